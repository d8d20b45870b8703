// decode.cu -- decode-side kernels of libgdn: the fused one-launch layer step
// (single token; the K=2 verify form with its rollback snapshot; the K = 2..8
// verify with a snapshot per position; the step that reads the snapshot an
// accepted count selects), the standalone gate / conv / recurrence / gated-norm
// kernels it is equal to bit for bit, and the verify commit.
//
// Decode is bound by HBM bandwidth on the recurrent state (128x128 fp32 per
// V head, read once and written once per step); everything else is small.
// Work split: one CTA per (sequence, V head, 128/NSPLIT value rows), 8 warps,
// each warp streaming 4*NG rows held in registers. The CTAs that share a QK
// head (r V heads x NSPLIT row slices) form one thread-block cluster, whose
// barrier orders every CTA's read of the shared Q/K conv history before its
// single owner rewrites it. The row slices of a head push their gated-norm
// partial sums into one another's shared memory (st.async, counted on the
// receiver's mbarrier), so no second cluster barrier is needed.
#include <type_traits>

#include "cluster.cuh"
#include "gdn_device.cuh"
#include "gdn_kernels.h"


namespace gdn {

// Bit 16: gdn_verify_commit saw an accepted count outside 1..2 (that sequence
// was left unchanged). Bit 128: a row slice of the fused step gave up (after
// 2 s) waiting for the other slices' norm partials; its outputs are then not
// valid. The one other wait in this file is the cluster barrier, which every
// CTA of a cluster reaches. Read and cleared by take_decode_device_error.
static __device__ int g_decode_error;
constexpr int kErrAcceptRange = 16;
constexpr int kErrNormWait = 128;
constexpr uint64_t kNormWaitNs = 2000000000ull;   // the bounded wait for a peer's norm partials

// The shared::cluster address of this CTA's shared-memory word p in the CTA of cluster rank cr.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t cr)
{
    const uint32_t local = (uint32_t)__cvta_generic_to_shared(p);
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(cr));
    return remote;
}

// Stores v into the shared memory of another CTA of the cluster and counts its 4 bytes
// on that CTA's mbarrier (both addresses from cluster_addr).
__device__ __forceinline__ void store_to_peer(uint32_t dst, float v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 :: "r"(dst), "r"(__float_as_uint(v)), "r"(bar) : "memory");
}

// Waits (bounded by the global timer) for phase `parity` of a local mbarrier that other
// CTAs of the cluster complete; acquire at cluster scope, so their stores are visible.
__device__ __forceinline__ bool wait_peers(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    uint64_t t0 = 0;
    for (int it = 0;; ++it) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        if (done)
            return true;
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (it == 0)
            t0 = t;
        else if (t - t0 > limit_ns)
            return false;
    }
}

// ------------------------------------------------------------------ decay gate
template <typename TIn>
__global__ void __launch_bounds__(256) decay_gate_kernel(const TIn *alpha, int64_t alpha_stride,
                                                         const float *dt, const float *A_log,
                                                         float *g, int rows, int H)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)rows * H)
        return;
    const int64_t r = i / H;
    const int h = (int)(i % H);
    GDN_CHECK(g_decode_error, r < rows && h < H);
    g[i] = decay_gate_f(load_act<TIn>(alpha + r * alpha_stride + h), __ldg(dt + h), __ldg(A_log + h));
}

// ------------------------------------------------------------------ recurrence
template <int NSPLIT>
__global__ void __launch_bounds__(256, 2) recurrence_decode_kernel(RecArgs a)
{
    constexpr int ROWS = kD / NSPLIT;
    constexpr int RPW = ROWS / 8;
    constexpr int NG = RPW / 4;
    __shared__ __align__(16) float sq[kD];
    __shared__ __align__(16) float sk[kD];
    __shared__ float sv[ROWS], sy[ROWS];
    __shared__ float sdecay[1], sbeta[1];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int b = blockIdx.y;
    const int h = blockIdx.x / NSPLIT, split = blockIdx.x % NSPLIT;
    const int hk = h / (a.Hv / a.Hq);
    const int row0 = split * ROWS;
    GDN_CHECK(g_decode_error, b < a.B && h < a.Hv && hk < a.Hq && row0 + ROWS <= kD);
    float *rows = a.state + (((size_t)b * a.Hv + h) * kD + row0 + warp * RPW) * kD;
    float4 r[NG][4];
    load_rows<NG>(rows, r);
    if (tid < kD)
        sq[tid] = __ldg(a.q + (int64_t)b * a.qkv_stride + hk * kD + tid);
    else
        sk[tid - kD] = __ldg(a.k + (int64_t)b * a.qkv_stride + hk * kD + (tid - kD));
    if (tid < ROWS)
        sv[tid] = __ldg(a.v + (int64_t)b * a.qkv_stride + h * kD + row0 + tid);
    if (tid == 255) {
        sdecay[0] = expf(__ldg(a.g + (size_t)b * a.Hv + h));
        sbeta[0] = __ldg(a.beta + (size_t)b * a.Hv + h);
    }
    __syncthreads();
    step_rows<NG, 1, false>(r, nullptr, sk, sq, sv, ROWS, sdecay, sbeta, sy, warp * RPW, a.scale);
    store_rows<NG>(r, rows);
    __syncthreads();
    if (tid < ROWS)
        a.y[((size_t)b * a.Hv + h) * kD + row0 + tid] = sy[tid];
}

// ------------------------------------------------------------------ gated norm
// One warp per (row, head); lane l holds elements l, 32+l, 64+l, 96+l.
template <typename TZ>
__global__ void __launch_bounds__(256) gated_norm_kernel(const float *y, const float *w,
                                                         const TZ *z, int64_t z_stride,
                                                         float *out, int rows, int Hv, float eps)
{
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= (int64_t)rows * Hv)
        return;
    const int64_t row = gw / Hv;
    const int h = (int)(gw % Hv);
    GDN_CHECK(g_decode_error, row < rows && h < Hv);
    const float *yr = y + gw * kD;
    float yv[4], bp[4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
        yv[m] = yr[32 * m + lane];
#pragma unroll
    for (int m = 0; m < 4; ++m)
        bp[m] = norm_block_partial(yv[m]);
    const float inv = norm_inv(bp[0], bp[1], bp[2], bp[3], eps);
    const TZ *zr = z + row * z_stride + (int64_t)h * kD;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int j = 32 * m + lane;
        out[gw * kD + j] = gated_out(yv[m], inv, __ldg(w + j), load_act<TZ>(zr + j));
    }
}

// ------------------------------------------------------------------ fused step
// NTOK = 1: one decode step. NTOK = 2: K=2 verify, snapshot after token 0, or
// (with the per-token snapshot layout) the generic K-token verify for K = 2..8.
//
// Order of a CTA's work, chosen so that no fence ever waits on the state
// loads or stores: (0) wait for the previous kernel in the stream (the launch
// is a programmatic dependent of it); (1) conv-window, gate, z and norm-gain
// loads, (2) state-row and conv-history loads, one memory round trip; (3) conv + SiLU, then cluster arrive (every
// read of the shared Q/K history is done); (4) L2, gates; (5) recurrence in
// registers, each 4-row group stored as soon as it is stepped (its stores
// overlap the later groups' arithmetic); (6) gated norm (when NSPLIT > 1: cluster
// wait, then each row slice of a head pushes its partial sums to the others and
// waits for theirs: one one-way trip instead of a second cluster barrier and
// remote reads, 3.64 -> 3.25 us per single-sequence step); (7) the single owner
// of each Q/K channel rewrites its history (after the cluster wait, which for
// NSPLIT == 1 comes here).
//
// TS is the storage type of the state and the output: float, or bf16 for the
// bf16-state decode (NTOK = 1 only), whose rows are widened to fp32 on load,
// stepped in fp32 and rounded to nearest even on store.
template <typename TIn, int NTOK, int NSPLIT, typename TS = float>
__global__ void __launch_bounds__(256, sizeof(TS) == 4 ? 2 : 3) decode_fused_kernel(FusedArgs a)
{
    static_assert(sizeof(TS) == 4 || NTOK == 1, "snapshots are float32");
    TS *const state = static_cast<TS *>(a.state);
    TS *const out = static_cast<TS *>(a.out);
    constexpr int ROWS = kD / NSPLIT;   // value rows of one head in this CTA
    constexpr int RPW = ROWS / 8;       // rows per warp
    constexpr int NG = RPW / 4;         // 4-row groups per warp
    constexpr int NBLK = ROWS / 32;     // 32-row norm blocks in this CTA
    constexpr bool SNAP = NTOK >= 2;
    // snapshot layouts: the two-token verify keeps the state and conv window after token
    // 0 (one entry); the generic form (conv_snap_entries == NTOK) keeps the state after
    // each of the first NTOK - 1 tokens ([B][NTOK-1][Hv][d][d]) and the conv window after
    // every token ([B][NTOK][conv_dim][W-1], the last one the committed window)
    const bool per_token = SNAP && a.conv_snap_entries == NTOK;
    __shared__ __align__(16) float sq[NTOK * kD];
    __shared__ __align__(16) float sk[NTOK * kD];
    __shared__ float sv[NTOK * ROWS], sy[NTOK * ROWS];
    __shared__ float sdecay[NTOK], sbeta[NTOK];
    __shared__ float sred[NTOK][8];
    __shared__ float spart[NTOK * NBLK];
    // the other row slices' partials, pushed by their CTAs: [sender slice][token][block]
    __shared__ float rpart[(NSPLIT > 1 ? NSPLIT : 1) * NTOK * NBLK];
    __shared__ __align__(8) uint64_t rbar;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.y;
    const int h = blockIdx.x / NSPLIT, split = blockIdx.x % NSPLIT;
    const int r = a.Hv / a.Hq;
    const int hk = h / r;
    const int csize = r * NSPLIT;                 // CTAs sharing QK head hk
    const int crank = blockIdx.x % csize;          // rank in the cluster
    const int W = a.W, cd = a.conv_dim;
    const int row0 = split * ROWS;
    const int64_t tok0 = (int64_t)b * NTOK;       // input row of token 0 of sequence b
    const TIn *xb = static_cast<const TIn *>(a.x) + tok0 * a.x_stride;
    float *histb = a.conv_state + (size_t)b * cd * (W - 1);

    const size_t head_off = ((size_t)b * a.Hv + h) * kD * kD;
    const size_t warp_off = (size_t)(row0 + warp * RPW) * kD;
    GDN_CHECK(g_decode_error, b < a.B && h < a.Hv && hk < a.Hq && split < NSPLIT && row0 + ROWS <= kD &&
                                  crank < csize);

    // (0) the layer parameters: the conv taps, the norm gain, dt and A_log. The launch is
    // a programmatic dependent of the previous kernel in the stream, so the CTA may be
    // resident while that kernel finishes; these loads are the only reads issued before
    // it has completed (the parameters are constant across steps and no kernel just
    // before a step writes them). Everything else may come from that kernel: the
    // activations from the projection before the step, the state and the conv history
    // from the previous step.
    const bool is_k = tid >= kD;
    const int c_qk = (is_k ? a.Hq * kD : 0) + hk * kD + (tid & (kD - 1));
    const int c_v = 2 * a.Hq * kD + h * kD + row0 + tid;
    GDN_CHECK(g_decode_error, c_qk < 2 * a.Hq * kD && (tid >= ROWS || (c_v >= 2 * a.Hq * kD && c_v < cd)));
    ConvWindow<NTOK> wqk, wv;
#pragma unroll
    for (int tau = 0; tau < kMaxW; ++tau) {
        wqk.w[tau] = tau < W ? __ldg(a.conv_w + (size_t)c_qk * W + tau) : 0.0f;
        wv.w[tau] = (tid < ROWS && tau < W) ? __ldg(a.conv_w + (size_t)c_v * W + tau) : 0.0f;
    }
    const float nw = tid < ROWS ? __ldg(a.norm_w + row0 + tid) : 0.0f;
    const bool gate_thread = tid >= ROWS && tid < ROWS + NTOK;
    float g_alpha = 0.0f, g_bl = 0.0f, g_dt = 0.0f, g_alog = 0.0f;
    if (gate_thread) {
        g_dt = __ldg(a.dt + h);
        g_alog = __ldg(a.A_log + h);
    }
    // the slices of a head push their norm partials to one another: each CTA's barrier
    // completes when the other slices' bytes have landed (initialised before the cluster
    // barrier that every CTA passes before it sends)
    if (NSPLIT > 1 && tid == 0) {
        const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&rbar);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar));
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     :: "r"(bar), "r"((uint32_t)((NSPLIT - 1) * NTOK * NBLK * 4)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // a grid of at most one wave starts while the previous kernel finishes: its CTAs
    // bring their state rows into L2 ahead of the wait. Nothing is read into registers
    // before the wait, and L2 is where every SM's stores land, so rows that kernel is
    // still writing are current there when the loads below read them.
    const bool one_wave = (long long)gridDim.x * gridDim.y <= 2LL * a.sm_count;
    if (NTOK == 1 && a.n_accept == nullptr && tid < 4 && one_wave) {
        const uint32_t quarter = ROWS * kD * sizeof(TS) / 4;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                     :: "l"(reinterpret_cast<const char *>(state + head_off + (size_t)row0 * kD) + tid * quarter),
                        "r"(quarter)
                     : "memory");
    }
    wait_previous_grid();
    // A launch of at most one wave lets the next kernel in the stream make its CTAs
    // resident from here on (they take free slots, read their parameters and prefetch
    // their rows, then wait for this whole grid): 3.66 -> 3.64 us per single-sequence
    // step. Larger launches trigger after their state stores, below, so that waiting
    // CTAs do not take slots from their later waves.
    if (one_wave)
        allow_next_grid();

    // (1) the conv windows' new rows, z and the gate inputs
    float zj[NTOK];
    auto load_inputs = [&]() {
#pragma unroll
        for (int e = 0; e < kMaxW - 1 + NTOK; ++e) {
            if (e >= W - 1 && e < W - 1 + NTOK) {
                wqk.win[e] = load_act<TIn>(xb + c_qk + (int64_t)(e - (W - 1)) * a.x_stride);
                if (tid < ROWS)
                    wv.win[e] = load_act<TIn>(xb + c_v + (int64_t)(e - (W - 1)) * a.x_stride);
            } else if (e >= W - 1 + NTOK) {
                wqk.win[e] = 0.0f;
                wv.win[e] = 0.0f;
            }
        }
        if (tid < ROWS) {
#pragma unroll
            for (int p = 0; p < NTOK; ++p)
                zj[p] = load_act<TIn>(static_cast<const TIn *>(a.z) + (tok0 + p) * a.z_stride +
                                      (int64_t)h * kD + row0 + tid);
        }
        if (gate_thread) {
            const int64_t row = tok0 + (tid - ROWS);
            g_alpha = load_act<TIn>(static_cast<const TIn *>(a.alpha) + row * a.gate_stride + h);
            g_bl = load_act<TIn>(static_cast<const TIn *>(a.beta_logit) + row * a.gate_stride + h);
        }
    };
    // (2) where the entering state and conv window are read: the live arrays, or, in the
    // step that follows a K-token verify, the snapshot sequence b's accepted count n
    // selects (n < K: the state after its n accepted tokens). The results always go to
    // the live arrays, so the rollback costs no copy. Then the conv windows' history.
    const TS *src_rows = state + head_off;
    const float *src_hist = histb;
    auto load_hist = [&]() {
        if (NTOK == 1 && a.n_accept != nullptr) {
            const int K = a.n_draft;
            int n = __ldg(a.n_accept + b);
            if (n < 1 || n > K) {
                if (blockIdx.x == 0 && tid == 0)
                    atomicOr(&g_decode_error, kErrAcceptRange);
                n = K;
            }
            if (n < K) {
                GDN_CHECK(g_decode_error, n - 1 < K - 1 && n - 1 < a.conv_snap_entries);
                src_rows = static_cast<const TS *>(a.state_snap) +
                           (((size_t)b * (K - 1) + (n - 1)) * a.Hv + h) * kD * kD;
                src_hist = a.conv_snap + ((size_t)b * a.conv_snap_entries + (n - 1)) * cd * (W - 1);
            }
        }
        conv_window_load_hist<NTOK>(src_hist + (size_t)c_qk * (W - 1), W, wqk);
        if (tid < ROWS)
            conv_window_load_hist<NTOK>(src_hist + (size_t)c_v * (W - 1), W, wv);
    };
    // Which group is requested first is a measured choice per form: the history first
    // for float32 rows with a whole head per CTA (batched decode 75.7 -> 69.6 us per
    // step, two-token verify 45.2 -> 43.2 us per launch), the new rows first otherwise
    // (single-sequence decode 4.56 -> 3.93 us per step, bf16 state 50.8 -> 48.7 us).
    if constexpr (NSPLIT == 1 && sizeof(TS) == 4) {
        load_hist();
        load_inputs();
    } else {
        load_inputs();
        load_hist();
    }

    // (3) this warp's state rows, float32 as float4; bf16 rows stay packed (half the
    // registers: 3 CTAs per SM)
    using Reg = typename std::conditional<sizeof(TS) == 4, float4, uint2>::type;
    Reg st[NG][4];
    load_rows<NG>(src_rows + warp_off, st);
    // A launch of more than one wave brings into L2, one wave ahead, the new rows
    // (the conv input row and the z row of a sequence) of the CTAs that will start about a wave
    // later: the CTA at the head of each such sequence row (NSPLIT == 1 and NTOK == 1
    // only) issues one bulk L2 prefetch per row, after its own loads, so the later
    // CTAs' first loads, on which their conv waits, hit L2 (batched decode with its
    // inputs copied in from the host each step: 79.4 -> 74.8 us per step, the kernel
    // alone unchanged)
    if (NTOK == 1 && NSPLIT == 1 && !one_wave && tid == 0) {
        const long long L = (long long)blockIdx.y * gridDim.x + blockIdx.x + 2LL * a.sm_count;
        if (L < (long long)gridDim.x * gridDim.y && L % gridDim.x == 0) {
            const long long bn = L / gridDim.x;
            const char *xr = reinterpret_cast<const char *>(static_cast<const TIn *>(a.x) + bn * a.x_stride);
            const char *zr = reinterpret_cast<const char *>(static_cast<const TIn *>(a.z) + bn * a.z_stride);
            const uint32_t xb = (uint32_t)(cd * sizeof(TIn)), zb = (uint32_t)(a.Hv * kD * sizeof(TIn));
            if ((reinterpret_cast<uintptr_t>(xr) & 15) == 0 && (xb & 15) == 0)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(xr), "r"(xb) : "memory");
            if ((reinterpret_cast<uintptr_t>(zr) & 15) == 0 && (zb & 15) == 0 &&
                (zr < xr || zr >= xr + xb))
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(zr), "r"(zb) : "memory");
        }
    }
    if constexpr (sizeof(TS) == 2) {
        // bf16 rows (3 CTAs per SM): also prefetch into L2 the state block of the
        // CTA one SM count later in launch order, about a third of a wave ahead
        // (measured: 52.3 -> 49.8 us per 64 x 48-head step; for float32 rows the
        // same prefetch slows the step, 84 -> 89 us, so it is not issued there)
        if (threadIdx.x < 4) {
            const long long L = (long long)blockIdx.y * gridDim.x + blockIdx.x + a.sm_count;
            if (L < (long long)gridDim.x * gridDim.y) {
                const int bb = (int)(L / gridDim.x), xx = (int)(L % gridDim.x);
                const TS *src = state + (((size_t)bb * a.Hv + xx / NSPLIT) * kD +
                                         (xx % NSPLIT) * ROWS) * kD;
                const uint32_t quarter = ROWS * kD * sizeof(TS) / 4;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                             :: "l"(reinterpret_cast<const char *>(src) + threadIdx.x * quarter),
                                "r"(quarter)
                             : "memory");
            }
        }
    }
    // (4) conv + SiLU; every read of the shared Q/K history is now complete: the
    // arrive below issues after the arithmetic that consumed those loads (a
    // warp issues in order), so it needs no release fence, which would also
    // wait for this warp's state loads still in flight
    float vals[NTOK];
#pragma unroll
    for (int p = 0; p < NTOK; ++p)
        vals[p] = silu_f(conv_window_pre<NTOK>(wqk, W, p));
    if (csize > 1)
        cluster_arrive_relaxed();

    // (4) V rows (exclusively owned: history rewritten at once), gates, Q/K L2
    if (tid < ROWS) {
#pragma unroll
        for (int p = 0; p < NTOK; ++p)
            sv[p * ROWS + tid] = silu_f(conv_window_pre<NTOK>(wv, W, p));
        float nh[kMaxW - 1];
        if (SNAP) {
#pragma unroll
            for (int p = 0; p < NTOK; ++p)
                if (per_token || p == 0) {
                    conv_window_history<NTOK>(wv, W, p + 1, nh);
                    store_history(a.conv_snap + ((size_t)(b * (per_token ? NTOK : 1) + p) * cd + c_v) * (W - 1),
                                  W, nh);
                }
        }
        conv_window_history<NTOK>(wv, W, NTOK, nh);
        store_history(histb + (size_t)c_v * (W - 1), W, nh);
    } else if (gate_thread) {
        const int p = tid - ROWS;
        sdecay[p] = expf(decay_gate_f(g_alpha, g_dt, g_alog));
        sbeta[p] = sigmoid_f(g_bl);
    }
#pragma unroll
    for (int p = 0; p < NTOK; ++p) {
        const float inv = head_l2_inv(vals[p], a.l2_eps, &sred[p][is_k ? 4 : 0], warp & 3, lane);
        (is_k ? sk : sq)[p * kD + (tid & (kD - 1))] = __fmul_rn(vals[p], inv);
    }
    __syncthreads();

    // (5) recurrence over this CTA's rows, in registers; the rows go back to HBM group
    // by group as they are finished
    float *snap_rows = nullptr;
    if (SNAP)
        snap_rows = static_cast<float *>(a.state_snap) + warp_off +
                    (per_token ? ((size_t)b * (NTOK - 1) * a.Hv + h) * kD * kD : head_off);
    step_rows<NG, NTOK, SNAP, TS, Reg>(st, snap_rows, sk, sq, sv, ROWS, sdecay, sbeta, sy, warp * RPW,
                                       a.scale, state + head_off + warp_off, per_token ? NTOK - 1 : 1,
                                       (size_t)a.Hv * kD * kD);
    // this CTA's state stores are issued: a dependent launch that follows may make its
    // CTAs resident (it waits for this whole grid before it reads anything)
    if (!one_wave)
        allow_next_grid();
    __syncthreads();

    // (6) gated RMSNorm: 32-row block partials, combined in block order. Row slices of
    // a head push theirs to the head's other slices (after cluster phase 0, which also
    // ends every CTA's reads of the shared Q/K history)
    if (NSPLIT > 1)
        cluster_wait_acquire();
#pragma unroll
    for (int i = warp; i < NTOK * NBLK; i += 8) {
        const int p = i / NBLK, bl = i % NBLK;
        const float s = norm_block_partial(sy[p * ROWS + bl * 32 + lane]);
        if (lane == 0) {
            spart[p * NBLK + bl] = s;
            if (NSPLIT > 1) {
#pragma unroll
                for (int o = 0; o < NSPLIT; ++o) {
                    if (o == split)
                        continue;
                    const uint32_t cr = (uint32_t)((h % r) * NSPLIT + o);
                    store_to_peer(cluster_addr(rpart + split * NTOK * NBLK + p * NBLK + bl, cr), s,
                                  cluster_addr(&rbar, cr));
                }
            }
        }
    }
    __syncthreads();
    if (NSPLIT > 1 && tid < ROWS &&
        !wait_peers((uint32_t)__cvta_generic_to_shared(&rbar), 0, kNormWaitNs) && tid == 0)
        atomicOr(&g_decode_error, kErrNormWait);
    if (tid < ROWS) {
#pragma unroll
        for (int p = 0; p < NTOK; ++p) {
            float bp[4];
#pragma unroll
            for (int bg = 0; bg < 4; ++bg) {
                const int owner = bg / NBLK, loc = bg % NBLK;
                bp[bg] = (NSPLIT == 1 || owner == split) ? spart[p * NBLK + loc]
                                                         : rpart[owner * NTOK * NBLK + p * NBLK + loc];
            }
            const float inv = norm_inv(bp[0], bp[1], bp[2], bp[3], a.rms_eps);
            const int j = row0 + tid;
            const int64_t row = tok0 + p;
            store_out(out + ((size_t)row * a.Hv + h) * kD + j,
                      gated_out(sy[p * ROWS + tid], inv, nw, zj[p]));
        }
    }


    // (7) Q/K history: each channel rewritten by exactly one CTA of the cluster,
    // after every CTA of the cluster has read it
    if (csize > 1 && NSPLIT == 1)
        cluster_wait_acquire();
    if (tid % csize == crank) {
        float *hist_c = histb + (size_t)c_qk * (W - 1);
        float nh[kMaxW - 1];
        if (SNAP) {
#pragma unroll
            for (int p = 0; p < NTOK; ++p)
                if (per_token || p == 0) {
                    conv_window_history<NTOK>(wqk, W, p + 1, nh);
                    store_history(a.conv_snap + ((size_t)(b * (per_token ? NTOK : 1) + p) * cd + c_qk) * (W - 1),
                                  W, nh);
                }
        }
        conv_window_history<NTOK>(wqk, W, NTOK, nh);
        store_history(hist_c, W, nh);
    }
}

// ------------------------------------------------------------------ commit
__global__ void __launch_bounds__(256) verify_commit_kernel(float *state, float *conv_state,
                                                            const float *state_snap,
                                                            const float *conv_snap,
                                                            const int32_t *n_accept,
                                                            int64_t state_elems, int64_t hist_elems)
{
    const int b = blockIdx.y;
    const int n = __ldg(n_accept + b);
    if (n < 1 || n > 2) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            atomicOr(&g_decode_error, kErrAcceptRange);
        return;
    }
    if (n == 2)
        return;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const float4 *src = reinterpret_cast<const float4 *>(state_snap + b * state_elems);
    float4 *dst = reinterpret_cast<float4 *>(state + b * state_elems);
    for (int64_t i = i0; i < state_elems / 4; i += stride)
        __stcs(dst + i, __ldcs(src + i));
    for (int64_t i = i0; i < hist_elems; i += stride)
        conv_state[b * hist_elems + i] = conv_snap[b * hist_elems + i];
}

// ------------------------------------------------------------------ host launchers
template <typename TIn, int NTOK, typename TS = float>
static cudaError_t fused_dispatch(const FusedArgs &a, cudaStream_t s)
{
    const int r = a.Hv / a.Hq;
    const int ns = pick_nsplit(a.B, a.Hv, r, a.sm_count);
    const dim3 grid(a.Hv * ns, a.B, 1);
    switch (ns) {
    case 1: return launch_cluster(decode_fused_kernel<TIn, NTOK, 1, TS>, grid, r, s, a, true);
    case 2: return launch_cluster(decode_fused_kernel<TIn, NTOK, 2, TS>, grid, r * 2, s, a, true);
    default: return launch_cluster(decode_fused_kernel<TIn, NTOK, 4, TS>, grid, r * 4, s, a, true);
    }
}

cudaError_t launch_decode_fused_bf16_state(const FusedArgs &a, bool bf16, cudaStream_t s)
{
    return bf16 ? fused_dispatch<__nv_bfloat16, 1, __nv_bfloat16>(a, s)
                : fused_dispatch<float, 1, __nv_bfloat16>(a, s);
}

template <typename TIn>
static cudaError_t fused_dispatch_ntok(const FusedArgs &a, int ntok, cudaStream_t s)
{
    switch (ntok) {
    case 1: return fused_dispatch<TIn, 1>(a, s);
    case 2: return fused_dispatch<TIn, 2>(a, s);
    case 3: return fused_dispatch<TIn, 3>(a, s);
    case 4: return fused_dispatch<TIn, 4>(a, s);
    case 5: return fused_dispatch<TIn, 5>(a, s);
    case 6: return fused_dispatch<TIn, 6>(a, s);
    case 7: return fused_dispatch<TIn, 7>(a, s);
    case 8: return fused_dispatch<TIn, 8>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_fused(const FusedArgs &a, bool bf16, int ntok, cudaStream_t s)
{
    return bf16 ? fused_dispatch_ntok<__nv_bfloat16>(a, ntok, s) : fused_dispatch_ntok<float>(a, ntok, s);
}

cudaError_t launch_decay_gate(const void *alpha, bool bf16, int64_t alpha_stride, const float *dt,
                              const float *A_log, float *g, int rows, int H, cudaStream_t s)
{
    const int64_t n = (int64_t)rows * H;
    const unsigned blocks = (unsigned)((n + 255) / 256);
    if (bf16)
        decay_gate_kernel<<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(alpha),
                                                 alpha_stride, dt, A_log, g, rows, H);
    else
        decay_gate_kernel<<<blocks, 256, 0, s>>>(static_cast<const float *>(alpha), alpha_stride,
                                                 dt, A_log, g, rows, H);
    return cudaGetLastError();
}

cudaError_t launch_recurrence_decode(const RecArgs &a, cudaStream_t s)
{
    const int r = a.Hv / a.Hq;
    const int ns = pick_nsplit(a.B, a.Hv, r, sm_count());
    const dim3 grid(a.Hv * ns, a.B, 1);
    switch (ns) {
    case 1: recurrence_decode_kernel<1><<<grid, 256, 0, s>>>(a); break;
    case 2: recurrence_decode_kernel<2><<<grid, 256, 0, s>>>(a); break;
    default: recurrence_decode_kernel<4><<<grid, 256, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_gated_norm(const float *y, const float *w, const void *z, bool bf16,
                              int64_t z_stride, float *out, int rows, int Hv, float eps,
                              cudaStream_t s)
{
    const int64_t n = (int64_t)rows * Hv;
    const unsigned blocks = (unsigned)((n + 7) / 8);
    if (bf16)
        gated_norm_kernel<<<blocks, 256, 0, s>>>(y, w, static_cast<const __nv_bfloat16 *>(z),
                                                 z_stride, out, rows, Hv, eps);
    else
        gated_norm_kernel<<<blocks, 256, 0, s>>>(y, w, static_cast<const float *>(z), z_stride,
                                                 out, rows, Hv, eps);
    return cudaGetLastError();
}

cudaError_t take_decode_device_error(int *code)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(int));
    if (e == cudaSuccess && v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(int));
    }
    *code = v;
    return e;
}

cudaError_t launch_verify_commit(float *state, float *conv_state, const float *state_snap,
                                 const float *conv_snap, const int32_t *n_accept, int B,
                                 int64_t state_elems, int64_t hist_elems, cudaStream_t s)
{
    const dim3 grid(64, B, 1);
    verify_commit_kernel<<<grid, 256, 0, s>>>(state, conv_state, state_snap, conv_snap, n_accept,
                                              state_elems, hist_elems);
    return cudaGetLastError();
}

}  // namespace gdn
