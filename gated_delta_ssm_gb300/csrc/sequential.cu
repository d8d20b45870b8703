// sequential.cu -- kernels that step T tokens of every sequence one token at
// a time with the state rows held in registers throughout:
//
//   recurrence_scan_kernel  the sequential scan of the recurrence alone
//                           ("fm_kernel_ssm.h", "Delta-rule recurrence": the
//                           naive scan kept as the permanent correctness
//                           reference for the chunked path);
//   layer_scan_kernel       the whole fused layer step (conv + SiLU + Q/K L2,
//                           gates, recurrence, gated RMSNorm) over T tokens,
//                           optionally writing the rollback snapshot of every
//                           position: the generic-K draft verification of
//                           "ssm_mamba.rs" (gdn_verify_fused_conv_kn and its
//                           batched form), extended from the conv window to
//                           the recurrent state;
//   commit_kn_kernel        the rollback to the accepted prefix.
//
// Per token, every value is computed by the same device functions in the same
// order as the single-step kernels of decode.cu, so a T-token scan equals T
// single steps bit for bit. The mapping is decode's: one CTA per (sequence,
// V head, 128/NSPLIT value rows), 8 lanes per 512-byte state row; the CTAs
// that share a QK head form a cluster, which orders every CTA's read of the
// shared Q/K conv history before its owner rewrites it and carries the
// gated-norm partial sums between row slices.
#include <cooperative_groups.h>

#include "cluster.cuh"
#include "gdn_device.cuh"
#include "gdn_kernels.h"

namespace cg = cooperative_groups;

namespace gdn {

// Bit 16: gdn_verify_commit_kn saw an accepted count outside 1..K (that
// sequence was left unchanged). Read and cleared by take_sequential_device_error.
static __device__ int g_seq_error;
constexpr int kErrAcceptRange = 16;

namespace {

// ------------------------------------------------------------------ recurrence scan
template <int NSPLIT>
__global__ void __launch_bounds__(256, 2) recurrence_scan_kernel(RecScanArgs a)
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
    GDN_CHECK(g_seq_error, b < a.B && h < a.Hv && hk < a.Hq && row0 + ROWS <= kD);
    float *rows = a.state + (((size_t)b * a.Hv + h) * kD + row0 + warp * RPW) * kD;
    float4 st[NG][4];
    load_rows<NG>(rows, st);

    // this thread's operands of a token: a q (tid < 128) or k channel, a v row
    // (tid < ROWS), and the gate pair (tid 255)
    const float *qk_src = (tid < kD ? a.q : a.k) + hk * kD + (tid & (kD - 1));
    const float *v_src = a.v + h * kD + row0 + tid;
    const int64_t row_b = (int64_t)b * a.T;
    float nqk = 0.0f, nv = 0.0f, ng = 0.0f, nb = 0.0f;
    auto fetch = [&](int t) {
        const int64_t row = row_b + t;
        nqk = __ldg(qk_src + row * a.qkv_stride);
        if (tid < ROWS)
            nv = __ldg(v_src + row * a.qkv_stride);
        if (tid == 255) {
            ng = __ldg(a.g + row * a.Hv + h);
            nb = __ldg(a.beta + row * a.Hv + h);
        }
    };
    fetch(0);
    for (int t = 0; t < a.T; ++t) {
        (tid < kD ? sq : sk)[tid & (kD - 1)] = nqk;
        if (tid < ROWS)
            sv[tid] = nv;
        if (tid == 255) {
            sdecay[0] = expf(ng);
            sbeta[0] = nb;
        }
        __syncthreads();
        if (t + 1 < a.T)
            fetch(t + 1);
        step_rows<NG, 1, false>(st, nullptr, sk, sq, sv, ROWS, sdecay, sbeta, sy, warp * RPW,
                                a.scale);
        __syncthreads();
        if (tid < ROWS)
            a.y[((row_b + t) * a.Hv + h) * kD + row0 + tid] = sy[tid];
    }
    store_rows<NG>(st, rows);
}

// ------------------------------------------------------------------ layer scan
// The window of one conv channel advanced by one token: the history after
// the token (window entries 1 .. W-1) followed by the next raw input.
__device__ __forceinline__ void roll_window(ConvWindow<1> &cw, int W, float x_next)
{
    float nh[kMaxW - 1];
    conv_window_history<1>(cw, W, 1, nh);
#pragma unroll
    for (int e = 0; e < kMaxW; ++e) {
        if (e < W - 1)
            cw.win[e] = nh[e];
        else if (e == W - 1)
            cw.win[e] = x_next;
    }
}

// The history held by a rolled window (its first W-1 entries).
__device__ __forceinline__ void window_history(const ConvWindow<1> &cw, float (&nh)[kMaxW - 1])
{
#pragma unroll
    for (int e = 0; e < kMaxW - 1; ++e)
        nh[e] = cw.win[e];
}

// Token p of sequence b: conv windows (Q/K channel for every thread, V row for
// tid < ROWS) and the gate thread's inputs are loaded one token ahead.
// Per token: conv + SiLU, V outputs and V snapshot, gates, Q/K L2 (its block
// reduction is the first barrier), Q/K snapshot, recurrence, state snapshot,
// gated norm (block partials; row slices of a head combine them through
// distributed shared memory, double-buffered by token parity).
template <typename TIn, int NSPLIT>
__global__ void __launch_bounds__(256, 2) layer_scan_kernel(LayerScanArgs a)
{
    constexpr int ROWS = kD / NSPLIT;
    constexpr int RPW = ROWS / 8;
    constexpr int NG = RPW / 4;
    constexpr int NBLK = ROWS / 32;
    __shared__ __align__(16) float sq[kD];
    __shared__ __align__(16) float sk[kD];
    __shared__ float sv[ROWS], sy[ROWS];
    __shared__ float sdecay[1], sbeta[1];
    __shared__ float sred[8];
    __shared__ float spart[2][NBLK];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.y;
    const int h = blockIdx.x / NSPLIT, split = blockIdx.x % NSPLIT;
    const int r = a.Hv / a.Hq;
    const int hk = h / r;
    const int csize = r * NSPLIT;
    const int crank = blockIdx.x % csize;
    const int W = a.W, cd = a.conv_dim, T = a.T;
    const int row0 = split * ROWS;
    const int64_t tok0 = (int64_t)b * T;
    const TIn *xb = static_cast<const TIn *>(a.x) + tok0 * a.x_stride;
    float *histb = a.conv_state + (size_t)b * cd * (W - 1);

    const size_t head_off = ((size_t)b * a.Hv + h) * kD * kD;
    const size_t warp_off = (size_t)(row0 + warp * RPW) * kD;
    GDN_CHECK(g_seq_error, b < a.B && h < a.Hv && hk < a.Hq && row0 + ROWS <= kD && crank < csize);
    float4 st[NG][4];
    load_rows<NG>(a.state + head_off + warp_off, st);

    const bool is_k = tid >= kD;
    const bool has_v = tid < ROWS;
    const bool gate_thread = tid == ROWS;
    const int c_qk = (is_k ? a.Hq * kD : 0) + hk * kD + (tid & (kD - 1));
    const int c_v = 2 * a.Hq * kD + h * kD + row0 + tid;
    ConvWindow<1> wqk, wv;
    conv_window_load<TIn, 1>(histb + (size_t)c_qk * (W - 1), xb + c_qk, a.x_stride,
                             a.conv_w + (size_t)c_qk * W, W, wqk);
    float nw = 0.0f, zc = 0.0f;
    if (has_v) {
        conv_window_load<TIn, 1>(histb + (size_t)c_v * (W - 1), xb + c_v, a.x_stride,
                                 a.conv_w + (size_t)c_v * W, W, wv);
        nw = __ldg(a.norm_w + row0 + tid);
        zc = load_act<TIn>(static_cast<const TIn *>(a.z) + tok0 * a.z_stride + (int64_t)h * kD +
                           row0 + tid);
    }
    float g_alpha = 0.0f, g_bl = 0.0f, g_dt = 0.0f, g_alog = 0.0f;
    if (gate_thread) {
        g_alpha = load_act<TIn>(static_cast<const TIn *>(a.alpha) + tok0 * a.gate_stride + h);
        g_bl = load_act<TIn>(static_cast<const TIn *>(a.beta_logit) + tok0 * a.gate_stride + h);
        g_dt = __ldg(a.dt + h);
        g_alog = __ldg(a.A_log + h);
    }
    cg::cluster_group cluster = cg::this_cluster();

    for (int p = 0; p < T; ++p) {
        const float pre_qk = conv_window_pre<1>(wqk, W, 0);
        const float pre_v = has_v ? conv_window_pre<1>(wv, W, 0) : 0.0f;
        if (p == 0 && csize > 1)
            cluster_arrive_release();   // this CTA's reads of the shared Q/K history are done

        // next token's raw inputs, in flight during this token's work
        const int64_t nrow = tok0 + (p + 1 < T ? p + 1 : p);
        const float xq_n = load_act<TIn>(static_cast<const TIn *>(a.x) + nrow * a.x_stride + c_qk);
        float xv_n = 0.0f, z_n = 0.0f, alpha_n = 0.0f, bl_n = 0.0f;
        if (has_v) {
            xv_n = load_act<TIn>(static_cast<const TIn *>(a.x) + nrow * a.x_stride + c_v);
            z_n = load_act<TIn>(static_cast<const TIn *>(a.z) + nrow * a.z_stride +
                                (int64_t)h * kD + row0 + tid);
        }
        if (gate_thread) {
            alpha_n = load_act<TIn>(static_cast<const TIn *>(a.alpha) + nrow * a.gate_stride + h);
            bl_n = load_act<TIn>(static_cast<const TIn *>(a.beta_logit) + nrow * a.gate_stride + h);
        }

        const float vqk = silu_f(pre_qk);
        if (has_v) {
            sv[tid] = silu_f(pre_v);
            roll_window(wv, W, xv_n);
            if (a.conv_snap) {
                float nh[kMaxW - 1];
                window_history(wv, nh);
                store_history(a.conv_snap + ((size_t)(tok0 + p) * cd + c_v) * (W - 1), W, nh);
            }
        } else if (gate_thread) {
            sdecay[0] = expf(decay_gate_f(g_alpha, g_dt, g_alog));
            sbeta[0] = sigmoid_f(g_bl);
            g_alpha = alpha_n;
            g_bl = bl_n;
        }
        const float inv = head_l2_inv(vqk, a.l2_eps, &sred[is_k ? 4 : 0], warp & 3, lane);
        (is_k ? sk : sq)[tid & (kD - 1)] = __fmul_rn(vqk, inv);
        roll_window(wqk, W, xq_n);
        if (a.conv_snap && tid % csize == crank) {
            float nh[kMaxW - 1];
            window_history(wqk, nh);
            store_history(a.conv_snap + ((size_t)(tok0 + p) * cd + c_qk) * (W - 1), W, nh);
        }
        __syncthreads();

        // each 4-row group goes out as soon as it is stepped: to this position's
        // snapshot, and after the last position to the state itself
        float *dst = p + 1 == T ? a.state + head_off + warp_off
                     : a.state_snap ? a.state_snap + (((size_t)b * (T - 1) + p) * a.Hv + h) * kD * kD +
                                          warp_off
                                    : nullptr;
        step_rows<NG, 1, false>(st, nullptr, sk, sq, sv, ROWS, sdecay, sbeta, sy, warp * RPW,
                                a.scale, dst);
        __syncthreads();

        const int slot = p & 1;
        if (warp < NBLK) {
            const float s = norm_block_partial(sy[warp * 32 + lane]);
            if (lane == 0)
                spart[slot][warp] = s;
        }
        if (NSPLIT > 1) {
            // the previous phase (history reads at p == 0, else the peers'
            // reads of token p-1's partials), then publish this token's
            cluster_wait_acquire();
            cluster_arrive_release();
            cluster_wait_acquire();
        } else {
            __syncthreads();
        }
        if (has_v) {
            float bp[4];
#pragma unroll
            for (int bg = 0; bg < 4; ++bg) {
                const int owner = bg / NBLK, loc = bg % NBLK;
                if (NSPLIT == 1) {
                    bp[bg] = spart[slot][loc];
                } else {
                    const float *peer = cluster.map_shared_rank(&spart[0][0], (h % r) * NSPLIT + owner);
                    bp[bg] = peer[slot * NBLK + loc];
                }
            }
            const float ninv = norm_inv(bp[0], bp[1], bp[2], bp[3], a.rms_eps);
            a.out[((size_t)(tok0 + p) * a.Hv + h) * kD + row0 + tid] = gated_out(sy[tid], ninv, nw, zc);
            zc = z_n;
        }
        if (NSPLIT > 1)
            cluster_arrive_relaxed();   // this CTA's reads of its peers' partials are done
    }

    if (has_v) {
        float nh[kMaxW - 1];
        window_history(wv, nh);
        store_history(histb + (size_t)c_v * (W - 1), W, nh);
    }
    // every CTA of the cluster has read the shared Q/K history (and, with row
    // slices, finished reading this CTA's partials)
    if (csize > 1)
        cluster_wait_acquire();
    if (tid % csize == crank) {
        float nh[kMaxW - 1];
        window_history(wqk, nh);
        store_history(histb + (size_t)c_qk * (W - 1), W, nh);
    }
}

// ------------------------------------------------------------------ commit
// Sequence b keeps its first n = n_accept[b] positions: n == K leaves the
// committed state; n < K restores snapshot n-1.
__global__ void __launch_bounds__(256) commit_kn_kernel(float *state, float *conv_state,
                                                        const float *state_snap,
                                                        const float *conv_snap,
                                                        const int32_t *n_accept, int K,
                                                        int64_t state_elems, int64_t hist_elems)
{
    const int b = blockIdx.y;
    const int n = __ldg(n_accept + b);
    if (n < 1 || n > K) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            atomicOr(&g_seq_error, kErrAcceptRange);
        return;
    }
    if (n == K)
        return;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const float4 *src =
        reinterpret_cast<const float4 *>(state_snap + ((size_t)b * (K - 1) + (n - 1)) * state_elems);
    float4 *dst = reinterpret_cast<float4 *>(state + (size_t)b * state_elems);
    for (int64_t i = i0; i < state_elems / 4; i += stride)
        __stcs(dst + i, __ldcs(src + i));
    const float *hsrc = conv_snap + ((size_t)b * K + (n - 1)) * hist_elems;
    for (int64_t i = i0; i < hist_elems; i += stride)
        conv_state[(size_t)b * hist_elems + i] = hsrc[i];
}

template <typename TIn>
cudaError_t layer_scan_dispatch(const LayerScanArgs &a, cudaStream_t s)
{
    const int r = a.Hv / a.Hq;
    const int ns = scan_nsplit(a.B, a.Hv, r, sm_count());
    const dim3 grid(a.Hv * ns, a.B, 1);
    switch (ns) {
    case 1: return launch_cluster(layer_scan_kernel<TIn, 1>, grid, r, s, a);
    case 2: return launch_cluster(layer_scan_kernel<TIn, 2>, grid, r * 2, s, a);
    default: return launch_cluster(layer_scan_kernel<TIn, 4>, grid, r * 4, s, a);
    }
}

}  // namespace

cudaError_t launch_recurrence_scan(const RecScanArgs &a, cudaStream_t s)
{
    const int ns = scan_nsplit(a.B, a.Hv, 1, sm_count());
    const dim3 grid(a.Hv * ns, a.B, 1);
    switch (ns) {
    case 1: recurrence_scan_kernel<1><<<grid, 256, 0, s>>>(a); break;
    case 2: recurrence_scan_kernel<2><<<grid, 256, 0, s>>>(a); break;
    default: recurrence_scan_kernel<4><<<grid, 256, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_layer_scan(const LayerScanArgs &a, bool bf16, cudaStream_t s)
{
    return bf16 ? layer_scan_dispatch<__nv_bfloat16>(a, s) : layer_scan_dispatch<float>(a, s);
}

cudaError_t launch_verify_commit_kn(float *state, float *conv_state, const float *state_snap,
                                    const float *conv_snap, const int32_t *n_accept, int B, int K,
                                    int64_t state_elems, int64_t hist_elems, cudaStream_t s)
{
    const dim3 grid(64, B, 1);
    commit_kn_kernel<<<grid, 256, 0, s>>>(state, conv_state, state_snap, conv_snap, n_accept, K,
                                          state_elems, hist_elems);
    return cudaGetLastError();
}

cudaError_t take_sequential_device_error(int *code)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_seq_error, sizeof(int));
    if (e == cudaSuccess && v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_seq_error, &zero, sizeof(int));
    }
    *code = v;
    return e;
}

}  // namespace gdn
