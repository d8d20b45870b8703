// prefill.cu -- chunked prefill in two passes, on the tcgen05 tensor cores.
//
// The chunk algebra is derived from the recurrence of "fm_kernel_ssm.h",
// section "Delta-rule recurrence", over 64-token chunks joined by ceil(T/64)
// sequential state links (the "Mamba-2 SSD chunked prefill scan" note of
// "ssm_mamba.rs"). Per (sequence, V head, chunk), with Gam_t the in-chunk
// cumulative decay, S_0 the entering state (plain orientation S[i][j], i the
// key index, j the value index), K, Q the L2-normalised key / query rows and
// V the value rows of the chunk:
//   A   = strictly lower part of diag(beta) (e^{Gam_t - Gam_s}) (K K^T)
//   T   = (I + A)^-1                                   (the chunk's UT transform)
//   X   = diag(beta) (V - diag(e^Gam) K S_0)
//   U   = T X                                          (the delta-rule updates)
//   O   = diag(e^Gam) Q S_0 + P U,  P = lower part (s <= t) of e^{Gam_t - Gam_s} (Q K^T)
//   S_C = e^{Gam_C} S_0 + K^T diag(e^{Gam_C - Gam}) U
//
// Pass 1 (prefill_ut_kernel) is parallel over every (sequence, QK head,
// chunk): it stages the chunk's raw Q and K rows in shared memory by tensor
// copy, runs the conv + SiLU + L2 on them, forms G = [Q; K] K^T on the tensor
// core, and for each V head of the group builds P (from Q K^T) and A (from
// K K^T) in parallel and solves T = (I + A)^-1 in 16-token blocks (diagonal
// blocks by forward substitution, the blocks below them by warp-level tensor
// core products), writing T and P as 16 KB two-part fp16 operand images to the
// caller's workspace. Nothing in it depends on the state.
//
// Pass 2 (prefill_chain_kernel) walks the chunks of one (sequence, V head)
// with the fp32 state master in tensor memory. Its warps are specialised:
//   * 16 epilogue warps (four per TMEM lane quarter, value row j = lane, 16 tokens each):
//     X (with the V rows' SiLU), U' and U, the state re-split, the state
//     write-back and the readout rows;
//   * 1 product warp: one lane issues every product as soon as its operands are
//     ready and its accumulator is free;
//   * 1 copy warp: one lane refills every workspace buffer as soon as the
//     products that read it are done;
//   * 8 conv warps: the conv of chunk c+1's V rows (from the staged rows) while
//     chunk c's products run, and the gated RMSNorm of chunk c's outputs.
// The products (transposed orientation, M = 128 value rows j, A operands in
// tensor memory, B operands in shared memory):
//   D1 = S_0^T [Q; K]^T        ((Q S_0)^T | (K S_0)^T)
//   D2 = X^T T^T = U^T         (the UT transform on the tensor core)
//   S^T += U'^T K              (U' = diag(e^{Gam_C - Gam}) U; K read MN-major)
//   (P U)^T = U^T P^T          (into D2 once U^T is read; O = e^Gam Q S_0 + P U is
//                               summed in the epilogue)
// so that the sequential part per chunk is three products and three short
// epilogues; everything that does not depend on the state runs ahead.
//
// Precision: every operand is an fp32 value split into two fp16 parts
// (x = x1 + x2, ~22 bits; products x1 y1 + x1 y2 + x2 y1), accumulation fp32.
//
// Every wait is bounded by the global timer (PrefillArgs::wait_ns); a wait that
// gives up sets a bit of the device error word, the other roles stop at their
// next wait, in-flight copies and products are drained, tensor memory is freed
// and the kernel returns.
#include <algorithm>

#include <cuda_fp16.h>

#include "gdn_device.cuh"
#include "gdn_kernels.h"
#include "tc_ptx.cuh"
#include "tma_map.cuh"

namespace gdn {

// Set when a bounded wait of a kernel in this file gives up; read and cleared
// by take_prefill_device_error.
static __device__ int g_device_error;

namespace {

constexpr int kC = 64;
constexpr uint32_t kErrChain = 1, kErrUT = 2, kErrDrain = 8;
// The normalised Q / K rows (entries at most 1) enter the tensor core scaled by
// 16, so that the low fp16 part of most entries is a normal number; every
// product that contains them is scaled back by the same power of two.
constexpr float kQK = 16.0f, kInvQK = 1.0f / 16.0f, kInvQK2 = 1.0f / 256.0f;

// ------------------------------------------------------------------ small helpers
// Tensor-core operands are fp32 values split into two fp16 parts, x = hi + lo
// (hi = fp16(x), lo = fp16(x - hi)): 22 significant bits for |x| >= 0.25 and an
// absolute representation error below 2^-25 for smaller x, at the price of
// fp16's range (every operand, i.e. the normalised Q/K rows, the state, X, U, P
// and T, must stay below 65504 in magnitude). Both pairs packed, element a in
// the low half.
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo)
{
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(__fsub_rn(a, hf.x), __fsub_rn(b, hf.y));
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Two-float arithmetic for the in-chunk cumulative decay Gam: its values reach
// hundreds while the decays exp(Gam_t - Gam_s) need the differences to full
// float precision, so Gam is carried as hi + lo (Knuth's TwoSum keeps the
// rounding error of every addition).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void two_add(float &h, float &l, float bh, float bl)
{
    float s, e;
    two_sum(h, bh, s, e);
    const float t = __fadd_rn(__fadd_rn(l, bl), e);
    h = __fadd_rn(s, t);
    l = __fsub_rn(t, __fsub_rn(h, s));
}

// exp((ah + al) - (bh + bl)) with the difference formed exactly before rounding
__device__ __forceinline__ float exp_diff(float ah, float al, float bh, float bl)
{
    float dh, de;
    two_sum(ah, -bh, dh, de);
    const float dl = __fadd_rn(de, __fsub_rn(al, bl));
    return __fmul_rn(expf(dh), __fadd_rn(1.0f, dl));
}

// The same with the hardware exponential (__expf): a relative error of a few
// 1e-6 at the largest in-chunk differences, for the 2 x 64 x 64 decay factors of
// P and A of every chunk and head
__device__ __forceinline__ float exp_diff_fast(float ah, float al, float bh, float bl)
{
    float dh, de;
    two_sum(ah, -bh, dh, de);
    const float dl = __fadd_rn(de, __fsub_rn(al, bl));
    return __fmul_rn(__expf(dh), __fadd_rn(1.0f, dl));
}

// 2^e for an integer e in [-126, 127], exactly
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

// One chunk's gate values ("fm_kernel_ssm.h" "Decay gate"; beta = sigmoid),
// formed in the chunk-parallel pass and copied whole to the chain pass.
//
// The chain keeps the fp32 state master scaled by a power of two, 2^rho S, with
// rho chosen per chunk from the gates so that the scaled state stays of order
// one however strongly it has decayed: the fp16 operand parts split from it
// (and the update U' that adds to it) then stay in fp16's normal range. Chunk c
// enters with rho_c and leaves with rho_{c+1} = next_rho(G, rho_c); the chain
// multiplies the factors below by those exact powers of two (2^-rho_c for eg,
// bg; 2^rho_{c+1} for egc; 2^(rho_{c+1} - rho_c) for ec).
struct Gates {
    float beta[kC];        // beta_t, 0 at or past the end of the call
    float gh[kC], gl[kC];  // Gam_t = g_0 + ... + g_t (two floats); g = 0 past the end
    float eg[kC];          // exp(Gam_t) / 16                   (scales 16 (Q S_0)^T)
    float egc[kC];         // exp(Gam_C - Gam_t) / 16, 0 past the end  (U' against 16 K)
    float bg[kC];          // beta_t exp(Gam_t) / 16            (scales 16 (K S_0)^T)
    float ec;              // exp(Gam_C)                        (the master's decay)
    float lc;              // log2 exp(Gam_C)
    float lu;              // max_t log2(beta_t exp(Gam_C - Gam_t)), -1e30 if no update
    float pad[13];
};
static_assert(sizeof(Gates) % 16 == 0, "gates travel by bulk copy");

// rho_{c+1}: with the entering scaled state of order one, the state after the
// chunk has magnitude about max(e^{Gam_C} 2^-rho_c, max_t beta_t e^{Gam_C - Gam_t})
// (times the values' scale); lmax is its log2 and rho_{c+1} = -lmax brings it
// back to order one. Since 2^rho_{c+1} <= 1 / (beta_t e^{Gam_C - Gam_t}), the
// update factors egc 2^rho_{c+1} stay bounded by 1 / (16 beta_t).
__device__ __forceinline__ int next_rho(const Gates *G, int rho)
{
    const float lmax = fmaxf(G->lc - (float)rho, G->lu);
    return (int)fminf(fmaxf(floorf(-lmax), 0.0f), 60.0f);
}

// Gates of tokens c0 .. c0+n-1 of sequence b, V head h; executed by one warp. With cf
// set, also the decays from each 16-token block start back to the earlier tokens:
// cf[64 (I - 1) + s] = exp(Gam_{16 I} - Gam_s) for I = 1, 2, 3 and s < 16 I (at most 1:
// Gam does not increase).
template <typename TIn>
__device__ __forceinline__ void chunk_gates(const PrefillArgs &a, int b, int h, int c0, int n, Gates *G,
                                            float *cf = nullptr)
{
    const int lane = threadIdx.x & 31;
    const float dtv = __ldg(a.dt + h), alog = __ldg(a.A_log + h);
    const int64_t row0 = (int64_t)b * a.T + c0;
    const TIn *al = static_cast<const TIn *>(a.alpha) + row0 * a.gate_stride + h;
    const TIn *bl = static_cast<const TIn *>(a.beta_logit) + row0 * a.gate_stride + h;
    float gv[2], bv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int t = 2 * lane + u;
        gv[u] = t < n ? decay_gate_f(load_act<TIn>(al + (int64_t)t * a.gate_stride), dtv, alog) : 0.0f;
        bv[u] = t < n ? sigmoid_f(load_act<TIn>(bl + (int64_t)t * a.gate_stride)) : 0.0f;
        G->beta[t] = bv[u];
    }
    // inclusive scan of the token pairs in two-float arithmetic
    float ph, pl;
    two_sum(gv[0], gv[1], ph, pl);
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float yh = __shfl_up_sync(0xffffffffu, ph, off);
        const float yl = __shfl_up_sync(0xffffffffu, pl, off);
        if (lane >= off)
            two_add(ph, pl, yh, yl);
    }
    float exh = __shfl_up_sync(0xffffffffu, ph, 1);
    float exl = __shfl_up_sync(0xffffffffu, pl, 1);
    if (lane == 0)
        exh = exl = 0.0f;
    float g0h = exh, g0l = exl;
    two_add(g0h, g0l, gv[0], 0.0f);
    float g1h = g0h, g1l = g0l;
    two_add(g1h, g1l, gv[1], 0.0f);
    const float gch = __shfl_sync(0xffffffffu, g1h, 31);
    const float gcl = __shfl_sync(0xffffffffu, g1l, 31);
    G->gh[2 * lane] = g0h;
    G->gl[2 * lane] = g0l;
    G->gh[2 * lane + 1] = g1h;
    G->gl[2 * lane + 1] = g1l;
    const float l2e = 1.4426950408889634f;
    const float dc0 = 2 * lane < n ? exp_diff(gch, gcl, g0h, g0l) : 0.0f;
    const float dc1 = 2 * lane + 1 < n ? exp_diff(gch, gcl, g1h, g1l) : 0.0f;
    float lu = -1e30f;   // log2 of the largest update factor of the warp's two tokens
    if (bv[0] > 0.0f && dc0 > 0.0f)
        lu = __log2f(bv[0]) + __fmul_rn(__fadd_rn(__fsub_rn(gch, g0h), __fsub_rn(gcl, g0l)), l2e);
    if (bv[1] > 0.0f && dc1 > 0.0f)
        lu = fmaxf(lu, __log2f(bv[1]) + __fmul_rn(__fadd_rn(__fsub_rn(gch, g1h), __fsub_rn(gcl, g1l)), l2e));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        lu = fmaxf(lu, __shfl_xor_sync(0xffffffffu, lu, m));
    const float e0 = __fmul_rn(exp_diff(g0h, g0l, 0.0f, 0.0f), kInvQK);
    const float e1 = __fmul_rn(exp_diff(g1h, g1l, 0.0f, 0.0f), kInvQK);
    G->eg[2 * lane] = e0;
    G->eg[2 * lane + 1] = e1;
    G->bg[2 * lane] = __fmul_rn(bv[0], e0);
    G->bg[2 * lane + 1] = __fmul_rn(bv[1], e1);
    G->egc[2 * lane] = __fmul_rn(dc0, kInvQK);
    G->egc[2 * lane + 1] = __fmul_rn(dc1, kInvQK);
    if (lane == 0) {
        G->ec = exp_diff(gch, gcl, 0.0f, 0.0f);
        G->lc = __fmul_rn(__fadd_rn(gch, gcl), l2e);
        G->lu = lu;
    }
    if (cf != nullptr) {
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int sidx = lane + 32 * u;
#pragma unroll
            for (int I = 1; I < 4; ++I)
                if (sidx < 16 * I)
                    cf[64 * (I - 1) + sidx] = exp_diff_fast(G->gh[16 * I], G->gl[16 * I], G->gh[sidx], G->gl[sidx]);
        }
    }
}

// conv + SiLU ("fm_kernel_ssm.h", "Causal depthwise conv1d + SiLU") of the
// NCH (4 or 8) channels ch0 .. ch0+NCH-1 for tokens t0 .. t0+7 of the chunk that
// starts at token c0 of the call; tokens at or past n give 0. With four taps the
// weights may come from a table in shared memory (wsm[e * wstride] = channel
// ch0 + e's taps) instead of global memory. Stream index
// s < 0 of the call reads the fp32 history, s >= T reads 0. With staged set,
// raw_s is the shared-window address of the chunk's rows of this channel's
// 128-channel head ([63 + W][128] bf16, row r = token c0 - (W-1) + r); otherwise
// x is read directly. Taps are summed oldest first.
template <int NCH, typename TIn>
__device__ __forceinline__ void load_row(const TIn *p, float (&v)[NCH]);
template <>
__device__ __forceinline__ void load_row<4, __nv_bfloat16>(const __nv_bfloat16 *p, float (&v)[4])
{
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xFFFF0000u);
    v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xFFFF0000u);
}
template <>
__device__ __forceinline__ void load_row<4, float>(const float *p, float (&v)[4])
{
    const float4 f = *reinterpret_cast<const float4 *>(p);
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
}

// Four bf16 channels of a staged row, by shared-window address (a plain shared
// load: these rows must not queue behind the warp's global traffic). Volatile so
// that it stays after the wait for the rows' copy.
__device__ __forceinline__ void lds_row4(uint32_t saddr, float (&v)[4])
{
    uint32_t x, y;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "r"(saddr));
    v[0] = __uint_as_float(x << 16); v[1] = __uint_as_float(x & 0xFFFF0000u);
    v[2] = __uint_as_float(y << 16); v[3] = __uint_as_float(y & 0xFFFF0000u);
}

template <typename TIn, int WC, int NCH, bool kSilu = true>
__device__ __forceinline__ void conv_block(const PrefillArgs &a, int b, int c0, int n, int ch0,
                                           int t0, bool staged, uint32_t raw_s, float (&out)[8][NCH],
                                           const float4 *wsm = nullptr, int wstride = 0)
{
    static_assert(NCH == 4, "staged rows are read four channels per thread");
    const int W = WC > 0 ? WC : a.W;
    constexpr int WM = WC > 0 ? WC : kMaxW;
    float w[NCH][WM];
#pragma unroll
    for (int e = 0; e < NCH; ++e) {
        if (WC == 4) {
            const float4 f = wsm != nullptr ? wsm[e * wstride]
                                            : __ldg(reinterpret_cast<const float4 *>(a.conv_w + (size_t)(ch0 + e) * 4));
            w[e][0] = f.x; w[e][1] = f.y; w[e][2] = f.z; w[e][3 % WM] = f.w;
        } else {
#pragma unroll
            for (int tau = 0; tau < WM; ++tau)
                w[e][tau] = tau < W ? __ldg(a.conv_w + (size_t)(ch0 + e) * W + tau) : 0.0f;
        }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int e = 0; e < NCH; ++e)
            out[t][e] = 0.0f;
    const int s0 = c0 + t0 - (W - 1);              // stream index of row 0 of the window
    const bool inside = s0 >= 0 && s0 + 7 + W - 1 < a.T;   // no history, no tail rows
    const TIn *xb = static_cast<const TIn *>(a.x) + ((int64_t)b * a.T + s0) * a.x_stride + ch0;
    const uint32_t rb = raw_s + (uint32_t)(t0 * kD + (ch0 & (kD - 1))) * 2u;
    const float *hist = a.conv_state + ((size_t)b * a.conv_dim + ch0) * (W - 1);
    // row rr of the window feeds tap rr - t of token t
    auto add_row = [&](int rr, const float (&v)[NCH]) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int tau = rr - t;
            if (tau >= 0 && tau < WM && (WC > 0 || tau < W)) {
#pragma unroll
                for (int e = 0; e < NCH; ++e)
                    out[t][e] = __fmaf_rn(v[e], w[e][tau], out[t][e]);
            }
        }
    };
    if (WC > 0 && staged && inside) {
        // every row of the window is a staged row: no branch between the loads and the sums
#pragma unroll
        for (int rr = 0; rr < 7 + WM; ++rr) {
            float v[NCH];
            lds_row4(rb + (uint32_t)(rr * kD * 2), v);
            add_row(rr, v);
        }
    } else {
#pragma unroll
        for (int rr = 0; rr < 7 + WM; ++rr) {
            if (WC == 0 && rr >= 7 + W)
                break;
            float v[NCH];
            const int s = s0 + rr;
            if (s >= 0 && s < a.T) {
                if (staged)
                    lds_row4(rb + (uint32_t)(rr * kD * 2), v);
                else
                    load_row<NCH, TIn>(xb + (int64_t)rr * a.x_stride, v);
            } else if (s < 0) {
#pragma unroll
                for (int e = 0; e < NCH; ++e)
                    v[e] = hist[(size_t)e * (W - 1) + (W - 1 + s)];
            } else {
#pragma unroll
                for (int e = 0; e < NCH; ++e)
                    v[e] = 0.0f;
            }
            add_row(rr, v);
        }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const bool live = t0 + t < n;
#pragma unroll
        for (int e = 0; e < NCH; ++e)
            out[t][e] = live ? (kSilu ? silu_f(out[t][e]) : out[t][e]) : 0.0f;
    }
}

// L2 normalisation of 8 token rows whose 128 channels are spread NCH per lane
// over 128 / NCH consecutive lanes ("ssm_mamba.rs" conv1d_update_l2norm;
// x / sqrt(sum x^2 + eps) as in "scr_state.hpp").
template <int NCH>
__device__ __forceinline__ void l2_rows(float (&v)[8][NCH], float eps, float post)
{
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        float ss = __fmul_rn(v[t][0], v[t][0]);
#pragma unroll
        for (int e = 1; e < NCH; ++e)
            ss = __fmaf_rn(v[t][e], v[t][e], ss);
#pragma unroll
        for (int m = (kD / NCH) / 2; m >= 1; m >>= 1)
            ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, m));
        const float inv = __fmul_rn(rsqrtf(__fadd_rn(ss, eps)), post);
#pragma unroll
        for (int e = 0; e < NCH; ++e)
            v[t][e] = __fmul_rn(v[t][e], inv);
    }
}

// Store 8 token rows x NCH channels (channels NCH*g .. of the head) as the two
// fp16 parts of a 128-byte-swizzled K-major tile with `rows` rows.
template <int NCH>
__device__ __forceinline__ void store_rows_split(uint8_t *hi, uint8_t *lo, int row0, int rows, int g,
                                                 const float (&v)[8][NCH])
{
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        uint32_t h[NCH / 2], l[NCH / 2];
#pragma unroll
        for (int e = 0; e < NCH / 2; ++e)
            split_pair(v[t][2 * e], v[t][2 * e + 1], h[e], l[e]);
        const uint32_t off = tc::sw128_offset(row0 + t, NCH * g, rows);
        if constexpr (NCH == 8) {
            *reinterpret_cast<uint4 *>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4 *>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
        } else {
            *reinterpret_cast<uint2 *>(hi + off) = make_uint2(h[0], h[1]);
            *reinterpret_cast<uint2 *>(lo + off) = make_uint2(l[0], l[1]);
        }
    }
}

// One tensor copy of a chunk's rows of a 128-channel head (no arrive: the caller
// sets the barrier's expected bytes once for all copies of a chunk).
__device__ __forceinline__ void rows_copy(const CUtensorMap *map, uint32_t dst, uint32_t mbar,
                                          int ch, int row, int b)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4}], [%5];"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(ch), "r"(row), "r"(b),
                    "r"(mbar)
                 : "memory");
}

// staged rows of one 128-channel head: (63 + W) rows of 128 bf16, padded to 1 KB
constexpr uint32_t kRawBox = ((kC + kMaxW - 1) * kD * 2 + 1023) / 1024 * 1024;

// ================================================================== pass 1
namespace p1 {
constexpr int kThreads = 256;
constexpr uint32_t RAWQ = 0, RAWK = kRawBox;       // staged Q and K rows of the QK head
constexpr uint32_t QK = 2 * kRawBox;               // [Q; K] two fp16 parts, [128 t'][128 i] sw128
constexpr uint32_t QK_LO = QK + 32768;
constexpr uint32_t AM = QK;                        // after G: A of two heads, fp32 [64][64]
constexpr uint32_t TB = QK + 32768;                // after G: T of two heads, fp32 [64][64]
constexpr uint32_t GATES = QK + 65536;             // two Gates
constexpr uint32_t CF = GATES + 2 * sizeof(Gates);   // two block-reference decay tables, [3][64]
constexpr uint32_t MBAR = CF + 2 * 3 * 64 * 4;
constexpr uint32_t SLOT = MBAR + 16;
constexpr uint32_t BYTES = SLOT + 16 + 1024;      // + alignment slack
static_assert(QK % 1024 == 0, "swizzled tiles on 1 KB boundaries");
}  // namespace p1

// A[t][s] and T[i][j] (fp32, 64 floats per row), float4 chunks XOR-swizzled by the row
__device__ __forceinline__ int a_idx(int t, int s) { return t * kC + ((((s >> 2) ^ (t & 15))) << 2) + (s & 3); }

// Warp-level 16 x 16 block products for the chunk's (I + A)^-1 (blocks too small for the
// CTA-wide tcgen05 products): D += A B with A 16 x 16 and B 16 x 8, fp16 operands, fp32
// accumulation; g = lane / 4 and q = lane % 4 index the PTX fragment layouts.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The 16 x 16 block at (r0, c0) of an a_idx-laid fp32 matrix as the A operand (two fp16 parts)
__device__ __forceinline__ void blk_a(const float *M, int r0, int c0, int lane, uint32_t (&hi)[4], uint32_t (&lo)[4])
{
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = r0 + g + 8 * (i & 1), col = c0 + 2 * q + 8 * (i >> 1);
        const float2 v = *reinterpret_cast<const float2 *>(M + a_idx(row, col));
        split_pair(v.x, v.y, hi[i], lo[i]);
    }
}
// The 16 x 8 block at (r0, c0) as the B operand (B[k][n] = M[r0 + k][c0 + n]), two fp16 parts
__device__ __forceinline__ void blk_b(const float *M, int r0, int c0, int lane, uint32_t (&hi)[2], uint32_t (&lo)[2])
{
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int row = r0 + 2 * q + 8 * i;
        split_pair(M[a_idx(row, c0 + g)], M[a_idx(row + 1, c0 + g)], hi[i], lo[i]);
    }
}
// D += A B with both operands in two fp16 parts (the product of the low parts is dropped)
__device__ __forceinline__ void mma_16816_x3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                             const uint32_t (&bh)[2], const uint32_t (&bl)[2])
{
    mma_16816(d, ah, bh[0], bh[1]);
    mma_16816(d, ah, bl[0], bl[1]);
    mma_16816(d, al, bh[0], bh[1]);
}
// A 16 x 16 accumulator (two 16 x 8 halves), times s, into the block at (r0, c0)
__device__ __forceinline__ void blk_store(float *M, int r0, int c0, int lane, const float (&d)[2][4], float s)
{
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 2; ++i)
            *reinterpret_cast<float2 *>(M + a_idx(r0 + g + 8 * i, c0 + 8 * h + 2 * q)) =
                make_float2(__fmul_rn(d[h][2 * i], s), __fmul_rn(d[h][2 * i + 1], s));
}

// One chunk's image in the workspace: T = (I + A)^-1 then P, each as two fp16
// parts of a [64][64] K-major core-matrix tile (8 KB per part), then the gates.
constexpr uint32_t kImgP = 16384, kImgGates = 32768;
static_assert(kImgGates + sizeof(Gates) <= kPrefillChunkImage, "chunk image layout");
__device__ __forceinline__ uint8_t *chunk_image(const PrefillArgs &a, int b, int h, int c)
{
    return a.ws + (((size_t)b * a.Hv + h) * a.n_chunks + c) * kPrefillChunkImage;
}

// The chunk's normalised Q rows then K rows of QK head hk (scaled by 16), each
// as two fp16 parts (16 KB each) of a [64 t][128 i] 128-byte-swizzled K-major
// tile: the chain pass copies them into shared memory as they are.
constexpr uint32_t kQKPart = 16384, kQKRows = 2 * kQKPart;
__device__ __forceinline__ uint8_t *qk_image(const PrefillArgs &a, int b, int hk, int c)
{
    return a.ws + (size_t)a.B * a.Hv * a.n_chunks * kPrefillChunkImage +
           (((size_t)b * a.Hq + hk) * a.n_chunks + c) * kPrefillQKImage;
}

template <typename TIn, int WC>
__global__ void __launch_bounds__(p1::kThreads, 2) prefill_ut_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                PrefillArgs a, int staged)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int r = a.Hv / a.Hq;
    const int W = WC > 0 ? WC : a.W;
    const int c0 = c * kC, n = min(kC, a.T - c0);
    GDN_CHECK(g_device_error, c < a.n_chunks && hk < a.Hq && b < a.B && n >= 1 && c0 + n <= a.T &&
                                  qk_image(a, b, hk, c) + kPrefillQKImage <= a.ws + a.ws_bytes &&
                                  chunk_image(a, b, hk * r + r - 1, c) + kPrefillChunkImage <= a.ws + a.ws_bytes);
    const uint32_t sbase = tc::smem_addr(smem);
    const uint32_t mb_raw = sbase + p1::MBAR, mb_mma = sbase + p1::MBAR + 8;
    Gates *gates = reinterpret_cast<Gates *>(smem + p1::GATES);
    float *cft = reinterpret_cast<float *>(smem + p1::CF);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + p1::SLOT + 4);
    const uint64_t lim = a.wait_ns;

    if (tid == 0) {
        tc::mbar_init(mb_raw, 1);
        tc::mbar_init(mb_mma, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (staged) {
            tc::mbar_expect_tx(mb_raw, 2u * (uint32_t)(kC + W - 1) * kD * 2);
            rows_copy(&xmap, sbase + p1::RAWQ, mb_raw, hk * kD, c0 - (W - 1), b);
            rows_copy(&xmap, sbase + p1::RAWK, mb_raw, a.Hq * kD + hk * kD, c0 - (W - 1), b);
        } else {
            tc::mbar_arrive(mb_raw);
        }
    }
    if (warp == 0)
        tc::tmem_alloc(sbase + p1::SLOT, 64);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + p1::SLOT);

    // the first head pair's gates, while the rows are in flight (they read nothing staged)
    if (warp < 2 && warp < r)
        chunk_gates<TIn>(a, b, hk * r + warp, c0, n, gates + warp, cft + warp * 192);

    // Q and K rows: conv + SiLU + L2 (warp = 8-token block, lane = 4 channels) -> [Q; K] tile
    bool ok = tc::mbar_wait_ns(mb_raw, 0, lim, abort);
    if (ok) {
#pragma unroll 1
        for (int part = 0; part < 2; ++part) {
            float v[8][4];
            conv_block<TIn, WC, 4>(a, b, c0, n, (part ? a.Hq * kD : 0) + hk * kD + 4 * lane, 8 * warp,
                                   staged != 0, sbase + (part ? p1::RAWK : p1::RAWQ), v);
            l2_rows<4>(v, a.l2_eps, kQK);
            store_rows_split<4>(smem + p1::QK, smem + p1::QK_LO, part * kC + 8 * warp, 2 * kC, lane, v);
        }
    } else {
        atomicOr(const_cast<int *>(abort), (int)kErrUT);
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    ok = *abort == 0;

    // G = [Q; K] K^T: rows 0..63 give Q K^T (for P), rows 64..127 K K^T (for A)
    const bool mma_issued = ok;
    if (ok && tid == 0) {
        // the chain pass's Q and K operands: rows 0..63 / 64..127 of each 8 KB column
        // block of the tile are the two column blocks of a 64-row tile (the swizzle
        // depends on the row within its 8-row group only)
        uint8_t *img = qk_image(a, b, hk, c);
#pragma unroll 1
        for (int i = 0; i < 8; ++i) {
            const int p = i >> 2, s = (i >> 1) & 1, cb = i & 1;
            tc::bulk_copy_s2g(img + p * kQKRows + s * kQKPart + cb * 8192,
                              sbase + p1::QK + s * 32768 + cb * 16384 + p * 8192, 8192);
        }
        tc::bulk_commit();
        const uint32_t id = tc::idesc_f16(128, 64);
#pragma unroll 1
        for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t kq = (kk >> 2) * (2 * kC * 128) + (kk & 3) * 32;
            const uint64_t a1 = tc::sdesc_sw128(sbase + p1::QK + kq);
            const uint64_t a2 = tc::sdesc_sw128(sbase + p1::QK_LO + kq);
            const uint64_t b1 = tc::sdesc_sw128(sbase + p1::QK + kC * 128 + kq);
            const uint64_t b2 = tc::sdesc_sw128(sbase + p1::QK_LO + kC * 128 + kq);
            tc::mma_f16(tmem, a1, b1, id, kk > 0);
            tc::mma_f16(tmem, a1, b2, id, 1);
            tc::mma_f16(tmem, a2, b1, id, 1);
        }
        tc::mma_commit(mb_mma);
    }
    if (ok && !tc::mbar_wait_ns(mb_mma, 0, lim, abort)) {
        atomicOr(const_cast<int *>(abort), (int)kErrUT);
        ok = false;
    }
    if (mma_issued && tid == 0)
        tc::bulk_wait_read();    // the tile's region is overwritten below
    tc::fence_after_sync();
    __syncthreads();
    ok = *abort == 0;

    float *Am = reinterpret_cast<float *>(smem + p1::AM);
    float *Tb = reinterpret_cast<float *>(smem + p1::TB);
    const int q4 = warp & 3, hsel = warp >> 2;
    const uint32_t lane_q = (uint32_t)(32 * q4) << 16;

#pragma unroll 1
    for (int hp = 0; ok && hp < r; hp += 2) {
        if (hp > 0 && warp < 2 && hp + warp < r)
            chunk_gates<TIn>(a, b, hk * r + hp + warp, c0, n, gates + warp, cft + warp * 192);
        tc::fence_smem_to_async();
        __syncthreads();
        if (tid == 0) {      // the gates travel with the chunk's image
#pragma unroll 1
            for (int u = 0; u < 2 && hp + u < r; ++u)
                tc::bulk_copy_s2g(chunk_image(a, b, hk * r + hp + u, c) + kImgGates,
                                  sbase + p1::GATES + u * (uint32_t)sizeof(Gates), sizeof(Gates));
            tc::bulk_commit();
        }
        const int hh = hp + hsel;
        // ---- P (TMEM lanes 0..63, the Q rows: warps 0, 1, 4, 5) and A (lanes 64..127, the
        //      K rows: warps 2, 3, 6, 7) of the pair's two heads, one token row per thread
        if (hh < r) {
            const Gates *G = gates + hsel;
            const int t = 32 * (q4 & 1) + lane;
            const bool is_a = q4 >= 2;
            const float gt = G->gh[t], gtl = G->gl[t];
            const float rowf = is_a ? __fmul_rn(G->beta[t], kInvQK2) : kInvQK2;
            uint8_t *pimg = chunk_image(a, b, hk * r + hh, c) + kImgP;
            float *A = Am + hsel * kC * kC;
            // Below the 16-token diagonal blocks the decay factors split at the start of the
            // row's block, exp(Gam_t - Gam_s) = exp(Gam_t - Gam_16I) exp(Gam_16I - Gam_s),
            // both factors at most 1; inside them each factor is formed on its own.
            const int I = t >> 4, Iw = (32 * (q4 & 1)) >> 4;  // the row's block, the warp's first
            const float rf = exp_diff_fast(gt, gtl, G->gh[16 * I], G->gl[16 * I]);
            const float *cfI = cft + hsel * 192 + 64 * (I > 0 ? I - 1 : 0);
            // one 16-column block of the row: A to shared memory, P as its two-part image
            auto store_blk = [&](int s0, const float (&o)[16]) {
                if (is_a) {
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq)
                        *reinterpret_cast<float4 *>(A + a_idx(t, s0 + 4 * qq)) =
                            make_float4(o[4 * qq], o[4 * qq + 1], o[4 * qq + 2], o[4 * qq + 3]);
                } else {
#pragma unroll
                    for (int hq = 0; hq < 2; ++hq) {
                        uint4 hi, lo;
                        split_pair(o[8 * hq], o[8 * hq + 1], hi.x, lo.x);
                        split_pair(o[8 * hq + 2], o[8 * hq + 3], hi.y, lo.y);
                        split_pair(o[8 * hq + 4], o[8 * hq + 5], hi.z, lo.z);
                        split_pair(o[8 * hq + 6], o[8 * hq + 7], hi.w, lo.w);
                        const uint32_t off = tc::km_offset(t, s0 + 8 * hq, kC);
                        *reinterpret_cast<uint4 *>(pimg + off) = hi;
                        *reinterpret_cast<uint4 *>(pimg + 8192 + off) = lo;
                    }
                }
            };
            // column blocks wholly below the warp's rows' diagonal blocks, or wholly above
#pragma unroll 1
            for (int J = 0; J < 4; ++J) {
                if (J == Iw || J == Iw + 1)                   // warp-uniform
                    continue;
                float o[16];
                if (J > Iw + 1) {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        o[e] = 0.0f;
                } else {
                    float gv[16];
                    tc::tmem_ld16(tmem + lane_q + 16 * J, gv);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        o[e] = t < n ? __fmul_rn(__fmul_rn(rowf, __fmul_rn(rf, cfI[16 * J + e])), gv[e]) : 0.0f;
                }
                store_blk(16 * J, o);
            }
            // the warp's own two row blocks: each lane forms the decay factors of its own
            // diagonal block only; of the other block, lanes of the second row block need
            // the part below their diagonal, lanes of the first the zero part above it
            {
                float ga[16], gb[16];
                tc::tmem_ld16(tmem + lane_q + 16 * Iw, ga);
                tc::tmem_ld16(tmem + lane_q + 16 * (Iw + 1), gb);
                const bool first = I == Iw;
                float od[16], oo[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int s = 16 * I + e;
                    const bool keep = t < n && (is_a ? s < t : s <= t);
                    od[e] = keep ? __fmul_rn(__fmul_rn(rowf, exp_diff_fast(gt, gtl, G->gh[s], G->gl[s])),
                                             first ? ga[e] : gb[e])
                                 : 0.0f;
                    oo[e] = !first && t < n
                                ? __fmul_rn(__fmul_rn(rowf, __fmul_rn(rf, cfI[16 * Iw + e])), ga[e])
                                : 0.0f;
                }
                store_blk(16 * I, od);
                store_blk(16 * (first ? Iw + 1 : Iw), oo);
            }
        }
        __syncthreads();
        // ---- T = (I + A)^-1 in 16-token blocks. Warp I of a head inverts the diagonal block
        //      T_II = (I + A_II)^-1 by forward substitution (lane j: column j) and clears the
        //      blocks right of it; then warp J walks block column J on its own:
        //      T_IJ = -T_II sum_{K=J}^{I-1} A_IK T_KJ for I = J+1 .. 3.
        const int hs = tid >> 7, wb = (tid >> 5) & 3;
        float *Tc = Tb + hs * kC * kC;
        const float *Ah = Am + hs * kC * kC;
        if (hp + hs < r) {
            const int r0 = 16 * wb;
            if (lane < 16) {
                float x[16];
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    x[q] = q == lane ? 1.0f : 0.0f;
                // four columns of the block at a time: rows q > e4 of A_II[:, e4 .. e4+3] as
                // float4 loads issued together, then four substitution steps from registers
#pragma unroll
                for (int e4 = 0; e4 < 16; e4 += 4) {
                    float4 ac[16];
#pragma unroll
                    for (int q = e4 + 1; q < 16; ++q)
                        ac[q] = *reinterpret_cast<const float4 *>(Ah + a_idx(r0 + q, r0 + e4));
#pragma unroll
                    for (int e = e4; e < e4 + 4 && e < 15; ++e)
#pragma unroll
                        for (int q = e + 1; q < 16; ++q) {
                            const float av = e == e4 ? ac[q].x : e == e4 + 1 ? ac[q].y : e == e4 + 2 ? ac[q].z : ac[q].w;
                            x[q] = __fmaf_rn(-av, x[e], x[q]);
                        }
                }
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    Tc[a_idx(r0 + q, r0 + lane)] = x[q];
            } else {
                const int w4 = 4 * (3 - wb);                    // float4 slots per row right of it
                for (int i = lane - 16; i < 16 * w4; i += 16)
                    *reinterpret_cast<float4 *>(Tc + a_idx(r0 + i / w4, 16 * (wb + 1) + 4 * (i % w4))) =
                        make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        }
        __syncthreads();
        if (hp + hs < r) {
            const int J = wb;
#pragma unroll 1
            for (int I = J + 1; I < 4; ++I) {
                float d[2][4] = {};
#pragma unroll 1
                for (int K = J; K < I; ++K) {
                    uint32_t ah[4], al[4];
                    blk_a(Ah, 16 * I, 16 * K, lane, ah, al);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t bh[2], bl[2];
                        blk_b(Tc, 16 * K, 16 * J + 8 * h, lane, bh, bl);
                        mma_16816_x3(d[h], ah, al, bh, bl);
                    }
                }
                // the sum goes through T_IJ's place to become the B operand of T_II (.)
                blk_store(Tc, 16 * I, 16 * J, lane, d, 1.0f);
                __syncwarp();
                uint32_t ah[4], al[4];
                blk_a(Tc, 16 * I, 16 * I, lane, ah, al);
                float e[2][4] = {};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t bh[2], bl[2];
                    blk_b(Tc, 16 * I, 16 * J + 8 * h, lane, bh, bl);
                    mma_16816_x3(e[h], ah, al, bh, bl);
                }
                __syncwarp();
                blk_store(Tc, 16 * I, 16 * J, lane, e, -1.0f);
                __syncwarp();
            }
        }
        __syncthreads();
        // ---- T -> two-part fp16 K-major image ([t][s], 8x8 core matrices) in the workspace
#pragma unroll 1
        for (int u = 0; u < 2; ++u) {
            if (hp + u >= r)
                break;
            const float *Tc = Tb + u * kC * kC;
            uint8_t *img = chunk_image(a, b, hk * r + hp + u, c);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int p = tid + 256 * k;                       // 16-byte chunk of a part
                const int t = ((p >> 6) << 3) | (p & 7), s8 = (p >> 3) & 7;
                const float4 f0 = *reinterpret_cast<const float4 *>(Tc + a_idx(t, 8 * s8));
                const float4 f1 = *reinterpret_cast<const float4 *>(Tc + a_idx(t, 8 * s8 + 4));
                uint4 hi, lo;
                split_pair(f0.x, f0.y, hi.x, lo.x);
                split_pair(f0.z, f0.w, hi.y, lo.y);
                split_pair(f1.x, f1.y, hi.z, lo.z);
                split_pair(f1.z, f1.w, hi.w, lo.w);
                *reinterpret_cast<uint4 *>(img + 16 * p) = hi;
                *reinterpret_cast<uint4 *>(img + 8192 + 16 * p) = lo;
            }
        }
        if (tid == 0)
            tc::bulk_wait_read();    // the gates' buffers are rewritten by the next pair
        __syncthreads();
    }

    if (tid == 0)
        tc::bulk_wait();             // the workspace copies are complete before the CTA ends
    if (tid == 0 && *abort) {
        atomicOr(&g_device_error, *abort);
        // the staged-row copy and the product may still be in flight
        if (!tc::mbar_wait_ns(mb_raw, 0, lim) || (mma_issued && !tc::mbar_wait_ns(mb_mma, 0, lim)))
            atomicOr(&g_device_error, (int)kErrDrain);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0)
        tc::tmem_dealloc(tmem, 64);
}

// ================================================================== pass 2
namespace p2 {
// warps 0-15: epilogue (four per TMEM lane quarter); warp 16: the products; warp 17: the
// workspace copies; warps 18-25: the V conv and the gated norm (8 tokens each). 26 warps
// of at most 72 registers fit the SM's 65536 registers with one CTA per SM. Each epilogue
// warp handles kEpiTok tokens of the chunk and kEpiCols columns of the state master for its
// 32 value rows. (Two epilogue warps per quarter, 32 tokens and 64 columns each, measured
// 1.280 against 1.257-1.275 ms for the 4 x 8192 prefill on one box, 1.358 against
// 1.281-1.290 ms on another; four conv warps with the sixteen took 2.31 ms.)
constexpr int kEpiWarps = 16, kEpiQ = kEpiWarps / 4;
constexpr int kEpiTok = kC / kEpiQ, kEpiCols = kD / kEpiQ;
static_assert(kEpiWarps == 8 || kEpiWarps == 16, "two or four epilogue warps per lane quarter");
constexpr int kIssuerWarp = kEpiWarps, kCopyWarp = kEpiWarps + 1, kConvWarp0 = kEpiWarps + 2;
constexpr int kConvWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps, kConvTok = kC / kConvWarps;
constexpr int kThreads = 32 * (kConvWarp0 + kConvWarps);
constexpr uint32_t QB = 0;                        // Q rows of the chunk: two parts, [64 t][128 i] sw128
constexpr uint32_t KB = 32768;                    // K rows, two buffers (even and odd chunks)
constexpr uint32_t VF = 98304;                    // V^T fp32 footprint [128 j][64 t], before SiLU
constexpr uint32_t TT = 131072;                   // T image of the current chunk (16 KB)
constexpr uint32_t PP = 147456;                   // P image of the current chunk (16 KB)
constexpr uint32_t OS = 163840;                   // O staging, fp32 [64 t][128 j]
constexpr uint32_t RAW = 196608;                  // staged rows of the V head
constexpr uint32_t GATES = RAW + kRawBox;         // two Gates buffers (even and odd chunks)
constexpr uint32_t MBAR = GATES + 2 * sizeof(Gates);
constexpr uint32_t SLOT = MBAR + 24 * 8;          // TMEM base, abort word
constexpr uint32_t CONVW = SLOT + 16;             // 4-tap conv weights of the V head
constexpr uint32_t BYTES = CONVW + kD * 16 + 1024;
static_assert(BYTES <= 232448, "shared memory budget");
static_assert(RAW % 1024 == 0 && KB % 1024 == 0, "tiles on 1 KB boundaries");
// barriers: copies (expected bytes), products (commits), and role hand-offs
enum { B_Q, B_K0, B_K1, B_T, B_G, B_P, B_RAW, B_M1, B_M1QA, B_M1Q, B_M2, B_M3, B_PU,
       B_RAWFREE, B_V, B_OSFREE,       // the conv threads arrive
       B_ST, B_X, B_U, B_UP, B_OR, B_OS,   // 256 epilogue threads arrive
       B_N };
static_assert(B_N <= 24, "barrier slots");
// TMEM columns: TS the fp32 state master (S^T), D1 = [(Q S_0)^T | (K S_0)^T], R1 the
// S_0^T operand (two fp16 parts; the low part's columns later hold U'^T), XU the
// X^T, then U^T operand (two parts), D2 = U^T, then (P U)^T
constexpr uint32_t TS = 0, D1 = 128, R1 = 256, XU = 384, D2 = 448;
}  // namespace p2

// fp32 V^T footprint: float4 q (tokens 4q .. 4q+3) of value row j; the 16-byte
// slot is XOR-ed with the row group so that both the conv's stores (rows 4
// apart) and a warp's row reads land on distinct bank groups.
__device__ __forceinline__ uint32_t foot_off(int j, int q)
{
    return (uint32_t)(p2::VF + (q >= 8 ? 16384 : 0) + (j >> 3) * 1024 + (q & 7) * 128 +
                      (((j & 7) ^ ((j >> 3) & 7)) << 4));
}

__device__ __forceinline__ void pack_split16(const float (&v)[16], uint32_t (&hi)[8], uint32_t (&lo)[8])
{
#pragma unroll
    for (int e = 0; e < 8; ++e)
        split_pair(v[2 * e], v[2 * e + 1], hi[e], lo[e]);
}

__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t (&v)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                    "r"(v[6]), "r"(v[7]));
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

// Four gate values of a norm row held as loaded (raw bits), so that a load issued
// early is waited for only where the values are used.
template <typename T> struct ZRaw;
template <> struct ZRaw<__nv_bfloat16> {
    uint2 u;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = __ldcs(reinterpret_cast<const uint2 *>(p)); }
    __device__ __forceinline__ void get(float (&v)[4]) const
    {
        v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xFFFF0000u);
        v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xFFFF0000u);
    }
};
template <> struct ZRaw<float> {
    float4 f;
    __device__ __forceinline__ void load(const float *p) { f = __ldcs(reinterpret_cast<const float4 *>(p)); }
    __device__ __forceinline__ void get(float (&v)[4]) const { v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w; }
};

template <typename TIn, int WC>
__global__ void __launch_bounds__(p2::kThreads, 1) prefill_chain_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                      PrefillArgs a, int staged, int zvec)
{
    using namespace p2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x, b = blockIdx.y;
    const int r = a.Hv / a.Hq, hk = h / r;
    const int W = WC > 0 ? WC : a.W;
    const int nch = a.n_chunks;
    GDN_CHECK(g_device_error, h < a.Hv && b < a.B && hk < a.Hq && (nch - 1) * kC < a.T &&
                                  qk_image(a, b, hk, nch - 1) + kPrefillQKImage <= a.ws + a.ws_bytes &&
                                  chunk_image(a, b, h, nch - 1) + kPrefillChunkImage <= a.ws + a.ws_bytes);
    const uint32_t sbase = tc::smem_addr(smem);
    const uint32_t mb = sbase + MBAR;
    auto bar = [&](int i) { return mb + 8u * (uint32_t)i; };
    volatile int *abort = reinterpret_cast<volatile int *>(smem + SLOT + 4);
    Gates *gbuf = reinterpret_cast<Gates *>(smem + GATES);
    float *Os = reinterpret_cast<float *>(smem + OS);
    const uint64_t lim = a.wait_ns;

    if (tid == 0) {
        for (int i = 0; i < B_N; ++i)
            tc::mbar_init(bar(i), i < B_RAWFREE ? 1 : i < B_ST ? kConvThreads : 32 * kEpiWarps);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0)
        tc::tmem_alloc(sbase + SLOT, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + SLOT);

    // a bounded wait that, on giving up, tells the other roles to stop
    auto waitb = [&](int i, uint32_t parity, uint64_t limit) -> bool {
        if (tc::mbar_wait_ns(bar(i), parity, limit, abort))
            return true;
        atomicOr(const_cast<int *>(abort), (int)kErrChain);
        return false;
    };

    if (warp >= kConvWarp0) {
        // ============================================ conv warps: chunk c's V rows, chunk c-1's norm
        const int cw = warp - kConvWarp0;
        const bool raw_issuer = tid == 32 * kConvWarp0;
        int raw_last = -1;
        auto issue_raw = [&](int cc) {
            tc::mbar_expect_tx(bar(B_RAW), (uint32_t)(kC + W - 1) * kD * 2);
            rows_copy(&xmap, sbase + RAW, bar(B_RAW), 2 * a.Hq * kD + h * kD, cc * kC - (W - 1), b);
            raw_last = cc;
        };
        if (staged && raw_issuer)
            issue_raw(0);
        // V rows: 16 tokens (16 cw ..) x 4 channels (4 lane ..) per thread; 4-tap weights
        // read once, channel 4 l + e at float4 [e][l] so that a warp's reads of one e
        // are consecutive
        const int v_ch = 2 * a.Hq * kD + h * kD + 4 * lane;
        const float4 *v_w = nullptr;
        if (WC == 4) {
            float4 *tab = reinterpret_cast<float4 *>(smem + CONVW);
            for (int i = tid - 32 * kConvWarp0; i < kD; i += kConvThreads)
                tab[i] = __ldg(reinterpret_cast<const float4 *>(a.conv_w + (size_t)(v_ch - 4 * lane + 4 * (i & 31) + (i >> 5)) * 4));
            asm volatile("bar.sync 1, %0;" :: "n"(kConvThreads) : "memory");   // the conv warps only
            v_w = tab + lane;
        }
        // gated-norm mapping: warp cw handles tokens cw, cw + 4, ...; lane holds channels 4 lane .. +3
        const float4 nw4 = __ldg(reinterpret_cast<const float4 *>(a.norm_w) + lane);
        // bf16 gate rows are held in registers from their load to the norm (2 per row);
        // float rows are loaded where they are used
        constexpr bool kZPre = sizeof(TIn) == 2;
        ZRaw<TIn> zpre[kZPre ? kConvTok : 1];
        auto z_rows = [&](int cc) {
            return static_cast<const TIn *>(a.z) + ((int64_t)b * a.T + (int64_t)cc * kC) * a.z_stride +
                   (int64_t)h * kD + 4 * lane;
        };
        // this warp's gate rows of chunk cc: brought into L2 early (a prefetch holds no
        // register, so nothing waits on it), loaded into registers once the V rows are out
        auto z_prefetch = [&](int cc) {
            const int n = min(kC, a.T - cc * kC);
            const TIn *zb = z_rows(cc);
#pragma unroll
            for (int i = 0; i < kConvTok; ++i)
                if (cw + kConvWarps * i < n)
                    asm volatile("prefetch.global.L2 [%0];" :: "l"(zb + (int64_t)(cw + kConvWarps * i) * a.z_stride));
        };
        auto z_fetch = [&](int cc) {
            if (!zvec || !kZPre)
                return;
            const int n = min(kC, a.T - cc * kC);
            const TIn *zb = z_rows(cc);
#pragma unroll
            for (int i = 0; i < kConvTok; ++i)
                if (cw + kConvWarps * i < n)
                    zpre[kZPre ? i : 0].load(zb + (int64_t)(cw + kConvWarps * i) * a.z_stride);
        };
        // ---- gated RMSNorm ("fm_kernel_ssm.h", "Gated RMSNorm") of chunk cc's staged rows,
        //      four rows at a time with no branch between them, so that their latencies
        //      overlap; rows at or past the end of the call are computed but not stored
        auto norm = [&](int cc) {
            const int c0 = cc * kC, n = min(kC, a.T - c0);
            const TIn *zb = z_rows(cc);
#pragma unroll
            for (int g = 0; g < kConvTok; g += 4) {
                float4 y[4];
                float ss[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int t = cw + kConvWarps * (g + r);
                    y[r] = *reinterpret_cast<const float4 *>(Os + t * kD + 4 * lane);
                    ss[r] = __fmul_rn(y[r].x, y[r].x);
                    ss[r] = __fmaf_rn(y[r].y, y[r].y, ss[r]);
                    ss[r] = __fmaf_rn(y[r].z, y[r].z, ss[r]);
                    ss[r] = __fmaf_rn(y[r].w, y[r].w, ss[r]);
                }
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        ss[r] = __fadd_rn(ss[r], __shfl_xor_sync(0xffffffffu, ss[r], m));
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int t = cw + kConvWarps * (g + r);
                    const bool live = t < n;
                    const float inv = rsqrtf(__fadd_rn(__fmul_rn(ss[r], 1.0f / kD), a.rms_eps));
                    float zv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    const TIn *zr = zb + (int64_t)t * a.z_stride;
                    if (zvec && kZPre) {
                        zpre[kZPre ? g + r : 0].get(zv);
                    } else if (live) {
                        if (zvec) {
                            load_row<4, TIn>(zr, zv);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                zv[e] = load_act<TIn>(zr + e);
                        }
                    }
                    float4 o;
                    o.x = gated_out(y[r].x, inv, nw4.x, zv[0]);
                    o.y = gated_out(y[r].y, inv, nw4.y, zv[1]);
                    o.z = gated_out(y[r].z, inv, nw4.z, zv[2]);
                    o.w = gated_out(y[r].w, inv, nw4.w, zv[3]);
                    const int64_t row = (int64_t)b * a.T + c0 + t;
                    if (live)
                        *reinterpret_cast<float4 *>(a.out + (row * a.Hv + h) * kD + 4 * lane) = o;
                }
            }
        };
        bool ok = true;
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
            const int c0 = c * kC, n = min(kC, a.T - c0);
            if (c > 0)
                z_prefetch(c - 1);
            if (staged && !(ok = waitb(B_RAW, c & 1, lim)))
                break;
            // V^T of chunk c before its SiLU (the epilogue applies it as it reads V for X,
            // which moves that work off these warps), 8 tokens at a time, written once
            // chunk c-1's X has read the footprint
            bool x_seen = c == 0;
#pragma unroll
            for (int k = 0; k < kConvTok / 8; ++k) {
                float v[8][4];
                conv_block<TIn, WC, 4, false>(a, b, c0, n, v_ch, kConvTok * cw + 8 * k, staged != 0, sbase + RAW,
                                       v, v_w, 32);
                if (!x_seen && !(ok = x_seen = waitb(B_X, (c - 1) & 1, lim)))
                    break;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = 4 * lane + e;
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        *reinterpret_cast<float4 *>(smem + foot_off(j, kConvTok / 4 * cw + 2 * k + q)) =
                            make_float4(v[4 * q][e], v[4 * q + 1][e], v[4 * q + 2][e], v[4 * q + 3][e]);
                }
            }
            if (!ok)
                break;
            tc::mbar_arrive(bar(B_V));
            if (staged && c + 1 < nch) {
                // the staged rows are read: the next chunk's may come in. The issuer's whole
                // warp waits, so that the warp stays converged for the work after it.
                tc::mbar_arrive(bar(B_RAWFREE));
                if (cw == 0) {
                    if ((ok = waitb(B_RAWFREE, c & 1, lim)) && raw_issuer)
                        issue_raw(c + 1);
                    __syncwarp();
                }
                if (!ok)
                    break;
            }
            // the norm of chunk c-1, whose rows the epilogue has staged
            if (c > 0) {
                z_fetch(c - 1);
                if (!(ok = waitb(B_OS, (c - 1) & 1, lim)))
                    break;
                norm(c - 1);
                tc::mbar_arrive(bar(B_OSFREE));
            }
        }
        if (ok && nch > 0) {
            z_fetch(nch - 1);
            if ((ok = waitb(B_OS, (nch - 1) & 1, lim)))
                norm(nch - 1);
        }
        // drain: the staged-row copy in flight lands before the CTA ends
        if (raw_issuer && raw_last >= 0 && !tc::mbar_wait_ns(bar(B_RAW), raw_last & 1, lim))
            atomicOr(&g_device_error, (int)kErrDrain);
    } else if (warp == kCopyWarp) {
        // ============================================ copies: the workspace images and gates
        // Lane 0 refills each shared-memory buffer from the workspace as soon as the products
        // or epilogues that read its previous contents are done, so that the issuing lane of
        // the products never waits behind a copy.
        if (lane == 0) {
            int q_last = -1, k_last0 = -1, k_last1 = -1, t_last = -1, g_last = -1, p_last = -1;
            auto issue_q = [&](int cc) {     // Q rows of chunk cc
                tc::mbar_expect_tx(bar(B_Q), kQKRows);
                tc::bulk_copy_g2s(sbase + QB, qk_image(a, b, hk, cc), kQKRows, bar(B_Q));
                q_last = cc;
            };
            auto issue_k = [&](int cc) {     // K rows of chunk cc, into the buffer of its parity
                const int kb = cc & 1;
                tc::mbar_expect_tx(bar(B_K0 + kb), kQKRows);
                tc::bulk_copy_g2s(sbase + KB + kb * kQKRows, qk_image(a, b, hk, cc) + kQKRows, kQKRows,
                                  bar(B_K0 + kb));
                (kb ? k_last1 : k_last0) = cc;
            };
            auto issue_t = [&](int cc) {     // T image of chunk cc
                tc::mbar_expect_tx(bar(B_T), 16384u);
                tc::bulk_copy_g2s(sbase + TT, chunk_image(a, b, h, cc), 16384u, bar(B_T));
                t_last = cc;
            };
            auto issue_g = [&](int cc) {     // gates of chunk cc, into the buffer of its parity
                tc::mbar_expect_tx(bar(B_G), (uint32_t)sizeof(Gates));
                tc::bulk_copy_g2s(sbase + GATES + (cc & 1) * (uint32_t)sizeof(Gates),
                                  chunk_image(a, b, h, cc) + kImgGates, (uint32_t)sizeof(Gates), bar(B_G));
                g_last = cc;
            };
            auto issue_p = [&](int cc) {     // P image of chunk cc
                tc::mbar_expect_tx(bar(B_P), 16384u);
                tc::bulk_copy_g2s(sbase + PP, chunk_image(a, b, h, cc) + kImgP, 16384u, bar(B_P));
                p_last = cc;
            };
            issue_k(0);
            if (nch > 1)
                issue_k(1);
            issue_q(0);
            issue_g(0);
            issue_t(0);
            issue_p(0);
            bool ok = true;
#pragma unroll 1
            // Each barrier waited on here cannot complete its next phase before this lane has
            // waited for the current one: that phase needs a copy this lane issues after the
            // wait (chunk c+1's gates, Q rows, T and P).
            for (int c = 0; ok && c + 1 < nch; ++c) {
                // chunk c+1's gates once every value row has read chunk c-1's (the buffer
                // of c+1's parity): the epilogue has finished chunk c-1 when it publishes X^T
                if (!(ok = waitb(B_X, c & 1, lim)))
                    break;
                issue_g(c + 1);
                // the Q rows once (Q S_0)^T has read chunk c's
                if (!(ok = waitb(B_M1Q, c & 1, lim)))
                    break;
                issue_q(c + 1);
                // chunk c's K buffer (read by K S_0 and the state update) and T (read by D2's
                // product) once the state update is done: a commit covers every earlier
                // product. K first: chunk c+2's first product waits for it, while T is needed
                // only after chunk c+1's X.
                if (!(ok = waitb(B_M3, c & 1, lim)))
                    break;
                if (c + 2 < nch)
                    issue_k(c + 2);
                issue_t(c + 1);
                // P once (P U)^T has read chunk c's
                if (!(ok = waitb(B_PU, c & 1, lim)))
                    break;
                issue_p(c + 1);
            }
            // drain: copies in flight land before the CTA releases its shared memory
            bool drained = true;
            if (q_last >= 0)
                drained &= tc::mbar_wait_ns(bar(B_Q), q_last & 1, lim);
            if (k_last0 >= 0)
                drained &= tc::mbar_wait_ns(bar(B_K0), (k_last0 >> 1) & 1, lim);
            if (k_last1 >= 0)
                drained &= tc::mbar_wait_ns(bar(B_K1), (k_last1 >> 1) & 1, lim);
            if (t_last >= 0)
                drained &= tc::mbar_wait_ns(bar(B_T), t_last & 1, lim);
            if (g_last >= 0)
                drained &= tc::mbar_wait_ns(bar(B_G), g_last & 1, lim);
            if (p_last >= 0)
                drained &= tc::mbar_wait_ns(bar(B_P), p_last & 1, lim);
            if (!drained)
                atomicOr(&g_device_error, (int)kErrDrain);
        }
        __syncwarp();
    } else if (warp == kIssuerWarp) {
        // ============================================ issuer: every product
        // Lane 0 walks the chunks, issuing each product as soon as its operands are ready and
        // its accumulator is free. Per chunk the tensor pipe, which runs products in issue
        // order, gets K S_0, part A of (Q S_0)^T, U = T X, part B of (Q S_0)^T, the state
        // update and (P U)^T: the three the next chunk waits for, with the readout's in the
        // gaps while the epilogue works.
        if (lane == 0) {
            int last_commit = -1;
            uint32_t last_phase = 0;
            auto commit = [&](int i, int c) {   // a commit tracks every product issued before it
                tc::mma_commit(bar(i));
                last_commit = i;
                last_phase = c & 1;
            };
            const uint32_t id64 = tc::idesc_f16(128, 64);
            const uint32_t id128 = tc::idesc_f16(128, 128);
            // D1[:, 64..127] = S_0^T K^T, once the K rows and S_0^T are ready
            auto issue_m1k = [&](int c) -> bool {
                const int kb = c & 1;
                // the first wait of the kernel takes its limit from first_wait_ns (a test hook)
                if (!waitb(B_K0 + kb, (c >> 1) & 1, c == 0 ? a.first_wait_ns : lim))
                    return false;
                if (!waitb(B_ST, c & 1, lim))
                    return false;
                tc::fence_after_sync();
                const uint32_t kt = sbase + KB + kb * kQKRows;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t ko = (kk >> 2) * 8192 + (kk & 3) * 32;   // column block, 16 channels
                    const uint32_t shi = tmem + R1 + 8 * kk, slo = tmem + R1 + 64 + 8 * kk;
                    const uint64_t k1 = tc::sdesc_sw128(kt + ko), k2 = tc::sdesc_sw128(kt + kQKPart + ko);
                    tc::mma_f16_ta(tmem + D1 + kC, shi, k1, id64, kk > 0);
                    tc::mma_f16_ta(tmem + D1 + kC, shi, k2, id64, 1);
                    tc::mma_f16_ta(tmem + D1 + kC, slo, k1, id64, 1);
                }
                commit(B_M1, c);
                return true;
            };
            // D1[:, 0..63] = S_0^T Q^T in two parts, so that the tensor pipe (which runs
            // products in issue order) holds no more of it before D2's product than fits
            // while the epilogue forms X. Part A, the terms of the low part of S_0^T (which
            // U'^T overwrites once D2 is done), once the Q rows are in and the previous
            // chunk's readout has read these columns:
            auto issue_m1q_lo = [&](int c) -> bool {
                if ((c > 0 && !waitb(B_OR, (c - 1) & 1, lim)) || !waitb(B_Q, c & 1, lim))
                    return false;
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t ko = (kk >> 2) * 8192 + (kk & 3) * 32;
                    const uint32_t slo = tmem + R1 + 64 + 8 * kk;
                    tc::mma_f16_ta(tmem + D1, slo, tc::sdesc_sw128(sbase + QB + ko), id64, kk > 0);
                }
                commit(B_M1QA, c);
                return true;
            };
            // part B, the terms of the high part (rewritten only after the state update),
            // issued right after D2's product
            auto issue_m1q_hi = [&](int c) {
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t ko = (kk >> 2) * 8192 + (kk & 3) * 32;
                    const uint32_t shi = tmem + R1 + 8 * kk;
                    tc::mma_f16_ta(tmem + D1, shi, tc::sdesc_sw128(sbase + QB + ko), id64, 1);
                    tc::mma_f16_ta(tmem + D1, shi, tc::sdesc_sw128(sbase + QB + kQKPart + ko), id64, 1);
                }
                commit(B_M1Q, c);
            };
            // D2 = X^T T^T, once every value row's X^T is in TMEM and T has arrived, then part
            // B of (Q S_0)^T. A commit tracks every product issued before it, so B_M2 also
            // covers part A: the epilogue that overwrites the low part of S_0^T with U'^T
            // waits for B_M2 only.
            auto issue_m2 = [&](int c) -> bool {
                if (!waitb(B_X, c & 1, lim) || !waitb(B_T, c & 1, lim))
                    return false;
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) {
                    const uint64_t b1 = tc::sdesc(sbase + TT + kk * 256, 128, 1024);
                    const uint64_t b2 = tc::sdesc(sbase + TT + 8192 + kk * 256, 128, 1024);
                    const uint32_t xhi = tmem + XU + 8 * kk, xlo = tmem + XU + 32 + 8 * kk;
                    tc::mma_f16_ta(tmem + D2, xhi, b1, id64, kk > 0);
                    tc::mma_f16_ta(tmem + D2, xhi, b2, id64, 1);
                    tc::mma_f16_ta(tmem + D2, xlo, b1, id64, 1);
                }
                commit(B_M2, c);
                issue_m1q_hi(c);
                return true;
            };
            // S^T += U'^T K (K rows read MN-major) once U'^T is written; then, once the U^T
            // operand is written and D2's columns have been read (B_UP) and P has arrived,
            // (P U)^T = U^T P^T into D2
            auto issue_m3 = [&](int c) -> bool {
                if (!waitb(B_U, c & 1, lim))
                    return false;
                tc::fence_after_sync();
                const uint32_t kt = sbase + KB + (c & 1) * kQKRows;
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) {
                    const uint32_t koff = kk * 2048;    // K rows 16kk.. : 8-row groups 1 KB apart
                    const uint64_t k1 = tc::sdesc_sw128_mn(kt + koff, 8192, 1024);
                    const uint64_t k2 = tc::sdesc_sw128_mn(kt + kQKPart + koff, 8192, 1024);
                    const uint32_t uphi = tmem + R1 + 64 + 8 * kk, uplo = tmem + R1 + 96 + 8 * kk;
                    tc::mma_f16_ta(tmem + TS, uphi, k1, id128 | tc::kIdescTransB, 1);
                    tc::mma_f16_ta(tmem + TS, uphi, k2, id128 | tc::kIdescTransB, 1);
                    tc::mma_f16_ta(tmem + TS, uplo, k1, id128 | tc::kIdescTransB, 1);
                }
                commit(B_M3, c);
                if (!waitb(B_UP, c & 1, lim) || !waitb(B_P, c & 1, lim))
                    return false;
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) {
                    const uint64_t p1d = tc::sdesc(sbase + PP + kk * 256, 128, 1024);
                    const uint64_t p2d = tc::sdesc(sbase + PP + 8192 + kk * 256, 128, 1024);
                    const uint32_t uhi = tmem + XU + 8 * kk, ulo = tmem + XU + 32 + 8 * kk;
                    tc::mma_f16_ta(tmem + D2, uhi, p1d, id64, kk > 0);
                    tc::mma_f16_ta(tmem + D2, uhi, p2d, id64, 1);
                    tc::mma_f16_ta(tmem + D2, ulo, p1d, id64, 1);
                }
                commit(B_PU, c);
                return true;
            };
            bool ok = true;
#pragma unroll 1
            for (int c = 0; ok && c < nch; ++c)
                ok = issue_m1k(c) && issue_m1q_lo(c) && issue_m2(c) && issue_m3(c);
            // drain: products in flight finish before the CTA releases TMEM
            if (last_commit >= 0 && !tc::mbar_wait_ns(bar(last_commit), last_phase, lim))
                atomicOr(&g_device_error, (int)kErrDrain);
        }
        __syncwarp();
    } else {
        // ============================================ epilogue warps: value row j
        const int q4 = warp & 3, hf = warp >> 2;
        const int j = 32 * q4 + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        float *state_row = a.state + (((size_t)b * a.Hv + h) * kD + j) * kD + kEpiCols * hf;
        // the S_0^T operand (R1, two parts) from the fp32 master (TS)
        auto state_operand = [&]() {
#pragma unroll
            for (int k = 0; k < kEpiCols / 16; ++k) {
                float sv[16];
                tc::tmem_ld16(tl + TS + kEpiCols * hf + 16 * k, sv);
                uint32_t hi[8], lo[8];
                pack_split16(sv, hi, lo);
                tmem_st8u(tl + R1 + kEpiCols / 2 * hf + 8 * k, hi);
                tmem_st8u(tl + R1 + 64 + kEpiCols / 2 * hf + 8 * k, lo);
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            tc::mbar_arrive(bar(B_ST));
        };
        // prologue: entering state -> fp32 master (TS) and the S_0^T operand (R1)
#pragma unroll
        for (int k = 0; k < kEpiCols / 16; ++k) {
            float v16[16];
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 f = __ldg(reinterpret_cast<const float4 *>(state_row + 16 * k + e));
                v16[e] = f.x; v16[e + 1] = f.y; v16[e + 2] = f.z; v16[e + 3] = f.w;
            }
            tc::tmem_st16(tl + TS + kEpiCols * hf + 16 * k, v16);
        }
        state_operand();
        bool ok = true;
        int rho = 0;   // this chunk's state scale
#pragma unroll 1
        for (int c = 0; ok && c < nch; ++c) {
            const uint32_t par = c & 1;
            ok = waitb(B_M1, par, lim) && waitb(B_V, par, lim) && waitb(B_G, par, lim);
            if (!ok)
                break;
            tc::fence_after_sync();
            const Gates *G = gbuf + (c & 1);
            const int rho_next = next_rho(G, rho);
            const float s_in = exp2i(-rho), s_out = exp2i(rho_next);
            // ---- X^T[j][t] = beta_t V[t][j] - beta_t e^{Gam_t} (K S_0)[t][j]; the state master
            //      scaled by e^{Gam_C} ahead of this chunk's update
#pragma unroll
            for (int p = 0; p < kEpiTok / 16; ++p) {
                const int tb0 = kEpiTok * hf + 16 * p;
                float ks[16];
                tc::tmem_ld16(tl + D1 + kC + tb0, ks);
                float x[16];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    float4 f = *reinterpret_cast<const float4 *>(smem + foot_off(j, tb0 / 4 + qq));
                    f.x = silu_f(f.x); f.y = silu_f(f.y); f.z = silu_f(f.z); f.w = silu_f(f.w);
                    const float4 bt = ld4(G->beta + tb0 + 4 * qq), bg = ld4(G->bg + tb0 + 4 * qq);
                    x[4 * qq + 0] = __fsub_rn(__fmul_rn(bt.x, f.x), __fmul_rn(__fmul_rn(bg.x, s_in), ks[4 * qq + 0]));
                    x[4 * qq + 1] = __fsub_rn(__fmul_rn(bt.y, f.y), __fmul_rn(__fmul_rn(bg.y, s_in), ks[4 * qq + 1]));
                    x[4 * qq + 2] = __fsub_rn(__fmul_rn(bt.z, f.z), __fmul_rn(__fmul_rn(bg.z, s_in), ks[4 * qq + 2]));
                    x[4 * qq + 3] = __fsub_rn(__fmul_rn(bt.w, f.w), __fmul_rn(__fmul_rn(bg.w, s_in), ks[4 * qq + 3]));
                }
                uint32_t hi[8], lo[8];
                pack_split16(x, hi, lo);
                tmem_st8u(tl + XU + tb0 / 2, hi);
                tmem_st8u(tl + XU + 32 + tb0 / 2, lo);
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            tc::mbar_arrive(bar(B_X));
            // the state master scaled by e^{Gam_C} while D2's product runs: only the state
            // update reads it, and that is issued after B_U (whose fence covers these stores)
            {
                const float ec = __fmul_rn(G->ec, exp2i(rho_next - rho));
#pragma unroll
                for (int k = 0; k < kEpiCols / 16; ++k) {
                    float sv[16];
                    tc::tmem_ld16(tl + TS + kEpiCols * hf + 16 * k, sv);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        sv[e] = __fmul_rn(sv[e], ec);
                    tc::tmem_st16(tl + TS + kEpiCols * hf + 16 * k, sv);
                }
            }
            // ---- U = T X (from D2): first U'^T = U^T diag(e^{Gam_C - Gam}) for the state
            //      update (B_U), then U^T for the output product (B_UP), which also reads D2's
            //      columns again before that product overwrites them
            if (!(ok = waitb(B_M2, par, lim)))
                break;
            tc::fence_after_sync();
#pragma unroll
            for (int p = 0; p < kEpiTok / 16; ++p) {
                const int tb0 = kEpiTok * hf + 16 * p;
                float u[16];
                tc::tmem_ld16(tl + D2 + tb0, u);
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const float4 g4 = ld4(G->egc + tb0 + 4 * qq);
                    u[4 * qq + 0] = __fmul_rn(u[4 * qq + 0], __fmul_rn(g4.x, s_out));
                    u[4 * qq + 1] = __fmul_rn(u[4 * qq + 1], __fmul_rn(g4.y, s_out));
                    u[4 * qq + 2] = __fmul_rn(u[4 * qq + 2], __fmul_rn(g4.z, s_out));
                    u[4 * qq + 3] = __fmul_rn(u[4 * qq + 3], __fmul_rn(g4.w, s_out));
                }
                uint32_t hi[8], lo[8];
                pack_split16(u, hi, lo);
                tmem_st8u(tl + R1 + 64 + tb0 / 2, hi);
                tmem_st8u(tl + R1 + 96 + tb0 / 2, lo);
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            tc::mbar_arrive(bar(B_U));
#pragma unroll
            for (int p = 0; p < kEpiTok / 16; ++p) {
                const int tb0 = kEpiTok * hf + 16 * p;
                float u[16];
                tc::tmem_ld16(tl + D2 + tb0, u);
                uint32_t hi[8], lo[8];
                pack_split16(u, hi, lo);
                tmem_st8u(tl + XU + tb0 / 2, hi);
                tmem_st8u(tl + XU + 32 + tb0 / 2, lo);
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            tc::mbar_arrive(bar(B_UP));
            // ---- the updated state: the next chunk's S_0^T operand (its first product follows)
            if (!(ok = waitb(B_M3, par, lim)))
                break;
            tc::fence_after_sync();
            if (c + 1 < nch) {
                state_operand();
            } else {
                // ---- final state back to HBM (S^T rows = the library layout), unscaled
                const float us = exp2i(-rho_next);
#pragma unroll
                for (int k = 0; k < kEpiCols / 16; ++k) {
                    float sv[16];
                    tc::tmem_ld16(tl + TS + kEpiCols * hf + 16 * k, sv);
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4 *>(state_row + 16 * k + e) =
                            make_float4(__fmul_rn(sv[e], us), __fmul_rn(sv[e + 1], us),
                                        __fmul_rn(sv[e + 2], us), __fmul_rn(sv[e + 3], us));
                }
            }
            // ---- O^T row j = e^{Gam} (Q S_0)^T + (P U)^T, scaled by 1/sqrt(d)
            //      (the two terms are added here, rounded, rather than in the accumulator: for a
            //      token whose readout nearly cancels this is the sum that decides its precision).
            //      (P U)^T's commit also covers (Q S_0)^T, issued before it.
            if (!(ok = waitb(B_PU, par, lim)))
                break;
            tc::fence_after_sync();
            float o[kEpiTok];
#pragma unroll
            for (int p = 0; p < kEpiTok / 16; ++p) {
                const int tb0 = kEpiTok * hf + 16 * p;
                float qs[16], pu[16];
                tc::tmem_ld16(tl + D1 + tb0, qs);
                tc::tmem_ld16(tl + D2 + tb0, pu);
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const float4 eg = ld4(G->eg + tb0 + 4 * qq);
                    const float egv[4] = {eg.x, eg.y, eg.z, eg.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int k = 4 * qq + e;
                        o[16 * p + k] = __fmul_rn(__fmaf_rn(qs[k], __fmul_rn(egv[e], s_in), pu[k]), a.scale);
                    }
                }
            }
            tc::fence_before_sync();
            tc::mbar_arrive(bar(B_OR));
            // ---- token-major staging for the conv warps' norm, once they have read chunk c-1's
            if (c > 0 && !(ok = waitb(B_OSFREE, (c - 1) & 1, lim)))
                break;
#pragma unroll
            for (int p = 0; p < kEpiTok / 16; ++p)
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    Os[(kEpiTok * hf + 16 * p + k) * kD + j] = o[16 * p + k];
            tc::mbar_arrive(bar(B_OS));
            rho = rho_next;
        }
    }

    // ---- teardown
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0 && *abort)
        atomicOr(&g_device_error, *abort);
    if (warp == 0)
        tc::tmem_dealloc(tmem, 512);
}

template <typename TIn>
__global__ void __launch_bounds__(256) prefill_history_kernel(float *conv_state, const TIn *x,
                                                              int64_t x_stride, int conv_dim, int W,
                                                              int T)
{
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const int b = blockIdx.y;
    if (c >= conv_dim)
        return;
    float *hist_c = conv_state + ((size_t)b * conv_dim + c) * (W - 1);
    float nh[kMaxW - 1];
    conv_history_after<TIn>(hist_c, x + (int64_t)b * T * x_stride + c, x_stride, W, T, nh);
    store_history(hist_c, W, nh);
}

template <typename TIn, int WC>
cudaError_t prefill_typed(const PrefillArgs &a, const CUtensorMap &map, int staged, cudaStream_t s)
{
    auto k1 = prefill_ut_kernel<TIn, WC>;
    auto k2 = prefill_chain_kernel<TIn, WC>;
    static const cudaError_t attr = [&] {
        cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p1::BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p2::BYTES);
        return e;
    }();
    if (attr != cudaSuccess)
        return attr;
    k1<<<dim3(a.n_chunks, a.Hq, a.B), p1::kThreads, p1::BYTES, s>>>(map, a, staged);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    // the gated norm reads 4 z values per lane with one vector load when rows allow it
    const size_t es = sizeof(TIn);
    const int zvec = (reinterpret_cast<uintptr_t>(a.z) % (4 * es) == 0 && (a.z_stride * es) % (4 * es) == 0) ? 1 : 0;
    k2<<<dim3(a.Hv, a.B, 1), p2::kThreads, p2::BYTES, s>>>(map, a, staged, zvec);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    prefill_history_kernel<TIn><<<dim3((a.conv_dim + 255) / 256, a.B, 1), 256, 0, s>>>(
        a.conv_state, static_cast<const TIn *>(a.x), a.x_stride, a.conv_dim, a.W, a.T);
    return cudaGetLastError();
}

}  // namespace

cudaError_t take_prefill_device_error(int *code)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int));
    if (e == cudaSuccess && v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    }
    *code = v;
    return e;
}

cudaError_t launch_prefill(const PrefillArgs &a, bool bf16, cudaStream_t s)
{
    CUtensorMap map;
    memset(&map, 0, sizeof map);
    // chunk rows of one 128-channel head, (63 + W) rows from token c0 - (W - 1); bf16 rows only
    const int staged = bf16 && encode_rows_map(&map, a.x, true, a.conv_dim, a.x_stride, a.T, a.B, kD,
                                               (uint32_t)(kC + a.W - 1))
                           ? 1 : 0;
    if (bf16)
        return a.W == 4 ? prefill_typed<__nv_bfloat16, 4>(a, map, staged, s)
                        : prefill_typed<__nv_bfloat16, 0>(a, map, staged, s);
    return a.W == 4 ? prefill_typed<float, 4>(a, map, staged, s) : prefill_typed<float, 0>(a, map, staged, s);
}

}  // namespace gdn
