// gdn_device.cuh -- device building blocks shared by every libgdn kernel.
//
// Every kernel that computes a given quantity calls the same function here,
// with explicit round-to-nearest intrinsics (no compiler contraction
// choices), so the fused decode step, the K=2 verify and the standalone
// entry points produce bit-identical results for the same inputs.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kD = 128;        // head_dim this library supports
constexpr int kMaxW = 8;       // largest conv tap count
constexpr float kSoftplusGuard = 20.0f;

// ------------------------------------------------------------------ loads
template <typename T>
__device__ __forceinline__ float load_act(const T *p);
template <>
__device__ __forceinline__ float load_act<float>(const float *p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_act<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat162float(__ldg(p));
}

// State rows are touched once per step: stream them past the caches.
__device__ __forceinline__ float4 ld_stream(const float *p)
{
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st_stream(float *p, float4 v)
{
    __stcs(reinterpret_cast<float4 *>(p), v);
}

// ------------------------------------------------------------------ checked build
// Range checks of the kernels' index arithmetic, compiled in by -DGDN_CHECKS (the
// checked library, libgdn_checked.so): a failing check sets bit 32 of the file's
// device-side error word (read by gdn_check_device) and the kernel goes on, so that a
// test sees the bit instead of a trap. Without the define the checks vanish.
constexpr int kErrRange = 32;
#ifdef GDN_CHECKS
#define GDN_CHECK(word, cond)                   \
    do {                                        \
        if (!(cond))                            \
            atomicOr(&(word), gdn::kErrRange);  \
    } while (0)
#else
#define GDN_CHECK(word, cond) \
    do {                      \
    } while (0)
#endif

// ------------------------------------------------------------------ scalar maps
// silu(x) = x * sigmoid(x) = x / (1 + e^-x), from the hardware exponential and
// the fast divide: a few ulp (about 1e-6 relative for |x| < 20), cheap enough
// for the multi-token conv paths, where the IEEE divide alone dominated the
// instruction count. Large negative x gives e^-x = inf and a quotient of 0;
// large positive x gives x.
__device__ __forceinline__ float silu_f(float x)
{
    return __fdividef(x, __fadd_rn(1.0f, __expf(-x)));
}

__device__ __forceinline__ float sigmoid_f(float x)
{
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-x)));
}

// Decay gate, "fm_kernel_ssm.h" section "Decay gate": g = a * softplus(alpha + dt),
// a = -exp(A_log), softplus guarded at 20 (identity above it). Returns g pre-exp.
__device__ __forceinline__ float decay_gate_f(float alpha, float dt, float A_log)
{
    const float a = -expf(A_log);
    const float v = __fadd_rn(alpha, dt);
    const float sp = v > kSoftplusGuard ? v : log1pf(expf(v));
    return __fmul_rn(a, sp);
}

// ------------------------------------------------------------------ conv
// Depthwise causal conv tap sum for one channel at token u of the call
// ("fm_kernel_ssm.h", "Causal depthwise conv1d + SiLU"): the window is the
// channel's input stream at tokens u-W+1 .. u, where stream index s < 0 reads
// the history hist_c[W-1+s] and s >= 0 reads the RAW input x_c[s * x_stride].
// Taps are summed oldest first.
template <typename TIn>
__device__ __forceinline__ float conv_stream_at(const float *hist_c, const TIn *x_c,
                                                int64_t x_stride, int W, int s)
{
    return s < 0 ? hist_c[W - 1 + s] : load_act<TIn>(x_c + (int64_t)s * x_stride);
}

template <typename TIn>
__device__ __forceinline__ float conv_pre(const float *hist_c, const TIn *x_c, int64_t x_stride,
                                          const float *w_c, int W, int u)
{
    float acc = __fmul_rn(conv_stream_at<TIn>(hist_c, x_c, x_stride, W, u - W + 1), __ldg(w_c));
    for (int tau = 1; tau < W; ++tau)
        acc = __fmaf_rn(conv_stream_at<TIn>(hist_c, x_c, x_stride, W, u - W + 1 + tau),
                        __ldg(w_c + tau), acc);
    return acc;
}

// New history (W-1 entries, oldest first) after the first n tokens of the call.
// Reads every value before the caller writes any, so hist may be updated in place.
template <typename TIn>
__device__ __forceinline__ void conv_history_after(const float *hist_c, const TIn *x_c,
                                                   int64_t x_stride, int W, int n,
                                                   float (&nh)[kMaxW - 1])
{
#pragma unroll
    for (int tau = 0; tau < kMaxW - 1; ++tau)
        if (tau < W - 1)
            nh[tau] = conv_stream_at<TIn>(hist_c, x_c, x_stride, W, n - (W - 1) + tau);
}

__device__ __forceinline__ void store_history(float *dst_c, int W, const float (&nh)[kMaxW - 1])
{
#pragma unroll
    for (int tau = 0; tau < kMaxW - 1; ++tau)
        if (tau < W - 1)
            dst_c[tau] = nh[tau];
}

// The same tap sum from a register window, for kernels that step NTOK tokens
// of one channel: win[e] holds the channel's stream at index e - (W-1)
// (history first, then the NTOK raw inputs), w[tau] its taps. Every load is
// independent (one memory round trip), and the arithmetic order is conv_pre's.
template <int NTOK>
struct ConvWindow {
    float win[kMaxW - 1 + NTOK];
    float w[kMaxW];
};

template <typename TIn, int NTOK>
__device__ __forceinline__ void conv_window_load(const float *hist_c, const TIn *x_c,
                                                 int64_t x_stride, const float *w_c, int W,
                                                 ConvWindow<NTOK> &cw)
{
#pragma unroll
    for (int e = 0; e < kMaxW - 1 + NTOK; ++e) {
        if (e < W - 1)
            cw.win[e] = hist_c[e];
        else if (e < W - 1 + NTOK)
            cw.win[e] = load_act<TIn>(x_c + (int64_t)(e - (W - 1)) * x_stride);
        else
            cw.win[e] = 0.0f;
    }
#pragma unroll
    for (int tau = 0; tau < kMaxW; ++tau)
        cw.w[tau] = tau < W ? __ldg(w_c + tau) : 0.0f;
}

// The history part of conv_window_load (the previous call may have written it)
template <int NTOK>
__device__ __forceinline__ void conv_window_load_hist(const float *hist_c, int W, ConvWindow<NTOK> &cw)
{
#pragma unroll
    for (int e = 0; e < kMaxW - 1; ++e)
        if (e < W - 1)
            cw.win[e] = hist_c[e];
}

template <int NTOK>
__device__ __forceinline__ float conv_window_pre(const ConvWindow<NTOK> &cw, int W, int p)
{
    float acc = __fmul_rn(cw.win[p], cw.w[0]);
#pragma unroll
    for (int tau = 1; tau < kMaxW; ++tau)
        if (tau < W && p + tau < kMaxW - 1 + NTOK)
            acc = __fmaf_rn(cw.win[p + tau], cw.w[tau], acc);
    return acc;
}

// History after the first n tokens: win[n .. n+W-2].
template <int NTOK>
__device__ __forceinline__ void conv_window_history(const ConvWindow<NTOK> &cw, int W, int n,
                                                    float (&nh)[kMaxW - 1])
{
#pragma unroll
    for (int tau = 0; tau < kMaxW - 1; ++tau) {
        nh[tau] = 0.0f;
#pragma unroll
        for (int nn = 0; nn <= NTOK; ++nn)
            if (nn == n && tau < W - 1 && nn + tau < kMaxW - 1 + NTOK)
                nh[tau] = cw.win[nn + tau];
    }
}

// ------------------------------------------------------------------ reductions
__device__ __forceinline__ float warp_sum32(float v)
{
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// Sum over the 8 lanes that share one state row (lanes 8g .. 8g+7).
__device__ __forceinline__ float row8_sum(float v)
{
    v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
    v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
    v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
    return v;
}

// L2 norm of one 128-channel head held one value per thread by 4 consecutive
// warps (thread i of the head = channel i). red4 is 4 floats of shared memory
// private to this head. Returns 1 / sqrt(sum v^2 + eps) to every thread.
// Caller must __syncthreads() between this and any reuse of red4.
// The head's 1 / sqrt(sum v^2 + eps) from its four 32-channel warp sums, in order.
__device__ __forceinline__ float l2_inv_of_partials(const float *red4, float eps)
{
    const float tot = __fadd_rn(__fadd_rn(__fadd_rn(red4[0], red4[1]), red4[2]), red4[3]);
    return rsqrtf(__fadd_rn(tot, eps));
}

__device__ __forceinline__ float head_l2_inv(float v, float eps, float *red4, int warp_in_head,
                                             int lane)
{
    float s = warp_sum32(__fmul_rn(v, v));
    if (lane == 0)
        red4[warp_in_head] = s;
    __syncthreads();
    return l2_inv_of_partials(red4, eps);
}

// ------------------------------------------------------------------ gated norm
// Sum of squares of one 32-row block of a head's readout (lane l holds row l of
// the block). The head total is ((b0 + b1) + b2) + b3 over its four blocks.
__device__ __forceinline__ float norm_block_partial(float y)
{
    return warp_sum32(__fmul_rn(y, y));
}

__device__ __forceinline__ float norm_inv(float b0, float b1, float b2, float b3, float eps)
{
    const float tot = __fadd_rn(__fadd_rn(__fadd_rn(b0, b1), b2), b3);
    return rsqrtf(__fadd_rn(__fmul_rn(tot, 1.0f / kD), eps));
}

// "fm_kernel_ssm.h", "Gated RMSNorm": ((y * inv) * w) * silu(z)
__device__ __forceinline__ float gated_out(float y, float inv, float w, float z)
{
    return __fmul_rn(__fmul_rn(__fmul_rn(y, inv), w), silu_f(z));
}

// ------------------------------------------------------------------ recurrence
// One warp advances 4*NG value rows of one head by NTOK tokens
// ("fm_kernel_ssm.h", "Delta-rule recurrence"). Each row of 128 floats is
// held by 8 lanes, 16 floats per lane: lane l of the warp owns row group
// rg = l / 8 and the float4 columns (m*8 + l%8), m = 0..3, so every float4
// load of the warp covers four complete 512-byte rows with 128-byte
// segments. Per row j and token, with decay = exp(g):
//   pk = row . k,  pq = row . q                    (old row, 8-lane sums)
//   delta = beta * (v_j - decay * pk)              (prediction on the decayed row)
//   row  <- decay * row + delta * k                (decay + rank-1 write)
//   y_j  = scale * (decay * pq + delta * (k . q))  (readout of the updated row)
// which is the page's read-after-write readout, expanded so that both dot
// products share one reduction.
//
// load_rows issues the warp's loads (callers issue them before their
// prologue so the HBM latency overlaps it); step_rows advances them in
// registers; store_rows writes them back:
//   rows       first row of this warp's block in global memory (row stride kD)
//   snap_rows  same rows in the snapshot buffer (used when SNAP): the rows after
//              token p go to snap_rows + p * snap_stride for p < n_snap
//   sk, sq     shared [NTOK][kD] normalised k, q
//   sv         shared [NTOK][v_stride] v, indexed by the row's local index
//   sdecay, sbeta shared [NTOK]
//   sy         shared [NTOK][v_stride] readout y (written by one lane per row)
//   local_row0 local index of this warp's first row
template <int NG>
__device__ __forceinline__ void load_rows(const float *rows, float4 (&r)[NG][4])
{
    const int lane = threadIdx.x & 31;
    const int rg = lane >> 3;
    const int sub = lane & 7;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
#pragma unroll
        for (int m = 0; m < 4; ++m)
            r[gi][m] = ld_stream(rows + (size_t)(gi * 4 + rg) * kD + (m * 8 + sub) * 4);
}

// Row registers to and from fp32 float4 (identity for float32 rows; packed bf16
// pairs are widened exactly and rounded to nearest even).
__device__ __forceinline__ float4 to_f4(float4 v) { return v; }
__device__ __forceinline__ float4 to_f4(uint2 u)
{
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ void from_f4(float4 v, float4 &r) { r = v; }
__device__ __forceinline__ void from_f4(float4 v, uint2 &r)
{
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    r.x = *reinterpret_cast<const uint32_t *>(&lo);
    r.y = *reinterpret_cast<const uint32_t *>(&hi);
}

// One float4 of a row to its storage type (streaming store; bf16: round to nearest even).
__device__ __forceinline__ void store_one(float *p, float4 v) { st_stream(p, v); }
__device__ __forceinline__ void store_one(__nv_bfloat16 *p, float4 v)
{
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&lo);
    u.y = *reinterpret_cast<const uint32_t *>(&hi);
    __stcs(reinterpret_cast<uint2 *>(p), u);
}

// final_rows, when given, receives each 4-row group as soon as its last token
// is applied, so the write traffic starts while later groups are still being
// stepped (the single-token kernels otherwise keep the rows until the norm).
template <int NG, int NTOK, bool SNAP, typename TSt = float, typename Reg = float4>
__device__ __forceinline__ void step_rows(Reg (&r)[NG][4], float *snap_rows,
                                          const float *sk, const float *sq, const float *sv,
                                          int v_stride, const float *sdecay, const float *sbeta,
                                          float *sy, int local_row0, float scale,
                                          TSt *final_rows = nullptr, int n_snap = 1,
                                          size_t snap_stride = 0)
{
    const int lane = threadIdx.x & 31;
    const int rg = lane >> 3;
    const int sub = lane & 7;
#pragma unroll
    for (int p = 0; p < NTOK; ++p) {
        float4 k4[4], q4[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            k4[m] = *reinterpret_cast<const float4 *>(sk + p * kD + (m * 8 + sub) * 4);
            q4[m] = *reinterpret_cast<const float4 *>(sq + p * kD + (m * 8 + sub) * 4);
        }
        float kq = __fmul_rn(k4[0].x, q4[0].x);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            if (m > 0)
                kq = __fmaf_rn(k4[m].x, q4[m].x, kq);
            kq = __fmaf_rn(k4[m].y, q4[m].y, kq);
            kq = __fmaf_rn(k4[m].z, q4[m].z, kq);
            kq = __fmaf_rn(k4[m].w, q4[m].w, kq);
        }
        kq = row8_sum(kq);
        const float decay = sdecay[p];
        const float beta = sbeta[p];
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            float4 f[4];
#pragma unroll
            for (int m = 0; m < 4; ++m)
                f[m] = to_f4(r[gi][m]);
            float pk = __fmul_rn(f[0].x, k4[0].x);
            float pq = __fmul_rn(f[0].x, q4[0].x);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (m > 0) {
                    pk = __fmaf_rn(f[m].x, k4[m].x, pk);
                    pq = __fmaf_rn(f[m].x, q4[m].x, pq);
                }
                pk = __fmaf_rn(f[m].y, k4[m].y, pk);
                pq = __fmaf_rn(f[m].y, q4[m].y, pq);
                pk = __fmaf_rn(f[m].z, k4[m].z, pk);
                pq = __fmaf_rn(f[m].z, q4[m].z, pq);
                pk = __fmaf_rn(f[m].w, k4[m].w, pk);
                pq = __fmaf_rn(f[m].w, q4[m].w, pq);
            }
            pk = row8_sum(pk);
            pq = row8_sum(pq);
            const int lrow = local_row0 + gi * 4 + rg;
            const float vj = sv[p * v_stride + lrow];
            const float delta = __fmul_rn(beta, __fsub_rn(vj, __fmul_rn(decay, pk)));
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                f[m].x = __fmaf_rn(delta, k4[m].x, __fmul_rn(decay, f[m].x));
                f[m].y = __fmaf_rn(delta, k4[m].y, __fmul_rn(decay, f[m].y));
                f[m].z = __fmaf_rn(delta, k4[m].z, __fmul_rn(decay, f[m].z));
                f[m].w = __fmaf_rn(delta, k4[m].w, __fmul_rn(decay, f[m].w));
                from_f4(f[m], r[gi][m]);
            }
            const float y = __fmul_rn(scale, __fmaf_rn(delta, kq, __fmul_rn(decay, pq)));
            if (sub == 0)
                sy[p * v_stride + lrow] = y;
            if (final_rows != nullptr && p == NTOK - 1) {
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    store_one(final_rows + (size_t)(gi * 4 + rg) * kD + (m * 8 + sub) * 4, f[m]);
            }
        }
        if constexpr (SNAP) {
            if (p < n_snap) {
#pragma unroll
                for (int gi = 0; gi < NG; ++gi)
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        st_stream(snap_rows + p * snap_stride + (size_t)(gi * 4 + rg) * kD + (m * 8 + sub) * 4,
                                  to_f4(r[gi][m]));
            }
        }
    }
}

// Write the advanced rows back (callers issue this late, after any cluster
// barrier, so no release fence waits on these stores).
template <int NG>
__device__ __forceinline__ void store_rows(const float4 (&r)[NG][4], float *rows)
{
    const int lane = threadIdx.x & 31;
    const int rg = lane >> 3;
    const int sub = lane & 7;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
#pragma unroll
        for (int m = 0; m < 4; ++m)
            st_stream(rows + (size_t)(gi * 4 + rg) * kD + (m * 8 + sub) * 4, r[gi][m]);
}

// bf16 storage of the same rows (the bf16-state decode): lane l holds the same
// 16 columns as above as four 8-byte groups of packed bf16 pairs (each warp
// load instruction covers 64 contiguous bytes of four rows). The rows stay
// packed in registers, half the registers of the float32 rows, and are widened
// exactly to fp32 group by group as they are stepped.
template <int NG>
__device__ __forceinline__ void load_rows(const __nv_bfloat16 *rows, uint2 (&r)[NG][4])
{
    const int lane = threadIdx.x & 31;
    const int rg = lane >> 3;
    const int sub = lane & 7;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
#pragma unroll
        for (int m = 0; m < 4; ++m)
            r[gi][m] = __ldcs(reinterpret_cast<const uint2 *>(
                rows + (size_t)(gi * 4 + rg) * kD + (m * 8 + sub) * 4));
}

// One output value in the storage type (bf16: round to nearest even).
__device__ __forceinline__ void store_out(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

}  // namespace gdn
