// prefill_tc.cu -- chunked prefill on the tcgen05 tensor cores.
//
// One CTA (8 warps) per (sequence, V head) walks the sequence in 64-token
// chunks. Per chunk, with Gam the in-chunk cumulative decay, S_0 the entering
// state in the plain orientation S[i][j] and the chunk algebra derived from the
// recurrence of "fm_kernel_ssm.h" section "Delta-rule recurrence" (64-token
// chunks with ceil(T/64) sequential links as in the "Mamba-2 SSD chunked
// prefill scan" note of "ssm_mamba.rs"):
//   G   = [Q; K] K^T                         tensor core   (QK^T and KK^T)
//   P   = e^{Gam_t-Gam_s} (QK^T)[t][s], s<=t  CUDA cores
//   A   = beta_t e^{Gam_t-Gam_s} (KK^T)[t][s], s<t      CUDA cores
//   KS  = S_0^T [Q; K]^T                     tensor core   ((Q S_0)^T, (K S_0)^T)
//   X   = beta V - beta e^{Gam} K S_0;  U = (I + A)^{-1} X by blocked forward
//         substitution, one value column per thread               CUDA cores
//   O^T = e^{Gam} (Q S_0)^T + U^T P^T        tensor core (accumulates onto KS)
//   S^T <- e^{Gam_C} S^T + U^T (diag(e^{Gam_C-Gam}) K)   tensor core (state in TMEM)
// then the gated RMSNorm of each token's O row. Every product is arranged
// so that M = 128 (the value index j, or the stacked [Q; K] token index),
// each TMEM lane holding one row of the result. Warps 4-7 run the V conv while
// the tensor core forms G and KS and warps 0-3 build P and A.
//
// Precision: operands are fp32 values split into bf16 parts, by default two
// (x = x1 + x2, ~16 bits; products x1 y1 + x1 y2 + x2 y1), with a three-part
// option on the readout products (kParts below). Accumulation is fp32 in
// TMEM. Against the fp64 scan the outputs stay within ~3e-5 and the state
// within ~2e-5, normwise per head, on the 4 x 8192 workload.
//
// Shared-memory operand tiles use the no-swizzle K-major core-matrix layout of
// tc_ptx.cuh, except the [Q; K] tile, which is 128-byte swizzled so that the
// conv's row stores do not conflict. The conv + SiLU + L2 and the gates of
// the chunk's tokens are computed in the CTA from the raw inputs; the conv
// history is rewritten by a second small kernel after every CTA has read it.
#include "gdn_device.cuh"
#include "gdn_kernels.h"
#include "tc_ptx.cuh"

namespace gdn {

// Set when a bounded wait of a kernel in this file gives up; read and cleared
// by take_prefill_device_error.
static __device__ int g_device_error;

namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;

// byte offsets in dynamic shared memory
// Tiles whose live ranges do not overlap share space: the third parts of
// [Q; K] and S^T are only read by the G and KS products, before T, P and
// (e^{Gam_C-Gam} K)^T are written.
constexpr uint32_t QK_HI = 0, QK_LO = 32768;        // [128 t'][128 i]  (Q rows, then K rows), 128-byte swizzled
constexpr uint32_t ST_HI = 65536, ST_LO = 98304;    // [128 j][128 i]   S^T
constexpr uint32_t KT_HI = 131072, KT_LO = 147456;  // [128 i][64 t]    (e^{Gam_C-Gam} K)^T
constexpr uint32_t ST_3 = 131072;                   // third part of S^T (in KT's space)
constexpr uint32_t XU_HI = 163840, XU_LO = 180224;  // [128 j][64 t]    U^T; V^T and O staging
constexpr uint32_t TT_HI = 196608;                  // [64 t][64 s]     A (fp32, 16 KB)
constexpr uint32_t PP_HI = 212992, PP_LO = 221184;  // [64 t][64 s]     P
constexpr uint32_t QK_3 = 196608;                   // third part of [Q; K] (in TT and PP's space)
// third parts of U^T and P, in the Q rows of [Q; K] (dead once G and KS are formed)
constexpr uint32_t XU_3 = QK_HI, PP_3 = QK_LO + 8192;

// The fp32 footprint of value row j in the X^T/U^T tile: float4 chunk q
// (tokens 4q .. 4q+3) of the row. Its 16-byte slot is XOR-ed with the row
// group (j / 8), so that the V conv's stores (eight rows of different 8-row
// groups per quarter-warp) and a warp's per-row reads both hit distinct bank
// groups. The two-part U^T operand written over it afterwards uses the plain
// core-matrix slots, so that write waits for every row's last read.
__host__ __device__ constexpr uint32_t foot_off(int j, int q)
{
    return (uint32_t)((q < 8 ? XU_HI : XU_LO) + (j >> 3) * 1024 + (q & 7) * 128 +
                      (((j & 7) ^ ((j >> 3) & 7)) << 4));
}

// Tokens per block of the blocked forward substitution U = (I + A)^{-1} X.
#ifndef GDN_SUBST_BLOCK
#define GDN_SUBST_BLOCK 8
#endif
constexpr int kSB = GDN_SUBST_BLOCK;
static_assert(kSB == 8 || kSB == 16, "8- or 16-token blocks");

// bf16 parts per fp32 operand on the readout products (G, KS, O): 2 parts and
// three product terms (~16 bits), or 3 parts and six terms (~24 bits). Two
// parts keep the outputs within ~3e-5 of the fp64 scan (normwise per head) on
// the 4 x 8192 workload and leave the state error (set by the two-part state
// update) unchanged; three parts (built with -DGDN_PREFILL_PARTS=3) give
// ~5e-6 at 14% more time.
#ifndef GDN_PREFILL_PARTS
#define GDN_PREFILL_PARTS 2
#endif
constexpr int kParts = GDN_PREFILL_PARTS;
static_assert(kParts == 2 || kParts == 3, "2 or 3 bf16 parts");
constexpr uint32_t SC_G = 229376, SC_BETA = SC_G + 256, SC_GAM = SC_BETA + 256,
                   SC_GAML = SC_GAM + 256, SC_EG = SC_GAML + 256, SC_EGC = SC_EG + 256,
                   SC_EGCC = SC_EGC + 256, SC_MBAR = SC_EGCC + 8, SC_TMEM = SC_MBAR + 32,
                   SC_ERR = SC_TMEM + 4, SMEM_BYTES = SC_ERR + 4;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(QK_HI % 1024 == 0 && QK_LO % 1024 == 0 && QK_3 % 1024 == 0,
              "swizzled [Q; K] tiles start on 1024-byte boundaries");

// TMEM columns
constexpr uint32_t TM_G = 0, TM_KS = 64, TM_S = 256, TM_COLS = 512;
constexpr int kWaitLimit = 1 << 26;

__device__ __forceinline__ void split8(const float (&v)[8], uint4 &hi, uint4 &lo)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 hh = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        const float2 hf = __bfloat1622float2(hh);
        const __nv_bfloat162 ll = __floats2bfloat162_rn(v[2 * e] - hf.x, v[2 * e + 1] - hf.y);
        h[e] = *reinterpret_cast<const uint32_t *>(&hh);
        l[e] = *reinterpret_cast<const uint32_t *>(&ll);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void split8x3(const float (&v)[8], uint4 &p1, uint4 &p2, uint4 &p3)
{
    uint32_t a[4], b[4], c[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h1 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        const float2 f1 = __bfloat1622float2(h1);
        const float r0 = v[2 * e] - f1.x, r1 = v[2 * e + 1] - f1.y;
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(r0, r1);
        const float2 f2 = __bfloat1622float2(h2);
        const __nv_bfloat162 h3 = __floats2bfloat162_rn(r0 - f2.x, r1 - f2.y);
        a[e] = *reinterpret_cast<const uint32_t *>(&h1);
        b[e] = *reinterpret_cast<const uint32_t *>(&h2);
        c[e] = *reinterpret_cast<const uint32_t *>(&h3);
    }
    p1 = make_uint4(a[0], a[1], a[2], a[3]);
    p2 = make_uint4(b[0], b[1], b[2], b[3]);
    p3 = make_uint4(c[0], c[1], c[2], c[3]);
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

// 8 consecutive channels of one input row as floats (16-byte aligned rows).
template <typename TIn>
__device__ __forceinline__ void load8(const TIn *p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float (&v)[8])
{
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        v[2 * e] = __uint_as_float(w[e] << 16);
        v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}
template <>
__device__ __forceinline__ void load8<float>(const float *p, float (&v)[8])
{
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// conv + SiLU of 8 channels (cb .. cb+7) for 8 tokens (t0 .. t0+7 of the call);
// tokens at or past T give 0. WC > 0 fixes the tap count at compile time so
// that all window loads issue together; WC == 0 reads it from the arguments.
template <typename TIn, int WC>
__device__ __forceinline__ void conv8x8(const PrefillArgs &a, int b, int cb, int t0,
                                        float (&out)[8][8])
{
    const int W = WC > 0 ? WC : a.W, T = a.T;
    const TIn *xb = static_cast<const TIn *>(a.x) + (int64_t)b * T * a.x_stride + cb;
    const float *hist = a.conv_state + ((size_t)b * a.conv_dim + cb) * (W - 1);
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            out[t][e] = 0.0f;
#pragma unroll
    for (int tau = 0; tau < (WC > 0 ? WC : kMaxW); ++tau) {
        if (tau >= W)
            break;
        float w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            w[e] = __ldg(a.conv_w + (size_t)(cb + e) * W + tau);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int s = t0 + t - (W - 1) + tau;    // stream index of this tap
            float v[8];
            if (s >= 0 && s < T) {
                load8<TIn>(xb + (int64_t)s * a.x_stride, v);
            } else if (s < 0) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[e] = hist[(size_t)e * (W - 1) + (W - 1 + s)];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[e] = 0.0f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                out[t][e] = __fmaf_rn(v[e], w[e], out[t][e]);
        }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            out[t][e] = t0 + t < T ? silu_f(out[t][e]) : 0.0f;
}

// The four-tap conv for a block whose window lies inside the call (every
// 8-token block but the first of a sequence): each of the 11 input rows is
// read once with a branch-free load (rows past the end of the call read the
// last row and are masked), so all loads issue together; SiLU uses the fast
// exponential.
template <typename TIn>
__device__ __forceinline__ void conv8x8_w4_inner(const PrefillArgs &a, int b, int cb, int t0,
                                                 float (&out)[8][8])
{
    const int T = a.T;
    const TIn *xb = static_cast<const TIn *>(a.x) + (int64_t)b * T * a.x_stride + cb;
    float w[8][4];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float4 f = __ldg(reinterpret_cast<const float4 *>(a.conv_w + (size_t)(cb + e) * 4));
        w[e][0] = f.x; w[e][1] = f.y; w[e][2] = f.z; w[e][3] = f.w;
    }
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            out[t][e] = 0.0f;
#pragma unroll
    for (int rr = 0; rr < 11; ++rr) {
        const int sidx = t0 - 3 + rr;                 // >= 0 on this path
        float v[8];
        load8<TIn>(xb + (int64_t)min(sidx, T - 1) * a.x_stride, v);
        const bool live = sidx < T;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            v[e] = live ? v[e] : 0.0f;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int tau = rr - t;                   // tap that row rr feeds for token t
            if (tau >= 0 && tau < 4) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    out[t][e] = __fmaf_rn(v[e], w[e][tau], out[t][e]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float x = out[t][e];
            out[t][e] = t0 + t < T ? __fdividef(x, 1.0f + __expf(-x)) : 0.0f;
        }
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(PrefillArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.y, h = blockIdx.x;
    const int hk = h / (a.Hv / a.Hq);
    const int T = a.T;
    const uint32_t sbase = tc::smem_addr(smem);
    // the [Q; K] tile's swizzle follows address bits 7-9: its atoms must be 1024-byte aligned
    if (sbase & 1023u) {
        if (threadIdx.x == 0)
            atomicOr(&g_device_error, 32);
        return;
    }
    float *sg = reinterpret_cast<float *>(smem + SC_G);
    float *sbeta = reinterpret_cast<float *>(smem + SC_BETA);
    float *sgam = reinterpret_cast<float *>(smem + SC_GAM);     // Gam, high part
    float *sgaml = reinterpret_cast<float *>(smem + SC_GAML);   // Gam, low part
    float *seg = reinterpret_cast<float *>(smem + SC_EG);
    float *segc = reinterpret_cast<float *>(smem + SC_EGC);
    float *segC = reinterpret_cast<float *>(smem + SC_EGCC);
    int *serr = reinterpret_cast<int *>(smem + SC_ERR);
    const uint32_t mbar = sbase + SC_MBAR;   // four barriers, 8 bytes apart
    float *state_h = a.state + ((size_t)b * a.Hv + h) * kD * kD;

    if (tid == 0) {
        for (int i = 0; i < 4; ++i)
            tc::mbar_init(mbar + 8 * i, 1);
        *serr = 0;
    }
    if (warp == 0)
        tc::tmem_alloc(sbase + SC_TMEM, TM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(smem + SC_TMEM);
    const uint32_t lane_q = (uint32_t)(32 * (warp & 3)) << 16;    // this warp's TMEM lane quarter
    const int jrow = 32 * (warp & 3) + lane;                       // TMEM lane = row index

    // ---- entering state: S^T rows into TMEM (fp32 master) and the bf16 hi/lo tile
    if (warp < 4) {
        const float *src = state_h + (size_t)jrow * kD;
#pragma unroll 1
        for (int c = 0; c < kD; c += 16) {
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 f = __ldg(reinterpret_cast<const float4 *>(src + c + e));
                v[e] = f.x; v[e + 1] = f.y; v[e + 2] = f.z; v[e + 3] = f.w;
            }
            tc::tmem_st16(tmem + lane_q + TM_S + c, v);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float w8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    w8[e] = v[8 * half + e];
                uint4 p1, p2, p3;
                split8x3(w8, p1, p2, p3);
                const uint32_t off = tc::km_offset(jrow, c + 8 * half, kD);
                *reinterpret_cast<uint4 *>(smem + ST_HI + off) = p1;
                *reinterpret_cast<uint4 *>(smem + ST_LO + off) = p2;
                if (kParts == 3)
                    *reinterpret_cast<uint4 *>(smem + ST_3 + off) = p3;
            }
        }
    }

    const float dtv = __ldg(a.dt + h), alog = __ldg(a.A_log + h);
    const TIn *alb = static_cast<const TIn *>(a.alpha) + (int64_t)b * T * a.gate_stride + h;
    const TIn *blb = static_cast<const TIn *>(a.beta_logit) + (int64_t)b * T * a.gate_stride + h;
    const uint32_t id_g = tc::idesc_bf16(128, 64), id_128 = tc::idesc_bf16(128, 128);
    int chunk = 0;

    for (int c0 = 0; c0 < T; c0 += kC, ++chunk) {
        const int n = min(kC, T - c0);
        const uint32_t par = chunk & 1;

        // ---- gate inputs of this chunk (warp 7): requested now, used after warp 7's
        // share of the conv below, so their latency hides under it
        float graw[2] = {0.0f, 0.0f}, braw[2] = {0.0f, 0.0f};
        if (warp == 7) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = 2 * lane + u;
                if (t < n) {
                    graw[u] = load_act<TIn>(alb + (int64_t)(c0 + t) * a.gate_stride);
                    braw[u] = load_act<TIn>(blb + (int64_t)(c0 + t) * a.gate_stride);
                }
            }
        }

        // ---- Q and K rows: conv + SiLU + L2 -> [Q; K] tile, and (e^{Gam_C-Gam} K)^T tile
        {
            const int part = warp >> 2;                         // 0: Q, 1: K
            const int t0 = 16 * (warp & 3) + 8 * (lane >> 4);   // first token (in chunk)
            const int grp = lane & 15;                          // 8-channel group of the head
            const int cb = (part ? a.Hq * kD : 0) + hk * kD + 8 * grp;
            float v[8][8];
            if (a.W == 4 && c0 + t0 >= 3)
                conv8x8_w4_inner<TIn>(a, b, cb, c0 + t0, v);
            else if (a.W == 4)
                conv8x8<TIn, 4>(a, b, cb, c0 + t0, v);
            else
                conv8x8<TIn, 0>(a, b, cb, c0 + t0, v);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                float ss = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    ss = __fmaf_rn(v[t][e], v[t][e], ss);
#pragma unroll
                for (int m = 1; m < 16; m <<= 1)
                    ss += __shfl_xor_sync(0xffffffffu, ss, m);
                const float inv = t0 + t < n ? rsqrtf(ss + a.l2_eps) : 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[t][e] *= inv;
                uint4 p1, p2, p3;
                split8x3(v[t], p1, p2, p3);
                // 128-byte swizzled rows: a quarter-warp's 16-byte stores (8 channel groups
                // of one token row) land on distinct bank groups
                const uint32_t off = tc::sw128_offset(part * kC + t0 + t, 8 * grp, 2 * kC);
                *reinterpret_cast<uint4 *>(smem + QK_HI + off) = p1;
                *reinterpret_cast<uint4 *>(smem + QK_LO + off) = p2;
                if (kParts == 3)
                    *reinterpret_cast<uint4 *>(smem + QK_3 + off) = p3;
            }
        }
        // ---- gates and in-chunk cumulative decay (warp 7); every reader comes after
        // the barrier that ends the conv
        if (warp == 7) {
            float gv[2], bv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = 2 * lane + u;
                gv[u] = t < n ? decay_gate_f(graw[u], dtv, alog) : 0.0f;
                bv[u] = t < n ? sigmoid_f(braw[u]) : 0.0f;
                sg[t] = gv[u];
                sbeta[t] = bv[u];
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
            sgam[2 * lane] = g0h;
            sgaml[2 * lane] = g0l;
            sgam[2 * lane + 1] = g1h;
            sgaml[2 * lane + 1] = g1l;
            seg[2 * lane] = exp_diff(g0h, g0l, 0.0f, 0.0f);
            seg[2 * lane + 1] = exp_diff(g1h, g1l, 0.0f, 0.0f);
            segc[2 * lane] = 2 * lane < n ? exp_diff(gch, gcl, g0h, g0l) : 0.0f;
            segc[2 * lane + 1] = 2 * lane + 1 < n ? exp_diff(gch, gcl, g1h, g1l) : 0.0f;
            if (lane == 0)
                *segC = exp_diff(gch, gcl, 0.0f, 0.0f);
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();

        // ---- G = [Q; K] K^T and KS = S^T [Q; K]^T on the tensor core
        if (tid == 0) {
#pragma unroll 1
            for (int kk = 0; kk < kD / 16; ++kk) {
                // [Q; K] tile: K slice kk at atom column kk / 4, 32 bytes per slice inside it
                const uint32_t kq = (kk >> 2) * (2 * kC * 128) + (kk & 3) * 32;
                const uint64_t a1 = tc::sdesc_sw128(sbase + QK_HI + kq);
                const uint64_t a2 = tc::sdesc_sw128(sbase + QK_LO + kq);
                const uint64_t a3 = tc::sdesc_sw128(sbase + QK_3 + kq);
                const uint64_t b1 = tc::sdesc_sw128(sbase + QK_HI + 8192 + kq);
                const uint64_t b2 = tc::sdesc_sw128(sbase + QK_LO + 8192 + kq);
                const uint64_t b3 = tc::sdesc_sw128(sbase + QK_3 + 8192 + kq);
                tc::mma_bf16(tmem + TM_G, a1, b1, id_g, kk > 0);
                tc::mma_bf16(tmem + TM_G, a1, b2, id_g, 1);
                tc::mma_bf16(tmem + TM_G, a2, b1, id_g, 1);
                if (kParts == 3) {
                    tc::mma_bf16(tmem + TM_G, a1, b3, id_g, 1);
                    tc::mma_bf16(tmem + TM_G, a2, b2, id_g, 1);
                    tc::mma_bf16(tmem + TM_G, a3, b1, id_g, 1);
                }
            }
            tc::mma_commit(mbar + 0);
#pragma unroll 1
            for (int kk = 0; kk < kD / 16; ++kk) {
                const uint32_t ko = kk * 256;
                const uint64_t a1 = tc::sdesc(sbase + ST_HI + ko, 128, 2048);
                const uint64_t a2 = tc::sdesc(sbase + ST_LO + ko, 128, 2048);
                const uint64_t a3 = tc::sdesc(sbase + ST_3 + ko, 128, 2048);
                const uint32_t kq = (kk >> 2) * (2 * kC * 128) + (kk & 3) * 32;
                const uint64_t b1 = tc::sdesc_sw128(sbase + QK_HI + kq);
                const uint64_t b2 = tc::sdesc_sw128(sbase + QK_LO + kq);
                const uint64_t b3 = tc::sdesc_sw128(sbase + QK_3 + kq);
                tc::mma_bf16(tmem + TM_KS, a1, b1, id_128, kk > 0);
                tc::mma_bf16(tmem + TM_KS, a1, b2, id_128, 1);
                tc::mma_bf16(tmem + TM_KS, a2, b1, id_128, 1);
                if (kParts == 3) {
                    tc::mma_bf16(tmem + TM_KS, a1, b3, id_128, 1);
                    tc::mma_bf16(tmem + TM_KS, a2, b2, id_128, 1);
                    tc::mma_bf16(tmem + TM_KS, a3, b1, id_128, 1);
                }
            }
            tc::mma_commit(mbar + 8);
        }

        // ---- V rows: conv + SiLU -> fp32 V^T staged in each value row's X^T footprint.
        // Warps 4-7 do this while the tensor core forms G and KS and warps 0-3 wait
        // for them and build P and A; the X^T/U^T tile is no operand of those products.
        if (warp >= 4) {
            const int t0 = 16 * (warp & 3) + 8 * (lane >> 4);
            const int grp = lane & 15;
            const int cb = 2 * a.Hq * kD + h * kD + 8 * grp;
            float v[8][8];
            if (a.W == 4 && c0 + t0 >= 3)
                conv8x8_w4_inner<TIn>(a, b, cb, c0 + t0, v);
            else if (a.W == 4)
                conv8x8<TIn, 4>(a, b, cb, c0 + t0, v);
            else
                conv8x8<TIn, 0>(a, b, cb, c0 + t0, v);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = 8 * grp + e;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int chunk4 = t0 / 4 + q;     // float4 chunk of the row (0..15)
                    const uint32_t off = foot_off(j, chunk4);
                    *reinterpret_cast<float4 *>(smem + off) =
                        make_float4(v[4 * q][e], v[4 * q + 1][e], v[4 * q + 2][e], v[4 * q + 3][e]);
                }
            }
        }
        // ---- P and A from G. With three parts both products must be done first
        // (their third parts share the space P, T and (e^{Gam_C-Gam} K)^T are written
        // to); with two parts only G is awaited here, and KS before X is formed.
        if (!tc::mbar_wait(mbar + 0, par, kWaitLimit))
            atomicOr(serr, 1);
        if (kParts == 3 && !tc::mbar_wait(mbar + 8, par, kWaitLimit))
            atomicOr(serr, 2);
        tc::fence_after_sync();
        if (warp < 4) {
            const int t = jrow & (kC - 1);
            const bool krow = jrow >= kC;
            const float gt = sgam[t], gtl = sgaml[t];
            const float bt = sbeta[t];
            const int tmax = (warp & 1) ? kC - 1 : kC / 2 - 1;   // largest token of this warp
#pragma unroll 1
            for (int c = 0; c < kC; c += 16) {
                if (c > tmax) {
                    // s > t everywhere in this block: P is zero there (an operand of the
                    // O product), A is never read there
                    if (!krow) {
                        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const uint32_t off = tc::km_offset(t, c + 8 * half, kC);
                            *reinterpret_cast<uint4 *>(smem + PP_HI + off) = zero;
                            *reinterpret_cast<uint4 *>(smem + PP_LO + off) = zero;
                            if (kParts == 3)
                                *reinterpret_cast<uint4 *>(smem + PP_3 + off) = zero;
                        }
                    }
                    continue;
                }
                float gv[16];
                tc::tmem_ld16(tmem + lane_q + TM_G + c, gv);
                float o[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int s = c + e;
                    const bool keep = t < n && (krow ? s < t : s <= t);
                    const float dec = keep ? exp_diff(gt, gtl, sgam[s], sgaml[s]) : 0.0f;
                    o[e] = krow ? bt * dec * gv[e] : dec * gv[e];
                }
                if (krow) {
                    // A, fp32, rows of 16 float4 chunks XOR-swizzled by the row index
                    float *row = reinterpret_cast<float *>(smem + TT_HI + t * 256);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<float4 *>(row + ((((c >> 2) + q) ^ (t & 15)) << 2)) =
                            make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                } else {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float w8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            w8[e] = o[8 * half + e];
                        uint4 p1, p2, p3;
                        split8x3(w8, p1, p2, p3);
                        const uint32_t off = tc::km_offset(t, c + 8 * half, kC);
                        *reinterpret_cast<uint4 *>(smem + PP_HI + off) = p1;
                        *reinterpret_cast<uint4 *>(smem + PP_LO + off) = p2;
                        if (kParts == 3)
                            *reinterpret_cast<uint4 *>(smem + PP_3 + off) = p3;
                    }
                }
            }
        }
        __syncthreads();

        if (warp >= 4) {
            const int tq = tid - 128;
            // ---- (e^{Gam_C-Gam} K)^T from the first two parts of the K rows: key row tq
            for (int t0 = 0; t0 < kC; t0 += 8) {
                float col[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const uint32_t off = tc::sw128_offset(kC + t0 + t, tq, 2 * kC);
                    const float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(smem + QK_HI + off)) +
                                     __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(smem + QK_LO + off));
                    col[t] = kv * segc[t0 + t];
                }
                uint4 hi, lo;
                split8(col, hi, lo);
                const uint32_t off = tc::km_offset(tq, t0, kC);
                *reinterpret_cast<uint4 *>(smem + KT_HI + off) = hi;
                *reinterpret_cast<uint4 *>(smem + KT_LO + off) = lo;
            }
            // ---- state accumulator scaled by e^{Gam_C} ahead of this chunk's update
            const float egC = *segC;
#pragma unroll 1
            for (int c2 = 0; c2 < kD; c2 += 16) {
                float sv[16];
                tc::tmem_ld16(tmem + lane_q + TM_S + c2, sv);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    sv[e] *= egC;
                tc::tmem_st16(tmem + lane_q + TM_S + c2, sv);
            }
        } else {
            if (kParts == 2) {
                if (!tc::mbar_wait(mbar + 8, par, kWaitLimit))
                    atomicOr(serr, 2);
                tc::fence_after_sync();
            }
            // ---- (Q S_0)^T scaled by e^{Gam}; X^T = beta V^T - beta e^{Gam} (K S_0)^T
#pragma unroll 1
            for (int c = 0; c < kC; c += 16) {
                float qv[16];
                tc::tmem_ld16(tmem + lane_q + TM_KS + c, qv);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    qv[e] *= seg[c + e];
                tc::tmem_st16(tmem + lane_q + TM_KS + c, qv);
            }
            // X^T row j = beta V^T - beta e^{Gam} (K S_0)^T, in registers (V^T was staged in
            // this thread's own footprint of the X^T/U^T tile)
            float xv[kC];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 f = *reinterpret_cast<const float4 *>(smem + foot_off(jrow, q));
                xv[4 * q] = f.x; xv[4 * q + 1] = f.y; xv[4 * q + 2] = f.z; xv[4 * q + 3] = f.w;
            }
#pragma unroll
            for (int c = 0; c < kC; c += 16) {
                float kv[16];
                tc::tmem_ld16(tmem + lane_q + TM_KS + kC + c, kv);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float bt = sbeta[c + e];
                    xv[c + e] = bt * xv[c + e] - bt * seg[c + e] * kv[e];
                }
            }
            // U = (I + A)^{-1} X by blocks of kSB tokens: (I + A) is unit lower triangular,
            // so u_t = x_t - sum_{s<t} A[t][s] u_s. Block b first takes the contributions
            // of the earlier blocks (their u read back from this thread's own footprint of
            // the X^T/U^T tile), then solves its diagonal block in registers. Rows of
            // A (fp32, XOR-swizzled float4 chunks) are read as broadcasts. The loops stay
            // rolled: the fully unrolled substitution did not fit the instruction cache.
            const float *Af = reinterpret_cast<const float *>(smem + TT_HI);
            auto ufoot = [&](int q) { return reinterpret_cast<float4 *>(smem + foot_off(jrow, q)); };
#pragma unroll
            for (int q = 0; q < 16; ++q)
                *ufoot(q) = make_float4(xv[4 * q], xv[4 * q + 1], xv[4 * q + 2], xv[4 * q + 3]);
#pragma unroll 1
            for (int b = 0; b < kC / kSB; ++b) {
                float acc0[kSB], acc1[kSB];
#pragma unroll
                for (int t = 0; t < kSB; ++t)
                    acc0[t] = acc1[t] = 0.0f;
#pragma unroll 1
                for (int sb = 0; sb < b; ++sb) {
                    float4 u4[kSB / 4];
#pragma unroll
                    for (int q = 0; q < kSB / 4; ++q)
                        u4[q] = *ufoot(sb * (kSB / 4) + q);
#pragma unroll
                    for (int t = 0; t < kSB; ++t) {
                        const int row = kSB * b + t;
                        const float *arow = Af + row * kC;
#pragma unroll
                        for (int q = 0; q < kSB / 4; ++q) {
                            const float4 a4 = *reinterpret_cast<const float4 *>(
                                arow + (((sb * (kSB / 4) + q) ^ (row & 15)) << 2));
                            acc0[t] = __fmaf_rn(a4.x, u4[q].x, acc0[t]);
                            acc1[t] = __fmaf_rn(a4.y, u4[q].y, acc1[t]);
                            acc0[t] = __fmaf_rn(a4.z, u4[q].z, acc0[t]);
                            acc1[t] = __fmaf_rn(a4.w, u4[q].w, acc1[t]);
                        }
                    }
                }
                float x[kSB];
#pragma unroll
                for (int q = 0; q < kSB / 4; ++q) {
                    const float4 f = *ufoot(b * (kSB / 4) + q);
                    x[4 * q] = f.x; x[4 * q + 1] = f.y; x[4 * q + 2] = f.z; x[4 * q + 3] = f.w;
                }
#pragma unroll
                for (int t = 0; t < kSB; ++t) {
                    const int row = kSB * b + t;
                    const float *arow = Af + row * kC;
                    float ad[kSB];
#pragma unroll
                    for (int q = 0; q < kSB / 4; ++q) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(
                            arow + (((b * (kSB / 4) + q) ^ (row & 15)) << 2));
                        ad[4 * q] = a4.x; ad[4 * q + 1] = a4.y; ad[4 * q + 2] = a4.z; ad[4 * q + 3] = a4.w;
                    }
                    float acc = __fadd_rn(acc0[t], acc1[t]);
#pragma unroll
                    for (int s2 = 0; s2 < t; ++s2)
                        acc = __fmaf_rn(ad[s2], x[s2], acc);
                    x[t] = __fsub_rn(x[t], acc);
                }
#pragma unroll
                for (int q = 0; q < kSB / 4; ++q)
                    *ufoot(b * (kSB / 4) + q) = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
            }
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 f = *ufoot(q);
                xv[4 * q] = f.x; xv[4 * q + 1] = f.y; xv[4 * q + 2] = f.z; xv[4 * q + 3] = f.w;
            }
            // U^T row j as the two-part operand of the O and state products; every row
            // of warps 0-3 has read its fp32 footprint back first (named barrier 1)
            asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll
            for (int c = 0; c < kC; c += 8) {
                float u8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    u8[e] = xv[c + e];
                uint4 p1, p2, p3;
                split8x3(u8, p1, p2, p3);
                const uint32_t off = tc::km_offset(jrow, c, kC);
                *reinterpret_cast<uint4 *>(smem + XU_HI + off) = p1;
                *reinterpret_cast<uint4 *>(smem + XU_LO + off) = p2;
                if (kParts == 3)
                    *reinterpret_cast<uint4 *>(smem + XU_3 + off) = p3;
            }
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();

        // ---- O^T += U^T P^T;  S^T += U^T (e^{Gam_C-Gam} K)
        if (tid == 0) {
#pragma unroll 1
            for (int kk = 0; kk < kC / 16; ++kk) {
                const uint32_t ko = kk * 256;
                const uint64_t ah = tc::sdesc(sbase + XU_HI + ko, 128, 1024);
                const uint64_t al = tc::sdesc(sbase + XU_LO + ko, 128, 1024);
                const uint64_t a3 = tc::sdesc(sbase + XU_3 + ko, 128, 1024);
                const uint64_t ph = tc::sdesc(sbase + PP_HI + ko, 128, 1024);
                const uint64_t pl = tc::sdesc(sbase + PP_LO + ko, 128, 1024);
                const uint64_t p3 = tc::sdesc(sbase + PP_3 + ko, 128, 1024);
                const uint64_t kh = tc::sdesc(sbase + KT_HI + ko, 128, 1024);
                const uint64_t kl = tc::sdesc(sbase + KT_LO + ko, 128, 1024);
                tc::mma_bf16(tmem + TM_KS, ah, ph, id_g, 1);
                tc::mma_bf16(tmem + TM_KS, ah, pl, id_g, 1);
                tc::mma_bf16(tmem + TM_KS, al, ph, id_g, 1);
                if (kParts == 3) {
                    tc::mma_bf16(tmem + TM_KS, ah, p3, id_g, 1);
                    tc::mma_bf16(tmem + TM_KS, al, pl, id_g, 1);
                    tc::mma_bf16(tmem + TM_KS, a3, ph, id_g, 1);
                }
                tc::mma_bf16(tmem + TM_S, ah, kh, id_128, 1);
                tc::mma_bf16(tmem + TM_S, ah, kl, id_128, 1);
                tc::mma_bf16(tmem + TM_S, al, kh, id_128, 1);
            }
            tc::mma_commit(mbar + 24);
        }
        // this chunk's z values for the gated norm (warp w: tokens w, w+8, ...), requested
        // now so that their latency hides under the products
        float zv[kC / 8][4];
        {
            const TIn *zb = static_cast<const TIn *>(a.z) + (int64_t)b * T * a.z_stride + (int64_t)h * kD;
#pragma unroll
            for (int i = 0; i < kC / 8; ++i) {
                const int t = warp + 8 * i;
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    zv[i][m] = t < n ? load_act<TIn>(zb + ((int64_t)c0 + t) * a.z_stride + 32 * m + lane) : 0.0f;
            }
        }
        if (!tc::mbar_wait(mbar + 24, par, kWaitLimit))
            atomicOr(serr, 8);
        tc::fence_after_sync();
        if (warp < 4) {
            // O (fp32, [t][j]) into the XU region for the row-wise norm
            float *O = reinterpret_cast<float *>(smem + XU_HI);
#pragma unroll 1
            for (int c = 0; c < kC; c += 16) {
                float ov[16];
                tc::tmem_ld16(tmem + lane_q + TM_KS + c, ov);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    O[(c + e) * kD + jrow] = ov[e];
            }
        } else {
            // next chunk's S^T operand (three parts) from the updated state
#pragma unroll 1
            for (int c = 0; c < kD; c += 16) {
                float sv[16];
                tc::tmem_ld16(tmem + lane_q + TM_S + c, sv);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float s8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        s8[e] = sv[8 * half + e];
                    uint4 p1, p2, p3;
                    split8x3(s8, p1, p2, p3);
                    const uint32_t off = tc::km_offset(jrow, c + 8 * half, kD);
                    *reinterpret_cast<uint4 *>(smem + ST_HI + off) = p1;
                    *reinterpret_cast<uint4 *>(smem + ST_LO + off) = p2;
                    if (kParts == 3)
                        *reinterpret_cast<uint4 *>(smem + ST_3 + off) = p3;
                }
            }
        }
        __syncthreads();

        // ---- gated RMSNorm of each token's output row (warp w: tokens w, w+8, ...)
        {
            const float *O = reinterpret_cast<const float *>(smem + XU_HI);
            float nwv[4];
#pragma unroll
            for (int m = 0; m < 4; ++m)
                nwv[m] = __ldg(a.norm_w + 32 * m + lane);
#pragma unroll
            for (int i = 0; i < kC / 8; ++i) {
                const int t = warp + 8 * i;
                if (t >= n)
                    break;
                float yv[4], bp[4];
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    yv[m] = O[t * kD + 32 * m + lane] * a.scale;
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    bp[m] = norm_block_partial(yv[m]);
                const float inv = norm_inv(bp[0], bp[1], bp[2], bp[3], a.rms_eps);
                float *outr = a.out + (((size_t)b * T + c0 + t) * a.Hv + h) * kD;
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    outr[32 * m + lane] = gated_out(yv[m], inv, nwv[m], zv[i][m]);
            }
        }
        __syncthreads();
        if (*serr)
            break;
    }

    // ---- final state back to HBM (S^T rows = the library layout)
    tc::fence_after_sync();
    if (warp < 4 && *serr == 0) {
        float *dst = state_h + (size_t)jrow * kD;
#pragma unroll 1
        for (int c = 0; c < kD; c += 16) {
            float v[16];
            tc::tmem_ld16(tmem + lane_q + TM_S + c, v);
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4 *>(dst + c + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
    }
    if (*serr) {
        if (tid == 0)
            atomicOr(&g_device_error, *serr);
        // MMAs may still be in flight: a second bounded chance for every barrier
        // before TMEM is released
        for (int i = 0; i < 4; ++i)
            if (i != 2)   // barrier 2 is not used
                tc::mbar_wait(mbar + 8 * i, (chunk & 1), kWaitLimit);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0)
        tc::tmem_dealloc(tmem, TM_COLS);
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

template <typename TIn>
cudaError_t prefill_typed(const PrefillArgs &a, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<TIn>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    prefill_tc_kernel<TIn><<<dim3(a.Hv, a.B, 1), kThreads, SMEM_BYTES, s>>>(a);
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

cudaError_t launch_prefill_tc(const PrefillArgs &a, bool bf16, cudaStream_t s)
{
    return bf16 ? prefill_typed<__nv_bfloat16>(a, s) : prefill_typed<float>(a, s);
}

}  // namespace gdn
