// prefill.cu -- chunked prefill of the gated-delta layer (fp32, CUDA cores).
//
// One CTA per (sequence, V head) walks the sequence in 64-token chunks with
// the 128x128 state resident in shared memory; nothing is staged through
// global memory between the phases of a chunk. The chunk algebra (plain
// orientation S[i][j], Gam_t = g_1 + ... + g_t inside the chunk, S_0 the state
// entering it) follows from the recurrence of "fm_kernel_ssm.h" section
// "Delta-rule recurrence" alone; the 64-token chunks joined by ceil(T/64)
// sequential links follow the "Mamba-2 SSD chunked prefill scan" note of
// "ssm_mamba.rs":
//   A[t][s] = beta_t e^{Gam_t - Gam_s} (k_t . k_s)        s < t
//   X       = diag(beta) V - diag(beta e^{Gam}) K S_0
//   U       = (I + A)^{-1} X                            forward substitution
//   O       = scale (diag(e^{Gam}) Q S_0 + P U),  P[t][s] = e^{Gam_t - Gam_s} (q_t . k_s), s <= t
//   S_C     = e^{Gam_C} S_0 + K^T diag(e^{Gam_C - Gam}) U
// then the gated RMSNorm of every token's O row. The conv + SiLU + L2 and the
// gates of the chunk's tokens are computed in the same CTA from the raw
// inputs; the conv history is rewritten by a second small kernel once every
// CTA has read it.
#include "gdn_device.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kC = 64;          // chunk length
constexpr int kLdQK = kD + 4;   // padded row stride of Q, K (float4 rows stay aligned)
constexpr int kLdP = kC + 4;    // padded row stride of A, P
constexpr int kThreads = 256;

struct PrefillSmem {
    float S[kD * kD];           // S[i][j]
    float Q[kC * kLdQK];        // Q[t][i]; reused for O[t][j]
    float K[kC * kLdQK];        // K[t][i]
    float V[kC * kD];           // V[t][j] -> X -> U -> e^{Gam_C - Gam_t} U
    float A[kC * kLdP];         // strictly lower (I + A) part
    float P[kC * kLdP];         // lower-triangular decayed Q K^T
    float g[kC], beta[kC], gam[kC], eg[kC], egc[kC];
    float egC;
};

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ float at(const float4 &v, int e)
{
    return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads, 1) prefill_chunk_kernel(PrefillArgs a)
{
    extern __shared__ __align__(16) float smem_raw[];
    PrefillSmem &sm = *reinterpret_cast<PrefillSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ty = tid >> 4, tx = tid & 15;
    const int b = blockIdx.y, h = blockIdx.x;
    const int hk = h / (a.Hv / a.Hq);
    const int W = a.W, cd = a.conv_dim, T = a.T;
    const TIn *xb = static_cast<const TIn *>(a.x) + (int64_t)b * T * a.x_stride;
    const TIn *zb = static_cast<const TIn *>(a.z) + (int64_t)b * T * a.z_stride;
    const TIn *alb = static_cast<const TIn *>(a.alpha) + (int64_t)b * T * a.gate_stride;
    const TIn *blb = static_cast<const TIn *>(a.beta_logit) + (int64_t)b * T * a.gate_stride;
    const float *histb = a.conv_state + (size_t)b * cd * (W - 1);
    float *state_h = a.state + ((size_t)b * a.Hv + h) * kD * kD;
    const float dtv = __ldg(a.dt + h), alog = __ldg(a.A_log + h);

    // load S (library layout [j][i]) into S[i][j]
    for (int idx = tid; idx < kD * kD; idx += kThreads) {
        const int j = idx >> 7, i = idx & (kD - 1);
        sm.S[i * kD + j] = state_h[idx];
    }

    for (int c0 = 0; c0 < T; c0 += kC) {
        const int n = min(kC, T - c0);
        // ---- conv + SiLU for the chunk's q, k (head hk) and v (head h) channels; gates
        for (int idx = tid; idx < kC * 3 * kD; idx += kThreads) {
            const int t = idx / (3 * kD), ch = idx % (3 * kD);
            int c;
            float *dst;
            if (ch < kD) {
                c = hk * kD + ch;
                dst = &sm.Q[t * kLdQK + ch];
            } else if (ch < 2 * kD) {
                c = a.Hq * kD + hk * kD + (ch - kD);
                dst = &sm.K[t * kLdQK + (ch - kD)];
            } else {
                c = 2 * a.Hq * kD + h * kD + (ch - 2 * kD);
                dst = &sm.V[t * kD + (ch - 2 * kD)];
            }
            float v = 0.0f;
            if (t < n)
                v = silu_f(conv_pre<TIn>(histb + (size_t)c * (W - 1), xb + c, a.x_stride,
                                         a.conv_w + (size_t)c * W, W, c0 + t));
            *dst = v;
        }
        if (tid < kC) {
            const int t = tid;
            float gv = 0.0f, bv = 0.0f;
            if (t < n) {
                const int64_t row = c0 + t;
                gv = decay_gate_f(load_act<TIn>(alb + row * a.gate_stride + h), dtv, alog);
                bv = sigmoid_f(load_act<TIn>(blb + row * a.gate_stride + h));
            }
            sm.g[t] = gv;
            sm.beta[t] = bv;
        }
        __syncthreads();

        // ---- L2 norm of the Q and K rows; cumulative decay
        for (int rr = warp; rr < 2 * kC; rr += 8) {
            if ((rr & (kC - 1)) >= n)
                continue;   // tail rows stay zero
            float *row = rr < kC ? &sm.Q[rr * kLdQK] : &sm.K[(rr - kC) * kLdQK];
            float v[4];
            float s = 0.0f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                v[m] = row[lane + 32 * m];
                s = __fmaf_rn(v[m], v[m], s);
            }
            const float inv = rsqrtf(__fadd_rn(warp_sum32(s), a.l2_eps));
#pragma unroll
            for (int m = 0; m < 4; ++m)
                row[lane + 32 * m] = __fmul_rn(v[m], inv);
        }
        if (warp == 0) {
            const float g0 = sm.g[2 * lane], g1 = sm.g[2 * lane + 1];
            float s = __fadd_rn(g0, g1);
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off)
                    s = __fadd_rn(s, y);
            }
            float ex = __shfl_up_sync(0xffffffffu, s, 1);
            if (lane == 0)
                ex = 0.0f;
            const float G0 = __fadd_rn(ex, g0);
            const float G1 = __fadd_rn(G0, g1);
            const float GC = __shfl_sync(0xffffffffu, G1, 31);
            sm.gam[2 * lane] = G0;
            sm.gam[2 * lane + 1] = G1;
            sm.eg[2 * lane] = expf(G0);
            sm.eg[2 * lane + 1] = expf(G1);
            sm.egc[2 * lane] = 2 * lane < n ? expf(__fsub_rn(GC, G0)) : 0.0f;
            sm.egc[2 * lane + 1] = 2 * lane + 1 < n ? expf(__fsub_rn(GC, G1)) : 0.0f;
            if (lane == 0)
                sm.egC = expf(GC);
        }
        __syncthreads();

        // ---- A (strictly lower, beta-scaled) and P (lower incl. diagonal)
        {
            float kk[4][4], qk[4][4];
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y)
                    kk[x][y] = qk[x][y] = 0.0f;
            for (int i = 0; i < kD; i += 4) {
                float4 kt[4], qt[4], ks[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    kt[x] = ld4(&sm.K[(ty + 16 * x) * kLdQK + i]);
                    qt[x] = ld4(&sm.Q[(ty + 16 * x) * kLdQK + i]);
                    ks[x] = ld4(&sm.K[(tx + 16 * x) * kLdQK + i]);
                }
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int y = 0; y < 4; ++y)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            kk[x][y] = __fmaf_rn(at(kt[x], e), at(ks[y], e), kk[x][y]);
                            qk[x][y] = __fmaf_rn(at(qt[x], e), at(ks[y], e), qk[x][y]);
                        }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) {
                    const int t = ty + 16 * x, s = tx + 16 * y;
                    const float dec = s <= t && t < n ? expf(__fsub_rn(sm.gam[t], sm.gam[s])) : 0.0f;
                    sm.A[t * kLdP + s] = s < t ? __fmul_rn(__fmul_rn(sm.beta[t], dec), kk[x][y]) : 0.0f;
                    sm.P[t * kLdP + s] = __fmul_rn(dec, qk[x][y]);
                }
        }

        // ---- X = beta V - beta e^{Gam} (K S_0), into V
        {
            float acc[4][8];
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 8; ++y)
                    acc[x][y] = 0.0f;
            for (int i = 0; i < kD; i += 4) {
                float4 kt[4];
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    kt[x] = ld4(&sm.K[(ty + 16 * x) * kLdQK + i]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 s0 = ld4(&sm.S[(i + e) * kD + 4 * tx]);
                    const float4 s1 = ld4(&sm.S[(i + e) * kD + 64 + 4 * tx]);
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float kv = at(kt[x], e);
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            acc[x][f] = __fmaf_rn(kv, at(s0, f), acc[x][f]);
                            acc[x][4 + f] = __fmaf_rn(kv, at(s1, f), acc[x][4 + f]);
                        }
                    }
                }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int t = ty + 16 * x;
                const float bt = sm.beta[t];
                const float be = __fmul_rn(bt, sm.eg[t]);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float *vp = &sm.V[t * kD + 64 * half + 4 * tx];
                    float4 v = ld4(vp);
                    v.x = __fsub_rn(__fmul_rn(bt, v.x), __fmul_rn(be, acc[x][4 * half + 0]));
                    v.y = __fsub_rn(__fmul_rn(bt, v.y), __fmul_rn(be, acc[x][4 * half + 1]));
                    v.z = __fsub_rn(__fmul_rn(bt, v.z), __fmul_rn(be, acc[x][4 * half + 2]));
                    v.w = __fsub_rn(__fmul_rn(bt, v.w), __fmul_rn(be, acc[x][4 * half + 3]));
                    st4(vp, v);
                }
            }
        }
        __syncthreads();

        // ---- U = (I + A)^{-1} X: forward substitution, one thread per value column
        if (tid < kD) {
            const int j = tid;
            for (int t = 1; t < n; ++t) {
                float s0 = 0.0f, s1 = 0.0f;
                int s = 0;
                for (; s + 1 < t; s += 2) {
                    s0 = __fmaf_rn(sm.A[t * kLdP + s], sm.V[s * kD + j], s0);
                    s1 = __fmaf_rn(sm.A[t * kLdP + s + 1], sm.V[(s + 1) * kD + j], s1);
                }
                if (s < t)
                    s0 = __fmaf_rn(sm.A[t * kLdP + s], sm.V[s * kD + j], s0);
                sm.V[t * kD + j] = __fsub_rn(sm.V[t * kD + j], __fadd_rn(s0, s1));
            }
        }
        __syncthreads();

        // ---- O = scale (e^{Gam} Q S_0 + P U)
        float o[4][8];
        {
            float acc[4][8];
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 8; ++y)
                    acc[x][y] = o[x][y] = 0.0f;
            for (int i = 0; i < kD; i += 4) {
                float4 qt[4];
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    qt[x] = ld4(&sm.Q[(ty + 16 * x) * kLdQK + i]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 s0 = ld4(&sm.S[(i + e) * kD + 4 * tx]);
                    const float4 s1 = ld4(&sm.S[(i + e) * kD + 64 + 4 * tx]);
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float qv = at(qt[x], e);
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            acc[x][f] = __fmaf_rn(qv, at(s0, f), acc[x][f]);
                            acc[x][4 + f] = __fmaf_rn(qv, at(s1, f), acc[x][4 + f]);
                        }
                    }
                }
            }
            for (int s = 0; s < kC; s += 4) {
                float4 pt[4];
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    pt[x] = ld4(&sm.P[(ty + 16 * x) * kLdP + s]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 u0 = ld4(&sm.V[(s + e) * kD + 4 * tx]);
                    const float4 u1 = ld4(&sm.V[(s + e) * kD + 64 + 4 * tx]);
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float pv = at(pt[x], e);
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            o[x][f] = __fmaf_rn(pv, at(u0, f), o[x][f]);
                            o[x][4 + f] = __fmaf_rn(pv, at(u1, f), o[x][4 + f]);
                        }
                    }
                }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float e = sm.eg[ty + 16 * x];
#pragma unroll
                for (int y = 0; y < 8; ++y)
                    o[x][y] = __fmul_rn(a.scale, __fmaf_rn(e, acc[x][y], o[x][y]));
            }
        }
        __syncthreads();   // every read of Q is done: O goes into Q's rows
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int half = 0; half < 2; ++half)
                st4(&sm.Q[(ty + 16 * x) * kLdQK + 64 * half + 4 * tx],
                    make_float4(o[x][4 * half], o[x][4 * half + 1], o[x][4 * half + 2], o[x][4 * half + 3]));
        // U rows scaled by e^{Gam_C - Gam_t} for the state update
        for (int idx = tid; idx < kC * kD / 4; idx += kThreads) {
            const int t = idx / (kD / 4);
            float4 u = ld4(&sm.V[idx * 4]);
            const float e = sm.egc[t];
            u.x = __fmul_rn(u.x, e);
            u.y = __fmul_rn(u.y, e);
            u.z = __fmul_rn(u.z, e);
            u.w = __fmul_rn(u.w, e);
            st4(&sm.V[idx * 4], u);
        }
        __syncthreads();

        // ---- gated RMSNorm of each token's O row -> out
        for (int t = warp; t < n; t += 8) {
            const float *orow = &sm.Q[t * kLdQK];
            float yv[4], bp[4];
#pragma unroll
            for (int m = 0; m < 4; ++m)
                yv[m] = orow[32 * m + lane];
#pragma unroll
            for (int m = 0; m < 4; ++m)
                bp[m] = norm_block_partial(yv[m]);
            const float inv = norm_inv(bp[0], bp[1], bp[2], bp[3], a.rms_eps);
            const int64_t row = (int64_t)c0 + t;
            const TIn *zr = zb + row * a.z_stride + (int64_t)h * kD;
            float *outr = a.out + (((size_t)b * T + row) * a.Hv + h) * kD;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int j = 32 * m + lane;
                outr[j] = gated_out(yv[m], inv, __ldg(a.norm_w + j), load_act<TIn>(zr + j));
            }
        }

        // ---- S <- e^{Gam_C} S + K^T (e^{Gam_C - Gam} U)
        {
            float acc[8][8];
#pragma unroll
            for (int x = 0; x < 8; ++x)
#pragma unroll
                for (int y = 0; y < 8; ++y)
                    acc[x][y] = 0.0f;
            for (int t = 0; t < n; ++t) {
                const float4 k0 = ld4(&sm.K[t * kLdQK + 8 * ty]);
                const float4 k1 = ld4(&sm.K[t * kLdQK + 8 * ty + 4]);
                const float4 u0 = ld4(&sm.V[t * kD + 4 * tx]);
                const float4 u1 = ld4(&sm.V[t * kD + 64 + 4 * tx]);
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const float kv = x < 4 ? at(k0, x) : at(k1, x - 4);
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        acc[x][f] = __fmaf_rn(kv, at(u0, f), acc[x][f]);
                        acc[x][4 + f] = __fmaf_rn(kv, at(u1, f), acc[x][4 + f]);
                    }
                }
            }
            const float egC = sm.egC;
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const int i = 8 * ty + x;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float *sp = &sm.S[i * kD + 64 * half + 4 * tx];
                    float4 s = ld4(sp);
                    s.x = __fmaf_rn(egC, s.x, acc[x][4 * half + 0]);
                    s.y = __fmaf_rn(egC, s.y, acc[x][4 * half + 1]);
                    s.z = __fmaf_rn(egC, s.z, acc[x][4 * half + 2]);
                    s.w = __fmaf_rn(egC, s.w, acc[x][4 * half + 3]);
                    st4(sp, s);
                }
            }
        }
        __syncthreads();
    }

    // store S back in the library layout
    for (int idx = tid; idx < kD * kD; idx += kThreads) {
        const int j = idx >> 7, i = idx & (kD - 1);
        state_h[idx] = sm.S[i * kD + j];
    }
}

// Rewrites every channel's history with the last W-1 raw inputs of the call
// (or the older history when the call had fewer tokens). Runs after the chunk
// kernel, which reads the old history.
template <typename TIn>
__global__ void __launch_bounds__(256) prefill_history_kernel_simt(float *conv_state, const TIn *x,
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
    const size_t smem = sizeof(PrefillSmem);
    cudaError_t e = cudaFuncSetAttribute(prefill_chunk_kernel<TIn>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    prefill_chunk_kernel<TIn><<<dim3(a.Hv, a.B, 1), kThreads, smem, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    prefill_history_kernel_simt<TIn><<<dim3((a.conv_dim + 255) / 256, a.B, 1), 256, 0, s>>>(
        a.conv_state, static_cast<const TIn *>(a.x), a.x_stride, a.conv_dim, a.W, a.T);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs &a, bool bf16, cudaStream_t s)
{
    return bf16 ? prefill_typed<__nv_bfloat16>(a, s) : prefill_typed<float>(a, s);
}

cudaError_t launch_prefill(const PrefillArgs &a, bool bf16, cudaStream_t s)
{
#ifdef GDN_PREFILL_SIMT
    return launch_prefill_simt(a, bf16, s);
#else
    return launch_prefill_tc(a, bf16, s);
#endif
}

}  // namespace gdn
