// conv.cu -- the standalone causal depthwise conv1d + SiLU with the per-head
// L2 norm of the Q and K channels ("fm_kernel_ssm.h", "Causal depthwise
// conv1d + SiLU"; "ssm_mamba.rs", conv1d_update_l2norm), over n tokens of
// every sequence.
//
// One token: the serial kernel (one thread per channel). Several tokens: a
// token-parallel kernel. The conv is a sliding window over INPUTS, so no
// output depends on another ("ssm_mamba.rs", the token-parallel prefill
// conv1d note); each output is the same tap sum in the same order and each
// head's L2 sum the same reduction tree, so all three kernels agree bit for
// bit. The tiled kernel (TMA-staged tiles, persistent CTAs) is used whenever
// the input rows meet the tensor-copy alignment; the token kernel (plain
// loads) covers the rest.
#include <algorithm>

#include "gdn_device.cuh"
#include "gdn_kernels.h"
#include "tc_ptx.cuh"
#include "tma_map.cuh"

namespace gdn {

// Bit 64: a wait of the tiled conv kernel for its tile copy gave up (that CTA
// stopped). Read and cleared by take_conv_device_error.
static __device__ int g_conv_error;
constexpr int kErrConvWait = 64;

namespace {

// One CTA of 128 threads per (128-channel head, sequence); thread i owns
// channel i of the head and scans the tokens of the call in order.
template <typename TIn>
__global__ void __launch_bounds__(kD) conv_update_kernel(ConvArgs a)
{
    __shared__ float red[2][4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.y;
    const int c = blockIdx.x * kD + tid;
    const bool is_qk = blockIdx.x < 2 * a.Hq;
    const int W = a.W;
    GDN_CHECK(g_conv_error, b < a.B && c < a.conv_dim);
    float *hist_c = a.conv_state + ((size_t)b * a.conv_dim + c) * (W - 1);
    const TIn *x_c = static_cast<const TIn *>(a.x) + (int64_t)b * a.T * a.x_stride + c;
    const float *w_c = a.conv_w + (size_t)c * W;
    float *out_c = a.out + (size_t)b * a.T * a.conv_dim + c;
    for (int t = 0; t < a.T; ++t) {
        float v = silu_f(conv_pre<TIn>(hist_c, x_c, a.x_stride, w_c, W, t));
        if (is_qk)
            v = __fmul_rn(v, head_l2_inv(v, a.l2_eps, red[t & 1], warp, lane));
        out_c[(size_t)t * a.conv_dim] = v;
    }
    float nh[kMaxW - 1];
    conv_history_after<TIn>(hist_c, x_c, a.x_stride, W, a.T, nh);
    store_history(hist_c, W, nh);
}

// Token-parallel form: one CTA of 256 threads per (128-channel head, tile of
// 2*TPT tokens, sequence). Thread (tg, i), tg = tid / 128, owns channel i of
// the head for the TPT tokens from t0 = tile*2*TPT + tg*TPT. Its window of
// TPT + W - 1 stream values (history entries for stream index < 0, raw
// inputs after) is loaded once, all loads independent; a warp's loads of one
// token are 32 consecutive channels. Only the first token group of the first
// tile reaches back into the history (TPT >= W - 1), and that group alone
// rewrites it, after its own reads: no other CTA touches the history.
template <typename TIn, int TPT>
__global__ void __launch_bounds__(256) conv_tokens_kernel(ConvArgs a)
{
    static_assert(TPT >= kMaxW - 1, "only token group 0 of tile 0 may read the history");
    constexpr int NWIN = kMaxW - 1 + TPT;
    __shared__ float red[2][TPT][4];
    const int tid = threadIdx.x, lane = tid & 31;
    const int i = tid & (kD - 1), tg = tid >> 7, wih = (tid >> 5) & 3;
    const int b = blockIdx.z;
    const int c = blockIdx.x * kD + i;
    const bool is_qk = blockIdx.x < 2 * a.Hq;
    const int W = a.W, T = a.T;
    const int t0 = (blockIdx.y * 2 + tg) * TPT;
    GDN_CHECK(g_conv_error, b < a.B && c < a.conv_dim && blockIdx.y * 2 * TPT < T);
    float *hist_c = a.conv_state + ((size_t)b * a.conv_dim + c) * (W - 1);
    const TIn *x_c = static_cast<const TIn *>(a.x) + (int64_t)b * T * a.x_stride + c;

    float w[kMaxW];
#pragma unroll
    for (int tau = 0; tau < kMaxW; ++tau)
        w[tau] = tau < W ? __ldg(a.conv_w + (size_t)c * W + tau) : 0.0f;
    // win[e] = stream value at index t0 - (W-1) + e
    float win[NWIN];
#pragma unroll
    for (int e = 0; e < NWIN; ++e) {
        const int s = t0 - (W - 1) + e;
        float v = 0.0f;
        if (e < W - 1 + TPT) {
            if (s < 0)
                v = hist_c[W - 1 + s];
            else if (s < T)
                v = load_act<TIn>(x_c + (int64_t)s * a.x_stride);
        }
        win[e] = v;
    }

    // token t0 + p: taps over win[p .. p+W-1], oldest first (conv_pre's order)
    float v[TPT];
#pragma unroll
    for (int p = 0; p < TPT; ++p) {
        float acc = __fmul_rn(win[p], w[0]);
#pragma unroll
        for (int tau = 1; tau < kMaxW; ++tau)
            if (tau < W)
                acc = __fmaf_rn(win[p + tau], w[tau], acc);
        v[p] = silu_f(acc);
    }
    if (is_qk) {   // uniform over the CTA
#pragma unroll
        for (int p = 0; p < TPT; ++p) {
            const float s2 = warp_sum32(__fmul_rn(v[p], v[p]));
            if (lane == 0)
                red[tg][p][wih] = s2;
        }
        __syncthreads();
#pragma unroll
        for (int p = 0; p < TPT; ++p)
            v[p] = __fmul_rn(v[p], l2_inv_of_partials(red[tg][p], a.l2_eps));
    }
    float *out_c = a.out + (size_t)b * T * a.conv_dim + c;
#pragma unroll
    for (int p = 0; p < TPT; ++p)
        if (t0 + p < T)
            out_c[(size_t)(t0 + p) * a.conv_dim] = v[p];

    if (t0 == 0) {
        float nh[kMaxW - 1];
        conv_history_after<TIn>(hist_c, x_c, a.x_stride, W, T, nh);
        store_history(hist_c, W, nh);
    }
}

constexpr int kTokensPerThread = 16;

// ------------------------------------------------------------------ tiled form
// Work item = (sequence b, 128-channel head, tile of kTT tokens), numbered
// head-fastest so that the CTAs in flight read neighbouring tiles of the same
// token rows. Each persistent CTA walks items gridDim.x apart; while it
// computes one item, the tensor copy of its next item's input rows
// (tokens t0-(W-1) .. t0+kTT-1, all 128 channels; rows before the sequence
// start or past its end arrive as zeros) lands in the other buffer.
//
// Thread (tg, i) = (tid / 128, tid % 128) computes channel i for the 32
// tokens t0 + 32 tg + p. The Q/K L2 sum of a token is formed in the order of
// a 32-lane xor butterfly (warp_sum32) per 32-channel group, here evaluated
// by one lane per token from shared memory: pairs 16 apart, then 8, 4, 2, 1;
// then the four group sums in order, as in head_l2_inv.
constexpr int kTT = 64;
constexpr int kTileRows = kTT + kMaxW - 1;
// Row stride of the per-warp squares buffer: 16-byte rows for vector reads,
// and 36 mod 32 = 4 keeps each quarter-warp's 16-byte reads on distinct banks.
constexpr int kSqStride = 36;

template <typename TIn>
struct TileLayout {
    static constexpr uint32_t tile = (kTileRows * kD * sizeof(TIn) + 1023) / 1024 * 1024;
    static constexpr uint32_t sq = 2 * tile;                   // [8 warps][32 tokens][36] float
    static constexpr uint32_t part = sq + 8 * 32 * 36 * 4;     // [2 tg][32 tokens][4 groups] float
    static constexpr uint32_t mbar = part + 2 * 32 * 4 * 4;    // two mbarriers
    static constexpr uint32_t flag = mbar + 16;
    static constexpr uint32_t bytes = flag + 16 + 1024;        // + alignment slack
};

template <typename TIn>
__device__ __forceinline__ float smem_act(const TIn *p);
template <>
__device__ __forceinline__ float smem_act<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float smem_act<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat162float(*p);
}

// WC = the tap count when fixed at compile time, 0 = a.W at run time.
template <typename TIn, int WC>
__global__ void __launch_bounds__(256) conv_tiles_kernel(const __grid_constant__ CUtensorMap xmap,
                                                         ConvArgs a, int n_tiles, int n_items)
{
    using L = TileLayout<TIn>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tg = tid >> 7, i = tid & (kD - 1), wih = warp & 3;
    const int W = WC > 0 ? WC : a.W;
    const int T = a.T;
    const int n_heads = a.conv_dim / kD;
    const uint32_t tx_bytes = (uint32_t)(kTT + W - 1) * kD * sizeof(TIn);
    const uint32_t tile0 = tc::smem_addr(smem);
    const uint32_t mbar0 = tc::smem_addr(smem + L::mbar);
    float *sq = reinterpret_cast<float *>(smem + L::sq) + warp * 32 * kSqStride;
    float *part = reinterpret_cast<float *>(smem + L::part) + tg * 32 * 4;
    int *sflag = reinterpret_cast<int *>(smem + L::flag);

    auto issue = [&](int item, int buf) {
        const int head = item % n_heads, rest = item / n_heads;
        tile_copy_3d(&xmap, tile0 + buf * L::tile, mbar0 + 8 * buf, tx_bytes, head * kD,
                  (rest % n_tiles) * kTT - (W - 1), rest / n_tiles);
    };
    if (tid == 0) {
        tc::mbar_init(mbar0, 1);
        tc::mbar_init(mbar0 + 8, 1);
        *sflag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if ((int)blockIdx.x < n_items)
            issue(blockIdx.x, 0);
    }
    __syncthreads();

    int k = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++k) {
        const int buf = k & 1;
        if (tid == 0 && item + (int)gridDim.x < n_items)
            issue(item + gridDim.x, buf ^ 1);
        if (!tc::mbar_wait_ns(mbar0 + 8 * buf, (k >> 1) & 1, k == 0 ? a.first_wait_ns : kDefaultWaitNs))
            *sflag = 1;
        __syncthreads();
        if (*sflag)
            break;

        const int head = item % n_heads, rest = item / n_heads;
        const int t0 = (rest % n_tiles) * kTT, b = rest / n_tiles;
        const int c = head * kD + i;
        GDN_CHECK(g_conv_error, b < a.B && c < a.conv_dim && t0 < T);
        const bool is_qk = head < 2 * a.Hq;
        const TIn *tl = reinterpret_cast<const TIn *>(smem + buf * L::tile) + i;   // column i
        float w[kMaxW];
#pragma unroll
        for (int tau = 0; tau < kMaxW; ++tau)
            w[tau] = tau < W ? __ldg(a.conv_w + (size_t)c * W + tau) : 0.0f;
        // tokens before the call: the first W-1 rows of tile 0 come from the history
        const bool from_hist = t0 == 0 && tg == 0;
        float *hist_c = a.conv_state + ((size_t)b * a.conv_dim + c) * (W - 1);
        float hreg[kMaxW - 1];
#pragma unroll
        for (int e = 0; e < kMaxW - 1; ++e)
            hreg[e] = (from_hist && e < W - 1) ? hist_c[e] : 0.0f;

        // this thread's 32 + W - 1 stream values, each read from shared memory once
        float xr[32 + kMaxW - 1];
#pragma unroll
        for (int r = 0; r < 32 + kMaxW - 1; ++r)
            xr[r] = r < 32 + W - 1 ? smem_act<TIn>(tl + (32 * tg + r) * kD) : 0.0f;
#pragma unroll
        for (int r = 0; r < kMaxW - 1; ++r)
            if (from_hist && r < W - 1)
                xr[r] = hreg[r];
        float v[32];
#pragma unroll
        for (int p = 0; p < 32; ++p) {
            float acc = __fmul_rn(xr[p], w[0]);
#pragma unroll
            for (int tau = 1; tau < kMaxW; ++tau)
                if (tau < W)
                    acc = __fmaf_rn(xr[p + tau], w[tau], acc);
            v[p] = silu_f(acc);
        }
        if (is_qk) {   // uniform over the CTA
#pragma unroll
            for (int p = 0; p < 32; ++p)
                sq[p * kSqStride + lane] = __fmul_rn(v[p], v[p]);
            __syncwarp();
            // lane = token: its 32 squares, four 16-byte loads at a time
            float row[32];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 f = *reinterpret_cast<const float4 *>(sq + lane * kSqStride + 4 * q);
                row[4 * q] = f.x;
                row[4 * q + 1] = f.y;
                row[4 * q + 2] = f.z;
                row[4 * q + 3] = f.w;
            }
            float s[16];
#pragma unroll
            for (int l = 0; l < 16; ++l)
                s[l] = __fadd_rn(row[l], row[l + 16]);
#pragma unroll
            for (int m = 8; m >= 1; m >>= 1)
#pragma unroll
                for (int l = 0; l < m; ++l)
                    s[l] = __fadd_rn(s[l], s[l + m]);
            part[lane * 4 + wih] = s[0];
            __syncthreads();
            const float inv = l2_inv_of_partials(part + lane * 4, a.l2_eps);
#pragma unroll
            for (int p = 0; p < 32; ++p)
                v[p] = __fmul_rn(v[p], __shfl_sync(0xffffffffu, inv, p));
        }
        float *out_c = a.out + ((size_t)b * T + t0 + 32 * tg) * a.conv_dim + c;
        if (t0 + kTT <= T) {
#pragma unroll
            for (int p = 0; p < 32; ++p)
                out_c[(size_t)p * a.conv_dim] = v[p];
        } else {
#pragma unroll
            for (int p = 0; p < 32; ++p)
                if (t0 + 32 * tg + p < T)
                    out_c[(size_t)p * a.conv_dim] = v[p];
        }
        if (from_hist) {
            const TIn *x_c = static_cast<const TIn *>(a.x) + (int64_t)b * T * a.x_stride + c;
            float nh[kMaxW - 1];
            conv_history_after<TIn>(hist_c, x_c, a.x_stride, W, T, nh);
            store_history(hist_c, W, nh);
        }
        __syncthreads();   // tile, sq and part are free for the next item
    }
    if (*sflag && tid == 0) {
        atomicOr(&g_conv_error, kErrConvWait);
        // let the copies this CTA issued finish before it exits
        tc::mbar_wait_ns(mbar0 + 8 * (k & 1), (k >> 1) & 1, kDefaultWaitNs);
        if (blockIdx.x + (k + 1) * gridDim.x < (unsigned)n_items)
            tc::mbar_wait_ns(mbar0 + 8 * ((k + 1) & 1), ((k + 1) >> 1) & 1, kDefaultWaitNs);
    }
}

// The [B][T][conv_dim] view of x, boxes of 128 channels x (kTT + W - 1) rows.
bool encode_x_map(CUtensorMap *map, const ConvArgs &a, bool bf16)
{
    return encode_rows_map(map, a.x, bf16, a.conv_dim, a.x_stride, a.T, a.B, kD,
                           (uint32_t)(kTT + a.W - 1));
}

template <typename TIn, int WC>
cudaError_t launch_tiles(const CUtensorMap &map, const ConvArgs &a, cudaStream_t s)
{
    using L = TileLayout<TIn>;
    auto kernel = conv_tiles_kernel<TIn, WC>;
    static int per_sm = [&] {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::bytes);
        int n = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, L::bytes);
        return n > 0 ? n : 1;
    }();
    const int sms = sm_count();
    const int n_tiles = (a.T + kTT - 1) / kTT;
    const int64_t n_items = (int64_t)a.B * n_tiles * (a.conv_dim / kD);
    if (n_items > INT32_MAX)
        return cudaErrorInvalidConfiguration;
    const int grid = (int)std::min<int64_t>(n_items, (int64_t)sms * per_sm);
    kernel<<<grid, 256, L::bytes, s>>>(map, a, n_tiles, (int)n_items);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv_update(const ConvArgs &a, bool bf16, cudaStream_t s)
{
    if (a.T == 1) {
        const dim3 grid(a.conv_dim / kD, a.B, 1);
        if (bf16)
            conv_update_kernel<__nv_bfloat16><<<grid, kD, 0, s>>>(a);
        else
            conv_update_kernel<float><<<grid, kD, 0, s>>>(a);
        return cudaGetLastError();
    }
    CUtensorMap map;
    if (encode_x_map(&map, a, bf16)) {
        if (bf16)
            return a.W == 4 ? launch_tiles<__nv_bfloat16, 4>(map, a, s)
                            : launch_tiles<__nv_bfloat16, 0>(map, a, s);
        return a.W == 4 ? launch_tiles<float, 4>(map, a, s) : launch_tiles<float, 0>(map, a, s);
    }
    constexpr int tile = 2 * kTokensPerThread;
    const dim3 grid(a.conv_dim / kD, (a.T + tile - 1) / tile, a.B);
    if (grid.y > 65535)
        return cudaErrorInvalidConfiguration;
    if (bf16)
        conv_tokens_kernel<__nv_bfloat16, kTokensPerThread><<<grid, 256, 0, s>>>(a);
    else
        conv_tokens_kernel<float, kTokensPerThread><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t take_conv_device_error(int *code)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_conv_error, sizeof(int));
    if (e == cudaSuccess && v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_conv_error, &zero, sizeof(int));
    }
    *code = v;
    return e;
}

}  // namespace gdn
