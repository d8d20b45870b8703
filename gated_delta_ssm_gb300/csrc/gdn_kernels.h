// gdn_kernels.h -- internal launch interface between the C ABI (abi.cu) and
// the kernel files. Not installed; the public interface is include/gdn.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

struct FusedArgs {
    void *state;           // [B][Hv][d][d], float (bf16 for the bf16-state step)
    float *conv_state;     // [B][conv_dim][W-1]
    void *state_snap;      // verify only, float
    float *conv_snap;      // verify only
    const void *x, *z, *alpha, *beta_logit;
    const float *conv_w, *dt, *A_log, *norm_w;
    void *out;             // [B][NTOK][Hv][d], the state's type
    int64_t x_stride, z_stride, gate_stride;
    int B, Hq, Hv, W, conv_dim;
    float l2_eps, rms_eps, scale;
    int sm_count;          // SMs of the device (the bf16-state step's L2 prefetch distance)
    // single-token step after a K-token verify (null: read state / conv_state): sequence b
    // starts from snapshot n-1 (state_snap [B][K-1][Hv][d][d], conv_snap [B][E][conv_dim][W-1])
    // when n = n_accept[b] < K, else from state / conv_state
    const int32_t *n_accept;
    int n_draft, conv_snap_entries;
};

struct ConvArgs {
    float *conv_state;
    const void *x;
    const float *conv_w;
    float *out;            // [B][T][conv_dim]
    int64_t x_stride;
    int B, Hq, Hv, W, conv_dim, T;
    float l2_eps;
    uint64_t first_wait_ns;  // limit of each CTA's first tile wait (global-timer ns)
};

struct RecArgs {
    float *state;
    const float *q, *k, *v;
    int64_t qkv_stride;
    const float *g, *beta;
    float *y;
    int B, Hq, Hv;
    float scale;
};

struct RecScanArgs {
    float *state;          // [B][Hv][d][d]
    const float *q, *k, *v;// token (b, t) at row b*T + t, qkv_stride apart
    int64_t qkv_stride;
    const float *g, *beta; // [B][T][Hv]
    float *y;              // [B][T][Hv][d]
    int B, Hq, Hv, T;
    float scale;
};

// The fused layer stepped token by token over T tokens of every sequence.
struct LayerScanArgs {
    float *state;          // [B][Hv][d][d]
    float *conv_state;     // [B][conv_dim][W-1]
    float *state_snap;     // [B][T-1][Hv][d][d] or null
    float *conv_snap;      // [B][T][conv_dim][W-1] or null
    const void *x, *z, *alpha, *beta_logit;
    const float *conv_w, *dt, *A_log, *norm_w;
    float *out;            // [B][T][Hv][d]
    int64_t x_stride, z_stride, gate_stride;
    int B, Hq, Hv, W, conv_dim, T;
    float l2_eps, rms_eps, scale;
};

struct PrefillArgs {
    float *state;
    float *conv_state;
    const void *x, *z, *alpha, *beta_logit;
    const float *conv_w, *dt, *A_log, *norm_w;
    float *out;            // [B][T][Hv][d]
    uint8_t *ws;           // workspace: chunk images, then [Q; K] images (prefill.cu)
    size_t ws_bytes;
    int64_t x_stride, z_stride, gate_stride;
    int B, Hq, Hv, W, conv_dim, T, n_chunks;
    float l2_eps, rms_eps, scale;
    uint64_t wait_ns;        // limit of every bounded wait (global-timer nanoseconds)
    uint64_t first_wait_ns;  // limit of the chain kernel's first wait
};

// Prefill workspace: per (sequence, V head, chunk) an image of (I + A)^-1, P and
// the chunk's gates; per (sequence, QK head, chunk) the chunk's normalised Q and
// K rows as tensor-core operands. All images are 1 KB multiples.
constexpr size_t kPrefillChunkImage = 34816;
constexpr size_t kPrefillQKImage = 65536;
inline size_t prefill_workspace_bytes(int B, int Hq, int Hv, int n_chunks)
{
    return (size_t)B * (size_t)n_chunks * ((size_t)Hv * kPrefillChunkImage + (size_t)Hq * kPrefillQKImage);
}

// Streaming multiprocessors of the current device, queried once per device.
int sm_count();

// Row slices per head of the single-token decode: enough CTAs (about four per
// SM) to keep every SM streaming state, without growing a cluster (r CTAs share
// a QK head, ns slices per head) past 4 CTAs by slicing. Past that the cluster's
// barriers and shared-memory exchanges cost more than the extra CTAs give
// (measured: one sequence of 32 V heads in 16 QK pairs, 3.92 us per step with
// 8-CTA clusters of 4 slices, 3.72 us with 4-CTA clusters of 2).
inline int pick_nsplit(int B, int Hv, int r, int sms)
{
    int ns = 1;
    while (ns < 4 && (int64_t)B * Hv * ns < 4 * (int64_t)sms && r * ns * 2 <= 4)
        ns *= 2;
    return ns;
}

// Row slices per head of the token-serial scans: as many as fill one wave of 2
// CTAs per SM without spilling into a second (a token-serial CTA's duration is
// its token count, so a partial second wave would double the time), within an
// 8-CTA cluster.
inline int scan_nsplit(int B, int Hv, int r, int sms)
{
    int ns = 1;
    while (ns < 4 && (int64_t)B * Hv * ns * 2 <= 2 * (int64_t)sms && r * ns * 2 <= 8)
        ns *= 2;
    return ns;
}

// Default limit of a bounded wait, and the test-only override of one prefill
// wait and of the tiled conv's first tile wait (0 = the default).
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
uint64_t first_wait_override_ns();

cudaError_t launch_decode_fused(const FusedArgs &a, bool bf16, int ntok, cudaStream_t s);
cudaError_t launch_decode_fused_bf16_state(const FusedArgs &a, bool bf16, cudaStream_t s);
cudaError_t launch_decay_gate(const void *alpha, bool bf16, int64_t alpha_stride, const float *dt,
                              const float *A_log, float *g, int rows, int H, cudaStream_t s);
cudaError_t launch_conv_update(const ConvArgs &a, bool bf16, cudaStream_t s);
cudaError_t launch_recurrence_decode(const RecArgs &a, cudaStream_t s);
cudaError_t launch_gated_norm(const float *y, const float *w, const void *z, bool bf16,
                              int64_t z_stride, float *out, int rows, int Hv, float eps,
                              cudaStream_t s);
cudaError_t launch_verify_commit(float *state, float *conv_state, const float *state_snap,
                                 const float *conv_snap, const int32_t *n_accept, int B,
                                 int64_t state_elems, int64_t hist_elems, cudaStream_t s);
cudaError_t take_decode_device_error(int *code);
cudaError_t launch_recurrence_scan(const RecScanArgs &a, cudaStream_t s);
cudaError_t launch_layer_scan(const LayerScanArgs &a, bool bf16, cudaStream_t s);
cudaError_t launch_verify_commit_kn(float *state, float *conv_state, const float *state_snap,
                                    const float *conv_snap, const int32_t *n_accept, int B, int K,
                                    int64_t state_elems, int64_t hist_elems, cudaStream_t s);
cudaError_t take_sequential_device_error(int *code);
cudaError_t take_conv_device_error(int *code);
cudaError_t take_prefill_device_error(int *code);
cudaError_t launch_prefill(const PrefillArgs &a, bool bf16, cudaStream_t s);

}  // namespace gdn
