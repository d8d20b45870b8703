// abi.cu -- the extern "C" entry points of libgdn (declared in include/gdn.h):
// host-side argument validation, then one launch on the caller's stream.
// Nothing here allocates, synchronises or keeps state between calls, beyond
// the thread-local last-error text and a per-device cache of the SM count.
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/gdn.h"
#include "../../include/gdn_testing.h"
#include "gdn_device.cuh"
#include "gdn_kernels.h"

namespace gdn {
namespace {
std::atomic<uint64_t> g_first_wait_ns{0};
constexpr int kMaxSmDevices = 64;
std::atomic<int> g_sm_count[kMaxSmDevices];   // 0 until queried
}
uint64_t first_wait_override_ns()
{
    const uint64_t v = g_first_wait_ns.load(std::memory_order_relaxed);
    return v != 0 ? v : kDefaultWaitNs;
}
int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 1;
    if (dev >= 0 && dev < kMaxSmDevices && (n = g_sm_count[dev].load(std::memory_order_relaxed)) > 0)
        return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return 1;   // the launch that follows reports the device's error
    if (dev >= 0 && dev < kMaxSmDevices)
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}
}  // namespace gdn

namespace {

thread_local char g_last_cuda_error[256] = "";

gdn_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess)
        return GDN_OK;
    snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s", cudaGetErrorName(e),
             cudaGetErrorString(e));
    return GDN_ERR_CUDA;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t act_size(gdn_dtype t) { return t == GDN_BF16 ? 2 : 4; }

bool valid_dtype(gdn_dtype t) { return t == GDN_F32 || t == GDN_BF16; }

cudaStream_t as_cuda(gdn_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Shape checks shared by every entry point that takes gdn_dims.
// need: bit 0 = x_stride used, bit 1 = z_stride used, bit 2 = gate_stride used.
gdn_status check_dims(const gdn_dims *d, int need)
{
    if (!d)
        return GDN_ERR_INVALID_ARG;
    if (d->n_seq < 1 || d->n_seq > 65535 || d->n_qk_heads < 1 || d->n_v_heads < 1 ||
        d->head_dim < 1 || d->d_conv < 1 || d->reserved != 0)
        return GDN_ERR_INVALID_ARG;
    if (d->n_v_heads % d->n_qk_heads != 0)
        return GDN_ERR_INVALID_ARG;
    const int64_t conv_dim = (int64_t)(2 * (int64_t)d->n_qk_heads + d->n_v_heads) * d->head_dim;
    if (conv_dim > (1 << 24))
        return GDN_ERR_INVALID_ARG;
    if ((need & 1) && d->x_stride < conv_dim)
        return GDN_ERR_INVALID_ARG;
    if ((need & 2) && d->z_stride < (int64_t)d->n_v_heads * d->head_dim)
        return GDN_ERR_INVALID_ARG;
    if ((need & 4) && d->gate_stride < d->n_v_heads)
        return GDN_ERR_INVALID_ARG;
    if (d->head_dim != gdn::kD)
        return GDN_ERR_UNSUPPORTED;
    if (d->d_conv < 2 || d->d_conv > gdn::kMaxW)
        return GDN_ERR_UNSUPPORTED;
    if (d->n_v_heads / d->n_qk_heads > 8)
        return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

gdn_status check_params(const gdn_params *p)
{
    if (!p || !p->conv_w || !p->dt || !p->A_log || !p->norm_w)
        return GDN_ERR_INVALID_ARG;
    if (!(p->l2_eps >= 0.0f) || !(p->rms_eps >= 0.0f))
        return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

int conv_dim_of(const gdn_dims *d) { return (2 * d->n_qk_heads + d->n_v_heads) * d->head_dim; }

// bf16_state: state and out are bf16 (single-token step only).
gdn_status fused_common(void *state, float *conv_state, float *state_snap, float *conv_snap,
                        const void *x, const void *z, const void *alpha, const void *beta_logit,
                        gdn_dtype act_dtype, const gdn_params *params, void *out,
                        const gdn_dims *dims, int ntok, bool bf16_state, gdn_stream_t stream,
                        const int32_t *n_accept = nullptr, int n_draft = 0,
                        int conv_snap_entries = 0)
{
    gdn_status st = check_dims(dims, 7);
    if (st != GDN_OK)
        return st;
    if ((st = check_params(params)) != GDN_OK)
        return st;
    if (!valid_dtype(act_dtype))
        return GDN_ERR_INVALID_ARG;
    if (!state || !conv_state || !x || !z || !alpha || !beta_logit || !out)
        return GDN_ERR_INVALID_ARG;
    if (ntok >= 2 && (!state_snap || !conv_snap))
        return GDN_ERR_INVALID_ARG;
    const size_t es = act_size(act_dtype);
    if (!aligned(state, 16) || (state_snap && !aligned(state_snap, 16)) || !aligned(x, es) ||
        !aligned(z, es) || !aligned(alpha, es) || !aligned(beta_logit, es) ||
        !aligned(out, bf16_state ? 2 : 4) || !aligned(conv_state, 4) ||
        (conv_snap && !aligned(conv_snap, 4)))
        return GDN_ERR_INVALID_ARG;
    gdn::FusedArgs a;
    a.state = state;
    a.conv_state = conv_state;
    a.state_snap = state_snap;
    a.conv_snap = conv_snap;
    a.x = x;
    a.z = z;
    a.alpha = alpha;
    a.beta_logit = beta_logit;
    a.conv_w = params->conv_w;
    a.dt = params->dt;
    a.A_log = params->A_log;
    a.norm_w = params->norm_w;
    a.out = out;
    a.x_stride = dims->x_stride;
    a.z_stride = dims->z_stride;
    a.gate_stride = dims->gate_stride;
    a.B = dims->n_seq;
    a.Hq = dims->n_qk_heads;
    a.Hv = dims->n_v_heads;
    a.W = dims->d_conv;
    a.conv_dim = conv_dim_of(dims);
    a.l2_eps = params->l2_eps;
    a.rms_eps = params->rms_eps;
    a.scale = 1.0f / sqrtf((float)dims->head_dim);
    a.sm_count = gdn::sm_count();
    a.n_accept = n_accept;
    a.n_draft = n_draft;
    a.conv_snap_entries = conv_snap_entries;
    if (bf16_state)
        return from_cuda(gdn::launch_decode_fused_bf16_state(a, act_dtype == GDN_BF16,
                                                             as_cuda(stream)));
    return from_cuda(gdn::launch_decode_fused(a, act_dtype == GDN_BF16, ntok, as_cuda(stream)));
}

gdn_status layer_scan_common(float *state, float *conv_state, float *state_snap, float *conv_snap,
                             const void *x, const void *z, const void *alpha,
                             const void *beta_logit, gdn_dtype act_dtype,
                             const gdn_params *params, float *out, const gdn_dims *dims,
                             int32_t n_tokens, gdn_stream_t stream)
{
    gdn_status st = check_dims(dims, 7);
    if (st != GDN_OK)
        return st;
    if ((st = check_params(params)) != GDN_OK)
        return st;
    if (!valid_dtype(act_dtype) || n_tokens < 1)
        return GDN_ERR_INVALID_ARG;
    if (!state || !conv_state || !x || !z || !alpha || !beta_logit || !out)
        return GDN_ERR_INVALID_ARG;
    const size_t es = act_size(act_dtype);
    if (!aligned(state, 16) || (state_snap && !aligned(state_snap, 16)) || !aligned(x, es) ||
        !aligned(z, es) || !aligned(alpha, es) || !aligned(beta_logit, es) || !aligned(out, 4) ||
        !aligned(conv_state, 4) || (conv_snap && !aligned(conv_snap, 4)))
        return GDN_ERR_INVALID_ARG;
    gdn::LayerScanArgs a;
    a.state = state;
    a.conv_state = conv_state;
    a.state_snap = n_tokens > 1 ? state_snap : nullptr;
    a.conv_snap = conv_snap;
    a.x = x;
    a.z = z;
    a.alpha = alpha;
    a.beta_logit = beta_logit;
    a.conv_w = params->conv_w;
    a.dt = params->dt;
    a.A_log = params->A_log;
    a.norm_w = params->norm_w;
    a.out = out;
    a.x_stride = dims->x_stride;
    a.z_stride = dims->z_stride;
    a.gate_stride = dims->gate_stride;
    a.B = dims->n_seq;
    a.Hq = dims->n_qk_heads;
    a.Hv = dims->n_v_heads;
    a.W = dims->d_conv;
    a.conv_dim = conv_dim_of(dims);
    a.T = n_tokens;
    a.l2_eps = params->l2_eps;
    a.rms_eps = params->rms_eps;
    a.scale = 1.0f / sqrtf((float)dims->head_dim);
    return from_cuda(gdn::launch_layer_scan(a, act_dtype == GDN_BF16, as_cuda(stream)));
}

// [p, p + pb) and [q, q + qb) share a byte
bool overlaps(const void *p, size_t pb, const void *q, size_t qb)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), c = reinterpret_cast<uintptr_t>(q);
    return a < c + qb && c < a + pb;
}

}  // namespace

extern "C" {

gdn_status gdn_decay_gate(const void *alpha, gdn_dtype alpha_dtype, int64_t alpha_stride,
                          const float *dt, const float *A_log, float *g, int32_t rows,
                          int32_t n_heads, gdn_stream_t stream)
{
    if (!alpha || !dt || !A_log || !g || rows < 1 || n_heads < 1 || alpha_stride < n_heads ||
        !valid_dtype(alpha_dtype) || !aligned(alpha, act_size(alpha_dtype)))
        return GDN_ERR_INVALID_ARG;
    return from_cuda(gdn::launch_decay_gate(alpha, alpha_dtype == GDN_BF16, alpha_stride, dt,
                                            A_log, g, rows, n_heads, as_cuda(stream)));
}

gdn_status gdn_conv_update(float *conv_state, const void *x, gdn_dtype x_dtype,
                           const float *conv_w, float *out, const gdn_dims *dims,
                           int32_t n_tokens, float l2_eps, gdn_stream_t stream)
{
    gdn_status st = check_dims(dims, 1);
    if (st != GDN_OK)
        return st;
    if (!conv_state || !x || !conv_w || !out || n_tokens < 1 || !valid_dtype(x_dtype) ||
        !(l2_eps >= 0.0f) || !aligned(x, act_size(x_dtype)))
        return GDN_ERR_INVALID_ARG;
    gdn::ConvArgs a;
    a.conv_state = conv_state;
    a.x = x;
    a.conv_w = conv_w;
    a.out = out;
    a.x_stride = dims->x_stride;
    a.B = dims->n_seq;
    a.Hq = dims->n_qk_heads;
    a.Hv = dims->n_v_heads;
    a.W = dims->d_conv;
    a.conv_dim = conv_dim_of(dims);
    a.T = n_tokens;
    a.l2_eps = l2_eps;
    a.first_wait_ns = gdn::first_wait_override_ns();
    return from_cuda(gdn::launch_conv_update(a, x_dtype == GDN_BF16, as_cuda(stream)));
}

gdn_status gdn_recurrence_decode(float *state, const float *q, const float *k, const float *v,
                                 int64_t qkv_stride, const float *g, const float *beta, float *y,
                                 const gdn_dims *dims, float scale, gdn_stream_t stream)
{
    gdn_status st = check_dims(dims, 0);
    if (st != GDN_OK)
        return st;
    if (!state || !q || !k || !v || !g || !beta || !y || !aligned(state, 16))
        return GDN_ERR_INVALID_ARG;
    if (dims->n_seq > 1 && qkv_stride < (int64_t)dims->n_v_heads * dims->head_dim)
        return GDN_ERR_INVALID_ARG;
    gdn::RecArgs a;
    a.state = state;
    a.q = q;
    a.k = k;
    a.v = v;
    a.qkv_stride = qkv_stride;
    a.g = g;
    a.beta = beta;
    a.y = y;
    a.B = dims->n_seq;
    a.Hq = dims->n_qk_heads;
    a.Hv = dims->n_v_heads;
    a.scale = scale;
    return from_cuda(gdn::launch_recurrence_decode(a, as_cuda(stream)));
}

gdn_status gdn_gated_norm(const float *y, const float *norm_w, const void *z, gdn_dtype z_dtype,
                          int64_t z_stride, float *out, int32_t rows, int32_t n_v_heads,
                          int32_t head_dim, float eps, gdn_stream_t stream)
{
    if (!y || !norm_w || !z || !out || rows < 1 || n_v_heads < 1 || head_dim < 1 ||
        !valid_dtype(z_dtype) || z_stride < (int64_t)n_v_heads * head_dim || !(eps >= 0.0f) ||
        !aligned(z, act_size(z_dtype)))
        return GDN_ERR_INVALID_ARG;
    if (head_dim != gdn::kD)
        return GDN_ERR_UNSUPPORTED;
    return from_cuda(gdn::launch_gated_norm(y, norm_w, z, z_dtype == GDN_BF16, z_stride, out, rows,
                                            n_v_heads, eps, as_cuda(stream)));
}

gdn_status gdn_decode_step(float *state, float *conv_state, const void *x, const void *z,
                           const void *alpha, const void *beta_logit, gdn_dtype act_dtype,
                           const gdn_params *params, float *out, const gdn_dims *dims,
                           gdn_stream_t stream)
{
    return fused_common(state, conv_state, nullptr, nullptr, x, z, alpha, beta_logit, act_dtype,
                        params, out, dims, 1, false, stream);
}

gdn_status gdn_decode_step_bf16_state(void *state, float *conv_state, const void *x,
                                      const void *z, const void *alpha, const void *beta_logit,
                                      gdn_dtype act_dtype, const gdn_params *params, void *out,
                                      const gdn_dims *dims, gdn_stream_t stream)
{
    return fused_common(state, conv_state, nullptr, nullptr, x, z, alpha, beta_logit, act_dtype,
                        params, out, dims, 1, true, stream);
}

gdn_status gdn_decode_step_select(float *state, float *conv_state, const float *state_snap,
                                  const float *conv_snap, int32_t conv_snap_entries,
                                  const int32_t *n_accept, int32_t n_draft, const void *x,
                                  const void *z, const void *alpha, const void *beta_logit,
                                  gdn_dtype act_dtype, const gdn_params *params, float *out,
                                  const gdn_dims *dims, gdn_stream_t stream)
{
    gdn_status st = check_dims(dims, 7);
    if (st != GDN_OK)
        return st;
    if (!n_accept || n_draft < 1)
        return GDN_ERR_INVALID_ARG;
    if (n_draft > 1) {
        if (!state_snap || !conv_snap || (conv_snap_entries != n_draft - 1 && conv_snap_entries != n_draft))
            return GDN_ERR_INVALID_ARG;
        const size_t B = (size_t)dims->n_seq, d = (size_t)dims->head_dim;
        const size_t sbytes = B * dims->n_v_heads * d * d * 4;
        const size_t hbytes = B * (size_t)conv_dim_of(dims) * (size_t)(dims->d_conv - 1) * 4;
        const size_t ssnap = sbytes * (size_t)(n_draft - 1), hsnap = hbytes * (size_t)conv_snap_entries;
        if (overlaps(state, sbytes, state_snap, ssnap) || overlaps(conv_state, hbytes, conv_snap, hsnap) ||
            overlaps(state, sbytes, conv_snap, hsnap) || overlaps(conv_state, hbytes, state_snap, ssnap))
            return GDN_ERR_INVALID_ARG;
    }
    return fused_common(state, conv_state, const_cast<float *>(state_snap), const_cast<float *>(conv_snap),
                        x, z, alpha, beta_logit, act_dtype, params, out, dims, 1, false, stream,
                        n_accept, n_draft, n_draft > 1 ? conv_snap_entries : 0);
}

gdn_status gdn_verify_k2(float *state, float *conv_state, float *state_snap, float *conv_snap,
                         const void *x, const void *z, const void *alpha, const void *beta_logit,
                         gdn_dtype act_dtype, const gdn_params *params, float *out,
                         const gdn_dims *dims, gdn_stream_t stream)
{
    if (state_snap == state || conv_snap == conv_state)
        return GDN_ERR_INVALID_ARG;
    return fused_common(state, conv_state, state_snap, conv_snap, x, z, alpha, beta_logit,
                        act_dtype, params, out, dims, 2, false, stream);
}

gdn_status gdn_verify_commit(float *state, float *conv_state, const float *state_snap,
                             const float *conv_snap, const int32_t *n_accept,
                             const gdn_dims *dims, gdn_stream_t stream)
{
    gdn_status st = check_dims(dims, 0);
    if (st != GDN_OK)
        return st;
    if (!state || !conv_state || !state_snap || !conv_snap || !n_accept || !aligned(state, 16) ||
        !aligned(state_snap, 16))
        return GDN_ERR_INVALID_ARG;
    const int64_t d = dims->head_dim;
    return from_cuda(gdn::launch_verify_commit(state, conv_state, state_snap, conv_snap, n_accept,
                                               dims->n_seq, (int64_t)dims->n_v_heads * d * d,
                                               (int64_t)conv_dim_of(dims) * (dims->d_conv - 1),
                                               as_cuda(stream)));
}

gdn_status gdn_recurrence_scan(float *state, const float *q, const float *k, const float *v,
                               int64_t qkv_stride, const float *g, const float *beta, float *y,
                               const gdn_dims *dims, int32_t n_tokens, float scale,
                               gdn_stream_t stream)
{
    gdn_status st = check_dims(dims, 0);
    if (st != GDN_OK)
        return st;
    if (!state || !q || !k || !v || !g || !beta || !y || !aligned(state, 16) || n_tokens < 1)
        return GDN_ERR_INVALID_ARG;
    if ((int64_t)dims->n_seq * n_tokens > 1 &&
        qkv_stride < (int64_t)dims->n_v_heads * dims->head_dim)
        return GDN_ERR_INVALID_ARG;
    gdn::RecScanArgs a;
    a.state = state;
    a.q = q;
    a.k = k;
    a.v = v;
    a.qkv_stride = qkv_stride;
    a.g = g;
    a.beta = beta;
    a.y = y;
    a.B = dims->n_seq;
    a.Hq = dims->n_qk_heads;
    a.Hv = dims->n_v_heads;
    a.T = n_tokens;
    a.scale = scale;
    return from_cuda(gdn::launch_recurrence_scan(a, as_cuda(stream)));
}

gdn_status gdn_layer_scan(float *state, float *conv_state, const void *x, const void *z,
                          const void *alpha, const void *beta_logit, gdn_dtype act_dtype,
                          const gdn_params *params, float *out, const gdn_dims *dims,
                          int32_t n_tokens, gdn_stream_t stream)
{
    return layer_scan_common(state, conv_state, nullptr, nullptr, x, z, alpha, beta_logit,
                             act_dtype, params, out, dims, n_tokens, stream);
}

gdn_status gdn_verify_kn(float *state, float *conv_state, float *state_snap, float *conv_snap,
                         const void *x, const void *z, const void *alpha, const void *beta_logit,
                         gdn_dtype act_dtype, const gdn_params *params, float *out,
                         const gdn_dims *dims, int32_t n_draft, gdn_stream_t stream)
{
    if (!conv_snap || (n_draft > 1 && !state_snap) || state_snap == state ||
        conv_snap == conv_state)
        return GDN_ERR_INVALID_ARG;
    // up to eight positions: the fused step kernel over all positions at once (state rows
    // held in registers, one snapshot entry per position); longer drafts: the layer scan.
    // Both give the bits of n_draft single steps.
    if (n_draft >= 2 && n_draft <= 8)
        return fused_common(state, conv_state, state_snap, conv_snap, x, z, alpha, beta_logit,
                            act_dtype, params, out, dims, n_draft, false, stream, nullptr, 0, n_draft);
    return layer_scan_common(state, conv_state, state_snap, conv_snap, x, z, alpha, beta_logit,
                             act_dtype, params, out, dims, n_draft, stream);
}

gdn_status gdn_verify_commit_kn(float *state, float *conv_state, const float *state_snap,
                                const float *conv_snap, const int32_t *n_accept,
                                const gdn_dims *dims, int32_t n_draft, gdn_stream_t stream)
{
    gdn_status st = check_dims(dims, 0);
    if (st != GDN_OK)
        return st;
    if (n_draft < 1 || !state || !conv_state || !conv_snap || !n_accept ||
        (n_draft > 1 && !state_snap) || !aligned(state, 16) ||
        (state_snap && !aligned(state_snap, 16)))
        return GDN_ERR_INVALID_ARG;
    const int64_t d = dims->head_dim;
    return from_cuda(gdn::launch_verify_commit_kn(
        state, conv_state, state_snap, conv_snap, n_accept, dims->n_seq, n_draft,
        (int64_t)dims->n_v_heads * d * d, (int64_t)conv_dim_of(dims) * (dims->d_conv - 1),
        as_cuda(stream)));
}

size_t gdn_prefill_workspace_bytes(const gdn_dims *dims, int32_t n_tokens, int32_t chunk)
{
    if (check_dims(dims, 0) != GDN_OK || n_tokens < 1 || chunk != 64)
        return 0;
    const int64_t n_chunks = ((int64_t)n_tokens + 63) / 64;
    return gdn::prefill_workspace_bytes(dims->n_seq, dims->n_qk_heads, dims->n_v_heads, (int)n_chunks);
}

gdn_status gdn_prefill_chunked(float *state, float *conv_state, const void *x, const void *z,
                               const void *alpha, const void *beta_logit, gdn_dtype act_dtype,
                               const gdn_params *params, float *out, const gdn_dims *dims,
                               int32_t n_tokens, int32_t chunk, void *workspace,
                               size_t workspace_bytes, gdn_stream_t stream)
{
    gdn_status st = check_dims(dims, 7);
    if (st != GDN_OK)
        return st;
    if ((st = check_params(params)) != GDN_OK)
        return st;
    if (!valid_dtype(act_dtype) || n_tokens < 1)
        return GDN_ERR_INVALID_ARG;
    if (!state || !conv_state || !x || !z || !alpha || !beta_logit || !out || !workspace)
        return GDN_ERR_INVALID_ARG;
    const size_t es = act_size(act_dtype);
    // the chunk kernels read 4 channels of a token row per 8- or 16-byte load
    if (!aligned(state, 16) || !aligned(x, 16) || (dims->x_stride * (int64_t)es) % 16 != 0 ||
        !aligned(params->conv_w, 16) || !aligned(workspace, 16) ||
        !aligned(z, es) || !aligned(alpha, es) || !aligned(beta_logit, es) || !aligned(out, 16))
        return GDN_ERR_INVALID_ARG;
    if (chunk != 64)
        return GDN_ERR_UNSUPPORTED;
    const size_t need = gdn_prefill_workspace_bytes(dims, n_tokens, chunk);
    if (need == 0 || workspace_bytes < need)
        return GDN_ERR_INVALID_ARG;
    const int64_t n_chunks = ((int64_t)n_tokens + 63) / 64;
    if (n_chunks > INT32_MAX)
        return GDN_ERR_INVALID_ARG;
    gdn::PrefillArgs a;
    a.state = state;
    a.conv_state = conv_state;
    a.x = x;
    a.z = z;
    a.alpha = alpha;
    a.beta_logit = beta_logit;
    a.conv_w = params->conv_w;
    a.dt = params->dt;
    a.A_log = params->A_log;
    a.norm_w = params->norm_w;
    a.out = out;
    a.ws = static_cast<uint8_t *>(workspace);
    a.ws_bytes = workspace_bytes;
    a.x_stride = dims->x_stride;
    a.z_stride = dims->z_stride;
    a.gate_stride = dims->gate_stride;
    a.B = dims->n_seq;
    a.Hq = dims->n_qk_heads;
    a.Hv = dims->n_v_heads;
    a.W = dims->d_conv;
    a.conv_dim = conv_dim_of(dims);
    a.T = n_tokens;
    a.n_chunks = (int)n_chunks;
    a.l2_eps = params->l2_eps;
    a.rms_eps = params->rms_eps;
    a.scale = 1.0f / sqrtf((float)dims->head_dim);
    a.wait_ns = gdn::kDefaultWaitNs;
    a.first_wait_ns = gdn::first_wait_override_ns();
    return from_cuda(gdn::launch_prefill(a, act_dtype == GDN_BF16, as_cuda(stream)));
}

// ------------------------------------------------------------------ allocation-free prefill
// Callers that cannot allocate device memory get the prefill's workspace from a
// fixed array owned by the library. It lives in this file so that the host side
// can resolve its device address here.
}  // extern "C"

namespace {
constexpr size_t kStaticScratchBytes = (size_t)16 << 20;   // 16 MiB of prefill workspace
__device__ __align__(256) uint8_t g_prefill_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_prefill_scratch on the current device, resolved once per
// device (the host-side symbol is only a stand-in for it).
gdn_status scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return from_cuda(e);
    if (dev < 0 || dev >= kMaxDevices)
        return GDN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_prefill_scratch);
        if (e != cudaSuccess)
            return from_cuda(e);
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}
}  // namespace

extern "C" {

gdn_status gdn_prefill_chunked_noalloc(float *state, float *conv_state, const void *x,
                                       const void *z, const void *alpha, const void *beta_logit,
                                       gdn_dtype act_dtype, const gdn_params *params, float *out,
                                       const gdn_dims *dims, int32_t n_tokens, int32_t chunk,
                                       gdn_stream_t stream)
{
    const size_t need = gdn_prefill_workspace_bytes(dims, n_tokens, chunk);
    if (need > kStaticScratchBytes) {
        snprintf(g_last_cuda_error, sizeof g_last_cuda_error,
                 "gdn_prefill_chunked_noalloc: %zu bytes of scratch needed, the static scratch "
                 "holds %zu", need, kStaticScratchBytes);
        return GDN_ERR_UNSUPPORTED;
    }
    void *scratch = nullptr;
    const gdn_status st = scratch_address(&scratch);
    if (st != GDN_OK)
        return st;
    return gdn_prefill_chunked(state, conv_state, x, z, alpha, beta_logit, act_dtype, params, out,
                               dims, n_tokens, chunk, scratch, kStaticScratchBytes, stream);
}

void gdn_testing_set_first_wait_ns(uint64_t ns)
{
    gdn::g_first_wait_ns.store(ns, std::memory_order_relaxed);
}

void gdn_testing_row_splits(int32_t n_seq, int32_t n_v_heads, int32_t r, int32_t sms,
                            int32_t *decode_split, int32_t *scan_split)
{
    *decode_split = gdn::pick_nsplit(n_seq, n_v_heads, r, sms);
    *scan_split = gdn::scan_nsplit(n_seq, n_v_heads, r, sms);
}

gdn_status gdn_check_device(int32_t *code)
{
    int a = 0, b = 0, c = 0, d = 0;
    gdn_status st = from_cuda(gdn::take_decode_device_error(&a));
    if (st == GDN_OK)
        st = from_cuda(gdn::take_prefill_device_error(&b));
    if (st == GDN_OK)
        st = from_cuda(gdn::take_sequential_device_error(&c));
    if (st == GDN_OK)
        st = from_cuda(gdn::take_conv_device_error(&d));
    const int all = a | b | c | d;
    if (code)
        *code = all;
    if (st != GDN_OK)
        return st;
    return all ? GDN_ERR_DEVICE : GDN_OK;
}

const char *gdn_last_cuda_error(void) { return g_last_cuda_error; }

const char *gdn_status_string(gdn_status s)
{
    switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_DEVICE: return "GDN_ERR_DEVICE";
    }
    return "unknown gdn_status";
}

const char *gdn_version(void) { return "libgdn 0.1.0 (sm_103a)"; }

}  // extern "C"
