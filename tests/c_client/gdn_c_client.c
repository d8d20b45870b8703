/*
 * A plain C client of libgdn: no Python, no C++. It fills a small layer's
 * inputs on the host, runs two single-token decode steps and, from the same
 * starting state, one two-token layer scan, and checks that the outputs,
 * states and conv histories agree bit for bit (the scan is defined to equal
 * the single steps). Prints "c client ok" and exits 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "gdn.h"

#define CHECK(call)                                                                   \
    do {                                                                              \
        gdn_status st_ = (call);                                                      \
        if (st_ != GDN_OK) {                                                          \
            fprintf(stderr, "%s: %s %s\n", #call, gdn_status_string(st_),             \
                    gdn_last_cuda_error());                                           \
            return 1;                                                                 \
        }                                                                             \
    } while (0)
#define CUDA(call)                                                                    \
    do {                                                                              \
        cudaError_t e_ = (call);                                                      \
        if (e_ != cudaSuccess) {                                                      \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));               \
            return 1;                                                                 \
        }                                                                             \
    } while (0)

static uint32_t rng = 12345u;
static float uniform(void) /* in (-1, 1) */
{
    rng = rng * 1664525u + 1013904223u;
    return (float)((int32_t)(rng >> 8) - (1 << 23)) / (float)(1 << 23);
}

static int fill(float **dev, size_t n, float scale)
{
    float *h = (float *)malloc(n * sizeof(float));
    if (!h)
        return 1;
    for (size_t i = 0; i < n; ++i)
        h[i] = scale * uniform();
    cudaError_t e = cudaMalloc((void **)dev, n * sizeof(float));
    if (e == cudaSuccess)
        e = cudaMemcpy(*dev, h, n * sizeof(float), cudaMemcpyHostToDevice);
    free(h);
    return e != cudaSuccess;
}

static int same(const float *a, const float *b, size_t n, const char *what)
{
    float *ha = (float *)malloc(n * sizeof(float)), *hb = (float *)malloc(n * sizeof(float));
    int ok = ha && hb && cudaMemcpy(ha, a, n * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess &&
             cudaMemcpy(hb, b, n * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess &&
             memcmp(ha, hb, n * sizeof(float)) == 0;
    if (!ok)
        fprintf(stderr, "%s differs\n", what);
    free(ha);
    free(hb);
    return ok;
}

int main(void)
{
    const int B = 2, Hq = 1, Hv = 2, d = 128, W = 4, T = 2;
    const int conv_dim = (2 * Hq + Hv) * d;
    gdn_dims dims = {B, Hq, Hv, d, W, 0, conv_dim, (int64_t)Hv * d, Hv};
    float *x, *z, *alpha, *blog, *conv_w, *dt, *A_log, *norm_w, *state0, *hist0;
    if (fill(&x, (size_t)B * T * conv_dim, 1.0f) || fill(&z, (size_t)B * T * Hv * d, 1.0f) ||
        fill(&alpha, (size_t)B * T * Hv, 1.0f) || fill(&blog, (size_t)B * T * Hv, 1.0f) ||
        fill(&conv_w, (size_t)conv_dim * W, 0.5f) || fill(&dt, Hv, 1.0f) ||
        fill(&A_log, Hv, 1.0f) || fill(&norm_w, d, 1.0f) ||
        fill(&state0, (size_t)B * Hv * d * d, 0.1f) || fill(&hist0, (size_t)B * conv_dim * (W - 1), 1.0f))
        return 1;
    const gdn_params params = {conv_w, dt, A_log, norm_w, 1e-6f, 1e-6f};
    const size_t ns = (size_t)B * Hv * d * d, nh = (size_t)B * conv_dim * (W - 1);
    const size_t no = (size_t)B * T * Hv * d;
    float *s1, *h1, *s2, *h2, *o1, *o2, *step;
    CUDA(cudaMalloc((void **)&s1, ns * 4));
    CUDA(cudaMalloc((void **)&s2, ns * 4));
    CUDA(cudaMalloc((void **)&h1, nh * 4));
    CUDA(cudaMalloc((void **)&h2, nh * 4));
    CUDA(cudaMalloc((void **)&o1, no * 4));
    CUDA(cudaMalloc((void **)&o2, no * 4));
    CUDA(cudaMalloc((void **)&step, (size_t)B * Hv * d * 4));
    CUDA(cudaMemcpy(s1, state0, ns * 4, cudaMemcpyDeviceToDevice));
    CUDA(cudaMemcpy(s2, state0, ns * 4, cudaMemcpyDeviceToDevice));
    CUDA(cudaMemcpy(h1, hist0, nh * 4, cudaMemcpyDeviceToDevice));
    CUDA(cudaMemcpy(h2, hist0, nh * 4, cudaMemcpyDeviceToDevice));

    /* two single-token steps: token t of sequence b is row b*T + t, so each step
       reads rows T apart */
    gdn_dims one = dims;
    one.x_stride = (int64_t)conv_dim * T;
    one.z_stride = (int64_t)Hv * d * T;
    one.gate_stride = (int64_t)Hv * T;
    for (int t = 0; t < T; ++t) {
        CHECK(gdn_decode_step(s1, h1, x + (size_t)t * conv_dim, z + (size_t)t * Hv * d,
                              alpha + (size_t)t * Hv, blog + (size_t)t * Hv, GDN_F32, &params, step,
                              &one, NULL));
        for (int b = 0; b < B; ++b)
            CUDA(cudaMemcpy(o1 + ((size_t)b * T + t) * Hv * d, step + (size_t)b * Hv * d,
                            (size_t)Hv * d * 4, cudaMemcpyDeviceToDevice));
    }
    /* one two-token scan from the same start */
    CHECK(gdn_layer_scan(s2, h2, x, z, alpha, blog, GDN_F32, &params, o2, &dims, T, NULL));
    CUDA(cudaDeviceSynchronize());
    int32_t code = -1;
    CHECK(gdn_check_device(&code));
    if (code != 0 || !same(o1, o2, no, "outputs") || !same(s1, s2, ns, "state") ||
        !same(h1, h2, nh, "conv history"))
        return 1;
    /* host-side validation: a null state is rejected before any launch */
    if (gdn_decode_step(NULL, h1, x, z, alpha, blog, GDN_F32, &params, step, &dims, NULL) !=
        GDN_ERR_INVALID_ARG)
        return 1;
    printf("c client ok: %s\n", gdn_version());
    return 0;
}
