// dgt_layer.cu -- the small kernels between the products of one decoder-layer
// decode step (batch 1): residual add + RMS norm, SiLU(gate) * up, and the
// grouped-query repeat that stands in for attention.
//
// Binade README, "Results" (decode speed: a whole model's per-token time with
// R4 weights against BF16) and "How it works" (the products are the only part
// the format changes).  Each step here has one fixed order, so a decode step
// with R4 weights and one with the same weights in BF16 give bit-identical
// outputs: the products are twins and these kernels are shared.
#include <cuda_runtime.h>

#include "../../include/dgt.h"
#include "dgt_device.cuh"
#include "dgt_launch.h"

namespace dgt {

constexpr uint32_t NORM_THREADS = 1024;
constexpr uint64_t NORM_MAX = 65536;

// One CTA: x += y (if y), then h = bf16((x * r) * gamma) with
// r = 1 / sqrt(ss / n + eps).  ss: thread t sums x_i^2 over i = t, t + 1024,
// ... in increasing i (fmaf from +0); each warp adds its lanes by the
// butterfly 16, 8, 4, 2, 1; warp 0 does the same over the 32 warp sums.
__global__ void __launch_bounds__(NORM_THREADS) k_add_rmsnorm(float *__restrict__ x, const float *__restrict__ y,
                                                             const uint16_t *__restrict__ gamma, uint32_t n,
                                                             float eps, uint16_t *__restrict__ h) {
    __shared__ float part[32];
    __shared__ float rs;
    pdl_trigger();
    pdl_wait();
    const uint32_t t = threadIdx.x, lane = t & 31, w = t >> 5;
    float acc = 0.0f;
    for (uint32_t i = t; i < n; i += NORM_THREADS) {
        float v = x[i];
        if (y) {
            v = v + y[i];
            x[i] = v;
        }
        acc = fmaf(v, v, acc);
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) acc += __shfl_xor_sync(DGT_FULL, acc, d);
    if (lane == 0) part[w] = acc;
    __syncthreads();
    if (w == 0) {
        float s = part[lane];
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) s += __shfl_xor_sync(DGT_FULL, s, d);
        if (lane == 0) rs = 1.0f / sqrtf(s / (float)n + eps);
    }
    __syncthreads();
    const float r = rs;
    for (uint32_t i = t; i < n; i += NORM_THREADS) {
        const float g = __uint_as_float((uint32_t)gamma[i] << 16);
        h[i] = f32_to_bf16_rne((x[i] * r) * g);
    }
}

// out = bf16((g / (1 + exp(-g))) * u), elementwise.
__global__ void __launch_bounds__(256) k_silu_mul(const float *__restrict__ g, const float *__restrict__ u,
                                                 uint64_t n, uint16_t *__restrict__ out) {
    pdl_trigger();
    pdl_wait();
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
        const float a = g[i];
        const float s = a / (1.0f + expf(-a));
        out[i] = f32_to_bf16_rne(s * u[i]);
    }
}

// Row r of gu holds [gate (n) | up (n)]: out[r, i] = bf16(silu(gate) * up),
// the same per-element arithmetic as k_silu_mul.
__global__ void __launch_bounds__(256) k_silu_mul_rows(const float *__restrict__ gu, uint32_t rows, uint64_t n,
                                                      uint16_t *__restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const uint64_t total = (uint64_t)rows * n;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t r = i / n, c = i - r * n;
        const float a = gu[r * 2 * n + c];
        const float s = a / (1.0f + expf(-a));
        out[i] = f32_to_bf16_rne(s * gu[r * 2 * n + n + c]);
    }
}

// out[i] = v[i mod n_in].
__global__ void __launch_bounds__(256) k_repeat(const uint16_t *__restrict__ v, uint64_t n_in, uint64_t n_out,
                                               uint16_t *__restrict__ out) {
    pdl_trigger();
    pdl_wait();
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_out;
         i += (uint64_t)gridDim.x * blockDim.x)
        out[i] = v[i % n_in];
}

// out[i] = fmaf(p[S-1], y[S-1][i], ... fmaf(p[0], y[0][i], +0)): the routed
// experts' outputs combined in slot order.
__global__ void __launch_bounds__(256) k_weighted_sum(const float *__restrict__ y, const float *__restrict__ p,
                                                     uint32_t slots, uint64_t n, float *__restrict__ out) {
    pdl_trigger();
    pdl_wait();
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
        float acc = 0.0f;
        for (uint32_t j = 0; j < slots; j++) acc = fmaf(p[j], y[(uint64_t)j * n + i], acc);
        out[i] = acc;
    }
}

static unsigned elem_grid(uint64_t n) {
    DeviceInfo di;
    const int sms = device_info(&di) == DGT_OK ? di.sms : 132;
    uint64_t g = (n + 255) / 256;
    if (g > (uint64_t)sms * 8) g = (uint64_t)sms * 8;
    return (unsigned)(g ? g : 1);
}

}  // namespace dgt

using namespace dgt;

extern "C" int dgt_add_rmsnorm(float *d_x, const float *d_y, const uint16_t *d_gamma, uint64_t n, float eps,
                               uint16_t *d_h, void *stream) {
    if (!d_x || !d_gamma || !d_h) return DGT_ERR_ARG;
    if (n == 0 || n > NORM_MAX) return DGT_ERR_SHAPE;
    if (!(eps >= 0.0f)) return DGT_ERR_ARG;
    return launch_pdl(k_add_rmsnorm, dim3(1), dim3(NORM_THREADS), 0, (cudaStream_t)stream, d_x, d_y, d_gamma,
                      (uint32_t)n, eps, d_h) == cudaSuccess
               ? DGT_OK
               : DGT_ERR_CUDA;
}

extern "C" int dgt_silu_mul(const float *d_g, const float *d_u, uint64_t n, uint16_t *d_out, void *stream) {
    if (!d_g || !d_u || !d_out) return DGT_ERR_ARG;
    if (n == 0) return DGT_OK;
    return launch_pdl(k_silu_mul, dim3(elem_grid(n)), dim3(256), 0, (cudaStream_t)stream, d_g, d_u, n, d_out) ==
                   cudaSuccess
               ? DGT_OK
               : DGT_ERR_CUDA;
}

extern "C" int dgt_silu_mul_rows(const float *d_gu, uint32_t rows, uint64_t n, uint16_t *d_out, void *stream) {
    if (!d_gu || !d_out) return DGT_ERR_ARG;
    if (n == 0 || rows == 0) return DGT_OK;
    const uint64_t total = (uint64_t)rows * n;
    if (total / rows != n) return DGT_ERR_SHAPE;
    return launch_pdl(k_silu_mul_rows, dim3(elem_grid(total)), dim3(256), 0, (cudaStream_t)stream, d_gu, rows, n,
                      d_out) == cudaSuccess
               ? DGT_OK
               : DGT_ERR_CUDA;
}

extern "C" int dgt_repeat(const uint16_t *d_v, uint64_t n_in, uint64_t n_out, uint16_t *d_out, void *stream) {
    if (!d_v || !d_out) return DGT_ERR_ARG;
    if (n_out == 0) return DGT_OK;
    if (n_in == 0) return DGT_ERR_SHAPE;
    return launch_pdl(k_repeat, dim3(elem_grid(n_out)), dim3(256), 0, (cudaStream_t)stream, d_v, n_in, n_out,
                      d_out) == cudaSuccess
               ? DGT_OK
               : DGT_ERR_CUDA;
}

extern "C" int dgt_weighted_sum(const float *d_y, const float *d_p, uint32_t slots, uint64_t n, float *d_out,
                                void *stream) {
    if (!d_y || !d_p || !d_out) return DGT_ERR_ARG;
    if (n == 0) return DGT_OK;
    if (slots == 0) return DGT_ERR_SHAPE;
    return launch_pdl(k_weighted_sum, dim3(elem_grid(n)), dim3(256), 0, (cudaStream_t)stream, d_y, d_p, slots, n,
                      d_out) == cudaSuccess
               ? DGT_OK
               : DGT_ERR_CUDA;
}
