// dgt_stats.cu -- exponent statistics of a BF16 tensor: the histogram of its
// 8-bit exponents and the entropy of each tile's own exponent distribution.
//
// Binade README, "How it works" ("No exponent locality": per-tile palettes
// gain only 0.011 to 0.027 bits per weight over a shuffled tensor, so one
// frequency table per tensor is used) and the exponent-statistics scripts it
// lists.  The per-tile entropy H_t = -sum_e (c_e / T) log2(c_e / T) is the
// cost in bits per weight of coding a tile's exponents with its own ideal
// table (side information not counted); comparing its mean over the tensor
// with the same mean over a shuffled copy measures how much locality a
// palette scheme could use.
#include <cuda_runtime.h>

#include "../../include/dgt.h"
#include "dgt_device.cuh"
#include "dgt_launch.h"

namespace dgt {

constexpr uint32_t STAT_WARPS = 8;
constexpr uint32_t STAT_MAX_TILE = 65536;

// One warp per tile (grid-stride): the tile's exponent counts in the warp's
// shared histogram, its bits T_t * H_t (fp64; bins summed lane by lane, then
// the butterfly 16, 8, 4, 2, 1) written to tile_bits[t]; the counts are added
// into the CTA's histogram, which is added into hist at the end.
__global__ void __launch_bounds__(STAT_WARPS * 32) k_exp_stats(const uint16_t *__restrict__ w, uint64_t n,
                                                               uint32_t tile, unsigned long long *__restrict__ hist,
                                                               double *__restrict__ tile_bits) {
    __shared__ uint32_t th[STAT_WARPS][256];
    __shared__ uint32_t ch[256];
    pdl_trigger();
    pdl_wait();
    const uint32_t lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
    for (uint32_t i = threadIdx.x; i < 256; i += blockDim.x) ch[i] = 0;
    __syncthreads();
    const uint64_t ntiles = (n + tile - 1) / tile;
    for (uint64_t t = (uint64_t)blockIdx.x * STAT_WARPS + wp; t < ntiles; t += (uint64_t)gridDim.x * STAT_WARPS) {
        for (uint32_t b = lane; b < 256; b += 32) th[wp][b] = 0;
        __syncwarp();
        const uint64_t base = t * tile;
        const uint32_t cnt = (uint32_t)min((uint64_t)tile, n - base);
        for (uint32_t i = lane; i < cnt; i += 32) atomicAdd(&th[wp][(w[base + i] >> 7) & 0xFFu], 1u);
        __syncwarp();
        double bits = 0.0;
        for (uint32_t b = lane; b < 256; b += 32) {
            const uint32_t c = th[wp][b];
            if (c) {
                bits -= (double)c * log2((double)c / (double)cnt);
                atomicAdd(&ch[b], c);
            }
        }
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) bits += __shfl_xor_sync(DGT_FULL, bits, d);
        if (lane == 0) tile_bits[t] = bits;
        __syncwarp();
    }
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < 256; i += blockDim.x)
        if (ch[i]) atomicAdd(&hist[i], (unsigned long long)ch[i]);
}

// One CTA: out = sum of v[0..m) in a fixed order (thread t adds i = t,
// t + 1024, ... in increasing i; warp butterflies; warp 0 over the warp sums).
__global__ void __launch_bounds__(1024) k_sum_f64(const double *__restrict__ v, uint64_t m, double *__restrict__ out) {
    __shared__ double part[32];
    pdl_trigger();
    pdl_wait();
    const uint32_t lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
    double acc = 0.0;
    for (uint64_t i = threadIdx.x; i < m; i += 1024) acc += v[i];
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) acc += __shfl_xor_sync(DGT_FULL, acc, d);
    if (lane == 0) part[wp] = acc;
    __syncthreads();
    if (wp == 0) {
        double s = part[lane];
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) s += __shfl_xor_sync(DGT_FULL, s, d);
        if (lane == 0) out[0] = s;
    }
}

// One warp: out = -sum_e (c_e / n) log2(c_e / n) over the tensor's exponent
// counts (bins lane by lane, then the butterfly 16, 8, 4, 2, 1).
__global__ void __launch_bounds__(32) k_hist_entropy(const unsigned long long *__restrict__ hist, uint64_t n,
                                                     double *__restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const uint32_t lane = threadIdx.x;
    double h = 0.0;
    for (uint32_t b = lane; b < 256; b += 32) {
        const unsigned long long c = hist[b];
        if (c) h -= ((double)c / (double)n) * log2((double)c / (double)n);
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) h += __shfl_xor_sync(DGT_FULL, h, d);
    if (lane == 0) out[0] = h;
}

}  // namespace dgt

using namespace dgt;

extern "C" int dgt_exponent_stats(const uint16_t *d_w, uint64_t n, uint32_t tile, uint64_t *d_hist,
                                  double *d_tile_bits, double *d_total_bits, void *stream) {
    if (!d_w || !d_hist || !d_tile_bits || !d_total_bits) return DGT_ERR_ARG;
    if (n == 0 || tile == 0 || tile > STAT_MAX_TILE) return DGT_ERR_SHAPE;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(d_hist, 0, 256 * sizeof(uint64_t), st) != cudaSuccess) return DGT_ERR_CUDA;
    DeviceInfo di;
    if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
    const uint64_t ntiles = (n + tile - 1) / tile;
    uint64_t grid = (ntiles + STAT_WARPS - 1) / STAT_WARPS;
    if (grid > (uint64_t)di.sms * 8) grid = (uint64_t)di.sms * 8;
    if (launch_pdl(k_exp_stats, dim3((unsigned)grid), dim3(STAT_WARPS * 32), 0, st, d_w, n, tile,
                   reinterpret_cast<unsigned long long *>(d_hist), d_tile_bits) != cudaSuccess)
        return DGT_ERR_CUDA;
    if (launch_pdl(k_sum_f64, dim3(1), dim3(1024), 0, st, (const double *)d_tile_bits, ntiles, d_total_bits) !=
        cudaSuccess)
        return DGT_ERR_CUDA;
    if (launch_pdl(k_hist_entropy, dim3(1), dim3(32), 0, st, (const unsigned long long *)d_hist, n,
                   d_total_bits + 1) != cudaSuccess)
        return DGT_ERR_CUDA;
    return DGT_OK;
}
