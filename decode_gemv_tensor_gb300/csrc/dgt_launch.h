// dgt_launch.h -- host-side launch helpers shared by libdgt's CUDA sources.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/dgt.h"

namespace dgt {

struct DeviceInfo {
    int device;
    int sms;
    int cc_major, cc_minor;
};

// The current device's SM count and compute capability, cached per device.
// Safe to call from several host threads at once: a cache entry is published
// (release) only after it is filled, and read only after that flag (acquire).
static inline int device_info(DeviceInfo *out) {
    static DeviceInfo cache[64];
    static std::atomic<bool> have[64];
    static std::mutex fill;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return DGT_ERR_CUDA;
    if (dev < 64 && have[dev].load(std::memory_order_acquire)) {
        *out = cache[dev];
        return DGT_OK;
    }
    DeviceInfo d;
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return DGT_ERR_CUDA;
    if (dev < 64) {
        std::lock_guard<std::mutex> lock(fill);
        if (!have[dev].load(std::memory_order_relaxed)) {
            cache[dev] = d;
            have[dev].store(true, std::memory_order_release);
        }
    }
    *out = d;
    return DGT_OK;
}

// Allow `smem` bytes of dynamic shared memory and report resident CTAs per SM.
static inline int prepare_kernel(const void *fn, size_t smem, int threads, int *blocks_per_sm) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DGT_ERR_CUDA;
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, smem) != cudaSuccess) return DGT_ERR_CUDA;
    *blocks_per_sm = b > 0 ? b : 1;
    return DGT_OK;
}

static inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream finishes (it must call pdl_wait() before
// touching anything that kernel writes, and write nothing before that).
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                     Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace dgt
