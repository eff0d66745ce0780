// host_copy.cu -- whole-array copies between device memory and host memory the
// device can address (pinned), done by a kernel on every SM instead of the copy
// engines: on this machine the copy engines move about 200 GB/s per direction
// over the CPU-GPU link, while loads and stores issued from all SMs keep enough
// requests in flight to use more of it.  Used by mpm_step_host.
#include "common.cuh"
#include "internal.h"

namespace mpm {

// Up to kMaxCopies arrays of the same byte size; src/dst device-addressable.
struct CopyTable {
    const void *src[kMaxCopies];
    void *dst[kMaxCopies];
    int count;
    int vec;            // 1: every pointer 16-byte aligned and the size a multiple of 16
    int64_t bytes;      // per array
};

// Every thread moves U elements a round, all loads issued before the stores.
template <typename E, int U>
__device__ __forceinline__ void copy_one(const E *__restrict__ s, E *__restrict__ d, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + (U - 1) * stride < n; i += U * stride) {
        E r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r[u] = s[i + u * stride];
#pragma unroll
        for (int u = 0; u < U; ++u) d[i + u * stride] = r[u];
    }
    for (; i < n; i += stride) d[i] = s[i];
}

__global__ void __launch_bounds__(256) k_copy_table(CopyTable t) {
    for (int a = 0; a < t.count; ++a) {
        if (t.vec)
            copy_one<uint4, 4>(static_cast<const uint4 *>(t.src[a]), static_cast<uint4 *>(t.dst[a]), t.bytes / 16);
        else
            copy_one<uint32_t, 8>(static_cast<const uint32_t *>(t.src[a]), static_cast<uint32_t *>(t.dst[a]),
                                  t.bytes / 4);
    }
}

// The device address of host memory the device can reach (pinned), or null.
void *device_view_of_host(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

mpm_status launch_copy_table(const void *const *src, void *const *dst, int count, int64_t bytes,
                             const DeviceInfo &dev, cudaStream_t st) {
    if (count < 0 || count > kMaxCopies || bytes < 0 || bytes % 4) return MPM_E_ARG;
    if (count == 0 || bytes == 0) return MPM_OK;
    CopyTable t{};
    t.count = count;
    t.bytes = bytes;
    t.vec = bytes % 16 == 0;
    for (int a = 0; a < count; ++a) {
        t.src[a] = src[a];
        t.dst[a] = dst[a];
        t.vec = t.vec && (reinterpret_cast<uintptr_t>(src[a]) % 16 == 0) &&
                (reinterpret_cast<uintptr_t>(dst[a]) % 16 == 0);
    }
    k_copy_table<<<dev.sms * 8, 256, 0, st>>>(t);
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

}  // namespace mpm
