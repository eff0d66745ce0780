// static_ws.cu -- mpm_bin_static: the binning call with a workspace that
// lives in the library itself (a fixed-size device array), for callers that
// cannot hand the library device memory of their own.
//
// The array is file-scope device memory, created by the CUDA runtime when
// this file's device code is loaded; the library never calls an allocator
// for it.  Its device address is looked up on every call, with the caller's
// device current (the lookup is cheap next to the binning), so no address
// outlives the context it belongs to.  Everything else is the ordinary
// mpm_bins_init + mpm_bin on that memory, so the results are the same as
// mpm_bin's.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/mpm.h"

namespace {

// One workspace per device (a __device__ variable has one instance per
// device context).  Nothing in it must be zero beforehand: mpm_bin clears the
// counters and status words it uses at the start of every call.
static __device__ __align__(256) unsigned char g_static_ws[MPM_STATIC_WORKSPACE_BYTES];

// Device address of g_static_ws on the current device (the first lookup on a
// device may load this file's device code).
mpm_status static_ws_ptr(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MPM_E_NO_DEVICE;
    }
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ? MPM_E_NO_DEVICE : MPM_E_CUDA;
    }
    *out = p;
    return MPM_OK;
}

}  // namespace

extern "C" mpm_status mpm_bin_static(const mpm_grid_desc *desc, const mpm_particles *parts, int flags,
                                     mpm_bins *out, void *stream) {
    if (!desc || !parts || !out || parts->n < 0) return MPM_E_ARG;
    const size_t need = mpm_workspace_bytes(desc, parts->n);
    if (need == 0) return MPM_E_ARG;  // invalid descriptor
    if (need > (size_t)MPM_STATIC_WORKSPACE_BYTES) return MPM_E_WORKSPACE;
    void *ws = nullptr;
    const mpm_status s = static_ws_ptr(&ws);
    if (s != MPM_OK) return s;
    const mpm_status si = mpm_bins_init(desc, parts->n, ws, MPM_STATIC_WORKSPACE_BYTES, out);
    if (si != MPM_OK) return si;
    return mpm_bin(desc, parts, out, flags, stream);
}
