// Backward pass for callers that cannot allocate device memory.
//
// Some callers of this library run where cudaMalloc is off limits: code that
// executes inside another framework's memory pool or allocator hooks,
// real-time or embedded loops that must not touch the allocator after start-up,
// and plugins that only ever receive the input and output buffers from their
// host.  fm_attn_bwd needs a caller-provided workspace (the fp32 dQ
// accumulator and the row sums D); fm_attn_bwd_noalloc takes that workspace
// from a fixed array compiled into the library instead.
//
// The array is a file-scope __device__ variable of FM_NOALLOC_SCRATCH_BYTES.
// A GPU that loads this part of the library (at the latest on the first call
// below) keeps the array until the process exits.  In host code the array's
// name is only a host-side stand-in, never a device address, so its device
// address is looked up once per device with cudaGetSymbolAddress.
#include <cuda_runtime.h>

#include <mutex>

#include "fm.h"
#include "fm_internal.h"

namespace {

static __device__ __align__(256) unsigned char fm_noalloc_scratch[FM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on the
// first call made with that device current.
fm_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, fm_noalloc_scratch) != cudaSuccess || !p) return FM_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return FM_OK;
}

}  // namespace

extern "C" fm_status fm_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                         int o_dtype, const float *lse, const void *dO, fm_bounds m,
                                         const void *plan, int B, int H, int N, int d, float scale,
                                         void *dq, void *dk, void *dv, int grad_dtype, int flags,
                                         int32_t *dev_status, fm_stream_t stream)
{
    const size_t need = fm_bwd_workspace_bytes(B, H, N, d);
    if (need == 0) return (d == 64 || d == 128) ? FM_ERR_INVALID_ARG : FM_ERR_UNSUPPORTED;
    if (need > (size_t)FM_NOALLOC_SCRATCH_BYTES) return FM_ERR_WORKSPACE;
    void *ws = nullptr;
    const fm_status st = scratch_address(&ws);
    if (st != FM_OK) return st;
    // The backward's preprocess zeroes the dQ accumulator and writes every D
    // before the main kernel reads them, so the previous call's contents of
    // the array never leak into this one.
    return fm_attn_bwd(q, k, v, o, o_dtype, lse, dO, m, plan, B, H, N, d, scale, dq, dk, dv,
                       grad_dtype, flags, ws, (size_t)FM_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
