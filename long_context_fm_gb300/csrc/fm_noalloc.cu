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
// address is looked up with cudaGetSymbolAddress, once per CUDA context: the
// cache is keyed by the context's process-unique id (cuCtxGetId), so a context
// created after a device reset, or a non-primary context made current by the
// caller, gets its own lookup instead of a stale address.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fm.h"
#include "fm_internal.h"

namespace {

static __device__ __align__(256) unsigned char fm_noalloc_scratch[FM_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*PFN_ctxGetCurrent)(CUcontext *);
typedef CUresult (*PFN_ctxGetId)(CUcontext, unsigned long long *);

std::mutex g_mu;
constexpr int kCacheSlots = 64;
struct Slot {
    unsigned long long ctx_id;   // 0 = empty (context ids start at 1)
    void *addr;
};
Slot g_cache[kCacheSlots] = {};
int g_next = 0;

// Driver entry points through the runtime (the library links no libcuda).
bool driver_fns(PFN_ctxGetCurrent *cur, PFN_ctxGetId *id)
{
    static PFN_ctxGetCurrent f_cur = nullptr;
    static PFN_ctxGetId f_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f_cur = reinterpret_cast<PFN_ctxGetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f_id = reinterpret_cast<PFN_ctxGetId>(p);
    });
    *cur = f_cur;
    *id = f_id;
    return f_cur && f_id;
}

// Device address of the scratch array in the current context, looked up on
// the first call made with that context current.
fm_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FM_ERR_CUDA;
    PFN_ctxGetCurrent get_cur;
    PFN_ctxGetId get_id;
    if (!driver_fns(&get_cur, &get_id)) return FM_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_cur(&ctx) != CUDA_SUCCESS) return FM_ERR_CUDA;
    void *p = nullptr;
    if (!ctx) {
        // No context is current yet: the symbol lookup makes the runtime
        // bind the device's primary context (it allocates nothing).
        if (cudaGetSymbolAddress(&p, fm_noalloc_scratch) != cudaSuccess || !p) return FM_ERR_CUDA;
        if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return FM_ERR_CUDA;
    }
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS || id == 0) return FM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    for (const Slot &s : g_cache)
        if (s.ctx_id == id) {
            *out = s.addr;
            return FM_OK;
        }
    if (!p && (cudaGetSymbolAddress(&p, fm_noalloc_scratch) != cudaSuccess || !p)) return FM_ERR_CUDA;
    g_cache[g_next] = Slot{id, p};          // oldest entry replaced once all slots are used
    g_next = (g_next + 1) % kCacheSlots;
    *out = p;
    return FM_OK;
}

}  // namespace

extern "C" fm_status fm_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                         int o_dtype, const float *lse, const void *dO, fm_bounds m,
                                         const void *plan, int B, int H, int N, int d, float scale,
                                         void *dq, void *dk, void *dv, int grad_dtype, int flags,
                                         int32_t *dev_status, fm_stream_t stream)
{
    // Shape errors are reported exactly as fm_attn_bwd reports them.
    const fm_status shapes = fm::check_shapes(B, H, N, d);
    if (shapes != FM_OK) return shapes;
    const size_t need = fm_bwd_workspace_bytes(B, H, N, d);
    if (need == 0) return FM_ERR_INVALID_ARG;
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
