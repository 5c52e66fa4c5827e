// C ABI entry points: argument validation, TMA descriptor encoding, launch
// sequencing and the per-kernel event profiler.  See include/fm.h for the
// contract of each call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "fm_internal.h"
#include "fm_ptx.cuh"

using namespace fm;

// Launchers in the kernel translation units.
fm_status fm_classify_launch(fm_bounds m, int q_row0, int Nq, int bq, int bk, void *plan, uint8_t *labels,
                             int32_t *status, cudaStream_t stream);
fm_status fm_bwd_pre_launch(const void *o, int o_f32, const void *dO, float *Dout, float *dq_acc,
                            int64_t rows, int d, cudaStream_t stream);
fm_status fm_bwd_post_launch(const float *dq_acc, void *dq, float scale, int64_t n, cudaStream_t stream);
fm_status fm_fwd_prepare(int d, bool precise);
fm_status fm_fwd_prepare_fp8();
fm_status fm_fwd_launch_fp8(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tvt,
                            const CUtensorMap &to, const FwdArgs &a, cudaStream_t stream);
fm_status fm_bwd_prepare(int d, bool precise);
fm_status fm_fwd_launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const CUtensorMap &to, const FwdArgs &a, int d, bool precise, cudaStream_t stream);
fm_status fm_bwd_main_launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const CUtensorMap &tdo, const CUtensorMap &tdk, const CUtensorMap &tdv,
                             const BwdArgs &a, int d, bool precise, cudaStream_t stream);

namespace {

constexpr int kAbiVersion = 6;

bool aligned16(const void *p) { return p && ((uintptr_t)p & 15u) == 0; }

// ---- driver entry point for tensor-map encoding --------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// bf16 [BH, N, d] viewed as 3-D (d, N, BH); box = 64 columns x `rows` rows,
// 128-byte swizzle, zero fill outside the tensor (ragged N).
bool make_tmap_bf16(CUtensorMap *map, const void *base, int BH, int N, int d, int rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// uint8 [BH, rows, cols] viewed as 3-D (cols, rows, BH); box = 128 columns x
// `box_rows` rows, 128-byte swizzle (one box spans a 128-byte row), zero fill.
bool make_tmap_u8(CUtensorMap *map, const void *base, int BH, int rows, int cols, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)rows * cols};
    const cuuint32_t box[3] = {128, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// O, fp32 or bf16 [BH, rows, d], viewed as 3-D (d, rows, BH) for TMA stores:
// box = 64 bytes (16 fp32 or 32 bf16 columns) x 32 rows, 64-byte swizzle; rows
// at or beyond `rows` are not written.
bool make_tmap_out(CUtensorMap *map, void *base, int BH, int rows, int d, bool f32)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t esz = f32 ? 4 : 2;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)d * esz, (cuuint64_t)rows * d * esz};
    const cuuint32_t box[3] = {(cuuint32_t)(64 / esz), 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base,
                          dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// dK or dV, fp32 or bf16 [BH, rows, d], viewed as 3-D (d, rows, BH) for TMA
// stores of 32 columns x 32 rows: fp32 boxes of 128-byte rows with the
// 128-byte swizzle, bf16 boxes of 64-byte rows with the 64-byte swizzle; rows
// at or beyond `rows` are not written.
bool make_tmap_grad(CUtensorMap *map, void *base, int BH, int rows, int d, bool f32)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t esz = f32 ? 4 : 2;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)d * esz, (cuuint64_t)rows * d * esz};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base,
                          dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

fm_status check_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FM_ERR_CUDA;
    static int cached[64];
    static std::once_flag once;
    std::call_once(once, [] { std::memset(cached, 0, sizeof(cached)); });
    if (dev < 0 || dev >= 64) return FM_ERR_UNSUPPORTED;
    if (cached[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FM_ERR_CUDA;
        cached[dev] = (major == 10 && minor == 3) ? 1 : 2;   // built for sm_103a only
    }
    return cached[dev] == 1 ? FM_OK : FM_ERR_UNSUPPORTED;
}

fm_status check_bounds(const fm_bounds &m, int B, int H, int N)
{
    if (!aligned16(m.lts) || !aligned16(m.lte) || !aligned16(m.uts) || !aligned16(m.ute))
        return FM_ERR_INVALID_ARG;
    if (m.B != B || m.N != N || !(m.Hm == 1 || m.Hm == H)) return FM_ERR_INVALID_ARG;
    return FM_OK;
}

// ---- wait test hook --------------------------------------------------------------
// One-shot, set only by fm_debug_wait_test: the next forward (kernel 0) or
// backward main (kernel 1) launch runs with a short wait bound and its first
// CTA withholds one tile load.
std::atomic<int> g_dbg_kernel{-1};
std::atomic<long long> g_dbg_limit{0};

void wait_test_args(int kernel, long long *limit, int *withhold)
{
    *limit = kWaitLimitCycles;
    *withhold = 0;
    int want = kernel;
    if (g_dbg_kernel.load(std::memory_order_acquire) == kernel &&
        g_dbg_kernel.compare_exchange_strong(want, -1, std::memory_order_acq_rel)) {
        *limit = g_dbg_limit.load(std::memory_order_acquire);
        *withhold = 1;
    }
}

// ---- profiler ------------------------------------------------------------------
struct ProfRec {
    int kernel;
    cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
constexpr size_t kProfMax = 4096;

}  // namespace

namespace fm {
int device_sm_count()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int v = cached[dev].load(std::memory_order_acquire);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 0;
    cached[dev].store(v, std::memory_order_release);
    return v;
}

fm_status check_shapes(int B, int H, int N, int d)
{
    if (B <= 0 || H <= 0 || N <= 0) return FM_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FM_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535) return FM_ERR_UNSUPPORTED;
    if ((int64_t)B * H * N * d > ((int64_t)1 << 40)) return FM_ERR_INVALID_ARG;
    if ((int64_t)B * H > (1 << 30)) return FM_ERR_UNSUPPORTED;
    return FM_OK;
}

ProfScope::ProfScope(int kernel, void *st) : slot(-1), stream(st)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on || g_prof.size() >= kProfMax) return;
    // Launches being captured into a graph are not timed (their events would
    // become graph nodes).
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing((cudaStream_t)st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return;
    ProfRec r{kernel, nullptr, nullptr};
    if (cudaEventCreate(&r.a) != cudaSuccess) return;
    if (cudaEventCreate(&r.b) != cudaSuccess) {
        cudaEventDestroy(r.a);
        return;
    }
    cudaEventRecord(r.a, (cudaStream_t)st);
    g_prof.push_back(r);
    slot = (int)g_prof.size() - 1;
}
ProfScope::~ProfScope()
{
    if (slot < 0) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (slot < (int)g_prof.size()) cudaEventRecord(g_prof[slot].b, (cudaStream_t)stream);
}
}  // namespace fm

// ---- wait-timeout self-test kernel ----------------------------------------------------
__global__ void fm_selftest_wait_kernel(long long limit, int32_t *status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);   // one arrival expected; nothing ever arrives
        fence_barrier_init();
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0, &abort_flag, status, limit);
    if (ok) set_status(status, -1);   // impossible: nothing completes the phase
}

// =====================================================================================
extern "C" {

const char *fm_status_string(fm_status st)
{
    switch (st) {
    case FM_OK: return "ok";
    case FM_ERR_INVALID_ARG: return "invalid argument";
    case FM_ERR_UNSUPPORTED: return "unsupported shape, tile size or device";
    case FM_ERR_UNREPRESENTABLE: return "mask not representable with two masked ranges per column";
    case FM_ERR_BAD_BOUNDS: return "mask bound outside [0, N]";
    case FM_ERR_PLAN_MISMATCH: return "plan does not match the call";
    case FM_ERR_WORKSPACE: return "workspace missing or too small";
    case FM_ERR_CUDA: return "CUDA error";
    case FM_ERR_TIMEOUT: return "device-side wait timed out";
    case FM_ERR_DEBUG_CHECK: return "device-side check of a debug build failed";
    }
    return "unknown status";
}

int fm_abi_version(void) { return kAbiVersion; }

size_t fm_plan_bytes_rows(int B, int Hm, int N, int q_row0, int Nq, int bq, int bk)
{
    PlanLayout L;
    if (!plan_layout(B, Hm, N, bq, bk, &L, q_row0, Nq)) return 0;
    return (size_t)L.total;
}

size_t fm_plan_bytes(int B, int Hm, int N, int bq, int bk)
{
    return fm_plan_bytes_rows(B, Hm, N, 0, N, bq, bk);
}

fm_status fm_tile_classify_rows(fm_bounds m, int q_row0, int Nq, int bq, int bk, void *plan, size_t plan_bytes,
                                uint8_t *labels, int32_t *dev_status, fm_stream_t stream)
{
    PlanLayout L;
    if (!plan_layout(m.B, m.Hm, m.N, bq, bk, &L, q_row0, Nq)) return FM_ERR_INVALID_ARG;
    if (!plan || ((uintptr_t)plan & 255u) || plan_bytes < (size_t)L.total) return FM_ERR_WORKSPACE;
    if (!dev_status || ((uintptr_t)dev_status & 3u)) return FM_ERR_INVALID_ARG;
    if (!aligned16(m.lts) || !aligned16(m.lte) || !aligned16(m.uts) || !aligned16(m.ute))
        return FM_ERR_INVALID_ARG;
    if ((int64_t)m.B * m.Hm > 65535) return FM_ERR_UNSUPPORTED;
    const fm_status dv = check_device();
    if (dv != FM_OK) return dv;
    return fm_classify_launch(m, q_row0, Nq, bq, bk, plan, labels, dev_status, (cudaStream_t)stream);
}

fm_status fm_tile_classify(fm_bounds m, int bq, int bk, void *plan, size_t plan_bytes, uint8_t *labels,
                           int32_t *dev_status, fm_stream_t stream)
{
    return fm_tile_classify_rows(m, 0, m.N, bq, bk, plan, plan_bytes, labels, dev_status, stream);
}

size_t fm_fwd_workspace_bytes(int B, int H, int N, int d)
{
    (void)B; (void)H; (void)N; (void)d;
    return 0;
}

fm_status fm_attn_fwd_rows(const void *q, const void *k, const void *v, fm_bounds m, const void *plan, int B,
                           int H, int N, int q_row0, int Nq, int d, float scale, void *o, int o_dtype, float *lse,
                           void *ws, size_t ws_bytes, int flags, int32_t *dev_status, fm_stream_t stream)
{
    (void)ws; (void)ws_bytes;
    if (flags & ~FM_FLAG_PRECISE) return FM_ERR_INVALID_ARG;
    fm_status st = check_shapes(B, H, N, d);
    if (st != FM_OK) return st;
    if ((st = check_bounds(m, B, H, N)) != FM_OK) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FM_ERR_INVALID_ARG;
    if (!dev_status || ((uintptr_t)dev_status & 3u)) return FM_ERR_INVALID_ARG;
    if (o_dtype != FM_DT_BF16 && o_dtype != FM_DT_F32) return FM_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return FM_ERR_INVALID_ARG;
    PlanLayout L;
    if (!plan_layout(B, m.Hm, N, 128, 128, &L, q_row0, Nq)) return FM_ERR_INVALID_ARG;
    if (!plan || ((uintptr_t)plan & 255u)) return FM_ERR_INVALID_ARG;
    if ((st = check_device()) != FM_OK) return st;
    CUtensorMap tq, tk, tv, to;
    if (!make_tmap_bf16(&tq, q, B * H, Nq, d, 128) || !make_tmap_bf16(&tk, k, B * H, N, d, 128) ||
        !make_tmap_bf16(&tv, v, B * H, N, d, 128) || !make_tmap_out(&to, o, B * H, Nq, d, o_dtype == FM_DT_F32))
        return FM_ERR_CUDA;
    FwdArgs a;
    a.lts = m.lts; a.lte = m.lte; a.uts = m.uts; a.ute = m.ute;
    a.plan = (const uint8_t *)plan; a.L = L;
    a.o = o; a.lse = lse; a.status = dev_status;
    a.B = B; a.H = H; a.Hm = m.Hm; a.N = N;
    a.q_row0 = q_row0; a.Nq = Nq;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.o_f32 = o_dtype == FM_DT_F32;
    a.descale = nullptr;
    wait_test_args(0, &a.wait_limit, &a.withhold);
    return fm_fwd_launch(tq, tk, tv, to, a, d, (flags & FM_FLAG_PRECISE) != 0, (cudaStream_t)stream);
}

fm_status fm_attn_fwd_fp8(const uint8_t *q8, const uint8_t *k8, const uint8_t *vt8, const float *descale,
                          fm_bounds m, const void *plan, int B, int H, int N, int d, float scale, void *o,
                          int o_dtype, float *lse, int32_t *dev_status, fm_stream_t stream)
{
    fm_status st = check_shapes(B, H, N, d);
    if (st != FM_OK) return st;
    if (d != 128 || N % 16 != 0) return FM_ERR_UNSUPPORTED;
    if ((st = check_bounds(m, B, H, N)) != FM_OK) return st;
    if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o) || !aligned16(lse))
        return FM_ERR_INVALID_ARG;
    if (!descale || ((uintptr_t)descale & 3u)) return FM_ERR_INVALID_ARG;
    if (!dev_status || ((uintptr_t)dev_status & 3u)) return FM_ERR_INVALID_ARG;
    if (o_dtype != FM_DT_BF16 && o_dtype != FM_DT_F32) return FM_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return FM_ERR_INVALID_ARG;
    PlanLayout L;
    if (!plan_layout(B, m.Hm, N, 128, 128, &L)) return FM_ERR_INVALID_ARG;
    if (!plan || ((uintptr_t)plan & 255u)) return FM_ERR_INVALID_ARG;
    if ((st = check_device()) != FM_OK) return st;
    CUtensorMap tq, tk, tvt, to;
    if (!make_tmap_u8(&tq, q8, B * H, N, d, 128) || !make_tmap_u8(&tk, k8, B * H, N, d, 128) ||
        !make_tmap_u8(&tvt, vt8, B * H, d, N, d) || !make_tmap_out(&to, o, B * H, N, d, o_dtype == FM_DT_F32))
        return FM_ERR_CUDA;
    FwdArgs a;
    a.lts = m.lts; a.lte = m.lte; a.uts = m.uts; a.ute = m.ute;
    a.plan = (const uint8_t *)plan; a.L = L;
    a.o = o; a.lse = lse; a.status = dev_status;
    a.B = B; a.H = H; a.Hm = m.Hm; a.N = N;
    a.q_row0 = 0; a.Nq = N;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.o_f32 = o_dtype == FM_DT_F32;
    a.descale = descale;
    a.wait_limit = kWaitLimitCycles;
    a.withhold = 0;
    return fm_fwd_launch_fp8(tq, tk, tvt, to, a, (cudaStream_t)stream);
}

fm_status fm_attn_fwd(const void *q, const void *k, const void *v, fm_bounds m, const void *plan, int B,
                      int H, int N, int d, float scale, void *o, int o_dtype, float *lse, void *ws,
                      size_t ws_bytes, int flags, int32_t *dev_status, fm_stream_t stream)
{
    return fm_attn_fwd_rows(q, k, v, m, plan, B, H, N, 0, N, d, scale, o, o_dtype, lse, ws, ws_bytes, flags,
                            dev_status, stream);
}

size_t fm_bwd_workspace_bytes(int B, int H, int N, int d)
{
    if (check_shapes(B, H, N, d) != FM_OK) return 0;
    const int64_t acc = align256((int64_t)B * H * N * d * 4);
    const int64_t dvec = align256((int64_t)B * H * N * 4);
    return (size_t)(acc + dvec);
}

fm_status fm_attn_bwd_rows(const void *q, const void *k, const void *v, const void *o, int o_dtype,
                           const float *lse, const void *dO, fm_bounds m, const void *plan, int B, int H,
                           int N, int q_row0, int Nq, int d, float scale, void *dq, void *dk, void *dv,
                           int grad_dtype, int flags, void *ws, size_t ws_bytes, int32_t *dev_status,
                           fm_stream_t stream)
{
    if (flags & ~FM_FLAG_PRECISE) return FM_ERR_INVALID_ARG;
    fm_status st = check_shapes(B, H, N, d);
    if (st != FM_OK) return st;
    if ((st = check_bounds(m, B, H, N)) != FM_OK) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return FM_ERR_INVALID_ARG;
    if (!dev_status || ((uintptr_t)dev_status & 3u)) return FM_ERR_INVALID_ARG;
    if ((o_dtype != FM_DT_BF16 && o_dtype != FM_DT_F32) ||
        (grad_dtype != FM_DT_BF16 && grad_dtype != FM_DT_F32))
        return FM_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return FM_ERR_INVALID_ARG;
    PlanLayout L;
    if (!plan_layout(B, m.Hm, N, 128, 128, &L, q_row0, Nq)) return FM_ERR_INVALID_ARG;
    const size_t need = fm_bwd_workspace_bytes(B, H, Nq, d);
    if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < need) return FM_ERR_WORKSPACE;
    if (!plan || ((uintptr_t)plan & 255u)) return FM_ERR_INVALID_ARG;
    if ((st = check_device()) != FM_OK) return st;
    CUtensorMap tq, tk, tv, tdo, tdk, tdv;
    float *dq_acc = reinterpret_cast<float *>(ws);
    if (!make_tmap_bf16(&tq, q, B * H, Nq, d, 64) || !make_tmap_bf16(&tk, k, B * H, N, d, 128) ||
        !make_tmap_bf16(&tv, v, B * H, N, d, 128) || !make_tmap_bf16(&tdo, dO, B * H, Nq, d, 64) ||
        !make_tmap_grad(&tdk, dk, B * H, N, d, grad_dtype == FM_DT_F32) ||
        !make_tmap_grad(&tdv, dv, B * H, N, d, grad_dtype == FM_DT_F32))
        return FM_ERR_CUDA;
    float *Dvec = reinterpret_cast<float *>((uint8_t *)ws + align256((int64_t)B * H * Nq * d * 4));
    const int64_t rows = (int64_t)B * H * Nq;
    cudaStream_t s = (cudaStream_t)stream;
    // fp32 gradients: dQ is accumulated (already scaled) in the caller's dq,
    // so no postprocess pass; bf16 gradients: unscaled in the workspace, then
    // scaled and converted by the postprocess.
    const bool dq_direct = grad_dtype == FM_DT_F32;
    if (dq_direct) dq_acc = reinterpret_cast<float *>(dq);
    if ((st = fm_bwd_pre_launch(o, o_dtype == FM_DT_F32, dO, Dvec, dq_acc, rows, d, s)) != FM_OK) return st;
    BwdArgs a;
    a.lts = m.lts; a.lte = m.lte; a.uts = m.uts; a.ute = m.ute;
    a.plan = (const uint8_t *)plan; a.L = L;
    a.lse = lse; a.Dvec = Dvec; a.dq_acc = dq_acc;
    a.dq_mul = dq_direct ? scale : 1.f;
    a.dk = dk; a.dv = dv; a.status = dev_status;
    a.B = B; a.H = H; a.Hm = m.Hm; a.N = N;
    a.q_row0 = q_row0; a.Nq = Nq;
    a.scale = scale; a.scale_log2 = scale * 1.4426950408889634f;
    a.g_f32 = grad_dtype == FM_DT_F32;
    wait_test_args(1, &a.wait_limit, &a.withhold);
    if ((st = fm_bwd_main_launch(tq, tk, tv, tdo, tdk, tdv, a, d, (flags & FM_FLAG_PRECISE) != 0, s)) != FM_OK)
        return st;
    return dq_direct ? FM_OK : fm_bwd_post_launch(dq_acc, dq, scale, rows * d, s);
}

fm_status fm_attn_bwd(const void *q, const void *k, const void *v, const void *o, int o_dtype,
                      const float *lse, const void *dO, fm_bounds m, const void *plan, int B, int H,
                      int N, int d, float scale, void *dq, void *dk, void *dv, int grad_dtype,
                      int flags, void *ws, size_t ws_bytes, int32_t *dev_status, fm_stream_t stream)
{
    return fm_attn_bwd_rows(q, k, v, o, o_dtype, lse, dO, m, plan, B, H, N, 0, N, d, scale, dq, dk, dv,
                            grad_dtype, flags, ws, ws_bytes, dev_status, stream);
}

struct fm_step_graph_st {
    cudaGraphExec_t exec;
};

fm_status fm_step_graph_create(const fm_step_args *a, fm_step_graph *graph)
{
    if (!graph) return FM_ERR_INVALID_ARG;
    *graph = nullptr;
    if (!a) return FM_ERR_INVALID_ARG;
    // Everything that is not a stream operation happens before the capture:
    // device check, the driver's tensor-map entry point, kernel attributes.
    fm_status st = check_device();
    if (st != FM_OK) return st;
    if (!encode_fn()) return FM_ERR_CUDA;
    if (a->d != 64 && a->d != 128) return FM_ERR_UNSUPPORTED;
    const bool precise = (a->flags & FM_FLAG_PRECISE) != 0;
    if ((st = fm_fwd_prepare(a->d, precise)) != FM_OK) return st;
    if (a->dO && (st = fm_bwd_prepare(a->d, precise)) != FM_OK) return st;
    cudaStream_t s = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return FM_ERR_CUDA;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaStreamDestroy(s);
        return FM_ERR_CUDA;
    }
    const fm_stream_t fs = (fm_stream_t)s;
    st = fm_tile_classify(a->mask, 128, 128, a->plan, a->plan_bytes, nullptr, a->dev_status, fs);
    if (st == FM_OK)
        st = fm_attn_fwd(a->q, a->k, a->v, a->mask, a->plan, a->B, a->H, a->N, a->d, a->scale, a->o, a->o_dtype,
                         a->lse, nullptr, 0, a->flags, a->dev_status, fs);
    if (st == FM_OK && a->dO)
        st = fm_attn_bwd(a->q, a->k, a->v, a->o, a->o_dtype, a->lse, a->dO, a->mask, a->plan, a->B, a->H, a->N,
                         a->d, a->scale, a->dq, a->dk, a->dv, a->grad_dtype, a->flags, a->ws, a->ws_bytes,
                         a->dev_status, fs);
    cudaGraph_t g = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(s, &g);
    if (st == FM_OK && (ec != cudaSuccess || !g)) st = FM_ERR_CUDA;
    cudaGraphExec_t exec = nullptr;
    if (st == FM_OK && cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) st = FM_ERR_CUDA;
    if (g) cudaGraphDestroy(g);
    cudaStreamDestroy(s);
    if (st != FM_OK) {
        if (exec) cudaGraphExecDestroy(exec);
        cudaGetLastError();   // a failed capture leaves no sticky error for the caller
        return st;
    }
    fm_step_graph h = new (std::nothrow) fm_step_graph_st{exec};
    if (!h) {
        cudaGraphExecDestroy(exec);
        return FM_ERR_CUDA;
    }
    *graph = h;
    return FM_OK;
}

fm_status fm_step_graph_launch(fm_step_graph graph, fm_stream_t stream)
{
    if (!graph) return FM_ERR_INVALID_ARG;
    return cudaGraphLaunch(graph->exec, (cudaStream_t)stream) == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

fm_status fm_step_graph_destroy(fm_step_graph graph)
{
    if (!graph) return FM_ERR_INVALID_ARG;
    const cudaError_t e = cudaGraphExecDestroy(graph->exec);
    delete graph;
    return e == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

fm_status fm_profile_begin(void)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto &r : g_prof) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_prof.clear();
    g_prof_on = true;
    return FM_OK;
}

int fm_profile_end(fm_kernel_time *out, int max_entries)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_on = false;
    int n = 0;
    bool err = false;
    for (auto &r : g_prof) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
            err = true;
        if (out && n < max_entries) {
            out[n].kernel = r.kernel;
            out[n].ms = ms;
            ++n;
        }
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_prof.clear();
    return err ? -1 : n;
}

fm_status fm_debug_wait_test(int kernel, long long limit_cycles)
{
    if ((kernel != 0 && kernel != 1 && kernel != -1) || (kernel >= 0 && (limit_cycles < 100000 ||
                                                                        limit_cycles > kWaitLimitCycles)))
        return FM_ERR_INVALID_ARG;
    g_dbg_limit.store(limit_cycles, std::memory_order_release);
    g_dbg_kernel.store(kernel, std::memory_order_release);
    return FM_OK;
}

fm_status fm_selftest_wait_timeout(long long limit_cycles, int32_t *dev_status, fm_stream_t stream)
{
    if (!dev_status || limit_cycles <= 0 || limit_cycles > kWaitLimitCycles) return FM_ERR_INVALID_ARG;
    const fm_status dv = check_device();
    if (dv != FM_OK) return dv;
    fm_selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit_cycles, dev_status);
    return cudaPeekAtLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

}  // extern "C"
