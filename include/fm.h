/*
 * fm.h — C ABI of the GB300 (sm_103a) FlashMask-style masked attention library.
 *
 * The method (FlashMask, arXiv 2410.01359, abstract): attention masks are
 * carried as O(N) column-wise bounds instead of a dense N x N matrix, and the
 * kernels use them to skip (Q-tile, KV-tile) blocks that are fully masked,
 * run fully visible blocks without any mask arithmetic, and apply the
 * per-element mask only on the remaining boundary blocks (blog post
 * "FlashMask技术", §2.2, three-way block decision).  The result is plain
 * masked softmax attention, exactly (blog §2.2, "mathematically
 * equivalent"; abstract, "without sacrificing computational accuracy").
 *
 * Mask encoding used throughout: for batch b, mask head hm and key column j,
 *     lower masked rows [lts_j, lte_j)   and   upper masked rows [uts_j, ute_j)
 * (half-open; start >= end is an empty range; all values in [0, N]).
 * Element (i, j) is masked when query row i lies in either range.  The
 * arrays are int32 [B, Hm, N], row-major; Hm is 1 (one mask for all heads)
 * or H (one mask per head).  Head h reads mask head (Hm == 1 ? 0 : h).
 *
 * Tensors: Q, K, V, dO are bf16 [B, H, N, d] contiguous (d = 64 or 128);
 * lse is fp32 [B, H, N] (natural log); outputs are bf16 or fp32 [B, H, N, d].
 *
 * Conventions
 *  - Memory: every buffer is allocated by the caller.  The library allocates
 *    no device memory and keeps no pointer after a call returns.
 *  - Device calls are asynchronous on the given stream (NULL = legacy
 *    default stream).  Argument errors are returned before anything is
 *    launched.  Errors the device detects (a bound outside [0, N], a plan
 *    that does not match the call, a pipeline wait that ran out) are written
 *    to the caller's int32 dev_status (zero it first; the first error wins)
 *    and read by the caller after synchronising.
 *  - Device pointers must be 16-byte aligned.
 *  - Thread safety: calls may be made from several host threads.
 */
#ifndef FM_H_
#define FM_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FM_API __attribute__((visibility("default")))
#else
#define FM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FM_OK = 0,
    FM_ERR_INVALID_ARG = 1,      /* null / misaligned pointer, bad size or dtype          */
    FM_ERR_UNSUPPORTED = 2,      /* head dim, tile size or device not supported          */
    FM_ERR_UNREPRESENTABLE = 3,  /* row-form mask with > 2 masked ranges in some column  */
    FM_ERR_BAD_BOUNDS = 4,       /* a bound outside [0, N] (host or device detected)     */
    FM_ERR_PLAN_MISMATCH = 5,    /* plan built for other shapes or tile sizes            */
    FM_ERR_WORKSPACE = 6,        /* workspace missing or too small                       */
    FM_ERR_CUDA = 7,             /* a CUDA runtime / driver call failed                  */
    FM_ERR_TIMEOUT = 8,          /* a bounded device-side wait ran out (kernel returned) */
    FM_ERR_DEBUG_CHECK = 9       /* a device-side check of an FM_DEBUG build failed      */
} fm_status;

enum { FM_TILE_SKIP = 0, FM_TILE_FULL = 1, FM_TILE_PARTIAL = 2 };
enum { FM_DT_BF16 = 0, FM_DT_F32 = 1 };

/* Flags of fm_attn_fwd / fm_attn_bwd.
 * FM_FLAG_PRECISE: the softmax probabilities P (forward and backward) and dS
 * (backward) enter the tensor-core products as two bf16 terms, x = hi + lo
 * with hi = bf16(x), lo = bf16(x - hi), instead of one bf16 rounding.  The
 * products keep ~16 significant bits of P and dS (more tensor-core work:
 * 1.5x the forward PV product, 1.6x the backward products).  Without it the
 * kernels use the usual FlashAttention arithmetic (bf16 P and dS operands,
 * fp32 accumulation).  Use it when gradients are large (|dQ| of tens), where
 * one bf16 rounding of dS and of O (through D) shows in the result. */
enum { FM_FLAG_PRECISE = 1 };

/* Same type as cudaStream_t, so a cudaStream_t can be passed directly. */
typedef struct CUstream_st *fm_stream_t;

/* Column-bound mask; the four pointers are DEVICE arrays int32 [B, Hm, N]. */
typedef struct {
    const int32_t *lts, *lte, *uts, *ute;
    int32_t B, Hm, N;
} fm_bounds;

/* Human-readable name of a status code (static storage). */
FM_API const char *fm_status_string(fm_status st);

/* Library ABI version (incremented when a signature changes). */
FM_API int fm_abi_version(void);

/*
 * fm_mask_from_rows — HOST, synchronous.
 * Passage: blog "FlashMask技术" §2.1 (causal example) and §3.3 (document
 * packing): one inclusive attend interval [cs_i, ce_i] per query row.
 * cs, ce: host int32 [B, Hm, N]; cs_i > ce_i is an empty row; otherwise
 * 0 <= cs_i <= ce_i < N is required (else FM_ERR_BAD_BOUNDS).
 * Writes the column form to host arrays lts, lte, uts, ute [B, Hm, N]:
 * for each column the rows that do NOT attend it must form at most two
 * ranges (else FM_ERR_UNREPRESENTABLE, outputs then undefined).  A masked
 * range that starts at row 0 is stored as the upper range, any other (or the
 * second of two) as the lower range; empty ranges are written canonically,
 * lower (N, N) and upper (0, 0).  Runs in O(N) per (b, hm).
 */
FM_API fm_status fm_mask_from_rows(const int32_t *cs, const int32_t *ce, int B, int Hm, int N,
                            int32_t *lts, int32_t *lte, int32_t *uts, int32_t *ute);

/*
 * fm_mask_from_row_intervals — HOST, synchronous.
 * Passage: blog "FlashMask技术" §6.1 item 1 (multi-interval extension:
 * several disjoint attend intervals per row, printed as row 0 -> (0, 100),
 * (200, 300) and row 1 -> (0, 50), (150, 250)), read with the inclusive
 * interval convention of §3.3.  The window-with-sink-tokens mask of the §5
 * streaming-inference example (row i attends [0, sink) and (i - window, i])
 * is such a two-interval row form.
 * starts, ends: host int32 [B, Hm, N, K], K >= 1 interval slots per row;
 * slot (s, e) with s > e is unused; otherwise 0 <= s <= e < N is required
 * (else FM_ERR_BAD_BOUNDS).  Row i attends the union of its intervals, which
 * may overlap, touch or come in any order.  Output and errors as for
 * fm_mask_from_rows (which is the K = 1 case, with identical results): each
 * column's non-attending rows must form at most two ranges, else
 * FM_ERR_UNREPRESENTABLE.  Runs in O(N K log K) per (b, hm).
 */
FM_API fm_status fm_mask_from_row_intervals(const int32_t *starts, const int32_t *ends, int K, int B,
                                     int Hm, int N, int32_t *lts, int32_t *lte, int32_t *uts,
                                     int32_t *ute);

/*
 * Compressed column bounds.  Passage: blog "FlashMask技术" §6.2 item 2
 * (memory compression, next step: differential encoding of the interval
 * vectors and 8-bit integers for the offsets).  Per 128-column block of each
 * of the four bound arrays of each (b, hm): the block's first value as int32
 * and the 127 column-to-column differences as int8 when all fit in
 * [-128, 127], else the block's int32 values; a directory of per-block
 * offsets lets every block decode on its own.  Causal, window, prefix and
 * document masks compress about 3.7x (16 bytes per column to about 4.3).
 *
 * fm_bounds_compressed_bytes — HOST: the exact size of the compressed form of
 *   these host bounds (int32 [B, Hm, N] each), 0 on bad arguments.
 * fm_bounds_compress — HOST, synchronous: writes it into out (out_bytes at
 *   least that size, else FM_ERR_WORKSPACE; bad arguments FM_ERR_INVALID_ARG).
 *   Bounds are stored as given (validated when classified).
 * fm_bounds_decompress — DEVICE, async: expands a compressed buffer (device,
 *   16-byte aligned, `bytes` long) into the caller's device arrays `out`
 *   (whose B, Hm, N must be those it was compressed with).  A buffer whose
 *   header or directory does not match (wrong magic or shape, an entry beyond
 *   the payload) writes FM_ERR_INVALID_ARG to dev_status and nothing is read
 *   beyond `bytes`.  B * Hm <= 65535.
 */
FM_API size_t fm_bounds_compressed_bytes(const int32_t *lts, const int32_t *lte, const int32_t *uts,
                                         const int32_t *ute, int B, int Hm, int N);
FM_API fm_status fm_bounds_compress(const int32_t *lts, const int32_t *lte, const int32_t *uts,
                                    const int32_t *ute, int B, int Hm, int N, void *out, size_t out_bytes);
FM_API fm_status fm_bounds_decompress(const void *cbounds, size_t bytes, fm_bounds out, int32_t *dev_status,
                                      fm_stream_t stream);

/*
 * Plan = tile labels plus, per Q tile, the ordered list of non-skip KV tiles
 * and, per KV tile, the list of non-skip Q tiles (blog §4.1 item 2: decide
 * before a KV block is loaded whether it is needed at all), plus the order in
 * which the attention kernels take their tiles: longest list first, in
 * half-octave length buckets, so that a tile with a long list (sink columns,
 * the first tiles of a long document) starts in the first wave.  Opaque
 * device buffer of fm_plan_bytes() bytes, 256-byte aligned, written by
 * fm_tile_classify and read by fm_attn_fwd / fm_attn_bwd.
 * bq, bk in {64, 128}; the attention kernels need bq = bk = 128.
 * Returns 0 for invalid sizes.
 */
FM_API size_t fm_plan_bytes(int B, int Hm, int N, int bq, int bk);

/*
 * fm_tile_classify — DEVICE, async.
 * Passage: blog §2.2 (skip / full GEMM / masked GEMM per block pair).  The
 * printed test is garbled; the decision implemented is: per KV tile take the
 * min and max of each canonicalised bound (empty lower -> (N, N), empty
 * upper -> (0, 0)) over its columns; for Q rows [qb, qe) the pair is
 *   SKIP    if all columns' lower ranges cover [qb, qe) or all upper ones do,
 *   FULL    if not SKIP and every lower and every upper range misses [qb, qe),
 *   PARTIAL otherwise (tile ends clipped to N).
 * labels (nullable): device uint8 [B, Hm, n_q, n_k] copy of the labels.
 * dev_status: device int32 (required).  Bounds outside [0, N] set
 * FM_ERR_BAD_BOUNDS there.  Three launches on the stream: per-tile bound
 * min/max, labels and lists, work order.
 */
FM_API fm_status fm_tile_classify(fm_bounds m, int bq, int bk, void *plan, size_t plan_bytes,
                           uint8_t *labels, int32_t *dev_status, fm_stream_t stream);

/* Workspace of fm_attn_fwd in bytes (may be 0: then ws may be NULL). */
FM_API size_t fm_fwd_workspace_bytes(int B, int H, int N, int d);

/*
 * fm_attn_fwd — DEVICE, async.
 * Passages: FlashAttention article §二.1-二.3 (tiling, max-subtracted
 * softmax, QK^T and PV fused on tensor cores), blog §2.2 and §4.1 items 2-3
 * (skip blocks before loading them, mask fused into the softmax on boundary
 * blocks only).  Computes, per (b, h),
 *     O = softmax(scale * Q K^T with masked entries removed) V,
 *     lse_i = ln sum_{j attended} exp(scale q_i.k_j)
 * with O_i = 0 and lse_i = -inf for a row that attends nothing.
 * q, k, v: device bf16 [B, H, N, d]; plan from fm_tile_classify(m, 128, 128);
 * o: device [B, H, N, d] of o_dtype (FM_DT_BF16 / FM_DT_F32);
 * lse: device fp32 [B, H, N]; ws: fm_fwd_workspace_bytes() bytes or NULL;
 * flags: 0 or FM_FLAG_PRECISE.
 */
FM_API fm_status fm_attn_fwd(const void *q, const void *k, const void *v, fm_bounds m, const void *plan,
                      int B, int H, int N, int d, float scale, void *o, int o_dtype, float *lse,
                      void *ws, size_t ws_bytes, int flags, int32_t *dev_status,
                      fm_stream_t stream);

/* Workspace of fm_attn_bwd in bytes: fp32 dQ accumulator [B,H,N,d] plus
 * fp32 D = rowsum(dO * O) [B,H,N].  (With fp32 gradients the kernels
 * accumulate dQ in the caller's dq buffer directly and the accumulator
 * part of the workspace is left untouched; the size is the same for both
 * gradient dtypes.) */
FM_API size_t fm_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * fm_attn_bwd — DEVICE, async.
 * Exact gradient of fm_attn_fwd's O with upstream dO (lse has no upstream
 * gradient); the pages use the method for training (abstract: SFT, LoRA,
 * DPO, RM), which needs these.  With P_ij = exp(scale q_i.k_j - lse_i) on
 * attended pairs (0 elsewhere), D_i = sum_k dO_ik O_ik:
 *     dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),
 *     dQ = scale dS K,  dK = scale dS^T Q.
 * Same tile skipping as the forward.  o, lse: the forward's outputs (o of
 * o_dtype); dq, dk, dv: device [B, H, N, d] of grad_dtype; flags: 0 or
 * FM_FLAG_PRECISE (with a precise backward, compute O with a precise forward
 * too: D is taken from O); ws: fm_bwd_workspace_bytes() bytes (overwritten).
 */
FM_API fm_status fm_attn_bwd(const void *q, const void *k, const void *v, const void *o, int o_dtype,
                      const float *lse, const void *dO, fm_bounds m, const void *plan, int B,
                      int H, int N, int d, float scale, void *dq, void *dk, void *dv,
                      int grad_dtype, int flags, void *ws, size_t ws_bytes, int32_t *dev_status,
                      fm_stream_t stream);

/*
 * fm_attn_bwd_noalloc — DEVICE, async.  No counterpart in the paper: this
 * entry point exists for callers that may not allocate device memory (code
 * running under another framework's allocator, latency-critical loops that
 * must not call cudaMalloc after start-up, plugins handed only their input
 * and output buffers).  Same contract and results as fm_attn_bwd, but the
 * workspace comes from a fixed array inside the library instead of the
 * caller, so nothing is allocated.
 * Limit: fm_bwd_workspace_bytes(B, H, N, d) <= FM_NOALLOC_SCRATCH_BYTES
 * (64 MiB: about 130,000 rows B*H*N at d = 128); larger sizes return
 * FM_ERR_WORKSPACE before anything is launched.
 * The first call made in a CUDA context (the device's primary context, or a
 * context the caller made current) looks up the array's device address in
 * that context; make that first call before any stream capture.  The lookup
 * is cached per context id, so a context created later (after
 * cudaDeviceReset, for example) gets a fresh lookup on its first call.
 * A device that has loaded the array keeps it until the process exits.
 * Shape errors return the same codes as fm_attn_bwd.
 * Every call uses the same array: calls whose work overlaps on the GPU (for
 * example on two streams) race and give wrong results; calls ordered on one
 * stream are safe.  Each call clears what it needs; nothing carries over.
 */
#define FM_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
FM_API fm_status fm_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                     int o_dtype, const float *lse, const void *dO, fm_bounds m,
                                     const void *plan, int B, int H, int N, int d, float scale,
                                     void *dq, void *dk, void *dv, int grad_dtype, int flags,
                                     int32_t *dev_status, fm_stream_t stream);

/*
 * Row windows — the same three calls for the Q rows [q_row0, q_row0 + Nq) of
 * the N x N mask against all N key columns: one rank's share of a sequence
 * split over several GPUs (blog §4.3, sequence-parallel integration: the
 * column intervals all-gathered, each rank computing the rows it holds;
 * key/value shards a window's rows never attend are skipped whole by the
 * tile labels).  q_row0 must be a multiple of 128 (of bq for
 * fm_tile_classify_rows), 1 <= Nq, q_row0 + Nq <= N; else FM_ERR_INVALID_ARG.
 * The bounds keep the whole mask ([B, Hm, N], global row numbers).
 *   Q, dO, O: [B, H, Nq, d]; lse: [B, H, Nq]; K, V: [B, H, N, d].
 *   fm_attn_bwd_rows: dQ [B, H, Nq, d] is complete; dK, dV [B, H, N, d]
 *   receive this window's contribution only (zero where it attends nothing):
 *   the contributions of all windows add up to the full gradients.  The
 *   workspace is fm_bwd_workspace_bytes(B, H, Nq, d).
 * The plan of a window is fm_plan_bytes_rows(...) bytes and is built by
 * fm_tile_classify_rows with the same window.  Whole mask: q_row0 = 0, Nq = N
 * (what fm_plan_bytes, fm_tile_classify, fm_attn_fwd and fm_attn_bwd do).
 */
FM_API size_t fm_plan_bytes_rows(int B, int Hm, int N, int q_row0, int Nq, int bq, int bk);
FM_API fm_status fm_tile_classify_rows(fm_bounds m, int q_row0, int Nq, int bq, int bk, void *plan,
                                size_t plan_bytes, uint8_t *labels, int32_t *dev_status,
                                fm_stream_t stream);
FM_API fm_status fm_attn_fwd_rows(const void *q, const void *k, const void *v, fm_bounds m,
                           const void *plan, int B, int H, int N, int q_row0, int Nq, int d,
                           float scale, void *o, int o_dtype, float *lse, void *ws, size_t ws_bytes,
                           int flags, int32_t *dev_status, fm_stream_t stream);
FM_API fm_status fm_attn_bwd_rows(const void *q, const void *k, const void *v, const void *o,
                           int o_dtype, const float *lse, const void *dO, fm_bounds m,
                           const void *plan, int B, int H, int N, int q_row0, int Nq, int d,
                           float scale, void *dq, void *dk, void *dv, int grad_dtype, int flags,
                           void *ws, size_t ws_bytes, int32_t *dev_status, fm_stream_t stream);

/*
 * FP8 forward — DEVICE, async.  Passage: blog "FlashMask技术" §4.2 (the
 * H100 path computes in FP8); per-tensor scaling is the plainest reading.
 * fm_quantize_fp8: e4m3 codes of a bf16 [B, H, N, d] tensor with one scale,
 *   descale = amax / 448 (1 if amax = 0), code = e4m3(x / descale) (fp32
 *   division, round to nearest even, saturating at +-448; inputs finite).
 *   transpose = 0: x8 is [B, H, N, d]; 1: x8 is [B, H, d, N] (N a multiple
 *   of 16, else FM_ERR_UNSUPPORTED) — the layout fm_attn_fwd_fp8 wants for V.
 *   descale: device float, written.  d = 64 or 128.
 * fm_attn_fwd_fp8: fm_attn_fwd (whole mask, standard mode, d = 128) on e4m3
 *   q8, k8 [B, H, N, d] and vt8 [B, H, d, N] with descale = device float[3]
 *   (Q, K, V): S = scale * dq * dk * Q8 K8^T, P rounded to e4m3 for the P V
 *   product (P <= 256 under the lazy rescale), O = dv * (P V) / sum P.  N a
 *   multiple of 16; d != 128 -> FM_ERR_UNSUPPORTED.  Same plan, bounds and
 *   outputs as fm_attn_fwd.
 */
FM_API fm_status fm_quantize_fp8(const void *x, int B, int H, int N, int d, int transpose, uint8_t *x8,
                          float *descale, fm_stream_t stream);
FM_API fm_status fm_attn_fwd_fp8(const uint8_t *q8, const uint8_t *k8, const uint8_t *vt8,
                          const float *descale, fm_bounds m, const void *plan, int B, int H, int N,
                          int d, float scale, void *o, int o_dtype, float *lse, int32_t *dev_status,
                          fm_stream_t stream);

/*
 * Step graphs — create / destroy HOST, synchronous; launch DEVICE, async.
 * One step of the path (fm_tile_classify, fm_attn_fwd and, when dO is given,
 * fm_attn_bwd; 128 x 128 tiles) captured once into a CUDA graph for a fixed
 * set of buffers and replayed with a single launch.  Passages: blog §6.2
 * item 1 (capture the compute pattern in a CUDA Graph) and FlashAttention
 * article §三.3 (CUDA Graphs to cut kernel-launch overhead, which dominates
 * small problems).  Every launch reads the current contents of
 * the buffers in fm_step_args: refill q, k, v, dO and the bounds in place
 * between launches.  The caller keeps every buffer allocated and unmoved until
 * fm_step_graph_destroy, zeroes dev_status before reading it, and does not run
 * two launches on the same buffers concurrently.
 * fm_step_graph_create: argument errors are those of the three calls (the
 * capture is discarded, nothing is allocated); args or graph NULL ->
 * FM_ERR_INVALID_ARG; a failed capture -> FM_ERR_CUDA.  *graph is written on
 * success only (else set to NULL).
 */
typedef struct {
    const void *q, *k, *v;          /* bf16 [B, H, N, d] */
    const void *dO;                 /* bf16 [B, H, N, d], or NULL: forward-only graph */
    fm_bounds mask;
    void *plan;                     /* fm_plan_bytes(B, Hm, N, 128, 128) bytes */
    size_t plan_bytes;
    void *o;                        /* [B, H, N, d] of o_dtype */
    int o_dtype;
    float *lse;                     /* [B, H, N] */
    void *dq, *dk, *dv;             /* [B, H, N, d] of grad_dtype; unused without dO */
    int grad_dtype;
    void *ws;                       /* fm_bwd_workspace_bytes(B, H, N, d); unused without dO */
    size_t ws_bytes;
    int B, H, N, d;
    float scale;
    int flags;                      /* FM_FLAG_PRECISE or 0 */
    int32_t *dev_status;
} fm_step_args;
typedef struct fm_step_graph_st *fm_step_graph;
FM_API fm_status fm_step_graph_create(const fm_step_args *args, fm_step_graph *graph);
FM_API fm_status fm_step_graph_launch(fm_step_graph graph, fm_stream_t stream);
FM_API fm_status fm_step_graph_destroy(fm_step_graph graph);

/*
 * Per-kernel timing (the library's own tracing).  fm_profile_begin starts
 * recording a CUDA event pair around every kernel the library launches
 * (process-wide, up to 4096 launches); fm_profile_end waits for those
 * events, writes up to max_entries (kernel id, milliseconds) records and
 * stops recording.  Returns the number of records written, or -1 on error.
 */
enum { FM_K_CLASSIFY_MINMAX = 0, FM_K_CLASSIFY_LISTS = 1, FM_K_FWD = 2, FM_K_BWD_PRE = 3,
       FM_K_BWD = 4, FM_K_BWD_POST = 5, FM_K_CLASSIFY_ORDER = 6, FM_K_FP8_AMAX = 7,
       FM_K_FP8_CONVERT = 8, FM_K_COUNT = 9 };
typedef struct {
    int32_t kernel;
    float ms;
} fm_kernel_time;
FM_API fm_status fm_profile_begin(void);
FM_API int fm_profile_end(fm_kernel_time *out, int max_entries);

/*
 * fm_debug_wait_test — HOST, test hook; nothing calls it in a product path.
 * Failure detection is tested on the real kernels without faulting the GPU:
 * after this call, the next fm_attn_fwd / fm_attn_fwd_rows launch
 * (kernel = 0) or fm_attn_bwd / fm_attn_bwd_rows launch (kernel = 1) made by
 * the process bounds every device-side wait by limit_cycles SM cycles
 * (100,000 .. the default bound of about 3e9) instead of the default, and
 * its first CTA withholds the load of its second K tile (forward) or of its
 * second Q/dO half (backward).  The wait for that load runs out: the kernel
 * writes FM_ERR_TIMEOUT to dev_status, raises its abort flag (every other
 * wait of the CTA then gives up), drains the copies and tensor-core products
 * it issued, frees its TMEM and returns; the CUDA context stays usable.
 * The switch is consumed by that one launch; kernel = -1 clears it.
 * Returns FM_ERR_INVALID_ARG for another kernel id or a limit out of range.
 */
FM_API fm_status fm_debug_wait_test(int kernel, long long limit_cycles);

/*
 * Self-test of the bounded wait used by every pipeline barrier: one CTA
 * waits on a barrier that nothing completes, gives up after about
 * limit_cycles SM clock cycles and writes FM_ERR_TIMEOUT to dev_status.
 * Lets failure detection be tested without hanging a GPU.
 */
FM_API fm_status fm_selftest_wait_timeout(long long limit_cycles, int32_t *dev_status,
                                   fm_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FM_H_ */
