// Compressed column bounds (blog "FlashMask技术" §6.2 item 2: differential
// encoding of the interval vectors, offsets stored as 8-bit integers).
//
// Format (little endian), for bounds int32 [B, Hm, N] x 4 (lts, lte, uts, ute):
//   header     uint32 magic "FMC1", int32 B, Hm, N, n_blk (= ceil(N / 128)),
//              int32 pad, int64 payload_bytes                      (32 bytes)
//   directory  uint32 [B*Hm][n_blk][4]: (payload offset << 1) | mode, one entry
//              per 128-column block of each bound array
//   payload    per entry, 4-byte aligned:
//              mode 0 (differential): int32 base = the block's first value,
//                      then int8 delta[k] = x[k + 1] - x[k] for the block's
//                      remaining columns (all deltas in [-128, 127])
//              mode 1 (raw): int32 x[k] for every column of the block
// A block's values are base + the prefix sums of its deltas, so blocks decode
// independently and in parallel.  Causal, window, prefix and document masks
// change their bounds by 0 or 1 per column except at document boundaries, so
// most blocks are differential: about 4.3 bytes per column instead of 16.
#include <cuda_runtime.h>

#include <cstring>
#include <vector>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace {

constexpr uint32_t kCompressMagic = 0x31434D46u;   // "FMC1"
constexpr int kBlk = 128;

struct CompressHeader {
    uint32_t magic;
    int32_t B, Hm, N, n_blk, pad;
    int64_t payload_bytes;
};
static_assert(sizeof(CompressHeader) == 32, "compressed-bounds header");

FM_HD int64_t dir_bytes(int64_t S, int n_blk) { return S * n_blk * 4 * 4; }

// Payload bytes of one block of one bound array, and its mode.
int64_t block_bytes(const int32_t *x, int ncol, int *mode)
{
    bool small = true;
    for (int k = 0; k + 1 < ncol && small; ++k) {
        const int64_t d = (int64_t)x[k + 1] - x[k];
        small = d >= -128 && d <= 127;
    }
    *mode = small ? 0 : 1;
    const int64_t raw = small ? 4 + (ncol - 1) : 4 * (int64_t)ncol;
    return (raw + 3) & ~int64_t(3);
}

bool args_ok(const int32_t *const arr[4], int B, int Hm, int N)
{
    if (B <= 0 || Hm <= 0 || N <= 0) return false;
    for (int q = 0; q < 4; ++q)
        if (!arr[q]) return false;
    return (int64_t)B * Hm * N < ((int64_t)1 << 40);
}

// Total compressed size, or -1 on bad arguments or a payload beyond 2 GB.
int64_t compressed_size(const int32_t *const arr[4], int B, int Hm, int N)
{
    if (!args_ok(arr, B, Hm, N)) return -1;
    const int n_blk = (N + kBlk - 1) / kBlk;
    const int64_t S = (int64_t)B * Hm;
    int64_t payload = 0;
    for (int64_t s = 0; s < S; ++s)
        for (int blk = 0; blk < n_blk; ++blk)
            for (int q = 0; q < 4; ++q) {
                int mode = 0;
                const int ncol = (blk + 1) * kBlk <= N ? kBlk : N - blk * kBlk;
                payload += block_bytes(arr[q] + s * N + (int64_t)blk * kBlk, ncol, &mode);
            }
    if (payload >= ((int64_t)1 << 31)) return -1;
    return (int64_t)sizeof(CompressHeader) + dir_bytes(S, n_blk) + payload;
}

}  // namespace

extern "C" size_t fm_bounds_compressed_bytes(const int32_t *lts, const int32_t *lte, const int32_t *uts,
                                             const int32_t *ute, int B, int Hm, int N)
{
    const int32_t *arr[4] = {lts, lte, uts, ute};
    const int64_t n = compressed_size(arr, B, Hm, N);
    return n < 0 ? 0 : (size_t)n;
}

extern "C" fm_status fm_bounds_compress(const int32_t *lts, const int32_t *lte, const int32_t *uts,
                                        const int32_t *ute, int B, int Hm, int N, void *out, size_t out_bytes)
{
    const int32_t *arr[4] = {lts, lte, uts, ute};
    const int64_t need = compressed_size(arr, B, Hm, N);
    if (need < 0) return FM_ERR_INVALID_ARG;
    if (!out || out_bytes < (size_t)need) return FM_ERR_WORKSPACE;
    const int n_blk = (N + kBlk - 1) / kBlk;
    const int64_t S = (int64_t)B * Hm;
    uint8_t *base = static_cast<uint8_t *>(out);
    uint32_t *dir = reinterpret_cast<uint32_t *>(base + sizeof(CompressHeader));
    uint8_t *payload = base + sizeof(CompressHeader) + dir_bytes(S, n_blk);
    int64_t off = 0;
    for (int64_t s = 0; s < S; ++s)
        for (int blk = 0; blk < n_blk; ++blk)
            for (int q = 0; q < 4; ++q) {
                const int32_t *x = arr[q] + s * N + (int64_t)blk * kBlk;
                const int ncol = (blk + 1) * kBlk <= N ? kBlk : N - blk * kBlk;
                int mode = 0;
                const int64_t nb = block_bytes(x, ncol, &mode);
                uint8_t *p = payload + off;
                std::memset(p, 0, (size_t)nb);
                if (mode == 0) {
                    std::memcpy(p, &x[0], 4);
                    for (int k = 0; k + 1 < ncol; ++k) p[4 + k] = (uint8_t)(int8_t)(x[k + 1] - x[k]);
                } else {
                    std::memcpy(p, x, 4 * (size_t)ncol);
                }
                dir[(s * n_blk + blk) * 4 + q] = (uint32_t)(off << 1) | (uint32_t)mode;
                off += nb;
            }
    CompressHeader h{kCompressMagic, B, Hm, N, n_blk, 0, off};
    std::memcpy(base, &h, sizeof h);
    return FM_OK;
}

namespace fm {

// One CTA per (b * Hm + hm, 128-column block), one thread per column: each of
// the four bound arrays of the block is copied (raw) or rebuilt as base plus
// the inclusive prefix sum of its deltas (a warp scan and a scan of the four
// warp totals).  Every directory entry is checked against the payload size
// before it is read; a buffer that does not match the call writes
// FM_ERR_INVALID_ARG to *status and nothing else.
__global__ void __launch_bounds__(kBlk) bounds_decompress_kernel(const uint8_t *cb, int64_t bytes, fm_bounds out,
                                                                  int32_t *status)
{
    const int blk = blockIdx.x;
    const int64_t s = blockIdx.y;
    const int k = threadIdx.x, lane = k & 31, w = k >> 5;
    const int N = out.N;
    const CompressHeader *h = reinterpret_cast<const CompressHeader *>(cb);
    const int n_blk = (N + kBlk - 1) / kBlk;
    const int64_t S = (int64_t)out.B * out.Hm;
    const int64_t head = (int64_t)sizeof(CompressHeader) + dir_bytes(S, n_blk);
    if (h->magic != kCompressMagic || h->B != out.B || h->Hm != out.Hm || h->N != N || h->n_blk != n_blk ||
        h->payload_bytes < 0 || head + h->payload_bytes > bytes) {
        if (k == 0) set_status(status, FM_ERR_INVALID_ARG);
        return;
    }
    const uint32_t *dir = reinterpret_cast<const uint32_t *>(cb + sizeof(CompressHeader));
    const uint8_t *payload = cb + head;
    const int ncol = (blk + 1) * kBlk <= N ? kBlk : N - blk * kBlk;
    int32_t *arr[4] = {const_cast<int32_t *>(out.lts), const_cast<int32_t *>(out.lte),
                       const_cast<int32_t *>(out.uts), const_cast<int32_t *>(out.ute)};
    __shared__ int wsum[kBlk / 32];
    for (int q = 0; q < 4; ++q) {
        const uint32_t e = dir[(s * n_blk + blk) * 4 + q];
        const int mode = (int)(e & 1u);
        const int64_t off = (int64_t)(e >> 1);
        const int64_t need = mode ? 4 * (int64_t)ncol : 4 + (ncol - 1);
        const bool in = (off & 3) == 0 && off + need <= h->payload_bytes;   // block-uniform
        if (!in) {
            if (k == 0) set_status(status, FM_ERR_INVALID_ARG);
            return;
        }
        const uint8_t *p = payload + off;
        int32_t x = 0;
        if (mode == 1) {
            if (k < ncol) x = reinterpret_cast<const int32_t *>(p)[k];
        } else {
            int v = (k >= 1 && k < ncol) ? (int)(int8_t)p[4 + k - 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            if (lane == 31) wsum[w] = v;
            __syncthreads();
            for (int ww = 0; ww < w; ++ww) v += wsum[ww];
            x = *reinterpret_cast<const int32_t *>(p) + v;
            __syncthreads();                     // wsum is rewritten for the next array
        }
        if (k < ncol) arr[q][s * N + (int64_t)blk * kBlk + k] = x;
    }
}

}  // namespace fm

extern "C" fm_status fm_bounds_decompress(const void *cbounds, size_t bytes, fm_bounds out, int32_t *dev_status,
                                          fm_stream_t stream)
{
    if (!cbounds || ((uintptr_t)cbounds & 15u) || !dev_status || ((uintptr_t)dev_status & 3u))
        return FM_ERR_INVALID_ARG;
    const int32_t *arr[4] = {out.lts, out.lte, out.uts, out.ute};
    for (int q = 0; q < 4; ++q)
        if (!arr[q] || ((uintptr_t)arr[q] & 15u)) return FM_ERR_INVALID_ARG;
    if (out.B <= 0 || out.Hm <= 0 || out.N <= 0) return FM_ERR_INVALID_ARG;
    const int64_t S = (int64_t)out.B * out.Hm;
    const int n_blk = (out.N + kBlk - 1) / kBlk;
    if (S > 65535) return FM_ERR_UNSUPPORTED;
    if ((int64_t)bytes < (int64_t)sizeof(CompressHeader) + dir_bytes(S, n_blk)) return FM_ERR_INVALID_ARG;
    fm::bounds_decompress_kernel<<<dim3(n_blk, (unsigned)S), kBlk, 0, (cudaStream_t)stream>>>(
        static_cast<const uint8_t *>(cbounds), (int64_t)bytes, out, dev_status);
    return cudaPeekAtLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}
