// FP8 (e4m3) inputs for the forward: per-tensor quantization of bf16 tensors.
//
// Passage: blog "FlashMask技术" §4.2 (the H100 path computes in FP8).  The scale
// rule is per tensor: descale = amax / 448 (448 = the largest finite e4m3
// value), codes = e4m3(x / descale) with the division in fp32, rounding to
// nearest even and saturating (cvt.rn.satfinite).  V is written transposed,
// [B, H, d, N], so that the P V product reads both operands K-major.
//
// Three launches: amax (grid-stride, one atomicMax per CTA on the float bits,
// which order like the values for non-negative floats), convert (reads the
// amax, HBM-bound: 2 bytes read and 1 written per element), and a one-thread
// finalize that replaces the amax by the descale.
#include <cuda_runtime.h>

#include <cstdint>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace fm {

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__global__ void __launch_bounds__(256) fp8_amax_kernel(const uint4 *x, int64_t n8, unsigned *amax_bits)
{
    float mx = 0.f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = x[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            mx = fmax3(mx, fabsf(bf16_to_f32(w[k] & 0xffffu)), fabsf(bf16_to_f32(w[k] >> 16)));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) mx = fmaxf(mx, red[w]);
        atomicMax(amax_bits, __float_as_uint(mx));
    }
}

__device__ __forceinline__ float descale_of(float amax) { return amax > 0.f ? amax / 448.f : 1.f; }

// Plain layout: 8 elements per thread.
__global__ void __launch_bounds__(256) fp8_convert_kernel(const uint4 *x, uint2 *out, int64_t n8, const float *amax)
{
    const float ds = descale_of(*amax);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = x[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t c[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint32_t lo = pack_e4m3x2(bf16_to_f32(w[2 * k] & 0xffffu) / ds, bf16_to_f32(w[2 * k] >> 16) / ds);
            const uint32_t hi = pack_e4m3x2(bf16_to_f32(w[2 * k + 1] & 0xffffu) / ds, bf16_to_f32(w[2 * k + 1] >> 16) / ds);
            c[k] = lo | (hi << 16);
        }
        out[i] = make_uint2(c[0], c[1]);
    }
}

// Transposed layout [BH][N][D] -> [BH][D][N]: one CTA per (64 rows, bh); the
// codes are transposed through shared memory.  N is a multiple of 16, so
// every 16-byte store lands on a 16-byte boundary.
template <int D>
__global__ void __launch_bounds__(256) fp8_convert_t_kernel(const uint16_t *x, uint8_t *out, int N, const float *amax)
{
    constexpr int R = 64;                     // rows (keys) per CTA
    __shared__ uint8_t tile[D][R + 16];
    const float ds = descale_of(*amax);
    const int n0 = blockIdx.x * R;
    const int64_t bh = blockIdx.y;
    const int t = threadIdx.x;
    // load: thread t converts row n0 + t / 4, columns [(t % 4) D / 4, ...)
    {
        const int r = t >> 2, c0 = (t & 3) * (D / 4);
        const int n = n0 + r;
#pragma unroll
        for (int c = 0; c < D / 4; c += 8) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (n < N) v = *reinterpret_cast<const uint4 *>(x + (bh * N + n) * D + c0 + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t e = pack_e4m3x2(bf16_to_f32(w[k] & 0xffffu) / ds, bf16_to_f32(w[k] >> 16) / ds);
                tile[c0 + c + 2 * k][r] = (uint8_t)(e & 0xff);
                tile[c0 + c + 2 * k + 1][r] = (uint8_t)(e >> 8);
            }
        }
    }
    __syncthreads();
    // store: column dd of the tile is R consecutive bytes of output row dd
    for (int idx = t; idx < D * (R / 16); idx += blockDim.x) {
        const int dd = idx / (R / 16), seg = idx % (R / 16);
        const int n = n0 + seg * 16;
        if (n >= N) continue;
        uint8_t *dst = out + (bh * D + dd) * N + n;
        const uint8_t *src = &tile[dd][seg * 16];
        uint4 v;
        uint8_t *vb = reinterpret_cast<uint8_t *>(&v);
#pragma unroll
        for (int b = 0; b < 16; ++b) vb[b] = src[b];
        *reinterpret_cast<uint4 *>(dst) = v;
    }
}

__global__ void fp8_finalize_kernel(float *descale)
{
    if (threadIdx.x == 0 && blockIdx.x == 0) *descale = descale_of(*descale);
}

}  // namespace fm

using namespace fm;

extern "C" fm_status fm_quantize_fp8(const void *x, int B, int H, int N, int d, int transpose, uint8_t *x8,
                                     float *descale, fm_stream_t stream)
{
    if (!x || !x8 || !descale || ((uintptr_t)x & 15u) || ((uintptr_t)x8 & 15u) || ((uintptr_t)descale & 3u))
        return FM_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || N <= 0) return FM_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FM_ERR_UNSUPPORTED;
    if (transpose && (N % 16) != 0) return FM_ERR_UNSUPPORTED;
    if ((int64_t)B * H * N * d > ((int64_t)1 << 40) || (int64_t)B * H > 65535) return FM_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t n8 = (int64_t)B * H * N * d / 8;
    const int blocks = (int)((n8 + 255) / 256 < 152 * 8 ? (n8 + 255) / 256 : 152 * 8);
    if (cudaMemsetAsync(descale, 0, sizeof(float), s) != cudaSuccess) return FM_ERR_CUDA;
    {
        ProfScope ps(kKFp8Amax, s);
        fp8_amax_kernel<<<blocks, 256, 0, s>>>((const uint4 *)x, n8, (unsigned *)descale);
    }
    {
        ProfScope ps(kKFp8Convert, s);
        if (!transpose)
            fp8_convert_kernel<<<blocks, 256, 0, s>>>((const uint4 *)x, (uint2 *)x8, n8, descale);
        else if (d == 128)
            fp8_convert_t_kernel<128><<<dim3((N + 63) / 64, B * H), 256, 0, s>>>((const uint16_t *)x, x8, N, descale);
        else
            fp8_convert_t_kernel<64><<<dim3((N + 63) / 64, B * H), 256, 0, s>>>((const uint16_t *)x, x8, N, descale);
    }
    fp8_finalize_kernel<<<1, 32, 0, s>>>(descale);
    return cudaPeekAtLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}
