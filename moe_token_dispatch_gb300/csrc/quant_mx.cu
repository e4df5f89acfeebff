// Microscaled FP8 (MXFP8) quantisation for the block-scaled expert GEMM, the
// MX form named by the "ThunderKittens 2.0 & FP8/NVFP4" item of the
// ThunderKittens tutorial page (the format itself is the MX formats'
// definition): 32 consecutive elements along the reduction dimension share
// one E8M0 scale 2^s,
//   s = floor(log2(amax)) - 8, clamped to [-127, 127]   (-127 for amax 0),
//   code_i = E4M3_rn_satfinite(v_i * 2^-s),   scale byte = s + 127,
// the product v * 2^-s formed in IEEE fp32 (a power-of-two scaling, rounded
// once), so the codes are a pure function of the bf16 inputs. Inputs are
// finite.
//   k_quant_rows_mx   activations x [T, D] -> codes [T, D] + scale bytes
//                     [T, D / 32] (one thread per block of 32).
//   k_quant_cols_mx   weights W [E, D, N] -> codes in the blocked layout of
//                     the FP8 GEMM (64-column x 128-code blocks, K-major
//                     inside) + scale bytes in the blocked layout the MX
//                     GEMM copies per K-step (below); done once per weight
//                     set, not per step.
// Scale layout of the weights (each unit of the MX GEMM covers 192 output
// columns): for column tile t (columns 192 t ..), K-step ks (codes
// 128 ks ..), one 1 KiB piece at ((e * NT + t) * KS + ks) * 1024, two 512-byte
// halves h (columns 192 t + 128 h ..), each 32 rows r of 16 bytes: bytes
// 4 g .. 4 g + 3 of row r hold the four 32-code blocks of column
// 192 t + 128 h + 32 g + r. That is the 32-row x 16-byte source a
// tcgen05.cp.32x128b copies into four TMEM columns; unused bytes are zero.
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pk_internal.h"

namespace pk {
namespace {

__device__ __forceinline__ float bf16_f32(uint32_t h) { return __uint_as_float(h << 16); }

// s of a block with largest magnitude amax (finite, >= 0)
__device__ __forceinline__ int mx_exponent(float amax) {
    const uint32_t field = __float_as_uint(amax) >> 23;  // amax >= 0: no sign bit
    if (field == 0) return -127;                         // 0 or below 2^-126: clamped
    const int s = static_cast<int>(field) - 127 - 8;
    return s < -127 ? -127 : (s > 127 ? 127 : s);
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xffffu) | (hi << 16);
}

// 32 bf16 (as 16 words) -> 32 codes (8 words) and the scale byte
__device__ __forceinline__ uint8_t mx_block(const uint32_t (&w)[16], uint32_t (&c)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        amax = fmaxf(amax, fmaxf(fabsf(bf16_f32(w[i] & 0xffffu)), fabsf(bf16_f32(w[i] >> 16))));
    const int s = mx_exponent(amax);
    const float m = ldexpf(1.0f, -s);  // exact power of two
#pragma unroll
    for (int i = 0; i < 8; ++i)
        c[i] = e4m3x4(__fmul_rn(bf16_f32(w[2 * i] & 0xffffu), m), __fmul_rn(bf16_f32(w[2 * i] >> 16), m),
                      __fmul_rn(bf16_f32(w[2 * i + 1] & 0xffffu), m),
                      __fmul_rn(bf16_f32(w[2 * i + 1] >> 16), m));
    return static_cast<uint8_t>(s + 127);
}

__global__ void __launch_bounds__(256) k_quant_rows_mx(const uint16_t* __restrict__ x, int64_t nblk,
                                                       uint8_t* __restrict__ q,
                                                       uint8_t* __restrict__ s) {
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblk;
         b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4* src = reinterpret_cast<const uint4*>(x + b * 32);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = src[i];
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
        uint32_t c[8];
        s[b] = mx_block(w, c);
        uint4* dst = reinterpret_cast<uint4*>(q + b * 32);
        dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
        dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
    }
}

// One thread per (column n, block of 32 d) of W[e]; grid (ceil(N / 128), D / 32, E).
__global__ void __launch_bounds__(128) k_quant_cols_mx(const uint16_t* __restrict__ W, int32_t D,
                                                       int32_t N, uint8_t* __restrict__ q,
                                                       uint8_t* __restrict__ sb) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    const int db = blockIdx.y, e = blockIdx.z;
    const uint16_t* col = W + (static_cast<int64_t>(e) * D + 32 * db) * N + n;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        w[i] = static_cast<uint32_t>(col[static_cast<int64_t>(2 * i) * N]) |
               (static_cast<uint32_t>(col[static_cast<int64_t>(2 * i + 1) * N]) << 16);
    uint32_t c[8];
    const uint8_t sbyte = mx_block(w, c);
    // codes: block (e, n / 64, d / 128), row n % 64, bytes (32 db) % 128 ..
    const int64_t NB = (N + 63) / 64, KS = D / 128;
    const int64_t row = ((e * NB + n / 64) * KS + db / 4) * 64 + n % 64;
    uint4* dst = reinterpret_cast<uint4*>(q + row * 128 + (32 * db) % 128);
    dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
    dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
    // scale: piece (e, n / 192, db / 4), half, row, group, block db % 4
    const int64_t NT = (N + 191) / 192;
    const int nl = n % 192, h = nl / 128, g = (nl % 128) / 32, r = nl % 32;
    sb[((e * NT + n / 192) * KS + db / 4) * 1024 + h * 512 + r * 16 + g * 4 + db % 4] = sbyte;
}

}  // namespace

size_t mx_weight_scale_bytes(int32_t E, int32_t D, int32_t N) {
    return static_cast<size_t>(E) * static_cast<size_t>((N + 191) / 192) *
           static_cast<size_t>(D / 128) * 1024u;
}

cudaError_t launch_quant_rows_mx(const uint16_t* x, int32_t T, int32_t D, uint8_t* q, uint8_t* s,
                                 cudaStream_t stream) {
    const int64_t nblk = static_cast<int64_t>(T) * (D / 32);
    if (nblk == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const int64_t blocks = (nblk + 255) / 256;
    const int grid = static_cast<int>(blocks < sms * 16 ? blocks : sms * 16);
    k_quant_rows_mx<<<grid, 256, 0, stream>>>(x, nblk, q, s);
    return cudaGetLastError();
}

cudaError_t launch_quant_cols_mx(const uint16_t* W, int32_t E, int32_t D, int32_t N, uint8_t* q,
                                 uint8_t* sb, cudaStream_t stream) {
    // padding of the code blocks past N reads as code 0, of the scale pieces as byte 0
    const int64_t qbytes = static_cast<int64_t>(E) * ((N + 63) / 64) * (D / 128) * 8192;
    cudaError_t err = cudaMemsetAsync(q, 0, static_cast<size_t>(qbytes), stream);
    if (err != cudaSuccess) return err;
    err = cudaMemsetAsync(sb, 0, mx_weight_scale_bytes(E, D, N), stream);
    if (err != cudaSuccess) return err;
    k_quant_cols_mx<<<dim3((N + 127) / 128, D / 32, E), 128, 0, stream>>>(W, D, N, q, sb);
    return cudaGetLastError();
}

}  // namespace pk
