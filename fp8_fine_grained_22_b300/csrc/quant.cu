// quant.cu -- fine-grained E4M3 quantisers (DeepSeek-V3 Technical Report,
// section 3.3.2, fine-grained quantization; 1x128 activation tiles, 128x128
// weight blocks, and the 128x1 token-wise transposed grouping the Wgrad GEMM
// needs, sections 3.3.1-3.3.3 and 3.5.2).
//
// Every group: amax = max |x|; s = fl32(amax / 448) (s = 1 for amax = 0);
// q = E4M3 RNE saturating conversion of fl32(x / s).  The divisions are
// IEEE round-to-nearest (no fast-math, no flush-to-zero), so the codes and
// scales are exact functions of the bf16 inputs.
//
// The kernels are HBM streams: 16-byte vector loads with the evict-first
// hint, group amax by warp shuffles (1x128) or a shared-memory tile
// (128x1, 128x128), conversion of pairs with the hardware E4M3x2 cvt.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace fp8fg {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float group_scale(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// E4M3 codes of x0 / s and x1 / s, x0 in the low byte.
__device__ __forceinline__ uint32_t quant_pair(float x0, float x1, float s) {
    float2 v = make_float2(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3));
}

// Four E4M3 codes packed little-endian.
__device__ __forceinline__ uint32_t quant_quad(float a, float b, float c, float d, float s) {
    return quant_pair(a, b, s) | (quant_pair(c, d, s) << 16);
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}

// ------------------------------------------------------------------ 1x128 --
// CTA: 64 rows x one 128-wide K group.  16 lanes per group, 8 elements per
// lane, 4 rows per thread (rows g, g+16, g+32, g+48) so that every thread has
// four 16-byte loads in flight.
constexpr int kQ1Rows = 64;

__global__ void __launch_bounds__(256) quant_act_1x128_kernel(const uint16_t* __restrict__ x,
                                                              int64_t M, int64_t ldx,
                                                              uint8_t* __restrict__ xq,
                                                              int64_t ldq,
                                                              float* __restrict__ sx) {
    const int l16 = threadIdx.x & 15;
    const int g = threadIdx.x >> 4;
    const int64_t kb = blockIdx.y;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kQ1Rows;
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + g + 16 * i;
        v[i] = (m < M) ? ld_stream_v4(x + m * ldx + kb * 128 + l16 * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + g + 16 * i;
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        float f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = bf16_lo(w[j]);
            f[2 * j + 1] = bf16_hi(w[j]);
        }
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float s = group_scale(amax);
        if (m < M) {
            uint2 q;
            q.x = quant_quad(f[0], f[1], f[2], f[3], s);
            q.y = quant_quad(f[4], f[5], f[6], f[7], s);
            *reinterpret_cast<uint2*>(xq + m * ldq + kb * 128 + l16 * 8) = q;
            if (l16 == 0) sx[kb * M + m] = s;
        }
    }
}

// ------------------------------------------------------------------ 128x1 --
// CTA: one 128-token group x 64 columns.  The bf16 tile is staged in shared
// memory; each thread then owns one column and a quarter of the 128 rows.
__global__ void __launch_bounds__(256) quant_act_128x1_kernel(const uint16_t* __restrict__ x,
                                                              int64_t M, int64_t K, int64_t ldx,
                                                              uint8_t* __restrict__ xqT,
                                                              float* __restrict__ sxT) {
    __shared__ __align__(16) uint16_t tile[128][64];
    __shared__ float part[4][64];
    const int t = threadIdx.x;
    const int64_t k0 = static_cast<int64_t>(blockIdx.x) * 64;
    const int64_t mb = blockIdx.y;
    const int64_t m0 = mb * 128;
    {
        const int ch = t & 7;
        uint4 v[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int row = (t >> 3) + 32 * p;
            v[p] = ld_stream_v4(x + (m0 + row) * ldx + k0 + ch * 8);
        }
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int row = (t >> 3) + 32 * p;
            *reinterpret_cast<uint4*>(&tile[row][ch * 8]) = v[p];
        }
    }
    __syncthreads();
    const int c = t & 63;
    const int qr = t >> 6;
    float f[32];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        f[i] = __uint_as_float(static_cast<uint32_t>(tile[qr * 32 + i][c]) << 16);
        amax = fmaxf(amax, fabsf(f[i]));
    }
    part[qr][c] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(part[0][c], part[1][c]), fmaxf(part[2][c], part[3][c]));
    const float s = group_scale(amax);
    if (qr == 0) sxT[mb * K + k0 + c] = s;
    uint4 o0, o1;
    o0.x = quant_quad(f[0], f[1], f[2], f[3], s);
    o0.y = quant_quad(f[4], f[5], f[6], f[7], s);
    o0.z = quant_quad(f[8], f[9], f[10], f[11], s);
    o0.w = quant_quad(f[12], f[13], f[14], f[15], s);
    o1.x = quant_quad(f[16], f[17], f[18], f[19], s);
    o1.y = quant_quad(f[20], f[21], f[22], f[23], s);
    o1.z = quant_quad(f[24], f[25], f[26], f[27], s);
    o1.w = quant_quad(f[28], f[29], f[30], f[31], s);
    uint8_t* dst = xqT + (k0 + c) * M + m0 + qr * 32;
    reinterpret_cast<uint4*>(dst)[0] = o0;
    reinterpret_cast<uint4*>(dst)[1] = o1;
}

// ---------------------------------------------------------------- 128x128 --
// CTA: one 128x128 block.  The bf16 block is held in registers (for the amax
// and the same-orientation output) and in shared memory (for the transposed
// output, one column per thread).
__global__ void __launch_bounds__(256) quant_weight_128x128_kernel(
    const uint16_t* __restrict__ w, int64_t K, int64_t N, int64_t ldw, uint8_t* __restrict__ wq,
    uint8_t* __restrict__ wqT, float* __restrict__ sw) {
    __shared__ __align__(16) uint16_t tile[128][128];
    __shared__ float part[8];
    const int t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 128;
    const int64_t k0 = static_cast<int64_t>(blockIdx.y) * 128;
    const int ch = t & 15;
    uint4 v[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const int row = (t >> 4) + 16 * p;
        v[p] = ld_stream_v4(w + (k0 + row) * ldw + n0 + ch * 8);
    }
    float amax = 0.0f;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const int row = (t >> 4) + 16 * p;
        *reinterpret_cast<uint4*>(&tile[row][ch * 8]) = v[p];
        const uint32_t wd[4] = {v[p].x, v[p].y, v[p].z, v[p].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(wd[j])), fabsf(bf16_hi(wd[j]))));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) part[warp] = amax;
    __syncthreads();
    amax = part[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, part[i]);
    const float s = group_scale(amax);
    if (t == 0) sw[blockIdx.x * (K / 128) + blockIdx.y] = s;
    if (wqT != nullptr) {
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int row = (t >> 4) + 16 * p;
            uint2 q;
            q.x = quant_quad(bf16_lo(v[p].x), bf16_hi(v[p].x), bf16_lo(v[p].y), bf16_hi(v[p].y), s);
            q.y = quant_quad(bf16_lo(v[p].z), bf16_hi(v[p].z), bf16_lo(v[p].w), bf16_hi(v[p].w), s);
            *reinterpret_cast<uint2*>(wqT + (k0 + row) * N + n0 + ch * 8) = q;
        }
    }
    if (wq != nullptr) {
        const int n = t & 127;
        const int h = t >> 7;
        uint8_t* dst = wq + (n0 + n) * K + k0 + h * 64;
#pragma unroll
        for (int c16 = 0; c16 < 4; ++c16) {
            float f[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                f[i] = __uint_as_float(static_cast<uint32_t>(tile[h * 64 + c16 * 16 + i][n]) << 16);
            uint4 o;
            o.x = quant_quad(f[0], f[1], f[2], f[3], s);
            o.y = quant_quad(f[4], f[5], f[6], f[7], s);
            o.z = quant_quad(f[8], f[9], f[10], f[11], s);
            o.w = quant_quad(f[12], f[13], f[14], f[15], s);
            reinterpret_cast<uint4*>(dst)[c16] = o;
        }
    }
}

}  // namespace fp8fg

using namespace fp8fg;

extern "C" int fp8_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                   int64_t ldq, float* sx, void* stream) {
    if (M < 0 || K <= 0 || K % 128 != 0 || ldx < K || ldq < K) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (x == nullptr || xq == nullptr || sx == nullptr) return FP8_ERR_NULL;
    if (ldx % 8 != 0 || ldq % 16 != 0 || !aligned(x, 16) || !aligned(xq, 16) || !aligned(sx, 4))
        return FP8_ERR_ALIGN;
    const int64_t gx = (M + kQ1Rows - 1) / kQ1Rows, gy = K / 128;
    if (gx > 0x7fffffff || gy > 65535) return FP8_ERR_UNSUPPORTED;
    quant_act_1x128_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), 256, 0,
                             static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(x), M, ldx, xq, ldq, sx);
    return launch_status();
}

extern "C" int fp8_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx,
                                   uint8_t* xqT, float* sxT, void* stream) {
    if (M < 0 || M % 128 != 0 || K <= 0 || K % 64 != 0 || ldx < K) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (x == nullptr || xqT == nullptr || sxT == nullptr) return FP8_ERR_NULL;
    if (ldx % 8 != 0 || !aligned(x, 16) || !aligned(xqT, 16) || !aligned(sxT, 4))
        return FP8_ERR_ALIGN;
    const int64_t gx = K / 64, gy = M / 128;
    if (gx > 0x7fffffff || gy > 65535) return FP8_ERR_UNSUPPORTED;
    quant_act_128x1_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), 256, 0,
                             static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(x), M, K, ldx, xqT, sxT);
    return launch_status();
}

extern "C" int fp8_quant_weight_128x128(const void* w, int64_t K, int64_t N, int64_t ldw,
                                        uint8_t* wq, uint8_t* wqT, float* sw, void* stream) {
    if (K < 0 || K % 128 != 0 || N < 0 || N % 128 != 0 || ldw < N) return FP8_ERR_SHAPE;
    if (K == 0 || N == 0) return FP8_OK;
    if (w == nullptr || sw == nullptr || (wq == nullptr && wqT == nullptr)) return FP8_ERR_NULL;
    if (ldw % 8 != 0 || !aligned(w, 16) || !aligned(wq, 16) || !aligned(wqT, 16) ||
        !aligned(sw, 4))
        return FP8_ERR_ALIGN;
    const int64_t gx = N / 128, gy = K / 128;
    if (gx > 0x7fffffff || gy > 65535) return FP8_ERR_UNSUPPORTED;
    quant_weight_128x128_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)),
                                  256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(w), K, N, ldw, wq, wqT, sw);
    return launch_status();
}

extern "C" const char* fp8_status_str(int status) {
    switch (status) {
        case FP8_OK: return "ok";
        case FP8_ERR_NULL: return "null pointer";
        case FP8_ERR_SHAPE: return "invalid shape or leading dimension";
        case FP8_ERR_ALIGN: return "misaligned pointer or stride";
        case FP8_ERR_UNSUPPORTED: return "unsupported configuration";
        case FP8_ERR_CUDA: return "CUDA error";
        case FP8_ERR_TIMEOUT: return "kernel barrier wait timed out";
        case FP8_ERR_DEVICE_SHAPE: return "invalid device-side offsets";
        default: return "unknown status";
    }
}
