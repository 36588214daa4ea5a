// quant.cu -- fine-grained E4M3 quantisers (DeepSeek-V3 Technical Report,
// section 3.3.2, fine-grained quantization; 1x128 activation tiles, 128x128
// weight blocks, and the 128x1 token-wise transposed grouping the Wgrad GEMM
// needs, sections 3.3.1-3.3.3 and 3.5.2).
//
// Every group: amax = max |x|; s = fl32(amax / 448) (s = 1 for amax = 0);
// q = E4M3 RNE saturating conversion of fl32(x / s).  The scale is an IEEE
// division and the quotients are correctly rounded (GroupDiv below); nothing
// is flushed to zero, so the codes and scales are exact functions of the
// bf16 inputs.
//
// The kernels are HBM streams: 16-byte vector loads with the evict-first
// hint, group amax by warp shuffles (1x128) or a shared-memory tile
// (128x1, 128x128), conversion of pairs with the hardware E4M3x2 cvt.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8fg {

// The 1x128, 128x1 and operand (128x128) kernels are persistent: a grid of a
// few CTAs per SM walks the tiles with a stride of the grid size, and each
// thread issues the loads of its next tile before it processes the current
// one, so HBM reads stay in flight through the compute and store phases.
// The per-expert 128x1 kernel runs one CTA per (token group, column block).
constexpr int kQuantThreads = 256;
constexpr int kQuantCtasPerSm = 4;

// ------------------------------------------------------------------ 1x128 --
// Tile: 64 rows x one 128-wide K group.  Four lanes per group, 32 elements
// (four 16-byte loads) per lane, one row per thread.  Tiles are numbered
// K-group fastest.
constexpr int kQ1Rows = 64;

__device__ __forceinline__ void load_1x128(const uint16_t* __restrict__ x, int64_t M, int64_t ldx,
                                           int64_t KB, int64_t t, int row, int l4, uint4 (&v)[4]) {
    const int64_t kb = t % KB;
    const int64_t m = (t / KB) * kQ1Rows + row;
    const uint16_t* src = x + m * ldx + kb * 128 + l4 * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (m < M) ? ld_stream_v4(src + 8 * i) : make_uint4(0, 0, 0, 0);
}

// Quantises the 1x128 tile whose bf16 values this thread holds in v (row
// `row` of the tile, lanes l4 = 0..3 of its four-lane group).
__device__ __forceinline__ void quant_1x128_tile(int64_t M, int64_t KB, uint8_t* __restrict__ xq,
                                                 int64_t ldq, float* __restrict__ sx, int64_t t,
                                                 int row, int l4, const uint4 (&v)[4]) {
    const int64_t kb = t % KB;
    const int64_t m = (t / KB) * kQ1Rows + row;
    uint32_t mx = absmax_bf16x2(v[0].x, v[0].y);
    mx = absmax_bf16x2(mx, absmax_bf16x2(v[0].z, v[0].w));
#pragma unroll
    for (int i = 1; i < 4; ++i) {
        mx = absmax_bf16x2(mx, absmax_bf16x2(v[i].x, v[i].y));
        mx = absmax_bf16x2(mx, absmax_bf16x2(v[i].z, v[i].w));
    }
    float amax = amax_of_pair(mx);
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float s = group_scale(amax);
    const GroupDiv dv(s);
    if (m < M) {
        uint4 o[2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t a = dv.quad_words(v[i].x, v[i].y);
            const uint32_t b = dv.quad_words(v[i].z, v[i].w);
            if (i & 1) {
                o[i >> 1].z = a;
                o[i >> 1].w = b;
            } else {
                o[i >> 1].x = a;
                o[i >> 1].y = b;
            }
        }
        uint4* dst = reinterpret_cast<uint4*>(xq + m * ldq + kb * 128 + l4 * 32);
        dst[0] = o[0];
        dst[1] = o[1];
        if (l4 == 0) sx[kb * M + m] = s;
    }
}

__global__ void __launch_bounds__(kQuantThreads) quant_act_1x128_kernel(
    const uint16_t* __restrict__ x, int64_t M, int64_t KB, int64_t ldx, uint8_t* __restrict__ xq,
    int64_t ldq, float* __restrict__ sx, int64_t tiles) {
    griddep_launch_dependents();  // the GEMM that follows may set up meanwhile
    const int l4 = threadIdx.x & 3;
    const int row = threadIdx.x >> 2;  // 0..63
    int64_t t = blockIdx.x;
    uint4 v[4];
    if (t < tiles) load_1x128(x, M, ldx, KB, t, row, l4, v);
    while (t < tiles) {
        const int64_t tn = t + gridDim.x;
        uint4 vn[4];
        if (tn < tiles) load_1x128(x, M, ldx, KB, tn, row, l4, vn);
        quant_1x128_tile(M, KB, xq, ldq, sx, t, row, l4, v);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = vn[i];
        t = tn;
    }
}

// ------------------------------------------------------------- 1x128 E5M6 --
// The same tiles and lanes as the 1x128 E4M3 kernel; each lane's 32 codes
// (12 bits each) fill 48 bytes of the packed row, stored as three 16-byte
// chunks.  Scale s = fl32(amax / 65024).
__device__ __forceinline__ void quant_1x128_e5m6_tile(int64_t M, int64_t KB,
                                                      uint8_t* __restrict__ xq, int64_t ldq,
                                                      float* __restrict__ sx, int64_t t, int row,
                                                      int l4, const uint4 (&v)[4]) {
    const int64_t kb = t % KB;
    const int64_t m = (t / KB) * kQ1Rows + row;
    uint32_t mx = absmax_bf16x2(v[0].x, v[0].y);
    mx = absmax_bf16x2(mx, absmax_bf16x2(v[0].z, v[0].w));
#pragma unroll
    for (int i = 1; i < 4; ++i) {
        mx = absmax_bf16x2(mx, absmax_bf16x2(v[i].x, v[i].y));
        mx = absmax_bf16x2(mx, absmax_bf16x2(v[i].z, v[i].w));
    }
    float amax = amax_of_pair(mx);
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 65024.0f);
    const GroupDiv dv(s, kE5M6FastMin);
    if (m < M) {
        uint32_t w[12];
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // 16-byte load i: eight elements
            const uint32_t words[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            uint32_t c[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float q0, q1;
                dv.quot2(bf16_lo(words[j]), bf16_hi(words[j]), q0, q1);
                c[2 * j] = e5m6_code(q0, (words[j] >> 15) & 1u);
                c[2 * j + 1] = e5m6_code(q1, words[j] >> 31);
            }
            pack_e5m6_8(c, w[3 * i], w[3 * i + 1], w[3 * i + 2]);
        }
        uint4* dst = reinterpret_cast<uint4*>(xq + m * ldq + kb * 192 + l4 * 48);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
        if (l4 == 0) sx[kb * M + m] = s;
    }
}

__global__ void __launch_bounds__(kQuantThreads) quant_act_1x128_e5m6_kernel(
    const uint16_t* __restrict__ x, int64_t M, int64_t KB, int64_t ldx, uint8_t* __restrict__ xq,
    int64_t ldq, float* __restrict__ sx, int64_t tiles) {
    griddep_launch_dependents();
    const int l4 = threadIdx.x & 3;
    const int row = threadIdx.x >> 2;  // 0..63
    int64_t t = blockIdx.x;
    uint4 v[4];
    if (t < tiles) load_1x128(x, M, ldx, KB, t, row, l4, v);
    while (t < tiles) {
        const int64_t tn = t + gridDim.x;
        uint4 vn[4];
        if (tn < tiles) load_1x128(x, M, ldx, KB, tn, row, l4, vn);
        quant_1x128_e5m6_tile(M, KB, xq, ldq, sx, t, row, l4, v);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = vn[i];
        t = tn;
    }
}

// ---------------------------------------------- power-of-two-scale 1x128 --
// As the 1x128 kernel, with the scale the smallest power of two 2^e such that
// amax / 2^e <= 448; writes the UE8M0 byte e + 127 instead of an FP32 scale.
__global__ void __launch_bounds__(kQuantThreads) quant_act_1x128_pow2_kernel(
    const uint16_t* __restrict__ x, int64_t M, int64_t KB, int64_t ldx, uint8_t* __restrict__ xq,
    int64_t ldq, uint8_t* __restrict__ se8, int64_t tiles) {
    griddep_launch_dependents();
    const int l4 = threadIdx.x & 3;
    const int row = threadIdx.x >> 2;
    int64_t t = blockIdx.x;
    uint4 v[4];
    if (t < tiles) load_1x128(x, M, ldx, KB, t, row, l4, v);
    while (t < tiles) {
        const int64_t tn = t + gridDim.x;
        uint4 vn[4];
        if (tn < tiles) load_1x128(x, M, ldx, KB, tn, row, l4, vn);
        const int64_t kb = t % KB;
        const int64_t m = (t / KB) * kQ1Rows + row;
        uint32_t mx = absmax_bf16x2(v[0].x, v[0].y);
        mx = absmax_bf16x2(mx, absmax_bf16x2(v[0].z, v[0].w));
#pragma unroll
        for (int i = 1; i < 4; ++i) {
            mx = absmax_bf16x2(mx, absmax_bf16x2(v[i].x, v[i].y));
            mx = absmax_bf16x2(mx, absmax_bf16x2(v[i].z, v[i].w));
        }
        float amax = amax_of_pair(mx);
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int e = pow2_exponent(amax);
        const float r = pow2_inverse(e);
        if (m < M) {
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                o[2 * i] = e4m3_scaled_pair(bf16_lo(v[i].x), bf16_hi(v[i].x), r) |
                           (e4m3_scaled_pair(bf16_lo(v[i].y), bf16_hi(v[i].y), r) << 16);
                o[2 * i + 1] = e4m3_scaled_pair(bf16_lo(v[i].z), bf16_hi(v[i].z), r) |
                               (e4m3_scaled_pair(bf16_lo(v[i].w), bf16_hi(v[i].w), r) << 16);
            }
            uint4* dst = reinterpret_cast<uint4*>(xq + m * ldq + kb * 128 + l4 * 32);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            if (l4 == 0) se8[kb * M + m] = static_cast<uint8_t>(e + 127);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = vn[i];
        t = tn;
    }
}

// ------------------------------------------- power-of-two-scale 128x128 --
// One CTA (256 threads) per 128x128 block: the block is staged in shared
// memory, its amax reduced, and the codes written K-major (wq[n][k]) through
// an XOR-swizzled shared transpose; the block's UE8M0 byte is written for
// each of its 128 rows n (se8[kb][n]).
__global__ void __launch_bounds__(256) quant_weight_128x128_pow2_kernel(
    const uint16_t* __restrict__ w, int64_t K, int64_t N, int64_t ldw, uint8_t* __restrict__ wq,
    uint8_t* __restrict__ se8) {
    griddep_launch_dependents();
    __shared__ __align__(16) uint16_t tile[128][128];
    __shared__ float part[8];
    const int t0 = threadIdx.x, lane = t0 & 31, warp = t0 >> 5;
    const int64_t NB = N / 128;
    const int64_t nb = blockIdx.x % NB, kb = blockIdx.x / NB;
    const int64_t n0 = nb * 128, k0 = kb * 128;
    const int ch = t0 & 15;
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (t0 >> 4) + 16 * i;
        const uint4 u = ld_stream_v4(w + (k0 + r) * ldw + n0 + ch * 8);
        *reinterpret_cast<uint4*>(&tile[r][ch * 8]) = u;
        mx = absmax_bf16x2(mx, absmax_bf16x2(u.x, u.y));
        mx = absmax_bf16x2(mx, absmax_bf16x2(u.z, u.w));
    }
    float amax = amax_of_pair(mx);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) part[warp] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(fmaxf(part[0], part[1]), fmaxf(part[2], part[3])),
                 fmaxf(fmaxf(part[4], part[5]), fmaxf(part[6], part[7])));
    const int e = pow2_exponent(amax);
    const float r = pow2_inverse(e);
    if (t0 < 128) se8[kb * N + n0 + t0] = static_cast<uint8_t>(e + 127);
    // thread: column pair (2cp, 2cp+1), rows rq*32 .. rq*32+31 -> 32 codes of
    // each of the two columns (wq rows n = 2cp, 2cp+1), k contiguous
    const int cp = t0 & 63, rq = t0 >> 6;
    uint32_t ca[8], cb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(&tile[rq * 32 + 4 * i + 2 * j][2 * cp]);
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(&tile[rq * 32 + 4 * i + 2 * j + 1][2 * cp]);
            // k = rq*32 + 4i + 2j and +1: column 2cp (lo halves), 2cp+1 (hi halves)
            lo |= e4m3_scaled_pair(bf16_lo(w0), bf16_lo(w1), r) << (16 * j);
            hi |= e4m3_scaled_pair(bf16_hi(w0), bf16_hi(w1), r) << (16 * j);
        }
        ca[i] = lo;
        cb[i] = hi;
    }
    __syncthreads();  // every value has been read: reuse the tile for the codes
    uint8_t* codes = reinterpret_cast<uint8_t*>(tile);  // [128 n][128 k], 16-byte chunks swizzled
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c = rq * 2 + h;  // 16-byte chunk of the k row
        const int na = 2 * cp, nbb = 2 * cp + 1;
        *reinterpret_cast<uint4*>(&codes[na * 128 + ((c ^ (na & 7)) << 4)]) =
            make_uint4(ca[4 * h], ca[4 * h + 1], ca[4 * h + 2], ca[4 * h + 3]);
        *reinterpret_cast<uint4*>(&codes[nbb * 128 + ((c ^ (nbb & 7)) << 4)]) =
            make_uint4(cb[4 * h], cb[4 * h + 1], cb[4 * h + 2], cb[4 * h + 3]);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = t0 + 256 * i;
        const int n = j >> 3, c = j & 7;
        *reinterpret_cast<uint4*>(wq + (n0 + n) * K + k0 + c * 16) =
            *reinterpret_cast<const uint4*>(&codes[n * 128 + ((c ^ (n & 7)) << 4)]);
    }
}

// ------------------------------------------------------------------ 128x1 --
// Tile: one 128-token group x 64 columns, staged in shared memory; each
// thread then owns a pair of adjacent columns (one 32-bit word per row: the
// warp reads a whole 128-byte row, no bank conflicts) and 16 of the 128
// rows, and converts both columns with one permute per four sign bits.
// Tiles are numbered column-block fastest.
__device__ __forceinline__ void load_128x1(const uint16_t* __restrict__ x, int64_t ldx,
                                           int64_t KC, int64_t t, int tid, uint4 (&v)[4]) {
    const int64_t k0 = (t % KC) * 64;
    const int64_t m0 = (t / KC) * 128;
    const int ch = tid & 7;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int row = (tid >> 3) + 32 * p;
        v[p] = ld_stream_v4(x + (m0 + row) * ldx + k0 + ch * 8);
    }
}

__global__ void __launch_bounds__(kQuantThreads) quant_act_128x1_kernel(
    const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx, uint8_t* __restrict__ xqT,
    float* __restrict__ sxT, int64_t tiles) {
    griddep_launch_dependents();  // the GEMM that follows may set up meanwhile
    __shared__ __align__(16) uint16_t tile[128][64];
    __shared__ float part[8][64];
    const int t0 = threadIdx.x;
    const int64_t KC = K / 64;
    const int cp = t0 & 31, rg = t0 >> 5;
    int64_t t = blockIdx.x;
    uint4 v[4];
    if (t < tiles) load_128x1(x, ldx, KC, t, t0, v);
    while (t < tiles) {
        const int64_t k0 = (t % KC) * 64;
        const int64_t mb = t / KC;
        {
            const int ch = t0 & 7;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int row = (t0 >> 3) + 32 * p;
                *reinterpret_cast<uint4*>(&tile[row][ch * 8]) = v[p];
            }
        }
        const int64_t tn = t + gridDim.x;
        if (tn < tiles) load_128x1(x, ldx, KC, tn, t0, v);  // next tile's loads in flight
        __syncthreads();
        uint32_t w[16];
        uint32_t mx = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            w[i] = *reinterpret_cast<const uint32_t*>(&tile[rg * 16 + i][2 * cp]);
            mx = absmax_bf16x2(mx, w[i]);  // per column: low half and high half
        }
        part[rg][2 * cp] = bf16_lo(mx);
        part[rg][2 * cp + 1] = bf16_hi(mx);
        __syncthreads();
        float amax_a = part[0][2 * cp], amax_b = part[0][2 * cp + 1];
#pragma unroll
        for (int j = 1; j < 8; ++j) {
            amax_a = fmaxf(amax_a, part[j][2 * cp]);
            amax_b = fmaxf(amax_b, part[j][2 * cp + 1]);
        }
        const float sa = group_scale(amax_a), sb = group_scale(amax_b);
        const GroupDiv da(sa), db(sb);
        if (rg == 0) {
            sxT[mb * K + k0 + 2 * cp] = sa;
            sxT[mb * K + k0 + 2 * cp + 1] = sb;
        }
        uint4 oa, ob;
        GroupDiv::halves(da, db, w[0], w[1], w[2], w[3], oa.x, ob.x);
        GroupDiv::halves(da, db, w[4], w[5], w[6], w[7], oa.y, ob.y);
        GroupDiv::halves(da, db, w[8], w[9], w[10], w[11], oa.z, ob.z);
        GroupDiv::halves(da, db, w[12], w[13], w[14], w[15], oa.w, ob.w);
        const int64_t r0 = mb * 128 + rg * 16;
        *reinterpret_cast<uint4*>(xqT + (k0 + 2 * cp) * M + r0) = oa;
        *reinterpret_cast<uint4*>(xqT + (k0 + 2 * cp + 1) * M + r0) = ob;
        __syncthreads();  // tile and part are rewritten by the next iteration
        t = tn;
    }
}

// ---------------------------------------------------- 128x1, per expert --
// The 128x1 grouping for a grouped Wgrad GEMM, whose contraction runs over
// each expert's own tokens: expert e's rows offsets[e] .. offsets[e+1]-1 of
// x form ceil(t_e / 128) groups of 128 tokens (the last one short).  The
// transposed codes of expert e start at the padded column pofs[e] (the sum of
// the previous experts' group counts x 128); a short group's missing tokens
// get code 0, which adds nothing to the product, and do not enter its amax.
// One CTA per (group, 64-column block) tile, tiles walked expert-major;
// CTAs past the last tile exit.
__global__ void __launch_bounds__(kQuantThreads) quant_act_128x1_grouped_kernel(
    const uint16_t* __restrict__ x, int64_t T, int64_t K, int64_t ldx,
    const int32_t* __restrict__ offsets, int E, uint8_t* __restrict__ xqT,
    float* __restrict__ sxT, int64_t Tp, int32_t* __restrict__ pofs) {
    griddep_launch_dependents();  // the GEMM that follows may set up meanwhile
    __shared__ __align__(16) uint16_t tile[128][64];
    __shared__ float part[4][64];
    __shared__ int64_t s_m0, s_p0;
    __shared__ int s_rows;
    const int t0 = threadIdx.x;
    const int64_t KC = K / 64;
    if (t0 == 0) {
        // locate this CTA's tile; CTA 0 also writes the padded offsets.  Expert
        // ranges outside [0, T] or decreasing count as empty (memory safety;
        // the results of such offsets are unspecified).
        int64_t t = blockIdx.x, padded = 0, lo = 0;
        int rows = 0;
        int64_t m0 = 0, p0 = 0;
        for (int e = 0; e < E; ++e) {
            if (blockIdx.x == 0) pofs[e] = static_cast<int32_t>(padded);
            int64_t hi = __ldg(offsets + e + 1);
            if (hi < lo || hi > T) hi = lo;
            const int64_t g = (hi - lo + 127) / 128;
            if (rows == 0 && t >= 0 && t < g * KC) {
                const int64_t grp = t / KC;
                m0 = lo + grp * 128;
                p0 = padded + grp * 128;
                rows = static_cast<int>(hi - m0 < 128 ? hi - m0 : 128);
                t = -(t % KC) - 1;  // remember the column block, stop matching
            } else if (rows == 0) {
                t -= g * KC;
            }
            padded += g * 128;
            lo = hi;
        }
        if (blockIdx.x == 0) pofs[E] = static_cast<int32_t>(padded);
        if (rows > 0 && p0 + 128 > Tp) rows = 0;  // capacity guard
        s_rows = rows;
        s_m0 = m0;
        s_p0 = rows > 0 ? p0 * KC + (-t - 1) : 0;  // padded column, column block
    }
    __syncthreads();
    const int rows = s_rows;
    if (rows == 0) return;
    const int64_t m0 = s_m0;
    const int64_t p0 = s_p0 / KC;
    const int64_t k0 = (s_p0 % KC) * 64;
    {
        const int ch = t0 & 7;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int row = (t0 >> 3) + 32 * p;
            const uint4 v = row < rows ? ld_stream_v4(x + (m0 + row) * ldx + k0 + ch * 8)
                                       : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(&tile[row][ch * 8]) = v;
        }
    }
    __syncthreads();
    const int c = t0 & 63;
    const int qr = t0 >> 6;
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
    const GroupDiv dv(s);
    if (qr == 0) sxT[(p0 / 128) * K + k0 + c] = s;
    uint4 o0, o1;
    o0.x = dv.quad(f[0], f[1], f[2], f[3]);
    o0.y = dv.quad(f[4], f[5], f[6], f[7]);
    o0.z = dv.quad(f[8], f[9], f[10], f[11]);
    o0.w = dv.quad(f[12], f[13], f[14], f[15]);
    o1.x = dv.quad(f[16], f[17], f[18], f[19]);
    o1.y = dv.quad(f[20], f[21], f[22], f[23]);
    o1.z = dv.quad(f[24], f[25], f[26], f[27]);
    o1.w = dv.quad(f[28], f[29], f[30], f[31]);
    uint8_t* dst = xqT + (k0 + c) * Tp + p0 + qr * 32;
    reinterpret_cast<uint4*>(dst)[0] = o0;
    reinterpret_cast<uint4*>(dst)[1] = o1;
}

// ---------------------------------------------------------------- 128x128 --
// The weight quantiser is the persistent kernel below run on weight blocks
// alone: one grid walks the blocks with a stride of the grid size, each CTA
// converting one 128x128 block from shared memory while the cp.async copy
// of its next block lands in a second buffer.  (One 128-thread CTA per
// block, without that overlap, was 7-15 % slower at every measured shape:
// the grid ran in whole waves of load, reduce, convert and store.)

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))), "l"(gmem)
                 : "memory");
}

// ------------------------------------------------- both Fprop operands --
// One persistent launch quantises the activation (1x128) and the weight
// (128x128) of one GEMM, or the weight alone.  Run as two kernels, the operands serialise: each
// kernel fills the SMs on its own, and neither is large enough to reach the
// HBM rate alone.  Here one grid walks a single list of items, weight blocks
// spread evenly among the activation tiles, with a stride of the grid size,
// prefetching the next item while it converts the current one: a weight
// block by cp.async into the other of two 32 KB shared buffers, an
// activation tile into registers.  The per-group arithmetic is the same code
// as the single-operand kernels.
constexpr int kPairThreads = 256;
constexpr int kPairCtasPerSm = 3;
constexpr int kPairSmem = 2 * 128 * 128 * 2;  // two bf16 blocks

struct PairArgs {
    const uint16_t* x;
    int64_t M, ldx, ldq, act_tiles;
    uint8_t* xq;
    float* sx;
    const uint16_t* w;
    int64_t N, ldw, w_tiles;
    uint8_t* wq;
    uint8_t* wqT;
    float* sw;
    int64_t KB;  // K / 128, shared by both operands
};

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_prev() {  // all groups but the newest
    asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// Item i of the list is a weight block when the count of weight blocks
// among items 0..i, floor((i + 1) W / total), steps up at i; *idx is then
// the block's index, else the activation tile's.
__device__ __forceinline__ bool pair_item(const PairArgs& p, int64_t i, int64_t* idx) {
    const int64_t total = p.w_tiles + p.act_tiles;
    const int64_t w_upto = ((i + 1) * p.w_tiles) / total;
    const bool is_w = w_upto > (i * p.w_tiles) / total;
    *idx = is_w ? w_upto - 1 : i - w_upto;
    return is_w;
}

// Starts the loads of item t: weight block t into `tile`, or activation
// tile t into v.
__device__ __forceinline__ void pair_issue(const PairArgs& p, bool is_w, int64_t t,
                                           uint16_t (*tile)[128], int row, int l4,
                                           uint4 (&v)[4]) {
    if (is_w) {
        const int64_t NB = p.N / 128;
        const int64_t n0 = (t % NB) * 128, k0 = (t / NB) * 128;
        const int ch = threadIdx.x & 15;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int r = (threadIdx.x >> 4) + 16 * q;
            cp_async16(&tile[r][ch * 8], p.w + (k0 + r) * p.ldw + n0 + ch * 8);
        }
    } else {
        load_1x128(p.x, p.M, p.ldx, p.KB, t, row, l4, v);
    }
}

// Converts the weight block t staged in `tile` (all 256 threads).  The
// transposed codes are staged in the first 16 KB of `tile` once every
// thread has read its values.  Ends with a barrier, after which `tile` and
// `part` may be reused.
__device__ __forceinline__ void pair_weight_block(const PairArgs& p, int64_t t,
                                                  uint16_t (*tile)[128], float* part) {
    const int t0 = threadIdx.x;
    const int lane = t0 & 31, warp = t0 >> 5;
    const int ch = t0 & 15;
    const int64_t NB = p.N / 128, K = p.KB * 128;
    const int64_t nb = t % NB, kb = t / NB;
    const int64_t n0 = nb * 128, k0 = kb * 128;
    uint32_t mx = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint4 u = *reinterpret_cast<const uint4*>(&tile[(t0 >> 4) + 16 * q][ch * 8]);
        mx = absmax_bf16x2(mx, absmax_bf16x2(u.x, u.y));
        mx = absmax_bf16x2(mx, absmax_bf16x2(u.z, u.w));
    }
    float amax = amax_of_pair(mx);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) part[warp] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(fmaxf(part[0], part[1]), fmaxf(part[2], part[3])),
                 fmaxf(fmaxf(part[4], part[5]), fmaxf(part[6], part[7])));
    const float s = group_scale(amax);
    const GroupDiv dv(s);
    if (t0 == 0) p.sw[nb * p.KB + kb] = s;
    if (p.wqT != nullptr) {
#pragma unroll 4
        for (int q = 0; q < 8; ++q) {
            const int r = (t0 >> 4) + 16 * q;
            const uint4 u = *reinterpret_cast<const uint4*>(&tile[r][ch * 8]);
            uint2 o;
            o.x = dv.quad_words(u.x, u.y);
            o.y = dv.quad_words(u.z, u.w);
            *reinterpret_cast<uint2*>(p.wqT + (k0 + r) * p.N + n0 + ch * 8) = o;
        }
    }
    if (p.wq != nullptr) {
        // columns 2cp, 2cp+1; rows rq*32 .. rq*32+31 in two chunks of 16
        // k values; codes staged as [n][k] rows with 16-byte chunks
        // XOR-swizzled by n & 7, then written out as 128-byte rows of wq.
        const int cp = t0 & 63;
        const int rq = t0 >> 6;
        uint4 oc[2][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t wv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                wv[i] = *reinterpret_cast<const uint32_t*>(&tile[rq * 32 + h * 16 + i][2 * cp]);
            uint4 o0, o1;
            dv.quad_halves(wv[0], wv[1], wv[2], wv[3], o0.x, o1.x);
            dv.quad_halves(wv[4], wv[5], wv[6], wv[7], o0.y, o1.y);
            dv.quad_halves(wv[8], wv[9], wv[10], wv[11], o0.z, o1.z);
            dv.quad_halves(wv[12], wv[13], wv[14], wv[15], o0.w, o1.w);
            oc[h][0] = o0;
            oc[h][1] = o1;
        }
        __syncthreads();  // every value of the block has been read
        uint8_t* codes = reinterpret_cast<uint8_t*>(tile);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = rq * 2 + h;  // 16-byte chunk of the 128-byte k row
            const int n_a = 2 * cp, n_b = 2 * cp + 1;
            *reinterpret_cast<uint4*>(&codes[n_a * 128 + ((c ^ (n_a & 7)) << 4)]) = oc[h][0];
            *reinterpret_cast<uint4*>(&codes[n_b * 128 + ((c ^ (n_b & 7)) << 4)]) = oc[h][1];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = t0 + kPairThreads * i;  // chunk j: row n = j / 8, chunk c = j % 8
            const int n = j >> 3, c = j & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(&codes[n * 128 + ((c ^ (n & 7)) << 4)]);
            *reinterpret_cast<uint4*>(p.wq + (n0 + n) * K + k0 + c * 16) = v;
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kPairThreads, kPairCtasPerSm) quant_fprop_pair_kernel(const PairArgs p) {
    griddep_launch_dependents();  // the GEMM that follows may set up meanwhile
    extern __shared__ __align__(128) uint8_t pair_smem[];
    __shared__ float part[kPairThreads / 32];
    uint16_t (*tiles)[128][128] = reinterpret_cast<uint16_t (*)[128][128]>(pair_smem);
    const int l4 = threadIdx.x & 3;
    const int row = threadIdx.x >> 2;  // 0..63
    const int64_t total = p.w_tiles + p.act_tiles;
    int64_t i = blockIdx.x;  // item; the same in every thread of the CTA
    int buf = 0;
    uint4 v[4];
    int64_t idx = 0;
    bool is_w = false;
    if (i < total) {
        is_w = pair_item(p, i, &idx);
        pair_issue(p, is_w, idx, tiles[0], row, l4, v);
    }
    cp_async_commit();
    while (i < total) {
        const int64_t in = i + gridDim.x;
        uint4 vn[4];
        int64_t idx_n = 0;
        bool is_w_n = false;
        if (in < total) {
            is_w_n = pair_item(p, in, &idx_n);
            pair_issue(p, is_w_n, idx_n, tiles[buf ^ 1], row, l4, vn);
        }
        cp_async_commit();  // possibly empty: one group per item keeps the count
        if (is_w) {
            cp_async_wait_prev();
            __syncthreads();
            pair_weight_block(p, idx, tiles[buf], part);
        } else {
            quant_1x128_tile(p.M, p.KB, p.xq, p.ldq, p.sx, idx, row, l4, v);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = vn[k];
        buf ^= 1;
        i = in;
        idx = idx_n;
        is_w = is_w_n;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Persistent grid: as many CTAs as can be resident at once (cached per
// kernel and device), never more than there are tiles.
template <auto kern>
static int64_t quant_grid(int64_t tiles) {
    static ContextCache<int> per_sm;
    const int sms = sm_count_current();
    int n = 0;
    if (sms <= 0 || per_sm.get(&n, [](int* v) {
            int b = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kQuantThreads, 0) !=
                    cudaSuccess ||
                b <= 0)
                b = 1;
            *v = b < kQuantCtasPerSm ? b : kQuantCtasPerSm;
            return static_cast<int>(FP8_OK);
        }) != FP8_OK)
        return tiles < 1024 ? tiles : 1024;
    const int64_t cap = static_cast<int64_t>(sms) * n;
    return tiles < cap ? tiles : cap;
}

}  // namespace fp8fg

using namespace fp8fg;

extern "C" fp8_status fp8_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                   int64_t ldq, float* sx, void* stream) {
    if (M < 0 || K <= 0 || K % 128 != 0 || ldx < K || ldq < K) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (x == nullptr || xq == nullptr || sx == nullptr) return FP8_ERR_NULL;
    if (ldx % 8 != 0 || ldq % 16 != 0 || !aligned(x, 16) || !aligned(xq, 16) || !aligned(sx, 4))
        return FP8_ERR_ALIGN;
    const int64_t tiles = ((M + kQ1Rows - 1) / kQ1Rows) * (K / 128);
    quant_act_1x128_kernel<<<static_cast<unsigned>(quant_grid<quant_act_1x128_kernel>(tiles)), kQuantThreads, 0,
                             static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(x), M, K / 128, ldx, xq, ldq, sx, tiles);
    return to_status(launch_status());
}

extern "C" fp8_status fp8_quant_act_1x128_e5m6(const void* x, int64_t M, int64_t K,
                                               int64_t ldx, uint8_t* xq, int64_t ldq_bytes,
                                               float* sx, void* stream) {
    if (M < 0 || K <= 0 || K % 128 != 0 || ldx < K || ldq_bytes < 3 * K / 2) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (x == nullptr || xq == nullptr || sx == nullptr) return FP8_ERR_NULL;
    if (ldx % 8 != 0 || ldq_bytes % 16 != 0 || !aligned(x, 16) || !aligned(xq, 16) ||
        !aligned(sx, 4))
        return FP8_ERR_ALIGN;
    const int64_t tiles = ((M + kQ1Rows - 1) / kQ1Rows) * (K / 128);
    quant_act_1x128_e5m6_kernel<<<static_cast<unsigned>(quant_grid<quant_act_1x128_e5m6_kernel>(tiles)),
                                  kQuantThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(x), M, K / 128, ldx, xq, ldq_bytes, sx, tiles);
    return to_status(launch_status());
}

extern "C" fp8_status fp8_quant_act_1x128_pow2(const void* x, int64_t M, int64_t K, int64_t ldx,
                                               uint8_t* xq, int64_t ldq, uint8_t* se8,
                                               void* stream) {
    if (M < 0 || K <= 0 || K % 128 != 0 || ldx < K || ldq < K) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (x == nullptr || xq == nullptr || se8 == nullptr) return FP8_ERR_NULL;
    if (ldx % 8 != 0 || ldq % 16 != 0 || !aligned(x, 16) || !aligned(xq, 16)) return FP8_ERR_ALIGN;
    const int64_t tiles = ((M + kQ1Rows - 1) / kQ1Rows) * (K / 128);
    quant_act_1x128_pow2_kernel<<<static_cast<unsigned>(quant_grid<quant_act_1x128_pow2_kernel>(tiles)),
                                  kQuantThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(x), M, K / 128, ldx, xq, ldq, se8, tiles);
    return to_status(launch_status());
}

extern "C" fp8_status fp8_quant_weight_128x128_pow2(const void* w, int64_t K, int64_t N,
                                                   int64_t ldw, uint8_t* wq, uint8_t* se8,
                                                   void* stream) {
    if (K < 0 || K % 128 != 0 || N < 0 || N % 128 != 0 || ldw < N) return FP8_ERR_SHAPE;
    if (K == 0 || N == 0) return FP8_OK;
    if (w == nullptr || wq == nullptr || se8 == nullptr) return FP8_ERR_NULL;
    if (ldw % 8 != 0 || !aligned(w, 16) || !aligned(wq, 16)) return FP8_ERR_ALIGN;
    const int64_t blocks = (N / 128) * (K / 128);
    if (blocks > 0x7fffffffLL) return FP8_ERR_UNSUPPORTED;
    quant_weight_128x128_pow2_kernel<<<static_cast<unsigned>(blocks), 256, 0,
                                       static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(w), K, N, ldw, wq, se8);
    return to_status(launch_status());
}

extern "C" fp8_status fp8_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx,
                                   uint8_t* xqT, float* sxT, void* stream) {
    if (M < 0 || M % 128 != 0 || K <= 0 || K % 64 != 0 || ldx < K) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (x == nullptr || xqT == nullptr || sxT == nullptr) return FP8_ERR_NULL;
    if (ldx % 8 != 0 || !aligned(x, 16) || !aligned(xqT, 16) || !aligned(sxT, 4))
        return FP8_ERR_ALIGN;
    const int64_t tiles = (M / 128) * (K / 64);
    quant_act_128x1_kernel<<<static_cast<unsigned>(quant_grid<quant_act_128x1_kernel>(tiles)), kQuantThreads, 0,
                             static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(x), M, K, ldx, xqT, sxT, tiles);
    return to_status(launch_status());
}

extern "C" fp8_status fp8_quant_act_128x1_grouped(const void* x, int64_t T, int64_t K, int64_t ldx,
                                           const int32_t* offsets, int32_t E, uint8_t* xqT,
                                           float* sxT, int64_t Tp, int32_t* pofs,
                                           void* stream) {
    if (T < 0 || K <= 0 || K % 64 != 0 || ldx < K || E < 1 || E > 65536 || Tp < 0 ||
        Tp % 128 != 0)
        return FP8_ERR_SHAPE;
    // every expert pads at most 127 tokens
    if (Tp < ((T + 127 * static_cast<int64_t>(E) + 127) / 128) * 128) return FP8_ERR_SHAPE;
    if (Tp > 0x7fffffffLL) return FP8_ERR_UNSUPPORTED;
    if (offsets == nullptr || pofs == nullptr) return FP8_ERR_NULL;
    if (T > 0 && (x == nullptr || xqT == nullptr || sxT == nullptr)) return FP8_ERR_NULL;
    if (ldx % 8 != 0 || !aligned(x, 16) || !aligned(xqT, 16) || !aligned(sxT, 4) ||
        !aligned(offsets, 4) || !aligned(pofs, 4))
        return FP8_ERR_ALIGN;
    // upper bound of the tiles: sum over experts of ceil(t_e / 128) groups x K/64
    const int64_t tiles = ((T + 127 * static_cast<int64_t>(E)) / 128 + 1) * (K / 64);
    if (tiles > 0x7fffffffLL) return FP8_ERR_UNSUPPORTED;
    quant_act_128x1_grouped_kernel<<<static_cast<unsigned>(tiles), kQuantThreads, 0,
                                     static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(x), T, K, ldx, offsets, E, xqT, sxT, Tp, pofs);
    return to_status(launch_status());
}

// Persistent grid of the operand kernel: as many CTAs as are resident (at
// most kPairCtasPerSm per SM), never more than there are items.
static int launch_pair(const PairArgs& p, cudaStream_t stream) {
    const int64_t total = p.act_tiles + p.w_tiles;
    if (total == 0) return FP8_OK;
    static ContextCache<int> per_sm;
    const int sms = sm_count_current();
    if (sms <= 0) return FP8_ERR_CUDA;
    int n = 0;
    const int st = per_sm.get(&n, [](int* v) {
        if (cudaFuncSetAttribute(quant_fprop_pair_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem) !=
            cudaSuccess)
            return static_cast<int>(FP8_ERR_CUDA);
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, quant_fprop_pair_kernel,
                                                          kPairThreads, kPairSmem) !=
                cudaSuccess ||
            b <= 0)
            return static_cast<int>(FP8_ERR_CUDA);
        *v = b < kPairCtasPerSm ? b : kPairCtasPerSm;
        return static_cast<int>(FP8_OK);
    });
    if (st != FP8_OK) return st;
    const int64_t cap = static_cast<int64_t>(sms) * n;
    const int64_t grid = total < cap ? total : cap;
    quant_fprop_pair_kernel<<<static_cast<unsigned>(grid), kPairThreads, kPairSmem, stream>>>(p);
    return launch_status();
}

extern "C" fp8_status fp8_quant_weight_128x128(const void* w, int64_t K, int64_t N, int64_t ldw,
                                        uint8_t* wq, uint8_t* wqT, float* sw, void* stream) {
    if (K < 0 || K % 128 != 0 || N < 0 || N % 128 != 0 || ldw < N) return FP8_ERR_SHAPE;
    if (K == 0 || N == 0) return FP8_OK;
    if (w == nullptr || sw == nullptr || (wq == nullptr && wqT == nullptr)) return FP8_ERR_NULL;
    if (ldw % 8 != 0 || !aligned(w, 16) || !aligned(wq, 16) || !aligned(wqT, 16) ||
        !aligned(sw, 4))
        return FP8_ERR_ALIGN;
    PairArgs p = {};
    p.w = static_cast<const uint16_t*>(w);
    p.N = N;
    p.ldw = ldw;
    p.wq = wq;
    p.wqT = wqT;
    p.sw = sw;
    p.w_tiles = (N / 128) * (K / 128);
    p.KB = K / 128;
    return to_status(launch_pair(p, static_cast<cudaStream_t>(stream)));
}

extern "C" fp8_status fp8_quant_fprop_operands(const void* x, int64_t M, int64_t K, int64_t ldx,
                                        uint8_t* xq, int64_t ldq, float* sx, const void* w,
                                        int64_t N, int64_t ldw, uint8_t* wq, uint8_t* wqT,
                                        float* sw, void* stream) {
    if (M < 0 || K < 0 || K % 128 != 0 || N < 0 || N % 128 != 0) return FP8_ERR_SHAPE;
    const bool act = M > 0 && K > 0, wgt = N > 0 && K > 0;
    if (act && (ldx < K || ldq < K)) return FP8_ERR_SHAPE;
    if (wgt && ldw < N) return FP8_ERR_SHAPE;
    if (!act && !wgt) return FP8_OK;
    if (act && (x == nullptr || xq == nullptr || sx == nullptr)) return FP8_ERR_NULL;
    if (wgt && (w == nullptr || sw == nullptr || (wq == nullptr && wqT == nullptr)))
        return FP8_ERR_NULL;
    if (act && (ldx % 8 != 0 || ldq % 16 != 0 || !aligned(x, 16) || !aligned(xq, 16) ||
                !aligned(sx, 4)))
        return FP8_ERR_ALIGN;
    if (wgt && (ldw % 8 != 0 || !aligned(w, 16) || !aligned(wq, 16) || !aligned(wqT, 16) ||
                !aligned(sw, 4)))
        return FP8_ERR_ALIGN;
    PairArgs p;
    p.x = static_cast<const uint16_t*>(x);
    p.M = act ? M : 0;
    p.ldx = ldx;
    p.ldq = ldq;
    p.xq = xq;
    p.sx = sx;
    p.act_tiles = act ? ((M + kQ1Rows - 1) / kQ1Rows) * (K / 128) : 0;
    p.w = static_cast<const uint16_t*>(w);
    p.N = wgt ? N : 128;
    p.ldw = ldw;
    p.wq = wq;
    p.wqT = wqT;
    p.sw = sw;
    p.w_tiles = wgt ? (N / 128) * (K / 128) : 0;
    p.KB = K / 128;
    return to_status(launch_pair(p, static_cast<cudaStream_t>(stream)));
}

extern "C" const char* fp8_status_str(fp8_status status) {
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
