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
#include "tensormap.cuh"

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

// Loads this lane's 32 elements of row m, K group kb (zeros past row M).
__device__ __forceinline__ void load_1x128(const uint16_t* __restrict__ x, uint32_t M, int64_t ldx,
                                           uint32_t kb, uint32_t m, int l4, uint4 (&v)[4]) {
    const uint16_t* src = x + static_cast<size_t>(m) * ldx + kb * 128 + l4 * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (m < M) ? ld_stream_v4(src + 8 * i) : make_uint4(0, 0, 0, 0);
}

// The same for tile t (64 rows x one K group, K group fastest), row `row`.
__device__ __forceinline__ void load_1x128_tile(const uint16_t* __restrict__ x, int64_t M, int64_t ldx,
                                                int64_t KB, int64_t t, int row, int l4, uint4 (&v)[4]) {
    const int64_t kb = t % KB;
    const int64_t m = (t / KB) * kQ1Rows + row;
    const uint16_t* src = x + m * ldx + kb * 128 + l4 * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (m < M) ? ld_stream_v4(src + 8 * i) : make_uint4(0, 0, 0, 0);
}

// Quantises the group (row m, K group kb) whose 32 bf16 values per lane
// this thread holds in v (lanes l4 = 0..3 of the row's four-lane group).
__device__ __forceinline__ void quant_1x128_group(uint32_t M, uint8_t* __restrict__ xq, int64_t ldq,
                                                  float* __restrict__ sx, uint32_t kb, uint32_t m, int l4,
                                                  const uint4 (&v)[4]) {
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        mx = absmax_acc(mx, v[i].x);
        mx = absmax_acc(mx, v[i].y);
        mx = absmax_acc(mx, v[i].z);
        mx = absmax_acc(mx, v[i].w);
    }
    mx &= 0x7FFF7FFFu;
    mx = absmax_acc(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = absmax_acc(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float s = group_scale(amax_of_pair(mx));
    const NegDiv dv(s, __frcp_rn(s));
    if (m < M) {
        uint4 o0, o1;
        if (s >= 0x1p-91f) {
            o0 = codes_1x128<true>(dv, v[0], v[1]);
            o1 = codes_1x128<true>(dv, v[2], v[3]);
        } else {
            o0 = codes_1x128<false>(dv, v[0], v[1]);
            o1 = codes_1x128<false>(dv, v[2], v[3]);
        }
        uint4* dst = reinterpret_cast<uint4*>(xq + static_cast<size_t>(m) * ldq + kb * 128 + l4 * 32);
        dst[0] = o0;
        dst[1] = o1;
        if (l4 == 0) sx[static_cast<size_t>(kb) * M + m] = s;
    }
}

__global__ void __launch_bounds__(kQuantThreads) quant_act_1x128_kernel(
    const uint16_t* __restrict__ x, uint32_t M, uint32_t KB, int64_t ldx, uint8_t* __restrict__ xq,
    int64_t ldq, float* __restrict__ sx, uint32_t tiles) {
    griddep_launch_dependents();  // the GEMM that follows may set up meanwhile
    const int l4 = threadIdx.x & 3;
    const int row = threadIdx.x >> 2;  // 0..63
    // tile t = mb * KB + kb, walked with the grid stride without division
    const uint32_t step = gridDim.x, step_q = step / KB, step_r = step % KB;
    uint32_t kb = blockIdx.x % KB, mb = blockIdx.x / KB;
    uint4 v[4];
    if (blockIdx.x < tiles) load_1x128(x, M, ldx, kb, mb * kQ1Rows + row, l4, v);
    for (uint32_t t = blockIdx.x; t < tiles; t += step) {
        uint32_t kbn = kb + step_r, mbn = mb + step_q;
        if (kbn >= KB) {
            kbn -= KB;
            ++mbn;
        }
        uint4 vn[4];
        if (t + step < tiles) load_1x128(x, M, ldx, kbn, mbn * kQ1Rows + row, l4, vn);  // in flight
        quant_1x128_group(M, xq, ldq, sx, kb, mb * kQ1Rows + row, l4, v);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = vn[i];
        kb = kbn;
        mb = mbn;
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
    if (t < tiles) load_1x128_tile(x, M, ldx, KB, t, row, l4, v);
    while (t < tiles) {
        const int64_t tn = t + gridDim.x;
        uint4 vn[4];
        if (tn < tiles) load_1x128_tile(x, M, ldx, KB, tn, row, l4, vn);
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
    if (t < tiles) load_1x128_tile(x, M, ldx, KB, t, row, l4, v);
    while (t < tiles) {
        const int64_t tn = t + gridDim.x;
        uint4 vn[4];
        if (tn < tiles) load_1x128_tile(x, M, ldx, KB, tn, row, l4, vn);
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
// Tile: one 128-token group x 64 columns (16 KB of bf16), brought by TMA
// with the 128-byte swizzle into a ring of kQ128x1Stages slots.  Warp w owns
// the tile's columns 8w .. 8w+7 (one 16-byte chunk of every row); lane
// (cp = lane & 3, g = lane >> 2) owns the column pair 8w+2cp, 8w+2cp+1 and
// rows 16g .. 16g+15.  The warps never wait for one another:
// - lane g reads its rows in the order 16g + (i ^ g), i = 0..15, so at every
//   step the eight lanes of a column pair read rows with different swizzle
//   phases, i.e. eight different bank groups (no conflicts);
// - a column's maximum is combined across its eight lanes by shuffles, and
//   the eight columns' scales are computed once each, by lanes 0-7;
// - the last warp to finish reading a slot (a shared counter) issues the
//   slot's next load.
// A lane's 16 codes per column leave in one 16-byte store, the XOR order
// undone by the byte permute that packs them; the eight lanes of a column
// write its 128-byte row of xqT together.  Tiles are numbered column-block
// fastest.
constexpr int kQ128x1Stages = 3;
constexpr int kQ128x1TileBytes = 128 * 64 * 2;
// 1 KB of slack to align the ring to the swizzle pattern; then the ring, the
// full barriers, the slot counters (reads done, loads issued) and the abort flag
constexpr int kQ128x1Smem = 1024 + kQ128x1Stages * (kQ128x1TileBytes + 16) + 16;

// Wait for a TMA load still in flight when the CTA gives up, so that the ring
// is not released under it; bounded like every other wait.
__device__ __forceinline__ void drain_load(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitLimit) return;
}

// Codes of 16 rows of two columns held as bf16 pairs (column a in the low
// halves of w[0..15], b in the high ones), sign bits flipped back.  Word m
// of oa packs the codes of w[4m .. 4m+3] through the byte selector sel
// (0x5410: memory order; the 128x1 kernel passes a lane-dependent order).
template <bool FAST>
__device__ __forceinline__ void codes_cols16(const NegDiv& da, const NegDiv& db, const uint32_t* w,
                                             uint32_t sel, uint32_t* oa, uint32_t* ob) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t a01 = da.ncodes2<FAST>(bf16_lo2(w[4 * m], w[4 * m + 1]));
        const uint32_t a23 = da.ncodes2<FAST>(bf16_lo2(w[4 * m + 2], w[4 * m + 3]));
        const uint32_t b01 = db.ncodes2<FAST>(bf16_hi2(w[4 * m], w[4 * m + 1]));
        const uint32_t b23 = db.ncodes2<FAST>(bf16_hi2(w[4 * m + 2], w[4 * m + 3]));
        oa[m] = prmt(a01, a23, sel) ^ kSignFlip4;
        ob[m] = prmt(b01, b23, sel) ^ kSignFlip4;
    }
}

__global__ void __launch_bounds__(kQuantThreads) quant_act_128x1_kernel(
    const __grid_constant__ CUtensorMap xmap, uint32_t M, uint32_t K, uint8_t* __restrict__ xqT,
    float* __restrict__ sxT, uint32_t tiles, unsigned* err_word) {
    griddep_launch_dependents();  // the GEMM that follows may set up meanwhile
    extern __shared__ __align__(16) uint8_t smem_q1[];
    uint8_t* ring = smem_q1 + ((1024u - (smem_addr(smem_q1) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + kQ128x1Stages * kQ128x1TileBytes);
    uint32_t* done = reinterpret_cast<uint32_t*>(full + kQ128x1Stages);  // warps done reading, per slot
    uint32_t* issued = done + kQ128x1Stages;                              // loads issued, per slot
    volatile int* abort_flag = reinterpret_cast<volatile int*>(issued + kQ128x1Stages);
    const int t0 = threadIdx.x, warp = t0 >> 5, lane = t0 & 31;
    const int cp = lane & 3, g = lane >> 2;
    const uint32_t KC = K / 64;
    const uint32_t step = gridDim.x;
    auto issue = [&](uint32_t tt, int s) {
        const uint32_t bar = smem_addr(&full[s]);
        mbar_arrive_expect_tx(bar, kQ128x1TileBytes);
        tma_load_2d(smem_addr(ring + s * kQ128x1TileBytes), &xmap, bar, static_cast<int>((tt % KC) * 64),
                    static_cast<int>((tt / KC) * 128));
        atomicAdd(&issued[s], 1u);
    };
    if (t0 == 0) {
        for (int s = 0; s < kQ128x1Stages; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            done[s] = 0;
            issued[s] = 0;
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&xmap);
        for (int s = 0; s < kQ128x1Stages; ++s)
            if (blockIdx.x + s * step < tiles) issue(blockIdx.x + s * step, s);
    }
    __syncthreads();
    // Byte offsets of this lane's words in a slot, for i & 7 = j (rows
    // 16g + (j ^ g), +8 for i >= 8): row 16g + u sits at 128 (16g + u) and its
    // chunk w at 16 (w ^ (row & 7)) = 16 (w ^ u).
    uint32_t off[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int u = j ^ g;
        off[j] = 2048 * g + 128 * u + 16 * (warp ^ u) + 4 * cp;
    }
    // Packing selector: the codes of rows i = 4m + t (t = 0, 1 in the first
    // source's low bytes, t = 2, 3 in the second's) go to byte t ^ (g & 3).
    uint32_t sel = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int t = b ^ (g & 3);
        sel |= static_cast<uint32_t>((t & 1) | ((t >> 1) << 2)) << (4 * b);
    }
    const bool swap_words = (g & 4) != 0;
    const uint32_t step_q = step / KC, step_r = step % KC;
    uint32_t kc = blockIdx.x % KC, mb = blockIdx.x / KC;
    uint32_t it = 0;
    for (uint32_t t = blockIdx.x; t < tiles; t += step, ++it) {
        const int s = static_cast<int>(it % kQ128x1Stages);
        if (!wait_bounded_warp(smem_addr(&full[s]), (it / kQ128x1Stages) & 1u, abort_flag, err_word)) break;
        const uint8_t* slot = ring + s * kQ128x1TileBytes;
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = *reinterpret_cast<const uint32_t*>(slot + off[i & 7] + 128 * (i & 8));
        // the last warp to finish with the slot refills it
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const uint32_t prev = atomicAdd(&done[s], 1u);
            const uint32_t tn = t + kQ128x1Stages * step;
            if (prev == 8u * (it / kQ128x1Stages) + 7u && tn < tiles) issue(tn, s);
        }
        uint32_t mx = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) mx = absmax_acc(mx, w[i]);
        mx &= 0x7FFF7FFFu;
        mx = absmax_acc(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = absmax_acc(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = absmax_acc(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        // lanes c = 0..7 (and their copies) take column 8w + c: its maximum
        // is half c & 1 of lane c >> 1's pair
        const int c8 = lane & 7;
        const uint32_t m2 = __shfl_sync(0xffffffffu, mx, c8 >> 1);
        const float sc = group_scale((c8 & 1) ? bf16_hi(m2) : bf16_lo(m2));
        const float rc = __frcp_rn(sc);
        const uint32_t k0 = kc * 64 + 8 * warp;
        if (lane < 8) sxT[static_cast<size_t>(mb) * K + k0 + lane] = sc;
        const float sa = __shfl_sync(0xffffffffu, sc, 2 * cp), ra = __shfl_sync(0xffffffffu, rc, 2 * cp);
        const float sb = __shfl_sync(0xffffffffu, sc, 2 * cp + 1), rb = __shfl_sync(0xffffffffu, rc, 2 * cp + 1);
        const NegDiv da(sa, ra), db(sb, rb);
        uint32_t oa[4], ob[4];
        if (sa >= 0x1p-91f && sb >= 0x1p-91f)
            codes_cols16<true>(da, db, w, sel, oa, ob);
        else
            codes_cols16<false>(da, db, w, sel, oa, ob);
        const uint4 va = swap_words ? make_uint4(oa[1], oa[0], oa[3], oa[2]) : make_uint4(oa[0], oa[1], oa[2], oa[3]);
        const uint4 vb = swap_words ? make_uint4(ob[1], ob[0], ob[3], ob[2]) : make_uint4(ob[0], ob[1], ob[2], ob[3]);
        uint8_t* dst = xqT + static_cast<size_t>(k0 + 2 * cp) * M + mb * 128 + 16 * g;
        *reinterpret_cast<uint4*>(dst) = va;
        *reinterpret_cast<uint4*>(dst + M) = vb;
        kc += step_r;
        mb += step_q;
        if (kc >= KC) {
            kc -= KC;
            ++mb;
        }
    }
    // A timed-out wait ends the loop early: a load still in flight into a
    // slot (at most one per slot) must land before the CTA releases the ring.
    __syncthreads();
    if (t0 == 0 && *abort_flag) {
        for (int s = 0; s < kQ128x1Stages; ++s) {
            const uint32_t n = *reinterpret_cast<volatile uint32_t*>(&issued[s]);
            if (n > 0) drain_load(smem_addr(&full[s]), (n - 1) & 1u);
        }
    }
}

// ------------------------------------------------------- 1x128 and 128x1 --
// Both quantisations of one activation from a single read of it (the Fprop
// operand and the transposed Wgrad operand of the same X or dY).  Tiles of
// 128 tokens x 128 columns arrive by TMA as two 64-column boxes with the
// 128-byte swizzle, in a two-slot ring.  Per tile:
// - 128x1: every warp does, for each 64-column half, what a warp of
//   quant_act_128x1_kernel does with its tile (column chunk w, XOR row order);
// - 1x128: the thread pair (2r, 2r+1) takes row r's 128-wide group, one half
//   each.  The odd thread walks its chunks in the order j ^ 4, so the pair's
//   reads of one row fall on different bank groups;
// - the last warp to finish with the slot issues its next two loads.
// Codes and scales are those of fp8_quant_act_1x128 and fp8_quant_act_128x1,
// bit for bit (the same per-group arithmetic).
constexpr int kQDualStages = 2;
constexpr int kQDualHalfBytes = 128 * 64 * 2;
constexpr int kQDualTileBytes = 2 * kQDualHalfBytes;
constexpr int kQDualSmem = 1024 + kQDualStages * (kQDualTileBytes + 16) + 16;

__global__ void __launch_bounds__(kQuantThreads) quant_act_dual_kernel(
    const __grid_constant__ CUtensorMap xmap, uint32_t M, uint32_t K, uint8_t* __restrict__ xq,
    int64_t ldq, float* __restrict__ sx, uint8_t* __restrict__ xqT, float* __restrict__ sxT,
    uint32_t tiles, unsigned* err_word) {
    griddep_launch_dependents();  // the GEMM that follows may set up meanwhile
    constexpr int S = kQDualStages;
    extern __shared__ __align__(16) uint8_t smem_qd[];
    uint8_t* ring = smem_qd + ((1024u - (smem_addr(smem_qd) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + S * kQDualTileBytes);
    uint32_t* done = reinterpret_cast<uint32_t*>(full + S);  // warps done reading, per slot
    uint32_t* issued = done + S;                              // loads issued, per slot
    volatile int* abort_flag = reinterpret_cast<volatile int*>(issued + S);
    const int t0 = threadIdx.x, warp = t0 >> 5, lane = t0 & 31;
    const int cp = lane & 3, g = lane >> 2;
    const uint32_t KC = K / 128;
    const uint32_t step = gridDim.x;
    auto issue = [&](uint32_t tt, int s) {
        const uint32_t bar = smem_addr(&full[s]);
        const uint32_t dst = smem_addr(ring + s * kQDualTileBytes);
        const int kx = static_cast<int>((tt % KC) * 128), my = static_cast<int>((tt / KC) * 128);
        mbar_arrive_expect_tx(bar, kQDualTileBytes);
        tma_load_2d(dst, &xmap, bar, kx, my);
        tma_load_2d(dst + kQDualHalfBytes, &xmap, bar, kx + 64, my);
        atomicAdd(&issued[s], 1u);
    };
    if (t0 == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            done[s] = 0;
            issued[s] = 0;
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&xmap);
        for (int s = 0; s < S; ++s)
            if (blockIdx.x + s * step < tiles) issue(blockIdx.x + s * step, s);
    }
    __syncthreads();
    // 128x1 part: this lane's word offsets in a 64-column half, packing
    // selector and word order, as in quant_act_128x1_kernel
    uint32_t off[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int u = j ^ g;
        off[j] = 2048 * g + 128 * u + 16 * (warp ^ u) + 4 * cp;
    }
    uint32_t sel = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int t = b ^ (g & 3);
        sel |= static_cast<uint32_t>((t & 1) | ((t >> 1) << 2)) << (4 * b);
    }
    const bool swap_words = (g & 4) != 0;
    // 1x128 part: row r, half h; chunk j of the half read in the order j ^ 4h
    const int r1 = t0 >> 1, h1 = t0 & 1;
    const uint32_t step_q = step / KC, step_r = step % KC;
    uint32_t kc = blockIdx.x % KC, mb = blockIdx.x / KC;
    uint32_t it = 0;
    uint32_t t = blockIdx.x;
    for (; t < tiles; t += step, ++it) {
        const int s = static_cast<int>(it % S);
        if (!wait_bounded_warp(smem_addr(&full[s]), (it / S) & 1u, abort_flag, err_word)) break;
        const uint8_t* slot = ring + s * kQDualTileBytes;
        // ---- 128x1: both halves
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
            const uint8_t* half = slot + h * kQDualHalfBytes;
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                w[i] = *reinterpret_cast<const uint32_t*>(half + off[i & 7] + 128 * (i & 8));
            uint32_t mx = 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) mx = absmax_acc(mx, w[i]);
            mx &= 0x7FFF7FFFu;
            mx = absmax_acc(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = absmax_acc(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = absmax_acc(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const int c8 = lane & 7;
            const uint32_t m2 = __shfl_sync(0xffffffffu, mx, c8 >> 1);
            const float sc = group_scale((c8 & 1) ? bf16_hi(m2) : bf16_lo(m2));
            const float rc = __frcp_rn(sc);
            const uint32_t k0 = kc * 128 + 64 * h + 8 * warp;
            if (lane < 8) sxT[static_cast<size_t>(mb) * K + k0 + lane] = sc;
            const float sa = __shfl_sync(0xffffffffu, sc, 2 * cp), ra = __shfl_sync(0xffffffffu, rc, 2 * cp);
            const float sb = __shfl_sync(0xffffffffu, sc, 2 * cp + 1), rb = __shfl_sync(0xffffffffu, rc, 2 * cp + 1);
            const NegDiv da(sa, ra), db(sb, rb);
            uint32_t oa[4], ob[4];
            if (sa >= 0x1p-91f && sb >= 0x1p-91f)
                codes_cols16<true>(da, db, w, sel, oa, ob);
            else
                codes_cols16<false>(da, db, w, sel, oa, ob);
            const uint4 va = swap_words ? make_uint4(oa[1], oa[0], oa[3], oa[2]) : make_uint4(oa[0], oa[1], oa[2], oa[3]);
            const uint4 vb = swap_words ? make_uint4(ob[1], ob[0], ob[3], ob[2]) : make_uint4(ob[0], ob[1], ob[2], ob[3]);
            uint8_t* dst = xqT + static_cast<size_t>(k0 + 2 * cp) * M + mb * 128 + 16 * g;
            *reinterpret_cast<uint4*>(dst) = va;
            *reinterpret_cast<uint4*>(dst + M) = vb;
        }
        // ---- 1x128: row r1's group, half h1
        {
            const uint8_t* rowp = slot + h1 * kQDualHalfBytes + r1 * 128;
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = *reinterpret_cast<const uint4*>(rowp + (((j ^ (4 * h1)) ^ (r1 & 7)) << 4));
            uint32_t mx = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                mx = absmax_acc(mx, v[j].x);
                mx = absmax_acc(mx, v[j].y);
                mx = absmax_acc(mx, v[j].z);
                mx = absmax_acc(mx, v[j].w);
            }
            mx &= 0x7FFF7FFFu;
            mx = absmax_acc(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            const float sc = group_scale(amax_of_pair(mx));
            const NegDiv dv(sc, __frcp_rn(sc));
            const uint32_t m = mb * 128 + r1;
            // v[2i], v[2i+1] hold chunks 2i ^ 4h1 and its successor: 16 codes
            // for bytes 16 (i ^ 2h1) .. of this half of the row
            uint8_t* dst = xq + static_cast<size_t>(m) * ldq + kc * 128 + 64 * h1;
            if (sc >= 0x1p-91f) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<uint4*>(dst + 16 * (i ^ (2 * h1))) = codes_1x128<true>(dv, v[2 * i], v[2 * i + 1]);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<uint4*>(dst + 16 * (i ^ (2 * h1))) = codes_1x128<false>(dv, v[2 * i], v[2 * i + 1]);
            }
            if (h1 == 0) sx[static_cast<size_t>(kc) * M + m] = sc;
        }
        // the last warp to finish with the slot refills it
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const uint32_t prev = atomicAdd(&done[s], 1u);
            const uint32_t tn = t + S * step;
            if (prev == 8u * (it / S) + 7u && tn < tiles) issue(tn, s);
        }
        kc += step_r;
        mb += step_q;
        if (kc >= KC) {
            kc -= KC;
            ++mb;
        }
    }
    // A timed-out wait ends the loop early: a load still in flight into a
    // slot (at most one per slot) must land before the CTA releases the ring.
    __syncthreads();
    if (t0 == 0 && *abort_flag) {
        for (int s = 0; s < S; ++s) {
            const uint32_t n = *reinterpret_cast<volatile uint32_t*>(&issued[s]);
            if (n > 0) drain_load(smem_addr(&full[s]), (n - 1) & 1u);
        }
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
    // ceil(w_tiles 2^32 / (w_tiles + act_tiles)): the weight blocks among
    // items 0..n-1 number floor(n w_frac / 2^32), which steps by 0 or 1 and
    // reaches w_tiles at n = total
    uint64_t w_frac;
};

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_prev() {  // all groups but the newest
    asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// Item i of the list is a weight block when the count of weight blocks
// among items 0..i, floor((i + 1) w_frac / 2^32), steps up at i; *idx is then
// the block's index, else the activation tile's.
__device__ __forceinline__ bool pair_item(const PairArgs& p, uint32_t i, uint32_t* idx) {
    const uint32_t w_upto = static_cast<uint32_t>(((i + 1ull) * p.w_frac) >> 32);
    const bool is_w = w_upto > static_cast<uint32_t>((static_cast<uint64_t>(i) * p.w_frac) >> 32);
    *idx = is_w ? w_upto - 1 : i - w_upto;
    return is_w;
}

// Starts the loads of item t: weight block t into `tile`, or activation
// tile t into v.
__device__ __forceinline__ void pair_issue(const PairArgs& p, bool is_w, uint32_t t,
                                           uint16_t (*tile)[128], int row, int l4,
                                           uint4 (&v)[4]) {
    if (is_w) {
        const uint32_t NB = static_cast<uint32_t>(p.N / 128);
        const size_t n0 = static_cast<size_t>(t % NB) * 128, k0 = static_cast<size_t>(t / NB) * 128;
        const int ch = threadIdx.x & 15;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int r = (threadIdx.x >> 4) + 16 * q;
            cp_async16(&tile[r][ch * 8], p.w + (k0 + r) * p.ldw + n0 + ch * 8);
        }
    } else {
        const uint32_t KB = static_cast<uint32_t>(p.KB);
        load_1x128(p.x, static_cast<uint32_t>(p.M), p.ldx, t % KB, (t / KB) * kQ1Rows + row, l4, v);
    }
}

// Converts the weight block t staged in `tile` (all 256 threads).  Thread
// (cp = t0 & 63, rq = t0 >> 6) reads the two columns n = 2cp, 2cp+1 over
// the rows k = 32 rq .. 32 rq + 31 and converts each element once; its codes
// then go to two staging areas over `tile` (the block is in registers by
// then): [n][k] rows for wq, with 16-byte chunks XOR-swizzled by (n >> 1) & 7,
// and [k][n] rows for wqT, two bytes per row.  Both leave as 16-byte rows
// pieces.  Ends with a barrier, after which `tile` and `part` may be reused.
__device__ __forceinline__ void pair_weight_block(const PairArgs& p, uint32_t t,
                                                  uint16_t (*tile)[128], float* part) {
    const int t0 = threadIdx.x;
    const int lane = t0 & 31, warp = t0 >> 5;
    const uint32_t NB = static_cast<uint32_t>(p.N / 128), KB = static_cast<uint32_t>(p.KB);
    const uint32_t nb = t % NB, kb = t / NB;
    const size_t n0 = static_cast<size_t>(nb) * 128, k0 = static_cast<size_t>(kb) * 128;
    const size_t K = static_cast<size_t>(KB) * 128;
    const int cp = t0 & 63, rq = t0 >> 6;
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = *reinterpret_cast<const uint32_t*>(&tile[32 * rq + i][2 * cp]);
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) mx = absmax_acc(mx, w[i]);
    mx &= 0x7FFF7FFFu;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = absmax_acc(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) part[warp] = amax_of_pair(mx);
    __syncthreads();  // the block maxima are published and every value is in registers
    const float amax = fmaxf(fmaxf(fmaxf(part[0], part[1]), fmaxf(part[2], part[3])),
                             fmaxf(fmaxf(part[4], part[5]), fmaxf(part[6], part[7])));
    const float s = group_scale(amax);
    const NegDiv dv(s, __frcp_rn(s));
    if (t0 == 0) p.sw[static_cast<size_t>(nb) * KB + kb] = s;
    uint32_t A[8], B[8];  // column 2cp / 2cp+1: word m holds rows 32rq + 4m .. +3
    if (s >= 0x1p-91f) {
        codes_cols16<true>(dv, dv, w, 0x5410u, A, B);
        codes_cols16<true>(dv, dv, w + 16, 0x5410u, A + 4, B + 4);
    } else {
        codes_cols16<false>(dv, dv, w, 0x5410u, A, B);
        codes_cols16<false>(dv, dv, w + 16, 0x5410u, A + 4, B + 4);
    }
    uint8_t* cq = reinterpret_cast<uint8_t*>(tile);  // wq codes [128 n][128 k]
    uint8_t* cqT = cq + 128 * 128;                     // wqT codes [128 k][128 n]
    if (p.wq != nullptr) {
        const int na = 2 * cp, nb2 = 2 * cp + 1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = 2 * rq + h;  // 16-byte chunk of the 128-byte k row
            *reinterpret_cast<uint4*>(&cq[na * 128 + ((c ^ ((na >> 1) & 7)) << 4)]) =
                make_uint4(A[4 * h], A[4 * h + 1], A[4 * h + 2], A[4 * h + 3]);
            *reinterpret_cast<uint4*>(&cq[nb2 * 128 + ((c ^ ((nb2 >> 1) & 7)) << 4)]) =
                make_uint4(B[4 * h], B[4 * h + 1], B[4 * h + 2], B[4 * h + 3]);
        }
    }
    if (p.wqT != nullptr) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const uint32_t lo = prmt(A[m], B[m], 0x5140u), hi = prmt(A[m], B[m], 0x7362u);
            uint8_t* d = cqT + (32 * rq + 4 * m) * 128 + 2 * cp;
            *reinterpret_cast<uint16_t*>(d) = static_cast<uint16_t>(lo);
            *reinterpret_cast<uint16_t*>(d + 128) = static_cast<uint16_t>(lo >> 16);
            *reinterpret_cast<uint16_t*>(d + 256) = static_cast<uint16_t>(hi);
            *reinterpret_cast<uint16_t*>(d + 384) = static_cast<uint16_t>(hi >> 16);
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = t0 + kPairThreads * i;  // chunk j: row j / 8, chunk j % 8
        const int r = j >> 3, c = j & 7;
        if (p.wq != nullptr)
            *reinterpret_cast<uint4*>(p.wq + (n0 + r) * K + k0 + c * 16) =
                *reinterpret_cast<const uint4*>(&cq[r * 128 + ((c ^ ((r >> 1) & 7)) << 4)]);
        if (p.wqT != nullptr)
            *reinterpret_cast<uint4*>(p.wqT + (k0 + r) * static_cast<size_t>(p.N) + n0 + c * 16) =
                *reinterpret_cast<const uint4*>(&cqT[r * 128 + c * 16]);
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
    const uint32_t total = static_cast<uint32_t>(p.w_tiles + p.act_tiles);
    const uint32_t KB = static_cast<uint32_t>(p.KB);
    uint32_t i = blockIdx.x;  // item; the same in every thread of the CTA
    int buf = 0;
    uint4 v[4];
    uint32_t idx = 0;
    bool is_w = false;
    if (i < total) {
        is_w = pair_item(p, i, &idx);
        pair_issue(p, is_w, idx, tiles[0], row, l4, v);
    }
    cp_async_commit();
    while (i < total) {
        const uint32_t in = i + gridDim.x;
        uint4 vn[4];
        uint32_t idx_n = 0;
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
            quant_1x128_group(static_cast<uint32_t>(p.M), p.xq, p.ldq, p.sx, idx % KB,
                              (idx / KB) * kQ1Rows + row, l4, v);
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
// Persistent grid: as many CTAs as are resident (at most kQuantCtasPerSm per
// SM), never more than there are tiles.  A kernel with dynamic shared memory
// gets its size limit raised here, once per context; 0 if that fails.
template <auto kern>
static int64_t quant_grid(int64_t tiles, int smem = 0) {
    static ContextCache<int> per_sm;
    const int sms = sm_count_current();
    int n = 0;
    const int st = sms <= 0 ? static_cast<int>(FP8_ERR_CUDA) : per_sm.get(&n, [smem](int* v) {
        if (smem > 0 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return static_cast<int>(FP8_ERR_CUDA);
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kQuantThreads, smem) != cudaSuccess ||
            b <= 0)
            b = 1;
        *v = b < kQuantCtasPerSm ? b : kQuantCtasPerSm;
        return static_cast<int>(FP8_OK);
    });
    if (st != FP8_OK) {
        if (smem > 0) return 0;
        return tiles < 1024 ? tiles : 1024;
    }
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
    if (M > 0x7fffffffLL || tiles > 0x7fffffffLL) return FP8_ERR_UNSUPPORTED;  // 32-bit tile walk
    quant_act_1x128_kernel<<<static_cast<unsigned>(quant_grid<quant_act_1x128_kernel>(tiles)), kQuantThreads, 0,
                             static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(x), static_cast<uint32_t>(M), static_cast<uint32_t>(K / 128), ldx, xq,
        ldq, sx, static_cast<uint32_t>(tiles));
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
    // 32-bit tile walk and TMA coordinates
    const int64_t tiles = (M / 128) * (K / 64);
    if (M > 0x7fffffffLL || K > 0x7fffffffLL || tiles > 0x7fffffffLL) return FP8_ERR_UNSUPPORTED;
    unsigned* err = device_error_word();
    if (err == nullptr) return FP8_ERR_CUDA;
    CUtensorMap xmap;
    if (make_map(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(K),
                 static_cast<uint64_t>(M), static_cast<uint64_t>(ldx) * 2, 64, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B) != FP8_OK)
        return FP8_ERR_CUDA;
    const int64_t grid = quant_grid<quant_act_128x1_kernel>(tiles, kQ128x1Smem);
    if (grid <= 0) return FP8_ERR_CUDA;
    quant_act_128x1_kernel<<<static_cast<unsigned>(grid), kQuantThreads, kQ128x1Smem,
                             static_cast<cudaStream_t>(stream)>>>(
        xmap, static_cast<uint32_t>(M), static_cast<uint32_t>(K), xqT, sxT,
        static_cast<uint32_t>(tiles), err);
    return to_status(launch_status());
}

extern "C" fp8_status fp8_quant_act_dual(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                         int64_t ldq, float* sx, uint8_t* xqT, float* sxT, void* stream) {
    if (M < 0 || M % 128 != 0 || K <= 0 || K % 128 != 0 || ldx < K || ldq < K) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (x == nullptr || xq == nullptr || sx == nullptr || xqT == nullptr || sxT == nullptr)
        return FP8_ERR_NULL;
    if (ldx % 8 != 0 || ldq % 16 != 0 || !aligned(x, 16) || !aligned(xq, 16) || !aligned(xqT, 16) ||
        !aligned(sx, 4) || !aligned(sxT, 4))
        return FP8_ERR_ALIGN;
    // 32-bit tile walk and TMA coordinates
    const int64_t tiles = (M / 128) * (K / 128);
    if (M > 0x7fffffffLL || K > 0x7fffffffLL || tiles > 0x7fffffffLL) return FP8_ERR_UNSUPPORTED;
    unsigned* err = device_error_word();
    if (err == nullptr) return FP8_ERR_CUDA;
    CUtensorMap xmap;
    if (make_map(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(K),
                 static_cast<uint64_t>(M), static_cast<uint64_t>(ldx) * 2, 64, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B) != FP8_OK)
        return FP8_ERR_CUDA;
    const int64_t grid = quant_grid<quant_act_dual_kernel>(tiles, kQDualSmem);
    if (grid <= 0) return FP8_ERR_CUDA;
    quant_act_dual_kernel<<<static_cast<unsigned>(grid), kQuantThreads, kQDualSmem,
                            static_cast<cudaStream_t>(stream)>>>(
        xmap, static_cast<uint32_t>(M), static_cast<uint32_t>(K), xq, ldq, sx, xqT, sxT,
        static_cast<uint32_t>(tiles), err);
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
    // 32-bit item walk and row indices
    if (total > 0x7fffffffLL || p.M > 0x7fffffffLL || p.N / 128 > 0x7fffffffLL || p.KB > 0x7fffffffLL)
        return FP8_ERR_UNSUPPORTED;
    PairArgs q = p;
    q.w_frac = ((static_cast<uint64_t>(p.w_tiles) << 32) + static_cast<uint64_t>(total) - 1) /
               static_cast<uint64_t>(total);
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
    quant_fprop_pair_kernel<<<static_cast<unsigned>(grid), kPairThreads, kPairSmem, stream>>>(q);
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
