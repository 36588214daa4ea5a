// gemm.cu -- block-scaled FP8 GEMM with per-128-K FP32 promotion on the
// sm_103a tensor cores (tcgen05 + tensor memory + TMA).
//
// Method (DeepSeek-V3 Technical Report, section 3.3.2 and Figure 7(b)): the
// tensor cores form the partial sum of each 128-wide K interval; that partial
// is promoted to FP32, multiplied by the A-row scale and the B scale of the
// interval, and accumulated in FP32 outside the tensor core.
//
// Blackwell mapping (the report's H800 design copied WGMMA register partials
// to CUDA-core registers; here the partials live in tensor memory), 384
// threads in three warpgroups:
//   warp 0      TMA producer: A tile 128x128 and B tile BNx128 (E4M3, 128-byte
//               swizzle) per K block into a STAGES-deep shared-memory ring.
//   warps 1, 3  MMA issuers (warp 1 also allocates TMEM): four tcgen05.mma
//               kind::f8f6f4 (K = 32 each) per K block into one of the TMEM
//               partial buffers (two of 256 FP32 columns, or four of 128),
//               then tcgen05.commit to release the smem stage and to signal
//               the epilogue.  Dense and pair kernels alternate K blocks
//               between warps 1 and 3; the others issue from warp 1.  Roles
//               run as whole warps with one elected lane issuing.
//   warp 2      scale loader of the per-column (Wgrad) mode: each K block's
//               A and B scales into a shared-memory ring by bulk copies.
//   warps 4..11 promotion epilogue, two per TMEM lane quadrant: tcgen05.ld the
//               partial of K block kb, acc += partial * (sa[m,kb] * sb[kb])
//               (or * sb[n,kb] per column in the Wgrad mode) with FP32 FMAs
//               in registers, release the TMEM buffer; after the last K
//               block, convert and store the tile through a swizzled
//               shared-memory staging buffer and TMA bulk stores.
// The dense 256-wide kernels run on CTA pairs (clusters of two) whose tensor
// cores act as one on a 256 x 256 tile (tcgen05 cta_group::2): each CTA
// loads its 128 rows of A and half of B, so shared memory moves A + B/2 per
// K block in each direction instead of A + B.
// Group modes: dense; grouped over rows (MoE Fprop and Dgrad: tiles walk the
// expert row offsets); grouped over K (MoE Wgrad: every expert has the same
// output tiles and contracts over its own padded token range).
// The kernel is persistent: one CTA (or CTA pair) per SM (pair of SMs) walks
// a static tile schedule.
// Every barrier wait is bounded; on expiry the kernel records
// FP8_ERR_TIMEOUT in a device error word, unwinds and frees its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"
#include "quant_math.cuh"
#include "tensormap.cuh"

namespace fp8fg {

// bit 0: a barrier wait timed out; bit 1: invalid grouped offsets
__device__ unsigned int g_dev_error;

constexpr int BM = 128;               // rows per tile (TMEM lanes)
constexpr int BK = 128;               // K block = promotion interval
constexpr int kEpiWarps = 8;          // 2 per TMEM lane quadrant
constexpr int kEpiWarp0 = 4;          // epilogue = warpgroups 1 and 2
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
// Register split (setmaxnreg): the kernel is compiled for kLaunchRegs per
// thread (the cap 384 threads leave); the control warpgroup drops to
// kCtrlRegs and the two epilogue warpgroups rise to kEpiRegs.  The split must
// not exceed the launch allocation, or setmaxnreg.inc would wait forever:
// 128 * kCtrlRegs + 256 * kEpiRegs == 384 * kLaunchRegs.  The host refuses to
// launch a build whose register count differs from kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 40;
constexpr int kEpiRegs = 232;
static_assert(128 * kCtrlRegs + 256 * kEpiRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kSmemLimit = 232448;    // 227 KB opt-in per CTA

// Output staging: each epilogue warp owns kOutSlots swizzled 4 KB boxes
// (32 rows x 128 bytes); a TMA store is only waited on when its slot comes
// round again, so the store of one tile overlaps the next tile's K loop.
constexpr int kOutSlots = 2;
constexpr int kBoxBytes = 32 * 128;

// Scale ring: warp 2 copies each K block's scales into shared memory ahead of
// the epilogue (cp.async, completion on an mbarrier): the A scales of the
// tile's 128 rows, then the B scales of its columns (one per 128-column
// block, or one per column in the per-row B-scale mode).  The epilogue reads
// them there and frees the slot, so no global load sits on its path and no
// barrier couples its warps.
constexpr int kScaleSlots = 8;

// BSPLIT = 2: a CTA pair shares the tile's B rows, each stage holds half
template <int BN, bool ROWSCALE, int BSPLIT = 1>
struct Cfg {
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN / BSPLIT * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int COLS = BN / 2;           // columns per epilogue thread
    // Tensor memory holds NBUF partial buffers of the whole tile (all 512
    // columns): two for 256-wide tiles, four for 128-wide ones.  With four,
    // an epilogue thread's 64 columns fit in registers next to its
    // accumulators, so it hands the buffer back before any arithmetic.
    static constexpr int NBUF = 512 / BN;
    static constexpr int TMEM_COLS = NBUF * BN;
    static constexpr int SB_FLOATS = ROWSCALE ? BN : 4;   // B scales in a slot (padded)
    static constexpr int SLOT_FLOATS = BM + SB_FLOATS;
    static constexpr int RING_BYTES = ROWSCALE ? kScaleSlots * SLOT_FLOATS * 4 : 0;
    static constexpr int CSTAGE_BYTES = kEpiWarps * kOutSlots * kBoxBytes;
    static constexpr int HEADER = 512;            // barriers, TMEM slot, flags
    static constexpr int FIXED = HEADER + 1023 + CSTAGE_BYTES + RING_BYTES;
    static constexpr int STAGES_FIT = (kSmemLimit - FIXED) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
    static constexpr int SMEM = FIXED + STAGES * STAGE_BYTES;
    static constexpr int NBARS = 2 * STAGES + 2 * NBUF + 2 + 2 * kScaleSlots;
    static_assert(STAGES >= 2, "pipeline too shallow");
    static_assert(NBARS * 8 <= HEADER - 16, "header too small for barriers");
    static_assert(TMEM_COLS == 512, "TMEM allocation must be a power of 2");
};

struct GemmParams {
    const float* sa;      // sa[kb * lds_a + row]
    int64_t lds_a;
    const float* sb;      // B scales (layout per bmode)
    int64_t ld_sb;        // ROW1x128: row stride of sb
    int64_t sb_expert;    // grouped: floats per expert in sb
    int bmode;            // FP8_BSCALE_*
    int64_t M;            // dense: rows of A and C; grouped: T
    int64_t N, K;
    void* c;
    int64_t ldc;          // elements
    const int32_t* offsets;  // grouped only
    int E;
    // Split-K tail of the dense CTA-pair kernels: tiles >= full_tiles (the
    // last, partial wave) are split along K into sk chunks; each chunk's FP32
    // partial goes to ws, and the last chunk of a tile to finish sums them.
    int64_t full_tiles;   // tiles computed whole (all of them when sk == 1)
    int sk;               // K chunks per tail tile (1: no split)
    float* ws;            // [tail unit][CTA rank][BM][BN] FP32 partials
    int* ws_cnt;          // [tail tile][CTA rank] arrivals; zero between launches
};

struct Tile {
    int64_t row0;     // first row of A / C
    int64_t row_end;  // rows >= row_end are not this tile's
    int64_t b_row0;   // first row of B (expert-major for grouped)
    int64_t n0;       // first output column
    int expert;
    // grouped-K (per-expert contraction) and split-K tail tiles:
    int64_t c_row0;   // first row of C (expert-major; grouped-K only)
    int kb_begin;     // first K block of the range
    int kb_count;     // K blocks of the range (grouped-K: 0 writes the tile as zeros)
    int64_t split;    // split-K tail unit index, or -1
};

template <int BN, bool GROUPED>
__device__ __forceinline__ bool get_tile(const GemmParams& p, int64_t t, Tile& ti) {
    const int64_t nblk = p.N / BN;
    if (!GROUPED) {
        const int64_t mblk = (p.M + BM - 1) / BM;
        if (t >= mblk * nblk) return false;
        const int64_t mb = t / nblk, nb = t % nblk;
        ti.row0 = mb * BM;
        ti.row_end = p.M;
        ti.n0 = nb * BN;
        ti.b_row0 = ti.n0;
        ti.expert = 0;
        return true;
    } else {
        // 32-bit arithmetic (the host keeps the tile count below 2^30)
        const int t32 = static_cast<int>(t), nb32 = static_cast<int>(nblk);
        int base = 0;
        for (int e = 0; e < p.E; ++e) {
            const int lo = __ldg(p.offsets + e), hi = __ldg(p.offsets + e + 1);
            const int n_e = ((hi - lo + BM - 1) / BM) * nb32;
            if (t32 < base + n_e) {
                const int local = t32 - base;
                const int mb = local / nb32, nb = local % nb32;
                ti.row0 = lo + mb * BM;
                ti.row_end = hi;
                ti.n0 = static_cast<int64_t>(nb) * BN;
                ti.b_row0 = static_cast<int64_t>(e) * p.N + ti.n0;
                ti.expert = e;
                return true;
            }
            base += n_e;
        }
        return false;
    }
}

// Grouped-K tiles (the per-expert Wgrad GEMM): every expert has the same
// (M/128) x (N/BN) output tiles; its contraction covers the padded token
// columns pofs[e] .. pofs[e+1]-1 of both operands (p.offsets = pofs).
template <int BN>
__device__ __forceinline__ bool get_tile_gk(const GemmParams& p, int64_t t, Tile& ti) {
    const int64_t nblk = p.N / BN;
    const int64_t per_expert = (p.M / BM) * nblk;
    if (t >= per_expert * p.E) return false;
    const int64_t e = t / per_expert, local = t % per_expert;
    const int64_t mb = local / nblk, nb = local % nblk;
    ti.row0 = mb * BM;
    ti.row_end = p.M;
    ti.n0 = nb * BN;
    ti.b_row0 = ti.n0;
    ti.expert = static_cast<int>(e);
    ti.c_row0 = e * p.M + mb * BM;
    const int32_t lo = __ldg(p.offsets + e), hi = __ldg(p.offsets + e + 1);
    ti.kb_begin = lo / BK;
    ti.kb_count = (hi - lo) / BK;
    return true;
}

// Dense tiles of a cluster of CM CTAs along M: cluster tile t covers the CM
// row blocks CM*mg .. CM*mg+CM-1 of one BN-wide column block; CTA `rank`
// takes row block CM*mg + rank (past M when M has fewer blocks: its rows read
// as zeros and are not stored, but it keeps the cluster's schedule) and, in
// a CTA pair, B rows n0 + rank*BN/2 .. + BN/2 - 1.
template <int BN, int CM>
__device__ __forceinline__ bool get_tile_cluster(const GemmParams& p, int64_t t64, uint32_t rank,
                                                 Tile& ti) {
    // 32-bit arithmetic throughout (the host keeps every count below 2^31):
    // the control warps walk this at 40 registers.
    const int t = static_cast<int>(t64);
    const int nblk = static_cast<int>(p.N / BN);
    const int mgroups = static_cast<int>(((p.M + BM - 1) / BM + CM - 1) / CM);
    const int KBt = static_cast<int>(p.K / BK);
    const int full = static_cast<int>(p.full_tiles);
    int tile = t;
    ti.split = -1;
    ti.kb_begin = 0;
    ti.kb_count = KBt;
    if (t >= full) {  // a K chunk of a tail tile
        const int u = t - full;
        const int c = u % p.sk;
        tile = full + u / p.sk;
        ti.kb_begin = (c * KBt) / p.sk;
        ti.kb_count = ((c + 1) * KBt) / p.sk - ti.kb_begin;
        ti.split = u;
    }
    if (tile >= mgroups * nblk) return false;
    const int mg = tile / nblk, nb = tile % nblk;
    ti.row0 = static_cast<int64_t>(mg * CM + static_cast<int>(rank)) * BM;
    ti.row_end = p.M;
    ti.n0 = static_cast<int64_t>(nb) * BN;
    ti.b_row0 = ti.n0;
    ti.expert = 0;
    return true;
}

// GM: 0 dense, 1 grouped over rows (MoE Fprop/Dgrad), 2 grouped over K (MoE Wgrad)
template <int BN, int GM>
__device__ __forceinline__ bool get_tile_gm(const GemmParams& p, int64_t t, Tile& ti) {
    if constexpr (GM == 2)
        return get_tile_gk<BN>(p, t, ti);
    else
        return get_tile<BN, GM == 1>(p, t, ti);
}

// CM = 2: dense tiles of a CTA pair, this CTA's share by its rank
// Grouped-row tiles of a CTA pair: every expert's rows are cut into 256-row
// pair blocks (the last one ragged), times N / BN column blocks; CTA `rank`
// takes the pair block's 128-row half `rank` (rows at or past the expert's
// end are computed from whatever A holds there and not stored).  32-bit
// arithmetic: the control warps walk this at 40 registers.
template <int BN, int CM>
__device__ __forceinline__ bool get_tile_grouped_pair(const GemmParams& p, int64_t t64, uint32_t rank,
                                                      Tile& ti) {
    const int t = static_cast<int>(t64);
    const int nblk = static_cast<int>(p.N / BN);
    int base = 0;
    for (int e = 0; e < p.E; ++e) {
        const int lo = __ldg(p.offsets + e), hi = __ldg(p.offsets + e + 1);
        const int n_e = ((hi - lo + CM * BM - 1) / (CM * BM)) * nblk;
        if (t < base + n_e) {
            const int local = t - base;
            const int mp = local / nblk, nb = local % nblk;
            ti.row0 = lo + (mp * CM + static_cast<int>(rank)) * BM;
            ti.row_end = hi;
            ti.n0 = static_cast<int64_t>(nb) * BN;
            ti.b_row0 = static_cast<int64_t>(e) * p.N + ti.n0;
            ti.expert = e;
            ti.kb_begin = 0;
            ti.kb_count = static_cast<int>(p.K / BK);
            ti.split = -1;
            return true;
        }
        base += n_e;
    }
    return false;
}

template <int BN, int GM, int CM>
__device__ __forceinline__ bool get_tile_any(const GemmParams& p, int64_t t, Tile& ti) {
    if constexpr (CM > 1 && GM == 1)
        return get_tile_grouped_pair<BN, CM>(p, t, cluster_ctarank(), ti);
    else if constexpr (CM > 1)
        return get_tile_cluster<BN, CM>(p, t, cluster_ctarank(), ti);
    else
        return get_tile_gm<BN, GM>(p, t, ti);
}

// Shared-memory matrix descriptor of a K-major operand tile whose rows are
// 128 bytes (one 128-byte swizzle atom wide), 8-row core groups 1024 bytes
// apart: start address, leading byte offset 16 (unused for this layout),
// stride byte offset 1024, descriptor version 1, swizzle mode 128B.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor: E4M3 x E4M3 -> FP32, A and B K-major, M x N = MM x BN
// (MM = 256 for a CTA pair).
template <int BN, int MM = BM>
__device__ __forceinline__ uint32_t idesc_e4m3_f32() {
    return (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) |
           (static_cast<uint32_t>(MM >> 4) << 24);
}

__device__ __forceinline__ void raise_error(volatile int* abort_flag, unsigned bits) {
    raise_device_error(abort_flag, &g_dev_error, bits);
}
// Barrier over the eight epilogue warps (named barrier 1, 256 threads).
__device__ __forceinline__ void epilogue_sync() {
    asm volatile("bar.sync 1, 256;" ::: "memory");
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return wait_bounded(bar, parity, abort_flag, &g_dev_error);
}
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag) {
    return wait_bounded_warp(bar, parity, abort_flag, &g_dev_error);
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

// Block-mode promotion of an accumulator pair (two FP32 values in one 64-bit
// word, low half first): acc += p * s as two scalar FFMAs.  The packed
// fma.rn.f32x2 form measured slower in the epilogue (it keeps one FMA pipe
// busy for twice as long); every lane is the same IEEE round-to-nearest
// operation either way.
__device__ __forceinline__ uint64_t fma_pair(uint32_t p0, uint32_t p1, float s, uint64_t acc) {
    const float lo = fmaf(__uint_as_float(p0), s, __uint_as_float(static_cast<uint32_t>(acc)));
    const float hi = fmaf(__uint_as_float(p1), s, __uint_as_float(static_cast<uint32_t>(acc >> 32)));
    return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}

__device__ __forceinline__ uint32_t bf16x2(uint64_t pair) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(u2f(static_cast<uint32_t>(pair)),
                                                   u2f(static_cast<uint32_t>(pair >> 32)));
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <int BN, bool OUT_BF16, bool ROWSCALE, int GM, int CM>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_blockscaled_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    constexpr bool GROUPED = GM == 1;  // tiles walk the expert row offsets
    constexpr bool GK = GM == 2;       // every expert contracts over its own K range
    // CM = 2 (dense only): a cluster of two CTAs on neighbouring SMs whose
    // tensor cores work as one (tcgen05 cta_group::2) on a 256 x BN tile.
    // Each CTA loads its 128 rows of A and half of the tile's BN rows of B;
    // the even CTA issues M = 256 MMAs that read both CTAs' shared memory
    // and write each CTA's 128 rows of D into its own tensor memory.  Per SM
    // and K block the shared memory then takes A + B/2 bytes from TMA and
    // gives A + B/2 to the tensor core, instead of A + B each way.
    //   full[s]    (even CTA) both CTAs' TMA bytes of stage s
    //   empty[s]   (both) the pair's MMAs have read stage s: one commit,
    //              multicast to both CTAs
    //   tfull[b]   (both) partial buffer b written: multicast commit
    //   tempty[b]  (even CTA) every epilogue warp of both CTAs has read b
    // The epilogue, the scale ring and the output store are per CTA.
    constexpr bool PAIR = CM == 2;
    static_assert(CM == 1 || PAIR, "one CTA, or a CTA pair");
    static_assert(!PAIR || GM != 2, "CTA pairs serve the dense and grouped-row kernels");
    using C = Cfg<BN, ROWSCALE, CM>;
    constexpr int S = C::STAGES;
    constexpr int NBUF = C::NBUF;
    constexpr int SR = kScaleSlots;
    extern __shared__ uint8_t smem_raw[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + C::HEADER - 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + C::HEADER - 12);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem_raw + C::HEADER - 8);
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + C::HEADER + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = base;
    uint8_t* cstage = base + S * C::STAGE_BYTES;
    float* ring = reinterpret_cast<float*>(cstage + C::CSTAGE_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // barriers: operand stages full / empty, TMEM partial buffers full
    // (MMA done) / empty (drained), the MMA drain on abort, scale slots
    // full (copies landed) / empty (read by every epilogue warp)
    // (32-bit shared-window addresses: one register each)
    const uint32_t bars_s = smem_addr(bars);
    auto bar_at = [bars_s](int i) { return bars_s + 8u * static_cast<uint32_t>(i); };
    auto full_bar = [&](int s) { return bar_at(s); };
    auto empty_bar = [&](int s) { return bar_at(S + s); };
    auto tfull_bar = [&](int b) { return bar_at(2 * S + b); };
    auto tempty_bar = [&](int b) { return bar_at(2 * S + NBUF + b); };
    const uint32_t drain_bar = bar_at(2 * S + 2 * NBUF);  // and the next one: one per MMA issuer
    auto sfull_bar = [&](int r) { return bar_at(2 * S + 2 * NBUF + 2 + r); };
    auto sempty_bar = [&](int r) { return bar_at(2 * S + 2 * NBUF + 2 + SR + r); };
    // The scale loader runs as a whole warp in the dense and grouped-K
    // kernels and as one lane in the grouped-row kernels (whose tile walk
    // over the expert offsets is kept to single lanes).
    constexpr int kLoaderLanes = GROUPED ? 1 : 32;
    // The ring carries the per-column B scales of the Wgrad mode.  In the
    // block modes the epilogue needs two scalars per K block and prefetches
    // them from global memory two K blocks ahead instead.
    constexpr bool kRing = ROWSCALE;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), CM * kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        mbar_init(drain_bar + 8u, 1);
        for (int r = 0; r < SR; ++r) {
            mbar_init(sfull_bar(r), 1);
            mbar_init(sempty_bar(r), kEpiWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_addr(tmem_slot), C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // the peer's barriers are initialised before any arrival targets them
    if constexpr (PAIR) cluster_sync();
    // Nothing above reads global memory.  The operands, scales and offsets
    // may come from the kernel launched just before this one (the launch
    // allows a programmatic dependency), so wait for it here.
    griddep_wait();
    if (GROUPED) {
        // offsets[0] == 0, non-decreasing, offsets[E] <= T; checked by all threads
        bool bad = false;
        if (threadIdx.x == 0) bad = (__ldg(p.offsets) != 0) || (__ldg(p.offsets + p.E) > p.M);
        for (int e = threadIdx.x; e < p.E; e += kThreads)
            bad |= __ldg(p.offsets + e + 1) < __ldg(p.offsets + e);
        if (bad) raise_error(abort_flag, kErrBadOffsets);
        __syncthreads();
    }
    if (GK) {
        // padded K offsets: pofs[0] == 0, non-decreasing multiples of 128, pofs[E] <= K
        bool bad = false;
        if (threadIdx.x == 0) bad = (__ldg(p.offsets) != 0) || (__ldg(p.offsets + p.E) > p.K);
        for (int e = threadIdx.x; e < p.E; e += kThreads) {
            const int32_t lo = __ldg(p.offsets + e), hi = __ldg(p.offsets + e + 1);
            bad |= hi < lo || (hi % BK) != 0;
        }
        if (bad) raise_error(abort_flag, kErrBadOffsets);
        __syncthreads();
    }
    const uint32_t tmem_base = *tmem_slot;
    const int64_t KB = p.K / BK;
    const bool aborted_at_start = *abort_flag != 0;

    if (warp < kEpiWarp0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    }
    // The producer and the MMA issuer run as whole warps in every kernel:
    // every lane walks the schedule and waits on the barriers, so descriptors
    // and coordinates are warp-uniform and one elected lane issues the
    // asynchronous operations (issued from a single divergent lane, each
    // tcgen05.mma costs about twice the issue cycles).  The 32-bit tile walks
    // fit the control warps' 40 registers.  Two MMA issuers in the dense and
    // grouped-row pair kernels.
    constexpr bool kWarpRoles = true;
    constexpr bool kTwoIssuers = GM == 0 || (GROUPED && PAIR);
    constexpr bool kKRange = GK || PAIR;  // tiles carry their own K range
    auto role_wait = [&](uint32_t bar, uint32_t parity) {
        return kWarpRoles ? wait_bar_warp(bar, parity, abort_flag) : wait_bar(bar, parity, abort_flag);
    };
    auto role_sync = [&]() {
        if (kWarpRoles) __syncwarp();
    };
    // Tile schedule: a cluster (or a lone CTA, CM = 1) walks the tiles
    // blockIdx.x / CM, + gridDim.x / CM, ...; every role walks the same list.
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if ((kWarpRoles || lane == 0) && !aborted_at_start) {
            const bool leader = kWarpRoles ? elect_one() : true;
            uint32_t it = 0;          // K blocks issued
            int s = 0;                // stage of K block it, and its ring pass parity
            uint32_t ph = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x / CM; ok; t += gridDim.x / CM) {
                Tile ti;
                if (!get_tile_any<BN, GM, CM>(p, t, ti)) break;
                const int64_t nkb = kKRange ? ti.kb_count : KB;
                const int64_t kbo = kKRange ? ti.kb_begin : 0;
                for (int64_t kb = 0; kb < nkb; ++kb, ++it) {
                    if (!role_wait(empty_bar(s), ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    if (leader) {
                        uint8_t* st = stages + s * C::STAGE_BYTES;
                        const int kx = static_cast<int>((kb + kbo) * BK);
                        if constexpr (PAIR) {
                            // both CTAs' bytes land on the even CTA's barrier
                            const uint32_t rank = cluster_ctarank();
                            if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2 * C::STAGE_BYTES);
                            const uint32_t fb = mapa_shared(full_bar(s), 0);
                            tma_load_2d_pair(smem_addr(st), &tmA, fb, kx, static_cast<int>(ti.row0));
                            tma_load_2d_pair(smem_addr(st + C::A_BYTES), &tmB, fb, kx,
                                             static_cast<int>(ti.b_row0 + rank * (BN / 2)));
                        } else {
                            mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
                            tma_load_2d(smem_addr(st), &tmA, full_bar(s), kx, static_cast<int>(ti.row0));
                            tma_load_2d(smem_addr(st + C::A_BYTES), &tmB, full_bar(s), kx,
                                        static_cast<int>(ti.b_row0));
                        }
                    }
                    role_sync();
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!PAIR && !ok && leader) {
                // let copies already issued land before the CTA can exit
                const uint32_t n = it < static_cast<uint32_t>(S) ? it : static_cast<uint32_t>(S);
                for (uint32_t i = it - n; i < it; ++i) {
                    const long long t0 = clock64();
                    while (!mbar_try_wait(full_bar(static_cast<int>(i % S)), (i / S) & 1u) &&
                           clock64() - t0 < (1LL << 24)) {
                    }
                }
            }
            if (PAIR && leader) {
                // The pair's MMAs have released the last stages: every copy
                // into this CTA has been read (so has landed) and the even
                // CTA's last commits to this CTA's barriers have arrived.
                const uint32_t n = it < static_cast<uint32_t>(S) ? it : static_cast<uint32_t>(S);
                for (uint32_t i = it - n; i < it; ++i)
                    if (!wait_bar(empty_bar(static_cast<int>(i % S)), (i / S) & 1u, abort_flag)) break;
            }
            role_sync();
        }
    } else if (warp == 1 || (kTwoIssuers && warp == 3)) {
        // -------------------------------------------------------- MMA issuers
        // Dense kernels: warp 1 issues the even K blocks (global count), warp
        // 3 the odd ones.  Issuing tcgen05.mma holds up the tensor-memory
        // loads of the epilogue warps on the issuing warp's SM sub-partition,
        // so the load is split between two sub-partitions.  Every K block's
        // MMAs and commits come from one thread, and consecutive K blocks use
        // different TMEM buffers.  The grouped kernels issue from warp 1
        // alone (their tile walk leaves no registers for the split).  A CTA
        // pair: the even CTA issues for both.
        const uint32_t mine = warp == 1 ? 0u : 1u;
        if ((kWarpRoles || lane == 0) && !aborted_at_start && (!PAIR || cluster_ctarank() == 0)) {
            const bool leader = kWarpRoles ? elect_one() : true;
            const uint32_t idesc = idesc_e4m3_f32<BN, CM * BM>();
            uint32_t kbg = 0;  // K blocks walked (both issuers walk all)
            int s = 0;         // stage of K block kbg and its ring pass parity
            uint32_t ph = 0;
            bool ok = true, issued = false;
            for (int64_t t = blockIdx.x / CM; ok; t += gridDim.x / CM) {
                Tile ti;
                if (!get_tile_any<BN, GM, CM>(p, t, ti)) break;
                const int64_t nkb = kKRange ? ti.kb_count : KB;
                for (int64_t kb = 0; kb < nkb; ++kb, ++kbg) {
                    if (kTwoIssuers && (kbg & 1u) != mine) {
                        if (++s == S) {
                            s = 0;
                            ph ^= 1u;
                        }
                        continue;
                    }
                    const uint32_t buf = kbg % NBUF, tph = (kbg / NBUF) & 1u;
                    // tempty: in a pair the peer's epilogue warps arrive from the other CTA
                    if (!role_wait(full_bar(s), ph) || !role_wait(tempty_bar(buf), tph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_addr = smem_addr(stages + s * C::STAGE_BYTES);
                    const uint64_t adesc = smem_desc_sw128(a_addr);
                    const uint64_t bdesc = smem_desc_sw128(a_addr + C::A_BYTES);
                    const uint32_t d = tmem_base + buf * BN;
                    if (leader) {
                        if constexpr (PAIR) {
#pragma unroll
                            for (int k = 0; k < BK / 32; ++k)
                                mma_f8f6f4_pair(d, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
                            mma_commit_pair_mc(tfull_bar(buf), 3);
                            mma_commit_pair_mc(empty_bar(s), 3);
                        } else {
#pragma unroll
                            for (int k = 0; k < BK / 32; ++k)  // K = 32 bytes per MMA: +2 in 16-byte units
                                mma_f8f6f4(d, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
                            mma_commit(tfull_bar(buf));
                            mma_commit(empty_bar(s));
                        }
                    }
                    role_sync();
                    issued = true;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok && issued && leader) {
                // wait (bounded) for every MMA this thread issued before TMEM is freed
                const uint32_t db = drain_bar + 8u * mine;
                if constexpr (PAIR)
                    mma_commit_pair(db);
                else
                    mma_commit(db);
                const long long t0 = clock64();
                while (!mbar_try_wait(db, 0) && clock64() - t0 < (1LL << 24)) {
                }
            }
            if (PAIR && ok && leader) {
                // every epilogue warp of both CTAs has read this issuer's last
                // partials: no arrival from the peer is still on its way here
                const uint32_t nb = kbg < static_cast<uint32_t>(NBUF) ? kbg : static_cast<uint32_t>(NBUF);
                for (uint32_t j = kbg - nb; j < kbg; ++j)
                    if ((!kTwoIssuers || (j & 1u) == mine) &&
                        !wait_bar(tempty_bar(static_cast<int>(j % NBUF)), (j / NBUF) & 1u, abort_flag))
                        break;
            }
            role_sync();
        }
    } else if (warp == 2) {
        // ------------------------------------------------------ scale loader
        // (per-column B scales only) Per K block, slot it % SR receives the
        // A scales of the tile's 128 rows, then the B scales of its BN
        // columns.  Where both runs are 16-byte aligned and all the tile's
        // rows are inside the operand, one lane copies each run with one
        // bulk copy counted on the slot's full barrier.  Otherwise (a ragged
        // last row block, unaligned scale arrays) the lanes copy 4-byte
        // elements (rows past the operand read row M-1: never stored), wait
        // for them, and one lane arrives.
        if (kRing && (kLoaderLanes == 32 || lane == 0) && !aborted_at_start) {
            uint32_t it = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x / CM; ok; t += gridDim.x / CM) {
                Tile ti;
                if (!get_tile_any<BN, GM, CM>(p, t, ti)) break;
                const int64_t nkb = kKRange ? ti.kb_count : KB;
                const int64_t kbo = kKRange ? ti.kb_begin : 0;
                for (int64_t kb = 0; kb < nkb; ++kb, ++it) {
                    const int r = static_cast<int>(it % SR);
                    const uint32_t ph = (it / SR) & 1u;
                    const bool got = kLoaderLanes == 32 ? wait_bar_warp(sempty_bar(r), ph ^ 1u, abort_flag)
                                                        : wait_bar(sempty_bar(r), ph ^ 1u, abort_flag);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    const uint32_t slot = smem_addr(ring + r * C::SLOT_FLOATS);
                    const int64_t kg = kb + kbo;
                    const float* sa_k = p.sa + kg * p.lds_a + ti.row0;
                    const float* sb_k = p.sb + kg * p.ld_sb + ti.n0;
                    const bool bulk = ti.row0 + BM <= p.M &&
                                      ((reinterpret_cast<uintptr_t>(sa_k) |
                                        reinterpret_cast<uintptr_t>(sb_k)) & 15u) == 0;
                    if (bulk) {
                        if (lane == 0) {
                            mbar_arrive_expect_tx(sfull_bar(r), 4 * (BM + BN));
                            bulk_load(slot, sa_k, 4 * BM, sfull_bar(r));
                            bulk_load(slot + 4 * BM, sb_k, 4 * BN, sfull_bar(r));
                        }
                    } else {
                        const int64_t last = p.M - 1 - ti.row0;  // offset of row M-1
                        for (int i = lane; i < BM; i += kLoaderLanes)
                            cp_async4(slot + 4 * i, sa_k + (i <= last ? i : last));
                        for (int i = lane; i < BN; i += kLoaderLanes)
                            cp_async4(slot + 4 * (BM + i), sb_k + i);
                        cp_async_wait_all();
                        if (kLoaderLanes == 32) __syncwarp();
                        if (lane == 0) mbar_arrive(sfull_bar(r));
                    }
                    if (kLoaderLanes == 32) __syncwarp();
                }
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------- promotion epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
        constexpr int COLS = C::COLS;
        constexpr int ELT = OUT_BF16 ? 2 : 4;
        const int ew = warp - kEpiWarp0;      // 0..7
        const int q = warp & 3;               // TMEM lane quadrant of this warp
        const int cg = ew >> 2;               // column half of the tile
        constexpr int BOX_COLS = 128 / ELT;  // one 128-byte swizzle row per box row
        uint8_t* my_cstage = cstage + ew * kOutSlots * kBoxBytes;
        uint32_t boxes = 0;  // TMA boxes this warp has stored so far
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + cg * COLS;
        uint32_t kbg = 0;
        bool ok = !aborted_at_start;
        // shared addresses of a thread's entries in slot 0: its row's A
        // scale, its columns' B scales (slot r adds r * SLOT_FLOATS * 4)
        const uint32_t sa_addr0 = smem_addr(ring) + 4u * (q * 32 + lane);
        const uint32_t sb_addr0 =
            smem_addr(ring) + 4u * (BM + (ROWSCALE ? cg * COLS : (cg * COLS) / 128));
        // a pair's tempty barriers are the even CTA's (8 bytes apart there too)
        const uint32_t tempty0 = PAIR ? mapa_shared(tempty_bar(0), 0) : tempty_bar(0);
        auto release_tmem = [&](uint32_t buf) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    mbar_arrive_remote(tempty0 + 8u * buf);
                else
                    mbar_arrive(tempty_bar(buf));
            }
        };
        auto release_slot = [&](int r) {
            __syncwarp();
            if (lane == 0) mbar_arrive(sempty_bar(r));
        };
        for (int64_t t = blockIdx.x / CM; ok; t += gridDim.x / CM) {
            Tile ti;
            if (!get_tile_any<BN, GM, CM>(p, t, ti)) break;
            const int row = static_cast<int>(ti.row0) + q * 32 + lane;
            const int row_end = static_cast<int>(ti.row_end);
            const int ncol0 = static_cast<int>(ti.n0) + cg * COLS;
            const int nkb = kKRange ? ti.kb_count : static_cast<int>(KB);
            const int kbo = kKRange ? ti.kb_begin : 0;
            // block modes: this row's A scales sa[kb * lds_a + row] and the
            // B scale of this thread's 128-column block, two K blocks ahead
            const bool row_in_alloc = row < p.M;
            const int lds_a = static_cast<int>(p.lds_a);
            const float* sa_g = p.sa + static_cast<int64_t>(kbo) * lds_a + (row_in_alloc ? row : 0);
            const float* sb_g = nullptr;
            int sb_gstep = 0;
            // scales of K blocks kb+1 and kb+2 (loaded two blocks ahead)
            float sa_next = 0.0f, sb_next = 0.0f, sa_next2 = 0.0f, sb_next2 = 0.0f;
            if constexpr (!kRing) {
                const int nb = ncol0 / 128;
                const bool blk = p.bmode == FP8_BSCALE_BLOCK128;
                const int KBi = static_cast<int>(KB);
                sb_gstep = blk ? 1 : static_cast<int>(p.N / 128);
                sb_g = p.sb + (GROUPED ? ti.expert * p.sb_expert : 0) + (blk ? nb * KBi : nb) +
                       static_cast<int64_t>(kbo) * sb_gstep;
                if (nkb > 0) {
                    sa_next = row_in_alloc ? __ldg(sa_g) : 0.0f;
                    sb_next = __ldg(sb_g);
                }
                if (nkb > 1) {
                    sa_next2 = row_in_alloc ? __ldg(sa_g + lds_a) : 0.0f;
                    sb_next2 = __ldg(sb_g + sb_gstep);
                }
            }

            uint64_t acc[COLS / 2];
#pragma unroll
            for (int i = 0; i < COLS / 2; ++i) acc[i] = 0;

            for (int kb = 0; kb < nkb; ++kb, ++kbg) {
                const int r = static_cast<int>(kbg % SR);
                const uint32_t buf = kbg % NBUF, tph = (kbg / NBUF) & 1u;
                float sa_cur = sa_next, sb_cur = sb_next;
                if constexpr (!kRing) {
                    sa_next = sa_next2;
                    sb_next = sb_next2;
                    if (kb + 2 < nkb) {
                        sa_next2 = row_in_alloc ? __ldg(sa_g + (kb + 2) * lds_a) : 0.0f;
                        sb_next2 = __ldg(sb_g + (kb + 2) * sb_gstep);
                    }
                }
                if ((kRing && !wait_bar_warp(sfull_bar(r), (kbg / SR) & 1u, abort_flag)) ||
                    !wait_bar_warp(tfull_bar(buf), tph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t slot_off = static_cast<uint32_t>(r) * (C::SLOT_FLOATS * 4);
                if constexpr (kRing) sa_cur = lds_f32(sa_addr0 + slot_off);
                const uint32_t taddr = t_lane + buf * BN;
                if constexpr (COLS == 64) {
                    // 64 columns: load all of them, hand the TMEM buffer
                    // back, then promote from registers
                    uint32_t ra[32], rb[32];
                    tmem_ld32(taddr, ra);
                    tmem_ld32(taddr + 32, rb);
                    tmem_wait_ld(ra);
                    tmem_wait_ld(rb);
                    release_tmem(buf);
                    if constexpr (!ROWSCALE) {
                        const float sc = sa_cur * sb_cur;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            acc[i] = fma_pair(ra[2 * i], ra[2 * i + 1], sc, acc[i]);
                            acc[16 + i] = fma_pair(rb[2 * i], rb[2 * i + 1], sc, acc[16 + i]);
                        }
                    } else {
                        // per column: (P * sb[col]) * sa + acc, packed FP32 pairs
                        const uint64_t sa2 = pack2(f2u(sa_cur), f2u(sa_cur));
                        const uint32_t sbp = sb_addr0 + slot_off;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 b4 = lds_f32x4(sbp + 16 * i);
                            const uint64_t p0 = fmul2(pack2(ra[4 * i], ra[4 * i + 1]),
                                                      pack2(f2u(b4.x), f2u(b4.y)));
                            const uint64_t p1 = fmul2(pack2(ra[4 * i + 2], ra[4 * i + 3]),
                                                      pack2(f2u(b4.z), f2u(b4.w)));
                            acc[2 * i] = ffma2(p0, sa2, acc[2 * i]);
                            acc[2 * i + 1] = ffma2(p1, sa2, acc[2 * i + 1]);
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 b4 = lds_f32x4(sbp + 128 + 16 * i);
                            const uint64_t p0 = fmul2(pack2(rb[4 * i], rb[4 * i + 1]),
                                                      pack2(f2u(b4.x), f2u(b4.y)));
                            const uint64_t p1 = fmul2(pack2(rb[4 * i + 2], rb[4 * i + 3]),
                                                      pack2(f2u(b4.z), f2u(b4.w)));
                            acc[16 + 2 * i] = ffma2(p0, sa2, acc[16 + 2 * i]);
                            acc[16 + 2 * i + 1] = ffma2(p1, sa2, acc[16 + 2 * i + 1]);
                        }
                        release_slot(r);
                    }
                } else if constexpr (ROWSCALE) {
                    // 128 columns, two FP32 operations each: (P * sb[col]) * sa + acc.
                    // 16-column TMEM loads, three in flight (three load latencies
                    // per K block; more staging registers than this do not fit);
                    // the TMEM buffer goes back once the last loads have landed,
                    // the scale slot after the last column's arithmetic.
                    // (packed FP32 pairs here: the scalar form needs more registers)
                    const uint64_t sa2 = pack2(f2u(sa_cur), f2u(sa_cur));
                    const uint32_t sbp = sb_addr0 + slot_off;
                    auto fma16 = [&](uint32_t (&rr)[16], int ch) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float4 b4 = lds_f32x4(sbp + 4u * (ch * 16 + 4 * i));
                            const uint64_t p0 = fmul2(pack2(rr[4 * i], rr[4 * i + 1]),
                                                      pack2(f2u(b4.x), f2u(b4.y)));
                            const uint64_t p1 = fmul2(pack2(rr[4 * i + 2], rr[4 * i + 3]),
                                                      pack2(f2u(b4.z), f2u(b4.w)));
                            acc[ch * 8 + 2 * i] = ffma2(p0, sa2, acc[ch * 8 + 2 * i]);
                            acc[ch * 8 + 2 * i + 1] = ffma2(p1, sa2, acc[ch * 8 + 2 * i + 1]);
                        }
                    };
                    // 16-column loads, three in flight: chunks 0-2, 3-5, 6-7
                    uint32_t r0[16], r1[16], r2[16];
                    tmem_ld16(taddr, r0);
                    tmem_ld16(taddr + 16, r1);
                    tmem_ld16(taddr + 32, r2);
                    tmem_wait_ld16(r0);
                    tmem_wait_ld16(r1);
                    tmem_wait_ld16(r2);
                    fma16(r0, 0);
                    tmem_ld16(taddr + 48, r0);
                    fma16(r1, 1);
                    tmem_ld16(taddr + 64, r1);
                    fma16(r2, 2);
                    tmem_ld16(taddr + 80, r2);
                    tmem_wait_ld16(r0);
                    tmem_wait_ld16(r1);
                    tmem_wait_ld16(r2);
                    fma16(r0, 3);
                    tmem_ld16(taddr + 96, r0);
                    fma16(r1, 4);
                    tmem_ld16(taddr + 112, r1);
                    fma16(r2, 5);
                    tmem_wait_ld16(r0);
                    tmem_wait_ld16(r1);
                    release_tmem(buf);
                    fma16(r0, 6);
                    fma16(r1, 7);
                    release_slot(r);
                } else {
                    const float sc = sa_cur * sb_cur;
                    // 128 columns in 32-column TMEM loads: two in flight from
                    // the start, and each freed register chunk is refilled at
                    // once, so the whole partial has landed after two load
                    // latencies; the TMEM buffer goes back to the MMA before
                    // the last FMAs
                    uint32_t ra[32], rb[32];
                    tmem_ld32(taddr, ra);
                    tmem_ld32(taddr + 32, rb);
                    tmem_wait_ld(ra);
                    tmem_wait_ld(rb);
                    auto fma_chunk = [&](uint32_t (&rr)[32], int ch) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            acc[ch * 16 + i] = fma_pair(rr[2 * i], rr[2 * i + 1], sc, acc[ch * 16 + i]);
                    };
                    fma_chunk(ra, 0);
                    tmem_ld32(taddr + 64, ra);
                    fma_chunk(rb, 1);
                    tmem_ld32(taddr + 96, rb);
                    tmem_wait_ld(ra);
                    tmem_wait_ld(rb);
                    release_tmem(buf);
                    fma_chunk(ra, 2);
                    fma_chunk(rb, 3);
                }
            }
            if (!ok) break;

            if constexpr (PAIR) {
                if (ti.split >= 0) {
                    // Split-K tail: park this K chunk's partial; the last chunk
                    // of the tile to arrive (per CTA half) sums all of them in
                    // chunk order and stores the tile.  Nothing waits.
                    const uint32_t rank = cluster_ctarank();
                    const int64_t tail = ti.split / p.sk;
                    // A CTA's partial is [warp][16-byte chunk][lane]: a warp's
                    // store or load of one chunk index covers 512 contiguous bytes.
                    constexpr int kChunks = COLS / 4;
                    auto part_at = [&](int64_t unit) {
                        return reinterpret_cast<float4*>(p.ws) +
                               ((unit * CM + rank) * kEpiWarps + ew) * (kChunks * 32) + lane;
                    };
                    float4* mine_p = part_at(ti.split);
#pragma unroll
                    for (int i = 0; i < kChunks; ++i)
                        mine_p[i * 32] = make_float4(u2f(static_cast<uint32_t>(acc[2 * i])),
                                                     u2f(static_cast<uint32_t>(acc[2 * i] >> 32)),
                                                     u2f(static_cast<uint32_t>(acc[2 * i + 1])),
                                                     u2f(static_cast<uint32_t>(acc[2 * i + 1] >> 32)));
                    epilogue_sync();
                    if (ew == 0 && lane == 0) {
                        __threadfence();
                        const int old = atomicAdd(p.ws_cnt + tail * CM + rank, 1);
                        *last_flag = old == p.sk - 1;
                    }
                    epilogue_sync();
                    if (!*last_flag) continue;  // another chunk completes the tile
                    __threadfence();
#pragma unroll
                    for (int i = 0; i < COLS / 2; ++i) acc[i] = 0;
                    for (int c = 0; c < p.sk; ++c) {
                        const float4* src = part_at(tail * p.sk + c);
#pragma unroll
                        for (int i = 0; i < kChunks; ++i) {
                            const float4 v = __ldcg(src + i * 32);
                            acc[2 * i] = pack2(f2u(u2f(static_cast<uint32_t>(acc[2 * i])) + v.x),
                                               f2u(u2f(static_cast<uint32_t>(acc[2 * i] >> 32)) + v.y));
                            acc[2 * i + 1] =
                                pack2(f2u(u2f(static_cast<uint32_t>(acc[2 * i + 1])) + v.z),
                                      f2u(u2f(static_cast<uint32_t>(acc[2 * i + 1] >> 32)) + v.w));
                        }
                    }
                    epilogue_sync();  // every thread has read the counter's flag
                    if (ew == 0 && lane == 0) p.ws_cnt[tail * CM + rank] = 0;  // for the next launch
                }
            }

            // ---------------------------------------------------- tile store
            // grouped-K: C is [E][M][N], the tile's rows start at c_row0 and are all valid
            const int wrow0 = static_cast<int>(GK ? ti.c_row0 : ti.row0) + q * 32;
            if (GK || wrow0 + 32 <= row_end) {
                // whole 32-row box valid: stage with the 128-byte swizzle, TMA store
#pragma unroll
                for (int bx = 0; bx < COLS / BOX_COLS; ++bx, ++boxes) {
                    uint8_t* slotc = my_cstage + (boxes % kOutSlots) * kBoxBytes;
                    // the store that last used this slot must have read it
                    if (lane == 0 && boxes >= static_cast<uint32_t>(kOutSlots))
                        bulk_wait_group_read<kOutSlots - 1>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4 v;
                        if (OUT_BF16) {
                            const int a0 = (bx * BOX_COLS + j * 8) / 2;
                            v = make_uint4(bf16x2(acc[a0]), bf16x2(acc[a0 + 1]), bf16x2(acc[a0 + 2]),
                                           bf16x2(acc[a0 + 3]));
                        } else {
                            const int a0 = (bx * BOX_COLS + j * 4) / 2;
                            v = make_uint4(static_cast<uint32_t>(acc[a0]),
                                           static_cast<uint32_t>(acc[a0] >> 32),
                                           static_cast<uint32_t>(acc[a0 + 1]),
                                           static_cast<uint32_t>(acc[a0 + 1] >> 32));
                        }
                        *reinterpret_cast<uint4*>(slotc + lane * 128 + ((j ^ (lane & 7)) << 4)) = v;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, smem_addr(slotc), ncol0 + bx * BOX_COLS, wrow0);
                        bulk_commit_group();
                    }
                }
            } else if (row < row_end) {
                // ragged rows: direct 16-byte stores of this thread's row
                uint8_t* dst = static_cast<uint8_t*>(p.c) +
                               (static_cast<int64_t>(row) * p.ldc + ncol0) * ELT;
#pragma unroll
                for (int j = 0; j < COLS * ELT / 16; ++j) {
                    uint4 v;
                    if (OUT_BF16) {
                        v = make_uint4(bf16x2(acc[4 * j]), bf16x2(acc[4 * j + 1]),
                                       bf16x2(acc[4 * j + 2]), bf16x2(acc[4 * j + 3]));
                    } else {
                        v = make_uint4(static_cast<uint32_t>(acc[2 * j]),
                                       static_cast<uint32_t>(acc[2 * j] >> 32),
                                       static_cast<uint32_t>(acc[2 * j + 1]),
                                       static_cast<uint32_t>(acc[2 * j + 1] >> 32));
                    }
                    reinterpret_cast<uint4*>(dst)[j] = v;
                }
            }
        }
        if (lane == 0) bulk_wait_group0();

    }

    tc_fence_before_sync();
    __syncthreads();
    // a pair frees its tensor memory together, once both CTAs are done with
    // it; neither leaves while the other may still write to its barriers
    if constexpr (PAIR) cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// -------------------------------------------------------------------- host --
// Split-K workspace of the dense CTA-pair kernels: 4 KB of arrival counters
// (two per tail tile, zero between launches), then one 128 x 256 FP32
// partial per CTA of each tail unit.  A tail has at most one unit per pair.
constexpr int64_t kSplitCounterBytes = 4096;
constexpr int64_t kSplitPartialBytes = 128 * 256 * 4;
static int64_t kSplitUnitsMax(int sms) { return sms / 2; }
static int64_t split_workspace_bytes(int sms) {
    return kSplitCounterBytes + kSplitUnitsMax(sms) * 2 * kSplitPartialBytes;
}

// Launch configuration of one kernel instance, per context: the register
// check, the shared-memory opt-in (a kernel attribute belongs to the context
// it was set in) and, for clusters, how many can be resident at once.
struct LaunchInfo {
    int ok;
    int max_clusters;  // CM > 1 only
};

template <int BN, bool OUT_BF16, bool ROWSCALE, int GM, int CM>
static int launch(const uint8_t* aq, int64_t a_rows, const uint8_t* bq, int64_t b_rows,
                  const GemmParams& p, int64_t tiles_upper, cudaStream_t stream) {
    using C = Cfg<BN, ROWSCALE, CM>;
    auto kern = gemm_blockscaled_kernel<BN, OUT_BF16, ROWSCALE, GM, CM>;
    const int sms = sm_count_current();
    if (sms <= 0) return FP8_ERR_CUDA;
    static ContextCache<LaunchInfo> info_cache;
    LaunchInfo info{};
    const int ast = info_cache.get(&info, [&](LaunchInfo* v) {
        // the setmaxnreg split is only safe for the register count it was sized for
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return static_cast<int>(FP8_ERR_CUDA);
        if (fa.numRegs != kLaunchRegs) return static_cast<int>(FP8_ERR_UNSUPPORTED);
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
            cudaSuccess)
            return static_cast<int>(FP8_ERR_CUDA);
        v->ok = 1;
        v->max_clusters = 0;
        if (CM > 1) {
            cudaLaunchAttribute ca[1];
            ca[0].id = cudaLaunchAttributeClusterDimension;
            ca[0].val.clusterDim.x = CM;
            ca[0].val.clusterDim.y = 1;
            ca[0].val.clusterDim.z = 1;
            cudaLaunchConfig_t qc = {};
            qc.gridDim = dim3(static_cast<unsigned>(CM * (sms / CM)));
            qc.blockDim = dim3(kThreads);
            qc.dynamicSmemBytes = C::SMEM;
            qc.attrs = ca;
            qc.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &qc) != cudaSuccess || n <= 0) {
                (void)cudaGetLastError();
                return static_cast<int>(FP8_ERR_UNSUPPORTED);
            }
            v->max_clusters = n;
        }
        return static_cast<int>(FP8_OK);
    });
    if (ast != FP8_OK) return ast;
    CUtensorMap ta, tb, tc;
    int st;
    if ((st = make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, aq, p.K, a_rows, p.K, BK, BM,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != FP8_OK)
        return st;
    // in a CTA pair each CTA loads BN / 2 rows of B
    if ((st = make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, bq, p.K, b_rows, p.K, BK, BN / CM,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != FP8_OK)
        return st;
    constexpr int ELT = OUT_BF16 ? 2 : 4;
    const int64_t c_rows = GM == 2 ? p.M * p.E : p.M;  // grouped-K: one [M][N] per expert
    if ((st = make_map(&tc, OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                       p.c, p.N, c_rows, p.ldc * ELT, 128 / ELT, 32,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != FP8_OK)
        return st;
    // CM > 1: tiles_upper counts cluster tiles, and the grid holds whole
    // clusters, no more than can be resident at once
    const int64_t slots = CM > 1 ? info.max_clusters : sms;
    const int64_t grid = CM * (tiles_upper < slots ? tiles_upper : slots);
    if (grid <= 0) return FP8_OK;
    GemmParams q = p;
    q.full_tiles = tiles_upper;
    q.sk = 1;
    if (CM > 1 && p.ws != nullptr) {
        // Split-K tail: when the last wave of whole tiles would leave at least
        // half the pairs idle, its tiles are cut along K into sk chunks and
        // reduced by the last chunk to finish.  Summing one chunk's partial
        // costs about three K blocks of MMA time (measured), so the tail
        // takes about KB/sk + 3 sk K blocks: sk ~ sqrt(KB/3), and only deep
        // contractions (48 K blocks or more) gain.
        const int64_t P = grid / CM;
        const int64_t full = (tiles_upper / P) * P, rem = tiles_upper - full;
        const int64_t KBt = p.K / BK;
        int64_t cap = 1;
        while (3 * (cap + 1) * (cap + 1) <= KBt + 3 * cap) ++cap;  // round(sqrt(KB / 3))
        int64_t sk = rem > 0 ? P / rem : 0;
        if (sk > cap) sk = cap;
        if (KBt >= 48 && sk >= 2 && rem * sk <= kSplitUnitsMax(sms) &&
            rem * CM * 4 <= kSplitCounterBytes) {
            q.full_tiles = full;
            q.sk = static_cast<int>(sk);
        }
    }
    // Programmatic stream serialisation: the CTAs may be scheduled while the
    // previous kernel on the stream finishes (once it allows it); they set
    // up barriers and tensor memory, then wait for it in griddep_wait.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CM;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = CM > 1 ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, q) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8_ERR_CUDA;
    }
    return launch_status();
}

// The dense 256-wide kernels run as CTA pairs (cta_group::2)
constexpr int kClusterM = 2;
static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <int GM>
static int dispatch(const uint8_t* aq, int64_t a_rows, const uint8_t* bq, int64_t b_rows,
                    GemmParams& p, int out_type, int64_t mblk_upper, cudaStream_t stream) {
    constexpr bool GROUPED = GM == 1;
    if constexpr (GM == 2) {
        // the per-expert Wgrad GEMM: per-column B scales, FP32 out
        (void)out_type;
        (void)mblk_upper;
        if (p.N % 256 == 0) {
            const int64_t tiles = static_cast<int64_t>(p.E) * (p.M / BM) * (p.N / 256);
            return launch<256, false, true, 2, 1>(aq, a_rows, bq, b_rows, p, tiles, stream);
        }
        const int64_t tiles = static_cast<int64_t>(p.E) * (p.M / BM) * (p.N / 128);
        return launch<128, false, true, 2, 1>(aq, a_rows, bq, b_rows, p, tiles, stream);
    } else {
        const bool rows = p.bmode == FP8_BSCALE_ROW1x128;
        if constexpr (!GROUPED) {
            // per-column B scales (the Wgrad GEMM)
            if (rows) {
                if (p.N % 256 == 0 && ceil_div(mblk_upper, kClusterM) * (p.N / 256) < (1LL << 30)) {
                    const int64_t tiles = ceil_div(mblk_upper, kClusterM) * (p.N / 256);
                    if (out_type == FP8_OUT_BF16)
                        return launch<256, true, true, 0, kClusterM>(aq, a_rows, bq, b_rows, p, tiles,
                                                                     stream);
                    return launch<256, false, true, 0, kClusterM>(aq, a_rows, bq, b_rows, p, tiles,
                                                                  stream);
                }
                const int64_t tiles = mblk_upper * (p.N / 128);
                if (out_type == FP8_OUT_BF16)
                    return launch<128, true, true, 0, 1>(aq, a_rows, bq, b_rows, p, tiles, stream);
                return launch<128, false, true, 0, 1>(aq, a_rows, bq, b_rows, p, tiles, stream);
            }
            // 256-wide tiles on CTA pairs: per SM and K block, shared memory
            // moves A + B/2 each way instead of A + B.  A single 128-row
            // block takes the one-CTA 128-wide kernel below instead: a pair
            // would idle one of its CTAs, and the cluster set-up dominates
            // such short launches (128 x 256 x 512: 8.5 us against 11.5 us)
            if (p.N % 256 == 0 && mblk_upper > 1 &&
                ceil_div(mblk_upper, kClusterM) * (p.N / 256) < (1LL << 30)) {
                const int64_t tiles = ceil_div(mblk_upper, kClusterM) * (p.N / 256);
                if (out_type == FP8_OUT_BF16)
                    return launch<256, true, false, 0, kClusterM>(aq, a_rows, bq, b_rows, p, tiles,
                                                                  stream);
                return launch<256, false, false, 0, kClusterM>(aq, a_rows, bq, b_rows, p, tiles,
                                                               stream);
            }
        }
        // grouped rows, 256 columns wide: CTA pairs over 256-row blocks of
        // each expert (at most one ragged block per expert) when the experts
        // average 192 rows or more.  With fewer (decode-sized batches) most
        // pairs would hold one expert's rows in one CTA only: measured 20 %
        // slower there than one CTA per 128-row tile, which stays.
        if constexpr (GROUPED) {
            const int64_t pair_blocks = (p.M + kClusterM * BM - 1) / (kClusterM * BM) + p.E;
            if (p.N % 256 == 0 && p.M >= 192 * static_cast<int64_t>(p.E) &&
                pair_blocks * (p.N / 256) < (1LL << 30)) {
                const int64_t tiles = pair_blocks * (p.N / 256);
                if (out_type == FP8_OUT_BF16)
                    return launch<256, true, false, GM, kClusterM>(aq, a_rows, bq, b_rows, p, tiles,
                                                                   stream);
                return launch<256, false, false, GM, kClusterM>(aq, a_rows, bq, b_rows, p, tiles,
                                                                stream);
            }
        }
        // grouped rows with few rows per expert: one CTA per 128 x 256 tile
        if constexpr (GROUPED) {
            if (p.N % 256 == 0) {
                const int64_t tiles = mblk_upper * (p.N / 256);
                if (out_type == FP8_OUT_BF16)
                    return launch<256, true, false, GM, 1>(aq, a_rows, bq, b_rows, p, tiles, stream);
                return launch<256, false, false, GM, 1>(aq, a_rows, bq, b_rows, p, tiles, stream);
            }
        }
        // N % 256 != 0: one CTA per 128 x 128 tile
        const int64_t tiles = mblk_upper * (p.N / 128);
        if (out_type == FP8_OUT_BF16)
            return launch<128, true, false, GM, 1>(aq, a_rows, bq, b_rows, p, tiles, stream);
        return launch<128, false, false, GM, 1>(aq, a_rows, bq, b_rows, p, tiles, stream);
    }
}

// ------------------------------------------------------------ MXFP8 variant
// Block-scaled GEMM for power-of-two group scales (the quantisers of
// fp8_quant_act_1x128_pow2 / fp8_quant_weight_128x128_pow2).  With such
// scales the per-group dequantisation can run inside the tensor core, which
// the report wishes for (section 3.5.2): tcgen05.mma kind::mxf8f6f4 with
// block scaling multiplies each 32-element K slice of a row of A and of B by
// its UE8M0 exponent (our 128-wide groups repeat one exponent over four
// slices) and accumulates the whole K range in FP32 in tensor memory, so the
// epilogue drains the accumulator once per tile instead of promoting one
// partial per K block.  Exact only because every scale is a power of two.
//
// Roles (384 threads): warp 0 TMA producer (A 128x128, B BNx128 per K block),
// warp 1 TMEM allocator and MMA issuer, warp 2 scale loader, warps 4..11
// epilogue.  Per K block the loader writes the scale bytes of the tile's 128
// A rows and BN B rows as 32-row x 128-bit matrices (row r of a 128-row group
// at bytes 16 (r % 32) + 4 (r / 32) .. + 3, its exponent repeated in all four
// bytes) next to the stage, and the MMA warp copies them into tensor memory
// (tcgen05.cp, four lane quadrants) ahead of the stage's MMAs: a row's scale
// word ends up at lane r % 32 of each quadrant, column r / 32.
constexpr int kMxSfSlots = 4;   // tensor-memory scale slots, 16 columns each

template <int BN>
struct MxCfg {
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SF_BYTES = 512 * (1 + BN / 128);  // A's matrix, then B's
    static constexpr int COLS = BN / 2;
    static constexpr int CSTAGE_BYTES = kEpiWarps * kOutSlots * kBoxBytes;
    static constexpr int HEADER = 256;
    static constexpr int FIXED = HEADER + 1023 + CSTAGE_BYTES;
    static constexpr int STAGES_FIT = (kSmemLimit - FIXED) / (STAGE_BYTES + SF_BYTES);
    static constexpr int STAGES = STAGES_FIT > 4 ? 4 : STAGES_FIT;
    static constexpr int SMEM = FIXED + STAGES * (STAGE_BYTES + SF_BYTES);
    static constexpr int TMEM_COLS = 512;
    static constexpr int SF_COL0 = 256;  // scale slots after the accumulator
    static_assert(STAGES >= 2, "pipeline too shallow");
    static_assert((2 * STAGES + 3) * 8 <= HEADER - 16, "header too small");
    static_assert(SF_COL0 + kMxSfSlots * 16 <= TMEM_COLS, "scale slots outside the allocation");
};

struct MxParams {
    const uint8_t* sa_e8;  // [K/128][M] UE8M0 bytes
    const uint8_t* sb_e8;  // [K/128][N]
    int64_t M, N, K;
    void* c;
    int64_t ldc;
};

// Shared-memory descriptor of a 32-row x 16-byte matrix, rows contiguous (no
// swizzle): 8-row core groups 128 bytes apart, descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sf(uint32_t addr) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 32) |
           (static_cast<uint64_t>(1) << 46);
}

// Instruction descriptor of the block-scaled MMA: E4M3 x E4M3, A and B
// K-major, N = BN, M = 128, UE8M0 scales; sf_id picks the byte of the scale
// words for both operands.
template <int BN>
__device__ __forceinline__ uint32_t idesc_mxf8_e4m3(uint32_t sf_id) {
    return (sf_id << 4) | (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
           (static_cast<uint32_t>(BM >> 4) << 24) | (sf_id << 29);
}

template <int BN, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    mxfp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const MxParams p) {
    using C = MxCfg<BN>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + C::HEADER - 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + C::HEADER - 12);
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + C::HEADER + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = base;
    uint8_t* cstage = base + S * C::STAGE_BYTES;
    uint8_t* sf_ring = cstage + C::CSTAGE_BYTES;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bars_s = smem_addr(bars);
    auto full_bar = [&](int s) { return bars_s + 8u * s; };              // TMA bytes + scale loader
    auto empty_bar = [&](int s) { return bars_s + 8u * (S + s); };       // MMAs of the stage done
    const uint32_t tfull_bar = bars_s + 8u * (2 * S);                    // a tile's accumulator done
    const uint32_t tempty_bar = bars_s + 8u * (2 * S + 1);               // drained by the epilogue
    const uint32_t drain_bar = bars_s + 8u * (2 * S + 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 2);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, kEpiWarps);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    griddep_wait();
    const uint32_t tmem_base = *tmem_slot;
    const int64_t KB = p.K / BK;
    const int64_t nblk = p.N / BN;
    const int64_t tiles = ((p.M + BM - 1) / BM) * nblk;

    // Tile schedule: a cluster (or a lone CTA, CM = 1) walks the tiles
    // blockIdx.x / CM, + gridDim.x / CM, ...; every role walks the same list.
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        const bool leader = elect_one();
        uint32_t it = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
            const int row0 = static_cast<int>((t / nblk) * BM), n0 = static_cast<int>((t % nblk) * BN);
            for (int64_t kb = 0; kb < KB; ++kb, ++it) {
                const int s = static_cast<int>(it % S);
                if (!wait_bar_warp(empty_bar(s), ((it / S) & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    uint8_t* st = stages + s * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
                    tma_load_2d(smem_addr(st), &tmA, full_bar(s), static_cast<int>(kb * BK), row0);
                    tma_load_2d(smem_addr(st + C::A_BYTES), &tmB, full_bar(s),
                                static_cast<int>(kb * BK), n0);
                }
                __syncwarp();
            }
        }
        if (!ok && leader) {
            const uint32_t n = it < static_cast<uint32_t>(S) ? it : static_cast<uint32_t>(S);
            for (uint32_t i = it - n; i < it; ++i) {
                const long long t0 = clock64();
                while (!mbar_try_wait(full_bar(static_cast<int>(i % S)), (i / S) & 1u) &&
                       clock64() - t0 < (1LL << 24)) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        const bool leader = elect_one();
        uint32_t it = 0, tc = 0;
        bool ok = true, issued = false;
        for (int64_t t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++tc) {
            // the previous tile's accumulator must have been read
            if (!wait_bar_warp(tempty_bar, (tc & 1u) ^ 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            for (int64_t kb = 0; kb < KB; ++kb, ++it) {
                const int s = static_cast<int>(it % S);
                if (!wait_bar_warp(full_bar(s), (it / S) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a_addr = smem_addr(stages + s * C::STAGE_BYTES);
                const uint64_t adesc = smem_desc_sw128(a_addr);
                const uint64_t bdesc = smem_desc_sw128(a_addr + C::A_BYTES);
                const uint32_t sf_s = smem_addr(sf_ring + s * C::SF_BYTES);
                const uint32_t sfa = tmem_base + C::SF_COL0 + 16u * (it % kMxSfSlots);
                const uint32_t sfb = sfa + 4;
                if (leader) {
                    tmem_cp_32x128b_warpx4(sfa, smem_desc_sf(sf_s));
#pragma unroll
                    for (int c = 0; c < BN / 128; ++c)
                        tmem_cp_32x128b_warpx4(sfb + 4 * c, smem_desc_sf(sf_s + 512 * (1 + c)));
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_mxf8f6f4(tmem_base, adesc + 2 * k, bdesc + 2 * k,
                                     idesc_mxf8_e4m3<BN>(static_cast<uint32_t>(k)), sfa, sfb,
                                     (kb > 0 || k > 0) ? 1u : 0u);
                    mma_commit(empty_bar(s));
                }
                __syncwarp();
                issued = true;
            }
            if (!ok) break;
            if (leader) mma_commit(tfull_bar);
            __syncwarp();
        }
        if (!ok && issued && leader) {
            mma_commit(drain_bar);
            const long long t0 = clock64();
            while (!mbar_try_wait(drain_bar, 0) && clock64() - t0 < (1LL << 24)) {
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------ scale loader
        uint32_t it = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
            const int64_t row0 = (t / nblk) * BM, n0 = (t % nblk) * BN;
            for (int64_t kb = 0; kb < KB; ++kb, ++it) {
                const int s = static_cast<int>(it % S);
                if (!wait_bar_warp(empty_bar(s), ((it / S) & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                uint8_t* sf = sf_ring + s * C::SF_BYTES;
                const uint8_t* ea = p.sa_e8 + kb * p.M;
                uint32_t w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int64_t r = row0 + lane + 32 * j;
                    w[j] = static_cast<uint32_t>(__ldg(ea + (r < p.M ? r : p.M - 1))) * 0x01010101u;
                }
                *reinterpret_cast<uint4*>(sf + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
                const uint8_t* eb = p.sb_e8 + kb * p.N + n0;
#pragma unroll
                for (int c = 0; c < BN / 128; ++c) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        w[j] = static_cast<uint32_t>(__ldg(eb + 128 * c + lane + 32 * j)) * 0x01010101u;
                    *reinterpret_cast<uint4*>(sf + 512 * (1 + c) + 16 * lane) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async_smem();  // the tensor-memory copy reads it
                __syncwarp();
                if (lane == 0) mbar_arrive(full_bar(s));
            }
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        // ---------------------------------------------------------- epilogue
        constexpr int COLS = C::COLS;
        constexpr int ELT = OUT_BF16 ? 2 : 4;
        constexpr int BOX_COLS = 128 / ELT;
        const int ew = warp - kEpiWarp0, q = warp & 3, cg = ew >> 2;
        uint8_t* my_cstage = cstage + ew * kOutSlots * kBoxBytes;
        uint32_t boxes = 0, tc = 0;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + cg * COLS;
        for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++tc) {
            if (!wait_bar_warp(tfull_bar, tc & 1u, abort_flag)) break;
            tc_fence_after_sync();
            const int row0 = static_cast<int>((t / nblk) * BM);
            const int ncol0 = static_cast<int>((t % nblk) * BN) + cg * COLS;
            const int row = row0 + q * 32 + lane;
            const int wrow0 = row0 + q * 32;
            const bool whole = wrow0 + 32 <= p.M;
            // 32 columns at a time; a box (128 bytes of each of 32 rows) is
            // 64 BF16 or 32 FP32 columns
#pragma unroll 1
            for (int ch = 0; ch < COLS / 32; ++ch) {
                uint32_t r[32];
                tmem_ld32(t_lane + 32 * ch, r);
                tmem_wait_ld(r);
                if (ch == COLS / 32 - 1) {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty_bar);  // accumulator free for the next tile
                }
                uint4 pc[OUT_BF16 ? 4 : 8];  // this chunk's 16-byte pieces of the row
#pragma unroll
                for (int i = 0; i < (OUT_BF16 ? 4 : 8); ++i) {
                    if (OUT_BF16)
                        pc[i] = make_uint4(bf16x2(pack2(r[8 * i], r[8 * i + 1])),
                                           bf16x2(pack2(r[8 * i + 2], r[8 * i + 3])),
                                           bf16x2(pack2(r[8 * i + 4], r[8 * i + 5])),
                                           bf16x2(pack2(r[8 * i + 6], r[8 * i + 7])));
                    else
                        pc[i] = make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
                }
                if (whole) {
                    // BF16: chunks 2b and 2b+1 fill box b's pieces 0-3 and 4-7
                    const int box_first = OUT_BF16 ? (ch % 2 == 0) : true;
                    const int piece0 = OUT_BF16 ? (ch % 2) * 4 : 0;
                    uint8_t* slotc = my_cstage + (boxes % kOutSlots) * kBoxBytes;
                    if (box_first) {
                        if (lane == 0 && boxes >= static_cast<uint32_t>(kOutSlots))
                            bulk_wait_group_read<kOutSlots - 1>();
                        __syncwarp();
                    }
#pragma unroll
                    for (int i = 0; i < (OUT_BF16 ? 4 : 8); ++i) {
                        const int j = piece0 + i;
                        *reinterpret_cast<uint4*>(slotc + lane * 128 + ((j ^ (lane & 7)) << 4)) = pc[i];
                    }
                    const bool box_done = OUT_BF16 ? (ch % 2 == 1) : true;
                    if (box_done) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            const int bx_col = ncol0 + (OUT_BF16 ? (ch / 2) * BOX_COLS : ch * BOX_COLS);
                            tma_store_2d(&tmC, smem_addr(slotc), bx_col, wrow0);
                            bulk_commit_group();
                        }
                        ++boxes;
                    }
                } else if (row < p.M) {
                    uint4* dst = reinterpret_cast<uint4*>(
                        static_cast<uint8_t*>(p.c) + (static_cast<int64_t>(row) * p.ldc + ncol0 + 32 * ch) * ELT);
#pragma unroll
                    for (int i = 0; i < (OUT_BF16 ? 4 : 8); ++i) dst[i] = pc[i];
                }
            }
        }
        if (lane == 0) bulk_wait_group0();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int BN, bool OUT_BF16>
static int mx_launch(const uint8_t* aq, const uint8_t* bq, const MxParams& p, cudaStream_t stream) {
    using C = MxCfg<BN>;
    auto kern = mxfp8_gemm_kernel<BN, OUT_BF16>;
    const int sms = sm_count_current();
    if (sms <= 0) return FP8_ERR_CUDA;
    static ContextCache<int> attr_cache;
    int ok = 0;
    const int ast = attr_cache.get(&ok, [&](int* v) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
            cudaSuccess)
            return static_cast<int>(FP8_ERR_CUDA);
        *v = 1;
        return static_cast<int>(FP8_OK);
    });
    if (ast != FP8_OK) return ast;
    CUtensorMap ta, tb, tc;
    int st;
    if ((st = make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, aq, p.K, p.M, p.K, BK, BM,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != FP8_OK)
        return st;
    if ((st = make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, bq, p.K, p.N, p.K, BK, BN,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != FP8_OK)
        return st;
    constexpr int ELT = OUT_BF16 ? 2 : 4;
    if ((st = make_map(&tc, OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                       p.c, p.N, p.M, p.ldc * ELT, 128 / ELT, 32, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        FP8_OK)
        return st;
    const int64_t tiles = ((p.M + BM - 1) / BM) * (p.N / BN);
    const int64_t grid = tiles < sms ? tiles : sms;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8_ERR_CUDA;
    }
    return launch_status();
}

// ------------------------------------------------ activation cast fused in
// The report wishes the FP8 conversion of activations were fused with the
// TMA access that brings them in (section 3.5.2).  This GEMM takes A as
// bfloat16 and quantises it 1x128 inside the kernel: per K block the producer
// TMA-loads the BF16 A tile (two 64-column boxes, 128-byte swizzle) into one
// of two staging slots, and a converter warpgroup (four warps) converts it
// with the arithmetic of fp8_quant_act_1x128 (four lanes per row,
// amax by shuffles, the same correctly rounded quotients), writing the E4M3
// codes straight into the stage's swizzled A tile the MMA reads and the row
// scales into a ring the epilogue reads.  Codes and scales are the bits the
// 1x128 quantiser produces, so the output is bitwise the output of
// quantise-then-fp8_gemm_blockscaled.  B is the pre-quantised weight (block
// scales, Fprop or the transposed Dgrad layout); tiles are 128 x 256.
// 512 threads: warpgroup 0 producer / MMA issuer (warps 2-3 idle), warpgroup
// 1 the converter (four warps), warpgroups 2-3 the epilogue.  Register split
// (setmaxnreg) within the launch's 512 x 128: 128 x 40 + 128 x 64 + 256 x 200
// = 64512.  The host refuses a build whose register count is not 128.
constexpr int kFzThreads = 512;
constexpr int kFzLaunchRegs = 128;
constexpr int kFzConvRegs = 64;
constexpr int kFzEpiRegs = 200;
constexpr int kFzConvWarp0 = 4, kFzConvWarps = 4, kFzEpiWarp0 = 8;
static_assert(128 * kCtrlRegs + 128 * kFzConvRegs + 256 * kFzEpiRegs <= kFzThreads * kFzLaunchRegs,
              "fused register split");
constexpr int kFzStages = 2;   // operand stages (FP8 A tile + B tile)
constexpr int kFzSlots = 2;    // BF16 A staging slots
constexpr int kFzSR = 8;       // A-scale ring slots
constexpr int kFzOutSlots = 1;

struct FzCfg {
    static constexpr int BN = 256;
    static constexpr int A_BYTES = BM * BK;              // FP8 A tile
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int X_BYTES = BM * BK * 2;           // BF16 A tile (two boxes)
    static constexpr int COLS = BN / 2;
    static constexpr int CSTAGE_BYTES = kEpiWarps * kFzOutSlots * kBoxBytes;
    static constexpr int RING_BYTES = kFzSR * BM * 4;
    static constexpr int HEADER = 512;
    static constexpr int SMEM = HEADER + 1023 + kFzStages * STAGE_BYTES + kFzSlots * X_BYTES +
                                CSTAGE_BYTES + RING_BYTES;
    static constexpr int NBUF = 2;
    static constexpr int NBARS = 2 * kFzStages + 2 * kFzSlots + 2 * NBUF + 1 + 2 * kFzSR;
    static_assert(SMEM <= kSmemLimit, "fused GEMM does not fit shared memory");
    static_assert(NBARS * 8 <= HEADER - 16, "header too small");
};

template <bool OUT_BF16, int GM>
__global__ void __launch_bounds__(kFzThreads, 1)
    gemm_fused_act_kernel(const __grid_constant__ CUtensorMap tmX,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    constexpr bool GROUPED = GM == 1;
    using C = FzCfg;
    constexpr int BN = C::BN, S = kFzStages, SX = kFzSlots, SR = kFzSR, NBUF = C::NBUF;
    extern __shared__ uint8_t smem_raw[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + C::HEADER - 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + C::HEADER - 12);
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + C::HEADER + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = base;
    uint8_t* xslots = stages + S * C::STAGE_BYTES;
    uint8_t* cstage = xslots + SX * C::X_BYTES;
    float* ring = reinterpret_cast<float*>(cstage + C::CSTAGE_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bars_s = smem_addr(bars);
    auto bar_at = [bars_s](int i) { return bars_s + 8u * static_cast<uint32_t>(i); };
    // stage full: B bytes + both converter warps; stage empty: MMAs done
    auto full_bar = [&](int s) { return bar_at(s); };
    auto empty_bar = [&](int s) { return bar_at(S + s); };
    // BF16 slot full: A bytes landed; slot empty: both converter warps read it
    auto xfull_bar = [&](int x) { return bar_at(2 * S + x); };
    auto xempty_bar = [&](int x) { return bar_at(2 * S + SX + x); };
    auto tfull_bar = [&](int b) { return bar_at(2 * S + 2 * SX + b); };
    auto tempty_bar = [&](int b) { return bar_at(2 * S + 2 * SX + NBUF + b); };
    const uint32_t drain_bar = bar_at(2 * S + 2 * SX + 2 * NBUF);
    // A-scale ring: full (both converter warps wrote), empty (all epilogue warps read)
    auto sfull_bar = [&](int r) { return bar_at(2 * S + 2 * SX + 2 * NBUF + 1 + r); };
    auto sempty_bar = [&](int r) { return bar_at(2 * S + 2 * SX + 2 * NBUF + 1 + SR + r); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1 + kFzConvWarps);
            mbar_init(empty_bar(s), 1);
        }
        for (int x = 0; x < SX; ++x) {
            mbar_init(xfull_bar(x), 1);
            mbar_init(xempty_bar(x), kFzConvWarps);
        }
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        for (int r = 0; r < SR; ++r) {
            mbar_init(sfull_bar(r), kFzConvWarps);
            mbar_init(sempty_bar(r), kEpiWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    griddep_wait();
    if (GROUPED) {
        bool bad = false;
        if (threadIdx.x == 0) bad = (__ldg(p.offsets) != 0) || (__ldg(p.offsets + p.E) > p.M);
        for (int e = threadIdx.x; e < p.E; e += kFzThreads)
            bad |= __ldg(p.offsets + e + 1) < __ldg(p.offsets + e);
        if (bad) raise_error(abort_flag, kErrBadOffsets);
        __syncthreads();
    }
    const uint32_t tmem_base = *tmem_slot;
    const int64_t KB = p.K / BK;
    const bool aborted_at_start = *abort_flag != 0;
    if (warp < kFzConvWarp0)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    else if (warp < kFzEpiWarp0)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kFzConvRegs));
    constexpr bool kWarpRoles = !GROUPED;
    auto role_wait = [&](uint32_t bar, uint32_t parity) {
        return kWarpRoles ? wait_bar_warp(bar, parity, abort_flag) : wait_bar(bar, parity, abort_flag);
    };
    auto role_sync = [&]() {
        if (kWarpRoles) __syncwarp();
    };

    // Tile schedule: a cluster (or a lone CTA, CM = 1) walks the tiles
    // blockIdx.x / CM, + gridDim.x / CM, ...; every role walks the same list.
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if ((kWarpRoles || lane == 0) && !aborted_at_start) {
            const bool leader = kWarpRoles ? elect_one() : true;
            uint32_t it = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; ok; t += gridDim.x) {
                Tile ti;
                if (!get_tile<BN, GROUPED>(p, t, ti)) break;
                for (int64_t kb = 0; kb < KB; ++kb, ++it) {
                    const int s = static_cast<int>(it % S), x = static_cast<int>(it % SX);
                    if (!role_wait(empty_bar(s), ((it / S) & 1u) ^ 1u) ||
                        !role_wait(xempty_bar(x), ((it / SX) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    if (leader) {
                        uint8_t* st = stages + s * C::STAGE_BYTES;
                        mbar_arrive_expect_tx(full_bar(s), C::B_BYTES);
                        tma_load_2d(smem_addr(st + C::A_BYTES), &tmB, full_bar(s),
                                    static_cast<int>(kb * BK), static_cast<int>(ti.b_row0));
                        uint8_t* xs = xslots + x * C::X_BYTES;
                        mbar_arrive_expect_tx(xfull_bar(x), C::X_BYTES);
                        tma_load_2d(smem_addr(xs), &tmX, xfull_bar(x), static_cast<int>(kb * BK),
                                    static_cast<int>(ti.row0));
                        tma_load_2d(smem_addr(xs + C::X_BYTES / 2), &tmX, xfull_bar(x),
                                    static_cast<int>(kb * BK + 64), static_cast<int>(ti.row0));
                    }
                    role_sync();
                }
            }
            role_sync();
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        if ((kWarpRoles || lane == 0) && !aborted_at_start) {
            const bool leader = kWarpRoles ? elect_one() : true;
            const uint32_t idesc = idesc_e4m3_f32<BN>();
            uint32_t it = 0;
            bool ok = true, issued = false;
            for (int64_t t = blockIdx.x; ok; t += gridDim.x) {
                Tile ti;
                if (!get_tile<BN, GROUPED>(p, t, ti)) break;
                for (int64_t kb = 0; kb < KB; ++kb, ++it) {
                    const int s = static_cast<int>(it % S);
                    const uint32_t buf = it % NBUF, tph = (it / NBUF) & 1u;
                    if (!role_wait(full_bar(s), (it / S) & 1u) || !role_wait(tempty_bar(buf), tph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_addr = smem_addr(stages + s * C::STAGE_BYTES);
                    const uint64_t adesc = smem_desc_sw128(a_addr);
                    const uint64_t bdesc = smem_desc_sw128(a_addr + C::A_BYTES);
                    const uint32_t d = tmem_base + buf * BN;
                    if (leader) {
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k)
                            mma_f8f6f4(d, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
                        mma_commit(tfull_bar(buf));
                        mma_commit(empty_bar(s));
                    }
                    role_sync();
                    issued = true;
                }
            }
            if (!ok && issued && leader) {
                mma_commit(drain_bar);
                const long long t0 = clock64();
                while (!mbar_try_wait(drain_bar, 0) && clock64() - t0 < (1LL << 24)) {
                }
            }
            role_sync();
        }
    } else if (warp >= kFzConvWarp0 && warp < kFzEpiWarp0) {
        // ------------------------------------------------ 1x128 A converter
        // Per pass 32 rows (8 per warp), four lanes per row, 32 elements per
        // lane held in registers (one 64-column box holds a lane pair's 64).
        if (!aborted_at_start) {
            const int w = warp - kFzConvWarp0, l4 = lane & 3, box = l4 >> 1, half = l4 & 1;
            uint32_t it = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; ok; t += gridDim.x) {
                Tile ti;
                if (!get_tile<BN, GROUPED>(p, t, ti)) break;
                for (int64_t kb = 0; kb < KB; ++kb, ++it) {
                    const int s = static_cast<int>(it % S), x = static_cast<int>(it % SX);
                    const int r8 = static_cast<int>(it % SR);
                    if (!wait_bar_warp(xfull_bar(x), (it / SX) & 1u, abort_flag) ||
                        !wait_bar_warp(empty_bar(s), ((it / S) & 1u) ^ 1u, abort_flag) ||
                        !wait_bar_warp(sempty_bar(r8), ((it / SR) & 1u) ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t xs = smem_addr(xslots + x * C::X_BYTES) + box * (C::X_BYTES / 2);
                    const uint32_t as = smem_addr(stages + s * C::STAGE_BYTES);
                    const uint32_t sa_slot = smem_addr(ring + r8 * BM);
#pragma unroll 1
                    for (int pass = 0; pass < BM / (8 * kFzConvWarps); ++pass) {
                        const int r = pass * 8 * kFzConvWarps + w * 8 + (lane >> 2);
                        const uint32_t rowx = xs + r * 128;
                        uint32_t v[16];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float4 f = lds_f32x4(rowx + (((half * 4 + i) ^ (r & 7)) << 4));
                            v[4 * i] = __float_as_uint(f.x);
                            v[4 * i + 1] = __float_as_uint(f.y);
                            v[4 * i + 2] = __float_as_uint(f.z);
                            v[4 * i + 3] = __float_as_uint(f.w);
                        }
                        uint32_t mx = absmax_bf16x2(v[0], v[1]);
#pragma unroll
                        for (int i = 1; i < 8; ++i) mx = absmax_bf16x2(mx, absmax_bf16x2(v[2 * i], v[2 * i + 1]));
                        float amax = amax_of_pair(mx);
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                        const float sc = group_scale(amax);
                        const GroupDiv dv(sc);
                        uint32_t o[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) o[i] = dv.quad_words(v[2 * i], v[2 * i + 1]);
                        // the row's 128 codes: 16-byte chunks 2 l4 and 2 l4 + 1 (swizzled)
                        const uint32_t rowa = as + r * 128;
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         rowa + (((2 * l4) ^ (r & 7)) << 4)),
                                     "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                                     : "memory");
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         rowa + (((2 * l4 + 1) ^ (r & 7)) << 4)),
                                     "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                                     : "memory");
                        if (l4 == 0)
                            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sa_slot + 4u * r), "f"(sc)
                                         : "memory");
                    }
                    fence_proxy_async_smem();  // the MMA reads the codes through the async proxy
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(xempty_bar(x));
                        mbar_arrive(sfull_bar(r8));
                        mbar_arrive(full_bar(s));
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp >= kFzEpiWarp0) {
        // ------------------------------------------------- promotion epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kFzEpiRegs));
        constexpr int COLS = C::COLS;
        constexpr int ELT = OUT_BF16 ? 2 : 4;
        constexpr int BOX_COLS = 128 / ELT;
        const int ew = warp - kFzEpiWarp0, q = warp & 3, cg = ew >> 2;
        uint8_t* my_cstage = cstage + ew * kFzOutSlots * kBoxBytes;
        uint32_t boxes = 0, it = 0;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + cg * COLS;
        const uint32_t sa_addr0 = smem_addr(ring) + 4u * (q * 32 + lane);
        bool ok = !aborted_at_start;
        for (int64_t t = blockIdx.x; ok; t += gridDim.x) {
            Tile ti;
            if (!get_tile<BN, GROUPED>(p, t, ti)) break;
            const int row = static_cast<int>(ti.row0) + q * 32 + lane;
            const int row_end = static_cast<int>(ti.row_end);
            const int ncol0 = static_cast<int>(ti.n0) + cg * COLS;
            const int KBi = static_cast<int>(KB);
            const int nb = ncol0 / 128;
            const bool blk = p.bmode == FP8_BSCALE_BLOCK128;
            const float* sb_g = p.sb + (GROUPED ? ti.expert * p.sb_expert : 0) + (blk ? nb * KBi : nb);
            const int sb_step = blk ? 1 : static_cast<int>(p.N / 128);
            float sb_next = __ldg(sb_g);
            uint64_t acc[COLS / 2];
#pragma unroll
            for (int i = 0; i < COLS / 2; ++i) acc[i] = 0;
            for (int kb = 0; kb < KBi; ++kb, ++it) {
                const float sb_cur = sb_next;
                if (kb + 1 < KBi) sb_next = __ldg(sb_g + (kb + 1) * sb_step);
                const int r8 = static_cast<int>(it % SR);
                const uint32_t buf = it % NBUF, tph = (it / NBUF) & 1u;
                if (!wait_bar_warp(sfull_bar(r8), (it / SR) & 1u, abort_flag) ||
                    !wait_bar_warp(tfull_bar(buf), tph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const float sc = lds_f32(sa_addr0 + 4u * BM * r8) * sb_cur;
                __syncwarp();
                if (lane == 0) mbar_arrive(sempty_bar(r8));
                const uint64_t sc2 = pack2(f2u(sc), f2u(sc));
                const uint32_t taddr = t_lane + buf * BN;
                // 16-column TMEM loads, two in flight (the 200-register budget)
                auto fma16 = [&](uint32_t (&rr)[16], int ch) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc[ch * 8 + i] = ffma2(pack2(rr[2 * i], rr[2 * i + 1]), sc2, acc[ch * 8 + i]);
                };
                uint32_t r0[16], r1[16];
                tmem_ld16(taddr, r0);
                tmem_ld16(taddr + 16, r1);
#pragma unroll
                for (int ch = 0; ch < COLS / 16; ch += 2) {
                    tmem_wait_ld16(r0);
                    tmem_wait_ld16(r1);
                    if (ch + 2 < COLS / 16) {
                        fma16(r0, ch);
                        tmem_ld16(taddr + (ch + 2) * 16, r0);
                        fma16(r1, ch + 1);
                        tmem_ld16(taddr + (ch + 3) * 16, r1);
                    } else {
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(tempty_bar(buf));
                        fma16(r0, ch);
                        fma16(r1, ch + 1);
                    }
                }
            }
            if (!ok) break;
            const int wrow0 = static_cast<int>(ti.row0) + q * 32;
            if (wrow0 + 32 <= row_end) {
#pragma unroll
                for (int bx = 0; bx < COLS / BOX_COLS; ++bx, ++boxes) {
                    uint8_t* slotc = my_cstage + (boxes % kFzOutSlots) * kBoxBytes;
                    if (lane == 0 && boxes >= static_cast<uint32_t>(kFzOutSlots))
                        bulk_wait_group_read<kFzOutSlots - 1>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4 v;
                        if (OUT_BF16) {
                            const int a0 = (bx * BOX_COLS + j * 8) / 2;
                            v = make_uint4(bf16x2(acc[a0]), bf16x2(acc[a0 + 1]), bf16x2(acc[a0 + 2]),
                                           bf16x2(acc[a0 + 3]));
                        } else {
                            const int a0 = (bx * BOX_COLS + j * 4) / 2;
                            v = make_uint4(static_cast<uint32_t>(acc[a0]), static_cast<uint32_t>(acc[a0] >> 32),
                                           static_cast<uint32_t>(acc[a0 + 1]),
                                           static_cast<uint32_t>(acc[a0 + 1] >> 32));
                        }
                        *reinterpret_cast<uint4*>(slotc + lane * 128 + ((j ^ (lane & 7)) << 4)) = v;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, smem_addr(slotc), ncol0 + bx * BOX_COLS, wrow0);
                        bulk_commit_group();
                    }
                }
            } else if (row < row_end) {
                uint8_t* dst = static_cast<uint8_t*>(p.c) + (static_cast<int64_t>(row) * p.ldc + ncol0) * ELT;
#pragma unroll
                for (int j = 0; j < COLS * ELT / 16; ++j) {
                    uint4 v;
                    if (OUT_BF16)
                        v = make_uint4(bf16x2(acc[4 * j]), bf16x2(acc[4 * j + 1]), bf16x2(acc[4 * j + 2]),
                                       bf16x2(acc[4 * j + 3]));
                    else
                        v = make_uint4(static_cast<uint32_t>(acc[2 * j]), static_cast<uint32_t>(acc[2 * j] >> 32),
                                       static_cast<uint32_t>(acc[2 * j + 1]),
                                       static_cast<uint32_t>(acc[2 * j + 1] >> 32));
                    reinterpret_cast<uint4*>(dst)[j] = v;
                }
            }
        }
        if (lane == 0) bulk_wait_group0();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, 512);
    }
}

template <bool OUT_BF16, int GM>
static int fz_launch(const void* x, int64_t ldx, int64_t x_rows, const uint8_t* bq, int64_t b_rows,
                     const GemmParams& p, int64_t tiles_upper, cudaStream_t stream) {
    using C = FzCfg;
    auto kern = gemm_fused_act_kernel<OUT_BF16, GM>;
    const int sms = sm_count_current();
    if (sms <= 0) return FP8_ERR_CUDA;
    static ContextCache<int> attr_cache;
    int ok = 0;
    const int ast = attr_cache.get(&ok, [&](int* v) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return static_cast<int>(FP8_ERR_CUDA);
        if (fa.numRegs != kFzLaunchRegs) return static_cast<int>(FP8_ERR_UNSUPPORTED);
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
            cudaSuccess)
            return static_cast<int>(FP8_ERR_CUDA);
        *v = 1;
        return static_cast<int>(FP8_OK);
    });
    if (ast != FP8_OK) return ast;
    CUtensorMap tx, tb, tc;
    int st;
    // BF16 A: boxes of 64 columns (128 bytes) x 128 rows, 128-byte swizzle
    if ((st = make_map(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, p.K, x_rows, ldx * 2, 64, BM,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != FP8_OK)
        return st;
    if ((st = make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, bq, p.K, b_rows, p.K, BK, C::BN,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != FP8_OK)
        return st;
    constexpr int ELT = OUT_BF16 ? 2 : 4;
    if ((st = make_map(&tc, OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                       p.c, p.N, p.M, p.ldc * ELT, 128 / ELT, 32, CU_TENSOR_MAP_SWIZZLE_128B)) != FP8_OK)
        return st;
    const int64_t grid = tiles_upper < sms ? tiles_upper : sms;
    if (grid <= 0) return FP8_OK;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kFzThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tx, tb, tc, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8_ERR_CUDA;
    }
    return launch_status();
}

}  // namespace fp8fg

using namespace fp8fg;

// Shared body of fp8_gemm_blockscaled and fp8_gemm_blockscaled_ws (ws: the
// split-K workspace, or null).
static int dense_gemm(const uint8_t* aq, const float* sa, const uint8_t* bq, const float* sb,
                      int bmode, int64_t M, int64_t N, int64_t K, void* c, int64_t ldc, int out_type,
                      void* ws, int64_t ws_bytes, void* stream) {
    if (M < 0 || N <= 0 || N % 128 != 0 || K <= 0 || K % 128 != 0 || ldc < N)
        return FP8_ERR_SHAPE;
    if (bmode < FP8_BSCALE_BLOCK128 || bmode > FP8_BSCALE_BLOCK128_T) return FP8_ERR_UNSUPPORTED;
    if (out_type != FP8_OUT_F32 && out_type != FP8_OUT_BF16) return FP8_ERR_UNSUPPORTED;
    if (M == 0) return FP8_OK;
    if (aq == nullptr || sa == nullptr || bq == nullptr || sb == nullptr || c == nullptr)
        return FP8_ERR_NULL;
    const int64_t elt = out_type == FP8_OUT_BF16 ? 2 : 4;
    if (!aligned(aq, 16) || !aligned(bq, 16) || !aligned(c, 16) || !aligned(sa, 4) ||
        !aligned(sb, 4) || (ldc * elt) % 16 != 0)
        return FP8_ERR_ALIGN;
    if (M > 0x7fffffffLL || N > 0x7fffffffLL || K > 0x7fffffffLL) return FP8_ERR_UNSUPPORTED;
    GemmParams p{};
    p.sa = sa;
    p.lds_a = M;
    p.sb = sb;
    p.ld_sb = N;
    p.sb_expert = 0;
    p.bmode = bmode;
    p.M = M;
    p.N = N;
    p.K = K;
    p.c = c;
    p.ldc = ldc;
    p.offsets = nullptr;
    p.E = 0;
    if (ws != nullptr) {
        const int sms = sm_count_current();
        if (sms <= 0) return FP8_ERR_CUDA;
        if (!aligned(ws, 16)) return FP8_ERR_ALIGN;
        if (ws_bytes < split_workspace_bytes(sms)) return FP8_ERR_SHAPE;
        p.ws_cnt = static_cast<int*>(ws);
        p.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kSplitCounterBytes);
    }
    return dispatch<0>(aq, M, bq, N, p, out_type, (M + BM - 1) / BM,
                       static_cast<cudaStream_t>(stream));
}

extern "C" fp8_status fp8_gemm_blockscaled(const uint8_t* aq, const float* sa, const uint8_t* bq,
                                    const float* sb, fp8_bscale_t bmode, int64_t M, int64_t N, int64_t K,
                                    void* c, int64_t ldc, fp8_out_t out_type, void* stream) {
    return to_status(dense_gemm(aq, sa, bq, sb, bmode, M, N, K, c, ldc, out_type, nullptr, 0, stream));
}

extern "C" fp8_status fp8_gemm_blockscaled_ws(const uint8_t* aq, const float* sa, const uint8_t* bq,
                                       const float* sb, fp8_bscale_t bmode, int64_t M, int64_t N,
                                       int64_t K, void* c, int64_t ldc, fp8_out_t out_type,
                                       void* workspace, int64_t workspace_bytes, void* stream) {
    if (workspace == nullptr) return FP8_ERR_NULL;
    return to_status(dense_gemm(aq, sa, bq, sb, bmode, M, N, K, c, ldc, out_type, workspace,
                                workspace_bytes, stream));
}

extern "C" int64_t fp8_gemm_blockscaled_workspace_size(void) {
    const int sms = sm_count_current();
    return sms > 0 ? split_workspace_bytes(sms) : -1;
}

// Shared body of the grouped entry points; bmode is BLOCK128 (Fprop: per-expert
// sb[N/128][K/128]) or BLOCK128_T (Dgrad: the Fprop weight scales read transposed).
static int grouped_gemm(const uint8_t* aq, const float* sa, const uint8_t* bq, const float* sb,
                        int bmode, const int32_t* offsets, int32_t E, int64_t T, int64_t N,
                        int64_t K, void* c, int out_type, void* stream) {
    if (E < 1 || E > 65536 || T < 0 || N <= 0 || N % 128 != 0 || K <= 0 || K % 128 != 0)
        return FP8_ERR_SHAPE;
    if (out_type != FP8_OUT_F32 && out_type != FP8_OUT_BF16) return FP8_ERR_UNSUPPORTED;
    if (T == 0) return FP8_OK;
    if (aq == nullptr || sa == nullptr || bq == nullptr || sb == nullptr || offsets == nullptr ||
        c == nullptr)
        return FP8_ERR_NULL;
    if (!aligned(aq, 16) || !aligned(bq, 16) || !aligned(c, 16) || !aligned(sa, 4) ||
        !aligned(sb, 4) || !aligned(offsets, 4))
        return FP8_ERR_ALIGN;
    if (T > 0x7fffffffLL || static_cast<int64_t>(E) * N > 0x7fffffffLL || K > 0x7fffffffLL)
        return FP8_ERR_UNSUPPORTED;
    GemmParams p{};
    p.sa = sa;
    p.lds_a = T;
    p.sb = sb;
    p.ld_sb = 0;
    p.sb_expert = (N / 128) * (K / 128);
    p.bmode = bmode;
    p.M = T;
    p.N = N;
    p.K = K;
    p.c = c;
    p.ldc = N;
    p.offsets = offsets;
    p.E = E;
    // every expert adds at most one ragged M block
    return dispatch<1>(aq, T, bq, static_cast<int64_t>(E) * N, p, out_type,
                          (T + BM - 1) / BM + E, static_cast<cudaStream_t>(stream));
}

extern "C" fp8_status fp8_gemm_mxfp8(const uint8_t* aq, const uint8_t* sa_e8, const uint8_t* bq,
                                     const uint8_t* sb_e8, int64_t M, int64_t N, int64_t K,
                                     void* c, int64_t ldc, fp8_out_t out_type, void* stream) {
    if (M < 0 || N <= 0 || N % 128 != 0 || K <= 0 || K % 128 != 0 || ldc < N) return FP8_ERR_SHAPE;
    if (out_type != FP8_OUT_F32 && out_type != FP8_OUT_BF16) return FP8_ERR_UNSUPPORTED;
    if (M == 0) return FP8_OK;
    if (aq == nullptr || sa_e8 == nullptr || bq == nullptr || sb_e8 == nullptr || c == nullptr)
        return FP8_ERR_NULL;
    const int64_t elt = out_type == FP8_OUT_BF16 ? 2 : 4;
    if (!aligned(aq, 16) || !aligned(bq, 16) || !aligned(c, 16) || (ldc * elt) % 16 != 0)
        return FP8_ERR_ALIGN;
    if (M > 0x7fffffffLL || N > 0x7fffffffLL || K > 0x7fffffffLL) return FP8_ERR_UNSUPPORTED;
    MxParams p{sa_e8, sb_e8, M, N, K, c, ldc};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N % 256 == 0)
        return to_status(out_type == FP8_OUT_BF16 ? mx_launch<256, true>(aq, bq, p, s)
                                                  : mx_launch<256, false>(aq, bq, p, s));
    return to_status(out_type == FP8_OUT_BF16 ? mx_launch<128, true>(aq, bq, p, s)
                                              : mx_launch<128, false>(aq, bq, p, s));
}

extern "C" fp8_status fp8_gemm_blockscaled_bf16a(const void* x, int64_t ldx, const uint8_t* bq,
                                                 const float* sb, fp8_bscale_t bmode, int64_t M,
                                                 int64_t N, int64_t K, void* c, int64_t ldc,
                                                 fp8_out_t out_type, void* stream) {
    if (M < 0 || N <= 0 || N % 256 != 0 || K <= 0 || K % 128 != 0 || ldc < N || ldx < K)
        return FP8_ERR_SHAPE;
    if (bmode != FP8_BSCALE_BLOCK128 && bmode != FP8_BSCALE_BLOCK128_T) return FP8_ERR_UNSUPPORTED;
    if (out_type != FP8_OUT_F32 && out_type != FP8_OUT_BF16) return FP8_ERR_UNSUPPORTED;
    if (M == 0) return FP8_OK;
    if (x == nullptr || bq == nullptr || sb == nullptr || c == nullptr) return FP8_ERR_NULL;
    const int64_t elt = out_type == FP8_OUT_BF16 ? 2 : 4;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(bq, 16) || !aligned(c, 16) ||
        !aligned(sb, 4) || (ldc * elt) % 16 != 0)
        return FP8_ERR_ALIGN;
    if (M > 0x7fffffffLL || N > 0x7fffffffLL || K > 0x7fffffffLL) return FP8_ERR_UNSUPPORTED;
    GemmParams p{};
    p.sb = sb;
    p.bmode = bmode;
    p.M = M;
    p.N = N;
    p.K = K;
    p.c = c;
    p.ldc = ldc;
    const int64_t tiles = ((M + BM - 1) / BM) * (N / 256);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return to_status(out_type == FP8_OUT_BF16 ? fz_launch<true, 0>(x, ldx, M, bq, N, p, tiles, s)
                                              : fz_launch<false, 0>(x, ldx, M, bq, N, p, tiles, s));
}

extern "C" fp8_status fp8_grouped_gemm_moe_bf16a(const void* x, int64_t ldx, const uint8_t* bq,
                                                 const float* sb, const int32_t* offsets,
                                                 int32_t E, int64_t T, int64_t N, int64_t K,
                                                 void* c, fp8_out_t out_type, void* stream) {
    if (E < 1 || E > 65536 || T < 0 || N <= 0 || N % 256 != 0 || K <= 0 || K % 128 != 0 || ldx < K)
        return FP8_ERR_SHAPE;
    if (out_type != FP8_OUT_F32 && out_type != FP8_OUT_BF16) return FP8_ERR_UNSUPPORTED;
    if (T == 0) return FP8_OK;
    if (x == nullptr || bq == nullptr || sb == nullptr || offsets == nullptr || c == nullptr)
        return FP8_ERR_NULL;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(bq, 16) || !aligned(c, 16) || !aligned(sb, 4) ||
        !aligned(offsets, 4))
        return FP8_ERR_ALIGN;
    if (T > 0x7fffffffLL || static_cast<int64_t>(E) * N > 0x7fffffffLL || K > 0x7fffffffLL)
        return FP8_ERR_UNSUPPORTED;
    GemmParams p{};
    p.sb = sb;
    p.sb_expert = (N / 128) * (K / 128);
    p.bmode = FP8_BSCALE_BLOCK128;
    p.M = T;
    p.N = N;
    p.K = K;
    p.c = c;
    p.ldc = N;
    p.offsets = offsets;
    p.E = E;
    const int64_t tiles = ((T + BM - 1) / BM + E) * (N / 256);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t b_rows = static_cast<int64_t>(E) * N;
    return to_status(out_type == FP8_OUT_BF16 ? fz_launch<true, 1>(x, ldx, T, bq, b_rows, p, tiles, s)
                                              : fz_launch<false, 1>(x, ldx, T, bq, b_rows, p, tiles, s));
}

extern "C" fp8_status fp8_grouped_gemm_moe(const uint8_t* aq, const float* sa, const uint8_t* bq,
                                    const float* sb, const int32_t* offsets, int32_t E, int64_t T,
                                    int64_t N, int64_t K, void* c, fp8_out_t out_type, void* stream) {
    return to_status(grouped_gemm(aq, sa, bq, sb, FP8_BSCALE_BLOCK128, offsets, E, T, N, K, c, out_type,
                        stream));
}

extern "C" fp8_status fp8_grouped_gemm_moe_dgrad(const uint8_t* aq, const float* sa, const uint8_t* bq,
                                          const float* sb, const int32_t* offsets, int32_t E,
                                          int64_t T, int64_t N, int64_t K, void* c, fp8_out_t out_type,
                                          void* stream) {
    return to_status(grouped_gemm(aq, sa, bq, sb, FP8_BSCALE_BLOCK128_T, offsets, E, T, N, K, c,
                        out_type, stream));
}

extern "C" fp8_status fp8_grouped_gemm_moe_wgrad(const uint8_t* aqT, const float* sa,
                                          const uint8_t* bqT, const float* sb,
                                          const int32_t* pofs, int32_t E, int64_t Tp, int64_t M,
                                          int64_t N, float* c, void* stream) {
    if (E < 1 || E > 65536 || Tp < 0 || Tp % 128 != 0 || M <= 0 || M % 128 != 0 || N <= 0 ||
        N % 128 != 0)
        return FP8_ERR_SHAPE;
    if (aqT == nullptr || sa == nullptr || bqT == nullptr || sb == nullptr || pofs == nullptr ||
        c == nullptr)
        return FP8_ERR_NULL;
    if (!aligned(aqT, 16) || !aligned(bqT, 16) || !aligned(c, 16) || !aligned(sa, 4) ||
        !aligned(sb, 4) || !aligned(pofs, 4))
        return FP8_ERR_ALIGN;
    if (Tp > 0x7fffffffLL || static_cast<int64_t>(E) * M > 0x7fffffffLL || N > 0x7fffffffLL)
        return FP8_ERR_UNSUPPORTED;
    if (Tp == 0) Tp = 128;  // every expert empty: no operand is read, outputs are zero
    GemmParams p{};
    p.sa = sa;
    p.lds_a = M;
    p.sb = sb;
    p.ld_sb = N;
    p.bmode = FP8_BSCALE_ROW1x128;
    p.M = M;
    p.N = N;
    p.K = Tp;
    p.c = c;
    p.ldc = N;
    p.offsets = pofs;
    p.E = E;
    return to_status(dispatch<2>(aqT, M, bqT, N, p, FP8_OUT_F32, 0, static_cast<cudaStream_t>(stream)));
}

// Self-test of the failure path: one thread waits, through the same bounded
// wait as the GEMM roles, on a barrier nothing ever arrives on.  The wait gives
// up after its limit (about two seconds), records FP8_ERR_TIMEOUT in the
// device error word and the kernel returns.
__global__ void selftest_wait_kernel() {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)wait_bar(smem_addr(&bar), 0, &abort_flag);
}

extern "C" fp8_status fp8_selftest_wait_timeout(void* stream) {
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>();
    return to_status(launch_status());
}

// Device address of the error word in the current context, for kernels of
// the other translation units (the library is built without relocatable
// device code, so they cannot name g_dev_error themselves).
unsigned* fp8fg::device_error_word() {
    static ContextCache<unsigned*> cache;
    unsigned* p = nullptr;
    if (cache.get(&p, [](unsigned** v) {
            void* a = nullptr;
            if (cudaGetSymbolAddress(&a, g_dev_error) != cudaSuccess) return static_cast<int>(FP8_ERR_CUDA);
            *v = static_cast<unsigned*>(a);
            return static_cast<int>(FP8_OK);
        }) != FP8_OK)
        return nullptr;
    return p;
}

extern "C" fp8_status fp8_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FP8_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_dev_error, sizeof v) != cudaSuccess) return FP8_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_dev_error, &zero, sizeof zero) != cudaSuccess)
        return FP8_ERR_CUDA;
    if (v & kErrTimeout) return FP8_ERR_TIMEOUT;
    if (v & kErrBadOffsets) return FP8_ERR_DEVICE_SHAPE;
    return FP8_OK;
}
