// dispatch.cu -- MoE dispatch packing with fine-grained FP8 quantisation.
//
// Before the expert GEMMs, every token's activation row is sent to the
// experts its router chose, in FP8 (DeepSeek-V3 Technical Report, section
// 3.3.3, low-precision communication: the activations before the MoE
// up-projections are quantised to FP8 with the same fine-grained scheme and
// dispatched in that form).  On one GPU with a block of local experts this is
// a gather: for every local expert e, the tokens routed to it, in ascending
// token order, are written one after another as 1x128-quantised E4M3 rows, so
// that the rows of expert e occupy offsets[e] .. offsets[e+1]-1 -- exactly
// the A operand, A scales and offsets of fp8_grouped_gemm_moe.  1x128
// quantisation is row-local, so quantising the gathered rows gives the same
// bits as gathering quantised rows; a token sent to two local experts is
// quantised once and stored twice.
//
// Three launches, no atomics on global memory, deterministic placement:
//   count  one CTA per 64-token chunk: per-chunk histogram of local experts
//          into counts[e][chunk];
//   scan   one warp per expert: exclusive prefix of counts over the chunks
//          (in place) and the expert's total;
//   pack   one CTA per (chunk, K slice), as many as are resident at once
//          (one wave): the exclusive scan of the totals gives offsets; the
//          chunk's (token, expert) pairs are ranked in token order in two
//          parallel passes over a 64-bit token mask per expert, and the
//          tokens that have a local expert are listed; then all warps
//          quantise those tokens' 1x128 groups (the arithmetic of
//          fp8_quant_act_1x128) and store each group's codes and scale at
//          every destination row.  Tokens routed only to other experts are
//          not read.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8fg {

constexpr int kChunk = 64;          // tokens per chunk (one 64-bit token mask per expert)
constexpr int kMaxTopk = 16;
constexpr int kMaxLocal = 1024;     // local experts
constexpr int kPackThreads = 256;   // 64 four-lane groups
constexpr int kCountThreads = 256;  // four lanes per token of a chunk
static_assert(kPackThreads == 4 * kChunk && kCountThreads == 4 * kChunk,
              "four lanes per token of a chunk");

// Local expert index of slot j of a token's top-k row, or -1 when the expert
// is not local or repeats an earlier slot of the same row.
__device__ __forceinline__ int local_slot(const int32_t* ids, int j, int expert_begin, int E) {
    const int64_t e = static_cast<int64_t>(ids[j]) - expert_begin;
    if (e < 0 || e >= E) return -1;
    for (int i = 0; i < j; ++i)
        if (ids[i] == ids[j]) return -1;
    return static_cast<int>(e);
}

// The chunk's top-k rows are read coalesced into shared memory; lane
// (token, sub) then takes the token's slots sub, sub + 4, ...
__global__ void __launch_bounds__(kCountThreads) moe_count_kernel(
    const int32_t* __restrict__ topk_ids, int64_t T, int topk, int expert_begin, int E,
    int nchunks, int32_t* __restrict__ counts) {
    __shared__ int hist[kMaxLocal];
    __shared__ int32_t s_ids[kChunk * kMaxTopk];
    const int tid = threadIdx.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kChunk;
    const int n_tok = static_cast<int>(T - t0 < kChunk ? T - t0 : kChunk);
    for (int e = tid; e < E; e += kCountThreads) hist[e] = 0;
    for (int i = tid; i < n_tok * topk; i += kCountThreads) s_ids[i] = __ldg(topk_ids + t0 * topk + i);
    __syncthreads();
    const int tl = tid >> 2, sub = tid & 3;
    if (tl < n_tok) {
        for (int j = sub; j < topk; j += 4) {
            const int e = local_slot(&s_ids[tl * topk], j, expert_begin, E);
            if (e >= 0) atomicAdd(&hist[e], 1);
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kCountThreads)
        counts[static_cast<int64_t>(e) * nchunks + blockIdx.x] = hist[e];
}

// counts[e][c] -> sum of counts[e][c'] over c' < c; totals[e] = sum over all c.
__global__ void __launch_bounds__(256) moe_scan_kernel(int32_t* __restrict__ counts,
                                                       int32_t* __restrict__ totals, int E,
                                                       int nchunks) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp;
    if (e >= E) return;  // whole warp
    int32_t* row = counts + static_cast<int64_t>(e) * nchunks;
    // lane l takes the consecutive chunks c0 .. c1-1: its sum (independent
    // loads), an exclusive scan of the lane sums, then its prefixes
    const int per = (nchunks + 31) / 32;
    const int c0 = lane * per < nchunks ? lane * per : nchunks;
    const int c1 = c0 + per < nchunks ? c0 + per : nchunks;
    int sum = 0;
    for (int c = c0; c < c1; ++c) sum += row[c];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    int run = incl - sum;
    for (int c = c0; c < c1; ++c) {
        const int v = row[c];
        row[c] = run;
        run += v;
    }
    if (lane == 31) totals[e] = incl;
}

__global__ void __launch_bounds__(kPackThreads) moe_pack_quant_kernel(
    const uint16_t* __restrict__ x, int64_t T, int64_t KB, int64_t ldx,
    const int32_t* __restrict__ topk_ids, int topk, int expert_begin, int E,
    const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ totals, int nchunks,
    int kb_per_slice, uint8_t* __restrict__ xq, float* __restrict__ sx, int64_t cap,
    int32_t* __restrict__ offsets, int32_t* __restrict__ token_ids) {
    griddep_launch_dependents();  // the grouped GEMM that follows may set up meanwhile
    __shared__ int32_t s_ids[kChunk * kMaxTopk];
    __shared__ int32_t s_dest[kChunk * kMaxTopk];
    __shared__ int32_t s_base[kMaxLocal];
    __shared__ unsigned long long s_tok[kMaxLocal];  // per expert: its tokens of the chunk
    __shared__ int32_t s_wsum[kPackThreads / 32];
    __shared__ int32_t s_active[kChunk];  // chunk tokens with a local expert, ascending
    __shared__ unsigned long long s_act;  // the same tokens as a mask
    __shared__ uint32_t s_vmask[kChunk];  // per token: its slots with a local expert
    __shared__ int32_t s_nd[kChunk];      // per active token: its destination rows,
    __shared__ int32_t s_dl[kChunk * kMaxTopk];  // in slot order
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int64_t t0 = static_cast<int64_t>(c) * kChunk;
    const int n_tok = static_cast<int>(T - t0 < kChunk ? T - t0 : kChunk);
    const bool first_cta = c == 0 && blockIdx.y == 0;

    for (int i = tid; i < n_tok * topk; i += kPackThreads) s_ids[i] = __ldg(topk_ids + t0 * topk + i);
    if (tid == 0) s_act = 0ull;
    if (tid < kChunk) s_vmask[tid] = 0u;

    // exclusive scan of the expert totals (four experts per thread) -> offsets
    int v[4], sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = tid * 4 + i;
        v[i] = e < E ? __ldg(totals + e) : 0;
        sum += v[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kPackThreads / 32 ? s_wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < kPackThreads / 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        if (lane < kPackThreads / 32) s_wsum[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    int excl = incl - sum + (warp > 0 ? s_wsum[warp - 1] : 0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = tid * 4 + i;
        if (e < E) {
            s_base[e] = excl + __ldg(chunk_base + static_cast<int64_t>(e) * nchunks + c);
            s_tok[e] = 0ull;
            if (first_cta) offsets[e] = excl;
        }
        excl += v[i];
    }
    if (first_cta && tid == 0) offsets[E] = s_wsum[kPackThreads / 32 - 1];
    __syncthreads();

    // Rank the chunk's (token, local expert) pairs in token order, lane
    // (token, sub) taking the token's slots sub, sub + 4, ...  Pass 1: each
    // slot's local expert (or -1) into s_dest, the token's bit in its
    // expert's mask and in the mask of tokens with a local expert, and the
    // slot's bit in the token's slot mask.  Pass 2: the destination row is the
    // expert's first row for this chunk plus the number of the expert's tokens
    // ahead of this one in the chunk; each active token's rows are also listed
    // compactly, so that the quantising groups store without scanning slots.
    const int tl = tid >> 2, sub = tid & 3;
    const unsigned long long below = (1ull << tl) - 1ull;
    if (tl < n_tok) {
        bool any = false;
        for (int j = sub; j < topk; j += 4) {
            const int e = local_slot(&s_ids[tl * topk], j, expert_begin, E);
            s_dest[tl * topk + j] = e;
            if (e >= 0) {
                atomicOr(&s_tok[e], 1ull << tl);
                atomicOr(&s_vmask[tl], 1u << j);
                any = true;
            }
        }
        if (any) atomicOr(&s_act, 1ull << tl);
    }
    __syncthreads();
    if (tl < n_tok) {
        const bool act = ((s_act >> tl) & 1ull) != 0;
        const int a = __popcll(s_act & below);  // the token's index among the active ones
        const uint32_t vm = s_vmask[tl];
        for (int j = sub; j < topk; j += 4) {
            const int e = s_dest[tl * topk + j];
            if (e >= 0) {
                const int d = s_base[e] + __popcll(s_tok[e] & below);
                s_dest[tl * topk + j] = d;
                s_dl[a * kMaxTopk + __popc(vm & ((1u << j) - 1u))] = d;
            }
        }
        // tokens with no local expert are never read
        if (sub == 0 && act) {
            s_active[a] = tl;
            s_nd[a] = __popc(vm);
        }
    }
    __syncthreads();
    const int n_active = __popcll(s_act);

    if (blockIdx.y == 0) {
        for (int i = tid; i < n_tok * topk; i += kPackThreads) {
            const int d = s_dest[i];
            if (d >= 0) token_ids[d] = static_cast<int32_t>(t0 + i / topk);
        }
    }

    // 1x128 groups (token, kb) of this K slice: four lanes per group, 32
    // elements per lane, the arithmetic of the 1x128 quantiser.  Item it is
    // (active token it / nkb, K block kb0 + it % nkb); each group walks its
    // items with a fixed stride, advancing the pair without division, and
    // issues the next item's loads before it converts the current one.
    const int kb0 = blockIdx.y * kb_per_slice;
    const int kb1 = static_cast<int>(KB < kb0 + kb_per_slice ? KB : kb0 + kb_per_slice);
    const int nkb = kb1 - kb0;
    const int items = n_active * nkb;
    const int l4 = tid & 3;
    const uint32_t gmask = 0xFu << (lane & ~3);
    const int64_t K = KB * 128;
    constexpr int kStep = kPackThreads / 4;
    const int step_q = kStep / nkb, step_r = kStep % nkb;
    int it = tid >> 2;
    int ia = it / nkb, ib = it % nkb;  // active-token index and K block within the slice
    uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0, q2 = q0, q3 = q0;
    if (it < items) {
        const uint16_t* src = x + (t0 + s_active[ia]) * ldx + static_cast<int64_t>(kb0 + ib) * 128 + l4 * 32;
        q0 = ld_stream_v4(src);
        q1 = ld_stream_v4(src + 8);
        q2 = ld_stream_v4(src + 16);
        q3 = ld_stream_v4(src + 24);
    }
    for (; it < items; it += kStep) {
        int na = ia + step_q, nb = ib + step_r;
        if (nb >= nkb) {
            nb -= nkb;
            ++na;
        }
        uint4 n0 = make_uint4(0, 0, 0, 0), n1 = n0, n2 = n0, n3 = n0;
        if (it + kStep < items) {  // the next item's loads, in flight during the conversion
            const uint16_t* src = x + (t0 + s_active[na]) * ldx + static_cast<int64_t>(kb0 + nb) * 128 + l4 * 32;
            n0 = ld_stream_v4(src);
            n1 = ld_stream_v4(src + 8);
            n2 = ld_stream_v4(src + 16);
            n3 = ld_stream_v4(src + 24);
        }
        const uint4 q[4] = {q0, q1, q2, q3};
        uint32_t mx = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            mx = absmax_acc(mx, q[i].x);
            mx = absmax_acc(mx, q[i].y);
            mx = absmax_acc(mx, q[i].z);
            mx = absmax_acc(mx, q[i].w);
        }
        mx &= 0x7FFF7FFFu;
        mx = absmax_acc(mx, __shfl_xor_sync(gmask, mx, 1));
        mx = absmax_acc(mx, __shfl_xor_sync(gmask, mx, 2));
        const float s = group_scale(amax_of_pair(mx));
        const NegDiv dv(s, __frcp_rn(s));
        uint4 o0, o1;
        if (s >= 0x1p-91f) {
            o0 = codes_1x128<true>(dv, q[0], q[1]);
            o1 = codes_1x128<true>(dv, q[2], q[3]);
        } else {
            o0 = codes_1x128<false>(dv, q[0], q[1]);
            o1 = codes_1x128<false>(dv, q[2], q[3]);
        }
        const int kb = kb0 + ib;
        const int nd = s_nd[ia];
        for (int k = 0; k < nd; ++k) {
            const int d = s_dl[ia * kMaxTopk + k];
            uint4* dst = reinterpret_cast<uint4*>(xq + static_cast<int64_t>(d) * K +
                                                  static_cast<int64_t>(kb) * 128 + l4 * 32);
            dst[0] = o0;
            dst[1] = o1;
            if (l4 == 0) sx[static_cast<int64_t>(kb) * cap + d] = s;
        }
        q0 = n0;
        q1 = n1;
        q2 = n2;
        q3 = n3;
        ia = na;
        ib = nb;
    }
}

struct DispatchPlan {
    int nchunks = 0;
    size_t count_ints = 0;  // counts[E][nchunks]
    size_t bytes = 0;       // counts + totals, 256-byte granules
};

static DispatchPlan dispatch_plan(int64_t T, int E) {
    DispatchPlan d;
    d.nchunks = static_cast<int>((T + kChunk - 1) / kChunk);
    d.count_ints = static_cast<size_t>(E) * d.nchunks;
    const size_t ints = d.count_ints + static_cast<size_t>(E);
    d.bytes = (ints * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
    return d;
}

static int dispatch_checks(int64_t T, int64_t K, int64_t ldx, int32_t topk, int32_t n_local,
                           int64_t cap) {
    if (T < 0 || K <= 0 || K % 128 != 0 || ldx < K || topk < 1 || topk > kMaxTopk ||
        n_local < 1 || n_local > kMaxLocal || cap < 0)
        return FP8_ERR_SHAPE;
    if (T > (static_cast<int64_t>(1) << 31) / kMaxTopk) return FP8_ERR_UNSUPPORTED;
    if (cap < T * std::min<int64_t>(topk, n_local) || cap > 0x7fffffffLL) return FP8_ERR_SHAPE;
    return FP8_OK;
}

// The three launches on a workspace of at least dispatch_plan().bytes.
static int dispatch_launch(const void* x, int64_t T, int64_t K, int64_t ldx,
                           const int32_t* topk_ids, int32_t topk, int32_t expert_begin,
                           int32_t n_local, uint8_t* xq, float* sx, int64_t cap,
                           int32_t* offsets, int32_t* token_ids, int32_t* scratch,
                           cudaStream_t stream) {
    const DispatchPlan d = dispatch_plan(T, n_local);
    int32_t* counts = scratch;
    int32_t* totals = scratch + d.count_ints;
    // (chunk, K slice) CTAs of the pack: as many slices per chunk as fit in
    // one wave of resident CTAs (a second, partial wave measured 20 % slower)
    const int sms = sm_count_current();
    if (sms <= 0) return FP8_ERR_CUDA;
    static ContextCache<int> per_sm;
    int resident = 0;
    const int ost = per_sm.get(&resident, [](int* v) {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, moe_pack_quant_kernel, kPackThreads, 0) !=
                cudaSuccess ||
            b < 1)
            return static_cast<int>(FP8_ERR_CUDA);
        *v = b;
        return static_cast<int>(FP8_OK);
    });
    if (ost != FP8_OK) return ost;
    const int64_t KB = K / 128;
    int64_t slices = static_cast<int64_t>(resident) * sms / d.nchunks;
    slices = std::max<int64_t>(1, std::min<int64_t>(slices, KB));
    const int kb_per_slice = static_cast<int>((KB + slices - 1) / slices);
    slices = (KB + kb_per_slice - 1) / kb_per_slice;

    moe_count_kernel<<<d.nchunks, kCountThreads, 0, stream>>>(topk_ids, T, topk, expert_begin,
                                                               n_local, d.nchunks, counts);
    moe_scan_kernel<<<(n_local + 7) / 8, 256, 0, stream>>>(counts, totals, n_local, d.nchunks);
    // (launching these two with programmatic stream serialisation, each
    // waiting for the one before in griddepcontrol.wait, measured 2 us slower)
    const dim3 grid(static_cast<unsigned>(d.nchunks), static_cast<unsigned>(slices));
    moe_pack_quant_kernel<<<grid, kPackThreads, 0, stream>>>(
        static_cast<const uint16_t*>(x), T, KB, ldx, topk_ids, topk, expert_begin, n_local,
        counts, totals, d.nchunks, kb_per_slice, xq, sx, cap, offsets, token_ids);
    return launch_status();
}

// Fixed device scratch for fp8_moe_dispatch_quant_noalloc: the per-chunk
// counts and per-expert totals of one call (n_local * ceil(T / 64) + n_local
// ints, at most 65536 = 256 KB).  One copy per device; every call overwrites
// the entries it reads, so nothing needs to start at zero.
constexpr size_t kDispatchScratchInts = static_cast<size_t>(1) << 16;
static __device__ __align__(256) int32_t g_dispatch_scratch[kDispatchScratchInts];

// Device address of g_dispatch_scratch in the CUDA context current on this
// thread, or nullptr.  Host code cannot use the array's name as a device
// address; the runtime's cudaGetSymbolAddress gives it, for the module as
// loaded into the current context.  It is looked up once per (device,
// context) -- with that context current -- and cached together with the
// context's id, so a call made in another context of the same device (a
// driver-API context of the caller's, or the primary context re-created
// after cudaDeviceReset) looks it up again instead of reusing an address
// that is not valid there.
static int32_t* dispatch_scratch() {
    static ContextCache<int32_t*> cache;
    int32_t* ptr = nullptr;
    const int st = cache.get(&ptr, [](int32_t** v) {
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(v), g_dispatch_scratch) != cudaSuccess)
            return static_cast<int>(FP8_ERR_CUDA);
        return static_cast<int>(FP8_OK);
    });
    return st == FP8_OK ? ptr : nullptr;
}

}  // namespace fp8fg

using namespace fp8fg;

extern "C" fp8_status fp8_moe_dispatch_workspace_size(int64_t T, int32_t n_local, size_t* bytes) {
    if (bytes == nullptr) return FP8_ERR_NULL;
    *bytes = 0;
    if (T < 0 || n_local < 1 || n_local > kMaxLocal) return FP8_ERR_SHAPE;
    if (T > (static_cast<int64_t>(1) << 31) / kMaxTopk) return FP8_ERR_UNSUPPORTED;
    *bytes = T == 0 ? 0 : dispatch_plan(T, n_local).bytes;
    return FP8_OK;
}

extern "C" fp8_status fp8_moe_dispatch_quant(const void* x, int64_t T, int64_t K, int64_t ldx,
                                      const int32_t* topk_ids, int32_t topk,
                                      int32_t expert_begin, int32_t n_local, uint8_t* xq,
                                      float* sx, int64_t cap, int32_t* offsets,
                                      int32_t* token_ids, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    int st = dispatch_checks(T, K, ldx, topk, n_local, cap);
    if (st != FP8_OK) return to_status(st);
    if (offsets == nullptr) return FP8_ERR_NULL;
    if (!aligned(offsets, 4)) return FP8_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        // no tokens: every expert is empty
        if (cudaMemsetAsync(offsets, 0, (static_cast<size_t>(n_local) + 1) * sizeof(int32_t), s) !=
            cudaSuccess)
            return FP8_ERR_CUDA;
        return FP8_OK;
    }
    if (x == nullptr || topk_ids == nullptr || xq == nullptr || sx == nullptr ||
        token_ids == nullptr || workspace == nullptr)
        return FP8_ERR_NULL;
    if (ldx % 8 != 0 || !aligned(x, 16) || !aligned(xq, 16) || !aligned(sx, 4) ||
        !aligned(topk_ids, 4) || !aligned(token_ids, 4) || !aligned(workspace, 256))
        return FP8_ERR_ALIGN;
    if (workspace_bytes < dispatch_plan(T, n_local).bytes) return FP8_ERR_SHAPE;
    return to_status(dispatch_launch(x, T, K, ldx, topk_ids, topk, expert_begin, n_local, xq, sx, cap,
                           offsets, token_ids, static_cast<int32_t*>(workspace), s));
}

extern "C" fp8_status fp8_moe_dispatch_quant_noalloc(const void* x, int64_t T, int64_t K, int64_t ldx,
                                              const int32_t* topk_ids, int32_t topk,
                                              int32_t expert_begin, int32_t n_local, uint8_t* xq,
                                              float* sx, int64_t cap, int32_t* offsets,
                                              int32_t* token_ids, void* stream) {
    int st = dispatch_checks(T, K, ldx, topk, n_local, cap);
    if (st != FP8_OK) return to_status(st);
    if (offsets == nullptr) return FP8_ERR_NULL;
    if (!aligned(offsets, 4)) return FP8_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (cudaMemsetAsync(offsets, 0, (static_cast<size_t>(n_local) + 1) * sizeof(int32_t), s) !=
            cudaSuccess)
            return FP8_ERR_CUDA;
        return FP8_OK;
    }
    if (x == nullptr || topk_ids == nullptr || xq == nullptr || sx == nullptr ||
        token_ids == nullptr)
        return FP8_ERR_NULL;
    if (ldx % 8 != 0 || !aligned(x, 16) || !aligned(xq, 16) || !aligned(sx, 4) ||
        !aligned(topk_ids, 4) || !aligned(token_ids, 4))
        return FP8_ERR_ALIGN;
    // the problem must fit the fixed scratch
    const DispatchPlan d = dispatch_plan(T, n_local);
    if (d.count_ints + static_cast<size_t>(n_local) > kDispatchScratchInts)
        return FP8_ERR_UNSUPPORTED;
    int32_t* scratch = dispatch_scratch();
    if (scratch == nullptr) return FP8_ERR_CUDA;
    return to_status(dispatch_launch(x, T, K, ldx, topk_ids, topk, expert_begin, n_local, xq, sx, cap,
                           offsets, token_ids, scratch, s));
}
