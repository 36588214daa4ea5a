// quant_math.cuh -- the per-group arithmetic of the E4M3 quantisers, shared
// by every kernel that emits fine-grained codes (the quantisers and the MoE
// dispatch packer) so that all of them produce identical codes and scales.
//
// Group scale s = fl32(amax / 448) (s = 1 for amax = 0); code = E4M3 RNE
// saturating conversion of the correctly rounded quotient x / s
// (DeepSeek-V3 Technical Report, section 3.3.2, fine-grained quantization).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace fp8fg {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float group_scale(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

__device__ __forceinline__ uint64_t f2x2(float lo, float hi) {
    return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Division of every element of a group by its scale s, correctly rounded,
// from one reciprocal per group.  Markstein's correction (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): with r = RN(1/s) and
// q0 = RN(x r), the residual e = x - q0 s is exact under a fused
// multiply-add and RN(q0 + e r) is the correctly rounded quotient x / s.
// Two lanes at a time with the packed FP32 instructions.  The sign of a zero
// quotient is taken from x (s > 0).  The residual is exact only while it does
// not underflow, i.e. for |x| >= 2^-102; with s >= 2^-91 every smaller x has
// |x / s| < 2^-11 and encodes to a signed zero whatever the last bit of its
// quotient, so the corrected path is used for s >= 2^-91 and groups with a
// smaller scale take the IEEE division.  The tests compare the resulting
// codes with IEEE division over every (x, amax) bf16 pair.
//
// fast_min: the smallest scale for which the corrected path is used.  Below
// |x| = 2^-102 the residual may be inexact; the path is still right when
// every such x gives a quotient the target format rounds to zero whatever
// its last bit: |x / s| < 2^-11 for E4M3 (s >= 2^-91, the default), and
// |x / s| < 2^-22 for E5M6 (s >= 2^-80, kE5M6FastMin).
constexpr float kE5M6FastMin = 0x1p-80f;

struct GroupDiv {
    float s;
    uint64_t r2, ns2;
    bool fast;
    __device__ __forceinline__ explicit GroupDiv(float scale, float fast_min = 0x1p-91f)
        : s(scale) {
        const float r = __frcp_rn(scale);
        r2 = f2x2(r, r);
        ns2 = f2x2(-scale, -scale);
        fast = scale >= fast_min;
    }
    // From a scale and its reciprocal computed elsewhere (r = RN(1 / scale)).
    __device__ __forceinline__ GroupDiv(float scale, float r, float fast_min) : s(scale) {
        r2 = f2x2(r, r);
        ns2 = f2x2(-scale, -scale);
        fast = scale >= fast_min;
    }
    // Correctly rounded quotients x0 / s, x1 / s (a zero may carry either sign).
    __device__ __forceinline__ void quot2(float x0, float x1, float& q0, float& q1) const {
        if (fast) {
            const uint64_t x2 = f2x2(x0, x1);
            const uint64_t a = mul2(x2, r2);
            const uint64_t e = fma2(a, ns2, x2);
            const uint64_t q = fma2(e, r2, a);
            q0 = __uint_as_float(static_cast<uint32_t>(q));
            q1 = __uint_as_float(static_cast<uint32_t>(q >> 32));
        } else {
            q0 = __fdiv_rn(x0, s);
            q1 = __fdiv_rn(x1, s);
        }
    }
    // E4M3 codes of x0 / s and x1 / s, x0 in the low byte
    __device__ __forceinline__ uint32_t pair(float x0, float x1) const {
        float q0, q1;
        if (fast) {
            const uint64_t x2 = f2x2(x0, x1);
            const uint64_t a = mul2(x2, r2);
            const uint64_t e = fma2(a, ns2, x2);
            const uint64_t q = fma2(e, r2, a);
            q0 = copysignf(__uint_as_float(static_cast<uint32_t>(q)), x0);
            q1 = copysignf(__uint_as_float(static_cast<uint32_t>(q >> 32)), x1);
        } else {
            q0 = __fdiv_rn(x0, s);
            q1 = __fdiv_rn(x1, s);
        }
        return static_cast<uint32_t>(
            __nv_cvt_float2_to_fp8x2(make_float2(q0, q1), __NV_SATFINITE, __NV_E4M3));
    }
    // four codes packed little-endian
    __device__ __forceinline__ uint32_t quad(float a, float b, float c, float d) const {
        return pair(a, b) | (pair(c, d) << 16);
    }

    // As pair(), but a zero quotient may carry the wrong sign: the callers
    // below set every code's sign bit from its input instead, one permute
    // for four inputs (for a nonzero quotient that bit is already right).
    __device__ __forceinline__ uint32_t pair_unsigned(float x0, float x1) const {
        float q0, q1;
        if (fast) {
            const uint64_t x2 = f2x2(x0, x1);
            const uint64_t a = mul2(x2, r2);
            const uint64_t e = fma2(a, ns2, x2);
            const uint64_t q = fma2(e, r2, a);
            q0 = __uint_as_float(static_cast<uint32_t>(q));
            q1 = __uint_as_float(static_cast<uint32_t>(q >> 32));
        } else {
            q0 = __fdiv_rn(x0, s);
            q1 = __fdiv_rn(x1, s);
        }
        return static_cast<uint32_t>(
            __nv_cvt_float2_to_fp8x2(make_float2(q0, q1), __NV_SATFINITE, __NV_E4M3));
    }
    // Codes of the four bf16 values of words w0, w1 in memory order
    // (lo w0, hi w0, lo w1, hi w1), packed little-endian.
    __device__ __forceinline__ uint32_t quad_words(uint32_t w0, uint32_t w1) const {
        const uint32_t c = pair_unsigned(bf16_lo(w0), bf16_hi(w0)) |
                           (pair_unsigned(bf16_lo(w1), bf16_hi(w1)) << 16);
        return c | (sign_bytes(w0, w1) & 0x80808080u);
    }
  private:
    __device__ __forceinline__ static uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t sel) {
        uint32_t d;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
        return d;
    }
    // 0xFF or 0x00 per byte: the signs of (lo w0, hi w0, lo w1, hi w1), each
    // the top bit of a bf16's high byte (bytes 1, 3, 5, 7) replicated.
    __device__ __forceinline__ static uint32_t sign_bytes(uint32_t w0, uint32_t w1) {
        return byte_perm(w0, w1, 0xFDB9);
    }
};

// ------------------------------------------------ negated-quotient codes --
// The streaming quantisers compute codes of the negated quotient and flip
// the sign bits afterwards.  With r = RN(1/s) and nr = -r:
//   a = RN(x nr) = -RN(x r),  e = RN(x + a s) = x - RN(x r) s (exact, as in
//   Markstein's correction above),  RN(e nr + a) = -RN(x / s),
// so the same three operations give the negated correctly rounded quotient,
// and a zero x gives a zero of the opposite sign (+0 + -0 rounds to +0 at
// the last step).  The E4M3 conversion is odd (RNE and saturation treat both
// signs alike), so code(x / s) = code(-(x / s)) ^ 0x80 for every finite x,
// signed zeros included, with no per-element sign repair.  The slow path
// (scales below the fast-path threshold) divides by -s in IEEE arithmetic,
// which is the same negated quotient.
struct NegDiv {
    uint64_t nr2, s2;
    float ns;
    __device__ __forceinline__ NegDiv(float scale, float r)
        : nr2(f2x2(-r, -r)), s2(f2x2(scale, scale)), ns(-scale) {}
    // Codes of -(x0 / s), -(x1 / s) (x0 in the low half of x2) in the low
    // two bytes, x0's first.
    template <bool FAST>
    __device__ __forceinline__ uint32_t ncodes2(uint64_t x2) const {
        uint64_t q;
        if (FAST) {
            const uint64_t a = mul2(x2, nr2);
            const uint64_t e = fma2(a, s2, x2);
            q = fma2(e, nr2, a);
        } else {
            q = f2x2(__fdiv_rn(__uint_as_float(static_cast<uint32_t>(x2)), ns),
                     __fdiv_rn(__uint_as_float(static_cast<uint32_t>(x2 >> 32)), ns));
        }
        return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(
            make_float2(__uint_as_float(static_cast<uint32_t>(q)), __uint_as_float(static_cast<uint32_t>(q >> 32))),
            __NV_SATFINITE, __NV_E4M3));
    }
};
constexpr uint32_t kSignFlip4 = 0x80808080u;

// The two bf16 values of a word as a packed FP32 pair (low half first).
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) {
    return f2x2(bf16_lo(w), bf16_hi(w));
}
// The low (or high) halves of two words as a packed FP32 pair, w0's first.
__device__ __forceinline__ uint64_t bf16_lo2(uint32_t w0, uint32_t w1) {
    return f2x2(bf16_lo(w0), bf16_lo(w1));
}
__device__ __forceinline__ uint64_t bf16_hi2(uint32_t w0, uint32_t w1) {
    return f2x2(bf16_hi(w0), bf16_hi(w1));
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Codes of 16 consecutive elements (eight words, memory order) of a group,
// sign bits flipped back, as one 16-byte store.
template <bool FAST>
__device__ __forceinline__ uint4 codes_1x128(const NegDiv& dv, const uint4& a, const uint4& b) {
    auto quad = [&](uint32_t w0, uint32_t w1) {
        return prmt(dv.ncodes2<FAST>(bf16x2_to_f2(w0)), dv.ncodes2<FAST>(bf16x2_to_f2(w1)), 0x5410u) ^
               kSignFlip4;
    };
    return make_uint4(quad(a.x, a.y), quad(a.z, a.w), quad(b.x, b.y), quad(b.z, b.w));
}

// ---------------------------------------------------- power-of-two scales --
// The smallest e with amax <= 448 * 2^e, clamped to the UE8M0 range
// [-127, 127]; e = 0 for amax = 0.  amax is a bfloat16 value (1 + m/128) 2^E:
// 448 = 1.75 * 2^8, so e = E - 8 when m <= 96 (mantissa <= 1.75) and E - 7
// otherwise; bfloat16 subnormals (and everything below 448 * 2^-128) clamp.
__device__ __forceinline__ int pow2_exponent(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int ef = static_cast<int>((b >> 23) & 0xFF);
    if (b == 0) return 0;
    if (ef == 0) return -127;
    const int e = ef - 127 - 8 + (((b >> 16) & 0x7F) > 96 ? 1 : 0);
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}
// 2^-e as a binary32 (e in [-127, 127]: 2^127 down to the subnormal 2^-127)
__device__ __forceinline__ float pow2_inverse(int e) {
    return e >= 127 ? 0x1p-127f : __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}
// E4M3 codes of x0 * r, x1 * r (r a power of two: the products are exact
// wherever the code can be nonzero), x0 in the low byte.
__device__ __forceinline__ uint32_t e4m3_scaled_pair(float x0, float x1, float r) {
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(x0 * r, x1 * r), __NV_SATFINITE, __NV_E4M3));
}

// ------------------------------------------------------------------ E5M6 --
// E5M6 (sign, 5-bit exponent with bias 15, 6-bit mantissa; exponent field 31
// reserved; largest finite 65024 = 0x7BF; subnormals m * 2^-20): the 12-bit
// code of a binary32 magnitude |q| with the given sign bit, rounded to nearest
// with ties to the even mantissa and saturated at 65024.
__device__ __forceinline__ uint32_t e5m6_code(float q, uint32_t neg) {
    const uint32_t a = __float_as_uint(q) & 0x7FFFFFFFu;
    uint32_t mag;
    if (a >= 0x477E0000u) {            // |q| >= 65024 (or infinite): saturate
        mag = 0x7BFu;
    } else if (a < 0x38800000u) {      // |q| < 2^-14: the grid m * 2^-20, m = 0..64
        // scaling by 2^20 is exact; m = 64 is 2^-14, whose code is 64 as well
        mag = __float2uint_rn(__uint_as_float(a) * 1048576.0f);
    } else {                           // keep 6 of the 23 mantissa bits, RNE
        const uint32_t r = a + 0xFFFFu + ((a >> 17) & 1u);
        mag = (r >> 17) - ((127u - 15u) << 6);
    }
    return (neg << 11) | mag;
}

// Eight 12-bit codes packed into three words, element i at bits 12 i .. 12 i + 11.
__device__ __forceinline__ void pack_e5m6_8(const uint32_t (&c)[8], uint32_t& w0, uint32_t& w1,
                                            uint32_t& w2) {
    w0 = c[0] | (c[1] << 12) | (c[2] << 24);
    w1 = (c[2] >> 8) | (c[3] << 4) | (c[4] << 16) | (c[5] << 28);
    w2 = (c[5] >> 4) | (c[6] << 8) | (c[7] << 20);
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}

// Largest magnitude in a word of two bf16 values, as a packed bf16 pair
// (exact: max and abs of bf16 values do not round).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
    const __nv_bfloat162 r = __hmax2(__habs2(*reinterpret_cast<const __nv_bfloat162*>(&a)),
                                     __habs2(*reinterpret_cast<const __nv_bfloat162*>(&b)));
    return *reinterpret_cast<const uint32_t*>(&r);
}
// Running maximum of magnitudes over words of bf16 pairs, one instruction a
// word: max.xorsign.abs gives max(|a|, |b|) per half with the XOR of the
// signs, so the magnitudes are exact and the sign bits meaningless until
// masked with 0x7FFF7FFF.
__device__ __forceinline__ uint32_t absmax_acc(uint32_t acc, uint32_t w) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(acc), "r"(w));
    return d;
}
__device__ __forceinline__ float amax_of_pair(uint32_t w) {
    return fmaxf(bf16_lo(w), bf16_hi(w));  // both halves already non-negative
}

}  // namespace fp8fg
