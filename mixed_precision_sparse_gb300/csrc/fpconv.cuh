// fpconv.cuh -- format conversions and error-free FP32 arithmetic on the integer and FP32
// pipes.
//
// On GB300 the FP64 unit issues about two operations per clock per SM, and the
// hardware FP64<->FP32 conversions run on that same unit. These helpers do the
// conversions the hot path needs with integer instructions instead, so that the only
// FP64 instructions left are the method's own FP64 arithmetic.
#pragma once
#include <cstdint>

namespace evocg {

// Round an FP64 value to a binary format with F fraction bits, an 8-bit exponent and
// bias 127 (F = 23: FP32, F = 7: BF16), to nearest with ties to even, in one rounding.
// Returns the target's bit pattern in the low 9 + F bits. Infinities map to infinities,
// NaN to a quiet NaN of the same sign, magnitudes past the largest finite value to
// infinity, FP64 subnormals to zero, and small values to the target's subnormals.
template <int F>
__host__ __device__ __forceinline__ uint32_t rne_bits_from_f64(uint64_t u)
{
    const uint32_t sign = (uint32_t)(u >> 63) << (F + 8);
    const uint64_t a = u & 0x7FFFFFFFFFFFFFFFull;
    const uint32_t kInf = 0xFFu << F;
    if (a >= 0x7FF0000000000000ull)
        return sign | (a == 0x7FF0000000000000ull ? kInf : (kInf | (1u << (F - 1))));
    const int ef = (int)(a >> 52);
    if (ef == 0) return sign;                         // zero or FP64 subnormal
    const int e = ef - 1023;
    const uint64_t sig = (a & 0x000FFFFFFFFFFFFFull) | 0x0010000000000000ull;
    int shift;
    uint32_t ebits;
    if (e >= -126) { shift = 52 - F; ebits = (uint32_t)(e + 127); }
    else { shift = 52 - F + (-126 - e); ebits = 0; }  // target subnormal: quantum 2^(-126-F)
    if (shift > 63) return sign;
    uint64_t q = sig >> shift;
    const uint64_t rem = sig & ((1ull << shift) - 1ull);
    const uint64_t half = 1ull << (shift - 1);
    q += (rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull;
    uint32_t out;
    if (ebits == 0) {
        out = (uint32_t)q;                            // may carry into the first normal
    } else {
        if (ebits >= 255u) return sign | kInf;
        out = (ebits << F) + (uint32_t)(q - (1ull << F));  // a carry bumps the exponent
        if (out >= kInf) out = kInf;
    }
    return sign | out;
}

// Exact FP32 -> FP64 conversion from the bit pattern.
__host__ __device__ __forceinline__ uint64_t f64_bits_from_f32(uint32_t u)
{
    const uint64_t sign = (uint64_t)(u >> 31) << 63;
    uint32_t a = u & 0x7FFFFFFFu;
    if (a == 0) return sign;
    if (a >= 0x7F800000u) {
        const uint64_t m = (uint64_t)(a & 0x7FFFFFu) << 29;
        return sign | 0x7FF0000000000000ull | m | (m ? 0x0008000000000000ull : 0ull);
    }
    int e = (int)(a >> 23);
    uint32_t m = a & 0x7FFFFFu;
    if (e == 0) {  // FP32 subnormal: normalise
        int lead = 31;
        while (!(m >> lead)) --lead;  // position of the leading one, 0..22
        e = 1 - (23 - lead);
        m = (m << (23 - lead)) & 0x7FFFFFu;
    }
    return sign | ((uint64_t)(e - 127 + 1023) << 52) | ((uint64_t)m << 29);
}

#ifdef __CUDACC__
// |x|'s high word from x's, by a 32-bit AND the compiler keeps as one (a 64-bit mask of the
// sign bit would be taken for an FP64 absolute value and run on the FP64 unit).
__device__ __forceinline__ uint32_t abs_hi(uint32_t hi)
{
    uint32_t r;
    asm("and.b32 %0, %1, 0x7fffffff;" : "=r"(r) : "r"(hi));
    return r;
}

// The same rounding as rne_bits_from_f64, with a short path for results in the target's
// normal range (FP64 exponents 897 .. 1150): the exponent and the top F fraction bits, rounded
// to nearest even on the dropped bits (a carry moves into the exponent), rebiased from 1023
// to 127. Zero, subnormal results, overflow, infinities and NaN take the general path.
template <int F>
__device__ __forceinline__ uint32_t rne_bits_dev(uint64_t u)
{
    const uint32_t hi = (uint32_t)(u >> 32), ahi = abs_hi(hi);
    if ((ahi >> 20) - 897u <= 253u) {
        constexpr int sh = 52 - F;
        const uint64_t a = ((uint64_t)ahi << 32) | (uint32_t)u;
        uint64_t q = a >> sh;
        const uint64_t rem = a & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
        q += (rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull;
        return ((hi >> 31) << (F + 8)) | ((uint32_t)q - ((uint32_t)(1023 - 127) << F));
    }
    return rne_bits_from_f64<F>(u);
}

__device__ __forceinline__ float f32_from_f64_rn(double x)
{
    return __uint_as_float(rne_bits_dev<23>((uint64_t)__double_as_longlong(x)));
}
__device__ __forceinline__ uint16_t bf16_from_f64_rn(double x)
{
    return (uint16_t)rne_bits_dev<7>((uint64_t)__double_as_longlong(x));
}
__device__ __forceinline__ double f64_from_f32(float f)
{
    return __longlong_as_double((long long)f64_bits_from_f32(__float_as_uint(f)));
}
__device__ __forceinline__ float f32_from_bf16(uint16_t h)
{
    return __uint_as_float((uint32_t)h << 16);
}
// 2^e as FP32 for e in [-126, 127].
__device__ __forceinline__ float pow2f(int e)
{
    return __uint_as_float((uint32_t)(e + 127) << 23);
}

// Error-free sum (Knuth's TwoSum): s + err == a + b exactly, s = fl(a + b).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &err)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Unevaluated FP32 pair accumulator: hi + lo holds a running sum to about 48 bits.
struct F32Pair {
    float hi = 0.f, lo = 0.f;
    __device__ __forceinline__ void add(float t)
    {
        float s, e;
        two_sum(hi, t, s, e);
        hi = s;
        lo = __fadd_rn(lo, e);
    }
    // add the exact product a*b (TwoProduct with one fused multiply-add)
    __device__ __forceinline__ void add_prod(float a, float b)
    {
        const float p = __fmul_rn(a, b);
        const float e = __fmaf_rn(a, b, -p);
        add(p);
        lo = __fadd_rn(lo, e);
    }
    __device__ __forceinline__ void merge(const F32Pair &o)
    {
        float s, e;
        two_sum(hi, o.hi, s, e);
        hi = s;
        lo = __fadd_rn(__fadd_rn(lo, o.lo), e);
    }
};
#endif

}  // namespace evocg
