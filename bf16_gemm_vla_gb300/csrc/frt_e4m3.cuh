// E4M3 encoding on the device, shared by the quantize kernels and the GEMM
// epilogue that quantizes its own output: round-to-nearest-even with
// saturation of an fp32 value, and the E4M3 byte of an IEEE fp32 quotient
// x / s computed through a reciprocal with a proven bracket.  Also the
// relaxed/acquire-release global accesses of the grid barriers that take a
// tensor's amax across CTAs.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace frt {
namespace {

// ------------------------------------------------------------------ E4M3 encode
//
// Round-to-nearest-even with saturation on the fp32 bit pattern.  For a
// magnitude a below the dialect's maximum:
//   a below the smallest normal 2^emin: the codes are spaced 2^(emin-3), so
//     the code is a * 2^(3-emin) rounded half-to-even (an exact power-of-two
//     scaling followed by an integer rounding; 8 lands on the smallest normal);
//   otherwise: keep 3 of the 23 mantissa bits, rounding half to even by
//     adding 0x7ffff plus the lowest kept bit (a carry steps into the next
//     binade), then re-bias the exponent from 127 to the dialect's bias.
// NaN -> the NaN code; a >= max (inf included) -> +-max; a negative value
// that rounds to zero keeps its sign in OCP (0x80) and is 0x00 in FNUZ.
template <bool kFnuz>
__device__ __forceinline__ uint32_t encode_e4m3(float v) {
  constexpr int kBias = kFnuz ? 8 : 7;
  constexpr float kMax = kFnuz ? 240.0f : 448.0f;
  constexpr uint32_t kMaxCode = kFnuz ? 0x7Fu : 0x7Eu;
  constexpr uint32_t kNanCode = kFnuz ? 0x80u : 0x7Fu;
  constexpr float kMinNormal = kFnuz ? 0.0078125f : 0.015625f;  // 2^(1 - bias)
  constexpr float kSubScale = kFnuz ? 1024.0f : 512.0f;         // 2^(3 - (1 - bias))
  const uint32_t u = __float_as_uint(v);
  const uint32_t sign = (u >> 24) & 0x80u;
  const float a = fabsf(v);
  if (!(a == a)) return kNanCode;
  if (a >= kMax) return sign | kMaxCode;
  uint32_t mag;
  if (a < kMinNormal) {
    mag = static_cast<uint32_t>(__float2int_rn(a * kSubScale));
  } else {
    const uint32_t ua = __float_as_uint(a);
    const uint32_t r = (ua + 0x7FFFFu + ((ua >> 20) & 1u)) >> 20;
    mag = r - static_cast<uint32_t>((127 - kBias) << 3);
  }
  if (kFnuz && mag == 0u) return 0u;
  return sign | mag;
}

// OCP E4M3 byte of a value by the hardware conversion (round to nearest
// even, saturating to +-448).  Used only for finite values in the E4M3
// normal range, where it agrees with encode_e4m3<false>.
__device__ __forceinline__ uint32_t cvt_e4m3_ocp(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// E4M3 byte of the IEEE fp32 quotient x / s.
//
// Fast path: q = x * r with r = RN(1/s).  q and RN(x/s) both lie within a
// relative 2^-23 of x / s (two and one roundings of at most 2^-24), so they
// are at most 6 fp32 steps apart (a step halves just below a power of two).
// E4M3 rounding is monotone and only changes at midpoints between codes,
// which in the E4M3 normal range are the fp32 values whose low 20 mantissa
// bits are 0x80000.  When q is finite, in the normal range, and at least 9
// steps from such a midpoint, q and RN(x/s) therefore encode to the same
// byte and q is encoded.  Every other element takes the IEEE division.
// `fast_ok` (uniform) says r is a positive normal number.
template <bool kFnuz>
__device__ __forceinline__ uint32_t quantize_one(float x, float s, float r, bool fast_ok) {
  constexpr uint32_t kMinNormalBits = kFnuz ? 0x3C000000u : 0x3C800000u;  // 2^-7 / 2^-6
  if (fast_ok) {
    const float q = x * r;
    const uint32_t u = __float_as_uint(q) & 0x7FFFFFFFu;
    const uint32_t m = u & 0xFFFFFu;
    const uint32_t d = m >= 0x80000u ? m - 0x80000u : 0x80000u - m;
    if (u >= kMinNormalBits && u < 0x7F800000u && d > 8u) {
      if constexpr (kFnuz)
        return encode_e4m3<true>(q);
      else
        return cvt_e4m3_ocp(q);
    }
  }
  return encode_e4m3<kFnuz>(__fdiv_rn(x, s));
}

// OCP E4M3 bytes of the IEEE fp32 quotients a / s and b / s (a in the low
// byte).  Fast path: with y = v * r (r = RN(1/s)), RN(v / s) lies within a
// relative 1.5 * 2^-23 of y, so inside [y (1 - 2^-20), y (1 + 2^-20)] even
// after the bracket's own rounding.  E4M3 rounding is monotone, so when
// both ends of the bracket encode to the same byte, so does RN(v / s).  Two
// hardware conversions give the ends of both elements' brackets; elements
// whose bracket straddles a rounding midpoint take the IEEE division.
__device__ __forceinline__ uint32_t cvt_e4m3x2_ocp(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 lanes in one 64-bit register, and their lane-wise products (each
// lane an IEEE round-to-nearest multiply, as the scalar one).
__device__ __forceinline__ unsigned long long f32x2(float lo, float hi) {
  unsigned long long d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}

__device__ __forceinline__ unsigned long long mul_f32x2(unsigned long long a,
                                                        unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint32_t cvt_e4m3x2_ocp(unsigned long long v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return cvt_e4m3x2_ocp(lo, hi);
}

__device__ __forceinline__ uint32_t quantize_pair_ocp(float a, float b, float s, float r,
                                                      bool fast_ok) {
  if (fast_ok) {
    // the pair's products and both brackets on packed lanes
    const unsigned long long y = mul_f32x2(f32x2(a, b), f32x2(r, r));
    const float kDown = 1.0f - 0x1p-20f, kUp = 1.0f + 0x1p-20f;
    const uint32_t c0 = cvt_e4m3x2_ocp(mul_f32x2(y, f32x2(kDown, kDown)));
    const uint32_t c1 = cvt_e4m3x2_ocp(mul_f32x2(y, f32x2(kUp, kUp)));
    if (c0 == c1) return c0;
    uint32_t out = 0;
    out |= ((c0 ^ c1) & 0x00FFu) ? encode_e4m3<false>(__fdiv_rn(a, s)) : (c0 & 0x00FFu);
    out |= ((c0 ^ c1) & 0xFF00u) ? encode_e4m3<false>(__fdiv_rn(b, s)) << 8 : (c0 & 0xFF00u);
    return out;
  }
  return encode_e4m3<false>(__fdiv_rn(a, s)) | (encode_e4m3<false>(__fdiv_rn(b, s)) << 8);
}


// NaN bytes (S.1111.111) of four OCP codes -> the positive NaN 0x7f.
__device__ __forceinline__ uint32_t canonical_nan_x4(uint32_t w) {
  const uint32_t t = (w & 0x7F7F7F7Fu) + 0x01010101u;  // bit 7 set where low 7 bits are 0x7f
  return w & ~(t & 0x80808080u);
}

// The elements of a vector whose bracket straddles a rounding midpoint (or
// all of them when the reciprocal is not normal): bytes where the bracket
// ends' codes lo_d/lo_u (elements 0-3) and hi_d/hi_u (4-7) differ take the
// IEEE division.  Out of line: rare, and kept out of the hot loop's code.
__device__ __noinline__ uint2 encode8_ocp_slow(float f0, float f1, float f2, float f3, float f4,
                                               float f5, float f6, float f7, float s,
                                               uint32_t lo_d, uint32_t lo_u, uint32_t hi_d,
                                               uint32_t hi_u, bool all) {
  const float f[8] = {f0, f1, f2, f3, f4, f5, f6, f7};
  uint32_t w[2] = {lo_d, hi_d};
  const uint32_t x[2] = {lo_d ^ lo_u, hi_d ^ hi_u};
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (all || ((x[h] >> (8 * e)) & 0xFFu)) {
        const uint32_t c = encode_e4m3<false>(__fdiv_rn(f[4 * h + e], s));
        w[h] = (w[h] & ~(0xFFu << (8 * e))) | (c << (8 * e));
      }
  return make_uint2(canonical_nan_x4(w[0]), canonical_nan_x4(w[1]));
}

// OCP E4M3 bytes of the IEEE fp32 quotients f[e] / s of 8 elements (element
// e in byte e % 4 of word e / 4), by the bracket of quantize_pair_ocp with
// one test for the whole vector; NaN bytes canonical.
__device__ __forceinline__ uint2 encode8_ocp(const float (&f)[8], float s, float r,
                                             bool fast_ok) {
  if (fast_ok) {
    const unsigned long long rr = f32x2(r, r);
    const float kDown = 1.0f - 0x1p-20f, kUp = 1.0f + 0x1p-20f;
    const unsigned long long dn = f32x2(kDown, kDown), up = f32x2(kUp, kUp);
    uint32_t d[4], u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const unsigned long long y = mul_f32x2(f32x2(f[2 * k], f[2 * k + 1]), rr);
      d[k] = cvt_e4m3x2_ocp(mul_f32x2(y, dn));
      u[k] = cvt_e4m3x2_ocp(mul_f32x2(y, up));
    }
    const uint32_t lo_d = d[0] | (d[1] << 16), hi_d = d[2] | (d[3] << 16);
    const uint32_t lo_u = u[0] | (u[1] << 16), hi_u = u[2] | (u[3] << 16);
    if (((lo_d ^ lo_u) | (hi_d ^ hi_u)) == 0u)
      return make_uint2(canonical_nan_x4(lo_d), canonical_nan_x4(hi_d));
    return encode8_ocp_slow(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7], s, lo_d, lo_u, hi_d,
                            hi_u, false);
  }
  return encode8_ocp_slow(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7], s, 0u, 0u, 0u, 0u,
                          true);
}

__device__ __forceinline__ bool recip_is_normal(float s, float r) {
  const uint32_t e = __float_as_uint(r) >> 23;  // r > 0: the exponent field
  return s > 0.0f && e - 1u < 254u;
}

// ------------------------------------------------------------------ grid-barrier words

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_gpu_u64(unsigned* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

}  // namespace
}  // namespace frt
