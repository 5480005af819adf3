// Bandwidth kernels: FNUZ -> OCP E4M3 re-encoding and E4M3 quantization.
//
// Both dialects put sign, 4 exponent bits and 3 mantissa bits in the same
// places; FNUZ's exponent bias is one larger, so a byte means half its OCP
// value, FNUZ has no -0 and its only NaN is 0x80 ("Real-time VLA inference
// on AMD hardware", "Different FP8 representation"; "Deploying
// DeepSeek-V4-Flash on AMD MI300X", "The FP8 dialect problem").
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "frt_device.cuh"
#include "frt_e4m3.cuh"
#include "frt_host.h"

namespace frt {
namespace {

// ------------------------------------------------------------------ FNUZ -> OCP
//
// Four bytes at a time in a 32-bit word (SIMD within a register).  Per byte,
// with magnitude g = b & 0x7f:
//   g >= 0x10 (exponent field >= 2): exponent field - 1, i.e. g - 8;
//   g <  0x10: value v * 2^-10 with v = g, on the OCP subnormal grid at v / 2:
//              (v >> 1) + ((v & 1) & ((v >> 1) & 1))  (round half to even);
//   sign kept (a negative tie to zero becomes 0x80); 0x80 (NaN) -> 0x7f.
// No byte's arithmetic carries into its neighbour: every intermediate below
// stays inside its byte lane.
__device__ __forceinline__ uint32_t fnuz_to_ocp_x4(uint32_t x) {
  const uint32_t sign = x & 0x80808080u;
  const uint32_t g = x & 0x7F7F7F7Fu;
  // high bit of each lane set where g >= 0x10 (g + 0x70 <= 0xef, no carry out)
  const uint32_t big_hi = (g + 0x70707070u) & 0x80808080u;
  const uint32_t big = (big_hi >> 7) * 0xFFu;  // 0xff lanes where g >= 0x10
  // g - 8 with a borrow guard bit in every lane
  const uint32_t dec = ((g | 0x80808080u) - 0x08080808u) & 0x7F7F7F7Fu;
  // small magnitudes: h = g >> 1 (3 bits), + 1 when g is odd and h is odd
  const uint32_t h = (g >> 1) & 0x07070707u;
  const uint32_t small = h + (g & h & 0x01010101u);
  uint32_t out = ((big & dec) | (~big & small)) | sign;
  // lanes that were exactly 0x80: g == 0 and sign set -> 0x7f
  const uint32_t zero_hi = ~(g + 0x7F7F7F7Fu) & 0x80808080u;
  const uint32_t nan_hi = zero_hi & sign;
  out ^= (nan_hi >> 7) * 0xFFu;  // 0x80 ^ 0xff = 0x7f
  return out;
}

__global__ void fnuz_to_ocp_vec_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                       size_t n16) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += stride) {
    uint4 v = in[i];
    v.x = fnuz_to_ocp_x4(v.x);
    v.y = fnuz_to_ocp_x4(v.y);
    v.z = fnuz_to_ocp_x4(v.z);
    v.w = fnuz_to_ocp_x4(v.w);
    out[i] = v;
  }
}

__global__ void fnuz_to_ocp_byte_kernel(const uint8_t* in, uint8_t* out, size_t n) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = static_cast<uint8_t>(fnuz_to_ocp_x4(in[i]) & 0xFFu);
}

// ------------------------------------------------------------------ quantize

constexpr int kQThreads = 256;
constexpr int kMaxPartials = 1024;  // per-tensor amax partials (one per block)
constexpr int kColRowsPerBlock = 64;

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// 8 consecutive elements of a row (16-byte aligned for bf16, 32 for fp32).
template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&f)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&f)[8]) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&f)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// 8 consecutive elements of a row as loaded (16 bytes of bf16, 32 of fp32),
// converted to fp32 after all of a thread's loads are in flight.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 v;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) {
    v = __ldg(reinterpret_cast<const uint4*>(p));
  }
  __device__ __forceinline__ void unpack(float (&f)[8]) const {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ void unpack(float (&f)[8]) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
};

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    v = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  }
  return v;  // valid in thread 0
}

// Offsets into a row-strided x of the flat vector indices a thread visits:
// i0, i0 + stride, i0 + 2 stride, ... (vector i = row i / vpr, vector i % vpr
// of the row).  The row and column are advanced by the fixed stride instead
// of divided out of each index (a 64-bit division per vector otherwise).
struct StridedWalk {
  int64_t vpr, ldx_v, dr, dc;  // vectors per row, row stride in vectors, stride split
  int64_t r, c;                // current row and vector within it
  __device__ StridedWalk(int64_t i0, int64_t stride, int64_t vpr_, int64_t ldx_v_)
      : vpr(vpr_), ldx_v(ldx_v_), dr(stride / vpr_), dc(stride % vpr_), r(i0 / vpr_),
        c(i0 % vpr_) {}
  __device__ int64_t offset() const { return r * ldx_v + c; }  // in vectors
  __device__ void next() {
    r += dr;
    c += dc;
    if (c >= vpr) {
      c -= vpr;
      ++r;
    }
  }
};

// Per-tensor pass 1: each block's max |x| (NaN ignored by fmaxf) -> partial[block].
// Vector path: VEC = 8 elements per load, kUnroll loads in flight per
// thread; scalar path: VEC = 1.
constexpr int kUnroll = 4;

template <typename T, int VEC>
__global__ void __launch_bounds__(kQThreads) amax_tensor_kernel(const T* __restrict__ x,
                                                               int64_t rows, int64_t cols,
                                                               int64_t ldx,
                                                               float* __restrict__ partial) {
  __shared__ float red[32];
  dev::grid_dependency_wait();  // x may come from the previous grid
  float m = 0.0f;
  const int64_t vpr = cols / VEC;  // vectors per row
  const int64_t total = rows * vpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const bool dense = ldx == cols;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  StridedWalk walk(first < total ? first : 0, stride, vpr > 0 ? vpr : 1, ldx / VEC);
  auto offset = [&](int64_t i) -> int64_t {  // element offset of vector i (walk at i)
    return dense ? i * VEC : walk.offset() * VEC;
  };
  for (int64_t i0 = first; i0 < total; i0 += kUnroll * stride) {
    if constexpr (VEC == 8) {
      float f[kUnroll][8];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = i0 + u * stride;
        if (i < total) {
          load8<T>(x + offset(i), f[u]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) f[u][e] = 0.0f;
        }
        if (!dense) walk.next();
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(f[u][e]));
    } else {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = i0 + u * stride;
        if (i < total) m = fmaxf(m, fabsf(to_f32<T>(x[offset(i)])));
        if (!dense) walk.next();
      }
    }
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) partial[blockIdx.x] = m;
  dev::grid_launch_dependents();  // the encode pass may start once every block is here
}

// Per-tensor pass 2: reduce the partials to amax, s = amax / max (1 if amax
// is 0) or the static scale, then q = E4M3(x / s).
template <typename T, int VEC, bool kFnuz>
__global__ void __launch_bounds__(kQThreads) encode_tensor_kernel(
    const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
    const float* __restrict__ partial, int npartial, const float* __restrict__ static_scale,
    uint8_t* __restrict__ q, float* __restrict__ scale_out) {
  __shared__ float red[32];
  __shared__ float s_sh;
  dev::grid_dependency_wait();  // the partials and x come from earlier grids
  const int64_t n_vec = rows * (cols / VEC);
  const int64_t n_threads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // a short pass lets the next grid (typically a GEMM fetching its weights)
  // start now; a long one triggers at its end so it does not compete
  const bool early = n_vec <= 2 * kUnroll * n_threads;
  if (early) dev::grid_launch_dependents();
  if (static_scale) {
    if (threadIdx.x == 0) s_sh = __ldg(static_scale);
  } else {
    float m = 0.0f;
    for (int i = threadIdx.x; i < npartial; i += blockDim.x) m = fmaxf(m, partial[i]);
    m = block_max(m, red);
    if (threadIdx.x == 0) s_sh = m == 0.0f ? 1.0f : __fdiv_rn(m, kFnuz ? 240.0f : 448.0f);
  }
  __syncthreads();
  const float s = s_sh;
  const float r = __frcp_rn(s);
  const bool fast_ok = recip_is_normal(s, r);
  if (blockIdx.x == 0 && threadIdx.x == 0 && scale_out) *scale_out = s;
  const int64_t vpr = cols / VEC;
  const int64_t total = rows * vpr;
  const int64_t stride = n_threads;
  const bool dense = ldx == cols;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  StridedWalk walk(first < total ? first : 0, stride, vpr > 0 ? vpr : 1, ldx / VEC);
  auto xoffset = [&](int64_t i) -> int64_t {  // element offset of vector i (walk at i)
    return dense ? i * VEC : walk.offset() * VEC;
  };
  if constexpr (VEC == 8) {
    // U loads of 8 elements in flight per thread (raw), then the encodes
    constexpr int U = sizeof(T) == 2 ? 6 : 4;
    auto body = [&](int64_t i0) {
      Raw8<T> v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + u * stride;
        if (i < total) v[u].load(x + xoffset(i));
        if (!dense) walk.next();
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + u * stride;
        if (i >= total) break;
        float f[8];
        v[u].unpack(f);
        uint2 w;
        if constexpr (kFnuz) {
          w = make_uint2(0u, 0u);
#pragma unroll
          for (int e = 0; e < 4; ++e) w.x |= quantize_one<true>(f[e], s, r, fast_ok) << (8 * e);
#pragma unroll
          for (int e = 0; e < 4; ++e) w.y |= quantize_one<true>(f[4 + e], s, r, fast_ok) << (8 * e);
        } else {
          w = encode8_ocp(f, s, r, fast_ok);
        }
        // q is dense: element (r, c) at r * cols + c = i * VEC
        *reinterpret_cast<uint2*>(q + i * VEC) = w;
      }
    };
    const int64_t span = U * stride;
    if (dense && !static_scale) {
      // the amax pass read x in the same grid-stride order: its last reads
      // are the ones still in L2, so this pass takes its spans last first
      for (int64_t j = first < total ? (total - first - 1) / span : -1; j >= 0; --j)
        body(first + j * span);
    } else {
      for (int64_t i0 = first; i0 < total; i0 += span) body(i0);
    }
  } else {
    for (int64_t i0 = first; i0 < total; i0 += kUnroll * stride) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = i0 + u * stride;
        if (i < total)
          q[i] = static_cast<uint8_t>(quantize_one<kFnuz>(to_f32<T>(x[xoffset(i)]), s, r, fast_ok));
        if (!dense) walk.next();
      }
    }
  }
  if (!early) dev::grid_launch_dependents();
}

// Per-tensor quantize in one grid, with the tensor resident on chip.
//
// Every CTA (all resident at once, at most one per SM) holds its part of x
// on chip -- in registers for tensors up to kRegCapacity 16-byte vectors,
// else in shared memory, bulk-copied as contiguous chunks -- and takes the
// max |x| of it as it arrives.  The CTAs then meet at a grid barrier in the
// workspace header, where the last to arrive turns the maximum into
// s = amax / max (1 if amax is 0); finally every CTA encodes its part from
// chip.  x is read from memory once.
//
// The barrier: each CTA reads the generation (after the previous grid has
// completed), folds its maximum into this call's running-maximum word (an
// integer atomic max on the fp32 bits, which orders non-negative floats as
// their values; the two words alternate between calls by the generation's
// parity) and arrives on the arrival count (acquire-release, so the count's
// read-modify-writes carry every CTA's maximum).  A CTA that sees the count
// complete (acquire) reads the maximum itself and turns it into s = amax /
// max (1 if amax is 0).  The last arrival does the same, then clears the
// other parity's maximum and the count for the next call and publishes the
// next generation together with s in one 64-bit store, which a CTA that
// missed the complete count (already cleared) takes s from.
// Waits are bounded; a CTA that gives up records a code in the header's
// status word and uses s = NaN, so the result is visibly invalid.
constexpr int kResThreads = 1024;   // shared-memory path
constexpr int kRegThreads = 512;    // register path
constexpr int kResChunk = 16384;    // bytes per bulk copy
constexpr int kResMaxChunks = 13;   // at most 208 KiB of a tensor per CTA
constexpr int kResSmem = kResChunk * kResMaxChunks;
constexpr int kRegVecs = 3;         // register path: 16-byte vectors per thread
constexpr int kHeaderFloats = 64;   // workspace header: 256 bytes
// header words: [0] arrivals, [1] status, [2] generation and [3] scale bits
// (one 64-bit word), [4] and [5] running max |x| (fp32 bits) of the calls
// with an even and an odd generation

template <typename T>
__device__ __forceinline__ int unpack16(const uint4& w, float (&f)[8]) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(ws[k] << 16);
      f[2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
    }
    return 8;
  } else {
    f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
    return 4;
  }
}

// E4M3 bytes of one 16-byte vector of x at q + e (8 or 4 elements).
template <typename T, bool kFnuz>
__device__ __forceinline__ void encode16(const uint4& w, float sc, float r, bool fast_ok,
                                         uint8_t* dst) {
  float f[8];
  unpack16<T>(w, f);
  uint32_t lo = 0, hi = 0;
  if constexpr (kFnuz) {
#pragma unroll
    for (int k = 0; k < 4; ++k) lo |= quantize_one<true>(f[k], sc, r, fast_ok) << (8 * k);
    if constexpr (sizeof(T) == 2) {
#pragma unroll
      for (int k = 0; k < 4; ++k) hi |= quantize_one<true>(f[4 + k], sc, r, fast_ok) << (8 * k);
    }
  } else if constexpr (sizeof(T) == 2) {
    const uint2 w2 = encode8_ocp(f, sc, r, fast_ok);
    lo = w2.x;
    hi = w2.y;
  } else {
    lo = canonical_nan_x4(quantize_pair_ocp(f[0], f[1], sc, r, fast_ok) |
                          (quantize_pair_ocp(f[2], f[3], sc, r, fast_ok) << 16));
  }
  if constexpr (sizeof(T) == 2)
    *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
  else
    *reinterpret_cast<uint32_t*>(dst) = lo;
}

template <typename T>
__device__ __forceinline__ float max16(const uint4& w, float m) {
  float f[8];
  const int ne = unpack16<T>(w, f);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (k < ne) m = fmaxf(m, fabsf(f[k]));
  return m;
}

// bf16: running max |x| over a 16-byte vector on packed bf16 pairs (sign
// bits cleared; __hmax2 returns the other operand for a NaN, as fmaxf).
// The maximum is exact, so the result equals the fp32 path's.
__device__ __forceinline__ uint32_t max_abs_bf16x8(uint32_t acc, const uint4& w) {
  __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&acc);
  const uint32_t ws[4] = {w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu, w.z & 0x7FFF7FFFu,
                          w.w & 0x7FFF7FFFu};
#pragma unroll
  for (int k = 0; k < 4; ++k) a = __hmax2(a, *reinterpret_cast<const __nv_bfloat162*>(&ws[k]));
  return *reinterpret_cast<const uint32_t*>(&a);
}

__device__ __forceinline__ float bf16x2_max_to_float(uint32_t acc) {
  return fmaxf(__uint_as_float(acc << 16), __uint_as_float(acc & 0xFFFF0000u));
}

// The grid barrier above.  m: this CTA's max |x| (valid in thread 0); g0:
// the generation read by thread 0 after the dependency wait; red: the block
// reduction buffer.  Returns s (or NaN if this CTA gave up) in every thread.
template <bool kFnuz>
__device__ __forceinline__ float grid_scale(float m, unsigned g0, unsigned* hdr, bool failed) {
  __shared__ float s_sh;
  if (threadIdx.x == 0) {
    bool fail = failed;
    float sc;
    auto scale_of = [](unsigned amax_bits) {
      const float a = __uint_as_float(amax_bits);
      return a == 0.0f ? 1.0f : __fdiv_rn(a, kFnuz ? 240.0f : 448.0f);
    };
    unsigned* run_max = hdr + 4 + (g0 & 1u);  // this call's; cleared by the previous one
    // m >= 0 and never NaN (fmaxf from 0): its bits order as its value.  The
    // max is ordered before the arrival by the arrival's release.
    atomicMax(run_max, __float_as_uint(m));
    const unsigned grid = gridDim.x;
    if (atom_add_acq_rel_gpu(hdr, 1u) == grid - 1) {
      // every other CTA's max was released before its arrival, and this
      // arrival's acquire orders the load after them
      sc = scale_of(ld_relaxed_gpu(run_max));
      // the resets reach memory before the next grid starts (grid
      // completion); a waiter that reads the cleared count takes s from
      // the published word instead
      hdr[4 + ((g0 + 1u) & 1u)] = 0u;
      hdr[0] = 0u;
      st_relaxed_gpu_u64(hdr + 2, static_cast<unsigned long long>(g0 + 1u) |
                                      (static_cast<unsigned long long>(__float_as_uint(sc)) << 32));
    } else {
      const uint64_t t0 = dev::globaltimer_ns();
      for (uint32_t it = 0;; ++it) {
        // the complete count (its acquire reads the last of the arrivals'
        // read-modify-writes, after which every max is visible) ...
        if (ld_acquire_gpu(hdr) == grid) {
          sc = scale_of(ld_relaxed_gpu(run_max));
          break;
        }
        // ... or, once the last arrival has cleared it, the published s
        // (looked at every fourth poll: the count is the usual signal)
        if ((it & 3u) == 3u) {
          const unsigned long long w = ld_relaxed_gpu_u64(hdr + 2);
          if (static_cast<unsigned>(w) != g0) {
            sc = __uint_as_float(static_cast<unsigned>(w >> 32));
            break;
          }
        }
        if ((it & 15u) == 15u && dev::globaltimer_ns() - t0 > dev::kWaitLimitNs) {
          fail = true;
          break;
        }
      }
    }
    if (fail) {
      sc = __uint_as_float(0x7FC00000u);
      atomicCAS(hdr + 1, 0u, 0x201u);
    }
    s_sh = sc;
  }
  __syncthreads();
  return s_sh;
}

// Register path: thread t of CTA b holds vectors t + 512 (b + G j), j < kRegVecs.
// A CTA takes at most 512 x 48 registers and no shared memory, so a GEMM CTA
// (the usual next grid) fits beside it: the next grid is let go at once,
// and its prologue and weight prefetch overlap this grid.
//
// With a static scale (calibrated, frozen) there is no amax and no barrier:
// each CTA encodes its part as soon as it holds it, and no header is used.
template <typename T, bool kFnuz>
__global__ void __maxnreg__(48) quantize_regs_kernel(
    const T* __restrict__ x, int64_t n_vec, uint8_t* __restrict__ q, float* __restrict__ scale_out,
    unsigned* __restrict__ hdr, const float* __restrict__ static_scale) {
  constexpr int VEC = 16 / sizeof(T);
  __shared__ float red[32];
  dev::grid_launch_dependents();
  dev::grid_dependency_wait();  // x (and a static scale) may come from the previous grid
  // (the previous grid is complete: its header words are visible)
  const unsigned g0 = (!static_scale && threadIdx.x == 0) ? ld_relaxed_gpu(hdr + 2) : 0u;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kRegThreads;
  const int64_t v0 = static_cast<int64_t>(blockIdx.x) * kRegThreads + threadIdx.x;
  uint4 w[kRegVecs];
#pragma unroll
  for (int j = 0; j < kRegVecs; ++j)
    w[j] = v0 + j * stride < n_vec ? __ldcs(xv + v0 + j * stride) : make_uint4(0, 0, 0, 0);
  float sc;
  if (static_scale) {
    sc = __ldg(static_scale);
  } else {
    float m = 0.0f;
    if constexpr (sizeof(T) == 2) {
      uint32_t m2 = 0u;
#pragma unroll
      for (int j = 0; j < kRegVecs; ++j) m2 = max_abs_bf16x8(m2, w[j]);
      m = bf16x2_max_to_float(m2);
    } else {
#pragma unroll
      for (int j = 0; j < kRegVecs; ++j) m = max16<T>(w[j], m);
    }
    m = block_max(m, red);
    sc = grid_scale<kFnuz>(m, g0, hdr, false);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && scale_out) *scale_out = sc;
  const float r = __frcp_rn(sc);
  const bool fast_ok = recip_is_normal(sc, r);
#pragma unroll
  for (int j = 0; j < kRegVecs; ++j)
    if (v0 + j * stride < n_vec) encode16<T, kFnuz>(w[j], sc, r, fast_ok, q + (v0 + j * stride) * VEC);
}

// Shared-memory path: CTA b holds the contiguous elements [b per_cta, +per_cta).
// With a static scale there is no amax and no barrier (and no header): each
// chunk is encoded as soon as its copy lands, so the slice streams through
// shared memory.
template <typename T, bool kFnuz>
__global__ void __launch_bounds__(kResThreads, 1) quantize_resident_kernel(
    const T* __restrict__ x, int64_t n, int64_t per_cta, uint8_t* __restrict__ q,
    float* __restrict__ scale_out, unsigned* __restrict__ hdr,
    const float* __restrict__ static_scale) {
  constexpr int VEC = 16 / sizeof(T);
  extern __shared__ __align__(128) uint8_t res[];
  __shared__ uint64_t bars[kResMaxChunks];
  __shared__ float red[32];
  const int tid = threadIdx.x;
  const int64_t e0 = static_cast<int64_t>(blockIdx.x) * per_cta;
  const int64_t e1 = e0 + per_cta < n ? e0 + per_cta : n;
  const uint32_t bytes = static_cast<uint32_t>((e1 > e0 ? e1 - e0 : 0) * sizeof(T));
  const int nchunks = static_cast<int>((bytes + kResChunk - 1) / kResChunk);
  const uint32_t bar0 = dev::smem_u32(bars);
  if (tid == 0) {
    for (int i = 0; i < nchunks; ++i) dev::mbar_init(bar0 + 8 * i, 1);
    dev::fence_mbar_init();
  }
  __syncthreads();
  dev::grid_dependency_wait();  // x may come from the previous grid
  unsigned g0 = 0;
  if (tid == 0) {
    if (!static_scale) g0 = ld_relaxed_gpu(hdr + 2);  // the previous grid is complete
    const uint64_t pol = dev::policy_evict_first();
    const uint8_t* src = reinterpret_cast<const uint8_t*>(x + e0);
    for (int i = 0; i < nchunks; ++i) {
      const uint32_t sz = bytes - i * kResChunk < kResChunk ? bytes - i * kResChunk : kResChunk;
      dev::mbar_arrive_expect_tx(bar0 + 8 * i, sz);
      dev::bulk_load(dev::smem_u32(res + i * kResChunk), src + i * kResChunk, sz, bar0 + 8 * i,
                     pol);
    }
  }
  if (static_scale) {
    const float sc = __ldg(static_scale);
    if (blockIdx.x == 0 && tid == 0 && scale_out) *scale_out = sc;
    const float r = __frcp_rn(sc);
    const bool fast_ok = recip_is_normal(sc, r);
    // each chunk as soon as its copy lands (bounded; a copy that never
    // lands leaves NaN codes for its chunk, so the result is visibly invalid)
    for (int i = 0; i < nchunks; ++i) {
      const bool landed = dev::mbar_wait(bar0 + 8 * i, 0, nullptr, nullptr, 0);
      const uint32_t v0 = static_cast<uint32_t>(i) * (kResChunk / 16);
      const uint32_t v1 = min(bytes / 16, v0 + kResChunk / 16);
      if (landed) {
        for (uint32_t v = v0 + tid; v < v1; v += kResThreads)
          encode16<T, kFnuz>(*reinterpret_cast<const uint4*>(res + v * 16), sc, r, fast_ok,
                             q + e0 + static_cast<int64_t>(v) * VEC);
      } else {
        for (uint32_t b = v0 * VEC + tid; b < v1 * VEC; b += kResThreads)
          q[e0 + b] = kFnuz ? 0x80u : 0x7Fu;
      }
    }
    // (the next grid's CTAs cannot share the SM with this one's shared
    // memory anyway: let it go only now, so that it does not compete)
    dev::grid_launch_dependents();
    return;
  }
  // max |x| of the slice, chunk by chunk as the copies land (NaN is ignored
  // by fmaxf)
  float m = 0.0f;
  uint32_t m2 = 0u;  // bf16: packed running max
  bool ok = true;
  for (int i = 0; i < nchunks; ++i) {
    ok = dev::mbar_wait(bar0 + 8 * i, 0, nullptr, nullptr, 0) && ok;
    const uint32_t sz = bytes - i * kResChunk < kResChunk ? bytes - i * kResChunk : kResChunk;
    for (uint32_t v = tid; v < sz / 16; v += kResThreads) {
      const uint4 w = *reinterpret_cast<const uint4*>(res + i * kResChunk + v * 16);
      if constexpr (sizeof(T) == 2)
        m2 = max_abs_bf16x8(m2, w);
      else
        m = max16<T>(w, m);
    }
  }
  if constexpr (sizeof(T) == 2) m = bf16x2_max_to_float(m2);
  m = block_max(m, red);
  const bool failed = __syncthreads_or(!ok);
  const float sc = grid_scale<kFnuz>(m, g0, hdr, failed);
  dev::grid_launch_dependents();  // every CTA is past the barrier
  if (blockIdx.x == 0 && tid == 0 && scale_out) *scale_out = sc;
  const float r = __frcp_rn(sc);
  const bool fast_ok = recip_is_normal(sc, r);
  for (uint32_t v = tid; v < bytes / 16; v += kResThreads)
    encode16<T, kFnuz>(*reinterpret_cast<const uint4*>(res + v * 16), sc, r, fast_ok,
                       q + e0 + static_cast<int64_t>(v) * VEC);
}

// Per-column pass 1: block (bx, by) covers columns [bx*256, +256) and rows
// [by*kColRowsPerBlock, +kColRowsPerBlock); partial[by * cols + c] = max |x|.
template <typename T>
__global__ void __launch_bounds__(kQThreads) amax_col_kernel(const T* __restrict__ x,
                                                            int64_t rows, int64_t cols,
                                                            int64_t ldx,
                                                            float* __restrict__ partial) {
  dev::grid_dependency_wait();
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kColRowsPerBlock;
  const int64_t r1 = min(rows, r0 + kColRowsPerBlock);
  float m = 0.0f;
  for (int64_t r = r0; r < r1; ++r) m = fmaxf(m, fabsf(to_f32<T>(x[r * ldx + c])));
  partial[static_cast<int64_t>(blockIdx.y) * cols + c] = m;
}

// Per-column pass 2: s[c] from the partials of column c (or the static
// scales), then q = E4M3(x / s[c]) for this block's rows.
template <typename T, bool kFnuz>
__global__ void __launch_bounds__(kQThreads) encode_col_kernel(
    const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
    const float* __restrict__ partial, int npartial, const float* __restrict__ static_scale,
    uint8_t* __restrict__ q, float* __restrict__ scale_out) {
  dev::grid_dependency_wait();
  dev::grid_launch_dependents();
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  float s;
  if (static_scale) {
    s = __ldg(static_scale + c);
  } else {
    float m = 0.0f;
    for (int i = 0; i < npartial; ++i) m = fmaxf(m, partial[static_cast<int64_t>(i) * cols + c]);
    s = m == 0.0f ? 1.0f : __fdiv_rn(m, kFnuz ? 240.0f : 448.0f);
  }
  if (blockIdx.y == 0 && scale_out) scale_out[c] = s;
  const float rs = __frcp_rn(s);
  const bool fast_ok = recip_is_normal(s, rs);
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kColRowsPerBlock;
  const int64_t r1 = min(rows, r0 + kColRowsPerBlock);
  for (int64_t r = r0; r < r1; ++r)
    q[r * cols + c] =
        static_cast<uint8_t>(quantize_one<kFnuz>(to_f32<T>(x[r * ldx + c]), s, rs, fast_ok));
}

// Blocks for a grid-stride pass over total_vecs vectors, kUnroll per thread
// per iteration: at most `per_sm` blocks per SM and `limit` in total.
int tensor_grid(int64_t total_vecs, int per_sm, int limit) {
  const int64_t want = ceil_div(total_vecs, static_cast<int64_t>(kQThreads) * kUnroll);
  const int64_t cap = static_cast<int64_t>(sm_count() > 0 ? sm_count() : 148) * per_sm;
  int64_t g = want < cap ? want : cap;
  if (g > limit) g = limit;
  return static_cast<int>(g < 1 ? 1 : g);
}

// Blocks of a kQThreads-thread kernel (no dynamic shared memory) resident per
// SM, queried once per device.  The two-kernel path sizes its grids to one
// wave: a dependent grid's blocks, launched early and waiting, then never hold
// the SM slots that later blocks of this grid would need.
template <typename Kern>
int blocks_per_sm(Kern kern, int* cache) {
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 4;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kQThreads, 0) != cudaSuccess ||
        n < 1) {
      cudaGetLastError();
      n = 4;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

template <typename T, int VEC>
int amax_blocks_per_sm() {
  static int cache[64] = {0};
  return blocks_per_sm(amax_tensor_kernel<T, VEC>, cache);
}

template <typename T, int VEC, bool kFnuz>
int encode_blocks_per_sm() {
  static int cache[64] = {0};
  return blocks_per_sm(encode_tensor_kernel<T, VEC, kFnuz>, cache);
}

// Sets the resident kernel's dynamic shared memory limit once per device.
template <typename T, bool kFnuz>
bool resident_ready() {
  static std::mutex mu;
  static bool set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!set[dev]) {
    if (cudaFuncSetAttribute(quantize_resident_kernel<T, kFnuz>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kResSmem) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    set[dev] = true;
  }
  return true;
}

template <typename T, bool kFnuz>
frt_status quantize_typed(const T* x, int64_t rows, int64_t cols, int64_t ldx, frt_scale_mode mode,
                          const float* static_scale, uint8_t* q, float* scale, float* ws_all,
                          cudaStream_t st) {
  // the workspace starts with the header of the one-grid path; partials follow
  unsigned* hdr = reinterpret_cast<unsigned*>(ws_all);
  float* ws = ws_all ? ws_all + kHeaderFloats : nullptr;
  if (mode == FRT_SCALE_PER_TENSOR) {
    const bool vec = aligned(x, 16) && aligned(q, 8) && cols % 8 == 0 && ldx % 8 == 0;
    const int64_t n = rows * cols;
    const int sms = sm_count() > 0 ? sm_count() : 148;
    const int64_t n_vec16 = n * static_cast<int64_t>(sizeof(T)) / 16;
    // (a static scale needs no workspace: no amax, no barrier)
    const bool ws_ok = static_scale || aligned(ws_all, 16);
    if (vec && ldx == cols && ws_ok &&
        n_vec16 <= static_cast<int64_t>(sms) * kRegThreads * kRegVecs) {
      // one grid, the tensor in registers: at most one CTA per SM
      const int grid = static_cast<int>(
          std::min<int64_t>(sms, ceil_div(n_vec16, static_cast<int64_t>(kRegThreads))));
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(grid);
      cfg.blockDim = dim3(kRegThreads);
      cfg.stream = st;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, quantize_regs_kernel<T, kFnuz>, x, n_vec16, q, scale,
                             static_scale ? nullptr : hdr, static_scale) != cudaSuccess) {
        cudaGetLastError();
        return FRT_ERR_CUDA;
      }
      note_launches(1);
      return launch_status();
    }
    if (vec && ldx == cols && ws_ok &&
        n * static_cast<int64_t>(sizeof(T)) <= static_cast<int64_t>(sms) * kResSmem &&
        resident_ready<T, kFnuz>()) {
      // one grid, the tensor resident in shared memory: slices of a multiple
      // of 64 elements, at most one CTA per SM
      int64_t per = ceil_div(n, static_cast<int64_t>(sms));
      per = ceil_div(per, static_cast<int64_t>(64)) * 64;
      const int grid = static_cast<int>(ceil_div(n, per));
      const size_t smem = static_cast<size_t>(
          ceil_div(per * static_cast<int64_t>(sizeof(T)), static_cast<int64_t>(kResChunk)) *
          kResChunk);
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(grid);
      cfg.blockDim = dim3(kResThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = st;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, quantize_resident_kernel<T, kFnuz>, x, n, per, q, scale,
                             static_scale ? nullptr : hdr, static_scale) != cudaSuccess) {
        cudaGetLastError();
        return FRT_ERR_CUDA;
      }
      note_launches(1);
      return launch_status();
    }
    const int64_t total = rows * (vec ? cols / 8 : cols);
    // one wave each; amax: one partial per block
    const int grid = tensor_grid(
        total, vec ? amax_blocks_per_sm<T, 8>() : amax_blocks_per_sm<T, 1>(), kMaxPartials);
    const int egrid = tensor_grid(
        total, vec ? encode_blocks_per_sm<T, 8, kFnuz>() : encode_blocks_per_sm<T, 1, kFnuz>(),
        1 << 20);
    // programmatic launches: each kernel's blocks may be scheduled while the
    // previous grid drains, and wait for it before reading its output
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cudaLaunchConfig_t ecfg;
    cfg.blockDim = dim3(kQThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ecfg = cfg;
    ecfg.gridDim = dim3(egrid);
    cudaError_t e = cudaSuccess;
    if (vec) {
      if (!static_scale)
        e = cudaLaunchKernelEx(&cfg, amax_tensor_kernel<T, 8>, x, rows, cols, ldx, ws);
      if (e == cudaSuccess)
        e = cudaLaunchKernelEx(&ecfg, encode_tensor_kernel<T, 8, kFnuz>, x, rows, cols, ldx,
                               static_cast<const float*>(ws), grid, static_scale, q, scale);
    } else {
      if (!static_scale)
        e = cudaLaunchKernelEx(&cfg, amax_tensor_kernel<T, 1>, x, rows, cols, ldx, ws);
      if (e == cudaSuccess)
        e = cudaLaunchKernelEx(&ecfg, encode_tensor_kernel<T, 1, kFnuz>, x, rows, cols, ldx,
                               static_cast<const float*>(ws), grid, static_scale, q, scale);
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      return FRT_ERR_CUDA;
    }
    note_launches(static_scale ? 1 : 2);
  } else {
    const dim3 grid(static_cast<unsigned>(ceil_div(cols, kQThreads)),
                    static_cast<unsigned>(ceil_div(rows, kColRowsPerBlock)));
    if (!static_scale) amax_col_kernel<T><<<grid, kQThreads, 0, st>>>(x, rows, cols, ldx, ws);
    encode_col_kernel<T, kFnuz><<<grid, kQThreads, 0, st>>>(x, rows, cols, ldx, ws,
                                                             static_cast<int>(grid.y),
                                                             static_scale, q, scale);
    note_launches(static_scale ? 1 : 2);
  }
  return launch_status();
}

}  // namespace
}  // namespace frt

extern "C" size_t frt_quantize_workspace_bytes(int64_t rows, int64_t cols, frt_scale_mode mode) {
  if (rows < 0 || cols < 0) return 0;
  const size_t header = static_cast<size_t>(frt::kHeaderFloats) * sizeof(float);
  if (mode == FRT_SCALE_PER_COL)
    return header +
           static_cast<size_t>(frt::ceil_div(rows, frt::kColRowsPerBlock) * cols) * sizeof(float);
  return header + static_cast<size_t>(frt::kMaxPartials) * sizeof(float);
}

extern "C" frt_status frt_quantize_e4m3(const void* x, frt_dtype x_dtype, int64_t rows,
                                        int64_t cols, int64_t ldx, frt_scale_mode mode,
                                        frt_dtype out_fmt, const float* static_scale, uint8_t* q,
                                        float* scale, void* workspace, size_t workspace_bytes,
                                        frt_stream_t stream) {
  using namespace frt;
  if (x_dtype != FRT_BF16 && x_dtype != FRT_F32) return FRT_ERR_INVALID_ARG;
  if (out_fmt != FRT_E4M3_OCP && out_fmt != FRT_E4M3_FNUZ) return FRT_ERR_INVALID_ARG;
  if (mode != FRT_SCALE_PER_TENSOR && mode != FRT_SCALE_PER_COL) return FRT_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || ldx < cols) return FRT_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FRT_OK;
  if (!x || !q) return FRT_ERR_INVALID_ARG;
  if (!static_scale && !workspace) return FRT_ERR_INVALID_ARG;
  if (rows > (1LL << 40) || cols > (1LL << 31)) return FRT_ERR_UNSUPPORTED_SHAPE;
  const size_t esize = x_dtype == FRT_BF16 ? 2 : 4;
  if (!aligned(x, esize) || (scale && !aligned(scale, 4)) ||
      (static_scale && !aligned(static_scale, 4)) || (workspace && !aligned(workspace, 4)))
    return FRT_ERR_MISALIGNED;
  if (!static_scale && workspace_bytes < frt_quantize_workspace_bytes(rows, cols, mode))
    return FRT_ERR_WORKSPACE_TOO_SMALL;
  float* ws = static_cast<float*>(workspace);
  cudaStream_t st = as_cuda(stream);
  const bool fnuz = out_fmt == FRT_E4M3_FNUZ;
  if (x_dtype == FRT_BF16) {
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    return fnuz ? quantize_typed<__nv_bfloat16, true>(xb, rows, cols, ldx, mode, static_scale, q,
                                                      scale, ws, st)
                : quantize_typed<__nv_bfloat16, false>(xb, rows, cols, ldx, mode, static_scale,
                                                       q, scale, ws, st);
  }
  const auto* xf = static_cast<const float*>(x);
  return fnuz ? quantize_typed<float, true>(xf, rows, cols, ldx, mode, static_scale, q, scale, ws,
                                            st)
              : quantize_typed<float, false>(xf, rows, cols, ldx, mode, static_scale, q, scale,
                                             ws, st);
}

extern "C" frt_status frt_fnuz_to_ocp(const uint8_t* in, uint8_t* out, size_t n,
                                      frt_stream_t stream) {
  using namespace frt;
  if (n == 0) return FRT_OK;
  if (!in || !out) return FRT_ERR_INVALID_ARG;
  const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
  if (a != b && a < b + n && b < a + n) return FRT_ERR_INVALID_ARG;  // partial overlap
  cudaStream_t st = as_cuda(stream);
  const int cap = (sm_count() > 0 ? sm_count() : 148) * 8;
  if (aligned(in, 16) && aligned(out, 16)) {
    const size_t n16 = n / 16;
    if (n16) {
      const int64_t want = ceil_div(static_cast<int64_t>(n16), 256);
      const int grid = static_cast<int>(want < cap ? want : cap);
      fnuz_to_ocp_vec_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(in),
                                                   reinterpret_cast<uint4*>(out), n16);
      note_launches(1);
    }
    const size_t tail = n - n16 * 16;
    if (tail) {
      fnuz_to_ocp_byte_kernel<<<1, 32, 0, st>>>(in + n16 * 16, out + n16 * 16, tail);
      note_launches(1);
    }
  } else {
    const int64_t want = ceil_div(static_cast<int64_t>(n), 256);
    const int grid = static_cast<int>(want < cap ? want : cap);
    fnuz_to_ocp_byte_kernel<<<grid, 256, 0, st>>>(in, out, n);
    note_launches(1);
  }
  return launch_status();
}

// ------------------------------------------------------------------ quantize without allocation
//
// Some callers cannot allocate device memory: a real-time control loop that
// forbids allocator calls once it is running, a plugin that only receives
// raw device pointers from a host application, or code that records a CUDA
// graph in a mode where allocation would break the capture.  For them,
// frt_quantize_e4m3_noalloc keeps its workspace (the 256-byte header of the
// one-grid path, zero from the moment the library loads, then the amax
// partials) in the fixed array below instead of a caller-provided one.
// Every GPU that loads the library holds the array until the process exits.

namespace frt {
namespace {

constexpr int64_t kNoAllocScratchFloats = 262144;  // 1 MiB of partials

static __device__ __align__(256) float g_noalloc_scratch[kHeaderFloats + kNoAllocScratchFloats];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
float* noalloc_scratch(frt_status* status) {
  static std::mutex mu;
  static float* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    *status = FRT_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      *status = FRT_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = static_cast<float*>(p);
  }
  return addr[dev];
}

}  // namespace
}  // namespace frt

extern "C" frt_status frt_quantize_e4m3_noalloc(const void* x, frt_dtype x_dtype, int64_t rows,
                                                int64_t cols, int64_t ldx, frt_scale_mode mode,
                                                frt_dtype out_fmt, const float* static_scale,
                                                uint8_t* q, float* scale, frt_stream_t stream) {
  using namespace frt;
  if (x_dtype != FRT_BF16 && x_dtype != FRT_F32) return FRT_ERR_INVALID_ARG;
  if (out_fmt != FRT_E4M3_OCP && out_fmt != FRT_E4M3_FNUZ) return FRT_ERR_INVALID_ARG;
  if (mode != FRT_SCALE_PER_TENSOR && mode != FRT_SCALE_PER_COL) return FRT_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || ldx < cols) return FRT_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FRT_OK;
  if (!x || !q) return FRT_ERR_INVALID_ARG;
  if (rows > (1LL << 40) || cols > (1LL << 31)) return FRT_ERR_UNSUPPORTED_SHAPE;
  const size_t esize = x_dtype == FRT_BF16 ? 2 : 4;
  if (!aligned(x, esize) || (scale && !aligned(scale, 4)) ||
      (static_scale && !aligned(static_scale, 4)))
    return FRT_ERR_MISALIGNED;
  // the scratch holds the header and at most kNoAllocScratchFloats partial maxima
  if (!static_scale && frt_quantize_workspace_bytes(rows, cols, mode) >
                           static_cast<size_t>(kHeaderFloats + kNoAllocScratchFloats) *
                               sizeof(float))
    return FRT_ERR_UNSUPPORTED_SHAPE;
  frt_status st = FRT_OK;
  float* ws = noalloc_scratch(&st);
  if (!ws) return st;
  cudaStream_t s = as_cuda(stream);
  const bool fnuz = out_fmt == FRT_E4M3_FNUZ;
  if (x_dtype == FRT_BF16) {
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    return fnuz ? quantize_typed<__nv_bfloat16, true>(xb, rows, cols, ldx, mode, static_scale, q,
                                                      scale, ws, s)
                : quantize_typed<__nv_bfloat16, false>(xb, rows, cols, ldx, mode, static_scale,
                                                       q, scale, ws, s);
  }
  const auto* xf = static_cast<const float*>(x);
  return fnuz ? quantize_typed<float, true>(xf, rows, cols, ldx, mode, static_scale, q, scale, ws, s)
              : quantize_typed<float, false>(xf, rows, cols, ldx, mode, static_scale, q, scale,
                                             ws, s);
}
