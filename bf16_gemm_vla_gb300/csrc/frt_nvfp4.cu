// NVFP4 (block-scaled 4-bit floats): quantize and GEMM.
//
// The FlashRT article names an NVFP4 path beside FP8 for the pi0.5 encoder
// FFN (section 7.2 of its table of contents, "NVFP4 path"; the use_fp4 /
// fp4_layers switches of its load_model listing) and gives no formula.  The
// format is read as E2M1 elements with one E4M3 scale per 16 consecutive
// elements along the reduction dimension K and one fp32 scale g per tensor
// (frt.h states the steps).
//
//   * Quantize: pass 1 folds the CTAs' maxima |x| into a workspace word;
//     pass 2 gives each thread one 16-element block: block maximum, E4M3
//     block scale, E2M1 codes (two per byte), and writes the block scale in
//     the GEMM's tiled layout.  The last CTA of pass 2 clears the workspace.
//   * GEMM: 128 x 128 output tiles, one CTA each, persistent.  A pipeline
//     stage holds one 256-element k-block of both operands (codes, 128 bytes
//     per row, 128-byte swizzle) and their four + four 512-byte scale atoms.
//     The MMA thread copies each atom into TMEM (tcgen05.cp) and issues the
//     block-scaled MMA (kind::mxf4nvf4, K = 64, four per k-block); the
//     epilogue multiplies by g_a g_w, adds the bias, applies the GELU and
//     stores bf16 by TMA.
//
// Scale layout ("tiled"), for a tensor of V vectors (rows of A, output
// channels of W) blocked along K: the scale of vector v, block j sits at
//   ((v / 128) * (K / 64) + j / 4) * 512 + 16 * (v % 32) + 4 * ((v % 128) / 32) + j % 4,
// so one 512-byte atom holds 128 vectors x 4 blocks (64 elements of K) as
// 32 lines of 16 bytes; line i carries vectors i, i + 32, i + 64, i + 96.
// tcgen05.cp .32x128b.warpx4 puts line i into TMEM lane i of every 32-lane
// quarter, 4 columns wide, which is where the MMA reads the scales of the
// 128 rows of one K = 64 step.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "frt_device.cuh"
#include "frt_e4m3.cuh"
#include "frt_epilogue.cuh"
#include "frt_host.h"
#include "frt_tma_host.h"

namespace frt {
namespace {

constexpr int kBlk = 16;  // elements per block scale
constexpr float kNvMaxProduct = 6.0f * 448.0f;  // E2M1 max x E4M3 max

__host__ __device__ inline int64_t sf_offset(int64_t v, int64_t j, int64_t kc_total) {
  return ((v / 128) * kc_total + j / 4) * 512 + 16 * (v % 32) + 4 * ((v % 128) / 32) + (j % 4);
}

// ------------------------------------------------------------------ element codes

// E2M1 code of an fp32 value, round to nearest with ties to the even code.
// The magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7); between two
// neighbours the midpoint goes to the one with mantissa bit 0: 0.25 -> 0,
// 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4; from 6 up
// (infinity included) the code saturates at 6.  The sign bit is kept, a
// value that rounds to zero included; NaN gives +0.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  if (!(y == y)) return 0u;
  const uint32_t sign = (__float_as_uint(y) >> 28) & 8u;
  const float a = fabsf(y);
  const uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                     (a >= 3.5f) + (a > 5.0f);
  return sign | c;
}

// E2M1 code of the IEEE fp32 quotient x / e, with r = RN(1 / e) a positive
// normal number (fast).  As for the E4M3 encode of the quantize kernels:
// RN(x / e) lies within a relative 1.5 * 2^-23 of y = x * r, so inside
// [y (1 - 2^-20), y (1 + 2^-20)] even after that bracket's own rounding; the
// code is monotone in the value, so when both ends of the bracket give the
// same code, so does RN(x / e).  Otherwise (y within a few ulps of a
// rounding boundary) the IEEE division decides.
__device__ __forceinline__ uint32_t e2m1_code_div(float x, float e, float r, bool fast) {
  if (fast) {
    const float y = x * r;
    const uint32_t lo = e2m1_code(y * (1.0f - 0x1p-20f));
    const uint32_t hi = e2m1_code(y * (1.0f + 0x1p-20f));
    if (lo == hi) return lo;
  }
  return e2m1_code(__fdiv_rn(x, e));
}

// E2M1 codes of the two fp32 lanes of v by the hardware conversion (round to
// nearest even, saturating at +-6, the sign of a zero kept): the low lane in
// the low nibble of the byte returned.  Not for NaN (E2M1 has no NaN code).
__device__ __forceinline__ uint32_t cvt_e2m1x2(unsigned long long v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Value of a non-negative OCP E4M3 byte (no NaN: the block scales saturate).
__device__ __forceinline__ float e4m3_value_pos(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  return e == 0 ? static_cast<float>(m) * 0x1p-9f
                : __uint_as_float(((e + 120u) << 23) | (m << 20));  // (1 + m/8) 2^(e-7)
}

template <typename T>
__device__ __forceinline__ float nv_to_f32(T v);
template <>
__device__ __forceinline__ float nv_to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float nv_to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// ------------------------------------------------------------------ quantize

constexpr int kNvQThreads = 256;

// Pass 1: max |x| over the tensor (NaN ignored by fmaxf), folded into ws[0].
// kVec: x is read as 16-byte vectors (cols and ldx multiples of the vector,
// x 16-byte aligned), four in flight per thread; else element by element.
template <typename T, bool kVec>
__global__ void __launch_bounds__(kNvQThreads) nvfp4_amax_kernel(const T* __restrict__ x,
                                                                  int64_t rows, int64_t cols,
                                                                  int64_t ldx, unsigned* ws) {
  constexpr int VEC = kVec ? 16 / static_cast<int>(sizeof(T)) : 1;
  constexpr int kU = 4;
  __shared__ float red[kNvQThreads / 32];
  dev::grid_dependency_wait();  // x may come from the previous grid
  float m = 0.0f;
  // (the host keeps rows * cols below 2^31: 32-bit index arithmetic)
  const uint32_t vpr = static_cast<uint32_t>(cols / VEC);
  const uint32_t total = static_cast<uint32_t>(rows) * vpr;
  const uint32_t stride = gridDim.x * kNvQThreads;
  for (uint32_t i0 = blockIdx.x * kNvQThreads + threadIdx.x; i0 < total; i0 += kU * stride) {
    if constexpr (kVec) {
      uint4 w[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const uint32_t i = i0 + u * stride;
        const uint32_t r = i / vpr, c = i - r * vpr;
        w[u] = i < total ? __ldg(reinterpret_cast<const uint4*>(x + r * ldx + c * VEC))
                         : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const uint32_t ww[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if constexpr (sizeof(T) == 2) {
            m = fmaxf(m, fabsf(__uint_as_float(ww[k] << 16)));
            m = fmaxf(m, fabsf(__uint_as_float(ww[k] & 0xFFFF0000u)));
          } else {
            m = fmaxf(m, fabsf(__uint_as_float(ww[k])));
          }
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const uint32_t i = i0 + u * stride;
        if (i < total) {
          const uint32_t r = i / vpr, c = i - r * vpr;
          m = fmaxf(m, fabsf(nv_to_f32<T>(x[r * ldx + c])));
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kNvQThreads / 32; ++w) m = fmaxf(m, red[w]);
    if (m > 0.0f) atomicMax(ws, __float_as_uint(m));  // m >= 0: bits order as values
  }
  dev::grid_launch_dependents();
}

// One thread per (vector v, block j).  kAlongRows: x is [K x V] (blocks run
// down the columns, e.g. a weight W[K x N]); else x is [V x K].  Codes are
// written in x's orientation, two per byte along K (element 2i in the low
// nibble): [V x K/2] or [K/2 x V]; block scales in the tiled layout, the
// vectors past V (up to the next multiple of 128) with scale 0.
template <typename T, bool kAlongRows>
__global__ void __launch_bounds__(kNvQThreads) nvfp4_encode_kernel(
    const T* __restrict__ x, int64_t V, int64_t Kd, int64_t ldx, const float* static_scale,
    unsigned* ws, uint8_t* __restrict__ q, uint8_t* __restrict__ sf, float* scale_out) {
  __shared__ float g_sh;
  dev::grid_dependency_wait();  // x, the amax word and a static scale come from earlier grids
  if (threadIdx.x == 0) {
    float g;
    if (static_scale) {
      g = __ldcg(static_scale);
    } else {
      const float amax = __uint_as_float(__ldcg(ws));
      g = amax == 0.0f ? 1.0f : __fdiv_rn(amax, kNvMaxProduct);
    }
    g_sh = g;
    if (blockIdx.x == 0 && scale_out) *scale_out = g;
  }
  __syncthreads();
  const float g = g_sh;
  const float d = __fmul_rn(6.0f, g);
  // RN(1 / d), for the block scales' bracket when it is a positive normal number
  const float rd = __frcp_rn(d);
  const bool fast_d = (__float_as_uint(rd) >> 23) - 1u < 254u;
  // (the host keeps vpad * nb below 2^31: 32-bit index arithmetic)
  const uint32_t nb = static_cast<uint32_t>(Kd / kBlk);  // blocks per vector
  const uint32_t vpad = static_cast<uint32_t>((V + 127) / 128 * 128);
  const int64_t kc_total = Kd / 64;
  const uint32_t total = vpad * nb;
  const uint32_t stride = gridDim.x * kNvQThreads;
  // block (v, j): vector v (a row of x, or a column when kAlongRows), its
  // elements 16 j ... 16 j + 15 in f; writes the codes and the block scale
  auto encode_block = [&](const float (&f)[kBlk], int64_t v, int64_t j) {
    float b = 0.0f;
    bool nan = false;
#pragma unroll
    for (int i = 0; i < kBlk; ++i) {
      b = fmaxf(b, fabsf(f[i]));
      nan |= f[i] != f[i];
    }
    // sb = E4M3(RN(b / d)) (b >= 0, d > 0: a non-negative byte), by the bracket of
    // the E4M3 quantize on z = b * RN(1 / d): both ends converted by one hardware
    // conversion, the IEEE division where their bytes differ
    const float z = b * rd;
    const uint32_t c2 = cvt_e4m3x2_ocp(z * (1.0f - 0x1p-20f), z * (1.0f + 0x1p-20f));
    const uint32_t sbyte = (fast_d && (c2 & 0xFFu) == (c2 >> 8))
                               ? (c2 & 0xFFu)
                               : encode_e4m3<false>(__fdiv_rn(b, d));
    const float e = __fmul_rn(e4m3_value_pos(sbyte), g);
    const float r = __frcp_rn(e);
    const bool fast = e > 0.0f && (__float_as_uint(r) >> 23) - 1u < 254u;
    // the 16 codes as 8 bytes, element 2 p in the low nibble of byte p (lo:
    // bytes 0-3, hi: bytes 4-7).  Fast path: the bracket of e2m1_code_div
    // on packed products, both ends converted by the hardware, one test for
    // the block; a block with a NaN, a bracket that straddles a rounding
    // boundary or no usable reciprocal takes the element-wise path.
    uint32_t lo = 0u, hi = 0u;
    bool done = false;
    if (fast && !nan) {
      const unsigned long long rr = f32x2(r, r);
      const unsigned long long dn = f32x2(1.0f - 0x1p-20f, 1.0f - 0x1p-20f);
      const unsigned long long up = f32x2(1.0f + 0x1p-20f, 1.0f + 0x1p-20f);
      uint32_t lo_u = 0u, hi_u = 0u;
#pragma unroll
      for (int p2 = 0; p2 < kBlk / 2; ++p2) {
        const unsigned long long y = mul_f32x2(f32x2(f[2 * p2], f[2 * p2 + 1]), rr);
        const uint32_t cd = cvt_e2m1x2(mul_f32x2(y, dn));
        const uint32_t cu = cvt_e2m1x2(mul_f32x2(y, up));
        if (p2 < 4) {
          lo |= cd << (8 * p2);
          lo_u |= cu << (8 * p2);
        } else {
          hi |= cd << (8 * (p2 - 4));
          hi_u |= cu << (8 * (p2 - 4));
        }
      }
      done = lo == lo_u && hi == hi_u;
    }
    if (!done) {
      lo = 0u;
      hi = 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        lo |= (e > 0.0f ? e2m1_code_div(f[i], e, r, fast) : 0u) << (4 * i);
        hi |= (e > 0.0f ? e2m1_code_div(f[8 + i], e, r, fast) : 0u) << (4 * i);
      }
    }
    if constexpr (kAlongRows) {
      // [K/2 x V]: byte (8 j + p, v) holds elements 16 j + 2 p (low) and + 1
#pragma unroll
      for (int p2 = 0; p2 < kBlk / 2; ++p2)
        q[(j * (kBlk / 2) + p2) * V + v] =
            static_cast<uint8_t>(((p2 < 4 ? lo : hi) >> (8 * (p2 & 3))) & 0xFFu);
    } else {
      *reinterpret_cast<uint2*>(q + v * (Kd / 2) + j * (kBlk / 2)) = make_uint2(lo, hi);
    }
    sf[sf_offset(v, j, kc_total)] = static_cast<uint8_t>(sbyte);
  };
  for (uint32_t t = blockIdx.x * kNvQThreads + threadIdx.x; t < total; t += stride) {
    int64_t v, j;
    if constexpr (kAlongRows) {  // consecutive threads: consecutive columns (coalesced)
      v = t % vpad;
      j = t / vpad;
    } else {  // consecutive threads: consecutive blocks of a row
      v = t / nb;
      j = t % nb;
    }
    if (v >= V) {
      sf[sf_offset(v, j, kc_total)] = 0u;  // padding vectors: scale 0
      continue;
    }
    float f[kBlk];
    if constexpr (kAlongRows) {
#pragma unroll
      for (int i = 0; i < kBlk; ++i) f[i] = nv_to_f32<T>(x[(j * kBlk + i) * ldx + v]);
    } else if constexpr (sizeof(T) == 2) {
      const uint4* src = reinterpret_cast<const uint4*>(x + v * ldx + j * kBlk);
      const uint4 w0 = src[0], w1 = src[1];
      const uint32_t ws8[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        f[2 * k] = __uint_as_float(ws8[k] << 16);
        f[2 * k + 1] = __uint_as_float(ws8[k] & 0xFFFF0000u);
      }
    } else {
      const float4* src = reinterpret_cast<const float4*>(x + v * ldx + j * kBlk);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 a = src[k];
        f[4 * k] = a.x; f[4 * k + 1] = a.y; f[4 * k + 2] = a.z; f[4 * k + 3] = a.w;
      }
    }
    encode_block(f, v, j);
  }
  // the amax word is read by every CTA before it counts itself done here; the
  // last one clears it (and the count) for the next call
  if (!static_scale) {
    __syncthreads();
    if (threadIdx.x == 0 && atomicAdd(ws + 1, 1u) == gridDim.x - 1) {
      ws[0] = 0u;
      ws[1] = 0u;
    }
  }
  dev::grid_launch_dependents();
}

// ------------------------------------------------------------------ GEMM

constexpr int kNvThreads = 192;  // copy warp, MMA warp, 4 epilogue warps
constexpr int kNvTile = 128;     // rows of a tile; channels of one half
constexpr int kNvOpBytes = kNvTile * 128;  // codes of 128 rows per k-block (256 elements)
constexpr int kNvSfBytes = 4 * 512;        // 4 scale atoms of 128 rows per k-block
constexpr uint32_t kNvTmemCols = 512;

// A tile is 128 rows x 128 channels: per K step (64 elements) one block-
// scaled MMA of 128 x 128.  TMEM: two accumulators of 128 columns (a tile's
// epilogue overlaps the next tile's MMAs), then per stage 16 columns of A
// scales and 16 of B scales.  (Tiles of 256 channels, two MMAs sharing the
// activations, were measured no faster: the k-block rate, not the bytes
// per FLOP, is the limit.)
struct NvCfg {
  static constexpr int kHalves = 1;
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = (1 + kHalves) * kNvOpBytes + (1 + kHalves) * kNvSfBytes;
  static constexpr int kOutOff = kStages * kStageBytes;
  static constexpr int kBiasOff = kOutOff + 4 * 2 * kWarpOutBytes;
  static constexpr int kBarOff = kBiasOff + 2 * kHalves * kNvTile * 4;
  static constexpr int kSmem = 1024 + kBarOff + 256;
  static constexpr int kAccBufs = 2;
  static constexpr uint32_t kAccCols = kHalves * kNvTile;
  static constexpr uint32_t kSfCol0 = kAccBufs * kAccCols;
  static constexpr uint32_t kSfColsPerStage = 16u * (1 + kHalves);
  static_assert(kSfCol0 + kStages * kSfColsPerStage <= kNvTmemCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct NvGemmArgs {
  const uint8_t* a_sf;
  const uint8_t* w_packed;
  const uint8_t* w_sf;
  const float* a_scale;  // g_a (1 float) or null (= 1)
  const float* w_scale;  // g_w (1 float) or null (= 1)
  const float* bias;     // N floats or null
  int M, N, act_cols;
  int kb_total;  // 256-element k-blocks
  int kc_total;  // 64-element scale chunks (K / 64)
  int tiles_m, num_tiles;
  int* dev_status;
};

__global__ void __launch_bounds__(kNvThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_out, const NvGemmArgs p) {
  using C = NvCfg;
  constexpr int kHalves = C::kHalves;
  constexpr int kNvStages = C::kStages;
  constexpr int kNvStageBytes = C::kStageBytes;
  constexpr int kTileN = kHalves * kNvTile;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (dev::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = dev::smem_u32(base);
  float* bias_s = reinterpret_cast<float*>(base + C::kBiasOff);  // [2 tiles][kTileN channels]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  const uint32_t full0 = dev::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kNvStages;
  const uint32_t tfull0 = empty0 + 8 * kNvStages;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t scale_bar = tempty0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kNvStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* gscale_s = reinterpret_cast<float*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNvStages; ++s) {
      dev::mbar_init(full0 + 8 * s, 1);
      dev::mbar_init(empty0 + 8 * s, 1);
    }
    dev::mbar_init(tfull0, 1);
    dev::mbar_init(tfull0 + 8, 1);
    dev::mbar_init(tempty0, 4);
    dev::mbar_init(tempty0 + 8, 4);
    dev::mbar_init(scale_bar, 1);
    *abort_flag = 0;
    dev::fence_mbar_init();
    dev::prefetch_tmap(&tmap_a);
    dev::prefetch_tmap(&tmap_out);
  }
  if (warp == 1) dev::tmem_alloc(dev::smem_u32(tmem_slot), kNvTmemCols);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  dev::grid_launch_dependents();

  const int first = static_cast<int>(blockIdx.x);
  const int step = static_cast<int>(gridDim.x);
  const int my_tiles = first < p.num_tiles ? (p.num_tiles - first + step - 1) / step : 0;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ copies
      const uint64_t pol_w = dev::policy_evict_normal();
      const uint64_t pol_a = dev::policy_evict_last();
      // the activations, their scales and g_a come from the previous grid
      dev::grid_dependency_wait();
      *gscale_s = __fmul_rn(p.a_scale ? __ldcg(p.a_scale) : 1.0f,
                            p.w_scale ? __ldcg(p.w_scale) : 1.0f);
      dev::mbar_arrive(scale_bar);
      int s = 0, issued = 0;
      uint32_t ph = 0;
      bool stop = false;
      for (int it = 0; it < my_tiles && !stop; ++it) {
        const int t = first + it * step;
        const int tm = t % p.tiles_m, tn = t / p.tiles_m;
        for (int kb = 0; kb < p.kb_total; ++kb) {
          if (!dev::mbar_wait(empty0 + 8 * s, (ph & 1) ^ 1, abort_flag, p.dev_status,
                              dev::kTimeoutProducer)) {
            stop = true;
            break;
          }
          const uint32_t st = sbase + s * kNvStageBytes;
          const uint32_t fb = full0 + 8 * s;
          dev::mbar_arrive_expect_tx(fb, kNvStageBytes);
          // stage: A codes, B codes of each half (128 channel rows apiece,
          // adjacent: one 128 x kTileN operand), A scales, B scales per half
          dev::tma_load_2d(st, &tmap_a, kb * 128, tm * kNvTile, fb, pol_a);
#pragma unroll
          for (int h = 0; h < kHalves; ++h) {
            const size_t nb = static_cast<size_t>(tn) * kHalves + h;
            dev::bulk_load(st + (1 + h) * kNvOpBytes,
                           p.w_packed + (nb * p.kb_total + kb) * kNvOpBytes, kNvOpBytes, fb,
                           pol_w);
            dev::bulk_load(st + (1 + kHalves) * kNvOpBytes + (1 + h) * kNvSfBytes,
                           p.w_sf + (nb * p.kc_total + 4 * kb) * 512, kNvSfBytes, fb, pol_w);
          }
          dev::bulk_load(st + (1 + kHalves) * kNvOpBytes,
                         p.a_sf + (static_cast<size_t>(tm) * p.kc_total + 4 * kb) * 512,
                         kNvSfBytes, fb, pol_a);
          ++issued;
          if (++s == kNvStages) {
            s = 0;
            ++ph;
          }
        }
      }
      // no copies in flight when the CTA leaves (bounded, even after an abort)
      for (int g = issued - kNvStages < 0 ? 0 : issued - kNvStages; g < issued; ++g)
        dev::mbar_wait(full0 + 8 * (g % kNvStages), (g / kNvStages) & 1, nullptr, p.dev_status,
                       dev::kTimeoutProducer);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ scales + MMA
      constexpr uint32_t idesc = dev::instr_desc_nvfp4(kNvTile, kNvTile);
      int s = 0;
      uint32_t ph = 0;
      bool stop = false;
      for (int it = 0; it < my_tiles && !stop; ++it) {
        const int b = it % C::kAccBufs;
        const uint32_t u = static_cast<uint32_t>(it / C::kAccBufs);
        if (!dev::mbar_wait(tempty0 + 8 * b, (u & 1) ^ 1, abort_flag, p.dev_status,
                            dev::kTimeoutMma))
          break;
        dev::tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b) * C::kAccCols;
        for (int kb = 0; kb < p.kb_total; ++kb) {
          if (!dev::mbar_wait(full0 + 8 * s, ph & 1, abort_flag, p.dev_status, dev::kTimeoutMma)) {
            stop = true;
            break;
          }
          dev::tc_fence_after();
          const uint32_t st = sbase + s * kNvStageBytes;
          const uint32_t sf_st = st + (1 + kHalves) * kNvOpBytes;  // A scales, then B per half
          const uint64_t ad = dev::smem_desc_sw128(st);
          // 16 columns of A scales, then 16 of B scales per half
          const uint32_t sfa = tmem + C::kSfCol0 + C::kSfColsPerStage * s;
          // the k-block's scale atoms first (copies and MMAs run in issue
          // order), then its MMAs back to back
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            dev::tmem_cp_32x128b_x4(sfa + 4u * k, dev::smem_desc_noswz(sf_st + 512 * k, 128, 128));
#pragma unroll
            for (int h = 0; h < kHalves; ++h)
              dev::tmem_cp_32x128b_x4(
                  sfa + 16u * (1 + h) + 4u * k,
                  dev::smem_desc_noswz(sf_st + (1 + h) * kNvSfBytes + 512 * k, 128, 128));
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int h = 0; h < kHalves; ++h)
              dev::mma_nvfp4(d + h * kNvTile, ad + 2 * k,
                             dev::smem_desc_sw128(st + (1 + h) * kNvOpBytes) + 2 * k, idesc,
                             sfa + 4u * k, sfa + 16u * (1 + h) + 4u * k, (kb | k) != 0);
          }
          dev::mma_commit(empty0 + 8 * s);
          if (++s == kNvStages) {
            s = 0;
            ++ph;
          }
        }
        dev::mma_commit(tfull0 + 8 * b);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int et = threadIdx.x - 64;
    const int ew = warp & 3;  // TMEM lane quarter
    const uint32_t lane_off = static_cast<uint32_t>(ew * 32) << 16;
    uint8_t* wbuf = base + C::kOutOff + (warp - 2) * 2 * kWarpOutBytes;
    const uint32_t wbuf_s = sbase + C::kOutOff + (warp - 2) * 2 * kWarpOutBytes;
    int wb = 0;
    // the four warps leave the tile loop together (named_all), so none is
    // left alone at a named barrier
    bool ok = dev::named_all(
        1, 128, dev::mbar_wait(scale_bar, 0, abort_flag, p.dev_status, dev::kTimeoutEpilogue));
    const float gs = *gscale_s;
    for (int it = 0; it < my_tiles && ok; ++it) {
      const int t = first + it * step;
      const int tm = t % p.tiles_m, tn = t / p.tiles_m;
      const int b = it % C::kAccBufs;
      const uint32_t u = static_cast<uint32_t>(it / C::kAccBufs);
      float* bs = bias_s + (it & 1) * kTileN;
#pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        const int n = tn * kTileN + h * kNvTile + et;
        bs[h * kNvTile + et] = (p.bias && n < p.N) ? __ldg(p.bias + n) : 0.0f;
      }
      ok = dev::named_all(1, 128, dev::mbar_wait(tfull0 + 8 * b, u & 1, abort_flag, p.dev_status,
                                                 dev::kTimeoutEpilogue));
      if (!ok) break;
      dev::tc_fence_after();
      const uint32_t tacc = tmem + lane_off + static_cast<uint32_t>(b) * C::kAccCols;
#pragma unroll 1
      for (int c = 0; c < kTileN; c += 32) {
        float v[32];
        dev::tmem_ld32(tacc + c, v);
        if (c + 32 == kTileN) {  // accumulator read out: back to the MMA thread
          dev::tc_fence_before();
          __syncwarp();
          if (lane == 0) dev::mbar_arrive(tempty0 + 8 * b);
        }
        const int n0 = tn * kTileN + c;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = lin(v[j], gs, bs[c + j]);
        if (n0 + 32 <= p.act_cols) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = gelu_tanh(v[j]);
        } else if (n0 < p.act_cols) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float gv = gelu_tanh(v[j]);
            v[j] = n0 + j < p.act_cols ? gv : v[j];
          }
        }
        if (n0 < p.N)
          warp_store<false, 32>(v, wbuf + wb * kWarpOutBytes, wbuf_s + wb * kWarpOutBytes,
                                &tmap_out, n0, tm * kNvTile + ew * 32, lane);
        wb ^= 1;
      }
    }
    // the TMA stores have read their staging buffers before the CTA leaves;
    // their writes are performed before the grid completes (and before a
    // dependent grid's wait returns), so the CTA does not wait for them
    if (lane == 0) dev::bulk_wait_read<0>();
  }
  dev::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, kNvTmemCols);
  }
}

// Pair tiles (more than 128 rows): 256 rows x kBN channels on a CTA pair
// (cta_group::2).  Each CTA holds 128 rows of A and their scales, half of
// the tile's channels of B, and the B scales of all kBN channels (each
// CTA's accumulator has the tile's kBN columns); per K step the even CTA
// issues one MMA of M = 256, N = kBN, and one scale copy per atom that takes
// each CTA's shared memory into its own TMEM.  Every copy of both CTAs
// completes on the leader's full barrier.  kBN = 256 leaves TMEM room for
// one accumulator only (its epilogue does not overlap the next tile's MMAs);
// kBN = 128 keeps two.
template <int kBN>
struct NvPairCfg {
  static constexpr int kGroups = kBN / kNvTile;  // 128-channel groups of a tile
  static constexpr int kAccBufs = kGroups == 2 ? 1 : 2;
  static constexpr int kStages = kGroups == 2 ? 5 : 6;
  static constexpr int kABytes = kNvOpBytes;     // 128 rows x 128 bytes
  static constexpr int kBBytes = kBN / 2 * 128;  // this CTA's channels x 128 bytes
  static constexpr int kSfaOff = kABytes + kBBytes;
  static constexpr int kSfbOff = kSfaOff + kNvSfBytes;
  static constexpr int kStageBytes = kSfbOff + kGroups * kNvSfBytes;
  static constexpr int kOutOff = kStages * kStageBytes;
  static constexpr int kBiasOff = kOutOff + 4 * 2 * kWarpOutBytes;
  static constexpr int kBarOff = kBiasOff + 2 * kBN * 4;
  static constexpr int kSmem = 1024 + kBarOff + 256;
  static constexpr uint32_t kAccCols = kBN;
  static constexpr uint32_t kSfCol0 = kAccBufs * kAccCols;
  static constexpr uint32_t kSfbCols = 4 * kGroups;  // B scale columns per K step
  static constexpr uint32_t kSfColsPerStage = 16 + 4 * kSfbCols;
  static_assert(kStageBytes % 1024 == 0, "stages keep the 128-byte swizzle's alignment");
  static_assert(kSfCol0 + kStages * kSfColsPerStage <= kNvTmemCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

template <int kBN>
__global__ void __launch_bounds__(kNvThreads, 1)
    gemm_nvfp4_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                           const __grid_constant__ CUtensorMap tmap_w,
                           const __grid_constant__ CUtensorMap tmap_sfa,
                           const __grid_constant__ CUtensorMap tmap_sfb,
                           const __grid_constant__ CUtensorMap tmap_out, const NvGemmArgs p) {
  using C = NvPairCfg<kBN>;
  constexpr int kS = C::kStages;
  constexpr int kG = C::kGroups;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (dev::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = dev::smem_u32(base);
  float* bias_s = reinterpret_cast<float*>(base + C::kBiasOff);  // [2 tiles][kBN channels]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  const uint32_t full0 = dev::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kS;
  const uint32_t tfull0 = empty0 + 8 * kS;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t scale_bar = tempty0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kS + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* gscale_s = reinterpret_cast<float*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = dev::cluster_ctarank();
  const int px = static_cast<int>(crank & 1u);  // CTA within the pair
  const bool leader = px == 0;
  const uint32_t lead_rank = crank & ~1u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kS; ++s) {
      dev::mbar_init(full0 + 8 * s, 1);
      dev::mbar_init(empty0 + 8 * s, 1);
    }
    dev::mbar_init(tfull0, 1);
    dev::mbar_init(tfull0 + 8, 1);
    // an accumulator is released by the epilogue warps of both CTAs
    dev::mbar_init(tempty0, 8);
    dev::mbar_init(tempty0 + 8, 8);
    dev::mbar_init(scale_bar, 1);
    *abort_flag = 0;
    dev::fence_mbar_init();
    dev::prefetch_tmap(&tmap_a);
    dev::prefetch_tmap(&tmap_w);
    dev::prefetch_tmap(&tmap_sfa);
    dev::prefetch_tmap(&tmap_sfb);
    dev::prefetch_tmap(&tmap_out);
  }
  if (warp == 1) dev::tmem_alloc_pair(dev::smem_u32(tmem_slot), kNvTmemCols);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  dev::grid_launch_dependents();
  // both CTAs' barriers are initialised (published by fence.mbarrier_init)
  // before either signals the other's; every cluster-barrier arrive and wait
  // below is executed by all 32 lanes of a warp together
  dev::cluster_arrive_relaxed();
  dev::cluster_wait();

  const int first = static_cast<int>(blockIdx.x >> 1);
  const int step = static_cast<int>(gridDim.x >> 1);
  const int my_tiles = first < p.num_tiles ? (p.num_tiles - first + step - 1) / step : 0;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ copies
      const uint64_t pol_w = dev::policy_evict_normal();
      const uint64_t pol_a = dev::policy_evict_last();
      struct Cur {
        int it, kb, tm, tn;
      };
      auto set_tile = [&](Cur& c) {
        const int t = first + c.it * step;
        c.tm = t % p.tiles_m;
        c.tn = t / p.tiles_m;
      };
      auto advance = [&](Cur& c) {
        if (++c.kb == p.kb_total) {
          c.kb = 0;
          if (++c.it < my_tiles) set_tile(c);
        }
      };
      auto full_bar = [&](int s) { return dev::map_to_rank(full0 + 8 * s, lead_rank); };
      // static data: this CTA's half of the tile's channels of the weight
      // k-tile (64 rows of the tile's group, or the CTA's own group of 128)
      // and the scales of all kBN channels (the leader arms the stage for
      // both CTAs' bytes)
      auto load_w = [&](const Cur& c, int s) {
        const uint32_t st = sbase + s * C::kStageBytes;
        if (leader) dev::mbar_arrive_expect_tx(full0 + 8 * s, 2u * C::kStageBytes);
        const int grp = kG * c.tn + (kG == 2 ? px : 0);
        dev::tma_load_3d_pair(st + C::kABytes, &tmap_w, 0, kG == 2 ? 0 : px * (kNvTile / 2),
                              grp * p.kb_total + c.kb, full_bar(s), pol_w);
#pragma unroll
        for (int g = 0; g < kG; ++g)
          dev::tma_load_2d_pair(st + C::kSfbOff + g * kNvSfBytes, &tmap_sfb, 0,
                                ((kG * c.tn + g) * p.kc_total + 4 * c.kb) * 2, full_bar(s),
                                pol_w);
      };
      // the previous grid's data: this CTA's 128 rows and their scales
      auto load_a = [&](const Cur& c, int s) {
        const uint32_t st = sbase + s * C::kStageBytes;
        dev::tma_load_2d_pair(st, &tmap_a, c.kb * 128, c.tm * 2 * kNvTile + px * kNvTile,
                              full_bar(s), pol_a);
        dev::tma_load_2d_pair(st + C::kSfaOff, &tmap_sfa, 0,
                              ((2 * c.tm + px) * p.kc_total + 4 * c.kb) * 2, full_bar(s), pol_a);
      };
      const int total = my_tiles * p.kb_total;
      const int npre = total < kS ? total : kS;
      Cur start = {0, 0, 0, 0};
      if (my_tiles > 0) set_tile(start);
      Cur cur = start;
      for (int g = 0; g < npre; ++g) {  // first use of each stage needs no wait
        load_w(cur, g);
        advance(cur);
      }
      dev::grid_dependency_wait();
      cur = start;
      for (int g = 0; g < npre; ++g) {
        load_a(cur, g);
        advance(cur);
      }
      *gscale_s = __fmul_rn(p.a_scale ? __ldcg(p.a_scale) : 1.0f,
                            p.w_scale ? __ldcg(p.w_scale) : 1.0f);
      dev::mbar_arrive(scale_bar);
      int issued = npre;
      int s = npre % kS;
      uint32_t ph = static_cast<uint32_t>(npre / kS);
      for (int g = npre; g < total; ++g) {
        if (!dev::mbar_wait(empty0 + 8 * s, (ph & 1) ^ 1, abort_flag, p.dev_status,
                            dev::kTimeoutProducer))
          break;
        load_w(cur, s);
        load_a(cur, s);
        advance(cur);
        issued = g + 1;
        if (++s == kS) {
          s = 0;
          ++ph;
        }
      }
      // no copies in flight when the CTA leaves: the copies complete on the
      // leader's barriers, so wait (bounded, even after an abort) until the
      // MMAs released the last use of every stage armed
      for (int g = issued - kS < 0 ? 0 : issued - kS; g < issued; ++g)
        dev::mbar_wait(empty0 + 8 * (g % kS), (g / kS) & 1, nullptr, p.dev_status,
                       dev::kTimeoutProducer);
    }
    __syncwarp();
    dev::cluster_arrive_relaxed();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ scales + MMA
      constexpr uint32_t idesc = dev::instr_desc_nvfp4(2 * kNvTile, kBN);
      const uint16_t pair_mask = static_cast<uint16_t>(3u << lead_rank);
      int s = 0;
      uint32_t ph = 0;
      bool stop = false;
      for (int it = 0; it < my_tiles && !stop; ++it) {
        const int b = it % C::kAccBufs;
        const uint32_t u = static_cast<uint32_t>(it / C::kAccBufs);
        if (!dev::mbar_wait_cluster(tempty0 + 8 * b, (u & 1) ^ 1, abort_flag, p.dev_status,
                                    dev::kTimeoutMma))
          break;
        dev::tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b) * C::kAccCols;
        for (int kb = 0; kb < p.kb_total; ++kb) {
          if (!dev::mbar_wait(full0 + 8 * s, ph & 1, abort_flag, p.dev_status, dev::kTimeoutMma)) {
            stop = true;
            break;
          }
          dev::tc_fence_after();
          const uint32_t st = sbase + s * C::kStageBytes;
          const uint32_t sfa = tmem + C::kSfCol0 + C::kSfColsPerStage * s;
          const uint32_t sfb = sfa + 16;
          // the k-block's scale atoms (copies and MMAs run in issue order),
          // then its MMAs; per K step 4 columns of A scales and kSfbCols of B
          // scales, channel n of the tile in column n / 32 (one atom per
          // 128-channel group)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            dev::tmem_cp_32x128b_x4_pair(sfa + 4u * k,
                                         dev::smem_desc_noswz(st + C::kSfaOff + 512 * k, 128, 128));
#pragma unroll
            for (int g = 0; g < kG; ++g)
              dev::tmem_cp_32x128b_x4_pair(
                  sfb + C::kSfbCols * k + 4u * g,
                  dev::smem_desc_noswz(st + C::kSfbOff + g * kNvSfBytes + 512 * k, 128, 128));
          }
          const uint64_t ad = dev::smem_desc_sw128(st);
          const uint64_t bd = dev::smem_desc_sw128(st + C::kABytes);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dev::mma_nvfp4_pair(d, ad + 2 * k, bd + 2 * k, idesc, sfa + 4u * k,
                                sfb + C::kSfbCols * k, (kb | k) != 0);
          dev::mma_commit_pair(empty0 + 8 * s, pair_mask);
          if (++s == kS) {
            s = 0;
            ++ph;
          }
        }
        dev::mma_commit_pair(tfull0 + 8 * b, pair_mask);
      }
    }
    __syncwarp();
    dev::cluster_arrive_relaxed();
  } else {
    // -------------------------------------------------------------- epilogue
    const int et = threadIdx.x - 64;
    const int ew = warp & 3;  // TMEM lane quarter
    const uint32_t lane_off = static_cast<uint32_t>(ew * 32) << 16;
    uint8_t* wbuf = base + C::kOutOff + (warp - 2) * 2 * kWarpOutBytes;
    const uint32_t wbuf_s = sbase + C::kOutOff + (warp - 2) * 2 * kWarpOutBytes;
    int wb = 0;
    bool bye = false;  // arrived on the pair's final cluster barrier
    // the four warps leave the tile loop together (named_all), so none is
    // left alone at a named barrier
    bool ok = dev::named_all(
        1, 128, dev::mbar_wait(scale_bar, 0, abort_flag, p.dev_status, dev::kTimeoutEpilogue));
    const float gs = *gscale_s;
    for (int it = 0; it < my_tiles && ok; ++it) {
      const int t = first + it * step;
      const int tm = t % p.tiles_m, tn = t / p.tiles_m;
      const int b = it % C::kAccBufs;
      const uint32_t u = static_cast<uint32_t>(it / C::kAccBufs);
      float* bs = bias_s + (it & 1) * kBN;
#pragma unroll
      for (int g = 0; g < kG; ++g) {
        const int n = tn * kBN + g * kNvTile + et;
        bs[g * kNvTile + et] = (p.bias && n < p.N) ? __ldg(p.bias + n) : 0.0f;
      }
      ok = dev::named_all(1, 128, dev::mbar_wait(tfull0 + 8 * b, u & 1, abort_flag, p.dev_status,
                                                 dev::kTimeoutEpilogue));
      if (!ok || it + 1 == my_tiles) {  // every MMA that reads the peer is done
        dev::cluster_arrive_relaxed();
        bye = true;
      }
      if (!ok) break;
      dev::tc_fence_after();
      const uint32_t tacc = tmem + lane_off + static_cast<uint32_t>(b) * C::kAccCols;
      const int row0 = tm * 2 * kNvTile + px * kNvTile + ew * 32;
#pragma unroll 1
      for (int c = 0; c < kBN; c += 32) {
        float v[32];
        dev::tmem_ld32(tacc + c, v);
        // accumulator read out: back to the MMA thread, if it will wait for it
        if (c + 32 == kBN && it + C::kAccBufs < my_tiles) {
          dev::tc_fence_before();
          __syncwarp();
          if (lane == 0) dev::mbar_arrive_cluster(dev::map_to_rank(tempty0 + 8 * b, lead_rank));
        }
        const int n0 = tn * kBN + c;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = lin(v[j], gs, bs[c + j]);
        if (n0 + 32 <= p.act_cols) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = gelu_tanh(v[j]);
        } else if (n0 < p.act_cols) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float gv = gelu_tanh(v[j]);
            v[j] = n0 + j < p.act_cols ? gv : v[j];
          }
        }
        if (n0 < p.N)
          warp_store<false, 32>(v, wbuf + wb * kWarpOutBytes, wbuf_s + wb * kWarpOutBytes,
                                &tmap_out, n0, row0, lane);
        wb ^= 1;
      }
    }
    if (!bye) dev::cluster_arrive_relaxed();
    // the TMA stores have read their staging buffers before the CTA leaves
    if (lane == 0) dev::bulk_wait_read<0>();
  }
  // neither CTA leaves (or frees TMEM) while the other may still take part
  // in its MMAs or signal its barriers
  dev::cluster_wait();
  dev::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    dev::tc_fence_after();
    dev::tmem_dealloc_pair(tmem, kNvTmemCols);
  }
}

// Shared-memory attribute of a GEMM kernel, once per device.
template <typename Kern>
cudaError_t set_smem_once(Kern kern, int smem, std::mutex& mu, bool (&set)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!set[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    set[dev] = true;
  }
  return cudaSuccess;
}

cudaError_t launch_nvfp4(const CUtensorMap& ta, const CUtensorMap& to, const NvGemmArgs& ga,
                         int sms, cudaStream_t stream) {
  static std::mutex mu;
  static bool set[64] = {false};
  cudaError_t e = set_smem_once(gemm_nvfp4_kernel, NvCfg::kSmem, mu, set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ga.num_tiles < sms ? ga.num_tiles : sms));
  cfg.blockDim = dim3(kNvThreads);
  cfg.dynamicSmemBytes = NvCfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_nvfp4_kernel, ta, to, ga);
}

// ga.num_tiles counts 256-row pair tiles; at most one pair per two SMs and
// no more pairs than can be resident at once (a persistent grid when there
// are more tiles).
template <int kBN>
cudaError_t launch_nvfp4_pair(const CUtensorMap& ta, const CUtensorMap& tw,
                              const CUtensorMap& tsa, const CUtensorMap& tsb,
                              const CUtensorMap& to, const NvGemmArgs& ga, int sms,
                              cudaStream_t stream) {
  using C = NvPairCfg<kBN>;
  auto kern = gemm_nvfp4_pair_kernel<kBN>;
  static std::mutex mu;
  static bool set[64] = {false};
  static int capacity[64] = {0};
  cudaError_t e = set_smem_once(kern, C::kSmem, mu, set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kNvThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  int dev = 0;
  cudaGetDevice(&dev);
  int cap = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && capacity[dev] == 0) {
      cfg.gridDim = dim3(2);
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = -1;  // unknown: one pair per two SMs
      }
      capacity[dev] = n;
    }
    cap = dev >= 0 && dev < 64 ? capacity[dev] : -1;
  }
  int pairs = sms / 2;
  if (cap > 0 && cap < pairs) pairs = cap;
  if (ga.num_tiles < pairs) pairs = ga.num_tiles;
  if (pairs < 1) pairs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, ta, tw, tsa, tsb, to, ga);
}

template <typename T>
frt_status quantize_nvfp4_typed(const T* x, int64_t rows, int64_t cols, int64_t ldx,
                                bool along_rows, const float* static_scale, uint8_t* q,
                                uint8_t* sf, float* scale, unsigned* ws, cudaStream_t st) {
  const int sms = sm_count() > 0 ? sm_count() : 148;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kNvQThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaSuccess;
  int launches = 1;
  if (!static_scale) {
    constexpr int VEC = 16 / static_cast<int>(sizeof(T));
    const bool vec = aligned(x, 16) && cols % VEC == 0 && ldx % VEC == 0;
    const int64_t units = rows * (vec ? cols / VEC : cols);
    cfg.gridDim = dim3(static_cast<unsigned>(
        std::max<int64_t>(1, std::min<int64_t>(ceil_div(units, 4 * kNvQThreads), 4 * sms))));
    e = vec ? cudaLaunchKernelEx(&cfg, nvfp4_amax_kernel<T, true>, x, rows, cols, ldx, ws)
            : cudaLaunchKernelEx(&cfg, nvfp4_amax_kernel<T, false>, x, rows, cols, ldx, ws);
    ++launches;
  }
  const int64_t V = along_rows ? cols : rows;
  const int64_t Kd = along_rows ? rows : cols;
  const int64_t total = ceil_div(V, 128) * 128 * (Kd / kBlk);
  // one block per thread (an uneven share of blocks per thread left most warps
  // waiting at the end-of-CTA barrier)
  cfg.gridDim = dim3(static_cast<unsigned>(std::max<int64_t>(1, ceil_div(total, kNvQThreads))));
  if (e == cudaSuccess)
    e = along_rows ? cudaLaunchKernelEx(&cfg, nvfp4_encode_kernel<T, true>, x, V, Kd, ldx,
                                        static_scale, ws, q, sf, scale)
                   : cudaLaunchKernelEx(&cfg, nvfp4_encode_kernel<T, false>, x, V, Kd, ldx,
                                        static_scale, ws, q, sf, scale);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FRT_ERR_CUDA;
  }
  note_launches(launches);
  return launch_status();
}

}  // namespace
}  // namespace frt

extern "C" size_t frt_nvfp4_scale_bytes(int64_t vectors, int64_t K) {
  if (vectors < 1 || K < 64 || K % 64 != 0) return 0;
  return static_cast<size_t>(frt::ceil_div(vectors, 128) * 128 * (K / 16));
}

extern "C" size_t frt_quantize_nvfp4_workspace_bytes(void) { return 16; }

extern "C" frt_status frt_quantize_nvfp4(const void* x, frt_dtype x_dtype, int64_t rows,
                                         int64_t cols, int64_t ldx, int blocks_along_rows,
                                         const float* static_scale, uint8_t* q, uint8_t* sf,
                                         size_t sf_bytes, float* scale, void* workspace,
                                         size_t workspace_bytes, frt_stream_t stream) {
  if (!x || !q || !sf) return FRT_ERR_INVALID_ARG;
  if (x_dtype != FRT_BF16 && x_dtype != FRT_F32) return FRT_ERR_INVALID_ARG;
  if (rows < 1 || cols < 1 || ldx < cols) return FRT_ERR_INVALID_ARG;
  const int64_t V = blocks_along_rows ? cols : rows;
  const int64_t Kd = blocks_along_rows ? rows : cols;
  if (Kd % 64 != 0) return FRT_ERR_UNSUPPORTED_SHAPE;
  if (frt::ceil_div(V, 128) * 128 * (Kd / 16) > (1LL << 31) - 1 || rows * cols > (1LL << 31) - 1)
    return FRT_ERR_UNSUPPORTED_SHAPE;
  if (sf_bytes < frt_nvfp4_scale_bytes(V, Kd)) return FRT_ERR_WORKSPACE_TOO_SMALL;
  if (!static_scale && (!workspace || workspace_bytes < 16)) return FRT_ERR_WORKSPACE_TOO_SMALL;
  const int esz = x_dtype == FRT_BF16 ? 2 : 4;
  if (!frt::aligned(x, 16) || (ldx * esz) % 16 != 0 || !frt::aligned(q, 16) ||
      (workspace && !frt::aligned(workspace, 16)) || (scale && !frt::aligned(scale, 4)) ||
      (static_scale && !frt::aligned(static_scale, 4)))
    return FRT_ERR_MISALIGNED;
  unsigned* ws = static_cast<unsigned*>(workspace);
  const cudaStream_t st = frt::as_cuda(stream);
  if (x_dtype == FRT_BF16)
    return frt::quantize_nvfp4_typed(static_cast<const __nv_bfloat16*>(x), rows, cols, ldx,
                                     blocks_along_rows != 0, static_scale, q, sf, scale, ws, st);
  return frt::quantize_nvfp4_typed(static_cast<const float*>(x), rows, cols, ldx,
                                   blocks_along_rows != 0, static_scale, q, sf, scale, ws, st);
}

extern "C" frt_status frt_gemm_nvfp4(const uint8_t* a_q, int64_t lda, const uint8_t* a_sf,
                                     const float* a_scale, const void* w_packed,
                                     const uint8_t* w_sf, const float* w_scale, const float* bias,
                                     int64_t M, int64_t N, int64_t K, frt_act act,
                                     int64_t act_cols, void* out, int64_t ldo, int* dev_status,
                                     frt_stream_t stream) {
  using namespace frt;
  if (!a_q || !a_sf || !w_packed || !w_sf || !out) return FRT_ERR_INVALID_ARG;
  if (act != FRT_ACT_NONE && act != FRT_ACT_GELU_TANH) return FRT_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || lda < K / 2 || ldo < N) return FRT_ERR_INVALID_ARG;
  if (act == FRT_ACT_GELU_TANH && (act_cols < 0 || act_cols > N)) return FRT_ERR_INVALID_ARG;
  if (K % 256 != 0 || N % 16 != 0) return FRT_ERR_UNSUPPORTED_SHAPE;
  if (M > (1LL << 31) - 1 || N > (1LL << 31) - 1 || K > (1LL << 31) - 1 ||
      ldo > (1LL << 31) - 1)
    return FRT_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(a_q, 16) || lda % 16 != 0 || !aligned(a_sf, 16) || !aligned(w_packed, 16) ||
      !aligned(w_sf, 16) || !aligned(out, 16) || ldo % 8 != 0 ||
      (a_scale && !aligned(a_scale, 4)) || (w_scale && !aligned(w_scale, 4)) ||
      (bias && !aligned(bias, 4)) || (dev_status && !aligned(dev_status, 4)))
    return FRT_ERR_MISALIGNED;
  auto encode = tensor_map_encoder();
  if (!encode) return FRT_ERR_CUDA;
  CUtensorMap ta, to;
  {
    // the codes as bytes [M x K/2], one box = 128 rows x 128 bytes (256
    // elements), 128-byte swizzle, zero fill past M
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lda)};
    const cuuint32_t box[2] = {128u, 128u};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a_q), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FRT_ERR_CUDA;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldo * 2)};
    const cuuint32_t box[2] = {32u, 32u};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FRT_ERR_CUDA;
  }
  NvGemmArgs ga;
  ga.a_sf = a_sf;
  ga.w_packed = static_cast<const uint8_t*>(w_packed);
  ga.w_sf = w_sf;
  ga.a_scale = a_scale;
  ga.w_scale = w_scale;
  ga.bias = bias;
  ga.M = static_cast<int>(M);
  ga.N = static_cast<int>(N);
  ga.act_cols = act == FRT_ACT_GELU_TANH ? static_cast<int>(act_cols) : 0;
  ga.kb_total = static_cast<int>(K / 256);
  ga.kc_total = static_cast<int>(K / 64);
  ga.tiles_m = static_cast<int>(ceil_div(M, kNvTile));
  ga.dev_status = dev_status;
  const int sms = sm_count() > 0 ? sm_count() : 148;
  cudaError_t e = cudaSuccess;
  if (M <= kNvTile) {
    ga.num_tiles = static_cast<int>(ga.tiles_m * ceil_div(N, kNvTile));
    e = launch_nvfp4(ta, to, ga, sms, as_cuda(stream));
  } else {
    // 256-row tiles on CTA pairs.  The weight codes as packed k-tiles
    // [tile][128 rows][128 bytes] (stored in their shared-memory image: no
    // swizzle), one box = the half of a tile's channels that one CTA holds;
    // the scales as lines of 256 bytes, one box = the four 512-byte atoms of
    // a k-block (zero fill past the last 128-row group)
    const int64_t nb_total = ceil_div(N, kNvTile);
    ga.tiles_m = static_cast<int>(ceil_div(M, 2 * kNvTile));
    CUtensorMap tw, tsa, tsb;
    const cuuint64_t wdims[3] = {128u, static_cast<cuuint64_t>(kNvTile),
                                 static_cast<cuuint64_t>(nb_total * ga.kb_total)};
    const cuuint64_t wstr[2] = {128u, static_cast<cuuint64_t>(kNvOpBytes)};
    // 256-channel tiles (one accumulator, twice the MACs per scale copy of
    // A) when they still give every SM pair a tile; else 128-channel tiles
    const bool wide = ga.tiles_m * ceil_div(N, 2 * kNvTile) >= sms / 2;
    const int bn = wide ? 2 * kNvTile : kNvTile;
    const cuuint32_t wbox[3] = {128u, static_cast<cuuint32_t>(bn / 2), 1u};
    const cuuint32_t estr3[3] = {1, 1, 1};
    const cuuint64_t adims[2] = {256u,
                                 static_cast<cuuint64_t>(ceil_div(M, kNvTile) * ga.kc_total * 2)};
    const cuuint64_t bdims[2] = {256u, static_cast<cuuint64_t>(nb_total * ga.kc_total * 2)};
    const cuuint64_t sstr[1] = {256u};
    const cuuint32_t sbox[2] = {256u, 8u};
    const cuuint32_t estr2[2] = {1, 1};
    if (encode(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(w_packed), wdims, wstr,
               wbox, estr3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a_sf), adims, sstr,
               sbox, estr2, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w_sf), bdims, sstr,
               sbox, estr2, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FRT_ERR_CUDA;
    ga.num_tiles = static_cast<int>(ga.tiles_m * ceil_div(N, bn));
    e = wide ? launch_nvfp4_pair<2 * kNvTile>(ta, tw, tsa, tsb, to, ga, sms, as_cuda(stream))
             : launch_nvfp4_pair<kNvTile>(ta, tw, tsa, tsb, to, ga, sms, as_cuda(stream));
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FRT_ERR_CUDA;
  }
  note_launches(1);
  return launch_status();
}
