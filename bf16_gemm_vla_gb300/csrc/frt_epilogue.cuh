// Epilogue pieces shared by the GEMM kernels: the tanh-GELU, the fused
// scale/bias step, bf16 packing, and one warp's bf16 output chunk staged in
// shared memory and written by a TMA tensor store.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "frt_device.cuh"

namespace frt {
namespace {

constexpr int kWarpOutBytes = 2048;  // one warp's bf16 output staging buffer

// tanh-GELU, 0.5 v (1 + tanh(u)) with u = sqrt(2/pi) (v + 0.044715 v^3),
// evaluated through the identity 0.5 (1 + tanh(u)) = 1 / (1 + exp(-2u)):
// the relative error stays near 1e-6 even where 1 + tanh(u) cancels
// (large negative v), and exp(-2u) -> inf gives the limit 0.
__device__ __forceinline__ float gelu_tanh(float v) {
  const float k2 = 1.5957691216057308f;  // 2 sqrt(2 / pi)
  const float t = k2 * fmaf(0.044715f * v, v * v, v);
  return __fdividef(v, 1.0f + __expf(-t));
}

__device__ __forceinline__ float lin(float acc, float cs, float b) { return fmaf(acc, cs, b); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Stages one warp's part of a bf16 output chunk in shared memory and
// writes it with a TMA tensor store (64-byte swizzle, 64-byte rows).
//   large M: 32 rows (the warp's TMEM lanes) x 32 channels; lane = row,
//     v[j] = channel x0 + j; box {32 ch, 32 rows}.
//   small M: kRows activation rows x 32 channels (the warp's lanes); lane =
//     channel x0 + lane, v[j] = row y0 + j; box {32 ch, kRows}.
// Each warp owns two staging buffers and alternates between them; lane 0
// issues the store and keeps the buffer's previous store tracked.
template <bool kSwap, int kRows>
__device__ __forceinline__ void warp_store(const float* v, uint8_t* buf, uint32_t buf_s,
                                           const CUtensorMap* tmap, int x0, int y0, int lane) {
  if (lane == 0) dev::bulk_wait_read<1>();  // this buffer's previous store has read it
  __syncwarp();
  if constexpr (!kSwap) {
    uint8_t* rowp = buf + lane * 64;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 w;
      w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
      w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
      w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
      w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
      *reinterpret_cast<uint4*>(rowp + ((q ^ ((lane >> 1) & 3)) << 4)) = w;
    }
  } else {
    const int cb = lane * 2;  // byte of this channel in a 64-byte row
#pragma unroll
    for (int j = 0; j < kRows; ++j)
      *reinterpret_cast<__nv_bfloat16*>(buf + j * 64 + (((cb >> 4) ^ ((j >> 1) & 3)) << 4) +
                                        (cb & 15)) = __float2bfloat16_rn(v[j]);
  }
  dev::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    dev::tma_store_2d(tmap, buf_s, x0, y0);
    dev::bulk_commit();
  }
}

}  // namespace
}  // namespace frt
