// The decoder block boundary in one kernel ("Real-time VLA inference on AMD
// hardware", section "Fusing the BF16 decoder boundary": the gated residual
// update and the adaptive RMS norm that follows it, once separate small
// kernels repeated through every decoder layer and denoising step, become
// one gate_residual_ada_norm_bf16 launch).  The page names the two steps
// but not the norm's parameters: the style row is read as [scale | shift |
// next gate], each H wide, with normed = rms_norm(r) * (1 + scale) + shift.
//
// Per row m of [M x H], with the style row [scale | shift | next gate]:
//   r        = bf16(fp32(residual + output * gate))   (one fused multiply-add)
//   inv      = 1 / sqrt(mean(r^2) + eps)               (fp32)
//   normed   = bf16(r * inv * (1 + scale) + shift)
//   next     = style's gate third, copied
// residual is updated in place.  One CTA per row: each thread holds 8
// elements per 16-byte vector, the sum of squares is a warp-shuffle and
// shared-memory reduction, and every tensor is read and written once.
#include <cuda_bf16.h>

#include "frt_device.cuh"
#include "frt_host.h"

namespace frt {
namespace {

constexpr int kNormThreads = 128;
constexpr int kNormVecs = 4;  // 16-byte vectors a thread holds (H <= 128 * 8 * 4 = 4096)

__device__ __forceinline__ void bf16x8_to_f32(const uint4& w, float (&f)[8]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(ws[k] << 16);
    f[2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  return make_uint4(f32x2_to_bf16x2(f[0], f[1]), f32x2_to_bf16x2(f[2], f[3]),
                    f32x2_to_bf16x2(f[4], f[5]), f32x2_to_bf16x2(f[6], f[7]));
}

__global__ void __launch_bounds__(kNormThreads) gate_residual_ada_norm_kernel(
    uint4* __restrict__ residual, const uint4* __restrict__ output, const uint4* __restrict__ gate,
    const uint4* __restrict__ style, int hv, float eps, uint4* __restrict__ normed,
    uint4* __restrict__ next_gate) {
  __shared__ float red[kNormThreads / 32];
  dev::grid_dependency_wait();  // every input may come from the previous grid
  dev::grid_launch_dependents();
  const int64_t row = blockIdx.x;
  const int64_t base = row * hv;       // this row's first vector (H / 8 per row)
  const int64_t sbase = row * 3 * hv;  // style row: scale, shift, next gate
  float r[kNormVecs][8];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < kNormVecs; ++i) {
    const int v = threadIdx.x + i * kNormThreads;
    if (v < hv) {
      float a[8], o[8], g[8];
      bf16x8_to_f32(residual[base + v], a);
      bf16x8_to_f32(output[base + v], o);
      bf16x8_to_f32(gate[base + v], g);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        // bf16 to fp32 is exact; the update is rounded to fp32 once, then
        // to bf16
        r[i][k] = __bfloat162float(__float2bfloat16_rn(fmaf(o[k], g[k], a[k])));
        ss = fmaf(r[i][k], r[i][k], ss);
      }
      residual[base + v] = f32_to_bf16x8(r[i]);
      next_gate[base + v] = style[sbase + 2 * hv + v];
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];  // same order in every thread
  const float inv = rsqrtf(tot / static_cast<float>(hv * 8) + eps);
#pragma unroll
  for (int i = 0; i < kNormVecs; ++i) {
    const int v = threadIdx.x + i * kNormThreads;
    if (v < hv) {
      float sc[8], sh[8], y[8];
      bf16x8_to_f32(style[sbase + v], sc);
      bf16x8_to_f32(style[sbase + hv + v], sh);
#pragma unroll
      for (int k = 0; k < 8; ++k) y[k] = fmaf(r[i][k] * inv, 1.0f + sc[k], sh[k]);
      normed[base + v] = f32_to_bf16x8(y);
    }
  }
}

}  // namespace
}  // namespace frt

extern "C" frt_status frt_gate_residual_ada_norm_bf16(void* residual, const void* output,
                                                      const void* gate, const void* style,
                                                      int64_t M, int64_t H, float eps,
                                                      void* normalized, void* next_gate,
                                                      frt_stream_t stream) {
  using namespace frt;
  if (M < 0 || H < 1 || !(eps >= 0.0f)) return FRT_ERR_INVALID_ARG;
  if (H % 8 != 0 || H > kNormThreads * 8 * kNormVecs || M > (1LL << 31) - 1)
    return FRT_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return FRT_OK;  // (empty tensors may have null pointers)
  if (!residual || !output || !gate || !style || !normalized || !next_gate)
    return FRT_ERR_INVALID_ARG;
  if (!aligned(residual, 16) || !aligned(output, 16) || !aligned(gate, 16) ||
      !aligned(style, 16) || !aligned(normalized, 16) || !aligned(next_gate, 16))
    return FRT_ERR_MISALIGNED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(M));
  cfg.blockDim = dim3(kNormThreads);
  cfg.stream = as_cuda(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gate_residual_ada_norm_kernel, static_cast<uint4*>(residual),
                         static_cast<const uint4*>(output), static_cast<const uint4*>(gate),
                         static_cast<const uint4*>(style), static_cast<int>(H / 8), eps,
                         static_cast<uint4*>(normalized),
                         static_cast<uint4*>(next_gate)) != cudaSuccess) {
    cudaGetLastError();
    return FRT_ERR_CUDA;
  }
  note_launches(1);
  return launch_status();
}
