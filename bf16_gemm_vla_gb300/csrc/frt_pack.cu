// Load-time weight packing ("Real-time VLA inference on AMD hardware",
// "Packing around the instruction": the static weights are rearranged once,
// at load, into the layout the matrix instruction reads, and stay at a fixed
// address for graph replay).
//
// The GB300 layout is the shared-memory operand image of the tensor-core
// kernels: W^T (one row of K bytes per output channel) cut into tiles of 128
// channels x 128 bytes of K, tile (nb, kb) at byte (nb * KB + kb) * 16384,
// channel r of the tile at byte r * 128, and the 16-byte chunk c of its K
// bytes stored at chunk position c ^ (r % 8) (the 128-byte swizzle).  One
// pipeline stage of the GEMM then loads a tile with one contiguous bulk copy.
#include <cuda_bf16.h>

#include "frt_host.h"

namespace frt {
namespace {

constexpr int kPackThreads = 256;
constexpr int kRowPitch = 132;  // bytes per staged channel row (odd word count)

// One CTA per packed tile (nb, kb).  Each thread owns a channel r (two
// threads per channel, splitting the K-bytes) and reads W[k, n] along k;
// neighbouring threads read neighbouring n, so global reads coalesce.  The
// tile is staged transposed in shared memory and written out as 16-byte
// chunks in swizzled order.
template <typename Tin, int kEsize>
__global__ void __launch_bounds__(kPackThreads) pack_kernel(const Tin* __restrict__ w, int64_t K,
                                                           int64_t N, int64_t ldw, int kb_total,
                                                           uint8_t* __restrict__ packed) {
  __shared__ __align__(16) uint8_t tile[128 * kRowPitch];
  const int nb = blockIdx.y;
  const int kb = blockIdx.x;
  constexpr int kElems = 128 / kEsize;  // K elements per tile row
  const int r = threadIdx.x & 127;
  const int half = threadIdx.x >> 7;
  const int64_t n = static_cast<int64_t>(nb) * 128 + r;
  const int64_t k0 = static_cast<int64_t>(kb) * kElems;
  for (int e = half * (kElems / 2); e < (half + 1) * (kElems / 2); ++e) {
    const int64_t k = k0 + e;
    const bool valid = n < N && k < K;
    if constexpr (kEsize == 1) {
      const uint8_t v = valid ? static_cast<uint8_t>(w[k * ldw + n]) : 0;
      tile[r * kRowPitch + e] = v;
    } else {
      uint16_t bits = 0;
      if (valid) {
        __nv_bfloat16 b;
        if constexpr (sizeof(Tin) == 4)
          b = __float2bfloat16_rn(static_cast<float>(w[k * ldw + n]));
        else
          b = w[k * ldw + n];
        bits = *reinterpret_cast<const uint16_t*>(&b);
      }
      tile[r * kRowPitch + 2 * e] = static_cast<uint8_t>(bits & 0xFF);
      tile[r * kRowPitch + 2 * e + 1] = static_cast<uint8_t>(bits >> 8);
    }
  }
  __syncthreads();
  uint8_t* dst = packed + (static_cast<size_t>(nb) * kb_total + kb) * 16384;
  for (int ch = threadIdx.x; ch < 128 * 8; ch += kPackThreads) {
    const int rr = ch >> 3;  // channel row
    const int p = ch & 7;    // stored chunk position
    const int c = p ^ (rr & 7);  // logical chunk held there
    const uint32_t* src = reinterpret_cast<const uint32_t*>(tile + rr * kRowPitch + c * 16);
    uint4 v;
    v.x = src[0];
    v.y = src[1];
    v.z = src[2];
    v.w = src[3];
    *reinterpret_cast<uint4*>(dst + rr * 128 + p * 16) = v;
  }
}

}  // namespace
}  // namespace frt

extern "C" size_t frt_packed_weight_bytes(int64_t K, int64_t N, frt_dtype packed_dtype) {
  if (K < 1 || N < 1) return 0;
  int esize;
  if (packed_dtype == FRT_BF16)
    esize = 2;
  else if (packed_dtype == FRT_E4M3_OCP)
    esize = 1;
  else
    return 0;
  return static_cast<size_t>(frt::ceil_div(N, 128) * frt::ceil_div(K * esize, 128)) * 16384;
}

extern "C" frt_status frt_pack_weights(const void* w, frt_dtype w_dtype, int64_t K, int64_t N,
                                       int64_t ldw, frt_dtype packed_dtype, void* packed,
                                       size_t packed_bytes, frt_stream_t stream) {
  using namespace frt;
  if (!w || !packed) return FRT_ERR_INVALID_ARG;
  if (K < 1 || N < 1 || ldw < N) return FRT_ERR_INVALID_ARG;
  const bool to_bf16 = packed_dtype == FRT_BF16 && (w_dtype == FRT_F32 || w_dtype == FRT_BF16);
  const bool to_fp8 = packed_dtype == FRT_E4M3_OCP && w_dtype == FRT_E4M3_OCP;
  if (!to_bf16 && !to_fp8) return FRT_ERR_INVALID_ARG;
  if (K > (1LL << 31) - 1 || N > (1LL << 31) - 1) return FRT_ERR_UNSUPPORTED_SHAPE;
  const size_t need = frt_packed_weight_bytes(K, N, packed_dtype);
  if (packed_bytes < need) return FRT_ERR_WORKSPACE_TOO_SMALL;
  const size_t in_esize = w_dtype == FRT_F32 ? 4 : (w_dtype == FRT_BF16 ? 2 : 1);
  if (!aligned(w, in_esize) || !aligned(packed, 16)) return FRT_ERR_MISALIGNED;
  const int esize = to_bf16 ? 2 : 1;
  const int kb_total = static_cast<int>(ceil_div(K * esize, 128));
  const int nb_total = static_cast<int>(ceil_div(N, 128));
  if (nb_total > 65535) return FRT_ERR_UNSUPPORTED_SHAPE;
  const dim3 grid(kb_total, nb_total);
  cudaStream_t st = as_cuda(stream);
  uint8_t* out = static_cast<uint8_t*>(packed);
  if (to_fp8)
    pack_kernel<uint8_t, 1><<<grid, kPackThreads, 0, st>>>(static_cast<const uint8_t*>(w), K, N,
                                                           ldw, kb_total, out);
  else if (w_dtype == FRT_F32)
    pack_kernel<float, 2><<<grid, kPackThreads, 0, st>>>(static_cast<const float*>(w), K, N, ldw,
                                                         kb_total, out);
  else
    pack_kernel<__nv_bfloat16, 2><<<grid, kPackThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(w), K, N, ldw, kb_total, out);
  note_launches(1);
  return launch_status();
}
