// FP8 (E4M3 x E4M3, tcgen05 kind::f8f6f4) and BF16 (kind::f16) GEMMs with
// the fused per-channel-scale + bias (+ tanh-GELU) epilogue and a bf16 store.
//
// The layer computes out = act(acc * a_scale * w_scale[n] + bias[n]) with
// acc = A[M x K] . W[K x N] in fp32 ("Real-time VLA inference on AMD
// hardware", "Merging gate and up": the bias lives in the GEMM epilogue).
// The pages split the work by row count ("FP8 helps the encoder and hurts
// the decoder"): an encoder GEMM with hundreds of rows is a dense
// contraction, the action decoder's few dozen rows make the GEMM stream its
// weights.  One kernel template serves both on GB300:
//
//   * large M ("normal" tiles): MMA M = 128 activation rows, MMA N = 256
//     output channels;
//   * small M ("swap" tiles): the product is taken transposed,
//     out^T = W^T . A^T, so the MMA's 128 rows cover output channels and
//     the few activation rows become the MMA N dimension (32/64/128).  The
//     weight tile is the operand that streams; every CTA reads 16 KiB
//     contiguous per pipeline stage.
//
// Both operands are K-major with the 128-byte swizzle.  Activations arrive
// by TMA (tensor map, zero fill past M and K); weights are pre-packed into
// the exact shared-memory image (see frt_pack.cu) and arrive by plain bulk
// copies.  Warp roles: warp 0 issues the copies, one thread of warp 1
// issues tcgen05.mma into a TMEM accumulator, warps 2-5 run the epilogue.
//
// When there are fewer output tiles than SMs, K is split across the CTAs of
// a thread-block cluster (grid z = cluster z = splits).  Each CTA writes its
// fp32 partial tile to its own shared memory; after a cluster barrier every
// CTA reduces a slice of the tile over all ranks, in rank order (so the
// result does not depend on timing), and applies the epilogue.  No global
// workspace and no atomics are involved.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "frt_device.cuh"
#include "frt_host.h"

namespace frt {
namespace {

constexpr int kThreads = 192;       // 6 warps: copy, MMA, 4 x epilogue
constexpr int kTile = 128;          // MMA M; channels per packed weight tile
constexpr int kKBytes = 128;        // bytes of K per pipeline stage
constexpr int kWTile = kTile * kKBytes;  // bytes of one packed weight tile
constexpr int kPipeBudget = 196608;      // shared memory for the stages
constexpr int kPitch = 129;         // floats per column of a split-K partial tile
constexpr int kMaxSplits = 8;       // portable cluster size

struct GemmArgs {
  const uint8_t* w_packed;
  const float* a_scale;  // 1 float or null (= 1)
  const float* w_scale;  // N floats or null (= 1)
  const float* bias;     // N floats or null (= 0)
  __nv_bfloat16* out;
  int64_t ldo;
  int M, N;
  int act_cols;
  int kb_total;  // 128-byte K blocks of the packed weight
  int nb_total;  // 128-channel groups of the packed weight
  int kb_per_split;
  int splits;
  int* dev_status;
};

template <bool kSwap, int kBN>
struct Cfg {
  static constexpr int kActRows = kSwap ? kBN : kTile;
  static constexpr int kWRows = kSwap ? kTile : kBN;
  static constexpr int kActBytes = kActRows * kKBytes;
  static constexpr int kWBytes = kWRows * kKBytes;
  static constexpr int kStageBytes = kActBytes + kWBytes;
  static constexpr int kStages = (kPipeBudget / kStageBytes) > 8 ? 8 : (kPipeBudget / kStageBytes);
  static constexpr int kPipeBytes = kStages * kStageBytes;
  static constexpr int kTmemCols = kBN;
  static constexpr int kPartialBytes = kBN * kPitch * 4;
  static constexpr int kSmemBytes = 1024 + kPipeBytes + 256;
  static_assert(kActBytes % 1024 == 0 && kWBytes % 1024 == 0, "operand tiles 1024-aligned");
  static_assert(kPartialBytes <= kPipeBytes, "partial tile fits in the stage buffers");
  static_assert(kBN == 32 || kBN == 64 || kBN == 128 || kBN == 256, "TMEM columns");
  static_assert(kStages >= 2, "pipeline depth");
};

__device__ __forceinline__ float gelu_tanh(float v) {
  const float k0 = 0.7978845608028654f;  // sqrt(2 / pi)
  const float u = k0 * (v + 0.044715f * v * v * v);
  return 0.5f * v * (1.0f + tanhf(u));
}

__device__ __forceinline__ float epi(float acc, float cs, float b, bool act) {
  const float v = fmaf(acc, cs, b);
  return act ? gelu_tanh(v) : v;
}

template <bool kFp8, bool kSwap, int kBN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_act, const GemmArgs p) {
  using C = Cfg<kSwap, kBN>;
  constexpr int kStages = C::kStages;
  constexpr int kEsize = kFp8 ? 1 : 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = dev::smem_u32(base);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kPipeBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t full0 = dev::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kStages;
  const uint32_t accum_bar = full0 + 16 * kStages;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      dev::mbar_init(full0 + 8 * s, 1);
      dev::mbar_init(empty0 + 8 * s, 1);
    }
    dev::mbar_init(accum_bar, 1);
    *abort_flag = 0;
    dev::fence_mbar_init();
    dev::prefetch_tmap(&tmap_act);
  }
  if (warp == 1) dev::tmem_alloc(dev::smem_u32(tmem_slot), C::kTmemCols);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int split = blockIdx.z;
  const int kb0 = split * p.kb_per_split;
  const int nkb = min(p.kb_per_split, p.kb_total - kb0);
  const int tile_n = blockIdx.x;
  const int tile_m = blockIdx.y;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- copies
    const uint64_t pol_w = dev::policy_evict_first();
    const uint64_t pol_a = dev::policy_evict_last();
    const int act_row0 = tile_m * C::kActRows;
    const int nb_first = kSwap ? tile_n : tile_n * (kBN / kTile);
    const int groups = kSwap ? 1 : min(kBN / kTile, p.nb_total - nb_first);
    const uint32_t tx = C::kActBytes + groups * kWTile;
    int issued = 0;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      if (!dev::mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, p.dev_status,
                          dev::kTimeoutProducer))
        break;
      const uint32_t st = sbase + s * C::kStageBytes;
      dev::mbar_arrive_expect_tx(full0 + 8 * s, tx);
      const int kb = kb0 + i;
      dev::tma_load_2d(st, &tmap_act, kb * (kKBytes / kEsize), act_row0, full0 + 8 * s, pol_a);
      for (int g = 0; g < groups; ++g) {
        const uint8_t* src =
            p.w_packed + (static_cast<size_t>(nb_first + g) * p.kb_total + kb) * kWTile;
        dev::bulk_load(st + C::kActBytes + g * kWTile, src, kWTile, full0 + 8 * s, pol_w);
      }
      issued = i + 1;
    }
    // Do not leave with copies in flight: wait (bounded, even after an
    // abort) for the last use of every stage that was armed.
    for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i) {
      const int s = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      dev::mbar_wait(full0 + 8 * s, ph, nullptr, p.dev_status, dev::kTimeoutProducer);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA
    constexpr uint32_t idesc = dev::instr_desc(kFp8, kTile, kBN);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      if (!dev::mbar_wait(full0 + 8 * s, ph, abort_flag, p.dev_status, dev::kTimeoutMma)) break;
      dev::tc_fence_after();
      const uint32_t st = sbase + s * C::kStageBytes;
      const uint32_t a_addr = kSwap ? st + C::kActBytes : st;
      const uint32_t b_addr = kSwap ? st : st + C::kActBytes;
      const uint64_t ad = dev::smem_desc_sw128(a_addr);
      const uint64_t bd = dev::smem_desc_sw128(b_addr);
#pragma unroll
      for (int k = 0; k < kKBytes / 32; ++k)
        dev::mma<kFp8>(tmem, ad + 2 * k, bd + 2 * k, idesc, (i | k) != 0);
      dev::mma_commit(empty0 + 8 * s);
    }
    dev::mma_commit(accum_bar);
  }

  // -------------------------------------------------------------------- epilogue
  float* part = reinterpret_cast<float*>(base);  // split-K partial tile [col][lane]
  bool ok = true;
  const int ew = warp & 3;         // TMEM lane quarter of this warp
  const int row = ew * 32 + lane;  // TMEM lane = tile row
  if (warp >= 2) {
    ok = dev::mbar_wait(accum_bar, 0, abort_flag, p.dev_status, dev::kTimeoutEpilogue);
    ok = __all_sync(0xffffffffu, ok);
    dev::tc_fence_after();
    const uint32_t taddr = tmem + (static_cast<uint32_t>(ew * 32) << 16);
    if (p.splits == 1) {
      const float as = p.a_scale ? __ldg(p.a_scale) : 1.0f;
      if constexpr (kSwap) {
        const int n = tile_n * kTile + row;
        const bool nvalid = ok && n < p.N;
        float cs = 1.0f, b = 0.0f;
        bool act = false;
        if (nvalid) {
          cs = as * (p.w_scale ? __ldg(p.w_scale + n) : 1.0f);
          b = p.bias ? __ldg(p.bias + n) : 0.0f;
          act = n < p.act_cols;
        }
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          float v[32];
          dev::tmem_ld32(taddr + c * 32, v);
          const int m0 = tile_m * kBN + c * 32;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int m = m0 + j;
            if (nvalid && m < p.M)
              p.out[static_cast<int64_t>(m) * p.ldo + n] = __float2bfloat16_rn(epi(v[j], cs, b, act));
          }
        }
      } else {
        const int m = tile_m * kTile + row;
        const bool mvalid = ok && m < p.M;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          float v[32];
          dev::tmem_ld32(taddr + c * 32, v);
          if (!mvalid) continue;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int n = tile_n * kBN + c * 32 + q * 8;
            if (n >= p.N) continue;
            __align__(16) __nv_bfloat16 o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float cs = as * (p.w_scale ? __ldg(p.w_scale + n + e) : 1.0f);
              const float b = p.bias ? __ldg(p.bias + n + e) : 0.0f;
              o[e] = __float2bfloat16_rn(epi(v[q * 8 + e], cs, b, n + e < p.act_cols));
            }
            *reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(m) * p.ldo + n) =
                *reinterpret_cast<const uint4*>(o);
          }
        }
      }
    } else {
      // split-K: this CTA's fp32 partial tile -> own shared memory, [col][lane]
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        float v[32];
        dev::tmem_ld32(taddr + c * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) part[(c * 32 + j) * kPitch + row] = v[j];
      }
    }
  }

  __syncwarp();
  if (p.splits > 1) {
    dev::cluster_sync();  // every partial tile of the cluster is written
    if (warp >= 2) {
      const uint32_t rank = dev::cluster_ctarank();
      const int S = p.splits;
      const float as = p.a_scale ? __ldg(p.a_scale) : 1.0f;
      const uint32_t part_s = dev::smem_u32(part);
      if constexpr (kSwap) {
        // columns = activation rows m; each CTA reduces a slice of them
        const int cpr = (kBN + S - 1) / S;
        const int c0 = rank * cpr;
        const int c1 = min(kBN, c0 + cpr);
        const int n = tile_n * kTile + row;
        const bool nvalid = ok && n < p.N;
        float cs = 1.0f, b = 0.0f;
        bool act = false;
        if (nvalid) {
          cs = as * (p.w_scale ? __ldg(p.w_scale + n) : 1.0f);
          b = p.bias ? __ldg(p.bias + n) : 0.0f;
          act = n < p.act_cols;
        }
        for (int c = c0; c < c1; ++c) {
          const int m = tile_m * kBN + c;
          if (!nvalid || m >= p.M) continue;
          const uint32_t off = part_s + static_cast<uint32_t>((c * kPitch + row) * 4);
          float acc = 0.0f;
          for (int s = 0; s < S; ++s) acc += dev::ld_dsmem_f32(dev::map_to_rank(off, s));
          p.out[static_cast<int64_t>(m) * p.ldo + n] = __float2bfloat16_rn(epi(acc, cs, b, act));
        }
      } else {
        // lanes = activation rows m; each CTA reduces a slice of rows, its
        // 128 epilogue threads walk the columns (coalesced stores)
        const int t = threadIdx.x - 64;
        const int rpr = (kTile + S - 1) / S;
        const int r0 = rank * rpr;
        const int r1 = min(kTile, r0 + rpr);
        for (int r = r0; r < r1; ++r) {
          const int m = tile_m * kTile + r;
          if (!ok || m >= p.M) break;
          for (int c = t; c < kBN; c += 128) {
            const int n = tile_n * kBN + c;
            if (n >= p.N) continue;
            const uint32_t off = part_s + static_cast<uint32_t>((c * kPitch + r) * 4);
            float acc = 0.0f;
            for (int s = 0; s < S; ++s) acc += dev::ld_dsmem_f32(dev::map_to_rank(off, s));
            const float cs = as * (p.w_scale ? __ldg(p.w_scale + n) : 1.0f);
            const float b = p.bias ? __ldg(p.bias + n) : 0.0f;
            p.out[static_cast<int64_t>(m) * p.ldo + n] =
                __float2bfloat16_rn(epi(acc, cs, b, n < p.act_cols));
          }
        }
      }
    }
    dev::cluster_sync();  // no CTA leaves while a peer still reads its tile
  }

  dev::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

struct Plan {
  bool swap;
  int bn;
  int splits;
  int kb_per_split;
  dim3 grid;
};

Plan make_plan(int64_t M, int64_t N, int64_t K, int esize) {
  Plan pl;
  const int kb = static_cast<int>(ceil_div(K * esize, kKBytes));
  const int nb = static_cast<int>(ceil_div(N, kTile));
  int tiles;
  if (M <= 128) {
    pl.swap = true;
    pl.bn = M <= 32 ? 32 : (M <= 64 ? 64 : 128);
    tiles = nb * static_cast<int>(ceil_div(M, pl.bn));
  } else {
    pl.swap = false;
    pl.bn = 256;
    tiles = static_cast<int>(ceil_div(N, 256) * ceil_div(M, kTile));
  }
  const int sms = sm_count() > 0 ? sm_count() : 148;
  int s = 1;
  if (tiles < sms) {
    s = sms / tiles;
    if (s > kMaxSplits) s = kMaxSplits;
    if (s > kb) s = kb;
    if (s < 1) s = 1;
  }
  pl.kb_per_split = static_cast<int>(ceil_div(kb, s));
  pl.splits = static_cast<int>(ceil_div(kb, pl.kb_per_split));
  if (pl.swap)
    pl.grid = dim3(nb, static_cast<unsigned>(ceil_div(M, pl.bn)), pl.splits);
  else
    pl.grid = dim3(static_cast<unsigned>(ceil_div(N, 256)), static_cast<unsigned>(ceil_div(M, kTile)),
                   pl.splits);
  return pl;
}

template <bool kFp8, bool kSwap, int kBN>
cudaError_t launch_one(const CUtensorMap& tm, const GemmArgs& a, const Plan& pl,
                       cudaStream_t stream) {
  using C = Cfg<kSwap, kBN>;
  auto kern = gemm_tc_kernel<kFp8, kSwap, kBN>;
  static std::mutex mu;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
      cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = pl.grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = pl.splits;
  cfg.attrs = attr;
  cfg.numAttrs = pl.splits > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tm, a);
}

template <bool kFp8>
cudaError_t dispatch(const CUtensorMap& tm, const GemmArgs& a, const Plan& pl,
                     cudaStream_t stream) {
  if (!pl.swap) return launch_one<kFp8, false, 256>(tm, a, pl, stream);
  switch (pl.bn) {
    case 32: return launch_one<kFp8, true, 32>(tm, a, pl, stream);
    case 64: return launch_one<kFp8, true, 64>(tm, a, pl, stream);
    default: return launch_one<kFp8, true, 128>(tm, a, pl, stream);
  }
}

frt_status gemm_common(bool fp8, const void* a, int64_t lda, const float* a_scale,
                       const void* w_packed, const float* w_scale, const float* bias, int64_t M,
                       int64_t N, int64_t K, frt_act act, int64_t act_cols, void* out,
                       int64_t ldo, int* dev_status, frt_stream_t stream) {
  const int esize = fp8 ? 1 : 2;
  if (!a || !w_packed || !out) return FRT_ERR_INVALID_ARG;
  if (fp8 && (!a_scale || !w_scale)) return FRT_ERR_INVALID_ARG;
  if (act != FRT_ACT_NONE && act != FRT_ACT_GELU_TANH) return FRT_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return FRT_ERR_INVALID_ARG;
  if (act == FRT_ACT_GELU_TANH && (act_cols < 0 || act_cols > N)) return FRT_ERR_INVALID_ARG;
  if (lda < K || ldo < N) return FRT_ERR_INVALID_ARG;
  if (N % 16 != 0 || K % (fp8 ? 32 : 16) != 0) return FRT_ERR_UNSUPPORTED_SHAPE;
  if (M > (1LL << 31) - 1 || N > (1LL << 31) - 1 || K > (1LL << 31) - 1)
    return FRT_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(a, 16) || (lda * esize) % 16 != 0 || !aligned(w_packed, 16) ||
      !aligned(out, 16) || ldo % 8 != 0)
    return FRT_ERR_MISALIGNED;
  if ((a_scale && !aligned(a_scale, 4)) || (w_scale && !aligned(w_scale, 4)) ||
      (bias && !aligned(bias, 4)) || (dev_status && !aligned(dev_status, 4)))
    return FRT_ERR_MISALIGNED;

  auto encode = tensor_map_encoder();
  if (!encode) return FRT_ERR_CUDA;
  const Plan pl = make_plan(M, N, K, esize);

  CUtensorMap tm;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lda * esize)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKBytes / esize),
                             static_cast<cuuint32_t>(pl.swap ? pl.bn : kTile)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(&tm, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      2, const_cast<void*>(a), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return FRT_ERR_CUDA;

  GemmArgs ga;
  ga.w_packed = static_cast<const uint8_t*>(w_packed);
  ga.a_scale = a_scale;
  ga.w_scale = w_scale;
  ga.bias = bias;
  ga.out = static_cast<__nv_bfloat16*>(out);
  ga.ldo = ldo;
  ga.M = static_cast<int>(M);
  ga.N = static_cast<int>(N);
  ga.act_cols = act == FRT_ACT_GELU_TANH ? static_cast<int>(act_cols) : 0;
  ga.kb_total = static_cast<int>(ceil_div(K * esize, kKBytes));
  ga.nb_total = static_cast<int>(ceil_div(N, kTile));
  ga.kb_per_split = pl.kb_per_split;
  ga.splits = pl.splits;
  ga.dev_status = dev_status;

  cudaError_t e = fp8 ? dispatch<true>(tm, ga, pl, as_cuda(stream))
                      : dispatch<false>(tm, ga, pl, as_cuda(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FRT_ERR_CUDA;
  }
  return launch_status();
}

}  // namespace
}  // namespace frt

extern "C" size_t frt_gemm_workspace_bytes(int64_t, int64_t, int64_t, frt_dtype) { return 0; }

extern "C" frt_status frt_gemm_fp8(const uint8_t* a_q, int64_t lda, const float* a_scale,
                                   const void* w_packed, const float* w_scale, const float* bias,
                                   int64_t M, int64_t N, int64_t K, frt_act act, int64_t act_cols,
                                   void* out, int64_t ldo, void* /*workspace*/,
                                   size_t /*workspace_bytes*/, int* dev_status,
                                   frt_stream_t stream) {
  return frt::gemm_common(true, a_q, lda, a_scale, w_packed, w_scale, bias, M, N, K, act,
                          act_cols, out, ldo, dev_status, stream);
}

extern "C" frt_status frt_gemm_bf16(const void* a, int64_t lda, const void* w_packed,
                                    const float* w_scale, const float* bias, int64_t M, int64_t N,
                                    int64_t K, frt_act act, int64_t act_cols, void* out,
                                    int64_t ldo, void* /*workspace*/, size_t /*workspace_bytes*/,
                                    int* dev_status, frt_stream_t stream) {
  return frt::gemm_common(false, a, lda, nullptr, w_packed, w_scale, bias, M, N, K, act, act_cols,
                          out, ldo, dev_status, stream);
}
