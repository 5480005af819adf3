// FP8 (E4M3 x E4M3, tcgen05 kind::f8f6f4) and BF16 (kind::f16) GEMMs with
// the fused per-channel-scale + bias (+ tanh-GELU, or the GeGLU of a merged
// gate/up) epilogue and a bf16 store.
//
// The layer computes out = act(acc * a_scale * w_scale[n] + bias[n]) with
// acc = A[M x K] . W[K x N] in fp32 ("Real-time VLA inference on AMD
// hardware", "Merging gate and up": the bias lives in the GEMM epilogue).
// The pages split the work by row count ("FP8 helps the encoder and hurts
// the decoder"): an encoder GEMM with hundreds of rows is a dense
// contraction, the action decoder's few dozen rows make the GEMM stream its
// weights.  One kernel template serves both on GB300:
//
//   * large M: 256-row tiles on CTA pairs (cta_group::2).  The two CTAs of a
//     cluster whose ranks differ in bit 0 each hold 128 activation rows and
//     half of the tile's 256 (or 128) output channels per k-block; the even
//     CTA issues one tcgen05.mma with M = 256 that reads both CTAs' shared
//     memory and writes each CTA's 128 accumulator rows into its own TMEM.
//     Per k-block a CTA ingests 32 KiB for 128 x 256 x 128 MACs instead of
//     48 KiB for a single-CTA 128 x 256 tile.
//   * small M ("swap" tiles): the product is taken transposed,
//     out^T = W^T . A^T, so the MMA's 128 rows cover output channels and
//     the few activation rows become the MMA N dimension (32/64/128).  The
//     weight tile is the operand that streams; a pipeline stage reads one
//     or two contiguous packed 16 KiB k-tiles of a channel group.
//
// Both operands are K-major with the 128-byte swizzle.  Activations arrive
// by TMA (zero fill past M and K); weights are pre-packed into the exact
// shared-memory image (frt_pack.cu) and arrive by bulk copies (single CTA)
// or by TMA over the packed buffer (pairs).  Warp roles: warp 0 issues the
// copies, one thread of warp 1 issues tcgen05.mma into TMEM, warps 2-5 run
// the epilogue (large M: bf16 staged in swizzled shared memory and written
// by TMA tensor stores; small M: each warp's rows staged in shared memory and
// written by 16-byte stores).
//
// Scheduling:
//   * without split-K the grid is persistent (one CTA, or pair, per SM walks
//     a strided tile list) and the TMEM accumulator is double-buffered, so a
//     tile's epilogue overlaps the next tile's mainloop;
//   * when there are fewer output tiles than SMs, K is split.  The tile's
//     columns are cut into chunks, each owned by one split; the other splits
//     hand their partial chunks to the owner -- inside a thread-block
//     cluster through shared memory (small M; large M without a workspace),
//     or through a caller workspace in global memory (pairs) -- and the
//     owner adds the partial sums in split order, a fixed order, so the
//     result does not depend on timing.
//
// With programmatic dependent launch, the first pipeline stages' weight
// tiles (static data) are fetched before the kernel waits for the previous
// grid; activations and the activation scale are read only after the wait
// (the copy warp reads the scale there and hands it to the epilogue through
// shared memory, so no epilogue waits on an L2 round trip).
//
// GeGLU (merged gate/up, gate channels first): a pair tile's CTAs hold the
// gate group and the matching up group of 128 outputs; a small-M tile's 128
// weight rows are 64 gate and the 64 matching up channels, and the up lanes
// hand their values to the gate lanes through shared memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "frt_device.cuh"
#include "frt_e4m3.cuh"
#include "frt_epilogue.cuh"
#include "frt_host.h"
#include "frt_tma_host.h"

namespace frt {
namespace {

constexpr int kThreads = 192;            // 6 warps: copy, MMA, 4 x epilogue
constexpr int kTile = 128;               // MMA M; channels per packed weight tile
constexpr int kKBytes = 128;             // bytes of K per pipeline stage
constexpr int kWTile = kTile * kKBytes;  // bytes of one packed weight tile
constexpr int kSmemMax = 232448;         // dynamic shared memory limit per CTA
constexpr int kPairMinSmem = 200 * 1024;  // shared memory floor of a pair CTA
constexpr int kOutBytes = 4 * 2 * kWarpOutBytes;  // 4 epilogue warps x 2 buffers
constexpr int kSwapStoreBytes = 32 * 64;          // small M: a warp's staged bf16 rows
constexpr int kBarRegion = 512;          // mbarriers, TMEM address, abort flag
constexpr int kMaxSplits = 8;            // portable cluster size
constexpr int kMaxStages = 8;
constexpr size_t kNextScaleHeaderBytes = 256;  // arrivals and running max of the next layer's scale

struct GemmArgs {
  const uint8_t* w_packed;
  const float* a_scale;  // 1 float or null (= 1)
  const float* w_scale;  // N floats or null (= 1)
  const float* bias;     // N floats or null (= 0)
  int M, N;
  int act_cols;
  // merged gate/up GEMM with the GeGLU fused: the output is gelu(gate) *
  // up.  Pairs (256-wide tiles): the tile's CTAs hold gate channel group tn
  // and up group f_groups + tn, 128 outputs per tile.  Small M: a tile's
  // 128 weight rows are 64 gate channels (64 tn ..) and the 64 up channels
  // of the same outputs, 64 outputs per tile.
  int geglu;
  int f_groups;  // F / 128, F = N / 2
  int kb_total;  // 128-byte K blocks of the packed weight
  int nb_total;  // 128-channel groups of the packed weight
  int kb_per_split;
  int splits;
  int tiles_m, tiles_n, num_tiles;
  int stages;          // pipeline depth
  int kbs;             // 128-byte k-blocks per pipeline stage (pairs: 2 when K allows)
  int chunk_cols;      // split-K: TMEM columns per chunk (32 large M, 8 small M)
  int recv_in_stages;  // split-K: receive buffers reuse the stage buffers
  int outbuf_off;      // shared-memory layout (bytes from the 1024-aligned base)
  int recv_off;
  int tail_off;        // per-channel scale/bias, then mbarriers
  int split_global;    // split-K partials exchanged through the workspace (pairs)
  __nv_bfloat16* out;  // small M: output rows written by the epilogue warps
  int ldo;
  float* ws_part;      // split_global: partial chunks, one slot per (tile, CTA, chunk, split)
  unsigned* ws_flag;   // split_global: per (tile, CTA, owner split) arrival counters
  int* dev_status;
  // The next FP8 layer's activation scale, taken from this layer's own bf16
  // output (s_cols 0: not asked for): s = amax / 448 over out[0:M, 0:s_cols]
  // (NaN ignored; 1 if the amax is 0), folded across the CTAs in s_hdr.
  int s_cols;
  float* s_out;    // receives s
  unsigned* s_hdr; // 256-byte header: [0] arrivals, [4] running max (fp32 bits)
};

template <bool kSwap, bool kPair, int kBN>
struct Cfg {
  static constexpr int kActRows = kSwap ? kBN : kTile;
  // a pair's CTAs each hold half of the tile's weight channels
  static constexpr int kWRows = kSwap ? kTile : (kPair ? kBN / 2 : kBN);
  static constexpr int kActBytes = kActRows * kKBytes;
  static constexpr int kWBytes = kWRows * kKBytes;
  static constexpr int kStageBytes = kActBytes + kWBytes;
  // output rows of a large-M tile: 128, or 256 for a CTA pair
  static constexpr int kTileRows = kPair ? 2 * kTile : kTile;
  // two accumulator buffers, so that a tile's epilogue overlaps the next
  // tile's mainloop (a pair's 256-column tiles take all 512 TMEM columns;
  // the host gives such a CTA enough shared memory that no other CTA that
  // allocates TMEM is resident beside it)
  static constexpr int kAccBufs = 2;
  static constexpr int kTmemCols = kAccBufs * kBN;
  static_assert(kActBytes % 1024 == 0 && kWBytes % 1024 == 0, "operand tiles 1024-aligned");
  static_assert(kBN == 32 || kBN == 64 || kBN == 128 || kBN == 256, "tile width");
  static_assert(kSwap || kBN >= 128, "large-M tiles are 128 x 128 or 128 x 256");
  static_assert(!(kSwap && kPair), "CTA pairs take large-M tiles");
};

// Small M: one warp's output rows.  Lane l holds channel n0 + l (n0 a
// multiple of 32) of rows y0 .. y0 + kRows - 1 (v[j] = row y0 + j).  The
// warp's kRows x 32 bf16 values are staged in `sb` (kRows x 64 bytes of
// this warp's shared memory) and written with one 16-byte store per lane and
// 8 rows (N and ldo are multiples of 8 and the output is 16-byte aligned, so
// a group of 8 channels is either whole or past N).  Rows >= M and channels
// >= N are not written.
template <int kRows>
__device__ __forceinline__ void store_rows(const float* v, const GemmArgs& p, int y0, int n0,
                                           int lane, __nv_bfloat16* sb) {
  __syncwarp();  // the previous chunk's reads of sb are done
#pragma unroll
  for (int j = 0; j < kRows; ++j) sb[j * 32 + lane] = __float2bfloat16_rn(v[j]);
  __syncwarp();
  const int seg = lane & 3;
  const int n = n0 + seg * 8;
#pragma unroll
  for (int r0 = 0; r0 < kRows; r0 += 8) {
    const int r = r0 + (lane >> 2);
    const uint4 w = *reinterpret_cast<const uint4*>(sb + r * 32 + seg * 8);
    if (y0 + r < p.M && n < p.N)
      *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(y0 + r) * p.ldo + n) = w;
  }
}

// Byte offset of float4 granule q of row r in a split-K partial chunk of
// 128 rows x cw floats (cw = 32 or 8); granules are XOR-swizzled by row so
// that row-per-thread reads and writes are free of bank conflicts.
__device__ __forceinline__ uint32_t chunk_off(int r, int q, int cw) {
  const int swz = cw == 32 ? (r & 7) : ((r >> 2) & 1);
  return static_cast<uint32_t>(r * cw * 4 + ((q ^ swz) << 4));
}

// ------------------------------------------------------------------ the next layer's scale
//
// The per-tensor E4M3 scale of the layer's own bf16 output, for the next FP8
// layer, taken in the epilogue instead of by a separate amax pass over the
// stored output: each epilogue thread keeps the running max |bf16(v)| of the
// outputs it stores in the first s_cols columns, each CTA folds its maximum
// into a header word after its last tile and arrives on an arrival count;
// the last CTA to arrive turns the maximum into s = amax / 448 (1 if 0),
// stores it and resets the header.  No CTA waits for another.  The encode
// with s is then the static-scale quantize of the stored output (a light
// pass over the output, which is still in L2).

__device__ __forceinline__ float bf16_round(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// max |x| over the 8 bf16 values of a 16-byte vector and a running bf16x2
// maximum (sign bits cleared; a NaN operand of __hmax2 yields the other
// one, as fmaxf: NaN is ignored).
__device__ __forceinline__ uint32_t max_abs_bf16x8(uint32_t acc, const uint4& w) {
  __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&acc);
  const uint32_t ws[4] = {w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu, w.z & 0x7FFF7FFFu,
                          w.w & 0x7FFF7FFFu};
#pragma unroll
  for (int k = 0; k < 4; ++k) a = __hmax2(a, *reinterpret_cast<const __nv_bfloat162*>(&ws[k]));
  return *reinterpret_cast<const uint32_t*>(&a);
}

// Large M: the running max over this thread's 32 bf16 outputs of row m,
// columns n0 .. n0 + 31 (n0 a multiple of 32; s_cols a multiple of 8), read
// back from the row the thread staged for the TMA store (64 bytes, 16-byte
// chunk c at c ^ sw): the stored values.
__device__ __forceinline__ void amax_row32_staged(const GemmArgs& p, float& amax,
                                                  const uint8_t* rowp, int sw, int m, int n0) {
  if (m >= p.M || n0 >= p.s_cols) return;
  const int nc = min(4, (p.s_cols - n0) >> 3);  // 8-column vectors inside s_cols
  uint32_t m2 = 0u;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (c < nc) m2 = max_abs_bf16x8(m2, *reinterpret_cast<const uint4*>(rowp + ((c ^ sw) << 4)));
  amax = fmaxf(amax, fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u)));
}

// Small M: the running max over the bf16 outputs of channel n for rows
// y0 .. y0 + kRows - 1.
template <int kRows>
__device__ __forceinline__ void amax_col(const GemmArgs& p, float& amax, const float* v, int y0,
                                         int n) {
  if (n >= p.s_cols) return;
#pragma unroll
  for (int j = 0; j < kRows; ++j)
    if (y0 + j < p.M) amax = fmaxf(amax, fabsf(bf16_round(v[j])));
}

// One thread per CTA, after the CTA's last output: folds the CTA's maximum m
// into the header and arrives; the last arrival stores s and resets the
// header for the next call.
__device__ __noinline__ void next_scale_arrive(const GemmArgs& p, float m) {
  unsigned* hdr = p.s_hdr;
  const unsigned nct = gridDim.x * gridDim.y * gridDim.z;
  // the header's previous user (an earlier grid on the stream) has completed
  dev::grid_dependency_wait();
  // m >= 0 and never NaN: its bits order as its value.  The running maximum
  // only grows within a call, so a CTA whose maximum is not above the value
  // it reads skips the atomic (fewer operations on the contended line).
  if (__uint_as_float(ld_relaxed_gpu(hdr + 4)) < m) atomicMax(hdr + 4, __float_as_uint(m));
  // the arrival releases this CTA's maximum; the last one acquires them all
  if (atom_add_acq_rel_gpu(hdr, 1u) == nct - 1) {
    const float a = __uint_as_float(ld_relaxed_gpu(hdr + 4));
    hdr[4] = 0u;
    hdr[0] = 0u;
    *p.s_out = a == 0.0f ? 1.0f : __fdiv_rn(a, 448.0f);
  }
}

template <bool kFp8, bool kSwap, bool kPair, int kBN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_act,
                   const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_out, const GemmArgs p) {
  using C = Cfg<kSwap, kPair, kBN>;
  constexpr int kEsize = kFp8 ? 1 : 2;
  const int stages = p.stages;
  // a stage holds kbs k-blocks: the activation tiles, then the weight tiles
  const int kbs = (kPair || kSwap) ? p.kbs : 1;
  const uint32_t act_bytes = static_cast<uint32_t>(kbs * C::kActBytes);
  const uint32_t stage_bytes = static_cast<uint32_t>(kbs * C::kStageBytes);
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, by pointer arithmetic on the shared array so
  // that accesses through it stay shared-memory loads and stores
  uint8_t* base = smem_raw + ((1024u - (dev::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = dev::smem_u32(base);
  float* col_sb = reinterpret_cast<float*>(base + p.tail_off);  // [2 bufs][scale, bias][kBN]
  uint64_t* bars = reinterpret_cast<uint64_t*>(col_sb + 4 * kBN);
  const uint32_t full0 = dev::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * stages;
  const uint32_t tfull0 = empty0 + 8 * stages;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t recv_bar = tempty0 + 16;
  const uint32_t scale_bar = recv_bar + 8;  // the activation scale is in a_scale_s
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * stages + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* a_scale_s = reinterpret_cast<float*>(tmem_slot + 2);
  float* amax_red = a_scale_s + 1;  // the epilogue warps' output maxima (next layer's scale)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool split = p.splits > 1;
  const int S = p.splits;
  // split-K partials meet in the workspace (global split; pairs only) or in
  // the shared memory of one cluster (cluster split)
  const bool gsplit = kPair && split && p.split_global;
  const bool csplit = split && !gsplit;
  // cluster layout: a pair's two CTAs along x, cluster-split ranks along z
  const uint32_t crank = (kPair || split) ? dev::cluster_ctarank() : 0u;
  const int px = kPair ? static_cast<int>(crank & 1u) : 0;  // CTA within the pair
  const int rank = gsplit ? static_cast<int>(blockIdx.z)
                          : (kPair ? static_cast<int>(crank >> 1) : static_cast<int>(crank));
  const bool leader = px == 0;  // issues the pair's MMAs
  const uint32_t lead_rank = crank & ~1u;
  // A pair without a cluster split meets once more before it frees TMEM.
  // Each warp arrives on that barrier as soon as it is done with everything
  // that crosses to the other CTA (the copy warp after its drain, the MMA
  // warp after its last commit, the epilogue after the last accumulator is
  // ready), all lanes together, and waits at the very end.  The arrivals
  // carry no memory ordering: the data that crosses was already ordered by
  // the mbarriers; this barrier only keeps either CTA from leaving early.
  const bool early_bye = kPair && !csplit;
  // cluster rank of the CTA that holds K split j of this CTA's rows
  auto split_cta = [&](int j) -> uint32_t {
    return kPair ? static_cast<uint32_t>(2 * j + px) : static_cast<uint32_t>(j);
  };

  // split-K chunks: chunk_cols TMEM columns each; rank j owns chunks
  // [cb(j), cb(j+1)) with cb(j) = ceil(j * NC / S)
  const int CW = p.chunk_cols;
  const int NC = split ? kBN / CW : 1;
  auto chunk_begin = [&](int j) { return (j * NC + S - 1) / S; };
  const int owned_max = split ? (NC + S - 1) / S : 0;
  const uint32_t chunk_bytes = static_cast<uint32_t>(kTile * CW * 4);
  const int own_c0 = split ? chunk_begin(rank) : 0;
  const int own_c1 = split ? chunk_begin(rank + 1) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      dev::mbar_init(full0 + 8 * s, 1);
      dev::mbar_init(empty0 + 8 * s, 1);
    }
    dev::mbar_init(tfull0, 1);
    dev::mbar_init(tfull0 + 8, 1);
    // accumulator released by every epilogue warp (of both CTAs of a pair)
    dev::mbar_init(tempty0, kPair ? 8 : 4);
    dev::mbar_init(tempty0 + 8, kPair ? 8 : 4);
    dev::mbar_init(recv_bar, 1);
    dev::mbar_init(scale_bar, 1);
    *abort_flag = 0;
    dev::fence_mbar_init();
    if (csplit)  // bytes this CTA receives: its own chunks from every peer
      dev::mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(S - 1) *
                                               static_cast<uint32_t>(own_c1 - own_c0) *
                                               chunk_bytes);
    dev::prefetch_tmap(&tmap_act);
    if (kPair) dev::prefetch_tmap(&tmap_w);
    dev::prefetch_tmap(&tmap_out);
  }
  if (warp == 1) {
    if constexpr (kPair)
      dev::tmem_alloc_pair(dev::smem_u32(tmem_slot), C::kTmemCols);
    else
      dev::tmem_alloc(dev::smem_u32(tmem_slot), C::kTmemCols);
  }
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the next grid on the stream may start its prologue (it waits for this
  // grid's completion before it reads or writes anything this grid touches)
  dev::grid_launch_dependents();
  // a pair signals mbarriers across its two CTAs from the first copy on:
  // both CTAs' barriers are initialised before either goes on.  (Every
  // cluster-barrier arrive and wait in this kernel is executed by all 32
  // lanes of a warp together.)
  if constexpr (kPair) {
    // the initialisation is published by fence.mbarrier_init (a release);
    // the arrival itself needs no ordering
    dev::cluster_arrive_relaxed();
    dev::cluster_wait();
  }
  // Split-K cluster barrier, phase 1: with dedicated receive buffers every
  // thread arrives now (its mbarriers are initialised); when the receive
  // buffers reuse the stage buffers, each thread arrives once this CTA's
  // MMAs can no longer read them.
  if (csplit && !p.recv_in_stages) dev::cluster_arrive_relaxed();

  // this CTA's tiles: split -> one tile and a K range; else a strided list
  // (a pair walks its list together)
  const int kb0 = split ? rank * p.kb_per_split : 0;
  const int nkb = split ? min(p.kb_per_split, p.kb_total - kb0) : p.kb_total;
  const int first_tile = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int t_step = split ? p.num_tiles : static_cast<int>(kPair ? gridDim.x >> 1 : gridDim.x);
  const int my_tiles = split ? 1 : (p.num_tiles - first_tile + t_step - 1) / t_step;
  auto tile_of = [&](int it, int& tm, int& tn) {
    const int t = first_tile + it * t_step;
    if (kSwap) {
      tn = t % p.tiles_n;
      tm = t / p.tiles_n;
    } else {  // rows fastest: the CTAs that share a weight tile run together
      tm = t % p.tiles_m;
      tn = t / p.tiles_m;
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ copies
      const uint64_t pol_w = kSwap ? dev::policy_evict_first() : dev::policy_evict_normal();
      const uint64_t pol_a = dev::policy_evict_last();
      const int units = (nkb + kbs - 1) / kbs;  // stages per tile
      const int total = my_tiles * units;
      // stage cursor: the walk's tile as (x, y), x the fastest coordinate of
      // tile_of, and the stage i within it; advanced without divisions (the
      // copy issue is on the critical path while the pipeline fills)
      struct Cur {
        int i, x, y;
      };
      const int inner = kSwap ? p.tiles_n : p.tiles_m;
      const int step_q = t_step / inner, step_r = t_step % inner;
      const Cur start = {0, first_tile % inner, first_tile / inner};
      auto advance = [&](Cur& c) {
        if (++c.i == units) {
          c.i = 0;
          c.x += step_r;
          c.y += step_q;
          if (c.x >= inner) {
            c.x -= inner;
            ++c.y;
          }
        }
      };
      // geometry of a stage: tile rows, first weight group, groups, tx bytes
      auto geom = [&](const Cur& c, int& tm, int& nbf, int& groups) -> uint32_t {
        tm = kSwap ? c.y : c.x;
        const int tn = kSwap ? c.x : c.y;
        if constexpr (kPair) {
          // 256-channel tiles: one 128-channel group per CTA; 128-channel
          // tiles: one half group per CTA.  Both CTAs' copies complete on
          // the leader's barrier.
          nbf = kBN == 256 ? (p.geglu ? (px ? p.f_groups + tn : tn) : 2 * tn + px) : tn;
          groups = 1;
          return 2u * stage_bytes;  // whole boxes (zero fill counts)
        }
        if constexpr (kSwap) {
          // the channel group's k-tiles of this stage are contiguous; the
          // copy stops at the group's last k-tile
          nbf = tn;
          groups = min(kbs, p.kb_total - (kb0 + c.i * kbs));
          return static_cast<uint32_t>(kbs * C::kActBytes + groups * kWTile);
        }
        nbf = tn * (kBN / kTile);
        groups = min(kBN / kTile, p.nb_total - nbf);
        return static_cast<uint32_t>(C::kActBytes + groups * kWTile);
      };
      // the stage's full barrier: a pair's is the leader's
      auto full_bar = [&](int s) -> uint32_t {
        return kPair ? dev::map_to_rank(full0 + 8 * s, lead_rank) : full0 + 8 * s;
      };
      auto arm = [&](int s, uint32_t tx) {
        if (!kPair || leader) dev::mbar_arrive_expect_tx(full0 + 8 * s, tx);
      };
      auto load_weights = [&](const Cur& c, int s, int nbf, int groups) {
        const uint32_t st = sbase + s * stage_bytes;
        const int kb = kb0 + c.i * kbs;
        if constexpr (kPair) {
          // packed tiles seen as [tile][128 rows][128 bytes]: one box takes
          // this CTA's rows of kbs consecutive k-tiles; tiles past the
          // weight (channels >= N) arrive as zeros
          const int half = kBN == 256 ? 0 : px;
          dev::tma_load_3d_pair(st + act_bytes, &tmap_w, 0, half * (kTile / 2),
                                nbf * p.kb_total + kb, full_bar(s), pol_w);
        } else if constexpr (kSwap) {
          if (p.geglu) {
            // rows 0-63: gate channels 64 nbf .. of the packed group nbf / 2,
            // rows 64-127: the up channels F + 64 nbf ..; a packed tile's rows
            // are 128 bytes, so a half group of one k-tile is 8 KiB (the
            // 128-byte swizzle repeats every 8 rows, so the halves keep it)
            const size_t half = static_cast<size_t>(nbf & 1) * (kWTile / 2);
            for (int q = 0; q < groups; ++q) {
              const uint8_t* sg = p.w_packed +
                                  (static_cast<size_t>(nbf >> 1) * p.kb_total + kb + q) * kWTile +
                                  half;
              const uint8_t* su =
                  p.w_packed +
                  (static_cast<size_t>(p.f_groups + (nbf >> 1)) * p.kb_total + kb + q) * kWTile +
                  half;
              const uint32_t dst = st + act_bytes + q * kWTile;
              dev::bulk_load(dst, sg, kWTile / 2, full0 + 8 * s, pol_w);
              dev::bulk_load(dst + kWTile / 2, su, kWTile / 2, full0 + 8 * s, pol_w);
            }
          } else {
            const uint8_t* src =
                p.w_packed + (static_cast<size_t>(nbf) * p.kb_total + kb) * kWTile;
            dev::bulk_load(st + act_bytes, src, static_cast<uint32_t>(groups * kWTile),
                           full0 + 8 * s, pol_w);
          }
        } else {
          for (int q = 0; q < groups; ++q) {
            const uint8_t* src =
                p.w_packed + (static_cast<size_t>(nbf + q) * p.kb_total + kb) * kWTile;
            dev::bulk_load(st + act_bytes + q * kWTile, src, kWTile, full0 + 8 * s, pol_w);
          }
        }
      };
      auto load_act = [&](const Cur& c, int s, int tm) {
        const int kb = kb0 + c.i * kbs;
        if constexpr (kPair) {
          // kbs > 1: activations seen as [k-block][row][128 bytes], one box
          // per stage; kbs = 1: the 2-D view (zero fill past K)
          if (kbs > 1)
            dev::tma_load_3d_pair(sbase + s * stage_bytes, &tmap_act, 0,
                                  tm * C::kTileRows + px * kTile, kb, full_bar(s), pol_a);
          else
            dev::tma_load_2d_pair(sbase + s * stage_bytes, &tmap_act, kb * (kKBytes / kEsize),
                                  tm * C::kTileRows + px * kTile, full_bar(s), pol_a);
        } else if (kbs > 1) {
          dev::tma_load_3d(sbase + s * stage_bytes, &tmap_act, 0, tm * C::kActRows, kb,
                           full0 + 8 * s, pol_a);
        } else {
          dev::tma_load_2d(sbase + s * stage_bytes, &tmap_act, kb * (kKBytes / kEsize),
                           tm * C::kActRows, full0 + 8 * s, pol_a);
        }
      };
      const int npre = total < stages ? total : stages;
      Cur cur = start;
      for (int g = 0; g < npre; ++g) {  // first use of each stage needs no wait
        int tm, nbf, groups;
        const uint32_t tx = geom(cur, tm, nbf, groups);
        arm(g, tx);
        load_weights(cur, g, nbf, groups);
        advance(cur);
      }
      dev::grid_dependency_wait();
      cur = start;
      for (int g = 0; g < npre; ++g) {
        int tm, nbf, groups;
        geom(cur, tm, nbf, groups);
        load_act(cur, g, tm);
        advance(cur);
      }
      // the activation scale comes from the previous grid: fetched here
      // (after the dependency wait, through L2) while the first stages land,
      // and handed to the epilogue through shared memory (the arrival
      // releases the store, the epilogue's wait acquires it)
      *a_scale_s = p.a_scale ? __ldcg(p.a_scale) : 1.0f;
      dev::mbar_arrive(scale_bar);
      int issued = npre;
      int s = npre % stages;
      uint32_t ph = static_cast<uint32_t>(npre / stages);
      for (int g = npre; g < total; ++g) {
        if (!dev::mbar_wait(empty0 + 8 * s, (ph & 1) ^ 1, abort_flag, p.dev_status,
                            dev::kTimeoutProducer))
          break;
        int tm, nbf, groups;
        const uint32_t tx = geom(cur, tm, nbf, groups);
        arm(s, tx);
        load_weights(cur, s, nbf, groups);
        load_act(cur, s, tm);
        advance(cur);
        issued = g + 1;
        if (++s == stages) {
          s = 0;
          ++ph;
        }
      }
      // Do not leave with copies in flight: wait (bounded, even after an
      // abort) for the last use of every stage that was armed.  A pair's
      // copies complete on the leader's barriers, so each of its CTAs waits
      // instead until the MMAs released its stages (which also means the
      // leader's commits to this CTA's barriers have landed).
      for (int g = issued - stages < 0 ? 0 : issued - stages; g < issued; ++g) {
        if constexpr (kPair)
          dev::mbar_wait(empty0 + 8 * (g % stages), (g / stages) & 1, nullptr, p.dev_status,
                         dev::kTimeoutProducer);
        else
          dev::mbar_wait(full0 + 8 * (g % stages), (g / stages) & 1, nullptr, p.dev_status,
                         dev::kTimeoutProducer);
      }
    }
    __syncwarp();
    if (early_bye) dev::cluster_arrive_relaxed();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA
      constexpr uint32_t idesc = dev::instr_desc(kFp8, C::kTileRows, kBN);
      const uint16_t pair_mask = static_cast<uint16_t>(3u << lead_rank);
      auto commit = [&](uint32_t bar) {
        if constexpr (kPair)
          dev::mma_commit_pair(bar, pair_mask);  // both CTAs' barriers at this offset
        else
          dev::mma_commit(bar);
      };
      int s = 0;
      uint32_t ph = 0;
      for (int it = 0; it < my_tiles; ++it) {
        const int b = it % C::kAccBufs;
        const uint32_t u = static_cast<uint32_t>(it / C::kAccBufs);
        const bool free_acc =
            kPair ? dev::mbar_wait_cluster(tempty0 + 8 * b, (u & 1) ^ 1, abort_flag, p.dev_status,
                                           dev::kTimeoutMma)
                  : dev::mbar_wait(tempty0 + 8 * b, (u & 1) ^ 1, abort_flag, p.dev_status,
                                   dev::kTimeoutMma);
        if (!free_acc) break;
        dev::tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b * kBN);
        bool stop = false;
        const int units = (nkb + kbs - 1) / kbs;
        for (int i = 0; i < units; ++i) {
          if (!dev::mbar_wait(full0 + 8 * s, ph & 1, abort_flag, p.dev_status,
                              dev::kTimeoutMma)) {
            stop = true;
            break;
          }
          dev::tc_fence_after();
          const uint32_t st = sbase + s * stage_bytes;
          // k-blocks of this stage inside this CTA's K range (a stage past
          // its end holds another range's or zero data, not multiplied)
          const int hk = min(kbs, nkb - i * kbs);
          for (int h = 0; h < hk; ++h) {
            const uint32_t a_addr =
                kSwap ? st + act_bytes + h * C::kWBytes : st + h * C::kActBytes;
            const uint32_t b_addr =
                kSwap ? st + h * C::kActBytes : st + act_bytes + h * C::kWBytes;
            const uint64_t ad = dev::smem_desc_sw128(a_addr);
            const uint64_t bd = dev::smem_desc_sw128(b_addr);
#pragma unroll
            for (int k = 0; k < kKBytes / 32; ++k) {
              if constexpr (kPair)
                dev::mma_pair<kFp8>(d, ad + 2 * k, bd + 2 * k, idesc, (i | h | k) != 0);
              else
                dev::mma<kFp8>(d, ad + 2 * k, bd + 2 * k, idesc, (i | h | k) != 0);
            }
          }
          commit(empty0 + 8 * s);
          if (++s == stages) {
            s = 0;
            ++ph;
          }
        }
        commit(tfull0 + 8 * b);
        if (stop) break;
      }
    }
    __syncwarp();
    if (early_bye) dev::cluster_arrive_relaxed();
  } else {
    // -------------------------------------------------------------- epilogue
    const int et = threadIdx.x - 64;  // 0..127
    const int ew = warp & 3;          // TMEM lane quarter of this warp
    const int row = ew * 32 + lane;   // TMEM lane = tile row
    const uint32_t lane_off = static_cast<uint32_t>(ew * 32) << 16;
    uint8_t* wbuf = base + p.outbuf_off + (warp - 2) * 2 * kWarpOutBytes;  // this warp's 2 buffers
    // small M: this warp's row-store staging (32 rows x 64 bytes), after the
    // GeGLU's lane-exchange buffers if there are any
    __nv_bfloat16* swap_sb = reinterpret_cast<__nv_bfloat16*>(
        base + p.outbuf_off + (p.geglu ? kOutBytes : 0) + (warp - 2) * kSwapStoreBytes);
    const uint32_t wbuf_s = sbase + p.outbuf_off + (warp - 2) * 2 * kWarpOutBytes;
    int wb = 0;
    bool ok = true;
    bool bye = false;  // arrived on the pair's final cluster barrier
    float amax = 0.0f;  // running max |bf16 output| in the first s_cols columns
    // a drained accumulator buffer goes back to the MMA issuer (the leader
    // of a pair, whose MMAs write both CTAs' TMEM)
    auto release_acc = [&](int b) {
      dev::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair)
          dev::mbar_arrive_cluster(dev::map_to_rank(tempty0 + 8 * b, lead_rank));
        else
          dev::mbar_arrive(tempty0 + 8 * b);
      }
    };
    for (int it = 0; it < my_tiles; ++it) {
      int tm, tn;
      tile_of(it, tm, tn);
      const int b = it % C::kAccBufs;
      const uint32_t u = static_cast<uint32_t>(it / C::kAccBufs);
      // per-channel weight scale and bias are load-time data: fetch them
      // while the MMAs run
      constexpr int kColsPerThread = kSwap ? 1 : kBN / 128;
      float wsc[kColsPerThread], wbi[kColsPerThread];
#pragma unroll
      for (int j = 0; j < kColsPerThread; ++j) {
        const int n = kSwap ? (p.geglu ? (row < 64 ? 0 : p.f_groups * kTile - 64) + tn * 64 + row
                                       : tn * kTile + row)
                            : (p.geglu ? (j ? p.f_groups : 0) * kTile + tn * kTile + et
                                       : tn * kBN + et + 128 * j);
        wsc[j] = n < p.N ? (p.w_scale ? __ldg(p.w_scale + n) : 1.0f) : 0.0f;
        wbi[j] = (n < p.N && p.bias) ? __ldg(p.bias + n) : 0.0f;
      }
      // the activation scale from the copy thread (waited once, bounded);
      // the tile's per-channel factors are staged before its accumulator is
      // waited for
      const bool scale_ok =
          it != 0 || dev::mbar_wait(scale_bar, 0, abort_flag, p.dev_status, dev::kTimeoutEpilogue);
      const float as = *a_scale_s;
      float* cs_s = col_sb + (it & 1) * 2 * kBN;  // per-channel scale and bias of the tile
      float* cb_s = cs_s + kBN;
      float lcs = 1.0f, lcb = 0.0f;
      bool lact = false;
      if constexpr (!kSwap) {
        // (the buffer was last read in tile it - 2: every warp has passed
        // tile it - 1's barrier below since)
#pragma unroll
        for (int j = 0; j < kColsPerThread; ++j) {
          cs_s[et + 128 * j] = as * wsc[j];
          cb_s[et + 128 * j] = wbi[j];
        }
        dev::named_sync(1, 128);
      } else {
        const int n = p.geglu ? (row < 64 ? 0 : p.f_groups * kTile - 64) + tn * 64 + row
                              : tn * kTile + row;
        if (n < p.N) {
          lcs = as * wsc[0];
          lcb = wbi[0];
          lact = !p.geglu && n < p.act_cols;
        }
      }
      // small-M GeGLU: the up lanes (64-127) hand their values to the gate
      // lanes through shared memory (two alternating buffers of 64 lanes x
      // 32 floats, one barrier of the epilogue warps per exchange)
      float* xbuf = reinterpret_cast<float*>(base + p.outbuf_off);
      auto geglu_rows = [&](float* v, int nv, int buf) -> bool {  // true: this lane stores
        float* xb = xbuf + buf * (64 * 32);
        if (row >= 64) {
          for (int j = 0; j < nv; ++j) xb[j * 64 + (row - 64)] = v[j];
        }
        dev::named_sync(1, 128);
        if (row < 64) {
          for (int j = 0; j < nv; ++j) v[j] = gelu_tanh(v[j]) * xb[j * 64 + row];
        }
        return row < 64;
      };
      ok = dev::mbar_wait(tfull0 + 8 * b, u & 1, abort_flag, p.dev_status,
                          dev::kTimeoutEpilogue) &&
           scale_ok;
      ok = __all_sync(0xffffffffu, ok);
      if (early_bye && it + 1 == my_tiles) {
        dev::cluster_arrive_relaxed();
        bye = true;
      }
      dev::tc_fence_after();
      const uint32_t tacc = tmem + lane_off + static_cast<uint32_t>(b * kBN);
      const int row0 = tm * C::kTileRows + px * kTile;  // large M: first output row of this CTA
      // epilogue of 32 accumulator columns starting at tile column c32, and
      // this warp's store of them
      auto finish32 = [&](float* v, int c32, int rows_of_tile_m0) {
        if constexpr (!kSwap) {
          const int n0 = tn * kBN + c32;
          const float4* cs4 = reinterpret_cast<const float4*>(cs_s + c32);
          const float4* cb4 = reinterpret_cast<const float4*>(cb_s + c32);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 sc = cs4[q];
            const float4 bi = cb4[q];
            v[4 * q + 0] = lin(v[4 * q + 0], sc.x, bi.x);
            v[4 * q + 1] = lin(v[4 * q + 1], sc.y, bi.y);
            v[4 * q + 2] = lin(v[4 * q + 2], sc.z, bi.z);
            v[4 * q + 3] = lin(v[4 * q + 3], sc.w, bi.w);
          }
          // (uniform across the warp: the chunk's columns).  The GELUs are
          // evaluated without a branch per element, so that the 32
          // independent evaluations interleave; a chunk that straddles
          // act_cols selects per element.
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
          warp_store<false, 32>(v, wbuf + wb * kWarpOutBytes, wbuf_s + wb * kWarpOutBytes,
                                &tmap_out, n0, row0 + ew * 32, lane);
          if (p.s_cols)
            amax_row32_staged(p, amax, wbuf + wb * kWarpOutBytes + lane * 64, (lane >> 1) & 3,
                           row0 + ew * 32 + lane, n0);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = lin(v[j], lcs, lcb);
          if (lact) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = gelu_tanh(v[j]);
          }
          if (!p.geglu) {
            if (p.s_cols) amax_col<32>(p, amax, v, rows_of_tile_m0 + c32, tn * kTile + row);
            store_rows<32>(v, p, rows_of_tile_m0 + c32, tn * kTile + ew * 32, lane, swap_sb);
          } else if (geglu_rows(v, 32, wb)) {
            if (p.s_cols) amax_col<32>(p, amax, v, rows_of_tile_m0 + c32, tn * 64 + row);
            store_rows<32>(v, p, rows_of_tile_m0 + c32, tn * 64 + ew * 32, lane, swap_sb);
          }
        }
        wb ^= 1;
      };

      if (!split) {
        if (kPair && kBN == 256 && p.geglu) {
          if constexpr (kPair && kBN == 256) {
          // ------------- fused GeGLU: columns [0, 128) hold the gate, [128,
          // 256) the up channels of the same 128 outputs
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) {
            float g[32], u[32];
            dev::tmem_ld32(tacc + c, g);
            dev::tmem_ld32(tacc + 128 + c, u);
            if (c + 32 == 128 && it + 1 < my_tiles) release_acc(b);
            const float4* gs4 = reinterpret_cast<const float4*>(cs_s + c);
            const float4* gb4 = reinterpret_cast<const float4*>(cb_s + c);
            const float4* us4 = reinterpret_cast<const float4*>(cs_s + 128 + c);
            const float4* ub4 = reinterpret_cast<const float4*>(cb_s + 128 + c);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 gs = gs4[q], gb = gb4[q], us = us4[q], ub = ub4[q];
              g[4 * q + 0] = gelu_tanh(lin(g[4 * q + 0], gs.x, gb.x)) * lin(u[4 * q + 0], us.x, ub.x);
              g[4 * q + 1] = gelu_tanh(lin(g[4 * q + 1], gs.y, gb.y)) * lin(u[4 * q + 1], us.y, ub.y);
              g[4 * q + 2] = gelu_tanh(lin(g[4 * q + 2], gs.z, gb.z)) * lin(u[4 * q + 2], us.z, ub.z);
              g[4 * q + 3] = gelu_tanh(lin(g[4 * q + 3], gs.w, gb.w)) * lin(u[4 * q + 3], us.w, ub.w);
            }
            warp_store<false, 32>(g, wbuf + wb * kWarpOutBytes, wbuf_s + wb * kWarpOutBytes,
                                  &tmap_out, tn * kTile + c, row0 + ew * 32, lane);
            if (p.s_cols)
              amax_row32_staged(p, amax, wbuf + wb * kWarpOutBytes + lane * 64, (lane >> 1) & 3,
                             row0 + ew * 32 + lane, tn * kTile + c);
            wb ^= 1;
          }
          }
        } else if constexpr (kBN >= 64) {
#pragma unroll 1
          for (int c = 0; c < kBN; c += 64) {
            float v[64];
            dev::tmem_ld64(tacc + c, v);
            // accumulator read out: back to the MMA unless this was the last tile
            if (c + 64 == kBN && it + 1 < my_tiles) release_acc(b);
            finish32(v, c, tm * kBN);
            finish32(v + 32, c + 32, tm * kBN);
          }
        } else {
          float v[32];
          dev::tmem_ld32(tacc, v);
          if (it + 1 < my_tiles) release_acc(b);
          finish32(v, 0, tm * kBN);
        }
      } else if (gsplit) {
        if constexpr (!kSwap) {
          // ------------- split-K: exchange partial chunks through the workspace
          // slot of (tile, CTA of the pair, chunk c, split j): 128 rows x 32
          // columns, float4 granule q of row r at (q * 128 + r)
          const int tile = first_tile;
          auto slot = [&](int c, int j) -> float4* {
            return reinterpret_cast<float4*>(p.ws_part) +
                   (static_cast<size_t>((tile * 2 + px) * NC + c) * S + j) * (kTile * 8);
          };
          auto flag = [&](int o) { return p.ws_flag + (tile * 2 + px) * S + o; };
          // the other splits' partials of this CTA's chunks come into the
          // stage buffers (idle once the accumulator is complete) by one bulk
          // copy per (chunk, split), a batch of whole chunks at a time (one
          // batch unless the splits are many): one wait for all of them
          const int remote = S - 1;
          const int per_batch =
              max(1, (p.stages * stage_bytes) / (remote * static_cast<int>(chunk_bytes)));
          auto fetch = [&](int c0, bool go) {  // one thread; completes a recv_bar phase
            if (!go) {
              dev::mbar_arrive(recv_bar);
              return;
            }
            const int c1 = min(own_c1, c0 + per_batch);
            const uint64_t pol = dev::policy_evict_first();
            // the partials were written by other CTAs' generic stores and
            // acquired through the counter; the copies read them through the
            // async proxy
            dev::fence_proxy_async_global();
            dev::mbar_arrive_expect_tx(recv_bar,
                                       static_cast<uint32_t>((c1 - c0) * remote) * chunk_bytes);
            for (int c = c0; c < c1; ++c) {
              int i = (c - c0) * remote;
              for (int r = 0; r < S; ++r) {
                if (r == rank) continue;
                dev::bulk_load(sbase + static_cast<uint32_t>(i++) * chunk_bytes, slot(c, r),
                               chunk_bytes, recv_bar, pol);
              }
            }
          };
          // 1. the chunks other splits own -> their slots
          for (int c = 0; c < NC; ++c) {
            if (c >= own_c0 && c < own_c1) continue;
            float v[32];
            dev::tmem_ld32(tacc + c * 32, v);
            float4* dst = slot(c, rank);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              __stcg(dst + q * kTile + row,
                     make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
          }
          // every epilogue thread's partial stores happen before the counter
          // increments below: the CTA barrier orders them before the
          // signalling thread's release, which is cumulative over them
          dev::named_sync(1, 128);
          if (et == 0) {
            for (int o = 0; o < S; ++o)
              if (o != rank && chunk_begin(o) < chunk_begin(o + 1)) dev::counter_add_release(flag(o));
            // 2. wait (bounded) until the other S - 1 splits have written
            //    this CTA's chunks, then return the counter to zero
            if (own_c1 > own_c0) {
              const bool got = dev::wait_counter(flag(rank), static_cast<unsigned>(S - 1),
                                                 abort_flag, p.dev_status, dev::kTimeoutEpilogue);
              if (got)
                *flag(rank) = 0u;
              else
                ok = false;
              fetch(own_c0, got);
            }
          }
          dev::named_sync(1, 128);
          ok = !*abort_flag && ok;
          // 3. own chunks: the S partials added in split order
          uint32_t rph = 0;
          for (int c0 = own_c0; c0 < own_c1; c0 += per_batch) {
            const int c1 = min(own_c1, c0 + per_batch);
            if (c0 != own_c0) {
              dev::named_sync(1, 128);  // every thread is done with the previous batch
              if (et == 0) fetch(c0, !*abort_flag);
            }
            // (no abort shortcut: copies in flight land before the CTA exits)
            ok = dev::mbar_wait(recv_bar, rph, nullptr, p.dev_status, dev::kTimeoutEpilogue) && ok;
            rph ^= 1u;
            for (int c = c0; c < c1; ++c) {
              float acc[32];
              dev::tmem_ld32(tacc + c * 32, acc);
              float sum[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) sum[j] = 0.0f;
              const float4* got = reinterpret_cast<const float4*>(
                  base + static_cast<size_t>((c - c0) * remote) * chunk_bytes);
              for (int r = 0; r < S; ++r) {
                if (r == rank) {
#pragma unroll
                  for (int j = 0; j < 32; ++j) sum[j] += acc[j];
                } else {
#pragma unroll
                  for (int q = 0; q < 8; ++q) {
                    const float4 x = got[q * kTile + row];
                    sum[4 * q] += x.x;
                    sum[4 * q + 1] += x.y;
                    sum[4 * q + 2] += x.z;
                    sum[4 * q + 3] += x.w;
                  }
                  got += kTile * 8;  // the next split's chunk
                }
              }
              finish32(sum, c * 32, 0);
            }
          }
        }
      } else {
        // ------------- split-K: exchange partial chunks inside the cluster
        const int owned = own_c1 - own_c0;
        if (p.recv_in_stages) dev::cluster_arrive();  // this CTA's stage buffers are free
        // 1. the chunks other ranks own -> this CTA's send buffer (stage region)
        if constexpr (kSwap) {
          // 8-column chunks, read from TMEM up to 64 columns (one wait) at a time
          constexpr int kPiece = kBN < 64 ? kBN : 64;
#pragma unroll 1
          for (int c64 = 0; c64 < kBN; c64 += kPiece) {
            const int cb = c64 / 8;
            if (cb >= own_c0 && cb + kPiece / 8 <= own_c1) continue;  // all owned
            float v[kPiece];
            if constexpr (kPiece == 64)
              dev::tmem_ld64(tacc + c64, v);
            else
              dev::tmem_ld32(tacc + c64, v);
#pragma unroll
            for (int j = 0; j < kPiece / 8; ++j) {
              const int c = cb + j;
              if (c >= own_c0 && c < own_c1) continue;
              uint8_t* dst = base + (c < own_c0 ? c : c - owned) * chunk_bytes;
              *reinterpret_cast<float4*>(dst + chunk_off(row, 0, 8)) =
                  make_float4(v[8 * j], v[8 * j + 1], v[8 * j + 2], v[8 * j + 3]);
              *reinterpret_cast<float4*>(dst + chunk_off(row, 1, 8)) =
                  make_float4(v[8 * j + 4], v[8 * j + 5], v[8 * j + 6], v[8 * j + 7]);
            }
          }
        } else {
          for (int c = 0; c < NC; ++c) {
            if (c >= own_c0 && c < own_c1) continue;
            uint8_t* dst = base + (c < own_c0 ? c : c - owned) * chunk_bytes;
            float v[32];
            dev::tmem_ld32(tacc + c * 32, v);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<float4*>(dst + chunk_off(row, q, 32)) =
                  make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
        }
        dev::fence_proxy_async_smem();
        if constexpr (kSwap) {
          // 2. after phase 1 (every peer initialised), each warp copies its
          //    own 32 rows of every chunk to the chunk's owner
          __syncwarp();
          dev::cluster_wait();
          if (lane < S && lane != rank) {
            const int o = lane;
            const int oc0 = chunk_begin(o), oc1 = chunk_begin(o + 1);
            const int slot = rank < o ? rank : rank - 1;
            const uint32_t bar = dev::map_to_rank(recv_bar, o);
            for (int c = oc0; c < oc1; ++c) {
              const int sp = c < own_c0 ? c : c - owned;
              const uint32_t rows_off = static_cast<uint32_t>(ew * 32 * CW * 4);
              const uint32_t dst = dev::map_to_rank(
                  sbase + p.recv_off +
                      static_cast<uint32_t>(slot * owned_max + (c - oc0)) * chunk_bytes + rows_off,
                  o);
              dev::bulk_copy_to_peer(dst, sbase + sp * chunk_bytes + rows_off,
                                     static_cast<uint32_t>(32 * CW * 4), bar);
            }
          }
        } else {
          dev::named_sync(1, 128);
          // 2. after phase 1 (every peer initialised and its receive buffer
          //    free), one bulk copy per owner
          dev::cluster_wait();
          if (et == 0) {
            for (int o = 0; o < S; ++o) {
              if (o == rank) continue;
              const int oc0 = chunk_begin(o), oc1 = chunk_begin(o + 1);
              const int sp0 = oc0 < own_c0 ? oc0 : oc0 - owned;
              const int slot = rank < o ? rank : rank - 1;
              const uint32_t dst = dev::map_to_rank(
                  sbase + p.recv_off + static_cast<uint32_t>(slot * owned_max) * chunk_bytes,
                  split_cta(o));
              dev::bulk_copy_to_peer(dst, sbase + sp0 * chunk_bytes,
                                     static_cast<uint32_t>(oc1 - oc0) * chunk_bytes,
                                     dev::map_to_rank(recv_bar, split_cta(o)));
            }
          }
        }
        // 3. own chunks: own partial + received partials, in rank order
        ok = dev::mbar_wait(recv_bar, 0, abort_flag, p.dev_status, dev::kTimeoutEpilogue) && ok;
        ok = __all_sync(0xffffffffu, ok);
        dev::cluster_arrive_relaxed();  // phase 2: every copy into this CTA has landed
        const uint8_t* recv = base + p.recv_off;
        if constexpr (kSwap) {
#pragma unroll 1
          for (int lc = 0; lc < owned; ++lc) {
            float own[8];
            dev::tmem_ld8(tacc + (own_c0 + lc) * 8, own);
            // the other ranks' partials (receive slot q holds rank q below
            // this CTA's rank, q + 1 from it on), loaded three slots ahead of
            // their additions
            float4 px[3][2];
            auto load_slot = [&](int q, float4 (&x)[2]) {
              const uint8_t* src = recv + (q * owned_max + lc) * chunk_bytes;
              x[0] = *reinterpret_cast<const float4*>(src + chunk_off(row, 0, 8));
              x[1] = *reinterpret_cast<const float4*>(src + chunk_off(row, 1, 8));
            };
#pragma unroll
            for (int q = 0; q < 3; ++q)
              if (q < S - 1) load_slot(q, px[q]);
            // the S partials added in rank order, this CTA's own at its rank
            float sum[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) sum[j] = 0.0f;
#pragma unroll
            for (int q = 0; q < kMaxSplits; ++q) {
              if (q == rank) {
#pragma unroll
                for (int j = 0; j < 8; ++j) sum[j] += own[j];
              }
              if (q < kMaxSplits - 1 && q < S - 1) {
                const float4(&x)[2] = px[q % 3];
                sum[0] += x[0].x; sum[1] += x[0].y; sum[2] += x[0].z; sum[3] += x[0].w;
                sum[4] += x[1].x; sum[5] += x[1].y; sum[6] += x[1].z; sum[7] += x[1].w;
                if (q + 3 < kMaxSplits - 1 && q + 3 < S - 1) load_slot(q + 3, px[q % 3]);
              }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) sum[j] = lin(sum[j], lcs, lcb);
            if (lact) {
#pragma unroll
              for (int j = 0; j < 8; ++j) sum[j] = gelu_tanh(sum[j]);
            }
            if (!p.geglu) {
              if (p.s_cols) amax_col<8>(p, amax, sum, tm * kBN + (own_c0 + lc) * 8, tn * kTile + row);
              store_rows<8>(sum, p, tm * kBN + (own_c0 + lc) * 8, tn * kTile + ew * 32, lane,
                            swap_sb);
            } else if (geglu_rows(sum, 8, lc & 1)) {  // the gate lanes: warps 0-1 of 4
              if (p.s_cols) amax_col<8>(p, amax, sum, tm * kBN + (own_c0 + lc) * 8, tn * 64 + row);
              store_rows<8>(sum, p, tm * kBN + (own_c0 + lc) * 8, tn * 64 + ew * 32, lane,
                            swap_sb);
            }
          }
        } else {
          for (int c = own_c0; c < own_c1; ++c) {
            const int lc = c - own_c0;
            float acc[32];
            dev::tmem_ld32(tacc + c * 32, acc);
            // partial sums added in rank order, this CTA's own at its rank
            float sum[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) sum[j] = 0.0f;
            for (int r = 0; r < S; ++r) {
              if (r == rank) {
#pragma unroll
                for (int j = 0; j < 32; ++j) sum[j] += acc[j];
              } else {
                const int slot = r < rank ? r : r - 1;
                const uint8_t* src = recv + (slot * owned_max + lc) * chunk_bytes;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const float4 x = *reinterpret_cast<const float4*>(src + chunk_off(row, q, 32));
                  sum[4 * q] += x.x;
                  sum[4 * q + 1] += x.y;
                  sum[4 * q + 2] += x.z;
                  sum[4 * q + 3] += x.w;
                }
              }
            }
            finish32(sum, c * 32, 0);
          }
        }
      }
      if (!ok) break;
    }
    if (early_bye && !bye) dev::cluster_arrive_relaxed();
    // the TMA stores have read their staging buffers before the CTA leaves;
    // their writes are performed before the grid completes (and before a
    // dependent grid's wait returns), so the CTA does not wait for them
    if (lane == 0) dev::bulk_wait_read<0>();
    if (p.s_cols) {
      // the next layer's scale: the CTA's maximum, folded in by one thread
      float m = amax;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) amax_red[warp - 2] = m;
      dev::named_sync(1, 128);
      if (et == 0)
        next_scale_arrive(p, fmaxf(fmaxf(amax_red[0], amax_red[1]),
                                   fmaxf(amax_red[2], amax_red[3])));
    }
  }

  if (csplit) {
    if (warp < 2) {  // the copy and MMA warps: both barrier phases
      if (p.recv_in_stages) dev::cluster_arrive();
      dev::cluster_wait();
      dev::cluster_arrive();
    }
    // phase 2: every CTA has received its chunks, so no copy out of this
    // CTA's shared memory is still in flight
    dev::cluster_wait();
  } else if constexpr (kPair) {
    // neither CTA of a pair leaves (or frees TMEM) while the other may still
    // take part in its MMAs or signal its barriers (every warp arrived above)
    dev::cluster_wait();
  }
  dev::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    dev::tc_fence_after();
    if constexpr (kPair)
      dev::tmem_dealloc_pair(tmem, C::kTmemCols);
    else
      dev::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

// Static per-shape choices (frozen at call time; the same shape always gets
// the same plan): tile kind and width, split-K factor, grid, pipeline depth.
struct Plan {
  bool swap;
  bool pair;  // 256-row tiles on CTA pairs (cta_group::2)
  int bn;
  int tiles_m, tiles_n, num_tiles;
  int splits;
  int kb_per_split;
  int chunk_cols;
  int stages;
  int kbs;  // k-blocks per stage
  bool recv_in_stages;
  bool split_global;  // split-K through the workspace (CTA pairs)
  bool geglu;         // merged gate/up with the GeGLU fused: 256-wide pair tiles, no split
  size_t ws_bytes;    // workspace the plan uses (split_global), else 0
  size_t ws_flag_bytes;
  int outbuf_off, recv_off, tail_off;
  int smem;
  dim3 grid;
};

// Shared-memory layout for a given depth; false if it needs more than `cap`.
bool layout(Plan& pl, int stage_bytes, int cap = kSmemMax) {
  const int pipe = pl.stages * stage_bytes;
  pl.outbuf_off = pipe;
  pl.recv_off = 0;
  // small M stages each warp's rows (2 KiB a warp) for 16-byte stores, after
  // the 16 KiB through which a GeGLU exchanges its up values (the large-M
  // output buffers)
  int tail = pipe + (pl.swap ? (pl.geglu ? kOutBytes : 0) + 4 * kSwapStoreBytes : kOutBytes);
  if (pl.splits > 1 && !pl.split_global) {
    const int nchunks = pl.bn / pl.chunk_cols;
    const int chunk = kTile * pl.chunk_cols * 4;
    const int owned_max = static_cast<int>(ceil_div(nchunks, pl.splits));
    const int owned_min = nchunks / pl.splits;
    const int recv = (pl.splits - 1) * owned_max * chunk;
    const int send = (nchunks - owned_min) * chunk;
    if (send > pipe) return false;
    if (!pl.recv_in_stages) {
      pl.recv_off = tail;
      tail += recv;
    } else {
      pl.recv_off = send;
      if (send + recv > pipe) return false;
    }
  }
  pl.tail_off = static_cast<int>(ceil_div(tail, 128) * 128);
  pl.smem = 1024 + pl.tail_off + 16 * pl.bn + kBarRegion;
  return pl.smem <= cap;
}

// Sets the kernel's dynamic shared memory limit once per device.
template <bool kFp8, bool kSwap, bool kPair, int kBN>
cudaError_t prepare_kernel() {
  static std::mutex mu;
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<kFp8, kSwap, kPair, kBN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  return cudaSuccess;
}

// Number of clusters of `s` split-K CTAs (times 2 for pairs) with `smem`
// bytes each that can be resident at once (cached per device and
// configuration).
template <bool kFp8, bool kSwap, bool kPair, int kBN>
int cluster_capacity(int s, int smem) {
  static std::mutex mu;
  static int cache[64][kMaxSplits + 1][8];
  static bool init = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (prepare_kernel<kFp8, kSwap, kPair, kBN>() != cudaSuccess) return 0;
  const int sb = (smem + 32767) / 32768;  // smem bucket of 32 KiB
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (auto& a : cache)
      for (auto& b : a)
        for (int& c : b) c = -1;
    init = true;
  }
  int& c = cache[dev][s][sb < 8 ? sb : 7];
  if (c < 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kPair ? 2 : 1, 1, static_cast<unsigned>(s));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(sb < 8 ? sb * 32768 : kSmemMax);
    if (cfg.dynamicSmemBytes > static_cast<size_t>(kSmemMax)) cfg.dynamicSmemBytes = kSmemMax;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = static_cast<unsigned>(s);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<kFp8, kSwap, kPair, kBN>, &cfg) !=
        cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    c = n;
  }
  return c;
}

template <bool kFp8>
int cluster_capacity_for(const Plan& pl, int s, int smem) {
  if (pl.pair)
    return pl.bn == 128 ? cluster_capacity<kFp8, false, true, 128>(s, smem)
                        : cluster_capacity<kFp8, false, true, 256>(s, smem);
  switch (pl.bn) {
    case 32: return cluster_capacity<kFp8, true, false, 32>(s, smem);
    case 64: return cluster_capacity<kFp8, true, false, 64>(s, smem);
    default: return cluster_capacity<kFp8, true, false, 128>(s, smem);
  }
}

// Places the pipeline and the split-K receive buffers: the deepest pipeline
// (up to `want` stages) with a dedicated receive region, or with the
// receive buffers inside the stage buffers if that allows a deeper one.
bool place_buffers(Plan& pl, int stage_bytes, int want, int cap = kSmemMax) {
  int best = 0;
  bool best_in_stages = false;
  for (int mode = 0; mode < (pl.splits > 1 && !pl.split_global ? 2 : 1); ++mode) {
    pl.recv_in_stages = mode == 1;
    for (int st = kMaxStages; st >= 2; --st) {
      if (!pl.recv_in_stages && st > want) continue;
      pl.stages = st;
      if (!layout(pl, stage_bytes, cap)) continue;
      const int eff = st < want ? st : want;
      if (eff > best) {
        best = eff;
        best_in_stages = pl.recv_in_stages;
      }
      break;
    }
  }
  if (best == 0) return false;
  pl.recv_in_stages = best_in_stages;
  for (int st = best_in_stages ? kMaxStages : want; st >= 2; --st) {
    pl.stages = st;
    if (layout(pl, stage_bytes, cap)) return true;
  }
  return false;
}

// Static per-shape choices (the same shape always gets the same plan): tile
// kind and width, split-K factor, grid and pipeline depth.  The split is the
// largest one that fits shared memory and keeps every cluster resident in
// one wave.
// Workspace of a global split: the arrival counters, then one 16 KiB slot per
// (tile, CTA of the pair, 32-column chunk, split).
void global_split_bytes(Plan& pl) {
  const int nchunks = pl.bn / pl.chunk_cols;
  pl.ws_flag_bytes = static_cast<size_t>(ceil_div(
                         static_cast<int64_t>(pl.num_tiles) * 2 * pl.splits * 4, 256)) * 256;
  pl.ws_bytes = pl.ws_flag_bytes + static_cast<size_t>(pl.num_tiles) * 2 * nchunks * pl.splits *
                                       static_cast<size_t>(kTile * pl.chunk_cols * 4);
}

Plan make_plan(int64_t M, int64_t N, int64_t K, int esize, bool fp8, size_t ws_avail,
               bool geglu = false) {
  Plan pl;
  pl.split_global = false;
  pl.geglu = geglu;
  pl.ws_bytes = 0;
  pl.ws_flag_bytes = 0;
  const int kb = static_cast<int>(ceil_div(K * esize, kKBytes));
  const int nb = static_cast<int>(ceil_div(N, kTile));
  const int sms = sm_count() > 0 ? sm_count() : 148;
  pl.pair = false;
  if (M <= 128) {
    pl.swap = true;
    pl.bn = M <= 32 ? 32 : (M <= 64 ? 64 : 128);
    pl.tiles_n = nb;
    pl.tiles_m = static_cast<int>(ceil_div(M, pl.bn));
    pl.chunk_cols = 8;
  } else {
    // 256-row tiles on CTA pairs: each CTA ingests 128 activation rows and
    // half of the tile's weight channels per k-block.  256 x 256 tiles carry
    // the most FLOPs per ingested byte; when they would leave most SMs idle
    // on a short K loop, 256 x 128 tiles fill the machine without a split-K
    // exchange.
    pl.swap = false;
    pl.pair = true;
    pl.tiles_m = static_cast<int>(ceil_div(M, 2 * kTile));
    const int64_t wide = 2 * pl.tiles_m * ceil_div(N, 256);  // CTAs
    const int64_t narrow = 2 * pl.tiles_m * ceil_div(N, 128);
    pl.bn = (!geglu && 2 * wide <= sms && narrow <= sms && kb <= 32) ? 128 : 256;
    pl.tiles_n = static_cast<int>(ceil_div(N, pl.bn));
    pl.chunk_cols = 32;
  }
  pl.num_tiles = pl.tiles_m * pl.tiles_n;
  const int ctas_per_tile = pl.pair ? 2 : 1;
  const int act_rows = pl.swap ? pl.bn : kTile;
  const int w_rows = pl.swap ? kTile : (pl.pair ? pl.bn / 2 : pl.bn);
  // pairs: several k-blocks per stage (one box per operand) when K is a
  // whole number of 128-byte k-blocks, so the activations can be seen as
  // [k-block][row][128 bytes]: fewer, larger copies.  Two for 256-channel
  // tiles (3 stages of 64 KiB), four for 128-channel tiles with 8 or more
  // k-blocks (2 stages of 96 KiB).
  const bool whole_kb = (K * esize) % kKBytes == 0;
  pl.kbs = (pl.pair && whole_kb && kb >= 2) ? ((pl.bn == 128 && kb >= 8) ? 4 : 2) : 1;
  int stage_bytes = pl.kbs * (act_rows + w_rows) * kKBytes;
  // a split's K range: a whole number of stages (cluster splits), or as even
  // as the split allows (splits through the workspace: a stage that runs
  // past the range is loaded whole and multiplied only as far as the range
  // goes, and the splits finish together)
  auto split_kb = [&](int s) {
    return static_cast<int>(ceil_div(ceil_div(kb, s), pl.kbs) * pl.kbs);
  };
  auto split_kb_even = [&](int s) { return static_cast<int>(ceil_div(kb, s)); };

  int s_max = 1, g_max = 1;
  // (a pair's GeGLU tile is finished whole: its gate and up halves would
  // meet in different split owners' chunks)
  if (pl.num_tiles * ctas_per_tile < sms && !(geglu && pl.pair)) {
    s_max = sms / (pl.num_tiles * ctas_per_tile);
    const int nchunks = pl.bn / pl.chunk_cols;
    if (s_max > nchunks) s_max = nchunks;
    if (s_max > kb) s_max = kb;
    if (s_max < 1) s_max = 1;
    g_max = pl.pair ? s_max : 1;  // a global split is not bounded by the cluster size
    if (s_max > kMaxSplits / ctas_per_tile) s_max = kMaxSplits / ctas_per_tile;
  }
  // CTA pairs: a split of K through the workspace, when the caller gave
  // enough of it and every pair of the grid can be resident at once (the
  // owners of each chunk wait for the other splits' partials).  It is taken
  // below only if it splits K further than a cluster can.
  Plan gpl = pl;
  bool have_g = false;
  for (int s = g_max; s >= 2 && !have_g; --s) {
    gpl.kb_per_split = split_kb_even(s);
    gpl.splits = static_cast<int>(ceil_div(kb, gpl.kb_per_split));
    if (gpl.splits < 2) break;
    gpl.split_global = true;
    global_split_bytes(gpl);
    // (the owners gather the other splits' partials of a chunk into their
    // stage buffers: at least one chunk's worth must fit)
    if (gpl.ws_bytes <= ws_avail && place_buffers(gpl, stage_bytes, kMaxStages) &&
        gpl.stages * stage_bytes >= (gpl.splits - 1) * kTile * gpl.chunk_cols * 4) {
      const int smem = gpl.smem < kPairMinSmem ? kPairMinSmem : gpl.smem;
      const int capacity = fp8 ? cluster_capacity_for<true>(gpl, 1, smem)
                               : cluster_capacity_for<false>(gpl, 1, smem);
      have_g = capacity >= gpl.num_tiles * gpl.splits;
    }
  }
  for (int s = s_max; s >= 1; --s) {
    if (pl.swap) {  // small M: two k-blocks per stage when each CTA has two or more
      pl.kbs = (whole_kb && ceil_div(kb, s) >= 2) ? 2 : 1;
      stage_bytes = pl.kbs * (act_rows + w_rows) * kKBytes;
    }
    pl.kb_per_split = split_kb(s);
    pl.splits = static_cast<int>(ceil_div(kb, pl.kb_per_split));
    // pipeline depth: small M takes just the CTA's k-blocks (a small
    // footprint lets a dependent grid's CTAs be resident early and
    // prefetch); large M and multi-tile walks take as many as fit
    int want = kMaxStages;
    if (pl.swap) {
      const int per_cta = static_cast<int>(ceil_div(pl.splits > 1 ? pl.kb_per_split : kb, pl.kbs));
      want = per_cta < 2 ? 2 : (per_cta > kMaxStages ? kMaxStages : per_cta);
      if (pl.splits == 1 && pl.num_tiles > sms) want = kMaxStages;
    }
    if (!place_buffers(pl, stage_bytes, want)) continue;
    if (pl.splits == 1) break;
    const int smem = pl.pair && pl.smem < kPairMinSmem ? kPairMinSmem : pl.smem;
    const int capacity = fp8 ? cluster_capacity_for<true>(pl, pl.splits, smem)
                             : cluster_capacity_for<false>(pl, pl.splits, smem);
    if (capacity >= pl.num_tiles) break;
  }
  // the workspace: deeper splits (no cluster size limit, no cluster
  // placement); a cluster's shared-memory exchange is cheaper at equal splits
  if (have_g && gpl.splits > pl.splits) pl = gpl;
  // a pair CTA takes all 512 TMEM columns: with at least kPairMinSmem of
  // shared memory no other GEMM CTA (each takes over 40 KiB) is resident
  // beside it, while the small CTAs of other kernels still are
  if (pl.pair && pl.smem < kPairMinSmem) pl.smem = kPairMinSmem;
  if (pl.split_global || pl.splits > 1) {
    pl.grid = dim3(static_cast<unsigned>(pl.num_tiles * ctas_per_tile), 1,
                   static_cast<unsigned>(pl.splits));
  } else {
    // persistent: one CTA (pair) per SM (two SMs), and no more CTAs (pairs)
    // than can be resident at once, so that the grid is one wave
    int units = sms / ctas_per_tile;
    const int cap = fp8 ? cluster_capacity_for<true>(pl, 1, pl.smem)
                        : cluster_capacity_for<false>(pl, 1, pl.smem);
    if (cap > 0 && cap < units) units = cap;
    pl.grid = dim3(static_cast<unsigned>((pl.num_tiles < units ? pl.num_tiles : units) *
                                         ctas_per_tile),
                   1, 1);
  }
  return pl;
}

template <bool kFp8, bool kSwap, bool kPair, int kBN>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tw, const CUtensorMap& to,
                       const GemmArgs& a, const Plan& pl, cudaStream_t stream) {
  auto kern = gemm_tc_kernel<kFp8, kSwap, kPair, kBN>;
  cudaError_t e = prepare_kernel<kFp8, kSwap, kPair, kBN>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = pl.grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kPair ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = pl.split_global ? 1 : pl.splits;
  cfg.attrs = attr;
  cfg.numAttrs = (kPair || pl.splits > 1) ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kern, ta, tw, to, a);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

template <bool kFp8>
cudaError_t dispatch(const CUtensorMap& ta, const CUtensorMap& tw, const CUtensorMap& to,
                     const GemmArgs& a, const Plan& pl, cudaStream_t stream) {
  if (pl.pair)
    return pl.bn == 128 ? launch_one<kFp8, false, true, 128>(ta, tw, to, a, pl, stream)
                        : launch_one<kFp8, false, true, 256>(ta, tw, to, a, pl, stream);
  switch (pl.bn) {
    case 32: return launch_one<kFp8, true, false, 32>(ta, tw, to, a, pl, stream);
    case 64: return launch_one<kFp8, true, false, 64>(ta, tw, to, a, pl, stream);
    default: return launch_one<kFp8, true, false, 128>(ta, tw, to, a, pl, stream);
  }
}

// The next layer's scale taken in a GEMM's epilogue (none when scale is null).
struct NextScale {
  int64_t cols;
  float* scale;
  void* hdr;
  size_t hdr_bytes;
};

frt_status gemm_common(bool fp8, const void* a, int64_t lda, const float* a_scale,
                       const void* w_packed, const float* w_scale, const float* bias, int64_t M,
                       int64_t N, int64_t K, frt_act act, int64_t act_cols, void* out,
                       int64_t ldo, void* workspace, size_t workspace_bytes, int* dev_status,
                       frt_stream_t stream, const NextScale& ns = NextScale{}) {
  const int esize = fp8 ? 1 : 2;
  if (!a || !w_packed || !out) return FRT_ERR_INVALID_ARG;
  if (fp8 && (!a_scale || !w_scale)) return FRT_ERR_INVALID_ARG;
  if (act != FRT_ACT_NONE && act != FRT_ACT_GELU_TANH && act != FRT_ACT_GEGLU)
    return FRT_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return FRT_ERR_INVALID_ARG;
  if (act == FRT_ACT_GELU_TANH && (act_cols < 0 || act_cols > N)) return FRT_ERR_INVALID_ARG;
  const bool geglu = act == FRT_ACT_GEGLU;
  const int64_t n_out = geglu ? N / 2 : N;  // GeGLU: gelu(gate) * up, N / 2 columns
  if (lda < K || ldo < n_out) return FRT_ERR_INVALID_ARG;
  if (geglu && N % 256 != 0) return FRT_ERR_UNSUPPORTED_SHAPE;
  if (ldo > (1LL << 31) - 1) return FRT_ERR_UNSUPPORTED_SHAPE;
  if (N % 16 != 0 || K % (fp8 ? 32 : 16) != 0) return FRT_ERR_UNSUPPORTED_SHAPE;
  if (M > (1LL << 31) - 1 || N > (1LL << 31) - 1 || K > (1LL << 31) - 1)
    return FRT_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(a, 16) || (lda * esize) % 16 != 0 || !aligned(w_packed, 16) ||
      !aligned(out, 16) || ldo % 8 != 0)
    return FRT_ERR_MISALIGNED;
  if ((a_scale && !aligned(a_scale, 4)) || (w_scale && !aligned(w_scale, 4)) ||
      (bias && !aligned(bias, 4)) || (dev_status && !aligned(dev_status, 4)))
    return FRT_ERR_MISALIGNED;
  if (ns.scale) {
    if (ns.cols < 1 || ns.cols > n_out || !ns.hdr) return FRT_ERR_INVALID_ARG;
    if (ns.cols % 8 != 0) return FRT_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(ns.scale, 4) || !aligned(ns.hdr, 16)) return FRT_ERR_MISALIGNED;
    if (ns.hdr_bytes < kNextScaleHeaderBytes) return FRT_ERR_WORKSPACE_TOO_SMALL;
  }

  const int64_t kb_total = ceil_div(K * esize, kKBytes);
  const int64_t nb_total = ceil_div(N, kTile);
  if (nb_total * kb_total * kTile > (1LL << 31) - 1) return FRT_ERR_UNSUPPORTED_SHAPE;

  auto encode = tensor_map_encoder();
  if (!encode) return FRT_ERR_CUDA;
  // a workspace that is missing or misaligned is not used
  const size_t ws_avail = (workspace && aligned(workspace, 256)) ? workspace_bytes : 0;
  const Plan pl = make_plan(M, N, K, esize, fp8, ws_avail, geglu);

  CUtensorMap ta, tw, to;
  if (pl.kbs > 1) {
    // activations as [k-block][row][128 bytes of K]; one box = the CTA's
    // rows of kbs consecutive k-blocks (zero fill past M and past the last
    // k-block)
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kKBytes / esize),
                                static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(kb_total)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(lda * esize),
                                   static_cast<cuuint64_t>(kKBytes)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kKBytes / esize),
                               static_cast<cuuint32_t>(pl.swap ? pl.bn : kTile),
                               static_cast<cuuint32_t>(pl.kbs)};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&ta, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void*>(a), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FRT_ERR_CUDA;
  } else {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lda * esize)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKBytes / esize),
                               static_cast<cuuint32_t>(pl.swap ? pl.bn : kTile)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&ta, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void*>(a), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FRT_ERR_CUDA;
  }
  if (pl.pair) {
    // packed weight tiles as [tile][128 rows][128 bytes] (the tiles are
    // stored in their shared-memory image, so no swizzle); one box = the 128
    // or 64 channels that a pair's CTA holds, of kbs consecutive k-tiles
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kKBytes), static_cast<cuuint64_t>(kTile),
                                static_cast<cuuint64_t>(nb_total * kb_total)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kKBytes),
                                   static_cast<cuuint64_t>(kWTile)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kKBytes), static_cast<cuuint32_t>(pl.bn / 2),
                               static_cast<cuuint32_t>(pl.kbs)};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(w_packed), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FRT_ERR_CUDA;
  } else {
    tw = ta;  // not read by the single-CTA kernels
  }
  {
    // output boxes, one per epilogue warp and chunk: {32 channels, 32 rows}
    // (small M split-K: {32 channels, 8 rows}), 64-byte swizzle
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(n_out), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldo * 2)};
    const cuuint32_t box[2] = {32u, (pl.swap && pl.splits > 1) ? 8u : 32u};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FRT_ERR_CUDA;
  }

  GemmArgs ga;
  ga.w_packed = static_cast<const uint8_t*>(w_packed);
  ga.a_scale = a_scale;
  ga.w_scale = w_scale;
  ga.bias = bias;
  ga.M = static_cast<int>(M);
  ga.N = static_cast<int>(N);
  ga.act_cols = act == FRT_ACT_GELU_TANH ? static_cast<int>(act_cols) : 0;
  ga.geglu = geglu ? 1 : 0;
  ga.f_groups = geglu ? static_cast<int>(N / 256) : 0;
  ga.kb_total = static_cast<int>(kb_total);
  ga.nb_total = static_cast<int>(nb_total);
  ga.kb_per_split = pl.kb_per_split;
  ga.splits = pl.splits;
  ga.tiles_m = pl.tiles_m;
  ga.tiles_n = pl.tiles_n;
  ga.num_tiles = pl.num_tiles;
  ga.stages = pl.stages;
  ga.kbs = pl.kbs;
  ga.chunk_cols = pl.chunk_cols;
  ga.recv_in_stages = pl.recv_in_stages ? 1 : 0;
  ga.outbuf_off = pl.outbuf_off;
  ga.recv_off = pl.recv_off;
  ga.tail_off = pl.tail_off;
  ga.split_global = pl.split_global ? 1 : 0;
  ga.out = static_cast<__nv_bfloat16*>(out);
  ga.ldo = static_cast<int>(ldo);
  ga.ws_flag = pl.split_global ? static_cast<unsigned*>(workspace) : nullptr;
  ga.ws_part = pl.split_global
                   ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.ws_flag_bytes)
                   : nullptr;
  ga.dev_status = dev_status;
  ga.s_cols = ns.scale ? static_cast<int>(ns.cols) : 0;
  ga.s_out = ns.scale;
  ga.s_hdr = ns.scale ? static_cast<unsigned*>(ns.hdr) : nullptr;

  cudaError_t e = fp8 ? dispatch<true>(ta, tw, to, ga, pl, as_cuda(stream))
                      : dispatch<false>(ta, tw, to, ga, pl, as_cuda(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FRT_ERR_CUDA;
  }
  return launch_status();
}

}  // namespace
}  // namespace frt

extern "C" size_t frt_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, frt_dtype a_dtype) {
  // only CTA-pair plans (M > 128) split K through the workspace
  if (M <= 128 || N < 1 || K < 1) return 0;
  if (a_dtype != FRT_E4M3_OCP && a_dtype != FRT_BF16) return 0;
  const bool fp8 = a_dtype == FRT_E4M3_OCP;
  const frt::Plan pl = frt::make_plan(M, N, K, fp8 ? 1 : 2, fp8, static_cast<size_t>(-1));
  return pl.ws_bytes;
}

extern "C" frt_status frt_gemm_fp8(const uint8_t* a_q, int64_t lda, const float* a_scale,
                                   const void* w_packed, const float* w_scale, const float* bias,
                                   int64_t M, int64_t N, int64_t K, frt_act act, int64_t act_cols,
                                   void* out, int64_t ldo, void* workspace,
                                   size_t workspace_bytes, int* dev_status,
                                   frt_stream_t stream) {
  return frt::gemm_common(true, a_q, lda, a_scale, w_packed, w_scale, bias, M, N, K, act,
                          act_cols, out, ldo, workspace, workspace_bytes, dev_status, stream);
}

extern "C" frt_status frt_gemm_bf16(const void* a, int64_t lda, const void* w_packed,
                                    const float* w_scale, const float* bias, int64_t M, int64_t N,
                                    int64_t K, frt_act act, int64_t act_cols, void* out,
                                    int64_t ldo, void* workspace, size_t workspace_bytes,
                                    int* dev_status, frt_stream_t stream) {
  return frt::gemm_common(false, a, lda, nullptr, w_packed, w_scale, bias, M, N, K, act, act_cols,
                          out, ldo, workspace, workspace_bytes, dev_status, stream);
}

extern "C" size_t frt_gemm_next_scale_workspace_bytes(void) {
  return frt::kNextScaleHeaderBytes;
}

extern "C" frt_status frt_gemm_fp8_next_scale(
    const uint8_t* a_q, int64_t lda, const float* a_scale, const void* w_packed,
    const float* w_scale, const float* bias, int64_t M, int64_t N, int64_t K, frt_act act,
    int64_t act_cols, void* out, int64_t ldo, int64_t scale_cols, float* scale,
    void* scale_workspace, size_t scale_workspace_bytes, void* workspace, size_t workspace_bytes,
    int* dev_status, frt_stream_t stream) {
  if (!scale) return FRT_ERR_INVALID_ARG;
  const frt::NextScale ns = {scale_cols, scale, scale_workspace, scale_workspace_bytes};
  return frt::gemm_common(true, a_q, lda, a_scale, w_packed, w_scale, bias, M, N, K, act,
                          act_cols, out, ldo, workspace, workspace_bytes, dev_status, stream, ns);
}

extern "C" frt_status frt_gemm_bf16_next_scale(
    const void* a, int64_t lda, const void* w_packed, const float* w_scale, const float* bias,
    int64_t M, int64_t N, int64_t K, frt_act act, int64_t act_cols, void* out, int64_t ldo,
    int64_t scale_cols, float* scale, void* scale_workspace, size_t scale_workspace_bytes,
    void* workspace, size_t workspace_bytes, int* dev_status, frt_stream_t stream) {
  if (!scale) return FRT_ERR_INVALID_ARG;
  const frt::NextScale ns = {scale_cols, scale, scale_workspace, scale_workspace_bytes};
  return frt::gemm_common(false, a, lda, nullptr, w_packed, w_scale, bias, M, N, K, act, act_cols,
                          out, ldo, workspace, workspace_bytes, dev_status, stream, ns);
}

extern "C" int frt_gemm_describe(int64_t M, int64_t N, int64_t K, frt_dtype a_dtype,
                                 size_t workspace_bytes, char* buf, size_t buf_len) {
  if (M < 1 || N < 1 || K < 1 || N % 16 != 0) return -1;
  if (M > (1LL << 31) - 1 || N > (1LL << 31) - 1 || K > (1LL << 31) - 1) return -1;
  if (a_dtype != FRT_E4M3_OCP && a_dtype != FRT_BF16) return -1;
  const bool fp8 = a_dtype == FRT_E4M3_OCP;
  if (K % (fp8 ? 32 : 16) != 0) return -1;
  const frt::Plan pl = frt::make_plan(M, N, K, fp8 ? 1 : 2, fp8, workspace_bytes);
  const unsigned cx = pl.pair ? 2u : 1u;
  const unsigned cz = pl.split_global ? 1u : static_cast<unsigned>(pl.splits);
  char line[256];
  const int n = std::snprintf(
      line, sizeof line,
      "kind=%s bn=%d kbs=%d stages=%d splits=%d global=%d tiles=%d grid=%u,%u,%u "
      "cluster=%u,1,%u smem=%d",
      pl.pair ? "pair" : "swap", pl.bn, pl.kbs, pl.stages, pl.splits, pl.split_global ? 1 : 0,
      pl.num_tiles, pl.grid.x, pl.grid.y, pl.grid.z, cx, cz, pl.smem);
  if (n < 0) return -1;
  if (buf && buf_len > 0) {
    const size_t c = static_cast<size_t>(n) < buf_len ? static_cast<size_t>(n) : buf_len - 1;
    std::memcpy(buf, line, c);
    buf[c] = '\0';
  }
  return n;
}
