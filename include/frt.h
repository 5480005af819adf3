/*
 * frt.h -- C ABI of libfrt: the quantized linear layers of a small-batch,
 * latency-bound VLA forward pass on GB300 (sm_103a).
 *
 * The path (sources cited by page title and section):
 *   - E4M3 activation quantization: amax, fp32 scale, round-to-nearest-even
 *     with saturation ("Real-time VLA inference on AMD hardware", "How
 *     FlashRT works": weights and activations are quantized to FP8);
 *   - FNUZ -> OCP re-encoding of imported E4M3 bytes: same bit layout,
 *     exponent bias off by one, a byte read in the wrong dialect is 2x off
 *     (same page, "Different FP8 representation"; "Deploying
 *     DeepSeek-V4-Flash on AMD MI300X", "The FP8 dialect problem");
 *   - load-time weight packing into the layout the tensor-core kernels read,
 *     at a fixed address for graph replay (first page, "Packing around the
 *     instruction");
 *   - FP8 and BF16 GEMMs, fp32 accumulation, with the per-channel scale,
 *     bias and optional tanh-GELU applied in the epilogue and a bf16 store
 *     (first page, "Merging gate and up": the bias is applied in the GEMM
 *     epilogue; a merged [W_gate, W_up] weight is one GEMM).
 *
 * Conventions shared by every entry point:
 *   - Pointers named x, q, w, packed, a, out, scale, bias, workspace and
 *     dev_status are DEVICE pointers; the caller owns every buffer.  The
 *     library never allocates or frees device memory and never synchronises
 *     the stream; work is enqueued on `stream` (NULL = the legacy default
 *     stream), so every call is legal inside CUDA stream capture and can be
 *     replayed from a CUDA graph with the same pointers and shapes.
 *   - Shapes and leading dimensions are in ELEMENTS.  Matrices are row-major.
 *   - Arguments are checked on the host before anything is enqueued; a
 *     failed check returns its status and enqueues nothing.  A launch
 *     failure returns FRT_ERR_CUDA (from cudaGetLastError).
 *   - The first call that launches a given kernel sets its function
 *     attributes (dynamic shared memory size); make one eager call of each
 *     entry point before capturing a graph.
 *   - Kernels run only on sm_103a (GB300); on any other device the launch
 *     fails with FRT_ERR_CUDA.
 */
#ifndef FRT_H_
#define FRT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-compatible with cudaStream_t / CUstream. */
typedef struct CUstream_st* frt_stream_t;

typedef enum {
  FRT_OK = 0,
  FRT_ERR_INVALID_ARG = 1,         /* null pointer, negative size, bad enum */
  FRT_ERR_UNSUPPORTED_SHAPE = 2,   /* a size constraint below is not met */
  FRT_ERR_MISALIGNED = 3,          /* a pointer or leading dimension is not aligned */
  FRT_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace or packed buffer smaller than required */
  FRT_ERR_CUDA = 5,                /* a CUDA runtime call or launch failed */
  FRT_ERR_TIMEOUT = 6              /* a device-side bounded wait expired (see dev_status) */
} frt_status;

typedef enum {
  FRT_F32 = 0,
  FRT_BF16 = 1,
  FRT_E4M3_OCP = 2,  /* OCP E4M3: bias 7, max 448, NaN = 0x7f/0xff, has -0 */
  FRT_E4M3_FNUZ = 3  /* FNUZ E4M3: bias 8, max 240, NaN = 0x80 only, no -0 */
} frt_dtype;

typedef enum {
  FRT_SCALE_PER_TENSOR = 0, /* one scale for the whole tensor */
  FRT_SCALE_PER_COL = 1     /* one scale per column c of a [rows x cols] tensor */
} frt_scale_mode;

typedef enum {
  FRT_ACT_NONE = 0,
  FRT_ACT_GELU_TANH = 1, /* 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))) */
  FRT_ACT_GEGLU = 2      /* merged gate/up: out = gelu_tanh(v_gate) * v_up, N / 2 columns */
} frt_act;

/* Version of this ABI (incremented on any signature change). */
int frt_abi_version(void);

/* Number of kernels this library has launched in this process (or recorded
 * into a stream capture: a captured call counts once, its graph's replays do
 * not), over all devices and threads.  For accounting only. */
unsigned long long frt_launch_count(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* frt_status_string(frt_status status);

/* ------------------------------------------------------------------------
 * E4M3 quantization ("Real-time VLA inference on AMD hardware", "How FlashRT
 * works" and "Different FP8 representation").
 *
 *   amax  = max |x| over the tensor (FRT_SCALE_PER_TENSOR) or over the rows
 *           of each column (FRT_SCALE_PER_COL); NaN elements are ignored.
 *   s     = amax / max_finite, one IEEE fp32 division (448 for OCP, 240 for
 *           FNUZ); s = 1 where amax == 0.  s is the DEQUANT multiplier:
 *           x ~= decode(q) * s.
 *   q     = E4M3(x / s), the quotient an IEEE fp32 division, encoded with
 *           round-to-nearest-even and saturation: NaN -> the NaN code (OCP
 *           0x7f, FNUZ 0x80), |v| >= max_finite (inf included) -> +-max;
 *           a negative value that rounds to zero is 0x80 in OCP, 0x00 in FNUZ.
 *
 * x         : [rows x cols] of x_dtype (FRT_BF16 or FRT_F32), row stride ldx.
 * out_fmt   : FRT_E4M3_OCP or FRT_E4M3_FNUZ.
 * static_scale: NULL -> compute amax and s as above.  Non-NULL -> device
 *           pointer to the scale(s) to use (1 float, or `cols` floats per
 *           column); amax is skipped and the workspace is not used (per
 *           tensor, a dense aligned x is encoded in one pass as its parts
 *           arrive on chip: no barrier between the CTAs).
 * q         : [rows x cols] bytes, contiguous (row stride cols).
 * scale     : device, receives s (1 float, or `cols` floats); may be NULL.
 * workspace : device memory of frt_quantize_workspace_bytes() bytes, 4-byte
 *             aligned (16-byte aligned to allow the one-grid path below).
 *             Its first 256 bytes are a header that must be zero-filled
 *             before the workspace's first use and is not written by the
 *             caller after that: every call leaves it ready for the next.
 *             The rest is scratch (amax partials).  Calls that share a
 *             workspace must be ordered on one stream.
 *             Per tensor, when x is dense (ldx == cols), 16-byte aligned and
 *             small enough to sit on chip (in registers up to 24 KiB per SM,
 *             else in shared memory up to 208 KiB per SM), one grid does
 *             both passes: each CTA holds its part of x, the CTAs meet at a
 *             barrier in the header (so the grid's CTAs, at most one per SM,
 *             must all be resident at once), and x is read once.  A CTA that
 *             waits there for over a second gives up: its part of q is NaN
 *             codes (and s is NaN if that CTA is the first, which writes
 *             it), and header word 1 (bytes 4-7) becomes nonzero (a record for the caller; no kernel reads
 *             it).  Every CTA still arrives at the barrier, so once all the
 *             call's CTAs have finished the header is ready for the next
 *             call again.  Only a header whose words were written by
 *             something other than these kernels needs zero-filling again.
 * Requires rows, cols >= 0, ldx >= cols; x, q, scale 4-byte aligned.
 * Vector paths are taken when x/q are 16-byte aligned and cols, ldx are
 * multiples of 8; other shapes take a scalar path with the same results.
 * rows * cols == 0 enqueues nothing and returns FRT_OK (scale is not written).
 * ---------------------------------------------------------------------- */
size_t frt_quantize_workspace_bytes(int64_t rows, int64_t cols, frt_scale_mode mode);

frt_status frt_quantize_e4m3(const void* x, frt_dtype x_dtype, int64_t rows, int64_t cols,
                             int64_t ldx, frt_scale_mode mode, frt_dtype out_fmt,
                             const float* static_scale, uint8_t* q, float* scale,
                             void* workspace, size_t workspace_bytes, frt_stream_t stream);

/* ------------------------------------------------------------------------
 * Quantization without allocation.  The source pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory --
 * a real-time control loop that forbids allocator calls once it runs, a
 * plugin that only receives raw device pointers from its host application,
 * or code recording a CUDA graph in a mode where allocating would break the
 * capture.  It computes exactly what frt_quantize_e4m3 computes, with the
 * same arguments minus the workspace: the workspace header and the amax
 * partials live in a fixed array inside the library (256 bytes + 1 MiB,
 * 262144 partials), which every GPU that loads the library keeps until the
 * process exits.
 *   - Nothing is allocated or freed, by this call or by any routine it calls.
 *   - Size limit (only when static_scale is NULL): the workspace that
 *     frt_quantize_workspace_bytes() reports must be at most 256 bytes +
 *     1 MiB -- always
 *     true per tensor; per column ceil(rows / 64) * cols <= 262144.  Larger
 *     shapes return FRT_ERR_UNSUPPORTED_SHAPE and enqueue nothing.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - All calls share the one array, and each call overwrites the partials
 *     it reads and leaves the header ready for the next call, so nothing needs
 *     clearing between calls; calls that overlap on the GPU (different
 *     streams, no ordering) race on it.  A one-grid call that gave up at
 *     its barrier (NaN scale and NaN codes, see frt_quantize_e4m3) still
 *     leaves the header ready for the next call once all its CTAs have
 *     finished (header word 1 keeps the give-up record; no kernel reads it).
 * ---------------------------------------------------------------------- */
frt_status frt_quantize_e4m3_noalloc(const void* x, frt_dtype x_dtype, int64_t rows, int64_t cols,
                                     int64_t ldx, frt_scale_mode mode, frt_dtype out_fmt,
                                     const float* static_scale, uint8_t* q, float* scale,
                                     frt_stream_t stream);

/* ------------------------------------------------------------------------
 * FNUZ -> OCP re-encoding of n E4M3 bytes ("Real-time VLA inference on AMD
 * hardware", "Different FP8 representation").  Each output byte is the OCP
 * code of the FNUZ byte's value: exponent field e >= 2 keeps sign and
 * mantissa with field e - 1 (exact); the 15 smallest FNUZ magnitudes land
 * on the OCP subnormal grid and round half to even (8 of them are ties), a
 * negative value rounding to zero becomes 0x80; the FNUZ NaN 0x80 -> 0x7f.
 * in == out (in place) is allowed; otherwise the ranges must not overlap.
 * n == 0 enqueues nothing.
 * ---------------------------------------------------------------------- */
frt_status frt_fnuz_to_ocp(const uint8_t* in, uint8_t* out, size_t n, frt_stream_t stream);

/* ------------------------------------------------------------------------
 * Load-time weight packing ("Real-time VLA inference on AMD hardware",
 * "Packing around the instruction"; merged gate/up = concatenate the
 * weights along N before packing, "Merging gate and up").
 *
 * W is logical [K x N], row-major with row stride ldw (column n = output
 * channel).  The packed buffer stores W^T in tiles of 128 channels x 128
 * bytes of K:
 *   NB = ceil(N / 128), KB = ceil(K * esize / 128)  (esize 1 for E4M3, 2 for bf16)
 *   tile (nb, kb) at byte offset (nb * KB + kb) * 16384;
 *   channel r = n - 128 nb owns bytes [r*128, r*128 + 128) of the tile;
 *   byte j of its 128 K-bytes (element k = kb*128/esize + j/esize,
 *   little-endian for bf16) sits at ((j / 16) ^ (r % 8)) * 16 + j % 16.
 *   Padding (n >= N, k >= K) is zero.
 * A tile copied byte for byte into 1024-byte-aligned shared memory is the
 * 128-byte-swizzled K-major operand image the tensor cores read.
 *
 * w_dtype -> packed_dtype:  FRT_F32 -> FRT_BF16 (round to nearest even),
 *                           FRT_BF16 -> FRT_BF16 (copy),
 *                           FRT_E4M3_OCP -> FRT_E4M3_OCP (bytes, copy).
 * packed must be 16-byte aligned and hold frt_packed_weight_bytes() bytes.
 * Returns 0 from frt_packed_weight_bytes for an unsupported packed_dtype.
 * ---------------------------------------------------------------------- */
size_t frt_packed_weight_bytes(int64_t K, int64_t N, frt_dtype packed_dtype);

frt_status frt_pack_weights(const void* w, frt_dtype w_dtype, int64_t K, int64_t N, int64_t ldw,
                            frt_dtype packed_dtype, void* packed, size_t packed_bytes,
                            frt_stream_t stream);

/* ------------------------------------------------------------------------
 * GEMMs with the fused epilogue ("Real-time VLA inference on AMD hardware",
 * "FP8 helps the encoder and hurts the decoder" and "Merging gate and up").
 *
 *   acc[m, n] = sum_k a[m, k] * w[k, n]            (fp32 accumulation)
 *   v         = acc * (a_scale * w_scale[n]) + bias[n]
 *   v         = gelu_tanh(v)   if act == FRT_ACT_GELU_TANH and n < act_cols
 *   out[m, n] = bf16(v)        (round to nearest even)
 *
 * act == FRT_ACT_GEGLU fuses the GeGLU of a merged gate/up layer ("Merging
 * gate and up"): w is [K x N] with the gate's F = N / 2 channels first and
 * the up channels after them (w_scale and bias likewise, N floats), and
 *   out[m, j] = bf16(gelu_tanh(v[m, j]) * v[m, F + j]),  0 <= j < F,
 * so out is [M x F] (ldo >= F); act_cols is ignored.  Requires N % 256 == 0
 * (else FRT_ERR_UNSUPPORTED_SHAPE).
 *
 * a_q / a   : [M x K] row-major, row stride lda; E4M3 OCP bytes (FP8) or
 *             bf16 (BF16); 16-byte aligned, lda * esize a multiple of 16.
 * a_scale   : device, 1 float (the activation's per-tensor dequant scale).
 * w_packed  : from frt_pack_weights with the same K and N (FRT_E4M3_OCP for
 *             frt_gemm_fp8, FRT_BF16 for frt_gemm_bf16); 16-byte aligned.
 *             Load-time data: the kernel starts fetching weight tiles before
 *             it waits for the previous kernel on the stream (programmatic
 *             dependent launch), so w_packed must be complete before that
 *             previous kernel started (pack at load time and synchronise, or
 *             leave at least one other kernel between the pack and the GEMM).
 *             Everything else (a, a_scale, w_scale, bias, out) may come from
 *             the previous kernel.
 * w_scale   : device, N floats (per output channel); NULL means 1.
 *             Required (non-NULL) for frt_gemm_fp8.
 * bias      : device, N floats; NULL means 0.
 * out       : bf16 [M x N], row stride ldo; 16-byte aligned, ldo a multiple of 8.
 * act_cols  : number of leading output columns the activation applies to
 *             (0 <= act_cols <= N; a merged gate/up GEMM passes N/2).
 * workspace : optional device scratch for split-K, 256-byte aligned, of at
 *             least frt_gemm_workspace_bytes() bytes (that function returns
 *             0 when the shape's plan has no use for one; a_dtype is
 *             FRT_E4M3_OCP for frt_gemm_fp8, FRT_BF16 for frt_gemm_bf16).
 *             It must be zero-filled before its first use.  Every call
 *             returns the arrival counters it holds to zero, so it is reused
 *             as it is (the rest of it holds dead partial sums), unless
 *             dev_status reports a timeout: then the caller zero-fills it
 *             again.  Calls
 *             that share a workspace must be ordered on one stream.  With
 *             NULL, a misaligned pointer or fewer bytes the GEMM takes a plan
 *             that needs none.  Either way split-K partial sums are added in
 *             a fixed order (across the CTAs of a thread-block cluster in
 *             shared memory, or through the workspace), so a given shape and
 *             workspace choice give bit-identical results run to run.
 * dev_status: optional device int.  Every wait inside the kernels is
 *             bounded (about one second); if one expires the kernel writes a
 *             nonzero code there (the first writer wins), abandons its tile
 *             and exits.  The caller reads it after synchronising; nonzero
 *             means the output is invalid.  The caller zeroes it once.
 * Requires M, N, K >= 1; N % 16 == 0; K % 32 == 0 (FP8) or K % 16 == 0
 * (BF16).  Any M works (row tails are masked).
 * ---------------------------------------------------------------------- */
size_t frt_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, frt_dtype a_dtype);

/* The launch plan frt_gemm_fp8 (a_dtype FRT_E4M3_OCP) or frt_gemm_bf16
 * (FRT_BF16) takes for an M x N x K problem given a usable workspace of
 * workspace_bytes bytes (with act != FRT_ACT_GEGLU; a GeGLU plan on CTA
 * pairs never splits K), as one line of space-separated key=value fields:
 *   kind    pair (256-row tiles on CTA pairs) or swap (M <= 128: channels on
 *           the MMA's M side);
 *   bn      tile width (channels for pair, rows for swap);
 *   kbs     128-byte k-blocks per pipeline stage; stages: pipeline depth;
 *   splits  split-K factor; global: 1 when the split meets in the workspace;
 *   tiles   output tiles the grid walks;
 *   grid    X,Y,Z CTAs; cluster: X,Y,Z CTAs; smem: bytes per CTA.
 * The same shape always gets the same plan (on one device).  Writes at most
 * buf_len bytes including the terminating NUL (nothing when buf is NULL or
 * buf_len is 0) and returns the length of the whole line, like snprintf;
 * returns -1 when the arguments do not describe a supported problem.  Needs
 * the current CUDA device (the plan depends on its SM count and on how many
 * clusters fit); launches nothing. */
int frt_gemm_describe(int64_t M, int64_t N, int64_t K, frt_dtype a_dtype, size_t workspace_bytes,
                      char* buf, size_t buf_len);

frt_status frt_gemm_fp8(const uint8_t* a_q, int64_t lda, const float* a_scale,
                        const void* w_packed, const float* w_scale, const float* bias,
                        int64_t M, int64_t N, int64_t K, frt_act act, int64_t act_cols,
                        void* out, int64_t ldo, void* workspace, size_t workspace_bytes,
                        int* dev_status, frt_stream_t stream);

frt_status frt_gemm_bf16(const void* a, int64_t lda, const void* w_packed, const float* w_scale,
                         const float* bias, int64_t M, int64_t N, int64_t K, frt_act act,
                         int64_t act_cols, void* out, int64_t ldo, void* workspace,
                         size_t workspace_bytes, int* dev_status, frt_stream_t stream);

/* ------------------------------------------------------------------------
 * GEMM that also takes the next FP8 layer's activation scale from its own
 * output.  The per-layer activation quantize is what the method spends
 * separate launches and passes on between the GEMMs ("Real-time VLA
 * inference on AMD hardware", "Fusing the BF16 decoder boundary", on the
 * launch count of a replayed forward); the part of it that reads the whole
 * tensor, the amax, is taken here in the epilogue of the GEMM that produces
 * the tensor, so the quantize left is one encode pass over the stored output
 * (frt_quantize_e4m3 with static_scale = scale).
 *
 * Computes exactly what frt_gemm_fp8 / frt_gemm_bf16 compute (same arguments,
 * same out) and, in the same launch,
 *   scale[0] = amax / 448 over the bf16 values out[0:M, 0:scale_cols]
 *              (NaN ignored; 1 if amax == 0; one IEEE fp32 division),
 * which is bit for bit the scale frt_quantize_e4m3(out[:, :scale_cols], per
 * tensor, OCP) computes; quantizing that view with static_scale = scale then
 * gives the same bytes as the dynamic quantize.
 *
 * scale_cols     : 1 <= scale_cols <= the output's columns (N, or N / 2 for
 *                  FRT_ACT_GEGLU), a multiple of 8 (else
 *                  FRT_ERR_UNSUPPORTED_SHAPE): the next layer reads the
 *                  first scale_cols columns.
 * scale          : device, receives the scale (1 float); required.
 * scale_workspace: device memory of frt_gemm_next_scale_workspace_bytes()
 *                  bytes, 16-byte aligned, zero-filled before its first use;
 *                  each CTA folds its maximum into it and the last one to do
 *                  so writes the scale and leaves it zero again.  No CTA
 *                  waits for another.  Calls that share it must be ordered
 *                  on one stream.
 * workspace, dev_status, stream: as for frt_gemm_fp8.
 * Allocates nothing; legal under stream capture.
 * ---------------------------------------------------------------------- */
size_t frt_gemm_next_scale_workspace_bytes(void);

frt_status frt_gemm_fp8_next_scale(const uint8_t* a_q, int64_t lda, const float* a_scale,
                                   const void* w_packed, const float* w_scale, const float* bias,
                                   int64_t M, int64_t N, int64_t K, frt_act act, int64_t act_cols,
                                   void* out, int64_t ldo, int64_t scale_cols, float* scale,
                                   void* scale_workspace, size_t scale_workspace_bytes,
                                   void* workspace, size_t workspace_bytes, int* dev_status,
                                   frt_stream_t stream);

frt_status frt_gemm_bf16_next_scale(const void* a, int64_t lda, const void* w_packed,
                                    const float* w_scale, const float* bias, int64_t M, int64_t N,
                                    int64_t K, frt_act act, int64_t act_cols, void* out,
                                    int64_t ldo, int64_t scale_cols, float* scale,
                                    void* scale_workspace, size_t scale_workspace_bytes,
                                    void* workspace, size_t workspace_bytes, int* dev_status,
                                    frt_stream_t stream);

/* ------------------------------------------------------------------------
 * NVFP4: 4-bit E2M1 values with block scales ("FlashRT" article, section 7.2
 * "NVFP4 path" for the pi0.5 encoder FFN, and the use_fp4 / fp4_layers
 * switches of its load_model listing; the pages give no formula).  Read as:
 * E2M1 elements (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; sign bit; -0 kept),
 * one E4M3 scale (OCP encoding, sign bit clear) per 16 consecutive elements
 * along the reduction dimension K, one fp32 scale g per tensor.  For a
 * tensor x, every step an IEEE fp32 operation rounded to nearest even:
 *   g    = amax(x) / (6 * 448)  (1 if amax is 0; NaN ignored), or given
 *   d    = 6 * g
 *   sb   = E4M3(b / d), b = max |x| over the 16-element block (saturating)
 *   e    = value(sb) * g
 *   q_i  = E2M1(x_i / e), round to nearest even, saturating at +-6, the sign
 *          kept for a value rounding to 0; NaN -> +0; q = 0 where e == 0
 *   x_i ~= value(q_i) * value(sb) * g
 *
 * Codes are stored two per byte along K, element 2i in the low nibble.
 * Block scales are stored "tiled", the layout the GEMM copies into tensor
 * memory: for V vectors (rows of an activation, output channels of a
 * weight), padded to a multiple of 128, the scale of vector v, block j is
 * byte ((v / 128) * (K / 64) + j / 4) * 512 + 16 * (v % 32)
 *       + 4 * ((v % 128) / 32) + j % 4;
 * padded vectors have scale 0.  frt_nvfp4_scale_bytes() is that buffer's
 * size (0 unless K % 64 == 0).
 *
 * frt_quantize_nvfp4: x [rows x cols] (FRT_BF16 or FRT_F32, row stride ldx,
 *   16-byte aligned, ldx * element size a multiple of 16).
 *   blocks_along_rows == 0: the vectors are the rows, K = cols (an
 *     activation [M x K]); q is [rows x cols / 2] bytes.
 *   blocks_along_rows != 0: the vectors are the columns, K = rows (a weight
 *     W[K x N]); q is [rows / 2 x cols] bytes (byte (i, n) holds elements
 *     (2i, n) low and (2i + 1, n) high): pack it for the GEMM with
 *     frt_pack_weights(q as bytes [K/2 x N], FRT_E4M3_OCP).
 *   K % 64 == 0 (else FRT_ERR_UNSUPPORTED_SHAPE); q 16-byte aligned.
 *   sf: device, sf_bytes >= frt_nvfp4_scale_bytes(V, K).
 *   static_scale: device, g, or NULL to take g from x's amax; scale receives
 *   g (may be NULL).  workspace: 16 bytes (frt_quantize_nvfp4_workspace_bytes),
 *   16-byte aligned, zero-filled before its first use and left zero by every
 *   call; needed when static_scale is NULL; calls sharing it are ordered on
 *   one stream.  Two launches (amax, encode), one with a static scale.
 *
 * frt_gemm_nvfp4: out = bf16(act(acc * (g_a * g_w) + bias[n])) with
 *   acc[m, n] = sum_k value(qa[m,k]) value(sa[m,k/16]) value(qw[k,n]) value(sw[n,k/16])
 *   in fp32 on the tensor cores (block-scaled MMA), GELU on the first
 *   act_cols columns (act FRT_ACT_NONE or FRT_ACT_GELU_TANH).
 *   a_q: [M x K/2] codes, row stride lda BYTES (lda >= K/2, lda % 16 == 0);
 *   a_sf: tiled scales of the M rows; a_scale: g_a (1 float, NULL = 1).
 *   w_packed: frt_pack_weights of the weight's [K/2 x N] code bytes;
 *   w_sf: tiled scales of the N channels; w_scale: g_w (1 float, NULL = 1).
 *   bias: N floats or NULL.  out: bf16 [M x N], row stride ldo (ldo % 8 ==
 *   0).  K % 256 == 0 and N % 16 == 0 (else FRT_ERR_UNSUPPORTED_SHAPE); all
 *   pointers 16-byte aligned.  The weights are load-time data (as for
 *   frt_gemm_fp8).  dev_status as for frt_gemm_fp8.  Allocates nothing;
 *   legal under stream capture.
 * ---------------------------------------------------------------------- */
size_t frt_nvfp4_scale_bytes(int64_t vectors, int64_t K);

size_t frt_quantize_nvfp4_workspace_bytes(void);

frt_status frt_quantize_nvfp4(const void* x, frt_dtype x_dtype, int64_t rows, int64_t cols,
                              int64_t ldx, int blocks_along_rows, const float* static_scale,
                              uint8_t* q, uint8_t* sf, size_t sf_bytes, float* scale,
                              void* workspace, size_t workspace_bytes, frt_stream_t stream);

frt_status frt_gemm_nvfp4(const uint8_t* a_q, int64_t lda, const uint8_t* a_sf,
                          const float* a_scale, const void* w_packed, const uint8_t* w_sf,
                          const float* w_scale, const float* bias, int64_t M, int64_t N, int64_t K,
                          frt_act act, int64_t act_cols, void* out, int64_t ldo, int* dev_status,
                          frt_stream_t stream);

/* ------------------------------------------------------------------------
 * The BF16 decoder block boundary in one kernel ("Real-time VLA inference on
 * AMD hardware", "Fusing the BF16 decoder boundary"), for each row m of an
 * [M x H] tensor:
 *   r[m, j]      = bf16(fp32(residual[m, j] + output[m, j] * gate[m, j]))
 *                  (one fused multiply-add in fp32, then round to bf16)
 *   inv[m]       = 1 / sqrt(mean_j r[m, j]^2 + eps)                (fp32)
 *   normalized   = bf16(r * inv * (1 + scale) + shift)
 *   next_gate    = gate part of style
 * style is [M x 3H]: scale in columns [0, H), shift in [H, 2H), the next
 * block's gate in [2H, 3H) (the page names the steps, not this layout: it is
 * a reading).  residual is updated in place to r.  All tensors bf16,
 * row-major and contiguous, 16-byte aligned; normalized and next_gate are
 * [M x H] outputs.  Requires H % 8 == 0 and H <= 4096 (else
 * FRT_ERR_UNSUPPORTED_SHAPE), eps >= 0.  M == 0 enqueues nothing.  Legal
 * under stream capture; allocates nothing.
 * ---------------------------------------------------------------------- */
frt_status frt_gate_residual_ada_norm_bf16(void* residual, const void* output, const void* gate,
                                           const void* style, int64_t M, int64_t H, float eps,
                                           void* normalized, void* next_gate, frt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FRT_H_ */
