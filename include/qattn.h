/*
 * qattn -- quantized flash-attention prefill for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libqattn.so.  The recipe it implements:
 *
 *   - K's per-channel mean is subtracted first.  Every score of a query row
 *     then moves by the same q.mu, which softmax ignores, so the result is
 *     unchanged while K's outlier channels shrink ("int8 Flash Attention on
 *     RDNA4: QK Wants Integers, PV Wants FP8", section "K's outliers, and the
 *     subtraction softmax does not notice").
 *   - Q and K become symmetric int8 codes with fp32 scales s = amax / 127
 *     ("QFlash: Bridging Quantization and Memory Efficiency in Vision
 *     Transformer Attention", section 4, eq. (1)-(2)); the score tile is the
 *     exact integer dot product of the codes (same page, eq. (3)).
 *   - The online softmax runs in fp32 with a running row maximum, so every
 *     P = exp(s - m) is <= 1 (ZINC post, section "The scale P needs is
 *     already sitting in a register").
 *   - P is scaled by the static 448 and rounded to fp8 e4m3; V is e4m3 with
 *     one fp32 scale per channel; PV accumulates in fp32 (ZINC post, section
 *     "fp8 is not faster, it is shaped correctly").
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers owned by the caller, unless stated.  The
 *     library allocates no device memory of its own except one error word per
 *     device.  Scratch memory is the caller's `workspace` of at least
 *     qattn_workspace_size() bytes; its contents need not be initialised.
 *   - Tensors are row-major.  Q-like tensors are [B][Hq][Nq][d], K/V-like
 *     tensors [B][Hkv][Nk][d].  bf16 tensors are passed as uint16_t bit
 *     patterns.  Every tensor pointer must be 16-byte aligned.  Outputs are
 *     dense.  The pre-pass calls (qattn_smooth_k, qattn_quantize_qk,
 *     qattn_quantize_v, qattn_prepare) also read inputs at any strides: an
 *     input's `*_strides` array gives its 4 strides in elements, in [B][H][N][d]
 *     order; the last must be 1 and the others non-negative multiples of 16
 *     bytes (so every row starts on a 16-byte boundary).  NULL = dense.  A
 *     packed projection output (e.g. [B][N][3][H][d] viewed as Q, K and V)
 *     is read in place, with no copy.
 *   - Supported head dims: d in {32, 64, 128}.  Hq must be a multiple of Hkv;
 *     query head h reads KV head h / (Hq / Hkv).  Limits (else
 *     QATTN_ERR_UNSUPPORTED): Nq, Nk <= 65535 * 128 and B * Hq <= 65535.
 *   - All calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Arguments are validated on the host first: an
 *     invalid call returns a status and launches nothing.  A launch failure
 *     returns QATTN_ERR_CUDA.  No call aborts or throws.
 *   - Empty problems (B, Hq or Nq equal to 0) return QATTN_OK and launch
 *     nothing.
 *   - Kernels never wait forever: a pipeline wait that exceeds its time limit
 *     makes the kernel record QATTN_ERR_TIMEOUT in the device error word and
 *     return early; qattn_get_error() reports it.
 *   - Launch log: with the environment variable QATTN_LOG set (to anything
 *     but "" or "0"; read once, at the library's first call), every call that launches
 *     work prints one line to stderr, "[qattn] <entry point> <shape>: <the
 *     kernels it launches>", and qattn_fwd_kernel_choice prints its answer.
 *     Unset, the library prints nothing.
 */
#ifndef QATTN_H_
#define QATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* qattn_stream_t; /* same type as cudaStream_t */

typedef enum {
  QATTN_OK = 0,
  QATTN_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad shape, bad enum */
  QATTN_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. d = 96)      */
  QATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed            */
  QATTN_ERR_TIMEOUT = 4,      /* a kernel's pipeline wait ran out (device)    */
  QATTN_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required   */
  QATTN_ERR_BOUNDS = 6        /* checked build: a kernel skipped an access whose
                                 index fell outside its buffer (device)        */
} qattn_status;

/* Scale granularity of Q and K codes ("QFlash", section 3.3: per tensor,
 * per head or per token; finer is allowed here because the softmax is fp32). */
typedef enum {
  QATTN_GRAN_TENSOR = 0, /* one scale for the whole tensor                   */
  QATTN_GRAN_HEAD = 1,   /* one scale per (batch, head): [B][H]              */
  QATTN_GRAN_BLOCK = 2   /* one per (batch, head, 128 tokens): [B][H][ceil(N/128)] */
} qattn_gran;

typedef enum { QATTN_BF16 = 0, QATTN_F32 = 1, QATTN_I8 = 2, QATTN_E4M3 = 3 } qattn_dtype;

/* Tokens per scale block and keys per softmax block. */
#define QATTN_BLOCK 128
/* q_pos0 value meaning "Nk - Nq" (the last query sits on the last key). */
#define QATTN_POS0_BOTTOM_RIGHT INT64_MIN

typedef struct {
  int64_t B, Hq, Hkv, Nq, Nk, d;
} qattn_shape;

/* How P is quantized for the PV product (qattn_params.pv_mode). */
typedef enum {
  QATTN_PV_E4M3 = 0,  /* the recipe: e4m3(448 P), static scale 448              */
  QATTN_PV_INT8 = 1   /* ablation: int8 rint(127 P), static scale 127 ("int8 Flash
                         Attention on RDNA4", "Then the easy matmul turns out to be
                         the hard one": the int8 PV that flushes P < 1/254 to 0) */
} qattn_pv_mode;

/* Which kernel qattn_fwd runs (qattn_params.fwd_kernel).  Both compute the same
 * recipe; they differ only in the order of the fp32 accumulations. */
typedef enum {
  QATTN_FWD_AUTO = 0,    /* the warp-level window kernel for Nq, Nk <= 64 (d in {32, 64},
                            no causal mask, pv_mode E4M3), else the persistent kernel    */
  QATTN_FWD_TC = 1,      /* the persistent tensor-core (tcgen05) kernel                  */
  QATTN_FWD_SHORT = 2    /* the warp-level kernels for short non-causal key sequences:
                            d in {32, 64}, 1 <= Nk <= 256, pv_mode E4M3, no causal mask
                            (else QATTN_ERR_UNSUPPORTED); no workspace, reads the int8 K
                            codes (k_carrier unused)                                    */
} qattn_fwd_kernel;

typedef struct {
  int32_t causal;           /* 1: key k is visible to query i iff k <= q_pos0 + i   */
  int32_t q_gran;           /* qattn_gran of the Q codes                           */
  int32_t k_gran;           /* qattn_gran of the K codes                           */
  int32_t out_dtype;        /* QATTN_F32 or QATTN_BF16                             */
  int64_t q_pos0;           /* key position of query row 0, or QATTN_POS0_BOTTOM_RIGHT */
  float sm_scale;           /* softmax scale; 0 -> fp32(1/sqrt(d))                 */
  int32_t pv_mode;          /* qattn_pv_mode; 0 for the recipe                     */
  int64_t bias_head_stride; /* elements between heads' bias matrices; 0 = shared   */
  int64_t kv_capacity;      /* qattn_decode: rows per (batch, KV head) in the cache
                               arrays (>= Nk, the rows in use); 0 = Nk               */
  int32_t fwd_kernel;       /* qattn_fwd_kernel; 0 = automatic                      */
} qattn_params;

/* Library version (major * 10000 + minor * 100 + patch). */
int qattn_version(void);

/* Human-readable text of a status.  Never NULL; the string is static. */
const char* qattn_status_string(qattn_status s);

/* Bytes of workspace that every entry point below accepts for this shape and
 * parameters (the maximum over them).  0 for an empty problem. */
size_t qattn_workspace_size(const qattn_shape* shape, const qattn_params* params);

/* Row stride, in bytes, of the transposed e4m3 V written by qattn_quantize_v:
 * Nk rounded up to a multiple of 16 (a TMA stride must be 16-byte aligned). */
int64_t qattn_v_ld(int64_t Nk);

/* a1 -- K channel mean ("int8 Flash Attention on RDNA4", section "K's outliers,
 * and the subtraction softmax does not notice": one reduction over the K
 * block, reused by every query tile).
 *   K          bf16 [B][Hkv][Nk][d]; k_strides as in the conventions (NULL = dense)
 *   k_mean  fp32 [B][Hkv][d] (out):
 *           mu = fp32( fp64( sum_t round_half_even(K * 2^24) ) * 2^-24 / Nk )
 *           The int64 fixed-point sum makes the result independent of the
 *           summation order.  Exact while Nk * max|K| < 2^29 (the sum stays
 *           below 2^53); Nk = 0 gives mu = 0.
 */
qattn_status qattn_smooth_k(const uint16_t* K, const int64_t* k_strides, const qattn_shape* shape,
                            float* k_mean, void* workspace, size_t workspace_bytes,
                            qattn_stream_t stream);

/* a2 -- Q/K to int8 codes ("QFlash", section 4, eq. (1)-(2)).
 * For each scale granule:  amax = max |x|;  inv = fp32(127 / amax) (0 if amax
 * is 0);  code = clamp(round_half_even(fp32(x * inv)), -127, 127);
 * scale = fp32(amax / 127).
 *   Q            bf16 [B][Hq][Nq][d]                          x = fp32(Q)
 *   K, k_dtype   QATTN_BF16: bf16 [B][Hkv][Nk][d];             x = fp32(fp32(K) - k_mean)
 *                QATTN_I8:   int8 codes of an int8 KV cache, used as they are
 *                            (dense only: QATTN_ERR_UNSUPPORTED otherwise).
 *   q_strides, k_strides  as in the conventions (NULL = dense)
 *   k_mean       fp32 [B][Hkv][d] (BF16 K; NULL = no mean subtraction)
 *   k_chan_scale fp32 [B][Hkv][d] per-channel scale of int8 K codes (I8 K only).
 *                It is folded into Q before Q is quantized,
 *                x = fp32(fp32(Q) * k_chan_scale[b][h / (Hq/Hkv)][c]), so the
 *                integer dot product with the stored codes stays exact, and
 *                every K scale written is 1.
 *   q_codes      int8 [B][Hq][Nq][d] (out)
 *   q_scales     fp32, params->q_gran layout (out)
 *   k_codes      int8 [B][Hkv][Nk][d] (out; BF16 K only, ignored for I8 K)
 *   k_scales     fp32, params->k_gran layout (out)
 *   k_carrier    NULL, or fp16 [B][Hkv][Nk][d] (out): the K codes (those
 *                written to k_codes, or the I8 K given) as exact fp16 values,
 *                the operand form of the tensor-core product; hand it to
 *                qattn_fwd to spare it a conversion pass.
 * Nk = 0: only Q is quantized; K, k_codes, k_scales and k_carrier may be NULL
 * and nothing is written for K.
 */
qattn_status qattn_quantize_qk(const uint16_t* Q, const int64_t* q_strides, const void* K,
                               const int64_t* k_strides, qattn_dtype k_dtype,
                               const float* k_mean, const float* k_chan_scale,
                               const qattn_shape* shape, const qattn_params* params,
                               int8_t* q_codes, float* q_scales, int8_t* k_codes,
                               float* k_scales, uint16_t* k_carrier, void* workspace,
                               size_t workspace_bytes, qattn_stream_t stream);

/* a3 -- V to e4m3 with one fp32 scale per (batch, KV head, channel) (ZINC
 * post, "fp8 is not faster": e4m3 PV; the per-channel scale factors out of the
 * PV sum onto the output channel).
 *   V, v_dtype   QATTN_BF16: bf16 [B][Hkv][Nk][d];  x = fp32(V)
 *                QATTN_I8:   int8 codes [B][Hkv][Nk][d] with v_chan_scale
 *                            fp32 [B][Hkv][d];       x = fp32(code)
 *   v_strides    as in the conventions (NULL = dense)
 *   amax_c = max_t |x|;  v8 = e4m3_rn_satfinite(fp32(x * fp32(448 / amax_c)))
 *   v_scales (out) fp32 [B][Hkv][d]: amax_c / 448 (BF16), or
 *                  fp32(fp32(v_chan_scale * amax_c) / 448) (I8)
 *   v8t (out)      e4m3 bytes [B][Hkv][d][ldv], TRANSPOSED (key index
 *                  fastest); bytes for keys Nk..ldv-1 are written as 0.
 *   ldv            row stride in bytes, >= qattn_v_ld(Nk), multiple of 16.
 */
qattn_status qattn_quantize_v(const void* V, const int64_t* v_strides, qattn_dtype v_dtype,
                              const float* v_chan_scale, const qattn_shape* shape,
                              uint8_t* v8t, int64_t ldv,
                              float* v_scales, void* workspace, size_t workspace_bytes,
                              qattn_stream_t stream);

/* a1-a3 in one or two launches, for bf16 Q, K and V: the same outputs, bit
 * for bit, as qattn_smooth_k, then qattn_quantize_qk (k_mean given, k_dtype
 * QATTN_BF16), then qattn_quantize_v (QATTN_BF16).
 * Block granules: launch 1 quantizes Q and reduces K's channel sums and V's
 * channel maxima (three independent jobs in one grid); launch 2 quantizes
 * K - mean (with the fp16 carriers when k_carrier is not NULL) and writes V's
 * transposed e4m3 codes.  Heads of at most 128 tokens with d <= 64 (e.g. Swin
 * windows): one launch, one warp per head.
 * Tensor granules (q_gran = k_gran = QATTN_GRAN_TENSOR; d in {32, 64}, Nk <=
 * 256, e.g. ViT's 197 tokens): launch 1, one warp per head, reduces max |Q|
 * and, per KV head, the channel mean, max |K - mean| and V's channel maxima,
 * and writes V's e4m3 codes; launch 2 writes the Q and K codes at the two
 * tensor scales -- two launches where the three calls take five.
 * The ZINC post's recipe runs these three steps before the attention kernel;
 * fusing them is this library's own step (fewer launches, fewer reads).
 *   Q            bf16 [B][Hq][Nq][d];  K, V  bf16 [B][Hkv][Nk][d]
 *   q_strides, k_strides, v_strides  as in the conventions (NULL = dense)
 *   k_mean (out) fp32 [B][Hkv][d]; the other outputs as for the three calls
 *   params       q_gran = k_gran = QATTN_GRAN_BLOCK, or both
 *                QATTN_GRAN_TENSOR within the limits above, else
 *                QATTN_ERR_UNSUPPORTED (use the three calls);
 *                Nk >= 1, else QATTN_ERR_UNSUPPORTED
 *                (qattn_prepare_launches answers which, on the host)
 *   ldv          >= qattn_v_ld(Nk), multiple of 16
 *   workspace    at least qattn_workspace_size() bytes.
 */
qattn_status qattn_prepare(const uint16_t* Q, const int64_t* q_strides, const uint16_t* K,
                           const int64_t* k_strides, const uint16_t* V, const int64_t* v_strides,
                           const qattn_shape* shape, const qattn_params* params,
                           int8_t* q_codes, float* q_scales, int8_t* k_codes, float* k_scales,
                           uint16_t* k_carrier, float* k_mean, uint8_t* v8t, int64_t ldv,
                           float* v_scales, void* workspace, size_t workspace_bytes,
                           qattn_stream_t stream);

/* qattn_quantize_v without a workspace, for callers that cannot allocate
 * device memory where they quantize V (an engine plugin handed only its
 * tensors, a serving loop that bans cudaMalloc because it can synchronise the
 * device, code running under an allocator it does not own).  The pages have no
 * counterpart to this entry point; it computes exactly what qattn_quantize_v
 * computes, with the same arguments minus the workspace.
 *   Scratch: one library-owned device array of 2^19 32-bit slots (2 MiB),
 *            held by every GPU that loads the library until the process exits.
 *   Limit:   B * Hkv * d <= 524288, else QATTN_ERR_UNSUPPORTED.
 *   Set-up:  the first call on a device looks up that array's device address
 *            (cudaGetSymbolAddress) with the device current, and again the
 *            first call in a new CUDA context of that device (after
 *            cudaDeviceReset); make such a first call before any stream
 *            capture.
 *   Sharing: every call uses the same array, which keeps the last call's
 *            contents; each call zeroes the slots it uses first.  Calls that
 *            overlap on the GPU (e.g. on two streams at once) race on the
 *            array: order them on one stream or with events.
 *   No cudaMalloc, cudaFree or allocating library routine is called.
 */
qattn_status qattn_quantize_v_noalloc(const void* V, qattn_dtype v_dtype,
                                      const float* v_chan_scale, const qattn_shape* shape,
                                      uint8_t* v8t, int64_t ldv, float* v_scales,
                                      qattn_stream_t stream);

/* a4-a10 -- fused attention forward (prefill).
 *   q_codes/q_scales, k_codes/k_scales   as written by qattn_quantize_qk
 *   k_carrier  NULL, or the fp16 carriers qattn_quantize_qk wrote for these
 *              K codes (then the workspace may be NULL / 0 bytes); with NULL
 *              the call first converts k_codes itself, in the workspace.
 *   v8t, ldv, v_scales                    as written by qattn_quantize_v
 *   bias   NULL, or fp32 [Nq][Nk] in natural-log units added to the scaled
 *          scores (one matrix per head if params->bias_head_stride != 0).
 *   O      (out) [B][Hq][Nq][d], fp32 or bf16 per params->out_dtype.
 *   lse    (out, nullable) fp32 [B][Hq][Nq]: natural log of the softmax
 *          denominator of the scaled scores (-inf for a fully masked row).
 * Per query row, over key blocks of 128 in ascending order:
 *   t = S * c_j (+ bias * log2 e), S the exact int32 score of the codes and
 *       c_j = fp32(fp32(fp32(sq * sk_j) * sm_scale) * log2 e);  masked -> -inf
 *   m' = max(m, max t);  alpha = 2^(m - m');  P = 2^(t - m') <= 1
 *   l = alpha * l + sum P;  O = alpha * O + e4m3(448 P) . V8
 *   out = O * v_scale / (448 l)   (0 for a row with no visible key)
 * Nk = 0: every row is fully masked; the call writes out = 0 and lse = -inf
 * with no attention kernel and reads no K, V or workspace argument.
 * ("QFlash", section 2.1 and Algorithm 1 for the blockwise loop; ZINC post for
 * P <= 1, the static 448 and e4m3.)  The QK^T product runs on the tensor cores
 * as exact small integers held in fp16 (kind::f16, fp32 accumulation: every
 * partial sum is an integer below 2^21, so no rounding occurs); PV runs as
 * kind::f8f6f4 e4m3 x e4m3 with fp32 accumulation.
 */
qattn_status qattn_fwd(const int8_t* q_codes, const float* q_scales, const int8_t* k_codes,
                       const uint16_t* k_carrier, const float* k_scales, const uint8_t* v8t,
                       int64_t ldv, const float* v_scales, const float* bias,
                       const qattn_shape* shape,
                       const qattn_params* params, void* O, float* lse, void* workspace,
                       size_t workspace_bytes, qattn_stream_t stream);

/* Decode on an int8 KV cache ("int8 Flash Attention on RDNA4", "What actually
 * changed for decode": at batch one both products are matrix-vector products
 * bound by the bytes of the cache, and an int8 cache halves them).  A few query
 * tokens per (batch, head) against Nk cached keys, read as stored: the K codes
 * for the scores and the V codes row-major, each V code rounded to e4m3 on the
 * fly as qattn_quantize_v rounds it.  The result is qattn_fwd's recipe on the
 * same codes (key blocks of 128 in ascending order, P relative to the running
 * max at each block), computed by a split over key blocks: every block's
 * scores and row maxima first, then each block's running max as a prefix
 * maximum, the chunks' shares of O and l, and their combination.
 *   q_codes/q_scales  as written by qattn_quantize_qk with k_dtype QATTN_I8
 *   k_codes      int8 [B][Hkv][cap][d], cap = params->kv_capacity (or Nk): the
 *                cache's K codes, rows 0..Nk-1 in use (of the mean-
 *                subtracted K; the mean lives in the cache header, "K's
 *                outliers, and the subtraction softmax does not notice")
 *   k_scales     as written by qattn_quantize_qk (all 1 for I8 K)
 *   v_codes      int8 [B][Hkv][cap][d]: the cache's V codes
 *   v_chan_scale fp32 [B][Hkv][d]: scale of each V channel's codes
 *   v_code_amax  fp32 [B][Hkv][d]: max |code| of each V channel over the
 *                cache (the cache header keeps it as tokens arrive)
 *   O, lse       as for qattn_fwd; params as for qattn_fwd (pv_mode 0, no bias)
 * Limits: 1 <= (Hq / Hkv) * Nq <= 16, d in {64, 128}, Nk >= 1 (a cache with
 * no rows in use is QATTN_ERR_UNSUPPORTED), pv_mode E4M3.  Workspace: at least
 * qattn_workspace_size() for this shape.
 */
qattn_status qattn_decode(const int8_t* q_codes, const float* q_scales, const int8_t* k_codes,
                          const float* k_scales, const int8_t* v_codes,
                          const float* v_chan_scale, const float* v_code_amax,
                          const qattn_shape* shape, const qattn_params* params, void* O,
                          float* lse, void* workspace, size_t workspace_bytes,
                          qattn_stream_t stream);

/* High-accuracy attention on an int8 KV cache with both products' other
 * operand split exact to 24 bits (Strata PR "prompt_attn_i8v3_kernel", "What
 * it does", "Operands"; "Measured": ~2e-6 max relative error against FP64).
 * Per (batch, query head): q' = fp32(q * k_chan_scale); per 64-channel group
 * s_g = fp32(max |q'| / 127) over the head's rows; X = rint(q'/s_g * 65536)
 * = h * 65536 + l * 256 + m; S = sum over groups of s_g * (h.k + l.k/256 +
 * m.k/65536) with exact integer dots against the K codes, combined in fp32;
 * an online softmax over 64-key chunks (fp32, P = 2^(t - m)); per (row,
 * chunk) s_p = max P / 127 and P's parts; O += s_p * (h.v + l.v/256 +
 * m.v/65536) against the V codes; out = O * v_chan_scale / l.
 *   Q            bf16 [B][Hq][Nq][d], device
 *   k_codes, v_codes  int8 [B][Hkv][cap][d] (cap = params->kv_capacity or Nk)
 *   k_chan_scale, v_chan_scale  fp32 [B][Hkv][d]: the codes' channel scales
 *   O, lse       as for qattn_fwd; params: causal, q_pos0, sm_scale,
 *                out_dtype, kv_capacity (granules, pv_mode and bias unused)
 * Limits: d in {64, 128}, B * Hq <= 65535.  Workspace: at least
 * qattn_workspace_size() (three fp16 planes of Q's parts and the group scales).
 * Nk = 0: out = 0 and lse = -inf, as for qattn_fwd.
 */
qattn_status qattn_fwd_exact24(const void* Q, const int8_t* k_codes, const float* k_chan_scale,
                               const int8_t* v_codes, const float* v_chan_scale,
                               const qattn_shape* shape, const qattn_params* params, void* O,
                               float* lse, void* workspace, size_t workspace_bytes,
                               qattn_stream_t stream);

/* QFlash's integer-only attention ("QFlash: Bridging Quantization and Memory
 * Efficiency in Vision Transformer Attention", Algorithm 1, sections 4.2-4.6)
 * on per-tensor int8 codes.  With s~ = fp32(fp32(fp32(sq * sk) * sm_scale) *
 * log2 e) and X0 = rint(1 / s~), per query row over key tiles of 64:
 *   S = q.k (int32);  m' = max(m, rowmax S), m starting at -2^21
 *   ShiftExp2(X <= 0) = ((R >> 1) + X0) >> -Q, X = Q X0 + R, Q = X / X0
 *       truncated toward zero (section 4.3, eq. (5)-(8))
 *   alpha = ShiftExp2(m - m');  P = ShiftExp2(S - m')
 *   Y = min((P * M) >> r, 127): P to int8 codes of scale 1/127, with
 *       ratio = fp32(127 s~), n = ceil(log2 ratio), r = 8 - n,
 *       M = rint(ratio 2^r) (section 4.4, eq. (9)-(10))
 *   l = floor(l * alpha / X0) + rowsum Y;  O = floor(O * alpha / X0) + Y.V
 *       (ScaleRelease, section 4.6: its definition is not given; this is the
 *       reading taken: the inverse scale 1/s~ approximated by the integer X0)
 *   out = clamp(floor(O / l), -127, 127): int8 codes of V's scale.
 *   q_codes  int8 [B][Hq][Nq][d], q_scale fp32[1] (device): its scale
 *   k_codes, v_codes  int8 [B][Hkv][Nk][d]; k_scale fp32[1] (device)
 *   O_codes  (out) int8 [B][Hq][Nq][d]
 *   params: sm_scale (0 -> fp32(1/sqrt(d))); causal must be 0
 * Limits: d in {32, 64, 128}, B * Hq <= 65535, 1 <= Nk <= 131072 (int32 O),
 * no mask, O_codes 16-byte aligned.  No workspace.  The scales are read on the
 * device: if s~ is not a positive finite number or 1/s~ > 2^30 the kernel
 * writes nothing and qattn_get_error() returns QATTN_ERR_INVALID_ARG.
 */
qattn_status qattn_fwd_intsoftmax(const int8_t* q_codes, const float* q_scale,
                                  const int8_t* k_codes, const float* k_scale,
                                  const int8_t* v_codes, const qattn_shape* shape,
                                  const qattn_params* params, int8_t* O_codes,
                                  qattn_stream_t stream);

/* Append T tokens to an int8 KV cache whose header keeps a running channel
 * mean of K (ZINC post, "K's outliers, and the subtraction softmax does not
 * notice": during decode K arrives one token at a time and the header keeps a
 * running mean, which lags by one token).  For token t at position
 * n = pos + t, per (batch, KV head, channel c), in fp32 with round-to-nearest:
 *   k_code = clamp(rint((K - mu) / s_k), -127, 127)   (mu of the n earlier tokens)
 *   mu     = mu + (K - mu) / (n + 1)
 *   v_code = clamp(rint(V / s_v), -127, 127);  amax = max(amax, |v_code|)
 *   K_new, V_new  bf16 [B][Hkv][T][d], device
 *   k_chan_scale, v_chan_scale  fp32 [B][Hkv][d], positive, device (the
 *                 cache's fixed per-channel scales)
 *   k_mean, v_code_amax  fp32 [B][Hkv][d], device, read and updated (the
 *                 header; zeros for an empty cache)
 *   k_codes, v_codes  int8 [B][Hkv][capacity][d], device; rows pos..pos+T-1
 *                 are written
 * Limits: 0 <= pos, pos + T <= capacity <= 2^24, 1 <= d <= 1024,
 * B * Hkv * d < 2^31.  T = 0 does nothing.  Pointers: non-null; bf16 2-byte
 * and fp32 4-byte aligned.  Asynchronous on the stream; no workspace.
 */
qattn_status qattn_kv_append(const void* K_new, const void* V_new, int64_t B, int64_t Hkv,
                             int64_t T, int64_t d, int64_t pos, int64_t capacity,
                             const float* k_chan_scale, const float* v_chan_scale,
                             float* k_mean, float* v_code_amax, int8_t* k_codes,
                             int8_t* v_codes, qattn_stream_t stream);

/* The int8 KV cache header's V part for a cache filled outside the library:
 * v_code_amax[b][h][c] = max over rows t < Nk of |v_codes[b][h][t][c]| (0 for
 * Nk = 0).  This is the per-channel maximum that qattn_kv_append keeps up to
 * date as it appends tokens and that qattn_decode turns into V's e4m3 scale
 * (ZINC post, "What actually changed for decode": the cache stores int8 codes
 * and the header carries what the kernels need about them).
 *   v_codes      int8 [B][Hkv][capacity][d], device, 16-byte aligned; rows
 *                0..Nk-1 are read (NULL allowed when Nk = 0)
 *   v_code_amax  (out) fp32 [B][Hkv][d], device, 4-byte aligned
 * Limits: d in {32, 64, 128}, 0 <= Nk <= capacity <= 2^24, B * Hkv <= 65535.
 * Asynchronous on the stream; no workspace.
 */
qattn_status qattn_kv_header_init(const int8_t* v_codes, int64_t B, int64_t Hkv, int64_t Nk,
                                  int64_t d, int64_t capacity, float* v_code_amax,
                                  qattn_stream_t stream);

/* a4 alone (debug) -- the int32 score tiles S = q_codes . k_codes^T
 * ("QFlash", eq. (3)), through the same tensor-core path as qattn_fwd.
 *   S (out) int32 [B][Hq][Nq][Nk]
 */
qattn_status qattn_debug_qk_scores(const int8_t* q_codes, const int8_t* k_codes,
                                   const qattn_shape* shape, int32_t* S, void* workspace,
                                   size_t workspace_bytes, qattn_stream_t stream);

/* Which kernel qattn_fwd runs for a shape and params (a qattn_fwd_kernel value:
 * QATTN_FWD_TC or QATTN_FWD_SHORT), or -1 if the call would be rejected
 * (invalid arguments, or QATTN_FWD_SHORT asked for a shape it does not
 * cover).  Host only, no device work. */
int qattn_fwd_kernel_choice(const qattn_shape* shape, const qattn_params* params);

/* How many kernels qattn_prepare launches for a shape and params (1 or 2; 0
 * for an empty problem), or -1 if it would reject them.  Host only. */
int qattn_prepare_launches(const qattn_shape* shape, const qattn_params* params);

/* The checked build (the library compiled with QATTN_CHECK=1, by
 * build.build(checked=True) into _lib/check/): the kernels guard the device
 * accesses whose indices they compute -- output rows and columns, scale
 * indices, cache rows, TMA coordinates -- against their buffers' extents; a
 * failing guard skips the access (nothing traps) and qattn_get_error()
 * returns QATTN_ERR_BOUNDS.  A stand-in for a memory checker where none can
 * run.  qattn_checked() is 1 in that build, 0 in the normal one (host only). */
int qattn_checked(void);

/* Runs one guard that fails for 16 of 32 threads and touches no memory: in
 * the checked build the next qattn_get_error() returns QATTN_ERR_BOUNDS, in
 * the normal build QATTN_OK -- a test of the reporting path. */
qattn_status qattn_debug_bounds_probe(qattn_stream_t stream);

/* Synchronises `stream`, then returns and clears the device error word of
 * the current device (QATTN_ERR_TIMEOUT if a kernel gave up on a wait,
 * QATTN_ERR_INVALID_ARG if a kernel found device-held scales outside its
 * domain). */
qattn_status qattn_get_error(qattn_stream_t stream);

/* Failure-path check (debug; no counterpart on the pages): one thread runs
 * the kernels' bounded pipeline wait on an mbarrier that nothing arrives at,
 * so the wait runs out after its time limit (about 2 s at the boost clock)
 * and takes the same exit as in the attention kernels: the abort flag is
 * raised, the timeout bit is set in the device error word, the kernel
 * returns.  The next qattn_get_error() then returns QATTN_ERR_TIMEOUT and
 * clears the word; the context stays usable.
 *   result  (out) device int32[2], 8-byte aligned: {1 if the wait reported
 *           success else 0, the abort flag} -- {0, 1} after a timeout.
 * QATTN_ERR_INVALID_ARG (nothing launched) for a NULL or misaligned result. */
qattn_status qattn_debug_wait_timeout(int32_t* result, qattn_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QATTN_H_ */
