// Internal launch interface between the C ABI (qattn_api.cu) and the
// kernels (quant_kernels.cu, attn_fwd.cu).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qattn {

// Launches `kernel` on stream s with programmatic stream serialization, so it
// may start while the previous kernel of the stream finishes (the kernels call
// pdl_wait before touching their inputs).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Streaming multiprocessors of the current device (1 if the query fails).
inline int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
  return n;
}

// Unique id (cuCtxGetId) of the CUDA context current on the calling thread;
// false when no context is current or the driver cannot say.  The library
// caches device addresses of its own __device__ symbols per device and per
// context, so that a context destroyed by cudaDeviceReset (and replaced by a
// new one) never leaves a stale address behind.
bool current_context_id(unsigned long long* id);

// Bits of the device error word.
constexpr unsigned int kErrTimeout = 1u;
constexpr unsigned int kErrDomain = 2u;  // device-held scales outside a kernel's domain

// The checked build's bounds-check words, one per kernel translation unit
// (qattn_check.cuh): each call reads and clears its unit's word (always 0 in
// the normal build).
unsigned int check_take_attn_fwd();
unsigned int check_take_quant();
unsigned int check_take_decode();
unsigned int check_take_short();
unsigned int check_take_exact24();
unsigned int check_take_intsm();
// One guard that fails for 16 of 32 threads, touching no memory (quant_kernels.cu).
cudaError_t launch_bounds_probe(cudaStream_t s);

struct AttnArgs {
  int B, Hq, Hkv, Nq, Nk, d;
  int causal;
  int pos0;  // key position of query row 0 (causal only)
  float sm_scale;
  int q_gran, k_gran;
  const float* q_scales;
  const float* k_scales;
  const float* v_scales;
  const float* bias;
  long long bias_head_stride;
  int pv_int8;  // P quantized as int8 rint(127 P) (ablation) instead of e4m3(448 P)
  void* out;
  int out_bf16;
  float* lse;
  unsigned int* err;
};

// ---- attn_short.cu: the recipe on the warp-level tensor cores for short
// non-causal key sequences (d in {32, 64}, Nk <= kShortMaxNk)
constexpr int kShortMaxNk = 256;
constexpr int kWindowMax = 64;  // Nq, Nk of the window kernel
bool attn_short_eligible(const AttnArgs& a);
cudaError_t launch_attn_short(const AttnArgs& a, const int8_t* q_codes, const int8_t* k_codes,
                              const uint8_t* v8t, long long ldv, cudaStream_t s);

// ---- quant_kernels.cu
// An input tensor [B][H][N][d] (bf16 or int8) at any strides, in elements: row
// t of (batch, head) bh = b H + h starts at p + b sB + h sH + t sN and its d
// elements are contiguous.  Dense: sB = H N d, sH = N d, sN = d.
struct Src {
  const void* p;
  long long sB, sH, sN;
  int H;
};
inline Src dense_src(const void* p, int H, long long N, int d) {
  return Src{p, static_cast<long long>(H) * N * d, N * d, static_cast<long long>(d), H};
}

cudaError_t launch_smooth_k(const Src& K, int BH, int Nk, int d, long long* ws, float* mu,
                            cudaStream_t s);
size_t smooth_k_ws_bytes(long long BH, long long Nk, long long d);

// One tensor to quantize per 128-token block rows (a2): X [B*H][N][d] bf16.
//   mode 0: x = X;  1: x = X - chan[b][h][:] (Hchan = H);
//   2: x = X * chan[b][h / group][:] (chan has Hchan heads, group = H / Hchan)
struct RowsJob {
  const uint16_t* X;
  long long sB, sH, sN;  // X's strides in elements (see Src)
  int H, N;
  const float* chan;
  int Hchan, group, gran;
  int8_t* codes;
  float* scales;
  float* ws_amax;  // B*H*nblk block maxima (tensor / head granules only)
  uint16_t* carrier;  // nullable: the codes again as exact fp16, same layout
  int nblk, BH;    // 128-token blocks per head; B*H (0: no job)
  float* ones;     // nullable (job 0 only): n_ones floats set to 1 by the
  long long n_ones;  // launch (the K scales of an int8 cache)
};
// Quantizes j0 (mode m0) and j1 (mode m1) in the same launches.  Supported:
// (m0, m1) = (0, 0), (0, 1), or (2, -) with j1.BH = 0.
cudaError_t launch_quantize_rows(const RowsJob& j0, int m0, const RowsJob& j1, int m1, int d,
                                 cudaStream_t s);
size_t quantize_rows_ws_bytes(long long B, long long H, long long N, int gran);
// The pre-pass for bf16 Q, K, V with block granules: jq (Q, mode 0), jk (K
// minus jk.chan = the mean it writes, mode 1), V's e4m3 transpose.  One launch
// for heads of at most 128 tokens and d <= 64, else two (ws zeroed here).
// ws: prepare_ws_bytes().
cudaError_t launch_prepare(const RowsJob& jq, const RowsJob& jk, const Src& V, int d,
                           uint8_t* v8t, long long ldv, float* v_scales, void* ws, cudaStream_t s);
size_t prepare_ws_bytes(long long BH, long long d);
int prepare_launch_count(int d, int Nq, int Nk);  // 1 for short heads, else 2
// The same pre-pass with tensor granules (jq.gran = jk.gran = 0): two launches,
// one warp per head, for d in {32, 64} and 1 <= Nk <= 256.  ws: 8 bytes (the
// two maxima, zeroed here).
bool prepare_tensor_eligible(int d, int Nq, int Nk);
cudaError_t launch_prepare_tensor(const RowsJob& jq, const RowsJob& jk, const Src& V, int d,
                                  uint8_t* v8t, long long ldv, float* v_scales, void* ws,
                                  cudaStream_t s);

cudaError_t launch_quantize_v(const Src& V, int is_i8, const float* chan, int BH, int Nk, int d,
                              uint8_t* v8t, long long ldv, float* v_scales, unsigned int* ws_amax,
                              cudaStream_t s);

cudaError_t launch_codes_to_f16(const int8_t* src, uint16_t* dst, size_t n, cudaStream_t s);

// max |code| per channel of int8 V codes [BH][rows][d], rows 0 .. Nk-1
// (out: [BH][d] fp32, zeroed first)
cudaError_t launch_v_code_amax(const int8_t* v_codes, int BH, int Nk, long long rows, int d,
                               float* out, cudaStream_t s);

// Rows that see no key (Nk = 0): out = 0 (out_bytes of it), lse = -inf for
// `rows` rows when lse is not null.
cudaError_t launch_no_key_rows(void* out, size_t out_bytes, float* lse, size_t rows, cudaStream_t s);

// ---- decode.cu
constexpr int kMaxDecodeRows = 16;  // (Hq / Hkv) * Nq rows per KV head

struct DecodeArgs {
  int B, Hq, Hkv, Nq, Nk, d;
  int causal;
  int pos0;
  float sm_scale;
  int q_gran, k_gran;
  const int8_t* q_codes;
  const float* q_scales;
  const int8_t* k_codes;
  const float* k_scales;
  const int8_t* v_codes;       // [B*Hkv][Nk][d], row-major as cached
  const float* v_chan_scale;   // [B*Hkv][d]
  const float* v_code_amax;    // [B*Hkv][d]: max |code| per channel
  void* out;
  int out_bf16;
  float* lse;
  // set by launch_decode: the split and the workspace regions
  int bpc;                        // key blocks per chunk
  int nch;                        // chunks per (batch, KV head)
  unsigned long long epoch;       // this call's tag (low 32 bits), unique per call
  unsigned long long* ctr;        // unit counter: (tag << 32) | units taken
  float* part_o;                  // [B*Hkv][nch][R][d]  chunk shares of O
  float* part_l;                  // [B*Hkv][nch][R]     their l
  float* part_m;                  // [B*Hkv][nch][R]     their running max
  unsigned long long* rec;        // [B*Hkv][nch][R]     chunk maxima: (tag << 32) | bits
  unsigned int* err;  // device error word (a bounded wait that ran out)
};
size_t decode_ws_bytes(long long B, long long Hq, long long Hkv, long long Nq, long long Nk,
                       long long d);
// tk, tv: maps over the int8 K and V codes [B*Hkv][Nk][d], box d x 128 x 1,
// 128-byte swizzle for d = 128, 64-byte for d = 64.
cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, DecodeArgs a, void* ws,
                          cudaStream_t s);
cudaError_t launch_kv_append(const uint16_t* K_new, const uint16_t* V_new, int BH, int d, int T,
                             int pos, long long cap, const float* k_chan_scale,
                             const float* v_chan_scale, float* k_mean, float* v_code_amax,
                             int8_t* k_codes, int8_t* v_codes, cudaStream_t s);

// ---- exact24.cu
struct Exact24Args {
  int B, Hq, Hkv, Nq, Nk, d;
  int causal;
  int pos0;
  float sm_scale;
  long long cap;                // cache rows per (batch, KV head)
  const void* Q;                // bf16 [B][Hq][Nq][d]
  const float* k_chan_scale;    // [B][Hkv][d]
  const int8_t* k_codes;        // [B][Hkv][cap][d]
  const int8_t* v_codes;
  const float* v_chan_scale;
  void* out;
  int out_bf16;
  float* lse;
  void* ws;                     // exact24_ws_bytes
  unsigned int* err;            // device error word (a bounded wait that ran out)
};
size_t exact24_ws_bytes(long long B, long long Hq, long long Hkv, long long Nq, long long Nk,
                        long long d);
cudaError_t launch_exact24(const Exact24Args& x, cudaStream_t s);

// ---- intsm.cu
cudaError_t launch_intsoftmax(int B, int Hq, int Hkv, int Nq, int Nk, int d, float sm_scale,
                              const int8_t* q_codes, const float* q_scale, const int8_t* k_codes,
                              const float* k_scale, const int8_t* v_codes, int8_t* out,
                              unsigned int* err, cudaStream_t s);

// 3-D tiled TMA map over a dense [planes][rows][inner] tensor (qattn_api.cu):
// row_stride_bytes between rows, plane_rows rows between planes (0 = rows);
// false if the driver entry point is missing or rejects the map.
bool encode_tiled_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
                     uint64_t rows, uint64_t planes, uint64_t row_stride_bytes, uint32_t box_inner,
                     uint32_t box_rows, CUtensorMapSwizzle swz, uint64_t plane_rows = 0);

// ---- attn_fwd.cu
// tq: int8 Q codes; tk: fp16 K carriers; tv: e4m3 V^T; to: the output
// [B*Hq][Nq][d] (bf16 or fp32) in boxes of 128-byte rows x 32 rows, 128B
// swizzle (unused, and may be left zero, for bf16 with d = 32).
cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, const AttnArgs& a, cudaStream_t s);
cudaError_t launch_qk_debug(const CUtensorMap& tq, const CUtensorMap& tk, int B, int Hq, int Hkv,
                            int Nq, int Nk, int d, int32_t* S, unsigned int* err,
                            cudaStream_t s);

}  // namespace qattn
