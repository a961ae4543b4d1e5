// The C ABI of libqattn.so (declared in include/qattn.h): host-side argument
// validation, workspace carving, TMA descriptor encoding and kernel launches.
// No entry point allocates device memory; every failure becomes a status.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <random>

#include <cuda.h>
#include <cuda_runtime.h>

#include "qattn.h"
#include "qattn_check.cuh"
#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {

bool current_context_id(unsigned long long* id) {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (!get_current || !get_id) return false;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return false;
  return get_id(c, id) == CUDA_SUCCESS;
}

}  // namespace qattn

namespace {

using qattn::AttnArgs;

// One error word per device; kernels OR error bits into it.
__device__ unsigned int g_qattn_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// The error word's device address per device, and the context it belongs to
// (0: unknown, resolved again on every call).
unsigned int* g_err_ptr[kMaxDevices] = {nullptr};
unsigned long long g_err_ctx[kMaxDevices] = {0};

// Tags of qattn_decode calls: a per-call count XOR a random per-process salt
// marks the chunk records and the unit counter a call writes in its workspace,
// so neither needs clearing between calls (stale contents carry another tag;
// the salt keeps zeros or small integers left in the memory from matching).
std::atomic<uint32_t> g_decode_count{0};
const uint32_t g_decode_salt = static_cast<uint32_t>(std::random_device{}());

uint32_t next_decode_tag() {
  for (;;) {
    const uint32_t t = (g_decode_count.fetch_add(1) + 1u) ^ g_decode_salt;
    if (t != 0u && t != 0xFFFFFFFFu) return t;
  }
}

// Device address of the error word in the current device's current context:
// cached per device and context (a new context after cudaDeviceReset resolves
// it again); nullptr on failure.
unsigned int* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned long long ctx = 0;
  const bool known = qattn::current_context_id(&ctx);
  std::lock_guard<std::mutex> lk(g_mu);
  if (known && g_err_ptr[dev] && g_err_ctx[dev] == ctx) return g_err_ptr[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_qattn_error_word) != cudaSuccess || p == nullptr) return nullptr;
  // the symbol lookup makes the device's primary context current if none was
  const bool now_known = known || qattn::current_context_id(&ctx);
  g_err_ptr[dev] = static_cast<unsigned int*>(p);
  g_err_ctx[dev] = now_known ? ctx : 0;
  return g_err_ptr[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// QATTN_LOG set to anything but "" or "0": every call that reaches its launch
// (and the host-only kernel-choice queries) prints one line on stderr naming
// the kernels it runs and the problem shape.  Read once per process.
bool log_on() {
  static const bool on = [] {
    const char* v = std::getenv("QATTN_LOG");
    return v != nullptr && v[0] != '\0' && !(v[0] == '0' && v[1] == '\0');
  }();
  return on;
}
#define QATTN_LOG_LINE(...)                         \
  do {                                              \
    if (log_on()) {                                 \
      std::fprintf(stderr, "[qattn] " __VA_ARGS__); \
      std::fputc('\n', stderr);                     \
    }                                               \
  } while (0)

const char* shape_str(const qattn_shape* s, char* buf, size_t n) {
  std::snprintf(buf, n, "B=%lld Hq=%lld Hkv=%lld Nq=%lld Nk=%lld d=%lld", static_cast<long long>(s->B),
                static_cast<long long>(s->Hq), static_cast<long long>(s->Hkv),
                static_cast<long long>(s->Nq), static_cast<long long>(s->Nk),
                static_cast<long long>(s->d));
  return buf;
}
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool valid_d(int64_t d) { return d == 32 || d == 64 || d == 128; }

// An input tensor [B][H][N][d] with element strides st (NULL: dense): the last
// stride must be 1 and the others non-negative multiples of 16 bytes (every
// row starts on a 16-byte boundary, as the vector loads need).
bool make_src(const void* p, const int64_t* st, int64_t H, int64_t N, int64_t d, int elem,
              qattn::Src* out) {
  if (!st) {
    *out = qattn::dense_src(p, static_cast<int>(H), N, static_cast<int>(d));
    return true;
  }
  if (st[3] != 1) return false;
  for (int i = 0; i < 3; ++i)
    if (st[i] < 0 || (st[i] * elem) % 16 != 0) return false;
  *out = qattn::Src{p, st[0], st[1], st[2], static_cast<int>(H)};
  return true;
}

bool is_dense(const int64_t* st, int64_t H, int64_t N, int64_t d) {
  return !st || (st[3] == 1 && st[2] == d && st[1] == N * d && st[0] == H * N * d);
}

// Shape checks shared by all entry points.  Returns QATTN_OK, or an error.
qattn_status check_shape(const qattn_shape* s) {
  if (!s) return QATTN_ERR_INVALID_ARG;
  if (s->B < 0 || s->Hq < 0 || s->Hkv < 0 || s->Nq < 0 || s->Nk < 0 || s->d <= 0)
    return QATTN_ERR_INVALID_ARG;
  if (s->Hkv == 0 || (s->Hq % s->Hkv) != 0) return QATTN_ERR_INVALID_ARG;
  if (!valid_d(s->d)) return QATTN_ERR_UNSUPPORTED;
  // Grid limits: 128-token tiles index gridDim.y/z (<= 65535), and (batch,
  // head) pairs index gridDim.y of the quantizers.
  const int64_t lim = int64_t{65535} * 128;
  if (s->Nq > lim || s->Nk > lim || s->B * s->Hq > 65535 || s->B > 65535)
    return QATTN_ERR_UNSUPPORTED;
  return QATTN_OK;
}

qattn_status check_params(const qattn_params* p) {
  if (!p) return QATTN_ERR_INVALID_ARG;
  if (p->q_gran < 0 || p->q_gran > 2 || p->k_gran < 0 || p->k_gran > 2) return QATTN_ERR_INVALID_ARG;
  if (p->out_dtype != QATTN_F32 && p->out_dtype != QATTN_BF16) return QATTN_ERR_INVALID_ARG;
  if (p->causal != 0 && p->causal != 1) return QATTN_ERR_INVALID_ARG;
  if (p->pv_mode != QATTN_PV_E4M3 && p->pv_mode != QATTN_PV_INT8) return QATTN_ERR_INVALID_ARG;
  if (p->bias_head_stride < 0 || p->kv_capacity < 0) return QATTN_ERR_INVALID_ARG;
  if (p->fwd_kernel < QATTN_FWD_AUTO || p->fwd_kernel > QATTN_FWD_SHORT) return QATTN_ERR_INVALID_ARG;
  if (!(p->sm_scale >= 0.f) || std::isinf(p->sm_scale)) return QATTN_ERR_INVALID_ARG;
  return QATTN_OK;
}

// The kernel qattn_fwd runs: the warp-level kernels for short non-causal key
// sequences, chosen automatically for windows (Nq, Nk <= 64, where the
// persistent kernel's 128-row tiles would be mostly empty) or when asked for;
// else the persistent one.  -1 when the requested kernel does not cover the
// shape.  Shape and params already validated.
int fwd_choice(const qattn_shape* shape, const qattn_params* params) {
  const bool short_ok = (shape->d == 32 || shape->d == 64) && !params->causal &&
                        params->pv_mode == QATTN_PV_E4M3 && shape->Nk >= 1 &&
                        shape->Nk <= qattn::kShortMaxNk;
  const bool window = short_ok && shape->Nq <= qattn::kWindowMax && shape->Nk <= qattn::kWindowMax;
  if (params->fwd_kernel == QATTN_FWD_SHORT) return short_ok ? QATTN_FWD_SHORT : -1;
  if (params->fwd_kernel == QATTN_FWD_AUTO && window) return QATTN_FWD_SHORT;
  return QATTN_FWD_TC;
}

int64_t pos0_of(const qattn_shape* s, const qattn_params* p) {
  return p->q_pos0 == QATTN_POS0_BOTTOM_RIGHT ? s->Nk - s->Nq : p->q_pos0;
}

qattn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QATTN_OK : QATTN_ERR_CUDA; }

bool empty_problem(const qattn_shape* s) { return s->B == 0 || s->Hq == 0 || s->Nq == 0; }

// Nk = 0: every row is fully masked, so out = 0 and lse = -inf, with no
// attention kernel.  Shape (non-empty) and params already validated.
qattn_status no_key_rows(const qattn_shape* shape, const qattn_params* params, void* O, float* lse,
                         cudaStream_t s) {
  const size_t rows = static_cast<size_t>(shape->B * shape->Hq * shape->Nq);
  const size_t esize = params->out_dtype == QATTN_BF16 ? 2 : 4;
  return from_cuda(qattn::launch_no_key_rows(O, rows * static_cast<size_t>(shape->d) * esize, lse, rows, s));
}

// Workspace regions of each entry point.
size_t ws_smooth(const qattn_shape* s) { return align256(qattn::smooth_k_ws_bytes(s->B * s->Hkv, s->Nk, s->d)); }
size_t ws_quant_qk(const qattn_shape* s, const qattn_params* p) {
  return align256(qattn::quantize_rows_ws_bytes(s->B, s->Hq, s->Nq, p ? p->q_gran : 0)) +
         align256(qattn::quantize_rows_ws_bytes(s->B, s->Hkv, s->Nk, p ? p->k_gran : 0));
}
size_t ws_quant_v(const qattn_shape* s) { return align256(static_cast<size_t>(s->B * s->Hkv * s->d) * 4); }
// fp16 carriers of the K codes (Q codes are widened inside the kernels).
size_t ws_carriers_k(const qattn_shape* s) { return align256(static_cast<size_t>(s->B * s->Hkv * s->Nk * s->d) * 2); }
size_t ws_fwd(const qattn_shape* s) { return ws_carriers_k(s); }
size_t ws_prepare(const qattn_shape* s) { return align256(qattn::prepare_ws_bytes(s->B * s->Hkv, s->d)); }

// 3-D tiled map over a dense [planes][rows][inner] tensor.
bool encode_3d(CUtensorMap* map, CUtensorMapDataType dt, size_t esize, const void* ptr,
               uint64_t inner, uint64_t rows, uint64_t planes, uint64_t row_stride_bytes,
               uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz,
               uint64_t plane_rows = 0) {  // rows between planes in memory; 0 = rows
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {inner, rows, planes};
  const cuuint64_t strides[2] = {row_stride_bytes, row_stride_bytes * (plane_rows ? plane_rows : rows)};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  (void)esize;
  return fn(map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace qattn {
bool encode_tiled_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
                     uint64_t rows, uint64_t planes, uint64_t row_stride_bytes, uint32_t box_inner,
                     uint32_t box_rows, CUtensorMapSwizzle swz, uint64_t plane_rows) {
  return encode_3d(map, dt, 0, ptr, inner, rows, planes, row_stride_bytes, box_inner, box_rows, swz,
                   plane_rows);
}
}  // namespace qattn

namespace {

// Map over the int8 Q codes [B*Hq][Nq][d]: one 128-row tile per load,
// unswizzled (the kernels widen it to fp16 themselves).
bool encode_q_codes(CUtensorMap* map, const void* ptr, int64_t planes, int64_t rows, int64_t d) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ptr, d, rows, planes, d,
                   static_cast<uint32_t>(d), 128, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Map over the fp16 carriers of K [B*Hkv][Nk][d].
bool encode_carrier(CUtensorMap* map, const void* ptr, int64_t planes, int64_t rows, int64_t d) {
  const uint32_t colblock = d >= 64 ? 64 : static_cast<uint32_t>(d);
  const CUtensorMapSwizzle swz = (colblock * 2 == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ptr, d, rows, planes, d * 2, colblock,
                   128, swz);
}

// Shapes the decode path serves: (Hq / Hkv) * Nq rows per KV head.
bool decode_shape_ok(const qattn_shape* s) {
  return s->Hkv > 0 && s->Nq >= 1 && (s->Hq / s->Hkv) * s->Nq <= qattn::kMaxDecodeRows &&
         (s->d == 64 || s->d == 128);
}

// The pipeline kernels' bounded mbarrier wait, run on a barrier that nothing
// arrives at: after its time limit it raises the abort flag, sets the timeout
// bit of the error word and returns false.  One thread; writes {1 if the wait
// reported success else 0, the abort flag} to result.
__global__ void wait_timeout_kernel(unsigned int* err, int* result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  abort_flag = 0;
  const uint32_t b = qattn::smem_u32(&bar);
  qattn::mbar_init(b, 1);
  qattn::fence_mbar_init();
  const bool ok = qattn::mbar_wait(b, 0, &abort_flag, err, qattn::kErrTimeout);
  result[0] = ok ? 1 : 0;
  result[1] = abort_flag;
}

}  // namespace

extern "C" {

int qattn_version(void) { return 100; }

const char* qattn_status_string(qattn_status s) {
  switch (s) {
    case QATTN_OK: return "ok";
    case QATTN_ERR_INVALID_ARG: return "invalid argument";
    case QATTN_ERR_UNSUPPORTED: return "unsupported shape or option";
    case QATTN_ERR_CUDA: return "CUDA error";
    case QATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case QATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case QATTN_ERR_BOUNDS: return "a kernel index fell outside its buffer (checked build)";
  }
  return "unknown status";
}

int64_t qattn_v_ld(int64_t Nk) { return Nk <= 0 ? 16 : ((Nk + 15) / 16) * 16; }

size_t qattn_workspace_size(const qattn_shape* shape, const qattn_params* params) {
  if (check_shape(shape) != QATTN_OK || empty_problem(shape)) return 0;
  size_t m = ws_smooth(shape);
  const size_t q = ws_quant_qk(shape, params);
  if (q > m) m = q;
  if (ws_quant_v(shape) > m) m = ws_quant_v(shape);
  if (ws_fwd(shape) > m) m = ws_fwd(shape);
  if (ws_prepare(shape) > m) m = ws_prepare(shape);
  if (decode_shape_ok(shape)) {
    const size_t dws = qattn::decode_ws_bytes(shape->B, shape->Hq, shape->Hkv, shape->Nq,
                                              shape->Nk, shape->d);
    if (dws > m) m = dws;
  }
  const size_t e24 = qattn::exact24_ws_bytes(shape->B, shape->Hq, shape->Hkv, shape->Nq, shape->Nk,
                                             shape->d);
  if (e24 > m) m = e24;
  return m;
}

qattn_status qattn_smooth_k(const uint16_t* K, const int64_t* k_strides, const qattn_shape* shape,
                            float* k_mean, void* workspace, size_t workspace_bytes,
                            qattn_stream_t stream) {
  qattn_status st = check_shape(shape);
  if (st != QATTN_OK) return st;
  if (shape->B == 0 || shape->Hkv == 0) return QATTN_OK;
  if (!k_mean || !aligned16(k_mean) || (shape->Nk > 0 && (!K || !aligned16(K)))) return QATTN_ERR_INVALID_ARG;
  qattn::Src ks;
  if (!make_src(K, k_strides, shape->Hkv, shape->Nk, shape->d, 2, &ks)) return QATTN_ERR_INVALID_ARG;
  const size_t need = ws_smooth(shape);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return QATTN_ERR_WORKSPACE;
  char sb[128];
  QATTN_LOG_LINE("qattn_smooth_k %s strided=%d: k_mean kernel (exact fixed-point channel sums)",
                 shape_str(shape, sb, sizeof sb), k_strides != nullptr);
  return from_cuda(qattn::launch_smooth_k(ks, static_cast<int>(shape->B * shape->Hkv),
                                          static_cast<int>(shape->Nk), static_cast<int>(shape->d),
                                          static_cast<long long*>(workspace), k_mean,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

qattn_status qattn_quantize_qk(const uint16_t* Q, const int64_t* q_strides, const void* K,
                               const int64_t* k_strides, qattn_dtype k_dtype,
                               const float* k_mean, const float* k_chan_scale,
                               const qattn_shape* shape, const qattn_params* params,
                               int8_t* q_codes, float* q_scales, int8_t* k_codes,
                               float* k_scales, uint16_t* k_carrier, void* workspace,
                               size_t workspace_bytes, qattn_stream_t stream) {
  qattn_status st = check_shape(shape);
  if (st != QATTN_OK) return st;
  if ((st = check_params(params)) != QATTN_OK) return st;
  if (k_dtype != QATTN_BF16 && k_dtype != QATTN_I8) return QATTN_ERR_INVALID_ARG;
  if (empty_problem(shape)) return QATTN_OK;
  const bool i8 = (k_dtype == QATTN_I8);
  if (!Q || !aligned16(Q) || !q_codes || !aligned16(q_codes) || !q_scales || (shape->Nk > 0 && !k_scales))
    return QATTN_ERR_INVALID_ARG;
  if (i8 && (!k_chan_scale || !aligned16(k_chan_scale))) return QATTN_ERR_INVALID_ARG;
  if (!i8 && shape->Nk > 0 && (!K || !aligned16(K) || !k_codes || !aligned16(k_codes))) return QATTN_ERR_INVALID_ARG;
  if (k_mean && (i8 || !aligned16(k_mean))) return QATTN_ERR_INVALID_ARG;
  if (k_carrier && !aligned16(k_carrier)) return QATTN_ERR_INVALID_ARG;
  qattn::Src qs, ks;
  if (!make_src(Q, q_strides, shape->Hq, shape->Nq, shape->d, 2, &qs)) return QATTN_ERR_INVALID_ARG;
  if (!make_src(K, k_strides, shape->Hkv, shape->Nk, shape->d, i8 ? 1 : 2, &ks)) return QATTN_ERR_INVALID_ARG;
  // int8 cache codes go to qattn_fwd as they are: dense only
  if (i8 && !is_dense(k_strides, shape->Hkv, shape->Nk, shape->d)) return QATTN_ERR_UNSUPPORTED;
  const size_t wq = align256(qattn::quantize_rows_ws_bytes(shape->B, shape->Hq, shape->Nq, params->q_gran));
  const size_t need = ws_quant_qk(shape, params);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return QATTN_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* ws_q = static_cast<float*>(workspace);
  float* ws_k = reinterpret_cast<float*>(static_cast<char*>(workspace) + wq);
  const int B = static_cast<int>(shape->B), Hq = static_cast<int>(shape->Hq);
  const int Hkv = static_cast<int>(shape->Hkv), d = static_cast<int>(shape->d);
  const int64_t nqb = (shape->Nq + 127) / 128, nkb = (shape->Nk + 127) / 128;
  qattn::RowsJob jq{};
  jq.X = Q;
  jq.sB = qs.sB;
  jq.sH = qs.sH;
  jq.sN = qs.sN;
  jq.H = Hq;
  jq.N = static_cast<int>(shape->Nq);
  jq.chan = i8 ? k_chan_scale : nullptr;
  jq.Hchan = i8 ? Hkv : 1;
  jq.group = i8 ? Hq / Hkv : 1;
  jq.gran = params->q_gran;
  jq.codes = q_codes;
  jq.scales = q_scales;
  jq.ws_amax = ws_q;
  jq.nblk = static_cast<int>(nqb);
  jq.BH = B * Hq;
  qattn::RowsJob jk{};
  if (i8) {
    // every K scale is 1: the Q quantizer's launch writes them
    jq.ones = k_scales;
    jq.n_ones = shape->Nk == 0                        ? 0
                : params->k_gran == QATTN_GRAN_TENSOR ? 1
                : params->k_gran == QATTN_GRAN_HEAD   ? shape->B * shape->Hkv
                                                      : shape->B * shape->Hkv * nkb;
    char sb[128];
    QATTN_LOG_LINE("qattn_quantize_qk %s int8 cache: quant_rows_kernel (Q with K's channel scales)%s",
                   shape_str(shape, sb, sizeof sb), k_carrier ? " + codes_to_f16_kernel" : "");
    cudaError_t e = qattn::launch_quantize_rows(jq, 2, jk, 0, d, s);
    if (e != cudaSuccess) return QATTN_ERR_CUDA;
    if (k_carrier && shape->Nk > 0) {
      e = qattn::launch_codes_to_f16(static_cast<const int8_t*>(K), k_carrier,
                                     static_cast<size_t>(shape->B * shape->Hkv * shape->Nk * d), s);
      if (e != cudaSuccess) return QATTN_ERR_CUDA;
    }
    return QATTN_OK;
  }
  if (shape->Nk > 0) {
    jk.X = static_cast<const uint16_t*>(K);
    jk.sB = ks.sB;
    jk.sH = ks.sH;
    jk.sN = ks.sN;
    jk.H = Hkv;
    jk.N = static_cast<int>(shape->Nk);
    jk.chan = k_mean;
    jk.Hchan = Hkv;
    jk.group = 1;
    jk.gran = params->k_gran;
    jk.codes = k_codes;
    jk.scales = k_scales;
    jk.ws_amax = ws_k;
    jk.carrier = k_carrier;
    jk.nblk = static_cast<int>(nkb);
    jk.BH = B * Hkv;
  }
  char sb[128];
  QATTN_LOG_LINE("qattn_quantize_qk %s granules q=%d k=%d mean=%d strided=%d: quant_rows_kernel, %d pass(es)",
                 shape_str(shape, sb, sizeof sb), params->q_gran, params->k_gran, k_mean != nullptr,
                 q_strides != nullptr || k_strides != nullptr,
                 (params->q_gran != QATTN_GRAN_BLOCK || (shape->Nk > 0 && params->k_gran != QATTN_GRAN_BLOCK)) ? 2 : 1);
  return from_cuda(qattn::launch_quantize_rows(jq, 0, jk, k_mean ? 1 : 0, d, s));
}

qattn_status qattn_prepare(const uint16_t* Q, const int64_t* q_strides, const uint16_t* K,
                           const int64_t* k_strides, const uint16_t* V, const int64_t* v_strides,
                           const qattn_shape* shape, const qattn_params* params,
                           int8_t* q_codes, float* q_scales, int8_t* k_codes, float* k_scales,
                           uint16_t* k_carrier, float* k_mean, uint8_t* v8t, int64_t ldv,
                           float* v_scales, void* workspace, size_t workspace_bytes,
                           qattn_stream_t stream) {
  qattn_status st = check_shape(shape);
  if (st != QATTN_OK) return st;
  if ((st = check_params(params)) != QATTN_OK) return st;
  if (empty_problem(shape)) return QATTN_OK;
  if (qattn_prepare_launches(shape, params) < 1) return QATTN_ERR_UNSUPPORTED;
  const bool tensor = params->q_gran == QATTN_GRAN_TENSOR;
  for (const void* p : {static_cast<const void*>(Q), static_cast<const void*>(K),
                        static_cast<const void*>(V), static_cast<const void*>(q_codes),
                        static_cast<const void*>(q_scales), static_cast<const void*>(k_codes),
                        static_cast<const void*>(k_scales), static_cast<const void*>(k_mean),
                        static_cast<const void*>(v8t), static_cast<const void*>(v_scales)})
    if (!p || !aligned16(p)) return QATTN_ERR_INVALID_ARG;
  if (k_carrier && !aligned16(k_carrier)) return QATTN_ERR_INVALID_ARG;
  if (ldv < qattn_v_ld(shape->Nk) || (ldv % 16) != 0) return QATTN_ERR_INVALID_ARG;
  const size_t need = ws_prepare(shape);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return QATTN_ERR_WORKSPACE;
  qattn::Src qs, ks, vs;
  if (!make_src(Q, q_strides, shape->Hq, shape->Nq, shape->d, 2, &qs) ||
      !make_src(K, k_strides, shape->Hkv, shape->Nk, shape->d, 2, &ks) ||
      !make_src(V, v_strides, shape->Hkv, shape->Nk, shape->d, 2, &vs))
    return QATTN_ERR_INVALID_ARG;
  const int B = static_cast<int>(shape->B), Hq = static_cast<int>(shape->Hq);
  const int Hkv = static_cast<int>(shape->Hkv), d = static_cast<int>(shape->d);
  qattn::RowsJob jq{};
  jq.X = Q;
  jq.sB = qs.sB;
  jq.sH = qs.sH;
  jq.sN = qs.sN;
  jq.H = Hq;
  jq.N = static_cast<int>(shape->Nq);
  jq.Hchan = 1;
  jq.group = 1;
  jq.gran = params->q_gran;
  jq.codes = q_codes;
  jq.scales = q_scales;
  jq.nblk = static_cast<int>((shape->Nq + 127) / 128);
  jq.BH = B * Hq;
  qattn::RowsJob jk{};
  jk.X = K;
  jk.sB = ks.sB;
  jk.sH = ks.sH;
  jk.sN = ks.sN;
  jk.H = Hkv;
  jk.N = static_cast<int>(shape->Nk);
  jk.chan = k_mean;
  jk.Hchan = Hkv;
  jk.group = 1;
  jk.gran = params->k_gran;
  jk.codes = k_codes;
  jk.scales = k_scales;
  jk.carrier = k_carrier;
  jk.nblk = static_cast<int>((shape->Nk + 127) / 128);
  jk.BH = B * Hkv;
  char sb[128];
  QATTN_LOG_LINE("qattn_prepare %s: %s", shape_str(shape, sb, sizeof sb),
                 tensor ? "prepare_tensor1_kernel + prepare_tensor2_kernel (tensor granules, two launches)"
                 : qattn::prepare_launch_count(d, jq.N, jk.N) == 1
                     ? "prepare_small_kernel (one warp per head, one launch)"
                     : "prepare1_kernel + prepare2_kernel (two launches)");
  if (tensor)
    return from_cuda(qattn::launch_prepare_tensor(jq, jk, vs, d, v8t, ldv, v_scales, workspace,
                                                  reinterpret_cast<cudaStream_t>(stream)));
  return from_cuda(qattn::launch_prepare(jq, jk, vs, d, v8t, ldv, v_scales, workspace,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

qattn_status qattn_quantize_v(const void* V, const int64_t* v_strides, qattn_dtype v_dtype,
                              const float* v_chan_scale,
                              const qattn_shape* shape, uint8_t* v8t, int64_t ldv,
                              float* v_scales, void* workspace, size_t workspace_bytes,
                              qattn_stream_t stream) {
  qattn_status st = check_shape(shape);
  if (st != QATTN_OK) return st;
  if (v_dtype != QATTN_BF16 && v_dtype != QATTN_I8) return QATTN_ERR_INVALID_ARG;
  if (shape->B == 0 || shape->Hkv == 0) return QATTN_OK;
  const bool i8 = (v_dtype == QATTN_I8);
  if (!v_scales || !aligned16(v_scales)) return QATTN_ERR_INVALID_ARG;
  if (shape->Nk > 0 && (!V || !aligned16(V) || !v8t || !aligned16(v8t))) return QATTN_ERR_INVALID_ARG;
  if (i8 && (!v_chan_scale || !aligned16(v_chan_scale))) return QATTN_ERR_INVALID_ARG;
  if (ldv < qattn_v_ld(shape->Nk) || (ldv % 16) != 0) return QATTN_ERR_INVALID_ARG;
  const size_t need = ws_quant_v(shape);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return QATTN_ERR_WORKSPACE;
  qattn::Src vs;
  if (!make_src(V, v_strides, shape->Hkv, shape->Nk, shape->d, i8 ? 1 : 2, &vs)) return QATTN_ERR_INVALID_ARG;
  char sb[128];
  QATTN_LOG_LINE("qattn_quantize_v %s %s strided=%d: v_amax_kernel + v_convert_kernel",
                 shape_str(shape, sb, sizeof sb), i8 ? "int8 codes" : "bf16", v_strides != nullptr);
  return from_cuda(qattn::launch_quantize_v(vs, i8 ? 1 : 0, v_chan_scale,
                                            static_cast<int>(shape->B * shape->Hkv),
                                            static_cast<int>(shape->Nk), static_cast<int>(shape->d),
                                            v8t, ldv, v_scales, static_cast<unsigned int*>(workspace),
                                            reinterpret_cast<cudaStream_t>(stream)));
}

qattn_status qattn_fwd(const int8_t* q_codes, const float* q_scales, const int8_t* k_codes,
                       const uint16_t* k_carrier, const float* k_scales, const uint8_t* v8t,
                       int64_t ldv,
                       const float* v_scales, const float* bias, const qattn_shape* shape,
                       const qattn_params* params, void* O, float* lse, void* workspace,
                       size_t workspace_bytes, qattn_stream_t stream) {
  qattn_status st = check_shape(shape);
  if (st != QATTN_OK) return st;
  if ((st = check_params(params)) != QATTN_OK) return st;
  if (empty_problem(shape)) return QATTN_OK;
  if (!q_codes || !aligned16(q_codes) || !q_scales || !O || !aligned16(O)) return QATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return QATTN_ERR_INVALID_ARG;
  if (params->pv_mode == QATTN_PV_INT8 && bias) return QATTN_ERR_UNSUPPORTED;  // ablation: no bias
  const int64_t pos0 = pos0_of(shape, params);
  if (params->causal && (pos0 <= -(int64_t{1} << 30) || pos0 >= (int64_t{1} << 30))) return QATTN_ERR_UNSUPPORTED;
  if (shape->Nk > 0) {
    if (!k_codes || !aligned16(k_codes) || !k_scales || !v8t || !aligned16(v8t) || !v_scales ||
        !aligned16(v_scales))
      return QATTN_ERR_INVALID_ARG;
    if (k_carrier && !aligned16(k_carrier)) return QATTN_ERR_INVALID_ARG;
    if (ldv < qattn_v_ld(shape->Nk) || (ldv % 16) != 0) return QATTN_ERR_INVALID_ARG;
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) return QATTN_ERR_INVALID_ARG;
  }
  const int choice = fwd_choice(shape, params);
  if (choice < 0) return QATTN_ERR_UNSUPPORTED;
  const bool use_short = choice == QATTN_FWD_SHORT;
  if (!use_short && !k_carrier && shape->Nk > 0) {  // the K codes are converted into the workspace
    const size_t need = ws_fwd(shape);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return QATTN_ERR_WORKSPACE;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (shape->Nk == 0) return no_key_rows(shape, params, O, lse, s);
  unsigned int* err = error_word();
  if (!err) return QATTN_ERR_CUDA;
  AttnArgs a{};
  a.B = static_cast<int>(shape->B);
  a.Hq = static_cast<int>(shape->Hq);
  a.Hkv = static_cast<int>(shape->Hkv);
  a.Nq = static_cast<int>(shape->Nq);
  a.Nk = static_cast<int>(shape->Nk);
  a.d = static_cast<int>(shape->d);
  a.causal = params->causal;
  a.pos0 = params->causal ? static_cast<int>(pos0) : 0;
  a.sm_scale = params->sm_scale > 0.f ? params->sm_scale
                                      : static_cast<float>(1.0 / std::sqrt(static_cast<double>(shape->d)));
  a.q_gran = params->q_gran;
  a.k_gran = params->k_gran;
  a.q_scales = q_scales;
  a.k_scales = k_scales;
  a.v_scales = v_scales;
  a.bias = bias;
  a.bias_head_stride = params->bias_head_stride;
  a.pv_int8 = params->pv_mode == QATTN_PV_INT8 ? 1 : 0;
  a.out = O;
  a.out_bf16 = params->out_dtype == QATTN_BF16;
  a.lse = lse;
  a.err = err;
  char sb[128];
  QATTN_LOG_LINE("qattn_fwd %s causal=%d pos0=%lld bias=%d pv=%s out=%s: %s%s", shape_str(shape, sb, sizeof sb),
                 params->causal, static_cast<long long>(pos0), bias != nullptr,
                 a.pv_int8 ? "int8" : "e4m3", a.out_bf16 ? "bf16" : "fp32",
                 use_short ? (qattn::attn_short_eligible(a) && shape->Nq <= qattn::kWindowMax &&
                                      shape->Nk <= qattn::kWindowMax
                                  ? "warp-level kernel (attn_window_kernel or attn_short_kernel)"
                                  : "warp-level kernel (attn_short_kernel)")
                           : "persistent tcgen05 kernel (attn_fwd_kernel), one CTA per SM",
                 use_short || k_carrier ? "" : " after codes_to_f16_kernel (K carriers in the workspace)");
  if (use_short) return from_cuda(qattn::launch_attn_short(a, q_codes, k_codes, v8t, ldv, s));
  const uint16_t* kc16 = k_carrier;
  if (!kc16) {  // convert the K codes into the workspace (checked above)
    uint16_t* w16 = static_cast<uint16_t*>(workspace);
    const cudaError_t e = qattn::launch_codes_to_f16(
        k_codes, w16, static_cast<size_t>(shape->B * shape->Hkv * shape->Nk * shape->d), s);
    if (e != cudaSuccess) return QATTN_ERR_CUDA;
    kc16 = w16;
  }
  CUtensorMap tq, tk, tv, to;
  std::memset(&to, 0, sizeof to);
  if (!encode_q_codes(&tq, q_codes, shape->B * shape->Hq, shape->Nq, shape->d) ||
      !encode_carrier(&tk, kc16, shape->B * shape->Hkv, shape->Nk, shape->d) ||
      !encode_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, v8t, static_cast<uint64_t>(shape->Nk),
                 static_cast<uint64_t>(shape->d), static_cast<uint64_t>(shape->B * shape->Hkv),
                 static_cast<uint64_t>(ldv), 128, static_cast<uint32_t>(shape->d),
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return QATTN_ERR_CUDA;
  if (!a.out_bf16 || shape->d >= 64) {  // the output map: boxes of 128-byte rows x 32 rows
    const size_t es = a.out_bf16 ? 2 : 4;
    if (!encode_3d(&to, a.out_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                   es, O, static_cast<uint64_t>(shape->d), static_cast<uint64_t>(shape->Nq),
                   static_cast<uint64_t>(shape->B * shape->Hq), static_cast<uint64_t>(shape->d) * es,
                   static_cast<uint32_t>(128 / es), 32, CU_TENSOR_MAP_SWIZZLE_128B))
      return QATTN_ERR_CUDA;
  }
  return from_cuda(qattn::launch_attn_fwd(tq, tk, tv, to, a, s));
}

qattn_status qattn_decode(const int8_t* q_codes, const float* q_scales, const int8_t* k_codes,
                          const float* k_scales, const int8_t* v_codes,
                          const float* v_chan_scale, const float* v_code_amax,
                          const qattn_shape* shape, const qattn_params* params, void* O,
                          float* lse, void* workspace, size_t workspace_bytes,
                          qattn_stream_t stream) {
  qattn_status st = check_shape(shape);
  if (st != QATTN_OK) return st;
  if ((st = check_params(params)) != QATTN_OK) return st;
  if (empty_problem(shape)) return QATTN_OK;
  if (!decode_shape_ok(shape) || shape->Nk == 0 || params->pv_mode != QATTN_PV_E4M3)
    return QATTN_ERR_UNSUPPORTED;
  if (params->kv_capacity != 0 &&
      (params->kv_capacity < shape->Nk || params->kv_capacity > (int64_t{1} << 31)))
    return QATTN_ERR_INVALID_ARG;
  if (!q_codes || !aligned16(q_codes) || !q_scales || !k_codes || !aligned16(k_codes) ||
      !k_scales || !v_codes || !aligned16(v_codes) || !v_chan_scale || !v_code_amax || !O ||
      !aligned16(O))
    return QATTN_ERR_INVALID_ARG;
  for (const void* f : {static_cast<const void*>(q_scales), static_cast<const void*>(k_scales),
                        static_cast<const void*>(v_chan_scale),
                        static_cast<const void*>(v_code_amax), static_cast<const void*>(lse)})
    if (reinterpret_cast<uintptr_t>(f) & 3u) return QATTN_ERR_INVALID_ARG;
  const int64_t pos0 = pos0_of(shape, params);
  if (params->causal && (pos0 <= -(int64_t{1} << 30) || pos0 >= (int64_t{1} << 30))) return QATTN_ERR_UNSUPPORTED;
  const size_t need = qattn::decode_ws_bytes(shape->B, shape->Hq, shape->Hkv, shape->Nq,
                                             shape->Nk, shape->d);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return QATTN_ERR_WORKSPACE;
  unsigned int* err = error_word();
  if (!err) return QATTN_ERR_CUDA;
  qattn::DecodeArgs a{};
  a.err = err;
  a.epoch = next_decode_tag();
  a.B = static_cast<int>(shape->B);
  a.Hq = static_cast<int>(shape->Hq);
  a.Hkv = static_cast<int>(shape->Hkv);
  a.Nq = static_cast<int>(shape->Nq);
  a.Nk = static_cast<int>(shape->Nk);
  a.d = static_cast<int>(shape->d);
  a.causal = params->causal;
  a.pos0 = params->causal ? static_cast<int>(pos0) : 0;
  a.sm_scale = params->sm_scale > 0.f ? params->sm_scale
                                      : static_cast<float>(1.0 / std::sqrt(static_cast<double>(shape->d)));
  a.q_gran = params->q_gran;
  a.k_gran = params->k_gran;
  a.q_codes = q_codes;
  a.q_scales = q_scales;
  a.k_codes = k_codes;
  a.k_scales = k_scales;
  a.v_codes = v_codes;
  a.v_chan_scale = v_chan_scale;
  a.v_code_amax = v_code_amax;
  a.out = O;
  a.out_bf16 = params->out_dtype == QATTN_BF16;
  a.lse = lse;
  // the cache's K and V codes, tiles of 128 keys swizzled for conflict-free reads
  CUtensorMap tk, tv;
  const CUtensorMapSwizzle swz = shape->d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const uint64_t planes = static_cast<uint64_t>(shape->B * shape->Hkv);
  const uint64_t cap = static_cast<uint64_t>(params->kv_capacity ? params->kv_capacity : shape->Nk);
  if (!encode_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, k_codes, shape->d, shape->Nk, planes,
                 shape->d, static_cast<uint32_t>(shape->d), 128, swz, cap) ||
      !encode_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, v_codes, shape->d, shape->Nk, planes,
                 shape->d, static_cast<uint32_t>(shape->d), 128, swz, cap))
    return QATTN_ERR_CUDA;
  char sb[128];
  QATTN_LOG_LINE("qattn_decode %s capacity=%lld: decode kernel over key chunks + chunk combine",
                 shape_str(shape, sb, sizeof sb), static_cast<long long>(cap));
  return from_cuda(qattn::launch_decode(tk, tv, a, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

qattn_status qattn_debug_qk_scores(const int8_t* q_codes, const int8_t* k_codes,
                                   const qattn_shape* shape, int32_t* S, void* workspace,
                                   size_t workspace_bytes, qattn_stream_t stream) {
  qattn_status st = check_shape(shape);
  if (st != QATTN_OK) return st;
  if (empty_problem(shape) || shape->Nk == 0) return QATTN_OK;
  if (!q_codes || !aligned16(q_codes) || !k_codes || !aligned16(k_codes) || !S || (reinterpret_cast<uintptr_t>(S) & 3u))
    return QATTN_ERR_INVALID_ARG;
  const size_t need = ws_fwd(shape);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return QATTN_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int* err = error_word();
  if (!err) return QATTN_ERR_CUDA;
  uint16_t* kc16 = static_cast<uint16_t*>(workspace);
  const cudaError_t e = qattn::launch_codes_to_f16(
      k_codes, kc16, static_cast<size_t>(shape->B * shape->Hkv * shape->Nk * shape->d), s);
  if (e != cudaSuccess) return QATTN_ERR_CUDA;
  CUtensorMap tq, tk;
  if (!encode_q_codes(&tq, q_codes, shape->B * shape->Hq, shape->Nq, shape->d) ||
      !encode_carrier(&tk, kc16, shape->B * shape->Hkv, shape->Nk, shape->d))
    return QATTN_ERR_CUDA;
  return from_cuda(qattn::launch_qk_debug(tq, tk, static_cast<int>(shape->B), static_cast<int>(shape->Hq),
                                          static_cast<int>(shape->Hkv), static_cast<int>(shape->Nq),
                                          static_cast<int>(shape->Nk), static_cast<int>(shape->d), S, err, s));
}

qattn_status qattn_fwd_exact24(const void* Q, const int8_t* k_codes, const float* k_chan_scale,
                              const int8_t* v_codes, const float* v_chan_scale,
                              const qattn_shape* shape, const qattn_params* params, void* O,
                              float* lse, void* workspace, size_t workspace_bytes,
                              qattn_stream_t stream) {
  qattn_status st = check_shape(shape);
  if (st != QATTN_OK) return st;
  if ((st = check_params(params)) != QATTN_OK) return st;
  if (empty_problem(shape)) return QATTN_OK;
  if (shape->d != 64 && shape->d != 128) return QATTN_ERR_UNSUPPORTED;
  if (shape->B * shape->Hq > 65535) return QATTN_ERR_UNSUPPORTED;
  if (!Q || !aligned16(Q) || !O || !aligned16(O) || !k_chan_scale || !v_chan_scale)
    return QATTN_ERR_INVALID_ARG;
  if (shape->Nk > 0 && (!k_codes || !aligned16(k_codes) || !v_codes || !aligned16(v_codes)))
    return QATTN_ERR_INVALID_ARG;
  for (const void* f : {static_cast<const void*>(k_chan_scale), static_cast<const void*>(v_chan_scale),
                        static_cast<const void*>(lse)})
    if (reinterpret_cast<uintptr_t>(f) & 3u) return QATTN_ERR_INVALID_ARG;
  if (params->kv_capacity != 0 &&
      (params->kv_capacity < shape->Nk || params->kv_capacity > (int64_t{1} << 31)))
    return QATTN_ERR_INVALID_ARG;
  const int64_t pos0 = pos0_of(shape, params);
  if (params->causal && (pos0 <= -(int64_t{1} << 30) || pos0 >= (int64_t{1} << 30))) return QATTN_ERR_UNSUPPORTED;
  if (shape->Nk == 0) return no_key_rows(shape, params, O, lse, reinterpret_cast<cudaStream_t>(stream));
  const size_t need = qattn::exact24_ws_bytes(shape->B, shape->Hq, shape->Hkv, shape->Nq, shape->Nk,
                                              shape->d);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return QATTN_ERR_WORKSPACE;
  qattn::Exact24Args a{};
  a.B = static_cast<int>(shape->B);
  a.Hq = static_cast<int>(shape->Hq);
  a.Hkv = static_cast<int>(shape->Hkv);
  a.Nq = static_cast<int>(shape->Nq);
  a.Nk = static_cast<int>(shape->Nk);
  a.d = static_cast<int>(shape->d);
  a.causal = params->causal;
  a.pos0 = params->causal ? static_cast<int>(pos0) : 0;
  a.sm_scale = params->sm_scale > 0.f ? params->sm_scale
                                      : static_cast<float>(1.0 / std::sqrt(static_cast<double>(shape->d)));
  a.cap = params->kv_capacity ? params->kv_capacity : shape->Nk;
  a.Q = Q;
  a.k_chan_scale = k_chan_scale;
  a.k_codes = k_codes;
  a.v_codes = v_codes;
  a.v_chan_scale = v_chan_scale;
  a.out = O;
  a.out_bf16 = params->out_dtype == QATTN_BF16;
  a.lse = lse;
  a.ws = workspace;
  char sb[128];
  a.err = error_word();
  if (!a.err) return QATTN_ERR_CUDA;
  QATTN_LOG_LINE("qattn_fwd_exact24 %s: q_split_kernel + k_rows_f16_kernel + v_t_f16_kernel + exact24_tc_kernel",
                 shape_str(shape, sb, sizeof sb));
  return from_cuda(qattn::launch_exact24(a, reinterpret_cast<cudaStream_t>(stream)));
}

qattn_status qattn_fwd_intsoftmax(const int8_t* q_codes, const float* q_scale,
                                 const int8_t* k_codes, const float* k_scale,
                                 const int8_t* v_codes, const qattn_shape* shape,
                                 const qattn_params* params, int8_t* O_codes,
                                 qattn_stream_t stream) {
  qattn_status st = check_shape(shape);
  if (st != QATTN_OK) return st;
  if ((st = check_params(params)) != QATTN_OK) return st;
  if (empty_problem(shape)) return QATTN_OK;
  if (shape->d != 32 && shape->d != 64 && shape->d != 128) return QATTN_ERR_UNSUPPORTED;
  // Nk <= 2^17 keeps |O| <= 127 * 128 * Nk inside int32
  if (params->causal || shape->Nk == 0 || shape->Nk > (int64_t{1} << 17) || shape->B * shape->Hq > 65535)
    return QATTN_ERR_UNSUPPORTED;
  if (!q_codes || !aligned16(q_codes) || !k_codes || !aligned16(k_codes) || !v_codes ||
      !aligned16(v_codes) || !O_codes || !aligned16(O_codes) || !q_scale || !k_scale)
    return QATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_scale) & 3u) || (reinterpret_cast<uintptr_t>(k_scale) & 3u))
    return QATTN_ERR_INVALID_ARG;
  const float sm = params->sm_scale > 0.f ? params->sm_scale
                                          : static_cast<float>(1.0 / std::sqrt(static_cast<double>(shape->d)));
  unsigned int* err = error_word();
  if (!err) return QATTN_ERR_CUDA;
  char sb[128];
  QATTN_LOG_LINE("qattn_fwd_intsoftmax %s: intsm_attn_kernel", shape_str(shape, sb, sizeof sb));
  return from_cuda(qattn::launch_intsoftmax(
      static_cast<int>(shape->B), static_cast<int>(shape->Hq), static_cast<int>(shape->Hkv),
      static_cast<int>(shape->Nq), static_cast<int>(shape->Nk), static_cast<int>(shape->d), sm, q_codes,
      q_scale, k_codes, k_scale, v_codes, O_codes, err, reinterpret_cast<cudaStream_t>(stream)));
}

qattn_status qattn_kv_append(const void* K_new, const void* V_new, int64_t B, int64_t Hkv,
                             int64_t T, int64_t d, int64_t pos, int64_t capacity,
                             const float* k_chan_scale, const float* v_chan_scale,
                             float* k_mean, float* v_code_amax, int8_t* k_codes,
                             int8_t* v_codes, qattn_stream_t stream) {
  if (B <= 0 || Hkv <= 0 || T < 0 || d < 1 || d > 1024 || pos < 0 || capacity < 0 ||
      pos + T > capacity || capacity > (int64_t{1} << 24) || B * Hkv * d >= (int64_t{1} << 31))
    return QATTN_ERR_INVALID_ARG;
  if (!K_new || !V_new || !k_chan_scale || !v_chan_scale || !k_mean || !v_code_amax ||
      !k_codes || !v_codes)
    return QATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(K_new) & 1u) || (reinterpret_cast<uintptr_t>(V_new) & 1u))
    return QATTN_ERR_INVALID_ARG;
  for (const void* f : {static_cast<const void*>(k_chan_scale), static_cast<const void*>(v_chan_scale),
                        static_cast<const void*>(k_mean), static_cast<const void*>(v_code_amax)})
    if (reinterpret_cast<uintptr_t>(f) & 3u) return QATTN_ERR_INVALID_ARG;
  if (T == 0) return QATTN_OK;
  QATTN_LOG_LINE("qattn_kv_append B=%lld Hkv=%lld T=%lld d=%lld pos=%lld capacity=%lld: kv_append_kernel",
                 static_cast<long long>(B), static_cast<long long>(Hkv), static_cast<long long>(T),
                 static_cast<long long>(d), static_cast<long long>(pos), static_cast<long long>(capacity));
  return from_cuda(qattn::launch_kv_append(
      static_cast<const uint16_t*>(K_new), static_cast<const uint16_t*>(V_new),
      static_cast<int>(B * Hkv), static_cast<int>(d), static_cast<int>(T), static_cast<int>(pos),
      static_cast<long long>(capacity), k_chan_scale, v_chan_scale, k_mean, v_code_amax, k_codes,
      v_codes, reinterpret_cast<cudaStream_t>(stream)));
}

qattn_status qattn_kv_header_init(const int8_t* v_codes, int64_t B, int64_t Hkv, int64_t Nk,
                                  int64_t d, int64_t capacity, float* v_code_amax,
                                  qattn_stream_t stream) {
  if (B <= 0 || Hkv <= 0 || Nk < 0 || capacity < Nk || capacity > (int64_t{1} << 24) ||
      B * Hkv > 65535 || !valid_d(d))
    return QATTN_ERR_INVALID_ARG;
  if (!v_code_amax || (reinterpret_cast<uintptr_t>(v_code_amax) & 3u)) return QATTN_ERR_INVALID_ARG;
  if (Nk > 0 && (!v_codes || !aligned16(v_codes))) return QATTN_ERR_INVALID_ARG;
  return from_cuda(qattn::launch_v_code_amax(v_codes, static_cast<int>(B * Hkv), static_cast<int>(Nk),
                                             static_cast<long long>(capacity), static_cast<int>(d),
                                             v_code_amax, reinterpret_cast<cudaStream_t>(stream)));
}

int qattn_fwd_kernel_choice(const qattn_shape* shape, const qattn_params* params) {
  if (check_shape(shape) != QATTN_OK || check_params(params) != QATTN_OK) return -1;
  const int c = fwd_choice(shape, params);
  char sb[128];
  QATTN_LOG_LINE("qattn_fwd_kernel_choice %s causal=%d: %s", shape_str(shape, sb, sizeof sb),
                 params->causal, c == QATTN_FWD_SHORT ? "warp-level" : c < 0 ? "rejected" : "persistent tcgen05");
  return c;
}

int qattn_checked(void) { return qattn::kChecked ? 1 : 0; }

qattn_status qattn_debug_bounds_probe(qattn_stream_t stream) {
  return from_cuda(qattn::launch_bounds_probe(reinterpret_cast<cudaStream_t>(stream)));
}

int qattn_prepare_launches(const qattn_shape* shape, const qattn_params* params) {
  if (check_shape(shape) != QATTN_OK || check_params(params) != QATTN_OK) return -1;
  if (shape->Nk < 1) return -1;
  const int d = static_cast<int>(shape->d), Nq = static_cast<int>(shape->Nq),
            Nk = static_cast<int>(shape->Nk);
  if (params->q_gran == QATTN_GRAN_TENSOR && params->k_gran == QATTN_GRAN_TENSOR) {
    if (!qattn::prepare_tensor_eligible(d, Nq, Nk)) return -1;
    return empty_problem(shape) ? 0 : 2;
  }
  if (params->q_gran != QATTN_GRAN_BLOCK || params->k_gran != QATTN_GRAN_BLOCK) return -1;
  if (empty_problem(shape)) return 0;
  return qattn::prepare_launch_count(d, Nq, Nk);
}

qattn_status qattn_debug_wait_timeout(int32_t* result, qattn_stream_t stream) {
  if (!result || (reinterpret_cast<uintptr_t>(result) & 7u)) return QATTN_ERR_INVALID_ARG;
  unsigned int* err = error_word();
  if (!err) return QATTN_ERR_CUDA;
  wait_timeout_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err, result);
  return from_cuda(cudaGetLastError());
}

qattn_status qattn_get_error(qattn_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return QATTN_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qattn_error_word, sizeof(v)) != cudaSuccess) return QATTN_ERR_CUDA;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_qattn_error_word, &zero, sizeof(zero)) != cudaSuccess) return QATTN_ERR_CUDA;
  }
  const unsigned int checks = qattn::check_take_attn_fwd() | qattn::check_take_quant() |
                              qattn::check_take_decode() | qattn::check_take_short() |
                              qattn::check_take_exact24() | qattn::check_take_intsm();
  if (v & qattn::kErrTimeout) return QATTN_ERR_TIMEOUT;
  if (checks != 0) return QATTN_ERR_BOUNDS;
  return (v & qattn::kErrDomain) ? QATTN_ERR_INVALID_ARG : QATTN_OK;
}

}  // extern "C"
