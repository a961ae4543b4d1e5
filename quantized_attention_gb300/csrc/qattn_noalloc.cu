// qattn_quantize_v_noalloc: qattn_quantize_v without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they quantize
// V: an inference-engine plugin that is handed only the tensors it must fill,
// a serving loop where cudaMalloc (which can synchronise the device) is banned
// on the hot path, or code that runs under an allocator it does not own.  For
// them this entry point keeps its scratch -- the per-channel amax of V -- in a
// file-scope device array owned by the library, so the call needs nothing but
// its inputs and outputs.
#include <mutex>

#include <cuda_runtime.h>

#include "qattn.h"
#include "qattn_internal.h"

namespace {

// Largest B * Hkv * d this entry point accepts (2 MiB of device memory, held by
// every GPU that loads the library until the process exits).
constexpr long long kNoAllocMaxChannels = 1ll << 19;

// One 32-bit amax slot per (batch, KV head, channel).  In host code this
// name is only a stand-in: its device address comes from
// cudaGetSymbolAddress, once per device and CUDA context.
static __device__ __align__(256) unsigned int g_v_amax_scratch[kNoAllocMaxChannels];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};  // 0: unknown, resolve every call

// Device address of the scratch array on the current device, resolved with
// that device current on the first call in each context (so after a
// cudaDeviceReset the new context gets its own address); nullptr on failure.
unsigned int* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned long long ctx = 0;
  const bool known = qattn::current_context_id(&ctx);
  std::lock_guard<std::mutex> lk(g_mu);
  if (known && g_scratch_ptr[dev] && g_scratch_ctx[dev] == ctx) return g_scratch_ptr[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_v_amax_scratch) != cudaSuccess || p == nullptr) return nullptr;
  // the symbol lookup makes the device's primary context current if none was
  const bool now_known = known || qattn::current_context_id(&ctx);
  g_scratch_ptr[dev] = static_cast<unsigned int*>(p);
  g_scratch_ctx[dev] = now_known ? ctx : 0;
  return g_scratch_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" qattn_status qattn_quantize_v_noalloc(const void* V, qattn_dtype v_dtype,
                                                 const float* v_chan_scale,
                                                 const qattn_shape* shape, uint8_t* v8t,
                                                 int64_t ldv, float* v_scales,
                                                 qattn_stream_t stream) {
  if (!shape) return QATTN_ERR_INVALID_ARG;
  if (shape->B < 0 || shape->Hkv <= 0 || shape->Nk < 0 || shape->Hq < 0 ||
      (shape->Hq % shape->Hkv) != 0)
    return QATTN_ERR_INVALID_ARG;
  if (shape->d != 32 && shape->d != 64 && shape->d != 128) return QATTN_ERR_UNSUPPORTED;
  if (shape->Nk > 65535ll * 128 || shape->B * shape->Hq > 65535 || shape->B > 65535)
    return QATTN_ERR_UNSUPPORTED;
  if (v_dtype != QATTN_BF16 && v_dtype != QATTN_I8) return QATTN_ERR_INVALID_ARG;
  if (shape->B == 0) return QATTN_OK;
  const long long channels = shape->B * shape->Hkv * shape->d;
  if (channels > kNoAllocMaxChannels) return QATTN_ERR_UNSUPPORTED;  // beyond the static scratch
  const bool i8 = (v_dtype == QATTN_I8);
  if (!v_scales || !aligned16(v_scales)) return QATTN_ERR_INVALID_ARG;
  if (shape->Nk > 0 && (!V || !aligned16(V) || !v8t || !aligned16(v8t))) return QATTN_ERR_INVALID_ARG;
  if (i8 && (!v_chan_scale || !aligned16(v_chan_scale))) return QATTN_ERR_INVALID_ARG;
  if (ldv < qattn_v_ld(shape->Nk) || (ldv % 16) != 0) return QATTN_ERR_INVALID_ARG;
  unsigned int* scratch = scratch_for_current_device();
  if (!scratch) return QATTN_ERR_CUDA;
  // launch_quantize_v zeroes the first B*Hkv*d slots before using them.
  const cudaError_t e = qattn::launch_quantize_v(
      qattn::dense_src(V, static_cast<int>(shape->Hkv), shape->Nk, static_cast<int>(shape->d)),
      i8 ? 1 : 0, v_chan_scale, static_cast<int>(shape->B * shape->Hkv),
      static_cast<int>(shape->Nk), static_cast<int>(shape->d), v8t, ldv, v_scales, scratch,
      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QATTN_OK : QATTN_ERR_CUDA;
}
