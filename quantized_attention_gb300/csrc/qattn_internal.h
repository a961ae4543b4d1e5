// Internal launch interface between the C ABI (qattn_api.cu) and the
// kernels (quant_kernels.cu, attn_fwd.cu).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qattn {

// Bits of the device error word.
constexpr unsigned int kErrTimeout = 1u;

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
  void* out;
  int out_bf16;
  float* lse;
  unsigned int* err;
};

// ---- quant_kernels.cu
cudaError_t launch_smooth_k(const uint16_t* K, int BH, int Nk, int d, long long* ws, float* mu,
                            cudaStream_t s);
size_t smooth_k_ws_bytes(long long BH, long long Nk, long long d);

cudaError_t launch_quantize_rows(const uint16_t* X, int B, int H, int N, int d, int mode,
                                 const float* chan, int Hchan, int gran, int8_t* codes,
                                 float* scales, float* ws_amax, cudaStream_t s);
size_t quantize_rows_ws_bytes(long long B, long long H, long long N, int gran);
cudaError_t launch_fill_ones(float* p, long long n, cudaStream_t s);

cudaError_t launch_quantize_v(const void* V, int is_i8, const float* chan, int BH, int Nk, int d,
                              uint8_t* v8t, long long ldv, float* v_scales, unsigned int* ws_amax,
                              cudaStream_t s);

cudaError_t launch_codes_to_f16(const int8_t* src, uint16_t* dst, size_t n, cudaStream_t s);

// ---- attn_fwd.cu
cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const AttnArgs& a, cudaStream_t s);
cudaError_t launch_qk_debug(const CUtensorMap& tq, const CUtensorMap& tk, int B, int Hq, int Hkv,
                            int Nq, int Nk, int d, int32_t* S, unsigned int* err,
                            cudaStream_t s);

}  // namespace qattn
