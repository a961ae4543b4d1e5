// HBM-bound pre-passes of the recipe: the K channel mean (a1), the symmetric
// int8 quantizer for Q and K (a2), the per-channel e4m3 quantizer for V with
// its transposed write (a3), and the int8 -> fp16 carrier conversion that
// feeds the f16 tensor-core path.
//
// Bit-exactness with the CPU oracle rests on: an integer (order-free) sum for
// the mean, IEEE divides/multiplies written as __fdiv_rn/__fmul_rn (no FMA
// contraction, no approximate reciprocal), round-half-even conversions
// (__float2ll_rn, __float2int_rn) and the hardware RN/satfinite e4m3 convert.
#include <cuda_fp16.h>

#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kThreads = 256;
constexpr int kTokPerChunk = 256;  // tokens per CTA in the reduction passes

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void unpack_i8x16(const uint4& v, float (&f)[16]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[4 * i + e] = static_cast<float>(static_cast<int8_t>((w[i] >> (8 * e)) & 0xFFu));
    }
  }
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) r = fmaxf(r, red[i]);
  return r;
}

// ------------------------------------------------------------------ a1
// Partial channel sums of round(K * 2^24) over one chunk of tokens.
__global__ void __launch_bounds__(kThreads) k_mean_partial_kernel(
    const uint16_t* __restrict__ K, int Nk, int d, int nchunks, long long* __restrict__ part) {
  extern __shared__ long long red64[];  // [rows per iteration][d]
  const int bh = blockIdx.y, chunk = blockIdx.x;
  const int vpr = d / 8;
  const int rpi = kThreads / vpr;
  const int v = threadIdx.x % vpr, r0 = threadIdx.x / vpr;
  long long acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const uint16_t* base = K + static_cast<size_t>(bh) * Nk * d;
  const int t_end = min(Nk, (chunk + 1) * kTokPerChunk);
  for (int t = chunk * kTokPerChunk + r0; t < t_end; t += rpi) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(base + static_cast<size_t>(t) * d) + v);
    float f[8];
    unpack_bf16x8(raw, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __float2ll_rn(__fmul_rn(f[e], 16777216.0f));
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red64[r0 * d + v * 8 + e] = acc[e];
  __syncthreads();
  for (int c = threadIdx.x; c < d; c += kThreads) {
    long long s = 0;
    for (int r = 0; r < rpi; ++r) s += red64[r * d + c];
    part[(static_cast<size_t>(bh) * nchunks + chunk) * d + c] = s;
  }
}

__global__ void k_mean_finish_kernel(const long long* __restrict__ part, int nchunks, int d,
                                     int Nk, float* __restrict__ mu) {
  const int bh = blockIdx.x;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    long long s = 0;
    for (int k = 0; k < nchunks; ++k) s += part[(static_cast<size_t>(bh) * nchunks + k) * d + c];
    double m = 0.0;
    if (Nk > 0) m = (__ll2double_rn(s) * 0x1p-24) / static_cast<double>(Nk);
    mu[static_cast<size_t>(bh) * d + c] = __double2float_rn(m);
  }
}

// ------------------------------------------------------------------ a2
// One CTA per (batch*head, 128-token block).  MODE 0: x = X; 1: x = X - chan
// (K minus its channel mean); 2: x = X * chan (Q times K's channel scale).
// pass 0 writes the block's amax (tensor/head granules); pass 1 quantizes.
template <int D, int MODE>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(
    const uint16_t* __restrict__ X, int H, int N, const float* __restrict__ chan, int Hchan,
    int group, int gran, int pass, int8_t* __restrict__ codes, float* __restrict__ scales,
    float* __restrict__ ws_amax, int nblk, int BH) {
  constexpr int VPR = D / 8;
  constexpr int NV = 128 * VPR / kThreads;
  __shared__ float red[kThreads / 32];
  const int bh = blockIdx.y, blk = blockIdx.x;
  const int b = bh / H, h = bh % H;
  const int t0 = blk * 128;
  const int rows = min(128, N - t0);
  const uint16_t* src = X + (static_cast<size_t>(bh) * N + t0) * D;
  const float* crow = nullptr;
  if (MODE != 0) crow = chan + (static_cast<size_t>(b) * Hchan + h / group) * D;

  float x[NV][8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = threadIdx.x + i * kThreads;
    const int r = v / VPR, cv = v % VPR;
    if (r < rows) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * D) + cv);
      float f[8];
      unpack_bf16x8(raw, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float y = f[e];
        if (MODE == 1) y = __fsub_rn(y, __ldg(crow + cv * 8 + e));
        if (MODE == 2) y = __fmul_rn(y, __ldg(crow + cv * 8 + e));
        x[i][e] = y;
        amax = fmaxf(amax, fabsf(y));
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[i][e] = 0.f;
    }
  }
  const float blk_amax = block_max(amax, red);
  if (pass == 0) {
    if (threadIdx.x == 0) ws_amax[static_cast<size_t>(bh) * nblk + blk] = blk_amax;
    return;
  }
  float g = blk_amax;
  if (gran != 2) {  // tensor (0) or head (1): reduce the granule's block maxima
    const int lo = (gran == 0) ? 0 : bh * nblk;
    const int hi = (gran == 0) ? BH * nblk : (bh + 1) * nblk;
    float m = 0.f;
    for (int i = lo + threadIdx.x; i < hi; i += kThreads) m = fmaxf(m, ws_amax[i]);
    g = block_max(m, red);
  }
  const float inv = (g > 0.f) ? __fdiv_rn(127.0f, g) : 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = threadIdx.x + i * kThreads;
    const int r = v / VPR, cv = v % VPR;
    if (r < rows) {
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int q = __float2int_rn(__fmul_rn(x[i][e], inv));
        q = max(-127, min(127, q));
        w[e / 4] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (e % 4));
      }
      *reinterpret_cast<uint2*>(codes + (static_cast<size_t>(bh) * N + t0 + r) * D + cv * 8) =
          make_uint2(w[0], w[1]);
    }
  }
  if (threadIdx.x == 0) {
    const float sc = __fdiv_rn(g, 127.0f);
    if (gran == 2) scales[static_cast<size_t>(bh) * nblk + blk] = sc;
    else if (gran == 1 && blk == 0) scales[bh] = sc;
    else if (gran == 0 && blk == 0 && bh == 0) scales[0] = sc;
  }
}

__global__ void fill_ones_kernel(float* p, long long n) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    p[i] = 1.0f;
}

// ------------------------------------------------------------------ a3
// Per-channel amax of V over one chunk of tokens, merged with atomicMax on
// the (non-negative) float bit patterns.
template <int D, bool I8>
__global__ void __launch_bounds__(kThreads) v_amax_kernel(const void* __restrict__ V, int Nk,
                                                         unsigned int* __restrict__ amax_bits) {
  constexpr int EPV = I8 ? 16 : 8;
  constexpr int VPR = D / EPV;
  constexpr int RPI = kThreads / VPR;
  __shared__ float red[RPI * D];
  const int bh = blockIdx.y, chunk = blockIdx.x;
  const int v = threadIdx.x % VPR, r0 = threadIdx.x / VPR;
  float mx[EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) mx[e] = 0.f;
  const size_t row_bytes = static_cast<size_t>(D) * (I8 ? 1 : 2);
  const uint8_t* base = static_cast<const uint8_t*>(V) + static_cast<size_t>(bh) * Nk * row_bytes;
  const int t_end = min(Nk, (chunk + 1) * kTokPerChunk);
  for (int t = chunk * kTokPerChunk + r0; t < t_end; t += RPI) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(base + t * row_bytes) + v);
    if constexpr (I8) {
      float f[16];
      unpack_i8x16(raw, f);
#pragma unroll
      for (int e = 0; e < 16; ++e) mx[e] = fmaxf(mx[e], fabsf(f[e]));
    } else {
      float f[8];
      unpack_bf16x8(raw, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], fabsf(f[e]));
    }
  }
#pragma unroll
  for (int e = 0; e < EPV; ++e) red[r0 * D + v * EPV + e] = mx[e];
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += kThreads) {
    float m = 0.f;
    for (int r = 0; r < RPI; ++r) m = fmaxf(m, red[r * D + c]);
    atomicMax(amax_bits + static_cast<size_t>(bh) * D + c, __float_as_uint(m));
  }
}

// Quantize a 128-key slice of one (batch, KV head) to e4m3 and write it
// transposed: v8t[bh][c][t0 .. t0+127].  Keys >= Nk are written as 0; the
// write stops at the row stride ldv.
template <int D, bool I8>
__global__ void __launch_bounds__(kThreads) v_convert_kernel(
    const void* __restrict__ V, int Nk, const unsigned int* __restrict__ amax_bits,
    const float* __restrict__ chan, uint8_t* __restrict__ v8t, long long ldv,
    float* __restrict__ v_scales) {
  constexpr int EPV = I8 ? 16 : 8;
  constexpr int VPR = D / EPV;
  constexpr int PITCH = D + 1;  // floats per tile row (odd: fewer bank conflicts)
  extern __shared__ float tile[];  // [128][PITCH]
  __shared__ float inv_s[D];
  const int bh = blockIdx.y;
  const int t0 = blockIdx.x * 128;
  const size_t row_bytes = static_cast<size_t>(D) * (I8 ? 1 : 2);
  const uint8_t* base = static_cast<const uint8_t*>(V) + static_cast<size_t>(bh) * Nk * row_bytes;
  for (int v = threadIdx.x; v < 128 * VPR; v += kThreads) {
    const int r = v / VPR, cv = v % VPR;
    const int t = t0 + r;
    float* dst = tile + r * PITCH + cv * EPV;
    if (t < Nk) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(base + t * row_bytes) + cv);
      if constexpr (I8) {
        float f[16];
        unpack_i8x16(raw, f);
#pragma unroll
        for (int e = 0; e < 16; ++e) dst[e] = f[e];
      } else {
        float f[8];
        unpack_bf16x8(raw, f);
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[e] = f[e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < EPV; ++e) dst[e] = 0.f;
    }
  }
  for (int c = threadIdx.x; c < D; c += kThreads) {
    const float a = __uint_as_float(amax_bits[static_cast<size_t>(bh) * D + c]);
    inv_s[c] = (a > 0.f) ? __fdiv_rn(448.0f, a) : 0.f;
    if (blockIdx.x == 0) {
      const size_t i = static_cast<size_t>(bh) * D + c;
      v_scales[i] = I8 ? __fdiv_rn(__fmul_rn(chan[i], a), 448.0f) : __fdiv_rn(a, 448.0f);
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < D * 8; idx += kThreads) {
    const int c = idx / 8, k = idx % 8;
    const long long pos = t0 + 16 * k;
    if (pos >= ldv) continue;
    const float inv = inv_s[c];
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float* col = tile + (16 * k + 4 * q) * PITCH + c;
      const uint32_t lo = cvt_e4m3x2(__fmul_rn(col[0], inv), __fmul_rn(col[PITCH], inv));
      const uint32_t hi = cvt_e4m3x2(__fmul_rn(col[2 * PITCH], inv), __fmul_rn(col[3 * PITCH], inv));
      w[q] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(v8t + (static_cast<size_t>(bh) * D + c) * ldv + pos) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ------------------------------------------------------------------ carriers
// int8 codes -> fp16 values (exact: |code| <= 127).
__global__ void codes_to_f16_kernel(const int8_t* __restrict__ src, uint16_t* __restrict__ dst,
                                    size_t n16) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src) + i);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c0 = static_cast<int8_t>((w[j] >> (16 * e)) & 0xFFu);
        const int c1 = static_cast<int8_t>((w[j] >> (16 * e + 8)) & 0xFFu);
        const uint32_t h0 = __half_as_ushort(__int2half_rn(c0));
        const uint32_t h1 = __half_as_ushort(__int2half_rn(c1));
        o[2 * j + e] = h0 | (h1 << 16);
      }
    }
    uint4* d = reinterpret_cast<uint4*>(dst) + 2 * i;
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

int grid_for(size_t n, int threads) {
  size_t g = (n + threads - 1) / threads;
  if (g > 152 * 16) g = 152 * 16;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

size_t smooth_k_ws_bytes(long long BH, long long Nk, long long d) {
  const long long nchunks = (Nk + kTokPerChunk - 1) / kTokPerChunk;
  return static_cast<size_t>(BH * nchunks * d) * sizeof(long long);
}

cudaError_t launch_smooth_k(const uint16_t* K, int BH, int Nk, int d, long long* partials,
                            float* mu, cudaStream_t s) {
  const int nchunks = (Nk + kTokPerChunk - 1) / kTokPerChunk;
  if (nchunks > 0) {
    const size_t smem = static_cast<size_t>(kThreads / (d / 8)) * d * sizeof(long long);
    k_mean_partial_kernel<<<dim3(nchunks, BH), kThreads, smem, s>>>(K, Nk, d, nchunks, partials);
  }
  k_mean_finish_kernel<<<BH, 128, 0, s>>>(partials, nchunks, d, Nk, mu);
  return cudaGetLastError();
}

size_t quantize_rows_ws_bytes(long long B, long long H, long long N, int gran) {
  if (gran == 2) return 0;
  return static_cast<size_t>(B * H * ((N + 127) / 128)) * sizeof(float);
}

template <int D>
static void quant_rows_dispatch(dim3 grid, cudaStream_t s, const uint16_t* X, int H, int N,
                                int mode, const float* chan, int Hchan, int group, int gran,
                                int pass, int8_t* codes, float* scales, float* ws, int nblk,
                                int BH) {
  if (mode == 0)
    quant_rows_kernel<D, 0><<<grid, kThreads, 0, s>>>(X, H, N, chan, Hchan, group, gran, pass,
                                                      codes, scales, ws, nblk, BH);
  else if (mode == 1)
    quant_rows_kernel<D, 1><<<grid, kThreads, 0, s>>>(X, H, N, chan, Hchan, group, gran, pass,
                                                      codes, scales, ws, nblk, BH);
  else
    quant_rows_kernel<D, 2><<<grid, kThreads, 0, s>>>(X, H, N, chan, Hchan, group, gran, pass,
                                                      codes, scales, ws, nblk, BH);
}

cudaError_t launch_quantize_rows(const uint16_t* X, int B, int H, int N, int d, int mode,
                                 const float* chan, int Hchan, int gran, int8_t* codes,
                                 float* scales, float* ws_amax, cudaStream_t s) {
  const int nblk = (N + 127) / 128;
  const int BH = B * H;
  const int group = (mode == 2) ? H / Hchan : 1;
  const dim3 grid(nblk, BH);
  for (int pass = (gran == 2 ? 1 : 0); pass < 2; ++pass) {
    switch (d) {
      case 32:
        quant_rows_dispatch<32>(grid, s, X, H, N, mode, chan, Hchan, group, gran, pass, codes,
                                scales, ws_amax, nblk, BH);
        break;
      case 64:
        quant_rows_dispatch<64>(grid, s, X, H, N, mode, chan, Hchan, group, gran, pass, codes,
                                scales, ws_amax, nblk, BH);
        break;
      default:
        quant_rows_dispatch<128>(grid, s, X, H, N, mode, chan, Hchan, group, gran, pass, codes,
                                 scales, ws_amax, nblk, BH);
    }
  }
  return cudaGetLastError();
}

cudaError_t launch_fill_ones(float* p, long long n, cudaStream_t s) {
  if (n > 0) fill_ones_kernel<<<grid_for(static_cast<size_t>(n), 256), 256, 0, s>>>(p, n);
  return cudaGetLastError();
}

template <int D, bool I8>
static void quantize_v_impl(const void* V, const float* chan, int BH, int Nk, uint8_t* v8t,
                            long long ldv, float* v_scales, unsigned int* ws, cudaStream_t s) {
  const int nchunks = (Nk + kTokPerChunk - 1) / kTokPerChunk;
  v_amax_kernel<D, I8><<<dim3(nchunks, BH), kThreads, 0, s>>>(V, Nk, ws);
  const int nt = static_cast<int>((ldv + 127) / 128);
  const size_t smem = static_cast<size_t>(128) * (D + 1) * sizeof(float);
  cudaFuncSetAttribute(v_convert_kernel<D, I8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(smem));
  v_convert_kernel<D, I8><<<dim3(nt, BH), kThreads, smem, s>>>(V, Nk, ws, chan, v8t, ldv, v_scales);
}

cudaError_t launch_quantize_v(const void* V, int is_i8, const float* chan, int BH, int Nk, int d,
                              uint8_t* v8t, long long ldv, float* v_scales, unsigned int* ws_amax,
                              cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(ws_amax, 0, static_cast<size_t>(BH) * d * sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  if (Nk == 0) return cudaMemsetAsync(v_scales, 0, static_cast<size_t>(BH) * d * sizeof(float), s);
#define QATTN_QV(DD)                                                             \
  if (is_i8)                                                                     \
    quantize_v_impl<DD, true>(V, chan, BH, Nk, v8t, ldv, v_scales, ws_amax, s);  \
  else                                                                           \
    quantize_v_impl<DD, false>(V, chan, BH, Nk, v8t, ldv, v_scales, ws_amax, s);
  switch (d) {
    case 32: QATTN_QV(32) break;
    case 64: QATTN_QV(64) break;
    default: QATTN_QV(128)
  }
#undef QATTN_QV
  return cudaGetLastError();
}

cudaError_t launch_codes_to_f16(const int8_t* src, uint16_t* dst, size_t n, cudaStream_t s) {
  const size_t n16 = n / 16;
  if (n16 > 0) codes_to_f16_kernel<<<grid_for(n16, 256), 256, 0, s>>>(src, dst, n16);
  return cudaGetLastError();
}

}  // namespace qattn
