// Throughput loops for the roofline denominators of the attention kernels:
// the 5th-generation tensor cores (tcgen05.mma kind::f16 and kind::f8f6f4,
// the two instructions the fused attention issues), the warp-level mma.sync
// paths (s8, f16, e4m3: the legacy tensor path the short-sequence, integer
// and exact-split kernels use) and the MUFU ex2 rate (one per attention
// score).  Each loop runs on every SM with its operands resident in shared
// memory or registers, so it measures the execution unit and nothing else.
#include <cstdint>

#include <cuda_runtime.h>

#include "qattn_peaks.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kTcThreads = 128;
constexpr int kTcSmem = 160 * 1024;  // more than half an SM: one CTA per SM
constexpr int kATileBytes = 128 * 128;  // A: 128 rows x 128 bytes, 128B swizzle
constexpr int kBTileBytes = 256 * 128;  // B: up to 256 rows x 128 bytes

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Start and end of a CTA's loop: SM clock cycles and global nanoseconds, so
// the clock the loop ran at is cycles / nanoseconds.
__device__ __forceinline__ void stamp(unsigned long long* clocks, unsigned long long c0,
                                      unsigned long long c1, unsigned long long n0,
                                      unsigned long long n1) {
  clocks[4 * blockIdx.x] = c0;
  clocks[4 * blockIdx.x + 1] = c1;
  clocks[4 * blockIdx.x + 2] = n0;
  clocks[4 * blockIdx.x + 3] = n1;
}

// Deterministic pseudo-random 32-bit words (a multiplicative hash).
__device__ __forceinline__ uint32_t hash32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

// Fills the operand tiles with finite values of the kind's format (fp16 for
// kind::f16, e4m3 bytes for kind::f8f6f4).
__device__ void fill_operands(uint8_t* smem, int bytes, bool f8) {
  uint32_t* w = reinterpret_cast<uint32_t*>(smem);
  for (int i = threadIdx.x; i < bytes / 4; i += blockDim.x) {
    const uint32_t h = hash32(i * 2654435761u + blockIdx.x);
    // the top exponent bit cleared: fp16 and e4m3 values below 2 in
    // magnitude with random sign and mantissa (never inf or NaN)
    w[i] = f8 ? (h & 0xBFBFBFBFu) : (h & 0xBFFFBFFFu);
  }
}

// tcgen05 loop: iters rounds of 4 MMAs (M = 128, N = n, one 128-byte K slice
// each: K = 16 for kind::f16, K = 32 for kind::f8f6f4) into one TMEM
// accumulator, issued by one thread; the stamps bracket the first issue and
// the completion of the last MMA.
template <bool F8>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_loop_kernel(int n, int iters, unsigned long long* clocks, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sA = base, sB = base + kATileBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kATileBytes + kBTileBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kATileBytes + kBTileBytes + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kATileBytes + kBTileBytes + 12);
  const int warp = threadIdx.x >> 5;
  fill_operands(smem, kATileBytes + kBTileBytes, F8);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(bar), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  fence_proxy_async_smem();  // the operand stores are seen by the MMA unit
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) {
    const uint32_t idesc = make_idesc(128, static_cast<uint32_t>(n), 0, 0);
    uint64_t ad[4], bd[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      ad[s] = smem_desc(sA + s * 32, 1024, kSwizzle128B);
      bd[s] = smem_desc(sB + s * 32, 1024, kSwizzle128B);
    }
    const unsigned long long g0 = global_ns(), t0 = cycles();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        if (F8) mma_f8(tmem, ad[s], bd[s], idesc, (i | s) ? 1u : 0u);
        else mma_f16(tmem, ad[s], bd[s], idesc, (i | s) ? 1u : 0u);
      }
    }
    mma_commit(smem_u32(bar));
    const bool ok = mbar_wait(smem_u32(bar), 0, abort_flag, err, kQattnPeakErrTimeout);
    const unsigned long long t1 = cycles(), g1 = global_ns();
    stamp(clocks, t0, ok ? t1 : t0, g0, ok ? g1 : g0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// The fused attention's MMA sequence per key block and query tile: 8
// kind::f16 MMAs (M = 128, N = 128, K = 16; S = Q K^T over 128 channels) into
// one accumulator, then 4 kind::f8f6f4 MMAs (N = 128, K = 32; O += P V over
// 128 keys) into a second; operands are the same 128-byte-row tiles (finite
// as fp16 and as e4m3).
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_mixed_loop_kernel(int iters, unsigned long long* clocks, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sA = base, sB = base + kATileBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kATileBytes + kBTileBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kATileBytes + kBTileBytes + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kATileBytes + kBTileBytes + 12);
  const int warp = threadIdx.x >> 5;
  {
    uint32_t* w = reinterpret_cast<uint32_t*>(smem);
    for (int i = threadIdx.x; i < (kATileBytes + kBTileBytes) / 4; i += blockDim.x)
      w[i] = hash32(i * 2654435761u + blockIdx.x) & 0xBFBFBFBFu;  // finite in both formats
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(bar), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) {
    const uint32_t idesc = make_idesc(128, 128, 0, 0);
    uint64_t ad[4], bd[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      ad[s] = smem_desc(sA + s * 32, 1024, kSwizzle128B);
      bd[s] = smem_desc(sB + s * 32, 1024, kSwizzle128B);
    }
    const unsigned long long g0 = global_ns(), t0 = cycles();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int s = 0; s < 8; ++s) mma_f16(tmem, ad[s & 3], bd[s & 3], idesc, (i | s) ? 1u : 0u);
#pragma unroll
      for (int s = 0; s < 4; ++s) mma_f8(tmem + 128, ad[s], bd[s], idesc, (i | s) ? 1u : 0u);
    }
    mma_commit(smem_u32(bar));
    const bool ok = mbar_wait(smem_u32(bar), 0, abort_flag, err, kQattnPeakErrTimeout);
    const unsigned long long t1 = cycles(), g1 = global_ns();
    stamp(clocks, t0, ok ? t1 : t0, g0, ok ? g1 : g0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// mma.sync loop: every warp runs 8 independent accumulator chains.
// kind 0: m16n8k32 s8 x s8 -> s32; 1: m16n8k16 f16 x f16 -> f32;
// 2: m16n8k32 e4m3 x e4m3 -> f32.
template <int KIND>
__global__ void __launch_bounds__(256)
    warp_mma_loop_kernel(int iters, unsigned long long* clocks, unsigned int* sink) {
  const uint32_t h = hash32(threadIdx.x + 977u * blockIdx.x);
  // operand registers: s8 codes, fp16 pairs below 2 or e4m3 bytes below 128
  // in magnitude (never inf or NaN)
  const uint32_t a0 = KIND == 1 ? (h & 0x37FF37FFu) : KIND == 2 ? (h & 0x6F6F6F6Fu) : h;
  const uint32_t a1 = a0 ^ 0x01010101u, a2 = a0 ^ 0x02020202u, a3 = a0 ^ 0x04040404u;
  const uint32_t b0 = a0 ^ 0x08080808u, b1 = a0 ^ 0x03030303u;
  uint32_t acc[8][4];
#pragma unroll
  for (int c = 0; c < 8; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[c][e] = 0u;
  const unsigned long long g0 = global_ns(), t0 = cycles();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      if (KIND == 0) {
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      } else if (KIND == 1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      } else {
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      }
    }
  }
  __syncthreads();
  const unsigned long long t1 = cycles(), g1 = global_ns();
  uint32_t x = 0;
#pragma unroll
  for (int c = 0; c < 8; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) x ^= acc[c][e];
  if (x == 0x9E3779B9u) atomicAdd(sink, 1u);  // keeps the chains live
  if (threadIdx.x == 0) stamp(clocks, t0, t1, g0, g1);
}

// MUFU ex2 loop: 8 independent chains per thread, x <- -2^x stays in [-1, -0.5].
__global__ void __launch_bounds__(256)
    ex2_loop_kernel(int iters, unsigned long long* clocks, unsigned int* sink) {
  float x[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) x[c] = -0.5f - 0.0625f * c - 1e-6f * threadIdx.x;
  const unsigned long long g0 = global_ns(), t0 = cycles();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = -ex2_approx(x[c]);
  }
  __syncthreads();
  const unsigned long long t1 = cycles(), g1 = global_ns();
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) s += x[c];
  if (s == 1.0f) atomicAdd(sink, 1u);
  if (threadIdx.x == 0) stamp(clocks, t0, t1, g0, g1);
}

}  // namespace
}  // namespace qattn

extern "C" int qattn_peak_loop(int kind, int n, int iters, int blocks,
                               unsigned long long* clocks, unsigned int* err,
                               unsigned int* sink, void* stream) {
  using namespace qattn;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (iters <= 0 || blocks <= 0 || !clocks || !err || !sink) return 1;
  switch (kind) {
    case QATTN_PEAK_TC_F16:
    case QATTN_PEAK_TC_F8: {
      if (n != 64 && n != 128 && n != 256) return 1;
      const bool f8 = kind == QATTN_PEAK_TC_F8;
      auto k = f8 ? tc_loop_kernel<true> : tc_loop_kernel<false>;
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) !=
          cudaSuccess)
        return 3;
      k<<<blocks, kTcThreads, kTcSmem, s>>>(n, iters, clocks, err);
      break;
    }
    case QATTN_PEAK_TC_ATTN_MIX: {
      if (cudaFuncSetAttribute(tc_mixed_loop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kTcSmem) != cudaSuccess)
        return 3;
      tc_mixed_loop_kernel<<<blocks, kTcThreads, kTcSmem, s>>>(iters, clocks, err);
      break;
    }
    case QATTN_PEAK_MMA_S8: warp_mma_loop_kernel<0><<<blocks, 256, 0, s>>>(iters, clocks, sink); break;
    case QATTN_PEAK_MMA_F16: warp_mma_loop_kernel<1><<<blocks, 256, 0, s>>>(iters, clocks, sink); break;
    case QATTN_PEAK_MMA_E4M3: warp_mma_loop_kernel<2><<<blocks, 256, 0, s>>>(iters, clocks, sink); break;
    case QATTN_PEAK_EX2: ex2_loop_kernel<<<blocks, 256, 0, s>>>(iters, clocks, sink); break;
    default: return 1;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
