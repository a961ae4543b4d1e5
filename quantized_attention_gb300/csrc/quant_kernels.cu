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

#include "qattn_check.cuh"
#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kThreads = 256;
constexpr int kTokPerChunk = 64;  // tokens per CTA in the reduction passes

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
// round_half_even(x * 2^24) for a bf16 bit pattern, with integer operations
// only (exact: x = M * 2^(e - 134) with the 8-bit significand M, so
// x * 2^24 = M * 2^(e - 110)).  Valid for finite |x| < 2^39.
__device__ __forceinline__ long long bf16_fix24(uint32_t b) {
  const int e = (b >> 7) & 0xFF;
  uint32_t M = b & 0x7Fu;
  int ee = e;
  if (e == 0) ee = 1;  // subnormal: no implicit bit
  else M |= 0x80u;
  const int sh = ee - 110;
  long long v;
  if (sh >= 0) {
    v = static_cast<long long>(M) << sh;
  } else {
    const int r = -sh;
    if (r > 9) {
      v = 0;  // M < 2^8, so M / 2^r < 1/2
    } else {
      uint32_t q = M >> r;
      const uint32_t rem = M & ((1u << r) - 1u), half = 1u << (r - 1);
      if (rem > half || (rem == half && (q & 1u))) ++q;
      v = q;
    }
  }
  return (b & 0x8000u) ? -v : v;
}

// round_half_even(x * 2^24) for many x at once, without 64-bit integer work.
// With y = x * 2^24 (exact) and C1 = 1.5 * 2^46 (ulp 2^23):
//   t  = fl(y + C1)            t = C1 + h * 2^23, h = rne(y / 2^23), |h| < 2^22
//   lo = y - (t - C1)          exact, |lo| <= 2^22
//   u  = fl(lo + C2)           C2 = 1.5 * 2^23 (ulp 1): u = C2 + rne(lo)
// so rne(y) = h * 2^23 + rne(lo) (h * 2^23 is even, so ties round alike), with
// h = bits(t) - bits(C1) and rne(lo) = bits(u) - bits(C2): integers that a
// thread sums in 32 bits (the bias terms are removed once, at the end).  Valid
// for |x| < 2^21; larger inputs take bf16_fix24.
constexpr float kFixScale = 0x1p24f;
constexpr float kFixC1 = 0x1.8p46f;
constexpr float kFixC2 = 0x1.8p23f;
constexpr uint32_t kFixC1Bits = 0x56C00000u;
constexpr uint32_t kFixC2Bits = 0x4B400000u;
constexpr uint32_t kFixMaxMag = 0x4A00u;  // bf16 magnitude bits of 2^21

// Accumulates the fixed-point values of the 8 bf16 in `raw` into the biased
// sums at/au (see above) and the largest magnitude pattern into mx.
__device__ __forceinline__ void fix24_accumulate8(const uint4& raw, uint32_t (&at)[8],
                                                  uint32_t (&au)[8], uint32_t& mx) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    mx = __vmaxu2(mx, w[e] & 0x7FFF7FFFu);
    const float2 x = make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
    const float2 t = ffma2(x, make_float2(kFixScale, kFixScale), make_float2(kFixC1, kFixC1));
    const float2 nhi = ffma2(t, make_float2(-1.f, -1.f), make_float2(kFixC1, kFixC1));  // -(t - C1)
    const float2 lo = ffma2(x, make_float2(kFixScale, kFixScale), nhi);
    const float2 u = fadd2(lo, make_float2(kFixC2, kFixC2));
    at[2 * e] += __float_as_uint(t.x);
    at[2 * e + 1] += __float_as_uint(t.y);
    au[2 * e] += __float_as_uint(u.x);
    au[2 * e + 1] += __float_as_uint(u.y);
  }
}

// Sum over NIT rows of one 16-byte column vector: the 8 channels' exact
// sums of round(K * 2^24).  Rows past the end were loaded as zeros.
template <int NIT>
__device__ __forceinline__ void fix24_column_sums(const uint4 (&raw)[NIT], long long (&sum)[8]) {
  uint32_t at[8], au[8], mx = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) at[e] = au[e] = 0u;
#pragma unroll
  for (int it = 0; it < NIT; ++it) fix24_accumulate8(raw[it], at, au, mx);
  if (max(mx & 0xFFFFu, mx >> 16) < kFixMaxMag) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int h = static_cast<int>(at[e] - NIT * kFixC1Bits);
      const int r = static_cast<int>(au[e] - NIT * kFixC2Bits);
      sum[e] = static_cast<long long>(h) * (1ll << 23) + r;
    }
  } else {  // some |x| >= 2^21: the general integer decode
#pragma unroll
    for (int e = 0; e < 8; ++e) sum[e] = 0;
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const uint32_t w[4] = {raw[it].x, raw[it].y, raw[it].z, raw[it].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sum[2 * e] += bf16_fix24(w[e] & 0xFFFFu);
        sum[2 * e + 1] += bf16_fix24(w[e] >> 16);
      }
    }
  }
}

// x = q * N + r (0 <= r < N) for x < 2^57, with M = floor((2^64 - 1) / N):
// q_est = floor(x * M / 2^64) is floor(x / N) or one less.
__device__ __forceinline__ void udivmod(unsigned long long x, uint32_t N, unsigned long long M,
                                        unsigned long long& q, unsigned long long& r) {
  q = __umul64hi(x, M);
  r = x - q * N;
  if (r >= N) {
    ++q;
    r -= N;
  }
}

// mu = fp32(fp64(S) * 2^-24 / N), computed as the correctly rounded fp32
// quotient |S| / N (then scaled by 2^-24) with integer long division -- no
// fp64, whose throughput on this part is a small fraction of fp32's.
// The two agree.  With A = |S| < 2^53 and N < 2^24, rounding A / N to fp64
// first could change the fp32 result only by landing exactly on an fp32
// rounding midpoint b != A / N, i.e. 0 < |A/N - b| <= 2^(e-53) for b in
// [2^e, 2^(e+1)).  But N (A/N - b) is a nonzero multiple of 2^(e-24), so
// |A/N - b| >= 2^(e-24) / N > 2^(e-48); and if e > 24, b is an integer, so
// |A/N - b| >= 1/N, which is > 2^(e-53) unless N >= 2^(53-e), and then
// A ~ N b > 2^53.  Both cases are impossible.
__device__ __forceinline__ float mean_of_fix24(long long S, uint32_t N, unsigned long long M) {
  if (S == 0) return 0.f;
  const unsigned long long A = S < 0 ? 0ull - static_cast<unsigned long long>(S)
                                     : static_cast<unsigned long long>(S);
  unsigned long long Q, R;
  udivmod(A, N, M, Q, R);  // A / N = (Q + R / N) * 2^-fr, fr = 0 so far
  int fr = 0;
  int bl = 64 - __clzll(static_cast<long long>(Q));
  while (bl < 25) {  // append quotient bits until Q holds 25 (24 + a guard bit)
    const int m = min(32, 25 - bl);
    unsigned long long q2, r2;
    udivmod(R << m, N, M, q2, r2);
    Q = (Q << m) | q2;
    R = r2;
    fr += m;
    bl = 64 - __clzll(static_cast<long long>(Q));
  }
  const int drop = bl - 25;
  const bool sticky = (R != 0) || (drop > 0 && (Q & ((1ull << drop) - 1ull)) != 0);
  const unsigned long long T = Q >> drop;  // 25 bits
  fr -= drop;
  uint32_t U = static_cast<uint32_t>(T >> 1);  // 24 bits, value U * 2^(1 - fr)
  if ((T & 1ull) && (sticky || (U & 1u))) ++U;  // round half to even
  int e = 1 - fr - 24;  // value / 2^24 = U * 2^e
  if (U == (1u << 24)) {
    U >>= 1;
    ++e;
  }
  const uint32_t bits = (static_cast<uint32_t>(e + 23 + 127) << 23) | (U - (1u << 23));
  return __uint_as_float(bits | (S < 0 ? 0x80000000u : 0u));
}

// First element of (batch, head) bh's slice of an input tensor.
template <typename T>
__device__ __forceinline__ const T* src_head(const Src& x, int bh) {
  const int b = bh / x.H, h = bh - b * x.H;
  return static_cast<const T*>(x.p) + static_cast<long long>(b) * x.sB + static_cast<long long>(h) * x.sH;
}

constexpr int kMeanRows = 8;  // rows per thread in the mean kernels

// Channel mean for short heads: one warp per (batch, head), all Nk rows
// (Nk <= 8 * 32 / (D / 8)); lanes = (row group, 16-byte column).
template <int D>
__global__ void __launch_bounds__(kThreads) k_mean_warp_kernel(const Src K, int BH, int Nk,
                                                              unsigned long long magic,
                                                              float* __restrict__ mu) {
  pdl_trigger();
  pdl_wait();
  constexpr int VPR = D / 8;
  constexpr int RG = 32 / VPR;
  const int bh = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (bh >= BH) return;
  const int lane = threadIdx.x & 31;
  const int v = lane % VPR, rg = lane / VPR;
  const uint16_t* base = src_head<uint16_t>(K, bh);
  uint4 raw[kMeanRows];
#pragma unroll
  for (int it = 0; it < kMeanRows; ++it) {
    const int t = rg + it * RG;
    raw[it] = (t < Nk) ? __ldg(reinterpret_cast<const uint4*>(base + static_cast<long long>(t) * K.sN) + v)
                       : make_uint4(0u, 0u, 0u, 0u);
  }
  long long sum[8];
  fix24_column_sums<kMeanRows>(raw, sum);
#pragma unroll
  for (int o = VPR; o < 32; o <<= 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) sum[e] += __shfl_xor_sync(0xffffffffu, sum[e], o);
  }
  // Every lane now holds its column's 8 sums; the RG lanes of a column share
  // the 8 divisions between them.
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (e % RG == rg)
      mu[static_cast<size_t>(bh) * D + v * 8 + e] =
          mean_of_fix24(sum[e], static_cast<uint32_t>(Nk), magic);
  }
}

// Channel mean over CTA-sized chunks of kMeanRows * (256 / (D / 8)) rows.
// MULTI = false: one chunk holds the whole head and the CTA writes mu.
// MULTI = true: each chunk adds its sums into acc[bh][c] with 64-bit atomics
// (integer, so the order does not matter) and the last CTA of the head to
// finish writes mu; acc and done must start at zero.
template <int D>
struct KMeanSmem {
  static constexpr int RG = kThreads / (D / 8);  // row groups per CTA
  long long red[RG][D];
  unsigned int last;
};

template <int D, bool MULTI>
__device__ __forceinline__ void k_mean_chunk(const Src& K, int Nk, int nchunks,
                                             unsigned long long magic,
                                             unsigned long long* __restrict__ acc,
                                             unsigned int* __restrict__ done, float* __restrict__ mu,
                                             int chunk, int bh, KMeanSmem<D>& sm) {
  constexpr int VPR = D / 8;           // 16-byte vectors per row
  constexpr int RG = KMeanSmem<D>::RG;
  constexpr int kChunk = RG * kMeanRows;
  auto& red = sm.red;
  unsigned int& last = sm.last;
  const int v = threadIdx.x % VPR, rg = threadIdx.x / VPR;
  const uint16_t* base = src_head<uint16_t>(K, bh);
  uint4 raw[kMeanRows];
#pragma unroll
  for (int it = 0; it < kMeanRows; ++it) {
    const int t = chunk * kChunk + rg + it * RG;
    raw[it] = (t < Nk) ? __ldg(reinterpret_cast<const uint4*>(base + static_cast<long long>(t) * K.sN) + v)
                       : make_uint4(0u, 0u, 0u, 0u);
  }
  long long sum[8];
  fix24_column_sums<kMeanRows>(raw, sum);
#pragma unroll
  for (int e = 0; e < 8; ++e) red[rg][v * 8 + e] = sum[e];
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += kThreads) {
    long long tot = 0;
#pragma unroll 8
    for (int r = 0; r < RG; ++r) tot += red[r][c];
    if (!MULTI) mu[static_cast<size_t>(bh) * D + c] = mean_of_fix24(tot, static_cast<uint32_t>(Nk), magic);
    else atomicAdd(acc + static_cast<size_t>(bh) * D + c, static_cast<unsigned long long>(tot));
  }
  if (!MULTI) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(done + bh, 1u) == static_cast<unsigned int>(nchunks - 1));
  __syncthreads();
  if (last) {
    __threadfence();
    for (int c = threadIdx.x; c < D; c += kThreads) {
      const long long tot =
          static_cast<long long>(atomicAdd(acc + static_cast<size_t>(bh) * D + c, 0ull));
      mu[static_cast<size_t>(bh) * D + c] = mean_of_fix24(tot, static_cast<uint32_t>(Nk), magic);
    }
  }
}

template <int D, bool MULTI>
__global__ void __launch_bounds__(kThreads) k_mean_kernel(const Src K, int Nk,
                                                         int nchunks, unsigned long long magic,
                                                         unsigned long long* __restrict__ acc,
                                                         unsigned int* __restrict__ done,
                                                         float* __restrict__ mu) {
  pdl_trigger();
  pdl_wait();
  __shared__ KMeanSmem<D> sm;
  k_mean_chunk<D, MULTI>(K, Nk, nchunks, magic, acc, done, mu, blockIdx.x, blockIdx.y, sm);
}

// ------------------------------------------------------------------ a2
// One CTA per (batch*head, 128-token block) of a job.  MODE 0: x = X;
// 1: x = X - chan (K minus its channel mean); 2: x = X * chan (Q times K's
// channel scale).  pass 0 writes the block's amax (tensor/head granules);
// pass 1 quantizes.  The raw bf16 vectors stay in registers and x is
// recomputed when quantizing, which halves the registers and doubles the
// CTAs per SM.
template <int D, int MODE>
__device__ __forceinline__ void load_x8(const uint4& raw, const float (&ch)[8], float (&x)[8]) {
  unpack_bf16x8(raw, x);
  if (MODE != 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (MODE == 1) ? __fsub_rn(x[e], ch[e]) : __fmul_rn(x[e], ch[e]);
  }
}

template <int D, int MODE>
__device__ __forceinline__ void quant_rows_body(const RowsJob& j, int bh, int blk, int pass,
                                                float* red) {
  constexpr int VPR = D / 8;
  constexpr int NV = 128 * VPR / kThreads;
  if (pass == 0 && j.gran == 2) return;  // block granules need no pre-pass
  const int b = bh / j.H, h = bh % j.H;
  const int t0 = blk * 128;
  const int rows = min(128, j.N - t0);
  const uint16_t* src = j.X + static_cast<long long>(b) * j.sB + static_cast<long long>(h) * j.sH +
                        static_cast<long long>(t0) * j.sN;
  // Every vector a thread handles is the same 8 channels (kThreads % VPR == 0).
  static_assert(kThreads % VPR == 0, "fixed channel group per thread");
  float ch[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (MODE != 0) {
    const float* crow = j.chan + (static_cast<size_t>(b) * j.Hchan + h / j.group) * D;
#pragma unroll
    for (int e = 0; e < 8; ++e) ch[e] = crow[(threadIdx.x % VPR) * 8 + e];  // written by the K mean pass
  }

  uint4 raw[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = threadIdx.x + i * kThreads;
    const int r = v / VPR, cv = v % VPR;
    raw[i] = (r < rows) ? __ldg(reinterpret_cast<const uint4*>(src + static_cast<long long>(r) * j.sN) + cv)
                        : make_uint4(0u, 0u, 0u, 0u);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = threadIdx.x + i * kThreads;
    if (v / VPR < rows) {
      float x[8];
      load_x8<D, MODE>(raw[i], ch, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
    }
  }
  const float blk_amax = block_max(amax, red);
  if (pass == 0) {
    if (threadIdx.x == 0) j.ws_amax[static_cast<size_t>(bh) * j.nblk + blk] = blk_amax;
    return;
  }
  float g = blk_amax;
  if (j.gran != 2) {  // tensor (0) or head (1): reduce the granule's block maxima
    const int lo = (j.gran == 0) ? 0 : bh * j.nblk;
    const int hi = (j.gran == 0) ? j.BH * j.nblk : (bh + 1) * j.nblk;
    float m = 0.f;
    for (int i = lo + threadIdx.x; i < hi; i += kThreads) m = fmaxf(m, j.ws_amax[i]);
    g = block_max(m, red);
  }
  const float inv = (g > 0.f) ? __fdiv_rn(127.0f, g) : 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = threadIdx.x + i * kThreads;
    const int r = v / VPR, cv = v % VPR;
    if (r < rows) {
      float x[8];
      load_x8<D, MODE>(raw[i], ch, x);
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int q = __float2int_rn(__fmul_rn(x[e], inv));
        q = max(-127, min(127, q));
        w[e / 4] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (e % 4));
      }
      const size_t off = (static_cast<size_t>(bh) * j.N + t0 + r) * D + cv * 8;
      if (!QATTN_IN_BOUNDS(bh < j.BH && t0 + r < j.N && cv * 8 < D)) continue;
      *reinterpret_cast<uint2*>(j.codes + off) = make_uint2(w[0], w[1]);
      if (j.carrier != nullptr) {
        uint4 h;
        codes4_to_f16x2(w[0], h.x, h.y);
        codes4_to_f16x2(w[1], h.z, h.w);
        *reinterpret_cast<uint4*>(j.carrier + off) = h;
      }
    }
  }
  if (threadIdx.x == 0) {
    const float sc = __fdiv_rn(g, 127.0f);
    if (j.gran == 2) j.scales[static_cast<size_t>(bh) * j.nblk + blk] = sc;
    else if (j.gran == 1 && blk == 0) j.scales[bh] = sc;
    else if (j.gran == 0 && blk == 0 && bh == 0) j.scales[0] = sc;
  }
}

// Q and K in one launch: blockIdx.x < j0.BH are (batch, head)s of job 0, the
// rest of job 1; blockIdx.y is the 128-token block.
template <int D, int M0, int M1>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(const RowsJob j0, const RowsJob j1,
                                                             int pass) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[kThreads / 32];
  if (pass == 1 && j0.n_ones > 0) {  // spread over every CTA of the launch
    const long long nthr = static_cast<long long>(gridDim.x) * gridDim.y * kThreads;
    for (long long i = (static_cast<long long>(blockIdx.y) * gridDim.x + blockIdx.x) * kThreads + threadIdx.x;
         i < j0.n_ones; i += nthr)
      j0.ones[i] = 1.0f;
  }
  const int x = blockIdx.x, blk = blockIdx.y;
  if (x < j0.BH) {
    if (blk < j0.nblk) quant_rows_body<D, M0>(j0, x, blk, pass, red);
  } else if (blk < j1.nblk) {
    quant_rows_body<D, M1>(j1, x - j0.BH, blk, pass, red);
  }
}

// ------------------------------------------------------------------ a3
// Per-channel amax of V over one chunk of tokens (every load issued before any
// is used), merged with atomicMax on the (non-negative) float bit patterns.
template <int D, bool I8>
struct VAmaxSmem {
  static constexpr int RPI = kThreads / (D / (I8 ? 16 : 8));  // rows per iteration
  float red[RPI * D];
};

template <int D, bool I8>
__device__ __forceinline__ void v_amax_chunk(const Src& V, int Nk,
                                             unsigned int* __restrict__ amax_bits, int chunk, int bh,
                                             VAmaxSmem<D, I8>& sm) {
  constexpr int EPV = I8 ? 16 : 8;
  constexpr int VPR = D / EPV;
  constexpr int RPI = VAmaxSmem<D, I8>::RPI;
  constexpr int NIT = (kTokPerChunk + RPI - 1) / RPI;
  float* red = sm.red;
  const int v = threadIdx.x % VPR, r0 = threadIdx.x / VPR;
  constexpr int kElem = I8 ? 1 : 2;  // bytes per element
  const uint8_t* base = reinterpret_cast<const uint8_t*>(src_head<uint8_t>(
      Src{V.p, V.sB * kElem, V.sH * kElem, V.sN * kElem, V.H}, bh));
  const long long row_bytes = V.sN * kElem;
  uint4 raw[NIT];
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int r = r0 + it * RPI;
    const int t = chunk * kTokPerChunk + r;
    raw[it] = (r < kTokPerChunk && t < Nk) ? __ldg(reinterpret_cast<const uint4*>(base + t * row_bytes) + v)
                                           : make_uint4(0u, 0u, 0u, 0u);
  }
  float mx[EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) mx[e] = 0.f;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    if constexpr (I8) {
      float f[16];
      unpack_i8x16(raw[it], f);
#pragma unroll
      for (int e = 0; e < 16; ++e) mx[e] = fmaxf(mx[e], fabsf(f[e]));
    } else {
      float f[8];
      unpack_bf16x8(raw[it], f);
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

template <int D, bool I8>
__global__ void __launch_bounds__(kThreads) v_amax_kernel(const Src V, int Nk,
                                                         unsigned int* __restrict__ amax_bits) {
  pdl_trigger();
  pdl_wait();
  __shared__ VAmaxSmem<D, I8> sm;
  v_amax_chunk<D, I8>(V, Nk, amax_bits, blockIdx.x, blockIdx.y, sm);
}

// Quantize a 128-key slice of one (batch, KV head) to e4m3 and write it
// transposed: v8t[bh][c][t0 .. t0+127].  Lane l of a warp owns keys
// 4l .. 4l+3 and reads, for each, 32 contiguous bytes of the row (two 16-byte
// vectors: a whole sector); each warp takes its own channel slices.  The four
// keys' e4m3 bytes of one channel form one word, stored at [c][4l] of a
// [D][128]-byte tile: the 32 lanes write 32 consecutive words (no bank
// conflict).  The tile leaves as 16-byte rows.  Keys >= Nk are written as 0;
// the write stops at the row stride ldv.
template <int D>
struct VConvSmem {
  __align__(16) uint8_t tile[D * 128];
  float inv_s[D];
};

template <int D, bool I8>
__device__ __forceinline__ void v_convert_slice(const Src& V, int Nk,
                                                const unsigned int* amax_bits,
                                                const float* __restrict__ chan,
                                                uint8_t* __restrict__ v8t, long long ldv,
                                                float* __restrict__ v_scales, int tblk, int bh,
                                                VConvSmem<D>& sm) {
  constexpr int EPV = I8 ? 16 : 8;        // channels per 16-byte vector
  constexpr int kSlices = D / (2 * EPV);  // 32-byte channel slices per key row
  constexpr int kWarps = kThreads / 32;
  constexpr int NS = (kSlices + kWarps - 1) / kWarps;  // slices per warp
  uint8_t* tile = sm.tile;
  float* inv_s = sm.inv_s;
  const int t0 = tblk * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kElem = I8 ? 1 : 2;  // bytes per element
  const uint8_t* base = reinterpret_cast<const uint8_t*>(src_head<uint8_t>(
      Src{V.p, V.sB * kElem, V.sH * kElem, V.sN * kElem, V.H}, bh));
  const long long row_bytes = V.sN * kElem;
  uint4 raw[NS][4][2];
#pragma unroll
  for (int u = 0; u < NS; ++u) {
    const int sl = warp + u * kWarps;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int t = t0 + 4 * lane + q;
      const bool in = (sl < kSlices) && (t < Nk);
      const uint4* src = reinterpret_cast<const uint4*>(base + t * row_bytes) + 2 * sl;
      raw[u][q][0] = in ? __ldg(src) : make_uint4(0u, 0u, 0u, 0u);
      raw[u][q][1] = in ? __ldg(src + 1) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  for (int c = threadIdx.x; c < D; c += kThreads) {
    const float a = __uint_as_float(amax_bits[static_cast<size_t>(bh) * D + c]);
    inv_s[c] = (a > 0.f) ? __fdiv_rn(448.0f, a) : 0.f;
    if (tblk == 0) {
      const size_t i = static_cast<size_t>(bh) * D + c;
      v_scales[i] = I8 ? __fdiv_rn(__fmul_rn(chan[i], a), 448.0f) : __fdiv_rn(a, 448.0f);
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < NS; ++u) {
    const int sl = warp + u * kWarps;
    if (sl >= kSlices) continue;
#pragma unroll
    for (int v = 0; v < 2; ++v) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const int c = (2 * sl + v) * EPV + e;
        const float sc = inv_s[c];
        float x[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 r4 = raw[u][q][v];
          if constexpr (I8) {
            const uint32_t w = (e < 4) ? r4.x : (e < 8) ? r4.y : (e < 12) ? r4.z : r4.w;
            x[q] = static_cast<float>(static_cast<int8_t>((w >> (8 * (e % 4))) & 0xFFu));
          } else {
            const uint32_t w = (e < 2) ? r4.x : (e < 4) ? r4.y : (e < 6) ? r4.z : r4.w;
            x[q] = __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
          }
        }
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(x[0], sc), __fmul_rn(x[1], sc));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(x[2], sc), __fmul_rn(x[3], sc));
        *reinterpret_cast<uint32_t*>(tile + c * 128 + 4 * lane) = lo | (hi << 16);
      }
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < D * 8; idx += kThreads) {
    const int c = idx / 8, k = idx % 8;
    const long long pos = t0 + 16 * k;
    if (pos >= ldv) continue;
    const uint4 w = *reinterpret_cast<const uint4*>(tile + c * 128 + 16 * k);
    *reinterpret_cast<uint4*>(v8t + (static_cast<size_t>(bh) * D + c) * ldv + pos) = w;
  }
}

template <int D, bool I8>
__global__ void __launch_bounds__(kThreads) v_convert_kernel(
    const Src V, int Nk, const unsigned int* amax_bits,
    const float* __restrict__ chan, uint8_t* __restrict__ v8t, long long ldv,
    float* __restrict__ v_scales) {
  pdl_trigger();
  pdl_wait();
  __shared__ VConvSmem<D> sm;
  v_convert_slice<D, I8>(V, Nk, amax_bits, chan, v8t, ldv, v_scales, blockIdx.x, blockIdx.y, sm);
}

// ------------------------------------------------------------------ a1-a3 in two launches
// The whole pre-pass for bf16 Q, K, V with block granules.  Launch 1: Q's
// codes | K's channel sums (the last CTA of a head writes its mean) | V's
// channel maxima -- three independent jobs in one grid.  Launch 2: K's codes
// (and carriers) from K minus its mean | V's e4m3 transpose.  Each CTA runs
// one of the bodies the separate kernels run, so the outputs are the same.
struct Prep1Args {
  RowsJob jq;
  Src K;
  Src V;
  int BHk, Nk, nkc, nvc;
  unsigned long long magic;
  unsigned long long* acc;
  unsigned int* done;
  float* mu;
  unsigned int* amax;
};

struct Prep2Args {
  RowsJob jk;
  Src V;
  int Nk, nvt;
  const unsigned int* amax;
  uint8_t* v8t;
  long long ldv;
  float* v_scales;
};

constexpr size_t cmax(size_t a, size_t b) { return a > b ? a : b; }

// 64 registers: four CTAs per SM, as the separate Q/K quantizer runs.
template <int D>
__global__ void __launch_bounds__(kThreads, 4) prepare1_kernel(const Prep1Args p) {
  pdl_trigger();
  pdl_wait();
  constexpr size_t kBytes =
      cmax(cmax(sizeof(KMeanSmem<D>), sizeof(VAmaxSmem<D, false>)), (kThreads / 32) * sizeof(float));
  __shared__ __align__(16) unsigned char sm[kBytes];
  int x = blockIdx.x;
  const int nq = p.jq.BH * p.jq.nblk;
  if (x < nq) {
    quant_rows_body<D, 0>(p.jq, x / p.jq.nblk, x % p.jq.nblk, 1, reinterpret_cast<float*>(sm));
    return;
  }
  x -= nq;
  const int nk = p.nkc * p.BHk;
  if (x < nk) {
    k_mean_chunk<D, true>(p.K, p.Nk, p.nkc, p.magic, p.acc, p.done, p.mu, x % p.nkc, x / p.nkc,
                          *reinterpret_cast<KMeanSmem<D>*>(sm));
    return;
  }
  x -= nk;
  v_amax_chunk<D, false>(p.V, p.Nk, p.amax, x % p.nvc, x / p.nvc,
                         *reinterpret_cast<VAmaxSmem<D, false>*>(sm));
}

template <int D>
__global__ void __launch_bounds__(kThreads) prepare2_kernel(const Prep2Args p) {
  pdl_trigger();
  pdl_wait();
  constexpr size_t kBytes = cmax(sizeof(VConvSmem<D>), (kThreads / 32) * sizeof(float));
  __shared__ __align__(16) unsigned char sm[kBytes];
  const int nk = p.jk.BH * p.jk.nblk;
  const int x = blockIdx.x;
  if (x < nk) {
    quant_rows_body<D, 1>(p.jk, x / p.jk.nblk, x % p.jk.nblk, 1, reinterpret_cast<float*>(sm));
    return;
  }
  const int y = x - nk;
  v_convert_slice<D, false>(p.V, p.Nk, p.amax, nullptr, p.v8t, p.ldv, p.v_scales, y % p.nvt, y / p.nvt,
                            *reinterpret_cast<VConvSmem<D>*>(sm));
}

// ------------------------------------------------------------------ a1-a3, short heads
// Heads of at most 128 tokens and d <= 64 (one block granule each, e.g. Swin
// windows; the V8^T tiles of d = 128 would not fit the static shared memory): one
// warp runs a head's whole pre-pass in one launch -- a KV head's channel mean
// (exact fixed-point sums), its K codes (and carriers), its V channel maxima and
// transposed e4m3 codes; a Q head's codes -- re-reading the head's few KB from
// L1 between passes.  The arithmetic is that of the bodies above, step by step.
constexpr int kSmallHead = 128;  // tokens per head at most
constexpr int kSmallWarps = 4;

struct SmallPrepArgs {
  Src Q, K, V;
  int BHq, BHk, Nq, Nk;
  unsigned long long magic;
  int8_t* q_codes;
  float* q_scales;
  int8_t* k_codes;
  float* k_scales;
  uint16_t* k_carrier;
  float* k_mean;
  uint8_t* v8t;
  long long ldv;
  float* v_scales;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// The 8 codes of x (8 channels) at inv, and (optionally) their fp16 carriers.
__device__ __forceinline__ void codes8(const float (&x)[8], float inv, int8_t* dst, uint16_t* carrier) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    int q = __float2int_rn(__fmul_rn(x[e], inv));
    q = max(-127, min(127, q));
    w[e / 4] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (e % 4));
  }
  *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
  if (carrier != nullptr) {
    uint4 h;
    codes4_to_f16x2(w[0], h.x, h.y);
    codes4_to_f16x2(w[1], h.z, h.w);
    *reinterpret_cast<uint4*>(carrier) = h;
  }
}

// Per-warp pieces of a short head's pre-pass.  Lane (rg, v) handles rows rg,
// rg + RG, ... and the 8 channels of 16-byte column v.
template <int D>
struct HeadLane {
  static constexpr int VPR = D / 8;    // 16-byte vectors per row
  static constexpr int RG = 32 / VPR;  // row groups per warp
  static constexpr int UNR = 8;        // rows a lane loads before it uses them
  int v, rg;
  __device__ explicit HeadLane(int lane) : v(lane % VPR), rg(lane / VPR) {}
  // Rows r0, r0 + RG, ... (UNR of them) of the lane's column; zeros past N.
  // rows of a head at a row stride of sN elements
  __device__ void load_rows(const uint16_t* head, long long sN, int N, int r0,
                            uint4 (&raw)[UNR]) const {
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u * RG;
      raw[u] = (r < N) ? *(reinterpret_cast<const uint4*>(head + static_cast<long long>(r) * sN) + v)
                       : make_uint4(0u, 0u, 0u, 0u);
    }
  }
};

// Brings a head's rows into L1 (prefetch.global.L1: no registers, no wait)
// so a later pass over them finds them there: each lane touches the lines of
// its own rows.
template <int D>
__device__ __forceinline__ void head_prefetch_l1(const HeadLane<D>& L, const uint16_t* head, long long sN,
                                                 int N) {
  for (int r = L.rg; r < N; r += HeadLane<D>::RG)
    asm volatile("prefetch.global.L1 [%0];" ::"l"(head + static_cast<long long>(r) * sN + 8 * L.v));
}

// The channel mean of a head's N rows (exact fixed-point sums), every lane of a
// column holding its 8 channels' means.
template <int D>
__device__ __forceinline__ void head_mean(const HeadLane<D>& L, const uint16_t* head, long long sN, int N,
                                          unsigned long long magic, float (&mu)[8]) {
  constexpr int RG = HeadLane<D>::RG, UNR = HeadLane<D>::UNR;
  long long sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int r0 = L.rg; r0 < N; r0 += UNR * RG) {
    uint4 raw[UNR];
    L.load_rows(head, sN, N, r0, raw);  // rows past N are zeros: they add nothing
    long long s8[8];
    fix24_column_sums<UNR>(raw, s8);
#pragma unroll
    for (int e = 0; e < 8; ++e) sum[e] += s8[e];
  }
#pragma unroll
  for (int o = HeadLane<D>::VPR; o < 32; o <<= 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) sum[e] += __shfl_xor_sync(0xffffffffu, sum[e], o);
  }
  // Every lane of a column now holds its 8 sums; the RG lanes of the column
  // share the 8 divisions (lane rg takes channels e = rg, rg + RG, ...) and
  // hand the means round: lane (e % RG) * VPR + v holds channel e's.
  constexpr int VPR = HeadLane<D>::VPR;
  static_assert(8 % RG == 0, "every lane of a column takes the same number of channels");
  constexpr int PER = 8 / RG;  // divisions per lane
  float own[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = L.rg + i * RG;  // < 8 for every lane when RG divides 8
    long long se = sum[0];
#pragma unroll
    for (int ee = 1; ee < 8; ++ee) se = (ee == e) ? sum[ee] : se;  // selects, no divergence
    own[i] = mean_of_fix24(se, static_cast<uint32_t>(N), magic);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) mu[e] = __shfl_sync(0xffffffffu, own[e / RG], (e % RG) * VPR + L.v);
}

// max |x - mu| (MINUS) or max |x| over a head's rows, over the whole warp.
template <int D, bool MINUS>
__device__ __forceinline__ float head_amax(const HeadLane<D>& L, const uint16_t* head, long long sN, int N,
                                           const float (&mu)[8]) {
  constexpr int RG = HeadLane<D>::RG, UNR = HeadLane<D>::UNR;
  float am = 0.f;
  for (int r0 = L.rg; r0 < N; r0 += UNR * RG) {
    uint4 raw[UNR];
    L.load_rows(head, sN, N, r0, raw);
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (r0 + u * RG >= N) break;
      float x[8];
      unpack_bf16x8(raw[u], x);
#pragma unroll
      for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(MINUS ? __fsub_rn(x[e], mu[e]) : x[e]));
    }
  }
  return warp_max(am);
}

// The head's codes rint((x [- mu]) * inv) (and carriers) at codes + row * D.
template <int D, bool MINUS>
__device__ __forceinline__ void head_codes(const HeadLane<D>& L, const uint16_t* head, long long sN, int N,
                                           const float (&mu)[8], float inv, int8_t* codes,
                                           uint16_t* carrier) {
  constexpr int RG = HeadLane<D>::RG, UNR = HeadLane<D>::UNR;
  for (int r0 = L.rg; r0 < N; r0 += UNR * RG) {
    uint4 raw[UNR];
    L.load_rows(head, sN, N, r0, raw);
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u * RG;
      if (r >= N) break;
      float x[8];
      unpack_bf16x8(raw[u], x);
      if (MINUS) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __fsub_rn(x[e], mu[e]);
      }
      const size_t off = static_cast<size_t>(r) * D + L.v * 8;
      codes8(x, inv, codes + off, carrier ? carrier + off : nullptr);
    }
  }
}

// Per-channel max |V| over a head's rows, every lane of a column holding its 8.
template <int D>
__device__ __forceinline__ void head_vamax(const HeadLane<D>& L, const uint16_t* head, long long sN, int N,
                                           float (&vm)[8]) {
  constexpr int RG = HeadLane<D>::RG, UNR = HeadLane<D>::UNR;
#pragma unroll
  for (int e = 0; e < 8; ++e) vm[e] = 0.f;
  for (int r0 = L.rg; r0 < N; r0 += UNR * RG) {
    uint4 raw[UNR];
    L.load_rows(head, sN, N, r0, raw);  // zero rows leave a maximum of |x| unchanged
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      float x[8];
      unpack_bf16x8(raw[u], x);
#pragma unroll
      for (int e = 0; e < 8; ++e) vm[e] = fmaxf(vm[e], fabsf(x[e]));
    }
  }
#pragma unroll
  for (int o = HeadLane<D>::VPR; o < 32; o <<= 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) vm[e] = fmaxf(vm[e], __shfl_xor_sync(0xffffffffu, vm[e], o));
  }
}

// The head's V8^T rows [D][ldv] (keys past N are 0): e4m3(fp32(x * sc)) per
// channel, through the warp's [D][TL] byte tile.  Here a lane takes UNR
// consecutive rows (not rows RG apart), so its 8 codes of one channel are 8
// consecutive bytes of the tile: one 8-byte store per channel.
template <int D, int TL>
__device__ __forceinline__ void head_v8t(const HeadLane<D>& L, const uint16_t* head, long long sN, int N,
                                         const float (&sc)[8], uint8_t* tile, uint8_t* v8t_head,
                                         long long ldv, int lane) {
  for (int i = lane; i < D * TL / 16; i += 32) reinterpret_cast<uint4*>(tile)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncwarp();
  constexpr int RG = HeadLane<D>::RG, UNR = HeadLane<D>::UNR;
  static_assert(UNR == 8, "two words of codes per channel");
  for (int base = 0; base < N; base += UNR * RG) {
    const int r0 = base + L.rg * UNR;
    if (r0 >= N) continue;  // (rows past N stay the tile's zeros)
    uint32_t w[8][2] = {};  // channel e: the codes of rows r0 .. r0 + 3, r0 + 4 .. r0 + 7
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u;
      const uint4 raw = (r < N) ? *(reinterpret_cast<const uint4*>(head + static_cast<long long>(r) * sN) + L.v)
                                : make_uint4(0u, 0u, 0u, 0u);  // 0 codes
      float x[8];
      unpack_bf16x8(raw, x);
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const uint32_t b2 = cvt_e4m3x2(__fmul_rn(x[e], sc[e]), __fmul_rn(x[e + 1], sc[e + 1]));
        w[e][u / 4] |= (b2 & 0xFFu) << (8 * (u % 4));
        w[e + 1][u / 4] |= (b2 >> 8) << (8 * (u % 4));
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
      *reinterpret_cast<uint2*>(tile + (L.v * 8 + e) * TL + r0) = make_uint2(w[e][0], w[e][1]);
  }
  __syncwarp();
  const int nchunk = static_cast<int>(ldv / 16);  // 16-byte chunks of a V8^T row
  for (int i = lane; i < D * nchunk; i += 32) {
    const int c = i / nchunk, k = i % nchunk;
    const uint4 w = (16 * k < TL) ? *reinterpret_cast<const uint4*>(tile + c * TL + 16 * k)
                                  : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(v8t_head + static_cast<size_t>(c) * ldv + 16 * k) = w;
  }
}

// Block granules, heads of at most 128 tokens: everything in one launch.  Six
// CTAs per SM (80 registers, a few spilled) run faster than four at 126.
template <int D>
__global__ void __launch_bounds__(kSmallWarps * 32, 6) prepare_small_kernel(const SmallPrepArgs p) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) uint8_t tiles[kSmallWarps][D * kSmallHead];  // V8^T of a warp's head
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the heavier KV heads take the first warps, the Q heads fill the tail
  int item = blockIdx.x * kSmallWarps + warp;
  item = (item < p.BHk) ? item + p.BHq : item - p.BHk;
  const HeadLane<D> L(lane);
  const float none[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (item < p.BHq) {  // ---- a Q head: block amax, codes, scale
    const int bh = item;
    const uint16_t* src = src_head<uint16_t>(p.Q, bh);
    const float g = head_amax<D, false>(L, src, p.Q.sN, p.Nq, none);
    const float inv = (g > 0.f) ? __fdiv_rn(127.0f, g) : 0.f;
    head_codes<D, false>(L, src, p.Q.sN, p.Nq, none, inv, p.q_codes + static_cast<size_t>(bh) * p.Nq * D,
                         nullptr);
    if (lane == 0) p.q_scales[bh] = __fdiv_rn(g, 127.0f);
    return;
  }
  const int bh = item - p.BHq;
  if (bh >= p.BHk) return;
  // ---- a KV head: channel mean, K - mean codes, V maxima and e4m3 codes
  const uint16_t* ks = src_head<uint16_t>(p.K, bh);
  const uint16_t* vs = src_head<uint16_t>(p.V, bh);
  head_prefetch_l1<D>(L, vs, p.V.sN, p.Nk);  // V's reads overlap K's passes
  float mu[8];
  head_mean<D>(L, ks, p.K.sN, p.Nk, p.magic, mu);
  if (L.rg == 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) p.k_mean[static_cast<size_t>(bh) * D + L.v * 8 + e] = mu[e];
  }
  const float g = head_amax<D, true>(L, ks, p.K.sN, p.Nk, mu);
  const float inv = (g > 0.f) ? __fdiv_rn(127.0f, g) : 0.f;
  const size_t hoff = static_cast<size_t>(bh) * p.Nk * D;
  head_codes<D, true>(L, ks, p.K.sN, p.Nk, mu, inv, p.k_codes + hoff,
                      p.k_carrier ? p.k_carrier + hoff : nullptr);
  if (lane == 0) p.k_scales[bh] = __fdiv_rn(g, 127.0f);
  float vm[8], sc[8];
  head_vamax<D>(L, vs, p.V.sN, p.Nk, vm);
  {
    // The RG lanes of a column share the column's 16 divisions (lane rg takes
    // channels e = rg, rg + RG, ...) and hand the factors 448 / max round, as
    // head_mean does with its means.
    constexpr int RG = HeadLane<D>::RG, VPR = HeadLane<D>::VPR, PER = 8 / RG;
    float own[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = L.rg + i * RG;
      float ve = vm[0];
#pragma unroll
      for (int ee = 1; ee < 8; ++ee) ve = (ee == e) ? vm[ee] : ve;  // selects, no divergence
      own[i] = (ve > 0.f) ? __fdiv_rn(448.0f, ve) : 0.f;
      p.v_scales[static_cast<size_t>(bh) * D + L.v * 8 + e] = __fdiv_rn(ve, 448.0f);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sc[e] = __shfl_sync(0xffffffffu, own[e / RG], (e % RG) * VPR + L.v);
  }
  head_v8t<D, kSmallHead>(L, vs, p.V.sN, p.Nk, sc, tiles[warp], p.v8t + static_cast<size_t>(bh) * D * p.ldv, p.ldv,
                          lane);
}

// Tensor granules (one scale for all of Q, one for all of K - mean), KV heads
// of at most 256 tokens with d <= 64 (e.g. ViT's 197 tokens): the pre-pass in
// two launches instead of five, one CTA per head.  A CTA's 256 threads hold a
// whole head in registers -- thread (g, v) the 8 channels of 16-byte column v
// of rows g * UNR .. g * UNR + UNR - 1 (UNR consecutive rows) -- so each head
// is read once per launch.  Launch 1: a Q head's max |x|; a K head's channel
// mean and max |K - mean|; a V head's channel maxima, scales and transposed
// e4m3 codes.  The two maxima merge into two words (Q, K) with atomicMax on
// their bit patterns (non-negative floats order as unsigned integers; the
// words start at 0).  Launch 2: the Q and K codes at the two tensor scales
// (K's with the fp16 carriers).  Q heads of more than 256 rows are taken 256
// rows at a time.  The arithmetic is that of the bodies above, step by step.
constexpr int kTensorHead = 256;  // rows a CTA holds at once (and KV tokens at most)

template <int D>
struct TensorLane {
  static constexpr int VPR = D / 8;                // 16-byte vectors per row
  static constexpr int RG = kThreads / VPR;        // row groups (32 or 64)
  static constexpr int UNR = kTensorHead / RG;     // consecutive rows per thread (8 or 4)
  static constexpr int kWarps = kThreads / 32;
  int v, g;
  __device__ TensorLane() : v(threadIdx.x % VPR), g(threadIdx.x / VPR) {}
  __device__ int row(int base, int u) const { return base + g * UNR + u; }
  // the thread's rows of the 256-row chunk at `base` (zeros past N)
  __device__ void load(const uint16_t* head, long long sN, int N, int base, uint4 (&raw)[UNR]) const {
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = row(base, u);
      raw[u] = (r < N) ? __ldg(reinterpret_cast<const uint4*>(head + static_cast<long long>(r) * sN) + v)
                       : make_uint4(0u, 0u, 0u, 0u);
    }
  }
};

struct TensorPrepArgs {
  Src Q, K, V;
  int BHq, BHk, Nq, Nk;
  unsigned long long magic;
  int8_t* q_codes;
  float* q_scales;
  int8_t* k_codes;
  float* k_scales;
  uint16_t* k_carrier;
  float* k_mean;
  uint8_t* v8t;
  long long ldv;
  float* v_scales;
  unsigned int* amax;  // [2]: max |Q|, max |K - mean| (bit patterns)
};

template <int D>
struct TensorSmem {
  union {
    long long sums[kThreads / 32][D];  // K: the warps' channel sums
    float vmax[kThreads / 32][D];      // V: the warps' channel maxima
  };
  float chan[D];                       // K's mean or V's 448 / amax per channel
  float red[kThreads / 32];
  uint8_t tile[D * kTensorHead];       // V8^T of the head [D][256]
};

// max over the CTA of a per-thread value >= 0.
__device__ __forceinline__ float cta_max(float v, float* red) { return block_max(v, red); }

template <int D>
__global__ void __launch_bounds__(kThreads, 3) prepare_tensor1_kernel(const TensorPrepArgs p) {
  pdl_trigger();
  pdl_wait();
  using TL = TensorLane<D>;
  constexpr int UNR = TL::UNR, VPR = TL::VPR;
  __shared__ __align__(16) TensorSmem<D> sm;
  const TL L;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // the heavier K and V heads take the first CTAs, the Q heads (a max and
  // nothing else) fill the tail
  int item = blockIdx.x;
  item = (item < 2 * p.BHk) ? item + p.BHq : item - 2 * p.BHk;
  if (item < p.BHq) {  // ---- a Q head: its max |x|
    const uint16_t* src = src_head<uint16_t>(p.Q, item);
    float am = 0.f;
    for (int base = 0; base < p.Nq; base += kTensorHead) {
      uint4 raw[UNR];
      L.load(src, p.Q.sN, p.Nq, base, raw);  // zero rows leave the maximum unchanged
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        float x[8];
        unpack_bf16x8(raw[u], x);
#pragma unroll
        for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(x[e]));
      }
    }
    am = cta_max(am, sm.red);
    if (threadIdx.x == 0) atomicMax(p.amax, __float_as_uint(am));
    return;
  }
  item -= p.BHq;
  if (item < p.BHk) {  // ---- a K head: channel mean, then max |K - mean|
    const int bh = item;
    uint4 raw[UNR];
    L.load(src_head<uint16_t>(p.K, bh), p.K.sN, p.Nk, 0, raw);
    long long sum[8];
    fix24_column_sums<UNR>(raw, sum);  // rows past Nk are zeros: they add nothing
#pragma unroll
    for (int o = VPR; o < 32; o <<= 1) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sum[e] += __shfl_xor_sync(0xffffffffu, sum[e], o);
    }
    if (lane < VPR) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sm.sums[warp][lane * 8 + e] = sum[e];
    }
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += kThreads) {
      long long tot = 0;
#pragma unroll
      for (int w = 0; w < TL::kWarps; ++w) tot += sm.sums[w][c];
      const float mu = mean_of_fix24(tot, static_cast<uint32_t>(p.Nk), p.magic);
      sm.chan[c] = mu;
      p.k_mean[static_cast<size_t>(bh) * D + c] = mu;
    }
    __syncthreads();
    float mu[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) mu[e] = sm.chan[L.v * 8 + e];
    L.load(src_head<uint16_t>(p.K, bh), p.K.sN, p.Nk, 0, raw);  // again, from L1
    float am = 0.f;
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (L.row(0, u) < p.Nk) {
        float x[8];
        unpack_bf16x8(raw[u], x);
#pragma unroll
        for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(__fsub_rn(x[e], mu[e])));
      }
    }
    am = cta_max(am, sm.red);
    if (threadIdx.x == 0) atomicMax(p.amax + 1, __float_as_uint(am));
    return;
  }
  item -= p.BHk;
  if (item >= p.BHk) return;
  // ---- a V head: channel maxima, scales, e4m3 codes through the [D][256] tile
  const int bh = item;
  uint4 raw[UNR];
  L.load(src_head<uint16_t>(p.V, bh), p.V.sN, p.Nk, 0, raw);
  float vm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int u = 0; u < UNR; ++u) {  // zero rows leave the maxima unchanged
    float x[8];
    unpack_bf16x8(raw[u], x);
#pragma unroll
    for (int e = 0; e < 8; ++e) vm[e] = fmaxf(vm[e], fabsf(x[e]));
  }
#pragma unroll
  for (int o = VPR; o < 32; o <<= 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) vm[e] = fmaxf(vm[e], __shfl_xor_sync(0xffffffffu, vm[e], o));
  }
  if (lane < VPR) {
#pragma unroll
    for (int e = 0; e < 8; ++e) sm.vmax[warp][lane * 8 + e] = vm[e];
  }
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += kThreads) {
    float m = 0.f;
#pragma unroll
    for (int w = 0; w < TL::kWarps; ++w) m = fmaxf(m, sm.vmax[w][c]);
    sm.chan[c] = (m > 0.f) ? __fdiv_rn(448.0f, m) : 0.f;
    p.v_scales[static_cast<size_t>(bh) * D + c] = __fdiv_rn(m, 448.0f);
  }
  __syncthreads();
  float sc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) sc[e] = sm.chan[L.v * 8 + e];
  // the thread's UNR consecutive keys of each of its channels: UNR bytes of a
  // tile row (zero rows give code 0, the padding the layout wants)
#pragma unroll
  for (int q = 0; q < UNR / 4; ++q) {  // keys 4q .. 4q + 3 of the thread's rows: one word per channel
    uint32_t b[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
    for (int u = 4 * q; u < 4 * q + 4; ++u) {
      float x[8];
      unpack_bf16x8(raw[u], x);
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const uint32_t b2 = cvt_e4m3x2(__fmul_rn(x[e], sc[e]), __fmul_rn(x[e + 1], sc[e + 1]));
        b[e] |= (b2 & 0xFFu) << (8 * (u % 4));
        b[e + 1] |= (b2 >> 8) << (8 * (u % 4));
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
      *reinterpret_cast<uint32_t*>(sm.tile + (L.v * 8 + e) * kTensorHead + L.g * UNR + 4 * q) = b[e];
  }
  __syncthreads();
  const int nchunk = static_cast<int>(p.ldv / 16);  // 16-byte chunks of a V8^T row
  uint8_t* dst = p.v8t + static_cast<size_t>(bh) * D * p.ldv;
  for (int i = threadIdx.x; i < D * nchunk; i += kThreads) {
    const int c = i / nchunk, k = i % nchunk;
    const uint4 w = (16 * k < kTensorHead) ? *reinterpret_cast<const uint4*>(sm.tile + c * kTensorHead + 16 * k)
                                           : make_uint4(0u, 0u, 0u, 0u);
    if (QATTN_IN_BOUNDS(bh < p.BHk && 16 * k + 16 <= p.ldv))
      *reinterpret_cast<uint4*>(dst + static_cast<size_t>(c) * p.ldv + 16 * k) = w;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) prepare_tensor2_kernel(const TensorPrepArgs p) {
  pdl_trigger();
  pdl_wait();  // the maxima and K's mean of launch 1
  using TL = TensorLane<D>;
  constexpr int UNR = TL::UNR;
  const TL L;
  const bool is_q = blockIdx.x < p.BHq;
  const int bh = is_q ? blockIdx.x : blockIdx.x - p.BHq;
  if (!is_q && bh >= p.BHk) return;
  const Src& X = is_q ? p.Q : p.K;
  const int N = is_q ? p.Nq : p.Nk;
  float mu[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (!is_q) {
#pragma unroll
    for (int e = 0; e < 8; ++e) mu[e] = p.k_mean[static_cast<size_t>(bh) * D + L.v * 8 + e];
  }
  const float g = __uint_as_float(p.amax[is_q ? 0 : 1]);
  const float inv = (g > 0.f) ? __fdiv_rn(127.0f, g) : 0.f;
  const uint16_t* src = src_head<uint16_t>(X, bh);
  int8_t* codes = (is_q ? p.q_codes : p.k_codes) + static_cast<size_t>(bh) * N * D;
  uint16_t* carrier = (!is_q && p.k_carrier) ? p.k_carrier + static_cast<size_t>(bh) * N * D : nullptr;
  for (int base = 0; base < N; base += kTensorHead) {
    uint4 raw[UNR];
    L.load(src, X.sN, N, base, raw);
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = L.row(base, u);
      if (r >= N) break;
      float x[8];
      unpack_bf16x8(raw[u], x);
      if (!is_q) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __fsub_rn(x[e], mu[e]);
      }
      const size_t off = static_cast<size_t>(r) * D + L.v * 8;
      if (QATTN_IN_BOUNDS(r < N && L.v * 8 < D)) codes8(x, inv, codes + off, carrier ? carrier + off : nullptr);
    }
  }
  if (bh == 0 && threadIdx.x == 0) (is_q ? p.q_scales : p.k_scales)[0] = __fdiv_rn(g, 127.0f);
}

// The checked build's reporting path: the guard fails for threads >= n.
__global__ void bounds_probe_kernel(int n) { (void)QATTN_IN_BOUNDS(static_cast<int>(threadIdx.x) < n); }

// ------------------------------------------------------------------ carriers
// int8 codes -> fp16 values (exact: |code| <= 127).
__global__ void codes_to_f16_kernel(const int8_t* src, uint16_t* __restrict__ dst,
                                    size_t n16) {
  pdl_trigger();
  pdl_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 raw = reinterpret_cast<const uint4*>(src)[i];  // may come from the kernel before
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
  (void)Nk;
  // 64-bit channel sums, then one completion counter per (batch, head)
  return static_cast<size_t>(BH * d) * sizeof(unsigned long long) + static_cast<size_t>(BH) * 4;
}

template <int D>
static cudaError_t smooth_k_t(const Src& K, int BH, int Nk, long long* ws, float* mu,
                              cudaStream_t s) {
  constexpr int kWarpRows = kMeanRows * 32 / (D / 8);
  constexpr int kChunk = kMeanRows * kThreads / (D / 8);
  const unsigned long long magic = ~0ull / static_cast<unsigned long long>(Nk);
  if (Nk <= kWarpRows) {
    const int per = kThreads / 32;
    return launch_pdl(k_mean_warp_kernel<D>, dim3((BH + per - 1) / per), dim3(kThreads), 0, s, K, BH, Nk,
                      magic, mu);
  }
  const int nchunks = (Nk + kChunk - 1) / kChunk;
  const dim3 grid(nchunks, BH);
  if (nchunks == 1) {
    return launch_pdl(k_mean_kernel<D, false>, grid, dim3(kThreads), 0, s, K, Nk, 1, magic,
                      static_cast<unsigned long long*>(nullptr),
                      static_cast<unsigned int*>(nullptr), mu);
  }
  unsigned long long* acc = reinterpret_cast<unsigned long long*>(ws);
  unsigned int* done = reinterpret_cast<unsigned int*>(acc + static_cast<size_t>(BH) * D);
  const cudaError_t e = cudaMemsetAsync(ws, 0, smooth_k_ws_bytes(BH, Nk, D), s);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_mean_kernel<D, true>, grid, dim3(kThreads), 0, s, K, Nk, nchunks, magic, acc,
                    done, mu);
}

cudaError_t launch_smooth_k(const Src& K, int BH, int Nk, int d, long long* ws, float* mu,
                            cudaStream_t s) {
  if (Nk == 0) return cudaMemsetAsync(mu, 0, static_cast<size_t>(BH) * d * sizeof(float), s);
  if (d == 32) return smooth_k_t<32>(K, BH, Nk, ws, mu, s);
  if (d == 64) return smooth_k_t<64>(K, BH, Nk, ws, mu, s);
  return smooth_k_t<128>(K, BH, Nk, ws, mu, s);
}

// Scratch: K channel sums and done counters, V channel maxima.
size_t prepare_ws_bytes(long long BH, long long d) {
  auto a256 = [](size_t x) { return (x + 255) / 256 * 256; };
  return a256(smooth_k_ws_bytes(BH, 0, d)) + a256(static_cast<size_t>(BH * d) * sizeof(unsigned int));
}

template <int D>
static cudaError_t prepare_t(const Prep1Args& p1, const Prep2Args& p2, cudaStream_t s) {
  const int g1 = p1.jq.BH * p1.jq.nblk + (p1.nkc + p1.nvc) * p1.BHk;
  cudaError_t e = launch_pdl(prepare1_kernel<D>, dim3(g1), dim3(kThreads), 0, s, p1);
  if (e != cudaSuccess) return e;
  const int g2 = p2.jk.BH * p2.jk.nblk + p2.nvt * p1.BHk;
  return launch_pdl(prepare2_kernel<D>, dim3(g2), dim3(kThreads), 0, s, p2);
}

int prepare_launch_count(int d, int Nq, int Nk) {
  return (d <= 64 && Nq <= kSmallHead && Nk <= kSmallHead) ? 1 : 2;
}

cudaError_t launch_prepare(const RowsJob& jq, const RowsJob& jk, const Src& V, int d,
                           uint8_t* v8t, long long ldv, float* v_scales, void* ws, cudaStream_t s) {
  const int BHk = jk.BH, Nk = jk.N;
  if (BHk <= 0 || Nk <= 0) return cudaErrorInvalidValue;
  if (jq.gran != 2 || jk.gran != 2) return cudaErrorInvalidValue;
  if (prepare_launch_count(d, jq.N, Nk) == 1) {  // short heads: one warp each, one launch
    SmallPrepArgs p{};
    p.Q = Src{jq.X, jq.sB, jq.sH, jq.sN, jq.H};
    p.K = Src{jk.X, jk.sB, jk.sH, jk.sN, jk.H};
    p.V = V;
    p.BHq = jq.BH;
    p.BHk = BHk;
    p.Nq = jq.N;
    p.Nk = Nk;
    p.magic = ~0ull / static_cast<unsigned long long>(Nk);
    p.q_codes = jq.codes;
    p.q_scales = jq.scales;
    p.k_codes = jk.codes;
    p.k_scales = jk.scales;
    p.k_carrier = jk.carrier;
    p.k_mean = const_cast<float*>(jk.chan);
    p.v8t = v8t;
    p.ldv = ldv;
    p.v_scales = v_scales;
    const dim3 grid((jq.BH + BHk + kSmallWarps - 1) / kSmallWarps);
    if (d == 32) return launch_pdl(prepare_small_kernel<32>, grid, dim3(kSmallWarps * 32), 0, s, p);
    return launch_pdl(prepare_small_kernel<64>, grid, dim3(kSmallWarps * 32), 0, s, p);
  }
  const size_t wsm = (smooth_k_ws_bytes(BHk, Nk, d) + 255) / 256 * 256;
  cudaError_t e = cudaMemsetAsync(ws, 0, prepare_ws_bytes(BHk, d), s);
  if (e != cudaSuccess) return e;
  Prep1Args p1{};
  p1.jq = jq;
  p1.K = Src{jk.X, jk.sB, jk.sH, jk.sN, jk.H};
  p1.V = V;
  p1.BHk = BHk;
  p1.Nk = Nk;
  p1.nkc = (Nk + kMeanRows * kThreads / (d / 8) - 1) / (kMeanRows * kThreads / (d / 8));
  p1.nvc = (Nk + kTokPerChunk - 1) / kTokPerChunk;
  p1.magic = ~0ull / static_cast<unsigned long long>(Nk);
  p1.acc = static_cast<unsigned long long*>(ws);
  p1.done = reinterpret_cast<unsigned int*>(p1.acc + static_cast<size_t>(BHk) * d);
  p1.mu = const_cast<float*>(jk.chan);
  p1.amax = reinterpret_cast<unsigned int*>(static_cast<char*>(ws) + wsm);
  Prep2Args p2{};
  p2.jk = jk;
  p2.V = V;
  p2.Nk = Nk;
  p2.nvt = static_cast<int>((ldv + 127) / 128);
  p2.amax = p1.amax;
  p2.v8t = v8t;
  p2.ldv = ldv;
  p2.v_scales = v_scales;
  switch (d) {
    case 32: return prepare_t<32>(p1, p2, s);
    case 64: return prepare_t<64>(p1, p2, s);
    default: return prepare_t<128>(p1, p2, s);
  }
}

unsigned int check_take_quant() { return check_take_local(); }

cudaError_t launch_bounds_probe(cudaStream_t s) {
  bounds_probe_kernel<<<1, 32, 0, s>>>(16);
  return cudaGetLastError();
}

bool prepare_tensor_eligible(int d, int Nq, int Nk) {
  (void)Nq;
  return (d == 32 || d == 64) && Nk >= 1 && Nk <= kTensorHead;
}

cudaError_t launch_prepare_tensor(const RowsJob& jq, const RowsJob& jk, const Src& V, int d,
                                  uint8_t* v8t, long long ldv, float* v_scales, void* ws,
                                  cudaStream_t s) {
  if (!prepare_tensor_eligible(d, jq.N, jk.N) || jq.gran != 0 || jk.gran != 0)
    return cudaErrorInvalidValue;
  TensorPrepArgs p{};
  p.Q = Src{jq.X, jq.sB, jq.sH, jq.sN, jq.H};
  p.K = Src{jk.X, jk.sB, jk.sH, jk.sN, jk.H};
  p.V = V;
  p.BHq = jq.BH;
  p.BHk = jk.BH;
  p.Nq = jq.N;
  p.Nk = jk.N;
  p.magic = ~0ull / static_cast<unsigned long long>(jk.N);
  p.q_codes = jq.codes;
  p.q_scales = jq.scales;
  p.k_codes = jk.codes;
  p.k_scales = jk.scales;
  p.k_carrier = jk.carrier;
  p.k_mean = const_cast<float*>(jk.chan);
  p.v8t = v8t;
  p.ldv = ldv;
  p.v_scales = v_scales;
  p.amax = static_cast<unsigned int*>(ws);
  cudaError_t e = cudaMemsetAsync(ws, 0, 2 * sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  const dim3 g1(jq.BH + 2 * jk.BH), g2(jq.BH + jk.BH);  // one CTA per Q, K, V head
  if (d == 32) {
    e = launch_pdl(prepare_tensor1_kernel<32>, g1, dim3(kThreads), 0, s, p);
    if (e != cudaSuccess) return e;
    return launch_pdl(prepare_tensor2_kernel<32>, g2, dim3(kThreads), 0, s, p);
  }
  e = launch_pdl(prepare_tensor1_kernel<64>, g1, dim3(kThreads), 0, s, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(prepare_tensor2_kernel<64>, g2, dim3(kThreads), 0, s, p);
}

size_t quantize_rows_ws_bytes(long long B, long long H, long long N, int gran) {
  if (gran == 2) return 0;
  return static_cast<size_t>(B * H * ((N + 127) / 128)) * sizeof(float);
}

template <int D>
static cudaError_t quant_rows_dispatch(dim3 grid, cudaStream_t s, const RowsJob& j0, int m0,
                                       const RowsJob& j1, int m1, int pass) {
  if (m0 == 0 && m1 == 1)
    return launch_pdl(quant_rows_kernel<D, 0, 1>, grid, dim3(kThreads), 0, s, j0, j1, pass);
  if (m0 == 0) return launch_pdl(quant_rows_kernel<D, 0, 0>, grid, dim3(kThreads), 0, s, j0, j1, pass);
  return launch_pdl(quant_rows_kernel<D, 2, 0>, grid, dim3(kThreads), 0, s, j0, j1, pass);
}

cudaError_t launch_quantize_rows(const RowsJob& j0, int m0, const RowsJob& j1, int m1, int d,
                                 cudaStream_t s) {
  if (!((m0 == 0 && (m1 == 0 || m1 == 1)) || (m0 == 2 && j1.BH == 0))) return cudaErrorInvalidValue;
  const int nblk = max(j0.nblk, j1.BH > 0 ? j1.nblk : 0);
  const int nx = j0.BH + j1.BH;
  if (nblk <= 0 || nx <= 0) return cudaSuccess;
  const dim3 grid(nx, nblk);
  const bool two_pass = (j0.BH > 0 && j0.gran != 2) || (j1.BH > 0 && j1.gran != 2);
  for (int pass = two_pass ? 0 : 1; pass < 2; ++pass) {
    cudaError_t e;
    switch (d) {
      case 32: e = quant_rows_dispatch<32>(grid, s, j0, m0, j1, m1, pass); break;
      case 64: e = quant_rows_dispatch<64>(grid, s, j0, m0, j1, m1, pass); break;
      default: e = quant_rows_dispatch<128>(grid, s, j0, m0, j1, m1, pass);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D, bool I8>
static cudaError_t quantize_v_impl(const Src& V, const float* chan, int BH, int Nk,
                                   uint8_t* v8t, long long ldv, float* v_scales, unsigned int* ws,
                                   cudaStream_t s) {
  const int nchunks = (Nk + kTokPerChunk - 1) / kTokPerChunk;
  cudaError_t e = launch_pdl(v_amax_kernel<D, I8>, dim3(nchunks, BH), dim3(kThreads), 0, s, V, Nk, ws);
  if (e != cudaSuccess) return e;
  const int nt = static_cast<int>((ldv + 127) / 128);
  return launch_pdl(v_convert_kernel<D, I8>, dim3(nt, BH), dim3(kThreads), 0, s, V, Nk,
                    static_cast<const unsigned int*>(ws), chan, v8t, ldv, v_scales);
}

cudaError_t launch_quantize_v(const Src& V, int is_i8, const float* chan, int BH, int Nk, int d,
                              uint8_t* v8t, long long ldv, float* v_scales, unsigned int* ws_amax,
                              cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(ws_amax, 0, static_cast<size_t>(BH) * d * sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  if (Nk == 0) return cudaMemsetAsync(v_scales, 0, static_cast<size_t>(BH) * d * sizeof(float), s);
#define QATTN_QV(DD)                                                                  \
  return is_i8 ? quantize_v_impl<DD, true>(V, chan, BH, Nk, v8t, ldv, v_scales, ws_amax, s) \
               : quantize_v_impl<DD, false>(V, chan, BH, Nk, v8t, ldv, v_scales, ws_amax, s);
  switch (d) {
    case 32: QATTN_QV(32)
    case 64: QATTN_QV(64)
    default: QATTN_QV(128)
  }
#undef QATTN_QV
}

// The int8 cache header's per-channel max |V code| over rows 0 .. Nk-1 of
// each (batch, KV head) slice of `rows` cached rows: the amax kernel of the
// int8 V path, writing the maxima straight into `out` (non-negative floats
// order like their bit patterns, so the kernel's integer atomic max applies).
cudaError_t launch_v_code_amax(const int8_t* v_codes, int BH, int Nk, long long rows, int d,
                               float* out, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(out, 0, static_cast<size_t>(BH) * d * sizeof(float), s);
  if (e != cudaSuccess || Nk == 0 || BH == 0) return e;
  const dim3 grid((Nk + kTokPerChunk - 1) / kTokPerChunk, BH);
  unsigned int* bits = reinterpret_cast<unsigned int*>(out);
  const Src v = dense_src(v_codes, 1, rows, d);  // (batch, head) slices of `rows` rows
  switch (d) {
    case 32: return launch_pdl(v_amax_kernel<32, true>, grid, dim3(kThreads), 0, s, v, Nk, bits);
    case 64: return launch_pdl(v_amax_kernel<64, true>, grid, dim3(kThreads), 0, s, v, Nk, bits);
    default: return launch_pdl(v_amax_kernel<128, true>, grid, dim3(kThreads), 0, s, v, Nk, bits);
  }
}

cudaError_t launch_codes_to_f16(const int8_t* src, uint16_t* dst, size_t n, cudaStream_t s) {
  const size_t n16 = n / 16;
  if (n16 == 0) return cudaSuccess;
  return launch_pdl(codes_to_f16_kernel, dim3(grid_for(n16, 256)), dim3(256), 0, s, src, dst, n16);
}

// ------------------------------------------------------------------ rows with no keys
__global__ void fill_u32_kernel(uint32_t* __restrict__ dst, size_t n, uint32_t v) {
  pdl_trigger();
  pdl_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    dst[i] = v;
}

cudaError_t launch_no_key_rows(void* out, size_t out_bytes, float* lse, size_t rows, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(out, 0, out_bytes, s);
  if (e != cudaSuccess || lse == nullptr || rows == 0) return e;
  return launch_pdl(fill_u32_kernel, dim3(grid_for(rows, 256)), dim3(256), 0, s,
                    reinterpret_cast<uint32_t*>(lse), rows, 0xFF800000u);  // -inf
}

}  // namespace qattn
