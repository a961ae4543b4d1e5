// High-accuracy attention on an int8 KV cache with operands split exact to 24
// bits (Strata PR "prompt_attn_i8v3_kernel", "What it does", "Operands": q
// scaled per (head, 64-dim group) and p per (row, chunk) to 127, then
// X = rint(x * 65536) = h * 65536 + l * 256 + m, three exact products with
// the stored int8 codes combined in fp32; "Measured": ~2e-6 max relative error
// against FP64).
//
// The exact products run on the 5th-generation tensor cores as fp16 x fp16
// with fp32 accumulation in TMEM (tcgen05.mma kind::f16; there is no int8
// kind on this part): h, l, m and the int8 codes are exact fp16 values, and a
// part's sum over 64 channels (or 64 keys) is an integer below
// 64 * 255 * 128 < 2^24, so no rounding occurs whatever the summation order.
// The K and V channel scales of the cache are factored out: K's is folded
// into q before the split, V's applied to the output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qattn_check.cuh"
#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kGroup = 64;   // q scale granule: 64 channels of a head
constexpr float kLog2e = 1.44269502162933349609375f;  // fp32(log2 e)
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kNegInf = -__builtin_huge_valf();

// x (fp32, |x| <= 127) -> X = rint(x * 65536) = h * 65536 + l * 256 + m with h,
// l signed and m unsigned bytes, returned as exact fp16 values.
__device__ __forceinline__ void split24(float x, __half& h, __half& l, __half& m) {
  const int X = __float2int_rn(__fmul_rn(x, 65536.0f));
  const int mm = X & 255;
  const int r = (X - mm) >> 8;
  const int ll = ((r + 128) & 255) - 128;
  const int hh = (r - ll) >> 8;
  h = __int2half_rn(hh);
  l = __int2half_rn(ll);
  m = __int2half_rn(mm);
}

// The same split for X = rint(y) given y = x * 65536 >= 0 (P's side), in fp32
// arithmetic only: every value below 2^24 is an exact integer, so floor, the
// products by 2^-8 and the differences are exact.  Returns (h, l, m) as floats.
__device__ __forceinline__ void split24_pos(float y, float& h, float& l, float& m) {
  const float X = rintf(y);
  const float r = floorf(X * 0.00390625f);           // X >> 8
  m = fmaf(-256.0f, r, X);                           // X & 255
  h = floorf((r + 128.0f) * 0.00390625f);            // so that l is a signed byte
  l = fmaf(-256.0f, h, r);
}

__device__ __forceinline__ uint32_t pack_f2h2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);  // exact: small integers
  return *reinterpret_cast<const uint32_t*>(&v);
}

// ---------------------------------------------------------------- q split
// One CTA per (batch, query head): s_g = fp32(max |q * s_k| / 127) over the
// head's rows and the 64 channels of group g, then every q' = fp32(q * s_k)
// becomes x = fp32(q' / s_g) and its three fp16 parts, stored [3][B*Hq][Nq][D].
template <int D>
__global__ void __launch_bounds__(256) q_split_kernel(const uint16_t* Q, const float* k_chan_scale,
                                                      int Hq, int Hkv, int Nq, __half* parts,
                                                      float* group_scale, size_t plane) {
  constexpr int NG = D / kGroup;
  __shared__ float red[256 / 32][NG];
  __shared__ float sg[NG];
  pdl_trigger();
  pdl_wait();
  const int bh = blockIdx.x, b = bh / Hq, h = bh % Hq;
  const float* sk = k_chan_scale + (static_cast<size_t>(b) * Hkv + h / (Hq / Hkv)) * D;
  const uint16_t* q = Q + static_cast<size_t>(bh) * Nq * D;
  const int c = threadIdx.x % D;  // each thread stays on one channel
  const float s = __ldg(sk + c);
  float amax = 0.f;
  for (size_t i = threadIdx.x; i < static_cast<size_t>(Nq) * D; i += 256)
    amax = fmaxf(amax, fabsf(__fmul_rn(bf16_bits_to_f32(q[i]), s)));
  // threads of a warp share one group (32 consecutive channels of the same 64)
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int g = 0; g < NG; ++g) red[warp][g] = (c / kGroup == g) ? amax : 0.f;
  }
  __syncthreads();
  if (threadIdx.x < NG) {
    float m = 0.f;
    for (int w = 0; w < 256 / 32; ++w) m = fmaxf(m, red[w][threadIdx.x]);
    sg[threadIdx.x] = __fdiv_rn(m, 127.0f);
    group_scale[static_cast<size_t>(bh) * NG + threadIdx.x] = sg[threadIdx.x];
  }
  __syncthreads();
  const float sgc = sg[c / kGroup];
  __half* ph = parts + static_cast<size_t>(bh) * Nq * D;
  for (size_t i = threadIdx.x; i < static_cast<size_t>(Nq) * D; i += 256) {
    const float qp = __fmul_rn(bf16_bits_to_f32(q[i]), s);
    const float x = (sgc > 0.f) ? __fdiv_rn(qp, sgc) : 0.f;
    __half hh, ll, mm;
    split24(x, hh, ll, mm);
    ph[i] = hh;
    ph[plane + i] = ll;
    ph[2 * plane + i] = mm;
  }
}

// ---------------------------------------------------------------- cache rows as fp16
// K codes [bkv][cap][D] -> exact fp16 rows [bkv][Nk][D] (the QK B operand).
__global__ void k_rows_f16_kernel(const int8_t* __restrict__ codes, long long cap, int Nk, int D,
                                  long long n16, uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int per_row = D / 16;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = i / per_row;  // bkv * Nk + key
    const int c16 = static_cast<int>(i % per_row);
    const long long bkv = row / Nk, key = row % Nk;
    if (!QATTN_IN_BOUNDS(key < cap)) continue;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(codes + (bkv * cap + key) * D) + c16);
    uint32_t h[8];
    codes4_to_f16x2(x.x, h[0], h[1]);
    codes4_to_f16x2(x.y, h[2], h[3]);
    codes4_to_f16x2(x.z, h[4], h[5]);
    codes4_to_f16x2(x.w, h[6], h[7]);
    uint4* d = reinterpret_cast<uint4*>(out + row * D) + 2 * c16;
    d[0] = make_uint4(h[0], h[1], h[2], h[3]);
    d[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// V codes [bkv][cap][D] -> exact fp16, transposed: [bkv][D][ldt] (key index
// fastest; keys Nk .. ldt-1 are 0), the PV B operand.  One CTA per (64 keys,
// bkv) through a [64][D] fp16 tile.
template <int D>
__global__ void __launch_bounds__(256) v_t_f16_kernel(const int8_t* __restrict__ codes, long long cap,
                                                      int Nk, long long ldt, uint16_t* __restrict__ out) {
  __shared__ uint16_t tile[64][D + 8];
  pdl_trigger();
  pdl_wait();
  const int k0 = blockIdx.x * 64, bkv = blockIdx.y;
  for (int i = threadIdx.x; i < 64 * D / 16; i += 256) {
    const int key = i / (D / 16), c16 = i % (D / 16);
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (k0 + key < Nk && QATTN_IN_BOUNDS(k0 + key < cap))
      x = __ldg(reinterpret_cast<const uint4*>(codes + (static_cast<long long>(bkv) * cap + k0 + key) * D) + c16);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 16; ++e)
      tile[key][16 * c16 + e] =
          __half_as_ushort(__int2half_rn(static_cast<int8_t>((w[e / 4] >> (8 * (e % 4))) & 0xFFu)));
  }
  __syncthreads();
  // channel c, keys k0 .. k0 + 63: 8 chunks of 8 fp16 (16 bytes), those past ldt skipped
  for (int i = threadIdx.x; i < D * 8; i += 256) {
    const int c = i / 8, q = i % 8;
    if (k0 + 8 * q >= ldt) continue;
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      h[e] = static_cast<uint32_t>(tile[8 * q + 2 * e][c]) | (static_cast<uint32_t>(tile[8 * q + 2 * e + 1][c]) << 16);
    *reinterpret_cast<uint4*>(out + (static_cast<long long>(bkv) * D + c) * ldt + k0 + 8 * q) =
        make_uint4(h[0], h[1], h[2], h[3]);
  }
}

// ---------------------------------------------------------------- attention
// One CTA per 128 query rows of one (batch, query head), on tcgen05:
//   warp 0   lane 0 issues the TMA loads: the tile's three q parts (once), a
//            ring of 64-key K chunks (fp16) and of V^T chunks (fp16);
//   warp 1   owns TMEM; lane 0 issues the MMAs;
//   warps 4-7 one query row per thread (row r = TMEM lane r).
// Per 64-key chunk j the MMA thread issues, per 64-channel group g and part p,
// the exact partial S_gp = q_part_p[:, g] . K_g^T (4 kind::f16 MMAs of
// 128 x 64 x 16, fp32 in TMEM: an integer below 2^24) into a ring of kNS
// 64-column slots; the row threads drain the partials in the oracle's order,
// S = sum_g sum_p (s_g 2^-8p) S_gp (fp32 multiply-adds), run the online
// softmax, split P per (row, chunk) into three exact fp16 parts in shared
// memory, and the MMA thread issues, per part, OP_p = P_p . V (4 MMAs of
// 128 x D x 16 into a ring of kNOP D-column slots), which the threads fold
// into their O registers: O = alpha O + sum_p (s_p 2^-8p) OP_p.  Issue order
// QK(j+1)'s first kNS partials before PV(j) overlaps the tensor work with the
// softmax; the rest after PV(j), whose operand P(j) depends on every partial
// of chunk j (issuing them earlier could wait on a slot only drained after
// PV(j)).
constexpr int kBM = 128;
constexpr int kCK = 64;   // keys per chunk (P scale granule, online-softmax block)
constexpr int kNS = 3;    // S partial slots (64 TMEM columns each)
constexpr int kNOP = 2;   // OP slots (D TMEM columns each)
constexpr int kTcThreads = 384;

template <int D>
struct TcCfg {
  static constexpr int NG = D / kGroup;                  // channel groups = 128-byte column blocks
  static constexpr int kNK = (D == 128) ? 2 : 4;          // K ring stages
  static constexpr int kNV = (D == 128) ? 2 : 4;          // V^T ring stages
  static constexpr int kQPart = NG * kBM * 128;           // one q part: NG blocks of [128][128 B]
  static constexpr int kKBytes = NG * kCK * 128;          // a K chunk: NG blocks of [64][128 B]
  static constexpr int kVBytes = D * 128;                 // a V^T chunk: [D][64 keys fp16]
  static constexpr int kPPart = kBM * 128;                // one P part: [128][64 keys fp16]
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 3 * kQPart;
  static constexpr int kOffV = kOffK + kNK * kKBytes;
  static constexpr int kOffP = kOffV + kNV * kVBytes;
  static constexpr int kOffBar = kOffP + 3 * kPPart;
  static constexpr int kSmemBytes = kOffBar + 256 + 4 * kBM * 4 + 1024;  // + barriers, row exchange, slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

enum {
  kTbQFull = 0,
  kTbKFull = 1,     // [4]
  kTbKEmpty = 5,    // [4]
  kTbVFull = 9,     // [4]
  kTbVEmpty = 13,   // [4]
  kTbSFull = 17,    // [3]
  kTbSFree = 20,    // [3]  128 row threads
  kTbPFull = 23,    //      128 row threads
  kTbOpFull = 24,   // [2]
  kTbOpFree = 26,   // [2]  128 row threads
  kTbXFull = 28,    // [2]  both halves of every row posted (256 row threads)
  kTbDrain = 30,
  kTbNum = 31
};
static_assert(8 * kTbNum + 8 <= 256, "barrier area (then the TMEM slot and the abort flag)");

struct Ex24TcArgs {
  int Hq, Hkv, Nq, Nk;
  int causal;
  int pos0;
  float cfac;  // fp32(sm_scale * log2 e)
  const float* group_scale;
  const float* v_chan_scale;
  void* out;
  int out_bf16;
  float* lse;
  unsigned int* err;
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    exact24_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const Ex24TcArgs a) {
  using C = TcCfg<D>;
  constexpr int NG = C::NG;
  constexpr int NPS = 3 * NG;  // partials per chunk
  extern __shared__ uint8_t smem_raw[];
  pdl_trigger();
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 8 * kTbNum);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 8 * kTbNum + 4);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto sQ = [&](int p, int g) { return base + C::kOffQ + p * C::kQPart + g * kBM * 128; };
  auto sK = [&](int st, int g) { return base + C::kOffK + st * C::kKBytes + g * kCK * 128; };
  auto sV = [&](int st) { return base + C::kOffV + st * C::kVBytes; };
  auto sP = [&](int p) { return base + C::kOffP + p * C::kPPart; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y, b = bh / a.Hq, h = bh % a.Hq;
  const int bkv = b * a.Hkv + h / (a.Hq / a.Hkv);
  const int q0 = blockIdx.x * kBM;
  const int last_row = min(q0 + kBM, a.Nq) - 1;
  const int kend = a.causal ? min(a.Nk, a.pos0 + last_row + 1) : a.Nk;
  const int nc = (kend + kCK - 1) / kCK;  // chunks; >= 1 (every row sees key 0)

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTbNum; ++i) {
      const bool rows = (i >= kTbSFree && i < kTbSFree + kNS) || i == kTbPFull ||
                        (i >= kTbOpFree && i < kTbOpFree + kNOP) || (i >= kTbXFull && i < kTbXFull + 2);
      mbar_init(bar(i), rows ? 2 * kBM : 1);  // both threads of every row
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the q parts, scales and fp16 cache rows of the kernels before

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(bar(kTbQFull), 3 * C::kQPart);
      for (int p = 0; p < 3; ++p)
        for (int g = 0; g < NG; ++g)
          tma_load_3d(sQ(p, g), &tmQ, bar(kTbQFull), g * kGroup, q0, p * static_cast<int>(gridDim.y) + bh);
      bool ok = true;
      int last_k[4] = {-1, -1, -1, -1}, last_v[4] = {-1, -1, -1, -1};
      for (int j = 0; ok && j < nc; ++j) {
        const int sk = j % C::kNK, sv = j % C::kNV;
        if (j >= C::kNK &&
            !(ok = mbar_wait(bar(kTbKEmpty + sk), ((j / C::kNK) - 1) & 1, abort_flag, a.err, kErrTimeout)))
          break;
        mbar_arrive_expect_tx(bar(kTbKFull + sk), C::kKBytes);
        for (int g = 0; g < NG; ++g) tma_load_3d(sK(sk, g), &tmK, bar(kTbKFull + sk), g * kGroup, j * kCK, bkv);
        last_k[sk] = j;
        if (j >= C::kNV &&
            !(ok = mbar_wait(bar(kTbVEmpty + sv), ((j / C::kNV) - 1) & 1, abort_flag, a.err, kErrTimeout)))
          break;
        mbar_arrive_expect_tx(bar(kTbVFull + sv), C::kVBytes);
        tma_load_3d(sV(sv), &tmV, bar(kTbVFull + sv), j * kCK, 0, bkv);
        last_v[sv] = j;
      }
      // every load this thread issued lands before the CTA may exit
      volatile int never = 0;
      mbar_wait(bar(kTbQFull), 0, &never, a.err, kErrTimeout);
      for (int st = 0; st < 4; ++st) {
        if (st < C::kNK && last_k[st] >= 0)
          mbar_wait(bar(kTbKFull + st), (last_k[st] / C::kNK) & 1, &never, a.err, kErrTimeout);
        if (st < C::kNV && last_v[st] >= 0)
          mbar_wait(bar(kTbVFull + st), (last_v[st] / C::kNV) & 1, &never, a.err, kErrTimeout);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA
      constexpr uint32_t idesc_qk = make_idesc(kBM, kCK, 0, 0);  // F16 x F16 -> F32, N = 64
      constexpr uint32_t idesc_pv = make_idesc(kBM, D, 0, 0);
      uint32_t sp = 0, op = 0;  // S partials / OP parts issued
      bool ok = mbar_wait(bar(kTbQFull), 0, abort_flag, a.err, kErrTimeout);
      // QK partials [from, to) of chunk j
      auto qk = [&](int j, int from, int to) -> bool {
        const int sk = j % C::kNK;
        if (from == 0 && !mbar_wait(bar(kTbKFull + sk), (j / C::kNK) & 1, abort_flag, a.err, kErrTimeout))
          return false;
        for (int u = from; u < to; ++u) {
          const int slot = sp % kNS;
          if (sp >= static_cast<uint32_t>(kNS) &&
              !mbar_wait(bar(kTbSFree + slot), ((sp / kNS) - 1) & 1, abort_flag, a.err, kErrTimeout))
            return false;
          tc_fence_after();
          const int g = u / 3, p = u % 3;
#pragma unroll
          for (int k = 0; k < kGroup / 16; ++k)
            mma_f16(tmem + 64 * slot, smem_desc(sQ(p, g) + 32 * k, 1024, kSwizzle128B),
                    smem_desc(sK(sk, g) + 32 * k, 1024, kSwizzle128B), idesc_qk, k > 0 ? 1u : 0u);
          mma_commit(bar(kTbSFull + slot));
          ++sp;
        }
        if (to == NPS) mma_commit(bar(kTbKEmpty + sk));
        return true;
      };
      auto pv = [&](int j) -> bool {
        const int sv = j % C::kNV;
        if (!mbar_wait(bar(kTbVFull + sv), (j / C::kNV) & 1, abort_flag, a.err, kErrTimeout) ||
            !mbar_wait(bar(kTbPFull), j & 1, abort_flag, a.err, kErrTimeout))
          return false;
        for (int p = 0; p < 3; ++p) {
          const int slot = op % kNOP;
          if (op >= static_cast<uint32_t>(kNOP) &&
              !mbar_wait(bar(kTbOpFree + slot), ((op / kNOP) - 1) & 1, abort_flag, a.err, kErrTimeout))
            return false;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kCK / 16; ++k)
            mma_f16(tmem + 64 * kNS + D * slot, smem_desc(sP(p) + 32 * k, 1024, kSwizzle128B),
                    smem_desc(sV(sv) + 32 * k, 1024, kSwizzle128B), idesc_pv, k > 0 ? 1u : 0u);
          mma_commit(bar(kTbOpFull + slot));
          ++op;
        }
        mma_commit(bar(kTbVEmpty + sv));
        return true;
      };
      constexpr int kAhead = (kNS < NPS) ? kNS : NPS;
      if (ok) ok = qk(0, 0, NPS);
      for (int j = 0; ok && j < nc; ++j) {
        if (j + 1 < nc && !(ok = qk(j + 1, 0, kAhead))) break;
        if (!(ok = pv(j))) break;
        if (j + 1 < nc && kAhead < NPS && !(ok = qk(j + 1, kAhead, NPS))) break;
      }
      mma_commit(bar(kTbDrain));
      volatile int never = 0;
      mbar_wait(bar(kTbDrain), 0, &never, a.err, kErrTimeout);
      if (!ok) *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ rows
    // Two threads per row: warps 4-7 take keys 0-31 of each chunk and O's
    // first D/2 columns, warps 8-11 keys 32-63 and the last D/2 columns.
    const int hf = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // TMEM lane and tile row
    const int row = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t prow = r * 128, sw = r & 7;
    constexpr int DH = D / 2;
    // [2 buffers][2 halves][128 rows]: the halves' row maxima (and, at the end,
    // row sums), exchanged through kTbXFull; buffer j & 1 is written again only
    // after every thread passed chunk j + 1's exchange, so after its reads
    float* xch = reinterpret_cast<float*>(smem + C::kOffBar + 256);
    auto exchange = [&](int n, float v, float& other) -> bool {
      const int xb = n & 1;
      xch[(xb * 2 + hf) * kBM + r] = v;
      mbar_arrive(bar(kTbXFull + xb));
      const bool okx = mbar_wait(bar(kTbXFull + xb), (n >> 1) & 1, abort_flag, a.err, kErrTimeout);
      if (!__all_sync(0xffffffffu, okx)) return false;
      other = xch[(xb * 2 + 1 - hf) * kBM + r];
      return true;
    };
    float gsc[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) gsc[g] = a.group_scale[static_cast<size_t>(bh) * NG + g];
    const int lim = a.causal ? min(a.Nk - 1, a.pos0 + row) : a.Nk - 1;  // last visible key
    float m = kNegInf, l = 0.f;  // l: this thread's share of the row sum
    float o[DH];
#pragma unroll
    for (int c = 0; c < DH; ++c) o[c] = 0.f;
    uint32_t sp = 0, op = 0;
    bool ok = true;
    for (int j = 0; j < nc; ++j) {
      const int kb = j * kCK + 32 * hf;  // this thread's first key of the chunk
      // ---- S = sum over groups and parts of (s_g 2^-8p) S_gp, in the oracle's order
      float S[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) S[k] = 0.f;
#pragma unroll
      for (int u = 0; u < NPS; ++u) {
        const int slot = sp % kNS;
        ok = mbar_wait(bar(kTbSFull + slot), (sp / kNS) & 1, abort_flag, a.err, kErrTimeout);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + 64 * slot + 32 * hf, v);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(kTbSFree + slot));
        ++sp;
        const int g = u / 3, p = u % 3;
        const float wgt = gsc[g] * ((p == 0) ? 1.f : (p == 1) ? (1.f / 256.f) : (1.f / 65536.f));
#pragma unroll
        for (int k = 0; k < 32; ++k) S[k] = fmaf(wgt, __uint_as_float(v[k]), S[k]);
      }
      if (!ok) break;
      // ---- t, mask, the row maximum (both halves), online softmax
      float mx = kNegInf;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const bool vis = row < a.Nq && kb + k <= lim;
        S[k] = vis ? __fmul_rn(S[k], a.cfac) : kNegInf;
        mx = fmaxf(mx, S[k]);
      }
      float mx_other;
      if (!(ok = exchange(j, mx, mx_other))) break;
      mx = fmaxf(mx, mx_other);
      const float mn = fmaxf(m, mx);
      const float al = (m == kNegInf) ? 0.f : ex2_approx(m - mn);
      const float ref = (mn == kNegInf) ? 0.f : mn;
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        S[k] = ex2_approx(S[k] - ref);
        sum += S[k];
      }
      l = al * l + sum;
      m = mn;
      // P's chunk maximum -> s_p = pmax / 127; x * 65536 = P * (65536 / s_p)
      const float pm = (mx == kNegInf) ? 0.f : ex2_approx(mx - ref);
      const float spc = __fdiv_rn(pm, 127.0f);
      const float ci = (spc > 0.f) ? __fdiv_rn(65536.0f, spc) : 0.f;
      // ---- the three parts of P, as fp16 rows of the three P tiles (128B swizzle)
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 16-byte chunk 4 hf + c: keys 8c .. 8c + 7 of this half
        uint32_t w[3][4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float ha, la, ma, hb, lb, mb;
          split24_pos(S[8 * c + 2 * e] * ci, ha, la, ma);
          split24_pos(S[8 * c + 2 * e + 1] * ci, hb, lb, mb);
          w[0][e] = pack_f2h2(ha, hb);
          w[1][e] = pack_f2h2(la, lb);
          w[2][e] = pack_f2h2(ma, mb);
        }
        const uint32_t off = prow + ((static_cast<uint32_t>(4 * hf + c) ^ sw) << 4);
#pragma unroll
        for (int p = 0; p < 3; ++p) st_shared_v4(sP(p) + off, w[p][0], w[p][1], w[p][2], w[p][3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kTbPFull));
      // ---- O = alpha O + sum_p (s_p 2^-8p) OP_p (this thread's D/2 columns)
#pragma unroll
      for (int c = 0; c < DH; ++c) o[c] *= al;
#pragma unroll
      for (int p = 0; p < 3; ++p) {
        const int slot = op % kNOP;
        ok = mbar_wait(bar(kTbOpFull + slot), (op / kNOP) & 1, abort_flag, a.err, kErrTimeout);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float w = spc * ((p == 0) ? 1.f : (p == 1) ? (1.f / 256.f) : (1.f / 65536.f));
#pragma unroll
        for (int cc = 0; cc < DH / 32; ++cc) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + 64 * kNS + D * slot + DH * hf + 32 * cc, v);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[32 * cc + k] = fmaf(w, __uint_as_float(v[k]), o[32 * cc + k]);
        }
        tc_fence_before();
        mbar_arrive(bar(kTbOpFree + slot));
        ++op;
      }
      if (!ok) break;
    }
    // the row sum: both halves' shares
    if (ok) {
      float l_other;
      if ((ok = exchange(nc, l, l_other))) l += l_other;
    }
    if (ok && row < a.Nq && QATTN_IN_BOUNDS(bh < static_cast<int>(gridDim.y))) {
      // ---- epilogue: O * s_v / l
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const float* svc = a.v_chan_scale + static_cast<size_t>(bkv) * D + DH * hf;
      const size_t idx = (static_cast<size_t>(bh) * a.Nq + row) * D + DH * hf;
#pragma unroll
      for (int c = 0; c < DH; c += 8) {
        float val[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) val[e] = o[c + e] * __ldg(svc + c + e) * inv;
        if (a.out_bf16) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 pr = __floats2bfloat162_rn(val[2 * e], val[2 * e + 1]);
            wv[e] = *reinterpret_cast<const uint32_t*>(&pr);
          }
          *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + idx + c) =
              make_uint4(wv[0], wv[1], wv[2], wv[3]);
        } else {
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + idx + c);
          dst[0] = make_float4(val[0], val[1], val[2], val[3]);
          dst[1] = make_float4(val[4], val[5], val[6], val[7]);
        }
      }
      if (a.lse && hf == 0)
        a.lse[static_cast<size_t>(bh) * a.Nq + row] = (l > 0.f) ? (m + __log2f(l)) * kLn2 : kNegInf;
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Workspace: the q parts [3][B*Hq][Nq][D] fp16, the group scales, K as fp16
// rows [B*Hkv][Nk][D], V^T as fp16 [B*Hkv][D][ldt].
struct Ex24Ws {
  size_t plane, off_gsc, off_k, off_v, total;
  long long ldt;
};
Ex24Ws ex24_ws(long long B, long long Hq, long long Hkv, long long Nq, long long Nk, long long d) {
  auto a256 = [](size_t x) { return (x + 255) / 256 * 256; };
  Ex24Ws w;
  w.plane = static_cast<size_t>(B * Hq * Nq * d);
  w.ldt = (Nk + 7) / 8 * 8;
  w.off_gsc = a256(3 * w.plane * 2);
  w.off_k = w.off_gsc + a256(static_cast<size_t>(B * Hq * (d / kGroup)) * 4);
  w.off_v = w.off_k + a256(static_cast<size_t>(B * Hkv * Nk * d) * 2);
  w.total = w.off_v + a256(static_cast<size_t>(B * Hkv * d * w.ldt) * 2);
  return w;
}

template <int D>
cudaError_t launch_t(const Exact24Args& x, cudaStream_t s) {
  const Ex24Ws w = ex24_ws(x.B, x.Hq, x.Hkv, x.Nq, x.Nk, D);
  char* ws = static_cast<char*>(x.ws);
  __half* parts = reinterpret_cast<__half*>(ws);
  float* gsc = reinterpret_cast<float*>(ws + w.off_gsc);
  uint16_t* k16 = reinterpret_cast<uint16_t*>(ws + w.off_k);
  uint16_t* vt16 = reinterpret_cast<uint16_t*>(ws + w.off_v);
  const int BHq = x.B * x.Hq, BHk = x.B * x.Hkv;
  CUtensorMap tq, tk, tv;
  if (!encode_tiled_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, parts, D, x.Nq, 3ull * BHq, D * 2, kGroup, kBM,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, k16, D, x.Nk, BHk, D * 2, kGroup, kCK,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, vt16, x.Nk, D, BHk, w.ldt * 2, kCK, D,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(q_split_kernel<D>, dim3(BHq), dim3(256), 0, s, static_cast<const uint16_t*>(x.Q),
                             x.k_chan_scale, x.Hq, x.Hkv, x.Nq, parts, gsc, w.plane);
  if (e != cudaSuccess) return e;
  const long long n16 = static_cast<long long>(BHk) * x.Nk * (D / 16);
  const int g16 = static_cast<int>(min(static_cast<long long>(num_sms()) * 8, (n16 + 255) / 256));
  e = launch_pdl(k_rows_f16_kernel, dim3(g16), dim3(256), 0, s, x.k_codes, x.cap, x.Nk, D, n16, k16);
  if (e != cudaSuccess) return e;
  e = launch_pdl(v_t_f16_kernel<D>, dim3((x.Nk + 63) / 64, BHk), dim3(256), 0, s, x.v_codes, x.cap, x.Nk,
                 w.ldt, vt16);
  if (e != cudaSuccess) return e;
  Ex24TcArgs a{};
  a.Hq = x.Hq;
  a.Hkv = x.Hkv;
  a.Nq = x.Nq;
  a.Nk = x.Nk;
  a.causal = x.causal;
  a.pos0 = x.pos0;
  a.cfac = x.sm_scale * kLog2e;  // one fp32 multiply, round to nearest
  a.group_scale = gsc;
  a.v_chan_scale = x.v_chan_scale;
  a.out = x.out;
  a.out_bf16 = x.out_bf16;
  a.lse = x.lse;
  a.err = x.err;
  constexpr int smem = TcCfg<D>::kSmemBytes;
  e = cudaFuncSetAttribute(exact24_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(exact24_tc_kernel<D>, dim3((x.Nq + kBM - 1) / kBM, BHq), dim3(kTcThreads), smem, s, tq,
                    tk, tv, a);
}

}  // namespace

unsigned int check_take_exact24() { return check_take_local(); }

size_t exact24_ws_bytes(long long B, long long Hq, long long Hkv, long long Nq, long long Nk,
                        long long d) {
  return ex24_ws(B, Hq, Hkv, Nq, Nk, d).total;
}

cudaError_t launch_exact24(const Exact24Args& x, cudaStream_t s) {
  return x.d == 64 ? launch_t<64>(x, s) : launch_t<128>(x, s);
}

}  // namespace qattn
