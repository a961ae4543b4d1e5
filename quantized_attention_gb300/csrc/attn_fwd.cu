// Fused quantized attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// One CTA owns one 128-row query tile of one (batch, head).  Warp roles:
//   warps 0-3 (128 threads, one query row each, TMEM lanes 0-127): read the
//     score tile from TMEM, scale and mask it, keep the running row max and
//     row sum in fp32, write P * 448 as e4m3 to shared memory, rescale the
//     TMEM output accumulator when the max grows, and run the epilogue.
//   warp 4: allocates TMEM; its lane 0 issues every TMA load and every MMA.
//
// Per key block j (128 keys):
//   S  = Q . K_j^T     tcgen05.mma kind::f16  (int8 codes held exactly in fp16,
//                      fp32 accumulation: every partial sum is an integer of
//                      magnitude <= d * 127^2 < 2^21, so the result is exact)
//   P8 = e4m3(448 * 2^(t - m))                 (softmax warps)
//   O += P8 . V8_j     tcgen05.mma kind::f8f6f4 (e4m3 x e4m3 -> fp32 in TMEM)
// The MMA thread issues PV_{j-1} before QK_j, so the commit that signals
// "S_j ready" also certifies that PV_{j-1} has finished with O and with the
// P buffer: the softmax warps may rescale O and overwrite P without another
// barrier.  Two CTAs share an SM, so one CTA's softmax overlaps the other's
// MMAs.
#include <cuda_bf16.h>

#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kBM = 128;  // query rows per tile (MMA M)
constexpr int kBN = 128;  // keys per block
constexpr int kThreads = 160;
constexpr float kLog2e = 1.44269502162933349609375f;   // fp32(log2 e)
constexpr float kLog2_448 = 8.8073549220576041f;       // log2(448)
constexpr float kLn2 = 0.69314718055994531f;

// Shared-memory plan for head dim D.  Q/K are fp16 carriers stored as
// column blocks of [128 rows][row_bytes] in the TMA/UMMA swizzled K-major
// layout (128-byte rows with the 128B swizzle, 64-byte rows with the 64B
// swizzle for D = 32).  V is e4m3 transposed, [D rows][128 keys]; P is e4m3
// [128 rows][128 keys]; both use 128-byte rows with the 128B swizzle.
template <int D>
struct Cfg {
  static constexpr int kColBlock = (D >= 64) ? 64 : D;  // fp16 elements per row of a block
  static constexpr int kRowBytes = kColBlock * 2;
  static constexpr int kNumColBlocks = D / kColBlock;
  static constexpr int kColBlockBytes = kBM * kRowBytes;
  static constexpr uint32_t kSwz = (kRowBytes == 128) ? kSwizzle128B : kSwizzle64B;
  static constexpr uint32_t kSBO = 8 * kRowBytes;  // bytes between 8-row groups
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kKBytes = kBN * D * 2;
  static constexpr int kVBytes = D * kBN;
  static constexpr int kPBytes = kBM * kBN;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kKBytes;
  static constexpr int kOffP = kOffV + kVBytes;
  static constexpr int kOffBar = kOffP + kPBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + barriers + alignment slack
  static constexpr uint32_t kTmemCols = 256;               // S: [0,128)  O: [128, 128+D)
  static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0, "tile alignment");
};

// S = Q . K^T for one 128 x 128 tile: D/16 MMAs of K = 16, fp32 into TMEM.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tmem_s, uint32_t sq, uint32_t sk) {
  using C = Cfg<D>;
  constexpr uint32_t idesc = make_idesc(kBM, kBN, 0, 0);  // F16 x F16 -> F32
  constexpr int kStepsPerBlock = C::kRowBytes / 32;       // 32 bytes = 16 fp16 per step
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    const uint32_t off = (s / kStepsPerBlock) * C::kColBlockBytes + (s % kStepsPerBlock) * 32;
    mma_f16(tmem_s, smem_desc(sq + off, C::kSBO, C::kSwz), smem_desc(sk + off, C::kSBO, C::kSwz),
            idesc, s > 0 ? 1u : 0u);
  }
}

// O (+)= P8 . V8 for one key block: 4 MMAs of K = 32 e4m3.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t sp, uint32_t sv, bool acc) {
  constexpr uint32_t idesc = make_idesc(kBM, D, 0, 0);  // E4M3 x E4M3 -> F32
#pragma unroll
  for (int s = 0; s < kBN / 32; ++s) {
    mma_f8(tmem_o, smem_desc(sp + s * 32, 1024, kSwizzle128B),
           smem_desc(sv + s * 32, 1024, kSwizzle128B), idesc, (acc || s > 0) ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void tma_tile(const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                         int row, int plane) {
  using C = Cfg<D>;
#pragma unroll
  for (int cb = 0; cb < C::kNumColBlocks; ++cb)
    tma_load_3d(dst + cb * C::kColBlockBytes, map, bar, cb * C::kColBlock, row, plane);
}

__device__ __forceinline__ float scale_of(const float* s, int gran, int bh, int nblk, int blk) {
  if (gran == 0) return __ldg(s);
  if (gran == 1) return __ldg(s + bh);
  return __ldg(s + static_cast<size_t>(bh) * nblk + blk);
}

enum Bar { kQFull = 0, kKFull, kVFull, kSFull, kPFull, kKEmpty, kVEmpty, kOFull, kDrain, kNumBars };

template <int D, bool BIAS>
__global__ void __launch_bounds__(kThreads, 2)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + C::kOffQ, sK = base + C::kOffK, sV = base + C::kOffV;
  const uint32_t sP = base + C::kOffP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 8 * kNumBars + 4);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, b = blockIdx.y;
  const int n_qt = (a.Nq + kBM - 1) / kBM;
  const int qt = n_qt - 1 - static_cast<int>(blockIdx.z);  // heaviest causal tiles first
  const int q0 = qt * kBM;
  const int hkv = h / (a.Hq / a.Hkv);
  const int bq = b * a.Hq + h, bkv = b * a.Hkv + hkv;

  int kend = a.Nk;  // one past the last key any row of this tile can see
  if (a.causal) {
    const long long last = static_cast<long long>(a.pos0) + min(q0 + kBM - 1, a.Nq - 1);
    kend = static_cast<int>(max(0LL, min(static_cast<long long>(a.Nk), last + 1)));
  }
  const int nb = (kend + kBN - 1) / kBN;

  if (nb == 0) {  // every row of the tile sees no key: output 0, lse -inf
    if (threadIdx.x < kBM) {
      const int qi = q0 + threadIdx.x;
      if (qi < a.Nq) {
        const size_t row = static_cast<size_t>(bq) * a.Nq + qi;
        for (int c = 0; c < D; ++c) {
          if (a.out_bf16) reinterpret_cast<__nv_bfloat16*>(a.out)[row * D + c] = __float2bfloat16(0.f);
          else reinterpret_cast<float*>(a.out)[row * D + c] = 0.f;
        }
        if (a.lse) a.lse[row] = -INFINITY;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    const uint32_t counts[kNumBars] = {1, 1, 1, 1, kBM, 1, 1, 1, 1};
    for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), counts[i]);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;

  if (warp == 4) {
    if (lane == 0) {
      // ------------------------------------------------ TMA + MMA issue
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int pend_k = -1, pend_v = -1;  // loads issued but not yet observed complete
      mbar_arrive_expect_tx(bar(kQFull), C::kQBytes);
      tma_tile<D>(&tmQ, sQ, bar(kQFull), q0, bq);
      mbar_arrive_expect_tx(bar(kKFull), C::kKBytes);
      tma_tile<D>(&tmK, sK, bar(kKFull), 0, bkv);
      pend_k = 0;
      mbar_arrive_expect_tx(bar(kVFull), C::kVBytes);
      tma_load_3d(sV, &tmV, bar(kVFull), 0, 0, bkv);
      pend_v = 0;
      bool ok = mbar_wait(bar(kQFull), 0, abort_flag, a.err, kErrTimeout);
      for (int j = 0; ok && j < nb; ++j) {
        if (!(ok = mbar_wait(bar(kKFull), j & 1, abort_flag, a.err, kErrTimeout))) break;
        pend_k = -1;
        if (j > 0) {
          if (!(ok = mbar_wait(bar(kPFull), (j - 1) & 1, abort_flag, a.err, kErrTimeout))) break;
          if (!(ok = mbar_wait(bar(kVFull), (j - 1) & 1, abort_flag, a.err, kErrTimeout))) break;
          pend_v = -1;
          tc_fence_after();
          issue_pv<D>(tO, sP, sV, j - 1 > 0);
          mma_commit(bar(kVEmpty));
        }
        tc_fence_after();
        issue_qk<D>(tS, sQ, sK);
        mma_commit(bar(kSFull));
        mma_commit(bar(kKEmpty));
        if (j + 1 < nb) {
          if (!(ok = mbar_wait(bar(kKEmpty), j & 1, abort_flag, a.err, kErrTimeout))) break;
          mbar_arrive_expect_tx(bar(kKFull), C::kKBytes);
          tma_tile<D>(&tmK, sK, bar(kKFull), (j + 1) * kBN, bkv);
          pend_k = (j + 1) & 1;
        }
        if (j > 0) {
          if (!(ok = mbar_wait(bar(kVEmpty), (j - 1) & 1, abort_flag, a.err, kErrTimeout))) break;
          mbar_arrive_expect_tx(bar(kVFull), C::kVBytes);
          tma_load_3d(sV, &tmV, bar(kVFull), j * kBN, 0, bkv);
          pend_v = j & 1;
        }
      }
      if (ok) {
        ok = mbar_wait(bar(kPFull), (nb - 1) & 1, abort_flag, a.err, kErrTimeout) &&
             mbar_wait(bar(kVFull), (nb - 1) & 1, abort_flag, a.err, kErrTimeout);
        if (ok) {
          pend_v = -1;
          tc_fence_after();
          issue_pv<D>(tO, sP, sV, nb - 1 > 0);
          mma_commit(bar(kOFull));
        }
      }
      // Let every MMA this thread issued finish before TMEM can be freed, and
      // let any TMA load still in flight land, each with a bounded wait.
      mma_commit(bar(kDrain));
      volatile int never = 0;
      mbar_wait(bar(kDrain), 0, &never, a.err, kErrTimeout);
      if (pend_k >= 0) mbar_wait(bar(kKFull), pend_k, &never, a.err, kErrTimeout);
      if (pend_v >= 0) mbar_wait(bar(kVFull), pend_v, &never, a.err, kErrTimeout);
      if (!ok) *abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warpgroup
    const int r = threadIdx.x;  // row within the tile == TMEM lane
    const int qi = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int nqb = (a.Nq + kBM - 1) / kBM, nkb = (a.Nk + kBN - 1) / kBN;
    const float sq = scale_of(a.q_scales, a.q_gran, bq, nqb, qt);
    const long long lim = static_cast<long long>(a.pos0) + qi;  // last visible key (causal)
    const float* brow = nullptr;
    if (BIAS) brow = a.bias + static_cast<size_t>(h) * a.bias_head_stride + static_cast<size_t>(min(qi, a.Nq - 1)) * a.Nk;
    const uint32_t prow = sP + r * 128;
    const uint32_t sw = r & 7;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      ok = mbar_wait(bar(kSFull), j & 1, abort_flag, a.err, kErrTimeout);
      if (!__all_sync(0xffffffffu, ok)) {  // keep the warp converged for tcgen05.ld
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s[kBN];
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i)
        tmem_ld32(tS + lane_base + i * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[i * 32]));
      tmem_wait_ld();
      const float sk = scale_of(a.k_scales, a.k_gran, bkv, nkb, j);
      const float c = __fmul_rn(__fmul_rn(__fmul_rn(sq, sk), a.sm_scale), kLog2e);
      const int kbase = j * kBN;
      long long lastk = static_cast<long long>(a.Nk) - 1;
      if (a.causal && lim < lastk) lastk = lim;
      const int nvis = static_cast<int>(max(0LL, min(static_cast<long long>(kBN), lastk - kbase + 1)));
      float m_blk = -INFINITY;
      if (!BIAS) {
        float mx = -INFINITY;
        if (nvis == kBN) {
#pragma unroll
          for (int k = 0; k < kBN; ++k) mx = fmaxf(mx, __uint_as_float(s[k]));
        } else {
#pragma unroll
          for (int k = 0; k < kBN; ++k)
            if (k < nvis) mx = fmaxf(mx, __uint_as_float(s[k]));
        }
        m_blk = (mx == -INFINITY) ? -INFINITY : __fmul_rn(mx, c);
      } else {
#pragma unroll
        for (int k = 0; k < kBN; ++k) {
          float t = -INFINITY;
          if (k < nvis) t = fmaf(__uint_as_float(s[k]), c, __fmul_rn(__ldg(brow + kbase + k), kLog2e));
          s[k] = __float_as_uint(t);
          m_blk = fmaxf(m_blk, t);
        }
      }
      const float m_new = fmaxf(m, m_blk);
      const bool dead = (m_new == -INFINITY);
      const float alpha = dead ? 1.f : ex2_approx(m - m_new);
      const float kneg = dead ? 0.f : (kLog2_448 - m_new);
      float sum = 0.f;
#pragma unroll
      for (int ch = 0; ch < kBN / 16; ++ch) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float p[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = ch * 16 + q * 4 + e;
            float x;
            if (!BIAS) x = fmaf(__uint_as_float(s[k]), c, kneg);
            else x = __uint_as_float(s[k]) + kneg;
            if (k >= nvis) x = -INFINITY;
            p[e] = ex2_approx(x);
            sum += p[e];
          }
          w[q] = cvt_e4m3x2(p[0], p[1]) | (cvt_e4m3x2(p[2], p[3]) << 16);
        }
        const uint32_t addr = prow + ((static_cast<uint32_t>(ch) ^ sw) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3])
                     : "memory");
      }
      l = fmaf(alpha, l, sum);
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + lane_base + cc * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + lane_base + cc * 32, o);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kPFull));
      m = m_new;
    }
    if (ok) ok = mbar_wait(bar(kOFull), 0, abort_flag, a.err, kErrTimeout);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const float* sv = a.v_scales + static_cast<size_t>(bkv) * D;
      const size_t row = static_cast<size_t>(bq) * a.Nq + qi;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + lane_base + cc * 32, o);
        tmem_wait_ld();
        if (qi < a.Nq) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(o[i]) * (__ldg(sv + cc * 32 + i) * inv_l);
          if (a.out_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + row * D + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 pr = __floats2bfloat162_rn(v[8 * i + 2 * e], v[8 * i + 2 * e + 1]);
                w[e] = *reinterpret_cast<const uint32_t*>(&pr);
              }
              dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + row * D + cc * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        }
      }
      if (a.lse && qi < a.Nq)
        a.lse[row] = (l > 0.f) ? (m + __log2f(l) - kLog2_448) * kLn2 : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Debug: the int32 score tile of one (q tile, k tile) through issue_qk.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    qk_debug_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    int Hq, int Hkv, int Nq, int Nk, int32_t* __restrict__ S, unsigned int* err) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + C::kOffQ, sK = base + C::kOffK;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 36);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x, qt = blockIdx.y, bq = blockIdx.z;
  const int b = bq / Hq, h = bq % Hq;
  const int bkv = b * Hkv + h / (Hq / Hkv);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    mbar_init(smem_u32(&bars[2]), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 4) {
    if (lane == 0) {
      const uint32_t full = smem_u32(&bars[0]);
      mbar_arrive_expect_tx(full, C::kQBytes + C::kKBytes);
      tma_tile<D>(&tmQ, sQ, full, qt * kBM, bq);
      tma_tile<D>(&tmK, sK, full, kt * kBN, bkv);
      volatile int never = 0;
      if (mbar_wait(full, 0, &never, err, kErrTimeout)) {
        tc_fence_after();
        issue_qk<D>(tmem, sQ, sK);
        mma_commit(smem_u32(&bars[1]));
        mma_commit(smem_u32(&bars[2]));
        mbar_wait(smem_u32(&bars[2]), 0, &never, err, kErrTimeout);
      } else {
        *abort_flag = 1;
      }
    }
    __syncwarp();
  } else {
    const int r = threadIdx.x;
    const bool ok = mbar_wait(smem_u32(&bars[1]), 0, abort_flag, err, kErrTimeout);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      uint32_t s[kBN];
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i)
        tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + i * 32,
                  *reinterpret_cast<uint32_t(*)[32]>(&s[i * 32]));
      tmem_wait_ld();
      const int qi = qt * kBM + r;
      if (qi < Nq) {
        int32_t* dst = S + (static_cast<size_t>(bq) * Nq + qi) * Nk + kt * kBN;
        const int ncol = min(kBN, Nk - kt * kBN);
#pragma unroll
        for (int k = 0; k < kBN; ++k)
          if (k < ncol) dst[k] = __float2int_rn(__uint_as_float(s[k]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

template <int D, bool BIAS>
cudaError_t launch_attn_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const AttnArgs& a, cudaStream_t s) {
  const int smem = Cfg<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, BIAS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.Hq, a.B, (a.Nq + kBM - 1) / kBM);
  attn_fwd_kernel<D, BIAS><<<grid, kThreads, smem, s>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dbg_t(const CUtensorMap& tq, const CUtensorMap& tk, int B, int Hq, int Hkv,
                         int Nq, int Nk, int32_t* S, unsigned int* err, cudaStream_t s) {
  const int smem = Cfg<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(qk_debug_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((Nk + kBN - 1) / kBN, (Nq + kBM - 1) / kBM, B * Hq);
  qk_debug_kernel<D><<<grid, kThreads, smem, s>>>(tq, tk, Hq, Hkv, Nq, Nk, S, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const AttnArgs& a, cudaStream_t s) {
  const bool bias = a.bias != nullptr;
  switch (a.d) {
    case 32: return bias ? launch_attn_t<32, true>(tq, tk, tv, a, s) : launch_attn_t<32, false>(tq, tk, tv, a, s);
    case 64: return bias ? launch_attn_t<64, true>(tq, tk, tv, a, s) : launch_attn_t<64, false>(tq, tk, tv, a, s);
    default: return bias ? launch_attn_t<128, true>(tq, tk, tv, a, s) : launch_attn_t<128, false>(tq, tk, tv, a, s);
  }
}

cudaError_t launch_qk_debug(const CUtensorMap& tq, const CUtensorMap& tk, int B, int Hq, int Hkv,
                            int Nq, int Nk, int d, int32_t* S, unsigned int* err,
                            cudaStream_t s) {
  switch (d) {
    case 32: return launch_dbg_t<32>(tq, tk, B, Hq, Hkv, Nq, Nk, S, err, s);
    case 64: return launch_dbg_t<64>(tq, tk, B, Hq, Hkv, Nq, Nk, S, err, s);
    default: return launch_dbg_t<128>(tq, tk, B, Hq, Hkv, Nq, Nk, S, err, s);
  }
}

}  // namespace qattn
