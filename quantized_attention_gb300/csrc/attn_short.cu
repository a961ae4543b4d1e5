// Attention for short key sequences (the ViT/DeiT and Swin-window shapes of
// "QFlash", Table 1: N = 197 or 49, d = 64 or 32, no causal mask): the same
// recipe as attn_fwd_kernel -- exact integer scores of the int8 codes, the fp32
// online softmax over 128-key blocks (P = 2^(t - m) <= 1, rescale whenever the
// row max grows), P8 = e4m3(448 P), O = alpha O + P8 . V8, out = O s_v / l --
// on the warp-level tensor cores.
//
// K codes and V8^T are converted once to exact fp16 in shared memory (int8
// codes and e4m3 values are fp16 values); QK^T and PV run on mma.m16n8k16 fp16
// with fp32 accumulation: the scores' partial sums are integers below 2^24
// (exact), and a P8 x V8 product is exact in fp32, as on the e4m3 tensor path.
// S stays in registers; the accumulator layout of two 8-key n-tiles is the A
// layout of one 16-key PV step, so P8 goes from registers straight into the PV
// product.  The expressions for c, t, m, alpha, P, l and the epilogue are those
// of the persistent kernel.
//
// Two kernels share that block step:
//   attn_window_kernel  Nq, Nk <= 64 (Swin windows): 4 warps cover a head's
//                       rows; each CTA loops over heads with the next head's
//                       raw codes loaded into registers under the current
//                       head's math (one 64-key block, S in 32 registers).
//   attn_short_kernel   Nk <= 256: 16 * W rows of one head per CTA, W <= 8
//                       warps sized to Nq, 128-key blocks in turn.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qattn_check.cuh"
#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kBlk = 128;      // keys per softmax block (the recipe's block)
constexpr int kMaxWarps = 8;   // 16 query rows per warp
constexpr int kWin = kWindowMax;  // rows and keys of the window kernel
constexpr int kWinThreads = 128;
constexpr float kLog2e = 1.44269502162933349609375f;  // fp32(log2 e)
constexpr float kLog2_448 = 8.8073549220576041f;      // log2(448)
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kNegInf = -__builtin_huge_valf();

struct ShortArgs {
  AttnArgs a;
  const int8_t* q_codes;
  const int8_t* k_codes;
  const uint8_t* v8t;
  long long ldv;
};

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ float scale_of(const float* s, int gran, int bh, int nblk, int blk) {
  if (gran == 0) return s[0];
  if (gran == 1) return s[bh];
  return s[static_cast<size_t>(bh) * nblk + blk];
}

// Sixteen int8 codes -> sixteen exact fp16 values at dst (32 bytes).
__device__ __forceinline__ void store_codes16_f16(uint8_t* dst, const uint4& x) {
  uint32_t hv[8];
  codes4_to_f16x2(x.x, hv[0], hv[1]);
  codes4_to_f16x2(x.y, hv[2], hv[3]);
  codes4_to_f16x2(x.z, hv[4], hv[5]);
  codes4_to_f16x2(x.w, hv[6], hv[7]);
  *reinterpret_cast<uint4*>(dst) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
  *reinterpret_cast<uint4*>(dst + 16) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
}

// Sixteen e4m3 bytes -> sixteen exact fp16 values at dst (32 bytes).
__device__ __forceinline__ void store_e4m3x16_f16(uint8_t* dst, const uint4& x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t hv[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    hv[2 * e] = e4m3x2_to_f16x2(w[e] & 0xFFFFu);
    hv[2 * e + 1] = e4m3x2_to_f16x2(w[e] >> 16);
  }
  *reinterpret_cast<uint4*>(dst) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
  *reinterpret_cast<uint4*>(dst + 16) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
}

// A lane's two rows (g and g + 8 of its warp's 16): running max and sum.
struct RowPair {
  float m_lo = kNegInf, m_hi = kNegInf, l_lo = 0.f, l_hi = 0.f;
};

// One key block of KB keys (nvis of them visible, from kbase) for a warp's 16
// rows: S from the fp16 Q rows (q_addr) and K rows (k_addr, pitch 2D + 16),
// the masked, scaled scores, the running max and alpha, O *= alpha, 448 P, its
// e4m3 codes and O += P8 . V8 (v_addr: V^T rows, pitch 2 KB + 16), and l.
// FRAG (with BIAS): the bias comes from bfrag, the lane's S-fragment-ordered
// values bias * log2 e (-inf past nvis) in shared memory, one float4 per
// 8-key n-tile at bfrag[32 n], instead of the rows.  FIRST: the row's first
// block (rp fresh, o zero), where O *= alpha and alpha l change nothing.
template <int D, bool BIAS, int KB, bool FRAG = false, bool FIRST = false>
__device__ __forceinline__ void block_step(uint32_t q_addr, uint32_t k_addr, uint32_t v_addr, int nvis,
                                           int kbase, float c_lo, float c_hi, const float* brow_lo,
                                           const float* brow_hi, int t4, RowPair& rp,
                                           float (&o)[D / 8][4], const float4* bfrag = nullptr) {
  constexpr int KS = D / 16;
  constexpr int NTO = D / 8;
  constexpr int kQKPitch = 2 * D + 16;
  constexpr int kVPitch = 2 * KB + 16;
  const int nstep = (nvis + 15) / 16;  // 16-key steps holding a visible key
  float S[KB / 8][4];
#pragma unroll
  for (int n = 0; n < KB / 8; ++n) S[n][0] = S[n][1] = S[n][2] = S[n][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(q_addr + ks * 32, a0, a1, a2, a3);
#pragma unroll
    for (int s = 0; s < KB / 16; ++s) {
      if (s < nstep) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(k_addr + 16 * s * kQKPitch + ks * 32, b0, b1, b2, b3);
        mma_f16_16816(S[2 * s], a0, a1, a2, a3, b0, b1);
        mma_f16_16816(S[2 * s + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
  if (!BIAS) {  // masked keys are -inf scores; c stays > 0 so -inf * c = -inf
    c_lo = fmaxf(c_lo, 0x1p-126f);
    c_hi = fmaxf(c_hi, 0x1p-126f);
  }
  float mx_lo = kNegInf, mx_hi = kNegInf;
#pragma unroll
  for (int n = 0; n < KB / 8; ++n) {
    float4 bf;
    if (FRAG) bf = bfrag[32 * n];  // n-tile n's entry of the lane (the lanes' entries interleave)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = 8 * n + 2 * t4 + (e & 1);
      float v = S[n][e];
      if (FRAG) {
        v = fmaf(v, (e < 2) ? c_lo : c_hi, e == 0 ? bf.x : e == 1 ? bf.y : e == 2 ? bf.z : bf.w);
      } else if (BIAS) {
        v = (key < nvis) ? fmaf(v, (e < 2) ? c_lo : c_hi,
                                __fmul_rn(((e < 2) ? brow_lo : brow_hi)[kbase + key], kLog2e))
                         : kNegInf;
      } else if (key >= nvis) {
        v = kNegInf;
      }
      S[n][e] = v;
    }
    mx_lo = fmax3(mx_lo, S[n][0], S[n][1]);
    mx_hi = fmax3(mx_hi, S[n][2], S[n][3]);
  }
#pragma unroll
  for (int sh = 1; sh < 4; sh <<= 1) {
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, sh));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, sh));
  }
  const float mb_lo = BIAS ? mx_lo : ((mx_lo == kNegInf) ? kNegInf : __fmul_rn(mx_lo, c_lo));
  const float mb_hi = BIAS ? mx_hi : ((mx_hi == kNegInf) ? kNegInf : __fmul_rn(mx_hi, c_hi));
  const float mn_lo = fmaxf(rp.m_lo, mb_lo), mn_hi = fmaxf(rp.m_hi, mb_hi);
  const bool dead_lo = (mn_lo == kNegInf), dead_hi = (mn_hi == kNegInf);
  const float al_lo = dead_lo ? 1.f : ex2_approx(rp.m_lo - mn_lo);
  const float al_hi = dead_hi ? 1.f : ex2_approx(rp.m_hi - mn_hi);
  const float kn_lo = dead_lo ? 0.f : (kLog2_448 - mn_lo);
  const float kn_hi = dead_hi ? 0.f : (kLog2_448 - mn_hi);
  rp.m_lo = mn_lo;
  rp.m_hi = mn_hi;
  if (!FIRST) {
#pragma unroll
    for (int n = 0; n < NTO; ++n) {  // O = alpha O (alpha = 1 is exact)
      o[n][0] *= al_lo;
      o[n][1] *= al_lo;
      o[n][2] *= al_hi;
      o[n][3] *= al_hi;
    }
  }
  float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
  for (int s = 0; s < KB / 16; ++s) {
    if (s < nstep) {
      uint32_t af[4];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int n = 2 * s + half;
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          p[e] = ex2_approx(BIAS ? (S[n][e] + ((e < 2) ? kn_lo : kn_hi))
                                 : fmaf(S[n][e], (e < 2) ? c_lo : c_hi, (e < 2) ? kn_lo : kn_hi));
        sum_lo += p[0] + p[1];
        sum_hi += p[2] + p[3];
        af[2 * half] = e4m3x2_to_f16x2(cvt_e4m3x2(p[0], p[1]));      // a0 / a2: row g
        af[2 * half + 1] = e4m3x2_to_f16x2(cvt_e4m3x2(p[2], p[3]));  // a1 / a3: row g + 8
      }
#pragma unroll
      for (int n = 0; n < NTO; n += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(v_addr + n * 8 * kVPitch + s * 32, b0, b1, b2, b3);
        mma_f16_16816(o[n], af[0], af[1], af[2], af[3], b0, b1);
        mma_f16_16816(o[n + 1], af[0], af[1], af[2], af[3], b2, b3);
      }
    }
  }
#pragma unroll
  for (int sh = 1; sh < 4; sh <<= 1) {
    sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, sh);
    sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, sh);
  }
  rp.l_lo = FIRST ? sum_lo : fmaf(al_lo, rp.l_lo, sum_lo);  // (alpha 0 l + sum = sum: l is 0)
  rp.l_hi = FIRST ? sum_hi : fmaf(al_hi, rp.l_hi, sum_hi);
}

// out = O s_v / l (l in units of 448 P) and lse for a lane's rows r_lo, r_hi.
// sv_pre: the lane's V channel scales (channels 8n + 2 t4, + 1), read ahead
// by the caller; else read here.
template <int D>
__device__ __forceinline__ void epilogue(const AttnArgs& a, int bh, int bkv, int r_lo, int r_hi, int t4,
                                         const RowPair& rp, const float (&o)[D / 8][4],
                                         const float2* sv_pre = nullptr) {
  const float* svp = a.v_scales + static_cast<size_t>(bkv) * D;
  const float il_lo = (rp.l_lo > 0.f) ? 1.f / rp.l_lo : 0.f, il_hi = (rp.l_hi > 0.f) ? 1.f / rp.l_hi : 0.f;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int c = 8 * n + 2 * t4;
    const float sv0 = sv_pre ? sv_pre[n].x : svp[c], sv1 = sv_pre ? sv_pre[n].y : svp[c + 1];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int row = half ? r_hi : r_lo;
      if (row >= a.Nq) continue;
      const float il = half ? il_hi : il_lo;
      const float v0 = o[n][2 * half] * (sv0 * il), v1 = o[n][2 * half + 1] * (sv1 * il);
      const size_t off = (static_cast<size_t>(bh) * a.Nq + row) * D + c;
      if (!QATTN_IN_BOUNDS(bh < a.B * a.Hq && c + 1 < D)) continue;
      if (a.out_bf16) {
        *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(a.out) + off) =
            __floats2bfloat162_rn(v0, v1);
      } else {
        *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + off) = make_float2(v0, v1);
      }
    }
  }
  if (a.lse && t4 == 0) {
    if (r_lo < a.Nq)
      a.lse[static_cast<size_t>(bh) * a.Nq + r_lo] =
          (rp.l_lo > 0.f) ? (rp.m_lo + __log2f(rp.l_lo) - kLog2_448) * kLn2 : kNegInf;
    if (r_hi < a.Nq)
      a.lse[static_cast<size_t>(bh) * a.Nq + r_hi] =
          (rp.l_hi > 0.f) ? (rp.m_hi + __log2f(rp.l_hi) - kLog2_448) * kLn2 : kNegInf;
  }
}

// ---------------------------------------------------------------- Nk <= 256
template <int D>
struct ShortSmem {
  static constexpr int kQKPitch = 2 * D + 16;    // bytes per fp16 row of Q or K (conflict-free ldmatrix)
  static constexpr int kVPitch = 2 * kBlk + 16;  // bytes per fp16 row of V^T (one channel, 128 keys)
  static constexpr int kK = kBlk * kQKPitch;
  static constexpr int kV = D * kVPitch;
  static constexpr int bytes(int warps) { return 16 * warps * kQKPitch + kK + kV; }
};

template <int D, bool BIAS>
__global__ void __launch_bounds__(kMaxWarps * 32, 2) attn_short_kernel(const ShortArgs sa) {
  using SM = ShortSmem<D>;
  const AttnArgs& a = sa.a;
  extern __shared__ __align__(16) uint8_t smem[];
  const int W = blockDim.x >> 5;
  uint8_t* sq = smem;
  uint8_t* sk = sq + 16 * W * SM::kQKPitch;
  uint8_t* sv = sk + SM::kK;
  pdl_trigger();
  pdl_wait();  // codes, scales and V8^T come from the kernels before this one
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int bh = blockIdx.y, b = bh / a.Hq, h = bh % a.Hq;
  const int bkv = b * a.Hkv + h / (a.Hq / a.Hkv);
  const int q0 = blockIdx.x * 16 * W;
  const int nqb = (a.Nq + kBlk - 1) / kBlk, nkb = (a.Nk + kBlk - 1) / kBlk;
  const int8_t* qg = sa.q_codes + static_cast<size_t>(bh) * a.Nq * D;
  const int8_t* kg = sa.k_codes + static_cast<size_t>(bkv) * a.Nk * D;
  const uint8_t* vg = sa.v8t + static_cast<size_t>(bkv) * D * sa.ldv;
  for (int v = threadIdx.x; v < 16 * W * (D / 16); v += blockDim.x) {  // Q rows (zeros past Nq)
    const int r = v / (D / 16), c16 = v % (D / 16);
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (q0 + r < a.Nq) x = *reinterpret_cast<const uint4*>(qg + static_cast<size_t>(q0 + r) * D + 16 * c16);
    store_codes16_f16(sq + r * SM::kQKPitch + c16 * 32, x);
  }
  const int r_lo = q0 + 16 * warp + g, r_hi = r_lo + 8;
  const bool active = q0 + 16 * warp < a.Nq;
  const float sq_lo = scale_of(a.q_scales, a.q_gran, bh, nqb, min(r_lo, a.Nq - 1) / kBlk);
  const float sq_hi = scale_of(a.q_scales, a.q_gran, bh, nqb, min(r_hi, a.Nq - 1) / kBlk);
  const float* brow_lo = nullptr;
  const float* brow_hi = nullptr;
  if (BIAS) {
    const float* bh0 = a.bias + static_cast<size_t>(h) * a.bias_head_stride;
    brow_lo = bh0 + static_cast<size_t>(min(r_lo, a.Nq - 1)) * a.Nk;
    brow_hi = bh0 + static_cast<size_t>(min(r_hi, a.Nq - 1)) * a.Nk;
  }
  RowPair rp;
  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  // ldmatrix row addresses: lane l gives row l % 8 of matrix l / 8
  const int mrow = lane & 7, mat = lane >> 3;
  const uint32_t q_addr = smem_u32(sq) + (16 * warp + mrow + (mat & 1) * 8) * SM::kQKPitch + (mat >> 1) * 16;
  const uint32_t k_addr = smem_u32(sk) + (mrow + (mat >> 1) * 8) * SM::kQKPitch + (mat & 1) * 16;
  const uint32_t v_addr = smem_u32(sv) + (mrow + (mat >> 1) * 8) * SM::kVPitch + (mat & 1) * 16;
  for (int j = 0; j < nkb; ++j) {
    const int kbase = j * kBlk;
    const int nvis = min(kBlk, a.Nk - kbase);
    const int nstep = (nvis + 15) / 16;
    __syncthreads();  // the previous block's K and V rows are read
    for (int v = threadIdx.x; v < nstep * 16 * (D / 16); v += blockDim.x) {  // K rows (zeros past Nk)
      const int key = v / (D / 16), c16 = v % (D / 16);
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (key < nvis) x = *reinterpret_cast<const uint4*>(kg + static_cast<size_t>(kbase + key) * D + 16 * c16);
      store_codes16_f16(sk + key * SM::kQKPitch + c16 * 32, x);
    }
    for (int v = threadIdx.x; v < D * nstep; v += blockDim.x) {  // V8^T: 16 keys of a channel per item
      const int c = v / nstep, k16 = v % nstep;
      store_e4m3x16_f16(sv + c * SM::kVPitch + 32 * k16,
                        *reinterpret_cast<const uint4*>(vg + static_cast<size_t>(c) * sa.ldv + kbase + 16 * k16));
    }
    __syncthreads();
    if (!active) continue;
    const float sk = scale_of(a.k_scales, a.k_gran, bkv, nkb, j);
    block_step<D, BIAS, kBlk>(q_addr, k_addr, v_addr, nvis, kbase,
                              __fmul_rn(__fmul_rn(__fmul_rn(sq_lo, sk), a.sm_scale), kLog2e),
                              __fmul_rn(__fmul_rn(__fmul_rn(sq_hi, sk), a.sm_scale), kLog2e), brow_lo,
                              brow_hi, t4, rp, o);
  }
  if (active) epilogue<D>(a, bh, bkv, r_lo, r_hi, t4, rp, o);
}

// ---------------------------------------------------------------- Nq, Nk <= 64
template <int D>
struct WinSmem {
  static constexpr int kQKPitch = 2 * D + 16;
  static constexpr int kVPitch = 2 * kWin + 16;
  static constexpr int kQ = kWin * kQKPitch;
  static constexpr int kBytes = 2 * kQ + D * kVPitch;  // Q rows, K rows, V^T rows
  static constexpr int kChunks = kWin * D / 16;         // 16-byte chunks of each of Q, K, V8^T
  static constexpr int kPer = kChunks / kWinThreads;    // per thread
};

// The raw codes of one head, kPer 16-byte chunks each of Q, K and V8^T per
// thread (zeros past Nq, Nk, and past V8^T's visible 16-key steps).
template <int D>
struct WinRaw {
  uint4 q[WinSmem<D>::kPer], k[WinSmem<D>::kPer], v[WinSmem<D>::kPer];
};

template <int D>
__device__ __forceinline__ void win_load(const ShortArgs& sa, int w, int bkv, WinRaw<D>& raw) {
  const AttnArgs& a = sa.a;
  const int8_t* qg = sa.q_codes + static_cast<size_t>(w) * a.Nq * D;
  const int8_t* kg = sa.k_codes + static_cast<size_t>(bkv) * a.Nk * D;
  const uint8_t* vg = sa.v8t + static_cast<size_t>(bkv) * D * sa.ldv;
  const int nstep = (a.Nk + 15) / 16;
#pragma unroll
  for (int i = 0; i < WinSmem<D>::kPer; ++i) {
    const int v = threadIdx.x + i * kWinThreads;
    const int r = v / (D / 16), c16 = v % (D / 16);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    raw.q[i] = (r < a.Nq) ? *reinterpret_cast<const uint4*>(qg + static_cast<size_t>(r) * D + 16 * c16) : z;
    raw.k[i] = (r < a.Nk) ? *reinterpret_cast<const uint4*>(kg + static_cast<size_t>(r) * D + 16 * c16) : z;
    const int c = v / (kWin / 16), k16 = v % (kWin / 16);
    raw.v[i] = (k16 < nstep) ? *reinterpret_cast<const uint4*>(vg + static_cast<size_t>(c) * sa.ldv + 16 * k16) : z;
  }
}

template <int D, bool BIAS>
__global__ void __launch_bounds__(kWinThreads, D == 32 ? 5 : 4) attn_window_kernel(const ShortArgs sa, int n_heads) {
  using SM = WinSmem<D>;
  const AttnArgs& a = sa.a;
  __shared__ __align__(16) uint8_t smem[SM::kBytes];
  uint8_t* sq = smem;
  uint8_t* sk = sq + SM::kQ;
  uint8_t* sv = sk + SM::kQ;
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int r_lo = 16 * warp + g, r_hi = r_lo + 8;
  const bool active = 16 * warp < a.Nq;
  const int mrow = lane & 7, mat = lane >> 3;
  const uint32_t q_addr = smem_u32(sq) + (16 * warp + mrow + (mat & 1) * 8) * SM::kQKPitch + (mat >> 1) * 16;
  const uint32_t k_addr = smem_u32(sk) + (mrow + (mat >> 1) * 8) * SM::kQKPitch + (mat & 1) * 16;
  const uint32_t v_addr = smem_u32(sv) + (mrow + (mat >> 1) * 8) * SM::kVPitch + (mat & 1) * 16;
  // BIAS: the lane's 32 bias values of its rows and S-fragment keys, times
  // log2 e, -inf past Nk (so fmaf(S, c, b) is the block step's masked t),
  // refilled only when the head index changes (never, when the grid is a
  // multiple of Hq: each CTA then sees one head index).  A lane reads back
  // only what it wrote, so no barrier guards the array.
  __shared__ float4 sbias[BIAS ? kWinThreads / 32 : 1][BIAS ? kWin / 8 : 1][32];
  int h_frag = -1;
  // The CTA's heads w = blockIdx.x + k G (G = gridDim.x), as (batch, head)
  // pairs stepped without divisions: (b, h) of w + G = (b + G / Hq, h + G % Hq),
  // carrying h >= Hq into b.
  const int grp = a.Hq / a.Hkv;
  const int db = static_cast<int>(gridDim.x) / a.Hq, dh = static_cast<int>(gridDim.x) % a.Hq;
  int b = static_cast<int>(blockIdx.x) / a.Hq, h = static_cast<int>(blockIdx.x) % a.Hq;
  auto kv_of = [&](int bb, int hh) { return bb * a.Hkv + hh / grp; };
  auto step = [&](int& bb, int& hh) {
    bb += db;
    hh += dh;
    if (hh >= a.Hq) {
      hh -= a.Hq;
      ++bb;
    }
  };
  WinRaw<D> raw;
  if (blockIdx.x < n_heads) win_load<D>(sa, blockIdx.x, kv_of(b, h), raw);
  for (int w = blockIdx.x; w < n_heads; w += gridDim.x, step(b, h)) {
    __syncthreads();  // the previous head's rows are read
    // the head's scales, read before the conversion so their latency hides
    // under it and the block step
    const int bkv = kv_of(b, h);
    const float sq_ = scale_of(a.q_scales, a.q_gran, w, 1, 0);
    const float sk_ = scale_of(a.k_scales, a.k_gran, bkv, 1, 0);
    float2 vsc[D / 8];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
      vsc[n] = *reinterpret_cast<const float2*>(a.v_scales + static_cast<size_t>(bkv) * D + 8 * n + 2 * t4);
#pragma unroll
    for (int i = 0; i < SM::kPer; ++i) {
      const int v = threadIdx.x + i * kWinThreads;
      const int r = v / (D / 16), c16 = v % (D / 16);
      store_codes16_f16(sq + r * SM::kQKPitch + c16 * 32, raw.q[i]);
      store_codes16_f16(sk + r * SM::kQKPitch + c16 * 32, raw.k[i]);
      const int c = v / (kWin / 16), k16 = v % (kWin / 16);
      store_e4m3x16_f16(sv + c * SM::kVPitch + 32 * k16, raw.v[i]);
    }
    if (w + gridDim.x < n_heads) {  // under this head's math
      int bn = b, hn = h;
      step(bn, hn);
      win_load<D>(sa, w + gridDim.x, kv_of(bn, hn), raw);
    }
    __syncthreads();
    if (!active) continue;
    const float c = __fmul_rn(__fmul_rn(__fmul_rn(sq_, sk_), a.sm_scale), kLog2e);
    if (BIAS && h != h_frag) {
      const float* bh0 = a.bias + static_cast<size_t>(h) * a.bias_head_stride;
      const float* brow_lo = bh0 + static_cast<size_t>(min(r_lo, a.Nq - 1)) * a.Nk;
      const float* brow_hi = bh0 + static_cast<size_t>(min(r_hi, a.Nq - 1)) * a.Nk;
#pragma unroll
      for (int n = 0; n < kWin / 8; ++n) {
        float bv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = 8 * n + 2 * t4 + (e & 1);
          bv[e] = (key < a.Nk) ? __fmul_rn(((e < 2) ? brow_lo : brow_hi)[key], kLog2e) : kNegInf;
        }
        sbias[warp][n][lane] = make_float4(bv[0], bv[1], bv[2], bv[3]);
      }
      h_frag = h;
    }
    RowPair rp;
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    block_step<D, BIAS, kWin, BIAS, true>(q_addr, k_addr, v_addr, a.Nk, 0, c, c, nullptr, nullptr, t4, rp, o,
                                    BIAS ? &sbias[warp][0][lane] : nullptr);
    epilogue<D>(a, w, bkv, r_lo, r_hi, t4, rp, o, vsc);
  }
}

template <int D, bool BIAS>
cudaError_t launch_short_t(const ShortArgs& sa, cudaStream_t s) {
  const int nblk = (sa.a.Nq + 15) / 16;
  const int per_head = (nblk + kMaxWarps - 1) / kMaxWarps;
  const int W = (nblk + per_head - 1) / per_head;
  const int smem = ShortSmem<D>::bytes(W);
  cudaError_t e = cudaFuncSetAttribute(attn_short_kernel<D, BIAS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       ShortSmem<D>::bytes(kMaxWarps));
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_short_kernel<D, BIAS>, dim3(per_head, sa.a.B * sa.a.Hq), dim3(32 * W), smem, s, sa);
}

template <int D, bool BIAS>
cudaError_t launch_window_t(const ShortArgs& sa, cudaStream_t s) {
  static const int slots = [] {
    int n = 0, dev = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_window_kernel<D, BIAS>, kWinThreads, 0) !=
            cudaSuccess || n < 1)
      n = 1;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
      sms = 1;
    return n * sms;
  }();
  const int n_heads = sa.a.B * sa.a.Hq;
  return launch_pdl(attn_window_kernel<D, BIAS>, dim3(min(n_heads, slots)), dim3(kWinThreads), 0, s, sa,
                    n_heads);
}

}  // namespace

unsigned int check_take_short() { return check_take_local(); }

bool attn_short_eligible(const AttnArgs& a) {
  return (a.d == 32 || a.d == 64) && !a.causal && !a.pv_int8 && a.Nk >= 1 && a.Nk <= kShortMaxNk &&
         a.Nq >= 1;
}

bool attn_window_eligible(const AttnArgs& a) {
  return attn_short_eligible(a) && a.Nq <= kWin && a.Nk <= kWin;
}

cudaError_t launch_attn_short(const AttnArgs& a, const int8_t* q_codes, const int8_t* k_codes,
                              const uint8_t* v8t, long long ldv, cudaStream_t s) {
  if (!attn_short_eligible(a)) return cudaErrorInvalidValue;
  const ShortArgs sa{a, q_codes, k_codes, v8t, ldv};
  const bool bias = a.bias != nullptr;
  if (attn_window_eligible(a)) {
    if (a.d == 32) return bias ? launch_window_t<32, true>(sa, s) : launch_window_t<32, false>(sa, s);
    return bias ? launch_window_t<64, true>(sa, s) : launch_window_t<64, false>(sa, s);
  }
  if (a.d == 32) return bias ? launch_short_t<32, true>(sa, s) : launch_short_t<32, false>(sa, s);
  return bias ? launch_short_t<64, true>(sa, s) : launch_short_t<64, false>(sa, s);
}

}  // namespace qattn
