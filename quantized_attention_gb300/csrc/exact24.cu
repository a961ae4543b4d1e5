// High-accuracy attention on an int8 KV cache with operands split exact to 24
// bits (Strata PR "prompt_attn_i8v3_kernel", "What it does", "Operands": q
// scaled per (head, 64-dim group) and p per (row, chunk) to 127, then
// X = rint(x * 65536) = h * 65536 + l * 256 + m, three exact products with
// the stored int8 codes combined in fp32; "Measured": ~2e-6 max relative error
// against FP64).
//
// The exact products run on the tensor cores as fp16 x fp16 with fp32
// accumulation (mma.m16n8k16, fragments by ldmatrix): h, l, m and the int8
// codes are exact fp16 values, and a part's sum over 64 channels (or 64 keys)
// is an integer below 64 * 255 * 127 < 2^24, so no rounding occurs.  (GB300 runs the warp-level
// fp16 MMA about four times faster than its int8 one.)  The K and V channel
// scales of the cache are factored out: K's is folded into q before the
// split, V's applied to the output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kGroup = 64;   // q scale granule: 64 channels of a head
constexpr int kChunk = 64;   // keys per chunk (P scale granule, online-softmax block)
constexpr int kRows = 64;    // query rows per CTA (4 warps x 16)
constexpr int kThreads = 128;
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

// D(16x8 f32) += A(16x16 f16) * B(16x8 f16).  a0/a2: row g, k = 2t, 2t+1 /
// 2t+8, 2t+9; a1/a3: row g + 8; b0/b1: column g, k = 2t, 2t+1 / 2t+8, 2t+9;
// d0, d1: row g, columns 2t, 2t+1; d2, d3: row g + 8.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

// ---------------------------------------------------------------- attention
template <int D>
struct Ex24Smem {
  static constexpr int kPitch = D * 2 + 16;         // bytes per fp16 row (8 rows hit 8 bank groups)
  static constexpr int kQ = 3 * kRows * kPitch;     // the three q parts
  static constexpr int kKV = kChunk * kPitch;       // K or V codes of a chunk as fp16
  static constexpr int kBytes = kQ + 2 * kKV;
};

struct Ex24Args {
  int B, Hq, Hkv, Nq, Nk;
  int causal;
  int pos0;
  float cfac;  // fp32(sm_scale * log2 e)
  long long cap;  // cache rows per (batch, KV head)
  const __half* parts;
  size_t plane;
  const float* group_scale;
  const int8_t* k_codes;
  const int8_t* v_codes;
  const float* v_chan_scale;
  void* out;
  int out_bf16;
  float* lse;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// CTA: 64 query rows of one (batch, query head); warp w owns rows 16w..16w+15.
// Per 64-key chunk the K and V codes are converted once to exact fp16 rows in
// shared memory; fragments come from ldmatrix (V transposed).  S = sum over
// groups and parts of weight * (part . K codes), fp32 multiply-adds;
// the online softmax; P per (row, chunk) to 127 and its three parts;
// O += sum of part weights * (part . V codes).
template <int D>
__global__ void __launch_bounds__(kThreads) exact24_attn_kernel(const Ex24Args a) {
  using SM = Ex24Smem<D>;
  constexpr int NG = D / kGroup;
  constexpr int NTO = D / 8;  // PV n-tiles (8 channels each)
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* sq = smem;
  uint8_t* sk = smem + SM::kQ;
  uint8_t* sv = smem + SM::kQ + SM::kKV;
  __shared__ float gs[NG];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int bh = blockIdx.y, b = bh / a.Hq, h = bh % a.Hq;
  const int bkv = b * a.Hkv + h / (a.Hq / a.Hkv);
  const int q0 = blockIdx.x * kRows;
  // the CTA's rows of the three q parts
  for (int v = threadIdx.x; v < 3 * kRows * (D / 8); v += kThreads) {
    const int p = v / (kRows * (D / 8)), rem = v % (kRows * (D / 8));
    const int r = rem / (D / 8), c8 = rem % (D / 8);
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (q0 + r < a.Nq)
      x = *reinterpret_cast<const uint4*>(a.parts + p * a.plane +
                                          (static_cast<size_t>(bh) * a.Nq + q0 + r) * D + c8 * 8);
    *reinterpret_cast<uint4*>(sq + (p * kRows + r) * SM::kPitch + c8 * 16) = x;
  }
  if (threadIdx.x < NG) gs[threadIdx.x] = a.group_scale[static_cast<size_t>(bh) * NG + threadIdx.x];
  const int r_lo = q0 + 16 * warp + g, r_hi = r_lo + 8;  // this lane's two rows
  float m_lo = kNegInf, m_hi = kNegInf, l_lo = 0.f, l_hi = 0.f;
  float o[NTO][4];
#pragma unroll
  for (int n = 0; n < NTO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  // ldmatrix row addresses: lane l gives row l % 8 of matrix l / 8
  const int mrow = lane & 7, mat = lane >> 3;
  const uint32_t q_addr = smem_u32(sq) + (16 * warp + mrow + (mat & 1) * 8) * SM::kPitch + (mat >> 1) * 16;
  const uint32_t k_addr = smem_u32(sk) + (mrow + (mat >> 1) * 8) * SM::kPitch + (mat & 1) * 16;
  const uint32_t v_addr = smem_u32(sv) + (mrow + (mat & 1) * 8) * SM::kPitch + (mat >> 1) * 16;
  // keys visible to the CTA's last row
  const int last_row = min(q0 + kRows, a.Nq) - 1;
  const int kend = a.causal ? min(a.Nk, a.pos0 + last_row + 1) : a.Nk;
  const int8_t* kg = a.k_codes + static_cast<size_t>(bkv) * a.cap * D;
  const int8_t* vg = a.v_codes + static_cast<size_t>(bkv) * a.cap * D;
  for (int k0 = 0; k0 < kend; k0 += kChunk) {
    __syncthreads();  // the previous chunk's tiles are read
    // K and V codes -> exact fp16 rows (zeros past Nk)
    for (int v = threadIdx.x; v < 2 * kChunk * (D / 16); v += kThreads) {
      const int which = v / (kChunk * (D / 16)), rem = v % (kChunk * (D / 16));
      const int key = rem / (D / 16), c16 = rem % (D / 16);
      const int8_t* src = which ? vg : kg;
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (k0 + key < a.Nk) x = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(k0 + key) * D) + c16);
      uint32_t hv[8];
      codes4_to_f16x2(x.x, hv[0], hv[1]);
      codes4_to_f16x2(x.y, hv[2], hv[3]);
      codes4_to_f16x2(x.z, hv[4], hv[5]);
      codes4_to_f16x2(x.w, hv[6], hv[7]);
      uint8_t* dst = (which ? sv : sk) + key * SM::kPitch + c16 * 32;
      *reinterpret_cast<uint4*>(dst) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
      *reinterpret_cast<uint4*>(dst + 16) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
    }
    __syncthreads();
    // ---- scores: 16 rows x 64 keys per warp, in the oracle's order
    float S[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) {
#pragma unroll
      for (int p = 0; p < 3; ++p) {
        float Sp[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) Sp[j][0] = Sp[j][1] = Sp[j][2] = Sp[j][3] = 0.f;
#pragma unroll 1
        for (int kk = 0; kk < kGroup / 16; ++kk) {
          const int ks = gr * (kGroup / 16) + kk;
          uint32_t a0, a1, a2, a3;
          ldsm_x4(q_addr + p * kRows * SM::kPitch + ks * 32, a0, a1, a2, a3);
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(k_addr + 8 * j * SM::kPitch + ks * 32, b0, b1, b2, b3);
            mma_f16_16816(Sp[j], a0, a1, a2, a3, b0, b1);
            mma_f16_16816(Sp[j + 1], a0, a1, a2, a3, b2, b3);
          }
        }
        const float wgt = gs[gr] * ((p == 0) ? 1.f : (p == 1) ? (1.f / 256.f) : (1.f / 65536.f));
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) S[j][e] = fmaf(wgt, Sp[j][e], S[j][e]);
      }
    }
    // ---- t, mask, online softmax (rows r_lo, r_hi; a row's 64 keys sit in
    // the 4 lanes of its quad)
    float mx_lo = kNegInf, mx_hi = kNegInf;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = k0 + 8 * j + 2 * t4 + (e & 1);
        const int row = (e < 2) ? r_lo : r_hi;
        const bool vis = key < a.Nk && row < a.Nq && (!a.causal || key <= a.pos0 + row);
        S[j][e] = vis ? __fmul_rn(S[j][e], a.cfac) : kNegInf;
      }
      mx_lo = fmaxf(mx_lo, fmaxf(S[j][0], S[j][1]));
      mx_hi = fmaxf(mx_hi, fmaxf(S[j][2], S[j][3]));
    }
#pragma unroll
    for (int sh = 1; sh < 4; sh <<= 1) {
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, sh));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, sh));
    }
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float al_lo = (m_lo == kNegInf) ? 0.f : ex2_approx(m_lo - mn_lo);
    const float al_hi = (m_hi == kNegInf) ? 0.f : ex2_approx(m_hi - mn_hi);
    const float ref_lo = (mn_lo == kNegInf) ? 0.f : mn_lo, ref_hi = (mn_hi == kNegInf) ? 0.f : mn_hi;
    float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      S[j][0] = ex2_approx(S[j][0] - ref_lo);
      S[j][1] = ex2_approx(S[j][1] - ref_lo);
      S[j][2] = ex2_approx(S[j][2] - ref_hi);
      S[j][3] = ex2_approx(S[j][3] - ref_hi);
      sum_lo += S[j][0] + S[j][1];
      sum_hi += S[j][2] + S[j][3];
    }
    l_lo = al_lo * l_lo + sum_lo;  // the lane's share; quad-summed at the end
    l_hi = al_hi * l_hi + sum_hi;
    m_lo = mn_lo;
    m_hi = mn_hi;
    // P's chunk maximum per row -> s_p = pmax / 127, x = P / s_p
    const float pm_lo = (mx_lo == kNegInf) ? 0.f : ex2_approx(mx_lo - ref_lo);
    const float pm_hi = (mx_hi == kNegInf) ? 0.f : ex2_approx(mx_hi - ref_hi);
    const float sp_lo = __fdiv_rn(pm_lo, 127.0f), sp_hi = __fdiv_rn(pm_hi, 127.0f);
    // x * 65536 = P * (65536 / s_p): one reciprocal per row
    const float ci_lo = (sp_lo > 0.f) ? __fdiv_rn(65536.0f, sp_lo) : 0.f;
    const float ci_hi = (sp_hi > 0.f) ? __fdiv_rn(65536.0f, sp_hi) : 0.f;
#pragma unroll
    for (int n = 0; n < NTO; ++n) {
      o[n][0] *= al_lo;
      o[n][1] *= al_lo;
      o[n][2] *= al_hi;
      o[n][3] *= al_hi;
    }
    // ---- PV: the three parts' A fragments (the S layout is the A layout),
    // then per half of the channels and per part an exact product, combined
    // into O with weights s_p, s_p/256, s_p/65536
    uint32_t af[3][4][4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int j = 2 * s + half;
        float v[3][4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          split24_pos(S[j][e] * ((e < 2) ? ci_lo : ci_hi), v[0][e], v[1][e], v[2][e]);
#pragma unroll
        for (int p = 0; p < 3; ++p) {
          af[p][s][2 * half] = pack_f2h2(v[p][0], v[p][1]);      // a0 / a2: row g
          af[p][s][2 * half + 1] = pack_f2h2(v[p][2], v[p][3]);  // a1 / a3: row g + 8
        }
      }
    }
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
#pragma unroll
      for (int p = 0; p < 3; ++p) {
        float op[NTO / 2][4];
#pragma unroll
        for (int n = 0; n < NTO / 2; ++n) op[n][0] = op[n][1] = op[n][2] = op[n][3] = 0.f;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
#pragma unroll
          for (int n = 0; n < NTO / 2; n += 2) {
            const int nt = hc * (NTO / 2) + n;
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(v_addr + 16 * s * SM::kPitch + nt * 16, b0, b1, b2, b3);
            mma_f16_16816(op[n], af[p][s][0], af[p][s][1], af[p][s][2], af[p][s][3], b0, b1);
            mma_f16_16816(op[n + 1], af[p][s][0], af[p][s][1], af[p][s][2], af[p][s][3], b2, b3);
          }
        }
        const float pw = (p == 0) ? 1.f : (p == 1) ? (1.f / 256.f) : (1.f / 65536.f);
        const float w_lo = sp_lo * pw, w_hi = sp_hi * pw;
#pragma unroll
        for (int n = 0; n < NTO / 2; ++n) {
          const int nt = hc * (NTO / 2) + n;
          o[nt][0] = fmaf(w_lo, op[n][0], o[nt][0]);
          o[nt][1] = fmaf(w_lo, op[n][1], o[nt][1]);
          o[nt][2] = fmaf(w_hi, op[n][2], o[nt][2]);
          o[nt][3] = fmaf(w_hi, op[n][3], o[nt][3]);
        }
      }
    }
  }
  // ---- epilogue: quad-sum l, O * s_v / l
#pragma unroll
  for (int sh = 1; sh < 4; sh <<= 1) {
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, sh);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, sh);
  }
  const float inv_lo = (l_lo > 0.f) ? 1.f / l_lo : 0.f, inv_hi = (l_hi > 0.f) ? 1.f / l_hi : 0.f;
  const float* svc = a.v_chan_scale + static_cast<size_t>(bkv) * D;
#pragma unroll
  for (int n = 0; n < NTO; ++n) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = (e < 2) ? r_lo : r_hi;
      if (row >= a.Nq) continue;
      const int c = 8 * n + 2 * t4 + (e & 1);
      const float val = o[n][e] * __ldg(svc + c) * ((e < 2) ? inv_lo : inv_hi);
      const size_t idx = (static_cast<size_t>(bh) * a.Nq + row) * D + c;
      if (a.out_bf16) reinterpret_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16(val);
      else reinterpret_cast<float*>(a.out)[idx] = val;
    }
  }
  if (a.lse && t4 == 0) {
    if (r_lo < a.Nq)
      a.lse[static_cast<size_t>(bh) * a.Nq + r_lo] = (l_lo > 0.f) ? (m_lo + __log2f(l_lo)) * kLn2 : kNegInf;
    if (r_hi < a.Nq)
      a.lse[static_cast<size_t>(bh) * a.Nq + r_hi] = (l_hi > 0.f) ? (m_hi + __log2f(l_hi)) * kLn2 : kNegInf;
  }
}

template <int D>
cudaError_t launch_t(const Exact24Args& x, cudaStream_t s) {
  const size_t plane = static_cast<size_t>(x.B) * x.Hq * x.Nq * D;
  __half* parts = static_cast<__half*>(x.ws);
  float* gsc = reinterpret_cast<float*>(static_cast<char*>(x.ws) + ((3 * plane * 2 + 255) / 256) * 256);
  cudaError_t e = launch_pdl(q_split_kernel<D>, dim3(x.B * x.Hq), dim3(256), 0, s,
                             static_cast<const uint16_t*>(x.Q), x.k_chan_scale, x.Hq, x.Hkv, x.Nq,
                             parts, gsc, plane);
  if (e != cudaSuccess) return e;
  Ex24Args a{};
  a.B = x.B;
  a.Hq = x.Hq;
  a.Hkv = x.Hkv;
  a.Nq = x.Nq;
  a.Nk = x.Nk;
  a.causal = x.causal;
  a.pos0 = x.pos0;
  a.cfac = x.sm_scale * kLog2e;  // one fp32 multiply, round to nearest
  a.cap = x.cap;
  a.parts = parts;
  a.plane = plane;
  a.group_scale = gsc;
  a.k_codes = x.k_codes;
  a.v_codes = x.v_codes;
  a.v_chan_scale = x.v_chan_scale;
  a.out = x.out;
  a.out_bf16 = x.out_bf16;
  a.lse = x.lse;
  constexpr int smem = Ex24Smem<D>::kBytes;
  e = cudaFuncSetAttribute(exact24_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(exact24_attn_kernel<D>, dim3((x.Nq + kRows - 1) / kRows, x.B * x.Hq), dim3(kThreads),
                    smem, s, a);
}

}  // namespace

size_t exact24_ws_bytes(long long B, long long Hq, long long Nq, long long d) {
  const long long plane = B * Hq * Nq * d;
  return static_cast<size_t>((3 * plane * 2 + 255) / 256 * 256 + (B * Hq * (d / kGroup) * 4 + 255) / 256 * 256);
}

cudaError_t launch_exact24(const Exact24Args& x, cudaStream_t s) {
  return x.d == 64 ? launch_t<64>(x, s) : launch_t<128>(x, s);
}

}  // namespace qattn
