// QFlash's integer-only attention ("QFlash: Bridging Quantization and Memory
// Efficiency in Vision Transformer Attention", Algorithm 1, sections 4.2-4.6):
// per-tensor int8 Q, K, V; S = q.k in int32; the running row max; ShiftExp2
// (X = Q X0 + R, 2^(s~ R) ~= s~ R / 2 + 1, so P = ((R >> 1) + X0) >> -Q at
// scale s~, eq. (5)-(8)); P requantized to int8 by a fixed-point multiplier
// (eq. (9)-(10)); row sums (eq. (11)); the accumulators rescaled by the
// max-offset factor alpha with ScaleRelease (read here as floor(x * alpha / X0);
// the paper defers its definition to an appendix not cited here) and O += P.V
// in int32; out = floor(O / l) as int8 codes of V's scale.
//
// Both products run on the warp-level fp16 tensor cores (mma.m16n8k16, fp32
// accumulation), which on this GPU run about four times the int8 warp MMA:
// the int8 codes and the P codes (0..127) are exact fp16 values and every
// partial sum is an integer below 2^24 (|q.k| <= 128^2 * 128 = 2^21; a tile's
// P.V <= 64 * 127 * 128), so the fp32 accumulator holds it exactly and the
// products are the int32 ones.  Every other step is integer arithmetic, so the
// result is bit-exact with the oracle.
//
// CTA: 16 * W query rows of one (batch, head), W <= 8 warps sized to Nq so a
// ViT row count (197) splits into two CTAs of 7 warps.  Per 64-key tile the
// K and V codes are staged by cp.async while the previous tile computes, then
// converted once to fp16 rows that ldmatrix reads (V transposed); S stays in
// registers and the P codes go straight into the A fragments of the PV
// product.
#include <cmath>
#include <cuda_runtime.h>

#include "qattn_check.cuh"
#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kTile = 64;        // keys per tile (Bc): the points where O is rescaled
constexpr int kMaxWarps = 8;     // 16 query rows per warp
constexpr int kM0 = -(1 << 21);  // initial running max
constexpr float kMaxX0 = 1073741824.0f;               // 2^30: a larger X0 leaves the int32 domain
constexpr float kLog2e = 1.44269502162933349609375f;  // fp32(log2 e)

struct IntsmConst {
  int x0;                   // rint(1 / s~)
  int M, r;                 // P requantization (P * M) >> r; r < 0 is stored as M = 128, r = 0
  uint32_t dm;              // floor(n / x0) = umulhi(n * 2^9, dm) >> dl for n < 2^23
  int dl;                   // ceil(log2 x0)
  uint32_t k0, k1;          // ShiftExp2 from an fp32's bits (below): -512 * kMagicBits, 2 x0 + kMagicBits
  unsigned long long cfix;  // floor(2^62 / x0)
};

// An fp32 holding an integer v with |v| <= 2^22 -> v: v + 1.5 * 2^23 is exact
// and carries v in its low mantissa bits.
constexpr float kMagic = 12582912.0f;
constexpr int kMagicBits = 0x4B400000;
__device__ __forceinline__ int f2i_small(float v) { return __float_as_int(v + kMagic) - kMagicBits; }

__device__ __forceinline__ uint32_t shr_clamped(uint32_t v, uint32_t s) {  // 0 once s >= 32
  uint32_t r;
  asm("shr.u32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(s));
  return r;
}

// The constants from the per-tensor scales, in the oracle's fp32 steps.
// False when s~ is not a positive finite number or X0 exceeds 2^30.
__device__ __forceinline__ bool intsm_constants(float sq, float sk, float sm_scale, IntsmConst& c) {
  const float st = __fmul_rn(__fmul_rn(__fmul_rn(sq, sk), sm_scale), kLog2e);
  const float inv = __fdiv_rn(1.0f, st);
  if (!(st > 0.f) || !(inv <= kMaxX0)) return false;
  c.x0 = max(1, __float2int_rn(inv));
  const float ratio = __fmul_rn(127.0f, st);
  int e;
  const float f = frexpf(ratio, &e);      // ratio = f * 2^e, f in [0.5, 1)
  const int n = (f == 0.5f) ? e - 1 : e;  // ceil(log2 ratio)
  c.r = 8 - n;
  c.M = __float2int_rn(ldexpf(ratio, c.r));  // exact scaling, then round
  if (c.r < 0) {  // ratio > 256: any P >= 1 saturates, as with a multiplier of 128
    c.M = 128;
    c.r = 0;
  }
  // division by the invariant x0 (Granlund and Montgomery, "Division by
  // Invariant Integers using Multiplication", 1994): with l = ceil(log2 x0)
  // and m = ceil(2^(23 + l) / x0) < 2^24 + 1, floor(n m / 2^(23 + l)) =
  // floor(n / x0) for every n < 2^23
  const unsigned long long x0u = static_cast<unsigned long long>(c.x0);
  c.dl = (c.x0 == 1) ? 0 : 32 - __clz(c.x0 - 1);
  c.dm = static_cast<uint32_t>(((1ull << (23 + c.dl)) + x0u - 1) / x0u);
  c.cfix = (1ull << 62) / x0u;
  c.k0 = 0u - 512u * static_cast<uint32_t>(kMagicBits);
  c.k1 = 2u * static_cast<uint32_t>(c.x0) + static_cast<uint32_t>(kMagicBits);
  return true;
}

// ShiftExp2 of X = -n <= 0 (0 <= n <= 2^22), given bits = the fp32 bits of
// n + 1.5 * 2^23: X = Q X0 + R with Q = -floor(n / X0) (truncation toward
// zero) and R = -(n mod X0), and ((R >> 1) + X0) >> -Q = (2 X0 - (n mod X0))
// >> (1 - Q), where 2 X0 - (n mod X0) = (floor(n / X0) + 2) X0 - n.
__device__ __forceinline__ int shift_exp2_bits(uint32_t bits, const IntsmConst& c) {
  const uint32_t q = __umulhi(bits * 512u + c.k0, c.dm) >> c.dl;  // floor(n / X0)
  const uint32_t u = q * static_cast<uint32_t>(c.x0) + (c.k1 - bits);
  return static_cast<int>(shr_clamped(u, q + 1));  // u <= 2 X0 <= 2^31
}

// P (scale s~) -> int8 code of scale 1/127: min((P * M) >> r, 127).  Narrow
// (X0 < 2^23, so P M < 2^31): one 32-bit product; else the 64-bit product as
// its two halves and a funnel shift (r <= 31).
template <bool Narrow>
__device__ __forceinline__ int requant(int P, const IntsmConst& c) {
  const uint32_t lo = static_cast<uint32_t>(P) * static_cast<uint32_t>(c.M);
  if (Narrow) return static_cast<int>(min(lo >> c.r, 127u));
  const uint32_t hi = __umulhi(static_cast<uint32_t>(P), static_cast<uint32_t>(c.M));
  return static_cast<int>(min(__funnelshift_r(lo, hi, c.r), 127u));
}

// ScaleRelease's per-row factor F = min(floor(alpha 2^31 / X0), 2^31 - 1):
// alpha * floor(2^62 / X0) / 2^31 falls short of alpha 2^31 / X0 by less
// than 1/2, so one step against the exact remainder completes the floor.
__device__ __forceinline__ int rescale_factor(int alpha, const IntsmConst& c) {
  const unsigned long long a = static_cast<unsigned long long>(alpha);
  const unsigned long long x0u = static_cast<unsigned long long>(c.x0);
  unsigned long long f = __umul64hi(a << 33, c.cfix);
  if ((a << 31) - f * x0u >= x0u) ++f;
  return static_cast<int>(min(f, 0x7fffffffull));
}

// ScaleRelease, floor(x * alpha / X0), for |x| < 2^31 and 0 <= alpha <= X0:
// (x F) >> 31 is within one of the quotient, and the remainder (in
// [-X0, 2 X0), exact in wrapping 32-bit arithmetic) gives the last step.
__device__ __forceinline__ int scale_release(int x, int alpha, int F, const IntsmConst& c) {
  int q = static_cast<int>((static_cast<long long>(x) * F) >> 31);
  const int rem = static_cast<int>(static_cast<uint32_t>(x) * static_cast<uint32_t>(alpha) -
                                   static_cast<uint32_t>(q) * static_cast<uint32_t>(c.x0));
  if (rem < 0) --q;
  else if (rem >= c.x0) ++q;
  return q;
}

// floor(o / l) for |o| < 2^31 and 1 <= l < 2^30, with Fi = min(floor(2^31 / l),
// 2^31 - 1): (o Fi) >> 31 is within one of the quotient and the remainder
// (in [-l, 2 l), exact in wrapping 32-bit arithmetic) gives the last step.
__device__ __forceinline__ int floor_div_recip(int o, int l, uint32_t Fi) {
  int q = static_cast<int>((static_cast<long long>(o) * static_cast<long long>(Fi)) >> 31);
  const int rem = static_cast<int>(static_cast<uint32_t>(o) - static_cast<uint32_t>(q) * static_cast<uint32_t>(l));
  if (rem < 0) --q;
  else if (rem >= l) ++q;
  return q;
}

// Two P codes (0..127) -> one f16x2 word: 0x6400 | y is the fp16 1024 + y,
// and one f16x2 subtraction of 1024 leaves y (exact).
__device__ __forceinline__ uint32_t codes2_to_f16x2(int y0, int y1) {
  const uint32_t w = 0x64006400u | static_cast<uint32_t>(y0) | (static_cast<uint32_t>(y1) << 16);
  uint32_t out;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(out) : "r"(w), "r"(0x64006400u));
  return out;
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

// 16 bytes global -> shared through L2; src_bytes 0 fills zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

struct IntsmArgs {
  int B, Hq, Hkv, Nq, Nk;
  float sm_scale;
  const int8_t* q_codes;
  const float* q_scale;
  const int8_t* k_codes;
  const float* k_scale;
  const int8_t* v_codes;
  int8_t* out;
  unsigned int* err;
};

template <int D>
struct IntsmSmem {
  static constexpr int kPitch = 2 * D + 16;     // bytes per fp16 row (conflict-free ldmatrix)
  static constexpr int kKV = kTile * kPitch;    // one tile of K or V as fp16 rows
  static constexpr int kStage = 2 * kTile * D;  // the next tile's K then V codes (int8)
  static constexpr int bytes(int warps) { return 16 * warps * kPitch + 2 * kKV + kStage; }
};

// The codes of keys k0..k0+63 into the staging area (zeros past Nk).
template <int D>
__device__ __forceinline__ void stage_tile(uint32_t st, const int8_t* kg, const int8_t* vg, int k0,
                                           int Nk) {
  constexpr int kChunks = kTile * D / 16;
  for (int v = threadIdx.x; v < 2 * kChunks; v += blockDim.x) {
    const int which = v / kChunks, rem = v % kChunks;
    const int key = rem / (D / 16), c16 = rem % (D / 16);
    const bool in = k0 + key < Nk;
    const int8_t* src = (which ? vg : kg) + (in ? static_cast<size_t>(k0 + key) * D + 16 * c16 : 0);
    cp_async16(st + 16 * v, src, in ? 16u : 0u);
  }
}

// Staged codes -> exact fp16 rows of K and V.
template <int D>
__device__ __forceinline__ void convert_tile(const uint8_t* st, uint8_t* sk, uint8_t* sv) {
  using SM = IntsmSmem<D>;
  constexpr int kChunks = kTile * D / 16;
  for (int v = threadIdx.x; v < 2 * kChunks; v += blockDim.x) {
    const int which = v / kChunks, rem = v % kChunks;
    const int key = rem / (D / 16), c16 = rem % (D / 16);
    const uint4 x = *reinterpret_cast<const uint4*>(st + 16 * v);
    uint32_t hv[8];
    codes4_to_f16x2(x.x, hv[0], hv[1]);
    codes4_to_f16x2(x.y, hv[2], hv[3]);
    codes4_to_f16x2(x.z, hv[4], hv[5]);
    codes4_to_f16x2(x.w, hv[6], hv[7]);
    uint8_t* dst = (which ? sv : sk) + key * SM::kPitch + c16 * 32;
    *reinterpret_cast<uint4*>(dst) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    *reinterpret_cast<uint4*>(dst + 16) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
  }
}

// One tile's softmax step for a lane's two rows (g and g + 8) from the exact
// fp32 scores S (the m16n8 accumulator layout): the new running max m'
// (quad-reduced), alpha = ShiftExp2(m - m'), the P codes Y =
// requant(ShiftExp2(S - m')) packed as the PV A fragments (the accumulator
// layout of 8 n-tiles is the A layout of 4 k-steps), and the lane's share of
// the row sums, quad-reduced.  Tail: keys at or past nvalid take no part.
template <bool Tail, bool Narrow>
__device__ __forceinline__ void softmax_tile(const float (&S)[8][4], int nvalid, int t4, const IntsmConst& c,
                                             float& m_lo, float& m_hi, int& al_lo, int& al_hi, int& sum_lo,
                                             int& sum_hi, uint32_t (&af)[4][4]) {
  float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const bool v0 = !Tail || 8 * j + 2 * t4 < nvalid, v1 = !Tail || 8 * j + 2 * t4 + 1 < nvalid;
    mx_lo = fmaxf(mx_lo, fmaxf(v0 ? S[j][0] : -INFINITY, v1 ? S[j][1] : -INFINITY));
    mx_hi = fmaxf(mx_hi, fmaxf(v0 ? S[j][2] : -INFINITY, v1 ? S[j][3] : -INFINITY));
  }
#pragma unroll
  for (int sh = 1; sh < 4; sh <<= 1) {
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, sh));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, sh));
  }
  const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
  // every score and the initial max are integers within 2^21 of zero, so all
  // differences below are exact and at most 2^22
  al_lo = shift_exp2_bits(__float_as_uint((mn_lo - m_lo) + kMagic), c);
  al_hi = shift_exp2_bits(__float_as_uint((mn_hi - m_hi) + kMagic), c);
  m_lo = mn_lo;
  m_hi = mn_hi;
  const float mb_lo = mn_lo + kMagic, mb_hi = mn_hi + kMagic;  // exact
  int s_lo = 0, s_hi = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    int Y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      Y[e] = requant<Narrow>(shift_exp2_bits(__float_as_uint(((e < 2) ? mb_lo : mb_hi) - S[j][e]), c), c);
      if (Tail && 8 * j + 2 * t4 + (e & 1) >= nvalid) Y[e] = 0;
    }
    s_lo += Y[0] + Y[1];
    s_hi += Y[2] + Y[3];
    af[j >> 1][2 * (j & 1)] = codes2_to_f16x2(Y[0], Y[1]);      // a0 / a2: row g
    af[j >> 1][2 * (j & 1) + 1] = codes2_to_f16x2(Y[2], Y[3]);  // a1 / a3: row g + 8
  }
#pragma unroll
  for (int sh = 1; sh < 4; sh <<= 1) {
    s_lo += __shfl_xor_sync(0xffffffffu, s_lo, sh);
    s_hi += __shfl_xor_sync(0xffffffffu, s_hi, sh);
  }
  sum_lo = s_lo;
  sum_hi = s_hi;
}

template <int D>
__global__ void __launch_bounds__(kMaxWarps * 32, D <= 64 ? 2 : 1) intsm_attn_kernel(const IntsmArgs a) {
  using SM = IntsmSmem<D>;
  constexpr int KS = D / 16;              // k-steps of QK^T
  constexpr int NTO = D / 8;              // PV n-tiles (8 channels each)
  constexpr int NTH = NTO < 8 ? NTO : 8;  // n-tiles per PV pass
  extern __shared__ __align__(16) uint8_t smem[];
  const int W = blockDim.x >> 5;
  uint8_t* sq = smem;
  uint8_t* sk = sq + 16 * W * SM::kPitch;
  uint8_t* sv = sk + SM::kKV;
  uint8_t* sst = sv + SM::kKV;
  pdl_trigger();
  pdl_wait();
  IntsmConst c;
  if (!intsm_constants(a.q_scale[0], a.k_scale[0], a.sm_scale, c)) {  // the same in every thread
    if (threadIdx.x == 0) atomicOr(a.err, kErrDomain);
    return;
  }
  const bool narrow = c.x0 < (1 << 23);  // P * M < 2^31
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int bh = blockIdx.y, b = bh / a.Hq, h = bh % a.Hq;
  const int bkv = b * a.Hkv + h / (a.Hq / a.Hkv);
  const int q0 = blockIdx.x * 16 * W;
  const int8_t* qg = a.q_codes + static_cast<size_t>(bh) * a.Nq * D;
  const int8_t* kg = a.k_codes + static_cast<size_t>(bkv) * a.Nk * D;
  const int8_t* vg = a.v_codes + static_cast<size_t>(bkv) * a.Nk * D;
  const uint32_t st_addr = smem_u32(sst);
  stage_tile<D>(st_addr, kg, vg, 0, a.Nk);
  // the CTA's Q rows as exact fp16 (zeros past Nq)
  for (int v = threadIdx.x; v < 16 * W * (D / 16); v += blockDim.x) {
    const int r = v / (D / 16), c16 = v % (D / 16);
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (q0 + r < a.Nq) x = *reinterpret_cast<const uint4*>(qg + static_cast<size_t>(q0 + r) * D + 16 * c16);
    uint32_t hv[8];
    codes4_to_f16x2(x.x, hv[0], hv[1]);
    codes4_to_f16x2(x.y, hv[2], hv[3]);
    codes4_to_f16x2(x.z, hv[4], hv[5]);
    codes4_to_f16x2(x.w, hv[6], hv[7]);
    uint8_t* dst = sq + r * SM::kPitch + c16 * 32;
    *reinterpret_cast<uint4*>(dst) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    *reinterpret_cast<uint4*>(dst + 16) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
  }
  cp_async_wait_all();
  __syncthreads();
  convert_tile<D>(sst, sk, sv);
  __syncthreads();

  float m_lo = static_cast<float>(kM0), m_hi = static_cast<float>(kM0);  // running max (integers)
  int l_lo = 0, l_hi = 0;
  int o[NTO][4];
#pragma unroll
  for (int n = 0; n < NTO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0;
  const bool active = q0 + 16 * warp < a.Nq;  // the warp has rows to compute
  // ldmatrix row addresses: lane l gives row l % 8 of matrix l / 8
  const int mrow = lane & 7, mat = lane >> 3;
  const uint32_t q_addr = smem_u32(sq) + (16 * warp + mrow + (mat & 1) * 8) * SM::kPitch + (mat >> 1) * 16;
  const uint32_t k_addr = smem_u32(sk) + (mrow + (mat >> 1) * 8) * SM::kPitch + (mat & 1) * 16;
  const uint32_t v_addr = smem_u32(sv) + (mrow + (mat & 1) * 8) * SM::kPitch + (mat >> 1) * 16;
  for (int k0 = 0; k0 < a.Nk; k0 += kTile) {
    const bool more = k0 + kTile < a.Nk;
    if (more) stage_tile<D>(st_addr, kg, vg, k0 + kTile, a.Nk);  // overlaps this tile's math
    if (active) {
      // ---- S = q.k for the warp's 16 rows and the tile's 64 keys (exact in fp32)
      float S[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(q_addr + ks * 32, a0, a1, a2, a3);
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(k_addr + 8 * j * SM::kPitch + ks * 32, b0, b1, b2, b3);
          mma_f16_16816(S[j], a0, a1, a2, a3, b0, b1);
          mma_f16_16816(S[j + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      // ---- the running max, alpha, and the P codes as the PV A fragments
      int al_lo, al_hi, sum_lo, sum_hi;
      uint32_t af[4][4];
      const int nvalid = a.Nk - k0;
      if (narrow) {
        if (nvalid >= kTile)
          softmax_tile<false, true>(S, kTile, t4, c, m_lo, m_hi, al_lo, al_hi, sum_lo, sum_hi, af);
        else
          softmax_tile<true, true>(S, nvalid, t4, c, m_lo, m_hi, al_lo, al_hi, sum_lo, sum_hi, af);
      } else {
        if (nvalid >= kTile)
          softmax_tile<false, false>(S, kTile, t4, c, m_lo, m_hi, al_lo, al_hi, sum_lo, sum_hi, af);
        else
          softmax_tile<true, false>(S, nvalid, t4, c, m_lo, m_hi, al_lo, al_hi, sum_lo, sum_hi, af);
      }
      // ---- l and O rescaled by alpha (ScaleRelease); the identity where the
      // max stayed (alpha = X0), nothing to do on the first tile (l = O = 0)
      if (k0 > 0 && __any_sync(0xffffffffu, (al_lo != c.x0) | (al_hi != c.x0))) {
        const int F_lo = rescale_factor(al_lo, c), F_hi = rescale_factor(al_hi, c);
        l_lo = scale_release(l_lo, al_lo, F_lo, c);
        l_hi = scale_release(l_hi, al_hi, F_hi, c);
#pragma unroll
        for (int n = 0; n < NTO; ++n) {
          o[n][0] = scale_release(o[n][0], al_lo, F_lo, c);
          o[n][1] = scale_release(o[n][1], al_lo, F_lo, c);
          o[n][2] = scale_release(o[n][2], al_hi, F_hi, c);
          o[n][3] = scale_release(o[n][3], al_hi, F_hi, c);
        }
      }
      l_lo += sum_lo;
      l_hi += sum_hi;
      // ---- O += Y.V, 64 channels per pass (exact: a tile's sums stay below 2^24)
#pragma unroll
      for (int hc = 0; hc < NTO / NTH; ++hc) {
        float op[NTH][4];
#pragma unroll
        for (int n = 0; n < NTH; ++n) op[n][0] = op[n][1] = op[n][2] = op[n][3] = 0.f;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
#pragma unroll
          for (int n = 0; n < NTH; n += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(v_addr + 16 * s * SM::kPitch + (hc * NTH + n) * 16, b0, b1, b2, b3);
            mma_f16_16816(op[n], af[s][0], af[s][1], af[s][2], af[s][3], b0, b1);
            mma_f16_16816(op[n + 1], af[s][0], af[s][1], af[s][2], af[s][3], b2, b3);
          }
        }
#pragma unroll
        for (int n = 0; n < NTH; ++n) {
#pragma unroll
          for (int e = 0; e < 4; ++e) o[hc * NTH + n][e] += f2i_small(op[n][e]);
        }
      }
    }
    if (more) {
      cp_async_wait_all();
      __syncthreads();  // this tile's fp16 rows are read; the next tile's codes have landed
      convert_tile<D>(sst, sk, sv);
      __syncthreads();
    }
  }
  if (!active) return;
  // ---- out = floor(O / l), int8 codes of V's scale
  const int r_lo = q0 + 16 * warp + g, r_hi = r_lo + 8;
  const int dl_lo = max(l_lo, 1), dl_hi = max(l_hi, 1);
  const uint32_t fi_lo = (dl_lo == 1) ? 0x7fffffffu : 0x80000000u / static_cast<uint32_t>(dl_lo);
  const uint32_t fi_hi = (dl_hi == 1) ? 0x7fffffffu : 0x80000000u / static_cast<uint32_t>(dl_hi);
#pragma unroll
  for (int n = 0; n < NTO; ++n) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int row = half ? r_hi : r_lo;
      if (row >= a.Nq) continue;
      const int dl = half ? dl_hi : dl_lo;
      const uint32_t fi = half ? fi_hi : fi_lo;
      const int v0 = min(127, max(-127, floor_div_recip(o[n][2 * half], dl, fi)));
      const int v1 = min(127, max(-127, floor_div_recip(o[n][2 * half + 1], dl, fi)));
      const uint16_t pair = static_cast<uint16_t>((v0 & 0xff) | ((v1 & 0xff) << 8));
      if (!QATTN_IN_BOUNDS(8 * n + 2 * t4 + 1 < D)) continue;
      *reinterpret_cast<uint16_t*>(a.out + (static_cast<size_t>(bh) * a.Nq + row) * D + 8 * n + 2 * t4) = pair;
    }
  }
}

template <int D>
cudaError_t launch_t(const IntsmArgs& a, cudaStream_t s) {
  // the 16-row blocks split evenly over the fewest CTAs of at most 8 warps
  const int nblk = (a.Nq + 15) / 16;
  const int per_head = (nblk + kMaxWarps - 1) / kMaxWarps;
  const int W = (nblk + per_head - 1) / per_head;
  cudaError_t e = cudaFuncSetAttribute(intsm_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       IntsmSmem<D>::bytes(kMaxWarps));
  if (e != cudaSuccess) return e;
  return launch_pdl(intsm_attn_kernel<D>, dim3(per_head, a.B * a.Hq), dim3(32 * W), IntsmSmem<D>::bytes(W),
                    s, a);
}

}  // namespace

unsigned int check_take_intsm() { return check_take_local(); }

cudaError_t launch_intsoftmax(int B, int Hq, int Hkv, int Nq, int Nk, int d, float sm_scale,
                              const int8_t* q_codes, const float* q_scale, const int8_t* k_codes,
                              const float* k_scale, const int8_t* v_codes, int8_t* out,
                              unsigned int* err, cudaStream_t s) {
  IntsmArgs a{B, Hq, Hkv, Nq, Nk, sm_scale, q_codes, q_scale, k_codes, k_scale, v_codes, out, err};
  if (d == 32) return launch_t<32>(a, s);
  if (d == 64) return launch_t<64>(a, s);
  return launch_t<128>(a, s);
}

}  // namespace qattn
