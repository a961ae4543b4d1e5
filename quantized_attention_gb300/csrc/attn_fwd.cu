// Fused quantized attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// Persistent kernel, one CTA per SM.  A work item is one (batch, head) and two
// consecutive 128-row query tiles (t0, t1); items are handed out heaviest
// first (causal) in a snake order over the CTAs.  Warp roles (12 warps):
//   warp 0      lane 0 issues every TMA load: the item's slot (its decoded
//               indices and scales, see ItemSlot), its two int8 Q tiles, a
//               ring of K stages and a ring of V^T stages;
//   warp 1      owns the 512 TMEM columns and issues the MMAs of tile t0 (the
//               whole warp runs the waits and forms the operand descriptors,
//               lane 0 issues the MMAs and commits);
//   warp 2      the same for tile t1;
//   warp 3      widens each item's int8 Q codes to exact fp16 in shared
//               memory (q_conv), running ahead of the softmax warps;
//   warps 4-7   softmax of tile t0, warps 8-11 softmax of tile t1 (one query
//               row per thread, row r = TMEM lane r), then the epilogue.
// TMEM: S_t at columns [128 t, 128 t + 128), O_t at [256 + 128 t, ...).
// Shared memory holds the e4m3 P_t tiles the PV MMAs read; the epilogue
// stages O through them for TMA stores.  K arrives as fp16 carriers.
// Per tile t and key block j:
//   softmax(t, j) loads S_t(j) from TMEM and at once releases it (s_free), so
//   the tile's MMA thread issues QK(t, j+1) -- S_t = Q_t . K_{j+1}^T,
//   kind::f16 on exact fp16 carriers of the int8 codes (every partial sum is
//   an integer below 2^21, so the fp32 accumulator holds it exactly) -- while
//   the softmax computes P; when P_t(j) is in shared memory and O_t rescaled
//   (p_full) it issues PV(t, j): O_t (+)= P_t . V8_j, kind::f8f6f4.
//   softmax(t, j+1) waits for PV(t, j) (pv_done) before it overwrites P_t or
//   rescales O_t.
// The two tiles run independently (their own softmax warps and MMA thread),
// sharing only the K / V stages, so the tensor core works on one tile while
// the other's softmax runs, and QK(t, j+1) overlaps softmax(t, j).
#include <cuda_bf16.h>

#include "qattn_check.cuh"
#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kBM = 128;  // query rows per tile (MMA M)
constexpr int kBN = 128;  // keys per block
constexpr int kThreads = 384;
constexpr float kLog2e = 1.44269502162933349609375f;  // fp32(log2 e)
constexpr float kLog2_448 = 8.8073549220576041f;      // log2(448)
constexpr float kLog2_127 = 6.9886846867721655f;      // log2(127)
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kNegInf = -__builtin_huge_valf();

// Shared-memory plan for head dim D.  Q and K are fp16 carriers stored as
// column blocks of [128 rows][row_bytes] in the TMA/UMMA swizzled K-major
// layout (128-byte rows and the 128B swizzle; 64-byte rows and the 64B
// swizzle for D = 32).  V is e4m3 transposed, [D rows][128 keys]; P is e4m3
// [128 rows][128 keys]; both 128-byte rows with the 128B swizzle.
// PQ: the int8 P ablation, whose P occupies two e4m3 planes per tile (see
// softmax_step); it buys that room with a 2-stage K ring for D >= 64.
template <int D, bool PQ = false>
struct Cfg {
  static constexpr int kColBlock = (D >= 64) ? 64 : D;  // fp16 elements per row of a block
  static constexpr int kRowBytes = kColBlock * 2;
  static constexpr int kNumColBlocks = D / kColBlock;
  static constexpr int kColBlockBytes = kBM * kRowBytes;
  static constexpr uint32_t kSwz = (kRowBytes == 128) ? kSwizzle128B : kSwizzle64B;
  static constexpr uint32_t kSBO = 8 * kRowBytes;  // bytes between 8-row groups
  static constexpr int kQS = (D == 128) ? 1 : 2;   // Q stages (each holds both tiles)
  static constexpr int kNK = (PQ && D >= 64) ? 2 : (D == 128) ? 3 : 4;  // K ring stages
  static constexpr int kNV = (D == 128) ? 2 : 4;   // V ring stages
  static constexpr int kQTileBytes = kBM * D * 2;
  static constexpr int kKBytes = kBN * D * 2;
  static constexpr int kVBytes = D * kBN;
  static constexpr int kPBytes = kBM * kBN;  // one e4m3 plane of P
  static constexpr int kPPlanes = PQ ? 2 : 1;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQS * 2 * kQTileBytes;
  static constexpr int kOffV = kOffK + kNK * kKBytes;
  static constexpr int kOffP = kOffV + kNV * kVBytes;
  // int8 Q codes as loaded: in the upper half of each fp16 Q tile for D = 128
  // (see convert_q_tile), in a region of their own for smaller D.
  static constexpr bool kQ8InPlace = (D == 128);
  static constexpr int kQ8Bytes = kBM * D;
  static constexpr int kOffQ8 = kOffP + 2 * kPPlanes * kPBytes;
  static constexpr int kOffBar = kOffQ8 + (kQ8InPlace ? 0 : kQS * 2 * kQ8Bytes);
  // Item slots (a ring of 2): the item's decoded indices, its Q scales per
  // tile, K's first block scale and V's D channel scales (see ItemSlot).
  static constexpr int kSlotBytes = 64 + 4 * D;
  static constexpr int kOffSlot = kOffBar + 512;
  static constexpr int kSmemBytes = kOffSlot + 2 * kSlotBytes + 1024;  // + alignment slack
  static_assert(kQTileBytes % 1024 == 0 && kKBytes % 1024 == 0 && kVBytes % 1024 == 0,
                "tile alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(!kQ8InPlace || (kColBlockBytes == kQTileBytes / 2 && kRowBytes == D),
                "in-place Q widening needs row r of the codes = row r of column block 1");
};

// Debug-kernel plan: one Q tile and one K tile.
template <int D>
struct DbgCfg {
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = Cfg<D>::kQTileBytes;
  static constexpr int kOffQ8 = kOffK + Cfg<D>::kKBytes;
  static constexpr int kOffBar = kOffQ8 + Cfg<D>::kQ8Bytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;
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

// The same with the operands' descriptors given (start address advanced by
// adding (offset >> 4) to the low word: addresses stay below 2^18).
template <int D>
__device__ __forceinline__ void issue_qk_d(uint32_t tmem_s, uint64_t dq, uint64_t dk) {
  using C = Cfg<D>;
  constexpr uint32_t idesc = make_idesc(kBM, kBN, 0, 0);
  constexpr int kStepsPerBlock = C::kRowBytes / 32;
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    const uint32_t off = (s / kStepsPerBlock) * C::kColBlockBytes + (s % kStepsPerBlock) * 32;
    mma_f16(tmem_s, dq + (off >> 4), dk + (off >> 4), idesc, s > 0 ? 1u : 0u);
  }
}
template <int D, bool PQ>
__device__ __forceinline__ void issue_pv_d(uint32_t tmem_o, uint64_t dp, uint64_t dv, bool acc) {
  constexpr uint32_t idesc = make_idesc(kBM, D, 0, 0);
#pragma unroll
  for (int pl = 0; pl < (PQ ? 2 : 1); ++pl) {
#pragma unroll
    for (int s = 0; s < kBN / 32; ++s) {
      mma_f8(tmem_o, dp + ((pl * kBM * kBN + s * 32) >> 4), dv + ((s * 32) >> 4), idesc,
             (acc || pl > 0 || s > 0) ? 1u : 0u);
    }
  }
}

// O (+)= P8 . V8 for one key block: 4 MMAs of K = 32 e4m3 per P plane (PQ:
// the high plane, then the low plane at sp + one plane, same V).
template <int D, bool PQ>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t sp, uint32_t sv, bool acc) {
  constexpr uint32_t idesc = make_idesc(kBM, D, 0, 0);  // E4M3 x E4M3 -> F32
#pragma unroll
  for (int pl = 0; pl < (PQ ? 2 : 1); ++pl) {
#pragma unroll
    for (int s = 0; s < kBN / 32; ++s) {
      mma_f8(tmem_o, smem_desc(sp + pl * kBM * kBN + s * 32, 1024, kSwizzle128B),
             smem_desc(sv + s * 32, 1024, kSwizzle128B), idesc,
             (acc || pl > 0 || s > 0) ? 1u : 0u);
    }
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

// int8 Q codes -> exact fp16 carriers.  The 128 calling threads each widen
// one row: thread r reads row r of the codes ([128 rows][D] bytes at `codes`)
// into registers, then writes it to the fp16 tile in the swizzled K-major
// layout the MMA descriptors expect.  With D = 128 the codes sit in the upper
// half of the fp16 tile itself: row r's codes then occupy exactly the bytes of
// row r of the second column block, which only thread r writes, after reading
// them -- so no thread needs to wait for another.  Chunks are visited starting
// at chunk r, so eight consecutive rows touch eight different bank groups.
template <int D>
__device__ __forceinline__ void convert_q_tile(uint32_t tile, uint32_t codes, int r) {
  using C = Cfg<D>;
  constexpr int kChunks = D / 16;  // 16-byte chunks of codes per row
  uint4 raw[kChunks];
  const uint32_t src = codes + r * D;
#pragma unroll
  for (int c = 0; c < kChunks; ++c) raw[c] = lds128(src + ((c + r) & (kChunks - 1)) * 16);
  const uint32_t sw = (C::kRowBytes == 128) ? (r & 7) : ((r >> 1) & 3);
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int cc = (c + r) & (kChunks - 1);
    uint32_t h[8];
    codes4_to_f16x2(raw[c].x, h[0], h[1]);
    codes4_to_f16x2(raw[c].y, h[2], h[3]);
    codes4_to_f16x2(raw[c].z, h[4], h[5]);
    codes4_to_f16x2(raw[c].w, h[6], h[7]);
    const int ch = cc * 16;                       // first channel of the chunk
    const uint32_t k0 = (ch % C::kColBlock) / 8;  // its 16-byte slot in the row
    const uint32_t row = tile + (ch / C::kColBlock) * C::kColBlockBytes + r * C::kRowBytes;
    sts128(row + ((k0 ^ sw) << 4), h[0], h[1], h[2], h[3]);
    sts128(row + (((k0 + 1) ^ sw) << 4), h[4], h[5], h[6], h[7]);
  }
}

__device__ __forceinline__ const float* scale_ptr(const float* s, int gran, int bh, int nblk, int blk) {
  if (gran == 0) return s;
  if (gran == 1) return s + bh;
  return s + static_cast<size_t>(bh) * nblk + blk;
}
// Checked build: whether (bh, blk) addresses one of the BH * nblk scales (the
// granule's array: 1, BH or BH * nblk floats).
__device__ __forceinline__ bool scale_in_range(int gran, int bh, int BH, int nblk, int blk) {
  return gran == 0 || (gran == 1 ? bh < BH : (bh < BH && blk < nblk));
}
__device__ __forceinline__ float scale_of(const float* s, int gran, int bh, int nblk, int blk) {
  return *scale_ptr(s, gran, bh, nblk, blk);
}

// Barrier slots.
enum {
  kBarQFull = 0,    // [2]  Q stage loaded
  kBarQEmpty = 2,   // [2]  Q stage free
  kBarKFull = 4,    // [4]  K stage loaded
  kBarKEmpty = 8,   // [4]  K stage free
  kBarVFull = 12,   // [4]  V stage loaded
  kBarVEmpty = 16,  // [4]  V stage free
  kBarSFull = 20,   // [2]  S_t ready (MMA commit)
  kBarSFree = 22,   // [2]  S_t loaded by the softmax (128 threads)
  kBarPFull = 24,   // [2]  P_t written, O_t rescaled (128 threads)
  kBarPVDone = 26,  // [2]  PV(t, j) finished (MMA commit)
  kBarDrain = 28,   // [2]  every MMA of the QK / PV issuer done (teardown)
  kBarQConv = 30,      // [2][2]  Q stage s, tile t widened to fp16 (the Q-widening warp)
  kBarSlotFull = 34,   // [2]  item slot written and its scales landed
  kBarSlotEmpty = 36,  // [2]  item slot read by every softmax thread (256 threads)
  kNumBars = 38
};

// Header of an item slot in shared memory; V's channel scales follow at byte
// 64.  The TMA thread writes the header and copies the scales in (cp.async for
// the three single floats, the bulk engine for V's), then arrives on the
// slot's full barrier, so the softmax warps neither decode the item nor wait
// for global loads of scales on their own critical path.
struct ItemSlot {
  int bq, bkv, h, q0, nb0, nb1;
  float sq[2];  // the Q scale of each tile's first row block (0 if the tile is empty)
  float sk0;    // the scale of K's first block
};

// One work item: (batch, head) x a pair of query tiles.
struct Item {
  int bq, bkv, h, q0;  // q0: first row of tile t0
  int nb[2];           // key blocks each tile visits (0: no visible key, or no row)
};

__device__ __forceinline__ Item decode_item(int w, const AttnArgs& a, int n_pairs) {
  const int BHq = a.B * a.Hq;
  Item it;
  const int pair = n_pairs - 1 - w / BHq;
  const int bq = w % BHq;
  const int b = bq / a.Hq;
  it.h = bq % a.Hq;
  it.bq = bq;
  it.bkv = b * a.Hkv + it.h / (a.Hq / a.Hkv);
  it.q0 = pair * 2 * kBM;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qs = it.q0 + t * kBM;
    int kend = 0;
    if (qs < a.Nq) {
      kend = a.Nk;
      if (a.causal) {
        const long long last = static_cast<long long>(a.pos0) + min(qs + kBM - 1, a.Nq - 1);
        kend = static_cast<int>(max(0LL, min(static_cast<long long>(a.Nk), last + 1)));
      }
    }
    it.nb[t] = (kend + kBN - 1) / kBN;
  }
  return it;
}

// k-th item of CTA c (snake order over rounds of G items); -1 if none.
__device__ __forceinline__ int item_index(int k, int c, int G, int n_items) {
  const int w = (k & 1) ? (k + 1) * G - 1 - c : k * G + c;
  return w < n_items ? w : -1;
}

// One softmax step for one query row and one key block.
//   s      the row's 128 scores: fp32 bit patterns of the integer scores, with
//          -inf for masked keys (without BIAS); with BIAS they are
//          overwritten by t = S c + bias log2e, and keys >= nvis are masked
//          (their bias is never read)
//   brow   BIAS: the row's bias for this block
//   c      the block's score scale (> 0 without BIAS, so -inf * c = -inf)
//   smax   without BIAS and with no masked key: the largest score of the
//          block (the TMEM read computed it); else NaN, and the maximum is
//          taken here
// Updates the running max m and sum l (l in units of 448 P), returns alpha
// and the e4m3 codes of 448 P packed four per word (key 4q + e in byte e).
// One body serves masked and unmasked blocks: a second, masked copy of this
// fully unrolled code would double the loop's instruction footprint.
template <bool BIAS, bool PQ>
__device__ __forceinline__ float softmax_step(uint32_t (&s)[kBN], float c, int nvis,
                                              const float* brow, float smax, float& m, float& l,
                                              uint32_t (&pw)[kBN / 4], uint32_t (&pw2)[kBN / 4]) {
  float mx = smax;
  if (BIAS || smax != smax) {
    if (BIAS) {  // only visible keys' bias is read: the row may end inside the block
#pragma unroll
      for (int k = 0; k < kBN; ++k) {
        float t = kNegInf;
        if (k < nvis) t = fmaf(__uint_as_float(s[k]), c, __fmul_rn(__ldg(brow + k), kLog2e));
        s[k] = __float_as_uint(t);
      }
    }
    float mx0 = kNegInf, mx1 = kNegInf, mx2 = kNegInf, mx3 = kNegInf;
#pragma unroll
    for (int k = 0; k < kBN; k += 8) {
      mx0 = fmax3(mx0, __uint_as_float(s[k]), __uint_as_float(s[k + 1]));
      mx1 = fmax3(mx1, __uint_as_float(s[k + 2]), __uint_as_float(s[k + 3]));
      mx2 = fmax3(mx2, __uint_as_float(s[k + 4]), __uint_as_float(s[k + 5]));
      mx3 = fmax3(mx3, __uint_as_float(s[k + 6]), __uint_as_float(s[k + 7]));
    }
    mx = fmax3(mx0, mx1, fmaxf(mx2, mx3));
  }
  float m_blk;
  if (BIAS) m_blk = mx;
  else m_blk = (mx == kNegInf) ? kNegInf : __fmul_rn(mx, c);
  const float m_new = fmaxf(m, m_blk);
  const bool dead = (m_new == kNegInf);
  const float alpha = dead ? 1.f : ex2_approx(m - m_new);
  const float kneg = dead ? 0.f : ((PQ ? kLog2_127 : kLog2_448) - m_new);
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                   make_float2(0.f, 0.f)};
#pragma unroll
  for (int k = 0; k < kBN; k += 4) {
    uint32_t half[2], half2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int kk = k + 2 * e;
      float2 x;
      if (BIAS) {
        x = fadd2(make_float2(__uint_as_float(s[kk]), __uint_as_float(s[kk + 1])),
                  make_float2(kneg, kneg));
      } else {
        x = ffma2(make_float2(__uint_as_float(s[kk]), __uint_as_float(s[kk + 1])),
                  make_float2(c, c), make_float2(kneg, kneg));
      }
      const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
      acc[(k / 2 + e) & 3] = fadd2(acc[(k / 2 + e) & 3], p);
      if (PQ) {  // code = rint(127 P) = 16 hi + lo; 16 hi and lo are exact e4m3 values
        const int ca = min(__float2int_rn(p.x), 127), cb = min(__float2int_rn(p.y), 127);
        half[e] = cvt_e4m3x2(static_cast<float>(ca & 0x70), static_cast<float>(cb & 0x70));
        half2[e] = cvt_e4m3x2(static_cast<float>(ca & 15), static_cast<float>(cb & 15));
      } else {
        half[e] = cvt_e4m3x2(p.x, p.y);
      }
    }
    pw[k / 4] = half[0] | (half[1] << 16);
    if (PQ) pw2[k / 4] = half2[0] | (half2[1] << 16);
  }
  const float2 a01 = fadd2(acc[0], acc[1]);
  const float2 a23 = fadd2(acc[2], acc[3]);
  const float2 tot = fadd2(a01, a23);
  l = fmaf(alpha, l, tot.x + tot.y);
  m = m_new;
  return alpha;
}

// softmax_step without BIAS or PQ for d <= 64, where a masked block (the
// ragged end of a short key sequence, e.g. ViT's 69-key second block) is a
// large share of the work.  Keys fall in four groups of 32: groups below
// nvis / 32 hold only visible keys and take their maximum from pmax (the TMEM
// read's maxima); the group holding the row's last visible key is masked
// (-inf) and maximized here; later groups hold no visible key and are skipped
// (P codes 0, nothing added to l).  Skipping is exact: their P would be 0 and
// adding 0 changes no sum.  The same arithmetic as softmax_step otherwise.
// (At d = 128 the per-group branches cost the block loop spills.)
__device__ __forceinline__ float softmax_step_groups(uint32_t (&s)[kBN], float c, int nvis,
                                                     const float (&pmax)[kBN / 32], bool masked,
                                                     float& m, float& l, uint32_t (&pw)[kBN / 4]) {
  constexpr int kG = kBN / 32;
  static_assert(kG == 4, "four 32-key groups per block");
  int ng = kG;  // groups with a visible key
  float mx;
  if (!masked) {
    mx = fmax3(pmax[0], pmax[1], fmaxf(pmax[2], pmax[3]));
  } else {
    ng = (nvis + 31) >> 5;
    const int nfull = nvis >> 5;
    mx = kNegInf;
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      if (g < nfull) {
        mx = fmaxf(mx, pmax[g]);
      } else if (g < ng) {  // the partial group
        float mx0 = kNegInf, mx1 = kNegInf;
#pragma unroll
        for (int k = 32 * g; k < 32 * g + 32; k += 4) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (k + e >= nvis) s[k + e] = 0xFF800000u;
          mx0 = fmax3(mx0, __uint_as_float(s[k]), __uint_as_float(s[k + 1]));
          mx1 = fmax3(mx1, __uint_as_float(s[k + 2]), __uint_as_float(s[k + 3]));
        }
        mx = fmax3(mx, mx0, mx1);
      }
    }
  }
  const float m_blk = (mx == kNegInf) ? kNegInf : __fmul_rn(mx, c);
  const float m_new = fmaxf(m, m_blk);
  const bool dead = (m_new == kNegInf);
  const float alpha = dead ? 1.f : ex2_approx(m - m_new);
  const float kneg = dead ? 0.f : (kLog2_448 - m_new);
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                   make_float2(0.f, 0.f)};
#pragma unroll
  for (int g = 0; g < kG; ++g) {
    if (g >= ng) {  // no visible key in the group
#pragma unroll
      for (int q = 8 * g; q < 8 * g + 8; ++q) pw[q] = 0u;
      continue;
    }
#pragma unroll
    for (int k = 32 * g; k < 32 * g + 32; k += 4) {
      uint32_t half[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kk = k + 2 * e;
        const float2 x = ffma2(make_float2(__uint_as_float(s[kk]), __uint_as_float(s[kk + 1])),
                               make_float2(c, c), make_float2(kneg, kneg));
        const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        acc[(k / 2 + e) & 3] = fadd2(acc[(k / 2 + e) & 3], p);
        half[e] = cvt_e4m3x2(p.x, p.y);
      }
      pw[k / 4] = half[0] | (half[1] << 16);
    }
  }
  const float2 a01 = fadd2(acc[0], acc[1]);
  const float2 a23 = fadd2(acc[2], acc[3]);
  const float2 tot = fadd2(a01, a23);
  l = fmaf(alpha, l, tot.x + tot.y);
  m = m_new;
  return alpha;
}

template <int D, bool BIAS, bool PQ>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const AttnArgs a, int n_items) {
  using C = Cfg<D, PQ>;
  extern __shared__ uint8_t smem_raw[];
  pdl_trigger();
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 8 * kNumBars + 4);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto sQ = [&](int qs, int t) { return base + C::kOffQ + (qs * 2 + t) * C::kQTileBytes; };
  auto sK = [&](int st) { return base + C::kOffK + st * C::kKBytes; };
  auto sV = [&](int st) { return base + C::kOffV + st * C::kVBytes; };
  auto sP = [&](int t) { return base + C::kOffP + t * C::kPPlanes * C::kPBytes; };
  auto sQ8 = [&](int qs, int t) {
    return C::kQ8InPlace ? sQ(qs, t) + C::kQTileBytes / 2
                         : base + C::kOffQ8 + (qs * 2 + t) * C::kQ8Bytes;
  };
  auto slot_hdr = [&](int sl) {
    return reinterpret_cast<ItemSlot*>(smem + C::kOffSlot + sl * C::kSlotBytes);
  };
  auto sSlot = [&](int sl) { return base + C::kOffSlot + sl * C::kSlotBytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int n_qt = (a.Nq + kBM - 1) / kBM;
  const int n_pairs = (n_qt + 1) / 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const bool softmax_side = (i >= kBarSFree && i < kBarSFree + 2) ||
                                (i >= kBarPFull && i < kBarPFull + 2);
      // Q, K and V stages are freed by both tiles' issuers.
      const bool shared_stage = (i >= kBarQEmpty && i < kBarQEmpty + 2) ||
                                (i >= kBarKEmpty && i < kBarKEmpty + 4) ||
                                (i >= kBarVEmpty && i < kBarVEmpty + 4);
      const bool slot_empty = i >= kBarSlotEmpty && i < kBarSlotEmpty + 2;
      mbar_init(bar(i), slot_empty ? 2 * kBM : softmax_side ? kBM : shared_stage ? 2 : 1);
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
  pdl_wait();  // the previous kernel's outputs (codes, scales, carriers) are visible

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA
      // Order per item: Q; then K runs one block ahead of V:
      // K0, K1, V0, K2, V1, ..., K(nb-1), V(nb-2), V(nb-1).
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int last_q[2] = {-1, -1}, last_k[4] = {-1, -1, -1, -1}, last_v[4] = {-1, -1, -1, -1};
      int last_slot[2] = {-1, -1};
      const int nqb = (a.Nq + kBM - 1) / kBM, nkb = (a.Nk + kBN - 1) / kBN;
      uint32_t kc = 0, vc = 0;
      int i = 0;
      bool ok = true;
      auto load_k = [&](int j, int bkv) -> bool {
        const int st = kc % C::kNK;
        if (kc >= static_cast<uint32_t>(C::kNK) &&
            !mbar_wait(bar(kBarKEmpty + st), ((kc / C::kNK) - 1) & 1, abort_flag, a.err, kErrTimeout))
          return false;
        (void)QATTN_IN_BOUNDS(j * kBN < a.Nk && bkv < a.B * a.Hkv);  // TMA coordinates
        mbar_arrive_expect_tx(bar(kBarKFull + st), C::kKBytes);
        tma_tile<D>(&tmK, sK(st), bar(kBarKFull + st), j * kBN, bkv);
        last_k[st] = static_cast<int>(kc++);
        return true;
      };
      auto load_v = [&](int j, int bkv) -> bool {
        const int st = vc % C::kNV;
        if (vc >= static_cast<uint32_t>(C::kNV) &&
            !mbar_wait(bar(kBarVEmpty + st), ((vc / C::kNV) - 1) & 1, abort_flag, a.err, kErrTimeout))
          return false;
        (void)QATTN_IN_BOUNDS(j * kBN < a.Nk && bkv < a.B * a.Hkv);  // TMA coordinates
        mbar_arrive_expect_tx(bar(kBarVFull + st), C::kVBytes);
        tma_load_3d(sV(st), &tmV, bar(kBarVFull + st), j * kBN, 0, bkv);
        last_v[st] = static_cast<int>(vc++);
        return true;
      };
      for (int k = 0; ok && k * G < n_items; ++k) {
        const int w = item_index(k, cta, G, n_items);
        if (w < 0) continue;
        const Item it = decode_item(w, a, n_pairs);
        {  // the item's slot: header, Q / K scales, V's channel scales
          const int sl = i & 1;
          if (i >= 2 && !(ok = mbar_wait(bar(kBarSlotEmpty + sl), ((i >> 1) - 1) & 1, abort_flag,
                                         a.err, kErrTimeout)))
            break;
          ItemSlot* hs = slot_hdr(sl);
          hs->bq = it.bq;
          hs->bkv = it.bkv;
          hs->h = it.h;
          hs->q0 = it.q0;
          hs->nb0 = it.nb[0];
          hs->nb1 = it.nb[1];
          for (int tt = 0; tt < 2; ++tt) {
            if (it.nb[tt] > 0 &&
                QATTN_IN_BOUNDS(scale_in_range(a.q_gran, it.bq, a.B * a.Hq, nqb, it.q0 / kBM + tt)))
              cp_async4(sSlot(sl) + offsetof(ItemSlot, sq) + 4 * tt,
                        scale_ptr(a.q_scales, a.q_gran, it.bq, nqb, it.q0 / kBM + tt));
            else
              hs->sq[tt] = 0.f;
          }
          if ((it.nb[0] > 0 || it.nb[1] > 0) &&
              QATTN_IN_BOUNDS(scale_in_range(a.k_gran, it.bkv, a.B * a.Hkv, nkb, 0)))
            cp_async4(sSlot(sl) + offsetof(ItemSlot, sk0), scale_ptr(a.k_scales, a.k_gran, it.bkv, nkb, 0));
          else
            hs->sk0 = 0.f;
          cp_async_mbar_arrive(bar(kBarSlotFull + sl));
          mbar_arrive_expect_tx(bar(kBarSlotFull + sl), 4 * D);
          if (QATTN_IN_BOUNDS(it.bkv < a.B * a.Hkv))  // (a skipped copy leaves the slot's wait to time out)
            bulk_g2s(sSlot(sl) + 64, a.v_scales + static_cast<size_t>(it.bkv) * D, 4 * D,
                     bar(kBarSlotFull + sl));
          last_slot[sl] = i;
        }
        const int qs = i % C::kQS;
        if (i >= C::kQS &&
            !(ok = mbar_wait(bar(kBarQEmpty + qs), ((i / C::kQS) - 1) & 1, abort_flag, a.err,
                             kErrTimeout)))
          break;
        (void)QATTN_IN_BOUNDS(it.bq < a.B * a.Hq && it.q0 < a.Nq);  // TMA coordinates
        mbar_arrive_expect_tx(bar(kBarQFull + qs), 2 * C::kQ8Bytes);  // int8 codes
        tma_load_3d(sQ8(qs, 0), &tmQ, bar(kBarQFull + qs), 0, it.q0, it.bq);
        tma_load_3d(sQ8(qs, 1), &tmQ, bar(kBarQFull + qs), 0, it.q0 + kBM, it.bq);
        last_q[qs] = i;
        const int nb = max(it.nb[0], it.nb[1]);
        if (nb > 0) ok = load_k(0, it.bkv);
        for (int j = 0; ok && j < nb; ++j) {
          if (j + 1 < nb && !(ok = load_k(j + 1, it.bkv))) break;
          ok = load_v(j, it.bkv);
        }
        ++i;
      }
      // Every load this thread issued lands before the CTA may exit.
      volatile int never = 0;
      for (int q = 0; q < C::kQS; ++q)
        if (last_q[q] >= 0)
          mbar_wait(bar(kBarQFull + q), (last_q[q] / C::kQS) & 1, &never, a.err, kErrTimeout);
      for (int st = 0; st < C::kNK; ++st)
        if (last_k[st] >= 0)
          mbar_wait(bar(kBarKFull + st), (last_k[st] / C::kNK) & 1, &never, a.err, kErrTimeout);
      for (int st = 0; st < C::kNV; ++st)
        if (last_v[st] >= 0)
          mbar_wait(bar(kBarVFull + st), (last_v[st] / C::kNV) & 1, &never, a.err, kErrTimeout);
      for (int sl = 0; sl < 2; ++sl)
        if (last_slot[sl] >= 0)
          mbar_wait(bar(kBarSlotFull + sl), (last_slot[sl] >> 1) & 1, &never, a.err, kErrTimeout);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ Q widening
    // Per item, as soon as its int8 Q codes land, the warp widens the rows of
    // each tile with keys to visit (lane l: rows l, l + 32, l + 64, l + 96)
    // and releases the tile's first QK (q_conv).  It runs ahead of the
    // softmax warps, so the next item's first QK is issued under this item's
    // last key block and epilogue.
    int i = 0;
    bool ok = true;
    for (int k = 0; ok && k * G < n_items; ++k) {
      const int w = item_index(k, cta, G, n_items);
      if (w < 0) continue;
      const Item it = decode_item(w, a, n_pairs);
      const int qs = i % C::kQS;
      if (it.nb[0] > 0 || it.nb[1] > 0) {
        ok = mbar_wait(bar(kBarQFull + qs), (i / C::kQS) & 1, abort_flag, a.err, kErrTimeout);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
      }
      // One q_conv phase per item and stage; a tile without keys is not
      // widened.  The barrier of stage s completes item i + kQS's phase only
      // after both issuers freed the stage from item i (q_empty), that is
      // after they waited for item i's phase: never two phases ahead.
      for (int t = 0; t < 2; ++t) {
        if (it.nb[t] > 0) {
#pragma unroll 1
          for (int rr = lane; rr < kBM; rr += 32) convert_q_tile<D>(sQ(qs, t), sQ8(qs, t), rr);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarQConv + 2 * qs + t));
      }
      ++i;
    }
    if (!ok && lane == 0) *abort_flag = 1;
  } else if (warp == 1 || warp == 2) {
    {
      // ------------------------------------------------------------ MMA
      // One issuing warp per query tile (warp 1: t0, warp 2: t1), so a tile
      // whose softmax runs ahead is never held back by the other.  Per item
      // it issues, in the order its softmax frees the inputs,
      //   QK(0), QK(1), PV(0), QK(2), PV(1), ..., PV(nb_t - 1)
      // where QK(b): S_t <- Q_t . K_b^T once K_b is loaded and softmax(t,
      // b-1) has loaded S_t (s_free), plus, for b = 0, once Q_t is widened;
      // PV(b): O_t (+)= P_t . V8_b once V_b is loaded and P_t(b) written
      // (p_full).  Each Q / K / V stage is freed by a commit from both issuers
      // (barrier count 2); a tile with fewer key blocks than its partner
      // still waits for and frees each remaining stage, in order, so neither
      // issuer can free a stage the other is still reading.
      const int t = warp - 1;
      uint32_t kvc = 0;          // K (and V) blocks of earlier items
      uint32_t nqk = 0, npv = 0;  // QKs / PVs issued for this tile
      int i = 0;
      bool ok = true;
      for (int k = 0; ok && k * G < n_items; ++k) {
        const int w = item_index(k, cta, G, n_items);
        if (w < 0) continue;
        const Item it = decode_item(w, a, n_pairs);
        const int qs = i % C::kQS;
        const int nb = max(it.nb[0], it.nb[1]);
        const int nbt = it.nb[t];
        if (nbt == 0) {  // nothing for this tile: free the item's Q stage
          if ((ok = mbar_wait(bar(kBarQFull + qs), (i / C::kQS) & 1, abort_flag, a.err, kErrTimeout)) && lane == 0)
            mma_commit(bar(kBarQEmpty + qs));
        }
        for (int b = 0; ok && b <= nb; ++b) {
          if (b < nb) {  // key block b
            const uint32_t kk = kvc + b;
            const int st = kk % C::kNK;
            if (!(ok = mbar_wait(bar(kBarKFull + st), (kk / C::kNK) & 1, abort_flag, a.err, kErrTimeout)))
              break;
            if (b < nbt) {
              if (nqk > 0 &&
                  !(ok = mbar_wait(bar(kBarSFree + t), (nqk - 1) & 1, abort_flag, a.err, kErrTimeout)))
                break;
              if (b == 0 &&  // the item's Q_t, widened by warp 3
                  !(ok = mbar_wait(bar(kBarQConv + 2 * qs + t), (i / C::kQS) & 1, abort_flag, a.err,
                                   kErrTimeout)))
                break;
              tc_fence_after();
              const uint64_t dq = smem_desc(sQ(qs, t), C::kSBO, C::kSwz), dk = smem_desc(sK(st), C::kSBO, C::kSwz);
              if (lane == 0) {
                issue_qk_d<D>(tmem + 128 * t, dq, dk);
                mma_commit(bar(kBarSFull + t));
              }
              ++nqk;
            }
            if (lane == 0) mma_commit(bar(kBarKEmpty + st));
            if (b == nbt - 1 && lane == 0) mma_commit(bar(kBarQEmpty + qs));  // the tile's last QK
          }
          if (b >= 1) {  // value block b - 1
            const uint32_t vv = kvc + b - 1;
            const int st = vv % C::kNV;
            if (!(ok = mbar_wait(bar(kBarVFull + st), (vv / C::kNV) & 1, abort_flag, a.err, kErrTimeout)))
              break;
            if (b - 1 < nbt) {
              if (!(ok = mbar_wait(bar(kBarPFull + t), npv & 1, abort_flag, a.err, kErrTimeout)))
                break;
              tc_fence_after();
              const uint64_t dp = smem_desc(sP(t), 1024, kSwizzle128B), dv = smem_desc(sV(st), 1024, kSwizzle128B);
              if (lane == 0) {
                issue_pv_d<D, PQ>(tmem + 256 + 128 * t, dp, dv, b > 1);
                mma_commit(bar(kBarPVDone + t));
              }
              ++npv;
            }
            if (lane == 0) mma_commit(bar(kBarVEmpty + st));
          }
        }
        kvc += nb;
        ++i;
      }
      // Every MMA this thread issued finishes before TMEM is freed.
      const int drain = kBarDrain + t;
      if (lane == 0) mma_commit(bar(drain));
      volatile int never = 0;
      mbar_wait(bar(drain), 0, &never, a.err, kErrTimeout);
      if (!ok && lane == 0) *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) / 4;  // tile of this warpgroup
    const int wq = warp & 3;       // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;  // row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + 128 * t, tO = tmem + 256 + 128 * t;
    const uint32_t prow = sP(t) + r * 128;
    const uint32_t sw = r & 7;
    const int nkb = (a.Nk + kBN - 1) / kBN;
    uint32_t sc = 0, pvc = 0;
    bool ok = true;
    int i = -1;  // items of this CTA so far
    for (int k = 0; ok && k * G < n_items; ++k) {
      const int w = item_index(k, cta, G, n_items);
      if (w < 0) continue;
      ++i;
      // the item as the TMA thread decoded it, with its scales (item slot)
      const int sl = i & 1;
      ok = mbar_wait(bar(kBarSlotFull + sl), (i >> 1) & 1, abort_flag, a.err, kErrTimeout);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const ItemSlot* hs = slot_hdr(sl);
      Item it;
      it.bq = hs->bq;
      it.bkv = hs->bkv;
      it.h = hs->h;
      it.q0 = hs->q0;
      it.nb[0] = hs->nb0;
      it.nb[1] = hs->nb1;
      const int q0t = it.q0 + t * kBM;
      const int qi = q0t + r;
      const int nbt = it.nb[t];
      if (nbt == 0) {  // no visible key for any row of this tile: output 0
        mbar_arrive(bar(kBarSlotEmpty + sl));
        const size_t row = static_cast<size_t>(it.bq) * a.Nq + qi;
        if (qi < a.Nq && QATTN_IN_BOUNDS(it.bq < a.B * a.Hq)) {
          for (int cidx = 0; cidx < D; ++cidx) {
            if (a.out_bf16)
              reinterpret_cast<__nv_bfloat16*>(a.out)[row * D + cidx] = __float2bfloat16(0.f);
            else
              reinterpret_cast<float*>(a.out)[row * D + cidx] = 0.f;
          }
          if (a.lse) a.lse[row] = kNegInf;
        }
        continue;
      }
      const float sq = hs->sq[t];
      float sk_next = hs->sk0;
      const int lim = a.causal ? min(a.Nk - 1, a.pos0 + qi) : a.Nk - 1;  // last visible key
      const int tile_lim = a.causal ? a.pos0 + q0t : a.Nk;  // blocks ending <= this need no causal mask
      const float* brow = nullptr;
      if (BIAS)
        brow = a.bias + static_cast<size_t>(it.h) * a.bias_head_stride +
               static_cast<size_t>(min(qi, a.Nq - 1)) * a.Nk;
      float m = kNegInf, l = 0.f;
      for (int j = 0; j < nbt; ++j) {
        const float sk = sk_next;
        if (j + 1 < nbt && QATTN_IN_BOUNDS(scale_in_range(a.k_gran, it.bkv, a.B * a.Hkv, nkb, j + 1)))
          sk_next = scale_of(a.k_scales, a.k_gran, it.bkv, nkb, j + 1);
        ok = mbar_wait(bar(kBarSFull + t), sc & 1, abort_flag, a.err, kErrTimeout);
        ++sc;
        if (!__all_sync(0xffffffffu, ok)) {  // keep the warp converged for tcgen05.ld
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s[kBN];
        float pmax[kBN / 32];  // the largest score of each 32-key group
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q)
          tmem_ld32_max(tS + lane_base + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[q * 32]),
                        pmax[q]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(kBarSFree + t));  // S_t may now be overwritten by the next QK
        float c = __fmul_rn(__fmul_rn(__fmul_rn(sq, sk), a.sm_scale), kLog2e);
        const int kbase = j * kBN;
        const bool need_mask = (kbase + kBN > a.Nk) || (kbase + kBN - 1 > tile_lim);
        const int nvis = need_mask ? max(0, min(kBN, lim - kbase + 1)) : kBN;
        constexpr bool kGroups = (D <= 64) && !BIAS && !PQ;  // softmax_step_groups
        if (!BIAS) {
          // Masked keys become -inf scores.  A zero (or subnormal) c would
          // turn them into NaN; c = FLT_MIN leaves every visible t = S c at
          // or within 2^-105 of the exact S c, so no P, alpha or l changes.
          c = fmaxf(c, 0x1p-126f);
          if (!kGroups && need_mask) {
#pragma unroll
            for (int k = 0; k < kBN; ++k)
              if (k >= nvis) s[k] = 0xFF800000u;
          }
        }
        uint32_t pw[kBN / 4], pw2[kBN / 4];
        const float* bk = BIAS ? brow + kbase : nullptr;
        float alpha;
        if constexpr (kGroups) {
          alpha = softmax_step_groups(s, c, nvis, pmax, need_mask, m, l, pw);
        } else {
          // the TMEM read's maxima serve unmasked blocks; masked keys are -inf
          // only after the read, so those blocks take the maximum themselves
          const float smax = (BIAS || need_mask) ? __int_as_float(0x7fc00000)
                                                 : fmax3(pmax[0], pmax[1], fmaxf(pmax[2], pmax[3]));
          alpha = softmax_step<BIAS, PQ>(s, c, nvis, bk, smax, m, l, pw, pw2);
        }
        if (j > 0) {  // PV(t, j-1) must be done with P_t and O_t
          ok = mbar_wait(bar(kBarPVDone + t), pvc & 1, abort_flag, a.err, kErrTimeout);
          ++pvc;
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (j == 0) {  // an earlier item's output store has read P_t's rows
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
        }
#pragma unroll
        for (int ch = 0; ch < kBN / 16; ++ch) {
          const uint32_t addr = prow + ((static_cast<uint32_t>(ch) ^ sw) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pw[4 * ch]),
                       "r"(pw[4 * ch + 1]), "r"(pw[4 * ch + 2]), "r"(pw[4 * ch + 3])
                       : "memory");
          if (PQ)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr + C::kPBytes),
                         "r"(pw2[4 * ch]), "r"(pw2[4 * ch + 1]), "r"(pw2[4 * ch + 2]),
                         "r"(pw2[4 * ch + 3])
                         : "memory");
        }
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // Rescale the O_t row: one TMEM round trip for all D columns.
          uint32_t o[D];
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc)
            tmem_ld32(tO + lane_base + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[cc * 32]));
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < D; q += 2) {
            const float2 v = fmul2(make_float2(__uint_as_float(o[q]), __uint_as_float(o[q + 1])),
                                   make_float2(alpha, alpha));
            o[q] = __float_as_uint(v.x);
            o[q + 1] = __float_as_uint(v.y);
          }
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc)
            tmem_st32(tO + lane_base + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[cc * 32]));
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + t));
      }
      if (!ok) break;
      ok = mbar_wait(bar(kBarPVDone + t), pvc & 1, abort_flag, a.err, kErrTimeout);  // last PV
      ++pvc;
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      // With the TMA store, the warp's 32 rows of O go out in 128-byte row
      // chunks (64 bf16 or 32 fp32 columns) staged in the warp's 32 rows of
      // P_t (free once the last PV is done; 128B swizzle as for P): one store
      // per warp and chunk writes whole lines, where a thread-per-row store
      // would touch 32 lines per instruction.  Rows past Nq are not written.
      const bool issue = lane == 0 && q0t + wq * 32 < a.Nq;
      const size_t row = static_cast<size_t>(it.bq) * a.Nq + qi;
      const int yo = q0t + wq * 32;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + lane_base + cc * 32, o);
        float svc[32];  // V's channel scales from the item slot (one broadcast read per 4)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 v4 = lds128(sSlot(sl) + 64 + (cc * 32 + 4 * q) * 4);
          svc[4 * q] = __uint_as_float(v4.x);
          svc[4 * q + 1] = __uint_as_float(v4.y);
          svc[4 * q + 2] = __uint_as_float(v4.z);
          svc[4 * q + 3] = __uint_as_float(v4.w);
        }
        tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = __uint_as_float(o[q]) * (svc[q] * inv_l);
        if (!a.out_bf16 || D >= 64) {  // TMA stores (all but bf16 rows of 64 bytes)
          const bool first_half = !a.out_bf16 || (cc & 1) == 0;  // a new 128-byte chunk starts
          if (first_half && cc > 0) {  // the previous chunk's store has read the stage
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
          if (a.out_bf16) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t wv[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 pr = __floats2bfloat162_rn(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
                wv[e] = *reinterpret_cast<const uint32_t*>(&pr);
              }
              const uint32_t c16 = static_cast<uint32_t>((cc & 1) * 4 + q);
              st_shared_v4(prow + ((c16 ^ sw) << 4), wv[0], wv[1], wv[2], wv[3]);
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_shared_v4(prow + ((static_cast<uint32_t>(q) ^ sw) << 4), __float_as_uint(v[4 * q]),
                           __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                           __float_as_uint(v[4 * q + 3]));
          }
          if (!a.out_bf16 || (cc & 1) == 1) {  // the 128-byte chunk is complete: store it
            fence_proxy_async_smem();
            __syncwarp();
            if (issue && QATTN_IN_BOUNDS(it.bq < a.B * a.Hq && yo < a.Nq)) {
              tma_store_3d(&tmO, prow - (static_cast<uint32_t>(lane) << 7), a.out_bf16 ? (cc / 2) * 64 : cc * 32, yo, it.bq);
              bulk_commit_group();
            }
          }
        } else if (qi < a.Nq && QATTN_IN_BOUNDS(it.bq < a.B * a.Hq)) {  // bf16 rows of 64 bytes (D = 32): direct stores
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + row * D + cc * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 pr = __floats2bfloat162_rn(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
              wv[e] = *reinterpret_cast<const uint32_t*>(&pr);
            }
            dst[q] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
      }
      mbar_arrive(bar(kBarSlotEmpty + sl));  // the slot's last read by this thread
      if (a.lse && qi < a.Nq && QATTN_IN_BOUNDS(it.bq < a.B * a.Hq))
        a.lse[row] = (l > 0.f) ? (m + __log2f(l) - (PQ ? kLog2_127 : kLog2_448)) * kLn2 : kNegInf;
    }
    if (lane == 0) bulk_wait_all();  // this warp's output stores are complete
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Debug: the int32 score tile of one (q tile, k tile) through issue_qk.
template <int D>
__global__ void __launch_bounds__(160, 1)
    qk_debug_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    int Hq, int Hkv, int Nq, int Nk, int32_t* __restrict__ S, unsigned int* err) {
  using C = DbgCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + C::kOffQ, sK = base + C::kOffK, sQ8 = base + C::kOffQ8;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 36);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x, qt = blockIdx.y, bq = blockIdx.z;
  const int b = bq / Hq, h = bq % Hq;
  const int bkv = b * Hkv + h / (Hq / Hkv);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);    // Q codes and K loaded
    mbar_init(smem_u32(&bars[1]), 1);    // S ready
    mbar_init(smem_u32(&bars[2]), 1);    // MMA drained
    mbar_init(smem_u32(&bars[3]), kBM);  // Q widened
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
      mbar_arrive_expect_tx(full, Cfg<D>::kQ8Bytes + Cfg<D>::kKBytes);
      tma_load_3d(sQ8, &tmQ, full, 0, qt * kBM, bq);
      tma_tile<D>(&tmK, sK, full, kt * kBN, bkv);
      volatile int never = 0;
      if (mbar_wait(full, 0, &never, err, kErrTimeout) &&
          mbar_wait(smem_u32(&bars[3]), 0, abort_flag, err, kErrTimeout)) {
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
    bool ok = mbar_wait(smem_u32(&bars[0]), 0, abort_flag, err, kErrTimeout);
    if (__all_sync(0xffffffffu, ok)) {
      convert_q_tile<D>(sQ, sQ8, r);
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars[3]));
      ok = mbar_wait(smem_u32(&bars[1]), 0, abort_flag, err, kErrTimeout);
    }
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

template <int D, bool BIAS, bool PQ = false>
cudaError_t launch_attn_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& to, const AttnArgs& a, cudaStream_t s) {
  const int smem = Cfg<D, PQ>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, BIAS, PQ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_qt = (a.Nq + kBM - 1) / kBM;
  const long long n_items = static_cast<long long>(a.B) * a.Hq * ((n_qt + 1) / 2);
  if (n_items <= 0) return cudaSuccess;
  const int grid = static_cast<int>(n_items < num_sms() ? n_items : num_sms());
  return launch_pdl(attn_fwd_kernel<D, BIAS, PQ>, dim3(grid), dim3(kThreads), smem, s, tq, tk, tv,
                    to, a, static_cast<int>(n_items));
}

template <int D>
cudaError_t launch_dbg_t(const CUtensorMap& tq, const CUtensorMap& tk, int B, int Hq, int Hkv,
                         int Nq, int Nk, int32_t* S, unsigned int* err, cudaStream_t s) {
  const int smem = DbgCfg<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(qk_debug_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((Nk + kBN - 1) / kBN, (Nq + kBM - 1) / kBM, B * Hq);
  qk_debug_kernel<D><<<grid, 160, smem, s>>>(tq, tk, Hq, Hkv, Nq, Nk, S, err);
  return cudaGetLastError();
}

}  // namespace

unsigned int check_take_attn_fwd() { return check_take_local(); }

cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, const AttnArgs& a, cudaStream_t s) {
  if (a.pv_int8) {  // the int8 P ablation (no bias)
    switch (a.d) {
      case 32: return launch_attn_t<32, false, true>(tq, tk, tv, to, a, s);
      case 64: return launch_attn_t<64, false, true>(tq, tk, tv, to, a, s);
      default: return launch_attn_t<128, false, true>(tq, tk, tv, to, a, s);
    }
  }
  const bool bias = a.bias != nullptr;
  switch (a.d) {
    case 32: return bias ? launch_attn_t<32, true>(tq, tk, tv, to, a, s) : launch_attn_t<32, false>(tq, tk, tv, to, a, s);
    case 64: return bias ? launch_attn_t<64, true>(tq, tk, tv, to, a, s) : launch_attn_t<64, false>(tq, tk, tv, to, a, s);
    default: return bias ? launch_attn_t<128, true>(tq, tk, tv, to, a, s) : launch_attn_t<128, false>(tq, tk, tv, to, a, s);
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
