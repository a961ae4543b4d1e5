// Decode on an int8 KV cache: a few query tokens per (batch, head) against a
// long cache of int8 K and V codes.  At batch one both attention products are
// matrix-vector products bound by the bytes of the cache ("int8 Flash
// Attention on RDNA4", "What actually changed for decode"), so this path
// streams the codes as stored -- K for the scores, V row-major for PV --
// split over key blocks so every SM reads.
//
// It computes the recipe of the prefill kernel on the same codes: blocks of
// 128 keys in ascending order, each block's P relative to the running max at
// that block.  The split over key blocks keeps that exactly: a chunk of blocks
// computes its scores, learns the running max before it from the chunk maxima
// of the earlier chunks (so each block's P = 2^(t - m_j) and its e4m3 code are
// the recipe's), and accumulates its share of O and l scaled to the running
// max at its last block; a second pass combines the chunks.  Rows are (query
// head of the KV group, token): r = g * Nq + i.
//
// The K and V tiles move by TMA (128-byte swizzle for d = 128, 64-byte for
// d = 64) through one ring of stages per CTA: a chunk's K tiles, then its V
// tiles, so the V reads start while the last scores are computed.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qattn_check.cuh"
#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kBlk = 128;  // keys per block (the recipe's key block)
constexpr int kCombineThreads = 256;
constexpr float kLog2e = 1.44269502162933349609375f;  // fp32(log2 e)
constexpr float kLog2_448 = 8.8073549220576041f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kNegInf = -__builtin_huge_valf();

__host__ __device__ constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Byte offset of 16-byte chunk c of key row r inside a TMA tile stored with
// the 128-byte (d = 128) or 64-byte (d = 64) swizzle: the chunk index is
// XORed with bits 7.. of the row's byte offset.
template <int D>
__device__ __forceinline__ int swz_chunk(int r, int c) {
  return r * D + 16 * (c ^ ((D == 128) ? (r & 7) : ((r >> 1) & 3)));
}

// Four int8 codes (byte e = code e) as exact fp32: the biased byte placed in
// the mantissa of 2^23, minus 2^23 + 128.
__device__ __forceinline__ void codes4_to_f32(uint32_t w, float2& c01, float2& c23) {
  const uint32_t x = w ^ 0x80808080u;
  const float2 bias = make_float2(-8388736.0f, -8388736.0f);
  c01 = fadd2(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540u)),
                          __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7541u))),
              bias);
  c23 = fadd2(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7542u)),
                          __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7543u))),
              bias);
}

// Four V codes of one key -> their e4m3 codes e4m3(fp32(code * inv_s)), byte e
// for channel e (the rounding qattn_quantize_v applies to the dequantized V).
__device__ __forceinline__ uint32_t v_codes_to_e4m3(uint32_t w, float4 iv) {
  float2 c01, c23;
  codes4_to_f32(w, c01, c23);
  const float2 x01 = fmul2(c01, make_float2(iv.x, iv.y));
  const float2 x23 = fmul2(c23, make_float2(iv.z, iv.w));
  return cvt_e4m3x2(x01.x, x01.y) | (cvt_e4m3x2(x23.x, x23.y) << 16);
}

// 4x4 byte transpose: y[e] byte i = x[i] byte e.
__device__ __forceinline__ void transpose4x4(const uint32_t (&x)[4], uint32_t (&y)[4]) {
  const uint32_t t0 = __byte_perm(x[0], x[1], 0x5140u), t1 = __byte_perm(x[0], x[1], 0x7362u);
  const uint32_t t2 = __byte_perm(x[2], x[3], 0x5140u), t3 = __byte_perm(x[2], x[3], 0x7362u);
  y[0] = __byte_perm(t0, t2, 0x5410u);
  y[1] = __byte_perm(t0, t2, 0x7632u);
  y[2] = __byte_perm(t1, t3, 0x5410u);
  y[3] = __byte_perm(t1, t3, 0x7632u);
}

// Q and K scales are written by the kernels just before this call (plain
// loads after the dependency wait, not the read-only path).
__device__ __forceinline__ float scale_at(const float* s, int gran, int bh, int nblk, int blk) {
  if (gran == 0) return s[0];
  if (gran == 1) return s[bh];
  return s[static_cast<size_t>(bh) * nblk + blk];
}

// Chunk records: one 64-bit word per (chunk, row) holding this call's tag in
// the high half and the chunk maximum's bits in the low half, so the value and
// its tag land in one store and need no fence (a fence here would wait for the
// tiles the CTA has in flight).
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Waits (bounded, like mbar_wait) until the record carries tag; returns its value.
__device__ __forceinline__ bool wait_record(const unsigned long long* rec, uint32_t tag, float& v,
                                            volatile int* abort_flag, unsigned int* err) {
  const unsigned long long t0 = cycles();
  for (uint32_t n = 0;; ++n) {
    const unsigned long long w = ld_relaxed_u64(rec);
    if (static_cast<uint32_t>(w >> 32) == tag) {
      v = __uint_as_float(static_cast<uint32_t>(w));
      return true;
    }
    if ((n & 63u) == 63u) {
      if (*abort_flag) return false;
      if (cycles() - t0 > kWaitTimeoutCycles) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
    __nanosleep(64);
  }
}

// ------------------------------------------------------------------ pass 1+2
// One kernel: CTA-units u = bkv * nch + c, each a chunk of bpc key blocks of
// one (batch, KV head), taken by persistent CTAs in increasing u.  A unit
// first computes its blocks' scores t = S c (the K tiles streamed through a
// ring of TMA stages) into shared memory and publishes its rows' chunk maximum
// (a record tagged with this call's epoch, release/acquire at GPU scope).  It
// then looks back at the records of the earlier chunks of its head -- the
// running max before the chunk -- and runs PV on the V tiles, which stream
// through the same ring right behind the K tiles.  A unit waits only on
// lower-numbered units, taken earlier by running CTAs, so the waits always
// end; each is bounded anyway.
//
// Scores: thread k owns key k of a block; exact int32 dot products on dp4a;
// the swizzled tile puts the 8 keys of a shared-memory phase in 8 bank groups
// and every lane reads the same Q chunk (a broadcast).
//
// PV: warp w multiplies P8 (rows x keys 32w..32w+31 of a block) by the
// block's V8 on the tensor cores (mma.m16n8k32, e4m3 x e4m3, fp32
// accumulation): every lane reads 16 (d = 128) or 8 (d = 64) channels of 8
// keys, rounds the codes to e4m3 as qattn_quantize_v does, and transposes 4x4
// byte groups into B fragments.  Keys of a 32-key step are permuted (fragment
// position 4t + i <-> key 8i + 2t, 16 + 4t + i <-> key 8i + 2t + 1) so the 8
// lanes of a shared-memory phase hit 8 bank groups; P8 uses the same
// permutation.  Lane group g = lane / 4 owns channels CPT*g .. CPT*g + CPT-1;
// n-tile (word w, byte e) column n is channel CPT*n + 4w + e.  Between blocks
// the accumulators are rescaled by 2^(m_prev - m_j), so the chunk's share ends
// relative to the running max at its last block.
constexpr int kThreads = 128;  // four warps
constexpr int kStages = 3;     // ring of K then V tiles

template <int D, int RMAX>
struct FusedSmem {
  static constexpr int kMaxBlocks = (RMAX <= 4) ? 8 : 4;  // key blocks per chunk, at most
  static constexpr int kChunkKeys = kMaxBlocks * kBlk;
  static constexpr int kTile = kBlk * D;  // 1024-byte multiple
  static constexpr int kRing = kStages * kTile;
  static constexpr int kQ = round_up(RMAX * D, 1024);           // the head's Q codes
  static constexpr int kT = RMAX * kChunkKeys * 4;               // t of the chunk (fp32)
  static constexpr int kP8 = kMaxBlocks * 4 * RMAX * 32;         // [block][step][row][32]
  static constexpr int kBytes = kRing + kQ + kT + kP8 + 1024;    // + alignment slack
  static constexpr int kRed = (kThreads / 32) * RMAX * D * 4;    // [warp][row][d]
  static_assert(kRed <= kRing, "reduction buffer does not fit");
};

template <int D, int RMAX>
__global__ void __launch_bounds__(kThreads)
    decode_fused_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecodeArgs a) {
  constexpr int NC = D / 16;    // 16-byte chunks per key row
  constexpr int CPT = D / 8;    // PV: channels per lane group
  constexpr int WPT = CPT / 4;  // their 32-bit words
  constexpr int NT = 4 * WPT;   // n-tiles a lane accumulates
  using SM = FusedSmem<D, RMAX>;
  constexpr int CK = SM::kChunkKeys;
  constexpr int MB = SM::kMaxBlocks;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = dsm_raw + ((1024u - (smem_u32(dsm_raw) & 1023u)) & 1023u);
  int8_t* qs = reinterpret_cast<int8_t*>(dsm + SM::kRing);
  float* tb = reinterpret_cast<float*>(dsm + SM::kRing + SM::kQ);
  uint8_t* p8 = dsm + SM::kRing + SM::kQ + SM::kT;
  float* red = reinterpret_cast<float*>(dsm);
  __shared__ float cf[MB][RMAX];    // score factor of block i, row r
  __shared__ float bmax[MB][RMAX];  // block maxima of the chunk
  __shared__ float mrun[MB][RMAX];  // running max at each block
  __shared__ float lblk[MB][RMAX];
  __shared__ float wmax[2][kThreads / 32][RMAX];
  __shared__ float mpoll[kThreads];
  __shared__ __align__(16) float inv_s[D];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ __align__(8) uint64_t qbar;
  __shared__ int abort_flag;
  __shared__ int unit_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.Hq / a.Hkv, R = G * a.Nq;
  const int nkb = (a.Nk + kBlk - 1) / kBlk, nqb = (a.Nq + kBlk - 1) / kBlk;
  const int units = a.B * a.Hkv * a.nch;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    mbar_init(smem_u32(&qbar), 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  // Units are taken in increasing order from a counter whose high half is this
  // call's tag: the first taker finds another value there (an earlier call's,
  // or whatever the workspace held) and claims the counter with a swap, so it
  // needs no reset.  A unit is only ever held by a running CTA, so the smallest
  // unfinished unit always has its predecessors done, whatever the residency
  // of the grid.  The kernels before this one in the stream do not touch it.
  const uint32_t tag = static_cast<uint32_t>(a.epoch);
  auto take = [&]() -> int {
    for (int attempt = 0; attempt < 64; ++attempt) {
      const unsigned long long cur = ld_relaxed_u64(a.ctr);
      if (static_cast<uint32_t>(cur >> 32) == tag)
        return static_cast<int>(static_cast<uint32_t>(atomicAdd(a.ctr, 1ull)));
      // another value (an earlier call's, or garbage): claim it for this call, unit 0
      if (atomicCAS(a.ctr, cur, (static_cast<unsigned long long>(tag) << 32) | 1ull) == cur) return 0;
    }
    atomicOr(a.err, kErrTimeout);  // unreachable while one call owns the workspace
    return units;
  };
  if (threadIdx.x == 0) unit_s = take();
  __syncthreads();
  pdl_wait();  // Q codes and scales come from the kernels before; the cache precedes this call
  uint32_t q0 = 0;  // ring items consumed by earlier units (every thread keeps the same count)
  uint32_t nu = 0;  // units done by this CTA (phase of qbar)
  for (int u = unit_s; u < units; ++nu) {
    const int bkv = u / a.nch, c = u % a.nch;
    const int b = bkv / a.Hkv, hkv = bkv % a.Hkv;
    const int j0 = c * a.bpc, nb = min(a.bpc, nkb - j0);
    const int items = 2 * nb;  // K tiles of the chunk, then its V tiles
    // thread 0: ring item i of this unit (K tile i, or V tile i - nb)
    auto issue = [&](int i) {
      const uint32_t q = q0 + i, slot = q % kStages;
      const uint32_t bar = smem_u32(&full[slot]);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kBlk * D));
      if (i < nb) tma_load_3d(smem_u32(dsm + slot * SM::kTile), &tmK, bar, 0, (j0 + i) * kBlk, bkv);
      else tma_load_3d(smem_u32(dsm + slot * SM::kTile), &tmV, bar, 0, (j0 + i - nb) * kBlk, bkv);
    };
    if (threadIdx.x == 0) {
      const uint32_t bar = smem_u32(&qbar);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(R * D));
      // rows r = g * Nq + i of the head are contiguous: heads hkv*G .. hkv*G+G-1
      bulk_g2s(smem_u32(qs), a.q_codes + (static_cast<size_t>(b) * a.Hq + hkv * G) * a.Nq * D,
               static_cast<uint32_t>(R * D), bar);
    }
    // score factors c = fp32(fp32(fp32(sq * sk) * sm_scale) * log2 e) and 448 / amax
    // (their loads go out ahead of the tiles)
    for (int idx = threadIdx.x; idx < nb * R; idx += kThreads) {
      const int i = idx / R, r = idx % R, g = r / a.Nq, ii = r % a.Nq;
      const float sq = scale_at(a.q_scales, a.q_gran, b * a.Hq + hkv * G + g, nqb, ii / kBlk);
      const float sk = scale_at(a.k_scales, a.k_gran, bkv, nkb, j0 + i);
      cf[i][r] = __fmul_rn(__fmul_rn(__fmul_rn(sq, sk), a.sm_scale), kLog2e);
    }
    for (int cc = threadIdx.x; cc < D; cc += kThreads) {
      const float am = __ldg(a.v_code_amax + static_cast<size_t>(bkv) * D + cc);
      inv_s[cc] = (am > 0.f) ? __fdiv_rn(448.0f, am) : 0.f;
    }
    if (threadIdx.x == 0)
      for (int i = 0; i < min(kStages, items); ++i) issue(i);
    __syncthreads();
    if (!mbar_wait(smem_u32(&qbar), nu & 1, &abort_flag, a.err, kErrTimeout)) return;
    // ---- scores of the chunk's blocks
    const int k = threadIdx.x;
    for (int i = 0; i < nb; ++i) {
      const uint32_t q = q0 + i;
      if (!mbar_wait(smem_u32(&full[q % kStages]), (q / kStages) & 1, &abort_flag, a.err,
                     kErrTimeout))
        return;
      const int8_t* ks = reinterpret_cast<const int8_t*>(dsm + (q % kStages) * SM::kTile);
      int acc[RMAX];
#pragma unroll
      for (int r = 0; r < RMAX; ++r) acc[r] = 0;
#pragma unroll
      for (int cc = 0; cc < NC; ++cc) {
        const uint4 kw = *reinterpret_cast<const uint4*>(ks + swz_chunk<D>(k, cc));
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          if (r < R) {
            const uint4 qw = *reinterpret_cast<const uint4*>(qs + r * D + cc * 16);
            acc[r] = __dp4a(static_cast<int>(kw.x), static_cast<int>(qw.x), acc[r]);
            acc[r] = __dp4a(static_cast<int>(kw.y), static_cast<int>(qw.y), acc[r]);
            acc[r] = __dp4a(static_cast<int>(kw.z), static_cast<int>(qw.z), acc[r]);
            acc[r] = __dp4a(static_cast<int>(kw.w), static_cast<int>(qw.w), acc[r]);
          }
        }
      }
      const int key = (j0 + i) * kBlk + k;
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        if (r < R) {
          const int ii = r % a.Nq;
          const bool vis = key < a.Nk && (!a.causal || key <= a.pos0 + ii);
          const float t = vis ? __fmul_rn(static_cast<float>(acc[r]), cf[i][r]) : kNegInf;
          tb[r * CK + i * kBlk + k] = t;
          float mx = t;
#pragma unroll
          for (int sh = 16; sh > 0; sh >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
          if (lane == 0) wmax[i & 1][warp][r] = mx;
        }
      }
      __syncthreads();  // the tile is read; the block's warp maxima are in
      if (threadIdx.x == 0 && i + kStages < items) issue(i + kStages);
      if (threadIdx.x < R) {
        const int r = threadIdx.x;
        bmax[i][r] = fmaxf(fmaxf(wmax[i & 1][0][r], wmax[i & 1][1][r]),
                           fmaxf(wmax[i & 1][2][r], wmax[i & 1][3][r]));
      }
    }
    __syncthreads();
    // ---- publish the chunk's maxima, then look back at the earlier chunks'
    const size_t rec0 = static_cast<size_t>(bkv) * a.nch;
    if (threadIdx.x < R) {
      const int r = threadIdx.x;
      float m = kNegInf;
      for (int i = 0; i < nb; ++i) m = fmaxf(m, bmax[i][r]);
      st_relaxed_u64(a.rec + (rec0 + c) * R + r,
                     (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(m));
    }
    // warps 1-3 poll: thread 32 + p * R + r reads row r of chunks p, p + pt, ...
    const int pt = (kThreads - 32) / R;
    const int pi = static_cast<int>(threadIdx.x) - 32;
    float mb = kNegInf;
    if (pi >= 0 && pi < pt * R) {
      const int r = pi % R;
      for (int cp = pi / R; cp < c; cp += pt) {
        float v;
        if (!wait_record(a.rec + (rec0 + cp) * R + r, tag, v, &abort_flag, a.err)) break;
        mb = fmaxf(mb, v);
      }
    }
    mpoll[threadIdx.x] = mb;
    __syncthreads();
    if (abort_flag) return;  // a look-back wait ran out (every thread sees it here)
    if (threadIdx.x < R) {
      const int r = threadIdx.x;
      float m = kNegInf;
      for (int p = 0; p < pt; ++p) m = fmaxf(m, mpoll[32 + p * R + r]);
      for (int i = 0; i < nb; ++i) {
        m = fmaxf(m, bmax[i][r]);
        mrun[i][r] = m;
      }
    }
    __syncthreads();
    // ---- P8 = e4m3(448 P), P = 2^(t - m_j), in fragment order; the block's
    // sum of 448 P (unquantized).  One warp per row; lane = key within a step.
    {
      const int f = (lane & 1) ? (16 + 4 * ((lane >> 1) & 3) + (lane >> 3))
                               : (4 * ((lane >> 1) & 3) + (lane >> 3));
      for (int r = warp; r < R; r += kThreads / 32) {
        const float* tr = tb + r * CK;
        for (int i = 0; i < nb; ++i) {
          const float mj = mrun[i][r];
          const float kneg = (mj == kNegInf) ? 0.f : (kLog2_448 - mj);
          float sum = 0.f;
#pragma unroll
          for (int st = 0; st < 4; ++st) {
            const float p = ex2_approx(__fadd_rn(tr[i * kBlk + 32 * st + lane], kneg));
            sum += p;
            p8[((i * 4 + st) * RMAX + r) * 32 + f] = static_cast<uint8_t>(cvt_e4m3x2(p, 0.f) & 0xFFu);
          }
#pragma unroll
          for (int sh = 16; sh > 0; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
          if (lane == 0) lblk[i][r] = sum;
        }
      }
    }
    __syncthreads();
    // ---- PV on the V tiles
    const int g = lane >> 2, t4 = lane & 3;
    const bool row_lo = g < R, row_hi = (RMAX > 8) && (g + 8 < R);
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    for (int i = 0; i < nb; ++i) {
      const uint32_t q = q0 + nb + i;
      if (!mbar_wait(smem_u32(&full[q % kStages]), (q / kStages) & 1, &abort_flag, a.err,
                     kErrTimeout))
        return;
      if (i > 0) {  // rescale to this block's running max (skipped while it holds)
        const float f0 =
            (row_lo && mrun[i][g] != kNegInf) ? ex2_approx(mrun[i - 1][g] - mrun[i][g]) : 1.f;
        const float f1 = (row_hi && mrun[i][g + 8] != kNegInf)
                             ? ex2_approx(mrun[i - 1][g + 8] - mrun[i][g + 8])
                             : 1.f;
        if (!__all_sync(0xffffffffu, f0 == 1.f && f1 == 1.f)) {
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            acc[n][0] *= f0;
            acc[n][1] *= f0;
            acc[n][2] *= f1;
            acc[n][3] *= f1;
          }
        }
      }
      const uint8_t* pa = p8 + ((i * 4 + warp) * RMAX) * 32;
      const uint32_t a0 = row_lo ? *reinterpret_cast<const uint32_t*>(pa + g * 32 + 4 * t4) : 0u;
      const uint32_t a2 = row_lo ? *reinterpret_cast<const uint32_t*>(pa + g * 32 + 16 + 4 * t4) : 0u;
      const uint32_t a1 =
          row_hi ? *reinterpret_cast<const uint32_t*>(pa + (g + 8) * 32 + 4 * t4) : 0u;
      const uint32_t a3 =
          row_hi ? *reinterpret_cast<const uint32_t*>(pa + (g + 8) * 32 + 16 + 4 * t4) : 0u;
      const uint8_t* vs = dsm + (q % kStages) * SM::kTile;
      uint32_t raw[8][WPT];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
          const int row = 32 * warp + 8 * ii + 2 * t4 + h;
          const uint8_t* src = vs + swz_chunk<D>(row, (CPT * g) >> 4) + ((CPT * g) & 15);
          if constexpr (WPT == 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(src);
            raw[4 * h + ii][0] = v.x;
            raw[4 * h + ii][1] = v.y;
            raw[4 * h + ii][2] = v.z;
            raw[4 * h + ii][3] = v.w;
          } else {
            const uint2 v = *reinterpret_cast<const uint2*>(src);
            raw[4 * h + ii][0] = v.x;
            raw[4 * h + ii][1] = v.y;
          }
        }
      }
#pragma unroll
      for (int w = 0; w < WPT; ++w) {
        const float4 iv = *reinterpret_cast<const float4*>(inv_s + CPT * g + 4 * w);
        uint32_t e0[4], e1[4], b0[4], b1[4];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
          e0[ii] = v_codes_to_e4m3(raw[ii][w], iv);
          e1[ii] = v_codes_to_e4m3(raw[4 + ii][w], iv);
        }
        transpose4x4(e0, b0);
        transpose4x4(e1, b1);
#pragma unroll
        for (int e = 0; e < 4; ++e) mma_e4m3_16832(acc[4 * w + e], a0, a1, a2, a3, b0[e], b1[e]);
      }
      __syncthreads();  // the tile is read
      if (threadIdx.x == 0 && nb + i + kStages < items) issue(nb + i + kStages);
    }
    q0 += items;
    // ---- reduce the four warps' shares; write the chunk's O share, l and m
#pragma unroll
    for (int w = 0; w < WPT; ++w) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int ch = CPT * (2 * t4 + cc) + 4 * w + e;
          if (row_lo) red[(warp * RMAX + g) * D + ch] = acc[4 * w + e][cc];
          if (row_hi) red[(warp * RMAX + g + 8) * D + ch] = acc[4 * w + e][2 + cc];
        }
      }
    }
    __syncthreads();
    const size_t pbase = (rec0 + c) * R;
    for (int idx = threadIdx.x; idx < R * D; idx += kThreads) {
      const int r = idx / D, ch = idx % D;
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) sum += red[(w * RMAX + r) * D + ch];
      a.part_o[(pbase + r) * D + ch] = sum;
    }
    if (threadIdx.x < R) {
      const int r = threadIdx.x;
      const float mend = mrun[nb - 1][r];
      float l = 0.f;
      if (mend != kNegInf)
        for (int i = 0; i < nb; ++i) l += lblk[i][r] * ex2_approx(mrun[i][r] - mend);
      a.part_l[pbase + r] = l;
      a.part_m[pbase + r] = mend;
    }
    // the next unit only now: taken earlier, a fast CTA would take units from
    // CTAs that have not started their first one yet.  With no more units
    // than CTAs, the first takes got them all.
    if (threadIdx.x == 0) unit_s = (units > static_cast<int>(gridDim.x)) ? take() : units;
    __syncthreads();  // red (the ring) and the unit's shared state are free again
    u = unit_s;
  }
  pdl_trigger();  // after every wait of this CTA: the combine pass may take the SM
}

// ------------------------------------------------------------------ combine
// One CTA per (row, batch * KV head).  Thread (chunk group cg, channel word
// c4) loads chunks cg, cg + CG, ... (their m, l and O slice in one batch),
// then scales them to the final max and the groups are summed.
template <int D>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const DecodeArgs a,
                                                                        int nchunks) {
  constexpr int TPC = D / 4;                 // threads per chunk row
  constexpr int CG = kCombineThreads / TPC;  // chunk groups
  constexpr int U = 8;                       // chunks per thread in one batch
  __shared__ float wm[kCombineThreads / 32];
  __shared__ __align__(16) float red[CG][D];
  __shared__ float redl[CG];
  const int r = blockIdx.x, bkv = blockIdx.y;
  const int b = bkv / a.Hkv, hkv = bkv % a.Hkv;
  const int G = a.Hq / a.Hkv, R = G * a.Nq;
  // V scale s_v = fp32(fp32(chan * amax) / 448), as qattn_quantize_v writes it; the
  // cache header precedes this call and the scores/PV pass released this grid
  // only after all its waits, so it is read before the dependency wait
  float sv = 0.f;
  if (threadIdx.x < D) {
    const size_t vc = static_cast<size_t>(bkv) * D + threadIdx.x;
    sv = __fdiv_rn(__fmul_rn(__ldg(a.v_chan_scale + vc), __ldg(a.v_code_amax + vc)), 448.0f);
  }
  pdl_wait();
  pdl_trigger();
  const size_t p0 = static_cast<size_t>(bkv) * nchunks * R + r;  // chunk c: p0 + c * R
  const int c4 = threadIdx.x % TPC, cg = threadIdx.x / TPC;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f, mf = kNegInf;
  for (int cb = cg; cb < nchunks; cb += U * CG) {
    float mc[U], lc[U];
    float4 oc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = cb + u * CG;
      const size_t pi = p0 + static_cast<size_t>(c) * R;
      const bool in = c < nchunks;
      mc[u] = in ? a.part_m[pi] : kNegInf;
      lc[u] = in ? a.part_l[pi] : 0.f;
      oc[u] = in ? *reinterpret_cast<const float4*>(a.part_o + pi * D + 4 * c4)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // the batch's max, then everything so far rescaled to it (online, in the
    // order of the recipe's combination: weights 2^(m_c - m_final))
    float mx = mf;
#pragma unroll
    for (int u = 0; u < U; ++u) mx = fmaxf(mx, mc[u]);
    if (mx != kNegInf) {
      const float f = (mf == kNegInf) ? 0.f : ex2_approx(mf - mx);
      l *= f;
      o.x *= f;
      o.y *= f;
      o.z *= f;
      o.w *= f;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float wgt = (mc[u] == kNegInf) ? 0.f : ex2_approx(mc[u] - mx);
        l = fmaf(wgt, lc[u], l);
        o.x = fmaf(wgt, oc[u].x, o.x);
        o.y = fmaf(wgt, oc[u].y, o.y);
        o.z = fmaf(wgt, oc[u].z, o.z);
        o.w = fmaf(wgt, oc[u].w, o.w);
      }
      mf = mx;
    }
  }
  // the groups' maxima -> the final max; each group's sums rescaled to it
  float gm = mf;
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, sh));
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = gm;
  __syncthreads();
  float mfin = wm[0];
#pragma unroll
  for (int w = 1; w < kCombineThreads / 32; ++w) mfin = fmaxf(mfin, wm[w]);
  const float f = (mf == kNegInf) ? 0.f : ex2_approx(mf - mfin);
  *reinterpret_cast<float4*>(&red[cg][4 * c4]) = make_float4(o.x * f, o.y * f, o.z * f, o.w * f);
  if (c4 == 0) redl[cg] = l * f;
  __syncthreads();
  const int g = r / a.Nq, i = r % a.Nq;
  const size_t row = (static_cast<size_t>(b) * a.Hq + hkv * G + g) * a.Nq + i;
  float lt = 0.f;
#pragma unroll
  for (int g2 = 0; g2 < CG; ++g2) lt += redl[g2];
  if (threadIdx.x < D && QATTN_IN_BOUNDS(b < a.B && hkv * G + g < a.Hq && i < a.Nq)) {
    const int c = threadIdx.x;
    float s = 0.f;
#pragma unroll
    for (int g2 = 0; g2 < CG; ++g2) s += red[g2][c];
    const float out = (lt > 0.f) ? s * (sv * (1.f / lt)) : 0.f;
    if (a.out_bf16) reinterpret_cast<__nv_bfloat16*>(a.out)[row * D + c] = __float2bfloat16(out);
    else reinterpret_cast<float*>(a.out)[row * D + c] = out;
  }
  if (threadIdx.x == 0 && a.lse)
    a.lse[row] = (lt > 0.f) ? (mfin + __log2f(lt) - kLog2_448) * kLn2 : kNegInf;
}

// ------------------------------------------------------------------ cache append
// One thread per (batch * KV head, channel), the T new tokens in order: a
// token's K is quantized against the header's running mean of the tokens
// before it, then the mean moves (the lag of one token the ZINC post
// describes); V codes raise the header's max |code|.  All steps are single
// IEEE fp32 operations, so the result is exact.
__global__ void kv_append_kernel(const uint16_t* K_new, const uint16_t* V_new, int BHd, int d,
                                 int T, int pos, long long cap, const float* k_chan_scale,
                                 const float* v_chan_scale, float* k_mean, float* v_code_amax,
                                 int8_t* k_codes, int8_t* v_codes) {
  pdl_trigger();
  pdl_wait();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= BHd) return;
  const int bh = idx / d, c = idx % d;
  float mu = k_mean[idx], am = v_code_amax[idx];
  const float sk = k_chan_scale[idx], sv = v_chan_scale[idx];
  for (int t = 0; t < T; ++t) {
    const size_t in = (static_cast<size_t>(bh) * T + t) * d + c;
    const float k = bf16_bits_to_f32(K_new[in]), v = bf16_bits_to_f32(V_new[in]);
    const int n = pos + t;
    const float diff = __fsub_rn(k, mu);
    const float qk = fminf(fmaxf(rintf(__fdiv_rn(diff, sk)), -127.f), 127.f);
    mu = __fadd_rn(mu, __fdiv_rn(diff, static_cast<float>(n + 1)));
    const float qv = fminf(fmaxf(rintf(__fdiv_rn(v, sv)), -127.f), 127.f);
    am = fmaxf(am, fabsf(qv));
    const size_t out = (static_cast<size_t>(bh) * cap + n) * d + c;
    k_codes[out] = static_cast<int8_t>(qk);
    v_codes[out] = static_cast<int8_t>(qv);
  }
  k_mean[idx] = mu;
  v_code_amax[idx] = am;
}

// CTAs of a kernel resident per SM.  Callers cache it: it depends only on the
// kernel and the device model.
template <typename Kernel>
int ctas_per_sm(Kernel kernel, int threads, int smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
      n < 1)
    n = 1;
  return n;
}

template <int D, int RMAX>
cudaError_t launch_decode_r(const CUtensorMap& tk, const CUtensorMap& tv, DecodeArgs a,
                            cudaStream_t s) {
  using SM = FusedSmem<D, RMAX>;
  const int BHkv = a.B * a.Hkv;
  const int nkb = (a.Nk + kBlk - 1) / kBlk;
  const int total = nkb * BHkv;
  cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel<D, RMAX>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
  if (e != cudaSuccess) return e;
  static const int occ = ctas_per_sm(decode_fused_kernel<D, RMAX>, kThreads, SM::kBytes);
  const int slots = num_sms() * occ;
  // chunks of about total / slots blocks (at most kMaxBlocks), one per resident CTA
  a.bpc = max(1, min(SM::kMaxBlocks, (total + slots - 1) / slots));
  a.nch = (nkb + a.bpc - 1) / a.bpc;
  const int units = a.nch * BHkv;
  e = launch_pdl(decode_fused_kernel<D, RMAX>, dim3(min(units, slots)), dim3(kThreads),
                 SM::kBytes, s, tk, tv, a);
  if (e != cudaSuccess) return e;
  const int R = (a.Hq / a.Hkv) * a.Nq;
  return launch_pdl(decode_combine_kernel<D>, dim3(R, BHkv), dim3(kCombineThreads), 0, s, a,
                    a.nch);
}

}  // namespace

unsigned int check_take_decode() { return check_take_local(); }

// Workspace, sized for the most chunks (one block each) so the layout does not
// depend on the GPU: the unit counter (64-bit), chunk shares O
// [B*Hkv][chunks][R][d], their l and m [B*Hkv][chunks][R], and the tagged
// chunk maxima [B*Hkv][chunks][R] (64-bit).
size_t decode_ws_bytes(long long B, long long Hq, long long Hkv, long long Nq, long long Nk,
                       long long d) {
  const long long R = (Hq / Hkv) * Nq;
  const long long nkb = (Nk + kBlk - 1) / kBlk;
  const long long BH = B * Hkv;
  auto a256 = [](long long x) { return static_cast<size_t>((x + 255) / 256 * 256); };
  return a256(8) +                     // unit counter
         a256(BH * nkb * R * d * 4) +  // chunk O
         2 * a256(BH * nkb * R * 4) +  // chunk l, m
         a256(BH * nkb * R * 8);       // chunk maxima records
}

cudaError_t launch_kv_append(const uint16_t* K_new, const uint16_t* V_new, int BH, int d, int T,
                             int pos, long long cap, const float* k_chan_scale,
                             const float* v_chan_scale, float* k_mean, float* v_code_amax,
                             int8_t* k_codes, int8_t* v_codes, cudaStream_t s) {
  const int n = BH * d;
  return launch_pdl(kv_append_kernel, dim3((n + 255) / 256), dim3(256), 0, s, K_new, V_new, n, d, T,
                    pos, cap, k_chan_scale, v_chan_scale, k_mean, v_code_amax, k_codes, v_codes);
}

cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, DecodeArgs a, void* ws,
                          cudaStream_t s) {
  const long long R = (a.Hq / a.Hkv) * a.Nq;
  const long long nkb = (a.Nk + kBlk - 1) / kBlk;
  const long long BH = static_cast<long long>(a.B) * a.Hkv;
  auto a256 = [](long long x) { return static_cast<size_t>((x + 255) / 256 * 256); };
  char* p = static_cast<char*>(ws);
  a.ctr = reinterpret_cast<unsigned long long*>(p);
  p += a256(8);
  a.part_o = reinterpret_cast<float*>(p);
  p += a256(BH * nkb * R * a.d * 4);
  a.part_l = reinterpret_cast<float*>(p);
  p += a256(BH * nkb * R * 4);
  a.part_m = reinterpret_cast<float*>(p);
  p += a256(BH * nkb * R * 4);
  a.rec = reinterpret_cast<unsigned long long*>(p);
  if (R <= 4)
    return a.d == 64 ? launch_decode_r<64, 4>(tk, tv, a, s) : launch_decode_r<128, 4>(tk, tv, a, s);
  return a.d == 64 ? launch_decode_r<64, kMaxDecodeRows>(tk, tv, a, s)
                   : launch_decode_r<128, kMaxDecodeRows>(tk, tv, a, s);
}

}  // namespace qattn
