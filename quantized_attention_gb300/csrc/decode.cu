// Decode on an int8 KV cache: a few query tokens per (batch, head) against a
// long cache of int8 K and V codes.  At batch one both attention products are
// matrix-vector products bound by the bytes of the cache ("int8 Flash
// Attention on RDNA4", "What actually changed for decode"), so this path
// streams the codes as stored -- K for the scores, V row-major for PV --
// split over key blocks so every SM reads.
//
// It computes the recipe of the prefill kernel on the same codes: blocks of
// 128 keys in ascending order, each block's P relative to the running max at
// that block.  The split keeps that exactly: pass 1 writes every block's
// scores t = S c and each row's block maximum; pass 2 rebuilds the running max
// of each block as a prefix maximum of the block maxima, so P = 2^(t - m_j)
// and its e4m3 code are the recipe's, and accumulates a chunk of blocks'
// share of O and l scaled to the running max at the chunk's end; pass 3
// combines the chunks.  Rows are (query head of the KV group, token):
// r = g * Nq + i.
//
// Both streaming passes move key blocks into shared memory with TMA (128-byte
// swizzle for d = 128, 64-byte for d = 64) through a ring of stages, so a CTA
// keeps several blocks in flight.  Pass 1 waits on the kernels before it and
// only then lets pass 2 launch; pass 2 can therefore start its V loads before
// its own wait (the cache was written before this call), overlapping the tail
// of pass 1.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kBlk = 128;         // keys per block (the recipe's key block)
constexpr int kScoreStages = 2;   // pass 1 ring depth (many CTAs per SM)
constexpr int kPvStages = 3;      // pass 2 ring depth
constexpr int kPvThreads = 128;   // four warps: warp w takes keys 32w .. 32w+31 of a block
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

// ------------------------------------------------------------------ pass 1
// Persistent CTAs of 128 threads; CTA c takes the key blocks gb = c, c + grid,
// ... of all (batch * KV head, block j) pairs, gb = bkv * nkb + j, through a
// ring of kScoreStages stages (the block's K codes by TMA, swizzled, and the
// head's Q rows by a bulk copy).  Thread k owns key j * 128 + k: the exact
// int32 dot products run on dp4a; the swizzle puts the 8 keys of a shared-
// memory phase in 8 different bank groups, and every lane reads the same Q
// chunk (a broadcast).  Writes t = S c (masked keys -inf) and each row's block
// maximum.
template <int D, int RMAX>
struct ScoreSmem {
  static constexpr int kK = kBlk * D;                           // K codes of a block
  static constexpr int kStage = round_up(kK + RMAX * D, 1024);  // + the head's Q codes
  static constexpr int kBytes = kScoreStages * kStage + 1024;   // + alignment slack
};

template <int D, int RMAX>
__global__ void __launch_bounds__(kBlk) decode_scores_kernel(const __grid_constant__ CUtensorMap tmK,
                                                             const DecodeArgs a) {
  constexpr int NC = D / 16;  // 16-byte chunks per key row
  using SM = ScoreSmem<D, RMAX>;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = dsm_raw + ((1024u - (smem_u32(dsm_raw) & 1023u)) & 1023u);
  __shared__ float cfv[2][RMAX];
  __shared__ float wmax[2][kBlk / 32][RMAX];
  __shared__ __align__(8) uint64_t full[kScoreStages];
  __shared__ int abort_flag;
  const int G = a.Hq / a.Hkv, R = G * a.Nq;
  const int nkb = (a.Nk + kBlk - 1) / kBlk, nqb = (a.Nq + kBlk - 1) / kBlk;
  const int total = nkb * a.B * a.Hkv;
  const int n_my = (total - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                   static_cast<int>(gridDim.x);
  const size_t tstride = static_cast<size_t>(nkb) * kBlk;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kScoreStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
  }
  __syncthreads();
  pdl_wait();     // Q codes and scales come from the kernels before; the cache may too
  pdl_trigger();  // only now: pass 2 may read the cache before its own wait
  // thread 0: the i-th block of this CTA into stage i % kScoreStages
  auto issue = [&](int i) {
    const int gb = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    const int bkv = gb / nkb, j = gb % nkb;
    const int b = bkv / a.Hkv, hkv = bkv % a.Hkv;
    const uint32_t st = smem_u32(dsm + (i % kScoreStages) * SM::kStage);
    const uint32_t bar = smem_u32(&full[i % kScoreStages]);
    // the TMA box is always 128 full rows (rows past Nk arrive as zeros)
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>((kBlk + R) * D));
    tma_load_3d(st, &tmK, bar, 0, j * kBlk, bkv);
    // rows r = g * Nq + i of the head are contiguous: heads hkv*G .. hkv*G+G-1
    bulk_g2s(st + SM::kK, a.q_codes + (static_cast<size_t>(b) * a.Hq + hkv * G) * a.Nq * D,
             static_cast<uint32_t>(R * D), bar);
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < min(kScoreStages, n_my); ++i) issue(i);
  // the scales of row r for the i-th block (threads r < R)
  auto load_scales = [&](int i, int r, float& sq, float& sk) {
    const int gb = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    const int bkv = gb / nkb, j = gb % nkb;
    const int b = bkv / a.Hkv, hkv = bkv % a.Hkv, g = r / a.Nq, ii = r % a.Nq;
    sq = scale_at(a.q_scales, a.q_gran, b * a.Hq + hkv * G + g, nqb, ii / kBlk);
    sk = scale_at(a.k_scales, a.k_gran, bkv, nkb, j);
  };
  auto cfac = [&](float sq, float sk) {
    return __fmul_rn(__fmul_rn(__fmul_rn(sq, sk), a.sm_scale), kLog2e);
  };
  if (threadIdx.x < R && n_my > 0) {
    float sq, sk;
    load_scales(0, threadIdx.x, sq, sk);
    cfv[0][threadIdx.x] = cfac(sq, sk);
  }
  __syncthreads();
  const int k = threadIdx.x;
  for (int i = 0; i < n_my; ++i) {
    const int s = i % kScoreStages;
    const int gb = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    const int bkv = gb / nkb, j = gb % nkb;
    float nsq = 0.f, nsk = 0.f;  // the next block's scales, in flight during the wait
    if (threadIdx.x < R && i + 1 < n_my) load_scales(i + 1, threadIdx.x, nsq, nsk);
    if (!mbar_wait(smem_u32(&full[s]), (i / kScoreStages) & 1, &abort_flag, a.err, kErrTimeout))
      return;
    const int8_t* ks = reinterpret_cast<const int8_t*>(dsm + s * SM::kStage);
    const int8_t* qs = ks + SM::kK;
    int acc[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) acc[r] = 0;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const uint4 kw = *reinterpret_cast<const uint4*>(ks + swz_chunk<D>(k, c));
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        if (r < R) {
          const uint4 qw = *reinterpret_cast<const uint4*>(qs + r * D + c * 16);
          acc[r] = __dp4a(static_cast<int>(kw.x), static_cast<int>(qw.x), acc[r]);
          acc[r] = __dp4a(static_cast<int>(kw.y), static_cast<int>(qw.y), acc[r]);
          acc[r] = __dp4a(static_cast<int>(kw.z), static_cast<int>(qw.z), acc[r]);
          acc[r] = __dp4a(static_cast<int>(kw.w), static_cast<int>(qw.w), acc[r]);
        }
      }
    }
    const int key = j * kBlk + k;
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      if (r < R) {
        const int ii = r % a.Nq;
        const bool vis = key < a.Nk && (!a.causal || key <= a.pos0 + ii);
        const float t = vis ? __fmul_rn(static_cast<float>(acc[r]), cfv[i & 1][r]) : kNegInf;
        a.t[(static_cast<size_t>(bkv) * R + r) * tstride + key] = t;
        float mx = t;
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
        if ((k & 31) == 0) wmax[i & 1][k >> 5][r] = mx;
      }
    }
    if (threadIdx.x < R && i + 1 < n_my) cfv[(i + 1) & 1][threadIdx.x] = cfac(nsq, nsk);
    __syncthreads();  // stage s is read; the block's warp maxima are in
    if (threadIdx.x == 0 && i + kScoreStages < n_my) issue(i + kScoreStages);
    if (threadIdx.x < R) {
      const int r = threadIdx.x;
      const float mx = fmaxf(fmaxf(wmax[i & 1][0][r], wmax[i & 1][1][r]),
                             fmaxf(wmax[i & 1][2][r], wmax[i & 1][3][r]));
      a.mblk[(static_cast<size_t>(bkv) * nkb + j) * R + r] = mx;
    }
  }
}

// ------------------------------------------------------------------ pass 2
// One CTA of four warps per (chunk of bpc key blocks, batch * KV head).  The
// chunk's t rows arrive by bulk copy and become the e4m3 codes of 448 P
// relative to each block's running max (the recipe's P8), stored in the
// A-fragment order of mma.m16n8k32; V blocks stream through a ring of TMA
// stages.  For each block, warp w multiplies P8 (rows x keys 32w..32w+31) by
// the block's V8 on the tensor cores (e4m3 x e4m3, fp32 accumulation): every
// lane reads 16 (d = 128) or 8 (d = 64) channels of 8 keys, rounds the codes
// to e4m3 as qattn_quantize_v does, and transposes 4x4 byte groups into B
// fragments.  Keys of a 32-key step are permuted (fragment position
// 4t + i <-> key 8i + 2t, 16 + 4t + i <-> key 8i + 2t + 1) so the 8 lanes of a
// shared-memory phase hit 8 bank groups of the swizzled tile; P8 uses the same
// permutation.  Channels: lane group g = lane / 4 owns channels CPT*g ..
// CPT*g + CPT-1; n-tile (word w, byte e) column n is channel CPT*n + 4w + e.
// Between blocks the accumulators are rescaled by 2^(m_prev - m_j), so the
// chunk's share ends relative to the running max at its last block.
template <int D, int RMAX>
struct PvSmem {
  static constexpr int kMaxBlocks = (RMAX <= 4) ? 8 : 4;  // key blocks per chunk, at most
  static constexpr int kChunkKeys = kMaxBlocks * kBlk;
  static constexpr int kStage = kBlk * D;  // 1024-byte multiple
  static constexpr int kRing = kPvStages * kStage;
  static constexpr int kT = RMAX * kChunkKeys * 4;               // t rows of the chunk (fp32)
  static constexpr int kP8 = kMaxBlocks * 4 * RMAX * 32;         // [block][step][row][32]
  static constexpr int kBytes = kRing + kT + kP8 + 1024;         // + alignment slack
  static constexpr int kRed = (kPvThreads / 32) * RMAX * D * 4;  // [warp][row][d]
  static_assert(kRed <= kRing, "reduction buffer does not fit");
};

template <int D, int RMAX>
__global__ void __launch_bounds__(kPvThreads) decode_pv_kernel(const __grid_constant__ CUtensorMap tmV,
                                                               const DecodeArgs a, int bpc) {
  constexpr int CPT = D / 8;    // channels per lane group
  constexpr int WPT = CPT / 4;  // their 32-bit words
  constexpr int NT = 4 * WPT;   // n-tiles a lane accumulates
  using SM = PvSmem<D, RMAX>;
  constexpr int CK = SM::kChunkKeys;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = dsm_raw + ((1024u - (smem_u32(dsm_raw) & 1023u)) & 1023u);
  float* tb = reinterpret_cast<float*>(dsm + SM::kRing);
  uint8_t* p8 = dsm + SM::kRing + SM::kT;
  float* red = reinterpret_cast<float*>(dsm);
  __shared__ float mrun[SM::kMaxBlocks][RMAX];
  __shared__ float lblk[SM::kMaxBlocks][RMAX];
  __shared__ float mpre[kPvThreads];
  __shared__ __align__(16) float inv_s[D];
  __shared__ __align__(8) uint64_t full[kPvStages];
  __shared__ __align__(8) uint64_t tbar;
  __shared__ int abort_flag;
  const int ch = blockIdx.x, bkv = blockIdx.y;
  const int c0 = ch * bpc;
  const int G = a.Hq / a.Hkv, R = G * a.Nq;
  const int nkb = (a.Nk + kBlk - 1) / kBlk;
  const int nb = min(bpc, nkb - c0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPvStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    mbar_init(smem_u32(&tbar), 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmV);
  }
  __syncthreads();
  // thread 0: V codes of the chunk's block jj into stage jj % kPvStages
  auto issue_v = [&](int jj) {
    const uint32_t bar = smem_u32(&full[jj % kPvStages]);
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kBlk * D));
    tma_load_3d(smem_u32(dsm + (jj % kPvStages) * SM::kStage), &tmV, bar, 0, (c0 + jj) * kBlk, bkv);
  };
  // The cache (V codes, their channel maxima) precedes this call; pass 1
  // released this grid only after its own wait, so it is complete here.
  if (threadIdx.x == 0)
    for (int jj = 0; jj < min(kPvStages, nb); ++jj) issue_v(jj);
  for (int c = threadIdx.x; c < D; c += kPvThreads) {
    const float am = __ldg(a.v_code_amax + static_cast<size_t>(bkv) * D + c);
    inv_s[c] = (am > 0.f) ? __fdiv_rn(448.0f, am) : 0.f;
  }
  pdl_wait();  // t and the block maxima come from pass 1
  pdl_trigger();
  const size_t tstride = static_cast<size_t>(nkb) * kBlk;
  if (threadIdx.x == 0) {
    const uint32_t bar = smem_u32(&tbar);
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(R * nb * kBlk * 4));
    for (int r = 0; r < R; ++r)
      bulk_g2s(smem_u32(tb + r * CK),
               a.t + (static_cast<size_t>(bkv) * R + r) * tstride + static_cast<size_t>(c0) * kBlk,
               static_cast<uint32_t>(nb * kBlk * 4), bar);
  }
  const float* mb = a.mblk + static_cast<size_t>(bkv) * nkb * R;
  // the running max before the chunk: max of the earlier blocks' maxima
  {
    const int r = threadIdx.x % R, part = threadIdx.x / R, parts = kPvThreads / R;
    float mx = kNegInf;
    if (part < parts)
      for (int jj = part; jj < c0; jj += parts) mx = fmaxf(mx, mb[static_cast<size_t>(jj) * R + r]);
    mpre[threadIdx.x] = mx;
  }
  __syncthreads();
  if (threadIdx.x < R) {
    const int r = threadIdx.x, parts = kPvThreads / R;
    float m = kNegInf;
    for (int p = 0; p < parts; ++p) m = fmaxf(m, mpre[p * R + r]);
    for (int jj = 0; jj < nb; ++jj) {
      m = fmaxf(m, mb[static_cast<size_t>(c0 + jj) * R + r]);
      mrun[jj][r] = m;
    }
  }
  __syncthreads();
  if (!mbar_wait(smem_u32(&tbar), 0, &abort_flag, a.err, kErrTimeout)) return;
  // P8 = e4m3(448 P), P = 2^(t - m_j) relative to the block's running max,
  // written in fragment order; the block's sum of 448 P (unquantized).  One
  // warp per row; lane = key within a 32-key step.
  {
    const int f = (lane & 1) ? (16 + 4 * ((lane >> 1) & 3) + (lane >> 3))
                             : (4 * ((lane >> 1) & 3) + (lane >> 3));
    for (int r = warp; r < R; r += kPvThreads / 32) {
      const float* tr = tb + r * CK;
      for (int jj = 0; jj < nb; ++jj) {
        const float mj = mrun[jj][r];
        const float kneg = (mj == kNegInf) ? 0.f : (kLog2_448 - mj);
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float p = ex2_approx(__fadd_rn(tr[jj * kBlk + 32 * q + lane], kneg));
          sum += p;
          p8[((jj * 4 + q) * RMAX + r) * 32 + f] = static_cast<uint8_t>(cvt_e4m3x2(p, 0.f) & 0xFFu);
        }
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
        if (lane == 0) lblk[jj][r] = sum;
      }
    }
  }
  __syncthreads();
  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  const bool row_lo = g < R, row_hi = (RMAX > 8) && (g + 8 < R);
  for (int jj = 0; jj < nb; ++jj) {
    const int s = jj % kPvStages;
    if (!mbar_wait(smem_u32(&full[s]), (jj / kPvStages) & 1, &abort_flag, a.err, kErrTimeout))
      return;
    if (jj > 0) {  // rescale to this block's running max (skipped while it holds)
      const float f0 =
          (row_lo && mrun[jj][g] != kNegInf) ? ex2_approx(mrun[jj - 1][g] - mrun[jj][g]) : 1.f;
      const float f1 = (row_hi && mrun[jj][g + 8] != kNegInf)
                           ? ex2_approx(mrun[jj - 1][g + 8] - mrun[jj][g + 8])
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
    // A fragments: P8 rows g, g + 8 of this warp's 32-key step
    const uint8_t* pa = p8 + ((jj * 4 + warp) * RMAX) * 32;
    const uint32_t a0 = row_lo ? *reinterpret_cast<const uint32_t*>(pa + g * 32 + 4 * t4) : 0u;
    const uint32_t a2 = row_lo ? *reinterpret_cast<const uint32_t*>(pa + g * 32 + 16 + 4 * t4) : 0u;
    const uint32_t a1 =
        row_hi ? *reinterpret_cast<const uint32_t*>(pa + (g + 8) * 32 + 4 * t4) : 0u;
    const uint32_t a3 =
        row_hi ? *reinterpret_cast<const uint32_t*>(pa + (g + 8) * 32 + 16 + 4 * t4) : 0u;
    // this lane's channels of its 8 keys: key 8i + 2t4 (+1 for h = 1) of the step
    const uint8_t* vs = dsm + s * SM::kStage;
    uint32_t raw[8][WPT];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = 32 * warp + 8 * i + 2 * t4 + h;
        const uint8_t* src = vs + swz_chunk<D>(row, (CPT * g) >> 4) + ((CPT * g) & 15);
        if constexpr (WPT == 4) {
          const uint4 v = *reinterpret_cast<const uint4*>(src);
          raw[4 * h + i][0] = v.x;
          raw[4 * h + i][1] = v.y;
          raw[4 * h + i][2] = v.z;
          raw[4 * h + i][3] = v.w;
        } else {
          const uint2 v = *reinterpret_cast<const uint2*>(src);
          raw[4 * h + i][0] = v.x;
          raw[4 * h + i][1] = v.y;
        }
      }
    }
#pragma unroll
    for (int w = 0; w < WPT; ++w) {
      const float4 iv = *reinterpret_cast<const float4*>(inv_s + CPT * g + 4 * w);
      uint32_t e0[4], e1[4], b0[4], b1[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        e0[i] = v_codes_to_e4m3(raw[i][w], iv);
        e1[i] = v_codes_to_e4m3(raw[4 + i][w], iv);
      }
      transpose4x4(e0, b0);
      transpose4x4(e1, b1);
#pragma unroll
      for (int e = 0; e < 4; ++e) mma_e4m3_16832(acc[4 * w + e], a0, a1, a2, a3, b0[e], b1[e]);
    }
    __syncthreads();  // stage s is read
    if (threadIdx.x == 0 && jj + kPvStages < nb) issue_v(jj + kPvStages);
  }
  // reduce the four warps' shares; write the chunk's O share
#pragma unroll
  for (int w = 0; w < WPT; ++w) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = CPT * (2 * t4 + cc) + 4 * w + e;
        if (row_lo) red[(warp * RMAX + g) * D + c] = acc[4 * w + e][cc];
        if (row_hi) red[(warp * RMAX + g + 8) * D + c] = acc[4 * w + e][2 + cc];
      }
    }
  }
  __syncthreads();
  const size_t pbase = (static_cast<size_t>(bkv) * gridDim.x + ch) * R;
  for (int idx = threadIdx.x; idx < R * D; idx += kPvThreads) {
    const int r = idx / D, c = idx % D;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kPvThreads / 32; ++w) sum += red[(w * RMAX + r) * D + c];
    a.part_o[(pbase + r) * D + c] = sum;
  }
  if (threadIdx.x < R) {
    const int r = threadIdx.x;
    const float mend = mrun[nb - 1][r];
    float l = 0.f;
    if (mend != kNegInf)
      for (int jj = 0; jj < nb; ++jj) l += lblk[jj][r] * ex2_approx(mrun[jj][r] - mend);
    a.part_l[pbase + r] = l;
    a.part_m[pbase + r] = mend;
  }
}

// ------------------------------------------------------------------ pass 3
// One CTA per (row, batch * KV head).  Thread (chunk group cg, channel word
// c4) sums chunks cg, cg + CG, ... scaled to the final max.
template <int D>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const DecodeArgs a,
                                                                        int nchunks) {
  constexpr int TPC = D / 4;                 // threads per chunk row
  constexpr int CG = kCombineThreads / TPC;  // chunk groups
  constexpr int U = 4;                       // chunks in flight per thread
  __shared__ float wm[kCombineThreads / 32];
  __shared__ __align__(16) float red[CG][D];
  __shared__ float redl[CG];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, bkv = blockIdx.y;
  const int b = bkv / a.Hkv, hkv = bkv % a.Hkv;
  const int G = a.Hq / a.Hkv, R = G * a.Nq;
  const size_t p0 = static_cast<size_t>(bkv) * nchunks * R + r;  // chunk c: p0 + c * R
  float mf = kNegInf;
  for (int c = threadIdx.x; c < nchunks; c += kCombineThreads)
    mf = fmaxf(mf, a.part_m[p0 + static_cast<size_t>(c) * R]);
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) mf = fmaxf(mf, __shfl_xor_sync(0xffffffffu, mf, sh));
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = mf;
  __syncthreads();
  mf = wm[0];
#pragma unroll
  for (int w = 1; w < kCombineThreads / 32; ++w) mf = fmaxf(mf, wm[w]);
  const int c4 = threadIdx.x % TPC, cg = threadIdx.x / TPC;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  if (mf != kNegInf) {
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
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float wgt = (mc[u] == kNegInf) ? 0.f : ex2_approx(mc[u] - mf);
        l = fmaf(wgt, lc[u], l);
        o.x = fmaf(wgt, oc[u].x, o.x);
        o.y = fmaf(wgt, oc[u].y, o.y);
        o.z = fmaf(wgt, oc[u].z, o.z);
        o.w = fmaf(wgt, oc[u].w, o.w);
      }
    }
  }
  *reinterpret_cast<float4*>(&red[cg][4 * c4]) = o;
  if (c4 == 0) redl[cg] = l;
  __syncthreads();
  const int g = r / a.Nq, i = r % a.Nq;
  const size_t row = (static_cast<size_t>(b) * a.Hq + hkv * G + g) * a.Nq + i;
  float lt = 0.f;
#pragma unroll
  for (int g2 = 0; g2 < CG; ++g2) lt += redl[g2];
  for (int c = threadIdx.x; c < D; c += kCombineThreads) {
    float s = 0.f;
#pragma unroll
    for (int g2 = 0; g2 < CG; ++g2) s += red[g2][c];
    // V scale s_v = fp32(fp32(chan * amax) / 448), as qattn_quantize_v writes it
    const size_t vc = static_cast<size_t>(bkv) * D + c;
    const float sv = __fdiv_rn(__fmul_rn(__ldg(a.v_chan_scale + vc), __ldg(a.v_code_amax + vc)), 448.0f);
    const float out = (lt > 0.f) ? s * (sv * (1.f / lt)) : 0.f;
    if (a.out_bf16) reinterpret_cast<__nv_bfloat16*>(a.out)[row * D + c] = __float2bfloat16(out);
    else reinterpret_cast<float*>(a.out)[row * D + c] = out;
  }
  if (threadIdx.x == 0 && a.lse)
    a.lse[row] = (lt > 0.f) ? (mf + __log2f(lt) - kLog2_448) * kLn2 : kNegInf;
}

// CTAs of a kernel resident per SM.  Callers cache it: it depends only on the
// kernel and the device model, and a wrong value changes the grid, not results.
template <typename Kernel>
int ctas_per_sm(Kernel kernel, int threads, int smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
      n < 1)
    n = 1;
  return n;
}

template <int D, int RMAX>
cudaError_t launch_decode_r(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                            cudaStream_t s) {
  const int BHkv = a.B * a.Hkv;
  const int nkb = (a.Nk + kBlk - 1) / kBlk;
  const int sms = num_sms();
  const int total = nkb * BHkv;
  // pass 1: a persistent grid filling every SM
  constexpr int ssmem = ScoreSmem<D, RMAX>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(decode_scores_kernel<D, RMAX>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, ssmem);
  if (e != cudaSuccess) return e;
  static const int occ1 = ctas_per_sm(decode_scores_kernel<D, RMAX>, kBlk, ssmem);
  const int g1 = min(total, sms * occ1);
  e = launch_pdl(decode_scores_kernel<D, RMAX>, dim3(g1), dim3(kBlk), ssmem, s, tk, a);
  if (e != cudaSuccess) return e;
  // pass 2: chunks sized so every resident CTA slot gets one
  using PS = PvSmem<D, RMAX>;
  e = cudaFuncSetAttribute(decode_pv_kernel<D, RMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PS::kBytes);
  if (e != cudaSuccess) return e;
  static const int occ2 = ctas_per_sm(decode_pv_kernel<D, RMAX>, kPvThreads, PS::kBytes);
  const int target = sms * occ2;
  const int bpc = max(1, min(PS::kMaxBlocks, (total + target - 1) / target));
  const int nchunks = (nkb + bpc - 1) / bpc;
  e = launch_pdl(decode_pv_kernel<D, RMAX>, dim3(nchunks, BHkv), dim3(kPvThreads), PS::kBytes, s,
                 tv, a, bpc);
  if (e != cudaSuccess) return e;
  const int R = (a.Hq / a.Hkv) * a.Nq;
  return launch_pdl(decode_combine_kernel<D>, dim3(R, BHkv), dim3(kCombineThreads), 0, s, a,
                    nchunks);
}

}  // namespace

// Workspace: t [B*Hkv][R][nkb*128], block maxima [B*Hkv][nkb][R], and the
// chunk shares O [B*Hkv][chunks][R][d], l and m [B*Hkv][chunks][R], sized for
// the most chunks (one block each) so the layout does not depend on the GPU.
size_t decode_ws_bytes(long long B, long long Hq, long long Hkv, long long Nq, long long Nk,
                       long long d) {
  const long long R = (Hq / Hkv) * Nq;
  const long long nkb = (Nk + kBlk - 1) / kBlk;
  const long long BH = B * Hkv;
  auto a256 = [](long long x) { return static_cast<size_t>((x + 255) / 256 * 256); };
  return a256(BH * R * nkb * kBlk * 4) +  // t
         a256(BH * nkb * R * 4) +          // block maxima
         a256(BH * nkb * R * d * 4) +      // chunk O
         2 * a256(BH * nkb * R * 4);       // chunk l, m
}

cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, DecodeArgs a, void* ws,
                          cudaStream_t s) {
  const long long R = (a.Hq / a.Hkv) * a.Nq;
  const long long nkb = (a.Nk + kBlk - 1) / kBlk;
  const long long BH = static_cast<long long>(a.B) * a.Hkv;
  auto a256 = [](long long x) { return static_cast<size_t>((x + 255) / 256 * 256); };
  char* p = static_cast<char*>(ws);
  a.t = reinterpret_cast<float*>(p);
  p += a256(BH * R * nkb * kBlk * 4);
  a.mblk = reinterpret_cast<float*>(p);
  p += a256(BH * nkb * R * 4);
  a.part_o = reinterpret_cast<float*>(p);
  p += a256(BH * nkb * R * a.d * 4);
  a.part_l = reinterpret_cast<float*>(p);
  p += a256(BH * nkb * R * 4);
  a.part_m = reinterpret_cast<float*>(p);
  if (R <= 4)
    return a.d == 64 ? launch_decode_r<64, 4>(tk, tv, a, s) : launch_decode_r<128, 4>(tk, tv, a, s);
  return a.d == 64 ? launch_decode_r<64, kMaxDecodeRows>(tk, tv, a, s)
                   : launch_decode_r<128, kMaxDecodeRows>(tk, tv, a, s);
}

}  // namespace qattn
