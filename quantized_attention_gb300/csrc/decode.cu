// Decode on an int8 KV cache: a few query tokens per (batch, head) against a
// long cache of int8 K and V codes.  At batch one both attention products are
// matrix-vector products bound by the bytes of the cache ("int8 Flash
// Attention on RDNA4", "What actually changed for decode"), so this path
// streams the codes as stored -- K for the scores, V row-major for PV -- on
// the CUDA cores, split over key blocks so every SM reads.
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
// Both streaming passes move a key block (or a chunk of them) into shared
// memory with one bulk copy, so a CTA has its whole share of the cache in
// flight at once.  Pass 1 waits on the kernels before it and only then lets
// pass 2 launch; pass 2 can therefore start its V copy before its own wait
// (the cache was written before this call), overlapping the tail of pass 1.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qattn_internal.h"
#include "sm103_ptx.cuh"

namespace qattn {
namespace {

constexpr int kBlk = 128;  // keys per block (the recipe's key block)
constexpr int kPvThreads = 256;
constexpr int kCombineThreads = 256;
constexpr int kChunkKeys = kDecodeChunk * kBlk;
constexpr float kLog2e = 1.44269502162933349609375f;  // fp32(log2 e)
constexpr float kLog2_448 = 8.8073549220576041f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kNegInf = -__builtin_huge_valf();

// The values of e4m3_rn_satfinite(x), e4m3_rn_satfinite(y) as fp32.
__device__ __forceinline__ float2 e4m3_values(float x, float y) {
  const uint32_t h = e4m3x2_to_f16x2(cvt_e4m3x2(x, y));
  return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16))));
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

// Q and K scales are written by the kernels just before this call (plain
// loads after the dependency wait, not the read-only path).
__device__ __forceinline__ float scale_at(const float* s, int gran, int bh, int nblk, int blk) {
  if (gran == 0) return s[0];
  if (gran == 1) return s[bh];
  return s[static_cast<size_t>(bh) * nblk + blk];
}

// Pass 1: one CTA of 128 threads per (key block j, batch * KV head); thread k
// owns key j * 128 + k.  The block's K codes arrive by one bulk copy; the
// exact int32 dot products run on dp4a, each thread walking the 16-byte
// chunks of its key row in a rotated order so the 8 threads of a shared-memory
// phase read 8 different bank groups.  Writes t = S c (masked keys -inf) and
// each row's block maximum.
template <int D, int RMAX>
__global__ void __launch_bounds__(kBlk) decode_scores_kernel(const DecodeArgs a) {
  constexpr int NC = D / 16;                // 16-byte chunks per key row
  constexpr int KSH = (D == 128) ? 0 : 1;   // log2 of key rows per 128 bytes
  __shared__ __align__(128) int8_t ks[kBlk * D];
  __shared__ __align__(16) int8_t qs[RMAX * D];
  __shared__ float cf[RMAX];
  __shared__ float wmax[kBlk / 32][RMAX];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int j = blockIdx.x, bkv = blockIdx.y;
  const int b = bkv / a.Hkv, hkv = bkv % a.Hkv;
  const int G = a.Hq / a.Hkv, R = G * a.Nq;
  const int nkb = (a.Nk + kBlk - 1) / kBlk, nqb = (a.Nq + kBlk - 1) / kBlk;
  const int nvalid = min(kBlk, a.Nk - j * kBlk);
  const uint32_t bar_a = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(bar_a, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();     // Q codes and K scales are written by the kernels before
  pdl_trigger();  // only now: pass 2 may read the cache before its own wait
  if (threadIdx.x == 0) {
    const int8_t* src = a.k_codes + (static_cast<size_t>(bkv) * a.Nk + static_cast<size_t>(j) * kBlk) * D;
    mbar_arrive_expect_tx(bar_a, static_cast<uint32_t>(nvalid * D));
    bulk_g2s(smem_u32(ks), src, static_cast<uint32_t>(nvalid * D), bar_a);
  }
  // the rows' Q codes: row r = g * Nq + i is query head hkv * G + g, token i
  for (int v = threadIdx.x; v < R * D / 16; v += kBlk) {
    const int r = v / (D / 16), cv = v % (D / 16);
    const int g = r / a.Nq, i = r % a.Nq;
    const int8_t* q = a.q_codes + ((static_cast<size_t>(b) * a.Hq + hkv * G + g) * a.Nq + i) * D;
    *reinterpret_cast<uint4*>(qs + r * D + cv * 16) = reinterpret_cast<const uint4*>(q)[cv];
  }
  if (threadIdx.x < R) {
    const int r = threadIdx.x, g = r / a.Nq, i = r % a.Nq;
    const float sq = scale_at(a.q_scales, a.q_gran, b * a.Hq + hkv * G + g, nqb, i / kBlk);
    const float sk = scale_at(a.k_scales, a.k_gran, bkv, nkb, j);
    cf[r] = __fmul_rn(__fmul_rn(__fmul_rn(sq, sk), a.sm_scale), kLog2e);
  }
  __syncthreads();
  if (!mbar_wait(bar_a, 0, &abort_flag, a.err, kErrTimeout)) return;
  const int k = threadIdx.x;
  int acc[RMAX];
#pragma unroll
  for (int r = 0; r < RMAX; ++r) acc[r] = 0;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int cc = (c + (k >> KSH)) & (NC - 1);
    const uint4 kw = *reinterpret_cast<const uint4*>(ks + k * D + cc * 16);
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
  const int key = j * kBlk + k;
  const size_t tstride = static_cast<size_t>(nkb) * kBlk;
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    if (r < R) {
      const int i = r % a.Nq;
      const bool vis = key < a.Nk && (!a.causal || key <= a.pos0 + i);
      const float t = vis ? __fmul_rn(static_cast<float>(acc[r]), cf[r]) : kNegInf;
      a.t[(static_cast<size_t>(bkv) * R + r) * tstride + key] = t;
      float mx = t;
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
      if ((k & 31) == 0) wmax[k >> 5][r] = mx;
    }
  }
  __syncthreads();
  if (threadIdx.x < R) {
    const int r = threadIdx.x;
    const float mx = fmaxf(fmaxf(wmax[0][r], wmax[1][r]), fmaxf(wmax[2][r], wmax[3][r]));
    a.mblk[(static_cast<size_t>(bkv) * nkb + j) * R + r] = mx;
  }
}

// Shared memory of pass 2 (dynamic): the chunk's V codes, then the weighted
// e4m3 P of the chunk [key][RMAX]; after the products both regions hold the
// reduction buffer of four rows [4][KG][D].
template <int D, int RMAX>
struct PvSmem {
  static constexpr int kV = kChunkKeys * D;
  static constexpr int kP = kChunkKeys * RMAX * 4;
  static constexpr int kBytes = kV + kP;
  static constexpr int kRed = 4 * (kPvThreads / (D / 4)) * D * 4;
  static_assert(kRed <= kBytes, "reduction buffer does not fit");
};

// Pass 2: one CTA per (chunk of kDecodeChunk blocks, batch * KV head).
// Thread (channel word cw = tid % (D/4), key group kg = tid / (D/4)) owns
// channels 4 cw .. 4 cw + 3 of keys kg, kg + KG, ... of the chunk.
template <int D, int RMAX>
__global__ void __launch_bounds__(kPvThreads) decode_pv_kernel(const DecodeArgs a) {
  constexpr int CW = D / 4;            // channel words (4 channels each)
  constexpr int KG = kPvThreads / CW;  // key groups
  constexpr int KPT = kBlk / KG;       // keys per thread per block
  extern __shared__ __align__(128) uint8_t dsm[];
  int8_t* vs = reinterpret_cast<int8_t*>(dsm);
  float* pw = reinterpret_cast<float*>(dsm + PvSmem<D, RMAX>::kV);
  float* red = reinterpret_cast<float*>(dsm);
  __shared__ float mrun[kDecodeChunk][RMAX];
  __shared__ float lblk[kDecodeChunk][RMAX];
  __shared__ float mpre[kPvThreads];
  __shared__ __align__(16) float inv_s[D];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int ch = blockIdx.x, bkv = blockIdx.y;
  const int c0 = ch * kDecodeChunk;
  const int G = a.Hq / a.Hkv, R = G * a.Nq;
  const int nkb = (a.Nk + kBlk - 1) / kBlk;
  const int nb = min(kDecodeChunk, nkb - c0);
  const int nv = min(kChunkKeys, a.Nk - c0 * kBlk);
  const uint32_t bar_a = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(bar_a, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // The cache (V codes, their channel maxima) precedes this call; pass 1
  // released this grid only after its own wait, so it is complete here.
  if (threadIdx.x == 0) {
    const int8_t* src = a.v_codes + (static_cast<size_t>(bkv) * a.Nk + static_cast<size_t>(c0) * kBlk) * D;
    mbar_arrive_expect_tx(bar_a, static_cast<uint32_t>(nv * D));
    bulk_g2s(smem_u32(vs), src, static_cast<uint32_t>(nv * D), bar_a);
  }
  for (int c = threadIdx.x; c < D; c += kPvThreads) {
    const float am = __ldg(a.v_code_amax + static_cast<size_t>(bkv) * D + c);
    inv_s[c] = (am > 0.f) ? __fdiv_rn(448.0f, am) : 0.f;
  }
  pdl_wait();  // t and the block maxima come from pass 1
  pdl_trigger();
  const size_t tstride = static_cast<size_t>(nkb) * kBlk;
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
  // P of each block relative to its running max; e4m3 of 448 P as a value,
  // times the block's weight 2^(m_j - m_end) to the running max at the
  // chunk's end; the block's sum of 448 P (unquantized).  One warp per row.
  for (int r = threadIdx.x / 32; r < R; r += kPvThreads / 32) {
    const float mend = mrun[nb - 1][r];
    const float* tr = a.t + (static_cast<size_t>(bkv) * R + r) * tstride + static_cast<size_t>(c0) * kBlk;
    for (int jj = 0; jj < nb; ++jj) {
      const float mj = mrun[jj][r];
      const float kneg = (mj == kNegInf) ? 0.f : (kLog2_448 - mj);
      const float w = (mend == kNegInf) ? 0.f : ex2_approx(mj - mend);
      float tv[kBlk / 32];
#pragma unroll
      for (int q = 0; q < kBlk / 32; ++q) tv[q] = tr[jj * kBlk + (threadIdx.x & 31) + 32 * q];
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < kBlk / 32; ++q) {
        const int kk = jj * kBlk + (threadIdx.x & 31) + 32 * q;
        const float p = ex2_approx(__fadd_rn(tv[q], kneg));
        sum += p;
        pw[kk * RMAX + r] = e4m3_values(p, 0.f).x * w;
      }
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, s);
      if ((threadIdx.x & 31) == 0) lblk[jj][r] = sum;
    }
  }
  // rows R .. RMAX-1 of the weights are read by the vector loads below
  for (int idx = threadIdx.x; idx < nb * kBlk * (RMAX - R); idx += kPvThreads) {
    const int kk = idx / (RMAX - R), r = R + idx % (RMAX - R);
    pw[kk * RMAX + r] = 0.f;
  }
  __syncthreads();
  if (!mbar_wait(bar_a, 0, &abort_flag, a.err, kErrTimeout)) return;
  // the chunk's share of O: keys past Nk carry P = 0 (their t is -inf)
  const int cw = threadIdx.x % CW, kg = threadIdx.x / CW;
  float2 o[RMAX][2];
#pragma unroll
  for (int r = 0; r < RMAX; ++r) o[r][0] = o[r][1] = make_float2(0.f, 0.f);
  const float2 iv01 = make_float2(inv_s[4 * cw], inv_s[4 * cw + 1]);
  const float2 iv23 = make_float2(inv_s[4 * cw + 2], inv_s[4 * cw + 3]);
  const uint32_t* vw = reinterpret_cast<const uint32_t*>(vs);
  for (int jj = 0; jj < nb; ++jj) {
#pragma unroll 4
    for (int q = 0; q < KPT; ++q) {
      const int kk = jj * kBlk + kg + q * KG;
      float2 c01, c23;
      codes4_to_f32(vw[kk * CW + cw], c01, c23);
      const float2 x01 = fmul2(c01, iv01), x23 = fmul2(c23, iv23);
      const float2 v01 = e4m3_values(x01.x, x01.y), v23 = e4m3_values(x23.x, x23.y);
#pragma unroll
      for (int r4 = 0; r4 < RMAX; r4 += 4) {
        if (r4 < R) {
          const float4 p4 = *reinterpret_cast<const float4*>(pw + kk * RMAX + r4);
          const float pr[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            o[r4 + e][0] = ffma2(make_float2(pr[e], pr[e]), v01, o[r4 + e][0]);
            o[r4 + e][1] = ffma2(make_float2(pr[e], pr[e]), v23, o[r4 + e][1]);
          }
        }
      }
    }
  }
  // reduce the key groups four rows at a time; write the chunk's O share
  const size_t pbase = (static_cast<size_t>(bkv) * gridDim.x + ch) * R;
#pragma unroll
  for (int r4 = 0; r4 < RMAX; r4 += 4) {
    if (r4 < R) {
      __syncthreads();  // the previous readers of this region are done
#pragma unroll
      for (int e = 0; e < 4; ++e)
        *reinterpret_cast<float4*>(red + ((e * KG) + kg) * D + 4 * cw) =
            make_float4(o[r4 + e][0].x, o[r4 + e][0].y, o[r4 + e][1].x, o[r4 + e][1].y);
      __syncthreads();
      for (int idx = threadIdx.x; idx < 4 * D; idx += kPvThreads) {
        const int e = idx / D, c = idx % D;
        if (r4 + e < R) {
          float s = 0.f;
#pragma unroll
          for (int g2 = 0; g2 < KG; ++g2) s += red[(e * KG + g2) * D + c];
          a.part_o[(pbase + r4 + e) * D + c] = s;
        }
      }
    }
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

// Pass 3: one CTA per (row, batch * KV head).  Thread (chunk group cg,
// channel word c4) sums chunks cg, cg + CG, ... scaled to the final max.
template <int D>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const DecodeArgs a,
                                                                        int nchunks) {
  constexpr int TPC = D / 4;                  // threads per chunk row
  constexpr int CG = kCombineThreads / TPC;   // chunk groups
  __shared__ float wm[kCombineThreads / 32];
  __shared__ __align__(16) float red[CG][D];
  __shared__ float redl[CG];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, bkv = blockIdx.y;
  const int b = bkv / a.Hkv, hkv = bkv % a.Hkv;
  const int G = a.Hq / a.Hkv, R = G * a.Nq;
  const size_t p0 = static_cast<size_t>(bkv) * nchunks * R + r;
  float mf = kNegInf;
  for (int c = threadIdx.x; c < nchunks; c += kCombineThreads)
    mf = fmaxf(mf, a.part_m[p0 + static_cast<size_t>(c) * R]);
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) mf = fmaxf(mf, __shfl_xor_sync(0xffffffffu, mf, s));
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = mf;
  __syncthreads();
  mf = wm[0];
#pragma unroll
  for (int w = 1; w < kCombineThreads / 32; ++w) mf = fmaxf(mf, wm[w]);
  const int c4 = threadIdx.x % TPC, cg = threadIdx.x / TPC;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  if (mf != kNegInf) {
#pragma unroll 4
    for (int c = cg; c < nchunks; c += CG) {
      const size_t pi = p0 + static_cast<size_t>(c) * R;
      const float mc = a.part_m[pi];
      const float lc = a.part_l[pi];
      const float4 oc = *reinterpret_cast<const float4*>(a.part_o + pi * D + 4 * c4);
      const float wgt = (mc == kNegInf) ? 0.f : ex2_approx(mc - mf);
      l = fmaf(wgt, lc, l);
      o.x = fmaf(wgt, oc.x, o.x);
      o.y = fmaf(wgt, oc.y, o.y);
      o.z = fmaf(wgt, oc.z, o.z);
      o.w = fmaf(wgt, oc.w, o.w);
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

template <int D, int RMAX>
cudaError_t launch_decode_r(const DecodeArgs& a, int nkb, int nchunks, cudaStream_t s) {
  const int BHkv = a.B * a.Hkv;
  cudaError_t e = launch_pdl(decode_scores_kernel<D, RMAX>, dim3(nkb, BHkv), dim3(kBlk), 0, s, a);
  if (e != cudaSuccess) return e;
  constexpr int smem = PvSmem<D, RMAX>::kBytes;
  e = cudaFuncSetAttribute(decode_pv_kernel<D, RMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_pv_kernel<D, RMAX>, dim3(nchunks, BHkv), dim3(kPvThreads), smem, s, a);
}

template <int D>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  const int nkb = (a.Nk + kBlk - 1) / kBlk;
  const int nchunks = (nkb + kDecodeChunk - 1) / kDecodeChunk;
  const int R = (a.Hq / a.Hkv) * a.Nq;
  cudaError_t e = (R <= 4) ? launch_decode_r<D, 4>(a, nkb, nchunks, s)
                           : launch_decode_r<D, kMaxDecodeRows>(a, nkb, nchunks, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_combine_kernel<D>, dim3(R, a.B * a.Hkv), dim3(kCombineThreads), 0, s,
                    a, nchunks);
}

}  // namespace

size_t decode_ws_bytes(long long B, long long Hq, long long Hkv, long long Nq, long long Nk,
                       long long d) {
  const long long R = (Hq / Hkv) * Nq;
  const long long nkb = (Nk + kBlk - 1) / kBlk;
  const long long nchunks = (nkb + kDecodeChunk - 1) / kDecodeChunk;
  const long long BH = B * Hkv;
  auto a256 = [](long long x) { return static_cast<size_t>((x + 255) / 256 * 256); };
  return a256(BH * R * nkb * kBlk * 4) +   // t
         a256(BH * nkb * R * 4) +           // block maxima
         a256(BH * nchunks * R * d * 4) +   // chunk O
         2 * a256(BH * nchunks * R * 4);    // chunk l, m
}

cudaError_t launch_decode(DecodeArgs a, void* ws, cudaStream_t s) {
  const long long R = (a.Hq / a.Hkv) * a.Nq;
  const long long nkb = (a.Nk + kBlk - 1) / kBlk;
  const long long nchunks = (nkb + kDecodeChunk - 1) / kDecodeChunk;
  const long long BH = static_cast<long long>(a.B) * a.Hkv;
  auto a256 = [](long long x) { return static_cast<size_t>((x + 255) / 256 * 256); };
  char* p = static_cast<char*>(ws);
  a.t = reinterpret_cast<float*>(p);
  p += a256(BH * R * nkb * kBlk * 4);
  a.mblk = reinterpret_cast<float*>(p);
  p += a256(BH * nkb * R * 4);
  a.part_o = reinterpret_cast<float*>(p);
  p += a256(BH * nchunks * R * a.d * 4);
  a.part_l = reinterpret_cast<float*>(p);
  p += a256(BH * nchunks * R * 4);
  a.part_m = reinterpret_cast<float*>(p);
  return a.d == 64 ? launch_decode_t<64>(a, s) : launch_decode_t<128>(a, s);
}

}  // namespace qattn
