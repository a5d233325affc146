// Fused latent decode attention (split-K) and its combine/epilogue.
//
// Method (page "PALU — True Low-Rank Latent Storage for Keys and Values",
// "How it works", decode step 3 and prefill step 6): attention over the
// reconstructed keys/values K = L^K V_g^T + mu_g.  Because V_g has orthonormal
// columns and the softmax weights sum to one, the same result follows in
// latent space:
//   score_t = scale * (q~ . L^K_t + q . mu^K),       q~ = q V^K
//   out     = (sum_t p_t L^V_t / sum_t p_t) V^V^T + mu^V
// and dequantized latents are L_t[j] = code_tj * s_bj + z_bj per 32-token
// block b.  The kernel never forms fp16 K or V (the page's "Adaptation notes"
// say its port reconstructs fp16 first; this is the fused form instead).
//
// GB300 design:
//  * Per (batch, KV head) stream, the cached 32-token block records are split
//    into chunks, one CTA each; each of the 4 warps walks every 4th block of
//    the chunk through its own ring of shared-memory stages fed by 1-D bulk
//    copies (TMA engine) with mbarrier completion, so many KB per SM are in
//    flight while the warp computes.
//  * Scores run on tensor cores: the block's key codes are the A operand
//    (tokens x channels, exact small integers in bf16, unpacked straight from
//    the packed words into register fragments), and the B operand is
//    q~_j * s_bj for the GQA query heads of the KV head (N = 8), split into a
//    bf16 hi + lo pair for ~16-bit accuracy; the zero-point term
//    sum_j q~_j z_bj + q . mu is added per block.
//  * Online softmax in base 2 (scale * log2 e folded into q~).
//  * Weighted sum on tensor cores: values dequantized to fp16 (one rounding
//    of code*s+z) as the A operand (channels x tokens), the probabilities as
//    the B operand (transposed in registers with movmatrix).
//  * Per-chunk (max, sum, latent accumulator) partials are merged by the
//    combine kernel, which also folds in the unquantized tail tokens and
//    applies V^V^T and + mu^V once per query head.
#include <math.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "palu_internal.cuh"

namespace palu {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

struct DecodeParams {
  CacheView k, v;
  const __half* q;
  float* ws;          // partials [B][Hkv][n_chunks][Gq][2 + rvp]
  int Hq, Hkv, Gq;
  int n_chunks, bpc;  // chunks per stream, blocks per chunk
  int rvp;            // padded value channels = 8 * v.n_oct
  int ns;             // ring stages per warp
  int stage_bytes;    // k.rec_bytes + v.rec_bytes
  int ring_off, merge_off;
  float scale_log2;   // softmax scale * log2(e)
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- key octet: exact codes (bf16 small integers) for the four (token row)
// registers k = 2*m + rh of this lane, plus the B fragment pair (hi, lo) of
// q~ * scale and the lane's share of sum_j q~_j z_j.
__device__ __forceinline__ void key_octet(const uint8_t* kr, int o, int n_hi_oct, int n_lo_oct, int szb, int npad,
                                          int lane, int c, float q0, float q1, uint32_t R[4], uint32_t& bh,
                                          uint32_t& bl, float& beta) {
  constexpr uint32_t M = 0x43004300u;  // bf16x2 (128, 128)
  if (o < n_hi_oct) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(kr + 128 * o + 4 * lane);
#pragma unroll
    for (int k = 0; k < 4; ++k) R[k] = sub_bf16x2(((w >> (4 * k)) & 0x000F000Fu) | M, M);
  } else {
    const int l = o - n_hi_oct, npair = n_lo_oct >> 1;
    const int off = l < 2 * npair ? 128 * n_hi_oct + 128 * (l >> 1) + 4 * lane + 2 * (l & 1)
                                  : 128 * n_hi_oct + 128 * npair + 2 * lane;
    const uint32_t hw = *reinterpret_cast<const uint16_t*>(kr + off);
    const uint32_t w = __byte_perm(hw, 0u, 0x4140);
#pragma unroll
    for (int k = 0; k < 4; ++k) R[k] = sub_bf16x2(((w >> (2 * k)) & 0x00030003u) | M, M);
  }
  const uint32_t s2 = *reinterpret_cast<const uint32_t*>(kr + szb + 16 * o + 4 * c);
  const uint32_t z2 = *reinterpret_cast<const uint32_t*>(kr + szb + 2 * npad + 16 * o + 4 * c);
  const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&s2));
  const float2 zf = __half22float2(*reinterpret_cast<const __half2*>(&z2));
  const float b0 = q0 * sf.x, b1 = q1 * sf.y;
  bh = pack_bf16x2(b0, b1);
  bl = pack_bf16x2(b0 - bf16_lo_to_f32(bh), b1 - bf16_hi_to_f32(bh));
  beta = fmaf(q0, zf.x, fmaf(q1, zf.y, beta));
}

// ---- value octet: fp16 dequantized latents for the four registers
// k = 2*kt + ch of this lane (channel g of the octet, token pairs).
template <bool VQ>
__device__ __forceinline__ void value_octet(const uint8_t* vr, int o, int n_hi_oct, int n_lo_oct, int szb, int lane,
                                            int g, uint32_t Lh[4]) {
  if constexpr (VQ) {
    constexpr uint32_t M = 0x64006400u;  // f16x2 (1024, 1024)
    uint32_t F[4];
    if (o < n_hi_oct) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(vr + 128 * o + 4 * lane);
#pragma unroll
      for (int k = 0; k < 4; ++k) F[k] = sub_f16x2(((w >> (4 * k)) & 0x000F000Fu) | M, M);
    } else {
      const int l = o - n_hi_oct, npair = n_lo_oct >> 1;
      const int off = l < 2 * npair ? 128 * n_hi_oct + 128 * (l >> 1) + 4 * lane + 2 * (l & 1)
                                    : 128 * n_hi_oct + 128 * npair + 2 * lane;
      const uint32_t hw = *reinterpret_cast<const uint16_t*>(vr + off);
      const uint32_t w = __byte_perm(hw, 0u, 0x4140);
#pragma unroll
      for (int k = 0; k < 4; ++k) F[k] = sub_f16x2(((w >> (2 * k)) & 0x00030003u) | M, M);
    }
    const uint32_t sz = *reinterpret_cast<const uint32_t*>(vr + szb + 4 * (8 * o + g));
    const uint32_t s2 = __byte_perm(sz, sz, 0x1010), z2 = __byte_perm(sz, sz, 0x3232);
#pragma unroll
    for (int k = 0; k < 4; ++k) Lh[k] = fma_f16x2(F[k], s2, z2);
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(vr + 512 * o + 16 * lane);
    Lh[0] = w.x;
    Lh[1] = w.y;
    Lh[2] = w.z;
    Lh[3] = w.w;
  }
}

template <int MAXKT, int MAXVT, bool VQ>
__global__ void __launch_bounds__(kThreads) latent_decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  float* q_s = reinterpret_cast<float*>(smem);        // [8][128]
  float* qt_s = q_s + 8 * kHeadDim;                    // [8][128] scaled q~ per padded key channel
  float* cq_s = qt_s + 8 * kHeadDim;                   // [8] scaled q . mu^K
  int* flag_s = reinterpret_cast<int*>(cq_s + 8);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 8 * kHeadDim * 4 * 2 + 64);
  uint8_t* ring = smem + p.ring_off;
  float* merge = reinterpret_cast<float*>(smem + p.merge_off);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int chunk = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int rvp = p.rvp, Gq = p.Gq;
  const long long len = __ldcg(&p.k.hdr->length);
  const long long n_full = len / kBlock;
  const long long blk0 = (long long)chunk * p.bpc;
  const long long blk1 = min(blk0 + (long long)p.bpc, n_full);
  float* part = p.ws + (((long long)b * p.Hkv + kh) * p.n_chunks + chunk) * (long long)Gq * (2 + rvp);

  if (tid == 0 && chunk == 0 && __ldcg(&p.v.hdr->length) != len) set_dev_error(p.k.hdr, PALU_DEVERR_LENGTH_MISMATCH);
  if (blk0 >= blk1) {
    for (int i = tid; i < Gq * (2 + rvp); i += kThreads) part[i] = (i % (2 + rvp)) == 0 ? -INFINITY : 0.f;
    return;
  }

  // ---- prologue: q, q~ (scaled, per padded key channel), c = q . mu^K (scaled)
  const int gk = kh / p.k.heads_per_group;
  for (int i = tid; i < 8 * kHeadDim; i += kThreads) {
    const int h = i / kHeadDim, d = i % kHeadDim;
    q_s[i] = h < Gq ? __half2float(p.q[((long long)b * p.Hq + (long long)kh * Gq + h) * kHeadDim + d]) : 0.f;
  }
  if (tid == 0) *flag_s = 0;
  if (lane == 0) {
    for (int s = 0; s < p.ns; ++s) mbar_init(&bars[warp * p.ns + s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  {
    const int pch = tid;
    const int rkp = 8 * p.k.n_oct;
    const int j = pch < rkp ? padded_to_channel(pch, p.k.r, p.k.n_hi, p.k.n_hi_oct, 1) : -1;
    float acc[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) acc[h] = 0.f;
    if (j >= 0) {
      const float4* row = reinterpret_cast<const float4*>(p.k.basisT + ((size_t)gk * p.k.r + j) * kHeadDim);
      for (int d4 = 0; d4 < kHeadDim / 4; ++d4) {
        const float4 vv = row[d4];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const float* qq = q_s + h * kHeadDim + 4 * d4;
          acc[h] = fmaf(qq[0], vv.x, fmaf(qq[1], vv.y, fmaf(qq[2], vv.z, fmaf(qq[3], vv.w, acc[h]))));
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 8; ++h) qt_s[h * kHeadDim + pch] = (h < Gq && j >= 0) ? acc[h] * p.scale_log2 : 0.f;
    if (tid < 8) {
      float s = 0.f;
      if (tid < Gq)
        for (int d = 0; d < kHeadDim; ++d) s = fmaf(q_s[tid * kHeadDim + d], p.k.mu[(size_t)gk * kHeadDim + d], s);
      cq_s[tid] = s * p.scale_log2;
    }
  }
  __syncthreads();

  const int n_oct_k = p.k.n_oct, n_oct_v = p.v.n_oct;
  const int KT = (n_oct_k + 1) >> 1, VT = (n_oct_v + 1) >> 1;
  float qk[2 * MAXKT][2];
#pragma unroll
  for (int o = 0; o < 2 * MAXKT; ++o) {
    qk[o][0] = o < n_oct_k ? qt_s[g * kHeadDim + 8 * o + 2 * c] : 0.f;
    qk[o][1] = o < n_oct_k ? qt_s[g * kHeadDim + 8 * o + 2 * c + 1] : 0.f;
  }
  const float cq = cq_s[g];
  const int szb_k = 128 * p.k.n_hi_oct + 64 * p.k.n_lo_oct, npad_k = 8 * n_oct_k;
  const int szb_v = 128 * p.v.n_hi_oct + 64 * p.v.n_lo_oct;
  const int rec_k = p.k.rec_bytes, rec_v = p.v.rec_bytes;

  // ---- this warp's blocks: blk0 + warp + 4 i
  const long long first = blk0 + warp;
  const int n_my = first < blk1 ? (int)((blk1 - first + kWarps - 1) / kWarps) : 0;
  uint8_t* wring = ring + (size_t)warp * p.ns * p.stage_bytes;
  uint64_t* wbar = bars + warp * p.ns;
  const long long stream = (long long)b * p.Hkv + kh;
  const uint8_t* kbase = p.k.blocks + stream * p.k.n_blk_cap * rec_k;
  const uint8_t* vbase = p.v.blocks + stream * p.v.n_blk_cap * rec_v;
  auto issue = [&](int i) {
    const int s = i % p.ns;
    const long long blk = first + (long long)i * kWarps;
    uint8_t* dst = wring + (size_t)s * p.stage_bytes;
    mbar_arrive_expect_tx(&wbar[s], (uint32_t)p.stage_bytes);
    bulk_g2s(dst, kbase + blk * rec_k, (uint32_t)rec_k, &wbar[s]);
    bulk_g2s(dst + rec_k, vbase + blk * rec_v, (uint32_t)rec_v, &wbar[s]);
  };
  if (lane == 0) {
    for (int i = 0; i < n_my && i < p.ns; ++i) issue(i);
  }
  __syncwarp();

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float acc[MAXVT][4];
#pragma unroll
  for (int mt = 0; mt < MAXVT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  int done = 0;
  bool timed_out = false;
  for (int i = 0; i < n_my; ++i) {
    const int s = i % p.ns;
    const uint32_t par = (uint32_t)((i / p.ns) & 1);
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&wbar[s], par));
    if (!ok) {
      timed_out = true;
      break;
    }
    const uint8_t* kr = wring + (size_t)s * p.stage_bytes;
    const uint8_t* vr = kr + rec_k;

    // ---- scores: C[token, head] over 2 m-tiles of 16 tokens
    float sc[2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m) sc[m][0] = sc[m][1] = sc[m][2] = sc[m][3] = 0.f;
    float beta = 0.f;
#pragma unroll
    for (int kt = 0; kt < MAXKT; ++kt) {
      if (kt < KT) {
        uint32_t RA[4], RB[4], bhA, blA, bhB = 0u, blB = 0u;
        key_octet(kr, 2 * kt, p.k.n_hi_oct, p.k.n_lo_oct, szb_k, npad_k, lane, c, qk[2 * kt][0], qk[2 * kt][1], RA,
                  bhA, blA, beta);
        if (2 * kt + 1 < n_oct_k) {
          key_octet(kr, 2 * kt + 1, p.k.n_hi_oct, p.k.n_lo_oct, szb_k, npad_k, lane, c, qk[2 * kt + 1][0],
                    qk[2 * kt + 1][1], RB, bhB, blB, beta);
        } else {
          RB[0] = RB[1] = RB[2] = RB[3] = 0u;
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          mma_bf16(sc[m], RA[2 * m], RA[2 * m + 1], RB[2 * m], RB[2 * m + 1], bhA, bhB);
          mma_bf16(sc[m], RA[2 * m], RA[2 * m + 1], RB[2 * m], RB[2 * m + 1], blA, blB);
        }
      }
    }
    beta += __shfl_xor_sync(0xffffffffu, beta, 1);
    beta += __shfl_xor_sync(0xffffffffu, beta, 2);
    beta += cq;  // head g
    const float be0 = __shfl_sync(0xffffffffu, beta, 8 * c);      // head 2c
    const float be1 = __shfl_sync(0xffffffffu, beta, 8 * c + 4);  // head 2c + 1
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      sc[m][0] += be0;
      sc[m][1] += be1;
      sc[m][2] += be0;
      sc[m][3] += be1;
    }

    // ---- online softmax (base 2) for heads 2c, 2c+1
    float bm0 = fmaxf(fmaxf(sc[0][0], sc[0][2]), fmaxf(sc[1][0], sc[1][2]));
    float bm1 = fmaxf(fmaxf(sc[0][1], sc[0][3]), fmaxf(sc[1][1], sc[1][3]));
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, x));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, x));
    }
    const float mn0 = fmaxf(m_run[0], bm0), mn1 = fmaxf(m_run[1], bm1);
    const float al0 = ex2(m_run[0] - mn0), al1 = ex2(m_run[1] - mn1);
    m_run[0] = mn0;
    m_run[1] = mn1;
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < MAXVT; ++mt) {
        acc[mt][0] *= al0;
        acc[mt][1] *= al1;
        acc[mt][2] *= al0;
        acc[mt][3] *= al1;
      }
      l_run[0] *= al0;
      l_run[1] *= al1;
    }
    float pr[2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      pr[m][0] = ex2(sc[m][0] - mn0);
      pr[m][1] = ex2(sc[m][1] - mn1);
      pr[m][2] = ex2(sc[m][2] - mn0);
      pr[m][3] = ex2(sc[m][3] - mn1);
    }
    l_run[0] += (pr[0][0] + pr[0][2]) + (pr[1][0] + pr[1][2]);
    l_run[1] += (pr[0][1] + pr[0][3]) + (pr[1][1] + pr[1][3]);
    // probabilities as the B operand (tokens x heads): transpose the 8x8 pieces
    uint32_t pb[2][2];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      pb[m][0] = movmatrix_t(pack_f16x2(pr[m][0], pr[m][1]));
      pb[m][1] = movmatrix_t(pack_f16x2(pr[m][2], pr[m][3]));
    }

    // ---- weighted sum of value latents: C[channel, head] += L^T P
#pragma unroll
    for (int mt = 0; mt < MAXVT; ++mt) {
      if (mt < VT) {
        uint32_t LA[4], LB[4];
        value_octet<VQ>(vr, 2 * mt, p.v.n_hi_oct, p.v.n_lo_oct, szb_v, lane, g, LA);
        if (2 * mt + 1 < n_oct_v) {
          value_octet<VQ>(vr, 2 * mt + 1, p.v.n_hi_oct, p.v.n_lo_oct, szb_v, lane, g, LB);
        } else {
          LB[0] = LB[1] = LB[2] = LB[3] = 0u;
        }
        mma_f16(acc[mt], LA[0], LB[0], LA[1], LB[1], pb[0][0], pb[0][1]);
        mma_f16(acc[mt], LA[2], LB[2], LA[3], LB[3], pb[1][0], pb[1][1]);
      }
    }
    __syncwarp();
    if (lane == 0 && i + p.ns < n_my) issue(i + p.ns);
    done = i + 1;
  }

  if (timed_out) {
    // drain this warp's copies still in flight (bounded), then report
    if (lane == 0) {
      set_dev_error(p.k.hdr, PALU_DEVERR_TIMEOUT);
      for (int i = done; i < n_my && i < done + p.ns; ++i) mbar_wait_bounded(&wbar[i % p.ns], (uint32_t)((i / p.ns) & 1));
      atomicOr(flag_s, 1);
    }
  }

  // ---- merge the 4 warps of the CTA
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], x);
    l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], x);
  }
  const int mstride = 2 + rvp;
  float* mw = merge + warp * 8 * mstride;
  if (g == 0) {
    mw[(2 * c) * mstride + 0] = n_my > 0 ? m_run[0] : -INFINITY;
    mw[(2 * c) * mstride + 1] = l_run[0];
    mw[(2 * c + 1) * mstride + 0] = n_my > 0 ? m_run[1] : -INFINITY;
    mw[(2 * c + 1) * mstride + 1] = l_run[1];
  }
#pragma unroll
  for (int mt = 0; mt < MAXVT; ++mt) {
    if (mt < VT) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int pch = 16 * mt + g + 8 * (e >> 1);
        const int h = 2 * c + (e & 1);
        if (pch < rvp) mw[h * mstride + 2 + pch] = acc[mt][e];
      }
    }
  }
  __syncthreads();
  if (*flag_s) {
    for (int i = tid; i < Gq * mstride; i += kThreads) part[i] = (i % mstride) == 0 ? -INFINITY : 0.f;
    return;
  }
  for (int i = tid; i < Gq * mstride; i += kThreads) {
    const int h = i / mstride, e = i % mstride;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, merge[(w * 8 + h) * mstride]);
    float out;
    if (e == 0) {
      out = M;
    } else {
      out = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw_ = merge[(w * 8 + h) * mstride];
        if (mw_ != -INFINITY) out += merge[(w * 8 + h) * mstride + e] * ex2(mw_ - M);
      }
    }
    part[i] = out;
  }
}

// One CTA of 8 warps per (batch, KV head); warp h finishes query head h:
// merge the chunk partials (log-sum-exp), fold in the unquantized tail tokens
// in fp32, then apply V^V^T and + mu^V once.  Every loop runs across lanes,
// so the kernel is a handful of dependent memory round trips long.
__global__ void __launch_bounds__(256) latent_combine_kernel(const DecodeParams p, void* out, int out_fp32) {
  __shared__ float q_s[8][kHeadDim];
  __shared__ float qt_s[8][kMaxRank];
  __shared__ float ol_s[8][kMaxRank];
  __shared__ float pt_s[8][kBlock];
  const int tid = threadIdx.x, h = tid >> 5, lane = tid & 31;
  const int kh = blockIdx.x, b = blockIdx.y;
  const int Gq = p.Gq, rvp = p.rvp, mstride = 2 + rvp;
  if (h >= Gq) return;
  const long long len = __ldcg(&p.k.hdr->length);
  const long long n_full = len / kBlock;
  const int n_tail = (int)(len % kBlock);
  const int gk = kh / p.k.heads_per_group, gv = kh / p.v.heads_per_group;
  const int rk = p.k.r, rv = p.v.r;
  const long long stream = (long long)b * p.Hkv + kh;
  const float* wpart = p.ws + stream * p.n_chunks * (long long)Gq * mstride + (long long)h * mstride;
  const long long cstride = (long long)Gq * mstride;

  // chunk maxima
  float M = -INFINITY;
  for (int ch = lane; ch < p.n_chunks; ch += 32) M = fmaxf(M, __ldcg(wpart + ch * cstride));
  // tail scores: lane t < n_tail owns token t
  float st = -INFINITY;
  if (n_tail > 0) {
    const __half* qh = p.q + ((long long)b * p.Hq + (long long)kh * Gq + h) * kHeadDim;
    for (int d = lane; d < kHeadDim; d += 32) q_s[h][d] = __half2float(qh[d]);
    __syncwarp();
    for (int j = lane; j < rk; j += 32) {
      const float4* row = reinterpret_cast<const float4*>(p.k.basisT + ((size_t)gk * rk + j) * kHeadDim);
      float a = 0.f;
#pragma unroll 8
      for (int d4 = 0; d4 < kHeadDim / 4; ++d4) {
        const float4 v = row[d4];
        a = fmaf(q_s[h][4 * d4], v.x,
                 fmaf(q_s[h][4 * d4 + 1], v.y, fmaf(q_s[h][4 * d4 + 2], v.z, fmaf(q_s[h][4 * d4 + 3], v.w, a))));
      }
      qt_s[h][j] = a;
    }
    float c = 0.f;
    for (int d = lane; d < kHeadDim; d += 32) c = fmaf(q_s[h][d], p.k.mu[(size_t)gk * kHeadDim + d], c);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    __syncwarp();
    if (lane < n_tail) {
      const float* tk = p.k.tail + (stream * kBlock + lane) * rk;
      float a = 0.f;
      for (int j = 0; j < rk; ++j) a = fmaf(qt_s[h][j], tk[j], a);
      st = (a + c) * p.scale_log2;
      M = fmaxf(M, st);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  // denominator
  float L = 0.f;
  for (int ch = lane; ch < p.n_chunks; ch += 32) {
    const float m = __ldcg(wpart + ch * cstride);
    if (m != -INFINITY) L += __ldcg(wpart + ch * cstride + 1) * ex2(m - M);
  }
  const float pt = lane < n_tail ? ex2(st - M) : 0.f;
  pt_s[h][lane] = pt;
  L += pt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float invL = 1.f / L;
  // latent accumulator per padded value channel, stored by real channel
  for (int pch = lane; pch < rvp; pch += 32) {
    const int j = padded_to_channel(pch, rv, p.v.n_hi, p.v.n_hi_oct, p.v.quantize);
    float a = 0.f;
    for (int ch = 0; ch < p.n_chunks; ++ch) {
      const float m = __ldcg(wpart + ch * cstride);
      if (m != -INFINITY) a = fmaf(__ldcg(wpart + ch * cstride + 2 + pch), ex2(m - M), a);
    }
    if (j >= 0) ol_s[h][j] = a;
  }
  __syncwarp();
  if (n_tail > 0) {
    for (int j = lane; j < rv; j += 32) {
      float a = ol_s[h][j];
      for (int t = 0; t < n_tail; ++t) {
        float lv;
        if (p.v.quantize) {
          lv = p.v.tail[(stream * kBlock + t) * rv + j];
        } else {
          const uint8_t* rec = p.v.blocks + (stream * p.v.n_blk_cap + n_full) * p.v.rec_bytes;
          const int k = 2 * (t >> 4) + ((t & 15) >> 3);
          const int ln = 4 * (j & 7) + ((t & 7) >> 1);
          lv = __half2float(*reinterpret_cast<const __half*>(rec + 512 * (j >> 3) + 16 * ln + 4 * k + 2 * (t & 1)));
        }
        a = fmaf(pt_s[h][t], lv, a);
      }
      ol_s[h][j] = a;
    }
  }
  __syncwarp();
  // epilogue: out[d] = (sum_j o_j V[d, j]) / L + mu[d]
  const float* bt = p.v.basisT + (size_t)gv * rv * kHeadDim;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int j = 0; j < rv; ++j) {
    const float oj = ol_s[h][j];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = fmaf(oj, bt[(size_t)j * kHeadDim + lane + 32 * e], o[e]);
  }
  const long long oi = ((long long)b * p.Hq + (long long)kh * Gq + h) * kHeadDim;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int d = lane + 32 * e;
    const float v = fmaf(o[e], invL, p.v.mu[(size_t)gv * kHeadDim + d]);
    if (out_fp32)
      static_cast<float*>(out)[oi + d] = v;
    else
      static_cast<__half*>(out)[oi + d] = __float2half_rn(v);
  }
}

// ------------------------------------------------------------------ host
struct DecodePlan {
  int MAXKT, MAXVT;
  bool VQ;
  int ns, stage_bytes, ring_off, merge_off, smem;
  int n_chunks, bpc, rvp;
  size_t ws_bytes;
};

static int round_tiles(int t) { return t <= 1 ? 1 : t <= 2 ? 2 : t <= 4 ? 4 : 8; }

typedef void (*DecodeKernel)(const DecodeParams);

static DecodeKernel pick_kernel(int kt, int vt, bool vq) {
#define PALU_K(A, B)                                                                     \
  if (kt == A && vt == B) return vq ? latent_decode_kernel<A, B, true> : latent_decode_kernel<A, B, false>;
  PALU_K(1, 1) PALU_K(1, 2) PALU_K(1, 4) PALU_K(1, 8)
  PALU_K(2, 1) PALU_K(2, 2) PALU_K(2, 4) PALU_K(2, 8)
  PALU_K(4, 1) PALU_K(4, 2) PALU_K(4, 4) PALU_K(4, 8)
  PALU_K(8, 1) PALU_K(8, 2) PALU_K(8, 4) PALU_K(8, 8)
#undef PALU_K
  return nullptr;
}

static palu_status plan_decode(const palu_cache* k, const palu_cache* v, int32_t Hq, DecodePlan* pl) {
  if (!k || !v || k->magic != kCacheMagic || v->magic != kCacheMagic)
    return fail(PALU_ERR_NOT_INITIALIZED, "key and value caches must be initialised");
  if (k->role != PALU_ROLE_KEY || v->role != PALU_ROLE_VALUE)
    return fail(PALU_ERR_INVALID_ARG, "k must be a key cache and v a value cache");
  if (k->batch != v->batch || k->kv_heads != v->kv_heads || k->capacity != v->capacity)
    return fail(PALU_ERR_INVALID_ARG, "key and value caches differ in batch, kv_heads or capacity");
  if (Hq < 1 || Hq % k->kv_heads != 0) return fail(PALU_ERR_INVALID_ARG, "q_heads must be a positive multiple of kv_heads");
  const int Gq = Hq / k->kv_heads;
  if (Gq > kMaxGq) return fail(PALU_ERR_UNSUPPORTED, "at most 8 query heads per KV head are supported");
  pl->MAXKT = round_tiles((k->n_oct + 1) / 2);
  pl->MAXVT = round_tiles((v->n_oct + 1) / 2);
  pl->VQ = v->quantize != 0;
  pl->stage_bytes = k->record_bytes + v->record_bytes;
  pl->ns = std::max(2, std::min(8, (64 * 1024) / (kWarps * pl->stage_bytes)));
  pl->rvp = 8 * v->n_oct;
  const int head = 8 * kHeadDim * 4 * 2 + 64;
  pl->ring_off = (int)align_up(head + 8 * kWarps * pl->ns, 128);
  pl->merge_off = (int)align_up(pl->ring_off + kWarps * pl->ns * pl->stage_bytes, 16);
  pl->smem = pl->merge_off + kWarps * 8 * (2 + pl->rvp) * 4;
  DecodeKernel kern = pick_kernel(pl->MAXKT, pl->MAXVT, pl->VQ);
  if (!kern) return fail(PALU_ERR_UNSUPPORTED, "no decode kernel for this rank");
  int per_sm = 0;
  palu_status st = kernel_occupancy(reinterpret_cast<const void*>(kern), kThreads, pl->smem, &per_sm);
  if (st != PALU_OK) return st;
  const int64_t streams = (int64_t)k->batch * k->kv_heads;
  const int64_t target = (int64_t)device_sm_count() * per_sm;
  int64_t nch = std::max<int64_t>(1, target / streams);
  nch = std::min<int64_t>(nch, std::max<int64_t>(1, k->n_blk_cap));
  const int64_t bpc = (k->n_blk_cap + nch - 1) / nch;
  nch = (k->n_blk_cap + bpc - 1) / bpc;
  pl->n_chunks = (int)std::max<int64_t>(1, nch);
  pl->bpc = (int)std::max<int64_t>(1, bpc);
  pl->ws_bytes = align_up(sizeof(float) * (size_t)streams * pl->n_chunks * Gq * (2 + pl->rvp), 256);
  return PALU_OK;
}

}  // namespace palu

using namespace palu;

extern "C" palu_status palu_decode_workspace_size(const palu_cache* k, const palu_cache* v, int32_t q_heads,
                                                  size_t* bytes) {
  DecodePlan pl;
  palu_status st = plan_decode(k, v, q_heads, &pl);
  if (st != PALU_OK) return st;
  if (!bytes) return fail(PALU_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = pl.ws_bytes;
  return PALU_OK;
}

extern "C" palu_status palu_decode_attn(const palu_cache* k, const palu_cache* v, const void* q, int32_t q_heads,
                                        float softmax_scale, void* out, int32_t out_fp32, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  DecodePlan pl;
  palu_status st = plan_decode(k, v, q_heads, &pl);
  if (st != PALU_OK) return st;
  if (!q || !out || !workspace) return fail(PALU_ERR_INVALID_ARG, "q, out and workspace must be non-NULL");
  if (((uintptr_t)q & 15) || ((uintptr_t)out & 15) || ((uintptr_t)workspace & 15))
    return fail(PALU_ERR_INVALID_ARG, "q, out and workspace must be 16-byte aligned");
  if (workspace_bytes < pl.ws_bytes)
    return fail(PALU_ERR_INVALID_ARG, "workspace too small: need " + std::to_string(pl.ws_bytes) + " bytes");
  if (k->length != v->length) return fail(PALU_ERR_INVALID_ARG, "key and value caches differ in length");
  if (k->length < 1) return fail(PALU_ERR_INVALID_ARG, "the caches are empty");
  DecodeParams p;
  p.k = make_view(k);
  p.v = make_view(v);
  p.q = static_cast<const __half*>(q);
  p.ws = static_cast<float*>(workspace);
  p.Hq = q_heads;
  p.Hkv = k->kv_heads;
  p.Gq = q_heads / k->kv_heads;
  p.n_chunks = pl.n_chunks;
  p.bpc = pl.bpc;
  p.rvp = pl.rvp;
  p.ns = pl.ns;
  p.stage_bytes = pl.stage_bytes;
  p.ring_off = pl.ring_off;
  p.merge_off = pl.merge_off;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)kHeadDim);
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  DecodeKernel kern = pick_kernel(pl.MAXKT, pl.MAXVT, pl.VQ);
  kern<<<dim3(pl.n_chunks, k->kv_heads, k->batch), kThreads, pl.smem, strm>>>(p);
  st = cuda_check(cudaGetLastError(), "latent_decode_kernel launch");
  if (st != PALU_OK) return st;
  latent_combine_kernel<<<dim3(k->kv_heads, k->batch), 256, 0, strm>>>(p, out, out_fp32);
  return cuda_check(cudaGetLastError(), "latent_combine_kernel launch");
}

// ------------------------------------------------------------------ allocation-free decode
// Some callers cannot allocate device memory while they decode: a plugin whose
// host application owns every device allocation, a serving loop that forbids
// allocation between steps to keep latency predictable, or a process whose
// device memory is already reserved in full by another pool.  For them
// palu_decode_attn_noalloc keeps the split-K partials in this fixed array,
// which every GPU that loads the library holds until the process exits.
namespace palu {
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of the scratch on the current device, looked up once per
// device.  In host code the array's name is only a stand-in for the symbol.
static palu_status noalloc_scratch(void** ptr) {
  static std::mutex mu;
  static std::map<int, void*> addr;
  int dev = 0;
  palu_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != PALU_OK) return st;
  std::lock_guard<std::mutex> lock(mu);
  auto it = addr.find(dev);
  if (it != addr.end()) {
    *ptr = it->second;
    return PALU_OK;
  }
  void* p = nullptr;
  st = cuda_check(cudaGetSymbolAddress(&p, g_decode_scratch), "cudaGetSymbolAddress(decode scratch)");
  if (st != PALU_OK) return st;
  addr[dev] = p;
  *ptr = p;
  return PALU_OK;
}
}  // namespace palu

extern "C" palu_status palu_decode_attn_noalloc(const palu_cache* k, const palu_cache* v, const void* q,
                                                int32_t q_heads, float softmax_scale, void* out, int32_t out_fp32,
                                                void* stream) {
  DecodePlan pl;
  palu_status st = plan_decode(k, v, q_heads, &pl);
  if (st != PALU_OK) return st;
  if (pl.ws_bytes > kNoAllocScratchBytes)
    return fail(PALU_ERR_UNSUPPORTED, "palu_decode_attn_noalloc: these caches need " + std::to_string(pl.ws_bytes) +
                                          " bytes of scratch but the library's fixed scratch holds " +
                                          std::to_string(kNoAllocScratchBytes) +
                                          "; call palu_decode_attn with a workspace instead");
  void* ws = nullptr;
  st = noalloc_scratch(&ws);
  if (st != PALU_OK) return st;
  return palu_decode_attn(k, v, q, q_heads, softmax_scale, out, out_fp32, ws, kNoAllocScratchBytes, stream);
}
