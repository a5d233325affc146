// Fused latent decode attention: one persistent kernel per call.
//
// Method (page "PALU — True Low-Rank Latent Storage for Keys and Values",
// "How it works", decode step 3 and prefill step 6): attention over the
// reconstructed keys/values K = L^K V_g^T + mu_g.  Because V_g has orthonormal
// columns and the softmax weights sum to one, the same result follows in
// latent space:
//   score_t = scale * (q~ . L^K_t + q . mu^K),       q~ = q V^K
//   out     = (sum_t p_t L^V_t / sum_t p_t) V^V^T + mu^V
// with dequantized latents L_t[j] = code_tj * s_bj + z_bj per 32-token block
// b.  No fp16 K or V is ever formed (the page's "Adaptation notes" describe a
// port that reconstructs fp16 first; this is the fused form instead).
//
// GB300 design:
//  * Persistent grid (resident CTAs only).  The flat range of full 32-token
//    blocks over all (batch, KV head) streams is split evenly over the CTAs, so
//    every SM gets the same number of blocks whatever the batch and head count.
//    A CTA walks its range stream by stream ("segments"); each of its 8 warps
//    takes a contiguous share of the segment and streams it through its own
//    ring of shared-memory stages (2 blocks of key and value records per stage,
//    two 1-D bulk copies on the TMA engine, mbarrier completion).  The first
//    stages are in flight before the per-segment prologue (q~ = q V^K) runs.
//  * Scores on tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate):
//    tokens x channels of exact small-integer codes as A, and as B the
//    query-side factor q~_j * s_bj for the GQA heads (N = 8) in fp16 as a
//    hi + lo pair (error-free HMUL2/HFMA2 split), with q~ prescaled by a power
//    of two so that every product stays inside fp16 range.  The zero-point
//    term sum_j q~_j z_bj rides on the same accumulators: an A operand whose
//    rows all hold z_b.  Codes are unpacked with one LOP3 per register pair
//    against per-field fp16 "magic" exponents, then one HSUB2.
//  * Online softmax in base 2 with a lazy running maximum: the maximum is only
//    raised (and the accumulators rescaled) when a score exceeds it by more
//    than 2^8, so the common path has no cross-lane reduction.  The row sums
//    come out of the tensor cores too (an all-ones A operand).
//  * Weighted sum on tensor cores: values dequantized once to fp16
//    (HFMA2 code*s+z) as A (channels x tokens), the probabilities as B.
//  * Each CTA merges its warps (log-sum-exp) into one partial per segment; a
//    per-stream ticket in the key cache's state picks the last contributor,
//    which merges the stream's partials, folds in the fp32 tail tokens and
//    applies V^V^T and + mu^V once per query head.
#pragma once

#include <math.h>

#include "palu_internal.cuh"

namespace palu {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = 32 * kDecWarps;
constexpr float kLazyTau = 8.f;     // log2 headroom before the running max is raised
// shared-memory header of a decode CTA (byte offsets)
constexpr int kDecQOff = 0;                           // q_s   fp32 [8][128]
constexpr int kDecQtOff = 4096;                       // qt_s  fp32 [8][128] scaled q~ per padded key channel
constexpr int kDecMuOff = 8192;                       // mu_s  fp32 [128]
constexpr int kDecCqOff = 8704;                       // cq_s  fp32 [8]
constexpr int kDecRedOff = 8736;                      // red_s fp32 [8]
constexpr int kDecFlagOff = 8768;                     // flags int [4]
constexpr int kDecBsOff = 8832;                       // B_s   fp32 [32][129] key basis rows (prologue)
constexpr int kDecBarOff = kDecBsOff + 32 * 129 * 4;  // mbarriers: [warps][ns], then the merge barrier

struct DecodeParams {
  CacheView k, v;
  const __half* q;
  void* out;
  float* ws;          // partials [streams][seg_max][Gq][2 + rvp]
  int out_fp32;
  int Hq, Hkv, Gq;
  int rvp;            // padded value channels = 8 * v.n_oct
  int ns;             // stages per warp ring
  int stage_bytes;    // 2 * (k.rec_bytes + v.rec_bytes)
  int ring_off;       // shared-memory offset of the rings (reused by the merges)
  int seg_max;        // partial slots per stream
  long long streams;  // batch * kv_heads
  float scale_log2;   // softmax scale * log2(e)
};

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// a * b - c, rounded once
__device__ __forceinline__ uint32_t hfms2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("{\n\t.reg .b32 t;\n\tneg.f16x2 t, %3;\n\tfma.rn.f16x2 %0, %1, %2, t;\n\t}"
      : "=r"(d)
      : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint32_t ld32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint32_t ld16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }

// 2^e as a float for |e| <= 126.
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

// ---- code unpack: 8 codes of one octet for this lane -> 4 fp16x2 registers
// holding the exact small integers.  Field k of the lane's word sits at bits
// 4k (4-bit) or 2k (2-bit) of each 16-bit half; OR-ing the field into the
// mantissa of an fp16 power of two 2^E whose unit in the last place lines up
// with the field's lowest bit gives 2^E + code, and one subtraction leaves the
// code.
__device__ __forceinline__ void unpack_hi(uint32_t w, uint32_t R[4]) {
  const uint32_t w8 = w >> 8;
  R[0] = sub_f16x2((w & 0x000F000Fu) | 0x64006400u, 0x64006400u);   // 1024 + c
  R[1] = sub_f16x2((w & 0x00F000F0u) | 0x54005400u, 0x54005400u);   //   64 + c
  R[2] = sub_f16x2((w8 & 0x000F000Fu) | 0x64006400u, 0x64006400u);
  R[3] = sub_f16x2((w8 & 0x00F000F0u) | 0x54005400u, 0x54005400u);
}
// hw: the octet's 16 bits (half 0 in bits 0-7, half 1 in bits 8-15).
__device__ __forceinline__ void unpack_lo(uint32_t hw, uint32_t R[4]) {
  const uint32_t w = __byte_perm(hw, 0u, 0x4140);
  R[0] = sub_f16x2((w & 0x00030003u) | 0x64006400u, 0x64006400u);   // 1024 + c
  R[1] = sub_f16x2((w & 0x000C000Cu) | 0x5C005C00u, 0x5C005C00u);   //  256 + c
  R[2] = sub_f16x2((w & 0x00300030u) | 0x54005400u, 0x54005400u);   //   64 + c
  R[3] = sub_f16x2((w & 0x00C000C0u) | 0x4C004C00u, 0x4C004C00u);   //   16 + c
}

// Record geometry of one cache as the kernel sees it.  C is the record class
// ceil(n_oct / 4) (for quantized records: the number of 4-bit octets); E is
// the exact octet count when it is a template argument (every offset is then
// a compile-time constant and no octet needs a presence test), or 0, in which
// case the counts are read from the cache and the last three octets of the
// class are tested at run time.
template <int C, int E, bool Q>
struct Geom {
  static constexpr int kMaxOct = E ? E : 4 * C;
  int n_oct_, sz_, z_, single_, rec_;
  __device__ __forceinline__ void init(const CacheView& v) {
    n_oct_ = v.n_oct;
    sz_ = 128 * v.n_hi_oct + 64 * v.n_lo_oct;
    z_ = sz_ + 16 * v.n_oct;
    single_ = (v.n_lo_oct & 1) ? v.n_oct - 1 : -1;
    rec_ = v.rec_bytes;
  }
  __device__ __forceinline__ bool present(int o) const {
    if constexpr (E > 0) return o < E;
    else return o < 4 * C - 3 || o < n_oct_;
  }
  __device__ __forceinline__ int sz() const {
    if constexpr (E > 0) return 128 * C + 64 * (E - C);
    else return sz_;
  }
  __device__ __forceinline__ int z() const {
    if constexpr (E > 0) return 128 * C + 64 * (E - C) + 16 * E;
    else return z_;
  }
  __device__ __forceinline__ int rec() const {
    if constexpr (E > 0) return Q ? 128 * C + 64 * (E - C) + 32 * E : 512 * E;
    else return rec_;
  }
  // lo octet stored alone (odd number of lo octets: the last one)
  __device__ __forceinline__ bool single(int o) const {
    if constexpr (E > 0) return ((E - C) & 1) && o == E - 1;
    else return o == single_;
  }
  // byte offset of octet o's word for this lane: a u32 for 4-bit octets, the
  // lane's u16 for 2-bit octets (pairs share u32 words, a lone one has u16s)
  __device__ __forceinline__ int word_off(int o, int lane) const {
    if (o < C) return 128 * o + 4 * lane;
    const int l = o - C;
    const int base = 128 * C + 128 * (l >> 1) + 2 * (l & 1);
    return base + (single(o) ? 2 : 4) * lane;
  }
};

__device__ __forceinline__ void mma16816_c(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1, const float c[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}
__device__ __forceinline__ void mma16816_0(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// One key octet of one block: exact codes, the B pair (hi, lo) of
// Q~ * s for the lane's head g and channels 2c, 2c+1, and the zero points.
template <class GK>
__device__ __forceinline__ void key_octet(const uint8_t* kr, const GK& gk, int o, uint32_t qh, uint32_t ql,
                                          int lane, int c, uint32_t R[4], uint32_t& bh, uint32_t& bl,
                                          uint32_t& z) {
  constexpr int KC = (GK::kMaxOct + 3) / 4;
  if (o < KC) unpack_hi(ld32(kr + gk.word_off(o, lane)), R);
  else unpack_lo(ld16(kr + gk.word_off(o, lane)), R);
  const uint32_t s2 = ld32(kr + gk.sz() + 16 * o + 4 * c);
  z = ld32(kr + gk.z() + 16 * o + 4 * c);
  bh = hmul2(qh, s2);
  bl = fma_f16x2(ql, s2, hfms2(qh, s2, bh));
}

// Scores of the two blocks of a stage.  sc[b][m][e]: 2^e * (q~ . codes*s) for
// block b, tokens 16m + g (+8 for e >= 2), heads 2c, 2c+1 (e & 1);
// zc = 2^e * (q . mu^K + q~ . z_b) with rows g = block 0 (zc[0..1]) and
// g + 8 = block 1 (zc[2..3]).
template <class GK>
__device__ __forceinline__ void key_stage(const uint8_t* kr0, const uint8_t* kr1, const GK& gk,
                                          const uint32_t (&Qh)[GK::kMaxOct], const uint32_t (&Ql)[GK::kMaxOct],
                                          const float (&CQ)[4], int lane, int c, float sc[2][2][4], float zc[4]) {
  constexpr int KO = GK::kMaxOct;
#pragma unroll
  for (int t = 0; t < (KO + 1) / 2; ++t) {
    const int oa = 2 * t, ob = 2 * t + 1;
    if (t > 0 && !gk.present(oa)) continue;  // only in class mode, and uniform
    const bool pb = ob < KO && gk.present(ob);
    uint32_t R[2][2][4], Bh[2][2], Bl[2][2], Z[2][2];
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint8_t* kr = b ? kr1 : kr0;
      key_octet(kr, gk, oa, Qh[oa], Ql[oa], lane, c, R[b][0], Bh[b][0], Bl[b][0], Z[b][0]);
      if (pb) {
        key_octet(kr, gk, ob, Qh[ob], Ql[ob], lane, c, R[b][1], Bh[b][1], Bl[b][1], Z[b][1]);
      } else {
        R[b][1][0] = R[b][1][1] = R[b][1][2] = R[b][1][3] = 0u;
        Bh[b][1] = Bl[b][1] = Z[b][1] = 0u;
      }
    }
    const uint32_t qhb = pb ? Qh[ob] : 0u, qlb = pb ? Ql[ob] : 0u;
    if (t == 0) mma16816_c(zc, Z[0][0], Z[1][0], Z[0][1], Z[1][1], Qh[oa], qhb, CQ);
    else mma16816(zc, Z[0][0], Z[1][0], Z[0][1], Z[1][1], Qh[oa], qhb);
    mma16816(zc, Z[0][0], Z[1][0], Z[0][1], Z[1][1], Ql[oa], qlb);
#pragma unroll
    for (int b = 0; b < 2; ++b) {
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        if (t == 0)
          mma16816_0(sc[b][m], R[b][0][2 * m], R[b][0][2 * m + 1], R[b][1][2 * m], R[b][1][2 * m + 1], Bh[b][0],
                     Bh[b][1]);
        else
          mma16816(sc[b][m], R[b][0][2 * m], R[b][0][2 * m + 1], R[b][1][2 * m], R[b][1][2 * m + 1], Bh[b][0],
                   Bh[b][1]);
        mma16816(sc[b][m], R[b][0][2 * m], R[b][0][2 * m + 1], R[b][1][2 * m], R[b][1][2 * m + 1], Bl[b][0],
                 Bl[b][1]);
      }
    }
  }
}

// ---- one value octet: fp16 latents for the lane's channel g of octet o and
// tokens (field k): registers k = 0..3.
template <bool VQ, class GV>
__device__ __forceinline__ void value_octet(const uint8_t* vr, int o, const GV& gv, int lane, int g,
                                            uint32_t L[4]) {
  if constexpr (VQ) {
    constexpr int VC = (GV::kMaxOct + 3) / 4;
    uint32_t F[4];
    if (o < VC) unpack_hi(ld32(vr + gv.word_off(o, lane)), F);
    else unpack_lo(ld16(vr + gv.word_off(o, lane)), F);
    const uint32_t sz = ld32(vr + gv.sz() + 4 * (8 * o + g));
    const uint32_t s2 = __byte_perm(sz, sz, 0x1010), z2 = __byte_perm(sz, sz, 0x3232);
#pragma unroll
    for (int k = 0; k < 4; ++k) L[k] = fma_f16x2(F[k], s2, z2);
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(vr + 512 * o + 16 * lane);
    L[0] = w.x;
    L[1] = w.y;
    L[2] = w.z;
    L[3] = w.w;
  }
}

template <bool VQ, class GV>
__device__ __forceinline__ void value_block(const uint8_t* vr, const GV& gv, int lane, int g,
                                            const uint32_t pb[2][2], float acc[(GV::kMaxOct + 1) / 2][4]) {
  constexpr int VO = GV::kMaxOct;
#pragma unroll
  for (int t = 0; t < (VO + 1) / 2; ++t) {
    const int oa = 2 * t, ob = 2 * t + 1;
    if (t > 0 && !gv.present(oa)) continue;
    const bool pbr = ob < VO && gv.present(ob);
    uint32_t La[4], Lb[4];
    value_octet<VQ>(vr, oa, gv, lane, g, La);
    if (pbr) {
      value_octet<VQ>(vr, ob, gv, lane, g, Lb);
    } else {
      Lb[0] = Lb[1] = Lb[2] = Lb[3] = 0u;
    }
    mma16816(acc[t], La[0], Lb[0], La[1], Lb[1], pb[0][0], pb[0][1]);
    mma16816(acc[t], La[2], Lb[2], La[3], Lb[3], pb[1][0], pb[1][1]);
  }
}

// Owner CTA of flat block i when T blocks are split evenly over G CTAs
// (CTA c covers [floor(cT/G), floor((c+1)T/G))).
__device__ __forceinline__ long long block_owner(long long i, long long T, long long G) {
  return ((i + 1) * G - 1) / T;
}

// ------------------------------------------------------------------ the kernel
// KC, VC: key / value record classes; KE, VE: exact octet counts, or 0 when
// the kernel serves every count of its class.
template <int KC, int VC, bool VQ, int KE, int VE>
__global__ void __launch_bounds__(kDecThreads, (KC + VC >= 7) ? 1 : 2) latent_decode_kernel(const DecodeParams p) {
  using GK = Geom<KC, KE, true>;
  using GV = Geom<VC, VE, VQ>;
  constexpr int KO = GK::kMaxOct, VT = (GV::kMaxOct + 1) / 2;
  extern __shared__ __align__(128) uint8_t smem[];
  float* q_s = reinterpret_cast<float*>(smem + kDecQOff);
  float* qt_s = reinterpret_cast<float*>(smem + kDecQtOff);
  float* mu_s = reinterpret_cast<float*>(smem + kDecMuOff);
  float* cq_s = reinterpret_cast<float*>(smem + kDecCqOff);
  float* red_s = reinterpret_cast<float*>(smem + kDecRedOff);
  int* flag_s = reinterpret_cast<int*>(smem + kDecFlagOff);  // [0] timed out, [1] this CTA merges
  float* B_s = reinterpret_cast<float*>(smem + kDecBsOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDecBarOff);  // [warps][ns], then the merge barrier
  uint8_t* ring = smem + p.ring_off;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const long long len = __ldcg(&p.k.hdr->length);
  const long long nf = len / kBlock;
  const long long T = p.streams * nf;
  // split over at most T CTAs, so every CTA that takes part owns >= 1 block
  // and the CTAs covering a stream are consecutive
  const long long G = T > 0 ? min((long long)gridDim.x, T) : (long long)gridDim.x, cta = blockIdx.x;
  const int ns = p.ns, Gq = p.Gq;
  GK geo_k;
  GV geo_v;
  geo_k.init(p.k);
  geo_v.init(p.v);
  const int rec_k = geo_k.rec(), rec_v = geo_v.rec();
  uint64_t* mbar = bars + kDecWarps * ns;

  if (tid == 0 && cta == 0 && __ldcg(&p.v.hdr->length) != len) set_dev_error(p.k.hdr, PALU_DEVERR_LENGTH_MISMATCH);
  long long R0 = 0, R1 = 0;
  if (T > 0) {
    if (cta >= G) return;
    R0 = cta * T / G;
    R1 = (cta + 1) * T / G;
    if (R0 >= R1) return;
  } else if (cta >= p.streams) {
    return;
  }

  // ---- one-time setup: zeroed rings (a stage's unused second block then
  // holds finite bytes), barriers
  {
    uint4* r4 = reinterpret_cast<uint4*>(ring);
    const int n16 = kDecWarps * ns * p.stage_bytes / 16;
    for (int i = tid; i < n16; i += kDecThreads) r4[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    for (int i = 0; i <= kDecWarps * ns; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    flag_s[0] = 0;
  }
  __syncthreads();

  const float max_s = __uint_as_float(__ldcg(&p.k.hdr->max_scale));
  uint8_t* wring = ring + (size_t)warp * ns * p.stage_bytes;
  uint64_t* wbar = bars + warp * ns;
  int slot = 0;           // this warp's next ring slot and its phase parity
  uint32_t par = 0;
  uint32_t merge_par = 0;

  long long X = T > 0 ? R0 / nf : cta;
  for (;;) {
    long long b0 = 0, b1 = 0, kslot = 0, nseg = 0;
    if (T > 0) {
      if (X * nf >= R1) break;
      b0 = max(R0, X * nf) - X * nf;
      b1 = min(R1, (X + 1) * nf) - X * nf;
      const long long c0 = block_owner(X * nf, T, G);
      nseg = block_owner(X * nf + nf - 1, T, G) - c0 + 1;
      kslot = cta - c0;
    } else if (X >= p.streams) {
      break;
    }
    const int b = (int)(X / p.Hkv), kh = (int)(X % p.Hkv);
    const bool dead = flag_s[0] != 0;

    // ---- this warp's contiguous share of the segment, two blocks per stage
    const long long nseg_blk = b1 - b0;
    const long long wb0 = b0 + warp * nseg_blk / kDecWarps, wb1 = b0 + (warp + 1) * nseg_blk / kDecWarps;
    const int n_my = (int)(wb1 - wb0), n_st = dead ? 0 : (n_my + 1) >> 1;
    const uint8_t* kbase = p.k.blocks + (size_t)X * p.k.n_blk_cap * rec_k;
    const uint8_t* vbase = p.v.blocks + (size_t)X * p.v.n_blk_cap * rec_v;
    auto issue = [&](int i, int s) {
      const long long blk = wb0 + 2LL * i;
      const int nb = (int)min(2LL, wb1 - blk);
      uint8_t* dst = wring + (size_t)s * p.stage_bytes;
      mbar_arrive_expect_tx(&wbar[s], (uint32_t)(nb * (rec_k + rec_v)));
      bulk_g2s(dst, kbase + blk * rec_k, (uint32_t)(nb * rec_k), &wbar[s]);
      bulk_g2s(dst + 2 * rec_k, vbase + blk * rec_v, (uint32_t)(nb * rec_v), &wbar[s]);
    };
    if (lane == 0) {
      int s = slot;
      for (int i = 0; i < n_st && i < ns; ++i) {
        issue(i, s);
        s = s + 1 == ns ? 0 : s + 1;
      }
    }

    // ---- prologue: q, mu^K and the key basis rows come in one batch of
    // loads; then q~ = q V^K (scaled, per padded key channel, one warp per
    // head, one lane per channel) and c = q . mu^K
    const int gk = kh / p.k.heads_per_group;
    const int npch = 8 * p.k.n_oct;
    const float* basis_g = p.k.basisT + (size_t)gk * p.k.r * kHeadDim;
    {
      const int h = tid >> 5, d4 = tid & 31;
      float4 qv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (h < Gq) {
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>(
                                    p.q + ((long long)b * p.Hq + (long long)kh * Gq + h) * kHeadDim) + d4);
        const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        qv = make_float4(lo.x, lo.y, hi.x, hi.y);
      }
      *reinterpret_cast<float4*>(q_s + h * kHeadDim + 4 * d4) = qv;
      if (tid < 32) *reinterpret_cast<float4*>(mu_s + 4 * tid) =
          __ldg(reinterpret_cast<const float4*>(p.k.mu + (size_t)gk * kHeadDim) + tid);
      for (int i = tid; i < 8 * kHeadDim; i += kDecThreads)
        if ((i & (kHeadDim - 1)) >= npch) qt_s[i] = 0.f;
    }
    float amax = 0.f;
    for (int ch = 0; ch < npch; ch += 32) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = tid + kDecThreads * u, r = i >> 5, c4 = i & 31, pch = ch + r;
        const int j = pch < npch ? padded_to_channel(pch, p.k.r, p.k.n_hi, p.k.n_hi_oct, 1) : -1;
        v[u] = j >= 0 ? __ldg(reinterpret_cast<const float4*>(basis_g + (size_t)j * kHeadDim) + c4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (ch > 0) __syncthreads();  // the previous chunk's readers are done
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = tid + kDecThreads * u, r = i >> 5, c4 = i & 31;
        float* dst = B_s + r * 129 + 4 * c4;
        dst[0] = v[u].x;
        dst[1] = v[u].y;
        dst[2] = v[u].z;
        dst[3] = v[u].w;
      }
      __syncthreads();
      const float* qh = q_s + warp * kHeadDim;
      const float* br = B_s + lane * 129;
      float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
      for (int d4 = 0; d4 < kHeadDim / 4; ++d4) {
        const float4 q4 = *reinterpret_cast<const float4*>(qh + 4 * d4);
        a0 = fmaf(q4.x, br[4 * d4], fmaf(q4.y, br[4 * d4 + 1], a0));
        a1 = fmaf(q4.z, br[4 * d4 + 2], fmaf(q4.w, br[4 * d4 + 3], a1));
      }
      const int pch = ch + lane;
      const float qt = (warp < Gq && pch < npch) ? (a0 + a1) * p.scale_log2 : 0.f;
      qt_s[warp * kHeadDim + pch] = qt;
      amax = fmaxf(amax, fabsf(qt));
    }
    {
      float s = 0.f;
      if (warp < Gq) {
        const float4 qq = *reinterpret_cast<const float4*>(q_s + warp * kHeadDim + 4 * lane);
        const float4 mm = *reinterpret_cast<const float4*>(mu_s + 4 * lane);
        s = fmaf(qq.x, mm.x, fmaf(qq.y, mm.y, fmaf(qq.z, mm.z, qq.w * mm.w)));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, o);
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      }
      if (lane == 0) {
        red_s[warp] = amax;
        cq_s[warp] = s * p.scale_log2;
      }
    }
    __syncthreads();
    // 2^e with |q~| 2^e max(1, max_s) < 2^14: every fp16 operand and product in
    // the score MMAs stays finite.
    amax = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) amax = fmaxf(amax, red_s[w]);
    const float xm = amax * fmaxf(1.f, max_s);
    int e = 0;
    if (xm > 0.f) {
      const int ex = (int)((__float_as_uint(xm) >> 23) & 0xFF) - 126;  // xm < 2^ex
      e = min(max(14 - ex, -120), 120);
    }
    const float two_e = pow2i(e), inv2e = pow2i(-e);
    uint32_t Qh[KO], Ql[KO];
#pragma unroll
    for (int o = 0; o < KO; ++o) {
      const float x0 = qt_s[g * kHeadDim + 8 * o + 2 * c] * two_e;
      const float x1 = qt_s[g * kHeadDim + 8 * o + 2 * c + 1] * two_e;
      Qh[o] = pack_f16x2(x0, x1);
      const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&Qh[o]));
      Ql[o] = pack_f16x2(x0 - hf.x, x1 - hf.y);
    }
    float CQ[4];
    CQ[0] = CQ[2] = cq_s[2 * c] * two_e;
    CQ[1] = CQ[3] = cq_s[2 * c + 1] * two_e;

    // ---- main loop
    float m_run[2] = {-INFINITY, -INFINITY}, thr[2] = {-INFINITY, -INFINITY};
    float l_acc[4] = {0.f, 0.f, 0.f, 0.f};
    float acc[VT][4];
#pragma unroll
    for (int t = 0; t < VT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    constexpr uint32_t kOnes = 0x3C003C00u;  // fp16x2 (1, 1)
    int done = 0;
    bool timed_out = false;
    for (int i = 0; i < n_st; ++i) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&wbar[slot], par));
      if (!ok) {
        timed_out = true;
        break;
      }
      const uint8_t* kr = wring + (size_t)slot * p.stage_bytes;
      const uint8_t* vr = kr + 2 * rec_k;
      const bool two = wb0 + 2LL * i + 1 < wb1;

      float sc[2][2][4], zc[4];
      key_stage(kr, kr + rec_k, geo_k, Qh, Ql, CQ, lane, c, sc, zc);
      if (!two) {
#pragma unroll
        for (int m = 0; m < 2; ++m) sc[1][m][0] = sc[1][m][1] = sc[1][m][2] = sc[1][m][3] = -INFINITY;
      }

      // lazy online softmax over the stage's 64 tokens (raw units: 2^e * log2);
      // raw score = sc + zc of its block and head
      float mx0 = fmaxf(fmaxf(fmaxf(sc[0][0][0], sc[0][0][2]), fmaxf(sc[0][1][0], sc[0][1][2])) + zc[0],
                        fmaxf(fmaxf(sc[1][0][0], sc[1][0][2]), fmaxf(sc[1][1][0], sc[1][1][2])) + zc[2]);
      float mx1 = fmaxf(fmaxf(fmaxf(sc[0][0][1], sc[0][0][3]), fmaxf(sc[0][1][1], sc[0][1][3])) + zc[1],
                        fmaxf(fmaxf(sc[1][0][1], sc[1][0][3]), fmaxf(sc[1][1][1], sc[1][1][3])) + zc[3]);
      if (__any_sync(0xffffffffu, mx0 > thr[0] || mx1 > thr[1])) {
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
        }
        const float n0 = fmaxf(m_run[0], mx0 * inv2e), n1 = fmaxf(m_run[1], mx1 * inv2e);
        const float a0 = ex2(m_run[0] - n0), a1 = ex2(m_run[1] - n1);
#pragma unroll
        for (int t = 0; t < VT; ++t) {
          acc[t][0] *= a0;
          acc[t][1] *= a1;
          acc[t][2] *= a0;
          acc[t][3] *= a1;
        }
        l_acc[0] *= a0;
        l_acc[1] *= a1;
        l_acc[2] *= a0;
        l_acc[3] *= a1;
        m_run[0] = n0;
        m_run[1] = n1;
        thr[0] = (n0 + kLazyTau) * two_e;
        thr[1] = (n1 + kLazyTau) * two_e;
      }
      uint32_t pb[2][2][2];
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        const float bias0 = fmaf(zc[2 * bb], inv2e, -m_run[0]), bias1 = fmaf(zc[2 * bb + 1], inv2e, -m_run[1]);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const float p0 = ex2(fmaf(sc[bb][m][0], inv2e, bias0)), p1 = ex2(fmaf(sc[bb][m][1], inv2e, bias1));
          const float p2 = ex2(fmaf(sc[bb][m][2], inv2e, bias0)), p3 = ex2(fmaf(sc[bb][m][3], inv2e, bias1));
          pb[bb][m][0] = movm_t(pack_f16x2(p0, p1));
          pb[bb][m][1] = movm_t(pack_f16x2(p2, p3));
        }
        // row sums on the tensor cores: all-ones A
        mma16816(l_acc, kOnes, kOnes, kOnes, kOnes, pb[bb][0][0], pb[bb][0][1]);
        mma16816(l_acc, kOnes, kOnes, kOnes, kOnes, pb[bb][1][0], pb[bb][1][1]);
      }
      value_block<VQ>(vr, geo_v, lane, g, pb[0], acc);
      value_block<VQ>(vr + rec_v, geo_v, lane, g, pb[1], acc);

      __syncwarp();
      if (lane == 0 && i + ns < n_st) issue(i + ns, slot);
      slot = slot + 1 == ns ? 0 : slot + 1;
      par ^= slot == 0 ? 1u : 0u;
      done = i + 1;
    }
    if (timed_out) {
      // drain this warp's copies still in flight (bounded), then report
      if (lane == 0) {
        set_dev_error(p.k.hdr, PALU_DEVERR_TIMEOUT);
        int s = slot;
        uint32_t pr = par;
        for (int i = done; i < n_st && i < done + ns; ++i) {
          mbar_wait_bounded(&wbar[s], pr);
          s = s + 1 == ns ? 0 : s + 1;
          pr ^= s == 0 ? 1u : 0u;
        }
        atomicOr(&flag_s[0], 1);
      }
    }

    // ---- merge the 8 warps of the CTA into the segment's partial
    __syncthreads();  // every warp is done with the ring
    const int ms = 2 + p.rvp;
    float* mw = reinterpret_cast<float*>(ring) + warp * 8 * ms;
    if (g == 0) {
      mw[(2 * c) * ms + 0] = n_my > 0 ? m_run[0] : -INFINITY;
      mw[(2 * c) * ms + 1] = l_acc[0];
      mw[(2 * c + 1) * ms + 0] = n_my > 0 ? m_run[1] : -INFINITY;
      mw[(2 * c + 1) * ms + 1] = l_acc[1];
    }
#pragma unroll
    for (int t = 0; t < VT; ++t) {
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const int pch = 16 * t + g + 8 * (e2 >> 1);
        if (pch < p.rvp) mw[(2 * c + (e2 & 1)) * ms + 2 + pch] = acc[t][e2];
      }
    }
    fence_proxy_async_smem();  // bulk copies will land on these bytes later
    __syncthreads();
    const bool bad = flag_s[0] != 0;
    // merge-phase layout of the ring (only the stream's last contributor
    // reads it): V basis, tails, the stream's partials, tail weights, merged
    // latents, denominators
    const int rk = p.k.r, rv = p.v.r;
    const int n_tail = (int)(len % kBlock);
    const int gv = kh / p.v.heads_per_group;
    const int tv_bytes = p.v.quantize ? kBlock * rv * 4 : rec_v;
    float* BV_s = reinterpret_cast<float*>(ring);                 // [rv][128]
    float* TK_s = BV_s + (size_t)rv * kHeadDim;                    // [32][rk]
    float* TV_s = TK_s + (size_t)kBlock * rk;                      // [32][rv] (or one fp16 record)
    float* P_s = TV_s + (tv_bytes + 15) / 16 * 4;                  // [nseg][Gq][ms] partials
    float* ST_s = P_s + (size_t)p.seg_max * Gq * ms;               // [8][32] tail scores, then weights
    float* O_s = ST_s + 8 * kBlock;                                // [8][128] merged latents
    float* L_s = O_s + 8 * kHeadDim;                               // [8]
    if (T > 0) {
      float* part = p.ws + ((size_t)X * p.seg_max + kslot) * (size_t)Gq * ms;
      const float* mrg = reinterpret_cast<const float*>(ring);
      for (int i = tid; i < Gq * ms; i += kDecThreads) {
        const int h = i / ms, e2 = i - h * ms;
        float out;
        if (bad) {
          out = e2 == 0 ? -INFINITY : 0.f;
        } else {
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, mrg[(w * 8 + h) * ms]);
          if (e2 == 0) {
            out = M;
          } else {
            out = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) {
              const float mw_ = mrg[(w * 8 + h) * ms];
              if (mw_ != -INFINITY) out = fmaf(mrg[(w * 8 + h) * ms + e2], ex2(mw_ - M), out);
            }
          }
        }
        part[i] = out;
      }
    }
    __syncthreads();  // the warp partials are consumed; the ring is free
    if (tid == 0) {
      // the V basis and the tails, fetched before the ticket so that the
      // last contributor finds them in place (the others just let them land)
      const uint32_t bytes = (uint32_t)rv * 512u + (n_tail > 0 ? (uint32_t)(kBlock * rk * 4 + tv_bytes) : 0u);
      mbar_arrive_expect_tx(mbar, bytes);
      bulk_g2s(BV_s, p.v.basisT + (size_t)gv * rv * kHeadDim, (uint32_t)rv * 512u, mbar);
      if (n_tail > 0) {
        bulk_g2s(TK_s, p.k.tail + (size_t)X * kBlock * rk, (uint32_t)(kBlock * rk * 4), mbar);
        const void* tv = p.v.quantize ? static_cast<const void*>(p.v.tail + (size_t)X * kBlock * rv)
                                      : static_cast<const void*>(p.v.blocks + ((size_t)X * p.v.n_blk_cap + nf) * rec_v);
        bulk_g2s(TV_s, tv, (uint32_t)tv_bytes, mbar);
      }
      int last = 1;
      if (T > 0) {
        // release: the CTA's partial (ordered by the barrier above) before the
        // ticket; acquire: the other contributors' partials after it
        __threadfence();
        const unsigned int t = atomicAdd(&p.k.tickets[X], 1u);
        last = t + 1 == (unsigned int)nseg;
        if (last) {
          p.k.tickets[X] = 0u;
          __threadfence();
        }
      }
      flag_s[1] = last;
    }
    __syncthreads();
    const bool merger = flag_s[1] != 0;
    const int nsg = T > 0 ? (int)nseg : 0;
    if (merger) {
      const float* wsx = p.ws + (size_t)X * p.seg_max * Gq * ms;
      for (int i = tid; i < nsg * Gq * ms; i += kDecThreads) P_s[i] = __ldcg(wsx + i);
    }
    const bool got = mbar_wait_bounded(mbar, merge_par);
    merge_par ^= 1u;
    if (!got && tid == 0) set_dev_error(p.k.hdr, PALU_DEVERR_TIMEOUT);
    __syncthreads();

    // ---- the stream's last contributor: merge partials + tail, project, + mu
    if (merger) {
      // tail scores (log2 units)
      for (int i = tid; i < n_tail * 8; i += kDecThreads) {
        const int t = i >> 3, h = i & 7;
        float sc_t = -INFINITY;
        if (h < Gq) {
          sc_t = cq_s[h];
          for (int j2 = 0; j2 < rk; ++j2) {
            const int pch = j2 < p.k.n_hi ? j2 : 8 * p.k.n_hi_oct + (j2 - p.k.n_hi);
            sc_t = fmaf(qt_s[h * kHeadDim + pch], TK_s[t * rk + j2], sc_t);
          }
        }
        ST_s[h * kBlock + t] = sc_t;
      }
      __syncthreads();
      // warp h: max, weights (over the partials' m), denominator
      if (warp < Gq) {
        const int h = warp;
        float M = -INFINITY;
        for (int sg = lane; sg < nsg; sg += 32) M = fmaxf(M, P_s[(sg * Gq + h) * ms]);
        const float st = lane < n_tail ? ST_s[h * kBlock + lane] : -INFINITY;
        M = fmaxf(M, st);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f;
        for (int sg = lane; sg < nsg; sg += 32) {
          const float m = P_s[(sg * Gq + h) * ms];
          const float w = m == -INFINITY ? 0.f : ex2(m - M);
          L = fmaf(w, P_s[(sg * Gq + h) * ms + 1], L);
          P_s[(sg * Gq + h) * ms] = w;
        }
        const float pt = lane < n_tail ? ex2(st - M) : 0.f;
        L += pt;
        __syncwarp();
        ST_s[h * kBlock + lane] = pt;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) L_s[h] = L;
      }
      __syncthreads();
      // merged latent per (head, real value channel)
      for (int i = tid; i < Gq * p.rvp; i += kDecThreads) {
        const int h = i / p.rvp, pch = i - h * p.rvp;
        const int j2 = padded_to_channel(pch, rv, p.v.n_hi, p.v.n_hi_oct, p.v.quantize);
        if (j2 < 0) continue;
        float a = 0.f;
        for (int sg = 0; sg < nsg; ++sg) a = fmaf(P_s[(sg * Gq + h) * ms], P_s[(sg * Gq + h) * ms + 2 + pch], a);
        for (int t = 0; t < n_tail; ++t) {
          float lv;
          if (p.v.quantize) {
            lv = TV_s[t * rv + j2];
          } else {
            const int kk = 2 * (t >> 4) + ((t & 15) >> 3);
            const int ln = 4 * (j2 & 7) + ((t & 7) >> 1);
            lv = __half2float(*reinterpret_cast<const __half*>(reinterpret_cast<const uint8_t*>(TV_s) +
                                                               512 * (j2 >> 3) + 16 * ln + 4 * kk + 2 * (t & 1)));
          }
          a = fmaf(ST_s[h * kBlock + t], lv, a);
        }
        O_s[h * kHeadDim + j2] = a;
      }
      __syncthreads();
      // out[h][d] = (sum_j o_hj V[d, j]) / L_h + mu[d]
      {
        const int d = tid & 127, h0 = (tid >> 7) * 4;
        float o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int j2 = 0; j2 < rv; ++j2) {
          const float bv = BV_s[j2 * kHeadDim + d];
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) o4[hh] = fmaf(O_s[(h0 + hh) * kHeadDim + j2], bv, o4[hh]);
        }
        const float mu = __ldg(p.v.mu + (size_t)gv * kHeadDim + d);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const int h = h0 + hh;
          if (h < Gq) {
            const float v = fmaf(o4[hh], 1.f / L_s[h], mu);
            const long long oi = ((long long)b * p.Hq + (long long)kh * Gq + h) * kHeadDim + d;
            if (p.out_fp32)
              static_cast<float*>(p.out)[oi] = v;
            else
              static_cast<__half*>(p.out)[oi] = __float2half_rn(v);
          }
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    ++X;
    if (T == 0) X += G - 1;
  }
}

typedef void (*DecodeKernel)(const DecodeParams);

// Instantiations are spread over translation units (parallel build):
// exact octet counts up to 8 on both sides, one unit per key count, and the
// class kernels for the larger ranks, one unit per key class.
template <int KE>
DecodeKernel decode_kernel_exact(int ve, bool vq);
template <int KC>
DecodeKernel decode_kernel_class(int vc, bool vq);

}  // namespace palu
