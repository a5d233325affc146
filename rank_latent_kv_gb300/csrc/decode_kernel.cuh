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
//  * Persistent grid (resident CTAs only, one per SM).  The flat range of full
//    32-token blocks over all (batch, KV head) streams is split evenly over
//    the warps of the grid (16, 12 or 8 a CTA), so every SM gets the same
//    number of blocks whatever the batch and head count.  A warp's range
//    covers at most two streams ("segments"); it streams them through its own
//    ring of shared-memory stages (2 blocks of key and value records per
//    stage, two 1-D bulk copies on the TMA engine, mbarrier completion).  The
//    first stages are in flight before the stream's query factors are read.
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
//  * Each CTA merges its warps (log-sum-exp) per stream, the CTA holding a
//    stream's last full block folds in the fp32 tail tokens, and every CTA
//    applies V^V^T to its merged latent (the projection is linear, so it
//    commutes with the final merge).  A CTA that covers a whole stream writes
//    the output; otherwise a per-stream ticket in the workspace picks the
//    stream's last CTA, which merges the projected partials and adds mu^V.
#pragma once

#include <math.h>

#include "palu_internal.cuh"

namespace palu {

constexpr int kMaxDecWarps = 16;  // warps per decode CTA: 16 (one CTA per SM) for the exact-octet
                                  // kernels, or 8 when their rings do not fit
constexpr int kMaxDecThreads = 32 * kMaxDecWarps;
// the per-class kernels: up to 12 warps (at most 168 registers a thread), or
// 8 when their rings do not fit
constexpr int kClassDecWarps = 12;
constexpr int kClassDecThreads = 32 * kClassDecWarps;
constexpr float kLazyTau = 8.f;   // log2 headroom before the running max is raised
constexpr int kDecFlagOff = 0;                  // decode CTA shared memory: flags int [2 * warps]
constexpr int kDecInfoOff = 8 * kMaxDecWarps;   // then the first CTA's streams' CTA ranges int [8]
constexpr int kDecBarOff = kDecInfoOff + 32;    // then mbarriers [warps][ns] + 2; the rings follow
// A partial (per segment and query head): m, l, two pad words, then the
// latent accumulator per padded value channel; 16-byte multiple, so one
// stream's partials move as a single bulk copy.
constexpr int kPartHead = 4;
// A projected partial (per CTA, stream and query head): m, l, two pad words,
// then sum_t p_t v_t over the head dimension.
constexpr int kOutHead = 4;
constexpr int kOutPart = kOutHead + kHeadDim;

struct DecodeParams {
  CacheView k, v;
  const __half* q;
  void* out;
  uint32_t* qpack;    // per stream and lane: Qh[ko], Ql[ko], CQ0, CQ1, 2^e, 2^-e  (qp_stride words)
  float* qt;          // per stream: scaled q~ [8][128] per padded key channel
  float* cq;          // per stream: scaled q . mu^K [8]
  float* ws;          // projected partials [streams][seg_max][Gq][kOutPart]
  uint32_t* tickets;  // per stream: CTAs done with the stream, then CTAs done with the launch (zeroed by the q-prep)
  int out_fp32;
  int Hq, Hkv, Gq;
  int rvp;            // padded value channels = 8 * v.n_oct
  int ns;             // stages per warp ring
  int stage_bytes;    // 2 * (k.rec_bytes + v.rec_bytes)
  int ring_off;       // shared-memory offset of the rings
  int wp_off;         // shared-memory offset of the warps' partials [warps][2][Gq][kPartHead + rvp]
  int end_off;        // shared-memory offset of the end phase's area (EndSmem)
  int end_off2;       // a second end area (two streams in parallel), or -1
  int seg_max;        // partial slots per stream
  int qp_ko;          // key octets held per lane in qpack
  int qp_stride;      // words per lane in qpack
  int dec_grid;       // CTAs of the decode launch
  int after_append;   // the preceding launch appended tokens: read nothing before it completes
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
// Programmatic dependent launch: wait for the preceding launch's results /
// let the next launch be scheduled.  Both are no-ops without the attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Named barrier over n threads (id 0 with the whole CTA is __syncthreads).
__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
// Bulk prefetch of global bytes into L2 (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
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
// (a & mask) | magic in one LOP3: the mask is an immediate, the magic comes
// in a register (an instruction takes one 32-bit immediate at most)
template <uint32_t kMask>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(kMask), "r"(magic));
  return d;
}
struct Magic {
  uint32_t m1024, m256, m64, m16;  // fp16x2 (2^E, 2^E) for E = 10, 8, 6, 4
};
__device__ __forceinline__ Magic make_magic() {
  Magic m;
  // through an opaque move so that the values stay in registers
  asm("mov.b32 %0, 0x64006400;" : "=r"(m.m1024));
  asm("mov.b32 %0, 0x5C005C00;" : "=r"(m.m256));
  asm("mov.b32 %0, 0x54005400;" : "=r"(m.m64));
  asm("mov.b32 %0, 0x4C004C00;" : "=r"(m.m16));
  return m;
}
__device__ __forceinline__ void unpack_hi(uint32_t w, const Magic& mg, uint32_t R[4]) {
  const uint32_t w8 = w >> 8;
  R[0] = sub_f16x2(and_or<0x000F000Fu>(w, mg.m1024), mg.m1024);   // 1024 + c
  R[1] = sub_f16x2(and_or<0x00F000F0u>(w, mg.m64), mg.m64);       //   64 + c
  R[2] = sub_f16x2(and_or<0x000F000Fu>(w8, mg.m1024), mg.m1024);
  R[3] = sub_f16x2(and_or<0x00F000F0u>(w8, mg.m64), mg.m64);
}
// hw: the octet's 16 bits (half 0 in bits 0-7, half 1 in bits 8-15).
__device__ __forceinline__ void unpack_lo(uint32_t hw, const Magic& mg, uint32_t R[4]) {
  const uint32_t w = __byte_perm(hw, 0u, 0x4140);
  R[0] = sub_f16x2(and_or<0x00030003u>(w, mg.m1024), mg.m1024);   // 1024 + c
  R[1] = sub_f16x2(and_or<0x000C000Cu>(w, mg.m256), mg.m256);     //  256 + c
  R[2] = sub_f16x2(and_or<0x00300030u>(w, mg.m64), mg.m64);       //   64 + c
  R[3] = sub_f16x2(and_or<0x00C000C0u>(w, mg.m16), mg.m16);       //   16 + c
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
// One key octet of one block: exact codes, the B pair (hi, lo) of
// Q~ * s for the lane's head g and channels 2c, 2c+1, and the zero points.
template <class GK>
__device__ __forceinline__ void key_octet(const uint8_t* kr, const GK& gk, int o, uint32_t qh, uint32_t ql,
                                          int lane, int c, const Magic& mg, uint32_t R[4], uint32_t& bh,
                                          uint32_t& bl, uint32_t& z) {
  constexpr int KC = (GK::kMaxOct + 3) / 4;
  if (o < KC) unpack_hi(ld32(kr + gk.word_off(o, lane)), mg, R);
  else unpack_lo(ld16(kr + gk.word_off(o, lane)), mg, R);
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
                                          const float (&CQ)[4], const float (&Z4)[4], int lane, int c, const Magic& mg,
                                          float sc[2][2][4], float zc[4]) {
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
      key_octet(kr, gk, oa, Qh[oa], Ql[oa], lane, c, mg, R[b][0], Bh[b][0], Bl[b][0], Z[b][0]);
      if (pb) {
        key_octet(kr, gk, ob, Qh[ob], Ql[ob], lane, c, mg, R[b][1], Bh[b][1], Bl[b][1], Z[b][1]);
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
          mma16816_c(sc[b][m], R[b][0][2 * m], R[b][0][2 * m + 1], R[b][1][2 * m], R[b][1][2 * m + 1], Bh[b][0],
                     Bh[b][1], Z4);
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
__device__ __forceinline__ void value_octet(const uint8_t* vr, int o, const GV& gv, int lane, int g, const Magic& mg,
                                            uint32_t L[4]) {
  if constexpr (VQ) {
    constexpr int VC = (GV::kMaxOct + 3) / 4;
    uint32_t F[4];
    if (o < VC) unpack_hi(ld32(vr + gv.word_off(o, lane)), mg, F);
    else unpack_lo(ld16(vr + gv.word_off(o, lane)), mg, F);
    const __half2 sz = *reinterpret_cast<const __half2*>(vr + gv.sz() + 4 * (8 * o + g));
    const __half2 s2 = __low2half2(sz), z2 = __high2half2(sz);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&F[k]), s2, z2);
      L[k] = *reinterpret_cast<const uint32_t*>(&r);
    }
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(vr + 512 * o + 16 * lane);
    L[0] = w.x;
    L[1] = w.y;
    L[2] = w.z;
    L[3] = w.w;
  }
}

template <bool VQ, class GV>
__device__ __forceinline__ void value_block(const uint8_t* vr, const GV& gv, int lane, int g, const Magic& mg,
                                            const uint32_t pb[2][2], float acc[(GV::kMaxOct + 1) / 2][4]) {
  constexpr int VO = GV::kMaxOct;
#pragma unroll
  for (int t = 0; t < (VO + 1) / 2; ++t) {
    const int oa = 2 * t, ob = 2 * t + 1;
    if (t > 0 && !gv.present(oa)) continue;
    const bool pbr = ob < VO && gv.present(ob);
    uint32_t La[4], Lb[4];
    value_octet<VQ>(vr, oa, gv, lane, g, mg, La);
    if (pbr) {
      value_octet<VQ>(vr, ob, gv, lane, g, mg, Lb);
    } else {
      Lb[0] = Lb[1] = Lb[2] = Lb[3] = 0u;
    }
    mma16816(acc[t], La[0], Lb[0], La[1], Lb[1], pb[0][0], pb[0][1]);
    mma16816(acc[t], La[2], Lb[2], La[3], Lb[3], pb[1][0], pb[1][1]);
  }
}

// Shared-memory area of the decode kernel's end phase (one stream at a time;
// it reuses the rings when they are large enough).  Byte offsets from its
// 16-byte aligned base, shared by the launch plan and the kernel.
struct EndLayout {
  int bv, qt, cq, tk, tv, st, ol, sw, hm, hl, wo, flag, bytes;
};
__host__ __device__ inline EndLayout end_layout(int rk, int rv, int v_quantize, int rec_v) {
  EndLayout e;
  e.bv = 0;                                   // V basis rows [rv][128]
  e.qt = e.bv + rv * kHeadDim * 4;            // scaled q~ [8][128]
  e.cq = e.qt + 8 * kHeadDim * 4;             // scaled q . mu^K [8]
  e.tk = e.cq + 32;                           // key tail latents [32][rk | 1]
  e.tv = e.tk + kBlock * (rk | 1) * 4;        // value tail [32][rv] (or the fp16 record)
  e.st = e.tv + (v_quantize ? kBlock * rv * 4 : rec_v);
  e.ol = e.st + 8 * kBlock * 4;               // tail scores, then weights [8][32]
  e.sw = e.ol + 8 * kHeadDim * 4;             // merged latents [8][128]
  e.hm = e.sw + 32 * 8 * 4;                   // weights of the warp segments [32][8]
  e.hl = e.hm + 32;                           // running max, sum, tail rescale [8]
  e.wo = e.hl + 32;
  e.flag = e.wo + 32;
  e.bytes = e.flag + 16;
  return e;
}
struct EndSmem {
  float *bv, *qt, *cq, *tk, *tv, *st, *ol, *sw, *hm, *hl, *wo;
  int* flag;
};
__device__ __forceinline__ EndSmem end_smem(uint8_t* base, const DecodeParams& p) {
  const EndLayout e = end_layout(p.k.r, p.v.r, p.v.quantize, p.v.rec_bytes);
  EndSmem s;
  s.bv = reinterpret_cast<float*>(base + e.bv);
  s.qt = reinterpret_cast<float*>(base + e.qt);
  s.cq = reinterpret_cast<float*>(base + e.cq);
  s.tk = reinterpret_cast<float*>(base + e.tk);
  s.tv = reinterpret_cast<float*>(base + e.tv);
  s.st = reinterpret_cast<float*>(base + e.st);
  s.ol = reinterpret_cast<float*>(base + e.ol);
  s.sw = reinterpret_cast<float*>(base + e.sw);
  s.hm = reinterpret_cast<float*>(base + e.hm);
  s.hl = reinterpret_cast<float*>(base + e.hl);
  s.wo = reinterpret_cast<float*>(base + e.wo);
  s.flag = reinterpret_cast<int*>(base + e.flag);
  return s;
}
__device__ __forceinline__ void store_out(const DecodeParams& p, long long i, float v) {
  if (p.out_fp32)
    static_cast<float*>(p.out)[i] = v;
  else
    static_cast<__half*>(p.out)[i] = __float2half_rn(v);
}

// Owner CTA of flat block i when T blocks are split evenly over G CTAs
// (CTA c covers [floor(cT/G), floor((c+1)T/G))).
__device__ __forceinline__ long long block_owner(long long i, long long T, long long G) {
  return ((i + 1) * G - 1) / T;
}

// ------------------------------------------------------------------ the kernel
// KC, VC: key / value record classes; KE, VE: exact octet counts, or 0 when
// the kernel serves every count of its class.  Launched after the q-prep
// kernel (programmatic dependent launch: the first copies are in flight
// before the packed query factors are read).
template <int KC, int VC, bool VQ, int KE, int VE>
__global__ void __launch_bounds__((KE > 0 && KE <= 8) ? kMaxDecThreads : kClassDecThreads, 1)
    latent_decode_kernel(const DecodeParams p) {
  using GK = Geom<KC, KE, true>;
  using GV = Geom<VC, VE, VQ>;
  constexpr int KO = GK::kMaxOct, VT = (GV::kMaxOct + 1) / 2;
  extern __shared__ __align__(128) uint8_t smem[];
  int* flag_s = reinterpret_cast<int*>(smem + kDecFlagOff);  // stream of each warp's two segments
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDecBarOff);  // [warps][ns]
  uint8_t* ring = smem + p.ring_off;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int nw = blockDim.x >> 5, nt = blockDim.x;  // 16, 12 or 8 warps
  // After a step prologue (one token appended per stream), this launch owns
  // the length update: the prologue leaves the stored length alone, every
  // CTA reads it as it was before the step, and the last CTA to finish
  // stores the new one.  Copies of blocks the prologue did not write may
  // start before its results are awaited; a block the appended token
  // completed may not.
  // With ragged lengths the split is that of the longest sequence (the
  // header length): every stream gets the same range of block positions, and
  // a warp skips the positions past its stream's own full blocks.
  const bool ragged = __ldcg(&p.k.hdr->ragged) != 0;
  const long long len0 = __ldcg(&p.k.hdr->length);
  const bool grows = p.after_append && len0 < p.k.capacity;
  const long long len = len0 + (grows ? 1 : 0);
  if (grows && (ragged || len % kBlock == 0)) grid_dep_wait();
  grid_dep_launch();
  const long long nf = len / kBlock;
  const long long T = p.streams * nf;
  // tokens of stream x at this launch (after a step prologue, one more)
  auto stream_len = [&](long long x) -> long long {
    return ragged ? __ldcg(p.k.seq_len + x / p.Hkv) + (grows ? 1 : 0) : len;
  };
  if (tid == 0 && blockIdx.x == 0) {
    bool bad = __ldcg(&p.v.hdr->length) != len0 || __ldcg(&p.v.hdr->ragged) != (ragged ? 1u : 0u);
    if (ragged && !bad)
      for (int b = 0; b < p.k.batch; ++b) bad |= __ldcg(p.k.seq_len + b) != __ldcg(p.v.seq_len + b);
    if (bad) set_dev_error(p.k.hdr, PALU_DEVERR_LENGTH_MISMATCH);
  }
  // every warp works on its own: the flat range of full blocks is split over
  // at most T warps, so each warp that takes part owns >= 1 block and the
  // warps covering a stream are consecutive
  const long long W = min((long long)gridDim.x * nw, T);
  const long long gw = (long long)blockIdx.x * nw + warp;
  const long long R0 = gw < W ? gw * T / W : 0, R1 = gw < W ? (gw + 1) * T / W : 0;
  const int ns = p.ns, Gq = p.Gq;
  GK geo_k;
  GV geo_v;
  geo_k.init(p.k);
  geo_v.init(p.v);
  const int rec_k = geo_k.rec(), rec_v = geo_v.rec();
  int* info_s = reinterpret_cast<int*>(smem + kDecInfoOff);  // x0, then (first, last CTA) of x0 and x0 + 1
  if (tid == 32) {
    // warm L2 with what the end phase will copy: the V basis rows of the
    // CTA's first and last stream, and the tails of a stream ending here;
    // and the CTA ranges of the CTA's first two streams, for the end phase
    long long x0 = 0, x1 = -1, b_end = -1;
    if (nf > 0) {
      const long long c0 = min((long long)blockIdx.x * nw, W), c1 = min(c0 + nw, W);
      if (c0 < c1) {
        b_end = c1 * T / W;
        x0 = (c0 * T / W) / nf;
        x1 = (b_end - 1) / nf;
      }
    } else {
      x0 = (long long)blockIdx.x * nw;
      x1 = min(x0 + nw, p.streams) - 1;
    }
    info_s[0] = (int)x0;
    for (int i = 0; i < 2; ++i) {
      const long long x = x0 + i;
      long long cf = x / nw, cl = cf;
      if (nf > 0) {
        cf = block_owner(x * nf, T, W) / nw;
        cl = block_owner(x * nf + nf - 1, T, W) / nw;
      }
      info_s[1 + 2 * i] = (int)cf;
      info_s[2 + 2 * i] = (int)cl;
    }
    if (x0 <= x1) {
      const int g0 = (int)(x0 % p.Hkv) / p.v.heads_per_group, g1 = (int)(x1 % p.Hkv) / p.v.heads_per_group;
      prefetch_l2(p.v.basisT + (size_t)g0 * p.v.r * kHeadDim, (uint32_t)p.v.r * 512u);
      if (g1 != g0) prefetch_l2(p.v.basisT + (size_t)g1 * p.v.r * kHeadDim, (uint32_t)p.v.r * 512u);
      if (!ragged && len % kBlock != 0 && b_end == (x1 + 1) * nf) {
        prefetch_l2(p.k.tail + (size_t)x1 * kBlock * p.k.r, (uint32_t)(kBlock * p.k.r * 4));
        if (p.v.quantize)
          prefetch_l2(p.v.tail + (size_t)x1 * kBlock * p.v.r, (uint32_t)(kBlock * p.v.r * 4));
        else
          prefetch_l2(p.v.blocks + ((size_t)x1 * p.v.n_blk_cap + nf) * p.v.rec_bytes, (uint32_t)p.v.rec_bytes);
      }
    }
  }

  // ---- one-time setup: barriers; the warps' partial slots (two segments
  // each) start at zero, so that the end phase can weigh every slot, with
  // weight 0 for the slots of other streams or of no segment
  if (tid == 0) {
    for (int i = 0; i < nw * ns + 2; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  const int ms = kPartHead + p.rvp;
  float* wp = reinterpret_cast<float*>(smem + p.wp_off) + (size_t)warp * 2 * Gq * ms;
  if (lane < 2) flag_s[2 * warp + lane] = -1;
  for (int i = lane; i < 2 * Gq * ms; i += 32) wp[i] = 0.f;
  __syncthreads();

  uint8_t* wring = ring + (size_t)warp * ns * p.stage_bytes;
  uint64_t* wbar = bars + warp * ns;
  int slot = 0;  // this warp's next ring slot and its phase parity
  uint32_t par = 0;
  bool first = true;
  const Magic mg = make_magic();
  // MMA operand quads of repeated constants, each value in its own register
  // (a zero C operand and an all-ones A operand, fp16x2 (1, 1))
  float Z4[4];
  uint32_t O4[4];
  asm volatile("mov.b32 %0, 0;" : "=f"(Z4[0]));
  asm volatile("mov.b32 %0, 0;" : "=f"(Z4[1]));
  asm volatile("mov.b32 %0, 0;" : "=f"(Z4[2]));
  asm volatile("mov.b32 %0, 0;" : "=f"(Z4[3]));
  asm volatile("mov.b32 %0, 0x3C003C00;" : "=r"(O4[0]));
  asm volatile("mov.b32 %0, 0x3C003C00;" : "=r"(O4[1]));
  asm volatile("mov.b32 %0, 0x3C003C00;" : "=r"(O4[2]));
  asm volatile("mov.b32 %0, 0x3C003C00;" : "=r"(O4[3]));

  bool timed_out = false;
  int seg = 0;
  for (long long X = R0 < R1 ? R0 / nf : 0; R0 < R1 && X * nf < R1; ++X, ++seg) {
    if (seg >= 2) {  // the launch plan gives every warp at most two streams
      set_dev_error(p.k.hdr, PALU_DEVERR_CAPACITY);
      break;
    }
    // ---- this warp's segment of stream X, two blocks per stage (clipped to
    // the stream's own full blocks)
    const long long nfX = ragged ? stream_len(X) / kBlock : nf;
    const long long wb1 = min(min(R1, (X + 1) * nf) - X * nf, nfX);
    const long long wb0 = min(max(R0, X * nf) - X * nf, wb1);
    const int n_my = (int)(wb1 - wb0), n_st = timed_out ? 0 : (n_my + 1) >> 1;
    // Stage i holds blocks 2i, 2i+1 of the warp's range.  Every stage reads
    // two real records, so that no byte the compute touches is stale: an odd
    // last stage takes the pair that ends at its block (its first slot, a
    // block counted already, is masked), or, for a one-block range, the pair
    // that starts there (second slot masked); a stream of one full block
    // cannot pair up, and its stage copies the block twice.
    const long long blk_last = nfX - 1;  // last full block of the stream
    int odd_shift = 0, odd_mask = 1;               // odd last stage: source shift, slot to mask
    if (n_my & 1) {
      if (n_my >= 2 || wb0 >= 1) {
        odd_shift = -1;
        odd_mask = 0;
      } else if (blk_last >= 1) {
        odd_shift = 0;
        odd_mask = 1;
      } else {
        odd_shift = 1;  // marker: duplicate
        odd_mask = 1;
      }
    }
    const uint8_t* kbase = p.k.blocks + ((size_t)X * p.k.n_blk_cap + wb0) * rec_k;
    const uint8_t* vbase = p.v.blocks + ((size_t)X * p.v.n_blk_cap + wb0) * rec_v;
    auto issue = [&](int i, int s) {
      uint8_t* dst = wring + s * p.stage_bytes;
      uint64_t* bar = &wbar[s];
      const bool odd_last = 2 * i + 1 >= n_my;
      const long long sb = 2LL * i + ((odd_last && odd_shift < 0) ? -1 : 0);
      const uint8_t* ks = kbase + sb * rec_k;
      const uint8_t* vs = vbase + sb * rec_v;
      mbar_arrive_expect_tx(bar, (uint32_t)(2 * (rec_k + rec_v)));
      if (odd_last && odd_shift > 0) {
        bulk_g2s(dst, ks, (uint32_t)rec_k, bar);
        bulk_g2s(dst + rec_k, ks, (uint32_t)rec_k, bar);
        bulk_g2s(dst + 2 * rec_k, vs, (uint32_t)rec_v, bar);
        bulk_g2s(dst + 2 * rec_k + rec_v, vs, (uint32_t)rec_v, bar);
      } else {
        bulk_g2s(dst, ks, (uint32_t)(2 * rec_k), bar);
        bulk_g2s(dst + 2 * rec_k, vs, (uint32_t)(2 * rec_v), bar);
      }
    };
    if (lane == 0) {
      int s = slot;
      for (int i = 0; i < n_st && i < ns; ++i) {
        issue(i, s);
        s = s + 1 == ns ? 0 : s + 1;
      }
    }
    if (first) {
      grid_dep_wait();  // the q-prep results
      first = false;
    }

    // ---- the lane's query factors for this stream
    uint32_t Qh[KO], Ql[KO];
    float CQ[4], two_e, inv2e;
    {
      const uint32_t* qp = p.qpack + ((size_t)X * 32 + lane) * p.qp_stride;
#pragma unroll
      for (int o = 0; o < KO; ++o) {
        Qh[o] = __ldcg(qp + o);
        Ql[o] = __ldcg(qp + KO + o);
      }
      CQ[0] = __uint_as_float(__ldcg(qp + 2 * KO));
      CQ[1] = __uint_as_float(__ldcg(qp + 2 * KO + 1));
      // distinct registers for the repeated values, so the quad needs no copies
      asm volatile("mov.b32 %0, %1;" : "=f"(CQ[2]) : "f"(CQ[0]));
      asm volatile("mov.b32 %0, %1;" : "=f"(CQ[3]) : "f"(CQ[1]));
      two_e = __uint_as_float(__ldcg(qp + 2 * KO + 2));
      inv2e = __uint_as_float(__ldcg(qp + 2 * KO + 3));
    }

    // ---- main loop
    float m_run[2] = {-INFINITY, -INFINITY}, thr[2] = {-INFINITY, -INFINITY};
    float l_acc[4] = {0.f, 0.f, 0.f, 0.f};
    float acc[VT][4];
#pragma unroll
    for (int t = 0; t < VT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    int done = 0;
    for (int i = 0; i < n_st; ++i) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&wbar[slot], par));
      if (!ok) {
        timed_out = true;
        break;
      }
      const uint8_t* kr = wring + slot * p.stage_bytes;
      const uint8_t* vr = kr + 2 * rec_k;
      const int masked = 2 * i + 1 < n_my ? -1 : odd_mask;  // slot whose scores are dropped

      float sc[2][2][4], zc[4];
      key_stage(kr, kr + rec_k, geo_k, Qh, Ql, CQ, Z4, lane, c, mg, sc, zc);
      if (masked >= 0) {
#pragma unroll
        for (int bb = 0; bb < 2; ++bb)
          if (bb == masked) {
#pragma unroll
            for (int m = 0; m < 2; ++m) sc[bb][m][0] = sc[bb][m][1] = sc[bb][m][2] = sc[bb][m][3] = -INFINITY;
          }
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
        mma16816(l_acc, O4[0], O4[1], O4[2], O4[3], pb[bb][0][0], pb[bb][0][1]);
        mma16816(l_acc, O4[0], O4[1], O4[2], O4[3], pb[bb][1][0], pb[bb][1][1]);
      }
      value_block<VQ>(vr, geo_v, lane, g, mg, pb[0], acc);
      value_block<VQ>(vr + rec_v, geo_v, lane, g, mg, pb[1], acc);

      __syncwarp();
      if (lane == 0 && i + ns < n_st) issue(i + ns, slot);
      slot = slot + 1 == ns ? 0 : slot + 1;
      par ^= slot == 0 ? 1u : 0u;
      done = i + 1;
    }
    if (timed_out && n_st > 0) {
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
      }
      __syncwarp();
    }

    // ---- the warp's partial for this segment (running max and sum per
    // head, latent accumulator per padded value channel), kept on chip
    float* part = wp + (size_t)seg * Gq * ms;
    if (lane == 0) flag_s[2 * warp + seg] = (int)X;
    if (g == 0) {
      if (2 * c < Gq) {
        part[(2 * c) * ms + 0] = timed_out ? -INFINITY : m_run[0];
        part[(2 * c) * ms + 1] = timed_out ? 0.f : l_acc[0];
      }
      if (2 * c + 1 < Gq) {
        part[(2 * c + 1) * ms + 0] = timed_out ? -INFINITY : m_run[1];
        part[(2 * c + 1) * ms + 1] = timed_out ? 0.f : l_acc[1];
      }
    }
#pragma unroll
    for (int t = 0; t < VT; ++t) {
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const int pch = 16 * t + g + 8 * (e2 >> 1), h = 2 * c + (e2 & 1);
        if (pch < p.rvp && h < Gq) part[h * ms + kPartHead + pch] = timed_out ? 0.f : acc[t][e2];
      }
    }
  }

  // ---- end phase, per stream this CTA touches: merge the warps (log-sum-exp),
  // fold in the fp32 tail tokens (the CTA holding the stream's last full
  // block; with no full block, CTA x / nw serves stream x), apply V^V^T, and
  // either finish the stream or leave a projected partial for the stream's
  // last CTA to merge.  A 16-warp CTA that covers two streams runs the two in
  // parallel, 8 warps and one end area each.
  __syncthreads();  // every warp is done with its ring and its partials
  grid_dep_wait();  // q~, c and the tickets come from the preceding launch
  // the CTA's streams, from the warps' segment flags (one per lane)
  const int fl = lane < 2 * nw ? flag_s[lane] : -1;
  int xlo, xhi;
  if (nf > 0) {
    int lo = fl >= 0 ? fl : 0x7fffffff, hi = fl;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    xlo = lo;
    xhi = hi;
  } else {
    xlo = blockIdx.x * nw;
    xhi = (int)min((long long)xlo + nw, p.streams) - 1;
  }
  const int rk = p.k.r, rv = p.v.r, tks = rk | 1, rvp = p.rvp;
  const float* wpa = reinterpret_cast<const float*>(smem + p.wp_off);

  // One stream x by the group of lnt threads (ltid = rank in the group) that
  // synchronises on named barrier bar_id, with end area es and barrier ebar.
  auto end_stream = [&](int x, const EndSmem& es, uint64_t* ebar, uint32_t& epar, int& bv_group, int ltid, int lnt,
                        int bar_id) {
    const int lw = ltid >> 5, lnw = lnt >> 5;
    const int hpt = (8 * kHeadDim + lnt - 1) / lnt;  // query heads per thread in the projection: 4, 3 or 2
    const int d = ltid & (kHeadDim - 1), h0 = (ltid >> 7) * hpt;
    long long c_first, c_last;
    const int xi = x - info_s[0];
    if (xi >= 0 && xi < 2) {
      c_first = info_s[1 + 2 * xi];
      c_last = info_s[2 + 2 * xi];
    } else {
      c_first = c_last = x / nw;
      if (nf > 0) {
        c_first = block_owner((long long)x * nf, T, W) / nw;
        c_last = block_owner((long long)x * nf + nf - 1, T, W) / nw;
      }
    }
    const int cslot = (int)(blockIdx.x - c_first), nseg = (int)(c_last - c_first + 1);
    const long long len_x = stream_len(x);  // this stream's tokens: its full blocks, then the tail
    const long long nf_x = len_x / kBlock;
    const int n_tail = (int)(len_x % kBlock);
    const bool tail_here = n_tail > 0 && blockIdx.x == c_last;
    const int kh = (int)(x % p.Hkv), bb = (int)(x / p.Hkv);
    const int gv = kh / p.v.heads_per_group;
    const bool new_basis = gv != bv_group;
    const bool copies = new_basis || tail_here;
    if (ltid == 0 && copies) {
      // the V basis rows (unless this group's are in place), and for the
      // tail: q~, c and the value tail (the area was last read through the
      // generic proxy: order those reads first)
      fence_proxy_async_smem();
      const uint32_t bv = new_basis ? (uint32_t)rv * 512u : 0u;
      const uint32_t tv = p.v.quantize ? (uint32_t)(kBlock * rv * 4) : (uint32_t)p.v.rec_bytes;
      asm volatile("fence.proxy.async.global;" ::: "memory");
      mbar_arrive_expect_tx(ebar, bv + (tail_here ? 4096u + 32u + tv : 0u));
      if (new_basis) bulk_g2s(es.bv, p.v.basisT + (size_t)gv * rv * kHeadDim, bv, ebar);
      if (tail_here) {
        bulk_g2s(es.qt, p.qt + (size_t)x * 8 * kHeadDim, 4096u, ebar);
        bulk_g2s(es.cq, p.cq + (size_t)x * 8, 32u, ebar);
        const void* src = p.v.quantize ? static_cast<const void*>(p.v.tail + (size_t)x * kBlock * rv)
                                       : static_cast<const void*>(p.v.blocks + ((size_t)x * p.v.n_blk_cap + nf_x) * p.v.rec_bytes);
        bulk_g2s(es.tv, src, tv, ebar);
      }
    }
    bv_group = gv;
    // the key tail [32][rk]: rows lw + lnw v, channels lane + 32 u; loaded
    // now, stored below at an odd row stride
    float tkv[4][4];
    if (tail_here) {
      const float* src = p.k.tail + (size_t)x * kBlock * rk;
#pragma unroll
      for (int v = 0; v < 4; ++v)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = lw + lnw * v, j = lane + 32 * u;
          tkv[v][u] = (t < kBlock && j < rk) ? __ldcg(src + t * rk + j) : 0.f;
        }
    }
    // per head: the maximum over the stream's warp segments, their weights
    // (zero for every other slot) and the sum; lane = slot
    const unsigned int wmask = __ballot_sync(0xffffffffu, fl == x);  // the warp segments of stream x
    for (int h = lw; h < Gq; h += lnw) {
      const bool in = (wmask >> lane) & 1u;
      const float mk = in ? wpa[((size_t)lane * Gq + h) * ms] : -INFINITY;
      const float lk = in ? wpa[((size_t)lane * Gq + h) * ms + 1] : 0.f;
      float M = mk;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float wk = mk == -INFINITY ? 0.f : ex2(mk - M);
      float L = wk * lk;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
      es.sw[lane * 8 + h] = wk;
      if (lane == 0) {
        es.hm[h] = M;
        es.hl[h] = L;
      }
    }
    bar_sync(bar_id, lnt);
    // merged latent per (head, real value channel), over the covering slots
    // in slot order (the slots of one stream are those of a run of warps)
    {
      const int k_lo = wmask ? __ffs(wmask) - 1 : 0, k_hi = wmask ? 32 - __clz(wmask) : 0;
      for (int i = ltid; i < Gq * rvp; i += lnt) {
        const int h = i / rvp, pch = i - h * rvp;
        const int j2 = padded_to_channel(pch, rv, p.v.n_hi, p.v.n_hi_oct, p.v.quantize);
        if (j2 < 0) continue;
        float v = 0.f;
#pragma unroll 4
        for (int k = k_lo; k < k_hi; ++k) v = fmaf(es.sw[k * 8 + h], wpa[((size_t)k * Gq + h) * ms + kPartHead + pch], v);
        es.ol[h * kHeadDim + j2] = v;
      }
    }
    if (tail_here) {
#pragma unroll
      for (int v = 0; v < 4; ++v)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = lw + lnw * v, j = lane + 32 * u;
          if (t < kBlock && j < rk) es.tk[t * tks + j] = tkv[v][u];
        }
    }
    bool got = true;
    if (copies) {
      got = mbar_wait_bounded(ebar, epar);
      epar ^= 1u;
      if (!got && ltid == 0) set_dev_error(p.k.hdr, PALU_DEVERR_TIMEOUT);
    }
    bar_sync(bar_id, lnt);
    if (tail_here) {
      // tail scores in log2 units (q~ and c carry the softmax scale): warp
      // per head, lane t
      for (int h = lw; h < Gq; h += lnw) {
        if (lane < n_tail) {
          const int t = lane;
          float sc_t = es.cq[h];
          const float* tkr = es.tk + t * tks;
          const float* qh = es.qt + h * kHeadDim;
          for (int j2 = 0; j2 < p.k.n_hi; ++j2) sc_t = fmaf(qh[j2], tkr[j2], sc_t);
          const float* ql = qh + 8 * p.k.n_hi_oct - p.k.n_hi;
          for (int j2 = p.k.n_hi; j2 < rk; ++j2) sc_t = fmaf(ql[j2], tkr[j2], sc_t);
          es.st[h * kBlock + t] = got ? sc_t : -INFINITY;
        }
        __syncwarp();
        const float m_old = es.hm[h];
        const float st = lane < n_tail ? es.st[h * kBlock + lane] : -INFINITY;
        float M = fmaxf(m_old, st);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float w_old = m_old == -INFINITY ? 0.f : ex2(m_old - M);
        const float pt = st == -INFINITY ? 0.f : ex2(st - M);
        float L = pt;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        __syncwarp();
        es.st[h * kBlock + lane] = pt;
        if (lane == 0) {
          es.hm[h] = M;
          es.hl[h] = fmaf(w_old, es.hl[h], L);
          es.wo[h] = w_old;
        }
      }
      bar_sync(bar_id, lnt);
      for (int i = ltid; i < Gq * rv; i += lnt) {
        const int h = i / rv, j2 = i - h * rv;
        float a = es.wo[h] * es.ol[h * kHeadDim + j2];
        for (int t = 0; t < n_tail; ++t) {
          float lv;
          if (p.v.quantize) {
            lv = es.tv[t * rv + j2];
          } else {
            // the partial block's fp16 record (fragment order)
            const int kk = 2 * (t >> 4) + ((t & 15) >> 3);
            const int ln = 4 * (j2 & 7) + ((t & 7) >> 1);
            lv = __half2float(*reinterpret_cast<const __half*>(reinterpret_cast<const uint8_t*>(es.tv) +
                                                               512 * (j2 >> 3) + 16 * ln + 4 * kk + 2 * (t & 1)));
          }
          a = fmaf(es.st[h * kBlock + t], lv, a);
        }
        es.ol[h * kHeadDim + j2] = a;
      }
      bar_sync(bar_id, lnt);
    }
    // o[h][d] = sum_j latent[h][j] V[d][j]: thread (d, hpt heads)
    float o4[4] = {0.f, 0.f, 0.f, 0.f};
    {
      int j2 = 0;
      for (; j2 + 4 <= rv; j2 += 4) {
        const float b0 = es.bv[j2 * kHeadDim + d], b1 = es.bv[(j2 + 1) * kHeadDim + d];
        const float b2 = es.bv[(j2 + 2) * kHeadDim + d], b3 = es.bv[(j2 + 3) * kHeadDim + d];
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          if (hh < hpt && h0 + hh < Gq) {
            const float4 o = *reinterpret_cast<const float4*>(es.ol + (h0 + hh) * kHeadDim + j2);
            o4[hh] = fmaf(o.x, b0, fmaf(o.y, b1, fmaf(o.z, b2, fmaf(o.w, b3, o4[hh]))));
          }
        }
      }
      for (; j2 < rv; ++j2) {
        const float bvj = es.bv[j2 * kHeadDim + d];
#pragma unroll
        for (int hh = 0; hh < 4; ++hh)
          if (hh < hpt && h0 + hh < Gq) o4[hh] = fmaf(es.ol[(h0 + hh) * kHeadDim + j2], bvj, o4[hh]);
      }
    }
    const float mu = __ldg(p.v.mu + (size_t)gv * kHeadDim + d);
    const long long out0 = ((long long)bb * p.Hq + (long long)kh * Gq) * kHeadDim + d;
    if (nseg == 1) {
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const int h = h0 + hh;
        if (hh < hpt && h < Gq) store_out(p, out0 + (long long)h * kHeadDim, fmaf(o4[hh], 1.f / es.hl[h], mu));
      }
    } else if (cslot < p.seg_max && nseg <= p.seg_max) {
      float* part = p.ws + ((size_t)x * p.seg_max + cslot) * (size_t)Gq * kOutPart;
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const int h = h0 + hh;
        if (hh < hpt && h < Gq) {
          part[(size_t)h * kOutPart + kOutHead + d] = o4[hh];
          if (d == 0) {
            part[(size_t)h * kOutPart] = es.hm[h];
            part[(size_t)h * kOutPart + 1] = es.hl[h];
          }
        }
      }
      bar_sync(bar_id, lnt);  // the group's partial is written
      if (ltid == 0) {
        asm volatile("fence.acq_rel.gpu;" ::: "memory");  // release the partial
        const unsigned int prev = atomicAdd(p.tickets + x, 1u);
        es.flag[0] = prev + 1 == (unsigned int)nseg ? 1 : 0;
      }
      bar_sync(bar_id, lnt);
      if (es.flag[0]) {
        // the stream's last CTA: merge the nseg projected partials, online
        // (running max per head), two partials' loads in flight at a time
        asm volatile("fence.acq_rel.gpu;" ::: "memory");  // acquire the others' partials
        const float* pbase = p.ws + (size_t)x * p.seg_max * Gq * kOutPart;
        float Mh[4], Lh[4], Oh[4];
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          Mh[hh] = -INFINITY;
          Lh[hh] = 0.f;
          Oh[hh] = 0.f;
        }
#pragma unroll 1
        for (int k0 = 0; k0 < nseg; k0 += 2) {
          float mv[2][4], lv[2][4], ov[2][4];
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
              const int h = h0 + hh;
              const bool ok = k0 + u < nseg && hh < hpt && h < Gq;
              const float* pk = pbase + ((size_t)(k0 + u) * Gq + h) * kOutPart;
              mv[u][hh] = ok ? __ldcg(pk) : -INFINITY;
              lv[u][hh] = ok ? __ldcg(pk + 1) : 0.f;
              ov[u][hh] = ok ? __ldcg(pk + kOutHead + d) : 0.f;
            }
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
              if (mv[u][hh] == -INFINITY) continue;
              const float Mn = fmaxf(Mh[hh], mv[u][hh]);
              const float a = ex2(Mh[hh] - Mn), w = ex2(mv[u][hh] - Mn);
              Lh[hh] = fmaf(Lh[hh], a, lv[u][hh] * w);
              Oh[hh] = fmaf(Oh[hh], a, ov[u][hh] * w);
              Mh[hh] = Mn;
            }
        }
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const int h = h0 + hh;
          if (hh < hpt && h < Gq) store_out(p, out0 + (long long)h * kHeadDim, fmaf(Oh[hh], 1.f / Lh[hh], mu));
        }
        if (ltid == 0) p.tickets[x] = 0u;
      }
    } else if (ltid == 0) {
      set_dev_error(p.k.hdr, PALU_DEVERR_CAPACITY);
    }
    bar_sync(bar_id, lnt);  // the end area is reused by the next stream
  };

  uint64_t* ebar = bars + nw * ns;  // the end phase's copies (two, for two groups)
  // two streams: two groups of 8 warps, each with its own end area and barrier
  const bool split = xhi == xlo + 1 && nw == kMaxDecWarps && p.end_off2 >= 0;
  const int half = (split && warp >= nw / 2) ? 1 : 0;
  const EndSmem es = end_smem(smem + (half ? p.end_off2 : p.end_off), p);
  uint32_t epar = 0;
  int bv_group = -1;
  const int x_first = split ? xlo + half : xlo, x_last = split ? xlo + half : xhi;
  for (int x = x_first; x <= x_last; ++x)
    end_stream(x, es, ebar + half, epar, bv_group, tid - half * (nt / 2), split ? nt / 2 : nt, split ? 1 + half : 0);
  if (grows) {
    // the last CTA stores the new length of both caches (every CTA read the
    // old one at its start, before it counted itself here)
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const unsigned int prev = atomicAdd(p.tickets + p.streams, 1u);
      if (prev + 1 == gridDim.x) {
        __threadfence();
        if (ragged) {
          advance_ragged_lengths(p.k, nullptr, 1);
          advance_ragged_lengths(p.v, nullptr, 1);
        } else {
          p.k.hdr->length = len;
          p.v.hdr->length = len;
        }
        p.tickets[p.streams] = 0u;
        __threadfence();
      }
    }
  }
}

typedef void (*DecodeKernel)(const DecodeParams);

// Instantiations are spread over translation units (parallel build):
// exact octet counts up to 8 on both sides, one unit per key count; exact
// wider records that common ranks produce (12 warps, as the class kernels);
// and the class kernels for the other larger ranks, one unit per key class.
template <int KE>
DecodeKernel decode_kernel_exact(int ve, bool vq);
DecodeKernel decode_kernel_wide(int ke, int ve, int kc, int vc, bool vq);  // nullptr when none
template <int KC>
DecodeKernel decode_kernel_class(int vc, bool vq);

}  // namespace palu
