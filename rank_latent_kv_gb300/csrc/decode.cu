// Host side of the fused latent decode attention: launch planning and the
// C entry points.  The kernel itself (and the method it follows) is described
// in decode_kernel.cuh.
#include <math.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "append_one.cuh"
#include "decode_kernel.cuh"

namespace palu {

// ------------------------------------------------------------------ q-prep
// One CTA per (batch, KV head) stream: q~ = q V^K and c = q . mu^K for its
// query heads, scaled by softmax scale * log2 e, and for the decode kernel the
// per-lane fp16 hi/lo factors prescaled by 2^e with
// |q~| 2^e max(1, largest stored scale) < 2^14, so that every fp16 operand and
// product of the score MMAs stays finite.
// Scratch of one stream's q-prep (16-byte aligned base).
struct QprepSmem {
  float (*q_s)[kHeadDim];
  float* mu_s;
  float* B_s;  // [32][129] basis rows, padded rows: conflict-free column reads
  float (*qt_s)[kHeadDim];
  float *red_s, *cq_s;
};
constexpr size_t kQprepSmemBytes = sizeof(float) * (8 * kHeadDim + kHeadDim + 32 * 129 + 8 * kHeadDim + 16);
__device__ __forceinline__ QprepSmem qprep_smem(uint8_t* base) {
  QprepSmem s;
  float* f = reinterpret_cast<float*>(base);
  s.q_s = reinterpret_cast<float(*)[kHeadDim]>(f);
  s.mu_s = f + 8 * kHeadDim;
  s.qt_s = reinterpret_cast<float(*)[kHeadDim]>(f + 9 * kHeadDim);
  s.B_s = f + 17 * kHeadDim;
  s.red_s = s.B_s + 32 * 129;
  s.cq_s = s.red_s + 8;
  return s;
}

// Stream X's q-prep by a 256-thread CTA.  max_s_floor: a scale the stream's
// blocks may hold that the header need not show yet (one this CTA just stored).
__device__ void qprep_stream(const DecodeParams& p, long long X, float max_s_floor, const QprepSmem& sm) {
  float (*q_s)[kHeadDim] = sm.q_s;
  float* mu_s = sm.mu_s;
  float* B_s = sm.B_s;
  float (*qt_s)[kHeadDim] = sm.qt_s;
  float* red_s = sm.red_s;
  float* cq_s = sm.cq_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = (int)(X / p.Hkv), kh = (int)(X % p.Hkv), Gq = p.Gq;
  const int gk = kh / p.k.heads_per_group;
  const int npch = 8 * p.k.n_oct;
  const float* basis_g = p.k.basisT + (size_t)gk * p.k.r * kHeadDim;
  {
    const int h = tid >> 5, d4 = tid & 31;
    float4 qv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h < Gq) {
      const uint2 raw =
          __ldg(reinterpret_cast<const uint2*>(p.q + ((long long)b * p.Hq + (long long)kh * Gq + h) * kHeadDim) + d4);
      const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
      const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
      qv = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    *reinterpret_cast<float4*>(&q_s[h][4 * d4]) = qv;
    if (tid < 32)
      *reinterpret_cast<float4*>(&mu_s[4 * tid]) = __ldg(reinterpret_cast<const float4*>(p.k.mu + (size_t)gk * kHeadDim) + tid);
    for (int i = tid; i < 8 * kHeadDim; i += 256)
      if ((i & (kHeadDim - 1)) >= npch) qt_s[i >> 7][i & (kHeadDim - 1)] = 0.f;
  }
  float amax = 0.f;
  for (int ch = 0; ch < npch; ch += 32) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = tid + 256 * u, r = i >> 5, c4 = i & 31, pch = ch + r;
      const int j = pch < npch ? padded_to_channel(pch, p.k.r, p.k.n_hi, p.k.n_hi_oct, 1) : -1;
      v[u] = j >= 0 ? __ldg(reinterpret_cast<const float4*>(basis_g + (size_t)j * kHeadDim) + c4)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (ch > 0) __syncthreads();  // the previous chunk's readers are done
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = tid + 256 * u, r = i >> 5, c4 = i & 31;
      float* dst = B_s + r * 129 + 4 * c4;
      dst[0] = v[u].x;
      dst[1] = v[u].y;
      dst[2] = v[u].z;
      dst[3] = v[u].w;
    }
    __syncthreads();
    const float* br = B_s + lane * 129;
    float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
    for (int d4 = 0; d4 < kHeadDim / 4; ++d4) {
      const float4 q4 = *reinterpret_cast<const float4*>(&q_s[warp][4 * d4]);
      a0 = fmaf(q4.x, br[4 * d4], fmaf(q4.y, br[4 * d4 + 1], a0));
      a1 = fmaf(q4.z, br[4 * d4 + 2], fmaf(q4.w, br[4 * d4 + 3], a1));
    }
    const int pch = ch + lane;
    const float qt = (warp < Gq && pch < npch) ? (a0 + a1) * p.scale_log2 : 0.f;
    if (pch < kHeadDim) qt_s[warp][pch] = qt;
    amax = fmaxf(amax, fabsf(qt));
  }
  {
    float s = 0.f;
    if (warp < Gq) {
      const float4 qq = *reinterpret_cast<const float4*>(&q_s[warp][4 * lane]);
      const float4 mm = *reinterpret_cast<const float4*>(&mu_s[4 * lane]);
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
  // scaled q~ and c for the combine's tail tokens
  for (int i = tid; i < 8 * kHeadDim; i += 256) p.qt[(size_t)X * 8 * kHeadDim + i] = qt_s[i >> 7][i & (kHeadDim - 1)];
  if (tid < 8) p.cq[(size_t)X * 8 + tid] = cq_s[tid];
  if (warp == 0) {
    amax = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) amax = fmaxf(amax, red_s[w]);
    const float max_s = fmaxf(__uint_as_float(__ldcg(&p.k.hdr->max_scale)), max_s_floor);
    const float xm = amax * fmaxf(1.f, max_s);
    int e = 0;
    if (xm > 0.f) {
      const int ex = (int)((__float_as_uint(xm) >> 23) & 0xFF) - 126;  // xm < 2^ex
      e = min(max(14 - ex, -120), 120);
    }
    const float two_e = pow2i(e), inv2e = pow2i(-e);
    const int g = lane >> 2, c = lane & 3, ko = p.qp_ko;
    uint32_t* qp = p.qpack + ((size_t)X * 32 + lane) * p.qp_stride;
    for (int o = 0; o < ko; ++o) {
      const float x0 = 8 * o + 2 * c < kHeadDim ? qt_s[g][8 * o + 2 * c] * two_e : 0.f;
      const float x1 = 8 * o + 2 * c + 1 < kHeadDim ? qt_s[g][8 * o + 2 * c + 1] * two_e : 0.f;
      const uint32_t hi = pack_f16x2(x0, x1);
      const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      qp[o] = hi;
      qp[ko + o] = pack_f16x2(x0 - hf.x, x1 - hf.y);
    }
    qp[2 * ko] = __float_as_uint(cq_s[2 * c] * two_e);
    qp[2 * ko + 1] = __float_as_uint(cq_s[2 * c + 1] * two_e);
    qp[2 * ko + 2] = __float_as_uint(two_e);
    qp[2 * ko + 3] = __float_as_uint(inv2e);
  }
}

__global__ void __launch_bounds__(256) latent_qprep_kernel(const DecodeParams p) {
  __shared__ __align__(16) uint8_t scratch[kQprepSmemBytes];
  grid_dep_launch();
  qprep_stream(p, blockIdx.x, 0.f, qprep_smem(scratch));
}

// ------------------------------------------------------------------ step prologue
// One decode step's work before attention (SURVEY "next" row: fused per-step
// pipeline), in one launch: grid (streams, 2).  CTA (X, 0) appends stream
// X's new key token and then prepares stream X's query factors (the prescale
// sees a block this append completed without waiting on other CTAs: only
// stream X's scales meet stream X's factors); CTA (X, 1) appends the new
// value token.  Each cache's last appending CTA publishes its new length.
__global__ void __launch_bounds__(256) latent_step_prologue_kernel(const DecodeParams p, const __half* k_new,
                                                                   const __half* v_new) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ uint64_t bar;
  const int tid = threadIdx.x;
  const long long X = blockIdx.x;
  const bool key = blockIdx.y == 0;
  const CacheView& cv = key ? p.k : p.v;
  const int h = (int)(X % p.Hkv), b = (int)(X / p.Hkv);
  const AppendSmem sm = append_smem(dsm, cv.r, cv.rec_bytes);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, (uint32_t)cv.r * 512u);
    bulk_g2s(sm.bas, cv.basisT + (size_t)(h / cv.heads_per_group) * cv.r * kHeadDim, (uint32_t)cv.r * 512u, &bar);
  }
  const long long p0 = __ldcg(&cv.hdr->length);
  __syncthreads();
  const bool got = mbar_wait_bounded(&bar, 0);
  if (!got && tid == 0) set_dev_error(cv.hdr, PALU_DEVERR_TIMEOUT);
  float s_new = 0.f;
  if (p0 + 1 > cv.capacity) {
    if (X == 0 && tid == 0) set_dev_error(cv.hdr, PALU_DEVERR_CAPACITY);
  } else {
    s_new = append_one_token(cv, (key ? k_new : v_new) + X * kHeadDim, p0, h, b, p.Hkv, sm);
    __syncthreads();
    if (tid == 0) publish_length(cv, p0, (unsigned int)p.streams);
  }
  if (key) {
    __syncthreads();  // the append's scratch is free
    qprep_stream(p, X, s_new, qprep_smem(dsm));
  }
}

// ------------------------------------------------------------------ combine
// One CTA per stream, after the decode kernel: merge the stream's partials
// (log-sum-exp), fold in the fp32 tail tokens, apply V^V^T and + mu^V.
// Dynamic shared memory: V basis [rv][128], tails, partials, tail weights,
// merged latents, denominators.
__global__ void __launch_bounds__(256) latent_combine_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t mbar, mbar_p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long X = blockIdx.x;
  const int b = (int)(X / p.Hkv), kh = (int)(X % p.Hkv), Gq = p.Gq;
  const int rk = p.k.r, rv = p.v.r, ms = kPartHead + p.rvp;
  const int gv = kh / p.v.heads_per_group;
  const int rec_v = p.v.rec_bytes;
  const int tv_bytes = p.v.quantize ? kBlock * rv * 4 : rec_v;
  float* BV_s = reinterpret_cast<float*>(smem);                 // [rv][128]
  float* TK_s = BV_s + (size_t)rv * kHeadDim;                    // [32][rk]
  float* TV_s = TK_s + (size_t)kBlock * rk;                      // [32][rv] (or one fp16 record)
  float* P_s = TV_s + (tv_bytes + 15) / 16 * 4;                  // [nseg][Gq][ms] partials
  float* ST_s = P_s + (size_t)p.seg_max * Gq * ms;               // [8][32] tail scores, then weights
  float* O_s = ST_s + 8 * kBlock;                                // [8][128] merged latents
  float* L_s = O_s + 8 * kHeadDim;                               // [8]

  // everything but the partials and q~ was written before the q-prep launch:
  // fetch it while the decode kernel is still running
  const long long len = __ldcg(&p.k.hdr->length);
  const long long nf = len / kBlock;
  const int n_tail = (int)(len % kBlock);
  const long long T = p.streams * nf;
  int nseg = 0;
  if (T > 0) {
    // the decode launch's warps that take part; one partial per CTA
    const long long W = min((long long)p.dec_grid * kDecWarps, T);
    nseg = (int)(block_owner(X * nf + nf - 1, T, W) / kDecWarps - block_owner(X * nf, T, W) / kDecWarps + 1);
  }
  const float mu_v = __ldg(p.v.mu + (size_t)gv * kHeadDim + (tid & 127));
  if (tid == 0) {
    mbar_init(&mbar, 1);
    mbar_init(&mbar_p, 1);
    fence_mbar_init();
    const uint32_t bytes = (uint32_t)rv * 512u + (n_tail > 0 ? (uint32_t)(kBlock * rk * 4 + tv_bytes) : 0u);
    mbar_arrive_expect_tx(&mbar, bytes);
    bulk_g2s(BV_s, p.v.basisT + (size_t)gv * rv * kHeadDim, (uint32_t)rv * 512u, &mbar);
    if (n_tail > 0) {
      bulk_g2s(TK_s, p.k.tail + (size_t)X * kBlock * rk, (uint32_t)(kBlock * rk * 4), &mbar);
      const void* tv = p.v.quantize ? static_cast<const void*>(p.v.tail + (size_t)X * kBlock * rv)
                                    : static_cast<const void*>(p.v.blocks + ((size_t)X * p.v.n_blk_cap + nf) * rec_v);
      bulk_g2s(TV_s, tv, (uint32_t)tv_bytes, &mbar);
    }
  }
  grid_dep_wait();  // the decode kernel's partials (and, through it, q~ and c)
  if (tid == 0) {
    // the stream's partials are contiguous: one bulk copy
    const uint32_t pbytes = (uint32_t)nseg * Gq * ms * 4u;
    asm volatile("fence.proxy.async.global;" ::: "memory");
    mbar_arrive_expect_tx(&mbar_p, pbytes);
    if (pbytes > 0) bulk_g2s(P_s, p.ws + (size_t)X * p.seg_max * Gq * ms, pbytes, &mbar_p);
  }
  __syncthreads();  // barriers initialised
  const bool got = mbar_wait_bounded(&mbar, 0) && mbar_wait_bounded(&mbar_p, 0);
  if (!got && tid == 0) set_dev_error(p.k.hdr, PALU_DEVERR_TIMEOUT);
  // tail scores (log2 units)
  const float* qt = p.qt + (size_t)X * 8 * kHeadDim;
  for (int i = tid; i < n_tail * 8; i += 256) {
    const int t = i >> 3, h = i & 7;
    float sc_t = -INFINITY;
    if (h < Gq) {
      sc_t = __ldcg(p.cq + (size_t)X * 8 + h);
      for (int j2 = 0; j2 < rk; ++j2) {
        const int pch = j2 < p.k.n_hi ? j2 : 8 * p.k.n_hi_oct + (j2 - p.k.n_hi);
        sc_t = fmaf(__ldcg(qt + h * kHeadDim + pch), TK_s[t * rk + j2], sc_t);
      }
    }
    ST_s[h * kBlock + t] = sc_t;
  }
  __syncthreads();
  // warp h: max, weights (over the partials' m), denominator
  if (warp < Gq) {
    const int h = warp;
    float M = -INFINITY;
    for (int sg = lane; sg < nseg; sg += 32) M = fmaxf(M, P_s[(sg * Gq + h) * ms]);
    const float st = lane < n_tail ? ST_s[h * kBlock + lane] : -INFINITY;
    M = fmaxf(M, st);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int sg = lane; sg < nseg; sg += 32) {
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
  for (int i = tid; i < Gq * p.rvp; i += 256) {
    const int h = i / p.rvp, pch = i - h * p.rvp;
    const int j2 = padded_to_channel(pch, rv, p.v.n_hi, p.v.n_hi_oct, p.v.quantize);
    if (j2 < 0) continue;
    float a4[4] = {0.f, 0.f, 0.f, 0.f};
    int sg = 0;
    for (; sg + 4 <= nseg; sg += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float* pr = P_s + ((size_t)(sg + u) * Gq + h) * ms;
        a4[u] = fmaf(pr[0], pr[kPartHead + pch], a4[u]);
      }
    }
    for (; sg < nseg; ++sg) {
      const float* pr = P_s + ((size_t)sg * Gq + h) * ms;
      a4[0] = fmaf(pr[0], pr[kPartHead + pch], a4[0]);
    }
    float a = (a4[0] + a4[1]) + (a4[2] + a4[3]);
    for (int t = 0; t < n_tail; ++t) {
      float lv;
      if (p.v.quantize) {
        lv = TV_s[t * rv + j2];
      } else {
        const int kk = 2 * (t >> 4) + ((t & 15) >> 3);
        const int ln = 4 * (j2 & 7) + ((t & 7) >> 1);
        lv = __half2float(*reinterpret_cast<const __half*>(reinterpret_cast<const uint8_t*>(TV_s) + 512 * (j2 >> 3) +
                                                           16 * ln + 4 * kk + 2 * (t & 1)));
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
    int j2 = 0;
    for (; j2 + 4 <= rv; j2 += 4) {
      const float b0 = BV_s[j2 * kHeadDim + d], b1 = BV_s[(j2 + 1) * kHeadDim + d];
      const float b2 = BV_s[(j2 + 2) * kHeadDim + d], b3 = BV_s[(j2 + 3) * kHeadDim + d];
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const float4 o = *reinterpret_cast<const float4*>(O_s + (h0 + hh) * kHeadDim + j2);
        o4[hh] = fmaf(o.x, b0, fmaf(o.y, b1, fmaf(o.z, b2, fmaf(o.w, b3, o4[hh]))));
      }
    }
    for (; j2 < rv; ++j2) {
      const float bv = BV_s[j2 * kHeadDim + d];
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) o4[hh] = fmaf(O_s[(h0 + hh) * kHeadDim + j2], bv, o4[hh]);
    }
    const float mu = mu_v;
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

struct DecodePlan {
  int KC, VC;
  bool VQ;
  int ns, stage_bytes, ring_off, wp_off, smem, grid, seg_max, rvp, qp_ko, qp_stride;
  size_t comb_smem;
  size_t qpack_off, qt_off, cq_off, part_off, ws_bytes;
  DecodeKernel kern;
};

static DecodeKernel pick_kernel(int ke, int ve, int kc, int vc, bool vq) {
  if (ke <= 8 && ve <= 8) {
    switch (ke) {
      case 1: return decode_kernel_exact<1>(ve, vq);
      case 2: return decode_kernel_exact<2>(ve, vq);
      case 3: return decode_kernel_exact<3>(ve, vq);
      case 4: return decode_kernel_exact<4>(ve, vq);
      case 5: return decode_kernel_exact<5>(ve, vq);
      case 6: return decode_kernel_exact<6>(ve, vq);
      case 7: return decode_kernel_exact<7>(ve, vq);
      case 8: return decode_kernel_exact<8>(ve, vq);
      default: return nullptr;
    }
  }
  switch (kc) {
    case 1: return decode_kernel_class<1>(vc, vq);
    case 2: return decode_kernel_class<2>(vc, vq);
    case 3: return decode_kernel_class<3>(vc, vq);
    case 4: return decode_kernel_class<4>(vc, vq);
    default: return nullptr;
  }
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
  // record class: ceil(n_oct / 4); for quantized records this is the number of
  // 4-bit octets, which fixes where every octet sits
  pl->KC = (k->n_oct + 3) / 4;
  pl->VC = (v->n_oct + 3) / 4;
  pl->VQ = v->quantize != 0;
  if (pl->VQ && pl->VC != v->n_hi_oct) return fail(PALU_ERR_UNSUPPORTED, "unexpected value record layout");
  if (pl->KC != k->n_hi_oct) return fail(PALU_ERR_UNSUPPORTED, "unexpected key record layout");
  pl->kern = pick_kernel(k->n_oct, v->n_oct, pl->KC, pl->VC, pl->VQ);
  if (!pl->kern) return fail(PALU_ERR_UNSUPPORTED, "no decode kernel for this rank");
  pl->qp_ko = (k->n_oct <= 8 && v->n_oct <= 8) ? k->n_oct : 4 * pl->KC;  // the kernel's key octets
  pl->qp_stride = (2 * pl->qp_ko + 4 + 3) / 4 * 4;
  const int rec_k = k->record_bytes, rec_v = v->record_bytes;
  pl->stage_bytes = 2 * (rec_k + rec_v);
  pl->ns = pl->stage_bytes <= 2048 ? 4 : pl->stage_bytes <= 6144 ? 3 : 2;
  pl->rvp = 8 * v->n_oct;
  pl->ring_off = (int)align_up(kDecBarOff + 8 * kDecWarps * pl->ns, 128);
  const int64_t streams = (int64_t)k->batch * k->kv_heads;
  const int sms = device_sm_count();
  const size_t rings = (size_t)kDecWarps * pl->ns * pl->stage_bytes;
  pl->wp_off = (int)align_up(pl->ring_off + rings, 16);
  pl->smem = (int)(pl->wp_off + (size_t)kDecWarps * 2 * Gq * (kPartHead + pl->rvp) * 4);
  if (pl->smem > 227 * 1024) return fail(PALU_ERR_UNSUPPORTED, "decode shared-memory plan exceeds 227 KB");
  int per_sm = 0;
  palu_status st = kernel_occupancy(reinterpret_cast<const void*>(pl->kern), kDecThreads, pl->smem, &per_sm);
  if (st != PALU_OK) return st;
  int64_t grid = (int64_t)sms * std::min(per_sm, 4);
  grid = std::min<int64_t>(grid, std::max<int64_t>(1, streams * k->n_blk_cap));
  // at least one warp per stream, so that no warp's range spans more than two
  // streams (extra CTAs, if any, simply run in a second wave)
  grid = std::max<int64_t>(grid, (streams + kDecWarps - 1) / kDecWarps);
  pl->grid = (int)std::max<int64_t>(1, grid);
  // the combine stages one stream's partials on chip (one per CTA that
  // touches the stream: at most ceil(CTAs / streams) + 1); with few streams,
  // use fewer CTAs so that they fit
  const int tv_bytes = v->quantize ? kBlock * v->rank * 4 : rec_v;
  const size_t comb_fixed = (size_t)v->rank * 512 + (size_t)128 * k->rank + align_up(tv_bytes, 16) +
                            8 * kBlock * 4 + 8 * kHeadDim * 4 + 32;
  const size_t per_seg = (size_t)Gq * (kPartHead + pl->rvp) * 4;
  const size_t comb_budget = 200 * 1024;
  pl->seg_max = (int)((pl->grid + streams - 1) / streams + 1);
  if (comb_fixed + pl->seg_max * per_seg > comb_budget) {
    const int64_t seg_fit = (int64_t)((comb_budget - comb_fixed) / per_seg);
    if (seg_fit < 2) return fail(PALU_ERR_UNSUPPORTED, "decode merge does not fit in shared memory");
    pl->grid = (int)std::max<int64_t>(1, std::min<int64_t>(pl->grid, streams * (seg_fit - 1)));
    pl->grid = (int)std::max<int64_t>(pl->grid, (streams + kDecWarps - 1) / kDecWarps);
    pl->seg_max = (int)((pl->grid + streams - 1) / streams + 1);
  }
  pl->comb_smem = comb_fixed + pl->seg_max * per_seg;
  if (pl->comb_smem > 227 * 1024) return fail(PALU_ERR_UNSUPPORTED, "decode merge does not fit in shared memory");
  // workspace: packed query factors, q~ and c per stream, partials
  pl->qpack_off = 0;
  pl->qt_off = align_up(pl->qpack_off + sizeof(uint32_t) * (size_t)streams * 32 * pl->qp_stride, 256);
  pl->cq_off = align_up(pl->qt_off + sizeof(float) * (size_t)streams * 8 * kHeadDim, 256);
  pl->part_off = align_up(pl->cq_off + sizeof(float) * (size_t)streams * 8, 256);
  pl->ws_bytes = align_up(pl->part_off + sizeof(float) * (size_t)streams * pl->seg_max * Gq * (kPartHead + pl->rvp), 256);
  return PALU_OK;
}

}  // namespace palu

using namespace palu;

namespace palu {
// Fills the launch parameters shared by palu_decode_attn and palu_decode_step.
static DecodeParams decode_params(const DecodePlan& pl, const palu_cache* k, const palu_cache* v, const void* q,
                                  int32_t q_heads, float softmax_scale, void* out, int32_t out_fp32,
                                  void* workspace) {
  DecodeParams p;
  p.k = make_view(k);
  p.v = make_view(v);
  p.q = static_cast<const __half*>(q);
  p.out = out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.qpack = reinterpret_cast<uint32_t*>(ws + pl.qpack_off);
  p.qt = reinterpret_cast<float*>(ws + pl.qt_off);
  p.cq = reinterpret_cast<float*>(ws + pl.cq_off);
  p.ws = reinterpret_cast<float*>(ws + pl.part_off);
  p.out_fp32 = out_fp32;
  p.Hq = q_heads;
  p.Hkv = k->kv_heads;
  p.Gq = q_heads / k->kv_heads;
  p.rvp = pl.rvp;
  p.ns = pl.ns;
  p.stage_bytes = pl.stage_bytes;
  p.ring_off = pl.ring_off;
  p.wp_off = pl.wp_off;
  p.seg_max = pl.seg_max;
  p.qp_ko = pl.qp_ko;
  p.qp_stride = pl.qp_stride;
  p.dec_grid = pl.grid;
  p.streams = (long long)k->batch * k->kv_heads;
  p.after_append = 0;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)kHeadDim);
  p.scale_log2 = scale * 1.4426950408889634f;
  return p;
}

// The decode kernel and the combine, each started while its predecessor
// finishes (programmatic dependent launch; each waits in-kernel).
static palu_status launch_decode_combine(const DecodePlan& pl, const DecodeParams& p, cudaStream_t strm) {
  const unsigned int n_streams = (unsigned int)p.streams;
  int per_sm = 0;
  palu_status st =
      kernel_occupancy(reinterpret_cast<const void*>(latent_combine_kernel), 256, (int)pl.comb_smem, &per_sm);
  if (st != PALU_OK) return st;
  // decode and combine each start while their predecessor finishes
  // (programmatic dependent launch; each waits in-kernel for the results)
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = strm;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  st = cuda_check(cudaLaunchKernelEx(&cfg, pl.kern, p), "latent_decode_kernel launch");
  if (st != PALU_OK) return st;
  cfg.gridDim = dim3(n_streams);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = pl.comb_smem;
  return cuda_check(cudaLaunchKernelEx(&cfg, latent_combine_kernel, p), "latent_combine_kernel launch");
}
}  // namespace palu

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
  DecodeParams p = decode_params(pl, k, v, q, q_heads, softmax_scale, out, out_fp32, workspace);
  p.after_append = 0;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  latent_qprep_kernel<<<(unsigned int)p.streams, 256, 0, strm>>>(p);
  st = cuda_check(cudaGetLastError(), "latent_qprep_kernel launch");
  if (st != PALU_OK) return st;
  return launch_decode_combine(pl, p, strm);
}

extern "C" palu_status palu_decode_step(palu_cache* k, palu_cache* v, const void* k_new, const void* v_new,
                                        const void* q, int32_t q_heads, float softmax_scale, void* out,
                                        int32_t out_fp32, void* workspace, size_t workspace_bytes, void* stream) {
  DecodePlan pl;
  palu_status st = plan_decode(k, v, q_heads, &pl);
  if (st != PALU_OK) return st;
  if (!k_new || !v_new || !q || !out || !workspace)
    return fail(PALU_ERR_INVALID_ARG, "k_new, v_new, q, out and workspace must be non-NULL");
  if ((((uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)q | (uintptr_t)out | (uintptr_t)workspace) & 15))
    return fail(PALU_ERR_INVALID_ARG, "k_new, v_new, q, out and workspace must be 16-byte aligned");
  if (workspace_bytes < pl.ws_bytes)
    return fail(PALU_ERR_INVALID_ARG, "workspace too small: need " + std::to_string(pl.ws_bytes) + " bytes");
  if (k->length != v->length) return fail(PALU_ERR_INVALID_ARG, "key and value caches differ in length");
  if (k->length + 1 > k->capacity)
    return fail(PALU_ERR_CAPACITY, "the caches are full (capacity " + std::to_string(k->capacity) + " tokens)");
  DecodeParams p = decode_params(pl, k, v, q, q_heads, softmax_scale, out, out_fp32, workspace);
  p.after_append = 1;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  const size_t smem = std::max({append_smem_bytes(k->rank, k->record_bytes),
                                append_smem_bytes(v->rank, v->record_bytes), kQprepSmemBytes});
  int per_sm = 0;
  st = kernel_occupancy(reinterpret_cast<const void*>(latent_step_prologue_kernel), 256, (int)smem, &per_sm);
  if (st != PALU_OK) return st;
  latent_step_prologue_kernel<<<dim3((unsigned int)p.streams, 2), 256, smem, strm>>>(p, static_cast<const __half*>(k_new),
                                                                                 static_cast<const __half*>(v_new));
  st = cuda_check(cudaGetLastError(), "latent_step_prologue_kernel launch");
  if (st != PALU_OK) return st;
  k->length += 1;
  v->length += 1;
  return launch_decode_combine(pl, p, strm);
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
