// The SVDq keys-only low-rank cache (page "veloxquant_mlx.cache.svdq_cache
// module", section "Design"): per-head bases and means, per-channel widths
// from the bit schedule (8, 4, 2, 1, 1, 0, 0, 0), fp16 values kept by the
// caller.  The append projects new keys (error-free float-pair dot products,
// so the fp32 latents are the correctly rounded ones), quantizes every block
// that completes (asymmetric min/max, blog post "VeloxQuant-MLX 0.8.0 adds
// KIVI", "What KIVI is") and packs the codes LSB-first; the decode computes
// each key score q~ . L_t + q . mean (q~ = q V_h) from the codes on the
// tensor cores (exact codes against an fp16 hi/lo pair of q~_j s_j, fp32
// accumulation) and streams the fp16 values through the tensor-core tile
// loop the dense comparator uses.
#include <math.h>

#include <algorithm>
#include <cstring>
#include <vector>

#include "splitk_attend.cuh"
#include "svdq.h"

namespace palu {

constexpr int32_t kSvdqMagic = 0x53564451;  // "SVDQ"
constexpr int kSvdqSchedule[8] = {8, 4, 2, 1, 1, 0, 0, 0};

struct SvdqHeader {
  long long length;
  unsigned int err;
  unsigned int ticket;
  unsigned int pad[12];
};
static_assert(sizeof(SvdqHeader) == 64, "SVDq state header size");

// Device state: header; per head (rank, kept channels, scale/zero offset,
// record bytes); per head and channel the code byte offset and the width;
// the transposed bases [H][r_max][D], the means [H][D], and mean . V as float
// pairs [H][r_max].
struct SvdqLayout {
  size_t head_off, coff_off, bits_off, basis_off, mu_off, mv_off, total;
};
inline SvdqLayout svdq_layout(int H, int r_max) {
  SvdqLayout s;
  s.head_off = 256;
  s.coff_off = align_up(s.head_off + sizeof(int) * 4 * (size_t)H, 256);
  s.bits_off = align_up(s.coff_off + sizeof(int) * (size_t)H * r_max, 256);
  s.basis_off = align_up(s.bits_off + sizeof(int) * (size_t)H * r_max, 256);
  s.mu_off = align_up(s.basis_off + sizeof(float) * (size_t)H * r_max * kHeadDim, 256);
  s.mv_off = align_up(s.mu_off + sizeof(float) * (size_t)H * kHeadDim, 256);
  s.total = align_up(s.mv_off + sizeof(float2) * (size_t)H * r_max, 256);
  return s;
}

struct SvdqView {
  uint8_t* blocks;
  float* tail;
  SvdqHeader* hdr;
  const int* head;      // [H][4]: rank, kept channels, scale/zero byte offset, record bytes of the head
  const int* coff;      // [H][r_max]: byte offset of channel j's codes in the record
  const int* cbits;     // [H][r_max]: width of channel j
  const float* basisT;  // [H][r_max][D]
  const float* mu;      // [H][D]
  const float2* mv;     // [H][r_max]
  long long n_blk_cap, capacity;
  int H, r_max, rec_bytes;
};

inline SvdqView svdq_view(const palu_svdq_cache* c) {
  SvdqView v;
  const SvdqLayout s = svdq_layout(c->kv_heads, c->r_max);
  uint8_t* st = static_cast<uint8_t*>(c->state);
  v.blocks = static_cast<uint8_t*>(c->blocks);
  v.tail = c->tail;
  v.hdr = reinterpret_cast<SvdqHeader*>(st);
  v.head = reinterpret_cast<const int*>(st + s.head_off);
  v.coff = reinterpret_cast<const int*>(st + s.coff_off);
  v.cbits = reinterpret_cast<const int*>(st + s.bits_off);
  v.basisT = reinterpret_cast<const float*>(st + s.basis_off);
  v.mu = reinterpret_cast<const float*>(st + s.mu_off);
  v.mv = reinterpret_cast<const float2*>(st + s.mv_off);
  v.n_blk_cap = c->n_blk_cap;
  v.capacity = c->capacity;
  v.H = c->kv_heads;
  v.r_max = c->r_max;
  v.rec_bytes = c->record_bytes;
  return v;
}

// Widths of a rank's channels: the schedule's 8 groups as equal contiguous
// groups, sizes differing by at most one, the larger groups first.
static void svdq_channel_bits(int r, std::vector<int>& bits) {
  bits.clear();
  for (int g = 0; g < 8; ++g) {
    const int n = r / 8 + (g < r % 8 ? 1 : 0);
    for (int i = 0; i < n; ++i) bits.push_back(kSvdqSchedule[g]);
  }
}

// Record geometry of one head: code offsets, kept channels, scale/zero
// offset, record bytes (a multiple of 16).
static int svdq_record(int r, std::vector<int>& offs, std::vector<int>& bits, int* kept, int* sz_off) {
  svdq_channel_bits(r, bits);
  offs.assign(r, 0);
  int o = 0, k = 0;
  for (int j = 0; j < r; ++j) {
    if (bits[j] == 0) break;
    offs[j] = o;
    o += 4 * bits[j];
    ++k;
  }
  *kept = k;
  *sz_off = o;
  return (int)align_up((size_t)(o + 4 * k), 16);
}

// ------------------------------------------------------------------ init
// One CTA per (head, direction j < rank): row j of the head's transposed
// basis and mean . V[:, j] in fp64, stored as a float pair.
__global__ void svdq_init_kernel(const float* __restrict__ basis, int ld, const float* __restrict__ mu, SvdqView v,
                                 const int* ranks_dev) {
  const int j = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  __shared__ double red[kHeadDim];
  const int r = ranks_dev[4 * h];
  float* basisT = const_cast<float*>(v.basisT);
  float* mu_out = const_cast<float*>(v.mu);
  float2* mv = const_cast<float2*>(v.mv);
  if (j >= r) return;  // uniform per CTA
  const float vj = basis[((size_t)h * kHeadDim + d) * ld + j];
  basisT[((size_t)h * v.r_max + j) * kHeadDim + d] = vj;
  const float m = mu[(size_t)h * kHeadDim + d];
  if (j == 0) mu_out[(size_t)h * kHeadDim + d] = m;
  red[d] = (double)m * (double)vj;
  __syncthreads();
  for (int s = kHeadDim / 2; s > 0; s >>= 1) {
    if (d < s) red[d] += red[d + s];
    __syncthreads();
  }
  if (d == 0) {
    const double t = red[0];
    const float hi = (float)t;
    mv[(size_t)h * v.r_max + j] = make_float2(hi, (float)(t - (double)hi));
  }
}

// ------------------------------------------------------------------ append
struct SvdqEncSmem {
  int xs, bas, lat, sz, rec, total;
};
__host__ __device__ inline int svdq_a16(int x) { return (x + 15) / 16 * 16; }
__host__ __device__ inline SvdqEncSmem svdq_enc_smem(int r_max, int rec_bytes) {
  SvdqEncSmem s;
  s.xs = 0;                                                      // half [32][D]
  s.bas = s.xs + kBlock * kHeadDim * 2;                          // float [r_max][D + 1]
  s.lat = s.bas + svdq_a16(4 * r_max * (kHeadDim + 1));          // float [32][r_max + 1]
  s.sz = s.lat + svdq_a16(4 * kBlock * (r_max + 1));             // half2 [r_max]
  s.rec = s.sz + svdq_a16(4 * r_max);                            // record
  s.total = s.rec + svdq_a16(rec_bytes);
  return s;
}

// grid (blocks touched, kv_heads, batch), 128 threads; two ordered launches
// (phase 1: every block the tokens reach except a last partial one; phase 2:
// that partial block and the new length), as the latent cache's append.
__global__ void __launch_bounds__(128) svdq_encode_kernel(SvdqView cv, const __half* __restrict__ x, long long T,
                                                          int phase) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, b = blockIdx.z, H = cv.H, rm = cv.r_max, ld = rm + 1;
  const int r = cv.head[4 * h], kept = cv.head[4 * h + 1], szo = cv.head[4 * h + 2];
  const SvdqEncSmem L = svdq_enc_smem(rm, cv.rec_bytes);
  __half* xs = reinterpret_cast<__half*>(smem + L.xs);
  float* bas = reinterpret_cast<float*>(smem + L.bas);
  float* lat = reinterpret_cast<float*>(smem + L.lat);
  __half2* sz = reinterpret_cast<__half2*>(smem + L.sz);
  uint8_t* rec = smem + L.rec;
  const long long p0 = __ldcg(&cv.hdr->length), p1 = p0 + T;
  const unsigned int n_cta = gridDim.x * gridDim.y * gridDim.z;
  if (p1 > cv.capacity) {
    if (blockIdx.x == 0 && h == 0 && b == 0 && tid == 0) atomicOr(&cv.hdr->err, (unsigned int)PALU_DEVERR_CAPACITY);
    return;  // nothing written, length unchanged (no CTA takes a ticket)
  }
  const long long blk = phase == 2 ? p1 / kBlock : p0 / kBlock + blockIdx.x;
  const long long lo = blk * kBlock;
  const bool last_partial = blk == p1 / kBlock && p1 % kBlock != 0;
  if (lo < p1 && last_partial == (phase == 2)) {
    const long long new_lo = lo > p0 ? lo : p0;
    const long long hi = (lo + kBlock < p1) ? lo + kBlock : p1;
    const int off_new = (int)(new_lo - lo), n_new = (int)(hi - new_lo);
    const bool complete = (hi - lo) == kBlock;
    const __half* xsrc = x + (((long long)b * H + h) * T + (new_lo - p0)) * kHeadDim;
    for (int i = tid; i < n_new * (kHeadDim / 8); i += blockDim.x) {
      const int t = i / (kHeadDim / 8), q = i % (kHeadDim / 8);
      reinterpret_cast<uint4*>(xs + (off_new + t) * kHeadDim)[q] =
          reinterpret_cast<const uint4*>(xsrc + (long long)t * kHeadDim)[q];
    }
    const float* bsrc = cv.basisT + (size_t)h * rm * kHeadDim;
    for (int i = tid; i < r * (kHeadDim / 4); i += blockDim.x) {
      const int j = i / (kHeadDim / 4), q = i % (kHeadDim / 4);
      const float4 v = reinterpret_cast<const float4*>(bsrc + (size_t)j * kHeadDim)[q];
      float* dst = bas + j * (kHeadDim + 1) + 4 * q;
      dst[0] = v.x;
      dst[1] = v.y;
      dst[2] = v.z;
      dst[3] = v.w;
    }
    __syncthreads();
    // projection: warp w takes tokens off_new + w + 4i, lane takes channels
    // lane + 32k; sum_d x_d V_dj as an unevaluated float pair, minus
    // mean . V[:, j], rounded once to fp32
    {
      float S[8][4], E[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) S[i][k] = E[i][k] = 0.f;
      const int nt = (n_new - warp + 3) / 4;
      for (int d = 0; d < kHeadDim; ++d) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = lane + 32 * k;
          v[k] = j < r ? bas[j * (kHeadDim + 1) + d] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (i < nt) {
            const float xv = __half2float(xs[(off_new + warp + 4 * i) * kHeadDim + d]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float pp, pe, s2, se;
              two_prod(xv, v[k], pp, pe);
              two_sum(S[i][k], pp, s2, se);
              S[i][k] = s2;
              E[i][k] = __fadd_rn(E[i][k], __fadd_rn(se, pe));
            }
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = lane + 32 * k;
        if (j < r) {
          const float2 m = cv.mv[(size_t)h * rm + j];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (i < nt) {
              float a, ae;
              two_sum(S[i][k], -m.x, a, ae);
              const float low = __fadd_rn(__fsub_rn(E[i][k], m.y), ae);
              lat[(off_new + warp + 4 * i) * ld + j] = __fadd_rn(a, low);
            }
          }
        }
      }
    }
    float* tail = cv.tail + ((long long)b * H + h) * kBlock * rm;
    if (complete) {
      for (int i = tid; i < off_new * r; i += blockDim.x) {
        const int t = i / r, j = i % r;
        lat[t * ld + j] = tail[t * rm + j];
      }
      for (int i = tid; i < cv.rec_bytes / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(rec)[i] = 0u;
      __syncthreads();
      // quantize and pack: thread per kept channel (its code words are its own)
      for (int j = tid; j < kept; j += blockDim.x) {
        float mn = lat[j], mx = lat[j];
        for (int t = 1; t < kBlock; ++t) {
          const float v = lat[t * ld + j];
          mn = fminf(mn, v);
          mx = fmaxf(mx, v);
        }
        const int wb = cv.cbits[(size_t)h * rm + j];
        const float qmax = (float)((1 << wb) - 1);
        const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), qmax));
        const __half zh = __float2half_rn(mn);
        const float s32 = __half2float(sh), z32 = __half2float(zh);
        sz[j] = __halves2half2(sh, zh);
        uint32_t* words = reinterpret_cast<uint32_t*>(rec + cv.coff[(size_t)h * rm + j]);
        for (int t = 0; t < kBlock; ++t) {
          float q = 0.f;
          if (s32 != 0.f) {
            q = rintf(__fdiv_rn(__fsub_rn(lat[t * ld + j], z32), s32));
            q = fminf(fmaxf(q, 0.f), qmax);
          }
          const int pos = t * wb;
          words[pos >> 5] |= (uint32_t)q << (pos & 31);
        }
      }
      __syncthreads();
      for (int j = tid; j < kept; j += blockDim.x) reinterpret_cast<__half2*>(rec + szo)[j] = sz[j];
      __syncthreads();
      uint8_t* gdst = cv.blocks + (((long long)b * H + h) * cv.n_blk_cap + blk) * cv.rec_bytes;
      if (bounds_ok(blk < cv.n_blk_cap, cv.hdr))  // (bounds-checking build)
        for (int i = tid; i < cv.rec_bytes / 16; i += blockDim.x)
          reinterpret_cast<uint4*>(gdst)[i] = reinterpret_cast<const uint4*>(rec)[i];
    } else {
      __syncthreads();
      for (int i = tid; i < n_new * r; i += blockDim.x) {
        const int t = off_new + i / r, j = i % r;
        tail[t * rm + j] = lat[t * ld + j];
      }
    }
  }
  if (phase != 2) return;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned int t = atomicAdd(&cv.hdr->ticket, 1u);
    if (t == n_cta - 1) {
      cv.hdr->length = p1;
      cv.hdr->ticket = 0u;
      __threadfence();
    }
  }
}

// ------------------------------------------------------------------ decode
struct SvdqDecParams {
  SvdqView k;
  const __half* v;
  const __half* q;
  float* ws;   // [streams][n_chunks][Gq][2 + D] partials
  long long v_cap, len;
  int Hq, Gq, n_chunks, tiles_per_chunk;
  float scale_log2;
};

// The query factors of stream X = (b, h) by the calling CTA's 128 threads, in
// fp32: qts[i][j] = q_i . V_h[:, j] for the stream's query heads i < Gq (0
// past the rank and for i >= Gq), cqs[i] = q_i . mean_h.  q_s: 4 KB of
// shared scratch.  Ends with a barrier.
__device__ __forceinline__ void svdq_query_factors(const SvdqDecParams& p, int h, int b, float* q_s, float* qts,
                                                   float* cqs) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rm = p.k.r_max, Gq = p.Gq, r = p.k.head[4 * h];
  for (int i = tid; i < 8 * kHeadDim; i += blockDim.x) {
    const int hq = i / kHeadDim, d = i % kHeadDim;
    q_s[i] = hq < Gq ? __half2float(p.q[((long long)b * p.Hq + (long long)h * Gq + hq) * kHeadDim + d]) : 0.f;
  }
  __syncthreads();
  // thread j: direction j of the head's basis against the 8 query rows
  for (int j = tid; j < rm; j += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    if (j < r) {
      const float4* row = reinterpret_cast<const float4*>(p.k.basisT + ((size_t)h * rm + j) * kHeadDim);
      for (int d4 = 0; d4 < kHeadDim / 4; ++d4) {
        const float4 v = __ldg(row + d4);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 qq = *reinterpret_cast<const float4*>(q_s + i * kHeadDim + 4 * d4);
          acc[i] = fmaf(qq.x, v.x, fmaf(qq.y, v.y, fmaf(qq.z, v.z, fmaf(qq.w, v.w, acc[i]))));
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) qts[i * rm + j] = acc[i];
  }
  // warp w: q_i . mean_h for i = w, w + 4
  for (int i = warp; i < 8; i += blockDim.x / 32) {
    const float4 m = __ldg(reinterpret_cast<const float4*>(p.k.mu + (size_t)h * kHeadDim) + lane);
    const float4 qq = *reinterpret_cast<const float4*>(q_s + i * kHeadDim + 4 * lane);
    float sm = fmaf(qq.x, m.x, fmaf(qq.y, m.y, fmaf(qq.z, m.z, qq.w * m.w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    if (lane == 0) cqs[i] = sm;
  }
  __syncthreads();
}

constexpr int kSvdqTile = 128;                           // tokens per tile: one 32-token block per warp
constexpr int kSvdqTileBytes = kSvdqTile * kHeadDim * 2;  // 32 KB of values
constexpr int kSvdqStages = 2;
constexpr int kSvdqRecSlack = 1024;  // bytes past the last staged record (see svdq_codes_frag)
static_assert(sizeof(float) * kSplitWarps * 8 * kSplitPartStride <= kSvdqTileBytes,
              "the end-of-chunk merge scratch fits in one value stage");
struct SvdqDecSmem {
  int vst, kst, qts, total;
};
__host__ __device__ inline SvdqDecSmem svdq_dec_smem(int r_max, int rec_bytes) {
  SvdqDecSmem s;
  s.vst = 0;                                                            // V tiles [stages][128][D] fp16, swizzled
  s.kst = s.vst + kSvdqStages * kSvdqTileBytes;                         // key records [stages][4][rec] + slack
  s.qts = s.kst + svdq_a16(kSvdqStages * 4 * rec_bytes + kSvdqRecSlack);  // q~ [8][r_max] and c [8]
  s.total = s.qts + svdq_a16(4 * (8 * r_max + 8));
  return s;
}

// The A fragment of one k-step (16 channels of one width W, tokens of one
// 16-row slice of a block) as exact fp16 codes.  The k-step's channel k holds
// its 32 codes in W words, token t at bit t*W; lane (g, c) needs channels 2c,
// 2c+1 (registers 0, 1) and 2c+8, 2c+9 (registers 2, 3) of tokens tb0 (16h+g)
// and tb0 + 8.  A byte permute gathers the two channels' bytes that hold a
// token's code into the low bytes of the two halves; the lane's bit mask
// keeps the code, ORed into the fp16 pattern of 1024 (code at mantissa bit
// o); one fp16x2 FMA by 2^-o with addend -1024 * 2^-o gives the code itself
// (every step exact).  cw: the words of channel 2c of the k-step.  Lanes
// whose channels lie past the class read codes of later channels or of the
// next record (finite, and multiplied by a zero B operand).
template <int W>
__device__ __forceinline__ void svdq_codes_frag(const uint32_t* cw, int tb0, uint32_t a[4]) {
  const int pos0 = tb0 * W, pos1 = pos0 + 8 * W;
  const int wi0 = pos0 >> 5, wi1 = pos1 >> 5;
  const uint32_t bs0 = (uint32_t)(pos0 & 31) >> 3, bs1 = (uint32_t)(pos1 & 31) >> 3;
  const int o = pos0 & 7;
  const uint32_t sel0 = bs0 | ((bs0 + 4u) << 8), sel1 = bs1 | ((bs1 + 4u) << 8);
  const uint32_t m = ((1u << W) - 1u) << o, M = m | (m << 16);
  const uint32_t mul = (uint32_t)(15 - o) << 10, add = 0x8000u | ((uint32_t)(25 - o) << 10);
  const uint32_t mul2 = mul | (mul << 16), add2 = add | (add << 16);
  a[0] = __byte_perm(cw[wi0], cw[W + wi0], sel0);
  a[1] = __byte_perm(cw[wi1], cw[W + wi1], sel1);
  a[2] = __byte_perm(cw[8 * W + wi0], cw[9 * W + wi0], sel0);
  a[3] = __byte_perm(cw[8 * W + wi1], cw[9 * W + wi1], sel1);
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = fma_f16x2((a[i] & M) | 0x64006400u, mul2, add2);
}

__device__ __forceinline__ float pow2f_(int e) { return __int_as_float((e + 127) << 23); }

// Channel offset of lane c's k-th channel (k = 0..3) within a 16-channel
// k-step: 2c, 2c+1, 2c+8, 2c+9.
__device__ __forceinline__ int svdq_kk(int k) { return (k & 1) + ((k >> 1) << 3); }

// grid (chunks, kv_heads, batch), 4 warps: each CTA a contiguous chunk of
// 128-token tiles of one stream.  Per tile: the value rows and the key
// records by cp.async into a 2-stage ring; warp w takes the tile's block w
// (32 tokens, two 16-row slices).  Scores of a quantized block on the tensor
// cores:
//   q~ . L_t + c = sum_j code_tj (q~_j s_j) + (c + sum_j q~_j z_j)
// with the codes as exact fp16 A operands (one k-step per width class of
// the schedule: 8, 4, 2 bits, then the 1-bit channels in one or two steps)
// and q~_j s_j as an fp16 hi + lo B pair prescaled by a power of two (the
// block's largest |q~_j s_j| near 2^14), fp32 accumulation; the partial
// block's tokens from their fp32 latents on the CUDA cores.  Then the online
// softmax and the weighted sum of the value rows on the tensor cores (the
// comparator's loop), slice by slice.
__global__ void __launch_bounds__(32 * kSplitWarps) svdq_decode_kernel(const SvdqDecParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int H = p.k.H, rm = p.k.r_max, Gq = p.Gq, rb = p.k.rec_bytes;
  const long long X = (long long)b * H + h;
  const int r = p.k.head[4 * h], szo = p.k.head[4 * h + 2];
  const SvdqDecSmem L = svdq_dec_smem(rm, rb);
  float* qts = reinterpret_cast<float*>(dsm + L.qts);
  float* cqs = qts + 8 * rm;
  const long long t0 = (long long)chunk * p.tiles_per_chunk * kSvdqTile;
  const long long t1 = min(t0 + (long long)p.tiles_per_chunk * kSvdqTile, p.len);
  float* part = p.ws + ((long long)X * p.n_chunks + chunk) * (long long)Gq * kSplitPartStride;
  if (t0 >= t1) {
    split_write_empty(Gq, part);
    return;
  }
  const int n_tiles = (int)((t1 - t0 + kSvdqTile - 1) / kSvdqTile);
  const long long nf = p.len / kBlock;  // full (quantized) blocks
  const uint8_t* kb = p.k.blocks + X * p.k.n_blk_cap * rb;
  const float* tail = p.k.tail + X * kBlock * rm;
  const uint32_t sbase = smem_addr(dsm);

  grid_dep_launch();  // the combine kernel may be scheduled; it waits for this grid

  // the head's width classes: group sizes r/8 (+1 for the first r%8 groups)
  const int n8 = r / 8 + (0 < r % 8), n4 = r / 8 + (1 < r % 8), n2 = r / 8 + (2 < r % 8);
  const int n1 = 2 * (r / 8) + (3 < r % 8) + (4 < r % 8);
  const int ksn[5] = {n8, n4, n2, min(n1, 16), max(n1 - 16, 0)};
  const int ksf[5] = {0, n8, n8 + n4, n8 + n4 + n2, n8 + n4 + n2 + 16};
  const int ksb[5] = {0, 32 * n8, 32 * n8 + 16 * n4, 32 * n8 + 16 * n4 + 8 * n2, 32 * n8 + 16 * n4 + 8 * n2 + 64};
  // this thread's cp.async slots: value rows (tid >> 4) + 8i, chunk tid & 15;
  // record chunks tid and tid + 128 of the tile's four records
  const int vrow = tid >> 4, vch = tid & 15;
  const char* vsrc = reinterpret_cast<const char*>(p.v + (X * p.v_cap + t0 + vrow) * kHeadDim + vch * 8);
  const char* vfall = reinterpret_cast<const char*>(p.v + (X * p.v_cap + t0) * kHeadDim);  // a row below len
  const uint32_t vdst = swz(sbase + L.vst, vrow, vch);
  const int rq = rb / 16;
  const int kbi0 = tid / rq, kq0 = tid % rq, kbi1 = (tid + 128) / rq, kq1 = (tid + 128) % rq;
  auto load_tile = [&](int tile, int stage) {
    const long long tt = t0 + (long long)tile * kSvdqTile;
    const char* src = vsrc + (long long)tile * kSvdqTileBytes;
    const uint32_t dst = vdst + stage * kSvdqTileBytes;
    if (tt + kSvdqTile <= t1) {
#pragma unroll
      for (int i = 0; i < kSvdqTile / 8; ++i)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + i * 8 * 256), "l"(src + i * 8 * 256)
                     : "memory");
    } else {
#pragma unroll
      for (int i = 0; i < kSvdqTile / 8; ++i) {
        const bool valid = tt + vrow + 8 * i < t1;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst + i * 8 * 256),
                     "l"(valid ? src + i * 8 * 256 : vfall), "r"(valid ? 16 : 0)
                     : "memory");
      }
    }
    // the key records of the tile's four blocks that are quantized
    const long long blk0 = tt / kBlock;
    const uint32_t kdst = sbase + L.kst + stage * 4 * rb;
    if (kbi0 < 4 && blk0 + kbi0 < nf)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(kdst + kbi0 * rb + 16 * kq0),
                   "l"(kb + (blk0 + kbi0) * rb + 16 * kq0)
                   : "memory");
    if (kbi1 < 4 && blk0 + kbi1 < nf)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(kdst + kbi1 * rb + 16 * kq1),
                   "l"(kb + (blk0 + kbi1) * rb + 16 * kq1)
                   : "memory");
    for (int i = tid + 256; i < 4 * rq; i += blockDim.x) {  // records over 512 bytes
      const int bi = i / rq, q = i % rq;
      if (blk0 + bi < nf)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(kdst + bi * rb + 16 * q),
                     "l"(kb + (blk0 + bi) * rb + 16 * q)
                     : "memory");
    }
  };

#pragma unroll
  for (int s = 0; s < kSvdqStages - 1; ++s) {
    if (s < n_tiles) load_tile(s, s);
    cp_async_commit();
  }
  // the stream's query factors while the first copies are in flight (every
  // CTA of the stream forms them; scratch: the second value stage, whose
  // first copy is issued only after the loop's first barrier)
  static_assert(kSvdqStages >= 2, "the query scratch uses the second value stage");
  svdq_query_factors(p, h, b, reinterpret_cast<float*>(dsm + L.vst + kSvdqTileBytes), qts, cqs);
  // lane's q~ of head g at its channels of each k-step (0 past the class)
  float qv[5][4];
#pragma unroll
  for (int ks = 0; ks < 5; ++ks)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int jj = 2 * c + svdq_kk(k);
      qv[ks][k] = jj < ksn[ks] ? qts[g * rm + ksf[ks] + jj] : 0.f;
    }
  const float cq_g = cqs[g];
  SplitState st;
  split_init(st);
  for (int tile = 0; tile < n_tiles; ++tile) {
    cp_async_wait<kSvdqStages - 2>();
    __syncthreads();
    const int nxt = tile + kSvdqStages - 1;
    if (nxt < n_tiles) load_tile(nxt, nxt % kSvdqStages);
    cp_async_commit();
    const int stage = tile % kSvdqStages;
    const long long tt = t0 + (long long)tile * kSvdqTile;
    const uint32_t vst = sbase + L.vst + stage * kSvdqTileBytes;
    const long long blk = tt / kBlock + warp;
    if (blk < nf) {
      // quantized block: B = q~_j s_j (hi + lo) once, then both slices
      const uint8_t* rec = dsm + L.kst + (stage * 4 + warp) * rb;
      const __half2* szr = reinterpret_cast<const __half2*>(rec + szo);
      float av[5][4];
      float mx = 0.f, cst = 0.f;
#pragma unroll
      for (int ks = 0; ks < 5; ++ks)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int jj = 2 * c + svdq_kk(k);
          float2 sz = make_float2(0.f, 0.f);
          if (jj < ksn[ks]) sz = __half22float2(szr[ksf[ks] + jj]);
          av[ks][k] = qv[ks][k] * sz.x;
          cst = fmaf(qv[ks][k], sz.y, cst);
          mx = fmaxf(mx, fabsf(av[ks][k]));
        }
#pragma unroll
      for (int x = 1; x < 4; x <<= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, x));
        cst += __shfl_xor_sync(0xffffffffu, cst, x);
      }
      const int e = min(141 - (int)((__float_as_uint(mx) >> 23) & 0xffu), 126);  // max|B| in [2^14, 2^15)
      const float S = pow2f_(e), invS = pow2f_(-e);
      uint32_t bh[5][2], bl[5][2];
#pragma unroll
      for (int ks = 0; ks < 5; ++ks) {
        const float x0 = av[ks][0] * S, x1 = av[ks][1] * S, x8 = av[ks][2] * S, x9 = av[ks][3] * S;
        bh[ks][0] = pack_f16x2(x0, x1);
        bh[ks][1] = pack_f16x2(x8, x9);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&bh[ks][0]));
        const float2 f89 = __half22float2(*reinterpret_cast<const __half2*>(&bh[ks][1]));
        bl[ks][0] = pack_f16x2(x0 - f01.x, x1 - f01.y);
        bl[ks][1] = pack_f16x2(x8 - f89.x, x9 - f89.y);
      }
      // heads 2c, 2c+1: their scale and constant from lanes 8c and 8c+4
      const float cfull = cst + cq_g;
      const float iA = __shfl_sync(0xffffffffu, invS, 8 * c) * p.scale_log2;
      const float iB = __shfl_sync(0xffffffffu, invS, 8 * c + 4) * p.scale_log2;
      const float cA = __shfl_sync(0xffffffffu, cfull, 8 * c) * p.scale_log2;
      const float cB = __shfl_sync(0xffffffffu, cfull, 8 * c + 4) * p.scale_log2;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int tb0 = 16 * half + g;
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 5; ++ks) {
          if (ksn[ks] == 0) continue;  // uniform
          uint32_t a[4];
          if (ks == 0) svdq_codes_frag<8>(reinterpret_cast<const uint32_t*>(rec + ksb[0]) + 16 * c, tb0, a);
          else if (ks == 1) svdq_codes_frag<4>(reinterpret_cast<const uint32_t*>(rec + ksb[1]) + 8 * c, tb0, a);
          else if (ks == 2) svdq_codes_frag<2>(reinterpret_cast<const uint32_t*>(rec + ksb[2]) + 4 * c, tb0, a);
          else svdq_codes_frag<1>(reinterpret_cast<const uint32_t*>(rec + ksb[ks]) + 2 * c, tb0, a);
          mma_f16(sc, a[0], a[1], a[2], a[3], bh[ks][0], bh[ks][1]);
          mma_f16(sc, a[0], a[1], a[2], a[3], bl[ks][0], bl[ks][1]);
        }
        // every token of a quantized block precedes the chunk's end
        sc[0] = fmaf(sc[0], iA, cA);
        sc[1] = fmaf(sc[1], iB, cB);
        sc[2] = fmaf(sc[2], iA, cA);
        sc[3] = fmaf(sc[3], iB, cB);
        split_softmax_pv(st, sc, vst, 32 * warp + 16 * half, lane);
      }
    } else {
      // the partial block (or past the end): fp32 latents
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const long long ta = tt + 32 * warp + 16 * half + g, tb = ta + 8;
        const bool va = ta < t1, vbv = tb < t1;
        float sc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (__any_sync(0xffffffffu, va)) {
          const float* la = tail + (va ? (ta % kBlock) : 0) * rm;
          const float* lb = tail + (vbv ? (tb % kBlock) : 0) * rm;
          const float* qa = qts + (2 * c) * rm;
          const float* qb = qa + rm;
          float s00 = cqs[2 * c], s01 = cqs[2 * c + 1], s10 = s00, s11 = s01;
          for (int j = 0; j < r; ++j) {
            const float x = __ldcg(la + j), y = __ldcg(lb + j), u = qa[j], w = qb[j];
            s00 = fmaf(u, x, s00);
            s01 = fmaf(w, x, s01);
            s10 = fmaf(u, y, s10);
            s11 = fmaf(w, y, s11);
          }
          sc[0] = va ? s00 * p.scale_log2 : -INFINITY;
          sc[1] = va ? s01 * p.scale_log2 : -INFINITY;
          sc[2] = vbv ? s10 * p.scale_log2 : -INFINITY;
          sc[3] = vbv ? s11 * p.scale_log2 : -INFINITY;
        }
        split_softmax_pv(st, sc, vst, 32 * warp + 16 * half, lane);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // the merge scratch reuses the value ring
  split_write_partial(st, reinterpret_cast<float(*)[8][kSplitPartStride]>(dsm + L.vst), warp, lane, Gq, part);
}

static int svdq_chunks(int64_t streams, int64_t seq, int smem, int* tiles_per_chunk) {
  int per_sm = 1;
  kernel_occupancy(reinterpret_cast<const void*>(svdq_decode_kernel), 32 * kSplitWarps, smem, &per_sm);
  const int64_t tiles = std::max<int64_t>(1, (seq + kSvdqTile - 1) / kSvdqTile);
  int64_t nch = std::max<int64_t>(1, (int64_t)device_sm_count() * per_sm / streams);
  nch = std::min(nch, tiles);
  const int64_t tpc = (tiles + nch - 1) / nch;
  *tiles_per_chunk = (int)tpc;
  return (int)((tiles + tpc - 1) / tpc);
}

static palu_status check_svdq(const palu_svdq_cache* c) {
  if (!c) return fail(PALU_ERR_INVALID_ARG, "cache is NULL");
  if (c->magic != kSvdqMagic) return fail(PALU_ERR_NOT_INITIALIZED, "the SVDq cache is not initialised");
  return PALU_OK;
}

static palu_status svdq_geometry(int32_t kv_heads, const int32_t* ranks, int* r_max, int* rec_bytes) {
  if (!ranks) return fail(PALU_ERR_INVALID_ARG, "ranks is NULL");
  *r_max = 0;
  *rec_bytes = 16;
  std::vector<int> offs, bits;
  for (int h = 0; h < kv_heads; ++h) {
    if (ranks[h] < 1 || ranks[h] > kMaxRank) return fail(PALU_ERR_INVALID_ARG, "every rank must be in [1, 128]");
    int kept, szo;
    *r_max = std::max(*r_max, (int)ranks[h]);
    *rec_bytes = std::max(*rec_bytes, svdq_record(ranks[h], offs, bits, &kept, &szo));
  }
  return PALU_OK;
}

}  // namespace palu

using namespace palu;

extern "C" palu_status palu_svdq_cache_size(int64_t batch, int32_t kv_heads, const int32_t* ranks, int64_t capacity,
                                            size_t* block_bytes, size_t* tail_bytes, size_t* state_bytes) {
  if (batch < 1 || kv_heads < 1 || capacity < 1) return fail(PALU_ERR_INVALID_ARG, "batch, kv_heads, capacity must be >= 1");
  if (batch * (int64_t)kv_heads > 65535LL * 64) return fail(PALU_ERR_UNSUPPORTED, "batch*kv_heads too large");
  int r_max, rb;
  palu_status st = svdq_geometry(kv_heads, ranks, &r_max, &rb);
  if (st != PALU_OK) return st;
  const int64_t n_blk = (capacity + kBlock - 1) / kBlock;
  if (block_bytes) *block_bytes = align_up((size_t)batch * kv_heads * n_blk * rb, 256);
  if (tail_bytes) *tail_bytes = align_up(sizeof(float) * (size_t)batch * kv_heads * kBlock * r_max, 256);
  if (state_bytes) *state_bytes = svdq_layout(kv_heads, r_max).total;
  return PALU_OK;
}

extern "C" palu_status palu_svdq_cache_init(palu_svdq_cache* cache, int64_t batch, int32_t kv_heads,
                                            const int32_t* ranks, int64_t capacity, const float* basis,
                                            int32_t basis_ld, const float* mu, void* blocks, void* tail, void* state,
                                            void* stream) {
  if (!cache) return fail(PALU_ERR_INVALID_ARG, "cache is NULL");
  size_t bb, tb, sb;
  palu_status st = palu_svdq_cache_size(batch, kv_heads, ranks, capacity, &bb, &tb, &sb);
  if (st != PALU_OK) return st;
  if (!basis || !mu || !blocks || !tail || !state) return fail(PALU_ERR_INVALID_ARG, "NULL buffer");
  if (((uintptr_t)blocks | (uintptr_t)tail | (uintptr_t)state) & 255)
    return fail(PALU_ERR_INVALID_ARG, "blocks, tail and state must be 256-byte aligned");
  int r_max, rb;
  svdq_geometry(kv_heads, ranks, &r_max, &rb);
  if (basis_ld < r_max) return fail(PALU_ERR_INVALID_ARG, "basis_ld must be >= the largest rank");
  palu_svdq_cache c;
  std::memset(&c, 0, sizeof(c));
  c.magic = kSvdqMagic;
  c.batch = (int32_t)batch;
  c.kv_heads = kv_heads;
  c.r_max = r_max;
  c.record_bytes = rb;
  c.capacity = capacity;
  c.n_blk_cap = (capacity + kBlock - 1) / kBlock;
  c.blocks = blocks;
  c.tail = static_cast<float*>(tail);
  c.state = state;
  c.length = 0;
  // per-head tables on the host, then copied
  const SvdqLayout sl = svdq_layout(kv_heads, r_max);
  std::vector<uint8_t> host(sl.basis_off, 0);
  int* head = reinterpret_cast<int*>(host.data() + sl.head_off);
  int* coff = reinterpret_cast<int*>(host.data() + sl.coff_off);
  int* cbits = reinterpret_cast<int*>(host.data() + sl.bits_off);
  std::vector<int> offs, bits;
  for (int h = 0; h < kv_heads; ++h) {
    int kept, szo;
    const int rbh = svdq_record(ranks[h], offs, bits, &kept, &szo);
    head[4 * h] = ranks[h];
    head[4 * h + 1] = kept;
    head[4 * h + 2] = szo;
    head[4 * h + 3] = rbh;
    for (int j = 0; j < ranks[h]; ++j) {
      coff[h * r_max + j] = offs[j];
      cbits[h * r_max + j] = bits[j];
    }
  }
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  uint8_t* s = static_cast<uint8_t*>(state);
  st = cuda_check(cudaMemsetAsync(s, 0, sl.total, strm), "cudaMemsetAsync(SVDq state)");
  if (st != PALU_OK) return st;
  st = cuda_check(cudaMemcpyAsync(s + sl.head_off, host.data() + sl.head_off, sl.basis_off - sl.head_off,
                                  cudaMemcpyHostToDevice, strm),
                  "copy SVDq tables");
  if (st != PALU_OK) return st;
  st = cuda_check(cudaStreamSynchronize(strm), "cudaStreamSynchronize");  // the host tables are pageable
  if (st != PALU_OK) return st;
  const SvdqView v = svdq_view(&c);
  svdq_init_kernel<<<dim3(r_max, kv_heads), kHeadDim, 0, strm>>>(basis, basis_ld, mu, v,
                                                                  reinterpret_cast<const int*>(s + sl.head_off));
  st = cuda_check(cudaGetLastError(), "svdq_init_kernel launch");
  if (st != PALU_OK) return st;
  *cache = c;
  return PALU_OK;
}

extern "C" palu_status palu_svdq_append(palu_svdq_cache* cache, const void* k, int64_t tokens, void* stream) {
  palu_status st = check_svdq(cache);
  if (st != PALU_OK) return st;
  if (tokens < 0) return fail(PALU_ERR_INVALID_ARG, "tokens must be >= 0");
  if (tokens == 0) return PALU_OK;
  if (!k || ((uintptr_t)k & 15)) return fail(PALU_ERR_INVALID_ARG, "k must be a non-NULL, 16-byte aligned device pointer");
  if (cache->length + tokens > cache->capacity)
    return fail(PALU_ERR_CAPACITY, "append of " + std::to_string(tokens) + " tokens to an SVDq cache holding " +
                                       std::to_string(cache->length) + " exceeds its capacity " +
                                       std::to_string(cache->capacity));
  const int64_t nblk = (tokens + kBlock - 1) / kBlock + 1;
  if (nblk > 2147483647LL) return fail(PALU_ERR_UNSUPPORTED, "too many tokens in one append");
  const int smem = svdq_enc_smem(cache->r_max, cache->record_bytes).total;
  int per_sm = 0;
  st = kernel_occupancy(reinterpret_cast<const void*>(svdq_encode_kernel), 128, smem, &per_sm);
  if (st != PALU_OK) return st;
  const SvdqView v = svdq_view(cache);
  for (int phase = 1; phase <= 2; ++phase) {
    svdq_encode_kernel<<<dim3(phase == 1 ? (unsigned)nblk : 1u, cache->kv_heads, cache->batch), 128, smem,
                         static_cast<cudaStream_t>(stream)>>>(v, static_cast<const __half*>(k), tokens, phase);
    st = cuda_check(cudaGetLastError(), "svdq_encode_kernel launch");
    if (st != PALU_OK) return st;
  }
  cache->length += tokens;
  return PALU_OK;
}

namespace palu {
struct SvdqWs {
  size_t part_off, total;
  int n_chunks, tpc, smem;
};
static palu_status svdq_ws(const palu_svdq_cache* c, int32_t q_heads, SvdqWs* w) {
  if (q_heads < 1 || q_heads % c->kv_heads) return fail(PALU_ERR_INVALID_ARG, "q_heads must be a multiple of kv_heads");
  const int Gq = q_heads / c->kv_heads;
  if (Gq > kMaxGq) return fail(PALU_ERR_UNSUPPORTED, "at most 8 query heads per KV head");
  const int64_t streams = (int64_t)c->batch * c->kv_heads;
  w->smem = svdq_dec_smem(c->r_max, c->record_bytes).total;
  w->n_chunks = svdq_chunks(streams, c->capacity, w->smem, &w->tpc);
  w->part_off = 0;
  w->total = align_up(sizeof(float) * (size_t)streams * w->n_chunks * Gq * kSplitPartStride, 256);
  return PALU_OK;
}
}  // namespace palu

extern "C" palu_status palu_svdq_decode_workspace_size(const palu_svdq_cache* cache, int32_t q_heads, size_t* bytes) {
  palu_status st = check_svdq(cache);
  if (st != PALU_OK) return st;
  if (!bytes) return fail(PALU_ERR_INVALID_ARG, "bytes is NULL");
  SvdqWs w;
  st = svdq_ws(cache, q_heads, &w);
  if (st != PALU_OK) return st;
  *bytes = w.total;
  return PALU_OK;
}

extern "C" palu_status palu_svdq_decode_attn(const palu_svdq_cache* cache, const void* v, int64_t v_cap, const void* q,
                                             int32_t q_heads, float softmax_scale, void* out, int32_t out_fp32,
                                             void* workspace, size_t workspace_bytes, void* stream) {
  palu_status st = check_svdq(cache);
  if (st != PALU_OK) return st;
  SvdqWs w;
  st = svdq_ws(cache, q_heads, &w);
  if (st != PALU_OK) return st;
  if (cache->length < 1) return fail(PALU_ERR_INVALID_ARG, "the SVDq cache is empty");
  if (v_cap < cache->length) return fail(PALU_ERR_INVALID_ARG, "v_cap must be >= the cache length");
  if (!v || !q || !out || !workspace) return fail(PALU_ERR_INVALID_ARG, "NULL pointer");
  if (((uintptr_t)v | (uintptr_t)q | (uintptr_t)out | (uintptr_t)workspace) & 15)
    return fail(PALU_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  if (workspace_bytes < w.total)
    return fail(PALU_ERR_INVALID_ARG, "workspace too small: need " + std::to_string(w.total) + " bytes");
  SvdqDecParams p;
  p.k = svdq_view(cache);
  p.v = static_cast<const __half*>(v);
  p.q = static_cast<const __half*>(q);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.ws = reinterpret_cast<float*>(ws + w.part_off);
  p.v_cap = v_cap;
  p.len = cache->length;
  p.Hq = q_heads;
  p.Gq = q_heads / cache->kv_heads;
  p.n_chunks = w.n_chunks;
  p.tiles_per_chunk = w.tpc;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)kHeadDim);
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  // in stream order (it reads what earlier launches wrote); the combine
  // kernel follows as its programmatic dependent
  svdq_decode_kernel<<<dim3(p.n_chunks, cache->kv_heads, (unsigned)cache->batch), 32 * kSplitWarps, w.smem, strm>>>(p);
  st = cuda_check(cudaGetLastError(), "svdq_decode_kernel launch");
  if (st != PALU_OK) return st;
  return split_combine(p.ws, cache->batch, q_heads, cache->kv_heads, p.n_chunks, out, out_fp32, strm);
}

extern "C" palu_status palu_svdq_sync(palu_svdq_cache* cache, uint32_t* device_error, void* stream) {
  palu_status st = check_svdq(cache);
  if (st != PALU_OK) return st;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  st = cuda_check(cudaStreamSynchronize(strm), "cudaStreamSynchronize");
  if (st != PALU_OK) return st;
  SvdqHeader h;
  st = cuda_check(cudaMemcpy(&h, cache->state, sizeof(h), cudaMemcpyDeviceToHost), "read SVDq state");
  if (st != PALU_OK) return st;
  cache->length = h.length;
  if (device_error) *device_error = h.err;
  if (h.err) {
    const unsigned int zero = 0;
    cudaMemcpy(static_cast<uint8_t*>(cache->state) + offsetof(SvdqHeader, err), &zero, sizeof(zero),
               cudaMemcpyHostToDevice);
    return fail(PALU_ERR_DEVICE, "SVDq device error word " + std::to_string(h.err));
  }
  return PALU_OK;
}
