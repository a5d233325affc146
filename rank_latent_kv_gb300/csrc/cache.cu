// Cache set-up and the encode/append kernel.
//
// Method (page "PALU — True Low-Rank Latent Storage for Keys and Values",
// "How it works"): prefill steps 4-5 and decode steps 1-2 -- project new
// tokens into the stored group basis, L = (x - mu_g) V_g, then mixed-bit
// quantize per (channel, 32-token group) with the asymmetric min/max
// quantizer (blog post "VeloxQuant-MLX 0.8.0 adds KIVI", "What KIVI is") and
// pack the codes LSB-first (blog post "How I built VeloxQuant-MLX", "The
// Bit-Packing Problem").
//
// The stored latents, scales, zeros and codes are those of the fp32 latents
// rounded once from an error-free (float-pair) dot product.  Complete blocks
// of quantized caches are projected on the tensor cores under a rigorous
// error bound, and the exact latent is formed only where a stored value
// depends on it; every other latent takes the float-pair path directly.
#include <math.h>

#include <algorithm>
#include <cstring>

#include "append_one.cuh"

namespace palu {

// ------------------------------------------------------------------ init
// One CTA per (group, direction j): copies column j of the caller's basis to
// row j of basisT, and forms mu_g . V_g[:, j] in fp64, stored as a float pair.
__global__ void cache_init_kernel(const float* __restrict__ basis, int ld, const float* __restrict__ mu,
                                  float* basisT, float* mu_out, float2* mv, StateHeader* hdr, int r) {
  const int g = blockIdx.y, j = blockIdx.x, d = threadIdx.x;
  __shared__ double red[kHeadDim];
  const float vj = basis[((size_t)g * kHeadDim + d) * ld + j];
  basisT[((size_t)g * r + j) * kHeadDim + d] = vj;
  const float m = mu[(size_t)g * kHeadDim + d];
  if (j == 0) mu_out[(size_t)g * kHeadDim + d] = m;
  red[d] = (double)m * (double)vj;
  __syncthreads();
  for (int s = kHeadDim / 2; s > 0; s >>= 1) {
    if (d < s) red[d] += red[d + s];
    __syncthreads();
  }
  if (d == 0) {
    const double t = red[0];
    const float hi = (float)t;
    mv[(size_t)g * r + j] = make_float2(hi, (float)(t - (double)hi));
  }
  if (g == 0 && j == 0 && d == 0) {
    hdr->length = 0;
    hdr->err = 0;
    hdr->ticket = 0;
    hdr->max_scale = 0;
    hdr->ragged = 0;
  }
}

// ------------------------------------------------------------------ encode
// Shared-memory plan of one encode CTA (one 32-token block of one stream).
// The staged basis comes last: the tensor-core path (every phase-1 CTA of a
// quantized cache) reads the basis from global memory and is launched
// without it.
struct EncodeSmem {
  int xs_off, lat_off, err_off, codes_off, sz_off, rec_off, work_off, basis_off, total;
};

__host__ __device__ inline int align16(int x) { return (x + 15) / 16 * 16; }

constexpr int kXsStride = kHeadDim + 8;  // halves per staged row: 272 B, so ldmatrix rows hit distinct banks

__host__ __device__ inline EncodeSmem encode_smem(int r, int rec_bytes) {
  EncodeSmem s;
  s.xs_off = 0;                                                        // half [32][136]
  s.lat_off = s.xs_off + kBlock * kXsStride * 2;                       // float [32][r+1]
  s.err_off = s.lat_off + align16(4 * kBlock * (r + 1));               // float [32][r+1]: bound of |L' - L|
  s.codes_off = s.err_off + align16(4 * kBlock * (r + 1));             // u8 [32][r]
  s.sz_off = s.codes_off + align16(kBlock * r);                        // half2 [r] (scale, zero)
  s.rec_off = s.sz_off + align16(4 * r);                               // record
  s.work_off = s.rec_off + align16(rec_bytes);                         // int [2] counts, u32 [4] warp maxima,
                                                                       // u16 [32 r] work list
  s.basis_off = s.work_off + align16(24 + 2 * kBlock * r);             // float [r][129] (exact path only)
  s.total = s.basis_off + align16(4 * r * (kHeadDim + 1));
  return s;
}

// One latent (x - mu_g) V_g[:, j] as the encoder stores it: sum_d x_d V_dj
// accumulated in order d = 0..127 as an unevaluated float pair (error-free
// products and sums), minus mu_g . V_g[:, j] (a float pair), rounded once to
// fp32.  Every exact latent of the encoder goes through this sequence, so
// the two projection paths below store identical values.
__device__ __forceinline__ void fp_acc(float& S, float& E, float xv, float v) {
  float pp, pe, s2, se;
  two_prod(xv, v, pp, pe);
  two_sum(S, pp, s2, se);
  S = s2;
  E = __fadd_rn(E, __fadd_rn(se, pe));
}
__device__ __forceinline__ float fp_finish(float S, float E, float2 m) {
  float a, ae;
  two_sum(S, -m.x, a, ae);
  const float low = __fadd_rn(__fsub_rn(E, m.y), ae);
  return __fadd_rn(a, low);
}
// Two fp32 lanes in one 64-bit register: the packed f32x2 arithmetic of
// this architecture (each element rounded to nearest, as the scalar forms).
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(f32x2 r, float& a, float& b) { asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r)); }
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// fp_acc on two float pairs at once, with the product carried negated
// (np = -x v): the same roundings as fp_acc element by element.
__device__ __forceinline__ void fp_acc2(f32x2& S, f32x2& E, f32x2 x, f32x2 v) {
  const f32x2 np = mul2(sub2(0ull, x), v);          // -p
  const f32x2 pe = fma2(x, v, np);                  // x v - p
  const f32x2 s2 = sub2(S, np);                     // S + p
  const f32x2 bb = sub2(s2, S);
  const f32x2 se = sub2(sub2(S, sub2(s2, bb)), add2(np, bb));  // (S - (s2 - bb)) + (p - bb)
  E = add2(E, add2(se, pe));
  S = s2;
}
// The same sum with four interleaved float pairs (d mod 4) merged by
// error-free sums at the end: about 48 significant bits like the sequential
// pair, so its fp32 rounding is the same except when the sum lies within
// about 2^-48 of a rounding boundary; a quarter of the dependent chain.  The
// four pairs advance two at a time in packed registers.
__device__ __noinline__ float exact_latent(const __half* xrow, const float* __restrict__ brow, float2 m) {
  f32x2 S01 = 0ull, E01 = 0ull, S23 = 0ull, E23 = 0ull;
#pragma unroll 8  // (eight rows' loads in flight: measured 2.75 -> 2.68 ms per layer against unroll 2)
  for (int d = 0; d < kHeadDim; d += 4) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(brow + d));
    const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(xrow + d));
    const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(xrow + d + 2));
    fp_acc2(S01, E01, pk2(x01.x, x01.y), pk2(v.x, v.y));
    fp_acc2(S23, E23, pk2(x23.x, x23.y), pk2(v.z, v.w));
  }
  float S[4], E[4];
  upk2(S01, S[0], S[1]);
  upk2(S23, S[2], S[3]);
  upk2(E01, E[0], E[1]);
  upk2(E23, E[2], E[3]);
  float s01, e01, s23, e23, s, e;
  two_sum(S[0], S[1], s01, e01);
  two_sum(S[2], S[3], s23, e23);
  two_sum(s01, s23, s, e);
  const float lo = __fadd_rn(__fadd_rn(__fadd_rn(E[0], E[1]), __fadd_rn(E[2], E[3])), __fadd_rn(__fadd_rn(e01, e23), e));
  return fp_finish(s, lo, m);
}

// The same latent computed by a whole warp (every lane calls): lane l takes
// terms 4l..4l+3 as a float pair, then the pairs merge over a butterfly of
// error-free sums (symmetric, so every lane ends with the same value).
__device__ __noinline__ float exact_latent_warp(const __half* xrow, const float* __restrict__ brow, float2 m,
                                                int lane) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(brow) + lane);
  const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(xrow + 4 * lane));
  const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(xrow + 4 * lane + 2));
  float S = 0.f, E = 0.f;
  fp_acc(S, E, x01.x, v.x);
  fp_acc(S, E, x01.y, v.y);
  fp_acc(S, E, x23.x, v.z);
  fp_acc(S, E, x23.y, v.w);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float S2 = __shfl_xor_sync(0xffffffffu, S, o), E2 = __shfl_xor_sync(0xffffffffu, E, o);
    float s, e;
    two_sum(S, S2, s, e);
    S = s;
    E = __fadd_rn(__fadd_rn(E, E2), e);
  }
  return fp_finish(S, E, m);
}

// f(t, j, L) for every (token, channel) entry of a work list of n, with L
// the entry's exact latent.  Whole warps of entries go one per lane; a short
// remainder (below 13 entries a warp per entry takes fewer instructions than
// one more pass of lanes) goes one entry per warp, starting with the warps
// that have no lane work.
template <class F>
__device__ __forceinline__ void run_exact(const uint16_t* work, int n, const __half* xs, const float* __restrict__ bT,
                                          const float2* __restrict__ mv, F&& f) {
  const int tid = threadIdx.x, nw = blockDim.x >> 5, warp = tid >> 5, lane = tid & 31;
  const int rem = (n & 31) < 13 ? (n & 31) : 0, full = n - rem;
  for (int i = tid; i < full; i += blockDim.x) {
    const int t = work[i] >> 7, j = work[i] & 127;
    f(t, j, exact_latent(xs + t * kXsStride, bT + (size_t)j * kHeadDim, mv[j]));
  }
  const int w0 = ((full + 31) >> 5) % nw;
  for (int k = (warp - w0 + nw) % nw; k < rem; k += nw) {
    const int t = work[full + k] >> 7, j = work[full + k] & 127;
    const float L = exact_latent_warp(xs + t * kXsStride, bT + (size_t)j * kHeadDim, mv[j], lane);
    if (lane == 0) f(t, j, L);
  }
}

// A float's bits mapped to an unsigned key of the same order (sign bit set
// for non-negative values, all bits inverted for negative ones; -0 below +0),
// and back: exact minima and maxima by integer comparisons.
__device__ __forceinline__ unsigned int f2key(float f) {
  const unsigned int b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key2f(unsigned int k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Append (t, j) for every set bit t of `bits` to a shared work list: one
// counter reservation per warp (every lane calls), a lane's entries together.
__device__ __forceinline__ void push_work(uint16_t* work, int* count, uint32_t bits, int j, int lane) {
  const int n = __popc(bits);
  int incl = n;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  int base = 0;
  if (lane == 31 && incl) base = atomicAdd(count, incl);
  base = __shfl_sync(0xffffffffu, base, 31) + incl - n;
  for (uint32_t m = bits; m; m &= m - 1u) work[base++] = (uint16_t)((__ffs(m) - 1) * 128 + j);
}

// The quantizer's code of a latent v (fp32 arithmetic, as the oracle):
// round((v - z) / s) clamped to [0, qmax]; 0 when s is 0.  Non-decreasing in v.
__device__ __forceinline__ float quant_code(float v, float z32, float s32, float qmax) {
  if (s32 == 0.f) return 0.f;
  return fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(v, z32), s32)), 0.f), qmax);
}

// Tensor-core projection of a complete block's new rows (quantized caches).
// L'_tj = x_t . (H_j + L_j) 2^-10 - mu.V_j, with H + L the fp16 hi/lo split
// of 2^10 V_g (mma.sync m16n8k16, the hi and lo products in separate fp32
// accumulators), for rows t >= off_new; the basis comes from global memory
// (L2) as B fragments.  A third chain forms S_tj = sum_d |x_d| |V_dj| (from
// |x| and the fp16 |H|), and err_tj = 2^-16 S_tj + 2^-21 |mu.V_j| bounds
// |L'_tj - L_tj| with margin: each of the eight accumulation steps of a
// chain adds a few units of 2^-24 of S_tj, the hi/lo split leaves 2^-22 S_tj,
// and the final roundings a few units of 2^-24 of S_tj + |mu.V_j|.
// Warp w of nw takes the 8-channel tiles w, w + nw, ... (two at a time);
// both 16-row tiles.
template <int NT>
__device__ __forceinline__ void project_tc(const __half* xs, const float* __restrict__ bT, float* lat, float* err,
                                           int r, const float2* mv, int off_new) {
  constexpr int nw = NT / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int n_nt = (r + 7) / 8;
  const uint32_t xbase = smem_addr(xs);
#pragma unroll 1
  for (int pass = 0; nw < 4 || pass < 2; ++pass) {  // (at most 16 tiles)
    if (warp + 2 * nw * pass >= n_nt) break;  // uniform
    float ah[2][2][4], al[2][2][4], aa[2][2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) ah[i][m][e] = al[i][m][e] = aa[i][m][e] = 0.f;
#pragma unroll 2
    for (int ks = 0; ks < kHeadDim / 16; ++ks) {
      uint32_t a[2][4], ab[2][4];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        ldsm_x4(a[m][0], a[m][1], a[m][2], a[m][3],
                xbase + 2 * ((16 * m + (lane & 15)) * kXsStride + 16 * ks + 8 * (lane >> 4)));
#pragma unroll
        for (int q = 0; q < 4; ++q) ab[m][q] = a[m][q] & 0x7fff7fffu;
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int nt = warp + 2 * nw * pass + nw * i;
        if (nt < n_nt) {  // uniform
          const int j = 8 * nt + g;
          float2 v01 = make_float2(0.f, 0.f), v89 = make_float2(0.f, 0.f);
          if (j < r) {
            const float* row = bT + (size_t)j * kHeadDim + 16 * ks + 2 * c;
            v01 = __ldg(reinterpret_cast<const float2*>(row));
            v89 = __ldg(reinterpret_cast<const float2*>(row + 8));
          }
          const float v[4] = {v01.x * 1024.f, v01.y * 1024.f, v89.x * 1024.f, v89.y * 1024.f};
          const uint32_t h01 = pack_f16x2(v[0], v[1]), h89 = pack_f16x2(v[2], v[3]);
          const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
          const float2 f89 = __half22float2(*reinterpret_cast<const __half2*>(&h89));
          const uint32_t l01 = pack_f16x2(v[0] - f01.x, v[1] - f01.y), l89 = pack_f16x2(v[2] - f89.x, v[3] - f89.y);
          const uint32_t b01 = h01 & 0x7fff7fffu, b89 = h89 & 0x7fff7fffu;
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            mma_f16(ah[i][m], a[m][0], a[m][1], a[m][2], a[m][3], h01, h89);
            mma_f16(al[i][m], a[m][0], a[m][1], a[m][2], a[m][3], l01, l89);
            mma_f16(aa[i][m], ab[m][0], ab[m][1], ab[m][2], ab[m][3], b01, b89);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int nt = warp + 2 * nw * pass + nw * i;
      if (nt >= n_nt) continue;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 8 * nt + 2 * c + (e & 1);
        if (j >= r) continue;
        const float2 mj = mv[j];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int t = 16 * m + g + 8 * (e >> 1);
          if (t < off_new) continue;
          const float pr = __fmul_rn(__fadd_rn(ah[i][m][e], al[i][m][e]), 1.f / 1024.f);
          lat[t * (r + 1) + j] = __fsub_rn(__fsub_rn(pr, mj.x), mj.y);
          // |H| is |V| 2^10 to within 2^-11 relative: 1.001 covers it and the chain's own rounding
          err[t * (r + 1) + j] = fmaf(aa[i][m][e], 0x1p-26f * 1.001f, fabsf(mj.x) * 0x1p-21f);
        }
      }
    }
  }
}

// grid (blocks touched, kv_heads, batch), NT threads: 64 for phase 1 of a
// quantized cache of rank <= 40 (every block takes the tensor-core path and
// one thread per channel needs no more), else 128.
// Two launches per append (phase 1, then phase 2 on the same stream): phase 1
// fills every block the tokens reach except a last, partial one; phase 2
// writes that partial block (the tail) and publishes the new length.  A
// single launch would race: the CTA completing the old partial block reads
// the tail rows the CTA of the new partial block overwrites.
// counts (device [batch], or NULL): sequence b appends the first counts[b]
// of its T rows; NULL appends all T rows of every sequence.
template <int NT>
__global__ void __launch_bounds__(NT, NT == 64 ? 12 : 6) encode_append_kernel(CacheView cv, const __half* __restrict__ x,
                                                                           long long T, int Hkv, int phase,
                                                                           const int* counts) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int r = cv.r;
  const EncodeSmem L = encode_smem(r, cv.rec_bytes);
  __half* xs = reinterpret_cast<__half*>(smem + L.xs_off);
  float* err = reinterpret_cast<float*>(smem + L.err_off);
  int* n_work = reinterpret_cast<int*>(smem + L.work_off);
  uint32_t* wmax_s = reinterpret_cast<uint32_t*>(smem + L.work_off + 8);  // each warp's largest scale
  uint16_t* work = reinterpret_cast<uint16_t*>(smem + L.work_off + 24);
  float* bas = reinterpret_cast<float*>(smem + L.basis_off);
  float* lat = reinterpret_cast<float*>(smem + L.lat_off);
  uint8_t* codes = smem + L.codes_off;
  __half2* sz = reinterpret_cast<__half2*>(smem + L.sz_off);
  uint8_t* rec = smem + L.rec_off;

  const int tid = threadIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const bool ragged = __ldcg(&cv.hdr->ragged) != 0;
  const long long p0 = ragged ? __ldcg(cv.seq_len + b) : __ldcg(&cv.hdr->length);
  const long long n_b = counts ? (long long)__ldcg(counts + b) : T;
  const long long p1 = p0 + n_b;
  const unsigned int n_cta = gridDim.x * gridDim.y * gridDim.z;

  if (!ragged && p1 > cv.capacity) {
    if (blockIdx.x == 0 && h == 0 && b == 0 && tid == 0) set_dev_error(cv.hdr, PALU_DEVERR_CAPACITY);
    return;  // nothing written, length unchanged (no CTA takes a ticket)
  }
  // ragged: a sequence whose append would pass the capacity (or whose count
  // is out of range) writes nothing and keeps its length
  const bool refused = ragged && (n_b < 0 || n_b > T || p1 > cv.capacity);
  if (refused && blockIdx.x == 0 && h == 0 && tid == 0) set_dev_error(cv.hdr, PALU_DEVERR_CAPACITY);

  // phase 1: block p0 / 32 + blockIdx.x; phase 2: the block holding token p1
  const long long blk = phase == 2 ? p1 / kBlock : p0 / kBlock + blockIdx.x;
  const long long lo = blk * kBlock;
  const bool last_partial = blk == p1 / kBlock && p1 % kBlock != 0;
  if (!refused && lo < p1 && last_partial == (phase == 2) && bounds_ok(blk < cv.n_blk_cap, cv.hdr)) {
    const long long new_lo = lo > p0 ? lo : p0;
    const long long hi = (lo + kBlock < p1) ? lo + kBlock : p1;
    const int off_new = (int)(new_lo - lo);
    const int n_new = (int)(hi - new_lo);
    const bool complete = (hi - lo) == kBlock;
    const int grp = h / cv.heads_per_group;

    // Quantized caches project a complete block on the tensor cores and
    // compute exact latents only where a stored value depends on them (see
    // the quantizer below); everything else takes the exact path for every
    // latent, from a staged copy of the basis.
    const bool tc = cv.quantize && complete;
    const float* bT = cv.basisT + (size_t)grp * r * kHeadDim;

    // stage the new tokens' rows (and, on the exact path, the group basis)
    if (tid < 2) n_work[tid] = 0;
    const __half* xsrc = x + (((long long)b * Hkv + h) * T + (new_lo - p0)) * kHeadDim;
    for (int i = tid; i < n_new * (kHeadDim / 8); i += blockDim.x) {
      const int t = i / (kHeadDim / 8), q = i % (kHeadDim / 8);
      reinterpret_cast<uint4*>(xs + (off_new + t) * kXsStride)[q] =
          reinterpret_cast<const uint4*>(xsrc + (long long)t * kHeadDim)[q];
    }
    const float* bsrc = bT;
    for (int i = tid; i < (tc ? 0 : r) * (kHeadDim / 4); i += blockDim.x) {
      const int j = i / (kHeadDim / 4), q = i % (kHeadDim / 4);
      const float4 v = reinterpret_cast<const float4*>(bsrc + (size_t)j * kHeadDim)[q];
      float* dst = bas + j * (kHeadDim + 1) + 4 * q;
      dst[0] = v.x;
      dst[1] = v.y;
      dst[2] = v.z;
      dst[3] = v.w;
    }
    __syncthreads();

    if (tc) {
      project_tc<NT>(xs, bT, lat, err, r, cv.mv + (size_t)grp * r, off_new);
    } else if constexpr (NT == 128) {  // (the host launches 64 threads only where tc holds)
      // projection: warp w takes tokens off_new + w + 4i, lane takes channels lane + 32k.
      // Each (token, channel) latent is sum_d x_d V_dj accumulated as an
      // unevaluated float pair (error-free products and sums), minus mu_g.V_g[:, j],
      // then rounded once to fp32.
      const int warp = tid >> 5, lane = tid & 31;
      float S[8][4], E[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) S[i][k] = E[i][k] = 0.f;
      const int nt = (n_new - warp + 3) / 4;  // tokens of this warp (may be <= 0)
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
            const float xv = __half2float(xs[(off_new + warp + 4 * i) * kXsStride + d]);
#pragma unroll
            for (int k = 0; k < 4; ++k) fp_acc(S[i][k], E[i][k], xv, v[k]);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = lane + 32 * k;
        if (j < r) {
          const float2 m = cv.mv[(size_t)grp * r + j];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < nt) lat[(off_new + warp + 4 * i) * (r + 1) + j] = fp_finish(S[i][k], E[i][k], m);
        }
      }
    }

    const long long rec_index = ((long long)b * Hkv + h) * cv.n_blk_cap + blk;
    uint8_t* gdst = cv.blocks + rec_index * cv.rec_bytes;
    float* tail = cv.quantize ? cv.tail + ((long long)b * Hkv + h) * kBlock * r : nullptr;

    if (cv.quantize) {
      if (complete) {
        // earlier tokens of this block come from the tail (exact)
        for (int i = tid; i < off_new * r; i += blockDim.x) {
          const int t = i / r, j = i % r;
          lat[t * (r + 1) + j] = tail[t * r + j];
          err[t * (r + 1) + j] = 0.f;
        }
        __syncthreads();
        {  // complete block of a quantized cache: tc holds
          // Each new latent is known to within its bound err (tail rows
          // exactly).  The block's minimum over a channel then lies in
          // [min (v - e), min (v + e)] and its maximum in [max (v - e),
          // max (v + e)]; zero = fp16(min) and scale = fp16(fl(fl(max - min)
          // / qmax)) are monotone in them, so when both ends of those
          // intervals give the same fp16 values they are the exact path's.
          // Only the other channels need exact latents, of the tokens that can
          // hold the minimum or maximum.  A code is taken from the bound
          // interval when the whole interval rounds to one code (the
          // quantizer is monotone), else from the exact latent.  One thread
          // per channel walks the block's 32 tokens (r <= blockDim.x);
          // the exact latents are computed by all threads from shared work
          // lists of (token, channel) pairs.
          const int warp = tid >> 5, lane = tid & 31, j = tid;
          const bool own = j < r;
          const uint32_t fresh = ~((1u << off_new) - 1u);  // tokens of this append (off_new <= 31)
          const int ld = r + 1;
          const float qmax = (float)((1 << (j < cv.n_hi ? 4 : 2)) - 1);
          uint32_t bmin = 0u, bmax = 0u;  // candidates of an uncertain channel
          bool certain = false;
          if (own) {
            float mh = INFINITY, ml = -INFINITY, lmin = INFINITY, hmax = -INFINITY;
#pragma unroll 8
            for (int t = 0; t < kBlock; ++t) {
              const float v = lat[t * ld + j], e = err[t * ld + j];
              const float vh = v + e, vl = v - e;
              mh = fminf(mh, vh);
              lmin = fminf(lmin, vl);
              ml = fmaxf(ml, vl);
              hmax = fmaxf(hmax, vh);
            }
            const __half za = __float2half_rn(lmin), zb = __float2half_rn(mh);
            const __half sa = __float2half_rn(__fdiv_rn(__fsub_rn(ml, mh), qmax));
            const __half sb = __float2half_rn(__fdiv_rn(__fsub_rn(hmax, lmin), qmax));
            // (zeros that round to +-0, and a scale of -0, go the exact way,
            // which orders -0 below +0)
            certain = __half_as_ushort(za) == __half_as_ushort(zb) && (__half_as_ushort(za) & 0x7fffu) != 0u &&
                      __half_as_ushort(sa) == __half_as_ushort(sb) && __half_as_ushort(sa) != 0x8000u;
            if (certain) {
              sz[j] = __halves2half2(sa, za);
            } else {
              // the candidates: tokens whose interval reaches below the smallest
              // upper end (minimum) or above the largest lower end (maximum)
#pragma unroll 8
              for (int t = 0; t < kBlock; ++t) {
                const float v = lat[t * ld + j], e = err[t * ld + j];
                if (v - e <= mh) bmin |= 1u << t;
                if (v + e >= ml) bmax |= 1u << t;
              }
            }
          }
          push_work(work, &n_work[0], (bmin | bmax) & fresh, j, lane);
          __syncthreads();
          run_exact(work, n_work[0], xs, bT, cv.mv + (size_t)grp * r,
                    [&](int tt, int jj, float L) { lat[tt * ld + jj] = L; });
          __syncthreads();
          uint32_t need = 0u, wmax = 0u;  // wmax: the fp32 bits of this channel's (non-negative) scale
          if (own) {
            if (!certain) {
              // minimum and maximum over the candidates' exact latents (an
              // unsigned key of the same order, so that the stored zero keeps
              // the sign of the minimum's zero as the oracle's)
              unsigned int kmn = 0xffffffffu, kmx = 0u;
              for (uint32_t m = bmin; m; m &= m - 1u) kmn = min(kmn, f2key(lat[(__ffs(m) - 1) * ld + j]));
              for (uint32_t m = bmax; m; m &= m - 1u) kmx = max(kmx, f2key(lat[(__ffs(m) - 1) * ld + j]));
              const float mn = key2f(kmn), mx = key2f(kmx);
              sz[j] = __halves2half2(__float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), qmax)), __float2half_rn(mn));
            }
            const __half2 szj = sz[j];
            const float s32 = __low2float(szj), z32 = __high2float(szj);
            wmax = __float_as_uint(s32);
            if (s32 == 0.f) {
              for (int t = 0; t < kBlock; ++t) codes[t * r + j] = 0;
            } else {
              // the exact code is round(fl((L - z) / s)) for some L in [v - e, v + e]:
              // it is known when that interval, scaled by an approximate 1/s and
              // widened by the approximation's error, lies inside one rounding
              // cell; else it is decided from the exact latent below
              float inv;
              asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(s32));
#pragma unroll 8
              for (int t = 0; t < kBlock; ++t) {
                const float v = lat[t * ld + j], e = err[t * ld + j];
                const float u = (v - z32) * inv, du = fmaf(e, inv, fmaf(fabsf(u), 0x1p-18f, 0x1p-20f));
                const float k = rintf(u);
                if (fabsf(u - k) + du >= 0.5f) need |= 1u << t;
                codes[t * r + j] = (uint8_t)fminf(fmaxf(k, 0.f), qmax);
              }
              // tokens whose exact latent is at hand: the candidates of an
              // uncertain channel and the earlier tokens of the block (tail)
              const uint32_t exact = bmin | bmax | ~fresh;
              need &= ~exact;
              for (uint32_t m = exact; m; m &= m - 1u) {
                const int t = __ffs(m) - 1;
                codes[t * r + j] = (uint8_t)quant_code(lat[t * ld + j], z32, s32, qmax);
              }
            }
          }
          push_work(work, &n_work[1], need, j, lane);
          wmax = __reduce_max_sync(0xffffffffu, wmax);
          if (lane == 0) wmax_s[warp] = wmax;
          __syncthreads();
          // the block's largest scale into the stream's and the cache's maxima:
          // one atomic each per block, and none when the stored value is as large
          if (tid == 0) {
            uint32_t m = wmax_s[0];
            for (int w = 1; w < NT / 32; ++w) m = max(m, wmax_s[w]);
            unsigned int* sm = &cv.smax[(long long)b * Hkv + h];
            if (m > __ldcg(sm)) atomicMax(sm, m);
            if (m > __ldcg(&cv.hdr->max_scale)) atomicMax(&cv.hdr->max_scale, m);
          }
          run_exact(work, n_work[1], xs, bT, cv.mv + (size_t)grp * r, [&](int tt, int jj, float L) {
            const __half2 szj = sz[jj];
            codes[tt * r + jj] =
                (uint8_t)quant_code(L, __high2float(szj), __low2float(szj), (float)((1 << (jj < cv.n_hi ? 4 : 2)) - 1));
          });
        }
        __syncthreads();
        // every byte of the record is written: the code area by the packer, the
        // scale / zero area below
        pack_codes(codes, r, cv.role, cv.n_hi, cv.n_hi_oct, cv.n_lo_oct, rec, tid, blockDim.x);
        // scale / zero per padded channel
        const int n_pad = 8 * cv.n_oct;
        const int szb = 128 * cv.n_hi_oct + 64 * cv.n_lo_oct;
        __half* r16 = reinterpret_cast<__half*>(rec + szb);
        for (int pch = tid; pch < n_pad; pch += blockDim.x) {
          const int j = padded_to_channel(pch, r, cv.n_hi, cv.n_hi_oct, 1);
          const __half2 v = j >= 0 ? sz[j] : __halves2half2(__float2half(0.f), __float2half(0.f));
          if (cv.role == PALU_ROLE_KEY) {
            r16[pch] = __low2half(v);
            r16[n_pad + pch] = __high2half(v);
          } else {
            r16[2 * pch] = __low2half(v);
            r16[2 * pch + 1] = __high2half(v);
          }
        }
        __syncthreads();
        for (int i = tid; i < cv.rec_bytes / 16; i += blockDim.x)
          reinterpret_cast<uint4*>(gdst)[i] = reinterpret_cast<const uint4*>(rec)[i];
      } else {
        __syncthreads();
        for (int i = tid; i < n_new * r; i += blockDim.x) {
          const int t = off_new + i / r, j = i % r;
          tail[t * r + j] = lat[t * (r + 1) + j];
        }
      }
    } else {
      // fp16 latents: read-modify-write the block record
      if (off_new > 0) {
        for (int i = tid; i < cv.rec_bytes / 16; i += blockDim.x)
          reinterpret_cast<uint4*>(rec)[i] = reinterpret_cast<const uint4*>(gdst)[i];
      } else {
        for (int i = tid; i < cv.rec_bytes / 16; i += blockDim.x)
          reinterpret_cast<uint4*>(rec)[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
      for (int i = tid; i < n_new * r; i += blockDim.x) {
        const int t = off_new + i / r, j = i % r;
        *reinterpret_cast<__half*>(rec + latent_off(t, j)) = __float2half_rn(lat[t * (r + 1) + j]);
      }
      __syncthreads();
      for (int i = tid; i < cv.rec_bytes / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(gdst)[i] = reinterpret_cast<const uint4*>(rec)[i];
    }
  }

  // the last CTA of phase 2 to finish publishes the new length(s)
  if (phase != 2) return;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned int t = atomicAdd(&cv.hdr->ticket, 1u);
    if (t == n_cta - 1) {
      if (ragged) advance_ragged_lengths(cv, counts, T);
      else cv.hdr->length = p1;
      cv.hdr->ticket = 0u;
      __threadfence();
    }
  }
}

// Decode-time append of a single token per stream: one CTA per (KV head,
// batch).  The group's basis rows come into shared memory with one bulk copy;
// append_one_token (append_one.cuh) does the rest.  The last CTA to finish
// publishes the new length.
constexpr int kEncOneThreads = 256;
__global__ void __launch_bounds__(kEncOneThreads) encode_one_kernel(CacheView cv, const __half* __restrict__ x,
                                                                    int Hkv) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ uint64_t bar;
  const int tid = threadIdx.x;
  const int h = blockIdx.x, b = blockIdx.y;
  const int r = cv.r;
  const AppendSmem sm = append_smem(dsm, r, cv.rec_bytes);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, (uint32_t)r * 512u);
    bulk_g2s(sm.bas, cv.basisT + (size_t)(h / cv.heads_per_group) * r * kHeadDim, (uint32_t)r * 512u, &bar);
  }
  const long long p0 = seq_length(cv, b);
  __syncthreads();  // barrier initialised
  const bool got = mbar_wait_bounded(&bar, 0);  // also drains the copy before any early exit
  if (!got && tid == 0) set_dev_error(cv.hdr, PALU_DEVERR_TIMEOUT);
  if (__ldcg(&cv.hdr->length) + 1 > cv.capacity) {
    // the longest sequence is full: nothing written, lengths unchanged (no CTA takes a ticket)
    if (h == 0 && b == 0 && tid == 0) set_dev_error(cv.hdr, PALU_DEVERR_CAPACITY);
    return;
  }
  append_one_token(cv, x + ((long long)b * Hkv + h) * kHeadDim, p0, h, b, Hkv, sm);
  __syncthreads();
  if (tid == 0) publish_length(cv, p0, gridDim.x * gridDim.y);
}

// Switches a cache to ragged lengths (once): every sequence starts from the
// shared length.
__global__ void cache_make_ragged_kernel(StateHeader* hdr, long long* seq_len, int batch) {
  if (hdr->ragged) return;
  for (int b = 0; b < batch; ++b) seq_len[b] = hdr->length;
  hdr->ragged = 1u;
  __threadfence();
}

// Per-sequence rollback: sequence b goes back to lengths[b] tokens when that
// is allowed (no growth; for quantized caches a block boundary or a length
// inside the current partial block), else keeps its length and the
// rollback error bit is set.
__global__ void cache_truncate_ragged_kernel(StateHeader* hdr, long long* seq_len, int batch,
                                             const long long* lengths, int quantize) {
  long long mx = 0;
  bool bad = false;
  for (int b = 0; b < batch; ++b) {
    const long long cur = seq_len[b], n = lengths[b];
    const bool ok = n >= 0 && n <= cur && (!quantize || n % kBlock == 0 || n / kBlock == cur / kBlock);
    const long long nl = ok ? n : cur;
    bad |= !ok;
    seq_len[b] = nl;
    mx = nl > mx ? nl : mx;
  }
  hdr->length = mx;
  if (bad) hdr->err |= PALU_DEVERR_ROLLBACK;
}

// Sets the device length (the host has checked that no quantized block is reopened).
// With ragged lengths every sequence longer than `length` goes back to it
// when the rollback rule allows (else it keeps its length and the rollback
// error bit is set); shorter sequences keep theirs.
__global__ void cache_truncate_kernel(StateHeader* hdr, long long* seq_len, int batch, long long length,
                                      int quantize) {
  if (hdr->ragged) {
    long long mx = 0;
    bool bad = false;
    for (int b = 0; b < batch; ++b) {
      const long long cur = seq_len[b];
      long long nl = cur;
      if (length < cur) {
        const bool ok = !quantize || length % kBlock == 0 || length / kBlock == cur / kBlock;
        bad |= !ok;
        if (ok) nl = length;
      }
      seq_len[b] = nl;
      mx = nl > mx ? nl : mx;
    }
    hdr->length = mx;
    if (bad) hdr->err |= PALU_DEVERR_ROLLBACK;
    return;
  }
  if (length > hdr->length) {
    hdr->err |= PALU_DEVERR_CAPACITY;
    return;
  }
  hdr->length = length;
}

// ------------------------------------------------------------------ host
static int64_t n_hi_of(const palu_config* cfg, int r) {
  const double v = ceil(cfg->hi_fraction * (double)r - 1e-9);
  return std::max<int64_t>(0, std::min<int64_t>(r, (int64_t)v));
}

static palu_status check_config(const palu_config* cfg) {
  if (!cfg) return fail(PALU_ERR_INVALID_ARG, "config is NULL");
  if (cfg->head_dim != kHeadDim) return fail(PALU_ERR_UNSUPPORTED, "head_dim must be 128");
  if (cfg->group_size != kBlock) return fail(PALU_ERR_UNSUPPORTED, "group_size must be 32");
  if (cfg->hi_bit != 4 || cfg->lo_bit != 2) return fail(PALU_ERR_UNSUPPORTED, "hi_bit must be 4 and lo_bit 2");
  if (!(cfg->hi_fraction >= 0.0 && cfg->hi_fraction <= 1.0))
    return fail(PALU_ERR_INVALID_ARG, "hi_fraction must be in [0, 1]");
  if (cfg->n_head_groups < 1) return fail(PALU_ERR_INVALID_ARG, "n_head_groups must be >= 1");
  return PALU_OK;
}

struct Geometry {
  int n_hi, n_hi_oct, n_lo_oct, n_oct, rec_bytes;
};

static Geometry geometry(const palu_config* cfg, int role, int r) {
  Geometry g;
  const bool quant = cfg->quantize || role == PALU_ROLE_KEY;
  if (quant) {
    g.n_hi = (int)n_hi_of(cfg, r);
    g.n_hi_oct = (g.n_hi + 7) / 8;
    g.n_lo_oct = (r - g.n_hi + 7) / 8;
    g.n_oct = g.n_hi_oct + g.n_lo_oct;
    g.rec_bytes = 128 * g.n_hi_oct + 64 * g.n_lo_oct + 4 * 8 * g.n_oct;
  } else {
    g.n_hi = 0;
    g.n_hi_oct = g.n_lo_oct = 0;
    g.n_oct = (r + 7) / 8;
    g.rec_bytes = 512 * g.n_oct;
  }
  return g;
}

static palu_status check_cache_args(const palu_config* cfg, int32_t role, int32_t rank, int64_t batch,
                                    int32_t kv_heads, int64_t capacity) {
  palu_status st = check_config(cfg);
  if (st != PALU_OK) return st;
  if (role != PALU_ROLE_KEY && role != PALU_ROLE_VALUE) return fail(PALU_ERR_INVALID_ARG, "role must be KEY or VALUE");
  if (role == PALU_ROLE_KEY && !cfg->quantize)
    return fail(PALU_ERR_INVALID_ARG, "quantize=0 (fp16 latents) applies to value caches only");
  if (rank < 1 || rank > kMaxRank) return fail(PALU_ERR_INVALID_ARG, "rank must be in [1, 128]");
  if (batch < 1 || kv_heads < 1 || capacity < 1) return fail(PALU_ERR_INVALID_ARG, "batch, kv_heads, capacity must be >= 1");
  if (kv_heads % cfg->n_head_groups != 0)
    return fail(PALU_ERR_INVALID_ARG, "kv_heads must be a multiple of n_head_groups (contiguous head groups)");
  if (batch * (int64_t)kv_heads > 65535 * 64LL) return fail(PALU_ERR_UNSUPPORTED, "batch*kv_heads too large");
  return PALU_OK;
}

}  // namespace palu

using namespace palu;

extern "C" palu_status palu_cache_size(const palu_config* cfg, int32_t role, int32_t rank, int64_t batch,
                                       int32_t kv_heads, int64_t capacity, size_t* block_bytes, size_t* tail_bytes,
                                       size_t* state_bytes) {
  palu_status st = check_cache_args(cfg, role, rank, batch, kv_heads, capacity);
  if (st != PALU_OK) return st;
  const Geometry g = geometry(cfg, role, rank);
  const int64_t n_blk = (capacity + kBlock - 1) / kBlock;
  const bool quant = cfg->quantize || role == PALU_ROLE_KEY;
  if (block_bytes) *block_bytes = align_up((size_t)batch * kv_heads * n_blk * g.rec_bytes, 256);
  if (tail_bytes) *tail_bytes = quant ? align_up(sizeof(float) * (size_t)batch * kv_heads * kBlock * rank, 256) : 0;
  if (state_bytes) *state_bytes = state_layout(cfg->n_head_groups, rank, batch, kv_heads).total;
  return PALU_OK;
}

extern "C" palu_status palu_cache_init(palu_cache* cache, const palu_config* cfg, int32_t role, int32_t rank,
                                       int64_t batch, int32_t kv_heads, int64_t capacity, const float* basis,
                                       int32_t basis_ld, const float* mu, void* blocks, void* tail, void* state,
                                       void* stream) {
  if (!cache) return fail(PALU_ERR_INVALID_ARG, "cache is NULL");
  palu_status st = check_cache_args(cfg, role, rank, batch, kv_heads, capacity);
  if (st != PALU_OK) return st;
  const bool quant = cfg->quantize || role == PALU_ROLE_KEY;
  if (!basis || !mu || !blocks || !state || (quant && !tail))
    return fail(PALU_ERR_INVALID_ARG, "basis, mu, blocks, state (and tail for quantized caches) must be non-NULL");
  if (basis_ld < rank) return fail(PALU_ERR_INVALID_ARG, "basis_ld must be >= rank");
  if (((uintptr_t)blocks | (uintptr_t)state | (uintptr_t)(tail ? tail : state)) & 255)
    return fail(PALU_ERR_INVALID_ARG, "blocks, tail and state must be 256-byte aligned");
  const Geometry g = geometry(cfg, role, rank);
  palu_cache c;
  std::memset(&c, 0, sizeof(c));
  c.magic = kCacheMagic;
  c.role = role;
  c.head_dim = kHeadDim;
  c.rank = rank;
  c.n_hi = g.n_hi;
  c.n_groups = cfg->n_head_groups;
  c.heads_per_group = kv_heads / cfg->n_head_groups;
  c.quantize = quant ? 1 : 0;
  c.batch = (int32_t)batch;
  c.kv_heads = kv_heads;
  c.n_hi_oct = g.n_hi_oct;
  c.n_lo_oct = g.n_lo_oct;
  c.n_oct = g.n_oct;
  c.record_bytes = g.rec_bytes;
  c.capacity = capacity;
  c.n_blk_cap = (capacity + kBlock - 1) / kBlock;
  c.blocks = blocks;
  c.tail = quant ? static_cast<float*>(tail) : nullptr;
  c.state = state;
  c.length = 0;
  const StateLayout sl = state_layout(c.n_groups, rank, batch, kv_heads);
  uint8_t* s = static_cast<uint8_t*>(state);
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  // every byte of the state (padding, largest scales, sequence lengths) and
  // of the tail starts at zero, so cache images are a function of the calls
  st = cuda_check(cudaMemsetAsync(s, 0, sl.total, strm), "cudaMemsetAsync(state)");
  if (st != PALU_OK) return st;
  if (quant) {
    st = cuda_check(cudaMemsetAsync(tail, 0, sizeof(float) * (size_t)batch * kv_heads * kBlock * rank, strm),
                    "cudaMemsetAsync(tail)");
    if (st != PALU_OK) return st;
  }
  cache_init_kernel<<<dim3(rank, c.n_groups), kHeadDim, 0, strm>>>(
      basis, basis_ld, mu, reinterpret_cast<float*>(s + sl.basis_off), reinterpret_cast<float*>(s + sl.mu_off),
      reinterpret_cast<float2*>(s + sl.mv_off), reinterpret_cast<StateHeader*>(s), rank);
  st = cuda_check(cudaGetLastError(), "cache_init_kernel launch");
  if (st != PALU_OK) return st;
  *cache = c;
  return PALU_OK;
}

static palu_status check_cache(const palu_cache* c, const char* name) {
  if (!c) return fail(PALU_ERR_INVALID_ARG, std::string(name) + " is NULL");
  if (c->magic != kCacheMagic) return fail(PALU_ERR_NOT_INITIALIZED, std::string(name) + " is not initialised");
  return PALU_OK;
}

// One phase of an append.  Phase 1 of a quantized cache covers complete
// blocks only, on the tensor-core path, and launches without the staged-basis
// area; at rank <= 40 it runs 64-thread CTAs (one thread per channel is
// enough, at most five channel tiles of the projection fall on each warp, and
// more CTAs fit an SM).  Measured on rank 33 and 53 keys and values of one
// layer: 1.32 -> 1.22 ms at rank 33, 1.53 -> 1.99 ms at rank 53.
static palu_status launch_encode(const palu_cache* cache, const CacheView& cv, const __half* x, int64_t tokens,
                                 int phase, const int32_t* counts, unsigned nblk, cudaStream_t strm) {
  const EncodeSmem es = encode_smem(cache->rank, cache->record_bytes);
  const bool tc = phase == 1 && cache->quantize;
  const int smem = tc ? es.basis_off : es.total;
  const bool narrow = tc && cache->rank <= 40;
  const void* kfn = narrow ? reinterpret_cast<const void*>(encode_append_kernel<64>)
                           : reinterpret_cast<const void*>(encode_append_kernel<128>);
  int per_sm = 0;
  palu_status st = kernel_occupancy(kfn, narrow ? 64 : 128, es.total, &per_sm);
  if (st != PALU_OK) return st;
  const dim3 grid(phase == 1 ? nblk : 1u, cache->kv_heads, cache->batch);
  if (narrow)
    encode_append_kernel<64><<<grid, 64, smem, strm>>>(cv, x, tokens, cache->kv_heads, phase, counts);
  else
    encode_append_kernel<128><<<grid, 128, smem, strm>>>(cv, x, tokens, cache->kv_heads, phase, counts);
  return cuda_check(cudaGetLastError(), "encode_append_kernel launch");
}

extern "C" palu_status palu_encode_append(palu_cache* cache, const void* x, int64_t tokens, void* stream) {
  palu_status st = check_cache(cache, "cache");
  if (st != PALU_OK) return st;
  if (tokens < 0) return fail(PALU_ERR_INVALID_ARG, "tokens must be >= 0");
  if (tokens == 0) return PALU_OK;
  if (!x || ((uintptr_t)x & 15)) return fail(PALU_ERR_INVALID_ARG, "x must be a non-NULL, 16-byte aligned device pointer");
  if (cache->length + tokens > cache->capacity)
    return fail(PALU_ERR_CAPACITY, "append of " + std::to_string(tokens) + " tokens to a cache holding " +
                                       std::to_string(cache->length) + " exceeds its capacity " +
                                       std::to_string(cache->capacity));
  const int64_t nblk = (tokens + kBlock - 1) / kBlock + 1;  // blocks touched from any start offset
  if (nblk > 2147483647LL) return fail(PALU_ERR_UNSUPPORTED, "too many tokens in one append");
  if (tokens == 1) {
    const int smem1 = (int)append_smem_bytes(cache->rank, cache->record_bytes);
    int per_sm1 = 0;
    st = kernel_occupancy(reinterpret_cast<const void*>(encode_one_kernel), kEncOneThreads, smem1, &per_sm1);
    if (st != PALU_OK) return st;
    encode_one_kernel<<<dim3(cache->kv_heads, cache->batch), kEncOneThreads, smem1, static_cast<cudaStream_t>(stream)>>>(
        make_view(cache), static_cast<const __half*>(x), cache->kv_heads);
    st = cuda_check(cudaGetLastError(), "encode_one_kernel launch");
    if (st != PALU_OK) return st;
    cache->length += 1;
    return PALU_OK;
  }
  const CacheView cv = make_view(cache);
  for (int phase = 1; phase <= 2; ++phase) {
    st = launch_encode(cache, cv, static_cast<const __half*>(x), tokens, phase, nullptr, (unsigned)nblk,
                       static_cast<cudaStream_t>(stream));
    if (st != PALU_OK) return st;
  }
  cache->length += tokens;
  return PALU_OK;
}

extern "C" palu_status palu_encode_append_ragged(palu_cache* cache, const void* x, int64_t tokens,
                                                 const int32_t* counts, void* stream) {
  palu_status st = check_cache(cache, "cache");
  if (st != PALU_OK) return st;
  if (tokens < 0) return fail(PALU_ERR_INVALID_ARG, "tokens must be >= 0");
  if (tokens == 0) return PALU_OK;
  if (!x || ((uintptr_t)x & 15)) return fail(PALU_ERR_INVALID_ARG, "x must be a non-NULL, 16-byte aligned device pointer");
  if (!counts || ((uintptr_t)counts & 3)) return fail(PALU_ERR_INVALID_ARG, "counts must be a non-NULL int32 device pointer");
  if (cache->batch > kMaxRaggedBatch)
    return fail(PALU_ERR_UNSUPPORTED, "ragged lengths are supported up to " + std::to_string(kMaxRaggedBatch) + " sequences");
  const int64_t nblk = (tokens + kBlock - 1) / kBlock + 1;  // blocks touched from any start offset
  if (nblk > 2147483647LL) return fail(PALU_ERR_UNSUPPORTED, "too many tokens in one append");
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  const CacheView cv = make_view(cache);
  cache_make_ragged_kernel<<<1, 1, 0, strm>>>(cv.hdr, cv.seq_len, cache->batch);
  st = cuda_check(cudaGetLastError(), "cache_make_ragged_kernel launch");
  if (st != PALU_OK) return st;
  for (int phase = 1; phase <= 2; ++phase) {
    st = launch_encode(cache, cv, static_cast<const __half*>(x), tokens, phase, counts, (unsigned)nblk, strm);
    if (st != PALU_OK) return st;
  }
  // the host count stays an upper bound of the longest sequence (the counts
  // are on the device); palu_cache_sync or palu_cache_lengths makes it exact
  cache->length = std::min<int64_t>(cache->length + tokens, cache->capacity);
  return PALU_OK;
}

extern "C" palu_status palu_cache_truncate_ragged(palu_cache* cache, const int64_t* lengths, void* stream) {
  palu_status st = check_cache(cache, "cache");
  if (st != PALU_OK) return st;
  if (!lengths || ((uintptr_t)lengths & 7)) return fail(PALU_ERR_INVALID_ARG, "lengths must be a non-NULL int64 device pointer");
  if (cache->batch > kMaxRaggedBatch)
    return fail(PALU_ERR_UNSUPPORTED, "ragged lengths are supported up to " + std::to_string(kMaxRaggedBatch) + " sequences");
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  const CacheView cv = make_view(cache);
  cache_make_ragged_kernel<<<1, 1, 0, strm>>>(cv.hdr, cv.seq_len, cache->batch);
  st = cuda_check(cudaGetLastError(), "cache_make_ragged_kernel launch");
  if (st != PALU_OK) return st;
  cache_truncate_ragged_kernel<<<1, 1, 0, strm>>>(cv.hdr, cv.seq_len, cache->batch,
                                                reinterpret_cast<const long long*>(lengths), cache->quantize);
  return cuda_check(cudaGetLastError(), "cache_truncate_ragged_kernel launch");
}

extern "C" palu_status palu_cache_lengths(palu_cache* cache, int64_t* lengths, void* stream) {
  palu_status st = check_cache(cache, "cache");
  if (st != PALU_OK) return st;
  if (!lengths) return fail(PALU_ERR_INVALID_ARG, "lengths is NULL");
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  st = cuda_check(cudaStreamSynchronize(strm), "cudaStreamSynchronize");
  if (st != PALU_OK) return st;
  const CacheView cv = make_view(cache);
  StateHeader h;
  st = cuda_check(cudaMemcpy(&h, cv.hdr, sizeof(h), cudaMemcpyDeviceToHost), "read cache state");
  if (st != PALU_OK) return st;
  if (h.ragged) {
    st = cuda_check(cudaMemcpy(lengths, cv.seq_len, sizeof(int64_t) * (size_t)cache->batch, cudaMemcpyDeviceToHost),
                    "read sequence lengths");
    if (st != PALU_OK) return st;
  } else {
    for (int b = 0; b < cache->batch; ++b) lengths[b] = h.length;
  }
  cache->length = h.length;
  return PALU_OK;
}

extern "C" palu_status palu_cache_truncate(palu_cache* cache, int64_t length, void* stream) {
  palu_status st = check_cache(cache, "cache");
  if (st != PALU_OK) return st;
  // (on a cache with ragged lengths the kernel sets every sequence to `length`
  // only if each allows it; palu_cache_truncate_ragged is the general call)
  if (length < 0 || length > cache->length)
    return fail(PALU_ERR_INVALID_ARG, "truncate length must be in [0, current length]");
  const int64_t open_block = (cache->length / kBlock) * kBlock;
  if (cache->quantize && length % kBlock != 0 && length < open_block)
    return fail(PALU_ERR_INVALID_ARG,
                "truncate to a length inside an already quantized 32-token block is not possible; use a multiple of 32");
  const CacheView cv = make_view(cache);
  cache_truncate_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(cv.hdr, cv.seq_len, cache->batch, length,
                                                                        cache->quantize);
  st = cuda_check(cudaGetLastError(), "cache_truncate_kernel launch");
  if (st != PALU_OK) return st;
  cache->length = length;
  return PALU_OK;
}

// ------------------------------------------------------------------ save / restore
// A cache image (the "prompt cache" of page "add TurboQuant KV cache
// compression": a saved prompt prefix reused by a later request): a fixed
// header, then the state (basis, mean, header with the largest stored
// scale), the records of the stream's stored blocks, and the fp32 tail.  Plain bytes in host memory; little-endian as the host.
namespace palu {
constexpr uint64_t kImageMagic = 0x50414C55494D4731ull;  // "PALUIMG1"
struct ImageHeader {
  uint64_t magic;
  int32_t role, head_dim, rank, n_hi, n_groups, heads_per_group, quantize, batch, kv_heads, record_bytes;
  int64_t length, n_blocks, state_bytes, block_bytes, tail_bytes;
  int32_t pad[10];
};
static_assert(sizeof(ImageHeader) == 128, "image header is 128 bytes");

// Records per stream that hold data at `length` tokens: the full blocks, and
// for unquantized caches the partial block too.
static int64_t stored_blocks(const palu_cache* c, int64_t length) {
  return c->quantize ? length / kBlock : (length + kBlock - 1) / kBlock;
}

static ImageHeader image_header(const palu_cache* c) {
  ImageHeader h;
  std::memset(&h, 0, sizeof(h));
  h.magic = kImageMagic;
  h.role = c->role;
  h.head_dim = c->head_dim;
  h.rank = c->rank;
  h.n_hi = c->n_hi;
  h.n_groups = c->n_groups;
  h.heads_per_group = c->heads_per_group;
  h.quantize = c->quantize;
  h.batch = c->batch;
  h.kv_heads = c->kv_heads;
  h.record_bytes = c->record_bytes;
  h.length = c->length;
  h.n_blocks = stored_blocks(c, c->length);
  h.state_bytes = (int64_t)state_layout(c->n_groups, c->rank, c->batch, c->kv_heads).total;
  h.block_bytes = (int64_t)c->batch * c->kv_heads * h.n_blocks * c->record_bytes;
  h.tail_bytes = c->quantize ? (int64_t)sizeof(float) * c->batch * c->kv_heads * kBlock * c->rank : 0;
  return h;
}

// After a restore: the image's length, a clear error word and ticket (the
// largest stored scale comes with the image's state).
__global__ void cache_restore_header_kernel(StateHeader* hdr, long long length) {
  hdr->length = length;
  hdr->err = 0u;
  hdr->ticket = 0u;
}
}  // namespace palu

extern "C" palu_status palu_cache_save_size(const palu_cache* cache, size_t* bytes) {
  palu_status st = check_cache(cache, "cache");
  if (st != PALU_OK) return st;
  if (!bytes) return fail(PALU_ERR_INVALID_ARG, "bytes is NULL");
  const ImageHeader h = image_header(cache);
  *bytes = sizeof(ImageHeader) + (size_t)(h.state_bytes + h.block_bytes + h.tail_bytes);
  return PALU_OK;
}

extern "C" palu_status palu_cache_save(const palu_cache* cache, void* host, size_t bytes, void* stream) {
  palu_status st = check_cache(cache, "cache");
  if (st != PALU_OK) return st;
  if (!host) return fail(PALU_ERR_INVALID_ARG, "host buffer is NULL");
  const ImageHeader h = image_header(cache);
  const size_t need = sizeof(ImageHeader) + (size_t)(h.state_bytes + h.block_bytes + h.tail_bytes);
  if (bytes < need) return fail(PALU_ERR_INVALID_ARG, "host buffer too small: need " + std::to_string(need) + " bytes");
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  uint8_t* dst = static_cast<uint8_t*>(host);
  std::memcpy(dst, &h, sizeof(h));
  dst += sizeof(h);
  st = cuda_check(cudaMemcpyAsync(dst, cache->state, (size_t)h.state_bytes, cudaMemcpyDeviceToHost, strm),
                  "cudaMemcpyAsync(state)");
  if (st != PALU_OK) return st;
  dst += h.state_bytes;
  if (h.block_bytes > 0) {
    // the stored prefix of every stream's records, gathered densely
    const size_t width = (size_t)h.n_blocks * cache->record_bytes;
    st = cuda_check(cudaMemcpy2DAsync(dst, width, cache->blocks, (size_t)cache->n_blk_cap * cache->record_bytes, width,
                                      (size_t)cache->batch * cache->kv_heads, cudaMemcpyDeviceToHost, strm),
                    "cudaMemcpy2DAsync(blocks)");
    if (st != PALU_OK) return st;
    dst += h.block_bytes;
  }
  if (h.tail_bytes > 0)
    st = cuda_check(cudaMemcpyAsync(dst, cache->tail, (size_t)h.tail_bytes, cudaMemcpyDeviceToHost, strm),
                    "cudaMemcpyAsync(tail)");
  return st;
}

extern "C" palu_status palu_cache_restore(palu_cache* cache, const void* host, size_t bytes, void* stream) {
  palu_status st = check_cache(cache, "cache");
  if (st != PALU_OK) return st;
  if (!host || bytes < sizeof(ImageHeader)) return fail(PALU_ERR_INVALID_ARG, "host image is NULL or too short");
  ImageHeader h;
  std::memcpy(&h, host, sizeof(h));
  if (h.magic != kImageMagic) return fail(PALU_ERR_INVALID_ARG, "not a cache image (bad magic)");
  const ImageHeader mine = image_header(cache);
  if (h.role != mine.role || h.head_dim != mine.head_dim || h.rank != mine.rank || h.n_hi != mine.n_hi ||
      h.n_groups != mine.n_groups || h.heads_per_group != mine.heads_per_group || h.quantize != mine.quantize ||
      h.batch != mine.batch || h.kv_heads != mine.kv_heads || h.record_bytes != mine.record_bytes)
    return fail(PALU_ERR_INVALID_ARG,
                "the image was saved from a cache of another role, rank, head grouping, quantization, batch or kv_heads");
  if (h.length < 0 || h.length > cache->capacity)
    return fail(PALU_ERR_CAPACITY, "the image holds " + std::to_string(h.length) + " tokens, the cache's capacity is " +
                                       std::to_string(cache->capacity));
  if (h.n_blocks != stored_blocks(cache, h.length) || h.state_bytes != mine.state_bytes ||
      h.block_bytes != (int64_t)cache->batch * cache->kv_heads * h.n_blocks * cache->record_bytes ||
      h.tail_bytes != mine.tail_bytes)
    return fail(PALU_ERR_INVALID_ARG, "inconsistent cache image header");
  const size_t need = sizeof(ImageHeader) + (size_t)(h.state_bytes + h.block_bytes + h.tail_bytes);
  if (bytes < need) return fail(PALU_ERR_INVALID_ARG, "host image too short: need " + std::to_string(need) + " bytes");
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  const uint8_t* src = static_cast<const uint8_t*>(host) + sizeof(h);
  st = cuda_check(cudaMemcpyAsync(cache->state, src, (size_t)h.state_bytes, cudaMemcpyHostToDevice, strm),
                  "cudaMemcpyAsync(state)");
  if (st != PALU_OK) return st;
  src += h.state_bytes;
  if (h.block_bytes > 0) {
    const size_t width = (size_t)h.n_blocks * cache->record_bytes;
    st = cuda_check(cudaMemcpy2DAsync(cache->blocks, (size_t)cache->n_blk_cap * cache->record_bytes, src, width, width,
                                      (size_t)cache->batch * cache->kv_heads, cudaMemcpyHostToDevice, strm),
                    "cudaMemcpy2DAsync(blocks)");
    if (st != PALU_OK) return st;
    src += h.block_bytes;
  }
  if (h.tail_bytes > 0) {
    st = cuda_check(cudaMemcpyAsync(cache->tail, src, (size_t)h.tail_bytes, cudaMemcpyHostToDevice, strm),
                    "cudaMemcpyAsync(tail)");
    if (st != PALU_OK) return st;
  }
  cache_restore_header_kernel<<<1, 1, 0, strm>>>(reinterpret_cast<StateHeader*>(cache->state), h.length);
  st = cuda_check(cudaGetLastError(), "cache_restore_header_kernel launch");
  if (st != PALU_OK) return st;
  cache->length = h.length;
  return PALU_OK;
}

extern "C" palu_status palu_cache_stats(const palu_cache* c, palu_stats* s) {
  palu_status st = check_cache(c, "cache");
  if (st != PALU_OK) return st;
  if (!s) return fail(PALU_ERR_INVALID_ARG, "stats is NULL");
  std::memset(s, 0, sizeof(*s));
  const double streams = (double)c->batch * c->kv_heads;
  const int64_t n_full = c->length / kBlock, n_tail = c->length % kBlock;
  s->length = c->length;
  s->rank = c->rank;
  s->n_hi = c->n_hi;
  const double code_bits = c->quantize ? (double)(c->n_hi * 4 + (c->rank - c->n_hi) * 2) : 16.0 * c->rank;
  if (c->quantize) {
    s->code_bytes = streams * n_full * kBlock * code_bits / 8.0;
    s->meta_bytes = streams * n_full * c->rank * 4.0;
    s->tail_bytes = streams * n_tail * c->rank * 4.0;
    s->record_bytes = streams * n_full * (double)c->record_bytes;
  } else {
    s->code_bytes = streams * c->length * c->rank * 2.0;
    s->record_bytes = streams * ((c->length + kBlock - 1) / kBlock) * (double)c->record_bytes;
  }
  s->basis_bytes = 4.0 * c->n_groups * (double)c->rank * kHeadDim + 4.0 * c->n_groups * kHeadDim;
  s->fp16_bytes = streams * c->length * kHeadDim * 2.0;
  s->effective_bits = code_bits / kHeadDim;
  s->bits_with_meta = c->quantize ? (code_bits + c->rank * 32.0 / kBlock) / kHeadDim : s->effective_bits;
  return PALU_OK;
}

namespace palu {
// One CTA waits, with the library's bounded wait, on an mbarrier that its
// thread 0 either completes (signal != 0) or leaves pending.  No copy is ever
// issued on the barrier, so nothing is in flight when the wait gives up and
// the CTA returns.  A wait that runs out sets the TIMEOUT bit, as every
// bounded wait of the library does.
__global__ void wait_probe_kernel(StateHeader* hdr, uint32_t limit, int signal) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && signal) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&bar)) : "memory");
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar, 0, limit));
  if (!ok && threadIdx.x == 0) set_dev_error(hdr, PALU_DEVERR_TIMEOUT);
}
}  // namespace palu

extern "C" palu_status palu_debug_wait_probe(palu_cache* c, uint32_t spin_limit, int32_t signal, void* stream) {
  palu_status st = check_cache(c, "cache");
  if (st != PALU_OK) return st;
  if (spin_limit < 1 || spin_limit > (1u << 20))
    return fail(PALU_ERR_INVALID_ARG, "spin_limit must be in [1, 2^20]");
  wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<StateHeader*>(c->state), spin_limit,
                                                                      signal ? 1 : 0);
  return cuda_check(cudaGetLastError(), "wait_probe_kernel launch");
}

extern "C" palu_status palu_cache_sync(palu_cache* c, uint32_t* device_error, void* stream) {
  palu_status st = check_cache(c, "cache");
  if (st != PALU_OK) return st;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  st = cuda_check(cudaStreamSynchronize(strm), "cudaStreamSynchronize");
  if (st != PALU_OK) return st;
  StateHeader h;
  st = cuda_check(cudaMemcpy(&h, c->state, sizeof(h), cudaMemcpyDeviceToHost), "read cache state");
  if (st != PALU_OK) return st;
  c->length = h.length;
  if (device_error) *device_error = h.err;
  if (h.err) {
    const unsigned int zero = 0;
    cudaMemcpy(static_cast<uint8_t*>(c->state) + offsetof(StateHeader, err), &zero, sizeof(zero),
               cudaMemcpyHostToDevice);
    return fail(PALU_ERR_DEVICE, "device error word 0x" + [](unsigned v) {
      char b[16];
      snprintf(b, sizeof(b), "%x", v);
      return std::string(b);
    }(h.err) + " (1 capacity, 2 copy wait timeout, 4 K/V length mismatch, 8 eigen-solver not converged)");
  }
  return PALU_OK;
}
