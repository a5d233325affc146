// Single-token append (decode steps 1-2 of page "PALU — True Low-Rank Latent
// Storage for Keys and Values", "How it works"): project the new token into
// the stored group basis, L = (x - mu_g) V_g, keep it in the fp32 tail, and
// when it completes a 32-token block quantize and pack the block (asymmetric
// min/max per channel, blog post "VeloxQuant-MLX 0.8.0 adds KIVI", "What KIVI
// is"; LSB-first fields, blog post "How I built VeloxQuant-MLX", "The
// Bit-Packing Problem").  Shared by the one-token append kernel and the fused
// decode-step prologue.
#pragma once

#include "palu_internal.cuh"

namespace palu {

// Pack a block's codes (codes[t * r + j], token t, channel j) into the code
// area of its quantized record, one storage unit per thread and step: a u32
// per lane of a 4-bit octet, a u16 per lane of a 2-bit octet (two 2-bit
// octets share a lane's u32; a lone last one has u16s), LSB-first fields.
// The layout: channel j -> (octet, slot), hi channels first; within an
// octet, lane = 4g + c and field k = 0..3 (bits 4k, or 2k, of a half), half
// 0/1 (bits 0-15 / 16-31, or 0-7 / 8-15).  Keys: token t = g + 8k, slot
// 2c + half.  Values: slot g, token t = 8k + 2c + half.  Padding channels of
// an octet hold code 0.  Every byte of the code area is written.
__device__ __forceinline__ void pack_codes(const uint8_t* codes, int r, int role, int n_hi, int n_hi_oct,
                                           int n_lo_oct, uint8_t* rec, int tid, int nthreads) {
  const int npair = n_lo_oct >> 1;
  const bool key = role == PALU_ROLE_KEY;
  for (int u = tid; u < 32 * (n_hi_oct + n_lo_oct); u += nthreads) {
    const int octet = u >> 5, lane = u & 31, g = lane >> 2, c = lane & 3;
    const bool hi = octet < n_hi_oct;
    const int j0 = hi ? 8 * octet : n_hi + 8 * (octet - n_hi_oct);
    const int jlim = hi ? n_hi : r;
    uint32_t w = 0u;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int j = j0 + (key ? 2 * c + half : g);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = key ? g + 8 * k : 8 * k + 2 * c + half;
        const uint32_t code = j < jlim ? codes[t * r + j] : 0u;
        w |= code << (hi ? 4 * k + 16 * half : 2 * k + 8 * half);
      }
    }
    if (hi) {
      *reinterpret_cast<uint32_t*>(rec + 128 * octet + 4 * lane) = w;
    } else {
      const int lo = octet - n_hi_oct;
      const int unit = 128 * n_hi_oct + (lo < 2 * npair ? 128 * (lo >> 1) + 4 * lane + 2 * (lo & 1) : 128 * npair + 2 * lane);
      *reinterpret_cast<uint16_t*>(rec + unit) = (uint16_t)w;
    }
  }
}

__device__ __forceinline__ int latent_off(int t, int j) {
  const int octet = j >> 3, slot = j & 7;
  const int k = 2 * (t >> 4) + ((t & 15) >> 3);
  const int lane = 4 * slot + ((t & 7) >> 1);
  return 512 * octet + 16 * lane + 4 * k + 2 * (t & 1);
}

// Shared-memory scratch of one single-token append, carved from a caller's
// buffer: the group's basis rows [r][128] (first, 128-byte aligned, filled by
// the caller), block latents [32][r+1], codes [32][r], (scale, zero) [r],
// and one record.
struct AppendSmem {
  float* bas;
  float* lat;
  uint8_t* codes;
  __half2* sz;
  uint8_t* rec;
};
__host__ __device__ inline size_t append_smem_bytes(int r, int rec_bytes) {
  auto a16 = [](size_t x) { return (x + 15) / 16 * 16; };
  return a16((size_t)r * kHeadDim * 4) + a16((size_t)kBlock * (r + 1) * 4) + a16((size_t)kBlock * r) +
         a16((size_t)r * 4) + a16((size_t)rec_bytes);
}
__device__ __forceinline__ AppendSmem append_smem(uint8_t* base, int r, int rec_bytes) {
  auto a16 = [](size_t x) { return (x + 15) / 16 * 16; };
  AppendSmem s;
  size_t o = 0;
  s.bas = reinterpret_cast<float*>(base + o);
  o += a16((size_t)r * kHeadDim * 4);
  s.lat = reinterpret_cast<float*>(base + o);
  o += a16((size_t)kBlock * (r + 1) * 4);
  s.codes = base + o;
  o += a16((size_t)kBlock * r);
  s.sz = reinterpret_cast<__half2*>(base + o);
  o += a16((size_t)r * 4);
  s.rec = base + o;
  (void)rec_bytes;
  return s;
}

// Projects one token (x: this stream's D fp16 values) onto the basis rows in
// sm.bas and stores its fp32 latent in row pos of sm.lat (stride r + 1).
// Every thread of the CTA calls it.  Eight lanes compute one latent channel:
// each holds 16 entries of x and of the basis row, forms exact products and
// float-pair partial sums, and a butterfly of error-free sums combines the 8
// partials; then mu_g . V_g[:, j] (a float pair) is subtracted and the result
// rounded once to fp32.
__device__ __forceinline__ void project_token(const CacheView& cv, const __half* __restrict__ x, int pos, int grp,
                                              const AppendSmem& sm) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
  const int r = cv.r, ld = r + 1;
  float* lat = sm.lat;
  (void)tid;
  // 8 lanes per channel, 4 channels per warp and pass: lane (q, i) = (lane / 8,
  // lane % 8) holds x[d] for d = 32u + 4i + (0..3), u < 4 (conflict-free
  // 128-bit basis reads: one 8-lane phase covers all 32 banks)
  const int lq = lane >> 3, li = lane & 7;
  float xv[16];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint2 w = *reinterpret_cast<const uint2*>(x + 32 * u + 4 * li);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
    const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
    xv[4 * u] = a.x;
    xv[4 * u + 1] = a.y;
    xv[4 * u + 2] = c.x;
    xv[4 * u + 3] = c.y;
  }
  for (int j0 = 4 * warp; j0 < r; j0 += 4 * nwarps) {  // warp-uniform trip count
    const int j = j0 + lq;
    float S = 0.f, E = 0.f;
    if (j < r) {
      const float* row = sm.bas + (size_t)j * kHeadDim + 4 * li;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 v = *reinterpret_cast<const float4*>(row + 32 * u);
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float pp, pe, s2, se;
          two_prod(xv[4 * u + e], vv[e], pp, pe);
          two_sum(S, pp, s2, se);
          S = s2;
          E = __fadd_rn(E, __fadd_rn(se, pe));
        }
      }
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
      const float E2 = __shfl_xor_sync(0xffffffffu, E, o);
      float s3, err;
      two_sum(S, S2, s3, err);
      S = s3;
      E = __fadd_rn(__fadd_rn(E, E2), err);
    }
    if (li == 0 && j < r) {
      const float2 m = cv.mv[(size_t)grp * r + j];
      float a, ae;
      two_sum(S, -m.x, a, ae);
      lat[pos * ld + j] = __fadd_rn(a, __fadd_rn(__fsub_rn(E, m.y), ae));
    }
  }
}

// Largest fp16 scale of the block that token x completes at position
// kBlock - 1 of stream (b, h), computed exactly as the append will store it
// (same projection, same quantizer arithmetic), without writing anything to
// the cache.  sm.bas must hold the group's basis rows.  Every thread calls it
// and gets the result.
__device__ __forceinline__ float completed_block_max_scale(const CacheView& cv, const __half* __restrict__ x, int h,
                                                           int b, int Hkv, const AppendSmem& sm) {
  const int tid = threadIdx.x, r = cv.r, ld = r + 1;
  const long long sidx = (long long)b * Hkv + h;
  __shared__ float smax2;
  if (tid == 0) smax2 = 0.f;
  project_token(cv, x, kBlock - 1, h / cv.heads_per_group, sm);
  const float* tail = cv.tail + sidx * kBlock * r;
  for (int i = tid; i < (kBlock - 1) * r; i += blockDim.x) sm.lat[(i / r) * ld + (i % r)] = __ldcg(tail + i);
  __syncthreads();
  for (int j = tid; j < r; j += blockDim.x) {
    float mn = sm.lat[j], mx = sm.lat[j];
    for (int t = 1; t < kBlock; ++t) {
      mn = fminf(mn, sm.lat[t * ld + j]);
      mx = fmaxf(mx, sm.lat[t * ld + j]);
    }
    const float qmax = j < cv.n_hi ? 15.f : 3.f;
    const float s32 = __half2float(__float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), qmax)));
    atomicMax(reinterpret_cast<unsigned int*>(&smax2), __float_as_uint(s32));
  }
  __syncthreads();
  return smax2;
}

// Appends one token (x: this stream's D fp16 values) at position p0 of stream
// (b, h).  Every thread of the CTA calls it; sm.bas must hold the group's
// basis rows.  Returns, in every thread, the largest fp16 scale of the block
// this token completed (0 if none).
__device__ __forceinline__ float append_one_token(const CacheView& cv, const __half* __restrict__ x, long long p0, int h, int b,
                                  int Hkv, const AppendSmem& sm) {
  const int tid = threadIdx.x;
  const int r = cv.r, ld = r + 1;
  const int pos = (int)(p0 % kBlock);
  const long long blk = p0 / kBlock;
  const long long sidx = (long long)b * Hkv + h;
  if (!bounds_ok(blk < cv.n_blk_cap, cv.hdr)) return 0.f;  // (bounds-checking build; uniform over the CTA)
  float* lat = sm.lat;
  __shared__ float smax;
  if (tid == 0) smax = 0.f;
  project_token(cv, x, pos, h / cv.heads_per_group, sm);
  __syncthreads();

  if (!cv.quantize) {
    uint8_t* gdst = cv.blocks + (sidx * cv.n_blk_cap + blk) * cv.rec_bytes;
    if (pos == 0) {
      // the block opens: clear its record, so the token slots not yet
      // written (and the padding channels) hold zeros, not stale bytes
      for (int i = tid; i < cv.rec_bytes / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(gdst)[i] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
    }
    for (int j = tid; j < r; j += blockDim.x)
      *reinterpret_cast<__half*>(gdst + latent_off(pos, j)) = __float2half_rn(lat[pos * ld + j]);
    return 0.f;
  }
  float* tail = cv.tail + sidx * kBlock * r;
  if (pos < kBlock - 1) {
    for (int j = tid; j < r; j += blockDim.x) tail[pos * r + j] = lat[pos * ld + j];
    return 0.f;
  }
  // the token completes the block: quantize and pack it like a prefill block
  uint8_t* rec = sm.rec;
  for (int i = tid; i < (kBlock - 1) * r; i += blockDim.x) lat[(i / r) * ld + (i % r)] = tail[i];
  __syncthreads();
  for (int j = tid; j < r; j += blockDim.x) {
    float mn = lat[j], mx = lat[j];
    for (int t = 1; t < kBlock; ++t) {
      mn = fminf(mn, lat[t * ld + j]);
      mx = fmaxf(mx, lat[t * ld + j]);
    }
    const float qmax = j < cv.n_hi ? 15.f : 3.f;
    const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), qmax));
    const __half zh = __float2half_rn(mn);
    const float s32 = __half2float(sh), z32 = __half2float(zh);
    sm.sz[j] = __halves2half2(sh, zh);
    atomicMax(&cv.hdr->max_scale, __float_as_uint(s32));
    atomicMax(&cv.smax[sidx], __float_as_uint(s32));
    atomicMax(reinterpret_cast<unsigned int*>(&smax), __float_as_uint(s32));
    for (int t = 0; t < kBlock; ++t) {
      float q = 0.f;
      if (s32 != 0.f) q = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(lat[t * ld + j], z32), s32)), 0.f), qmax);
      sm.codes[t * r + j] = (uint8_t)q;
    }
  }
  __syncthreads();
  pack_codes(sm.codes, r, cv.role, cv.n_hi, cv.n_hi_oct, cv.n_lo_oct, rec, tid, blockDim.x);
  const int n_pad = 8 * cv.n_oct;
  const int szb = 128 * cv.n_hi_oct + 64 * cv.n_lo_oct;
  __half* r16 = reinterpret_cast<__half*>(rec + szb);
  for (int pch = tid; pch < n_pad; pch += blockDim.x) {
    const int j = padded_to_channel(pch, r, cv.n_hi, cv.n_hi_oct, 1);
    const __half2 v = j >= 0 ? sm.sz[j] : __halves2half2(__float2half(0.f), __float2half(0.f));
    if (cv.role == PALU_ROLE_KEY) {
      r16[pch] = __low2half(v);
      r16[n_pad + pch] = __high2half(v);
    } else {
      r16[2 * pch] = __low2half(v);
      r16[2 * pch + 1] = __high2half(v);
    }
  }
  __syncthreads();
  uint8_t* gdst = cv.blocks + (sidx * cv.n_blk_cap + blk) * cv.rec_bytes;
  for (int i = tid; i < cv.rec_bytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(gdst)[i] = reinterpret_cast<const uint4*>(rec)[i];
  return smax;
}

// Called by one thread of each of the n_cta CTAs that appended one token at
// p0 (their sequence's position), after its CTA's writes: the last to arrive
// advances the length(s).
__device__ __forceinline__ void publish_length(const CacheView& cv, long long p0, unsigned int n_cta) {
  __threadfence();
  const unsigned int t = atomicAdd(&cv.hdr->ticket, 1u);
  if (t == n_cta - 1) {
    if (cv.hdr->ragged) advance_ragged_lengths(cv, nullptr, 1);
    else cv.hdr->length = p0 + 1;
    cv.hdr->ticket = 0u;
    __threadfence();
  }
}

}  // namespace palu
