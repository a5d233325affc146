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
  float (*qt_s)[kHeadDim];
  float *red_s, *cq_s;
};
constexpr size_t kQprepSmemBytes = sizeof(float) * (8 * kHeadDim + kHeadDim + 8 * kHeadDim + 16);
__device__ __forceinline__ QprepSmem qprep_smem(uint8_t* base) {
  QprepSmem s;
  float* f = reinterpret_cast<float*>(base);
  s.q_s = reinterpret_cast<float(*)[kHeadDim]>(f);
  s.mu_s = f + 8 * kHeadDim;
  s.qt_s = reinterpret_cast<float(*)[kHeadDim]>(f + 9 * kHeadDim);
  s.red_s = f + 17 * kHeadDim;
  s.cq_s = s.red_s + 8;
  return s;
}

// Stream X's q-prep by a 256-thread CTA.  max_s_floor: a scale the stream's
// blocks may hold that its largest-scale word need not show yet (the largest
// of a block this step completes).  bas_s: the group's key basis rows [r][128] in shared
// memory, if the caller holds them (else they are read from global memory).
// q~ is one pass per 32 padded key channels: 8 lanes per channel, each with
// 16 entries of the basis row (d = 4i + 32u, conflict-free 128-bit reads)
// and of every query head, a 3-level butterfly for the 8 heads' sums.
__device__ void qprep_stream(const DecodeParams& p, long long X, float max_s_floor, const QprepSmem& sm,
                             const float* bas_s = nullptr) {
  float (*q_s)[kHeadDim] = sm.q_s;
  float* mu_s = sm.mu_s;
  float (*qt_s)[kHeadDim] = sm.qt_s;
  float* red_s = sm.red_s;
  float* cq_s = sm.cq_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = (int)(X / p.Hkv), kh = (int)(X % p.Hkv), Gq = p.Gq;
  const int gk = kh / p.k.heads_per_group;
  const int npch = 8 * p.k.n_oct;
  const float* basis_g = p.k.basisT + (size_t)gk * p.k.r * kHeadDim;
  // the stream's own largest stored scale: no other stream's append moves it
  const float max_s = fmaxf(__uint_as_float(__ldcg(&p.k.smax[X])), max_s_floor);
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
  __syncthreads();
  float amax = 0.f;
  const int jq = tid >> 3, li = tid & 7;
  for (int ch = 0; ch < npch; ch += 32) {
    const int pch = ch + jq;
    const int j = pch < npch ? padded_to_channel(pch, p.k.r, p.k.n_hi, p.k.n_hi_oct, 1) : -1;
    float acc[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) acc[h] = 0.f;
    if (j >= 0) {
      const float* row = (bas_s ? bas_s : basis_g) + (size_t)j * kHeadDim + 4 * li;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 v = bas_s ? *reinterpret_cast<const float4*>(row + 32 * u)
                               : __ldg(reinterpret_cast<const float4*>(row + 32 * u));
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const float4 q4 = *reinterpret_cast<const float4*>(&q_s[h][4 * li + 32 * u]);
          acc[h] = fmaf(q4.x, v.x, fmaf(q4.y, v.y, fmaf(q4.z, v.z, fmaf(q4.w, v.w, acc[h]))));
        }
      }
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1)
#pragma unroll
      for (int h = 0; h < 8; ++h) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], o);
    if (li == 0 && pch < npch) {
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float qt = h < Gq ? acc[h] * p.scale_log2 : 0.f;
        qt_s[h][pch] = qt;
        amax = fmaxf(amax, fabsf(qt));
      }
    }
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
  // scaled q~ and c for the tail tokens; the stream's ticket starts at zero
  for (int i = tid; i < 8 * kHeadDim; i += 256) p.qt[(size_t)X * 8 * kHeadDim + i] = qt_s[i >> 7][i & (kHeadDim - 1)];
  if (tid < 8) p.cq[(size_t)X * 8 + tid] = cq_s[tid];
  if (tid == 0) p.tickets[X] = 0u;
  if (tid == 0 && X == 0) p.tickets[p.streams] = 0u;
  // prescale 2^e with |q~| 2^e max(1, largest stored scale) < 2^14, and the
  // per-lane fp16 hi/lo factors: thread (lane l, octet o)
  amax = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) amax = fmaxf(amax, red_s[w]);
  const float xm = amax * fmaxf(1.f, max_s);
  int e = 0;
  if (xm > 0.f) {
    const int ex = (int)((__float_as_uint(xm) >> 23) & 0xFF) - 126;  // xm < 2^ex
    e = min(max(14 - ex, -120), 120);
  }
  const float two_e = pow2i(e), inv2e = pow2i(-e);
  const int g = lane >> 2, c = lane & 3, ko = p.qp_ko;
  uint32_t* qp = p.qpack + ((size_t)X * 32 + lane) * p.qp_stride;
  for (int o = warp; o < ko; o += 8) {
    const float x0 = 8 * o + 2 * c < kHeadDim ? qt_s[g][8 * o + 2 * c] * two_e : 0.f;
    const float x1 = 8 * o + 2 * c + 1 < kHeadDim ? qt_s[g][8 * o + 2 * c + 1] * two_e : 0.f;
    const uint32_t hi = pack_f16x2(x0, x1);
    const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    qp[o] = hi;
    qp[ko + o] = pack_f16x2(x0 - hf.x, x1 - hf.y);
  }
  if (warp == 0) {
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
// One decode step's work before attention (the fused per-step pipeline), in
// one launch: grid (streams, 3).  CTA (X, 0) appends stream X's new key
// token, CTA (X, 1) the new value token, CTA (X, 2) prepares stream X's
// query factors; the three run side by side.  The stored lengths
// stay as they were: the decode launch that follows advances them.
// Launched as a programmatic dependent: the basis rows, which no launch
// writes, are fetched before waiting for the preceding launch.  The q-prep
// recomputes the largest scale of a block this step completes (exactly as
// the key append stores it) instead of waiting for the append, so the
// result is the same as that of the separate calls.
__global__ void __launch_bounds__(256) latent_step_prologue_kernel(const DecodeParams p, const __half* k_new,
                                                                   const __half* v_new) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ uint64_t bar;
  const int tid = threadIdx.x;
  const long long X = blockIdx.x;
  const int role = blockIdx.y;  // 0 key append, 1 value append, 2 q-prep
  const CacheView& cv = role == 1 ? p.v : p.k;
  const int h = (int)(X % p.Hkv), b = (int)(X / p.Hkv);
  const AppendSmem sm = append_smem(dsm, cv.r, cv.rec_bytes);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, (uint32_t)cv.r * 512u);
    bulk_g2s(sm.bas, cv.basisT + (size_t)(h / cv.heads_per_group) * cv.r * kHeadDim, (uint32_t)cv.r * 512u, &bar);
  }
  grid_dep_wait();
  grid_dep_launch();
  const long long p0 = seq_length(cv, b);  // this sequence's position
  __syncthreads();
  const bool got = mbar_wait_bounded(&bar, 0);
  if (!got && tid == 0) set_dev_error(cv.hdr, PALU_DEVERR_TIMEOUT);
  if (role == 2) {
    // a block this step completes holds scales the header may not show yet:
    // the q-prep takes them from the same arithmetic the key append runs
    float s_floor = 0.f;
    if (p0 + 1 <= cv.capacity && p0 % kBlock == kBlock - 1)
      s_floor = completed_block_max_scale(cv, k_new + X * kHeadDim, h, b, p.Hkv, sm);
    __syncthreads();
    qprep_stream(p, X, s_floor, qprep_smem(dsm + append_smem_bytes(cv.r, cv.rec_bytes)), sm.bas);
    return;
  }
  if (p0 + 1 > cv.capacity) {
    if (X == 0 && tid == 0) set_dev_error(cv.hdr, PALU_DEVERR_CAPACITY);
  } else {
    append_one_token(cv, (role == 0 ? k_new : v_new) + X * kHeadDim, p0, h, b, p.Hkv, sm);
  }
}

struct DecodePlan {
  int KC, VC;
  bool VQ;
  int nw, ns, stage_bytes, ring_off, wp_off, end_off, end_off2, smem, grid, seg_max, rvp, qp_ko, qp_stride;
  size_t qpack_off, qt_off, cq_off, tick_off, part_off, ws_bytes;
  DecodeKernel kern;
};

// The decode kernel for the records' octet counts; *ko: the key octets it
// holds per lane (the q-prep's packing).
static DecodeKernel pick_kernel(int ke, int ve, int kc, int vc, bool vq, int* ko) {
  *ko = ke;
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
  if (DecodeKernel kw = decode_kernel_wide(ke, ve, kc, vc, vq)) return kw;
  *ko = 4 * kc;
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
  pl->kern = pick_kernel(k->n_oct, v->n_oct, pl->KC, pl->VC, pl->VQ, &pl->qp_ko);
  if (!pl->kern) return fail(PALU_ERR_UNSUPPORTED, "no decode kernel for this rank");
  pl->qp_stride = (2 * pl->qp_ko + 4 + 3) / 4 * 4;
  const int rec_k = k->record_bytes, rec_v = v->record_bytes;
  pl->stage_bytes = 2 * (rec_k + rec_v);
  pl->ns = pl->stage_bytes <= 2048 ? 4 : pl->stage_bytes <= 6144 ? 3 : 2;
  pl->rvp = 8 * v->n_oct;
  const int64_t streams = (int64_t)k->batch * k->kv_heads;
  const int sms = device_sm_count();
  // the end phase reuses the rings when they are large enough
  const EndLayout el = end_layout(k->rank, v->rank, v->quantize, rec_v);
  // one CTA per SM with as many warps as the kernel's registers allow (16
  // for the exact-octet kernels, 12 for the per-class ones) when the rings
  // fit: every warp of an SM then has the same scheduling age, and their
  // ranges end together; else 8
  const bool exact = k->n_oct <= 8 && v->n_oct <= 8;
  for (int nw = exact ? kMaxDecWarps : kClassDecWarps; nw >= 8; nw = nw > 8 ? 8 : 0) {
    pl->nw = nw;
    pl->ring_off = (int)align_up(kDecBarOff + 8 * (nw * pl->ns + 2), 128);
    const size_t rings = (size_t)nw * pl->ns * pl->stage_bytes;
    pl->wp_off = (int)align_up(pl->ring_off + rings, 16);
    const size_t wp_end = pl->wp_off + (size_t)nw * 2 * Gq * (kPartHead + pl->rvp) * 4;
    pl->end_off = (size_t)el.bytes <= rings ? pl->ring_off : (int)align_up(wp_end, 16);
    pl->smem = (int)std::max(wp_end, (size_t)pl->end_off + el.bytes);
    // a second end area inside the rings, for a CTA that finishes two streams at once
    const size_t el16 = align_up(el.bytes, 16);
    pl->end_off2 = (nw == kMaxDecWarps && 2 * el16 <= rings) ? (int)(pl->ring_off + el16) : -1;
    if (pl->smem <= 227 * 1024) break;
  }
  if (pl->smem > 227 * 1024) return fail(PALU_ERR_UNSUPPORTED, "decode shared-memory plan exceeds 227 KB");
  int per_sm = 0;
  palu_status st = kernel_occupancy(reinterpret_cast<const void*>(pl->kern), 32 * pl->nw, pl->smem, &per_sm);
  if (st != PALU_OK) return st;
  int64_t grid = (int64_t)sms * std::min(per_sm, 4);
  grid = std::min<int64_t>(grid, std::max<int64_t>(1, streams * k->n_blk_cap));
  // at least one warp per stream, so that no warp's range spans more than two
  // streams (extra CTAs, if any, simply run in a second wave)
  grid = std::max<int64_t>(grid, (streams + pl->nw - 1) / pl->nw);
  pl->grid = (int)std::max<int64_t>(1, grid);
  // CTAs that touch one stream: at most ceil(CTAs / streams) + 1
  pl->seg_max = (int)((pl->grid + streams - 1) / streams + 1);
  // workspace: packed query factors, q~ and c per stream, tickets, partials
  pl->qpack_off = 0;
  pl->qt_off = align_up(pl->qpack_off + sizeof(uint32_t) * (size_t)streams * 32 * pl->qp_stride, 256);
  pl->cq_off = align_up(pl->qt_off + sizeof(float) * (size_t)streams * 8 * kHeadDim, 256);
  pl->tick_off = align_up(pl->cq_off + sizeof(float) * (size_t)streams * 8, 256);
  pl->part_off = align_up(pl->tick_off + sizeof(uint32_t) * (size_t)(streams + 1), 256);
  pl->ws_bytes = align_up(pl->part_off + sizeof(float) * (size_t)streams * pl->seg_max * Gq * kOutPart, 256);
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
  p.tickets = reinterpret_cast<uint32_t*>(ws + pl.tick_off);
  p.out_fp32 = out_fp32;
  p.Hq = q_heads;
  p.Hkv = k->kv_heads;
  p.Gq = q_heads / k->kv_heads;
  p.rvp = pl.rvp;
  p.ns = pl.ns;
  p.stage_bytes = pl.stage_bytes;
  p.ring_off = pl.ring_off;
  p.wp_off = pl.wp_off;
  p.end_off = pl.end_off;
  p.end_off2 = pl.end_off2;
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

// The decode kernel, started while its predecessor finishes (programmatic
// dependent launch; it waits in-kernel for the query factors).
static palu_status launch_decode(const DecodePlan& pl, const DecodeParams& p, cudaStream_t strm) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(32 * pl.nw);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = strm;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, pl.kern, p), "latent_decode_kernel launch");
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
  return launch_decode(pl, p, strm);
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
  const size_t smem = std::max(append_smem_bytes(v->rank, v->record_bytes),
                               append_smem_bytes(k->rank, k->record_bytes) + kQprepSmemBytes);
  int per_sm = 0;
  st = kernel_occupancy(reinterpret_cast<const void*>(latent_step_prologue_kernel), 256, (int)smem, &per_sm);
  if (st != PALU_OK) return st;
  {
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned int)p.streams, 3);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = strm;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    st = cuda_check(cudaLaunchKernelEx(&cfg, latent_step_prologue_kernel, p, static_cast<const __half*>(k_new),
                                       static_cast<const __half*>(v_new)),
                    "latent_step_prologue_kernel launch");
  }
  if (st != PALU_OK) return st;
  k->length += 1;
  v->length += 1;
  return launch_decode(pl, p, strm);
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
