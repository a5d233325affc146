// Host side of the fused latent decode attention: launch planning and the
// C entry points.  The kernel itself (and the method it follows) is described
// in decode_kernel.cuh.
#include <math.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "decode_kernel.cuh"

namespace palu {

struct DecodePlan {
  int KC, VC;
  bool VQ;
  int ns, stage_bytes, ring_off, smem, grid, seg_max, rvp;
  size_t ws_bytes;
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
  const int rec_k = k->record_bytes, rec_v = v->record_bytes;
  pl->stage_bytes = 2 * (rec_k + rec_v);
  pl->ns = pl->stage_bytes <= 2048 ? 4 : pl->stage_bytes <= 6144 ? 3 : 2;
  pl->rvp = 8 * v->n_oct;
  pl->ring_off = (int)align_up(kDecBarOff + 8 * (kDecWarps * pl->ns + 1), 128);
  const int64_t streams = (int64_t)k->batch * k->kv_heads;
  const int sms = device_sm_count();
  // shared memory: header, then the rings, which the merges reuse; the merge
  // layout needs the partial slots per stream, which follow from the grid,
  // which follows from the occupancy
  const size_t rings = std::max((size_t)kDecWarps * pl->ns * pl->stage_bytes,
                                (size_t)kDecWarps * 8 * (2 + pl->rvp) * 4);
  int per_sm = 0;
  palu_status st = kernel_occupancy(reinterpret_cast<const void*>(pl->kern), kDecThreads,
                                    (int)(pl->ring_off + rings), &per_sm);
  if (st != PALU_OK) return st;
  int64_t grid = (int64_t)sms * std::min(per_sm, 4);
  grid = std::min<int64_t>(grid, std::max<int64_t>(streams, streams * k->n_blk_cap));
  pl->grid = (int)std::max<int64_t>(1, grid);
  const int tv_bytes = v->quantize ? kBlock * v->rank * 4 : rec_v;
  const size_t merge_fixed = (size_t)v->rank * 512 + (size_t)128 * k->rank + align_up(tv_bytes, 16) +
                             8 * kBlock * 4 + 8 * kHeadDim * 4 + 32;
  const size_t per_seg = (size_t)Gq * (2 + pl->rvp) * 4;
  pl->seg_max = (int)((pl->grid + streams - 1) / streams + 1);
  const size_t merge_budget = 200 * 1024 - (size_t)pl->ring_off;
  if (merge_fixed + pl->seg_max * per_seg > merge_budget) {
    // few streams: fewer CTAs, so that one stream's partials fit on chip
    const int64_t seg_fit = (int64_t)((merge_budget - merge_fixed) / per_seg);
    if (seg_fit < 2) return fail(PALU_ERR_UNSUPPORTED, "decode merge does not fit in shared memory");
    pl->grid = (int)std::max<int64_t>(1, std::min<int64_t>(pl->grid, streams * (seg_fit - 1)));
    pl->seg_max = (int)((pl->grid + streams - 1) / streams + 1);
  }
  const size_t merge_bytes = merge_fixed + pl->seg_max * per_seg;
  pl->smem = (int)(pl->ring_off + std::max(rings, merge_bytes));
  if (pl->smem > 227 * 1024) return fail(PALU_ERR_UNSUPPORTED, "decode shared-memory plan exceeds 227 KB");
  if (merge_bytes > rings) {
    st = kernel_occupancy(reinterpret_cast<const void*>(pl->kern), kDecThreads, pl->smem, &per_sm);
    if (st != PALU_OK) return st;
    // a smaller grid only lowers the number of partial slots a stream needs
    pl->grid = (int)std::min<int64_t>(pl->grid, (int64_t)sms * std::min(per_sm, 4));
  }
  pl->ws_bytes = align_up(sizeof(float) * (size_t)streams * pl->seg_max * Gq * (2 + pl->rvp), 256);
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
  p.out = out;
  p.ws = static_cast<float*>(workspace);
  p.out_fp32 = out_fp32;
  p.Hq = q_heads;
  p.Hkv = k->kv_heads;
  p.Gq = q_heads / k->kv_heads;
  p.rvp = pl.rvp;
  p.ns = pl.ns;
  p.stage_bytes = pl.stage_bytes;
  p.ring_off = pl.ring_off;
  p.seg_max = pl.seg_max;
  p.streams = (long long)k->batch * k->kv_heads;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)kHeadDim);
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  pl.kern<<<pl.grid, kDecThreads, pl.smem, strm>>>(p);
  return cuda_check(cudaGetLastError(), "latent_decode_kernel launch");
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
