// Comparator: split-K single-token decode attention on uncompressed fp16 K/V.
//
// This is the dense baseline the latent cache is measured against: the same
// decode attention (softmax(q K^T * scale) V, GQA query heads sharing one
// K/V read) on the [S, D] fp16 tensors the method avoids storing.  Tensor-core
// scores and weighted sums, online softmax, CTA-wide cp.async pipeline over
// 64-token tiles staged through swizzled shared memory.
#include <math.h>

#include <algorithm>

#include "splitk_attend.cuh"

namespace palu {

constexpr int kF16Warps = kSplitWarps;
constexpr int kF16Tile = kSplitTile;  // tokens per stage (16 per warp)
constexpr int kF16Stages = 3;
constexpr int kF16TileBytes = kSplitTileBytes;  // 16 KB per tensor

struct F16Params {
  const __half *k, *v, *q;
  float* ws;  // [B][Hkv][n_chunks][Gq][2 + 128]
  long long seq, seq_cap;
  int Hq, Hkv, Gq, n_chunks, tiles_per_chunk;
  float scale_log2;
};

__global__ void __launch_bounds__(32 * kF16Warps) fp16_decode_kernel(const F16Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float merge[kF16Warps][8][kSplitPartStride];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int chunk = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int Gq = p.Gq;
  const long long t0 = (long long)chunk * p.tiles_per_chunk * kF16Tile;
  const long long t1 = min(t0 + (long long)p.tiles_per_chunk * kF16Tile, p.seq);
  float* part = p.ws + (((long long)b * p.Hkv + kh) * p.n_chunks + chunk) * (long long)Gq * kSplitPartStride;
  if (t0 >= t1) {
    split_write_empty(Gq, part);
    return;
  }
  const int n_tiles = (int)((t1 - t0 + kF16Tile - 1) / kF16Tile);
  const long long stream = (long long)b * p.Hkv + kh;
  const __half* kb = p.k + stream * p.seq_cap * kHeadDim;
  const __half* vb = p.v + stream * p.seq_cap * kHeadDim;
  const uint32_t sbase = smem_addr(smem);

  auto load_tile = [&](int tile, int stage) {
    const long long tt = t0 + (long long)tile * kF16Tile;
#pragma unroll
    for (int i = 0; i < (kF16Tile * 16) / (32 * kF16Warps); ++i) {
      const int idx = tid + i * 32 * kF16Warps;
      const int row = idx >> 4, ch = idx & 15;
      const bool valid = tt + row < t1;
      const long long tok = valid ? tt + row : t0;
      const int sz = valid ? 16 : 0;
      const uint32_t dk = swz(sbase + stage * 2 * kF16TileBytes, row, ch);
      const uint32_t dv = dk + kF16TileBytes;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dk), "l"(kb + tok * kHeadDim + ch * 8),
                   "r"(sz)
                   : "memory");
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dv), "l"(vb + tok * kHeadDim + ch * 8),
                   "r"(sz)
                   : "memory");
    }
  };

  uint32_t qb[8][2];
  split_load_q(qb, p.q + ((long long)b * p.Hq + (long long)kh * Gq + g) * kHeadDim, g < Gq, c);

#pragma unroll
  for (int s = 0; s < kF16Stages - 1; ++s) {
    if (s < n_tiles) load_tile(s, s);
    cp_async_commit();
  }
  SplitState st;
  split_init(st);

  for (int tile = 0; tile < n_tiles; ++tile) {
    cp_async_wait<kF16Stages - 2>();
    __syncthreads();
    const int nxt = tile + kF16Stages - 1;
    if (nxt < n_tiles) load_tile(nxt, nxt % kF16Stages);
    cp_async_commit();
    const uint32_t kst = sbase + (tile % kF16Stages) * 2 * kF16TileBytes;
    const int r0 = 16 * warp;  // this warp's 16 tokens of the tile
    split_tile(st, qb, kst, kst + kF16TileBytes, r0, lane, t0 + (long long)tile * kF16Tile + r0, t1, p.scale_log2);
  }
  cp_async_wait<0>();
  split_write_partial(st, merge, warp, lane, Gq, part);
}

// One CTA per (KV head, batch, query head of the group); thread d: channel d.
// Launched as a programmatic dependent of the split kernel: it may start
// early and waits here for the partials.
__global__ void split_combine_kernel(const float* ws, int Hq, int Hkv, int n_chunks, void* out, int out_fp32) {
  const int kh = blockIdx.x, b = blockIdx.y, h = blockIdx.z, d = threadIdx.x;
  const int Gq = Hq / Hkv, mstride = kSplitPartStride;
  grid_dep_wait();
  const float* wp = ws + ((long long)b * Hkv + kh) * n_chunks * (long long)Gq * mstride + (long long)h * mstride;
  float M = -INFINITY;
  for (int ch = 0; ch < n_chunks; ++ch) M = fmaxf(M, wp[(long long)ch * Gq * mstride]);
  float L = 0.f, a = 0.f;
  for (int ch = 0; ch < n_chunks; ++ch) {
    const float* pc = wp + (long long)ch * Gq * mstride;
    const float m = pc[0];
    if (m == -INFINITY) continue;
    const float w = ex2f_(m - M);
    L += pc[1] * w;
    a += pc[2 + d] * w;
  }
  const long long oi = ((long long)b * Hq + (long long)kh * Gq + h) * kHeadDim + d;
  const float o = a / L;
  if (out_fp32)
    static_cast<float*>(out)[oi] = o;
  else
    static_cast<__half*>(out)[oi] = __float2half_rn(o);
}

palu_status split_combine(const float* ws, long long batch, int Hq, int Hkv, int n_chunks, void* out, int out_fp32,
                          cudaStream_t stream) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(Hkv, (unsigned)batch, Hq / Hkv);
  cfg.blockDim = dim3(kHeadDim);
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, split_combine_kernel, ws, Hq, Hkv, n_chunks, out, out_fp32),
                    "split_combine_kernel launch");
}

static int f16_chunks(int64_t batch, int32_t kv_heads, int64_t seq_cap, int* tiles_per_chunk) {
  const int smem = kF16Stages * 2 * kF16TileBytes;
  int per_sm = 1;
  kernel_occupancy(reinterpret_cast<const void*>(fp16_decode_kernel), 32 * kF16Warps, smem, &per_sm);
  const int64_t tiles = std::max<int64_t>(1, (seq_cap + kF16Tile - 1) / kF16Tile);
  const int64_t streams = batch * kv_heads;
  int64_t nch = std::max<int64_t>(1, (int64_t)device_sm_count() * per_sm / streams);
  nch = std::min(nch, tiles);
  const int64_t tpc = (tiles + nch - 1) / nch;
  *tiles_per_chunk = (int)tpc;
  return (int)((tiles + tpc - 1) / tpc);
}

}  // namespace palu

using namespace palu;

extern "C" palu_status palu_fp16_decode_workspace_size(int64_t batch, int32_t kv_heads, int64_t seq_cap,
                                                       int32_t q_heads, size_t* bytes) {
  if (batch < 1 || kv_heads < 1 || seq_cap < 1 || q_heads < 1 || q_heads % kv_heads)
    return fail(PALU_ERR_INVALID_ARG, "bad shapes");
  if (q_heads / kv_heads > kMaxGq) return fail(PALU_ERR_UNSUPPORTED, "at most 8 query heads per KV head");
  if (!bytes) return fail(PALU_ERR_INVALID_ARG, "bytes is NULL");
  int tpc;
  const int nch = f16_chunks(batch, kv_heads, seq_cap, &tpc);
  *bytes = align_up(sizeof(float) * (size_t)batch * kv_heads * nch * (q_heads / kv_heads) * (2 + kHeadDim), 256);
  return PALU_OK;
}

extern "C" palu_status palu_fp16_decode_attn(const void* k, const void* v, int64_t batch, int32_t kv_heads,
                                             int64_t seq, int64_t seq_cap, const void* q, int32_t q_heads,
                                             float softmax_scale, void* out, int32_t out_fp32, void* workspace,
                                             size_t workspace_bytes, void* stream) {
  size_t need = 0;
  palu_status st = palu_fp16_decode_workspace_size(batch, kv_heads, seq_cap, q_heads, &need);
  if (st != PALU_OK) return st;
  if (seq < 1 || seq > seq_cap) return fail(PALU_ERR_INVALID_ARG, "seq must be in [1, seq_cap]");
  if (!k || !v || !q || !out || !workspace) return fail(PALU_ERR_INVALID_ARG, "NULL pointer");
  if (((uintptr_t)k | (uintptr_t)v | (uintptr_t)q | (uintptr_t)out | (uintptr_t)workspace) & 15)
    return fail(PALU_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  if (workspace_bytes < need) return fail(PALU_ERR_INVALID_ARG, "workspace too small");
  F16Params p;
  p.k = static_cast<const __half*>(k);
  p.v = static_cast<const __half*>(v);
  p.q = static_cast<const __half*>(q);
  p.ws = static_cast<float*>(workspace);
  p.seq = seq;
  p.seq_cap = seq_cap;
  p.Hq = q_heads;
  p.Hkv = kv_heads;
  p.Gq = q_heads / kv_heads;
  p.n_chunks = f16_chunks(batch, kv_heads, seq_cap, &p.tiles_per_chunk);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)kHeadDim);
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  const int smem = kF16Stages * 2 * kF16TileBytes;
  fp16_decode_kernel<<<dim3(p.n_chunks, kv_heads, (unsigned)batch), 32 * kF16Warps, smem, strm>>>(p);
  st = cuda_check(cudaGetLastError(), "fp16_decode_kernel launch");
  if (st != PALU_OK) return st;
  return split_combine(p.ws, batch, q_heads, kv_heads, p.n_chunks, out, out_fp32, strm);
}
