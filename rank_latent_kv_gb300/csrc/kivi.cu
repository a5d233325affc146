// KIVI-2bit comparator: cache append (quantize whole blocks, keep the rest in
// an fp16 window) and split-K decode attention that dequantizes the codes
// into fp16 tiles in shared memory and runs the tensor-core core of the
// dense comparator on them.
//
// Method: blog post "VeloxQuant-MLX 0.8.0 adds KIVI", section "What KIVI is"
// (per-channel keys, per-token values, fp16 residual window, asymmetric
// min/max quantizer, 2 bits, groups of 32).
#include <math.h>

#include <algorithm>

#include "kivi.h"
#include "splitk_attend.cuh"

namespace palu {

constexpr int32_t kKiviMagic = 0x4B495649;  // "KIVI"
constexpr int kKiviHalf = 1536;             // key or value part of a record
constexpr int kKiviRecord = 2 * kKiviHalf;
constexpr int kKiviMetaOff = 1024;          // scale/zero after the 32 x 16 u16 code words
constexpr int kKiviWindowHalfs = 2 * kBlock * kHeadDim;  // per stream: keys then values
constexpr int kKiviStages = 3;
constexpr int kKiviStageBytes = 2 * kKiviRecord;  // the two blocks of a 64-token tile
constexpr int kKiviSmem = kKiviStages * kKiviStageBytes + 2 * kSplitTileBytes;
constexpr float kKiviQmax = 3.f;            // 2^2 - 1

// ---------------------------------------------------------------- append

struct KiviAppendParams {
  uint8_t* records;
  __half* window;
  const __half *k, *v;
  long long n_blk_cap, t0, T, j_first, w_first;
};

// One CTA per (completed block, stream): gather the block's 32 rows (tokens
// before t0 from the window, the rest from the input), quantize keys per
// channel and values per (token, 32-channel group), pack the record.
__global__ void __launch_bounds__(128) kivi_quantize_kernel(const KiviAppendParams p) {
  __shared__ __align__(16) __half xs[2][kBlock][kHeadDim];
  __shared__ uint8_t cs[2][kBlock][kHeadDim];
  const int tid = threadIdx.x;
  const long long s = blockIdx.y, j = p.j_first + blockIdx.x;
  for (int idx = tid; idx < 2 * kBlock * 16; idx += blockDim.x) {
    const int tsr = idx >> 9, row = (idx >> 4) & 31, ch = idx & 15;
    const long long tok = (long long)kBlock * j + row;
    const __half* src = tok < p.t0 ? p.window + (s * kKiviWindowHalfs + (tsr * kBlock + row) * kHeadDim + ch * 8)
                                   : (tsr ? p.v : p.k) + ((s * p.T + (tok - p.t0)) * kHeadDim + ch * 8);
    *reinterpret_cast<uint4*>(&xs[tsr][row][ch * 8]) = *reinterpret_cast<const uint4*>(src);
  }
  __syncthreads();
  uint8_t* rec = p.records + (s * p.n_blk_cap + j) * kKiviRecord;
  {
    // keys: one group per channel over the block's 32 tokens
    const int d = tid;
    float mn = INFINITY, mx = -INFINITY;
    for (int t = 0; t < kBlock; ++t) {
      const float x = __half2float(xs[0][t][d]);
      mn = fminf(mn, x);
      mx = fmaxf(mx, x);
    }
    const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), kKiviQmax));
    const __half zh = __float2half_rn(mn);
    const float s32 = __half2float(sh), z32 = __half2float(zh);
    for (int t = 0; t < kBlock; ++t) {
      float q = 0.f;
      if (s32 != 0.f)
        q = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(__half2float(xs[0][t][d]), z32), s32)), 0.f), kKiviQmax);
      cs[0][t][d] = (uint8_t)q;
    }
    reinterpret_cast<__half*>(rec + kKiviMetaOff)[d] = sh;
    reinterpret_cast<__half*>(rec + kKiviMetaOff + 2 * kHeadDim)[d] = zh;
  }
  {
    // values: one group per (token, 32 consecutive channels)
    const int t = tid >> 2, g = tid & 3;
    float mn = INFINITY, mx = -INFINITY;
    for (int c = 0; c < 32; ++c) {
      const float x = __half2float(xs[1][t][32 * g + c]);
      mn = fminf(mn, x);
      mx = fmaxf(mx, x);
    }
    const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), kKiviQmax));
    const __half zh = __float2half_rn(mn);
    const float s32 = __half2float(sh), z32 = __half2float(zh);
    for (int c = 0; c < 32; ++c) {
      float q = 0.f;
      if (s32 != 0.f)
        q = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(__half2float(xs[1][t][32 * g + c]), z32), s32)), 0.f), kKiviQmax);
      cs[1][t][32 * g + c] = (uint8_t)q;
    }
    *reinterpret_cast<__half2*>(rec + kKiviHalf + kKiviMetaOff + 4 * (4 * t + g)) = __halves2half2(sh, zh);
  }
  __syncthreads();
  // pack: u16 #u = (token u / 16, chunk u % 16); channel 8 ch + 2k + h at bits 2k + 8h
  for (int idx = tid; idx < 2 * 256; idx += blockDim.x) {
    const int tsr = idx >> 8, w = idx & 255;
    uint32_t word = 0;
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
      const int u = 2 * w + hw, t = u >> 4, ch = u & 15;
      uint32_t x16 = 0;
#pragma unroll
      for (int sl = 0; sl < 8; ++sl) x16 |= (uint32_t)cs[tsr][t][8 * ch + sl] << (2 * (sl >> 1) + 8 * (sl & 1));
      word |= x16 << (16 * hw);
    }
    reinterpret_cast<uint32_t*>(rec + tsr * kKiviHalf)[w] = word;
  }
}

// One CTA per stream: the appended tokens after the last completed block go
// to the window (row = token % 32).  Runs after kivi_quantize_kernel, which
// may still read the window rows of the block the append completes.
__global__ void __launch_bounds__(128) kivi_window_kernel(const KiviAppendParams p) {
  const long long s = blockIdx.x;
  const int n_rows = (int)(p.t0 + p.T - p.w_first);
  for (int idx = threadIdx.x; idx < 2 * n_rows * 16; idx += blockDim.x) {
    const int tsr = idx / (n_rows * 16), rem = idx % (n_rows * 16), ch = rem & 15;
    const long long tok = p.w_first + (rem >> 4);
    const __half* src = (tsr ? p.v : p.k) + ((s * p.T + (tok - p.t0)) * kHeadDim + ch * 8);
    __half* dst = p.window + (s * kKiviWindowHalfs + (tsr * kBlock + (int)(tok & 31)) * kHeadDim + ch * 8);
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

// ---------------------------------------------------------------- decode

struct KiviDecodeParams {
  const uint8_t* records;
  const __half* window;
  const __half* q;
  float* ws;  // [B][Hkv][n_chunks][Gq][2 + 128]
  long long n_blk_cap, seq, nblk_full;
  int win, Hq, Hkv, Gq, n_chunks, tiles_per_chunk;
  float scale_log2;
};

__device__ __forceinline__ void sts128(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Eight 2-bit codes of one (token, chunk) word -> eight fp16 code*scale+zero.
// The even channels sit in the low byte, the odd ones in the high byte: after
// spreading the high byte to bits 16..23, pair k is (y >> 2k) & 3 in each
// half; OR-ing 0x6400 (fp16 1024) makes 1024 + code exactly, and subtracting
// 1024 leaves the code, exact in fp16.  One rounding in the fused multiply-add.
__device__ __forceinline__ uint4 dequant8(uint32_t cw, const uint4& s, const uint4& z) {
  const uint32_t y = (cw & 0xFFu) | ((cw & 0xFF00u) << 8);
  const uint32_t magic = 0x64006400u;
  uint4 o;
  o.x = fma_f16x2(sub_f16x2((y & 0x00030003u) | magic, magic), s.x, z.x);
  o.y = fma_f16x2(sub_f16x2(((y >> 2) & 0x00030003u) | magic, magic), s.y, z.y);
  o.z = fma_f16x2(sub_f16x2(((y >> 4) & 0x00030003u) | magic, magic), s.z, z.z);
  o.w = fma_f16x2(sub_f16x2(((y >> 6) & 0x00030003u) | magic, magic), s.w, z.w);
  return o;
}

static_assert(sizeof(float) * kSplitWarps * 8 * kSplitPartStride <= kKiviStages * kKiviStageBytes,
              "the warp merge area fits in the stage buffers");

__global__ void __launch_bounds__(32 * kSplitWarps, 4) kivi_decode_kernel(const KiviDecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int chunk = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int Gq = p.Gq;
  const long long t0 = (long long)chunk * p.tiles_per_chunk * kSplitTile;
  const long long t1 = min(t0 + (long long)p.tiles_per_chunk * kSplitTile, p.seq);
  float* part = p.ws + (((long long)b * p.Hkv + kh) * p.n_chunks + chunk) * (long long)Gq * kSplitPartStride;
  if (t0 >= t1) {
    split_write_empty(Gq, part);
    return;
  }
  const int n_tiles = (int)((t1 - t0 + kSplitTile - 1) / kSplitTile);
  const long long stream = (long long)b * p.Hkv + kh;
  const uint8_t* rb = p.records + stream * p.n_blk_cap * kKiviRecord;
  const __half* wb = p.window + stream * kKiviWindowHalfs;
  const uint32_t kt = smem_addr(smem + kKiviStages * kKiviStageBytes), vt = kt + kSplitTileBytes;

  // the records of the tile's two blocks (those that are stored) -> stage
  auto load_stage = [&](int tile, int stage) {
    const long long jb = (t0 + (long long)tile * kSplitTile) / kBlock;
#pragma unroll
    for (int i = 0; i < kKiviStageBytes / 16 / (32 * kSplitWarps); ++i) {
      const int idx = tid + i * 32 * kSplitWarps;
      const int h = idx / (kKiviRecord / 16), off = (idx % (kKiviRecord / 16)) * 16;
      const long long j = jb + h;
      if (j < p.nblk_full) cp_async16(smem + stage * kKiviStageBytes + h * kKiviRecord + off, rb + j * kKiviRecord + off);
    }
  };

  uint32_t qb[8][2];
  split_load_q(qb, p.q + ((long long)b * p.Hq + (long long)kh * Gq + g) * kHeadDim, g < Gq, c);

#pragma unroll
  for (int s = 0; s < kKiviStages - 1; ++s) {
    if (s < n_tiles) load_stage(s, s);
    cp_async_commit();
  }
  SplitState st;
  split_init(st);
  const int ch = tid & 15, rq = tid >> 4;  // dequantization: chunk, first row

  for (int tile = 0; tile < n_tiles; ++tile) {
    cp_async_wait<kKiviStages - 2>();
    __syncthreads();  // the stage has landed; every warp is done with the previous tile's K/V
    const int nxt = tile + kKiviStages - 1;
    if (nxt < n_tiles) load_stage(nxt, nxt % kKiviStages);
    cp_async_commit();
    const long long jb = (t0 + (long long)tile * kSplitTile) / kBlock;
    const uint8_t* sb = smem + (tile % kKiviStages) * kKiviStageBytes;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const long long j = jb + h;
      const uint8_t* rec = sb + h * kKiviRecord;
      if (j < p.nblk_full) {
        const uint4 ks = *reinterpret_cast<const uint4*>(rec + kKiviMetaOff + 16 * ch);
        const uint4 kz = *reinterpret_cast<const uint4*>(rec + kKiviMetaOff + 2 * kHeadDim + 16 * ch);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rb_ = rq + 8 * i, row = kBlock * h + rb_;
          const uint32_t cwk = *reinterpret_cast<const uint16_t*>(rec + 2 * (16 * rb_ + ch));
          sts128(swz(kt, row, ch), dequant8(cwk, ks, kz));
          const uint32_t cwv = *reinterpret_cast<const uint16_t*>(rec + kKiviHalf + 2 * (16 * rb_ + ch));
          const uint32_t m = *reinterpret_cast<const uint32_t*>(rec + kKiviHalf + kKiviMetaOff + 4 * (4 * rb_ + (ch >> 2)));
          const uint32_t s2 = __byte_perm(m, 0u, 0x1010), z2 = __byte_perm(m, 0u, 0x3232);
          sts128(swz(vt, row, ch), dequant8(cwv, make_uint4(s2, s2, s2, s2), make_uint4(z2, z2, z2, z2)));
        }
      } else {
        // the window block (rows past the window are zero), or no block at all
        const int n_win = (j == p.nblk_full) ? p.win : 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rb_ = rq + 8 * i, row = kBlock * h + rb_;
          uint4 kk = make_uint4(0u, 0u, 0u, 0u), vv = kk;
          if (rb_ < n_win) {
            kk = *reinterpret_cast<const uint4*>(wb + rb_ * kHeadDim + 8 * ch);
            vv = *reinterpret_cast<const uint4*>(wb + (kBlock + rb_) * kHeadDim + 8 * ch);
          }
          sts128(swz(kt, row, ch), kk);
          sts128(swz(vt, row, ch), vv);
        }
      }
    }
    __syncthreads();  // the tile's K/V are in shared memory
    const int r0 = 16 * warp;
    split_tile(st, qb, kt, vt, r0, lane, t0 + (long long)tile * kSplitTile + r0, t1, p.scale_log2);
  }
  cp_async_wait<0>();
  // every stage was consumed in the loop (no copy is in flight) and the last
  // tile's dequantization ended before the barrier above: the stage buffers
  // are free for the warps' merge
  split_write_partial(st, reinterpret_cast<float (*)[8][kSplitPartStride]>(smem), warp, lane, Gq, part);
}

static palu_status kivi_chunks(long long batch, int kv_heads, long long seq, int* n_chunks, int* tiles_per_chunk) {
  int per_sm = 1;
  palu_status st =
      kernel_occupancy(reinterpret_cast<const void*>(kivi_decode_kernel), 32 * kSplitWarps, kKiviSmem, &per_sm);
  if (st != PALU_OK) return st;
  const long long tiles = std::max<long long>(1, (seq + kSplitTile - 1) / kSplitTile);
  const long long streams = batch * kv_heads;
  long long nch = std::max<long long>(1, (long long)device_sm_count() * std::max(per_sm, 1) / streams);
  nch = std::min(nch, tiles);
  const long long tpc = (tiles + nch - 1) / nch;
  *tiles_per_chunk = (int)tpc;
  *n_chunks = (int)((tiles + tpc - 1) / tpc);
  return PALU_OK;
}

static palu_status check_kivi(const palu_kivi_cache* c) {
  if (!c) return fail(PALU_ERR_INVALID_ARG, "cache is NULL");
  if (c->magic != kKiviMagic) return fail(PALU_ERR_NOT_INITIALIZED, "KIVI cache not initialised (palu_kivi_cache_init)");
  return PALU_OK;
}

}  // namespace palu

using namespace palu;

extern "C" palu_status palu_kivi_cache_size(int64_t batch, int32_t kv_heads, int64_t capacity, size_t* record_bytes,
                                            size_t* window_bytes) {
  if (batch < 1 || kv_heads < 1 || capacity < 1) return fail(PALU_ERR_INVALID_ARG, "batch, kv_heads and capacity must be >= 1");
  if (!record_bytes || !window_bytes) return fail(PALU_ERR_INVALID_ARG, "NULL output pointer");
  const size_t streams = (size_t)batch * (size_t)kv_heads;
  *record_bytes = align_up(streams * (size_t)(capacity / kBlock) * kKiviRecord, 256);
  *window_bytes = align_up(streams * kKiviWindowHalfs * sizeof(__half), 256);
  return PALU_OK;
}

extern "C" palu_status palu_kivi_cache_init(palu_kivi_cache* cache, int64_t batch, int32_t kv_heads, int64_t capacity,
                                            void* records, void* window) {
  if (!cache) return fail(PALU_ERR_INVALID_ARG, "cache is NULL");
  size_t rb = 0, wb = 0;
  palu_status st = palu_kivi_cache_size(batch, kv_heads, capacity, &rb, &wb);
  if (st != PALU_OK) return st;
  if (batch > 65535) return fail(PALU_ERR_UNSUPPORTED, "batch must be <= 65535");
  if (batch * kv_heads > 65535) return fail(PALU_ERR_UNSUPPORTED, "batch * kv_heads must be <= 65535");
  if (!window || (rb > 0 && !records)) return fail(PALU_ERR_INVALID_ARG, "NULL buffer");
  if (((uintptr_t)records | (uintptr_t)window) & 15) return fail(PALU_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  cache->magic = kKiviMagic;
  cache->batch = (int32_t)batch;
  cache->kv_heads = kv_heads;
  cache->bits = 2;
  cache->capacity = capacity;
  cache->n_blk_cap = capacity / kBlock;
  cache->records = records;
  cache->window = window;
  cache->length = 0;
  return PALU_OK;
}

extern "C" palu_status palu_kivi_append(palu_kivi_cache* cache, const void* k, const void* v, int64_t tokens,
                                        void* stream) {
  palu_status st = check_kivi(cache);
  if (st != PALU_OK) return st;
  if (tokens < 0) return fail(PALU_ERR_INVALID_ARG, "tokens must be >= 0");
  if (tokens == 0) return PALU_OK;
  if (!k || !v) return fail(PALU_ERR_INVALID_ARG, "k or v is NULL");
  if (((uintptr_t)k | (uintptr_t)v) & 15) return fail(PALU_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  if (cache->length + tokens > cache->capacity)
    return fail(PALU_ERR_CAPACITY, "append of " + std::to_string(tokens) + " tokens to a KIVI cache holding " +
                                       std::to_string(cache->length) + " of " + std::to_string(cache->capacity));
  KiviAppendParams p;
  p.records = static_cast<uint8_t*>(cache->records);
  p.window = static_cast<__half*>(cache->window);
  p.k = static_cast<const __half*>(k);
  p.v = static_cast<const __half*>(v);
  p.n_blk_cap = cache->n_blk_cap;
  p.t0 = cache->length;
  p.T = tokens;
  const long long t_end = p.t0 + tokens;
  p.j_first = p.t0 / kBlock;
  p.w_first = std::max<long long>(p.t0, t_end / kBlock * kBlock);
  const long long n_complete = t_end / kBlock - p.t0 / kBlock;
  const unsigned streams = (unsigned)((long long)cache->batch * cache->kv_heads);
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  if (n_complete > 0) {
    kivi_quantize_kernel<<<dim3((unsigned)n_complete, streams), 128, 0, strm>>>(p);
    st = cuda_check(cudaGetLastError(), "kivi_quantize_kernel launch");
    if (st != PALU_OK) return st;
  }
  if (t_end % kBlock) {
    kivi_window_kernel<<<streams, 128, 0, strm>>>(p);
    st = cuda_check(cudaGetLastError(), "kivi_window_kernel launch");
    if (st != PALU_OK) return st;
  }
  cache->length = t_end;
  return PALU_OK;
}

extern "C" palu_status palu_kivi_decode_workspace_size(const palu_kivi_cache* cache, int32_t q_heads, size_t* bytes) {
  palu_status st = check_kivi(cache);
  if (st != PALU_OK) return st;
  if (!bytes) return fail(PALU_ERR_INVALID_ARG, "bytes is NULL");
  if (q_heads < 1 || q_heads % cache->kv_heads) return fail(PALU_ERR_INVALID_ARG, "q_heads must be a multiple of kv_heads");
  if (q_heads / cache->kv_heads > kMaxGq) return fail(PALU_ERR_UNSUPPORTED, "at most 8 query heads per KV head");
  int nch = 1, tpc = 1;
  st = kivi_chunks(cache->batch, cache->kv_heads, cache->capacity, &nch, &tpc);
  if (st != PALU_OK) return st;
  *bytes = align_up(sizeof(float) * (size_t)cache->batch * cache->kv_heads * nch * (q_heads / cache->kv_heads) *
                        kSplitPartStride,
                    256);
  return PALU_OK;
}

extern "C" palu_status palu_kivi_decode_attn(const palu_kivi_cache* cache, const void* q, int32_t q_heads,
                                             float softmax_scale, void* out, int32_t out_fp32, void* workspace,
                                             size_t workspace_bytes, void* stream) {
  palu_status st = check_kivi(cache);
  if (st != PALU_OK) return st;
  if (cache->length < 1) return fail(PALU_ERR_INVALID_ARG, "the KIVI cache is empty");
  if (!q || !out || !workspace) return fail(PALU_ERR_INVALID_ARG, "NULL pointer");
  if (((uintptr_t)q | (uintptr_t)out | (uintptr_t)workspace) & 15)
    return fail(PALU_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  size_t need = 0;
  st = palu_kivi_decode_workspace_size(cache, q_heads, &need);
  if (st != PALU_OK) return st;
  if (workspace_bytes < need) return fail(PALU_ERR_INVALID_ARG, "workspace too small");
  KiviDecodeParams p;
  p.records = static_cast<const uint8_t*>(cache->records);
  p.window = static_cast<const __half*>(cache->window);
  p.q = static_cast<const __half*>(q);
  p.ws = static_cast<float*>(workspace);
  p.n_blk_cap = cache->n_blk_cap;
  p.seq = cache->length;
  p.nblk_full = cache->length / kBlock;
  p.win = (int)(cache->length % kBlock);
  p.Hq = q_heads;
  p.Hkv = cache->kv_heads;
  p.Gq = q_heads / cache->kv_heads;
  st = kivi_chunks(cache->batch, cache->kv_heads, cache->length, &p.n_chunks, &p.tiles_per_chunk);
  if (st != PALU_OK) return st;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)kHeadDim);
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  kivi_decode_kernel<<<dim3(p.n_chunks, cache->kv_heads, (unsigned)cache->batch), 32 * kSplitWarps, kKiviSmem, strm>>>(p);
  st = cuda_check(cudaGetLastError(), "kivi_decode_kernel launch");
  if (st != PALU_OK) return st;
  return split_combine(p.ws, cache->batch, q_heads, cache->kv_heads, p.n_chunks, out, out_fp32, strm);
}
