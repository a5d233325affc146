// Internal definitions shared by the libpalu translation units: the device
// state layout, the error plumbing and thin inline-PTX wrappers for the
// sm_103a instructions the kernels use (warp-level MMA, movmatrix, ldmatrix,
// cp.async, bulk copies with mbarrier completion).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "palu.h"

namespace palu {

constexpr int kHeadDim = 128;
constexpr int kBlock = 32;          // tokens per quantization group
constexpr int kMaxRank = 128;
constexpr int kMaxGq = 8;           // query heads per KV head (one n8 MMA tile)
constexpr int32_t kCacheMagic = 0x50414C55;  // "PALU"

// Bounded spin on an mbarrier: try_wait already suspends for a while per
// attempt, so this bounds the wait to well under a minute on any clock.
constexpr uint32_t kSpinLimit = 1u << 22;

// ---------------------------------------------------------------- state
// Device state of a cache, in one caller-owned buffer:
//   [0, 64)        header: length, error word, ticket, largest stored scale, ragged flag
//   basisT         fp32 [n_groups][rank][D]   (row j = direction j)
//   mu             fp32 [n_groups][D]
//   mv             fp32 [n_groups][rank][2]   mu_g . V_g[:, j] as a float pair (hi, lo)
//   smax           u32  [batch * kv_heads]    largest stored fp16 scale per stream
//   seq_len        i64  [batch]               tokens per sequence (ragged caches)
struct StateHeader {
  long long length;        // tokens of every sequence; with ragged lengths, the largest
  unsigned int err;
  unsigned int ticket;
  unsigned int max_scale;  // bits of the largest fp16 scale stored so far in any stream (a non-negative float)
  unsigned int ragged;     // 1: seq_len holds each sequence's own length (set by the ragged calls)
  unsigned int pad[10];
};
static_assert(sizeof(StateHeader) == 64, "state header size");

struct StateLayout {
  size_t basis_off, mu_off, mv_off, smax_off, slen_off, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// One largest-scale word per stream (batch * kv_heads) follows mv, then one
// length per sequence.
inline StateLayout state_layout(int n_groups, int rank, long long batch, long long kv_heads) {
  StateLayout s;
  s.basis_off = 256;
  s.mu_off = align_up(s.basis_off + sizeof(float) * (size_t)n_groups * rank * kHeadDim, 256);
  s.mv_off = align_up(s.mu_off + sizeof(float) * (size_t)n_groups * kHeadDim, 256);
  s.smax_off = align_up(s.mv_off + sizeof(float) * 2 * (size_t)n_groups * rank, 256);
  s.slen_off = align_up(s.smax_off + sizeof(unsigned int) * (size_t)(batch * kv_heads), 256);
  s.total = align_up(s.slen_off + sizeof(long long) * (size_t)batch, 256);
  return s;
}

// Ragged per-sequence lengths are supported up to this many sequences.
constexpr int kMaxRaggedBatch = 4096;

// Everything a kernel needs to know about one cache.
struct CacheView {
  uint8_t* blocks;
  float* tail;
  StateHeader* hdr;
  const float* basisT;   // [n_g][r][D]
  const float* mu;       // [n_g][D]
  const float2* mv;      // [n_g][r]
  unsigned int* smax;    // [batch * kv_heads] bits of each stream's largest stored fp16 scale
  long long* seq_len;    // [batch] tokens per sequence (authoritative when hdr->ragged)
  int64_t n_blk_cap;
  int64_t capacity;
  int r, n_hi, n_hi_oct, n_lo_oct, n_oct, rec_bytes;
  int heads_per_group, quantize, role, batch, kv_heads;
};

inline CacheView make_view(const palu_cache* c) {
  CacheView v;
  StateLayout s = state_layout(c->n_groups, c->rank, c->batch, c->kv_heads);
  uint8_t* st = static_cast<uint8_t*>(c->state);
  v.blocks = static_cast<uint8_t*>(c->blocks);
  v.tail = c->tail;
  v.hdr = reinterpret_cast<StateHeader*>(st);
  v.basisT = reinterpret_cast<const float*>(st + s.basis_off);
  v.mu = reinterpret_cast<const float*>(st + s.mu_off);
  v.mv = reinterpret_cast<const float2*>(st + s.mv_off);
  v.smax = reinterpret_cast<unsigned int*>(st + s.smax_off);
  v.seq_len = reinterpret_cast<long long*>(st + s.slen_off);
  v.n_blk_cap = c->n_blk_cap;
  v.capacity = c->capacity;
  v.r = c->rank;
  v.n_hi = c->n_hi;
  v.n_hi_oct = c->n_hi_oct;
  v.n_lo_oct = c->n_lo_oct;
  v.n_oct = c->n_oct;
  v.rec_bytes = c->record_bytes;
  v.heads_per_group = c->heads_per_group;
  v.quantize = c->quantize;
  v.role = c->role;
  v.batch = c->batch;
  v.kv_heads = c->kv_heads;
  return v;
}

// Tokens held by sequence b, read on the device: its own length when the
// cache has ragged lengths, else the shared one.
__device__ __forceinline__ long long seq_length(const CacheView& v, long long b) {
  return __ldcg(&v.hdr->ragged) ? __ldcg(v.seq_len + b) : __ldcg(&v.hdr->length);
}

// Ragged lengths: every sequence's length advances by its own count (counts,
// device [batch]) or by `delta` when counts is NULL; a sequence whose append
// would pass the capacity keeps its length (its CTAs wrote nothing).  The
// shared length becomes the largest.  One thread, after every CTA of the
// append has read the old lengths.
__device__ __forceinline__ void advance_ragged_lengths(const CacheView& cv, const int* counts, long long delta) {
  long long mx = 0;
  for (int b = 0; b < cv.batch; ++b) {
    const long long l0 = cv.seq_len[b];
    const long long n = counts ? (long long)counts[b] : delta;
    const long long l1 = (n >= 0 && l0 + n <= cv.capacity) ? l0 + n : l0;
    cv.seq_len[b] = l1;
    mx = l1 > mx ? l1 : mx;
  }
  cv.hdr->length = mx;
}

// Real latent channel of padded channel p (octet p/8, slot p%8), or -1 for padding.
__host__ __device__ inline int padded_to_channel(int p, int r, int n_hi, int n_hi_oct, int quantize) {
  int o = p >> 3, slot = p & 7;
  if (!quantize) return p < r ? p : -1;
  if (o < n_hi_oct) {
    int j = 8 * o + slot;
    return j < n_hi ? j : -1;
  }
  int j = n_hi + 8 * (o - n_hi_oct) + slot;
  return j < r ? j : -1;
}

// ---------------------------------------------------------------- errors
void set_error(const std::string& msg);
palu_status fail(palu_status st, const std::string& msg);
palu_status cuda_check(cudaError_t e, const char* what);
int device_sm_count();
// Sets the kernel's dynamic shared-memory limit to `smem` (once per kernel,
// smem and device) and returns its resident CTAs per SM; cached, so calls made
// while a stream is being captured issue no CUDA API calls after the first.
palu_status kernel_occupancy(const void* kernel, int threads, int smem, int* per_sm);

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// Arrive once (release semantics: this thread's earlier writes, and those of
// threads that synchronised with it before, are visible to the waiter).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; returns false if the limit (try_wait attempts) ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// D = A(16x16) * B(16x8) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 b16 matrix held in the standard fragment layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t fma_f16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Error-free product and sum in fp32 (explicit round-to-nearest intrinsics so
// the compiler can neither contract nor reassociate them).
__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
  p = __fmul_rn(a, b);
  e = __fmaf_rn(a, b, -p);
}
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void set_dev_error(StateHeader* hdr, unsigned int bit) {
  if (hdr) atomicOr(&hdr->err, bit);
}

// The bounds-checking build (compiled with -DPALU_DEBUG_BOUNDS=1, the library
// libpalu_debug.so): the kernels check the block indices of their streaming
// global accesses (the decode's record copies, the encode's record writes and
// its rows of x) against the cache's extents.  A failed check sets
// PALU_DEVERR_BOUNDS in the cache's error word and the access is skipped or
// redirected to the cache's first block, so that nothing out of range is
// touched and every wait still completes.  The default build compiles the
// checks out: bounds_ok is then constant true.
#ifndef PALU_DEBUG_BOUNDS
#define PALU_DEBUG_BOUNDS 0
#endif
template <class Header>  // a cache state header with an `unsigned int err` word
__device__ __forceinline__ bool bounds_ok(bool ok, Header* hdr) {
#if PALU_DEBUG_BOUNDS
  if (!ok && hdr) atomicOr(&hdr->err, (unsigned int)PALU_DEVERR_BOUNDS);
  return ok;
#else
  (void)ok;
  (void)hdr;
  return true;
#endif
}

}  // namespace palu
