/*
 * libpalu — the SVDq keys-only low-rank cache (page "veloxquant_mlx.cache.
 * svdq_cache module", section "Design"), for GB300 (sm_103a).
 *
 * Keys of each KV head are centred by the head's own mean and projected on
 * the head's own basis (rank r_h, from an explicit rank or the energy
 * threshold 0.95), then quantized per (channel, 32-token group) with the
 * asymmetric min/max quantizer at the width the bit schedule
 * (8, 4, 2, 1, 1, 0, 0, 0) gives the channel's group of equal contiguous
 * channel groups (most significant first; a 0-bit channel is not stored and
 * reads back as 0).  Values are not compressed: they stay fp16, in the
 * caller's own buffer.  Decode attention runs on the key codes directly:
 * scores q . K_t = q~ . L_t + q . mean with q~ = q V_h, as
 * sum_j code_tj (q~_j s_j) + (q . mean + sum_j q~_j z_j): the codes exact,
 * q~_j s_j as an fp16 hi/lo pair (about 22 significant bits), fp32
 * accumulation; the zero term and the partial block's fp32 latents in fp32.
 *
 * The per-head fit is palu_fit with n_head_groups = kv_heads (one head per
 * group); its group ranks are the per-head ranks, and its basis [kv_heads,
 * D, D] and mean [kv_heads, D] are the inputs of palu_svdq_cache_init.
 *
 * Conventions as in palu.h: caller-owned device memory, asynchronous calls on
 * `stream`, host argument checks, a device error word (capacity, bounded
 * wait) reported by palu_svdq_sync.
 *
 * Block record of a (batch, head, 32-token block), a storage format of this
 * library (the page fixes the widths; the bit order is the LSB-first packing
 * of blog post "How I built VeloxQuant-MLX", "The Bit-Packing Problem"): the
 * kept channels' codes, channel after channel, token t of a b-bit channel at
 * bit t*b of the channel's 4*b bytes; then one fp16 (scale, zero) pair per
 * kept channel; records of all heads share one 16-byte multiple stride.
 */
#ifndef PALU_SVDQ_H
#define PALU_SVDQ_H

#include "palu.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t magic;
  int32_t batch, kv_heads, r_max, record_bytes;
  int32_t pad0;
  int64_t capacity;          /* tokens */
  int64_t n_blk_cap;         /* 32-token block records per stream */
  void* blocks;              /* device [batch, kv_heads, n_blk_cap, record_bytes] */
  float* tail;               /* device [batch, kv_heads, 32, r_max] fp32: latents of the partial block */
  void* state;               /* device: header, per-head tables, bases, means */
  int64_t length;            /* tokens appended (host count) */
} palu_svdq_cache;

/* Byte sizes of the cache's three device buffers for per-head ranks
 * (host int32 [kv_heads], each in 1..128). */
palu_status palu_svdq_cache_size(int64_t batch, int32_t kv_heads, const int32_t* ranks, int64_t capacity,
                                 size_t* block_bytes, size_t* tail_bytes, size_t* state_bytes);

/* Initialise an empty cache on caller-owned buffers (256-byte aligned, at
 * least the sizes above).
 *   ranks   host int32 [kv_heads]: head h keeps columns 0..ranks[h]-1.
 *   basis   device fp32 [kv_heads, D, basis_ld] (palu_fit's basis with one
 *           head per group: basis_ld = D); mu device fp32 [kv_heads, D].
 * The bases and means are copied into `state`. */
palu_status palu_svdq_cache_init(palu_svdq_cache* cache, int64_t batch, int32_t kv_heads, const int32_t* ranks,
                                 int64_t capacity, const float* basis, int32_t basis_ld, const float* mu,
                                 void* blocks, void* tail, void* state, void* stream);

/* Project, quantize and append `tokens` keys (prefill steps 1-4 when empty,
 * decode steps 1-2 afterwards): k device fp16 [batch, kv_heads, tokens, D],
 * 16-byte aligned.  Latents are the fp32 rounding of (k - mean_h) V_h; a
 * 32-token block is quantized when its last token arrives, until then its
 * latents wait in the fp32 tail (so appends of any sizes store the codes of
 * one long append).  Two kernel launches. */
palu_status palu_svdq_append(palu_svdq_cache* cache, const void* k, int64_t tokens, void* stream);

/* Device workspace for palu_svdq_decode_attn. */
palu_status palu_svdq_decode_workspace_size(const palu_svdq_cache* cache, int32_t q_heads, size_t* bytes);

/* Single-token decode attention (decode step 3): every cached token of each
 * stream, keys from the codes (and the fp32 tail), values from v.
 *   v     device fp16 [batch, kv_heads, v_cap, D]: tokens 0..length-1 are used.
 *   q     device fp16 [batch, q_heads, D]; query head h reads KV head
 *         h / (q_heads / kv_heads) (at most 8 per KV head).
 *   out   device [batch, q_heads, D], fp32 if out_fp32 else fp16.
 * Two kernel launches: split attention (each CTA forms its stream's query
 * factors), then the combine. */
palu_status palu_svdq_decode_attn(const palu_svdq_cache* cache, const void* v, int64_t v_cap, const void* q,
                                  int32_t q_heads, float softmax_scale, void* out, int32_t out_fp32,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Synchronise, refresh cache->length from the device and report and clear
 * the device error word (PALU_ERR_DEVICE with the bits in *device_error). */
palu_status palu_svdq_sync(palu_svdq_cache* cache, uint32_t* device_error, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PALU_SVDQ_H */
