/*
 * KIVI-2bit KV cache and its decode attention: the compressed comparator the
 * latent cache is measured against, beside the dense fp16 one in palu.h.
 *
 * The method (blog post "VeloxQuant-MLX 0.8.0 adds KIVI", section "What KIVI
 * is"; its usage example sets 2 bits, group size 32, residual length 32):
 * keys are quantized per channel -- one fp16 (scale, zero) per (channel,
 * 32-token group) -- and values per token -- one per (token, 32-channel
 * group) -- with the asymmetric min/max quantizer
 *     zero = min(g), scale = (max(g) - min(g)) / 3, code = round((g - zero) / scale)
 * and the most recent tokens are kept exactly in an fp16 window.  Reading of
 * the window: a key group needs 32 whole tokens, so a 32-token block is
 * quantized (keys and values together) when its 32nd token arrives; the
 * window holds the tokens after the last complete block (0..31 of them).
 *
 * Conventions are those of palu.h (status codes, palu_last_error(), caller-
 * owned device memory, asynchronous calls on `stream`, argument errors
 * reported before anything is launched).  Supported: head_dim 128, 2-bit
 * codes, query heads per KV head 1..8, fp16 inputs.
 */
#ifndef PALU_KIVI_H
#define PALU_KIVI_H

#include "palu.h"

#ifdef __cplusplus
extern "C" {
#endif

/* A KIVI cache of one layer (keys and values together).  Plain data: fill it
 * with palu_kivi_cache_init(); do not edit fields afterwards.
 * Block record of stream s = (b, kv head), block j (3072 bytes at
 * records + (s * n_blk_cap + j) * 3072): the key part, then the value part,
 * 1536 bytes each:
 *   codes  one little-endian u16 per (token t, 8-channel chunk c) at byte
 *          2 (16 t + c); channel 8c + 2k + h (k 0..3, h 0..1) at bits 2k + 8h.
 *   keys   then fp16 scale[128] and fp16 zero[128] (one per channel).
 *   values then one fp16 (scale, zero) pair per (token t, 32-channel group g)
 *          at byte 1024 + 4 (4 t + g) of the value part.
 * Window of stream s: fp16 [2 (keys, values)][32][128] at window + s * 16384
 * bytes; rows 0 .. length % 32 - 1 hold the tokens after the last block. */
typedef struct {
  int32_t magic;
  int32_t batch, kv_heads;
  int32_t bits;               /* 2 */
  int64_t capacity;           /* tokens per stream */
  int64_t n_blk_cap;          /* block records per stream: capacity / 32 */
  void* records;              /* device [batch, kv_heads, n_blk_cap, 3072] bytes */
  void* window;               /* device [batch, kv_heads, 2, 32, 128] fp16 */
  int64_t length;             /* tokens per stream (host count) */
} palu_kivi_cache;

/* Byte sizes (multiples of 256) of the records and window buffers. */
palu_status palu_kivi_cache_size(int64_t batch, int32_t kv_heads, int64_t capacity, size_t* record_bytes,
                                 size_t* window_bytes);

/* Describe an empty cache (length 0) on caller-owned device buffers of at
 * least palu_kivi_cache_size bytes, 16-byte aligned.  Launches nothing. */
palu_status palu_kivi_cache_init(palu_kivi_cache* cache, int64_t batch, int32_t kv_heads, int64_t capacity,
                                 void* records, void* window);

/* Append `tokens` tokens of keys and values to every stream.
 *   k, v  device fp16 [batch, kv_heads, tokens, 128], contiguous, 16-byte aligned.
 * Every block completed by the append is quantized (scale and zero rounded to
 * fp16, codes computed in fp32 against the rounded values, round half to
 * even, clamped to 0..3; a zero scale gives code 0) and written as a record;
 * the remaining tokens go to the window.  Appending one token at a time stores
 * exactly what one long append stores.  PALU_ERR_CAPACITY (nothing launched)
 * past the capacity.  One or two kernel launches; advances cache->length. */
palu_status palu_kivi_append(palu_kivi_cache* cache, const void* k, const void* v, int64_t tokens, void* stream);

/* Device workspace needed by palu_kivi_decode_attn (sized for any length up
 * to the capacity). */
palu_status palu_kivi_decode_workspace_size(const palu_kivi_cache* cache, int32_t q_heads, size_t* bytes);

/* Single-token decode attention over the cache's cache->length tokens:
 *   out = softmax(softmax_scale * q K_hat^T) V_hat
 * with K_hat = code * scale + zero per channel group, V_hat likewise per
 * token group, and the window's rows as stored.  The codes are dequantized
 * to fp16 inside the kernel (one rounding of code * scale + zero) and never
 * written back.
 *   q    device fp16 [batch, q_heads, 128]; query head h reads KV head
 *        h / (q_heads / kv_heads).
 *   out  device [batch, q_heads, 128], fp32 if out_fp32 else fp16.
 *   softmax_scale 0 selects 1/sqrt(128).
 *   workspace  device scratch of palu_kivi_decode_workspace_size bytes.
 * The cache must hold at least one token.  Two kernel launches (split
 * attention over the blocks, then the merge of the splits). */
palu_status palu_kivi_decode_attn(const palu_kivi_cache* cache, const void* q, int32_t q_heads, float softmax_scale,
                                  void* out, int32_t out_fp32, void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PALU_KIVI_H */
