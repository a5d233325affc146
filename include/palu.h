/*
 * libpalu — group-head low-rank latent KV cache (PALU style) for GB300 (sm_103a).
 *
 * The method (page "PALU — True Low-Rank Latent Storage for Keys and Values",
 * section "How it works"): the KV heads of a layer are split into contiguous
 * head groups; per group, keys (and separately values) of the prefill are
 * centred by their mean mu_g and projected on a shared basis V_g (D x r) from
 * a truncated SVD; the cache stores only the latent codes [S, r], mixed-bit
 * quantized per (channel, 32-token group) -- the top quarter of channels by
 * singular value at 4 bits, the rest at 2 bits -- with the asymmetric min/max
 * quantizer of the blog post "VeloxQuant-MLX 0.8.0 adds KIVI" ("What KIVI
 * is").  Single-token decode attention runs on the codes directly.
 *
 * Conventions for every call:
 *  - Pointers named as device pointers must point to memory of the current
 *    CUDA device; the caller allocates and owns all memory.  Host pointers are
 *    named as such.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous on it unless stated otherwise.
 *  - A call returns PALU_OK or an error code; palu_last_error() then gives a
 *    message for the calling thread.  Argument errors are detected on the host
 *    before anything is launched.  Conditions only the device can see (append
 *    past capacity while replaying a captured graph, a bounded wait that ran
 *    out, K/V length mismatch, eigen-solver not converged) set bits of the
 *    cache's device error word, reported by palu_cache_sync().
 *  - Supported: head_dim 128, group_size 32, hi_bit 4, lo_bit 2, rank 1..128,
 *    query heads per KV head 1..8, fp16 inputs.
 */
#ifndef PALU_H
#define PALU_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PALU_OK = 0,
  PALU_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or configuration */
  PALU_ERR_UNSUPPORTED = 2,   /* valid by the method but not built here (e.g. head_dim != 128) */
  PALU_ERR_CAPACITY = 3,      /* append beyond the cache capacity */
  PALU_ERR_NOT_INITIALIZED = 4,
  PALU_ERR_CUDA = 5,          /* a CUDA runtime call failed */
  PALU_ERR_DEVICE = 6         /* a kernel reported an error through the device error word */
} palu_status;

/* Energy reading for the rank threshold ("retain 90% of singular value
 * energy", section "Usage"): cumulative sum of singular values (default) or
 * of squared singular values. */
enum { PALU_ENERGY_SIGMA = 0, PALU_ENERGY_SIGMA2 = 1 };

/* Which tensor a cache holds; keys and values use different record layouts. */
enum { PALU_ROLE_KEY = 0, PALU_ROLE_VALUE = 1 };

/* Bits of the device error word. */
enum {
  PALU_DEVERR_CAPACITY = 1u,        /* append beyond capacity (nothing written) */
  PALU_DEVERR_TIMEOUT = 2u,         /* a bounded wait on a copy ran out */
  PALU_DEVERR_LENGTH_MISMATCH = 4u, /* key and value caches differ in length */
  PALU_DEVERR_NOT_CONVERGED = 8u,   /* eigen-solver hit its sweep limit */
  PALU_DEVERR_ROLLBACK = 16u,       /* a per-sequence rollback was refused (that sequence kept its length) */
  PALU_DEVERR_BOUNDS = 32u          /* bounds-checking build only (PALU_DEBUG_BOUNDS): a kernel found a
                                       computed block index out of range and skipped that access */
};

/* Configuration, mirroring the page's KVCacheConfig fields (section "Usage"):
 * palu_rank, palu_energy_threshold, palu_n_head_groups, palu_hi_bit,
 * palu_lo_bit, palu_hi_fraction, palu_group_size, palu_quantize_values. */
typedef struct {
  int32_t head_dim;          /* D; must be 128 */
  int32_t n_head_groups;     /* KV heads are split into this many contiguous groups */
  int32_t rank;              /* > 0: explicit rank; 0: rank from energy_threshold */
  int32_t energy_mode;       /* PALU_ENERGY_SIGMA or PALU_ENERGY_SIGMA2 */
  double energy_threshold;   /* fraction of energy retained, (0, 1] */
  double hi_fraction;        /* fraction of channels (by singular value) at hi_bit: n_hi = ceil(f*r) */
  int32_t hi_bit;            /* 4 */
  int32_t lo_bit;            /* 2 */
  int32_t group_size;        /* tokens per quantization group: 32 */
  int32_t quantize;          /* 1: mixed-bit codes; 0: fp16 latents (value caches only) */
} palu_config;

/* A cache for one tensor (K or V) of one layer.  Plain data: copying it
 * copies the description, not the device buffers.  Fill it with
 * palu_cache_init(); do not edit fields afterwards. */
typedef struct {
  int32_t magic;
  int32_t role;
  int32_t head_dim, rank, n_hi, n_groups, heads_per_group, quantize;
  int32_t batch, kv_heads;
  int32_t n_hi_oct, n_lo_oct, n_oct, record_bytes;
  int64_t capacity;          /* tokens */
  int64_t n_blk_cap;         /* 32-token block records per stream */
  void* blocks;              /* device [batch, kv_heads, n_blk_cap, record_bytes] */
  float* tail;               /* device [batch, kv_heads, 32, rank] fp32 (quantized caches) */
  void* state;               /* device state: length, error word, basis, mean */
  int64_t length;            /* tokens appended through this descriptor (host count) */
} palu_cache;

typedef struct {
  int64_t length;            /* tokens per stream */
  int32_t rank, n_hi;
  double code_bytes;         /* packed code bits of the real channels of full blocks / 8 */
  double meta_bytes;         /* fp16 scale+zero of the real channels of full blocks */
  double tail_bytes;         /* fp32 latents of the partial block (fp16 latents if unquantized) */
  double record_bytes;       /* bytes of block records in use, including channel padding */
  double basis_bytes;        /* V_g and mu_g of all groups, fp32 */
  double fp16_bytes;         /* what the [S, D] fp16 tensor would take */
  double effective_bits;     /* code bits per element: (n_hi*hi_bit + (r-n_hi)*lo_bit)/D, 16r/D unquantized */
  double bits_with_meta;     /* including scale/zero metadata */
} palu_stats;

/* Message for the last error on the calling thread ("" if none). */
const char* palu_last_error(void);

/* Library version string. */
const char* palu_version(void);

/* Fill cfg with the page's defaults: head_dim 128, 4 groups, energy
 * threshold 0.90 (sigma reading), 4/2 bits, hi_fraction 0.25, group 32,
 * quantized values. */
palu_status palu_config_default(palu_config* cfg);

/* Device workspace needed by palu_fit for x of [batch, kv_heads, seq, D]. */
palu_status palu_fit_workspace_size(const palu_config* cfg, int64_t batch, int32_t kv_heads,
                                    int64_t seq, size_t* bytes);

/* Fit the group bases of one tensor of one layer from its prefill
 * (section "How it works", prefill steps 1-3).
 *   x        device fp16 [batch, kv_heads, seq, D], contiguous, 16-byte aligned.
 *   basis    device fp32 [n_groups, D, D]: basis[g, d, j] is entry d of
 *            direction j; directions sorted by descending singular value,
 *            each with its largest-magnitude entry positive.
 *   mu       device fp32 [n_groups, D]: per-group mean of the stacked rows.
 *   eigvals  device fp64 [n_groups, D]: squared singular values, descending.
 *   rank_out host int32: r = minimum over groups of the selected rank.
 *   group_ranks host int32 [n_groups] (may be NULL): rank selected per group.
 * Rows of group g are all (batch, head in group, token) triples.  The centred
 * Gram matrix is built on tensor cores and reduced in fp64; a one-block
 * cyclic Jacobi solver diagonalises it.  This call synchronises `stream` once
 * (the rank is needed on the host to size the cache). */
palu_status palu_fit(const palu_config* cfg, const void* x, int64_t batch, int32_t kv_heads,
                     int64_t seq, void* workspace, size_t workspace_bytes, float* basis,
                     float* mu, double* eigvals, int32_t* rank_out, int32_t* group_ranks,
                     void* stream);

/* Fit n_tensors tensors of the same shape in one call (for example the keys
 * and values of every layer after a prefill): every tensor's Gram matrices
 * first, then one eigensolve launch over all their head groups (one SM per
 * group, up to 256 groups a launch), then one synchronisation of `stream`.
 * The outputs equal those of palu_fit on each tensor alone.
 *   cfgs       host [n_tensors] configurations (each its own grouping,
 *              rank rule and threshold).
 *   x, basis, mu, eigvals  host [n_tensors] arrays of device pointers, each
 *              as in palu_fit; every x[t] must hold batch x kv_heads x seq x D
 *              fp16 values (the call has only the pointers and cannot check).
 *   rank_out   host int32 [n_tensors].
 *   group_ranks host int32 [sum of n_head_groups], tensor after tensor (may
 *              be NULL).
 *   workspace  device, 256-byte aligned, at least
 *              palu_fit_batch_workspace_size bytes.
 * Errors: argument errors before any launch; PALU_ERR_DEVICE if an
 * eigensolve did not converge (the first such tensor is reported). */
palu_status palu_fit_batch_workspace_size(const palu_config* cfgs, int32_t n_tensors, int64_t batch,
                                          int32_t kv_heads, int64_t seq, size_t* bytes);
palu_status palu_fit_batch(const palu_config* cfgs, int32_t n_tensors, const void* const* x, int64_t batch,
                           int32_t kv_heads, int64_t seq, void* workspace, size_t workspace_bytes,
                           float* const* basis, float* const* mu, double* const* eigvals, int32_t* rank_out,
                           int32_t* group_ranks, void* stream);

/* Byte sizes of the three device buffers of a cache (all 256-byte aligned
 * sizes): block records, fp32 tail (0 for unquantized values) and state. */
palu_status palu_cache_size(const palu_config* cfg, int32_t role, int32_t rank, int64_t batch,
                            int32_t kv_heads, int64_t capacity, size_t* block_bytes,
                            size_t* tail_bytes, size_t* state_bytes);

/* Initialise an empty cache (length 0) on caller-owned buffers.
 *   basis    device fp32 [n_groups, D, basis_ld]; columns 0..rank-1 of each
 *            group are used (e.g. palu_fit's output with basis_ld = D).
 *   mu       device fp32 [n_groups, D].
 *   blocks, tail, state: device buffers of at least the sizes given by
 *            palu_cache_size, 256-byte aligned; tail may be NULL when the
 *            cache is unquantized.
 * The basis and mean are copied into `state`; the caller may free them after
 * the call has completed on `stream`. */
palu_status palu_cache_init(palu_cache* cache, const palu_config* cfg, int32_t role, int32_t rank,
                            int64_t batch, int32_t kv_heads, int64_t capacity, const float* basis,
                            int32_t basis_ld, const float* mu, void* blocks, void* tail,
                            void* state, void* stream);

/* Project `tokens` new tokens into the stored bases, quantize and append
 * (prefill steps 4-5 when the cache is empty; decode steps 1-2 afterwards).
 *   x  device fp16 [batch, kv_heads, tokens, D], contiguous, 16-byte aligned.
 * Latents are computed to fp32 accuracy, (x - mu_g) V_g.  A 32-token block is
 * quantized when its last token arrives; until then its latents wait
 * unquantized in the tail, so appending one token at a time stores exactly the
 * codes of one long append.  Reads and advances the device-side length, so a
 * captured graph of appends stays correct when replayed. */
palu_status palu_encode_append(palu_cache* cache, const void* x, int64_t tokens, void* stream);

/* Device workspace needed by palu_decode_attn. */
palu_status palu_decode_workspace_size(const palu_cache* k, const palu_cache* v, int32_t q_heads,
                                       size_t* bytes);

/* Single-token decode attention over the latent cache (decode step 3),
 * computed from the packed codes without reconstructing K or V:
 *   scores_t = softmax_scale * (q~ . L^K_t + q . mu^K),  q~ = q V^K
 *   out      = (sum_t p_t L^V_t / sum_t p_t) (V^V)^T + mu^V
 * over every cached token, including the one appended this step.
 *   q    device fp16 [batch, q_heads, D]; query head h reads KV head
 *        h / (q_heads / kv_heads).
 *   out  device [batch, q_heads, D], fp32 if out_fp32 else fp16.
 *   softmax_scale 0 selects 1/sqrt(D).
 *   workspace  device scratch of palu_decode_workspace_size bytes (packed
 *        query factors, per-stream tickets and partial results); no initial
 *        contents are needed.
 * k and v must have the same batch, kv_heads and length.  Two kernel
 * launches on `stream` (the query factors, then the split attention over
 * the code blocks, whose last CTA per stream merges that stream's partials);
 * calls that share a workspace must not overlap on the GPU. */
palu_status palu_decode_attn(const palu_cache* k, const palu_cache* v, const void* q,
                             int32_t q_heads, float softmax_scale, void* out, int32_t out_fp32,
                             void* workspace, size_t workspace_bytes, void* stream);

/* One decode step of one layer: append one token of k and one of v to every
 * (batch, KV head) stream (decode steps 1-2), then attend with q over every
 * cached token including the new one (decode step 3); the same results as
 * palu_encode_append(k, k_new, 1), palu_encode_append(v, v_new, 1) and
 * palu_decode_attn(k, v, q, ...) in that order.  The "fused per-step
 * pipeline" of this library: two kernel launches instead of four (the two
 * appends and the query factors share one launch).
 *   k_new, v_new  device fp16 [batch, kv_heads, D] (one token per stream).
 *   q, out, softmax_scale, out_fp32, workspace  as for palu_decode_attn
 *        (workspace of palu_decode_workspace_size bytes).
 * Errors: as palu_encode_append (capacity: PALU_ERR_CAPACITY, nothing
 * launched) and palu_decode_attn.  Updates k->length and v->length. */
palu_status palu_decode_step(palu_cache* k, palu_cache* v, const void* k_new, const void* v_new,
                             const void* q, int32_t q_heads, float softmax_scale, void* out, int32_t out_fp32,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Roll the cache back to `length` tokens (e.g. to reuse a prompt prefix or
 * drop rejected speculative tokens).  Allowed when length is a multiple of 32
 * (a block boundary) or lies inside the current partial block, i.e. whenever
 * no already-quantized block has to be reopened; 0 <= length <= current
 * length.  Sets the device-side length with a one-thread kernel, so it can be
 * captured in a graph together with appends. */
palu_status palu_cache_truncate(palu_cache* cache, int64_t length, void* stream);

/* Ragged per-sequence lengths (page "add TurboQuant KV cache compression",
 * the pull request's description and review: prompts of different lengths
 * in one batch, a restored prompt prefix, speculative rollback).  The
 * sequences of a batch keep one basis and mean per head group; a sequence's
 * KV heads share its length, and its blocks and tail follow the uniform rules
 * at its own positions.  The first ragged call switches the cache to
 * per-sequence lengths (each sequence starting from the shared one); every
 * later append, decode step and decode attention then works at each
 * sequence's own position, and decode attention of sequence b covers exactly
 * its own tokens.  Up to 4096 sequences (PALU_ERR_UNSUPPORTED beyond).
 * cache->length (host) becomes an upper bound of the longest sequence;
 * palu_cache_sync or palu_cache_lengths makes it exact (do that before
 * palu_cache_save).  Every sequence must hold at least one token when
 * attention runs.
 *
 * palu_encode_append_ragged: sequence b appends the first counts[b] of its
 *   `tokens` rows of x.
 *     x       device fp16 [batch, kv_heads, tokens, D], contiguous, 16-byte aligned.
 *     counts  device int32 [batch], each in [0, tokens] (device memory, so a
 *             captured graph can replay with new counts).
 *   A sequence whose append would pass the capacity (or whose count is out
 *   of range) writes nothing and keeps its length, and PALU_DEVERR_CAPACITY
 *   is set.  Three kernel launches on `stream`.
 * palu_cache_truncate_ragged: sequence b goes back to lengths[b] tokens
 *   (device int64 [batch]) under palu_cache_truncate's rule (no growth; for
 *   quantized caches a multiple of 32 or a length inside the current partial
 *   block); a refused sequence keeps its length and PALU_DEVERR_ROLLBACK is
 *   set.  (palu_cache_truncate on a ragged cache rolls every longer sequence
 *   back to its length, under the same rule.)
 * palu_cache_lengths: synchronises `stream` and writes each sequence's
 *   length into lengths (host int64 [batch]; the shared length for a cache
 *   without ragged lengths); refreshes cache->length. */
palu_status palu_encode_append_ragged(palu_cache* cache, const void* x, int64_t tokens, const int32_t* counts,
                                      void* stream);
palu_status palu_cache_truncate_ragged(palu_cache* cache, const int64_t* lengths, void* stream);
palu_status palu_cache_lengths(palu_cache* cache, int64_t* lengths, void* stream);

/* Cache save and restore (the prompt cache of page "add TurboQuant KV cache
 * compression", the pull request's description and review: the cache of a
 * prompt prefix saved and reused by a later request).  An image
 * holds a fixed 128-byte header, the cache's state (basis, mean, largest
 * stored scale), the records of every stream's stored blocks, and the fp32
 * tail: host memory, plain bytes.
 * palu_cache_save_size: bytes of the image of `cache` at cache->length (the
 *   host count; after graph replays call palu_cache_sync first).
 * palu_cache_save: copies the image into `host` (>= that many bytes),
 *   asynchronously on `stream` (the header is written at once; the device
 *   bytes are there when the stream has passed the call; pinned host memory
 *   makes the copies asynchronous).
 * palu_cache_restore: copies an image into `cache`, which must have been
 *   initialised with the same role, rank, head grouping, quantization, batch
 *   and kv_heads (its basis and mean are replaced by the image's) and a
 *   capacity of at least the image's length (else PALU_ERR_CAPACITY);
 *   another kind of image is refused with PALU_ERR_INVALID_ARG.  Sets
 *   cache->length and the device length, clears the device error word.
 *   The caller owns both buffers. */
palu_status palu_cache_save_size(const palu_cache* cache, size_t* bytes);
palu_status palu_cache_save(const palu_cache* cache, void* host, size_t bytes, void* stream);
palu_status palu_cache_restore(palu_cache* cache, const void* host, size_t bytes, void* stream);

/* palu_decode_attn without a caller workspace, for callers that cannot
 * allocate device memory while decoding (a plugin whose host application owns
 * every allocation, a serving loop that forbids allocation between steps, a
 * process whose device memory is reserved in full by another pool).  The
 * method's pages have no counterpart: this is a library convenience.
 *   Same arguments and results as palu_decode_attn, minus the workspace.
 *   The split-K partials live in a fixed 4 MiB device array inside the
 *   library (held on every GPU that loads it, until exit); caches whose
 *   partials need more (palu_decode_workspace_size > 4 MiB) are rejected with
 *   PALU_ERR_UNSUPPORTED and a message giving both sizes.
 *   The first call on a device looks up the array's device address with
 *   cudaGetSymbolAddress; make that first call before any stream capture.
 *   Nothing in the array needs to start at zero: each call writes every
 *   partial before reading it, and the array keeps the last call's
 *   contents.  All calls on one device share that device's copy, so calls
 *   that may overlap on the GPU (e.g. issued on different streams) race and
 *   must be serialised by the caller.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
palu_status palu_decode_attn_noalloc(const palu_cache* k, const palu_cache* v, const void* q,
                                     int32_t q_heads, float softmax_scale, void* out, int32_t out_fp32,
                                     void* stream);

/* Byte accounting of a cache (section "Evidence": compressed bytes against
 * fp16 bytes; section "Effective bit-width").  Host only. */
palu_status palu_cache_stats(const palu_cache* cache, palu_stats* stats);

/* Synchronise `stream`, read the device length and error word, update
 * cache->length and clear the error word.  Returns PALU_ERR_DEVICE (with the
 * bits in the message and in *device_error if not NULL) when it was set. */
palu_status palu_cache_sync(palu_cache* cache, uint32_t* device_error, void* stream);

/* Test hook for the device error path (the group-size guard of page "add
 * TurboQuant KV cache compression", review thread, asks for actionable
 * errors instead of silent failure; this lets a test see one without faulting
 * the GPU).  Launches one CTA that waits, with the library's bounded wait and
 * a limit of spin_limit attempts (1 .. 2^20), on a shared-memory barrier
 * that it completes itself when signal != 0 and otherwise leaves pending.
 * No copy is issued on the barrier, so nothing is in flight when the wait
 * gives up.  A wait that runs out sets PALU_DEVERR_TIMEOUT in the cache's
 * device error word, reported by palu_cache_sync().  The cache is not
 * otherwise touched.  Asynchronous on `stream`. */
palu_status palu_debug_wait_probe(palu_cache* cache, uint32_t spin_limit, int32_t signal, void* stream);

/* Comparator: plain split-K decode attention on uncompressed fp16 K and V
 * (the dense baseline the latent cache is measured against).
 *   k, v  device fp16 [batch, kv_heads, seq_cap, D]; tokens 0..seq-1 are used.
 *   q     device fp16 [batch, q_heads, D];  out as in palu_decode_attn. */
palu_status palu_fp16_decode_workspace_size(int64_t batch, int32_t kv_heads, int64_t seq_cap,
                                            int32_t q_heads, size_t* bytes);
palu_status palu_fp16_decode_attn(const void* k, const void* v, int64_t batch, int32_t kv_heads,
                                  int64_t seq, int64_t seq_cap, const void* q, int32_t q_heads,
                                  float softmax_scale, void* out, int32_t out_fp32,
                                  void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PALU_H */
