/*
 * kvc.h -- C ABI of the static KV-cache decode library (libkvc.so, sm_103a).
 *
 * The library implements one decode step over a KV cache that is allocated
 * once, at full capacity, and never reallocated:
 *
 *   1. kvc_append: write the new token's K and V rows into the fixed buffer
 *      at cache_index (slice assignment, never concatenation);
 *   2. kvc_decode_attn: one query row per head attends over every live cache
 *      row, softmax(q K^T / sqrt(d_head)) V, with each KV head shared by
 *      n_heads / n_kv_heads query heads (grouped-query attention).
 *
 * Sources for the operations:
 *   - "KV-Cache Mechanics" (DantinoX docs), AR Static KV-Cache: the cache is
 *     pre-allocated at model construction with shape
 *     [B, H_kv, max_context, head_size] per layer; prefill writes at
 *     cache_index 0, each decode step at cache_index = tokens so far.
 *   - "KV Cache Optimization: GQA Audit, In-Place Buffers, Persistent
 *     Prompts", #2 In-place KV cache updates (After): append slice-assigns
 *     rows [valid, valid + T_new) of one [B, H, capacity, D] buffer per K and
 *     V; reads are sliced to the live length so padded rows are not attended.
 *     #1 GQA-aware KV cache audit: K/V are stored with n_kv_heads heads.
 *   - "10.3 -- KV cache implementation details", section 5 (the decode loop,
 *     step-by-step): append k_t, v_t to the layer's cache, then attention of
 *     the single query row against the entire cache -- "the only place the
 *     cache is read"; section 4.2: GQA shares each KV head across
 *     n_heads / g query heads; sections 2 and 4.4: the cache-size formula.
 *
 * Conventions for every call:
 *   - All tensors are dense, row-major, innermost dimension contiguous, in
 *     the cache's element type (kvc_dtype).  Device pointers are CUDA device
 *     memory of the device that was current at kvc_alloc; host pointers are
 *     marked "host".
 *   - The caller owns every buffer (cache, inputs, outputs, workspace).  The
 *     library owns only the kvc_cache handle; it never allocates device
 *     memory and never frees caller memory.
 *   - Calls that take a stream enqueue asynchronously on it (stream is a
 *     cudaStream_t passed as void*; NULL means the legacy default stream).
 *     Their return value reports only errors detectable on the host before
 *     launch; nothing is enqueued when it is not KVC_OK.  Errors that depend
 *     on device-resident values (cache_index, valid_len) are recorded in a
 *     device error word inside the workspace and read with kvc_get_error.
 *   - The library is stateless with respect to sequence lengths: the caller
 *     tracks them (passing cache_index to append and valid_len to attention)
 *     exactly as the optimisation note's KVCache tracks validLengths.
 *     Rewinding a sequence is lowering its length on the caller's side.
 *   - Calls on one handle that overlap on the GPU (different streams without
 *     ordering) race on the workspace; order them on one stream.
 *   - Every kernel is launched with programmatic stream serialization: its
 *     set-up may overlap the previous kernel on the stream, and it touches no
 *     global memory before that kernel has completed and its writes are
 *     visible, so stream order holds as for ordinary launches.  A kernel the
 *     caller launches right after a library call with the same attribute, and
 *     that does not wait (griddepcontrol.wait) itself, may start before the
 *     library's kernel has finished.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVC_ABI_VERSION 1

/* Status codes.  KVC_OK is 0; every other value is an error. */
typedef enum {
    KVC_OK = 0,
    KVC_ERR_INVALID = 1,      /* bad argument: null pointer, shape, layer, dtype */
    KVC_ERR_CAPACITY = 2,     /* an append would pass max_context */
    KVC_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    KVC_ERR_WORKSPACE = 4,    /* workspace missing or smaller than kvc_workspace_bytes */
    KVC_ERR_TIMEOUT = 5,      /* a bounded wait inside a kernel gave up (device word) */
    KVC_ERR_DEVICE_INDEX = 6, /* a device-resident cache_index / valid_len was out of range */
    KVC_ERR_UNSUPPORTED = 7,  /* configuration outside the compiled kernel set */
    KVC_ERR_ALIGNMENT = 8     /* a pointer is not 16-byte aligned */
} kvc_status;

/* Element type of the cache, of q / k_new / v_new, and of the output.
 * Bytes per element p: bf16 2, fp32 4, fp16 2 ("10.3", section 2). */
/* KVC_INT8: an int8 cache ("10.3", section 4.4: the cache stored as int8,
 * p = 1 byte per element) with one fp32 scale per cache row (one token of
 * one KV head), held in two caller-owned scale arrays bound by
 * kvc_alloc_scaled.  A row of d_h values x is stored as
 * code = rint(x * (127 / absmax)) in [-127, 127] with scale = absmax / 127
 * (fp32 arithmetic, round half to even; scale 0 for a row of zeros), and the
 * attention reads code * scale.  The activations of such a cache -- q, out,
 * k_new, v_new -- are bf16.  Built for d_h = 128. */
typedef enum { KVC_BF16 = 0, KVC_FP32 = 1, KVC_FP16 = 2, KVC_INT8 = 3 } kvc_dtype;

/* Model shape of one static cache.
 *   n_layers     L, number of per-layer caches held in one allocation
 *   batch        B, sequences
 *   n_heads      H, query heads
 *   n_kv_heads   H_kv, KV heads; must divide H (g = H / H_kv query heads share one)
 *   d_head       d_h, head width: 32, 64, 128 or 256
 *   max_context  T_max, rows allocated per (layer, sequence, KV head)
 *   dtype        kvc_dtype
 * Supported head groups g = n_heads / n_kv_heads: 1 to 8 for every cache
 * type and head width; 16, 32 and 64 (multi-query attention, "10.3" section
 * 4.1: one KV head shared by all query heads, g = n_heads) for 16-bit caches
 * (KVC_BF16, KVC_FP16) with d_head 64 or 128. */
typedef struct {
    int32_t n_layers;
    int32_t batch;
    int32_t n_heads;
    int32_t n_kv_heads;
    int32_t d_head;
    int32_t max_context;
    int32_t dtype;
} kvc_config;

typedef struct kvc_cache kvc_cache; /* opaque handle */

/* ---- host-only queries (no GPU needed) -------------------------------- */

/* Library ABI version (KVC_ABI_VERSION). */
int32_t kvc_abi_version(void);

/* Human-readable name of a status code; never NULL. */
const char *kvc_status_str(int32_t status);

/* Check a configuration on the host: KVC_OK, KVC_ERR_INVALID (nonsense
 * shape) or KVC_ERR_UNSUPPORTED (no compiled kernel for it). */
kvc_status kvc_check_config(const kvc_config *cfg);

/* Bytes of the whole static cache, K and V, all layers:
 *   2 * n_layers * n_kv_heads * d_head * max_context * batch * p
 * ("10.3", section 2 boxed formula with n_kv_heads as in section 4.4; the
 * "Key-value cache" lesson record's payload estimate).  0 if cfg is invalid. */
uint64_t kvc_cache_bytes(const kvc_config *cfg);

/* Growth of one sequence's cache per token: 2 * n_layers * n_kv_heads *
 * d_head * p ("10.3", section 2.2; lesson record "per token per sequence").
 * 0 if cfg is invalid. */
uint64_t kvc_bytes_per_token(const kvc_config *cfg);

/* Bytes of device workspace kvc_alloc needs for cfg: split partials
 * (max, sum, accumulator per split of each sequence/KV head/query head),
 * one counter per (sequence, KV head), and the device error word.
 * 0 if cfg is invalid.  The workspace starts with the int32 error word at
 * byte 0 and the int32 arrival counters [B * H_kv] at byte 256 (for
 * diagnostics; the rest of its layout is private). */
uint64_t kvc_workspace_bytes(const kvc_config *cfg);

/* Bytes of ONE of the two scale arrays of an int8 cache: one fp32 per row,
 * n_layers * batch * n_kv_heads * max_context * 4, laid out [L, B, H_kv,
 * T_max].  0 for other cache types or an invalid cfg.  (The cache-size
 * formula, kvc_cache_bytes, counts the codes only, as the pages do.) */
uint64_t kvc_scale_bytes(const kvc_config *cfg);

/* ---- handle -------------------------------------------------------------- */

/* Bind caller-owned device buffers to a new handle.
 *   k_base, v_base  device, each n_layers * batch * n_kv_heads * max_context
 *                   * d_head elements, laid out [L, B, H_kv, T_max, d_h]
 *                   (layer l's cache starts at element
 *                   l * B * H_kv * T_max * d_h); 16-byte aligned.
 *   workspace       device, ws_bytes >= kvc_workspace_bytes(cfg); 16-byte
 *                   aligned.  kvc_alloc zeroes it (synchronously); it must
 *                   not be used for anything else while the handle lives.
 *   out             host; receives the handle on KVC_OK, untouched otherwise.
 * Uses the current CUDA device; later calls must run with it current.
 * Returns KVC_ERR_INVALID / _UNSUPPORTED / _ALIGNMENT / _WORKSPACE / _CUDA. */
/* kvc_alloc for int8 caches (cfg->dtype == KVC_INT8): k_base and v_base
 * hold the codes (one byte per element, same layout as above) and k_scale,
 * v_scale (device, kvc_scale_bytes(cfg) each, 16-byte aligned) the per-row
 * fp32 scales.  The other arguments, and the errors, are kvc_alloc's;
 * KVC_ERR_INVALID for another dtype or a missing scale array.  kvc_alloc
 * itself refuses KVC_INT8 (KVC_ERR_INVALID). */
kvc_status kvc_alloc_scaled(const kvc_config *cfg, void *k_base, void *v_base, void *k_scale,
                            void *v_scale, void *workspace, uint64_t ws_bytes, kvc_cache **out);

/* ---- paged caches ----------------------------------------------------------- */

/* Bytes of ONE pool of a paged cache with num_blocks physical blocks per
 * layer: n_layers * num_blocks * n_kv_heads * 16 * d_head elements.  0 for an
 * invalid cfg or num_blocks <= 0 (and for int8 caches, which are not paged). */
uint64_t kvc_pool_bytes(const kvc_config *cfg, int32_t num_blocks);

/* A paged cache ("10.3", section 7, PagedAttention: the cache allocated in
 * fixed-size blocks of 16 tokens, made logically contiguous by a block
 * table).  Per layer, K and V each live in a pool of num_blocks physical
 * blocks, laid out [L, num_blocks, H_kv, 16, d_h] (layer l's pool starts at
 * element l * num_blocks * H_kv * 16 * d_h); block_table (device, int32
 * [B, max_context / 16], caller-owned, shared by the layers) maps logical
 * block j of sequence b to a physical block, so token p of sequence b lives in
 * block block_table[b, p / 16] at slot p % 16.  The caller may change the
 * table between calls (it is read at every launch; blocks may be shared
 * read-only between sequences).  kvc_append and kvc_decode_step write through
 * the table, kvc_decode_attn and kvc_decode_step read through it; rows past a
 * sequence's live length are never read.  A table entry outside
 * [0, num_blocks) is recorded as KVC_ERR_DEVICE_INDEX and its rows are
 * neither read nor written.  cfg->max_context must be a multiple of 16.
 * Built for 16-bit caches with head groups of 2 to 8, 16, 32 or 64 and d_h of 64 or 128
 * (KVC_ERR_UNSUPPORTED otherwise); kvc_prefill_attn returns
 * KVC_ERR_UNSUPPORTED on a paged handle.  Other arguments and errors as for
 * kvc_alloc. */
kvc_status kvc_alloc_paged(const kvc_config *cfg, void *k_pool, void *v_pool, int32_t num_blocks,
                           const int32_t *block_table, void *workspace, uint64_t ws_bytes,
                           kvc_cache **out);

kvc_status kvc_alloc(const kvc_config *cfg, void *k_base, void *v_base,
                     void *workspace, uint64_t ws_bytes, kvc_cache **out);

/* Release the handle (host memory only).  Caller buffers stay untouched.
 * NULL is accepted. */
void kvc_free(kvc_cache *h);

/* Override the number of context splits (CTAs) of kvc_decode_attn: 0 restores
 * the automatic choice, otherwise 1..1024.  Results agree across split
 * counts up to fp32 rounding. */
kvc_status kvc_set_num_splits(kvc_cache *h, int32_t n);

/* Limit, in nanoseconds of GPU wall time, of one wait inside the decode
 * kernels: the wait of a sequence's last context split for the partial
 * results the other splits publish (the split combine, which has no
 * counterpart on the pages).  0 restores the default of 1 s.  When
 * the limit runs out the kernel records KVC_ERR_TIMEOUT in the device error
 * word, abandons the launch (its output rows are undefined) and returns;
 * kvc_get_error then reports it and resets the split counters, after which
 * the handle works normally again.  Every other wait (the copies into shared
 * memory, and the drain of copies in flight before a block exits) keeps the
 * 1 s default, so no block ever exits with a copy still landing.  A short
 * limit is meant for diagnostics: under load the other splits may
 * legitimately take longer than it. */
kvc_status kvc_set_wait_timeout_ns(kvc_cache *h, uint64_t ns);

/* ---- the decode step ------------------------------------------------------ */

/* In-place append ("KV Cache Optimization...", #2 After; "10.3", section 5:
 * "Append k_t, v_t to the layer's KV cache"):
 *   K_l[b, j, cache_index[b] + t, :] = k_new[b, j, t, :]   for t < T_new
 * and the same for V, for every sequence b and KV head j.  A pure byte copy;
 * no other cache row is written.
 *   layer        0 <= layer < n_layers
 *   k_new, v_new device, [B, H_kv, T_new, d_h], 16-byte aligned
 *   cache_index  device int32 [B]: write position of each sequence (its live
 *                length before the append).  A sequence whose
 *                cache_index[b] < 0 or cache_index[b] + T_new > max_context is
 *                skipped and KVC_ERR_DEVICE_INDEX is recorded.
 *   T_new        rows per sequence, 0 <= T_new <= max_context (0: no-op)
 * For an int8 cache k_new / v_new are bf16 and each row is quantised as it
 * is written (codes and the row's scale; see KVC_INT8).
 * Host errors: KVC_ERR_INVALID, KVC_ERR_CAPACITY (T_new > max_context),
 * KVC_ERR_ALIGNMENT, KVC_ERR_CUDA. */
kvc_status kvc_append(kvc_cache *h, int32_t layer, const void *k_new,
                      const void *v_new, const int32_t *cache_index,
                      int32_t T_new, void *stream);

/* Single-query decode attention ("10.3", section 5, attention bullet):
 *   out[b, i, :] = softmax_j( q[b, i, :] . K_l[b, i / g, j, :] / sqrt(d_h) )
 *                  . V_l[b, i / g, j, :]       over j < valid_len[b]
 * with g = n_heads / n_kv_heads (query head i reads KV head i / g, the
 * contiguous grouping).  Rows at or past valid_len[b] never reach the
 * output: the 16-bit and fp32 kernels never read them; on an int8 cache a
 * ragged last tile may be copied whole (codes of up to 127 rows past
 * valid_len[b], within max_context), and those codes are discarded
 * unused (their scales are never read).
 * Arithmetic: fp32 products and accumulation, one round-to-nearest-even to
 * the cache type at the end.
 *   layer           0 <= layer < n_layers
 *   q               device, [B, H, d_h], 16-byte aligned
 *   valid_len       device int32 [B]: live rows of each sequence, counting
 *                   this step's appended row.  A sequence with valid_len[b]
 *                   < 1 or > max_context is skipped (its output rows are left
 *                   unwritten) and KVC_ERR_DEVICE_INDEX is recorded.
 *   max_valid_hint  host; 0, or an upper bound on valid_len used only to size
 *                   the launch without a device-to-host read.
 *   out             device, [B, H, d_h]
 * Host errors: KVC_ERR_INVALID, KVC_ERR_ALIGNMENT, KVC_ERR_CUDA. */
kvc_status kvc_decode_attn(kvc_cache *h, int32_t layer, const void *q,
                           const int32_t *valid_len, int32_t max_valid_hint,
                           void *out, void *stream);

/* One whole decode step of one layer ("10.3", section 5, the decode loop:
 * append k_t, v_t to the layer's cache, then attend with the single query
 * row over the entire cache): for every sequence b the new rows go to
 * position valid_len[b] - 1, then the attention of kvc_decode_attn runs over
 * rows [0, valid_len[b]).  The result equals kvc_append(h, layer, k_new,
 * v_new, valid_len[b] - 1, T_new = 1) followed by kvc_decode_attn with the
 * same arguments: the cache bytes are identical and the output agrees to
 * fp32 rounding.  It is one launch, which reads the new rows straight from
 * k_new / v_new (an int8 cache: quantises them, with the codes and scale
 * kvc_append would write) while it streams the older ones, and stores them
 * into the cache.
 *   layer, q, max_valid_hint, out   as for kvc_decode_attn
 *   k_new, v_new    device, [B, H_kv, 1, d_h], 16-byte aligned
 *   valid_len       device int32 [B]: live rows after this step's append.  A
 *                   sequence with valid_len[b] < 1 or > max_context gets no
 *                   append and no output, and KVC_ERR_DEVICE_INDEX is
 *                   recorded.
 * Host errors: KVC_ERR_INVALID, KVC_ERR_ALIGNMENT, KVC_ERR_CUDA. */
kvc_status kvc_decode_step(kvc_cache *h, int32_t layer, const void *q,
                           const void *k_new, const void *v_new,
                           const int32_t *valid_len, int32_t max_valid_hint,
                           void *out, void *stream);

/* ---- chunked prefill ------------------------------------------------------ */

/* Causal attention of a chunk of T_new new tokens per sequence over the static
 * cache ("KV-Cache Mechanics", AR Static KV-Cache: prefill fills the cache from
 * cache_index, decoding continues from there; "10.3", section 3, prefill vs.
 * decode).  The chunk's K and V rows must already be in the cache at rows
 * [cache_index[b], cache_index[b] + T_new) (kvc_append with the same
 * cache_index and T_new).  For every sequence b, query head i and chunk
 * position t:
 *   out[b, i, t, :] = softmax_j( q[b, i, t, :] . K_l[b, i / g, j, :] / sqrt(d_h) )
 *                     . V_l[b, i / g, j, :]     over j <= cache_index[b] + t
 * i.e. the decode attention of each chunk token over the rows up to and
 * including its own (the pages leave the mask implicit; causal is the reading
 * under which one pass, chunks and decode steps agree).  Rows past a token's
 * own position are never read.  Arithmetic: fp32 products and accumulation,
 * one round-to-nearest-even to the cache type.  Built for 16-bit caches with
 * d_h of 64 or 128 (KVC_ERR_UNSUPPORTED otherwise).
 *   layer        0 <= layer < n_layers
 *   q            device, [B, H, T_new, d_h], 16-byte aligned
 *   cache_index  device int32 [B]: row of each sequence's first chunk token.
 *                A sequence with cache_index[b] < 0 or cache_index[b] + T_new
 *                > max_context is skipped (output rows unwritten) and
 *                KVC_ERR_DEVICE_INDEX is recorded.
 *   T_new        chunk length, 0 <= T_new <= max_context (0: no-op)
 *   out          device, [B, H, T_new, d_h]
 * Host errors: KVC_ERR_INVALID, KVC_ERR_CAPACITY, KVC_ERR_UNSUPPORTED,
 * KVC_ERR_ALIGNMENT, KVC_ERR_CUDA. */
kvc_status kvc_prefill_attn(kvc_cache *h, int32_t layer, const void *q,
                            const int32_t *cache_index, int32_t T_new,
                            void *out, void *stream);

/* ---- decode without any device allocation ------------------------------- */

/* Size of the library's built-in scratch array used by kvc_decode_attn_static:
 * 4 MiB of device memory, held on every GPU that loads the library until the
 * process exits. */
#define KVC_STATIC_SCRATCH_BYTES (4u * 1024u * 1024u)

/* The pages have no counterpart to this call; it exists for users of the
 * library, not for the method.
 *
 * Same attention as kvc_decode_attn, for callers that cannot allocate device
 * memory: code whose device memory is owned by someone else (a host framework
 * that budgets every byte itself, a plugin interface that passes only the
 * tensors of the call) can neither call cudaMalloc nor hand the library the
 * workspace that kvc_alloc binds.  This call needs no handle and no
 * workspace: it keeps the split partials and per-(sequence, KV head)
 * counters in a fixed array compiled into the library
 * (KVC_STATIC_SCRATCH_BYTES) and allocates nothing.
 *   cfg             host; the cache shape, as for kvc_alloc
 *   layer           0 <= layer < cfg->n_layers
 *   k_base, v_base  device caches laid out as for kvc_alloc, 16-byte aligned
 *   q, valid_len, max_valid_hint, out, stream   as for kvc_decode_attn
 * Returns KVC_ERR_WORKSPACE when the configuration needs more scratch than
 * the array holds (about (152 + B*H_kv) * (H/H_kv) * (d_head + 2) * 4 bytes
 * on a 152-SM GPU); KVC_ERR_INVALID, _ALIGNMENT, _UNSUPPORTED, _CUDA as
 * kvc_decode_attn.
 * The first call on a device does a one-time set-up there (looks up the
 * array's device address and the device limits); make that first call before
 * any stream capture.  Every call shares the one array and clears its
 * counters on the stream first, so calls that overlap on the GPU (streams
 * without ordering between them) race; order them on one stream.  A sequence
 * with valid_len[b] outside [1, max_context] is skipped (its output rows are
 * left unwritten).  This call has no handle: errors found on the device
 * (KVC_ERR_DEVICE_INDEX, KVC_ERR_TIMEOUT) go to the array's own error word,
 * which kvc_static_get_error reads and clears; it keeps the first error until
 * then. */
kvc_status kvc_decode_attn_static(const kvc_config *cfg, int32_t layer,
                                  const void *k_base, const void *v_base,
                                  const void *q, const int32_t *valid_len,
                                  int32_t max_valid_hint, void *out, void *stream);

/* The error word of the scratch array that kvc_decode_attn_static uses on the
 * current device (no counterpart on the pages, like that call): synchronise
 * the stream, then read and clear the word.  KVC_OK if no such call recorded
 * an error since the last read, otherwise the first recorded code:
 * KVC_ERR_DEVICE_INDEX (a valid_len outside [1, max_context]; that sequence
 * was skipped) or KVC_ERR_TIMEOUT (a bounded wait gave up; that call's
 * output is undefined, and the next call clears the split counters it may
 * have left set).  The word is shared by every such call on the device, so
 * read it between calls to tell them apart.  Allocates nothing.
 * KVC_ERR_CUDA if the synchronisation or the copy fails. */
kvc_status kvc_static_get_error(void *stream);

/* Synchronise the stream, then read and clear the device error word.
 * Returns KVC_OK if no kernel recorded an error since the last call,
 * otherwise the first recorded code (KVC_ERR_DEVICE_INDEX or
 * KVC_ERR_TIMEOUT).  After KVC_ERR_TIMEOUT the split counters are reset too.
 * KVC_ERR_CUDA if the synchronisation or the copy fails. */
kvc_status kvc_get_error(kvc_cache *h, void *stream);

/* ---- MLA latent cache --------------------------------------------------- */

/* "10.3 -- KV cache implementation details", section 4.3 (Multi-head Latent
 * Attention): the cache holds one latent vector c of width d_latent per token
 * -- a single tensor, no separate K and V -- and head h rebuilds its key and
 * value rows from it by up-projections, k = W_UK[h] c and v = W_UV[h] c with
 * W_UK[h], W_UV[h] of shape [d_head, d_latent].  Decode attention is
 *   out[b, h] = sum_t softmax_t(q[b, h] . k_t / sqrt(d_head)) v_t
 * over the live rows t < valid_len[b].  The library evaluates it in the
 * absorbed order -- q~ = W_UK[h]^T q (rounded once to the cache type),
 * attention of q~ over the latents, W_UV[h] applied to the attended latent
 * (folded over the splits in fp32, then rounded once to the cache type for
 * the tensor-core product) -- reading every latent row once for all heads.
 * Size: n_layers * d_latent * max_context * batch * p bytes ("10.3" §4.3).
 *
 * Shapes the kernels take: KVC_BF16 or KVC_FP16, n_heads 8, 16, or a
 * multiple of 16 up to 128 (taken 16 heads per CTA, the head groups of one
 * split side by side in the grid so that they read its latent rows from
 * memory once between them), d_latent 128, 256 or 512, d_head 16..256 in
 * multiples of 16; others are KVC_ERR_UNSUPPORTED.  Conventions (ownership, streams, device error word)
 * as for the calls above. */
typedef struct {
    int32_t n_layers;
    int32_t batch;
    int32_t n_heads;
    int32_t d_head;       /* width of the rebuilt key and value rows, and of q and out */
    int32_t d_latent;     /* d_c */
    int32_t max_context;
    int32_t dtype;        /* kvc_dtype */
} kvc_mla_config;

typedef struct kvc_mla_cache kvc_mla_cache; /* opaque handle */

/* Bytes of the latent cache [n_layers, batch, max_context, d_latent]; 0 for an
 * invalid configuration. */
uint64_t kvc_mla_cache_bytes(const kvc_mla_config *cfg);

/* Workspace bytes kvc_mla_alloc needs: the error word, the absorbed queries
 * [B, H, d_latent] and the split partials of up to 256 + B splits. */
uint64_t kvc_mla_workspace_bytes(const kvc_mla_config *cfg);

/* Bind a caller-owned latent cache and workspace to a new handle.
 *   cfg        host
 *   c_base     device, kvc_mla_cache_bytes(cfg) bytes, 16-byte aligned; the
 *              latents of layer l start at l * B * max_context * d_latent
 *              elements
 *   workspace  device, >= kvc_mla_workspace_bytes(cfg), 256-byte aligned;
 *              kvc_mla_alloc zeroes its error word (synchronously); it must
 *              not be used for anything else while the handle lives
 *   out        host; receives the handle
 * Host errors: KVC_ERR_INVALID, KVC_ERR_UNSUPPORTED, KVC_ERR_ALIGNMENT,
 * KVC_ERR_WORKSPACE, KVC_ERR_CUDA. */
kvc_status kvc_mla_alloc(const kvc_mla_config *cfg, void *c_base, void *workspace,
                         uint64_t ws_bytes, kvc_mla_cache **out);

void kvc_mla_free(kvc_mla_cache *h);

/* Number of splits (CTAs) of the attention launch: 0 automatic, else
 * 1..256. */
kvc_status kvc_mla_set_num_splits(kvc_mla_cache *h, int32_t n);

/* Write T_new latent rows per sequence at cache_index[b].
 *   c_new        device, [B, T_new, d_latent], 16-byte aligned
 *   cache_index  device int32 [B]; a sequence whose rows would leave
 *                [0, max_context) is skipped and KVC_ERR_DEVICE_INDEX recorded
 * Host errors: KVC_ERR_INVALID, KVC_ERR_CAPACITY, KVC_ERR_ALIGNMENT, KVC_ERR_CUDA. */
kvc_status kvc_mla_append(kvc_mla_cache *h, int32_t layer, const void *c_new,
                          const int32_t *cache_index, int32_t T_new, void *stream);

/* MLA decode attention of one layer.
 *   q          device, [B, n_heads, d_head], 16-byte aligned
 *   w_uk, w_uv device, [n_heads, d_head, d_latent] each, 16-byte aligned
 *   valid_len  device int32 [B]: live latent rows of each sequence; a value
 *              outside [1, max_context] skips the sequence (out unwritten) and
 *              records KVC_ERR_DEVICE_INDEX
 *   max_valid_hint  host upper bound of valid_len (sizes the grid), 0 = max_context
 *   out        device, [B, n_heads, d_head]
 * Three launches on the stream: absorb, attention over the latents, combine
 * with the up-projection.
 * Host errors: KVC_ERR_INVALID, KVC_ERR_ALIGNMENT, KVC_ERR_CUDA. */
kvc_status kvc_mla_decode_attn(kvc_mla_cache *h, int32_t layer, const void *q,
                               const void *w_uk, const void *w_uv,
                               const int32_t *valid_len, int32_t max_valid_hint,
                               void *out, void *stream);

/* The decode step of one layer: write c_new [B, d_latent] (device, 16-byte
 * aligned) at row valid_len[b] - 1, then kvc_mla_decode_attn.  The append
 * rides in the absorb launch (three launches in all). */
kvc_status kvc_mla_decode_step(kvc_mla_cache *h, int32_t layer, const void *q,
                               const void *c_new, const void *w_uk, const void *w_uv,
                               const int32_t *valid_len, int32_t max_valid_hint,
                               void *out, void *stream);

/* As kvc_get_error, for an MLA handle. */
kvc_status kvc_mla_get_error(kvc_mla_cache *h, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
