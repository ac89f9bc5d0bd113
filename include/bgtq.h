/*
 * bgtq.h — C ABI of the Block-GTQ packed-cache decode library (GB300, sm_103a).
 *
 * The method: "RoPE-Aware Bit Allocation for KV-Cache Quantization".  Under
 * RoPE a key's contribution to a logit is a sum over 2-D frequency blocks
 * (English abstract); Block-GTQ scores each RoPE block of each (layer, KV
 * head) with a label-free energy from calibration data and greedily assigns
 * integer bit widths by marginal gain under the TQ-MSE 4^-b distortion rate
 * (English abstract; paper review §1 Key Terms, §3 Method & Key Results).
 * Values use uniform TQ-MSE.  The packed-cache serving path attends directly
 * on the compressed cache, never materialising an fp16 KV cache (abstract;
 * review §1 "Packed-Cache", Figure 2).
 *
 * Conventions for every entry point:
 *   - Return value: BGTQ_OK (0) or a negative BGTQ_ERR_* code; the message of
 *     the last failure on the calling thread is returned by bgtq_last_error().
 *   - "device" pointers are CUDA device memory owned by the caller; "host"
 *     pointers are ordinary host memory owned by the caller.  The library
 *     allocates device memory only in bgtq_plan_create (its read-only tables,
 *     freed by bgtq_plan_destroy).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is enqueued asynchronously on it; no call
 *     synchronises the host except bgtq_plan_create/destroy.
 *   - The quantize-append and decode kernels launch with programmatic
 *     dependent launch: each may start while the previous kernel on the
 *     stream is still running, does its plan-static set-up, and waits for
 *     that kernel to finish before it reads q, k, v, pos_start or the cache.
 *     The decode kernel reads seq_lens BEFORE that wait, so seq_lens must not
 *     be written by a kernel that triggers its dependents early (no kernel
 *     of this library writes it; ordinary kernels and copies are fine).
 *   - head_dim must be 128.  Inputs must be finite: NaN/Inf inputs give
 *     unspecified codes, never a fault.
 *   - Errors discovered on the device (positions beyond the cache capacity,
 *     sequence lengths beyond capacity) are OR-ed into an optional device
 *     status word (BGTQ_STATUS_* bits) and the offending work is skipped.
 *
 * Cache layout of one layer (all caller-owned device memory, see
 * bgtq_cache_bytes):
 *   k_codes [B][H][capacity][16*bK] bytes  one K record per token
 *   v_codes [B][H][capacity/2][32*bV] bytes one V record per token pair
 *   k_norm, v_norm [B][H][capacity] float   per-token norms (side data)
 * with bK = bits_per_key / 128, bV = v_bits, capacity even.
 * A paged cache (page_table != NULL in bgtq_cache) stores the same records in
 * pools of pages of P tokens: the arrays above with [B] -> [n_pages] and
 * capacity -> P, and sequence b's position pos in page page_table[b][pos / P]
 * at row pos mod P.  Size the pools with bgtq_cache_bytes(plan, n_pages, P).
 */
#ifndef BGTQ_H
#define BGTQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BGTQ_OK 0
#define BGTQ_ERR_INVALID_ARG (-1)
#define BGTQ_ERR_UNSUPPORTED (-2)
#define BGTQ_ERR_CAPACITY (-3)
#define BGTQ_ERR_WORKSPACE (-4)
#define BGTQ_ERR_CUDA (-5)
#define BGTQ_ERR_DEVICE_CHECK (-6)

/* device status bits */
#define BGTQ_STATUS_APPEND_CAPACITY 1 /* pos_start + t_new > capacity: that sequence was skipped */
#define BGTQ_STATUS_SEQLEN_CAPACITY 2 /* seq_len > capacity or < 0: clamped */
#define BGTQ_STATUS_PAGE_RANGE 4      /* a page_table entry outside [0, n_pages) was met: writes to that
                                         page skipped, reads use page 0 (output unspecified) */
#define BGTQ_STATUS_BOUNDS 16         /* library built with BGTQ_DEBUG_BOUNDS only: an index (record slot,
                                         position against the capacity, page entry, table entry) failed
                                         its range check; that access was skipped */
#define BGTQ_STATUS_TIMEOUT 8         /* a wait inside a pipelined kernel gave up after 2 s: that launch
                                         skipped the rest of its work (output unspecified); never expected,
                                         reported instead of hanging the GPU */

/* plan flags */
#define BGTQ_PLAN_HOST_ONLY 1 /* build the tables on the host only (inspection, no GPU needed) */

typedef struct bgtq_plan bgtq_plan;

/* One layer's packed cache.  Passed by pointer; the struct itself is read on
 * the host only.  k_codes and v_codes must be 16-byte aligned (the kernels
 * copy whole records with 16-byte asynchronous copies), the norms 4-byte
 * aligned; INVALID_ARG otherwise. */
typedef struct {
    void* k_codes;    /* device, [B][H][capacity][16*bK] bytes */
    float* k_norm;    /* device, [B][H][capacity] */
    void* v_codes;    /* device, [B][H][capacity/2][32*bV] bytes */
    float* v_norm;    /* device, [B][H][capacity] */
    int64_t capacity; /* tokens per (sequence, head); must be even */
    /* Optional fp16 recent-key buffer (abstract: results are quoted "without
     * an fp16 recent-key buffer", so the option exists).  recent = W > 0:
     * every append also copies the fp16 keys of its last W tokens into ring
     * slot (position mod W) of k_recent, and decode uses those exact keys for
     * positions [seq_len - W, seq_len) (values stay packed).  recent = 0:
     * none (k_recent may be NULL). */
    void* k_recent;   /* device, [B][H][recent][128] half, 16-byte aligned */
    int64_t recent;   /* W, 0 <= W <= capacity */
    /* Optional paging (serving without a per-sequence reservation; NULL =
     * contiguous, the fields below ignored).  page_table[b][i] is the pool
     * page that holds positions i P .. i P + P - 1 of sequence b; a page
     * that an append writes must not be mapped twice.
     * page_table is read by the decode kernel before it waits for the previous
     * kernel (like seq_lens): it must not be written by a kernel that triggers
     * its dependents early.  capacity must equal max_pages * page_tokens
     * and be at most 2^21. */
    const int32_t* page_table; /* device, [B][max_pages] */
    int64_t max_pages;         /* entries per row of page_table, >= 1 */
    int64_t page_tokens;       /* P: a power of two, 16 <= P <= 2^20 */
    int64_t n_pages;           /* pages in the pools, >= 1 */
} bgtq_cache;

/* Message of the last failure on this thread ("" if none).  Never NULL. */
const char* bgtq_last_error(void);

/*
 * bgtq_alloc_bits — Block-GTQ allocation for one (layer, KV head).
 * Source: abstract ("computes a label-free energy score for each RoPE block
 * and greedily allocates integer bit widths by marginal gain"), review §3
 * (the gain uses the TQ-MSE 4^-b rate within the budget).
 *   calib_keys_fp16  host, [n][head_dim] IEEE half bit patterns, keys as cached
 *                    (RoPE applied)
 *   bits_per_key     even, >= 0: bits spent per key (K3 = 384); every greedy
 *                    step gives one bit to both coordinates of a block
 *   b_max            1..8, largest width of a block
 *   rope_layout      0 = half-split blocks (i, i+64), 1 = interleaved (2i, 2i+1)
 *   block_bits_out   host, [head_dim/2] widths (sum = bits_per_key/2)
 *   energy_out       host, [head_dim/2] float64 energies, may be NULL
 * Energy: s_i = (1/n) sum_t (k_t[lo_i]^2 + k_t[hi_i]^2) in float64.  Greedy:
 * the block maximising s_i*4^-b_i among b_i < b_max gets the next bit, ties
 * to the smaller index.  Host only; never touches the GPU.
 * Errors: INVALID_ARG for n <= 0, odd or oversized budgets, b_max out of range.
 */
int bgtq_alloc_bits(const uint16_t* calib_keys_fp16, int64_t n, int head_dim, int bits_per_key, int b_max,
                    int rope_layout, uint8_t* block_bits_out, double* energy_out);

/*
 * bgtq_plan_create — codec tables of one layer (all KV heads).
 * Source: TQ-MSE "rotates then quantises" with a near-optimal distortion rate
 * (review §1 Key Terms); per-block widths from Block-GTQ (abstract).
 *   n_kv_heads       KV heads of the layer (H)
 *   group            query heads per KV head (G, 1..8); query head h reads
 *                    KV head h / G
 *   bits_per_key     multiple of 128 (bK = bits_per_key/128 words per lane slice)
 *   v_bits           1..5, uniform value width
 *   block_bits       host, [H][head_dim/2] widths from bgtq_alloc_bits
 *   energy           host, [H][head_dim/2] energies from bgtq_alloc_bits
 *   seed             per-layer seed of the random rotation signs
 *   rope_layout      as in bgtq_alloc_bits
 *   flags            0, or BGTQ_PLAN_HOST_ONLY
 * Builds, per head: the codec order (width classes cut into aligned
 * power-of-two rotation pieces), whitening, SplitMix64 rotation signs, the
 * Lloyd-Max codebooks (fp16 centroids, float32 thresholds), the lane layout
 * of the K record, and copies them to the current CUDA device (synchronous).
 * Errors: INVALID_ARG (sizes, widths not summing to the budget);
 * UNSUPPORTED (head_dim != 128, no balanced lane layout for an allocation);
 * CUDA (device allocation or copy failed).
 */
int bgtq_plan_create(bgtq_plan** out, int head_dim, int n_kv_heads, int group, int bits_per_key, int v_bits,
                     const uint8_t* block_bits, const double* energy, uint64_t seed, int rope_layout, int flags);

/* Frees the plan and its device tables (synchronous).  NULL is accepted. */
int bgtq_plan_destroy(bgtq_plan* plan);

/*
 * Host views of a plan's tables, for inspection and for checking them against
 * an independent implementation.  The pointers stay valid until the plan is
 * destroyed.  head in [0, H).
 *   n_coded      coded coordinates of the head's keys (widths > 0)
 *   perm         [128] codec index -> original dim (first n_coded valid)
 *   width        [128] code width of each codec index
 *   piece        [128] rotation piece size of each codec index
 *   sign_k       [128] +1/-1 rotation signs of the keys (codec order)
 *   sign_v       [128] +1/-1 rotation signs of the values
 *   whiten       [128] float whitening multiplier of each codec index
 *   dewhiten     [128] float de-whitening multiplier of each codec index
 *   slot_pair    [4][16] K record lane layout: codec pair in each lane slot
 *   slot_offset  [4][16] bit offset of each slot's field inside its lane slice
 */
typedef struct {
    int n_coded;
    const uint8_t* perm;
    const uint8_t* width;
    const uint8_t* piece;
    const int8_t* sign_k;
    const int8_t* sign_v;
    const float* whiten;
    const float* dewhiten;
    const uint8_t* slot_pair;
    const uint16_t* slot_offset;
} bgtq_head_tables;

int bgtq_plan_get_head(const bgtq_plan* plan, int head, bgtq_head_tables* out);

/*
 * bgtq_plan_save / bgtq_plan_load — a plan as bytes (to keep a calibration
 * with a model, or to build it on another host).  The paper has no
 * counterpart; a plan is a deterministic function of its inputs (the
 * Block-GTQ widths and energies of every head, the group, budgets, seed and
 * RoPE layout), so those are what is stored, in a versioned, checksummed,
 * little-endian record; loading runs bgtq_plan_create on them and rebuilds
 * every table bit for bit.
 *   bgtq_plan_save: buf host (NULL: only *bytes is set), capacity its size;
 *                   *bytes = the record's size.  INVALID_ARG if capacity is
 *                   too small.
 *   bgtq_plan_load: buf/bytes a record from bgtq_plan_save; flags as for
 *                   bgtq_plan_create (BGTQ_PLAN_HOST_ONLY: no device tables).
 *                   INVALID_ARG for a foreign, truncated or corrupted record
 *                   (magic, size, checksum), UNSUPPORTED for another format
 *                   version, and bgtq_plan_create's errors.
 */
int bgtq_plan_save(const bgtq_plan* plan, void* buf, size_t capacity, size_t* bytes);
int bgtq_plan_load(bgtq_plan** out, const void* buf, size_t bytes, int flags);

/* Codebook of one width (0..8): 2^width fp16-exact centroids as floats and
 * 2^width - 1 float thresholds (host pointers owned by the plan). */
int bgtq_plan_get_codebook(const bgtq_plan* plan, int width, const float** centroids, const float** thresholds,
                           int* n_levels);

/* Codes of n quotients u at one width (0..8) through the plan's code-search
 * cell tables, on the host: the number of width-`width` thresholds <= u[i]
 * (TQ-MSE's nearest-centroid rule, review §1 Key Terms; the bulk encoder
 * takes its codes from the same tables).  u, codes: host arrays of n floats /
 * int32; a NaN is INVALID_ARG (the codes of the quotients before it are then
 * written, the rest not).  For checking the tables against a plain count. */
int bgtq_plan_code(const bgtq_plan* plan, int width, const float* u, int64_t n, int32_t* codes);

/* Byte sizes of one layer's cache buffers for `batch` sequences of `capacity`
 * tokens (capacity even); for a paged cache, of the pools: batch = n_pages,
 * capacity = page_tokens.  Host only. */
int bgtq_cache_bytes(const bgtq_plan* plan, int batch, int64_t capacity, size_t* k_codes_bytes,
                     size_t* v_codes_bytes, size_t* norm_bytes);

/*
 * bgtq_quantize_append — encode and store new tokens (prefill chunk or one
 * decode token).  Source: the packed cache is written from compressed K/V
 * (abstract, packed-cache serving path); TQ-MSE encoder (review §1).
 *   k_fp16, v_fp16   device, [batch][H][t_new][128] half (RoPE applied to K)
 *   pos_start        device, [batch] int32: first cache position written for
 *                    each sequence (not modified)
 *   cache            host pointer to the layer's cache descriptor
 *   dev_status       device int32 or NULL: BGTQ_STATUS_APPEND_CAPACITY is
 *                    OR-ed in and the sequence skipped when pos_start +
 *                    t_new > capacity or pos_start < 0
 * Per token: rotate (whitened keys / raw values), store the float norm, code
 * every coordinate against the Lloyd-Max thresholds, bit-pack at exactly the
 * budget.  Bits of other tokens that share a V pair record are preserved.
 * Errors: INVALID_ARG (null pointers, batch/t_new < 0, odd capacity,
 * host-only plan); CUDA (launch failure).
 */
int bgtq_quantize_append(const bgtq_plan* plan, void* stream, const void* k_fp16, const void* v_fp16, int batch,
                         int t_new, const int32_t* pos_start, const bgtq_cache* cache, int32_t* dev_status);

/* Workspace bytes bgtq_decode_attn needs for `batch` sequences no longer than
 * max_len.  The workspace must be zero-filled once before first use (its
 * counters are returned to zero by every call). */
int bgtq_decode_attn_workspace(const bgtq_plan* plan, int batch, int64_t max_len, size_t* bytes);

/*
 * bgtq_decode_attn — one decode step of attention on the packed cache.
 * Source: packed-cache serving path that works on compressed K/V without an
 * fp16 KV cache (abstract; review §1 "Packed-Cache", Figure 2).
 *   q_fp16       device, [batch][H*G][128] half, RoPE applied
 *   cache        host pointer to the layer's cache descriptor
 *   seq_lens     device, [batch] int32 valid tokens per sequence (not modified);
 *                values above capacity are clamped (status bit 2)
 *   max_len      host upper bound of seq_lens (sizes the split-K grid)
 *   out          device, [batch][H*G][128], half (out_dtype 0) or float (1)
 *   softmax_scale  logit scale, e.g. 1/sqrt(128)
 *   workspace    device scratch of bgtq_decode_attn_workspace bytes (zeroed
 *                once before the first call)
 *   dev_status   device int32 or NULL
 * Computes o_g = sum_t softmax_t(scale * q_g . k_t) v_t over the dequantised
 * cache: the query is rotated once into the codec domain, K/V codes are
 * streamed from HBM and decoded by codebook lookup, the contractions run on
 * tensor cores, and split-K partials are merged by the last CTA of each
 * (sequence, head).  An empty sequence yields zeros.
 * Errors: INVALID_ARG, WORKSPACE (too small), UNSUPPORTED (bK > 3 or G > 8),
 * CUDA.
 */
int bgtq_decode_attn(const bgtq_plan* plan, void* stream, const void* q_fp16, const bgtq_cache* cache,
                     const int32_t* seq_lens, int64_t max_len, int batch, void* out, int out_dtype,
                     float softmax_scale, void* workspace, size_t ws_bytes, int32_t* dev_status);

/*
 * bgtq_decode_step — one decode step of one layer in a single launch: the
 * new token of every sequence is quantize-appended to the packed cache and
 * attention then runs over the updated cache.
 * Source: the packed-cache serving path (abstract; review §1 "Packed-Cache",
 * Figure 2): each step appends the new token's compressed K/V and attends on
 * the compressed cache.
 *   k_new_fp16, v_new_fp16  device, [batch][H][128] half: the new token
 *   pos_new      device, [batch] int32 cache position of the new token (read
 *                before the kernel waits for the previous kernel, like
 *                seq_lens); usually seq_lens[b] - 1
 *   all other arguments as bgtq_decode_attn (same workspace size)
 * The result equals bgtq_quantize_append (t_new = 1, pos_start = pos_new)
 * followed by bgtq_decode_attn: the same codes, norms and records are
 * written and the attention sees them.  A position outside [0, capacity)
 * appends nothing and sets BGTQ_STATUS_APPEND_CAPACITY.
 * Errors: as bgtq_decode_attn.
 */
int bgtq_decode_step(const bgtq_plan* plan, void* stream, const void* q_fp16, const void* k_new_fp16,
                     const void* v_new_fp16, const int32_t* pos_new, const bgtq_cache* cache,
                     const int32_t* seq_lens, int64_t max_len, int batch, void* out, int out_dtype,
                     float softmax_scale, void* workspace, size_t ws_bytes, int32_t* dev_status);

/*
 * bgtq_prefill_attn — prefill of a prompt into an empty cache in one launch:
 * causal attention over the prompt's own fp16 K/V, and the packed records of
 * positions 0 .. t-1 written to the cache.
 * Source: the packed cache is written at prefill and read at decode (review
 * §1 "Packed-Cache"); fusing the quantizer into attention is named as future
 * work on the LogQuant page (section "중요성 및 주장").
 *   q_fp16       device, [batch][H*G][t][128] half, RoPE applied, 16-byte aligned
 *   k_fp16, v_fp16  device, [batch][H][t][128] half, 16-byte aligned
 *   t            prompt length, 0 <= t <= capacity
 *   cache        host pointer to the layer's cache descriptor (contiguous or
 *                paged; with a recent-key buffer its last W keys are copied too)
 *   out          device, [batch][H*G][t][128], half (out_dtype 0) or float (1),
 *                16-byte aligned
 *   softmax_scale  logit scale, e.g. 1/sqrt(128)
 *   dev_status   device int32 or NULL
 * Row i of query head g computes sum_{j <= i} softmax_j(scale q_i . k_j) v_j
 * with the keys and values as given (fp16 tensor-core products, fp32
 * accumulation, probabilities rounded to fp16); the records are those
 * bgtq_quantize_append writes for the same tokens at pos_start = 0, bit for
 * bit.  Prefill onto a non-empty cache (a later chunk) is not covered.
 * Errors: INVALID_ARG (pointers, alignment, dtype, scale), CAPACITY (t >
 * capacity), CUDA.
 */
int bgtq_prefill_attn(const bgtq_plan* plan, void* stream, const void* q_fp16, const void* k_fp16,
                      const void* v_fp16, int batch, int t, const bgtq_cache* cache, void* out, int out_dtype,
                      float softmax_scale, int32_t* dev_status);

/*
 * bgtq_prefill_chunk_workspace — bytes of device scratch that
 * bgtq_prefill_chunk_attn needs for `batch` sequences whose prefixes are at
 * most max_prefix tokens: every prefix token's decoded rows (raw centroids,
 * fp16, K and V) and its two norms, (512 + 8) bytes per (sequence, KV head,
 * position up to max_prefix rounded up to 128).
 */
int bgtq_prefill_chunk_workspace(const bgtq_plan* plan, int batch, int64_t max_prefix, size_t* bytes);

/*
 * bgtq_prefill_chunk_attn — a later chunk of a long prompt onto a cache that
 * already holds positions 0 .. P0-1 of each sequence: the packed records of
 * positions P0 .. P0+c-1 are written (bgtq_quantize_append at pos_start = P0,
 * bit for bit) and chunk row i attends, in one softmax, the P0 cached keys as
 * stored (dequantised) and the chunk's keys 0 .. i as given, values likewise.
 * Source: the packed cache is what earlier chunks left (review §1
 * "Packed-Cache"); a quantizer fused into attention is future work on the
 * LogQuant page (section "중요성 및 주장").
 *   q_fp16       device, [batch][H*G][c][128] half, RoPE applied, 16-byte aligned
 *   k_fp16, v_fp16  device, [batch][H][c][128] half (the chunk), 16-byte aligned
 *   c            chunk length, 0 <= c <= capacity
 *   dev_pos_start  device int32 [batch]: P0 of each sequence; a sequence with
 *                P0 < 0 or P0 + c > capacity is skipped (nothing written to
 *                the cache, zero output rows, BGTQ_STATUS_APPEND_CAPACITY); one
 *                with P0 > max_prefix gets zero output rows and
 *                BGTQ_STATUS_SEQLEN_CAPACITY (its records are still appended)
 *   max_prefix   host bound of every P0, 0 <= max_prefix <= capacity
 *   cache        host pointer to the layer's descriptor, contiguous or paged,
 *                without a recent-key buffer
 *   out          device, [batch][H*G][c][128], half (out_dtype 0) or float
 *                (1), 16-byte aligned
 *   softmax_scale  logit scale, e.g. 1/sqrt(128)
 *   workspace    device scratch of bgtq_prefill_chunk_workspace(plan, batch,
 *                max_prefix) bytes, 256-byte aligned (contents not kept)
 *   dev_status   device int32 or NULL
 * Three launches on `stream`: the append, the decode of the prefix records
 * into the workspace (each prefix token once), the attention (tcgen05).  The
 * chunk part is computed as in bgtq_prefill_attn; the prefix part in the
 * codecs' own domains (rotated query, raw centroids, norms in fp32) with fp16
 * hi + lo splits of the query and of the probabilities, fp32 accumulation.
 * Errors: INVALID_ARG (pointers, alignment, dtype, scale), CAPACITY (c or
 * max_prefix > capacity), WORKSPACE (too small), UNSUPPORTED (a recent-key
 * buffer, bK > 3, bV > 4, sizes past 2^31 rows), CUDA.
 */
int bgtq_prefill_chunk_attn(const bgtq_plan* plan, void* stream, const void* q_fp16, const void* k_fp16,
                            const void* v_fp16, int batch, int c, const int32_t* dev_pos_start, int64_t max_prefix,
                            const bgtq_cache* cache, void* out, int out_dtype, float softmax_scale, void* workspace,
                            size_t ws_bytes, int32_t* dev_status);

/*
 * bgtq_decode_attn_noalloc — bgtq_decode_attn for callers that cannot
 * allocate device memory (a fixed memory budget, an allocator or pool that
 * must not be bypassed, a host runtime without a device allocator).  The
 * paper has no counterpart; this is a convenience of the library.
 *   Same arguments and results as bgtq_decode_attn, minus the workspace: the
 *   split-merge scratch is one built-in device array of 2 MiB that every GPU
 *   which loads the library keeps until the process exits.  No call
 *   allocates or frees memory.
 *   Every call looks up that array's address on the current device (a
 *   host-side lookup, so a reset and re-created context is followed); the
 *   first call on a device may load the library's device code, so make it
 *   before any stream capture.  Every call shares the array and it keeps the
 *   last call's contents (its counters are cleared by each call), so calls
 *   that overlap on the GPU race; order them on one stream.
 * Errors: as bgtq_decode_attn; WORKSPACE when the problem needs more than the
 * built-in 2 MiB of scratch (then use bgtq_decode_attn with a workspace).
 */
int bgtq_decode_attn_noalloc(const bgtq_plan* plan, void* stream, const void* q_fp16, const bgtq_cache* cache,
                             const int32_t* seq_lens, int64_t max_len, int batch, void* out, int out_dtype,
                             float softmax_scale, int32_t* dev_status);

/*
 * bgtq_logit_mae — RoPE-logit fidelity diagnostic: for every query head, the
 * mean absolute error of the attention logits computed from the packed keys
 * against the keys as given,
 *   mae[b][g] = (1/t) sum_{s < t} | softmax_scale (q_g . k_s - q_g . khat_s) |
 * over cache positions 0..t-1 (khat = the dequantised cached key).
 * Source: review §3 Method & Key Results (Block-GTQ lowers the RoPE-logit
 * error against uniform TQ-MSE at matched budgets; plan a uniform baseline
 * with every block at bK bits and equal energies); English abstract (the
 * logit is a sum over 2-D frequency blocks).
 *   q_fp16      device, [batch][H*G][128] half
 *   k_fp16      device, [batch][H][t][128] half (8-byte aligned): the keys
 *               that were appended at positions 0..t-1
 *   cache       host pointer to the descriptor of the cache holding them
 *   mae         device, [batch][H*G] float, overwritten
 * q.khat is computed in the key codec domain as the decode kernel does; the
 * result is float32 (summation order not fixed).
 * Errors: INVALID_ARG (t > capacity, NULL, misaligned k, host-only plan),
 * UNSUPPORTED (G > 8), CUDA.
 */
int bgtq_logit_mae(const bgtq_plan* plan, void* stream, const void* q_fp16, const void* k_fp16,
                   const bgtq_cache* cache, int64_t t, int batch, float softmax_scale, float* mae);

/*
 * bgtq_dequant_debug — decode cached tokens [t0, t1) of (sequence b, head)
 * back to float32, for inspection and parity checks.
 *   k_out, v_out  device, [t1-t0][128] float (either may be NULL)
 *   codec_domain  0: original dims (inverse rotation, de-whitening, scatter);
 *                 1: codec-domain reconstruction rho * centroid per codec index
 * Errors: INVALID_ARG (ranges outside the capacity, host-only plan), CUDA.
 */
int bgtq_dequant_debug(const bgtq_plan* plan, void* stream, const bgtq_cache* cache, int batch, int b, int head,
                       int64_t t0, int64_t t1, float* k_out, float* v_out, int codec_domain);

#ifdef __cplusplus
}
#endif

#endif /* BGTQ_H */
