/*
 * fw_attn.h -- C ABI of the GB300 (sm_103a) ragged softmax attention library.
 *
 * Two operations, both fused online-softmax attention that never materialises
 * the probability matrix (running max m, running sum l and a rescaled output
 * accumulator o, "Flywheel Attention: Attention Kernels Built for the TPU",
 * section 1, the FlashAttention recurrence):
 *
 *   fw_paged_decode    -- grouped-query decode over a paged, ragged KV cache
 *                         addressed through block_table[batch, logical_page]
 *                         ("Writing Page Attention with PyPTO", sections 1.2-1.3
 *                         and 5.2), with split-KV partials merged by a
 *                         log-sum-exp combine ("TokenSpeed-MLA 2.0.1", decode:
 *                         a split-KV attention kernel plus a reduction kernel).
 *   fw_varlen_prefill  -- ragged varlen prefill without padding, Q and KV packs
 *                         given by cumulative sequence lengths, causal or not
 *                         ("TokenSpeed-MLA 2.0.1", capability summary, MLA Prefill).
 *
 * Conventions shared by every entry point
 *   - Tensors are passed as fw_tensor_t: a DEVICE pointer, a dtype, up to 5
 *     dimensions and strides IN ELEMENTS.  The caller owns every tensor; the
 *     library never frees or retains them past the call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  They never synchronise the host and never copy device data to
 *     the host; split planning uses shapes only (max_pages * page_size bounds
 *     every sequence).
 *   - Arithmetic: BF16 inputs, FP32 accumulation and softmax state, BF16 output
 *     rounded to nearest even, FP32 LSE.  LSE is the NATURAL log of
 *     sum_j exp(scale * <q, k_j>) over the visible keys.
 *   - Grouped-query heads: query head h reads KV head h / (Hq / Hkv), so
 *     consecutive query heads share a KV head (PyPTO section 1.3: KV head 1
 *     serves query heads 5-9 at 40 Q / 8 KV heads).
 *   - Rows with no visible key produce a zero output row and LSE = -inf
 *     ("TokenSpeed-MLA 2.0.1", SM107 decode section).
 *   - Errors: invalid shapes, dtypes, strides or alignment return a status and
 *     launch nothing; fw_last_error() then describes the problem.  A CUDA
 *     launch failure returns FW_ERR_CUDA.  A device-side wait that exceeds its
 *     time limit does not trap: the kernel records FW_ERR_DEVICE_TIMEOUT in a
 *     device status word and exits; read it with fw_get_device_status().
 */
#ifndef FW_ATTN_H
#define FW_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *fw_stream_t; /* identical to cudaStream_t */

typedef enum {
    FW_OK = 0,
    FW_ERR_INVALID_ARG = 1,     /* inconsistent shapes / dtypes / strides / NULL data */
    FW_ERR_UNSUPPORTED = 2,     /* valid but not implemented (head dim, page size, ...) */
    FW_ERR_WORKSPACE = 3,       /* caller workspace too small, or allocation failed */
    FW_ERR_CUDA = 4,            /* a CUDA runtime / driver call failed */
    FW_ERR_DEVICE_TIMEOUT = 5   /* a kernel gave up waiting (reported by fw_get_device_status) */
} fw_status_t;

typedef enum { FW_BF16 = 0, FW_F32 = 1, FW_I32 = 2, FW_FP8_E4M3 = 3 } fw_dtype_t;

typedef struct {
    void *data;          /* device pointer (may be NULL only when every extent is 0) */
    int32_t dtype;       /* fw_dtype_t */
    int32_t ndim;        /* 1..5 */
    int64_t shape[5];
    int64_t stride[5];   /* in elements */
} fw_tensor_t;

/*
 * Paged grouped-query decode.
 *
 *   q           [B, q_len, Hq, Dk]            BF16, last dim contiguous
 *   k_cache     [num_pages, ps, Hkv, Dk]      BF16, last dim contiguous
 *   v_cache     [num_pages, ps, Hkv, Dv]      BF16, last dim contiguous; may be a
 *                                             strided view of k_cache (latent heads:
 *                                             V = the first Dv columns of each K row)
 *   block_table [B, max_pages]                I32; entry [b, p] is the physical page of
 *                                             logical page p of row b.  Entries at or
 *                                             past ceil(seq_lens[b] / ps) are never read
 *                                             (PyPTO section 9.1) and may hold anything.
 *   seq_lens    [B]                           I32; keys of row b, including the q_len
 *                                             new tokens; 0 <= seq_lens[b] <= max_pages*ps.
 *   scale       softmax scale applied to <q, k> before the max (PyPTO section 6.2).
 *   out         [B, q_len, Hq, Dv]            BF16, written.
 *   lse         [B, q_len, Hq]                F32, written; may be NULL.
 *
 * With q_len > 1 the query tokens are causal and bottom-right aligned: token
 * t sees keys 0 .. seq_lens[b] - q_len + t.  With q_len = 1 every key is seen.
 *
 * Supported: Dk = Dv in {128, 256}; Hq % Hkv == 0 (any group size); page sizes
 * 8, 16, 32, 64, 128 or any multiple of 128;
 * 1 <= q_len <= 4; strides multiples of 8 elements and 16-byte aligned base
 * pointers (tensor-memory-accelerator addressing).
 *
 * Split-KV: the keys of a row may be cut across CTAs (see fw_decode_plan_t);
 * the FP32 partials (normalised output + log2-sum-exp per row per piece) are
 * merged by a combine kernel.  Three launches per call: plan (one block),
 * attention, combine.  The plan and the partials live in a workspace:
 * caller-provided through fw_set_workspace(), else an internal buffer grown
 * on demand with cudaMalloc (grow it once, outside any stream capture, by an
 * initial call with the largest shapes).
 */
fw_status_t fw_paged_decode(const fw_tensor_t *q, const fw_tensor_t *k_cache,
                            const fw_tensor_t *v_cache, const fw_tensor_t *block_table,
                            const fw_tensor_t *seq_lens, float scale,
                            fw_tensor_t *out, fw_tensor_t *lse, fw_stream_t stream);

/*
 * fw_paged_decode for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for users of the library.
 *
 * Who needs it: code that runs where cudaMalloc is off limits -- a plugin whose
 * host runtime owns every byte of device memory and forbids allocation in its
 * execute step, or a latency-critical loop that cannot take the implicit
 * device synchronisation or the out-of-memory failure an allocation may
 * bring.  fw_paged_decode may grow an internal workspace with cudaMalloc the
 * first time it sees larger shapes; this variant never allocates anything.
 *
 * Arguments, layouts, supported shapes and results are those of
 * fw_paged_decode; a workspace set with fw_set_workspace() is not used.  Its
 * scratch (the tile prefix table and the split-KV partials) is a fixed
 * 64 MiB array in the library's device image, held by every GPU that loads
 * the library until the process exits.  Shapes whose scratch
 * (fw_decode_plan_t.workspace_bytes) exceeds 64 MiB return FW_ERR_WORKSPACE
 * and launch nothing.  That size follows the block table's width
 * (max_pages x page_size keys per row, the longest row the call could see),
 * not the seq_lens values, which stay on the device: a caller with short
 * rows in a wide table can pass a narrower view of the table (fewer
 * columns, same row stride) to fit.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  Every call shares the one array and nothing in
 * it needs to start at zero (each value is written before it is read within a
 * call), but calls whose kernels overlap on the GPU -- different streams, or
 * several host threads -- race on it: order them.
 */
fw_status_t fw_paged_decode_noalloc(const fw_tensor_t *q, const fw_tensor_t *k_cache,
                                    const fw_tensor_t *v_cache, const fw_tensor_t *block_table,
                                    const fw_tensor_t *seq_lens, float scale,
                                    fw_tensor_t *out, fw_tensor_t *lse, fw_stream_t stream);

/*
 * fw_paged_decode over an FP8 KV cache ("TokenSpeed-MLA 2.0.1", decode: FP8
 * inputs, BF16 output).
 *
 *   k_cache, v_cache  [num_pages, page_size, Hkv, 128]  FP8_E4M3 (OCP E4M3
 *                     bytes); key j's values are k_scale * e4m3(byte) and
 *                     v_scale * e4m3(byte), one scale per cache
 *   q, block_table, seq_lens, scale, out, lse, stream: as fw_paged_decode
 *                     (q BF16, out BF16, lse F32 natural log)
 *
 * Supported: Dk = Dv = 128, the query-head groupings, q_len 1-4 and page
 * sizes of fw_paged_decode; cache strides multiples of 16 bytes.  The
 * tensor cores read the E4M3 bytes as stored; the result is that of FP16
 * products of the FP8 values with FP16-exact queries and probabilities and
 * FP32 sums: each BF16 query row is scaled by a power of two and carried as
 * two E4M3 terms (exact for every element down to 2^-10 of the row's largest
 * magnitude), each probability is rounded to FP16 and carried as four E5M2
 * terms (exact).  The same workspace as fw_paged_decode
 * (fw_paged_decode_workspace_size with the same shapes); errors as
 * fw_paged_decode, plus FW_ERR_INVALID_ARG for a non-finite or non-positive
 * k_scale / v_scale.
 */
fw_status_t fw_paged_decode_fp8(const fw_tensor_t *q, const fw_tensor_t *k_cache,
                                const fw_tensor_t *v_cache, const fw_tensor_t *block_table,
                                const fw_tensor_t *seq_lens, float scale, float k_scale, float v_scale,
                                fw_tensor_t *out, fw_tensor_t *lse, fw_stream_t stream);

/*
 * Paged decode with a sliding window ("TokenSpeed-MLA 2.0.1", window_left),
 * over a BF16 or an FP8_E4M3 cache (chosen by k_cache's dtype).
 *
 *   window_left  -1: no window (the call equals fw_paged_decode or
 *                fw_paged_decode_fp8); W >= 0: query token t of row b sees only
 *                keys max(0, n - q_len + t - W) .. n - q_len + t, n =
 *                seq_lens[b] -- its own position and the W before it.
 *   k_scale, v_scale  the FP8 cache scales; must be 1 for a BF16 cache.
 *   other arguments   as fw_paged_decode / fw_paged_decode_fp8.
 *
 * The walk of a row starts at the KV tile holding its first visible key, so
 * the work scales with the window, not the row.  Block-table entries of pages
 * wholly before key max(0, n - q_len - W) are never read and those pages are
 * never loaded: a cache may drop pages that left the window.  Supported: the
 * layouts of fw_paged_decode (Dk = Dv in {128, 256}, and the latent Dk 576 /
 * Dv 512, where TokenSpeed defines window_left) and of fw_paged_decode_fp8.
 * FW_ERR_INVALID_ARG for W < -1 or BF16 caches with scales other than 1.
 * Same workspace as fw_paged_decode.
 */
fw_status_t fw_paged_decode_window(const fw_tensor_t *q, const fw_tensor_t *k_cache,
                                   const fw_tensor_t *v_cache, const fw_tensor_t *block_table,
                                   const fw_tensor_t *seq_lens, float scale, float k_scale, float v_scale,
                                   int32_t window_left, fw_tensor_t *out, fw_tensor_t *lse,
                                   fw_stream_t stream);

/*
 * fw_paged_decode_masked -- decode, causal or not ("TokenSpeed-MLA 2.0.1", MLA
 * decode: causal_mask supports causal and non-causal execution; window_left
 * bounds row i's history to start at max(0, K - q_len - window_left + i)).
 *
 *   causal       1: query token t of a row with n keys sees keys up to its own
 *                position n - q_len + t (as fw_paged_decode); 0: every token
 *                sees all n keys.  With q_len = 1 both are the same.
 *   window_left  -1: none; W >= 0: the keys a token sees start at
 *                max(0, n - q_len + t - W), causal or not.
 *   other arguments   as fw_paged_decode_window (BF16 or FP8_E4M3 caches,
 *                the scales applying to FP8 ones).
 *
 * Errors as fw_paged_decode_window; FW_ERR_UNSUPPORTED for a non-causal
 * sliding window on the grouped-query layouts with q_len > 1 (served for the
 * latent layout).  Same workspace as fw_paged_decode.
 */
fw_status_t fw_paged_decode_masked(const fw_tensor_t *q, const fw_tensor_t *k_cache,
                                   const fw_tensor_t *v_cache, const fw_tensor_t *block_table,
                                   const fw_tensor_t *seq_lens, float scale, int32_t causal,
                                   int32_t window_left, float k_scale, float v_scale,
                                   fw_tensor_t *out, fw_tensor_t *lse, fw_stream_t stream);

/*
 * KV-cache append ("Writing Page Attention with PyPTO", sections 4.2-4.3).
 *
 *   k_new, v_new  [B, q_len, Hkv, D]   BF16, last dim contiguous, strides
 *                                      multiples of 8 elements, 16-byte aligned;
 *                                      v_new may be NULL together with v_cache
 *                                      (a latent cache whose values are a view
 *                                      of its keys)
 *   slot_mapping  [B * q_len] or [B, q_len]  I32, contiguous; the token row of
 *                                      each new token inside its layer; -1 marks
 *                                      a warm-up token
 *   layer_base_rows   first token row of the layer in the (possibly packed
 *                     multi-layer) cache, 0 <= layer_base_rows < pages * ps
 *   k_cache, v_cache  [pages, ps, Hkv, D]  BF16 or FP8_E4M3 (both the same);
 *                     written
 *   k_scale, v_scale  FP8 caches: the stored code is E4M3(x / scale) -- IEEE
 *                     single-precision division, nearest with ties to even,
 *                     finite overflow saturating to +-448; 1 for BF16 caches
 *                     (which take the BF16 bits unchanged).
 *
 * Token (b, t), KV head h goes to token row
 *   r = layer_base_rows + max(slot_mapping[b * q_len + t], 0),
 * page r / ps, slot r % ps: the warm-up slot -1 is clamped to 0 before the
 * layer base is added, so a layer never writes the previous layer's last row.
 * Nothing else in the caches changes.  Tokens sharing a row (repeated
 * warm-up slots) race: each 16-byte group of that row (8 BF16 or 8 E4M3
 * values of one head) ends up holding one of theirs.  A row at
 * or past pages * ps records FW_ERR_INVALID_ARG in the device status word
 * and is skipped.  One launch; no workspace.
 */
fw_status_t fw_kv_append(const fw_tensor_t *k_new, const fw_tensor_t *v_new, const fw_tensor_t *slot_mapping,
                         int64_t layer_base_rows, fw_tensor_t *k_cache, fw_tensor_t *v_cache, float k_scale,
                         float v_scale, fw_stream_t stream);

/*
 * Append the new tokens, then decode: fw_kv_append followed by
 * fw_paged_decode_window on the layer, with the append folded into the
 * decode's plan launch (no extra launch; the attention launch starts after
 * it, so it reads the new rows).
 *
 *   k_cache, v_cache  the (packed) caches of fw_kv_append; the attention reads
 *                     the layer's pages, pages layer_base_rows / ps onward, so
 *                     block_table entries count pages from the layer's first
 *                     page and layer_base_rows must be a multiple of ps
 *   q, block_table, seq_lens, scale, k_scale, v_scale, window_left, out, lse:
 *                     as fw_paged_decode_window (seq_lens include the new
 *                     tokens, which normally occupy each row's last q_len
 *                     positions)
 *
 * Supported: the grouped-query layouts (BF16 Dk = Dv in {128, 256}, FP8 128);
 * the latent layout returns FW_ERR_UNSUPPORTED (append it with fw_kv_append).
 */
fw_status_t fw_paged_decode_append(const fw_tensor_t *q, const fw_tensor_t *k_new, const fw_tensor_t *v_new,
                                   const fw_tensor_t *slot_mapping, int64_t layer_base_rows,
                                   fw_tensor_t *k_cache, fw_tensor_t *v_cache,
                                   const fw_tensor_t *block_table, const fw_tensor_t *seq_lens, float scale,
                                   float k_scale, float v_scale, int32_t window_left,
                                   fw_tensor_t *out, fw_tensor_t *lse, fw_stream_t stream);

/*
 * Workspace bytes fw_paged_decode needs for these shapes (data pointers are
 * not read).  Writes the size to *bytes.  It holds the tile prefix table
 * (B + 3 int32) and rows * max_pieces * (Dv + 1) * 4 bytes of partials, with
 * rows = B * q_len * Hq: one FP32 partial output row plus one FP32 LSE per
 * row per split ("TokenSpeed-MLA 2.0.1", packed-query paragraph, 513 floats
 * per row at Dv 512).
 */
fw_status_t fw_paged_decode_workspace_size(const fw_tensor_t *q, const fw_tensor_t *k_cache,
                                           const fw_tensor_t *v_cache,
                                           const fw_tensor_t *block_table, size_t *bytes);

/*
 * Ragged varlen prefill.
 *
 *   q            [total_q, Hq, Dk]   BF16
 *   k            [total_k, Hkv, Dk]  BF16
 *   v            [total_k, Hkv, Dv]  BF16
 *   cu_seqlens_q [B + 1]             I32 prefix sums of the query lengths (cu[0] = 0)
 *   cu_seqlens_k [B + 1]             I32 prefix sums of the key lengths; may differ from Q's
 *   causal       nonzero: row r of a sequence (0-based) sees keys 0 .. r + Lk - Lq
 *                (bottom-right alignment); zero: every key of its sequence.
 *   out          [total_q, Hq, Dv]   BF16, written
 *   lse          [total_q, Hq]       F32, written; may be NULL
 *
 * Supported: Dk = Dv in {128, 256}; Hq % Hkv == 0; strides multiples of 8
 * elements, 16-byte aligned base pointers.  cu_seqlens_q[B] must equal total_q
 * and cu_seqlens_k[B] must not exceed total_k (checked on the device: a
 * sequence reaching past the packed tensors is skipped and flagged in the
 * device status word as FW_ERR_INVALID_ARG).
 */
fw_status_t fw_varlen_prefill(const fw_tensor_t *q, const fw_tensor_t *k, const fw_tensor_t *v,
                              const fw_tensor_t *cu_seqlens_q, const fw_tensor_t *cu_seqlens_k,
                              int causal, float scale, fw_tensor_t *out, fw_tensor_t *lse,
                              fw_stream_t stream);

/*
 * Caller-owned workspace for the CURRENT device (ptr = NULL, bytes = 0 returns
 * to the internal buffer).  The library never frees it.  Calls on one device
 * that share the workspace must be ordered (same stream, or synchronised).
 */
fw_status_t fw_set_workspace(void *ptr, size_t bytes, fw_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device: 0 when every kernel since the last read finished normally,
 * else the fw_status_t code of the first failure (FW_ERR_DEVICE_TIMEOUT when a
 * kernel abandoned a wait, FW_ERR_INVALID_ARG for a bad sequence extent).
 */
fw_status_t fw_get_device_status(fw_stream_t stream, int32_t *code);

/*
 * Device event counters, accumulated by every call on the current device
 * since the last read.  Synchronises `stream`, copies the first n (1..4)
 * counters into values[0..n-1] and resets all of them to zero.
 *
 *   FW_COUNTER_PREFILL_REPLAYS  (query row, KV tile) steps of the prefill
 *       static-anchor softmax whose running-sum check failed, so the tile was
 *       replayed with the rescaling form ("Flywheel Attention", section 3.1:
 *       the check raises a flag and the block is recomputed, appendix A)
 *   FW_COUNTER_LATENT_RESCALES  (query row, key step) steps of the latent-head
 *       decode whose anchor moved because a score rose more than 64 log2 units
 *       above it
 */
typedef enum {
    FW_COUNTER_PREFILL_REPLAYS = 0,
    FW_COUNTER_LATENT_RESCALES = 1
} fw_counter_t;

fw_status_t fw_read_counters(fw_stream_t stream, int64_t *values, int32_t n);

/* Message for the last failing call on this host thread ("" if none). */
const char *fw_last_error(void);

/* Tunables, mostly for tests and measurement. */
typedef enum {
    FW_OPT_DECODE_CHUNK_TOKENS = 0, /* force the keys per CTA range (multiple of 128; 0 = auto) */
    FW_OPT_WAIT_TIMEOUT_MS = 1,     /* device wait limit before giving up (default 2000) */
    FW_OPT_KERNEL_TIMING = 2,       /* 1: record CUDA events around each attention kernel */
    FW_OPT_MAX_CTAS = 3,            /* cap on persistent CTAs (0 = one per SM) */
    FW_OPT_PREFILL_SOFTMAX = 4,     /* prefill softmax: 0 = static anchor with a check and replay
                                       ("Flywheel Attention", section 3.1, default); 1 = online
                                       softmax with a conditional rescale (the base moves when a
                                       row max rises more than 8 log2 units).  Same result up to
                                       rounding; kept for comparison. */
    FW_OPT_TEST_STALL = 5           /* test hook, default 0.  1: the grouped-query decode kernel's
                                       copy warp first waits on a barrier that nothing completes,
                                       so that wait runs out after FW_OPT_WAIT_TIMEOUT_MS: the call
                                       records FW_ERR_DEVICE_TIMEOUT (read by fw_get_device_status)
                                       and its outputs are not valid.  Nothing is copied or
                                       multiplied before the wait, so no work is left in flight. */
} fw_option_t;

fw_status_t fw_set_option(int32_t option, int64_t value);

/*
 * With FW_OPT_KERNEL_TIMING on, the summed device time (ms) of the attention
 * kernels (decode or prefill main kernel, not the combine) since the last
 * read and the number of such launches.  Synchronises the device.  Resets the
 * accumulators.
 */
fw_status_t fw_kernel_timing_read(double *total_ms, int64_t *launches);

/* Total kernels this library has launched in this process (all kinds). */
int64_t fw_launch_count(void);

/*
 * Host-side decode plan for given shapes (no device access), exposed so the
 * planner can be checked without a GPU.  num_sms <= 0 queries the current
 * device.  Fields are written on success.
 *
 * Scheduling: the (batch row, KV head, row group) units are laid end to end
 * in the order of their 128-key tiles, each preceded by a few empty slots
 * that stand for the cost of starting a piece (none for the latent layout);
 * each persistent CTA takes equal contiguous ranges of that sequence (span
 * decided on the device from seq_lens, never below min_span_tiles unless
 * forced), so CTAs carry equal work, piece starts included.  A unit cut by
 * range boundaries becomes pieces whose FP32 partials a combine kernel
 * merges.  When the grid is a multiple of Hkv > 1 (grouped-query heads), the
 * KV heads ride on the CTA index instead: the sequence holds the (batch row,
 * row group) units, and CTA c walks the ranges c / Hkv, c / Hkv + grid / Hkv,
 * ... for KV head c % Hkv, so the Hkv CTAs that read one token row's heads
 * run side by side.
 */
typedef struct {
    int32_t group;            /* G = Hq / Hkv */
    int32_t rows_per_unit;    /* NQ: MMA N extent holding the (token, head) rows of one unit */
    int32_t tokens_per_unit;  /* query tokens one unit covers (whole head groups) */
    int32_t heads_per_unit;   /* query heads one unit covers */
    int32_t row_groups;       /* units per (batch row, KV head) */
    int32_t min_span_tiles;   /* fewest KV tiles in one CTA range (the forced span when set) */
    int32_t max_pieces;       /* upper bound of split-KV pieces of one unit */
    int64_t num_units;        /* B * Hkv * row_groups */
    int64_t partial_bytes;    /* rows * max_pieces * (Dv + 1) * 4: FP32 partial rows + LSE */
    int64_t workspace_bytes;  /* partial_bytes + the tile prefix table + alignment */
    int32_t grid;             /* persistent CTAs launched */
} fw_decode_plan_t;

fw_status_t fw_plan_decode(int32_t batch, int32_t q_len, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim_v, int64_t max_kv_len,
                           int32_t num_sms, fw_decode_plan_t *plan);

#ifdef __cplusplus
}
#endif

#endif /* FW_ATTN_H */
