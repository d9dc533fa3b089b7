// Internal interfaces between the C ABI (abi.cu) and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fw {

// Launches `kernel` so that it may start while the previous kernel in the
// stream still runs (programmatic stream serialization); the kernel calls
// pdl_wait() before it reads anything that kernel wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_after_previous(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                         cudaStream_t stream, const Args &...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kKvTile = 128;          // keys per KV tile (MMA M extent in decode, N in prefill)

// Device event counters (the FW_COUNTER_* indices of the C ABI).
constexpr int kCounterPrefillReplays = 0;   // (query row, KV tile) steps the static-anchor check replayed
constexpr int kCounterLatentRescales = 1;   // (query row, key step) steps whose latent anchor moved
constexpr int kNumCounters = 4;
constexpr int kSoftmaxStartWarp = 2;  // decode: warps 2..5 run the softmax / epilogue

constexpr int kDecodeMinSpan = 8;     // decode: fewest KV tiles one CTA range holds (auto mode)
constexpr int kLatentMinSpan = 32;    // latent-head decode: the same, for its heavier tiles
// What starting a piece costs a decode CTA, in KV tiles of streaming (the
// next unit's Q, the pipeline refill, the previous piece's epilogue): a
// clock64 trace of the FP8 kernel puts a piece boundary at ~8,400 cycles
// against ~1,425 per tile inside a piece.  The planned tile sequence gives
// every unit this many empty slots before its tiles, so equal ranges of it
// carry equal work, piece starts included.
constexpr int kDecodePieceCostBf16 = 4;
constexpr int kDecodePieceCostFp8 = 5;
constexpr int kLatentRows = 64;       // latent-head decode: query heads per CTA (MMA N of one CTA)
constexpr int kLatentPairRows = 128;  // latent-head decode on CTA pairs: query heads per pair

// One decode launch, fully resolved on the host.
//
// Scheduling: the (batch row, KV head, row group) units are laid end to end
// in that order, each contributing ceil(n_b / 128) KV tiles; the plan kernel
// writes the exclusive prefix PB[b] of these tile counts per batch row, the
// total T and the range span.  CTA c then processes the global tile ranges
// [r * span, (r + 1) * span) for r = c, c + grid, ...; the part of a unit
// inside one range is a "piece" and writes a split-KV partial unless the unit
// fits in a single range.  With head_ride the KV head leaves the unit: the
// units are (batch row, row group), and CTA c takes KV head c % Hkv over the
// ranges c / Hkv, c / Hkv + grid / Hkv, ...; the Hkv CTAs of one range then
// read the heads of the same token rows at the same time (one DRAM row and,
// for 128-byte FP8 rows, one 256-byte L2 fetch serve two of them).
// KV-cache append ("Writing Page Attention with PyPTO", section 4.3): row
// (b, t, kv head) of the new keys/values goes to cache token row
// layer_base + max(slot_mapping[b * q_len + t], 0).  rows = 0: nothing.
struct AppendParams {
    int64_t rows;                              // B * q_len * Hkv
    int q_len, Hkv, Dk, Dv, ps;
    int kv8;                                   // 1: E4M3 caches, code of x / scale
    float k_scale, v_scale;
    const uint16_t *k_new, *v_new;             // [B, q_len, Hkv, D] bf16; v_new may be null
    int64_t kn_stride[3], vn_stride[3];        // elements (b, t, head); last dim contiguous
    const int32_t *slot_mapping;               // [B * q_len]
    int64_t layer_base, cache_rows;            // token rows; cache_rows = pages * ps
    void *k_cache, *v_cache;                   // [pages, ps, Hkv, D]
    int64_t kc_stride[3], vc_stride[3];        // elements (page, slot, head)
};

struct DecodeParams {
    int B, q_len, Hq, Hkv, G, ps, max_pages, num_pages;
    int head_mode;        // 0: a unit holds whole head groups for tokens_per_unit tokens;
                          // 1: a unit holds `rows` consecutive heads of one token
    int rows;             // NQ: padded MMA N extent
    int tokens_per_unit, heads_per_unit, head_chunks, row_groups, units_per_row;
    int forced_span;      // KV tiles per range, 0 = auto
    int min_span;         // lower bound of the auto span
    int max_pieces;       // workspace slots per query row
    int grid;             // CTAs of the attention kernel
    int range_groups;     // 1: CTA c takes ranges c, c + grid, ...; R > 1: the R row groups of
                          // a unit ride on the CTA index (CTA c runs row group c % R over ranges
                          // c / R, c / R + grid / R, ...), so they read the same keys together
    int Dv;
    int packed;           // latent heads: 1 when q rows are read through the flattened (token, head)
                          // axis (one KV head, q contiguous over it): a row group is `rows` consecutive
                          // packed rows t * Hq + h and may straddle tokens ("TokenSpeed-MLA 2.0.1",
                          // packed-query paragraph); 0: one token's heads per row group
    int window_left;      // < 0: none; else token t sees keys max(0, n - q_len + t - W) .. n - q_len + t
    int causal;           // 1: token t sees keys up to its own position n - q_len + t; 0: all n keys
    AppendParams app;     // appended by the plan launch's extra blocks before the attention reads
    int32_t *plan;        // [0] = T, [1] = span, [2 .. 2 + B] = PB
    const int32_t *block_table; int64_t bt_stride;
    const int32_t *seq_lens;
    void *out; int64_t out_stride[4];          // [B, q_len, Hq, Dv] bf16
    float *lse; int64_t lse_stride[3];         // [B, q_len, Hq] or nullptr
    float *ws_o;                               // [B*q_len*Hq, max_pieces, Dv]
    float *ws_lse;                             // [B*q_len*Hq, max_pieces] (log2 units)
    float scale_log2;                          // scale * log2(e) (times k_scale for an FP8 cache)
    float out_scale;                           // v_scale for an FP8 cache, else 1
    uint64_t timeout_ns;
    int *status;                               // device status word
    unsigned long long *counters;              // device event counters (FW_COUNTER_*)
    int test_stall;                            // test hook: the producer first waits on a barrier nothing completes
    int piece_cost;                            // empty slots before each unit's tiles in the planned sequence
    int head_ride;        // 1: the KV heads ride on the CTA index (CTA c runs KV head c % Hkv over
                          // ranges c / Hkv, c / Hkv + grid / Hkv, ... of the (batch row, row group)
                          // units), so the Hkv CTAs reading one token row's heads run side by side
};

// One varlen prefill launch.  The plan kernel lists the units (sequence,
// query head, pair of consecutive 128-row query tiles) longest first; the
// CTAs (CTA pairs at head dim 256) take list entries in that order as they
// free up, from a counter in the plan.
struct PrefillParams {
    int B, Hq, Hkv, G, causal, Dv;
    int online;           // 0: static anchor with check and replay; 1: online softmax, conditional rescale
    int64_t total_q, total_k;
    const int32_t *cu_q, *cu_k;
    void *out; int64_t out_stride[3];          // [total_q, Hq, Dv] bf16
    float *lse; int64_t lse_stride[2];         // [total_q, Hq] or nullptr
    float scale_log2;
    uint64_t timeout_ns;
    int *status;
    unsigned long long *counters;              // device event counters (FW_COUNTER_*)
    int32_t *plan;        // [0] = entries, [1] = pairs, [2 .. 2 + B] = pair prefix PP, [3 + B] = next entry
                          // to hand out (CTAs take entries in list order as they free up)
    int32_t *list;        // entries pair_index * Hq + head, sorted by cost, longest first
    int64_t list_capacity;
    int grid;
};

// plan kernel + attention kernel + combine kernel, in stream order
cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                          const CUtensorMap &tm_v, int head_dim, cudaStream_t stream,
                          cudaEvent_t timing_start, cudaEvent_t timing_stop, int *launches);
size_t decode_smem_bytes(int head_dim, int rows);
cudaError_t launch_decode_plan(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_decode_combine(const DecodeParams &p, int head_dim_v, cudaStream_t stream);
// Standalone KV-cache append (the fused form runs inside launch_decode_plan).
cudaError_t launch_kv_append(const AppendParams &a, int *status, cudaStream_t stream);

// Latent-head decode (Dk = 576, Dv = 512, row groups of 64 query heads):
// plan kernel + attention kernel + combine kernel, in stream order
cudaError_t launch_latent_decode(const DecodeParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                 const CUtensorMap &tm_v, cudaStream_t stream, cudaEvent_t timing_start,
                                 cudaEvent_t timing_stop, int *launches);
size_t latent_decode_smem_bytes();

// The same on CTA pairs (row groups of 128 query heads, cta_group::2 MMAs)
cudaError_t launch_latent_pair_decode(const DecodeParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                      const CUtensorMap &tm_v, cudaStream_t stream, cudaEvent_t timing_start,
                                      cudaEvent_t timing_stop, int *launches);
size_t latent_pair_decode_smem_bytes();

// Decode over an FP8 E4M3 KV cache (Dk = Dv = 128): plan + attention + combine
cudaError_t launch_decode_fp8(const DecodeParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, cudaStream_t stream, cudaEvent_t timing_start,
                              cudaEvent_t timing_stop, int *launches);

// plan kernel + attention kernel, in stream order
cudaError_t launch_prefill(const PrefillParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                           const CUtensorMap &tm_v, int head_dim, cudaStream_t stream,
                           cudaEvent_t timing_start, cudaEvent_t timing_stop, int *launches);

}  // namespace fw
