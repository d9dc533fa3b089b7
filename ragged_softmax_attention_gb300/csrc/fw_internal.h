// Internal interfaces between the C ABI (abi.cu) and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fw {

constexpr int kKvTile = 128;          // keys per KV tile (MMA M extent in decode, N in prefill)
constexpr int kSoftmaxStartWarp = 2;  // decode: warps 2..5 run the softmax / epilogue

// One decode launch, fully resolved on the host.
struct DecodeParams {
    int B, q_len, Hq, Hkv, G, ps, max_pages, num_pages;
    int head_mode;        // 0: a unit holds whole head groups for tokens_per_unit tokens;
                          // 1: a unit holds `rows` consecutive heads of one token
    int rows;             // NQ: padded MMA N extent
    int tokens_per_unit, heads_per_unit, head_chunks, row_groups;
    int chunk_tokens, max_splits;
    int64_t num_units;
    const int32_t *block_table; int64_t bt_stride;
    const int32_t *seq_lens;
    void *out; int64_t out_stride[4];          // [B, q_len, Hq, Dv] bf16
    float *lse; int64_t lse_stride[3];         // [B, q_len, Hq] or nullptr
    float *ws_o;                               // [B*q_len*Hq, max_splits, Dv]
    float *ws_lse;                             // [B*q_len*Hq, max_splits] (log2 units)
    float scale_log2;                          // scale * log2(e)
    uint64_t timeout_ns;
    int *status;                               // device status word
};

struct CombineParams {
    int B, q_len, Hq, Dv, chunk_tokens, max_splits;
    const int32_t *seq_lens;
    const float *ws_o, *ws_lse;
    void *out; int64_t out_stride[4];
    float *lse; int64_t lse_stride[3];
    int max_kv_len;
};

struct PrefillParams {
    int B, Hq, Hkv, G, causal;
    int64_t total_q, total_k;
    const int32_t *cu_q, *cu_k;
    void *out; int64_t out_stride[3];          // [total_q, Hq, Dv] bf16
    float *lse; int64_t lse_stride[2];
    float scale_log2;
    uint64_t timeout_ns;
    int *status;
    int32_t *work_counter;                      // zeroed before launch
    const int32_t *work_list;                   // planned (seq, q_tile) list, longest first
    int32_t *work_count;                        // number of entries (device)
    int max_q_tiles;
};

cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                          const CUtensorMap &tm_v, int head_dim, int grid, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream);
size_t decode_smem_bytes(int head_dim, int rows);

cudaError_t launch_prefill(const PrefillParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                           const CUtensorMap &tm_v, int head_dim, int grid, int64_t plan_entries,
                           cudaStream_t stream);
cudaError_t launch_prefill_plan(const PrefillParams &p, int32_t *work_list, int32_t *work_count,
                                int64_t capacity, cudaStream_t stream);

}  // namespace fw
