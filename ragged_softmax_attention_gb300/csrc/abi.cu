// C ABI of the library: argument validation, planning, tensor-map encoding,
// workspace and status-word management, and kernel launches.  Every entry
// point is declared and documented in include/fw_attn.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "fw_attn.h"
#include "fw_internal.h"

namespace {

__device__ int g_fw_status = 0;
__device__ unsigned long long g_fw_counters[fw::kNumCounters];

constexpr int kMaxDevices = 64;

thread_local char t_error[512] = "";

fw_status_t fail(fw_status_t st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_error, sizeof t_error, fmt, ap);
    va_end(ap);
    return st;
}

fw_status_t ok() {
    t_error[0] = '\0';
    return FW_OK;
}

struct DeviceState {
    bool init = false;
    int num_sms = 0;
    int *status = nullptr;          // device address of g_fw_status
    unsigned long long *counters = nullptr;  // device address of g_fw_counters
    void *ws = nullptr;             // internal workspace
    size_t ws_bytes = 0;
    void *user_ws = nullptr;        // caller workspace
    size_t user_ws_bytes = 0;
    void *noalloc_scratch = nullptr; // device address of g_noalloc_scratch on this device
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<int64_t> g_launches{0};
int64_t g_opt_chunk = 0;
int64_t g_opt_timeout_ms = 2000;
int64_t g_opt_timing = 0;
int64_t g_opt_max_ctas = 0;
int64_t g_opt_prefill_online = 0;
int64_t g_opt_test_stall = 0;

struct TimedLaunch { cudaEvent_t a, b; };
std::vector<TimedLaunch> g_timed;      // pending event pairs
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pooled_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

fw_status_t device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FW_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(FW_ERR_UNSUPPORTED, "device index %d out of range", dev);
    DeviceState &d = g_dev[dev];
    if (!d.init) {
        e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(FW_ERR_CUDA, "multiprocessor count: %s", cudaGetErrorString(e));
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return fail(FW_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300); device %d is sm_%d%d",
                        dev, major, minor);
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_fw_status);
        if (e != cudaSuccess) return fail(FW_ERR_CUDA, "status word address: %s", cudaGetErrorString(e));
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.counters), g_fw_counters);
        if (e != cudaSuccess) return fail(FW_ERR_CUDA, "counter address: %s", cudaGetErrorString(e));
        d.init = true;
    }
    *out = &d;
    return FW_OK;
}

// ---------------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

fw_status_t get_encoder() {
    if (g_encode) return FW_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(FW_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return FW_OK;
}

// Tensor map with 128-byte swizzle; dims/strides innermost first, strides
// in bytes for dims 1..rank-1.  L2 fetches are promoted to 256 bytes unless
// the caller knows the other half of each 256-byte block is someone else's.
fw_status_t encode_map(CUtensorMap *tm, CUtensorMapDataType type, const void *base, int rank, const uint64_t *dims,
                       const uint64_t *strides_bytes, const uint32_t *box, const char *what,
                       CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
    if (fw_status_t s = get_encoder()) return s;
    uint32_t elem[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(tm, type, (cuuint32_t)rank, const_cast<void *>(base),
                          dims, strides_bytes, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FW_ERR_INVALID_ARG, "tensor map for %s rejected (CUresult %d)", what, (int)r);
    return FW_OK;
}

fw_status_t encode_bf16(CUtensorMap *tm, const void *base, int rank, const uint64_t *dims,
                        const uint64_t *strides_bytes, const uint32_t *box, const char *what) {
    return encode_map(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes, box, what);
}

// ----------------------------------------------------------------- validation

const char *dtype_name(int32_t d) {
    switch (d) {
        case FW_BF16: return "bf16"; case FW_F32: return "f32"; case FW_I32: return "i32";
        case FW_FP8_E4M3: return "fp8_e4m3"; default: return "?";
    }
}

fw_status_t check_tensor(const fw_tensor_t *t, const char *name, int ndim, int32_t dtype, bool allow_null = false) {
    if (!t) return allow_null ? FW_OK : fail(FW_ERR_INVALID_ARG, "%s is NULL", name);
    if (t->ndim != ndim) return fail(FW_ERR_INVALID_ARG, "%s: expected %d dims, got %d", name, ndim, t->ndim);
    if (t->dtype != dtype)
        return fail(FW_ERR_INVALID_ARG, "%s: expected dtype %s, got %s", name, dtype_name(dtype), dtype_name(t->dtype));
    int64_t numel = 1;
    for (int i = 0; i < ndim; ++i) {
        if (t->shape[i] < 0) return fail(FW_ERR_INVALID_ARG, "%s: negative extent", name);
        if (t->stride[i] < 0) return fail(FW_ERR_INVALID_ARG, "%s: negative stride", name);
        numel *= t->shape[i];
    }
    if (numel > 0 && !t->data) return fail(FW_ERR_INVALID_ARG, "%s: NULL data", name);
    if (numel > 0 && t->stride[ndim - 1] != 1 && t->shape[ndim - 1] > 1)
        return fail(FW_ERR_INVALID_ARG, "%s: last dimension must be contiguous", name);
    return FW_OK;
}

// Tensors read through the tensor memory accelerator: 16-byte aligned base,
// every outer stride a multiple of 16 bytes (8 BF16 or 16 FP8 elements).
fw_status_t check_tma_layout(const fw_tensor_t *t, const char *name) {
    if (reinterpret_cast<uintptr_t>(t->data) % 16 != 0)
        return fail(FW_ERR_INVALID_ARG, "%s: base pointer must be 16-byte aligned", name);
    const int64_t per16 = t->dtype == FW_FP8_E4M3 ? 16 : 8;
    for (int i = 0; i + 1 < t->ndim; ++i)
        if (t->stride[i] % per16 != 0)
            return fail(FW_ERR_INVALID_ARG, "%s: stride[%d] = %lld is not a multiple of %lld elements", name, i,
                        (long long)t->stride[i], (long long)per16);
    return FW_OK;
}

fw_status_t check_output_layout(const fw_tensor_t *t, const char *name) {
    if (reinterpret_cast<uintptr_t>(t->data) % 16 != 0)
        return fail(FW_ERR_INVALID_ARG, "%s: base pointer must be 16-byte aligned", name);
    for (int i = 0; i + 1 < t->ndim; ++i)
        if (t->stride[i] % 2 != 0)
            return fail(FW_ERR_INVALID_ARG, "%s: stride[%d] must be even", name, i);
    return FW_OK;
}

bool supported_page_size(int64_t ps) {
    if (ps == 8 || ps == 16 || ps == 32 || ps == 64 || ps == 128) return true;
    return ps > 128 && ps % 128 == 0 && ps <= (1 << 20);
}

// --------------------------------------------------------------------- planner

fw_status_t plan_decode(int32_t B, int32_t q_len, int32_t Hq, int32_t Hkv, int32_t Dv, int64_t max_kv_len,
                        int32_t num_sms, fw_decode_plan_t *pl) {
    if (B < 0 || q_len < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_kv_len < 0 || Dv < 1)
        return fail(FW_ERR_INVALID_ARG, "invalid decode shapes");
    if (num_sms <= 0) return fail(FW_ERR_INVALID_ARG, "num_sms must be positive");
    fw_decode_plan_t p{};
    const int G = Hq / Hkv;
    p.group = G;
    const bool latent = (Dv == 512);
    if (latent) {
        // Latent heads (Dk = 576, Dv = 512): a row group is `rows` consecutive
        // query rows of a (batch row, KV head) unit -- 128 on a CTA pair, 64
        // on one CTA -- whose q_len * G / rows row groups share its tile
        // ranges and ride on the worker (pair or CTA) index.  With one KV head
        // the rows are packed (token, head) rows t * G + h ("TokenSpeed-MLA
        // 2.0.1", packed-query paragraph): ceil(q_len * G / rows) groups, only
        // the last one padded.  With several KV heads a group holds one
        // token's heads, so G must be a multiple of 64.
        int rows;
        if (Hkv == 1)
            rows = (int64_t)q_len * G >= fw::kLatentPairRows ? fw::kLatentPairRows : fw::kLatentRows;
        else if (G % fw::kLatentRows == 0)
            rows = G % fw::kLatentPairRows == 0 ? fw::kLatentPairRows : fw::kLatentRows;
        else
            return fail(FW_ERR_UNSUPPORTED, "latent decode with several KV heads needs the query heads per KV "
                        "head (%d) to be a multiple of %d", G, fw::kLatentRows);
        p.tokens_per_unit = 1;
        p.heads_per_unit = rows;
        p.rows_per_unit = rows;
        p.row_groups = (int32_t)(((int64_t)q_len * G + rows - 1) / rows);
        const int ctas_per_group = rows == fw::kLatentPairRows ? 2 : 1;
        if ((int64_t)p.row_groups * ctas_per_group > num_sms)
            return fail(FW_ERR_UNSUPPORTED, "more row groups than SMs");
    } else
    // Fold query tokens next to the heads of a KV group: the largest F that
    // divides q_len with G * F within the 32-row N budget ("TokenSpeed-MLA
    // 2.0.1", fold_sq_factor, with 32 rows instead of 128 because here the
    // query rows sit on the MMA N axis).  Groups wider than 32 heads are cut
    // into 32-head chunks, one token each.
    if (G <= 32) {
        int F = 1;
        for (int f = 1; f <= q_len; ++f)
            if (q_len % f == 0 && G * f <= 32) F = f;
        p.tokens_per_unit = F;
        p.heads_per_unit = G;
        p.rows_per_unit = G * F <= 16 ? 16 : 32;
        p.row_groups = q_len / F;
    } else {
        p.tokens_per_unit = 1;
        p.heads_per_unit = 32;
        p.rows_per_unit = 32;
        p.row_groups = q_len * ((G + 31) / 32);
    }
    p.num_units = (int64_t)B * Hkv * p.row_groups;
    const int64_t tiles_max = (max_kv_len + fw::kKvTile - 1) / fw::kKvTile;
    if (p.num_units * ((tiles_max > 0 ? tiles_max : 1) + fw::kDecodePieceCostFp8) >= (1LL << 31))
        return fail(FW_ERR_UNSUPPORTED, "decode too large for 32-bit tile indices");
    int64_t span = g_opt_chunk > 0 ? (g_opt_chunk + fw::kKvTile - 1) / fw::kKvTile
                                   : (latent ? fw::kLatentMinSpan : fw::kDecodeMinSpan);
    p.min_span_tiles = (int32_t)span;
    // A unit of t tiles meets at most ceil(t / span) + 1 ranges.
    p.max_pieces = (int32_t)((tiles_max + span - 1) / span + 1);
    const int64_t rows = (int64_t)B * q_len * Hq;
    p.partial_bytes = rows * p.max_pieces * (int64_t)(Dv + 1) * 4;
    const int64_t plan_bytes = ((B + 3) * 4 + 255) / 256 * 256;
    const int64_t o_bytes = (rows * p.max_pieces * (int64_t)Dv * 4 + 255) / 256 * 256;
    p.workspace_bytes = plan_bytes + o_bytes + rows * p.max_pieces * 4;
    int64_t grid = num_sms;
    if (g_opt_max_ctas > 0 && grid > g_opt_max_ctas) grid = g_opt_max_ctas;
    if (latent) {
        // whole groups of row-group workers (a worker is a CTA pair at 128 rows)
        const int64_t per = (int64_t)p.row_groups * (p.rows_per_unit == fw::kLatentPairRows ? 2 : 1);
        grid = grid / per * per;
        if (grid < per) grid = per;
    }
    p.grid = (int32_t)(grid > 0 ? grid : 1);
    *pl = p;
    return FW_OK;
}

fw_status_t get_workspace(DeviceState *d, size_t bytes, cudaStream_t stream, void **ptr) {
    *ptr = nullptr;
    if (bytes == 0) return FW_OK;
    if (d->user_ws) {
        if (d->user_ws_bytes < bytes)
            return fail(FW_ERR_WORKSPACE, "caller workspace holds %zu bytes, %zu needed", d->user_ws_bytes, bytes);
        *ptr = d->user_ws;
        return FW_OK;
    }
    if (d->ws_bytes < bytes) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaStreamIsCapturing(stream, &cs);
        if (cs != cudaStreamCaptureStatusNone)
            return fail(FW_ERR_WORKSPACE, "workspace must grow to %zu bytes during stream capture; "
                        "make one call with these shapes before capturing", bytes);
        if (d->ws) cudaFree(d->ws);
        d->ws = nullptr;
        d->ws_bytes = 0;
        cudaError_t e = cudaMalloc(&d->ws, bytes);
        if (e != cudaSuccess) return fail(FW_ERR_WORKSPACE, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
        d->ws_bytes = bytes;
    }
    *ptr = d->ws;
    return FW_OK;
}

}  // namespace

// ============================================================== entry points

extern "C" {

const char *fw_last_error(void) { return t_error; }

int64_t fw_launch_count(void) { return g_launches.load(); }

fw_status_t fw_set_option(int32_t option, int64_t value) {
    std::lock_guard<std::mutex> lk(g_mu);
    switch (option) {
        case FW_OPT_DECODE_CHUNK_TOKENS:
            if (value < 0 || value % fw::kKvTile) return fail(FW_ERR_INVALID_ARG, "chunk must be a multiple of 128");
            g_opt_chunk = value; return ok();
        case FW_OPT_WAIT_TIMEOUT_MS:
            if (value < 1) return fail(FW_ERR_INVALID_ARG, "timeout must be positive");
            g_opt_timeout_ms = value; return ok();
        case FW_OPT_KERNEL_TIMING: g_opt_timing = value ? 1 : 0; return ok();
        case FW_OPT_MAX_CTAS:
            if (value < 0) return fail(FW_ERR_INVALID_ARG, "max CTAs must be >= 0");
            g_opt_max_ctas = value; return ok();
        case FW_OPT_PREFILL_SOFTMAX:
            if (value != 0 && value != 1) return fail(FW_ERR_INVALID_ARG, "prefill softmax mode must be 0 or 1");
            g_opt_prefill_online = value; return ok();
        case FW_OPT_TEST_STALL: g_opt_test_stall = value ? 1 : 0; return ok();
        default: return fail(FW_ERR_INVALID_ARG, "unknown option %d", option);
    }
}

fw_status_t fw_kernel_timing_read(double *total_ms, int64_t *launches) {
    std::lock_guard<std::mutex> lk(g_mu);
    double sum = 0.0;
    int64_t n = 0;
    for (auto &t : g_timed) {
        cudaError_t e = cudaEventSynchronize(t.b);
        float ms = 0.f;
        if (e == cudaSuccess && cudaEventElapsedTime(&ms, t.a, t.b) == cudaSuccess) { sum += ms; ++n; }
        g_event_pool.push_back(t.a);
        g_event_pool.push_back(t.b);
    }
    g_timed.clear();
    if (total_ms) *total_ms = sum;
    if (launches) *launches = n;
    return ok();
}

fw_status_t fw_plan_decode(int32_t batch, int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim_v, int64_t max_kv_len, int32_t num_sms, fw_decode_plan_t *plan) {
    if (!plan) return fail(FW_ERR_INVALID_ARG, "plan is NULL");
    std::lock_guard<std::mutex> lk(g_mu);
    if (num_sms <= 0) {
        DeviceState *d = nullptr;
        if (fw_status_t s = device_state(&d)) return s;
        num_sms = d->num_sms;
    }
    if (fw_status_t s = plan_decode(batch, q_len, num_q_heads, num_kv_heads, head_dim_v, max_kv_len, num_sms, plan))
        return s;
    return ok();
}

fw_status_t fw_set_workspace(void *ptr, size_t bytes, fw_stream_t stream) {
    (void)stream;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState *d = nullptr;
    if (fw_status_t s = device_state(&d)) return s;
    if (!ptr && bytes) return fail(FW_ERR_INVALID_ARG, "NULL workspace with nonzero size");
    if (ptr && reinterpret_cast<uintptr_t>(ptr) % 256 != 0)
        return fail(FW_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    d->user_ws = ptr;
    d->user_ws_bytes = ptr ? bytes : 0;
    return ok();
}

fw_status_t fw_get_device_status(fw_stream_t stream, int32_t *code) {
    if (!code) return fail(FW_ERR_INVALID_ARG, "code is NULL");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState *d = nullptr;
    if (fw_status_t s = device_state(&d)) return s;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(FW_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    int v = 0;
    e = cudaMemcpy(&v, d->status, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(FW_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    const int zero = 0;
    cudaMemcpy(d->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    *code = v;
    return ok();
}

fw_status_t fw_read_counters(fw_stream_t stream, int64_t *values, int32_t n) {
    if (!values || n < 1 || n > fw::kNumCounters) return fail(FW_ERR_INVALID_ARG, "need 1 to %d counters", fw::kNumCounters);
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState *d = nullptr;
    if (fw_status_t s = device_state(&d)) return s;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(FW_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    unsigned long long v[fw::kNumCounters] = {};
    e = cudaMemcpy(v, d->counters, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(FW_ERR_CUDA, "counter read: %s", cudaGetErrorString(e));
    const unsigned long long zero[fw::kNumCounters] = {};
    e = cudaMemcpy(d->counters, zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(FW_ERR_CUDA, "counter reset: %s", cudaGetErrorString(e));
    for (int i = 0; i < n; ++i) values[i] = (int64_t)v[i];
    return ok();
}

static fw_status_t decode_shapes(const fw_tensor_t *q, const fw_tensor_t *k_cache, const fw_tensor_t *v_cache,
                                 const fw_tensor_t *block_table) {
    if (fw_status_t s = check_tensor(q, "q", 4, FW_BF16)) return s;
    // BF16 caches, or FP8 caches (fw_paged_decode_fp8): both of one type
    const int32_t kv_type = k_cache && k_cache->dtype == FW_FP8_E4M3 ? FW_FP8_E4M3 : FW_BF16;
    if (fw_status_t s = check_tensor(k_cache, "k_cache", 4, kv_type)) return s;
    if (fw_status_t s = check_tensor(v_cache, "v_cache", 4, kv_type)) return s;
    if (fw_status_t s = check_tensor(block_table, "block_table", 2, FW_I32)) return s;
    const int64_t B = q->shape[0], Hq = q->shape[2], Dk = q->shape[3];
    const int64_t P = k_cache->shape[0], ps = k_cache->shape[1], Hkv = k_cache->shape[2];
    if (k_cache->shape[3] != Dk) return fail(FW_ERR_INVALID_ARG, "k_cache head dim %lld != q head dim %lld",
                                             (long long)k_cache->shape[3], (long long)Dk);
    if (v_cache->shape[0] != P || v_cache->shape[1] != ps || v_cache->shape[2] != Hkv)
        return fail(FW_ERR_INVALID_ARG, "v_cache [P, ps, Hkv] must match k_cache");
    if (block_table->shape[0] != B) return fail(FW_ERR_INVALID_ARG, "block_table rows != batch");
    if (block_table->shape[1] > 0 && block_table->stride[1] != 1)
        return fail(FW_ERR_INVALID_ARG, "block_table rows must be contiguous");
    if (Hkv < 1 || Hq % Hkv != 0) return fail(FW_ERR_INVALID_ARG, "Hq (%lld) must be a multiple of Hkv (%lld)",
                                              (long long)Hq, (long long)Hkv);
    if (ps < 1) return fail(FW_ERR_INVALID_ARG, "page size must be positive");
    return FW_OK;
}

fw_status_t fw_paged_decode_workspace_size(const fw_tensor_t *q, const fw_tensor_t *k_cache,
                                           const fw_tensor_t *v_cache, const fw_tensor_t *block_table,
                                           size_t *bytes) {
    if (!bytes) return fail(FW_ERR_INVALID_ARG, "bytes is NULL");
    if (fw_status_t s = decode_shapes(q, k_cache, v_cache, block_table)) return s;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState *d = nullptr;
    if (fw_status_t s = device_state(&d)) return s;
    fw_decode_plan_t pl;
    const int64_t max_kv = block_table->shape[1] * k_cache->shape[1];
    if (fw_status_t s = plan_decode((int32_t)q->shape[0], (int32_t)q->shape[1], (int32_t)q->shape[2],
                                    (int32_t)k_cache->shape[2], (int32_t)v_cache->shape[3], max_kv, d->num_sms, &pl))
        return s;
    *bytes = (size_t)pl.workspace_bytes;
    return ok();
}

// Host side of a KV-cache append: the new rows, their slots, the layer base.
struct AppendArgs {
    const fw_tensor_t *k_new, *v_new, *slot_mapping;
    int64_t layer_base_rows;
};

// Validates an append into [pages, ps, Hkv, D] caches and fills the kernel's
// parameters ("Writing Page Attention with PyPTO", section 4.3).
static fw_status_t build_append(const AppendArgs &aa, const fw_tensor_t *k_cache, const fw_tensor_t *v_cache,
                                float k_scale, float v_scale, fw::AppendParams *ap) {
    if (!k_cache) return fail(FW_ERR_INVALID_ARG, "k_cache is NULL");
    const bool kv8 = k_cache->dtype == FW_FP8_E4M3;
    if (!kv8 && k_cache->dtype != FW_BF16) return fail(FW_ERR_INVALID_ARG, "caches must be BF16 or FP8_E4M3");
    if (fw_status_t s = check_tensor(k_cache, "k_cache", 4, k_cache->dtype)) return s;
    if (fw_status_t s = check_tensor(aa.k_new, "k_new", 4, FW_BF16)) return s;
    if ((aa.v_new == nullptr) != (v_cache == nullptr))
        return fail(FW_ERR_INVALID_ARG, "v_new and v_cache go together (both or neither)");
    if (v_cache) {
        if (fw_status_t s = check_tensor(v_cache, "v_cache", 4, k_cache->dtype)) return s;
        if (fw_status_t s = check_tensor(aa.v_new, "v_new", 4, FW_BF16)) return s;
    }
    const fw_tensor_t *sm = aa.slot_mapping;
    if (!sm || sm->dtype != FW_I32 || sm->ndim < 1 || sm->ndim > 2)
        return fail(FW_ERR_INVALID_ARG, "slot_mapping must be an I32 [B * q_len] or [B, q_len] tensor");
    const int64_t B = aa.k_new->shape[0], q_len = aa.k_new->shape[1], Hkv = aa.k_new->shape[2];
    const int64_t Dk = aa.k_new->shape[3];
    const int64_t P = k_cache->shape[0], ps = k_cache->shape[1];
    const int64_t sm_n = sm->ndim == 1 ? sm->shape[0] : sm->shape[0] * sm->shape[1];
    const bool sm_contig = sm->ndim == 1 ? (sm->shape[0] <= 1 || sm->stride[0] == 1)
                                         : ((sm->shape[1] <= 1 || sm->stride[1] == 1) &&
                                            (sm->shape[0] <= 1 || sm->stride[0] == sm->shape[1]));
    if (sm_n != B * q_len || !sm_contig || (sm_n > 0 && !sm->data))
        return fail(FW_ERR_INVALID_ARG, "slot_mapping must hold B * q_len contiguous entries");
    if (k_cache->shape[2] != Hkv || k_cache->shape[3] != Dk)
        return fail(FW_ERR_INVALID_ARG, "k_new [B, q_len, Hkv, D] does not match k_cache [pages, ps, Hkv, D]");
    int64_t Dv = 0;
    if (v_cache) {
        Dv = aa.v_new->shape[3];
        if (aa.v_new->shape[0] != B || aa.v_new->shape[1] != q_len || aa.v_new->shape[2] != Hkv ||
            v_cache->shape[0] != P || v_cache->shape[1] != ps || v_cache->shape[2] != Hkv || v_cache->shape[3] != Dv)
            return fail(FW_ERR_INVALID_ARG, "v_new / v_cache shapes do not match k_new / k_cache");
    }
    if (Dk < 8 || Dk % 8 || (v_cache && (Dv < 8 || Dv % 8)))
        return fail(FW_ERR_UNSUPPORTED, "appended head dims must be positive multiples of 8");
    if (P < 1 || ps < 1) return fail(FW_ERR_INVALID_ARG, "empty cache");
    if (aa.layer_base_rows < 0 || aa.layer_base_rows >= P * ps)
        return fail(FW_ERR_INVALID_ARG, "layer_base_rows %lld outside the cache's %lld token rows",
                    (long long)aa.layer_base_rows, (long long)(P * ps));
    if (kv8 && !(std::isfinite(k_scale) && std::isfinite(v_scale) && k_scale > 0.f && v_scale > 0.f))
        return fail(FW_ERR_INVALID_ARG, "k_scale and v_scale must be finite and positive");
    if (!kv8 && (k_scale != 1.f || v_scale != 1.f))
        return fail(FW_ERR_INVALID_ARG, "k_scale and v_scale must be 1 for BF16 caches");
    if (B * q_len > 0) {
        if (fw_status_t s = check_tma_layout(aa.k_new, "k_new")) return s;
        if (fw_status_t s = check_tma_layout(k_cache, "k_cache")) return s;
        if (v_cache) {
            if (fw_status_t s = check_tma_layout(aa.v_new, "v_new")) return s;
            if (fw_status_t s = check_tma_layout(v_cache, "v_cache")) return s;
        }
    }
    fw::AppendParams a{};
    a.rows = B * q_len * Hkv;
    a.q_len = (int)q_len; a.Hkv = (int)Hkv; a.Dk = (int)Dk; a.Dv = (int)Dv; a.ps = (int)ps;
    a.kv8 = kv8 ? 1 : 0;
    a.k_scale = k_scale; a.v_scale = v_scale;
    a.k_new = static_cast<const uint16_t *>(aa.k_new->data);
    a.v_new = v_cache ? static_cast<const uint16_t *>(aa.v_new->data) : nullptr;
    for (int i = 0; i < 3; ++i) {
        a.kn_stride[i] = aa.k_new->stride[i];
        a.vn_stride[i] = v_cache ? aa.v_new->stride[i] : 0;
        a.kc_stride[i] = k_cache->stride[i];
        a.vc_stride[i] = v_cache ? v_cache->stride[i] : 0;
    }
    a.slot_mapping = static_cast<const int32_t *>(sm->data);
    a.layer_base = aa.layer_base_rows;
    a.cache_rows = P * ps;
    a.k_cache = k_cache->data;
    a.v_cache = v_cache ? v_cache->data : nullptr;
    *ap = a;
    return FW_OK;
}

// Shared body of the decode entry points.  `fixed_ws` selects where the
// scratch comes from: nullptr = the workspace fw_set_workspace() set or the
// internal buffer (fw_paged_decode); otherwise that device range of
// `fixed_bytes` bytes, which is never grown (fw_paged_decode_noalloc).
static fw_status_t paged_decode_impl(const fw_tensor_t *q, const fw_tensor_t *k_cache, const fw_tensor_t *v_cache,
                                     const fw_tensor_t *block_table, const fw_tensor_t *seq_lens, float scale,
                                     fw_tensor_t *out, fw_tensor_t *lse, fw_stream_t stream_,
                                     void *(*fixed_ws)(DeviceState *, fw_status_t *), size_t fixed_bytes,
                                     bool kv8 = false, float k_scale = 1.f, float v_scale = 1.f,
                                     int32_t window_left = -1, bool any_cache = false,
                                     const AppendArgs *append = nullptr, bool causal = true) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    // A fused append writes the packed cache at layer_base + max(slot, 0); the
    // attention then reads the layer's pages, a view from layer_base on.
    fw::AppendParams app{};
    fw_tensor_t k_view, v_view;
    if (append) {
        if (fw_status_t s = build_append(*append, k_cache, v_cache, k_scale, v_scale, &app)) return s;
        if (append->layer_base_rows % k_cache->shape[1] != 0)
            return fail(FW_ERR_INVALID_ARG, "layer_base_rows must be a multiple of the page size");
        const int64_t first_page = append->layer_base_rows / k_cache->shape[1];
        const int64_t esz = k_cache->dtype == FW_FP8_E4M3 ? 1 : 2;
        k_view = *k_cache;
        v_view = *v_cache;
        k_view.data = static_cast<char *>(k_cache->data) + first_page * k_cache->stride[0] * esz;
        v_view.data = static_cast<char *>(v_cache->data) + first_page * v_cache->stride[0] * esz;
        k_view.shape[0] -= first_page;
        v_view.shape[0] -= first_page;
        k_cache = &k_view;
        v_cache = &v_view;
    }
    if (fw_status_t s = decode_shapes(q, k_cache, v_cache, block_table)) return s;
    if (any_cache) kv8 = k_cache->dtype == FW_FP8_E4M3;
    if (kv8 != (k_cache->dtype == FW_FP8_E4M3))
        return fail(FW_ERR_INVALID_ARG, kv8 ? "fw_paged_decode_fp8 takes FP8_E4M3 caches"
                                            : "FP8 caches go through fw_paged_decode_fp8");
    if (!kv8 && (k_scale != 1.f || v_scale != 1.f))
        return fail(FW_ERR_INVALID_ARG, "k_scale and v_scale must be 1 for BF16 caches");
    if (window_left < -1) return fail(FW_ERR_INVALID_ARG, "window_left must be -1 (no window) or >= 0");
    if (kv8 && !(std::isfinite(k_scale) && std::isfinite(v_scale) && k_scale > 0.f && v_scale > 0.f))
        return fail(FW_ERR_INVALID_ARG, "k_scale and v_scale must be finite and positive");
    if (fw_status_t s = check_tensor(seq_lens, "seq_lens", 1, FW_I32)) return s;
    if (fw_status_t s = check_tensor(out, "out", 4, FW_BF16)) return s;
    if (fw_status_t s = check_tensor(lse, "lse", 3, FW_F32, true)) return s;
    const int64_t B = q->shape[0], q_len = q->shape[1], Hq = q->shape[2], Dk = q->shape[3];
    const int64_t P = k_cache->shape[0], ps = k_cache->shape[1], Hkv = k_cache->shape[2];
    const int64_t Dv = v_cache->shape[3];
    const int64_t max_pages = block_table->shape[1];
    if (seq_lens->shape[0] != B || (B > 0 && seq_lens->stride[0] != 1))
        return fail(FW_ERR_INVALID_ARG, "seq_lens must be a contiguous [B] vector");
    if (out->shape[0] != B || out->shape[1] != q_len || out->shape[2] != Hq || out->shape[3] != Dv)
        return fail(FW_ERR_INVALID_ARG, "out must be [B, q_len, Hq, Dv]");
    if (lse && (lse->shape[0] != B || lse->shape[1] != q_len || lse->shape[2] != Hq))
        return fail(FW_ERR_INVALID_ARG, "lse must be [B, q_len, Hq]");
    if (!std::isfinite(scale)) return fail(FW_ERR_INVALID_ARG, "scale must be finite");
    const bool latent = !kv8 && (Dk == 576 && Dv == 512);
    // The grouped-query kernels anchor a row's window at its causal bound;
    // the latent ones keep both bounds per row.
    if (!causal && window_left >= 0 && !latent && q_len > 1)
        return fail(FW_ERR_UNSUPPORTED, "non-causal decode with a sliding window is served for the latent layout "
                    "(or q_len = 1)");
    if (latent && append)
        return fail(FW_ERR_UNSUPPORTED, "the fused append serves the grouped-query layouts (append latent rows "
                    "with fw_kv_append)");
    if (kv8 && !(Dk == 128 && Dv == 128))
        return fail(FW_ERR_UNSUPPORTED, "FP8 decode head dims (Dk=%lld, Dv=%lld): supported Dk = Dv = 128",
                    (long long)Dk, (long long)Dv);
    if (!latent && !(Dk == Dv && (Dk == 128 || Dk == 256)))
        return fail(FW_ERR_UNSUPPORTED, "decode head dims (Dk=%lld, Dv=%lld): supported Dk = Dv in {128, 256} "
                    "and the latent (576, 512)", (long long)Dk, (long long)Dv);
    if (!latent && Dv == 512)
        return fail(FW_ERR_UNSUPPORTED, "Dv = 512 is served for the latent layout (Dk = 576) only");
    if (q_len < 1 || q_len > 4) return fail(FW_ERR_UNSUPPORTED, "q_len must be in [1, 4]");
    if (!supported_page_size(ps))
        return fail(FW_ERR_UNSUPPORTED, "page size %lld: supported 8, 16, 32, 64, 128 or multiples of 128",
                    (long long)ps);
    if (B == 0) return ok();
    if (P < 1 || max_pages < 1) return fail(FW_ERR_INVALID_ARG, "empty page pool or block table");
    if (P > (1LL << 31) - 1 || max_pages * ps > (1LL << 30))
        return fail(FW_ERR_UNSUPPORTED, "page pool or sequence bound too large");
    if (fw_status_t s = check_tma_layout(q, "q")) return s;
    if (fw_status_t s = check_tma_layout(k_cache, "k_cache")) return s;
    if (fw_status_t s = check_tma_layout(v_cache, "v_cache")) return s;
    if (fw_status_t s = check_output_layout(out, "out")) return s;
    if (lse && reinterpret_cast<uintptr_t>(lse->data) % 4) return fail(FW_ERR_INVALID_ARG, "lse misaligned");

    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState *d = nullptr;
    if (fw_status_t s = device_state(&d)) return s;
    fw_decode_plan_t pl;
    if (fw_status_t s = plan_decode((int32_t)B, (int32_t)q_len, (int32_t)Hq, (int32_t)Hkv, (int32_t)Dv,
                                    max_pages * ps, d->num_sms, &pl))
        return s;
    void *ws = nullptr;
    if (fixed_ws) {
        if ((size_t)pl.workspace_bytes > fixed_bytes)
            return fail(FW_ERR_WORKSPACE, "these shapes need %lld bytes of decode scratch; the fixed scratch "
                        "holds %zu bytes", (long long)pl.workspace_bytes, fixed_bytes);
        fw_status_t st = FW_OK;
        ws = fixed_ws(d, &st);
        if (st != FW_OK) return st;
    } else if (fw_status_t s = get_workspace(d, (size_t)pl.workspace_bytes, stream, &ws)) {
        return s;
    }

    fw::DecodeParams p{};
    p.B = (int)B; p.q_len = (int)q_len; p.Hq = (int)Hq; p.Hkv = (int)Hkv; p.G = pl.group;
    p.ps = (int)ps; p.max_pages = (int)max_pages; p.num_pages = (int)P;
    p.rows = pl.rows_per_unit;
    p.head_mode = (latent || pl.group > 32) ? 1 : 0;
    p.tokens_per_unit = pl.tokens_per_unit;
    p.heads_per_unit = pl.heads_per_unit;
    p.head_chunks = p.head_mode ? (pl.group + pl.heads_per_unit - 1) / pl.heads_per_unit : 1;
    p.row_groups = pl.row_groups;
    p.units_per_row = latent ? (int)Hkv : (int)Hkv * pl.row_groups;
    p.range_groups = latent ? pl.row_groups : 1;
    // Grouped-query heads: the KV heads ride on the CTA index when the grid
    // holds whole groups of Hkv CTAs (same-box A/B at the Qwen3 shape: BF16
    // decode 4.0 % and FP8 decode 3.5 % faster).
    if (!latent && Hkv > 1 && pl.grid % Hkv == 0) {
        p.head_ride = 1;
        p.units_per_row = pl.row_groups;
        p.range_groups = (int)Hkv;
    }
    p.forced_span = g_opt_chunk > 0 ? pl.min_span_tiles : 0;
    p.min_span = pl.min_span_tiles;
    p.max_pieces = pl.max_pieces;
    p.grid = pl.grid;
    p.Dv = (int)Dv;
    // Packed latent rows: row groups straddle tokens, so q is read through
    // its flattened (token, head) axis, which must then be one stride.
    p.packed = latent && Hkv == 1 && pl.group % pl.rows_per_unit != 0;
    if (p.packed && q_len > 1 && q->stride[1] != Hq * q->stride[2])
        return fail(FW_ERR_UNSUPPORTED, "packed latent query rows need q contiguous over (token, head): "
                    "stride[1] = %lld, expected %lld", (long long)q->stride[1], (long long)(Hq * q->stride[2]));
    p.window_left = window_left;
    p.causal = causal ? 1 : 0;
    p.app = app;
    p.block_table = static_cast<const int32_t *>(block_table->data);
    p.bt_stride = block_table->stride[0];
    p.seq_lens = static_cast<const int32_t *>(seq_lens->data);
    p.out = out->data;
    for (int i = 0; i < 4; ++i) p.out_stride[i] = out->stride[i];
    p.lse = lse ? static_cast<float *>(lse->data) : nullptr;
    if (lse) for (int i = 0; i < 3; ++i) p.lse_stride[i] = lse->stride[i];
    const int64_t rows = B * q_len * Hq;
    char *wsb = static_cast<char *>(ws);
    const int64_t plan_bytes = ((B + 3) * 4 + 255) / 256 * 256;
    const int64_t o_bytes = (rows * pl.max_pieces * Dv * 4 + 255) / 256 * 256;
    p.plan = reinterpret_cast<int32_t *>(wsb);
    p.ws_o = reinterpret_cast<float *>(wsb + plan_bytes);
    p.ws_lse = reinterpret_cast<float *>(wsb + plan_bytes + o_bytes);
    p.scale_log2 = scale * (kv8 ? k_scale : 1.f) * 1.4426950408889634f;
    p.out_scale = kv8 ? v_scale : 1.f;
    p.timeout_ns = (uint64_t)g_opt_timeout_ms * 1000000ull;
    p.status = d->status;
    p.counters = d->counters;
    p.test_stall = g_opt_test_stall ? 1 : 0;
    p.piece_cost = latent ? 0 : kv8 ? fw::kDecodePieceCostFp8 : fw::kDecodePieceCostBf16;

    CUtensorMap tq, tk, tv;
    if (p.packed) {
        // Packed latent rows: [B][q_len * Hq rows][Dk], 64 rows per box (a
        // pair's CTAs load one box each); rows past the end read as zeros.
        const uint64_t dims[3] = {(uint64_t)Dk, (uint64_t)(q_len * Hq), (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)q->stride[2] * 2, (uint64_t)q->stride[0] * 2};
        const uint32_t box[3] = {64, (uint32_t)fw::kLatentRows, 1};
        if (fw_status_t s = encode_bf16(&tq, q->data, 3, dims, strides, box, "q")) return s;
    } else {
        // Latent heads: each CTA loads 64 query rows (a pair splits its 128).
        const uint32_t box_h = p.head_mode == 0 ? (uint32_t)pl.group
                             : latent ? (uint32_t)fw::kLatentRows : (uint32_t)pl.heads_per_unit;
        const uint32_t box_t = p.head_mode == 0 ? (uint32_t)pl.tokens_per_unit : 1u;
        const uint64_t dims[4] = {(uint64_t)Dk, (uint64_t)Hq, (uint64_t)q_len, (uint64_t)B};
        const uint64_t strides[3] = {(uint64_t)q->stride[2] * 2, (uint64_t)q->stride[1] * 2, (uint64_t)q->stride[0] * 2};
        const uint32_t box[4] = {64, box_h, box_t, 1};
        if (fw_status_t s = encode_bf16(&tq, q->data, 4, dims, strides, box, "q")) return s;
    }
    {
        // BF16: boxes of 64 columns (128 bytes); FP8: one box spans the whole
        // 128-byte row of 128 E4M3 values.
        const uint32_t rows_box = (uint32_t)(ps < fw::kKvTile ? ps : fw::kKvTile);
        const uint64_t esz = kv8 ? 1 : 2;
        const CUtensorMapDataType type = kv8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const uint64_t dk[4] = {(uint64_t)Dk, (uint64_t)Hkv, (uint64_t)ps, (uint64_t)P};
        const uint64_t sk[3] = {(uint64_t)k_cache->stride[2] * esz, (uint64_t)k_cache->stride[1] * esz,
                                (uint64_t)k_cache->stride[0] * esz};
        const uint32_t box[4] = {kv8 ? 128u : 64u, 1, rows_box, 1};
        // A 128-byte FP8 row is followed in memory by another head's row
        // unless the slots are 128 bytes apart (one KV head): promoting its
        // fetch to 256 bytes pulls that row through DRAM for another CTA,
        // which uses it from L2 when the heads ride on the CTA index (that
        // CTA reads the same token rows at the same time) and mostly comes
        // too late otherwise (measured: 1.4x the algorithmic bytes with 8 KV
        // heads), so only riding heads get 256 bytes.  BF16 rows of 256 bytes
        // or more use both halves.
        auto promo_for = [&](const fw_tensor_t *c) {
            const bool narrow_row = kv8 && (uint64_t)Dk * esz == 128 && (uint64_t)c->stride[1] * esz != 128 &&
                                    !p.head_ride;
            return narrow_row ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
        };
        if (fw_status_t s = encode_map(&tk, type, k_cache->data, 4, dk, sk, box, "k_cache", promo_for(k_cache)))
            return s;
        const uint64_t dv[4] = {(uint64_t)Dv, (uint64_t)Hkv, (uint64_t)ps, (uint64_t)P};
        const uint64_t sv[3] = {(uint64_t)v_cache->stride[2] * esz, (uint64_t)v_cache->stride[1] * esz,
                                (uint64_t)v_cache->stride[0] * esz};
        if (fw_status_t s = encode_map(&tv, type, v_cache->data, 4, dv, sv, box, "v_cache", promo_for(v_cache)))
            return s;
    }
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    if (g_opt_timing) { ev0 = pooled_event(); ev1 = pooled_event(); }
    int launched = 0;
    cudaError_t e = kv8 ? fw::launch_decode_fp8(p, tq, tk, tv, stream, ev0, ev1, &launched)
                  : latent ? (pl.rows_per_unit == fw::kLatentPairRows
                                  ? fw::launch_latent_pair_decode(p, tq, tk, tv, stream, ev0, ev1, &launched)
                                  : fw::launch_latent_decode(p, tq, tk, tv, stream, ev0, ev1, &launched))
                           : fw::launch_decode(p, tq, tk, tv, (int)Dk, stream, ev0, ev1, &launched);
    g_launches.fetch_add(launched);
    if (e != cudaSuccess) return fail(FW_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    if (ev0) g_timed.push_back({ev0, ev1});
    return ok();
}

fw_status_t fw_paged_decode(const fw_tensor_t *q, const fw_tensor_t *k_cache, const fw_tensor_t *v_cache,
                            const fw_tensor_t *block_table, const fw_tensor_t *seq_lens, float scale,
                            fw_tensor_t *out, fw_tensor_t *lse, fw_stream_t stream) {
    return paged_decode_impl(q, k_cache, v_cache, block_table, seq_lens, scale, out, lse, stream, nullptr, 0);
}

fw_status_t fw_paged_decode_fp8(const fw_tensor_t *q, const fw_tensor_t *k_cache, const fw_tensor_t *v_cache,
                                const fw_tensor_t *block_table, const fw_tensor_t *seq_lens, float scale,
                                float k_scale, float v_scale, fw_tensor_t *out, fw_tensor_t *lse,
                                fw_stream_t stream) {
    return paged_decode_impl(q, k_cache, v_cache, block_table, seq_lens, scale, out, lse, stream, nullptr, 0,
                             true, k_scale, v_scale);
}

fw_status_t fw_paged_decode_append(const fw_tensor_t *q, const fw_tensor_t *k_new, const fw_tensor_t *v_new,
                                   const fw_tensor_t *slot_mapping, int64_t layer_base_rows, fw_tensor_t *k_cache,
                                   fw_tensor_t *v_cache, const fw_tensor_t *block_table,
                                   const fw_tensor_t *seq_lens, float scale, float k_scale, float v_scale,
                                   int32_t window_left, fw_tensor_t *out, fw_tensor_t *lse, fw_stream_t stream) {
    if (!k_cache || !v_cache || !k_new || !v_new) return fail(FW_ERR_INVALID_ARG, "caches and new rows are required");
    const AppendArgs aa{k_new, v_new, slot_mapping, layer_base_rows};
    return paged_decode_impl(q, k_cache, v_cache, block_table, seq_lens, scale, out, lse, stream, nullptr, 0,
                             false, k_scale, v_scale, window_left, true, &aa);
}

fw_status_t fw_kv_append(const fw_tensor_t *k_new, const fw_tensor_t *v_new, const fw_tensor_t *slot_mapping,
                         int64_t layer_base_rows, fw_tensor_t *k_cache, fw_tensor_t *v_cache, float k_scale,
                         float v_scale, fw_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const AppendArgs aa{k_new, v_new, slot_mapping, layer_base_rows};
    fw::AppendParams app{};
    if (fw_status_t s = build_append(aa, k_cache, v_cache, k_scale, v_scale, &app)) return s;
    if (app.rows == 0) return ok();
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState *d = nullptr;
    if (fw_status_t s = device_state(&d)) return s;
    cudaError_t e = fw::launch_kv_append(app, d->status, stream);
    if (e != cudaSuccess) return fail(FW_ERR_CUDA, "append launch: %s", cudaGetErrorString(e));
    g_launches.fetch_add(1);
    return ok();
}

fw_status_t fw_paged_decode_window(const fw_tensor_t *q, const fw_tensor_t *k_cache, const fw_tensor_t *v_cache,
                                   const fw_tensor_t *block_table, const fw_tensor_t *seq_lens, float scale,
                                   float k_scale, float v_scale, int32_t window_left, fw_tensor_t *out,
                                   fw_tensor_t *lse, fw_stream_t stream) {
    return paged_decode_impl(q, k_cache, v_cache, block_table, seq_lens, scale, out, lse, stream, nullptr, 0,
                             false, k_scale, v_scale, window_left, true);
}

fw_status_t fw_paged_decode_masked(const fw_tensor_t *q, const fw_tensor_t *k_cache, const fw_tensor_t *v_cache,
                                   const fw_tensor_t *block_table, const fw_tensor_t *seq_lens, float scale,
                                   int32_t causal, int32_t window_left, float k_scale, float v_scale,
                                   fw_tensor_t *out, fw_tensor_t *lse, fw_stream_t stream) {
    return paged_decode_impl(q, k_cache, v_cache, block_table, seq_lens, scale, out, lse, stream, nullptr, 0,
                             false, k_scale, v_scale, window_left, true, nullptr, causal != 0);
}

// ----------------------------------------------------- decode without allocation
//
// Fixed decode scratch for fw_paged_decode_noalloc: the tile prefix table and
// the split-KV partials of one call.  It is part of the library's device
// image, so every GPU that loads the library holds these 64 MiB until the
// process exits.  Host code must not hand the array's name to a kernel (on
// the host it is only a stand-in symbol); the device address is looked up
// below, once per device, and cached.
}  // extern "C"

static constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static void *noalloc_scratch(DeviceState *d, fw_status_t *st) {
    if (!d->noalloc_scratch) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr) {
            *st = fail(FW_ERR_CUDA, "device address of the fixed decode scratch: %s", cudaGetErrorString(e));
            return nullptr;
        }
        d->noalloc_scratch = ptr;
    }
    *st = FW_OK;
    return d->noalloc_scratch;
}

extern "C" {

fw_status_t fw_paged_decode_noalloc(const fw_tensor_t *q, const fw_tensor_t *k_cache, const fw_tensor_t *v_cache,
                                    const fw_tensor_t *block_table, const fw_tensor_t *seq_lens, float scale,
                                    fw_tensor_t *out, fw_tensor_t *lse, fw_stream_t stream) {
    return paged_decode_impl(q, k_cache, v_cache, block_table, seq_lens, scale, out, lse, stream,
                             noalloc_scratch, kNoAllocScratchBytes);
}

fw_status_t fw_varlen_prefill(const fw_tensor_t *q, const fw_tensor_t *k, const fw_tensor_t *v,
                              const fw_tensor_t *cu_seqlens_q, const fw_tensor_t *cu_seqlens_k, int causal,
                              float scale, fw_tensor_t *out, fw_tensor_t *lse, fw_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (fw_status_t s = check_tensor(q, "q", 3, FW_BF16)) return s;
    if (fw_status_t s = check_tensor(k, "k", 3, FW_BF16)) return s;
    if (fw_status_t s = check_tensor(v, "v", 3, FW_BF16)) return s;
    if (fw_status_t s = check_tensor(cu_seqlens_q, "cu_seqlens_q", 1, FW_I32)) return s;
    if (fw_status_t s = check_tensor(cu_seqlens_k, "cu_seqlens_k", 1, FW_I32)) return s;
    if (fw_status_t s = check_tensor(out, "out", 3, FW_BF16)) return s;
    if (fw_status_t s = check_tensor(lse, "lse", 2, FW_F32, true)) return s;
    const int64_t total_q = q->shape[0], Hq = q->shape[1], Dk = q->shape[2];
    const int64_t total_k = k->shape[0], Hkv = k->shape[1];
    const int64_t Dv = v->shape[2];
    const int64_t B = cu_seqlens_q->shape[0] - 1;
    if (k->shape[2] != Dk) return fail(FW_ERR_INVALID_ARG, "k head dim must match q");
    if (v->shape[0] != total_k || v->shape[1] != Hkv) return fail(FW_ERR_INVALID_ARG, "v must be [total_k, Hkv, Dv]");
    if (B < 0 || cu_seqlens_k->shape[0] != B + 1)
        return fail(FW_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must both hold B + 1 entries");
    if ((B >= 0 && cu_seqlens_q->stride[0] != 1 && B + 1 > 1) || (cu_seqlens_k->stride[0] != 1 && B + 1 > 1))
        return fail(FW_ERR_INVALID_ARG, "cu_seqlens must be contiguous");
    if (out->shape[0] != total_q || out->shape[1] != Hq || out->shape[2] != Dv)
        return fail(FW_ERR_INVALID_ARG, "out must be [total_q, Hq, Dv]");
    if (lse && (lse->shape[0] != total_q || lse->shape[1] != Hq))
        return fail(FW_ERR_INVALID_ARG, "lse must be [total_q, Hq]");
    if (Hkv < 1 || Hq % Hkv != 0) return fail(FW_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
    if (!std::isfinite(scale)) return fail(FW_ERR_INVALID_ARG, "scale must be finite");
    if (!(Dk == Dv && (Dk == 128 || Dk == 256)))
        return fail(FW_ERR_UNSUPPORTED, "prefill head dims (Dk=%lld, Dv=%lld): supported Dk = Dv in {128, 256}",
                    (long long)Dk, (long long)Dv);
    if (total_q >= (1LL << 31) || total_k >= (1LL << 31)) return fail(FW_ERR_UNSUPPORTED, "too many tokens");
    if (B == 0 || total_q == 0) return ok();
    if (fw_status_t s = check_tma_layout(q, "q")) return s;
    if (fw_status_t s = check_tma_layout(k, "k")) return s;
    if (fw_status_t s = check_tma_layout(v, "v")) return s;
    if (fw_status_t s = check_tma_layout(out, "out")) return s;   // rows are written as 16-byte vectors
    if (lse && reinterpret_cast<uintptr_t>(lse->data) % 4) return fail(FW_ERR_INVALID_ARG, "lse misaligned");
    const int64_t capacity = ((total_q + 127) / 128 + B) * Hq;
    if (capacity >= (1LL << 31)) return fail(FW_ERR_UNSUPPORTED, "too many query tiles");

    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState *d = nullptr;
    if (fw_status_t s = device_state(&d)) return s;
    const int64_t plan_bytes = ((B + 4) * 4 + 255) / 256 * 256;
    const int64_t ws_bytes = plan_bytes + capacity * 4;
    void *ws = nullptr;
    if (fw_status_t s = get_workspace(d, (size_t)ws_bytes, stream, &ws)) return s;

    fw::PrefillParams p{};
    p.B = (int)B; p.Hq = (int)Hq; p.Hkv = (int)Hkv; p.G = (int)(Hq / Hkv); p.causal = causal ? 1 : 0;
    p.Dv = (int)Dv;
    p.online = g_opt_prefill_online ? 1 : 0;
    p.total_q = total_q; p.total_k = total_k;
    p.cu_q = static_cast<const int32_t *>(cu_seqlens_q->data);
    p.cu_k = static_cast<const int32_t *>(cu_seqlens_k->data);
    p.out = out->data;
    for (int i = 0; i < 3; ++i) p.out_stride[i] = out->stride[i];
    p.lse = lse ? static_cast<float *>(lse->data) : nullptr;
    if (lse) for (int i = 0; i < 2; ++i) p.lse_stride[i] = lse->stride[i];
    p.scale_log2 = scale * 1.4426950408889634f;
    p.timeout_ns = (uint64_t)g_opt_timeout_ms * 1000000ull;
    p.status = d->status;
    p.counters = d->counters;
    p.plan = static_cast<int32_t *>(ws);
    p.list = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + plan_bytes);
    p.list_capacity = capacity;
    int64_t grid = d->num_sms;
    if (g_opt_max_ctas > 0 && grid > g_opt_max_ctas) grid = g_opt_max_ctas;
    if (Dk == 256) grid = grid < 2 ? 2 : grid & ~int64_t(1);   // whole CTA pairs
    p.grid = (int)grid;

    CUtensorMap tq, tk, tv;
    {
        const uint64_t dq[3] = {(uint64_t)Dk, (uint64_t)Hq, (uint64_t)total_q};
        const uint64_t sq[2] = {(uint64_t)q->stride[1] * 2, (uint64_t)q->stride[0] * 2};
        const uint32_t box[3] = {64, 1, 128};
        if (fw_status_t s = encode_bf16(&tq, q->data, 3, dq, sq, box, "q")) return s;
        if (total_k > 0) {
            const uint64_t dk[3] = {(uint64_t)Dk, (uint64_t)Hkv, (uint64_t)total_k};
            const uint64_t sk[2] = {(uint64_t)k->stride[1] * 2, (uint64_t)k->stride[0] * 2};
            // Head dim 256 runs on CTA pairs that each load half (64 keys) of a K tile.
            const uint32_t kbox[3] = {64, 1, Dk == 256 ? 64u : 128u};
            if (fw_status_t s = encode_bf16(&tk, k->data, 3, dk, sk, kbox, "k")) return s;
            const uint64_t dv[3] = {(uint64_t)Dv, (uint64_t)Hkv, (uint64_t)total_k};
            const uint64_t sv[2] = {(uint64_t)v->stride[1] * 2, (uint64_t)v->stride[0] * 2};
            if (fw_status_t s = encode_bf16(&tv, v->data, 3, dv, sv, box, "v")) return s;
        } else {
            // No keys anywhere: every query tile walks zero KV tiles, so these
            // maps are never used; they only need to be valid descriptors.
            tk = tq;
            tv = tq;
        }
    }
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    if (g_opt_timing) { ev0 = pooled_event(); ev1 = pooled_event(); }
    int launched = 0;
    cudaError_t e = fw::launch_prefill(p, tq, tk, tv, (int)Dk, stream, ev0, ev1, &launched);
    g_launches.fetch_add(launched);
    if (e != cudaSuccess) return fail(FW_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    if (ev0) g_timed.push_back({ev0, ev1});
    return ok();
}

}  // extern "C"
