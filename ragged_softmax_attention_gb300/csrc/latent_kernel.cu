// Latent-head paged decode, sm_103a: every KV head is one 576-wide latent row
// per key, and V is its first 512 columns ("TokenSpeed-MLA 2.0.1", decode:
// kv_cache [pages, page_size, 576] with v = kv_cache[..., :512], 128 query
// heads over one KV head, up to four query tokens).
//
// Why its own kernel.  A 128-key tile of 576-wide keys is 144 KB of shared
// memory and 128 query rows of a 512-wide O fill all 512 TMEM columns, so the
// layout of the grouped-query decode kernel does not carry over.  Here:
//   * a CTA holds 64 query rows (64 consecutive heads of one token) on the MMA
//     N axis and 128 keys on M (swap-AB, as in the grouped-query kernel):
//       S^T [128 keys x 64]  = K_tile [128 x 576] * Q^T
//       O^T [512 x 64]      += V_tile^T [512 x 128] * P^T [128 x 64]
//     TMEM: two S^T buffers (2 x 64 columns) + O^T (4 x 64 columns);
//   * Q^T stays in shared memory (72 KB) for the whole piece; keys stream
//     through a ring of four 32 KB slots, one 128-key x 128-column chunk per
//     slot: five chunks feed a tile's QK^T (the last one is the 64-column
//     rotary part), four more (the V columns, read again from L2) feed its PV;
//   * the row groups of a (batch row, KV head) unit -- q_len tokens x Hq/64
//     head blocks -- ride on the CTA index: CTA c runs row group c % R over the
//     tile ranges c / R, c / R + grid / R, ..., so the R CTAs that read the
//     same keys run side by side and the keys come from DRAM about once.
//
// Softmax: Flywheel's static anchor ("Flywheel Attention", section 3.1 and
// appendix A).  A row's anchor is the scaled max of the first tile of the
// piece; P = 2^(s * scale * log2 e - anchor) afterwards with no running max.
// The check is per element: while no exponent exceeds 64 every p, the row sum
// and O stay far inside FP32 range, so the result equals the rescaling form
// up to rounding; a tile in which some exponent exceeds it moves the affected
// anchors to that tile's row max, rescales l and O^T, and recomputes P before
// the MMA reads it.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0     TMA producer: Q^T of each piece, then the key chunks in the
//              order the MMAs consume them (page walk through block_table);
//              V rows past the end of a sequence are zeroed before release.
//   warp 1     MMA issuer (one thread) and TMEM owner: QK^T of tile j+1 goes
//              out before PV of tile j, so the softmax of tile j overlaps it.
//   warps 2-5  softmax (thread = key of the tile) and epilogue (thread = O^T
//              lane = one of 128 value columns of a chunk).
#include <cuda_bf16.h>

#include "fw_internal.h"
#include "fw_ptx.cuh"
#include "decode_common.cuh"

namespace fw {

namespace {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kAnchorSlack = 64.0f;                  // log2 units above the anchor before a rescale

constexpr int kDk = 576, kDv = 512;
constexpr int kRows = kLatentRows;                     // 64 query rows per CTA
constexpr int kSlots = 4;
constexpr int kHalfBytes = kKvTile * 128;              // 128 keys x 64 columns, 128-byte swizzle
constexpr int kSlotBytes = 2 * kHalfBytes;             // 128 keys x 128 columns
constexpr int kQChunkBytes = kRows * 128;              // 64 rows x 64 columns
constexpr int kQBytes = kRows * kDk * 2;               // 9 chunks
constexpr int kPBytes = kKvTile * kRows * 2;           // P^T: one 128-byte row (64 query rows) per key
constexpr int kQkChunks = 5;                           // 4 x 128 columns + 64 rotary columns
constexpr int kPvChunks = kDv / 128;
constexpr int kOffQ = 0;
constexpr int kOffRing = kOffQ + kQBytes;
constexpr int kOffP = kOffRing + kSlots * kSlotBytes;
constexpr int kOffBar = kOffP + kPBytes;
constexpr int kNumBars = 2 * kSlots + 2 + 2 + 1 + 1 + 1 + 1 + 1 + 1;
constexpr int kOffRed = kOffBar + ((kNumBars * 8 + 127) / 128) * 128;
constexpr int kOffMisc = kOffRed + 8 * kRows * 4;       // [4][64] partials + [64] anchors, factors, upper/lower limits
constexpr int kSmemBytes = kOffMisc + 16 + 1024;        // + alignment slack
static_assert(kOffRing % 1024 == 0 && kOffP % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA exceeded");
constexpr uint32_t kTmemCols = 512;                     // 2 x 64 (S^T) + 4 x 64 (O^T) = 384 used
constexpr uint32_t kColO = 2 * kRows;
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kRows, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kRows, true, true);

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const WaitCtx &w, int lane) {
    int ok = 1;
    if (lane == 0) ok = mbar_wait(bar, parity, w) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Named barrier over `count` threads that also returns whether any of them
// passed `pred` (PTX bar.red.or).
__device__ __forceinline__ bool named_bar_any(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(pred ? 1u : 0u), "r"(id), "r"(count) : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ int clamp_len(const DecodeParams &p, int n) {
    const int cap = p.max_pages * p.ps;
    return n < 0 ? 0 : (n > cap ? cap : n);
}

// kPacked: row groups may straddle tokens (packed rows), so visibility is
// per row; otherwise every row of a group is one token's and shares it.
template <bool kPacked>
__global__ void __launch_bounds__(192, 1)
latent_decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem + kOffQ;
    uint8_t *sRing = smem + kOffRing;
    uint8_t *sP = smem + kOffP;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *slot_full = bars;
    uint64_t *slot_empty = slot_full + kSlots;
    uint64_t *s_full = slot_empty + kSlots;        // [2]
    uint64_t *s_free = s_full + 2;                 // [2]
    uint64_t *q_full = s_free + 2;                 // [1]
    uint64_t *q_empty = q_full + 1;                // [1]
    uint64_t *p_full = q_empty + 1;                // [1]
    uint64_t *pv_done = p_full + 1;                // [1]: PV j landed (also frees P^T)
    uint64_t *drain = pv_done + 1;                 // [1]
    uint64_t *tail_bar = drain + 1;                // [1]: producer-side landing of a tail V chunk
    float *red = reinterpret_cast<float *>(smem + kOffRed);        // [4][64] per-warp row partials
    float *anchor_s = red + 4 * kRows;                             // [64] row anchors
    float *alpha_s = anchor_s + kRows;                             // [64] rescale factors / 1 / L
    int *lim_s = reinterpret_cast<int *>(alpha_s + kRows);         // [64] end of the keys each row sees
    int *lo_s = lim_s + kRows;                                     // [64] first key each row sees
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) { mbar_init(&slot_full[i], 1); mbar_init(&slot_empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&s_full[i], 1); mbar_init(&s_free[i], 4); }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(p_full, 4);
        mbar_init(pv_done, 1);
        mbar_init(drain, 1);
        mbar_init(tail_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();                                    // the plan (and appended rows) of this call are written
    const WaitCtx wc{p.status, p.timeout_ns, abort_flag};

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        uint32_t m = 0, nq = 0, ntail = 0;
        const int box_rows = p.ps < kKvTile ? p.ps : kKvTile;
        // One ring slot: chunk c (128 columns, or the 64 rotary ones) of the
        // 128-key tile starting at key ts of row b.  Pages past the piece's
        // end are not loaded; with `zero_tail`, rows at or past k_end are
        // cleared once the copy has landed (their V values may be anything,
        // and a zero probability times a NaN would still be NaN).
        // Physical pages of the 128-key tile at key ts of row b: lane l holds
        // the tile's l-th page (l < pages in the tile).  Read one tile ahead
        // of use, so no chunk load waits on the block table.
        // Pages below a tile are powers of two: shifts instead of divisions.
        const int ps_shift = __ffs(p.ps) - 1;
        // Leading pages of the tile at ts wholly before the page holding the
        // window's first key (lo_page) are never looked up nor loaded.
        auto skip_of = [&](int ts, int lo_page) { return p.ps >= kKvTile ? 0 : max(0, lo_page - (ts >> ps_shift)); };
        auto tile_pages = [&](int b, int ts, int k_end, int lo_page) {
            int npages = 1;
            if (p.ps < kKvTile) npages = min(kKvTile >> ps_shift, (k_end - ts + p.ps - 1) >> ps_shift);
            int phys = 0;
            if (lane >= skip_of(ts, lo_page) && lane < npages)
                phys = __ldg(p.block_table + (int64_t)b * p.bt_stride + (p.ps < kKvTile ? ts >> ps_shift : ts / p.ps) +
                             lane);
            return phys;
        };
        auto load_chunk = [&](int g, int ts, int k_end, int lo_page, int phys, const CUtensorMap *tm, int c,
                              bool zero_tail) -> bool {
            const uint32_t s = m % kSlots;
            if (!warp_wait(&slot_empty[s], ((m / kSlots) & 1) ^ 1, wc, lane)) return false;
            const int halves = c < 4 ? 2 : 1;
            int npages = 1, slot0 = 0;
            if (p.ps < kKvTile) npages = min(kKvTile >> ps_shift, (k_end - ts + p.ps - 1) >> ps_shift);
            else slot0 = ts % p.ps;
            const int skip = min(npages, skip_of(ts, lo_page));
            const bool load = lane >= skip && lane < npages;
            if (load && (unsigned)phys >= (unsigned)p.num_pages) { record_error(p.status, 1); phys = 0; }
            const bool zero = zero_tail && (ts + kKvTile > k_end || skip > 0);
            uint64_t *bar = zero ? tail_bar : &slot_full[s];
            const uint32_t bytes = (uint32_t)((npages - skip) * box_rows * 128 * halves);
            uint8_t *dst = sRing + s * kSlotBytes;
            if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
            __syncwarp();
            if (load) {
                for (int h = 0; h < halves; ++h)
                    tma_load_4d(smem_u32(dst + h * kHalfBytes + lane * box_rows * 128), tm, bar,
                                c * 128 + h * 64, g, slot0, phys);
            }
            if (zero) {
                const bool landed = warp_wait(tail_bar, ntail & 1, wc, lane);
                if (!landed) {
                    if (lane == 0) mbar_wait_drain(tail_bar, ntail & 1, wc);
                    __syncwarp();
                    return false;
                }
                ++ntail;
                // Rows at or past k_end, and rows of pages skipped before the window.
                const int r0 = min(kKvTile, k_end - ts), rh = skip * p.ps;
                for (int idx = lane; idx < (kKvTile - r0) * 16; idx += 32) {
                    const int row = r0 + (idx >> 4);
                    const int h = (idx >> 3) & 1;
                    reinterpret_cast<uint4 *>(dst + h * kHalfBytes + row * 128)[idx & 7] = make_uint4(0, 0, 0, 0);
                }
                for (int idx = lane; idx < min(rh, r0) * 16; idx += 32) {
                    const int row = idx >> 4;
                    const int h = (idx >> 3) & 1;
                    reinterpret_cast<uint4 *>(dst + h * kHalfBytes + row * 128)[idx & 7] = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&slot_full[s]);
            }
            ++m;
            return true;
        };
        bool ok = true;
        int pb = -1, pg = 0, pts = 0, pend_end = 0, pend_lo = 0, pphys = 0;   // the tile whose PV is still to be fed
        dec::LatentIter it;
        it.init(p, blockIdx.x, gridDim.x);
        dec::LatentPiece x;
        while (ok && it.next(p, x)) {
            if (!warp_wait(q_empty, (nq & 1) ^ 1, wc, lane)) { ok = false; break; }
            if (lane == 0) {
                mbar_arrive_expect_tx(q_full, (uint32_t)kQBytes);
                for (int c = 0; c < kDk / 64; ++c) {
                    if (kPacked)       // rows past the last (token, head) read as zeros
                        tma_load_3d(smem_u32(sQ + c * kQChunkBytes), &tm_q, q_full, c * 64, x.row0, x.b);
                    else
                        tma_load_4d(smem_u32(sQ + c * kQChunkBytes), &tm_q, q_full, c * 64, x.h0, x.t, x.b);
                }
            }
            __syncwarp();
            ++nq;
            const int lo_page = x.lo / p.ps;
            int nphys = tile_pages(x.b, x.k_begin, x.k_end, lo_page);
            for (int i = 0; i < x.ntiles && ok; ++i) {
                const int ts = x.k_begin + i * kKvTile;
                const int phys = nphys;
                if (i + 1 < x.ntiles) nphys = tile_pages(x.b, ts + kKvTile, x.k_end, lo_page);
                for (int c = 0; c < kQkChunks && ok; ++c)
                    ok = load_chunk(x.g, ts, x.k_end, lo_page, phys, &tm_k, c, false);
                if (pb >= 0)
                    for (int c = 0; c < kPvChunks && ok; ++c)
                        ok = load_chunk(pg, pts, pend_end, pend_lo, pphys, &tm_v, c, true);
                pb = x.b; pg = x.g; pts = ts; pend_end = x.k_end; pend_lo = lo_page; pphys = phys;
            }
        }
        if (ok && pb >= 0)
            for (int c = 0; c < kPvChunks && ok; ++c)
                ok = load_chunk(pg, pts, pend_end, pend_lo, pphys, &tm_v, c, true);
        // Do not leave the CTA while copies it issued may still land.
        if (lane == 0) {
            for (uint32_t k = 0; k < (uint32_t)kSlots && k < m; ++k) {
                const uint32_t j = m - 1 - k;
                mbar_wait_drain(&slot_full[j % kSlots], (j / kSlots) & 1, wc);
            }
            if (nq > 0) mbar_wait_drain(q_full, (nq - 1) & 1, wc);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            uint32_t m = 0, nq = 0, jt = 0, npv = 0;
            const uint32_t q_base = smem_u32(sQ);
            const uint32_t ring_base = smem_u32(sRing);
            const uint32_t p_base = smem_u32(sP);
            auto wait_slot = [&](uint32_t mm) { return mbar_wait(&slot_full[mm % kSlots], (mm / kSlots) & 1, wc); };
            auto issue_qk = [&](bool last_of_piece) -> bool {
                const uint32_t sb = jt & 1;
                if (!mbar_wait(&s_free[sb], ((jt >> 1) & 1) ^ 1, wc)) return false;
                for (int c = 0; c < kQkChunks; ++c) {
                    if (!wait_slot(m)) return false;
                    tc_fence_after();
                    const uint32_t slot = ring_base + (m % kSlots) * kSlotBytes;
                    const int nk = c < 4 ? 8 : 4;
                    for (int kk = 0; kk < nk; ++kk) {
                        const uint64_t a = sdesc_sw128(slot + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(q_base + (2 * c + (kk >> 2)) * kQChunkBytes + (kk & 3) * 32,
                                                       16, 1024);
                        mma_bf16_ss(tmem + sb * kRows, a, b, kIdescQK, (c > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&slot_empty[m % kSlots]);
                    ++m;
                }
                mma_commit(&s_full[sb]);
                if (last_of_piece) mma_commit(q_empty);
                ++jt;
                return true;
            };
            auto issue_pv = [&](bool first) -> bool {
                if (!mbar_wait(p_full, npv & 1, wc)) return false;
                for (int c = 0; c < kPvChunks; ++c) {
                    if (!wait_slot(m)) return false;
                    tc_fence_after();
                    const uint32_t slot = ring_base + (m % kSlots) * kSlotBytes;
#pragma unroll
                    for (int kk = 0; kk < kKvTile / 16; ++kk) {
                        const uint64_t a = sdesc_sw128(slot + kk * 16 * 128, kHalfBytes, 1024);
                        const uint64_t b = sdesc_sw128(p_base + kk * 16 * 128, 8192, 1024);
                        mma_bf16_ss(tmem + kColO + c * kRows, a, b, kIdescPV, (first && kk == 0) ? 0u : 1u);
                    }
                    mma_commit(&slot_empty[m % kSlots]);
                    ++m;
                }
                mma_commit(pv_done);
                ++npv;
                return true;
            };
            bool ok = true, pend = false, pend_first = false;
            dec::LatentIter it;
            it.init(p, blockIdx.x, gridDim.x);
            dec::LatentPiece x;
            while (ok && it.next(p, x)) {
                if (!mbar_wait(q_full, nq & 1, wc)) { ok = false; break; }
                tc_fence_after();
                ++nq;
                for (int i = 0; i < x.ntiles && ok; ++i) {
                    ok = issue_qk(i == x.ntiles - 1);
                    if (ok && pend) ok = issue_pv(pend_first);
                    pend = true;
                    pend_first = (i == 0);
                }
            }
            if (ok && pend) issue_pv(pend_first);
            mma_commit(drain);
            mbar_wait_drain(drain, 0, wc);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- softmax / epilogue
        // The 128 threads meet at named barriers, which cannot time out, so a
        // failed wait does not leave the loop: after an abort every wait
        // returns at once and the warps run through their remaining (bounded)
        // iterations together; the status word disowns what they write.
        // Per-row state shared by all threads (anchors, rescale factors) lives
        // in shared memory; each thread keeps only its keys' partial row sums.
        const int q4 = warp & 3;                        // TMEM lane quadrant of this warp
        const int key = q4 * 32 + lane;                 // key of the tile / value column of a chunk
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const float c2 = p.scale_log2;
        uint32_t jt = 0;
        // Scaled, masked row maxima of the S^T buffer at `sa`: every warp
        // reduces over its 32 keys into red[q4][r]; after the barrier thread
        // r < 64 may combine row r.
        auto row_max_partials = [&](uint32_t sa, int tok, bool uni, bool vis) {
#pragma unroll
            for (int c = 0; c < kRows; c += 16) {
                float s16[16];
                tmem_ld16(sa + c, s16);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float v =
                        warp_max((uni ? vis : (tok >= lo_s[c + k] && tok < lim_s[c + k])) ? s16[k] * c2 : kNegInf);
                    if (lane == 0) red[q4 * kRows + c + k] = v;
                }
            }
            named_bar_sync(1, 128);
        };
        auto red4 = [&](int r) {
            return fmaxf(fmaxf(red[r], red[kRows + r]), fmaxf(red[2 * kRows + r], red[3 * kRows + r]));
        };
        dec::LatentIter it;
        it.init(p, blockIdx.x, gridDim.x);
        dec::LatentPiece x;
        while (it.next(p, x)) {
            // Row r sees keys lo_s[r] .. lim_s[r] - 1: from its window's first
            // key (0 without a window) to its token's causal bound; nothing
            // for a padding row past the last packed row.  Rows of one group
            // may belong to different tokens.
            if (key < kRows) {
                const int gr = x.row0 + key;
                const int pos = x.n - p.q_len + gr / p.G;             // the row's own key position
                const bool real = gr < p.q_len * p.G;
                lim_s[key] = real ? min(x.k_end, p.causal ? pos + 1 : x.n) : 0;
                lo_s[key] = real && p.window_left >= 0 ? max(0, pos - p.window_left) : 0;
            }
            named_bar_sync(1, 128);
            // A key inside every row's range is visible to all rows, one
            // outside all of them to none: one test then serves the row set
            // (always, unless the rows straddle a token boundary near it).
            int hi_min = lim_s[0], hi_max = hi_min, lo_min = lo_s[0], lo_max = lo_min;
            for (int r = 1; r < kRows; ++r) {
                hi_min = min(hi_min, lim_s[r]);
                hi_max = max(hi_max, lim_s[r]);
                lo_min = min(lo_min, lo_s[r]);
                lo_max = max(lo_max, lo_s[r]);
            }
            float l_part[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r) l_part[r] = 0.f;
            for (int i = 0; i < x.ntiles; ++i, ++jt) {
                const int tok = x.k_begin + i * kKvTile + key;
                const bool vis = tok >= lo_max && tok < hi_min;
                const bool uni = !kPacked || vis || tok < lo_min || tok >= hi_max;
                const uint32_t sb = jt & 1;
                mbar_wait(&s_full[sb], (jt >> 1) & 1, wc);
                tc_fence_after();
                const uint32_t sa = tmem + lane_off + sb * kRows;
                if (i == 0) {
                    // anchor_s[r]: row r's exponent offset, its max over this
                    // first tile (0 for a row that sees no key here, and hence
                    // none later in the piece).
                    row_max_partials(sa, tok, uni, vis);
                    if (key < kRows) {
                        const float m = red4(key);
                        anchor_s[key] = m == kNegInf ? 0.f : m;
                    }
                    named_bar_sync(1, 128);
                }
                // The check comes first: the largest exponent this tile would
                // raise any row to (a max-only pass; on a piece's first tile the
                // anchors are this tile's maxima and nothing can exceed them).
                float xmax = kNegInf;
                if (i > 0) {   // all lanes: tcgen05.ld is warp-collective
#pragma unroll
                    for (int c = 0; c < kRows; c += 16) {
                        float s16[16];
                        tmem_ld16(sa + c, s16);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 16; k += 4) {
                            const float4 a = *reinterpret_cast<const float4 *>(anchor_s + c + k);
                            float e0 = fmaf(s16[k], c2, -a.x), e1 = fmaf(s16[k + 1], c2, -a.y);
                            float e2 = fmaf(s16[k + 2], c2, -a.z), e3 = fmaf(s16[k + 3], c2, -a.w);
                            if (!uni) {            // rows of two tokens meet near this key
                                const int4 L = *reinterpret_cast<const int4 *>(lim_s + c + k);
                                const int4 F = *reinterpret_cast<const int4 *>(lo_s + c + k);
                                e0 = tok >= F.x && tok < L.x ? e0 : kNegInf; e1 = tok >= F.y && tok < L.y ? e1 : kNegInf;
                                e2 = tok >= F.z && tok < L.z ? e2 : kNegInf; e3 = tok >= F.w && tok < L.w ? e3 : kNegInf;
                            }
                            xmax = fmaxf(xmax, fmaxf(fmaxf(e0, e1), fmaxf(e2, e3)));
                        }
                    }
                    if (uni && !vis) xmax = kNegInf;
                }
                if (named_bar_any(1, 128, xmax > kAnchorSlack)) {
                    // Some score rose more than kAnchorSlack above its anchor:
                    // move those anchors to this tile's row max and rescale l
                    // and O^T (once the previous PV has landed).
                    row_max_partials(sa, tok, uni, vis);
                    if (key < kRows) {                   // whole warps: q4 0-1
                        const float mx = red4(key);
                        float a = 1.f;
                        const bool move = mx > anchor_s[key] + kAnchorSlack;
                        if (move) {
                            a = ex2_approx(anchor_s[key] - mx);
                            anchor_s[key] = mx;
                        }
                        alpha_s[key] = a;
                        const unsigned moved = __ballot_sync(0xffffffffu, move);
                        if (lane == 0) count_events(p.counters, kCounterLatentRescales, __popc(moved));
                    }
                    named_bar_sync(1, 128);
#pragma unroll
                    for (int r = 0; r < kRows; ++r) l_part[r] *= alpha_s[r];
                    mbar_wait(pv_done, (jt - 1) & 1, wc);
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < kPvChunks; ++c) {
#pragma unroll
                        for (int r0 = 0; r0 < kRows; r0 += 16) {
                            float o[16];
                            const uint32_t ta = tmem + lane_off + kColO + c * kRows + r0;
                            tmem_ld16(ta, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 16; ++k) o[k] *= alpha_s[r0 + k];
                            tmem_st16(ta, o);
                        }
                    }
                    tmem_wait_st();
                }
                // P^T row of this key for the 64 query rows, packed in pairs;
                // the row sums take the FP32 probabilities.
                uint32_t pk[kRows / 2];
#pragma unroll
                for (int c = 0; c < kRows; c += 16) {
                    float s16[16];
                    tmem_ld16(sa + c, s16);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; k += 4) {
                        const float4 a = *reinterpret_cast<const float4 *>(anchor_s + c + k);
                        float p0 = ex2_approx(fmaf(s16[k], c2, -a.x)), p1 = ex2_approx(fmaf(s16[k + 1], c2, -a.y));
                        float p2 = ex2_approx(fmaf(s16[k + 2], c2, -a.z)), p3 = ex2_approx(fmaf(s16[k + 3], c2, -a.w));
                        // Masking by selection (an invisible key's score may be
                        // anything); per row only when two tokens meet near the key.
                        if (kPacked && !uni) {
                            const int4 L = *reinterpret_cast<const int4 *>(lim_s + c + k);
                            const int4 F = *reinterpret_cast<const int4 *>(lo_s + c + k);
                            p0 = tok >= F.x && tok < L.x ? p0 : 0.f; p1 = tok >= F.y && tok < L.y ? p1 : 0.f;
                            p2 = tok >= F.z && tok < L.z ? p2 : 0.f; p3 = tok >= F.w && tok < L.w ? p3 : 0.f;
                        } else {
                            p0 = vis ? p0 : 0.f; p1 = vis ? p1 : 0.f; p2 = vis ? p2 : 0.f; p3 = vis ? p3 : 0.f;
                        }
                        l_part[c + k] += p0;
                        l_part[c + k + 1] += p1;
                        l_part[c + k + 2] += p2;
                        l_part[c + k + 3] += p3;
                        pk[(c + k) >> 1] = pack_bf16x2(p0, p1);
                        pk[((c + k) >> 1) + 1] = pack_bf16x2(p2, p3);
                    }
                }
                // The P^T buffer is free once the previous PV has landed.
                mbar_wait(pv_done, (jt & 1) ^ 1, wc);
                uint8_t *prow = sP + key * 128;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    *reinterpret_cast<uint4 *>(prow + ((u ^ (key & 7)) << 4)) =
                        make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) { mbar_arrive(&s_free[sb]); mbar_arrive(p_full); }
            }
            // ------------------------------------------------------ epilogue
            // Row sums: red[q4][r] = this warp's part; thread r < 64 writes
            // 1 / L_r (or 0 for a row that saw no key) and the LSE.
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const float v = warp_sum(l_part[r]);
                if (lane == 0) red[q4 * kRows + r] = v;
            }
            named_bar_sync(1, 128);
            // Packed row gr of the unit is token gr / G, head g * G + gr % G;
            // rows past q_len * G are padding and write nothing.
            const int qG = p.q_len * p.G;
            const int64_t wrow_b = (int64_t)x.b * p.q_len * p.Hq;      // workspace row of (b, 0, 0)
            if (key < kRows) {
                const float L = (red[key] + red[kRows + key]) + (red[2 * kRows + key] + red[3 * kRows + key]);
                alpha_s[key] = L > 0.f ? 1.f / L : 0.f;
                const float lse2 = L > 0.f ? anchor_s[key] + __log2f(L) : kNegInf;
                const int gr = x.row0 + key;
                if (gr < qG) {
                    const int t = gr / p.G, h = x.g * p.G + gr % p.G;
                    if (x.single) {
                        if (p.lse)
                            p.lse[x.b * p.lse_stride[0] + t * p.lse_stride[1] + h * p.lse_stride[2]] =
                                lse2 * 0.69314718055994531f;
                    } else {
                        p.ws_lse[(wrow_b + (int64_t)t * p.Hq + h) * p.max_pieces + x.k] = lse2;
                    }
                }
            }
            named_bar_sync(1, 128);
            mbar_wait(pv_done, (jt - 1) & 1, wc);
            tc_fence_after();
            // Thread = value column c * 128 + key; a warp stores 32 consecutive
            // columns of one row at a time.
            __nv_bfloat16 *obase = reinterpret_cast<__nv_bfloat16 *>(p.out) + x.b * p.out_stride[0] + key;
            float *wbase = p.ws_o + key;
#pragma unroll 1
            for (int c = 0; c < kPvChunks; ++c) {
#pragma unroll 1
                for (int r0 = 0; r0 < kRows; r0 += 16) {
                    float o[16];
                    tmem_ld16(tmem + lane_off + kColO + c * kRows + r0, o);
                    tmem_wait_ld();
                    const int gr0 = x.row0 + r0;
                    int t = gr0 / p.G, hl = gr0 % p.G;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        if (gr0 + k < qG) {
                            const int h = x.g * p.G + hl;
                            const float v = o[k] * alpha_s[r0 + k];
                            if (x.single)
                                obase[t * p.out_stride[1] + h * p.out_stride[2] + c * 128] = __float2bfloat16_rn(v);
                            else
                                wbase[((wrow_b + (int64_t)t * p.Hq + h) * p.max_pieces + x.k) * kDv + c * 128] = v;
                        }
                        if (++hl == p.G) { hl = 0; ++t; }
                    }
                }
            }
            tc_fence_before();
            // The next piece rewrites red, anchor_s and alpha_s.
            named_bar_sync(1, 128);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    pdl_launch_dependents();                       // the combine kernel may launch
}

}  // namespace

size_t latent_decode_smem_bytes() { return kSmemBytes; }

cudaError_t launch_latent_decode(const DecodeParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                                 const CUtensorMap &tv, cudaStream_t stream, cudaEvent_t timing_start,
                                 cudaEvent_t timing_stop, int *launches) {
    *launches = 0;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(latent_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(latent_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    cudaError_t e = launch_decode_plan(p, stream);
    if (e != cudaSuccess) return e;
    ++*launches;
    if (timing_start) cudaEventRecord(timing_start, stream);
    // An ordinary launch, as for the CTA-pair kernel (programmatic
    // serialization under the plan kernel measured slower there).
    if (p.packed) latent_decode_kernel<true><<<p.grid, 192, kSmemBytes, stream>>>(p, tq, tk, tv);
    else latent_decode_kernel<false><<<p.grid, 192, kSmemBytes, stream>>>(p, tq, tk, tv);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ++*launches;
    if (timing_stop) cudaEventRecord(timing_stop, stream);
    if (p.max_pieces > 1) {
        e = launch_decode_combine(p, kDv, stream);
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    return cudaSuccess;
}

}  // namespace fw
