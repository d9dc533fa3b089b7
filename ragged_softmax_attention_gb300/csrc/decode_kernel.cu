// Paged grouped-query decode, sm_103a.
//
// The work unit is (batch row b, KV head g, row group): the query rows a unit
// holds are the (token, head) pairs of the query heads that share KV head g
// ("Writing Page Attention with PyPTO", section 1.3: one task = one batch row
// + one KV head + its five query heads; "TokenSpeed-MLA 2.0.1": query tokens
// folded next to the heads).  Units are laid end to end in the global order
// of their 128-key tiles and every persistent CTA takes equal contiguous tile
// ranges, so the work per CTA differs by at most one tile however ragged the
// batch is.  A unit cut by a range boundary becomes several pieces whose
// FP32 partials (split-KV) the combine kernel merges.
//
// Orientation.  A decode unit has few query rows (5 at 40 Q / 8 KV heads), so
// the KV tile takes the 128-wide MMA M axis and the padded query rows take N:
//   S^T [128 keys x NQ]  = K_tile [128 x D]  * Q^T            (tcgen05, TMEM)
//   O^T [D x NQ]        += V_tile^T [D x 128] * P^T [128 x NQ] (tcgen05, TMEM)
// Every softmax thread then owns one key of the tile and holds that key's
// score for every query row, so exp2 work spreads over 128 threads.
//
// Warp roles (192 threads, one CTA per SM, persistent over units):
//   warp 0     TMA producer: walks block_table[b, logical_page] and loads the
//              K and V pages of each 128-key tile into separate smem rings
//              (PyPTO section 5.2 page lookup; "TokenSpeed-MLA 2.0.1": K and V
//              loads do not wait on each other), plus the unit's Q rows.
//   warp 1     MMA issuer (one thread) and TMEM owner.
//   warps 2-5  online softmax in base 2 with a conditional rescale (the base
//              moves only when a row's max rises by more than 8 log2 units,
//              "TokenSpeed-MLA 2.0.1", softmax precision paragraph), P^T to
//              smem, O^T correction in TMEM when the base moves, epilogue.
// Handoffs are mbarriers: k_full/k_empty, v_full/v_empty, q_full/q_empty,
// s_full/s_free, p_full/p_free, pv_done -- the READY events of PyPTO
// section 8.3 with the double-buffered S and P slots playing its ring.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "decode_common.cuh"
#include "fw_internal.h"
#include "fw_ptx.cuh"

namespace fw {

namespace {

using namespace dec;

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D, int NQ>
struct DecodeCfg {
    static constexpr int kChunks = D / 64;                 // 128-byte swizzle column blocks
    static constexpr int kChunkBytes = kKvTile * 128;       // one 64-column block of a tile
    static constexpr int kTileBytes = kKvTile * D * 2;
    static constexpr int kKStages = (D == 128) ? 3 : (NQ == 16 ? 2 : 1);
    static constexpr int kVStages = (D == 128) ? 3 : 1;
    static constexpr int kQBytes = NQ * D * 2;
    static constexpr int kPBytes = NQ * kKvTile * 2;
    static constexpr int kDvTiles = D / 128;
    static constexpr int kTmemNeed = (2 + kDvTiles) * NQ;
    static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128 : 256;
    // shared memory map (offsets from a 1024-aligned base)
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffQ = kOffV + kVStages * kTileBytes;
    static constexpr int kOffP = kOffQ + 2 * kQBytes;
    static constexpr int kOffBar = kOffP + 2 * kPBytes;
    static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 2 + 2 + 2 + 2 + 2 + 2 + 1 + 1 + 1;
    static constexpr int kOffRedMax = kOffBar + kNumBars * 8;
    static constexpr int kOffRedSum = kOffRedMax + 2 * 4 * NQ * 4;
    static constexpr int kOffMisc = kOffRedSum + 4 * NQ * 4;
    // The row tables (PB and the lengths) take what is left of the budget.
    static constexpr int kOffRows = kOffMisc + 16;
    static constexpr int kRowCap = (232448 - 1024 - kOffRows) / 4 > 4096 ? 4096 : (232448 - 1024 - kOffRows) / 4;
    static constexpr int kSmemBytes = kOffRows + kRowCap * 4 + 1024;   // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA exceeded");
    static constexpr uint32_t kIdescQK = idesc_bf16_f32(128, NQ, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, NQ, true, false);
};

template <int D, int NQ>
__global__ void __launch_bounds__(192, 1)
paged_decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    using C = DecodeCfg<D, NQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sK = smem + C::kOffK;
    uint8_t *sV = smem + C::kOffV;
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sP = smem + C::kOffP;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *k_full = bars;
    uint64_t *k_empty = k_full + C::kKStages;
    uint64_t *v_full = k_empty + C::kKStages;
    uint64_t *v_empty = v_full + C::kVStages;
    uint64_t *q_full = v_empty + C::kVStages;
    uint64_t *q_empty = q_full + 2;
    uint64_t *s_full = q_empty + 2;
    uint64_t *s_free = s_full + 2;
    uint64_t *p_full = s_free + 2;
    uint64_t *p_free = p_full + 2;
    uint64_t *pv_done = p_free + 2;
    uint64_t *drain = pv_done + 1;
    uint64_t *never = drain + 1;                   // test hook: no thread ever arrives on it
    float *red_max = reinterpret_cast<float *>(smem + C::kOffRedMax);   // [2][4][NQ]
    float *red_sum = reinterpret_cast<float *>(smem + C::kOffRedSum);   // [4][NQ]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kKStages; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
        for (int i = 0; i < C::kVStages; ++i) { mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], 1); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1);
            mbar_init(&s_full[i], 1); mbar_init(&s_free[i], 4);
            mbar_init(&p_full[i], 4); mbar_init(&p_free[i], 1);
        }
        mbar_init(pv_done, 1);
        mbar_init(drain, 1);
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) { tmem_alloc(tmem_slot, C::kTmemCols); tmem_relinquish(); }
    // Zero the Q and P slots once: padding rows then contribute exact zeros.
    for (int i = threadIdx.x; i < (2 * C::kQBytes + 2 * C::kPBytes) / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(sQ)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();                                    // the plan (and appended rows) of this call are written
    const WaitCtx wc{p.status, p.timeout_ns, abort_flag};
    const RowTables rows = cache_row_tables(p, reinterpret_cast<int32_t *>(smem + C::kOffRows), C::kRowCap);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int jt = 0, ju = 0, issued_k = 0, issued_v = 0;
        const int box_rows = p.ps < kKvTile ? p.ps : kKvTile;
        const int pages_per_tile = p.ps < kKvTile ? kKvTile / p.ps : 1;
        const uint32_t q_rows = p.head_mode == 0 ? (uint32_t)(p.G * p.tokens_per_unit) : (uint32_t)p.rows;
        // Test hook for the bounded waits: before anything is copied, wait on
        // a barrier that nothing completes.  The wait runs out, records
        // FW_ERR_DEVICE_TIMEOUT and raises the abort flag; the other roles'
        // waits then return at once and the CTA winds down with no copy or
        // MMA in flight.
        if (p.test_stall && !warp_wait(never, 0, wc, lane)) goto producer_done;
        PieceIter it;
        it.init(p, rows);
        Unit x;
        while (it.next(p, x)) {
            const int qs = ju & 1;
            if (!warp_wait(&q_empty[qs], ((ju >> 1) & 1) ^ 1, wc, lane)) goto producer_done;
            if (lane == 0) {
                int h0, t0;
                if (p.head_mode == 0) { h0 = x.g * p.G; t0 = x.rg * p.tokens_per_unit; }
                else { t0 = x.rg / p.head_chunks; h0 = x.g * p.G + (x.rg % p.head_chunks) * p.rows; }
                mbar_arrive_expect_tx(&q_full[qs], C::kChunks * q_rows * 128u);
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(smem_u32(sQ + qs * C::kQBytes + c * NQ * 128), &tm_q, &q_full[qs],
                                c * 64, h0, t0, x.b);
            }
            __syncwarp();
            // Physical page numbers of the piece, 64 logical pages at a time in
            // two 32-entry register windows (lane l holds page win + l and
            // win + 32 + l); the next window is fetched while the current one
            // is in use, so no tile waits on a block-table read.  Entries past
            // the row's last page are never read (PyPTO section 9.1), nor, under
            // a sliding window, those of pages wholly before the window.
            const int32_t *bt_row = p.block_table + (int64_t)x.b * p.bt_stride;
            const int lp_end = ceil_div_i(x.k_end, p.ps);
            const int lp_first = x.lo / p.ps;
            int win = x.k_begin / p.ps;
            auto bt_at = [&](int lp) { return (lp >= lp_first && lp < lp_end) ? __ldg(bt_row + lp) : 0; };
            int cur = bt_at(win + lane);
            int nxt = bt_at(win + 32 + lane);
            for (int i = 0; i < x.ntiles; ++i, ++jt) {
                const int ts = x.k_begin + i * kKvTile;
                const int lp0 = ts / p.ps;
                const int slot0 = p.ps < kKvTile ? 0 : ts % p.ps;
                int npages = 1;
                if (p.ps < kKvTile) npages = min(pages_per_tile, ceil_div_i(x.k_end - ts, p.ps));
                if (lp0 >= win + 32) {
                    win += 32;
                    cur = nxt;
                    nxt = bt_at(win + 32 + lane);
                }
                // Leading pages of the tile wholly before the window are not
                // loaded (their rows are masked and their V rows zeroed).
                const int skip = min(npages, max(0, lp_first - lp0));
                const bool load = lane >= skip && lane < npages;
                const int idx = lp0 + lane - win;          // < 64 since npages <= 16
                const int from_cur = __shfl_sync(0xffffffffu, cur, idx & 31);
                const int from_nxt = __shfl_sync(0xffffffffu, nxt, idx & 31);
                int phys = idx < 32 ? from_cur : from_nxt;
                if (load && (unsigned)phys >= (unsigned)p.num_pages) { record_error(p.status, 1); phys = 0; }
                const uint32_t bytes = (uint32_t)((npages - skip) * box_rows * 128 * C::kChunks);
                const int ks = jt % C::kKStages;
                if (!warp_wait(&k_empty[ks], ((jt / C::kKStages) & 1) ^ 1, wc, lane)) goto producer_done;
                if (lane == 0) mbar_arrive_expect_tx(&k_full[ks], bytes);
                __syncwarp();
                if (load) {
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_4d(smem_u32(sK + ks * C::kTileBytes + c * C::kChunkBytes + lane * box_rows * 128),
                                    &tm_k, &k_full[ks], c * 64, x.g, slot0, phys);
                }
                issued_k = jt + 1;
                const int vs = jt % C::kVStages;
                if (!warp_wait(&v_empty[vs], ((jt / C::kVStages) & 1) ^ 1, wc, lane)) goto producer_done;
                if (lane == 0) mbar_arrive_expect_tx(&v_full[vs], bytes);
                __syncwarp();
                if (load) {
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_4d(smem_u32(sV + vs * C::kTileBytes + c * C::kChunkBytes + lane * box_rows * 128),
                                    &tm_v, &v_full[vs], c * 64, x.g, slot0, phys);
                }
                issued_v = jt + 1;
            }
            ++ju;
        }
    producer_done:
        // Do not leave the CTA while copies it issued may still land.
        if (lane == 0) {
            for (int k = 0; k < C::kKStages && k < issued_k; ++k) {
                const int j = issued_k - 1 - k;
                mbar_wait_drain(&k_full[j % C::kKStages], (j / C::kKStages) & 1, wc);
            }
            for (int k = 0; k < C::kVStages && k < issued_v; ++k) {
                const int j = issued_v - 1 - k;
                mbar_wait_drain(&v_full[j % C::kVStages], (j / C::kVStages) & 1, wc);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            int jt = 0, ju = 0, pend = -1;
            bool pend_first = false;
            // Descriptors at the tile bases, stepped by one integer add per
            // operand and instruction.
            const SDesc v_d = sdesc_sw128_split(smem_u32(sV), C::kChunkBytes, 1024);
            const SDesc k_d = sdesc_sw128_split(smem_u32(sK), 16, 1024);
            const SDesc p_d = sdesc_sw128_split(smem_u32(sP), 16, 1024);
            const SDesc q_d = sdesc_sw128_split(smem_u32(sQ), 16, 1024);
            auto issue_pv = [&](int jj, bool first) -> bool {
                const int vs = jj % C::kVStages;
                const int pb = jj & 1;
                if (!mbar_wait(&v_full[vs], (jj / C::kVStages) & 1, wc)) return false;
                if (!mbar_wait(&p_full[pb], (jj >> 1) & 1, wc)) return false;
                tc_fence_after();
                const SDesc v_s{v_d.lo + (uint32_t)(vs * C::kTileBytes) / 16u, v_d.hi};
                const SDesc p_s{p_d.lo + (uint32_t)(pb * C::kPBytes) / 16u, p_d.hi};
#pragma unroll
                for (int dvt = 0; dvt < C::kDvTiles; ++dvt) {
#pragma unroll
                    for (int kk = 0; kk < kKvTile / 16; ++kk) {
                        const uint64_t a = sdesc_at(v_s, (2 * dvt) * C::kChunkBytes + kk * 16 * 128);
                        const uint64_t b = sdesc_at(p_s, (kk >> 2) * NQ * 128 + (kk & 3) * 32);
                        mma_bf16_ss(tmem + 2 * NQ + dvt * NQ, a, b, C::kIdescPV, (first && kk == 0) ? 0u : 1u);
                    }
                }
                mma_commit(&v_empty[vs]);
                mma_commit(&p_free[pb]);
                mma_commit(pv_done);
                return true;
            };
            PieceIter it;
            it.init(p, rows);
            Unit x;
            while (it.next(p, x)) {
                const int qs = ju & 1;
                if (!mbar_wait(&q_full[qs], (ju >> 1) & 1, wc)) goto mma_done;
                for (int i = 0; i < x.ntiles; ++i, ++jt) {
                    const int ks = jt % C::kKStages;
                    const int sb = jt & 1;
                    if (!mbar_wait(&k_full[ks], (jt / C::kKStages) & 1, wc)) goto mma_done;
                    if (!mbar_wait(&s_free[sb], ((jt >> 1) & 1) ^ 1, wc)) goto mma_done;
                    tc_fence_after();
                    const SDesc k_s{k_d.lo + (uint32_t)(ks * C::kTileBytes) / 16u, k_d.hi};
                    const SDesc q_s{q_d.lo + (uint32_t)(qs * C::kQBytes) / 16u, q_d.hi};
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t a = sdesc_at(k_s, (kk >> 2) * C::kChunkBytes + (kk & 3) * 32);
                        const uint64_t b = sdesc_at(q_s, (kk >> 2) * NQ * 128 + (kk & 3) * 32);
                        mma_bf16_ss(tmem + sb * NQ, a, b, C::kIdescQK, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&k_empty[ks]);
                    mma_commit(&s_full[sb]);
                    if (i == x.ntiles - 1) mma_commit(&q_empty[qs]);
                    if (pend >= 0 && !issue_pv(pend, pend_first)) goto mma_done;
                    pend = jt;
                    pend_first = (i == 0);
                }
                ++ju;
            }
            if (pend >= 0) issue_pv(pend, pend_first);
        mma_done:
            mma_commit(drain);
            mbar_wait_drain(drain, 0, wc);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- softmax / epilogue
        // These 128 threads meet at named barriers, which cannot time out, so
        // a failed wait does not leave the loop: after an abort every wait
        // returns at once and the warps run through their remaining (bounded)
        // iterations in lockstep, producing garbage that the recorded status
        // word disowns.
        const int q4 = warp & 3;                       // TMEM lane quadrant of this warp
        const int row_in_tile = q4 * 32 + lane;        // key of the tile / dv lane this thread owns
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        int jt = 0;
        PieceIter it;
        it.init(p, rows);
        Unit x;
        while (it.next(p, x)) {
            int lim[NQ];
            int nrows = 0;
#pragma unroll
            for (int r = 0; r < NQ; ++r) {
                int t, h;
                const bool ok = unit_row(p, x, r, t, h);
                lim[r] = ok ? (p.causal ? min(x.n, x.n - p.q_len + t + 1) : x.n) : 0;
                if (ok) nrows = r + 1;
            }
            // Sliding window: a row with visible-key bound lim sees keys
            // lim - 1 - W .. lim - 1, i.e. lim - tok <= W + 1.
            const int wp1 = p.window_left < 0 ? 0x7fffffff : p.window_left + 1;
            float m_ref[NQ], l_part[NQ];
#pragma unroll
            for (int r = 0; r < NQ; ++r) { m_ref[r] = kNegInf; l_part[r] = 0.f; }
            for (int i = 0; i < x.ntiles; ++i, ++jt) {
                const int ts = x.k_begin + i * kKvTile;
                const int tok = ts + row_in_tile;
                const int sb = jt & 1;
                mbar_wait(&s_full[sb], (jt >> 1) & 1, wc);
                tc_fence_after();
                float s[NQ];
#pragma unroll
                for (int c = 0; c < NQ; c += 16)
                    tmem_ld16(tmem + lane_off + sb * NQ + c, *reinterpret_cast<float(*)[16]>(&s[c]));
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[sb]);
                float* rm = red_max + (jt & 1) * 4 * NQ;
#pragma unroll
                for (int r = 0; r < NQ; ++r) s[r] = (tok < lim[r] && lim[r] - tok <= wp1) ? s[r] * p.scale_log2 : kNegInf;
                warp_rows_reduce<NQ, true>(s, lane, rm + q4 * NQ);
                named_bar_sync(1, 128);
                bool need = false;
                float mx[NQ];
#pragma unroll
                for (int r = 0; r < NQ; ++r) {
                    // Padding rows hold -inf everywhere: mx = -inf, no rescale.
                    mx[r] = fmaxf(fmaxf(rm[r], rm[NQ + r]), fmaxf(rm[2 * NQ + r], rm[3 * NQ + r]));
                    need |= mx[r] > m_ref[r] + kRescaleThreshold;
                }
                if (need) {
                    float alpha[NQ];
#pragma unroll
                    for (int r = 0; r < NQ; ++r) {
                        const float mn = fmaxf(m_ref[r], mx[r]);
                        alpha[r] = (mn == kNegInf) ? 1.f : ex2_approx(m_ref[r] - mn);
                        l_part[r] *= alpha[r];
                        m_ref[r] = mn;
                    }
                    if (i > 0) {
                        // Rescale the accumulated O^T once PV(jt - 1) has landed.
                        // s_full(jt) was committed after PV(jt - 2) was issued,
                        // so pv_done is at most one phase behind here.
                        mbar_wait(pv_done, (jt - 1) & 1, wc);
                        tc_fence_after();
#pragma unroll
                        for (int dvt = 0; dvt < C::kDvTiles; ++dvt) {
#pragma unroll
                            for (int c = 0; c < NQ; c += 16) {
                                float o[16];
                                const uint32_t ta = tmem + lane_off + 2 * NQ + dvt * NQ + c;
                                tmem_ld16(ta, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int k = 0; k < 16; ++k) o[k] *= alpha[c + k];
                                tmem_st16(ta, o);
                            }
                        }
                        tmem_wait_st();
                    }
                }
                if (ts + kKvTile > x.n || ts < x.lo) {
                    // Keys past the row's end or before its window: their V
                    // rows may hold anything (unloaded pages, poisoned slots).
                    // Zero them so that the exact-zero probabilities cannot
                    // meet a NaN in the MMA.
                    const int vs = jt % C::kVStages;
                    mbar_wait(&v_full[vs], (jt / C::kVStages) & 1, wc);
                    if (tok >= x.n || tok < x.lo) {
#pragma unroll
                        for (int c = 0; c < C::kChunks; ++c) {
                            uint4 *row = reinterpret_cast<uint4 *>(sV + vs * C::kTileBytes + c * C::kChunkBytes +
                                                                   row_in_tile * 128);
#pragma unroll
                            for (int k = 0; k < 8; ++k) row[k] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                const int pb = jt & 1;
                mbar_wait(&p_free[pb], ((jt >> 1) & 1) ^ 1, wc);
                uint8_t *pbuf = sP + pb * C::kPBytes;
#pragma unroll
                for (int r = 0; r < NQ; ++r) {
                    // Masked keys and padding rows have s = -inf: p = 0 exactly.
                    const float mu = (m_ref[r] == kNegInf) ? 0.f : m_ref[r];
                    const float pr = ex2_approx(s[r] - mu);
                    l_part[r] += pr;
                    *reinterpret_cast<__nv_bfloat16 *>(pbuf + sw128_offset(r, row_in_tile, NQ)) = __float2bfloat16_rn(pr);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[pb]);
            }
            // ------------------------------------------------------ epilogue
            {
                warp_rows_reduce<NQ, false>(l_part, lane, red_sum + q4 * NQ);
                named_bar_sync(1, 128);
                float L[NQ];
#pragma unroll
                for (int r = 0; r < NQ; ++r)
                    L[r] = (red_sum[r] + red_sum[NQ + r]) + (red_sum[2 * NQ + r] + red_sum[3 * NQ + r]);
                // O^T is final once PV(jt - 2) and PV(jt - 1), the unit's
                // last, have landed.  These are the P-buffer waits of tiles jt
                // and jt + 1: each buffer's phase is at most one behind, while
                // a parity wait on pv_done alone could pass with PV(jt - 2)
                // still in flight.
                mbar_wait(&p_free[jt & 1], ((jt >> 1) & 1) ^ 1, wc);
                mbar_wait(&p_free[(jt + 1) & 1], (((jt + 1) >> 1) & 1) ^ 1, wc);
                tc_fence_after();
#pragma unroll
                for (int dvt = 0; dvt < C::kDvTiles; ++dvt) {
                    float o[NQ];
#pragma unroll
                    for (int c = 0; c < NQ; c += 16)
                        tmem_ld16(tmem + lane_off + 2 * NQ + dvt * NQ + c, *reinterpret_cast<float(*)[16]>(&o[c]));
                    tmem_wait_ld();
                    const int dv = dvt * 128 + row_in_tile;
#pragma unroll
                    for (int r = 0; r < NQ; ++r) {
                        int t, h;
                        if (r >= nrows || !unit_row(p, x, r, t, h)) continue;
                        const float val = L[r] > 0.f ? o[r] / L[r] : 0.f;
                        if (x.single) {
                            __nv_bfloat16 *op = reinterpret_cast<__nv_bfloat16 *>(p.out) + x.b * p.out_stride[0] +
                                                t * p.out_stride[1] + h * p.out_stride[2];
                            op[dv] = __float2bfloat16_rn(val);
                        } else {
                            const int64_t row = ((int64_t)x.b * p.q_len + t) * p.Hq + h;
                            p.ws_o[(row * p.max_pieces + x.k) * D + dv] = val;
                        }
                    }
                }
                if (row_in_tile < nrows) {
                    const int r = row_in_tile;
                    int t, h;
                    if (unit_row(p, x, r, t, h)) {
                        float lse2 = kNegInf;
#pragma unroll
                        for (int k = 0; k < NQ; ++k)
                            if (k == r && L[k] > 0.f) lse2 = m_ref[k] + __log2f(L[k]);
                        if (x.single) {
                            if (p.lse)
                                p.lse[x.b * p.lse_stride[0] + t * p.lse_stride[1] + h * p.lse_stride[2]] =
                                    lse2 * 0.69314718055994531f;
                        } else {
                            const int64_t row = ((int64_t)x.b * p.q_len + t) * p.Hq + h;
                            p.ws_lse[row * p.max_pieces + x.k] = lse2;
                        }
                    }
                }
                tc_fence_before();
                named_bar_sync(1, 128);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
    pdl_launch_dependents();                       // the combine kernel may launch
}

template <int D, int NQ>
cudaError_t launch_t(const DecodeParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                     const CUtensorMap &tv, cudaStream_t stream) {
    using C = DecodeCfg<D, NQ>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<D, NQ>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    cudaError_t le = launch_after_previous(paged_decode_kernel<D, NQ>, dim3(p.grid), dim3(192), C::kSmemBytes,
                                           stream, p, tq, tk, tv);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

// ---------------------------------------------------------------- append
//
// One warp per (b, t, kv head) row: 16-byte loads of eight BF16 values,
// stored as they are or as eight E4M3 codes of x / scale (IEEE division,
// round to nearest even, saturating: the conversion instruction's
// satfinite form).  A slot whose row falls outside the cache records
// FW_ERR_INVALID_ARG and writes nothing.

__device__ void append_rows(const AppendParams &a, int block, int nblocks, int *status) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int64_t r = (int64_t)block * wpb + warp; r < a.rows; r += (int64_t)nblocks * wpb) {
        const int h = (int)(r % a.Hkv);
        const int64_t bt = r / a.Hkv;                    // b * q_len + t
        const int t = (int)(bt % a.q_len);
        const int64_t b = bt / a.q_len;
        int64_t slot = __ldg(a.slot_mapping + bt);
        if (slot < 0) slot = 0;                          // clamp before adding the layer base
        const int64_t row = a.layer_base + slot;
        if (row >= a.cache_rows) {
            if (lane == 0) record_error(status, 1 /* FW_ERR_INVALID_ARG */);
            continue;
        }
        const int64_t page = row / a.ps, off = row % a.ps;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const uint16_t *src = pass ? a.v_new : a.k_new;
            if (!src) break;
            const int64_t *ss = pass ? a.vn_stride : a.kn_stride;
            const int64_t *cs = pass ? a.vc_stride : a.kc_stride;
            const int D = pass ? a.Dv : a.Dk;
            const float sc = pass ? a.v_scale : a.k_scale;
            const uint16_t *srow = src + b * ss[0] + t * ss[1] + h * ss[2];
            const int64_t dst = page * cs[0] + off * cs[1] + h * cs[2];
            for (int d = lane * 8; d < D; d += 256) {
                const uint4 v = *reinterpret_cast<const uint4 *>(srow + d);
                if (a.kv8) {
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    uint32_t out[2];
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const float x0 = __fdiv_rn(__uint_as_float(w[e] << 16), sc);
                        const float x1 = __fdiv_rn(__uint_as_float(w[e] & 0xffff0000u), sc);
                        const float x2 = __fdiv_rn(__uint_as_float(w[e + 1] << 16), sc);
                        const float x3 = __fdiv_rn(__uint_as_float(w[e + 1] & 0xffff0000u), sc);
                        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
                        const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(x2, x3), __NV_SATFINITE, __NV_E4M3);
                        out[e >> 1] = lo | (hi << 16);
                    }
                    uint8_t *base = static_cast<uint8_t *>(pass ? a.v_cache : a.k_cache);
                    *reinterpret_cast<uint2 *>(base + dst + d) = make_uint2(out[0], out[1]);
                } else {
                    uint16_t *base = static_cast<uint16_t *>(pass ? a.v_cache : a.k_cache);
                    *reinterpret_cast<uint4 *>(base + dst + d) = v;
                }
            }
        }
    }
}

__global__ void __launch_bounds__(256) kv_append_kernel(const __grid_constant__ AppendParams a, int *status) {
    append_rows(a, blockIdx.x, gridDim.x, status);
}

// ------------------------------------------------------------------- plan
//
// One block: exclusive prefix PB[b] of the KV tiles each batch row puts in
// the global order (the tiles from the window's first key, or from key 0,
// to ceil(n_b / 128), for each of its units), the total
// T and the range span; rows with no keys get their zero output and -inf LSE
// here, since no range ever covers them.
__global__ void __launch_bounds__(1024) decode_plan_kernel(const __grid_constant__ DecodeParams p) {
    pdl_launch_dependents();                         // the attention kernel waits for this grid to finish
    if (blockIdx.x > 0) {                            // the launch's extra blocks append the new tokens
        append_rows(p.app, blockIdx.x - 1, gridDim.x - 1, p.status);
        return;
    }
    __shared__ int warp_sums[32];
    __shared__ int carry_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t *PB = p.plan + 2;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < p.B; base += 1024) {
        const int b = base + tid;
        const int n = b < p.B ? clamp_len(p, __ldg(p.seq_lens + b)) : 0;
        const int rt = row_tiles(p, n);
        const int t = rt > 0 ? (p.piece_cost + rt) * p.units_per_row : 0;   // each unit: empty slots, then its tiles
        int incl = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += v;
            }
            warp_sums[lane] = w;                     // inclusive over warps
        }
        __syncthreads();
        const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + incl - t;
        if (b < p.B) PB[b] = carry_s + before;
        __syncthreads();
        if (tid == 0) carry_s += warp_sums[31];
        __syncthreads();
    }
    if (tid == 0) {
        const int T = carry_s;
        PB[p.B] = T;
        int span = p.forced_span;
        if (span <= 0) span = max(p.min_span, ceil_div_i(T, max(1, p.grid / max(1, p.range_groups))));
        p.plan[0] = T;
        p.plan[1] = span;
    }
    // Empty rows.
    const int64_t rows = (int64_t)p.B * p.q_len * p.Hq;
    for (int64_t r = tid; r < rows; r += blockDim.x) {
        const int b = (int)(r / ((int64_t)p.q_len * p.Hq));
        if (clamp_len(p, __ldg(p.seq_lens + b)) != 0) continue;
        const int h = (int)(r % p.Hq);
        const int t = (int)((r / p.Hq) % p.q_len);
        __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(p.out) + b * p.out_stride[0] + t * p.out_stride[1] +
                           h * p.out_stride[2];
        for (int dv = 0; dv < p.Dv; ++dv) o[dv] = __float2bfloat16(0.f);
        if (p.lse) p.lse[b * p.lse_stride[0] + t * p.lse_stride[1] + h * p.lse_stride[2]] = kNegInf;
    }
}

// ------------------------------------------------------------------ combine
//
// Merge the split-KV partials of each query row: with per-piece normalised
// outputs o_i and log2-sum-exp values e_i, L = log2 sum_i 2^{e_i} and
// out = sum_i 2^{e_i - L} o_i.  This is the rescale of the online recurrence
// applied across whole pieces ("Flywheel Attention", section 1; the reduction
// kernel of "TokenSpeed-MLA 2.0.1", decode).  One warp per row, float4 loads;
// rows whose unit fits one range were written by the attention kernel.

template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const __grid_constant__ DecodeParams p) {
    pdl_wait();                                      // the attention kernel's partials are written
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)p.B * p.q_len * p.Hq;
    const int64_t row = (int64_t)blockIdx.x * 4 + warp;
    if (row >= rows) return;
    const int h = (int)(row % p.Hq);
    const int t = (int)((row / p.Hq) % p.q_len);
    const int b = (int)(row / ((int64_t)p.Hq * p.q_len));
    const int32_t *PB = p.plan + 2;
    const int span = max(1, __ldg(p.plan + 1));
    const int pb0 = __ldg(PB + b);
    const int vb = (__ldg(PB + b + 1) - pb0) / p.units_per_row;   // slots per unit
    if (vb == 0) return;                             // empty row: written by the plan kernel
    const int tb = vb - p.piece_cost;
    const int g = h / p.G;
    // Row groups that ride on the CTA index share their unit's tile range.
    const int rg = (p.range_groups > 1 && !p.head_ride) ? 0
                 : p.head_mode == 0 ? t / p.tokens_per_unit
                                    : t * p.head_chunks + (h - g * p.G) / p.rows;
    // With the KV heads riding on the CTA index a row's units are its row groups.
    const int unit = p.head_ride ? rg : g * (p.range_groups > 1 ? 1 : p.row_groups) + rg;
    const int pstart = pb0 + unit * vb + p.piece_cost;
    const int npieces = (pstart + tb - 1) / span - pstart / span + 1;
    if (npieces <= 1) return;
    const float *lse_row = p.ws_lse + row * p.max_pieces;
    float m = kNegInf;
    for (int i = lane; i < npieces; i += 32) m = fmaxf(m, lse_row[i]);
    m = warp_max(m);
    constexpr int V = D / 32;                        // floats per lane
    float acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k) acc[k] = 0.f;
    float wsum = 0.f;
    if (m != kNegInf) {
        for (int i = 0; i < npieces; ++i) {
            const float w = ex2_approx(lse_row[i] - m);  // 0 for an empty piece (e = -inf)
            wsum += w;
            const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + (row * p.max_pieces + i) * D) + lane * (V / 4);
#pragma unroll
            for (int k = 0; k < V / 4; ++k) {
                const float4 v = src[k];
                acc[4 * k + 0] += w * v.x; acc[4 * k + 1] += w * v.y;
                acc[4 * k + 2] += w * v.z; acc[4 * k + 3] += w * v.w;
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(p.out) + b * p.out_stride[0] + t * p.out_stride[1] +
                       h * p.out_stride[2] + lane * V;
#pragma unroll
    for (int k = 0; k < V; k += 2)
        *reinterpret_cast<__nv_bfloat162 *>(o + k) = __floats2bfloat162_rn(acc[k] * inv, acc[k + 1] * inv);
    if (lane == 0 && p.lse)
        p.lse[b * p.lse_stride[0] + t * p.lse_stride[1] + h * p.lse_stride[2]] =
            (m == kNegInf) ? kNegInf : (m + __log2f(wsum)) * 0.69314718055994531f;
}

}  // namespace

size_t decode_smem_bytes(int head_dim, int rows) {
    if (head_dim == 128) return rows == 16 ? DecodeCfg<128, 16>::kSmemBytes : DecodeCfg<128, 32>::kSmemBytes;
    return rows == 16 ? DecodeCfg<256, 16>::kSmemBytes : DecodeCfg<256, 32>::kSmemBytes;
}

// Blocks of 32 warps that cover the append rows (at most 64 blocks; each
// warp walks rows with the grid's stride).
static unsigned append_blocks(const AppendParams &a, int warps_per_block) {
    if (a.rows <= 0) return 0;
    const int64_t b = (a.rows + warps_per_block - 1) / warps_per_block;
    return (unsigned)(b < 64 ? b : 64);
}

cudaError_t launch_decode_plan(const DecodeParams &p, cudaStream_t stream) {
    decode_plan_kernel<<<1 + append_blocks(p.app, 32), 1024, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_kv_append(const AppendParams &a, int *status, cudaStream_t stream) {
    const unsigned grid = append_blocks(a, 8);
    if (grid == 0) return cudaSuccess;
    kv_append_kernel<<<grid, 256, 0, stream>>>(a, status);
    return cudaGetLastError();
}

cudaError_t launch_decode_combine(const DecodeParams &p, int head_dim_v, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.B * p.q_len * p.Hq;
    const unsigned grid = (unsigned)((rows + 3) / 4);
    if (head_dim_v == 128) return launch_after_previous(combine_kernel<128>, dim3(grid), dim3(128), 0, stream, p);
    if (head_dim_v == 256) return launch_after_previous(combine_kernel<256>, dim3(grid), dim3(128), 0, stream, p);
    if (head_dim_v == 512) return launch_after_previous(combine_kernel<512>, dim3(grid), dim3(128), 0, stream, p);
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                          const CUtensorMap &tv, int head_dim, cudaStream_t stream,
                          cudaEvent_t timing_start, cudaEvent_t timing_stop, int *launches) {
    *launches = 0;
    cudaError_t e = launch_decode_plan(p, stream);
    if (e != cudaSuccess) return e;
    ++*launches;
    if (timing_start) cudaEventRecord(timing_start, stream);
    if (head_dim == 128 && p.rows == 16) e = launch_t<128, 16>(p, tq, tk, tv, stream);
    else if (head_dim == 128 && p.rows == 32) e = launch_t<128, 32>(p, tq, tk, tv, stream);
    else if (head_dim == 256 && p.rows == 16) e = launch_t<256, 16>(p, tq, tk, tv, stream);
    else if (head_dim == 256 && p.rows == 32) e = launch_t<256, 32>(p, tq, tk, tv, stream);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    ++*launches;
    if (timing_stop) cudaEventRecord(timing_stop, stream);
    if (p.max_pieces > 1) {
        e = launch_decode_combine(p, head_dim, stream);
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    return cudaSuccess;
}

}  // namespace fw
