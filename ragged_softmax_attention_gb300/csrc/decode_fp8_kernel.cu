// Paged grouped-query decode over an FP8 E4M3 KV cache, sm_103a.
//
// "TokenSpeed-MLA 2.0.1" (decode): FP8 inputs, BF16 output.  The cache holds
// E4M3 bytes with one scale per cache (k = k_scale * e4m3, v = v_scale *
// e4m3); HBM traffic per key is half that of a BF16 cache, which is what a
// bandwidth-bound decode gains.
//
// The tensor cores read the E4M3 tiles as TMA lands them (kind::f8f6f4, 32
// keys or dims per instruction): nothing widens K or V.  The 16-bit sides of
// the two products enter as sums of 8-bit terms stacked along the MMA's N
// axis, so one instruction covers all terms while reading its K or V slice
// once:
//   * Q: each BF16 query row is scaled by a power of two 2^e (its largest
//     magnitude lands in [128, 256)) and split into hi + mid E4M3 terms.
//     Every BF16 value of the row down to 2^-10 of that maximum is exactly
//     hi + mid (8 significant bits = two 4-bit terms); S = S_hi + S_mid and
//     2^-e folds into the row's score scale, k_scale too.
//   * P: each probability is rounded to FP16 (as a 16-bit MMA would take it)
//     and split into four E5M2 terms; E5M2 is FP16's upper byte, so the four
//     terms (3 significant bits each) give the FP16 value exactly across
//     FP16's range.  O = O_1 + O_2 + O_3 + O_4, v_scale in the epilogue.
// The arithmetic therefore matches a kernel that widens K and V to FP16 and
// runs FP16 MMAs on FP16 queries and probabilities.
//
// Layout and schedule follow the BF16 decode kernel (swap-AB: S^T [128 keys x
// 2 NQ] = K * [Q_hi; Q_mid]^T, O^T [128 x 4 NQ] += V^T * [P_1..P_4]^T with V^T
// read MN-major straight from the 128-byte key rows; balanced tile ranges;
// split-KV pieces merged by the combine kernel).  Roles:
//   * warp 0 (TMA): per tile one ring stage holding the K and the V tile;
//   * warp 1 issues QK^T (4 instructions) and PV (4 instructions), one
//     commit each: qk_done publishes S; kv_empty frees the ring stage and the
//     P buffer and, for the rescale and the epilogue, marks O^T;
//   * warps 2-9: softmax, two warps per TMEM lane quadrant (thread = key),
//     each with half of the unit's query rows; they also build the Q terms
//     once per unit and zero the V rows of keys past a row's end, so NaN bytes
//     in unused slots never meet an MMA.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "decode_common.cuh"
#include "fw_internal.h"
#include "fw_ptx.cuh"

namespace fw {

namespace {

using namespace dec;

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;   // log2 units: 2^(s - base) stays below 2^8
// Probabilities are taken relative to base - kHeadroom: at most 2^15, inside
// FP16's (and E5M2's) range, with small ones clear of the subnormals.  l
// carries the same factor and the LSE subtracts it again.
constexpr float kHeadroom = 7.0f;
constexpr int D = 128;
constexpr int kQTerms = 2;   // E4M3 terms of a scaled BF16 query
constexpr int kPTerms = 4;   // E5M2 terms of an FP16 probability
constexpr int kSoftmaxThreads = 256;

// kind::f8f6f4 instruction descriptor: FP32 accumulation, A E4M3, B E4M3 (0)
// or E5M2 (1), A K-major or MN-major, B K-major.
__host__ __device__ constexpr uint32_t idesc_f8_f32(uint32_t M, uint32_t N, bool a_mn_major, uint32_t b_fmt) {
    return (1u << 4) | (b_fmt << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Byte offset of (row, col) in a K-major tile of 128-byte rows, 128B swizzle.
__device__ __forceinline__ uint32_t sw128_byte(uint32_t row, uint32_t col) {
    return row * 128u + ((((col >> 4) ^ (row & 7u))) << 4) + (col & 15u);
}

template <int NQ, int R>
struct F8Cfg {
    static constexpr int kStages = NQ == 16 ? 5 : 4;           // ring stages (K tile + V tile each)
    static constexpr int kTileBytes = kKvTile * D;              // 128 keys x 128 E4M3 bytes
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kQ16Bytes = NQ * D * 2;                // BF16 query rows, two 64-column chunks
    static constexpr int kQ8Bytes = kQTerms * NQ * D;           // B of QK^T: row = term * NQ + query row
    static constexpr int kPBytes = kPTerms * NQ * kKvTile;      // B of PV: row = term * NQ + query row
    static constexpr int kRH = R / 2;                           // query rows per softmax warp
    // shared memory map (offsets from a 1024-aligned base)
    static constexpr int kOffRing = 0;
    static constexpr int kOffQ16 = kOffRing + kStages * kStageBytes;
    static constexpr int kOffQ8 = kOffQ16 + 2 * kQ16Bytes;
    static constexpr int kOffP = kOffQ8 + 2 * kQ8Bytes;
    static constexpr int kOffBar = kOffP + 2 * kPBytes;
    static constexpr int kNumBars = 3 * kStages + 4 * 2 + 3 * 2 + 1;
    static constexpr int kOffRedMax = (kOffBar + kNumBars * 8 + 15) / 16 * 16;
    static constexpr int kOffRedSum = kOffRedMax + 2 * 4 * R * 4;
    static constexpr int kOffQExp = kOffRedSum + 4 * R * 4;
    static constexpr int kOffMisc = kOffQExp + 2 * NQ * 4;
    // The row tables (PB and the lengths) take what is left of the budget.
    static constexpr int kOffRows = kOffMisc + 16;
    static constexpr int kRowCap = (232448 - 1024 - kOffRows) / 4 > 4096 ? 4096 : (232448 - 1024 - kOffRows) / 4;
    static constexpr int kSmemBytes = kOffRows + kRowCap * 4 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA exceeded");
    static_assert(kRH % 4 == 0, "softmax rows per warp");
    // TMEM: two S^T buffers (Q terms side by side), then O^T (P terms side by side)
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kSCols = kQTerms * NQ;
    static constexpr uint32_t kColO = 2 * kSCols;
    static constexpr uint32_t kTmemCols = (kColO + kPTerms * NQ) <= 128 ? 128 : 256;
    static_assert(kColO + kPTerms * NQ <= kTmemCols, "TMEM columns");
    static constexpr uint32_t kIdescQK = idesc_f8_f32(128, kQTerms * NQ, false, 0);
    static constexpr uint32_t kIdescPV = idesc_f8_f32(128, kPTerms * NQ, true, 1);
};

// NQ: query rows per unit on the MMA N axis (16 or 32); R: rows the softmax
// carries (8 when a unit holds at most 8 query rows, else NQ).
template <int NQ, int R>
__global__ void __launch_bounds__(320, 1)
paged_decode_fp8_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    using C = F8Cfg<NQ, R>;
    static_assert(R == 8 || R == NQ, "softmax rows");
    constexpr int S = C::kStages;
    constexpr int RH = C::kRH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem + C::kOffRing;
    uint8_t *sQ16 = smem + C::kOffQ16;
    uint8_t *sQ8 = smem + C::kOffQ8;
    uint8_t *sP = smem + C::kOffP;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *k_full = bars;                   // [S] K tile landed
    uint64_t *v_full = k_full + S;             // [S] V tile landed
    uint64_t *kv_empty = v_full + S;           // [S] PV of the stage's tile done: stage, P buffer, O^T
    uint64_t *q16_full = kv_empty + S;         // [2] BF16 Q landed
    uint64_t *q16_free = q16_full + 2;         // [2] BF16 Q read (softmax warps)
    uint64_t *q8_full = q16_free + 2;          // [2] Q terms written (softmax warps)
    uint64_t *q8_free = q8_full + 2;           // [2] the unit's last QK^T done
    uint64_t *qk_done = q8_free + 2;           // [2] S buffer of tile j & 1 ready
    uint64_t *s_free = qk_done + 2;            // [2] S buffer read (softmax warps)
    uint64_t *p_full = s_free + 2;             // [2] P terms written (softmax warps)
    uint64_t *drain = p_full + 2;              // [1]
    float *red_max = reinterpret_cast<float *>(smem + C::kOffRedMax);   // [2][4][R]
    float *red_sum = reinterpret_cast<float *>(smem + C::kOffRedSum);   // [4][R]
    int *q_exp = reinterpret_cast<int *>(smem + C::kOffQExp);           // [2][NQ]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&k_full[i], 1); mbar_init(&v_full[i], 1); mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q16_full[i], 1); mbar_init(&q16_free[i], 8);
            mbar_init(&q8_full[i], 8); mbar_init(&q8_free[i], 1);
            mbar_init(&qk_done[i], 1); mbar_init(&s_free[i], 8); mbar_init(&p_full[i], 8);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) { tmem_alloc(tmem_slot, C::kTmemCols); tmem_relinquish(); }
    // Zero the query and probability buffers once: padding rows stay exact zeros.
    for (int i = threadIdx.x; i < (C::kOffBar - C::kOffQ16) / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(sQ16)[i] = make_uint4(0, 0, 0, 0);
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
        int jt = 0, ju = 0, issued = 0;
        const int box_rows = p.ps < kKvTile ? p.ps : kKvTile;
        const int pages_per_tile = p.ps < kKvTile ? kKvTile / p.ps : 1;
        const uint32_t q_rows = p.head_mode == 0 ? (uint32_t)(p.G * p.tokens_per_unit) : (uint32_t)p.rows;
        PieceIter it;
        it.init(p, rows);
        Unit x;
        while (it.next(p, x)) {
            const int qs = ju & 1;
            if (!warp_wait(&q16_free[qs], ((ju >> 1) & 1) ^ 1, wc, lane)) goto producer_done;
            if (lane == 0) {
                int h0, t0;
                if (p.head_mode == 0) { h0 = x.g * p.G; t0 = x.rg * p.tokens_per_unit; }
                else { t0 = x.rg / p.head_chunks; h0 = x.g * p.G + (x.rg % p.head_chunks) * p.rows; }
                mbar_arrive_expect_tx(&q16_full[qs], 2u * q_rows * 128u);
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    tma_load_4d(smem_u32(sQ16 + qs * C::kQ16Bytes + c * NQ * 128), &tm_q, &q16_full[qs], c * 64, h0,
                                t0, x.b);
            }
            __syncwarp();
            {
                // Physical page numbers, 64 logical pages at a time in two
                // 32-entry register windows (lane l holds page win + l and
                // win + 32 + l), the next window fetched while the current one
                // is in use: no tile waits on a block-table read (a read per tile
                // on the copy warp's path measured as the bound of this kernel).
                // Entries past the row's last page, or wholly before its window,
                // are never read.
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
                    // Leading pages wholly before the window are neither looked
                    // up nor loaded (their rows are masked, their V rows zeroed).
                    const int skip = min(npages, max(0, lp_first - lp0));
                    const bool load = lane >= skip && lane < npages;
                    const int idx = lp0 + lane - win;          // < 64 for loading lanes (npages <= 16)
                    const int from_cur = __shfl_sync(0xffffffffu, cur, idx & 31);
                    const int from_nxt = __shfl_sync(0xffffffffu, nxt, idx & 31);
                    int phys = idx < 32 ? from_cur : from_nxt;
                    if (load && (unsigned)phys >= (unsigned)p.num_pages) { record_error(p.status, 1); phys = 0; }
                    const uint32_t bytes = (uint32_t)((npages - skip) * box_rows * 128);
                    const int s = jt % S;
                    if (!warp_wait(&kv_empty[s], ((jt / S) & 1) ^ 1, wc, lane)) goto producer_done;
                    uint8_t *stage = ring + s * C::kStageBytes;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&k_full[s], bytes);
                        mbar_arrive_expect_tx(&v_full[s], bytes);
                    }
                    __syncwarp();
                    if (load) {
                        tma_load_4d(smem_u32(stage + lane * box_rows * 128), &tm_k, &k_full[s], 0, x.g, slot0, phys);
                        tma_load_4d(smem_u32(stage + C::kTileBytes + lane * box_rows * 128), &tm_v, &v_full[s], 0,
                                    x.g, slot0, phys);
                    }
                    issued = jt + 1;
                }
            }
            ++ju;
        }
    producer_done:
        if (lane == 0) {
            for (int k = 0; k < S && k < issued; ++k) {
                const int j = issued - 1 - k;
                mbar_wait_drain(&k_full[j % S], (j / S) & 1, wc);
                mbar_wait_drain(&v_full[j % S], (j / S) & 1, wc);
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
            const SDesc ring_d = sdesc_sw128_split(smem_u32(ring), 16, 1024);
            const SDesc p_d = sdesc_sw128_split(smem_u32(sP), 16, 1024);
            const SDesc q_d = sdesc_sw128_split(smem_u32(sQ8), 16, 1024);
            auto issue_pv = [&](int jj, bool first) -> bool {
                const int s = jj % S;
                const int pb = jj & 1;
                if (!mbar_wait(&v_full[s], (jj / S) & 1, wc)) return false;
                if (!mbar_wait(&p_full[pb], (jj >> 1) & 1, wc)) return false;
                tc_fence_after();
                const SDesc v_s{ring_d.lo + (uint32_t)(s * C::kStageBytes + C::kTileBytes) / 16u, ring_d.hi};
                const SDesc p_s{p_d.lo + (uint32_t)(pb * C::kPBytes) / 16u, p_d.hi};
#pragma unroll
                for (int kk = 0; kk < kKvTile / 32; ++kk) {
                    // A = V^T, MN-major: 32 key rows of 128 bytes per step.
                    const uint64_t a = sdesc_at(v_s, kk * 32 * 128);
                    const uint64_t b = sdesc_at(p_s, kk * 32);
                    mma_f8_ss(tmem + C::kColO, a, b, C::kIdescPV, (first && kk == 0) ? 0u : 1u);
                }
                mma_commit(&kv_empty[s]);
                return true;
            };
            PieceIter it;
            it.init(p, rows);
            Unit x;
            while (it.next(p, x)) {
                const int qs = ju & 1;
                // The previous unit's last PV goes out before this unit's Q
                // terms are awaited: the softmax warps build them only after
                // their epilogue, which waits for that PV.
                if (pend >= 0) {
                    if (!issue_pv(pend, pend_first)) goto mma_done;
                    pend = -1;
                }
                if (!mbar_wait(&q8_full[qs], (ju >> 1) & 1, wc)) goto mma_done;
                for (int i = 0; i < x.ntiles; ++i, ++jt) {
                    const int s = jt % S;
                    const int sb = jt & 1;
                    if (!mbar_wait(&k_full[s], (jt / S) & 1, wc)) goto mma_done;
                    if (!mbar_wait(&s_free[sb], ((jt >> 1) & 1) ^ 1, wc)) goto mma_done;
                    tc_fence_after();
                    const SDesc k_s{ring_d.lo + (uint32_t)(s * C::kStageBytes) / 16u, ring_d.hi};
                    const SDesc q_s{q_d.lo + (uint32_t)(qs * C::kQ8Bytes) / 16u, q_d.hi};
#pragma unroll
                    for (int kk = 0; kk < D / 32; ++kk) {
                        const uint64_t a = sdesc_at(k_s, kk * 32);
                        const uint64_t b = sdesc_at(q_s, kk * 32);
                        mma_f8_ss(tmem + C::kColS + sb * C::kSCols, a, b, C::kIdescQK, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&qk_done[sb]);
                    if (i == x.ntiles - 1) mma_commit(&q8_free[qs]);
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
        // Thread = key of the tile (TMEM lane) and, in the epilogue, value
        // column; warp pair (w, w + 4) shares a lane quadrant and splits the
        // rows.  Waits that fail do not change the control flow; the bounded
        // iterations wind down under the recorded status.
        const int q4 = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r0 = half * RH;
        const int key = q4 * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const int st = threadIdx.x - 64;                       // 0..255
        int jt = 0, ju = 0;
        PieceIter it;
        it.init(p, rows);
        Unit x;
        // ---- query terms of unit nu: BF16 row * 2^e = hi + mid, both E4M3.
        // Built for the next unit before this unit's epilogue, so that the
        // MMA warp can start the next unit's QK^T while the epilogue waits
        // for the last PV and writes O.
        auto build_q8 = [&](int nu) {
            const int qs = nu & 1;
            mbar_wait(&q16_full[qs], (nu >> 1) & 1, wc);
            mbar_wait(&q8_free[qs], ((nu >> 1) & 1) ^ 1, wc);
            {
                constexpr int TPR = kSoftmaxThreads / NQ;          // threads per query row
                constexpr int EPT = D / TPR;                       // elements per thread (8 or 16)
                const int rq = st / TPR;
                const int c0 = (st % TPR) * EPT;
                float y[EPT];
                const uint8_t *q16 = sQ16 + qs * C::kQ16Bytes + (c0 >> 6) * NQ * 128 + rq * 128;
#pragma unroll
                for (int u = 0; u < EPT / 8; ++u) {
                    const int unit = ((c0 & 63) >> 3) + u;
                    const uint4 w = *reinterpret_cast<const uint4 *>(q16 + ((unit ^ (rq & 7)) << 4));
                    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        y[8 * u + 2 * e] = __uint_as_float(wd[e] << 16);
                        y[8 * u + 2 * e + 1] = __uint_as_float(wd[e] & 0xffff0000u);
                    }
                }
                float amax = 0.f;
#pragma unroll
                for (int e = 0; e < EPT; ++e) amax = fmaxf(amax, fabsf(y[e]));
#pragma unroll
                for (int o = TPR / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                int ex = 0;
                if (amax > 0.f && amax <= 3.0e38f) ex = min(100, max(-100, 7 - ilogbf(amax)));
                const float mul = __int_as_float((ex + 127) << 23);     // 2^ex, exact
                uint8_t hi[EPT], mid[EPT];
#pragma unroll
                for (int e = 0; e < EPT; e += 2) {
                    const float a = y[e] * mul, b = y[e + 1] * mul;
                    const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
                    const float2 hb = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3)));
                    const __nv_fp8x2_storage_t m2 =
                        __nv_cvt_float2_to_fp8x2(make_float2(a - hb.x, b - hb.y), __NV_SATFINITE, __NV_E4M3);
                    hi[e] = (uint8_t)(h2 & 0xff); hi[e + 1] = (uint8_t)(h2 >> 8);
                    mid[e] = (uint8_t)(m2 & 0xff); mid[e + 1] = (uint8_t)(m2 >> 8);
                }
                uint8_t *q8 = sQ8 + qs * C::kQ8Bytes;
#pragma unroll
                for (int t = 0; t < kQTerms; ++t) {
                    const uint8_t *src = t == 0 ? hi : mid;
                    const uint32_t row = (uint32_t)(t * NQ + rq);
#pragma unroll
                    for (int e = 0; e < EPT; e += 8) {
                        uint2 v;
                        v.x = src[e] | (src[e + 1] << 8) | (src[e + 2] << 16) | ((uint32_t)src[e + 3] << 24);
                        v.y = src[e + 4] | (src[e + 5] << 8) | (src[e + 6] << 16) | ((uint32_t)src[e + 7] << 24);
                        *reinterpret_cast<uint2 *>(q8 + sw128_byte(row, (uint32_t)(c0 + e))) = v;
                    }
                }
                if (st % TPR == 0) q_exp[qs * NQ + rq] = ex;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) { mbar_arrive(&q16_free[qs]); mbar_arrive(&q8_full[qs]); }
            named_bar_sync(3, kSoftmaxThreads);                   // q_exp of unit nu visible
        };
        // Token, head and visible-key bound of this warp's rows of a unit.
        // Warps of up to 4 rows work them out for the next unit while the
        // current one runs (with the next unit's descriptor, fetched then
        // too), so a piece boundary waits on neither; wider warps, short of
        // registers, work them out at the unit's start and again in its
        // epilogue.
        constexpr bool kKeepRows = RH <= 4;
        constexpr int KR = kKeepRows ? RH : 1;
        struct Rows {
            int t[KR], h[KR], lim[RH];
            unsigned ok;
            int nrows;
        };
        auto rows_of = [&](const Unit &u, Rows &w) {
            w.ok = 0;
            w.nrows = 0;
#pragma unroll
            for (int r = 0; r < RH; ++r) {
                int t, h;
                const bool ok = unit_row(p, u, r0 + r, t, h);
                if constexpr (kKeepRows) {
                    w.t[r] = t;
                    w.h[r] = h;
                }
                if (ok) { w.ok |= 1u << r; w.nrows = r + 1; }
                w.lim[r] = ok ? (p.causal ? min(u.n, u.n - p.q_len + t + 1) : u.n) : 0;
            }
        };
        bool have = it.next(p, x);
        if (have) build_q8(0);
        Rows cur, nxt;
        if (have) rows_of(x, cur);
        Unit nx;
        while (have) {
            const int qs = ju & 1;
            if (!kKeepRows) rows_of(x, cur);
            const int nrows = cur.nrows;
            const unsigned row_ok = cur.ok;
            int lim[RH];
            float rs[RH];
#pragma unroll
            for (int r = 0; r < RH; ++r) {
                lim[r] = cur.lim[r];
                rs[r] = p.scale_log2 * __int_as_float((127 - q_exp[qs * NQ + r0 + r]) << 23);
            }
            auto row_of = [&](int r, int &t, int &h) -> bool {
                if constexpr (kKeepRows) {
                    t = cur.t[r];
                    h = cur.h[r];
                    return (row_ok >> r) & 1u;
                } else {
                    return unit_row(p, x, r0 + r, t, h);
                }
            };
            // The next unit's descriptor (and rows), while this unit runs.
            bool next_unit = false;
            if constexpr (kKeepRows) {
                next_unit = it.next(p, nx);
                if (next_unit) rows_of(nx, nxt);
            }
            // Sliding window: a row with visible-key bound lim sees keys
            // lim - 1 - W .. lim - 1, i.e. lim - tok <= W + 1.
            const int wp1 = p.window_left < 0 ? 0x7fffffff : p.window_left + 1;
            float m_ref[RH], l_part[RH];
#pragma unroll
            for (int r = 0; r < RH; ++r) { m_ref[r] = kNegInf; l_part[r] = 0.f; }
            for (int i = 0; i < x.ntiles; ++i, ++jt) {
                const int ts = x.k_begin + i * kKvTile;
                const int tok = ts + key;
                const int sb = jt & 1;
                mbar_wait(&qk_done[sb], (jt >> 1) & 1, wc);
                tc_fence_after();
                float s[RH], sm[RH];
                tmem_ld_cols<RH>(tmem + lane_off + C::kColS + sb * C::kSCols + r0, s);
                tmem_ld_cols<RH>(tmem + lane_off + C::kColS + sb * C::kSCols + NQ + r0, sm);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[sb]);
                float *rm = red_max + (jt & 1) * 4 * R;
#pragma unroll
                for (int r = 0; r < RH; ++r)
                    s[r] = (tok < lim[r] && lim[r] - tok <= wp1) ? (s[r] + sm[r]) * rs[r] : kNegInf;
                warp_rows_reduce<RH, true>(s, lane, rm + q4 * R + r0);
                named_bar_sync(1 + half, 128);
                bool need = false;
                float mx[RH];
#pragma unroll
                for (int r = 0; r < RH; r += 4) {
                    // Padding rows hold -inf everywhere: mx = -inf, no rescale.
                    float4 m4 = *reinterpret_cast<const float4 *>(rm + r0 + r);
#pragma unroll
                    for (int q = 1; q < 4; ++q) {
                        const float4 o4 = *reinterpret_cast<const float4 *>(rm + q * R + r0 + r);
                        m4.x = fmaxf(m4.x, o4.x); m4.y = fmaxf(m4.y, o4.y);
                        m4.z = fmaxf(m4.z, o4.z); m4.w = fmaxf(m4.w, o4.w);
                    }
                    mx[r] = m4.x; mx[r + 1] = m4.y; mx[r + 2] = m4.z; mx[r + 3] = m4.w;
                }
#pragma unroll
                for (int r = 0; r < RH; ++r) need |= mx[r] > m_ref[r] + kRescaleThreshold;
                if (need) {
                    float alpha[RH];
#pragma unroll
                    for (int r = 0; r < RH; ++r) {
                        const float mn = fmaxf(m_ref[r], mx[r]);
                        alpha[r] = (mn == kNegInf) ? 1.f : ex2_approx(m_ref[r] - mn);
                        l_part[r] *= alpha[r];
                        m_ref[r] = mn;
                    }
                    if (i > 0) {
                        // Rescale once PV(jt - 1) has landed; PV(jt - 2) has,
                        // as qk_done(jt) was committed after it was issued.
                        mbar_wait(&kv_empty[(jt - 1) % S], ((jt - 1) / S) & 1, wc);
                        tc_fence_after();
#pragma unroll
                        for (int t = 0; t < kPTerms; ++t) {
                            float o[RH];
                            const uint32_t ta = tmem + lane_off + C::kColO + t * NQ + r0;
                            tmem_ld_cols<RH>(ta, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < RH; ++k) o[k] *= alpha[k];
                            tmem_st_cols<RH>(ta, o);
                        }
                        tmem_wait_st();
                    }
                }
                if (half == 0 && (ts + kKvTile > x.n || ts < x.lo)) {
                    // Keys past the row's end or before its window: their V
                    // rows may hold anything (unloaded pages, poisoned slots).
                    // Zero them so that the exact-zero probabilities cannot
                    // meet a NaN in the MMA.
                    const int s = jt % S;
                    mbar_wait(&v_full[s], (jt / S) & 1, wc);
                    if (tok >= x.n || tok < x.lo) {
                        uint4 *row = reinterpret_cast<uint4 *>(ring + s * C::kStageBytes + C::kTileBytes + key * 128);
#pragma unroll
                        for (int k = 0; k < 8; ++k) row[k] = make_uint4(0, 0, 0, 0);
                    }
                }
                const int pb = jt & 1;
                if (jt >= 2) mbar_wait(&kv_empty[(jt - 2) % S], ((jt - 2) / S) & 1, wc);   // PV(jt - 2) read P buffer pb
                uint8_t *pbuf = sP + pb * C::kPBytes;
#pragma unroll
                for (int r = 0; r < RH; r += 2) {
                    // Masked keys and padding rows have s = -inf: p = 0 exactly.
                    const float mu0 = (m_ref[r] == kNegInf) ? 0.f : m_ref[r] - kHeadroom;
                    const float mu1 = (m_ref[r + 1] == kNegInf) ? 0.f : m_ref[r + 1] - kHeadroom;
                    const float p0 = ex2_approx(s[r] - mu0);
                    const float p1 = ex2_approx(s[r + 1] - mu1);
                    l_part[r] += p0;
                    l_part[r + 1] += p1;
                    // FP16 value -> four E5M2 terms: round, subtract exactly, repeat.
                    __half2 h = __floats2half2_rn(p0, p1);
#pragma unroll
                    for (int t = 0; t < kPTerms; ++t) {
                        const __nv_fp8x2_storage_t e2 =
                            __nv_cvt_halfraw2_to_fp8x2(__half2_raw(h), __NV_SATFINITE, __NV_E5M2);
                        pbuf[sw128_byte((uint32_t)(t * NQ + r0 + r), (uint32_t)key)] = (uint8_t)(e2 & 0xff);
                        pbuf[sw128_byte((uint32_t)(t * NQ + r0 + r + 1), (uint32_t)key)] = (uint8_t)(e2 >> 8);
                        if (t + 1 < kPTerms) h = __hsub2(h, __half2(__nv_cvt_fp8x2_to_halfraw2(e2, __NV_E5M2)));
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[pb]);
            }
            if constexpr (!kKeepRows) next_unit = it.next(p, nx);
            if (next_unit) build_q8(ju + 1);
            // ------------------------------------------------------ epilogue
            {
                warp_rows_reduce<RH, false>(l_part, lane, red_sum + q4 * R + r0);
                named_bar_sync(1 + half, 128);
                float L[RH];
#pragma unroll
                for (int r = 0; r < RH; ++r)
                    L[r] = (red_sum[r0 + r] + red_sum[R + r0 + r]) + (red_sum[2 * R + r0 + r] + red_sum[3 * R + r0 + r]);
                // O^T is final once PV(jt - 2) and PV(jt - 1), the unit's
                // last, have landed.  The softmax waits each stage's phases in
                // order, so neither wait can be two phases behind.
                if (jt >= 2) mbar_wait(&kv_empty[(jt - 2) % S], ((jt - 2) / S) & 1, wc);
                mbar_wait(&kv_empty[(jt - 1) % S], ((jt - 1) / S) & 1, wc);
                tc_fence_after();
                float o[RH];
#pragma unroll
                for (int r = 0; r < RH; ++r) o[r] = 0.f;
#pragma unroll
                for (int t = 0; t < kPTerms; ++t) {
                    float ot[RH];
                    tmem_ld_cols<RH>(tmem + lane_off + C::kColO + t * NQ + r0, ot);
                    tmem_wait_ld();
#pragma unroll
                    for (int r = 0; r < RH; ++r) o[r] += ot[r];
                }
                const int dv = key;
#pragma unroll
                for (int r = 0; r < RH; ++r) {
                    int t, h;
                    if (r >= nrows || !row_of(r, t, h)) continue;
                    const float val = L[r] > 0.f ? o[r] / L[r] * p.out_scale : 0.f;
                    if (x.single) {
                        __nv_bfloat16 *op = reinterpret_cast<__nv_bfloat16 *>(p.out) + x.b * p.out_stride[0] +
                                            t * p.out_stride[1] + h * p.out_stride[2];
                        op[dv] = __float2bfloat16_rn(val);
                    } else {
                        const int64_t row = ((int64_t)x.b * p.q_len + t) * p.Hq + h;
                        p.ws_o[(row * p.max_pieces + x.k) * D + dv] = val;
                    }
                }
                if (q4 == 0 && lane < nrows && ((row_ok >> lane) & 1u)) {
                    const int r = lane;
                    {
                        int t = 0, h = 0;
                        float lse2 = kNegInf;
#pragma unroll
                        for (int k = 0; k < RH; ++k) {
                            if (k != r) continue;
                            row_of(k, t, h);
                            if (L[k] > 0.f) lse2 = m_ref[k] - kHeadroom + __log2f(L[k]);
                        }
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
                named_bar_sync(1 + half, 128);
            }
            ++ju;
            x = nx;
            if (kKeepRows) cur = nxt;
            have = next_unit;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
    pdl_launch_dependents();                       // the combine kernel may launch
}

template <int NQ, int R>
cudaError_t launch_fp8_t(const DecodeParams &p, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         cudaStream_t stream) {
    using C = F8Cfg<NQ, R>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(paged_decode_fp8_kernel<NQ, R>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    cudaError_t le = launch_after_previous(paged_decode_fp8_kernel<NQ, R>, dim3(p.grid), dim3(320), C::kSmemBytes,
                                           stream, p, tq, tk, tv);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_fp8(const DecodeParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                              const CUtensorMap &tv, cudaStream_t stream, cudaEvent_t timing_start,
                              cudaEvent_t timing_stop, int *launches) {
    *launches = 0;
    cudaError_t e = launch_decode_plan(p, stream);
    if (e != cudaSuccess) return e;
    ++*launches;
    if (timing_start) cudaEventRecord(timing_start, stream);
    const bool narrow = p.head_mode == 0 && p.G * p.tokens_per_unit <= 8;
    if (p.rows == 16 && narrow) e = launch_fp8_t<16, 8>(p, tq, tk, tv, stream);
    else if (p.rows == 16) e = launch_fp8_t<16, 16>(p, tq, tk, tv, stream);
    else if (p.rows == 32) e = launch_fp8_t<32, 32>(p, tq, tk, tv, stream);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    ++*launches;
    if (timing_stop) cudaEventRecord(timing_stop, stream);
    if (p.max_pieces > 1) {
        e = launch_decode_combine(p, D, stream);
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    return cudaSuccess;
}

}  // namespace fw
