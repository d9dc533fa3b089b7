// Latent-head paged decode on CTA pairs, sm_103a: the layout of
// "TokenSpeed-MLA 2.0.1" (decode: kv_cache [pages, page_size, 576], values =
// its first 512 columns, 128 query heads over one KV head, up to four query
// tokens), for query-head groups that are a multiple of 128 heads.
//
// Why a pair.  128 query rows of a 512-wide O take all 512 TMEM columns of
// one SM, and 128 rows of 576-wide queries take 144 KB of its shared memory,
// so one SM can hold only 64 rows (the one-CTA latent kernel), which puts
// the MMA at N = 64 and makes every key byte copied into shared memory feed
// 64 rows.  Two SMs of a cluster share the 128 rows of one token instead,
// with tcgen05.mma.cta_group::2 issued by CTA 0 for both (swap-AB):
//   S^T [256 keys x 128 rows]  = K_step [256 x 576] * Q^T
//     CTA r holds keys [128r, 128r + 128) of the step (A, its TMEM lanes) and
//     query rows [64r, 64r + 64) (B, split between the pair);
//   O^T [512 x 128 rows]      += V_step^T [512 x 256] * P^T [256 x 128]
//     as two MMAs of 256 value columns; CTA r holds columns
//     [256h + 128r, 256h + 128r + 128) of half h (A, its TMEM lanes) and
//     P^T for its 64 rows over all 256 keys (B).
// Each SM so runs MMAs at N = 128 and every copied key byte feeds 128 rows.
// TMEM per CTA: two S^T buffers (2 x 128 columns) + O^T (2 x 128 columns).
//
// The softmax warps of CTA r own its 128 keys of a step (thread = key, one
// warp per TMEM lane quadrant and row half) and write P^T rows of those keys
// into the shared memory of the CTA that holds each row half (their own, or
// the partner's through distributed shared memory).  Flywheel's static anchor
// ("Flywheel Attention", section 3.1 and appendix A): a row's anchor is the
// scaled maximum of the first step of a piece over both CTAs' keys, then
// P = 2^(s * scale * log2 e - anchor) with no running max; each step checks
// every exponent against a 64 log2-unit slack, the two CTAs exchange the
// verdict, and a step that fails on either side moves the affected anchors to
// that step's row maxima and rescales l and O^T (the form with rescaling is
// exact for any input; the anchored one equals it up to rounding).
//
// Warp roles (320 threads, one CTA per SM, clusters of two):
//   warp 0     TMA producer of its CTA: its Q^T rows, its keys' four 128-column
//              chunks and 64 rotary columns for QK^T, then its value columns
//              of all 256 keys for PV (read again from L2); copies complete
//              on CTA 0's barriers.
//   warp 1     CTA 0: MMA issuer for the pair (QK^T of step j+1 before PV of
//              step j, so the softmax of step j overlaps it); TMEM owner.
//   warps 2-9  softmax and epilogue (thread = key; then thread = O^T lane).
#include <cuda_bf16.h>

#include "decode_common.cuh"
#include "fw_internal.h"
#include "fw_pair.cuh"
#include "fw_ptx.cuh"

namespace fw {

namespace {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kAnchorSlack = 64.0f;                  // log2 units above the anchor before a rescale

constexpr int kDk = 576, kDv = 512;
constexpr int kRowsCta = 64;                           // query rows each CTA loads (half of MMA N)
constexpr int kKeysCta = kKvTile;                      // keys of a step in one CTA (half of MMA M)
constexpr int kStepKeys = 2 * kKeysCta;
constexpr int kSlots = 3;
constexpr int kHalfBytes = kKeysCta * 128;             // 128 keys x 64 columns, 128-byte swizzle
constexpr int kSlotBytes = 2 * kHalfBytes;             // 128 keys x 128 columns
constexpr int kQChunkBytes = kRowsCta * 128;           // 64 rows x 64 columns
constexpr int kQBytes = kRowsCta * kDk * 2;            // 9 chunks
constexpr int kPBytes = kStepKeys * kRowsCta * 2;      // P^T: one 128-byte row (64 query rows) per key
constexpr int kOffQ = 0;
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kOffRing = kOffP + kPBytes;
constexpr int kOffRot = kOffRing + kSlots * kSlotBytes;
constexpr int kOffBar = kOffRot + kHalfBytes;
// mbarrier array: index of each group (every pointer derives from these, so
// the count cannot drift from the layout)
constexpr int kBarSlotFull = 0;                        // [kSlots], CTA 0's count both CTAs' copies
constexpr int kBarSlotEmpty = kBarSlotFull + kSlots;   // [kSlots]
constexpr int kBarRotFull = kBarSlotEmpty + kSlots;    // [1], CTA 0's
constexpr int kBarRotEmpty = kBarRotFull + 1;          // [1]
constexpr int kBarQFull = kBarRotEmpty + 1;            // [1], CTA 0's
constexpr int kBarQEmpty = kBarQFull + 1;              // [1]
constexpr int kBarSFull = kBarQEmpty + 1;              // [2]
constexpr int kBarSFree = kBarSFull + 2;               // [2], CTA 0's count both CTAs' softmax warps
constexpr int kBarPFull = kBarSFree + 2;               // [1], CTA 0's: one arrival per CTA once its P^T is whole
constexpr int kBarPvDone = kBarPFull + 1;              // [1]: PV j landed (frees both CTAs' P^T)
constexpr int kBarX = kBarPvDone + 1;                  // [2]: the partner's part of an exchange arrived
constexpr int kBarDrain = kBarX + 2;                   // [1]
constexpr int kBarTail = kBarDrain + 1;                // [2]: a producer warp's landing of a value chunk with a tail
constexpr int kBarPTx = kBarTail + 2;                  // [1]: the partner's P^T rows landed in this CTA
constexpr int kNumBars = kBarPTx + 1;
constexpr int kThreads = 352;                          // 11 warps: see the roles below
constexpr int kOffX = kOffBar + ((kNumBars * 8 + 127) / 128) * 128;
constexpr int kOffRed = kOffX + (2 * 128 + 32) * 4;    // xr[2][128] from the partner, xf[2] + pad
constexpr int kOffMisc = kOffRed + 8 * 128 * 4;        // red[4][128], anchors, factors, upper and lower limits
constexpr int kSmemBytes = kOffMisc + 16 + 1024;       // + alignment slack
static_assert(kOffP % 1024 == 0 && kOffRing % 1024 == 0 && kOffRot % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA exceeded");
constexpr uint32_t kColO = 256;
constexpr uint32_t kIdescQK = idesc_bf16_f32(256, 2 * kRowsCta, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(256, 2 * kRowsCta, true, true);

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
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

// kPacked: row groups may straddle tokens (packed rows), so visibility is
// per row; otherwise every row of a group is one token's and shares it.
template <bool kPacked>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
latent_pair_decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem + kOffQ;
    uint8_t *sP = smem + kOffP;
    uint8_t *sRing = smem + kOffRing;
    uint8_t *sRot = smem + kOffRot;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *slot_full = bars + kBarSlotFull;
    uint64_t *slot_empty = bars + kBarSlotEmpty;
    uint64_t *rot_full = bars + kBarRotFull;
    uint64_t *rot_empty = bars + kBarRotEmpty;
    uint64_t *q_full = bars + kBarQFull;
    uint64_t *q_empty = bars + kBarQEmpty;
    uint64_t *s_full = bars + kBarSFull;
    uint64_t *s_free = bars + kBarSFree;
    uint64_t *p_full = bars + kBarPFull;
    uint64_t *pv_done = bars + kBarPvDone;
    uint64_t *xbar = bars + kBarX;
    uint64_t *drain = bars + kBarDrain;
    uint64_t *tail_bar = bars + kBarTail;
    uint64_t *p_tx = bars + kBarPTx;
    float *xr = reinterpret_cast<float *>(smem + kOffX);           // [2][128] written by the partner
    uint32_t *xf = reinterpret_cast<uint32_t *>(xr + 2 * 128);     // [2] partner's flag
    float *red = reinterpret_cast<float *>(smem + kOffRed);        // [4][128] per-quadrant row partials
    float *anchor_s = red + 4 * 128;                               // [128] row anchors
    float *alpha_s = anchor_s + 128;                               // [128] rescale factors / 1 / L
    int *lim_s = reinterpret_cast<int *>(alpha_s + 128);           // [128] end of the keys each row sees
    int *lo_s = lim_s + 128;                                       // [128] first key each row sees
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const uint32_t peer = rank ^ 1u;
    const int pair = (int)blockIdx.x >> 1, npairs = (int)gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) { mbar_init(&slot_full[i], 2); mbar_init(&slot_empty[i], 1); }
        mbar_init(rot_full, 2);
        mbar_init(rot_empty, 1);
        mbar_init(q_full, 2);
        mbar_init(q_empty, 1);
        for (int i = 0; i < 2; ++i) { mbar_init(&s_full[i], 1); mbar_init(&s_free[i], 16); mbar_init(&xbar[i], 1); }
        mbar_init(p_full, 2);
        mbar_init(pv_done, 1);
        mbar_init(drain, 1);
        mbar_init(&tail_bar[0], 1);
        mbar_init(&tail_bar[1], 1);
        mbar_init(p_tx, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) { tmem_alloc_pair(tmem_slot, 512); tmem_relinquish_pair(); }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                            // both CTAs' barriers exist before any remote use
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();                                    // the plan (and appended rows) of this call are written
    const WaitCtx wc{p.status, p.timeout_ns, abort_flag};

    if (warp == 0 || warp == 10) {
        // ------------------------------------------------------------ producers
        // Two warps walk the same item sequence; warp 0 (pw 0) copies the ring
        // items of even index, Q and the rotary chunks, warp 10 (pw 1) the
        // ring items of odd index.  (An L2 prefetch of the pages a few steps
        // ahead made the call ~12% slower: the four row-group pairs of a
        // request already walk its keys side by side.)
        const int pw = warp == 0 ? 0 : 1;
        uint64_t *my_tail = &tail_bar[pw];
        uint32_t m = 0, nq = 0, nr = 0, ntail = 0;
        const int box_rows = p.ps < kKeysCta ? p.ps : kKeysCta;
        // Pages holding keys [ks, ks + 128) below k_end; lane l < that count
        // gets the l-th one's physical page (read one step ahead of use).
        // Pages below a half are powers of two: shifts instead of divisions.
        const int ps_shift = __ffs(p.ps) - 1;
        auto npages_of = [&](int ks, int k_end) -> int {
            if (ks >= k_end) return 0;
            if (p.ps >= kKeysCta) return 1;
            return min(kKeysCta >> ps_shift, (k_end - ks + p.ps - 1) >> ps_shift);
        };
        // Logical page of key ks.
        auto page_of = [&](int ks) { return p.ps < kKeysCta ? ks >> ps_shift : ks / p.ps; };
        // Leading pages of keys [ks, ks + 128) wholly before the page holding
        // the window's first key (lo_page): never looked up nor loaded.
        auto skip_of = [&](int ks, int lo_page) -> int {
            return p.ps >= kKeysCta ? 0 : max(0, lo_page - (ks >> ps_shift));
        };
        // The load is issued a step before the page is copied; its range
        // check waits until then (in fill), so the walk never stalls on it.
        auto lookup = [&](int b, int ks, int k_end, int lo_page) -> int {
            int phys = 0;
            if (lane >= skip_of(ks, lo_page) && lane < npages_of(ks, k_end))
                phys = __ldg(p.block_table + (int64_t)b * p.bt_stride + page_of(ks) + lane);
            return phys;
        };
        // Keys [ks, ks + 128) below k_end, `ncb` 64-column blocks from column
        // col0, into dst ([block][128 keys][128 B]); counted on CTA 0's `full`
        // (one arrival per CTA).  With zero_tail, rows at or past k_end are
        // cleared first: their values may be anything, and a zero probability
        // times a NaN is still NaN.
        auto fill = [&](uint64_t *full, uint8_t *dst, const CUtensorMap *tm, int g, int col0, int ncb, int ks,
                        int k_end, int lo_page, int phys, bool zero_tail) -> bool {
            const int np = npages_of(ks, k_end);
            const int skip = min(np, skip_of(ks, lo_page));
            const bool load = lane >= skip && lane < np;
            const int slot0 = p.ps >= kKeysCta ? ks % p.ps : 0;
            const uint32_t full0 = cluster_addr(full, 0);
            if (load && (unsigned)phys >= (unsigned)p.num_pages) { record_error(p.status, 1); phys = 0; }
            const uint32_t bytes = (uint32_t)((np - skip) * box_rows * 128 * ncb);
            if (!(zero_tail && (ks + kKeysCta > k_end || skip > 0))) {
                if (lane == 0) mbar_arrive_expect_tx_relaxed_cluster(full0, bytes);
                __syncwarp();
                if (load)
                    for (int c = 0; c < ncb; ++c)
                        tma_load_4d_pair(smem_u32(dst + c * kHalfBytes + lane * box_rows * 128), tm, full0,
                                         col0 + c * 64, g, slot0, phys);
                return true;
            }
            if (np > skip) {
                if (lane == 0) mbar_arrive_expect_tx(my_tail, bytes);
                __syncwarp();
                if (load)
                    for (int c = 0; c < ncb; ++c)
                        tma_load_4d(smem_u32(dst + c * kHalfBytes + lane * box_rows * 128), tm, my_tail,
                                    col0 + c * 64, g, slot0, phys);
                if (!dec::warp_wait(my_tail, ntail & 1, wc, lane)) {
                    if (lane == 0) mbar_wait_drain(my_tail, ntail & 1, wc);
                    __syncwarp();
                    return false;
                }
                ++ntail;
            }
            // Rows of pages skipped before the window, and rows at or past k_end.
            const int r0 = max(0, k_end - ks), rh = skip * p.ps;
            for (int idx = lane; idx < (kKeysCta - r0) * 8 * ncb; idx += 32) {
                const int row = r0 + idx / (8 * ncb);
                const int rem = idx % (8 * ncb);
                reinterpret_cast<uint4 *>(dst + (rem >> 3) * kHalfBytes + row * 128)[rem & 7] = make_uint4(0, 0, 0, 0);
            }
            for (int idx = lane; idx < min(rh, r0) * 8 * ncb; idx += 32) {
                const int row = idx / (8 * ncb);
                const int rem = idx % (8 * ncb);
                reinterpret_cast<uint4 *>(dst + (rem >> 3) * kHalfBytes + row * 128)[rem & 7] = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0) mbar_arrive(full);        // CTA 0's own barrier: CTA-scope release
                else mbar_arrive_cluster(full0);
            }
            return true;
        };
        bool ok = true, pend = false;
        int pg = 0, pts = 0, pend_end = 0, pend_lo = 0, pph0 = 0, pph1 = 0;   // the step whose PV is still to be fed
        int lo_page = 0;                                                        // page of the piece's first key
        // This CTA's value columns of both key halves of the pending step.
        auto feed_pv = [&]() -> bool {
            for (int v = 0; v < 4; ++v, ++m) {
                if ((int)(m & 1) != pw) continue;
                const int dh = v >> 1, kh = v & 1;
                const uint32_t sl = m % kSlots;
                if (!dec::warp_wait(&slot_empty[sl], ((m / kSlots) & 1) ^ 1, wc, lane)) return false;
                if (!fill(&slot_full[sl], sRing + sl * kSlotBytes, &tm_v, pg, dh * 256 + (int)rank * 128, 2,
                          pts + kh * kKeysCta, pend_end, pend_lo, kh ? pph1 : pph0, true))
                    return false;
            }
            return true;
        };
        dec::LatentIter it;
        it.init(p, pair, npairs);
        dec::LatentPiece x;
        while (ok && it.next(p, x)) {
            if (pw == 0 && !dec::warp_wait(q_empty, (nq & 1) ^ 1, wc, lane)) { ok = false; break; }
            if (pw == 0 && lane == 0) {
                const uint32_t q_full0 = cluster_addr(q_full, 0);
                mbar_arrive_expect_tx_relaxed_cluster(q_full0, (uint32_t)kQBytes);
                for (int c = 0; c < kDk / 64; ++c) {
                    if (kPacked)       // rows past the last (token, head) read as zeros
                        tma_load_3d_pair(smem_u32(sQ + c * kQChunkBytes), &tm_q, q_full0, c * 64,
                                         x.row0 + (int)rank * kRowsCta, x.b);
                    else
                        tma_load_4d_pair(smem_u32(sQ + c * kQChunkBytes), &tm_q, q_full0, c * 64,
                                         x.h0 + (int)rank * kRowsCta, x.t, x.b);
                }
            }
            __syncwarp();
            ++nq;
            const int nsteps = (x.ntiles + 1) >> 1;
            lo_page = x.lo / p.ps;
            int ph0 = lookup(x.b, x.k_begin, x.k_end, lo_page), ph1 = lookup(x.b, x.k_begin + kKeysCta, x.k_end, lo_page);
            for (int s = 0; s < nsteps && ok; ++s) {
                const int ts = x.k_begin + s * kStepKeys;
                const int c0 = ph0, c1 = ph1;
                if (s + 1 < nsteps) {
                    ph0 = lookup(x.b, ts + kStepKeys, x.k_end, lo_page);
                    ph1 = lookup(x.b, ts + kStepKeys + kKeysCta, x.k_end, lo_page);
                }
                const int own_ks = ts + (int)rank * kKeysCta;
                const int own_ph = rank ? c1 : c0;
                for (int c = 0; c < 4 && ok; ++c, ++m) {
                    if ((int)(m & 1) != pw) continue;
                    const uint32_t sl = m % kSlots;
                    if (!dec::warp_wait(&slot_empty[sl], ((m / kSlots) & 1) ^ 1, wc, lane)) { ok = false; break; }
                    ok = fill(&slot_full[sl], sRing + sl * kSlotBytes, &tm_k, x.g, c * 128, 2, own_ks, x.k_end,
                              lo_page, own_ph, false);
                }
                if (!ok) break;
                if (pw == 0) {
                    if (!dec::warp_wait(rot_empty, (nr & 1) ^ 1, wc, lane)) { ok = false; break; }
                    ok = fill(rot_full, sRot, &tm_k, x.g, 512, 1, own_ks, x.k_end, lo_page, own_ph, false);
                }
                ++nr;
                if (ok && pend) ok = feed_pv();
                pend = true; pg = x.g; pts = ts; pend_end = x.k_end; pend_lo = lo_page; pph0 = c0; pph1 = c1;
            }
        }
        if (ok && pend) ok = feed_pv();
        // CTA 0's full barriers complete only once both CTAs' copies have
        // landed; CTA 0 drains them here, before the pair's final cluster
        // barrier, so neither CTA leaves with a copy in flight.
        if (rank == 0 && pw == 0 && lane == 0) {
            for (uint32_t k = 0; k < (uint32_t)kSlots && k < m; ++k) {
                const uint32_t j = m - 1 - k;
                mbar_wait_drain(&slot_full[j % kSlots], (j / kSlots) & 1, wc);
            }
            if (nr > 0) mbar_wait_drain(rot_full, (nr - 1) & 1, wc);
            if (nq > 0) mbar_wait_drain(q_full, (nq - 1) & 1, wc);
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------- MMA (CTA 0 only)
        if (rank == 0 && lane == 0) {
            uint32_t m = 0, nq = 0, nr = 0, jt = 0, npv = 0;
            uint32_t si = 0, sph = 0;                  // ring slot of item m and its phase bit
            // Descriptors at the tile bases; the loops add compile-time
            // offsets (one integer add per operand and instruction).
            const SDesc q_k = sdesc_sw128_split(smem_u32(sQ), 16, 1024);               // Q^T, K-major
            const SDesc ring_k = sdesc_sw128_split(smem_u32(sRing), 16, 1024);          // key chunks, K-major
            const SDesc ring_mn = sdesc_sw128_split(smem_u32(sRing), kHalfBytes, 1024); // value chunks, MN-major
            const SDesc rot_k = sdesc_sw128_split(smem_u32(sRot), 16, 1024);
            const SDesc p_mn = sdesc_sw128_split(smem_u32(sP), 8192, 1024);             // P^T, MN-major
            // The slot of item m lands on the CTA-0 barrier; the copies are
            // TMA transfers completing on it, so a CTA-scope acquire suffices.
            auto wait_slot = [&]() { return mbar_wait(&slot_full[si], sph, wc); };
            auto next_slot = [&]() {
                ++m;
                if (++si == (uint32_t)kSlots) { si = 0; sph ^= 1u; }
            };
            auto issue_qk = [&](bool last_of_piece) -> bool {
                const uint32_t sb = jt & 1;
                if (!mbar_wait_cluster(&s_free[sb], ((jt >> 1) & 1) ^ 1, wc)) return false;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    if (!wait_slot()) return false;
                    tc_fence_after();
                    const SDesc slot_k{ring_k.lo + si * (kSlotBytes >> 4), ring_k.hi};
                    const SDesc q_c{q_k.lo + (uint32_t)c * (2 * kQChunkBytes >> 4), q_k.hi};
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t a = sdesc_at(slot_k, (kk >> 2) * kHalfBytes + (kk & 3) * 32);
                        const uint64_t b = sdesc_at(q_c, (kk >> 2) * kQChunkBytes + (kk & 3) * 32);
                        mma_pair_ss(tmem + sb * 128, a, b, kIdescQK, (c > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit_pair(&slot_empty[si]);
                    next_slot();
                }
                if (!mbar_wait(rot_full, nr & 1, wc)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t a = sdesc_at(rot_k, kk * 32);
                    const uint64_t b = sdesc_at(q_k, 8 * kQChunkBytes + kk * 32);
                    mma_pair_ss(tmem + sb * 128, a, b, kIdescQK, 1u);
                }
                mma_commit_pair(rot_empty);
                ++nr;
                mma_commit_pair(&s_full[sb]);
                if (last_of_piece) mma_commit_pair(q_empty);
                ++jt;
                return true;
            };
            auto issue_pv = [&](bool first) -> bool {
                if (!mbar_wait_cluster(p_full, npv & 1, wc)) return false;
                tc_fence_after();
#pragma unroll 1
                for (int v = 0; v < 4; ++v) {
                    const int dh = v >> 1, kh = v & 1;
                    if (!wait_slot()) return false;
                    tc_fence_after();
                    const SDesc slot_mn{ring_mn.lo + si * (kSlotBytes >> 4), ring_mn.hi};
                    const SDesc p_h{p_mn.lo + (uint32_t)kh * (kKeysCta * 128 >> 4), p_mn.hi};
                    const uint32_t o_col = tmem + kColO + (uint32_t)dh * 128;
#pragma unroll
                    for (int kk = 0; kk < kKeysCta / 16; ++kk) {
                        const uint64_t a = sdesc_at(slot_mn, kk * 16 * 128);
                        const uint64_t b = sdesc_at(p_h, kk * 16 * 128);
                        mma_pair_ss(o_col, a, b, kIdescPV, (first && kh == 0 && kk == 0) ? 0u : 1u);
                    }
                    mma_commit_pair(&slot_empty[si]);
                    next_slot();
                }
                mma_commit_pair(pv_done);
                ++npv;
                return true;
            };
            bool ok = true, pend = false, pend_first = false;
            dec::LatentIter it;
            it.init(p, pair, npairs);
            dec::LatentPiece x;
            while (ok && it.next(p, x)) {
                if (!mbar_wait(q_full, nq & 1, wc)) { ok = false; break; }
                tc_fence_after();
                ++nq;
                const int nsteps = (x.ntiles + 1) >> 1;
                for (int s = 0; s < nsteps && ok; ++s) {
                    ok = issue_qk(s == nsteps - 1);
                    if (ok && pend) ok = issue_pv(pend_first);
                    pend = true;
                    pend_first = (s == 0);
                }
            }
            if (ok && pend) issue_pv(pend_first);
            // No MMA of the pair may still run when the pair frees TMEM.
            mma_commit_pair(drain);
            mbar_wait_drain(drain, 0, wc);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- softmax / epilogue
        // Thread = key (q4 * 32 + lane) of this CTA's half of a step, for the
        // 64 query rows of its warp's half; in the epilogue, thread = O^T lane
        // (value column) for the same 64 rows.  The 256 threads meet at named
        // barriers, which cannot time out, so a failed wait does not leave the
        // loop: after an abort every wait returns at once and the warps run
        // through their remaining (bounded) iterations together; the status
        // word disowns what they write.  Both CTAs run the same exchanges in
        // the same order (counter xc), so the per-row state they derive from
        // them -- anchors, rescale factors, row sums -- is identical.
        const int sw = warp - 2;                         // 0..7
        const int q4 = warp & 3;                         // TMEM lane quadrant of this warp
        const int half = sw >> 2;                        // query rows [64 half, 64 half + 64)
        const int key = q4 * 32 + lane;
        const int tsw = sw * 32 + lane;                  // 0..255; < 128 combines row tsw
        const int row_base = half * kRowsCta;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const float c2 = p.scale_log2;
        uint32_t jt = 0, xc = 0;
        auto xwait = [&](uint32_t k) { mbar_wait_cluster(&xbar[k & 1], (k >> 1) & 1, wc); };
        // Row values of this CTA (thread tsw < 128 holds row tsw's) go to the
        // partner; every thread returns once the partner's have arrived in
        // xr[xc & 1].  Advances xc.
        auto exchange_rows = [&](float own) {
            const uint32_t par = xc & 1;
            if (tsw == 0) mbar_arrive_expect_tx(&xbar[par], 128 * 4);        // the partner's 128 values
            if (tsw < 128)
                st_async_u32(cluster_addr(&xr[par * 128 + tsw], peer), __float_as_uint(own),
                             cluster_addr(&xbar[par], peer));
            xwait(xc);
            ++xc;
            return par;
        };
        // Per-row maxima of the scaled, masked scores of S^T at `sa` over this
        // CTA's keys: red[q4][row] per warp, then thread tsw < 128 combines row
        // tsw; returns it (other threads: -inf).
        auto rows_max_own = [&](uint32_t sa, int tok, bool uni, bool vis) -> float {
#pragma unroll
            for (int c = 0; c < kRowsCta; c += 16) {
                float v[16];
                tmem_ld16(sa + c, v);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    v[k] = (uni ? vis : (tok >= lo_s[row_base + c + k] && tok < lim_s[row_base + c + k])) ? v[k] * c2
                                                                                                    : kNegInf;
                dec::warp_rows_reduce<16, true>(v, lane, red + q4 * 128 + row_base + c);
            }
            named_bar_sync(1, 256);
            return tsw < 128 ? fmaxf(fmaxf(red[tsw], red[128 + tsw]), fmaxf(red[256 + tsw], red[384 + tsw]))
                             : kNegInf;
        };
        dec::LatentIter it;
        it.init(p, pair, npairs);
        dec::LatentPiece x;
        while (it.next(p, x)) {
            // Row r sees keys lo_s[r] .. lim_s[r] - 1 of the piece: from its
            // window's first key (0 without a window) to its token's causal
            // bound, and no key past the piece (a step's second half may lie
            // beyond a piece that holds an odd number of tiles; those keys
            // belong to the next); nothing for a padding row past the last
            // packed row.  Rows of one group may belong to different tokens.
            if (tsw < 128) {
                const int gr = x.row0 + tsw;
                const int pos = x.n - p.q_len + gr / p.G;             // the row's own key position
                const bool real = gr < p.q_len * p.G;
                lim_s[tsw] = real ? min(x.k_end, p.causal ? pos + 1 : x.n) : 0;
                lo_s[tsw] = real && p.window_left >= 0 ? max(0, pos - p.window_left) : 0;
            }
            named_bar_sync(1, 256);
            // A key inside every row's range is visible to all of the warp's 64
            // rows, one outside all of them to none: then one test serves the
            // whole row set (always, unless the rows straddle a token boundary
            // near this key).
            int hi_min = lim_s[row_base], hi_max = hi_min, lo_min = lo_s[row_base], lo_max = lo_min;
            for (int r = 1; r < kRowsCta; ++r) {
                hi_min = min(hi_min, lim_s[row_base + r]);
                hi_max = max(hi_max, lim_s[row_base + r]);
                lo_min = min(lo_min, lo_s[row_base + r]);
                lo_max = max(lo_max, lo_s[row_base + r]);
            }
            const int nsteps = (x.ntiles + 1) >> 1;
            float lp[2][32];
#pragma unroll
            for (int r = 0; r < 32; ++r) { lp[0][r] = 0.f; lp[1][r] = 0.f; }
            for (int s = 0; s < nsteps; ++s, ++jt) {
                const int tok = x.k_begin + s * kStepKeys + (int)rank * kKeysCta + key;
                const bool vis = tok >= lo_max && tok < hi_min;
                const bool uni = !kPacked || vis || tok < lo_min || tok >= hi_max;
                const uint32_t sb = jt & 1;
                mbar_wait(&s_full[sb], (jt >> 1) & 1, wc);
                tc_fence_after();
                const uint32_t sa = tmem + lane_off + sb * 128 + row_base;
                if (s == 0) {
                    // anchor_s[r]: row r's max over the piece's first step, both
                    // CTAs' keys (0 for a row that sees no key here, and hence
                    // none later in the piece).
                    const float own = rows_max_own(sa, tok, uni, vis);
                    const uint32_t par = exchange_rows(own);
                    if (tsw < 128) {
                        const float mx = fmaxf(own, xr[par * 128 + tsw]);
                        anchor_s[tsw] = mx == kNegInf ? 0.f : mx;
                    }
                    named_bar_sync(1, 256);
                } else {
                    // The check: the largest exponent this step would raise any
                    // row to, on either CTA.
                    // (tcgen05.ld is warp-collective: every lane loads, and a
                    // lane whose key no row sees discards what it loaded.)
                    float xmax = kNegInf;
#pragma unroll
                    for (int c = 0; c < kRowsCta; c += 16) {
                        float s16[16];
                        tmem_ld16(sa + c, s16);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 16; k += 4) {
                            const float4 a = *reinterpret_cast<const float4 *>(anchor_s + row_base + c + k);
                            float e0 = fmaf(s16[k], c2, -a.x), e1 = fmaf(s16[k + 1], c2, -a.y);
                            float e2 = fmaf(s16[k + 2], c2, -a.z), e3 = fmaf(s16[k + 3], c2, -a.w);
                            if (!uni) {            // rows of two tokens meet near this key
                                const int4 L = *reinterpret_cast<const int4 *>(lim_s + row_base + c + k);
                                const int4 F = *reinterpret_cast<const int4 *>(lo_s + row_base + c + k);
                                e0 = tok >= F.x && tok < L.x ? e0 : kNegInf; e1 = tok >= F.y && tok < L.y ? e1 : kNegInf;
                                e2 = tok >= F.z && tok < L.z ? e2 : kNegInf; e3 = tok >= F.w && tok < L.w ? e3 : kNegInf;
                            }
                            xmax = fmaxf(xmax, fmaxf(fmaxf(e0, e1), fmaxf(e2, e3)));
                        }
                    }
                    if (uni && !vis) xmax = kNegInf;
                    const bool mine = named_bar_any(1, 256, xmax > kAnchorSlack);
                    const uint32_t par = xc & 1;
                    if (tsw == 0) {
                        mbar_arrive_expect_tx(&xbar[par], 4);                   // the partner's verdict
                        st_async_u32(cluster_addr(&xf[par], peer), mine ? 1u : 0u, cluster_addr(&xbar[par], peer));
                    }
                    xwait(xc);
                    ++xc;
                    if (mine || xf[par] != 0u) {
                        // Some score rose more than kAnchorSlack above its anchor:
                        // move those anchors to this step's row max and rescale l
                        // and O^T (once the previous PV has landed).
                        const float own = rows_max_own(sa, tok, uni, vis);
                        const uint32_t par2 = exchange_rows(own);
                        if (tsw < 128) {                 // whole warps: sw 0-3
                            const float mx = fmaxf(own, xr[par2 * 128 + tsw]);
                            float a = 1.f;
                            const bool move = mx > anchor_s[tsw] + kAnchorSlack;
                            if (move) {
                                a = ex2_approx(anchor_s[tsw] - mx);
                                anchor_s[tsw] = mx;
                            }
                            alpha_s[tsw] = a;
                            const unsigned moved = __ballot_sync(0xffffffffu, move);
                            if (rank == 0 && lane == 0) count_events(p.counters, kCounterLatentRescales, __popc(moved));
                        }
                        named_bar_sync(1, 256);
#pragma unroll
                        for (int r = 0; r < 32; ++r) {
                            lp[0][r] *= alpha_s[row_base + r];
                            lp[1][r] *= alpha_s[row_base + 32 + r];
                        }
                        mbar_wait(pv_done, (jt - 1) & 1, wc);
                        tc_fence_after();
#pragma unroll 1
                        for (int i = 0; i < 2 * kRowsCta; i += 8) {      // (value half, 8 rows)
                            float o[8];
                            const int r0 = i & (kRowsCta - 1);
                            const uint32_t ta = tmem + lane_off + kColO + (i / kRowsCta) * 128 + row_base + r0;
                            tmem_ld8(ta, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 8; ++k) o[k] *= alpha_s[row_base + r0 + k];
                            tmem_st8(ta, o);
                        }
                        tmem_wait_st();
                    }
                }
                // P^T row of this key for the warp's 64 query rows, packed in
                // pairs (the row sums take the FP32 probabilities), computed
                // while the previous PV may still run.
                uint32_t pk[kRowsCta / 2];
#pragma unroll
                for (int c = 0; c < kRowsCta; c += 16) {
                    float s16[16];
                    tmem_ld16(sa + c, s16);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; k += 4) {
                        const float4 a = *reinterpret_cast<const float4 *>(anchor_s + row_base + c + k);
                        float p0 = ex2_approx(fmaf(s16[k], c2, -a.x)), p1 = ex2_approx(fmaf(s16[k + 1], c2, -a.y));
                        float p2 = ex2_approx(fmaf(s16[k + 2], c2, -a.z)), p3 = ex2_approx(fmaf(s16[k + 3], c2, -a.w));
                        // Masking by selection (an invisible key's score may be
                        // anything); per row only when two tokens meet near the key.
                        if (kPacked && !uni) {
                            const int4 L = *reinterpret_cast<const int4 *>(lim_s + row_base + c + k);
                            const int4 F = *reinterpret_cast<const int4 *>(lo_s + row_base + c + k);
                            p0 = tok >= F.x && tok < L.x ? p0 : 0.f; p1 = tok >= F.y && tok < L.y ? p1 : 0.f;
                            p2 = tok >= F.z && tok < L.z ? p2 : 0.f; p3 = tok >= F.w && tok < L.w ? p3 : 0.f;
                        } else {
                            p0 = vis ? p0 : 0.f; p1 = vis ? p1 : 0.f; p2 = vis ? p2 : 0.f; p3 = vis ? p3 : 0.f;
                        }
                        const int li = (c + k) >> 5, lj = (c + k) & 31;
                        lp[li][lj] += p0; lp[li][lj + 1] += p1; lp[li][lj + 2] += p2; lp[li][lj + 3] += p3;
                        pk[(c + k) >> 1] = pack_bf16x2(p0, p1);
                        pk[((c + k) >> 1) + 1] = pack_bf16x2(p2, p3);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed_cluster(cluster_addr(&s_free[sb], 0));
                // Both CTAs' P^T buffers are free once the previous PV has landed.
                mbar_wait(pv_done, (jt & 1) ^ 1, wc);
                // Into the CTA that holds the warp's row half (128-byte swizzle):
                // plain stores here, asynchronous ones into the partner, whose
                // p_tx counts their bytes.
                const int krow = (int)rank * kKeysCta + key;
                if (half == (int)rank) {
                    uint8_t *prow = sP + krow * 128;
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        *reinterpret_cast<uint4 *>(prow + ((u ^ (krow & 7)) << 4)) =
                            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                    fence_proxy_async_smem();
                } else {
                    const uint32_t prow = cluster_addr(sP + krow * 128, peer);
                    const uint32_t ptx = cluster_addr(p_tx, peer);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        st_async_v4(prow + ((u ^ (krow & 7)) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                                    pk[4 * u + 3], ptx);
                }
                named_bar_sync(1, 256);
                // This CTA's P^T is whole once its own warps' stores are done
                // (the barrier) and the partner's 16 KB have landed (p_tx);
                // one thread makes them visible to the tensor core and tells
                // the MMA issuer.
                if (tsw == 0) {
                    mbar_arrive_expect_tx(p_tx, kKeysCta * 128);
                    mbar_wait_cluster(p_tx, jt & 1, wc);
                    fence_proxy_async_smem();
                    if (rank == 0) mbar_arrive(p_full);
                    else mbar_arrive_cluster(cluster_addr(p_full, 0));
                }
            }
            // ------------------------------------------------------ epilogue
            // Row sums over both CTAs' keys: red[q4][row] per warp, thread
            // tsw < 128 adds row tsw's four parts and the partner's sum, then
            // writes 1 / L (0 for a row that saw no key) and the LSE.
            dec::warp_rows_reduce<32, false>(lp[0], lane, red + q4 * 128 + row_base);
            dec::warp_rows_reduce<32, false>(lp[1], lane, red + q4 * 128 + row_base + 32);
            named_bar_sync(1, 256);
            const float own = tsw < 128 ? (red[tsw] + red[128 + tsw]) + (red[256 + tsw] + red[384 + tsw]) : 0.f;
            const uint32_t par = exchange_rows(own);
            // Packed row gr of the unit is token gr / G, head g * G + gr % G;
            // rows past q_len * G are padding and write nothing.
            const int qG = p.q_len * p.G;
            const int64_t wrow_b = (int64_t)x.b * p.q_len * p.Hq;      // workspace row of (b, 0, 0)
            if (tsw < 128) {
                const float L = own + xr[par * 128 + tsw];
                alpha_s[tsw] = L > 0.f ? 1.f / L : 0.f;
                const float lse2 = L > 0.f ? anchor_s[tsw] + __log2f(L) : kNegInf;
                const int gr = x.row0 + tsw;
                if (rank == 0 && gr < qG) {
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
            named_bar_sync(1, 256);
            mbar_wait(pv_done, (jt - 1) & 1, wc);
            tc_fence_after();
            // Thread = value column dh * 256 + rank * 128 + key; a warp stores
            // 32 consecutive columns of one row at a time.
            const int col = (int)rank * 128 + key;
            __nv_bfloat16 *obase = reinterpret_cast<__nv_bfloat16 *>(p.out) + x.b * p.out_stride[0] + col;
            float *wbase = p.ws_o + col;
#pragma unroll 1
            for (int dh = 0; dh < 2; ++dh) {
#pragma unroll 1
                for (int r0 = 0; r0 < kRowsCta; r0 += 16) {
                    float o[16];
                    tmem_ld16(tmem + lane_off + kColO + dh * 128 + row_base + r0, o);
                    tmem_wait_ld();
                    const int gr0 = x.row0 + row_base + r0;
                    int t = gr0 / p.G, hl = gr0 % p.G;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        if (gr0 + k < qG) {
                            const int h = x.g * p.G + hl;
                            const float v = o[k] * alpha_s[row_base + r0 + k];
                            if (x.single)
                                obase[t * p.out_stride[1] + h * p.out_stride[2] + dh * 256] = __float2bfloat16_rn(v);
                            else
                                wbase[((wrow_b + (int64_t)t * p.Hq + h) * p.max_pieces + x.k) * kDv + dh * 256] = v;
                        }
                        if (++hl == p.G) { hl = 0; ++t; }
                    }
                }
            }
            tc_fence_before();
            // The next piece rewrites red, anchor_s and alpha_s.
            named_bar_sync(1, 256);
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                            // no MMA, copy, store or arrive of the pair is left
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
    pdl_launch_dependents();                       // the combine kernel may launch
}

}  // namespace

size_t latent_pair_decode_smem_bytes() { return kSmemBytes; }

cudaError_t launch_latent_pair_decode(const DecodeParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                                      const CUtensorMap &tv, cudaStream_t stream, cudaEvent_t timing_start,
                                      cudaEvent_t timing_stop, int *launches) {
    *launches = 0;
    if (p.grid % 2 != 0) return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(latent_pair_decode_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(latent_pair_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    cudaError_t e = launch_decode_plan(p, stream);
    if (e != cudaSuccess) return e;
    ++*launches;
    if (timing_start) cudaEventRecord(timing_start, stream);
    // An ordinary launch: starting under the plan kernel (programmatic
    // serialization) measured ~2% slower for this kernel.
    if (p.packed) latent_pair_decode_kernel<true><<<p.grid, kThreads, kSmemBytes, stream>>>(p, tq, tk, tv);
    else latent_pair_decode_kernel<false><<<p.grid, kThreads, kSmemBytes, stream>>>(p, tq, tk, tv);
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
