// Ragged (varlen) prefill, sm_103a: packed Q [total_q, Hq, D], K/V
// [total_k, Hkv, D] described by cumulative sequence lengths, causal
// (bottom-right aligned) or not ("TokenSpeed-MLA 2.0.1", MLA Prefill: ragged
// varlen FMHA without padding, Q and KV packs may differ).
//
// Orientation: a 128-row query tile is the MMA M axis, a 128-key tile is N:
//   S [128 x 128]  = Q_tile * K_tile^T          (tcgen05, FP32 in TMEM)
//   O [128 x D]   += P [128 x 128] * V_tile      (tcgen05, FP32 in TMEM)
// with the static-anchor softmax of "Flywheel Attention", section 3.1 and
// appendix A, in base 2: each row's anchor is the max of its first visible
// tile, P = 2^(s - anchor) needs no running max, and a check of the running
// sum after each tile replays the tile with the online rescale (section 1
// recurrence) when a score could have outgrown the anchor.
//
// D = 128: a unit is two consecutive query tiles of one head that share every
// K/V tile load; S and O of both live in TMEM (4 x 128 columns) and two
// softmax warpgroups alternate with the tensor core: while one group turns
// its S into P, the MMA warp runs the other tile's PV and QK ("Flywheel
// Attention", section 1: two compute groups alternate so that one's softmax
// overlaps the other's matmuls).  D = 256: the same two query tiles run on a
// pair of CTAs (varlen_prefill_pair_kernel below), one tile each, with
// cta_group::2 MMAs whose K and V operands the pair splits between its SMs.
//
// Warp roles: warp 0 TMA producer (Q tiles, then K_j / V_j through a ring of
// shared-memory slots), warp 1 MMA issuer of query tile 0 and TMEM owner,
// warp 2 MMA issuer of query tile 1 (warp 3 idle),
// then one warpgroup per query tile (thread = query row: the row max and sum
// are thread-local; the row of S stays in registers).
#include <cuda_bf16.h>

#include "fw_internal.h"
#include "fw_ptx.cuh"
#include "fw_pair.cuh"

namespace fw {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();
// Budget on a row's running sum of 2^(s - anchor): 2^32 keeps l and every
// entry of O (|O| <= l * max|v|) far inside FP32 for |v| < 2^90; Flywheel's
// appendix A derives its budget the same way, in natural-log units.
constexpr float kAnchorBudget = 4294967296.0f;
// Online mode: the base moves only when a row max rises more than this many
// log2 units above it ("TokenSpeed-MLA 2.0.1" keeps its base for rises up to
// 8 in split mode), so every p <= 2^8.
constexpr float kRescaleSlack = 8.0f;
constexpr int kQTile = 128;
constexpr int kCostBins = 4096;

// Head dim 128, two query tiles per CTA.
struct PrefillCfg {
    static constexpr int D = 128;
    static constexpr int kNumQ = 2;                             // query tiles per unit
    static constexpr int kChunks = D / 64;
    static constexpr int kChunkBytes = 128 * 128;              // 128 rows x 64 bf16 columns
    static constexpr int kTileBytes = 128 * D * 2;              // one Q, K or V tile
    static constexpr int kSlotBytes = kTileBytes;
    static constexpr int kSlots = 4;                            // K/V ring slots
    static constexpr int kOffQ = 0;
    static constexpr int kOffRing = kOffQ + kNumQ * kTileBytes;
    static constexpr int kOffBar = kOffRing + kSlots * kSlotBytes;
    // mbarrier array: index of each group (every pointer below derives from
    // these, so the count cannot drift from the layout)
    static constexpr int kBarSlotFull = 0;                      // [kSlots]
    static constexpr int kBarSlotEmpty = kBarSlotFull + kSlots;  // [kSlots]
    static constexpr int kBarQFull = kBarSlotEmpty + kSlots;     // [1]
    static constexpr int kBarQEmpty = kBarQFull + 1;             // [1]
    static constexpr int kBarSFull = kBarQEmpty + 1;             // [2] per query tile
    static constexpr int kBarPFull = kBarSFull + 2;              // [2]
    static constexpr int kBarPvDone = kBarPFull + 2;             // [2]
    static constexpr int kBarDrain = kBarPvDone + 2;             // [2]
    static constexpr int kBarIssued = kBarDrain + 2;             // [2]
    static constexpr int kBarPHalf = kBarIssued + 2;             // [2]
    static constexpr int kBarPvhDone = kBarPHalf + 2;            // [2]
    static constexpr int kSchedSlots = 4;                        // unit records in flight
    static constexpr int kBarSchedFull = kBarPvhDone + 2;        // [kSchedSlots]
    static constexpr int kBarSchedEmpty = kBarSchedFull + kSchedSlots;  // [kSchedSlots]
    static constexpr int kNumBars = kBarSchedEmpty + kSchedSlots;
    // Readers of a unit record: the two issuers and the eight softmax warps.
    static constexpr int kSchedReaders = 2 + 8;
    static constexpr int kOffSched = (kOffBar + kNumBars * 8 + 63) / 64 * 64;
    static constexpr int kOffMisc = kOffSched + 64 * kSchedSlots;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA exceeded");
    // warpgroup 0: producer (warp 0), MMA (warp 1), two idle warps; then one
    // softmax warpgroup per query tile
    static constexpr int kThreads = 128 + kNumQ * 128;
    // hd 128 launches 384 threads at 168 registers (64512 in all); the split
    // below gives 128 x 80 + 256 x 208 = 63488 <= 64512.  (72 / 216 left
    // the control warps, which also run the unit queue, short: 2.5% slower.)
    static constexpr uint32_t kRegsControl = 80;
    static constexpr uint32_t kRegsSoftmax = 208;
    static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= 384 * 168, "register split");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kKvTile, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
    // TMEM columns: the two tiles' S buffers, then their O accumulators
    __device__ static constexpr uint32_t s_col(int tile) { return (uint32_t)tile * 128u; }
    __device__ static constexpr uint32_t o_col(int tile) { return 256u + (uint32_t)tile * 128u; }
};

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

// Bulk prefetch of one tensor-map box into L2 (no shared memory, no barrier).
__device__ __forceinline__ void l2_prefetch_3d(const void *tmap, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 :: "l"(tmap), "r"(c0), "r"(c1), "r"(c2) : "memory");
}

// Ring order of a unit's K and V tiles when one issuer's QKs run two tiles
// ahead of its PVs (the CTA-pair kernel): K_0 K_1, then V_j followed by
// K_{j+2} -- the order the issuer consumes them, so a ring of a few items
// always holds the next loads.  (The two-tile kernel uses K_0 V_0 K_1 V_1 ...)
__device__ __forceinline__ int ring_pos_v(int j, int n) {
    return min(2, n) + j + min(j, max(0, n - 2));
}
__device__ __forceinline__ int ring_pos_k(int j, int n) {
    return j < 2 ? j : ring_pos_v(j - 2, n) + 1;
}

struct Seq {
    int q0, k0, Lq, Lk;
    bool ok;
};

__device__ __forceinline__ Seq load_seq(const PrefillParams &p, int i) {
    Seq s;
    s.q0 = __ldg(p.cu_q + i);
    s.k0 = __ldg(p.cu_k + i);
    const int q1 = __ldg(p.cu_q + i + 1);
    const int k1 = __ldg(p.cu_k + i + 1);
    s.ok = s.q0 >= 0 && s.k0 >= 0 && q1 >= s.q0 && k1 >= s.k0 && q1 <= p.total_q && k1 <= p.total_k;
    s.Lq = s.ok ? q1 - s.q0 : 0;
    s.Lk = s.ok ? k1 - s.k0 : 0;
    return s;
}

// Keys a query tile sees: [0, kv_limit); the last row decides for causal.
__device__ __forceinline__ int tile_kv_limit(const PrefillParams &p, const Seq &s, int t) {
    if (t * kQTile >= s.Lq) return 0;
    if (!p.causal) return s.Lk;
    const int q_last = min(s.Lq, (t + 1) * kQTile) - 1;
    return max(0, min(s.Lk, q_last + s.Lk - s.Lq + 1));
}

__device__ __forceinline__ int tile_kv_tiles(const PrefillParams &p, const Seq &s, int t) {
    return ceil_div_i(tile_kv_limit(p, s, t), kKvTile);
}

// One unit of work: (sequence, head, pair of query tiles 2*pair and 2*pair+1).
// 64 bytes, 16-aligned: a unit record is copied whole into the queues, the
// partner CTA's in four 16-byte stores.
struct alignas(16) PUnit {
    int seq, h, g;
    Seq s;
    int tile[2];       // query tile index, -1 if absent
    int nkv[2];        // KV tiles each query tile walks
    int nmax;
    int pad_[3];
};
static_assert(sizeof(PUnit) == 64, "a unit record fills one 64-byte slot");

__device__ __forceinline__ void decode_entry(const PrefillParams &p, int e, PUnit &u, int num_q) {
    const int32_t *PP = p.plan + 2;
    const int gp = e / p.Hq;
    u.h = e - gp * p.Hq;
    u.g = u.h / p.G;
    int lo = 0, hi = p.B - 1;                          // largest seq with PP[seq] <= gp
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(PP + mid) <= gp) lo = mid; else hi = mid - 1;
    }
    u.seq = lo;
    u.s = load_seq(p, lo);
    const int pair = gp - __ldg(PP + lo);
    const int nqt = ceil_div_i(u.s.Lq, kQTile);
    u.nmax = 0;
    for (int x = 0; x < 2; ++x) {
        const int t = num_q == 2 ? 2 * pair + x : (x == 0 ? pair : -1);
        u.tile[x] = (t >= 0 && t < nqt) ? t : -1;
        u.nkv[x] = u.tile[x] >= 0 ? tile_kv_tiles(p, u.s, t) : 0;
        u.nmax = max(u.nmax, u.nkv[x]);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <bool kOnline>
__global__ void __launch_bounds__(PrefillCfg::kThreads, 1)
varlen_prefill_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    using C = PrefillCfg;
    constexpr int D = C::D;
    constexpr int NQ = C::kNumQ;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sRing = smem + C::kOffRing;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *slot_full = bars + C::kBarSlotFull;
    uint64_t *slot_empty = bars + C::kBarSlotEmpty;
    uint64_t *q_full = bars + C::kBarQFull;
    uint64_t *q_empty = bars + C::kBarQEmpty;
    uint64_t *s_full = bars + C::kBarSFull;
    uint64_t *p_full = bars + C::kBarPFull;
    uint64_t *pv_done = bars + C::kBarPvDone;
    uint64_t *drain = bars + C::kBarDrain;
    uint64_t *issued = bars + C::kBarIssued;         // step handoff between the two issuers
    uint64_t *p_half = bars + C::kBarPHalf;          // first half of P (keys 0..63) written
    uint64_t *pvh_done = bars + C::kBarPvhDone;      // the PV of that half complete
    uint64_t *sched_full = bars + C::kBarSchedFull;  // unit record k written by the producer
    uint64_t *sched_empty = bars + C::kBarSchedEmpty;  // unit record k read by every role
    PUnit *sched = reinterpret_cast<PUnit *>(smem + C::kOffSched);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kSlots; ++i) { mbar_init(&slot_full[i], 1); mbar_init(&slot_empty[i], NQ); }
        mbar_init(q_full, 1);
        mbar_init(q_empty, NQ);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1); mbar_init(&p_full[i], 4); mbar_init(&pv_done[i], 1); mbar_init(&drain[i], 1);
            mbar_init(&issued[i], 1);
            mbar_init(&p_half[i], 4); mbar_init(&pvh_done[i], 1);
        }
        for (int i = 0; i < C::kSchedSlots; ++i) {
            mbar_init(&sched_full[i], 1); mbar_init(&sched_empty[i], C::kSchedReaders);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) { tmem_alloc(tmem_slot, C::kTmemCols); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();                                    // the plan of this call is written
    const int count = p.plan[0];                   // (read only after the wait)
    const WaitCtx wc{p.status, p.timeout_ns, abort_flag};
    // Units are handed out in list order (longest first) to whichever CTA
    // frees up: the producer takes the next entry from the call's counter
    // and publishes the decoded unit in shared memory for the other roles,
    // who so never walk the list themselves.  A record with seq < 0 ends
    // the CTA's work.  (A static snake over the list left CTAs finishing
    // 2.06-2.23 ms apart on the varlen workload.)
    // Readers copy the fields they use out of record k, then free it.
    auto wait_unit = [&](int k) -> const PUnit * {
        const int sl = k % C::kSchedSlots;
        return mbar_wait(&sched_full[sl], (k / C::kSchedSlots) & 1, wc) ? &sched[sl] : nullptr;
    };
    auto free_unit = [&](int k) { mbar_arrive(&sched_empty[k % C::kSchedSlots]); };

    if (warp < 4) {
      setmaxnreg_dec<C::kRegsControl>();
      if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t rp = 0, nu = 0, issued = 0;
            bool ok = true;
            for (int k = 0; ok; ++k, ++nu) {
                const int idx = atomicAdd(p.plan + 3 + p.B, 1);      // the call's next entry
                PUnit u;
                if (idx < count) decode_entry(p, __ldg(p.list + idx), u, NQ);
                else u.seq = -1;
                {
                    const int sl = k % C::kSchedSlots;
                    if (!mbar_wait(&sched_empty[sl], ((k / C::kSchedSlots) & 1) ^ 1, wc)) break;
                    sched[sl] = u;
                    mbar_arrive(&sched_full[sl]);          // release: the record is visible to its readers
                }
                if (u.seq < 0) break;
                if (!mbar_wait(q_empty, (nu & 1) ^ 1, wc)) break;
                uint32_t bytes = 0;
                for (int x = 0; x < NQ; ++x) if (u.tile[x] >= 0) bytes += C::kTileBytes;
                mbar_arrive_expect_tx(q_full, bytes);
                for (int x = 0; x < NQ; ++x) {
                    if (u.tile[x] < 0) continue;
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(smem_u32(sQ + x * C::kTileBytes + c * C::kChunkBytes), &tm_q, q_full,
                                    c * 64, u.h, u.s.q0 + u.tile[x] * kQTile);
                }
                // K_j and V_j of the unit, in that order, through the slot ring.
                for (int j = 0; j < u.nmax && ok; ++j) {
                    for (int kv = 0; kv < 2 && ok; ++kv, ++rp) {
                        const int sl = rp % C::kSlots;
                        ok = mbar_wait(&slot_empty[sl], ((rp / C::kSlots) & 1) ^ 1, wc);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&slot_full[sl], C::kTileBytes);
#pragma unroll
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_3d(smem_u32(sRing + sl * C::kSlotBytes + c * C::kChunkBytes),
                                        kv == 0 ? (const void *)&tm_k : (const void *)&tm_v, &slot_full[sl],
                                        c * 64, u.g, u.s.k0 + j * kKvTile);
                        issued = rp + 1;
                    }
                }
            }
            for (uint32_t k = 0; k < (uint32_t)C::kSlots && k < issued; ++k) {
                const uint32_t r = issued - 1 - k;
                mbar_wait_drain(&slot_full[r % C::kSlots], (r / C::kSlots) & 1, wc);
            }
        }
        __syncwarp();
      } else if (warp == 1 || warp == 2) {
        // ----------------------------------------------------------------- MMA
        // One issuing thread per query tile, so neither tile's MMAs queue
        // behind the other's issue: warp 1 drives tile 0, warp 2 tile 1.
        if (lane == 0) {
            const int x = warp - 1;
            uint32_t rp = 0, nu = 0, qk_cnt = 0, pv_cnt = 0;
            auto wait_slot = [&](uint32_t r) {
                return mbar_wait(&slot_full[r % C::kSlots], (r / C::kSlots) & 1, wc);
            };
            // Pushes only: a thread's tcgen05.mma issue advances at the tensor
            // core's pace, and any wait between pushes lets the pipe drain, so
            // each step waits for everything first and commits afterwards.
            auto wait_tile = [&](uint32_t r) { return wait_slot(r); };
            auto release_tile = [&](uint32_t r) { mma_commit(&slot_empty[r % C::kSlots]); };
            // Descriptors at the tile bases; the loops add compile-time offsets
            // (one integer add per operand: at N = 128 an MMA takes 64 cycles,
            // too few to rebuild two descriptors in the issuing thread).
            const SDesc q_k = sdesc_sw128_split(smem_u32(sQ + x * C::kTileBytes), 16, 1024);
            const SDesc ring_k = sdesc_sw128_split(smem_u32(sRing), 16, 1024);
            const SDesc ring_v = sdesc_sw128_split(smem_u32(sRing), C::kChunkBytes, 1024);
            auto push_qk = [&](uint32_t r_k) {
                const uint32_t sc = C::s_col(x);
                const SDesc kd{ring_k.lo + (r_k % C::kSlots) * (C::kSlotBytes >> 4), ring_k.hi};
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = sdesc_at(q_k, (kk >> 2) * C::kChunkBytes + (kk & 3) * 32);
                    const uint64_t b = sdesc_at(kd, (kk >> 2) * C::kChunkBytes + (kk & 3) * 32);
                    mma_bf16_ss(tmem + sc, a, b, C::kIdescQK, kk > 0 ? 1u : 0u);
                }
            };
            auto commit_qk = [&]() {
                mma_commit(&s_full[x]);
                ++qk_cnt;
            };
            // P was written over the first 64 columns of this tile's S buffer
            // (two BF16 per 32-bit column): A operand straight from TMEM.  The
            // softmax hands it over in two halves of 64 keys, and each half's
            // four MMAs go out as soon as it is there.
            auto push_pv_half = [&](uint32_t r_v, int half, bool first) {
                const uint32_t p_col = C::s_col(x);
                const SDesc vd{ring_v.lo + (r_v % C::kSlots) * (C::kSlotBytes >> 4), ring_v.hi};
#pragma unroll
                for (int k4 = 0; k4 < kKvTile / 32; ++k4) {
                    const int kk = half * (kKvTile / 32) + k4;
                    const uint64_t b = sdesc_at(vd, kk * 16 * 128);
                    mma_bf16_ts(tmem + C::o_col(x), tmem + p_col + kk * 8, b, C::kIdescPV,
                                (first && kk == 0) ? 0u : 1u);
                }
            };
            // pv_done completes once per unit, after the tile's last PV (the
            // epilogue's wait): within the unit, S_{j+1} landing already
            // implies PV_j complete (the same thread's earlier MMAs).
            auto commit_pv = [&](bool last) {
                if (last) mma_commit(&pv_done[x]);
                ++pv_cnt;
            };
            // Each issuing thread releases every ring position of the unit
            // exactly once (slot_empty counts one arrival per issuer): after its
            // last MMA reading the slot, or -- for a KV tile this query tile
            // does not reach -- once the load has landed, so that no release
            // can run a full ring ahead of the producer.
            auto release_unused = [&](uint32_t r) -> bool {
                if (!wait_tile(r)) return false;
                release_tile(r);
                return true;
            };
            // Alternation (two issuers): step j of tile 1 starts once tile 0 has
            // pushed the PV of its step j, and step j of tile 0 once tile 1 has
            // pushed the PV of its step j-1, so the tensor core runs the tiles'
            // PV+QK groups in turns while the other tile's softmax works -- the
            // two-group ping-pong.  The skew between the issuers stays within
            // one step, so each waits on at most the newest phase of the other's
            // `issued` barrier.
            uint32_t other = 0;                            // steps the other tile issued so far
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const PUnit *ur = wait_unit(k);
                const bool got = ur && ur->seq >= 0;
                const int nmax = got ? ur->nmax : 0;
                const int n = got ? ur->nkv[x] : 0;
                const int n_other = got ? ur->nkv[1 - x] : 0;
                free_unit(k);
                if (!got) break;
                if (!mbar_wait(q_full, nu & 1, wc)) break;
                tc_fence_after();
                const uint32_t r0 = rp;                       // K_j at r0 + 2j, V_j at r0 + 2j + 1
                auto pos_k = [&](int j) { return r0 + 2u * (uint32_t)j; };
                auto pos_v = [&](int j) { return r0 + 2u * (uint32_t)j + 1u; };
                constexpr int step = 1;                       // QK_{j+1} goes out with PV_j
                // prologue: the first `step` QKs
                for (int j = 0; j < step && j < nmax && ok; ++j) {
                    const uint32_t rk = pos_k(j);
                    if (j < n) {
                        if (!wait_tile(rk)) { ok = false; break; }
                        tc_fence_after();
                        push_qk(rk);
                        commit_qk();
                        release_tile(rk);
                    } else {
                        ok = release_unused(rk);
                    }
                }
                for (int j = 0; j < nmax && ok; ++j) {
                    const int jn = j + step;
                    const uint32_t rv = pos_v(j);
                    const uint32_t rk = jn < nmax ? pos_k(jn) : 0u;
                    const bool mine = j < n, next_mine = jn < n;
                    if (mine) {
                        {
                            // tile 1 follows tile 0's step j; tile 0 follows tile 1's step j-1
                            const int dep = x == 1 ? j : j - 1;
                            if (dep >= 0 && dep < n_other && !mbar_wait(&issued[1 - x], (other + dep) & 1, wc)) {
                                ok = false; break;
                            }
                        }
                        // The ring holds K_{j+step} before V_j is released (its items
                        // need only older items consumed), so PV and QK go out back
                        // to back.
                        if (!wait_tile(rv) || (next_mine && !wait_tile(rk)) ||
                            !mbar_wait(&p_half[x], pv_cnt & 1u, wc)) {
                            ok = false; break;
                        }
                        tc_fence_after();
                        push_pv_half(rv, 0, j == 0);
                        mma_commit(&pvh_done[x]);       // read only by a late replay
                        if (!mbar_wait(&p_full[x], pv_cnt & 1u, wc)) { ok = false; break; }
                        tc_fence_after();
                        push_pv_half(rv, 1, false);
                        // Hand the turn over while this step's QK is still being
                        // pushed: the other issuer's waits then overlap that push,
                        // and its PV queues right behind it instead of after an
                        // empty pipe.
                        mbar_arrive(&issued[x]);
                        if (next_mine) push_qk(rk);
                        commit_pv(j == n - 1);
                        release_tile(rv);
                        if (next_mine) { commit_qk(); release_tile(rk); }
                    } else if (!release_unused(rv)) {
                        ok = false; break;
                    }
                    if (jn < nmax && !next_mine && !release_unused(rk)) { ok = false; break; }
                }
                if (!ok) break;
                other += n_other;
                rp = r0 + (uint32_t)(2 * nmax);
                mma_commit(q_empty);
                ++nu;
            }
            mma_commit(&drain[x]);
            mbar_wait_drain(&drain[x], 0, wc);
        }
        __syncwarp();
      }
    } else {
        setmaxnreg_inc<C::kRegsSoftmax>();
        // ------------------------------------------------- softmax / epilogue
        // Warpgroup x owns query tile x of each unit; thread = one query row.
        // A failed wait does not change the control flow (no block-level
        // barriers here; each warp arrives on its own), so aborts wind down
        // through the remaining bounded iterations.
        const int x = (warp - 4) >> 2;
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const bool scale_pos = p.scale_log2 >= 0.f;
        uint32_t s_cnt = 0, pv_units = 0;
        // Completion of the last PV of this tile's unit number i.
        auto wait_pv = [&](uint32_t i) {
            mbar_wait(&pv_done[x], i & 1u, wc);
            tc_fence_after();
        };
        // The softmax warps hold their unit's record until its epilogue, which
        // reads the output row from it (fewer registers across the tile loop).
        for (int k = 0;; ++k) {
            const PUnit *ur = wait_unit(k);
            const bool got = ur && ur->seq >= 0;
            const int tile = got ? ur->tile[x] : -1;
            if (tile < 0) {
                __syncwarp();
                if (lane == 0) free_unit(k);
                if (!got) break;
                continue;
            }
            const int Lq = ur->s.Lq, Lk = ur->s.Lk;
            const int nkv = ur->nkv[x];
            const int q_row = tile * kQTile + row;               // row within the sequence
            const bool row_valid = q_row < Lq;
            const int lim = !p.causal ? Lk : max(0, min(Lk, q_row + Lk - Lq + 1));
            float m_ref = kNegInf, l_sum = 0.f;
            for (int j = 0; j < nkv; ++j, ++s_cnt) {
                mbar_wait(&s_full[x], s_cnt & 1u, wc);
                tc_fence_after();
                const uint32_t sa = tmem + lane_off + C::s_col(x);
                const int key0 = j * kKvTile;
                // The whole row of S in registers with one TMEM round trip.
                // Masked keys (past the causal limit or the sequence end) get the
                // value that exponentiates to 0 for this scale's sign.
                float sv[kKvTile];
                auto load_s = [&]() {
#pragma unroll
                    for (int c = 0; c < kKvTile / 32; ++c) tmem_ld32(sa + c * 32, sv + c * 32);
                    tmem_wait_ld();
                    if (key0 + kKvTile > lim) {
#pragma unroll
                        for (int i = 0; i < kKvTile; ++i)
                            if (key0 + i >= lim) sv[i] = scale_pos ? kNegInf : -kNegInf;
                    }
                };
                load_s();
                // Scaled row max of keys [lo, 128) of this tile (-inf when every
                // one is masked), 8 independent chains over the raw scores.
                auto row_max = [&](int lo) -> float {
                    float e8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) e8[i] = sv[lo + i];
                    if (scale_pos) {
#pragma unroll
                        for (int i = lo + 8; i < kKvTile; ++i) e8[i & 7] = fmaxf(e8[i & 7], sv[i]);
                    } else {
#pragma unroll
                        for (int i = lo + 8; i < kKvTile; ++i) e8[i & 7] = fminf(e8[i & 7], sv[i]);
                    }
                    const float ext = scale_pos
                        ? fmaxf(fmaxf(fmaxf(e8[0], e8[1]), fmaxf(e8[2], e8[3])), fmaxf(fmaxf(e8[4], e8[5]), fmaxf(e8[6], e8[7])))
                        : fminf(fminf(fminf(e8[0], e8[1]), fminf(e8[2], e8[3])), fminf(fminf(e8[4], e8[5]), fminf(e8[6], e8[7])));
                    return (ext == kNegInf || ext == -kNegInf) ? kNegInf : ext * p.scale_log2;
                };
                // P = 2^(s * scale * log2(e) - anchor) as BF16, packed two per
                // 32-bit register, for keys [64h, 64h + 64); returns their sum
                // (8 independent chains).  Each score dies as its probability is
                // formed, so the rows of S and P never both sit in registers in
                // full.
                uint32_t pk[kKvTile / 2];
                auto exp_half = [&](int h, float anchor) -> float {
                    const float mu = (anchor == kNegInf) ? 0.f : anchor;
                    float a8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) a8[i] = 0.f;
#pragma unroll
                    for (int i = 0; i < kKvTile / 2; i += 2) {
                        const int k = h * (kKvTile / 2) + i;
                        const float p0 = ex2_approx(fmaf(sv[k], p.scale_log2, -mu));
                        const float p1 = ex2_approx(fmaf(sv[k + 1], p.scale_log2, -mu));
                        a8[(i >> 1) & 7] += p0 + p1;
                        pk[k >> 1] = pack_bf16x2(p0, p1);
                    }
                    return ((a8[0] + a8[1]) + (a8[2] + a8[3])) + ((a8[4] + a8[5]) + (a8[6] + a8[7]));
                };
                // Half h of P over columns [32h, 32h + 32) of this tile's S
                // buffer, then handed to the MMA warp: p_half releases the PV of
                // keys 0..63 while the exponent pass of keys 64..127 runs, p_full
                // the rest (warp-collective TMEM stores).  P overwrites the
                // tile's only S buffer, which PV_{j-1} reads: that PV has landed,
                // since the same thread issued it before QK_j, whose completion
                // s_full reported.
                auto publish_half = [&](int h, bool store) {
                    if (store) {
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            tmem_st16u(sa + h * 32 + c * 16,
                                       *reinterpret_cast<const uint32_t(*)[16]>(pk + h * 32 + c * 16));
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(h == 0 ? &p_half[x] : &p_full[x]);
                };
                // Static anchor ("Flywheel Attention", section 3.1 and appendix
                // A): a row's anchor is the max of the first tile in which it sees
                // a key and does not move on the fast path, so the exponent pass
                // needs no running max.
                // O *= alpha for this thread's row (warp-collective TMEM
                // access; the caller makes sure no PV into O is in flight).
                auto rescale_o = [&](float alpha) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        const uint32_t oa = tmem + lane_off + C::o_col(x) + c * 32;
                        tmem_ld32(oa, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(oa, o);
                    }
                    tmem_wait_st();
                };
                // Slow path of the static anchor: half h of a tile whose check
                // failed in some row (warp-collective).  It works straight from
                // TMEM, 32 columns at a time in rolled loops, so that the hot
                // path carries neither its code nor its registers.  Rows with
                // `over` move their anchor to the max of the scores still in
                // TMEM (keys [64h, 128): the first half's P has overwritten keys
                // 0..63 once published), l is rescaled -- and for h = 1 also the
                // first half's sum t0, whose P already went to the MMA -- O is
                // rescaled (for h = 1 once that half's PV has landed), and P of
                // keys [64h, 64h + 64) is recomputed and written over columns
                // [32h, 32h + 32).  Returns the half's new sum.
                auto replay_half = [&](int h, bool over, bool rescale, float &t0) -> float {
                    float ext = scale_pos ? kNegInf : -kNegInf;
#pragma unroll 1
                    for (int c = 2 * h; c < 4; ++c) {
                        float v[32];
                        tmem_ld32(sa + c * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (key0 + c * 32 + i < lim) ext = scale_pos ? fmaxf(ext, v[i]) : fminf(ext, v[i]);
                    }
                    const float m_tile = (ext == kNegInf || ext == -kNegInf) ? kNegInf : ext * p.scale_log2;
                    float alpha = 1.f;
                    if (over) {
                        const float m_new = fmaxf(m_ref, m_tile);
                        alpha = ex2_approx(m_ref - m_new);
                        l_sum *= alpha;
                        if (h == 1) t0 *= alpha;
                        m_ref = m_new;
                    }
                    if (h == 1) {
                        mbar_wait(&pvh_done[x], s_cnt & 1u, wc);
                        tc_fence_after();
                    }
                    if (rescale) {
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            float o[32];
                            const uint32_t oa = tmem + lane_off + C::o_col(x) + c * 32;
                            tmem_ld32(oa, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= alpha;
                            tmem_st32(oa, o);
                        }
                        tmem_wait_st();
                    }
                    const float mu = (m_ref == kNegInf) ? 0.f : m_ref;
                    float sum = 0.f;
#pragma unroll 1
                    for (int c = 2 * h; c < 2 * h + 2; ++c) {
                        float v[32];
                        uint32_t q[16];
                        tmem_ld32(sa + c * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const bool in0 = key0 + c * 32 + i < lim, in1 = key0 + c * 32 + i + 1 < lim;
                            const float p0 = in0 ? ex2_approx(fmaf(v[i], p.scale_log2, -mu)) : 0.f;
                            const float p1 = in1 ? ex2_approx(fmaf(v[i + 1], p.scale_log2, -mu)) : 0.f;
                            sum += p0 + p1;
                            q[i >> 1] = pack_bf16x2(p0, p1);
                        }
                        tmem_st16u(sa + c * 16, q);
                    }
                    return sum;
                };
                float tsum0, tsum1;
                if constexpr (kOnline) {
                    // Online softmax with a conditional rescale ("Flywheel
                    // Attention", section 1): the tile's row max is taken every
                    // tile, and the base moves to it (l and O rescaled) only when
                    // it rose more than kRescaleSlack above the base.  PV_{j-1}
                    // has landed, since S_j has.
                    const float m_tile = row_max(0);
                    const bool up = m_tile > m_ref + kRescaleSlack;
                    if (__any_sync(0xffffffffu, up)) {
                        float alpha = 1.f;
                        if (up) {
                            alpha = ex2_approx(m_ref - m_tile);    // 0 while the row had no base
                            l_sum *= alpha;
                            m_ref = m_tile;
                        }
                        if (j > 0) rescale_o(alpha);
                    }
                    tsum0 = exp_half(0, m_ref);
                    publish_half(0, true);
                    tsum1 = exp_half(1, m_ref);
                    publish_half(1, true);
                } else {
                    if (m_ref == kNegInf) m_ref = row_max(0);
                    // The check, once per half before the MMA sees it: every p <=
                    // l, so a running sum within the budget proves no score rose
                    // more than log2(budget) above the anchor (appendix A, claim
                    // 2).  A row that fails (or overflowed) replays that half with
                    // the rescaling softmax (prefill_replay_half): its anchor
                    // moves to the new max, l and O are rescaled, P is recomputed.
                    tsum0 = exp_half(0, m_ref);
                    bool over = !(l_sum + tsum0 <= kAnchorBudget);
                    unsigned replay = __ballot_sync(0xffffffffu, over);
                    if (replay) {
                        // Nothing of this tile has reached the MMA, and PV_{j-1}
                        // has landed, since S_j has.
                        if (lane == 0) count_events(p.counters, kCounterPrefillReplays, __popc(replay));
                        tsum0 = replay_half(0, over, j > 0, tsum0);
                        publish_half(0, false);
                    } else {
                        publish_half(0, true);
                    }
                    tsum1 = exp_half(1, m_ref);
                    over = !(l_sum + tsum0 + tsum1 <= kAnchorBudget);
                    replay = __ballot_sync(0xffffffffu, over);
                    if (replay) {
                        // The first half went out with the old anchor: it is
                        // rescaled in O once its PV has landed (pvh_done).
                        if (lane == 0) count_events(p.counters, kCounterPrefillReplays, __popc(replay));
                        tsum1 = replay_half(1, over, true, tsum0);
                        publish_half(1, false);
                    } else {
                        publish_half(1, true);
                    }
                }
                l_sum += tsum0 + tsum1;
            }
            // ------------------------------------------------------ epilogue
            const int q0 = sched[k % C::kSchedSlots].s.q0, head = sched[k % C::kSchedSlots].h;
            __syncwarp();
            if (lane == 0) free_unit(k);
            __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                  (int64_t)(q0 + q_row) * p.out_stride[0] + (int64_t)head * p.out_stride[1];
            if (nkv > 0) {
                wait_pv(pv_units++);
                const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(tmem + lane_off + C::o_col(x) + c * 32, o);
                    tmem_wait_ld();
                    if (row_valid) {
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            uint4 v;
                            v.x = pack_bf16x2(o[8 * w + 0] * inv, o[8 * w + 1] * inv);
                            v.y = pack_bf16x2(o[8 * w + 2] * inv, o[8 * w + 3] * inv);
                            v.z = pack_bf16x2(o[8 * w + 4] * inv, o[8 * w + 5] * inv);
                            v.w = pack_bf16x2(o[8 * w + 6] * inv, o[8 * w + 7] * inv);
                            *reinterpret_cast<uint4 *>(orow + c * 32 + w * 8) = v;
                        }
                    }
                }
                tc_fence_before();
            } else if (row_valid) {
                for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4 *>(orow)[c] = make_uint4(0, 0, 0, 0);
            }
            if (row_valid && p.lse)
                p.lse[(int64_t)(q0 + q_row) * p.lse_stride[0] + (int64_t)head * p.lse_stride[1]] =
                    l_sum > 0.f ? (m_ref + __log2f(l_sum)) * 0.69314718055994531f : kNegInf;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// ------------------------------------------------- head dim 256, CTA pairs
//
// A cluster of two CTAs runs one unit of two consecutive 128-row query tiles
// (tile 2u in CTA 0, tile 2u+1 in CTA 1) with tcgen05.mma.cta_group::2,
// issued by CTA 0 for both:
//   S [256 x 128]  = Q [256 x 256] * K_tile^T      M = 256 rows, N = 128 keys
//   O [256 x 256] += P [256 x 128] * V_tile        M = 256 rows, N = 256 columns
// Each CTA holds its own query tile (A) and its TMEM holds its own 128 rows
// of S and O; the B operands are split between the pair: CTA r loads keys
// [64r, 64r + 64) of each K tile and value columns [128r, 128r + 128) of each
// V tile.  Every SM so moves 64 KiB of K/V per 128-key step instead of 128
// KiB, which is what a one-tile CTA at head dim 256 was bound by.
//
// Synchronisation across the pair: both CTAs' copies complete on CTA 0's
// barriers (slot_full, q_full); CTA 0's commits arrive on both CTAs'
// barriers (multicast: slot_empty, q_empty, s_full, pv_done); CTA 0's four
// softmax warps and one thread of CTA 1 (after its warps meet) arrive on CTA
// 0's p_full.

constexpr int kPairSlots = 5;
constexpr int kPairSlotBytes = 32768;          // half a K tile (64 x 256) or half a V tile (128 x 128)
constexpr int kPairQBytes = 128 * 256 * 2;
constexpr int kPairOffRing = kPairQBytes;
constexpr int kPairOffBar = kPairOffRing + kPairSlots * kPairSlotBytes;
// mbarrier array of the pair kernel, as above
constexpr int kPairBarSlotFull = 0;                            // [kPairSlots]
constexpr int kPairBarSlotEmpty = kPairBarSlotFull + kPairSlots;  // [kPairSlots]
constexpr int kPairBarQFull = kPairBarSlotEmpty + kPairSlots;  // [1]
constexpr int kPairBarQEmpty = kPairBarQFull + 1;              // [1]
constexpr int kPairBarSFull = kPairBarQEmpty + 1;              // [2]
constexpr int kPairBarPFull = kPairBarSFull + 2;               // [2]
constexpr int kPairBarPvDone = kPairBarPFull + 2;              // [2]
constexpr int kPairBarDrain = kPairBarPvDone + 2;              // [1]
constexpr int kPairSchedSlots = 4;                             // unit records in flight
constexpr int kPairBarSchedFull = kPairBarDrain + 1;           // [kPairSchedSlots], each CTA's own
constexpr int kPairBarSchedEmpty = kPairBarSchedFull + kPairSchedSlots;  // [kPairSchedSlots], CTA 0's
constexpr int kPairNumBars = kPairBarSchedEmpty + kPairSchedSlots;
// Readers of a unit record that arrive on CTA 0's sched_empty: CTA 0's issuer
// and four softmax warps, CTA 1's producer and (one arrival for) its softmax
// warps.
constexpr int kPairSchedReaders = 1 + 4 + 1 + 1;
constexpr int kPairOffSched = (kPairOffBar + kPairNumBars * 8 + 63) / 64 * 64;   // 16-byte stores land here
constexpr int kPairOffMisc = kPairOffSched + 64 * kPairSchedSlots;
constexpr int kPairSmemBytes = kPairOffMisc + 16 + 1024;
static_assert(kPairSmemBytes <= 232448, "shared memory budget of one CTA exceeded");
constexpr uint32_t kPairIdescQK = idesc_bf16_f32(256, 128, false, false);
constexpr uint32_t kPairIdescPV = idesc_bf16_f32(256, 256, false, true);


template <bool kOnline>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
varlen_prefill_pair_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    constexpr int D = 256;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem;
    uint8_t *sRing = smem + kPairOffRing;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kPairOffBar);
    uint64_t *slot_full = bars + kPairBarSlotFull;       // CTA 0's count both CTAs' copies
    uint64_t *slot_empty = bars + kPairBarSlotEmpty;
    uint64_t *q_full = bars + kPairBarQFull;             // CTA 0's counts both Q tiles
    uint64_t *q_empty = bars + kPairBarQEmpty;
    uint64_t *s_full = bars + kPairBarSFull;
    uint64_t *p_full = bars + kPairBarPFull;             // CTA 0's: its 4 warps + one arrival of CTA 1
    uint64_t *pv_done = bars + kPairBarPvDone;
    uint64_t *drain = bars + kPairBarDrain;              // CTA 0's MMAs all complete
    uint64_t *sched_full = bars + kPairBarSchedFull;     // unit record k in this CTA
    uint64_t *sched_empty = bars + kPairBarSchedEmpty;   // CTA 0's: record k read in both CTAs
    PUnit *sched = reinterpret_cast<PUnit *>(smem + kPairOffSched);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kPairOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kPairOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPairSlots; ++i) { mbar_init(&slot_full[i], 1); mbar_init(&slot_empty[i], 1); }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < 2; ++i) { mbar_init(&s_full[i], 1); mbar_init(&p_full[i], 5); mbar_init(&pv_done[i], 1); }
        mbar_init(drain, 1);
        for (int i = 0; i < kPairSchedSlots; ++i) {
            mbar_init(&sched_full[i], 1); mbar_init(&sched_empty[i], kPairSchedReaders);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) { tmem_alloc_pair(tmem_slot, 512); tmem_relinquish_pair(); }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                                  // both CTAs' barriers exist before any remote use
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();                                    // the plan of this call is written
    const int count = p.plan[0];                   // (read only after the wait)
    const WaitCtx wc{p.status, p.timeout_ns, abort_flag};
    // Units are handed out in list order to whichever pair frees up: CTA 0's
    // producer takes the next entry from the call's counter, decodes it and
    // writes the unit record into both CTAs' queues; every other role of
    // the pair reads its own CTA's copy and frees it on CTA 0's barrier.  A
    // record with seq < 0 ends the pair's work.
    auto wait_unit = [&](int k) -> const PUnit * {
        const int sl = k % kPairSchedSlots;
        return mbar_wait_cluster(&sched_full[sl], (k / kPairSchedSlots) & 1, wc) ? &sched[sl] : nullptr;
    };
    auto free_unit = [&](int k) {
        const int sl = k % kPairSchedSlots;
        if (rank == 0) mbar_arrive(&sched_empty[sl]);
        else mbar_arrive_cluster(cluster_addr(&sched_empty[sl], 0));
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t q_full0 = cluster_addr(q_full, 0);
            uint32_t rp = 0, nu = 0;
            bool ok = true;
            for (int k = 0; ok; ++k, ++nu) {
                PUnit u;
                if (rank == 0) {
                    const int idx = atomicAdd(p.plan + 3 + p.B, 1);    // the call's next entry
                    if (idx < count) decode_entry(p, __ldg(p.list + idx), u, 2);
                    else u.seq = -1;
                    const int sl = k % kPairSchedSlots;
                    if (!mbar_wait_cluster(&sched_empty[sl], ((k / kPairSchedSlots) & 1) ^ 1, wc)) break;
                    sched[sl] = u;
                    const uint4 *w = reinterpret_cast<const uint4 *>(&u);
                    const uint32_t peer = cluster_addr(&sched[sl], 1);
#pragma unroll
                    for (int i = 0; i < (int)sizeof(PUnit) / 16; ++i)
                        st_cluster_v4(peer + 16u * i, w[i].x, w[i].y, w[i].z, w[i].w);
                    mbar_arrive(&sched_full[sl]);
                    mbar_arrive_cluster(cluster_addr(&sched_full[sl], 1));   // release: the copy is visible
                } else {
                    const PUnit *ur = wait_unit(k);
                    if (ur) u = *ur;
                    else u.seq = -1;
                    free_unit(k);
                }
                if (u.seq < 0) break;
                if (!mbar_wait(q_empty, (nu & 1) ^ 1, wc)) break;
                // A CTA whose tile does not exist loads its partner's rows
                // (finite values; its outputs are never written).
                const int tile = u.tile[rank] >= 0 ? u.tile[rank] : u.tile[0];
                if (rank == 0) mbar_arrive_expect_tx(q_full, 2u * kPairQBytes);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d_pair(smem_u32(sQ + c * 128 * 128), &tm_q, q_full0, c * 64, u.h,
                                     u.s.q0 + tile * kQTile);
                const int n = u.nmax;
                auto prefetch_tile = [&](int j) {
                    if (j >= n) return;
                    const int key = u.s.k0 + j * kKvTile;
                    for (int c = 0; c < D / 64; ++c) l2_prefetch_3d(&tm_k, c * 64, u.g, key + (int)rank * 64);
                    for (int c = 0; c < 2; ++c) l2_prefetch_3d(&tm_v, (int)rank * 128 + c * 64, u.g, key);
                };
                for (int j = 0; j < 2; ++j) prefetch_tile(j);
                // This CTA's half of K_j or V_j, as one ring item.
                auto load_half = [&](bool is_v, int j) {
                    const int sl = rp % kPairSlots;
                    ok = mbar_wait(&slot_empty[sl], ((rp / kPairSlots) & 1) ^ 1, wc);
                    if (!ok) return;
                    if (rank == 0) mbar_arrive_expect_tx(&slot_full[sl], 2u * kPairSlotBytes);
                    const uint32_t full0 = cluster_addr(&slot_full[sl], 0);
                    const uint32_t dst = smem_u32(sRing + sl * kPairSlotBytes);
                    const int key = u.s.k0 + j * kKvTile;
                    if (!is_v) {
#pragma unroll
                        for (int c = 0; c < D / 64; ++c)          // 64 keys x 64 columns per box
                            tma_load_3d_pair(dst + c * 64 * 128, &tm_k, full0, c * 64, u.g, key + (int)rank * 64);
                    } else {
#pragma unroll
                        for (int c = 0; c < 2; ++c)                // 128 keys x 64 columns per box
                            tma_load_3d_pair(dst + c * 128 * 128, &tm_v, full0, (int)rank * 128 + c * 64, u.g, key);
                        prefetch_tile(j + 2);
                    }
                    ++rp;
                };
                for (int j = 0; j < 2 && j < n && ok; ++j) load_half(false, j);
                for (int j = 0; j < n && ok; ++j) {
                    load_half(true, j);
                    if (ok && j + 2 < n) load_half(false, j + 2);
                }
            }
            // CTA 0's slot_full / q_full phases complete only once both CTAs'
            // copies have landed; CTA 0 drains them below, before the pair's
            // final cluster barrier, so neither CTA leaves with a copy in flight.
            if (rank == 0) {
                for (uint32_t k = 0; k < (uint32_t)kPairSlots && k < rp; ++k) {
                    const uint32_t r = rp - 1 - k;
                    mbar_wait_drain(&slot_full[r % kPairSlots], (r / kPairSlots) & 1, wc);
                }
                if (nu > 0) mbar_wait_drain(q_full, (nu - 1) & 1, wc);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------- MMA (CTA 0 only)
        if (rank == 0 && lane == 0) {
            uint32_t rp = 0, nu = 0, qk_cnt = 0, pv_cnt = 0;
            // Descriptors at the tile bases, stepped by compile-time offsets.
            const SDesc q_k = sdesc_sw128_split(smem_u32(sQ), 16, 1024);
            const SDesc ring_k = sdesc_sw128_split(smem_u32(sRing), 16, 1024);
            const SDesc ring_v = sdesc_sw128_split(smem_u32(sRing), 128 * 128, 1024);
            auto wait_slot = [&](uint32_t r) {
                return mbar_wait(&slot_full[r % kPairSlots], (r / kPairSlots) & 1, wc);
            };
            auto push_qk = [&](uint32_t r_k) {
                const uint32_t sc = (qk_cnt & 1u) * 128u;
                const SDesc kd{ring_k.lo + (r_k % kPairSlots) * (kPairSlotBytes >> 4), ring_k.hi};
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = sdesc_at(q_k, (kk >> 2) * 128 * 128 + (kk & 3) * 32);
                    const uint64_t b = sdesc_at(kd, (kk >> 2) * 64 * 128 + (kk & 3) * 32);
                    mma_pair_ss(tmem + sc, a, b, kPairIdescQK, kk > 0 ? 1u : 0u);
                }
            };
            auto commit_qk = [&]() { mma_commit_pair(&s_full[qk_cnt & 1u]); ++qk_cnt; };
            // P sits over the first 64 columns of the tile's S buffer, two BF16
            // per column, in each CTA's TMEM.
            auto push_pv = [&](uint32_t r_v, bool first) {
                const uint32_t p_col = (pv_cnt & 1u) * 128u;
                const SDesc vd{ring_v.lo + (r_v % kPairSlots) * (kPairSlotBytes >> 4), ring_v.hi};
#pragma unroll
                for (int kk = 0; kk < kKvTile / 16; ++kk) {
                    const uint64_t b = sdesc_at(vd, kk * 16 * 128);
                    mma_pair_ts(tmem + 256u, tmem + p_col + kk * 8, b, kPairIdescPV, (first && kk == 0) ? 0u : 1u);
                }
            };
            auto commit_pv = [&]() { mma_commit_pair(&pv_done[pv_cnt & 1u]); ++pv_cnt; };
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const PUnit *ur = wait_unit(k);
                const bool got = ur && ur->seq >= 0;
                const int n = got ? ur->nmax : 0;
                free_unit(k);
                if (!got) break;
                if (!mbar_wait(q_full, nu & 1, wc)) break;
                tc_fence_after();
                const uint32_t r0 = rp;
                auto pos_k = [&](int j) { return r0 + (uint32_t)ring_pos_k(j, n); };
                auto pos_v = [&](int j) { return r0 + (uint32_t)ring_pos_v(j, n); };
                for (int j = 0; j < 2 && j < n && ok; ++j) {
                    const uint32_t rk = pos_k(j);
                    if (!wait_slot(rk)) { ok = false; break; }
                    tc_fence_after();
                    push_qk(rk);
                    commit_qk();
                    mma_commit_pair(&slot_empty[rk % kPairSlots]);
                }
                for (int j = 0; j < n && ok; ++j) {
                    const bool next = j + 2 < n;
                    const uint32_t rv = pos_v(j);
                    const uint32_t rk = next ? pos_k(j + 2) : 0u;
                    if (!wait_slot(rv) || (next && !wait_slot(rk)) ||
                        !mbar_wait_cluster(&p_full[pv_cnt & 1u], (pv_cnt >> 1) & 1u, wc)) {
                        ok = false; break;
                    }
                    tc_fence_after();
                    push_pv(rv, j == 0);
                    if (next) push_qk(rk);
                    commit_pv();
                    mma_commit_pair(&slot_empty[rv % kPairSlots]);
                    if (next) { commit_qk(); mma_commit_pair(&slot_empty[rk % kPairSlots]); }
                }
                if (!ok) break;
                rp = r0 + (uint32_t)(2 * n);
                mma_commit_pair(q_empty);
                ++nu;
            }
            // No MMA of the pair may still run when the pair frees TMEM.
            mma_commit_pair(drain);
            mbar_wait_drain(drain, 0, wc);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------- softmax / epilogue
        // Thread = one row of this CTA's query tile.  Every unit walks the
        // pair's KV tiles; a tile past this CTA's causal reach is fully masked
        // (zero probabilities).  A CTA whose tile does not exist still takes
        // part (its P gates CTA 0's PV) and writes nothing.
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const bool scale_pos = p.scale_log2 >= 0.f;
        uint32_t s_cnt = 0, pv_cnt = 0;
        auto wait_pv = [&](uint32_t i) {
            mbar_wait(&pv_done[i & 1u], (i >> 1) & 1u, wc);
            tc_fence_after();
        };
        for (int k = 0;; ++k) {
            const PUnit *ur = wait_unit(k);
            bool got = ur && ur->seq >= 0;
            const int tile0 = got ? ur->tile[0] : 0, tile_r = got ? ur->tile[rank] : -1;
            const int q0 = got ? ur->s.q0 : 0, Lq = got ? ur->s.Lq : 0, Lk = got ? ur->s.Lk : 0;
            const int head = got ? ur->h : 0;
            const int n = got ? ur->nmax : 0;
            // CTA 0's warps free the record one by one; CTA 1's meet first and
            // send one cluster-scope arrival.
            __syncwarp();
            if (rank == 0) {
                if (lane == 0) free_unit(k);
            } else {
                named_bar_sync(2, 128);
                if (warp == 4 && lane == 0) free_unit(k);
                // After an abort (some wait ran out) all four warps leave
                // together, so none is left alone at a named barrier.
                if (*abort_flag) got = false;
            }
            if (!got) break;
            const bool tile_ok = tile_r >= 0;
            const int q_row = (tile_ok ? tile_r : tile0) * kQTile + row;
            const bool row_valid = tile_ok && q_row < Lq;
            const int lim = !p.causal ? Lk : max(0, min(Lk, q_row + Lk - Lq + 1));
            float m_ref = kNegInf, l_sum = 0.f;
            for (int j = 0; j < n; ++j, ++s_cnt) {
                const uint32_t sb = s_cnt & 1u;
                mbar_wait(&s_full[sb], (s_cnt >> 1) & 1u, wc);
                tc_fence_after();
                const uint32_t sa = tmem + lane_off + sb * 128u;
                const int key0 = j * kKvTile;
                float sv[kKvTile];
                auto load_s = [&]() {
#pragma unroll
                    for (int c = 0; c < kKvTile / 32; ++c) tmem_ld32(sa + c * 32, sv + c * 32);
                    tmem_wait_ld();
                    if (key0 + kKvTile > lim) {
#pragma unroll
                        for (int i = 0; i < kKvTile; ++i)
                            if (key0 + i >= lim) sv[i] = scale_pos ? kNegInf : -kNegInf;
                    }
                };
                load_s();
                auto row_max = [&]() -> float {
                    float e8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) e8[i] = sv[i];
                    if (scale_pos) {
#pragma unroll
                        for (int i = 8; i < kKvTile; ++i) e8[i & 7] = fmaxf(e8[i & 7], sv[i]);
                    } else {
#pragma unroll
                        for (int i = 8; i < kKvTile; ++i) e8[i & 7] = fminf(e8[i & 7], sv[i]);
                    }
                    const float ext = scale_pos
                        ? fmaxf(fmaxf(fmaxf(e8[0], e8[1]), fmaxf(e8[2], e8[3])), fmaxf(fmaxf(e8[4], e8[5]), fmaxf(e8[6], e8[7])))
                        : fminf(fminf(fminf(e8[0], e8[1]), fminf(e8[2], e8[3])), fminf(fminf(e8[4], e8[5]), fminf(e8[6], e8[7])));
                    return (ext == kNegInf || ext == -kNegInf) ? kNegInf : ext * p.scale_log2;
                };
                uint32_t pk[kKvTile / 2];
                auto exp_pass = [&](float anchor) -> float {
                    const float mu = (anchor == kNegInf) ? 0.f : anchor;
                    float a8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) a8[i] = 0.f;
#pragma unroll
                    for (int i = 0; i < kKvTile; i += 2) {
                        const float p0 = ex2_approx(fmaf(sv[i], p.scale_log2, -mu));
                        const float p1 = ex2_approx(fmaf(sv[i + 1], p.scale_log2, -mu));
                        a8[(i >> 1) & 7] += p0 + p1;
                        pk[i >> 1] = pack_bf16x2(p0, p1);
                    }
                    return ((a8[0] + a8[1]) + (a8[2] + a8[3])) + ((a8[4] + a8[5]) + (a8[6] + a8[7]));
                };
                auto store_p = [&]() {
#pragma unroll
                    for (int c = 0; c < kKvTile / 32; ++c)
                        tmem_st16u(sa + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + c * 16));
                };
                // Static anchor and the running-sum check, as in the one-CTA
                // kernel; P(j) goes to S buffer j & 1, which PV(j-1) does not read.
                // O *= alpha for this thread's row, once PV(j-1) has landed
                // (warp-collective TMEM access).
                auto rescale_o = [&](float alpha) {
                    wait_pv(pv_cnt + j - 1);
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        const uint32_t oa = tmem + lane_off + 256u + c * 32;
                        tmem_ld32(oa, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(oa, o);
                    }
                    tmem_wait_st();
                };
                float tsum;
                if constexpr (kOnline) {
                    // Online softmax with a conditional rescale, as in the one-CTA kernel.
                    const float m_tile = row_max();
                    const bool up = m_tile > m_ref + kRescaleSlack;
                    if (__any_sync(0xffffffffu, up)) {
                        float alpha = 1.f;
                        if (up) {
                            alpha = ex2_approx(m_ref - m_tile);    // 0 while the row had no base
                            l_sum *= alpha;
                            m_ref = m_tile;
                        }
                        if (j > 0) rescale_o(alpha);
                    }
                    tsum = exp_pass(m_ref);
                } else {
                    if (m_ref == kNegInf) m_ref = row_max();
                    tsum = exp_pass(m_ref);
                    // The check: every p <= l, so a running sum within the budget
                    // proves no score rose more than log2(budget) above the anchor
                    // (appendix A, claim 2).  A row that fails (or overflowed)
                    // replays the tile with the rescaling softmax: its anchor moves
                    // to the new max, l and O are rescaled, P is recomputed before
                    // the MMA sees it.  The scores come back from TMEM, which P
                    // has not overwritten yet.
                    const bool over = !(l_sum + tsum <= kAnchorBudget);
                    const unsigned replay = __ballot_sync(0xffffffffu, over);
                    if (replay) {
                        if (lane == 0) count_events(p.counters, kCounterPrefillReplays, __popc(replay));
                        // The scores are read twice so that they are not held in
                        // registers across the O rescale.
                        load_s();
                        const float m_tile = row_max();
                        float alpha = 1.f;
                        if (over) {
                            const float m_new = fmaxf(m_ref, m_tile);
                            alpha = ex2_approx(m_ref - m_new);
                            l_sum *= alpha;
                            m_ref = m_new;
                        }
                        if (j > 0) rescale_o(alpha);
                        load_s();
                        tsum = exp_pass(m_ref);    // all lanes: unchanged rows recompute the same P
                    }
                }
                store_p();
                l_sum += tsum;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                // CTA 0's warps arrive on their own CTA's barrier; CTA 1's meet
                // first and send one cluster-scope arrival (each such release
                // costs the arriving thread a long fence: one per step, not
                // four; 0.387 -> 0.365 ms per call).
                if (rank == 0) {
                    if (lane == 0) mbar_arrive(&p_full[s_cnt & 1u]);
                } else {
                    named_bar_sync(1, 128);
                    if (warp == 4 && lane == 0) mbar_arrive_cluster(cluster_addr(&p_full[s_cnt & 1u], 0));
                }
            }
            // ------------------------------------------------------ epilogue
            __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                  (int64_t)(q0 + q_row) * p.out_stride[0] + (int64_t)head * p.out_stride[1];
            if (n > 0) {
                wait_pv(pv_cnt + n - 1);
                const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(tmem + lane_off + 256u + c * 32, o);
                    tmem_wait_ld();
                    if (row_valid) {
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            uint4 v;
                            v.x = pack_bf16x2(o[8 * w + 0] * inv, o[8 * w + 1] * inv);
                            v.y = pack_bf16x2(o[8 * w + 2] * inv, o[8 * w + 3] * inv);
                            v.z = pack_bf16x2(o[8 * w + 4] * inv, o[8 * w + 5] * inv);
                            v.w = pack_bf16x2(o[8 * w + 6] * inv, o[8 * w + 7] * inv);
                            *reinterpret_cast<uint4 *>(orow + c * 32 + w * 8) = v;
                        }
                    }
                }
                tc_fence_before();
            } else if (row_valid) {
                for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4 *>(orow)[c] = make_uint4(0, 0, 0, 0);
            }
            if (row_valid && p.lse)
                p.lse[(int64_t)(q0 + q_row) * p.lse_stride[0] + (int64_t)head * p.lse_stride[1]] =
                    l_sum > 0.f ? (m_ref + __log2f(l_sum)) * 0.69314718055994531f : kNegInf;
            pv_cnt += n;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                                  // no MMA, copy or remote arrive of the pair is left
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

// ------------------------------------------------------------------- plan
//
// One block.  PP[i] = exclusive prefix of the unit pairs per sequence; each
// (pair, head) entry goes into the list ordered by its KV-tile cost, largest
// first (counting sort): handed out in that order as CTAs (or CTA pairs)
// free up, it balances them.
// Sequences whose cumulative lengths reach past the packed tensors are left
// out and reported in the status word.
__global__ void __launch_bounds__(1024) prefill_plan_kernel(const __grid_constant__ PrefillParams p, int num_q) {
    pdl_launch_dependents();                         // the attention kernel waits for this grid to finish
    __shared__ int warp_sums[32];
    __shared__ int carry_s;
    __shared__ int bins[kCostBins];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t *PP = p.plan + 2;
    if (tid == 0) carry_s = 0;
    for (int i = tid; i < kCostBins; i += blockDim.x) bins[i] = 0;
    __syncthreads();
    for (int base = 0; base < p.B; base += 1024) {
        const int i = base + tid;
        int pairs = 0;
        if (i < p.B) {
            const Seq s = load_seq(p, i);
            if (!s.ok) record_error(p.status, 1);
            const int nqt = ceil_div_i(s.Lq, kQTile);
            pairs = num_q == 2 ? (nqt + 1) / 2 : nqt;
        }
        int incl = pairs;
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
            warp_sums[lane] = w;
        }
        __syncthreads();
        if (i < p.B) PP[i] = carry_s + (warp > 0 ? warp_sums[warp - 1] : 0) + incl - pairs;
        __syncthreads();
        if (tid == 0) carry_s += warp_sums[31];
        __syncthreads();
    }
    const int NP = carry_s;
    if (tid == 0) PP[p.B] = NP;
    __syncthreads();
    // cost of a pair: KV tiles of both of its query tiles
    auto pair_bin = [&](int gp, int &seq_out) {
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (PP[mid] <= gp) lo = mid; else hi = mid - 1;
        }
        seq_out = lo;
        const Seq s = load_seq(p, lo);
        const int pair = gp - PP[lo];
        int cost = 0;
        if (num_q == 2) {
            cost = tile_kv_tiles(p, s, 2 * pair) + tile_kv_tiles(p, s, 2 * pair + 1);
        } else {
            cost = 2 * tile_kv_tiles(p, s, pair);
        }
        return kCostBins - 1 - min(cost, kCostBins - 1);     // largest cost first
    };
    for (int gp = tid; gp < NP; gp += blockDim.x) {
        int sq;
        atomicAdd(&bins[pair_bin(gp, sq)], 1);
    }
    __syncthreads();
    {
        // Exclusive scan of the bins: each thread scans its run of
        // kCostBins / blockDim.x consecutive bins, then the run totals are
        // scanned across the block (warp shuffles + one warp over warp sums).
        constexpr int kPer = kCostBins / 1024;
        static_assert(kCostBins % 1024 == 0, "bins per thread");
        int run[kPer], tot = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) { run[i] = bins[tid * kPer + i]; tot += run[i]; }
        int incl = tot;
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
            warp_sums[lane] = w;
        }
        __syncthreads();
        int acc = (warp > 0 ? warp_sums[warp - 1] : 0) + incl - tot;
#pragma unroll
        for (int i = 0; i < kPer; ++i) { bins[tid * kPer + i] = acc; acc += run[i]; }
    }
    __syncthreads();
    for (int gp = tid; gp < NP; gp += blockDim.x) {
        int sq;
        const int pos = atomicAdd(&bins[pair_bin(gp, sq)], 1);
        if ((int64_t)(pos + 1) * p.Hq <= p.list_capacity)
            for (int h = 0; h < p.Hq; ++h) p.list[(int64_t)pos * p.Hq + h] = gp * p.Hq + h;
    }
    if (tid == 0) {
        p.plan[0] = (int64_t)NP * p.Hq <= p.list_capacity ? NP * p.Hq : 0;
        p.plan[1] = NP;
        p.plan[3 + p.B] = 0;                         // the attention kernel's next entry to hand out
        if ((int64_t)NP * p.Hq > p.list_capacity) record_error(p.status, 3);
    }
}

template <bool kOnline>
cudaError_t launch_tiles(const PrefillParams &p, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         cudaStream_t stream) {
    using C = PrefillCfg;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(varlen_prefill_kernel<kOnline>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    cudaError_t le = launch_after_previous(varlen_prefill_kernel<kOnline>, dim3(p.grid), dim3(C::kThreads),
                                           C::kSmemBytes, stream, p, tq, tk, tv);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

template <bool kOnline>
cudaError_t launch_pair(const PrefillParams &p, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        cudaStream_t stream) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(varlen_prefill_pair_kernel<kOnline>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    cudaError_t le = launch_after_previous(varlen_prefill_pair_kernel<kOnline>, dim3(p.grid & ~1), dim3(256),
                                           kPairSmemBytes, stream, p, tq, tk, tv);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                           const CUtensorMap &tv, int head_dim, cudaStream_t stream,
                           cudaEvent_t timing_start, cudaEvent_t timing_stop, int *launches) {
    *launches = 0;
    prefill_plan_kernel<<<1, 1024, 0, stream>>>(p, 2);           // units of two query tiles at both head dims
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ++*launches;
    if (timing_start) cudaEventRecord(timing_start, stream);
    if (head_dim == 128) e = p.online ? launch_tiles<true>(p, tq, tk, tv, stream) : launch_tiles<false>(p, tq, tk, tv, stream);
    else if (head_dim == 256) e = p.online ? launch_pair<true>(p, tq, tk, tv, stream) : launch_pair<false>(p, tq, tk, tv, stream);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    ++*launches;
    if (timing_stop) cudaEventRecord(timing_stop, stream);
    return cudaSuccess;
}

}  // namespace fw
