// Paged grouped-query decode over an FP8 E4M3 KV cache, sm_103a.
//
// "TokenSpeed-MLA 2.0.1" (decode): FP8 inputs, BF16 output.  The cache holds
// E4M3 bytes with one scale per cache (k = k_scale * e4m3, v = v_scale *
// e4m3); HBM traffic per key is half that of a BF16 cache, which is what a
// bandwidth-bound decode gains.  The arithmetic keeps 16-bit operands: every
// E4M3 value is exact in FP16, so converter warps widen the K and V tiles to
// FP16 next to the tensor core and the MMAs run kind::f16 with FP16 A and B
// (queries converted from BF16 once per unit, probabilities written as FP16);
// k_scale folds into the score scale, v_scale into the epilogue.
//
// Layout and schedule follow the BF16 decode kernel (swap-AB: S^T [128 keys x
// NQ] = K * Q^T, O^T [128 x NQ] += V^T * P^T; balanced tile ranges; split-KV
// pieces merged by the combine kernel).  Differences:
//   * warp 0 (TMA) loads 16 KiB FP8 tiles (128 keys x 128 bytes) into two
//     byte rings, one for K and one for V;
//   * warps 6-9 convert, one thread per key: the K row into TMEM as the A
//     operand of QK^T (thread = key = TMEM lane, 2 FP16 per column), the V
//     row into a swizzled FP16 tile in shared memory (the A operand of PV);
//     keys past the piece's end become zeros, so NaN bytes in unused slots
//     never meet the MMAs;
//   * warp 1 issues the MMAs (QK^T in TS form), warps 2-5 run the softmax
//     with the conditional rescale of the BF16 kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_common.cuh"
#include "fw_internal.h"
#include "fw_ptx.cuh"

namespace fw {

namespace {

using namespace dec;

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;   // log2 units: 2^(s - base) stays below 2^8
// Probabilities go to the MMA as FP16, whose normal range starts at 2^-14;
// they are taken relative to base - kHeadroom (at most 2^15, inside FP16's
// 65504) so that small ones keep their precision.  l carries the same factor,
// and the LSE subtracts it again.
constexpr float kHeadroom = 7.0f;
constexpr int D = 128;

// Instruction descriptor, kind::f16 with FP16 A/B and FP32 accumulation.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t M, uint32_t N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) | ((N >> 3) << 17) |
           ((M >> 4) << 24);
}

// Two E4M3 bytes (the lower address in the low byte) to two FP16 values
// (the lower address in the low half).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
    return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <int NQ>
struct Fp8Cfg {
    static constexpr int kStages8 = NQ == 16 ? 4 : 3;          // FP8 tiles in flight per ring
    static constexpr int kTile8Bytes = kKvTile * D;             // 128 keys x 128 bytes
    static constexpr int kChunkBytes = kKvTile * 128;           // 64 FP16 columns of a tile
    static constexpr int kTile16Bytes = 2 * kChunkBytes;
    static constexpr int kQBytes = NQ * D * 2;
    static constexpr int kPBytes = NQ * kKvTile * 2;
    // shared memory map (offsets from a 1024-aligned base)
    static constexpr int kOffK8 = 0;
    static constexpr int kOffV8 = kOffK8 + kStages8 * kTile8Bytes;
    static constexpr int kOffV16 = kOffV8 + kStages8 * kTile8Bytes;
    static constexpr int kOffQ = kOffV16 + 2 * kTile16Bytes;
    static constexpr int kOffP = kOffQ + 2 * kQBytes;
    static constexpr int kOffBar = kOffP + 2 * kPBytes;
    static constexpr int kNumBars = 4 * kStages8 + 2 * 2 + 2 * 2 + 2 + 2 + 2 + 2 + 2 + 1 + 1;
    static constexpr int kOffRedMax = kOffBar + kNumBars * 8;
    static constexpr int kOffRedSum = kOffRedMax + 2 * 4 * NQ * 4;
    static constexpr int kOffMisc = kOffRedSum + 4 * NQ * 4;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA exceeded");
    static_assert(kOffRedMax % 16 == 0, "row maxima are read as float4");
    // TMEM: two FP16 K tiles (64 columns each), two S^T buffers, O^T
    static constexpr uint32_t kColK = 0;
    static constexpr uint32_t kColS = 128;
    static constexpr uint32_t kColO = kColS + 2 * NQ;
    static constexpr uint32_t kTmemCols = 256;
    static constexpr uint32_t kIdescQK = idesc_f16_f32(128, NQ, false, false);
    static constexpr uint32_t kIdescPV = idesc_f16_f32(128, NQ, true, false);
};

// NQ: query rows on the MMA N axis (16 or 32); R: rows the softmax carries
// (8 when a unit holds at most 8 query rows, else NQ).
template <int NQ, int R>
__global__ void __launch_bounds__(320, 1)
paged_decode_fp8_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    using C = Fp8Cfg<NQ>;
    static_assert(R == 8 || R == NQ, "softmax rows");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sK8 = smem + C::kOffK8;
    uint8_t *sV8 = smem + C::kOffV8;
    uint8_t *sV16 = smem + C::kOffV16;
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sP = smem + C::kOffP;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *k8_full = bars;
    uint64_t *k8_empty = k8_full + C::kStages8;
    uint64_t *v8_full = k8_empty + C::kStages8;
    uint64_t *v8_empty = v8_full + C::kStages8;
    uint64_t *k16_full = v8_empty + C::kStages8;      // [2]
    // One commit per MMA group: qk_done[b] (QK of tile j, b = j & 1) frees
    // the FP16 K buffer b and publishes S buffer b; pv_done[b] (PV of tile j)
    // frees the FP16 V buffer and the P buffer b.  A commit costs the tensor
    // pipe about as much as an N = 16 MMA, so each event has one barrier,
    // waited on by every role that needs it.
    uint64_t *qk_done = k16_full + 2;                  // [2]
    uint64_t *v16_full = qk_done + 2;                  // [2]
    uint64_t *pv_done = v16_full + 2;                  // [2]
    uint64_t *q_full = pv_done + 2;                    // [2] BF16 Q landed
    uint64_t *q16 = q_full + 2;                        // [2] Q converted to FP16
    uint64_t *q_empty = q16 + 2;                       // [2]
    uint64_t *s_free = q_empty + 2;                    // [2]
    uint64_t *p_full = s_free + 2;                     // [2]
    uint64_t *drain = p_full + 2;                      // [1]
    float *red_max = reinterpret_cast<float *>(smem + C::kOffRedMax);   // [2][4][NQ]
    float *red_sum = reinterpret_cast<float *>(smem + C::kOffRedSum);   // [4][NQ]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages8; ++i) {
            mbar_init(&k8_full[i], 1); mbar_init(&k8_empty[i], 4);
            mbar_init(&v8_full[i], 1); mbar_init(&v8_empty[i], 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k16_full[i], 4); mbar_init(&qk_done[i], 1);
            mbar_init(&v16_full[i], 4); mbar_init(&pv_done[i], 1);
            mbar_init(&q_full[i], 1); mbar_init(&q16[i], 4); mbar_init(&q_empty[i], 1);
            mbar_init(&s_free[i], 4);
            mbar_init(&p_full[i], 4);
        }
        mbar_init(drain, 1);
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
    const WaitCtx wc{p.status, p.timeout_ns, abort_flag};

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int jt = 0, ju = 0, issued = 0;
        const int box_rows = p.ps < kKvTile ? p.ps : kKvTile;
        const int pages_per_tile = p.ps < kKvTile ? kKvTile / p.ps : 1;
        const uint32_t q_rows = p.head_mode == 0 ? (uint32_t)(p.G * p.tokens_per_unit) : (uint32_t)p.rows;
        PieceIter it;
        it.init(p);
        Unit x;
        while (it.next(p, x)) {
            const int qs = ju & 1;
            if (!warp_wait(&q_empty[qs], ((ju >> 1) & 1) ^ 1, wc, lane)) goto producer_done;
            if (lane == 0) {
                int h0, t0;
                if (p.head_mode == 0) { h0 = x.g * p.G; t0 = x.rg * p.tokens_per_unit; }
                else { t0 = x.rg / p.head_chunks; h0 = x.g * p.G + (x.rg % p.head_chunks) * p.rows; }
                mbar_arrive_expect_tx(&q_full[qs], 2u * q_rows * 128u);
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    tma_load_4d(smem_u32(sQ + qs * C::kQBytes + c * NQ * 128), &tm_q, &q_full[qs], c * 64, h0, t0,
                                x.b);
            }
            __syncwarp();
            {
                const int32_t *bt_row = p.block_table + (int64_t)x.b * p.bt_stride;
                for (int i = 0; i < x.ntiles; ++i, ++jt) {
                    const int ts = x.k_begin + i * kKvTile;
                    const int slot0 = p.ps < kKvTile ? 0 : ts % p.ps;
                    int npages = 1;
                    if (p.ps < kKvTile) npages = min(pages_per_tile, ceil_div_i(x.k_end - ts, p.ps));
                    int phys = 0;
                    if (lane < npages) {
                        phys = __ldg(bt_row + ts / p.ps + lane);
                        if ((unsigned)phys >= (unsigned)p.num_pages) { record_error(p.status, 1); phys = 0; }
                    }
                    const uint32_t bytes = (uint32_t)(npages * box_rows * 128);
                    const int s8 = jt % C::kStages8;
                    const uint32_t par = ((jt / C::kStages8) & 1) ^ 1;
                    if (!warp_wait(&k8_empty[s8], par, wc, lane)) goto producer_done;
                    if (lane == 0) mbar_arrive_expect_tx(&k8_full[s8], bytes);
                    __syncwarp();
                    if (lane < npages)
                        tma_load_4d(smem_u32(sK8 + s8 * C::kTile8Bytes + lane * box_rows * 128), &tm_k, &k8_full[s8],
                                    0, x.g, slot0, phys);
                    if (!warp_wait(&v8_empty[s8], par, wc, lane)) goto producer_done;
                    if (lane == 0) mbar_arrive_expect_tx(&v8_full[s8], bytes);
                    __syncwarp();
                    if (lane < npages)
                        tma_load_4d(smem_u32(sV8 + s8 * C::kTile8Bytes + lane * box_rows * 128), &tm_v, &v8_full[s8],
                                    0, x.g, slot0, phys);
                    issued = jt + 1;
                }
            }
            ++ju;
        }
    producer_done:
        if (lane == 0) {
            for (int k = 0; k < C::kStages8 && k < issued; ++k) {
                const int j = issued - 1 - k;
                mbar_wait_drain(&k8_full[j % C::kStages8], (j / C::kStages8) & 1, wc);
                mbar_wait_drain(&v8_full[j % C::kStages8], (j / C::kStages8) & 1, wc);
            }
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ------------------------------------------------------------ convert
        // Thread = key of the tile (its TMEM lane for K); keys at or past the
        // piece's end become zeros.  Waits that fail do not change the control
        // flow (each warp arrives on its own), so aborts wind down.
        const int q4 = warp & 3;
        const int key = q4 * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const int tq = threadIdx.x - 192;                 // 0..127
        int jt = 0, ju = 0;
        PieceIter it;
        it.init(p);
        Unit x;
        while (it.next(p, x)) {
            // Q of this unit: BF16 -> FP16 in place (each element keeps its
            // position, so the swizzled layout needs no remapping).
            const int qs = ju & 1;
            mbar_wait(&q_full[qs], (ju >> 1) & 1, wc);
            {
                uint32_t *qw = reinterpret_cast<uint32_t *>(sQ + qs * C::kQBytes);
                for (int i = tq; i < C::kQBytes / 4; i += 128) {
                    const uint32_t w = qw[i];
                    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
                    qw[i] = pack_half2(lo, hi);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&q16[qs]);
            for (int i = 0; i < x.ntiles; ++i, ++jt) {
                const int valid = x.k_end - (x.k_begin + i * kKvTile);   // keys of the tile inside the piece
                const bool live = key < valid;
                const int s8 = jt % C::kStages8;
                const uint32_t par8 = (jt / C::kStages8) & 1;
                const int b16 = jt & 1;
                const uint32_t par16 = ((jt >> 1) & 1) ^ 1;
                // K row -> TMEM lane `key`, 64 columns of FP16 pairs.
                mbar_wait(&k8_full[s8], par8, wc);
                mbar_wait(&qk_done[b16], par16, wc);      // QK(jt - 2) read this buffer
                tc_fence_after();
                const uint8_t *krow = sK8 + s8 * C::kTile8Bytes + key * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 r[2];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        r[k] = *reinterpret_cast<const uint4 *>(krow + (((2 * c + k) ^ (key & 7)) << 4));
                        if (!live) r[k] = make_uint4(0, 0, 0, 0);
                    }
                    uint32_t w16[16];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint32_t wd[4] = {r[k].x, r[k].y, r[k].z, r[k].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            w16[8 * k + 2 * e] = e4m3x2_to_f16x2((uint16_t)(wd[e] & 0xffffu));
                            w16[8 * k + 2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(wd[e] >> 16));
                        }
                    }
                    tmem_st16u(tmem + lane_off + C::kColK + b16 * 64 + c * 16, w16);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&k8_empty[s8]);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&k16_full[b16]);
                // V row -> swizzled FP16 tile (two 64-column chunks)
                mbar_wait(&v8_full[s8], par8, wc);
                mbar_wait(&pv_done[b16], par16, wc);      // PV(jt - 2) read this buffer
                const uint8_t *vrow = sV8 + s8 * C::kTile8Bytes + key * 128;
                uint8_t *v16 = sV16 + b16 * C::kTile16Bytes;
#pragma unroll 4
                for (int u = 0; u < 8; ++u) {              // FP8 unit u = columns 16u .. 16u + 15
                    uint4 r = *reinterpret_cast<const uint4 *>(vrow + ((u ^ (key & 7)) << 4));
                    if (!live) r = make_uint4(0, 0, 0, 0);
                    const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
                    uint32_t h[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        h[2 * e] = e4m3x2_to_f16x2((uint16_t)(wd[e] & 0xffffu));
                        h[2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(wd[e] >> 16));
                    }
                    const int chunk = u >> 2;                // 64 columns per chunk
                    const int unit = (u & 3) * 2;            // 8 FP16 columns per 16-byte unit
                    uint8_t *rowp = v16 + chunk * C::kChunkBytes + key * 128;
                    *reinterpret_cast<uint4 *>(rowp + ((unit ^ (key & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4 *>(rowp + (((unit + 1) ^ (key & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&v8_empty[s8]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&v16_full[b16]);
            }
            ++ju;
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            int jt = 0, ju = 0, pend = -1;
            bool pend_first = false;
            auto issue_pv = [&](int jj, bool first) -> bool {
                const int b16 = jj & 1;
                const int pb = jj & 1;
                if (!mbar_wait(&v16_full[b16], (jj >> 1) & 1, wc)) return false;
                if (!mbar_wait(&p_full[pb], (jj >> 1) & 1, wc)) return false;
                tc_fence_after();
                const uint32_t v_base = smem_u32(sV16 + b16 * C::kTile16Bytes);
                const uint32_t p_base = smem_u32(sP + pb * C::kPBytes);
#pragma unroll
                for (int kk = 0; kk < kKvTile / 16; ++kk) {
                    const uint64_t a = sdesc_sw128(v_base + kk * 16 * 128, C::kChunkBytes, 1024);
                    const uint64_t b = sdesc_sw128(p_base + (kk >> 2) * NQ * 128 + (kk & 3) * 32, 16, 1024);
                    mma_bf16_ss(tmem + C::kColO, a, b, C::kIdescPV, (first && kk == 0) ? 0u : 1u);
                }
                mma_commit(&pv_done[b16]);
                return true;
            };
            PieceIter it;
            it.init(p);
            Unit x;
            while (it.next(p, x)) {
                const int qs = ju & 1;
                if (!mbar_wait(&q16[qs], (ju >> 1) & 1, wc)) goto mma_done;
                for (int i = 0; i < x.ntiles; ++i, ++jt) {
                    const int b16 = jt & 1;
                    const int sb = jt & 1;
                    if (!mbar_wait(&k16_full[b16], (jt >> 1) & 1, wc)) goto mma_done;
                    if (!mbar_wait(&s_free[sb], ((jt >> 1) & 1) ^ 1, wc)) goto mma_done;
                    tc_fence_after();
                    const uint32_t q_base = smem_u32(sQ + qs * C::kQBytes);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t b = sdesc_sw128(q_base + (kk >> 2) * NQ * 128 + (kk & 3) * 32, 16, 1024);
                        mma_bf16_ts(tmem + C::kColS + sb * NQ, tmem + C::kColK + b16 * 64 + kk * 8, b, C::kIdescQK,
                                    kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&qk_done[b16]);
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
    } else if (warp >= 2) {
        // ------------------------------------------------- softmax / epilogue
        // As in the BF16 decode kernel: thread = key of the tile, all NQ rows
        // of its S^T column in registers, conditional rescale; P as FP16.
        const int q4 = warp & 3;
        const int row_in_tile = q4 * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        int jt = 0;
        PieceIter it;
        it.init(p);
        Unit x;
        while (it.next(p, x)) {
            int lim[R];
            int nrows = 0;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                int t, h;
                const bool ok = unit_row(p, x, r, t, h);
                lim[r] = ok ? min(x.n, x.n - p.q_len + t + 1) : 0;
                if (ok) nrows = r + 1;
            }
            float m_ref[R], l_part[R];
#pragma unroll
            for (int r = 0; r < R; ++r) { m_ref[r] = kNegInf; l_part[r] = 0.f; }
            for (int i = 0; i < x.ntiles; ++i, ++jt) {
                const int ts = x.k_begin + i * kKvTile;
                const int tok = ts + row_in_tile;
                const int sb = jt & 1;
                mbar_wait(&qk_done[sb], (jt >> 1) & 1, wc);
                tc_fence_after();
                float s[R];
                tmem_ld_cols<R>(tmem + lane_off + C::kColS + sb * NQ, s);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[sb]);
                float *rm = red_max + (jt & 1) * 4 * R;
#pragma unroll
                for (int r = 0; r < R; ++r) s[r] = (tok < lim[r]) ? s[r] * p.scale_log2 : kNegInf;
                warp_rows_reduce<R, true>(s, lane, rm + q4 * R);
                named_bar_sync(1, 128);
                bool need = false;
                float mx[R];
#pragma unroll
                for (int r = 0; r < R; r += 4) {
                    // Padding rows hold -inf everywhere: mx = -inf, no rescale.
                    float4 m4 = *reinterpret_cast<const float4 *>(rm + r);
#pragma unroll
                    for (int q = 1; q < 4; ++q) {
                        const float4 o4 = *reinterpret_cast<const float4 *>(rm + q * R + r);
                        m4.x = fmaxf(m4.x, o4.x); m4.y = fmaxf(m4.y, o4.y);
                        m4.z = fmaxf(m4.z, o4.z); m4.w = fmaxf(m4.w, o4.w);
                    }
                    mx[r] = m4.x; mx[r + 1] = m4.y; mx[r + 2] = m4.z; mx[r + 3] = m4.w;
                }
#pragma unroll
                for (int r = 0; r < R; ++r) need |= mx[r] > m_ref[r] + kRescaleThreshold;
                if (need) {
                    float alpha[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float mn = fmaxf(m_ref[r], mx[r]);
                        alpha[r] = (mn == kNegInf) ? 1.f : ex2_approx(m_ref[r] - mn);
                        l_part[r] *= alpha[r];
                        m_ref[r] = mn;
                    }
                    if (i > 0) {
                        // Rescale once PV(jt - 1) has landed (the P-buffer wait
                        // of tile jt + 1); PV(jt - 2) has, as qk_done(jt) was
                        // committed after it was issued.
                        mbar_wait(&pv_done[(jt + 1) & 1], (((jt + 1) >> 1) & 1) ^ 1, wc);
                        tc_fence_after();
                        float o[R];
                        const uint32_t ta = tmem + lane_off + C::kColO;
                        tmem_ld_cols<R>(ta, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < R; ++k) o[k] *= alpha[k];
                        tmem_st_cols<R>(ta, o);
                        tmem_wait_st();
                    }
                }
                const int pb = jt & 1;
                mbar_wait(&pv_done[pb], ((jt >> 1) & 1) ^ 1, wc);     // PV(jt - 2) read P buffer pb
                uint8_t *pbuf = sP + pb * C::kPBytes;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    // Masked keys and padding rows have s = -inf: p = 0 exactly.
                    // Rows R..NQ-1 of P stay at the zeros written at start.
                    const float mu = (m_ref[r] == kNegInf) ? 0.f : m_ref[r] - kHeadroom;
                    const float pr = ex2_approx(s[r] - mu);
                    l_part[r] += pr;
                    *reinterpret_cast<__half *>(pbuf + sw128_offset(r, row_in_tile, NQ)) = __float2half_rn(pr);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[pb]);
            }
            // ------------------------------------------------------ epilogue
            {
                warp_rows_reduce<R, false>(l_part, lane, red_sum + q4 * R);
                named_bar_sync(1, 128);
                float L[R];
#pragma unroll
                for (int r = 0; r < R; ++r)
                    L[r] = (red_sum[r] + red_sum[R + r]) + (red_sum[2 * R + r] + red_sum[3 * R + r]);
                // O^T is final once PV(jt - 2) and PV(jt - 1), the unit's
                // last, have landed: the P-buffer waits of tiles jt and jt + 1.
                // Each buffer's barrier is at most one phase behind its waiter,
                // so the parity waits are unambiguous.
                mbar_wait(&pv_done[jt & 1], ((jt >> 1) & 1) ^ 1, wc);
                mbar_wait(&pv_done[(jt + 1) & 1], (((jt + 1) >> 1) & 1) ^ 1, wc);
                tc_fence_after();
                float o[R];
                tmem_ld_cols<R>(tmem + lane_off + C::kColO, o);
                tmem_wait_ld();
                const int dv = row_in_tile;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    int t, h;
                    if (r >= nrows || !unit_row(p, x, r, t, h)) continue;
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
                if (row_in_tile < nrows) {
                    const int r = row_in_tile;
                    int t, h;
                    if (unit_row(p, x, r, t, h)) {
                        float lse2 = kNegInf;
#pragma unroll
                        for (int k = 0; k < R; ++k)
                            if (k == r && L[k] > 0.f) lse2 = m_ref[k] - kHeadroom + __log2f(L[k]);
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
}

template <int NQ, int R>
cudaError_t launch_fp8_t(const DecodeParams &p, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         cudaStream_t stream) {
    using C = Fp8Cfg<NQ>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(paged_decode_fp8_kernel<NQ, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    paged_decode_fp8_kernel<NQ, R><<<p.grid, 320, C::kSmemBytes, stream>>>(p, tq, tk, tv);
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
