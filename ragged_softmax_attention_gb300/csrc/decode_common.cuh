// Scheduling helpers shared by the paged-decode kernels (BF16 and FP8 KV):
// the pieces of a CTA's tile ranges over the (batch row, KV head, row group)
// units, the query row a unit's N-axis position holds, and warp reductions.
#pragma once

#include "fw_internal.h"
#include "fw_ptx.cuh"

namespace fw {
namespace dec {

struct Unit {                 // one piece: a unit's tiles inside one CTA range
    int b, g, rg, n, lo, k_begin, k_end, ntiles;   // lo: first key any row of the unit may see
    int k, npieces;
    bool single;
};

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int clamp_len(const DecodeParams &p, int n) {
    const int cap = p.max_pages * p.ps;
    return n < 0 ? 0 : (n > cap ? cap : n);
}

// First key any query row of a row with n keys may see: max(0, n - q_len -
// W) under a sliding window of W ("TokenSpeed-MLA 2.0.1", window_left), else
// 0.  The row's walk starts at the tile holding it; pages wholly before it
// are never read.
__device__ __forceinline__ int window_first_key(const DecodeParams &p, int n) {
    return p.window_left < 0 ? 0 : max(0, n - p.q_len - p.window_left);
}

// KV tiles a row with n keys walks (per unit).
__device__ __forceinline__ int row_tiles(const DecodeParams &p, int n) {
    return ceil_div_i(n, kKvTile) - window_first_key(p, n) / kKvTile;
}

// The per-row slot prefix PB[0..B] and the sequence lengths, copied into
// shared memory once per CTA when the batch fits (else read in place): the
// piece walk then finds the next unit without a global load, which at every
// piece boundary cost the softmax warps ~2,000 cycles.  All threads of the
// CTA call it, after the plan is visible.
struct RowTables {
    const int32_t *pb;
    const int32_t *lens;
};
__device__ __forceinline__ RowTables cache_row_tables(const DecodeParams &p, int32_t *smem_rows, int cap) {
    if (p.B + 1 + p.B > cap) return RowTables{p.plan + 2, p.seq_lens};
    for (int i = threadIdx.x; i <= p.B; i += blockDim.x) smem_rows[i] = p.plan[2 + i];
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) smem_rows[p.B + 1 + i] = __ldg(p.seq_lens + i);
    __syncthreads();
    return RowTables{smem_rows, smem_rows + p.B + 1};
}

// Walks the pieces of this CTA's tile ranges; every role runs its own copy
// and sees the same sequence.  With the KV heads riding on the CTA index
// (head_ride) the CTA's head is fixed and the units of a row are its row
// groups.
struct PieceIter {
    int T, span, range, step, g_ride, pos, end, b;
    RowTables rt;

    __device__ void init(const DecodeParams &p, RowTables tables) {
        rt = tables;
        T = __ldg(p.plan + 0);
        span = max(1, __ldg(p.plan + 1));
        if (p.head_ride) {
            range = blockIdx.x / p.Hkv;
            step = gridDim.x / p.Hkv;
            g_ride = blockIdx.x % p.Hkv;
        } else {
            range = blockIdx.x;
            step = gridDim.x;
            g_ride = 0;
        }
        pos = 0;
        end = 0;
        b = -1;
        open_range();
    }
    __device__ void open_range() {
        const long long lo = (long long)range * span;
        pos = lo < T ? (int)lo : T;
        end = (int)min((long long)T, lo + span);
        b = -1;
    }
    __device__ bool next(const DecodeParams &p, Unit &x) {
        const int32_t *PB = rt.pb;
        for (;;) {
            while (pos >= end) {
                range += step;
                if ((long long)range * span >= T) return false;
                open_range();
            }
            if (b < 0) {
                int lo = 0, hi = p.B - 1;              // largest b with PB[b] <= pos
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (PB[mid] <= pos) lo = mid; else hi = mid - 1;
                }
                b = lo;
            } else {
                // Within a range the walk only moves forward, mostly into the
                // next row: a scan costs one dependent load per row crossed,
                // where a fresh binary search costs log2(B).
                while (pos >= PB[b + 1]) ++b;
            }
            // Row b holds units_per_row units of vb slots: piece_cost empty
            // ones, then the unit's tb tiles.
            const int pb0 = PB[b];
            const int vb = (PB[b + 1] - pb0) / p.units_per_row;
            const int off = pos - pb0;
            const int u = off / vb;
            const int vl = off - u * vb;
            if (vl < p.piece_cost) {                   // empty slots carry no tiles
                pos += p.piece_cost - vl;
                continue;
            }
            const int tb = vb - p.piece_cost;
            const int tl = vl - p.piece_cost;
            const int th = min(tb, tl + (end - pos));
            const int pstart = pb0 + u * vb + p.piece_cost;   // the unit's first tile
            x.b = b;
            if (p.head_ride) {
                x.g = g_ride;
                x.rg = u;
            } else {
                x.g = u / p.row_groups;
                x.rg = u - x.g * p.row_groups;
            }
            x.n = clamp_len(p, rt.lens[b]);
            x.lo = window_first_key(p, x.n);
            const int t0 = x.lo / kKvTile;               // the walk starts at the window's first tile
            x.k_begin = (t0 + tl) * kKvTile;
            x.k_end = min(x.n, (t0 + th) * kKvTile);
            x.ntiles = th - tl;
            x.k = (pstart + tl) / span - pstart / span;
            x.npieces = (pstart + tb - 1) / span - pstart / span + 1;
            x.single = (x.npieces == 1);
            pos += th - tl;
            return true;
        }
    }
};

// Latent-head decode: one piece is a (batch row, KV head) unit's tiles inside
// one tile range, for one row group: packed rows row0 .. row0 + rows of the
// unit, packed row i being token i / G, head g * G + i % G (when G is a
// multiple of `rows` a group is one token's heads h0 .. h0 + rows).
struct LatentPiece {
    int b, g, t, h0, row0, n, lo, k_begin, k_end, ntiles, k;   // lo: first key any row may see
    bool single;
};

// Walks the pieces of worker `idx` of `count` (a CTA, or a CTA pair): tile
// ranges idx / R, idx / R + count / R, ... over the units laid end to end in
// tile order, for row group idx % R (R = range_groups), so the R workers that
// read the same keys run side by side.  Every role runs its own copy and
// sees the same sequence.  Latent plans carry no empty slots
// (piece_cost = 0: the host never sets it for them), so a unit's slots are its
// tiles; keeping that case out of this walk keeps the pair kernel's roles
// within their registers.
struct LatentIter {
    int T, span, range, step, pos, end, b, rg;

    __device__ void init(const DecodeParams &p, int idx, int count) {
        T = __ldg(p.plan + 0);
        span = max(1, __ldg(p.plan + 1));
        step = max(1, count / p.range_groups);
        range = idx / p.range_groups;
        rg = idx % p.range_groups;
        open_range();
    }
    __device__ void open_range() {
        const long long lo = (long long)range * span;
        pos = lo < T ? (int)lo : T;
        end = (int)min((long long)T, lo + span);
        b = -1;
    }
    __device__ bool next(const DecodeParams &p, LatentPiece &x) {
        const int32_t *PB = p.plan + 2;
        while (pos >= end) {
            range += step;
            if ((long long)range * span >= T) return false;
            open_range();
        }
        if (b < 0 || pos >= __ldg(PB + b + 1)) {
            int lo = 0, hi = p.B - 1;              // largest b with PB[b] <= pos
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (__ldg(PB + mid) <= pos) lo = mid; else hi = mid - 1;
            }
            b = lo;
        }
        const int pb0 = __ldg(PB + b);
        const int tb = (__ldg(PB + b + 1) - pb0) / p.units_per_row;
        const int off = pos - pb0;
        const int u = off / tb;
        const int tl = off - u * tb;
        const int th = min(tb, tl + (end - pos));
        const int pstart = pb0 + u * tb;
        x.b = b;
        x.g = u;
        x.row0 = rg * p.rows;
        x.t = x.row0 / p.G;
        x.h0 = u * p.G + x.row0 % p.G;
        x.n = clamp_len(p, __ldg(p.seq_lens + b));
        x.lo = window_first_key(p, x.n);
        const int t0 = x.lo / kKvTile;               // the walk starts at the window's first tile
        x.k_begin = (t0 + tl) * kKvTile;
        x.k_end = min(x.n, (t0 + th) * kKvTile);
        x.ntiles = th - tl;
        x.k = (pstart + tl) / span - pstart / span;
        x.single = ((pstart + tb - 1) / span == pstart / span);
        pos += th - tl;
        return true;
    }
};

// Query row r of unit x -> (token t, head h); false if the row is padding.
__device__ __forceinline__ bool unit_row(const DecodeParams &p, const Unit &x, int r, int &t, int &h) {
    if (p.head_mode == 0) {
        const int tt = r / p.G;
        t = x.rg * p.tokens_per_unit + tt;
        h = x.g * p.G + (r - tt * p.G);
        return tt < p.tokens_per_unit && t < p.q_len;
    }
    t = x.rg / p.head_chunks;
    const int hh = (x.rg % p.head_chunks) * p.rows + r;
    h = x.g * p.G + hh;
    return hh < p.G;
}

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

// Reduces each of the NQ per-lane values over the warp (max or sum) and
// stores row r's result to dst[r].  Reduce-scatter: every butterfly stage
// sends the half of the remaining rows that the partner lane keeps, so the
// warp issues NQ - 1 + (5 - log2 NQ) shuffles instead of 5 NQ, and the
// shuffles of one stage are independent of each other.
template <int NQ, bool kMax>
__device__ __forceinline__ void warp_rows_reduce(const float (&v)[NQ], int lane, float *dst) {
    static_assert(NQ == 4 || NQ == 8 || NQ == 16 || NQ == 32, "rows per warp reduction");
    float a[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) a[i] = v[i];
    int row = 0;
#pragma unroll
    for (int st = 0; st < 5; ++st) {
        const int off = 16 >> st;
        const int half = NQ >> (st + 1);
        if (half >= 1) {
            const bool hi = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float send = hi ? a[i] : a[half + i];
                const float keep = hi ? a[half + i] : a[i];
                const float got = __shfl_xor_sync(0xffffffffu, send, off);
                a[i] = kMax ? fmaxf(keep, got) : keep + got;
            }
            row += hi ? half : 0;
        } else {
            const float got = __shfl_xor_sync(0xffffffffu, a[0], off);
            a[0] = kMax ? fmaxf(a[0], got) : a[0] + got;
        }
    }
    if ((lane & (32 / NQ - 1)) == 0) dst[row] = a[0];
}

// R consecutive 32-bit TMEM columns of this warp's lane quadrant.
template <int R>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[R]) {
    static_assert(R % 4 == 0, "columns in groups of 4");
    if constexpr (R % 16 == 0) {
#pragma unroll
        for (int c = 0; c < R; c += 16) tmem_ld16(taddr + c, *reinterpret_cast<float(*)[16]>(&v[c]));
    } else if constexpr (R % 8 == 0) {
#pragma unroll
        for (int c = 0; c < R; c += 8) tmem_ld8(taddr + c, *reinterpret_cast<float(*)[8]>(&v[c]));
    } else {
#pragma unroll
        for (int c = 0; c < R; c += 4) tmem_ld4(taddr + c, *reinterpret_cast<float(*)[4]>(&v[c]));
    }
}
template <int R>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float (&v)[R]) {
    static_assert(R % 4 == 0, "columns in groups of 4");
    if constexpr (R % 16 == 0) {
#pragma unroll
        for (int c = 0; c < R; c += 16) tmem_st16(taddr + c, *reinterpret_cast<const float(*)[16]>(&v[c]));
    } else if constexpr (R % 8 == 0) {
#pragma unroll
        for (int c = 0; c < R; c += 8) tmem_st8(taddr + c, *reinterpret_cast<const float(*)[8]>(&v[c]));
    } else {
#pragma unroll
        for (int c = 0; c < R; c += 4) tmem_st4(taddr + c, *reinterpret_cast<const float(*)[4]>(&v[c]));
    }
}

// One lane waits, the whole warp learns the outcome (keeps the warp converged).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const WaitCtx &w, int lane) {
    int ok = 1;
    if (lane == 0) ok = mbar_wait(bar, parity, w) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

}  // namespace dec
}  // namespace fw
