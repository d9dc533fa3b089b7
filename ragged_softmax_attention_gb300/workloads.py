"""Seeded synthetic inputs for paged decode and ragged (varlen) prefill.

This module only draws random tensors and index structures: values, sequence
lengths, physical page permutations and block tables.  It holds none of the
attention arithmetic, so both the CUDA path and the fp64 oracle can be fed from
it without sharing any of the method's computation.

Shapes follow the pages' workloads:
  * "Writing Page Attention with PyPTO", section 1 (Qwen3-14B decode: 40 Q heads,
    8 KV heads, head_dim 128, 128-token pages, block_table[batch, logical_page]);
  * "TokenSpeed-MLA 2.0.1", capability summary (ragged varlen prefill packed by
    cumulative sequence lengths; latent-head decode with q_len 4, kv 80K, page 64);
  * "Flywheel Attention", section 4.1 (causal forward at head_dim 256, batch 1).

Seeds: values use ``value_seed`` (1234 + workload index), sequence lengths seed
99, the physical page permutation seed 7.  Slots of the page pool that no
sequence covers (spare pages and the tail of each sequence's last page) are
filled with NaN, so any read outside the ragged extent poisons the result.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

SEQ_LEN_SEED = 99
PAGE_PERM_SEED = 7


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    q_len: int
    num_q_heads: int
    num_kv_heads: int
    head_dim_qk: int
    head_dim_v: int
    page_size: int
    scale: float
    seq_lens: Optional[tuple] = None          # fixed lengths (one per batch row)
    seq_len_range: Optional[tuple] = None     # inclusive uniform integer range
    latent: bool = False                      # V = first head_dim_v columns of each K row
    kv_fp8: bool = False                      # K/V caches in FP8 E4M3 with one scale each
    value_seed: int = 1234
    spare_pages: int = 3                      # NaN-filled pool pages no sequence uses

    @property
    def max_seq_len(self) -> int:
        if self.seq_lens is not None:
            return max(self.seq_lens) if self.seq_lens else 0
        return self.seq_len_range[1]

    @property
    def max_pages(self) -> int:
        return max(1, -(-self.max_seq_len // self.page_size))


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim_qk: int
    head_dim_v: int
    causal: bool
    scale: float
    seq_lens: Optional[tuple] = None
    seq_len_range: Optional[tuple] = None
    value_seed: int = 1234


WORKLOADS = {
    "tiny_paged_decode": DecodeWorkload(
        "tiny_paged_decode", batch=2, q_len=1, num_q_heads=8, num_kv_heads=2,
        head_dim_qk=128, head_dim_v=128, page_size=16, scale=1.0 / math.sqrt(128),
        seq_lens=(37, 200), value_seed=1234, spare_pages=0),
    "qwen3_14b_paged_decode": DecodeWorkload(
        "qwen3_14b_paged_decode", batch=64, q_len=1, num_q_heads=40, num_kv_heads=8,
        head_dim_qk=128, head_dim_v=128, page_size=128, scale=1.0 / math.sqrt(128),
        seq_len_range=(512, 32768), value_seed=1235),
    "varlen_gqa_prefill": PrefillWorkload(
        "varlen_gqa_prefill", num_seqs=16, num_q_heads=32, num_kv_heads=8,
        head_dim_qk=128, head_dim_v=128, causal=True, scale=1.0 / math.sqrt(128),
        seq_len_range=(256, 8192), value_seed=1236),
    "qwen3_14b_paged_decode_fp8": DecodeWorkload(
        "qwen3_14b_paged_decode_fp8", batch=64, q_len=1, num_q_heads=40, num_kv_heads=8,
        head_dim_qk=128, head_dim_v=128, page_size=128, scale=1.0 / math.sqrt(128.0),
        seq_len_range=(512, 32768), kv_fp8=True, value_seed=1235),
    "dense_causal_mha_hd256": PrefillWorkload(
        "dense_causal_mha_hd256", num_seqs=1, num_q_heads=16, num_kv_heads=16,
        head_dim_qk=256, head_dim_v=256, causal=True, scale=1.0 / 16.0,
        seq_lens=(8192,), value_seed=1237),
    "latent_paged_decode": DecodeWorkload(
        "latent_paged_decode", batch=32, q_len=4, num_q_heads=128, num_kv_heads=1,
        head_dim_qk=576, head_dim_v=512, page_size=64, scale=0.07216882,
        seq_lens=(81920,) * 32, latent=True, value_seed=1238),
}


def draw_seq_lens(num: int, lo: int, hi: int, seed: int = SEQ_LEN_SEED) -> list:
    """Integers uniform in [lo, hi], drawn from a seeded CPU generator."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randint(lo, hi + 1, (num,), generator=g).tolist()


def workload_seq_lens(wl) -> list:
    if wl.seq_lens is not None:
        return list(wl.seq_lens)
    n = wl.batch if isinstance(wl, DecodeWorkload) else wl.num_seqs
    return draw_seq_lens(n, wl.seq_len_range[0], wl.seq_len_range[1])


def _randn(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_block_table(seq_lens: Sequence[int], page_size: int, max_pages: int,
                     spare_pages: int = 0, mapping: str = "random",
                     seed: int = PAGE_PERM_SEED):
    """Assign physical pages to every (batch, logical page) a sequence covers.

    mapping: "random" (seeded permutation of the pool), "identity", "reverse"
    or "shared_prefix" (all rows share their first common full pages), the
    adversarial tables of "Writing Page Attention with PyPTO", section 10.2.
    Unused entries hold -1.  Returns (block_table [B, max_pages] int32 CPU
    tensor, num_pages).
    """
    B = len(seq_lens)
    pages_per_row = [-(-int(n) // page_size) for n in seq_lens]
    bt = torch.full((B, max_pages), -1, dtype=torch.int32)
    if mapping == "shared_prefix":
        shared = min(int(n) for n in seq_lens) // page_size // 2 if B else 0
        used = shared + sum(p - shared for p in pages_per_row)
    else:
        shared = 0
        used = sum(pages_per_row)
    num_pages = used + spare_pages
    if mapping in ("random", "shared_prefix"):
        g = torch.Generator(device="cpu").manual_seed(seed)
        perm = torch.randperm(num_pages, generator=g).tolist()
    elif mapping == "identity":
        perm = list(range(num_pages))
    elif mapping == "reverse":
        perm = list(range(num_pages))[::-1]
    else:
        raise ValueError(f"unknown page mapping {mapping!r}")
    nxt = shared
    for b in range(B):
        for p in range(pages_per_row[b]):
            if p < shared:
                bt[b, p] = perm[p]
            else:
                bt[b, p] = perm[nxt]
                nxt += 1
    return bt, num_pages


def make_decode_inputs(wl: DecodeWorkload, device="cpu", seq_lens=None, mapping="random",
                       poison=True):
    """Seeded inputs for one paged decode call.

    Returns a dict with q [B, q_len, Hq, Dk], k_cache [P, ps, Hkv, Dk],
    v_cache [P, ps, Hkv, Dv] (a strided view of k_cache for latent heads),
    block_table [B, max_pages] int32, seq_lens [B] int32 and scale.
    """
    lens = list(seq_lens) if seq_lens is not None else workload_seq_lens(wl)
    max_pages = max(1, max([-(-int(n) // wl.page_size) for n in lens] + [wl.max_pages]))
    bt, num_pages = make_block_table(lens, wl.page_size, max_pages, wl.spare_pages, mapping)
    gen = torch.Generator(device=device).manual_seed(wl.value_seed)
    q = _randn((wl.batch, wl.q_len, wl.num_q_heads, wl.head_dim_qk), gen, device)
    k_cache = _randn((num_pages, wl.page_size, wl.num_kv_heads, wl.head_dim_qk), gen, device)
    if wl.latent:
        v_cache = k_cache[..., : wl.head_dim_v]
    else:
        v_cache = _randn((num_pages, wl.page_size, wl.num_kv_heads, wl.head_dim_v), gen, device)
    k_scale = v_scale = 1.0
    if wl.kv_fp8:
        # One scale per cache: the largest magnitude maps to E4M3's largest
        # finite value (448), so no value saturates.
        k_scale = float(k_cache.float().abs().amax()) / 448.0
        v_scale = float(v_cache.float().abs().amax()) / 448.0
        k_cache = (k_cache.float() / k_scale).to(torch.float8_e4m3fn)
        v_cache = (v_cache.float() / v_scale).to(torch.float8_e4m3fn)
    if poison:
        covered = torch.zeros((num_pages, wl.page_size), dtype=torch.bool)
        for b, n in enumerate(lens):
            for j in range(0, int(n), wl.page_size):
                cnt = min(wl.page_size, int(n) - j)
                covered[int(bt[b, j // wl.page_size]), :cnt] = True
        mask = (~covered).to(device)
        if wl.kv_fp8:                         # E4M3 NaN: S.1111.111
            k_cache.view(torch.uint8)[mask] = 0x7F
            if not wl.latent:
                v_cache.view(torch.uint8)[mask] = 0x7F
        else:
            nan = float("nan")
            k_cache[mask] = nan
            if not wl.latent:
                v_cache[mask] = nan
    return {
        "q": q,
        "k_cache": k_cache,
        "v_cache": v_cache,
        "block_table": bt.to(device),
        "seq_lens": torch.tensor(lens, dtype=torch.int32, device=device),
        "scale": float(wl.scale),
        "k_scale": k_scale,
        "v_scale": v_scale,
        "num_pages": num_pages,
    }


def make_prefill_inputs(wl: PrefillWorkload, device="cpu", seq_lens_q=None, seq_lens_k=None):
    """Seeded packed inputs for one varlen prefill call.

    Returns q [total_q, Hq, Dk], k [total_k, Hkv, Dk], v [total_k, Hkv, Dv],
    cu_seqlens_q / cu_seqlens_k [B+1] int32, plus the scale and causal flag.
    Q and KV packs may differ (seq_lens_k given separately).
    """
    lq = list(seq_lens_q) if seq_lens_q is not None else workload_seq_lens(wl)
    lk = list(seq_lens_k) if seq_lens_k is not None else list(lq)
    assert len(lq) == len(lk)
    cu_q = [0]
    cu_k = [0]
    for a, b in zip(lq, lk):
        cu_q.append(cu_q[-1] + int(a))
        cu_k.append(cu_k[-1] + int(b))
    gen = torch.Generator(device=device).manual_seed(wl.value_seed)
    q = _randn((cu_q[-1], wl.num_q_heads, wl.head_dim_qk), gen, device)
    k = _randn((cu_k[-1], wl.num_kv_heads, wl.head_dim_qk), gen, device)
    v = _randn((cu_k[-1], wl.num_kv_heads, wl.head_dim_v), gen, device)
    return {
        "q": q, "k": k, "v": v,
        "cu_seqlens_q": torch.tensor(cu_q, dtype=torch.int32, device=device),
        "cu_seqlens_k": torch.tensor(cu_k, dtype=torch.int32, device=device),
        "causal": bool(wl.causal),
        "scale": float(wl.scale),
    }
