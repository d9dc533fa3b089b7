"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test ties the oracle to something other than itself: a closed form, a
special case that reduces to a library routine (torch's scaled-dot-product
attention and logsumexp in float64), an invariant, or a worked example printed
on the pages (stored under tests/golden/ with its citation).  A second group
shows the pages' reformulations (online recurrence, split-KV merge, the
delayed-rescale FIFO) reach the oracle's one-shot result.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import planning
from ragged_softmax_attention_gb300.workloads import (DecodeWorkload, PrefillWorkload,
                                                      make_block_table, make_decode_inputs,
                                                      make_prefill_inputs)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def tiny_decode(batch=3, q_len=1, hq=8, hkv=2, d=32, dv=None, ps=4, lens=(5, 1, 13), seed=3,
                mapping="random", latent=False):
    wl = DecodeWorkload("t", batch=batch, q_len=q_len, num_q_heads=hq, num_kv_heads=hkv,
                        head_dim_qk=d, head_dim_v=dv or d, page_size=ps, scale=1.0 / math.sqrt(d),
                        seq_lens=tuple(lens), value_seed=seed, spare_pages=2, latent=latent)
    return wl, make_decode_inputs(wl, "cpu", mapping=mapping)


def dense_kv(inp, b):
    """Gather batch row b's keys/values into a dense [n, Hkv, D] copy (plain indexing)."""
    n = int(inp["seq_lens"][b])
    ps = inp["k_cache"].shape[1]
    idx_page = [int(inp["block_table"][b, j // ps]) for j in range(n)]
    idx_slot = [j % ps for j in range(n)]
    k = inp["k_cache"][idx_page, idx_slot]
    v = inp["v_cache"][idx_page, idx_slot]
    return k, v


def sdpa_decode_reference(inp, b):
    """torch float64 scaled_dot_product_attention over a dense gathered copy.

    GQA by repeat_interleave (consecutive query heads share a KV head), causal
    bottom-right mask for q_len > 1 given explicitly as a boolean mask.
    """
    q = inp["q"][b].double()                        # [q_len, Hq, D]
    k, v = dense_kv(inp, b)
    q_len, hq, _ = q.shape
    hkv = k.shape[1]
    n = k.shape[0]
    k = k.double().repeat_interleave(hq // hkv, dim=1)
    v = v.double().repeat_interleave(hq // hkv, dim=1)
    mask = torch.zeros(q_len, n, dtype=torch.bool)
    for t in range(q_len):
        mask[t, : max(0, n - q_len + t + 1)] = True
    out = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1), attn_mask=mask,
        scale=inp["scale"])                         # [Hq, q_len, Dv]
    scores = torch.einsum("thd,nhd->htn", q, k) * inp["scale"]
    scores = scores.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(scores, dim=-1)           # [Hq, q_len]
    return out.transpose(0, 1).reshape(q_len * hq, -1).numpy(), lse.transpose(0, 1).reshape(-1).numpy()


# --------------------------------------------------------------- library routine

@pytest.mark.parametrize("q_len,lens,ps,mapping", [
    (1, (5, 1, 13), 4, "random"),
    (1, (16, 17, 3), 8, "reverse"),
    (3, (7, 9, 12), 4, "random"),
    (4, (4, 30, 11), 16, "shared_prefix"),
])
def test_decode_matches_sdpa_on_dense_copy(q_len, lens, ps, mapping):
    wl, inp = tiny_decode(q_len=q_len, lens=lens, ps=ps, mapping=mapping)
    out, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"])
    rows_per_b = q_len * wl.num_q_heads
    for b in range(wl.batch):
        ref_o, ref_l = sdpa_decode_reference(inp, b)
        np.testing.assert_allclose(out[b * rows_per_b:(b + 1) * rows_per_b], ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b * rows_per_b:(b + 1) * rows_per_b], ref_l, rtol=0, atol=1e-12)


def test_prefill_matches_sdpa_per_sequence():
    wl = PrefillWorkload("p", num_seqs=3, num_q_heads=6, num_kv_heads=3, head_dim_qk=16,
                         head_dim_v=8, causal=True, scale=0.3, value_seed=5)
    lq, lk = [5, 1, 9], [7, 4, 9]
    inp = make_prefill_inputs(wl, "cpu", lq, lk)
    out, lse = oracle.varlen_prefill(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"],
                                     inp["cu_seqlens_k"], True, wl.scale)
    cq, ck = inp["cu_seqlens_q"].tolist(), inp["cu_seqlens_k"].tolist()
    for i in range(3):
        q = inp["q"][cq[i]:cq[i + 1]].double().transpose(0, 1)
        k = inp["k"][ck[i]:ck[i + 1]].double().repeat_interleave(2, dim=1).transpose(0, 1)
        v = inp["v"][ck[i]:ck[i + 1]].double().repeat_interleave(2, dim=1).transpose(0, 1)
        Lq, Lk = lq[i], lk[i]
        mask = torch.ones(Lq, Lk, dtype=torch.bool).tril(diagonal=Lk - Lq)   # bottom-right
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=wl.scale)
        ref = ref.transpose(0, 1).reshape(Lq * 6, -1).numpy()
        np.testing.assert_allclose(out[cq[i] * 6:cq[i + 1] * 6], ref, rtol=0, atol=1e-12)
        s = torch.einsum("hqd,hkd->hqk", q, k) * wl.scale
        ref_l = torch.logsumexp(s.masked_fill(~mask, float("-inf")), -1).transpose(0, 1).reshape(-1)
        np.testing.assert_allclose(lse[cq[i] * 6:cq[i + 1] * 6], ref_l.numpy(), rtol=0, atol=1e-12)


def test_noncausal_prefill_dense_matches_sdpa():
    wl = PrefillWorkload("p", num_seqs=2, num_q_heads=4, num_kv_heads=4, head_dim_qk=8,
                         head_dim_v=8, causal=False, scale=0.5, value_seed=9)
    inp = make_prefill_inputs(wl, "cpu", [3, 6], [10, 2])
    out, _ = oracle.varlen_prefill(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"],
                                   inp["cu_seqlens_k"], False, wl.scale)
    q = inp["q"][:3].double().transpose(0, 1)
    k = inp["k"][:10].double().transpose(0, 1)
    v = inp["v"][:10].double().transpose(0, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=0.5)
    np.testing.assert_allclose(out[:12], ref.transpose(0, 1).reshape(12, -1).numpy(), atol=1e-12, rtol=0)


# ------------------------------------------------------------------ closed forms

def _bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


def test_seq_len_one_returns_that_value_row():
    """PyPTO section 10.1: seq_len = 1 -> context equals the selected V row."""
    wl, inp = tiny_decode(lens=(1, 1, 1), ps=4)
    out, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"])
    G = wl.num_q_heads // wl.num_kv_heads
    for b in range(3):
        page = int(inp["block_table"][b, 0])
        for h in range(wl.num_q_heads):
            r = b * wl.num_q_heads + h
            v = inp["v_cache"][page, 0, h // G].double().numpy()
            np.testing.assert_array_equal(out[r], v)
            k = inp["k_cache"][page, 0, h // G].double()
            s = float((inp["q"][b, 0, h].double() * k).sum()) * inp["scale"]
            assert abs(lse[r] - s) < 1e-12


def test_constant_values_give_that_constant():
    wl, inp = tiny_decode(lens=(9, 4, 13))
    c = torch.linspace(-3, 3, wl.head_dim_v).to(torch.bfloat16)
    inp["v_cache"][:] = c
    out, _ = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                 inp["seq_lens"], inp["scale"])
    np.testing.assert_allclose(out, np.broadcast_to(c.double().numpy(), out.shape), atol=1e-13, rtol=0)


def test_identical_keys_give_mean_value_and_log_n():
    wl, inp = tiny_decode(lens=(6, 11, 2))
    inp["k_cache"][:] = inp["k_cache"][0, 0]
    out, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"])
    G = wl.num_q_heads // wl.num_kv_heads
    for b in range(3):
        kk, vv = dense_kv(inp, b)
        n = kk.shape[0]
        for h in range(wl.num_q_heads):
            r = b * wl.num_q_heads + h
            np.testing.assert_allclose(out[r], vv[:, h // G].double().mean(0).numpy(), atol=1e-13, rtol=0)
            s = float((inp["q"][b, 0, h].double() * kk[0, h // G].double()).sum()) * inp["scale"]
            assert abs(lse[r] - (s + math.log(n))) < 1e-12


def test_two_key_closed_form():
    """Two keys with scores a and 0: weights e^a/(1+e^a) and 1/(1+e^a)."""
    a = 1.09375                            # 1 + 12/128: exact in bf16, close to ln 3
    q = torch.zeros(1, 1, 1, 4, dtype=torch.bfloat16); q[..., 0] = 1
    k = torch.zeros(1, 2, 1, 4, dtype=torch.bfloat16); k[0, 0, 0, 0] = a
    v = torch.zeros(1, 2, 1, 2, dtype=torch.bfloat16)
    v[0, 0, 0] = _bf16([2.0, -1.0]); v[0, 1, 0] = _bf16([-6.0, 0.5])
    out, lse = oracle.paged_decode(q, k, v, torch.tensor([[0]], dtype=torch.int32),
                                   torch.tensor([2], dtype=torch.int32), 1.0)
    w1 = math.exp(a) / (1 + math.exp(a))
    assert abs(out[0, 0] - (2.0 * w1 - 6.0 * (1 - w1))) < 1e-14
    assert abs(out[0, 1] - (-1.0 * w1 + 0.5 * (1 - w1))) < 1e-14
    assert abs(lse[0] - math.log(1 + math.exp(a))) < 1e-14


def test_gqa_mapping_worked_example():
    """PyPTO section 1.3: with 40 Q / 8 KV heads, KV head 1 serves Q heads 5-9."""
    g = _golden("pypto_worked_examples.json")["task_mapping"]
    wl = DecodeWorkload("m", batch=2, q_len=1, num_q_heads=40, num_kv_heads=8, head_dim_qk=16,
                        head_dim_v=4, page_size=4, scale=0.25, seq_lens=(5, 7), value_seed=2)
    inp = make_decode_inputs(wl, "cpu")
    v = inp["v_cache"]
    v[:, :, :, :] = 0
    v[:, :, g["kv_head"], :] = 7.0
    out, _ = oracle.paged_decode(inp["q"], inp["k_cache"], v, inp["block_table"], inp["seq_lens"], 0.25)
    b = g["batch"]
    for h in range(40):
        expect = 7.0 if h in g["q_heads"] else 0.0
        np.testing.assert_allclose(out[b * 40 + h], np.full(4, expect), atol=1e-13, rtol=0)


def test_empty_rows_zero_output_minus_inf_lse():
    """Rows with no visible key: zero output and -inf LSE (TokenSpeed SM107 section)."""
    wl, inp = tiny_decode(q_len=4, lens=(0, 2, 5), ps=4)
    out, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"])
    H = wl.num_q_heads
    # batch 0: n = 0, every row empty; batch 1: n = 2, tokens t = 0, 1 see nothing (2 - 4 + t + 1 <= 0)
    empty = list(range(0, 4 * H)) + [4 * H + t * H + h for t in range(2) for h in range(H)]
    assert np.all(out[empty] == 0) and np.all(np.isneginf(lse[empty]))
    rest = np.setdiff1d(np.arange(out.shape[0]), empty)
    assert np.all(np.isfinite(lse[rest]))


# ------------------------------------------------------------------- invariants

def test_page_permutation_invariance():
    """Physical page placement must not matter (PyPTO sections 5.2, 10.2)."""
    wl, inp = tiny_decode(lens=(13, 7, 16), ps=4, mapping="identity")
    base = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                               inp["seq_lens"], inp["scale"])
    P = inp["k_cache"].shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(11))
    inv = torch.empty_like(perm); inv[perm] = torch.arange(P)
    k2 = inp["k_cache"][perm]           # new page i holds old page perm[i]
    v2 = inp["v_cache"][perm]
    bt = inp["block_table"].clone()
    valid = bt >= 0
    bt[valid] = inv[bt[valid].long()].to(torch.int32)
    moved = oracle.paged_decode(inp["q"], k2, v2, bt, inp["seq_lens"], inp["scale"])
    np.testing.assert_array_equal(base[0], moved[0])
    np.testing.assert_array_equal(base[1], moved[1])


def test_gqa_equals_mha_with_repeated_kv_heads():
    wl, inp = tiny_decode(hq=6, hkv=2, lens=(5, 9, 3))
    out, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"])
    k_rep = inp["k_cache"].repeat_interleave(3, dim=2)
    v_rep = inp["v_cache"].repeat_interleave(3, dim=2)
    out2, lse2 = oracle.paged_decode(inp["q"], k_rep, v_rep, inp["block_table"], inp["seq_lens"],
                                     inp["scale"])
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_key_shift_moves_lse_only():
    """Adding one vector u to every key adds scale*<q,u> to each score of a row."""
    wl, inp = tiny_decode(lens=(6, 3, 10), d=8)
    g = torch.Generator().manual_seed(4)
    k = (torch.randint(-16, 16, inp["k_cache"].shape, generator=g) / 8.0).to(torch.bfloat16)
    u = (torch.randint(-8, 8, (8,), generator=g) / 4.0)
    k2 = (k.float() + u).to(torch.bfloat16)
    assert torch.equal(k2.float() - k.float(), u.expand_as(k.float()))   # exact in bf16
    o1, l1 = oracle.paged_decode(inp["q"], k, inp["v_cache"], inp["block_table"], inp["seq_lens"], 0.5)
    o2, l2 = oracle.paged_decode(inp["q"], k2, inp["v_cache"], inp["block_table"], inp["seq_lens"], 0.5)
    shift = 0.5 * (inp["q"][:, 0].double() @ u.double()).reshape(-1).numpy()
    np.testing.assert_allclose(o1, o2, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l2 - l1, shift, atol=1e-12, rtol=0)


def test_lse_bounds():
    wl, inp = tiny_decode(lens=(13, 2, 40), ps=8)
    _, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                 inp["seq_lens"], inp["scale"])
    G = wl.num_q_heads // wl.num_kv_heads
    for b in range(3):
        k, _ = dense_kv(inp, b)
        n = k.shape[0]
        for h in range(wl.num_q_heads):
            s = (k[:, h // G].double() @ inp["q"][b, 0, h].double()) * inp["scale"]
            m = float(s.max())
            assert m - 1e-12 <= lse[b * wl.num_q_heads + h] <= m + math.log(n) + 1e-12


def test_varlen_equals_each_sequence_alone():
    wl = PrefillWorkload("p", num_seqs=3, num_q_heads=4, num_kv_heads=2, head_dim_qk=8,
                         head_dim_v=8, causal=True, scale=0.4, value_seed=8)
    inp = make_prefill_inputs(wl, "cpu", [4, 6, 3])
    out, lse = oracle.varlen_prefill(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"],
                                     inp["cu_seqlens_k"], True, 0.4)
    cu = inp["cu_seqlens_q"].tolist()
    for i in range(3):
        a, b = cu[i], cu[i + 1]
        one = torch.tensor([0, b - a], dtype=torch.int32)
        o1, l1 = oracle.varlen_prefill(inp["q"][a:b], inp["k"][a:b], inp["v"][a:b], one, one, True, 0.4)
        np.testing.assert_array_equal(out[a * 4:b * 4], o1)
        np.testing.assert_array_equal(lse[a * 4:b * 4], l1)


def test_decode_equals_prefill_over_identity_pages():
    """Causal prefill with Lq = q_len over a sequence of n keys equals paged decode."""
    wl, inp = tiny_decode(q_len=3, lens=(9, 5, 12), ps=4, mapping="identity", hq=4, hkv=2)
    dec_o, dec_l = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                       inp["seq_lens"], inp["scale"])
    for b in range(3):
        k, v = dense_kv(inp, b)
        q = inp["q"][b]
        cq = torch.tensor([0, 3], dtype=torch.int32)
        ck = torch.tensor([0, k.shape[0]], dtype=torch.int32)
        o, l = oracle.varlen_prefill(q, k, v, cq, ck, True, inp["scale"])
        np.testing.assert_array_equal(dec_o[b * 12:(b + 1) * 12], o)
        np.testing.assert_array_equal(dec_l[b * 12:(b + 1) * 12], l)


def sdpa_masked_reference(inp, b, causal, window):
    """float64 SDPA over a dense gathered copy with an explicit boolean mask:
    token t's own position is pos = n - q_len + t; causal, it sees keys up to
    pos, otherwise all n; a window W starts the range at max(0, pos - W)."""
    q = inp["q"][b].double()
    k, v = dense_kv(inp, b)
    q_len, hq, _ = q.shape
    n, hkv = k.shape[0], k.shape[1]
    k = k.double().repeat_interleave(hq // hkv, dim=1)
    v = v.double().repeat_interleave(hq // hkv, dim=1)
    mask = torch.zeros(q_len, n, dtype=torch.bool)
    for t in range(q_len):
        pos = n - q_len + t
        hi = min(n, pos + 1) if causal else n
        lo = max(0, pos - window) if window >= 0 else 0
        mask[t, lo:max(lo, hi)] = True
    scores = torch.einsum("thd,nhd->htn", q, k) * inp["scale"]
    scores = scores.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(scores, dim=-1)
    p = torch.softmax(scores, dim=-1).nan_to_num(0.0)
    out = torch.einsum("htn,nhd->thd", p, v)
    return out.reshape(q_len * hq, -1).numpy(), lse.transpose(0, 1).reshape(-1).numpy()


@pytest.mark.parametrize("window", [-1, 0, 3, 7])
def test_noncausal_decode_matches_masked_sdpa(window):
    """TokenSpeed's non-causal decode: every token sees all n keys (a window
    still starts at its own position minus W); float64 reference built from
    the mask definition, GQA by repeat_interleave."""
    wl, inp = tiny_decode(q_len=3, lens=(9, 2, 14), hq=4, hkv=2, ps=4)
    out, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"], window_left=window, causal=False)
    for b in range(3):
        ref_o, ref_l = sdpa_masked_reference(inp, b, causal=False, window=window)
        np.testing.assert_allclose(out[b * 12:(b + 1) * 12], ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b * 12:(b + 1) * 12], ref_l, rtol=0, atol=1e-12)
    # the same mask builder reproduces the causal oracle (guards the builder itself)
    out_c, _ = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"], window_left=window)
    ref_c, _ = sdpa_masked_reference(inp, 0, causal=True, window=window)
    np.testing.assert_allclose(out_c[:12], ref_c, rtol=0, atol=1e-12)


def test_noncausal_decode_equals_noncausal_prefill_over_identity_pages():
    """Non-causal prefill with Lq = q_len over n keys equals non-causal paged decode."""
    wl, inp = tiny_decode(q_len=3, lens=(9, 5, 12), ps=4, mapping="identity", hq=4, hkv=2)
    dec_o, dec_l = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                       inp["seq_lens"], inp["scale"], causal=False)
    for b in range(3):
        k, v = dense_kv(inp, b)
        cq = torch.tensor([0, 3], dtype=torch.int32)
        ck = torch.tensor([0, k.shape[0]], dtype=torch.int32)
        o, l = oracle.varlen_prefill(inp["q"][b], k, v, cq, ck, False, inp["scale"])
        np.testing.assert_array_equal(dec_o[b * 12:(b + 1) * 12], o)
        np.testing.assert_array_equal(dec_l[b * 12:(b + 1) * 12], l)


def test_noncausal_equals_causal_at_one_token():
    wl, inp = tiny_decode(q_len=1, lens=(9, 1, 6))
    a = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"],
                            inp["scale"], causal=False)
    c = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"],
                            inp["scale"])
    np.testing.assert_array_equal(a[0], c[0])
    np.testing.assert_array_equal(a[1], c[1])


def test_latent_value_prefix_view():
    """V as the first Dv columns of the K rows (TokenSpeed decode, one KV cache)."""
    wl, inp = tiny_decode(hq=4, hkv=1, d=24, dv=16, lens=(7, 3, 9), latent=True)
    assert inp["v_cache"].data_ptr() == inp["k_cache"].data_ptr()
    out, _ = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                 inp["seq_lens"], inp["scale"])
    out2, _ = oracle.paged_decode(inp["q"], inp["k_cache"], inp["k_cache"][..., :16].contiguous(),
                                  inp["block_table"], inp["seq_lens"], inp["scale"])
    np.testing.assert_array_equal(out, out2)


def test_row_subset_matches_full():
    wl, inp = tiny_decode(lens=(5, 9, 2))
    full = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                               inp["seq_lens"], inp["scale"])
    rows = [23, 0, 7, 16]
    sub = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                              inp["seq_lens"], inp["scale"], rows=rows)
    np.testing.assert_array_equal(full[0][rows], sub[0])
    np.testing.assert_array_equal(full[1][rows], sub[1])


def test_oracle_rejects_out_of_range_page():
    wl, inp = tiny_decode(lens=(5, 9, 2))
    bt = inp["block_table"].clone()
    bt[1, 0] = 10_000
    with pytest.raises(ValueError):
        oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], bt, inp["seq_lens"], 1.0)


# ------------------------------------------- the pages' reformulations reach it

def _row_scores(inp, b, h):
    G = inp["q"].shape[2] // inp["k_cache"].shape[2]
    k, v = dense_kv(inp, b)
    s = (k[:, h // G].double() @ inp["q"][b, 0, h].double()).numpy() * inp["scale"]
    return s, v[:, h // G].double().numpy()


def online_softmax(s, v, block, threshold=None):
    """Flywheel section 1 recurrence (m, l, o per block); with `threshold` the
    base is kept unless the max rises by more than that many log2 units
    (TokenSpeed: 4 unsplit / 8 split)."""
    m, l, o = -math.inf, 0.0, np.zeros(v.shape[1])
    for a in range(0, len(s), block):
        sb, vb = s[a:a + block], v[a:a + block]
        m_new = max(m, float(sb.max()))
        if threshold is not None and m != -math.inf and (m_new - m) / math.log(2) <= threshold:
            m_new = m                                   # keep the stale base
        r = math.exp(m - m_new) if m != -math.inf else 0.0
        p = np.exp(sb - m_new)
        l = r * l + p.sum()
        o = r * o + p @ vb
        m = m_new
    return o / l, m + math.log(l)


@pytest.mark.parametrize("block", [1, 16, 512])
@pytest.mark.parametrize("threshold", [None, 4, 8])
def test_online_recurrence_equals_one_shot(block, threshold):
    wl, inp = tiny_decode(lens=(700, 129, 513), ps=128, d=16, hq=4, hkv=2, seed=21)
    out, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"])
    for b in range(3):
        for h in range(4):
            s, v = _row_scores(inp, b, h)
            o, l = online_softmax(s * 4.0, v, block, threshold)   # sharper scores stress the rescale
            o_ref, l_ref = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"],
                                               inp["block_table"], inp["seq_lens"],
                                               inp["scale"] * 4.0, rows=[b * 4 + h])
            np.testing.assert_allclose(o, o_ref[0], atol=1e-12, rtol=0)
            assert abs(l - l_ref[0]) < 1e-11


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8])
def test_split_kv_lse_merge_equals_one_shot(splits):
    """Split the keys, normalise each part, merge with weights exp(lse_i - L)."""
    wl, inp = tiny_decode(lens=(300, 41, 97), ps=16, d=16, hq=4, hkv=2, seed=22)
    out, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"])
    for b in range(3):
        for h in range(4):
            s, v = _row_scores(inp, b, h)
            edges = np.linspace(0, len(s), splits + 1).astype(int)
            parts = []
            for i in range(splits):
                sb, vb = s[edges[i]:edges[i + 1]], v[edges[i]:edges[i + 1]]
                if len(sb) == 0:
                    parts.append((np.zeros(v.shape[1]), -math.inf))
                    continue
                mb = sb.max()
                p = np.exp(sb - mb)
                parts.append((p @ vb / p.sum(), mb + math.log(p.sum())))
            L = max(pl for _, pl in parts)
            L = L + math.log(sum(math.exp(pl - L) for _, pl in parts))
            o = sum(math.exp(pl - L) * po for po, pl in parts)
            r = b * 4 + h
            np.testing.assert_allclose(o, out[r], atol=1e-12, rtol=0)
            assert abs(L - lse[r]) < 1e-12


def test_delayed_rescale_fifo_pipeline_equals_one_shot():
    """PyPTO sections 6.3, 8.1, 8.4: stacks of 512, PV collected two ticks later
    with the FIFO's pending0; the final O / l equals the one-shot result."""
    g = _golden("pypto_worked_examples.json")["rescale_fifo"]
    sched = planning.rescale_fifo_schedule(4)
    assert [list(x) for x in sched[:2]] == g["collections"]
    wl, inp = tiny_decode(lens=(1700, 513, 511), ps=128, d=16, hq=4, hkv=2, seed=23)
    for b in range(3):
        for h in (0, 3):
            s, v = _row_scores(inp, b, h)
            s = s * 3.0
            stacks = -(-len(s) // 512)
            m, l = -math.inf, 0.0
            pv, r = {}, {}
            o = np.zeros(v.shape[1])
            pending = [1.0, 1.0]
            for tick in range(stacks + 2):
                if tick >= 2:                      # consume(stack = tick - 2)
                    o = pending[0] * o + pv[tick - 2]
                if tick < stacks:                  # produce(stack = tick): softmax + PV numerator
                    sb = s[tick * 512:(tick + 1) * 512]
                    m_new = max(m, float(sb.max()))
                    r[tick] = math.exp(m - m_new) if m != -math.inf else 0.0
                    p = np.exp(sb - m_new)
                    l = r[tick] * l + p.sum()
                    m = m_new
                    pv[tick] = p @ v[tick * 512:(tick + 1) * 512]
                pending = [pending[1], r[tick] if tick < stacks else 1.0]
            o_ref, l_ref = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"],
                                               inp["block_table"], inp["seq_lens"],
                                               inp["scale"] * 3.0, rows=[b * 4 + h])
            np.testing.assert_allclose(o / l, o_ref[0], atol=1e-12, rtol=0)


# ---------------------------------------------------------- printed examples

def test_pypto_worked_examples():
    g = _golden("pypto_worked_examples.json")
    t = g["task_mapping"]
    assert planning.task_mapping(t["task"], t["num_kv_heads"], t["group"]) == (t["batch"], t["kv_head"], t["q_head_begin"])
    gr = g["granularity"]
    assert planning.page_count(gr["seq_len"], gr["page_size"]) == gr["pages"]
    assert planning.stack_count(gr["seq_len"], gr["stack_tokens"]) == gr["stacks"]
    assert planning.last_stack_tokens(gr["seq_len"], gr["stack_tokens"]) == gr["last_stack_valid_tokens"]
    gs = g["grid_stride"]
    n_tasks = gs["active_batch"] * gs["num_kv_heads"]
    for core, tasks in gs["tasks"].items():
        assert planning.grid_stride_tasks(int(core), n_tasks, gs["num_cores"]) == tasks
    two = gs["two_row_batch"]
    busy = [c for c in range(gs["num_cores"]) if planning.grid_stride_tasks(c, two["num_tasks"], gs["num_cores"])]
    assert len(busy) == two["busy_cores"]
    assert [c for c in range(gs["num_cores"]) if c not in busy] == two["idle_cores"]
    ring = g["ring"]
    assert ring["cores"] * ring["slots"] * ring["rows_per_slot"] == ring["rows"]


def test_tokenspeed_worked_examples():
    g = _golden("tokenspeed_worked_examples.json")
    f = g["fold"]
    F = planning.fold_factor(f["num_heads"], f["q_len"])
    assert F == f["F"] and f["num_heads"] * F == f["H_eff"] and f["q_len"] // F == f["q_len_eff"]
    for H, q_len, tiles in g["packed_q_tiles"]["cases"]:
        assert planning.packed_q_tiles(H, q_len) == tiles
    w = g["split_workspace"]
    assert planning.split_workspace_bytes(2, 128, 4, 1) == 0
    assert planning.split_workspace_bytes(2, 128, 4, 3) == 2 * 128 * 4 * 3 * w["floats_per_row_per_split_at_d512"] * 4
    # No factor above one divides q_len = 3 with H = 64 under 128 rows.
    assert planning.fold_factor(64, 3) == 1 and planning.fold_factor(16, 4) == 4


def test_flywheel_static_anchor_budget():
    g = _golden("flywheel_appendix_a.json")
    tau = planning.static_anchor_tau(g["n_keys"], g["v_max"], g["delta"], g["fp32_log_max"])
    assert round(tau) == g["tau_about"]
    assert round(tau - math.log(g["n_keys"])) == g["replay_margin_about"]
    # The refusal threshold is crossed only at N = exp(88.7 - ln Vmax - delta - 20) keys.
    n_star = math.exp(g["fp32_log_max"] - math.log(g["v_max"]) - g["delta"] - g["refuse_below"])
    assert planning.static_anchor_tau(n_star * 1.01) < g["refuse_below"] < planning.static_anchor_tau(n_star * 0.99)


# ------------------------------------------------------------ FP8 KV cache

def tiny_decode_fp8(batch=3, q_len=1, hq=8, hkv=2, d=32, ps=4, lens=(5, 1, 13), seed=13):
    wl = DecodeWorkload("t8", batch=batch, q_len=q_len, num_q_heads=hq, num_kv_heads=hkv,
                        head_dim_qk=d, head_dim_v=d, page_size=ps, scale=1.0 / math.sqrt(d),
                        seq_lens=tuple(lens), value_seed=seed, spare_pages=2, kv_fp8=True)
    return wl, make_decode_inputs(wl, "cpu")


def test_e4m3_decoding_matches_torch_for_every_byte():
    """The oracle's E4M3 decoder (written from the format definition) against
    torch's float8_e4m3fn conversion, all 256 codes, NaN codes included."""
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).tolist()
    for b in range(256):
        v = oracle.e4m3_to_double(b)
        assert (math.isnan(v) and math.isnan(ref[b])) or v == ref[b], b
    # closed forms: 1.0, the largest finite value, the smallest subnormal, NaN
    assert oracle.e4m3_to_double(0x38) == 1.0 and oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9 and oracle.e4m3_to_double(0xB8) == -1.0
    assert math.isnan(oracle.e4m3_to_double(0x7F)) and math.isnan(oracle.e4m3_to_double(0xFF))


def _dequantized_dense(inp, b, name, scale):
    """Row b's keys or values as float64: bytes gathered through the block
    table (plain indexing on the uint8 view), decoded by torch, times the scale."""
    n = int(inp["seq_lens"][b])
    ps = inp[name].shape[1]
    pages = [int(inp["block_table"][b, j // ps]) for j in range(n)]
    slots = [j % ps for j in range(n)]
    raw = inp[name].view(torch.uint8)[pages, slots]
    return raw.view(torch.float8_e4m3fn).to(torch.float64) * scale


@pytest.mark.parametrize("q_len,lens", [(1, (5, 1, 13)), (3, (7, 9, 12))])
def test_fp8_kv_decode_matches_sdpa_on_dequantized_copy(q_len, lens):
    wl, inp = tiny_decode_fp8(q_len=q_len, lens=lens)
    out, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"], k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    hq, hkv = wl.num_q_heads, wl.num_kv_heads
    for b in range(wl.batch):
        k = _dequantized_dense(inp, b, "k_cache", inp["k_scale"]).repeat_interleave(hq // hkv, dim=1)
        v = _dequantized_dense(inp, b, "v_cache", inp["v_scale"]).repeat_interleave(hq // hkv, dim=1)
        q = inp["q"][b].double()
        n = k.shape[0]
        mask = torch.zeros(q_len, n, dtype=torch.bool)
        for t in range(q_len):
            mask[t, : max(0, n - q_len + t + 1)] = True
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1), attn_mask=mask, scale=inp["scale"])
        sc = (torch.einsum("thd,nhd->htn", q, k) * inp["scale"]).masked_fill(~mask, float("-inf"))
        rows = slice(b * q_len * hq, (b + 1) * q_len * hq)
        np.testing.assert_allclose(out[rows], ref.transpose(0, 1).reshape(q_len * hq, -1).numpy(), atol=1e-12)
        np.testing.assert_allclose(lse[rows], torch.logsumexp(sc, -1).transpose(0, 1).reshape(-1).numpy(),
                                   atol=1e-12)


def test_fp8_scales_fold_into_score_scale_and_output():
    """k_scale multiplies every score like the softmax scale does; v_scale
    multiplies the output and leaves the LSE alone."""
    wl, inp = tiny_decode_fp8()
    args = (inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"])
    o1, l1 = oracle.paged_decode(*args, 0.3, k_scale=2.0, v_scale=1.0)
    o2, l2 = oracle.paged_decode(*args, 0.6, k_scale=1.0, v_scale=1.0)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)
    o3, l3 = oracle.paged_decode(*args, 0.3, k_scale=2.0, v_scale=3.0)
    np.testing.assert_allclose(o3, 3.0 * o1, atol=1e-12)
    np.testing.assert_allclose(l3, l1, atol=1e-12)


# ------------------------------------------------------------ sliding window
# "TokenSpeed-MLA 2.0.1", window_left: token t of a row with n keys sees keys
# max(0, n - q_len + t - W) .. n - q_len + t.

def _window_mask(q_len, n, window_left):
    mask = torch.zeros(q_len, n, dtype=torch.bool)
    for t in range(q_len):
        hi = n - q_len + t                         # last visible key (bottom-right causal)
        if hi < 0:
            continue
        lo = max(0, hi - window_left)
        mask[t, lo:hi + 1] = True
    return mask


@pytest.mark.parametrize("q_len,lens,ps,window", [
    (1, (5, 1, 13), 4, 0), (1, (16, 17, 3), 8, 3), (2, (9, 30, 2), 4, 7), (4, (20, 6, 33), 8, 5),
    (3, (40, 41, 12), 16, 16)])
def test_window_matches_sdpa_on_dense_copy(q_len, lens, ps, window):
    wl, inp = tiny_decode(q_len=q_len, lens=lens, ps=ps, seed=17)
    out, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"], window_left=window)
    hq, hkv = wl.num_q_heads, wl.num_kv_heads
    for b in range(wl.batch):
        k, v = dense_kv(inp, b)
        n = k.shape[0]
        q = inp["q"][b].double()
        k = k.double().repeat_interleave(hq // hkv, dim=1)
        v = v.double().repeat_interleave(hq // hkv, dim=1)
        mask = _window_mask(q_len, n, window)
        sc = (torch.einsum("thd,nhd->htn", q, k) * inp["scale"]).masked_fill(~mask, float("-inf"))
        w = torch.softmax(sc, -1).nan_to_num(0.0)  # rows with no visible key: zero output
        ref = torch.einsum("htn,nhd->thd", w, v).reshape(q_len * hq, -1).numpy()
        rows = slice(b * q_len * hq, (b + 1) * q_len * hq)
        np.testing.assert_allclose(out[rows], ref, atol=1e-12)
        np.testing.assert_allclose(lse[rows], torch.logsumexp(sc, -1).transpose(0, 1).reshape(-1).numpy(),
                                   atol=1e-12)


def test_window_zero_sees_own_position_only():
    """W = 0: token t sees exactly key n - q_len + t, so out = that value row
    and lse = that score (closed form)."""
    wl, inp = tiny_decode(q_len=3, lens=(7, 12, 5), ps=4, seed=19)
    out, lse = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                   inp["seq_lens"], inp["scale"], window_left=0)
    G = wl.num_q_heads // wl.num_kv_heads
    for b in range(wl.batch):
        k, v = dense_kv(inp, b)
        n = k.shape[0]
        for t in range(wl.q_len):
            j = n - wl.q_len + t
            for h in range(wl.num_q_heads):
                r = (b * wl.q_len + t) * wl.num_q_heads + h
                np.testing.assert_allclose(out[r], v[j, h // G].double().numpy(), atol=1e-12)
                s = inp["scale"] * float((inp["q"][b, t, h].double() * k[j, h // G].double()).sum())
                assert abs(lse[r] - s) < 1e-12


def test_window_wider_than_row_is_no_window():
    wl, inp = tiny_decode(q_len=2, lens=(9, 30, 2), ps=4, seed=21)
    args = (inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"], inp["scale"])
    o0, l0 = oracle.paged_decode(*args)
    o1, l1 = oracle.paged_decode(*args, window_left=30)
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)


def test_window_never_reads_pages_before_it():
    """Pages wholly before every token's window may be evicted: their table
    entries can hold anything and their contents NaN (a cache that drops keys
    leaving the window)."""
    wl, inp = tiny_decode(q_len=2, lens=(40, 37, 9), ps=4, seed=23)
    W = 6
    args = (inp["q"], inp["k_cache"], inp["v_cache"])
    o0, l0 = oracle.paged_decode(*args, inp["block_table"], inp["seq_lens"], inp["scale"], window_left=W)
    bt = inp["block_table"].clone()
    kc, vc = inp["k_cache"].clone(), inp["v_cache"].clone()
    for b in range(wl.batch):
        n = int(inp["seq_lens"][b])
        first = max(0, n - wl.q_len - W)           # smallest lower bound of the row
        for pg in range(first // wl.page_size):
            kc[int(bt[b, pg])] = float("nan")
            vc[int(bt[b, pg])] = float("nan")
        for pg in range(first // wl.page_size):
            bt[b, pg] = -1
    o1, l1 = oracle.paged_decode(inp["q"], kc, vc, bt, inp["seq_lens"], inp["scale"], window_left=W)
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)


# ----------------------------------------------------------------- KV append
# "Writing Page Attention with PyPTO", section 4.3: row (b, t) goes to cache
# token row layer_base + max(slot, 0); a cache canary shows only those rows
# change (section 10.2).

def test_e4m3_encoding_round_trips_every_code_and_matches_torch():
    for code in range(256):
        if (code & 0x7F) == 0x7F:
            continue                                  # NaN patterns
        x = oracle.e4m3_to_double(code)
        assert oracle.e4m3_from_float(x) == code, hex(code)
    g = torch.Generator().manual_seed(3)
    xs = torch.cat([torch.randn(4000, generator=g) * 40, torch.randn(1000, generator=g) * 0.01])
    # midpoints between neighbouring codes: ties go to the even code
    mids = [(oracle.e4m3_to_double(c) + oracle.e4m3_to_double(c + 1)) / 2 for c in range(0, 0x7E)]
    xs = torch.cat([xs, torch.tensor(mids, dtype=torch.float32), -torch.tensor(mids, dtype=torch.float32)])
    ref = xs.to(torch.float8_e4m3fn).view(torch.uint8)
    for x, r in zip(xs.tolist(), ref.tolist()):
        assert oracle.e4m3_from_float(x) == r, x
    for x, code in ((448.0, 0x7E), (460.0, 0x7E), (1e30, 0x7E), (float("inf"), 0x7E), (-1e30, 0xFE)):
        assert oracle.e4m3_from_float(x) == code


def _append_case(q_len=2, fp8=False, seed=5):
    wl, inp = tiny_decode(batch=3, q_len=q_len, hq=8, hkv=2, d=32, ps=4, lens=(7, 12, 5), seed=seed)
    g = torch.Generator().manual_seed(seed + 100)
    k_new = torch.randn(3, q_len, 2, 32, generator=g).to(torch.bfloat16)
    v_new = torch.randn(3, q_len, 2, 32, generator=g).to(torch.bfloat16)
    kc, vc = inp["k_cache"], inp["v_cache"]
    if fp8:
        kc = (kc.float().nan_to_num(0.0) / 0.05).clamp(-448, 448).to(torch.float8_e4m3fn)
        vc = (vc.float().nan_to_num(0.0) / 0.05).clamp(-448, 448).to(torch.float8_e4m3fn)
    return wl, inp, k_new, v_new, kc, vc


@pytest.mark.parametrize("fp8", [False, True])
def test_append_changes_only_the_addressed_rows(fp8):
    wl, inp, k_new, v_new, kc, vc = _append_case(fp8=fp8)
    ps, P = kc.shape[1], kc.shape[0]
    slots = torch.tensor([3, 17, 20, 9, 30, 1], dtype=torch.int32)
    kc2, vc2 = oracle.kv_append(k_new, v_new, slots, 4, kc, vc, k_scale=0.05, v_scale=0.05)
    raw = (lambda t: t.view(torch.uint8)) if fp8 else (lambda t: t.view(torch.int16))
    changed = (raw(kc2) != raw(kc)).flatten(2).any(-1) | (raw(vc2) != raw(vc)).flatten(2).any(-1)
    rows = {int(4 + s) for s in slots}
    for page in range(P):
        for off in range(ps):
            if page * ps + off not in rows:
                assert not changed[page, off].any(), (page, off)
    for i, s in enumerate(slots.tolist()):
        b, t = divmod(i, wl.q_len)
        page, off = divmod(4 + s, ps)
        if fp8:
            want_k = (k_new[b, t].float() / 0.05).to(torch.float8_e4m3fn).view(torch.uint8)
            assert torch.equal(kc2[page, off].view(torch.uint8), want_k)
        else:
            assert torch.equal(kc2[page, off], k_new[b, t])
            assert torch.equal(vc2[page, off], v_new[b, t])


def test_warmup_slot_is_clamped_before_the_layer_base():
    """Slot -1 with a nonzero layer base writes the layer's row 0, never the
    previous layer's last row (section 4.3 and the test note of section 10.2)."""
    wl, inp, k_new, v_new, kc, vc = _append_case(q_len=1)
    base = 8
    slots = torch.tensor([-1, 5, -1], dtype=torch.int32)
    kc2, vc2 = oracle.kv_append(k_new, v_new, slots, base, kc, vc)
    ps = kc.shape[1]
    prev_page, prev_off = divmod(base - 1, ps)
    assert torch.equal(kc2[prev_page, prev_off].view(torch.int16), kc[prev_page, prev_off].view(torch.int16))
    page, off = divmod(base, ps)
    assert torch.equal(kc2[page, off], k_new[2, 0])     # the last of the two -1 writers
    page, off = divmod(base + 5, ps)
    assert torch.equal(vc2[page, off], v_new[1, 0])


def test_append_then_decode_matches_sdpa_with_the_new_keys():
    """New tokens appended at each row's last q_len positions are the keys the
    decode then attends to: equal to SDPA on the dense copy with those rows."""
    wl, inp, k_new, v_new, kc, vc = _append_case(q_len=2, seed=9)
    ps = kc.shape[1]
    lens = inp["seq_lens"]
    slots = []
    for b in range(wl.batch):
        for t in range(wl.q_len):
            pos = int(lens[b]) - wl.q_len + t
            slots.append(int(inp["block_table"][b, pos // ps]) * ps + pos % ps)
    kc2, vc2 = oracle.kv_append(k_new, v_new, torch.tensor(slots, dtype=torch.int32), 0, kc, vc)
    inp2 = dict(inp)
    inp2["k_cache"], inp2["v_cache"] = kc2, vc2
    out, lse = oracle.paged_decode(inp2["q"], kc2, vc2, inp["block_table"], lens, inp["scale"])
    for b in range(wl.batch):
        ref_o, ref_l = sdpa_decode_reference(inp2, b)
        k_dense, _ = dense_kv(inp2, b)
        n = int(lens[b])
        assert torch.equal(k_dense[n - wl.q_len:], k_new[b])
        rows = slice(b * wl.q_len * wl.num_q_heads, (b + 1) * wl.q_len * wl.num_q_heads)
        np.testing.assert_allclose(out[rows], ref_o, atol=1e-12)
        np.testing.assert_allclose(lse[rows], ref_l, atol=1e-12)


# ------------------------------------------- the error-bound scale (absv)
# absv = sum_j p_j |v_j| / l: the same softmax weights applied to |v|.  The
# GPU tests scale their bound for rounding P to BF16 ("Writing Page Attention
# with PyPTO", section 6.3) by it, so it is pinned like the output itself.

@pytest.mark.parametrize("q_len,lens,ps,mapping", [
    (1, (5, 1, 13), 4, "random"),
    (3, (7, 9, 12), 4, "reverse"),
])
def test_absv_matches_sdpa_on_absolute_values(q_len, lens, ps, mapping):
    wl, inp = tiny_decode(q_len=q_len, lens=lens, ps=ps, mapping=mapping)
    out, lse, absv = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                         inp["seq_lens"], inp["scale"], with_absv=True)
    inp_abs = dict(inp, v_cache=inp["v_cache"].abs())
    rows_per_b = q_len * wl.num_q_heads
    for b in range(wl.batch):
        ref_o, _ = sdpa_decode_reference(inp_abs, b)
        np.testing.assert_allclose(absv[b * rows_per_b:(b + 1) * rows_per_b], ref_o, rtol=0, atol=1e-12)
    # Asking for absv changes nothing else.
    o2, l2 = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                 inp["seq_lens"], inp["scale"])
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)
    assert np.all(absv >= np.abs(out) - 1e-12)                  # |sum p v| <= sum p |v|


def test_absv_closed_forms():
    """Non-negative values: absv = out; one key: absv = |that value row|; a
    row with no key: 0."""
    wl, inp = tiny_decode(lens=(5, 1, 0))
    inp_pos = dict(inp, v_cache=inp["v_cache"].abs())
    out, _, absv = oracle.paged_decode(inp_pos["q"], inp_pos["k_cache"], inp_pos["v_cache"], inp["block_table"],
                                       inp["seq_lens"], inp["scale"], with_absv=True)
    fin = np.isfinite(out)
    np.testing.assert_allclose(absv[fin], out[fin], rtol=0, atol=1e-12)
    _, _, absv = oracle.paged_decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                     inp["seq_lens"], inp["scale"], with_absv=True)
    k, v = dense_kv(inp, 1)                                     # batch row 1 holds one key
    hq, hkv = wl.num_q_heads, wl.num_kv_heads
    for h in range(hq):
        np.testing.assert_array_equal(absv[hq + h], v[0, h // (hq // hkv)].double().abs().numpy())
    assert np.all(absv[2 * hq:] == 0.0)


def test_absv_prefill_and_fp8_match_sdpa_on_absolute_values():
    wl = PrefillWorkload("p", num_seqs=2, num_q_heads=4, num_kv_heads=2, head_dim_qk=16,
                         head_dim_v=8, causal=True, scale=0.3, value_seed=5)
    inp = make_prefill_inputs(wl, "cpu", [5, 9], [7, 9])
    _, _, absv = oracle.varlen_prefill(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"],
                                       inp["cu_seqlens_k"], True, wl.scale, with_absv=True)
    q = inp["q"][:5].double().transpose(0, 1)
    k = inp["k"][:7].double().repeat_interleave(2, dim=1).transpose(0, 1)
    v = inp["v"][:7].double().abs().repeat_interleave(2, dim=1).transpose(0, 1)
    mask = torch.ones(5, 7, dtype=torch.bool).tril(diagonal=2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=wl.scale)
    np.testing.assert_allclose(absv[:20], ref.transpose(0, 1).reshape(20, -1).numpy(), rtol=0, atol=1e-12)

    wl8, inp8 = tiny_decode_fp8()
    _, _, absv8 = oracle.paged_decode(inp8["q"], inp8["k_cache"], inp8["v_cache"], inp8["block_table"],
                                      inp8["seq_lens"], inp8["scale"], k_scale=inp8["k_scale"],
                                      v_scale=inp8["v_scale"], with_absv=True)
    hq, hkv = wl8.num_q_heads, wl8.num_kv_heads
    for b in range(wl8.batch):
        kk = _dequantized_dense(inp8, b, "k_cache", inp8["k_scale"]).repeat_interleave(hq // hkv, dim=1)
        vv = _dequantized_dense(inp8, b, "v_cache", inp8["v_scale"]).abs().repeat_interleave(hq // hkv, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            inp8["q"][b].double().transpose(0, 1), kk.transpose(0, 1), vv.transpose(0, 1), scale=inp8["scale"])
        np.testing.assert_allclose(absv8[b * hq:(b + 1) * hq], ref.transpose(0, 1).reshape(hq, -1).numpy(),
                                   rtol=0, atol=1e-12)
