"""KV-cache append on the GPU, standalone and fused into the decode, against
the fp64 oracle ("Writing Page Attention with PyPTO", sections 4.2-4.3 and
10.2: token (b, t) goes to cache token row layer_base + max(slot, 0); a cache
canary shows nothing else changes; a nonzero layer base with the warm-up slot
-1 stays inside the layer).

The appended caches are compared byte for byte with the oracle's (BF16 bits,
or E4M3 codes of x / scale); the fused append + decode is compared with the
oracle's append followed by its decode of the layer, on a packed two-layer
cache, for BF16 and FP8 caches, with and without a sliding window.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from ragged_softmax_attention_gb300.workloads import WORKLOADS, DecodeWorkload, make_decode_inputs
from tests.gpu_common import BF16_UNIT, FP16_UNIT, built_library, compare, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fw():
    lib = built_library()
    lib.set_option(lib.FW_OPT_DECODE_CHUNK_TOKENS, 0)
    yield lib
    lib.set_option(lib.FW_OPT_DECODE_CHUNK_TOKENS, 0)


def raw(t):
    return t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t.view(torch.int16)


def new_rows(B, q_len, hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    k = (torch.randn(B, q_len, hkv, d, generator=g) * 3).to(torch.bfloat16)
    v = (torch.randn(B, q_len, hkv, d, generator=g) * 3).to(torch.bfloat16)
    return k, v


def caches(P, ps, hkv, d, fp8, seed):
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn(P, ps, hkv, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(P, ps, hkv, d, generator=g).to(torch.bfloat16)
    if fp8:
        kc, vc = (kc.float() * 20).to(torch.float8_e4m3fn), (vc.float() * 20).to(torch.float8_e4m3fn)
    return kc, vc


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("d,ps", [(128, 16), (128, 128), (256, 64)])
def test_append_matches_oracle_bytewise(fw, fp8, d, ps):
    if fp8 and d != 128:
        pytest.skip("FP8 caches are served at head dim 128")
    B, q_len, hkv, P = 5, 3, 4, 40
    k_new, v_new = new_rows(B, q_len, hkv, d, seed=d + ps)
    kc, vc = caches(P, ps, hkv, d, fp8, seed=7)
    base = 8 * ps
    slots = torch.randperm(P * ps - base, generator=torch.Generator().manual_seed(3))[:B * q_len].to(torch.int32)
    ks, vs = (0.013, 0.021) if fp8 else (1.0, 1.0)
    ref_k, ref_v = oracle.kv_append(k_new, v_new, slots, base, kc, vc, k_scale=ks, v_scale=vs)
    dk, dv = kc.cuda(), vc.cuda()
    fw.kv_append(k_new.cuda(), v_new.cuda(), slots.cuda(), base, dk, dv, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    assert torch.equal(raw(dk.cpu()), raw(ref_k))
    assert torch.equal(raw(dv.cpu()), raw(ref_v))


def test_fp8_append_rounding_edges(fw):
    """Values at E4M3 midpoints (ties to even), beyond 448 (saturation), tiny
    values flushing to signed zero: the stored codes equal the oracle's."""
    B, q_len, hkv, d, ps, P = 2, 1, 1, 128, 16, 4
    mids = [(oracle.e4m3_to_double(c) + oracle.e4m3_to_double(c + 1)) / 2 for c in range(0, 0x7E)]
    vals = mids[:120] + [500.0, -1e4, 1e-30, -1e-30, 448.0, -448.0, 0.0, -0.0]
    x = torch.tensor(vals[:d] + [1.0] * max(0, d - len(vals)), dtype=torch.float32).to(torch.bfloat16)
    k_new = x.view(1, 1, 1, d).repeat(B, q_len, hkv, 1).contiguous()
    v_new = (-k_new).contiguous()
    kc, vc = caches(P, ps, hkv, d, True, seed=9)
    slots = torch.tensor([5, 40], dtype=torch.int32)
    ref_k, ref_v = oracle.kv_append(k_new, v_new, slots, 0, kc, vc, k_scale=1.0, v_scale=1.0)
    dk, dv = kc.cuda(), vc.cuda()
    fw.kv_append(k_new.cuda(), v_new.cuda(), slots.cuda(), 0, dk, dv, k_scale=1.0, v_scale=1.0)
    torch.cuda.synchronize()
    assert torch.equal(raw(dk.cpu()), raw(ref_k))
    assert torch.equal(raw(dv.cpu()), raw(ref_v))


def test_warmup_slots_stay_inside_the_layer(fw):
    """Slot -1 with a nonzero layer base: the layer's row 0 holds the warm-up
    tokens' values (each 16-byte group from one of them, the writers race);
    the previous layer's last row and every other row keep their bytes."""
    B, q_len, hkv, d, ps, P = 4, 1, 2, 128, 16, 20
    k_new, v_new = new_rows(B, q_len, hkv, d, seed=11)
    kc, vc = caches(P, ps, hkv, d, False, seed=12)
    base = 5 * ps
    slots = torch.tensor([-1, 7, -1, 30], dtype=torch.int32)
    dk, dv = kc.cuda(), vc.cuda()
    fw.kv_append(k_new.cuda(), v_new.cuda(), slots.cuda(), base, dk, dv)
    torch.cuda.synchronize()
    dk, dv = dk.cpu(), dv.cpu()
    p0, o0 = divmod(base, ps)
    for got, new in ((dk[p0, o0], k_new), (dv[p0, o0], v_new)):
        g = got.view(hkv, d // 8, 8)
        a, b2 = new[0, 0].view(hkv, d // 8, 8), new[2, 0].view(hkv, d // 8, 8)
        same = (g == a).all(-1) | (g == b2).all(-1)
        assert same.all(), "a 16-byte group of the warm-up row comes from neither warm-up token"
    # every row but the warm-up row: exactly the oracle's result without the repeat
    ref_k, ref_v = oracle.kv_append(k_new, v_new, slots, base, kc, vc)
    mask = torch.ones(P, ps, dtype=torch.bool)
    mask[p0, o0] = False
    assert torch.equal(raw(dk)[mask], raw(ref_k)[mask])
    assert torch.equal(raw(dv)[mask], raw(ref_v)[mask])


def test_slot_outside_the_cache_is_reported_and_skipped(fw):
    B, q_len, hkv, d, ps, P = 2, 1, 2, 128, 16, 6
    k_new, v_new = new_rows(B, q_len, hkv, d, seed=13)
    kc, vc = caches(P, ps, hkv, d, False, seed=14)
    slots = torch.tensor([3, P * ps], dtype=torch.int32)      # the second is one row past the end
    dk, dv = kc.cuda(), vc.cuda()
    fw.kv_append(k_new.cuda(), v_new.cuda(), slots.cuda(), 0, dk, dv)
    torch.cuda.synchronize()
    assert fw.device_status() == 1                           # FW_ERR_INVALID_ARG
    ref_k, ref_v = oracle.kv_append(k_new[:1], v_new[:1], slots[:1], 0, kc, vc)
    assert torch.equal(raw(dk.cpu()), raw(ref_k))
    assert torch.equal(raw(dv.cpu()), raw(ref_v))


def test_latent_keys_only(fw):
    """A latent cache (576-wide keys, values a view of them): append keys only."""
    B, q_len, d, ps, P = 3, 2, 576, 64, 8
    k_new, _ = new_rows(B, q_len, 1, d, seed=15)
    kc, _ = caches(P, ps, 1, d, False, seed=16)
    slots = torch.tensor([0, 1, 100, 101, 300, 511], dtype=torch.int32)
    dk = kc.cuda()
    fw.kv_append(k_new.cuda(), None, slots.cuda(), 0, dk, None)
    torch.cuda.synchronize()
    ref = kc.clone()
    for i, s in enumerate(slots.tolist()):
        b, t = divmod(i, q_len)
        ref[s // ps, s % ps] = k_new[b, t]
    assert torch.equal(raw(dk.cpu()), raw(ref))


def _layer_case(wl, fp8, seed):
    """A packed two-layer cache: layer 0 then layer 1 (the decoded one), each
    with its own pages; new tokens at each row's last q_len positions."""
    inp = make_decode_inputs(wl, "cpu")
    kl, vl = inp["k_cache"], inp["v_cache"]
    P, ps = kl.shape[0], kl.shape[1]
    k0, v0 = caches(P, ps, wl.num_kv_heads, wl.head_dim_qk, fp8, seed=seed)
    if fp8:
        kl, vl = k0.clone(), v0.clone()                      # finite E4M3 layer contents
    kp = torch.cat([k0, kl]).contiguous()
    vp = torch.cat([v0, vl]).contiguous()
    base = P * ps
    k_new, v_new = new_rows(wl.batch, wl.q_len, wl.num_kv_heads, wl.head_dim_qk, seed=seed + 1)
    lens = inp["seq_lens"]
    slots = []
    for b in range(wl.batch):
        for t in range(wl.q_len):
            pos = int(lens[b]) - wl.q_len + t
            slots.append(int(inp["block_table"][b, pos // ps]) * ps + pos % ps if pos >= 0 else -1)
    return inp, kp, vp, base, k_new, v_new, torch.tensor(slots, dtype=torch.int32)


@pytest.mark.parametrize("fp8,window", [(False, -1), (False, 50), (True, -1), (True, 50)])
@pytest.mark.parametrize("q_len", [1, 3])
def test_fused_append_then_decode(fw, fp8, window, q_len):
    wl = DecodeWorkload("app", batch=4, q_len=q_len, num_q_heads=8, num_kv_heads=2, head_dim_qk=128,
                        head_dim_v=128, page_size=16, scale=1.0 / math.sqrt(128), seq_lens=(3, 129, 300, 1029),
                        kv_fp8=fp8, value_seed=71, spare_pages=3)
    inp, kp, vp, base, k_new, v_new, slots = _layer_case(wl, fp8, seed=31)
    ks, vs = (0.02, 0.02) if fp8 else (1.0, 1.0)
    ref_k, ref_v = oracle.kv_append(k_new, v_new, slots, base, kp, vp, k_scale=ks, v_scale=vs)
    P = inp["k_cache"].shape[0]
    ref_o, ref_l, ref_a = oracle.paged_decode(inp["q"], ref_k[P:], ref_v[P:], inp["block_table"], inp["seq_lens"],
                                              inp["scale"], k_scale=ks, v_scale=vs, window_left=window, with_absv=True)
    dk, dv = kp.cuda(), vp.cuda()
    d = to_device(inp)
    out, lse = fw.paged_decode_append(d["q"], k_new.cuda(), v_new.cuda(), slots.cuda(), base, dk, dv,
                                      d["block_table"], d["seq_lens"], d["scale"], k_scale=ks, v_scale=vs,
                                      window_left=window)
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    assert torch.equal(raw(dk.cpu()), raw(ref_k))            # layer 0 untouched, layer 1 appended
    assert torch.equal(raw(dv.cpu()), raw(ref_v))
    compare(out, lse, ref_o, ref_l, what=f"fused append fp8={fp8} window={window} q_len={q_len}", absv=ref_a,
            p_unit=FP16_UNIT if fp8 else BF16_UNIT)


def test_fused_append_argument_checks_launch_nothing(fw):
    wl = DecodeWorkload("app", batch=2, q_len=1, num_q_heads=8, num_kv_heads=2, head_dim_qk=128,
                        head_dim_v=128, page_size=16, scale=0.1, seq_lens=(30, 40), value_seed=3, spare_pages=2)
    inp, kp, vp, base, k_new, v_new, slots = _layer_case(wl, False, seed=41)
    d = to_device(inp)
    dk, dv = kp.cuda(), vp.cuda()
    args = (d["q"], k_new.cuda(), v_new.cuda(), slots.cuda())
    rest = (dk, dv, d["block_table"], d["seq_lens"], d["scale"])
    before = fw.launch_count()
    with pytest.raises(fw.FwError):                            # base not a multiple of the page size
        fw.paged_decode_append(*args, base + 3, *rest)
    with pytest.raises(fw.FwError):                            # base outside the cache
        fw.paged_decode_append(*args, 10 ** 9, *rest)
    with pytest.raises(fw.FwError):                            # BF16 cache with a scale
        fw.paged_decode_append(*args, base, *rest, k_scale=2.0)
    with pytest.raises(fw.FwError):                            # slot_mapping of the wrong length
        fw.paged_decode_append(d["q"], k_new.cuda(), v_new.cuda(), slots[:1].cuda(), base, *rest)
    assert fw.launch_count() == before
    assert torch.equal(raw(dk.cpu()), raw(kp))


def test_fused_append_full_size_qwen3(fw):
    """The Qwen3-14B-shaped decode with its new token appended by the fused
    call (a packed two-layer cache would double 4.4 GB; here the layer is the
    whole cache, base 0): the appended rows equal the new tokens and sampled
    rows match the oracle's decode of the updated cache."""
    wl = WORKLOADS["qwen3_14b_paged_decode"]
    d = make_decode_inputs(wl, "cuda")
    ps = wl.page_size
    lens, bt = d["seq_lens"].cpu(), d["block_table"].cpu()
    slots = torch.tensor([int(bt[b, (int(lens[b]) - 1) // ps]) * ps + (int(lens[b]) - 1) % ps
                          for b in range(wl.batch)], dtype=torch.int32)
    k_new, v_new = new_rows(wl.batch, 1, wl.num_kv_heads, 128, seed=77)
    out, lse = fw.paged_decode_append(d["q"], k_new.cuda(), v_new.cuda(), slots.cuda(), 0, d["k_cache"],
                                      d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    g = torch.Generator().manual_seed(5)
    for b in torch.randperm(wl.batch, generator=g)[:8].tolist():
        s = int(slots[b])
        assert torch.equal(d["k_cache"][s // ps, s % ps].cpu(), k_new[b, 0])
        npg = -(-int(lens[b]) // ps)
        pages = bt[b, :npg].long()
        k = d["k_cache"][pages.cuda()].cpu()
        v = d["v_cache"][pages.cuda()].cpu()
        sub_bt = torch.arange(npg, dtype=torch.int32).unsqueeze(0)
        heads = torch.randperm(wl.num_q_heads, generator=g)[:4].tolist()
        o_ref, l_ref, a_ref = oracle.paged_decode(d["q"][b:b + 1].cpu(), k, v, sub_bt, lens[b:b + 1], wl.scale, rows=heads, with_absv=True)
        compare(out[b, 0, heads], lse[b, 0, heads], o_ref, l_ref, f"b{b}", absv=a_ref)
