"""Pins of the oracle's KV slots, window visibility and attention (CPU only).

The decode-step attention is brute-forced against a second formulation: the cache
writes are simulated position by position to find which position each slot holds,
an explicit 0/1 mask is built from the window definition, and numpy computes the
softmax over the masked logits.
"""
import numpy as np
import pytest
import torch

from quantized_attention_layer_gb300 import workloads as wl


def test_ring_slot_arithmetic_brute_force(orc):
    for C in (1, 3, 8):
        owner = {}
        for P in range(3 * C):
            owner[P % C] = P                       # simulate the ring writes
            assert orc.kv_slot(P, C, True) == P % C
            for s in range(C):
                assert orc.slot_position(s, P, C, True) == owner.get(s, -1)
    for C in (5, 16):
        for P in range(C):
            assert orc.kv_slot(P, C, False) == P
            for s in range(C):
                assert orc.slot_position(s, P, C, False) == (s if s <= P else -1)


def test_visible_key_count_matches_the_kv_seq_len_rule(orc):
    # gemma4/gpu_full_attn.rs, "Dense flash_attn_vec": a ring of capacity = window
    # attends to min(seq_pos + 1, capacity) entries; a global layer to seq_pos + 1.
    for W in (1, 4, 7):
        for P in range(30):
            n_sl = sum(orc.key_visible(p, P, True, W) for p in range(-3, P + 5))
            n_full = sum(orc.key_visible(p, P, False, W) for p in range(-3, P + 5))
            assert n_sl == min(P + 1, W)
            assert n_full == P + 1


def _tiny(layer_type, C, W, ring, hd=16, nh=2, nkv=1, softcap=0.0, seed=100):
    return wl.Workload(name="tiny", hidden=64, num_heads=nh, num_kv_heads=nkv, head_dim=hd,
                       layer_type=layer_type, window=W, kv_capacity=C, ring=ring, batch=1,
                       rope_theta=1e4, seed=seed, seq_pos=0, softcap=softcap)


def _explicit_mask_attention(w, q, kc, vc, P):
    """Second formulation: simulate writes, explicit mask, numpy softmax."""
    C, hd, g = w.kv_capacity, w.head_dim, w.group
    owner = np.full(C, -1)
    for p in range(P + 1):
        owner[p % C if w.ring else p] = p
    sliding = w.layer_type == wl.SLIDING
    mask = np.array([owner[s] >= 0 and owner[s] <= P and (not sliding or owner[s] > P - w.window)
                     for s in range(C)])
    K = orc_bf16(kc)[0]
    V = orc_bf16(vc)[0]
    o = np.empty((w.num_heads, hd))
    for h in range(w.num_heads):
        s = w.attn_scale * (K[h // g] @ q[h])
        if w.softcap > 0:
            s = w.softcap * np.tanh(s / w.softcap)
        s = np.where(mask, s, -np.inf)
        p = np.exp(s - s.max())
        o[h] = (p / p.sum()) @ V[h // g]
    return o


def orc_bf16(bits):
    import oracle
    return oracle.bf16_to_f64(bits)


@pytest.mark.parametrize("layer_type,ring", [(wl.SLIDING, False), (wl.SLIDING, True),
                                             (wl.FULL, False)])
def test_decode_attention_brute_force_mask(orc, layer_type, ring):
    for C in (4, 8, 16):
        for W in ((1, 2, 3, C) if layer_type == wl.SLIDING else (0,)):
            if ring and W != C:
                continue
            w = _tiny(layer_type, C, W, ring, seed=C * 10 + W)
            weights = wl.make_weights(w)
            kv = wl.make_kv_cache(w)
            x = wl.make_x(w)
            for P in range(0, (3 * C) if ring else C):
                r = orc.decode_step(w, weights, x, [P], kv["k_cache"], kv["v_cache"])
                ref = _explicit_mask_attention(w, r["q"][0], r["k_cache"], r["v_cache"], P)
                assert np.max(np.abs(r["attn"][0] - ref)) <= 1e-12, (C, W, P)


def test_attend_weights_sum_to_one_and_one_key_returns_v(orc):
    rng = np.random.default_rng(0)
    hd, n = 16, 11
    K = torch.randn(n, hd, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    V = torch.randn(n, hd, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    q = rng.normal(size=hd) * 3
    o, wts = orc.attend(q, K, V, np.arange(n))
    assert abs(wts.sum() - 1.0) <= 1e-14 and np.all(wts > 0)
    o1, w1 = orc.attend(q, K, V, [7])
    assert w1[0] == 1.0
    assert np.array_equal(o1, V[7].to(torch.float64).numpy())


def test_attend_is_invariant_to_slot_order(orc):
    rng = np.random.default_rng(5)
    hd, n = 32, 40
    K = torch.randn(n, hd, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    V = torch.randn(n, hd, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    q = rng.normal(size=hd)
    rows = np.arange(0, n, 2)
    o1, _ = orc.attend(q, K, V, rows)
    o2, _ = orc.attend(q, K, V, rng.permutation(rows))
    assert np.max(np.abs(o1 - o2)) <= 1e-14


def test_softcap_applies_to_logits_before_the_softmax(orc):
    hd = 8
    K = torch.zeros(2, hd)
    K[0, 0], K[1, 0] = 1.0, -1.0
    K = K.to(torch.bfloat16)
    V = torch.eye(2, hd).to(torch.bfloat16)
    q = np.zeros(hd)
    q[0] = 6.0                       # raw logits +6 and -6
    _, w_nocap = orc.attend(q, K, V, [0, 1])
    assert abs(w_nocap[0] / w_nocap[1] - np.exp(12.0)) <= 1e-10 * np.exp(12.0)
    cap = 0.5
    _, w_cap = orc.attend(q, K, V, [0, 1], softcap=cap)
    s = cap * np.tanh(np.array([6.0, -6.0]) / cap)
    assert np.all(np.abs(s) < cap)
    expect = np.exp(s - s.max()) / np.exp(s - s.max()).sum()
    assert np.allclose(w_cap, expect, rtol=1e-14, atol=0)
    assert w_cap[0] / w_cap[1] <= np.exp(2 * cap) * (1 + 1e-12)
    _, w_huge = orc.attend(q, K, V, [0, 1], softcap=1e12)
    assert np.allclose(w_huge, w_nocap, rtol=1e-9, atol=1e-300)


def test_ring_equals_linear_sliding_window(orc):
    W, P = 8, 39
    lin = _tiny(wl.SLIDING, 40, W, False, seed=7)
    ring = _tiny(wl.SLIDING, W, W, True, seed=7)
    weights = wl.make_weights(lin)
    x = wl.make_x(lin)
    kv = wl.make_kv_cache(lin)
    kr = torch.empty((1, 1, W, lin.head_dim), dtype=torch.bfloat16)
    vr = torch.empty_like(kr)
    for p in range(P - W + 1, P + 1):
        kr[0, 0, p % W] = kv["k_cache"][0, 0, p]
        vr[0, 0, p % W] = kv["v_cache"][0, 0, p]
    a = orc.decode_step(lin, weights, x, [P], kv["k_cache"], kv["v_cache"])
    b = orc.decode_step(ring, weights, x, [P], kr, vr)
    assert np.max(np.abs(a["attn"] - b["attn"])) <= 1e-13
    assert np.max(np.abs(a["out"] - b["out"])) <= 1e-12
