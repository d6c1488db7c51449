"""Whole-layer pins of the oracle (CPU only).

* a closed-form layer: permutation Q8_0 weights at position 0 with one visible key;
* the q and k heads in closed form at a later position: distinct permutation Wq and Wk,
  distinct q_norm / k_norm weights, RoPE angles that are exact powers of two applied as
  complex rotations (so a swapped projection, a norm applied after RoPE, or RoPE left off
  one of q and k all fail);
* the verify block of L tokens equals L decode steps one after another;
* a batch of sequences equals the sequences stepped one by one.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_layer_gb300 import workloads as wl


def _perm_q8_0(perm, cols):
    """Q8_0 bytes of the 0/1 matrix with W[r, perm[r]] = 1 (d = 1.0 = fp16 0x3C00)."""
    rows = len(perm)
    blk = np.zeros((rows, cols // 32, 34), dtype=np.uint8)
    blk[:, :, 0] = 0x00
    blk[:, :, 1] = 0x3C
    for r, c in enumerate(perm):
        blk[r, c // 32, 2 + c % 32] = 1
    return blk.reshape(rows, -1)


@pytest.mark.parametrize("v_unit_norm", [False, True])
def test_closed_form_layer_with_permutation_weights(orc, v_unit_norm):
    # H = nh * hd so that o_proj is square; GQA group 2.
    w = wl.Workload(name="perm", hidden=64, num_heads=4, num_kv_heads=2, head_dim=16,
                    layer_type=wl.FULL, window=0, kv_capacity=4, ring=False, batch=1,
                    rope_theta=1e4, seed=9, seq_pos=0, v_unit_norm=v_unit_norm)
    rng = np.random.default_rng(9)
    pv = rng.permutation(64)[:32]
    po = rng.permutation(64)
    weights = wl.make_weights(w)
    weights["wv"] = _perm_q8_0(pv, 64)
    weights["wo"] = _perm_q8_0(po, 64)
    x = wl.make_x(w)
    kv = wl.make_kv_cache(w)
    r = orc.decode_step(w, weights, x, [0], kv["k_cache"], kv["v_cache"])

    xd = x.to(torch.float64).numpy()[0]
    w_in = weights["w_in"].to(torch.float64).numpy()
    n = xd * w_in / np.sqrt(np.mean(xd * xd) + w.eps)       # input RMSNorm
    v = n[pv].reshape(2, 16)                                   # V projection
    if v_unit_norm:
        v = v / np.sqrt(np.mean(v * v, axis=1, keepdims=True) + w.eps)
    v_b = np.array([[oracle.bf16_scalar_to_f64(oracle.f64_to_bf16(t)) for t in row] for row in v])
    o = np.concatenate([v_b[0], v_b[0], v_b[1], v_b[1]])     # one key: o = V; head h -> h // 2
    y = o[po]                                                  # O projection
    assert np.max(np.abs(r["v"][0] - v)) <= 1e-14
    assert np.array_equal(r["attn"][0].reshape(-1), o)
    assert np.max(np.abs(r["out"][0] - (xd + y))) <= 1e-14
    # the appended slot holds exactly the bf16 rounding of v; other slots are untouched
    vc = r["v_cache"].reshape(2, 4, 16)
    assert np.array_equal(oracle.bf16_to_f64(vc[:, 0, :]), v_b)
    assert np.array_equal(vc[:, 1:, :], oracle.bf16_bits(kv["v_cache"]).reshape(2, 4, 16)[:, 1:, :])


@pytest.mark.parametrize("P", [5, 77])
def test_closed_form_q_and_k_heads_at_a_later_position(orc, P):
    # theta = 2^8 with head_dim 16: inverse frequencies 256^(-2i/16) = 2^-i exactly, so the
    # angle of pair i is P * 2^-i.  The rotation of the NeoX pair (u_i, u_{i+8}) is the
    # complex product (u_i + j u_{i+8}) * e^{j phi_i}.
    hd, nh, nkv, H = 16, 4, 2, 64
    w = wl.Workload(name="qkpin", hidden=H, num_heads=nh, num_kv_heads=nkv, head_dim=hd,
                    layer_type=wl.FULL, window=0, kv_capacity=P + 3, ring=False, batch=1,
                    rope_theta=256.0, seed=31, seq_pos=P)
    rng = np.random.default_rng(31)
    pq = rng.permutation(H)             # Wq: 64 rows, each picks one input column
    pk = rng.permutation(H)[:nkv * hd]  # Wk: 32 rows, a different choice of columns
    weights = wl.make_weights(w)
    weights["wq"] = _perm_q8_0(pq, H)
    weights["wk"] = _perm_q8_0(pk, H)
    w_q = weights["w_q"].to(torch.float64).numpy()
    w_k = weights["w_k"].to(torch.float64).numpy()
    assert np.min(np.abs(w_q - w_k)) > 0  # a swap of the two norm weights shows
    x = wl.make_x(w)
    kv = wl.make_kv_cache(w)
    r = orc.decode_step(w, weights, x, [P], kv["k_cache"], kv["v_cache"])

    xd = x.to(torch.float64).numpy()[0]
    w_in = weights["w_in"].to(torch.float64).numpy()
    n = xd * w_in / np.sqrt(np.mean(xd * xd) + w.eps)
    rot = np.exp(1j * P * np.ldexp(1.0, -np.arange(hd // 2)))

    def head(t, wn):
        u = t * wn / np.sqrt(np.mean(t * t) + w.eps)  # per-head RMSNorm, then RoPE
        z = (u[:hd // 2] + 1j * u[hd // 2:]) * rot
        return np.concatenate([z.real, z.imag])

    q = np.stack([head(n[pq[h * hd:(h + 1) * hd]], w_q) for h in range(nh)])
    k = np.stack([head(n[pk[h * hd:(h + 1) * hd]], w_k) for h in range(nkv)])
    assert np.max(np.abs(r["q"][0] - q)) <= 1e-13
    assert np.max(np.abs(r["k"][0] - k)) <= 1e-13
    # the key row lands at slot P as the bf16 rounding of k
    kc = r["k_cache"].reshape(nkv, w.kv_capacity, hd)
    kb = np.array([[oracle.f64_to_bf16(t) for t in row] for row in k], dtype=np.uint16)
    assert np.array_equal(kc[:, P, :], kb)


def test_verify_block_equals_sequential_decode_steps(orc):
    w = wl.Workload(name="ver", hidden=96, num_heads=4, num_kv_heads=2, head_dim=16,
                    layer_type=wl.FULL, window=0, kv_capacity=24, ring=False, batch=1,
                    rope_theta=1e4, seed=21, base_pos=10, verify_len=5, softcap=30.0)
    weights = wl.make_weights(w)
    x = wl.make_x(w)
    kv = wl.make_kv_cache(w)
    ver = orc.verify_block(w, weights, x, 10, kv["k_cache"], kv["v_cache"])
    kc, vc = kv["k_cache"], kv["v_cache"]
    for i in range(5):
        step = orc.decode_step(w, weights, x[i:i + 1], [10 + i], kc, vc)
        kc = torch.from_numpy(step["k_cache"].view(np.int16)).view(torch.bfloat16)
        vc = torch.from_numpy(step["v_cache"].view(np.int16)).view(torch.bfloat16)
        for key in ("q", "k", "v", "attn", "out"):
            assert np.max(np.abs(step[key][0] - ver[key][i])) <= 1e-13, (key, i)
    assert np.array_equal(oracle.bf16_bits(kc), ver["k_cache"])
    assert np.array_equal(oracle.bf16_bits(vc), ver["v_cache"])


def test_global_layer_verify_block_equals_sequential_decode_steps(orc):
    # the global layer's width and variants (hd 512, no V projection, RoPE frequency
    # factors, post-attention norm, GQA group 4) through both paths of the oracle
    w = wl.Workload(name="verglob", hidden=128, num_heads=4, num_kv_heads=1, head_dim=512,
                    layer_type=wl.FULL, window=0, kv_capacity=20, ring=False, batch=1,
                    rope_theta=1e6, seed=24, base_pos=9, verify_len=4, k_eq_v=True,
                    rope_freq_factors=True, post_norm=True)
    weights = wl.make_weights(w)
    assert weights["wv"] is None and weights["rope_ff"] is not None
    x = wl.make_x(w)
    kv = wl.make_kv_cache(w)
    ver = orc.verify_block(w, weights, x, 9, kv["k_cache"], kv["v_cache"])
    kc, vc = kv["k_cache"], kv["v_cache"]
    for i in range(4):
        step = orc.decode_step(w, weights, x[i:i + 1], [9 + i], kc, vc)
        kc = torch.from_numpy(step["k_cache"].view(np.int16)).view(torch.bfloat16)
        vc = torch.from_numpy(step["v_cache"].view(np.int16)).view(torch.bfloat16)
        for key in ("q", "k", "v", "attn", "out"):
            assert np.max(np.abs(step[key][0] - ver[key][i])) <= 1e-12, (key, i)
    assert np.array_equal(oracle.bf16_bits(kc), ver["k_cache"])
    assert np.array_equal(oracle.bf16_bits(vc), ver["v_cache"])


def test_sliding_verify_block_matches_decode_steps(orc):
    w = wl.Workload(name="versl", hidden=64, num_heads=2, num_kv_heads=1, head_dim=32,
                    layer_type=wl.SLIDING, window=6, kv_capacity=32, ring=False, batch=1,
                    rope_theta=1e4, seed=22, base_pos=12, verify_len=4)
    weights = wl.make_weights(w)
    x = wl.make_x(w)
    kv = wl.make_kv_cache(w)
    ver = orc.verify_block(w, weights, x, 12, kv["k_cache"], kv["v_cache"])
    kc, vc = kv["k_cache"], kv["v_cache"]
    for i in range(4):
        step = orc.decode_step(w, weights, x[i:i + 1], [12 + i], kc, vc)
        kc = torch.from_numpy(step["k_cache"].view(np.int16)).view(torch.bfloat16)
        vc = torch.from_numpy(step["v_cache"].view(np.int16)).view(torch.bfloat16)
        assert np.max(np.abs(step["out"][0] - ver["out"][i])) <= 1e-13


def test_batch_equals_independent_sequences(orc):
    w = wl.Workload(name="batch", hidden=64, num_heads=4, num_kv_heads=2, head_dim=16,
                    layer_type=wl.SLIDING, window=8, kv_capacity=8, ring=True, batch=3,
                    rope_theta=1e4, seed=23, seq_pos_range=(8, 40))
    weights = wl.make_weights(w)
    x = wl.make_x(w)
    kv = wl.make_kv_cache(w)
    pos = wl.make_positions(w)
    full = orc.decode_step(w, weights, x, pos, kv["k_cache"], kv["v_cache"])
    one = w.replace(batch=1)
    for b in range(3):
        r = orc.decode_step(one, weights, x[b:b + 1], pos[b:b + 1], kv["k_cache"][b:b + 1],
                            kv["v_cache"][b:b + 1])
        for key in ("q", "attn", "out"):
            assert np.array_equal(r[key][0], full[key][b])
        assert np.array_equal(r["k_cache"][0], full["k_cache"][b])


def test_decode_rejects_out_of_range_positions(orc):
    w = wl.TINY_SLIDING
    weights = wl.make_weights(w)
    kv = wl.make_kv_cache(w)
    with pytest.raises(ValueError):
        orc.decode_step(w, weights, wl.make_x(w), [w.kv_capacity], kv["k_cache"], kv["v_cache"])
