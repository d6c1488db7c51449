"""Pins of the oracle's Gemma decode variants (CPU only).

* RoPE frequency factors [P1 fused head norm + RoPE, freq factors on global layers;
  P2 rope_freqs.weight]: read as phi_i = pos * theta^(-2i/hd) / f_i.  Pinned by the
  position scaling (f = 2 at position 2p is the plain rotation at p), by f = 1 being the
  plain rotation, by per-pair locality (a factor moves only its own pair) and by norms;
* k_eq_v [P2 model.rs: no v_proj when k_eq_v; P1 GPU V norm of attn_k] and the
  post-attention RMSNorm before the residual add [P1 fused post-attention norm + add]:
  a closed-form layer with permutation weights at position 0, one visible key.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_layer_gb300 import workloads as wl

from test_oracle_layer import _perm_q8_0


def test_rope_frequency_factors_scale_the_position(orc):
    rng = np.random.default_rng(3)
    hd = 64
    u = rng.standard_normal(hd)
    plain = oracle.rope_neox(u, 37, 1e4)
    assert np.array_equal(oracle.rope_neox(u, 37, 1e4, np.ones(hd // 2)), plain)
    # f = 2 everywhere at position 74 is the plain rotation at 37
    assert np.max(np.abs(oracle.rope_neox(u, 74, 1e4, np.full(hd // 2, 2.0)) - plain)) < 1e-12
    # a factor moves only its own pair (i, i + hd/2)
    f = np.ones(hd // 2)
    f[5] = 3.0
    got = oracle.rope_neox(u, 37, 1e4, f)
    mask = np.ones(hd, dtype=bool)
    mask[[5, 5 + hd // 2]] = False
    assert np.array_equal(got[mask], plain[mask])
    assert not np.allclose(got[~mask], plain[~mask])
    # the pair's angle is divided by its factor: at position 3 * 37 it is the plain angle
    got3 = oracle.rope_neox(u, 3 * 37, 1e4, f)
    assert np.max(np.abs(got3[~mask] - plain[~mask])) < 1e-12
    # rotations preserve each pair's norm
    g = rng.uniform(1.0, 4.0, hd // 2)
    r = oracle.rope_neox(u, 1234, 1e6, g)
    h = hd // 2
    assert np.allclose(r[:h] ** 2 + r[h:] ** 2, u[:h] ** 2 + u[h:] ** 2, rtol=1e-13, atol=0)


@pytest.mark.parametrize("k_eq_v,post_norm", [(True, False), (False, True), (True, True)])
def test_closed_form_layer_k_eq_v_and_post_norm(orc, k_eq_v, post_norm):
    w = wl.Workload(name="perm_v", hidden=64, num_heads=4, num_kv_heads=2, head_dim=16,
                    layer_type=wl.FULL, window=0, kv_capacity=4, ring=False, batch=1,
                    rope_theta=1e4, seed=9, seq_pos=0, k_eq_v=k_eq_v, post_norm=post_norm)
    rng = np.random.default_rng(11)
    pk = rng.permutation(64)[:32]
    pv = rng.permutation(64)[:32]
    po = rng.permutation(64)
    weights = wl.make_weights(w)
    assert (weights["wv"] is None) == k_eq_v
    weights["wk"] = _perm_q8_0(pk, 64)
    if not k_eq_v:
        weights["wv"] = _perm_q8_0(pv, 64)
    weights["wo"] = _perm_q8_0(po, 64)
    x = wl.make_x(w)
    kv = wl.make_kv_cache(w)
    r = orc.decode_step(w, weights, x, [0], kv["k_cache"], kv["v_cache"])

    xd = x.to(torch.float64).numpy()[0]
    w_in = weights["w_in"].to(torch.float64).numpy()
    n = xd * w_in / np.sqrt(np.mean(xd * xd) + w.eps)
    # V: the raw K projection, unit-RMS-normalised per head (k_eq_v), else the V projection
    v = (n[pk] if k_eq_v else n[pv]).reshape(2, 16)
    if k_eq_v:
        v = v / np.sqrt(np.mean(v * v, axis=1, keepdims=True) + w.eps)
    v_b = np.array([[oracle.bf16_scalar_to_f64(oracle.f64_to_bf16(t)) for t in row] for row in v])
    o = np.concatenate([v_b[0], v_b[0], v_b[1], v_b[1]])
    y = o[po]
    if post_norm:
        w_post = weights["w_post"].to(torch.float64).numpy()
        y = y * w_post / np.sqrt(np.mean(y * y) + w.eps)
    assert np.max(np.abs(r["v"][0] - v)) <= 1e-14
    assert np.array_equal(r["attn"][0].reshape(-1), o)
    assert np.max(np.abs(r["out"][0] - (xd + y))) <= 1e-14
    if k_eq_v:
        # at position 0 RoPE is the identity: with unit k_norm weights K equals V
        weights["w_k"] = torch.ones(16, dtype=torch.float32)
        r1 = orc.decode_step(w, weights, x, [0], kv["k_cache"], kv["v_cache"])
        assert np.array_equal(r1["k"], r1["v"])


def test_post_norm_output_is_invariant_to_the_o_proj_scale(orc):
    w = wl.Workload(name="post", hidden=128, num_heads=4, num_kv_heads=2, head_dim=32,
                    layer_type=wl.SLIDING, window=8, kv_capacity=32, ring=False, batch=1,
                    rope_theta=1e4, seed=12, seq_pos=20, post_norm=True)
    weights = wl.make_weights(w)
    x = wl.make_x(w)
    kv = wl.make_kv_cache(w)
    a = orc.decode_step(w, weights, x, [20], kv["k_cache"], kv["v_cache"])
    # doubling every fp16 scale of Wo (exact) doubles y; RMSNorm(2y) = RMSNorm(y) up to eps
    wo = np.array(weights["wo"], dtype=np.uint8).reshape(-1, 34).copy()
    d = wo[:, :2].copy().view(np.float16)
    wo[:, :2] = (d * np.float16(2)).view(np.uint8)
    weights["wo"] = wo.reshape(np.array(weights["wo"]).shape)
    b = orc.decode_step(w, weights, x, [20], kv["k_cache"], kv["v_cache"])
    y_a = a["out"][0] - x.to(torch.float64).numpy()[0]
    y_b = b["out"][0] - x.to(torch.float64).numpy()[0]
    assert np.max(np.abs(y_a - y_b)) < 1e-5 * np.max(np.abs(y_a))
    # and with the weights of the norm the output's RMS is fixed by w_post alone
    w_post = weights["w_post"].to(torch.float64).numpy()
    assert abs(np.sqrt(np.mean((y_a / w_post) ** 2)) - 1.0) < 1e-5


def test_frequency_factors_of_two_rotate_like_half_the_position(orc):
    base = wl.Workload(name="ff", hidden=128, num_heads=4, num_kv_heads=2, head_dim=32,
                       layer_type=wl.FULL, window=0, kv_capacity=64, ring=False, batch=1,
                       rope_theta=1e6, seed=13, seq_pos=40)
    weights = wl.make_weights(base)
    x = wl.make_x(base)
    kv = wl.make_kv_cache(base)
    wf = base.replace(rope_freq_factors=True)
    wff = dict(weights)
    wff["rope_ff"] = torch.full((16,), 2.0)
    a = orc.decode_step(wf, wff, x, [40], kv["k_cache"], kv["v_cache"])
    b = orc.decode_step(base, weights, x, [20], kv["k_cache"], kv["v_cache"])
    assert np.max(np.abs(a["q"] - b["q"])) < 1e-12
    assert np.max(np.abs(a["k"] - b["k"])) < 1e-12
