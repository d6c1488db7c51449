"""Pins of the oracle's drafter pieces (CPU only).

The drafter layer of the speculative-decoding page attends over the committed context, its
new context rows and the block's own rows, bidirectionally within the block on a full layer
and causally (with the window) on a sliding one; its context rows are projected by Wk and Wv
without the input norm.

* a bidirectional block of one row is the causal block;
* every row of a bidirectional block equals the attention of that row's query over the
  explicit key set [0, last position of the block], computed by the single-query routine;
* on a sliding layer the flag changes nothing;
* the context rows in closed form: permutation Wk and Wv, power-of-two RoPE angles applied
  as complex rotations, the bf16 rounding in the cache slots.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_layer_gb300 import workloads as wl

from test_oracle_layer import _perm_q8_0


def _layer(**kw):
    base = dict(name="draft", hidden=96, num_heads=4, num_kv_heads=2, head_dim=16,
                layer_type=wl.FULL, window=0, kv_capacity=40, ring=False, batch=1,
                rope_theta=1e4, seed=51, base_pos=20, verify_len=6, attn_scale=0.25)
    base.update(kw)
    return wl.Workload(**base)


def test_one_row_bidirectional_block_is_causal(orc):
    w = _layer(verify_len=1)
    weights, x, kv = wl.make_weights(w), wl.make_x(w), wl.make_kv_cache(w)
    a = orc.verify_block(w, weights, x, 20, kv["k_cache"], kv["v_cache"])
    b = orc.verify_block(w.replace(block_bidir=True), weights, x, 20, kv["k_cache"], kv["v_cache"])
    for key in ("q", "attn", "out"):
        assert np.array_equal(a[key], b[key])


def test_bidirectional_rows_see_the_whole_block(orc):
    w = _layer(block_bidir=True)
    weights, x, kv = wl.make_weights(w), wl.make_x(w), wl.make_kv_cache(w)
    r = orc.verify_block(w, weights, x, 20, kv["k_cache"], kv["v_cache"])
    last = 20 + 6 - 1
    rows = np.arange(last + 1)
    kc = r["k_cache"].reshape(2, 40, 16)
    vc = r["v_cache"].reshape(2, 40, 16)
    for i in range(6):
        for h in range(4):
            o, wts = orc.attend(r["q"][i, h], kc[h // 2], vc[h // 2], rows, scale=0.25)
            assert np.max(np.abs(o - r["attn"][i, h])) <= 1e-13
            assert abs(wts.sum() - 1.0) < 1e-13
    # and they differ from the causal block for every row but the last
    c = orc.verify_block(w.replace(block_bidir=False), weights, x, 20, kv["k_cache"], kv["v_cache"])
    assert np.array_equal(c["attn"][5], r["attn"][5])
    assert all(np.max(np.abs(c["attn"][i] - r["attn"][i])) > 1e-6 for i in range(5))


def test_flag_leaves_sliding_layers_causal(orc):
    w = _layer(layer_type=wl.SLIDING, window=9)
    weights, x, kv = wl.make_weights(w), wl.make_x(w), wl.make_kv_cache(w)
    a = orc.verify_block(w, weights, x, 20, kv["k_cache"], kv["v_cache"])
    b = orc.verify_block(w.replace(block_bidir=True), weights, x, 20, kv["k_cache"], kv["v_cache"])
    assert np.array_equal(a["attn"], b["attn"])


@pytest.mark.parametrize("S,base", [(1, 0), (3, 11)])
def test_context_rows_closed_form(orc, S, base):
    hd, nkv, H = 16, 2, 64
    w = wl.Workload(name="ctx", hidden=H, num_heads=4, num_kv_heads=nkv, head_dim=hd,
                    layer_type=wl.FULL, window=0, kv_capacity=base + S + 2, ring=False, batch=1,
                    rope_theta=256.0, seed=52)
    rng = np.random.default_rng(52 + S)
    pk = rng.permutation(H)[:nkv * hd]
    pv = rng.permutation(H)[:nkv * hd]
    weights = wl.make_weights(w)
    weights["wk"] = _perm_q8_0(pk, H)
    weights["wv"] = _perm_q8_0(pv, H)
    x = wl.make_x(w, rows=S)
    kv = wl.make_kv_cache(w)
    r = orc.ctx_append(w, weights, x, base, kv["k_cache"], kv["v_cache"])
    w_k = weights["w_k"].to(torch.float64).numpy()
    xd = x.to(torch.float64).numpy()
    for i in range(S):
        rot = np.exp(1j * (base + i) * np.ldexp(1.0, -np.arange(hd // 2)))
        for h in range(nkv):
            t = xd[i, pk[h * hd:(h + 1) * hd]]          # no input norm on context rows
            u = t * w_k / np.sqrt(np.mean(t * t) + w.eps)
            z = (u[:hd // 2] + 1j * u[hd // 2:]) * rot
            k = np.concatenate([z.real, z.imag])
            assert np.max(np.abs(r["k"][i, h] - k)) <= 1e-13
            assert np.array_equal(r["v"][i, h], xd[i, pv[h * hd:(h + 1) * hd]])
    kc = r["k_cache"].reshape(nkv, w.kv_capacity, hd)
    for i in range(S):
        kb = np.array([[oracle.f64_to_bf16(t) for t in row] for row in r["k"][i]], dtype=np.uint16)
        assert np.array_equal(kc[:, base + i, :], kb)
