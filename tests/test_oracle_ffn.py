"""Pins of the oracle's dense FFN half (CPU only).

The layer's feed-forward half on the gemma4 page (encode_one_layer, the dense MLP groups
and the end-of-layer norm): pre-FF RMSNorm, gate and up projections, GELU(gate) * up, the
down projection, then the post-FF RMSNorm of the down output added to the residual and the
sum scaled by the layer scalar.  What pins it:

* the GELU is the tanh form: torch's tanh-approximate GELU in fp64, and within the known
  gap (under 5e-4) of the erf form but measurably apart from it;
* selection matrices for the three projections give every value in closed form, so a
  transposed operand, a swapped gate/up or a missing norm fails;
* a zero down projection leaves out = h * scalar exactly (RMSNorm of zero is zero);
* with eps = 0 the post-FF norm makes out invariant to scaling the down projection, and
  the pre-FF norm makes a invariant to scaling h;
* a per-channel scalar equal everywhere matches the single scalar; batch rows are
  independent.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from quantized_attention_layer_gb300 import workloads as wl

from test_oracle_layer import _perm_q8_0


def _ffn(**kw):
    base = dict(name="ffn_t", hidden=64, intermediate=128, batch=1, seed=61)
    base.update(kw)
    return wl.FfnWorkload(**base)


def test_gelu_is_the_tanh_form():
    xs = np.linspace(-9.0, 9.0, 3601)
    ours = np.array([oracle.gelu_tanh(x) for x in xs])
    ref = torch.nn.functional.gelu(torch.from_numpy(xs), approximate="tanh").numpy()
    assert np.max(np.abs(ours - ref)) <= 1e-15 * np.maximum(1.0, np.abs(xs)).max()
    erf_form = np.array([0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0))) for x in xs])
    gap = np.max(np.abs(ours - erf_form))
    assert 1e-4 < gap < 5e-4
    assert oracle.gelu_tanh(0.0) == 0.0


def test_closed_form_with_selection_weights(orc):
    f = _ffn()
    H, I = f.hidden, f.intermediate
    rng = np.random.default_rng(61)
    pg, pu = rng.integers(0, H, I), rng.integers(0, H, I)
    pd = rng.permutation(I)[:H]
    w = wl.make_ffn_weights(f)
    w["w_gate"], w["w_up"], w["w_down"] = _perm_q8_0(pg, H), _perm_q8_0(pu, H), _perm_q8_0(pd, I)
    h = wl.make_ffn_input(f, rows=2)
    r = orc.ffn_step(f, w, h)
    hd = h.to(torch.float64).numpy()
    w_pre = w["w_pre"].to(torch.float64).numpy()
    w_post = w["w_post"].to(torch.float64).numpy()
    s = float(w["scalar"][0])
    for b in range(2):
        x = hd[b]
        n = x * w_pre / np.sqrt(np.mean(x * x) + f.eps)
        a = np.array([oracle.gelu_tanh(t) for t in n[pg]]) * n[pu]
        d = a[pd]
        out = (x + d * w_post / np.sqrt(np.mean(d * d) + f.eps)) * s
        assert np.max(np.abs(r["a"][b] - a)) <= 1e-13
        assert np.max(np.abs(r["out"][b] - out)) <= 1e-13
    # gate and up are not interchangeable: GELU applies to the gate only
    w2 = dict(w, w_gate=w["w_up"], w_up=w["w_gate"])
    r2 = orc.ffn_step(f, w2, h)
    assert np.max(np.abs(r2["a"] - r["a"])) > 1e-3


def test_zero_down_projection_leaves_the_scaled_residual(orc):
    f = _ffn(scalar_per_channel=True)
    w = wl.make_ffn_weights(f)
    zero = np.array(w["w_down"], copy=True).reshape(f.hidden, -1, 34)
    zero[:, :, 0:2] = 0  # every block scale 0
    w["w_down"] = zero.reshape(f.hidden, -1)
    h = wl.make_ffn_input(f, rows=3)
    r = orc.ffn_step(f, w, h)
    want = h.to(torch.float64).numpy() * w["scalar"].to(torch.float64).numpy()[None, :]
    assert np.array_equal(r["out"], want)


def _scale_q8_0(m, k):
    """The Q8_0 matrix times 2^k, exactly (each fp16 block scale times 2^k)."""
    blk = np.array(m, copy=True).reshape(m.shape[0], -1, 34)
    d = blk[:, :, 0:2].copy().view(np.float16) * np.float16(2.0 ** k)
    blk[:, :, 0:2] = d.view(np.uint8)
    return blk.reshape(m.shape[0], -1)


def test_norms_make_the_result_scale_invariant(orc):
    f = _ffn(eps=0.0)
    w = wl.make_ffn_weights(f)
    h = wl.make_ffn_input(f, rows=2)
    r = orc.ffn_step(f, w, h)
    # post-FF norm: a scaled down projection gives the same output
    r2 = orc.ffn_step(f, dict(w, w_down=_scale_q8_0(w["w_down"], 3)), h)
    assert np.max(np.abs(r2["out"] - r["out"])) <= 1e-12 * np.max(np.abs(r["out"]))
    # pre-FF norm: a scaled input gives the same activation; out moves by the residual only
    r3 = orc.ffn_step(f, w, (h.to(torch.float32) * 4.0).to(torch.bfloat16))
    assert np.max(np.abs(r3["a"] - r["a"])) <= 1e-12 * np.max(np.abs(r["a"]))
    s = float(w["scalar"][0])
    extra = 3.0 * h.to(torch.float64).numpy() * s
    assert np.max(np.abs(r3["out"] - r["out"] - extra)) <= 1e-12 * np.max(np.abs(r3["out"]))


def test_scalar_forms_and_batch_rows(orc):
    f = _ffn()
    w = wl.make_ffn_weights(f)
    h = wl.make_ffn_input(f, rows=3)
    r = orc.ffn_step(f, w, h)
    c = float(w["scalar"][0])
    fv = f.replace(scalar_per_channel=True)
    wv = dict(w, scalar=torch.full((f.hidden,), c, dtype=torch.float32))
    rv = orc.ffn_step(fv, wv, h)
    assert np.array_equal(rv["out"], r["out"])
    for b in range(3):
        rb = orc.ffn_step(f, w, h[b:b + 1])
        assert np.array_equal(rb["out"][0], r["out"][b])
        assert np.array_equal(rb["a"][0], r["a"][b])


def test_rejects_bad_shapes(orc):
    f = _ffn(hidden=48)
    w = wl.make_ffn_weights(_ffn())
    with pytest.raises(ValueError):
        orc.ffn_step(f, w, wl.make_ffn_input(_ffn()))
