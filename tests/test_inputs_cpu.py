"""The seeded input recipe: every buffer is a pure function of (workload seed, buffer), drawn
from a stream of its own, with the distributions the design notes state."""
import numpy as np
import torch

from quantized_attention_layer_gb300 import workloads as wl

SMALL = wl.Workload(name="inputs", hidden=128, num_heads=4, num_kv_heads=2, head_dim=64,
                    layer_type=wl.SLIDING, window=16, kv_capacity=32, ring=False, batch=2,
                    rope_theta=1e4, seed=11, seq_pos_range=(3, 30), post_norm=True,
                    rope_freq_factors=True)


def _same(a, b):
    if a is None or b is None:
        return a is None and b is None
    if isinstance(a, torch.Tensor):
        return torch.equal(a, b)
    return np.array_equal(a, b)


def test_inputs_are_a_function_of_the_seed():
    for make in (wl.make_weights, wl.make_x, wl.make_positions, wl.make_kv_cache):
        a, b = make(SMALL), make(SMALL)
        if isinstance(a, dict):
            assert a.keys() == b.keys() and all(_same(a[k], b[k]) for k in a), make.__name__
        else:
            assert _same(a, b), make.__name__
    other = wl.make_weights(SMALL.replace(seed=12))
    assert not np.array_equal(other["wq"], wl.make_weights(SMALL)["wq"])


def test_buffers_draw_from_streams_of_their_own():
    # a larger cache leaves the weights, the layer input and the positions as they were
    big = SMALL.replace(kv_capacity=64, window=32)
    w0, w1 = wl.make_weights(SMALL), wl.make_weights(big)
    assert all(_same(w0[k], w1[k]) for k in w0)
    assert torch.equal(wl.make_x(SMALL), wl.make_x(big))
    # a wider hidden size leaves the per-head norm weights as they were
    wide = wl.make_weights(SMALL.replace(hidden=256))
    assert torch.equal(wide["w_q"], w0["w_q"]) and torch.equal(wide["w_k"], w0["w_k"])


def test_q8_0_blocks_follow_the_recipe():
    raw = wl.make_weights(SMALL)["wq"]
    rows, nb = SMALL.q_rows, SMALL.hidden // 32
    assert raw.dtype == np.uint8 and raw.shape == (rows, nb * 34)
    blocks = raw.reshape(rows, nb, 34)
    d = blocks[:, :, 0:2].copy().view(np.float16).astype(np.float64)
    q = blocks[:, :, 2:].view(np.int8)
    assert d.min() >= 0.001 - 1e-6 and d.max() <= 0.02 + 2e-5  # U[0.001, 0.02] in fp16
    assert q.min() >= -127 and q.max() <= 127                 # U[-127, 127], never -128
    assert q.min() == -127 and q.max() == 127                 # the whole range is drawn


def test_norm_weights_factors_and_caches_follow_the_recipe():
    w = wl.make_weights(SMALL)
    for k in ("w_in", "w_q", "w_k", "w_post"):
        assert w[k].dtype == torch.float32 and 0.5 <= w[k].min() and w[k].max() < 1.5, k
    ff = w["rope_ff"]
    assert ff.shape == (SMALL.head_dim // 2,) and 1.0 <= ff.min() and ff.max() < 4.0
    kv = wl.make_kv_cache(SMALL)
    kc = kv["k_cache"]
    assert kc.dtype == torch.bfloat16
    assert tuple(kc.shape) == (SMALL.batch, SMALL.num_kv_heads, SMALL.kv_capacity, SMALL.head_dim)
    assert abs(float(kc.float().std()) - 1.0) < 0.05 and not torch.equal(kc, kv["v_cache"])
    pos = wl.make_positions(SMALL)
    assert pos.dtype == np.int32 and pos.min() >= 3 and pos.max() <= 30


def test_quantised_kv_signs_are_plus_or_minus_one_and_seeded():
    s = wl.make_tq_signs(512, 7)
    assert s.dtype == np.int8 and set(np.unique(s)) == {-1, 1}
    assert np.array_equal(s, wl.make_tq_signs(512, 7))
    assert not np.array_equal(s, wl.make_tq_signs(512, 8))
