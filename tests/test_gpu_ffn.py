"""GPU parity of the dense FFN half (libhfa's hfa_ffn_step through its C ABI) against the
oracle.

* gelu(gate) * up (the a tap) and the layer output before rounding, per batch row, within
  relative L2 2e-3 of the oracle's fp64 values;
* the bf16 output is the round-to-nearest-even of the kernel's own f32 value, byte for
  byte, and differs from the oracle's bf16 rounding no more often than the float error
  explains (the same flip bound as the KV append);
* shapes: several k-splits and stages per CTA, ragged batches inside each batch tile
  (1..4, 5..8, 9..16 rows), a per-channel layer scalar, and the decode shape of the pages'
  dense MLP (2816 -> 5760 -> 2816) at batch 1 and 16;
* repeated steps on one object (the partial sums of one step are never read by the next),
  a CUDA-graph replay with new inputs, and two objects used in turn.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_layer_gb300 import hfa, workloads as wl

from parity import REL_L2, flip_bound, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_layer_gb300 import build
    build.build()
    oracle.build()


def _run(ffn, f, h):
    B = h.shape[0]
    hd = h.cuda()
    out = torch.empty((B, f.hidden), dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty((B, f.hidden), dtype=torch.float32, device="cuda")
    a = torch.empty((B, f.intermediate), dtype=torch.float32, device="cuda")
    ffn.hfa_ffn_step(hd, out, out32, a)
    ffn.hfa_ffn_check_status()
    torch.cuda.synchronize()
    return {"out_bf16": out.cpu(), "out": out32.cpu().numpy(), "a": a.cpu().numpy()}


def _check(f, got, ref, label=""):
    B = got["out"].shape[0]
    for b in range(B):
        ea = rel_l2(got["a"][b], ref["a"][b])
        eo = rel_l2(got["out"][b], ref["out"][b])
        assert ea <= REL_L2, f"{label} row {b}: a rel L2 {ea:.3e}"
        assert eo <= REL_L2, f"{label} row {b}: out rel L2 {eo:.3e}"
    # the bf16 output is the RNE of the kernel's own f32 value
    own = oracle.bf16_bits(torch.from_numpy(got["out"]).to(torch.bfloat16))
    gb = oracle.bf16_bits(got["out_bf16"])
    assert np.array_equal(own, gb), f"{label}: bf16 output is not the rounding of the f32 output"
    flips = int(np.count_nonzero(gb != ref["out_bf16"]))
    e, allowed = flip_bound(got["out"], ref["out"])
    assert flips <= allowed, f"{label}: {flips} bf16 flips, {e:.1f} expected"


def _make(f, max_batch=None):
    weights = wl.make_ffn_weights(f)
    ffn = hfa.Ffn(hfa.ffn_desc_for(f, max_batch=max_batch), hfa.ffn_weights_to_device(weights))
    return ffn, weights


@pytest.mark.parametrize("H,I,B", [(256, 512, 1), (512, 1024, 3), (1024, 2048, 5), (768, 1536, 12),
                                   (512, 2048, 16)])
def test_small_shapes(orc, H, I, B):
    f = wl.FFN_B1.replace(name="ffn_s", hidden=H, intermediate=I, batch=B, seed=80 + B)
    ffn, weights = _make(f)
    h = wl.make_ffn_input(f)
    got = _run(ffn, f, h)
    ref = orc.ffn_step(f, weights, h)
    _check(f, got, ref, f"H={H} I={I} B={B}")
    ffn.hfa_ffn_destroy()


@pytest.mark.parametrize("H,I,B,max_batch", [(352, 480, 1, 1), (352, 480, 1, 8), (96, 160, 3, 3),
                                             (32, 32, 1, 1), (1056, 2880, 16, 16)])
def test_odd_block_counts_and_tiny_shapes(orc, H, I, B, max_batch):
    # block counts with odd factors (11, 15, 3, 1 blocks of 32), fewer outputs than CTAs,
    # and a batch below the planned batch tiles
    f = wl.FFN_B1.replace(name="ffn_odd", hidden=H, intermediate=I, batch=B, seed=94 + H)
    ffn, weights = _make(f, max_batch=max_batch)
    h = wl.make_ffn_input(f)
    _check(f, _run(ffn, f, h), orc.ffn_step(f, weights, h), f"H={H} I={I} B={B}/{max_batch}")
    ffn.hfa_ffn_destroy()


def test_per_channel_scalar_and_batch_below_max(orc):
    f = wl.FFN_B1.replace(name="ffn_v", hidden=512, intermediate=1536, batch=6, seed=88,
                          scalar_per_channel=True)
    ffn, weights = _make(f, max_batch=16)  # plan for 16 rows, run 6 and then 1
    for rows in (6, 1):
        h = wl.make_ffn_input(f, rows=rows)
        got = _run(ffn, f, h)
        _check(f, got, orc.ffn_step(f, weights, h), f"rows={rows}")
    ffn.hfa_ffn_destroy()


@pytest.mark.parametrize("B", [1, 16])
def test_decode_shape(orc, B):
    f = wl.FFN_B1.replace(batch=B)
    ffn, weights = _make(f)
    plan = ffn.hfa_ffn_plan_info()
    assert plan["s1"] >= 1 and plan["stages2"] >= 1
    h = wl.make_ffn_input(f)
    got = _run(ffn, f, h)
    _check(f, got, orc.ffn_step(f, weights, h), f"2816x5760 B={B}")
    ffn.hfa_ffn_destroy()


def test_repeated_steps_and_two_objects(orc):
    f1 = wl.FFN_B1.replace(name="ffn_r1", hidden=512, intermediate=1024, batch=2, seed=90)
    f2 = f1.replace(name="ffn_r2", seed=91)
    ffn1, w1 = _make(f1)
    ffn2, w2 = _make(f2)
    for step in range(3):
        for ffn, f, w in ((ffn1, f1, w1), (ffn2, f2, w2)):
            h = wl.bf16_normal((2, f.hidden), torch.Generator().manual_seed(1000 * step + f.seed))
            _check(f, _run(ffn, f, h), orc.ffn_step(f, w, h), f"{f.name} step {step}")
    ffn1.hfa_ffn_destroy()
    ffn2.hfa_ffn_destroy()


def test_graph_replay_with_new_inputs(orc):
    f = wl.FFN_B1.replace(name="ffn_g", hidden=1024, intermediate=2048, batch=1, seed=92)
    ffn, weights = _make(f)
    h = torch.empty((1, f.hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((1, f.hidden), dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty((1, f.hidden), dtype=torch.float32, device="cuda")
    a = torch.empty((1, f.intermediate), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    h.copy_(wl.make_ffn_input(f).cuda())
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        ffn.hfa_ffn_step(h, out, out32, a, stream=s)  # warm-up outside the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ffn.hfa_ffn_step(h, out, out32, a, stream=s)
    for k in range(3):
        hk = wl.bf16_normal((1, f.hidden), torch.Generator().manual_seed(500 + k))
        h.copy_(hk.cuda())
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ffn.hfa_ffn_check_status()
        got = {"out_bf16": out.cpu(), "out": out32.cpu().numpy(), "a": a.cpu().numpy()}
        _check(f, got, orc.ffn_step(f, weights, hk), f"replay {k}")
    ffn.hfa_ffn_destroy()


def test_step_validation():
    f = wl.FFN_B1.replace(name="ffn_e", hidden=256, intermediate=512, batch=2, seed=93)
    ffn, _ = _make(f)
    h = torch.zeros((3, 256), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((3, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(hfa.HfaError) as ei:
        ffn.hfa_ffn_step(h, out)  # 3 rows > max_batch 2
    assert ei.value.status == hfa.HFA_EINVAL
    with pytest.raises(hfa.HfaError) as ei:
        ffn.hfa_ffn_step(h[:2], out.view(-1)[1:513].view(2, 256))  # misaligned output
    assert ei.value.status == hfa.HFA_EINVAL
    ffn.hfa_ffn_destroy()
