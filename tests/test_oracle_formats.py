"""Pins of the oracle's number formats and Q8_0 mat-vec (CPU only).

Each test checks the oracle against something other than itself: an exhaustive
library conversion, hand-made fixtures under tests/golden/, the Q8_0 quantiser as the
gemma4/model.rs page states it, or an independent blockwise formulation.
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_f16_decode_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decode_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.bf16_scalar_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_rounding_golden(orc):
    n = 0
    for line in open(os.path.join(GOLDEN, "bf16_rounding.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        parts = line.split()
        # columns: expression (may contain spaces), hex pattern, note words
        hex_idx = next(i for i, p in enumerate(parts) if p.startswith("0x"))
        expr = " ".join(parts[:hex_idx])
        expected = int(parts[hex_idx], 16)
        value = eval(expr, {"__builtins__": {}})
        assert orc.f64_to_bf16(value) == expected, (expr, hex(orc.f64_to_bf16(value)))
        n += 1
    assert n >= 10


def test_bf16_rounding_matches_torch_on_binary32(orc):
    # For values exactly representable in binary32, torch's binary32 -> bf16
    # conversion (round to nearest even) is a library reference.
    rng = np.random.default_rng(7)
    pats = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    f = pats.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f64_to_bf16(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)


def _golden_blocks():
    blocks, values = [], []
    for line in open(os.path.join(GOLDEN, "q8_0_blocks.txt")):
        if line.startswith("block "):
            blocks.append(bytes(int(t, 16) for t in line.split()[1:]))
        elif line.startswith("values "):
            values.append([float(t) for t in line.split()[1:]])
    return blocks, values


def test_q8_0_dequant_golden(orc):
    blocks, values = _golden_blocks()
    assert len(blocks) == len(values) >= 5
    for blk, vals in zip(blocks, values):
        assert len(blk) == 34
        got = orc.q8_0_dequant(np.frombuffer(blk, dtype=np.uint8), 32)[0]
        assert np.array_equal(got, np.array(vals)), (blk.hex(), got)


def _quantise_like_the_page(v):
    """The gemma4/model.rs Q8_0 re-quantiser: d = amax/127, q = round(v/d) clamped."""
    rows, cols = v.shape
    out = np.zeros((rows, cols // 32, 34), dtype=np.uint8)
    for r in range(rows):
        for b in range(cols // 32):
            blk = v[r, 32 * b:32 * b + 32].astype(np.float32)
            amax = float(np.max(np.abs(blk)))
            d = np.float32(amax / 127.0) if amax > 0 else np.float32(0)
            inv = np.float32(1.0) / d if d != 0 else np.float32(0)
            q = np.clip(np.round(blk * inv), -127, 127).astype(np.int8)
            out[r, b, 0:2] = np.array([np.float16(d)]).view(np.uint8)
            out[r, b, 2:] = q.view(np.uint8)
    return out.reshape(rows, -1)


def test_q8_0_page_quantiser_round_trip(orc):
    rng = np.random.default_rng(3)
    v = rng.normal(size=(6, 128)).astype(np.float32)
    blocks = _quantise_like_the_page(v)
    deq = orc.q8_0_dequant(blocks, 128)
    for r in range(6):
        for b in range(4):
            seg = v[r, 32 * b:32 * b + 32].astype(np.float64)
            d = float(np.max(np.abs(seg))) / 127.0
            # rounding to the grid costs at most d/2; the fp16 scale adds a relative 2^-11
            assert np.max(np.abs(deq[r, 32 * b:32 * b + 32] - seg)) <= d * (0.5 + 127 * 2**-10)


def test_q8_0_matvec_blockwise_equals_dense(orc):
    from quantized_attention_layer_gb300 import workloads as wl
    g = torch.Generator().manual_seed(11)
    rows, cols = 48, 256
    blocks = wl.q8_0_blocks(rows, cols, g)
    x = np.random.default_rng(1).normal(size=cols)
    y = orc.q8_0_matvec(blocks, rows, cols, x)
    yb = orc.q8_0_matvec(blocks, rows, cols, x, blockwise=True)
    assert np.max(np.abs(y - yb)) <= 1e-12 * np.max(np.abs(y))


def test_q8_0_matvec_one_hot_columns(orc):
    from quantized_attention_layer_gb300 import workloads as wl
    g = torch.Generator().manual_seed(12)
    rows, cols = 16, 96
    blocks = wl.q8_0_blocks(rows, cols, g)
    raw = blocks.reshape(rows, cols // 32, 34)
    for c in (0, 1, 31, 32, 63, 95):
        x = np.zeros(cols)
        x[c] = 1.0
        y = orc.q8_0_matvec(blocks, rows, cols, x)
        b, i = divmod(c, 32)
        d = raw[:, b, 0:2].copy().view(np.float16).astype(np.float64)[:, 0]
        q = raw[:, b, 2 + i].view(np.int8).astype(np.float64)
        assert np.array_equal(y, d * q)


def test_q8_0_zero_scale_block_contributes_nothing(orc):
    from quantized_attention_layer_gb300 import workloads as wl
    blocks = wl.q8_0_blocks(4, 64, torch.Generator().manual_seed(13)).reshape(4, 2, 34).copy()
    blocks[:, 1, 0:2] = 0
    x = np.zeros(64)
    x[32:] = np.random.default_rng(2).normal(size=32)
    assert np.array_equal(orc.q8_0_matvec(blocks.reshape(4, -1), 4, 64, x), np.zeros(4))


def test_bf16_matvec_matches_numpy_matmul(orc):
    w = (torch.randn(40, 64, generator=torch.Generator().manual_seed(5)) * 0.02).to(torch.bfloat16)
    x = np.random.default_rng(4).normal(size=64)
    ref = w.to(torch.float64).numpy() @ x
    got = orc.bf16_matvec(w, x)
    assert np.max(np.abs(got - ref)) <= 1e-14 * np.max(np.abs(ref)) * 64
