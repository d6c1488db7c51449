"""The weight re-layout done at layer creation, read back and undone (GPU).

hfa_layer_create copies the Q8_0 blocks (34 bytes: fp16 scale, 32 int8) into 544-byte
MMA tiles and the bf16 matrices into 128 x 64 swizzled tiles; only the placement of the
bytes may change.  This test decodes the tiles returned by hfa_debug_weight_tiles with the
layout stated in hfa.h, written out here independently of the library, and compares the
result with the original blocks byte for byte: scales, the +128 bias of every weight
byte, the lane and word order, the k-split order and the swizzle.
"""
import numpy as np
import pytest
import torch

from quantized_attention_layer_gb300 import hfa, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_layer_gb300 import build
    build.build()


def k_split_blocks(nb):
    """Blocks per k-split: the largest divisor of the block count up to 16."""
    return max(d for d in range(1, 17) if nb % d == 0)


def undo_q8_tiles(tiles, rows, cols):
    """Q8_0 tile bytes -> [rows, cols/32, 34] blocks (hfa.h, hfa_debug_weight_tiles)."""
    nb = cols // 32
    nbs = k_split_blocks(nb)
    R = rows // 16
    t = tiles.reshape(nb // nbs, R, nbs, 544)
    out = np.zeros((rows, nb, 34), dtype=np.uint8)
    for s in range(nb // nbs):
        for r in range(R):
            for bb in range(nbs):
                b = s * nbs + bb
                tile = t[s, r, bb]
                words = tile[:512].reshape(32, 4, 4)  # lane, word, byte
                for lane in range(32):
                    g, tt = lane // 4, lane % 4
                    for ks in range(2):
                        for h in range(2):
                            row = 16 * r + g + 8 * h
                            c0 = 16 * ks + 2 * tt
                            for e, c in enumerate((c0, c0 + 1, c0 + 8, c0 + 9)):
                                out[row, b, 2 + c] = (int(words[lane, 2 * ks + h, e]) - 128) & 0xFF
                sc = tile[512:].reshape(8, 2, 2)  # g, (row g, row g + 8), fp16 bytes
                for g in range(8):
                    out[16 * r + g, b, 0:2] = sc[g, 0]
                    out[16 * r + g + 8, b, 0:2] = sc[g, 1]
    return out


def undo_bf16_tiles(tiles, rows, K):
    """bf16 tile bytes -> [rows, K] uint16 (128 x 64 tiles, 128-byte swizzle)."""
    t = tiles.reshape(rows // 128, K // 64, 128, 8, 16)  # m, c, r, position, byte
    out = np.zeros((rows, K), dtype=np.uint16)
    for r in range(128):
        for j in range(8):
            blk = t[:, :, r, j ^ (r % 8), :]          # [m, c, 16 bytes] = 8 bf16 values
            vals = blk.copy().view(np.uint16)          # [m, c, 8]
            for m in range(rows // 128):
                out[m * 128 + r].reshape(K // 64, 8, 8)[:, j, :] = vals[m]
    return out


@pytest.mark.parametrize("hidden", [2048, 1088], ids=["4splits", "odd_blocks"])
def test_q8_0_tiles_round_trip(hidden):
    # hidden 1088 = 34 blocks: k-splits of 2 blocks (the largest divisor up to 16)
    w = wl.Workload(name="rp", hidden=hidden, num_heads=4, num_kv_heads=2, head_dim=128,
                    layer_type=wl.FULL, window=0, kv_capacity=64, ring=False, batch=1,
                    rope_theta=1e6, seed=61)
    weights = wl.make_weights(w)
    layer = hfa.Layer(hfa.desc_for(w), hfa.weights_to_device(w, weights))
    qkv = layer.hfa_debug_weight_tiles(0).cpu().numpy()
    wo = layer.hfa_debug_weight_tiles(1).cpu().numpy()
    layer.hfa_destroy()
    src_qkv = np.concatenate([weights[n].reshape(-1, hidden // 32, 34) for n in ("wq", "wk", "wv")])
    assert np.array_equal(undo_q8_tiles(qkv, src_qkv.shape[0], hidden), src_qkv)
    src_o = weights["wo"].reshape(hidden, -1, 34)
    assert np.array_equal(undo_q8_tiles(wo, hidden, w.q_rows), src_o)


def test_bf16_tiles_round_trip():
    w = wl.Workload(name="rpb", hidden=512, num_heads=4, num_kv_heads=2, head_dim=128,
                    layer_type=wl.FULL, window=0, kv_capacity=64, ring=False, batch=1,
                    rope_theta=1e6, seed=62, weights_bf16=True, verify_len=16)
    weights = wl.make_weights(w)
    layer = hfa.Layer(hfa.desc_for(w), hfa.weights_to_device(w, weights))
    qkv = layer.hfa_debug_weight_tiles(2).cpu().numpy()
    wo = layer.hfa_debug_weight_tiles(3).cpu().numpy()
    layer.hfa_destroy()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    src_qkv = np.concatenate([bits(weights[n]) for n in ("wq", "wk", "wv")])
    assert np.array_equal(undo_bf16_tiles(qkv, src_qkv.shape[0], w.hidden), src_qkv)
    assert np.array_equal(undo_bf16_tiles(wo, w.hidden, w.q_rows), bits(weights["wo"]))


def test_weight_tiles_of_an_absent_buffer_are_refused():
    w = wl.TINY_SLIDING
    layer = hfa.Layer(hfa.desc_for(w), hfa.weights_to_device(w, wl.make_weights(w)))
    with pytest.raises(hfa.HfaError):
        layer.hfa_debug_weight_tiles(2)  # a Q8_0 layer holds no bf16 tiles
    layer.hfa_destroy()
