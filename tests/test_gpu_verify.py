"""GPU parity of the multi-token verify block (tcgen05 projections) against the oracle."""
import pytest
import torch

import oracle
from quantized_attention_layer_gb300 import workloads as wl

from parity import check_verify, run_gpu_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_layer_gb300 import build
    build.build()
    oracle.build()


def _case(w, L, base):
    weights = wl.make_weights(w)
    x = wl.make_x(w, rows=L)
    kv = wl.make_kv_cache(w)
    gpu = run_gpu_verify(w, weights, x, base, kv)
    ref = oracle.verify_block(w, weights, x, base, kv["k_cache"], kv["v_cache"])
    return check_verify(w, base, gpu, ref, kv)


def test_verify_block_full_size():
    w = wl.VERIFY_L16
    _case(w, w.verify_len, w.base_pos)


@pytest.mark.parametrize("L", [1, 5, 16])
def test_verify_block_small_lengths(L):
    w = wl.Workload(name=f"ver{L}", hidden=1024, num_heads=8, num_kv_heads=2, head_dim=128,
                    layer_type=wl.FULL, window=0, kv_capacity=700, ring=False, batch=1,
                    rope_theta=1e6, seed=90 + L, weights_bf16=True, verify_len=16, base_pos=0)
    _case(w, L, 300)


def test_verify_block_sliding_window_softcap_hd64():
    w = wl.Workload(name="ver_sl", hidden=512, num_heads=8, num_kv_heads=4, head_dim=64,
                    layer_type=wl.SLIDING, window=100, kv_capacity=600, ring=False, batch=1,
                    rope_theta=1e4, seed=95, weights_bf16=True, verify_len=16, base_pos=0,
                    softcap=30.0)
    _case(w, 12, 450)


def test_verify_block_at_position_zero():
    w = wl.Workload(name="ver0", hidden=512, num_heads=4, num_kv_heads=2, head_dim=128,
                    layer_type=wl.FULL, window=0, kv_capacity=64, ring=False, batch=1,
                    rope_theta=1e6, seed=96, weights_bf16=True, verify_len=16, base_pos=0)
    _case(w, 16, 0)


@pytest.mark.parametrize("k_eq_v,ff,post", [(True, True, True), (False, False, True),
                                           (True, False, False)], ids=["all", "post", "keqv"])
def test_verify_block_gemma_variants(k_eq_v, ff, post):
    # no V projection, RoPE frequency factors, post-attention RMSNorm (the pages' global
    # layer), each against the oracle
    w = wl.Workload(name="ver_var", hidden=1024, num_heads=8, num_kv_heads=2, head_dim=128,
                    layer_type=wl.FULL, window=0, kv_capacity=700, ring=False, batch=1,
                    rope_theta=1e6, seed=97, weights_bf16=True, verify_len=16, base_pos=0,
                    k_eq_v=k_eq_v, rope_freq_factors=ff, post_norm=post)
    _case(w, 13, 400)


def test_verify_block_hd256_cluster_across_row_tiles():
    # a 256-wide head spans two 128-row GEMM tiles: the k-split cluster holds both tiles'
    # splits, and the head epilogue adds rows from either tile's CTAs
    w = wl.Workload(name="ver256", hidden=1024, num_heads=8, num_kv_heads=2, head_dim=256,
                    layer_type=wl.FULL, window=0, kv_capacity=600, ring=False, batch=1,
                    rope_theta=1e6, seed=98, weights_bf16=True, verify_len=16, base_pos=0)
    _case(w, 16, 500)


def test_verify_block_sliding_hd256_softcap_short_block():
    w = wl.Workload(name="ver256s", hidden=512, num_heads=4, num_kv_heads=1, head_dim=256,
                    layer_type=wl.SLIDING, window=200, kv_capacity=900, ring=False, batch=1,
                    rope_theta=1e4, seed=99, weights_bf16=True, verify_len=16, base_pos=0,
                    softcap=30.0)
    _case(w, 7, 850)


@pytest.mark.parametrize("window,softcap", [(100, 30.0), (40, 0.0)], ids=["w100cap", "w40"])
def test_verify_block_hd128_sliding(window, softcap):
    # head_dim 128 runs the tensor-core attention: window starts inside a 64-key stage,
    # keys before the window and after each row's position masked, with and without softcap
    w = wl.Workload(name=f"ver128s{window}", hidden=1024, num_heads=8, num_kv_heads=2,
                    head_dim=128, layer_type=wl.SLIDING, window=window, kv_capacity=700,
                    ring=False, batch=1, rope_theta=1e4, seed=101, weights_bf16=True,
                    verify_len=16, base_pos=0, softcap=softcap)
    _case(w, 11, 517)


def test_verify_block_repeats_bit_for_bit():
    # no atomics on the data path: two runs on the same inputs agree in every bit
    w = wl.VERIFY_L16
    weights = wl.make_weights(w)
    x = wl.make_x(w, rows=w.verify_len)
    kv = wl.make_kv_cache(w)
    a = run_gpu_verify(w, weights, x, w.base_pos, kv)
    b = run_gpu_verify(w, weights, x, w.base_pos, kv)
    for key in ("out_bf16", "q", "k", "v", "attn", "out"):
        assert torch.equal(a[key], b[key]), key
