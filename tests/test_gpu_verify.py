"""GPU parity of the multi-token verify block (tcgen05 projections) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_layer_gb300 import hfa, workloads as wl

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


def test_verify_block_global_layer_hd512_32k():
    # the pages' global layer (16 query heads of 512 dims over 2 KV heads, no V projection,
    # RoPE frequency factors, post-attention norm), 8 tokens at the end of a 32K context
    w = wl.VERIFY_GLOBAL
    _case(w, w.verify_len, w.base_pos)


def test_verify_block_hd512_sliding_softcap_ragged():
    # 312 visible keys (not a multiple of the 32-key stage), the window's first key inside
    # a stage, two CTAs per key chunk each writing half of the output dims
    w = wl.Workload(name="ver512s", hidden=1024, num_heads=8, num_kv_heads=2, head_dim=512,
                    layer_type=wl.SLIDING, window=300, kv_capacity=1300, ring=False, batch=1,
                    rope_theta=1e4, seed=103, weights_bf16=True, verify_len=16, base_pos=0,
                    softcap=30.0)
    _case(w, 13, 1111)


def test_verify_block_hd512_short_context_variants():
    # fewer keys than one stage per chunk; V projected and unit-normed
    w = wl.Workload(name="ver512v", hidden=512, num_heads=4, num_kv_heads=1, head_dim=512,
                    layer_type=wl.FULL, window=0, kv_capacity=96, ring=False, batch=1,
                    rope_theta=1e6, seed=104, weights_bf16=True, verify_len=16, base_pos=0,
                    v_unit_norm=True, rope_freq_factors=True, post_norm=True)
    _case(w, 16, 20)


@pytest.mark.parametrize("w", [wl.VERIFY_L16, wl.VERIFY_GLOBAL], ids=lambda w: w.name)
def test_verify_block_repeats_bit_for_bit(w):
    # no atomics on the data path: two runs on the same inputs agree in every bit (at hd
    # 512 the output also passes through the TMEM accumulator and its rare rescales)
    weights = wl.make_weights(w)
    x = wl.make_x(w, rows=w.verify_len)
    kv = wl.make_kv_cache(w)
    a = run_gpu_verify(w, weights, x, w.base_pos, kv)
    b = run_gpu_verify(w, weights, x, w.base_pos, kv)
    for key in ("out_bf16", "q", "k", "v", "attn", "out"):
        assert torch.equal(a[key], b[key]), key


# ---------------------------------------------------------------- the drafter's blocks

def test_bidirectional_block_full_size():
    w = wl.VERIFY_L16.replace(name="ver_bidir", block_bidir=True)
    _case(w, w.verify_len, w.base_pos)


@pytest.mark.parametrize("hd", [64, 128, 256, 512])
def test_bidirectional_block_head_dims(hd):
    w = wl.Workload(name=f"bidir{hd}", hidden=1024, num_heads=8, num_kv_heads=2, head_dim=hd,
                    layer_type=wl.FULL, window=0, kv_capacity=700, ring=False, batch=1,
                    rope_theta=1e6, seed=99, weights_bf16=True, verify_len=16, base_pos=0,
                    block_bidir=True)
    _case(w, 11, 350)


def _drafter_step(w, S, L, base):
    """Context rows then the block, on the GPU and in the oracle; both checked."""
    from parity import bits_of, check_verify, flip_bound, rel_l2
    weights = wl.make_weights(w)
    g = torch.Generator().manual_seed(w.seed + 5)
    x_ctx = wl.bf16_normal((S, w.hidden), g)
    x = wl.make_x(w, rows=L)
    kv = wl.make_kv_cache(w)
    layer = hfa.Layer(hfa.desc_for(w, debug_taps=True), hfa.weights_to_device(w, weights))
    kc, vc = kv["k_cache"].cuda(), kv["v_cache"].cuda()
    layer.hfa_ctx_append(x_ctx.cuda(), base, kc, vc)
    taps = layer.hfa_debug_taps(S)
    torch.cuda.synchronize()
    ref_ctx = oracle.ctx_append(w, weights, x_ctx, base, kv["k_cache"], kv["v_cache"])
    n_flip, expected = 0, 0.0
    for key in ("k", "v"):
        got = taps[key].cpu().numpy()
        assert rel_l2(got, ref_ctx[key]) <= 2e-3
        cache = bits_of((kc if key == "k" else vc).cpu()).reshape(w.num_kv_heads, w.kv_capacity, w.head_dim)
        own = np.array([oracle.f64_to_bf16(float(t)) for t in got.ravel()], dtype=np.uint16)
        rows = cache[:, base:base + S, :].transpose(1, 0, 2).ravel()
        assert np.array_equal(rows, own), "context bytes are not the RNE of the kernel's fp32"
        ref_rows = ref_ctx[key + "_cache"].reshape(cache.shape)[:, base:base + S, :].transpose(1, 0, 2).ravel()
        n_flip += int((rows != ref_rows).sum())
        expected += flip_bound(got, ref_ctx[key])[0]
    assert n_flip <= expected + 4 * np.sqrt(expected) + 4
    kv_mid = {"k_cache": kc.cpu(), "v_cache": vc.cpu()}
    out = torch.empty((L, w.hidden), dtype=torch.bfloat16, device="cuda")
    layer.hfa_verify_block(x.cuda(), base + S, kc, vc, out)
    layer.hfa_check_device_status()
    gpu = {"out_bf16": out, "k_cache": kc, "v_cache": vc}
    gpu.update(layer.hfa_debug_taps(L))
    torch.cuda.synchronize()
    gpu = {k: v.cpu() for k, v in gpu.items()}
    layer.hfa_destroy()
    kc_ref = torch.from_numpy(ref_ctx["k_cache"].view(np.int16)).view(torch.bfloat16)
    vc_ref = torch.from_numpy(ref_ctx["v_cache"].view(np.int16)).view(torch.bfloat16)
    ref = oracle.verify_block(w, weights, x, base + S, kc_ref, vc_ref)
    return check_verify(w, base + S, gpu, ref, kv_mid)


def test_drafter_step_full_layer():
    # context rows, then a bidirectional block with the drafter's 1/sqrt(hd) scale
    w = wl.Workload(name="draft_full", hidden=1024, num_heads=8, num_kv_heads=2, head_dim=128,
                    layer_type=wl.FULL, window=0, kv_capacity=600, ring=False, batch=1,
                    rope_theta=1e6, seed=101, weights_bf16=True, verify_len=16, base_pos=0,
                    block_bidir=True, attn_scale=128 ** -0.5)
    _drafter_step(w, S=5, L=8, base=300)


def test_drafter_step_sliding_layer_stays_causal():
    w = wl.Workload(name="draft_sl", hidden=1024, num_heads=8, num_kv_heads=4, head_dim=256,
                    layer_type=wl.SLIDING, window=64, kv_capacity=500, ring=False, batch=1,
                    rope_theta=1e4, seed=102, weights_bf16=True, verify_len=16, base_pos=0,
                    block_bidir=True, attn_scale=256 ** -0.5)
    _drafter_step(w, S=16, L=8, base=200)


def test_drafter_step_global_layer_hd512():
    # context rows (at most max_verify_len = 8) through the 512-wide K/V epilogue (no V
    # projection), then the block
    w = wl.GLOBAL_32K.replace(name="draft_global", kv_capacity=2000, weights_bf16=True,
                              verify_len=8, seq_pos=None, block_bidir=True,
                              attn_scale=512 ** -0.5)
    _drafter_step(w, S=8, L=8, base=1500)
