"""GPU parity of the decode step (libhfa through its C ABI) against the fp64 oracle.

Cases: the four decode workloads at full size, small cases that span several GEMV
tiles and attention stages with ragged tails, and the degenerate cases of the method
(one visible key, a ring that has not wrapped, V unit norm, softcap, mixed positions).
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_layer_gb300 import hfa, workloads as wl

from parity import REL_L2, bits_of, check_decode, rel_l2, run_gpu_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_layer_gb300 import build
    build.build()
    oracle.build()


def _case(w: wl.Workload, pos=None):
    weights = wl.make_weights(w)
    x = wl.make_x(w)
    kv = wl.make_kv_cache(w)
    pos = wl.make_positions(w) if pos is None else np.asarray(pos, dtype=np.int32)
    gpu = run_gpu_decode(w, weights, x, pos, kv)
    ref = oracle.decode_step(w, weights, x, pos, kv["k_cache"], kv["v_cache"])
    return check_decode(w, pos, gpu, ref, kv), gpu, ref


@pytest.mark.parametrize("w", [wl.TINY_SLIDING, wl.FULL_32K, wl.SLIDING_B16, wl.FULL_128K_B4],
                         ids=lambda w: w.name)
def test_full_size_workloads(w):
    report, _, _ = _case(w)
    print(w.name, report)


SMALL = wl.Workload(name="small_full", hidden=512, num_heads=8, num_kv_heads=2, head_dim=128,
                    layer_type=wl.FULL, window=0, kv_capacity=1000, ring=False, batch=3,
                    rope_theta=1e6, seed=31, seq_pos_range=(0, 999))


def test_small_full_ragged_positions():
    # positions are not multiples of the 64-key stage; the chunks end mid-stage
    _case(SMALL, pos=[0, 77, 999])


def test_one_visible_key_returns_v_exactly():
    w = SMALL.replace(batch=1)
    report, gpu, _ = _case(w, pos=[0])
    # with a single key the attention output is the appended (bf16) V row itself
    v_row = oracle.bf16_to_f64(bits_of(gpu["v_cache"]).reshape(1, 2, 1000, 128)[0, :, 0, :])
    attn = gpu["attn"].numpy()[0]
    for h in range(8):
        assert np.array_equal(attn[h].astype(np.float64), v_row[h // 4])


@pytest.mark.parametrize("hd", [64, 256])
def test_other_head_dims_sliding_linear(hd):
    w = wl.Workload(name=f"sl{hd}", hidden=512, num_heads=4, num_kv_heads=2, head_dim=hd,
                    layer_type=wl.SLIDING, window=200, kv_capacity=700, ring=False, batch=2,
                    rope_theta=1e4, seed=40 + hd, seq_pos_range=(0, 699))
    _case(w, pos=[150, 613])


# The pages' global layer (hd 512, 16/2 heads, k_eq_v, frequency factors, post norm) at 32K;
# hidden 2816 splits the QKV rows into k-splits of 11 blocks.
GLOBAL_32K = wl.GLOBAL_32K


def test_global_layer_hd512_32k_context():
    _case(GLOBAL_32K)


def test_hd512_ragged_batch_plain_layer():
    # three sequences of 1, 7 and 40 key tiles of 32 keys, with V projected and no variants
    w = GLOBAL_32K.replace(name="hd512_b3", hidden=1024, kv_capacity=1300, batch=3,
                           k_eq_v=False, rope_freq_factors=False, post_norm=False,
                           seq_pos=None, softcap=30.0)
    _case(w, pos=[0, 200, 1279])


def test_fewer_key_tiles_than_ctas_with_many_units():
    # 16 sequences of 1..6 key tiles (104 tiles for 152 CTAs): CTAs without tiles sit both
    # inside units and on their first tiles; every unit's records must combine exactly once
    w = wl.Workload(name="units16", hidden=512, num_heads=4, num_kv_heads=2, head_dim=64,
                    layer_type=wl.FULL, window=0, kv_capacity=700, ring=False, batch=16,
                    rope_theta=1e6, seed=45, seq_pos_range=(0, 699))
    _case(w, pos=[0, 130, 260, 390, 520, 650, 3, 140, 300, 450, 600, 699, 77, 255, 256, 511])


def test_ring_before_and_after_wrap():
    w = wl.Workload(name="ring", hidden=256, num_heads=4, num_kv_heads=1, head_dim=64,
                    layer_type=wl.SLIDING, window=256, kv_capacity=256, ring=True, batch=4,
                    rope_theta=1e4, seed=50, seq_pos_range=(0, 2000))
    _case(w, pos=[5, 255, 256, 1999])


def test_v_unit_norm_and_softcap():
    w = SMALL.replace(v_unit_norm=True, softcap=20.0, batch=2)
    _case(w, pos=[500, 999])


def test_gqa_group_five_like_the_long_context_layer():
    w = wl.Workload(name="g5", hidden=640, num_heads=10, num_kv_heads=2, head_dim=128,
                    layer_type=wl.FULL, window=0, kv_capacity=3000, ring=False, batch=4,
                    rope_theta=1e6, seed=60, softcap=50.0, seq_pos_range=(2000, 2999))
    _case(w)


def test_host_entry_point_matches_device_entry_point():
    w = SMALL.replace(batch=2)
    weights = wl.make_weights(w)
    x = wl.make_x(w)
    pos = np.array([10, 900], dtype=np.int32)
    kv = wl.make_kv_cache(w)
    dev = run_gpu_decode(w, weights, x, pos, kv, debug_taps=False)
    layer = hfa.Layer(hfa.desc_for(w), hfa.weights_to_device(w, weights))
    kc, vc = kv["k_cache"].cuda(), kv["v_cache"].cuda()
    out_h = torch.empty((2, w.hidden), dtype=torch.bfloat16).pin_memory()
    layer.hfa_decode_step_host(x.pin_memory(), pos, kc, vc, out_h)
    assert rel_l2(oracle.bf16_to_f64(bits_of(out_h)), oracle.bf16_to_f64(bits_of(dev["out_bf16"]))) < 1e-5
    layer.hfa_destroy()


def test_repeated_steps_reset_their_accumulators():
    w = SMALL.replace(batch=2)
    weights = wl.make_weights(w)
    layer = hfa.Layer(hfa.desc_for(w, debug_taps=True), hfa.weights_to_device(w, weights))
    x = wl.make_x(w)
    pos = np.array([100, 200], dtype=np.int32)
    kv = wl.make_kv_cache(w)
    outs = []
    for _ in range(3):
        r = run_gpu_decode(w, weights, x, pos, kv, debug_taps=True, layer=layer)
        outs.append(r["out"].numpy())
    # every sum of the step is added in a fixed order (split-K partials, attention
    # records): repeated steps agree bit for bit
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    layer.hfa_destroy()


def test_successor_prefetch_leaves_results_unchanged():
    w = SMALL.replace(batch=2)
    weights = wl.make_weights(w)
    dev_w = hfa.weights_to_device(w, weights)
    a = hfa.Layer(hfa.desc_for(w, debug_taps=True), dev_w)
    b = hfa.Layer(hfa.desc_for(w, debug_taps=True), dev_w)
    x = wl.make_x(w)
    pos = np.array([100, 999], dtype=np.int32)
    kv = wl.make_kv_cache(w)
    plain = run_gpu_decode(w, weights, x, pos, kv, debug_taps=True, layer=a)
    a.hfa_set_successor(b)
    hinted = run_gpu_decode(w, weights, x, pos, kv, debug_taps=True, layer=a)
    for key in ("out_bf16", "q", "k", "v", "attn", "out", "k_cache", "v_cache"):
        assert torch.equal(hinted[key], plain[key]), key
    other = wl.Workload(name="other", hidden=512, num_heads=4, num_kv_heads=2, head_dim=128,
                        layer_type=wl.FULL, window=0, kv_capacity=64, ring=False, batch=1,
                        rope_theta=1e6, seed=32, seq_pos=10)
    c = hfa.Layer(hfa.desc_for(other), hfa.weights_to_device(other, wl.make_weights(other)))
    with pytest.raises(hfa.HfaError) as e:
        a.hfa_set_successor(c)
    assert e.value.status == hfa.HFA_EINVAL
    a.hfa_set_successor(None)
    for L in (a, b, c):
        L.hfa_destroy()


def test_rejected_calls_touch_nothing():
    w = SMALL.replace(batch=1)
    weights = wl.make_weights(w)
    layer = hfa.Layer(hfa.desc_for(w), hfa.weights_to_device(w, weights))
    kv = wl.make_kv_cache(w)
    kc, vc = kv["k_cache"].cuda(), kv["v_cache"].cuda()
    x = wl.make_x(w).cuda()
    out = torch.zeros((1, w.hidden), dtype=torch.bfloat16, device="cuda")
    bad_pos = np.array([w.kv_capacity], dtype=np.int32)
    with pytest.raises(hfa.HfaError) as e:
        layer.hfa_decode_step(x, torch.from_numpy(bad_pos).cuda(), bad_pos, kc, vc, out)
    assert e.value.status == hfa.HFA_ERANGE
    with pytest.raises(hfa.HfaError) as e:
        pos = np.array([3], dtype=np.int32)
        layer.hfa_decode_step(x.view(-1)[1:].view(torch.bfloat16)[: w.hidden].view(1, -1),
                              torch.from_numpy(pos).cuda(), pos, kc, vc, out)
    assert e.value.status == hfa.HFA_EINVAL
    torch.cuda.synchronize()
    assert torch.equal(kc.cpu().view(torch.int16), kv["k_cache"].view(torch.int16))
    assert torch.count_nonzero(out).item() == 0
    layer.hfa_check_device_status()
    layer.hfa_destroy()


def test_bounded_wait_gives_up_reports_and_recovers():
    # the failure path without a fault: CTA 0's consumers wait on a barrier nothing
    # completes; the wait gives up after its bound, the step ends with its error word
    # set, hfa_check_device_status reports it and resets, and the next step is correct
    w = SMALL.replace(batch=2)
    weights = wl.make_weights(w)
    layer = hfa.Layer(hfa.desc_for(w, debug_taps=True), hfa.weights_to_device(w, weights))
    x = wl.make_x(w)
    pos = np.array([100, 999], dtype=np.int32)
    kv = wl.make_kv_cache(w)
    before = run_gpu_decode(w, weights, x, pos, kv, debug_taps=True, layer=layer)
    kc, vc = kv["k_cache"].cuda(), kv["v_cache"].cuda()
    out = torch.empty((len(pos), w.hidden), dtype=torch.bfloat16, device="cuda")
    layer.hfa_debug_stall_next_step()
    layer.hfa_decode_step(x.cuda(), torch.from_numpy(pos).cuda(), pos, kc, vc, out)
    with pytest.raises(hfa.HfaError) as e:
        layer.hfa_check_device_status()
    assert e.value.status == hfa.HFA_EDEVICE
    assert "bounded wait" in str(e.value)
    layer.hfa_check_device_status()  # the record was cleared
    # steps after the reset: the same result as before the stall, bit for bit
    for _ in range(2):
        after = run_gpu_decode(w, weights, x, pos, kv, debug_taps=True, layer=layer)
        for key in ("out_bf16", "attn", "out"):
            assert torch.equal(after[key], before[key]), key
    layer.hfa_destroy()


@pytest.mark.parametrize("k_eq_v,ff,post", [(True, True, True), (True, False, False),
                                           (False, True, False), (False, False, True)],
                         ids=["all", "keqv", "ff", "post"])
def test_gemma_variants_full_layer(k_eq_v, ff, post):
    # no V projection (V = unit-normed raw K), RoPE frequency factors, post-attention
    # RMSNorm: the pages' global-layer variants, each against the oracle
    w = SMALL.replace(name="small_var", k_eq_v=k_eq_v, rope_freq_factors=ff, post_norm=post)
    _case(w, pos=[0, 77, 999])


def test_post_norm_batch_of_sixteen_sliding_ring():
    # 16 rows: every CTA's share of the outputs straddles rows, so the row statistic is
    # summed over the CTAs that share each row
    w = wl.SLIDING_B16.replace(name="b16_post", post_norm=True, rope_freq_factors=True)
    _case(w)


def test_post_norm_off_again_and_factors_cleared():
    w = SMALL.replace(name="small_toggle", post_norm=True, rope_freq_factors=True)
    weights = wl.make_weights(w)
    layer = hfa.Layer(hfa.desc_for(w, debug_taps=True), hfa.weights_to_device(w, weights))
    x = wl.make_x(w)
    pos = np.array([5, 600, 999], dtype=np.int32)
    kv = wl.make_kv_cache(w)
    layer.hfa_set_post_norm(None)
    layer.hfa_set_rope_freq_factors(None)
    gpu = run_gpu_decode(w, weights, x, pos, kv, debug_taps=True, layer=layer)
    plain = SMALL.replace(name="small_plain")
    ref = oracle.decode_step(plain, weights, x, pos, kv["k_cache"], kv["v_cache"])
    check_decode(plain, pos, gpu, ref, kv)
    with pytest.raises(hfa.HfaError) as e:
        layer.hfa_set_rope_freq_factors(np.zeros(w.head_dim // 2, dtype=np.float32))
    assert e.value.status == hfa.HFA_EINVAL
    layer.hfa_destroy()
