"""The allocation-free attention entry point against the workspace one (GPU).

hfa_attention_decode_noalloc exists for callers that cannot allocate device memory
where they run attention (an engine that fixes its device memory at start-up, a plugin
whose host owns the allocator, code that must not let cudaMalloc synchronise the
device); it keeps its scratch in a static device array.  This file is collected last on
purpose.  It checks, through the C ABI, two calls in a row against hfa_attention_decode
with a caller-allocated workspace, within the parity tolerance of the other tests, and
that a batch too large for the static scratch is refused.
"""
import numpy as np
import pytest
import torch

from quantized_attention_layer_gb300 import hfa, workloads as wl

from parity import REL_L2, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_layer_gb300 import build
    build.build()


def _inputs(w, pos, seed):
    kv = wl.make_kv_cache(w)
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((len(pos), w.num_heads, w.head_dim), generator=g).cuda()
    posd = torch.from_numpy(np.asarray(pos, dtype=np.int32)).cuda()
    return q, posd, kv["k_cache"].cuda(), kv["v_cache"].cuda()


@pytest.mark.parametrize("w,calls", [
    (wl.FULL_32K, ([32767], [20000])),
    (wl.Workload(name="ring_b4", hidden=256, num_heads=8, num_kv_heads=4, head_dim=256,
                 layer_type=wl.SLIDING, window=1024, kv_capacity=1024, ring=True, batch=4,
                 rope_theta=1e4, seed=81), ([1023, 5000, 77, 3000], [1500, 2047, 1024, 9999])),
], ids=["full_32k", "ring_hd256_b4"])
def test_noalloc_matches_workspace_entry_point_twice(w, calls):
    desc = hfa.attn_desc_for(w)
    for i, pos in enumerate(calls):
        q, posd, kc, vc = _inputs(w, pos, seed=100 + i)
        ws = torch.zeros(hfa.hfa_attention_workspace_bytes(desc, len(pos)), dtype=torch.uint8,
                         device="cuda")
        o_ref = torch.empty_like(q)
        hfa.hfa_attention_decode(desc, q, posd, pos, kc, vc, ws, o_ref)
        o = torch.full_like(q, float("nan"))
        hfa.hfa_attention_decode_noalloc(desc, q, posd, pos, kc, vc, o)
        torch.cuda.synchronize()
        assert torch.isfinite(o).all()
        for b in range(len(pos)):
            assert rel_l2(o[b].cpu().numpy(), o_ref[b].cpu().numpy()) <= REL_L2


def test_noalloc_refuses_a_batch_beyond_its_static_scratch():
    w = wl.Workload(name="huge", hidden=256, num_heads=8, num_kv_heads=8, head_dim=256,
                    layer_type=wl.FULL, window=0, kv_capacity=64, ring=False, batch=512,
                    rope_theta=1e4, seed=82)
    desc = hfa.attn_desc_for(w)
    pos = np.full(512, 10, dtype=np.int32)
    q = torch.zeros((512, 8, 256), device="cuda")
    kc = torch.zeros((512, 8, 64, 256), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    with pytest.raises(hfa.HfaError) as e:
        hfa.hfa_attention_decode_noalloc(desc, q, torch.from_numpy(pos).cuda(), pos, kc, kc, o)
    assert e.value.status == hfa.HFA_ERANGE
    assert "static scratch" in str(e.value)


def test_noalloc_allocates_nothing_after_its_first_call():
    # the first call on a device looks up the static array (and may load the module that
    # holds it); after that, free device memory must not move across calls
    w = wl.FULL_32K.replace(kv_capacity=4096, seq_pos=4095)
    desc = hfa.attn_desc_for(w)
    pos = [4095]
    q, posd, kc, vc = _inputs(w, pos, seed=7)
    o = torch.empty_like(q)
    hfa.hfa_attention_decode_noalloc(desc, q, posd, pos, kc, vc, o)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        hfa.hfa_attention_decode_noalloc(desc, q, posd, pos, kc, vc, o)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.isfinite(o).all()
