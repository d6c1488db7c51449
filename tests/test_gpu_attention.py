"""GPU parity of the attention step alone (hfa_attention_decode) against the oracle.

Queries are drawn directly (unit-RMS rows like the output of the per-head norm, scaled
so the logits span the range of the layer's), the cache is the seeded bf16 cache, and
the oracle attends over the explicit list of visible slots of each sequence.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_layer_gb300 import hfa, workloads as wl

from parity import REL_L2, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_layer_gb300 import build
    build.build()
    oracle.build()


def _visible_slots(w, P):
    sl = w.layer_type == wl.SLIDING
    return [s for s in range(w.kv_capacity)
            if (p := oracle.slot_position(s, P, w.kv_capacity, w.ring)) >= 0
            and oracle.key_visible(p, P, sl, w.window)]


def run_attention(w, pos, q_scale=1.0, seed=0, workspace=None):
    kv = wl.make_kv_cache(w)
    B = len(pos)
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, w.num_heads, w.head_dim), generator=g) * q_scale
    desc = hfa.attn_desc_for(w)
    if workspace is None:
        nbytes = hfa.hfa_attention_workspace_bytes(desc, B)
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    o = torch.empty((B, w.num_heads, w.head_dim), device="cuda")
    posd = torch.from_numpy(np.asarray(pos, dtype=np.int32)).cuda()
    kc, vc = kv["k_cache"].cuda(), kv["v_cache"].cuda()
    hfa.hfa_attention_decode(desc, q.cuda(), posd, pos, kc, vc, workspace, o)
    torch.cuda.synchronize()
    assert int(workspace[:4].view(torch.int32).item()) == 0, "device status word set"
    kb = oracle.bf16_bits(kv["k_cache"]).reshape(B, w.num_kv_heads, w.kv_capacity, w.head_dim)
    vb = oracle.bf16_bits(kv["v_cache"]).reshape(kb.shape)
    worst = 0.0
    for b, P in enumerate(pos):
        rows = np.array(_visible_slots(w, int(P)), dtype=np.int64)
        for h in range(w.num_heads):
            kvh = h // w.group
            ref, _ = oracle.attend(q[b, h].double().numpy(), kb[b, kvh], vb[b, kvh], rows,
                                   scale=w.attn_scale, softcap=w.softcap)
            worst = max(worst, rel_l2(o[b, h].cpu().numpy(), ref))
    return worst, workspace


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_attention_alone_sliding_and_full(hd):
    w = wl.Workload(name=f"a{hd}", hidden=256, num_heads=8, num_kv_heads=2, head_dim=hd,
                    layer_type=wl.SLIDING, window=300, kv_capacity=1100, ring=False, batch=3,
                    rope_theta=1e4, seed=70 + hd)
    worst, _ = run_attention(w, [0, 299, 1099], q_scale=1.0)
    assert worst <= REL_L2, worst
    w = w.replace(layer_type=wl.FULL, window=0, softcap=30.0)
    worst, _ = run_attention(w, [63, 64, 1099], q_scale=2.0)
    assert worst <= REL_L2, worst


def test_attention_alone_reuses_its_workspace():
    w = wl.Workload(name="ws", hidden=256, num_heads=4, num_kv_heads=1, head_dim=128,
                    layer_type=wl.FULL, window=0, kv_capacity=5000, ring=False, batch=2,
                    rope_theta=1e4, seed=77)
    worst1, ws = run_attention(w, [4999, 1234], seed=1)
    worst2, _ = run_attention(w, [4321, 17], seed=2, workspace=ws)
    assert worst1 <= REL_L2 and worst2 <= REL_L2


def test_attention_alone_at_the_32k_layer_size():
    w = wl.FULL_32K
    worst, _ = run_attention(w, [32767], q_scale=1.0)
    assert worst <= REL_L2, worst
