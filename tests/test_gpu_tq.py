"""GPU parity of the quantised KV cache (libhfa through its C ABI) against the oracle.

* the library's Lloyd-Max codebook equals the oracle's (both computed from the definition);
* the encode on append: codes and f32 norms equal, byte for byte, to the oracle's encoding
  of the same f32 rows (both take the decisions in double precision; a code may differ only
  for a value within 1e-9 of a cell boundary, where the two independently converged
  codebooks may place it apart -- counted, expected 0), and every other slot unchanged;
* the attention over codes (4-, 5-, 6- and 8-bit, head dims 64 to 512, ring, sliding window,
  softcap, the hybrid raw-K layout) against the oracle on the same seeded codes, within
  relative L2 2e-3 per sequence and head group;
* encode followed by attention against the oracle's encode followed by its attention.
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


def unpack(codes, hd, bits):
    if bits != 4:  # 5-, 6- and 8-bit codes: one byte per element
        return codes.astype(np.int64)
    return np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[:-1] + (hd,)).astype(np.int64)


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_codebook_matches_the_oracle(bits):
    fmt = hfa.TqFormat(128, bits, wl.make_tq_signs(128, 1))
    c, _, _ = oracle.lloyd_max_normal(bits)
    got = fmt.codebook().astype(np.float64)
    assert got.size == c.size and np.max(np.abs(got - c)) < 1e-6
    fmt.destroy()


@pytest.mark.parametrize("hd,bits,ring", [(64, 4, False), (128, 8, False), (256, 4, True),
                                          (512, 8, False), (128, 4, True), (128, 5, False),
                                          (256, 6, True)])
def test_append_codes_equal_the_oracle(hd, bits, ring):
    B, nkv, C = 3, 2, 40
    signs = wl.make_tq_signs(hd, hd + bits)
    fmt = hfa.TqFormat(hd, bits, signs)
    g = torch.Generator().manual_seed(hd * 10 + bits)
    x = torch.randn((B, nkv, hd), generator=g) * torch.rand((B, nkv, 1), generator=g) * 4
    pos = np.array([0, 39, 77], dtype=np.int32) if ring else np.array([0, 17, 39], dtype=np.int32)
    cb, nb = fmt.code_bytes, fmt.blocks
    codes = torch.full((B, nkv, C, cb), 0xA5, dtype=torch.uint8, device="cuda")
    norms = torch.full((B, nkv, C, nb), -1.0, dtype=torch.float32, device="cuda")
    fmt.hfa_tq_append(x.cuda(), torch.from_numpy(pos).cuda(), pos, nkv, C, ring, codes, norms)
    torch.cuda.synchronize()
    codes, norms = codes.cpu().numpy(), norms.cpu().numpy()
    cent, bnd, _ = oracle.lloyd_max_normal(bits)
    ref_c, ref_n = oracle.tq_encode_rows(x.numpy().astype(np.float64), signs, bits, bnd)
    near = 0
    for b, P in enumerate(pos):
        slot = P % C if ring else P
        assert np.array_equal(norms[b, :, slot, :], ref_n[b])
        got, want = unpack(codes[b, :, slot, :], hd, bits), unpack(ref_c[b], hd, bits)
        diff = got != want
        if diff.any():
            # only a value on a boundary (to 1e-9) of the two codebooks may differ
            u = np.stack([oracle.tq_rotate(r, signs) for r in x[b].numpy().astype(np.float64)])
            B_ = min(hd, 256)
            e = u / np.repeat(ref_n[b].astype(np.float64), B_, axis=1)
            dist = np.min(np.abs(e[..., None] - bnd[None, None, 1:-1]), axis=-1)
            assert np.all(dist[diff] < 1e-9) and np.all(np.abs(got - want)[diff] == 1)
            near += int(diff.sum())
        untouched = np.ones(C, dtype=bool)
        untouched[slot] = False
        assert np.all(codes[b][:, untouched] == 0xA5) and np.all(norms[b][:, untouched] == -1.0)
    assert near <= 2
    fmt.destroy()


def _synthetic_tq_cache(B, nkv, C, hd, bits, seed):
    """Seeded synthetic coded cache: codes uniform over the levels, norms ~U[0.5, 1.5]."""
    g = torch.Generator().manual_seed(seed)
    cb = hd // 2 if bits == 4 else hd
    nb = hd // min(hd, 256)
    top = 256 if bits in (4, 8) else 1 << bits  # nibble pairs / bytes over every code
    codes = torch.randint(0, top, (B, nkv, C, cb), generator=g, dtype=torch.uint8)
    norms = torch.rand((B, nkv, C, nb), generator=g) + 0.5
    return codes, norms


def _visible_rows(w, P):
    if w.ring:
        n = min(P + 1, w.kv_capacity)
        return np.arange(n)
    lo = max(0, P - w.window + 1) if w.layer_type == wl.SLIDING else 0
    return np.arange(lo, P + 1)


def _run_tq_attention(w, bits, pos, hybrid=False, seed=0):
    B, nkv, C, hd, nh = len(pos), w.num_kv_heads, w.kv_capacity, w.head_dim, w.num_heads
    signs = wl.make_tq_signs(hd, seed)
    fmt = hfa.TqFormat(hd, bits, signs)
    kc, kn = _synthetic_tq_cache(B, nkv, C, hd, bits, seed + 1)
    vc, vn = _synthetic_tq_cache(B, nkv, C, hd, bits, seed + 2)
    kraw = wl.bf16_normal((B, nkv, C, hd), torch.Generator().manual_seed(seed + 3)) if hybrid else None
    q = torch.randn((B, nh, hd), generator=torch.Generator().manual_seed(seed + 4))
    desc = hfa.attn_desc_for(w)
    max_keys = max(len(_visible_rows(w, int(P))) for P in pos)
    ws = torch.zeros(hfa.hfa_attention_tq_workspace_bytes(desc, B, max_keys), dtype=torch.uint8,
                     device="cuda")
    o = torch.full((B, nh, hd), float("nan"), device="cuda")
    fmt.hfa_attention_decode_tq(desc, q.cuda(), torch.from_numpy(np.asarray(pos, dtype=np.int32)).cuda(),
                                pos, None if hybrid else kc.cuda(), None if hybrid else kn.cuda(),
                                kraw.cuda() if hybrid else None, vc.cuda(), vn.cuda(), ws, o)
    torch.cuda.synchronize()
    o = o.cpu().numpy()
    cent, _, _ = oracle.lloyd_max_normal(bits)
    G = nh // nkv
    worst = 0.0
    for b, P in enumerate(pos):
        rows = _visible_rows(w, int(P))
        for kvh in range(nkv):
            ref = np.stack([oracle.attend_tq(
                q[b, kvh * G + g].numpy(), signs, bits, cent,
                None if hybrid else kc[b, kvh].numpy(), None if hybrid else kn[b, kvh].numpy(),
                vc[b, kvh].numpy(), vn[b, kvh].numpy(), rows, scale=w.attn_scale, softcap=w.softcap,
                k_bf16=kraw[b, kvh] if hybrid else None) for g in range(G)])
            worst = max(worst, rel_l2(o[b, kvh * G:(kvh + 1) * G], ref))
    fmt.destroy()
    print(w.name, bits, "hybrid" if hybrid else "coded", "rel L2", worst)
    assert worst <= REL_L2


def test_attention_over_codes_32k_context_8bit():
    w = wl.FULL_32K.replace(name="tq_full_32k", kv_capacity=32768)
    _run_tq_attention(w, 8, [32767], seed=21)


@pytest.mark.parametrize("hd,bits", [(64, 4), (128, 4), (256, 8), (512, 4), (512, 8), (128, 5),
                                     (64, 6), (512, 6)])
def test_attention_over_codes_head_dims(hd, bits):
    nh = 16 if hd == 512 else 8
    w = wl.Workload(name=f"tq{hd}", hidden=256, num_heads=nh, num_kv_heads=2, head_dim=hd,
                    layer_type=wl.FULL, window=0, kv_capacity=1500, ring=False, batch=3,
                    rope_theta=1e6, seed=22)
    _run_tq_attention(w, bits, [0, 700, 1499], seed=hd + bits)


def test_attention_over_codes_ring_softcap():
    w = wl.Workload(name="tq_ring", hidden=256, num_heads=8, num_kv_heads=4, head_dim=256,
                    layer_type=wl.SLIDING, window=1024, kv_capacity=1024, ring=True, batch=4,
                    rope_theta=1e4, seed=23, softcap=30.0)
    _run_tq_attention(w, 4, [5, 1023, 1024, 5000], seed=31)


def test_attention_over_codes_linear_sliding_window():
    w = wl.Workload(name="tq_sl", hidden=256, num_heads=4, num_kv_heads=2, head_dim=128,
                    layer_type=wl.SLIDING, window=300, kv_capacity=2000, ring=False, batch=2,
                    rope_theta=1e4, seed=24)
    _run_tq_attention(w, 8, [250, 1999], seed=32)


def test_hybrid_raw_keys_coded_values():
    # the pages' hybrid sliding layer: raw keys, 8-bit coded values, head_dim 256
    w = wl.Workload(name="tq_hybrid", hidden=256, num_heads=16, num_kv_heads=8, head_dim=256,
                    layer_type=wl.SLIDING, window=1024, kv_capacity=1024, ring=True, batch=2,
                    rope_theta=1e4, seed=25)
    _run_tq_attention(w, 8, [1500, 600], hybrid=True, seed=33)


@pytest.mark.parametrize("hybrid", [False, True])
def test_group_of_eight_4bit_values(hybrid):
    # eight query heads per KV head (the largest group), 4-bit value codes, head_dim 128,
    # keys coded or raw
    w = wl.Workload(name="tq_g8", hidden=256, num_heads=16, num_kv_heads=2, head_dim=128,
                    layer_type=wl.FULL, window=0, kv_capacity=3000, ring=False, batch=2,
                    rope_theta=1e6, seed=26)
    _run_tq_attention(w, 4, [2999, 77], hybrid=hybrid, seed=34)


def test_hybrid_raw_keys_head_dim_512():
    # raw keys at hd 512 (two norm blocks per value row): the CUDA-core kernel
    w = wl.Workload(name="tq_hyb512", hidden=256, num_heads=16, num_kv_heads=2, head_dim=512,
                    layer_type=wl.FULL, window=0, kv_capacity=700, ring=False, batch=2,
                    rope_theta=1e6, seed=27)
    _run_tq_attention(w, 8, [699, 40], hybrid=True, seed=35)


def test_global_layer_shape_32k_context_4bit():
    # the pages' global layer with a coded cache: 16 query heads over 2 KV heads, hd 512
    w = wl.Workload(name="tq_global", hidden=256, num_heads=16, num_kv_heads=2, head_dim=512,
                    layer_type=wl.FULL, window=0, kv_capacity=32768, ring=False, batch=1,
                    rope_theta=1e6, seed=28)
    _run_tq_attention(w, 4, [32767], seed=36)


@pytest.mark.parametrize("hd,nh,nkv", [(128, 32, 8), (512, 16, 2)])
def test_repeated_calls_are_bit_identical(hd, nh, nkv):
    # the chunk records are merged once, in a fixed order, by the last CTA of each unit
    # (one level at hd 128 with 19 chunks, two levels at hd 512): every call gives the
    # same bits, however the CTAs happen to finish
    C, B, bits = 8192, 1, 8
    w = wl.Workload(name="tq_det", hidden=256, num_heads=nh, num_kv_heads=nkv, head_dim=hd,
                    layer_type=wl.FULL, window=0, kv_capacity=C, ring=False, batch=B,
                    rope_theta=1e6, seed=29)
    desc = hfa.attn_desc_for(w)
    fmt = hfa.TqFormat(hd, bits, wl.make_tq_signs(hd, 37))
    kc, kn = _synthetic_tq_cache(B, nkv, C, hd, bits, 38)
    vc, vn = _synthetic_tq_cache(B, nkv, C, hd, bits, 39)
    kc, kn, vc, vn = kc.cuda(), kn.cuda(), vc.cuda(), vn.cuda()
    q = torch.randn((B, nh, hd), generator=torch.Generator().manual_seed(40)).cuda()
    pos = np.array([C - 1], dtype=np.int32)
    posd = torch.from_numpy(pos).cuda()
    ws = torch.zeros(hfa.hfa_attention_tq_workspace_bytes(desc, B, C), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for _ in range(6):
        o = torch.full((B, nh, hd), float("nan"), device="cuda")
        fmt.hfa_attention_decode_tq(desc, q, posd, pos, kc, kn, None, vc, vn, ws, o)
        torch.cuda.synchronize()
        outs.append(o.cpu())
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))
    assert torch.isfinite(outs[0]).all()
    fmt.destroy()


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_encode_then_attend_matches_the_oracle_pipeline(bits):
    # f32 K/V rows appended one position at a time by the library's encoder, then attended;
    # the oracle encodes the same rows itself and attends over its own codes
    B, nkv, nh, hd, C = 1, 2, 4, 128, 96
    signs = wl.make_tq_signs(hd, 40 + bits)
    fmt = hfa.TqFormat(hd, bits, signs)
    g = torch.Generator().manual_seed(41 + bits)
    K = torch.randn((C, B, nkv, hd), generator=g)
    V = torch.randn((C, B, nkv, hd), generator=g)
    q = torch.randn((B, nh, hd), generator=g)
    kc = torch.zeros((B, nkv, C, fmt.code_bytes), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    kn = torch.zeros((B, nkv, C, fmt.blocks), device="cuda")
    vn = torch.zeros_like(kn)
    for p in range(C):
        pos = np.array([p], dtype=np.int32)
        pd = torch.from_numpy(pos).cuda()
        fmt.hfa_tq_append(K[p].cuda().contiguous(), pd, pos, nkv, C, False, kc, kn)
        fmt.hfa_tq_append(V[p].cuda().contiguous(), pd, pos, nkv, C, False, vc, vn)
    w = wl.Workload(name="tq_e2e", hidden=256, num_heads=nh, num_kv_heads=nkv, head_dim=hd,
                    layer_type=wl.FULL, window=0, kv_capacity=C, ring=False, batch=B,
                    rope_theta=1e6, seed=42)
    desc = hfa.attn_desc_for(w)
    P = C - 1
    ws = torch.zeros(hfa.hfa_attention_tq_workspace_bytes(desc, B, C), dtype=torch.uint8, device="cuda")
    o = torch.empty((B, nh, hd), device="cuda")
    fmt.hfa_attention_decode_tq(desc, q.cuda(), torch.tensor([P], dtype=torch.int32, device="cuda"),
                                np.array([P], dtype=np.int32), kc, kn, None, vc, vn, ws, o)
    torch.cuda.synchronize()
    cent, bnd, _ = oracle.lloyd_max_normal(bits)
    rkc, rkn = oracle.tq_encode_rows(K[:, 0].numpy().astype(np.float64).transpose(1, 0, 2), signs, bits, bnd)
    rvc, rvn = oracle.tq_encode_rows(V[:, 0].numpy().astype(np.float64).transpose(1, 0, 2), signs, bits, bnd)
    rows = np.arange(C)
    for kvh in range(nkv):
        for gq in range(nh // nkv):
            h = kvh * (nh // nkv) + gq
            ref = oracle.attend_tq(q[0, h].numpy(), signs, bits, cent, rkc[kvh], rkn[kvh], rvc[kvh],
                                   rvn[kvh], rows)
            assert rel_l2(o[0, h].cpu().numpy(), ref) <= REL_L2
    fmt.destroy()
