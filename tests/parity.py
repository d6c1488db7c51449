"""Helpers of the GPU parity tests: run libhfa and the oracle on the same inputs.

Tolerance (stated by the layer's accuracy target): per sequence and per tensor, the
relative L2 error ||gpu - oracle|| / ||oracle|| must be <= 2e-3 for every float output
(q after RoPE, k, v, attention output, layer output).  Integer / byte results are exact:
the appended cache slot equals the bf16 rounding of the kernel's own fp32 value, and
differs from the oracle's rounding only where a bf16 rounding midpoint lies between the
kernel's fp32 value and the oracle's fp64 value and the two agree to 2^-16 of the head
row's RMS (both bytes are then correct roundings of values inside the float
tolerance); every other slot is unchanged, byte for byte.

The number of such flips is bounded, not only their place.  An element flips when a
rounding midpoint falls between the kernel's value t and the oracle's value v, which for a
midpoint placed at random happens with probability |t - v| / ulp(v).  The expected count E
is the sum of those probabilities over the appended values; the flips counted must not
exceed E + 4 sqrt(E) + 4 (far in the tail of the count's distribution), so flips occur only
at the rate that the measured float error explains.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from quantized_attention_layer_gb300 import hfa, workloads as wl

REL_L2 = 2e-3
MIDPOINT_WINDOW = 2.0 ** -16


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def bits_of(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_bits(t.cpu())


def run_gpu_decode(w: wl.Workload, weights, x, pos, kv, debug_taps=True, layer=None):
    dev_w = hfa.weights_to_device(w, weights)
    own = layer is None
    if own:
        layer = hfa.Layer(hfa.desc_for(w, debug_taps=debug_taps), dev_w)
    kc = kv["k_cache"].cuda()
    vc = kv["v_cache"].cuda()
    xd = x.cuda()
    posd = torch.from_numpy(np.asarray(pos, dtype=np.int32)).cuda()
    out = torch.empty((len(pos), w.hidden), dtype=torch.bfloat16, device="cuda")
    layer.hfa_decode_step(xd, posd, pos, kc, vc, out)
    layer.hfa_check_device_status()
    res = {"out_bf16": out, "k_cache": kc, "v_cache": vc}
    if debug_taps:
        res.update(layer.hfa_debug_taps(len(pos)))
    torch.cuda.synchronize()
    res = {k: v.cpu() for k, v in res.items()}
    if own:
        layer.hfa_destroy()
    return res


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values around |v| (8 significant bits; subnormal quantum below)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 7)


def flip_bound(t: np.ndarray, v: np.ndarray):
    """(expected flips, allowed flips) of appended values t (kernel) against v (oracle)."""
    t = np.asarray(t, dtype=np.float64).ravel()
    v = np.asarray(v, dtype=np.float64).ravel()
    e = float(np.sum(np.minimum(1.0, np.abs(t - v) / bf16_ulp(v))))
    return e, e + 4.0 * np.sqrt(e) + 4.0


def check_append(w: wl.Workload, pos, gpu, ref, kv_before, tap_key):
    """Bytes of the appended slot and every untouched slot (see module docstring)."""
    cache_key = tap_key + "_cache"
    g = bits_of(gpu[cache_key]).reshape(len(pos), w.num_kv_heads, w.kv_capacity, w.head_dim)
    r = ref[cache_key].reshape(g.shape)
    before = bits_of(kv_before[cache_key]).reshape(g.shape)
    tap = gpu[tap_key].numpy()                     # fp32 values the kernel rounded
    ref_val = ref[tap_key]                         # fp64 values of the oracle
    n_mid = 0
    for b, P in enumerate(pos):
        slot = P % w.kv_capacity if w.ring else P
        got = g[b, :, slot, :]
        own = np.array([[oracle.f64_to_bf16(float(v)) for v in row] for row in tap[b]],
                       dtype=np.uint16)
        assert np.array_equal(got, own), "appended bytes are not the RNE of the kernel's fp32"
        diff = got != r[b, :, slot, :]
        if diff.any():
            # allowed only where a bf16 rounding midpoint lies between the kernel's fp32
            # value and the oracle's fp64 value, and the two are close (2^-16 of the
            # head row's RMS: far inside the float tolerance)
            mid = 0.5 * (oracle.bf16_to_f64(got[diff]) + oracle.bf16_to_f64(r[b, :, slot, :][diff]))
            v = ref_val[b][diff]
            t = tap[b][diff].astype(np.float64)
            rms = np.sqrt(np.mean(ref_val[b] ** 2, axis=-1, keepdims=True))
            rms = np.broadcast_to(rms, ref_val[b].shape)[diff]
            assert np.all((t - mid) * (v - mid) <= 0), "append differs without a midpoint between"
            assert np.all(np.abs(t - v) <= MIDPOINT_WINDOW * rms), "append differs off-midpoint"
            n_mid += int(diff.sum())
        mask = np.ones(w.kv_capacity, dtype=bool)
        mask[slot] = False
        assert np.array_equal(g[b][:, mask, :], before[b][:, mask, :]), "an untouched slot changed"
    expected, allowed = flip_bound(tap[:len(pos)], ref_val[:len(pos)])
    assert n_mid <= allowed, f"{n_mid} flipped bytes, {expected:.2f} expected (at most {allowed:.1f})"
    return n_mid, round(expected, 3)


def check_decode(w: wl.Workload, pos, gpu, ref, kv_before, tol=REL_L2):
    report = {}
    B = len(pos)
    for key in ("q", "k", "v", "attn", "out"):
        report[key] = max(rel_l2(gpu[key][b].numpy(), ref[key][b]) for b in range(B))
    # bf16 output: exactly the RNE of the kernel's own fp32 output, which meets the
    # float tolerance above (a per-element ulp bound would not survive x + y cancelling)
    own = np.array([oracle.f64_to_bf16(float(v)) for v in gpu["out"].numpy().ravel()],
                   dtype=np.uint16)
    report["out_bf16_exact"] = bool(np.array_equal(bits_of(gpu["out_bf16"]).ravel(), own))
    report["out_bf16_rel_l2"] = rel_l2(oracle.bf16_to_f64(bits_of(gpu["out_bf16"])),
                                       ref["out"].reshape(B, -1))
    report["k_midpoints"] = check_append(w, pos, gpu, ref, kv_before, "k")
    report["v_midpoints"] = check_append(w, pos, gpu, ref, kv_before, "v")
    print(w.name, report)
    for key in ("q", "k", "v", "attn", "out"):
        assert report[key] <= tol, f"{key}: rel L2 {report[key]:.3e} > {tol}"
    assert report["out_bf16_exact"], "bf16 out is not the RNE of the kernel's fp32 out"
    return report


def run_gpu_verify(w: wl.Workload, weights, x, base, kv):
    layer = hfa.Layer(hfa.desc_for(w, debug_taps=True), hfa.weights_to_device(w, weights))
    kc, vc = kv["k_cache"].cuda(), kv["v_cache"].cuda()
    L = x.shape[0]
    out = torch.empty((L, w.hidden), dtype=torch.bfloat16, device="cuda")
    layer.hfa_verify_block(x.cuda(), base, kc, vc, out)
    layer.hfa_check_device_status()
    res = {"out_bf16": out, "k_cache": kc, "v_cache": vc}
    res.update(layer.hfa_debug_taps(L))
    torch.cuda.synchronize()
    res = {k: v.cpu() for k, v in res.items()}
    layer.hfa_destroy()
    return res


def check_verify(w: wl.Workload, base, gpu, ref, kv_before, tol=REL_L2):
    """Float taps per token within tol; appended rows as in check_append; the rest of
    the cache unchanged."""
    L = gpu["q"].shape[0]
    report = {}
    for key in ("q", "k", "v", "attn", "out"):
        report[key] = max(rel_l2(gpu[key][i].numpy(), ref[key][i]) for i in range(L))
    own = np.array([oracle.f64_to_bf16(float(v)) for v in gpu["out"].numpy().ravel()],
                   dtype=np.uint16)
    report["out_bf16_exact"] = bool(np.array_equal(bits_of(gpu["out_bf16"]).ravel(), own))
    n_mid = 0
    expected = 0.0
    for key in ("k", "v"):
        g = bits_of(gpu[key + "_cache"]).reshape(w.num_kv_heads, w.kv_capacity, w.head_dim)
        r = ref[key + "_cache"].reshape(g.shape)
        before = bits_of(kv_before[key + "_cache"]).reshape(g.shape)
        tap = gpu[key].numpy()                       # [L, nkv, hd]
        for i in range(L):
            slot = base + i
            got = g[:, slot, :]
            own_b = np.array([[oracle.f64_to_bf16(float(v)) for v in row] for row in tap[i]],
                             dtype=np.uint16)
            assert np.array_equal(got, own_b), "appended bytes are not the RNE of the kernel's fp32"
            diff = got != r[:, slot, :]
            if diff.any():
                mid = 0.5 * (oracle.bf16_to_f64(got[diff]) + oracle.bf16_to_f64(r[:, slot, :][diff]))
                v = ref[key][i][diff]
                t = tap[i][diff].astype(np.float64)
                rms = np.broadcast_to(np.sqrt(np.mean(ref[key][i] ** 2, axis=-1, keepdims=True)),
                                      ref[key][i].shape)[diff]
                assert np.all((t - mid) * (v - mid) <= 0)
                assert np.all(np.abs(t - v) <= MIDPOINT_WINDOW * rms)
                n_mid += int(diff.sum())
        mask = np.ones(w.kv_capacity, dtype=bool)
        mask[base:base + L] = False
        assert np.array_equal(g[:, mask, :], before[:, mask, :]), "an untouched slot changed"
        e, _ = flip_bound(tap, ref[key][:L])
        expected += e
    allowed = expected + 4.0 * np.sqrt(expected) + 4.0
    assert n_mid <= allowed, f"{n_mid} flipped bytes, {expected:.2f} expected (at most {allowed:.1f})"
    report["midpoints"] = (n_mid, round(expected, 3), 2 * L * w.num_kv_heads * w.head_dim)
    print(w.name, report)
    for key in ("q", "k", "v", "attn", "out"):
        assert report[key] <= tol, f"{key}: rel L2 {report[key]:.3e} > {tol}"
    assert report["out_bf16_exact"]
    return report
