"""CPU oracle for the attention-layer decode step (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  It wraps ``liborc.so`` (built from ``hfa_oracle.cpp`` by
:func:`build`) with ctypes and converts numpy / torch CPU buffers.  It never touches
the CUDA library and the CUDA library never touches it.

Parity status per function (pins live in ``tests/test_oracle_*.py``):

* f16 / bf16 conversions: pinned (exhaustive library comparison, hand-made midpoints)
* Q8_0 dequantisation and mat-vec: pinned (hand-made blocks, page quantiser round
  trip, blockwise == dense, one-hot columns)
* RMSNorm: pinned (all-ones closed form from the drafter smoke test, unit RMS)
* RoPE: pinned (hand-computed angles, norm, composition, relative position)
* slots / visibility / attention: pinned (brute-force explicit mask, permutation,
  one key, softcap bound, ring == linear window)
* quantised KV cache (Lloyd-Max codebook, FWHT rotation, encode / decode, attention
  over codes): pinned (textbook Lloyd-Max values and closed forms, the Hadamard matrix
  from its popcount definition, brute-force nearest centroid, attention over codes ==
  attention over the dequantised cache)
* decode step / verify block: pinned by a closed-form layer (permutation weights at
  position 0), by the q and k heads in closed form at later positions (permutation Wq
  and Wk, distinct norm weights, power-of-two RoPE angles), and by consistency (verify of L tokens == L decode steps; batch ==
  independent sequences).  The pages print no whole-layer values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hfa_oracle.cpp")
_SRCS = [_SRC, os.path.join(_HERE, "tq_oracle.cpp")]
_HDRS = [os.path.join(_HERE, "hfa_oracle.h"), os.path.join(_HERE, "tq_oracle.h")]
_LIB_PATH = os.path.join(_HERE, "liborc.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (OpenMP when available)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(f) for f in _SRCS + _HDRS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp"] + _SRCS + ["-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OrcDesc(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int), ("num_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("layer_type", ctypes.c_int), ("window", ctypes.c_int),
        ("eps", ctypes.c_double), ("rope_theta", ctypes.c_double),
        ("attn_scale", ctypes.c_double), ("softcap", ctypes.c_double),
        ("kv_capacity", ctypes.c_int), ("ring", ctypes.c_int),
        ("v_unit_norm", ctypes.c_int), ("weights_bf16", ctypes.c_int),
        ("k_eq_v", ctypes.c_int), ("rope_freq_factors", ctypes.c_void_p),
        ("w_post", ctypes.c_void_p), ("block_bidir", ctypes.c_int),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            L.orc_bf16_to_f64.restype = ctypes.c_double
            L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.orc_f64_to_bf16.restype = ctypes.c_uint16
            L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
            L.orc_f16_to_f64.restype = ctypes.c_double
            L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
            L.orc_q8_0_dequant_row.argtypes = [P, ctypes.c_int, P]
            L.orc_q8_0_matvec.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P]
            L.orc_q8_0_matvec_blockwise.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P]
            L.orc_bf16_matvec.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P]
            L.orc_rmsnorm.argtypes = [P, P, ctypes.c_int, ctypes.c_double, P]
            L.orc_rope_neox.argtypes = [P, ctypes.c_int, ctypes.c_double, ctypes.c_double]
            L.orc_rope_neox_ff.argtypes = [P, ctypes.c_int, ctypes.c_double, ctypes.c_double, P]
            L.orc_kv_slot.restype = ctypes.c_long
            L.orc_kv_slot.argtypes = [ctypes.c_long, ctypes.c_long, ctypes.c_int]
            L.orc_key_visible.restype = ctypes.c_int
            L.orc_key_visible.argtypes = [ctypes.c_long, ctypes.c_long, ctypes.c_int, ctypes.c_long]
            L.orc_slot_position.restype = ctypes.c_long
            L.orc_slot_position.argtypes = [ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_int]
            L.orc_attend.argtypes = [P, P, P, ctypes.c_int, P, ctypes.c_long, ctypes.c_double,
                                     ctypes.c_double, P, P]
            step_args = [ctypes.POINTER(OrcDesc), P, P, P, P, P, P, P, P]
            L.orc_decode_step.restype = ctypes.c_int
            L.orc_decode_step.argtypes = step_args + [P, ctypes.c_int, P, P, P, P, P, P, P, P]
            L.orc_verify_block.restype = ctypes.c_int
            L.orc_verify_block.argtypes = step_args + [ctypes.c_int, ctypes.c_int, P, P, P, P, P,
                                                       P, P, P]
            L.orc_lloyd_max_normal.restype = ctypes.c_int
            L.orc_lloyd_max_normal.argtypes = [ctypes.c_int, P, P]
            L.orc_lloyd_max_mse.restype = ctypes.c_double
            L.orc_lloyd_max_mse.argtypes = [ctypes.c_int, P, P]
            L.orc_fwht.argtypes = [P, ctypes.c_int]
            L.orc_tq_rotate.argtypes = [P, ctypes.c_int, P]
            L.orc_tq_unrotate.argtypes = [P, ctypes.c_int, P]
            L.orc_tq_code_bytes.restype = ctypes.c_int
            L.orc_tq_code_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
            L.orc_tq_blocks.restype = ctypes.c_int
            L.orc_tq_blocks.argtypes = [ctypes.c_int]
            L.orc_tq_encode_row.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, P, P]
            L.orc_tq_decode_row.argtypes = [P, P, ctypes.c_int, ctypes.c_int, P, P]
            L.orc_attend_tq.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P, P,
                                        ctypes.c_long, ctypes.c_double, ctypes.c_double, P]
            L.orc_ctx_append.restype = ctypes.c_int
            L.orc_ctx_append.argtypes = [ctypes.POINTER(OrcDesc), P, P, P, P, ctypes.c_int,
                                         ctypes.c_int, P, P, P, P]
            L.orc_gelu_tanh.restype = ctypes.c_double
            L.orc_gelu_tanh.argtypes = [ctypes.c_double]
            L.orc_ffn_step.restype = ctypes.c_int
            L.orc_ffn_step.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, P, P, P, P, P,
                                       P, ctypes.c_int, P, ctypes.c_int, P, P, P]
            L.orc_num_threads.restype = ctypes.c_int
            L.orc_set_num_threads.argtypes = [ctypes.c_int]
            _lib = L
    return _lib


# ------------------------------------------------------------------ array helpers

def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def as_np(t, dtype) -> np.ndarray:
    """numpy view/copy of a CPU tensor or array with the given dtype, C-contiguous."""
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.view(torch.int16)
        t = t.numpy()
    a = np.ascontiguousarray(t)
    if a.dtype != dtype:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def bf16_bits(t) -> np.ndarray:
    return as_np(t, np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 -> float64 (bit shift into binary32)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def desc_from(w, weights: Optional[Dict] = None, keep: Optional[list] = None) -> OrcDesc:
    """The oracle's layer description; the variant tables of `weights` (frequency factors,
    post-attention norm weight) are referenced by pointer, their arrays appended to `keep`
    so that they outlive the call."""
    ff = wp = None
    if weights is not None:  # only the variants the workload turns on
        if getattr(w, "rope_freq_factors", False) and weights.get("rope_ff") is not None:
            ff = as_np(weights["rope_ff"], np.float32)
        if getattr(w, "post_norm", False) and weights.get("w_post") is not None:
            wp = as_np(weights["w_post"], np.float32)
    if keep is not None:
        keep.extend([ff, wp])
    return OrcDesc(hidden=w.hidden, num_heads=w.num_heads, num_kv_heads=w.num_kv_heads,
                   head_dim=w.head_dim, layer_type=w.layer_type, window=w.window, eps=w.eps,
                   rope_theta=w.rope_theta, attn_scale=w.attn_scale, softcap=w.softcap,
                   kv_capacity=w.kv_capacity, ring=int(w.ring), v_unit_norm=int(w.v_unit_norm),
                   weights_bf16=int(w.weights_bf16), k_eq_v=int(getattr(w, "k_eq_v", False)),
                   rope_freq_factors=None if ff is None else ff.ctypes.data,
                   w_post=None if wp is None else wp.ctypes.data,
                   block_bidir=int(getattr(w, "block_bidir", False)))


def _weight_np(w, t):
    if t is None:
        return None
    return as_np(t, np.uint16) if w.weights_bf16 else as_np(t, np.uint8)


# ------------------------------------------------------------------ scalar wrappers

def f64_to_bf16(v: float) -> int:
    return int(lib().orc_f64_to_bf16(float(v)))


def bf16_scalar_to_f64(b: int) -> float:
    return float(lib().orc_bf16_to_f64(int(b)))


def f16_to_f64(h: int) -> float:
    return float(lib().orc_f16_to_f64(int(h)))


def q8_0_dequant(blocks: np.ndarray, cols: int) -> np.ndarray:
    blocks = as_np(blocks, np.uint8).reshape(-1, cols // 32 * 34)
    out = np.empty((blocks.shape[0], cols), dtype=np.float64)
    for r in range(blocks.shape[0]):
        lib().orc_q8_0_dequant_row(_ptr(blocks[r]), cols, _ptr(out[r]))
    return out


def q8_0_matvec(blocks, rows, cols, x, blockwise=False) -> np.ndarray:
    blocks = as_np(blocks, np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(rows, dtype=np.float64)
    fn = lib().orc_q8_0_matvec_blockwise if blockwise else lib().orc_q8_0_matvec
    fn(_ptr(blocks), rows, cols, _ptr(x), _ptr(y))
    return y


def bf16_matvec(w, x) -> np.ndarray:
    wb = as_np(w, np.uint16)
    rows, cols = wb.shape
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(rows, dtype=np.float64)
    lib().orc_bf16_matvec(_ptr(wb), rows, cols, _ptr(x), _ptr(y))
    return y


def rmsnorm(x, w=None, eps=1e-6) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    wa = None if w is None else as_np(w, np.float32)
    y = np.empty_like(x)
    lib().orc_rmsnorm(_ptr(x), _ptr(wa), x.size, float(eps), _ptr(y))
    return y


def rope_neox(u, pos, theta, freq_factors=None) -> np.ndarray:
    u = np.array(u, dtype=np.float64, copy=True)
    if freq_factors is None:
        lib().orc_rope_neox(_ptr(u), u.size, float(pos), float(theta))
    else:
        ff = np.ascontiguousarray(np.asarray(freq_factors, dtype=np.float32))
        lib().orc_rope_neox_ff(_ptr(u), u.size, float(pos), float(theta), _ptr(ff))
    return u


def kv_slot(pos, cap, ring) -> int:
    return int(lib().orc_kv_slot(pos, cap, int(ring)))


def key_visible(p, P, sliding, window) -> bool:
    return bool(lib().orc_key_visible(p, P, int(sliding), window))


def slot_position(slot, P, cap, ring) -> int:
    return int(lib().orc_slot_position(slot, P, cap, int(ring)))


def attend(q, k_rows_bf16, v_rows_bf16, rows, scale=1.0, softcap=0.0):
    """Attention of one query over explicit cache rows; returns (o, weights)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    kb = as_np(k_rows_bf16, np.uint16)
    vb = as_np(v_rows_bf16, np.uint16)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    hd = q.size
    o = np.empty(hd, dtype=np.float64)
    wts = np.empty(max(rows.size, 1), dtype=np.float64)
    lib().orc_attend(_ptr(q), _ptr(kb), _ptr(vb), hd, _ptr(rows), rows.size, float(scale),
                     float(softcap), _ptr(wts), _ptr(o))
    return o, wts[:rows.size]


# ------------------------------------------------------------------ layer entry points

def decode_step(w, weights: Dict, x, seq_pos, k_cache, v_cache) -> Dict[str, np.ndarray]:
    """Run the oracle decode step on copies of the caches; returns every tap."""
    keep: list = []
    d = desc_from(w, weights, keep)
    B = int(np.asarray(seq_pos).size)
    H, nh, nkv, hd = w.hidden, w.num_heads, w.num_kv_heads, w.head_dim
    xb = bf16_bits(x).reshape(B, H)
    pos = np.ascontiguousarray(np.asarray(seq_pos, dtype=np.int32))
    kc = bf16_bits(k_cache).copy()
    vc = bf16_bits(v_cache).copy()
    out = {"q": np.empty((B, nh, hd)), "k": np.empty((B, nkv, hd)), "v": np.empty((B, nkv, hd)),
           "attn": np.empty((B, nh, hd)), "out": np.empty((B, H)),
           "out_bf16": np.empty((B, H), dtype=np.uint16)}
    wq, wk, wv, wo = (_weight_np(w, weights[n]) for n in ("wq", "wk", "wv", "wo"))
    norms = [as_np(weights[n], np.float32) for n in ("w_in", "w_q", "w_k")]
    rc = lib().orc_decode_step(ctypes.byref(d), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo),
                               *[_ptr(a) for a in norms], _ptr(xb), _ptr(pos), B, _ptr(kc),
                               _ptr(vc), _ptr(out["q"]), _ptr(out["k"]), _ptr(out["v"]),
                               _ptr(out["attn"]), _ptr(out["out"]), _ptr(out["out_bf16"]))
    if rc != 0:
        raise ValueError("oracle decode_step rejected its arguments")
    out["k_cache"], out["v_cache"] = kc, vc
    return out


def verify_block(w, weights: Dict, x, base_pos, k_cache, v_cache) -> Dict[str, np.ndarray]:
    keep: list = []
    d = desc_from(w, weights, keep)
    H, nh, nkv, hd = w.hidden, w.num_heads, w.num_kv_heads, w.head_dim
    xb = bf16_bits(x).reshape(-1, H)
    L = xb.shape[0]
    kc = bf16_bits(k_cache).copy()
    vc = bf16_bits(v_cache).copy()
    out = {"q": np.empty((L, nh, hd)), "k": np.empty((L, nkv, hd)), "v": np.empty((L, nkv, hd)),
           "attn": np.empty((L, nh, hd)), "out": np.empty((L, H)),
           "out_bf16": np.empty((L, H), dtype=np.uint16)}
    wq, wk, wv, wo = (_weight_np(w, weights[n]) for n in ("wq", "wk", "wv", "wo"))
    norms = [as_np(weights[n], np.float32) for n in ("w_in", "w_q", "w_k")]
    rc = lib().orc_verify_block(ctypes.byref(d), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo),
                                *[_ptr(a) for a in norms], _ptr(xb), L, int(base_pos), _ptr(kc),
                                _ptr(vc), _ptr(out["q"]), _ptr(out["k"]), _ptr(out["v"]),
                                _ptr(out["attn"]), _ptr(out["out"]), _ptr(out["out_bf16"]))
    if rc != 0:
        raise ValueError("oracle verify_block rejected its arguments")
    out["k_cache"], out["v_cache"] = kc, vc
    return out


def ctx_append(w, weights: Dict, x_ctx, base_pos, k_cache, v_cache) -> Dict[str, np.ndarray]:
    """The drafter's context rows appended to copies of the caches; returns k, v and caches."""
    keep: list = []
    d = desc_from(w, weights, keep)
    H, nkv, hd = w.hidden, w.num_kv_heads, w.head_dim
    xb = bf16_bits(x_ctx).reshape(-1, H)
    S = xb.shape[0]
    kc = bf16_bits(k_cache).copy()
    vc = bf16_bits(v_cache).copy()
    out = {"k": np.empty((S, nkv, hd)), "v": np.empty((S, nkv, hd))}
    wk, wv = _weight_np(w, weights["wk"]), _weight_np(w, weights["wv"])
    rc = lib().orc_ctx_append(ctypes.byref(d), _ptr(wk), _ptr(wv),
                              _ptr(as_np(weights["w_k"], np.float32)), _ptr(xb), S, int(base_pos),
                              _ptr(kc), _ptr(vc), _ptr(out["k"]), _ptr(out["v"]))
    if rc != 0:
        raise ValueError("oracle ctx_append rejected its arguments")
    out["k_cache"], out["v_cache"] = kc, vc
    return out


def gelu_tanh(x: float) -> float:
    return float(lib().orc_gelu_tanh(float(x)))


def ffn_step(f, weights: Dict, h) -> Dict[str, np.ndarray]:
    """The dense FFN half for the rows of h (bf16 [B, H]); returns a, out and out_bf16."""
    H, I = f.hidden, f.intermediate
    hb = bf16_bits(h).reshape(-1, H)
    B = hb.shape[0]
    out = {"a": np.empty((B, I)), "out": np.empty((B, H)), "out_bf16": np.empty((B, H), dtype=np.uint16)}
    wg, wu, wd = (as_np(weights[n], np.uint8) for n in ("w_gate", "w_up", "w_down"))
    norms = [as_np(weights[n], np.float32) for n in ("w_pre", "w_post", "scalar")]
    rc = lib().orc_ffn_step(H, I, float(f.eps), _ptr(wg), _ptr(wu), _ptr(wd), _ptr(norms[0]),
                            _ptr(norms[1]), _ptr(norms[2]), norms[2].size, _ptr(hb), B,
                            _ptr(out["a"]), _ptr(out["out"]), _ptr(out["out_bf16"]))
    if rc != 0:
        raise ValueError("oracle ffn_step rejected its arguments")
    return out


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# ------------------------------------------------------------------ quantised KV cache

def lloyd_max_normal(bits: int):
    """(centroids [2^bits], boundaries [2^bits + 1], rounds) of the N(0,1) Lloyd-Max quantiser."""
    levels = 1 << bits
    c = np.empty(levels, dtype=np.float64)
    b = np.empty(levels + 1, dtype=np.float64)
    rounds = lib().orc_lloyd_max_normal(levels, _ptr(c), _ptr(b))
    return c, b, int(rounds)


def lloyd_max_mse(centroids, boundaries) -> float:
    c = np.ascontiguousarray(centroids, dtype=np.float64)
    b = np.ascontiguousarray(boundaries, dtype=np.float64)
    return float(lib().orc_lloyd_max_mse(c.size, _ptr(c), _ptr(b)))


def fwht(x) -> np.ndarray:
    x = np.array(x, dtype=np.float64, copy=True)
    lib().orc_fwht(_ptr(x), x.size)
    return x


def tq_rotate(x, signs) -> np.ndarray:
    x = np.array(x, dtype=np.float64, copy=True)
    s = np.ascontiguousarray(signs, dtype=np.int8)
    lib().orc_tq_rotate(_ptr(x), x.size, _ptr(s))
    return x


def tq_unrotate(x, signs) -> np.ndarray:
    x = np.array(x, dtype=np.float64, copy=True)
    s = np.ascontiguousarray(signs, dtype=np.int8)
    lib().orc_tq_unrotate(_ptr(x), x.size, _ptr(s))
    return x


def tq_code_bytes(hd: int, bits: int) -> int:
    return int(lib().orc_tq_code_bytes(hd, bits))


def tq_blocks(hd: int) -> int:
    return int(lib().orc_tq_blocks(hd))


def tq_encode_rows(x, signs, bits, boundaries):
    """Encode rows x [..., hd] -> (codes uint8 [..., code_bytes], norms f32 [..., blocks])."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    hd = x.shape[-1]
    rows = x.reshape(-1, hd)
    s = np.ascontiguousarray(signs, dtype=np.int8)
    b = np.ascontiguousarray(boundaries, dtype=np.float64)
    cb, nb = tq_code_bytes(hd, bits), tq_blocks(hd)
    codes = np.empty((rows.shape[0], cb), dtype=np.uint8)
    norms = np.empty((rows.shape[0], nb), dtype=np.float32)
    for r in range(rows.shape[0]):
        lib().orc_tq_encode_row(_ptr(rows[r]), hd, _ptr(s), int(bits), _ptr(b), _ptr(codes[r]),
                                _ptr(norms[r]))
    return codes.reshape(x.shape[:-1] + (cb,)), norms.reshape(x.shape[:-1] + (nb,))


def tq_decode_rows(codes, norms, hd, bits, centroids) -> np.ndarray:
    """Decode rows into the rotated domain: [..., hd] float64."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    norms = np.ascontiguousarray(norms, dtype=np.float32)
    c = np.ascontiguousarray(centroids, dtype=np.float64)
    cr = codes.reshape(-1, codes.shape[-1])
    nr = norms.reshape(-1, norms.shape[-1])
    out = np.empty((cr.shape[0], hd), dtype=np.float64)
    for r in range(cr.shape[0]):
        lib().orc_tq_decode_row(_ptr(cr[r]), _ptr(nr[r]), hd, int(bits), _ptr(c), _ptr(out[r]))
    return out.reshape(codes.shape[:-1] + (hd,))


def attend_tq(q, signs, bits, centroids, k_codes, k_norms, v_codes, v_norms, rows,
              scale=1.0, softcap=0.0, k_bf16=None) -> np.ndarray:
    """Attention of one query over rows of a TQ cache (k_codes None: hybrid, raw bf16 keys)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    hd = q.size
    s = np.ascontiguousarray(signs, dtype=np.int8)
    c = np.ascontiguousarray(centroids, dtype=np.float64)
    kc = None if k_codes is None else np.ascontiguousarray(k_codes, dtype=np.uint8)
    kn = None if k_norms is None else np.ascontiguousarray(k_norms, dtype=np.float32)
    kb = None if k_bf16 is None else as_np(k_bf16, np.uint16)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    vn = np.ascontiguousarray(v_norms, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty(hd, dtype=np.float64)
    lib().orc_attend_tq(_ptr(q), hd, int(bits), _ptr(s), _ptr(c), _ptr(kc), _ptr(kn), _ptr(kb),
                        _ptr(vc), _ptr(vn), _ptr(rows), rows.size, float(scale), float(softcap),
                        _ptr(o))
    return o
