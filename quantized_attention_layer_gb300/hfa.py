"""ctypes binding of libhfa (include/hfa.h): argument marshalling only.

Every step of the decode path runs in the CUDA kernels of libhfa.so; this module
converts torch tensors to raw pointers and checks return codes.  There is no CPU
fallback: if the library is missing, :func:`lib` raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libhfa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "hfa.h")

HFA_OK, HFA_EINVAL, HFA_ERANGE, HFA_ENOMEM, HFA_ECUDA, HFA_EUNSUPPORTED, HFA_EDEVICE = \
    0, -1, -2, -3, -4, -5, -6
STATUS_NAMES = {0: "HFA_OK", -1: "HFA_EINVAL", -2: "HFA_ERANGE", -3: "HFA_ENOMEM",
                -4: "HFA_ECUDA", -5: "HFA_EUNSUPPORTED", -6: "HFA_EDEVICE"}

HFA_F_V_UNIT_NORM = 0x1
HFA_F_WEIGHTS_BF16 = 0x2
HFA_F_RING = 0x4
HFA_F_DEBUG_TAPS = 0x8
HFA_F_K_EQ_V = 0x10
HFA_F_BLOCK_BIDIR = 0x20


class HfaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class hfa_layer_desc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("num_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("layer_type", ctypes.c_int), ("window", ctypes.c_int),
                ("eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("attn_scale", ctypes.c_float), ("softcap", ctypes.c_float),
                ("kv_capacity", ctypes.c_int), ("max_batch", ctypes.c_int),
                ("max_verify_len", ctypes.c_int), ("flags", ctypes.c_uint)]


class hfa_attn_desc(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("layer_type", ctypes.c_int),
                ("window", ctypes.c_int), ("kv_capacity", ctypes.c_int),
                ("attn_scale", ctypes.c_float), ("softcap", ctypes.c_float),
                ("flags", ctypes.c_uint)]


class hfa_ffn_desc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("intermediate", ctypes.c_int), ("eps", ctypes.c_float),
                ("scalar_len", ctypes.c_int), ("max_batch", ctypes.c_int)]


def attn_desc_for(w: wl.Workload) -> hfa_attn_desc:
    return hfa_attn_desc(num_heads=w.num_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                         layer_type=w.layer_type, window=w.window, kv_capacity=w.kv_capacity,
                         attn_scale=w.attn_scale, softcap=w.softcap,
                         flags=HFA_F_RING if w.ring else 0)


_lib = None


def lib():
    """Load libhfa.so (raises when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run quantized_attention_layer_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        P, I, C = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
        L.hfa_layer_create.restype = C
        L.hfa_layer_create.argtypes = [ctypes.POINTER(hfa_layer_desc), P, P, P, P, P, P, P, P,
                                       ctypes.POINTER(P)]
        L.hfa_decode_step.restype = C
        L.hfa_decode_step.argtypes = [P, P, P, P, P, I, P, P, P]
        L.hfa_decode_step_host.restype = C
        L.hfa_decode_step_host.argtypes = [P, P, P, P, I, P, P, P]
        L.hfa_verify_block.restype = C
        L.hfa_verify_block.argtypes = [P, P, P, I, I, P, P, P]
        L.hfa_ctx_append.restype = C
        L.hfa_ctx_append.argtypes = [P, P, P, I, I, P, P]
        L.hfa_destroy.restype = C
        L.hfa_destroy.argtypes = [P]
        L.hfa_set_successor.restype = C
        L.hfa_set_successor.argtypes = [P, P]
        L.hfa_set_step_stamps.restype = C
        L.hfa_set_step_stamps.argtypes = [P, P]
        L.hfa_step_stamp_rows.restype = C
        L.hfa_step_stamp_rows.argtypes = [P]
        L.hfa_weight_tile_bytes.restype = ctypes.c_size_t
        L.hfa_weight_tile_bytes.argtypes = [P, I]
        L.hfa_debug_weight_tiles.restype = C
        L.hfa_debug_weight_tiles.argtypes = [P, I, P, ctypes.c_size_t, P]
        L.hfa_debug_stall_next_step.restype = C
        L.hfa_debug_stall_next_step.argtypes = [P]
        L.hfa_set_rope_freq_factors.restype = C
        L.hfa_set_rope_freq_factors.argtypes = [P, P, P]
        L.hfa_set_post_norm.restype = C
        L.hfa_set_post_norm.argtypes = [P, P, P]
        L.hfa_last_error.restype = ctypes.c_char_p
        L.hfa_last_error.argtypes = [P]
        L.hfa_debug_taps.restype = C
        L.hfa_debug_taps.argtypes = [P, P, P, P, P, P, P]
        L.hfa_check_device_status.restype = C
        L.hfa_check_device_status.argtypes = [P, P]
        L.hfa_set_kernel_timing.restype = C
        L.hfa_set_kernel_timing.argtypes = [P, I]
        L.hfa_kernel_times.restype = C
        L.hfa_kernel_times.argtypes = [P, I, ctypes.POINTER(ctypes.c_char_p),
                                       ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]
        L.hfa_plan_info.restype = C
        L.hfa_plan_info.argtypes = [P, I, ctypes.POINTER(ctypes.c_int)]
        L.hfa_attention_workspace_bytes.restype = ctypes.c_size_t
        L.hfa_attention_workspace_bytes.argtypes = [ctypes.POINTER(hfa_attn_desc), I]
        L.hfa_attention_decode.restype = C
        L.hfa_attention_decode.argtypes = [ctypes.POINTER(hfa_attn_desc), P, P, P, P, I, P, P, P,
                                           ctypes.c_size_t, P]
        L.hfa_attention_decode_noalloc.restype = C
        L.hfa_attention_decode_noalloc.argtypes = [ctypes.POINTER(hfa_attn_desc), P, P, P, P, I,
                                                   P, P, P]
        L.hfa_tq_create.restype = C
        L.hfa_tq_create.argtypes = [I, I, P, ctypes.POINTER(P)]
        L.hfa_tq_destroy.restype = C
        L.hfa_tq_destroy.argtypes = [P]
        L.hfa_tq_code_bytes.restype = I
        L.hfa_tq_code_bytes.argtypes = [P]
        L.hfa_tq_blocks.restype = I
        L.hfa_tq_blocks.argtypes = [P]
        L.hfa_tq_codebook.restype = I
        L.hfa_tq_codebook.argtypes = [P, P, I]
        L.hfa_tq_append.restype = C
        L.hfa_tq_append.argtypes = [P, P, P, P, P, I, I, I, I, P, P]
        L.hfa_attention_tq_workspace_bytes.restype = ctypes.c_size_t
        L.hfa_attention_tq_workspace_bytes.argtypes = [ctypes.POINTER(hfa_attn_desc), I, I]
        L.hfa_attention_decode_tq.restype = C
        L.hfa_attention_decode_tq.argtypes = [ctypes.POINTER(hfa_attn_desc), P, P, P, P, P, I,
                                              P, P, P, P, P, P, ctypes.c_size_t, P]
        L.hfa_ffn_create.restype = C
        L.hfa_ffn_create.argtypes = [ctypes.POINTER(hfa_ffn_desc), P, P, P, P, P, P, P,
                                     ctypes.POINTER(P)]
        L.hfa_ffn_destroy.restype = C
        L.hfa_ffn_destroy.argtypes = [P]
        L.hfa_ffn_step.restype = C
        L.hfa_ffn_step.argtypes = [P, P, P, I, P, P, P]
        L.hfa_ffn_check_status.restype = C
        L.hfa_ffn_check_status.argtypes = [P, P]
        L.hfa_ffn_last_error.restype = ctypes.c_char_p
        L.hfa_ffn_last_error.argtypes = [P]
        L.hfa_ffn_set_stamps.restype = C
        L.hfa_ffn_set_stamps.argtypes = [P, P]
        L.hfa_ffn_stamp_rows.restype = C
        L.hfa_ffn_stamp_rows.argtypes = [P]
        L.hfa_ffn_plan_info.restype = C
        L.hfa_ffn_plan_info.argtypes = [P, I, ctypes.POINTER(ctypes.c_int)]
        _lib = L
    return _lib


def header_functions() -> List[str]:
    """Names of the functions include/hfa.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hfa_[a-z_0-9]+)\s*\(", text)))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def hfa_attention_workspace_bytes(desc: hfa_attn_desc, batch: int) -> int:
    return int(lib().hfa_attention_workspace_bytes(ctypes.byref(desc), int(batch)))


def hfa_attention_decode(desc: hfa_attn_desc, q: torch.Tensor, seq_pos_dev: torch.Tensor,
                         seq_pos_host, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         workspace: torch.Tensor, o: torch.Tensor, stream=None) -> torch.Tensor:
    pos_h = np.ascontiguousarray(seq_pos_host, dtype=np.int32)
    st = lib().hfa_attention_decode(ctypes.byref(desc), _stream_ptr(stream), _ptr(q),
                                    _ptr(seq_pos_dev), ctypes.c_void_p(pos_h.ctypes.data),
                                    int(pos_h.size), _ptr(k_cache), _ptr(v_cache), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _ptr(o))
    if st != HFA_OK:
        raise HfaError(st, lib().hfa_last_error(None).decode())
    return o


def hfa_attention_decode_noalloc(desc: hfa_attn_desc, q: torch.Tensor, seq_pos_dev: torch.Tensor,
                                 seq_pos_host, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                 o: torch.Tensor, stream=None) -> torch.Tensor:
    """hfa_attention_decode with the library's static scratch instead of a workspace."""
    pos_h = np.ascontiguousarray(seq_pos_host, dtype=np.int32)
    st = lib().hfa_attention_decode_noalloc(ctypes.byref(desc), _stream_ptr(stream), _ptr(q),
                                            _ptr(seq_pos_dev), ctypes.c_void_p(pos_h.ctypes.data),
                                            int(pos_h.size), _ptr(k_cache), _ptr(v_cache), _ptr(o))
    if st != HFA_OK:
        raise HfaError(st, lib().hfa_last_error(None).decode())
    return o


class TqFormat:
    """A quantised-KV format (hfa_tq_create ... hfa_tq_destroy)."""

    def __init__(self, head_dim: int, bits: int, signs: np.ndarray):
        self.head_dim, self.bits = int(head_dim), int(bits)
        self._signs = np.ascontiguousarray(signs, dtype=np.int8)
        self._h = ctypes.c_void_p()
        st = lib().hfa_tq_create(self.head_dim, self.bits, ctypes.c_void_p(self._signs.ctypes.data),
                                 ctypes.byref(self._h))
        if st != HFA_OK:
            raise HfaError(st, lib().hfa_last_error(None).decode())

    @property
    def code_bytes(self) -> int:
        return int(lib().hfa_tq_code_bytes(self._h))

    @property
    def blocks(self) -> int:
        return int(lib().hfa_tq_blocks(self._h))

    def codebook(self) -> np.ndarray:
        c = np.empty(1 << self.bits, dtype=np.float32)
        n = lib().hfa_tq_codebook(self._h, ctypes.c_void_p(c.ctypes.data), c.size)
        return c[:n]

    def hfa_tq_append(self, x: torch.Tensor, seq_pos_dev: torch.Tensor, seq_pos_host, nkv: int,
                      capacity: int, ring: bool, codes: torch.Tensor, norms: torch.Tensor,
                      stream=None) -> None:
        pos_h = np.ascontiguousarray(seq_pos_host, dtype=np.int32)
        st = lib().hfa_tq_append(self._h, _stream_ptr(stream), _ptr(x), _ptr(seq_pos_dev),
                                 ctypes.c_void_p(pos_h.ctypes.data), int(pos_h.size), int(nkv),
                                 int(capacity), int(bool(ring)), _ptr(codes), _ptr(norms))
        if st != HFA_OK:
            raise HfaError(st, lib().hfa_last_error(None).decode())

    def hfa_attention_decode_tq(self, desc: hfa_attn_desc, q: torch.Tensor, seq_pos_dev: torch.Tensor,
                                seq_pos_host, k_codes, k_norms, k_raw, v_codes, v_norms,
                                workspace: torch.Tensor, o: torch.Tensor, stream=None) -> torch.Tensor:
        pos_h = np.ascontiguousarray(seq_pos_host, dtype=np.int32)
        st = lib().hfa_attention_decode_tq(
            ctypes.byref(desc), self._h, _stream_ptr(stream), _ptr(q), _ptr(seq_pos_dev),
            ctypes.c_void_p(pos_h.ctypes.data), int(pos_h.size), _ptr(k_codes), _ptr(k_norms),
            _ptr(k_raw), _ptr(v_codes), _ptr(v_norms), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(o))
        if st != HFA_OK:
            raise HfaError(st, lib().hfa_last_error(None).decode())
        return o

    def destroy(self) -> None:
        if self._h:
            lib().hfa_tq_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def hfa_attention_tq_workspace_bytes(desc: hfa_attn_desc, batch: int, max_keys: int) -> int:
    return int(lib().hfa_attention_tq_workspace_bytes(ctypes.byref(desc), int(batch), int(max_keys)))


def desc_for(w: wl.Workload, max_batch: Optional[int] = None, max_verify_len: Optional[int] = None,
             debug_taps: bool = False) -> hfa_layer_desc:
    flags = w.flags | (HFA_F_DEBUG_TAPS if debug_taps else 0)
    return hfa_layer_desc(
        hidden=w.hidden, num_heads=w.num_heads, num_kv_heads=w.num_kv_heads,
        head_dim=w.head_dim, layer_type=w.layer_type, window=w.window, eps=w.eps,
        rope_theta=w.rope_theta, attn_scale=w.attn_scale, softcap=w.softcap,
        kv_capacity=w.kv_capacity,
        max_batch=max_batch if max_batch is not None else max(1, w.batch),
        max_verify_len=max_verify_len if max_verify_len is not None else w.verify_len,
        flags=flags)


def weights_to_device(w: wl.Workload, weights: Dict, device="cuda") -> Dict[str, torch.Tensor]:
    out = {}
    for k, v in weights.items():
        if v is None:  # an absent tensor (no V projection, no variant table)
            out[k] = None
            continue
        if isinstance(v, np.ndarray):
            v = torch.from_numpy(np.ascontiguousarray(v))
        out[k] = v.to(device).contiguous()
    return out


class Layer:
    """One attention layer held by libhfa (hfa_layer_create ... hfa_destroy)."""

    def __init__(self, desc: hfa_layer_desc, dev_weights: Dict[str, torch.Tensor], stream=None):
        self.desc = desc
        self._h = ctypes.c_void_p()
        st = lib().hfa_layer_create(
            ctypes.byref(desc), _ptr(dev_weights["wq"]), _ptr(dev_weights["wk"]),
            _ptr(dev_weights["wv"]), _ptr(dev_weights["wo"]), _ptr(dev_weights["w_in"]),
            _ptr(dev_weights["w_q"]), _ptr(dev_weights["w_k"]), _stream_ptr(stream),
            ctypes.byref(self._h))
        if st != HFA_OK:
            raise HfaError(st, lib().hfa_last_error(None).decode())
        # the Gemma variants the weights carry: RoPE frequency factors, post-attention norm
        if dev_weights.get("rope_ff") is not None:
            self.hfa_set_rope_freq_factors(dev_weights["rope_ff"].cpu().numpy(), stream)
        if dev_weights.get("w_post") is not None:
            self.hfa_set_post_norm(dev_weights["w_post"], stream)

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    def _check(self, st: int):
        if st != HFA_OK:
            raise HfaError(st, lib().hfa_last_error(self._h).decode())

    def hfa_decode_step(self, x: torch.Tensor, seq_pos_dev: torch.Tensor, seq_pos_host: np.ndarray,
                        k_cache: torch.Tensor, v_cache: torch.Tensor, out: torch.Tensor,
                        stream=None) -> torch.Tensor:
        pos_h = np.ascontiguousarray(seq_pos_host, dtype=np.int32)
        self._check(lib().hfa_decode_step(self._h, _stream_ptr(stream), _ptr(x), _ptr(seq_pos_dev),
                                          ctypes.c_void_p(pos_h.ctypes.data), int(pos_h.size),
                                          _ptr(k_cache), _ptr(v_cache), _ptr(out)))
        return out

    def hfa_decode_step_host(self, x_host: torch.Tensor, seq_pos_host: np.ndarray,
                             k_cache: torch.Tensor, v_cache: torch.Tensor, out_host: torch.Tensor,
                             stream=None) -> torch.Tensor:
        pos_h = np.ascontiguousarray(seq_pos_host, dtype=np.int32)
        self._check(lib().hfa_decode_step_host(self._h, _stream_ptr(stream), _ptr(x_host),
                                               ctypes.c_void_p(pos_h.ctypes.data), int(pos_h.size),
                                               _ptr(k_cache), _ptr(v_cache), _ptr(out_host)))
        return out_host

    def hfa_verify_block(self, x: torch.Tensor, base_pos: int, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, out: torch.Tensor, stream=None) -> torch.Tensor:
        self._check(lib().hfa_verify_block(self._h, _stream_ptr(stream), _ptr(x), int(x.shape[0]),
                                           int(base_pos), _ptr(k_cache), _ptr(v_cache), _ptr(out)))
        return out

    def hfa_ctx_append(self, x_ctx: torch.Tensor, base_pos: int, k_cache: torch.Tensor,
                       v_cache: torch.Tensor, stream=None) -> None:
        self._check(lib().hfa_ctx_append(self._h, _stream_ptr(stream), _ptr(x_ctx),
                                         int(x_ctx.shape[0]), int(base_pos), _ptr(k_cache),
                                         _ptr(v_cache)))

    def hfa_debug_taps(self, rows: int, stream=None) -> Dict[str, torch.Tensor]:
        d = self.desc
        dev = torch.device("cuda")
        t = {"q": torch.empty((rows, d.num_heads, d.head_dim), device=dev),
             "k": torch.empty((rows, d.num_kv_heads, d.head_dim), device=dev),
             "v": torch.empty((rows, d.num_kv_heads, d.head_dim), device=dev),
             "attn": torch.empty((rows, d.num_heads, d.head_dim), device=dev),
             "out": torch.empty((rows, d.hidden), device=dev)}
        self._check(lib().hfa_debug_taps(self._h, _stream_ptr(stream), _ptr(t["q"]), _ptr(t["k"]),
                                          _ptr(t["v"]), _ptr(t["attn"]), _ptr(t["out"])))
        return t

    def hfa_check_device_status(self, stream=None) -> None:
        self._check(lib().hfa_check_device_status(self._h, _stream_ptr(stream)))

    def hfa_set_rope_freq_factors(self, factors: Optional[np.ndarray], stream=None) -> None:
        ff = None if factors is None else np.ascontiguousarray(factors, dtype=np.float32)
        self._check(lib().hfa_set_rope_freq_factors(
            self._h, None if ff is None else ctypes.c_void_p(ff.ctypes.data), _stream_ptr(stream)))

    def hfa_set_post_norm(self, w_post: Optional[torch.Tensor], stream=None) -> None:
        self._check(lib().hfa_set_post_norm(self._h, None if w_post is None else _ptr(w_post),
                                            _stream_ptr(stream)))

    def hfa_set_step_stamps(self, stamps: Optional[torch.Tensor]) -> None:
        """Timer stamps of later decode steps into `stamps` (int64 [rows, 16], device), or off."""
        self._check(lib().hfa_set_step_stamps(self._h, _ptr(stamps)))

    def hfa_step_stamp_rows(self) -> int:
        return int(lib().hfa_step_stamp_rows(self._h))

    def hfa_debug_weight_tiles(self, which: int, stream=None) -> torch.Tensor:
        """The library's copy of weight buffer `which` (see hfa.h) as a uint8 device tensor."""
        n = int(lib().hfa_weight_tile_bytes(self._h, int(which)))
        if n == 0:
            raise HfaError(HFA_EINVAL, f"the layer has no weight buffer {which}")
        dst = torch.empty(n, dtype=torch.uint8, device="cuda")
        self._check(lib().hfa_debug_weight_tiles(self._h, int(which), _ptr(dst), n,
                                                 _stream_ptr(stream)))
        return dst

    def hfa_debug_stall_next_step(self) -> None:
        self._check(lib().hfa_debug_stall_next_step(self._h))

    def hfa_set_successor(self, next_layer: Optional["Layer"]) -> None:
        self._check(lib().hfa_set_successor(self._h, next_layer._h if next_layer else None))

    def hfa_set_kernel_timing(self, enable: bool) -> None:
        lib().hfa_set_kernel_timing(self._h, int(bool(enable)))

    def hfa_kernel_times(self) -> Dict[str, tuple]:
        n = 16
        names = (ctypes.c_char_p * n)()
        ms = (ctypes.c_float * n)()
        cnt = (ctypes.c_int * n)()
        k = lib().hfa_kernel_times(self._h, n, names, ms, cnt)
        return {names[i].decode(): (float(ms[i]), int(cnt[i])) for i in range(max(k, 0))}

    def hfa_plan_info(self) -> Dict[str, int]:
        v = (ctypes.c_int * 5)()
        lib().hfa_plan_info(self._h, 5, v)
        return {"attn_tiles": v[0], "keys_per_tile": v[1], "step_grid": v[2],
                "num_sms": v[4]}

    def hfa_destroy(self) -> None:
        if self._h:
            lib().hfa_destroy(self._h)
            self._h = ctypes.c_void_p()

    close = hfa_destroy

    def __del__(self):
        try:
            self.hfa_destroy()
        except Exception:
            pass


def ffn_desc_for(f: wl.FfnWorkload, max_batch: Optional[int] = None) -> hfa_ffn_desc:
    return hfa_ffn_desc(hidden=f.hidden, intermediate=f.intermediate, eps=f.eps,
                        scalar_len=f.hidden if f.scalar_per_channel else 1,
                        max_batch=int(max_batch or f.batch))


def ffn_weights_to_device(weights: Dict, device="cuda") -> Dict[str, torch.Tensor]:
    out = {}
    for k in ("w_gate", "w_up", "w_down"):
        out[k] = torch.from_numpy(np.ascontiguousarray(weights[k])).to(device)
    for k in ("w_pre", "w_post", "scalar"):
        out[k] = torch.as_tensor(weights[k], dtype=torch.float32).contiguous().to(device)
    return out


class Ffn:
    """The dense FFN half (hfa_ffn_create ... hfa_ffn_destroy)."""

    def __init__(self, desc: hfa_ffn_desc, dev_weights: Dict[str, torch.Tensor], stream=None):
        self.desc = desc
        self._h = ctypes.c_void_p()
        w = dev_weights
        st = lib().hfa_ffn_create(ctypes.byref(desc), _ptr(w["w_gate"]), _ptr(w["w_up"]),
                                  _ptr(w["w_down"]), _ptr(w["w_pre"]), _ptr(w["w_post"]),
                                  _ptr(w["scalar"]), _stream_ptr(stream), ctypes.byref(self._h))
        if st != HFA_OK:
            raise HfaError(st, lib().hfa_ffn_last_error(None).decode())

    def _check(self, st: int):
        if st != HFA_OK:
            raise HfaError(st, lib().hfa_ffn_last_error(self._h).decode())

    def hfa_ffn_step(self, h: torch.Tensor, out: torch.Tensor, out_f32: Optional[torch.Tensor] = None,
                     a: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        self._check(lib().hfa_ffn_step(self._h, _stream_ptr(stream), _ptr(h), int(h.shape[0]),
                                       _ptr(out), _ptr(out_f32), _ptr(a)))
        return out

    def hfa_ffn_check_status(self, stream=None) -> None:
        self._check(lib().hfa_ffn_check_status(self._h, _stream_ptr(stream)))

    def hfa_ffn_set_stamps(self, stamps: Optional[torch.Tensor]) -> None:
        self._check(lib().hfa_ffn_set_stamps(self._h, _ptr(stamps)))

    def hfa_ffn_stamp_rows(self) -> int:
        return int(lib().hfa_ffn_stamp_rows(self._h))

    def hfa_ffn_plan_info(self) -> Dict[str, int]:
        v = (ctypes.c_int * 16)()
        n = lib().hfa_ffn_plan_info(self._h, 16, v)
        names = ["grid", "nt_max", "s1", "nbs1", "rgs1", "stages1", "s2", "nbs2", "rgs2", "stages2"]
        return {names[i]: int(v[i]) for i in range(min(n, len(names)))}

    def hfa_ffn_destroy(self) -> None:
        if self._h:
            lib().hfa_ffn_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.hfa_ffn_destroy()
        except Exception:
            pass
