"""Seeded synthetic workloads for the single-layer decode step and the verify block.

This module only *draws* inputs: random Q8_0 blocks, bf16 activations and KV caches,
norm weights and positions.  It holds none of the layer's arithmetic (no norm, no
projection, no rounding of computed values), so both the CPU oracle and the CUDA
library can consume the very same buffers.

The five workloads follow the shapes and value distributions of the layer
descriptions they stand in for:

* Q8_0 weights: 32-value blocks of 34 bytes -- a little-endian fp16 scale ``d``
  followed by 32 signed bytes -- as written by the Q8_0 re-quantiser on the
  ``gemma4/model.rs`` page (lm_head Q8_0 section).  Here the bytes are drawn
  directly: ``q ~ U[-127, 127]`` and ``d ~ U[0.001, 0.02]`` (rounded to fp16).
* bf16 dense weights (verify block): ``~ N(0, 0.02)``.
* activations ``x`` and the prefilled KV cache: bf16 ``~ N(0, 1)``.
* RMSNorm weights (input, q_norm, k_norm): f32 ``~ U[0.5, 1.5]``.
* KV cache layout: head-major ``[B, n_kv_heads, capacity, head_dim]``, the layout of
  the dense KV buffers on the ``gemma4/model.rs`` page (``dense_kvs`` field).

Random numbers come from ``torch.Generator`` on the CPU, seeded per workload.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np
import torch

SLIDING = 0
FULL = 1

F_V_UNIT_NORM = 1 << 0
F_WEIGHTS_BF16 = 1 << 1
F_RING = 1 << 2
F_K_EQ_V = 1 << 4
F_BLOCK_BIDIR = 1 << 5


@dataclasses.dataclass(frozen=True)
class Workload:
    """One layer configuration plus the step it is exercised on."""

    name: str
    hidden: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    layer_type: int            # SLIDING or FULL
    window: int                # used iff SLIDING
    kv_capacity: int
    ring: bool                 # sliding ring buffer: slot = pos % capacity
    batch: int
    rope_theta: float
    seed: int
    eps: float = 1e-6
    attn_scale: float = 1.0
    softcap: float = 0.0
    weights_bf16: bool = False  # dense bf16 weights instead of Q8_0
    verify_len: int = 0         # > 0: multi-token verify block of this length
    base_pos: int = 0           # verify: first position of the block
    seq_pos: Optional[int] = None        # decode: one position for every sequence
    seq_pos_range: Optional[tuple] = None  # decode: per-sequence U[lo, hi]
    v_unit_norm: bool = False
    # Gemma decode variants: no V projection (V = unit-normed raw K), per-pair RoPE
    # frequency factors, RMSNorm of the o_proj output before the residual add
    k_eq_v: bool = False
    rope_freq_factors: bool = False
    post_norm: bool = False
    # the drafter's block attention: every row of a verify block sees the whole block on a
    # full layer (sliding layers stay causal)
    block_bidir: bool = False

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def q_rows(self) -> int:
        return self.num_heads * self.head_dim

    @property
    def kv_rows(self) -> int:
        return self.num_kv_heads * self.head_dim

    @property
    def flags(self) -> int:
        f = 0
        if self.v_unit_norm:
            f |= F_V_UNIT_NORM
        if self.weights_bf16:
            f |= F_WEIGHTS_BF16
        if self.ring:
            f |= F_RING
        if self.k_eq_v:
            f |= F_K_EQ_V
        if self.block_bidir:
            f |= F_BLOCK_BIDIR
        return f

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five layer workloads.  Readings of points the layer descriptions leave open
# (theta of the sliding batch, eps, context N -> seq_pos N-1 with capacity N, the
# ring prefill) are listed with their reasons in the design notes.
TINY_SLIDING = Workload(
    name="tiny_sliding", hidden=256, num_heads=4, num_kv_heads=2, head_dim=64,
    layer_type=SLIDING, window=64, kv_capacity=128, ring=False, batch=1,
    rope_theta=1e4, seed=0, seq_pos=127)
FULL_32K = Workload(
    name="full_b1_32k", hidden=4096, num_heads=32, num_kv_heads=8, head_dim=128,
    layer_type=FULL, window=0, kv_capacity=32768, ring=False, batch=1,
    rope_theta=1e6, seed=1, seq_pos=32767)
SLIDING_B16 = Workload(
    name="sliding_b16_ring1024", hidden=4096, num_heads=16, num_kv_heads=8,
    head_dim=256, layer_type=SLIDING, window=1024, kv_capacity=1024, ring=True,
    batch=16, rope_theta=1e4, seed=2, seq_pos_range=(1024, 8192))
VERIFY_L16 = Workload(
    name="verify_l16_8k", hidden=4096, num_heads=32, num_kv_heads=8, head_dim=128,
    layer_type=FULL, window=0, kv_capacity=8208, ring=False, batch=1,
    rope_theta=1e6, seed=3, weights_bf16=True, verify_len=16, base_pos=8192)
FULL_128K_B4 = Workload(
    name="full_b4_128k_softcap", hidden=5120, num_heads=40, num_kv_heads=8,
    head_dim=128, layer_type=FULL, window=0, kv_capacity=131072, ring=False,
    batch=4, rope_theta=1e6, seed=4, seq_pos=131071, softcap=50.0)

WORKLOADS: List[Workload] = [TINY_SLIDING, FULL_32K, SLIDING_B16, VERIFY_L16, FULL_128K_B4]

# The pages' global layer: 16 query heads of 512 dims over 2 KV heads (GQA group 8), full
# attention, no V projection (V = unit-normed raw K), RoPE frequency factors and the
# post-attention norm; hidden 2816 (the dense model's width) at a 32K context.
GLOBAL_32K = Workload(name="global_hd512_32k", hidden=2816, num_heads=16, num_kv_heads=2,
                      head_dim=512, layer_type=FULL, window=0, kv_capacity=32768, ring=False,
                      batch=1, rope_theta=1e6, seed=70, seq_pos=32767, k_eq_v=True,
                      rope_freq_factors=True, post_norm=True)
# The verify block on the global layer at a 32K context: GQA group 8 admits blocks of up to
# 8 tokens (64 query rows per KV head), here the last 8 positions of the cache.
VERIFY_GLOBAL = dataclasses.replace(GLOBAL_32K, name="verify_global_hd512_32k", seq_pos=None,
                                    weights_bf16=True, verify_len=8, base_pos=32760)
# A drafter step on the verify shape: 16 context rows appended at 8176..8191 (K/V
# projections only), then a 16-token block at 8192..8207, bidirectional within the block,
# scale 1/sqrt(hd).
DRAFTER_L16 = dataclasses.replace(VERIFY_L16, name="drafter_l16_8k", block_bidir=True,
                                  attn_scale=128 ** -0.5)
DRAFTER_CTX_ROWS = 16

BY_NAME: Dict[str, Workload] = {w.name: w for w in WORKLOADS + [GLOBAL_32K, VERIFY_GLOBAL,
                                                                 DRAFTER_L16]}


def _gen(seed: int, stream: int) -> torch.Generator:
    # one independent stream per buffer so that shrinking one buffer in a test never
    # changes the others
    return torch.Generator().manual_seed(seed * 1000 + stream)


def q8_0_blocks(rows: int, cols: int, g: torch.Generator, d_mean: Optional[float] = None) -> np.ndarray:
    """Random Q8_0 matrix ``[rows, cols]`` as raw bytes ``uint8 [rows, cols/32*34]``.

    Byte layout per 32-value block: bytes 0-1 the fp16 scale (little endian),
    bytes 2..33 the 32 signed 8-bit values in column order.  Scales ~U[0.001, 0.02], or
    ~U[0.5, 1.5] * d_mean when d_mean is given.
    """
    assert cols % 32 == 0
    nb = cols // 32
    q = torch.randint(-127, 128, (rows, nb, 32), generator=g, dtype=torch.int8)
    u = torch.rand((rows, nb), generator=g, dtype=torch.float32)
    d = (u * 0.019 + 0.001 if d_mean is None else (u + 0.5) * d_mean).to(torch.float16)
    out = np.empty((rows, nb, 34), dtype=np.uint8)
    out[:, :, 0:2] = d.numpy().view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:] = q.numpy().view(np.uint8)
    return out.reshape(rows, nb * 34)


def bf16_normal(shape, g: torch.Generator, std: float = 1.0) -> torch.Tensor:
    t = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t = t * std
    return t.to(torch.bfloat16)


def norm_weight(n: int, g: torch.Generator) -> torch.Tensor:
    return torch.rand((n,), generator=g, dtype=torch.float32) + 0.5


def make_weights(w: Workload) -> Dict[str, object]:
    """Layer weights: Q/K/V/O as Q8_0 byte arrays (numpy) or bf16 tensors, norms f32."""
    H, qr, kr = w.hidden, w.q_rows, w.kv_rows
    out: Dict[str, object] = {}
    shapes = {"wq": (qr, H), "wk": (kr, H), "wv": (kr, H), "wo": (H, qr)}
    for i, (name, (r, c)) in enumerate(shapes.items()):
        g = _gen(w.seed, 10 + i)
        if name == "wv" and w.k_eq_v:
            out[name] = None  # the layer has no V projection
        elif w.weights_bf16:
            out[name] = bf16_normal((r, c), g, std=0.02)
        else:
            out[name] = q8_0_blocks(r, c, g)
    out["w_in"] = norm_weight(H, _gen(w.seed, 20))
    out["w_q"] = norm_weight(w.head_dim, _gen(w.seed, 21))
    out["w_k"] = norm_weight(w.head_dim, _gen(w.seed, 22))
    # per-pair RoPE frequency factors, U[1, 4] (the pages load them from the model file)
    out["rope_ff"] = (torch.rand((w.head_dim // 2,), generator=_gen(w.seed, 23),
                                 dtype=torch.float32) * 3.0 + 1.0) if w.rope_freq_factors else None
    out["w_post"] = norm_weight(H, _gen(w.seed, 24)) if w.post_norm else None
    return out


def make_positions(w: Workload) -> np.ndarray:
    """Per-sequence decode position ``seq_pos`` (int32 [B])."""
    if w.seq_pos_range is not None:
        lo, hi = w.seq_pos_range
        g = _gen(w.seed, 30)
        return torch.randint(lo, hi + 1, (w.batch,), generator=g, dtype=torch.int32).numpy()
    pos = w.seq_pos if w.seq_pos is not None else w.base_pos
    return np.full((w.batch,), pos, dtype=np.int32)


def make_x(w: Workload, rows: Optional[int] = None) -> torch.Tensor:
    """Layer input ``x`` bf16 ``[rows, hidden]`` (rows = batch, or verify length)."""
    if rows is None:
        rows = w.verify_len if w.verify_len else w.batch
    return bf16_normal((rows, w.hidden), _gen(w.seed, 40))


def make_kv_cache(w: Workload) -> Dict[str, torch.Tensor]:
    """Prefilled KV cache, bf16 ``[B, n_kv, capacity, head_dim]``, every slot ~N(0,1).

    Every slot holds a random row; which slots the step may read is decided by the
    positions and the window, never by the contents.
    """
    shape = (w.batch, w.num_kv_heads, w.kv_capacity, w.head_dim)
    return {"k_cache": bf16_normal(shape, _gen(w.seed, 50)),
            "v_cache": bf16_normal(shape, _gen(w.seed, 51))}


def make_tq_signs(head_dim: int, seed: int) -> np.ndarray:
    """The +-1 sign pre-multiply of a quantised-KV format (int8 [head_dim]), seeded."""
    g = _gen(seed, 60)
    return (torch.randint(0, 2, (head_dim,), generator=g, dtype=torch.int8) * 2 - 1).numpy()


@dataclasses.dataclass(frozen=True)
class FfnWorkload:
    """The dense FFN half of a layer: hidden H, intermediate I, batch rows."""

    name: str
    hidden: int
    intermediate: int
    batch: int
    seed: int
    eps: float = 1e-6
    scalar_per_channel: bool = False

    def replace(self, **kw) -> "FfnWorkload":
        return dataclasses.replace(self, **kw)


# the dense MLP of the pages' decode (2816 -> 5760 gate and up, back to 2816), batch 1
FFN_B1 = FfnWorkload(name="ffn_b1", hidden=2816, intermediate=5760, batch=1, seed=6)
FFN_B16 = FfnWorkload(name="ffn_b16", hidden=2816, intermediate=5760, batch=16, seed=7)
FFN_BY_NAME: Dict[str, FfnWorkload] = {f.name: f for f in (FFN_B1, FFN_B16)}


def make_ffn_weights(f: FfnWorkload) -> Dict[str, object]:
    """Q8_0 gate, up [I, H] and down [H, I], f32 norm weights ~U[0.5, 1.5], the layer
    scalar ~U[0.5, 1.5] (one value or one per channel).  The Q8_0 scales are sized so that
    each weight has standard deviation about 1/sqrt(fan-in) (q ~U{-127..127} has standard
    deviation ~73.3): the gate pre-activations are then O(1), where GELU is not linear."""
    H, I = f.hidden, f.intermediate
    q_std = 73.3
    out: Dict[str, object] = {
        "w_gate": q8_0_blocks(I, H, _gen(f.seed, 70), d_mean=1.0 / (q_std * H ** 0.5)),
        "w_up": q8_0_blocks(I, H, _gen(f.seed, 71), d_mean=1.0 / (q_std * H ** 0.5)),
        "w_down": q8_0_blocks(H, I, _gen(f.seed, 72), d_mean=1.0 / (q_std * I ** 0.5)),
        "w_pre": norm_weight(H, _gen(f.seed, 73)),
        "w_post": norm_weight(H, _gen(f.seed, 74)),
        "scalar": norm_weight(H if f.scalar_per_channel else 1, _gen(f.seed, 75)),
    }
    return out


def make_ffn_input(f: FfnWorkload, rows: Optional[int] = None) -> torch.Tensor:
    """The FFN input h (the attention half's output), bf16 [rows, H] ~N(0, 1)."""
    return bf16_normal((rows or f.batch, f.hidden), _gen(f.seed, 76))
