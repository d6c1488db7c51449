"""CPU checks of the C-ABI library: it builds, loads, and exports every declared symbol.

No compute call is made here (there is no GPU); argument checks that run before any
CUDA call are exercised where the call needs no device.
"""
import ctypes
import os

import pytest

from quantized_attention_layer_gb300 import build, hfa


@pytest.fixture(scope="module")
def libhfa():
    build.build()
    return hfa.lib()


def test_header_declares_the_boundary():
    names = hfa.header_functions()
    for required in ("hfa_layer_create", "hfa_decode_step", "hfa_verify_block", "hfa_destroy",
                     "hfa_last_error", "hfa_debug_taps", "hfa_decode_step_host"):
        assert required in names


def test_library_exports_every_declared_symbol(libhfa):
    for name in hfa.header_functions():
        assert hasattr(libhfa, name), f"libhfa.so does not export {name}"


def test_create_rejects_bad_descriptors_before_touching_a_device(libhfa):
    from quantized_attention_layer_gb300 import workloads as wl
    bad = [
        dict(hidden=100),             # not a multiple of 32
        dict(head_dim=96),            # unsupported head_dim
        dict(num_kv_heads=3),         # nh % nkv != 0
        dict(max_batch=17),
        dict(kv_capacity=0),
    ]
    for kw in bad:
        d = hfa.desc_for(wl.TINY_SLIDING)
        for k, v in kw.items():
            setattr(d, k, v)
        h = ctypes.c_void_p()
        dummy = ctypes.c_void_p(16)
        st = libhfa.hfa_layer_create(ctypes.byref(d), dummy, dummy, dummy, dummy, dummy, dummy,
                                     dummy, None, ctypes.byref(h))
        assert st in (hfa.HFA_EINVAL, hfa.HFA_EUNSUPPORTED), (kw, st)
        assert not h.value
        assert libhfa.hfa_last_error(None)


def _create_status(libhfa, d):
    h = ctypes.c_void_p()
    dummy = ctypes.c_void_p(16)
    st = libhfa.hfa_layer_create(ctypes.byref(d), dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                 None, ctypes.byref(h))
    assert not h.value
    return st


def test_hidden_statuses_follow_the_block_format(libhfa):
    from quantized_attention_layer_gb300 import workloads as wl
    d = hfa.desc_for(wl.TINY_SLIDING)
    d.hidden = 100  # not whole 32-value blocks: an invalid layer
    assert _create_status(libhfa, d) == hfa.HFA_EINVAL
    d.hidden = 96   # whole Q8_0 blocks, but not a multiple of 64: valid, not covered
    assert _create_status(libhfa, d) == hfa.HFA_EUNSUPPORTED
    assert b"multiples of 64" in libhfa.hfa_last_error(None)


def test_verify_refuses_caches_past_32_bit_rows(libhfa):
    from quantized_attention_layer_gb300 import workloads as wl
    d = hfa.desc_for(wl.VERIFY_L16)
    d.num_kv_heads = 256
    d.num_heads = 256
    d.kv_capacity = (1 << 23) + 1  # 256 x (2^23 + 1) rows: past 2^31
    assert _create_status(libhfa, d) == hfa.HFA_EUNSUPPORTED
    assert b"32-bit" in libhfa.hfa_last_error(None)


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="a valid descriptor with placeholder weights must not reach a GPU")
def test_global_layer_passes_validation_for_decode_and_verify(libhfa):
    # head dim 512 with a verify length is a covered shape: without a GPU the create stops
    # at the device query, after the descriptor checks
    from quantized_attention_layer_gb300 import workloads as wl
    for w in (wl.GLOBAL_32K, wl.VERIFY_GLOBAL):
        d = hfa.desc_for(w)
        assert d.head_dim == 512 and (d.max_verify_len > 0) == (w is wl.VERIFY_GLOBAL)
        assert _create_status(libhfa, d) == hfa.HFA_EDEVICE, libhfa.hfa_last_error(None)
        assert b"no CUDA device" in libhfa.hfa_last_error(None)


def test_ring_needs_capacity_equal_to_window(libhfa):
    from quantized_attention_layer_gb300 import workloads as wl
    d = hfa.desc_for(wl.SLIDING_B16)
    d.kv_capacity = 2048
    h = ctypes.c_void_p()
    dummy = ctypes.c_void_p(16)
    st = libhfa.hfa_layer_create(ctypes.byref(d), dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                 None, ctypes.byref(h))
    assert st == hfa.HFA_EINVAL


def test_null_handle_is_rejected(libhfa):
    assert libhfa.hfa_decode_step(None, None, None, None, None, 1, None, None, None) == hfa.HFA_EINVAL
    assert libhfa.hfa_destroy(None) == hfa.HFA_EINVAL


def test_quantised_kv_format_rejects_bad_arguments_before_any_device_call(libhfa):
    import numpy as np
    h = ctypes.c_void_p()
    ok = np.ones(128, dtype=np.int8)
    bad = ok.copy()
    bad[5] = 0
    P = lambda a: ctypes.c_void_p(a.ctypes.data)  # noqa: E731
    assert libhfa.hfa_tq_create(128, 3, P(ok), ctypes.byref(h)) == hfa.HFA_EUNSUPPORTED
    assert libhfa.hfa_tq_create(128, 7, P(ok), ctypes.byref(h)) == hfa.HFA_EUNSUPPORTED
    assert libhfa.hfa_tq_create(96, 8, P(ok), ctypes.byref(h)) == hfa.HFA_EUNSUPPORTED
    assert libhfa.hfa_tq_create(128, 8, P(bad), ctypes.byref(h)) == hfa.HFA_EINVAL
    assert b"signs[5]" in libhfa.hfa_last_error(None)
    assert libhfa.hfa_tq_create(128, 8, None, ctypes.byref(h)) == hfa.HFA_EINVAL
    assert not h.value


def test_ffn_create_rejects_bad_descriptors_before_any_device_call(libhfa):
    h = ctypes.c_void_p()
    dummy = ctypes.c_void_p(16)  # never dereferenced: every case fails validation first

    def create(**kw):
        base = dict(hidden=256, intermediate=512, eps=1e-6, scalar_len=1, max_batch=1)
        base.update(kw)
        d = hfa.hfa_ffn_desc(**base)
        return libhfa.hfa_ffn_create(ctypes.byref(d), dummy, dummy, dummy, dummy, dummy, dummy,
                                     None, ctypes.byref(h))

    assert create(hidden=48) == hfa.HFA_EINVAL          # not whole Q8_0 blocks
    assert create(intermediate=0) == hfa.HFA_EINVAL
    assert create(scalar_len=7) == hfa.HFA_EINVAL       # one scalar or one per channel
    assert create(max_batch=17) == hfa.HFA_EUNSUPPORTED
    assert create(max_batch=0) == hfa.HFA_EUNSUPPORTED
    assert create(eps=-1.0) == hfa.HFA_EINVAL
    assert b"eps" in libhfa.hfa_ffn_last_error(None)
    d = hfa.hfa_ffn_desc(hidden=256, intermediate=512, eps=1e-6, scalar_len=1, max_batch=1)
    assert libhfa.hfa_ffn_create(ctypes.byref(d), None, dummy, dummy, dummy, dummy, dummy, None,
                                 ctypes.byref(h)) == hfa.HFA_EINVAL
    assert not h.value
    assert libhfa.hfa_ffn_step(None, None, None, 1, None, None, None) == hfa.HFA_EINVAL
    assert libhfa.hfa_ffn_destroy(None) == hfa.HFA_EINVAL
