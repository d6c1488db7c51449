"""Pins of the quantised-KV (TurboQuant) oracle, CPU only.

* the Lloyd-Max quantiser of N(0,1): the 2-level closed form (centroids +-sqrt(2/pi),
  mean squared error 1 - 2/pi), the published 4- and 8-level tables (Max, "Quantizing for
  minimum distortion", IRE Trans. Inform. Theory, 1960: levels, thresholds and error to
  the printed digits), for 16, 32, 64 and 256 levels the two optimality conditions checked
  with scipy's truncated-normal mean, and the Panter-Dite high-resolution error
  (sqrt(3) pi / 2) 4^-bits approached from below as the bit count grows;
* the normalised FWHT against the Hadamard matrix built from its popcount definition;
* the encoder against a brute-force nearest-centroid search in the documented packing (4-bit
  nibbles; 5-, 6- and 8-bit codes one byte per element);
* attention over codes against attention over the dequantised, un-rotated cache, written
  out here in the original domain (orthogonality of the rotation and the sign undo).
"""
import math

import numpy as np
import pytest

import oracle


def hadamard(n):
    i = np.arange(n)
    pop = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pop % 2 == 0, 1.0, -1.0) / math.sqrt(n)


def signs_for(hd, seed):
    return np.where(np.random.default_rng(seed).random(hd) < 0.5, -1, 1).astype(np.int8)


# ------------------------------------------------------------------ Lloyd-Max

def test_two_level_quantiser_closed_form(orc):
    c, b, _ = oracle.lloyd_max_normal(1)
    assert abs(c[1] - math.sqrt(2 / math.pi)) < 1e-12 and abs(c[0] + c[1]) < 1e-15
    assert b[1] == 0.0
    assert abs(oracle.lloyd_max_mse(c, b) - (1 - 2 / math.pi)) < 1e-12


@pytest.mark.parametrize("bits,levels,thresholds,mse", [
    (2, [0.4528, 1.5104], [0.9816], 0.1175),
    (3, [0.2451, 0.7560, 1.3440, 2.1520], [0.5006, 1.0500, 1.7480], 0.03454),
])
def test_published_quantiser_tables(orc, bits, levels, thresholds, mse):
    c, b, _ = oracle.lloyd_max_normal(bits)
    half = len(c) // 2
    assert np.max(np.abs(c[half:] - levels)) < 6e-4
    assert np.max(np.abs(b[half + 1:-1] - thresholds)) < 6e-4
    assert abs(oracle.lloyd_max_mse(c, b) - mse) < 1e-4


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_optimality_conditions(orc, bits):
    from scipy.stats import norm, truncnorm
    c, b, _ = oracle.lloyd_max_normal(bits)
    n = len(c)
    assert np.all(np.diff(c) > 0) and np.max(np.abs(c + c[::-1])) < 1e-12  # sorted, symmetric
    assert np.max(np.abs(b[1:-1] - 0.5 * (c[:-1] + c[1:]))) < 1e-15       # nearest neighbour
    # centroid condition: each level is the mean of N(0, 1) on its cell
    means = np.array([truncnorm.mean(b[i], b[i + 1]) for i in range(n)])
    assert np.max(np.abs(means - c)) < 5e-9
    # mean squared error against direct numerical integration of the cell errors
    num = sum(norm.expect(lambda x, ci=c[i]: (x - ci) ** 2, lb=b[i], ub=b[i + 1]) for i in range(n))
    assert abs(num - oracle.lloyd_max_mse(c, b)) < 1e-9


def test_high_resolution_asymptote(orc):
    # Panter-Dite: the optimal b-bit quantiser of N(0, 1) has mean squared error
    # (sqrt(3) pi / 2) 4^-b as b grows; the exact quantisers approach it from below
    r = []
    for bits in (4, 5, 6, 7, 8):
        c, b, _ = oracle.lloyd_max_normal(bits)
        r.append(oracle.lloyd_max_mse(c, b) * 4.0 ** bits / (math.sqrt(3.0) * math.pi / 2.0))
    assert all(0.85 < x < 1.0 for x in r) and all(x < y for x, y in zip(r, r[1:]))
    assert r[-1] > 0.99


# ------------------------------------------------------------------ rotation

@pytest.mark.parametrize("n", [8, 64, 256])
def test_fwht_is_the_normalised_hadamard_matrix(orc, n):
    x = np.random.default_rng(n).normal(size=n)
    assert np.max(np.abs(oracle.fwht(x) - hadamard(n) @ x)) < 1e-13
    assert np.max(np.abs(oracle.fwht(oracle.fwht(x)) - x)) < 1e-13  # involution


@pytest.mark.parametrize("hd", [64, 128, 256, 512])
def test_rotation_blocks_and_inverse(orc, hd):
    s = signs_for(hd, hd)
    x = np.random.default_rng(hd + 1).normal(size=hd)
    B = min(hd, 256)
    want = np.concatenate([hadamard(B) @ (s[k:k + B] * x[k:k + B]) for k in range(0, hd, B)])
    r = oracle.tq_rotate(x, s)
    assert np.max(np.abs(r - want)) < 1e-12
    assert np.max(np.abs(oracle.tq_unrotate(r, s) - x)) < 1e-12


# ------------------------------------------------------------------ encoder

def unpack(codes, hd, bits):
    if bits != 4:  # 5-, 6- and 8-bit codes: one byte per element
        return codes.astype(np.int64)
    lo, hi = codes & 15, codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (hd,)).astype(np.int64)


@pytest.mark.parametrize("hd,bits", [(64, 4), (128, 8), (256, 4), (512, 8), (128, 5), (256, 6)])
def test_encoder_is_the_nearest_centroid(orc, hd, bits):
    s = signs_for(hd, 7)
    c, b, _ = oracle.lloyd_max_normal(bits)
    x = np.random.default_rng(hd * bits).normal(size=(20, hd)) * 3.0
    codes, norms = oracle.tq_encode_rows(x, s, bits, b)
    B = min(hd, 256)
    got = unpack(codes, hd, bits)
    for r in range(20):
        u = np.concatenate([hadamard(B) @ (s[k:k + B] * x[r, k:k + B]) for k in range(0, hd, B)])
        for k in range(0, hd, B):
            nrm = math.sqrt(np.mean(u[k:k + B] ** 2))
            assert norms[r, k // B] == np.float32(nrm)
            e = u[k:k + B] / nrm
            want = np.argmin(np.abs(e[:, None] - c[None, :]), axis=1)  # brute force
            assert np.array_equal(got[r, k:k + B], want)


def test_encoder_scale_invariance_and_zero_row(orc):
    hd, bits = 128, 4
    s = signs_for(hd, 8)
    _, b, _ = oracle.lloyd_max_normal(bits)
    x = np.random.default_rng(9).normal(size=(1, hd))
    c1, n1 = oracle.tq_encode_rows(x, s, bits, b)
    c2, n2 = oracle.tq_encode_rows(x * 8.0, s, bits, b)
    assert np.array_equal(c1, c2) and n2[0, 0] == 8.0 * n1[0, 0]
    cz, nz = oracle.tq_encode_rows(np.zeros((1, hd)), s, bits, b)
    assert nz[0, 0] == 0.0 and np.all(unpack(cz, hd, bits) == len(b) // 2)  # 0 -> upper cell


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_round_trip_error_matches_the_quantiser(orc, bits):
    hd = 256
    s = signs_for(hd, 10)
    c, b, _ = oracle.lloyd_max_normal(bits)
    x = np.random.default_rng(11).normal(size=(400, hd))
    codes, norms = oracle.tq_encode_rows(x, s, bits, b)
    u = np.stack([oracle.tq_rotate(r, s) for r in x])
    uh = oracle.tq_decode_rows(codes, norms, hd, bits, c)
    rel = np.mean(np.sum((u - uh) ** 2, axis=1) / np.sum(u ** 2, axis=1))
    mse = oracle.lloyd_max_mse(c, b)
    assert 0.8 * mse < rel < 1.2 * mse
    back = np.stack([oracle.tq_unrotate(r, s) for r in uh])  # error is the same un-rotated
    assert abs(np.mean(np.sum((x - back) ** 2, axis=1) / np.sum(x ** 2, axis=1)) - rel) < 1e-12


# ------------------------------------------------------------------ attention

def softmax_attention(q, K, V, scale, softcap):
    s = scale * (K @ q)
    if softcap > 0:
        s = softcap * np.tanh(s / softcap)
    p = np.exp(s - s.max())
    return (p / p.sum()) @ V


@pytest.mark.parametrize("hd,bits,softcap", [(128, 8, 0.0), (256, 4, 30.0), (512, 8, 0.0),
                                             (128, 6, 0.0), (64, 5, 20.0)])
def test_attention_over_codes_is_attention_over_the_dequantised_cache(orc, hd, bits, softcap):
    rng = np.random.default_rng(hd + bits)
    s = signs_for(hd, 12)
    c, b, _ = oracle.lloyd_max_normal(bits)
    n = 50
    k = rng.normal(size=(n, hd))
    v = rng.normal(size=(n, hd))
    q = rng.normal(size=hd)
    kc, kn = oracle.tq_encode_rows(k, s, bits, b)
    vc, vn = oracle.tq_encode_rows(v, s, bits, b)
    rows = np.array([3, 0, 17, 49, 22, 8])
    got = oracle.attend_tq(q, s, bits, c, kc, kn, vc, vn, rows, scale=0.125, softcap=softcap)
    K = np.stack([oracle.tq_unrotate(r, s) for r in oracle.tq_decode_rows(kc[rows], kn[rows], hd, bits, c)])
    V = np.stack([oracle.tq_unrotate(r, s) for r in oracle.tq_decode_rows(vc[rows], vn[rows], hd, bits, c)])
    want = softmax_attention(q, K, V, 0.125, softcap)
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want))


def test_hybrid_attention_raw_keys_coded_values(orc):
    import torch
    hd, bits = 256, 8
    rng = np.random.default_rng(13)
    s = signs_for(hd, 14)
    c, b, _ = oracle.lloyd_max_normal(bits)
    kb = torch.from_numpy(rng.normal(size=(30, hd)).astype(np.float32)).to(torch.bfloat16)
    v = rng.normal(size=(30, hd))
    vc, vn = oracle.tq_encode_rows(v, s, bits, b)
    q = rng.normal(size=hd)
    rows = np.arange(0, 30, 3)
    got = oracle.attend_tq(q, s, bits, c, None, None, vc, vn, rows, k_bf16=kb)
    K = kb.to(torch.float64).numpy()[rows]
    V = np.stack([oracle.tq_unrotate(r, s) for r in oracle.tq_decode_rows(vc[rows], vn[rows], hd, bits, c)])
    want = softmax_attention(q, K, V, 1.0, 0.0)
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want))
