"""Pins of the oracle's FP8 (e4m3) KV-cache path to things other than itself (CPU only).

The FP8 cache is the QuantSpec path of cuDNN FE-OSS "Gated Attention Block (SM107)"
(API: static per-tensor scales, dtype torch.float8_e4m3fn): K = k_descale * e4m3(code),
V = v_descale * e4m3(code).  Each pin catches a plausible mistake:
  * the e4m3 decoder: every one of the 256 codes against torch's float8_e4m3fn
    conversion (a library routine), and closed forms of the format (bias 7,
    subnormals m * 2^-9, 448 the largest value, NaN at S.1111.111);
  * the attention over FP8 pools: with power-of-two descales every K/V value is
    exactly a BF16 value, so the FP8 oracle must give bit for bit what the
    (separately pinned) BF16 oracle gives on those BF16 pools;
  * brute-force loops on tiny inputs with non-power-of-two descales, values taken
    from the library conversion;
  * which operand each descale scales: O is linear in v_descale, and k_descale
    only multiplies the scores (it folds into the scale); swapping the two fails.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gated_gqa_attention_gb300 import workloads


def _codes(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).numpy()


def _values(t: torch.Tensor, descale: float) -> np.ndarray:
    """Library dequantisation: torch's float8_e4m3fn -> float64, times the descale."""
    return t.to(torch.float64).numpy() * descale


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_e4m3_all_codes_match_library():
    c = np.arange(256, dtype=np.uint8)
    got = oracle.double_from_e4m3(c)
    want = torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))  # -0.0 at 0x80


def test_e4m3_closed_forms():
    # e4m3 ("fn"): 1 sign, 4 exponent bits (bias 7), 3 fraction bits, no infinities
    cases = {
        0x00: 0.0, 0x38: 1.0, 0xB8: -1.0, 0x40: 2.0, 0x3C: 1.5, 0x30: 0.5,
        0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x0F: 1.875 * 2.0 ** -6,
        0x7E: 448.0, 0xFE: -448.0, 0x77: 240.0, 0x78: 256.0,
    }
    for code, v in cases.items():
        assert oracle.double_from_e4m3([code])[0] == v, hex(code)
    assert math.isnan(oracle.double_from_e4m3([0x7F])[0])
    assert math.isnan(oracle.double_from_e4m3([0xFF])[0])
    assert math.copysign(1.0, oracle.double_from_e4m3([0x80])[0]) == -1.0


def _tiny_fp8(seed, lengths, hq, hkv, d, scale=None, slots=None):
    return workloads.make(lengths, seed=seed, hq=hq, hkv=hkv, head_dim=d, layout="perm", pool_slots=slots,
                          scale=scale if scale is not None else 1.0 / math.sqrt(d), kv="e4m3")


@pytest.mark.parametrize("seed,lengths,hq,hkv,d,kd,vd", [
    (31, [5, 0, 9], 4, 2, 16, 2.0 ** -3, 2.0 ** -5),
    (32, [33, 1, 17], 16, 2, 256, 2.0 ** -6, 2.0 ** -6),
    (33, [12, 40], 6, 2, 32, 2.0 ** 2, 2.0 ** -9),
])
def test_fp8_decode_equals_bf16_decode_when_values_are_bf16(seed, lengths, hq, hkv, d, kd, vd):
    inp = _tiny_fp8(seed, lengths, hq, hkv, d)
    # power-of-two descale: descale * e4m3(code) has <= 4 significant bits -> exact in BF16
    kb = torch.from_numpy(_values(inp["k_pool"], kd)).to(torch.bfloat16)
    vb = torch.from_numpy(_values(inp["v_pool"], vd)).to(torch.bfloat16)
    assert np.array_equal(kb.to(torch.float64).numpy(), _values(inp["k_pool"], kd))
    for splits, window, sinks in [(0, 0, None), (3, 0, None), (0, 7, None), (0, 0, np.linspace(-1, 2, hq))]:
        f8 = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                           inp["kv_indices"], inp["scale"], num_splits=splits, window=window, sinks=sinks,
                           k_descale=kd, v_descale=vd)
        bf = oracle.decode(inp["q"], inp["gate"], kb, vb, inp["kv_indptr"], inp["kv_indices"], inp["scale"],
                           num_splits=splits, window=window, sinks=sinks)
        assert np.array_equal(f8.o_f64, bf.o_f64, equal_nan=True)
        assert np.array_equal(f8.lse, bf.lse, equal_nan=True)
        assert np.array_equal(f8.out, bf.out)


def _brute_force_fp8(inp, kd, vd):
    """Pure-Python loops, math.fsum, values from the library conversion."""
    q = inp["q"].to(torch.float64).numpy()
    k = _values(inp["k_pool"], kd)
    v = _values(inp["v_pool"], vd)
    ip = inp["kv_indptr"].tolist()
    ix = inp["kv_indices"].tolist()
    B, Hq, D = q.shape
    G = Hq // k.shape[1]
    O = np.zeros((B, Hq, D))
    for b in range(B):
        rows = ix[ip[b]:ip[b + 1]]
        for h in range(Hq):
            if not rows:
                continue
            s = [inp["scale"] * math.fsum(q[b, h, dd] * k[r, h // G, dd] for dd in range(D)) for r in rows]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            z = math.fsum(w)
            for dd in range(D):
                O[b, h, dd] = math.fsum(w[j] * v[r, h // G, dd] for j, r in enumerate(rows)) / z
    return O


@pytest.mark.parametrize("seed,lengths,hq,hkv,d", [
    (41, [5], 4, 2, 8), (42, [1, 7, 3], 6, 2, 16), (43, [16, 0, 9], 8, 8, 4), (44, [12, 3], 9, 3, 12),
])
def test_fp8_decode_brute_force(seed, lengths, hq, hkv, d):
    inp = _tiny_fp8(seed, lengths, hq, hkv, d)
    kd, vd = 0.0137, 0.0291  # not powers of two, and different
    res = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                        inp["kv_indices"], inp["scale"], k_descale=kd, v_descale=vd)
    want = _brute_force_fp8(inp, kd, vd)
    np.testing.assert_allclose(res.o_f64, want, rtol=1e-12, atol=1e-15)
    assert np.array_equal(res.o_bf16, oracle.bf16_from_double(res.o_f64))
    assert np.array_equal(res.out, oracle.gate(res.o_bf16, _bf16_bits(inp["gate"])))
    # a planted mistake -- the two descales swapped -- fails the same comparison
    bad = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                        inp["kv_indices"], inp["scale"], k_descale=vd, v_descale=kd)
    assert not np.allclose(bad.o_f64, want, rtol=1e-6, atol=1e-9)


def test_fp8_descales_scale_the_right_operand():
    inp = _tiny_fp8(51, [20, 9, 33], 16, 2, 64)
    args = (inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"], inp["kv_indices"])
    base = oracle.decode(*args, inp["scale"], k_descale=0.02, v_descale=0.03)
    # O is linear in v_descale; the LSE does not depend on it
    v2 = oracle.decode(*args, inp["scale"], k_descale=0.02, v_descale=0.03 * 2.5)
    np.testing.assert_allclose(v2.o_f64, 2.5 * base.o_f64, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(v2.lse, base.lse, rtol=1e-15, atol=0)
    # k_descale multiplies the scores only: it folds into the scale
    k2 = oracle.decode(*args, inp["scale"] * 0.02 / 0.05, k_descale=0.05, v_descale=0.03)
    np.testing.assert_allclose(k2.o_f64, base.o_f64, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(k2.lse, base.lse, rtol=1e-13, atol=0)
    # ... and it does change the result (the scores are not constant)
    k3 = oracle.decode(*args, inp["scale"], k_descale=0.05, v_descale=0.03)
    assert not np.allclose(k3.o_f64, base.o_f64, rtol=1e-6)
