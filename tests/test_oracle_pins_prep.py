"""Pins of the oracle for the step before attention (Q/K RMSNorm, partial RoPE, KV
write; cuDNN FE-OSS "Gated Attention Block (SM107)", Overview stages (2)+(3)).

* RMSNorm against the library torch.nn.functional.rms_norm in float64.
* RoPE against a complex-number rotation (y_i + i y_j) * e^{i theta} on numpy
  complex128 (an independent formulation of the rotate-half convention), and the
  closed forms theta = 0, pi/2, pi.
* Scale invariance (eps = 0), pass-through of the gate and V, untouched pool rows.
* A planted mistake (the sine sign flipped) fails the rotation pin."""
import math

import numpy as np
import pytest
import torch

import oracle

HQ, HKV, D = 4, 2, 256


def bf16(x) -> np.ndarray:
    return torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f64(bits) -> np.ndarray:
    return oracle.double_from_bf16(bits)


def make(B, rope_dim, theta=None, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    qgkv = bf16(rng.standard_normal((B, (2 * HQ + 2 * HKV) * D)) * scale)
    wq = bf16(rng.uniform(0.5, 1.5, D))
    wk = bf16(rng.uniform(0.5, 1.5, D))
    if theta is None:
        theta = rng.uniform(0, 2 * math.pi, (B, rope_dim // 2))
    ang = np.concatenate([theta, theta], axis=1) if rope_dim else np.zeros((B, 0))
    cos_t, sin_t = bf16(np.cos(ang)), bf16(np.sin(ang))
    slots = rng.permutation(50)[:B].astype(np.int32)
    kp = bf16(rng.standard_normal((50, HKV, D)))
    vp = bf16(rng.standard_normal((50, HKV, D)))
    return qgkv, wq, wk, cos_t, sin_t, slots, kp, vp


def run(qgkv, wq, wk, cos_t, sin_t, rope_dim, slots, kp, vp, eps=1e-6):
    return oracle.qk_norm_rope_kv_write(qgkv, wq, wk, eps, cos_t, sin_t, rope_dim, slots, kp, vp, HQ, HKV, D)


def test_rmsnorm_against_library():
    qgkv, wq, wk, cs, sn, slots, kp, vp = make(3, 0)
    qo, go, kpo, vpo = run(qgkv, wq, wk, cs, sn, 0, slots, kp, vp)       # rope_dim = 0: norm only
    x = torch.from_numpy(f64(qgkv)).view(3, -1)
    for b in range(3):
        for h in range(HQ):
            ref = torch.nn.functional.rms_norm(x[b, h * D:(h + 1) * D], (D,), torch.from_numpy(f64(wq)), 1e-6)
            assert np.array_equal(qo[b, h], oracle.bf16_from_double(ref.numpy()))
        for h in range(HKV):
            off = (2 * HQ + h) * D
            ref = torch.nn.functional.rms_norm(x[b, off:off + D], (D,), torch.from_numpy(f64(wk)), 1e-6)
            assert np.array_equal(kpo[slots[b], h], oracle.bf16_from_double(ref.numpy()))


@pytest.mark.parametrize("rope_dim", [64, 128, 256])
def test_rope_against_complex_rotation(rope_dim):
    B = 3
    qgkv, wq, wk, cs, sn, slots, kp, vp = make(B, rope_dim, seed=rope_dim)
    qo, go, kpo, vpo = run(qgkv, None, None, cs, sn, rope_dim, slots, kp, vp)   # no norm: rope only
    x = f64(qgkv).reshape(B, -1)
    c, s = f64(cs), f64(sn)
    half = rope_dim // 2
    for b in range(B):
        for h in range(HQ):
            y = x[b, h * D:(h + 1) * D]
            # the two halves as one complex number; rotation by the (rounded) angle's cos/sin
            z = (y[:half] + 1j * y[half:rope_dim]) * (c[b, :half] + 1j * s[b, :half])
            want = np.concatenate([z.real, z.imag, y[rope_dim:]])
            assert np.array_equal(qo[b, h], oracle.bf16_from_double(want))


def test_rope_closed_forms():
    B, r = 3, 64
    qgkv, wq, wk, cs, sn, slots, kp, vp = make(B, r, seed=3)
    x = f64(qgkv).reshape(B, -1)
    for theta, fn in [(0.0, lambda y: y),                                                 # identity
                      (math.pi / 2, lambda y: np.concatenate([-y[32:64], y[:32], y[64:]])),  # rotate half
                      (math.pi, lambda y: np.concatenate([-y[:64], y[64:]]))]:            # negate
        ang = np.full((B, r), theta)
        c = bf16(np.round(np.cos(ang), 12))
        s = bf16(np.round(np.sin(ang), 12))
        qo, _, kpo, _ = run(qgkv, None, None, c, s, r, slots, kp, vp)
        for b in range(B):
            assert np.array_equal(qo[b, 0], oracle.bf16_from_double(fn(x[b, :D])))


def test_scale_invariance_and_pass_through():
    B = 4
    qgkv, wq, wk, cs, sn, slots, kp, vp = make(B, 64, seed=9)
    a = run(qgkv, wq, wk, cs, sn, 64, slots, kp, vp, eps=0.0)
    doubled = bf16(f64(qgkv) * 4.0)                       # exact: a power of two
    b_ = run(doubled, wq, wk, cs, sn, 64, slots, kp, vp, eps=0.0)
    assert np.array_equal(a[0], b_[0])                    # q_out: RMSNorm removes the scale
    assert np.array_equal(a[2][slots], b_[2][slots])      # new K rows likewise
    qo, go, kpo, vpo = a
    row = qgkv.reshape(B, -1)
    for b in range(B):
        assert np.array_equal(go[b].reshape(-1), row[b, HQ * D:2 * HQ * D])                    # gate copied
        assert np.array_equal(vpo[slots[b]].reshape(-1), row[b, (2 * HQ + HKV) * D:])           # V written
    untouched = np.setdiff1d(np.arange(50), slots)
    assert np.array_equal(kpo[untouched], kp[untouched]) and np.array_equal(vpo[untouched], vp[untouched])


def test_planted_sine_sign_mistake_is_caught():
    B, r = 2, 64
    qgkv, wq, wk, cs, sn, slots, kp, vp = make(B, r, seed=11)
    flipped = bf16(-f64(sn))                               # the mistake: rotation the wrong way
    qo, _, _, _ = run(qgkv, None, None, cs, flipped, r, slots, kp, vp)
    x = f64(qgkv).reshape(B, -1)
    c, s = f64(cs), f64(sn)
    y = x[0, :D]
    z = (y[:32] + 1j * y[32:64]) * (c[0, :32] + 1j * s[0, :32])
    want = oracle.bf16_from_double(np.concatenate([z.real, z.imag, y[64:]]))
    assert not np.array_equal(qo[0, 0], want)
