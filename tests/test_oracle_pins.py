"""Pins of the FP64 oracle to things other than itself (CPU only).

Each pin is chosen so a plausible mistake in the oracle fails it:
  * BF16 rounding: a library conversion (torch float32 -> bfloat16), hand-derived
    ties and subnormal/overflow cases, and the identity on every BF16 value.
  * sigmoid: every one of the 65 536 gate codes against a 50-digit mpmath
    evaluation rounded by an independent RNE (wrong sign, base, or double
    rounding would show up here).
  * gate product: closed forms (sigmoid(0) = 1/2 halves o exactly; saturation
    leaves o unchanged) and a float32 library product.
  * attention: brute-force pure-Python loops on tiny inputs, the library SDPA in
    float64 (GQA mapping, scale, transposed operands), closed forms (q = 0 or
    equal keys -> mean of V; one key -> that V row), the split-merge
    formulation for many split counts, placement invariance, zero length.
  * sensitivity: planted mistakes (a dropped scale, a flipped gate sign, a
    wrong head mapping) fail the same comparisons.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gated_gqa_attention_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_float(b) -> np.ndarray:
    return oracle.double_from_bf16(b)


# --------------------------------------------------------------------------- rounding

def test_bf16_rounding_golden():
    path = os.path.join(GOLDEN, "bf16_rounding_cases.txt")
    n = 0
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        lit, hexbits = line.split()[:2]
        got = int(oracle.bf16_from_double([float(lit)])[0])
        assert got == int(hexbits, 16), (lit, hex(got), hexbits)
        n += 1
    assert n >= 15


def test_bf16_rounding_matches_library_for_float32_inputs():
    # For doubles that are exact float32 values, direct RNE to BF16 must equal
    # torch's float32 -> bfloat16 conversion (round-to-nearest-even).
    g = torch.Generator().manual_seed(123)
    bits = torch.randint(0, 2**32, (200_000,), generator=g, dtype=torch.int64).to(torch.int64)
    bits = bits.to(torch.int32).view(torch.float32)
    f = bits[torch.isfinite(bits)]
    # add ties and near-ties explicitly: low 16 bits = 0x8000 and neighbours
    tie_bits = (torch.randint(0, 2**15, (20_000,), generator=g).to(torch.int32) << 16) | 0x8000
    ties = tie_bits.view(torch.float32)
    more = torch.cat([ties, (tie_bits + 1).view(torch.float32), (tie_bits - 1).view(torch.float32)])
    f = torch.cat([f, more[torch.isfinite(more)]])
    want = bf16_bits(f.to(torch.bfloat16))
    got = oracle.bf16_from_double(f.double().numpy())
    assert np.array_equal(got, want)


def test_bf16_rounding_identity_on_all_codes():
    codes = np.arange(65536, dtype=np.uint16)
    x = bits_to_float(codes)
    got = oracle.bf16_from_double(x)
    finite_or_inf = ~np.isnan(x)
    assert np.array_equal(got[finite_or_inf], codes[finite_or_inf])
    assert np.all((got[~finite_or_inf] & 0x7FFF) > 0x7F80)  # NaN stays NaN


def test_bf16_rounding_no_double_rounding():
    # Just above a BF16 tie at a precision finer than float32: direct rounding
    # goes up, rounding through float32 would land on the tie and go to even.
    rng = np.random.default_rng(5)
    for _ in range(2000):
        code = int(rng.integers(0x0080, 0x7F00)) & ~1   # even code, normal range
        lo = bits_to_float(np.array([code], np.uint16))[0]
        hi = bits_to_float(np.array([code + 1], np.uint16))[0]
        mid = (lo + hi) / 2
        eps = (hi - lo) * 2.0**-30
        assert oracle.bf16_from_double([mid])[0] == code          # tie -> even
        assert oracle.bf16_from_double([mid + eps])[0] == code + 1  # above tie -> up
        assert oracle.bf16_from_double([mid - eps])[0] == code      # below tie -> down


# --------------------------------------------------------------------------- sigmoid

def _mp_rne_bf16(v) -> int:
    """Independent RNE of a positive mpmath number to BF16 bits (no ties occur:
    the sigmoid of a nonzero BF16 value is transcendental)."""
    import mpmath
    if v == 0:
        return 0
    e = int(mpmath.floor(mpmath.log(v, 2)))
    # guard log rounding at exact powers of two
    if mpmath.mpf(2) ** e > v:
        e -= 1
    elif mpmath.mpf(2) ** (e + 1) <= v:
        e += 1
    qexp = max(e - 7, -133)
    r = v / mpmath.mpf(2) ** qexp
    n = int(mpmath.floor(r + mpmath.mpf("0.5")))
    assert r + mpmath.mpf("0.5") != n, "unexpected exact tie"
    val = n * 2.0**qexp
    if val >= 2.0**128:
        return 0x7F80
    return int(np.array([val], np.float32).view(np.uint32)[0] >> 16)


def test_sigmoid_all_codes_against_50_digit_reference():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    codes = np.arange(65536, dtype=np.uint16)
    got = oracle.sigmoid_bf16(codes)
    x = bits_to_float(codes)
    mismatches = []
    for c in range(65536):
        xv = x[c]
        if np.isnan(xv):
            assert (got[c] & 0x7FFF) > 0x7F80
            continue
        if np.isinf(xv):
            want = 0x3F80 if xv > 0 else 0x0000
        elif xv == 0.0:
            want = 0x3F00
        else:
            want = _mp_rne_bf16(1 / (1 + mpmath.exp(-mpmath.mpf(float(xv)))))
        if int(got[c]) != want:
            mismatches.append((c, int(got[c]), want))
    assert not mismatches, mismatches[:10]


def test_sigmoid_closed_forms_golden():
    for line in open(os.path.join(GOLDEN, "sigmoid_closed_forms.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        g, want = line.split()[:2]
        got = int(oracle.sigmoid_bf16(np.array([int(g, 16)], np.uint16))[0])
        assert got == int(want, 16), (g, hex(got), want)


# --------------------------------------------------------------------------- gate

def test_gate_closed_forms():
    rng = np.random.default_rng(7)
    o = bf16_bits((torch.from_numpy(rng.standard_normal(4096)).float() * 3).to(torch.bfloat16))
    # sigmoid(0) = 1/2: out = o / 2 exactly (no underflow at these magnitudes)
    out = oracle.gate(o, np.zeros_like(o))
    half = bf16_bits((torch.from_numpy(bits_to_float(o)).float() * 0.5).to(torch.bfloat16))
    assert np.array_equal(out, half)
    # saturation: BF16 sigmoid(g) == 1 for g >= 7 -> out = o
    g7 = np.full_like(o, 0x40E0)
    assert np.array_equal(oracle.gate(o, g7), o)
    # g = -inf -> sigmoid 0 -> out = signed zero
    gm = np.full_like(o, 0xFF80)
    out = oracle.gate(o, gm)
    assert np.array_equal(out, (o & 0x8000))


def test_gate_product_matches_float32_library_product():
    # The product of two BF16 values is exact in float32 (normal range), so the
    # library float32 multiply followed by torch's RNE cast is the same result.
    rng = np.random.default_rng(8)
    o = bf16_bits(torch.from_numpy(rng.standard_normal(50_000)).float().to(torch.bfloat16))
    g = bf16_bits((torch.from_numpy(rng.standard_normal(50_000)).float() * 4).to(torch.bfloat16))
    s = oracle.sigmoid_bf16(g)
    prod = torch.from_numpy(bits_to_float(o).astype(np.float32)) * torch.from_numpy(bits_to_float(s).astype(np.float32))
    want = bf16_bits(prod.to(torch.bfloat16))
    assert np.array_equal(oracle.gate(o, g), want)


# --------------------------------------------------------------------------- attention

def _tiny(seed, lengths, hq, hkv, d, slots=None, scale=None, gate_std=2.0):
    inp = workloads.make(lengths, seed=seed, hq=hq, hkv=hkv, head_dim=d, layout="perm",
                         pool_slots=slots, gate_std=gate_std,
                         scale=scale if scale is not None else 1.0 / math.sqrt(d))
    return inp


def _brute_force(inp):
    """Pure-Python loops, math.fsum: the definition written out on tiny inputs."""
    q = bits_to_float(bf16_bits(inp["q"]))
    k = bits_to_float(bf16_bits(inp["k_pool"]))
    v = bits_to_float(bf16_bits(inp["v_pool"]))
    ip = inp["kv_indptr"].tolist()
    ix = inp["kv_indices"].tolist()
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
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
    (11, [5], 4, 2, 8), (12, [1, 7, 3], 6, 2, 16), (13, [16, 0, 9], 8, 8, 4),
    (14, [12, 3], 9, 3, 12), (15, [2, 2, 2], 16, 2, 32),
])
def test_decode_brute_force(seed, lengths, hq, hkv, d):
    inp = _tiny(seed, lengths, hq, hkv, d)
    res = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                        inp["kv_indices"], inp["scale"])
    want = _brute_force(inp)
    np.testing.assert_allclose(res.o_f64, want, rtol=1e-12, atol=1e-14)
    # the rounding stages follow from O by the pinned rounding / gate functions
    assert np.array_equal(res.o_bf16, oracle.bf16_from_double(res.o_f64))
    assert np.array_equal(res.out, oracle.gate(res.o_bf16, bf16_bits(inp["gate"])))


def _sdpa_reference(inp):
    q = torch.from_numpy(bits_to_float(bf16_bits(inp["q"])))
    k = torch.from_numpy(bits_to_float(bf16_bits(inp["k_pool"])))
    v = torch.from_numpy(bits_to_float(bf16_bits(inp["v_pool"])))
    ip = inp["kv_indptr"].tolist()
    ix = inp["kv_indices"].long()
    B, Hq, D = q.shape
    O = torch.zeros(B, Hq, D, dtype=torch.float64)
    lse = torch.full((B, Hq), -math.inf, dtype=torch.float64)
    for b in range(B):
        rows = ix[ip[b]:ip[b + 1]]
        if rows.numel() == 0:
            continue
        kb = k[rows].transpose(0, 1)  # [Hkv, L, D]
        vb = v[rows].transpose(0, 1)
        qb = q[b][:, None, :]          # [Hq, 1, D]
        O[b] = torch.nn.functional.scaled_dot_product_attention(
            qb[None], kb[None], vb[None], scale=inp["scale"], enable_gqa=True)[0, :, 0]
        G = Hq // k.shape[1]
        scores = torch.einsum("hd,hld->hl", q[b], kb.repeat_interleave(G, dim=0)) * inp["scale"]
        lse[b] = torch.logsumexp(scores, dim=-1)
    return O.numpy(), lse.numpy()


@pytest.mark.parametrize("seed,lengths,hq,hkv,d", [
    (21, [37, 64, 1, 0, 129], 16, 2, 256), (22, [50, 17], 6, 2, 64), (23, [33], 12, 4, 32),
    (24, [100, 3, 77], 16, 16, 16),
])
def test_decode_against_library_sdpa(seed, lengths, hq, hkv, d):
    inp = _tiny(seed, lengths, hq, hkv, d)
    res = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                        inp["kv_indices"], inp["scale"])
    O, lse = _sdpa_reference(inp)
    np.testing.assert_allclose(res.o_f64, O, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(res.lse, lse, rtol=1e-12, atol=1e-12)


def test_decode_closed_form_mean_of_v():
    inp = _tiny(31, [40, 7], 16, 2, 256)
    # q = 0: every score is 0, the softmax is uniform, O is the mean of the rows
    inp["q"] = torch.zeros_like(inp["q"])
    res = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                        inp["kv_indices"], inp["scale"])
    v = bits_to_float(bf16_bits(inp["v_pool"]))
    ip, ix = inp["kv_indptr"].tolist(), inp["kv_indices"].numpy()
    for b in range(2):
        rows = ix[ip[b]:ip[b + 1]]
        for h in range(16):
            np.testing.assert_allclose(res.o_f64[b, h], v[rows, h // 8].mean(axis=0), rtol=1e-13, atol=1e-15)
    # equal keys: same uniform softmax with a nonzero q
    inp2 = _tiny(32, [25], 16, 2, 256)
    rows = inp2["kv_indices"].long()
    inp2["k_pool"][rows] = inp2["k_pool"][rows[0]].clone()
    res2 = oracle.decode(inp2["q"], inp2["gate"], inp2["k_pool"], inp2["v_pool"], inp2["kv_indptr"],
                         inp2["kv_indices"], inp2["scale"])
    v2 = bits_to_float(bf16_bits(inp2["v_pool"]))
    for h in range(16):
        np.testing.assert_allclose(res2.o_f64[0, h], v2[rows.numpy(), h // 8].mean(axis=0), rtol=1e-13, atol=1e-15)


def test_decode_single_key_is_exact():
    inp = _tiny(33, [1, 1, 1], 16, 2, 256)
    res = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                        inp["kv_indices"], inp["scale"])
    vb = bf16_bits(inp["v_pool"])
    for b in range(3):
        slot = int(inp["kv_indices"][b])
        for h in range(16):
            assert np.array_equal(res.o_bf16[b, h], vb[slot, h // 8])
            assert np.array_equal(res.o_f64[b, h], bits_to_float(vb[slot, h // 8]))


def test_decode_zero_length_rows():
    inp = _tiny(34, [0, 5, 0], 16, 2, 256)
    res = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                        inp["kv_indices"], inp["scale"])
    for b in (0, 2):
        assert np.all(res.o_f64[b] == 0.0)
        assert np.all(res.out[b] == 0)          # +0, not -0
        assert np.all(np.isneginf(res.lse[b]))
    assert np.count_nonzero(res.out[1]) > 0.9 * res.out[1].size


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 16, 128])
def test_split_merge_invariance(splits):
    inp = _tiny(41, [300, 1, 0, 129, 64], 16, 2, 256)
    direct = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                           inp["kv_indices"], inp["scale"])
    split = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                          inp["kv_indices"], inp["scale"], num_splits=splits)
    np.testing.assert_allclose(split.o_f64, direct.o_f64, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(split.lse, direct.lse, rtol=1e-13, atol=1e-13)


def test_placement_invariance():
    inp = _tiny(42, [80, 33], 16, 2, 256, slots=200)
    res = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                        inp["kv_indices"], inp["scale"])
    perm = torch.randperm(200, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(200)
    k2, v2 = inp["k_pool"][perm], inp["v_pool"][perm]        # new row r holds old row perm[r]
    idx2 = inv[inp["kv_indices"].long()].to(torch.int32)
    res2 = oracle.decode(inp["q"], inp["gate"], k2, v2, inp["kv_indptr"], idx2, inp["scale"])
    assert np.array_equal(res.o_f64, res2.o_f64)
    assert np.array_equal(res.out, res2.out)


def test_pairs_subset_matches_full():
    inp = _tiny(43, [70, 20, 9], 16, 2, 256)
    full = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                         inp["kv_indices"], inp["scale"])
    pairs = np.array([[2, 15], [0, 3], [1, 8]])
    sub = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                        inp["kv_indices"], inp["scale"], pairs=pairs)
    for b, h in pairs:
        assert np.array_equal(sub.out[b, h], full.out[b, h])
        assert np.array_equal(sub.o_f64[b, h], full.o_f64[b, h])


def test_rejects_out_of_range_index():
    inp = _tiny(44, [4], 16, 2, 256, slots=10)
    bad = inp["kv_indices"].clone()
    bad[2] = 10
    with pytest.raises(ValueError):
        oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"], bad, inp["scale"])


# --------------------------------------------------------------------------- sensitivity

def test_pins_reject_planted_mistakes():
    """Mistakes planted in the oracle's evaluation (on the CPU) fail the pins."""
    inp = _tiny(51, [40, 13], 16, 2, 64)
    O_ref, _ = _sdpa_reference(inp)
    args = (inp["k_pool"], inp["v_pool"], inp["kv_indptr"], inp["kv_indices"])
    # 1. dropped scale
    bad = oracle.decode(inp["q"], inp["gate"], *args, 1.0)
    assert not np.allclose(bad.o_f64, O_ref, rtol=1e-6)
    # 2. wrong GQA mapping (h % Hkv instead of h // G): permute the query heads
    G = 8
    perm = [(h % 2) * G + h // 2 for h in range(16)]
    q_wrong = inp["q"][:, perm]
    bad = oracle.decode(q_wrong, inp["gate"], *args, inp["scale"])
    assert not np.allclose(bad.o_f64[:, perm], O_ref, rtol=1e-6)
    # 3. flipped gate sign: sigmoid(-g) instead of sigmoid(g)
    codes = np.arange(0x3F00, 0x4100, dtype=np.uint16)  # gates in [0.5, 8)
    flipped = oracle.sigmoid_bf16(codes ^ 0x8000)
    right = oracle.sigmoid_bf16(codes)
    assert np.count_nonzero(flipped != right) > 400
    # 4. double rounding through float32 differs from direct rounding
    x = 1 + 2.0**-8 + 2.0**-30
    via_f32 = int(bf16_bits(torch.tensor([x], dtype=torch.float64).float().to(torch.bfloat16))[0])
    assert via_f32 != int(oracle.bf16_from_double([x])[0])


# --------------------------------------------------------------------------- window and sinks

def _ref_args(inp):
    return (inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"], inp["kv_indices"],
            inp["scale"])


def _window_truncated(inp, W):
    """The same batch with each sequence cut to its last W positions (CSR rebuilt)."""
    ip = inp["kv_indptr"].tolist()
    ix = inp["kv_indices"]
    parts, new = [], [0]
    for b in range(len(ip) - 1):
        L = ip[b + 1] - ip[b]
        first = max(0, L - W)
        parts.append(ix[ip[b] + first:ip[b + 1]])
        new.append(new[-1] + (L - first))
    out = dict(inp)
    out["kv_indices"] = torch.cat(parts) if parts else ix[:0]
    out["kv_indptr"] = torch.tensor(new, dtype=torch.int32)
    return out


@pytest.mark.parametrize("W", [1, 3, 16, 100])
def test_window_equals_full_attention_on_the_last_rows(W):
    inp = _tiny(61, [40, 7, 0, 130, 16], 16, 2, 64)
    res = oracle.decode(*_ref_args(inp), window=W)
    trunc = _window_truncated(inp, W)
    O_ref, lse_ref = _sdpa_reference(trunc)       # library SDPA on the kept rows
    np.testing.assert_allclose(res.o_f64, O_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(res.lse, lse_ref, rtol=1e-12, atol=1e-12)
    bf = _brute_force(trunc)                        # brute force on the kept rows
    np.testing.assert_allclose(res.o_f64, bf, rtol=1e-12, atol=1e-14)


def test_window_special_cases():
    inp = _tiny(62, [40, 7, 1], 16, 2, 64)
    full = oracle.decode(*_ref_args(inp))
    wide = oracle.decode(*_ref_args(inp), window=10_000)      # W >= L: unchanged
    assert np.array_equal(full.out, wide.out) and np.array_equal(full.o_f64, wide.o_f64)
    one = oracle.decode(*_ref_args(inp), window=1)            # W = 1: the last row exactly
    v = bits_to_float(bf16_bits(inp["v_pool"]))
    ip, ix = inp["kv_indptr"].tolist(), inp["kv_indices"].tolist()
    for b in range(3):
        last = ix[ip[b + 1] - 1]
        for h in range(16):
            assert np.array_equal(one.o_f64[b, h], v[last, h // 8])
    split = oracle.decode(*_ref_args(inp), window=5, num_splits=3)
    direct = oracle.decode(*_ref_args(inp), window=5)
    np.testing.assert_allclose(split.o_f64, direct.o_f64, rtol=1e-12, atol=1e-14)


def _sdpa_with_sink_key(inp, sinks):
    """Sinks restated as one extra key per (b, h) whose score is the sink and whose
    value row is zero, through the library SDPA in float64."""
    q = torch.from_numpy(bits_to_float(bf16_bits(inp["q"])))
    k = torch.from_numpy(bits_to_float(bf16_bits(inp["k_pool"])))
    v = torch.from_numpy(bits_to_float(bf16_bits(inp["v_pool"])))
    ip = inp["kv_indptr"].tolist()
    ix = inp["kv_indices"].long()
    B, Hq, D = q.shape
    G = Hq // k.shape[1]
    sc = inp["scale"]
    O = torch.zeros(B, Hq, D, dtype=torch.float64)
    lse = torch.zeros(B, Hq, dtype=torch.float64)
    for b in range(B):
        rows = ix[ip[b]:ip[b + 1]]
        for h in range(Hq):
            qh = q[b, h]
            ksink = qh * (sinks[h] / (sc * float(qh @ qh)))        # sc * q . ksink == sink
            kb = torch.cat([k[rows, h // G], ksink[None]])
            vb = torch.cat([v[rows, h // G], torch.zeros(1, D, dtype=torch.float64)])
            O[b, h] = torch.nn.functional.scaled_dot_product_attention(
                qh[None, None, None], kb[None, None], vb[None, None], scale=sc)[0, 0, 0]
            lse[b, h] = torch.logsumexp(kb @ qh * sc, dim=0)
    return O.numpy(), lse.numpy()


def test_sinks_as_an_extra_zero_value_key():
    inp = _tiny(63, [40, 7, 0, 90], 16, 2, 64)
    sinks = np.linspace(-3.0, 4.0, 16)
    res = oracle.decode(*_ref_args(inp), sinks=sinks)
    O_ref, lse_ref = _sdpa_with_sink_key(inp, sinks)
    np.testing.assert_allclose(res.o_f64, O_ref, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(res.lse, lse_ref, rtol=1e-12, atol=1e-12)
    # with a window as well: the sink joins the windowed softmax
    resw = oracle.decode(*_ref_args(inp), sinks=sinks, window=9)
    O_w, lse_w = _sdpa_with_sink_key(_window_truncated(inp, 9), sinks)
    np.testing.assert_allclose(resw.o_f64, O_w, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(resw.lse, lse_w, rtol=1e-12, atol=1e-12)


def test_sinks_closed_forms():
    inp = _tiny(64, [30, 5], 16, 2, 64)
    inp["q"] = torch.zeros_like(inp["q"])                  # every score 0
    sinks = np.linspace(-2.0, 2.0, 16)
    res = oracle.decode(*_ref_args(inp), sinks=sinks)
    v = bits_to_float(bf16_bits(inp["v_pool"]))
    ip, ix = inp["kv_indptr"].tolist(), inp["kv_indices"].numpy()
    for b in range(2):
        rows = ix[ip[b]:ip[b + 1]]
        L = len(rows)
        for h in range(16):
            want = v[rows, h // 8].sum(axis=0) / (L + math.exp(sinks[h]))   # sum V / (L + e^sink)
            np.testing.assert_allclose(res.o_f64[b, h], want, rtol=1e-13, atol=1e-15)
            assert abs(res.lse[b, h] - math.log(L + math.exp(sinks[h]))) < 1e-12
    none = oracle.decode(*_ref_args(inp))
    minus_inf = oracle.decode(*_ref_args(inp), sinks=np.full(16, -np.inf))
    assert np.array_equal(none.o_f64, minus_inf.o_f64) and np.array_equal(none.out, minus_inf.out)
    empty = _tiny(65, [0, 3], 16, 2, 64)
    r = oracle.decode(*_ref_args(empty), sinks=sinks)
    assert np.all(r.o_f64[0] == 0.0) and np.allclose(r.lse[0], sinks)  # L = 0: O = 0, lse = sink
