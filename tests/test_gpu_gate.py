"""The gate epilogue on the GPU, bit-exact against the FP64 oracle.

FreeToken PR #781 "Fuse the BF16 attention output sigmoid gate into the existing
Triton decode stage2" (Summary, Correctness): out = RNE_bf16(o * RNE_bf16(sigmoid(g)))
must equal the unfused sigmoid-then-multiply element by element, so the gate
stage has exactly one correct result per (o, gate) pair.  The sigmoid depends on
the gate code alone, so testing all 65 536 gate codes proves it completely.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def bits_tensor(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(a.astype(np.uint16).view(np.int16)).view(torch.bfloat16)


def tensor_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_bit_exact(got: np.ndarray, want: np.ndarray):
    nan_g = (got & 0x7FFF) > 0x7F80
    nan_w = (want & 0x7FFF) > 0x7F80
    assert np.array_equal(nan_g, nan_w), np.flatnonzero(nan_g != nan_w)[:10]
    bad = np.flatnonzero((got != want) & ~nan_w)
    assert bad.size == 0, [(int(i), hex(int(got[i])), hex(int(want[i]))) for i in bad[:10]]


def run_gate(gda, o: np.ndarray, g: np.ndarray) -> np.ndarray:
    out = gda.gate(bits_tensor(o).cuda(), bits_tensor(g).cuda())
    torch.cuda.synchronize()
    return tensor_bits(out)


O_SPECIAL = [0x3F80, 0xBF80, 0x0000, 0x8000, 0x4060, 0x0001, 0x8003, 0x007F, 0x0080, 0x7F7F, 0xFF7F,
             0x7F80, 0xFF80, 0x7FC0, 0x3C00, 0x4300, 0x3F81, 0x1234, 0x00FF, 0x0100]


def test_gate_all_gate_codes(gda):
    codes = np.arange(65536, dtype=np.uint16)
    rng = np.random.default_rng(0)
    o_vals = O_SPECIAL + [int(x) for x in rng.integers(0, 65536, 12)]
    o = np.repeat(np.array(o_vals, np.uint16), 65536)
    g = np.tile(codes, len(o_vals))
    assert_bit_exact(run_gate(gda, o, g), oracle.gate(o, g))


def test_gate_all_o_codes(gda):
    codes = np.arange(65536, dtype=np.uint16)
    g_vals = [0x0000, 0x8000, 0x3F80, 0xBF80, 0x40E0, 0xC0E0, 0x42C8, 0xC2C8, 0x7F80, 0xFF80, 0x7FC0,
              0x3E00, 0xBE00, 0x4120, 0xC120, 0xC1A0, 0xC2A0, 0xC2B0]
    o = np.tile(codes, len(g_vals))
    g = np.repeat(np.array(g_vals, np.uint16), 65536)
    assert_bit_exact(run_gate(gda, o, g), oracle.gate(o, g))


def test_gate_random_pairs_and_ragged_tail(gda):
    rng = np.random.default_rng(1)
    for n in (1, 7, 8, 9, 1000003):
        o = rng.integers(0, 65536, n).astype(np.uint16)
        g = rng.integers(0, 65536, n).astype(np.uint16)
        assert_bit_exact(run_gate(gda, o, g), oracle.gate(o, g))


def test_gate_subnormal_products(gda):
    # products below the float normal range are rounded once, from the exact value
    o_codes = np.concatenate([np.arange(0x0001, 0x0400), np.arange(0x8001, 0x8400)]).astype(np.uint16)
    g_codes = np.arange(0xC000, 0xC2C0, 3, dtype=np.uint16)  # gates in [-2, -96): small sigmoids
    o = np.repeat(o_codes, g_codes.size)
    g = np.tile(g_codes, o_codes.size)
    assert_bit_exact(run_gate(gda, o, g), oracle.gate(o, g))


def test_gate_does_not_modify_inputs_and_allows_in_place(gda):
    rng = np.random.default_rng(2)
    o = bits_tensor(rng.integers(0, 0x7F00, 4096).astype(np.uint16)).cuda()
    g = bits_tensor(rng.integers(0, 65536, 4096).astype(np.uint16)).cuda()
    o0, g0 = o.clone(), g.clone()
    out = gda.gate(o, g)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o0.view(torch.int16))
    assert torch.equal(g.view(torch.int16), g0.view(torch.int16))
    gda.gate(o, g, out=o)   # out may alias o
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), out.view(torch.int16))
