"""Prefill / extend gated SDPA on the GPU (tcgen05 kernel) against the FP64 oracle.

cuDNN FE-OSS "Gated Attention Block (SM107)", Overview stages (4)-(5) with fuse_gate:
O = softmax(Q K^T * scale + mask) V with GQA, out = RNE(RNE(O) * RNE(sigmoid(gate))).
Tolerance as in the decode tests: |err| <= 4e-3 + 1.6e-2 |ref| on the gated output
(P is rounded to BF16 before the PV product, sums in FP32)."""
import numpy as np
import pytest
import torch

import oracle
from canary import Guarded, check_all
from gated_gqa_attention_gb300 import workloads

pytestmark = pytest.mark.gpu

ATOL, RTOL = 4e-3, 1.6e-2


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_close(got, want, rows=None):
    g = oracle.double_from_bf16(got)
    w = oracle.double_from_bf16(want)
    if rows is not None:
        idx = tuple(np.asarray(rows).T)
        g, w = g[idx], w[idx]
    bad = np.abs(g - w) > ATOL + RTOL * np.abs(w)
    assert not bad.any(), "%d / %d out of tolerance, worst %.3g" % (bad.sum(), bad.size, np.abs(g - w).max())
    return float(np.abs(g - w).max()) if g.size else 0.0


def to_cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run(gda, d, gate=True, lse=None, out=None):
    out = gda.prefill(d["q"], d["gate"] if gate else None, d["k"], d["v"], kv_lens=d["kv_lens"], lse=lse,
                      out=out, scale=d["scale"], causal=d["causal"])
    torch.cuda.synchronize()
    return bits(out)


def reference(inp, rows=None):
    return oracle.prefill(inp["q"], inp["gate"], inp["k"], inp["v"], inp["scale"], causal=inp["causal"],
                          kv_lens=inp["kv_lens"], rows=rows)


CASES = [
    # B, Sq, Skv, Hq, Hkv, causal, kv_lens
    (1, 128, 128, 1, 1, True, None),            # one CTA, one diagonal
    (1, 128, 128, 1, 1, False, None),
    (1, 200, 200, 2, 1, True, None),            # ragged query and key tails
    (2, 300, 300, 4, 2, False, None),
    (1, 77, 333, 2, 2, True, None),             # extend: 77 new tokens after 256 cached
    (3, 130, 190, 4, 1, True, [190, 64, 0]),    # padded keys; an empty sequence (dead rows)
    (2, 256, 256, 32, 2, True, None),           # the page's head geometry
    (1, 64, 1000, 2, 2, False, [700]),
]


@pytest.mark.parametrize("B,Sq,Skv,Hq,Hkv,causal,kv_lens", CASES)
def test_prefill_parity(gda, B, Sq, Skv, Hq, Hkv, causal, kv_lens):
    inp = workloads.make_prefill(B, Sq, Skv, seed=500 + Sq + Skv, hq=Hq, hkv=Hkv, causal=causal, kv_lens=kv_lens)
    dev = to_cuda(inp)
    ref = reference(inp)
    # out and lse inside 0xFF guard bands (canary.Guarded)
    out, lse = Guarded.like(dev["q"]), Guarded((B, Hq, Sq), torch.float32, fill=float("nan"))
    check_close(run(gda, dev, lse=lse.t, out=out.t), ref.out)
    check_all(out=out, lse=lse)
    got_lse = lse.t.cpu().numpy()
    live = np.isfinite(ref.lse)
    np.testing.assert_allclose(got_lse[live], ref.lse[live], atol=2e-3, rtol=1e-4)
    assert np.all(np.isneginf(got_lse[~live]))
    assert gda.prefill_read_error() == 0


def test_prefill_unfused_and_deterministic(gda):
    inp = workloads.make_prefill(2, 160, 160, seed=41, hq=4, hkv=2, causal=True)
    dev = to_cuda(inp)
    ref = reference(inp)
    check_close(run(gda, dev, gate=False), ref.o_bf16)
    a = run(gda, dev)
    b = run(gda, dev)
    assert np.array_equal(a, b)
    # the fused gate equals the standalone gate applied to the unfused output, bit for bit
    o = run(gda, dev, gate=False)
    assert np.array_equal(a, oracle.gate(o, bits(inp["gate"])))


def test_prefill_scores_that_move_the_max(gda):
    """Keys that grow along the sequence force repeated rescaling of O in TMEM."""
    inp = workloads.make_prefill(1, 256, 512, seed=43, hq=2, hkv=1, causal=False)
    ramp = torch.linspace(0.2, 6.0, 512)[None, :, None, None]
    inp["k"] = (inp["k"].float() * ramp).to(torch.bfloat16)
    inp["scale"] = 0.25
    dev = to_cuda(inp)
    check_close(run(gda, dev), reference(inp).out)


@pytest.mark.parametrize("key", ["p1_s512_causal", "p1_s4096_causal", "p1_s4096_dense", "p4_extend_q1024_kv8192"])
def test_prefill_workload_sampled(gda, key):
    # one random query row from every (128-query block, head, sequence) tile -- each a
    # CTA of the kernel -- plus random rows and the corners; out and lse inside guard bands
    inp = workloads.make_prefill_workload(key)
    dev = to_cuda(inp)
    B, Sq, Hq = inp["q"].shape[:3]
    out, lse = Guarded.like(dev["q"]), Guarded((B, Hq, Sq), torch.float32)
    got = run(gda, dev, lse=lse.t, out=out.t)
    check_all(out=out, lse=lse)
    rng = np.random.default_rng(3)
    nblk = (Sq + 127) // 128
    bb, qb, hh = np.meshgrid(np.arange(B), np.arange(nblk), np.arange(Hq), indexing="ij")
    bb, qb, hh = bb.ravel(), qb.ravel(), hh.ravel()
    ii = np.minimum(qb * 128 + rng.integers(0, 128, bb.size), Sq - 1)
    per_tile = np.stack([bb, ii, hh], axis=1)
    rnd = np.stack([rng.integers(0, B, 48), rng.integers(0, Sq, 48), rng.integers(0, Hq, 48)], axis=1)
    rows = np.concatenate([per_tile, rnd, [[0, 0, 0], [B - 1, Sq - 1, Hq - 1], [0, Sq - 1, 0]]]).astype(np.int32)
    ref = reference(inp, rows=rows)
    check_close(got, ref.out, rows=rows)
    idx = (rows[:, 0], rows[:, 2], rows[:, 1])
    got_lse = lse.t.cpu().numpy()[idx]
    np.testing.assert_allclose(got_lse, ref.lse[idx], atol=2e-3, rtol=1e-4)
    assert gda.prefill_read_error() == 0


def test_prefill_gate_covers_every_bf16_code(gda):
    """O = 1 exactly (one visible key whose V row is 1.0), so out = RNE(sigmoid(g)):
    all 65 536 gate codes through the fused epilogue against the oracle's sigmoid."""
    B, Sq, Hq, D = 1, 16, 16, 256
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(B, Sq, Hq, D)
    inp = workloads.make_prefill(B, Sq, 1, seed=7, hq=Hq, hkv=1, causal=False)
    inp["gate"] = codes.view(torch.bfloat16)
    inp["v"] = torch.ones_like(inp["v"])
    dev = to_cuda(inp)
    got = run(gda, dev)
    want = oracle.sigmoid_bf16(codes.numpy().view(np.uint16))
    g, w = oracle.double_from_bf16(got), oracle.double_from_bf16(want)
    nan = np.isnan(w)
    assert np.array_equal(np.isnan(g), nan)
    assert np.array_equal(got[~nan], want[~nan])


_FIRST_USE = r'''
import numpy as np, torch
import gated_gqa_attention_gb300 as gda
torch.manual_seed(0)
q = torch.randn(1, 256, 8, 256, device="cuda").to(torch.bfloat16)
gate = (2 * torch.randn(1, 256, 8, 256, device="cuda")).to(torch.bfloat16)
k = torch.randn(1, 256, 2, 256, device="cuda").to(torch.bfloat16)
v = torch.randn(1, 256, 2, 256, device="cuda").to(torch.bfloat16)
torch.cuda.synchronize()
a, b = torch.cuda.Stream(), torch.cuda.Stream()
outs = []
for s in (a, b):      # the first two calls of the process, back to back on two streams
    with torch.cuda.stream(s):
        outs.append(gda.prefill(q, gate, k, v, scale=0.0625, causal=True))
torch.cuda.synchronize()
again = gda.prefill(q, gate, k, v, scale=0.0625, causal=True)
g = torch.cuda.CUDAGraph()
side = torch.cuda.Stream()
side.wait_stream(torch.cuda.current_stream())
with torch.cuda.stream(side):
    with torch.cuda.graph(g):
        captured = gda.prefill(q, gate, k, v, scale=0.0625, causal=True)
g.replay()
torch.cuda.synchronize()
for o in outs + [captured]:
    assert torch.equal(o.view(torch.int16), again.view(torch.int16))
assert gda.prefill_read_error() == 0
print("first-use ok")
'''


def test_first_use_on_two_streams_and_capture():
    # The per-device sigmoid table is built and waited for on first use, so a second
    # stream's first call cannot read it early; capture after first use replays the
    # same bits.  A fresh process, so this really is the library's first prefill.
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_USE], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "first-use ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
