"""Decode-kernel variants on the GPU against the FP64 oracle: sliding window,
attention sinks, any GQA group size (FreeToken PR #781, Automatic dispatch and
Correctness: window, sinks, custom scale and non-power-of-two GQA groups are the
cases of the general path).  Same tolerance as the main parity tests."""
import numpy as np
import pytest
import torch

import oracle
from gated_gqa_attention_gb300 import workloads

pytestmark = pytest.mark.gpu

ATOL, RTOL = 4e-3, 1.6e-2
LENS = [0, 1, 5, 63, 64, 65, 200, 1000, 16, 129, 4096]


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_close(got, want):
    g = oracle.double_from_bf16(got)
    w = oracle.double_from_bf16(want)
    bad = np.abs(g - w) > ATOL + RTOL * np.abs(w)
    assert not bad.any(), "%d / %d out of tolerance, worst %.3g" % (bad.sum(), bad.size, np.abs(g - w).max())


def run(gda, inp, **kw):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    sinks = kw.pop("sinks", None)
    lse = kw.pop("lse", None)
    out = gda.decode_ex(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"],
                        scale=d["scale"], sinks=None if sinks is None else torch.as_tensor(
                            sinks, dtype=torch.float32).cuda(), lse=lse, **kw)
    torch.cuda.synchronize()
    return bits(out)


def reference(inp, **kw):
    return oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                         inp["kv_indices"], inp["scale"], **kw)


@pytest.fixture(scope="module")
def batch():
    return workloads.make(LENS, seed=201, layout="perm", pool_slots=8000)


@pytest.mark.parametrize("variant", [1, 2, 3])
@pytest.mark.parametrize("window", [1, 7, 64, 300, 100_000])
def test_sliding_window(gda, batch, variant, window):
    ref = reference(batch, window=window)
    for splits in (0, 3):
        check_close(run(gda, batch, window=window, num_splits=splits, variant=variant), ref.out)


@pytest.mark.parametrize("variant", [1, 2, 3])
def test_attention_sinks(gda, batch, variant):
    rng = np.random.default_rng(5)
    sinks = rng.normal(0.0, 3.0, 16).astype(np.float32)
    sinks[3] = -np.inf                     # a head without a sink
    sinks[7] = 40.0                        # a sink that dominates the softmax
    ref = reference(batch, sinks=sinks.astype(np.float64))
    for splits in (0, 5):
        check_close(run(gda, batch, sinks=sinks, num_splits=splits, variant=variant), ref.out)


def test_sinks_lse_and_empty_rows(gda, batch):
    sinks = np.linspace(-2, 2, 16).astype(np.float32)
    ref = reference(batch, sinks=sinks.astype(np.float64))
    lse = torch.empty(len(LENS), 16, dtype=torch.float32, device="cuda")
    got = run(gda, batch, sinks=sinks, lse=lse)
    check_close(got, ref.out)
    np.testing.assert_allclose(lse.cpu().numpy(), ref.lse, atol=2e-3, rtol=1e-4)   # L = 0 rows: lse = sink
    assert np.all(got[0] == 0)


@pytest.mark.parametrize("hq,hkv", [(16, 16), (16, 8), (6, 2), (16, 4), (12, 2), (14, 2), (32, 2), (20, 2), (15, 1),
                                     (48, 2), (24, 1), (40, 2), (64, 2), (56, 1)])
@pytest.mark.parametrize("variant", [1, 2, 3])
def test_gqa_group_sizes(gda, hq, hkv, variant):
    inp = workloads.make([1, 37, 300, 0, 129], seed=300 + hq + hkv, hq=hq, hkv=hkv, layout="perm", pool_slots=1000)
    ref = reference(inp)
    for splits in (0, 4):
        check_close(run(gda, inp, num_splits=splits, variant=variant), ref.out)


def test_everything_together(gda):
    inp = workloads.make([700, 1, 0, 2500, 90], seed=401, hq=12, hkv=2, layout="pages", page=16,
                         pool_slots=4000, scale=0.09, peaky_frac=0.02)
    sinks = np.linspace(-1, 3, 12).astype(np.float32)
    ref = reference(inp, window=333, sinks=sinks.astype(np.float64))
    lse = torch.empty(5, 12, dtype=torch.float32, device="cuda")
    got = run(gda, inp, window=333, sinks=sinks, lse=lse)
    check_close(got, ref.out)
    np.testing.assert_allclose(lse.cpu().numpy(), ref.lse, atol=2e-3, rtol=1e-4)


def test_window_on_the_ragged_workload(gda):
    inp = workloads.make_workload("b224_ragged")
    pairs = np.array([(b, h) for b in range(0, 224, 7) for h in (0, 5, 8, 15)])
    ref = reference(inp, window=1024, pairs=pairs)
    got = run(gda, inp, window=1024)
    idx = tuple(pairs.T)
    check_close(got[idx], ref.out[idx])


# G > 8 on the MMA kernel: the groups of 8 query heads go in teams (pairs for 2 or 4
# groups on 8 warps, threes otherwise on 6 warps); one piece per (sequence, KV head,
# team) serves every group of the team, a share of the CTA's warps each, and stage 2
# reads the partial of (piece, group of the team) at piece * team + group.  G = 20 and
# G = 24 are one three; G = 40 (5 groups) and G = 56 (7 groups) leave the last three
# with empty groups; G = 32 is two pairs.  Long ragged batches make pieces cross
# sequences and CTAs; a window, sinks, the LSE and explicit splits go through the same
# mapping.  The TMA variant (3) runs the same case per virtual head.
@pytest.mark.parametrize("hq,hkv", [(32, 2), (20, 2), (16, 1), (30, 3), (40, 2), (48, 2), (24, 1), (64, 2),
                                    (80, 2), (56, 1)])
def test_team_groups_long_ragged(gda, hq, hkv):
    lens = [4096, 1, 0, 3000, 777, 65, 2049, 16, 5000, 129, 1500, 2]
    inp = workloads.make(lens, seed=500 + hq + hkv, hq=hq, hkv=hkv, layout="perm", pool_slots=20000,
                         peaky_frac=0.01)
    ref = reference(inp)
    for kw in ({}, {"min_chunk": 16}, {"num_splits": 7}, {"variant": 3}):
        check_close(run(gda, inp, **kw), ref.out)
    sinks = np.linspace(-2.0, 2.0, hq).astype(np.float32)
    ref = reference(inp, window=1000, sinks=sinks.astype(np.float64))
    lse = torch.empty(len(lens), hq, dtype=torch.float32, device="cuda")
    check_close(run(gda, inp, window=1000, sinks=sinks, lse=lse), ref.out)
    np.testing.assert_allclose(lse.cpu().numpy(), ref.lse, atol=2e-3, rtol=1e-4)


@pytest.mark.parametrize("hq", [32, 48])
def test_team_groups_workload_sample(gda, hq):
    # b64_l4096's lengths with Hq = 32 or 48, Hkv = 2 (G = 16: one pair; G = 24: one
    # three), sampled (sequence, head) pairs
    inp = workloads.make([4096] * 64, seed=77, hq=hq, hkv=2, layout="perm", pool_slots=64 * 4096 + 1000)
    heads = sorted({0, 7, 8, 15, 16, hq // 2 - 1, hq // 2, hq - 9, hq - 8, hq - 1})
    pairs = np.array([(b, h) for b in range(0, 64, 9) for h in heads])
    ref = reference(inp, pairs=pairs)
    got = run(gda, inp)
    idx = tuple(pairs.T)
    check_close(got[idx], ref.out[idx])


@pytest.mark.parametrize("hq", [32, 48])
def test_team_groups_deterministic_and_placement_invariant(gda, hq):
    # the team kernel merges the warps of a group in a fixed order: repeated calls and
    # a permuted pool (same rows at other slots) give the same bits
    inp = workloads.make([4096, 700, 1, 2500], seed=611, hq=hq, hkv=2, layout="perm", pool_slots=9000)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    n = inp["k_pool"].shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n)
    moved = dict(inp)
    moved["k_pool"] = inp["k_pool"][perm]
    moved["v_pool"] = inp["v_pool"][perm]
    moved["kv_indices"] = inv[inp["kv_indices"].long()].to(torch.int32)
    for kw in ({}, {"num_splits": 5}):
        a, b, c = run(gda, inp, **kw), run(gda, inp, **kw), run(gda, moved, **kw)
        assert np.array_equal(a, b) and np.array_equal(a, c)


@pytest.mark.parametrize("hq", [32, 48])
def test_team_groups_check_indices(gda, hq):
    inp = workloads.make([300, 200], seed=612, hq=hq, hkv=2, layout="perm", pool_slots=600)
    ws = torch.empty(gda.workspace_bytes(2, hq, 2, 256, 0), dtype=torch.uint8, device="cuda")
    gda.workspace_init(ws)
    run(gda, inp, workspace=ws, check_indices=True)
    assert gda.read_error(ws) == 0
    bad = inp["kv_indices"].clone()
    bad[17] = 600         # == num_slots: out of range
    bad[450] = -1
    run(gda, dict(inp, kv_indices=bad), workspace=ws, check_indices=True)
    assert gda.read_error(ws) & gda.DEVERR_INDEX


@pytest.mark.parametrize("hq", [24, 48, 80])
def test_team_groups_caller_workspace_sizes(gda, hq):
    # the caller-sized workspace (workspace_bytes) holds the team schedule's partials
    # (pairs at G = 12, threes at G = 24 and 40) in automatic and explicit-split modes,
    # with a window too
    lens = [1, 4096, 33, 2000, 0, 5000, 65]
    inp = workloads.make(lens, seed=613, hq=hq, hkv=2, layout="perm", pool_slots=12000)
    for splits, window in ((0, 0), (3, 0), (0, 700)):
        ws = torch.empty(gda.workspace_bytes(len(lens), hq, 2, 256, splits), dtype=torch.uint8, device="cuda")
        gda.workspace_init(ws)
        ref = reference(inp, window=window)
        check_close(run(gda, inp, workspace=ws, num_splits=splits, window=window), ref.out)
        assert gda.read_error(ws) == 0


@pytest.mark.parametrize("hq", [32, 48])
def test_team_groups_many_segments(gda, hq):
    # more (sequence, KV head, team) segments than CTAs: the stream schedule charges a
    # cost per segment start (the stage-1 and stage-2 views of the pieces must agree),
    # with pairs (hq 32) and threes (hq 48)
    rng = np.random.default_rng(700 + hq)
    lens = [int(x) for x in rng.integers(1, 600, 160)]
    lens[5] = 0
    lens[77] = 4000
    inp = workloads.make(lens, seed=701 + hq, hq=hq, hkv=2, layout="perm", pool_slots=sum(lens) + 500)
    ref = reference(inp)
    for kw in ({}, {"max_len": max(lens), "total_len": sum(lens)}, {"num_splits": 3}):
        check_close(run(gda, inp, **kw), ref.out)

