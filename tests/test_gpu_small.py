"""The one-kernel small-batch decode path (a thread-block cluster of 8 CTAs per
(sequence, KV head), partial states merged in distributed shared memory, the gate
in the same kernel), taken when the caller passes a host-known length bound
max_len <= 1024.  Against the FP64 oracle under the tolerance of the other decode
tests: |gpu - oracle| <= 4e-3 + 1.6e-2 |oracle|; windows, sinks, lse, empty
sequences, GQA group sizes, the ungated output, and the page's B1 / B4 workloads."""
import numpy as np
import pytest
import torch

import oracle
from canary import Guarded, check_all
from gated_gqa_attention_gb300 import workloads

pytestmark = pytest.mark.gpu

ATOL, RTOL = 4e-3, 1.6e-2
LENS = [0, 1, 65, 1000, 129, 1024]   # 12 (sequence, KV head) pairs: one wave of clusters


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_close(got, want):
    g = oracle.double_from_bf16(got)
    w = oracle.double_from_bf16(want)
    bad = np.abs(g - w) > ATOL + RTOL * np.abs(w)
    assert not bad.any(), "%d / %d out of tolerance, worst %.3g" % (bad.sum(), bad.size, np.abs(g - w).max())


def to_cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run(gda, inp, max_len, workspace=None, **kw):
    d = to_cuda(inp)
    sinks = kw.pop("sinks", None)
    out = gda.decode_ex(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"],
                        scale=d["scale"], max_len=max_len, workspace=workspace,
                        sinks=None if sinks is None else torch.as_tensor(sinks, dtype=torch.float32).cuda(), **kw)
    torch.cuda.synchronize()
    return bits(out)


def reference(inp, **kw):
    return oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                         inp["kv_indices"], inp["scale"], **kw)


def test_one_wave_holds_the_test_batches(gda):
    # the test batches take the 8-CTA clusters (one wave, <= 128 positions per CTA)
    assert gda.small_path_cluster(2 * len(LENS), 1024) == 8
    assert gda.small_path_cluster(2 * len(LENS), 1025) == 0       # beyond the length bound
    assert gda.small_path_cluster(10_000, 128) == 0               # beyond one wave


@pytest.fixture(scope="module")
def batch():
    inp = workloads.make(LENS, seed=211, layout="perm", pool_slots=8000)
    return inp, reference(inp)


def test_cluster_path_is_taken_and_matches(gda, batch):
    # the cluster path writes no partials: a sentinel-filled workspace stays untouched
    # past its header, while the split path (no bound) fills it
    inp, ref = batch
    B, Hq, D = inp["q"].shape
    Hkv = inp["k_pool"].shape[1]
    nbytes = gda.workspace_bytes(B, Hq, Hkv, D, 0)
    ws = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    gda.workspace_init(ws)
    got = run(gda, inp, max(LENS), workspace=ws)
    check_close(got, ref.out)
    assert bool((ws[256:] == 0xA5).all()), "partials were written: the split path ran"
    got2 = run(gda, inp, 0, workspace=ws)
    check_close(got2, ref.out)
    assert not bool((ws[256:] == 0xA5).all())


def test_bound_below_the_lengths_is_still_correct(gda, batch):
    inp, ref = batch
    check_close(run(gda, inp, 5), ref.out)


def test_deterministic(gda, batch):
    inp, _ = batch
    assert np.array_equal(run(gda, inp, 1024), run(gda, inp, 1024))


@pytest.mark.parametrize("window", [1, 7, 64, 300, 100_000])
def test_window(gda, batch, window):
    inp, _ = batch
    check_close(run(gda, inp, 1024, window=window), reference(inp, window=window).out)


def test_sinks_lse_and_empty_rows(gda, batch):
    inp, _ = batch
    rng = np.random.default_rng(7)
    sinks = rng.normal(0.0, 3.0, 16).astype(np.float32)
    sinks[3] = -np.inf                     # a head without a sink
    sinks[7] = 40.0                        # a sink that dominates the softmax
    ref = reference(inp, sinks=sinks.astype(np.float64))
    # out and lse inside 0xFF guard bands (canary.Guarded)
    out, lse = Guarded((len(LENS), 16, 256), torch.bfloat16), Guarded((len(LENS), 16), torch.float32)
    got = run(gda, inp, 1024, sinks=sinks, lse=lse.t, out=out.t)
    check_all(out=out, lse=lse)
    check_close(got, ref.out)
    np.testing.assert_allclose(lse.t.cpu().numpy(), ref.lse, atol=2e-3, rtol=1e-4)
    assert np.all(got[0] == 0)             # L = 0: O = 0 whatever the sink


def test_lse_without_sinks(gda, batch):
    inp, ref = batch
    lse = torch.empty(len(LENS), 16, dtype=torch.float32, device="cuda")
    check_close(run(gda, inp, 1024, lse=lse), ref.out)
    got = lse.cpu().numpy()
    assert np.all(np.isneginf(got[0])) and np.all(np.isneginf(ref.lse[0]))
    np.testing.assert_allclose(got[1:], ref.lse[1:], atol=2e-3, rtol=1e-4)


def test_ungated_output(gda, batch):
    inp, ref = batch
    check_close(run(gda, inp, 1024, fuse_gate=False), ref.o_bf16)


# group sizes the path takes (G <= 8; B * Hkv <= 12 pairs for B = 3)
@pytest.mark.parametrize("hq,hkv", [(6, 2), (16, 4), (12, 2), (14, 2), (4, 4), (2, 1), (8, 1)])
def test_gqa_group_sizes(gda, hq, hkv):
    inp = workloads.make([37, 300, 0], seed=500 + hq + hkv, hq=hq, hkv=hkv, layout="perm", pool_slots=1000)
    check_close(run(gda, inp, 300), reference(inp).out)


@pytest.mark.parametrize("key", ["b1_l512", "b4_ragged"])
def test_page_workloads(gda, key):
    inp = workloads.make_workload(key)
    B = inp["q"].shape[0]
    out, lse = Guarded((B, 16, 256), torch.bfloat16), Guarded((B, 16), torch.float32)
    got = run(gda, inp, int(max(inp["lengths"])), out=out.t, lse=lse.t)
    check_all(out=out, lse=lse)
    check_close(got, reference(inp).out)


def test_step_host_takes_the_cluster_path(gda):
    # gda_decode_step_host reads the longest length from kv_indptr on the host: B4
    # ragged runs as one kernel, and its result equals decode_ex with that bound bit
    # for bit
    inp = workloads.make_workload("b4_ragged")
    d = to_cuda(inp)
    B, Hq, D = inp["q"].shape
    nnz = inp["kv_indices"].numel()
    _, total = gda.step_layout(B, Hq, D, nnz)
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    gda.pack_step(host_in, inp["q"], inp["gate"], inp["kv_indptr"], inp["kv_indices"])
    host_out = torch.empty(B, Hq, D, dtype=torch.bfloat16).pin_memory()
    gda.decode_step_host(host_in, None, d["k_pool"], d["v_pool"], None, host_out, B, Hq, nnz, scale=inp["scale"],
                         map_in=True, map_out=True)
    want = run(gda, inp, int(max(inp["lengths"])))
    assert np.array_equal(bits(host_out), want)
    check_close(bits(host_out), reference(inp).out)


@pytest.mark.parametrize("B,lmax,C", [(16, 512, 4), (32, 256, 2), (48, 128, 1)])
def test_smaller_clusters(gda, B, lmax, C):
    # more pairs than 8-CTA clusters fit at once: 4-, 2- and 1-CTA clusters (each CTA at
    # most 128 positions), same parity and no partials written
    rng = np.random.default_rng(B)
    lens = [int(x) for x in rng.integers(0, lmax + 1, B)]
    lens[0], lens[1] = lmax, 0
    inp = workloads.make(lens, seed=600 + B, layout="perm", pool_slots=sum(lens) + 100)
    Hkv = inp["k_pool"].shape[1]
    assert gda.small_path_cluster(B * Hkv, lmax) == C
    _, Hq, D = inp["q"].shape
    ws = torch.full((gda.workspace_bytes(B, Hq, Hkv, D, 0),), 0xA5, dtype=torch.uint8, device="cuda")
    gda.workspace_init(ws)
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    got = run(gda, inp, lmax, workspace=ws, lse=lse)
    assert bool((ws[256:] == 0xA5).all()), "partials were written: the split path ran"
    ref = reference(inp)
    check_close(got, ref.out)
    np.testing.assert_allclose(lse.cpu().numpy(), ref.lse, atol=2e-3, rtol=1e-4)


def _check_fp8(got, want, v_scale):
    # the FP8 tests' tolerance: the absolute term grows with the V scale
    g = oracle.double_from_bf16(got)
    w = oracle.double_from_bf16(want)
    bad = np.abs(g - w) > ATOL * max(1.0, v_scale) + RTOL * np.abs(w)
    assert not bad.any(), "%d / %d out of tolerance, worst %.3g" % (bad.sum(), bad.size, np.abs(g - w).max())


@pytest.mark.parametrize("key", ["b1_l512", "b4_ragged"])
def test_e4m3_pools(gda, key):
    # an FP8 (e4m3) cache through the one-kernel path: K and V widened to FP16 while
    # staged, Q to FP16 with one power-of-two factor, the descales folded in
    inp = workloads.make_workload(key, kv="e4m3")
    ml = int(max(inp["lengths"]))
    d = to_cuda(inp)
    B, Hq, D = inp["q"].shape
    Hkv = inp["k_pool"].shape[1]
    assert gda.small_path_cluster(B * Hkv, ml) > 0
    ws = torch.full((gda.workspace_bytes(B, Hq, Hkv, D, 0),), 0xA5, dtype=torch.uint8, device="cuda")
    gda.workspace_init(ws)
    for kd, vd in ((inp["k_descale"], inp["v_descale"]), (inp["k_descale"] * 0.5, inp["v_descale"] * 3.5)):
        out = gda.decode_ex(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"],
                            scale=inp["scale"], max_len=ml, workspace=ws, k_descale=kd, v_descale=vd)
        torch.cuda.synchronize()
        assert bool((ws[256:] == 0xA5).all()), "partials were written: the split path ran"
        ref = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                            inp["kv_indices"], inp["scale"], k_descale=kd, v_descale=vd)
        _check_fp8(bits(out), ref.out, vd / inp["v_descale"])


def test_e4m3_sinks_window_lse(gda):
    inp = workloads.make([0, 1, 65, 700, 129, 1024], seed=77, layout="perm", pool_slots=4000, kv="e4m3")
    d = to_cuda(inp)
    sinks = np.linspace(-2, 2, 16).astype(np.float32)
    lse = torch.empty(6, 16, dtype=torch.float32, device="cuda")
    out = gda.decode_ex(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"],
                        scale=inp["scale"], max_len=1024, window=300, lse=lse,
                        sinks=torch.as_tensor(sinks).cuda(), k_descale=inp["k_descale"], v_descale=inp["v_descale"])
    torch.cuda.synchronize()
    ref = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"], inp["kv_indices"],
                        inp["scale"], window=300, sinks=sinks.astype(np.float64), k_descale=inp["k_descale"],
                        v_descale=inp["v_descale"])
    _check_fp8(bits(out), ref.out, 1.0)
    np.testing.assert_allclose(lse.cpu().numpy(), ref.lse, atol=2e-3, rtol=1e-4)


def test_step_host_e4m3(gda):
    # the host-memory step over an FP8 cache: the same bits as decode_ex with the bound
    # the step reads from kv_indptr (the longest length)
    inp = workloads.make_workload("b4_ragged", kv="e4m3")
    d = to_cuda(inp)
    B, Hq, D = inp["q"].shape
    nnz = inp["kv_indices"].numel()
    _, total = gda.step_layout(B, Hq, D, nnz)
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    gda.pack_step(host_in, inp["q"], inp["gate"], inp["kv_indptr"], inp["kv_indices"])
    host_out = torch.empty(B, Hq, D, dtype=torch.bfloat16).pin_memory()
    kd, vd = inp["k_descale"], inp["v_descale"]
    gda.decode_step_host(host_in, None, d["k_pool"], d["v_pool"], None, host_out, B, Hq, nnz, scale=inp["scale"],
                         map_in=True, map_out=True, k_descale=kd, v_descale=vd)
    want = gda.decode_ex(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"],
                         scale=inp["scale"], max_len=int(max(inp["lengths"])), k_descale=kd, v_descale=vd)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host_out), bits(want))
    ref = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"], inp["kv_indices"],
                        inp["scale"], k_descale=kd, v_descale=vd)
    _check_fp8(bits(host_out), ref.out, 1.0)
