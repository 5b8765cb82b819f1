"""Gated decode attention on the GPU against the FP64 oracle, through the C ABI.

Tolerance (per element of the BF16 output): |gpu - oracle| <= 4e-3 + 1.6e-2 |oracle|,
the allclose form of "within 2 BF16 ulp of the output"; the gate stage is
bit-exact for identical O (test_fused_equals_unfused_bitwise).  Small cases span
several 64-token tiles, ragged tails, empty and single-key sequences; the five
named workloads run at full size with every (sequence, head) checked.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from canary import Guarded, check_all
from gated_gqa_attention_gb300 import workloads

pytestmark = pytest.mark.gpu

ATOL, RTOL = 4e-3, 1.6e-2


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run(gda, dev, **kw):
    return gda.decode_ex(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"],
                         dev["kv_indices"], scale=dev["scale"], **kw)


def reference(inp, pairs=None):
    return oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                         inp["kv_indices"], inp["scale"], pairs=pairs)


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    # BF16 codes on one ordered integer line (sign-magnitude: +0 and -0 coincide)
    def ordered(x):
        x = np.asarray(x).astype(np.int64) & 0xFFFF
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def check_close(got_bits: np.ndarray, want_bits: np.ndarray, pairs=None):
    g = oracle.double_from_bf16(got_bits)
    w = oracle.double_from_bf16(want_bits)
    gb, wb = np.asarray(got_bits), np.asarray(want_bits)
    if pairs is not None:
        idx = tuple(np.asarray(pairs).T)
        g, w, gb, wb = g[idx], w[idx], gb[idx], wb[idx]
    err = np.abs(g - w)
    lim = ATOL + RTOL * np.abs(w)
    bad = err > lim
    assert not bad.any(), "%d / %d elements out of tolerance; worst err %.3g at ref %.3g" % (
        bad.sum(), bad.size, err.max(), w.flat[np.argmax(err - lim)])
    rms = math.sqrt(float(np.mean(w * w))) if w.size else 1.0
    rms = rms or 1.0
    ulp = bf16_ulp_distance(gb, wb)
    return dict(max_abs=float(err.max()) if err.size else 0.0, max_rel_rms=float(err.max() / rms) if err.size else 0.0,
                max_ulp=int(ulp.max()) if ulp.size else 0)


SMALL = [0, 1, 5, 63, 64, 65, 200, 1000, 777, 16, 129]


@pytest.fixture(scope="module")
def small_case():
    inp = workloads.make(SMALL, seed=101, layout="perm", pool_slots=6000, gate_std=2.0)
    return inp, reference(inp)


@pytest.mark.parametrize("variant", [1, 2, 3])
@pytest.mark.parametrize("splits", [0, 1, 3, 8, 64])
def test_small_ragged_parity(gda, small_case, variant, splits):
    inp, ref = small_case
    dev = to_cuda(inp)
    out, lse, ws = guarded_io(gda, dev, splits)
    run(gda, dev, num_splits=splits, variant=variant, out=out.t, lse=lse.t, workspace=ws.t)
    check_all(out=out, lse=lse, workspace=ws)
    check_close(bits(out.t), ref.out)
    got_lse, fin = lse.t.cpu().numpy().astype(np.float64), np.isfinite(ref.lse)
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref.lse))
    np.testing.assert_allclose(got_lse[fin], ref.lse[fin], atol=2e-3, rtol=1e-4)


def guarded_io(gda, dev, splits):
    """out, lse and a workspace, each inside 0xFF guard bands (canary.Guarded)."""
    B, Hq, D = dev["q"].shape
    Hkv = dev["k_pool"].shape[1]
    out = Guarded.like(dev["q"])
    lse = Guarded((B, Hq), torch.float32)
    ws = Guarded((max(gda.workspace_bytes(B, Hq, Hkv, D, splits), 256),), torch.uint8)
    gda.workspace_init(ws.t)
    return out, lse, ws


@pytest.mark.parametrize("min_chunk", [1, 16, 64, 100, 1000])
def test_auto_chunking_parity(gda, small_case, min_chunk):
    inp, ref = small_case
    out = run(gda, to_cuda(inp), num_splits=0, min_chunk=min_chunk)
    torch.cuda.synchronize()
    check_close(bits(out), ref.out)


def test_gda_decode_internal_workspace(gda, small_case):
    inp, ref = small_case
    dev = to_cuda(inp)
    for splits in (0, 5):
        out = gda.decode(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"],
                         dev["kv_indices"], scale=dev["scale"], num_splits=splits)
        torch.cuda.synchronize()
        check_close(bits(out), ref.out)
    assert gda.read_error() == 0


def test_decode_step_host_matches_decode(gda, small_case):
    # host block in, decode, host result out: the same bits as gda.decode on device
    # tensors, within tolerance of the oracle; a second step reuses the staging with
    # changed inputs and without waiting inside the call
    inp, ref = small_case
    dev = to_cuda(inp)
    B, Hq, D = inp["q"].shape
    nnz = inp["kv_indices"].numel()
    off, total = gda.step_layout(B, Hq, D, nnz)
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    gda.pack_step(host_in, inp["q"], inp["gate"], inp["kv_indptr"], inp["kv_indices"])
    dev_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    dev_out = torch.empty_like(dev["q"])
    host_out = torch.empty(B, Hq, D, dtype=torch.bfloat16).pin_memory()
    for splits in (0, 5):
        want = gda.decode(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"], dev["kv_indices"],
                          scale=inp["scale"], num_splits=splits)
        torch.cuda.synchronize()
        # copies, or the kernels reading / writing the pinned host buffers in place
        for map_in in (False, True):
            for map_out in (False, True):
                host_out.fill_(7.0)
                gda.decode_step_host(host_in, None if map_in else dev_in, dev["k_pool"], dev["v_pool"],
                                     None if map_out else dev_out, host_out, B, Hq, nnz, scale=inp["scale"],
                                     num_splits=splits, map_in=map_in, map_out=map_out)
                assert np.array_equal(bits(host_out), bits(want)), (splits, map_in, map_out)
        check_close(bits(host_out), ref.out)
    # a second step: other q and gate through the same block, no wait inside the call
    inp2 = dict(inp, q=inp["q"].flip(1).contiguous(), gate=(-inp["gate"]).contiguous())
    gda.pack_step(host_in, inp2["q"], inp2["gate"], inp["kv_indptr"], inp["kv_indices"])
    step = gda.StepHost(host_in, None, dev["k_pool"], dev["v_pool"], None, host_out, B, Hq, nnz,
                        scale=inp["scale"], map_in=True, map_out=True, synchronize=False)
    step()
    torch.cuda.current_stream().synchronize()
    check_close(bits(host_out), reference(inp2).out)
    assert gda.read_error() == 0


def test_fused_equals_unfused_bitwise(gda, small_case):
    inp, ref = small_case
    dev = to_cuda(inp)
    for variant in (1, 2, 3):
        fused = run(gda, dev, variant=variant)
        o_only = run(gda, dev, variant=variant, fuse_gate=False)
        unfused = gda.gate(o_only, dev["gate"])
        torch.cuda.synchronize()
        assert np.array_equal(bits(fused), bits(unfused))
        # the ungated output is RNE_bf16(O): compare with the oracle's O
        check_close(bits(o_only), ref.o_bf16)


def test_deterministic_and_inputs_unmodified(gda, small_case):
    inp, _ = small_case
    dev = to_cuda(inp)
    before = {k: v.clone() for k, v in dev.items() if isinstance(v, torch.Tensor)}
    a = run(gda, dev)
    b = run(gda, dev)
    torch.cuda.synchronize()
    assert np.array_equal(bits(a), bits(b))
    for k, v in before.items():
        assert torch.equal(v.view(torch.uint8) if v.dtype == torch.bfloat16 else v,
                           dev[k].view(torch.uint8) if v.dtype == torch.bfloat16 else dev[k]), k


def test_placement_invariance_bitwise(gda, small_case):
    inp, _ = small_case
    dev = to_cuda(inp)
    n = inp["k_pool"].shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n)
    dev2 = dict(dev)
    dev2["k_pool"] = inp["k_pool"][perm].cuda()
    dev2["v_pool"] = inp["v_pool"][perm].cuda()
    dev2["kv_indices"] = inv[inp["kv_indices"].long()].to(torch.int32).cuda()
    for splits in (0, 4):
        a = run(gda, dev, num_splits=splits)
        b = run(gda, dev2, num_splits=splits)
        torch.cuda.synchronize()
        assert np.array_equal(bits(a), bits(b))


def test_single_key_and_empty_rows_exact(gda):
    inp = workloads.make([1, 0, 1, 1, 0], seed=7, layout="perm", pool_slots=50)
    ref = reference(inp)
    for variant in (1, 2, 3):
        out = run(gda, to_cuda(inp), variant=variant)
        torch.cuda.synchronize()
        got = bits(out)
        assert np.array_equal(got, ref.out)            # one key: O = V row exactly
        assert np.all(got[[1, 4]] == 0)                # empty: +0


def test_lse_output(gda, small_case):
    inp, ref = small_case
    dev = to_cuda(inp)
    lse = torch.empty(len(SMALL), 16, dtype=torch.float32, device="cuda")
    run(gda, dev, lse=lse, num_splits=3)
    torch.cuda.synchronize()
    got = lse.cpu().numpy().astype(np.float64)
    want = ref.lse
    fin = np.isfinite(want)
    assert np.array_equal(np.isneginf(got), np.isneginf(want))
    np.testing.assert_allclose(got[fin], want[fin], atol=2e-3, rtol=1e-4)


def test_custom_scale_and_peaky_scores(gda):
    inp = workloads.make([300, 41, 1, 2048], seed=12, layout="perm", pool_slots=3000, qkv_std=2.5,
                         peaky_frac=0.05, peaky_scale=4.0, scale=0.11)
    ref = reference(inp)
    for variant in (1, 2, 3):
        out = run(gda, to_cuda(inp), variant=variant, num_splits=0)
        torch.cuda.synchronize()
        check_close(bits(out), ref.out)


def test_check_indices_flags_bad_rows(gda):
    inp = workloads.make([40, 30], seed=13, layout="perm", pool_slots=100)
    dev = to_cuda(inp)
    ws = torch.empty(gda.workspace_bytes(2, 16, 2, 256, 0), dtype=torch.uint8, device="cuda")
    gda.workspace_init(ws)
    run(gda, dev, workspace=ws, check_indices=True)
    assert gda.read_error(ws) == 0
    bad = dev["kv_indices"].clone()
    bad[5] = 100          # == num_slots: out of range
    bad[50] = -3
    dev["kv_indices"] = bad
    run(gda, dev, workspace=ws, check_indices=True)
    assert gda.read_error(ws) & gda.DEVERR_INDEX
    assert gda.read_error(ws) == 0   # cleared by the previous read


def test_empty_batch_is_a_no_op(gda):
    q = torch.empty(0, 16, 256, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(4, 2, 256, dtype=torch.bfloat16, device="cuda")
    indptr = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.zeros(0, dtype=torch.int32, device="cuda")
    out = gda.decode(q, q, pool, pool, indptr, idx, scale=0.0625)
    assert out.shape == (0, 16, 256)


def test_graph_replay_with_changed_inputs(gda):
    inp1 = workloads.make([100, 260, 7], seed=21, layout="perm", pool_slots=600)
    inp2 = workloads.make([100, 260, 7], seed=22, layout="perm", pool_slots=600)
    dev = to_cuda(inp1)
    ws = torch.empty(gda.workspace_bytes(3, 16, 2, 256, 0), dtype=torch.uint8, device="cuda")
    gda.workspace_init(ws)
    out = torch.empty_like(dev["q"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(gda, dev, out=out, workspace=ws)   # warm-up (sets kernel attributes) before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(gda, dev, out=out, workspace=ws)
    for inp in (inp1, inp2, inp1):
        for k in ("q", "gate", "k_pool", "v_pool", "kv_indptr", "kv_indices"):
            dev[k].copy_(inp[k])
        g.replay()
        torch.cuda.synchronize()
        check_close(bits(out), reference(inp).out)


def test_internal_workspace_refuses_growth_during_capture(gda):
    inp = workloads.make([64] * 300, seed=23, layout="perm", pool_slots=30_000)
    dev = to_cuda(inp)
    g = torch.cuda.CUDAGraph()
    with pytest.raises(gda.GdaError) as ei:
        with torch.cuda.graph(g):
            gda.decode(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"],
                       dev["kv_indices"], scale=dev["scale"], num_splits=32)
    assert ei.value.status == -7
    # after gda_reserve the same capture succeeds
    gda.reserve(300, 16, 2, 256, 32)
    out = torch.empty_like(dev["q"])
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        gda.decode(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"],
                   dev["kv_indices"], out=out, scale=dev["scale"], num_splits=32)
    g2.replay()
    torch.cuda.synchronize()
    pairs = [(b, h) for b in (0, 123, 299) for h in (0, 7, 8, 15)]
    check_close(bits(out), reference(inp, pairs=pairs).out, pairs=pairs)


def test_graph_stays_valid_after_internal_workspace_growth(gda):
    # a graph captured on the internal workspace keeps that buffer: growing the
    # workspace later (gda_reserve, or a larger eager gda_decode) must not free it,
    # so the replay still gives the oracle's result
    inp = workloads.make([100, 260, 7], seed=24, layout="perm", pool_slots=600)
    dev = to_cuda(inp)
    gda.reserve(3, 16, 2, 256, 8)
    out = torch.empty_like(dev["q"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gda.decode(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"], dev["kv_indices"],
                   out=out, scale=dev["scale"], num_splits=8)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gda.decode(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"], dev["kv_indices"],
                   out=out, scale=dev["scale"], num_splits=8)
    # growth past anything this process used: 512 sequences x 2 KV heads x 256 splits
    # (2 GiB of partials); the drop in free memory shows that a new buffer came
    free0 = torch.cuda.mem_get_info()[0]
    gda.reserve(512, 16, 2, 256, 256)
    assert free0 - torch.cuda.mem_get_info()[0] >= gda.workspace_bytes(512, 16, 2, 256, 256) // 2
    big = workloads.make([33] * 40, seed=25, layout="perm", pool_slots=2000)
    dbig = to_cuda(big)
    out_big = gda.decode(dbig["q"], dbig["gate"], dbig["k_pool"], dbig["v_pool"], dbig["kv_indptr"],
                         dbig["kv_indices"], scale=dbig["scale"], num_splits=200)
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    check_close(bits(out), reference(inp).out)
    check_close(bits(out_big), reference(big).out)
    assert gda.read_error() == 0


# ------------------------------------------------------------------ the named workloads, full size

_cache = {}


def workload_case(key):
    if key not in _cache:
        _cache.clear()
        inp = workloads.make_workload(key)
        _cache[key] = (inp, reference(inp), to_cuda(inp))
    return _cache[key]


@pytest.mark.parametrize("key,splits", [
    ("b1_l512", 8), ("b1_l512", 0), ("b4_ragged", 0), ("b4_ragged", 4),
    ("b64_l4096", 0), ("b64_l4096", 19),
    ("b224_ragged", 0), ("b224_ragged", 8),
    ("b8_l131072", 0), ("b8_l131072", 16), ("b8_l131072", 32), ("b8_l131072", 64), ("b8_l131072", 128),
])
def test_workload_parity(gda, key, splits):
    inp, ref, dev = workload_case(key)
    out, lse, ws = guarded_io(gda, dev, splits)
    run(gda, dev, num_splits=splits, out=out.t, lse=lse.t, workspace=ws.t)
    check_all(out=out, lse=lse, workspace=ws)
    stats = check_close(bits(out.t), ref.out)
    assert gda.read_error(ws.t) == 0
    print(key, splits, stats)


@pytest.mark.parametrize("variant", [2, 3])
def test_workload_parity_other_variants(gda, variant):
    inp, ref, dev = workload_case("b64_l4096")
    out = run(gda, dev, num_splits=0, variant=variant)
    torch.cuda.synchronize()
    check_close(bits(out), ref.out)


@pytest.mark.parametrize("lens", [[5000], [2048] * 4, [3000, 2900, 3100], [700] * 24, [64] * 40])
def test_host_planned_splits(gda, lens):
    # max_len with the exact total: the host applies the split rule and uniform
    # splits run as explicit ones -- the same bits as that explicit count, and the
    # oracle's result within the tolerance
    inp = workloads.make(lens, seed=71 + len(lens), layout="perm", pool_slots=sum(lens) + 500)
    ref = reference(inp)
    dev = to_cuda(inp)
    S = gda.auto_splits(len(lens), 2, 152, max(lens), sum(lens))
    # variant MMA (not AUTO) keeps the call off the one-kernel cluster path
    planned = run(gda, dev, max_len=max(lens), total_len=sum(lens), variant=1)
    torch.cuda.synchronize()
    check_close(bits(planned), ref.out)
    explicit = run(gda, dev, num_splits=S, variant=1) if S > 0 else run(gda, dev, variant=1)
    torch.cuda.synchronize()
    assert np.array_equal(bits(planned), bits(explicit))
