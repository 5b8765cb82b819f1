"""FP8 (e4m3) KV-cache decode on the GPU against the FP64 oracle.

The cache holds e4m3 codes with per-tensor descales (cuDNN FE-OSS "Gated Attention
Block (SM107)", API, QuantSpec: static per-tensor scales, torch.float8_e4m3fn);
q and gate stay BF16 and the output is the BF16 gated result of the BF16 path, so
the tolerance is the same |err| <= 4e-3 + 1.6e-2 |ref| on the gated output.  Its
absolute term is for V values of unit scale (the workloads' std-1 data); where a
test re-reads the codes with a larger v_descale, V and the kernel's absolute
error grow by the same factor, and so does that term.
VARIANT_AUTO and VARIANT_MMA select the same FP8 stage-1 kernel; both are called."""
import numpy as np
import pytest
import torch

import oracle
from canary import Guarded, check_all
from gated_gqa_attention_gb300 import workloads

pytestmark = pytest.mark.gpu

ATOL, RTOL = 4e-3, 1.6e-2
LENS = [0, 1, 5, 63, 64, 65, 200, 1000, 16, 129, 4096, 17]
FORMS = [0, 1]  # VARIANT_AUTO, VARIANT_MMA (the same kernel)


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_close(got, want, pairs=None, v_scale=1.0):
    g = oracle.double_from_bf16(got)
    w = oracle.double_from_bf16(want)
    if pairs is not None:
        idx = tuple(np.asarray(pairs).T)
        g, w = g[idx], w[idx]
    bad = np.abs(g - w) > ATOL * max(1.0, v_scale) + RTOL * np.abs(w)
    assert not bad.any(), "%d / %d out of tolerance, worst %.3g" % (bad.sum(), bad.size, np.abs(g - w).max())
    return float(np.abs(g - w).max()) if g.size else 0.0


def to_cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run(gda, d, **kw):
    sinks = kw.pop("sinks", None)
    out = gda.decode_ex(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"],
                        scale=kw.pop("scale", d["scale"]), k_descale=kw.pop("k_descale", d["k_descale"]),
                        v_descale=kw.pop("v_descale", d["v_descale"]),
                        sinks=None if sinks is None else torch.as_tensor(sinks, dtype=torch.float32).cuda(), **kw)
    torch.cuda.synchronize()
    return bits(out)


def reference(inp, **kw):
    kd = kw.pop("k_descale", inp["k_descale"])
    vd = kw.pop("v_descale", inp["v_descale"])
    return oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"],
                         inp["kv_indices"], kw.pop("scale", inp["scale"]), k_descale=kd, v_descale=vd, **kw)


@pytest.fixture(scope="module")
def batch():
    inp = workloads.make(LENS, seed=301, layout="perm", pool_slots=9000, kv="e4m3")
    return inp, to_cuda(inp)


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("splits", [0, 1, 3, 16, 64])
def test_small_ragged_parity(gda, batch, form, splits):
    inp, dev = batch
    ref = reference(inp)
    check_close(run(gda, dev, num_splits=splits, variant=form), ref.out)


@pytest.mark.parametrize("min_chunk", [16, 64, 1000])
def test_auto_chunking_parity(gda, batch, min_chunk):
    inp, dev = batch
    ref = reference(inp)
    for form in FORMS:
        check_close(run(gda, dev, min_chunk=min_chunk, variant=form), ref.out)


@pytest.mark.parametrize("kd,vd", [(0.0137, 0.0291), (1.0, 1.0), (2.0 ** -7, 3.5), (1e-4, 1e-3)])
def test_descales(gda, batch, kd, vd):
    inp, dev = batch
    ref = reference(inp, k_descale=kd, v_descale=vd)
    for form in FORMS:
        check_close(run(gda, dev, k_descale=kd, v_descale=vd, variant=form), ref.out, v_scale=vd / inp["v_descale"])


def test_lse_unfused_and_simple_entry_point(gda, batch):
    inp, dev = batch
    ref = reference(inp)
    B = len(LENS)
    lse = torch.empty(B, 16, dtype=torch.float32, device="cuda")
    check_close(run(gda, dev, lse=lse), ref.out)
    ok = np.isfinite(ref.lse)
    np.testing.assert_allclose(lse.cpu().numpy()[ok], ref.lse[ok], atol=2e-3, rtol=1e-4)
    assert np.all(np.isneginf(lse.cpu().numpy()[~ok]))
    # unfused first half: RNE_bf16(O)
    check_close(run(gda, dev, fuse_gate=False), ref.o_bf16)
    # gda_decode_e4m3 (library-owned workspace)
    out = gda.decode(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"], dev["kv_indices"],
                     scale=dev["scale"], k_descale=dev["k_descale"], v_descale=dev["v_descale"])
    torch.cuda.synchronize()
    check_close(bits(out), ref.out)


def test_deterministic_and_inputs_unmodified(gda, batch):
    inp, dev = batch
    k0, v0 = dev["k_pool"].clone(), dev["v_pool"].clone()
    for form in FORMS:
        a = run(gda, dev, variant=form)
        b = run(gda, dev, variant=form)
        assert np.array_equal(a, b)
    assert torch.equal(k0.view(torch.uint8), dev["k_pool"].view(torch.uint8))
    assert torch.equal(v0.view(torch.uint8), dev["v_pool"].view(torch.uint8))


@pytest.mark.parametrize("window", [1, 7, 64, 300, 100_000])
def test_sliding_window(gda, batch, window):
    inp, dev = batch
    ref = reference(inp, window=window)
    for splits in (0, 3):
        check_close(run(gda, dev, window=window, num_splits=splits), ref.out)


def test_attention_sinks(gda, batch):
    inp, dev = batch
    rng = np.random.default_rng(7)
    sinks = rng.normal(0.0, 3.0, 16).astype(np.float32)
    sinks[2] = -np.inf
    sinks[9] = 40.0
    ref = reference(inp, sinks=sinks.astype(np.float64))
    for splits in (0, 5):
        check_close(run(gda, dev, sinks=sinks, num_splits=splits), ref.out)


@pytest.mark.parametrize("hq,hkv", [(16, 16), (16, 8), (6, 2), (12, 2), (32, 2), (24, 1), (16, 1), (40, 2),
                                    (64, 2)])
def test_group_sizes(gda, hq, hkv):
    # G > 8: the groups of 8 go in pairs (one piece, one read of the rows per pair); G =
    # 24 and 20 leave the second pair half empty, G = 32 is two pairs
    inp = workloads.make([0, 3, 77, 600, 1500], seed=311, hq=hq, hkv=hkv, layout="perm", pool_slots=3000,
                         kv="e4m3")
    dev = to_cuda(inp)
    ref = reference(inp)
    for splits in (0, 4):
        check_close(run(gda, dev, num_splits=splits), ref.out)


@pytest.mark.parametrize("hq,hkv", [(32, 2), (48, 2)])
def test_pairs_long_ragged_window_sinks_lse(gda, hq, hkv):
    # pairs over a long ragged batch: pieces cross sequences and CTAs, the partner warps
    # meet at every step; a window, sinks and the LSE go through the same mapping, and
    # repeated calls give the same bits
    lens = [4096, 1, 0, 3000, 777, 65, 2049, 16, 5000, 129, 1500, 2]
    inp = workloads.make(lens, seed=520 + hq, hq=hq, hkv=hkv, layout="perm", pool_slots=20000, peaky_frac=0.01,
                         kv="e4m3")
    dev = to_cuda(inp)
    ref = reference(inp)
    for kw in ({}, {"min_chunk": 16}, {"num_splits": 7}):
        a = run(gda, dev, **kw)
        check_close(a, ref.out)
        assert np.array_equal(a, run(gda, dev, **kw))
    sinks = np.linspace(-2.0, 2.0, hq).astype(np.float32)
    ref = reference(inp, window=1000, sinks=sinks.astype(np.float64))
    lse = torch.empty(len(lens), hq, dtype=torch.float32, device="cuda")
    check_close(run(gda, dev, window=1000, sinks=sinks, lse=lse), ref.out)
    np.testing.assert_allclose(lse.cpu().numpy(), ref.lse, atol=2e-3, rtol=1e-4)


def test_all_codes_and_extreme_q(gda):
    """Codes drawn uniformly over every finite e4m3 value (subnormals and +-448
    included); q rows that are zero, tiny, huge, or a single spike."""
    inp = workloads.make([1, 40, 333, 2048], seed=321, layout="perm", pool_slots=4000, kv="e4m3")
    g = torch.Generator().manual_seed(9)
    finite = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
    for name in ("k_pool", "v_pool"):
        pick = torch.randint(0, finite.numel(), inp[name].shape, generator=g)
        inp[name] = finite[pick].view(torch.float8_e4m3fn)
    q = inp["q"].clone()
    q[0] = 0.0
    q[1, :8] *= 1e-30
    q[2, :8] *= 1e20
    q[3, 8:] = 0.0
    q[3, 8:, 5] = 3.0
    inp["q"] = q
    inp["k_descale"], inp["v_descale"] = 2.0 ** -9, 0.01
    dev = to_cuda(inp)
    ref = reference(inp)
    v_std = float(np.std(inp["v_pool"].to(torch.float64).numpy())) * inp["v_descale"]
    for form in FORMS:
        for splits in (0, 7):
            check_close(run(gda, dev, num_splits=splits, variant=form), ref.out, v_scale=v_std)


def test_pairs_scale_q_per_group(gda):
    """G = 16 runs the two groups of 8 query heads of a KV head as one piece; each group
    gets its own power-of-two factor into FP16, so a group of ordinary magnitude next
    to a group ~2^66 larger keeps its scores (one shared factor would flush it to
    zero and flatten its softmax)."""
    inp = workloads.make([1, 300, 2048, 77], seed=331, hq=32, hkv=2, layout="perm", pool_slots=3000,
                         kv="e4m3")
    q = inp["q"].clone()
    q[:, 0:8] *= 1e20        # group 0 of KV head 0
    q[:, 24:32] *= 1e-20     # group 1 of KV head 1
    q[2, 8:16] *= 1e-30      # group 1 of KV head 0, one sequence: tiny
    inp["q"] = q
    dev = to_cuda(inp)
    ref = reference(inp)
    for splits in (0, 5):
        check_close(run(gda, dev, num_splits=splits), ref.out)


def test_pairs_many_segments_and_bad_indices(gda):
    # G = 16 pairs with more (sequence, KV head, pair) segments than CTAs (the
    # cost-weighted stream schedule), then one bad index under check_indices
    rng = np.random.default_rng(341)
    lens = [int(x) for x in rng.integers(1, 600, 160)]
    lens[9] = 0
    lens[100] = 3000
    inp = workloads.make(lens, seed=342, hq=32, hkv=2, layout="perm", pool_slots=sum(lens) + 500, kv="e4m3")
    dev = to_cuda(inp)
    ref = reference(inp)
    for kw in ({}, {"max_len": max(lens), "total_len": sum(lens)}, {"num_splits": 3}):
        check_close(run(gda, dev, **kw), ref.out)
    B, Hq, D = dev["q"].shape
    ws = torch.empty(gda.workspace_bytes(B, Hq, 2, D, 0), dtype=torch.uint8, device="cuda")
    gda.workspace_init(ws)
    bad = dev["kv_indices"].clone()
    bad[1234] = 10 ** 8
    gda.decode_ex(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"], bad,
                  scale=dev["scale"], k_descale=dev["k_descale"], v_descale=dev["v_descale"],
                  check_indices=True, workspace=ws)
    assert gda.read_error(ws) == gda.DEVERR_INDEX


def test_check_indices_flags_bad_rows(gda, batch):
    inp, dev = batch
    bad = dev["kv_indices"].clone()
    bad[3] = 10 ** 8
    B, Hq, D = dev["q"].shape
    ws = torch.empty(gda.workspace_bytes(B, Hq, 2, D, 0), dtype=torch.uint8, device="cuda")
    gda.workspace_init(ws)
    gda.decode_ex(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"], dev["kv_indices"],
                  scale=dev["scale"], k_descale=dev["k_descale"], v_descale=dev["v_descale"],
                  check_indices=True, workspace=ws)
    assert gda.read_error(ws) == 0
    gda.decode_ex(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"], bad,
                  scale=dev["scale"], k_descale=dev["k_descale"], v_descale=dev["v_descale"],
                  check_indices=True, workspace=ws)
    assert gda.read_error(ws) == gda.DEVERR_INDEX
    assert gda.read_error(ws) == 0  # cleared by the first read


def test_unsupported_forms_are_refused(gda, batch):
    inp, dev = batch
    for variant in (2, 3):
        with pytest.raises(gda.GdaError) as ei:
            run(gda, dev, variant=variant)
        assert ei.value.status == -4
    with pytest.raises(gda.GdaError) as ei:
        run(gda, dev, k_descale=float("nan"))
    assert ei.value.status == -10


# ------------------------------------------------------------------ the named workloads over an FP8 cache, full size

_cache = {}


def workload_case(key):
    if key not in _cache:
        _cache.clear()
        inp = workloads.make_workload(key, kv="e4m3")
        _cache[key] = (inp, reference(inp), to_cuda(inp))
    return _cache[key]


@pytest.mark.parametrize("key,splits,form", [
    ("b1_l512", 8, 0), ("b1_l512", 0, 0), ("b4_ragged", 0, 0), ("b4_ragged", 0, 1),
    ("b64_l4096", 0, 0), ("b64_l4096", 0, 1), ("b64_l4096", 19, 0),
    ("b224_ragged", 0, 0), ("b224_ragged", 8, 1),
    ("b8_l131072", 0, 0), ("b8_l131072", 64, 1),
])
def test_workload_parity(gda, key, splits, form):
    # out, lse and the workspace inside 0xFF guard bands (canary.Guarded)
    inp, ref, dev = workload_case(key)
    B, Hq, D = inp["q"].shape
    out, lse = Guarded.like(dev["q"]), Guarded((B, Hq), torch.float32)
    ws = Guarded((gda.workspace_bytes(B, Hq, inp["k_pool"].shape[1], D, splits),), torch.uint8)
    gda.workspace_init(ws.t)
    got = run(gda, dev, num_splits=splits, variant=form, out=out.t, lse=lse.t, workspace=ws.t)
    check_all(out=out, lse=lse, workspace=ws)
    worst = check_close(got, ref.out)
    assert gda.read_error(ws.t) == 0
    print(key, splits, form, worst)
