"""The allocation-free entry point, gda_decode_noalloc.

Some callers may not allocate device memory: a serving loop whose GPU memory was
reserved up front, a pooled allocator that owns every byte, a thread that must
never block on the driver's allocator.  gda_decode_noalloc serves them with a
fixed scratch area that the library declares statically on every device.  These
tests call it through the C ABI and check it against gda_decode, the entry point
with a library-owned workspace, on two calls in a row (the second reuses the
scratch as the first left it).  Both calls run the same kernels on the same plan,
so they must agree bit for bit; both are also checked against the FP64 oracle.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import gated_gqa_attention_gb300 as gda_mod
import oracle
from gated_gqa_attention_gb300 import build, workloads

ATOL, RTOL = 4e-3, 1.6e-2   # the decode parity tolerance used by every other test


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _check_oracle(got_bits, inp):
    ref = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"], inp["kv_indices"],
                        inp["scale"])
    g = oracle.double_from_bf16(got_bits)
    w = oracle.double_from_bf16(ref.out)
    bad = np.abs(g - w) > ATOL + RTOL * np.abs(w)
    assert not bad.any(), "%d elements out of tolerance" % int(bad.sum())


def _call_noalloc(lib, d, out, num_splits):
    vp = ctypes.c_void_p
    return lib.gda_decode_noalloc(
        vp(d["q"].data_ptr()), vp(d["gate"].data_ptr()), vp(d["k_pool"].data_ptr()), vp(d["v_pool"].data_ptr()),
        vp(d["kv_indptr"].data_ptr()), vp(d["kv_indices"].data_ptr()), vp(out.data_ptr()),
        d["q"].shape[0], d["q"].shape[1], d["k_pool"].shape[1], d["q"].shape[2], d["scale"], num_splits,
        vp(torch.cuda.current_stream().cuda_stream))


def test_noalloc_rejects_sizes_beyond_the_scratch():
    # host-side size check: answered before any CUDA call, so it needs no GPU
    build.build()
    lib = gda_mod.load()
    vp = ctypes.c_void_p
    args = [vp(256)] * 7
    assert lib.gda_workspace_bytes(508, 16, 2, 256, 0) <= gda_mod.NOALLOC_SCRATCH_BYTES
    assert lib.gda_workspace_bytes(509, 16, 2, 256, 0) > gda_mod.NOALLOC_SCRATCH_BYTES
    assert lib.gda_decode_noalloc(*args, 509, 16, 2, 256, 0.0625, 0, None) == -6     # automatic: > 508
    assert lib.gda_decode_noalloc(*args, 511, 16, 2, 256, 0.0625, 2, None) == -6     # 511 * 2 > 1020
    assert lib.gda_decode_noalloc(None, *args[1:], 4, 16, 2, 256, 0.0625, 0, None) == -1


def _run_twice(gda, lib, inp, num_splits):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    ref = gda.decode(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"],
                     scale=d["scale"], num_splits=num_splits)
    torch.cuda.synchronize()
    want = _bits(ref)
    _check_oracle(want, inp)
    outs = [torch.full_like(d["q"], float("nan")) for _ in range(2)]
    # the first call on a device looks up the scratch address (and may load the
    # module); from the second call on, nothing may change the free device memory
    assert _call_noalloc(lib, d, outs[0], num_splits) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for out in outs:
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        assert _call_noalloc(lib, d, out, num_splits) == 0
        torch.cuda.synchronize()
        assert np.array_equal(_bits(out), want)
    assert torch.cuda.mem_get_info()[0] == free0


@pytest.mark.gpu
def test_noalloc_matches_gda_decode_twice(gda):
    lib = gda.load()
    for num_splits in (0, 5):
        inp = workloads.make([0, 1, 300, 1000, 4096, 77, 16], seed=77 + num_splits, layout="perm",
                             pool_slots=8000)
        _run_twice(gda, lib, inp, num_splits)


@pytest.mark.gpu
def test_noalloc_at_the_largest_accepted_size(gda):
    # B = 508 in automatic mode fills the 16 MiB scratch exactly (Hq 16, Hkv 2, D 256);
    # B = 509 is refused above
    lib = gda.load()
    lens = [int(x) for x in np.random.default_rng(5).integers(1, 65, 508)]
    inp = workloads.make(lens, seed=78, layout="perm", pool_slots=sum(lens) + 100)
    _run_twice(gda, lib, inp, 0)
