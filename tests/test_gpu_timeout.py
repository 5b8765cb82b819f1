"""The bounded-wait failure path on the GPU, made to run out on purpose.

The kernels that wait on mbarriers -- the prefill kernel and the TMA-ring decode
stage 1 -- give up a pipeline wait after a limit of SM cycles, record
GDA_DEVERR_TIMEOUT in their error word, wait (under the normal limit) for the copies
and MMAs they already started, and return (cuDNN FE-OSS "Gated Attention Block
(SM107)", Forward: a typed error, not a hang).  gda_debug_wait_limit shortens the
limit to a few hundred cycles, far below the latency of the first TMA load, so the
first wait of every CTA gives up.  Each test checks that the call returns, that the
error word carries the timeout bit, and that the next call with the normal limit on
the same stream gives the oracle's result with a clean error word.  One small case
each; no wait is left without a limit."""
import numpy as np
import pytest
import torch

import oracle
from gated_gqa_attention_gb300 import workloads

pytestmark = pytest.mark.gpu

ATOL, RTOL = 4e-3, 1.6e-2
SHORT = 200          # SM cycles
TIMEOUT_BIT = 0x2


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_close(got, want):
    g = oracle.double_from_bf16(got)
    w = oracle.double_from_bf16(want)
    assert np.all(np.abs(g - w) <= ATOL + RTOL * np.abs(w))


def test_prefill_wait_limit_gives_a_typed_timeout(gda):
    inp = workloads.make_prefill(1, 256, 256, seed=91, hq=2, hkv=1, causal=True)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    call = lambda: gda.prefill(dev["q"], dev["gate"], dev["k"], dev["v"], scale=inp["scale"], causal=True,
                               error_word=err)
    call()                                  # first use on the device (table, attributes) at the normal limit
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    try:
        gda.debug_wait_limit(SHORT)
        call()
        torch.cuda.synchronize()            # the call returns: no hang
    finally:
        gda.debug_wait_limit(0)
    assert int(err.item()) & TIMEOUT_BIT
    err.zero_()
    out = call()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_close(bits(out), oracle.prefill(inp["q"], inp["gate"], inp["k"], inp["v"], inp["scale"], causal=True).out)


def test_tma_ring_decode_wait_limit_gives_a_typed_timeout(gda):
    inp = workloads.make([300, 77, 1000], seed=92, layout="perm", pool_slots=2000)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    ws = torch.empty(gda.workspace_bytes(3, 16, 2, 256, 0), dtype=torch.uint8, device="cuda")
    gda.workspace_init(ws)
    call = lambda: gda.decode_ex(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"],
                                 dev["kv_indices"], workspace=ws, scale=inp["scale"], variant=gda.VARIANT_TMA)
    call()
    assert gda.read_error(ws) == 0
    try:
        gda.debug_wait_limit(SHORT)
        call()
        torch.cuda.synchronize()
    finally:
        gda.debug_wait_limit(0)
    assert gda.read_error(ws) & TIMEOUT_BIT   # read and cleared
    out = call()
    assert gda.read_error(ws) == 0
    ref = oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"], inp["kv_indices"],
                        inp["scale"])
    check_close(bits(out), ref.out)
