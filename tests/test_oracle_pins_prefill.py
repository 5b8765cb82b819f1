"""Pins of the prefill / extend oracle (gated SDPA over per-sequence K and V) to
things other than itself (CPU only).

cuDNN FE-OSS "Gated Attention Block (SM107)", Overview stages (4)-(5): O =
softmax(Q K^T * scale + mask) V with GQA, O *= sigmoid(GATE) after the dead-row
select.  Each pin catches a plausible mistake:
  * the library SDPA (torch, float64, explicit boolean mask, GQA) on causal,
    dense, extend (Sq < Skv) and padded (kv_lens) cases -- a shifted causal
    diagonal, a wrong head mapping or a transposed operand fails it;
  * brute-force pure-Python loops on tiny inputs;
  * the decode oracle: query i of a causal prefill is a decode token whose KV rows
    are keys 0 .. i + (L - Sq);
  * closed forms: the first causal query sees one key (O = that V row exactly),
    q = 0 gives the mean of the visible V rows, a dead row gives O = 0, lse = -inf;
  * the gate stage follows from O by the pinned rounding and gate functions.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gated_gqa_attention_gb300 import workloads


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(t):
    return t.to(torch.float64)


def _mask(B, Sq, Skv, causal, kv_lens, shift=0):
    """[B, Sq, Skv] boolean visibility (True = attend)."""
    m = torch.zeros(B, Sq, Skv, dtype=torch.bool)
    for b in range(B):
        L = Skv if kv_lens is None else int(kv_lens[b])
        j = torch.arange(Skv)[None, :]
        i = torch.arange(Sq)[:, None]
        vis = j < L
        if causal:
            vis = vis & (j <= i + (L - Sq) + shift)
        m[b] = vis
    return m


def _library(inp, shift=0):
    """torch SDPA in float64 with an explicit mask; dead rows -> 0."""
    q, k, v = _f64(inp["q"]), _f64(inp["k"]), _f64(inp["v"])
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    m = _mask(B, Sq, Skv, inp["causal"], inp["kv_lens"], shift)
    out = torch.zeros(B, Sq, Hq, D, dtype=torch.float64)
    lse = torch.full((B, Hq, Sq), -math.inf, dtype=torch.float64)
    for b in range(B):
        live = m[b].any(dim=1)
        if not live.any():
            continue
        qb = q[b].transpose(0, 1)[:, live]             # [Hq, n, D]
        kb = k[b].transpose(0, 1)                      # [Hkv, Skv, D]
        vb = v[b].transpose(0, 1)
        mb = m[b][live][None, None]                    # [1, 1, n, Skv]
        o = torch.nn.functional.scaled_dot_product_attention(qb[None], kb[None], vb[None], attn_mask=mb,
                                                             scale=inp["scale"], enable_gqa=True)[0]
        out[b, live] = o.transpose(0, 1)
        s = torch.einsum("hnd,hjd->hnj", qb, kb.repeat_interleave(Hq // Hkv, dim=0)) * inp["scale"]
        s = s.masked_fill(~mb[0], -math.inf)
        lse[b][:, live] = torch.logsumexp(s, dim=-1)
    return out.numpy(), lse.numpy()


CASES = [
    # B, Sq, Skv, Hq, Hkv, D, causal, kv_lens
    (1, 37, 37, 4, 2, 16, True, None),
    (2, 20, 20, 6, 2, 32, False, None),
    (2, 9, 30, 4, 1, 8, True, None),            # extend: 9 new tokens after 21 cached
    (3, 16, 24, 8, 2, 16, True, [24, 10, 0]),    # padded KV, one empty sequence (dead rows)
    (2, 12, 12, 4, 4, 64, False, [5, 12]),
    (1, 64, 64, 32, 2, 256, True, None),        # the page's head geometry
]


@pytest.mark.parametrize("B,Sq,Skv,Hq,Hkv,D,causal,kv_lens", CASES)
def test_prefill_against_library_sdpa(B, Sq, Skv, Hq, Hkv, D, causal, kv_lens):
    inp = workloads.make_prefill(B, Sq, Skv, seed=1000 + Sq + D, hq=Hq, hkv=Hkv, head_dim=D, causal=causal,
                                 kv_lens=kv_lens)
    res = oracle.prefill(inp["q"], inp["gate"], inp["k"], inp["v"], inp["scale"], causal=causal,
                         kv_lens=inp["kv_lens"])
    want, lse = _library(inp)
    np.testing.assert_allclose(res.o_f64, want, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(res.lse, lse, rtol=1e-12, atol=1e-12)
    assert np.array_equal(res.o_bf16, oracle.bf16_from_double(res.o_f64))
    assert np.array_equal(res.out, oracle.gate(res.o_bf16, _bits(inp["gate"])))
    if causal:
        # a causal diagonal shifted by one key is a different result
        bad, _ = _library(inp, shift=1)
        assert not np.allclose(bad, want, rtol=1e-6, atol=1e-9)


def _brute(inp):
    q, k, v = _f64(inp["q"]).numpy(), _f64(inp["k"]).numpy(), _f64(inp["v"]).numpy()
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    O = np.zeros_like(q)
    for b in range(B):
        L = Skv if inp["kv_lens"] is None else int(inp["kv_lens"][b])
        for i in range(Sq):
            keys = [j for j in range(L) if (not inp["causal"]) or j <= i + (L - Sq)]
            for h in range(Hq):
                if not keys:
                    continue
                s = [inp["scale"] * math.fsum(q[b, i, h, d] * k[b, j, h // G, d] for d in range(D)) for j in keys]
                m = max(s)
                w = [math.exp(x - m) for x in s]
                z = math.fsum(w)
                for d in range(D):
                    O[b, i, h, d] = math.fsum(wj * v[b, j, h // G, d] for wj, j in zip(w, keys)) / z
    return O


@pytest.mark.parametrize("B,Sq,Skv,Hq,Hkv,D,causal,kv_lens", [
    (1, 5, 5, 2, 1, 4, True, None), (2, 3, 7, 4, 2, 8, True, [7, 4]), (1, 6, 6, 3, 3, 4, False, None),
])
def test_prefill_brute_force(B, Sq, Skv, Hq, Hkv, D, causal, kv_lens):
    inp = workloads.make_prefill(B, Sq, Skv, seed=77 + D, hq=Hq, hkv=Hkv, head_dim=D, causal=causal, kv_lens=kv_lens)
    res = oracle.prefill(inp["q"], inp["gate"], inp["k"], inp["v"], inp["scale"], causal=causal,
                         kv_lens=inp["kv_lens"])
    np.testing.assert_allclose(res.o_f64, _brute(inp), rtol=1e-12, atol=1e-14)


def test_prefill_rows_match_the_decode_oracle():
    B, Sq, Skv, Hq, Hkv, D = 2, 11, 29, 8, 2, 32
    inp = workloads.make_prefill(B, Sq, Skv, seed=5, hq=Hq, hkv=Hkv, head_dim=D, causal=True, kv_lens=[29, 17])
    res = oracle.prefill(inp["q"], inp["gate"], inp["k"], inp["v"], inp["scale"], causal=True, kv_lens=inp["kv_lens"])
    # each (b, i) becomes one decode token over keys 0 .. i + (L - Sq) of sequence b
    qs, gs, indptr, indices = [], [], [0], []
    pool_k = inp["k"].reshape(B * Skv, Hkv, D)
    pool_v = inp["v"].reshape(B * Skv, Hkv, D)
    for b in range(B):
        L = int(inp["kv_lens"][b])
        for i in range(Sq):
            last = min(L - 1, i + (L - Sq))
            qs.append(inp["q"][b, i])
            gs.append(inp["gate"][b, i])
            indices.extend(b * Skv + j for j in range(last + 1))
            indptr.append(len(indices))
    dec = oracle.decode(torch.stack(qs), torch.stack(gs), pool_k, pool_v, np.array(indptr, np.int32),
                        np.array(indices, np.int32), inp["scale"])
    np.testing.assert_allclose(res.o_f64.reshape(B * Sq, Hq, D), dec.o_f64, rtol=1e-13, atol=1e-15)
    assert np.array_equal(res.out.reshape(B * Sq, Hq, D), dec.out)
    np.testing.assert_allclose(res.lse.transpose(0, 2, 1).reshape(B * Sq, Hq), dec.lse, rtol=1e-13, atol=1e-13)


def test_prefill_closed_forms():
    B, S, Hq, Hkv, D = 2, 8, 4, 2, 16
    inp = workloads.make_prefill(B, S, S, seed=9, hq=Hq, hkv=Hkv, head_dim=D, causal=True, kv_lens=[8, 0])
    res = oracle.prefill(inp["q"], inp["gate"], inp["k"], inp["v"], inp["scale"], causal=True, kv_lens=inp["kv_lens"])
    v = _f64(inp["v"]).numpy()
    # query 0 of a plain causal prefill sees key 0 only: O = v_0 exactly, lse = its score
    for h in range(Hq):
        assert np.array_equal(res.o_f64[0, 0, h], v[0, 0, h // 2])
        s0 = inp["scale"] * float(np.dot(_f64(inp["q"][0, 0, h]).numpy(), _f64(inp["k"][0, 0, h // 2]).numpy()))
        assert abs(res.lse[0, h, 0] - s0) < 1e-12
    # an empty sequence: dead rows everywhere
    assert np.all(res.o_f64[1] == 0) and np.all(res.out[1] == 0) and np.all(np.isneginf(res.lse[1]))
    # q = 0: uniform weights over the visible keys -> their mean (dense: all keys)
    inp0 = dict(inp, q=torch.zeros_like(inp["q"]), kv_lens=None)
    r0 = oracle.prefill(inp0["q"], inp0["gate"], inp0["k"], inp0["v"], inp0["scale"], causal=False)
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_allclose(r0.o_f64[b, 3, h], v[b, :, h // 2].mean(axis=0), rtol=1e-14, atol=1e-15)
            np.testing.assert_allclose(r0.lse[b, h, 3], math.log(S), rtol=1e-15)


def test_prefill_rows_subset_matches_full():
    inp = workloads.make_prefill(2, 10, 14, seed=3, hq=4, hkv=2, head_dim=16, causal=True)
    full = oracle.prefill(inp["q"], inp["gate"], inp["k"], inp["v"], inp["scale"], causal=True)
    rows = [(0, 0, 1), (1, 9, 3), (1, 4, 0)]
    sub = oracle.prefill(inp["q"], inp["gate"], inp["k"], inp["v"], inp["scale"], causal=True, rows=rows)
    for b, i, h in rows:
        assert np.array_equal(sub.o_f64[b, i, h], full.o_f64[b, i, h])
        assert np.array_equal(sub.out[b, i, h], full.out[b, i, h])
        assert sub.lse[b, h, i] == full.lse[b, h, i]
