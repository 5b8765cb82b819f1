"""Seeded synthetic decode workloads (inputs only; none of the method's arithmetic).

The five workloads are the decode shapes the gated-attention pages measure or
serve, built from seeded random numbers because no page ships data:

1. ``b1_l512``      B=1, KV length 512, a 1024-slot pool, slots a random
                    subset (FreeToken PR #781, Automatic dispatch and Kernel
                    window: query [1,16,256], two KV heads, CSR capacity 512).
2. ``b4_ragged``    B=4, lengths 512/495/478/461 over a shuffled 4096-slot pool
                    (FreeToken PR #781, Kernel window, the B4 row).
3. ``b64_l4096``    B=64, length 4096, 16-slot pages placed at random in a
                    300 000-slot pool (the bandwidth workload).
4. ``b224_ragged``  B=224, lengths uniform in [1, 6142], slots a permutation of
                    the pool, 1% of referenced K rows scaled by 3 (a peaky
                    softmax); the shape of ROCm/ATOM PR #838's CONC=224,
                    ISL 4094 / OSL 2048 serving run.
5. ``b8_l131072``   B=8, length 131072, 64-slot pages in random order.

Every workload has Hq=16, Hkv=2, D=256, scale 1/16 and BF16 q / gate / K / V
drawn from normal distributions (gate standard deviation 2, except workload 4
where it is 1).  Draw order, all from one ``torch.Generator`` seeded with the
workload's seed: lengths (if random) -> slot layout -> peaky-row mask -> q ->
gate -> K pool -> V pool.  Values are drawn in float32, scaled, then rounded to
BF16 (round-to-nearest-even).  Every pool row is filled, referenced or not.

FP8 KV cache (``kv="e4m3"``): the same float32 draws of the pools are divided by a
per-tensor descale, saturated to the e4m3 range (+-448) and converted to
torch.float8_e4m3fn; the descale is the one a 6-sigma calibration gives,
6 * std * (largest row factor) / 448, rounded to float32.  q and gate stay BF16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

HQ, HKV, HEAD_DIM = 16, 2, 256
E4M3_MAX = 448.0
DEFAULT_SCALE = 1.0 / 16.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    lengths: Optional[Sequence[int]]     # None -> drawn uniform in [len_lo, len_hi]
    len_lo: int
    len_hi: int
    layout: str                          # "subset" | "pages" | "perm"
    pool_slots: Optional[int]            # None -> exactly the referenced count
    page: int
    gate_std: float
    peaky_frac: float
    seed: int
    num_splits: int                      # split count the workload names (0: automatic)
    hq: int = HQ
    hkv: int = HKV
    head_dim: int = HEAD_DIM
    scale: float = DEFAULT_SCALE


WORKLOADS: List[Workload] = [
    Workload("b1_l512", 1, [512], 0, 0, "subset", 1024, 1, 2.0, 0.0, 0, 8),
    Workload("b4_ragged", 4, [512, 495, 478, 461], 0, 0, "subset", 4096, 1, 2.0, 0.0, 1, 0),
    Workload("b64_l4096", 64, [4096] * 64, 0, 0, "pages", 300_000, 16, 2.0, 0.0, 2, 0),
    Workload("b224_ragged", 224, None, 1, 6142, "perm", None, 1, 1.0, 0.01, 3, 0),
    Workload("b8_l131072", 8, [131072] * 8, 0, 0, "pages", 1_048_576, 64, 2.0, 0.0, 4, 128),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def workload(key) -> Workload:
    """Look a workload up by name or by its 1-based number."""
    if isinstance(key, int):
        return WORKLOADS[key - 1]
    if isinstance(key, str) and key.isdigit():
        return WORKLOADS[int(key) - 1]
    return BY_NAME[key]


def _randn_bf16(gen: torch.Generator, rows: int, cols: int, std: float,
                row_scale: Optional[torch.Tensor] = None) -> torch.Tensor:
    """[rows, cols] BF16 of N(0, std^2) values, drawn in float32 chunks on the
    generator's device.

    ``row_scale`` (float32 [rows]) multiplies rows in float32 before the
    rounding to BF16."""
    out = torch.empty(rows, cols, dtype=torch.bfloat16, device=gen.device)
    if row_scale is not None:
        row_scale = row_scale.to(gen.device)
    chunk = max(1, (1 << 24) // max(cols, 1))
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        x = torch.randn(r1 - r0, cols, generator=gen, dtype=torch.float32, device=gen.device)
        if std != 1.0:
            x.mul_(std)
        if row_scale is not None:
            x.mul_(row_scale[r0:r1, None])
        out[r0:r1] = x.to(torch.bfloat16)
    return out


def _randn_e4m3(gen: torch.Generator, rows: int, cols: int, std: float, descale: float,
                row_scale: Optional[torch.Tensor] = None) -> torch.Tensor:
    """[rows, cols] float8_e4m3fn codes of the same float32 draws as _randn_bf16,
    divided by ``descale`` and saturated at +-448."""
    out = torch.empty(rows, cols, dtype=torch.float8_e4m3fn, device=gen.device)
    if row_scale is not None:
        row_scale = row_scale.to(gen.device)
    chunk = max(1, (1 << 24) // max(cols, 1))
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        x = torch.randn(r1 - r0, cols, generator=gen, dtype=torch.float32, device=gen.device)
        if std != 1.0:
            x.mul_(std)
        if row_scale is not None:
            x.mul_(row_scale[r0:r1, None])
        x.div_(descale).clamp_(-E4M3_MAX, E4M3_MAX)
        out[r0:r1] = x.to(torch.float8_e4m3fn)
    return out


def _layout(gen: torch.Generator, lengths: List[int], layout: str, pool_slots: Optional[int],
            page: int):
    nnz = int(sum(lengths))
    if layout == "subset":
        slots = pool_slots if pool_slots is not None else nnz
        assert slots >= nnz
        idx = torch.randperm(slots, generator=gen)[:nnz].to(torch.int32)
    elif layout == "perm":
        slots = nnz if pool_slots is None else pool_slots
        idx = torch.randperm(slots, generator=gen)[:nnz].to(torch.int32)
    elif layout == "pages":
        pages_needed = [int(math.ceil(L / page)) for L in lengths]
        total_pages = sum(pages_needed)
        slots = pool_slots if pool_slots is not None else total_pages * page
        pool_pages = slots // page
        assert pool_pages >= total_pages, "pool too small for the pages"
        order = torch.randperm(pool_pages, generator=gen)[:total_pages]
        parts = []
        p = 0
        for L, npg in zip(lengths, pages_needed):
            pg = order[p:p + npg]
            p += npg
            s = (pg[:, None] * page + torch.arange(page)[None, :]).reshape(-1)[:L]
            parts.append(s)
        idx = (torch.cat(parts) if parts else torch.empty(0, dtype=torch.int64)).to(torch.int32)
    else:
        raise ValueError(layout)
    return idx, slots


def make(lengths: Sequence[int], *, seed: int, hq: int = HQ, hkv: int = HKV,
         head_dim: int = HEAD_DIM, layout: str = "perm", pool_slots: Optional[int] = None,
         page: int = 1, gate_std: float = 2.0, qkv_std: float = 1.0, peaky_frac: float = 0.0,
         peaky_scale: float = 3.0, scale: float = DEFAULT_SCALE, random_lengths=None,
         kv: str = "bf16", values_device: Optional[str] = None) -> dict:
    """Build one decode batch on the CPU.

    Returns a dict of CPU tensors ``q, gate`` [B, Hq, D] bf16, ``k_pool, v_pool``
    [slots, Hkv, D] bf16 (float8_e4m3fn with ``kv="e4m3"``), ``kv_indptr`` [B+1]
    int32, ``kv_indices`` [nnz] int32, plus ``scale``, ``lengths``, ``num_slots``
    and the pools' ``k_descale`` / ``v_descale`` (1.0 for BF16 pools).
    ``random_lengths=(lo, hi, B)`` draws the lengths uniformly from [lo, hi] first.
    ``values_device="cuda"``: the lengths, layout and peaky-row mask are drawn as
    above, but q, gate and the pools from a CUDA generator seeded with ``seed`` and
    left on the device (the same distributions, other values; seconds instead of a
    minute for the largest pools, for timing runs)."""
    if kv not in ("bf16", "e4m3"):
        raise ValueError(kv)
    gen = torch.Generator().manual_seed(seed)
    if random_lengths is not None:
        lo, hi, bsz = random_lengths
        lengths = torch.randint(lo, hi + 1, (bsz,), generator=gen).tolist()
    lengths = [int(L) for L in lengths]
    B = len(lengths)
    idx, slots = _layout(gen, lengths, layout, pool_slots, page)
    row_scale = None
    if peaky_frac > 0.0:
        picked = torch.rand(idx.numel(), generator=gen) < peaky_frac
        row_scale = torch.ones(slots, dtype=torch.float32)
        row_scale[idx[picked].long()] = peaky_scale
    if values_device is not None:
        gen = torch.Generator(device=values_device).manual_seed(seed)
    q = _randn_bf16(gen, B * hq, head_dim, qkv_std).view(B, hq, head_dim)
    g = _randn_bf16(gen, B * hq, head_dim, gate_std).view(B, hq, head_dim)
    k_scale = None
    if row_scale is not None:
        k_scale = row_scale.repeat_interleave(hkv)
    if kv == "e4m3":
        peak = peaky_scale if peaky_frac > 0.0 else 1.0
        k_descale = float(torch.tensor(6.0 * qkv_std * max(peak, 1.0) / E4M3_MAX, dtype=torch.float32))
        v_descale = float(torch.tensor(6.0 * qkv_std / E4M3_MAX, dtype=torch.float32))
        k_pool = _randn_e4m3(gen, slots * hkv, head_dim, qkv_std, k_descale, k_scale).view(slots, hkv, head_dim)
        v_pool = _randn_e4m3(gen, slots * hkv, head_dim, qkv_std, v_descale).view(slots, hkv, head_dim)
    else:
        k_descale = v_descale = 1.0
        k_pool = _randn_bf16(gen, slots * hkv, head_dim, qkv_std, k_scale).view(slots, hkv, head_dim)
        v_pool = _randn_bf16(gen, slots * hkv, head_dim, qkv_std).view(slots, hkv, head_dim)
    indptr = torch.zeros(B + 1, dtype=torch.int32)
    if B:
        indptr[1:] = torch.tensor(lengths, dtype=torch.int64).cumsum(0).to(torch.int32)
    return dict(q=q, gate=g, k_pool=k_pool, v_pool=v_pool, kv_indptr=indptr, kv_indices=idx,
                scale=float(scale), lengths=lengths, num_slots=slots, k_descale=k_descale,
                v_descale=v_descale, kv=kv)


def make_workload(key, batch_limit: Optional[int] = None, seed: Optional[int] = None, kv: str = "bf16",
                  values_device: Optional[str] = None) -> dict:
    """Inputs of one of the five named workloads (``batch_limit`` keeps the
    first sequences only, for bounded CPU timing; the draw is unchanged;
    ``seed`` replaces the workload's seed, e.g. for independent replicas;
    ``kv="e4m3"`` gives the same workload over an FP8 KV cache;
    ``values_device`` as in make())."""
    w = workload(key)
    rl = (w.len_lo, w.len_hi, w.batch) if w.lengths is None else None
    d = make(w.lengths if w.lengths is not None else [], seed=w.seed if seed is None else seed, hq=w.hq, hkv=w.hkv,
             head_dim=w.head_dim, layout=w.layout, pool_slots=w.pool_slots, page=w.page,
             gate_std=w.gate_std, peaky_frac=w.peaky_frac, scale=w.scale, random_lengths=rl, kv=kv,
             values_device=values_device)
    d["workload"] = w
    d["num_splits"] = w.num_splits
    if batch_limit is not None and batch_limit < len(d["lengths"]):
        d = truncate_batch(d, batch_limit)
    return d


def truncate_batch(d: dict, nb: int) -> dict:
    """Keep the first ``nb`` sequences of a batch (same pools)."""
    e = dict(d)
    nnz = int(d["kv_indptr"][nb])
    e["q"] = d["q"][:nb].contiguous()
    e["gate"] = d["gate"][:nb].contiguous()
    e["kv_indptr"] = d["kv_indptr"][:nb + 1].clone()
    e["kv_indices"] = d["kv_indices"][:nnz].clone()
    e["lengths"] = d["lengths"][:nb]
    return e


def metric_bytes(lengths: Sequence[int], hq: int = HQ, hkv: int = HKV, head_dim: int = HEAD_DIM,
                 kv_bytes: int = 2) -> int:
    """Algorithmic HBM bytes of one call: every referenced K and V row once
    (``kv_bytes`` per element: 2 for BF16, 1 for e4m3), plus q, gate and out."""
    n = int(sum(lengths))
    return n * hkv * head_dim * kv_bytes * 2 + 3 * len(lengths) * hq * head_dim * 2


# ------------------------------------------------------------------ prefill / extend

PREFILL_HQ, PREFILL_HKV = 32, 2


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    batch: int
    sq: int                 # query tokens per sequence
    skv: int                # key/value tokens per sequence (the queries are the last sq of them)
    causal: bool
    seed: int
    hq: int = PREFILL_HQ
    hkv: int = PREFILL_HKV
    head_dim: int = HEAD_DIM
    gate_std: float = 2.0


# The geometry of cuDNN FE-OSS "Gated Attention Block (SM107)", Performance: B=1,
# h_q=32, h_kv=2, d=256, causal and dense (no mask); the sequence lengths are
# this module's choice (the page's tables did not survive extraction).
PREFILL_WORKLOADS: List[PrefillWorkload] = [
    PrefillWorkload("p1_s4096_causal", 1, 4096, 4096, True, 10),
    PrefillWorkload("p1_s4096_dense", 1, 4096, 4096, False, 11),
    PrefillWorkload("p1_s512_causal", 1, 512, 512, True, 12),
    PrefillWorkload("p4_extend_q1024_kv8192", 4, 1024, 8192, True, 13),
]
PREFILL_BY_NAME = {w.name: w for w in PREFILL_WORKLOADS}


def make_prefill(batch: int, sq: int, skv: int, *, seed: int, hq: int = PREFILL_HQ, hkv: int = PREFILL_HKV,
                 head_dim: int = HEAD_DIM, gate_std: float = 2.0, qkv_std: float = 1.0,
                 scale: Optional[float] = None, causal: bool = True, kv_lens=None) -> dict:
    """Prefill / extend inputs on the CPU: q, gate [B, Sq, Hq, D] and k, v [B, Skv, Hkv, D]
    BF16 drawn from N(0, std^2) (draw order q, gate, k, v from one generator seeded
    with ``seed``), plus ``scale`` (1/sqrt(D) by default), ``causal`` and ``kv_lens``
    ([B] int32 or None)."""
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, batch * sq * hq, head_dim, qkv_std).view(batch, sq, hq, head_dim)
    g = _randn_bf16(gen, batch * sq * hq, head_dim, gate_std).view(batch, sq, hq, head_dim)
    k = _randn_bf16(gen, batch * skv * hkv, head_dim, qkv_std).view(batch, skv, hkv, head_dim)
    v = _randn_bf16(gen, batch * skv * hkv, head_dim, qkv_std).view(batch, skv, hkv, head_dim)
    kl = None if kv_lens is None else torch.tensor(list(kv_lens), dtype=torch.int32)
    return dict(q=q, gate=g, k=k, v=v, scale=float(scale if scale is not None else 1.0 / math.sqrt(head_dim)),
                causal=bool(causal), kv_lens=kl)


def make_prefill_workload(key: str, seed: Optional[int] = None) -> dict:
    w = PREFILL_BY_NAME[key]
    d = make_prefill(w.batch, w.sq, w.skv, seed=w.seed if seed is None else seed, hq=w.hq, hkv=w.hkv,
                     head_dim=w.head_dim, gate_std=w.gate_std, causal=w.causal)
    d["workload"] = w
    return d


def prefill_flops(batch: int, sq: int, skv: int, hq: int, head_dim: int, causal: bool, kv_lens=None) -> int:
    """Algorithmic FLOPs of one prefill call: 4 * D per visible (query, key) pair per
    query head (QK^T and PV, multiply-add = 2)."""
    total = 0
    for b in range(batch):
        L = skv if kv_lens is None else int(kv_lens[b])
        if causal:
            off = L - sq
            # visible keys of query i: min(L, max(0, i + off + 1))
            vis = sum(min(L, max(0, i + off + 1)) for i in range(sq))
        else:
            vis = sq * L
        total += vis
    return 4 * head_dim * hq * total
