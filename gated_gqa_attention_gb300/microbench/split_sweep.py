"""Split-count sweep (needs a GPU): for batches of B equal-length sequences, B in
{1, 2, 4, 8, 16, 32, 64, 128} and L in {512, 2048, 8192, 32768} (B * L at most 2^21
positions), the µs per call of gda_decode_ex with every explicit split count
S in {1, 2, 4, ..., 128}, with the automatic schedule (num_splits = 0, no length
bound: stage 1 + stage 2, the rule applied to kv_indptr on the device), and with
the library's full dispatch (automatic, the batch's longest length and its total
passed: the one-kernel cluster path where it applies, else the rule applied on the
host and uniform splits launched as explicit ones).  Each is a CUDA graph of 4
calls, replayed.  The table gives, per bucket, the argmin over S and the automatic
schedule's time against it: the measured basis of the split choice ("chosen per
(B, length) from measured time", FreeToken PR #781, Performance).

Inputs are made on the device from seeded generators (N(0, 1) q, gate and K/V rows,
slots a random permutation of the pool), Hq = 16, Hkv = 2, D = 256: timing only.

    python -m gated_gqa_attention_gb300.microbench splits [out.json]
    python -m gated_gqa_attention_gb300.microbench splits cross    (the crossover table)
"""
import json
import sys

import torch

import gated_gqa_attention_gb300 as gda
from gated_gqa_attention_gb300.microbench.decode_paths import _per_call_us

HQ, HKV, D = 16, 2, 256
SPLITS = (1, 2, 4, 8, 16, 32, 64, 128)
MAX_POSITIONS = 1 << 21


def _batch(B, L, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    n = B * L
    slots = n + 64
    mk = lambda *s: torch.randn(*s, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    q, gate = mk(B, HQ, D), mk(B, HQ, D)
    k_pool, v_pool = mk(slots, HKV, D), mk(slots, HKV, D)
    indptr = (torch.arange(B + 1, device="cuda", dtype=torch.int64) * L).to(torch.int32)
    indices = torch.randperm(slots, generator=g, device="cuda")[:n].to(torch.int32)
    return q, gate, k_pool, v_pool, indptr, indices


def main(out_path=None):
    gda.load()
    rows = []
    print("%4s %6s | %s | %9s %9s %6s | %9s" % ("B", "L", " ".join("%8s" % ("S=%d" % s) for s in SPLITS), "best S",
                                                "auto", "a/best", "dispatch"))
    for B in (1, 2, 4, 8, 16, 32, 64, 128):
        for L in (512, 2048, 8192, 32768):
            if B * L > MAX_POSITIONS:
                continue
            q, gate, kp, vp, indptr, idx = _batch(B, L, seed=1000 + B + L)
            out = torch.empty_like(q)
            t = {}
            for S in SPLITS + (0,):
                ws = torch.empty(gda.workspace_bytes(B, HQ, HKV, D, S), dtype=torch.uint8, device="cuda")
                gda.workspace_init(ws)
                t[S] = _per_call_us(lambda: gda.decode_ex(q, gate, kp, vp, indptr, idx, out=out, workspace=ws,
                                                          scale=D ** -0.5, num_splits=S), calls=100)
            ws = torch.empty(gda.workspace_bytes(B, HQ, HKV, D, 0), dtype=torch.uint8, device="cuda")
            gda.workspace_init(ws)
            disp = _per_call_us(lambda: gda.decode_ex(q, gate, kp, vp, indptr, idx, out=out, workspace=ws,
                                                      scale=D ** -0.5, max_len=L, total_len=B * L), calls=100)
            best = min(SPLITS, key=lambda s: t[s])
            row = {"B": B, "L": L, "us_by_splits": {str(s): round(t[s], 3) for s in SPLITS},
                   "best_splits": best, "best_us": round(t[best], 3), "auto_us": round(t[0], 3),
                   "dispatch_us": round(disp, 3), "cluster": gda.small_path_cluster(B * HKV, L)}
            rows.append(row)
            print("%4d %6d | %s | %4d %4.1f %9.2f %6.3f | %9.2f" % (
                B, L, " ".join("%8.2f" % t[s] for s in SPLITS), best, t[best], t[0], t[0] / t[best], disp), flush=True)
            del q, gate, kp, vp, indptr, idx, out, ws
            torch.cuda.empty_cache()
    if out_path:
        with open(out_path, "w") as f:
            json.dump(rows, f, indent=1)



# Where uniform splits and the stream schedule cross: (B, L, S) with S the one-wave
# uniform count, timed against the automatic schedule (the stream there)
CROSS = [(64, 3072, 1), (64, 4096, 1), (64, 5120, 1), (64, 6144, 1), (32, 6144, 2), (32, 8192, 2), (32, 10240, 2),
         (16, 12288, 4), (16, 16384, 4), (16, 20480, 4), (8, 2048, 8), (8, 2048, 9), (8, 32768, 8), (8, 32768, 9),
         (4, 2048, 16), (4, 2048, 19), (4, 32768, 16), (4, 32768, 19), (2, 32768, 32), (2, 32768, 38),
         (1, 32768, 64), (1, 32768, 76), (48, 4096, 1), (48, 8192, 1), (24, 8192, 3), (24, 8192, 2)]


def crossover():
    """Explicit uniform splits against the automatic schedule around the rule's bounds
    (positions per CTA near 3072; the power of two below the wave bound against the
    bound itself; waves that leave CTAs idle)."""
    gda.load()
    for B, L, S in CROSS:
        q, gate, kp, vp, indptr, idx = _batch(B, L, seed=5)
        out = torch.empty_like(q)
        t = {}
        for s in (0, S):
            ws = torch.empty(gda.workspace_bytes(B, HQ, HKV, D, s), dtype=torch.uint8, device="cuda")
            gda.workspace_init(ws)
            t[s] = _per_call_us(lambda: gda.decode_ex(q, gate, kp, vp, indptr, idx, out=out, workspace=ws,
                                                      scale=D ** -0.5, num_splits=s), calls=200)
        print("B %3d L %6d per-CTA %6d | auto %8.2f | S=%3d %8.2f | S/auto %.3f" % (
            B, L, (HKV * B * L + 151) // 152, t[0], S, t[S], t[S] / t[0]), flush=True)
        del q, gate, kp, vp, indptr, idx, out, ws
        torch.cuda.empty_cache()


if __name__ == "__main__":
    if len(sys.argv) > 1 and sys.argv[1] == "cross":
        crossover()
    else:
        main(sys.argv[1] if len(sys.argv) > 1 else None)
