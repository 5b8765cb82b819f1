"""Decode-path sweep (needs a GPU): for B in {1, 4, 8, 12, 16, 24, 32, 48, 64} and
equal lengths L in {128, 256, 512, 1024, 2048}, the µs per call of gda_decode_ex with the
length bound (the library picks the one-kernel cluster path when it applies), without
it (the split path, split count chosen on the device), and on the split path with the
bound and the batch's total (variant MMA, split count chosen on the host), each a CUDA
graph of 4 calls replayed; the cluster size gda_small_path_cluster chose is printed
beside them."""
import torch

import gated_gqa_attention_gb300 as gda
from gated_gqa_attention_gb300 import workloads


def _per_call_us(f, calls=200):
    for _ in range(5):
        f()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            for _ in range(4):
                f()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(calls // 4):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / calls * 1e3


def main():
    gda.load()
    print("%3s %5s %9s %12s %10s %13s %6s" % ("B", "L", "cluster C", "one-kernel", "split", "split (host)",
                                               "ratio"))
    for B in (1, 4, 8, 12, 16, 24, 32, 48, 64):
        for L in (128, 256, 512, 1024, 2048):
            inp = workloads.make([L] * B, seed=7, layout="perm", pool_slots=max(4096, B * L + 100))
            d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
            out = torch.empty_like(d["q"])
            _, Hq, D = d["q"].shape
            Hkv = d["k_pool"].shape[1]
            ws = torch.empty(gda.workspace_bytes(B, Hq, Hkv, D, 0), dtype=torch.uint8, device="cuda")
            gda.workspace_init(ws)
            t = {}
            for ml in (L, 0):
                t[ml] = _per_call_us(lambda: gda.decode_ex(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["kv_indptr"],
                                                           d["kv_indices"], out=out, workspace=ws, scale=inp["scale"],
                                                           max_len=ml))
            th = _per_call_us(lambda: gda.decode_ex(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["kv_indptr"],
                                                    d["kv_indices"], out=out, workspace=ws, scale=inp["scale"],
                                                    max_len=L, total_len=B * L, variant=gda.VARIANT_MMA))
            print("%3d %5d %9d %9.2f us %7.2f us %10.2f us %6.2f" % (B, L, gda.small_path_cluster(B * Hkv, L), t[L],
                                                                    t[0], th, t[L] / min(t[0], th)), flush=True)


if __name__ == "__main__":
    main()
