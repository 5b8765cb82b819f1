"""Build and run a probe (needs a GPU):

    python -m gated_gqa_attention_gb300.microbench [gather|mma|tma|issue|paths|splits]

gather: how scattered K/V rows stream (16-byte loads, cp.async, 1-D bulk copies);
mma:    tcgen05.mma throughput per instruction shape (M = 128, N = 64 / 128 / 256,
        A from TMEM or shared memory, B K-major or MN-major);
tma:    tensor-map (cp.async.bulk.tensor) throughput for [64 x 256] BF16 tiles of an
        L2-resident [1, S, 2, 256] tensor through 2 / 4 / 6-stage rings;
issue:  how waits in the MMA-issuing thread stall the tensor pipe, and the attention
        mainloop's MMA schedules (64-key tiles, 128-key tiles with one or two issuers);
paths:  the decode's one-kernel cluster path against the split path over batch and
        length (decode_paths.py);
splits: every explicit split count against the automatic schedule per (batch, length)
        bucket (split_sweep.py; an optional second argument names a JSON output, or
        `cross` times uniform splits against the stream schedule near the rule's bounds)."""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
PROBES = {"gather": "gather_probe.cu", "mma": "mma_probe.cu", "tma": "tma_probe.cu", "issue": "issue_probe.cu"}


def main():
    which = sys.argv[1] if len(sys.argv) > 1 else "gather"
    if which == "paths":
        from gated_gqa_attention_gb300.microbench import decode_paths
        decode_paths.main()
        return
    if which == "splits":
        from gated_gqa_attention_gb300.microbench import split_sweep
        if len(sys.argv) > 2 and sys.argv[2] == "cross":
            split_sweep.crossover()
        else:
            split_sweep.main(sys.argv[2] if len(sys.argv) > 2 else None)
        return
    src = os.path.join(HERE, PROBES[which])
    exe = os.path.join(HERE, which + "_probe")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-o", exe, src],
                   check=True)
    sys.exit(subprocess.run([exe]).returncode)


if __name__ == "__main__":
    main()
