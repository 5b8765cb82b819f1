"""Build and run the gather probe (needs a GPU): python -m gated_gqa_attention_gb300.microbench"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))


def main():
    src = os.path.join(HERE, "gather_probe.cu")
    exe = os.path.join(HERE, "gather_probe")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-o", exe, src],
                   check=True)
    sys.exit(subprocess.run([exe]).returncode)


if __name__ == "__main__":
    main()
