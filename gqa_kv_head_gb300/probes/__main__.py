"""Build memory_probe.cu for sm_103a and run it (needs a GPU)."""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "csrc")


def main():
    from ..build import ARCH, _nvcc
    out_dir = os.path.join(os.path.dirname(HERE), "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "memory_probe")
    cmd = [_nvcc(), *ARCH, "-O3", "-std=c++17", "-I", CSRC, os.path.join(HERE, "memory_probe.cu"), "-o", exe, "-lcuda"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        return 1
    return subprocess.run([exe]).returncode


if __name__ == "__main__":
    sys.exit(main())
