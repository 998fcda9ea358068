"""Builds and runs the one-GPU microbenchmarks (msk_micro.cu) and prints
their JSON lines.

  python -m moe_decode_step_persistent_gb300.micro.run [--out FILE]

The instruction-cache kernels are generated into _build/ (gen_bodies.py);
one nvcc invocation for sm_103a; the program prints one JSON object per
probe."""

from __future__ import annotations

import argparse
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")


def nvcc() -> str:
    env = os.environ.get("NVCC")
    if env:
        return env
    return "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"


def build() -> str:
    os.makedirs(BUILD, exist_ok=True)
    bodies = os.path.join(BUILD, "icache_bodies.cuh")
    subprocess.run([sys.executable, os.path.join(HERE, "gen_bodies.py"), bodies], check=True)
    exe = os.path.join(BUILD, "msk_micro")
    cmd = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-I", BUILD,
           os.path.join(HERE, "msk_micro.cu"), "-o", exe]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout.decode(errors="replace"))
    return exe


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--out", default=None, help="also write the JSON lines to this file")
    p.add_argument("--build-only", action="store_true")
    args = p.parse_args(argv)
    exe = build()
    if args.build_only:
        print(exe)
        return 0
    r = subprocess.run([exe], stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    out = r.stdout.decode(errors="replace")
    sys.stdout.write(out)
    if args.out:
        with open(args.out, "w") as f:
            f.write(out)
    return r.returncode


if __name__ == "__main__":
    sys.exit(main())
