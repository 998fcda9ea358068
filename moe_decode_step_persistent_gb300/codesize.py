"""Code size of the layer kernel, per instantiation, against a budget.

The pages warn that a kernel this large pays an instruction-cache bill: the
SM's instruction cache holds about 128 KB while their per-layer kernels are
215-314 KB, and a launch that runs each phase once fetches each phase's code
from L2 ([orcarouter] "Tre bollette che un kernel così grande deve pagare").
This module measures ours without reading any instruction: it compiles the
layer kernel's translation unit to a cubin with the library's own flags and
reads the ELF section headers, whose `.text.<kernel>` sizes are the bytes of
code of each kernel instantiation (all phase functions of a launch are in
it).  Nothing else of the cubin is read.

  python -m moe_decode_step_persistent_gb300.codesize      # prints the table
"""

from __future__ import annotations

import json
import os
import struct
import subprocess
import sys

from . import build as B

CUBIN = os.path.join(B.LIBDIR, "msk_layer.cubin")

#: budget per layer-kernel instantiation, bytes of .text
BUDGET_BYTES = 240 * 1024


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(os.path.join(B.CSRC, f)) > t for f in os.listdir(B.CSRC))


def compile_cubin(force: bool = False) -> str:
    """nvcc -cubin of csrc/msk_layer.cu with the library's flags."""
    if force or _stale(CUBIN):
        os.makedirs(B.LIBDIR, exist_ok=True)
        cmd = [B.nvcc(), *B.ARCH, *[f for f in B.FLAGS if f not in ("-Xcompiler", "-fPIC")], "-cubin",
               os.path.join(B.CSRC, "msk_layer.cu"), "-o", CUBIN + ".tmp"]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout.decode(errors='replace')}")
        os.replace(CUBIN + ".tmp", CUBIN)
    return CUBIN


def section_sizes(path: str) -> dict:
    """{section name: size} from the ELF64 section header table."""
    with open(path, "rb") as f:
        b = f.read()
    if b[:4] != b"\x7fELF" or b[4] != 2:
        raise ValueError(f"{path}: not an ELF64 file")
    shoff = struct.unpack_from("<Q", b, 0x28)[0]
    shentsize, shnum, shstrndx = struct.unpack_from("<HHH", b, 0x3A)
    hdrs = [struct.unpack_from("<IIQQQQ", b, shoff + i * shentsize) for i in range(shnum)]
    stroff = hdrs[shstrndx][4]
    out = {}
    for name, _typ, _flags, _addr, _off, size in hdrs:
        end = b.index(b"\0", stroff + name)
        out[b[stroff + name:end].decode()] = size
    return out


def kernel_text_sizes(force: bool = False) -> dict:
    """{kernel instantiation (mangled name): .text bytes} of the layer kernel."""
    secs = section_sizes(compile_cubin(force))
    return {n[len(".text."):]: s for n, s in secs.items() if n.startswith(".text.") and "msk_layer_kernel" in n}


def main(argv=None):
    sizes = kernel_text_sizes(force="--force" in (argv or sys.argv[1:]))
    for name, size in sorted(sizes.items()):
        print(f"{size:8d} B  {size / 1024:7.1f} KB  {'OK ' if size <= BUDGET_BYTES else 'OVER'}  {name}")
    print(json.dumps({"budget_bytes": BUDGET_BYTES, "text_bytes": sizes}))


if __name__ == "__main__":
    main()
