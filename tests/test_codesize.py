"""The layer kernel's code-size budget (CPU: compiles to a cubin and reads
the ELF section headers only).

The pages' per-layer kernels were 215-314 KB against an instruction cache of
about 128 KB per SM, with measurable slowdowns when code does not fit
([orcarouter] "Tre bollette che un kernel così grande deve pagare"); every
instantiation of ours must stay within the budget set in
moe_decode_step_persistent_gb300/codesize.py."""

import shutil

import pytest


@pytest.mark.skipif(shutil.which("nvcc") is None and not __import__("os").path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc not available")
def test_layer_kernel_within_code_budget():
    from moe_decode_step_persistent_gb300 import codesize as CS
    sizes = CS.kernel_text_sizes()
    assert len(sizes) == 4, sizes  # head_dim 64 / 128, timing on / off
    for name, size in sizes.items():
        assert size <= CS.BUDGET_BYTES, f"{name}: {size} bytes of code > budget {CS.BUDGET_BYTES}"


def test_section_reader_on_a_handmade_elf(tmp_path):
    """The header reader against an ELF64 file assembled by hand: two named
    sections of known sizes."""
    import struct
    from moe_decode_step_persistent_gb300 import codesize as CS
    names = b"\0.shstrtab\0.text.k1\0.text.k2\0"
    hdr = bytearray(64)
    hdr[:4] = b"\x7fELF"
    hdr[4] = 2
    body = names
    shoff = 64 + len(body)
    shoff += (-shoff) % 8
    struct.pack_into("<Q", hdr, 0x28, shoff)
    struct.pack_into("<HHH", hdr, 0x3A, 64, 4, 1)
    secs = [(0, 0, 0), (1, 64, len(names)), (11, 0, 1234), (20, 0, 98765)]
    sh = b"".join(struct.pack("<IIQQQQ", n, 1, 0, 0, off, size) + bytes(24) for n, off, size in secs)
    data = bytes(hdr) + body + bytes(shoff - 64 - len(body)) + sh
    p = tmp_path / "x.elf"
    p.write_bytes(data)
    got = CS.section_sizes(str(p))
    assert got[".text.k1"] == 1234 and got[".text.k2"] == 98765 and got[".shstrtab"] == len(names)
