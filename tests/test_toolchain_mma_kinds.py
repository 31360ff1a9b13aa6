"""Which tcgen05.mma kinds the toolchain accepts for sm_103a (compile only, no GPU).

Evidence behind two scope decisions:
  * the W4A8 variant of "W4A8量化计算优化" §2.1-§3.2 (LiquidQuant: 4-bit weights turned
    into int8 by one IMAD and one XOR, then an int8 x int8 -> int32 tensor-core GEMM)
    needs the int8 MMA, tcgen05.mma.kind::i8; ptxas rejects that kind for sm_103a, so the
    variant cannot be built on this GPU;
  * the block-scaled FP4 kinds that "量化开销对比" §5 calls Blackwell's native route A
    (MXFP4 / NVFP4, a hardware block-32 E8M0 scale) are accepted, as is kind::f16, the
    kind every kernel of this library uses.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

NVCC = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"

_HEAD = "#include <cstdint>\n"
_MMA = {
    "f16": "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;",
    "i8": "tcgen05.mma.cta_group::1.kind::i8 [%0], %1, %2, %3, p;",
}
_MMA_BS = {
    "mxf8f6f4": "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;",
    "mxf4": "tcgen05.mma.cta_group::1.kind::mxf4.block_scale [%0], %1, %2, %3, [%4], [%5], p;",
    "mxf4nvf4": ("tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
                 "[%0], %1, %2, %3, [%4], [%5], p;"),
}


def _kernel(kind):
    if kind in _MMA:
        return (_HEAD + "__global__ void k(uint32_t d, uint64_t a, uint64_t b, uint32_t i) {\n"
                "  asm volatile(\"{\\n\\t.reg .pred p;\\n\\tsetp.ne.b32 p, %4, 0;\\n\\t"
                + _MMA[kind] + "\\n\\t}\" :: \"r\"(d), \"l\"(a), \"l\"(b), \"r\"(i), \"r\"(1));\n}\n")
    return (_HEAD + "__global__ void k(uint32_t d, uint64_t a, uint64_t b, uint32_t i, uint32_t sa,"
            " uint32_t sb) {\n"
            "  asm volatile(\"{\\n\\t.reg .pred p;\\n\\tsetp.ne.b32 p, %6, 0;\\n\\t"
            + _MMA_BS[kind] + "\\n\\t}\" :: \"r\"(d), \"l\"(a), \"l\"(b), \"r\"(i), \"r\"(sa), "
            "\"r\"(sb), \"r\"(1));\n}\n")


def _compile(kind):
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "k.cu")
        open(src, "w").write(_kernel(kind))
        r = subprocess.run([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-c", src, "-o",
                            os.path.join(d, "k.o")], capture_output=True, text=True)
        return r.returncode, r.stdout + r.stderr


pytestmark = pytest.mark.skipif(not os.path.exists(NVCC), reason="nvcc not available")


@pytest.mark.parametrize("kind", ["f16", "mxf8f6f4", "mxf4", "mxf4nvf4"])
def test_kind_is_accepted_for_sm103a(kind):
    rc, out = _compile(kind)
    assert rc == 0, out


def test_int8_kind_is_rejected_for_sm103a():
    rc, out = _compile("i8")
    assert rc != 0
    assert ".kind::i8" in out and "sm_103a" in out and "not supported" in out, out
