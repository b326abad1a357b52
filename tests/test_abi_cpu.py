"""Host-side checks of the C-ABI library: it builds, loads, exports every
symbol include/q1gemv.h declares, and rejects bad arguments before touching a
device.  No call here launches a kernel (no GPU needed)."""
import ctypes
import os
import re

import pytest

from decode_q1_gemv_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q1gemv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z][a-z0-9_]*)\s*\(", text)) - {"defined"})


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    assert set(binding.EXPORTS) == set(names), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_library_exports_are_c_symbols():
    """nm -D shows the entry points unmangled (extern "C")."""
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in syms, name


@pytest.mark.parametrize("rows,n,expect", [
    (1, 128, 256 * 4 * 18),           # rows pad to a 256-row panel group, blocks to 4
    (32, 1024, 256 * 8 * 18),
    (257, 1024, 512 * 8 * 18),
    (4096, 4096, 4096 * 32 * 18),     # exactly 18 bytes per 128 weights
    (4096, 14336, 4096 * 112 * 18),
    (128256, 4096, 128256 * 32 * 18),
    (100, 640, 256 * 8 * 18),         # 5 blocks pad to 8
])
def test_packed_bytes(lib, rows, n, expect):
    assert binding.packed_bytes(rows, n) == expect


@pytest.mark.parametrize("rows,n", [(0, 128), (-1, 128), (1, 0), (1, 64), (1, 200), (1, 1 << 25), (1 << 27, 128)])
def test_packed_bytes_rejects_bad_shapes(lib, rows, n):
    with pytest.raises(binding.Q1Error):
        binding.packed_bytes(rows, n)
    assert "bad shape" in binding.last_error()


def test_null_pointers_rejected_on_host(lib):
    """Argument checks run on the host and return Q1_ERR_ARG with a message."""
    assert lib.q1_0_pack(None, 4, 128, None, None) == binding.Q1_ERR_ARG
    assert "q1_0_pack" in binding.last_error()
    assert lib.q1_0_gemv(None, 4, 128, None, None, None, None) == binding.Q1_ERR_ARG
    assert "q1_0_gemv" in binding.last_error()
    assert lib.q1_0_gemm_small(None, 4, 128, 3, None, None, None, None) == binding.Q1_ERR_ARG
    assert lib.q8_quantize_act(None, 1, 128, None, None, None) == binding.Q1_ERR_ARG
    assert lib.q1_0_unpack(None, 4, 128, None, None) == binding.Q1_ERR_ARG


def test_shape_limits_rejected_on_host(lib):
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the shape check fails first
    assert lib.q1_0_gemv(fake, 4, 100, fake, fake, fake, None) == binding.Q1_ERR_ARG
    assert lib.q1_0_gemm_small(fake, 4, 128, 0, fake, fake, fake, None) == binding.Q1_ERR_ARG
    assert lib.q1_0_gemm_small(fake, 4, 128, 65, fake, fake, fake, None) == binding.Q1_ERR_ARG
    assert "nvec" in binding.last_error()
    assert lib.q8_quantize_act(fake, 1, 48, fake, fake, None) == binding.Q1_ERR_ARG


def test_misaligned_pointers_rejected_on_host(lib):
    ok = ctypes.c_void_p(0x10000)
    bad = ctypes.c_void_p(0x10004)
    assert lib.q1_0_gemv(bad, 4, 128, ok, ok, ok, None) == binding.Q1_ERR_ARG
    assert "aligned" in binding.last_error()
    assert lib.q1_0_gemv(ok, 4, 128, ok, ok, bad, None) == binding.Q1_ERR_ARG
    assert lib.q1_0_pack(ctypes.c_void_p(0x10001), 4, 128, ok, None) == binding.Q1_ERR_ARG


def test_oracle_and_library_share_no_code():
    """The library sources never include or name the oracle, and vice versa."""
    csrc = os.path.join(ROOT, "decode_q1_gemv_gb300", "csrc")
    for fn in os.listdir(csrc):
        text = open(os.path.join(csrc, fn)).read()
        assert "oracle" not in text.lower(), fn
        assert "q1o_" not in text, fn
    pkg = os.path.join(ROOT, "decode_q1_gemv_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            text = open(os.path.join(pkg, fn)).read()
            assert "import oracle" not in text and "from oracle" not in text, fn
    otext = open(os.path.join(ROOT, "oracle", "q1_oracle.c")).read()
    assert "#include \"" not in otext
    otext_py = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert "import decode_q1_gemv_gb300" not in otext_py and "from decode_q1_gemv_gb300" not in otext_py
