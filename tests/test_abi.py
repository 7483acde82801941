"""The C ABI without a GPU: the library builds, loads and exports every entry
point include/moe_layout.h declares; host-only calls agree with the oracle."""
import ctypes
import os
import re
import subprocess

import pytest

import oracle
from combine_moe_layout_gb300 import _binding as B
from combine_moe_layout_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_layout.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("moe_buffer_sizes", "moe_layout", "moe_dispatch", "moe_layout_dispatch", "moe_combine",
              "moe_get_error", "moe_reset"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(_build.build())
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} is declared but not exported"
    nm = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = set(re.findall(r"\bT (moe_\w+)", nm.stdout))
        assert set(declared_functions()) <= exported


def test_every_declared_entry_point_has_a_python_name():
    """The binding calls each C entry point by its own name, and the package exports it."""
    import combine_moe_layout_gb300 as pkg
    for name in declared_functions():
        assert callable(getattr(B, name, None)), f"{name} has no binding"
        assert getattr(pkg, name, None) is getattr(B, name), f"{name} is not exported by the package"


def test_library_is_built_for_sm_103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)


@pytest.mark.parametrize("shape", [
    (2, 16, 128, 8, 2, 16, 0), (8, 128, 7168, 256, 8, 128, 1), (8, 4096, 4096, 8, 2, 4096, 0),
    (16, 256, 7168, 256, 8, 256, 0), (8, 4096, 7168, 256, 8, 4096, 1), (64, 128, 7168, 256, 8, 128, 1),
    (8, 128, 7168, 256, 8, 128, 2),
])
def test_buffer_sizes_agree_with_the_oracle(shape):
    R, T, H, E, k, M, dt = shape
    got = B.moe_buffer_sizes(B.MoeDesc(R, T, H, E, k, M, dt, 0))
    want = oracle.buffer_sizes(R, T, H, E, k, M, dt)
    assert got == want


@pytest.mark.parametrize("shape", [
    (3, 16, 128, 8, 2, 16, 0),    # E % R
    (2, 17, 128, 8, 2, 16, 0),    # T > max_m
    (2, 16, 130, 8, 2, 16, 0),    # bf16 row not whole 16-byte vectors
    (2, 16, 192, 8, 2, 16, 1),    # fp8 hidden not whole 128-element blocks
    (2, 16, 128, 8, 9, 16, 0),    # k > E
    (2, 16, 128, 64, 17, 16, 0),  # k > 16
    (2, 16, 128, 8, 2, 16, 3),    # unknown dtype
    (2, 16, 192, 8, 2, 16, 2),    # bf16 rows quantised on dispatch need whole 128-element blocks
    (0, 16, 128, 8, 2, 16, 0),    # no ranks
])
def test_invalid_descs_are_rejected_on_the_host(shape):
    R, T, H, E, k, M, dt = shape
    with pytest.raises(B.MoeError) as e:
        B.moe_buffer_sizes(B.MoeDesc(R, T, H, E, k, M, dt, 0))
    assert e.value.status == B.MOE_EINVAL


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5):
        assert B.moe_status_string(code) != "unknown status"
    assert B.moe_status_string(99) == "unknown status"


def test_fused_kernel_count_is_a_host_query():
    decode = B.MoeDesc(8, 128, 7168, 256, 8, 128, 1, 0)
    prefill = B.MoeDesc(8, 4096, 7168, 256, 8, 4096, 1, 0)
    assert B.moe_layout_dispatch_kernels(decode) == 1
    assert B.moe_layout_dispatch_kernels(prefill) == 2
    assert B.moe_layout_dispatch_kernels(B.MoeDesc(8, 0, 7168, 256, 8, 128, 1, 0)) == 1
