"""The C ABI library builds for sm_103a, loads without a GPU, and exports
every entry point include/moe.h declares (no compute call is made here)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libpath():
    from mixture_experts_ffn_histogram_gb300 import _build
    return _build.build()


def test_header_declares_the_block(libpath):
    names = declared_functions()
    for required in ("moe_route_histogram", "moe_permute", "moe_permute_bwd",
                     "moe_grouped_gemm_fc1_swiglu", "moe_grouped_gemm_fc1_swiglu_bwd",
                     "moe_grouped_gemm_fc2", "moe_grouped_gemm_fc2_bwd", "moe_combine",
                     "moe_combine_bwd", "moe_workspace_bytes", "moe_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"
    nm = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = set(re.findall(r"\bT (moe_[a-z0-9_]+)$", nm.stdout, flags=re.M))
        assert set(declared_functions()) <= exported


def test_binding_names_match_the_header(libpath):
    from mixture_experts_ffn_histogram_gb300 import binding
    assert set(binding.ENTRY_POINTS) == set(declared_functions())
    for n in declared_functions():
        if n != "moe_status_string":
            assert callable(getattr(binding, n))


def test_host_only_queries(libpath):
    from mixture_experts_ffn_histogram_gb300 import binding as B
    assert B.moe_abi_version() == 4
    d = B.dims(32768, 2816, 128, 8, 704)
    ws = B.moe_workspace_bytes(d)
    assert ws >= 32768 * 8 * 2 * 704 * 2 and ws % 256 == 0
    assert B.moe_workspace_bytes(B.dims(16, 100, 8, 2, 64)) == 0      # unsupported dims
    assert "expert id" in B.status_string(B.MOE_ERR_DEVICE)


def test_compiled_for_sm103a_only(libpath):
    from mixture_experts_ffn_histogram_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
