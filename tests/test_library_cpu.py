"""CPU checks of the library boundary: the shared library builds, loads
without a GPU and exports every entry point the header declares; the Python
package refuses to import without it; the binding validates arguments before
touching the library."""

import os
import re
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "txl_relattn.h")
PKG = os.path.join(ROOT, "transformer_xl_relative_txl_gb300")
LIB = os.path.join(PKG, "libtxl_relattn.so")


def _build_if_missing():
    if not os.path.exists(LIB):
        sys.path.insert(0, ROOT)
        import importlib.util

        spec = importlib.util.spec_from_file_location("txl_build", os.path.join(PKG, "build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:TXL_API\s+)?(?:int|size_t|const char\*|txl_status)\s+(txl_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("txl_relattn_forward", "txl_relattn_forward_static", "txl_relattn_forward_roll",
              "txl_relattn_backward", "txl_mem_update",
              "txl_sinusoid_rel",
              "txl_get_device_status",
              "txl_status_string", "txl_version"):
        assert n in names


def test_library_exports_every_declared_symbol():
    _build_if_missing()
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    import ctypes

    lib = ctypes.CDLL(LIB)
    for n in declared_functions():
        getattr(lib, n)
    lib.txl_version.restype = ctypes.c_int
    assert lib.txl_version() == 150
    lib.txl_status_string.restype = ctypes.c_char_p
    assert lib.txl_status_string(5) == b"TXL_ERR_DEVICE_TIMEOUT"


def test_package_import_fails_loudly_without_library(tmp_path):
    dst = tmp_path / "transformer_xl_relative_txl_gb300"
    shutil.copytree(PKG, dst, ignore=shutil.ignore_patterns("*.so", "__pycache__", "csrc"))
    code = "import transformer_xl_relative_txl_gb300"
    res = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True)
    assert res.returncode != 0 and "ImportError" in res.stderr


def test_binding_rejects_host_tensors_before_calling():
    _build_if_missing()
    import torch

    import transformer_xl_relative_txl_gb300 as txl

    q = torch.zeros(1, 4, 2, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    r = torch.zeros(8, 2, 64, dtype=torch.bfloat16)
    u = torch.zeros(2, 64)
    with pytest.raises(ValueError):
        txl.txl_relattn_forward(q, k, k, r, u, u, q.clone())
    with pytest.raises(ValueError):
        txl.txl_relattn_forward(q, k[:, :5], k, r, u, u, q.clone())
