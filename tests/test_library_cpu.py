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
    assert lib.txl_version() == 160
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


def _split_model(nqt, bh, W, M, sms):
    """The pair kernel's split choice restated: CTAs start in launch order on
    the SM that frees first (whole units longest query tile first, then the
    halves of the split tiles' units); a CTA costs its key steps plus 3; the
    count k of split tiles (0 to 2, halves of at least two steps) with the
    shortest launch wins, the smaller k on a tie."""
    import heapq

    def steps(qt):
        return min(M + 128 * qt + 127, M + W - 1) // 64 + 1

    def span(k):
        loads = [0] * sms
        heapq.heapify(loads)
        costs = [3 + steps(qt) for qt in range(nqt - k - 1, -1, -1) for _ in range(bh)]
        for j in range(2 * k):
            n = steps(nqt - 1 - j // 2)
            costs += [3 + (n - n // 2 if j % 2 else n // 2)] * bh
        for c in costs:
            heapq.heappush(loads, heapq.heappop(loads) + c)
        return max(loads)

    best, best_span = 0, span(0)
    for k in range(1, min(nqt, 2) + 1):
        if steps(nqt - k) < 4:
            break
        v = span(k)
        if v < best_span:
            best, best_span = k, v
    return best


def test_pair_kernel_split_choice():
    """The backward pair kernel's host-side split choice (test hook, no GPU
    needed) against the list-scheduling model it is defined by, over the
    bench's workloads and a grid of small shapes."""
    _build_if_missing()
    import ctypes

    lib = ctypes.CDLL(LIB)
    f = lib.txl_debug_pair_split_tiles
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 5
    # the bench's workloads: wide splits its last query tile, base does not
    assert f(6, 64, 768, 768, 152) == 1
    assert f(4, 176, 512, 512, 152) == 0
    assert f(1, 64, 128, 1600, 152) == 1
    cases = [(nqt, bh, W, M, sms) for nqt, W in ((1, 100), (2, 200), (3, 300), (4, 512), (6, 768))
             for bh in (1, 7, 64, 200) for M in (0, 8, 512, 1600) for sms in (148, 152)]
    for nqt, bh, W, M, sms in cases:
        got = f(nqt, bh, W, M, sms)
        assert got == _split_model(nqt, bh, W, M, sms), (nqt, bh, W, M, sms, got)
        assert 0 <= got <= min(nqt, 2)
    assert f(-1, 1, 1, 0, 152) == -1 and f(1, 1, 1, 0, 0) == -1


C_CALLER = r"""
#include <stdio.h>
#include "txl_relattn.h"

int main(void) {
  int stride = 0, table[64];
  /* host-only calls: no device is touched */
  int plan = txl_debug_unit_plan(2, 2, 300, 37, 5, table, 64, &stride);
  printf("%d %s %d %d %d %d\n", txl_version(), txl_status_string(TXL_ERR_ALIAS),
         txl_debug_pair_split_tiles(6, 64, 768, 768, 152), plan, stride, table[0]);
  return 0;
}
"""


def test_header_serves_a_c_program(tmp_path):
    """The boundary is a C ABI: the header compiles as C99 with all warnings
    and a C program links against the library and calls it (host-only entry
    points, so no GPU is needed)."""
    _build_if_missing()
    gcc = shutil.which("gcc") or pytest.skip("no C compiler")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, str(src), "-o", str(exe), "-L", PKG, "-ltxl_relattn",
                    "-Wl,-rpath," + PKG], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    import transformer_xl_relative_txl_gb300 as txl

    assert int(out[0]) == txl.txl_version()
    assert out[1] == txl.txl_status_string(3)
    assert out[2:] == ["1", "0", "4", "0"]  # split choice at wide; plan rows of 3 units + the -1
