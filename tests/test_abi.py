"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports
every function include/ep.h declares, and rejects bad arguments before any
CUDA call."""
import ctypes
import os
import re

import pytest

from combine_ep_get_03_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = cuda_build.build()
    return ctypes.CDLL(path)


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(ep_\w+)\s*\(", text))
    return names


def test_header_declares_the_boundary():
    assert {"ep_handle_create", "ep_handle_destroy", "ep_get_dispatch_layout", "ep_get_num_recv", "ep_dispatch",
            "ep_combine", "ep_low_latency_dispatch", "ep_low_latency_combine", "ep_get_device_status",
            "ep_status_str"} <= _declared()


def test_every_declared_symbol_is_exported(lib):
    for name in sorted(_declared()):
        assert hasattr(lib, name), name


def test_status_strings(lib):
    lib.ep_status_str.restype = ctypes.c_char_p
    assert [lib.ep_status_str(i).decode() for i in range(7)] == [
        "EP_OK", "EP_ERR_INVALID_ARG", "EP_ERR_CUDA", "EP_ERR_CAPACITY", "EP_ERR_BAD_EXPERT", "EP_ERR_TIMEOUT",
        "EP_ERR_STATE"]


def test_argument_checks_precede_cuda(lib):
    out = ctypes.c_void_p()
    create = lib.ep_handle_create
    create.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_void_p)]
    for args in [(0, 16, 2, 512, 8), (4, 18, 2, 512, 8), (4, 16, 0, 512, 8), (4, 16, 33, 512, 8),
                 (4, 16, 2, 500, 8), (4, 16, 2, 512, 0), (2048, 2048, 2, 512, 8)]:
        assert create(*args, ctypes.byref(out)) == 1, args
        assert out.value is None
    assert create(4, 16, 2, 512, 8, None) == 1
    # NULL handles
    for name in ("ep_get_dispatch_layout", "ep_dispatch", "ep_combine", "ep_low_latency_dispatch",
                 "ep_low_latency_combine", "ep_get_device_status", "ep_get_num_recv", "ep_check_wait_timeout"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        nargs = {"ep_get_dispatch_layout": 7, "ep_dispatch": 12, "ep_combine": 6, "ep_low_latency_dispatch": 11,
                 "ep_low_latency_combine": 6, "ep_get_device_status": 2, "ep_get_num_recv": 5,
                 "ep_check_wait_timeout": 2}[name]
        fn.argtypes = [ctypes.c_void_p] * nargs
        assert fn(*([None] * nargs)) == 1, name
    lib.ep_handle_destroy.argtypes = [ctypes.c_void_p]
    assert lib.ep_handle_destroy(None) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from combine_ep_get_03_gb300 import ep
    monkeypatch.setattr(ep, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(ep, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        ep.lib()


def test_header_is_plain_c_and_links(tmp_path):
    """include/ep.h compiles as C99 (no C++ in the boundary) and a C program
    links against the library and calls its host-only entry points."""
    import subprocess
    path = cuda_build.build()
    src = tmp_path / "use_ep.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "ep.h"
int main(void) {
  int64_t rows = 0, bytes = 0;
  ep_status_t st = ep_get_buffer_size_hint(8, 256, 8, 7168, 1024, EP_FP8_E4M3, EP_LAYOUT_EXPERT_MAJOR, 128,
                                           &rows, &bytes);
  if (st != EP_OK || rows != 8192LL * 8 + 256LL * 127) return 1;
  if (strcmp(ep_status_str(EP_ERR_CAPACITY), "EP_ERR_CAPACITY") != 0) return 2;
  if (ep_handle_destroy(NULL) != EP_OK) return 3;
  if (ep_handle_topk_idx_bits(NULL) != 0) return 4;
  printf("ok %lld %lld\n", (long long)rows, (long long)bytes);
  return 0;
}
''')
    exe = tmp_path / "use_ep"
    libdir = os.path.dirname(path)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
           "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(path), "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.startswith("ok "), (r.returncode, r.stdout, r.stderr)
