"""The C-ABI library: it builds, loads without a GPU and exports what include/vbs.h declares."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vbs.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?(?:int|char|void)\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def libpath():
    from verify_bs_step_gb300 import _build
    return _build.build()


def test_exports_match_header(libpath):
    names = header_functions()
    assert len(names) >= 24, names
    lib = ctypes.CDLL(libpath)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True, check=True)
    exported = {ln.split()[-1] for ln in out.stdout.splitlines() if " T " in ln}
    assert exported == set(names), exported ^ set(names)


def test_binding_declares_every_entry_point(libpath):
    import verify_bs_step_gb300 as vbs
    assert set(vbs.SIGNATURES) == set(header_functions())
    L = vbs.lib()
    assert L.vbs_version() == 100
    assert L.vbs_strerror(-1) == b"invalid argument"
    assert L.vbs_strerror(-3).startswith(b"out of memory")
    assert L.vbs_strerror(12345) == b"unknown status"


def test_host_checks_reject_bad_arguments_before_any_launch(libpath):
    import verify_bs_step_gb300 as vbs
    L = vbs.lib()
    ctx = ctypes.c_void_p()
    bad_inits = [
        (0, 4, 100), (2, 0, 100), (2, 17, 100), (2, 4, 1),         # batch, W (1..16), V >= 2
    ]
    for B, W, V in bad_inits:
        st = L.bs_init(ctypes.byref(ctx), B, W, V, -1, 0.6, 0, 0, 8, 0, -1, 1, None)
        assert st == vbs.EINVAL and ctx.value is None
    assert L.bs_init(ctypes.byref(ctx), 2, 4, 100, 100, 0.6, 0, 0, 8, 0, -1, 1, None) == vbs.EINVAL   # eos >= V
    assert L.bs_init(ctypes.byref(ctx), 2, 4, 100, 5, 0.6, 3, 0, 8, 0, -1, 1, None) == vbs.EINVAL     # mode
    assert L.bs_init(ctypes.byref(ctx), 2, 4, 100, 5, 0.6, 0, 2, 8, 0, -1, 1, None) == vbs.EINVAL     # lp kind
    assert L.bs_init(ctypes.byref(ctx), 2, 4, 100, 5, 0.6, 0, 0, 8, 0, -1, 7, None) == vbs.EINVAL     # dtype
    assert L.bs_init(ctypes.byref(ctx), 1 << 16, 16, 1 << 16, 5, 0.6, 0, 0, 8, 0, -1, 1, None) == vbs.EINVAL
    assert L.bs_step(None, None, 0, None, None, None, None, None) == vbs.EINVAL
    assert L.bs_destroy(None) == vbs.OK
    assert L.bpd_verify(None, None, 4, 0, 100, 1, -1, None, None, None, None) == vbs.EINVAL        # k = 0
    assert L.bpd_verify(None, None, 4, 33, 100, 1, -1, None, None, None, None) == vbs.EINVAL       # k > 32
    assert L.bpd_verify(None, None, 4, 8, 100, 1, -1, None, None, None, None) == vbs.EINVAL        # NULLs
    assert L.bpd_propose(None, 0, 4, 100, 1, None, None) == vbs.OK                                 # empty batch
    assert L.kv_reorder(None, None, None, None, 4, 1, None) == vbs.EINVAL
    assert L.kv_paged_init(ctypes.byref(ctx), None, 1, 1, 1, 16, 1, None, None) == vbs.EINVAL
