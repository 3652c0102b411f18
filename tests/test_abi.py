"""The C-ABI library loads without a GPU, exports every entry point that
include/pps.h declares, and rejects malformed arguments before touching the
device."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(pps_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("pps_kv_append", "pps_attn_plan", "pps_attn_run", "pps_plan_destroy"):
        assert want in names


def test_every_declared_symbol_is_exported(pps):
    lib = pps.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings_and_version(pps):
    assert pps.status_string(0) == "ok"
    for code in range(-7, 0):
        assert pps.status_string(code) != "unknown status"
    assert pps.version() >= 100


def _tiny_tables():
    q_indptr = np.array([0, 1, 3], np.int32)
    kv_len = np.array([5, 20], np.int32)
    page_indptr = np.array([0, 1, 3], np.int32)
    page_indices = np.array([0, 1, 2], np.int32)
    return q_indptr, kv_len, page_indptr, page_indices


@pytest.mark.parametrize("mutate,err", [
    (lambda t: t[1].__setitem__(0, 0), "invalid argument"),          # kv_len < q_len
    (lambda t: t[3].__setitem__(2, 9), "malformed page table"),      # page id out of range
    (lambda t: t[1].__setitem__(1, 40), "malformed page table"),     # page list too short
    (lambda t: t[0].__setitem__(1, 4), "invalid argument"),          # q_indptr not monotone
])
def test_plan_rejects_malformed_tables(pps, mutate, err):
    t = [a.copy() for a in _tiny_tables()]
    mutate(t)
    with pytest.raises(pps.PPSError, match=err):
        pps.attn_plan(*t, 8, 2, 64, 16, 4)


def test_plan_rejects_unsupported_shapes(pps):
    t = _tiny_tables()
    for hq, hkv, d, p in [(8, 2, 96, 16), (8, 2, 64, 24), (12, 1, 64, 16), (8, 3, 64, 16)]:
        with pytest.raises(pps.PPSError):
            pps.attn_plan(*t, hq, hkv, d, p, 4)


def test_empty_batch_plans(pps):
    plan = pps.attn_plan(np.array([0], np.int32), np.zeros(0, np.int32), np.array([0], np.int32),
                         np.zeros(0, np.int32), 8, 2, 64, 16, 4)
    info = plan.info()
    assert info["num_bw_tasks"] == 0 and info["num_mma_tasks"] == 0
    plan.destroy()


def test_missing_library_fails_loudly(tmp_path):
    """Without libpps.so the binding raises; it never falls back to another path."""
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "import paged_prefix_shared_gb300 as p\n"
        "p.LIB_PATH = %r\n"
        "try:\n"
        "    p.attn_plan([0, 1], [1], [0, 1], [0], 8, 2, 64, 16, 1)\n"
        "except p.PPSError as e:\n"
        "    print('raised:', e)\n"
        "    sys.exit(0)\n"
        "sys.exit(3)\n" % (ROOT, str(tmp_path / "absent" / "libpps.so")))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "missing" in r.stdout
