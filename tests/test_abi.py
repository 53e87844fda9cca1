"""The C-ABI library loads and exports every declared entry point (no GPU needed).

Also checks host-side argument validation, which runs before any CUDA call.
"""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build
    build()
    import paged_kv_cache_261_gb300 as pa
    return pa


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pagedattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary_calls():
    names = _declared_functions()
    for must in ("pa_paged_kv_write", "pa_paged_attention_decode", "pa_copy_blocks",
                 "pa_decode_workspace_bytes", "pa_get_device_error", "pa_alloc_create",
                 "pa_alloc_append", "pa_alloc_fork", "pa_alloc_free_seq"):
        assert must in names


def test_library_exports_every_declared_symbol(pa):
    lib = pa.lib()
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert missing == []


def test_status_strings(pa):
    assert pa.status_string(0) == "PA_OK"
    assert pa.status_string(-5) == "PA_ERR_DEVICE_INDEX"
    assert pa.status_string(-99) == "PA_ERR_UNKNOWN"
    assert pa.version() >= 100


def test_workspace_size_formula(pa):
    # one partition -> no workspace; else B*H*P*(2 + D) floats (+ alignment pad)
    assert pa.decode_workspace_bytes(4, 8, 128, 512, 512) == 0
    n = pa.decode_workspace_bytes(4, 8, 128, 513, 512)
    P = 2
    assert n >= 4 * 8 * P * (2 + 128) * 4 and n < 4 * 8 * P * (2 + 128) * 4 + 256


def _decode(pa, **kw):
    args = dict(out=16, q=16, kc=16, vc=16, bt=16, mb=4, cl=16, B=2, H=8, Hk=2, D=128, bs=16, nb=64,
                scale=0.1, maxctx=0, part=0, ws=None, wsb=0, dtype=2, stream=None)
    args.update(kw)
    a = args
    return pa.lib().pa_paged_attention_decode(a["out"], a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["cl"],
                                              a["B"], a["H"], a["Hk"], a["D"], a["bs"], a["nb"], a["scale"],
                                              a["maxctx"], a["part"], a["ws"], a["wsb"], a["dtype"], a["stream"])


@pytest.mark.parametrize("bad,code", [
    (dict(H=6, Hk=4), -1),          # heads not a multiple of kv heads
    (dict(D=96), -2),               # head_dim not supported
    (dict(bs=12), -2),              # block size not a power of two
    (dict(H=64, Hk=2), -2),         # group above 16
    (dict(part=100), -1),           # partition not a multiple of 128
    (dict(dtype=7), -1),            # unknown dtype
    (dict(out=None), -1),           # null pointer
    (dict(q=8), -1),                # misaligned pointer
    (dict(nb=0), -1),
    (dict(B=-1), -1),
])
def test_decode_rejects_bad_arguments_on_the_host(pa, bad, code):
    assert _decode(pa, **bad) == code


def test_decode_with_no_sequences_is_a_no_op(pa):
    assert _decode(pa, B=0) == 0


def test_write_and_copy_reject_bad_arguments(pa):
    L = pa.lib()
    assert L.pa_paged_kv_write(16, 16, 16, 4, 16, 16, 8, 16, 8, 128, 9, None) == -1
    assert L.pa_paged_kv_write(16, 16, 16, 4, 16, 16, 8, 16, 1, 6, 2, None) == -2   # 12-byte rows
    assert L.pa_paged_kv_write(16, 16, 16, 0, 16, 16, 8, 16, 8, 128, 2, None) == 0  # nothing to do
    assert L.pa_copy_blocks(16, 16, 16, -1, 8, 16, 8, 128, 2, None) == -1
    assert L.pa_copy_blocks(16, 16, 16, 0, 8, 16, 8, 128, 2, None) == 0


def test_get_device_error_requires_output_pointer(pa):
    assert pa.lib().pa_get_device_error(None, None) == -1


def test_package_import_fails_loudly_without_the_library(tmp_path):
    # a copy of the package without _build/ must refuse to import
    import shutil
    import subprocess
    import sys
    dst = tmp_path / "paged_kv_cache_261_gb300"
    shutil.copytree(os.path.join(ROOT, "paged_kv_cache_261_gb300"), dst,
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    r = subprocess.run([sys.executable, "-c", "import paged_kv_cache_261_gb300"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode != 0 and "libpagedattn.so is missing" in r.stderr
