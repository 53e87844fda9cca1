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
                 "pa_paged_kv_write_fp8", "pa_paged_attention_decode_fp8",
                 "pa_paged_attention_decode_fp8_append", "pa_paged_attention_decode_append",
                 "pa_decode_workspace_bytes", "pa_get_device_error", "pa_alloc_create",
                 "pa_alloc_append", "pa_alloc_fork", "pa_alloc_free_seq"):
        assert must in names


def test_library_exports_every_declared_symbol(pa):
    lib = pa.lib()
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert missing == []


def test_bounded_wait_check_validates_on_the_host(pa):
    # refused before any CUDA call: a bound outside [1 us, 1 s], a misaligned report
    L = pa.lib()
    assert L.pa_check_bounded_wait(0, None, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_check_bounded_wait(2_000_000_000, None, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_check_bounded_wait(1_000_000, 12, None) == pa.PA_ERR_INVALID_ARG


def test_automatic_partition_size(pa):
    # 1024 tokens once num_seqs * ceil(max_context_len / 1024) >= 64, else 512; explicit sizes pass through
    assert pa.decode_partition_size(64, 4096) == 1024          # the 8B-shaped batch
    assert pa.decode_partition_size(8, 131072) == 1024         # long context
    assert pa.decode_partition_size(16, 4096) == 1024          # exactly 64 partitions
    assert pa.decode_partition_size(15, 4096) == 512
    assert pa.decode_partition_size(1, 20000) == 512
    assert pa.decode_partition_size(10, 100, 256) == 256
    # the workspace is sized for the partitions the call will use
    assert pa.decode_workspace_bytes(64, 32, 128, 4096, 0) == pa.decode_workspace_bytes(64, 32, 128, 4096, 1024)
    assert pa.decode_workspace_bytes(4, 32, 128, 4096, 0) == pa.decode_workspace_bytes(4, 32, 128, 4096, 512)


def _shared_rule(num_seqs, groups, kvh, max_prefix, max_ctx, sms=152):
    # the documented estimate: ceil(items / SMs) * (tiles per item + 1.4), minimised
    # over multiples of 128 from 512 to the longest prefix, ties to the larger; then
    # grown to cover whole contexts (<= 8192) when one partition holds each prefix
    if groups <= 0 or kvh <= 0 or max_prefix <= 0:
        return 512
    best, best_cost = None, None
    top = max(min(-(-max_prefix // 128) * 128, 65536), 512)
    for part in range(512, top + 1, 128):
        items = groups * kvh * -(-max_prefix // part)
        cost = -(-items // sms) * (-(-min(part, max_prefix) // 128) + 1.4)
        if best is None or cost <= best_cost:
            best, best_cost = part, cost
    whole = -(-max_ctx // 128) * 128
    if best >= max_prefix and best < whole <= 8192 and num_seqs * kvh >= 2 * sms:
        best = whole
    return best


def test_automatic_shared_partition_size(pa):
    # the forked-sampling batch: 256 sequences in 32 groups of 8, 992 shared tokens,
    # contexts up to 1257 tokens, 8 kv heads -> one partition per group and kv head,
    # grown to cover whole contexts (1280: no merge)
    assert pa.decode_shared_partition_size(256, 32, 8, 992, 1257) == 1280
    assert pa.decode_shared_partition_size(64, 8, 8, 992, 1257) == 512      # 8 groups: two partitions each
    assert pa.decode_shared_partition_size(32, 4, 8, 992, 1257) == 512      # too few private items to grow
    assert pa.decode_shared_partition_size(256, 0, 8, 992, 1257) == 512     # no groups
    assert pa.decode_shared_partition_size(256, 32, 8, 0, 1257) == 512      # nothing shared
    assert pa.decode_shared_partition_size(256, 32, 8, 992, 1257, 256) == 256   # explicit sizes pass through
    assert pa.decode_shared_partition_size(256, 32, 8, 300, 1257) == 1280   # never below 512; grown
    assert pa.decode_shared_partition_size(256, 32, 8, 992, 20000) == 1024  # contexts too long to cover
    for args in [(8, 1, 8, 32768, 40000), (256, 32, 8, 32768, 33000), (20, 4, 1, 5000, 6000),
                 (1600, 200, 8, 4096, 4500), (6, 3, 2, 100000, 100100), (512, 64, 8, 2000, 8192)]:
        got = pa.decode_shared_partition_size(*args)
        assert got == _shared_rule(*args), (args, got)
        assert got % 128 == 0 and got >= 512
        # the workspace sized for the automatic choice (0) covers it
        assert pa.decode_shared_workspace_bytes(64, 32, 128, args[4], 0) >= \
            pa.decode_shared_workspace_bytes(64, 32, 128, args[4], got)


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


def _decode_fp8(pa, **kw):
    args = dict(out=16, q=16, kc=16, vc=16, bt=16, mb=4, cl=16, B=2, H=8, Hk=2, D=128, bs=16, nb=64,
                scale=0.1, ks=0.05, vs=0.05, maxctx=0, part=0, ws=None, wsb=0, dtype=2, stream=None)
    args.update(kw)
    a = args
    return pa.lib().pa_paged_attention_decode_fp8(a["out"], a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["cl"],
                                                  a["B"], a["H"], a["Hk"], a["D"], a["bs"], a["nb"], a["scale"],
                                                  a["ks"], a["vs"], a["maxctx"], a["part"], a["ws"], a["wsb"],
                                                  a["dtype"], a["stream"])


@pytest.mark.parametrize("bad,code", [
    (dict(dtype=0), -2),            # fp32 queries: not supported on the 8-bit path
    (dict(dtype=3), -1),            # the storage code is not a query type
    (dict(dtype=9), -1),
    (dict(ks=0.0), -1),             # scales must be finite and positive
    (dict(vs=-1.0), -1),
    (dict(ks=float("inf")), -1),
    (dict(vs=float("nan")), -1),
    (dict(D=64), -2),               # head_dim 128 only
    (dict(bs=4), -2),               # block size 8..128
    (dict(bs=256), -2),
    (dict(H=6, Hk=4), -1),
    (dict(q=8), -1),
])
def test_decode_fp8_rejects_bad_arguments_on_the_host(pa, bad, code):
    assert _decode_fp8(pa, **bad) == code


def test_decode_fp8_with_no_sequences_is_a_no_op(pa):
    assert _decode_fp8(pa, B=0) == 0


def test_write_fp8_rejects_bad_arguments(pa):
    L = pa.lib()
    ok = dict(k=16, v=16, sm=16, T=4, kc=16, vc=16, nb=8, bs=16, hk=8, d=128, ks=0.1, vs=0.1, dt=2)

    def w(**kw):
        a = dict(ok, **kw)
        return L.pa_paged_kv_write_fp8(a["k"], a["v"], a["sm"], a["T"], a["kc"], a["vc"], a["nb"], a["bs"],
                                       a["hk"], a["d"], a["ks"], a["vs"], a["dt"], None)
    assert w(dt=3) == -1                 # source must be fp32, fp16 or bf16
    assert w(ks=0.0) == -1 and w(vs=float("inf")) == -1
    assert w(hk=1, d=8) == -2            # rows of 8 codes: not a multiple of 16
    assert w(T=0) == 0                   # nothing to do
    assert w(k=8) == -1                  # misaligned
    assert w(T=2 ** 40) == -2            # one thread per 16-element run: beyond one launch
    # copy_blocks takes the 8-bit storage code
    assert L.pa_copy_blocks(16, 16, 16, 0, 8, 16, 8, 128, 3, None) == 0


def test_decode_append_rejects_bad_arguments(pa):
    L = pa.lib()

    def call(k_new=16, v_new=16, slots=16, B=4):
        return L.pa_paged_attention_decode_append(16, 16, k_new, v_new, slots, 16, 16, 16, 8, 16, B, 8, 2, 128, 16,
                                                  64, 0.1, 0, 0, None, 0, 2, None)
    assert call(B=0) == 0                # nothing to do
    assert call(k_new=None) == -1 and call(slots=None) == -1
    assert call(v_new=8) == -1           # misaligned


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


def test_every_compute_call_refuses_host_tensors(pa):
    """No CPU fallback: each compute entry point rejects host tensors before any
    work, and leaves its output untouched."""
    import torch
    B, H, Hk, D, bs, NB, MB = 2, 4, 2, 128, 16, 8, 4
    kc = torch.zeros(NB, bs, Hk, D, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    kc8 = torch.zeros(NB, bs, Hk, D, dtype=torch.uint8)
    vc8 = torch.zeros_like(kc8)
    q = torch.ones(B, H, D, dtype=torch.bfloat16)
    out = torch.full_like(q, 7.0)
    kn = torch.zeros(B, Hk, D, dtype=torch.bfloat16)
    vn = torch.zeros_like(kn)
    slots = torch.tensor([0, 16], dtype=torch.int32)
    bt = torch.arange(B * MB, dtype=torch.int32).view(B, MB)
    cl = torch.tensor([1, 1], dtype=torch.int32)
    qsl = torch.tensor([0, 1, 2], dtype=torch.int32)
    pairs = torch.tensor([[0, 1]], dtype=torch.int32)
    calls = {
        "paged_kv_write": lambda: pa.paged_kv_write(kn, vn, slots, kc, vc),
        "paged_attention_decode": lambda: pa.paged_attention_decode(out, q, kc, vc, bt, cl, 0.1),
        "paged_attention_decode_append": lambda: pa.paged_attention_decode_append(out, q, kn, vn, slots, kc, vc, bt,
                                                                                  cl, 0.1),
        "paged_attention_prefill": lambda: pa.paged_attention_prefill(out, q, kc, vc, bt, cl, qsl, 0.1, 1),
        "paged_attention_decode_shared": lambda: pa.paged_attention_decode_shared(
            out, q, kc, vc, bt, cl, torch.zeros(B, dtype=torch.int32), torch.zeros(1, B, dtype=torch.int32), 0.1),
        "copy_blocks": lambda: pa.copy_blocks(kc, vc, pairs),
        "paged_kv_write_fp8": lambda: pa.paged_kv_write_fp8(kn, vn, slots, kc8, vc8, 1.0, 1.0),
        "paged_attention_decode_fp8": lambda: pa.paged_attention_decode_fp8(out, q, kc8, vc8, bt, cl, 0.1, 1.0,
                                                                            1.0),
    }
    for name, call in calls.items():
        with pytest.raises(ValueError, match="must be a CUDA tensor"):
            call()
        assert torch.all(out == 7.0), name
