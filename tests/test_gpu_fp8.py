"""GPU parity of the 8-bit (OCP FP8 E4M3) cache path against the CPU oracle.

Scatter and block copy: bit-exact codes. Decode: max/mean abs error within
2e-2 / 2e-3 for bf16 and fp16 outputs. The kernel multiplies the codes as
stored; the query enters as two E4M3 terms (exact for bf16, 8 significant
bits for f16) and each softmax weight as two E4M3 terms (about a bf16's
precision), so the error budget is that of the 16-bit decode (P in 16 bits,
fp32 accumulation, the output rounded once).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_cases import (FP8_POISON, assert_close, dev, gpu_decode_fp8, oracle_decode_fp8, pa_mod, to_f64)

pytestmark = pytest.mark.gpu

S = workloads.FP8_SCALE


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def pa():
    return pa_mod()


def _errors_clear(pa):
    assert pa.get_device_error() == 0


def _nan_code(c):
    return (c & 0x7F) == 0x7F


# ---------------------------------------------------------------------------
# scatter with quantisation
# ---------------------------------------------------------------------------

def _write_both(pa, rows_k, rows_v, slots, NB, bs, Hk, D, k_scale, v_scale, src):
    """GPU and oracle scatter of the same float32 rows (rounded to src on both sides) into caches
    pre-filled with 0xAB; returns (gpu K, gpu V, oracle K, oracle V) as uint8."""
    d = dev()
    tdt = workloads.torch_dtype(src)
    T = rows_k.shape[0]
    kc = torch.full((NB, bs, Hk, D), 0xAB, dtype=torch.uint8, device=d)
    vc = torch.full_like(kc, 0xAB)
    pa.paged_kv_write_fp8(torch.from_numpy(rows_k).to(d).to(tdt).reshape(T, Hk, D).contiguous(),
                          torch.from_numpy(rows_v).to(d).to(tdt).reshape(T, Hk, D).contiguous(),
                          torch.as_tensor(slots, device=d), kc, vc, k_scale, v_scale)
    torch.cuda.synchronize()
    ok = np.full((NB, bs, Hk, D), 0xAB, np.uint8)
    ov = ok.copy()
    oracle.kv_write_fp8(workloads.to_storage_numpy(rows_k, src), workloads.to_storage_numpy(rows_v, src),
                        slots, ok, ov, k_scale, v_scale, src)
    return kc.cpu().numpy(), vc.cpu().numpy(), ok, ov


@pytest.mark.parametrize("src", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("k_scale,v_scale", [(S, S), (2.0 ** -8, 0.37), (1024.0, 3.0e-3)])
def test_write_fp8_bit_exact(pa, src, k_scale, v_scale):
    """Ragged token count, -1 slots, scales that round normally, saturate (k / 2^-8
    exceeds 448) and reach the subnormal codes and signed zeros (k / 1024)."""
    Hk, D, bs, NB, T = 8, 128, 16, 12, 37
    rng = np.random.default_rng(501)
    slots = rng.choice(NB * bs, T, replace=False).astype(np.int32)
    slots[[3, 20]] = -1
    keys = np.arange(T, dtype=np.int64) + 77
    pos = np.arange(T, dtype=np.int64)
    rk = workloads.content_rows(5, workloads.TID_K, keys, pos, Hk * D)
    rv = workloads.content_rows(5, workloads.TID_V, keys, pos, Hk * D)
    gk, gv, ok, ov = _write_both(pa, rk, rv, slots, NB, bs, Hk, D, float(k_scale), float(v_scale), src)
    assert np.array_equal(gk, ok)
    assert np.array_equal(gv, ov)
    _errors_clear(pa)


def test_write_fp8_special_values(pa):
    """Infinities saturate to +-448, NaN gives a NaN code, -0 keeps its sign,
    exact midpoints between codes round to the even code."""
    pos = oracle.e4m3_to_float64(np.arange(0x00, 0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)            # 126 exact midpoints
    special = np.array([np.inf, -np.inf, np.nan, -0.0, 0.0, 1e-45, -1e-45, 448.0, 464.0, -1e9,
                        2.0 ** -10, -(2.0 ** -10)], np.float32)
    vals = np.concatenate([mids, -mids, special]).astype(np.float32)
    row = 16
    n = -(-vals.shape[0] // row) * row
    x = np.zeros(n, np.float32)
    x[: vals.shape[0]] = vals
    rows = x.reshape(-1, row)
    T = rows.shape[0]
    slots = np.arange(T, dtype=np.int32)
    gk, gv, ok, ov = _write_both(pa, rows, rows[::-1].copy(), slots, 2, T, 1, row, 1.0, 1.0, "f32")
    for g, o in ((gk, ok), (gv, ov)):
        g, o = g.reshape(-1), o.reshape(-1)
        nan = _nan_code(o)
        assert np.array_equal(_nan_code(g), nan)
        assert np.array_equal(g[~nan], o[~nan])
    _errors_clear(pa)


def test_write_fp8_bad_slot_sets_the_error(pa):
    d = dev()
    kc = torch.zeros((4, 4, 1, 64), dtype=torch.uint8, device=d)
    vc = torch.zeros_like(kc)
    k = torch.ones((3, 1, 64), dtype=torch.bfloat16, device=d)
    slots = torch.tensor([2, 16, -7], dtype=torch.int32, device=d)
    pa.paged_kv_write_fp8(k, k, slots, kc, vc, 1.0, 1.0)
    assert pa.get_device_error() & pa.PA_DEVERR_SLOT
    assert int((kc != 0).sum()) == 64 and int(kc.view(-1, 64)[2, 0]) == 0x38   # code of 1.0


def test_copy_blocks_fp8_bit_exact(pa):
    rng = np.random.default_rng(502)
    NB, bs, Hk, D = 24, 16, 2, 128
    d = dev()
    kc = torch.from_numpy(rng.integers(0, 256, (NB, bs, Hk, D), dtype=np.uint8)).to(d)
    vc = torch.from_numpy(rng.integers(0, 256, (NB, bs, Hk, D), dtype=np.uint8)).to(d)
    ok, ov = kc.cpu().numpy(), vc.cpu().numpy()
    pairs = np.array([[0, 5], [3, 7], [11, 2], [4, 20]], np.int32)
    pa.copy_blocks(kc, vc, torch.as_tensor(pairs, device=d))
    oracle.copy_blocks(ok, ov, pairs, "e4m3")
    assert np.array_equal(kc.cpu().numpy(), ok) and np.array_equal(vc.cpu().numpy(), ov)
    _errors_clear(pa)


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

RAGGED = np.array([1, 7, 0, 128, 129, 300, 513, 1000, 1024, 77], np.int32)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("bs", [8, 16, 128])
@pytest.mark.parametrize("H,Hk", [(8, 8), (32, 8), (16, 2), (32, 2)])
def test_decode_fp8_ragged_contexts(pa, dtype, bs, H, Hk):
    """Contexts of 0, 1, a tile, a tile plus one, several partitions and ragged
    tails; group sizes 1, 4, 8 and 16; the newest token of each written by the
    8-bit scatter."""
    w = workloads.make_decode(f"fp8_{dtype}_{bs}_{H}_{Hk}", 503 + bs + H, RAGGED, H, Hk, 128, bs, dtype)
    out, _, _ = gpu_decode_fp8(w, max_context_len=int(RAGGED.max()))
    ref = oracle_decode_fp8(w, range(w.num_seqs))
    got = to_f64(out)
    assert np.all(got[2] == 0.0)                        # empty context
    assert_close(got, ref, dtype, f"fp8 {dtype} bs{bs} H{H}/{Hk}")
    _errors_clear(pa)


@pytest.mark.parametrize("bs,H,Hk,dtype", [(32, 12, 4, "bf16"), (64, 24, 8, "f16"), (32, 6, 2, "f16")])
def test_decode_fp8_padded_groups_and_block_sizes(pa, bs, H, Hk, dtype):
    """G = 3 (padded to 4 columns) and block sizes 32 / 64."""
    w = workloads.make_decode(f"fp8_g{H // Hk}_{bs}", 511 + bs, RAGGED, H, Hk, 128, bs, dtype)
    out, _, _ = gpu_decode_fp8(w, max_context_len=int(RAGGED.max()))
    assert_close(to_f64(out), oracle_decode_fp8(w, range(w.num_seqs)), dtype, f"fp8 bs{bs} H{H}/{Hk} {dtype}")
    _errors_clear(pa)


def test_decode_fp8_many_partitions_split_the_launch(pa):
    rng = np.random.default_rng(512)
    ctx = rng.integers(19000, 20000, size=64).astype(np.int32)
    ctx[[5, 40]] = [1, 20000]
    w = workloads.make_decode("fp8_many_items", 512, ctx, 32, 8, 128, 16, "bf16")
    out, _, _ = gpu_decode_fp8(w, max_context_len=20000, partition_size=128)
    seqs = [0, 5, 30, 31, 32, 40, 63]
    assert_close(to_f64(out)[seqs], oracle_decode_fp8(w, seqs), "bf16", "fp8 split launch")
    _errors_clear(pa)


@pytest.mark.parametrize("partition_size", [128, 256, 1024])
def test_decode_fp8_partition_sizes(pa, partition_size):
    w = workloads.make_decode("fp8_parts", 509, RAGGED, 32, 8, 128, 16, "bf16")
    out, _, _ = gpu_decode_fp8(w, partition_size=partition_size, max_context_len=int(RAGGED.max()))
    assert_close(to_f64(out), oracle_decode_fp8(w, range(w.num_seqs)), "bf16", f"partition {partition_size}")
    _errors_clear(pa)


def test_decode_fp8_llama8b_full_batch(pa):
    w = workloads.llama8b_decode()
    out, _, _ = gpu_decode_fp8(w)
    assert_close(to_f64(out), oracle_decode_fp8(w, range(w.num_seqs)), "bf16", "fp8 llama8b_decode")
    _errors_clear(pa)


def test_decode_fp8_long_context_sampled(pa):
    w = workloads.long_context()
    out, _, _ = gpu_decode_fp8(w, max_context_len=int(w.context_lens.max()), partition_size=512)
    seqs = [int(np.argmin(w.context_lens)), int(np.argmax(w.context_lens))]
    assert_close(to_f64(out)[seqs], oracle_decode_fp8(w, seqs), "bf16", "fp8 long_context")
    # every row is a convex combination of V rows: finite and within the V range
    o = to_f64(out)
    vmax = max(240 * S, workloads.CONTENT_MAX * 1.0001)
    assert np.all(np.isfinite(o)) and np.abs(o).max() <= vmax + 0.05
    _errors_clear(pa)


def test_decode_fp8_mixed_serving_sampled(pa):
    w = workloads.mixed_serving(block_size=16, dtype="f16")
    out, _, _ = gpu_decode_fp8(w, max_context_len=int(w.context_lens.max()))
    rng = np.random.default_rng(16)
    seqs = np.unique(np.concatenate([rng.choice(w.num_seqs, 48, replace=False),
                                     [int(np.argmax(w.context_lens)), int(np.argmin(w.context_lens))]]))
    assert_close(to_f64(out)[seqs], oracle_decode_fp8(w, seqs), "f16", "fp8 mixed f16")
    _errors_clear(pa)


def test_decode_fp8_large_batch_runs_in_chunks(pa):
    rng = np.random.default_rng(504)
    ctx = rng.integers(0, 1200, size=2500).astype(np.int32)
    w = workloads.make_decode("fp8_big_batch", 504, ctx, 16, 4, 128, 16, "bf16")
    out, _, _ = gpu_decode_fp8(w, max_context_len=int(ctx.max()), partition_size=256)
    seqs = np.concatenate([np.arange(0, 2500, 37), [1023, 1024, 1025, 2047, 2048, 2499]])
    assert_close(to_f64(out)[seqs], oracle_decode_fp8(w, seqs), "bf16", "fp8 2500 sequences")
    _errors_clear(pa)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_decode_fp8_query_magnitudes_per_head(pa, dtype):
    """The query enters the 8-bit MMAs as two E4M3 terms after a power-of-two scale
    chosen per head. Heads of one group get magnitudes 2^-130 (bf16 subnormals; f16
    flushes them to zero), 2^-12, 2^4 and exactly 0 (a uniform softmax): each head's
    scale is its own, and the clamped and all-zero cases still match the oracle."""
    w = workloads.make_decode("fp8_qmag", 508, np.array([1, 100, 700, 1500], np.int32), 16, 4, 128, 16, dtype)
    d = dev()
    dt = workloads.torch_dtype(dtype)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, FP8_POISON, dtype=torch.uint8, device=d)
    vc = torch.full(shape, FP8_POISON, dtype=torch.uint8, device=d)
    w.fill_cache_torch(kc, vc, include_newest=True)
    factor = torch.tensor([2.0 ** -130, 2.0 ** -12, 2.0 ** 4, 0.0], dtype=torch.float64)
    factor = factor.repeat(w.num_heads // 4)[None, :, None]
    q64 = w.q_values(like=kc).double().cpu() * factor
    q = q64.to(dt).to(d).contiguous()
    out = torch.full_like(q, float("nan"))
    pa.paged_attention_decode_fp8(out, q, kc, vc, torch.as_tensor(w.block_tables, device=d),
                                  torch.as_tensor(w.context_lens, device=d), w.scale, S, S)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    seqs = np.arange(w.num_seqs)
    view = w.compact_host_view(seqs, include_newest=True, codes=True)
    qh = workloads.to_storage_numpy(q.float().cpu().numpy(), dtype)
    ref = oracle.paged_attention_fp8(qh, view["key_cache"], view["value_cache"], view["block_tables"],
                                     view["context_lens"], w.scale, S, S, dtype,
                                     num_threads=oracle.num_host_threads())
    assert_close(to_f64(out), ref, dtype, f"fp8 query magnitudes {dtype}")


def test_decode_fp8_single_token_is_dequantised_v(pa):
    """ctx = 1: the softmax weight is 1, so out = v_scale * decoded(V code) rounded once."""
    w = workloads.make_decode("fp8_one", 505, np.array([1, 1, 1], np.int32), 16, 4, 128, 8, "bf16")
    out, kc, vc = gpu_decode_fp8(w, write_newest=False)
    vq = torch.float8_e4m3fn
    for b in range(3):
        blk = int(w.block_tables[b, 0])
        v = vc[blk, 0].view(vq).float() * torch.tensor(S, dtype=torch.float32)
        want = v.repeat_interleave(4, dim=0).to(torch.bfloat16)
        assert torch.equal(out[b].cpu(), want.cpu())
    _errors_clear(pa)


def test_decode_fp8_matches_16bit_decode_of_the_dequantised_cache(pa):
    """With power-of-two scales every dequantised element is exact in bf16: the
    16-bit kernel on those values and the 8-bit kernel on the codes compute the
    same thing (only the place of the k_scale factor differs)."""
    w = workloads.llama8b_decode(num_seqs=16)
    ks, vs = 2.0 ** -5, 2.0 ** -6
    out8, kc, vc = gpu_decode_fp8(w, write_newest=False, k_scale=ks, v_scale=vs)
    kb = (kc.view(torch.float8_e4m3fn).float() * ks).to(torch.bfloat16)
    vb = (vc.view(torch.float8_e4m3fn).float() * vs).to(torch.bfloat16)
    d = dev()
    q = w.q_values(like=kc).to(torch.bfloat16).contiguous()
    out16 = torch.empty_like(q)
    pa.paged_attention_decode(out16, q, kb, vb, torch.as_tensor(w.block_tables, device=d),
                              torch.as_tensor(w.context_lens, device=d), w.scale)
    torch.cuda.synchronize()
    diff = (out8.float() - out16.float()).abs()
    assert float(diff.max()) <= 1e-2 and float(diff.mean()) <= 1e-4
    _errors_clear(pa)


def test_decode_fp8_accepts_float8_typed_caches(pa):
    w = workloads.make_decode("fp8_view", 506, np.array([300, 5], np.int32), 8, 2, 128, 16, "bf16")
    out, kc, vc = gpu_decode_fp8(w, write_newest=False)
    d = dev()
    q = w.q_values(like=kc).to(torch.bfloat16).contiguous()
    out2 = torch.empty_like(q)
    pa.paged_attention_decode_fp8(out2, q, kc.view(torch.float8_e4m3fn), vc.view(torch.float8_e4m3fn),
                                  torch.as_tensor(w.block_tables, device=d),
                                  torch.as_tensor(w.context_lens, device=d), w.scale, S, S)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_decode_fp8_bad_block_id_reads_zeros(pa):
    w = workloads.make_decode("fp8_badid", 507, np.array([300, 300], np.int32), 8, 2, 128, 16, "bf16")
    d = dev()
    kc = torch.full((w.num_blocks, 16, 2, 128), FP8_POISON, dtype=torch.uint8, device=d)
    vc = torch.full_like(kc, FP8_POISON)
    w.fill_cache_torch(kc, vc, include_newest=True)
    bad = w.block_tables.copy()
    bad[1, 3] = w.num_blocks + 9
    bad[1, 5] = -3
    q = w.q_values(like=kc).to(torch.bfloat16).contiguous()
    out = torch.empty_like(q)
    pa.paged_attention_decode_fp8(out, q, kc, vc, torch.as_tensor(bad, device=d),
                                  torch.as_tensor(w.context_lens, device=d), w.scale, S, S)
    assert pa.get_device_error() & pa.PA_DEVERR_BLOCK_ID
    ref = oracle_decode_fp8(w, [0], write_newest=False)
    assert_close(to_f64(out)[:1], ref, "bf16", "unaffected sequence")
    assert torch.isfinite(out.float()).all()
