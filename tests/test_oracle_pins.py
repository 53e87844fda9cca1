"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test names what fixes the expected value: a fixture made from the pages
(tests/golden/), a closed form, a textbook special case, or a library routine
(torch's scaled_dot_product_attention in float64 on contiguous K/V, numpy's and
torch's own float16/bfloat16 widening).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import read_golden


def _dense_case(B, H, Hk, D, ctxs, bs, seed, nb=None, dtype="f32"):
    """Random paged case: contiguous K/V per sequence placed on a shuffled pool."""
    rng = np.random.default_rng(seed)
    ctxs = np.asarray(ctxs, dtype=np.int32)
    nbs = (ctxs + bs - 1) // bs
    total = int(nbs.sum())
    nb = nb or max(total + 3, 1)
    perm = rng.permutation(nb).astype(np.int32)
    mb = max(int(nbs.max()), 1)
    tables = np.full((B, mb), -1, np.int32)
    kc = np.zeros((nb, bs, Hk, D), np.float64)
    vc = np.zeros_like(kc)
    K = [rng.standard_normal((int(c), Hk, D)) for c in ctxs]
    V = [rng.standard_normal((int(c), Hk, D)) for c in ctxs]
    off = 0
    for b in range(B):
        tables[b, : nbs[b]] = perm[off: off + nbs[b]]
        off += nbs[b]
        for t in range(int(ctxs[b])):
            kc[tables[b, t // bs], t % bs] = K[b][t]
            vc[tables[b, t // bs], t % bs] = V[b][t]
    q = rng.standard_normal((B, H, D))
    return q, kc, vc, tables, ctxs, K, V


def _sdpa(q, K, V, scale):
    """torch float64 SDPA of one sequence: q [H, D], K/V [ctx, Hk, D]."""
    H = q.shape[0]
    Hk = K.shape[1]
    qt = torch.from_numpy(q).reshape(1, H, 1, -1)
    kt = torch.from_numpy(np.ascontiguousarray(K.transpose(1, 0, 2)))[None]
    vt = torch.from_numpy(np.ascontiguousarray(V.transpose(1, 0, 2)))[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale,
                                                         enable_gqa=(Hk != H))
    return o.reshape(H, -1).numpy()


# --------------------------------------------------------------------------
# attention = dense attention over the concatenated K/V (page 2, demo 2)
# pinned against a library routine
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bs", [1, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("H,Hk", [(4, 4), (8, 2), (6, 1)])
def test_attention_matches_torch_sdpa(bs, H, Hk):
    ctxs = [1, 5, 17, 33, 64, 100]
    q, kc, vc, bt, cl, K, V = _dense_case(len(ctxs), H, Hk, 16, ctxs, bs, seed=bs * 31 + H)
    scale = 0.3
    out = oracle.paged_attention(q, kc, vc, bt, cl, scale, "f64")
    for b in range(len(ctxs)):
        ref = _sdpa(q[b], K[b], V[b], scale)
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)


def test_tiny_workload_matches_torch_sdpa():
    w = workloads.tiny_fp32()
    view = w.compact_host_view(range(w.num_seqs), include_newest=True)
    q = w.q_values().astype(np.float32)
    out = oracle.paged_attention(q, view["key_cache"], view["value_cache"], view["block_tables"],
                                 view["context_lens"], w.scale, "f32")
    for b in range(w.num_seqs):
        K, V = w.contiguous_kv(b)
        ref = _sdpa(q[b].astype(np.float64), K.astype(np.float64), V.astype(np.float64), w.scale)
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# closed forms and textbook special cases
# --------------------------------------------------------------------------

def _single(q, K, V, scale, bs=2):
    """One sequence, one kv head: q [H, D], K/V [ctx, D]."""
    ctx, D = K.shape
    nb = (ctx + bs - 1) // bs
    kc = np.zeros((nb, bs, 1, D))
    vc = np.zeros_like(kc)
    for t in range(ctx):
        kc[t // bs, t % bs, 0] = K[t]
        vc[t // bs, t % bs, 0] = V[t]
    bt = np.arange(nb, dtype=np.int32)[None]
    cl = np.array([ctx], np.int32)
    return oracle.paged_attention(q[None], kc, vc, bt, cl, scale, "f64")[0]


def test_two_token_logistic_closed_form():
    # K rows are basis vectors e0, e1 and V rows e2, e3, so the two scores are
    # (a, b) and the output is (0, 0, sigmoid(a - b), sigmoid(b - a)).
    for a, b in [(0.3, -1.1), (2.0, 2.0), (-4.0, 3.5)]:
        K = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
        V = np.array([[0, 0, 1.0, 0], [0, 0, 0, 1.0]])
        out = _single(np.array([[a, b, 0.0, 0.0]]), K, V, 1.0)
        sig = 1.0 / (1.0 + math.exp(-(a - b)))
        np.testing.assert_allclose(out[0], [0, 0, sig, 1 - sig], rtol=0, atol=1e-15)


def test_single_token_returns_v0_exactly():
    rng = np.random.default_rng(3)
    K = rng.standard_normal((1, 8))
    V = rng.standard_normal((1, 8))
    out = _single(rng.standard_normal((3, 8)), K, V, 0.7)
    assert np.array_equal(out, np.repeat(V, 3, axis=0))


def test_zero_query_gives_mean_of_v():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((37, 8))
    V = rng.standard_normal((37, 8))
    out = _single(np.zeros((2, 8)), K, V, 1.0, bs=4)
    np.testing.assert_allclose(out, np.repeat(V.mean(0, keepdims=True), 2, 0), rtol=0, atol=1e-14)


def test_equal_keys_give_mean_of_v():
    rng = np.random.default_rng(5)
    K = np.repeat(rng.standard_normal((1, 8)), 21, axis=0)
    V = rng.standard_normal((21, 8))
    out = _single(rng.standard_normal((1, 8)), K, V, 1.0, bs=8)
    np.testing.assert_allclose(out[0], V.mean(0), rtol=0, atol=1e-14)


def test_peaky_scores_select_the_argmax_value_without_overflow():
    # scores of order 1e4: a softmax without the max shift overflows to inf/nan
    rng = np.random.default_rng(6)
    K = rng.standard_normal((50, 8))
    V = rng.standard_normal((50, 8))
    q = rng.standard_normal((1, 8)) * 3000.0
    out = _single(q, K, V, 1.0, bs=16)
    s = K @ q[0]
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0], V[int(np.argmax(s))], rtol=0, atol=1e-12)


def test_gqa_head_map_groups_are_contiguous():
    # V of kv head j is the constant j + 1, so every query head h must return
    # h // G + 1 (contiguous groups of G = H / Hk query heads per kv head).
    H, Hk, D, bs = 6, 2, 4, 4
    rng = np.random.default_rng(7)
    ctx = 9
    kc = rng.standard_normal((3, bs, Hk, D))
    vc = np.zeros_like(kc)
    for j in range(Hk):
        vc[:, :, j, :] = j + 1.0
    bt = np.array([[2, 0, 1]], np.int32)
    out = oracle.paged_attention(rng.standard_normal((1, H, D)), kc, vc, bt,
                                 np.array([ctx], np.int32), 0.5, "f64")
    expect = np.array([h // (H // Hk) + 1.0 for h in range(H)])
    np.testing.assert_allclose(out[0], np.repeat(expect[:, None], D, 1), rtol=0, atol=1e-14)


def test_value_affine_equivariance():
    # the weights sum to one, so out(a V + c) = a out(V) + c
    q, kc, vc, bt, cl, _, _ = _dense_case(3, 4, 2, 8, [7, 30, 64], 8, seed=8)
    o1 = oracle.paged_attention(q, kc, vc, bt, cl, 0.4, "f64")
    o2 = oracle.paged_attention(q, kc, 2.5 * vc - 1.25, bt, cl, 0.4, "f64")
    np.testing.assert_allclose(o2, 2.5 * o1 - 1.25, rtol=0, atol=1e-12)


def test_softmax_weights_sum_to_one_and_are_positive():
    q, kc, vc, bt, cl, _, _ = _dense_case(2, 4, 4, 16, [33, 129], 16, seed=9)
    for b in range(2):
        for h in range(4):
            w, _ = oracle.attention_weights(q, kc, vc, bt, cl, 0.25, "f64", b, h)
            assert w.shape == (cl[b],)
            assert np.all(w > 0)
            assert abs(w.sum() - 1.0) <= 1e-12


def test_empty_context_gives_zeros():
    q, kc, vc, bt, cl, _, _ = _dense_case(3, 2, 2, 8, [5, 0, 9], 4, seed=10)
    out = oracle.paged_attention(q, kc, vc, bt, cl, 0.5, "f64")
    assert np.all(out[1] == 0.0)
    assert np.any(out[0] != 0.0)


def test_physical_placement_does_not_change_the_result():
    # Paging changes where K/V live, not what is computed (page 2, demo 2):
    # the same contents on a different permutation of the pool give identical bits.
    w = workloads.llama8b_decode(num_seqs=3, dtype="f32")
    w.context_lens = np.array([40, 97, 16], np.int32)
    q = w.q_values()
    v1 = w.compact_host_view(range(3), rng_seed=1, include_newest=True)
    v2 = w.compact_host_view(range(3), rng_seed=2, include_newest=True)
    assert not np.array_equal(v1["block_tables"], v2["block_tables"])
    o1 = oracle.paged_attention(q, v1["key_cache"], v1["value_cache"], v1["block_tables"],
                                v1["context_lens"], w.scale, "f32")
    o2 = oracle.paged_attention(q, v2["key_cache"], v2["value_cache"], v2["block_tables"],
                                v2["context_lens"], w.scale, "f32")
    assert np.array_equal(o1, o2)


def test_block_size_invariance():
    # Same token contents at block sizes 8/16/32 (the mixed serving sweep) give
    # identical bits, because only the gather changes.
    outs = []
    for bs in (8, 16, 32):
        w = workloads.mixed_serving(block_size=bs, dtype="f32", num_seqs=6, extra_write=16)
        view = w.compact_host_view(range(6), include_newest=True)
        outs.append(oracle.paged_attention(w.q_values(), view["key_cache"], view["value_cache"],
                                           view["block_tables"], view["context_lens"], w.scale, "f32"))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_context_beyond_table_is_rejected():
    q, kc, vc, bt, cl, _, _ = _dense_case(1, 2, 2, 8, [9], 4, seed=11)
    with pytest.raises(ValueError):
        oracle.paged_attention(q, kc, vc, bt, np.array([bt.shape[1] * 4 + 1], np.int32), 1.0, "f64")


def test_bad_block_id_is_rejected():
    q, kc, vc, bt, cl, _, _ = _dense_case(1, 2, 2, 8, [9], 4, seed=12)
    bt = bt.copy()
    bt[0, 1] = kc.shape[0]
    with pytest.raises(ValueError):
        oracle.paged_attention(q, kc, vc, bt, cl, 1.0, "f64")


# --------------------------------------------------------------------------
# storage decoding (pinned against numpy / torch widening)
# --------------------------------------------------------------------------

def _roundtrip_ctx1(vals_storage, dtype):
    """Attention with one token returns V0 exactly, so out == decode(V0)."""
    n = vals_storage.shape[0]
    V = vals_storage.reshape(1, 1, 1, n)
    K = np.zeros_like(V)
    q = np.zeros((1, 1, n), dtype=vals_storage.dtype)
    return oracle.paged_attention(q, K, V, np.zeros((1, 1), np.int32), np.array([1], np.int32),
                                  1.0, dtype)[0, 0]


def test_f16_decoding_matches_numpy_for_every_finite_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    h = bits.view(np.float16)
    h = h[np.isfinite(h)]
    out = _roundtrip_ctx1(np.ascontiguousarray(h), "f16")
    assert np.array_equal(out, h.astype(np.float64))


def test_bf16_decoding_matches_torch_for_every_finite_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16)
    ref = t.to(torch.float64).numpy()
    keep = np.isfinite(ref)
    out = _roundtrip_ctx1(np.ascontiguousarray(bits[keep]), "bf16")
    assert np.array_equal(out, ref[keep])


# --------------------------------------------------------------------------
# scatter and block copy: hand-made fixtures
# --------------------------------------------------------------------------

def _rows(txt):
    return np.array([[float(x) for x in r.split()] for r in txt.split("|")])


def test_scatter_small_fixture():
    g = read_golden("scatter_small.txt")
    nb, bs, row = int(g["num_blocks"][0]), int(g["block_size"][0]), int(g["row_elems"][0])
    slots = np.array([int(x) for x in g["slots"][0].split()], np.int32)
    k = _rows(g["k_rows"][0])
    v = _rows(g["v_rows"][0])
    kc = np.zeros((nb, bs, row))
    vc = np.zeros_like(kc)
    bad = oracle.kv_write(k, v, slots, kc, vc, "f64")
    assert bad == 0
    ek = np.zeros_like(kc)
    ev = np.zeros_like(vc)
    for e in g["expect"]:
        blk, off, k0, k1, v0, v1 = [float(x) for x in e.split()]
        ek[int(blk), int(off)] = [k0, k1]
        ev[int(blk), int(off)] = [v0, v1]
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_scatter_counts_and_skips_invalid_slots():
    kc = np.zeros((2, 4, 3))
    vc = np.zeros_like(kc)
    k = np.ones((3, 3))
    bad = oracle.kv_write(k, k, np.array([8, -2, 1], np.int32), kc, vc, "f64")
    assert bad == 2
    assert kc[0, 1].tolist() == [1, 1, 1] and kc.sum() == 3


def test_scatter_is_bit_exact_for_bf16_bits():
    rng = np.random.default_rng(13)
    bits = rng.integers(0, 65536, size=(5, 8), dtype=np.uint16)
    kc = np.zeros((4, 4, 8), np.uint16)
    vc = np.zeros_like(kc)
    slots = np.array([3, 15, -1, 0, 9], np.int32)
    oracle.kv_write(bits, bits ^ 0xFFFF, slots, kc, vc, "bf16")
    flat_k, flat_v = kc.reshape(16, 8), vc.reshape(16, 8)
    for t, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(flat_k[s], bits[t]) and np.array_equal(flat_v[s], bits[t] ^ 0xFFFF)


def test_copy_small_fixture():
    g = read_golden("copy_small.txt")
    nb, bs, row = int(g["num_blocks"][0]), int(g["block_size"][0]), int(g["row_elems"][0])
    kc = np.array([10 * i + np.arange(bs * row) for i in range(nb)], float).reshape(nb, bs, row)
    vc = kc + 100
    pairs = _rows(g["pairs"][0]).astype(np.int32)
    bad = oracle.copy_blocks(kc, vc, pairs, "f64")
    assert bad == 0
    expect = [float(x) for x in g["expect_k_first"][0].split()]
    assert kc[:, 0, 0].tolist() == expect
    assert np.array_equal(kc[2], kc[0]) and np.array_equal(kc[1], kc[3])
    assert np.array_equal(vc[2], kc[0] + 100) and np.array_equal(vc[1], kc[3] + 100)
    assert kc[0].ravel().tolist() == [0, 1, 2, 3] and kc[3].ravel().tolist() == [30, 31, 32, 33]


def test_copy_skips_invalid_pairs():
    kc = np.arange(12.0).reshape(3, 2, 2)
    vc = kc.copy()
    bad = oracle.copy_blocks(kc, vc, np.array([[0, 3], [-1, 1], [2, 1]], np.int32), "f64")
    assert bad == 2
    assert np.array_equal(kc[1], kc[2])


# --------------------------------------------------------------------------
# the input generator: full-mantissa N(0, 1) stand-in, identical in numpy and
# torch, rounded to the storage dtypes exactly as torch's casts round
# --------------------------------------------------------------------------

def test_generator_values_full_mantissa_and_numpy_torch_agree():
    keys = np.arange(512, dtype=np.int64) * 977
    pos = np.arange(512, dtype=np.int64) * 13
    a = workloads.content_rows(5, 1, keys, pos, 1024)
    b = workloads.content_rows(5, 1, torch.from_numpy(keys), torch.from_numpy(pos), 1024).numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # every value is n / 2^21 for an odd integer n: an exact float32, within the stated bound
    n = a.astype(np.float64) * 2.0 ** 21
    assert np.all(n == np.round(n)) and np.all(np.mod(n, 2) == 1)
    assert np.abs(a).max() <= workloads.CONTENT_MAX
    # full mantissa: almost no value is exact in bf16 or fp16
    for dt in ("f16", "bf16"):
        r = workloads.rounded(a, dt)
        assert np.mean(r != a) > 0.99
    # an N(0, 1) stand-in: moments and the distance of the empirical CDF to the normal one
    x = np.sort(a.astype(np.float64).ravel())
    assert abs(x.mean()) < 0.01 and abs(x.std() - 0.998) < 0.01
    cdf = 0.5 * (1.0 + np.vectorize(math.erf)(x[::97] / math.sqrt(2.0)))
    emp = (np.arange(x.size)[::97] + 0.5) / x.size
    assert np.abs(cdf - emp).max() < 0.01


def test_storage_rounding_matches_torch_casts():
    """The host side of the parity tests rounds float32 to bf16 and fp16 with
    to_storage_numpy; the device side uses torch's casts. Both must round to
    nearest even: ties of either parity, carries into the exponent, overflow,
    subnormals, signed zeros, infinities and NaN."""
    rng = np.random.default_rng(9)
    hi = rng.integers(0, 1 << 16, size=4096, dtype=np.uint64)
    low = np.concatenate([np.full(1024, 0x8000), np.full(1024, 0x7FFF), np.full(1024, 0x8001),
                          rng.integers(0, 1 << 16, size=1024)]).astype(np.uint64)
    bits = ((hi << 16) | low).astype(np.uint32)
    x = bits.view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 3.3895314e38, -3.3895314e38, 65520.0, 65519.0,
                        6.0e-8, 2.0 ** -25, -(2.0 ** -24), 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                        1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], np.float32)
    x = np.concatenate([x, special, workloads.content_rows(1, 0, np.arange(64), np.arange(64), 256).ravel()])
    t = torch.from_numpy(x.copy())
    got = workloads.to_storage_numpy(x, "bf16")
    want = t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan]) and np.all(got[nan] == 0x7FC0)
    got16 = workloads.to_storage_numpy(x, "f16").view(np.uint16)
    want16 = t.to(torch.float16).numpy().view(np.uint16)
    assert np.array_equal(got16[~nan], want16[~nan])
    assert np.array_equal(workloads.rounded(x, "bf16")[~nan],
                          t.to(torch.bfloat16).float().numpy()[~nan])
