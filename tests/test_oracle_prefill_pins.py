"""Pins of the oracle's chunked-prefill attention (no GPU)."""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _host_case(pw, rng_seed=3):
    """Oracle inputs: compact paged cache with the chunk already written."""
    w = pw.base
    view = w.compact_host_view(range(w.num_seqs), rng_seed=rng_seed, include_newest=True)
    q = pw.q_values().astype(np.float32)
    return q, view


def _sdpa_chunk(q, K, V, q_len, scale):
    """torch float64 SDPA of one sequence's chunk with an explicit causal mask:
    query i (position ctx - q_len + i) sees keys 0..ctx - q_len + i."""
    ctx = K.shape[0]
    H, Hk = q.shape[1], K.shape[1]
    qt = torch.from_numpy(q.astype(np.float64).transpose(1, 0, 2))[None]          # [1, H, q_len, D]
    kt = torch.from_numpy(np.ascontiguousarray(K.astype(np.float64).transpose(1, 0, 2)))[None]
    vt = torch.from_numpy(np.ascontiguousarray(V.astype(np.float64).transpose(1, 0, 2)))[None]
    pos = np.arange(ctx - q_len, ctx)[:, None]
    mask = torch.from_numpy(np.arange(ctx)[None, :] <= pos)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale,
                                                         enable_gqa=(H != Hk))
    return o[0].numpy().transpose(1, 0, 2)


@pytest.mark.parametrize("H,Hk,bs", [(8, 2, 16), (4, 4, 4), (6, 1, 32)])
def test_prefill_matches_torch_sdpa_with_causal_mask(H, Hk, bs):
    prior = np.array([0, 5, 37, 100], np.int32)
    q_lens = np.array([7, 1, 20, 33], np.int32)
    pw = workloads.make_prefill("pin", 9, prior, q_lens, H, Hk, 32, bs, "f32")
    q, view = _host_case(pw)
    out = oracle.paged_prefill(q, view["key_cache"], view["value_cache"], view["block_tables"],
                               view["context_lens"], pw.query_start_loc, pw.base.scale, "f32")
    qs = pw.query_start_loc
    for b in range(pw.base.num_seqs):
        K, V = pw.base.contiguous_kv(b)
        ref = _sdpa_chunk(q[qs[b]:qs[b + 1]], K, V, int(q_lens[b]), pw.base.scale)
        np.testing.assert_allclose(out[qs[b]:qs[b + 1]], ref, rtol=0, atol=1e-12)


def test_full_prefill_matches_sdpa_is_causal():
    prior = np.zeros(2, np.int32)
    q_lens = np.array([19, 40], np.int32)
    pw = workloads.make_prefill("pin_full", 4, prior, q_lens, 4, 2, 16, 8, "f32")
    q, view = _host_case(pw)
    out = oracle.paged_prefill(q, view["key_cache"], view["value_cache"], view["block_tables"],
                               view["context_lens"], pw.query_start_loc, pw.base.scale, "f32")
    qs = pw.query_start_loc
    for b in range(2):
        K, V = pw.base.contiguous_kv(b)
        qt = torch.from_numpy(q[qs[b]:qs[b + 1]].astype(np.float64).transpose(1, 0, 2))[None]
        kt = torch.from_numpy(np.ascontiguousarray(K.astype(np.float64).transpose(1, 0, 2)))[None]
        vt = torch.from_numpy(np.ascontiguousarray(V.astype(np.float64).transpose(1, 0, 2)))[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=pw.base.scale,
                                                               enable_gqa=True)[0].numpy().transpose(1, 0, 2)
        np.testing.assert_allclose(out[qs[b]:qs[b + 1]], ref, rtol=0, atol=1e-12)


def test_single_query_chunks_reduce_to_decode():
    # a chunk of one token is a decode step: same result as the (pinned) decode oracle
    prior = np.array([4, 0, 63, 200], np.int32)
    pw = workloads.make_prefill("pin_dec", 12, prior, np.ones(4, np.int32), 8, 2, 64, 16, "f32")
    q, view = _host_case(pw)
    out = oracle.paged_prefill(q, view["key_cache"], view["value_cache"], view["block_tables"],
                               view["context_lens"], pw.query_start_loc, pw.base.scale, "f32")
    dec = oracle.paged_attention(q, view["key_cache"], view["value_cache"], view["block_tables"],
                                 view["context_lens"], pw.base.scale, "f32")
    assert np.array_equal(out, dec)


def test_last_query_of_a_chunk_equals_decode_of_the_whole_context():
    prior = np.array([10, 77], np.int32)
    q_lens = np.array([5, 16], np.int32)
    pw = workloads.make_prefill("pin_last", 13, prior, q_lens, 4, 2, 32, 8, "f32")
    q, view = _host_case(pw)
    out = oracle.paged_prefill(q, view["key_cache"], view["value_cache"], view["block_tables"],
                               view["context_lens"], pw.query_start_loc, pw.base.scale, "f32")
    last = pw.query_start_loc[1:] - 1
    dec = oracle.paged_attention(np.ascontiguousarray(q[last]), view["key_cache"], view["value_cache"],
                                 view["block_tables"], view["context_lens"], pw.base.scale, "f32")
    assert np.array_equal(out[last], dec)


def test_prefill_rejects_a_chunk_longer_than_the_context():
    pw = workloads.make_prefill("pin_bad", 1, np.array([3], np.int32), np.array([4], np.int32), 2, 2, 16, 4, "f32")
    q, view = _host_case(pw)
    with pytest.raises(ValueError):
        oracle.paged_prefill(q, view["key_cache"], view["value_cache"], view["block_tables"],
                             np.array([3], np.int32), pw.query_start_loc, 1.0, "f32")
