"""Shared drivers for the GPU parity tests: run one workload through the library
and through the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

TOL = {"f32": (1e-5, 1e-5), "f16": (2e-2, 2e-3), "bf16": (2e-2, 2e-3)}


def pa_mod():
    from __graft_entry__ import build
    build()
    import paged_kv_cache_261_gb300 as pa
    return pa


def dev():
    return torch.device("cuda", 0)


def gpu_decode(w: workloads.DecodeWorkload, partition_size=0, max_context_len=0, poison=True,
               write_newest=True, workspace=None):
    """Fill a device cache, scatter the newest tokens with paged_kv_write, decode.

    Unused cache slots hold NaN when poison is set, so any read of a slot that
    is not part of a context shows up in the output."""
    pa = pa_mod()
    d = dev()
    dt = workloads.torch_dtype(w.dtype)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    fill = float("nan") if poison else 0.0
    kc = torch.full(shape, fill, dtype=dt, device=d)
    vc = torch.full(shape, fill, dtype=dt, device=d)
    w.fill_cache_torch(kc, vc, include_newest=not write_newest)
    if write_newest:
        kn, vn = w.newest_kv(like=kc)
        pa.paged_kv_write(kn.to(dt).contiguous(), vn.to(dt).contiguous(),
                          torch.as_tensor(w.slot_mapping, device=d), kc, vc)
    q = w.q_values(like=kc).to(dt).contiguous()
    out = torch.full_like(q, float("nan"))
    pa.paged_attention_decode(out, q, kc, vc, torch.as_tensor(w.block_tables, device=d),
                              torch.as_tensor(w.context_lens, device=d), w.scale,
                              block_size=w.block_size, num_kv_heads=w.num_kv_heads,
                              max_context_len=max_context_len, partition_size=partition_size,
                              workspace=workspace)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_decode(w: workloads.DecodeWorkload, seqs) -> np.ndarray:
    """float64 [len(seqs), H, D]: oracle scatter of the newest tokens + oracle decode."""
    seqs = np.asarray(seqs, dtype=np.int64)
    view = w.compact_host_view(seqs, include_newest=False)
    kc = workloads.to_storage_numpy(view["key_cache"], w.dtype)
    vc = workloads.to_storage_numpy(view["value_cache"], w.dtype)
    kn, vn = w.newest_kv()
    row = w.num_kv_heads * w.head_dim
    oracle.kv_write(workloads.to_storage_numpy(kn[seqs].reshape(-1, row), w.dtype),
                    workloads.to_storage_numpy(vn[seqs].reshape(-1, row), w.dtype),
                    view["slot_mapping"], kc, vc, w.dtype)
    q = workloads.to_storage_numpy(w.q_values()[seqs], w.dtype)
    return oracle.paged_attention(q, kc, vc, view["block_tables"], view["context_lens"], w.scale,
                                  w.dtype, num_threads=oracle.num_host_threads())


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    tmax, tmean = TOL[dtype]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= tmax, f"{what}: max abs err {err.max():.3e} > {tmax}"
    assert err.mean() <= tmean, f"{what}: mean abs err {err.mean():.3e} > {tmean}"
    return float(err.max()), float(err.mean())


def check_newest_rows(w: workloads.DecodeWorkload, kc: torch.Tensor, vc: torch.Tensor):
    """Bit-exact: the rows paged_kv_write put at each newest slot."""
    live = w.slot_mapping >= 0
    slots = torch.as_tensor(w.slot_mapping[live].astype(np.int64), device=kc.device)
    row = w.num_kv_heads * w.head_dim
    got_k = kc.view(-1, row)[slots].float().cpu().numpy()
    got_v = vc.view(-1, row)[slots].float().cpu().numpy()
    kn, vn = w.newest_kv()
    assert np.array_equal(got_k, workloads.rounded(kn.reshape(-1, row)[live], w.dtype))
    assert np.array_equal(got_v, workloads.rounded(vn.reshape(-1, row)[live], w.dtype))


# ---------------------------------------------------------------------------
# 8-bit (E4M3) cache
# ---------------------------------------------------------------------------

FP8_POISON = 0x7F      # the E4M3 NaN pattern in every slot no context uses


def gpu_decode_fp8(w: workloads.DecodeWorkload, partition_size=0, max_context_len=0, write_newest=True,
                   k_scale=workloads.FP8_SCALE, v_scale=workloads.FP8_SCALE, workspace=None):
    """uint8 caches filled with codes, the newest tokens scattered (quantised) from
    w.dtype rows with paged_kv_write_fp8, then the 8-bit decode."""
    pa = pa_mod()
    d = dev()
    dt = workloads.torch_dtype(w.dtype)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, FP8_POISON, dtype=torch.uint8, device=d)
    vc = torch.full(shape, FP8_POISON, dtype=torch.uint8, device=d)
    w.fill_cache_torch(kc, vc, include_newest=not write_newest)
    if write_newest:
        kn, vn = w.newest_kv(like=kc)
        pa.paged_kv_write_fp8(kn.to(dt).contiguous(), vn.to(dt).contiguous(),
                              torch.as_tensor(w.slot_mapping, device=d), kc, vc, k_scale, v_scale)
    q = w.q_values(like=kc).to(dt).contiguous()
    out = torch.full_like(q, float("nan"))
    pa.paged_attention_decode_fp8(out, q, kc, vc, torch.as_tensor(w.block_tables, device=d),
                                  torch.as_tensor(w.context_lens, device=d), w.scale, k_scale, v_scale,
                                  max_context_len=max_context_len, partition_size=partition_size,
                                  workspace=workspace)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_decode_fp8(w: workloads.DecodeWorkload, seqs, write_newest=True, k_scale=workloads.FP8_SCALE,
                      v_scale=workloads.FP8_SCALE) -> np.ndarray:
    """float64 [len(seqs), H, D]: oracle 8-bit scatter of the newest tokens + oracle decode."""
    seqs = np.asarray(seqs, dtype=np.int64)
    view = w.compact_host_view(seqs, include_newest=not write_newest, codes=True)
    kc, vc = view["key_cache"], view["value_cache"]
    if write_newest:
        kn, vn = w.newest_kv()
        row = w.num_kv_heads * w.head_dim
        oracle.kv_write_fp8(workloads.to_storage_numpy(kn[seqs].reshape(-1, row), w.dtype),
                            workloads.to_storage_numpy(vn[seqs].reshape(-1, row), w.dtype),
                            view["slot_mapping"], kc, vc, k_scale, v_scale, w.dtype)
    q = workloads.to_storage_numpy(w.q_values()[seqs], w.dtype)
    return oracle.paged_attention_fp8(q, kc, vc, view["block_tables"], view["context_lens"], w.scale,
                                      k_scale, v_scale, w.dtype, num_threads=oracle.num_host_threads())
