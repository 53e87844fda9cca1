"""A decode step -- scatter of the newest tokens, then decode -- captured in a CUDA
graph and replayed.

The replays give the eagerly computed outputs bit for bit and follow new inputs
written in place (a graph reads the buffers it was captured with, not copies).
The calls inside launch with programmatic stream serialization, which capture
keeps as programmatic edges; with a caller's workspace they allocate nothing and
never synchronise, which is what makes a step capturable. Both cache paths: 16-bit
and 8-bit (E4M3)."""
import pytest
import torch

import workloads
from gpu_cases import dev, pa_mod

pytestmark = pytest.mark.gpu

S = workloads.FP8_SCALE


@pytest.fixture(scope="module")
def pa():
    return pa_mod()


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_step_replays_as_a_cuda_graph(pa, fp8):
    w = workloads.llama8b_decode(num_seqs=16)
    d = dev()
    dt = workloads.torch_dtype(w.dtype)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.zeros(shape, dtype=torch.uint8 if fp8 else dt, device=d)
    vc = torch.zeros_like(kc)
    w.fill_cache_torch(kc, vc, include_newest=False)
    kn, vn = w.newest_kv(like=kc)
    kn, vn = kn.to(dt).contiguous(), vn.to(dt).contiguous()
    q = w.q_values(like=kc).to(dt).contiguous()
    slots = torch.as_tensor(w.slot_mapping, device=d)
    bt = torch.as_tensor(w.block_tables, device=d)
    cl = torch.as_tensor(w.context_lens, device=d)
    mc = int(w.context_lens.max())
    ws = torch.empty(max(pa.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim, mc, 0), 16),
                     dtype=torch.uint8, device=d)
    out = torch.full_like(q, float("nan"))

    def step():
        if fp8:
            pa.paged_kv_write_fp8(kn, vn, slots, kc, vc, S, S)
            pa.paged_attention_decode_fp8(out, q, kc, vc, bt, cl, w.scale, S, S, max_context_len=mc, workspace=ws)
        else:
            pa.paged_kv_write(kn, vn, slots, kc, vc)
            pa.paged_attention_decode(out, q, kc, vc, bt, cl, w.scale, max_context_len=mc, workspace=ws)

    # first calls outside capture (per-device set-up: kernel attributes, error word)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = out.clone()
    assert torch.isfinite(ref.float()).all()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)

    # new query values in place: the replay computes with them, as an eager step does
    q.copy_((q.float() * -0.5).to(dt))
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    got = out.clone()
    out.fill_(float("nan"))
    step()
    torch.cuda.synchronize()
    assert torch.equal(got, out) and not torch.equal(got, ref)
    assert pa.get_device_error() == 0
