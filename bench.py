"""Benchmark of the paged decode step on GB300.

One step = one pass of the hot path over one synthetic batch: the scatter of
the step's new tokens into their cache slots (paged_kv_write), the
copy-on-write block copies when the workload has them (copy_blocks), and decode
attention over the paged cache (split-K partition kernel + merge kernel).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload llama8b_decode|long_context|mixed_serving|shared_prefix|chunked_prefill]

Prints one JSON line (rank 0). ``value`` is algorithmic bytes per step (K and V
of every context once, q, out, the table entries and lengths used, plus the
written and copied rows) divided by the device time per step, in GB/s, summed
over ranks (each rank runs its own replica of the workload: the path has no
exchange step). The reference arm (--impl reference) times the CPU oracle on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged decode attn KV GB/s & tokens/s on 1×GB300; fraction of HBM peak"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Device-code sources of the kernel each workload's roofline line is about; a
# recorded DRAM-traffic figure is used only while these files are unchanged.
_KERNEL_SOURCES = {
    "decode_tc": ["decode_tc.cu", "decode_order.cuh", "sm100.cuh", "common.cuh", "tma_maps.cuh", "kernels.h"],
    "decode_fp8": ["decode_fp8.cu", "decode_order.cuh", "sm100.cuh", "common.cuh", "tma_maps.cuh", "kernels.h",
                   "kernels_fp8.h", "fp8_encode.cuh"],
    "prefill_tc": ["prefill_tc.cu", "prefill_common.cuh", "sm100.cuh", "common.cuh", "tma_maps.cuh", "kernels.h"],
    # the sharing-aware decode's two passes: group mode of the prefill kernel + the
    # tensor-core decode (its record is the DRAM bytes of both launches of one call)
    "shared_decode": ["prefill_tc.cu", "prefill_common.cuh", "decode_tc.cu", "decode_order.cuh", "sm100.cuh",
                      "common.cuh", "tma_maps.cuh", "kernels.h"],
}

DECODE_WORKLOADS = ("llama8b_decode", "long_context", "mixed_serving")
FP8_WORKLOADS = tuple(n + "_fp8" for n in DECODE_WORKLOADS)


def traffic_family(workload: str) -> str:
    """The kernel family whose sources key a workload's DRAM-traffic record."""
    if workload == "chunked_prefill":
        return "prefill_tc"
    if workload == "shared_prefix":
        return "shared_decode"
    return "decode_fp8" if workload.endswith("_fp8") else "decode_tc"


def base_workload(name: str):
    """(decode workload builder, 8-bit cache?) of a workload name."""
    fp8 = name.endswith("_fp8")
    base = name[: -len("_fp8")] if fp8 else name
    return {"llama8b_decode": workloads.llama8b_decode, "long_context": workloads.long_context,
            "mixed_serving": workloads.mixed_serving}[base], fp8


def code_only(text: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed to one
    space: what a compiler sees, so that a change to prose alone keeps a
    kernel's recorded counters valid. String and character literals are kept
    as written."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_digest(kernel: str = "decode_tc"):
    """Digest of the code (comments and layout aside) of a kernel's sources."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_261_gb300", "csrc")
    for name in _KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str = "decode_tc"):
    """DRAM bytes per launch of the workload's dominant kernel from the committed
    ncu summary, if it was taken on the current sources of that kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
        ent = rec.get(workload)
        if ent and ent.get("source_digest") == source_digest(kernel):
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.path = os.path.join("/tmp", f"pa_clocks_{os.getpid()}.csv")
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.remove(self.path)
        return self.summarise(lines)

    @staticmethod
    def summarise(lines):
        """Median SM clock, the highest max clock and the throttle reasons seen
        (any sample with the reason "Active") from the CSV samples; None if no
        sample parsed."""
        rows = []
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 8:
                rows.append(parts)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def max_over_ranks(ms: float, device) -> float:
    """Slowest rank's time (the job is done when the last replica is done)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world: int, step_bytes: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs one replica of the step."""
    return world * step_bytes / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# device state of one workload
# ---------------------------------------------------------------------------

class Step:
    """Device-resident inputs of one step and the calls that run it."""

    def __init__(self, name: str, device):
        import torch

        import paged_kv_cache_261_gb300 as pa
        self.pa = pa
        self.name = name
        self.device = device
        self.copy_pairs = None
        self.copy_bytes = 0
        self.fp8 = False
        if name == "shared_prefix":
            w, extra = self._shared_prefix_state()
        else:
            build_w, self.fp8 = base_workload(name)
            w = build_w()
            extra = None
        self.w = w
        self.k_scale = self.v_scale = workloads.FP8_SCALE
        dt = workloads.torch_dtype(w.dtype)
        self.tdtype = dt
        shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
        cdt = torch.uint8 if self.fp8 else dt           # 8-bit caches hold E4M3 codes
        self.kc = torch.zeros(shape, dtype=cdt, device=device)
        self.vc = torch.zeros(shape, dtype=cdt, device=device)
        w.fill_cache_torch(self.kc, self.vc, include_newest=False)
        if name.startswith("mixed_serving"):
            k, v = w.extra_write_rows(like=self.kc)
            self.slots = torch.as_tensor(w.extra_write_slots, device=device)
        else:
            k, v = w.newest_kv(like=self.kc)
            self.slots = torch.as_tensor(w.slot_mapping, device=device)
        self.k_new = k.to(dt).contiguous()
        self.v_new = v.to(dt).contiguous()
        if name.startswith("mixed_serving"):
            # the decode batch's own newest tokens are already in the cache
            kn, vn = w.newest_kv(like=self.kc)
            self.write(kn.to(dt).contiguous(), vn.to(dt).contiguous(),
                       torch.as_tensor(w.slot_mapping, device=device))
        if extra is not None:
            self.copy_pairs = torch.as_tensor(extra, device=device)
            es = 2
            self.copy_bytes = 2 * 2 * extra.shape[0] * w.block_size * w.row_elems * es
        self.q = w.q_values(like=self.kc).to(dt).contiguous()
        self.out = torch.empty_like(self.q)
        self.bt = torch.as_tensor(w.block_tables, device=device)
        self.cl = torch.as_tensor(w.context_lens, device=device)
        self.max_ctx = int(w.context_lens.max())
        # the long-context configuration names its split-K partition (512 tokens); the
        # others leave it to the library's automatic choice
        self.part = 512 if name.startswith("long_context") else 0
        self.ws = torch.empty(max(pa.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim,
                                                            self.max_ctx, self.part), 16),
                              dtype=torch.uint8, device=device)
        self.shared = None
        self.unique_kv_bytes = None
        if name == "shared_prefix":
            # each prompt's shared blocks are read once for its 8 samples
            pl, gm = pa.prefix_groups(w.block_tables, w.context_lens, w.block_size, max_members=8)
            self.shared = (torch.as_tensor(pl, device=device), torch.as_tensor(gm, device=device),
                           int(pl.max()) if pl.size else 0)
            self.ws = torch.empty(pa.decode_shared_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim,
                                                                   self.max_ctx, 0), dtype=torch.uint8,
                                  device=device)
            lead_prefix = sum(int(pl[row[0]]) for row in gm)
            uniq_tokens = int((w.context_lens.astype(np.int64) - pl).sum()) + lead_prefix
            self.unique_kv_bytes = uniq_tokens * w.row_elems * 2 * 2
        es = {"f32": 4, "f16": 2, "bf16": 2}[w.dtype]
        ce = 1 if self.fp8 else es                        # bytes of one cache element
        ab = w.algorithmic_bytes(cache_elem_bytes=ce)
        self.decode_bytes = ab["decode"]
        self.kv_bytes = ab["kv"]
        self.decode_unique_bytes = self.decode_bytes
        if self.unique_kv_bytes is not None:
            self.decode_unique_bytes = self.decode_bytes - self.kv_bytes + self.unique_kv_bytes
        ntok = int(self.slots.shape[0])
        self.write_bytes = 2 * ntok * w.row_elems * (es + ce) + 4 * ntok
        self.step_bytes = self.decode_bytes + self.write_bytes + self.copy_bytes
        # a step whose new tokens are the batch's own newest ones (not mixed serving's
        # extra write, not the 8-bit or shared paths) runs as one decode-with-append
        # call: the tensor-core decode writes each token before reading its block
        self.append = self.shared is None and not name.startswith("mixed_serving")
        self.launches_per_step = (0 if self.append else 1) + (1 if self.copy_pairs is not None else 0) + 1 + (
            1 if pa.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim, self.max_ctx, self.part) else 0)
        if self.shared is not None:
            self.launches_per_step = 1 + 1 + 3     # copy, write, shared pass + private pass + merge
        torch.cuda.synchronize()

    def _shared_prefix_state(self):
        """Allocator replay of the shared-prefix workload (library allocator).
        The step's copy_blocks duplicates each prompt's partial block into a
        spare block per copy-on-write pair, which leaves the decode inputs intact."""
        pa = self.pa
        sc = workloads.shared_prefix()
        npairs = (sc.samples_per_prompt - 1) * sc.num_prompts
        nb = sc.pool_blocks() + npairs
        a = pa.BlockAllocator(nb, sc.block_size)
        pairs = []
        for p in range(sc.num_prompts):
            a.add_seq(p)
            a.append(p, sc.prompt_len)
            for j in range(sc.samples_per_prompt):
                a.fork(p, 1000 + p * sc.samples_per_prompt + j)
            a.free_seq(p)
        for s in range(sc.num_samples):
            _, pr = a.append(1000 + s, int(sc.private[s]) + 1)
            pairs += pr.tolist()
        spare = [a.alloc() for _ in range(len(pairs))]
        ids = np.arange(sc.num_samples) + 1000
        mb = max(len(a.block_table(int(i))) for i in ids)
        tables, _ = a.export(ids, mb)
        w = sc.workload(tables, nb)
        extra = np.array([[src, dst] for (src, _), dst in zip(pairs, spare)], np.int32)
        return w, extra

    def write(self, k, v, slots):
        if self.fp8:
            self.pa.paged_kv_write_fp8(k, v, slots, self.kc, self.vc, self.k_scale, self.v_scale)
        else:
            self.pa.paged_kv_write(k, v, slots, self.kc, self.vc)

    def decode(self, q, bt, cl, prefix=None, new=None):
        """The decode call; new = (k, v, slots) of the step's tokens for a decode with append."""
        pa = self.pa
        if new is not None and self.fp8:
            k, v, slots = new
            pa.paged_attention_decode_fp8_append(self.out, q, k, v, slots, self.kc, self.vc, bt, cl, self.w.scale,
                                                 self.k_scale, self.v_scale, max_context_len=self.max_ctx,
                                                 partition_size=self.part, workspace=self.ws)
        elif new is not None:
            k, v, slots = new
            pa.paged_attention_decode_append(self.out, q, k, v, slots, self.kc, self.vc, bt, cl, self.w.scale,
                                             max_context_len=self.max_ctx, partition_size=self.part,
                                             workspace=self.ws)
        elif self.shared is not None:
            pl, gm, mp = self.shared if prefix is None else prefix
            pa.paged_attention_decode_shared(self.out, q, self.kc, self.vc, bt, cl, pl, gm, self.w.scale,
                                             max_context_len=self.max_ctx, max_prefix_len=mp, workspace=self.ws)
        elif self.fp8:
            pa.paged_attention_decode_fp8(self.out, q, self.kc, self.vc, bt, cl, self.w.scale, self.k_scale,
                                          self.v_scale, max_context_len=self.max_ctx, partition_size=self.part,
                                          workspace=self.ws)
        else:
            pa.paged_attention_decode(self.out, q, self.kc, self.vc, bt, cl, self.w.scale,
                                      max_context_len=self.max_ctx, partition_size=self.part, workspace=self.ws)

    def decode_call(self):
        """The step's decode call alone (with its write when it is a decode with append)."""
        self.decode(self.q, self.bt, self.cl, new=(self.k_new, self.v_new, self.slots) if self.append else None)

    def run(self):
        """One step: copy-on-write copies, the scatter of the new tokens, the decode."""
        if self.copy_pairs is not None:
            self.pa.copy_blocks(self.kc, self.vc, self.copy_pairs)
        if not self.append:
            self.write(self.k_new, self.v_new, self.slots)
        self.decode_call()

    def config(self):
        w = self.w
        return {"workload": self.name, "num_seqs": w.num_seqs, "num_heads": w.num_heads,
                "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                "num_blocks": w.num_blocks, "context_total": int(w.context_lens.sum()),
                "context_min": int(w.context_lens.min()), "context_max": int(w.context_lens.max()),
                "written_tokens": int(self.slots.shape[0]),
                "write": ("fused: decode with append (each sequence's new token written by the decode kernel)"
                          if self.append else "separate scatter launch"),
                "copied_blocks": 0 if self.copy_pairs is None else int(self.copy_pairs.shape[0]),
                "partition_size": (self.pa.decode_shared_partition_size(w.num_seqs, int(self.shared[1].shape[0]),
                                                                        w.num_kv_heads, self.shared[2], self.max_ctx)
                                   if self.shared is not None else
                                   self.pa.decode_partition_size(w.num_seqs, self.max_ctx, self.part)),
                "shared_prefix_decode": self.shared is not None,
                "unique_kv_bytes": self.unique_kv_bytes,
                "kv_cache": (f"e4m3 codes, k_scale = v_scale = {self.k_scale:.9g}" if self.fp8 else w.dtype),
                "decode_kernel": "decode_fp8" if self.fp8 else os.environ.get("PA_DECODE_KERNEL", "auto"),
                "l2": self.l2_note()}

    def l2_note(self):
        mib = 2.0 ** 20
        if self.unique_kv_bytes is not None:
            return (f"{self.unique_kv_bytes / mib:.0f} MiB of unique K/V per step vs {L2_BYTES / mib:.0f} MiB L2: "
                    f"steps run back to back (no flush); the decode roofline times each call after an L2 flush")
        return (f"inputs larger than L2: {self.kv_bytes / 1e9:.2f} GB of K/V read per step "
                f"vs {L2_BYTES / mib:.0f} MiB L2; no flush")


class PrefillStep:
    """Chunked-prefill step: scatter the chunk's K/V, then every chunk row attends."""

    def __init__(self, device):
        import torch

        import paged_kv_cache_261_gb300 as pa
        self.pa = pa
        self.name = "chunked_prefill"
        self.pw = pw = workloads.chunked_prefill()
        w = pw.base
        self.w = w
        dt = workloads.torch_dtype(w.dtype)
        shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
        self.kc = torch.zeros(shape, dtype=dt, device=device)
        self.vc = torch.zeros(shape, dtype=dt, device=device)
        workloads.fill_prior_torch(pw, self.kc, self.vc)
        k, v = pw.chunk_kv(like=self.kc)
        self.k_new, self.v_new = k.to(dt).contiguous(), v.to(dt).contiguous()
        self.slots = torch.as_tensor(pw.chunk_slots(), device=device)
        self.q = pw.q_values(like=self.kc).to(dt).contiguous()
        self.out = torch.empty_like(self.q)
        self.bt = torch.as_tensor(w.block_tables, device=device)
        self.cl = torch.as_tensor(w.context_lens, device=device)
        self.qs = torch.as_tensor(pw.query_start_loc, device=device)
        self.max_q = int(pw.q_lens.max())
        self.flops = pw.flops()
        self.launches_per_step = 2
        torch.cuda.synchronize()

    def prefill(self):
        self.pa.paged_attention_prefill(self.out, self.q, self.kc, self.vc, self.bt, self.cl, self.qs,
                                        self.w.scale, self.max_q)

    def run(self):
        self.pa.paged_kv_write(self.k_new, self.v_new, self.slots, self.kc, self.vc)
        self.prefill()

    def config(self):
        w, pw = self.w, self.pw
        return {"workload": self.name, "num_seqs": w.num_seqs, "num_heads": w.num_heads,
                "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                "query_tokens": pw.total_q, "chunk": self.max_q,
                "prior_min": int((w.context_lens - pw.q_lens).min()),
                "prior_max": int((w.context_lens - pw.q_lens).max()),
                "l2": self.l2_note()}

    def l2_note(self):
        w, pw = self.w, self.pw
        mib = 2.0 ** 20
        row = w.num_kv_heads * w.head_dim * 2
        kv = int(w.context_lens.sum()) * row * 2
        q = pw.total_q * w.num_heads * w.head_dim * 2
        return (f"inputs larger than L2: {q / mib:.0f} MiB of queries + {kv / mib:.0f} MiB of K/V read per step "
                f"(+ {q / mib:.0f} MiB of output and {pw.total_q * row * 2 / mib:.0f} MiB of chunk K/V written) "
                f"vs {L2_BYTES / mib:.0f} MiB L2; no flush")


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------

SETTLE_S = 0.3          # warm-up wall time while the clock sampler starts
KERNEL_WARM = 10        # untimed calls before a kernel-timing loop
KERNEL_RUNS = 5         # event-bracketed runs of back-to-back calls
KERNEL_CALLS = 50       # calls per run
BRACKETED_CALLS = 50    # individually bracketed calls (upper-bound cross-check)


def warm_up(torch, step, warmup: int, min_s: float = SETTLE_S) -> int:
    """At least `warmup` untimed steps, continuing until min_s of wall time has
    passed so that clocks have settled under load when the timed region starts
    (the clock sampler starts meanwhile, with the GPU busy rather than idle).
    Returns the number of warm-up steps run."""
    n = 0
    t = time.perf_counter()
    while n < warmup or time.perf_counter() - t < min_s:
        for _ in range(8):
            step()
            n += 1
        torch.cuda.synchronize()
    return n


def time_calls(torch, call, runs: int = KERNEL_RUNS, calls: int = KERNEL_CALLS, warm: int = KERNEL_WARM):
    """Device time of one call in steady state: `warm` untimed calls, then `runs`
    runs of `calls` back-to-back calls, each run between two CUDA events on the
    launching stream. Returns (median over the runs of ms per call, calls timed)."""
    for _ in range(warm):
        call()
    torch.cuda.synchronize()
    per = []
    for _ in range(runs):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(calls):
            call()
        b.record()
        b.synchronize()
        per.append(a.elapsed_time(b) / calls)
    return statistics.median(per), runs * calls


def time_calls_bracketed(torch, call, n: int = BRACKETED_CALLS, flush=None):
    """Median ms of `n` calls each bracketed alone by two CUDA events (so none
    overlaps its predecessor's tail). flush: a uint8 CUDA buffer larger than L2,
    overwritten before every call so that no call finds its inputs in L2."""
    evs = []
    for _ in range(n):
        if flush is not None:
            flush.fill_(0x5A)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(x.elapsed_time(y) for x, y in evs)


def l2_flush_buffer(torch, device):
    return torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)


def checked_roofline(achieved: float, peak: float, kernel_ms: float, ms_per_step: float, tol: float = 1.05):
    """frac, or None with the reason, when the kernel time or the rate is not
    physically consistent with the step it sits in."""
    if kernel_ms > tol * ms_per_step:
        return None, f"kernel time {kernel_ms:.4f} ms exceeds the step's {ms_per_step:.4f} ms"
    if achieved > 1.2 * peak:
        return None, f"achieved {achieved:.0f} above 1.2 x peak {peak:.0f}"
    return achieved / peak, None


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except Exception:
        return {}


def run_prefill(args, device, rank, world):
    """Timed loop of the chunked-prefill step (TFLOP/s of causal attention)."""
    import torch
    st = PrefillStep(device)
    st.run()
    torch.cuda.synchronize()
    if st.pa.get_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")
    sampler = ClockSampler(None) if rank == 0 else None
    nwarm = warm_up(torch, st.run, max(args.warmup, 3))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record()
    for _ in range(args.steps):
        st.run()
    t1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler is not None else None
    ms = max_over_ranks(t0.elapsed_time(t1), device) / args.steps
    kern_ms, ncalls = time_calls(torch, st.prefill)
    peaks = load_peaks()
    # the kernel is timed alone, in short runs (clocks stay at their maximum), so the
    # denominator is the burst GEMM figure, not the power-capped sustained one
    peak = float(peaks.get("bf16_tflops", 1900.0))
    achieved = st.flops / (kern_ms * 1e-3) / 1e12
    frac, why = checked_roofline(achieved, peak, kern_ms, ms)
    line = {"metric": "paged chunked-prefill attention TFLOP/s on 1×GB300 (causal, packed chunks)",
            "value": world * st.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": nwarm, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": st.w.dtype, "data": "synthetic",
            "config": st.config(), "tokens_per_s": world * st.pw.total_q / (ms * 1e-3),
            "roofline": {"kernel": "prefill_tc_kernel", "bound": "tensor", "achieved": achieved, "peak": peak,
                         "peak_kind": "measured bf16_tflops (burst)" if "bf16_tflops" in peaks
                         else "fallback", "unit": "TFLOP/s", "frac": frac,
                         "algorithmic_flops_per_launch": st.flops, "kernel_ms": kern_ms,
                         "timed_launches": ncalls,
                         "timing": f"median over {KERNEL_RUNS} event-bracketed runs of {KERNEL_CALLS} back-to-back "
                                   f"prefill calls, after the timed steps",
                         "traffic": recorded_traffic("chunked_prefill", traffic_family("chunked_prefill"))},
            "gpu_launches": st.launches_per_step * args.steps, "clocks": clocks}
    if why:
        line["roofline"]["frac_null_reason"] = why
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(w, n_seqs: int, fp8: bool = False):
    """Host inputs of the oracle for the first n_seqs sequences (storage dtype;
    E4M3 codes for an 8-bit cache)."""
    seqs = np.arange(n_seqs)
    view = w.compact_host_view(seqs, include_newest=False, codes=fp8)
    if fp8:
        kc, vc = view["key_cache"], view["value_cache"]
    else:
        kc = workloads.to_storage_numpy(view["key_cache"], w.dtype)
        vc = workloads.to_storage_numpy(view["value_cache"], w.dtype)
    kn, vn = w.newest_kv()
    row = w.row_elems
    kn = workloads.to_storage_numpy(kn[seqs].reshape(-1, row), w.dtype)
    vn = workloads.to_storage_numpy(vn[seqs].reshape(-1, row), w.dtype)
    q = workloads.to_storage_numpy(w.q_values()[seqs], w.dtype)
    return dict(kc=kc, vc=vc, kn=kn, vn=vn, q=q, slots=view["slot_mapping"], bt=view["block_tables"],
                cl=view["context_lens"], fp8=fp8)


def oracle_step(w, s, threads):
    """One oracle pass over the sample: newest-token scatter, then decode."""
    import oracle
    kc, vc = s["kc"].copy(), s["vc"].copy()
    if s["fp8"]:
        S = workloads.FP8_SCALE
        oracle.kv_write_fp8(s["kn"], s["vn"], s["slots"], kc, vc, S, S, w.dtype)
        return oracle.paged_attention_fp8(s["q"], kc, vc, s["bt"], s["cl"], w.scale, S, S, w.dtype,
                                          num_threads=threads)
    oracle.kv_write(s["kn"], s["vn"], s["slots"], kc, vc, w.dtype)
    return oracle.paged_attention(s["q"], kc, vc, s["bt"], s["cl"], w.scale, w.dtype, num_threads=threads)


def sample_bytes(w, n_seqs, fp8: bool = False):
    es = {"f32": 4, "f16": 2, "bf16": 2}[w.dtype]
    ce = 1 if fp8 else es
    ctx = w.context_lens[:n_seqs].astype(np.int64)
    nb = (ctx + w.block_size - 1) // w.block_size
    return (int(ctx.sum()) * w.row_elems * 2 * ce + 2 * n_seqs * w.num_heads * w.head_dim * es
            + 4 * int(nb.sum()) + 4 * n_seqs + 2 * n_seqs * w.row_elems * (es + ce))


def pick_sample(w, threads, budget_s, fp8: bool = False):
    """Largest prefix of sequences whose oracle pass fits the time budget."""
    s1 = oracle_sample(w, 1, fp8)
    t = time.perf_counter()
    oracle_step(w, s1, threads)
    dt = time.perf_counter() - t
    per_tok = dt / max(int(w.context_lens[0]), 1)
    # threads help once there are several (seq, kv-head) items
    eff = max(1.0, min(threads, 8 * w.num_kv_heads) / 1.5)
    n, tot = 0, 0.0
    while n < w.num_seqs and tot + per_tok * w.context_lens[n] / eff <= budget_s:
        tot += per_tok * w.context_lens[n] / eff
        n += 1
    return max(n, 1)


def cpu_baseline(w, fp8: bool = False, budget_s=15.0, min_time_s=10.0):
    """The oracle, as it stands, on the host cores: a prefix of the batch sized to
    the budget, passes repeated until about min_time_s of CPU work."""
    import oracle
    threads = oracle.num_host_threads()
    n = pick_sample(w, threads, budget_s, fp8)
    s = oracle_sample(w, n, fp8)
    passes = 0
    t = time.perf_counter()
    while True:
        oracle_step(w, s, threads)
        passes += 1
        dt = time.perf_counter() - t
        if dt >= min_time_s or passes >= 1000:
            break
    return {"value": passes * sample_bytes(w, n, fp8) / dt / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"first {n} of {w.num_seqs} sequences ({int(w.context_lens[:n].sum())} context tokens): "
                      f"newest-token scatter + decode, {passes} passes in {dt:.1f} s"}


def run_reference(args, budget_total_s: float = 90.0):
    """The oracle, as it stands, on the host cores (the reference arm): each step
    one pass over a prefix of the batch sized so that warm-up and timed steps
    together take about budget_total_s."""
    import oracle
    name = args.workload
    if name not in DECODE_WORKLOADS + FP8_WORKLOADS:
        name = "llama8b_decode"
    build_w, fp8 = base_workload(name)
    w = build_w()
    threads = oracle.num_host_threads()
    budget = budget_total_s / max(args.steps + args.warmup, 1)
    n = pick_sample(w, threads, budget, fp8)
    s = oracle_sample(w, n, fp8)
    for _ in range(args.warmup):
        oracle_step(w, s, threads)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, s, threads)
    dt = (time.perf_counter() - t) / max(args.steps, 1)
    value = sample_bytes(w, n, fp8) / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "num_seqs": w.num_seqs, "sampled_seqs": n},
            "tokens_per_s": n / dt,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"first {n} of {w.num_seqs} sequences per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from __graft_entry__ import build
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()

    if args.workload == "chunked_prefill":
        run_prefill(args, device, rank, world)
        if world > 1:
            dist.destroy_process_group()
        return
    st = Step(args.workload, device)
    st.run()
    torch.cuda.synchronize()
    if st.pa.get_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_id) if rank == 0 else None
    nwarm = warm_up(torch, st.run, max(args.warmup, 3))
    if world > 1:
        dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record()
    for _ in range(args.steps):
        st.run()
    t1.record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler is not None else None
    ms = max_over_ranks(t0.elapsed_time(t1), device)
    ms_step = ms / args.steps
    if st.pa.get_device_error() != 0:
        raise RuntimeError("device error word set during the timed steps")

    # the decode call's own device time, after the timed steps
    peak, peak_kind = hbm_peak()
    roof = decode_roofline(torch, st, device, peak, peak_kind, ms_step)

    # end to end through the public API: pinned host inputs in, result out, every step
    e2e = run_e2e(st, args, device)
    w = st.w
    secondary = []
    if not args.no_secondary and args.workload == "llama8b_decode":
        # the other configuration the 70 % target names, measured in the same run
        del st
        torch.cuda.empty_cache()
        secondary.append(secondary_record(torch, "long_context", device, peak, peak_kind))
        torch.cuda.empty_cache()
        st = None

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    step_bytes, config, launches = roof.pop("_step_bytes"), roof.pop("_config"), roof.pop("_launches_per_step")
    value = job_gbs(world, step_bytes, ms_step)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": nwarm, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded counter-based generator)",
        "config": config,
        "tokens_per_s": world * w.num_seqs / (ms_step * 1e-3),
        "kv_tokens_per_s": world * int(w.context_lens.sum()) / (ms_step * 1e-3),
        "hbm_fraction": value / world / peak,
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    if secondary:
        line["secondary"] = secondary
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.workload.endswith("_fp8"))
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def decode_roofline(torch, st: "Step", device, peak: float, peak_kind: str, ms_step: float | None):
    """Roofline of the decode call of a step: algorithmic bytes per call over its
    device time in steady state (back-to-back calls), checked against the step
    time. For the shared-prefix workload the bytes are the unique bytes (each
    shared block once) and every call is timed alone after an L2 flush, so that
    no call finds the previous call's blocks in L2."""
    shared = st.shared is not None
    if shared:
        flush = l2_flush_buffer(torch, device)
        for _ in range(KERNEL_WARM):
            st.decode_call()
        kern_ms = time_calls_bracketed(torch, st.decode_call, flush=flush)
        ncalls, bracketed = BRACKETED_CALLS, kern_ms
        timing = (f"median of {BRACKETED_CALLS} decode calls, each between its own two CUDA events after an "
                  f"L2 flush (a {2 * L2_BYTES >> 20} MiB write)")
        del flush
        bytes_ = st.decode_unique_bytes
    else:
        kern_ms, ncalls = time_calls(torch, st.decode_call)
        bracketed = time_calls_bracketed(torch, st.decode_call)
        timing = (f"median over {KERNEL_RUNS} runs of {KERNEL_CALLS} back-to-back decode calls, each run between "
                  f"two CUDA events on the launching stream, after the timed steps")
        bytes_ = st.decode_bytes
    achieved = bytes_ / (kern_ms * 1e-3) / 1e9
    ref_ms = ms_step if ms_step is not None else kern_ms
    frac, why = checked_roofline(achieved, peak, kern_ms, ref_ms)
    kernel = (("decode call: decode_fp8_kernel (partitions; writes the new tokens) + merge" if st.append
               else "decode_fp8_kernel + merge") if st.fp8 else
              ("decode call: shared-prefix pass (prefill_tc_kernel, group mode) + private decode_tc_kernel pass "
               "(joining the shared partials; a merge only when one partition does not cover every context)")
              if shared else
              "decode call: decode_tc_kernel (partitions; writes the new tokens) + merge")
    roof = {"kernel": kernel, "bound": "hbm", "achieved": achieved, "peak": peak,
            "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s", "frac": frac,
            "algorithmic_bytes_per_launch": bytes_, "decode_ms": kern_ms, "timed_launches": ncalls,
            "timing": timing, "decode_ms_bracketed_median": bracketed,
            "traffic": recorded_traffic(st.name, traffic_family(st.name))}
    if shared:
        roof["logical_bytes_per_launch"] = st.decode_bytes
        roof["bytes"] = "unique: every shared prefix block counted once per group"
    if why:
        roof["frac_null_reason"] = why
    roof["_step_bytes"] = st.step_bytes
    roof["_config"] = st.config()
    roof["_launches_per_step"] = st.launches_per_step
    return roof


def secondary_record(torch, name: str, device, peak: float, peak_kind: str):
    """The decode roofline of another workload, measured in the same run."""
    st = Step(name, device)
    st.run()
    torch.cuda.synchronize()
    if st.pa.get_device_error() != 0:
        raise RuntimeError(f"device error word set on {name}")
    roof = decode_roofline(torch, st, device, peak, peak_kind, None)
    for k in ("_step_bytes", "_launches_per_step"):
        roof.pop(k)
    cfg = roof.pop("_config")
    roof = {"workload": name, "config": {k: cfg[k] for k in ("num_seqs", "num_heads", "num_kv_heads", "head_dim",
                                                             "block_size", "context_total", "context_min",
                                                             "context_max", "partition_size", "kv_cache", "l2")},
            **roof}
    del st
    return roof


def run_e2e(st: Step, args, device):
    """Per step, through the public calls: the step's inputs (q, new K/V, slot
    mapping, block tables, lengths) copied host -> device from one pinned staging
    buffer in one copy (each input 256-byte aligned in it; the calls take views of
    the device copy), the decode with its write, and a device -> host copy of the
    output into pinned memory. As in a serving loop the device holds two input and
    two output buffers: step i + 1's inputs are copied, and step i - 1's output
    read back, on their own streams while step i computes; events order each
    buffer's reuse (a copy into input buffer j waits for the decode two steps back
    to finish reading it; that decode's output is on the host before step i + 2
    writes output buffer j again)."""
    import torch
    n = min(max(args.steps, 200), 2000)
    items = [("q", st.q), ("k", st.k_new), ("v", st.v_new), ("slots", st.slots), ("bt", st.bt), ("cl", st.cl)]
    if st.shared is not None:
        items += [("pl", st.shared[0]), ("gm", st.shared[1])]
    host = {k: t.cpu().contiguous() for k, t in items}
    layout, off = {}, 0
    for k, t in host.items():
        nbytes = t.numel() * t.element_size()
        layout[k] = (off, nbytes)
        off += (nbytes + 255) // 256 * 256
    stage_h = torch.empty(max(off, 256), dtype=torch.uint8, pin_memory=True)
    for k, t in host.items():
        o, nb = layout[k]
        stage_h[o:o + nb].copy_(t.view(-1).view(torch.uint8))
    stage_d = [torch.empty_like(stage_h, device=device) for _ in range(2)]
    dev_in = [{k: sd[o:o + nb].view(host[k].dtype).view(host[k].shape) for k, (o, nb) in layout.items()}
              for sd in stage_d]
    out_d = [st.out, torch.empty_like(st.out)]
    out_h = [torch.empty(st.out.shape, dtype=st.out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(nb for _, nb in layout.values())
    d2h = out_h[0].numel() * out_h[0].element_size()
    comp = torch.cuda.current_stream(device)
    h2d_s, d2h_s = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of buffer j on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]    # decode of buffer j finished
    ev_out = [torch.cuda.Event() for _ in range(2)]     # output j on the host

    def one(i):
        j = i & 1
        h2d_s.wait_event(ev_done[j])
        with torch.cuda.stream(h2d_s):
            stage_d[j].copy_(stage_h, non_blocking=True)
        ev_in[j].record(h2d_s)
        comp.wait_event(ev_in[j])
        comp.wait_event(ev_out[j])
        if st.copy_pairs is not None:
            st.pa.copy_blocks(st.kc, st.vc, st.copy_pairs)
        d = dev_in[j]
        new = (d["k"], d["v"], d["slots"])
        if not st.append:
            st.write(*new)
        prefix = (d["pl"], d["gm"], st.shared[2]) if st.shared is not None else None
        st.out = out_d[j]
        st.decode(d["q"], d["bt"], d["cl"], prefix, new=new if st.append else None)
        ev_done[j].record(comp)
        d2h_s.wait_event(ev_done[j])
        with torch.cuda.stream(d2h_s):
            out_h[j].copy_(out_d[j], non_blocking=True)
        ev_out[j].record(d2h_s)

    def drain():
        for j in range(2):
            comp.wait_event(ev_out[j])

    for i in range(4):
        one(i)
    drain()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    h2d_s.wait_stream(comp)
    d2h_s.wait_stream(comp)
    for i in range(n):
        one(i)
    drain()
    b.record(comp)
    torch.cuda.synchronize()
    st.out = out_d[0]
    # every step computes the same output; the two host copies must agree with the device
    if not (torch.equal(out_h[0], out_h[1]) and torch.equal(out_h[0], out_d[0].cpu())):
        raise RuntimeError("end-to-end outputs differ between steps")
    ms = a.elapsed_time(b) / n
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return {"value": world * st.step_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "steps": n, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": "one pinned H2D copy and one D2H copy per step, double-buffered on their own streams"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_decode",
                    choices=[*DECODE_WORKLOADS, *FP8_WORKLOADS, "shared_prefix", "chunked_prefill"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the long-context decode record that the 8B-shaped run adds")
    args = ap.parse_args()
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        run_reference(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
