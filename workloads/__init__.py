"""Seeded synthetic inputs for the paged KV cache decode path.

This module only *draws* inputs: token contents, context lengths, physical block
pools, block tables, slot mappings and the event scripts of the sharing workloads.
It holds none of the attention, scatter, copy or allocation arithmetic. The CPU
oracle (``oracle/``) and the CUDA library (``paged_kv_cache_261_gb300``) both
consume what it makes; neither is imported here.

Token contents come from a counter-based generator. Element ``e`` of the row that
tensor ``tid`` (K, V or q) holds for content key ``key`` at position ``pos`` is a
pure integer function of ``(seed, tid, key, pos, e)``: the centred sum of twelve
independent uniforms on [0, 1), an Irwin-Hall stand-in for N(0, 1) (standard
deviation 0.998, range about +-5.66). Eleven of the uniforms carry 4 bits and
one carries 20, so the sum is continuous to 2^-21 and a value has up to 24
significant bits: it is an exact float32 (the fp32 workloads use it as it is)
with a full mantissa, and the 16-bit workloads store it rounded to nearest-even
in fp16 or bf16 -- the same rounding on both sides (``to_storage_numpy`` here,
torch's casts on the device), so the oracle reads exactly the values the GPU
reads. The integer code runs on numpy arrays and on torch tensors (host or
device) and yields identical bits on both, which lets a test regenerate on the
host exactly the rows that were generated on the device.

Shapes follow the cache layout ``[num_blocks, block_size, num_kv_heads,
head_dim]``. A table entry of -1 marks an unused logical block.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

M32 = 0xFFFFFFFF

TID_K = 0
TID_V = 1
TID_Q = 2

DTYPES = ("f32", "f16", "bf16")


# ---------------------------------------------------------------------------
# counter-based generator (numpy or torch, int64 arithmetic only)
# ---------------------------------------------------------------------------

def _is_torch(x) -> bool:
    return type(x).__module__.startswith("torch")


def _mix32(x):
    """32-bit integer finaliser on int64 arrays holding values in [0, 2**32).

    Every product stays below 2**59, so int64 never overflows and numpy and
    torch give the same bits."""
    x = (((x >> 16) ^ x) * 0x045D9F3B) & M32
    x = (((x >> 16) ^ x) * 0x045D9F3B) & M32
    return (x >> 16) ^ x


def _mix_scalar(v: int) -> int:
    v &= M32
    v = (((v >> 16) ^ v) * 0x045D9F3B) & M32
    v = (((v >> 16) ^ v) * 0x045D9F3B) & M32
    return (v >> 16) ^ v


# Largest magnitude content_rows can return: 11862015 / 2**21.
CONTENT_MAX = 11862015.0 / 2097152.0


def _irwin_hall(keys):
    """keys: int64 array in [0, 2**32). Returns float32 values in [-CONTENT_MAX, CONTENT_MAX].

    Twelve uniforms on [0, 1): eleven 4-bit ones (nibbles of two hashes) and one
    20-bit one (a nibble of the first hash extended by the second hash's top 16
    bits). Their sum minus its mean is n / 2**21 for an odd integer n with
    |n| <= 11862015 < 2**24, so the float32 conversion and the scaling are exact."""
    a = _mix32(keys)
    b = _mix32(keys ^ 0x5BD1E995)
    s = a & 15
    for i in range(1, 8):
        s = s + ((a >> (4 * i)) & 15)
    for i in range(4):
        s = s + ((b >> (4 * i)) & 15)
    f = b >> 16
    n = 2 * (s * 65536 + f) - (180 * 65536 + 65535)
    if _is_torch(n):
        import torch
        return n.to(torch.float32) / 2097152.0
    return n.astype(np.float32) / np.float32(2097152.0)


def content_rows(seed: int, tid: int, keys, positions, row_elems: int):
    """Rows of token contents.

    keys, positions: int64 arrays (numpy or torch) of equal length n.
    Returns float32 [n, row_elems] on the same library/device as ``keys``.
    """
    h = _mix_scalar(seed * 0x9E3779B1 + tid * 0x7FEB352D)
    r = _mix32(((_mix32((keys + h) & M32)) + positions * 0x2C1B3C6D) & M32)
    if _is_torch(keys):
        import torch
        e = torch.arange(row_elems, dtype=torch.int64, device=keys.device)
    else:
        e = np.arange(row_elems, dtype=np.int64)
    ek = (e * 0x297A2D39) & M32
    return _irwin_hall(r[:, None] ^ ek[None, :])


def content_codes(seed: int, tid: int, keys, positions, row_elems: int):
    """Rows of 8-bit cache contents: OCP FP8 E4M3 codes drawn directly as bits.

    Same keying as ``content_rows``; returns uint8 [n, row_elems]. Each code has a
    random sign, a random 3-bit mantissa and an exponent field drawn uniformly
    from {0 (subnormal), 4, 5, ..., 14}: magnitudes from 2^-9 to 240, never the
    NaN pattern. With a scale of 5.625 / 448 the decoded values span about
    [-3, 3], inside the range of the float rows. No quantisation is involved.
    """
    h = _mix_scalar(seed * 0x9E3779B1 + tid * 0x7FEB352D + 0x3C6EF372)
    r = _mix32(((_mix32((keys + h) & M32)) + positions * 0x2C1B3C6D) & M32)
    if _is_torch(keys):
        import torch
        e = torch.arange(row_elems, dtype=torch.int64, device=keys.device)
    else:
        e = np.arange(row_elems, dtype=np.int64)
    ek = (e * 0x297A2D39) & M32
    x = _mix32(r[:, None] ^ ek[None, :])
    ex = ((x >> 8) & 0xFFFF) % 12
    ex = ex + 3 * (ex > 0)                      # 0, or 4..14
    code = ((x >> 31) << 7) | (ex << 3) | (x & 7)
    if _is_torch(code):
        import torch
        return code.to(torch.uint8)
    return code.astype(np.uint8)


FP8_SCALE = 5.625 / 448.0     # maps [-5.625, 5.625] onto [-448, 448]; rarer larger rows saturate


# ---------------------------------------------------------------------------
# bf16 / f16 storage helpers (round to nearest even, as torch's casts do)
# ---------------------------------------------------------------------------

def _bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest with ties to even; any NaN
    becomes 0x7FC0 (torch's canonical bf16 NaN). Infinities and overflow follow
    from the same carry."""
    u = x.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = r.astype(np.uint16)
    out[np.isnan(x)] = 0x7FC0
    return out


def to_storage_numpy(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values -> numpy array holding them in the storage dtype, rounded
    to nearest even: f32 -> float32 (unchanged), f16 -> float16, bf16 -> uint16
    bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "f16":
        with np.errstate(over="ignore"):
            return x.astype(np.float16)
    if dtype == "bf16":
        return _bf16_bits_rne(x)
    raise ValueError(dtype)


def storage_to_float64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Inverse of to_storage_numpy on stored values (exact)."""
    if dtype == "bf16":
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def rounded(x, dtype: str):
    """float32 values as the storage dtype holds them (numpy or torch input)."""
    if _is_torch(x):
        return x.to(torch_dtype(dtype)).float()
    return storage_to_float64(to_storage_numpy(x, dtype), dtype).astype(np.float32)


def torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

@dataclass
class DecodeWorkload:
    """One decode batch: per-sequence contexts laid out through block tables.

    Sequence b holds positions [0, context_lens[b]). Its content at position pos
    comes from key prefix_key[b] when pos < prefix_len[b], else from own_key[b]
    (the shared-prefix workload shares prompt contents across samples).
    The newest token (pos = context_lens[b] - 1) is the one the step writes with
    paged_kv_write; slot_mapping[b] is its slot, or -1 when context_lens[b] == 0.
    """
    name: str
    seed: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: str
    scale: float
    q_mult: float
    context_lens: np.ndarray          # int32 [B]
    block_tables: np.ndarray          # int32 [B, MB]
    slot_mapping: np.ndarray          # int32 [B]
    own_key: np.ndarray               # int64 [B]
    prefix_key: np.ndarray            # int64 [B]
    prefix_len: np.ndarray            # int64 [B]
    extra_write_slots: np.ndarray | None = None   # int32 [T] (mixed serving step)
    extra_write_key0: int = 1 << 24
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def row_elems(self) -> int:
        return self.num_kv_heads * self.head_dim

    def content_keys(self, seq_idx, positions):
        """Content key per (seq, pos); arrays of the same library."""
        if _is_torch(positions):
            import torch
            dev = positions.device
            own = torch.as_tensor(self.own_key, device=dev)[seq_idx]
            pk = torch.as_tensor(self.prefix_key, device=dev)[seq_idx]
            pl = torch.as_tensor(self.prefix_len, device=dev)[seq_idx]
            return torch.where(positions < pl, pk, own)
        own = self.own_key[seq_idx]
        return np.where(positions < self.prefix_len[seq_idx], self.prefix_key[seq_idx], own)

    def kv_rows(self, tid: int, seq_idx, positions):
        """float32 [n, num_kv_heads*head_dim] rows for (seq_idx[i], positions[i])."""
        keys = self.content_keys(seq_idx, positions)
        return content_rows(self.seed, tid, keys, positions, self.row_elems)

    def kv_codes(self, tid: int, seq_idx, positions):
        """uint8 [n, num_kv_heads*head_dim] E4M3 codes for an 8-bit cache."""
        keys = self.content_keys(seq_idx, positions)
        return content_codes(self.seed, tid, keys, positions, self.row_elems)

    def _cache_rows(self, tid: int, seq_idx, positions, codes: bool):
        return self.kv_codes(tid, seq_idx, positions) if codes else self.kv_rows(tid, seq_idx, positions)

    def q_values(self, like=None):
        """float32 [B, H, D] queries (q_mult applied; callers round to the storage dtype)."""
        B, H, D = self.num_seqs, self.num_heads, self.head_dim
        if like is not None and _is_torch(like):
            import torch
            keys = torch.as_tensor(self.own_key, device=like.device)
            pos = torch.zeros_like(keys)
        else:
            keys = self.own_key.astype(np.int64)
            pos = np.zeros_like(keys)
        rows = content_rows(self.seed, TID_Q, keys, pos, H * D)
        return (rows * self.q_mult).reshape(B, H, D)

    def newest_kv(self, like=None):
        """float32 ([B, Hk, D], [B, Hk, D]): K and V rows of each newest token.
        Rows of sequences with context 0 are zero (their slot is -1)."""
        ctx = self.context_lens.astype(np.int64)
        pos = np.maximum(ctx - 1, 0)
        idx = np.arange(self.num_seqs, dtype=np.int64)
        if like is not None and _is_torch(like):
            import torch
            idx_t = torch.as_tensor(idx, device=like.device)
            pos_t = torch.as_tensor(pos, device=like.device)
            k = self.kv_rows(TID_K, idx_t, pos_t)
            v = self.kv_rows(TID_V, idx_t, pos_t)
            live = torch.as_tensor(ctx > 0, device=like.device)[:, None]
            k = torch.where(live, k, torch.zeros_like(k))
            v = torch.where(live, v, torch.zeros_like(v))
        else:
            k = self.kv_rows(TID_K, idx, pos)
            v = self.kv_rows(TID_V, idx, pos)
            k[ctx == 0] = 0
            v[ctx == 0] = 0
        shp = (self.num_seqs, self.num_kv_heads, self.head_dim)
        return k.reshape(shp), v.reshape(shp)

    def extra_write_rows(self, like=None):
        """K, V rows [T, Hk, D] of the mixed serving step's extra tokens."""
        T = int(self.extra_write_slots.shape[0])
        keys = np.arange(T, dtype=np.int64) + self.extra_write_key0
        pos = np.zeros(T, dtype=np.int64)
        if like is not None and _is_torch(like):
            import torch
            keys = torch.as_tensor(keys, device=like.device)
            pos = torch.as_tensor(pos, device=like.device)
        k = content_rows(self.seed, TID_K, keys, pos, self.row_elems)
        v = content_rows(self.seed, TID_V, keys, pos, self.row_elems)
        shp = (T, self.num_kv_heads, self.head_dim)
        return k.reshape(shp), v.reshape(shp)

    # -- placement of the pre-step cache contents ---------------------------

    def _positions(self, seqs, include_newest: bool):
        """(seq_idx, pos) int64 arrays for the tokens the cache holds before the step."""
        ctx = self.context_lens.astype(np.int64)[seqs]
        n = ctx if include_newest else np.maximum(ctx - 1, 0)
        seq_idx = np.repeat(np.asarray(seqs, dtype=np.int64), n)
        starts = np.repeat(np.cumsum(n) - n, n)
        pos = np.arange(int(n.sum()), dtype=np.int64) - starts
        return seq_idx, pos

    def _slots(self, seq_idx, pos):
        bs = self.block_size
        phys = self.block_tables[seq_idx, pos // bs].astype(np.int64)
        if np.any(phys < 0):
            raise ValueError("table entry missing for a live position")
        return phys * bs + pos % bs

    def fill_cache_torch(self, key_cache, value_cache, include_newest=False,
                         seqs=None, chunk_tokens=1 << 16):
        """Write the pre-step contents into device (or host) torch caches; uint8
        caches receive E4M3 codes (``kv_codes``), others float rows.

        Uses plain torch indexing; the library under test is not involved."""
        import torch
        codes = key_cache.dtype == torch.uint8
        seqs = np.arange(self.num_seqs) if seqs is None else np.asarray(seqs)
        seq_idx, pos = self._positions(seqs, include_newest)
        slots = self._slots(seq_idx, pos)
        kflat = key_cache.view(-1, self.row_elems)
        vflat = value_cache.view(-1, self.row_elems)
        dev = key_cache.device
        for s in range(0, seq_idx.shape[0], chunk_tokens):
            si = torch.as_tensor(seq_idx[s:s + chunk_tokens], device=dev)
            pi = torch.as_tensor(pos[s:s + chunk_tokens], device=dev)
            sl = torch.as_tensor(slots[s:s + chunk_tokens], device=dev)
            kflat[sl] = self._cache_rows(TID_K, si, pi, codes).to(key_cache.dtype)
            vflat[sl] = self._cache_rows(TID_V, si, pi, codes).to(value_cache.dtype)

    def contiguous_kv(self, b: int, include_newest: bool = True):
        """float32 ([ctx, Hk, D], [ctx, Hk, D]) for sequence b, in position order."""
        ctx = int(self.context_lens[b])
        n = ctx if include_newest else max(ctx - 1, 0)
        seq_idx = np.full(n, b, dtype=np.int64)
        pos = np.arange(n, dtype=np.int64)
        shp = (n, self.num_kv_heads, self.head_dim)
        return (self.kv_rows(TID_K, seq_idx, pos).reshape(shp),
                self.kv_rows(TID_V, seq_idx, pos).reshape(shp))

    def _rows_host(self, seq_idx, pos, codes: bool = False):
        """numpy K and V rows (float32, or uint8 codes), generated with torch's CPU threads."""
        import torch
        si = torch.from_numpy(np.ascontiguousarray(seq_idx))
        pi = torch.from_numpy(np.ascontiguousarray(pos))
        return (self._cache_rows(TID_K, si, pi, codes).numpy(), self._cache_rows(TID_V, si, pi, codes).numpy())

    def compact_host_view(self, seqs, rng_seed: int = 7, include_newest=False, chunk: int = 16384,
                          codes: bool = False):
        """A small host paged cache holding only ``seqs``.

        The chosen sequences' logical blocks are placed on a fresh random
        permutation of a pool just big enough for them. Returns a dict with
        float32 caches (uint8 E4M3 codes when ``codes``), int32
        block_tables/context_lens for the chosen rows and the newest-token slots
        in the new pool."""
        seqs = np.asarray(seqs, dtype=np.int64)
        bs = self.block_size
        ctx = self.context_lens.astype(np.int64)[seqs]
        nb = (ctx + bs - 1) // bs
        total = int(nb.sum())
        perm = np.random.default_rng(rng_seed).permutation(max(total, 1)).astype(np.int32)
        mb = max(int(nb.max()) if nb.size else 1, 1)
        tables = np.full((seqs.shape[0], mb), -1, dtype=np.int32)
        off = 0
        for i, n in enumerate(nb):
            tables[i, :n] = perm[off:off + n]
            off += n
        nblk = max(total, 1)
        kc = np.zeros((nblk, bs, self.num_kv_heads, self.head_dim), np.uint8 if codes else np.float32)
        vc = np.zeros_like(kc)
        kflat = kc.reshape(-1, self.row_elems)
        vflat = vc.reshape(-1, self.row_elems)
        for i, b in enumerate(seqs):
            c = int(ctx[i])
            n = c if include_newest else max(c - 1, 0)
            for s in range(0, n, chunk):
                p = np.arange(s, min(n, s + chunk), dtype=np.int64)
                slot = tables[i, p // bs].astype(np.int64) * bs + p % bs
                k, v = self._rows_host(np.full(p.shape[0], int(b), np.int64), p, codes)
                kflat[slot] = k
                vflat[slot] = v
        newest = np.full(seqs.shape[0], -1, np.int32)
        for i, c in enumerate(ctx):
            if c > 0:
                newest[i] = tables[i, (c - 1) // bs] * bs + (c - 1) % bs
        return dict(key_cache=kc, value_cache=vc, block_tables=tables,
                    context_lens=ctx.astype(np.int32), slot_mapping=newest,
                    num_blocks=nblk)

    def algorithmic_bytes(self, cache_elem_bytes: int | None = None) -> dict:
        """Bytes a decode step must move at minimum (K and V once per (seq, kv-head),
        q in, out back, the table entries used and the lengths). cache_elem_bytes:
        size of a cache element when it differs from the dtype's (1 for 8-bit)."""
        s = {"f32": 4, "f16": 2, "bf16": 2}[self.dtype]
        c = s if cache_elem_bytes is None else cache_elem_bytes
        ctx = self.context_lens.astype(np.int64)
        nb = (ctx + self.block_size - 1) // self.block_size
        kv = int(ctx.sum()) * self.num_kv_heads * self.head_dim * 2 * c
        qo = 2 * self.num_seqs * self.num_heads * self.head_dim * s
        meta = 4 * int(nb.sum()) + 4 * self.num_seqs
        write = 2 * int((ctx > 0).sum()) * self.row_elems * (s + c) + 4 * self.num_seqs
        return dict(kv=kv, qo=qo, meta=meta, decode=kv + qo + meta, write=write)


def _tables_from_pool(ctx: np.ndarray, block_size: int, perm: np.ndarray, mb: int | None = None):
    nb = (ctx.astype(np.int64) + block_size - 1) // block_size
    if mb is None:
        mb = max(int(nb.max()), 1)
    tables = np.full((ctx.shape[0], mb), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nb):
        tables[b, :n] = perm[off:off + n]
        off += n
    return tables, off


def _newest_slots(ctx, tables, bs):
    out = np.full(ctx.shape[0], -1, np.int32)
    for b, c in enumerate(ctx):
        if c > 0:
            out[b] = tables[b, (c - 1) // bs] * bs + (c - 1) % bs
    return out


def make_decode(name: str, seed: int, ctx: np.ndarray, num_heads: int, num_kv_heads: int,
                head_dim: int, block_size: int, dtype: str, q_mult: float = 1.0,
                pool_slack: float = 0.10, num_blocks: int | None = None,
                extra_write: int = 0, mb: int | None = None, scale: float | None = None) -> DecodeWorkload:
    """Generic builder: contexts ``ctx`` laid out on a shuffled pool."""
    rng = np.random.default_rng(seed + 7919)
    ctx = np.asarray(ctx, dtype=np.int32)
    nb = (ctx.astype(np.int64) + block_size - 1) // block_size
    need = int(nb.sum()) + (extra_write + block_size - 1) // block_size
    if num_blocks is None:
        num_blocks = max(int(math.ceil((1.0 + pool_slack) * need)), 1)
    if num_blocks < need:
        raise ValueError("pool too small")
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables, used = _tables_from_pool(ctx, block_size, perm, mb)
    extra = None
    if extra_write:
        free_blocks = perm[used:].astype(np.int64)
        free_slots = (free_blocks[:, None] * block_size + np.arange(block_size)[None, :]).reshape(-1)
        extra = rng.choice(free_slots, extra_write, replace=False).astype(np.int32)
    B = ctx.shape[0]
    return DecodeWorkload(
        name=name, seed=seed, num_heads=num_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=block_size, num_blocks=num_blocks, dtype=dtype,
        scale=(1.0 / math.sqrt(head_dim)) if scale is None else scale, q_mult=q_mult,
        context_lens=ctx, block_tables=tables,
        slot_mapping=_newest_slots(ctx, tables, block_size),
        own_key=np.arange(B, dtype=np.int64), prefix_key=np.zeros(B, np.int64),
        prefix_len=np.zeros(B, np.int64), extra_write_slots=extra)


# -- the five named workloads ------------------------------------------------

def tiny_fp32(seed: int = 1001) -> DecodeWorkload:
    """4 sequences of 5/17/33/64 tokens, 4 q heads = 4 kv heads, head_dim 64,
    block_size 4, 64-block pool consumed in the order of a seeded permutation."""
    rng = np.random.default_rng(seed)
    ctx = np.array([5, 17, 33, 64], dtype=np.int32)
    perm = rng.permutation(64).astype(np.int32)
    tables, _ = _tables_from_pool(ctx, 4, perm)
    B = 4
    return DecodeWorkload(
        name="tiny_fp32", seed=seed, num_heads=4, num_kv_heads=4, head_dim=64,
        block_size=4, num_blocks=64, dtype="f32", scale=1.0 / 8.0, q_mult=1.0,
        context_lens=ctx, block_tables=tables, slot_mapping=_newest_slots(ctx, tables, 4),
        own_key=np.arange(B, dtype=np.int64), prefix_key=np.zeros(B, np.int64),
        prefix_len=np.zeros(B, np.int64))


def llama8b_decode(seed: int = 1002, num_seqs: int = 64, dtype: str = "bf16",
                   block_size: int = 16) -> DecodeWorkload:
    """Batch 64, 32 q heads / 8 kv heads, head_dim 128, bf16, block_size 16,
    contexts uniform in [512, 4096], pool = total need + 10%, shuffled."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(512, 4097, size=num_seqs).astype(np.int32)
    return make_decode("llama8b_decode", seed, ctx, 32, 8, 128, block_size, dtype)


def long_context(seed: int = 1003, num_seqs: int = 8, dtype: str = "bf16") -> DecodeWorkload:
    """Batch 8, contexts uniform in [32768, 131072], 64 q heads / 8 kv heads,
    head_dim 128, bf16, block_size 16, q doubled for a peaky softmax."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(32768, 131073, size=num_seqs).astype(np.int32)
    return make_decode("long_context", seed, ctx, 64, 8, 128, 16, dtype, q_mult=2.0)


def mixed_serving(seed: int = 1005, block_size: int = 16, dtype: str = "bf16",
                  num_seqs: int = 512, extra_write: int = 2048) -> DecodeWorkload:
    """Batch 512 with lognormal contexts (median 600, sigma 1.0, clipped to
    [16, 8192]) plus a 2048-token write to distinct random free slots. The
    contexts and contents do not depend on block_size or dtype."""
    rng = np.random.default_rng(seed)
    ctx = np.clip(np.round(rng.lognormal(math.log(600.0), 1.0, size=num_seqs)), 16, 8192).astype(np.int32)
    w = make_decode(f"mixed_serving_bs{block_size}_{dtype}", seed, ctx, 32, 8, 128,
                    block_size, dtype, extra_write=extra_write)
    return w


@dataclass
class SharedPrefixScript:
    """Event script of the shared-prefix sampling workload.

    num_prompts prompts of prompt_len tokens are prefilled, each is forked into
    samples_per_prompt samples, then sample s appends private[s] earlier tokens
    plus one current token. Samples append in index order."""
    seed: int
    num_prompts: int
    samples_per_prompt: int
    prompt_len: int
    private: np.ndarray           # int64 [num_prompts * samples_per_prompt]
    block_size: int
    num_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    dtype: str = "bf16"

    @property
    def num_samples(self) -> int:
        return self.num_prompts * self.samples_per_prompt

    def pool_blocks(self) -> int:
        bs = self.block_size
        prompt_blocks = (self.prompt_len + bs - 1) // bs
        ctx = self.prompt_len + self.private + 1
        private_blocks = ((ctx + bs - 1) // bs) - (self.prompt_len // bs)
        need = self.num_prompts * prompt_blocks + int(private_blocks.sum())
        return int(math.ceil(1.1 * need)) + 8

    def workload(self, block_tables: np.ndarray, num_blocks: int) -> DecodeWorkload:
        """The decode batch after every sample's current token, laid out on the
        tables an allocator produced (rows in sample order)."""
        S = self.num_samples
        ctx = (self.prompt_len + self.private + 1).astype(np.int32)
        prompt_of = np.arange(S, dtype=np.int64) // self.samples_per_prompt
        return DecodeWorkload(
            name="shared_prefix", seed=self.seed, num_heads=self.num_heads,
            num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
            block_size=self.block_size, num_blocks=num_blocks, dtype=self.dtype,
            scale=1.0 / math.sqrt(self.head_dim), q_mult=1.0, context_lens=ctx,
            block_tables=block_tables.astype(np.int32),
            slot_mapping=_newest_slots(ctx, block_tables, self.block_size),
            own_key=np.arange(S, dtype=np.int64) + (1 << 20),
            prefix_key=prompt_of, prefix_len=np.full(S, self.prompt_len, np.int64))


def shared_prefix(seed: int = 1004, num_prompts: int = 32, samples_per_prompt: int = 8,
                  prompt_len: int = 1000, max_private: int = 256,
                  block_size: int = 16) -> SharedPrefixScript:
    rng = np.random.default_rng(seed)
    private = rng.integers(0, max_private + 1, size=num_prompts * samples_per_prompt).astype(np.int64)
    return SharedPrefixScript(seed=seed, num_prompts=num_prompts,
                              samples_per_prompt=samples_per_prompt, prompt_len=prompt_len,
                              private=private, block_size=block_size)


WORKLOADS = {
    "tiny_fp32": tiny_fp32,
    "llama8b_decode": llama8b_decode,
    "long_context": long_context,
    "shared_prefix": shared_prefix,
    "mixed_serving": mixed_serving,
}


# ---------------------------------------------------------------------------
# chunked prefill
# ---------------------------------------------------------------------------

@dataclass
class PrefillWorkload:
    """A chunked-prefill batch on top of a decode-style layout.

    ``base`` holds the contexts *including* each sequence's chunk, so its
    block tables, pool and token contents apply unchanged; sequence b's chunk is
    its last q_lens[b] positions. Query rows are packed in sequence order;
    query_start_loc[b] is the first row of sequence b."""
    base: DecodeWorkload
    q_lens: np.ndarray                 # int32 [B]

    @property
    def query_start_loc(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    def chunk_index(self):
        """(seq_idx, pos) int64 arrays of every query row, in packed order."""
        ctx = self.base.context_lens.astype(np.int64)
        ql = self.q_lens.astype(np.int64)
        seq_idx = np.repeat(np.arange(ctx.shape[0], dtype=np.int64), ql)
        starts = np.repeat(np.cumsum(ql) - ql, ql)
        i = np.arange(int(ql.sum()), dtype=np.int64) - starts
        return seq_idx, ctx[seq_idx] - ql[seq_idx] + i

    def q_values(self, like=None):
        """float32 [total_q, H, D] queries (q_mult applied)."""
        w = self.base
        seq_idx, pos = self.chunk_index()
        keys = w.own_key[seq_idx]
        if like is not None and _is_torch(like):
            import torch
            keys = torch.as_tensor(keys, device=like.device)
            pos = torch.as_tensor(pos + 1, device=like.device)
        else:
            pos = pos + 1
        rows = content_rows(w.seed, TID_Q, keys, pos, w.num_heads * w.head_dim)
        return (rows * w.q_mult).reshape(-1, w.num_heads, w.head_dim)

    def chunk_kv(self, like=None):
        """K, V rows [total_q, Hk, D] of the chunk positions (written before attending)."""
        w = self.base
        seq_idx, pos = self.chunk_index()
        if like is not None and _is_torch(like):
            import torch
            seq_idx = torch.as_tensor(seq_idx, device=like.device)
            pos = torch.as_tensor(pos, device=like.device)
        shp = (-1, w.num_kv_heads, w.head_dim)
        return w.kv_rows(TID_K, seq_idx, pos).reshape(shp), w.kv_rows(TID_V, seq_idx, pos).reshape(shp)

    def chunk_slots(self) -> np.ndarray:
        seq_idx, pos = self.chunk_index()
        return self.base._slots(seq_idx, pos).astype(np.int32)

    def flops(self) -> int:
        """Scores plus weighted sum: 4 * D flops per (query row, head, visible key)."""
        w = self.base
        ctx = w.context_lens.astype(np.int64)
        ql = self.q_lens.astype(np.int64)
        visible = (ctx - ql) * ql + ql * (ql + 1) // 2
        return int(4 * w.head_dim * w.num_heads * visible.sum())


def make_prefill(name: str, seed: int, prior: np.ndarray, q_lens: np.ndarray, num_heads: int,
                 num_kv_heads: int, head_dim: int, block_size: int, dtype: str) -> PrefillWorkload:
    """Sequences with `prior` cached tokens each receiving a chunk of q_lens tokens."""
    prior = np.asarray(prior, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    base = make_decode(name, seed, prior + q_lens, num_heads, num_kv_heads, head_dim, block_size, dtype)
    return PrefillWorkload(base=base, q_lens=q_lens)


def chunked_prefill(seed: int = 1006, num_seqs: int = 16, chunk: int = 512,
                    dtype: str = "bf16") -> PrefillWorkload:
    """16 sequences, each with U[0, 3584] cached tokens and a 512-token chunk;
    32 q heads / 8 kv heads, head_dim 128, bf16, block_size 16."""
    rng = np.random.default_rng(seed)
    prior = rng.integers(0, 3585, size=num_seqs)
    return make_prefill("chunked_prefill", seed, prior, np.full(num_seqs, chunk), 32, 8, 128, 16, dtype)


def fill_prior_torch(pw: PrefillWorkload, key_cache, value_cache, chunk_tokens: int = 1 << 16):
    """Write every sequence's cached tokens before its chunk (positions < ctx - q_len)."""
    import torch
    w = pw.base
    prior = (w.context_lens - pw.q_lens).astype(np.int64)
    seq_idx = np.repeat(np.arange(w.num_seqs, dtype=np.int64), prior)
    starts = np.repeat(np.cumsum(prior) - prior, prior)
    pos = np.arange(int(prior.sum()), dtype=np.int64) - starts
    slots = w._slots(seq_idx, pos) if seq_idx.size else np.zeros(0, np.int64)
    kflat = key_cache.view(-1, w.row_elems)
    vflat = value_cache.view(-1, w.row_elems)
    dev = key_cache.device
    for s in range(0, seq_idx.shape[0], chunk_tokens):
        si = torch.as_tensor(seq_idx[s:s + chunk_tokens], device=dev)
        pi = torch.as_tensor(pos[s:s + chunk_tokens], device=dev)
        sl = torch.as_tensor(slots[s:s + chunk_tokens], device=dev)
        kflat[sl] = w.kv_rows(TID_K, si, pi).to(key_cache.dtype)
        vflat[sl] = w.kv_rows(TID_V, si, pi).to(value_cache.dtype)


def make_shared_groups(seed: int, groups, singles: int, num_heads: int, num_kv_heads: int,
                       head_dim: int, block_size: int, dtype: str) -> DecodeWorkload:
    """Sequences sharing leading blocks by reference, as forks produce them.

    groups: list of (members, shared_blocks, max_private) -- each group's members
    share `shared_blocks` full blocks of one prompt (same physical blocks, same
    contents) and then hold 0..max_private private tokens each. `singles` more
    sequences share nothing. Shapes and contents are seeded."""
    rng = np.random.default_rng(seed)
    bs = block_size
    ctx, pkey, plen = [], [], []
    layout = []                                   # (group id or -1, shared blocks)
    for gi, (members, shared, max_priv) in enumerate(groups):
        for _ in range(members):
            priv = int(rng.integers(0, max_priv + 1))
            ctx.append(shared * bs + priv)
            pkey.append(gi)
            plen.append(shared * bs)
            layout.append((gi, shared))
    for _ in range(singles):
        ctx.append(int(rng.integers(1, 1500)))
        pkey.append(0)
        plen.append(0)
        layout.append((-1, 0))
    ctx = np.array(ctx, np.int32)
    B = ctx.shape[0]
    nb_total = sum(g[1] for g in groups) + int(((ctx + bs - 1) // bs).sum()) + 8
    num_blocks = int(1.1 * nb_total) + 8
    perm = rng.permutation(num_blocks).astype(np.int32)
    mb = max(int(((ctx + bs - 1) // bs).max()), 1)
    tables = np.full((B, mb), -1, np.int32)
    off = 0
    group_blocks = {}
    for gi, (_, shared, _) in enumerate(groups):
        group_blocks[gi] = perm[off:off + shared]
        off += shared
    for b in range(B):
        gi, shared = layout[b]
        n = int((ctx[b] + bs - 1) // bs)
        if gi >= 0:
            tables[b, :shared] = group_blocks[gi]
        for j in range(shared, n):
            tables[b, j] = perm[off]
            off += 1
    own = np.arange(B, dtype=np.int64) + (1 << 20)
    return DecodeWorkload(
        name="shared_groups", seed=seed, num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        block_size=bs, num_blocks=num_blocks, dtype=dtype, scale=1.0 / math.sqrt(head_dim), q_mult=1.0,
        context_lens=ctx, block_tables=tables, slot_mapping=_newest_slots(ctx, tables, bs), own_key=own,
        prefix_key=np.array(pkey, np.int64), prefix_len=np.array(plen, np.int64))


# ---------------------------------------------------------------------------
# beam search (fork / prune / copy-on-write of the last block)
# ---------------------------------------------------------------------------

@dataclass
class BeamScript:
    """Seeded beam-search event script.

    A prompt of prompt_len tokens is prefilled, then `steps` decode steps run
    with beam width k: at each step every surviving beam proposes candidates
    and k of them survive; parents[s][i] is the beam (index into the previous
    step's survivors) that survivor i extends. A parent may have several
    children (they fork) or none (it is dropped). The choices are drawn from
    the seed -- no model is involved."""
    seed: int
    prompt_len: int
    steps: int
    k: int
    block_size: int
    parents: list

    @property
    def final_len(self) -> int:
        return self.prompt_len + self.steps


def beam_search_script(seed: int = 1007, prompt_len: int = 64, steps: int = 32, k: int = 4,
                       block_size: int = 16) -> BeamScript:
    """Prompt 64 tokens, 32 steps, block size 16 (the shape of the pages' beam demo)."""
    rng = np.random.default_rng(seed)
    parents = []
    width = 1
    for _ in range(steps):
        # survivors concentrate on a few parents, as beams do
        weights = rng.dirichlet(np.full(width, 0.6))
        parents.append(sorted(int(x) for x in rng.choice(width, size=k, p=weights)))
        width = k
    return BeamScript(seed=seed, prompt_len=prompt_len, steps=steps, k=k, block_size=block_size,
                      parents=parents)
