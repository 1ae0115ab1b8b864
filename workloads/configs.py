"""Seeded synthetic workloads for paged GQA attention over a block arena.

The shapes and structure follow the pages "Building Kshipra" part 3
(kshipra-3): the KV cache is an arena of fixed-size blocks reserved once and
handed out from a free list (section 1, "Block-Arena KV Cache"); several
requests may point at the same physical prefix blocks (section 3, "Radix-Tree
Prefix Cache"); a prompt is processed in chunks whose tokens sit at absolute
positions after the cached prefix (section 4, "Chunked Prefill"); one
scheduler step mixes prefill chunks with single-token decodes under a token
budget (section 5, "Continuous Batching").  The pages give no concrete data,
so every tensor here is drawn N(0, 1) and rounded to the storage dtype.

Recipe (fixed draw order per workload, numpy PCG64 seeded with the config's
index): lengths -> block permutation -> q -> k -> v.  Keys and values are drawn
for every position 0..ctx-1 of every sequence (the cached prefix and the new
chunk), in logical order; rows of the shared system prefix are drawn once and
reused by every sequence that shares it.

Nothing in this module rotates, scales, masks or normalises: it only draws
numbers and lays out block tables.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Sequence

import numpy as np
import torch

DTYPE_CODES = {"f16": 0, "bf16": 1}

CONFIG_NAMES = ("tiny", "llama-decode", "chunked-prefill", "mixed", "long-decode")

# block-table entries past a sequence's last block hold this value; no kernel
# may read them
TABLE_POISON = -1

_CHUNK = 1 << 24  # values per normal draw, to bound host memory


def f16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE binary16 (nearest, ties to even); bits.

    Uses torch's vectorised CPU cast, which rounds like numpy's but is far
    faster on the hundreds of millions of values the large workloads draw.
    """
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bfloat16 (nearest, ties to even); bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


class _NormalBits:
    """Draws N(0, 1) float32 values chunk by chunk into reused buffers and
    writes their dtype bits in place (large fresh arrays are slow to touch)."""

    def __init__(self, rng: np.random.Generator, dtype: str):
        self.rng = rng
        self.dtype = dtype
        self.f32 = np.empty(_CHUNK, dtype=np.float32)
        self.t32 = torch.from_numpy(self.f32)
        self.t16 = torch.empty(_CHUNK, dtype=torch.float16)

    def fill(self, out: np.ndarray) -> None:
        flat = out.reshape(-1)
        n = flat.size
        for lo in range(0, n, _CHUNK):
            m = min(n, lo + _CHUNK) - lo
            self.rng.standard_normal(out=self.f32[:m], dtype=np.float32)
            if self.dtype == "f16":
                self.t16[:m].copy_(self.t32[:m])
                flat[lo:lo + m] = self.t16[:m].view(torch.int16).numpy().view(np.uint16)
            else:
                flat[lo:lo + m] = bf16_bits_from_f32(self.f32[:m])

    def new(self, shape) -> np.ndarray:
        out = np.empty(shape, dtype=np.uint16)
        self.fill(out)
        return out


@dataclass
class Workload:
    """One batch of the hot path: new query tokens plus the full KV history.

    ``q`` holds the raw (unrotated) query rows of this step, token-major
    ``[T, Hq, d]`` in ``query_start_loc`` order.  ``k_all``/``v_all`` hold the
    raw key/value rows of every position of every sequence, ``[sum ctx, Hkv,
    d]``, sequence after sequence, positions ascending (``kv_start`` gives the
    offsets).  Positions ``[0, P_s)`` form the cached prefix, ``[P_s, ctx_s)``
    the tokens appended in this step.  All tensors are raw IEEE bits
    (``uint16``).
    """

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    theta: float
    scale: float
    prefix_lens: np.ndarray
    query_lens: np.ndarray
    num_blocks: int
    block_tables: np.ndarray
    q: np.ndarray
    k_all: np.ndarray
    v_all: np.ndarray
    shared_prefix_len: int = 0
    shared_seqs: tuple = ()

    # ---- derived layout -------------------------------------------------
    @property
    def dtype_code(self) -> int:
        return DTYPE_CODES[self.dtype]

    @property
    def num_seqs(self) -> int:
        return int(len(self.prefix_lens))

    @property
    def context_lens(self) -> np.ndarray:
        return (self.prefix_lens + self.query_lens).astype(np.int32)

    @property
    def query_start_loc(self) -> np.ndarray:
        out = np.zeros(self.num_seqs + 1, dtype=np.int32)
        np.cumsum(self.query_lens, out=out[1:])
        return out

    @property
    def kv_start(self) -> np.ndarray:
        out = np.zeros(self.num_seqs + 1, dtype=np.int64)
        np.cumsum(self.context_lens.astype(np.int64), out=out[1:])
        return out

    @property
    def num_tokens(self) -> int:
        return int(self.query_lens.sum())

    @property
    def positions(self) -> np.ndarray:
        """Absolute position of every query token (prefix length + index)."""
        parts = [np.arange(p, p + n, dtype=np.int32) for p, n in zip(self.prefix_lens, self.query_lens)]
        return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int32)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def max_query_len(self) -> int:
        return int(self.query_lens.max()) if self.num_seqs else 0

    def _row_index(self, which: str) -> np.ndarray:
        ks = self.kv_start
        parts = []
        for s in range(self.num_seqs):
            p, n = int(self.prefix_lens[s]), int(self.query_lens[s])
            if which == "step":
                parts.append(np.arange(ks[s] + p, ks[s] + p + n))
            else:
                parts.append(np.arange(ks[s], ks[s] + p))
        return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)

    def step_kv(self):
        """(k_new, v_new): raw rows of the tokens appended in this step."""
        idx = self._row_index("step")
        return self.k_all[idx], self.v_all[idx]

    def prefix_batch(self):
        """Arguments of the set-up append that fills the cached prefixes.

        Returns ``(k_rows, v_rows, query_start_loc, positions)``.
        """
        idx = self._row_index("prefix")
        qsl = np.zeros(self.num_seqs + 1, dtype=np.int32)
        np.cumsum(self.prefix_lens, out=qsl[1:])
        parts = [np.arange(0, p, dtype=np.int32) for p in self.prefix_lens]
        pos = np.concatenate(parts) if parts else np.zeros(0, dtype=np.int32)
        return self.k_all[idx], self.v_all[idx], qsl, pos


def _assign_blocks(rng, context_lens, block_size, spare, shared_prefix_len, shared_seqs):
    nblk = [(int(c) + block_size - 1) // block_size for c in context_lens]
    if shared_prefix_len % block_size:
        raise ValueError("shared prefix must fill whole blocks")
    n_shared = shared_prefix_len // block_size
    shared = set(int(s) for s in shared_seqs)
    private = [nb - (n_shared if s in shared else 0) for s, nb in enumerate(nblk)]
    num_blocks = (n_shared if shared else 0) + sum(private) + spare
    perm = rng.permutation(num_blocks).astype(np.int32)
    width = max(nblk) if nblk else 1
    table = np.full((len(nblk), max(width, 1)), TABLE_POISON, dtype=np.int32)
    shared_ids = perm[:n_shared] if shared else perm[:0]
    off = len(shared_ids)
    for s, nb in enumerate(nblk):
        j = 0
        if s in shared:
            table[s, :n_shared] = shared_ids
            j = n_shared
        table[s, j:nb] = perm[off:off + private[s]]
        off += private[s]
    return num_blocks, table


def build_workload(name: str, rng: np.random.Generator, *, num_q_heads: int, num_kv_heads: int,
                   head_dim: int, block_size: int, dtype: str, theta: float,
                   prefix_lens: Sequence[int], query_lens: Sequence[int], spare_blocks: int = 0,
                   shared_prefix_len: int = 0, shared_seqs: Sequence[int] = ()) -> Workload:
    """Finish a workload whose lengths are already drawn: blocks, q, k, v."""
    prefix = np.asarray(prefix_lens, dtype=np.int64).reshape(-1)
    qlen = np.asarray(query_lens, dtype=np.int64).reshape(-1)
    ctx = prefix + qlen
    for s in shared_seqs:
        if prefix[s] < shared_prefix_len:
            raise ValueError("a sharing sequence must hold the whole shared prefix in its cache")
    num_blocks, table = _assign_blocks(rng, ctx, block_size, spare_blocks, shared_prefix_len, shared_seqs)
    T = int(qlen.sum())
    gen = _NormalBits(rng, dtype)
    q = gen.new((T, num_q_heads, head_dim))

    shared = set(int(s) for s in shared_seqs)
    starts = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int64)

    def draw_rows():
        # shared prefix rows once, then each sequence's own rows, drawn in place
        out = np.empty((int(ctx.sum()), num_kv_heads, head_dim), dtype=np.uint16)
        first = None
        for s in sorted(shared):
            o = int(starts[s])
            if first is None:
                gen.fill(out[o:o + shared_prefix_len])
                first = o
            else:
                out[o:o + shared_prefix_len] = out[first:first + shared_prefix_len]
        for s in range(len(ctx)):
            o = int(starts[s]) + (shared_prefix_len if s in shared else 0)
            gen.fill(out[o:int(starts[s + 1])])
        return out

    k_all = draw_rows()
    v_all = draw_rows()
    return Workload(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                    block_size=block_size, dtype=dtype, theta=float(theta), scale=1.0 / math.sqrt(head_dim),
                    prefix_lens=prefix, query_lens=qlen, num_blocks=num_blocks, block_tables=table, q=q,
                    k_all=k_all, v_all=v_all, shared_prefix_len=shared_prefix_len if shared else 0,
                    shared_seqs=tuple(sorted(shared)))


def _rescale_to_total(raw: np.ndarray, total: int, lo: int, hi: int) -> np.ndarray:
    """Integers in [lo, hi] summing to ``total``, proportional to raw - lo.

    Largest-remainder rounding; lengths that would pass ``hi`` are clamped and
    their overflow is handed to the others (water filling).
    """
    n = len(raw)
    if not n * lo <= total <= n * hi:
        raise ValueError("total out of range")
    excess = (np.asarray(raw, dtype=np.int64) - lo).astype(np.float64)
    cap = hi - lo
    alloc = np.zeros(n, dtype=np.int64)
    active = list(range(n))
    remaining = total - n * lo
    while remaining > 0 and active:
        w = excess[active]
        if w.sum() <= 0:
            w = np.ones(len(active))
        share = remaining * w / w.sum()
        fl = np.floor(share).astype(np.int64)
        left = remaining - int(fl.sum())
        order = sorted(range(len(active)), key=lambda i: (-(share[i] - fl[i]), i))
        for i in order[:left]:
            fl[i] += 1
        still = []
        remaining = 0
        for i, a in enumerate(active):
            v = alloc[a] + fl[i]
            if v >= cap:
                remaining += int(v - cap)
                alloc[a] = cap
            else:
                alloc[a] = v
                still.append(a)
        active = still
    return alloc + lo


def make_config(name: str, seed: int | None = None) -> Workload:
    """The five named workloads; ``seed`` defaults to the config's index."""
    idx = CONFIG_NAMES.index(name)
    rng = np.random.Generator(np.random.PCG64(idx if seed is None else seed))
    llama = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, theta=5.0e5)
    if name == "tiny":
        return build_workload(name, rng, num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                              dtype="f16", theta=1.0e4, prefix_lens=[40, 23], query_lens=[17, 1],
                              spare_blocks=10)
    if name == "llama-decode":
        ctx = rng.integers(512, 4096, size=64, endpoint=True)
        return build_workload(name, rng, block_size=16, dtype="f16", prefix_lens=ctx - 1,
                              query_lens=np.ones(64, dtype=np.int64), spare_blocks=64, **llama)
    if name == "chunked-prefill":
        return build_workload(name, rng, block_size=16, dtype="f16", prefix_lens=[0, 1024, 2048, 3000],
                              query_lens=[512] * 4, **llama)
    if name == "mixed":
        budget, n_chunks, n_dec = 2048, 8, 200
        raw = rng.integers(128, 512, size=n_chunks, endpoint=True)
        chunk = _rescale_to_total(raw, budget - n_dec, 128, 512)
        p_shared = rng.integers(512, 4096, size=4, endpoint=True)
        p_other = rng.integers(0, 4096, size=4, endpoint=True)
        ctx_dec_shared = rng.integers(513, 8192, size=28, endpoint=True)
        ctx_dec_other = rng.integers(128, 8192, size=n_dec - 28, endpoint=True)
        prefix = np.concatenate([p_shared, p_other, ctx_dec_shared - 1, ctx_dec_other - 1])
        qlen = np.concatenate([chunk, np.ones(n_dec, dtype=np.int64)])
        shared = list(range(0, 4)) + list(range(8, 8 + 28))
        return build_workload(name, rng, block_size=16, dtype="f16", prefix_lens=prefix, query_lens=qlen,
                              spare_blocks=64, shared_prefix_len=512, shared_seqs=shared, **llama)
    if name == "long-decode":
        return build_workload(name, rng, block_size=32, dtype="bf16", prefix_lens=[32767] * 16,
                              query_lens=[1] * 16, **llama)
    raise KeyError(name)


def describe(w: Workload) -> dict:
    """Short, JSON-friendly summary of a workload's shape."""
    return {"workload": w.name, "num_seqs": w.num_seqs, "num_tokens": w.num_tokens,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "dtype": w.dtype, "num_blocks": w.num_blocks,
            "max_context_len": w.max_context_len, "rope_theta": w.theta}
