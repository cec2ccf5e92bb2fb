"""Seeded synthetic inputs for KPool indexer selection.

This module draws random numbers and lays out shapes; it holds none of the
method's arithmetic (no pooling, scoring, selection or expansion). Both the
CUDA path's tests and benchmark and the oracle's tests take their inputs from
here, so the two sides always see the same bytes: a test draws once (on the
CPU for small cases, on the GPU for the large ones) and copies to the other
side.

The shapes follow the GLM-5.3-Flash indexer the pages describe: 32 index heads
("spark_model/layers/glm5next_dsa/tp.rs", module docs), index_topk = 2048 and
kpool = 4 ("NVIDIA/Megatron-LM pull request #8299", section "Change"), head
dimension 128. The pages measure on real model activations, which are not
available here; these seeded draws stand in for them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    seqlens: tuple
    heads: int
    head_dim: int
    kpool: int
    index_topk: int
    scale: float
    dtype: str            # "bf16" or "f32": dtype of q and k (w is always fp32)
    values: str           # "normal": q,k ~ N(0,1), w ~ U(0,1)
                          # "integer": q,k uniform in {-2..2}, w uniform in {0,1/4,..,1}
    seed: int
    dup_every: int = 0    # >0: pool p with p % dup_every == dup_every-1 copies the
                          # kpool keys of a uniformly drawn earlier pool (exact ties)
    description: str = field(default="", compare=False)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens)

    @property
    def budget(self) -> int:
        return self.index_topk // self.kpool

    @property
    def width(self) -> int:
        return self.index_topk + self.kpool

    def cu_seqlens(self) -> torch.Tensor:
        cu = [0]
        for n in self.seqlens:
            cu.append(cu[-1] + int(n))
        return torch.tensor(cu, dtype=torch.int32)

    def causal_pairs(self) -> int:
        """Number of (query row, eligible pool) pairs: sum over rows of floor((t+1)/kpool)."""
        total = 0
        for L in self.seqlens:
            # sum_{m=1..L} floor(m/kpool), in closed form
            n, r = divmod(int(L), self.kpool)
            total += self.kpool * n * (n - 1) // 2 + n * (r + 1)
        return total

    def num_pools(self) -> int:
        return sum(int(L) // self.kpool for L in self.seqlens)


_S128 = 1.0 / math.sqrt(128.0)

TINY = Workload("tiny", (64,), 4, 32, 4, 16, 1.0 / math.sqrt(32.0), "f32", "normal", 1,
                description="Tiny causal: 1 x 64 tokens, kpool 4, H 4, d 32, index_topk 16, fp32")
TIE_HEAVY = Workload("tie_heavy", (4096, 4096), 32, 128, 4, 2048, 1.0 / 16.0, "bf16", "integer", 2,
                     dup_every=8,
                     description="Tie-heavy exact: 2 x 4096 tokens, integer-valued bf16, ties at the cutoff")
VARLEN = Workload("varlen", (8192, 16384, 3072, 5120), 32, 128, 4, 2048, _S128, "bf16", "normal", 3,
                  description="Packed varlen THD: lengths 8192/16384/3072/5120 (32768 tokens)")
LONG_128K = Workload("long_128k", (131072,), 32, 128, 4, 2048, _S128, "bf16", "normal", 4,
                     description="Long causal: 1 x 131072 tokens")
PAGES_512K = Workload("pages_512k", (524288,), 32, 128, 4, 2048, _S128, "bf16", "normal", 5,
                      description="Pages-scale causal: 1 x 524288 tokens")

ALL = (TINY, TIE_HEAVY, VARLEN, LONG_128K, PAGES_512K)
BY_NAME = {w.name: w for w in ALL}


def custom(name: str, seqlens, heads: int, head_dim: int, kpool: int, index_topk: int, scale: float,
           dtype: str = "bf16", values: str = "normal", seed: int = 0, dup_every: int = 0) -> Workload:
    return Workload(name, tuple(int(s) for s in seqlens), heads, head_dim, kpool, index_topk, scale,
                    dtype, values, seed, dup_every)


def generate(wl: Workload, device="cpu") -> dict:
    """Draw q [T,H,d], k [T,d] (dtype), w [T,H] fp32 and cu_seqlens [S+1] int32 on `device`.

    The generator is torch's, seeded with wl.seed (Philox on CUDA, MT19937 on the
    CPU), so the bytes depend on the device; callers that need both sides copy.
    """
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed)
    T, H, d = wl.total_tokens, wl.heads, wl.head_dim
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    if wl.values == "normal":
        q = torch.randn((T, H, d), generator=g, device=device, dtype=torch.float32).to(tdt)
        k = torch.randn((T, d), generator=g, device=device, dtype=torch.float32).to(tdt)
        w = torch.rand((T, H), generator=g, device=device, dtype=torch.float32)
    elif wl.values == "integer":
        q = torch.randint(-2, 3, (T, H, d), generator=g, device=device, dtype=torch.int32).to(tdt)
        k = torch.randint(-2, 3, (T, d), generator=g, device=device, dtype=torch.int32).to(tdt)
        w = torch.randint(0, 5, (T, H), generator=g, device=device, dtype=torch.int32).to(torch.float32) / 4.0
    else:
        raise ValueError(f"unknown value recipe {wl.values!r}")
    cu = wl.cu_seqlens()
    if wl.dup_every > 0:
        _plant_duplicate_pools(k, cu, wl.kpool, wl.dup_every, wl.seed)
    return {"q": q, "k": k, "w": w, "cu_seqlens": cu.to(device)}


def _plant_duplicate_pools(k: torch.Tensor, cu: torch.Tensor, kpool: int, every: int, seed: int) -> None:
    """Copy the kpool keys of a random earlier pool onto every `every`-th pool (in place)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 7919)
    for b in range(len(cu) - 1):
        start, L = int(cu[b]), int(cu[b + 1] - cu[b])
        n = L // kpool
        if n < every:
            continue
        dst = torch.arange(every - 1, n, every)
        # draw src uniformly in [0, dst): floor(u * dst)
        u = torch.rand(len(dst), generator=g, dtype=torch.float64)
        src = torch.minimum((u * dst.to(torch.float64)).floor().to(torch.int64), dst - 1)
        for s_pool, d_pool in zip(src.tolist(), dst.tolist()):
            a = start + s_pool * kpool
            z = start + d_pool * kpool
            k[z:z + kpool] = k[a:a + kpool]


def sample_rows(wl: Workload, count: int, seed: int = 12345) -> torch.Tensor:
    """A stratified sample of global rows: each sequence's first and last rows, rows at
    every kpool phase near the ends and around local row index_topk (where a row's
    eligible pools first exceed the budget), and uniform draws (sorted, unique, int64)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    cu = wl.cu_seqlens().tolist()
    picks = set()
    span = 2 * wl.kpool
    for b in range(wl.num_seqs):
        s, e = cu[b], cu[b + 1]
        if e <= s:
            continue
        for t in list(range(s, min(e, s + span + 1))) + list(range(max(s, e - span), e)):
            picks.add(t)
        mid = s + wl.index_topk
        for t in range(max(s, mid - span), min(e, mid + span + 1)):
            picks.add(t)
    T = wl.total_tokens
    while len(picks) < min(count, T):  # uniform draws until `count` distinct rows
        picks.update(torch.randint(0, T, (count - len(picks),), generator=g).tolist())
    return torch.tensor(sorted(picks), dtype=torch.int64)


# --------------------------------------------------------------- explicit query rows
#
# The decode / short-query case: a few query rows, each at a position of one key
# sequence, score that sequence's pooled-key cache. The pages' example is one
# decode token at a 262,144-token context scoring 65,536 pools
# ("spark_model/layers/glm5next_dsa/tp.rs", module docs, "Why the indexer is
# REPLICATED"); a batch of such sequences stands in for a decode batch.


@dataclass(frozen=True)
class RowsWorkload:
    name: str
    seqlens: tuple        # key sequences (the cache)
    rows: tuple           # ((seq, pos), ...) of the query rows; pos < 0 means seqlens[seq] + pos
    heads: int
    head_dim: int
    kpool: int
    index_topk: int
    scale: float
    dtype: str
    values: str
    seed: int
    dup_every: int = 0
    description: str = field(default="", compare=False)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens)

    @property
    def num_rows(self) -> int:
        return len(self.rows)

    @property
    def budget(self) -> int:
        return self.index_topk // self.kpool

    @property
    def width(self) -> int:
        return self.index_topk + self.kpool

    def cu_seqlens(self) -> torch.Tensor:
        return Workload("", self.seqlens, 1, 1, 1, 1, 1.0, "f32", "normal", 0).cu_seqlens()

    def row_positions(self):
        """(seq, pos) of every row with negative positions resolved."""
        out = []
        for b, t in self.rows:
            out.append((int(b), int(t) if t >= 0 else int(self.seqlens[b]) + int(t)))
        return out

    def global_rows(self):
        cu = self.cu_seqlens().tolist()
        return [cu[b] + t for b, t in self.row_positions()]

    def scored_pairs(self) -> int:
        return sum((t + 1) // self.kpool for _, t in self.row_positions())


DECODE_SMALL = RowsWorkload(
    "decode_small", (5000, 12345, 2, 8191),
    ((0, -1), (1, -1), (3, -1), (2, 1), (0, 0), (0, 2), (0, 3), (1, 2047), (1, 2048), (1, 6000), (3, 4099),
     (3, 4095), (1, -2), (0, 1234), (3, 2049), (1, -1)),
    32, 128, 4, 2048, _S128, "bf16", "normal", 11,
    description="Decode rows against four key caches (5000/12345/2/8191 tokens) at assorted positions")
DECODE_TIE = RowsWorkload(
    "decode_tie", (4096, 6000),
    ((0, -1), (1, -1), (0, 2051), (1, 4999), (0, 100), (1, -3)),
    32, 128, 4, 2048, 1.0 / 16.0, "bf16", "integer", 12, dup_every=8,
    description="Integer-valued decode rows with duplicated pools (exact ties at the cutoff)")
DECODE_262K = RowsWorkload(
    "decode_262k", (262144,) * 16, tuple((b, -1) for b in range(16)),
    32, 128, 4, 2048, _S128, "bf16", "normal", 13,
    description="Decode batch: 16 sequences x 262,144-token caches, one new query row each (65,536 pools)")

ROWS_ALL = (DECODE_SMALL, DECODE_TIE, DECODE_262K)
ROWS_BY_NAME = {w.name: w for w in ROWS_ALL}


def generate_rows(wl: RowsWorkload, device="cpu") -> dict:
    """Draw the key cache k [T,d], cu_seqlens, and the rows' q [R,H,d], w [R,H], row_seq, row_pos."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed)
    T, H, d, R = wl.total_tokens, wl.heads, wl.head_dim, wl.num_rows
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    if wl.values == "normal":
        k = torch.randn((T, d), generator=g, device=device, dtype=torch.float32).to(tdt)
        q = torch.randn((R, H, d), generator=g, device=device, dtype=torch.float32).to(tdt)
        w = torch.rand((R, H), generator=g, device=device, dtype=torch.float32)
    elif wl.values == "integer":
        k = torch.randint(-2, 3, (T, d), generator=g, device=device, dtype=torch.int32).to(tdt)
        q = torch.randint(-2, 3, (R, H, d), generator=g, device=device, dtype=torch.int32).to(tdt)
        w = torch.randint(0, 5, (R, H), generator=g, device=device, dtype=torch.int32).to(torch.float32) / 4.0
    else:
        raise ValueError(f"unknown value recipe {wl.values!r}")
    cu = wl.cu_seqlens()
    if wl.dup_every > 0:
        _plant_duplicate_pools(k, cu, wl.kpool, wl.dup_every, wl.seed)
    pos = wl.row_positions()
    row_seq = torch.tensor([b for b, _ in pos], dtype=torch.int32)
    row_pos = torch.tensor([t for _, t in pos], dtype=torch.int32)
    return {"k": k, "q": q, "w": w, "cu_seqlens": cu.to(device), "row_seq": row_seq.to(device),
            "row_pos": row_pos.to(device)}
