"""Seeded synthetic inputs for range-masked attention.

This module is shared by the oracle tests and by the CUDA path's tests and benchmark, so
both sides see identical inputs.  It holds no attention arithmetic: only random draws,
slice lists and the workload descriptions.

Conventions (the pages leave the random-number recipe open):
  * "seed s": one ``torch.Generator('cpu')`` seeded with s; q, k, v, dO are drawn in that
    order with ``torch.randn(..., dtype=float32)`` and rounded to bfloat16.
  * Document lengths (packed-document workload) come from a second generator seeded with
    the same s, drawing ``randint(128, 4097)`` until the running sum reaches the total;
    the last document is truncated so the lengths sum exactly to the total.
  * Slice type codes follow the flex_flash_attn_func interface (MagiAttention issue #180,
    "Using dummy/padded attention slices ..."): 0 = FULL, 1 = CAUSAL.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch

FULL = 0
CAUSAL = 1


@dataclass
class Workload:
    """One attention problem: shapes, slices and the input seed."""

    name: str
    total: int                 # packed tokens (q and k share the token axis here)
    hq: int
    hkv: int
    d: int
    seed: int
    q_ranges: List[Tuple[int, int]]
    k_ranges: List[Tuple[int, int]]
    types: List[int]
    softcap: float = 0.0
    softmax_scale: Optional[float] = None   # None -> 1/sqrt(d)
    backward: bool = True
    pad_to: int = 0                          # append start==end dummies up to this many slices
    doc_lengths: List[int] = field(default_factory=list)

    @property
    def n_slices(self) -> int:
        return len(self.types)

    def padded(self) -> "Workload":
        """Return a copy whose slice list is padded with [0,0)x[0,0) FULL dummies."""
        n = max(self.pad_to, len(self.types))
        extra = n - len(self.types)
        w = Workload(**{**self.__dict__})
        w.q_ranges = list(self.q_ranges) + [(0, 0)] * extra
        w.k_ranges = list(self.k_ranges) + [(0, 0)] * extra
        w.types = list(self.types) + [FULL] * extra
        return w


def make_generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def draw_qkv(total_q: int, total_k: int, hq: int, hkv: int, d: int, seed: int,
             with_dout: bool = True):
    """q:[Nq,Hq,d], k,v:[Nk,Hkv,d], dO:[Nq,Hq,d] as bf16 CPU tensors, N(0,1) before rounding."""
    g = make_generator(seed)
    q = torch.randn(total_q, hq, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(total_k, hkv, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(total_k, hkv, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    do = None
    if with_dout:
        do = torch.randn(total_q, hq, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return q, k, v, do


def draw_document_lengths(total: int, seed: int, lo: int = 128, hi: int = 4096) -> List[int]:
    g = make_generator(seed)
    lens: List[int] = []
    s = 0
    while s < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        n = min(n, total - s)
        lens.append(n)
        s += n
    return lens


def ranges_tensors(w: Workload):
    """(q_ranges [R,2] int32, k_ranges [R,2] int32, types [R] int32) CPU tensors."""
    qr = torch.tensor(w.q_ranges, dtype=torch.int32).reshape(-1, 2)
    kr = torch.tensor(w.k_ranges, dtype=torch.int32).reshape(-1, 2)
    ty = torch.tensor(w.types, dtype=torch.int32).reshape(-1)
    return qr, kr, ty


# --------------------------------------------------------------------------------------
# The five workloads.  Sizes, slice lists, seeds and flags follow the benchmark
# configurations of this project; the page-1 shape (2048 tokens, 8/2 heads, d 64, FULL then
# CAUSAL slice, padded to 20) is the one the MagiAttention issue's parity script uses.
# --------------------------------------------------------------------------------------

def tiny() -> Workload:
    return Workload(
        name="tiny_256", total=256, hq=2, hkv=1, d=64, seed=0,
        q_ranges=[(0, 128), (128, 256)], k_ranges=[(0, 128), (0, 256)], types=[FULL, CAUSAL],
        softmax_scale=1.0 / 8.0, pad_to=4)


def page1() -> Workload:
    return Workload(
        name="page1_2048_gqa", total=2048, hq=8, hkv=2, d=64, seed=0,
        q_ranges=[(0, 1024), (1024, 2048)], k_ranges=[(0, 1024), (0, 2048)],
        types=[FULL, CAUSAL], pad_to=20)


def documents() -> Workload:
    total = 16384
    lens = draw_document_lengths(total, seed=1)
    qr, kr, ty = [], [], []
    s = 0
    for n in lens:
        qr.append((s, s + n))
        kr.append((s, s + n))
        ty.append(CAUSAL)
        s += n
    return Workload(name="docs_16k", total=total, hq=16, hkv=16, d=128, seed=1,
                    q_ranges=qr, k_ranges=kr, types=ty, backward=False, doc_lengths=lens)


def sliding_softcap() -> Workload:
    total = 32768
    qr, kr, ty = [], [], []
    for b in range(total // 256):
        lo = 256 * b
        qr.append((lo, lo + 256)); kr.append((lo, lo + 256)); ty.append(CAUSAL)
        qr.append((lo, lo + 256)); kr.append((max(0, lo - 1024), lo)); ty.append(FULL)
    return Workload(name="sliding_32k_softcap", total=total, hq=32, hkv=8, d=128, seed=2,
                    q_ranges=qr, k_ranges=kr, types=ty, softcap=30.0)


def long_causal() -> Workload:
    total = 65536
    return Workload(
        name="long_causal_64k_prefix", total=total, hq=16, hkv=4, d=128, seed=3,
        q_ranges=[(0, total), (0, 4096), (0, 4096)],
        k_ranges=[(0, total), (0, 4096), (0, 4096)],
        types=[CAUSAL, FULL, FULL])


def long_causal_16k() -> Workload:
    """The long-causal recipe at a quarter of the length (profiling-sized: inputs > L2)."""
    total = 16384
    return Workload(
        name="long_causal_16k_prefix", total=total, hq=16, hkv=4, d=128, seed=3,
        q_ranges=[(0, total), (0, 4096), (0, 4096)],
        k_ranges=[(0, total), (0, 4096), (0, 4096)],
        types=[CAUSAL, FULL, FULL])


ALL = {w.name: w for w in (tiny(), page1(), documents(), sliding_softcap(), long_causal(), long_causal_16k())}
ORDER = ["tiny_256", "page1_2048_gqa", "docs_16k", "sliding_32k_softcap", "long_causal_64k_prefix"]


def get(name: str) -> Workload:
    return ALL[name]


# --------------------------------------------------------------------------------------
# Random slice sets for parity tests (overlapping, unaligned, zero-length, q_len != k_len).
# --------------------------------------------------------------------------------------

def random_slices(total_q: int, total_k: int, n: int, seed: int, p_dummy: float = 0.15,
                  p_causal: float = 0.5):
    g = make_generator(seed + 7919)

    def ri(lo, hi):  # inclusive lo, exclusive hi
        if hi <= lo:
            return lo
        return int(torch.randint(lo, hi, (1,), generator=g).item())

    qr, kr, ty = [], [], []
    for _ in range(n):
        u = float(torch.rand((), generator=g).item())
        if u < p_dummy:
            a = ri(0, total_q + 1)
            b = ri(0, total_k + 1)
            form = ri(0, 3)
            if form == 0:
                qr.append((a, a)); kr.append((0, total_k))
            elif form == 1:
                qr.append((0, total_q)); kr.append((b, b))
            else:
                qr.append((a, a)); kr.append((b, b))
            ty.append(ri(0, 2))
            continue
        qs = ri(0, total_q)
        qe = ri(qs + 1, total_q + 1)
        ks = ri(0, total_k)
        ke = ri(ks + 1, total_k + 1)
        qr.append((qs, qe)); kr.append((ks, ke))
        ty.append(CAUSAL if float(torch.rand((), generator=g).item()) < p_causal else FULL)
    return qr, kr, ty


def random_page_table(n_logical: int, n_pages: int, seed: int) -> torch.Tensor:
    """Distinct physical pages for n_logical logical pages out of a pool of n_pages (a seeded
    random permutation prefix), int32 -- the page table of a paged key/value cache."""
    g = make_generator(seed)
    return torch.randperm(n_pages, generator=g)[:n_logical].to(torch.int32)

# --------------------------------------------------------------------------------------
# Decoding batches: n_seq sequences, each with q_len new query tokens at the end of its
# kv_len keys (one CAUSAL slice per sequence: bottom-right alignment makes the new tokens see
# every earlier key), packed one sequence after another on both token axes.
# --------------------------------------------------------------------------------------

@dataclass
class DecodeWorkload:
    name: str
    n_seq: int
    q_len: int
    kv_len: int
    hq: int
    hkv: int
    d: int
    seed: int

    @property
    def total_q(self) -> int:
        return self.n_seq * self.q_len

    @property
    def total_k(self) -> int:
        return self.n_seq * self.kv_len

    def slices(self):
        qr = [(s * self.q_len, (s + 1) * self.q_len) for s in range(self.n_seq)]
        kr = [(s * self.kv_len, (s + 1) * self.kv_len) for s in range(self.n_seq)]
        return qr, kr, [CAUSAL] * self.n_seq

    def draw(self):
        """q [n_seq * q_len, Hq, d], k, v [n_seq * kv_len, Hkv, d]: bf16 N(0,1), seeded."""
        g = make_generator(self.seed)
        q = torch.randn(self.total_q, self.hq, self.d, generator=g).to(torch.bfloat16)
        k = torch.randn(self.total_k, self.hkv, self.d, generator=g).to(torch.bfloat16)
        v = torch.randn(self.total_k, self.hkv, self.d, generator=g).to(torch.bfloat16)
        return q, k, v


DECODE = {w.name: w for w in (
    DecodeWorkload("decode_64x8k_g4", n_seq=64, q_len=1, kv_len=8192, hq=16, hkv=4, d=128, seed=11),
    DecodeWorkload("decode_8x64k_g8", n_seq=8, q_len=1, kv_len=65536, hq=16, hkv=2, d=128, seed=12),
)}
