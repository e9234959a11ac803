"""Seeded synthetic inputs for block-sparse top-k GQA attention.

This module only *generates inputs*: Q/K/V values, top-k block index lists
(``q2k``), page tables and KV lengths.  It holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle can consume its output.

Randomness is counter based: every value is a pure function of
``(seed, stream, element index)``, evaluated with exact int64 tensor ops, so
the same call gives bit-identical tensors on the CPU and on a CUDA device.

* Integer hash: the two-round xorshift-multiply 32-bit hash published by
  C. Wellons ("Hash Prospector", constants 0x21f0aaad / 0x735a2d97, shifts
  16/15/15), chained over the seed, the stream id and the index words.
* N(0,1) bf16: the top 16 bits of a hash pick one of 65536 equiprobable
  quantiles ``Phi^-1((i + 0.5) / 65536)`` (float64, then rounded to bf16).
* Distinct picks: R. Floyd's sampling algorithm (Bentley & Floyd, CACM 1987),
  run for all rows at once; draw order is kept.
* Random permutation prefixes: partial Fisher-Yates.

Pattern recipes follow the workloads of the MSA sparse-attention test and
benchmark page (``test_sparse_atten.py``: ``generate_test_data``,
``_build_pattern_q2k``, ``_bottom_right_causal_visible_blocks``) with the
selection rule fixed per workload:

* ``q2k_perm_prefix``: non-causal, first ``topk`` entries of a fresh
  permutation of all blocks (``generate_test_data``, non-causal branch).
* ``q2k_causal_sink``: block 0, the diagonal (last visible) block, then
  ``topk-2`` distinct uniform picks from the other visible blocks.
* ``q2k_causal_uniform``: the diagonal block, then ``topk-1`` distinct uniform
  picks from the other visible blocks.
* ``q2k_decode``: the last visible block, then ``topk-1`` distinct uniform picks
  from the other visible blocks (paged decode, positions ``seqused-Sq..``).

When a query sees ``V <= topk`` blocks it takes all of them (fixed slots first,
then the rest ascending) and pads with -1.  Rows with ``V == 0`` are all -1.
"""

from __future__ import annotations

import itertools
import math
from dataclasses import dataclass, field
from typing import Optional

import torch

MASK32 = 0xFFFFFFFF
_H1 = 0x21F0AAAD
_H2 = 0x735A2D97

# Stream ids: one per kind of draw, so no two draws share a counter space.
STREAM_Q = 1
STREAM_K = 2
STREAM_V = 3
STREAM_Q2K = 4
STREAM_PAGES = 5
STREAM_AUX = 6

DEFAULT_SEED = 42
BLK = 128


# ---------------------------------------------------------------------------
# counter-based integer hash (exact int64 arithmetic, CPU == CUDA)
# ---------------------------------------------------------------------------

def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for 0 <= x < 2^32, without int64 overflow."""
    lo = x * (c & 0xFFFF)
    hi = ((x * (c >> 16)) & 0xFFFF) << 16
    return (lo + hi) & MASK32


def hash32(x: torch.Tensor) -> torch.Tensor:
    """Wellons' low-bias 32-bit hash; ``x`` int64 holding values < 2^32."""
    x = x & MASK32
    x = x ^ (x >> 16)
    x = _mul32(x, _H1)
    x = x ^ (x >> 15)
    x = _mul32(x, _H2)
    x = x ^ (x >> 15)
    return x


def _hash_int(v: int) -> int:
    return int(hash32(torch.tensor([v & MASK32], dtype=torch.int64))[0])


def stream_key(seed: int, stream: int) -> int:
    return _hash_int(stream ^ _hash_int(seed))


def counter_u32(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """32 random bits per element of ``idx`` (int64, >= 0, < 2^62)."""
    key = stream_key(seed, stream)
    lo = idx & MASK32
    hi = idx >> 32
    if bool((hi == 0).all()):
        return hash32(lo ^ _hash_int(key))
    return hash32(lo ^ hash32(hi ^ key))


def uniform_below(bits: torch.Tensor, n: torch.Tensor) -> torch.Tensor:
    """Map 32 random bits to an integer in [0, n) (multiply-high, n < 2^30)."""
    return (bits * n) >> 32


# ---------------------------------------------------------------------------
# N(0,1) bf16 values
# ---------------------------------------------------------------------------

_QUANTILES: dict = {}


def _normal_table(device) -> torch.Tensor:
    key = str(device)
    if key not in _QUANTILES:
        p = (torch.arange(65536, dtype=torch.float64) + 0.5) / 65536.0
        tab = torch.special.ndtri(p).to(torch.bfloat16)
        _QUANTILES[key] = tab.to(device)
    return _QUANTILES[key]


def normal_bf16(shape, seed: int, stream: int, device="cpu",
                chunk: int = 1 << 26, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """bf16 tensor ~N(0,1); element i = table[hash(seed, stream, i) >> 16]."""
    numel = math.prod(shape)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    tab = _normal_table(flat.device)
    for start in range(0, numel, chunk):
        n = min(chunk, numel - start)
        idx = torch.arange(start, start + n, dtype=torch.int64, device=flat.device)
        bits = counter_u32(seed, stream, idx)
        flat[start:start + n] = tab[bits >> 16]
    return out


# ---------------------------------------------------------------------------
# top-k block index generators
# ---------------------------------------------------------------------------

def causal_visible_blocks(q_pos: torch.Tensor, kv_len: int, sq: int, blk: int, nblk: int) -> torch.Tensor:
    """Blocks a bottom-right-causal query at local position ``q_pos`` can see."""
    limit = q_pos + (kv_len - sq)
    return torch.clamp(torch.div(limit, blk, rounding_mode="floor") + 1, 0, nblk)


def _rand_bits(seed: int, stream: int, row_ids: torch.Tensor, draw: int) -> torch.Tensor:
    # 64 draws per row at most; counter = row * 64 + draw.
    return counter_u32(seed, stream, row_ids * 64 + draw)


def _floyd_distinct(seed: int, stream: int, row_ids: torch.Tensor, n: torch.Tensor, k: int) -> torch.Tensor:
    """k distinct picks from [0, n) per row (requires n >= k), Floyd's method."""
    rows = row_ids.numel()
    chosen = torch.empty((rows, k), dtype=torch.int64, device=row_ids.device)
    for e in range(k):
        j = n - k + e
        t = uniform_below(_rand_bits(seed, stream, row_ids, e), j + 1)
        if e > 0:
            dup = (chosen[:, :e] == t[:, None]).any(dim=1)
            t = torch.where(dup, j, t)
        chosen[:, e] = t
    return chosen


def _fill_pattern(V: torch.Tensor, topk: int, fixed: list, rand_lo: int,
                  seed: int, stream: int, row_ids: torch.Tensor) -> torch.Tensor:
    """Build rows of ``topk`` slots.

    ``fixed`` lists per-row tensors of forced blocks (e.g. block 0, diagonal),
    ``rand_lo`` is the first block of the random range, whose size is
    ``V - len(fixed)``.  Rows with V <= topk take all visible blocks.
    """
    rows = V.numel()
    dev = V.device
    out = torch.full((rows, topk), -1, dtype=torch.int64, device=dev)
    nfix = len(fixed)
    big = V > topk
    # rows that see more than topk blocks: fixed slots + random distinct picks
    if bool(big.any()):
        bi = big.nonzero().flatten()
        for s, f in enumerate(fixed):
            out[bi, s] = f[bi]
        picks = _floyd_distinct(seed, stream, row_ids[bi], V[bi] - nfix, topk - nfix)
        out[bi, nfix:] = picks + rand_lo
    # rows that see V <= topk blocks: fixed slots, then the others ascending
    small = (~big) & (V > 0)
    if bool(small.any()):
        si = small.nonzero().flatten()
        Vs = V[si]
        ar = torch.arange(topk, dtype=torch.int64, device=dev)[None, :].expand(si.numel(), topk)
        # candidate list: all visible blocks ascending, with the fixed ones moved to the front
        cand = ar.clone()
        if nfix:
            fx = torch.stack([f[si] for f in fixed], dim=1)  # [n, nfix]
            # blocks that are not fixed, ascending
            is_fixed = (ar[:, :, None] == fx[:, None, :]).any(dim=2)
            key = torch.where(is_fixed, torch.full_like(ar, -1), ar)
            key = torch.where(ar < Vs[:, None], key, torch.full_like(ar, 1 << 40))
            # fixed blocks that are visible and distinct go first, in slot order
            fx_valid = fx < Vs[:, None]
            for s in range(1, nfix):
                fx_valid[:, s] &= ~(fx[:, :s] == fx[:, s:s + 1]).any(dim=1)
            order_key = torch.cat([
                torch.where(fx_valid, torch.arange(nfix, device=dev)[None, :] - nfix - 1, torch.full_like(fx, 1 << 41)),
                torch.where(key >= 0, key, torch.full_like(key, 1 << 41)),
            ], dim=1)
            vals = torch.cat([fx, ar], dim=1)
            srt = torch.argsort(order_key, dim=1, stable=True)
            cand = torch.gather(vals, 1, srt)[:, :topk]
        cand = torch.where(ar < Vs[:, None], cand, torch.full_like(cand, -1))
        out[si] = cand
    return out


def q2k_perm_prefix(B: int, Hkv: int, Sq: int, nblk: int, topk: int, seed: int = DEFAULT_SEED,
                    device="cpu") -> torch.Tensor:
    """[B,Hkv,Sq,topk] int32: first ``topk`` entries of a random permutation of 0..nblk-1."""
    rows = B * Hkv * Sq
    row_ids = torch.arange(rows, dtype=torch.int64, device=device)
    arr = torch.arange(nblk, dtype=torch.int64, device=device)[None, :].repeat(rows, 1)
    for i in range(topk):
        j = i + uniform_below(_rand_bits(seed, STREAM_Q2K, row_ids, i),
                              torch.full_like(row_ids, nblk - i))
        ai = arr[:, i].clone()
        aj = torch.gather(arr, 1, j[:, None])[:, 0]
        arr[:, i] = aj
        arr.scatter_(1, j[:, None], ai[:, None])
    return arr[:, :topk].to(torch.int32).view(B, Hkv, Sq, topk)


def _causal_rows(B, Hkv, Sq, kv_len, blk, nblk, device):
    s = torch.arange(Sq, dtype=torch.int64, device=device)
    V = causal_visible_blocks(s, kv_len, Sq, blk, nblk)
    V = V[None, None, :].expand(B, Hkv, Sq).reshape(-1)
    row_ids = torch.arange(B * Hkv * Sq, dtype=torch.int64, device=device)
    return V, row_ids


def q2k_causal_sink(B: int, Hkv: int, Sq: int, Skv: int, topk: int, blk: int = BLK,
                    seed: int = DEFAULT_SEED, device="cpu") -> torch.Tensor:
    """[B,Hkv,Sq,topk]: block 0, the diagonal block, topk-2 distinct random others."""
    nblk = (Skv + blk - 1) // blk
    V, row_ids = _causal_rows(B, Hkv, Sq, Skv, blk, nblk, device)
    zero = torch.zeros_like(V)
    diag = V - 1
    out = _fill_pattern(V, topk, [zero, diag], 1, seed, STREAM_Q2K, row_ids)
    return out.to(torch.int32).view(B, Hkv, Sq, topk)


def q2k_causal_uniform(B: int, Hkv: int, Sq: int, Skv: int, topk: int, blk: int = BLK,
                       seed: int = DEFAULT_SEED, device="cpu") -> torch.Tensor:
    """[B,Hkv,Sq,topk]: the diagonal block, then topk-1 distinct random others."""
    nblk = (Skv + blk - 1) // blk
    V, row_ids = _causal_rows(B, Hkv, Sq, Skv, blk, nblk, device)
    diag = V - 1
    out = _fill_pattern(V, topk, [diag], 0, seed, STREAM_Q2K, row_ids)
    return out.to(torch.int32).view(B, Hkv, Sq, topk)


def q2k_decode(B: int, Hkv: int, Sq: int, seqused: torch.Tensor, topk: int, blk: int = BLK,
               seed: int = DEFAULT_SEED, device="cpu") -> torch.Tensor:
    """[B,Hkv,Sq,topk] for paged decode.

    Query i of sequence b sits at position ``seqused[b] - Sq + i`` and sees keys
    up to that position.  Slots: last visible block, then topk-1 distinct
    random others (or every visible block when there are at most topk).
    """
    su = seqused.to(torch.int64).to(device)
    i = torch.arange(Sq, dtype=torch.int64, device=device)
    pos = su[:, None] - Sq + i[None, :]                                   # [B, Sq]
    V = torch.clamp(torch.div(pos, blk, rounding_mode="floor") + 1, min=0)  # [B, Sq]
    V = torch.where(pos >= 0, V, torch.zeros_like(V))
    V = V[:, None, :].expand(B, Hkv, Sq).reshape(-1)
    row_ids = torch.arange(B * Hkv * Sq, dtype=torch.int64, device=device)
    last = V - 1
    out = _fill_pattern(V, topk, [last], 0, seed, STREAM_Q2K, row_ids)
    return out.to(torch.int32).view(B, Hkv, Sq, topk)


def shuffled_page_table(B: int, pages_per_seq: int, seed: int = DEFAULT_SEED, device="cpu") -> torch.Tensor:
    """[B, pages_per_seq] int32: one random permutation of all B*pages_per_seq pages."""
    n = B * pages_per_seq
    idx = torch.arange(n, dtype=torch.int64, device=device)
    keys = counter_u32(seed, STREAM_PAGES, idx) * n + idx  # distinct sort keys
    perm = torch.argsort(keys)
    return perm.to(torch.int32).view(B, pages_per_seq)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

@dataclass
class PrefillSpec:
    """Dense-KV prefill workload: Q [B,Sq,Hq,D], K/V [B,Skv,Hkv,D], q2k [B,Hkv,Sq,topk]."""
    name: str
    B: int
    Sq: int
    Skv: int
    Hkv: int
    qpk: int
    topk: int
    causal: bool
    pattern: str            # "perm_prefix" | "sink" | "uniform"
    D: int = 128
    blk: int = BLK
    kv_format: str = "bf16"  # "bf16" | "nvfp4"
    seed: int = DEFAULT_SEED

    @property
    def Hq(self) -> int:
        return self.Hkv * self.qpk

    @property
    def nblk(self) -> int:
        return (self.Skv + self.blk - 1) // self.blk


@dataclass
class DecodeSpec:
    """Paged decode workload: pool [num_pages,page,Hkv,D], page_table [B,pages_per_seq]."""
    name: str
    B: int
    Sq: int
    Hkv: int
    qpk: int
    topk: int
    kv_len: int
    trim: int
    D: int = 128
    page: int = BLK
    seed: int = DEFAULT_SEED

    @property
    def Hq(self) -> int:
        return self.Hkv * self.qpk

    @property
    def pages_per_seq(self) -> int:
        return (self.kv_len + self.page - 1) // self.page

    @property
    def num_pages(self) -> int:
        return self.B * self.pages_per_seq

    @property
    def seqused(self) -> int:
        return max(1, self.kv_len - self.trim)


# The prefill workloads: a tiny non-causal case, then causal 32K, 48K and 384K
# cases (the last also with NVFP4 K/V).  paged_decode_spec gives the decode sweep.
TINY_NONCAUSAL_1K = PrefillSpec("tiny_noncausal_1k", B=1, Sq=1024, Skv=1024, Hkv=1, qpk=2, topk=4,
                                causal=False, pattern="perm_prefix")
CAUSAL_SINK_32K = PrefillSpec("causal_sink_32k", B=1, Sq=32768, Skv=32768, Hkv=4, qpk=16, topk=16,
                              causal=True, pattern="sink")
CAUSAL_UNIFORM_48K = PrefillSpec("causal_uniform_48k", B=1, Sq=49152, Skv=49152, Hkv=1, qpk=16, topk=16,
                                 causal=True, pattern="uniform")
CAUSAL_SINK_384K = PrefillSpec("causal_sink_384k", B=1, Sq=393216, Skv=393216, Hkv=1, qpk=2, topk=16,
                               causal=True, pattern="sink")
CAUSAL_SINK_384K_NVFP4 = PrefillSpec("causal_sink_384k_nvfp4", B=1, Sq=393216, Skv=393216, Hkv=1, qpk=2,
                                     topk=16, causal=True, pattern="sink", kv_format="nvfp4")
DECODE_SWEEP_L = tuple(1024 << i for i in range(8))   # 1K .. 128K


def paged_decode_spec(kv_len: int) -> DecodeSpec:
    return DecodeSpec(f"paged_decode_{kv_len // 1024}k", B=32, Sq=8, Hkv=4, qpk=16, topk=16,
                      kv_len=kv_len, trim=17)


def make_prefill_q2k(spec: PrefillSpec, device="cpu") -> torch.Tensor:
    if spec.pattern == "perm_prefix":
        return q2k_perm_prefix(spec.B, spec.Hkv, spec.Sq, spec.nblk, spec.topk, spec.seed, device)
    if spec.pattern == "sink":
        return q2k_causal_sink(spec.B, spec.Hkv, spec.Sq, spec.Skv, spec.topk, spec.blk, spec.seed, device)
    if spec.pattern == "uniform":
        return q2k_causal_uniform(spec.B, spec.Hkv, spec.Sq, spec.Skv, spec.topk, spec.blk, spec.seed, device)
    raise ValueError(f"unknown pattern {spec.pattern!r}")


def make_prefill_inputs(spec: PrefillSpec, device="cpu") -> dict:
    """Q, K, V (bf16) and q2k (int32) for a dense prefill workload."""
    q = normal_bf16((spec.B, spec.Sq, spec.Hq, spec.D), spec.seed, STREAM_Q, device)
    k = normal_bf16((spec.B, spec.Skv, spec.Hkv, spec.D), spec.seed, STREAM_K, device)
    v = normal_bf16((spec.B, spec.Skv, spec.Hkv, spec.D), spec.seed, STREAM_V, device)
    q2k = make_prefill_q2k(spec, device)
    return {"q": q, "k": k, "v": v, "q2k": q2k}


def make_decode_inputs(spec: DecodeSpec, device="cpu") -> dict:
    """Q [B*Sq,Hq,D], K/V pools [num_pages,page,Hkv,D], page_table, seqused, q2k."""
    q = normal_bf16((spec.B * spec.Sq, spec.Hq, spec.D), spec.seed, STREAM_Q, device)
    k = normal_bf16((spec.num_pages, spec.page, spec.Hkv, spec.D), spec.seed, STREAM_K, device)
    v = normal_bf16((spec.num_pages, spec.page, spec.Hkv, spec.D), spec.seed, STREAM_V, device)
    pt = shuffled_page_table(spec.B, spec.pages_per_seq, spec.seed, device)
    seqused = torch.full((spec.B,), spec.seqused, dtype=torch.int32, device=device)
    q2k = q2k_decode(spec.B, spec.Hkv, spec.Sq, seqused, spec.topk, spec.page, spec.seed, device)
    return {"q": q, "k_pool": k, "v_pool": v, "page_table": pt, "seqused": seqused, "q2k": q2k}


@dataclass
class VarlenSpec:
    """Ragged prefill batch: sequence b has q_lens[b] queries and k_lens[b] keys.

    Q [total_q,Hq,D], K/V [total_k,Hkv,D], q2k [Hkv,total_q,topk] with block ids
    local to each sequence; cu_seqlens_q / cu_seqlens_k are the prefix sums.
    """
    name: str
    q_lens: tuple
    k_lens: tuple
    Hkv: int
    qpk: int
    topk: int
    causal: bool
    pattern: str            # "perm_prefix" | "sink" | "uniform"
    D: int = 128
    blk: int = BLK
    seed: int = DEFAULT_SEED

    @property
    def B(self) -> int:
        return len(self.q_lens)

    @property
    def Hq(self) -> int:
        return self.Hkv * self.qpk

    @property
    def total_q(self) -> int:
        return int(sum(self.q_lens))

    @property
    def total_k(self) -> int:
        return int(sum(self.k_lens))


def make_varlen_inputs(spec: VarlenSpec, device="cpu") -> dict:
    """Q, K, V (bf16), q2k [Hkv,total_q,topk] and cu_seqlens_q/k (int32).

    Each sequence's selections follow the pattern of a batch-1 prefill of its
    own lengths (seed + 7919 * b, so sequences differ)."""
    q = normal_bf16((spec.total_q, spec.Hq, spec.D), spec.seed, STREAM_Q, device)
    k = normal_bf16((spec.total_k, spec.Hkv, spec.D), spec.seed, STREAM_K, device)
    v = normal_bf16((spec.total_k, spec.Hkv, spec.D), spec.seed, STREAM_V, device)
    parts = []
    for b, (sq, sk) in enumerate(zip(spec.q_lens, spec.k_lens)):
        ps = PrefillSpec(f"{spec.name}_{b}", B=1, Sq=int(sq), Skv=int(sk), Hkv=spec.Hkv, qpk=spec.qpk,
                         topk=spec.topk, causal=spec.causal, pattern=spec.pattern, D=spec.D, blk=spec.blk,
                         seed=spec.seed + 7919 * b)
        parts.append(make_prefill_q2k(ps, device)[0])          # [Hkv, sq, topk]
    q2k = torch.cat(parts, dim=1).contiguous()
    cu = lambda lens: torch.tensor([0] + list(itertools.accumulate(int(x) for x in lens)), dtype=torch.int32,
                                   device=device)
    return {"q": q, "k": k, "v": v, "q2k": q2k, "cu_seqlens_q": cu(spec.q_lens), "cu_seqlens_k": cu(spec.k_lens)}


def sample_query_rows(total_q: int, n: int, seed: int = DEFAULT_SEED, must=()) -> list:
    """Sorted sample of ``n`` distinct global query ids plus ``must`` (edges)."""
    idx = torch.arange(max(n, 1), dtype=torch.int64)
    picks = uniform_below(counter_u32(seed, STREAM_AUX, idx), torch.full_like(idx, total_q))
    out = set(int(x) for x in picks.tolist()[:n])
    out.update(int(m) for m in must if 0 <= m < total_q)
    return sorted(out)
