"""Float64 CPU oracle for block-sparse top-k GQA attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg use this package.  It loads ``liboracle.so`` (built from ``oracle.c`` by
``oracle.build``) through ctypes and shares nothing with the CUDA library.
Every function states the passage it follows in ``oracle.c``.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        path = _build.library_path()
        if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_build.source_path()):
            _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        I64 = ctypes.c_int64
        D = ctypes.c_double
        L.oracle_sparse_attn.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, I, D, P, P, I64, P, P, I]
        L.oracle_sparse_attn.restype = I
        L.oracle_sparse_attn_paged.argtypes = [P, P, P, P, I, P, P, I, I, I, I, I, I, I, I, D, P, I64, P, P, I]
        L.oracle_sparse_attn_paged.restype = I
        L.oracle_build_k2q_csr.argtypes = [P, I, I, I, I, I, I, P, P, P, P, P]
        L.oracle_build_k2q_csr.restype = I
        L.oracle_sparse_attn_varlen.argtypes = [P, P, P, P, P, P, P, I, P, I, I, I, I, I, I, I, D, D, P, I64, P,
                                                P, P, I]
        L.oracle_sparse_attn_varlen.restype = I
        L.oracle_build_k2q_csr_varlen.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P]
        L.oracle_build_k2q_csr_varlen.restype = I
        L.oracle_nvfp4_quantize.argtypes = [P, I64, I, P, P]
        L.oracle_nvfp4_dequantize.argtypes = [P, P, I64, I, P]
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_double.restype = D
        L.oracle_e4m3_from_double_rne_sat.argtypes = [D]
        L.oracle_e4m3_from_double_rne_sat.restype = ctypes.c_uint8
        L.oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_to_double.restype = D
        L.oracle_e2m1_from_double_rne_sat.argtypes = [D]
        L.oracle_e2m1_from_double_rne_sat.restype = ctypes.c_uint8
        L.oracle_default_threads.restype = I
        _LIB = L
    return _LIB


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 numpy array of bf16 bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x.astype(np.int32, copy=False))
    return np.ascontiguousarray(x.detach().cpu().contiguous().numpy().astype(np.int32, copy=False))


def default_threads() -> int:
    return int(lib().oracle_default_threads())


def sparse_attn(q, k, v, q2k, *, causal: bool, scale: Optional[float] = None, blk: int = 128,
                seqused=None, rows: Optional[Sequence[int]] = None, nthreads: int = 0,
                return_threads: bool = False):
    """Dense-KV oracle (oracle.c ``oracle_sparse_attn``).

    q [B,Sq,Hq,D], k/v [B,Skv,Hkv,D] bf16; q2k [B,Hkv,Sq,topk] int32.
    Returns (O [n,Hq,D] float64, LSE [n,Hq] float64) for the queries ``rows``
    (global ids b*Sq+s) or for all B*Sq queries.
    """
    B, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    topk = q2k.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    sel = _i32(q2k)
    su = None if seqused is None else _i32(seqused)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = B * Sq if r is None else r.size
    o = np.zeros((n, Hq, D), dtype=np.float64)
    lse = np.zeros((n, Hq), dtype=np.float64)
    th = lib().oracle_sparse_attn(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(sel), B, Sq, Skv, Hq, Hkv, D, blk, topk,
                                  int(bool(causal)), float(scale), _ptr(su), _ptr(r), n, _ptr(o), _ptr(lse),
                                  int(nthreads))
    return (o, lse, th) if return_threads else (o, lse)


def sparse_attn_paged(q, k_pool, v_pool, page_table, seqused, q2k, *, causal: bool = True,
                      scale: Optional[float] = None, rows: Optional[Sequence[int]] = None,
                      nthreads: int = 0, return_threads: bool = False):
    """Paged-KV oracle (oracle.c ``oracle_sparse_attn_paged``).

    q [B*Sq,Hq,D]; pools [num_pages,page,Hkv,D]; page_table [B,max_pages];
    seqused [B]; q2k [B,Hkv,Sq,topk].  Returns (O [n,Hq,D], LSE [n,Hq]).
    """
    total_q, Hq, D = q.shape
    num_pages, page, Hkv, _ = k_pool.shape
    B, max_pages = page_table.shape
    Sq = total_q // B
    topk = q2k.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k_pool), _bf16_bits(v_pool)
    pt, su, sel = _i32(page_table), _i32(seqused), _i32(q2k)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = total_q if r is None else r.size
    o = np.zeros((n, Hq, D), dtype=np.float64)
    lse = np.zeros((n, Hq), dtype=np.float64)
    th = lib().oracle_sparse_attn_paged(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pt), max_pages, _ptr(su), _ptr(sel),
                                        B, Sq, Hq, Hkv, D, page, topk, int(bool(causal)), float(scale),
                                        _ptr(r), n, _ptr(o), _ptr(lse), int(nthreads))
    return (o, lse, th) if return_threads else (o, lse)


def sparse_attn_varlen(q, k, v, q2k, cu_seqlens_q, cu_seqlens_k=None, *, causal: bool,
                       scale: Optional[float] = None, temperature: Optional[float] = None, blk: int = 128,
                       page_table=None, seqused=None, rows: Optional[Sequence[int]] = None, nthreads: int = 0):
    """Varlen / paged / every-block oracle (oracle.c ``oracle_sparse_attn_varlen``).

    q [total_q,Hq,D]; dense k/v [total_k,Hkv,D] with cu_seqlens_k, or pools
    [num_pages,blk,Hkv,D] with page_table [B,max_pages]; q2k [Hkv,total_q,topk]
    (sequence-local ids) or None for every block.  Returns (O [n,Hq,D],
    LSE [n,Hq]) and, when ``temperature`` is given, the temperature LSE [n,Hq].
    """
    total_q, Hq, D = q.shape
    Hkv = k.shape[-2]
    cq = _i32(cu_seqlens_q)
    B = cq.size - 1
    ck = None if cu_seqlens_k is None else _i32(cu_seqlens_k)
    pt = None if page_table is None else _i32(page_table)
    max_pages = 0 if pt is None else pt.shape[1]
    if pt is None and ck is None:
        raise ValueError("dense K/V needs cu_seqlens_k")
    topk = 0 if q2k is None else q2k.shape[-1]
    sel = None if q2k is None else _i32(q2k)
    su = None if seqused is None else _i32(seqused)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = total_q if r is None else r.size
    o = np.zeros((n, Hq, D), dtype=np.float64)
    lse = np.zeros((n, Hq), dtype=np.float64)
    lt = np.zeros((n, Hq), dtype=np.float64) if temperature is not None else None
    lib().oracle_sparse_attn_varlen(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(sel), _ptr(cq), _ptr(ck), _ptr(pt),
                                    max_pages, _ptr(su), B, Hq, Hkv, D, blk, topk, int(bool(causal)), float(scale),
                                    float(temperature) if temperature is not None else 0.0, _ptr(r), n, _ptr(o),
                                    _ptr(lse), _ptr(lt), int(nthreads))
    return (o, lse) if lt is None else (o, lse, lt)


def build_k2q_csr_varlen(q2k, cu_seqlens_q, cu_seqlens_k, blk: int = 128, seqused=None):
    """Varlen k->q CSR oracle (oracle.c ``oracle_build_k2q_csr_varlen``).

    q2k [Hkv,total_q,topk] (sequence-local ids).  Returns dict(row_ptr
    [Hkv,total_rows+1], q_indices, qsplit [Hkv,total_q*topk], split_counts
    [total_q,Hkv]); total_rows = sum of ceil(kv_len_b / blk).
    """
    Hkv, total_q, topk = q2k.shape
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    B = cq.size - 1
    rows = int(sum((int(ck[b + 1]) - int(ck[b]) + blk - 1) // blk for b in range(B)))
    cap = total_q * topk
    sel = _i32(q2k)
    su = None if seqused is None else _i32(seqused)
    row_ptr = np.zeros((Hkv, rows + 1), dtype=np.int32)
    qi = np.zeros((Hkv, cap), dtype=np.int32)
    qs = np.zeros((Hkv, cap), dtype=np.int32)
    sc = np.zeros((total_q, Hkv), dtype=np.int32)
    lib().oracle_build_k2q_csr_varlen(_ptr(sel), _ptr(cq), _ptr(ck), B, Hkv, topk, blk, _ptr(su), _ptr(row_ptr),
                                      _ptr(qi), _ptr(qs), _ptr(sc))
    return {"row_ptr": row_ptr, "q_indices": qi, "qsplit": qs, "split_counts": sc}


def build_k2q_csr(q2k, Skv: int, blk: int = 128, seqused=None):
    """k->q CSR oracle (oracle.c ``oracle_build_k2q_csr``).

    Returns dict(row_ptr [Hkv,B*nblk+1], q_indices [Hkv,B*Sq*topk],
    qsplit [Hkv,B*Sq*topk], split_counts [B*Sq,Hkv]), all int32.
    """
    B, Hkv, Sq, topk = q2k.shape
    nblk = (Skv + blk - 1) // blk
    rows = B * nblk
    cap = B * Sq * topk
    sel = _i32(q2k)
    su = None if seqused is None else _i32(seqused)
    row_ptr = np.zeros((Hkv, rows + 1), dtype=np.int32)
    qi = np.zeros((Hkv, cap), dtype=np.int32)
    qs = np.zeros((Hkv, cap), dtype=np.int32)
    sc = np.zeros((B * Sq, Hkv), dtype=np.int32)
    lib().oracle_build_k2q_csr(_ptr(sel), B, Hkv, Sq, Skv, topk, blk, _ptr(su), _ptr(row_ptr), _ptr(qi),
                               _ptr(qs), _ptr(sc))
    return {"row_ptr": row_ptr, "q_indices": qi, "qsplit": qs, "split_counts": sc}


def nvfp4_quantize(x):
    """bf16 [..., D] -> (packed uint8 [..., D/2], scales uint8 e4m3 [..., D/16])."""
    xb = _bf16_bits(x)
    shape = xb.shape
    D = shape[-1]
    rows = xb.size // D
    packed = np.zeros(shape[:-1] + (D // 2,), dtype=np.uint8)
    scales = np.zeros(shape[:-1] + (D // 16,), dtype=np.uint8)
    lib().oracle_nvfp4_quantize(_ptr(xb), rows, D, _ptr(packed), _ptr(scales))
    return packed, scales


def nvfp4_dequantize(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """(packed, scales) -> bf16 bits uint16 [..., D]."""
    packed = np.ascontiguousarray(packed)
    scales = np.ascontiguousarray(scales)
    D = packed.shape[-1] * 2
    rows = packed.size // (D // 2)
    out = np.zeros(packed.shape[:-1] + (D,), dtype=np.uint16)
    lib().oracle_nvfp4_dequantize(_ptr(packed), _ptr(scales), rows, D, _ptr(out))
    return out


def e4m3_decode(b: int) -> float:
    return float(lib().oracle_e4m3_to_double(b))


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_e4m3_from_double_rne_sat(x))


def e2m1_decode(c: int) -> float:
    return float(lib().oracle_e2m1_to_double(c))


def e2m1_encode(x: float) -> int:
    return int(lib().oracle_e2m1_from_double_rne_sat(x))


def bf16_bits_to_float64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
