"""Python binding of libmsa (GB300 block-sparse top-k GQA attention).

Each function marshals torch CUDA tensors into the matching C-ABI call of
include/msa.h; every step of the computation runs in the library's kernels.
PyTorch provides device memory and the current stream only.
"""

from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass
from typing import Optional

import torch

from ._lib import (MSA_KV_BF16, MSA_KV_FP8, MSA_KV_NVFP4, MSA_PARTIAL_BF16, MSA_PARTIAL_FP16, MSA_PARTIAL_FP32,  # noqa: F401
                   MSA_STATUS_DUPLICATE, MSA_STATUS_FATAL_MASK, MSA_STATUS_INDEX_RANGE, MSA_STATUS_LAUNCH,
                   MSA_STATUS_PAGE_RANGE, MSA_STATUS_PLAN_OVERFLOW, MSA_STATUS_SHAPE, MSA_STATUS_TIMEOUT, FwdOptions,
                   MsaError, check, lib)

BLK = 128


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ws(nbytes: int, device) -> torch.Tensor:
    # 256-byte aligned by the caching allocator (blocks are 512-byte aligned)
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of {dtype}")


_FP8 = getattr(torch, "float8_e4m3fn", None)


def _kv_format(kv_format: str, k, v, k_scales, v_scales) -> int:
    """Checks the K/V tensors of a format name and returns its MSA_KV_* code."""
    if kv_format == "bf16":
        _need(k, torch.bfloat16, "k")
        _need(v, torch.bfloat16, "v")
        return MSA_KV_BF16
    if kv_format == "fp8":
        for t, n in ((k, "k"), (v, "v")):
            if not (t.is_cuda and t.is_contiguous() and t.dtype in (torch.uint8, _FP8)):
                raise ValueError(f"{n} must be a contiguous CUDA tensor of e4m3 bytes (float8_e4m3fn or uint8)")
        return MSA_KV_FP8
    if kv_format == "nvfp4":
        for t, n in ((k, "k"), (v, "v"), (k_scales, "k_scales"), (v_scales, "v_scales")):
            _need(t, torch.uint8, n)
        return MSA_KV_NVFP4
    raise ValueError(f"unknown kv_format {kv_format!r}")


@dataclass
class K2qCsr:
    """Output of msa_build_k2q_csr plus the work plan of the prefill kernel."""
    row_ptr: torch.Tensor       # [Hkv, B*nblk+1] int32
    q_indices: torch.Tensor     # [Hkv, B*Sq*topk] int32
    qsplit: torch.Tensor        # [Hkv, B*Sq*topk] int32
    split_counts: torch.Tensor  # [B*Sq, Hkv] int32
    plan: torch.Tensor          # opaque uint8 buffer
    B: int
    Hkv: int
    Sq: int
    Skv: int
    topk: int
    qhead_per_kv: int


def csr_buffers(B: int, Hkv: int, Sq: int, Skv: int, topk: int, qhead_per_kv: int, device) -> tuple:
    """Allocates (K2qCsr, workspace) for msa_build_k2q_csr."""
    L = lib()
    nblk = math.ceil(Skv / BLK)
    cap = B * Sq * topk
    plan_bytes = L.msa_plan_size(B, Hkv, Sq, Skv, topk, BLK, qhead_per_kv)
    ws_bytes = L.msa_k2q_csr_workspace_size(B, Hkv, Sq, Skv, topk, BLK)
    if plan_bytes == 0 or ws_bytes == 0:
        raise ValueError("unsupported CSR shape")
    csr = K2qCsr(
        row_ptr=torch.empty((Hkv, B * nblk + 1), dtype=torch.int32, device=device),
        q_indices=torch.empty((Hkv, cap), dtype=torch.int32, device=device),
        qsplit=torch.empty((Hkv, cap), dtype=torch.int32, device=device),
        split_counts=torch.empty((B * Sq, Hkv), dtype=torch.int32, device=device),
        plan=torch.empty(plan_bytes, dtype=torch.uint8, device=device),
        B=B, Hkv=Hkv, Sq=Sq, Skv=Skv, topk=topk, qhead_per_kv=qhead_per_kv)
    return csr, _ws(ws_bytes, device)


def build_k2q_csr(q2k: torch.Tensor, Skv: int, qhead_per_kv: int, seqused: Optional[torch.Tensor] = None,
                  out: Optional[K2qCsr] = None, workspace: Optional[torch.Tensor] = None,
                  status: Optional[torch.Tensor] = None, stream=None) -> K2qCsr:
    """msa_build_k2q_csr: q2k [B,Hkv,Sq,topk] int32 -> K2qCsr (plan included)."""
    _need(q2k, torch.int32, "q2k")
    B, Hkv, Sq, topk = q2k.shape
    if out is None or workspace is None:
        out, workspace = csr_buffers(B, Hkv, Sq, Skv, topk, qhead_per_kv, q2k.device)
    if seqused is not None:
        _need(seqused, torch.int32, "seqused")
    rc = lib().msa_build_k2q_csr(_p(q2k), B, Hkv, Sq, Skv, topk, BLK, qhead_per_kv, _p(seqused), _p(out.row_ptr),
                                 _p(out.q_indices), _p(out.qsplit), _p(out.split_counts), _p(out.plan),
                                 out.plan.numel(), _p(workspace), workspace.numel(), _p(status), _stream(stream))
    check(rc, "msa_build_k2q_csr")
    return out


@dataclass
class K2qCsrVarlen:
    """Output of msa_build_k2q_csr_varlen plus the work plan (ragged batch)."""
    row_ptr: torch.Tensor       # [Hkv, total_rows+1] int32
    q_indices: torch.Tensor     # [Hkv, total_q*topk] int32
    qsplit: torch.Tensor        # [Hkv, total_q*topk] int32
    split_counts: torch.Tensor  # [total_q, Hkv] int32
    plan: torch.Tensor          # opaque uint8 buffer
    cu_seqlens_q: torch.Tensor  # [B+1] int32
    cu_seqlens_k: torch.Tensor  # [B+1] int32
    B: int
    Hkv: int
    total_q: int
    topk: int
    qhead_per_kv: int


def build_k2q_csr_varlen(q2k: torch.Tensor, cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                         max_seqlen_q: int, max_seqlen_k: int, qhead_per_kv: int, total_rows: Optional[int] = None,
                         seqused: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                         stream=None) -> K2qCsrVarlen:
    """msa_build_k2q_csr_varlen: q2k [Hkv,total_q,topk] int32 + cu_seqlens -> K2qCsrVarlen.

    ``total_rows`` (the row capacity) defaults to sum_b ceil(keys_b / 128), read
    from cu_seqlens_k on the host."""
    _need(q2k, torch.int32, "q2k")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    Hkv, total_q, topk = q2k.shape
    B = cu_seqlens_q.numel() - 1
    if total_rows is None:
        lens = cu_seqlens_k.cpu().diff()
        total_rows = int(((lens + BLK - 1) // BLK).sum())
    total_rows = max(1, int(total_rows))
    L = lib()
    plan_bytes = L.msa_plan_varlen_size(Hkv, total_q, total_rows, topk, BLK, qhead_per_kv)
    ws_bytes = L.msa_k2q_csr_varlen_workspace_size(B, Hkv, total_q, max_seqlen_q, max_seqlen_k, total_rows, topk, BLK)
    if plan_bytes == 0 or ws_bytes == 0:
        raise ValueError("unsupported varlen CSR shape")
    dev = q2k.device
    out = K2qCsrVarlen(
        row_ptr=torch.empty((Hkv, total_rows + 1), dtype=torch.int32, device=dev),
        q_indices=torch.empty((Hkv, total_q * topk), dtype=torch.int32, device=dev),
        qsplit=torch.empty((Hkv, total_q * topk), dtype=torch.int32, device=dev),
        split_counts=torch.empty((total_q, Hkv), dtype=torch.int32, device=dev),
        plan=torch.empty(plan_bytes, dtype=torch.uint8, device=dev),
        cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k, B=B, Hkv=Hkv, total_q=total_q, topk=topk,
        qhead_per_kv=qhead_per_kv)
    ws = _ws(ws_bytes, dev)
    if seqused is not None:
        _need(seqused, torch.int32, "seqused")
    rc = L.msa_build_k2q_csr_varlen(_p(q2k), _p(cu_seqlens_q), _p(cu_seqlens_k), B, Hkv, total_q, max_seqlen_q,
                                    max_seqlen_k, total_rows, topk, BLK, qhead_per_kv, _p(seqused), _p(out.row_ptr),
                                    _p(out.q_indices), _p(out.qsplit), _p(out.split_counts), _p(out.plan),
                                    out.plan.numel(), _p(ws), ws.numel(), _p(status), _stream(stream))
    check(rc, "msa_build_k2q_csr_varlen")
    out._workspace = ws  # kept alive until the stream has used it
    return out


def _opts(partial_dtype: int, lse_temperature_scale: float, lse_temperature: Optional[torch.Tensor],
          qk_fp8: bool = False):
    o = FwdOptions()
    o.partial_dtype = int(partial_dtype)
    o.lse_temperature_scale = float(lse_temperature_scale)
    o.lse_temperature = None if lse_temperature is None else lse_temperature.data_ptr()
    o.qk_fp8 = int(bool(qk_fp8))
    return o


def sparse_attn_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, csr: K2qCsrVarlen, *, causal: bool,
                           softmax_scale: Optional[float] = None, kv_format: str = "bf16",
                           k_scales: Optional[torch.Tensor] = None, v_scales: Optional[torch.Tensor] = None,
                           partial_dtype: int = MSA_PARTIAL_BF16, lse_temperature_scale: Optional[float] = None,
                           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                           stream=None):
    """msa_sparse_attn_fwd_varlen: q [total_q,Hq,D], k/v [total_k,Hkv,D] -> (O, LSE[, temperature LSE]).

    q of e4m3 bytes (float8_e4m3fn or uint8) with kv_format "fp8" runs S = Q K^T as an fp8 MMA."""
    qk_fp8 = q.dtype in (torch.uint8, _FP8)
    if qk_fp8:
        if not (q.is_cuda and q.is_contiguous()) or kv_format != "fp8":
            raise ValueError("e4m3 q needs a contiguous CUDA tensor and kv_format 'fp8'")
    else:
        _need(q, torch.bfloat16, "q")
    total_q, Hq, D = q.shape
    fmt = _kv_format(kv_format, k, v, k_scales, v_scales)
    total_k, Hkv = k.shape[0], k.shape[1]
    if out is None:
        out = torch.empty((total_q, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    lse_t = None
    if lse_temperature_scale is not None:
        lse_t = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    opts = _opts(partial_dtype, 1.0 if lse_temperature_scale is None else lse_temperature_scale, lse_t, qk_fp8)
    L = lib()
    if workspace is None:
        n = L.msa_sparse_attn_fwd_varlen_workspace_size(total_q, Hq, csr.topk, D, ctypes.byref(opts))
        if n == 0:
            raise ValueError("unsupported varlen forward shape or options")
        workspace = _ws(n, q.device)
    scale = -1.0 if softmax_scale is None else float(softmax_scale)
    rc = L.msa_sparse_attn_fwd_varlen(_p(q), _p(k), _p(v), fmt, _p(k_scales), _p(v_scales), _p(csr.q_indices),
                                      _p(csr.qsplit), _p(csr.split_counts), _p(csr.plan), _p(csr.cu_seqlens_q),
                                      _p(csr.cu_seqlens_k), csr.B, total_q, total_k, Hq, Hkv, D, BLK, csr.topk,
                                      int(bool(causal)), scale, ctypes.byref(opts), _p(out), _p(lse),
                                      _p(workspace), workspace.numel(), _p(status), _stream(stream))
    check(rc, "msa_sparse_attn_fwd_varlen")
    return (out, lse) if lse_t is None else (out, lse, lse_t)


def fwd_workspace(B: int, Sq: int, Hq: int, topk: int, device) -> torch.Tensor:
    n = lib().msa_sparse_attn_fwd_workspace_size(B, Sq, Hq, topk, 128)
    if n == 0:
        raise ValueError("unsupported forward shape")
    return _ws(n, device)


def sparse_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, csr: K2qCsr, *, causal: bool,
                    softmax_scale: Optional[float] = None, kv_format: str = "bf16",
                    k_scales: Optional[torch.Tensor] = None, v_scales: Optional[torch.Tensor] = None,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    return_lse: bool = True, workspace: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None, stream=None):
    """msa_sparse_attn_fwd: q [B,Sq,Hq,D], k/v [B,Skv,Hkv,D] (or NVFP4 packed) -> (O, LSE)."""
    _need(q, torch.bfloat16, "q")
    B, Sq, Hq, D = q.shape
    fmt = _kv_format(kv_format, k, v, k_scales, v_scales)
    Skv, Hkv = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = fwd_workspace(B, Sq, Hq, csr.topk, q.device)
    scale = -1.0 if softmax_scale is None else float(softmax_scale)
    rc = lib().msa_sparse_attn_fwd(_p(q), _p(k), _p(v), fmt, _p(k_scales), _p(v_scales), _p(csr.row_ptr),
                                   _p(csr.q_indices), _p(csr.qsplit), _p(csr.split_counts), _p(csr.plan), B, Sq,
                                   Skv, Hq, Hkv, D, BLK, csr.topk, int(bool(causal)), scale, _p(out), _p(lse),
                                   _p(workspace), workspace.numel(), _p(status), _stream(stream))
    check(rc, "msa_sparse_attn_fwd")
    return out, lse


def sparse_attn_fwd_partial(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, csr: K2qCsr, *, causal: bool,
                            workspace: torch.Tensor, softmax_scale: Optional[float] = None, kv_format: str = "bf16",
                            k_scales: Optional[torch.Tensor] = None, v_scales: Optional[torch.Tensor] = None,
                            status: Optional[torch.Tensor] = None, stream=None) -> None:
    """msa_sparse_attn_fwd_partial: the attention tiles only (split partials into ``workspace``)."""
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    fmt = _kv_format(kv_format, k, v, k_scales, v_scales)
    scale = -1.0 if softmax_scale is None else float(softmax_scale)
    rc = lib().msa_sparse_attn_fwd_partial(_p(q), _p(k), _p(v), fmt, _p(k_scales), _p(v_scales), _p(csr.q_indices),
                                           _p(csr.qsplit), _p(csr.plan), B, Sq, Skv, Hq, Hkv, D, BLK, csr.topk,
                                           int(bool(causal)), scale, _p(workspace), workspace.numel(), _p(status),
                                           _stream(stream))
    check(rc, "msa_sparse_attn_fwd_partial")


def sparse_attn_combine(csr: K2qCsr, Hq: int, out: torch.Tensor, lse: Optional[torch.Tensor],
                        workspace: torch.Tensor, stream=None) -> None:
    """msa_sparse_attn_combine: LSE combine of the partials in ``workspace`` into ``out`` / ``lse``."""
    rc = lib().msa_sparse_attn_combine(_p(csr.split_counts), csr.B, csr.Sq, Hq, csr.Hkv, 128, csr.topk, _p(out),
                                       _p(lse), _p(workspace), workspace.numel(), _stream(stream))
    check(rc, "msa_sparse_attn_combine")


def paged_workspace(B: int, Sq: int, Hq: int, Hkv: int, topk: int, max_pages: int, device) -> torch.Tensor:
    n = lib().msa_sparse_attn_paged_fwd_workspace_size(B, Sq, Hq, Hkv, 128, topk, max_pages)
    if n == 0:
        raise ValueError("unsupported decode shape")
    return _ws(n, device)


def paged_fwd_launches(B: int, Sq: int, Hq: int, Hkv: int, topk: int, max_pages: int) -> int:
    """msa_sparse_attn_paged_fwd_launches: kernels one decode call of this shape
    launches on the current device (1 or 2; topk = 0 for the dense mode)."""
    n = lib().msa_sparse_attn_paged_fwd_launches(B, Sq, Hq, Hkv, 128, topk, max_pages)
    if n < 0:
        raise MsaError(n, "msa_sparse_attn_paged_fwd_launches")
    return n


def sparse_attn_paged_fwd(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, page_table: torch.Tensor,
                          seqused: torch.Tensor, q2k: torch.Tensor, *, causal: bool = True,
                          softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                          lse: Optional[torch.Tensor] = None, return_lse: bool = True,
                          workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                          stream=None):
    """msa_sparse_attn_paged_fwd: q [B*Sq,Hq,D], pools [num_pages,page,Hkv,D] -> (O, LSE)."""
    _need(q, torch.bfloat16, "q")
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(v_pool, torch.bfloat16, "v_pool")
    _need(page_table, torch.int32, "page_table")
    _need(seqused, torch.int32, "seqused")
    _need(q2k, torch.int32, "q2k")
    total_q, Hq, D = q.shape
    num_pages, page, Hkv, _ = k_pool.shape
    B, max_pages = page_table.shape
    Sq = total_q // B
    topk = q2k.shape[-1]
    if out is None:
        out = torch.empty((total_q, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = paged_workspace(B, Sq, Hq, Hkv, topk, max_pages, q.device)
    scale = -1.0 if softmax_scale is None else float(softmax_scale)
    rc = lib().msa_sparse_attn_paged_fwd(_p(q), _p(k_pool), _p(v_pool), num_pages, _p(page_table), max_pages,
                                         _p(seqused), _p(q2k), B, Sq, Hq, Hkv, D, page, topk, int(bool(causal)),
                                         scale, _p(out), _p(lse), _p(workspace), workspace.numel(), _p(status),
                                         _stream(stream))
    check(rc, "msa_sparse_attn_paged_fwd")
    return out, lse


def paged_attn_fwd(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, page_table: torch.Tensor,
                   seqused: torch.Tensor, q2k: Optional[torch.Tensor] = None, *, kv_format: str = "bf16",
                   causal: bool = True, softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None, stream=None):
    """msa_paged_attn_fwd: paged decode over bf16 or e4m3 pools [num_pages,page,Hkv,D]; q2k None is the
    dense mode (every block of each sequence)."""
    _need(q, torch.bfloat16, "q")
    _need(page_table, torch.int32, "page_table")
    _need(seqused, torch.int32, "seqused")
    fmt = _kv_format(kv_format, k_pool, v_pool, None, None)
    total_q, Hq, D = q.shape
    num_pages, page, Hkv, _ = k_pool.shape
    B, max_pages = page_table.shape
    Sq = total_q // B
    topk = 0
    if q2k is not None:
        _need(q2k, torch.int32, "q2k")
        topk = q2k.shape[-1]
    if out is None:
        out = torch.empty((total_q, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    L = lib()
    if workspace is None:
        n = L.msa_paged_attn_fwd_workspace_size(B, Sq, Hq, Hkv, D, topk, max_pages)
        if n == 0:
            raise ValueError("unsupported paged decode shape")
        workspace = _ws(n, q.device)
    scale = -1.0 if softmax_scale is None else float(softmax_scale)
    rc = L.msa_paged_attn_fwd(_p(q), _p(k_pool), _p(v_pool), fmt, num_pages, _p(page_table), max_pages, _p(seqused),
                              _p(q2k), B, Sq, Hq, Hkv, D, page, topk, int(bool(causal)), scale, _p(out), _p(lse),
                              _p(workspace), workspace.numel(), _p(status), _stream(stream))
    check(rc, "msa_paged_attn_fwd")
    return out, lse


def nvfp4_quantize(x: torch.Tensor, stream=None):
    """msa_nvfp4_quantize: bf16 [..., D] -> (packed uint8 [..., D/2], e4m3 scales uint8 [..., D/16])."""
    _need(x, torch.bfloat16, "x")
    D = x.shape[-1]
    rows = x.numel() // D
    packed = torch.empty(x.shape[:-1] + (D // 2,), dtype=torch.uint8, device=x.device)
    scales = torch.empty(x.shape[:-1] + (D // 16,), dtype=torch.uint8, device=x.device)
    rc = lib().msa_nvfp4_quantize(_p(x), rows, D, _p(packed), _p(scales), _stream(stream))
    check(rc, "msa_nvfp4_quantize")
    return packed, scales


def new_status(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_status(word: int) -> int:
    """msa_check_status on a status word already read back to the host: 0 (MSA_OK) or -5 (MSA_ERR_DEVICE)."""
    w = ctypes.c_uint32(int(word) & 0xFFFFFFFF)
    return int(lib().msa_check_status(ctypes.cast(ctypes.pointer(w), ctypes.c_void_p)))


def read_status(status: torch.Tensor, stream=None) -> int:
    """msa_read_status: synchronises the stream and returns the status bits."""
    host = ctypes.c_uint32(0)
    rc = lib().msa_read_status(_p(status), ctypes.cast(ctypes.pointer(host), ctypes.c_void_p), _stream(stream))
    if rc not in (0, -5):
        check(rc, "msa_read_status")
    return int(host.value)
