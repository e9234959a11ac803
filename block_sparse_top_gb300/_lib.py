"""ctypes loader for libmsa.so (the C ABI declared in include/msa.h).

There is no fallback: if the library is missing the import of the binding
fails with an error naming the build step.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmsa.so")

MSA_OK = 0
MSA_ERR_INVALID_ARG = -1
MSA_ERR_UNSUPPORTED = -2
MSA_ERR_WORKSPACE = -3
MSA_ERR_CUDA = -4
MSA_ERR_DEVICE = -5

MSA_STATUS_INDEX_RANGE = 0x1
MSA_STATUS_DUPLICATE = 0x2
MSA_STATUS_PAGE_RANGE = 0x4
MSA_STATUS_PLAN_OVERFLOW = 0x8
MSA_STATUS_TIMEOUT = 0x10
MSA_STATUS_LAUNCH = 0x20
MSA_STATUS_SHAPE = 0x40
MSA_STATUS_FATAL_MASK = (MSA_STATUS_PAGE_RANGE | MSA_STATUS_PLAN_OVERFLOW | MSA_STATUS_TIMEOUT | MSA_STATUS_LAUNCH
                         | MSA_STATUS_SHAPE)

MSA_KV_BF16 = 0
MSA_KV_NVFP4 = 1
MSA_KV_FP8 = 2

MSA_PARTIAL_BF16 = 0
MSA_PARTIAL_FP16 = 1
MSA_PARTIAL_FP32 = 2


class FwdOptions(ctypes.Structure):
    """msa_fwd_options (include/msa.h)."""
    _fields_ = [("partial_dtype", ctypes.c_int), ("lse_temperature_scale", ctypes.c_float),
                ("lse_temperature", ctypes.c_void_p), ("qk_fp8", ctypes.c_int)]


class MsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {_status_string(code)} ({code})")


_lib = None


def _status_string(code: int) -> str:
    try:
        return lib().msa_status_string(code).decode()
    except Exception:  # pragma: no cover - only when the library itself is broken
        return "status"


def lib():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m block_sparse_top_gb300.build` "
                           "(or __graft_entry__.build()); there is no CPU fallback")
    _lib = load(LIB_PATH)
    return _lib


def load(path: str):
    """Opens a build of the library at `path` with the C signatures of include/msa.h."""
    L = ctypes.CDLL(path)
    P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    L.msa_status_string.argtypes = [I]
    L.msa_status_string.restype = ctypes.c_char_p
    L.msa_version.restype = I
    L.msa_check_status.argtypes = [P]
    L.msa_check_status.restype = I
    L.msa_read_status.argtypes = [P, P, P]
    L.msa_read_status.restype = I
    L.msa_k2q_csr_workspace_size.argtypes = [I, I, I, I, I, I]
    L.msa_k2q_csr_workspace_size.restype = SZ
    L.msa_plan_size.argtypes = [I, I, I, I, I, I, I]
    L.msa_plan_size.restype = SZ
    L.msa_build_k2q_csr.argtypes = [P, I, I, I, I, I, I, I, P, P, P, P, P, P, SZ, P, SZ, P, P]
    L.msa_build_k2q_csr.restype = I
    L.msa_sparse_attn_fwd_workspace_size.argtypes = [I, I, I, I, I]
    L.msa_sparse_attn_fwd_workspace_size.restype = SZ
    L.msa_sparse_attn_fwd.argtypes = [P, P, P, I, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, P, P, SZ,
                                      P, P]
    L.msa_sparse_attn_fwd.restype = I
    L.msa_sparse_attn_fwd_partial.argtypes = [P, P, P, I, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, SZ, P, P]
    L.msa_sparse_attn_fwd_partial.restype = I
    L.msa_sparse_attn_combine.argtypes = [P, I, I, I, I, I, I, P, P, P, SZ, P]
    L.msa_sparse_attn_combine.restype = I
    L.msa_sparse_attn_paged_fwd_workspace_size.argtypes = [I, I, I, I, I, I, I]
    L.msa_sparse_attn_paged_fwd_workspace_size.restype = SZ
    L.msa_sparse_attn_paged_fwd_launches.argtypes = [I, I, I, I, I, I, I]
    L.msa_sparse_attn_paged_fwd_launches.restype = I
    L.msa_sparse_attn_paged_fwd.argtypes = [P, P, P, I, P, I, P, P, I, I, I, I, I, I, I, I, F, P, P, P, SZ, P, P]
    L.msa_sparse_attn_paged_fwd.restype = I
    L.msa_k2q_csr_varlen_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
    L.msa_k2q_csr_varlen_workspace_size.restype = SZ
    L.msa_plan_varlen_size.argtypes = [I, I, I, I, I, I]
    L.msa_plan_varlen_size.restype = SZ
    L.msa_build_k2q_csr_varlen.argtypes = [P, P, P, I, I, I, I, I, I, I, I, I, P, P, P, P, P, P, SZ, P, SZ, P, P]
    L.msa_build_k2q_csr_varlen.restype = I
    L.msa_sparse_attn_fwd_varlen_workspace_size.argtypes = [I, I, I, I, P]
    L.msa_sparse_attn_fwd_varlen_workspace_size.restype = SZ
    L.msa_sparse_attn_fwd_varlen.argtypes = [P, P, P, I, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P,
                                             P, P, P, SZ, P, P]
    L.msa_sparse_attn_fwd_varlen.restype = I
    L.msa_paged_attn_fwd_workspace_size.argtypes = [I, I, I, I, I, I, I]
    L.msa_paged_attn_fwd_workspace_size.restype = SZ
    L.msa_paged_attn_fwd.argtypes = [P, P, P, I, I, P, I, P, P, I, I, I, I, I, I, I, I, F, P, P, P, SZ, P, P]
    L.msa_paged_attn_fwd.restype = I
    L.msa_nvfp4_quantize.argtypes = [P, I64, I, P, P, P]
    L.msa_nvfp4_quantize.restype = I
    return L


def check(code: int, where: str) -> None:
    if code != MSA_OK:
        raise MsaError(code, where)
