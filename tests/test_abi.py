"""CPU checks of the C-ABI library: it loads, exports every symbol msa.h declares,
answers size queries and rejects bad arguments before touching the device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


@pytest.fixture(scope="module")
def L():
    from block_sparse_top_gb300 import build
    build.build()
    from block_sparse_top_gb300 import _lib
    return _lib.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_\w+)\s*\(", src)))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for n in ("msa_build_k2q_csr", "msa_sparse_attn_fwd", "msa_sparse_attn_paged_fwd"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    assert L.msa_version() == 101
    for code in (0, -1, -2, -3, -4, -5):
        assert L.msa_status_string(code).startswith(b"MSA_")


def test_check_status_reads_a_host_word_without_cuda(L):
    """msa_check_status classifies a status word the caller already holds on the host."""
    from block_sparse_top_gb300 import _lib
    cases = {0: 0, _lib.MSA_STATUS_INDEX_RANGE: 0, _lib.MSA_STATUS_DUPLICATE: 0,
             _lib.MSA_STATUS_INDEX_RANGE | _lib.MSA_STATUS_DUPLICATE: 0,
             _lib.MSA_STATUS_PAGE_RANGE: -5, _lib.MSA_STATUS_PLAN_OVERFLOW: -5, _lib.MSA_STATUS_TIMEOUT: -5,
             _lib.MSA_STATUS_LAUNCH: -5, _lib.MSA_STATUS_DUPLICATE | _lib.MSA_STATUS_TIMEOUT: -5}
    for word, want in cases.items():
        w = ctypes.c_uint32(word)
        assert L.msa_check_status(ctypes.cast(ctypes.pointer(w), ctypes.c_void_p)) == want, hex(word)
    assert L.msa_check_status(None) == -1


def test_size_queries(L):
    # 32K causal workload: plan holds at least one unit per row plus nnz / 64
    assert L.msa_plan_size(1, 4, 32768, 32768, 16, 128, 16) > 64
    assert L.msa_plan_size(1, 4, 32768, 32768, 16, 128, 3) == 0          # qhead_per_kv 3 unsupported
    assert L.msa_k2q_csr_workspace_size(1, 4, 32768, 32768, 16, 64) == 0  # blk_kv 64 unsupported
    ws = L.msa_sparse_attn_fwd_workspace_size(1, 1024, 2, 4, 128)
    assert ws >= 1024 * 4 * 2 * (256 + 4)
    assert L.msa_sparse_attn_fwd_workspace_size(1, 1024, 2, 4, 64) == 0
    assert L.msa_sparse_attn_paged_fwd_workspace_size(32, 8, 64, 4, 128, 16, 1024) > 0


def test_decode_size_queries(L):
    # sparse and dense (topk 0) paged decode; the dense plan holds every block
    sparse = L.msa_paged_attn_fwd_workspace_size(32, 8, 64, 4, 128, 16, 1024)
    dense = L.msa_paged_attn_fwd_workspace_size(32, 8, 64, 4, 128, 0, 1024)
    assert sparse == L.msa_sparse_attn_paged_fwd_workspace_size(32, 8, 64, 4, 128, 16, 1024)
    assert dense > sparse > 0
    # the sparse entry point has no dense mode; unsupported shapes give 0
    assert L.msa_sparse_attn_paged_fwd_workspace_size(32, 8, 64, 4, 128, 0, 1024) == 0
    assert L.msa_paged_attn_fwd_workspace_size(32, 8, 64, 4, 128, 5, 1024) == 0       # topk 5
    assert L.msa_paged_attn_fwd_workspace_size(32, 8, 48, 4, 128, 16, 1024) == 0      # qhead_per_kv 12
    assert L.msa_paged_attn_fwd_workspace_size(32, 8, 64, 4, 128, 16, 8193) == 0      # max_pages past 8192
    # groups: B * Hkv * ceil(Sq / (128 / qpk)) at most 49152
    assert L.msa_paged_attn_fwd_workspace_size(12288, 1, 64, 4, 128, 16, 8) > 0       # 49152 groups
    assert L.msa_paged_attn_fwd_workspace_size(12289, 1, 64, 4, 128, 16, 8) == 0      # one more


def test_decode_launch_count_query(L):
    # 1K keys (8 pages, unions of at most 8 blocks) and 128 groups: one launch
    # on any device with at least 128 SMs; 4K keys (unions up to 32): two
    assert L.msa_sparse_attn_paged_fwd_launches(32, 8, 64, 4, 128, 16, 8) == 1
    assert L.msa_sparse_attn_paged_fwd_launches(32, 8, 64, 4, 128, 16, 16) == 1     # 2K: unions of <= 16
    assert L.msa_sparse_attn_paged_fwd_launches(32, 8, 64, 4, 128, 16, 32) == 2
    assert L.msa_sparse_attn_paged_fwd_launches(32, 8, 64, 4, 128, 0, 8) == 1       # dense mode, 8 pages
    assert L.msa_sparse_attn_paged_fwd_launches(4096, 8, 64, 4, 128, 16, 8) == 2    # more groups than SMs
    # shapes the decode calls reject give their error codes
    assert L.msa_sparse_attn_paged_fwd_launches(32, 8, 64, 4, 128, 5, 8) == -2      # topk 5: unsupported
    assert L.msa_sparse_attn_paged_fwd_launches(32, 8, 63, 4, 128, 16, 8) == -1     # Hq % Hkv
    assert L.msa_sparse_attn_paged_fwd_launches(32, 8, 64, 4, 128, -1, 8) == -1


def test_bad_arguments_are_rejected_before_launch(L):
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    null = None
    # null pointers
    assert L.msa_build_k2q_csr(null, 1, 1, 8, 128, 4, 128, 2, null, null, null, null, null, null, 0, null, 0,
                               null, null) == -1
    # unsupported topk (5) and head dim (64)
    args = [fake] * 5
    assert L.msa_build_k2q_csr(fake, 1, 1, 8, 128, 5, 128, 2, null, *args[:4], null, 0, fake, 1 << 20, null,
                               null) == -2
    rc = L.msa_sparse_attn_fwd(fake, fake, fake, 0, null, null, fake, fake, fake, fake, fake, 1, 8, 128, 2, 1, 64,
                               128, 4, 0, 0.0, fake, null, fake, 1 << 30, null, null)
    assert rc == -2
    # workspace too small
    rc = L.msa_sparse_attn_fwd(fake, fake, fake, 0, null, null, fake, fake, fake, fake, fake, 1, 8, 128, 2, 1, 128,
                               128, 4, 0, 0.0, fake, null, fake, 16, null, null)
    assert rc == -3
    rc = L.msa_sparse_attn_paged_fwd(fake, fake, fake, 8, fake, 4, fake, fake, 2, 8, 64, 4, 128, 64, 16, 1, 0.0,
                                     fake, null, fake, 1 << 30, null, null)
    assert rc == -2   # page size 64
    # general paged decode: kv_format must be bf16 or e4m3; a q2k with topk 0 is invalid
    rc = L.msa_paged_attn_fwd(fake, fake, fake, 1, 8, fake, 4, fake, fake, 2, 8, 64, 4, 128, 128, 16, 1, 0.0,
                              fake, null, fake, 1 << 30, null, null)
    assert rc == -1   # MSA_KV_NVFP4 pools are not a decode format
    rc = L.msa_paged_attn_fwd(fake, fake, fake, 0, 8, fake, 4, fake, fake, 2, 8, 64, 4, 128, 128, 0, 1, 0.0,
                              fake, null, fake, 1 << 30, null, null)
    assert rc == -1
    # dense mode (q2k NULL), workspace too small
    rc = L.msa_paged_attn_fwd(fake, fake, fake, 0, 8, fake, 4, fake, null, 2, 8, 64, 4, 128, 128, 0, 1, 0.0,
                              fake, null, fake, 16, null, null)
    assert rc == -3
    assert L.msa_nvfp4_quantize(fake, 4, 100, fake, fake, null) == -1   # D % 16 != 0


def test_binding_fails_loudly_without_the_library(monkeypatch):
    from block_sparse_top_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", os.path.join(ROOT, "does-not-exist.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.lib()


def test_generator_is_deterministic_on_cpu():
    import torch
    import msa_synth as s
    a = s.normal_bf16((64, 128), 42, s.STREAM_Q)
    b = s.normal_bf16((64, 128), 42, s.STREAM_Q)
    c = s.normal_bf16((64, 128), 43, s.STREAM_Q)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))
    q = s.q2k_causal_sink(1, 2, 300, 1024, 16)
    assert torch.equal(q, s.q2k_causal_sink(1, 2, 300, 1024, 16))
