"""The paged decode entry point that allocates nothing (msa_sparse_attn_paged_fwd_noalloc).

It serves callers that cannot allocate device memory when they run a decode
step; its scratch is a static device array inside the library.  This test
calls it through the C ABI twice in a row and checks each result against the
allocating entry point (msa_sparse_attn_paged_fwd with a caller workspace),
within the parity tolerances, and each result against the float64 oracle.
The file sorts last so that a stop-at-first-failure run has already run
every other test.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import msa_synth as synth
import oracle
from parity import assert_attn_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_REL = 1e-3


def _call_noalloc(L, d, spec, o, lse, status):
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn = L.msa_sparse_attn_paged_fwd_noalloc
    fn.argtypes = [P, P, P, I, P, I, P, P, I, I, I, I, I, I, I, I, F, P, P, P, P]
    fn.restype = I
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(p(d["q"]), p(d["k_pool"]), p(d["v_pool"]), spec.num_pages, p(d["page_table"]), spec.pages_per_seq,
              p(d["seqused"]), p(d["q2k"]), spec.B, spec.Sq, spec.Hq, spec.Hkv, 128, 128, spec.topk, 1, -1.0,
              p(o), p(lse), p(status), stream)


def _close(a_o, a_l, b_o, b_l):
    err = (a_o.float() - b_o.float()).abs()
    assert err.max().item() <= O_MAX_ABS and err.mean().item() <= O_MEAN_ABS
    assert torch.equal(torch.isneginf(a_l), torch.isneginf(b_l))
    fin = torch.isfinite(b_l)
    rel = ((a_l[fin] - b_l[fin]).abs() / b_l[fin].abs().clamp_min(1e-6)).max().item()
    assert rel <= LSE_REL


@pytest.mark.parametrize("L_kv", [4096, 32768])
def test_noalloc_decode_matches_allocating_entry_point_twice(L_kv):
    import block_sparse_top_gb300 as msa
    L = msa.lib()
    spec = synth.paged_decode_spec(L_kv)
    d = synth.make_decode_inputs(spec, device=DEV)
    ref_o, ref_l = msa.sparse_attn_paged_fwd(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seqused"],
                                             d["q2k"])
    rows = synth.sample_query_rows(spec.B * spec.Sq, 24, must=[0, 7, 255])
    o_ref, l_ref = oracle.sparse_attn_paged(d["q"].cpu(), d["k_pool"].cpu(), d["v_pool"].cpu(),
                                            d["page_table"].cpu(), d["seqused"].cpu(), d["q2k"].cpu(), rows=rows)
    for _ in range(2):
        o = torch.full_like(d["q"], float("nan"))
        lse = torch.full(d["q"].shape[:2], float("nan"), dtype=torch.float32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = _call_noalloc(L, d, spec, o, lse, status)
        assert rc == 0, L.msa_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) & 0x1C == 0
        _close(o, lse, ref_o, ref_l)
        assert_attn_close(o[rows], lse[rows], o_ref, l_ref, f"noalloc L={L_kv}")


def union_scratch_bytes(B, Sq, Hkv, qpk, topk, max_pages, sms):
    """The no-alloc decode's scratch for a shape, as its header states it."""
    up = lambda x: (x + 255) // 256 * 256
    n = min(Sq, 128 // qpk)
    G = B * Hkv * math.ceil(Sq / (128 // qpk))
    U = min(n * topk, max_pages)
    wq = math.ceil((128 // qpk) / 32)
    return (up(4 * G * U) + up(4 * G * U * wq) + up(4 * (G + 1)) + up(4 * G) + up(4 * sms * 2 * 128)
            + up(4 * sms * 2 * 128 * 128))


def test_noalloc_decode_rejects_shapes_beyond_its_scratch():
    import block_sparse_top_gb300 as msa
    L = msa.lib()
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    # 16384 sequences x 4 KV heads at 64K tokens need about twice the 32 MiB static scratch
    spec = synth.DecodeSpec("too_big", B=16384, Sq=8, Hkv=4, qpk=16, topk=16, kv_len=65536, trim=0)
    need = union_scratch_bytes(spec.B, spec.Sq, spec.Hkv, spec.qpk, spec.topk, spec.pages_per_seq, sms)
    assert need > 2 * (32 << 20)
    # the shapes the parity test above uses fit
    for L_kv in (4096, 32768):
        sp = synth.paged_decode_spec(L_kv)
        assert union_scratch_bytes(sp.B, sp.Sq, sp.Hkv, sp.qpk, sp.topk, sp.pages_per_seq, sms) <= (32 << 20)
    t = torch.zeros(16, dtype=torch.bfloat16, device=DEV)
    d = {"q": t, "k_pool": t, "v_pool": t, "page_table": t, "seqused": t, "q2k": t}
    rc = _call_noalloc(L, d, spec, t, t, t)
    assert rc == -3   # MSA_ERR_WORKSPACE, returned before any launch
