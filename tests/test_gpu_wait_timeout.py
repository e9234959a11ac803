"""Bounded waits: every wait in the kernels gives up after a time limit, raises
MSA_STATUS_TIMEOUT, drains its copies and MMAs and exits, leaving the context
usable.

A test build of the library (never the product) is compiled with a 2 ms wait
limit and with CTA 0 never signalling its first unit's K/V block: a flag that
nothing sets.  The forward through that build must return with the timeout bit
in the status word (msa_check_status: MSA_ERR_DEVICE), and the product
library's next call on the same context must be correct.
"""

import ctypes
import os

import pytest
import torch

import msa_synth as synth
import oracle
from parity import assert_attn_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _wait_test_lib():
    from block_sparse_top_gb300 import _lib, build
    d = os.path.join(build.ROOT, "_build", "waittest")
    path = build.build(defines=("MSA_TEST_WAIT_LIMIT_NS=2000000ull", "MSA_TEST_DROP_KV_ARRIVAL"),
                       lib_path=os.path.join(d, "libmsa_waittest.so"), build_dir=d)
    return _lib.load(path)


def test_dropped_arrival_times_out_and_the_context_stays_usable():
    import block_sparse_top_gb300 as msa
    spec = synth.PrefillSpec("wait", B=1, Sq=1000, Skv=2048, Hkv=2, qpk=16, topk=8, causal=True, pattern="sink")
    x = synth.make_prefill_inputs(spec, device=DEV)
    csr = msa.build_k2q_csr(x["q2k"], spec.Skv, spec.qpk)
    ws = msa.fwd_workspace(spec.B, spec.Sq, spec.Hq, spec.topk, DEV)
    o = torch.zeros_like(x["q"])
    lse = torch.zeros((spec.B, spec.Sq, spec.Hq), dtype=torch.float32, device=DEV)
    status = msa.new_status(DEV)
    WL = _wait_test_lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = WL.msa_sparse_attn_fwd(p(x["q"]), p(x["k"]), p(x["v"]), msa.MSA_KV_BF16, None, None, p(csr.row_ptr),
                                p(csr.q_indices), p(csr.qsplit), p(csr.split_counts), p(csr.plan), spec.B, spec.Sq,
                                spec.Skv, spec.Hq, spec.Hkv, 128, 128, spec.topk, 1, -1.0, p(o), p(lse), p(ws),
                                ws.numel(), p(status), stream)
    assert rc == 0
    torch.cuda.synchronize()  # returns: the kernel gave up instead of hanging
    word = int(status.item()) & 0xFFFFFFFF
    assert word & msa.MSA_STATUS_TIMEOUT
    assert msa.check_status(word) == -5  # MSA_ERR_DEVICE
    # the context is intact: the product library's call is right
    status2 = msa.new_status(DEV)
    o2, l2 = msa.sparse_attn_fwd(x["q"], x["k"], x["v"], csr, causal=True, status=status2)
    assert msa.read_status(status2) & msa.MSA_STATUS_FATAL_MASK == 0
    rows = synth.sample_query_rows(spec.Sq, 32, must=[0, 127, 999])
    o_ref, l_ref = oracle.sparse_attn(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["q2k"].cpu(), causal=True,
                                      rows=rows)
    assert_attn_close(o2.view(-1, spec.Hq, 128)[rows], l2.view(-1, spec.Hq)[rows], o_ref, l_ref, "after timeout")
