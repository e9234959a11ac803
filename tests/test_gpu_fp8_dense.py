"""GPU e4m3 (FP8) K/V staged to bf16 and the dense paged decode mode vs the float64 oracle.

FP8 K/V: the oracle runs on the e4m3 values decoded exactly (the oracle's
e4m3 decode is pinned against torch.float8_e4m3fn on all 256 codes), and the
FP8 run equals the bf16 run on the decoded K/V bit for bit (staging is exact).
Dense decode (q2k = NULL): the oracle's every-block selection over the pool.
"""

import numpy as np
import pytest
import torch

import msa_synth as synth
import oracle
from parity import assert_attn_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _e4m3_lut() -> torch.Tensor:
    """bf16 bits of every e4m3 code, from the oracle's decode (exact in bf16)."""
    vals = np.array([oracle.e4m3_decode(b) if (b & 0x7F) != 0x7F else 0.0 for b in range(256)], dtype=np.float32)
    return torch.from_numpy((vals.view(np.uint32) >> 16).astype(np.int16))


def to_fp8(x: torch.Tensor):
    """(e4m3 bytes of x, the bf16 tensor those bytes decode to)."""
    b = x.float().to(torch.float8_e4m3fn).view(torch.uint8)
    dec = _e4m3_lut()[b.cpu().long()].view(torch.bfloat16)
    return b.contiguous(), dec


@pytest.mark.parametrize("spec", [
    synth.PrefillSpec("fp8_sink_qpk16", B=1, Sq=1500, Skv=2048, Hkv=2, qpk=16, topk=16, causal=True, pattern="sink"),
    synth.PrefillSpec("fp8_uniform_qpk2", B=2, Sq=1000, Skv=1100, Hkv=1, qpk=2, topk=8, causal=True,
                      pattern="uniform"),
], ids=lambda s: s.name)
def test_fp8_kv_prefill_matches_oracle_and_decoded_bf16_exactly(spec):
    import block_sparse_top_gb300 as msa
    x = synth.make_prefill_inputs(spec, device=DEV)
    k8, kd = to_fp8(x["k"])
    v8, vd = to_fp8(x["v"])
    csr = msa.build_k2q_csr(x["q2k"], spec.Skv, spec.qpk)
    o8, l8 = msa.sparse_attn_fwd(x["q"], k8, v8, csr, causal=True, kv_format="fp8")
    ob, lb = msa.sparse_attn_fwd(x["q"], kd.to(DEV), vd.to(DEV), csr, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o8, ob) and torch.equal(l8, lb)
    o_ref, l_ref = oracle.sparse_attn(x["q"].cpu(), kd, vd, x["q2k"].cpu(), causal=True)
    assert_attn_close(o8.view(-1, spec.Hq, 128), l8.view(-1, spec.Hq), o_ref, l_ref, spec.name)


def test_fp8_kv_varlen_with_temperature():
    import block_sparse_top_gb300 as msa
    spec = synth.VarlenSpec("fp8_ragged", q_lens=(600, 77), k_lens=(1024, 900), Hkv=2, qpk=8, topk=8, causal=True,
                            pattern="sink")
    x = synth.make_varlen_inputs(spec, device=DEV)
    k8, kd = to_fp8(x["k"])
    v8, vd = to_fp8(x["v"])
    csr = msa.build_k2q_csr_varlen(x["q2k"], x["cu_seqlens_q"], x["cu_seqlens_k"], 600, 1024, spec.qpk)
    o, lse, lt = msa.sparse_attn_fwd_varlen(x["q"], k8, v8, csr, causal=True, kv_format="fp8",
                                            lse_temperature_scale=1.5)
    torch.cuda.synchronize()
    o_ref, l_ref, t_ref = oracle.sparse_attn_varlen(x["q"].cpu(), kd, vd, x["q2k"].cpu(), x["cu_seqlens_q"].cpu(),
                                                    x["cu_seqlens_k"].cpu(), causal=True, temperature=1.5)
    assert_attn_close(o, lse, o_ref, l_ref, "fp8 ragged")
    assert_attn_close(o, lt, o_ref, t_ref, "fp8 ragged temperature lse")


@pytest.mark.parametrize("L", [2048, 32768])
def test_fp8_paged_decode_matches_oracle_and_decoded_bf16_exactly(L):
    import block_sparse_top_gb300 as msa
    spec = synth.paged_decode_spec(L)
    d = synth.make_decode_inputs(spec, device=DEV)
    k8, kd = to_fp8(d["k_pool"])
    v8, vd = to_fp8(d["v_pool"])
    status = msa.new_status(DEV)
    o8, l8 = msa.paged_attn_fwd(d["q"], k8, v8, d["page_table"], d["seqused"], d["q2k"], kv_format="fp8",
                                status=status)
    assert msa.read_status(status) & msa.MSA_STATUS_FATAL_MASK == 0
    ob, lb = msa.sparse_attn_paged_fwd(d["q"], kd.to(DEV), vd.to(DEV), d["page_table"], d["seqused"], d["q2k"])
    torch.cuda.synchronize()
    assert torch.equal(o8, ob) and torch.equal(l8, lb)
    rows = synth.sample_query_rows(spec.B * spec.Sq, 24, must=[0, 7, 255])
    o_ref, l_ref = oracle.sparse_attn_paged(d["q"].cpu(), kd, vd, d["page_table"].cpu(), d["seqused"].cpu(),
                                            d["q2k"].cpu(), rows=rows)
    assert_attn_close(o8[rows], l8[rows], o_ref, l_ref, f"fp8 decode {L}")


def D(name, **kw):
    base = dict(B=4, Sq=8, Hkv=2, qpk=16, topk=16, kv_len=2048, trim=17)
    base.update(kw)
    return synth.DecodeSpec(name, **base)


@pytest.mark.parametrize("spec", [
    synth.paged_decode_spec(1024),
    synth.paged_decode_spec(4096),
    D("dense_qpk4_sq3", qpk=4, Sq=3, kv_len=3000, trim=5),
    D("dense_qpk1", qpk=1, Sq=8, kv_len=1024, trim=100),
    D("dense_short", qpk=16, Sq=8, kv_len=128, trim=123),   # seqused 5 < Sq: early queries see nothing
    D("dense_qpk2_many_groups", qpk=2, Sq=150, kv_len=2048, trim=300),
    # one long sequence and one KV head: every CTA holds a piece of the one
    # group (512 blocks, 64 pieces merged by the CTA finishing last)
    D("dense_one_group_64k", B=1, Hkv=1, Sq=8, qpk=16, kv_len=65536, trim=17),
], ids=lambda s: s.name)
def test_dense_decode_matches_oracle(spec):
    import block_sparse_top_gb300 as msa
    d = synth.make_decode_inputs(spec, device=DEV)
    status = msa.new_status(DEV)
    o, lse = msa.paged_attn_fwd(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seqused"], None,
                                status=status)
    assert msa.read_status(status) & msa.MSA_STATUS_FATAL_MASK == 0
    B, Sq = spec.B, spec.Sq
    cu_q = torch.arange(0, B * Sq + 1, Sq, dtype=torch.int32)
    rows = None if B * Sq <= 64 else synth.sample_query_rows(B * Sq, 48, must=[0, Sq - 1, B * Sq - 1])
    o_ref, l_ref = oracle.sparse_attn_varlen(d["q"].cpu(), d["k_pool"].cpu(), d["v_pool"].cpu(), None, cu_q,
                                             causal=True, page_table=d["page_table"].cpu(),
                                             seqused=d["seqused"].cpu(), rows=rows)
    og, lg = (o, lse) if rows is None else (o[rows], lse[rows])
    assert_attn_close(og, lg, o_ref, l_ref, spec.name)


@pytest.mark.parametrize("qpk,topk", [(16, 16), (8, 8), (2, 16), (1, 4)])
def test_fp8_qk_bf16_pv_matches_oracle(qpk, topk):
    """e4m3 Q and K with S = Q K^T as an fp8 MMA, e4m3 V staged to bf16 for the
    bf16 P V: the oracle runs on the decoded e4m3 values (exact in bf16)."""
    import block_sparse_top_gb300 as msa
    spec = synth.VarlenSpec(f"qk8_{qpk}", q_lens=(700, 129, 40), k_lens=(1024, 2048, 512), Hkv=2, qpk=qpk, topk=topk,
                            causal=True, pattern="sink")
    x = synth.make_varlen_inputs(spec, device=DEV)
    q8, qd = to_fp8(x["q"])
    k8, kd = to_fp8(x["k"])
    v8, vd = to_fp8(x["v"])
    csr = msa.build_k2q_csr_varlen(x["q2k"], x["cu_seqlens_q"], x["cu_seqlens_k"], 700, 2048, spec.qpk)
    status = msa.new_status(DEV)
    o, lse, lt = msa.sparse_attn_fwd_varlen(q8.to(DEV), k8, v8, csr, causal=True, kv_format="fp8",
                                            lse_temperature_scale=0.75, status=status)
    assert msa.read_status(status) & msa.MSA_STATUS_FATAL_MASK == 0
    o_ref, l_ref, t_ref = oracle.sparse_attn_varlen(qd, kd, vd, x["q2k"].cpu(), x["cu_seqlens_q"].cpu(),
                                                    x["cu_seqlens_k"].cpu(), causal=True, temperature=0.75)
    assert_attn_close(o, lse, o_ref, l_ref, spec.name)
    assert_attn_close(o, lt, o_ref, t_ref, spec.name + " temperature lse")
