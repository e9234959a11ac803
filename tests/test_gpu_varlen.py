"""GPU ragged batches (msa_build_k2q_csr_varlen + msa_sparse_attn_fwd_varlen) vs the float64 oracle.

The CSR is bit-exact against the oracle's varlen CSR, the plan covers every
(row, query) once, the attention output is compared element by element with
the oracle's varlen attention, and a ragged batch whose sequences all have the
same lengths gives the uniform entry points' output bit for bit.
"""

import numpy as np
import pytest
import torch

import msa_synth as synth
import oracle
from parity import assert_attn_close
from test_gpu_csr import _check_plan

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def V(name, q_lens, k_lens, **kw):
    base = dict(Hkv=2, qpk=16, topk=8, causal=True, pattern="sink")
    base.update(kw)
    return synth.VarlenSpec(name, q_lens=tuple(q_lens), k_lens=tuple(k_lens), **base)


SPECS = [
    V("ragged_sink_qpk16", (700, 1, 129, 300), (1024, 256, 1000, 300)),
    V("ragged_uniform_qpk8", (1500, 64, 257), (2048, 4096, 640), qpk=8, topk=16, pattern="uniform"),
    V("ragged_qpk2_topk4", (900, 33), (1024, 900), qpk=2, topk=4, Hkv=3),
    V("ragged_qpk1_topk32", (600, 1200), (4096, 1280), qpk=1, topk=32, Hkv=1),
    V("ragged_q_longer_than_kv", (700, 50), (256, 1024), qpk=4, topk=4),
    V("ragged_noncausal", (100, 300, 7), (512, 1024, 640), qpk=4, topk=4, causal=False, pattern="perm_prefix"),
]


def _row_off(spec):
    out = [0]
    for kl in spec.k_lens:
        out.append(out[-1] + -(-kl // 128))
    return out


def _run(spec, x, kv_format="bf16", k=None, v=None, k_scales=None, v_scales=None, status=None):
    import block_sparse_top_gb300 as msa
    own = status is None
    if own:
        status = msa.new_status(DEV)
    csr = msa.build_k2q_csr_varlen(x["q2k"], x["cu_seqlens_q"], x["cu_seqlens_k"], max(spec.q_lens),
                                   max(spec.k_lens), spec.qpk, status=status)
    res = msa.sparse_attn_fwd_varlen(x["q"], x["k"] if k is None else k, x["v"] if v is None else v, csr,
                                     causal=spec.causal, kv_format=kv_format, k_scales=k_scales, v_scales=v_scales,
                                     status=status)
    torch.cuda.synchronize()
    if own:
        st = msa.read_status(status)
        assert st & msa.MSA_STATUS_FATAL_MASK == 0, f"fatal device status {st:#x}"
    return csr, res


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_varlen_csr_bit_exact_and_plan_covers_every_pair(spec):
    x = synth.make_varlen_inputs(spec, device=DEV)
    import block_sparse_top_gb300 as msa
    csr = msa.build_k2q_csr_varlen(x["q2k"], x["cu_seqlens_q"], x["cu_seqlens_k"], max(spec.q_lens),
                                   max(spec.k_lens), spec.qpk)
    ref = oracle.build_k2q_csr_varlen(x["q2k"].cpu(), x["cu_seqlens_q"].cpu(), x["cu_seqlens_k"].cpu())
    for key in ("row_ptr", "q_indices", "qsplit", "split_counts"):
        assert np.array_equal(getattr(csr, key).cpu().numpy(), ref[key]), key
    _check_plan(csr, _row_off(spec))


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_varlen_attention_matches_oracle(spec):
    x = synth.make_varlen_inputs(spec, device=DEV)
    _, (o, lse) = _run(spec, x)
    o_ref, l_ref = oracle.sparse_attn_varlen(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["q2k"].cpu(),
                                             x["cu_seqlens_q"].cpu(), x["cu_seqlens_k"].cpu(), causal=spec.causal)
    assert_attn_close(o, lse, o_ref, l_ref, spec.name)


def test_varlen_nvfp4_matches_oracle_and_dequantised_bf16_exactly():
    import block_sparse_top_gb300 as msa
    spec = V("ragged_nvfp4", (500, 130, 64), (1024, 300, 2048), qpk=2, topk=8)
    x = synth.make_varlen_inputs(spec, device=DEV)
    kp, ks = msa.nvfp4_quantize(x["k"])
    vp, vs = msa.nvfp4_quantize(x["v"])
    _, (o4, l4) = _run(spec, x, kv_format="nvfp4", k=kp, v=vp, k_scales=ks, v_scales=vs)
    kq, kqs = oracle.nvfp4_quantize(x["k"].cpu())
    vq, vqs = oracle.nvfp4_quantize(x["v"].cpu())
    kd = torch.from_numpy(oracle.nvfp4_dequantize(kq, kqs).view(np.int16)).view(torch.bfloat16)
    vd = torch.from_numpy(oracle.nvfp4_dequantize(vq, vqs).view(np.int16)).view(torch.bfloat16)
    o_ref, l_ref = oracle.sparse_attn_varlen(x["q"].cpu(), kd, vd, x["q2k"].cpu(), x["cu_seqlens_q"].cpu(),
                                             x["cu_seqlens_k"].cpu(), causal=True)
    assert_attn_close(o4, l4, o_ref, l_ref, spec.name)
    _, (ob, lb) = _run(spec, x, k=kd.to(DEV), v=vd.to(DEV))
    assert torch.equal(o4, ob) and torch.equal(l4, lb)


def test_equal_lengths_give_the_uniform_result_bit_for_bit():
    """Three sequences of 1000 queries / 2048 keys as a ragged batch equal the
    uniform B=3 call: same CSR, same plan, same kernels."""
    import block_sparse_top_gb300 as msa
    B, Sq, Skv, Hkv, qpk, topk = 3, 1000, 2048, 2, 16, 16
    spec = synth.PrefillSpec("u3", B=B, Sq=Sq, Skv=Skv, Hkv=Hkv, qpk=qpk, topk=topk, causal=True, pattern="sink")
    x = synth.make_prefill_inputs(spec, device=DEV)
    csr = msa.build_k2q_csr(x["q2k"], Skv, qpk)
    o_u, l_u = msa.sparse_attn_fwd(x["q"], x["k"], x["v"], csr, causal=True)
    q2k_v = x["q2k"].permute(1, 0, 2, 3).reshape(Hkv, B * Sq, topk).contiguous()
    cu_q = torch.arange(0, B * Sq + 1, Sq, dtype=torch.int32, device=DEV)
    cu_k = torch.arange(0, B * Skv + 1, Skv, dtype=torch.int32, device=DEV)
    csr_v = msa.build_k2q_csr_varlen(q2k_v, cu_q, cu_k, Sq, Skv, qpk)
    o_v, l_v = msa.sparse_attn_fwd_varlen(x["q"].view(B * Sq, spec.Hq, 128), x["k"].view(B * Skv, Hkv, 128),
                                          x["v"].view(B * Skv, Hkv, 128), csr_v, causal=True)
    torch.cuda.synchronize()
    for key in ("row_ptr", "q_indices", "qsplit", "split_counts"):
        assert torch.equal(getattr(csr, key), getattr(csr_v, key)), key
    assert torch.equal(o_u.view(B * Sq, spec.Hq, 128), o_v) and torch.equal(l_u.view(B * Sq, spec.Hq), l_v)


def test_mid_size_ragged_batch_sampled():
    spec = V("ragged_mid", (9000, 2500, 16384, 1), (9000, 12288, 16384, 128), Hkv=2, qpk=16, topk=16)
    x = synth.make_varlen_inputs(spec, device=DEV)
    _, (o, lse) = _run(spec, x)
    cq = [0, 9000, 11500, 27884, 27885]
    rows = synth.sample_query_rows(spec.total_q, 48, must=[0, 127, 128, 8999, 9000, 11499, 11500, 27883, 27884])
    o_ref, l_ref = oracle.sparse_attn_varlen(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["q2k"].cpu(),
                                             x["cu_seqlens_q"].cpu(), x["cu_seqlens_k"].cpu(), causal=True, rows=rows)
    assert cq[-1] == spec.total_q
    assert_attn_close(o[rows], lse[rows], o_ref, l_ref, spec.name)


def test_inconsistent_cu_seqlens_drop_the_sequence_and_set_the_shape_bit():
    """Sequences whose query range runs backwards, or exceeds the declared
    maximum, are dropped with MSA_STATUS_SHAPE; queries that no kept sequence
    holds get O = 0, LSE = -inf; the kept sequence is exact."""
    import block_sparse_top_gb300 as msa
    spec = V("bad_cu", (300, 200, 100), (512, 512, 512), qpk=4, topk=4)
    x = synth.make_varlen_inputs(spec, device=DEV)
    # sequence 1 runs 300 -> 250 (backwards); sequence 2 then holds 350 > 300 queries
    bad_q = torch.tensor([0, 300, 250, 600], dtype=torch.int32, device=DEV)
    status = msa.new_status(DEV)
    csr = msa.build_k2q_csr_varlen(x["q2k"], bad_q, x["cu_seqlens_k"], 300, 512, spec.qpk, status=status)
    o, lse = msa.sparse_attn_fwd_varlen(x["q"], x["k"], x["v"], csr, causal=True, status=status)
    st = msa.read_status(status)
    assert st & msa.MSA_STATUS_SHAPE
    o_ref, l_ref = oracle.sparse_attn_varlen(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["q2k"].cpu(),
                                             x["cu_seqlens_q"].cpu(), x["cu_seqlens_k"].cpu(), causal=True,
                                             rows=list(range(300)))
    assert_attn_close(o[:300], lse[:300], o_ref, l_ref, "bad_cu sequence 0")
    assert torch.isneginf(lse[300:]).all() and (o[300:] == 0).all()


# --------------------------------------------------------------------------- temperature LSE, partial dtypes

TEMP_SPEC = V("ragged_temp", (700, 129, 300), (1024, 1000, 2048), qpk=16, topk=8)


@pytest.mark.parametrize("T", [0.5, 2.0])
@pytest.mark.parametrize("kv_format", ["bf16", "nvfp4"])
def test_temperature_lse_matches_oracle(T, kv_format):
    import block_sparse_top_gb300 as msa
    spec = TEMP_SPEC
    x = synth.make_varlen_inputs(spec, device=DEV)
    k, v, kw = x["k"], x["v"], {}
    if kv_format == "nvfp4":
        k, ks = msa.nvfp4_quantize(x["k"])
        v, vs = msa.nvfp4_quantize(x["v"])
        kw = {"kv_format": "nvfp4", "k_scales": ks, "v_scales": vs}
        kd = torch.from_numpy(oracle.nvfp4_dequantize(*oracle.nvfp4_quantize(x["k"].cpu())).view(np.int16))
        vd = torch.from_numpy(oracle.nvfp4_dequantize(*oracle.nvfp4_quantize(x["v"].cpu())).view(np.int16))
        k_ref, v_ref = kd.view(torch.bfloat16), vd.view(torch.bfloat16)
    else:
        k_ref, v_ref = x["k"].cpu(), x["v"].cpu()
    status = msa.new_status(DEV)
    csr = msa.build_k2q_csr_varlen(x["q2k"], x["cu_seqlens_q"], x["cu_seqlens_k"], max(spec.q_lens),
                                   max(spec.k_lens), spec.qpk, status=status)
    o, lse, lt = msa.sparse_attn_fwd_varlen(x["q"], k, v, csr, causal=True, lse_temperature_scale=T, status=status,
                                            **kw)
    assert msa.read_status(status) & msa.MSA_STATUS_FATAL_MASK == 0
    o_ref, l_ref, t_ref = oracle.sparse_attn_varlen(x["q"].cpu(), k_ref, v_ref, x["q2k"].cpu(),
                                                    x["cu_seqlens_q"].cpu(), x["cu_seqlens_k"].cpu(), causal=True,
                                                    temperature=T)
    assert_attn_close(o, lse, o_ref, l_ref, f"temp {T} {kv_format}")
    # the temperature LSE, same bar as the LSE
    assert_attn_close(o, lt, o_ref, t_ref, f"temperature lse {T} {kv_format}")
    # the forward without the temperature output is unchanged by it
    o2, l2 = msa.sparse_attn_fwd_varlen(x["q"], k, v, csr, causal=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("qpk,topk", [(16, 16), (4, 32), (2, 8)])
def test_partial_dtypes_match_oracle_and_fp32_is_at_least_as_close(qpk, topk):
    import block_sparse_top_gb300 as msa
    spec = V(f"ragged_part_{qpk}", (3000, 700, 1), (4096, 2048, 640), qpk=qpk, topk=topk, Hkv=2)
    x = synth.make_varlen_inputs(spec, device=DEV)
    csr = msa.build_k2q_csr_varlen(x["q2k"], x["cu_seqlens_q"], x["cu_seqlens_k"], max(spec.q_lens),
                                   max(spec.k_lens), spec.qpk)
    o_ref, l_ref = oracle.sparse_attn_varlen(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["q2k"].cpu(),
                                             x["cu_seqlens_q"].cpu(), x["cu_seqlens_k"].cpu(), causal=True)
    errs = {}
    for pd in (msa.MSA_PARTIAL_BF16, msa.MSA_PARTIAL_FP16, msa.MSA_PARTIAL_FP32):
        status = msa.new_status(DEV)
        o, lse = msa.sparse_attn_fwd_varlen(x["q"], x["k"], x["v"], csr, causal=True, partial_dtype=pd,
                                            status=status)
        assert msa.read_status(status) & msa.MSA_STATUS_FATAL_MASK == 0
        errs[pd] = assert_attn_close(o, lse, o_ref, l_ref, f"partial dtype {pd}")
    # fp32 partials drop the partials' rounding: never less accurate on average
    assert errs[msa.MSA_PARTIAL_FP32][1] <= errs[msa.MSA_PARTIAL_BF16][1]


def test_peaked_softmax_with_large_scores():
    """A softmax scale of 8 spreads the scores over hundreds of units, so a
    row's softmax is nearly one-hot; P of the row max is exactly 1 and the
    output still matches the oracle."""
    import block_sparse_top_gb300 as msa
    spec = V("ragged_big_scores", (600, 300), (1024, 2048), qpk=8, topk=8)
    x = synth.make_varlen_inputs(spec, device=DEV)
    csr = msa.build_k2q_csr_varlen(x["q2k"], x["cu_seqlens_q"], x["cu_seqlens_k"], max(spec.q_lens),
                                   max(spec.k_lens), spec.qpk)
    o, lse = msa.sparse_attn_fwd_varlen(x["q"], x["k"], x["v"], csr, causal=True, softmax_scale=8.0)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.sparse_attn_varlen(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["q2k"].cpu(),
                                             x["cu_seqlens_q"].cpu(), x["cu_seqlens_k"].cpu(), causal=True,
                                             scale=8.0)
    assert_attn_close(o, lse, o_ref, l_ref, "large scores")
