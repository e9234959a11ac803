"""GPU block-sparse prefill (msa_build_k2q_csr + msa_sparse_attn_fwd) vs the float64 oracle."""

import math

import numpy as np
import pytest
import torch

import msa_synth as synth
import oracle
from parity import assert_attn_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def run_gpu(x, spec, kv_format="bf16", k=None, v=None, k_scales=None, v_scales=None, status=None):
    import block_sparse_top_gb300 as msa
    own = status is None
    if own:
        status = msa.new_status(DEV)
    csr = msa.build_k2q_csr(x["q2k"], spec.Skv, spec.qpk, status=status)
    o, lse = msa.sparse_attn_fwd(x["q"], x["k"] if k is None else k, x["v"] if v is None else v, csr,
                                 causal=spec.causal, kv_format=kv_format, k_scales=k_scales, v_scales=v_scales,
                                 status=status)
    torch.cuda.synchronize()
    if own:
        st = msa.read_status(status)
        assert st & msa.MSA_STATUS_FATAL_MASK == 0, f"fatal device status {st:#x}"
    return o, lse


def check_spec(spec, rows=None, q2k=None):
    x = synth.make_prefill_inputs(spec, device=DEV)
    if q2k is not None:
        x["q2k"] = q2k.to(DEV)
    o, lse = run_gpu(x, spec)
    o_ref, l_ref = oracle.sparse_attn(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["q2k"].cpu(),
                                      causal=spec.causal, rows=rows)
    og = o.view(-1, spec.Hq, 128)
    lg = lse.view(-1, spec.Hq)
    if rows is not None:
        og, lg = og[rows], lg[rows]
    return assert_attn_close(og, lg, o_ref, l_ref, spec.name)


def P(name, **kw):
    base = dict(B=1, Sq=1000, Skv=1024, Hkv=2, qpk=16, topk=8, causal=True, pattern="sink")
    base.update(kw)
    return synth.PrefillSpec(name, **base)


SMALL = [
    synth.TINY_NONCAUSAL_1K,
    P("sink_qpk16_ragged", Sq=700, Skv=1024),
    P("sink_qpk8_topk16", qpk=8, topk=16, Sq=1500, Skv=2048),
    P("uniform_qpk4", qpk=4, pattern="uniform", Sq=2100, Skv=2048, topk=16),
    P("uniform_qpk2_topk32", qpk=2, pattern="uniform", Sq=4100, Skv=4096, topk=32, Hkv=1),
    P("sink_qpk1_topk4", qpk=1, topk=4, Sq=900, Skv=1024, Hkv=3),
    P("q_shorter_than_kv", Sq=300, Skv=2048, topk=16),
    P("q_longer_than_kv", Sq=1300, Skv=640, topk=4),
    P("kv_not_block_multiple", Sq=500, Skv=1000, topk=8),
    P("batch3_noncausal", B=3, Sq=200, Skv=512, causal=False, pattern="perm_prefix", topk=4, qpk=4),
]


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
def test_prefill_matches_oracle(spec):
    check_spec(spec)


def test_prefill_messy_indices_and_empty_queries():
    spec = P("messy", Sq=400, Skv=1024, topk=8, qpk=4, causal=False, pattern="perm_prefix")
    g = torch.Generator().manual_seed(3)
    q2k = torch.randint(-3, 10, (1, 2, 400, 8), generator=g, dtype=torch.int32)  # ids 8, 9 out of range
    q2k[0, :, 7] = -1            # query 7 selects nothing: O = 0, LSE = -inf
    q2k[0, 0, 9] = 3             # query 9 names block 3 eight times: counts once
    import block_sparse_top_gb300 as msa
    status = msa.new_status(DEV)
    x = synth.make_prefill_inputs(spec, device=DEV)
    x["q2k"] = q2k.to(DEV)
    o, lse = run_gpu(x, spec, status=status)
    st = msa.read_status(status)
    assert st & msa.MSA_STATUS_INDEX_RANGE and st & msa.MSA_STATUS_DUPLICATE
    o_ref, l_ref = oracle.sparse_attn(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), q2k, causal=False)
    assert_attn_close(o.view(-1, spec.Hq, 128), lse.view(-1, spec.Hq), o_ref, l_ref, "messy")
    assert torch.isneginf(lse[0, 7]).all() and (o[0, 7] == 0).all()


def test_prefill_custom_scale_and_repeat_calls_are_identical():
    import block_sparse_top_gb300 as msa
    spec = P("scale", Sq=512, Skv=1024)
    x = synth.make_prefill_inputs(spec, device=DEV)
    csr = msa.build_k2q_csr(x["q2k"], spec.Skv, spec.qpk)
    o1, l1 = msa.sparse_attn_fwd(x["q"], x["k"], x["v"], csr, causal=True, softmax_scale=0.05)
    o2, l2 = msa.sparse_attn_fwd(x["q"], x["k"], x["v"], csr, causal=True, softmax_scale=0.05)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o_ref, l_ref = oracle.sparse_attn(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["q2k"].cpu(), causal=True,
                                      scale=0.05)
    assert_attn_close(o1.view(-1, spec.Hq, 128), l1.view(-1, spec.Hq), o_ref, l_ref, "scale")


@pytest.mark.parametrize("spec", [P("split_sink", Sq=1500, Skv=2048, topk=16),
                                  P("split_qpk2", qpk=2, Hkv=3, Sq=2000, Skv=2048, topk=8, pattern="uniform")],
                         ids=lambda s: s.name)
def test_partial_then_combine_equals_fwd(spec):
    """msa_sparse_attn_fwd_partial then msa_sparse_attn_combine, called
    separately, give msa_sparse_attn_fwd's output bit for bit."""
    import block_sparse_top_gb300 as msa
    x = synth.make_prefill_inputs(spec, device=DEV)
    csr = msa.build_k2q_csr(x["q2k"], spec.Skv, spec.qpk)
    ws = msa.fwd_workspace(spec.B, spec.Sq, spec.Hq, spec.topk, DEV)
    o2 = torch.empty_like(x["q"])
    l2 = torch.empty((spec.B, spec.Sq, spec.Hq), dtype=torch.float32, device=DEV)
    msa.sparse_attn_fwd_partial(x["q"], x["k"], x["v"], csr, causal=True, workspace=ws)
    msa.sparse_attn_combine(csr, spec.Hq, o2, l2, ws)
    o1, l1 = msa.sparse_attn_fwd(x["q"], x["k"], x["v"], csr, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o_ref, l_ref = oracle.sparse_attn(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["q2k"].cpu(), causal=True)
    assert_attn_close(o2.view(-1, spec.Hq, 128), l2.view(-1, spec.Hq), o_ref, l_ref, spec.name)


MID = [
    # several waves, tens of units per CTA, many single-chunk units
    P("mid_sink_two_waves", Hkv=1, Sq=16384, Skv=16384, topk=16),
    P("mid_uniform_topk4", Hkv=2, Sq=12000, Skv=12288, topk=4, pattern="uniform"),
    P("mid_qpk2_sink", Hkv=1, qpk=2, Sq=70000, Skv=70016, topk=8),
]


@pytest.mark.parametrize("spec", MID, ids=lambda s: s.name)
def test_prefill_mid_size_sampled(spec):
    total = spec.B * spec.Sq
    rows = synth.sample_query_rows(total, 64, must=[0, 127, 128, 8191, 8192, total - 1])
    check_spec(spec, rows=rows)


FULL = [synth.CAUSAL_SINK_32K, synth.CAUSAL_UNIFORM_48K, synth.CAUSAL_SINK_384K]


@pytest.mark.parametrize("spec", FULL, ids=lambda s: s.name)
def test_prefill_full_size_sampled(spec):
    total = spec.B * spec.Sq
    edges = [0, 1, 15, 16, 127, 128, 129, 255, 2047, 2048, total // 2, total - 129, total - 128, total - 2, total - 1]
    rows = synth.sample_query_rows(total, 48, must=edges)
    check_spec(spec, rows=rows)


# --------------------------------------------------------------------------- NVFP4

def test_nvfp4_quantiser_bit_exact_vs_oracle():
    import block_sparse_top_gb300 as msa
    x = synth.normal_bf16((4096, 128), 9, synth.STREAM_AUX, device=DEV)
    x[0, :16] = 0
    x[1] *= 40.0
    x[2] *= 1e-3
    pk, sc = msa.nvfp4_quantize(x)
    torch.cuda.synchronize()
    pk_ref, sc_ref = oracle.nvfp4_quantize(x.cpu())
    assert np.array_equal(sc.cpu().numpy(), sc_ref)
    assert np.array_equal(pk.cpu().numpy(), pk_ref)


@pytest.mark.parametrize("spec", [P("nvfp4_qpk2", qpk=2, Hkv=1, Sq=3000, Skv=3072, topk=16),
                                  P("nvfp4_qpk16", Sq=700, Skv=1024)], ids=lambda s: s.name)
def test_nvfp4_kv_matches_oracle_and_dequantised_bf16_exactly(spec):
    import block_sparse_top_gb300 as msa
    x = synth.make_prefill_inputs(spec, device=DEV)
    kp, ks = msa.nvfp4_quantize(x["k"])
    vp, vs = msa.nvfp4_quantize(x["v"])
    o4, l4 = run_gpu(x, spec, kv_format="nvfp4", k=kp, v=vp, k_scales=ks, v_scales=vs)
    # oracle on its own quantisation, dequantised (bf16 exact)
    kq, kqs = oracle.nvfp4_quantize(x["k"].cpu())
    vq, vqs = oracle.nvfp4_quantize(x["v"].cpu())
    kd = torch.from_numpy(oracle.nvfp4_dequantize(kq, kqs).view(np.int16)).view(torch.bfloat16)
    vd = torch.from_numpy(oracle.nvfp4_dequantize(vq, vqs).view(np.int16)).view(torch.bfloat16)
    o_ref, l_ref = oracle.sparse_attn(x["q"].cpu(), kd, vd, x["q2k"].cpu(), causal=spec.causal)
    assert_attn_close(o4.view(-1, spec.Hq, 128), l4.view(-1, spec.Hq), o_ref, l_ref, spec.name)
    # dequantise-on-load is exact: the bf16 run on the dequantised K/V is bit-identical
    ob, lb = run_gpu(x, spec, k=kd.to(DEV), v=vd.to(DEV))
    assert torch.equal(o4, ob) and torch.equal(l4, lb)


def test_nvfp4_full_size_sampled():
    import block_sparse_top_gb300 as msa
    spec = synth.CAUSAL_SINK_384K_NVFP4
    x = synth.make_prefill_inputs(spec, device=DEV)
    kp, ks = msa.nvfp4_quantize(x["k"])
    vp, vs = msa.nvfp4_quantize(x["v"])
    o, lse = run_gpu(x, spec, kv_format="nvfp4", k=kp, v=vp, k_scales=ks, v_scales=vs)
    total = spec.Sq
    rows = synth.sample_query_rows(total, 32, must=[0, 128, total - 1])
    kq, kqs = oracle.nvfp4_quantize(x["k"].cpu())
    vq, vqs = oracle.nvfp4_quantize(x["v"].cpu())
    # the whole quantiser output, codes and scales of both K and V, is bit-exact
    assert np.array_equal(kp.cpu().numpy(), kq) and np.array_equal(ks.cpu().numpy(), kqs)
    assert np.array_equal(vp.cpu().numpy(), vq) and np.array_equal(vs.cpu().numpy(), vqs)
    kd = torch.from_numpy(oracle.nvfp4_dequantize(kq, kqs).view(np.int16)).view(torch.bfloat16)
    vd = torch.from_numpy(oracle.nvfp4_dequantize(vq, vqs).view(np.int16)).view(torch.bfloat16)
    o_ref, l_ref = oracle.sparse_attn(x["q"].cpu(), kd, vd, x["q2k"].cpu(), causal=True, rows=rows)
    assert_attn_close(o.view(-1, spec.Hq, 128)[rows], lse.view(-1, spec.Hq)[rows], o_ref, l_ref, spec.name)


def test_generator_identical_on_cpu_and_gpu():
    a = synth.normal_bf16((3, 1000, 7), 42, synth.STREAM_K, device=DEV).cpu()
    b = synth.normal_bf16((3, 1000, 7), 42, synth.STREAM_K)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(synth.q2k_causal_sink(1, 2, 3000, 4096, 16, device=DEV).cpu(),
                       synth.q2k_causal_sink(1, 2, 3000, 4096, 16))
