"""GPU block-sparse paged decode (msa_sparse_attn_paged_fwd) vs the float64 oracle."""

import numpy as np
import pytest
import torch

import msa_synth as synth
import oracle
from parity import assert_attn_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def run_case(spec, rows=None, mutate=None):
    import block_sparse_top_gb300 as msa
    d = synth.make_decode_inputs(spec, device=DEV)
    if mutate:
        mutate(d)
    status = msa.new_status(DEV)
    o, lse = msa.sparse_attn_paged_fwd(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seqused"], d["q2k"],
                                       status=status)
    st = msa.read_status(status)
    o_ref, l_ref = oracle.sparse_attn_paged(d["q"].cpu(), d["k_pool"].cpu(), d["v_pool"].cpu(),
                                            d["page_table"].cpu(), d["seqused"].cpu(), d["q2k"].cpu(), rows=rows)
    og, lg = (o, lse) if rows is None else (o[rows], lse[rows])
    assert_attn_close(og, lg, o_ref, l_ref, spec.name)
    return st, o, lse


@pytest.mark.parametrize("L", [1024, 2048, 4096, 8192])
def test_decode_sweep_small_full_parity(L):
    st, _, _ = run_case(synth.paged_decode_spec(L))
    assert st == 0


@pytest.mark.parametrize("L", [16384, 32768, 65536, 131072])
def test_decode_sweep_large_sampled(L):
    spec = synth.paged_decode_spec(L)
    rows = synth.sample_query_rows(spec.B * spec.Sq, 24, must=[0, 7, 255])
    run_case(spec, rows=rows)


def D(name, **kw):
    base = dict(B=4, Sq=8, Hkv=2, qpk=16, topk=16, kv_len=2048, trim=17)
    base.update(kw)
    return synth.DecodeSpec(name, **base)


EDGE = [
    D("qpk1_sq3", qpk=1, Sq=3, topk=4),
    D("qpk2_many_groups", qpk=2, Sq=150, topk=8, kv_len=8192, trim=100),
    D("qpk4_topk32", qpk=4, Sq=8, topk=32, kv_len=8192),
    D("qpk8_sq1", qpk=8, Sq=1, topk=16, kv_len=16384),
    D("short_kv", qpk=16, Sq=8, topk=16, kv_len=128, trim=123),   # seqused 5 < Sq: early queries see nothing
    D("trim_zero", qpk=16, Sq=8, topk=4, kv_len=1024, trim=0),
    # three query groups per (sequence, KV head), the last one partial: consecutive
    # groups of one head share nothing, their Q tiles must not be reused
    D("qpk16_three_groups", qpk=16, Sq=20, topk=8, kv_len=4096, Hkv=3),
    # one group only: its ~120 union blocks are shared out between CTAs (at
    # least 8 units each), and the CTA finishing last merges ~14 pieces
    D("one_group_many_pieces", B=1, Hkv=1, Sq=8, qpk=16, topk=16, kv_len=131072, trim=17),
    # two groups of ~57 blocks and 152 SMs: cut groups whose pieces lie in
    # different numbers of CTAs, some CTAs holding the end of one group and the
    # start of the next
    D("two_groups_cut", B=2, Hkv=1, Sq=8, qpk=16, topk=16, kv_len=8192, trim=17),
]


@pytest.mark.parametrize("spec", EDGE, ids=lambda s: s.name)
def test_decode_edge_cases(spec):
    run_case(spec)


def test_decode_bad_page_entry_sets_status_and_skips_block():
    spec = D("bad_page", kv_len=1024, topk=4)

    def mutate(d):
        d["page_table"][1, 0] = 10 ** 6          # out of the pool: block skipped, status bit set

    import block_sparse_top_gb300 as msa
    d = synth.make_decode_inputs(spec, device=DEV)
    mutate(d)
    status = msa.new_status(DEV)
    o, lse = msa.sparse_attn_paged_fwd(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seqused"], d["q2k"],
                                       status=status)
    st = msa.read_status(status)
    assert st & msa.MSA_STATUS_PAGE_RANGE
    # sequences whose pages are valid are unaffected
    rows = list(range(0, 8)) + list(range(16, 32))
    o_ref, l_ref = oracle.sparse_attn_paged(d["q"].cpu(), d["k_pool"].cpu(), d["v_pool"].cpu(),
                                            d["page_table"].cpu().clamp(max=spec.num_pages - 1),
                                            d["seqused"].cpu(), d["q2k"].cpu(), rows=rows)
    assert_attn_close(o[rows], lse[rows], o_ref, l_ref, "bad_page")


def test_decode_repeat_calls_identical():
    import block_sparse_top_gb300 as msa
    spec = synth.paged_decode_spec(4096)
    d = synth.make_decode_inputs(spec, device=DEV)
    a = msa.sparse_attn_paged_fwd(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seqused"], d["q2k"])
    b = msa.sparse_attn_paged_fwd(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seqused"], d["q2k"])
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_peaked_scores_rescale_accumulated_rows():
    """With a softmax scale of 8 a row's later blocks often hold a max far
    above the reference of its accumulated piece, so the decode rescales the
    accumulated O row; the result still matches the oracle."""
    import block_sparse_top_gb300 as msa
    spec = synth.paged_decode_spec(8192)
    d = synth.make_decode_inputs(spec, device=DEV)
    o, lse = msa.sparse_attn_paged_fwd(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seqused"], d["q2k"],
                                       softmax_scale=8.0)
    torch.cuda.synchronize()
    rows = synth.sample_query_rows(spec.B * spec.Sq, 48, must=[0, 7, 255])
    o_ref, l_ref = oracle.sparse_attn_paged(d["q"].cpu(), d["k_pool"].cpu(), d["v_pool"].cpu(),
                                            d["page_table"].cpu(), d["seqused"].cpu(), d["q2k"].cpu(), rows=rows,
                                            scale=8.0)
    assert_attn_close(o[rows], lse[rows], o_ref, l_ref, "decode peaked")


def test_decode_uneven_unions_one_launch():
    """Unions of at most 16 blocks run as one launch, each CTA planning and
    holding its own group whatever the union sizes: here one group keeps all
    16 blocks, one keeps 4 and the rest only their last visible block."""
    spec = D("uneven_unions", B=4, Sq=8, Hkv=2, qpk=16, topk=16, kv_len=2048, trim=17)

    def mutate(d):
        q2k = d["q2k"]                     # [B, Hkv, Sq, topk], slot 0 = last visible block
        keep = torch.ones_like(q2k, dtype=torch.bool)
        keep[:, :, :, 1:] = False
        keep[0, 0] = True                  # the long group: every slot
        keep[1, 1, :, :4] = True           # a short one: four slots per query
        d["q2k"] = torch.where(keep, q2k, torch.full_like(q2k, -1))

    st, _, _ = run_case(spec, mutate=mutate)
    assert st == 0
