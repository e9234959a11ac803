"""GPU k->q CSR and work plan vs the oracle: bit-exact, through the C ABI."""

import numpy as np
import pytest
import torch

import msa_synth as synth
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _gpu_csr(q2k, Skv, qpk, seqused=None):
    import block_sparse_top_gb300 as msa
    status = msa.new_status(DEV)
    csr = msa.build_k2q_csr(q2k.to(DEV), Skv, qpk, seqused=None if seqused is None else seqused.to(DEV),
                            status=status)
    st = msa.read_status(status)
    return csr, st


def _check_equal(csr, ref):
    assert np.array_equal(csr.row_ptr.cpu().numpy(), ref["row_ptr"])
    assert np.array_equal(csr.q_indices.cpu().numpy(), ref["q_indices"])
    assert np.array_equal(csr.qsplit.cpu().numpy(), ref["qsplit"])
    assert np.array_equal(csr.split_counts.cpu().numpy(), ref["split_counts"])


def plan_units(plan: torch.Tensor, row_off):
    """Decodes a plan buffer: header ints and units as (head, row, start, count),
    row = row_off[seq] + block (units are {int16 head, int16 block, int32 seq,
    int32 start, int32 count})."""
    words = plan.cpu().view(torch.int32).numpy()
    work = int(words[0])
    raw = words[16:16 + 4 * work].reshape(-1, 4)
    head = (raw[:, 0] & 0xFFFF).astype(np.int64)
    blk = (raw[:, 0] >> 16).astype(np.int64)
    seq = raw[:, 1].astype(np.int64)
    rows = np.asarray(row_off, dtype=np.int64)[seq] + blk
    return words, [(int(h), int(r), int(st), int(c)) for h, r, st, c in zip(head, rows, raw[:, 2], raw[:, 3])]


def _check_plan(csr, row_off=None):
    if row_off is None:  # uniform batch: sequence b owns rows b*nblk ..
        nblk = -(-csr.Skv // 128)
        row_off = [b * nblk for b in range(csr.B)]
    plan, units = plan_units(csr.plan, row_off)
    work, cap, qpk, qpu = plan[:4]
    assert work <= cap and qpk == csr.qhead_per_kv
    rp = csr.row_ptr.cpu().numpy()
    rows = rp.shape[1] - 1
    covered = np.zeros((csr.Hkv, rows), dtype=np.int64)
    seen = set()
    for h, r, start, count in units:
        assert 0 < count <= qpu
        assert rp[h, r] <= start and start + count <= rp[h, r + 1]
        covered[h, r] += count
        for x in range(start, start + count):
            assert (h, x) not in seen
            seen.add((h, x))
    assert np.array_equal(covered, np.diff(rp, axis=1))
    # units run head-major, then wave by wave
    W = int(plan[4])
    qi = csr.q_indices.cpu().numpy()
    order = [(int(h), int(qi[h, start]) // W) for h, r, start, count in units]
    assert order == sorted(order)


CASES = [
    ("tiny_noncausal", synth.TINY_NONCAUSAL_1K),
    ("sink_small", synth.PrefillSpec("s", B=2, Sq=1000, Skv=2048, Hkv=3, qpk=16, topk=16, causal=True,
                                     pattern="sink")),
    ("uniform_small", synth.PrefillSpec("u", B=1, Sq=3000, Skv=2500, Hkv=1, qpk=2, topk=8, causal=True,
                                        pattern="uniform")),
    ("topk32_q_gt_kv", synth.PrefillSpec("t", B=1, Sq=5000, Skv=4096, Hkv=2, qpk=1, topk=32, causal=True,
                                         pattern="sink")),
]


@pytest.mark.parametrize("name,spec", CASES, ids=[c[0] for c in CASES])
def test_csr_bit_exact(name, spec):
    q2k = synth.make_prefill_q2k(spec)
    ref = oracle.build_k2q_csr(q2k, spec.Skv)
    csr, st = _gpu_csr(q2k, spec.Skv, spec.qpk)
    _check_equal(csr, ref)
    _check_plan(csr)
    assert st == 0


def test_csr_messy_indices_and_seqused():
    B, Hkv, Sq, Skv, topk = 2, 2, 333, 1024, 8
    g = torch.Generator().manual_seed(5)
    q2k = torch.randint(-4, 12, (B, Hkv, Sq, topk), generator=g, dtype=torch.int32)
    seqused = torch.tensor([1024, 300], dtype=torch.int32)
    ref = oracle.build_k2q_csr(q2k, Skv, seqused=seqused)
    csr, st = _gpu_csr(q2k, Skv, 4, seqused)
    _check_equal(csr, ref)
    _check_plan(csr)
    assert st & 0x1 and st & 0x2   # out-of-range and duplicate ids were seen


def test_csr_block_selected_by_no_query_and_empty_queries():
    B, Hkv, Sq, Skv, topk = 1, 1, 256, 1024, 4
    q2k = torch.full((B, Hkv, Sq, topk), -1, dtype=torch.int32)
    q2k[0, 0, ::2, 0] = 0
    q2k[0, 0, ::3, 1] = 5   # blocks 1-4, 6, 7 stay empty; odd queries not divisible by 3 select nothing
    ref = oracle.build_k2q_csr(q2k, Skv)
    csr, _ = _gpu_csr(q2k, Skv, 16)
    _check_equal(csr, ref)
    _check_plan(csr)


@pytest.mark.parametrize("spec", [synth.CAUSAL_SINK_32K, synth.CAUSAL_UNIFORM_48K, synth.CAUSAL_SINK_384K],
                         ids=lambda s: s.name)
def test_csr_bit_exact_full_size(spec):
    q2k = synth.make_prefill_q2k(spec, device=DEV)
    csr, st = _gpu_csr(q2k, spec.Skv, spec.qpk)
    ref = oracle.build_k2q_csr(q2k.cpu(), spec.Skv)
    _check_equal(csr, ref)
    assert st == 0
    # the plan's units cover every row exactly (cheap invariant at full size)
    plan = csr.plan.cpu().view(torch.int32).numpy()
    work = plan[0]
    units = plan[16:16 + 4 * work].reshape(-1, 4)
    assert units[:, 3].sum() == int(csr.row_ptr[:, -1].sum())


def test_csr_deterministic_across_runs():
    spec = synth.PrefillSpec("d", B=1, Sq=4096, Skv=4096, Hkv=2, qpk=16, topk=16, causal=True, pattern="sink")
    q2k = synth.make_prefill_q2k(spec, device=DEV)
    a, _ = _gpu_csr(q2k, spec.Skv, spec.qpk)
    a = [t.clone() for t in (a.row_ptr, a.q_indices, a.qsplit, a.split_counts)]
    for _ in range(3):
        b, _ = _gpu_csr(q2k, spec.Skv, spec.qpk)
        for x, y in zip(a, (b.row_ptr, b.q_indices, b.qsplit, b.split_counts)):
            assert torch.equal(x, y)


def test_csr_q2k_view_not_16_byte_aligned():
    """A q2k view starting 4 bytes past a 16-byte boundary takes the builder's
    scalar loads and gives the same CSR as the oracle."""
    spec = synth.PrefillSpec("a", B=1, Sq=1000, Skv=2048, Hkv=2, qpk=4, topk=8, causal=True, pattern="sink")
    q2k = synth.make_prefill_q2k(spec)
    flat = torch.empty(q2k.numel() + 1, dtype=torch.int32, device=DEV)
    view = flat[1:].view(q2k.shape)
    view.copy_(q2k.to(DEV))
    assert view.data_ptr() % 16 == 4
    ref = oracle.build_k2q_csr(q2k, spec.Skv)
    csr, st = _gpu_csr(view, spec.Skv, spec.qpk)
    _check_equal(csr, ref)
    _check_plan(csr)
    assert st == 0
