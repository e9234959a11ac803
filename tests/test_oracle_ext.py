"""Pins for the oracle's varlen, temperature-LSE and every-block paths.

Each check rests on something other than the function under test:

* varlen: a ragged batch equals the uniform oracle (pinned on its own in
  test_oracle.py) run on each sequence's slice, which is how the test page's
  varlen reference defines it; with every block selected it equals textbook
  softmax attention per sequence (numpy / scipy);
* temperature LSE: at T = 1 it is the LSE; with constant keys it is
  c / T + ln |visible| (closed form); with every block selected it is scipy's
  logsumexp of the scaled scores divided by T;
* every-block selection (q2k = None): equals the paged oracle given a q2k that
  lists every block, and dense causal attention on the truncated sequence;
* varlen CSR: brute-force enumeration, and the uniform CSR oracle when all
  sequences have the same lengths.
"""

import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import msa_synth as synth
import oracle


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.float().double().numpy()


def _assert_close(o, lse, o_ref, lse_ref, tol=1e-10):
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=0, atol=tol)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=tol)


VARLEN = [
    synth.VarlenSpec("vl_sink", q_lens=(300, 77, 512), k_lens=(640, 200, 512), Hkv=2, qpk=4, topk=4,
                     causal=True, pattern="sink"),
    synth.VarlenSpec("vl_uniform_q_longer", q_lens=(260, 129), k_lens=(256, 1000), Hkv=1, qpk=2, topk=8,
                     causal=True, pattern="uniform"),
    synth.VarlenSpec("vl_noncausal", q_lens=(40, 1, 90), k_lens=(512, 1000, 640), Hkv=2, qpk=1, topk=4,
                     causal=False, pattern="perm_prefix"),
]


def _slices(spec, x):
    cq, ck = x["cu_seqlens_q"].tolist(), x["cu_seqlens_k"].tolist()
    for b in range(spec.B):
        q = x["q"][cq[b]:cq[b + 1]].unsqueeze(0)
        k = x["k"][ck[b]:ck[b + 1]].unsqueeze(0)
        v = x["v"][ck[b]:ck[b + 1]].unsqueeze(0)
        sel = x["q2k"][:, cq[b]:cq[b + 1]].unsqueeze(0).contiguous()      # [1,Hkv,Sq_b,topk]
        yield b, cq[b], cq[b + 1], q, k, v, sel


@pytest.mark.parametrize("spec", VARLEN, ids=lambda s: s.name)
def test_varlen_equals_uniform_oracle_per_sequence(spec):
    x = synth.make_varlen_inputs(spec)
    o, l = oracle.sparse_attn_varlen(x["q"], x["k"], x["v"], x["q2k"], x["cu_seqlens_q"], x["cu_seqlens_k"],
                                     causal=spec.causal)
    for b, q0, q1, q, k, v, sel in _slices(spec, x):
        ob, lb = oracle.sparse_attn(q, k, v, sel, causal=spec.causal)
        _assert_close(o[q0:q1], l[q0:q1], ob, lb, tol=1e-12)


def test_varlen_rows_subset_matches_full_run():
    spec = VARLEN[0]
    x = synth.make_varlen_inputs(spec)
    o, l = oracle.sparse_attn_varlen(x["q"], x["k"], x["v"], x["q2k"], x["cu_seqlens_q"], x["cu_seqlens_k"],
                                     causal=True)
    rows = [0, 299, 300, 376, 377, 888]
    os_, ls = oracle.sparse_attn_varlen(x["q"], x["k"], x["v"], x["q2k"], x["cu_seqlens_q"], x["cu_seqlens_k"],
                                        causal=True, rows=rows)
    _assert_close(os_, ls, o[rows], l[rows], tol=0)


def _dense_rows(q, k, v, causal, scale, temp=None):
    """Textbook attention for one sequence: q [Sq,Hq,D], k/v [Skv,Hkv,D]."""
    Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[0], k.shape[1]
    qpk = Hq // Hkv
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    O = np.zeros((Sq, Hq, D))
    L = np.full((Sq, Hq), -np.inf)
    T = np.full((Sq, Hq), -np.inf)
    for hq in range(Hq):
        h = hq // qpk
        S = scale * qf[:, hq] @ kf[:, h].T
        for s in range(Sq):
            n = Skv if not causal else max(0, min(Skv, s + (Skv - Sq) + 1))
            if n == 0:
                continue
            row = S[s, :n]
            L[s, hq] = logsumexp(row)
            if temp is not None:
                T[s, hq] = logsumexp(row / temp)
            O[s, hq] = softmax(row) @ vf[:n, h]
    return O, L, T


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_every_block_equals_dense_attention_per_sequence(causal):
    spec = synth.VarlenSpec("vl_dense", q_lens=(130, 60, 256), k_lens=(256, 300, 128), Hkv=1, qpk=2, topk=4,
                            causal=causal, pattern="sink")
    x = synth.make_varlen_inputs(spec)
    # every block of each sequence, in a scrambled slot order, padded with -1
    q2k = torch.full_like(x["q2k"], -1)
    cq = x["cu_seqlens_q"].tolist()
    for b in range(spec.B):
        nb = -(-spec.k_lens[b] // 128)
        q2k[:, cq[b]:cq[b + 1], :nb] = torch.arange(nb - 1, -1, -1, dtype=torch.int32)
    o, l, lt = oracle.sparse_attn_varlen(x["q"], x["k"], x["v"], q2k, x["cu_seqlens_q"], x["cu_seqlens_k"],
                                         causal=causal, temperature=0.7)
    scale = 1 / math.sqrt(128)
    for b, q0, q1, q, k, v, _ in _slices(spec, x):
        O, L, T = _dense_rows(q[0], k[0], v[0], causal, scale, temp=0.7)
        _assert_close(o[q0:q1], l[q0:q1], O, L)
        fin = np.isfinite(T)
        assert np.array_equal(np.isneginf(lt[q0:q1]), np.isneginf(T))
        np.testing.assert_allclose(lt[q0:q1][fin], T[fin], rtol=0, atol=1e-10)


def test_temperature_one_is_the_lse():
    spec = VARLEN[0]
    x = synth.make_varlen_inputs(spec)
    o, l, lt = oracle.sparse_attn_varlen(x["q"], x["k"], x["v"], x["q2k"], x["cu_seqlens_q"], x["cu_seqlens_k"],
                                         causal=True, temperature=1.0)
    assert np.array_equal(np.isneginf(lt), np.isneginf(l))
    fin = np.isfinite(l)
    np.testing.assert_allclose(lt[fin], l[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("T", [0.25, 3.0])
def test_temperature_lse_closed_form_for_constant_keys(T):
    """All keys equal k: every visible score is c = scale q.k, so lse_T = c / T + ln n."""
    Sq, Skv, Hkv, qpk, D = 20, 1024, 1, 2, 128
    q = synth.normal_bf16((Sq, Hkv * qpk, D), 3, synth.STREAM_Q)
    kbar = synth.normal_bf16((D,), 11, synth.STREAM_AUX)
    k = kbar.view(1, 1, D).expand(Skv, Hkv, D).contiguous()
    v = synth.normal_bf16((Skv, Hkv, D), 3, synth.STREAM_V)
    q2k = synth.q2k_perm_prefix(1, Hkv, Sq, 8, 3, seed=5)[0]           # [Hkv, Sq, 3]
    cu_q = torch.tensor([0, Sq], dtype=torch.int32)
    cu_k = torch.tensor([0, Skv], dtype=torch.int32)
    scale = 1 / math.sqrt(D)
    _, l, lt = oracle.sparse_attn_varlen(q, k, v, q2k, cu_q, cu_k, causal=False, temperature=T)
    qf, kf = _f64(q), _f64(kbar)
    for s in range(Sq):
        for g in range(qpk):
            c = scale * qf[s, g] @ kf
            n = 3 * 128
            assert abs(lt[s, g] - (c / T + math.log(n))) < 1e-10
            assert abs(l[s, g] - (c + math.log(n))) < 1e-10


def _to_pool(k, pt, page=128):
    """Scatter dense [B,L,Hkv,D] into a pool [num_pages,page,Hkv,D] through page_table."""
    B, L, Hkv, D = k.shape
    pool = torch.zeros((pt.numel(), page, Hkv, D), dtype=k.dtype)
    for b in range(B):
        for j in range(pt.shape[1]):
            seg = k[b, j * page:(j + 1) * page]
            pool[int(pt[b, j]), :seg.shape[0]] = seg
    return pool


def test_every_block_paged_equals_listed_blocks_and_dense_causal():
    B, Sq, L, Hkv, qpk, D = 3, 8, 640, 2, 4, 128
    Hq = Hkv * qpk
    q = synth.normal_bf16((B * Sq, Hq, D), 8, synth.STREAM_Q)
    k = synth.normal_bf16((B, L, Hkv, D), 8, synth.STREAM_K)
    v = synth.normal_bf16((B, L, Hkv, D), 8, synth.STREAM_V)
    pt = synth.shuffled_page_table(B, L // 128, seed=9)
    kp, vp = _to_pool(k, pt), _to_pool(v, pt)
    seqused = torch.tensor([L - 17, 130, 5], dtype=torch.int32)
    cu_q = torch.arange(0, B * Sq + 1, Sq, dtype=torch.int32)
    o, l = oracle.sparse_attn_varlen(q, kp, vp, None, cu_q, causal=True, page_table=pt, seqused=seqused)
    # the same selection written out: every block of the page table
    nb = L // 128
    q2k = torch.arange(nb, dtype=torch.int32).expand(B, Hkv, Sq, nb).contiguous()
    o2, l2 = oracle.sparse_attn_paged(q, kp, vp, pt, seqused, q2k, causal=True)
    _assert_close(o, l, o2, l2, tol=1e-12)
    scale = 1 / math.sqrt(D)
    for b in range(B):
        n = int(seqused[b])
        O, Lr, _ = _dense_rows(q[b * Sq:(b + 1) * Sq], k[b, :n], v[b, :n], True, scale)
        _assert_close(o[b * Sq:(b + 1) * Sq], l[b * Sq:(b + 1) * Sq], O, Lr)


# ---------------------------------------------------------------------------
# varlen CSR
# ---------------------------------------------------------------------------

def _csr_varlen_brute(q2k: np.ndarray, q_lens, k_lens, blk=128, seqused=None):
    Hkv, total_q, topk = q2k.shape
    row_off = [0]
    for kl in k_lens:
        row_off.append(row_off[-1] + -(-kl // blk))
    cq = [0]
    for ql in q_lens:
        cq.append(cq[-1] + ql)
    out = {}
    for h in range(Hkv):
        rows = [[] for _ in range(row_off[-1])]
        for b in range(len(q_lens)):
            kv = k_lens[b] if seqused is None else int(seqused[b])
            nvalid = min(row_off[b + 1] - row_off[b], -(-kv // blk))
            for gq in range(cq[b], cq[b + 1]):
                seen = []
                for t in range(topk):
                    j = int(q2k[h, gq, t])
                    if 0 <= j < nvalid and j not in seen:
                        rows[row_off[b] + j].append((gq, len(seen)))
                        seen.append(j)
        out[h] = rows
    return out


@pytest.mark.parametrize("case", ["sink", "messy"])
def test_varlen_csr_matches_brute_force(case):
    if case == "sink":
        spec = synth.VarlenSpec("vlc", q_lens=(300, 1, 129), k_lens=(640, 128, 1000), Hkv=2, qpk=4, topk=8,
                                causal=True, pattern="sink")
        x = synth.make_varlen_inputs(spec)
        q2k, seqused = x["q2k"].numpy(), None
    else:  # duplicates, out-of-range and negative ids, seqused trimming
        spec = synth.VarlenSpec("vlm", q_lens=(30, 50), k_lens=(512, 300), Hkv=1, qpk=2, topk=6, causal=False,
                                pattern="sink")
        x = synth.make_varlen_inputs(spec)
        rng = np.random.default_rng(1)
        q2k = rng.integers(-3, 6, size=(1, 80, 6)).astype(np.int32)
        seqused = np.array([400, 130], dtype=np.int32)
    c = oracle.build_k2q_csr_varlen(q2k, x["cu_seqlens_q"], x["cu_seqlens_k"], seqused=seqused)
    ref = _csr_varlen_brute(q2k, spec.q_lens, spec.k_lens, seqused=seqused)
    for h in range(spec.Hkv):
        rows = ref[h]
        assert c["row_ptr"][h].tolist() == [0] + list(np.cumsum([len(r) for r in rows]))
        flat = [qq for r in rows for (qq, _) in r]
        nnz = len(flat)
        assert c["q_indices"][h, :nnz].tolist() == flat
        assert c["qsplit"][h, :nnz].tolist() == [qq | (rk << 24) for r in rows for (qq, rk) in r]
        assert (c["q_indices"][h, nnz:] == -1).all() and (c["qsplit"][h, nnz:] == -1).all()
        for gq in range(spec.total_q):
            n = sum(1 for r in rows for (qq, _) in r if qq == gq)
            assert c["split_counts"][gq, h] == n


def test_varlen_csr_with_equal_lengths_equals_uniform_csr():
    B, Hkv, Sq, Skv, topk = 3, 2, 200, 512, 8
    q2k = synth.q2k_causal_sink(B, Hkv, Sq, Skv, topk, seed=4)          # [B,Hkv,Sq,topk]
    flat = q2k.permute(1, 0, 2, 3).reshape(Hkv, B * Sq, topk).contiguous()
    cu_q = torch.arange(0, B * Sq + 1, Sq, dtype=torch.int32)
    cu_k = torch.arange(0, B * Skv + 1, Skv, dtype=torch.int32)
    a = oracle.build_k2q_csr_varlen(flat, cu_q, cu_k)
    b = oracle.build_k2q_csr(q2k, Skv)
    for key in ("row_ptr", "q_indices", "qsplit", "split_counts"):
        assert np.array_equal(a[key], b[key]), key
