"""Pins for the float64 oracle: each check rests on something other than the oracle.

* dense equivalence: selecting every block reduces sparse attention to plain
  (optionally bottom-right causal) softmax attention, computed here with numpy
  matmuls and scipy's logsumexp/softmax;
* closed forms: constant keys give O = mean of the visible values and
  LSE = scale*q.k + ln|visible|; a single visible key gives O = v, LSE = scale*q.k;
* invariances: slot order, duplicate ids and padding do not change the result;
* the LSE merge law over disjoint block sets (the rule the split-KV combine uses);
* paging: a shuffled page table over the same tokens gives the dense result,
  and seqused trimming equals attention over the truncated sequence;
* CSR: brute-force enumeration on tiny inputs;
* NVFP4: the pages' e2m1 table, e4m3 against torch's float8_e4m3fn, and the
  quantiser's rounding choices against brute force over all codes.
"""

import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import msa_synth as synth
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.float().double().numpy()


def _rand_inputs(B, Sq, Skv, Hkv, qpk, D=128, seed=7):
    Hq = Hkv * qpk
    q = synth.normal_bf16((B, Sq, Hq, D), seed, synth.STREAM_Q)
    k = synth.normal_bf16((B, Skv, Hkv, D), seed, synth.STREAM_K)
    v = synth.normal_bf16((B, Skv, Hkv, D), seed, synth.STREAM_V)
    return q, k, v


def _dense_reference(q, k, v, causal, kv_len=None, scale=None):
    """Textbook softmax attention with GQA and bottom-right causal mask (numpy)."""
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    qpk = Hq // Hkv
    scale = 1 / math.sqrt(D) if scale is None else scale
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    O = np.zeros((B, Sq, Hq, D))
    L = np.full((B, Sq, Hq), -np.inf)
    for b in range(B):
        n = Skv if kv_len is None else int(kv_len[b])
        for hq in range(Hq):
            h = hq // qpk
            S = scale * qf[b, :, hq, :] @ kf[b, :n, h, :].T          # [Sq, n]
            mask = np.ones_like(S, dtype=bool)
            if causal:
                t = np.arange(n)[None, :]
                s = np.arange(Sq)[:, None]
                mask = t <= s + (n - Sq)
            for s_ in range(Sq):
                row = S[s_][mask[s_]]
                if row.size == 0:
                    continue
                L[b, s_, hq] = logsumexp(row)
                O[b, s_, hq] = softmax(row) @ vf[b, :n, h, :][mask[s_]]
    return O.reshape(B * Sq, Hq, D), L.reshape(B * Sq, Hq)


def _assert_close(o, lse, o_ref, lse_ref, tol=1e-10):
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=0, atol=tol)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=tol)


# ---------------------------------------------------------------------------
# dense equivalence
# ---------------------------------------------------------------------------

def test_all_blocks_noncausal_equals_dense_attention():
    B, Sq, Skv, Hkv, qpk = 2, 48, 512, 2, 2
    q, k, v = _rand_inputs(B, Sq, Skv, Hkv, qpk)
    q2k = synth.q2k_perm_prefix(B, Hkv, Sq, 4, 4, seed=3)          # every block, random order
    o, l = oracle.sparse_attn(q, k, v, q2k, causal=False)
    o_ref, l_ref = _dense_reference(q, k, v, causal=False)
    _assert_close(o, l, o_ref, l_ref)


@pytest.mark.parametrize("Sq,Skv", [(200, 512), (512, 512), (600, 384)])
def test_all_blocks_causal_equals_dense_causal_attention(Sq, Skv):
    B, Hkv, qpk = 1, 2, 4
    q, k, v = _rand_inputs(B, Sq, Skv, Hkv, qpk)
    nblk = Skv // 128
    topk = 8
    q2k = torch.full((B, Hkv, Sq, topk), -1, dtype=torch.int32)
    q2k[..., :nblk] = torch.arange(nblk, dtype=torch.int32)
    o, l = oracle.sparse_attn(q, k, v, q2k, causal=True)
    o_ref, l_ref = _dense_reference(q, k, v, causal=True)
    _assert_close(o, l, o_ref, l_ref)
    if Sq > Skv:  # leading queries see no key at all: O = 0, LSE = -inf
        assert np.isneginf(l[0]).all() and (o[0] == 0).all()


def test_partial_last_block_masks_keys_past_kv_length():
    # Skv not a multiple of the block size: keys >= Skv do not exist.
    B, Sq, Skv, Hkv, qpk = 1, 40, 300, 1, 2
    q, k, v = _rand_inputs(B, Sq, Skv, Hkv, qpk)
    q2k = torch.tensor([0, 1, 2, -1], dtype=torch.int32).expand(B, Hkv, Sq, 4).contiguous()
    o, l = oracle.sparse_attn(q, k, v, q2k, causal=False)
    o_ref, l_ref = _dense_reference(q, k, v, causal=False)
    _assert_close(o, l, o_ref, l_ref)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def test_constant_keys_give_mean_of_values_and_log_count():
    B, Sq, Skv, Hkv, qpk, D = 1, 16, 1024, 1, 2, 128
    q, _, v = _rand_inputs(B, Sq, Skv, Hkv, qpk)
    kbar = synth.normal_bf16((D,), 11, synth.STREAM_AUX)
    k = kbar.view(1, 1, 1, D).expand(B, Skv, Hkv, D).contiguous()
    q2k = synth.q2k_perm_prefix(B, Hkv, Sq, 8, 3, seed=5)            # 3 distinct blocks of 8
    o, l = oracle.sparse_attn(q, k, v, q2k, causal=False)
    scale = 1 / math.sqrt(D)
    vf, qf, kf = _f64(v), _f64(q), _f64(kbar)
    for s in range(Sq):
        toks = np.concatenate([np.arange(128 * j, 128 * j + 128) for j in q2k[0, 0, s].tolist()])
        mean_v = vf[0, toks, 0, :].mean(axis=0)
        for g in range(qpk):
            np.testing.assert_allclose(o[s, g], mean_v, atol=1e-12)
            assert abs(l[s, g] - (scale * qf[0, s, g] @ kf + math.log(len(toks)))) < 1e-10


def test_single_visible_key_returns_its_value():
    # causal, Sq == Skv: query 0 sees exactly key 0 when it selects block 0.
    B, Sq, Skv, Hkv, qpk, D = 1, 256, 256, 1, 4, 128
    q, k, v = _rand_inputs(B, Sq, Skv, Hkv, qpk)
    q2k = torch.full((B, Hkv, Sq, 4), -1, dtype=torch.int32)
    q2k[..., 0] = 0
    o, l = oracle.sparse_attn(q, k, v, q2k, causal=True)
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    for g in range(qpk):
        np.testing.assert_array_equal(o[0, g], vf[0, 0, 0])
        assert abs(l[0, g] - qf[0, 0, g] @ kf[0, 0, 0] / math.sqrt(D)) < 1e-12


def test_query_without_valid_block_is_zero_and_minus_inf():
    q, k, v = _rand_inputs(1, 8, 256, 1, 2)
    q2k = torch.full((1, 1, 8, 4), -1, dtype=torch.int32)
    q2k[0, 0, 3, 1] = 7        # out of range: padding
    q2k[0, 0, 5, 0] = 1        # valid
    o, l = oracle.sparse_attn(q, k, v, q2k, causal=False)
    for s in range(8):
        if s == 5:
            assert np.isfinite(l[s]).all()
        else:
            assert np.isneginf(l[s]).all() and (o[s] == 0).all()


# ---------------------------------------------------------------------------
# invariances and the merge law
# ---------------------------------------------------------------------------

def test_slot_order_duplicates_and_padding_do_not_matter():
    B, Sq, Skv, Hkv, qpk = 1, 64, 1024, 2, 2
    q, k, v = _rand_inputs(B, Sq, Skv, Hkv, qpk)
    q2k = synth.q2k_causal_sink(B, Hkv, Sq, Skv, 8, seed=9)
    o, l = oracle.sparse_attn(q, k, v, q2k, causal=True)
    g = torch.Generator().manual_seed(0)
    perm = torch.randperm(8, generator=g)
    shuffled = q2k[..., perm]
    o2, l2 = oracle.sparse_attn(q, k, v, shuffled, causal=True)
    _assert_close(o2, l2, o, l, tol=1e-12)
    # append duplicates of every slot plus padding: topk 8 -> 17 slots
    dup = torch.cat([q2k, q2k.flip(-1), torch.full_like(q2k[..., :1], -1)], dim=-1)
    o3, l3 = oracle.sparse_attn(q, k, v, dup, causal=True)
    _assert_close(o3, l3, o, l, tol=1e-12)


def test_lse_merge_law_over_disjoint_block_sets():
    B, Sq, Skv, Hkv, qpk = 1, 32, 2048, 1, 4
    q, k, v = _rand_inputs(B, Sq, Skv, Hkv, qpk)
    q2k = synth.q2k_perm_prefix(B, Hkv, Sq, 16, 8, seed=13)
    oa, la = oracle.sparse_attn(q, k, v, q2k[..., :3].contiguous(), causal=False)
    ob, lb = oracle.sparse_attn(q, k, v, q2k[..., 3:].contiguous(), causal=False)
    o, l = oracle.sparse_attn(q, k, v, q2k, causal=False)
    lm = np.logaddexp(la, lb)
    om = np.exp(la - lm)[..., None] * oa + np.exp(lb - lm)[..., None] * ob
    _assert_close(om, lm, o, l, tol=1e-12)


# ---------------------------------------------------------------------------
# paged KV
# ---------------------------------------------------------------------------

def _to_pool(k, page_table, page=128):
    """Scatter dense [B,S,H,D] into a [num_pages,page,H,D] pool through page_table."""
    B, S, H, D = k.shape
    mp = page_table.shape[1]
    pool = torch.zeros((B * mp, page, H, D), dtype=k.dtype)
    for b in range(B):
        for j in range(mp):
            seg = k[b, j * page:(j + 1) * page]
            pool[int(page_table[b, j]), :seg.shape[0]] = seg
    return pool


def test_paged_shuffled_pool_equals_truncated_dense():
    B, Sq, L, Hkv, qpk, trim = 3, 8, 1024, 2, 4, 17
    Hq = Hkv * qpk
    q, k, v = _rand_inputs(B, Sq, L, Hkv, qpk)
    pt = synth.shuffled_page_table(B, L // 128, seed=21)
    kp, vp = _to_pool(k, pt), _to_pool(v, pt)
    seqused = torch.tensor([L - trim, L - 128 - 5, 300], dtype=torch.int32)
    q2k = synth.q2k_decode(B, Hkv, Sq, seqused, 4, seed=2)
    o, l = oracle.sparse_attn_paged(q.reshape(B * Sq, Hq, 128), kp, vp, pt, seqused, q2k, causal=True)
    for b in range(B):
        n = int(seqused[b])
        ob, lb = oracle.sparse_attn(q[b:b + 1], k[b:b + 1, :n].contiguous(), v[b:b + 1, :n].contiguous(),
                                    q2k[b:b + 1], causal=True)
        _assert_close(o[b * Sq:(b + 1) * Sq], l[b * Sq:(b + 1) * Sq], ob, lb, tol=1e-12)


def test_paged_all_blocks_equals_dense_causal_attention():
    B, Sq, L, Hkv, qpk = 2, 8, 512, 1, 4
    Hq = Hkv * qpk
    q, k, v = _rand_inputs(B, Sq, L, Hkv, qpk)
    pt = synth.shuffled_page_table(B, L // 128, seed=4)
    seqused = torch.tensor([L, L - 100], dtype=torch.int32)
    q2k = torch.arange(4, dtype=torch.int32).expand(B, Hkv, Sq, 4).contiguous()
    o, l = oracle.sparse_attn_paged(q.reshape(B * Sq, Hq, 128), _to_pool(k, pt), _to_pool(v, pt), pt,
                                    seqused, q2k, causal=True)
    o_ref, l_ref = _dense_reference(q, k, v, causal=True, kv_len=seqused.tolist())
    _assert_close(o, l, o_ref, l_ref)


# ---------------------------------------------------------------------------
# CSR
# ---------------------------------------------------------------------------

def _csr_brute(q2k: np.ndarray, Skv, blk=128, seqused=None):
    B, Hkv, Sq, topk = q2k.shape
    nblk = -(-Skv // blk)
    out = {}
    for h in range(Hkv):
        rows = [[] for _ in range(B * nblk)]
        for b in range(B):
            kv = Skv if seqused is None else int(seqused[b])
            nvalid = min(nblk, -(-kv // blk))
            for s in range(Sq):
                seen = []
                for t in range(topk):
                    j = int(q2k[b, h, s, t])
                    if 0 <= j < nvalid and j not in seen:
                        rows[b * nblk + j].append((b * Sq + s, len(seen)))
                        seen.append(j)
        out[h] = rows
    return out


@pytest.mark.parametrize("case", ["sink", "perm", "messy"])
def test_csr_matches_brute_force(case):
    if case == "sink":
        B, Hkv, Sq, Skv, topk = 2, 2, 300, 640, 8
        q2k = synth.q2k_causal_sink(B, Hkv, Sq, Skv, topk, seed=1).numpy()
        seqused = None
    elif case == "perm":
        B, Hkv, Sq, Skv, topk = 1, 3, 77, 1024, 4
        q2k = synth.q2k_perm_prefix(B, Hkv, Sq, 8, topk, seed=2).numpy()
        seqused = None
    else:  # duplicates, out-of-range ids, negative ids, seqused trimming
        B, Hkv, Sq, Skv, topk = 2, 1, 50, 512, 6
        rng = np.random.default_rng(0)
        q2k = rng.integers(-3, 6, size=(B, Hkv, Sq, topk)).astype(np.int32)
        seqused = np.array([512, 200], dtype=np.int32)
    c = oracle.build_k2q_csr(q2k, Skv, seqused=seqused)
    ref = _csr_brute(q2k, Skv, seqused=seqused)
    cap = B * Sq * topk
    for h in range(Hkv):
        rows = ref[h]
        counts = [len(r) for r in rows]
        assert c["row_ptr"][h].tolist() == [0] + list(np.cumsum(counts))
        flat = [qq for r in rows for (qq, _) in r]
        nnz = len(flat)
        assert c["q_indices"][h, :nnz].tolist() == flat
        assert (c["q_indices"][h, nnz:] == -1).all() and (c["qsplit"][h, nnz:] == -1).all()
        packed = [qq | (rk << 24) for r in rows for (qq, rk) in r]
        assert c["qsplit"][h, :nnz].tolist() == packed
        # each query's split ids are 0..count-1 and count matches split_counts
        per_q = {}
        for qq, rk in [x for r in rows for x in r]:
            per_q.setdefault(qq, []).append(rk)
        for qq in range(B * Sq):
            got = sorted(per_q.get(qq, []))
            assert got == list(range(len(got)))
            assert c["split_counts"][qq, h] == len(got)
        assert c["q_indices"].shape[1] == cap


# ---------------------------------------------------------------------------
# NVFP4
# ---------------------------------------------------------------------------

def _golden_e2m1():
    tab = {}
    with open(os.path.join(GOLDEN, "e2m1_table.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            c, v = line.split()
            tab[int(c)] = float(v)
    return tab


def test_e2m1_decode_matches_table_on_the_pages():
    for c, v in _golden_e2m1().items():
        assert oracle.e2m1_decode(c) == v


def test_e4m3_decode_matches_torch_float8_e4m3fn():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got)
        else:
            assert got == ref[c], c


def test_e4m3_encode_matches_torch_rounding_in_range():
    g = torch.Generator().manual_seed(1)
    x = torch.cat([torch.rand(4000, generator=g, dtype=torch.float64) * 448,
                   torch.rand(4000, generator=g, dtype=torch.float64) * 0.05,
                   torch.tensor([0.0, 2 ** -10, 2 ** -9 * 1.5, 2 ** -9 * 2.5, 447.9, 448.0, 1.0625, 1.1875])])
    x32 = x.float()   # the quantiser rounds binary32 quotients
    ref = x32.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for xi, r in zip(x32.double().tolist(), ref.tolist()):
        assert oracle.e4m3_encode(xi) == r, xi


def test_nvfp4_quantiser_choices_are_nearest_even_by_brute_force():
    x = synth.normal_bf16((64, 128), 5, synth.STREAM_AUX)
    x[0, :16] = 0                          # all-zero group
    x[1, :16] = torch.linspace(-6, 6, 16)  # exact grid points after scaling
    packed, scales = oracle.nvfp4_quantize(x)
    xf = _f64(x)
    e4 = np.array([oracle.e4m3_decode(c) for c in range(256)])
    e2 = np.array([oracle.e2m1_decode(c) for c in range(16)])
    for r in range(64):
        for gi in range(8):
            grp = xf[r, gi * 16:(gi + 1) * 16]
            amax = np.float32(np.abs(grp).max())
            target = float(np.float32(amax) / np.float32(6.0))
            sc = scales[r, gi]
            # nearest e4m3 (finite, >= 0); ties to even code
            cand = [(abs(e4[c] - target), c & 1, c) for c in range(0x7F) if not math.isnan(e4[c])]
            best = min(cand)[2]
            assert e4[sc] == e4[best], (r, gi)
            s = np.float32(e4[sc])
            for i in range(16):
                byte = packed[r, (gi * 16 + i) // 2]
                code = (byte >> 4) if i & 1 else (byte & 0xF)
                if s == 0:
                    assert code == 0
                    continue
                y = float(np.float32(grp[i]) / s)
                mags = [(abs(abs(y) - e2[c]), c & 1, c) for c in range(8)]
                want = min(mags)[2] if abs(y) < 6 else 7
                assert (code & 7) == want, (r, gi, i, y)
                if want:
                    assert (code >> 3) == (1 if y < 0 else 0)


def test_nvfp4_dequant_is_exact_product_and_close_to_input():
    x = synth.normal_bf16((32, 128), 6, synth.STREAM_AUX)
    packed, scales = oracle.nvfp4_quantize(x)
    deq = oracle.nvfp4_dequantize(packed, scales)
    xh = oracle.bf16_bits_to_float64(deq)
    e4 = np.array([oracle.e4m3_decode(c) for c in range(256)])
    e2 = np.array([oracle.e2m1_decode(c) for c in range(16)])
    for r in range(32):
        for i in range(128):
            byte = packed[r, i // 2]
            code = (byte >> 4) if i & 1 else (byte & 0xF)
            assert xh[r, i] == e2[code] * e4[scales[r, i // 16]]
    # relative to the group's amax, the e2m1 grid error is at most 1/6 + scale rounding
    xf = _f64(x)
    for r in range(32):
        for gi in range(8):
            a = np.abs(xf[r, gi * 16:(gi + 1) * 16]).max()
            err = np.abs(xf[r, gi * 16:(gi + 1) * 16] - xh[r, gi * 16:(gi + 1) * 16]).max()
            assert err <= a * (1 / 6 + 1 / 16) + 1e-12


def test_supported_shape_sets_on_the_pages():
    with open(os.path.join(GOLDEN, "supported_shapes.txt")) as f:
        sets = {ln.split()[0]: [int(x) for x in ln.split()[1:]] for ln in f if ln.strip() and not ln.startswith("#")}
    assert sets["topk"] == [4, 8, 16, 32]
    assert sets["qhead_per_kv"] == [1, 2, 4, 8, 16]
    assert sets["head_dim"] == [128]
