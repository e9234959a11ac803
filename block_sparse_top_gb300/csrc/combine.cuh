// combine.cuh -- split partial layout (written by the tile kernel, read by
// the LSE combine) and the merge of one output piece.
//
// A (query, KV head) pair is a group g = gq * Hkv + h; its split partials are
// contiguous:
//   o_part    [B*Sq][Hkv][topk][D/8][qhead_per_kv][8] of the partial type
//             (bf16 by default, fp16 or fp32 on request), the unnormalised
//             U_s = sum_k exp(scale (s_k - m_s)) v_k of split s, m_s its
//             reference max (the first half-row's max unless the second
//             exceeds it by more than the tile kernel's bound);
//   stat_part [B*Sq][Hkv][topk][qhead_per_kv] float2 (a_s = scale m_s, l_s).
// Split s alone normalises to U_s / l_s with lse_s = a_s + ln l_s, so
//   LSE = logsumexp_s lse_s = A + ln sum_s l_s exp(a_s - A)      (A = max a_s)
//   O   = sum_s exp(lse_s - LSE) U_s / l_s = sum_s exp(a_s - A) U_s / sum_s l_s exp(a_s - A)
// (interface.py _sparse_atten_csr_varlen_forward: per-split O and LSE merged
// by LSE; test_sparse_atten.py sparse_attention_ref: a row with no visible key
// has O = 0 and LSE = -inf).  A split with a non-finite a_s has weight 0.
#pragma once
#include "common.cuh"

namespace msa {

// Bytes of one stored piece (8 values): bf16 and fp16 partials 16, fp32 32.
__host__ __device__ inline int part_piece_bytes(int part_dtype) { return part_dtype == MSA_PARTIAL_FP32 ? 32 : 16; }

__host__ __device__ inline int64_t part_o_index(int64_t grp, int topk, int qpk, int split, int c, int j) {
    return ((grp * topk + split) * 16 + c) * qpk + j;  // in pieces
}
__host__ __device__ inline int64_t part_stat_index(int64_t grp, int topk, int qpk, int split, int j) {
    return (grp * topk + split) * qpk + j;
}

// One stored piece of partial type PD (MSA_PARTIAL_*): raw words and their 8 values.
template <int PD>
struct PartPiece {
    uint4 w[PD == MSA_PARTIAL_FP32 ? 2 : 1];
    __device__ __forceinline__ void load(const char *p, bool smem) {
        const uint4 *q = reinterpret_cast<const uint4 *>(p);
#pragma unroll
        for (int i = 0; i < (PD == MSA_PARTIAL_FP32 ? 2 : 1); ++i) w[i] = smem ? q[i] : __ldcs(q + i);
    }
    __device__ __forceinline__ float val(int i) const {
        if (PD == MSA_PARTIAL_FP32) {
            const uint4 &u = w[i >> 2];
            const uint32_t x = (i & 3) == 0 ? u.x : (i & 3) == 1 ? u.y : (i & 3) == 2 ? u.z : u.w;
            return __uint_as_float(x);
        }
        const uint32_t x = (i >> 1) == 0 ? w[0].x : (i >> 1) == 1 ? w[0].y : (i >> 1) == 2 ? w[0].z : w[0].w;
        if (PD == MSA_PARTIAL_FP16) {
            const __half2 h = *reinterpret_cast<const __half2 *>(&x);
            return (i & 1) ? __high2float(h) : __low2float(h);
        }
        return (i & 1) ? bf16_hi(x) : bf16_lo(x);
    }
};

// Merges the first n of topk splits of piece (group grp, 8-dim chunk c, head j
// of the group) into out (8 bf16) and lse_out.  Every load of a batch of BATCH
// splits is issued before any is used (only the first n slots are read);
// batches merge online with a running max.  SMEM: the
// group's partials and statistics were staged in shared memory (o_part and
// stat_part point at the copy, grp 0).  PD: the partials' storage type.
template <int MAXS, int PD, int BATCH = 16, bool SMEM = false>
__device__ __forceinline__ void combine_piece(const void *__restrict__ o_part, const float2 *__restrict__ stat_part,
                                              int64_t grp, int n, int topk, int qpk, int c, int j, uint4 &out,
                                              float &lse_out) {
    constexpr int PB = PD == MSA_PARTIAL_FP32 ? 32 : 16;
    const char *src = static_cast<const char *>(o_part) + part_o_index(grp, topk, qpk, 0, c, j) * PB;
    const float2 *st = stat_part + part_stat_index(grp, topk, qpk, 0, j);
    const int64_t o_stride = 16 * (int64_t)qpk * PB;
    float mx = -INFINITY, den = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int s0 = 0; s0 < (MAXS < n ? MAXS : n); s0 += BATCH) {
        PartPiece<PD> v[BATCH];
        float2 sv[BATCH];
#pragma unroll
        for (int t = 0; t < BATCH; ++t)
            if (s0 + t < n) v[t].load(src + (s0 + t) * o_stride, SMEM);
#pragma unroll
        for (int t = 0; t < BATCH; ++t)
            sv[t] = (s0 + t < n) ? (SMEM ? st[(s0 + t) * qpk] : __ldg(st + (int64_t)(s0 + t) * qpk))
                                 : make_float2(-INFINITY, 0.f);
        float bm = mx;
#pragma unroll
        for (int t = 0; t < BATCH; ++t)
            if (isfinite(sv[t].x)) bm = fmaxf(bm, sv[t].x);
        if (bm > mx) {
            const float r = __expf(mx - bm);  // 0 when mx is -inf
            den *= r;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] *= r;
            mx = bm;
        }
#pragma unroll
        for (int t = 0; t < BATCH; ++t) {
            if (!isfinite(sv[t].x)) continue;
            const float e = __expf(sv[t].x - mx);
            den += e * sv[t].y;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += e * v[t].val(i);
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    out.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    out.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    lse_out = den > 0.f ? mx + logf(den) : -INFINITY;
}

// Temperature LSE of (group grp, head j) from its first n splits' temperature
// statistics (a_s = m_s scale / T, l_s = sum 2^(x / T)): the logsumexp of
// a_s + ln l_s, -inf when no split has a finite a_s.
__device__ __forceinline__ float combine_lse_temp(const float2 *__restrict__ stat_temp, int64_t grp, int n, int topk,
                                                  int qpk, int j) {
    const float2 *st = stat_temp + part_stat_index(grp, topk, qpk, 0, j);
    float mx = -INFINITY;
    for (int s = 0; s < n; ++s) {
        const float a = __ldg(st + (int64_t)s * qpk).x;
        if (isfinite(a)) mx = fmaxf(mx, a);
    }
    if (mx == -INFINITY) return -INFINITY;
    float den = 0.f;
    for (int s = 0; s < n; ++s) {
        const float2 v = __ldg(st + (int64_t)s * qpk);
        if (isfinite(v.x)) den += v.y * __expf(v.x - mx);
    }
    return den > 0.f ? mx + logf(den) : -INFINITY;
}

}  // namespace msa
