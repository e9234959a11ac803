// attn_mma.cuh -- warp-level bf16 MMA helpers (mma.sync m16n8k16, ldmatrix) on
// XOR-swizzled 128 x 128 bf16 shared-memory tiles (row = 256 B = 16 chunks of
// 16 B; chunk c of row r is stored at chunk c ^ (r & 7)).
#pragma once
#include "common.cuh"

namespace msa {

__device__ __forceinline__ uint32_t swz_off(int row, int chunk) {
    return (uint32_t)(row * 256 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// max of three floats in one instruction (sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// S[16 x 128] = Q_rows[16 x 128] . K[128 x 128]^T for the warp's 16 query
// rows starting at `row0` of the Q tile; acc[nt][4] in the m16n8 C layout.
__device__ __forceinline__ void warp_qk(uint32_t q_base, uint32_t k_base, int row0, float (&acc)[16][4]) {
    int lane = threadIdx.x & 31;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t a0, a1, a2, a3;
        int arow = row0 + (lane & 15);
        int achunk = 2 * kk + (lane >> 4);
        ldsm_x4(q_base + swz_off(arow, achunk), a0, a1, a2, a3);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            uint32_t b0, b1, b2, b3;
            int brow = np * 16 + (lane & 7) + ((lane >> 4) << 3);
            int bchunk = 2 * kk + ((lane >> 3) & 1);
            ldsm_x4(k_base + swz_off(brow, bchunk), b0, b1, b2, b3);
            mma_bf16(acc[2 * np], a0, a1, a2, a3, b0, b1);
            mma_bf16(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
    }
}

// O[16 x 128] += P[16 x 128 keys] . V[128 keys x 128 d]; P given as the S
// accumulator layout already converted to bf16 pairs: pk[nt][0] = row g,
// pk[nt][1] = row g + 8 (keys 8nt + 2t, +1).
__device__ __forceinline__ void warp_pv(uint32_t v_base, const uint32_t (&pk)[16][2], float (&o)[16][4]) {
    int lane = threadIdx.x & 31;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t a0 = pk[2 * kk][0], a1 = pk[2 * kk][1], a2 = pk[2 * kk + 1][0], a3 = pk[2 * kk + 1][1];
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
            uint32_t b0, b1, b2, b3;
            int vrow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            int vchunk = 2 * dp + (lane >> 4);
            ldsm_x4_t(v_base + swz_off(vrow, vchunk), b0, b1, b2, b3);
            mma_bf16(o[2 * dp], a0, a1, a2, a3, b0, b1);
            mma_bf16(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
        }
    }
}

// Byte offset of 16-byte chunk c (0..15) of row r in a TMA tile stored as two
// 128-byte-swizzled half tiles [2][128 rows][128 B] (1024-byte aligned base).
__device__ __forceinline__ uint32_t tma_tile_off(int row, int chunk) {
    return (uint32_t)((chunk >> 3) * 16384 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// A fragments (m16n8k16 layout) of 16 query rows x 128 dims read straight
// from global memory: qf[kk] = {a0, a1, a2, a3} of k-step kk.  row_g and
// row_g8 point at the rows of this thread's groupID and groupID + 8 (or are
// null for rows that do not exist, which read as zero).
__device__ __forceinline__ void load_q_frags(const __nv_bfloat16 *row_g, const __nv_bfloat16 *row_g8,
                                             uint32_t (&qf)[8][4]) {
    const int t = threadIdx.x & 3;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const int col = kk * 16 + 2 * t;
        qf[kk][0] = row_g ? *reinterpret_cast<const uint32_t *>(row_g + col) : 0u;
        qf[kk][1] = row_g8 ? *reinterpret_cast<const uint32_t *>(row_g8 + col) : 0u;
        qf[kk][2] = row_g ? *reinterpret_cast<const uint32_t *>(row_g + col + 8) : 0u;
        qf[kk][3] = row_g8 ? *reinterpret_cast<const uint32_t *>(row_g8 + col + 8) : 0u;
    }
}

// S[16 x 128] = Q (register fragments) . K^T with K in a TMA half-tile pair.
__device__ __forceinline__ void warp_qk_tma(const uint32_t (&qf)[8][4], uint32_t k_base, float (&acc)[16][4]) {
    int lane = threadIdx.x & 31;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            uint32_t b0, b1, b2, b3;
            int brow = np * 16 + (lane & 7) + ((lane >> 4) << 3);
            int bchunk = 2 * kk + ((lane >> 3) & 1);
            ldsm_x4(k_base + tma_tile_off(brow, bchunk), b0, b1, b2, b3);
            mma_bf16(acc[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
            mma_bf16(acc[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
        }
    }
}

// S[16 x 128] = Q . K^T with Q in a warp-private XOR-swizzled 16-row tile
// (swz_off layout) and K in a TMA half-tile pair.
__device__ __forceinline__ void warp_qk_qs_tma(uint32_t q_base, uint32_t k_base, float (&acc)[16][4]) {
    int lane = threadIdx.x & 31;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(q_base + swz_off(lane & 15, 2 * kk + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            uint32_t b0, b1, b2, b3;
            int brow = np * 16 + (lane & 7) + ((lane >> 4) << 3);
            int bchunk = 2 * kk + ((lane >> 3) & 1);
            ldsm_x4(k_base + tma_tile_off(brow, bchunk), b0, b1, b2, b3);
            mma_bf16(acc[2 * np], a0, a1, a2, a3, b0, b1);
            mma_bf16(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
    }
}

// Half-block forms: keys [64*kh, 64*kh + 64) only.
__device__ __forceinline__ void warp_qk_qs_tma_half(uint32_t q_base, uint32_t k_base, int kh, float (&acc)[8][4]) {
    int lane = threadIdx.x & 31;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(q_base + swz_off(lane & 15, 2 * kk + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t b0, b1, b2, b3;
            int brow = kh * 64 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
            int bchunk = 2 * kk + ((lane >> 3) & 1);
            ldsm_x4(k_base + tma_tile_off(brow, bchunk), b0, b1, b2, b3);
            mma_bf16(acc[2 * np], a0, a1, a2, a3, b0, b1);
            mma_bf16(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
    }
}
__device__ __forceinline__ void warp_pv_tma_half(uint32_t v_base, int kh, const uint32_t (&pk)[8][2],
                                                 float (&o)[16][4]) {
    int lane = threadIdx.x & 31;
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {
        const int kk = kh * 4 + kq;
        uint32_t a0 = pk[2 * kq][0], a1 = pk[2 * kq][1], a2 = pk[2 * kq + 1][0], a3 = pk[2 * kq + 1][1];
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
            uint32_t b0, b1, b2, b3;
            int vrow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            int vchunk = 2 * dp + (lane >> 4);
            ldsm_x4_t(v_base + tma_tile_off(vrow, vchunk), b0, b1, b2, b3);
            mma_bf16(o[2 * dp], a0, a1, a2, a3, b0, b1);
            mma_bf16(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
        }
    }
}

// O[16 x 128] += P . V with V in a TMA half-tile pair.
__device__ __forceinline__ void warp_pv_tma(uint32_t v_base, const uint32_t (&pk)[16][2], float (&o)[16][4]) {
    int lane = threadIdx.x & 31;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t a0 = pk[2 * kk][0], a1 = pk[2 * kk][1], a2 = pk[2 * kk + 1][0], a3 = pk[2 * kk + 1][1];
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
            uint32_t b0, b1, b2, b3;
            int vrow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            int vchunk = 2 * dp + (lane >> 4);
            ldsm_x4_t(v_base + tma_tile_off(vrow, vchunk), b0, b1, b2, b3);
            mma_bf16(o[2 * dp], a0, a1, a2, a3, b0, b1);
            mma_bf16(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
        }
    }
}

// e4m3 (fn) byte -> float, exact.
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
    uint32_t e = (b >> 3) & 0xF, m = b & 7;
    float v = (e == 0) ? (float)m * (1.0f / 512.0f) : __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (b & 0x80) ? -v : v;
}

// e2m1 code (4 bits) -> float.
__device__ __forceinline__ float e2m1_to_float(uint32_t c) {
    // magnitudes 0, .5, 1, 1.5 (m < 4) and 2, 3, 4, 6 (m >= 4)
    const uint32_t m = c & 7;
    float v = (m < 4) ? 0.5f * (float)m : (float)(1u << ((m >> 1) - 1)) * (1.0f + 0.5f * (float)(m & 1));
    return (c & 8) ? -v : v;
}

// e4m3 byte -> its value as bf16 in both halves of a word.  The seven
// magnitude bits placed at bit 20 of an f32 (exponent field low four bits,
// mantissa top three) read as 2^-120 times the e4m3 value, subnormal codes
// included, so one exact multiply by 2^120 gives the value; it has at most
// four significant bits, so the bf16 truncation is exact too.
__device__ __forceinline__ uint32_t e4m3_to_bf16x2(uint32_t b) {
    const float f = __uint_as_float(((b & 0x7Fu) << 20) | ((b & 0x80u) << 24)) * 0x1p120f;
    const uint32_t h = __float_as_uint(f) >> 16;
    return h | (h << 16);
}

// Eight e2m1 codes (code i in nibble i of x) -> eight bf16, element 2i in the
// low half of w[i].  The bf16 bytes of the eight magnitudes {0, .5, 1, 1.5, 2,
// 3, 4, 6} are two byte tables (low bytes 00 00 80 c0 00 40 80 c0, high bytes
// 00 3f 3f 3f 40 40 40 40) that one byte permute each looks up for four codes
// at a time; two more permutes interleave low and high bytes, and the codes'
// sign bits (bit 3 of each nibble) become the bf16 sign bits.  Integer ops
// only: nothing on the special-function pipe the softmax uses.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t x, uint32_t (&w)[4]) {
    const uint32_t mag = x & 0x77777777u, sg = x & 0x88888888u;
    const uint32_t lo03 = __byte_perm(0xC0800000u, 0xC0804000u, mag);
    const uint32_t hi03 = __byte_perm(0x3F3F3F00u, 0x40404040u, mag);
    const uint32_t lo47 = __byte_perm(0xC0800000u, 0xC0804000u, mag >> 16);
    const uint32_t hi47 = __byte_perm(0x3F3F3F00u, 0x40404040u, mag >> 16);
    w[0] = __byte_perm(lo03, hi03, 0x5140) | ((sg << 12) & 0x8000u) | ((sg << 24) & 0x80000000u);
    w[1] = __byte_perm(lo03, hi03, 0x7362) | ((sg << 4) & 0x8000u) | ((sg << 16) & 0x80000000u);
    w[2] = __byte_perm(lo47, hi47, 0x5140) | ((sg >> 4) & 0x8000u) | ((sg << 8) & 0x80000000u);
    w[3] = __byte_perm(lo47, hi47, 0x7362) | ((sg >> 12) & 0x8000u) | (sg & 0x80000000u);
}

// bf16x2 product, round to nearest (exact for e2m1 x e4m3: at most six
// significant bits).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 32 NVFP4 values (16 packed bytes, two groups of 16) and their two e4m3
// scales (low byte: first group) -> 32 bf16 in four 16-byte chunks.
__device__ __forceinline__ void nvfp4_piece_to_bf16(uint4 packed, uint32_t scales2, uint4 (&out)[4]) {
    const uint32_t s0 = e4m3_to_bf16x2(scales2 & 0xFFu), s1 = e4m3_to_bf16x2((scales2 >> 8) & 0xFFu);
    const uint32_t words[4] = {packed.x, packed.y, packed.z, packed.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t w[4];
        e2m1x8_to_bf16(words[c], w);
        const uint32_t s = c < 2 ? s0 : s1;
        out[c] = make_uint4(bf16x2_mul(w[0], s), bf16x2_mul(w[1], s), bf16x2_mul(w[2], s), bf16x2_mul(w[3], s));
    }
}

// Two e4m3 values (low 16 bits of x, first value in the low byte) -> f16x2,
// exactly (every e4m3 value, subnormals included, is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t x) {
    uint32_t d;
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n" : "=r"(d) : "r"(x));
    return d;
}

// 16 e4m3 values (16 bytes, first value in the lowest byte) -> 16 bf16 in two
// 16-byte chunks, exactly (at most four significant bits each).
__device__ __forceinline__ void e4m3x16_to_bf16(uint4 v, uint4 (&out)[2]) {
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t f = e4m3x2_to_f16x2(words[i] >> (16 * h));
            const float2 g = __half22float2(*reinterpret_cast<const __half2 *>(&f));
            w[2 * i + h] = pack_bf16x2(g.x, g.y);
        }
    }
    out[0] = make_uint4(w[0], w[1], w[2], w[3]);
    out[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Stages 128 token rows of e4m3 values (128 bytes each, row t at src + t *
// row_stride) as bf16 into a 128-byte-swizzled tile [2 column halves][128
// rows][128 B] at shared address `tile` (halves 16384 bytes apart), exactly;
// rows t >= nrows are zero.  One warp: lane l converts the 16-byte piece l % 8
// (values 16 (l % 8) .. + 15: column half (l % 8) / 4) of rows l / 8 + 4 i,
// with eight loads in flight before any is used.
__device__ __forceinline__ void e4m3_rows_to_tile(uint32_t tile, const uint8_t *src, int64_t row_stride, int nrows,
                                                  int lane) {
    const int pc = lane & 7, r0 = lane >> 3;
    const uint32_t half = tile + (uint32_t)(pc >> 2) * 16384u;
#pragma unroll 1
    for (int rb = r0; rb < 128; rb += 32) {
        uint4 pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = rb + 4 * i;
            pk[i] = r < nrows ? __ldg(reinterpret_cast<const uint4 *>(src + (int64_t)r * row_stride) + pc)
                              : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint4 o4[2];
            e4m3x16_to_bf16(pk[i], o4);
            const int r = rb + 4 * i;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int ch = (pc & 3) * 2 + c;  // 16-byte chunk of the 128-byte row
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(half + (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4))),
                             "r"(o4[c].x), "r"(o4[c].y), "r"(o4[c].z), "r"(o4[c].w));
            }
        }
    }
}

}  // namespace msa
