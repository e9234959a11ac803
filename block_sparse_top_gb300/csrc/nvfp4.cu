// nvfp4.cu -- NVFP4 encoder for K/V rows: per group of 16 values along D,
// scale = e4m3_rne_satfinite(amax / 6) and code = e2m1_rne_satfinite(x / scale)
// (both quotients binary32), e2m1 element 2i in the low nibble.
//
// Source: interface.py sparse_atten_nvfp4_kv_func docstring (e2m1 data two per
// byte, one e4m3 scale per 16 elements along D) and the vLLM sparse-MLA test
// page (_E2M1_TABLE {0,.5,1,1.5,2,3,4,6}, sign in bit 3, low nibble first).
#include <cuda_fp8.h>

#include "attn_mma.cuh"

namespace msa {
namespace {

// |y| -> e2m1 magnitude code, round to nearest, ties to the even code,
// saturating at 6 (code 7).  Midpoints: .25 .75 1.25 1.75 2.5 3.5 5.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
    float a = fabsf(y);
    uint32_t c = (a <= 0.25f) ? 0u
               : (a < 0.75f)  ? 1u
               : (a <= 1.25f) ? 2u
               : (a < 1.75f)  ? 3u
               : (a <= 2.5f)  ? 4u
               : (a < 3.5f)   ? 5u
               : (a <= 5.0f)  ? 6u
                              : 7u;
    return (y < 0.f) ? (c | 8u) : c;
}

__global__ void nvfp4_quantize_kernel(const __nv_bfloat16 *__restrict__ x, int64_t groups, int gpr,
                                      uint8_t *__restrict__ packed, uint8_t *__restrict__ scales) {
    int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gi >= groups) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + gi * 16);
    uint4 a = src[0], b = src[1];
    uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_lo(w[i]);
        v[2 * i + 1] = bf16_hi(w[i]);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    float q6 = __fdiv_rn(amax, 6.0f);
    __nv_fp8_storage_t sb = __nv_cvt_float_to_fp8(q6, __NV_SATFINITE, __NV_E4M3);
    float sf = e4m3_to_float((uint32_t)sb);
    uint32_t out[2] = {0u, 0u};
    if (sf > 0.f) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            uint32_t c = e2m1_code(__fdiv_rn(v[i], sf));
            out[i >> 3] |= c << (4 * (i & 7));
        }
    }
    *reinterpret_cast<uint2 *>(packed + gi * 8) = make_uint2(out[0], out[1]);
    scales[gi] = (uint8_t)sb;
    (void)gpr;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" int msa_nvfp4_quantize(const void *x, int64_t rows, int D, uint8_t *packed, uint8_t *scales,
                                  cudaStream_t stream) {
    if (!x || !packed || !scales || rows < 0 || D <= 0 || D % 16) return MSA_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(packed, 8)) return MSA_ERR_INVALID_ARG;
    if (rows == 0) return MSA_OK;
    int64_t groups = rows * (D / 16);
    int threads = 256;
    int64_t blocks = ceil_div(groups, threads);
    nvfp4_quantize_kernel<<<(unsigned)blocks, threads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(x), groups,
                                                                     D / 16, packed, scales);
    MSA_LAUNCH_CHECK();
    return MSA_OK;
}
