// common.cuh -- shared device/host helpers of libmsa (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa.h"

#define MSA_CUDA_TRY(expr)                                  \
    do {                                                    \
        cudaError_t _e = (expr);                            \
        if (_e != cudaSuccess) return MSA_ERR_CUDA;         \
    } while (0)

#define MSA_LAUNCH_CHECK()                                  \
    do {                                                    \
        if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA; \
    } while (0)

namespace msa {

constexpr int kBlk = 128;      // KV block = page = 128 tokens
constexpr int kD = 128;        // head dimension
constexpr int kMaxNblk = 8192; // CSR builder bitmap limit (blocks per sequence)

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool supported_topk(int t) { return t == 4 || t == 8 || t == 16 || t == 32; }
inline bool supported_qpk(int q) { return q == 1 || q == 2 || q == 4 || q == 8 || q == 16; }
inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device status word (OR of MSA_STATUS_* bits); tolerates a null pointer.
__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

// Programmatic dependent launch.  A kernel launched by launch_pdl may be
// scheduled while the previous kernel on its stream is still finishing: it
// runs its prologue (barrier set-up, tensor-memory allocation), then
// grid_dependency_wait() blocks until the previous kernel has completed and
// its writes are visible, so nothing that kernel produces may be read, and
// nothing it reads may be written, before that call (a kernel launched the
// ordinary way returns from it at once).  grid_dependents_launch() lets the
// next kernel on the stream be scheduled in the same way.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              A &&...args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<A &&>(args)...);
}

// ---------------------------------------------------------------------------
// Work plan shared by the CSR builder (writer) and the prefill kernel (reader)
// ---------------------------------------------------------------------------
// A unit is (KV head, KV block blk of sequence seq, first q_indices position,
// query count); its queries are processed in chunks of 128/qhead_per_kv
// queries, 128 rows each.
struct PlanHeader {
    int32_t work_count;  // units written (device side, no host readback)
    int32_t capacity;    // units the buffer holds
    int32_t qhead_per_kv;
    int32_t q_per_unit;
    int32_t wave_queries;  // queries per wave (units run head-major, then wave-major)
    int32_t nwaves;
    int32_t reserved[10];
};
static_assert(sizeof(PlanHeader) == 64, "plan header is 64 bytes");

struct PlanUnit {
    int16_t head;   // KV head h
    int16_t blk;    // KV block j within the sequence (tokens 128 j ..)
    int32_t seq;    // sequence b
    int32_t start;  // first position in q_indices[h]
    int32_t count;  // queries in this unit
};
static_assert(sizeof(PlanUnit) == 16, "plan unit is 16 bytes");
constexpr int kMaxHkv = 32767;  // KV heads a plan unit can name

inline int q_per_chunk(int qpk) { return 128 / qpk; }
// Queries per unit (its K/V block is loaded once for all its chunks): 8
// chunks for qhead_per_kv >= 8, 16 below, where a chunk holds 32 or more
// queries, units are few per block and a dequantised (NVFP4, e4m3) block is
// converted once per unit.  Tile times against 8 chunks: 32K qpk 16 +1 %,
// 48K qpk 16 +3 % at 16 chunks; 384K qpk 2 bf16 -3.4 %, NVFP4 -20 %.
inline int q_per_unit(int qpk) { return (qpk >= 8 ? 8 : 16) * q_per_chunk(qpk); }

// Queries per wave.  Units run head-major, then wave by wave, and a unit never
// crosses a wave, so W trades the reach of the queries the CTAs read at one
// time against unit length (a unit's K/V block is loaded once for all its
// chunks).  W is sized by the split partials one (KV head, wave) pass writes
// -- W * qhead_per_kv * topk rows of D bf16 plus two floats -- at about 512
// MiB for qhead_per_kv >= 8 (on the 32K causal workload the tiles took 2.263
// ms at 256 MiB, 2.246 at 512, 2.255 at 1024, 2.277 at 2048) and 2048 MiB for
// qhead_per_kv <= 4, whose chunks hold 32 or more queries and whose units are
// short (the 384K qhead_per_kv 2 workload: 0.173 -> 0.181 of peak in bf16,
// 0.117 -> 0.132 with NVFP4 K/V, against 512 MiB).
inline int64_t wave_queries(int64_t total_q, int qpk, int topk) {
    const int64_t per_q = (int64_t)qpk * topk * (kD * 2 + 8);
    const int64_t budget = (int64_t)(qpk >= 8 ? 512 : 2048) << 20;
    int64_t w = ((budget / per_q) + 64) / 128 * 128;  // nearest multiple of 128
    if (w < 128) w = 128;
    return w > total_q ? total_q : w;
}
inline int64_t num_waves(int64_t total_q, int qpk, int topk) {
    return ceil_div(total_q, wave_queries(total_q, qpk, topk));
}

// Units of a plan over `rows` CSR rows per KV head and total_q queries: every
// (head, row, wave) segment adds at most one partial unit.
inline int64_t plan_capacity(int64_t rows, int64_t total_q, int Hkv, int topk, int qpk) {
    const int64_t nnz = total_q * topk;
    int64_t segs = rows * num_waves(total_q, qpk, topk);
    if (segs > nnz) segs = nnz;
    const int64_t per_head = segs + ceil_div(nnz, q_per_unit(qpk));
    return per_head * Hkv;
}

// ---------------------------------------------------------------------------
// bf16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared async copy (L2 only), optionally zero-filled.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid = true) {
    int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
// 4-byte global->shared async copy (through L1).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

}  // namespace msa
