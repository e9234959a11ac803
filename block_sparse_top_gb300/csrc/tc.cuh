// tc.cuh -- Blackwell (sm_100 family, built for sm_103a) building blocks in
// inline PTX: mbarriers with bounded waits, TMA tiled loads, tcgen05 tensor
// memory allocation, MMA (A from shared memory or tensor memory), commit and
// tensor-memory loads/stores.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace msa {
namespace tc {

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(addr), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t addr) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(addr) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t addr, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(addr), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// L2 prefetch of the 128-byte line holding `p`.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}

// Non-blocking probe of an mbarrier phase (for a thread that polls several).
__device__ __forceinline__ bool mbar_test(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits are bounded in time: a wait that has not completed within
// kWaitLimitNs of the device's global nanosecond timer gives up.  (A test
// build of the library sets a short limit to check the abort path.)
#ifdef MSA_TEST_WAIT_LIMIT_NS
constexpr uint64_t kWaitLimitNs = MSA_TEST_WAIT_LIMIT_NS;
#else
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second
#endif
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Bounded wait: gives up after kWaitLimitNs, raises the CTA abort flag and
// the device status bit so every role can drain and exit; returns false at
// once when another role has raised the abort flag.
// The polling loop of mbar_wait, out of line: a wait that does not complete at
// its first try costs far more than the call, and every call site stays small.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t addr, uint32_t parity, volatile int *abort_flag,
                                                   uint32_t *status, uint32_t status_bit) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(addr, parity)) return true;
        if ((i & 63u) == 0u) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > kWaitLimitNs) break;
        }
    }
    *abort_flag = 1;
    set_status(status, status_bit);
    return false;
}
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity, volatile int *abort_flag, uint32_t *status,
                                          uint32_t status_bit) {
    if (mbar_try_wait(addr, parity)) return true;
    return mbar_wait_slow(addr, parity, abort_flag, status, status_bit);
}

// cp.async completion tracked by an mbarrier (no-increment arrive).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t addr) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(addr) : "memory");
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t mbar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
        "[%2];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t mbar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];\n" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar), "r"(c0), "r"(c1)
        : "memory");
}
// Four rows r0..r3 (box one row high) at column c0 into four consecutive
// 128-byte rows of shared memory.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap *map, uint32_t mbar, int c0, int r0,
                                            int r1, int r2, int r3) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4, %5, %6, %7}], [%2];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
        : "memory");
}
// L2 policy that keeps lines resident (evict last); used for data a CTA
// re-reads while streaming writes pass through L2.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap *map, uint32_t mbar, int c0, int c1,
                                                 int c2, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
        "%4, %5}], [%2], %6;\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, uint32_t mbar, int c0, int c1,
                                                 uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
        "%4}], [%2], %5;\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar), "r"(c0), "r"(c1), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t mbar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, "
        "%6}], [%2];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, uint32_t mbar, int c0, int c1,
                                            int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, "
        "%7}], [%2];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}
__device__ __forceinline__ void tma_gather4_hint(uint32_t dst, const CUtensorMap *map, uint32_t mbar, int c0, int r0,
                                                 int r1, int r2, int r3, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "l"(pol)
        : "memory");
}
// Contiguous global -> shared copy of `bytes` (a multiple of 16; both
// addresses 16-byte aligned) completing on an mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory
// ---------------------------------------------------------------------------
// Executed by one full warp.  Writes the allocated base address to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: descriptors
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (16-byte units), version 1, layout type 2.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 accumulate.
// a_mn / b_mn: operand stored MN-major (transposed) instead of K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | ((uint32_t)a_mn << 15)        // A major
           | ((uint32_t)b_mn << 16)        // B major
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Instruction descriptor for kind::f8f6f4 with e4m3 A/B (format code 0),
// fp32 accumulate, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                       // D format: f32
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// D[tmem] (+)= A[smem desc] * B[smem desc], e4m3 operands (K = 32 per instruction)
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
// Eight kind::f16 MMAs (K = 16 each) into d_tmem from one asm block: the
// first overwrites D, the other seven accumulate; A and B from shared memory
// (descriptors a[i], b[i]).
__device__ __forceinline__ void mma_ss8(uint32_t d_tmem, const uint64_t (&a)[8], const uint64_t (&b)[8],
                                        uint32_t idesc) {
    asm volatile(
        "{\n .reg .pred p0, p1;\n setp.ne.b32 p0, %1, %1;\n setp.eq.b32 p1, %1, %1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %1, p0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %17, %1, p1;\n}\n" ::"r"(d_tmem),
        "r"(idesc), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]), "l"(b[0]),
        "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7])
        : "memory");
}
// The same with A in tensor memory (columns a[i]) and B from shared memory.
__device__ __forceinline__ void mma_ts8(uint32_t d_tmem, const uint32_t (&a)[8], const uint64_t (&b)[8],
                                        uint32_t idesc) {
    asm volatile(
        "{\n .reg .pred p0, p1;\n setp.ne.b32 p0, %1, %1;\n setp.eq.b32 p1, %1, %1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %10, %1, p0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %11, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %12, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %13, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %14, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %15, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %16, %1, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %17, %1, p1;\n}\n" ::"r"(d_tmem),
        "r"(idesc), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "l"(b[0]),
        "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7])
        : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on an mbarrier once all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
                 : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory <-> registers (32 lanes x 32 bit, per warp quarter)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// 128 consecutive columns of the warp's 32 lanes (one full S or O row per thread).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
#define MSA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                  "=r"(r[i + 6]), "=r"(r[i + 7])
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,"
        "%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,"
        "%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
        "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,"
        "%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n"
        : MSA_R8(0), MSA_R8(8), MSA_R8(16), MSA_R8(24), MSA_R8(32), MSA_R8(40), MSA_R8(48), MSA_R8(56), MSA_R8(64),
          MSA_R8(72), MSA_R8(80), MSA_R8(88), MSA_R8(96), MSA_R8(104), MSA_R8(112), MSA_R8(120)
        : "r"(taddr));
#undef MSA_R8
}
// Stores r[0..63] into 64 consecutive columns.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[128]) {
#define MSA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                  "r"(r[i + 6]), "r"(r[i + 7])
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,"
        "%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n" ::"r"(taddr),
        MSA_W8(0), MSA_W8(8), MSA_W8(16), MSA_W8(24), MSA_W8(32), MSA_W8(40), MSA_W8(48), MSA_W8(56)
        : "memory");
#undef MSA_W8
}
// Stores r[0..127] into 128 consecutive columns (a whole O row per thread).
__device__ __forceinline__ void tmem_st128(uint32_t taddr, const uint32_t (&r)[128]) {
#define MSA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                  "r"(r[i + 6]), "r"(r[i + 7])
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x128.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,"
        "%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,"
        "%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,"
        "%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,"
        "%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127,%128};\n" ::"r"(taddr),
        MSA_W8(0), MSA_W8(8), MSA_W8(16), MSA_W8(24), MSA_W8(32), MSA_W8(40), MSA_W8(48), MSA_W8(56), MSA_W8(64),
        MSA_W8(72), MSA_W8(80), MSA_W8(88), MSA_W8(96), MSA_W8(104), MSA_W8(112), MSA_W8(120)
        : "memory");
#undef MSA_W8
}
// 64 consecutive columns of the warp's 32 lanes (half an S or O row per
// thread), as two 32-column loads.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    tmem_ld32(taddr + 32u, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
}
// Stores r[0..31] into 32 consecutive columns.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[64]) {
#define MSA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                  "r"(r[i + 6]), "r"(r[i + 7])
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        MSA_W8(0), MSA_W8(8), MSA_W8(16), MSA_W8(24)
        : "memory");
#undef MSA_W8
}
// Stores r[0..31] into 32 consecutive columns (from a 32-register array).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
#define MSA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                  "r"(r[i + 6]), "r"(r[i + 7])
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        MSA_W8(0), MSA_W8(8), MSA_W8(16), MSA_W8(24)
        : "memory");
#undef MSA_W8
}
// Stores r[0..15] into 16 consecutive columns (from a 32-register array).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[32]) {
#define MSA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                  "r"(r[i + 6]), "r"(r[i + 7])
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16};\n" ::"r"(taddr),
                 MSA_W8(0), MSA_W8(8)
                 : "memory");
#undef MSA_W8
}
// Stores r[0..63] into 64 consecutive columns (from a 64-register array).
__device__ __forceinline__ void tmem_st64h(uint32_t taddr, const uint32_t (&r)[64]) {
#define MSA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                  "r"(r[i + 6]), "r"(r[i + 7])
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,"
        "%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n" ::"r"(taddr),
        MSA_W8(0), MSA_W8(8), MSA_W8(16), MSA_W8(24), MSA_W8(32), MSA_W8(40), MSA_W8(48), MSA_W8(56)
        : "memory");
#undef MSA_W8
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled
// tile of 128-byte rows whose base is 1024-byte aligned.
__host__ __device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

}  // namespace tc

// ---------------------------------------------------------------------------
// host: TMA descriptor creation through the driver entry point
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 4D bf16 view of a K or V cache [tokens][heads][128]: dims {64 elements,
// tokens, 2 column halves, heads} with byte strides {heads*256, 128, 256} and
// box {64, 128, 2, 1}: one copy brings a whole 128-token block of one head as
// [half][128 tokens][128 B], 128-byte swizzled (halves 16384 bytes apart).
inline bool make_kv_map(CUtensorMap *map, const void *base, int heads, int64_t tokens) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[4] = {64, (cuuint64_t)tokens, 2, (cuuint64_t)heads};
    cuuint64_t strides[3] = {(cuuint64_t)heads * 256, 128, 256};
    cuuint32_t box[4] = {64, 128, 2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3D e4m3 view of a K cache [tokens][heads][128 bytes]: dims {128, tokens,
// heads} with byte strides {heads*128, 128} and box {128, 128, 1}: one copy
// brings a 128-token block of one head as [128 tokens][128 B], 128-byte swizzled.
inline bool make_k8_map(CUtensorMap *map, const void *base, int heads, int64_t tokens) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)tokens, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)heads * 128, 128};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// e4m3 query rows [rows][128 bytes]: qpk >= 8, one box per (query, KV head)
// group as 4D {128, 8 rows, qpk/8 octets, groups} (strides {128, 1024,
// qpk*128}, box {128, 8, qpk/8, 1}: [octet][8 rows][128 B], octets 1024 bytes
// apart); qpk < 8, 2D rows {128, rows} with a one-row box for tile::gather4.
inline bool make_q8_map(CUtensorMap *map, const void *base, int64_t rows, int qpk) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    CUresult r;
    if (qpk >= 8) {
        const int64_t groups = rows / qpk;
        cuuint64_t dims[4] = {128, 8, (cuuint64_t)(qpk / 8), (cuuint64_t)groups};
        cuuint64_t strides[3] = {128, 1024, (cuuint64_t)qpk * 128};
        cuuint32_t box[4] = {128, 8, (cuuint32_t)(qpk / 8), 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[2] = {128, (cuuint64_t)rows};
        cuuint64_t strides[1] = {128};
        cuuint32_t box[2] = {128, 1};
        cuuint32_t estr[2] = {1, 1};
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

// 3D bf16 view of queries [tokens][Hq][128]: dims {128 elements, Hq heads,
// tokens} with byte strides {256, Hq*256} and box {64, qpk, 128/qpk}: one copy
// brings one column half of the qpk heads of a KV head for 128/qpk
// consecutive tokens as 128 rows (row = token * qpk + head) of 128 bytes,
// 128-byte swizzled (rows past the last token are zero).
inline bool make_q_heads_map(CUtensorMap *map, const void *base, int64_t tokens, int Hq, int qpk) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)Hq, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {256, (cuuint64_t)Hq * 256};
    cuuint32_t box[3] = {64, (cuuint32_t)qpk, (cuuint32_t)(128 / qpk)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2D bf16 map over the query rows [rows][128]: box {64, box_rows}; box_rows
// = 1 is the gather4 form (four arbitrary rows per copy).
inline bool make_q_map(CUtensorMap *map, const void *base, int64_t rows, int box_rows) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    cuuint64_t strides[1] = {128 * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 5D bf16 view of the query rows for qhead_per_kv >= 8, one box per (query,
// KV head) group of qpk rows: dims {64 elements, 8 rows, 2 column halves,
// qpk/8 row octets, groups} with byte strides {256, 128, 2048, qpk*256} and
// box {64, 8, 2, qpk/8, 1}.  A box lands as [octet][half][8 rows][128 B] with
// the 128-byte swizzle: each (octet, half) is one 1024-byte K-major atom, so
// the chunk's row octets sit 2048 bytes apart and its halves 1024 bytes apart.
inline bool make_q_group_map(CUtensorMap *map, const void *base, int64_t groups, int qpk) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[5] = {64, 8, 2, (cuuint64_t)(qpk / 8), (cuuint64_t)groups};
    cuuint64_t strides[4] = {256, 128, 2048, (cuuint64_t)qpk * 256};
    cuuint32_t box[5] = {64, 8, 2, (cuuint32_t)(qpk / 8), 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace msa
