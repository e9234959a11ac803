// csr.cu -- deterministic k->q CSR inversion and the prefill work plan.
//
// Source: interface.py module docstring (q2k [Hkv,total_q,topK] is inverted
// into k2q_row_ptr [Hkv,total_rows+1] and k2q_q_indices [Hkv,total_q*topK])
// and test_sparse_atten.py test_scheduler_builds_packed_qsplit_metadata /
// test_k2q_csr_builder_matches_torch_reference (bit-exact CSR, packed
// q | split << 24, work items bounded by the per-CTA query target, every row
// covered).
//
// Three passes over tiles of 128 queries of one (sequence, KV head):
//   1. hist: a 128-bit mask per KV block (bit i = query i of the tile names
//      the block) built in shared memory; per-tile counts written out.
//   2. scan: per block, exclusive scan of the tile counts (tile offsets inside
//      the row) and row totals; then per head an inclusive scan of the row
//      totals gives row_ptr.
//   3. scatter: position = row_ptr + tile offset + popcount of the mask bits
//      below the query, so each row lists its queries in ascending order with
//      no atomics on positions (bit-deterministic).
// The plan then cuts every row into units of at most 8 chunks of 128 rows,
// ordered by KV head, then by wave: wave w holds the queries [w*W, (w+1)*W)
// (W: wave_queries in common.cuh).
#include <algorithm>

#include "common.cuh"

namespace msa {
namespace {

constexpr int kTileQ = 128;  // queries per CSR tile (4 x 32-bit mask words)

struct CsrShape {
    int B, Hkv, Sq, Skv, topk, nblk, ntiles;
    int64_t rows, cap;
};

// Validity of one slot: 0 <= j < nvalid and not named by an earlier slot.
__device__ __forceinline__ bool slot_valid(const int32_t *sel, int t, int nvalid, uint32_t *status) {
    int j = sel[t];
    if (j < 0) return false;
    if (j >= nvalid) {
        set_status(status, MSA_STATUS_INDEX_RANGE);
        return false;
    }
    for (int u = 0; u < t; ++u)
        if (sel[u] == j) {
            set_status(status, MSA_STATUS_DUPLICATE);
            return false;
        }
    return true;
}

__device__ __forceinline__ int seq_nvalid(const int32_t *seqused, int b, int Skv, int nblk) {
    int64_t kv = seqused ? (int64_t)seqused[b] : (int64_t)Skv;
    int64_t n = ceil_div(kv, kBlk);
    if (n > nblk) n = nblk;
    if (n < 0) n = 0;
    return (int)n;
}

// Builds the per-block query masks of one tile in shared memory.
__device__ void build_masks(uint32_t *masks, const int32_t *q2k, const int32_t *seqused, const CsrShape &s,
                            int tile, int b, int h, uint32_t *status, int32_t *split_counts) {
    for (int i = threadIdx.x; i < s.nblk * 4; i += blockDim.x) masks[i] = 0u;
    __syncthreads();
    int i = threadIdx.x;
    int sq = tile * kTileQ + i;
    if (sq < s.Sq) {
        int nvalid = seq_nvalid(seqused, b, s.Skv, s.nblk);
        const int32_t *sel = q2k + (((int64_t)b * s.Hkv + h) * s.Sq + sq) * s.topk;
        int cnt = 0;
        for (int t = 0; t < s.topk; ++t) {
            if (!slot_valid(sel, t, nvalid, status)) continue;
            atomicOr(&masks[sel[t] * 4 + (i >> 5)], 1u << (i & 31));
            ++cnt;
        }
        if (split_counts) split_counts[((int64_t)b * s.Sq + sq) * s.Hkv + h] = cnt;
    }
    __syncthreads();
}

__global__ void csr_hist_kernel(const int32_t *__restrict__ q2k, const int32_t *__restrict__ seqused, CsrShape s,
                                int32_t *__restrict__ tile_counts, int32_t *__restrict__ split_counts,
                                uint32_t *status) {
    extern __shared__ uint32_t masks[];
    int tile = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
    build_masks(masks, q2k, seqused, s, tile, b, h, status, split_counts);
    int32_t *out = tile_counts + (((int64_t)h * s.B + b) * s.ntiles + tile) * s.nblk;
    for (int j = threadIdx.x; j < s.nblk; j += blockDim.x) {
        const uint32_t *m = masks + j * 4;
        out[j] = __popc(m[0]) + __popc(m[1]) + __popc(m[2]) + __popc(m[3]);
    }
}

// Column scan: for each (h, b, j) turn the tile counts into exclusive offsets
// within the row and write the row total to row_ptr[h][b*nblk + j + 1].
// Block (32, 32): threadIdx.x = block id offset, threadIdx.y = tile range.
// blockDim = (32 block columns, ty tile slices): slice y sums its run of
// tiles, thread y = 0 scans the ty slice sums, each slice rewrites its run.
__global__ void csr_colscan_kernel(int32_t *__restrict__ tile_counts, int32_t *__restrict__ row_ptr, CsrShape s) {
    __shared__ int32_t part[32][33];
    const int ty = blockDim.y;
    int j = blockIdx.x * 32 + threadIdx.x;
    int b = blockIdx.y, h = blockIdx.z;
    int per = (s.ntiles + ty - 1) / ty;
    int t0 = threadIdx.y * per;
    int t1 = min(t0 + per, s.ntiles);
    int32_t *base = tile_counts + ((int64_t)h * s.B + b) * s.ntiles * (int64_t)s.nblk;
    int32_t sum = 0;
    if (j < s.nblk)
        for (int t = t0; t < t1; ++t) sum += base[(int64_t)t * s.nblk + j];
    part[threadIdx.y][threadIdx.x] = sum;
    __syncthreads();
    if (threadIdx.y == 0) {
        int32_t run = 0;
        for (int y = 0; y < ty; ++y) {
            int32_t v = part[y][threadIdx.x];
            part[y][threadIdx.x] = run;
            run += v;
        }
        if (j < s.nblk) row_ptr[(int64_t)h * (s.rows + 1) + (int64_t)b * s.nblk + j + 1] = run;
    }
    __syncthreads();
    if (j < s.nblk) {
        int32_t run = part[threadIdx.y][threadIdx.x];
        for (int t = t0; t < t1; ++t) {
            int32_t v = base[(int64_t)t * s.nblk + j];
            base[(int64_t)t * s.nblk + j] = run;
            run += v;
        }
    }
}

// In-place scan of n int32 per blockIdx.x segment (segment stride `stride`),
// one CTA of 1024 threads per segment.  Each pass stages kScanItems * 1024
// values through shared memory with coalesced loads and stores; thread t
// scans values [t*kScanItems, (t+1)*kScanItems) of the pass.  exclusive != 0:
// out[i] = sum_{<i}; the segment total goes to totals[blockIdx.x] when
// totals != nullptr.
constexpr int kScanItems = 8;
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads) segment_scan_kernel(int32_t *data, int64_t n, int64_t stride,
                                                                    int exclusive, int32_t *totals) {
    __shared__ int32_t tile[kScanItems * kScanThreads + kScanItems * kScanThreads / 32];  // padded rows
    __shared__ int32_t warp_sums[32];
    int32_t *d = data + blockIdx.x * stride;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // padding of one word per 32 keeps a thread's run free of bank conflicts
    auto slot = [](int i) { return i + (i >> 5); };
    int32_t carry = 0;  // identical in every thread
    for (int64_t base = 0; base < n; base += (int64_t)kScanThreads * kScanItems) {
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            const int i = k * kScanThreads + tid;
            tile[slot(i)] = (base + i < n) ? d[base + i] : 0;
        }
        __syncthreads();
        int32_t v[kScanItems];
        int32_t tsum = 0;
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            v[k] = tile[slot(tid * kScanItems + k)];
            tsum += v[k];
        }
        int32_t x = tsum;  // inclusive scan of the thread sums
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        int32_t run = carry + x - tsum + (warp > 0 ? warp_sums[warp - 1] : 0);  // exclusive start of the thread
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            const int32_t incl = run + v[k];
            tile[slot(tid * kScanItems + k)] = exclusive ? run : incl;
            run = incl;
        }
        carry += warp_sums[31];
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            const int i = k * kScanThreads + tid;
            if (base + i < n) d[base + i] = tile[slot(i)];
        }
        __syncthreads();  // tile and warp_sums are rewritten by the next pass
    }
    if (totals && threadIdx.x == 0) totals[blockIdx.x] = carry;
}

__global__ void csr_scatter_kernel(const int32_t *__restrict__ q2k, const int32_t *__restrict__ seqused, CsrShape s,
                                   const int32_t *__restrict__ tile_off, const int32_t *__restrict__ row_ptr,
                                   int32_t *__restrict__ q_indices, int32_t *__restrict__ qsplit) {
    extern __shared__ uint32_t masks[];
    int tile = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
    build_masks(masks, q2k, seqused, s, tile, b, h, nullptr, nullptr);
    int i = threadIdx.x;
    int sq = tile * kTileQ + i;
    if (sq >= s.Sq) return;
    int nvalid = seq_nvalid(seqused, b, s.Skv, s.nblk);
    const int32_t *sel = q2k + (((int64_t)b * s.Hkv + h) * s.Sq + sq) * s.topk;
    const int32_t *off = tile_off + (((int64_t)h * s.B + b) * s.ntiles + tile) * s.nblk;
    const int32_t *rp = row_ptr + (int64_t)h * (s.rows + 1) + (int64_t)b * s.nblk;
    int32_t *qi = q_indices + (int64_t)h * s.cap;
    int32_t *qs = qsplit + (int64_t)h * s.cap;
    int32_t gq = (int32_t)((int64_t)b * s.Sq + sq);
    int w = i >> 5;
    uint32_t below = (1u << (i & 31)) - 1u;
    int rank = 0;
    for (int t = 0; t < s.topk; ++t) {
        if (!slot_valid(sel, t, nvalid, nullptr)) continue;
        int j = sel[t];
        const uint32_t *m = masks + j * 4;
        int r = __popc(m[w] & below);
        for (int x = 0; x < w; ++x) r += __popc(m[x]);
        int64_t pos = (int64_t)rp[j] + off[j] + r;
        qi[pos] = gq;
        qs[pos] = gq | (rank << 24);
        ++rank;
    }
}

__global__ void csr_tail_kernel(const int32_t *__restrict__ row_ptr, CsrShape s, int32_t *__restrict__ q_indices,
                                int32_t *__restrict__ qsplit) {
    int h = blockIdx.y;
    int64_t nnz = row_ptr[(int64_t)h * (s.rows + 1) + s.rows];
    for (int64_t i = nnz + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < s.cap;
         i += (int64_t)gridDim.x * blockDim.x) {
        q_indices[(int64_t)h * s.cap + i] = -1;
        qsplit[(int64_t)h * s.cap + i] = -1;
    }
}

// First position in the ascending run a[lo, hi) holding a value >= key.
__device__ __forceinline__ int32_t lower_bound(const int32_t *a, int32_t lo, int32_t hi, int32_t key) {
    while (lo < hi) {
        int32_t mid = lo + ((hi - lo) >> 1);
        if (a[mid] < key) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Segment (head h, wave w, row r) = the queries of row r in [w*W, (w+1)*W);
// the flat index is head-major, then wave-major, so the unit list runs one
// KV head at a time (its K/V stays in L2) and, within it, wave by wave (the
// CTAs read the Q rows of one wave's queries at a time).
struct PlanShape {
    int64_t W, nwaves;
    int qpu;
};

__device__ __forceinline__ void segment_range(const int32_t *row_ptr, const int32_t *q_indices, const CsrShape &s,
                                              const PlanShape &ps, int64_t idx, int &h, int64_t &r, int32_t &lo,
                                              int32_t &hi) {
    const int64_t per_head = ps.nwaves * s.rows;
    h = (int)(idx / per_head);
    const int64_t rem = idx % per_head;
    const int64_t w = rem / s.rows;
    r = rem % s.rows;
    const int32_t *rp = row_ptr + (int64_t)h * (s.rows + 1);
    const int32_t *qi = q_indices + (int64_t)h * s.cap;
    const int32_t b0 = rp[r], b1 = rp[r + 1];
    lo = lower_bound(qi, b0, b1, (int32_t)(w * ps.W));
    hi = lower_bound(qi, lo, b1, (int32_t)((w + 1) * ps.W));
}

// Units per segment: ceil(count / q_per_unit).
__global__ void plan_count_kernel(const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ q_indices,
                                  CsrShape s, PlanShape ps, int32_t *__restrict__ units_per_seg) {
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= ps.nwaves * s.Hkv * s.rows) return;
    int h;
    int64_t r;
    int32_t lo, hi;
    segment_range(row_ptr, q_indices, s, ps, idx, h, r, lo, hi);
    units_per_seg[idx] = (hi - lo + ps.qpu - 1) / ps.qpu;
}

__global__ void plan_write_kernel(const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ q_indices,
                                  CsrShape s, PlanShape ps, const int32_t *__restrict__ unit_off,
                                  const int32_t *__restrict__ total, PlanHeader *plan, PlanUnit *units, int capacity,
                                  int qpk, uint32_t *status) {
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx == 0) {
        int32_t tot = *total;
        if (tot > capacity) {
            set_status(status, MSA_STATUS_PLAN_OVERFLOW);
            tot = capacity;
        }
        plan->work_count = tot;
        plan->capacity = capacity;
        plan->qhead_per_kv = qpk;
        plan->q_per_unit = ps.qpu;
        plan->wave_queries = (int32_t)ps.W;
        plan->nwaves = (int32_t)ps.nwaves;
    }
    if (idx >= ps.nwaves * s.Hkv * s.rows) return;
    int h;
    int64_t r;
    int32_t lo, hi;
    segment_range(row_ptr, q_indices, s, ps, idx, h, r, lo, hi);
    const int32_t c = hi - lo;
    const int32_t u0 = unit_off[idx];
    for (int32_t u = 0; u * ps.qpu < c; ++u) {
        if (u0 + u >= capacity) break;
        PlanUnit pu;
        pu.head = h;
        pu.row = (int32_t)r;
        pu.start = lo + u * ps.qpu;
        pu.count = min(ps.qpu, c - u * ps.qpu);
        units[u0 + u] = pu;
    }
}

CsrShape make_shape(int B, int Hkv, int Sq, int Skv, int topk) {
    CsrShape s;
    s.B = B; s.Hkv = Hkv; s.Sq = Sq; s.Skv = Skv; s.topk = topk;
    s.nblk = (int)ceil_div(Skv, kBlk);
    s.ntiles = (int)ceil_div(Sq, kTileQ);
    s.rows = (int64_t)B * s.nblk;
    s.cap = (int64_t)B * Sq * topk;
    return s;
}

struct CsrWorkspace {
    size_t tile_counts, units_per_row, total, bytes;
};

PlanShape make_plan_shape(const CsrShape &s, int qpk) {
    PlanShape ps;
    ps.W = wave_queries(s.B, s.Sq, qpk, s.topk);
    ps.nwaves = num_waves(s.B, s.Sq, qpk, s.topk);
    ps.qpu = q_per_unit(qpk);
    return ps;
}

// Segments (head, wave, row) of the plan; qpk 16 gives the smallest waves,
// hence the most of them.
int64_t max_segments(const CsrShape &s) {
    return num_waves(s.B, s.Sq, 16, s.topk) * s.Hkv * s.rows;
}

CsrWorkspace csr_workspace_layout(const CsrShape &s) {
    CsrWorkspace w;
    size_t off = 0;
    w.tile_counts = off;
    off = align_up(off + sizeof(int32_t) * (size_t)s.Hkv * s.B * s.ntiles * s.nblk, 256);
    w.units_per_row = off;
    off = align_up(off + sizeof(int32_t) * (size_t)max_segments(s), 256);
    w.total = off;
    off = align_up(off + 256, 256);
    w.bytes = off;
    return w;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" size_t msa_k2q_csr_workspace_size(int B, int Hkv, int Sq, int Skv, int topk, int blk_kv) {
    if (B <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || topk <= 0 || blk_kv != kBlk) return 0;
    return csr_workspace_layout(make_shape(B, Hkv, Sq, Skv, topk)).bytes;
}

extern "C" size_t msa_plan_size(int B, int Hkv, int Sq, int Skv, int topk, int blk_kv, int qhead_per_kv) {
    if (B <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || topk <= 0 || blk_kv != kBlk || !supported_qpk(qhead_per_kv))
        return 0;
    return sizeof(PlanHeader) + sizeof(PlanUnit) * (size_t)plan_capacity(B, Hkv, Sq, Skv, topk, qhead_per_kv);
}

extern "C" int msa_build_k2q_csr(const int32_t *q2k, int B, int Hkv, int Sq, int Skv, int topk, int blk_kv,
                                 int qhead_per_kv, const int32_t *seqused, int32_t *row_ptr, int32_t *q_indices,
                                 int32_t *qsplit, int32_t *split_counts, void *plan, size_t plan_bytes,
                                 void *workspace, size_t ws_bytes, uint32_t *status_dev, cudaStream_t stream) {
    if (!q2k || !row_ptr || !q_indices || !qsplit || !split_counts || !workspace) return MSA_ERR_INVALID_ARG;
    if (B <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || topk <= 0) return MSA_ERR_INVALID_ARG;
    if (blk_kv != kBlk || !supported_topk(topk) || !supported_qpk(qhead_per_kv)) return MSA_ERR_UNSUPPORTED;
    if ((int64_t)B * Sq >= (1 << 24)) return MSA_ERR_UNSUPPORTED;
    CsrShape s = make_shape(B, Hkv, Sq, Skv, topk);
    if (s.nblk > kMaxNblk) return MSA_ERR_UNSUPPORTED;
    CsrWorkspace w = csr_workspace_layout(s);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    if (plan && (plan_bytes < msa_plan_size(B, Hkv, Sq, Skv, topk, blk_kv, qhead_per_kv) || !aligned(plan, 16)))
        return MSA_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    int32_t *tile_counts = reinterpret_cast<int32_t *>(ws + w.tile_counts);

    size_t mask_smem = sizeof(uint32_t) * 4 * (size_t)s.nblk;
    static bool smem_set = false;
    if (!smem_set) {
        MSA_CUDA_TRY(cudaFuncSetAttribute(csr_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          sizeof(uint32_t) * 4 * kMaxNblk));
        MSA_CUDA_TRY(cudaFuncSetAttribute(csr_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          sizeof(uint32_t) * 4 * kMaxNblk));
        smem_set = true;
    }
    dim3 tgrid(s.ntiles, B, Hkv);
    csr_hist_kernel<<<tgrid, kTileQ, mask_smem, stream>>>(q2k, seqused, s, tile_counts, split_counts, status_dev);
    MSA_LAUNCH_CHECK();
    dim3 cgrid((unsigned)ceil_div(s.nblk, 32), B, Hkv);
    csr_colscan_kernel<<<cgrid, dim3(32, (unsigned)std::min(32, s.ntiles)), 0, stream>>>(tile_counts, row_ptr, s);
    MSA_LAUNCH_CHECK();
    // row_ptr[h][0] = 0, then inclusive scan of the row totals in [1, rows]
    MSA_CUDA_TRY(cudaMemset2DAsync(row_ptr, sizeof(int32_t) * (s.rows + 1), 0, sizeof(int32_t), Hkv, stream));
    segment_scan_kernel<<<Hkv, 1024, 0, stream>>>(row_ptr + 1, s.rows, s.rows + 1, 0, nullptr);
    MSA_LAUNCH_CHECK();
    csr_scatter_kernel<<<tgrid, kTileQ, mask_smem, stream>>>(q2k, seqused, s, tile_counts, row_ptr, q_indices,
                                                             qsplit);
    MSA_LAUNCH_CHECK();
    int tail_blocks = (int)std::min<int64_t>(ceil_div(s.cap, 256), 1024);
    csr_tail_kernel<<<dim3(tail_blocks, Hkv), 256, 0, stream>>>(row_ptr, s, q_indices, qsplit);
    MSA_LAUNCH_CHECK();

    if (plan) {
        PlanShape ps = make_plan_shape(s, qhead_per_kv);
        int32_t *ups = reinterpret_cast<int32_t *>(ws + w.units_per_row);
        int32_t *total = reinterpret_cast<int32_t *>(ws + w.total);
        int64_t n = ps.nwaves * Hkv * s.rows;
        int blocks = (int)ceil_div(n, 256);
        plan_count_kernel<<<blocks, 256, 0, stream>>>(row_ptr, q_indices, s, ps, ups);
        MSA_LAUNCH_CHECK();
        segment_scan_kernel<<<1, 1024, 0, stream>>>(ups, n, 0, 1, total);
        MSA_LAUNCH_CHECK();
        PlanHeader *ph = static_cast<PlanHeader *>(plan);
        PlanUnit *units = reinterpret_cast<PlanUnit *>(ph + 1);
        int capacity = (int)plan_capacity(B, Hkv, Sq, Skv, topk, qhead_per_kv);
        plan_write_kernel<<<blocks, 256, 0, stream>>>(row_ptr, q_indices, s, ps, ups, total, ph, units, capacity,
                                                      qhead_per_kv, status_dev);
        MSA_LAUNCH_CHECK();
    }
    return MSA_OK;
}
