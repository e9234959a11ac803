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
//
// Uniform batches (B sequences of Sq queries and Skv keys, q2k
// [B][Hkv][Sq][topk]) and ragged ones (interface.py sparse_atten_func:
// cu_seqlens_q / cu_seqlens_k, q2k [Hkv][total_q][topk] with block ids local
// to each sequence) run the same kernels; for a ragged batch a first kernel
// turns the cu_seqlens into a per-sequence table {first query, queries, keys,
// first CSR row} (sequence b owns rows row0_b .. row0_b + ceil(keys/128) - 1),
// dropping with MSA_STATUS_SHAPE any sequence whose ranges are inconsistent
// or do not fit the sizes the caller declared.
#include <algorithm>

#include "common.cuh"

namespace msa {
namespace {

constexpr int kTileQ = 128;  // queries per CSR tile (4 x 32-bit mask words)

struct CsrShape {
    int B, Hkv, Sq, Skv, topk, nblk, ntiles;  // ragged: Sq, Skv, nblk, ntiles are per-sequence maxima
    int64_t rows, cap, total_q;
    const int4 *seqs;  // ragged: per sequence {first query, queries, keys, first row}; uniform: null
};

// One sequence's queries, keys, block count and first CSR row.
struct Seq {
    int64_t q0, row0;
    int sq, kv, nblk;
};

__device__ __forceinline__ Seq seq_info(const CsrShape &s, int b) {
    Seq x;
    if (s.seqs) {
        const int4 e = s.seqs[b];
        x.q0 = e.x;
        x.sq = e.y;
        x.kv = e.z;
        x.row0 = e.w;
    } else {
        x.q0 = (int64_t)b * s.Sq;
        x.sq = s.Sq;
        x.kv = s.Skv;
        x.row0 = (int64_t)b * s.nblk;
    }
    x.nblk = (int)ceil_div(x.kv, kBlk);
    return x;
}

// The top-k list of query sl (local) of sequence b, KV head h.
__device__ __forceinline__ const int32_t *sel_of(const int32_t *q2k, const CsrShape &s, const Seq &x, int b, int h,
                                                 int sl) {
    return s.seqs ? q2k + ((int64_t)h * s.total_q + x.q0 + sl) * s.topk
                  : q2k + (((int64_t)b * s.Hkv + h) * s.Sq + sl) * s.topk;
}

// Blocks of sequence b a query may name: those below the used KV length.
__device__ __forceinline__ int seq_nvalid(const int32_t *seqused, int b, const Seq &x) {
    int64_t kv = seqused ? (int64_t)seqused[b] : (int64_t)x.kv;
    int64_t n = ceil_div(kv, kBlk);
    if (n > x.nblk) n = x.nblk;
    if (n < 0) n = 0;
    return (int)n;
}

// One query's top-k list in registers (ids[0 .. topk), topk <= 32; read as
// 16-byte vectors when the list is 16-byte aligned -- topk is a multiple of 4,
// so it is whenever q2k is) and the mask of its valid slots: bit t set when
// slot t names a block 0 <= j < nvalid that no earlier slot named.  With a
// status word, an id at or past nvalid raises MSA_STATUS_INDEX_RANGE and a
// repeated id MSA_STATUS_DUPLICATE.
__device__ __forceinline__ uint32_t load_slots(const int32_t *sel, int topk, int nvalid, uint32_t *status,
                                               int (&ids)[32]) {
    const bool vec = (reinterpret_cast<uintptr_t>(sel) & 15u) == 0;
#pragma unroll
    for (int t4 = 0; t4 < 8; ++t4) {
        int4 v = make_int4(-1, -1, -1, -1);
        if (4 * t4 < topk) {
            if (vec) {
                v = __ldg(reinterpret_cast<const int4 *>(sel) + t4);
            } else {
                v = make_int4(__ldg(sel + 4 * t4), __ldg(sel + 4 * t4 + 1), __ldg(sel + 4 * t4 + 2),
                              __ldg(sel + 4 * t4 + 3));
            }
        }
        ids[4 * t4 + 0] = v.x;
        ids[4 * t4 + 1] = v.y;
        ids[4 * t4 + 2] = v.z;
        ids[4 * t4 + 3] = v.w;
    }
    uint32_t valid = 0u;
    bool range = false, dup = false;
#pragma unroll
    for (int t = 0; t < 32; ++t) {
        if (t >= topk) break;
        const int j = ids[t];
        if (j < 0) continue;
        if (j >= nvalid) {
            range = true;
            continue;
        }
        bool seen = false;
#pragma unroll
        for (int u = 0; u < t; ++u) seen |= ids[u] == j;
        if (seen) {
            dup = true;
            continue;
        }
        valid |= 1u << t;
    }
    if (status && range) set_status(status, MSA_STATUS_INDEX_RANGE);
    if (status && dup) set_status(status, MSA_STATUS_DUPLICATE);
    return valid;
}

// Ragged batches: the per-sequence table and row offsets row_off [B+1] from
// cu_seqlens_q / cu_seqlens_k.  One CTA; sequences are scanned in passes of
// blockDim.x.  A sequence with a decreasing range, a start below 0, queries
// past total_q, more queries or keys than the declared maxima, or rows past
// total_rows is dropped (no queries, no keys) and raises MSA_STATUS_SHAPE.
__global__ void __launch_bounds__(1024) csr_seq_kernel(const int32_t *__restrict__ cu_q,
                                                       const int32_t *__restrict__ cu_k, int B, int64_t total_q,
                                                       int64_t total_rows, int max_sq, int max_kv, int4 *seqs,
                                                       int32_t *row_off, uint32_t *status) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry_s;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < B; base += blockDim.x) {
        const int b = base + threadIdx.x;
        int q0 = 0, sq = 0, kv = 0, nb = 0;
        if (b < B) {
            q0 = cu_q[b];
            const int q1 = cu_q[b + 1], k0 = cu_k[b], k1 = cu_k[b + 1];
            sq = q1 - q0;
            kv = k1 - k0;
            const bool ok = q0 >= 0 && sq >= 0 && (int64_t)q1 <= total_q && sq <= max_sq && k0 >= 0 && kv >= 0 &&
                            kv <= max_kv;
            if (!ok) {
                set_status(status, MSA_STATUS_SHAPE);
                sq = kv = 0;
            }
            nb = (int)ceil_div(kv, kBlk);
        }
        int32_t x = nb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int32_t incl = x + (warp > 0 ? warp_sums[warp - 1] : 0) + carry_s;
        int32_t row0 = incl - nb;
        if (b < B) {
            if ((int64_t)incl > total_rows) {  // rows past the declared capacity: drop the sequence
                set_status(status, MSA_STATUS_SHAPE);
                sq = kv = 0;
                row0 = (int32_t)total_rows;
            }
            seqs[b] = make_int4(q0, sq, kv, row0);
            row_off[b] = row0;
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry_s = incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        row_off[B] = carry_s > total_rows ? (int32_t)total_rows : carry_s;
        if ((int64_t)cu_q[B] != total_q) set_status(status, MSA_STATUS_SHAPE);  // queries outside every sequence
    }
}

// Builds the per-block query masks of one tile in shared memory.
__device__ void build_masks(uint32_t *masks, const int32_t *q2k, const int32_t *seqused, const CsrShape &s,
                            const Seq &x, int tile, int b, int h, uint32_t *status, int32_t *split_counts) {
    for (int i = threadIdx.x; i < x.nblk * 4; i += blockDim.x) masks[i] = 0u;
    __syncthreads();
    int i = threadIdx.x;
    int sq = tile * kTileQ + i;
    if (sq < x.sq) {
        int ids[32];
        const uint32_t valid = load_slots(sel_of(q2k, s, x, b, h, sq), s.topk, seq_nvalid(seqused, b, x), status, ids);
#pragma unroll
        for (int t = 0; t < 32; ++t)
            if ((valid >> t) & 1u) atomicOr(&masks[ids[t] * 4 + (i >> 5)], 1u << (i & 31));
        if (split_counts) split_counts[(x.q0 + sq) * s.Hkv + h] = __popc(valid);
    }
    __syncthreads();
}

__global__ void csr_hist_kernel(const int32_t *__restrict__ q2k, const int32_t *__restrict__ seqused, CsrShape s,
                                int32_t *__restrict__ tile_counts, int32_t *__restrict__ split_counts,
                                int32_t *__restrict__ row_ptr, uint32_t *status) {
    extern __shared__ uint32_t masks[];
    int tile = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
    grid_dependency_wait();  // the previous kernel on the stream may still read split_counts
    grid_dependents_launch();
    // uniform batch: row_ptr[h][0] = 0 (the column scan writes every other entry)
    if (!s.seqs && tile == 0 && b == 0 && threadIdx.x == 0) row_ptr[(int64_t)h * (s.rows + 1)] = 0;
    const Seq x = seq_info(s, b);
    if (tile * kTileQ >= x.sq) return;  // past this sequence's queries (whole CTA)
    build_masks(masks, q2k, seqused, s, x, tile, b, h, status, split_counts);
    int32_t *out = tile_counts + (((int64_t)h * s.B + b) * s.ntiles + tile) * s.nblk;
    for (int j = threadIdx.x; j < x.nblk; j += blockDim.x) {
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
    grid_dependency_wait();  // the previous CSR step
    grid_dependents_launch();
    __shared__ int32_t part[32][33];
    const int ty = blockDim.y;
    int j = blockIdx.x * 32 + threadIdx.x;
    int b = blockIdx.y, h = blockIdx.z;
    const Seq x = seq_info(s, b);
    if (blockIdx.x * 32 >= x.nblk) return;  // past this sequence's blocks (whole CTA)
    const int ntiles = (int)ceil_div(x.sq, kTileQ);
    int per = (ntiles + ty - 1) / ty;
    int t0 = threadIdx.y * per;
    int t1 = min(t0 + per, ntiles);
    int32_t *base = tile_counts + ((int64_t)h * s.B + b) * s.ntiles * (int64_t)s.nblk;
    int32_t sum = 0;
    if (j < x.nblk)
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
        if (j < x.nblk) row_ptr[(int64_t)h * (s.rows + 1) + x.row0 + j + 1] = run;
    }
    __syncthreads();
    if (j < x.nblk) {
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
    grid_dependency_wait();  // the previous CSR step
    grid_dependents_launch();
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
    grid_dependency_wait();  // the previous CSR step
    grid_dependents_launch();
    extern __shared__ uint32_t masks[];
    int tile = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
    const Seq x = seq_info(s, b);
    if (tile * kTileQ >= x.sq) return;  // past this sequence's queries (whole CTA)
    build_masks(masks, q2k, seqused, s, x, tile, b, h, nullptr, nullptr);
    int i = threadIdx.x;
    int sq = tile * kTileQ + i;
    if (sq >= x.sq) return;
    int ids[32];
    const uint32_t valid = load_slots(sel_of(q2k, s, x, b, h, sq), s.topk, seq_nvalid(seqused, b, x), nullptr, ids);
    const int32_t *off = tile_off + (((int64_t)h * s.B + b) * s.ntiles + tile) * s.nblk;
    const int32_t *rp = row_ptr + (int64_t)h * (s.rows + 1) + x.row0;
    int32_t *qi = q_indices + (int64_t)h * s.cap;
    int32_t *qs = qsplit + (int64_t)h * s.cap;
    int32_t gq = (int32_t)(x.q0 + sq);
    int w = i >> 5;
    uint32_t below = (1u << (i & 31)) - 1u;
    // every slot's row start and tile offset are loaded before any is used
    int base[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) base[t] = ((valid >> t) & 1u) ? rp[ids[t]] + off[ids[t]] : 0;
    int rank = 0;
#pragma unroll
    for (int t = 0; t < 32; ++t) {
        if (!((valid >> t) & 1u)) continue;
        const uint32_t *m = masks + ids[t] * 4;
        int r = __popc(m[w] & below);
        for (int y = 0; y < w; ++y) r += __popc(m[y]);
        const int64_t pos = (int64_t)base[t] + r;
        qi[pos] = gq;
        qs[pos] = gq | (rank << 24);
        ++rank;
    }
}

__global__ void csr_tail_kernel(const int32_t *__restrict__ row_ptr, CsrShape s, int32_t *__restrict__ q_indices,
                                int32_t *__restrict__ qsplit) {
    grid_dependency_wait();  // the previous CSR step
    grid_dependents_launch();
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
    const int32_t *row_off;  // ragged: first row of each sequence [B+1]; uniform: null
    // uniform batch with Sq a multiple of 128: every wave boundary is a tile
    // boundary, so a row's position of query b Sq + 128 t is row_ptr plus the
    // column scan's offset of tile t (tile_off), with no search; else null
    const int32_t *tile_off;
};

// Sequence and block of global row r.
__device__ __forceinline__ void row_owner(const CsrShape &s, const PlanShape &ps, int64_t r, int &seq, int &blk) {
    if (!ps.row_off) {
        seq = (int)(r / s.nblk);
        blk = (int)(r % s.nblk);
        return;
    }
    int lo = 0, hi = s.B;  // last b with row_off[b] <= r (sequences without rows are skipped)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ps.row_off[mid] <= r) lo = mid;
        else hi = mid;
    }
    seq = lo;
    blk = (int)(r - ps.row_off[lo]);
}

__device__ __forceinline__ void segment_range(const int32_t *row_ptr, const int32_t *q_indices, const CsrShape &s,
                                              const PlanShape &ps, int64_t idx, int &h, int64_t &r, int32_t &lo,
                                              int32_t &hi) {
    const int64_t per_head = ps.nwaves * s.rows;
    h = (int)(idx / per_head);
    const int64_t rem = idx % per_head;
    const int64_t w = rem / s.rows;
    r = rem % s.rows;
    const int32_t *rp = row_ptr + (int64_t)h * (s.rows + 1);
    const int32_t b0 = rp[r], b1 = rp[r + 1];
    if (ps.tile_off) {
        const int b = (int)(r / s.nblk), j = (int)(r % s.nblk);
        const int32_t *off = ps.tile_off + (int64_t)h * s.B * s.ntiles * s.nblk + (int64_t)b * s.ntiles * s.nblk + j;
        auto pos = [&](int64_t q) -> int32_t {  // first position of the row holding a query >= q
            const int64_t sl = q - (int64_t)b * s.Sq;
            if (sl <= 0) return b0;
            if (sl >= s.Sq) return b1;
            return b0 + off[(sl / kTileQ) * s.nblk];
        };
        lo = pos(w * ps.W);
        hi = pos((w + 1) * ps.W);
        return;
    }
    const int32_t *qi = q_indices + (int64_t)h * s.cap;
    lo = lower_bound(qi, b0, b1, (int32_t)(w * ps.W));
    hi = lower_bound(qi, lo, b1, (int32_t)((w + 1) * ps.W));
}

// Units per segment: ceil(count / q_per_unit).
__global__ void plan_count_kernel(const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ q_indices,
                                  CsrShape s, PlanShape ps, int32_t *__restrict__ units_per_seg) {
    grid_dependency_wait();  // the previous CSR step
    grid_dependents_launch();
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
    grid_dependency_wait();  // the previous CSR step
    grid_dependents_launch();
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
    if (c == 0) return;
    const int32_t u0 = unit_off[idx];
    int seq, blk;
    row_owner(s, ps, r, seq, blk);
    for (int32_t u = 0; u * ps.qpu < c; ++u) {
        if (u0 + u >= capacity) break;
        PlanUnit pu;
        pu.head = (int16_t)h;
        pu.blk = (int16_t)blk;
        pu.seq = seq;
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
    s.total_q = (int64_t)B * Sq;
    s.cap = s.total_q * topk;
    s.seqs = nullptr;
    return s;
}

// Ragged batch: Sq / Skv are the per-sequence maxima, rows the declared row capacity.
CsrShape make_varlen_shape(int B, int Hkv, int64_t total_q, int max_sq, int max_kv, int64_t total_rows, int topk) {
    CsrShape s = make_shape(B, Hkv, max_sq, max_kv, topk);
    s.rows = total_rows;
    s.total_q = total_q;
    s.cap = total_q * topk;
    return s;
}

struct CsrWorkspace {
    size_t tile_counts, units_per_row, total, seqs, row_off, bytes;
};

PlanShape make_plan_shape(const CsrShape &s, int qpk) {
    PlanShape ps;
    ps.W = wave_queries(s.total_q, qpk, s.topk);
    ps.nwaves = num_waves(s.total_q, qpk, s.topk);
    ps.qpu = q_per_unit(qpk);
    ps.row_off = nullptr;
    ps.tile_off = nullptr;
    return ps;
}

// Segments (head, wave, row) of the plan; qpk 16 gives the smallest waves,
// hence the most of them.
int64_t max_segments(const CsrShape &s) {
    return num_waves(s.total_q, 16, s.topk) * s.Hkv * s.rows;
}

CsrWorkspace csr_workspace_layout(const CsrShape &s, bool ragged) {
    CsrWorkspace w;
    size_t off = 0;
    w.tile_counts = off;
    off = align_up(off + sizeof(int32_t) * (size_t)s.Hkv * s.B * s.ntiles * s.nblk, 256);
    w.units_per_row = off;
    off = align_up(off + sizeof(int32_t) * (size_t)max_segments(s), 256);
    w.total = off;
    off = align_up(off + 256, 256);
    w.seqs = off;
    if (ragged) off = align_up(off + sizeof(int4) * (size_t)s.B, 256);
    w.row_off = off;
    if (ragged) off = align_up(off + sizeof(int32_t) * ((size_t)s.B + 1), 256);
    w.bytes = off;
    return w;
}

// Common argument checks of both builders (shape s already made).
int check_csr_args(const CsrShape &s, int topk, int blk_kv, int qpk) {
    if (blk_kv != kBlk || !supported_topk(topk) || !supported_qpk(qpk)) return MSA_ERR_UNSUPPORTED;
    if (s.total_q >= (1 << 24) || s.nblk > kMaxNblk || s.Hkv > kMaxHkv || s.B > 65535) return MSA_ERR_UNSUPPORTED;
    if (s.rows >= ((int64_t)1 << 31) || s.cap >= ((int64_t)1 << 31)) return MSA_ERR_UNSUPPORTED;
    if ((int64_t)s.ntiles > 65535 * 1024) return MSA_ERR_UNSUPPORTED;
    return MSA_OK;
}

// The CSR passes and the plan, once the shape (and, ragged, its sequence
// table in the workspace) is set.
int csr_launch(const CsrShape &s, const int32_t *q2k, int qhead_per_kv, const int32_t *seqused, int32_t *row_ptr,
               int32_t *q_indices, int32_t *qsplit, int32_t *split_counts, void *plan, char *ws,
               const CsrWorkspace &w, const int32_t *row_off, uint32_t *status_dev, cudaStream_t stream) {
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
    dim3 tgrid(s.ntiles, s.B, s.Hkv);
    // The CSR kernels are chained with programmatic dependent launch: each
    // waits for the one before it (grid_dependency_wait) at its start.
    MSA_CUDA_TRY(launch_pdl(csr_hist_kernel, tgrid, dim3(kTileQ), mask_smem, stream, q2k, seqused, s, tile_counts,
                            split_counts, row_ptr, status_dev));
    if (s.seqs) {
        // rows past the sequences' blocks (capacity above need) count 0 (a
        // uniform batch's row_ptr[h][0] is written by the histogram kernel)
        MSA_CUDA_TRY(cudaMemsetAsync(row_ptr, 0, sizeof(int32_t) * (size_t)(s.rows + 1) * s.Hkv, stream));
    }
    dim3 cgrid((unsigned)ceil_div(s.nblk, 32), s.B, s.Hkv);
    MSA_CUDA_TRY(launch_pdl(csr_colscan_kernel, cgrid, dim3(32, (unsigned)std::min(32, s.ntiles)), 0, stream,
                            tile_counts, row_ptr, s));
    // inclusive scan of the row totals in [1, rows]
    MSA_CUDA_TRY(launch_pdl(segment_scan_kernel, dim3(s.Hkv), dim3(kScanThreads), 0, stream, row_ptr + 1, s.rows,
                            s.rows + 1, 0, (int32_t *)nullptr));
    MSA_CUDA_TRY(launch_pdl(csr_scatter_kernel, tgrid, dim3(kTileQ), mask_smem, stream, q2k, seqused, s,
                            (const int32_t *)tile_counts, (const int32_t *)row_ptr, q_indices, qsplit));
    int tail_blocks = (int)std::min<int64_t>(ceil_div(s.cap, 256), 1024);
    MSA_CUDA_TRY(launch_pdl(csr_tail_kernel, dim3(tail_blocks, s.Hkv), dim3(256), 0, stream, (const int32_t *)row_ptr,
                            s, q_indices, qsplit));

    if (plan) {
        PlanShape ps = make_plan_shape(s, qhead_per_kv);
        ps.row_off = row_off;
        if (!s.seqs && s.Sq % kTileQ == 0 && ps.W % kTileQ == 0) ps.tile_off = tile_counts;
        int32_t *ups = reinterpret_cast<int32_t *>(ws + w.units_per_row);
        int32_t *total = reinterpret_cast<int32_t *>(ws + w.total);
        int64_t n = ps.nwaves * s.Hkv * s.rows;
        int blocks = (int)ceil_div(n, 256);
        MSA_CUDA_TRY(launch_pdl(plan_count_kernel, dim3(blocks), dim3(256), 0, stream, (const int32_t *)row_ptr,
                                (const int32_t *)q_indices, s, ps, ups));
        MSA_CUDA_TRY(launch_pdl(segment_scan_kernel, dim3(1), dim3(kScanThreads), 0, stream, ups, n, (int64_t)0, 1,
                                total));
        PlanHeader *ph = static_cast<PlanHeader *>(plan);
        PlanUnit *units = reinterpret_cast<PlanUnit *>(ph + 1);
        int capacity = (int)plan_capacity(s.rows, s.total_q, s.Hkv, s.topk, qhead_per_kv);
        MSA_CUDA_TRY(launch_pdl(plan_write_kernel, dim3(blocks), dim3(256), 0, stream, (const int32_t *)row_ptr,
                                (const int32_t *)q_indices, s, ps, (const int32_t *)ups, (const int32_t *)total, ph,
                                units, capacity, qhead_per_kv, status_dev));
    }
    return MSA_OK;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" size_t msa_k2q_csr_workspace_size(int B, int Hkv, int Sq, int Skv, int topk, int blk_kv) {
    if (B <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || topk <= 0 || blk_kv != kBlk) return 0;
    return csr_workspace_layout(make_shape(B, Hkv, Sq, Skv, topk), false).bytes;
}

extern "C" size_t msa_plan_size(int B, int Hkv, int Sq, int Skv, int topk, int blk_kv, int qhead_per_kv) {
    if (B <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || topk <= 0 || blk_kv != kBlk || !supported_qpk(qhead_per_kv))
        return 0;
    const CsrShape s = make_shape(B, Hkv, Sq, Skv, topk);
    return sizeof(PlanHeader) + sizeof(PlanUnit) * (size_t)plan_capacity(s.rows, s.total_q, Hkv, topk, qhead_per_kv);
}

extern "C" int msa_build_k2q_csr(const int32_t *q2k, int B, int Hkv, int Sq, int Skv, int topk, int blk_kv,
                                 int qhead_per_kv, const int32_t *seqused, int32_t *row_ptr, int32_t *q_indices,
                                 int32_t *qsplit, int32_t *split_counts, void *plan, size_t plan_bytes,
                                 void *workspace, size_t ws_bytes, uint32_t *status_dev, cudaStream_t stream) {
    if (!q2k || !row_ptr || !q_indices || !qsplit || !split_counts || !workspace) return MSA_ERR_INVALID_ARG;
    if (B <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || topk <= 0) return MSA_ERR_INVALID_ARG;
    const CsrShape s = make_shape(B, Hkv, Sq, Skv, topk);
    const int rc = check_csr_args(s, topk, blk_kv, qhead_per_kv);
    if (rc != MSA_OK) return rc;
    const CsrWorkspace w = csr_workspace_layout(s, false);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    if (plan && (plan_bytes < msa_plan_size(B, Hkv, Sq, Skv, topk, blk_kv, qhead_per_kv) || !aligned(plan, 16)))
        return MSA_ERR_WORKSPACE;
    return csr_launch(s, q2k, qhead_per_kv, seqused, row_ptr, q_indices, qsplit, split_counts, plan,
                      static_cast<char *>(workspace), w, nullptr, status_dev, stream);
}

extern "C" size_t msa_k2q_csr_varlen_workspace_size(int B, int Hkv, int total_q, int max_seqlen_q, int max_seqlen_k,
                                                    int total_rows, int topk, int blk_kv) {
    if (B <= 0 || Hkv <= 0 || total_q <= 0 || max_seqlen_q <= 0 || max_seqlen_k <= 0 || total_rows <= 0 ||
        topk <= 0 || blk_kv != kBlk)
        return 0;
    return csr_workspace_layout(make_varlen_shape(B, Hkv, total_q, max_seqlen_q, max_seqlen_k, total_rows, topk),
                                true)
        .bytes;
}

extern "C" size_t msa_plan_varlen_size(int Hkv, int total_q, int total_rows, int topk, int blk_kv,
                                       int qhead_per_kv) {
    if (Hkv <= 0 || total_q <= 0 || total_rows <= 0 || topk <= 0 || blk_kv != kBlk || !supported_qpk(qhead_per_kv))
        return 0;
    return sizeof(PlanHeader) + sizeof(PlanUnit) * (size_t)plan_capacity(total_rows, total_q, Hkv, topk, qhead_per_kv);
}

extern "C" int msa_build_k2q_csr_varlen(const int32_t *q2k, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                        int B, int Hkv, int total_q, int max_seqlen_q, int max_seqlen_k,
                                        int total_rows, int topk, int blk_kv, int qhead_per_kv,
                                        const int32_t *seqused, int32_t *row_ptr, int32_t *q_indices,
                                        int32_t *qsplit, int32_t *split_counts, void *plan, size_t plan_bytes,
                                        void *workspace, size_t ws_bytes, uint32_t *status_dev,
                                        cudaStream_t stream) {
    if (!q2k || !cu_seqlens_q || !cu_seqlens_k || !row_ptr || !q_indices || !qsplit || !split_counts || !workspace)
        return MSA_ERR_INVALID_ARG;
    if (B <= 0 || Hkv <= 0 || total_q <= 0 || max_seqlen_q <= 0 || max_seqlen_k <= 0 || total_rows <= 0 ||
        topk <= 0)
        return MSA_ERR_INVALID_ARG;
    CsrShape s = make_varlen_shape(B, Hkv, total_q, max_seqlen_q, max_seqlen_k, total_rows, topk);
    const int rc = check_csr_args(s, topk, blk_kv, qhead_per_kv);
    if (rc != MSA_OK) return rc;
    const CsrWorkspace w = csr_workspace_layout(s, true);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    if (plan && (plan_bytes < msa_plan_varlen_size(Hkv, total_q, total_rows, topk, blk_kv, qhead_per_kv) ||
                 !aligned(plan, 16)))
        return MSA_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    // a query outside every kept sequence keeps 0 splits (O = 0, LSE = -inf)
    MSA_CUDA_TRY(cudaMemsetAsync(split_counts, 0, sizeof(int32_t) * (size_t)total_q * Hkv, stream));
    int4 *seqs = reinterpret_cast<int4 *>(ws + w.seqs);
    int32_t *row_off = reinterpret_cast<int32_t *>(ws + w.row_off);
    csr_seq_kernel<<<1, 1024, 0, stream>>>(cu_seqlens_q, cu_seqlens_k, B, total_q, total_rows, max_seqlen_q,
                                           max_seqlen_k, seqs, row_off, status_dev);
    MSA_LAUNCH_CHECK();
    s.seqs = seqs;
    return csr_launch(s, q2k, qhead_per_kv, seqused, row_ptr, q_indices, qsplit, split_counts, plan, ws, w, row_off,
                      status_dev, stream);
}
