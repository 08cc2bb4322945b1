// Expert-sorted permutation of routed top-k pairs (qmoe_align_sort).
//
// Grouping all experts' projections into one launch needs the pairs ordered by
// expert, and the scatter back must keep a deterministic order ("perf(qmoe):
// group prefill expert matmuls", description).  The order here is the stable
// one: within an expert, slots follow ascending pair id p = t*k + j.
//
// Up to 2048 pairs (one chunk) a single CTA does all of it in one launch;
// above, three launches, none of which lets an atomic decide an order:
//   1. hist:    each CTA owns a contiguous chunk of kChunk pairs and counts
//               them per expert (shared-memory counters).
//   2. scan:    one CTA turns the [chunk][expert] histograms into per-chunk
//               base slots (exclusive over chunks within an expert, plus the
//               expert's offset) and writes counts and offsets.
//   3. scatter: each CTA walks its chunk again in pair order; a pair's slot
//               is its chunk base + the running count of earlier equal ids,
//               so the result is the stable counting sort.
// The scan also derives the GEMMs' token-tile schedule, and the scatter
// gives every slot and every pair its row in the token tiles (so the permute
// and intermediate kernels look it up instead of searching the offsets).
#include "qmoe_common.cuh"
#include "mx_tiles.cuh"

namespace qmoe {

constexpr int kChunk = 2048;          // pairs per chunk (one CTA)
constexpr int kThreads = 1024;        // threads per CTA in hist/scatter (two rounds per chunk)
constexpr int kMaxExperts = 4096;     // shared-memory counter bound
constexpr int kScanThreads = 1024;

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive scan of one value per thread over a 1024-thread CTA; `total`
// receives the sum (every thread).  ws: 33 ints of shared memory.
__device__ int block_exclusive_scan(int v, int32_t* ws, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = ws[lane];
        int wi = w;
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += u;
        }
        ws[lane] = wi - w;
        if (lane == 31) ws[32] = wi;
    }
    __syncthreads();
    const int r = ws[warp] + incl - v;
    total = ws[32];
    __syncthreads();  // ws may be reused right after
    return r;
}

// Token-tile schedule for the tensor-core GEMMs from the counts of experts
// e0..e1 (this thread's, E <= 4 * 1024): tile_start[e] = prefix over experts
// of ceil(count[e] / nmax), tile_start[E] = number of tiles.
__device__ void write_tile_schedule(const int (&cnt)[4], int e0, int e1, int E, int nmax, int32_t* ws,
                                    int32_t* __restrict__ tile_start) {
    int local = 0;
    for (int e = e0; e < e1; ++e) local += (cnt[e - e0] + nmax - 1) / nmax;
    int total;
    int base = block_exclusive_scan(local, ws, total);
    for (int e = e0; e < e1; ++e) {
        tile_start[e] = base;
        base += (cnt[e - e0] + nmax - 1) / nmax;
    }
    if (threadIdx.x == 0) tile_start[E] = total;
}

// Per-chunk expert histogram: counts do not depend on order, so shared-memory
// atomics are fine here.
__global__ void __launch_bounds__(kThreads)
align_hist_kernel(const int32_t* __restrict__ ids, int64_t P, int E, int nchunks, int32_t* __restrict__ hist,
                  int32_t* __restrict__ dev_status) {
    extern __shared__ int32_t cnt[];
    const int tid = threadIdx.x;
    pdl_sync();
    for (int e = tid; e < E; e += kThreads) cnt[e] = 0;
    __syncthreads();
    const int64_t p0 = (int64_t)blockIdx.x * kChunk;
    int bad = 0;
    for (int i = tid; i < kChunk; i += kThreads) {
        const int64_t p = p0 + i;
        if (p < P) {
            const int e = ids[p];
            if (e >= 0 && e < E)
                atomicAdd(&cnt[e], 1);
            else
                bad = 1;
        }
    }
    if (__syncthreads_or(bad) && tid == 0) atomicOr(dev_status, QMOE_DEV_BAD_EXPERT_ID);
    int32_t* out = hist + (size_t)blockIdx.x * E;
    for (int e = tid; e < E; e += kThreads) out[e] = cnt[e];
}

// One CTA: per expert, chunk bases exclusive over chunks (loads issued eight
// at a time so they overlap), counts, offsets, the -1 tail of sorted ids and
// (tile_start non-null) the token-tile schedule.
__global__ void __launch_bounds__(kScanThreads)
align_scan_kernel(int32_t* __restrict__ hist, int64_t P, int E, int nchunks, int nmax, int32_t* __restrict__ counts,
                  int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_pair_ids, int32_t* __restrict__ tile_start,
                  int32_t* __restrict__ slot_dest) {
    __shared__ int32_t ws[33];
    const int tid = threadIdx.x;
    pdl_sync();
    const int per = (E + kScanThreads - 1) / kScanThreads;  // <= 4 (E <= kMaxExperts)
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int cnt[4] = {0, 0, 0, 0};
    int local = 0;
    for (int e = e0; e < e1; ++e) {
        int run = 0;
        for (int c0 = 0; c0 < nchunks; c0 += 8) {
            int32_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = (c0 + j < nchunks) ? hist[(size_t)(c0 + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (c0 + j < nchunks) hist[(size_t)(c0 + j) * E + e] = run;
                run += v[j];
            }
        }
        counts[e] = run;
        cnt[e - e0] = run;
        local += run;
    }
    int total_valid;
    int base = block_exclusive_scan(local, ws, total_valid);
    for (int e = e0; e < e1; ++e) {
        offsets[e] = base;
        for (int c = 0; c < nchunks; ++c) hist[(size_t)c * E + e] += base;
        base += cnt[e - e0];
    }
    if (tid == 0) offsets[E] = total_valid;
    for (int64_t s = (int64_t)total_valid + tid; s < P; s += kScanThreads) {
        sorted_pair_ids[s] = -1;
        if (slot_dest) slot_dest[s] = -1;
    }
    if (tile_start) write_tile_schedule(cnt, e0, e1, E, nmax, ws, tile_start);
}

// The chunk's pairs in pair order onto their slots: cur[e] enters as the
// chunk's first slot of expert e and is advanced past the chunk's pairs.
// With slot_dest, each slot also gets its token-tile row
// tile_start[e] * nmax + (slot - offsets[e]) (offsets and tile_start are
// complete in global memory: written before this CTA's barrier, or by an
// earlier kernel; read from L2), and pair_dest[p] the same row of pair p
// (-1 for an invalid id).
__device__ void scatter_chunk(const int32_t* __restrict__ ids, int64_t P, int E, int64_t p0, int32_t* cur,
                              int32_t* __restrict__ sorted_pair_ids, int32_t* __restrict__ pair_slot,
                              const int32_t* offsets, const int32_t* tile_start, int nmax, int32_t* slot_dest,
                              int32_t* pair_dest) {
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int round = 0; round < kChunk / kThreads; ++round) {
        const int64_t r0 = p0 + round * kThreads;
        if (r0 >= P) break;  // CTA-uniform
        // only warps that hold pairs of this round take a turn
        const int64_t warps_left = (P - r0 + 31) / 32;
        const int nw = warps_left < kThreads / 32 ? (int)warps_left : kThreads / 32;
        const int64_t p = r0 + tid;
        int e = -1;
        if (p < P) e = ids[p];
        const bool valid = (p < P) && e >= 0 && e < E;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1);
        const uint32_t before = peers & lanemask_lt();
        int slot = -1;
        for (int w = 0; w < nw; ++w) {
            if (warp == w) {
                if (valid) slot = cur[e] + __popc(before);
                __syncwarp();
                if (valid && before == 0) cur[e] += __popc(peers);
            }
            __syncthreads();
        }
        if (p < P) {
            pair_slot[p] = slot;
            int dst = -1;
            if (valid) {
                sorted_pair_ids[slot] = (int32_t)p;
                if (slot_dest) {
                    dst = __ldcg(tile_start + e) * nmax + slot - __ldcg(offsets + e);
                    slot_dest[slot] = dst;
                }
            }
            if (pair_dest) pair_dest[p] = dst;
        }
    }
}

// Stable scatter: the CTA walks its chunk in two rounds of 1024 pairs; inside
// a round the 32 warps take turns (in pair order) on the per-expert cursors,
// each warp ranking equal ids among its lanes with match-any.  A pair's slot
// is therefore its chunk base + the number of earlier pairs of the same
// expert in the chunk: the stable counting sort.
__global__ void __launch_bounds__(kThreads)
align_scatter_kernel(const int32_t* __restrict__ ids, int64_t P, int E, int nchunks,
                     const int32_t* __restrict__ hist, int32_t* __restrict__ sorted_pair_ids,
                     int32_t* __restrict__ pair_slot, const int32_t* __restrict__ offsets,
                     const int32_t* __restrict__ tile_start, int nmax, int32_t* __restrict__ slot_dest,
                     int32_t* __restrict__ pair_dest) {
    extern __shared__ int32_t cur[];
    const int tid = threadIdx.x;
    pdl_sync();
    const int32_t* base = hist + (size_t)blockIdx.x * E;
    for (int e = tid; e < E; e += kThreads) cur[e] = base[e];
    __syncthreads();
    scatter_chunk(ids, P, E, (int64_t)blockIdx.x * kChunk, cur, sorted_pair_ids, pair_slot, offsets, tile_start, nmax,
                  slot_dest, pair_dest);
}

// One CTA for at most one chunk of pairs: histogram, scan (counts, offsets,
// tile schedule) and the stable scatter of the three-launch path, in one launch.
__global__ void __launch_bounds__(kThreads)
align_small_kernel(const int32_t* __restrict__ ids, int64_t P, int E, int nmax, int32_t* __restrict__ counts,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_pair_ids,
                   int32_t* __restrict__ pair_slot, int32_t* __restrict__ tile_start, int32_t* __restrict__ slot_dest,
                   int32_t* __restrict__ pair_dest, int32_t* __restrict__ dev_status) {
    extern __shared__ int32_t cur[];  // per-expert counts, then cursors
    __shared__ int32_t ws[33];
    const int tid = threadIdx.x;
    pdl_sync();
    for (int e = tid; e < E; e += kThreads) cur[e] = 0;
    __syncthreads();
    int bad = 0;
    for (int64_t p = tid; p < P; p += kThreads) {
        const int e = ids[p];
        if (e >= 0 && e < E)
            atomicAdd(&cur[e], 1);
        else
            bad = 1;
    }
    if (__syncthreads_or(bad) && tid == 0) atomicOr(dev_status, QMOE_DEV_BAD_EXPERT_ID);
    const int per = (E + kThreads - 1) / kThreads;  // <= 4
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int cnt[4] = {0, 0, 0, 0};
    int local = 0;
    for (int e = e0; e < e1; ++e) {
        cnt[e - e0] = cur[e];
        local += cnt[e - e0];
    }
    int total_valid;
    int base = block_exclusive_scan(local, ws, total_valid);  // also orders the reads above before the writes
    for (int e = e0; e < e1; ++e) {
        counts[e] = cnt[e - e0];
        offsets[e] = base;
        cur[e] = base;
        base += cnt[e - e0];
    }
    if (tid == 0) offsets[E] = total_valid;
    for (int64_t s = (int64_t)total_valid + tid; s < P; s += kThreads) {
        sorted_pair_ids[s] = -1;
        if (slot_dest) slot_dest[s] = -1;
    }
    if (tile_start) write_tile_schedule(cnt, e0, e1, E, nmax, ws, tile_start);
    __syncthreads();
    scatter_chunk(ids, P, E, 0, cur, sorted_pair_ids, pair_slot, offsets, tile_start, nmax, slot_dest, pair_dest);
}

size_t align_ws_bytes(int64_t P, int E) {
    const int64_t nchunks = (P + kChunk - 1) / kChunk;
    return (size_t)((nchunks * E * 4 + 255) / 256 * 256);
}

int align_sort_launch(int64_t P, int E, const int32_t* ids, int32_t* counts, int32_t* offsets,
                      int32_t* sorted_pair_ids, int32_t* pair_slot, int32_t* dev_status, int32_t* hist,
                      int nmax, int32_t* tile_start, cudaStream_t stream) {
    const int nchunks = (int)((P + kChunk - 1) / kChunk);
    const size_t smem = (size_t)E * sizeof(int32_t);
    int32_t* slot_dest = tile_start ? tile_start + schedule_ints(E) : nullptr;
    int32_t* pair_dest = slot_dest ? slot_dest + slot_ints(P) : nullptr;
    if (smem > 48 * 1024) {
        cudaFuncSetAttribute(align_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(align_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(align_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    }
    if (nchunks <= 1)
        return launch_pdl(align_small_kernel, 1, kThreads, smem, stream, ids, P, E, nmax, counts, offsets,
                          sorted_pair_ids, pair_slot, tile_start, slot_dest, pair_dest, dev_status);
    int rc = launch_pdl(align_hist_kernel, nchunks, kThreads, smem, stream, ids, P, E, nchunks, hist, dev_status);
    if (rc == QMOE_OK)
        rc = launch_pdl(align_scan_kernel, 1, kScanThreads, 0, stream, hist, P, E, nchunks, nmax, counts, offsets,
                        sorted_pair_ids, tile_start, slot_dest);
    if (rc == QMOE_OK)
        rc = launch_pdl(align_scatter_kernel, nchunks, kThreads, smem, stream, ids, P, E, nchunks, hist,
                        sorted_pair_ids, pair_slot, offsets, tile_start, nmax, slot_dest, pair_dest);
    return rc;
}

// Where the tile schedule lives inside the routing workspace.
int32_t* tile_schedule_in(void* ws, const qmoe_dims* d) {
    return reinterpret_cast<int32_t*>(static_cast<char*>(ws) + align_ws_bytes((int64_t)d->T * d->k, d->E));
}

}  // namespace qmoe

extern "C" size_t qmoe_workspace_bytes(const qmoe_dims* d) {
    if (!qmoe::dims_ok(d)) return 0;
    const int64_t P = (int64_t)d->T * d->k;
    // histograms, the GEMM schedule (tile offsets over experts), each slot's and each pair's token-tile row
    return qmoe::align_ws_bytes(P, d->E) + (size_t)(qmoe::schedule_ints(d->E) + 2 * qmoe::slot_ints(P)) * 4;
}

extern "C" int qmoe_align_sort(const qmoe_dims* d, const int32_t* topk_ids, int32_t* counts, int32_t* offsets,
                               int32_t* sorted_pair_ids, int32_t* pair_slot, int32_t* dev_status, void* ws,
                               size_t ws_bytes, qmoe_stream_t stream) {
    using namespace qmoe;
    if (!dims_ok(d)) return QMOE_ERR_ARG;
    const int64_t P = (int64_t)d->T * d->k;
    if (!counts || !offsets || !dev_status || !ws) return QMOE_ERR_ARG;
    if (P > 0 && (!topk_ids || !sorted_pair_ids || !pair_slot)) return QMOE_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return QMOE_ERR_ARG;
    if (d->E > kMaxExperts) return QMOE_ERR_UNSUPPORTED;
    if (ws_bytes < align_ws_bytes(P, d->E)) return QMOE_ERR_ARG;
    if (ws_bytes < qmoe_workspace_bytes(d)) return QMOE_ERR_ARG;
    return align_sort_launch(P, d->E, topk_ids, counts, offsets, sorted_pair_ids, pair_slot, dev_status,
                             static_cast<int32_t*>(ws), mxt::nmax_for(d), tile_schedule_in(ws, d),
                             (cudaStream_t)stream);
}
