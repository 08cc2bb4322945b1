// Expert-sorted permutation of routed top-k pairs (qmoe_align_sort).
//
// Grouping all experts' projections into one launch needs the pairs ordered by
// expert, and the scatter back must keep a deterministic order ("perf(qmoe):
// group prefill expert matmuls", description).  The order here is the stable
// one: within an expert, slots follow ascending pair id p = t*k + j.
//
// Up to 2048 pairs (one chunk) a single CTA does all of it in one launch;
// above, two launches, none of which lets an atomic decide an order:
//   1. hist:    each CTA owns a contiguous chunk of kChunk pairs and counts
//               them per expert (shared-memory counters).
//   2. scatter: each CTA sums the [chunk][expert] histograms into per-expert
//               totals and its chunk's base slots (the exclusive prefix over
//               chunks plus the expert's offset, from a block scan), then
//               walks its chunk in pair order: a pair's slot is its chunk base
//               plus the number of earlier pairs of the same expert, counted
//               per warp, so the result is the stable counting sort.  CTA 0
//               writes counts and offsets.
// The scan also derives the GEMMs' token-tile schedule, and the scatter
// gives every slot and every pair its row in the token tiles (so the permute
// and intermediate kernels look it up instead of searching the offsets).
#include "qmoe_common.cuh"
#include "mx_tiles.cuh"

namespace qmoe {

constexpr int kChunk = 2048;          // pairs per chunk (one CTA)
constexpr int kThreads = 1024;        // threads per CTA in hist/scatter (two rounds per chunk)
constexpr int kMaxExperts = 4096;     // shared-memory counter bound

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

// Per-expert totals and this chunk's bases from the [chunk][expert] histogram
// (every CTA of the scatter launch does this for itself), then the offsets and
// the token-tile schedule by block scans: offs/tst are this CTA's copies in
// shared memory; CTA 0 also writes counts, offsets, tile_start and the -1 tail
// of the sorted ids to global memory.
__device__ void scan_chunk_bases(const int32_t* __restrict__ hist, int64_t P, int E, int nchunks, int chunk, int nmax,
                                 int32_t* cur, int32_t* offs, int32_t* tst, int32_t* ws, int32_t* __restrict__ counts,
                                 int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_pair_ids,
                                 int32_t* __restrict__ tile_start, int32_t* __restrict__ slot_dest) {
    const int tid = threadIdx.x;
    const bool writer = chunk == 0;
    const int per = (E + kThreads - 1) / kThreads;  // <= 4 (E <= kMaxExperts)
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int cnt[4] = {0, 0, 0, 0}, pre[4] = {0, 0, 0, 0};
    int local = 0;
    for (int e = e0; e < e1; ++e) {
        int run = 0, mine = 0;
        for (int c0 = 0; c0 < nchunks; c0 += 8) {  // loads issued eight at a time so they overlap
            int32_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = (c0 + j < nchunks) ? hist[(size_t)(c0 + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (c0 + j == chunk) mine = run;
                run += v[j];
            }
        }
        cnt[e - e0] = run;
        pre[e - e0] = mine;
        local += run;
    }
    int total_valid;
    int base = block_exclusive_scan(local, ws, total_valid);
    for (int e = e0; e < e1; ++e) {
        offs[e] = base;
        cur[e] = base + pre[e - e0];
        if (writer) {
            counts[e] = cnt[e - e0];
            offsets[e] = base;
        }
        base += cnt[e - e0];
    }
    if (tid == 0) {
        offs[E] = total_valid;
        if (writer) offsets[E] = total_valid;
    }
    if (tile_start) {
        int lt = 0;
        for (int e = e0; e < e1; ++e) lt += (cnt[e - e0] + nmax - 1) / nmax;
        int ntiles;
        int tb = block_exclusive_scan(lt, ws, ntiles);
        for (int e = e0; e < e1; ++e) {
            tst[e] = tb;
            if (writer) tile_start[e] = tb;
            tb += (cnt[e - e0] + nmax - 1) / nmax;
        }
        if (tid == 0) {
            tst[E] = ntiles;
            if (writer) tile_start[E] = ntiles;
        }
    }
    if (writer)
        for (int64_t s = (int64_t)total_valid + tid; s < P; s += kThreads) {
            sorted_pair_ids[s] = -1;
            if (slot_dest) slot_dest[s] = -1;
        }
}

// The chunk's pairs in pair order onto their slots: cur[e] enters as the
// chunk's first slot of expert e and is advanced past the chunk's pairs.  Per
// round of 1024 pairs each warp counts its pairs per expert (one byte per
// warp and expert in wcnt: at most 32); a pair's slot is cur[e] plus the
// counts of the earlier warps plus its rank among its own warp's equal ids,
// so the order is the stable one with four barriers a round.  With
// slot_dest, each slot also gets its token-tile row
// tst[e] * nmax + (slot - offs[e]), and pair_dest[p] the same row of pair p
// (-1 for an invalid id).
__device__ void scatter_chunk(const int32_t* __restrict__ ids, int64_t P, int E, int64_t p0, int32_t* cur,
                              uint8_t* wcnt, int32_t* __restrict__ sorted_pair_ids, int32_t* __restrict__ pair_slot,
                              const int32_t* offs, const int32_t* tst, int nmax, int32_t* slot_dest,
                              int32_t* pair_dest) {
    const int tid = threadIdx.x, warp = tid >> 5;
    uint32_t* wz = reinterpret_cast<uint32_t*>(wcnt);  // 32 * E bytes: a multiple of 4
    for (int round = 0; round < kChunk / kThreads; ++round) {
        const int64_t r0 = p0 + round * kThreads;
        if (r0 >= P) break;  // CTA-uniform
        for (int i = tid; i < 8 * E; i += kThreads) wz[i] = 0u;
        __syncthreads();
        const int64_t p = r0 + tid;
        int e = -1;
        if (p < P) e = ids[p];
        const bool valid = (p < P) && e >= 0 && e < E;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1);
        const uint32_t before = peers & lanemask_lt();
        if (valid && before == 0) wcnt[warp * E + e] = (uint8_t)__popc(peers);
        __syncthreads();
        int slot = -1;
        if (valid) {
            int pre = 0;
            for (int w = 0; w < warp; ++w) pre += wcnt[w * E + e];
            slot = cur[e] + pre + __popc(before);
        }
        __syncthreads();  // every read of cur for these 1024 pairs is done
        for (int ee = tid; ee < E; ee += kThreads) {
            int add = 0;
#pragma unroll 8
            for (int w = 0; w < 32; ++w) add += wcnt[w * E + ee];
            cur[ee] += add;
        }
        if (p < P) {
            pair_slot[p] = slot;
            int dst = -1;
            if (valid) {
                sorted_pair_ids[slot] = (int32_t)p;
                if (slot_dest) {
                    dst = tst[e] * nmax + slot - offs[e];
                    slot_dest[slot] = dst;
                }
            }
            if (pair_dest) pair_dest[p] = dst;
        }
        __syncthreads();  // wcnt and cur settled before the next round
    }
}

// Shared memory of the scan-and-scatter kernels: cur[E], offs[E+1], tst[E+1] ints, then the
// per-warp expert counts (32 x E bytes).
inline size_t scatter_smem_bytes(int E) { return (size_t)(3 * E + 2) * 4 + (size_t)32 * E; }

// Second launch of the multi-chunk path: each CTA derives its chunk's bases
// (and the offsets and tile schedule) from the histograms, then scatters its
// chunk.  CTA 0 writes the per-expert outputs.
__global__ void __launch_bounds__(kThreads)
align_scan_scatter_kernel(const int32_t* __restrict__ ids, int64_t P, int E, int nchunks,
                          const int32_t* __restrict__ hist, int nmax, int32_t* __restrict__ counts,
                          int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_pair_ids,
                          int32_t* __restrict__ pair_slot, int32_t* __restrict__ tile_start,
                          int32_t* __restrict__ slot_dest, int32_t* __restrict__ pair_dest) {
    extern __shared__ int32_t sm[];
    int32_t* cur = sm;
    int32_t* offs = cur + E;
    int32_t* tst = offs + E + 1;
    uint8_t* wcnt = reinterpret_cast<uint8_t*>(tst + E + 1);
    __shared__ int32_t ws[33];
    pdl_sync();
    scan_chunk_bases(hist, P, E, nchunks, blockIdx.x, nmax, cur, offs, tst, ws, counts, offsets, sorted_pair_ids,
                     tile_start, slot_dest);
    __syncthreads();
    scatter_chunk(ids, P, E, (int64_t)blockIdx.x * kChunk, cur, wcnt, sorted_pair_ids, pair_slot, offs, tst, nmax,
                  slot_dest, pair_dest);
}

// One CTA for at most one chunk of pairs: histogram, scan (counts, offsets,
// tile schedule) and the stable scatter, in one launch.
__global__ void __launch_bounds__(kThreads)
align_small_kernel(const int32_t* __restrict__ ids, int64_t P, int E, int nmax, int32_t* __restrict__ counts,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_pair_ids,
                   int32_t* __restrict__ pair_slot, int32_t* __restrict__ tile_start, int32_t* __restrict__ slot_dest,
                   int32_t* __restrict__ pair_dest, int32_t* __restrict__ dev_status) {
    extern __shared__ int32_t sm[];
    int32_t* cur = sm;  // per-expert counts, then cursors
    int32_t* offs = cur + E;
    int32_t* tst = offs + E + 1;
    uint8_t* wcnt = reinterpret_cast<uint8_t*>(tst + E + 1);
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
        offs[e] = base;
        cur[e] = base;
        base += cnt[e - e0];
    }
    if (tid == 0) {
        offsets[E] = total_valid;
        offs[E] = total_valid;
    }
    for (int64_t s = (int64_t)total_valid + tid; s < P; s += kThreads) {
        sorted_pair_ids[s] = -1;
        if (slot_dest) slot_dest[s] = -1;
    }
    if (tile_start) {
        int lt = 0;
        for (int e = e0; e < e1; ++e) lt += (cnt[e - e0] + nmax - 1) / nmax;
        int ntiles;
        int tb = block_exclusive_scan(lt, ws, ntiles);
        for (int e = e0; e < e1; ++e) {
            tst[e] = tb;
            tile_start[e] = tb;
            tb += (cnt[e - e0] + nmax - 1) / nmax;
        }
        if (tid == 0) {
            tst[E] = ntiles;
            tile_start[E] = ntiles;
        }
    }
    __syncthreads();
    scatter_chunk(ids, P, E, 0, cur, wcnt, sorted_pair_ids, pair_slot, offs, tst, nmax, slot_dest, pair_dest);
}

size_t align_ws_bytes(int64_t P, int E) {
    const int64_t nchunks = (P + kChunk - 1) / kChunk;
    return (size_t)((nchunks * E * 4 + 255) / 256 * 256);
}

int align_sort_launch(int64_t P, int E, const int32_t* ids, int32_t* counts, int32_t* offsets,
                      int32_t* sorted_pair_ids, int32_t* pair_slot, int32_t* dev_status, int32_t* hist,
                      int nmax, int32_t* tile_start, cudaStream_t stream) {
    const int nchunks = (int)((P + kChunk - 1) / kChunk);
    const size_t hsmem = (size_t)E * sizeof(int32_t);
    const size_t ssmem = scatter_smem_bytes(E);
    int32_t* slot_dest = tile_start ? tile_start + schedule_ints(E) : nullptr;
    int32_t* pair_dest = slot_dest ? slot_dest + slot_ints(P) : nullptr;
    if (hsmem > 48 * 1024)
        cudaFuncSetAttribute(align_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hsmem);
    if (ssmem > 48 * 1024) {
        cudaFuncSetAttribute(align_scan_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssmem);
        cudaFuncSetAttribute(align_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssmem);
    }
    if (nchunks <= 1)
        return launch_pdl(align_small_kernel, 1, kThreads, ssmem, stream, ids, P, E, nmax, counts, offsets,
                          sorted_pair_ids, pair_slot, tile_start, slot_dest, pair_dest, dev_status);
    int rc = launch_pdl(align_hist_kernel, nchunks, kThreads, hsmem, stream, ids, P, E, nchunks, hist, dev_status);
    if (rc == QMOE_OK)
        rc = launch_pdl(align_scan_scatter_kernel, nchunks, kThreads, ssmem, stream, ids, P, E, nchunks, hist, nmax,
                        counts, offsets, sorted_pair_ids, pair_slot, tile_start, slot_dest, pair_dest);
    return rc;
}

// Kernels align_sort_launch starts for P pairs: one CTA's single launch up to
// one chunk, else the histogram and the scan-and-scatter.
int align_sort_launches(int64_t P) { return (P + kChunk - 1) / kChunk <= 1 ? 1 : 2; }

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
