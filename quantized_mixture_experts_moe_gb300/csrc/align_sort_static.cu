// qmoe_align_sort_static_scratch: the routing sort without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they route
// tokens: code running inside a framework that owns every allocation through
// its own pool, a plugin whose host forbids cudaMalloc after start-up, or a
// runtime that must not allocate on its latency path.  This entry point gives
// them the same sort as qmoe_align_sort with the per-chunk histogram scratch
// held in a fixed array that lives in device memory for as long as the
// library is loaded.  It allocates nothing: no cudaMalloc, cudaFree or other
// allocating call.
#include <mutex>

#include "qmoe_common.cuh"

namespace qmoe {
size_t align_ws_bytes(int64_t P, int E);
int align_sort_launch(int64_t P, int E, const int32_t* ids, int32_t* counts, int32_t* offsets,
                      int32_t* sorted_pair_ids, int32_t* pair_slot, int32_t* dev_status, int32_t* hist,
                      int nmax, int32_t* tile_start, cudaStream_t stream);
}  // namespace qmoe

// The scratch every call shares: QMOE_STATIC_SCRATCH_BYTES bytes on every GPU
// that loads the library, held until the process exits.  Each call rewrites
// every histogram entry it later reads, so nothing has to start at zero.
static __device__ __align__(256) int32_t g_align_scratch[QMOE_STATIC_SCRATCH_BYTES / sizeof(int32_t)];

namespace {

constexpr int kMaxDevices = 64;
int32_t* g_scratch_ptr[kMaxDevices];  // written once per device, under g_scratch_mu, after a successful lookup
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  The host-side
// name g_align_scratch is only a stand-in for the symbol, never a device
// address, so it is resolved per device with that device current.  Only a
// successful lookup is kept: a failed one (say, a transient error while the
// module loads) is tried again on the next call.
int32_t* scratch_on_current_device(int* status) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = QMOE_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_align_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();  // clear the lookup error so a later launch check does not report it
            *status = QMOE_ERR_CUDA;
            return nullptr;
        }
        g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *status = QMOE_OK;
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int qmoe_align_sort_static_scratch(const qmoe_dims* d, const int32_t* topk_ids, int32_t* counts,
                                              int32_t* offsets, int32_t* sorted_pair_ids, int32_t* pair_slot,
                                              int32_t* dev_status, qmoe_stream_t stream) {
    using namespace qmoe;
    if (!dims_ok(d)) return QMOE_ERR_ARG;
    const int64_t P = (int64_t)d->T * d->k;
    if (!counts || !offsets || !dev_status) return QMOE_ERR_ARG;
    if (P > 0 && (!topk_ids || !sorted_pair_ids || !pair_slot)) return QMOE_ERR_ARG;
    if (d->E > 4096) return QMOE_ERR_UNSUPPORTED;
    if (align_ws_bytes(P, d->E) > (size_t)QMOE_STATIC_SCRATCH_BYTES) return QMOE_ERR_UNSUPPORTED;
    int st = QMOE_OK;
    int32_t* scratch = scratch_on_current_device(&st);
    if (st != QMOE_OK) return st;
    // no GEMM tile schedule here: the GEMM calls take the routing workspace that holds it
    return align_sort_launch(P, d->E, topk_ids, counts, offsets, sorted_pair_ids, pair_slot, dev_status, scratch, 0,
                             nullptr, (cudaStream_t)stream);
}
