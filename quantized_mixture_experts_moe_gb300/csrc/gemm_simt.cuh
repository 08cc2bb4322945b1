// Arguments of the grouped expert GEMM launchers.
#pragma once
#include <stdint.h>
#include <cuda_runtime.h>

namespace qmoe {

struct SimtArgs {
    int T, k, H, I, E;
    const void* act;        // stage 1: activations [T, H]; stage 2: intermediate [P, I] (slot order)
    const void* act_s;      // activation / intermediate scales (scheme-dependent)
    const void* w;          // packed expert weights
    const void* w_s;        // weight scales
    const int32_t* offsets; // [E+1]
    const int32_t* sorted;  // [P] slot -> pair id (stage 1)
    void* out;              // stage 1: intermediate; stage 2: y bf16 [P, H]
    void* out_s;            // stage 1 MXFP4: intermediate scales
    int32_t* dbg_acc;       // W8A8: raw int32 accumulators (nullable)
};

int gemm_simt(int scheme, int stage, const SimtArgs& a, cudaStream_t st);

}  // namespace qmoe
