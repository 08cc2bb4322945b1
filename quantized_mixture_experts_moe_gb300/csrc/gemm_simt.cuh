// Arguments of the grouped W8A8 SIMT GEMM launcher.
#pragma once
#include <stdint.h>
#include <cuda_runtime.h>

namespace qmoe {

struct SimtArgs {
    int T, k, H, I, E;
    const void* act;        // stage 1: int8 activations [T, H]; stage 2: int8 intermediate [P, I] (slot order)
    const void* act_s;      // fp32 per-row activation / intermediate scales
    const void* w;          // int8 expert weights
    const void* w_s;        // fp32 per-output-row weight scales
    const int32_t* offsets; // [E+1]
    const int32_t* sorted;  // [P] slot -> pair id (stage 1)
    void* out;              // stage 1: fp32 h [P, I]; stage 2: y bf16 [P, H]
    int32_t* dbg_acc;       // raw int32 accumulators (nullable)
};

int gemm_simt_w8a8(int stage, const SimtArgs& a, cudaStream_t st);

}  // namespace qmoe
