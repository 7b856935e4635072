// Internal declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Device-side copy of the validated forward arguments.
struct FwdParams {
    int B, T, H, dk, dv;
    int gate_kind;          // kda_gate
    int scale_v;            // beta scales v
    int has_beta;
    const void *q, *k, *v, *g, *beta;
    const float *h0;
    void *o;
    float *ht;
    int *status;            // first word of the workspace
};

// Device-side copy of the validated DPLR arguments.
struct DplrParams {
    int B, T, H, dk, dv;
    int gate_kind;          // kda_gate
    const void *q, *k, *v, *a, *b, *g;
    const float *h0;
    void *o;
    float *ht;
    int *status;            // first word of the workspace
};

// Device status codes written into the workspace word (first error wins).
enum : int { kDevOk = 0, kDevTimeout = 1 };

// float32 CUDA-core path (any gate kind; inputs float32).
cudaError_t launch_fwd_simt_f32(const FwdParams &p, int g_is_bf16, cudaStream_t s);

// bf16 tcgen05 path; returns cudaErrorNotSupported for shapes it does not take.
cudaError_t launch_fwd_tc_bf16(const FwdParams &p, int g_is_bf16, cudaStream_t s);

// float32 CUDA-core DPLR chunk forward (inputs float32 or bf16).
cudaError_t launch_dplr_fwd_simt(const DplrParams &p, int in_bf16, int g_is_bf16, cudaStream_t s);

// Per-token transition norms; maxes (2 floats) is cleared on the stream first.
cudaError_t launch_dplr_factor_norms(const DplrParams &p, int in_bf16, int g_is_bf16, float *rho, float *nrm,
                                     float *maxes, cudaStream_t s);

}  // namespace kda
