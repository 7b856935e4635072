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
    const int *cu_seqlens;  // packed sequences: [B + 1] row offsets into a [1, T, H, d] batch, or null
    uint8_t *zrec;          // bf16 path: Z records (fwd_zrec_bytes), or null to build Z in the scan kernel
    int strong_token;       // nonzero, new for every call: see kStatusStrongWord
};

// Device-side copy of the validated DPLR arguments.
struct DplrParams {
    int B, T, H, dk, dv;
    int gate_kind;          // kda_gate
    int clip;               // clip the decay to 1/rho (eq. (7) of "How to make GDN2 more stable")
    const void *q, *k, *v, *a, *b, *g;
    const float *h0;
    void *o;
    float *ht;
    int *status;            // first word of the workspace
    // backward only
    const void *grad_o;
    const float *grad_ht;
    void *grad_q, *grad_k, *grad_v, *grad_a, *grad_b, *grad_g;
    float *grad_h0;
    // workspace arrays, by head, then chunk slot: NS = B ceil(T / C) slots for dense
    // batches, B + ceil(T / C) for packed sequences (dplr_bwd_carve)
    float *ws_S;            // [H, NS + B, dv, dk] states before each chunk, then the final state
    float *ws_dS;           // [H, NS, dv, dk] gradients of the state after each chunk
    float *ws_prep;         // [H, NS] chunk records (state-independent operands)
    float *ws_x;            // backward: [H, NS, C, dv] X of every chunk
    float *ws_dc;           // backward: [H, NS, C, dv] dC of every chunk
    const int *cu_seqlens;  // packed sequences: [B + 1] row offsets into a [1, T, H, d] batch, or null
};

// Device-side copy of the validated backward arguments.
struct BwdParams {
    int B, T, H, dk, dv;
    int gate_kind;          // kda_gate
    int scale_v;            // beta scales v
    int has_beta;
    const void *q, *k, *v, *g, *beta;
    const float *h0;
    const void *grad_o;     // [B, T, H, dv]
    const float *grad_ht;   // [B, H, dv, dk] or null
    void *grad_q, *grad_k, *grad_v, *grad_g, *grad_beta;
    float *grad_h0;
    // workspace arrays, by head, then chunk slot (bwd_carve): NS = B ceil(T / 32) slots for
    // dense batches, B + ceil(T / 32) for packed sequences
    float *ws_S;            // [H, NS + B, dv, dk] states before each chunk, then the final state
    float *ws_dS;           // [H, NS, dv, dk] gradients of the state after each chunk
    float *ws_prep;         // [H, NS] chunk records (state-independent operands)
    float *ws_vnew;         // [H, NS, C, dv] V_new of every chunk
    float *ws_du;           // [H, NS, C, dv] dU of every chunk
    int *status;
    const int *cu_seqlens;  // packed sequences: [B + 1] row offsets into a [1, T, H, d] batch, or null
};

// Device status codes written into the workspace word (first error wins).
enum : int { kDevOk = 0, kDevTimeout = 1, kDevDecayRange = 2 };
// Word of the 256-byte status block that holds the polling budget of the bounded waits
// (iterations before a wait gives up; 0 = the library default).
constexpr int kStatusBoundWord = 7;
// Word where the single-kernel bf16 forward notes the call's strong_token when a chunk's decay
// is past the one-product Gram's range; a second launch then redoes the call with the sub-chunk
// Gram, and exits at once when the word holds another call's token.
constexpr int kStatusStrongWord = 8;

// float32 CUDA-core path (any gate kind; inputs float32).
cudaError_t launch_fwd_simt_f32(const FwdParams &p, int g_is_bf16, cudaStream_t s);

// bf16 tcgen05 path; returns cudaErrorNotSupported for shapes it does not take.
cudaError_t launch_fwd_tc_bf16(const FwdParams &p, int g_is_bf16, cudaStream_t s);
// Bytes of Z records the bf16 forward uses (16 KB per chunk slot and head).
size_t fwd_zrec_bytes(int B, int T, int H, bool packed);

// float32 CUDA-core DPLR chunk forward (inputs float32 or bf16) and the bytes
// of chunk records it keeps in the workspace.
size_t dplr_fwd_record_bytes(int B, int T, int H, int dk, int dv, bool packed);
cudaError_t launch_dplr_fwd_simt(const DplrParams &p, int in_bf16, int g_is_bf16, cudaStream_t s);

// float32 CUDA-core DPLR backward (inputs float32 or bf16), its workspace bytes and the
// carving of those bytes (at ws, 16-byte aligned) into p's ws_* arrays.
cudaError_t launch_dplr_bwd_simt(const DplrParams &p, int in_bf16, int g_is_bf16, cudaStream_t s);
size_t dplr_bwd_state_bytes(int B, int T, int H, int dk, int dv, bool packed);
void dplr_bwd_carve(DplrParams &p, float *ws);

// Per-token transition norms; maxes (2 floats) is cleared on the stream first.
cudaError_t launch_dplr_factor_norms(const DplrParams &p, int in_bf16, int g_is_bf16, float *rho, float *nrm,
                                     float *maxes, cudaStream_t s);

// Backward: bytes of chunk states, records and chunk products the kernels keep in the
// workspace, and the carving of those bytes (at ws, 16-byte aligned) into p's ws_* arrays.
size_t bwd_state_bytes(int B, int T, int H, int dk, int dv, bool packed);
void bwd_carve(BwdParams &p, float *ws);

// float32 CUDA-core backward (inputs float32 or bf16).
cudaError_t launch_bwd_simt(const BwdParams &p, int in_bf16, int g_is_bf16, cudaStream_t s);

}  // namespace kda
