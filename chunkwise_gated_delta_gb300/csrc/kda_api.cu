// C-ABI layer: argument validation, workspace query, dispatch, status words.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"
#include "kda_internal.h"

namespace {

constexpr size_t kStatusBytes = 256;   // the status word, padded to one aligned block

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t dtype_size(kda_dtype d) { return d == KDA_F32 ? 4 : 2; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || !na || !nb) return false;
    auto x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

kda_status validate(const kda_fwd_args *a) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->B < 1 || a->T < 1 || a->H < 1) return KDA_ERR_INVALID_ARG;
    if (a->dk < 1 || a->dv < 1) return KDA_ERR_INVALID_ARG;
    if (a->chunk != 0 && a->chunk < 1) return KDA_ERR_INVALID_ARG;
    if (a->dtype != KDA_BF16 && a->dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
    if (a->g_dtype != KDA_BF16 && a->g_dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
    if (a->gate_kind != KDA_GATE_NONE && a->gate_kind != KDA_GATE_SCALAR && a->gate_kind != KDA_GATE_CHANNEL)
        return KDA_ERR_INVALID_ARG;
    if ((a->gate_kind == KDA_GATE_NONE) != (a->g == nullptr)) return KDA_ERR_INVALID_ARG;
    if (a->flags & ~KDA_FLAG_BETA_SCALES_V) return KDA_ERR_INVALID_ARG;
    if (!a->q || !a->k || !a->v || !a->o) return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {a->q, a->k, a->v, a->g, a->beta, a->h0, a->o, a->ht, a->workspace};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    // sizes: reject products that overflow 63 bits
    const double elems = (double)a->B * a->T * a->H * (a->dk > a->dv ? a->dk : a->dv);
    if (elems > 9.0e18 / 8 || (double)a->B * a->T * a->H > 2.0e9) return KDA_ERR_INVALID_ARG;
    if (a->dk != 64 && a->dk != 128) return KDA_ERR_UNSUPPORTED;
    if (a->dv != 64 && a->dv != 128) return KDA_ERR_UNSUPPORTED;
    if (a->chunk != 0 && a->chunk != 64) return KDA_ERR_UNSUPPORTED;
    // outputs must not alias inputs
    const size_t es = dtype_size(a->dtype);
    const size_t nbt = (size_t)a->B * a->T * a->H;
    const size_t o_bytes = nbt * a->dv * es;
    const size_t state_bytes = (size_t)a->B * a->H * a->dv * a->dk * 4;
    const size_t ht_bytes = a->ht ? state_bytes : 0;
    const size_t g_bytes = a->gate_kind == KDA_GATE_CHANNEL ? nbt * a->dk * dtype_size(a->g_dtype)
                           : a->gate_kind == KDA_GATE_SCALAR ? nbt * dtype_size(a->g_dtype) : 0;
    struct R { const void *p; size_t n; } ins[] = {
        {a->q, nbt * a->dk * es}, {a->k, nbt * a->dk * es}, {a->v, nbt * a->dv * es}, {a->g, g_bytes},
        {a->beta, a->beta ? nbt * es : 0}, {a->h0, a->h0 ? state_bytes : 0},
        {a->workspace, a->workspace_bytes}};
    for (const R &r : ins) {
        if (overlaps(a->o, o_bytes, r.p, r.n)) return KDA_ERR_INVALID_ARG;
        if (overlaps(a->ht, ht_bytes, r.p, r.n)) return KDA_ERR_INVALID_ARG;
    }
    if (overlaps(a->o, o_bytes, a->ht, ht_bytes)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

}  // namespace

extern "C" {

size_t kda_chunk_fwd_workspace(const kda_fwd_args *args) {
    if (validate(args) != KDA_OK) return 0;
    return kStatusBytes;
}

kda_status kda_chunk_fwd(const kda_fwd_args *args, kda_stream_t stream) {
    kda_status st = validate(args);
    if (st != KDA_OK) return st;
    if (!args->workspace || args->workspace_bytes < kStatusBytes) return KDA_ERR_WORKSPACE;

    kda::FwdParams p{};
    p.B = args->B; p.T = args->T; p.H = args->H; p.dk = args->dk; p.dv = args->dv;
    p.gate_kind = args->gate_kind;
    p.scale_v = (args->flags & KDA_FLAG_BETA_SCALES_V) ? 1 : 0;
    p.has_beta = args->beta != nullptr;
    p.q = args->q; p.k = args->k; p.v = args->v; p.g = args->g; p.beta = args->beta;
    p.h0 = args->h0; p.o = args->o; p.ht = args->ht;
    p.status = static_cast<int *>(args->workspace);

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int g_bf16 = args->g_dtype == KDA_BF16;
    cudaError_t e;
    if (args->dtype == KDA_F32)
        e = kda::launch_fwd_simt_f32(p, g_bf16, s);
    else
        e = kda::launch_fwd_tc_bf16(p, g_bf16, s);
    if (e == cudaErrorNotSupported) return KDA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_status_read(void *workspace, kda_stream_t stream) {
    if (!workspace || !aligned16(workspace)) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (word != kda::kDevOk) {
        if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return KDA_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    return word == kda::kDevOk ? KDA_OK : word == kda::kDevTimeout ? KDA_ERR_TIMEOUT : KDA_ERR_CUDA;
}

const char *kda_status_string(kda_status status) {
    switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported configuration";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

}  // extern "C"
