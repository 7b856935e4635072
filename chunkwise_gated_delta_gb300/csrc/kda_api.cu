// C-ABI layer: argument validation, workspace query, dispatch, status words.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

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
    if (a->cu_seqlens && (reinterpret_cast<uintptr_t>(a->cu_seqlens) & 3u)) return KDA_ERR_INVALID_ARG;
    // sizes: reject products that overflow 63 bits
    const double elems = (double)a->B * a->T * a->H * (a->dk > a->dv ? a->dk : a->dv);
    if (elems > 9.0e18 / 8 || (double)a->B * a->T * a->H > 2.0e9) return KDA_ERR_INVALID_ARG;
    if (a->dk != 64 && a->dk != 128) return KDA_ERR_UNSUPPORTED;
    if (a->dv != 64 && a->dv != 128) return KDA_ERR_UNSUPPORTED;
    if (a->chunk != 0 && a->chunk != 64) return KDA_ERR_UNSUPPORTED;
    // the tensor-core forward is laid out for 128 key channels (fp32 inputs take 64 too)
    if (a->dtype == KDA_BF16 && a->dk != 128) return KDA_ERR_UNSUPPORTED;
    // the bf16 forward reads a per-channel gate as bf16 tiles
    if (a->dtype == KDA_BF16 && a->gate_kind == KDA_GATE_CHANNEL && a->g_dtype != KDA_BF16)
        return KDA_ERR_UNSUPPORTED;
    // outputs must not alias inputs (packed sequences: one [1, T, H, d] batch)
    const size_t es = dtype_size(a->dtype);
    const size_t nbt = (size_t)(a->cu_seqlens ? 1 : a->B) * a->T * a->H;
    const size_t o_bytes = nbt * a->dv * es;
    const size_t state_bytes = (size_t)a->B * a->H * a->dv * a->dk * 4;
    const size_t ht_bytes = a->ht ? state_bytes : 0;
    const size_t g_bytes = a->gate_kind == KDA_GATE_CHANNEL ? nbt * a->dk * dtype_size(a->g_dtype)
                           : a->gate_kind == KDA_GATE_SCALAR ? nbt * dtype_size(a->g_dtype) : 0;
    struct R { const void *p; size_t n; } ins[] = {
        {a->q, nbt * a->dk * es}, {a->k, nbt * a->dk * es}, {a->v, nbt * a->dv * es}, {a->g, g_bytes},
        {a->beta, a->beta ? nbt * es : 0}, {a->h0, a->h0 ? state_bytes : 0},
        {a->workspace, a->workspace_bytes}, {a->cu_seqlens, a->cu_seqlens ? (size_t)(a->B + 1) * 4 : 0}};
    for (const R &r : ins) {
        if (overlaps(a->o, o_bytes, r.p, r.n)) return KDA_ERR_INVALID_ARG;
        if (overlaps(a->ht, ht_bytes, r.p, r.n)) return KDA_ERR_INVALID_ARG;
    }
    if (overlaps(a->o, o_bytes, a->ht, ht_bytes)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

kda_status validate_dplr_common(const dplr_fwd_args *a) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->B < 1 || a->T < 1 || a->H < 1) return KDA_ERR_INVALID_ARG;
    if (a->dk < 1) return KDA_ERR_INVALID_ARG;
    if (a->chunk != 0 && a->chunk < 1) return KDA_ERR_INVALID_ARG;
    if (a->dtype != KDA_BF16 && a->dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
    if (a->g_dtype != KDA_BF16 && a->g_dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
    if (a->gate_kind != KDA_GATE_NONE && a->gate_kind != KDA_GATE_SCALAR && a->gate_kind != KDA_GATE_CHANNEL)
        return KDA_ERR_INVALID_ARG;
    if ((a->gate_kind == KDA_GATE_NONE) != (a->g == nullptr)) return KDA_ERR_INVALID_ARG;
    if (!a->a || !a->b) return KDA_ERR_INVALID_ARG;
    if (a->flags & ~DPLR_FLAG_CLIP_GATE) return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {a->q, a->k, a->v, a->a, a->b, a->g, a->h0, a->o, a->ht, a->workspace};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (a->cu_seqlens && (reinterpret_cast<uintptr_t>(a->cu_seqlens) & 3u)) return KDA_ERR_INVALID_ARG;
    const double elems = (double)a->B * a->T * a->H * (a->dk > 256 ? a->dk : 256);
    if (elems > 9.0e18 / 8 || (double)a->B * a->T * a->H > 2.0e9) return KDA_ERR_INVALID_ARG;
    if (a->dk != 64 && a->dk != 128) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

kda_status validate_dplr(const dplr_fwd_args *a) {
    kda_status st = validate_dplr_common(a);
    if (st != KDA_OK) return st;
    if (!a->q || !a->k || !a->v || !a->o || a->dv < 1) return KDA_ERR_INVALID_ARG;
    if (a->dv % 32 != 0 || a->dv > 256) return KDA_ERR_UNSUPPORTED;
    if (a->chunk != 0 && a->chunk != 32) return KDA_ERR_UNSUPPORTED;
    const size_t es = dtype_size(a->dtype);
    const size_t nbt = (size_t)(a->cu_seqlens ? 1 : a->B) * a->T * a->H;   // packed: one [1, T, H, d] batch
    const size_t o_bytes = nbt * a->dv * es;
    const size_t state_bytes = (size_t)a->B * a->H * a->dv * a->dk * 4;
    const size_t ht_bytes = a->ht ? state_bytes : 0;
    const size_t g_bytes = a->gate_kind == KDA_GATE_CHANNEL ? nbt * a->dk * dtype_size(a->g_dtype)
                           : a->gate_kind == KDA_GATE_SCALAR ? nbt * dtype_size(a->g_dtype) : 0;
    struct R { const void *p; size_t n; } ins[] = {
        {a->q, nbt * a->dk * es}, {a->k, nbt * a->dk * es}, {a->v, nbt * a->dv * es},
        {a->a, nbt * a->dk * es}, {a->b, nbt * a->dk * es}, {a->g, g_bytes},
        {a->h0, a->h0 ? state_bytes : 0}, {a->workspace, a->workspace_bytes},
        {a->cu_seqlens, a->cu_seqlens ? (size_t)(a->B + 1) * 4 : 0}};
    for (const R &r : ins) {
        if (overlaps(a->o, o_bytes, r.p, r.n)) return KDA_ERR_INVALID_ARG;
        if (overlaps(a->ht, ht_bytes, r.p, r.n)) return KDA_ERR_INVALID_ARG;
    }
    if (overlaps(a->o, o_bytes, a->ht, ht_bytes)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

kda_status validate_bwd(const kda_bwd_args *a) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->B < 1 || a->T < 1 || a->H < 1 || a->dk < 1 || a->dv < 1) return KDA_ERR_INVALID_ARG;
    if (a->chunk != 0 && a->chunk < 1) return KDA_ERR_INVALID_ARG;
    if (a->dtype != KDA_BF16 && a->dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
    if (a->g_dtype != KDA_BF16 && a->g_dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
    if (a->gate_kind != KDA_GATE_NONE && a->gate_kind != KDA_GATE_SCALAR && a->gate_kind != KDA_GATE_CHANNEL)
        return KDA_ERR_INVALID_ARG;
    if ((a->gate_kind == KDA_GATE_NONE) != (a->g == nullptr)) return KDA_ERR_INVALID_ARG;
    if ((a->g == nullptr) != (a->grad_g == nullptr)) return KDA_ERR_INVALID_ARG;
    if ((a->beta == nullptr) != (a->grad_beta == nullptr)) return KDA_ERR_INVALID_ARG;
    if (a->flags & ~KDA_FLAG_BETA_SCALES_V) return KDA_ERR_INVALID_ARG;
    if (!a->q || !a->k || !a->v || !a->grad_o || !a->grad_q || !a->grad_k || !a->grad_v)
        return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {a->q, a->k, a->v, a->g, a->beta, a->h0, a->grad_o, a->grad_ht, a->grad_q,
                          a->grad_k, a->grad_v, a->grad_g, a->grad_beta, a->grad_h0, a->workspace};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (a->cu_seqlens && (reinterpret_cast<uintptr_t>(a->cu_seqlens) & 3u)) return KDA_ERR_INVALID_ARG;
    const double elems = (double)a->B * a->T * a->H * (a->dk > a->dv ? a->dk : a->dv);
    if (elems > 9.0e18 / 8 || (double)a->B * a->T * a->H > 2.0e9) return KDA_ERR_INVALID_ARG;
    if (a->dk != 64 && a->dk != 128) return KDA_ERR_UNSUPPORTED;
    if (a->dv != 64 && a->dv != 128) return KDA_ERR_UNSUPPORTED;
    if (a->chunk != 0 && a->chunk != 32) return KDA_ERR_UNSUPPORTED;
    const size_t es = dtype_size(a->dtype);
    const size_t nbt = (size_t)(a->cu_seqlens ? 1 : a->B) * a->T * a->H;   // packed: one [1, T, H, d] batch
    const size_t state_bytes = (size_t)a->B * a->H * a->dv * a->dk * 4;
    const size_t g_bytes = a->gate_kind == KDA_GATE_CHANNEL ? nbt * a->dk * dtype_size(a->g_dtype)
                           : a->gate_kind == KDA_GATE_SCALAR ? nbt * dtype_size(a->g_dtype) : 0;
    struct R { const void *p; size_t n; };
    const R ins[] = {{a->q, nbt * a->dk * es}, {a->k, nbt * a->dk * es}, {a->v, nbt * a->dv * es},
                     {a->g, g_bytes}, {a->beta, a->beta ? nbt * es : 0}, {a->h0, a->h0 ? state_bytes : 0},
                     {a->grad_o, nbt * a->dv * es}, {a->grad_ht, a->grad_ht ? state_bytes : 0},
                     {a->workspace, a->workspace_bytes},
                     {a->cu_seqlens, a->cu_seqlens ? (size_t)(a->B + 1) * 4 : 0}};
    const R outs[] = {{a->grad_q, nbt * a->dk * es}, {a->grad_k, nbt * a->dk * es},
                      {a->grad_v, nbt * a->dv * es}, {a->grad_g, g_bytes},
                      {a->grad_beta, a->grad_beta ? nbt * es : 0}, {a->grad_h0, a->grad_h0 ? state_bytes : 0}};
    for (const R &o : outs) {
        for (const R &r : ins)
            if (overlaps(o.p, o.n, r.p, r.n)) return KDA_ERR_INVALID_ARG;
        for (const R &o2 : outs)
            if (&o2 != &o && overlaps(o.p, o.n, o2.p, o2.n)) return KDA_ERR_INVALID_ARG;
    }
    return KDA_OK;
}

size_t bwd_workspace_bytes(const kda_bwd_args *a) {
    return kStatusBytes + kda::bwd_state_bytes(a->B, a->T, a->H, a->dk, a->dv, a->cu_seqlens != nullptr);
}

kda::DplrParams dplr_params(const dplr_fwd_args *args) {
    kda::DplrParams p{};
    p.B = args->B; p.T = args->T; p.H = args->H; p.dk = args->dk; p.dv = args->dv;
    p.gate_kind = args->gate_kind;
    p.clip = (args->flags & DPLR_FLAG_CLIP_GATE) ? 1 : 0;
    p.q = args->q; p.k = args->k; p.v = args->v; p.a = args->a; p.b = args->b; p.g = args->g;
    p.h0 = args->h0; p.o = args->o; p.ht = args->ht;
    p.status = static_cast<int *>(args->workspace);
    p.cu_seqlens = args->cu_seqlens;
    return p;
}

kda_status validate_dplr_bwd(const dplr_bwd_args *a) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->B < 1 || a->T < 1 || a->H < 1 || a->dk < 1 || a->dv < 1) return KDA_ERR_INVALID_ARG;
    if (a->chunk != 0 && a->chunk < 1) return KDA_ERR_INVALID_ARG;
    if (a->dtype != KDA_BF16 && a->dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
    if (a->g_dtype != KDA_BF16 && a->g_dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
    if (a->gate_kind != KDA_GATE_NONE && a->gate_kind != KDA_GATE_SCALAR && a->gate_kind != KDA_GATE_CHANNEL)
        return KDA_ERR_INVALID_ARG;
    if ((a->gate_kind == KDA_GATE_NONE) != (a->g == nullptr)) return KDA_ERR_INVALID_ARG;
    if ((a->g == nullptr) != (a->grad_g == nullptr)) return KDA_ERR_INVALID_ARG;
    if (a->flags & ~DPLR_FLAG_CLIP_GATE) return KDA_ERR_INVALID_ARG;
    if (!a->q || !a->k || !a->v || !a->a || !a->b || !a->grad_o || !a->grad_q || !a->grad_k || !a->grad_v ||
        !a->grad_a || !a->grad_b)
        return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {a->q, a->k, a->v, a->a, a->b, a->g, a->h0, a->grad_o, a->grad_ht, a->grad_q, a->grad_k,
                          a->grad_v, a->grad_a, a->grad_b, a->grad_g, a->grad_h0, a->workspace};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (a->cu_seqlens && (reinterpret_cast<uintptr_t>(a->cu_seqlens) & 3u)) return KDA_ERR_INVALID_ARG;
    const double elems = (double)a->B * a->T * a->H * (a->dk > a->dv ? a->dk : a->dv);
    if (elems > 9.0e18 / 8 || (double)a->B * a->T * a->H > 2.0e9) return KDA_ERR_INVALID_ARG;
    if (a->dk != 64 && a->dk != 128) return KDA_ERR_UNSUPPORTED;
    if (a->dv != 64 && a->dv != 128) return KDA_ERR_UNSUPPORTED;
    if (a->chunk != 0 && a->chunk != 16) return KDA_ERR_UNSUPPORTED;
    const size_t es = dtype_size(a->dtype);
    const size_t nbt = (size_t)(a->cu_seqlens ? 1 : a->B) * a->T * a->H;   // packed: one [1, T, H, d] batch
    const size_t state_bytes = (size_t)a->B * a->H * a->dv * a->dk * 4;
    const size_t g_bytes = a->gate_kind == KDA_GATE_CHANNEL ? nbt * a->dk * dtype_size(a->g_dtype)
                           : a->gate_kind == KDA_GATE_SCALAR ? nbt * dtype_size(a->g_dtype) : 0;
    struct R { const void *p; size_t n; };
    const R ins[] = {{a->q, nbt * a->dk * es}, {a->k, nbt * a->dk * es}, {a->v, nbt * a->dv * es},
                     {a->a, nbt * a->dk * es}, {a->b, nbt * a->dk * es}, {a->g, g_bytes},
                     {a->h0, a->h0 ? state_bytes : 0}, {a->grad_o, nbt * a->dv * es},
                     {a->grad_ht, a->grad_ht ? state_bytes : 0}, {a->workspace, a->workspace_bytes},
                     {a->cu_seqlens, a->cu_seqlens ? (size_t)(a->B + 1) * 4 : 0}};
    const R outs[] = {{a->grad_q, nbt * a->dk * es}, {a->grad_k, nbt * a->dk * es},
                      {a->grad_v, nbt * a->dv * es}, {a->grad_a, nbt * a->dk * es},
                      {a->grad_b, nbt * a->dk * es}, {a->grad_g, g_bytes},
                      {a->grad_h0, a->grad_h0 ? state_bytes : 0}};
    for (const R &o : outs) {
        for (const R &r : ins)
            if (overlaps(o.p, o.n, r.p, r.n)) return KDA_ERR_INVALID_ARG;
        for (const R &o2 : outs)
            if (&o2 != &o && overlaps(o.p, o.n, o2.p, o2.n)) return KDA_ERR_INVALID_ARG;
    }
    return KDA_OK;
}

size_t dplr_bwd_workspace_bytes(const dplr_bwd_args *a) {
    return kStatusBytes + kda::dplr_bwd_state_bytes(a->B, a->T, a->H, a->dk, a->dv, a->cu_seqlens != nullptr);
}

kda_status from_cuda(cudaError_t e) {
    if (e == cudaErrorNotSupported) return KDA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Streaming multiprocessors of the current device (0 if the query fails).
int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Chunk-record bytes of the two-kernel bf16 forward, 0 where the single kernel is the faster
// form: float32 inputs, and batches whose single-kernel CTAs (one per 64-value slice of each
// sequence and head) fill between half and all of the SMs in one wave -- there every SM builds
// its own chunks' operands next to its scan and no records travel through HBM, while fewer CTAs
// leave most SMs idle and more CTAs take several waves, where the chunk-parallel record kernel
// on every SM wins.
size_t fwd_record_bytes(const kda_fwd_args *a) {
    if (a->dtype != KDA_BF16) return 0;
    const long long ctas = (long long)a->B * a->H * (a->dv / 64);
    const int sms = sm_count();
    if (sms > 0 && 2 * ctas > sms && ctas <= sms) return 0;
    return kda::fwd_zrec_bytes(a->B, a->T, a->H, a->cu_seqlens != nullptr);
}

}  // namespace

extern "C" {

size_t kda_chunk_fwd_workspace(const kda_fwd_args *args) {
    if (validate(args) != KDA_OK) return 0;
    return kStatusBytes + fwd_record_bytes(args);
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
    p.cu_seqlens = args->cu_seqlens;
    {
        static std::atomic<unsigned> calls{0};
        unsigned t = ++calls;
        if ((int)t == 0) t = ++calls;                // never 0, the status block's initial value
        p.strong_token = (int)t;
    }
    if (const size_t zbytes = fwd_record_bytes(args)) {
        // the full workspace holds the chunk records of the two-kernel form; the status word
        // alone selects the single-kernel form
        if (args->workspace_bytes >= kStatusBytes + zbytes) {
            if (!aligned16(args->workspace)) return KDA_ERR_INVALID_ARG;
            p.zrec = static_cast<uint8_t *>(args->workspace) + kStatusBytes;
        }
    }

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

size_t dplr_chunk_fwd_workspace(const dplr_fwd_args *args) {
    if (validate_dplr(args) != KDA_OK) return 0;
    return kStatusBytes + kda::dplr_fwd_record_bytes(args->B, args->T, args->H, args->dk, args->dv,
                                                     args->cu_seqlens != nullptr);
}

kda_status dplr_chunk_fwd(const dplr_fwd_args *args, kda_stream_t stream) {
    kda_status st = validate_dplr(args);
    if (st != KDA_OK) return st;
    const size_t need = kStatusBytes + kda::dplr_fwd_record_bytes(args->B, args->T, args->H, args->dk, args->dv,
                                                                  args->cu_seqlens != nullptr);
    if (!args->workspace || args->workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(args->workspace)) return KDA_ERR_INVALID_ARG;   // vector and async copies into it
    kda::DplrParams p = dplr_params(args);
    p.ws_prep = reinterpret_cast<float *>(static_cast<unsigned char *>(args->workspace) + kStatusBytes);
    return from_cuda(kda::launch_dplr_fwd_simt(p, args->dtype == KDA_BF16, args->g_dtype == KDA_BF16,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

size_t dplr_chunk_bwd_workspace(const dplr_bwd_args *args) {
    if (validate_dplr_bwd(args) != KDA_OK) return 0;
    return dplr_bwd_workspace_bytes(args);
}

kda_status dplr_chunk_bwd(const dplr_bwd_args *args, kda_stream_t stream) {
    kda_status st = validate_dplr_bwd(args);
    if (st != KDA_OK) return st;
    if (!args->workspace || args->workspace_bytes < dplr_bwd_workspace_bytes(args)) return KDA_ERR_WORKSPACE;
    if (!aligned16(args->workspace)) return KDA_ERR_INVALID_ARG;   // vector and async copies into it
    kda::DplrParams p{};
    p.B = args->B; p.T = args->T; p.H = args->H; p.dk = args->dk; p.dv = args->dv;
    p.gate_kind = args->gate_kind;
    p.clip = (args->flags & DPLR_FLAG_CLIP_GATE) ? 1 : 0;
    p.q = args->q; p.k = args->k; p.v = args->v; p.a = args->a; p.b = args->b; p.g = args->g; p.h0 = args->h0;
    p.grad_o = args->grad_o; p.grad_ht = args->grad_ht;
    p.grad_q = args->grad_q; p.grad_k = args->grad_k; p.grad_v = args->grad_v;
    p.grad_a = args->grad_a; p.grad_b = args->grad_b; p.grad_g = args->grad_g; p.grad_h0 = args->grad_h0;
    p.cu_seqlens = args->cu_seqlens;
    unsigned char *ws = static_cast<unsigned char *>(args->workspace);
    p.status = reinterpret_cast<int *>(ws);
    kda::dplr_bwd_carve(p, reinterpret_cast<float *>(ws + kStatusBytes));
    return from_cuda(kda::launch_dplr_bwd_simt(p, args->dtype == KDA_BF16, args->g_dtype == KDA_BF16,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

kda_status dplr_factor_norms(const dplr_fwd_args *args, float *rho, float *norm, float *maxes,
                             kda_stream_t stream) {
    kda_status st = validate_dplr_common(args);
    if (st != KDA_OK) return st;
    const size_t nbt = (size_t)(args->cu_seqlens ? 1 : args->B) * args->T * args->H;
    const void *outs[] = {rho, norm, maxes};
    for (const void *p : outs)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    const size_t in_bytes = nbt * args->dk * dtype_size(args->dtype);
    const size_t g_bytes = args->gate_kind == KDA_GATE_CHANNEL ? nbt * args->dk * dtype_size(args->g_dtype)
                           : args->gate_kind == KDA_GATE_SCALAR ? nbt * dtype_size(args->g_dtype) : 0;
    struct R { const void *p; size_t n; } outr[] = {{rho, rho ? nbt * 4 : 0}, {norm, norm ? nbt * 4 : 0},
                                                     {maxes, maxes ? size_t{8} : size_t{0}}};
    for (const R &o : outr) {
        if (overlaps(o.p, o.n, args->a, in_bytes) || overlaps(o.p, o.n, args->b, in_bytes) ||
            overlaps(o.p, o.n, args->g, g_bytes))
            return KDA_ERR_INVALID_ARG;
    }
    if (overlaps(rho, outr[0].n, norm, outr[1].n) || overlaps(rho, outr[0].n, maxes, outr[2].n) ||
        overlaps(norm, outr[1].n, maxes, outr[2].n))
        return KDA_ERR_INVALID_ARG;
    return from_cuda(kda::launch_dplr_factor_norms(dplr_params(args), args->dtype == KDA_BF16,
                                                   args->g_dtype == KDA_BF16, rho, norm, maxes,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

size_t kda_chunk_bwd_workspace(const kda_bwd_args *args) {
    if (validate_bwd(args) != KDA_OK) return 0;
    return bwd_workspace_bytes(args);
}

kda_status kda_chunk_bwd(const kda_bwd_args *args, kda_stream_t stream) {
    kda_status st = validate_bwd(args);
    if (st != KDA_OK) return st;
    if (!args->workspace || args->workspace_bytes < bwd_workspace_bytes(args)) return KDA_ERR_WORKSPACE;
    if (!aligned16(args->workspace)) return KDA_ERR_INVALID_ARG;   // vector and async copies into it
    kda::BwdParams p{};
    p.B = args->B; p.T = args->T; p.H = args->H; p.dk = args->dk; p.dv = args->dv;
    p.gate_kind = args->gate_kind;
    p.scale_v = (args->flags & KDA_FLAG_BETA_SCALES_V) ? 1 : 0;
    p.has_beta = args->beta != nullptr;
    p.q = args->q; p.k = args->k; p.v = args->v; p.g = args->g; p.beta = args->beta; p.h0 = args->h0;
    p.grad_o = args->grad_o; p.grad_ht = args->grad_ht;
    p.grad_q = args->grad_q; p.grad_k = args->grad_k; p.grad_v = args->grad_v;
    p.grad_g = args->grad_g; p.grad_beta = args->grad_beta; p.grad_h0 = args->grad_h0;
    p.cu_seqlens = args->cu_seqlens;
    unsigned char *ws = static_cast<unsigned char *>(args->workspace);
    p.status = reinterpret_cast<int *>(ws);
    kda::bwd_carve(p, reinterpret_cast<float *>(ws + kStatusBytes));
    return from_cuda(kda::launch_bwd_simt(p, args->dtype == KDA_BF16, args->g_dtype == KDA_BF16,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_status_read(void *workspace, kda_stream_t stream) {
    if (!workspace || !aligned16(workspace)) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (word != kda::kDevOk) {
        // the status word and the words after it that locate the first wait that ran out (the
        // wait budget in word kStatusBoundWord is the caller's and stays)
        if (cudaMemsetAsync(workspace, 0, kda::kStatusBoundWord * sizeof(int), s) != cudaSuccess)
            return KDA_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    switch (word) {
    case kda::kDevOk: return KDA_OK;
    case kda::kDevTimeout: return KDA_ERR_TIMEOUT;
    case kda::kDevDecayRange: return KDA_ERR_RANGE;
    default: return KDA_ERR_CUDA;
    }
}

const char *kda_status_string(kda_status status) {
    switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported configuration";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_TIMEOUT: return "device-side wait timed out";
    case KDA_ERR_RANGE: return "log-decay outside the range of a kernel";
    }
    return "unknown status";
}

}  // extern "C"
