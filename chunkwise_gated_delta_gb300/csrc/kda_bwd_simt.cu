// Backward of the chunkwise gated delta rule (KDA and its special cases),
// chunk length C = 32, float32 accumulation: the chunk products are warp-level
// tf32 tensor-core MMAs for bf16 inputs and exact float32 products on the CUDA
// cores for fp32 inputs.
//
// Page "Kimi Delta Attention backward" derives, per chunk [t] and with dS the
// gradient of the state after the chunk:
//
//   dU   = K-> Diag(gamma^C) dS^T + (Q<- K->^T * M)^T dO
//   dW   = -dU S_prev
//   dQ<- = dO S_prev + (dO V_new^T * M) K->
//   dV   = Diag(beta) A~^T dU
//   dA~  = (dW K<-^T + dU V^T) Diag(beta),      dX~ = -A~^T dA~ A~^T
//   dK<- = Diag(beta) A~^T dW + (Diag(beta) dX~ * M_{-1}) K->
//   dK-> = V_new dS Diag(gamma^C) + (dO V_new^T * M)^T Q<- + (Diag(beta) dX~ * M_{-1})^T K<-
//   dbeta = diag(A~^T dW K<-^T) + diag(A~^T dU V^T) + diag(dX~ (K<- K->^T * M_{-1})^T)
//   dlogGamma = dQ<- * Q<- + dK<- * K<- - dK-> * K->,  last row + diag(S^T dS)
//   dg = in-chunk suffix sum of dlogGamma,  dq = dQ<- * Gamma,  dk = dK<- * Gamma + dK-> / Gamma
//   dS_prev = dS Diag(gamma^C) + dO^T Q<- - dU^T W
//
// (dW against S_[t-1]; dK-> with the output term the page's final
// combination carries.)  Four kernels:
//   prep  one CTA per (chunk, head, sequence): everything of a chunk that does
//         not depend on the state (A~, P, N, W, U, K~, Q<-, gamma^C) into a
//         chunk record in the workspace;
//   A     forward scan per (value slice, head, sequence) from the records: the
//         state before every chunk, the final state and V_new, into the
//         workspace;
//   B     reverse scan per (value slice, head, sequence) from the records: dS
//         after every chunk and dU into the workspace, and dh0;
//   C     one CTA per (chunk, head, sequence): every other gradient of the chunk,
//         from its record, V_new, dU and the stored S_prev, S_next and dS.
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "packed_seq.cuh"
#include "warp_gemm.cuh"

namespace kda {
namespace {

constexpr int kC = 32;       // chunk length
constexpr int kThreads = 256;
constexpr int kThreadsC = 512;   // the gradient kernel: 16 warps to hide the latency of its L2 reads

using seq::Seq;
__host__ __device__ __forceinline__ int chunk_slots(int B, int T, bool packed) {
    return seq::chunk_slots<kC>(B, T, packed);
}
__device__ __forceinline__ Seq seq_of(const BwdParams &p, int b) { return seq::seq_of<kC>(p, b); }
__device__ __forceinline__ bool chunk_of(const BwdParams &p, int &b, int &n, Seq &sq) {
    return seq::chunk_of<kC>(p, b, n, sq);
}
__device__ __forceinline__ size_t chunk_index(const BwdParams &p, const Seq &sq, int h, int n) {
    return seq::chunk_index<kC>(p, sq, h, n);
}
__device__ __forceinline__ size_t state_index(const BwdParams &p, const Seq &sq, int b, int h, int n) {
    return seq::state_index<kC>(p, sq, b, h, n);
}

template <typename T> __device__ __forceinline__ float ld(const T *p, size_t i);
template <> __device__ __forceinline__ float ld<float>(const float *p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
template <typename T> __device__ __forceinline__ void st(T *p, size_t i, float x);
template <> __device__ __forceinline__ void st<float>(float *p, size_t i, float x) { p[i] = x; }
template <> __device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

template <typename Tin>
__device__ void load_beta(const BwdParams &p, size_t row, int h, int nvalid, float *beta) {
    const Tin *bp = static_cast<const Tin *>(p.beta);
    const int tid = threadIdx.x;
    if (tid < kC) beta[tid] = (p.has_beta && tid < nvalid) ? ld(bp, (row + tid) * p.H + h) : 0.f;
}

// Gamma, Q<-, K<-, K-> of the chunk starting at row `row` of its batch, with row stride
// SK: all threads load the raw
// tiles, then one thread per key channel runs the in-chunk cumsum of g down
// its column in shared memory (rows past nvalid are zero, Gamma held at its
// last value); gam[d] = gamma^C.  Gm and Ql may be null (the raw g then waits
// in Kr); gsc holds C floats (scalar gates).  Contains one barrier; the
// caller synchronises before reading the tiles.
template <int DK, int SK, typename Tin, typename Tg, int NT = kThreads>
__device__ void load_rescaled_par(const BwdParams &p, size_t row, int h, int nvalid, float *Gm, float *Ql,
                                  float *Kl, float *Kr, float *gam, float *gsc) {
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tg *g = static_cast<const Tg *>(p.g);
    const int tid = threadIdx.x;
    float *graw = Gm ? Gm : Kr;
    const size_t r0 = (row * p.H + h) * DK, rs = (size_t)p.H * DK;
    wg::load_tile<kC, DK, SK, NT>(k + r0, rs, nvalid, Kl);
    if (Ql) wg::load_tile<kC, DK, SK, NT>(q + r0, rs, nvalid, Ql);
    if (p.gate_kind == KDA_GATE_CHANNEL) wg::load_tile<kC, DK, SK, NT>(g + r0, rs, nvalid, graw);
    if (p.gate_kind == KDA_GATE_SCALAR && tid < kC)
        gsc[tid] = tid < nvalid ? ld(g, (row + tid) * p.H + h) : 0.f;
    __syncthreads();
    if (tid < DK) {
        const int d = tid;
        float G = 0.f, gm = 1.f;
        for (int c = 0; c < kC; ++c) {
            const float gv = p.gate_kind == KDA_GATE_CHANNEL ? graw[c * SK + d]
                             : p.gate_kind == KDA_GATE_SCALAR ? gsc[c] : 0.f;
            if (c < nvalid) {
                G += gv;
                gm = expf(G);
            }
            const float kv = Kl[c * SK + d];
            Kl[c * SK + d] = kv * gm;
            Kr[c * SK + d] = kv / gm;
            if (Ql) Ql[c * SK + d] *= gm;
            if (Gm) Gm[c * SK + d] = gm;
        }
        gam[d] = gm;
    }
}

// A~ = (I + Diag(beta) N)^{-1} for a strictly lower N in Nm (row stride SC):
// the unit lower triangular inverse in two levels (page "DeltaNet", section
// 4.2, block form): the two 16x16 diagonal blocks by forward substitution
// side by side (one column per thread of the first warp), then the
// off-diagonal block A21 = -A22 L21 A11 by two parallel products (Tm is a
// [C][SC] scratch).  Starts after, and ends with, a barrier.
template <int SC>
__device__ void block_inverse(const float *beta, const float *Nm, float *Am, float *Tm) {
    constexpr int HB = kC / 2;
    const int tid = threadIdx.x;
    if (tid < kC) {
        const int blk = tid / HB, c = blk * HB + tid % HB;     // column c of diagonal block blk
        for (int i = blk * HB; i < blk * HB + HB; ++i) {
            float y = 0.f;
            if (i == c) y = 1.f;
            else if (i > c)
                for (int j = c; j < i; ++j) y -= beta[i] * Nm[i * SC + j] * Am[j * SC + c];
            Am[i * SC + c] = y;
        }
        for (int i = 0; i < HB; ++i) Am[(blk == 0 ? i : HB + i) * SC + (blk == 0 ? HB : 0) + tid % HB] = 0.f;
    }
    __syncthreads();
    // Tm = L21 A11 (rows HB.., cols ..HB), L21 = Diag(beta) N21
    for (int idx = tid; idx < HB * HB; idx += blockDim.x) {
        const int i = HB + idx / HB, j = idx % HB;
        float acc = 0.f;
        for (int l = j; l < HB; ++l) acc += beta[i] * Nm[i * SC + l] * Am[l * SC + j];
        Tm[i * SC + j] = acc;
    }
    __syncthreads();
    // A21 = -A22 Tm
    for (int idx = tid; idx < HB * HB; idx += blockDim.x) {
        const int i = HB + idx / HB, j = idx % HB;
        float acc = 0.f;
        for (int l = HB; l <= i; ++l) acc -= Am[i * SC + l] * Tm[l * SC + j];
        Am[i * SC + j] = acc;
    }
    __syncthreads();
}

// Row strides of the shared tiles: = 4 (mod 32), so that the 8 x 4 fragment
// reads of the warp-tiled products mostly avoid bank conflicts.
__host__ __device__ constexpr int pad4(int n) { return n + 4; }
constexpr int kSC4 = pad4(kC);

// ------------------------------------------------------------------ chunk records
// Everything of a chunk that does not depend on the state, written once by the
// prep kernel (float32): A~, P = Q<- K->^T * M, N = K<- K->^T * M_{-1},
// W = A~ Diag(beta) K<-, U = A~ Diag(beta) V (or A~ V), K~ = K-> Diag(gamma^C),
// Q<- and gamma^C.
__host__ __device__ constexpr size_t rec_floats(int dk, int dv) {
    return (size_t)3 * kC * kC + (size_t)3 * kC * dk + (size_t)kC * dv + dk;
}
template <int DK, int DV>
struct Rec {
    static constexpr int A = 0, P = kC * kC, N = 2 * kC * kC, W = 3 * kC * kC, U = W + kC * DK, KT = U + kC * DV,
                         QL = KT + kC * DK, GC = QL + kC * DK;
    static_assert(rec_floats(DK, DV) == (size_t)GC + DK && rec_floats(DK, DV) % 4 == 0, "record layout");
};

// ------------------------------------------------------------------ prep kernel
// One CTA per (chunk, head, sequence).
template <int DK, int DV, typename Tin, typename Tg, bool TF32>
__global__ void __launch_bounds__(kThreads) kda_bwd_prep_kernel(const BwdParams p) {
    constexpr int SK = pad4(DK), SV = pad4(DV), SC = kSC4;
    using R = Rec<DK, DV>;
    extern __shared__ float smem[];
    float *Gm = smem;                  // [C][SK]  raw gate, then Gamma
    float *Ql = Gm + kC * SK;          // [C][SK]
    float *Kl = Ql + kC * SK;          // [C][SK]
    float *Kr = Kl + kC * SK;          // [C][SK]
    float *Vm = Kr + kC * SK;          // [C][SV]
    float *Nm = Vm + kC * SV;          // [C][SC]
    float *Am = Nm + kC * SC;          // [C][SC]
    float *Tm = Am + kC * SC;          // [C][SC]
    float *beta = Tm + kC * SC;        // [C]
    float *gsc = beta + kC;            // [C]
    float *gam = gsc + kC;             // [DK]

    const int tid = threadIdx.x, h = blockIdx.y;
    int b, n;
    Seq sq;
    if (!chunk_of(p, b, n, sq)) return;
    const int H = p.H;
    const int t0 = n * kC, nvalid = min(kC, sq.len - t0);
    const size_t row = (size_t)sq.row0 + t0;
    const Tin *v = static_cast<const Tin *>(p.v);
    float *rec = p.ws_prep + chunk_index(p, sq, h, n) * rec_floats(DK, DV);
    const bool sv = p.scale_v != 0;

    load_beta<Tin>(p, row, h, nvalid, beta);
    wg::load_tile<kC, DV, SV, kThreads>(v + (row * H + h) * DV, (size_t)H * DV, nvalid, Vm);
    load_rescaled_par<DK, SK, Tin, Tg>(p, row, h, nvalid, Gm, Ql, Kl, Kr, gam, gsc);
    __syncthreads();
    {
        auto bKr = [&](int d, int j) { return Kr[j * SK + d]; };
        wg::gemm_pair<kC, TF32>(
            DK, [&](int i, int d) { return Ql[i * SK + d]; }, bKr, DK, [&](int i, int d) { return Kl[i * SK + d]; },
            bKr, [&](int i, int j, float pv, float nv) {
                rec[R::P + i * kC + j] = j <= i ? pv : 0.f;
                const float nn = j < i ? nv : 0.f;
                Nm[i * SC + j] = nn;
                rec[R::N + i * kC + j] = nn;
            });
    }
    for (int idx = tid; idx < kC * DK; idx += kThreads) {
        const int i = idx / DK, d = idx % DK;
        rec[R::KT + idx] = Kr[i * SK + d] * gam[d];
        rec[R::QL + idx] = Ql[i * SK + d];
    }
    for (int d = tid; d < DK; d += kThreads) rec[R::GC + d] = gam[d];
    __syncthreads();
    block_inverse<SC>(beta, Nm, Am, Tm);
    for (int idx = tid; idx < kC * kC; idx += kThreads) rec[R::A + idx] = Am[(idx / kC) * SC + idx % kC];
    wg::gemm<DK, TF32>(
        kC, [&](int i, int j) { return Am[i * SC + j] * beta[j]; }, [&](int j, int d) { return Kl[j * SK + d]; },
        [&](int i, int d, float x) { rec[R::W + i * DK + d] = x; });
    wg::gemm<DV, TF32>(
        kC, [&](int i, int j) { return Am[i * SC + j] * (sv ? beta[j] : 1.f); },
        [&](int j, int e) { return Vm[j * SV + e]; }, [&](int i, int e, float x) { rec[R::U + i * DV + e] = x; });
}

template <int DK, int DV>
constexpr size_t prep_smem_bytes() {
    return sizeof(float) * ((size_t)4 * kC * pad4(DK) + kC * pad4(DV) + 3 * kC * kSC4 + 2 * kC + DK);
}

// ------------------------------------------------------------------ kernel A
// The forward state scan from the chunk records: V_new = U - W S^T,
// S <- S Diag(gamma^C) + V_new^T K~.  One CTA per (64-wide value slice, head, sequence).
// The records of chunk n + 1 travel (cp.async, double buffer) while chunk n computes.
constexpr int kDVD = 64;     // value rows per CTA in the two scans

// A scan's [kDVD][DK] state block between shared memory (row stride SK) and global rows of DK
// floats, 16 bytes per access (rows 16-byte aligned on both sides); a null source reads zeros.
template <int DK, int SK>
__device__ __forceinline__ void block_to_shared(const float *src, float *dst) {
    constexpr int V = DK / 4;
    for (int idx = threadIdx.x; idx < kDVD * V; idx += kThreads) {
        const int e = idx / V, d = (idx % V) * 4;
        *reinterpret_cast<float4 *>(dst + e * SK + d) =
            src ? *reinterpret_cast<const float4 *>(src + (size_t)e * DK + d) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}
template <int DK, int SK>
__device__ __forceinline__ void block_to_global(const float *src, float *dst) {
    constexpr int V = DK / 4;
    for (int idx = threadIdx.x; idx < kDVD * V; idx += kThreads) {
        const int e = idx / V, d = (idx % V) * 4;
        *reinterpret_cast<float4 *>(dst + (size_t)e * DK + d) = *reinterpret_cast<const float4 *>(src + e * SK + d);
    }
}
template <int DK>
__host__ __device__ constexpr int states_buf_floats() {
    return 2 * kC * pad4(DK) + kC * pad4(kDVD) + DK;       // W, K~, U (then V_new), gamma^C
}
template <int DK, int DV, bool TF32>
__global__ void __launch_bounds__(kThreads) kda_bwd_states_kernel(const BwdParams p) {
    constexpr int SK = pad4(DK), SV = pad4(kDVD), BUF = states_buf_floats<DK>();
    using R = Rec<DK, DV>;
    extern __shared__ float smem[];
    float *Sm = smem;                  // [DVS][SK]
    float *bufs = Sm + kDVD * SK;      // 2 x BUF

    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * kDVD, h = blockIdx.y, b = blockIdx.z;
    const int H = p.H, dv = p.dv;
    const Seq sq = seq_of(p, b);
    const int N = sq.nch;
    const size_t head = (size_t)b * H + h;
    float *Sws = p.ws_S + state_index(p, sq, b, h, 0) * dv * DK;
    const float *recs = p.ws_prep + chunk_index(p, sq, h, 0) * rec_floats(DK, DV);
    float *vnew = p.ws_vnew + chunk_index(p, sq, h, 0) * kC * dv;
    auto issue = [&](int n) {
        const float *rec = recs + (size_t)n * rec_floats(DK, DV);
        float *bf = bufs + (n & 1) * BUF;
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::W, DK, bf);
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::KT, DK, bf + kC * SK);
        wg::load_tile_async<kC, kDVD, SV, kThreads>(rec + R::U + e0, DV, bf + 2 * kC * SK);
        wg::load_tile_async<1, DK, DK, kThreads>(rec + R::GC, DK, bf + 2 * kC * SK + kC * SV);
    };

    block_to_shared<DK, SK>(p.h0 ? p.h0 + (head * dv + e0) * DK : nullptr, Sm);
    issue(0);
    wg::cp_async_commit();
    for (int n = 0; n < N; ++n) {
        float *Wm = bufs + (n & 1) * BUF, *KT = Wm + kC * SK, *Um = KT + kC * SK, *gam = Um + kC * SV;
        __syncthreads();               // S is final for chunk n; chunk n - 1's buffer is free
        block_to_global<DK, SK>(Sm, Sws + ((size_t)n * dv + e0) * DK);
        if (n + 1 < N) issue(n + 1);
        wg::cp_async_commit();         // (an empty group on the last chunk keeps the count)
        wg::cp_async_wait<1>();        // chunk n's tiles have landed (this thread's copies)
        __syncthreads();               // ... and everyone's
        float *vn = vnew + (size_t)n * kC * dv + e0;     // V_new rows of this chunk
        wg::gemm<kDVD, TF32>(
            DK, [&](int i, int d) { return Wm[i * SK + d]; }, [&](int d, int e) { return Sm[e * SK + d]; },
            [&](int i, int e, float x) {
                const float y = Um[i * SV + e] - x;
                Um[i * SV + e] = y;
                vn[(size_t)i * dv + e] = y;
            });
        __syncthreads();
        // S rows e of the slice, 32 at a time
#pragma unroll
        for (int eo = 0; eo < kDVD; eo += 32)
            wg::gemm<DK, TF32>(
                kC, [&](int e, int c) { return Um[c * SV + eo + e]; }, [&](int c, int d) { return KT[c * SK + d]; },
                [&](int e, int d, float x) { Sm[(eo + e) * SK + d] = Sm[(eo + e) * SK + d] * gam[d] + x; });
    }
    __syncthreads();
    block_to_global<DK, SK>(Sm, Sws + ((size_t)N * dv + e0) * DK);
}

// ------------------------------------------------------------------ kernel B
// The reverse scan from the chunk records: dU = K~ dS^T + P^T dO,
// dS <- dS Diag(gamma^C) + dO^T Q<- - dU^T W.  One CTA per (64-wide value slice, head,
// sequence): the records of a head are read by dv / 64 CTAs, and the records and dO rows of
// chunk n - 1 travel (cp.async, double buffer) while chunk n computes.
template <int DK, typename Tin>
__host__ __device__ constexpr int dstate_buf_floats() {
    // W, Q<-, K~ [C][SK]; P [C][SC]; gamma^C [DK]; raw dO rows [C][DVD] of Tin
    return 3 * kC * pad4(DK) + kC * kSC4 + DK + (kC * kDVD * (int)sizeof(Tin) + 3) / 4;
}
template <int DK, int DV, typename Tin, bool TF32>
__global__ void __launch_bounds__(kThreads) kda_bwd_dstate_kernel(const BwdParams p) {
    constexpr int SK = pad4(DK), SV = pad4(kDVD), SC = kSC4, BUF = dstate_buf_floats<DK, Tin>();
    using R = Rec<DK, DV>;
    extern __shared__ float smem[];
    float *dS = smem;                  // [DVD][SK]
    float *dO = dS + kDVD * SK;        // [C][SV]
    float *dU = dO + kC * SV;          // [C][SV]
    float *bufs = dU + kC * SV;        // 2 x BUF

    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * kDVD, h = blockIdx.y, b = blockIdx.z;
    const int H = p.H, dv = p.dv;
    const Seq sq = seq_of(p, b);
    const int N = sq.nch;
    const Tin *dop = static_cast<const Tin *>(p.grad_o);
    const size_t head = (size_t)b * H + h;
    float *dSws = p.ws_dS + chunk_index(p, sq, h, 0) * dv * DK;
    const float *recs = p.ws_prep + chunk_index(p, sq, h, 0) * rec_floats(DK, DV);
    float *dus = p.ws_du + chunk_index(p, sq, h, 0) * kC * dv;
    // buffer (n & 1) holds chunk n's tiles
    auto issue = [&](int n) {
        const float *rec = recs + (size_t)n * rec_floats(DK, DV);
        float *bf = bufs + (n & 1) * BUF;
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::W, DK, bf);
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::QL, DK, bf + kC * SK);
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::KT, DK, bf + 2 * kC * SK);
        wg::load_tile_async<kC, kC, SC, kThreads>(rec + R::P, kC, bf + 3 * kC * SK);
        wg::load_tile_async<1, DK, DK, kThreads>(rec + R::GC, DK, bf + 3 * kC * SK + kC * SC);
        const int t0 = n * kC;
        wg::load_raw_async<kC, kDVD, Tin, kThreads>(dop + (((size_t)sq.row0 + t0) * H + h) * dv + e0,
                                                    (size_t)H * dv, min(kC, sq.len - t0),
                                                    reinterpret_cast<Tin *>(bf + 3 * kC * SK + kC * SC + DK));
    };

    block_to_shared<DK, SK>(p.grad_ht ? p.grad_ht + (head * dv + e0) * DK : nullptr, dS);
    if (N > 0) issue(N - 1);
    wg::cp_async_commit();
    for (int n = N - 1; n >= 0; --n) {
        float *Wm = bufs + (n & 1) * BUF, *QL = Wm + kC * SK, *KT = QL + kC * SK, *Pm = KT + kC * SK;
        float *gam = Pm + kC * SC;
        const Tin *draw = reinterpret_cast<const Tin *>(gam + DK);
        __syncthreads();               // dS is final for chunk n; chunk n + 1's buffer is free
        block_to_global<DK, SK>(dS, dSws + ((size_t)n * dv + e0) * DK);
        if (n > 0) issue(n - 1);
        wg::cp_async_commit();         // (an empty group on the last step keeps the count)
        wg::cp_async_wait<1>();        // chunk n's tiles have landed (this thread's copies)
        __syncthreads();               // ... and everyone's
        wg::to_f32<kC, kDVD, SV, Tin, kThreads>(draw, dO);
        __syncthreads();
        float *du = dus + (size_t)n * kC * dv + e0;       // dU rows of this chunk
        wg::gemm2<kDVD, TF32>(
            DK, [&](int i, int d) { return KT[i * SK + d]; }, [&](int d, int e) { return dS[e * SK + d]; }, kC,
            [&](int i, int j) { return Pm[j * SC + i]; }, [&](int j, int e) { return dO[j * SV + e]; },
            [&](int i, int e, float x) {
                dU[i * SV + e] = x;
                du[(size_t)i * dv + e] = x;
            });
        __syncthreads();
        // dS rows e of the slice, 32 at a time
#pragma unroll
        for (int eo = 0; eo < kDVD; eo += 32)
            wg::gemm2<DK, TF32>(
                kC, [&](int e, int c) { return dO[c * SV + eo + e]; }, [&](int c, int d) { return QL[c * SK + d]; },
                kC, [&](int e, int c) { return -dU[c * SV + eo + e]; }, [&](int c, int d) { return Wm[c * SK + d]; },
                [&](int e, int d, float x) { dS[(eo + e) * SK + d] = dS[(eo + e) * SK + d] * gam[d] + x; });
    }
    __syncthreads();
    if (p.grad_h0) block_to_global<DK, SK>(dS, p.grad_h0 + (head * dv + e0) * DK);
}

// ------------------------------------------------------------------ kernel C

template <int DK, int DV>
constexpr size_t grad_smem_floats() {
    return (size_t)8 * kC * pad4(DK) + (size_t)4 * kC * pad4(DV) + (size_t)5 * kC * kSC4 + 2 * kC + 2 * DK;
}

// Products run as warp-tiled 32 x N blocks (warp_gemm.cuh): tf32 tensor-core
// MMAs for bf16 inputs (TF32), exact float32 for float32 inputs.
template <int DK, int DV, typename Tin, typename Tg, bool TF32>
__global__ void __launch_bounds__(kThreadsC) kda_bwd_grad_kernel(const BwdParams p) {
    constexpr int SK = pad4(DK), SV = pad4(DV), SC = kSC4;
    extern __shared__ float smem[];
    float *Gm = smem;                  // [C][SK]  Gamma
    float *Ql = Gm + kC * SK;          // [C][SK]
    float *Kl = Ql + kC * SK;          // [C][SK]
    float *Kr = Kl + kC * SK;          // [C][SK]
    float *Wm = Kr + kC * SK;          // [C][SK]  W, then dW
    float *dQl = Wm + kC * SK;         // [C][SK]
    float *dKl = dQl + kC * SK;        // [C][SK]  A~^T dW, then dK<-
    float *dKr = dKl + kC * SK;        // [C][SK]
    float *Vm = dKr + kC * SK;         // [C][SV]
    float *dO = Vm + kC * SV;          // [C][SV]
    float *Vn = dO + kC * SV;          // [C][SV]  U, V_new, then A~^T dU
    float *dU = Vn + kC * SV;          // [C][SV]
    float *Nm = dU + kC * SV;          // [C][SC]  K<- K->^T * M_{-1}
    float *Am = Nm + kC * SC;          // [C][SC]  A~
    float *Pm = Am + kC * SC;          // [C][SC]  P, then dO V_new^T * M
    float *dA = Pm + kC * SC;          // [C][SC]  dA~, then dX~
    float *Tm = dA + kC * SC;          // [C][SC]  scratch
    float *beta = Tm + kC * SC;        // [C]
    float *dbeta = beta + kC;          // [C]
    float *gam = dbeta + kC;           // [DK]
    float *lastrow = gam + DK;         // [DK] diag(S_next^T dS)

    const int tid = threadIdx.x, h = blockIdx.y;
    int b, n;
    Seq sq;
    if (!chunk_of(p, b, n, sq)) return;
    const int H = p.H;
    const int t0 = n * kC, nvalid = min(kC, sq.len - t0);
    const size_t row = (size_t)sq.row0 + t0;
    const Tin *v = static_cast<const Tin *>(p.v);
    const Tin *dop = static_cast<const Tin *>(p.grad_o);
    const size_t ci = chunk_index(p, sq, h, n);
    const float *Sp = p.ws_S + state_index(p, sq, b, h, n) * DV * DK;     // state before the chunk
    const float *Sn = Sp + (size_t)DV * DK;                                 // state after the chunk
    const float *dS = p.ws_dS + ci * DV * DK;                               // gradient of the state after
    const bool sv = p.scale_v != 0;

    // The stored states stream through a ring of four tile buffers that are free until the
    // state products below end (W, dQ<-, dK<-, dK->): slabs of 32 rows, in the order they are
    // consumed -- S_prev slabs, then (dS, S_next) slab pairs -- by cp.async, the first four
    // issued now so that they travel during the loads and the first product.
    constexpr int NS = DV / kC, NL = 3 * NS;
    float *ring[4] = {Wm, dKl, dQl, dKr};
    auto slab_src = [&](int k) -> const float * {
        if (k < NS) return Sp + (size_t)k * kC * DK;
        return (((k - NS) & 1) ? Sn : dS) + (size_t)((k - NS) >> 1) * kC * DK;
    };
    int issued = 0;
    auto issue_upto = [&](int end) {
        for (; issued < end && issued < NL; ++issued) {
            wg::load_tile_async<kC, DK, SK, kThreadsC>(slab_src(issued), DK, ring[issued & 3]);
            wg::cp_async_commit();
        }
    };
    // A~, P, N of the chunk record and the chunk's V_new and dU (float32, written by the prep kernel
    // and the scans) by cp.async too: one group, committed before the slabs' and waited for after
    // the loads below
    {
        using R = Rec<DK, DV>;
        const float *rec = p.ws_prep + ci * rec_floats(DK, DV);
        wg::load_tile_async<kC, kC, SC, kThreadsC>(rec + R::A, kC, Am);
        wg::load_tile_async<kC, kC, SC, kThreadsC>(rec + R::P, kC, Pm);
        wg::load_tile_async<kC, kC, SC, kThreadsC>(rec + R::N, kC, Nm);
        wg::load_tile_async<kC, DV, SV, kThreadsC>(p.ws_vnew + ci * kC * DV, DV, Vn);
        wg::load_tile_async<kC, DV, SV, kThreadsC>(p.ws_du + ci * kC * DV, DV, dU);
        wg::cp_async_commit();
    }
    static_assert(NL >= 4, "four slab groups follow the tiles' group");
    issue_upto(4);

    // ---- loads: Gamma and the rescaled tiles, v, dO, beta
    load_rescaled_par<DK, SK, Tin, Tg, kThreadsC>(p, row, h, nvalid, Gm, Ql, Kl, Kr, gam, dbeta);
    load_beta<Tin>(p, row, h, nvalid, beta);
    {
        const size_t r0 = (row * H + h) * DV, rs = (size_t)H * DV;
        wg::load_tile<kC, DV, SV, kThreadsC>(v + r0, rs, nvalid, Vm);
        wg::load_tile<kC, DV, SV, kThreadsC>(dop + r0, rs, nvalid, dO);
    }
    wg::cp_async_wait<4>();            // the tiles' group (at most the four slab groups after it in flight)
    __syncthreads();
    // ---- dO V_new^T * M (into Pm)
    wg::gemm<kC, TF32, 16>(
        DV, [&](int i, int e) { return dO[i * SV + e]; }, [&](int e, int j) { return Vn[j * SV + e]; },
        [&](int i, int j, float x) { Pm[i * SC + j] = j <= i ? x : 0.f; });
    __syncthreads();
    // ---- dW = -dU S_prev ; dQ<- = dO S_prev + (dO V_new^T * M) K-> ;
    //      dK-> = V_new dS Diag(gamma^C) + (dO V_new^T * M)^T Q<- ; and diag(S_next^T dS)
    //      for the gamma^C row, from the slab ring.  A unit consumes slabs a..bl; before it,
    //      the buffers of every earlier slab are free, so slabs up to a + 3 may be in flight.
    {
        constexpr int NT = wg::ntiles<DK, 16>();
        int r0, c0;
        wg::origin<DK, 16>(r0, c0);
        float aW[NT][4] = {}, aQ[NT][4] = {}, aK[NT][4] = {}, aK2[NT][4] = {};
        float last = 0.f;                  // diag(S_next^T dS), column tid
        for (int u = 0; u < 2 * NS; ++u) {
            const int a = u < NS ? u : NS + 2 * (u - NS), bl = u < NS ? a : a + 1;
            issue_upto(a + 4);
            switch (issued - 1 - bl) {     // this thread's copies of slabs <= bl have landed
                case 0: wg::cp_async_wait<0>(); break;
                case 1: wg::cp_async_wait<1>(); break;
                case 2: wg::cp_async_wait<2>(); break;
                default: wg::cp_async_wait<3>(); break;
            }
            __syncthreads();
            if (u < NS) {
                const int s0 = u * kC;
                const float *slab = ring[a & 3];
                auto bS = [&](int e, int d) { return slab[e * SK + d]; };
                wg::tile<NT, TF32>(aW, r0, c0, kC, [&](int i, int e) { return dU[i * SV + s0 + e]; }, bS);
                wg::tile<NT, TF32>(aQ, r0, c0, kC, [&](int i, int e) { return dO[i * SV + s0 + e]; }, bS);
            } else {
                const int s0 = (u - NS) * kC;
                const float *dsl = ring[a & 3], *snl = ring[(a + 1) & 3];
                wg::tile<NT, TF32>(aK, r0, c0, kC, [&](int i, int e) { return Vn[i * SV + s0 + e]; },
                                   [&](int e, int d) { return dsl[e * SK + d]; });
                if (tid < DK)
#pragma unroll 4
                    for (int e = 0; e < kC; ++e) last += snl[e * SK + tid] * dsl[e * SK + tid];
            }
            __syncthreads();
        }
        if (tid < DK) lastrow[tid] = last;
        wg::tile<NT, TF32>(aQ, r0, c0, kC, [&](int i, int j) { return Pm[i * SC + j]; },
                           [&](int j, int d) { return Kr[j * SK + d]; });
        wg::tile<NT, TF32>(aK2, r0, c0, kC, [&](int i, int j) { return Pm[j * SC + i]; },
                           [&](int j, int d) { return Ql[j * SK + d]; });
        wg::store<NT>(aW, r0, c0, [&](int i, int d, float x) { Wm[i * SK + d] = -x; });
        wg::store<NT>(aQ, r0, c0, [&](int i, int d, float x) { dQl[i * SK + d] = x; });
        wg::store_pair<NT>(aK, aK2, r0, c0, [&](int i, int d, float x1, float x2) { dKr[i * SK + d] = x1 * gam[d] + x2; });
    }
    __syncthreads();
    // ---- A~^T dW (into dKl), A~^T dU (into Vn), dA~ = dW K<-^T Diag(beta) + dU V^T Diag(beta) (or dU V^T)
    auto aAt = [&](int i, int j) { return Am[j * SC + i]; };
    wg::gemm<DK, TF32, 16>(
        kC, aAt, [&](int j, int d) { return Wm[j * SK + d]; }, [&](int i, int d, float x) { dKl[i * SK + d] = x; });
    wg::gemm<DV, TF32, 16>(
        kC, aAt, [&](int j, int e) { return dU[j * SV + e]; }, [&](int i, int e, float x) { Vn[i * SV + e] = x; });
    wg::gemm_pair<kC, TF32, 16>(
        DK, [&](int i, int d) { return Wm[i * SK + d]; }, [&](int d, int j) { return Kl[j * SK + d]; }, DV,
        [&](int i, int e) { return dU[i * SV + e]; }, [&](int e, int j) { return Vm[j * SV + e]; },
        [&](int i, int j, float xw, float xu) { dA[i * SC + j] = xw * beta[j] + xu * (sv ? beta[j] : 1.f); });
    __syncthreads();
    // ---- dbeta, first two terms: diag(A~^T dW K<-^T) + diag(A~^T dU V^T) ; Tm = dA~ A~^T
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int i = warp; i < kC; i += kThreadsC / 32) {
            float acc = 0.f;
            for (int d = lane; d < DK; d += 32) acc += dKl[i * SK + d] * Kl[i * SK + d];
            if (sv)
                for (int e = lane; e < DV; e += 32) acc += Vn[i * SV + e] * Vm[i * SV + e];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) dbeta[i] = acc;
        }
    }
    wg::gemm<kC, TF32, 16>(
        kC, [&](int i, int l) { return dA[i * SC + l]; }, [&](int l, int j) { return Am[j * SC + l]; },
        [&](int i, int j, float x) { Tm[i * SC + j] = x; });
    __syncthreads();
    // ---- dX~ = -A~^T (dA~ A~^T)
    wg::gemm<kC, TF32, 16>(
        kC, aAt, [&](int l, int j) { return Tm[l * SC + j]; }, [&](int i, int j, float x) { dA[i * SC + j] = -x; });
    __syncthreads();
    // ---- dbeta third term diag(dX~ N^T); E = (Diag(beta) dX~) * M_{-1} into Tm
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int i = warp; i < kC; i += kThreadsC / 32) {
            float acc = dA[i * SC + lane] * Nm[i * SC + lane];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) dbeta[i] += acc;
        }
    }
    for (int idx = tid; idx < kC * kC; idx += kThreadsC) {
        const int i = idx / kC, j = idx % kC;
        Tm[i * SC + j] = j < i ? beta[i] * dA[i * SC + j] : 0.f;
    }
    __syncthreads();
    // ---- dK<- = Diag(beta) A~^T dW + E K-> ; dK-> += E^T K<-
    wg::gemm<DK, TF32, 16>(
        kC, [&](int i, int j) { return Tm[i * SC + j]; }, [&](int j, int d) { return Kr[j * SK + d]; },
        [&](int i, int d, float x) { dKl[i * SK + d] = beta[i] * dKl[i * SK + d] + x; });
    wg::gemm<DK, TF32, 16>(
        kC, [&](int i, int j) { return Tm[j * SC + i]; }, [&](int j, int d) { return Kl[j * SK + d]; },
        [&](int i, int d, float x) { dKr[i * SK + d] += x; });
    __syncthreads();
    // ---- outputs: dq, dk, dv, dbeta, and dg from the suffix sums of dlogGamma
    Tin *gq = static_cast<Tin *>(p.grad_q);
    Tin *gk = static_cast<Tin *>(p.grad_k);
    Tin *gv = static_cast<Tin *>(p.grad_v);
    for (int idx = tid; idx < kC * DK; idx += kThreadsC) {
        const int i = idx / DK, d = idx % DK;
        if (i < nvalid) {
            const size_t off = ((row + i) * H + h) * DK + d;
            const float gm = Gm[i * SK + d];
            st(gq, off, dQl[i * SK + d] * gm);
            st(gk, off, dKl[i * SK + d] * gm + dKr[i * SK + d] / gm);
        }
    }
    for (int idx = tid; idx < kC * DV; idx += kThreadsC) {
        const int i = idx / DV, e = idx % DV;
        if (i < nvalid)
            st(gv, ((row + i) * H + h) * DV + e, (sv ? beta[i] : 1.f) * Vn[i * SV + e]);
    }
    if (p.has_beta && tid < nvalid)
        st(static_cast<Tin *>(p.grad_beta), (row + tid) * H + h, dbeta[tid]);
    if (p.gate_kind != KDA_GATE_NONE) {
        // diag(S_next^T dS) for the gamma^C row, then suffix sums down each channel
        Tg *gg = static_cast<Tg *>(p.grad_g);
        const float *acc_last = lastrow;   // diag(S_next^T dS), from the state pass above
        if (p.gate_kind == KDA_GATE_CHANNEL) {
            for (int d = tid; d < DK; d += kThreadsC) {
                float run = acc_last[d];
                for (int i = kC - 1; i >= 0; --i) {
                    run += dQl[i * SK + d] * Ql[i * SK + d] + dKl[i * SK + d] * Kl[i * SK + d] -
                           dKr[i * SK + d] * Kr[i * SK + d];
                    if (i < nvalid) st(gg, ((row + i) * H + h) * DK + d, run);
                }
            }
        } else {
            // scalar gate: the channel sum of the per-channel gradient
            const int warp = tid >> 5, lane = tid & 31;
            float *rowsum = dbeta;     // reuse: C floats (dbeta was already written out)
            __syncthreads();
            for (int i = warp; i < kC; i += kThreadsC / 32) {
                float acc = 0.f;
                for (int d = lane; d < DK; d += 32)
                    acc += dQl[i * SK + d] * Ql[i * SK + d] + dKl[i * SK + d] * Kl[i * SK + d] -
                           dKr[i * SK + d] * Kr[i * SK + d];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                if (lane == 0) rowsum[i] = acc;
            }
            __syncthreads();
            if (tid == 0) {
                float run = 0.f;
                for (int d = 0; d < DK; ++d) run += acc_last[d];
                for (int i = kC - 1; i >= 0; --i) {
                    run += rowsum[i];
                    if (i < nvalid) st(gg, (row + i) * H + h, run);
                }
            }
        }
    }
}

template <int DK>
constexpr size_t states_smem_bytes() {
    return sizeof(float) * ((size_t)kDVD * pad4(DK) + 2 * states_buf_floats<DK>());
}
template <int DK, typename Tin>
constexpr size_t dstate_smem_bytes() {
    return sizeof(float) * ((size_t)kDVD * pad4(DK) + 2 * kC * pad4(kDVD) + 2 * dstate_buf_floats<DK, Tin>());
}

template <typename F>
cudaError_t set_smem(F *fn, size_t bytes) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int DK, int DV, typename Tin, typename Tg>
cudaError_t launch_all(const BwdParams &p, cudaStream_t s) {
    constexpr bool kTf32 = sizeof(Tin) == 2;        // bf16 inputs: tf32 tensor-core products
    const bool packed = p.cu_seqlens != nullptr;
    cudaError_t e;
    const size_t sp = prep_smem_bytes<DK, DV>(), sa = states_smem_bytes<DK>(), sb = dstate_smem_bytes<DK, Tin>();
    static_assert(dstate_smem_bytes<128, float>() <= 227 * 1024, "kernel B shared memory");
    const size_t sc = sizeof(float) * grad_smem_floats<DK, DV>();
    static_assert(sizeof(float) * grad_smem_floats<128, 128>() <= 227 * 1024, "kernel C shared memory");
    if ((e = set_smem(kda_bwd_prep_kernel<DK, DV, Tin, Tg, kTf32>, sp)) != cudaSuccess) return e;
    if ((e = set_smem(kda_bwd_states_kernel<DK, DV, kTf32>, sa)) != cudaSuccess) return e;
    if ((e = set_smem(kda_bwd_dstate_kernel<DK, DV, Tin, kTf32>, sb)) != cudaSuccess) return e;
    if ((e = set_smem(kda_bwd_grad_kernel<DK, DV, Tin, Tg, kTf32>, sc)) != cudaSuccess) return e;
    const dim3 gscan(p.dv / kDVD, p.H, p.B);
    const dim3 gchunk = seq::chunk_grid<kC>(p.B, p.T, p.H, packed);
    kda_bwd_prep_kernel<DK, DV, Tin, Tg, kTf32><<<gchunk, kThreads, sp, s>>>(p);
    kda_bwd_states_kernel<DK, DV, kTf32><<<gscan, kThreads, sa, s>>>(p);
    kda_bwd_dstate_kernel<DK, DV, Tin, kTf32><<<gscan, kThreads, sb, s>>>(p);
    kda_bwd_grad_kernel<DK, DV, Tin, Tg, kTf32><<<gchunk, kThreadsC, sc, s>>>(p);
    return cudaGetLastError();
}

template <typename Tin, typename Tg>
cudaError_t launch_typed(const BwdParams &p, cudaStream_t s) {
    if (p.dk == 64 && p.dv == 64) return launch_all<64, 64, Tin, Tg>(p, s);
    if (p.dk == 64 && p.dv == 128) return launch_all<64, 128, Tin, Tg>(p, s);
    if (p.dk == 128 && p.dv == 64) return launch_all<128, 64, Tin, Tg>(p, s);
    if (p.dk == 128 && p.dv == 128) return launch_all<128, 128, Tin, Tg>(p, s);
    return cudaErrorNotSupported;
}

}  // namespace

size_t bwd_state_bytes(int B, int T, int H, int dk, int dv, bool packed) {
    const size_t NS = chunk_slots(B, T, packed);
    return sizeof(float) * (size_t)H * ((2 * NS + B) * dv * dk + NS * rec_floats(dk, dv) + 2 * NS * kC * dv);
}

void bwd_carve(BwdParams &p, float *ws) {
    const size_t NS = chunk_slots(p.B, p.T, p.cu_seqlens != nullptr), H = p.H, st = (size_t)p.dv * p.dk;
    p.ws_S = ws;                                     // [H][NS + B state slots][dv][dk]
    p.ws_dS = p.ws_S + H * (NS + p.B) * st;          // [H][NS][dv][dk]
    p.ws_prep = p.ws_dS + H * NS * st;               // [H][NS] records
    p.ws_vnew = p.ws_prep + H * NS * rec_floats(p.dk, p.dv);
    p.ws_du = p.ws_vnew + H * NS * kC * p.dv;        // [H][NS][C][dv] each
}

cudaError_t launch_bwd_simt(const BwdParams &p, int in_bf16, int g_is_bf16, cudaStream_t s) {
    if (in_bf16)
        return g_is_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(p, s) : launch_typed<__nv_bfloat16, float>(p, s);
    return g_is_bf16 ? launch_typed<float, __nv_bfloat16>(p, s) : launch_typed<float, float>(p, s);
}

}  // namespace kda
