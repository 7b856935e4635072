// Backward of the general gated DPLR recurrence, chunk length C = 16, float32
// accumulation: the chunk products are warp-level tf32 tensor-core MMAs for
// bf16 inputs and exact float32 products on the CUDA cores for fp32 inputs.
//
// Page "Diagonal Plus Low Rank", section 3 derives, per chunk [t], with
// F = I + (B<- A->^T * M_{-1}), E = F^{-1}, W = E B<-,
// C = -E (B<- K->^T * M_{-1}) V, V_1 = V, V_2 = C - W S_prev^T and dS the
// gradient of the state after the chunk:
//
//   dC   = A-> Diag(gamma^C) dS^T + (Q<- A->^T * M)^T dO
//   dV_1 = K-> Diag(gamma^C) dS^T + (Q<- K->^T * M)^T dO,     dW = -dC S_prev
//   dE   = -dC V^T (B<- K->^T * M_{-1})^T + dW B<-^T,           dF = -E^T dE E^T
//   dQ<- = dO S_prev + (dO V_1^T * M) K-> + (dO V_2^T * M) A->
//   dB<- = E^T dW - (E^T dC V^T * M_{-1}) K-> + (dF * M_{-1}) A->
//   dK-> = (dO V_1^T * M)^T Q<- - (E^T dC V^T * M_{-1})^T B<- + V_1 dS Diag(gamma^C)
//   dA-> = (dO V_2^T * M)^T Q<- + (dF * M_{-1})^T B<- + V_2 dS Diag(gamma^C)
//   dV   = dV_1 - (B<- K->^T * M_{-1})^T E^T dC
//   dlogGamma = dQ<- * Q<- + dB<- * B<- - dK-> * K-> - dA-> * A->,  last row + diag(S^T dS)
//   dS_prev = dS Diag(gamma^C) + dO^T Q<- - dC^T W
//
// (dW against S_[t-1]; dB from dB<-; the state-update terms of dK-> and dA->,
// which the page's lines omit.)  With the clip of page "How to make GDN2 more
// stable", eq. (7), the gate is g' = min(g, -log rho): the gradient of g' goes
// to g where g < -log rho, and to -log rho elsewhere, from where it reaches a
// and b through the derivative of eq. (4).
//
// Four kernels, as for the KDA backward: a chunk-parallel prep kernel writes the
// state-independent operands of every chunk (W, K-> and A-> times gamma^C,
// Q<-, C, E, N_bk, P_k, P_a) once; the forward state scan and the reverse dS
// scan per (32-wide value slice, head, sequence) keep X and dC; then one CTA per
// (chunk, head, sequence) for every other gradient.
#include <cuda_bf16.h>

#include "dplr_common.cuh"
#include "kda_internal.h"
#include "packed_seq.cuh"
#include "warp_gemm.cuh"

namespace kda {
namespace {

using dplr::ldf;
using dplr::stf;

constexpr int kC = 16;       // chunk length
constexpr int kDVS = 32;
constexpr int kThreads = 256;

// Row strides = 4 (mod 32) for the fragment reads of the warp-tiled products.
__host__ __device__ constexpr int pad4(int n) { return n + 4; }
constexpr int kSC4 = pad4(kC);

// E = (I + Nm)^{-1} for a strictly lower 16 x 16 Nm: forward substitution,
// one column per thread of the first warp.  Starts after, ends with, a barrier.
template <int SC>
__device__ void inverse16(const float *Nm, float *Em) {
    if (threadIdx.x < kC) {
        const int c = threadIdx.x;
        for (int i = 0; i < kC; ++i) {
            float y = 0.f;
            if (i == c) y = 1.f;
            else if (i > c)
                for (int j = c; j < i; ++j) y -= Nm[i * SC + j] * Em[j * SC + c];
            Em[i * SC + c] = y;
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------------ chunk records
// Everything of a chunk that does not depend on the state (float32), written
// once by the prep kernel: W = E B<-, K~ = K-> Diag(gamma^C), A~ = A-> Diag(gamma^C),
// Q<-, C = -E (B<- K->^T * M_{-1}) V, E, N_bk = B<- K->^T * M_{-1}, P_k, P_a and gamma^C.
__host__ __device__ constexpr size_t bwd_rec_floats(int dk, int dv) {
    return (size_t)4 * kC * dk + (size_t)kC * dv + (size_t)4 * kC * kC + dk;
}
template <int DK, int DV>
struct BRec {
    static constexpr int W = 0, KG = kC * DK, AG = 2 * kC * DK, QL = 3 * kC * DK, CC = 4 * kC * DK,
                         E = CC + kC * DV, NK = E + kC * kC, PK = NK + kC * kC, PA = PK + kC * kC,
                         GC = PA + kC * kC;
    static_assert(bwd_rec_floats(DK, DV) == (size_t)GC + DK && bwd_rec_floats(DK, DV) % 4 == 0, "record");
};

// ------------------------------------------------------------------ prep kernel
// One CTA per (chunk, head, sequence).  Products run as warp-tiled blocks
// (warp_gemm.cuh): tf32 tensor-core MMAs for bf16 inputs (TF32), exact float32
// for float32 inputs.
template <int DK, int DV, typename Tin, typename Tg, bool TF32>
__global__ void __launch_bounds__(kThreads) dplr_bwd_prep_kernel(const DplrParams p) {
    constexpr int SK = pad4(DK), SV = pad4(DV), SC = kSC4;
    using R = BRec<DK, DV>;
    extern __shared__ float smem[];
    float4 *rows = reinterpret_cast<float4 *>(smem);      // [C]
    float *Gm = smem + 4 * kC;           // [C][SK]  raw gate, then Gamma
    float *Ql = Gm + kC * SK;
    float *Kr = Ql + kC * SK;
    float *Ar = Kr + kC * SK;
    float *Bl = Ar + kC * SK;
    float *Vm = Bl + kC * SK;            // [C][SV]
    float *T1 = Vm + kC * SV;            // [C][SV]  N_bk V
    float *Nm = T1 + kC * SV;            // [C][SC]
    float *Em = Nm + kC * SC;
    float *Nk = Em + kC * SC;
    float *gam = Nk + kC * SC;           // [DK]
    float *gsc = gam + DK;               // [C]

    const int tid = threadIdx.x, h = blockIdx.y;
    int b, n;
    seq::Seq sq;
    if (!seq::chunk_of<kC>(p, b, n, sq)) return;
    const int H = p.H;
    const int t0 = n * kC, nvalid = min(kC, sq.len - t0);
    const size_t row = (size_t)sq.row0 + t0;
    const Tin *v = static_cast<const Tin *>(p.v);
    float *rec = p.ws_prep + seq::chunk_index<kC>(p, sq, h, n) * bwd_rec_floats(DK, DV);

    if (p.clip) {
        dplr::row_rho<DK, kC, Tin>(p, row, h, nvalid, rows);
        __syncthreads();
    }
    wg::load_tile<kC, DV, SV, kThreads>(v + (row * H + h) * DV, (size_t)H * DV, nvalid, Vm);
    dplr::load_rescaled_par<DK, SK, kC, Tin, Tg>(p, row, h, nvalid, rows, Gm, Ql, Kr, Ar, Bl, gam, gsc);
    __syncthreads();
    {
        auto bAr = [&](int d, int j) { return Ar[j * SK + d]; };
        auto bKr = [&](int d, int j) { return Kr[j * SK + d]; };
        auto aBl = [&](int i, int d) { return Bl[i * SK + d]; };
        auto aQl = [&](int i, int d) { return Ql[i * SK + d]; };
        wg::gemm16_pair<kC, TF32>(DK, aBl, bAr, DK, aBl, bKr, [&](int i, int j, float x, float y) {
            Nm[i * SC + j] = j < i ? x : 0.f;
            const float nk = j < i ? y : 0.f;
            Nk[i * SC + j] = nk;
            rec[R::NK + i * kC + j] = nk;
        });
        wg::gemm16_pair<kC, TF32>(DK, aQl, bKr, DK, aQl, bAr, [&](int i, int j, float x, float y) {
            rec[R::PK + i * kC + j] = j <= i ? x : 0.f;
            rec[R::PA + i * kC + j] = j <= i ? y : 0.f;
        });
    }
    for (int idx = tid; idx < kC * DK; idx += kThreads) {
        const int i = idx / DK, d = idx % DK;
        rec[R::KG + idx] = Kr[i * SK + d] * gam[d];
        rec[R::AG + idx] = Ar[i * SK + d] * gam[d];
        rec[R::QL + idx] = Ql[i * SK + d];
    }
    for (int d = tid; d < DK; d += kThreads) rec[R::GC + d] = gam[d];
    __syncthreads();
    inverse16<SC>(Nm, Em);
    for (int idx = tid; idx < kC * kC; idx += kThreads) rec[R::E + idx] = Em[(idx / kC) * SC + idx % kC];
    wg::gemm16<DK, TF32>(
        kC, [&](int i, int j) { return Em[i * SC + j]; }, [&](int j, int d) { return Bl[j * SK + d]; },
        [&](int i, int d, float x) { rec[R::W + i * DK + d] = x; });
    wg::gemm16<DV, TF32>(
        kC, [&](int i, int j) { return Nk[i * SC + j]; }, [&](int j, int e) { return Vm[j * SV + e]; },
        [&](int i, int e, float x) { T1[i * SV + e] = x; });
    __syncthreads();
    wg::gemm16<DV, TF32>(
        kC, [&](int i, int j) { return Em[i * SC + j]; }, [&](int j, int e) { return T1[j * SV + e]; },
        [&](int i, int e, float x) { rec[R::CC + i * DV + e] = -x; });
}

template <int DK, int DV>
constexpr size_t prep_smem_bytes() {
    return sizeof(float) * ((size_t)4 * kC + 5 * kC * pad4(DK) + 2 * kC * pad4(DV) + 3 * kC * kSC4 + DK + kC);
}

// The two scans read each chunk's record tiles (and v or dO) through a ring of
// kRing buffers filled by cp.async: chunk n computes while chunks n + 1 and n + 2
// are in flight.
constexpr int kRing = 3;

// ------------------------------------------------------------------ kernel A
// The forward state scan from the records: X = C - W S^T (kept for the
// gradient kernel), S <- S Diag(gamma^C) + V^T K~ + X^T A~.
template <int DK, typename Tin>
__host__ __device__ constexpr int states_buf_floats() {
    // W, K~, A~ [C][SK]; C slice [C][SV]; gamma^C [DK]; raw v rows [C][DVS] of Tin
    return 3 * kC * pad4(DK) + kC * pad4(kDVS) + DK + (kC * kDVS * (int)sizeof(Tin) + 3) / 4;
}
template <int DK, int DV, typename Tin, bool TF32>
__global__ void __launch_bounds__(kThreads) dplr_bwd_states_kernel(const DplrParams p) {
    constexpr int SK = pad4(DK), SV = pad4(kDVS), BUF = states_buf_floats<DK, Tin>();
    using R = BRec<DK, DV>;
    extern __shared__ float smem[];
    float *Sm = smem;                    // [DVS][SK]
    float *Vm = Sm + kDVS * SK;          // [C][SV]
    float *Xm = Vm + kC * SV;            // [C][SV]
    float *ring = Xm + kC * SV;          // kRing x BUF

    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * kDVS, h = blockIdx.y, b = blockIdx.z;
    const int H = p.H, dv = p.dv;
    const seq::Seq sq = seq::seq_of<kC>(p, b);
    const int N = sq.nch, T = sq.len;
    const size_t row0 = sq.row0, ci0 = seq::chunk_index<kC>(p, sq, h, 0);
    const Tin *v = static_cast<const Tin *>(p.v);
    const size_t head = (size_t)b * H + h;
    float *Sws = p.ws_S + seq::state_index<kC>(p, sq, b, h, 0) * dv * DK;
    const float *recs = p.ws_prep + ci0 * bwd_rec_floats(DK, DV);
    auto issue = [&](int n) {
        const float *rec = recs + (size_t)n * bwd_rec_floats(DK, DV);
        float *bf = ring + (n % kRing) * BUF;
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::W, DK, bf);
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::KG, DK, bf + kC * SK);
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::AG, DK, bf + 2 * kC * SK);
        wg::load_tile_async<kC, kDVS, SV, kThreads>(rec + R::CC + e0, DV, bf + 3 * kC * SK);
        wg::load_tile_async<1, DK, DK, kThreads>(rec + R::GC, DK, bf + 3 * kC * SK + kC * SV);
        wg::load_raw_async<kC, kDVS, Tin, kThreads>(v + ((row0 + n * kC) * H + h) * dv + e0, (size_t)H * dv,
                                                    min(kC, T - n * kC),
                                                    reinterpret_cast<Tin *>(bf + 3 * kC * SK + kC * SV + DK));
    };

    for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
        const int e = idx / DK, d = idx % DK;
        Sm[e * SK + d] = p.h0 ? p.h0[(head * dv + e0 + e) * DK + d] : 0.f;
    }
    for (int n = 0; n < kRing - 1; ++n) {
        if (n < N) issue(n);
        wg::cp_async_commit();
    }
    for (int n = 0; n < N; ++n) {
        float *Wm = ring + (n % kRing) * BUF, *KG = Wm + kC * SK, *AG = KG + kC * SK, *Cs = AG + kC * SK;
        float *gam = Cs + kC * SV;
        const Tin *vraw = reinterpret_cast<const Tin *>(gam + DK);
        __syncthreads();                 // S is final for chunk n; chunk n - 1's buffer is free
        for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
            const int e = idx / DK, d = idx % DK;
            Sws[((size_t)n * dv + e0 + e) * DK + d] = Sm[e * SK + d];
        }
        if (n + kRing - 1 < N) issue(n + kRing - 1);
        wg::cp_async_commit();           // (empty groups at the end keep the count)
        wg::cp_async_wait<kRing - 1>();  // chunk n's copies (this thread's) have landed
        __syncthreads();
        wg::to_f32<kC, kDVS, SV, Tin, kThreads>(vraw, Vm);
        float *xs = p.ws_x + ((ci0 + n) * kC) * (size_t)dv + e0;
        wg::gemm16<kDVS, TF32>(
            DK, [&](int i, int d) { return Wm[i * SK + d]; }, [&](int d, int e) { return Sm[e * SK + d]; },
            [&](int i, int e, float x) {
                const float y = Cs[i * SV + e] - x;
                Xm[i * SV + e] = y;
                xs[(size_t)i * dv + e] = y;
            });
        __syncthreads();
        wg::gemm2<DK, TF32>(
            kC, [&](int e, int c) { return Vm[c * SV + e]; }, [&](int c, int d) { return KG[c * SK + d]; }, kC,
            [&](int e, int c) { return Xm[c * SV + e]; }, [&](int c, int d) { return AG[c * SK + d]; },
            [&](int e, int d, float x) { Sm[e * SK + d] = Sm[e * SK + d] * gam[d] + x; });
    }
    __syncthreads();
    for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
        const int e = idx / DK, d = idx % DK;
        Sws[((size_t)N * dv + e0 + e) * DK + d] = Sm[e * SK + d];
    }
}

// ------------------------------------------------------------------ kernel B
// The reverse scan from the records: dC = A~ dS^T + P_a^T dO (kept for the
// gradient kernel), dS <- dS Diag(gamma^C) + dO^T Q<- - dC^T W.
template <int DK, typename Tin>
__host__ __device__ constexpr int dstate_buf_floats() {
    // W, A~, Q<- [C][SK]; P_a [C][SC]; gamma^C [DK]; raw dO rows [C][DVS] of Tin
    return 3 * kC * pad4(DK) + kC * kSC4 + DK + (kC * kDVS * (int)sizeof(Tin) + 3) / 4;
}
template <int DK, int DV, typename Tin, bool TF32>
__global__ void __launch_bounds__(kThreads) dplr_bwd_dstate_kernel(const DplrParams p) {
    constexpr int SK = pad4(DK), SV = pad4(kDVS), SC = kSC4, BUF = dstate_buf_floats<DK, Tin>();
    using R = BRec<DK, DV>;
    extern __shared__ float smem[];
    float *dS = smem;                    // [DVS][SK]
    float *dO = dS + kDVS * SK;          // [C][SV]
    float *dC = dO + kC * SV;            // [C][SV]
    float *ring = dC + kC * SV;          // kRing x BUF

    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * kDVS, h = blockIdx.y, b = blockIdx.z;
    const int H = p.H, dv = p.dv;
    const seq::Seq sq = seq::seq_of<kC>(p, b);
    const int N = sq.nch, T = sq.len;
    const size_t row0 = sq.row0, ci0 = seq::chunk_index<kC>(p, sq, h, 0);
    const Tin *dop = static_cast<const Tin *>(p.grad_o);
    const size_t head = (size_t)b * H + h;
    float *dSws = p.ws_dS + ci0 * dv * DK;
    const float *recs = p.ws_prep + ci0 * bwd_rec_floats(DK, DV);
    // step i handles chunk N - 1 - i (the scan runs backwards)
    auto issue = [&](int i) {
        const int n = N - 1 - i;
        const float *rec = recs + (size_t)n * bwd_rec_floats(DK, DV);
        float *bf = ring + (i % kRing) * BUF;
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::W, DK, bf);
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::AG, DK, bf + kC * SK);
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::QL, DK, bf + 2 * kC * SK);
        wg::load_tile_async<kC, kC, SC, kThreads>(rec + R::PA, kC, bf + 3 * kC * SK);
        wg::load_tile_async<1, DK, DK, kThreads>(rec + R::GC, DK, bf + 3 * kC * SK + kC * SC);
        wg::load_raw_async<kC, kDVS, Tin, kThreads>(dop + ((row0 + n * kC) * H + h) * dv + e0,
                                                    (size_t)H * dv, min(kC, T - n * kC),
                                                    reinterpret_cast<Tin *>(bf + 3 * kC * SK + kC * SC + DK));
    };

    for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
        const int e = idx / DK, d = idx % DK;
        dS[e * SK + d] = p.grad_ht ? p.grad_ht[(head * dv + e0 + e) * DK + d] : 0.f;
    }
    for (int i = 0; i < kRing - 1; ++i) {
        if (i < N) issue(i);
        wg::cp_async_commit();
    }
    for (int i = 0; i < N; ++i) {
        const int n = N - 1 - i;
        float *Wm = ring + (i % kRing) * BUF, *AG = Wm + kC * SK, *QL = AG + kC * SK, *Pa = QL + kC * SK;
        float *gam = Pa + kC * SC;
        const Tin *draw = reinterpret_cast<const Tin *>(gam + DK);
        __syncthreads();                 // dS is final for chunk n; the previous step's buffer is free
        for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
            const int e = idx / DK, d = idx % DK;
            dSws[((size_t)n * dv + e0 + e) * DK + d] = dS[e * SK + d];
        }
        if (i + kRing - 1 < N) issue(i + kRing - 1);
        wg::cp_async_commit();
        wg::cp_async_wait<kRing - 1>();
        __syncthreads();
        wg::to_f32<kC, kDVS, SV, Tin, kThreads>(draw, dO);
        __syncthreads();
        float *dcs = p.ws_dc + ((ci0 + n) * kC) * (size_t)dv + e0;
        wg::gemm16_2<kDVS, TF32>(
            DK, [&](int r, int d) { return AG[r * SK + d]; }, [&](int d, int e) { return dS[e * SK + d]; }, kC,
            [&](int r, int j) { return Pa[j * SC + r]; }, [&](int j, int e) { return dO[j * SV + e]; },
            [&](int r, int e, float x) {
                dC[r * SV + e] = x;
                dcs[(size_t)r * dv + e] = x;
            });
        __syncthreads();
        wg::gemm2<DK, TF32>(
            kC, [&](int e, int c) { return dO[c * SV + e]; }, [&](int c, int d) { return QL[c * SK + d]; }, kC,
            [&](int e, int c) { return -dC[c * SV + e]; }, [&](int c, int d) { return Wm[c * SK + d]; },
            [&](int e, int d, float x) { dS[e * SK + d] = dS[e * SK + d] * gam[d] + x; });
    }
    __syncthreads();
    if (p.grad_h0) {
        for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
            const int e = idx / DK, d = idx % DK;
            p.grad_h0[(head * dv + e0 + e) * DK + d] = dS[e * SK + d];
        }
    }
}

// ------------------------------------------------------------------ kernel C
template <int DK, int DV>
constexpr size_t grad_smem_floats() {
    return (size_t)4 * kC + (size_t)10 * kC * pad4(DK) + (size_t)5 * kC * pad4(DV) + (size_t)12 * kC * kSC4 + DK +
           3 * kC + DK + 32 * pad4(DK) + kC * pad4(DV);
}

template <int DK, int DV, typename Tin, typename Tg, bool TF32>
__global__ void __launch_bounds__(kThreads) dplr_bwd_grad_kernel(const DplrParams p) {
    constexpr int SK = pad4(DK), SV = pad4(DV), SC = kSC4;
    extern __shared__ float smem[];
    float4 *rows = reinterpret_cast<float4 *>(smem);      // [C] (|a|^2, |b|^2, a.b, -log rho)
    float *Gm = smem + 4 * kC;           // [C][SK] Gamma
    float *Ql = Gm + kC * SK;
    float *Kr = Ql + kC * SK;
    float *Ar = Kr + kC * SK;
    float *Bl = Ar + kC * SK;
    float *Wm = Bl + kC * SK;            // W, then dW
    float *dQl = Wm + kC * SK;           // dQ<-, then dlogGamma, then dg'
    float *dKr = dQl + kC * SK;
    float *dAr = dKr + kC * SK;
    float *dBl = dAr + kC * SK;
    float *Vm = dBl + kC * SK;           // [C][SV]
    float *dO = Vm + kC * SV;
    float *V2 = dO + kC * SV;
    float *dC = V2 + kC * SV;
    float *Ym = dC + kC * SV;            // Nk V, then E^T dC
    float *Nm = Ym + kC * SV;            // [C][SC] B<- A->^T * M_{-1}
    float *Em = Nm + kC * SC;
    float *Nk = Em + kC * SC;            // B<- K->^T * M_{-1}
    float *Pk = Nk + kC * SC;            // Q<- K->^T * M
    float *Pa = Pk + kC * SC;            // Q<- A->^T * M
    float *O1 = Pa + kC * SC;            // dO V^T * M
    float *O2 = O1 + kC * SC;            // dO V_2^T * M
    float *Z1 = O2 + kC * SC;            // dC V^T
    float *dE = Z1 + kC * SC;
    float *Gx = dE + kC * SC;            // E^T dC V^T * M_{-1}
    float *dF = Gx + kC * SC;
    float *Tt = dF + kC * SC;
    float *gam = Tt + kC * SC;           // [DK]
    float *rsum = gam + DK;              // [C] row sums / dL/d(-log rho)
    float *aux = rsum + kC;              // [C]
    float *gsc = aux + kC;               // [C]
    float *lastrow = gsc + kC;           // [DK] diag(S_next^T dS)
    float *slab = lastrow + DK;          // [32][SK] staged state rows
    float *dVs = slab + 32 * SK;         // [C][SV] K-> Diag(gamma^C) dS^T

    const int tid = threadIdx.x, h = blockIdx.y;
    int b, n;
    seq::Seq sq;
    if (!seq::chunk_of<kC>(p, b, n, sq)) return;
    const int H = p.H;
    const int t0 = n * kC, nvalid = min(kC, sq.len - t0);
    const size_t row = (size_t)sq.row0 + t0, ci = seq::chunk_index<kC>(p, sq, h, n);
    const Tin *v = static_cast<const Tin *>(p.v);
    const Tin *dop = static_cast<const Tin *>(p.grad_o);
    const float *Sp = p.ws_S + seq::state_index<kC>(p, sq, b, h, n) * DV * DK;
    const float *Sn = Sp + (size_t)DV * DK;
    const float *dS = p.ws_dS + ci * DV * DK;

    if (p.clip) {
        dplr::row_rho<DK, kC, Tin>(p, row, h, nvalid, rows);
        __syncthreads();
    }
    {
        const size_t r0 = (row * H + h) * DV, rs = (size_t)H * DV;
        wg::load_tile<kC, DV, SV, kThreads>(v + r0, rs, nvalid, Vm);
        wg::load_tile<kC, DV, SV, kThreads>(dop + r0, rs, nvalid, dO);
    }
    dplr::load_rescaled_par<DK, SK, kC, Tin, Tg>(p, row, h, nvalid, rows, Gm, Ql, Kr, Ar, Bl, gam, gsc);
    __syncthreads();
    // E, N_bk, P_k, P_a and W from the chunk record; V_2 (= X) and dC from the scans
    {
        using R = BRec<DK, DV>;
        const float *rec = p.ws_prep + ci * bwd_rec_floats(DK, DV);
        wg::load_tile<kC, kC, SC, kThreads>(rec + R::E, kC, kC, Em);
        wg::load_tile<kC, kC, SC, kThreads>(rec + R::NK, kC, kC, Nk);
        wg::load_tile<kC, kC, SC, kThreads>(rec + R::PK, kC, kC, Pk);
        wg::load_tile<kC, kC, SC, kThreads>(rec + R::PA, kC, kC, Pa);
        wg::load_tile<kC, DK, SK, kThreads>(rec + R::W, DK, kC, Wm);
        wg::load_tile<kC, DV, SV, kThreads>(p.ws_x + ci * kC * DV, DV, kC, V2);
        wg::load_tile<kC, DV, SV, kThreads>(p.ws_dc + ci * kC * DV, DV, kC, dC);
    }
    __syncthreads();
    // O1 = dO V^T * M ; O2 = dO V_2^T * M ; Z1 = dC V^T
    {
        auto aDO = [&](int i, int e) { return dO[i * SV + e]; };
        auto bV = [&](int e, int j) { return Vm[j * SV + e]; };
        wg::gemm16_pair<kC, TF32>(DV, aDO, bV, DV, aDO, [&](int e, int j) { return V2[j * SV + e]; },
                                  [&](int i, int j, float x, float y) {
                                      O1[i * SC + j] = j <= i ? x : 0.f;
                                      O2[i * SC + j] = j <= i ? y : 0.f;
                                  });
        wg::gemm16<kC, TF32>(DV, [&](int i, int e) { return dC[i * SV + e]; }, bV,
                             [&](int i, int j, float x) { Z1[i * SC + j] = x; });
    }
    __syncthreads();
    // dW = -dC S_prev ; dQ<- ; dK-> and dA-> without their F/G terms ; the dS term of dV ;
    // diag(S_next^T dS) for the gamma^C row.  The stored states stream through
    // shared memory 32 rows at a time (16-byte loads).
    {
        constexpr int NT = wg::nt16<DK>();
        int c0;
        wg::origin16<DK>(c0);
        float aW[NT][4] = {}, aQ[NT][4] = {}, aK[NT][4] = {}, aA[NT][4] = {}, aK2[NT][4] = {}, aA2[NT][4] = {};
        for (int s0 = 0; s0 < DV; s0 += 32) {
            wg::load_tile<32, DK, SK, kThreads>(Sp + (size_t)s0 * DK, DK, 32, slab);
            __syncthreads();
            auto bS = [&](int e, int d) { return slab[e * SK + d]; };
            wg::tile<NT, TF32>(aW, 0, c0, 32, [&](int i, int e) { return dC[i * SV + s0 + e]; }, bS);
            wg::tile<NT, TF32>(aQ, 0, c0, 32, [&](int i, int e) { return dO[i * SV + s0 + e]; }, bS);
            __syncthreads();
        }
        float last = 0.f;                    // diag(S_next^T dS), column tid
        for (int s0 = 0; s0 < DV; s0 += 32) {
            wg::load_tile<32, DK, SK, kThreads>(dS + (size_t)s0 * DK, DK, 32, slab);
            float sn[32];
            if (tid < DK)
#pragma unroll
                for (int e = 0; e < 32; ++e) sn[e] = Sn[(size_t)(s0 + e) * DK + tid];
            __syncthreads();
            auto bS = [&](int e, int d) { return slab[e * SK + d]; };
            wg::tile<NT, TF32>(aK, 0, c0, 32, [&](int i, int e) { return Vm[i * SV + s0 + e]; }, bS);
            wg::tile<NT, TF32>(aA, 0, c0, 32, [&](int i, int e) { return V2[i * SV + s0 + e]; }, bS);
            wg::gemm16<32, TF32>(
                DK, [&](int i, int d) { return Kr[i * SK + d] * gam[d]; }, [&](int d, int e) { return slab[e * SK + d]; },
                [&](int i, int e, float x) { dVs[i * SV + s0 + e] = x; });
            if (tid < DK)
#pragma unroll
                for (int e = 0; e < 32; ++e) last += sn[e] * slab[e * SK + tid];
            __syncthreads();
        }
        if (tid < DK) lastrow[tid] = last;
        wg::tile<NT, TF32>(aQ, 0, c0, kC, [&](int i, int j) { return O1[i * SC + j]; },
                           [&](int j, int d) { return Kr[j * SK + d]; });
        wg::tile<NT, TF32>(aQ, 0, c0, kC, [&](int i, int j) { return O2[i * SC + j]; },
                           [&](int j, int d) { return Ar[j * SK + d]; });
        auto bQl = [&](int j, int d) { return Ql[j * SK + d]; };
        wg::tile<NT, TF32>(aK2, 0, c0, kC, [&](int i, int j) { return O1[j * SC + i]; }, bQl);
        wg::tile<NT, TF32>(aA2, 0, c0, kC, [&](int i, int j) { return O2[j * SC + i]; }, bQl);
        wg::store<NT>(aW, 0, c0, [&](int i, int d, float x) { Wm[i * SK + d] = -x; });
        wg::store<NT>(aQ, 0, c0, [&](int i, int d, float x) { dQl[i * SK + d] = x; });
        wg::store_pair<NT>(aK, aK2, 0, c0, [&](int i, int d, float x1, float x2) { dKr[i * SK + d] = x1 * gam[d] + x2; });
        wg::store_pair<NT>(aA, aA2, 0, c0, [&](int i, int d, float x1, float x2) { dAr[i * SK + d] = x1 * gam[d] + x2; });
    }
    wg::gemm16<DV, TF32>(
        kC, [&](int i, int j) { return Em[j * SC + i]; }, [&](int j, int e) { return dC[j * SV + e]; },
        [&](int i, int e, float x) { Ym[i * SV + e] = x; });
    __syncthreads();
    // dE = -Z1 Nk^T + dW B<-^T ; G = (Y V^T) * M_{-1}
    wg::gemm16_2<kC, TF32>(
        kC, [&](int i, int l) { return -Z1[i * SC + l]; }, [&](int l, int j) { return Nk[j * SC + l]; }, DK,
        [&](int i, int d) { return Wm[i * SK + d]; }, [&](int d, int j) { return Bl[j * SK + d]; },
        [&](int i, int j, float x) { dE[i * SC + j] = x; });
    wg::gemm16<kC, TF32>(
        DV, [&](int i, int e) { return Ym[i * SV + e]; }, [&](int e, int j) { return Vm[j * SV + e]; },
        [&](int i, int j, float x) { Gx[i * SC + j] = j < i ? x : 0.f; });
    __syncthreads();
    // dF = -E^T dE E^T (only dF * M_{-1} is used)
    wg::gemm16<kC, TF32>(
        kC, [&](int i, int l) { return dE[i * SC + l]; }, [&](int l, int j) { return Em[j * SC + l]; },
        [&](int i, int j, float x) { Tt[i * SC + j] = x; });
    __syncthreads();
    wg::gemm16<kC, TF32>(
        kC, [&](int i, int l) { return Em[l * SC + i]; }, [&](int l, int j) { return Tt[l * SC + j]; },
        [&](int i, int j, float x) { dF[i * SC + j] = j < i ? -x : 0.f; });
    __syncthreads();
    // dB<- = E^T dW - G K-> + (dF * M_{-1}) A-> ; dK-> -= G^T B<- ; dA-> += (dF * M_{-1})^T B<-
    wg::gemm16_3<DK, TF32>(
        kC, [&](int i, int j) { return Em[j * SC + i]; }, [&](int j, int d) { return Wm[j * SK + d]; }, kC,
        [&](int i, int j) { return -Gx[i * SC + j]; }, [&](int j, int d) { return Kr[j * SK + d]; }, kC,
        [&](int i, int j) { return dF[i * SC + j]; }, [&](int j, int d) { return Ar[j * SK + d]; },
        [&](int i, int d, float x) { dBl[i * SK + d] = x; });
    {
        auto bBl = [&](int j, int d) { return Bl[j * SK + d]; };
        wg::gemm16_pair<DK, TF32>(
            kC, [&](int i, int j) { return Gx[j * SC + i]; }, bBl, kC, [&](int i, int j) { return dF[j * SC + i]; }, bBl,
            [&](int i, int d, float xg, float xf) {
                dKr[i * SK + d] -= xg;
                dAr[i * SK + d] += xf;
            });
    }
    // dV = K-> Diag(gamma^C) dS^T + P_k^T dO - Nk^T (E^T dC)
    {
        Tin *gv = static_cast<Tin *>(p.grad_v);
        wg::gemm16_2<DV, TF32>(
            kC, [&](int i, int j) { return Pk[j * SC + i]; }, [&](int j, int e) { return dO[j * SV + e]; }, kC,
            [&](int i, int j) { return -Nk[j * SC + i]; }, [&](int j, int e) { return Ym[j * SV + e]; },
            [&](int i, int e, float x) {
                if (i < nvalid) stf(gv, ((row + i) * H + h) * DV + e, x + dVs[i * SV + e]);
            });
    }
    __syncthreads();
    // dq, dk ; dlogGamma into dQl
    Tin *gq = static_cast<Tin *>(p.grad_q);
    Tin *gk = static_cast<Tin *>(p.grad_k);
    for (int idx = tid; idx < kC * DK; idx += kThreads) {
        const int i = idx / DK, d = idx % DK;
        const float gm = Gm[i * SK + d], dq = dQl[i * SK + d];
        if (i < nvalid) {
            const size_t off = ((row + i) * H + h) * DK + d;
            stf(gq, off, dq * gm);
            stf(gk, off, dKr[i * SK + d] / gm);
        }
        dQl[i * SK + d] = dq * Ql[i * SK + d] + dBl[i * SK + d] * Bl[i * SK + d] - dKr[i * SK + d] * Kr[i * SK + d] -
                          dAr[i * SK + d] * Ar[i * SK + d];
    }
    __syncthreads();
    // dg' = in-chunk suffix sums of dlogGamma, the gamma^C row adding diag(S_next^T dS)
    const bool channel = p.gate_kind == KDA_GATE_CHANNEL;
    for (int d = tid; d < DK; d += kThreads) {
        float run = lastrow[d];              // diag(S_next^T dS), from the state pass above
        for (int i = kC - 1; i >= 0; --i) {
            run += dQl[i * SK + d];
            dQl[i * SK + d] = run;
        }
    }
    __syncthreads();
    Tg *gg = static_cast<Tg *>(p.grad_g);
    const Tg *graw = static_cast<const Tg *>(p.g);
    const int warp = tid >> 5, lane = tid & 31;
    if (channel) {
        for (int i = warp; i < kC; i += kThreads / 32) {
            float lost = 0.f;
            if (i < nvalid) {
                const size_t tok = (row + i) * H + h;
                for (int d = lane; d < DK; d += 32) {
                    const float dgp = dQl[i * SK + d];
                    const bool keep = !p.clip || ldf(graw, tok * DK + d) < rows[i].w;
                    stf(gg, tok * DK + d, keep ? dgp : 0.f);
                    if (!keep) lost += dgp;
                }
            }
            lost = dplr::warp_sum(lost);
            if (lane == 0) rsum[i] = lost;
        }
    } else {
        // one decay per token (scalar gate, or the clip acting on no gate): dg'_t = sum over channels
        for (int i = warp; i < kC; i += kThreads / 32) {
            float acc = 0.f;
            for (int d = lane; d < DK; d += 32) acc += dQl[i * SK + d];
            acc = dplr::warp_sum(acc);
            if (lane == 0) {
                float lost = 0.f;
                if (i < nvalid) {
                    const size_t tok = (row + i) * H + h;
                    const float g0 = p.gate_kind == KDA_GATE_SCALAR ? ldf(graw, tok) : 0.f;
                    const bool keep = !p.clip || g0 < rows[i].w;
                    if (p.gate_kind == KDA_GATE_SCALAR) stf(gg, tok, keep ? acc : 0.f);
                    if (!keep) lost = acc;
                }
                rsum[i] = lost;
            }
        }
    }
    __syncthreads();
    // da, db; with the clip, plus dL/d(-log rho) * d(-log rho)/d(a, b) through eq. (4)
    if (tid < kC) {
        const int i = tid;
        float sa = 0.f, sb = 0.f;
        if (p.clip && i < nvalid) {
            const float4 r = rows[i];
            const float na = sqrtf(r.x), nb = sqrtf(r.y), eta = na * nb;
            const float R = sqrtf(fmaxf(eta * eta - 4.f * r.z + 4.f, 1e-30f));
            const float rho = 0.5f * (eta + R);
            const float scale = -rsum[i] / rho;      // dL/d rho
            // d rho/d a = 0.5 ((1 + eta/R) |b|/|a| a - 2 b / R), and symmetrically for b
            const float f = 0.5f * (1.f + eta / R);
            sa = scale * f * (na > 0.f ? nb / na : 0.f);
            sb = scale * f * (nb > 0.f ? na / nb : 0.f);
            rsum[i] = scale / R;                     // coefficient of the cross terms
        }
        aux[i] = sa;
        Tt[i] = sb;                                  // Tt is free again
    }
    __syncthreads();
    Tin *ga = static_cast<Tin *>(p.grad_a);
    Tin *gb = static_cast<Tin *>(p.grad_b);
    const Tin *araw = static_cast<const Tin *>(p.a);
    const Tin *braw = static_cast<const Tin *>(p.b);
    for (int idx = tid; idx < kC * DK; idx += kThreads) {
        const int i = idx / DK, d = idx % DK;
        if (i >= nvalid) continue;
        const size_t off = ((row + i) * H + h) * DK + d;
        const float gm = Gm[i * SK + d];
        float da = dAr[i * SK + d] / gm, db = dBl[i * SK + d] * gm;
        if (p.clip) {
            const float av = ldf(araw, off), bv = ldf(braw, off), cross = rsum[i];
            da += aux[i] * av - cross * bv;
            db += Tt[i] * bv - cross * av;
        }
        stf(ga, off, da);
        stf(gb, off, db);
    }
}

template <int DK, typename Tin>
constexpr size_t states_smem_bytes() {
    return sizeof(float) * ((size_t)kDVS * pad4(DK) + 2 * kC * pad4(kDVS) + kRing * states_buf_floats<DK, Tin>());
}
template <int DK, typename Tin>
constexpr size_t dstate_smem_bytes() {
    return sizeof(float) * ((size_t)kDVS * pad4(DK) + 2 * kC * pad4(kDVS) + kRing * dstate_buf_floats<DK, Tin>());
}

template <typename F>
cudaError_t set_smem(F *fn, size_t bytes) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int DK, int DV, typename Tin, typename Tg>
cudaError_t launch_all(const DplrParams &p, cudaStream_t s) {
    constexpr bool kTf32 = sizeof(Tin) == 2;        // bf16 inputs: tf32 tensor-core products
    cudaError_t e;
    const size_t sp = prep_smem_bytes<DK, DV>(), sa = states_smem_bytes<DK, Tin>(), sb = dstate_smem_bytes<DK, Tin>();
    const size_t sc = sizeof(float) * grad_smem_floats<DK, DV>();
    static_assert(sizeof(float) * grad_smem_floats<128, 128>() <= 227 * 1024, "kernel C shared memory");
    if ((e = set_smem(dplr_bwd_prep_kernel<DK, DV, Tin, Tg, kTf32>, sp)) != cudaSuccess) return e;
    if ((e = set_smem(dplr_bwd_states_kernel<DK, DV, Tin, kTf32>, sa)) != cudaSuccess) return e;
    if ((e = set_smem(dplr_bwd_dstate_kernel<DK, DV, Tin, kTf32>, sb)) != cudaSuccess) return e;
    if ((e = set_smem(dplr_bwd_grad_kernel<DK, DV, Tin, Tg, kTf32>, sc)) != cudaSuccess) return e;
    const dim3 gscan(p.dv / kDVS, p.H, p.B), gchunk = seq::chunk_grid<kC>(p.B, p.T, p.H, p.cu_seqlens != nullptr);
    dplr_bwd_prep_kernel<DK, DV, Tin, Tg, kTf32><<<gchunk, kThreads, sp, s>>>(p);
    dplr_bwd_states_kernel<DK, DV, Tin, kTf32><<<gscan, kThreads, sa, s>>>(p);
    dplr_bwd_dstate_kernel<DK, DV, Tin, kTf32><<<gscan, kThreads, sb, s>>>(p);
    dplr_bwd_grad_kernel<DK, DV, Tin, Tg, kTf32><<<gchunk, kThreads, sc, s>>>(p);
    return cudaGetLastError();
}

template <typename Tin, typename Tg>
cudaError_t launch_typed(const DplrParams &p, cudaStream_t s) {
    if (p.dk == 64 && p.dv == 64) return launch_all<64, 64, Tin, Tg>(p, s);
    if (p.dk == 64 && p.dv == 128) return launch_all<64, 128, Tin, Tg>(p, s);
    if (p.dk == 128 && p.dv == 64) return launch_all<128, 64, Tin, Tg>(p, s);
    if (p.dk == 128 && p.dv == 128) return launch_all<128, 128, Tin, Tg>(p, s);
    return cudaErrorNotSupported;
}

}  // namespace

size_t dplr_bwd_state_bytes(int B, int T, int H, int dk, int dv, bool packed) {
    const size_t NS = seq::chunk_slots<kC>(B, T, packed);
    return sizeof(float) * (size_t)H * ((2 * NS + B) * dv * dk + NS * bwd_rec_floats(dk, dv) + 2 * NS * kC * dv);
}

void dplr_bwd_carve(DplrParams &p, float *ws) {
    const size_t NS = seq::chunk_slots<kC>(p.B, p.T, p.cu_seqlens != nullptr), H = p.H;
    const size_t st = (size_t)p.dv * p.dk;
    p.ws_S = ws;                                     // [H][NS + B state slots][dv][dk]
    p.ws_dS = p.ws_S + H * (NS + p.B) * st;          // [H][NS][dv][dk]
    p.ws_prep = p.ws_dS + H * NS * st;               // [H][NS] records
    p.ws_x = p.ws_prep + H * NS * bwd_rec_floats(p.dk, p.dv);
    p.ws_dc = p.ws_x + H * NS * kC * p.dv;           // [H][NS][C][dv] each
}

cudaError_t launch_dplr_bwd_simt(const DplrParams &p, int in_bf16, int g_is_bf16, cudaStream_t s) {
    if (in_bf16)
        return g_is_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(p, s) : launch_typed<__nv_bfloat16, float>(p, s);
    return g_is_bf16 ? launch_typed<float, __nv_bfloat16>(p, s) : launch_typed<float, float>(p, s);
}

}  // namespace kda
