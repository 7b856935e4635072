// Kernels for the general gated DPLR recurrence, float32 accumulation (warp-level
// tf32 tensor-core products for bf16 inputs, exact float32 products for fp32)
//
//     S_t = S_{t-1} Diag(alpha_t) (I - b_t a_t^T) + v_t k_t^T,   o_t = S_t q_t
//
// (page "Diagonal Plus Low Rank", section 2), evaluated in the chunk form
// that page derives.  Per chunk [t] (length C = 32, so every tile of a
// (value slice, head, batch) fits in shared memory; the chunk length does not
// change the result):
//
//   Gamma = exp(in-chunk cumsum g);  Q<- = Q*Gamma, K-> = K/Gamma,
//   A-> = A/Gamma, B<- = B*Gamma;
//   E = (I + (B<- A->^T * M_{-1}))^{-1};   W = E B<-;
//   C = -E (B<- K->^T * M_{-1}) V;          X = C - W S^T;
//   O = Q<- S^T + (Q<- K->^T * M) V + (Q<- A->^T * M) X;
//   S <- (S + V^T K-> + X^T A->) Diag(gamma^C).
//
// Two kernels: a chunk-parallel prep kernel writes, per chunk, everything that
// does not depend on the state (W, Q<- - P_a W, K-> and A-> times gamma^C, C
// and the chunk-local output P_k V + P_a C) into the workspace; the scan then
// needs three products per chunk.
//
// Also the per-token transition norms of page "How to make GDN2 more stable":
// eq. (4) for I - b a^T, and the largest singular value of the full factor
// Diag(alpha)(I - b a^T), for which the page has no closed form, by
// bisection on inertia counts of its Gram matrix.
#include <cuda_bf16.h>

#include "dplr_common.cuh"
#include "kda_internal.h"
#include "packed_seq.cuh"
#include "warp_gemm.cuh"

namespace kda {
namespace {

constexpr int kC = 32;      // chunk length
constexpr int kDVS = 32;    // value channels per CTA
constexpr int kThreads = 256;

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Row strides = 4 (mod 32) for the fragment reads of the warp-tiled products.
__host__ __device__ constexpr int pad4(int n) { return n + 4; }

// ------------------------------------------------------------------ chunk records
// Everything of a chunk that does not depend on the state (float32), written
// once by the prep kernel: W = E B<-, Qt = Q<- - P_a W, K~ = K-> Diag(gamma^C),
// A~ = A-> Diag(gamma^C), C = -E (B<- K->^T * M_{-1}) V, the chunk-local output
// O_loc = P_k V + P_a C, and gamma^C; so that per chunk
//   X = C - W S^T,  O = Qt S^T + O_loc,  S <- S Diag(gamma^C) + V^T K~ + X^T A~.
__host__ __device__ constexpr size_t dplr_rec_floats(int dk, int dv) {
    return (size_t)4 * kC * dk + (size_t)2 * kC * dv + dk;
}
template <int DK, int DV>
struct DRec {
    static constexpr int W = 0, QT = kC * DK, KG = 2 * kC * DK, AG = 3 * kC * DK, CC = 4 * kC * DK,
                         OL = CC + kC * DV, GC = OL + kC * DV;
    static_assert(dplr_rec_floats(DK, DV) == (size_t)GC + DK && dplr_rec_floats(DK, DV) % 4 == 0, "record");
};

template <int DK>
__host__ __device__ constexpr bool prep_aliases() { return 3 * kC * pad4(kC) <= kC * pad4(DK); }

// One CTA per (chunk, head, sequence).  Products run as warp-tiled 32 x N blocks
// (warp_gemm.cuh): tf32 tensor-core MMAs for bf16 inputs (TF32), exact float32
// for float32 inputs.
template <int DK, int DV, typename Tin, typename Tg, bool TF32>
__global__ void __launch_bounds__(kThreads)
dplr_fwd_prep_kernel(const DplrParams p) {
    constexpr int SK = pad4(DK), SC = pad4(kC), SV = pad4(DV);
    using R = DRec<DK, DV>;
    extern __shared__ float smem[];
    // Where three C x C tiles fit a key-wide tile (dk = 128), tiles that die early hand their
    // space on, so two CTAs fit an SM for dv <= 128: Gamma's tile holds three Gram tiles once
    // the rescaled tiles exist, and K->'s holds E, the inverse's scratch and M1 once the K~
    // and A~ records are written.
    constexpr bool kAlias = prep_aliases<DK>();
    float4 *rows = reinterpret_cast<float4 *>(smem);   // [C] eq. (4) data per row (clip)
    float *Gm = smem + 4 * kC;        // [C][SK]  raw gate, then Gamma
    float *Ql = Gm + kC * SK;         // [C][SK]
    float *Kr = Ql + kC * SK;         // [C][SK]
    float *Ar = Kr + kC * SK;         // [C][SK]
    float *Bl = Ar + kC * SK;         // [C][SK]
    float *Vm = Bl + kC * SK;         // [C][SV]
    float *Pa = Vm + kC * SV;         // [C][SC]  Q<- A->^T * M
    float *gam = Pa + kC * SC;        // [DK]
    float *gsc = gam + DK;            // [C]
    float *extra = gsc + kC;          // 6 x [C][SC] when the tiles do not alias
    float *Lab = kAlias ? Gm : extra; // [C][SC]  B<- A->^T * M_{-1}   (Gamma's tile, after the rescaling)
    float *Lbk = Lab + kC * SC;       // [C][SC]  B<- K->^T * M_{-1}
    float *Pk = Lbk + kC * SC;        // [C][SC]  Q<- K->^T * M
    float *Em = kAlias ? Kr : Pk + kC * SC;   // [C][SC]  E           (K->'s tile, after the records)
    float *Ts = Em + kC * SC;         // [C][SC]  scratch of the inverse, then P_a E
    float *M1 = Ts + kC * SC;         // [C][SC]  E (B<- K->^T * M_{-1})

    const int tid = threadIdx.x, h = blockIdx.y;
    int b, n;
    seq::Seq sq;
    if (!seq::chunk_of<kC>(p, b, n, sq)) return;
    const int H = p.H;
    const int t0 = n * kC, nvalid = min(kC, sq.len - t0);
    const size_t row = (size_t)sq.row0 + t0;
    const Tin *v = static_cast<const Tin *>(p.v);
    float *rec = p.ws_prep + seq::chunk_index<kC>(p, sq, h, n) * dplr_rec_floats(DK, DV);

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
        wg::gemm_pair<kC, TF32>(DK, aBl, bAr, DK, aBl, bKr, [&](int i, int j, float x, float y) {
            Lab[i * SC + j] = j < i ? x : 0.f;
            Lbk[i * SC + j] = j < i ? y : 0.f;
        });
        wg::gemm_pair<kC, TF32>(DK, aQl, bKr, DK, aQl, bAr, [&](int i, int j, float x, float y) {
            Pk[i * SC + j] = j <= i ? x : 0.f;
            Pa[i * SC + j] = j <= i ? y : 0.f;
        });
    }
    for (int idx = tid; idx < kC * DK; idx += kThreads) {
        const int i = idx / DK, d = idx % DK;
        rec[R::KG + idx] = Kr[i * SK + d] * gam[d];
        rec[R::AG + idx] = Ar[i * SK + d] * gam[d];
    }
    for (int d = tid; d < DK; d += kThreads) rec[R::GC + d] = gam[d];
    __syncthreads();
    dplr::block_inverse32<SC>(Lab, Em, Ts);
    // M1 = E Lbk ; P_a E (into Ts)
    wg::gemm_pair<kC, TF32>(
        kC, [&](int i, int j) { return Em[i * SC + j]; }, [&](int j, int l) { return Lbk[j * SC + l]; }, kC,
        [&](int i, int j) { return Pa[i * SC + j]; }, [&](int j, int l) { return Em[j * SC + l]; },
        [&](int i, int l, float x, float y) {
            M1[i * SC + l] = x;
            Ts[i * SC + l] = y;
        });
    __syncthreads();
    // P_k - (P_a E) Lbk (into Pk)
    wg::gemm<kC, TF32>(
        kC, [&](int i, int j) { return Ts[i * SC + j]; }, [&](int j, int l) { return Lbk[j * SC + l]; },
        [&](int i, int l, float x) { Pk[i * SC + l] -= x; });
    // W = E B<- ; Qt = Q<- - (P_a E) B<-
    wg::gemm_pair<DK, TF32>(
        kC, [&](int i, int j) { return Em[i * SC + j]; }, [&](int j, int d) { return Bl[j * SK + d]; }, kC,
        [&](int i, int j) { return Ts[i * SC + j]; }, [&](int j, int d) { return Bl[j * SK + d]; },
        [&](int i, int d, float w, float pw) {
            rec[R::W + i * DK + d] = w;
            rec[R::QT + i * DK + d] = Ql[i * SK + d] - pw;
        });
    __syncthreads();
    // C = -M1 V ; O_loc = (P_k - P_a E Lbk) V
    wg::gemm_pair<DV, TF32>(
        kC, [&](int i, int j) { return M1[i * SC + j]; }, [&](int j, int e) { return Vm[j * SV + e]; }, kC,
        [&](int i, int j) { return Pk[i * SC + j]; }, [&](int j, int e) { return Vm[j * SV + e]; },
        [&](int i, int e, float c, float ol) {
            rec[R::CC + i * DV + e] = -c;
            rec[R::OL + i * DV + e] = ol;
        });
}

template <int DK, int DV>
constexpr size_t prep_smem_bytes() {
    return sizeof(float) * (size_t)(4 * kC + 5 * kC * pad4(DK) + kC * pad4(DV) + kC * pad4(kC) + DK + kC +
                                    (prep_aliases<DK>() ? 0 : 6 * kC * pad4(kC)));
}

// One CTA per (32-wide value slice, head, batch): the serial scan over the
// chunk records.  The records (and v) of chunk n + 1 travel by cp.async into a
// second buffer while chunk n computes.
template <int DK, typename Tin>
__host__ __device__ constexpr int scan_buf_floats() {
    // W, Qt, K~, A~ [C][SK]; C and O_loc slices [C][SV]; gamma^C [DK]; raw v rows [C][DVS] of Tin
    return 4 * kC * pad4(DK) + 2 * kC * pad4(kDVS) + DK + (kC * kDVS * (int)sizeof(Tin) + 3) / 4;
}
template <int DK, int DV, typename Tin, bool TF32>
__global__ void __launch_bounds__(kThreads)
dplr_fwd_simt_kernel(const DplrParams p) {
    constexpr int SK = pad4(DK), SV = pad4(kDVS), BUF = scan_buf_floats<DK, Tin>();
    using R = DRec<DK, DV>;
    extern __shared__ float smem[];
    float *Sm = smem;                 // [DVS][SK] state slice
    float *Vm = Sm + kDVS * SK;       // [C][SV]  v slice (float)
    float *Xm = Vm + kC * SV;         // [C][SV]  X
    float *bufs = Xm + kC * SV;       // 2 x BUF

    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * kDVS;
    const int h = blockIdx.y, b = blockIdx.z;
    const int H = p.H, dv = p.dv;
    const seq::Seq sq = seq::seq_of<kC>(p, b);
    const int N = sq.nch, T = sq.len;
    const size_t row0 = sq.row0;
    const Tin *v = static_cast<const Tin *>(p.v);
    Tin *o = static_cast<Tin *>(p.o);
    const float *recs = p.ws_prep + seq::chunk_index<kC>(p, sq, h, 0) * dplr_rec_floats(DK, DV);
    auto issue = [&](int n) {
        const float *rec = recs + (size_t)n * dplr_rec_floats(DK, DV);
        float *bf = bufs + (n & 1) * BUF;
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::W, DK, bf);
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::QT, DK, bf + kC * SK);
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::KG, DK, bf + 2 * kC * SK);
        wg::load_tile_async<kC, DK, SK, kThreads>(rec + R::AG, DK, bf + 3 * kC * SK);
        wg::load_tile_async<kC, kDVS, SV, kThreads>(rec + R::CC + e0, DV, bf + 4 * kC * SK);
        wg::load_tile_async<kC, kDVS, SV, kThreads>(rec + R::OL + e0, DV, bf + 4 * kC * SK + kC * SV);
        wg::load_tile_async<1, DK, DK, kThreads>(rec + R::GC, DK, bf + 4 * kC * SK + 2 * kC * SV);
        wg::load_raw_async<kC, kDVS, Tin, kThreads>(v + ((row0 + n * kC) * H + h) * dv + e0, (size_t)H * dv,
                                                    min(kC, T - n * kC),
                                                    reinterpret_cast<Tin *>(bf + 4 * kC * SK + 2 * kC * SV + DK));
    };

    for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
        const int e = idx / DK, d = idx % DK;
        Sm[e * SK + d] = p.h0 ? p.h0[(((size_t)b * H + h) * dv + e0 + e) * DK + d] : 0.f;
    }
    issue(0);
    wg::cp_async_commit();
    for (int n = 0; n < N; ++n) {
        const int t0 = n * kC, nvalid = min(kC, T - t0);
        float *Wm = bufs + (n & 1) * BUF, *QT = Wm + kC * SK, *KG = QT + kC * SK, *AG = KG + kC * SK;
        float *Cs = AG + kC * SK, *Os = Cs + kC * SV, *gC = Os + kC * SV;
        const Tin *vraw = reinterpret_cast<const Tin *>(gC + DK);
        __syncthreads();                  // chunk n - 1 is done with the other buffer
        if (n + 1 < N) issue(n + 1);
        wg::cp_async_commit();            // (an empty group on the last chunk keeps the count)
        wg::cp_async_wait<1>();           // chunk n's copies (this thread's) have landed
        __syncthreads();
        wg::to_f32<kC, kDVS, SV, Tin, kThreads>(vraw, Vm);
        __syncthreads();
        // X = C - W S^T ; O = Qt S^T + O_loc
        {
            auto bS = [&](int d, int e) { return Sm[e * SK + d]; };
            wg::gemm_pair<kDVS, TF32>(
                DK, [&](int i, int d) { return Wm[i * SK + d]; }, bS, DK, [&](int i, int d) { return QT[i * SK + d]; },
                bS, [&](int i, int e, float ws, float qs) {
                    Xm[i * SV + e] = Cs[i * SV + e] - ws;
                    if (i < nvalid) o[((row0 + t0 + i) * H + h) * dv + e0 + e] = from_f<Tin>(Os[i * SV + e] + qs);
                });
        }
        __syncthreads();
        // S <- S Diag(gamma^C) + V^T K~ + X^T A~
        wg::gemm2<DK, TF32>(
            kC, [&](int e, int c) { return Vm[c * SV + e]; }, [&](int c, int d) { return KG[c * SK + d]; }, kC,
            [&](int e, int c) { return Xm[c * SV + e]; }, [&](int c, int d) { return AG[c * SK + d]; },
            [&](int e, int d, float x) { Sm[e * SK + d] = Sm[e * SK + d] * gC[d] + x; });
    }
    __syncthreads();
    if (p.ht) {
        for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
            const int e = idx / DK, d = idx % DK;
            p.ht[(((size_t)b * H + h) * dv + e0 + e) * DK + d] = Sm[e * SK + d];
        }
    }
}

template <int DK, typename Tin>
constexpr size_t dplr_smem_bytes() {
    return sizeof(float) * (size_t)(kDVS * pad4(DK) + 2 * kC * pad4(kDVS) + 2 * scan_buf_floats<DK, Tin>());
}

template <int DK, int DV, typename Tin, typename Tg>
cudaError_t launch_dkv(const DplrParams &p, cudaStream_t s) {
    constexpr bool kTf32 = sizeof(Tin) == 2;        // bf16 inputs: tf32 tensor-core products
    const size_t sp = prep_smem_bytes<DK, DV>(), sm = dplr_smem_bytes<DK, Tin>();
    static_assert(dplr_smem_bytes<128, float>() <= 227 * 1024, "scan shared memory");
    static_assert(prep_smem_bytes<128, 256>() <= 227 * 1024, "shared memory");
    cudaError_t e = cudaFuncSetAttribute(dplr_fwd_prep_kernel<DK, DV, Tin, Tg, kTf32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dplr_fwd_simt_kernel<DK, DV, Tin, kTf32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm);
    if (e != cudaSuccess) return e;
    dplr_fwd_prep_kernel<DK, DV, Tin, Tg, kTf32>
        <<<seq::chunk_grid<kC>(p.B, p.T, p.H, p.cu_seqlens != nullptr), kThreads, sp, s>>>(p);
    dplr_fwd_simt_kernel<DK, DV, Tin, kTf32><<<dim3(p.dv / kDVS, p.H, p.B), kThreads, sm, s>>>(p);
    return cudaGetLastError();
}

template <int DK, typename Tin, typename Tg>
cudaError_t launch_dk(const DplrParams &p, cudaStream_t s) {
    switch (p.dv) {
    case 32: return launch_dkv<DK, 32, Tin, Tg>(p, s);
    case 64: return launch_dkv<DK, 64, Tin, Tg>(p, s);
    case 96: return launch_dkv<DK, 96, Tin, Tg>(p, s);
    case 128: return launch_dkv<DK, 128, Tin, Tg>(p, s);
    case 160: return launch_dkv<DK, 160, Tin, Tg>(p, s);
    case 192: return launch_dkv<DK, 192, Tin, Tg>(p, s);
    case 224: return launch_dkv<DK, 224, Tin, Tg>(p, s);
    case 256: return launch_dkv<DK, 256, Tin, Tg>(p, s);
    }
    return cudaErrorNotSupported;
}

template <typename Tin, typename Tg>
cudaError_t launch_typed(const DplrParams &p, cudaStream_t s) {
    if (p.dk == 64) return launch_dk<64, Tin, Tg>(p, s);
    if (p.dk == 128) return launch_dk<128, Tin, Tg>(p, s);
    return cudaErrorNotSupported;
}

// ---------------------------------------------------------------- factor norms
// One warp per token; lane l holds channels l, l+32, l+64, l+96 (dk <= 128).
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}

// Largest singular value of M = D - u a^T with D = Diag(alpha), u = D b.
// M^T M = D^2 + P K P^T with P = [a, r], r = D u, K = [[s, -1], [-1, 0]],
// s = u^T u: a diagonal matrix plus a rank-2 term of either sign.  For a
// shift lambda that is no alpha_i^2, Haynsworth's inertia additivity applied
// to [[D^2 - lambda, P], [P^T, -K^{-1}]] counts the eigenvalues of M^T M
// above lambda:
//     #{i : alpha_i^2 > lambda} + pos(N) - pos(-K^{-1}),
//     N = -K^{-1} - P^T (D^2 - lambda)^{-1} P = [[-R11, 1 - R12], [1 - R12, s - R22]],
// with pos(-K^{-1}) = 1 (its determinant is -1).  The count is monotone in
// lambda, so bisection on "count >= 1" over [0, (max alpha + |u||a|)^2]
// brackets the largest eigenvalue (the spectral-bisection method of Sturm
// counts, with the count taken from the inertia of a 2x2 matrix).
template <int R>
__device__ float factor_norm_inertia(const float (&av)[R], const float (&al)[R], const float (&bv)[R]) {
    float r[R], d2[R];
    float dmax = 0.f, su = 0.f, sa = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const float u = al[i] * bv[i];
        r[i] = al[i] * u;
        d2[i] = al[i] * al[i];
        dmax = fmaxf(dmax, al[i]);
        su += u * u;
        sa += av[i] * av[i];
    }
    dmax = warp_max(dmax);
    const float s = warp_sum(su);
    sa = warp_sum(sa);
    const float top = dmax + sqrtf(s * sa);
    float lo = 0.f, hi = top * top * (1.f + 1e-6f) + 1e-30f;
    for (int it = 0; it < 64; ++it) {
        float mid = 0.5f * (lo + hi);
        if (!(mid > lo && mid < hi)) break;
        bool pole = false;
#pragma unroll
        for (int i = 0; i < R; ++i) pole |= d2[i] == mid;
        if (__any_sync(0xffffffffu, pole)) mid = nextafterf(mid, hi);
        float r11 = 0.f, r12 = 0.f, r22 = 0.f, above = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float w = 1.f / (d2[i] - mid);
            r11 += av[i] * av[i] * w;
            r12 += av[i] * r[i] * w;
            r22 += r[i] * r[i] * w;
            above += d2[i] > mid ? 1.f : 0.f;
        }
        r11 = warp_sum(r11);
        r12 = warp_sum(r12);
        r22 = warp_sum(r22);
        above = warp_sum(above);
        const float n11 = -r11, n12 = 1.f - r12, n22 = s - r22;
        const float det = n11 * n22 - n12 * n12, tr = n11 + n22;
        const float pos = det < 0.f ? 1.f : (tr > 0.f ? (det > 0.f ? 2.f : 1.f) : 0.f);
        if (above + pos - 1.f >= 1.f) lo = mid;
        else hi = mid;
    }
    return sqrtf(0.5f * (lo + hi));
}

template <typename Tin, typename Tg>
__global__ void __launch_bounds__(256)
dplr_factor_norm_kernel(const DplrParams p, float *rho, float *nrm, float *maxes) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long ntok = (long)(p.cu_seqlens ? 1 : p.B) * p.T * p.H;   // packed: one [1, T] batch
    if (warp >= ntok) return;
    const int dk = p.dk;
    const Tin *a = static_cast<const Tin *>(p.a);
    const Tin *bb = static_cast<const Tin *>(p.b);
    const Tg *g = static_cast<const Tg *>(p.g);
    float av[4], bv[4], gv[4], al[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int d = lane + 32 * r;
        const bool ok = d < dk;
        av[r] = ok ? to_f(a[(size_t)warp * dk + d]) : 0.f;
        bv[r] = ok ? to_f(bb[(size_t)warp * dk + d]) : 0.f;
        gv[r] = 0.f;
        if (p.gate_kind == KDA_GATE_CHANNEL) gv[r] = ok ? to_f(g[(size_t)warp * dk + d]) : 0.f;
        else if (p.gate_kind == KDA_GATE_SCALAR) gv[r] = to_f(g[warp]);
    }
    // eq. (4): ||I - eta k j^T||_2 for unit k, j with eta = |a||b| and c = cos(a, b)
    const float na2 = warp_sum(av[0] * av[0] + av[1] * av[1] + av[2] * av[2] + av[3] * av[3]);
    const float nb2 = warp_sum(bv[0] * bv[0] + bv[1] * bv[1] + bv[2] * bv[2] + bv[3] * bv[3]);
    const float ab = warp_sum(av[0] * bv[0] + av[1] * bv[1] + av[2] * bv[2] + av[3] * bv[3]);
    const float r4 = dplr::rho_eq4(na2, nb2, ab);
    // decay, clipped to 1/rho by eq. (7) when asked
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const float gc = p.clip ? fminf(gv[r], -logf(r4)) : gv[r];
        al[r] = (lane + 32 * r < dk) ? expf(gc) : 0.f;
    }
    const float sig = factor_norm_inertia(av, al, bv);
    if (lane == 0) {
        if (rho) rho[warp] = r4;
        if (nrm) nrm[warp] = sig;
        if (maxes) {   // non-negative floats order like their bit patterns
            atomicMax(reinterpret_cast<int *>(maxes), __float_as_int(r4));
            atomicMax(reinterpret_cast<int *>(maxes) + 1, __float_as_int(sig));
        }
    }
}

}  // namespace

size_t dplr_fwd_record_bytes(int B, int T, int H, int dk, int dv, bool packed) {
    return sizeof(float) * (size_t)H * seq::chunk_slots<kC>(B, T, packed) * dplr_rec_floats(dk, dv);
}

cudaError_t launch_dplr_fwd_simt(const DplrParams &p, int in_bf16, int g_is_bf16, cudaStream_t s) {
    if (in_bf16)
        return g_is_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(p, s) : launch_typed<__nv_bfloat16, float>(p, s);
    return g_is_bf16 ? launch_typed<float, __nv_bfloat16>(p, s) : launch_typed<float, float>(p, s);
}

cudaError_t launch_dplr_factor_norms(const DplrParams &p, int in_bf16, int g_is_bf16, float *rho, float *nrm,
                                     float *maxes, cudaStream_t s) {
    const long ntok = (long)(p.cu_seqlens ? 1 : p.B) * p.T * p.H;
    const long blocks = (ntok * 32 + 255) / 256;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidValue;
    if (maxes) {
        cudaError_t e = cudaMemsetAsync(maxes, 0, 2 * sizeof(float), s);
        if (e != cudaSuccess) return e;
    }
    if (in_bf16) {
        if (g_is_bf16)
            dplr_factor_norm_kernel<__nv_bfloat16, __nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(p, rho, nrm, maxes);
        else
            dplr_factor_norm_kernel<__nv_bfloat16, float><<<(unsigned)blocks, 256, 0, s>>>(p, rho, nrm, maxes);
    } else {
        if (g_is_bf16)
            dplr_factor_norm_kernel<float, __nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(p, rho, nrm, maxes);
        else
            dplr_factor_norm_kernel<float, float><<<(unsigned)blocks, 256, 0, s>>>(p, rho, nrm, maxes);
    }
    return cudaGetLastError();
}

}  // namespace kda
