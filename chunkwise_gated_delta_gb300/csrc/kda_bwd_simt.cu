// Backward of the chunkwise gated delta rule (KDA and its special cases),
// float32 arithmetic on CUDA cores, chunk length C = 32.
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
// combination carries.)  Three kernels:
//   A  forward scan per (value slice, head, batch): the state before every
//      chunk and the final state, into the workspace;
//   B  reverse scan per (value slice, head, batch): dS after every chunk into
//      the workspace, and dh0;
//   C  one CTA per (chunk, head, batch): every other gradient of the chunk,
//      from the stored S_prev, S_next and dS.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kC = 32;       // chunk length
constexpr int kSC = kC + 1;  // padded row stride of [C][C] tiles
constexpr int kDVS = 32;     // value rows per CTA in the scans
constexpr int kThreads = 256;

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

// Gamma, Q<-, K<-, K-> of one chunk (rows past nvalid are zero, Gamma held at
// its last value), one key channel per thread; gam[d] = gamma^C.
template <int DK, typename Tin, typename Tg>
__device__ void load_rescaled(const BwdParams &p, int b, int h, int t0, int nvalid, float *Gm, float *Ql,
                              float *Kl, float *Kr, float *gam) {
    constexpr int SK = DK + 1;
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tg *g = static_cast<const Tg *>(p.g);
    const int tid = threadIdx.x;
    if (tid < DK) {
        const int d = tid;
        float G = 0.f, gm = 1.f;
        for (int c = 0; c < kC; ++c) {
            float qv = 0.f, kv = 0.f;
            if (c < nvalid) {
                const size_t row = ((size_t)b * p.T + t0 + c) * p.H + h;
                if (Ql) qv = ld(q, row * DK + d);
                kv = ld(k, row * DK + d);
                if (p.gate_kind == KDA_GATE_CHANNEL) G += ld(g, row * DK + d);
                else if (p.gate_kind == KDA_GATE_SCALAR) G += ld(g, row);
                gm = expf(G);
            }
            if (Gm) Gm[c * SK + d] = gm;
            if (Ql) Ql[c * SK + d] = qv * gm;
            Kl[c * SK + d] = kv * gm;
            Kr[c * SK + d] = kv / gm;
        }
        gam[d] = gm;
    }
}

template <typename Tin>
__device__ void load_beta(const BwdParams &p, int b, int h, int t0, int nvalid, float *beta) {
    const Tin *bp = static_cast<const Tin *>(p.beta);
    const int tid = threadIdx.x;
    if (tid < kC) beta[tid] = (p.has_beta && tid < nvalid) ? ld(bp, ((size_t)b * p.T + t0 + tid) * p.H + h) : 0.f;
}

// A~ = (I + Diag(beta) N)^{-1} with N = K<- K->^T * M_{-1}: N into Nm (strict
// lower part, zero elsewhere), then the inverse by forward substitution, one
// column per thread of the first warp.  Ends with a barrier.
template <int DK>
__device__ void wy_inverse(const float *Kl, const float *Kr, const float *beta, float *Nm, float *Am) {
    constexpr int SK = DK + 1;
    const int tid = threadIdx.x;
    for (int idx = tid; idx < kC * kC; idx += kThreads) {
        const int i = idx / kC, j = idx % kC;
        float acc = 0.f;
        if (j < i)
            for (int d = 0; d < DK; ++d) acc += Kl[i * SK + d] * Kr[j * SK + d];
        Nm[i * kSC + j] = acc;
    }
    __syncthreads();
    if (tid < kC) {
        const int c = tid;
        for (int i = 0; i < kC; ++i) {
            float y = 0.f;
            if (i == c) y = 1.f;
            else if (i > c)
                for (int j = c; j < i; ++j) y -= beta[i] * Nm[i * kSC + j] * Am[j * kSC + c];
            Am[i * kSC + c] = y;
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------------ kernel A
template <int DK, typename Tin, typename Tg>
__global__ void __launch_bounds__(kThreads) kda_bwd_states_kernel(const BwdParams p) {
    constexpr int SK = DK + 1, SV = kDVS + 1;
    extern __shared__ float smem[];
    float *Kl = smem;                  // [C][SK]
    float *Kr = Kl + kC * SK;          // [C][SK]
    float *Wm = Kr + kC * SK;          // [C][SK]
    float *Sm = Wm + kC * SK;          // [DVS][SK]
    float *Nm = Sm + kDVS * SK;        // [C][SC]
    float *Am = Nm + kC * kSC;         // [C][SC]
    float *Vm = Am + kC * kSC;         // [C][SV]  v slice, then U, then V_new
    float *gam = Vm + kC * SV;         // [DK]
    float *beta = gam + DK;            // [C]

    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * kDVS, h = blockIdx.y, b = blockIdx.z;
    const int T = p.T, H = p.H, dv = p.dv, N = (T + kC - 1) / kC;
    const Tin *v = static_cast<const Tin *>(p.v);
    const size_t head = (size_t)b * H + h;
    float *Sws = p.ws_S + head * (size_t)(N + 1) * dv * DK;

    for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
        const int e = idx / DK, d = idx % DK;
        Sm[e * SK + d] = p.h0 ? p.h0[(head * dv + e0 + e) * DK + d] : 0.f;
    }
    for (int n = 0; n < N; ++n) {
        const int t0 = n * kC, nvalid = min(kC, T - t0);
        __syncthreads();
        for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
            const int e = idx / DK, d = idx % DK;
            Sws[((size_t)n * dv + e0 + e) * DK + d] = Sm[e * SK + d];
        }
        load_rescaled<DK, Tin, Tg>(p, b, h, t0, nvalid, nullptr, nullptr, Kl, Kr, gam);
        load_beta<Tin>(p, b, h, t0, nvalid, beta);
        for (int idx = tid; idx < kC * kDVS; idx += kThreads) {
            const int c = idx / kDVS, e = idx % kDVS;
            Vm[c * SV + e] = c < nvalid ? ld(v, (((size_t)b * T + t0 + c) * H + h) * dv + e0 + e) : 0.f;
        }
        __syncthreads();
        wy_inverse<DK>(Kl, Kr, beta, Nm, Am);
        // W = A~ Diag(beta) K<-
        for (int idx = tid; idx < kC * DK; idx += kThreads) {
            const int i = idx / DK, d = idx % DK;
            float acc = 0.f;
            for (int j = 0; j <= i; ++j) acc += Am[i * kSC + j] * beta[j] * Kl[j * SK + d];
            Wm[i * SK + d] = acc;
        }
        // U = A~ Diag(beta) V (or A~ V), column by column in place: row i needs rows j <= i
        if (tid < kDVS) {
            const int e = tid;
            for (int i = kC - 1; i >= 0; --i) {
                float acc = 0.f;
                for (int j = 0; j <= i; ++j) acc += Am[i * kSC + j] * (p.scale_v ? beta[j] : 1.f) * Vm[j * SV + e];
                Vm[i * SV + e] = acc;
            }
        }
        __syncthreads();
        // V_new = U - W S^T
        for (int idx = tid; idx < kC * kDVS; idx += kThreads) {
            const int i = idx / kDVS, e = idx % kDVS;
            float acc = Vm[i * SV + e];
            for (int d = 0; d < DK; ++d) acc -= Wm[i * SK + d] * Sm[e * SK + d];
            Vm[i * SV + e] = acc;
        }
        __syncthreads();
        // S <- (S + V_new^T K->) Diag(gamma^C)
        for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
            const int e = idx / DK, d = idx % DK;
            float acc = Sm[e * SK + d];
            for (int c = 0; c < kC; ++c) acc += Vm[c * SV + e] * Kr[c * SK + d];
            Sm[e * SK + d] = acc * gam[d];
        }
    }
    __syncthreads();
    for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
        const int e = idx / DK, d = idx % DK;
        Sws[((size_t)N * dv + e0 + e) * DK + d] = Sm[e * SK + d];
    }
}

// ------------------------------------------------------------------ kernel B
template <int DK, typename Tin, typename Tg>
__global__ void __launch_bounds__(kThreads) kda_bwd_dstate_kernel(const BwdParams p) {
    constexpr int SK = DK + 1, SV = kDVS + 1;
    extern __shared__ float smem[];
    float *Ql = smem;                  // [C][SK]
    float *Kl = Ql + kC * SK;          // [C][SK]
    float *Kr = Kl + kC * SK;          // [C][SK]
    float *Wm = Kr + kC * SK;          // [C][SK]
    float *dS = Wm + kC * SK;          // [DVS][SK]
    float *Nm = dS + kDVS * SK;        // [C][SC]
    float *Am = Nm + kC * kSC;         // [C][SC]
    float *Pm = Am + kC * kSC;         // [C][SC]
    float *dO = Pm + kC * kSC;         // [C][SV]
    float *dU = dO + kC * SV;          // [C][SV]
    float *gam = dU + kC * SV;         // [DK]
    float *beta = gam + DK;            // [C]

    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * kDVS, h = blockIdx.y, b = blockIdx.z;
    const int T = p.T, H = p.H, dv = p.dv, N = (T + kC - 1) / kC;
    const Tin *dop = static_cast<const Tin *>(p.grad_o);
    const size_t head = (size_t)b * H + h;
    float *dSws = p.ws_dS + head * (size_t)N * dv * DK;

    for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
        const int e = idx / DK, d = idx % DK;
        dS[e * SK + d] = p.grad_ht ? p.grad_ht[(head * dv + e0 + e) * DK + d] : 0.f;
    }
    for (int n = N - 1; n >= 0; --n) {
        const int t0 = n * kC, nvalid = min(kC, T - t0);
        __syncthreads();
        for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
            const int e = idx / DK, d = idx % DK;
            dSws[((size_t)n * dv + e0 + e) * DK + d] = dS[e * SK + d];
        }
        load_rescaled<DK, Tin, Tg>(p, b, h, t0, nvalid, nullptr, Ql, Kl, Kr, gam);
        load_beta<Tin>(p, b, h, t0, nvalid, beta);
        for (int idx = tid; idx < kC * kDVS; idx += kThreads) {
            const int c = idx / kDVS, e = idx % kDVS;
            dO[c * SV + e] = c < nvalid ? ld(dop, (((size_t)b * T + t0 + c) * H + h) * dv + e0 + e) : 0.f;
        }
        __syncthreads();
        // P = Q<- K->^T * M
        for (int idx = tid; idx < kC * kC; idx += kThreads) {
            const int i = idx / kC, j = idx % kC;
            float acc = 0.f;
            if (j <= i)
                for (int d = 0; d < DK; ++d) acc += Ql[i * SK + d] * Kr[j * SK + d];
            Pm[i * kSC + j] = acc;
        }
        wy_inverse<DK>(Kl, Kr, beta, Nm, Am);
        // W = A~ Diag(beta) K<-
        for (int idx = tid; idx < kC * DK; idx += kThreads) {
            const int i = idx / DK, d = idx % DK;
            float acc = 0.f;
            for (int j = 0; j <= i; ++j) acc += Am[i * kSC + j] * beta[j] * Kl[j * SK + d];
            Wm[i * SK + d] = acc;
        }
        // dU = K-> Diag(gamma^C) dS^T + P^T dO
        for (int idx = tid; idx < kC * kDVS; idx += kThreads) {
            const int i = idx / kDVS, e = idx % kDVS;
            float acc = 0.f;
            for (int d = 0; d < DK; ++d) acc += Kr[i * SK + d] * gam[d] * dS[e * SK + d];
            for (int j = i; j < kC; ++j) acc += Pm[j * kSC + i] * dO[j * SV + e];
            dU[i * SV + e] = acc;
        }
        __syncthreads();
        // dS <- dS Diag(gamma^C) + dO^T Q<- - dU^T W
        for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
            const int e = idx / DK, d = idx % DK;
            float acc = dS[e * SK + d] * gam[d];
            for (int c = 0; c < kC; ++c) acc += dO[c * SV + e] * Ql[c * SK + d] - dU[c * SV + e] * Wm[c * SK + d];
            dS[e * SK + d] = acc;
        }
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
    return (size_t)8 * kC * (DK + 1) + (size_t)4 * kC * (DV + 1) + (size_t)5 * kC * kSC + 2 * kC + DK;
}

template <int DK, int DV, typename Tin, typename Tg>
__global__ void __launch_bounds__(kThreads) kda_bwd_grad_kernel(const BwdParams p) {
    constexpr int SK = DK + 1, SV = DV + 1;
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
    float *Am = Nm + kC * kSC;         // [C][SC]  A~
    float *Pm = Am + kC * kSC;         // [C][SC]  P, then dO V_new^T * M
    float *dA = Pm + kC * kSC;         // [C][SC]  dA~, then dX~
    float *Tm = dA + kC * kSC;         // [C][SC]  scratch
    float *beta = Tm + kC * kSC;       // [C]
    float *dbeta = beta + kC;          // [C]
    float *gam = dbeta + kC;           // [DK]

    const int tid = threadIdx.x;
    const int n = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int T = p.T, H = p.H, N = (T + kC - 1) / kC;
    const int t0 = n * kC, nvalid = min(kC, T - t0);
    const Tin *v = static_cast<const Tin *>(p.v);
    const Tin *dop = static_cast<const Tin *>(p.grad_o);
    const size_t head = (size_t)b * H + h;
    const float *Sp = p.ws_S + (head * (N + 1) + n) * (size_t)DV * DK;      // state before the chunk
    const float *Sn = Sp + (size_t)DV * DK;                                 // state after the chunk
    const float *dS = p.ws_dS + (head * N + n) * (size_t)DV * DK;           // gradient of the state after

    load_rescaled<DK, Tin, Tg>(p, b, h, t0, nvalid, Gm, Ql, Kl, Kr, gam);
    load_beta<Tin>(p, b, h, t0, nvalid, beta);
    for (int idx = tid; idx < kC * DV; idx += kThreads) {
        const int c = idx / DV, e = idx % DV;
        const size_t off = (((size_t)b * T + t0 + c) * H + h) * DV + e;
        Vm[c * SV + e] = c < nvalid ? ld(v, off) : 0.f;
        dO[c * SV + e] = c < nvalid ? ld(dop, off) : 0.f;
    }
    __syncthreads();
    // P = Q<- K->^T * M ; N and A~
    for (int idx = tid; idx < kC * kC; idx += kThreads) {
        const int i = idx / kC, j = idx % kC;
        float acc = 0.f;
        if (j <= i)
            for (int d = 0; d < DK; ++d) acc += Ql[i * SK + d] * Kr[j * SK + d];
        Pm[i * kSC + j] = acc;
    }
    wy_inverse<DK>(Kl, Kr, beta, Nm, Am);
    const float vscale = p.scale_v ? 1.f : 0.f;   // beta scales v: U = A~ Diag(beta) V, else A~ V
    // W = A~ Diag(beta) K<- ; U = A~ Diag(beta) V
    for (int idx = tid; idx < kC * DK; idx += kThreads) {
        const int i = idx / DK, d = idx % DK;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc += Am[i * kSC + j] * beta[j] * Kl[j * SK + d];
        Wm[i * SK + d] = acc;
    }
    for (int idx = tid; idx < kC * DV; idx += kThreads) {
        const int i = idx / DV, e = idx % DV;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc += Am[i * kSC + j] * (vscale != 0.f ? beta[j] : 1.f) * Vm[j * SV + e];
        Vn[i * SV + e] = acc;
    }
    __syncthreads();
    // V_new = U - W S_prev^T ; dU = K-> Diag(gamma^C) dS^T + P^T dO
    for (int idx = tid; idx < kC * DV; idx += kThreads) {
        const int i = idx / DV, e = idx % DV;
        float acc = Vn[i * SV + e], au = 0.f;
        for (int d = 0; d < DK; ++d) {
            acc -= Wm[i * SK + d] * Sp[(size_t)e * DK + d];
            au += Kr[i * SK + d] * gam[d] * dS[(size_t)e * DK + d];
        }
        for (int j = i; j < kC; ++j) au += Pm[j * kSC + i] * dO[j * SV + e];
        Vn[i * SV + e] = acc;
        dU[i * SV + e] = au;
    }
    __syncthreads();
    // dO V_new^T * M (into Pm)
    for (int idx = tid; idx < kC * kC; idx += kThreads) {
        const int i = idx / kC, j = idx % kC;
        float acc = 0.f;
        if (j <= i)
            for (int e = 0; e < DV; ++e) acc += dO[i * SV + e] * Vn[j * SV + e];
        Pm[i * kSC + j] = acc;
    }
    __syncthreads();
    // dW = -dU S_prev ; dQ<- = dO S_prev + (dO V_new^T * M) K-> ;
    // dK-> = V_new dS Diag(gamma^C) + (dO V_new^T * M)^T Q<-
    for (int idx = tid; idx < kC * DK; idx += kThreads) {
        const int i = idx / DK, d = idx % DK;
        float aw = 0.f, aq = 0.f, ak = 0.f;
        for (int e = 0; e < DV; ++e) {
            const float sp = Sp[(size_t)e * DK + d], ds = dS[(size_t)e * DK + d];
            aw -= dU[i * SV + e] * sp;
            aq += dO[i * SV + e] * sp;
            ak += Vn[i * SV + e] * ds;
        }
        ak *= gam[d];
        for (int j = 0; j <= i; ++j) aq += Pm[i * kSC + j] * Kr[j * SK + d];
        for (int j = i; j < kC; ++j) ak += Pm[j * kSC + i] * Ql[j * SK + d];
        Wm[i * SK + d] = aw;
        dQl[i * SK + d] = aq;
        dKr[i * SK + d] = ak;
    }
    __syncthreads();
    // A~^T dW (into dKl) and A~^T dU (into Vn)
    for (int idx = tid; idx < kC * DK; idx += kThreads) {
        const int i = idx / DK, d = idx % DK;
        float acc = 0.f;
        for (int j = i; j < kC; ++j) acc += Am[j * kSC + i] * Wm[j * SK + d];
        dKl[i * SK + d] = acc;
    }
    for (int idx = tid; idx < kC * DV; idx += kThreads) {
        const int i = idx / DV, e = idx % DV;
        float acc = 0.f;
        for (int j = i; j < kC; ++j) acc += Am[j * kSC + i] * dU[j * SV + e];
        Vn[i * SV + e] = acc;
    }
    // dA~ = dW K<-^T Diag(beta) + dU V^T Diag(beta)  (dU V^T unscaled when beta does not scale v)
    for (int idx = tid; idx < kC * kC; idx += kThreads) {
        const int i = idx / kC, j = idx % kC;
        float aw = 0.f, au = 0.f;
        for (int d = 0; d < DK; ++d) aw += Wm[i * SK + d] * Kl[j * SK + d];
        for (int e = 0; e < DV; ++e) au += dU[i * SV + e] * Vm[j * SV + e];
        dA[i * kSC + j] = aw * beta[j] + au * (vscale != 0.f ? beta[j] : 1.f);
    }
    __syncthreads();
    // dbeta, first two terms: diag(A~^T dW K<-^T) + diag(A~^T dU V^T)
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int i = warp; i < kC; i += kThreads / 32) {
            float acc = 0.f;
            for (int d = lane; d < DK; d += 32) acc += dKl[i * SK + d] * Kl[i * SK + d];
            if (vscale != 0.f)
                for (int e = lane; e < DV; e += 32) acc += Vn[i * SV + e] * Vm[i * SV + e];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) dbeta[i] = acc;
        }
    }
    // dX~ = -A~^T dA~ A~^T: Tm = dA~ A~^T, then dA = -A~^T Tm
    for (int idx = tid; idx < kC * kC; idx += kThreads) {
        const int i = idx / kC, j = idx % kC;
        float acc = 0.f;
        for (int l = 0; l <= j; ++l) acc += dA[i * kSC + l] * Am[j * kSC + l];
        Tm[i * kSC + j] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < kC * kC; idx += kThreads) {
        const int i = idx / kC, j = idx % kC;
        float acc = 0.f;
        for (int l = i; l < kC; ++l) acc -= Am[l * kSC + i] * Tm[l * kSC + j];
        dA[i * kSC + j] = acc;
    }
    __syncthreads();
    // dbeta third term diag(dX~ N^T); E = (Diag(beta) dX~) * M_{-1} into Tm
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int i = warp; i < kC; i += kThreads / 32) {
            float acc = dA[i * kSC + lane] * Nm[i * kSC + lane];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) dbeta[i] += acc;
        }
    }
    for (int idx = tid; idx < kC * kC; idx += kThreads) {
        const int i = idx / kC, j = idx % kC;
        Tm[i * kSC + j] = j < i ? beta[i] * dA[i * kSC + j] : 0.f;
    }
    __syncthreads();
    // dK<- = Diag(beta) A~^T dW + E K-> ; dK-> += E^T K<-
    for (int idx = tid; idx < kC * DK; idx += kThreads) {
        const int i = idx / DK, d = idx % DK;
        float al = beta[i] * dKl[i * SK + d], ar = dKr[i * SK + d];
        for (int j = 0; j < i; ++j) al += Tm[i * kSC + j] * Kr[j * SK + d];
        for (int j = i + 1; j < kC; ++j) ar += Tm[j * kSC + i] * Kl[j * SK + d];
        dKl[i * SK + d] = al;
        dKr[i * SK + d] = ar;
    }
    __syncthreads();
    // outputs: dq, dk, dv, dbeta, and dg from the suffix sums of dlogGamma
    Tin *gq = static_cast<Tin *>(p.grad_q);
    Tin *gk = static_cast<Tin *>(p.grad_k);
    Tin *gv = static_cast<Tin *>(p.grad_v);
    for (int idx = tid; idx < kC * DK; idx += kThreads) {
        const int i = idx / DK, d = idx % DK;
        if (i < nvalid) {
            const size_t off = (((size_t)b * T + t0 + i) * H + h) * DK + d;
            const float gm = Gm[i * SK + d];
            st(gq, off, dQl[i * SK + d] * gm);
            st(gk, off, dKl[i * SK + d] * gm + dKr[i * SK + d] / gm);
        }
    }
    for (int idx = tid; idx < kC * DV; idx += kThreads) {
        const int i = idx / DV, e = idx % DV;
        if (i < nvalid)
            st(gv, (((size_t)b * T + t0 + i) * H + h) * DV + e, (vscale != 0.f ? beta[i] : 1.f) * Vn[i * SV + e]);
    }
    if (p.has_beta && tid < nvalid)
        st(static_cast<Tin *>(p.grad_beta), ((size_t)b * T + t0 + tid) * H + h, dbeta[tid]);
    if (p.gate_kind != KDA_GATE_NONE) {
        // diag(S_next^T dS) for the gamma^C row, then suffix sums down each channel
        Tg *gg = static_cast<Tg *>(p.grad_g);
        float *acc_last = Tm;          // DK floats (Tm is free now)
        for (int d = tid; d < DK; d += kThreads) {
            float acc = 0.f;
            for (int e = 0; e < DV; ++e) acc += Sn[(size_t)e * DK + d] * dS[(size_t)e * DK + d];
            acc_last[d] = acc;
        }
        __syncthreads();
        if (p.gate_kind == KDA_GATE_CHANNEL) {
            for (int d = tid; d < DK; d += kThreads) {
                float run = acc_last[d];
                for (int i = kC - 1; i >= 0; --i) {
                    run += dQl[i * SK + d] * Ql[i * SK + d] + dKl[i * SK + d] * Kl[i * SK + d] -
                           dKr[i * SK + d] * Kr[i * SK + d];
                    if (i < nvalid) st(gg, (((size_t)b * T + t0 + i) * H + h) * DK + d, run);
                }
            }
        } else {
            // scalar gate: the channel sum of the per-channel gradient
            const int warp = tid >> 5, lane = tid & 31;
            float *rowsum = dbeta;     // reuse: C floats (dbeta was already written out)
            __syncthreads();
            for (int i = warp; i < kC; i += kThreads / 32) {
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
                    if (i < nvalid) st(gg, ((size_t)b * T + t0 + i) * H + h, run);
                }
            }
        }
    }
}

template <int DK>
constexpr size_t states_smem_bytes() {
    return sizeof(float) * ((size_t)3 * kC * (DK + 1) + kDVS * (DK + 1) + 2 * kC * kSC + kC * (kDVS + 1) + DK + kC);
}
template <int DK>
constexpr size_t dstate_smem_bytes() {
    return sizeof(float) *
           ((size_t)4 * kC * (DK + 1) + kDVS * (DK + 1) + 3 * kC * kSC + 2 * kC * (kDVS + 1) + DK + kC);
}

template <typename F>
cudaError_t set_smem(F *fn, size_t bytes) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int DK, int DV, typename Tin, typename Tg>
cudaError_t launch_all(const BwdParams &p, cudaStream_t s) {
    const int N = (p.T + kC - 1) / kC;
    cudaError_t e;
    const size_t sa = states_smem_bytes<DK>(), sb = dstate_smem_bytes<DK>();
    const size_t sc = sizeof(float) * grad_smem_floats<DK, DV>();
    static_assert(sizeof(float) * grad_smem_floats<128, 128>() <= 227 * 1024, "kernel C shared memory");
    if ((e = set_smem(kda_bwd_states_kernel<DK, Tin, Tg>, sa)) != cudaSuccess) return e;
    if ((e = set_smem(kda_bwd_dstate_kernel<DK, Tin, Tg>, sb)) != cudaSuccess) return e;
    if ((e = set_smem(kda_bwd_grad_kernel<DK, DV, Tin, Tg>, sc)) != cudaSuccess) return e;
    const dim3 gscan(p.dv / kDVS, p.H, p.B), ggrad(N, p.H, p.B);
    kda_bwd_states_kernel<DK, Tin, Tg><<<gscan, kThreads, sa, s>>>(p);
    kda_bwd_dstate_kernel<DK, Tin, Tg><<<gscan, kThreads, sb, s>>>(p);
    kda_bwd_grad_kernel<DK, DV, Tin, Tg><<<ggrad, kThreads, sc, s>>>(p);
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

size_t bwd_state_bytes(int B, int T, int H, int dk, int dv) {
    const size_t N = (T + kC - 1) / kC;
    return sizeof(float) * (size_t)B * H * (2 * N + 1) * dv * dk;
}

cudaError_t launch_bwd_simt(const BwdParams &p, int in_bf16, int g_is_bf16, cudaStream_t s) {
    if (in_bf16)
        return g_is_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(p, s) : launch_typed<__nv_bfloat16, float>(p, s);
    return g_is_bf16 ? launch_typed<float, __nv_bfloat16>(p, s) : launch_typed<float, float>(p, s);
}

}  // namespace kda
