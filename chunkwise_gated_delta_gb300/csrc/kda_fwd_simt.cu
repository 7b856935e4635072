// float32 CUDA-core kernel for the chunkwise gated delta rule.
//
// Computes the chunk form recapped on page "Kimi Delta Attention backward"
// ("forward recap") in float32 throughout, one CTA per (value slice, head,
// batch).  It serves float32 inputs, whose tolerance (1e-5 relative) no
// tensor-core precision below fp32 meets.  Per chunk [t], with
// G = in-chunk cumsum of g:
//
//   L = Diag(beta)(K<- K->^T * M_{-1}),  P = Q<- K->^T * M,  whose entries
//       sum_d k_id k_jd exp(G_id - G_jd) and q_id k_jd exp(G_id - G_jd)
//       (i >= j) are formed in the log domain, as page "Gated Linear
//       Attention", section 5.3 does for strong decay: no factor exceeds 1,
//       where K-> = K / Gamma alone would overflow once G < -88;
//   A~ = (I + L)^{-1} by forward substitution, one column per thread (page
//       "DeltaNet", section 4.2 gives the unit-lower-triangular inverse);
//   V_new = U - W S^T = A~ (Diag(beta) V - Diag(beta) (K<- S^T))  (or A~ V -
//       A~ Diag(beta) (K<- S^T) when beta does not scale v), K<- = K exp(G);
//   O = Q<- S^T + P V_new,  Q<- = Q exp(G);
//   S <- S Diag(gamma^C) + V_new^T (K exp(G_C - G))  (page "Gated Linear
//       Attention", section 5.2 writes the state step in this factored form).
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kC = 64;      // chunk length
constexpr int kDVS = 32;    // value channels per CTA
constexpr int kThreads = 256;

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <int DK, typename Tg>
__global__ void __launch_bounds__(kThreads)
fwd_simt_kernel(const FwdParams p) {
    constexpr int SK = DK + 1;     // padded row stride of [C][DK] tiles
    constexpr int SC = kC + 1;     // padded row stride of [C][C] tiles
    constexpr int SV = kDVS + 1;
    extern __shared__ float smem[];
    float *Qm = smem;                 // [C][SK]  raw q
    float *Km = Qm + kC * SK;         // [C][SK]  raw k
    float *Gm = Km + kC * SK;         // [C][SK]  G (in-chunk cumsum of g)
    float *Lm = Gm + kC * SK;         // [C][SC]  strictly lower Gram, beta rows
    float *Pm = Lm + kC * SC;         // [C][SC]  inclusive-lower Q<- K->^T
    float *Ym = Pm + kC * SC;         // [C][SC]  A~ = (I + L)^{-1}
    float *Vm = Ym + kC * SC;         // [C][SV]  raw v slice
    float *Um = Vm + kC * SV;         // [C][SV]  V_new
    float *KS = Um + kC * SV;         // [C][SV]  K<- S^T
    float *Sm = KS + kC * SV;         // [DVS][SK] state slice
    float *bet = Sm + kDVS * SK;      // [C]
    float *gC = bet + kC;             // [DK] gamma^C
    float *GC = gC + DK;              // [DK] log gamma^C

    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * kDVS;
    const int h = blockIdx.y, b = blockIdx.z;
    const int T = p.T, H = p.H, dv = p.dv;
    // rows of this sequence: dense batches (b, 0, T); packed sequences (0, cu[b], cu[b+1] - cu[b])
    int rb = b, tb = 0, len = T;
    if (p.cu_seqlens) {
        const int lo = min(max(p.cu_seqlens[b], 0), T);
        const int hi = min(max(p.cu_seqlens[b + 1], lo), T);
        rb = 0; tb = lo; len = hi - lo;
    }
    const float *q = static_cast<const float *>(p.q);
    const float *k = static_cast<const float *>(p.k);
    const float *v = static_cast<const float *>(p.v);
    const Tg *g = static_cast<const Tg *>(p.g);
    const float *beta = static_cast<const float *>(p.beta);
    float *o = static_cast<float *>(p.o);

    for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
        int e = idx / DK, d = idx % DK;
        float s0 = 0.f;
        if (p.h0) s0 = p.h0[(((size_t)b * H + h) * dv + e0 + e) * DK + d];
        Sm[e * SK + d] = s0;
    }

    for (int t0 = 0; t0 < len; t0 += kC) {
        const int nvalid = min(kC, len - t0);
        __syncthreads();
        // ---- prologue: raw q, k and G, one key channel per thread (G held past nvalid)
        if (tid < DK) {
            const int d = tid;
            float G = 0.f;
            for (int c = 0; c < kC; ++c) {
                float qv = 0.f, kv = 0.f;
                if (c < nvalid) {
                    size_t row = ((size_t)rb * T + tb + t0 + c) * H + h;
                    qv = q[row * DK + d];
                    kv = k[row * DK + d];
                    if (p.gate_kind == KDA_GATE_CHANNEL) G += to_f(g[row * DK + d]);
                    else if (p.gate_kind == KDA_GATE_SCALAR) G += to_f(g[row]);
                }
                Qm[c * SK + d] = qv;
                Km[c * SK + d] = kv;
                Gm[c * SK + d] = G;
            }
            gC[d] = expf(G);
            GC[d] = G;
        }
        for (int idx = tid; idx < kC * kDVS; idx += kThreads) {
            int c = idx / kDVS, e = idx % kDVS;
            float vv = 0.f;
            if (c < nvalid) vv = v[(((size_t)rb * T + tb + t0 + c) * H + h) * dv + e0 + e];
            Vm[c * SV + e] = vv;
        }
        if (tid < kC) {
            float bv = 0.f;
            if (p.has_beta && tid < nvalid) bv = beta[((size_t)rb * T + tb + t0 + tid) * H + h];
            bet[tid] = bv;
        }
        __syncthreads();
        // ---- Gram matrices in the log domain; K<- S^T
        for (int idx = tid; idx < kC * kC; idx += kThreads) {
            int i = idx / kC, j = idx % kC;
            float l = 0.f, pp = 0.f;
            if (j <= i) {
                for (int d = 0; d < DK; ++d) {
                    const float f = expf(Gm[i * SK + d] - Gm[j * SK + d]) * Km[j * SK + d];
                    l += Km[i * SK + d] * f;
                    pp += Qm[i * SK + d] * f;
                }
            }
            Lm[i * SC + j] = (j < i) ? bet[i] * l : 0.f;
            Pm[i * SC + j] = pp;
        }
        for (int idx = tid; idx < kC * kDVS; idx += kThreads) {
            int i = idx / kDVS, e = idx % kDVS;
            float acc = 0.f;
            for (int d = 0; d < DK; ++d) acc += Km[i * SK + d] * expf(Gm[i * SK + d]) * Sm[e * SK + d];
            KS[i * SV + e] = acc;
        }
        __syncthreads();
        // ---- A~ = (I + L)^{-1}: column c solved by forward substitution
        if (tid < kC) {
            const int c = tid;
            for (int i = 0; i < kC; ++i) {
                float y = 0.f;
                if (i == c) y = 1.f;
                else if (i > c) {
                    for (int j = c; j < i; ++j) y -= Lm[i * SC + j] * Ym[j * SC + c];
                }
                Ym[i * SC + c] = y;
            }
        }
        __syncthreads();
        // ---- V_new = A~ (Diag(beta) V - Diag(beta) K<- S^T)  (Diag(beta) V -> V when beta does not scale v)
        for (int idx = tid; idx < kC * kDVS; idx += kThreads) {
            int i = idx / kDVS, e = idx % kDVS;
            float acc = 0.f;
            for (int j = 0; j <= i; ++j)
                acc += Ym[i * SC + j] * ((p.scale_v ? bet[j] : 1.f) * Vm[j * SV + e] - bet[j] * KS[j * SV + e]);
            Um[i * SV + e] = acc;
        }
        __syncthreads();
        // ---- O = Q<- S^T + P V_new
        for (int idx = tid; idx < kC * kDVS; idx += kThreads) {
            int i = idx / kDVS, e = idx % kDVS;
            float acc = 0.f;
            for (int d = 0; d < DK; ++d) acc += Qm[i * SK + d] * expf(Gm[i * SK + d]) * Sm[e * SK + d];
            for (int j = 0; j <= i; ++j) acc += Pm[i * SC + j] * Um[j * SV + e];
            if (i < nvalid) o[(((size_t)rb * T + tb + t0 + i) * H + h) * dv + e0 + e] = acc;
        }
        __syncthreads();
        // ---- S <- S Diag(gamma^C) + V_new^T (K exp(G_C - G))
        for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
            int e = idx / DK, d = idx % DK;
            float acc = 0.f;
            for (int c = 0; c < kC; ++c) acc += Um[c * SV + e] * Km[c * SK + d] * expf(GC[d] - Gm[c * SK + d]);
            Sm[e * SK + d] = Sm[e * SK + d] * gC[d] + acc;
        }
    }
    __syncthreads();
    if (p.ht) {
        for (int idx = tid; idx < kDVS * DK; idx += kThreads) {
            int e = idx / DK, d = idx % DK;
            p.ht[(((size_t)b * H + h) * dv + e0 + e) * DK + d] = Sm[e * SK + d];
        }
    }
}

template <int DK>
constexpr size_t simt_smem_bytes() {
    return sizeof(float) * (size_t)(3 * kC * (DK + 1) + 3 * kC * (kC + 1) + 3 * kC * (kDVS + 1) +
                                    kDVS * (DK + 1) + kC + 2 * DK);
}

template <int DK, typename Tg>
cudaError_t launch_dk(const FwdParams &p, cudaStream_t s) {
    const size_t smem = simt_smem_bytes<DK>();
    cudaError_t e = cudaFuncSetAttribute(fwd_simt_kernel<DK, Tg>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.dv / kDVS, p.H, p.B);
    fwd_simt_kernel<DK, Tg><<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt_f32(const FwdParams &p, int g_is_bf16, cudaStream_t s) {
    if (p.dk == 64) return g_is_bf16 ? launch_dk<64, __nv_bfloat16>(p, s) : launch_dk<64, float>(p, s);
    if (p.dk == 128) return g_is_bf16 ? launch_dk<128, __nv_bfloat16>(p, s) : launch_dk<128, float>(p, s);
    return cudaErrorNotSupported;
}

}  // namespace kda
