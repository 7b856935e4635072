// Device helpers shared by the DPLR forward and backward kernels.
//
// The gated DPLR recurrence S_t = S_{t-1} Diag(alpha_t)(I - b_t a_t^T) + v_t k_t^T
// (page "Diagonal Plus Low Rank", section 2) in its chunk form needs, per
// chunk, Gamma = exp(in-chunk cumsum of the log-decay) and the rescaled tiles
// Q<- = Q * Gamma, K-> = K / Gamma, A-> = A / Gamma, B<- = B * Gamma.
//
// With the clip of page "How to make GDN2 more stable", eq. (7), the decay of
// token t is min(D_t, 1/rho_t), rho_t = ||I - b_t a_t^T||_2 from eq. (4):
// in log space g'_t = min(g_t, -log rho_t), with eta = |a||b| and
// c = a.b / eta, rho = (eta + sqrt(eta^2 - 4 eta c + 4)) / 2.
#pragma once

#include <cuda_bf16.h>

#include "kda_internal.h"
#include "warp_gemm.cuh"

namespace kda {
namespace dplr {

template <typename T> __device__ __forceinline__ float ldf(const T *p, size_t i);
template <> __device__ __forceinline__ float ldf<float>(const float *p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
template <typename T> __device__ __forceinline__ void stf(T *p, size_t i, float x);
template <> __device__ __forceinline__ void stf<float>(float *p, size_t i, float x) { p[i] = x; }
template <> __device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Eq. (4) for one token from |a|^2, |b|^2 and a.b.
__device__ __forceinline__ float rho_eq4(float na2, float nb2, float ab) {
    const float eta = sqrtf(na2 * nb2);
    const float cosv = eta > 0.f ? ab / eta : 1.f;
    return 0.5f * (eta + sqrtf(fmaxf(eta * eta - 4.f * eta * cosv + 4.f, 0.f)));
}

// Per row c < C of the chunk starting at row `row0` of its batch: rows[c] = (|a|^2, |b|^2,
// a.b, -log rho) (zeros past nvalid).  One warp per row; no barrier inside.
template <int DK, int C, typename Tin>
__device__ void row_rho(const DplrParams &p, size_t row0, int h, int nvalid, float4 *rows) {
    const Tin *a = static_cast<const Tin *>(p.a);
    const Tin *bb = static_cast<const Tin *>(p.b);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int c = warp; c < C; c += nwarps) {
        float na2 = 0.f, nb2 = 0.f, ab = 0.f;
        if (c < nvalid) {
            const size_t row = ((row0 + c) * p.H + h) * DK;
            for (int d = lane; d < DK; d += 32) {
                const float av = ldf(a, row + d), bv = ldf(bb, row + d);
                na2 += av * av;
                nb2 += bv * bv;
                ab += av * bv;
            }
        }
        na2 = warp_sum(na2);
        nb2 = warp_sum(nb2);
        ab = warp_sum(ab);
        if (lane == 0) rows[c] = make_float4(na2, nb2, ab, c < nvalid ? -logf(rho_eq4(na2, nb2, ab)) : 0.f);
    }
}




// Gamma and the rescaled tiles of the chunk starting at row `row0` of its batch (rows
// past nvalid zero, Gamma held
// at its last value; gam[d] = gamma^C): all threads load the raw tiles first
// (16-byte vector loads, 256 threads), then one thread per key channel runs the
// (optionally clipped) cumsum down its column in shared memory.  Gm is required
// (it holds the raw gate in between); Ql, Kr, Ar, Bl may be null; gsc holds C
// floats (scalar gates); `rows` comes from row_rho when p.clip is set (a
// barrier must separate the two).  Contains one barrier; the caller
// synchronises before reading the tiles.
template <int DK, int SK, int C, typename Tin, typename Tg>
__device__ void load_rescaled_par(const DplrParams &p, size_t row0, int h, int nvalid, const float4 *rows,
                                  float *Gm, float *Ql, float *Kr, float *Ar, float *Bl, float *gam, float *gsc) {
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *a = static_cast<const Tin *>(p.a);
    const Tin *bb = static_cast<const Tin *>(p.b);
    const Tg *g = static_cast<const Tg *>(p.g);
    const int tid = threadIdx.x, nt = blockDim.x;
    const size_t r0 = (row0 * p.H + h) * DK, rs = (size_t)p.H * DK;
    if (Ql) wg::load_tile<C, DK, SK, 256>(q + r0, rs, nvalid, Ql);
    if (Kr) wg::load_tile<C, DK, SK, 256>(k + r0, rs, nvalid, Kr);
    if (Ar) wg::load_tile<C, DK, SK, 256>(a + r0, rs, nvalid, Ar);
    if (Bl) wg::load_tile<C, DK, SK, 256>(bb + r0, rs, nvalid, Bl);
    if (p.gate_kind == KDA_GATE_CHANNEL) wg::load_tile<C, DK, SK, 256>(g + r0, rs, nvalid, Gm);
    if (tid < C) {
        float gv = 0.f;
        if (tid < nvalid && p.gate_kind == KDA_GATE_SCALAR) gv = ldf(g, (row0 + tid) * p.H + h);
        gsc[tid] = gv;
    }
    __syncthreads();
    for (int d = tid; d < DK; d += nt) {
        float G = 0.f, gm = 1.f;
        for (int c = 0; c < C; ++c) {
            if (c < nvalid) {
                float gv = p.gate_kind == KDA_GATE_CHANNEL ? Gm[c * SK + d] : gsc[c];   // channel: staged above
                if (p.clip) gv = fminf(gv, rows[c].w);
                G += gv;
                gm = expf(G);
            }
            Gm[c * SK + d] = gm;
            if (Ql) Ql[c * SK + d] *= gm;
            if (Kr) Kr[c * SK + d] /= gm;
            if (Ar) Ar[c * SK + d] /= gm;
            if (Bl) Bl[c * SK + d] *= gm;
        }
        gam[d] = gm;
    }
}

// E = (I + Nm)^{-1} for a strictly lower Nm (row stride SC, C = 32): the two
// 16x16 diagonal blocks by forward substitution side by side, then
// E21 = -E22 N21 E11 by two parallel products (Tm: [C][SC] scratch).  Starts
// after, and ends with, a barrier.
template <int SC>
__device__ void block_inverse32(const float *Nm, float *Em, float *Tm) {
    constexpr int C = 32, HB = 16;
    const int tid = threadIdx.x, nt = blockDim.x;
    if (tid < C) {
        const int blk = tid / HB, c = blk * HB + tid % HB;
        for (int i = blk * HB; i < blk * HB + HB; ++i) {
            float y = 0.f;
            if (i == c) y = 1.f;
            else if (i > c)
                for (int j = c; j < i; ++j) y -= Nm[i * SC + j] * Em[j * SC + c];
            Em[i * SC + c] = y;
        }
        for (int i = 0; i < HB; ++i) Em[(blk == 0 ? i : HB + i) * SC + (blk == 0 ? HB : 0) + tid % HB] = 0.f;
    }
    __syncthreads();
    for (int idx = tid; idx < HB * HB; idx += nt) {
        const int i = HB + idx / HB, j = idx % HB;
        float acc = 0.f;
        for (int l = j; l < HB; ++l) acc += Nm[i * SC + l] * Em[l * SC + j];
        Tm[i * SC + j] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < HB * HB; idx += nt) {
        const int i = HB + idx / HB, j = idx % HB;
        float acc = 0.f;
        for (int l = HB; l <= i; ++l) acc -= Em[i * SC + l] * Tm[l * SC + j];
        Em[i * SC + j] = acc;
    }
    __syncthreads();
}

}  // namespace dplr
}  // namespace kda
