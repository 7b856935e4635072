// Warp-tiled products for the chunk-parallel backward kernels.
//
// A CTA of 8 (or 16) warps computes a 32 x N block (N in {32, 64, 128}) of a
// product sum_k A(i, k) B(k, n): warp w owns rows 16 (w & 1) .. +16 and a
// column range of N / 4 (or N / 8), i.e. tiles of 16 x 8.  Operands come
// through accessor functors (shared or global memory, any layout or
// transform).  TF32 = true issues warp-level m16n8k8 tf32 tensor-core MMAs
// with float32 accumulation (operands rounded to tf32); TF32 = false computes
// the same fragment elements exactly in float32 on the CUDA cores.
#pragma once

#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace kda {
namespace wg {

using tc::mma_tf32_16x8x8;
using tc::to_tf32;

// acc[nt][q] is element (row0 + g + 8 (q >> 1), col0 + 8 nt + 2 t + (q & 1)) of the tile,
// g = lane / 4, t = lane % 4 (the m16n8 accumulator layout).
template <int NT, bool TF32, typename FA, typename FB>
__device__ __forceinline__ void tile(float (&acc)[NT][4], int row0, int col0, int K, const FA &A, const FB &B) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    if constexpr (TF32) {
#pragma unroll 2
        for (int k0 = 0; k0 < K; k0 += 8) {
            const uint32_t a[4] = {to_tf32(A(row0 + g, k0 + t)), to_tf32(A(row0 + g + 8, k0 + t)),
                                   to_tf32(A(row0 + g, k0 + t + 4)), to_tf32(A(row0 + g + 8, k0 + t + 4))};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int n = col0 + 8 * nt + g;
                const uint32_t b[2] = {to_tf32(B(k0 + t, n)), to_tf32(B(k0 + t + 4, n))};
                mma_tf32_16x8x8(acc[nt], a, b);
            }
        }
    } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = row0 + g + 8 * (q >> 1), n = col0 + 8 * nt + 2 * t + (q & 1);
                float s = 0.f;
#pragma unroll 4
                for (int k = 0; k < K; ++k) s += A(r, k) * B(k, n);
                acc[nt][q] += s;
            }
    }
}

// Calls epi(row, col, value) for every element of this thread's fragments.
template <int NT, typename FE>
__device__ __forceinline__ void store(const float (&acc)[NT][4], int row0, int col0, const FE &epi) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) epi(row0 + g + 8 * (q >> 1), col0 + 8 * nt + 2 * t + (q & 1), acc[nt][q]);
}

// Tiles of a 32 x N block over NW warps (8 or 16): warp w owns rows
// 16 (w & 1) .. +16 and columns (w >> 1) N / (NW / 2) .. + N / (NW / 2); when
// that is narrower than one 8-column tile (N = 32 with 16 warps) the warps
// past the tiles sit out.
template <int N, int NW>
__host__ __device__ constexpr int ntiles() { return N / (NW / 2) >= 8 ? N / (NW / 2) / 8 : 1; }

// Calls epi(row, col, a1, a2) for two accumulators of the same tile shape.
template <int NT, typename FE>
__device__ __forceinline__ void store_pair(const float (&a1)[NT][4], const float (&a2)[NT][4], int row0, int col0,
                                           const FE &epi) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q)
            epi(row0 + g + 8 * (q >> 1), col0 + 8 * nt + 2 * t + (q & 1), a1[nt][q], a2[nt][q]);
}

// This warp's tile origin in a 32 x N block; false when the warp has no tile.
template <int N, int NW = 8>
__device__ __forceinline__ bool origin(int &row0, int &col0) {
    const int w = threadIdx.x >> 5;
    constexpr int W = N / (NW / 2) >= 8 ? N / (NW / 2) : 8;     // columns per warp pair
    row0 = 16 * (w & 1);
    col0 = (w >> 1) * W;
    return col0 < N;
}

// out(i, n) = epi(i, n, sum_k A(i, k) B(k, n)) over a 32 x N block.
template <int N, bool TF32, int NW = 8, typename FA, typename FB, typename FE>
__device__ __forceinline__ void gemm(int K, const FA &A, const FB &B, const FE &epi) {
    constexpr int NT = ntiles<N, NW>();
    int r0, c0;
    if (!origin<N, NW>(r0, c0)) return;
    float acc[NT][4] = {};
    tile<NT, TF32>(acc, r0, c0, K, A, B);
    store<NT>(acc, r0, c0, epi);
}

// out(i, n) = epi(i, n, sum_k A1 B1 + sum_k A2 B2).
template <int N, bool TF32, int NW = 8, typename FA1, typename FB1, typename FA2, typename FB2, typename FE>
__device__ __forceinline__ void gemm2(int K1, const FA1 &A1, const FB1 &B1, int K2, const FA2 &A2, const FB2 &B2,
                                      const FE &epi) {
    constexpr int NT = ntiles<N, NW>();
    int r0, c0;
    if (!origin<N, NW>(r0, c0)) return;
    float acc[NT][4] = {};
    tile<NT, TF32>(acc, r0, c0, K1, A1, B1);
    tile<NT, TF32>(acc, r0, c0, K2, A2, B2);
    store<NT>(acc, r0, c0, epi);
}

// out(i, n) = epi(i, n, sum_k A1 B1, sum_k A2 B2): two products kept apart.
template <int N, bool TF32, int NW = 8, typename FA1, typename FB1, typename FA2, typename FB2, typename FE>
__device__ __forceinline__ void gemm_pair(int K1, const FA1 &A1, const FB1 &B1, int K2, const FA2 &A2,
                                          const FB2 &B2, const FE &epi) {
    constexpr int NT = ntiles<N, NW>();
    int r0, c0;
    if (!origin<N, NW>(r0, c0)) return;
    float a1[NT][4] = {}, a2[NT][4] = {};
    tile<NT, TF32>(a1, r0, c0, K1, A1, B1);
    tile<NT, TF32>(a2, r0, c0, K2, A2, B2);
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q)
            epi(r0 + g + 8 * (q >> 1), c0 + 8 * nt + 2 * t + (q & 1), a1[nt][q], a2[nt][q]);
}

// ---- 16-row blocks (16-token chunks): warp w owns columns w N / 8 .. + N / 8 (N >= 64),
// or one 16 x 8 tile for N in {16, 32} (warps past N / 8 sit out).
template <int N>
__host__ __device__ constexpr int nt16() { return N >= 64 ? N / 64 : 1; }

template <int N>
__device__ __forceinline__ bool origin16(int &col0) {
    const int w = threadIdx.x >> 5;
    if constexpr (N >= 64) {
        col0 = w * (N / 8);
        return true;
    } else {
        col0 = w * 8;
        return w < N / 8;
    }
}

template <int N, bool TF32, typename FA, typename FB, typename FE>
__device__ __forceinline__ void gemm16(int K, const FA &A, const FB &B, const FE &epi) {
    constexpr int NT = nt16<N>();
    int c0;
    if (!origin16<N>(c0)) return;
    float acc[NT][4] = {};
    tile<NT, TF32>(acc, 0, c0, K, A, B);
    store<NT>(acc, 0, c0, epi);
}

template <int N, bool TF32, typename FA1, typename FB1, typename FA2, typename FB2, typename FE>
__device__ __forceinline__ void gemm16_2(int K1, const FA1 &A1, const FB1 &B1, int K2, const FA2 &A2, const FB2 &B2,
                                         const FE &epi) {
    constexpr int NT = nt16<N>();
    int c0;
    if (!origin16<N>(c0)) return;
    float acc[NT][4] = {};
    tile<NT, TF32>(acc, 0, c0, K1, A1, B1);
    tile<NT, TF32>(acc, 0, c0, K2, A2, B2);
    store<NT>(acc, 0, c0, epi);
}

template <int N, bool TF32, typename FA1, typename FB1, typename FA2, typename FB2, typename FA3, typename FB3,
          typename FE>
__device__ __forceinline__ void gemm16_3(int K1, const FA1 &A1, const FB1 &B1, int K2, const FA2 &A2, const FB2 &B2,
                                         int K3, const FA3 &A3, const FB3 &B3, const FE &epi) {
    constexpr int NT = nt16<N>();
    int c0;
    if (!origin16<N>(c0)) return;
    float acc[NT][4] = {};
    tile<NT, TF32>(acc, 0, c0, K1, A1, B1);
    tile<NT, TF32>(acc, 0, c0, K2, A2, B2);
    tile<NT, TF32>(acc, 0, c0, K3, A3, B3);
    store<NT>(acc, 0, c0, epi);
}

template <int N, bool TF32, typename FA1, typename FB1, typename FA2, typename FB2, typename FE>
__device__ __forceinline__ void gemm16_pair(int K1, const FA1 &A1, const FB1 &B1, int K2, const FA2 &A2,
                                            const FB2 &B2, const FE &epi) {
    constexpr int NT = nt16<N>();
    int c0;
    if (!origin16<N>(c0)) return;
    float a1[NT][4] = {}, a2[NT][4] = {};
    tile<NT, TF32>(a1, 0, c0, K1, A1, B1);
    tile<NT, TF32>(a2, 0, c0, K2, A2, B2);
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) epi(g + 8 * (q >> 1), c0 + 8 * nt + 2 * t + (q & 1), a1[nt][q], a2[nt][q]);
}

// ---- staging of [rows][D] tiles from global memory
// 8 consecutive elements as floats: one 16-byte load for bf16, two for fp32.
__device__ __forceinline__ float ldf1(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float ldf1(float x) { return x; }
__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void ld8(const float *p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Rows c < R of a row-major source (row c at src + c * rs elements, D columns,
// 16-byte aligned) into dst[c * SD + d] as floats; rows >= nvalid become zero.
// Every thread issues all of its loads before its shared-memory stores.
template <int R, int D, int SD, int NT, typename T>
__device__ __forceinline__ void load_tile(const T *src, size_t rs, int nvalid, float *dst) {
    static_assert(D % 8 == 0 && SD % 4 == 0, "tile shape");
    constexpr int V = D / 8, TOT = R * V, IT = (TOT + NT - 1) / NT;
    float x[IT][8];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int idx = threadIdx.x + it * NT;
        const int c = idx / V, d0 = (idx % V) * 8;
        if (idx < TOT && c < nvalid) {
            ld8(src + (size_t)c * rs + d0, x[it]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) x[it][j] = 0.f;
        }
    }
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int idx = threadIdx.x + it * NT;
        if (idx < TOT) {
            const int c = idx / V, d0 = (idx % V) * 8;
            float4 *q = reinterpret_cast<float4 *>(dst + c * SD + d0);
            q[0] = make_float4(x[it][0], x[it][1], x[it][2], x[it][3]);
            q[1] = make_float4(x[it][4], x[it][5], x[it][6], x[it][7]);
        }
    }
}

// Asynchronous copy of an R x D float32 tile (global row stride rs floats, shared row stride SD;
// every row start 16-byte aligned) by cp.async, 16 bytes per request, NT threads.  Completes
// through cp_async_commit / cp_async_wait, so the next chunk's tiles can travel while the
// current chunk computes.
template <int R, int D, int SD, int NT>
__device__ __forceinline__ void load_tile_async(const float *src, size_t rs, float *dst) {
    static_assert(D % 4 == 0 && SD % 4 == 0, "tile shape");
    constexpr int V = D / 4, TOT = R * V;
    for (int idx = threadIdx.x; idx < TOT; idx += NT) {
        const int c = idx / V, d0 = (idx % V) * 4;
        const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(dst + c * SD + d0));
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(src + (size_t)c * rs + d0)
                     : "memory");
    }
}
// The raw rows of an R x D tile of T (bf16 or float) into a shared staging tile with row stride D,
// rows at or past nvalid zero-filled; every row start 16-byte aligned.  to_f32 converts it.
template <int R, int D, typename T, int NT>
__device__ __forceinline__ void load_raw_async(const T *src, size_t rs, int nvalid, T *dst) {
    constexpr int E = 16 / sizeof(T), V = D / E, TOT = R * V;   // elements per request, requests per row
    static_assert(D % E == 0, "tile shape");
    for (int idx = threadIdx.x; idx < TOT; idx += NT) {
        const int c = idx / V, d0 = (idx % V) * E;
        const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(dst + c * D + d0));
        const int bytes = c < nvalid ? 16 : 0;                   // 0: the request writes zeros
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s),
                     "l"(src + (size_t)min(c, max(nvalid - 1, 0)) * rs + d0), "r"(bytes)
                     : "memory");
    }
}
template <int R, int D, int SD, typename T, int NT>
__device__ __forceinline__ void to_f32(const T *stage, float *dst) {
    for (int idx = threadIdx.x; idx < R * D; idx += NT) dst[(idx / D) * SD + idx % D] = ldf1(stage[idx]);
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed groups are still in flight.
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace wg
}  // namespace kda
