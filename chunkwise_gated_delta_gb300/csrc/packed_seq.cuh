// Rows and chunk slots of the sequences of a dense or a packed batch, for the
// float32 chunk kernels whose chunk-parallel CTAs write per-chunk records.
//
// Dense batches: sequence b holds rows b T .. b T + T - 1 of the [B, T] batch
// and chunk slots b N .. b N + N - 1 (N = ceil(T / C)).  Packed sequences
// (cu_seqlens): sequence b holds rows lo .. hi - 1 of the one [1, T] batch
// (offsets clamped into [0, T]) and chunk slots b + floor(lo / C) + n.  The next
// sequence's first slot lies at least ceil((hi - lo) / C) further on, so no two
// sequences share a slot, and B + ceil(T / C) slots hold them all, whatever the
// offsets (clamped ones included).  The states before each chunk take one more
// slot per sequence (its final state): state slot = chunk slot + b.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace kda {
namespace seq {

struct Seq {
    int row0;    // first row of the sequence in its batch (b T, or lo)
    int len;     // rows
    int slot0;   // first chunk slot
    int nch;     // chunks
};

template <int C>
__host__ __device__ __forceinline__ int chunk_slots(int B, int T, bool packed) {
    const int N = (T + C - 1) / C;
    return packed ? B + N : B * N;
}

// P: a parameter block with B, T and cu_seqlens (null for a dense batch).
template <int C, class P>
__host__ __device__ __forceinline__ Seq seq_of(const P &p, int b) {
    const int N = (p.T + C - 1) / C;
    if (!p.cu_seqlens) return Seq{b * p.T, p.T, b * N, N};
    const int lo = min(max(p.cu_seqlens[b], 0), p.T);
    const int hi = min(max(p.cu_seqlens[b + 1], lo), p.T);
    return Seq{lo, hi - lo, b + lo / C, (hi - lo + C - 1) / C};
}

// The sequence and chunk of chunk slot s of a packed batch: the last sequence whose first
// slot is at or before s, by bisection.  False for a slot no sequence uses.
template <int C, class P>
__host__ __device__ __forceinline__ bool slot_of(const P &p, int s, int &b, int &n, Seq &sq) {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seq_of<C>(p, mid).slot0 <= s) lo = mid;
        else hi = mid - 1;
    }
    b = lo;
    sq = seq_of<C>(p, b);
    n = s - sq.slot0;
    return n >= 0 && n < sq.nch;
}

// The sequence and chunk of a chunk-parallel CTA: grid (N, H, B) for dense batches;
// (chunk slots, H, 1) for packed sequences (slot_of).  False for a slot no sequence uses
// (the whole CTA then returns).
template <int C, class P>
__device__ __forceinline__ bool chunk_of(const P &p, int &b, int &n, Seq &sq) {
    if (!p.cu_seqlens) {
        b = blockIdx.z;
        n = blockIdx.x;
        sq = seq_of<C>(p, b);
        return true;
    }
    return slot_of<C>(p, (int)blockIdx.x, b, n, sq);
}

// Grid of the chunk-parallel kernels.
template <int C>
inline dim3 chunk_grid(int B, int T, int H, bool packed) {
    return packed ? dim3(chunk_slots<C>(B, T, true), H, 1) : dim3((T + C - 1) / C, H, B);
}

// Workspace index of chunk n of a sequence for head h, arrays laid out [H][slots]: chunk
// slots (records and per-chunk products), and state slots (the state before each chunk,
// then the final one).
template <int C, class P>
__host__ __device__ __forceinline__ size_t chunk_index(const P &p, const Seq &sq, int h, int n) {
    return (size_t)h * chunk_slots<C>(p.B, p.T, p.cu_seqlens != nullptr) + sq.slot0 + n;
}
template <int C, class P>
__host__ __device__ __forceinline__ size_t state_index(const P &p, const Seq &sq, int b, int h, int n) {
    return (size_t)h * (chunk_slots<C>(p.B, p.T, p.cu_seqlens != nullptr) + p.B) + sq.slot0 + b + n;
}

}  // namespace seq
}  // namespace kda
