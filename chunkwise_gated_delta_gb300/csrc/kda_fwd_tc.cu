// Fused tcgen05 kernel for the chunkwise KDA forward (bf16 in, fp32 accumulate,
// fp32 state), GB300 / sm_103a.
//
// One CTA owns one (batch, head, 64-wide value slice) and walks its chunks in
// order.  The chunk form it evaluates is the one recapped on page "Kimi Delta
// Attention backward" ("forward recap"), regrouped so every tensor-core
// product has M = 128 rows:
//
//   [beta K<- ; Q<-] K->^T      = [L ; P]          (Gram, one MMA)
//   Z' (I + L_{strict}) = [I ; P],  Z = Z' Diag(beta) = [T ; P T]
//        with T = (I + L)^{-1} Diag(beta): block back-substitution over
//        16-column blocks (page "DeltaNet" 4.2, block form 2), the 16x16
//        diagonal blocks inverted by warp shuffles, the block products as
//        tf32 warp MMAs, 16 rows of Z' per warp
//   Z K<-                       = [W ; P W]
//   Z V                         = [U ; P U]        (into the accumulator D1)
//   D1 += [-W ; Q<- - P W] S^T  = [V_new ; O]      (state-dependent, one MMA)
//   K->^T V_new                 = dS^T,  S <- (S + dS) Diag(gamma^C)
//
// O = Q<- S^T + (Q<- K->^T * M) V_new expands to (Q<- - P W) S^T + P U, which
// is why the output rides in the lower half of the state-dependent product;
// the state step uses the factored form of page "Gated Linear Attention" 5.2.
//
// Warp roles (384 threads):
//   warps 0-3  "chain": the serial part -- the state S^T (128 key channels x
//              64 values) in fp32 registers, one key channel per thread.
//   warps 4-11 "WY": everything that does not depend on S.
//
// Two forms.
//   Records (two kernels, when the caller's workspace holds them): a
//   chunk-parallel kernel computes, for every chunk, Gamma, the rescaled tiles
//   and Z -- the Gram, the inverse and the back-substitution, which dominate
//   the state-independent work -- and writes them as a chunk record (the bf16
//   tile images Z, Q<-, K<-, K-> and gamma^C).  The scan kernel then runs one
//   CTA per (batch, head, 64-wide value slice); its WY warps only form
//   [W ; P W] = Z K<-, [U ; P U] = Z V and A_chain, with Z and K<- double
//   buffered, while the chain warps load Q<- (into A_chain's slot), K-> and
//   gamma^C two chunks ahead.
//   Single kernel (a 256-byte workspace): the WY warps build Z themselves.
//   With dv = 128 the two value-slice CTAs of a head form a cluster and split
//   that work by chunk parity: CTA r builds the chunks n with n % 2 == r and
//   copies their slot tiles (A_chain, K->, gamma^C) and Z into the other CTA's
//   shared memory; each CTA still runs the state scan of every chunk for its
//   own value slice and forms its own [U ; P U] = Z V.  With dv = 64 one CTA
//   does it all.
//
// Warps reach every aligned instruction (bar.sync, tcgen05.ld) converged: each
// block that only the issuing thread runs is followed by __syncwarp().
//
// Every wait on an mbarrier is bounded; on timeout the kernel writes the
// status word (and where it gave up, in the words after it), turns every later
// wait into a no-op and runs to its end.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_internal.h"
#include "tc_common.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kC = 64;        // chunk length
constexpr int kDK = 128;      // key dim
constexpr int kDVS = 64;      // value channels per CTA
constexpr int kChainThreads = 128;
constexpr int kWyThreads = 256;
constexpr int kThreads = kChainThreads + kWyThreads;
constexpr float kLog2e = 1.4426950408889634f;

// ---- shared memory map (byte offsets from a 1024-aligned base).  Operand
// tiles are bf16 column blocks of 64 with 128-byte swizzle.
constexpr uint32_t OFF_AG = 0;           // [beta K<- ; Q<-] 128 x 128 K-major.  Raw g lands in its
                                         // rows 0-63 and raw q in rows 64-127; after the Gram,
                                         // rows 0-63 hold the diagonal-block inverses (fp32).
constexpr uint32_t OFF_KR = 32768;       // K-> 64 x 128 (K-major B); then L (fp32), then Z
constexpr uint32_t OFF_KL = 49152;       // raw k, then K<- 64 x 128 (MN-major B)
constexpr uint32_t OFF_V0 = 65536;       // v slice [64][64] (MN-major B), slot 0
constexpr uint32_t OFF_V1 = 73728;       // slot 1
constexpr uint32_t OFF_ACH0 = 81920;     // [-W ; Q'] 128 x 128 K-major, slot 0
constexpr uint32_t OFF_ACH1 = 114688;    // slot 1
constexpr uint32_t OFF_KT0 = 147456;     // K-> 64 x 128 (MN-major A of dS), slot 0
constexpr uint32_t OFF_KT1 = 163840;     // slot 1
constexpr uint32_t OFF_ZIN = 180224;     // Z received from the other CTA of the pair
constexpr uint32_t OFF_ST = 196608;      // S^T 128 x 64 (MN-major B); V_new in its first 8 KB
constexpr uint32_t OFF_OST = 212992;     // O staging [64][64] for the TMA store
constexpr uint32_t OFF_MISC = 221184;
constexpr uint32_t MISC_GC = 0;          // gamma^C [2][128] f32            (1024 B)
constexpr uint32_t MISC_BETA = 1024;     // beta [2][64] f32                 (512 B)
constexpr uint32_t MISC_GS = 1536;       // scalar gate [2][64] f32          (512 B)
constexpr uint32_t MISC_TOT = 2048;      // cumsum partials [8][128] f32     (4096 B)
constexpr uint32_t MISC_BAR = 6144;      // mbarriers [24] u64               (192 B)
constexpr uint32_t MISC_TSLOT = 6400;    // TMEM base address
constexpr uint32_t MISC_ABORT = 6404;    // abort flag
constexpr uint32_t kMiscBytes = 6656;
constexpr uint32_t kSmemBytes = OFF_MISC + kMiscBytes + 1024;   // + alignment slack of the dynamic base
static_assert(MISC_GC + 2 * 128 * 4 <= MISC_BETA, "misc layout");
static_assert(MISC_BETA + 2 * 64 * 4 <= MISC_GS, "misc layout");
static_assert(MISC_GS + 2 * 64 * 4 <= MISC_TOT, "misc layout");
static_assert(MISC_TOT + 8 * 128 * 4 <= MISC_BAR, "misc layout");
static_assert(MISC_BAR + 24 * 8 <= MISC_TSLOT, "misc layout");
static_assert(MISC_ABORT + 4 <= kMiscBytes, "misc layout");
static_assert(OFF_OST + 8192 <= OFF_MISC, "tile layout");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");


// bytes one CTA of a pair sends the other per chunk it builds: Z (st.async) and the slot tiles
// (bulk copies)
constexpr uint32_t kPushBytes = 16384 + 32768 + 16384 + 512;
// One chunk's record (Z kernel -> scan kernel): images of the bf16 tiles the scan kernel reads.
constexpr uint32_t REC_Z = 0;            // Z, K-major 128 x 64
constexpr uint32_t REC_Q = 16384;        // Q<-, 64 x 128 (rows 64-127 of the A_G tile)
constexpr uint32_t REC_KL = 32768;       // K<-, MN-major 64 x 128
constexpr uint32_t REC_KR = 49152;       // K->, 64 x 128 (the slot tile)
constexpr uint32_t REC_GC = 65536;       // gamma^C [128] f32
constexpr uint32_t kRecBytes = 66048;

// ---- TMEM columns
constexpr uint32_t TM_G = 0;      // Gram [L ; P], 64 cols
constexpr uint32_t TM_WQ = 128;   // [W ; P W], 128 cols
constexpr uint32_t TM_D1 = 256;   // [U ; P U] -> [V_new ; O], 2 slots x 64 cols
constexpr uint32_t TM_S = 384;    // dS^T, 64 cols
constexpr uint32_t kTmemCols = 512;

// mbarrier indices
enum {
    B_RAW = 0, B_V0, B_V1, B_GRAM, B_W2, B_WYR0, B_WYR1, B_C10, B_C11, B_C20, B_C21, B_E10, B_E11,
    B_RX, B_PFREE, B_FIN0, B_FIN1, B_ZK0, B_ZK1, B_SL0, B_SL1, kNumBars
};
static_assert(kNumBars <= 24, "mbarrier slots");

__device__ __forceinline__ uint32_t off_ach(int s) { return s ? OFF_ACH1 : OFF_ACH0; }
__device__ __forceinline__ uint32_t off_kt(int s) { return s ? OFF_KT1 : OFF_KT0; }
__device__ __forceinline__ uint32_t off_v(int s) { return s ? OFF_V1 : OFF_V0; }

struct Ctx {
    uint8_t *base;
    uint64_t *bars;
    volatile int *abort;
    int *status;
    uint32_t tmem;
    uint32_t rank;     // rank in the pair (0 without a pair)
    const uint8_t *zrec;   // Z record of chunk 0 of this (sequence, head); chunk n at zrec + n * zstride
    size_t zstride;
};

// A wait ran out: the CTA stops waiting, and the status word says so.  The
// first wait to run out in the launch also leaves where it was in the next
// words of the status block: barrier index + 1, parity, thread, block (x, y, z
// in bytes 0-2).
__device__ __forceinline__ void record_timeout(const Ctx &c, int idx, uint32_t parity) {
    *c.abort = 1;
    atomicCAS(c.status, kDevOk, kDevTimeout);
    if (atomicCAS(c.status + 1, 0, idx + 1) == 0) {
        c.status[2] = (int)parity;
        c.status[3] = (int)threadIdx.x;
        c.status[4] = (int)(blockIdx.x | (blockIdx.y << 8) | (blockIdx.z << 16));
    }
}
// A wait given up because another thread of the CTA gave up: the two issuing threads (chain
// leader 0, WY leader 128) leave the barrier they were on in words 5 and 6.
__device__ __forceinline__ void note_abort(const Ctx &c, int idx, uint32_t parity) {
    if (threadIdx.x == 0) atomicCAS(c.status + 5, 0, idx + 1 + 256 * (int)parity);
    if (threadIdx.x == kChainThreads) atomicCAS(c.status + 6, 0, idx + 1 + 256 * (int)parity);
}

// Bounded wait that becomes a no-op once any thread of the CTA has given up.
__device__ __noinline__ void wait_bar(const Ctx &c, int idx, uint32_t parity) {
    uint64_t *bar = c.bars + idx;
    for (uint32_t i = 0; i < kWaitBound; ++i) {
        if (mbar_try_wait(bar, parity)) return;
        if (*c.abort) {
            note_abort(c, idx, parity);
            return;
        }
    }
    record_timeout(c, idx, parity);
}
// The same for barriers completed from the other CTA of the pair.
__device__ __noinline__ void wait_bar_cluster(const Ctx &c, int idx, uint32_t parity) {
    uint64_t *bar = c.bars + idx;
    for (uint32_t i = 0; i < kWaitBound; ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return;
        if (*c.abort) {
            note_abort(c, idx, parity);
            return;
        }
    }
    record_timeout(c, idx, parity);
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void st_u128(uint8_t *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}
__device__ __forceinline__ void st_u64(uint8_t *p, uint2 v) { *reinterpret_cast<uint2 *>(p) = v; }
__device__ __forceinline__ uint2 pack4(float a, float b, float c, float d) {
    return make_uint2(pack_bf16(a, b), pack_bf16(c, d));
}
__device__ __forceinline__ float4 ld_bf16x4(const uint8_t *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
// 32 fp32 values -> 64 bytes of bf16 at (row, col .. col+31) of a SW128 tile with `rows` rows.
__device__ __forceinline__ void store_row32_bf16(uint8_t *tile, uint32_t rows, uint32_t row, uint32_t col,
                                                 const float *v) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
        st_u128(tile + sw128_offset(rows, row, col + 8 * q), pack_bf16(v[8 * q], v[8 * q + 1]),
                pack_bf16(v[8 * q + 2], v[8 * q + 3]), pack_bf16(v[8 * q + 4], v[8 * q + 5]),
                pack_bf16(v[8 * q + 6], v[8 * q + 7]));
}

// A row of Z (128 x 64 K-major tile): also sent to the other CTA of the pair at `remote`
// (its address of `tile`) by asynchronous stores that complete on its barrier `rbar`.
template <bool REMOTE>
__device__ __forceinline__ void store_row32_z(uint8_t *tile, uint32_t remote, uint32_t rbar, uint32_t row, uint32_t col,
                                              const float *v) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t off = sw128_offset(128, row, col + 8 * q);
        const uint32_t a = pack_bf16(v[8 * q], v[8 * q + 1]), b = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
        const uint32_t c = pack_bf16(v[8 * q + 4], v[8 * q + 5]), d = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
        st_u128(tile + off, a, b, c, d);
        if (REMOTE) st_async_u128(remote + off, a, b, c, d, rbar);
    }
}

template <typename T> __device__ __forceinline__ float ldg_f(const T *p);
template <> __device__ __forceinline__ float ldg_f<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
template <> __device__ __forceinline__ float ldg_f<float>(const float *p) { return *p; }

// ---- fp32 [64][64] scratch for the inverse, with an XOR swizzle on column
// bits 2-4: float4 groups stay contiguous, and row walks spread over the banks.
__device__ __forceinline__ uint32_t sidx(uint32_t i, uint32_t j) { return i * 64u + (j ^ ((i & 7u) << 2)); }

struct Scratch {
    uint8_t *base;
    __device__ __forceinline__ float *L(uint32_t i, uint32_t j) const {
        return reinterpret_cast<float *>(base + OFF_KR) + sidx(i, j);
    }
    // Y lives in the dead beta K<- rows of the A_G tile: rows 0-31 at +0, rows 32-63 at +16 KB.
    __device__ __forceinline__ float *Y(uint32_t i, uint32_t j) const {
        return reinterpret_cast<float *>(base + OFF_AG + (i >= 32 ? 16384u : 0u)) + sidx(i & 31u, j);
    }
};

// Where a (batch, head) sequence lives: tensor-map batch coordinate, first row
// and length.  Dense batches: (b, 0, T).  Packed variable-length batches
// (cu_seqlens): (0, cu_seqlens[b], cu_seqlens[b + 1] - cu_seqlens[b]).
struct Seq {
    int bt, t0, len;
};
__device__ __forceinline__ Seq seq_of(const FwdParams &p, int b) {
    if (!p.cu_seqlens) return Seq{b, 0, p.T};
    const int lo = min(max(p.cu_seqlens[b], 0), p.T);      // offsets clamped into [0, T]
    const int hi = min(max(p.cu_seqlens[b + 1], lo), p.T);
    return Seq{0, lo, hi - lo};
}
// Z record slot of chunk 0 of sequence b.  Dense: b * ceil(T / C).  Packed:
// b + floor(t0 / C), which never collides with the next sequence's slots
// (floor(t0 / C) + ceil(len / C) <= floor((t0 + len) / C) + 1), so B + ceil(T / C)
// slots per head cover every packing.
__device__ __forceinline__ int zslot0(const FwdParams &p, int b, const Seq &sq) {
    return p.cu_seqlens ? b + sq.t0 / kC : b * ((p.T + kC - 1) / kC);
}

// Accumulator fragments of a 16x16 block (two 16x8 halves) -> tf32 A fragments of the
// same block (k-steps 0 and 1), times `sign`, by shuffles within the warp.
__device__ __forceinline__ void frag_c_to_a(const float (&x)[2][4], uint32_t (&a)[2][4], int lane, float sign) {
    const int g = lane >> 2, t = lane & 3;
    const int s0 = 4 * g + (t >> 1), s1 = s0 + 2;
    const bool odd = (t & 1) != 0;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const float v0 = __shfl_sync(0xffffffffu, x[ks][0], s0), v1 = __shfl_sync(0xffffffffu, x[ks][1], s0);
        const float v2 = __shfl_sync(0xffffffffu, x[ks][2], s0), v3 = __shfl_sync(0xffffffffu, x[ks][3], s0);
        const float w0 = __shfl_sync(0xffffffffu, x[ks][0], s1), w1 = __shfl_sync(0xffffffffu, x[ks][1], s1);
        const float w2 = __shfl_sync(0xffffffffu, x[ks][2], s1), w3 = __shfl_sync(0xffffffffu, x[ks][3], s1);
        a[ks][0] = to_tf32(sign * (odd ? v1 : v0));
        a[ks][1] = to_tf32(sign * (odd ? v3 : v2));
        a[ks][2] = to_tf32(sign * (odd ? w1 : w0));
        a[ks][3] = to_tf32(sign * (odd ? w3 : w2));
    }
}

// ---- Gamma and the rescaled tiles of one chunk, in place.  Raw g (channel
// gate) sits in A_G rows 0-63, raw q in A_G rows 64-127 and raw k in the
// 64-row tile at `kraw`.  Q<- replaces the raw q; GRAM: beta K<- goes to A_G
// rows 0-63 and K-> to the K-> tile (the Gram's operands); SCAN: K<- goes to
// the K<- tile.  K-> (packed bf16, 8 rows x 4 columns per thread) and gamma^C
// (4 columns) come back for the chunk's slot.  Rows at or past `live_rows`
// are zero; `bet` and `gs` hold the chunk's beta and scalar gate.  The 256 WY
// threads (index wt), 4 columns x 8 rows each; one barrier inside.
//   With `rec` non-null, Q<-, K<-, K-> and gamma^C also go to that chunk record.
template <int GATE, bool GRAM, bool SCAN>
__device__ __forceinline__ void rescale_tiles(uint8_t *base, uint32_t kraw, int wt, int live_rows, const float *bet,
                                              const float *gs, float *tot, uint2 (&krv)[8], float4 &gcv,
                                              uint8_t *rec = nullptr) {
    const int cg = wt & 31, rg = wt >> 5;
    const int col = 4 * cg;
    float G[8][4];
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int row = rg * 8 + r;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (row >= live_rows) {
        } else if (GATE == KDA_GATE_CHANNEL) {
            const float4 gg = ld_bf16x4(base + OFF_AG + sw128_offset(128, row, col));
            x[0] = gg.x; x[1] = gg.y; x[2] = gg.z; x[3] = gg.w;
        } else if (GATE == KDA_GATE_SCALAR) {
            x[0] = x[1] = x[2] = x[3] = gs[row];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) { a[e] += x[e]; G[r][e] = a[e]; }
    }
    *reinterpret_cast<float4 *>(tot + rg * kDK + col) = make_float4(a[0], a[1], a[2], a[3]);
    named_sync(2, kWyThreads);
    float pre[4] = {0.f, 0.f, 0.f, 0.f}, all[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 t4 = *reinterpret_cast<const float4 *>(tot + q * kDK + col);
        const float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (q < rg) pre[e] += tv[e];
            all[e] += tv[e];
        }
    }
    gcv = make_float4(__expf(all[0]), __expf(all[1]), __expf(all[2]), __expf(all[3]));
    if (rec && rg == 0) *reinterpret_cast<float4 *>(rec + REC_GC + 4 * col) = gcv;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int row = rg * 8 + r;
        const uint32_t o64 = sw128_offset(64, row, col);
        const uint32_t otop = sw128_offset(128, row, col), obot = sw128_offset(128, 64 + row, col);
        const bool live = row < live_rows;
        const float4 q4 = live ? ld_bf16x4(base + OFF_AG + obot) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 k4 = live ? ld_bf16x4(base + kraw + o64) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float qv[4] = {q4.x, q4.y, q4.z, q4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
        const float bb = bet[row];
        float kl[4], kr4[4], ql[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float g2 = (G[r][e] + pre[e]) * kLog2e;   // G in base-2 units
            const float ev = ex2_approx(g2), iv = ex2_approx(-g2);
            kl[e] = kv[e] * ev;
            kr4[e] = kv[e] * iv;
            ql[e] = qv[e] * ev;
        }
        const uint2 kr = pack4(kr4[0], kr4[1], kr4[2], kr4[3]);
        if (GRAM) st_u64(base + OFF_AG + otop, pack4(bb * kl[0], bb * kl[1], bb * kl[2], bb * kl[3]));
        st_u64(base + OFF_AG + obot, pack4(ql[0], ql[1], ql[2], ql[3]));
        if (GRAM) st_u64(base + OFF_KR + o64, kr);
        if (SCAN) st_u64(base + OFF_KL + o64, pack4(kl[0], kl[1], kl[2], kl[3]));
        krv[r] = kr;
        if (rec) {
            st_u64(rec + REC_Q + o64, pack4(ql[0], ql[1], ql[2], ql[3]));
            st_u64(rec + REC_KL + o64, pack4(kl[0], kl[1], kl[2], kl[3]));
            st_u64(rec + REC_KR + o64, kr);
        }
    }
}

// ---- Z = [T ; P T] of one chunk (GLA: [I ; P]) from its rescaled tiles, as a
// bf16 K-major 128 x 64 tile in the K-> tile: the Gram [beta K<- ; Q<-] K->^T
// into TMEM, L and the inverses of its 16x16 diagonal blocks, the block
// back-substitution, the beta scaling.  The 256 WY threads enter after the
// barrier that follows their stores of the rescaled tiles; `ph` is the parity
// of the Gram barrier.  Returns the first of the 16 Z rows this warp wrote;
// ends without a barrier.
template <bool GLA>
__device__ int build_z(const Ctx &c, int wt, const float *bet, uint32_t ph) {
    uint8_t *base = c.base;
    const int ww = wt >> 5, lane = wt & 31;
    const int quarter = ww & 3, half = ww >> 2;
    const bool leader = wt == 0;
    const Scratch sc{base};
    // ---------------- Gram: D_G = [beta K<- ; Q<-] K->^T   (M128 N64 K128)
    if (leader) {
        tc_fence_after();
        const uint32_t a0 = smem_u32(base + OFF_AG), b0 = smem_u32(base + OFF_KR);
        const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16(c.tmem + TM_G, desc_kmajor(a0, 128, ks), desc_kmajor(b0, 64, ks), id, ks > 0);
        mma_commit(c.bars + B_GRAM);
    }
    __syncwarp();
    wait_bar(c, B_GRAM, ph);
    tc_fence_after();
    __syncwarp();                            // the TMEM loads below are warp-collective

    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int row = quarter * 32 + lane;   // TMEM lane owned by this thread

    if (!GLA) {
        // ---- L (strictly lower, rows carry beta) to fp32 scratch in the K-> tile (dead now)
        if (quarter < 2) {
            float v[32];
            tmem_ld32(c.tmem + TM_G + lane_base + half * 32, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int col = half * 32 + 4 * q;
                float4 f;
                f.x = col + 0 < row ? v[4 * q + 0] : 0.f;
                f.y = col + 1 < row ? v[4 * q + 1] : 0.f;
                f.z = col + 2 < row ? v[4 * q + 2] : 0.f;
                f.w = col + 3 < row ? v[4 * q + 3] : 0.f;
                *reinterpret_cast<float4 *>(sc.L(row, col)) = f;
            }
            if (quarter == half) {
                // Level 0 of the inverse: this warp holds the two 16x16 diagonal blocks of its
                // 32 rows (one row per lane).  Row-wise forward substitution,
                // Y[r] = e_r - sum_{j<r} L[r][j] Y[j], rows of the block exchanged by shuffles.
                const int seg = lane >> 4, r = lane & 15;
                float lr[16], y[16];
#pragma unroll
                for (int cc = 0; cc < 16; ++cc) {
                    lr[cc] = seg ? v[16 + cc] : v[cc];
                    y[cc] = (cc == r) ? 1.f : 0.f;
                }
#pragma unroll
                for (int jj = 0; jj < 15; ++jj) {
                    const float lj = (r > jj) ? lr[jj] : 0.f;
#pragma unroll
                    for (int cc = 0; cc <= jj; ++cc) {
                        const float yj = __shfl_sync(0xffffffffu, y[cc], jj, 16);
                        y[cc] -= lj * yj;
                    }
                }
                const int o = quarter * 32 + seg * 16;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    *reinterpret_cast<float4 *>(sc.Y(row, o + 4 * c4)) =
                        make_float4(y[4 * c4], y[4 * c4 + 1], y[4 * c4 + 2], y[4 * c4 + 3]);
            }
        }
        named_sync(2, kWyThreads);
    }

    // ---------------- Z' (I + L) = [I ; P] by block back-substitution over 16-column blocks,
    // 16 rows of Z' per warp: Z'_b = ([I ; P]_b - sum_{b' > b} Z'_{b'} L_{b'b}) Y_bb with
    // Y_bb = (I + L_bb)^{-1} (block form 2 of page "DeltaNet" 4.2, on the transposed system).
    // Then Z = Z' Diag(beta) = [T ; P T].  For GLA (beta = 0, v unscaled) Z = [I ; P].
    float zb[4][2][4];                                     // Z' blocks, accumulator-fragment layout
    const int r0 = quarter * 32 + half * 16;               // first row of Z' owned by this warp
    {
        const int g = lane >> 2, t = lane & 3;
        uint32_t za[4][2][4];                              // -Z' blocks as tf32 A fragments
#pragma unroll
        for (int bb = 3; bb >= 0; --bb) {
            float acc[2][4];
            if (quarter < 2) {                             // identity rows
#pragma unroll
                for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        acc[nh][e] = (r0 + g + 8 * (e >> 1) == 16 * bb + 8 * nh + 2 * t + (e & 1)) ? 1.f : 0.f;
            } else {                                       // rows of P = Q<- K->^T * M (inclusive)
                float pv[8];
                tmem_ld16x256b_x2(c.tmem + TM_G + ((uint32_t)r0 << 16) + 16 * bb, pv);
                const int i0 = r0 - 64;
#pragma unroll
                for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        acc[nh][e] = (16 * bb + 8 * nh + 2 * t + (e & 1) <= i0 + g + 8 * (e >> 1)) ? pv[4 * nh + e]
                                                                                                  : 0.f;
            }
            if (!GLA) {
#pragma unroll
                for (int bp = bb + 1; bp < 4; ++bp)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                        for (int nh = 0; nh < 2; ++nh) {
                            const uint32_t bf[2] = {to_tf32(*sc.L(16 * bp + 8 * ks + t, 16 * bb + 8 * nh + g)),
                                                    to_tf32(*sc.L(16 * bp + 8 * ks + t + 4, 16 * bb + 8 * nh + g))};
                            mma_tf32_16x8x8(acc[nh], za[bp][ks], bf);
                        }
                uint32_t af[2][4];
                frag_c_to_a(acc, af, lane, 1.f);
#pragma unroll
                for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                    for (int e = 0; e < 4; ++e) zb[bb][nh][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                    for (int nh = 0; nh < 2; ++nh) {
                        const uint32_t bf[2] = {to_tf32(*sc.Y(16 * bb + 8 * ks + t, 16 * bb + 8 * nh + g)),
                                                to_tf32(*sc.Y(16 * bb + 8 * ks + t + 4, 16 * bb + 8 * nh + g))};
                        mma_tf32_16x8x8(zb[bb][nh], af[ks], bf);
                    }
                if (bb > 0) frag_c_to_a(zb[bb], za[bb], lane, -1.f);
            } else {
#pragma unroll
                for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                    for (int e = 0; e < 4; ++e) zb[bb][nh][e] = acc[nh][e];
            }
        }
    }
    if (!GLA) named_sync(2, kWyThreads);                   // every warp is done with L in the K-> tile
    // ---------------- Z = Z' Diag(beta) -> bf16 K-major 128 x 64 tile in the K-> tile
    {
        const int g = lane >> 2, t = lane & 3;
        uint8_t *zt = base + OFF_KR;
#pragma unroll
        for (int bb = 0; bb < 4; ++bb)
#pragma unroll
            for (int nh = 0; nh < 2; ++nh) {
                const int c0 = 16 * bb + 8 * nh + 2 * t;
                float b0 = 1.f, b1 = 1.f;
                if (!GLA) {
                    const float2 b2 = *reinterpret_cast<const float2 *>(bet + c0);
                    b0 = b2.x;
                    b1 = b2.y;
                }
                *reinterpret_cast<uint32_t *>(zt + sw128_offset(128, r0 + g, c0)) =
                    pack_bf16(zb[bb][nh][0] * b0, zb[bb][nh][1] * b1);
                *reinterpret_cast<uint32_t *>(zt + sw128_offset(128, r0 + g + 8, c0)) =
                    pack_bf16(zb[bb][nh][2] * b0, zb[bb][nh][3] * b1);
            }
    }
    return r0;
}

// ============================================================================
// WY warps: everything of a chunk that does not depend on the state.
// ============================================================================
template <int GATE, bool GLA, bool PAIR, bool ZREC, typename Tg>
__device__ void wy_role(const Ctx &c, const FwdParams &p, const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                        const CUtensorMap *tm_g, const CUtensorMap *tm_v, int e0, int h, Seq sq, int nchunks) {
    uint8_t *base = c.base;
    const int wt = threadIdx.x - kChainThreads;          // 0..255
    const int ww = wt >> 5;                              // WY warp 0..7
    const int lane = threadIdx.x & 31;
    const int quarter = ww & 3;                          // TMEM lane quarter (warp index mod 4)
    const int half = ww >> 2;                            // column half
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int row = quarter * 32 + lane;                 // TMEM lane owned by this thread
    const bool leader = wt == 0;
    const int T = p.T, H = p.H;
    float *gC = reinterpret_cast<float *>(base + OFF_MISC + MISC_GC);
    float *betas = reinterpret_cast<float *>(base + OFF_MISC + MISC_BETA);
    float *gss = reinterpret_cast<float *>(base + OFF_MISC + MISC_GS);
    float *tot = reinterpret_cast<float *>(base + OFF_MISC + MISC_TOT);
    const __nv_bfloat16 *betag = static_cast<const __nv_bfloat16 *>(p.beta);
    const Tg *gsg = static_cast<const Tg *>(p.g);
    const uint32_t raw_bytes = (GATE == KDA_GATE_CHANNEL ? 3u : 2u) * 16384u;
    const Scratch sc{base};
    const int step = PAIR ? 2 : 1;                       // distance between chunks this CTA builds
    const int first = PAIR ? (int)c.rank : 0;
    auto owns = [&](int n) { return !PAIR || (n & 1) == (int)c.rank; };

    // raw tiles land where their rescaled versions go: g -> A_G rows 0-63,
    // q -> A_G rows 64-127, k -> K<- tile
    auto issue_raw = [&](int n) {
        mbar_arrive_expect_tx(c.bars + B_RAW, raw_bytes);
        for (int blk = 0; blk < 2; ++blk) {
            tma_load_4d(base + OFF_AG + blk * 16384 + 8192, tm_q, c.bars + B_RAW, blk * 64, h, sq.t0 + n * kC, sq.bt);
            tma_load_4d(base + OFF_KL + blk * 8192, tm_k, c.bars + B_RAW, blk * 64, h, sq.t0 + n * kC, sq.bt);
            if (GATE == KDA_GATE_CHANNEL)
                tma_load_4d(base + OFF_AG + blk * 16384, tm_g, c.bars + B_RAW, blk * 64, h, sq.t0 + n * kC, sq.bt);
        }
    };
    // With records: Z and K<- of chunk n, the operands of its products, into buffer n & 1 --
    // (the K-> tile, the K<- tile) or (the Z-in tile, A_G rows 0-127 of column block 0), which
    // nothing else uses without a pair.  The chain loads the rest of the record into the slot.
    auto issue_zk = [&](int n) {
        const uint8_t *r = c.zrec + (size_t)n * c.zstride;
        const int bf = n & 1;
        uint64_t *bar = c.bars + B_ZK0 + bf;
        mbar_arrive_expect_tx(bar, 32768u);
        bulk_load(base + (bf ? OFF_ZIN : OFF_KR), r + REC_Z, 16384u, bar);
        bulk_load(base + (bf ? OFF_AG : OFF_KL), r + REC_KL, 16384u, bar);
    };
    auto issue_v = [&](int n) {
        const int s = n & 1;
        mbar_arrive_expect_tx(c.bars + B_V0 + s, 8192u);
        tma_load_4d(base + off_v(s), tm_v, c.bars + B_V0 + s, e0, h, sq.t0 + n * kC, sq.bt);
    };
    // per-token scalars of chunk n: beta and (GDN) the scalar log-decay
    auto load_scalars = [&](int n, float &bv, float &gv) {
        bv = 0.f; gv = 0.f;
        const int t = n * kC + wt;
        if (wt < kC && t < sq.len) {
            const size_t row = ((size_t)sq.bt * T + sq.t0 + t) * H + h;
            if (p.has_beta) bv = __bfloat162float(betag[row]);
            if (GATE == KDA_GATE_SCALAR) gv = ldg_f<Tg>(gsg + row);
        }
    };

    if (leader) {
        if (ZREC) {
            issue_zk(0);
            if (nchunks > 1) issue_zk(1);
        } else if (first < nchunks) {
            issue_raw(first);
        }
        issue_v(0);                          // nchunks >= 1: empty sequences return before the roles
        if (nchunks > 1) issue_v(1);
    }
    __syncwarp();
    if (!ZREC) {
        float bv, gv;
        load_scalars(first, bv, gv);
        if (wt < kC) { betas[wt] = bv; gss[wt] = gv; }
    }
    named_sync(2, kWyThreads);

    for (int n = 0; n < nchunks; ++n) {
        const int s = n & 1;
        const uint32_t ph2 = (uint32_t)((n >> 1) & 1);

        if (!owns(n)) continue;              // the chain warps take the other CTA's chunks

        // ---------------- a chunk this CTA builds
        const int m = PAIR ? (n >> 1) : n;                   // index among the chunks built here
        const uint32_t phm = (uint32_t)(m & 1);
        const int sb = m & 1;                                // scalar buffer
        const float *bet = betas + sb * kC;
        float nb = 0.f, ng = 0.f;
        const uint32_t peer_base = PAIR ? map_to_rank(smem_u32(base), c.rank ^ 1u) : 0u;
        uint2 krv[8];
        float4 gcv;
        int r0 = 0;                                          // first of the 16 Z rows this warp built

        if constexpr (!ZREC) {
            if (n + step < nchunks) load_scalars(n + step, nb, ng);   // prefetch next built chunk's scalars
            wait_bar(c, B_RAW, phm);
            // ---------------- prologue: Gamma and the rescaled tiles, in place.  K-> and gamma^C also
            // go to the chunk's slot, written at the end (the slot may still be in use).
            rescale_tiles<GATE, true, true>(base, OFF_KL, wt, sq.len - n * kC, bet, gss + sb * kC, tot, krv, gcv);
            fence_proxy_async_smem();
            named_sync(2, kWyThreads);

            r0 = build_z<GLA>(c, wt, bet, phm);
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(2, kWyThreads);
        }

        // ---------------- Z K<- -> [W ; P W],  Z V -> D1[s] = [U ; P U]
        if (leader) {
            wait_bar(c, B_V0 + s, ph2);
            if (ZREC) wait_bar(c, B_ZK0 + s, ph2);               // buffer n & 1 holds Z and K<-
            if (n >= 2) wait_bar(c, B_E10 + s, (uint32_t)(((n - 2) >> 1) & 1));   // D1[s] drained
            tc_fence_after();
            const uint32_t a0 = smem_u32(base + (ZREC && s ? OFF_ZIN : OFF_KR));
            if (!GLA) {
                const uint32_t bk = smem_u32(base + (ZREC && s ? OFF_AG : OFF_KL));
                const uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(c.tmem + TM_WQ, desc_kmajor(a0, 128, ks), desc_mnmajor(bk, 64, ks), id, ks > 0);
            }
            const uint32_t bv = smem_u32(base + off_v(s));
            const uint32_t id = idesc_bf16(128, 64, 0, 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(c.tmem + TM_D1 + s * 64, desc_kmajor(a0, 128, ks), desc_mnmajor(bv, 64, ks), id, ks > 0);
            mma_commit(c.bars + B_W2);
        }
        __syncwarp();                        // aligned TMEM loads and barriers below need whole warps
        wait_bar(c, B_W2, phm);
        tc_fence_after();
        if (leader && n + 2 < nchunks) issue_v(n + 2);           // v[s] consumed
        if (ZREC && leader && n + 2 < nchunks) issue_zk(n + 2);      // buffer n & 1: its products are done
        __syncwarp();
        if (n >= 2) wait_bar(c, B_C20 + s, (uint32_t)(((n - 2) >> 1) & 1));   // own scan done with slot s
        // the other CTA of a pair is done with chunk n - 2, whose slot tiles and Z it received from
        // here: the slot and its Z-in tile may be rewritten
        if (PAIR && m >= 1) wait_bar_cluster(c, B_PFREE, (uint32_t)((m - 1) & 1));
        if (ZREC) wait_bar(c, B_SL0 + s, ph2);                 // Q<- (in A_chain[s]), K->, gamma^C of chunk n
        __syncwarp();
        if (PAIR) {
            // the other CTA forms its own [U ; P U] = Z V: send this warp's 16 rows of Z (the
            // products above only read the tile)
            const uint8_t *zt = base + OFF_KR;
            const uint32_t rbar = peer_base + OFF_MISC + MISC_BAR + 8u * B_RX;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const int id = lane + 32 * k4;
                const uint32_t off = sw128_offset(128, r0 + (id >> 3), (id & 7) * 8);
                const uint4 u = *reinterpret_cast<const uint4 *>(zt + off);
                st_async_u128(peer_base + OFF_ZIN + off, u.x, u.y, u.z, u.w, rbar);
            }
        }

        // ---------------- A_chain[s] = [-W ; Q<- - P W]  (K-major 128 x 128), 64 columns per thread
        {
            uint8_t *ach = base + off_ach(s);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int col = half * 64 + cc * 32;
                float v[32];
                if (!GLA) {
                    tmem_ld32(c.tmem + TM_WQ + lane_base + col, v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.f;
                }
                if (quarter < 2) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = -v[j];
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        // Q<-: rows 64-127 of A_G, or (records) of A_chain[s] itself, replaced in place
                        const uint4 u = *reinterpret_cast<const uint4 *>((ZREC ? ach : base + OFF_AG) +
                                                                         sw128_offset(128, row, col + 8 * q));
                        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[e]));
                            v[8 * q + 2 * e] = f.x - v[8 * q + 2 * e];
                            v[8 * q + 2 * e + 1] = f.y - v[8 * q + 2 * e + 1];
                        }
                    }
                }
                store_row32_bf16(ach, 128, row, col, v);
            }
        }
        // ---------------- K-> and gamma^C into slot s (and the other CTA's slot s)
        if constexpr (!ZREC) {
            const int cg = wt & 31, rg = wt >> 5;
            const int col = 4 * cg;
            uint8_t *kt = base + off_kt(s);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const uint32_t o64 = sw128_offset(64, rg * 8 + r, col);
                st_u64(kt + o64, krv[r]);
            }
            if (rg == 0) *reinterpret_cast<float4 *>(gC + s * kDK + col) = gcv;
        }
        if (!ZREC && wt < kC && n + step < nchunks) {
            betas[(sb ^ 1) * kC + wt] = nb;
            gss[(sb ^ 1) * kC + wt] = ng;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_sync(2, kWyThreads);
        if (leader) {
            mbar_arrive(c.bars + B_WYR0 + s);
            if (!ZREC && n + step < nchunks) issue_raw(n + step);   // A_G and the K<- tile are free again
            if (PAIR) {
                // the slot buffers go to the other CTA's slot s by bulk copy (it is done with
                // chunk n - 2: checked above)
                const uint32_t rbar = peer_base + OFF_MISC + MISC_BAR + 8u * B_RX;
                const uint32_t gc_off = OFF_MISC + MISC_GC + (uint32_t)s * 512u;
                mbar_arrive_expect_tx_remote(rbar, kPushBytes);
                bulk_copy_to_peer(peer_base + off_ach(s), base + off_ach(s), 32768u, rbar);
                bulk_copy_to_peer(peer_base + off_kt(s), base + off_kt(s), 16384u, rbar);
                bulk_copy_to_peer(peer_base + gc_off, base + gc_off, 512u, rbar);
            }
        }
        __syncwarp();                        // the leader's warp reaches the next barrier converged
    }
    // drain: every MMA this thread issued has completed before TMEM is freed
    if (leader) {
        mma_commit(c.bars + B_FIN1);
        wait_bar(c, B_FIN1, 0);
    }
    __syncwarp();
}

// ============================================================================
// Chain warps: the serial state scan and the output.
// ============================================================================
template <bool PAIR, bool ZREC>
__device__ void chain_role(const Ctx &c, const FwdParams &p, const CUtensorMap *tm_v, const CUtensorMap *tm_o,
                           int e0, int h, int b, Seq sq, int nchunks) {
    uint8_t *base = c.base;
    const int j = threadIdx.x;                  // key channel == TMEM lane
    const int warp = j >> 5;
    const bool leader = j == 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float *gC = reinterpret_cast<const float *>(base + OFF_MISC + MISC_GC);
    const int H = p.H, dv = p.dv;

    float S[kDVS];
#pragma unroll
    for (int e = 0; e < kDVS; ++e)
        S[e] = p.h0 ? p.h0[(((size_t)b * H + h) * dv + e0 + e) * kDK + j] : 0.f;

    auto write_state = [&]() {
        uint8_t *st = base + OFF_ST;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            st_u128(st + sw128_offset(128, j, q * 8), pack_bf16(S[8 * q], S[8 * q + 1]),
                    pack_bf16(S[8 * q + 2], S[8 * q + 3]), pack_bf16(S[8 * q + 4], S[8 * q + 5]),
                    pack_bf16(S[8 * q + 6], S[8 * q + 7]));
        fence_proxy_async_smem();
        tc_fence_before();
        named_sync(1, kChainThreads);
    };
    write_state();

    // With records the slot inputs of chunk n come straight from its record into slot n & 1:
    // Q<- into rows 64-127 of A_chain (the WY warps turn it into Q<- - P W in place), K-> and
    // gamma^C.  Issued once the slot's previous chunk is done with it, two chunks ahead.
    auto issue_slot = [&](int n) {
        const uint8_t *r = c.zrec + (size_t)n * c.zstride;
        const int sl = n & 1;
        uint64_t *bar = c.bars + B_SL0 + sl;
        mbar_arrive_expect_tx(bar, 2u * 16384u + 512u);
        for (int blk = 0; blk < 2; ++blk)
            bulk_load(base + off_ach(sl) + blk * 16384 + 8192, r + REC_Q + blk * 8192, 8192u, bar);
        bulk_load(base + off_kt(sl), r + REC_KR, 16384u, bar);
        bulk_load(base + OFF_MISC + MISC_GC + sl * 512, r + REC_GC, 512u, bar);
    };
    if (ZREC && leader) {
        issue_slot(0);
        if (nchunks > 1) issue_slot(1);
    }
    __syncwarp();

    for (int n = 0; n < nchunks; ++n) {
        const int s = n & 1;
        const uint32_t ph2 = (uint32_t)((n >> 1) & 1);
        const bool peer_chunk = PAIR && (n & 1) != (int)c.rank;
        if (peer_chunk) {
            // built by the other CTA: wait until its WY warps have written A_chain, K->, gamma^C
            // and Z here, and for this slice's v; [U ; P U] = Z V goes right before the state product
            if (leader) wait_bar(c, B_V0 + s, ph2);
            __syncwarp();
            wait_bar_cluster(c, B_RX, (uint32_t)((n >> 1) & 1));
            fence_proxy_async_smem();    // the received tiles are read by the tensor core next
        } else {
            wait_bar(c, B_WYR0 + s, ph2);
            if (ZREC) wait_bar(c, B_SL0 + s, ph2);      // gamma^C and K-> of the slot, loaded here
        }
        tc_fence_after();
        const float gam = gC[s * kDK + j];

        // ---- D1[s] (+)= [-W ; Q'] S^T   (M128 N64 K128)
        if (leader) {
            const uint32_t id = idesc_bf16(128, 64, 0, 1);
            if (peer_chunk) {
                const uint32_t az = smem_u32(base + OFF_ZIN), bv = smem_u32(base + off_v(s));
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(c.tmem + TM_D1 + s * 64, desc_kmajor(az, 128, ks), desc_mnmajor(bv, 64, ks), id,
                             ks > 0);
            }
            const uint32_t a0 = smem_u32(base + off_ach(s)), b0 = smem_u32(base + OFF_ST);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(c.tmem + TM_D1 + s * 64, desc_kmajor(a0, 128, ks), desc_mnmajor(b0, 128, ks), id, 1);
            mma_commit(c.bars + B_C10 + s);
        }
        __syncwarp();
        wait_bar(c, B_C10 + s, ph2);
        tc_fence_after();
        if (peer_chunk && leader && n + 2 < nchunks) {
            // v[s] has been read: fetch the slice of chunk n + 2
            mbar_arrive_expect_tx(c.bars + B_V0 + s, 8192u);
            tma_load_4d(base + off_v(s), tm_v, c.bars + B_V0 + s, e0, h, sq.t0 + (n + 2) * kC, sq.bt);
        }
        __syncwarp();

        // ---- rows 0-63: V_new -> bf16 MN-major B tile in the first half of the S^T tile (its
        //      product is done), then dS^T = K->^T V_new.  Rows 64-127: O -> staging tile, or,
        //      for the last chunk of a packed sequence, straight to its rows (a 64-row TMA store
        //      would run into the next sequence).
        const bool direct_o = p.cu_seqlens != nullptr && (n + 1) * kC > sq.len;
        {
            const int r = (warp & 1) * 32 + (j & 31);
            uint8_t *dst = base + (warp < 2 ? OFF_ST : OFF_OST);
            float v[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                tmem_ld32(c.tmem + TM_D1 + s * 64 + lane_base + cc * 32, v);
                if (warp >= 2 && direct_o) {
                    if (n * kC + r < sq.len) {
                        __nv_bfloat16 *orow =
                            static_cast<__nv_bfloat16 *>(p.o) +
                            (((size_t)sq.bt * p.T + sq.t0 + n * kC + r) * p.H + h) * p.dv + e0 + cc * 32;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4 *>(orow + 8 * q) =
                                make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                                           pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
                    }
                } else {
                    store_row32_bf16(dst, 64, r, cc * 32, v);
                }
            }
            fence_proxy_async_smem();
            if (warp < 2) {
                named_sync(3, 64);
                if (leader) {
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(base + off_kt(s)), b0 = smem_u32(base + OFF_ST);
                    const uint32_t id = idesc_bf16(128, 64, 1, 1);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(c.tmem + TM_S, desc_mnmajor(a0, 64, ks), desc_mnmajor(b0, 64, ks), id, ks > 0);
                    mma_commit(c.bars + B_C20 + s);
                }
                __syncwarp();
            }
        }
        tc_fence_before();
        named_sync(1, kChainThreads);
        if (leader) {
            tc_fence_after();
            mbar_arrive(c.bars + B_E10 + s);                        // D1[s] drained
            if (!direct_o) {
                tma_store_4d(tm_o, base + OFF_OST, e0, h, sq.t0 + n * kC, sq.bt);
                tma_store_commit();
            }
        }
        __syncwarp();
        wait_bar(c, B_C20 + s, ph2);
        tc_fence_after();
        if (ZREC && leader && n + 2 < nchunks) issue_slot(n + 2);   // slot s: both products are done
        __syncwarp();
        {
            float v[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                tmem_ld32(c.tmem + TM_S + lane_base + cc * 32, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) S[cc * 32 + e] = gam * (S[cc * 32 + e] + v[e]);
            }
        }
        if (leader) tma_store_wait_read0();                       // staging tile free for the next chunk
        __syncwarp();
        write_state();
        if (peer_chunk && leader)                                  // done with the other CTA's chunk n
            mbar_arrive_remote(map_to_rank(smem_u32(c.bars + B_PFREE), c.rank ^ 1u));
    }
    if (p.ht) {
#pragma unroll
        for (int e = 0; e < kDVS; ++e) p.ht[(((size_t)b * H + h) * dv + e0 + e) * kDK + j] = S[e];
    }
    if (leader) {
        tma_store_wait_all0();
        mma_commit(c.bars + B_FIN0);
        wait_bar(c, B_FIN0, 0);
    }
    __syncwarp();
}

template <int GATE, bool GLA, bool PAIR, bool ZREC, typename Tg>
__global__ void __launch_bounds__(kThreads, 1)
kda_fwd_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_g,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o) {
    static_assert(!(PAIR && ZREC), "with records each value slice builds every chunk itself");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctx c;
    c.base = base;
    c.bars = reinterpret_cast<uint64_t *>(base + OFF_MISC + MISC_BAR);
    c.abort = reinterpret_cast<volatile int *>(base + OFF_MISC + MISC_ABORT);
    c.status = p.status;
    c.rank = PAIR ? cluster_ctarank() : 0u;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + OFF_MISC + MISC_TSLOT);

    const int e0 = blockIdx.x * kDVS, h = blockIdx.y, b = blockIdx.z;
    const Seq sq = seq_of(p, b);
    const int nchunks = (sq.len + kC - 1) / kC;
    c.zrec = ZREC ? p.zrec + ((size_t)zslot0(p, b, sq) * p.H + h) * kRecBytes : nullptr;
    c.zstride = (size_t)p.H * kRecBytes;
    if (nchunks == 0) {                     // empty sequence: ht = h0; nothing else is set up
        if (p.ht)
            for (int i = threadIdx.x; i < kDVS * kDK; i += kThreads) {
                const size_t off = (((size_t)b * p.H + h) * p.dv + e0 + i / kDK) * kDK + i % kDK;
                p.ht[off] = p.h0 ? p.h0[off] : 0.f;
            }
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(c.bars + i, 1);
        *c.abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(tslot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();           // the peer's barriers exist before any remote access
    tc_fence_after();
    c.tmem = *tslot;

    if (threadIdx.x < kChainThreads)
        chain_role<PAIR, ZREC>(c, p, &tm_v, &tm_o, e0, h, b, sq, nchunks);
    else
        wy_role<GATE, GLA, PAIR, ZREC, Tg>(c, p, &tm_q, &tm_k, &tm_g, &tm_v, e0, h, sq, nchunks);

    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();           // no remote access into a CTA that has exited
    tc_fence_after();
    if (threadIdx.x < 32) tmem_dealloc(c.tmem, kTmemCols);
}

// ============================================================================
// Z records: the part of every chunk that needs the Gram and the inverse,
// chunk-parallel ahead of the scan kernel.
// ============================================================================
// One CTA per (chunk, head, sequence) computes Gamma, the rescaled tiles and
// Z = [T ; P T] (GLA: [I ; P]) with the scan kernel's own code (rescale_tiles,
// build_z) and stores Z as the 16 KB image of the bf16 tile that the scan
// kernel's products read, so that kernel loads it with one bulk copy instead
// of building it.  Shared memory: the A_G and K-> tiles at the scan kernel's
// offsets (raw k lands in the K-> tile and becomes K-> in place), then the
// scalars, the cumsum partials and the barriers.
constexpr uint32_t OFF_WMISC = 49152;
constexpr uint32_t WM_BETA = 0;          // beta [64] f32
constexpr uint32_t WM_GS = 256;          // scalar gate [64] f32
constexpr uint32_t WM_TOT = 512;         // cumsum partials [8][128] f32
constexpr uint32_t WM_BAR = 4608;        // mbarriers [kNumBars] u64
constexpr uint32_t WM_TSLOT = 4800;      // TMEM base address
constexpr uint32_t WM_ABORT = 4804;      // abort flag
constexpr uint32_t kWMiscBytes = 4864;
constexpr uint32_t kZSmemBytes = OFF_WMISC + kWMiscBytes + 1024;
constexpr uint32_t kZTmemCols = 64;      // the Gram [L ; P]
static_assert(OFF_KR + 16384 <= OFF_WMISC, "Z kernel tile layout");
static_assert(WM_BAR + kNumBars * 8 <= WM_TSLOT, "Z kernel misc layout");
static_assert(WM_ABORT + 4 <= kWMiscBytes, "Z kernel misc layout");

template <int GATE, bool GLA, typename Tg>
__global__ void __launch_bounds__(kWyThreads, 4)
kda_fwd_z_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int n = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const Seq sq = seq_of(p, b);
    if (n * kC >= sq.len) return;           // past the end of this sequence (or an empty one)
    const int wt = threadIdx.x;
    Ctx c;
    c.base = base;
    c.bars = reinterpret_cast<uint64_t *>(base + OFF_WMISC + WM_BAR);
    c.abort = reinterpret_cast<volatile int *>(base + OFF_WMISC + WM_ABORT);
    c.status = p.status;
    c.rank = 0;
    c.zrec = nullptr;
    c.zstride = 0;
    float *betas = reinterpret_cast<float *>(base + OFF_WMISC + WM_BETA);
    float *gss = reinterpret_cast<float *>(base + OFF_WMISC + WM_GS);
    float *tot = reinterpret_cast<float *>(base + OFF_WMISC + WM_TOT);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + OFF_WMISC + WM_TSLOT);
    const int T = p.T, H = p.H;

    if (wt == 0) {
        mbar_init(c.bars + B_RAW, 1);
        mbar_init(c.bars + B_GRAM, 1);
        *c.abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (wt < 32) {
        tmem_alloc(tslot, kZTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = *tslot;

    if (wt == 0) {
        // raw g -> A_G rows 0-63, raw q -> A_G rows 64-127, raw k -> the K-> tile
        mbar_arrive_expect_tx(c.bars + B_RAW, (GATE == KDA_GATE_CHANNEL ? 3u : 2u) * 16384u);
        for (int blk = 0; blk < 2; ++blk) {
            tma_load_4d(base + OFF_AG + blk * 16384 + 8192, &tm_q, c.bars + B_RAW, blk * 64, h, sq.t0 + n * kC, sq.bt);
            tma_load_4d(base + OFF_KR + blk * 8192, &tm_k, c.bars + B_RAW, blk * 64, h, sq.t0 + n * kC, sq.bt);
            if (GATE == KDA_GATE_CHANNEL)
                tma_load_4d(base + OFF_AG + blk * 16384, &tm_g, c.bars + B_RAW, blk * 64, h, sq.t0 + n * kC, sq.bt);
        }
    }
    __syncwarp();
    if (wt < kC) {
        float bv = 0.f, gv = 0.f;
        const int t = n * kC + wt;
        if (t < sq.len) {
            const size_t row = ((size_t)sq.bt * T + sq.t0 + t) * H + h;
            if (p.has_beta) bv = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.beta)[row]);
            if (GATE == KDA_GATE_SCALAR) gv = ldg_f<Tg>(static_cast<const Tg *>(p.g) + row);
        }
        betas[wt] = bv;
        gss[wt] = gv;
    }
    wait_bar(c, B_RAW, 0);
    __syncthreads();                        // the scalars

    uint8_t *rec = p.zrec + ((size_t)(zslot0(p, b, sq) + n) * H + h) * kRecBytes;
    uint2 krv[8];
    float4 gcv;
    rescale_tiles<GATE, true, false>(base, OFF_KR, wt, sq.len - n * kC, betas, gss, tot, krv, gcv, rec);
    fence_proxy_async_smem();
    __syncthreads();
    build_z<GLA>(c, wt, betas, 0);
    fence_proxy_async_smem();               // the Z stores, before the bulk copy reads them
    __syncthreads();
    if (wt == 0) {
        bulk_store(rec + REC_Z, base + OFF_KR, 16384u);
        tma_store_commit();
        tma_store_wait_read0();             // shared memory may go once the copy has read it
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (wt < 32) tmem_dealloc(c.tmem, kZTmemCols);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// [B, T, H, D] tensor as a 4-D map (D, H, T, B) with 64 x 1 x 64 x 1 boxes, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, uint32_t es, int B, int T, int H, int D) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * es, (cuuint64_t)H * D * es, (cuuint64_t)T * H * D * es};
    cuuint32_t box[4] = {64, 1, 64, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, dt, 4, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int GATE, bool GLA, bool ZREC, typename Tg>
cudaError_t launch_scan(const FwdParams &p, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &g,
                        const CUtensorMap &v, const CUtensorMap &o, cudaStream_t s) {
    // Without records the two value slices of a head split the chunks they build (a pair);
    // with records building a chunk is light, and each slice builds every chunk itself.
    dim3 grid(p.dv / kDVS, p.H, p.B);
    if constexpr (!ZREC) {
      if (p.dv == 2 * kDVS) {
        auto kern = kda_fwd_tc_kernel<GATE, GLA, true, false, Tg>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, p, q, k, g, v, o);
      }
    }
    auto kern = kda_fwd_tc_kernel<GATE, GLA, false, ZREC, Tg>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kSmemBytes, s>>>(p, q, k, g, v, o);
    return cudaGetLastError();
}

// With Z records (p.zrec set): the chunk-parallel Z kernel, then the scan
// kernel that loads Z; otherwise the scan kernel alone, building Z itself.
template <int GATE, bool GLA, typename Tg>
cudaError_t launch_variant(const FwdParams &p, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &g,
                           const CUtensorMap &v, const CUtensorMap &o, cudaStream_t s) {
    if (!p.zrec) return launch_scan<GATE, GLA, false, Tg>(p, q, k, g, v, o, s);
    auto zk = kda_fwd_z_kernel<GATE, GLA, Tg>;
    cudaError_t e = cudaFuncSetAttribute(zk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kZSmemBytes);
    if (e != cudaSuccess) return e;
    zk<<<dim3((p.T + kC - 1) / kC, p.H, p.B), kWyThreads, kZSmemBytes, s>>>(p, q, k, g);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_scan<GATE, GLA, true, Tg>(p, q, k, g, v, o, s);
}

}  // namespace

size_t fwd_zrec_bytes(int B, int T, int H, bool packed) {
    const size_t nc = (size_t)(T + kC - 1) / kC;
    return (packed ? (size_t)B + nc : (size_t)B * nc) * (size_t)H * kRecBytes;
}

cudaError_t launch_fwd_tc_bf16(const FwdParams &p, int g_is_bf16, cudaStream_t s) {
    if (p.dk != kDK || (p.dv != kDVS && p.dv != 2 * kDVS)) return cudaErrorNotSupported;
    const bool gla = !p.scale_v;
    if (gla && p.has_beta) return cudaErrorNotSupported;     // unscaled v with a delta term: DPLR entry
    if (p.gate_kind == KDA_GATE_CHANNEL && !g_is_bf16) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mg, mv, mo;
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int mb = p.cu_seqlens ? 1 : p.B;          // packed sequences: one [1, T, H, d] tensor
    if (!make_map(&mq, p.q, bf, 2, mb, p.T, p.H, p.dk) || !make_map(&mk, p.k, bf, 2, mb, p.T, p.H, p.dk) ||
        !make_map(&mv, p.v, bf, 2, mb, p.T, p.H, p.dv) || !make_map(&mo, p.o, bf, 2, mb, p.T, p.H, p.dv))
        return cudaErrorInvalidValue;
    mg = mq;
    if (p.gate_kind == KDA_GATE_CHANNEL && !make_map(&mg, p.g, bf, 2, mb, p.T, p.H, p.dk))
        return cudaErrorInvalidValue;
    if (p.gate_kind == KDA_GATE_CHANNEL) {
        return gla ? launch_variant<KDA_GATE_CHANNEL, true, __nv_bfloat16>(p, mq, mk, mg, mv, mo, s)
                   : launch_variant<KDA_GATE_CHANNEL, false, __nv_bfloat16>(p, mq, mk, mg, mv, mo, s);
    }
    if (p.gate_kind == KDA_GATE_SCALAR) {
        if (gla) return cudaErrorNotSupported;
        return g_is_bf16 ? launch_variant<KDA_GATE_SCALAR, false, __nv_bfloat16>(p, mq, mk, mg, mv, mo, s)
                         : launch_variant<KDA_GATE_SCALAR, false, float>(p, mq, mk, mg, mv, mo, s);
    }
    if (gla) return cudaErrorNotSupported;
    return launch_variant<KDA_GATE_NONE, false, __nv_bfloat16>(p, mq, mk, mg, mv, mo, s);
}

}  // namespace kda
