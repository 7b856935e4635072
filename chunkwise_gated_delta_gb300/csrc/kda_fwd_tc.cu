// tcgen05 kernels for the chunkwise KDA forward (bf16 in, fp32 accumulate,
// fp32 state), GB300 / sm_103a.
//
// The chunk form evaluated is the one recapped on page "Kimi Delta Attention
// backward" ("forward recap"), regrouped so every tensor-core product has
// M = 128 rows:
//
//   [beta K<- ; Q<-] K->^T      = [L ; P]          (Gram, one MMA; a chunk whose decay
//                                                    K-> cannot represent takes the sub-chunk
//                                                    form of "Gated Linear Attention" 5.3)
//   Z' (I + L_{strict}) = [I ; P],  Z = Z' Diag(beta) = [T ; P T]
//        with T = (I + L)^{-1} Diag(beta): block back-substitution over
//        16-column blocks (page "DeltaNet" 4.2, block form 2), the 16x16
//        diagonal blocks inverted by warp shuffles, the block products as
//        tf32 warp MMAs, 16 rows of Z' per warp
//   Z K<-                       = [W ; P W]
//   Z V                         = [U ; P U]        (into the accumulator D1)
//   D1 += [-W ; Q<- - P W] S^T  = [V_new ; O]      (state-dependent, one MMA)
//   K->^T V_new                 = dS^T,  S <- (S + dS) Diag(gamma^C)   (single kernel)
//   K~^T V_new                  = dS^T,  S <- S Diag(gamma^C) + dS     (records, and a chunk
//                                        past K->'s range),  K~ = K-> Diag(gamma^C)
//
// O = Q<- S^T + (Q<- K->^T * M) V_new expands to (Q<- - P W) S^T + P U, which
// is why the output rides in the lower half of the state-dependent product;
// the state step uses the factored form of page "Gated Linear Attention" 5.2
// (K~ = K exp(G_C - G) is bounded by |K| at any decay).
//
// Two forms.
//   Records (two kernels, when the caller's workspace holds them): the
//   chunk-parallel Z kernel computes, for every chunk, Gamma, the rescaled
//   tiles, Z, [W ; P W] and A_chain = [-W ; Q<- - P W] -- everything that
//   does not depend on the state -- and writes the bf16 tile images of Z,
//   A_chain and K~ and gamma^C as the chunk's record.  The record scan
//   kernel then runs one CTA per (batch, head, 64-wide value slice) and takes
//   three products per chunk (Z V, A_chain S^T, K~^T V_new).
//   Single kernel (a 256-byte workspace, or batches that fill one wave): one
//   CTA per (batch, head, 64-wide value slice) walks its chunks in order with
//   two warp roles (384 threads): warps 0-3 "chain", the serial part -- the
//   state S^T (128 key channels x 64 values) in fp32 registers, one key
//   channel per thread; warps 4-11 "WY", everything that does not depend on
//   S, Z included.  With dv = 128 the two value-slice CTAs of a head form a
//   cluster and split the WY work by chunk parity: CTA r builds the chunks n
//   with n % 2 == r and copies their slot tiles (A_chain, K->, gamma^C) and Z
//   into the other CTA's shared memory; each CTA still runs the state scan of
//   every chunk for its own value slice and forms its own [U ; P U] = Z V.
//   With dv = 64 one CTA does it all.
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
constexpr uint32_t OFF_KT0 = 147456;     // K-> (or K~) 64 x 128 (MN-major A of dS), slot 0
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
// One chunk's record (Z kernel -> record scan kernel): images of the bf16 tiles whose
// products the scan forms, plus gamma^C.
constexpr uint32_t REC_Z = 0;            // Z = [T ; P T], K-major 128 x 64 (A of Z V)
constexpr uint32_t REC_A = 16384;        // A_chain = [-W ; Q<- - P W], K-major 128 x 128 (A of A_chain S^T)
constexpr uint32_t REC_KR = 49152;       // K~ = K exp(G_C - G), 64 x 128 (MN-major A of K~^T V_new)
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
    B_RX, B_PFREE, B_FIN0, B_FIN1, B_RAWK, B_RAWQ, B_STRONG, kNumBars
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
    uint32_t bound;    // polling iterations a bounded wait takes before it gives up
    bool short_polls;  // a caller's budget: each poll suspends for at most kShortPollNs
    uint32_t rank;     // rank in the pair (0 without a pair)
    const uint8_t *zrec;   // record of chunk 0 of this (sequence, head); chunk n at zrec + n * zstride
    size_t zstride;
};

// A wait ran out: the CTA stops waiting, and the status word says so.  The
// first wait to run out in the launch also leaves where it was in the next
// words of the status block: barrier index + 1, parity, thread, block (x, y, z
// in bytes 0-2).
__device__ __forceinline__ void record_timeout(volatile int *abort, int *status, int idx, uint32_t parity) {
    *abort = 1;
    atomicCAS(status, kDevOk, kDevTimeout);
    if (atomicCAS(status + 1, 0, idx + 1) == 0) {
        status[2] = (int)parity;
        status[3] = (int)threadIdx.x;
        status[4] = (int)(blockIdx.x | (blockIdx.y << 8) | (blockIdx.z << 16));
    }
}
// A wait given up because another thread of the CTA gave up: the two issuing threads (chain
// leader 0, WY leader 128) leave the barrier they were on in words 5 and 6.
__device__ __forceinline__ void note_abort(int *status, int idx, uint32_t parity) {
    if (threadIdx.x == 0) atomicCAS(status + 5, 0, idx + 1 + 256 * (int)parity);
    if (threadIdx.x == kChainThreads) atomicCAS(status + 6, 0, idx + 1 + 256 * (int)parity);
}

// Bounded wait that becomes a no-op once any thread of the CTA has given up.  The
// first probe is inline: most waits end within it, and a call to the out-of-line
// loop would move the caller's live registers through local memory.  Probes use
// try_wait, which suspends the thread until the phase completes or a hardware time
// limit passes; under a caller's budget the first probe does not block and each
// later poll suspends for at most kShortPollNs, so the budget counts short polls.
// The out-of-line loops take plain values, not the context: a reference to it would
// keep the context in local memory for every inline use.
constexpr uint32_t kShortPollNs = 32;
// Returns whether the phase completed (false: the wait gave up, or another thread had).
__device__ __noinline__ bool wait_bar_slow(uint64_t *bars, volatile int *abort, int *status, uint32_t bound,
                                           bool short_polls, int idx, uint32_t parity) {
    uint64_t *bar = bars + idx;
    for (uint32_t i = 0; i < bound; ++i) {
        if (short_polls ? mbar_try_wait_for(bar, parity, kShortPollNs) : mbar_try_wait(bar, parity)) return true;
        if (*abort) {
            note_abort(status, idx, parity);
            return false;
        }
    }
    record_timeout(abort, status, idx, parity);
    return false;
}
__device__ __forceinline__ bool wait_bar(const Ctx &c, int idx, uint32_t parity) {
    uint64_t *bar = c.bars + idx;
    if (c.short_polls ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(c.bars, c.abort, c.status, c.bound, c.short_polls, idx, parity);
}

// Wait for a phase that an asynchronous operation this thread started completes -- a copy into
// shared memory, a commit of tensor-core products -- whatever the abort flag says: nothing may
// still write this CTA's shared memory or TMEM when it frees TMEM or exits.  These operations
// complete by themselves, so the library's default bound applies (never the caller's budget);
// running out is recorded like any other timeout.
__device__ __noinline__ void drain_bar_slow(uint64_t *bar, volatile int *abort, int *status, int idx,
                                            uint32_t parity) {
    for (uint32_t i = 0; i < kWaitBound; ++i)
        if (mbar_try_wait(bar, parity)) return;
    record_timeout(abort, status, idx, parity);
}
__device__ __forceinline__ void drain_bar(const Ctx &c, int idx, uint32_t parity) {
    if (!mbar_try_wait(c.bars + idx, parity)) drain_bar_slow(c.bars + idx, c.abort, c.status, idx, parity);
}
__device__ __noinline__ void drain_bar_cluster_slow(uint64_t *bar, volatile int *abort, int *status, int idx,
                                                    uint32_t parity) {
    for (uint32_t i = 0; i < kWaitBound; ++i)
        if (mbar_try_wait_cluster(bar, parity)) return;
    record_timeout(abort, status, idx, parity);
}
__device__ __forceinline__ void drain_bar_cluster(const Ctx &c, int idx, uint32_t parity) {
    if (!mbar_try_wait_cluster(c.bars + idx, parity))
        drain_bar_cluster_slow(c.bars + idx, c.abort, c.status, idx, parity);
}
// The budget of the bounded waits: word kStatusBoundWord of the status block, or the default.
__device__ __forceinline__ uint32_t wait_bound_of(const int *status) {
    const int b = status[kStatusBoundWord];
    return b > 0 ? (uint32_t)b : kWaitBound;
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// A named barrier that also returns whether `pred` held in any of its threads.
__device__ __forceinline__ bool named_sync_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void st_u128(uint8_t *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
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
// Record slot of chunk 0 of sequence b.  Dense: b * ceil(T / C).  Packed:
// b + floor(t0 / C), which never collides with the next sequence's slots
// (floor(t0 / C) + ceil(len / C) <= floor((t0 + len) / C) + 1), so B + ceil(T / C)
// slots per head cover every packing.
__device__ __forceinline__ int zslot0(const FwdParams &p, int b, const Seq &sq) {
    return p.cu_seqlens ? b + sq.t0 / kC : b * ((p.T + kC - 1) / kC);
}

// ---- Gamma and the rescaled tiles of one chunk, in place.  Raw g (channel
// gate) sits in A_G rows 0-63, raw q in A_G rows 64-127 and raw k in the
// 64-row tile at `kraw`.  Q<- replaces the raw q; GRAM: beta K<- goes to A_G
// rows 0-63 and K-> to the K-> tile (the Gram's operands); SCAN: K<- goes to
// the K<- tile.  Rows at or past `live_rows` are zero; `bet` and `gs` hold the
// chunk's beta and scalar gate.  The 256 WY threads (index wt): warp w owns
// rows 8w .. 8w + 7, its lanes 16 column groups of 8 (one 16-byte piece of a
// swizzled row) by 2 row halves, so every load and store moves 16 bytes and
// the in-chunk cumsum is a 4-row sum, one shuffle and one exchange of warp
// totals through `tot` (one barrier).  SCAN: K-> of the thread's 4 rows comes
// back in `krv` for the chunk's slot; the thread holding row 63 (`has_gam`)
// also returns gamma^C of its 8 columns in `gam`.
//   REC (the Z kernel of the record form): A_G rows 0-63 get K<- itself (beta is
// applied to the rows of L instead, so the tile is also the B operand of Z K<-),
// and K~ = K exp(G_C - G) and gamma^C go straight to the chunk record `rec`.
//   Returns whether this thread saw a column whose decay K-> cannot represent
// (G_C below -kFastLog2): the callers vote on it at their next barrier, and a
// chunk so marked is done again by strong_prologue.  STRONG (that second pass):
// K-> is not formed (its tile gets zeros), K~ is formed directly and goes to
// `krv` in place of K->, and every thread returns gamma^C in `gam`.
__device__ __forceinline__ void unpack_bf16x8(const uint4 u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ uint4 pack_bf16x8(const float (&x)[8]) {
    return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}

// Largest in-chunk log-decay magnitude (base 2) the rescaled tiles of the one-product Gram
// represent: K-> = K 2^{-G} and the products of K-> stay finite in fp32 with a margin of 2^28
// for the sums.  G_C, the chunk's total, is the extreme of G for g <= 0; a chunk whose G_C is
// below -kFastLog2 in any channel takes the sub-chunk Gram (strong_gram) instead.
constexpr float kFastLog2 = 100.f;

template <int GATE, bool GRAM, bool SCAN, bool REC, bool STRONG, typename PreQK>
__device__ __forceinline__ bool rescale_tiles(uint8_t *base, uint32_t kraw, int wt, int live_rows, const float *bet,
                                              const float *gs, float *tot, uint4 (&krv)[4], float (&gam)[8],
                                              bool &has_gam, PreQK &&pre_qk, uint8_t *rec = nullptr) {
    const int w = wt >> 5, lane = wt & 31;
    const int cq = lane & 15, rsub = lane >> 4;
    const int r0 = 8 * w + 4 * rsub;                 // first of the thread's 4 rows
    const int col = 8 * cq;                          // first of its 8 columns
    // byte offset of (r0 + i, col) in a 64-row / 128-row swizzled tile: r0 & 7 == 4 rsub
    const uint32_t sw = (uint32_t)((cq & 7) ^ (4 * rsub));
    const uint32_t o64 = (uint32_t)(cq >> 3) * 8192u + (uint32_t)r0 * 128u;
    const uint32_t o128 = (uint32_t)(cq >> 3) * 16384u + (uint32_t)r0 * 128u;
    auto off64 = [&](int i) { return o64 + (uint32_t)i * 128u + ((sw ^ (uint32_t)i) << 4); };
    auto off128 = [&](int i) { return o128 + (uint32_t)i * 128u + ((sw ^ (uint32_t)i) << 4); };

    constexpr bool ALLGC = REC || STRONG;            // every thread needs G_C of its columns
    float G[4][8];                                   // in-chunk cumsum of g, base-2 units, this thread's rows
    float gc2[8];                                    // ALLGC: G_C of this thread's columns, base 2
    bool strong_here = false;                        // a column of this thread past the fast form's range
    has_gam = (w == 7 && rsub == 1);
    if constexpr (GATE == KDA_GATE_NONE) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) G[i][e] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) { gam[e] = 1.f; gc2[e] = 0.f; }
    } else {
        float a[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = r0 + i;
            float x[8];
            if (GATE == KDA_GATE_CHANNEL) {
                const uint4 u = row < live_rows ? *reinterpret_cast<const uint4 *>(base + OFF_AG + off128(i))
                                                : make_uint4(0u, 0u, 0u, 0u);
                unpack_bf16x8(u, x);
            } else {
                const float s = row < live_rows ? gs[row] : 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = s;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) { a[e] += x[e]; G[i][e] = a[e]; }
        }
        // the lower half-warp (rows + 4) adds the upper half's 4-row total; lanes 16-31 then hold
        // the warp's 8-row total, which goes to the other warps through `tot`
        float pre[8], rest[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float own = a[e];                  // this thread's 4-row sum
            const float up = __shfl_up_sync(0xffffffffu, own, 16);
            pre[e] = rsub ? up : 0.f;
            a[e] = own + pre[e];                     // lanes 16-31: the warp's 8-row total
            // what the chunk adds after this thread's last row, starting with the lower
            // half-warp's rows for the upper half (the warp total from lanes 16-31 less its own)
            const float dn = __shfl_down_sync(0xffffffffu, a[e], 16);
            rest[e] = rsub ? 0.f : dn - own;
        }
        if (rsub) {
            *reinterpret_cast<float4 *>(tot + w * kDK + col) = make_float4(a[0], a[1], a[2], a[3]);
            *reinterpret_cast<float4 *>(tot + w * kDK + col + 4) = make_float4(a[4], a[5], a[6], a[7]);
        }
        named_sync(2, kWyThreads);
        for (int q = 0; q < w; ++q) {                // warp-uniform bound
            const float4 t0 = *reinterpret_cast<const float4 *>(tot + q * kDK + col);
            const float4 t1 = *reinterpret_cast<const float4 *>(tot + q * kDK + col + 4);
            pre[0] += t0.x; pre[1] += t0.y; pre[2] += t0.z; pre[3] += t0.w;
            pre[4] += t1.x; pre[5] += t1.y; pre[6] += t1.z; pre[7] += t1.w;
        }
        if (ALLGC) {
            for (int q = w + 1; q < 8; ++q) {        // warp-uniform bound
                const float4 t0 = *reinterpret_cast<const float4 *>(tot + q * kDK + col);
                const float4 t1 = *reinterpret_cast<const float4 *>(tot + q * kDK + col + 4);
                rest[0] += t0.x; rest[1] += t0.y; rest[2] += t0.z; rest[3] += t0.w;
                rest[4] += t1.x; rest[5] += t1.y; rest[6] += t1.z; rest[7] += t1.w;
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float p2 = pre[e] * kLog2e;
            // G_C, the chunk's total log-decay (base 2): this thread's running sum plus the rest
            gc2[e] = fmaf(G[3][e] + rest[e], kLog2e, p2);
#pragma unroll
            for (int i = 0; i < 4; ++i) G[i][e] = fmaf(G[i][e], kLog2e, p2);
            // ALLGC: every thread; else the one holding row 63, whose G[3] is G_C
            const float gce = ALLGC ? gc2[e] : G[3][e];
            gam[e] = ex2_approx(gce);
            strong_here |= (ALLGC || has_gam) && gce < -kFastLog2;
        }
    }
    if (REC && has_gam) {
        *reinterpret_cast<float4 *>(rec + REC_GC + 4 * col) = make_float4(gam[0], gam[1], gam[2], gam[3]);
        *reinterpret_cast<float4 *>(rec + REC_GC + 4 * col + 16) = make_float4(gam[4], gam[5], gam[6], gam[7]);
    }
    pre_qk();                                        // q and k may land later than g
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool live = r0 + i < live_rows;
        const uint4 uq = live ? *reinterpret_cast<const uint4 *>(base + OFF_AG + off128(i) + 8192u)
                              : make_uint4(0u, 0u, 0u, 0u);
        const uint4 uk = live ? *reinterpret_cast<const uint4 *>(base + kraw + off64(i)) : make_uint4(0u, 0u, 0u, 0u);
        float qv[8], kv[8], kl[8], kr[8], ql[8], kt[8];
        unpack_bf16x8(uq, qv);
        unpack_bf16x8(uk, kv);
        const float bb = (REC || !GRAM) ? 1.f : bet[r0 + i];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if constexpr (GATE == KDA_GATE_NONE) {
                kl[e] = kv[e]; kr[e] = kv[e]; ql[e] = qv[e]; kt[e] = kv[e];
            } else {
                const float ev = ex2_approx(G[i][e]);
                kl[e] = kv[e] * ev;
                ql[e] = qv[e] * ev;
                // K~ = K exp(G_C - G): K-> gamma^C where K-> is finite, else directly
                if (!STRONG) {
                    kr[e] = kv[e] * ex2_approx(-G[i][e]);
                    if (REC) kt[e] = kr[e] * gam[e];
                } else {
                    kr[e] = 0.f;
                    kt[e] = kv[e] * ex2_approx(gc2[e] - G[i][e]);
                }
            }
        }
        const uint4 krp = pack_bf16x8(kr);
        *reinterpret_cast<uint4 *>(base + OFF_AG + off128(i) + 8192u) = pack_bf16x8(ql);
        if (GRAM) {
            float bk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) bk[e] = bb * kl[e];
            *reinterpret_cast<uint4 *>(base + OFF_AG + off128(i)) = pack_bf16x8(bk);
            *reinterpret_cast<uint4 *>(base + OFF_KR + off64(i)) = krp;
        }
        if (SCAN) *reinterpret_cast<uint4 *>(base + OFF_KL + off64(i)) = pack_bf16x8(kl);
        if (SCAN) krv[i] = STRONG ? pack_bf16x8(kt) : krp;
        if (REC) *reinterpret_cast<uint4 *>(rec + REC_KR + off64(i)) = pack_bf16x8(kt);
    }
    return strong_here;
}
// Slot image of the rows a thread of rescale_tiles produced (its 4 rows x 8 columns) and, from
// the thread that holds row 63, gamma^C of its 8 columns.  The rows are K->, or K~ for a chunk
// that took the sub-chunk Gram (`strong`), which the chain learns from the sign bit of gamma^C
// (stored negated; -0 where gamma^C underflows).
__device__ __forceinline__ void store_kr_slot(uint8_t *kt, float *gc, int wt, const uint4 (&krv)[4],
                                              const float (&gam)[8], bool has_gam, bool strong) {
    const int w = wt >> 5, lane = wt & 31;
    const int cq = lane & 15, rsub = lane >> 4;
    const int r0 = 8 * w + 4 * rsub;
    const uint32_t sw = (uint32_t)((cq & 7) ^ (4 * rsub));
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4 *>(kt + (uint32_t)(cq >> 3) * 8192u + (uint32_t)(r0 + i) * 128u +
                                   ((sw ^ (uint32_t)i) << 4)) = krv[i];
    if (has_gam) {
        const float sg = strong ? -1.f : 1.f;
        *reinterpret_cast<float4 *>(gc + 8 * cq) = make_float4(sg * gam[0], sg * gam[1], sg * gam[2], sg * gam[3]);
        *reinterpret_cast<float4 *>(gc + 8 * cq + 4) =
            make_float4(sg * gam[4], sg * gam[5], sg * gam[6], sg * gam[7]);
    }
}

// ---- Fragment images of the block back-substitution's B operands: tf32
// values in the order the warp MMAs read them, 256 floats per 16x16 block
// ([k-step][n-half][lane][2]).  The k index of every 8-wide k-step is taken
// in the order 0, 2, 4, 6 | 1, 3, 5, 7 (slot t holds k = 2t, slot t + 4 holds
// k = 2t + 1), which makes an accumulator fragment (row g, columns 2t, 2t + 1)
// the A fragment of the next product as it stands: no shuffles.
__device__ __forceinline__ int frag_pos(int r, int cc) {   // element (r, cc) of a 16x16 block
    return (((r >> 3) * 2 + (cc >> 3)) * 32 + 4 * (cc & 7) + ((r & 7) >> 1)) * 2 + (r & 1);
}
// Accumulator fragment of a 16x8 half (columns 2t, 2t + 1 of rows g, g + 8) as the
// k-permuted tf32 A fragment of one k-step, times `sign`.
__device__ __forceinline__ void acc_as_a(const float (&x)[4], uint32_t (&a)[4], float sign) {
    a[0] = to_tf32(sign * x[0]);
    a[1] = to_tf32(sign * x[2]);
    a[2] = to_tf32(sign * x[1]);
    a[3] = to_tf32(sign * x[3]);
}
__device__ __forceinline__ void stmatrix_x4(uint32_t addr, const uint32_t (&r)[4]) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

// ---- Z = [T ; P T] of one chunk (GLA: [I ; P]) from its rescaled tiles, as a
// bf16 K-major 128 x 64 tile in the K-> tile: the Gram [beta K<- ; Q<-] K->^T
// into TMEM, L and the inverses of its 16x16 diagonal blocks, the block
// back-substitution, the beta scaling.  The 256 WY threads enter after the
// barrier that follows their stores of the rescaled tiles; `ph` is the parity
// of the Gram barrier.  `yfrag` (4 KB, free by then) receives the diagonal-block
// inverses and the K-> tile, dead after the Gram, the off-diagonal blocks of L,
// both as fragment images.  Returns the first of the 16 Z rows this warp wrote;
// ends without a barrier.
//   REC: rows 0-63 of the Gram are K<- K->^T (A_G holds K<-, not beta K<-), so
// beta scales them as they leave TMEM.
//   strong: the sub-chunk Gram is already in TMEM; the Gram barrier is committed with no product,
// so that its phases stay one per chunk.
template <bool GLA, bool REC = false>
__device__ int build_z(const Ctx &c, int wt, const float *bet, uint32_t ph, float *yfrag, bool strong) {
    uint8_t *base = c.base;
    const int ww = wt >> 5, lane = wt & 31;
    const int quarter = ww & 3, half = ww >> 2;
    const bool leader = wt == 0;
    float *lfrag = reinterpret_cast<float *>(base + OFF_KR);
    // ---------------- Gram: D_G = [beta K<- ; Q<-] K->^T   (M128 N64 K128)
    if (leader) {
        tc_fence_after();
        if (!strong) {
            const uint32_t a0 = smem_u32(base + OFF_AG), b0 = smem_u32(base + OFF_KR);
            const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(c.tmem + TM_G, desc_kmajor(a0, 128, ks), desc_kmajor(b0, 64, ks), id, ks > 0);
        }
        mma_commit(c.bars + B_GRAM);
    }
    __syncwarp();
    wait_bar(c, B_GRAM, ph);
    tc_fence_after();
    __syncwarp();                            // the TMEM loads below are warp-collective

    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int row = quarter * 32 + lane;   // TMEM lane owned by this thread

    if (!GLA) {
        // ---- L (strictly lower, rows carry beta): the off-diagonal blocks as fragment images in
        //      the (dead) K-> tile; the two diagonal blocks of the warps on the diagonal inverted
        if (quarter < 2) {
            float v[32];
            tmem_ld32(c.tmem + TM_G + lane_base + half * 32, v);
            if (REC) {
                const float br = bet[row];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] *= br;
            }
            const int brow = row >> 4, rr = row & 15;
            // the Gram barrier above has ordered the tensor core's reads of the K-> tile
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                const int bc = 2 * half + hb;
                if (bc < brow) {
                    float *dst = lfrag + (brow * (brow - 1) / 2 + bc) * 256;
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) dst[frag_pos(rr, cc)] = __uint_as_float(to_tf32(v[16 * hb + cc]));
                }
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
                float *yb = yfrag + ((quarter * 32 + seg * 16) >> 4) * 256;
#pragma unroll
                for (int cc = 0; cc < 16; ++cc) yb[frag_pos(r, cc)] = __uint_as_float(to_tf32(y[cc]));
            }
        }
        named_sync(2, kWyThreads);
    }

    // ---------------- Z' (I + L) = [I ; P] by block back-substitution over 16-column blocks,
    // 16 rows of Z' per warp: Z'_b = ([I ; P]_b - sum_{b' > b} Z'_{b'} L_{b'b}) Y_bb with
    // Y_bb = (I + L_bb)^{-1} (block form 2 of page "DeltaNet" 4.2, on the transposed system).
    // Z' = [T' ; P T'] with T' lower triangular and P lower triangular, so the blocks right of
    // the warp's own row block R are zero and are skipped.  Then Z = Z' Diag(beta) = [T ; P T],
    // kept as packed bf16 in the stmatrix register order.  For GLA (beta = 0, v unscaled)
    // Z = [I ; P].
    const int r0 = quarter * 32 + half * 16;               // first row of Z' owned by this warp
    const int R = (r0 & 63) >> 4;
    uint32_t zp[4][4];                                     // Z blocks, bf16 pairs, stmatrix order
    {
        const int g = lane >> 2, t = lane & 3;
        uint32_t za[4][2][4];                              // -Z' blocks as k-permuted tf32 A fragments
#pragma unroll
        for (int bb = 3; bb >= 0; --bb) {
            if (bb > R) {
#pragma unroll
                for (int m = 0; m < 4; ++m) zp[bb][m] = 0u;
                continue;
            }
            float acc[2][4];
            if (quarter < 2) {                             // identity rows
#pragma unroll
                for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        acc[nh][e] = (bb == R && g + 8 * (e >> 1) == 8 * nh + 2 * t + (e & 1)) ? 1.f : 0.f;
            } else {                                       // rows of P = Q<- K->^T * M (inclusive)
                float pv[8];
                tmem_ld16x256b_x2(c.tmem + TM_G + ((uint32_t)r0 << 16) + 16 * bb, pv);
#pragma unroll
                for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        acc[nh][e] = (bb < R || 8 * nh + 2 * t + (e & 1) <= g + 8 * (e >> 1)) ? pv[4 * nh + e] : 0.f;
            }
            float zb[2][4];
            if (!GLA) {
#pragma unroll
                for (int bp = bb + 1; bp < 4; ++bp) {
                    if (bp > R) continue;
                    const float *lb = lfrag + (bp * (bp - 1) / 2 + bb) * 256;
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                        for (int nh = 0; nh < 2; ++nh) {
                            const float2 lf = *reinterpret_cast<const float2 *>(lb + ((ks * 2 + nh) * 32 + lane) * 2);
                            const uint32_t bf[2] = {__float_as_uint(lf.x), __float_as_uint(lf.y)};
                            mma_tf32_16x8x8(acc[nh], za[bp][ks], bf);
                        }
                }
                uint32_t af[2][4];
                acc_as_a(acc[0], af[0], 1.f);
                acc_as_a(acc[1], af[1], 1.f);
                const float *yb = yfrag + bb * 256;
#pragma unroll
                for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                    for (int e = 0; e < 4; ++e) zb[nh][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                    for (int nh = 0; nh < 2; ++nh) {
                        const float2 yf = *reinterpret_cast<const float2 *>(yb + ((ks * 2 + nh) * 32 + lane) * 2);
                        const uint32_t bf[2] = {__float_as_uint(yf.x), __float_as_uint(yf.y)};
                        mma_tf32_16x8x8(zb[nh], af[ks], bf);
                    }
                if (bb > 0) {
                    acc_as_a(zb[0], za[bb][0], -1.f);
                    acc_as_a(zb[1], za[bb][1], -1.f);
                }
            } else {
#pragma unroll
                for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                    for (int e = 0; e < 4; ++e) zb[nh][e] = acc[nh][e];
            }
#pragma unroll
            for (int nh = 0; nh < 2; ++nh) {
                float b0 = 1.f, b1 = 1.f;
                if (!GLA) {
                    const float2 b2 = *reinterpret_cast<const float2 *>(bet + 16 * bb + 8 * nh + 2 * t);
                    b0 = b2.x;
                    b1 = b2.y;
                }
                zp[bb][2 * nh] = pack_bf16(zb[nh][0] * b0, zb[nh][1] * b1);       // rows g
                zp[bb][2 * nh + 1] = pack_bf16(zb[nh][2] * b0, zb[nh][3] * b1);   // rows g + 8
            }
        }
    }
    if (!GLA) named_sync(2, kWyThreads);                   // every warp is done with L in the K-> tile
    // ---------------- Z -> bf16 K-major 128 x 64 tile in the K-> tile: one stmatrix per 16x16 block,
    // lane l giving the address of row l & 7 of 8x8 matrix l >> 3 (rows + 8 for odd matrices,
    // columns + 8 for the last two)
    {
        const uint32_t zt = smem_u32(base + OFF_KR);
        const int mi = lane >> 3;
        const uint32_t zrow = (uint32_t)(r0 + (lane & 7) + 8 * (mi & 1));
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) stmatrix_x4(zt + sw128_offset(128, zrow, 16 * bb + 8 * (mi >> 1)), zp[bb]);
    }
    return r0;
}

// ============================================================================
// Chunks past the one-product Gram's range: the sub-chunk Gram.
// ============================================================================
// [beta K<- ; Q<-] K->^T factors exp(G_i - G_j) as Gamma_i / Gamma_j, whose 1 / Gamma_j overflows
// once a chunk's log-decay passes -kFastLog2 (base 2).  Such a chunk takes the secondary chunking
// of page "Gated Linear Attention", section 5.3, with 16-token sub-chunks:
//   - pairs of different sub-chunks (I > J) as bf16 tensor-core products, with the end of
//     sub-chunk I - 1 as reference, R_I = G at row 16 I - 1: rows i of sub-chunk I scaled by
//     2^{G_i - R_I} <= 1 (one A tile serves every I) and rows j < 16 I of K by 2^{R_I - G_j} <= 1
//     (a B tile per I), so no factor exceeds 1;
//   - pairs within a sub-chunk element by element in fp32, sum_d x_id k_jd 2^{G_id - G_jd}, at
//     full precision.
// The result lands in the Gram's TMEM columns as the one-product Gram leaves it (rows 0-63:
// [beta] K<- K->^T, rows 64-127: Q<- K->^T; the parts build_z reads), with no limit on the decay.
// The 256 WY threads enter after the prologue has written its tiles and with no copy into A_G,
// the K-> tile or the raw k tile in flight; they read q, k and g from global memory (L2), use
// A_G, the K-> tile, `scratch` (4 KB) and TMEM columns kStrongCol .. kStrongCol + 63 as scratch,
// and end with the raw g, q and k tiles fetched back into place for the prologue, which then
// runs again.  Returns the completed-phase count of B_STRONG.
constexpr uint32_t kStrongCol = 64;      // TMEM columns 64-127: free while the Gram is formed
struct StrongArgs {
    const __nv_bfloat16 *q, *k;         // [.., H, 128] rows of the batch
    const void *g;                      // channel gate, same layout (type Tg), or null
    const float *gs;                    // scalar gate of the chunk's rows (shared memory), or null
    const float *bet;                   // beta of the chunk's rows for rows 0-63, or null (unscaled)
    float *scratch;                     // 4 KB of shared memory
    size_t row0;                        // global row (b T + t) of the chunk's first token
    int H, h, live;                     // heads, this head, valid rows of the chunk
    const CUtensorMap *tm_q, *tm_k, *tm_g;   // tm_g: null unless the gate is per channel
    int tma_t, tma_b;                   // TMA token and batch coordinates of the chunk
    uint32_t kraw;                      // offset of the raw k tile
};

template <int GATE, typename Tg>
__device__ __forceinline__ uint32_t strong_gram(const Ctx &c, const StrongArgs &a, int wt, uint32_t sph) {
    uint8_t *base = c.base;
    const int d = wt & 127, part = wt >> 7;          // key channel; part 0: k side, part 1: q side
    const int ww = wt >> 5, lane = wt & 31, quarter = ww & 3, half = ww >> 2;
    const bool leader = wt == 0;
    bool ok = true;                                  // every wait here ended complete
    int armed = -1;                                  // leader: phase count of the newest phase it armed
    auto grow = [&](int r) -> float {                // log-decay of row r, channel d, base 2
        if (r >= a.live) return 0.f;
        const float x = GATE == KDA_GATE_CHANNEL
                            ? ldg_f<Tg>(static_cast<const Tg *>(a.g) + ((a.row0 + r) * a.H + a.h) * kDK + d)
                            : a.gs[r];
        return x * kLog2e;
    };
    auto raw = [&](const __nv_bfloat16 *t, int r) -> __nv_bfloat16 {
        return r < a.live ? t[((a.row0 + r) * a.H + a.h) * kDK + d] : __float2bfloat16_rn(0.f);
    };

    // ---- the A tile in A_G: row i of sub-chunk I scaled by 2^{G_i - R_I}; rows 0-63 from k
    //      (times beta), rows 64-127 from q.  R keeps R_I of channel d.
    float R[4];
    {
        const __nv_bfloat16 *x = part ? a.q : a.k;
        float G = 0.f;
#pragma unroll
        for (int I = 0; I < 4; ++I) {
            R[I] = G;
#pragma unroll 1
            for (int r0 = 16 * I; r0 < 16 * I + 16; r0 += 8) {
                float gv[8], xv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    gv[i] = grow(r0 + i);
                    xv[i] = __bfloat162float(raw(x, r0 + i));
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = r0 + i;
                    G += gv[i];
                    float v = xv[i] * ex2_approx(G - R[I]);
                    if (!part && a.bet) v *= a.bet[r];
                    *reinterpret_cast<__nv_bfloat16 *>(base + OFF_AG + sw128_offset(128, part * 64 + r, d)) =
                        __float2bfloat16_rn(v);
                }
            }
        }
    }
    auto ref = [&](int I) { return I == 0 ? R[0] : I == 1 ? R[1] : I == 2 ? R[2] : R[3]; };

    // ---- sub-chunk pairs I > J: B = rows j < 16 I of k scaled by 2^{R_I - G_j} in the K-> tile,
    //      D = A B^T (N = 16 I) into the spare columns, whose rows of sub-chunk I go to the Gram's
#pragma unroll 1
    for (int I = 1; I < 4; ++I) {
        if (part == 0) {
            const float RI = ref(I);
            float G = 0.f;
#pragma unroll 1
            for (int j0 = 0; j0 < 16 * I; j0 += 8) {
                float gv[8], kv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    gv[i] = grow(j0 + i);
                    kv[i] = __bfloat162float(raw(a.k, j0 + i));
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    G += gv[i];
                    *reinterpret_cast<__nv_bfloat16 *>(base + OFF_KR + sw128_offset(64, j0 + i, d)) =
                        __float2bfloat16_rn(kv[i] * ex2_approx(RI - G));
                }
            }
        }
        fence_proxy_async_smem();                    // A and B, before the tensor core reads them
        named_sync(2, kWyThreads);
        if (leader && ok) {
            tc_fence_after();
            const uint32_t a0 = smem_u32(base + OFF_AG), b0 = smem_u32(base + OFF_KR);
            const uint32_t id = idesc_bf16(128, 16 * I, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(c.tmem + kStrongCol, desc_kmajor(a0, 128, ks), desc_kmajor(b0, 64, ks), id, ks > 0);
            mma_commit(c.bars + B_STRONG);
            armed = (int)sph;
        }
        __syncwarp();
        ok &= wait_bar(c, B_STRONG, sph & 1u);
        ++sph;
        tc_fence_after();
        // rows of sub-chunk I: lanes 16 (I & 1) .. of quarter I / 2 (rows of L) and 2 + I / 2 (of P)
        if (half == 0 && (quarter == (I >> 1) || quarter == 2 + (I >> 1))) {
            const uint32_t lb = (uint32_t)(quarter * 32) << 16;
            const bool mine = (lane >> 4) == (I & 1);
#pragma unroll 1
            for (int cc = 0; cc * 32 < 16 * I; ++cc) {
                float o[32], nw[32];
                __syncwarp();
                tmem_ld32(c.tmem + TM_G + lb + 32 * cc, o);
                tmem_ld32(c.tmem + kStrongCol + lb + 32 * cc, nw);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = mine ? nw[e] : o[e];
                tmem_st32(c.tmem + TM_G + lb + 32 * cc, o);
            }
        }
        tc_fence_before();
        named_sync(2, kWyThreads);                   // the B tile and the spare columns are free again
    }

    // ---- pairs within sub-chunk I, in fp32.  G, k, q of its 16 rows go to the K-> tile as
    //      [channel][row] arrays (a warp's threads read distinct rows of one channel: distinct
    //      banks); one thread per entry: 136 of P (i >= j), 120 of L (i > j).
    float *sG = reinterpret_cast<float *>(base + OFF_KR);                       // [128][16] f32
    __nv_bfloat16 *sk = reinterpret_cast<__nv_bfloat16 *>(base + OFF_KR + 8192);   // [128][16]
    __nv_bfloat16 *sq = sk + 128 * 16;                                              // [128][16]
    int ei, ej;                                      // this thread's entry
    const bool isP = wt < 136;
    {
        int e = isP ? wt : wt - 136, i = isP ? 0 : 1;
        while (e >= (isP ? i + 1 : i)) {             // row i holds i + 1 (P) or i (L) entries
            e -= isP ? i + 1 : i;
            ++i;
        }
        ei = i;
        ej = e;
    }
#pragma unroll 1
    for (int I = 0; I < 4; ++I) {
        if (part == 0) {
            float G = ref(I);
#pragma unroll 4
            for (int j = 0; j < 16; ++j) {
                G += grow(16 * I + j);
                sG[d * 16 + j] = G;
            }
        } else {
#pragma unroll 4
            for (int j = 0; j < 16; ++j) {
                sk[d * 16 + j] = raw(a.k, 16 * I + j);
                sq[d * 16 + j] = raw(a.q, 16 * I + j);
            }
        }
        named_sync(2, kWyThreads);
        {
            const __nv_bfloat16 *xs = isP ? sq : sk;
            float acc = 0.f;
#pragma unroll 4
            for (int dd = 0; dd < kDK; ++dd)
                acc = fmaf(__bfloat162float(xs[dd * 16 + ei]) * __bfloat162float(sk[dd * 16 + ej]),
                           ex2_approx(sG[dd * 16 + ei] - sG[dd * 16 + ej]), acc);
            if (!isP && a.bet) acc *= a.bet[16 * I + ei];
            a.scratch[(isP ? 256 : 0) + ei * 16 + ej] = acc;
        }
        named_sync(2, kWyThreads);
        // into columns 16 I .. 16 I + 15 of the sub-chunk's rows (entries above the diagonal: 0)
        if (half == 0 && (quarter == (I >> 1) || quarter == 2 + (I >> 1))) {
            const uint32_t lb = (uint32_t)(quarter * 32) << 16;
            const bool mine = (lane >> 4) == (I & 1), pq = quarter >= 2;
            const int ii = lane & 15;
            const uint32_t cc = (uint32_t)(16 * I) & ~31u;
            const float *src = a.scratch + (pq ? 256 : 0) + ii * 16;
            float o[32];
            __syncwarp();
            tmem_ld32(c.tmem + TM_G + lb + cc, o);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const float val = (pq ? jj <= ii : jj < ii) ? src[jj] : 0.f;
                if (I & 1) o[16 + jj] = mine ? val : o[16 + jj];   // I & 1: the same in the whole warp
                else o[jj] = mine ? val : o[jj];
            }
            tmem_st32(c.tmem + TM_G + lb + cc, o);
        }
        tc_fence_before();
        named_sync(2, kWyThreads);                   // the staged rows and `scratch` are free again
    }

    // ---- the raw tiles back into place: g into A_G rows 0-63, q into rows 64-127, k into its tile
    fence_proxy_async_smem();
    named_sync(2, kWyThreads);
    if (leader && ok) {
        mbar_arrive_expect_tx(c.bars + B_STRONG, (a.tm_g ? 3u : 2u) * 16384u);
        for (int blk = 0; blk < 2; ++blk) {
            tma_load_4d(base + OFF_AG + blk * 16384 + 8192, a.tm_q, c.bars + B_STRONG, blk * 64, a.h, a.tma_t,
                        a.tma_b);
            if (a.tm_g)
                tma_load_4d(base + OFF_AG + blk * 16384, a.tm_g, c.bars + B_STRONG, blk * 64, a.h, a.tma_t, a.tma_b);
            tma_load_4d(base + a.kraw + blk * 8192, a.tm_k, c.bars + B_STRONG, blk * 64, a.h, a.tma_t, a.tma_b);
        }
        armed = (int)sph;
    }
    __syncwarp();
    ok &= wait_bar(c, B_STRONG, sph & 1u);
    ++sph;
    // a wait gave up: the newest product or copy issued here completes before the tiles are
    // touched again (the phases before it completed first)
    if (leader && !ok && armed >= 0) drain_bar(c, B_STRONG, (uint32_t)armed & 1u);
    return sph;
}

// A chunk the prologue marked: the sub-chunk Gram, then the prologue again over the refetched
// raw tiles in its STRONG form.  Out of line, so that the rarely taken path does not weigh on the
// registers of the loops around it; returns what the prologue returns in registers (K~ rows for
// the chunk's slot, gamma^C) and the completed-phase count of B_STRONG.  Ends, like the ordinary
// prologue and its barrier, with the tiles written and visible to the tensor core.
struct StrongOut {
    uint4 krv[4];
    float gam[8];
    uint32_t sph;
};
template <int GATE, bool SCAN, bool REC, typename Tg>
__device__ __noinline__ StrongOut strong_prologue(const Ctx c, const StrongArgs a, int wt, uint32_t sph,
                                                  const float *bet, uint8_t *rec) {
    StrongOut out;
    out.sph = strong_gram<GATE, Tg>(c, a, wt, sph);
    bool has_gam;
    rescale_tiles<GATE, true, SCAN, REC, true>(c.base, a.kraw, wt, a.live, bet, a.gs, a.scratch, out.krv, out.gam,
                                               has_gam, [] {}, rec);
    fence_proxy_async_smem();
    named_sync(2, kWyThreads);
    return out;
}

// ============================================================================
// WY warps: everything of a chunk that does not depend on the state.
// ============================================================================
// STRONG: the instance that takes the sub-chunk Gram for a chunk past the one-product Gram's
// range; the other instance only notes such a chunk (kStatusStrongWord) for the launch that follows.
template <int GATE, bool GLA, bool PAIR, bool STRONG, typename Tg>
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
    const int step = PAIR ? 2 : 1;                       // distance between chunks this CTA builds
    const int first = PAIR ? (int)c.rank : 0;
    auto owns = [&](int n) { return !PAIR || (n & 1) == (int)c.rank; };

    // raw tiles land where their rescaled versions go: g -> A_G rows 0-63 (free once the Gram
    // has read beta K<-), k -> the K<- tile (free once Z K<- has read it), q -> A_G rows 64-127
    // (free once A_chain has read Q<-); each is fetched for the next chunk as soon as its tile frees
    // A barrier is re-armed only after the issuing thread's own wait on its previous phase has
    // ended with the phase complete: while `clean` (every wait of this thread so far did, kept in
    // a register), it issues; after a wait gave up it issues no more copies.  So each barrier has
    // at most one copy in flight, and the last phase it issued on each is drained at the end.
    // `mi` is the index, among the chunks this CTA builds, of the chunk fetched.
    bool clean = true;
    int last_g = -1, last_k = -1, last_q = -1, last_v[2] = {-1, -1};
    uint32_t sph = 0;                                    // completed phases of the sub-chunk Gram's barrier
    auto issue_g = [&](int n, int mi) {
        if (GATE != KDA_GATE_CHANNEL || !clean) return;
        last_g = mi;
        mbar_arrive_expect_tx(c.bars + B_RAW, 16384u);
        for (int blk = 0; blk < 2; ++blk)
            tma_load_4d(base + OFF_AG + blk * 16384, tm_g, c.bars + B_RAW, blk * 64, h, sq.t0 + n * kC, sq.bt);
    };
    auto issue_k = [&](int n, int mi) {
        if (!clean) return;
        last_k = mi;
        mbar_arrive_expect_tx(c.bars + B_RAWK, 16384u);
        for (int blk = 0; blk < 2; ++blk)
            tma_load_4d(base + OFF_KL + blk * 8192, tm_k, c.bars + B_RAWK, blk * 64, h, sq.t0 + n * kC, sq.bt);
    };
    auto issue_q = [&](int n, int mi) {
        if (!clean) return;
        last_q = mi;
        mbar_arrive_expect_tx(c.bars + B_RAWQ, 16384u);
        for (int blk = 0; blk < 2; ++blk)
            tma_load_4d(base + OFF_AG + blk * 16384 + 8192, tm_q, c.bars + B_RAWQ, blk * 64, h, sq.t0 + n * kC,
                        sq.bt);
    };
    auto issue_v = [&](int n) {
        const int s = (n & 1) ^ (int)c.rank;
        if (!clean) return;
        last_v[s] = n;
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
        if (first < nchunks) {
            issue_g(first, 0);
            issue_k(first, 0);
            issue_q(first, 0);
        }
        issue_v(0);                          // nchunks >= 1: empty sequences return before the roles
        if (nchunks > 1) issue_v(1);
    }
    __syncwarp();
    {
        float bv, gv;
        load_scalars(first, bv, gv);
        if (wt < kC) { betas[wt] = bv; gss[wt] = gv; }
    }
    named_sync(2, kWyThreads);

    for (int n = 0; n < nchunks; ++n) {
        // slot of chunk n: a pair keeps the chunks it builds in slot 0 and the other CTA's in slot 1
        const int s = (n & 1) ^ (int)c.rank;
        const uint32_t ph2 = (uint32_t)((n >> 1) & 1);

        if (!owns(n)) continue;              // the chain warps take the other CTA's chunks

        // ---------------- a chunk this CTA builds
        const int m = PAIR ? (n >> 1) : n;                   // index among the chunks built here
        const uint32_t phm = (uint32_t)(m & 1);
        const int sb = m & 1;                                // scalar buffer
        const float *bet = betas + sb * kC;
        float nb = 0.f, ng = 0.f;
        const uint32_t peer_base = PAIR ? map_to_rank(smem_u32(base), c.rank ^ 1u) : 0u;
        uint4 krv[4];
        float gam[8];
        bool has_gam, strong;
        int r0 = 0;                                          // first of the 16 Z rows this warp built

        {
            if (n + step < nchunks) load_scalars(n + step, nb, ng);   // prefetch next built chunk's scalars
            if (GATE == KDA_GATE_CHANNEL) clean &= wait_bar(c, B_RAW, phm);
            // ---------------- prologue: Gamma and the rescaled tiles, in place.  K-> and gamma^C also
            // go to the chunk's slot, written at the end (the slot may still be in use).
            auto pre_qk = [&] {
                clean &= wait_bar(c, B_RAWQ, phm);
                clean &= wait_bar(c, B_RAWK, phm);
            };
            const bool mark = rescale_tiles<GATE, true, true, false, false>(
                base, OFF_KL, wt, sq.len - n * kC, bet, gss + sb * kC, tot, krv, gam, has_gam, pre_qk);
            fence_proxy_async_smem();
            if constexpr (!STRONG) {
                // outputs of this call are redone by the STRONG launch: note it, go on
                if (mark) p.status[kStatusStrongWord] = p.strong_token;
                named_sync(2, kWyThreads);
                strong = false;
            } else {
                strong = named_sync_or(2, kWyThreads, mark);
            }
            if (STRONG && strong) {
                const StrongArgs sa{static_cast<const __nv_bfloat16 *>(p.q),
                                    static_cast<const __nv_bfloat16 *>(p.k),
                                    GATE == KDA_GATE_CHANNEL ? p.g : nullptr,
                                    gss + sb * kC,
                                    bet,
                                    tot,
                                    (size_t)sq.bt * T + sq.t0 + n * kC,
                                    H,
                                    h,
                                    sq.len - n * kC,
                                    tm_q,
                                    tm_k,
                                    GATE == KDA_GATE_CHANNEL ? tm_g : nullptr,
                                    sq.t0 + n * kC,
                                    sq.bt,
                                    OFF_KL};
                const StrongOut so = strong_prologue<GATE, true, false, Tg>(c, sa, wt, sph, bet, nullptr);
#pragma unroll
                for (int i = 0; i < 4; ++i) krv[i] = so.krv[i];
#pragma unroll
                for (int e = 0; e < 8; ++e) gam[e] = so.gam[e];
                sph = so.sph;
            }

            r0 = build_z<GLA>(c, wt, bet, phm, tot, strong);
            // the Gram has read beta K<-: the next chunk's g may land in its rows
            if (leader && n + step < nchunks) issue_g(n + step, m + 1);
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(2, kWyThreads);
        }

        // ---------------- Z K<- -> [W ; P W],  Z V -> D1[s] = [U ; P U]
        if (leader) {
            clean &= wait_bar(c, B_V0 + s, ph2);
            if (n >= 2) wait_bar(c, B_E10 + s, (uint32_t)(((n - 2) >> 1) & 1));   // D1[s] drained
            tc_fence_after();
            const uint32_t a0 = smem_u32(base + OFF_KR);
            const uint32_t bk = smem_u32(base + OFF_KL);
            if (!GLA && s == 0) {
                // slot 0: the v tile directly follows the two 64-column blocks of K<-, and D1[0] the
                // [W ; P W] columns, so Z [K<- | V] = [[W ; P W] | [U ; P U]] is one N = 192 product
                static_assert(OFF_V0 == OFF_KL + 16384 && TM_D1 == TM_WQ + 128, "merged Z [K<- | V] layout");
                const uint32_t id = idesc_bf16(128, 192, 0, 1);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(c.tmem + TM_WQ, desc_kmajor(a0, 128, ks), desc_mnmajor(bk, 64, ks), id, ks > 0);
            } else {
                if (!GLA) {
                    const uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(c.tmem + TM_WQ, desc_kmajor(a0, 128, ks), desc_mnmajor(bk, 64, ks), id, ks > 0);
                }
                const uint32_t bv = smem_u32(base + off_v(s));
                const uint32_t id = idesc_bf16(128, 64, 0, 1);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(c.tmem + TM_D1 + s * 64, desc_kmajor(a0, 128, ks), desc_mnmajor(bv, 64, ks), id,
                             ks > 0);
            }
            mma_commit(c.bars + B_W2);
        }
        __syncwarp();                        // aligned TMEM loads and barriers below need whole warps
        wait_bar(c, B_W2, phm);
        tc_fence_after();
        if (leader && n + 2 < nchunks) issue_v(n + 2);           // v[s] consumed
        if (leader && n + step < nchunks) issue_k(n + step, m + 1);    // the K<- tile is consumed
        __syncwarp();
        if (n >= 2) wait_bar(c, B_C20 + s, (uint32_t)(((n - 2) >> 1) & 1));   // own scan done with slot s
        // the other CTA of a pair is done with the chunk sent before, whose slot tiles and Z it
        // received here: its slot 1 and Z-in tile may be rewritten.  The two waits of the exchange
        // between the CTAs of a pair (this one, and the receiver's for the chunk) are drain waits:
        // both CTAs run every chunk whatever their other waits did, so every chunk is sent and
        // received, at most one is in flight towards a CTA, and none is when it exits.
        if (PAIR && m >= 1) drain_bar_cluster(c, B_PFREE, (uint32_t)((m - 1) & 1));
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
                        // Q<-: rows 64-127 of A_G
                        const uint4 u = *reinterpret_cast<const uint4 *>(base + OFF_AG +
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
        // ---------------- K-> (K~) and gamma^C into slot s (and the other CTA's slot s)
        store_kr_slot(base + off_kt(s), gC + s * kDK, wt, krv, gam, has_gam, strong);
        if (wt < kC && n + step < nchunks) {
            betas[(sb ^ 1) * kC + wt] = nb;
            gss[(sb ^ 1) * kC + wt] = ng;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_sync(2, kWyThreads);
        if (leader) {
            mbar_arrive(c.bars + B_WYR0 + s);
            if (n + step < nchunks) issue_q(n + step, m + 1);      // A_chain has read Q<-
            if (PAIR) {
                // the slot buffers go to slot 1 of the other CTA, which keeps the chunks built here
                // there, by bulk copy (it is done with chunk n - 2: checked above)
                const int ps = s ^ 1;
                const uint32_t rbar = peer_base + OFF_MISC + MISC_BAR + 8u * B_RX;
                const uint32_t gc_src = OFF_MISC + MISC_GC + (uint32_t)s * 512u;
                const uint32_t gc_dst = OFF_MISC + MISC_GC + (uint32_t)ps * 512u;
                mbar_arrive_expect_tx_remote(rbar, kPushBytes);
                bulk_copy_to_peer(peer_base + off_ach(ps), base + off_ach(s), 32768u, rbar);
                bulk_copy_to_peer(peer_base + off_kt(ps), base + off_kt(s), 16384u, rbar);
                bulk_copy_to_peer(peer_base + gc_dst, base + gc_src, 512u, rbar);
            }
        }
        __syncwarp();                        // the leader's warp reaches the next barrier converged
    }
    // drain, also after a wait gave up: every product issued here is done and the newest copy
    // into each raw tile has landed before TMEM is freed and the CTA exits
    if (leader) {
        mma_commit(c.bars + B_FIN1);
        drain_bar(c, B_FIN1, 0);
        if (last_g >= 0) drain_bar(c, B_RAW, (uint32_t)(last_g & 1));
        if (last_k >= 0) drain_bar(c, B_RAWK, (uint32_t)(last_k & 1));
        if (last_q >= 0) drain_bar(c, B_RAWQ, (uint32_t)(last_q & 1));
        // v slots: a pair's slot 1 (the other CTA's chunks) is drained by the chain leader, which
        // arms its later phases (an earlier phase than the last one would alias by parity with
        // a phase that is still open)
        for (int sl = 0; sl < (PAIR ? 1 : 2); ++sl)
            if (last_v[sl] >= 0) drain_bar(c, B_V0 + sl, (uint32_t)((last_v[sl] >> 1) & 1));
    }
    __syncwarp();
}

// ============================================================================
// Chain warps: the serial state scan and the output.
// ============================================================================
template <bool PAIR, bool STRONG>
__device__ void chain_role(const Ctx &c, const FwdParams &p, const CUtensorMap *tm_v, const CUtensorMap *tm_o,
                           int e0, int h, int b, Seq sq, int nchunks) {
    uint8_t *base = c.base;
    const int j = threadIdx.x;                  // key channel == TMEM lane
    const int warp = j >> 5;
    const bool leader = j == 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float *gC = reinterpret_cast<const float *>(base + OFF_MISC + MISC_GC);
    const int H = p.H, dv = p.dv;
    bool clean = true;                          // every wait of this thread has ended complete
    int last_v = -1;                            // newest v copy this thread issued (chunk index)

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


    for (int n = 0; n < nchunks; ++n) {
        const int s = (n & 1) ^ (int)c.rank;   // a pair: own chunks in slot 0, the other CTA's in slot 1
        const uint32_t ph2 = (uint32_t)((n >> 1) & 1);
        const bool peer_chunk = PAIR && (n & 1) != (int)c.rank;
        if (peer_chunk) {
            // built by the other CTA: wait until its WY warps have written A_chain, K->, gamma^C
            // and Z here, and for this slice's v; [U ; P U] = Z V goes right before the state product
            if (leader) clean &= wait_bar(c, B_V0 + s, ph2);
            __syncwarp();
            drain_bar_cluster(c, B_RX, (uint32_t)((n >> 1) & 1));   // an exchange wait (see the WY warps)
            fence_proxy_async_smem();    // the received tiles are read by the tensor core next
        } else {
            wait_bar(c, B_WYR0 + s, ph2);
        }
        tc_fence_after();
        // gamma^C; its sign bit marks a chunk whose slot holds K~ instead of K-> (same in every thread)
        const float gsg = gC[s * kDK + j];
        const bool ktilde = STRONG && signbit(gsg);
        const float gam = STRONG ? fabsf(gsg) : gsg;

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
        if (peer_chunk && leader && n + 2 < nchunks && clean) {
            // v[s] has been read: fetch the slice of chunk n + 2 (its wait on chunk n's copy above
            // ended complete; after a wait gave up no more copies are issued)
            last_v = n + 2;
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
        {
            float v[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                tmem_ld32(c.tmem + TM_S + lane_base + cc * 32, v);
                if (!ktilde) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) S[cc * 32 + e] = gam * (S[cc * 32 + e] + v[e]);   // dS^T = K->^T V_new
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) S[cc * 32 + e] = fmaf(gam, S[cc * 32 + e], v[e]);   // dS^T = K~^T V_new
                }
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
        drain_bar(c, B_FIN0, 0);
        if (PAIR) {
            // slot 1 of a pair: the newest v copy into it, issued here or, when the chain issued
            // none, by the WY leader at the start (the first of the other CTA's chunks)
            const int first_peer = c.rank ? 0 : 1;
            const int lv = last_v >= 0 ? last_v : (first_peer < nchunks ? first_peer : -1);
            if (lv >= 0) drain_bar(c, B_V1, (uint32_t)((lv >> 1) & 1));
        }
    }
    __syncwarp();
}

// STRONG: the second launch of a call, which redoes the call with the sub-chunk Gram when the
// first noted a chunk past the one-product Gram's range, and exits at once otherwise (both CTAs of
// a pair read the same word, so they decide alike).
template <int GATE, bool GLA, bool PAIR, bool STRONG, typename Tg>
__global__ void __launch_bounds__(kThreads, 1)
kda_fwd_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_g,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o) {
    if (STRONG) {
        grid_dep_wait();                    // the first launch of the call is done and visible
        if (*reinterpret_cast<volatile const int *>(p.status + kStatusStrongWord) != p.strong_token) return;
    } else {
        grid_dep_launch();                  // the second launch may take SMs as this one's blocks finish
    }
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctx c;
    c.base = base;
    c.bars = reinterpret_cast<uint64_t *>(base + OFF_MISC + MISC_BAR);
    c.abort = reinterpret_cast<volatile int *>(base + OFF_MISC + MISC_ABORT);
    c.status = p.status;
    c.bound = wait_bound_of(p.status);
    c.short_polls = c.bound != kWaitBound;
    c.rank = PAIR ? cluster_ctarank() : 0u;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + OFF_MISC + MISC_TSLOT);

    const int e0 = blockIdx.x * kDVS, h = blockIdx.y, b = blockIdx.z;
    const Seq sq = seq_of(p, b);
    const int nchunks = (sq.len + kC - 1) / kC;
    c.zrec = nullptr;
    c.zstride = 0;
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
        chain_role<PAIR, STRONG>(c, p, &tm_v, &tm_o, e0, h, b, sq, nchunks);
    else
        wy_role<GATE, GLA, PAIR, STRONG, Tg>(c, p, &tm_q, &tm_k, &tm_g, &tm_v, e0, h, sq, nchunks);

    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();           // no remote access into a CTA that has exited
    tc_fence_after();
    if (threadIdx.x < 32) tmem_dealloc(c.tmem, kTmemCols);
}

// ============================================================================
// Chunk records: every state-independent operand of a chunk, chunk-parallel
// ahead of the record scan kernel.
// ============================================================================
// One CTA per (chunk, head, sequence) computes Gamma, the rescaled tiles and
// Z = [T ; P T] with the single kernel's code (rescale_tiles, build_z), then
// [W ; P W] = Z K<- on the tensor core and A_chain = [-W ; Q<- - P W], and
// stores the images of the bf16 tiles Z, A_chain and K~ (and gamma^C) as the
// chunk's record, which the scan kernel loads with bulk copies.  Shared
// memory: the A_G and K-> tiles at the single kernel's offsets (raw k lands in
// the K-> tile and becomes K-> in place; A_G becomes [K<- ; Q<-], then
// A_chain), then the scalars, the cumsum partials and the barriers.
constexpr uint32_t OFF_WMISC = 49152;
constexpr uint32_t WM_BETA = 0;          // beta [64] f32
constexpr uint32_t WM_GS = 256;          // scalar gate [64] f32
constexpr uint32_t WM_TOT = 512;         // cumsum partials [8][128] f32
constexpr uint32_t WM_BAR = 4608;        // mbarriers [kNumBars] u64
constexpr uint32_t WM_TSLOT = 4800;      // TMEM base address
constexpr uint32_t WM_ABORT = 4804;      // abort flag
constexpr uint32_t kWMiscBytes = 4864;
constexpr uint32_t kZSmemBytes = OFF_WMISC + kWMiscBytes + 1024;
constexpr uint32_t kZTmemCols = 128;     // the Gram [L ; P] (64), then [W ; P W] (128)
static_assert(OFF_KR + 16384 <= OFF_WMISC, "Z kernel tile layout");
static_assert(WM_BAR + kNumBars * 8 <= WM_TSLOT, "Z kernel misc layout");
static_assert(WM_ABORT + 4 <= kWMiscBytes, "Z kernel misc layout");

template <int GATE, bool GLA, typename Tg>
__global__ void __launch_bounds__(kWyThreads, 4)
kda_fwd_z_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // one-dimensional grid, chunk-major with the last chunk first: the records the scan reads
    // first are written last and are still in L2 when it starts
    const int nch = (p.T + kC - 1) / kC;
    const int per_chunk = p.H * p.B;
    const int h = (int)(blockIdx.x % (unsigned)p.H), b = (int)((blockIdx.x / (unsigned)p.H) % (unsigned)p.B);
    const int n = nch - 1 - (int)(blockIdx.x / (unsigned)per_chunk);
    const Seq sq = seq_of(p, b);
    grid_dep_launch();                      // the record scan may take SMs as this kernel's blocks finish
    if (n * kC >= sq.len) return;           // past the end of this sequence (or an empty one)
    const int wt = threadIdx.x;
    Ctx c;
    c.base = base;
    c.bars = reinterpret_cast<uint64_t *>(base + OFF_WMISC + WM_BAR);
    c.abort = reinterpret_cast<volatile int *>(base + OFF_WMISC + WM_ABORT);
    c.status = p.status;
    c.bound = wait_bound_of(p.status);
    c.short_polls = c.bound != kWaitBound;
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
        mbar_init(c.bars + B_FIN0, 1);
        mbar_init(c.bars + B_STRONG, 1);
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
    uint4 krv[4];
    float gam[8];
    bool has_gam;
    const bool mark = rescale_tiles<GATE, true, false, true, false>(base, OFF_KR, wt, sq.len - n * kC, betas, gss,
                                                                    tot, krv, gam, has_gam, [] {}, rec);
    fence_proxy_async_smem();
    bool strong = false;                    // no gate: no decay, no sub-chunk path compiled
    if constexpr (GATE == KDA_GATE_NONE) __syncthreads();
    else strong = __syncthreads_or(mark) != 0;
    if (strong) {
        const StrongArgs sa{static_cast<const __nv_bfloat16 *>(p.q),
                            static_cast<const __nv_bfloat16 *>(p.k),
                            GATE == KDA_GATE_CHANNEL ? p.g : nullptr,
                            gss,
                            nullptr,
                            tot,
                            (size_t)sq.bt * T + sq.t0 + n * kC,
                            H,
                            h,
                            sq.len - n * kC,
                            &tm_q,
                            &tm_k,
                            GATE == KDA_GATE_CHANNEL ? &tm_g : nullptr,
                            sq.t0 + n * kC,
                            sq.bt,
                            OFF_KR};
        strong_prologue<GATE, false, true, Tg>(c, sa, wt, 0u, betas, rec);
    }
    // the cumsum partials are dead: their 4 KB hold the diagonal-block inverses
    build_z<GLA, true>(c, wt, betas, 0, tot, strong);
    fence_proxy_async_smem();               // the Z stores, before the bulk copy and the tensor core read them
    tc_fence_before();
    __syncthreads();                        // and every warp is done with the Gram's TMEM columns
    tc_fence_after();
    if (wt == 0) {
        bulk_store(rec + REC_Z, base + OFF_KR, 16384u);
        tma_store_commit();
        // [W ; P W] = Z K<-  (M128 N128 K64) over the Gram's columns.  K<- is rows 0-63 of A_G,
        // read as an MN-major B tile: 16 K rows per step, its two 64-wide N blocks 16 KB apart.
        // GLA (beta = 0): W = 0, no product.
        if (!GLA) {
            const uint32_t a0 = smem_u32(base + OFF_KR), b0 = smem_u32(base + OFF_AG);
            const uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(c.tmem + TM_G, desc_kmajor(a0, 128, ks), sdesc_sw128(b0 + ks * 2048u, 16384u, 1024u), id,
                         ks > 0);
        }
        mma_commit(c.bars + B_GRAM);
    }
    __syncwarp();
    wait_bar(c, B_GRAM, 1);
    tc_fence_after();
    // A_chain = [-W ; Q<- - P W] in place over A_G = [K<- ; Q<-] (the product has read K<-):
    // TMEM lane quarter ww & 3, 64 columns per warp
    {
        const int ww = wt >> 5, quarter = ww & 3, half = ww >> 2;
        const int row = quarter * 32 + (wt & 31);
        uint8_t *ag = base + OFF_AG;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int col = half * 64 + cc * 32;
            float v[32];
            if (!GLA) {
                tmem_ld32(c.tmem + TM_G + ((uint32_t)(quarter * 32) << 16) + col, v);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0.f;
            }
            if (quarter < 2) {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = -v[e];
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(ag + sw128_offset(128, row, col + 8 * q));
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[e]));
                        v[8 * q + 2 * e] = f.x - v[8 * q + 2 * e];
                        v[8 * q + 2 * e + 1] = f.y - v[8 * q + 2 * e + 1];
                    }
                }
            }
            store_row32_bf16(ag, 128, row, col, v);
        }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (wt == 0) {
        bulk_store(rec + REC_A, base + OFF_AG, 32768u);
        tma_store_commit();
        tma_store_wait_read0();             // shared memory may go once the copies have read it
        // drain, also after a wait gave up: the products are done and the tiles have landed
        mma_commit(c.bars + B_FIN0);
        drain_bar(c, B_FIN0, 0);
        drain_bar(c, B_RAW, 0);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (wt < 32) tmem_dealloc(c.tmem, kZTmemCols);
}

// ============================================================================
// Record scan kernel: the state recursion over the chunk records.
// ============================================================================
// One CTA per (value slice, head, sequence).  The records carry every
// state-independent operand, so a chunk takes three products:
//   D1 = Z V = [U ; P U]                  (issued by the loader, one chunk ahead)
//   D1 += A_chain S^T = [V_new ; O]       (the state product)
//   dS^T = K~^T V_new,   S <- S Diag(gamma^C) + dS
// The CTA's SV = NH W values are split into NH halves of W, each a chain of four
// warps with its own accumulator columns, S^T and V_new tiles and barriers, so
// the halves can run out of step.  Warp 4 NH loads the records (bulk copies)
// and the v tiles (TMA) and issues Z V for the whole slice.  A record takes
// about a chunk's time to arrive, so A_chain, K~, gamma^C and v of chunk n go
// to entry n % RD of an RD-deep ring, loaded RD chunks ahead, and Z V of chunk
// n runs up to two chunks ahead into accumulator slot n % RD, its Z from entry
// n % 2 of a two-deep ring.  V_new takes the front of the half's S^T tile,
// which the state product has read by then.
//   Configurations: one 64-wide slice (NH = 1, W = 64, RD = 3); both slices of
// a dv = 128 head in one CTA (NH = 2, W = 64, RD = 2: the record and Z tiles
// serve both halves, half the CTAs, for batches of more heads than one wave
// of SMs holds).  Two 32-wide halves of a 64-wide slice (NH = 2, W = 32, RD =
// 3, MN-major B tiles with 64-byte swizzle) give the same values and measured
// no faster: the halves run in step, the products' latency dominates.
template <int NH_, int W_, int RD_> struct ScanCfg {
    static constexpr int NH = NH_, W = W_, RD = RD_;
    static constexpr int SV = NH * W;                    // values per CTA
    static constexpr int kThreads = 128 * NH + 32;
    static constexpr uint32_t R_ACH = 0, R_KT = 32768, R_V = 49152;
    static constexpr uint32_t R_SLOT = R_V + 128u * SV;  // ring entry: A_chain, K~, v (64 rows x SV)
    static constexpr uint32_t OFF_Z = RD * R_SLOT;       // two entries: Z
    static constexpr uint32_t OFF_ST = OFF_Z + 2 * 16384;    // S^T (then V_new) of each half, 256 SV bytes in all
    static constexpr uint32_t OFF_GC = OFF_ST + 256u * SV;   // gamma^C [RD][128] f32
    static constexpr uint32_t OFF_BAR = OFF_GC + 1536;   // mbarriers
    static constexpr uint32_t OFF_TSLOT = OFF_BAR + 256;
    static constexpr uint32_t OFF_ABORT = OFF_TSLOT + 4;
    static constexpr uint32_t kSmem = OFF_ABORT + 60 + 1024;   // + alignment slack of the dynamic base
    static constexpr uint32_t kRTx = 32768u + 16384u + 512u + 128u * SV, kZTx = 16384u;
    // TMEM: [U ; P U] -> [V_new ; O] in RD slots of SV columns (half h at + h W), then dS^T
    static constexpr uint32_t TS_D1 = 0, TS_DS = RD * SV;
    static constexpr uint32_t kTmemCols = (RD + 1) * SV <= 256 ? 256 : 512;
    static_assert(RD >= 2 && RD <= 3 && (RD + 1) * SV <= 512, "scan configuration");
    static_assert(kSmem <= 232448, "shared memory per CTA");
};
using ScanSlice = ScanCfg<1, 64, 3>;     // one 64-wide value slice per CTA
using ScanHead = ScanCfg<2, 64, 2>;      // both slices of a dv = 128 head per CTA

// Ring entry / accumulator slot n % 3: FULLR, RFREE (one arrival per half), ZV, D1FREE (one
// arrival per half); Z entry n % 2: FULLZ; C1 / C2: [half][chunk parity].
enum { SB_FULLR = 0, SB_RFREE = 3, SB_ZV = 6, SB_D1FREE = 9, SB_FULLZ = 12, SB_C1 = 14, SB_C2 = 18, SB_FINL = 22,
       SB_FINC = 23, kScanBars = 25 };
static_assert(kScanBars * 8 <= 256, "scan barriers");

// 64-byte swizzle (MN-major operand tiles of 32 bf16 columns, one 64-byte row
// each, 512-byte atoms of 8 rows): byte offset of column c < 32 of row r.
__device__ __forceinline__ uint32_t sw64_offset(uint32_t r, uint32_t c) {
    return r * 64u + ((((c >> 3) ^ (r >> 1)) & 3u) << 4) + ((c & 7u) << 1);
}
// Descriptor of K-step ks (16 K rows) of such a tile: 8-row groups 512 bytes apart.
__device__ __forceinline__ uint64_t desc_mn32(uint32_t base, uint32_t ks) {
    uint64_t d = 0;
    const uint32_t saddr = base + ks * 1024u;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((8192u >> 4) & 0x3FFFu) << 16;   // stride between 32-wide blocks (one block: unused)
    d |= (uint64_t)((512u >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;                         // descriptor version for tcgen05
    d |= (uint64_t)4u << 61;                         // 64-byte swizzle
    return d;
}

// W bf16 values of one row of a half's MN-major tile (SW128 with 64 columns, SW64 with 32).
template <int W>
__device__ __forceinline__ void store_half_row(uint8_t *tile, uint32_t rows, uint32_t r, const float *v) {
#pragma unroll
    for (int q = 0; q < W / 8; ++q) {
        const uint32_t off = W == 64 ? sw128_offset(rows, r, 8 * q) : sw64_offset(r, 8 * q);
        st_u128(tile + off, pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
    }
}
template <int W>
__device__ __forceinline__ uint64_t desc_half(uint32_t base, uint32_t krows, uint32_t ks) {
    return W == 64 ? desc_mnmajor(base, krows, ks) : desc_mn32(base, ks);
}
template <int W> __device__ __forceinline__ void tmem_ld_half(uint32_t taddr, float (&v)[W]) {
    tmem_ld32(taddr, *reinterpret_cast<float(*)[32]>(&v[0]));
    if constexpr (W == 64) tmem_ld32(taddr + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
}

// One half's chain: thread t of the half owns key channel t (its TMEM lane) and
// the W state values S[ev0 .. ev0 + W)[t] in registers.
template <class G>
__device__ void scan_chain(const Ctx &c, const FwdParams &p, int half, int e0, int h, int b, Seq sq,
                           int nchunks) {
    constexpr int W = G::W, RD = G::RD, SV = G::SV;
    constexpr int PW = G::NH == 2 && W == 64 ? 32 : W;   // columns per TMEM load
    uint8_t *base = c.base;
    const int t = threadIdx.x - 128 * half;
    const int warp = t >> 5;                             // TMEM lane quarter
    const bool leader = t == 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int ev0 = e0 + half * W;
    const int H = p.H, dv = p.dv;
    const int bar_id = 1 + half;
    uint8_t *st = base + G::OFF_ST + half * 128 * W * 2;
    uint8_t *vn = st;                                    // V_new: 64 rows at the front of the S^T tile
    const float *gc = reinterpret_cast<const float *>(base + G::OFF_GC);
    const uint32_t col = (uint32_t)(half * W);

    float S[W];
#pragma unroll
    for (int e = 0; e < W; ++e) S[e] = p.h0 ? p.h0[(((size_t)b * H + h) * dv + ev0 + e) * kDK + t] : 0.f;

    auto write_state = [&]() {
        store_half_row<W>(st, 128, t, S);
        fence_proxy_async_smem();
        tc_fence_before();
        named_sync(bar_id, 128);
    };
    write_state();

    const uint32_t id1 = idesc_bf16(128, W, 0, 1), id2 = idesc_bf16(128, W, 1, 1);
    for (int n = 0; n < nchunks; ++n) {
        const int s = n & 1, ri = n % RD;
        const uint32_t ph = (uint32_t)((n >> 1) & 1), phr = (uint32_t)((n / RD) & 1);
        uint8_t *slot = base + ri * G::R_SLOT;
        wait_bar(c, SB_FULLR + ri, phr);                 // A_chain, K~ and gamma^C of the record
        wait_bar(c, SB_ZV + ri, phr);                    // D1[ri] = [U ; P U]
        tc_fence_after();
        const float gam = gc[ri * kDK + t];

        // ---- D1[s] += A_chain S^T   (M128 N=W K128)
        if (leader) {
            const uint32_t a0 = smem_u32(slot + G::R_ACH), b0 = smem_u32(st);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(c.tmem + G::TS_D1 + ri * SV + col, desc_kmajor(a0, 128, ks), desc_half<W>(b0, 128, ks), id1,
                         1);
            mma_commit(c.bars + SB_C1 + half * 2 + s);
        }
        __syncwarp();
        wait_bar(c, SB_C1 + half * 2 + s, ph);
        tc_fence_after();

        // ---- rows 0-63 (warps 0, 1): V_new -> the half's V_new tile, then dS^T = K~^T V_new;
        //      rows 64-127 (warps 2, 3): O -> o, stored while that product runs
        {
            // in pieces of PW columns: with two 64-wide halves a whole row would not fit the registers
            const int r = (warp & 1) * 32 + (t & 31);
            float v[W];
            if constexpr (PW == W) {
                tmem_ld_half<W>(c.tmem + G::TS_D1 + ri * SV + col + lane_base, v);
                if (warp < 2) store_half_row<W>(vn, 64, r, v);
            } else {
                // the O rows (warps 2, 3) go out piece by piece at once
#pragma unroll
                for (int pc = 0; pc < W / PW; ++pc) {
                    float u[PW];
                    tmem_ld32(c.tmem + G::TS_D1 + ri * SV + col + pc * PW + lane_base, u);
                    if (warp < 2) {
#pragma unroll
                        for (int q = 0; q < PW / 8; ++q)
                            st_u128(vn + sw128_offset(64, r, pc * PW + 8 * q), pack_bf16(u[8 * q], u[8 * q + 1]),
                                    pack_bf16(u[8 * q + 2], u[8 * q + 3]), pack_bf16(u[8 * q + 4], u[8 * q + 5]),
                                    pack_bf16(u[8 * q + 6], u[8 * q + 7]));
                    } else if (n * kC + r < sq.len) {
                        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.o) +
                                              (((size_t)sq.bt * p.T + sq.t0 + n * kC + r) * H + h) * dv + ev0 + pc * PW;
#pragma unroll
                        for (int q = 0; q < PW / 8; ++q)
                            *reinterpret_cast<uint4 *>(orow + 8 * q) =
                                make_uint4(pack_bf16(u[8 * q], u[8 * q + 1]), pack_bf16(u[8 * q + 2], u[8 * q + 3]),
                                           pack_bf16(u[8 * q + 4], u[8 * q + 5]), pack_bf16(u[8 * q + 6], u[8 * q + 7]));
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(bar_id, 128);
            // ---- dS^T = K~^T V_new   (M128 N=W K64)
            if (leader) {
                tc_fence_after();
                mbar_arrive(c.bars + SB_D1FREE + ri);    // this half's columns of D1[ri] are drained
                const uint32_t a0 = smem_u32(slot + G::R_KT), b0 = smem_u32(vn);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(c.tmem + G::TS_DS + col, desc_mnmajor(a0, 64, ks), desc_half<W>(b0, 64, ks), id2, ks > 0);
                mma_commit(c.bars + SB_C2 + half * 2 + s);
            }
            __syncwarp();
            if (PW == W && warp >= 2 && n * kC + r < sq.len) {
                __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.o) +
                                      (((size_t)sq.bt * p.T + sq.t0 + n * kC + r) * H + h) * dv + ev0;
#pragma unroll
                for (int q = 0; q < W / 8; ++q)
                    *reinterpret_cast<uint4 *>(orow + 8 * q) =
                        make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                                   pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
            }
        }
        wait_bar(c, SB_C2 + half * 2 + s, ph);
        tc_fence_after();
        if (leader) mbar_arrive(c.bars + SB_RFREE + ri);  // this half is done with ring entry ri
        __syncwarp();
#pragma unroll
        for (int pc = 0; pc < W / PW; ++pc) {
            float v[PW];
            if constexpr (PW == W) tmem_ld_half<W>(c.tmem + G::TS_DS + col + lane_base, v);
            else tmem_ld32(c.tmem + G::TS_DS + col + pc * PW + lane_base, v);
#pragma unroll
            for (int e = 0; e < PW; ++e)                // S Diag(gamma^C) + dS, dS^T = K~^T V_new
                S[pc * PW + e] = fmaf(gam, S[pc * PW + e], v[e]);
        }
        write_state();
    }
    if (p.ht) {
#pragma unroll
        for (int e = 0; e < W; ++e) p.ht[(((size_t)b * H + h) * dv + ev0 + e) * kDK + t] = S[e];
    }
    if (leader) {                                       // every product issued here is done
        mma_commit(c.bars + SB_FINC + half);
        drain_bar(c, SB_FINC + half, 0);
    }
    __syncwarp();
}

// The loader (one thread): chunk n's A_chain, K~, gamma^C and v tile into ring
// entry n % RD, its Z into entry n % 2 of the Z ring, and D1[n % RD] = Z V as
// soon as those are in and chunk n - RD has drained the slot.
template <class G>
__device__ void scan_loader(const Ctx &c, const FwdParams &p, const CUtensorMap *tm_v, int e0, int h, Seq sq,
                            int nchunks) {
    constexpr int RD = G::RD, SV = G::SV;
    uint8_t *base = c.base;
    // A ring entry is re-armed only after this thread's own wait on its previous copy (in zv)
    // ended with it landed: while `clean` (every wait of this thread so far did) it issues, after
    // a wait gave up it issues no more copies.  One copy in flight per barrier, the newest drained
    // at the end.
    int last_r = -1, last_z = -1;                        // newest record / Z copy issued
    bool clean = true;
    auto issue_r = [&](int n) {
        const uint8_t *r = c.zrec + (size_t)n * c.zstride;
        const int ri = n % RD;
        uint8_t *slot = base + ri * G::R_SLOT;
        uint64_t *bar = c.bars + SB_FULLR + ri;
        if (!clean) return;
        last_r = n;
        mbar_arrive_expect_tx(bar, G::kRTx);
        bulk_load(slot + G::R_ACH, r + REC_A, 32768u, bar);
        bulk_load(slot + G::R_KT, r + REC_KR, 16384u, bar);
        bulk_load(base + G::OFF_GC + ri * 512, r + REC_GC, 512u, bar);
        for (int vb = 0; vb < SV / 64; ++vb)           // 64-wide column blocks of the v tile
            tma_load_4d(slot + G::R_V + vb * 8192, tm_v, bar, e0 + 64 * vb, h, sq.t0 + n * kC, sq.bt);
    };
    auto issue_z = [&](int n) {
        const uint8_t *r = c.zrec + (size_t)n * c.zstride;
        uint64_t *bar = c.bars + SB_FULLZ + (n & 1);
        if (!clean) return;
        last_z = n;
        mbar_arrive_expect_tx(bar, G::kZTx);
        bulk_load(base + G::OFF_Z + (n & 1) * 16384, r + REC_Z, 16384u, bar);
    };
    auto zv = [&](int n) {
        const int ri = n % RD;
        clean &= wait_bar(c, SB_FULLR + ri, (uint32_t)((n / RD) & 1));       // v
        clean &= wait_bar(c, SB_FULLZ + (n & 1), (uint32_t)((n >> 1) & 1));  // Z
        if (n >= RD) wait_bar(c, SB_D1FREE + ri, (uint32_t)(((n - RD) / RD) & 1));   // chunk n - RD drained D1[ri]
        tc_fence_after();
        const uint32_t a0 = smem_u32(base + G::OFF_Z + (n & 1) * 16384), b0 = smem_u32(base + ri * G::R_SLOT + G::R_V);
        const uint32_t id = idesc_bf16(128, SV, 0, 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(c.tmem + G::TS_D1 + ri * SV, desc_kmajor(a0, 128, ks), desc_mnmajor(b0, 64, ks), id, ks > 0);
        mma_commit(c.bars + SB_ZV + ri);
    };
    if ((threadIdx.x & 31) == 0) {
        for (int n = 0; n < RD && n < nchunks; ++n) {
            issue_r(n);
            if (n < 2) issue_z(n);
        }
        zv(0);
        if (nchunks > 1) zv(1);
        for (int n = 0; n < nchunks; ++n) {
            if (n + 2 < nchunks) {
                wait_bar(c, SB_ZV + n % RD, (uint32_t)((n / RD) & 1));    // Z V of chunk n has read its Z
                issue_z(n + 2);
            }
            if (n + RD < nchunks) {
                wait_bar(c, SB_RFREE + n % RD, (uint32_t)((n / RD) & 1));  // chunk n is done with its entry
                issue_r(n + RD);
            }
            if (n + 2 < nchunks) zv(n + 2);
        }
        // drain, also after a wait gave up: the newest copy into every entry has landed and every
        // product issued here is done before the CTA frees TMEM and exits
        for (int m = last_r; m >= 0 && m > last_r - RD; --m)
            drain_bar(c, SB_FULLR + m % RD, (uint32_t)((m / RD) & 1));
        for (int m = last_z; m >= 0 && m > last_z - 2; --m) drain_bar(c, SB_FULLZ + (m & 1), (uint32_t)((m >> 1) & 1));
        mma_commit(c.bars + SB_FINL);
        drain_bar(c, SB_FINL, 0);
    }
    __syncwarp();
}

template <class G>
__global__ void __launch_bounds__(G::kThreads, 1)
kda_fwd_scan_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_v) {
    constexpr int NH = G::NH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctx c;
    c.base = base;
    c.bars = reinterpret_cast<uint64_t *>(base + G::OFF_BAR);
    c.abort = reinterpret_cast<volatile int *>(base + G::OFF_ABORT);
    c.status = p.status;
    c.bound = wait_bound_of(p.status);
    c.short_polls = c.bound != kWaitBound;
    c.rank = 0;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + G::OFF_TSLOT);
    const int e0 = blockIdx.x * G::SV, h = blockIdx.y, b = blockIdx.z;
    const Seq sq = seq_of(p, b);
    const int nchunks = (sq.len + kC - 1) / kC;
    c.zrec = p.zrec + ((size_t)zslot0(p, b, sq) * p.H + h) * kRecBytes;
    c.zstride = (size_t)p.H * kRecBytes;
    if (nchunks == 0) {                     // empty sequence: ht = h0; nothing else is set up
        if (p.ht)
            for (int i = threadIdx.x; i < G::SV * kDK; i += G::kThreads) {
                const size_t off = (((size_t)b * p.H + h) * p.dv + e0 + i / kDK) * kDK + i % kDK;
                p.ht[off] = p.h0 ? p.h0[off] : 0.f;
            }
        return;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kScanBars; ++i)
            mbar_init(c.bars + i, ((i >= SB_RFREE && i < SB_ZV) || (i >= SB_D1FREE && i < SB_FULLZ))
                                      ? (uint32_t)NH : 1u);   // RFREE, D1FREE: one arrival per half
        *c.abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(tslot, G::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = *tslot;
    grid_dep_wait();                        // the Z kernel is done and its records are visible

    if (threadIdx.x < 128 * NH)
        scan_chain<G>(c, p, threadIdx.x >> 7, e0, h, b, sq, nchunks);
    else
        scan_loader<G>(c, p, &tm_v, e0, h, sq, nchunks);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x < 32) tmem_dealloc(c.tmem, G::kTmemCols);
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

template <int GATE, bool GLA, bool STRONG, typename Tg>
cudaError_t launch_single_one(const FwdParams &p, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &g,
                              const CUtensorMap &v, const CUtensorMap &o, cudaStream_t s) {
    // The two value slices of a head (dv = 128) split the chunks they build (a pair).
    dim3 grid(p.dv / kDVS, p.H, p.B);
    {
      if (p.dv == 2 * kDVS) {
        auto kern = kda_fwd_tc_kernel<GATE, GLA, true, STRONG, Tg>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = STRONG ? 2 : 1;
        return cudaLaunchKernelEx(&cfg, kern, p, q, k, g, v, o);
      }
    }
    auto kern = kda_fwd_tc_kernel<GATE, GLA, false, STRONG, Tg>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = STRONG ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p, q, k, g, v, o);
}

// The single kernel as two launches: the first, with only the one-product Gram, notes a chunk
// whose decay is past its range; the second redoes the whole call with the sub-chunk Gram if the
// first noted one, and exits at once otherwise.  (The sub-chunk path compiled into the first
// kernel would cost it registers in its chunk loop; the second launch costs a few microseconds,
// fewer as a programmatic dependent launch, whose blocks take SMs as the first launch's finish
// and wait for its completion in the hardware.)  GATE_NONE has no decay: one launch.
template <int GATE, bool GLA, typename Tg>
cudaError_t launch_single(const FwdParams &p, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &g,
                          const CUtensorMap &v, const CUtensorMap &o, cudaStream_t s) {
    cudaError_t e = launch_single_one<GATE, GLA, false, Tg>(p, q, k, g, v, o, s);
    if (e != cudaSuccess || GATE == KDA_GATE_NONE) return e;
    return launch_single_one<GATE, GLA, true, Tg>(p, q, k, g, v, o, s);
}

template <class G>
cudaError_t launch_record_scan_cfg(const FwdParams &p, const CUtensorMap &v, cudaStream_t s) {
    auto kern = kda_fwd_scan_kernel<G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G::kSmem);
    if (e != cudaSuccess) return e;
    // a programmatic dependent launch: its blocks set up while the Z kernel's last blocks run
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.dv / G::SV, p.H, p.B);
    cfg.blockDim = dim3(G::kThreads, 1, 1);
    cfg.dynamicSmemBytes = G::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, v);
}

// The record scan's configuration: both value slices of a dv = 128 head in one CTA when one
// CTA per 64-wide slice would take more than one wave of SMs (the head form halves the waves);
// otherwise one CTA per slice, whose products run on a tensor pipe of their own.
constexpr int kScanHeadPolicy = 1;       // 0: slices always, 1: heads for multi-wave batches, 2: heads always
cudaError_t launch_record_scan(const FwdParams &p, const CUtensorMap &v, cudaStream_t s) {
    if (p.dv == 2 * kDVS && kScanHeadPolicy != 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                      cudaSuccess)
            sms = 0;
        const long long slice_ctas = 2LL * p.B * p.H;
        if (kScanHeadPolicy == 2 || (sms > 0 && slice_ctas > sms)) return launch_record_scan_cfg<ScanHead>(p, v, s);
    }
    return launch_record_scan_cfg<ScanSlice>(p, v, s);
}

// With chunk records (p.zrec set): the chunk-parallel Z kernel, then the record
// scan kernel; otherwise the single kernel, building Z itself.
template <int GATE, bool GLA, typename Tg>
cudaError_t launch_variant(const FwdParams &p, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &g,
                           const CUtensorMap &v, const CUtensorMap &o, cudaStream_t s) {
    {
        if (!p.zrec) return launch_single<GATE, GLA, Tg>(p, q, k, g, v, o, s);
        auto zk = kda_fwd_z_kernel<GATE, GLA, Tg>;
        cudaError_t e = cudaFuncSetAttribute(zk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kZSmemBytes);
        if (e != cudaSuccess) return e;
        const long long nblk = (long long)((p.T + kC - 1) / kC) * p.H * p.B;
        if (nblk > 0x7fffffffLL) return cudaErrorInvalidValue;
        zk<<<dim3((unsigned)nblk), kWyThreads, kZSmemBytes, s>>>(p, q, k, g);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return launch_record_scan(p, v, s);
    }
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
