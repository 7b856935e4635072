/*
 * kda.h -- C ABI of the GB300 (sm_103a) chunkwise gated delta-rule library.
 *
 * Recurrence (page "Diagonal Plus Low Rank", section 2, opening equation):
 *
 *     S_t = S_{t-1} Diag(alpha_t) (I - b_t a_t^T) + v_t k_t^T,   o_t = S_t q_t,
 *     S in R^{dv x dk},  alpha_t = exp(g_t),  S_{-1} = h0 (0 when absent).
 *
 * kda_chunk_fwd evaluates the KDA specialisation a = k, b = beta k with beta
 * scaling v (same page, "relation to KDA"; page "How to make GDN2 more
 * stable", eq. (1)) by the chunkwise form recapped on page "Kimi Delta
 * Attention backward" ("forward recap"):
 *
 *     Gamma = exp(in-chunk cumsum g),  Q<- = Q*Gamma, K<- = K*Gamma, K-> = K/Gamma,
 *     A~ = (I + Diag(beta)(K<- K->^T * M_{-1}))^{-1},
 *     W = A~ Diag(beta) K<-,  U = A~ Diag(beta) V,
 *     V_new = U - W S^T,  O = Q<- S^T + (Q<- K->^T * M) V_new,
 *     S <- S Diag(gamma^C) + V_new^T K-> Diag(gamma^C).
 *
 * The same call covers GDN (gate_kind = KDA_GATE_SCALAR), DeltaNet
 * (gate_kind = KDA_GATE_NONE) and GLA (beta = NULL and the flag
 * KDA_FLAG_BETA_SCALES_V cleared, so S_t = S_{t-1} Diag(alpha_t) + v_t k_t^T;
 * page "Gated Linear Attention", section 5.1).
 *
 * Conventions
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates or frees device memory.
 *   - Sequence tensors are contiguous [B, T, H, d] (d fastest); the state
 *     tensors h0 / ht are contiguous [B, H, dv, dk] float32 (row = value
 *     channel, column = key channel).  Device pointers must be 16-byte
 *     aligned, workspaces included (KDA_ERR_INVALID_ARG otherwise, where the
 *     entry point reads its workspace with vector or asynchronous copies).
 *   - Calls are asynchronous on the given stream.  Argument errors are
 *     detected on the host before anything is launched and nothing is
 *     written; the return value says which.  Errors found on the device
 *     (a bounded wait that ran out) are recorded in the first word of the
 *     workspace and read back with kda_status_read.  The forward also leaves,
 *     in words 1-6 of the workspace, where the first wait ran out (barrier,
 *     phase, thread, block, and the barriers its two issuing threads were on)
 *     for diagnosis; kda_status_read clears them with the status word.
 *   - Word 7 of the workspace (bytes 28-31, int32) is read by the bf16
 *     forward's kernels: when positive, the number of short polls (each
 *     suspends the waiting thread for at most about 32 ns) a bounded wait
 *     makes before it gives up (0: the library's default, far above any wait
 *     that ends).  It exists to exercise the failure path: a
 *     budget too small for the waits makes the launch end early with
 *     KDA_ERR_TIMEOUT recorded and its outputs undefined, after every copy
 *     and tensor-core product the kernels started has completed, so the next
 *     call runs normally.  kda_status_read leaves it as it is.
 *   - Word 8 of the workspace (bytes 32-35) belongs to the bf16 forward's
 *     single-kernel form, which notes there a call that needs its second
 *     launch (see kda_chunk_fwd); callers do not write it.
 *   - Outputs must not alias inputs.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kda_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,  /* null pointer, bad size, misalignment, bad enum */
    KDA_ERR_UNSUPPORTED = -2,  /* valid but not implemented (e.g. dk = 96) */
    KDA_ERR_WORKSPACE = -3,    /* workspace missing or smaller than the query */
    KDA_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed */
    KDA_ERR_TIMEOUT = -5,      /* a device-side bounded wait gave up */
    KDA_ERR_RANGE = -6         /* reserved: a log-decay beyond a kernel's range (no kernel of
                                  this version has such a limit; see kda_chunk_fwd) */
} kda_status;

typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype;

typedef enum {
    KDA_GATE_NONE = 0,     /* alpha = 1 (DeltaNet); g must be NULL */
    KDA_GATE_SCALAR = 1,   /* g [B, T, H]: one log-decay per token and head (GDN) */
    KDA_GATE_CHANNEL = 2   /* g [B, T, H, dk]: per-channel log-decay (KDA, GLA) */
} kda_gate;

/* beta scales v (KDA, GDN, DeltaNet).  Cleared: v enters unscaled (GLA). */
#define KDA_FLAG_BETA_SCALES_V 1u

typedef struct {
    int B, T, H;           /* batch, sequence length (any T >= 1), heads */
    int dk, dv;            /* key / value head dims: 64 or 128 each; bfloat16 inputs need
                              dk = 128 (dk = 64 returns KDA_ERR_UNSUPPORTED: the tensor-core
                              kernels are laid out for 128 key channels; float32 inputs take 64) */
    int chunk;             /* chunk length C; 64 (0 selects 64) */
    kda_dtype dtype;       /* dtype of q, k, v, beta and o */
    kda_gate gate_kind;
    kda_dtype g_dtype;     /* dtype of g (log-decay, g <= 0 expected) */
    unsigned flags;        /* KDA_FLAG_* */
    const void *q;         /* [B, T, H, dk] */
    const void *k;         /* [B, T, H, dk] */
    const void *v;         /* [B, T, H, dv] */
    const void *g;         /* see kda_gate; NULL iff gate_kind == KDA_GATE_NONE */
    const void *beta;      /* [B, T, H] in dtype; NULL means beta = 0 */
    const float *h0;       /* [B, H, dv, dk] initial state, or NULL (zero) */
    void *o;               /* [B, T, H, dv] output, dtype */
    float *ht;             /* [B, H, dv, dk] final state, or NULL (not written) */
    void *workspace;       /* device buffer, zero-filled before its first use */
    size_t workspace_bytes;
    /*
     * Packed variable-length batches, or NULL.  When given: B sequences lie
     * back to back in [1, T, H, d] tensors (q, k, v, g, beta, o), sequence i
     * in rows cu_seqlens[i] .. cu_seqlens[i + 1] - 1; h0 / ht stay [B, H, dv, dk],
     * one state per sequence.  A DEVICE array of B + 1 int32 with
     * 0 = cu_seqlens[0] <= ... <= cu_seqlens[B] = T, read by the kernels
     * (offsets outside [0, T] are clamped there); empty sequences are allowed
     * (their ht is h0).  Each sequence is independent: no state crosses a
     * boundary.  The pages batch only dense [B, T] sequences; this is a
     * boundary extension.
     */
    const int32_t *cu_seqlens;
} kda_fwd_args;

/*
 * Bytes of workspace kda_chunk_fwd runs fastest with for these arguments (0
 * on bad args): 256 for the status word, plus, for bfloat16 inputs, one
 * 66048-byte chunk record per chunk slot and head -- B * ceil(T / 64) slots,
 * or B + ceil(T / 64) with cu_seqlens -- except for batches whose
 * single-kernel CTAs fill between half and all of the SMs (there the query
 * returns 256 and the forward runs its single-kernel form).
 */
size_t kda_chunk_fwd_workspace(const kda_fwd_args *args);

/*
 * Chunkwise forward of the gated delta rule (KDA and its special cases).
 * Writes o, and ht when non-NULL.  float32 inputs run a float32 CUDA-core
 * kernel; bfloat16 inputs run the tcgen05 tensor-core path (bf16 operands,
 * fp32 accumulation, fp32 state).
 *
 * The workspace must be at least 256 bytes (KDA_ERR_WORKSPACE otherwise).
 * For bfloat16 inputs and workspace_bytes >= kda_chunk_fwd_workspace(args)
 * (when that is more than 256) the forward takes two kernels: a
 * chunk-parallel one writes every chunk's record into the workspace --
 * Z = [T ; P T] (T = (I + L)^{-1} Diag(beta) with L the masked
 * beta K<- K->^T, P the masked Q<- K->^T: the forward recap of page "Kimi
 * Delta Attention backward"), A_chain = [-W ; Q<- - P W] with W = T K<-
 * (GLA, beta = 0: Z = [I ; P], A_chain = [0 ; Q<-]), the rescaled K-> and
 * gamma^C -- then the scan kernel reads them; the
 * workspace must then be 16-byte aligned (KDA_ERR_INVALID_ARG otherwise).
 * With a smaller workspace, or where the query returns 256 (a batch whose
 * single-kernel CTAs, one per 64 values of each sequence and head, fill
 * between half of the GPU's SMs and all of them: there that form is faster),
 * the scan kernel builds Z itself in one kernel; both forms compute the same
 * values up to bf16 rounding (the record form applies beta to the rows of L
 * after the Gram product, the single kernel to the bf16 K<- operand before it).
 *
 * The decay has no range limit.  The bf16 path forms a chunk's Gram with one
 * tensor-core product over tiles rescaled by Gamma and 1/Gamma (page "Gated
 * Linear Attention", section 5.2) while the chunk's total log-decay, sum of g
 * over its 64 tokens, stays above -100 ln 2 (about -69) in every channel; a
 * chunk past that (detected on the device, chunk by chunk) takes that page's
 * secondary chunking (section 5.3): 16-token sub-chunks, products between
 * sub-chunks against a per-sub-chunk reference, pairs within a sub-chunk
 * element by element in float32.  float32 inputs form every Gram in the log
 * domain.  In the single-kernel form such a chunk makes the call take a
 * second launch (the first notes the call in word 8 of the status block, the
 * second redoes the call with the sub-chunk Gram; without such a chunk the
 * second launch exits at once).  A captured graph replays both launches with
 * the note of the capture: once a replay has met such a chunk, the second
 * launch of every later replay on the same workspace redoes the call too
 * (same results, at the sub-chunk form's cost) until the caller clears the
 * status block.
 */
kda_status kda_chunk_fwd(const kda_fwd_args *args, kda_stream_t stream);

/*
 * kda_chunk_fwd without a workspace from the caller, in its single-kernel
 * form.  The papers have no counterpart: this is library plumbing.
 *
 * Some callers cannot allocate device memory where they call the forward:
 * frameworks whose caching allocator owns all device memory and forbids
 * allocations outside its own arenas, plugins and embedded hosts that hand
 * the library nothing but the input and output tensors, and latency-critical
 * paths that cannot afford cudaMalloc, which may synchronise the device.
 * This entry point takes the same arguments as kda_chunk_fwd (workspace and
 * workspace_bytes are ignored) and uses instead an array owned by the
 * library: 256 bytes per device, held from library load until process exit.
 *   - Every call looks up the device address of the current device's array
 *     (a lookup, not an allocation: the address belongs to the current CUDA
 *     context, so none is kept between calls); the first call on a device may
 *     load the library's device code, so make it before any stream capture.
 *     `stream` must belong to the current device (KDA_ERR_INVALID_ARG
 *     otherwise).
 *   - Every call clears the array's status word on `stream`, then launches.
 *     All calls share the array, so calls that overlap on the GPU (unordered
 *     streams) race on it.
 *   - Runs the single-kernel form of kda_chunk_fwd (no chunk records), whose
 *     scratch is the 256-byte status block at any problem size, so no size
 *     that kda_chunk_fwd accepts is too large for the array.
 *   - A device-side wait that runs out is recorded in the shared array and
 *     cleared by the next call; to observe it, use kda_chunk_fwd with your
 *     own workspace and kda_status_read.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
kda_status kda_chunk_fwd_noalloc(const kda_fwd_args *args, kda_stream_t stream);

/* -------------------------------------------------------------- backward */

/*
 * Backward of kda_chunk_fwd: given dL/do (grad_o) and dL/dht (grad_ht), the
 * gradients of L with respect to q, k, v, g, beta and h0.  It follows the
 * chunk backward of page "Kimi Delta Attention backward": per chunk, in
 * reverse, with dS the gradient of the state after the chunk,
 *     dU = K-> Diag(gamma^C) dS^T + (Q<- K->^T * M)^T dO,   dW = -dU S_[t-1],
 *     dS_[t-1] = dS Diag(gamma^C) + dO^T Q<- - dU^T W,
 * then dQ, dK (both the K<- and K-> paths, with the output term), dV,
 * dbeta (the form without beta^{-1}), dlog Gamma and its in-chunk suffix sum
 * for dg.  The forward states are recomputed, not read from the forward call.
 * Same variants as kda_chunk_fwd (gate kinds, beta NULL, the v-scaling flag).
 */
typedef struct {
    int B, T, H;           /* as kda_fwd_args */
    int dk, dv;            /* 64 or 128 each */
    int chunk;             /* 0 (library's choice) or 32; the result does not depend on it */
    kda_dtype dtype;       /* dtype of q, k, v, beta, grad_o and of grad_q, grad_k, grad_v, grad_beta */
    kda_gate gate_kind;
    kda_dtype g_dtype;     /* dtype of g and of grad_g */
    unsigned flags;        /* KDA_FLAG_* */
    const void *q, *k, *v, *g, *beta;   /* the forward's inputs, layouts of kda_fwd_args */
    const float *h0;       /* [B, H, dv, dk] or NULL */
    const void *grad_o;    /* [B, T, H, dv] dL/do */
    const float *grad_ht;  /* [B, H, dv, dk] dL/dht, or NULL (zero) */
    void *grad_q;          /* [B, T, H, dk] out */
    void *grad_k;          /* [B, T, H, dk] out */
    void *grad_v;          /* [B, T, H, dv] out */
    void *grad_g;          /* layout of g, out; NULL iff g is NULL */
    void *grad_beta;       /* [B, T, H] out; NULL iff beta is NULL */
    float *grad_h0;        /* [B, H, dv, dk] out, or NULL (not written) */
    void *workspace;       /* device buffer of kda_chunk_bwd_workspace bytes; its first 256
                              bytes zero-filled before the first use */
    size_t workspace_bytes;
    /*
     * Packed variable-length batches, or NULL: as in kda_fwd_args (B sequences back
     * to back in [1, T, H, d] tensors -- q, k, v, g, beta, grad_o and the gradients of
     * those -- h0, grad_ht and grad_h0 one [H, dv, dk] state per sequence, a DEVICE
     * array of B + 1 int32 offsets, clamped into [0, T] by the kernels).  Gradients
     * do not cross a sequence boundary; an empty sequence's grad_h0 is its grad_ht.
     */
    const int32_t *cu_seqlens;
} kda_bwd_args;

/*
 * Bytes of workspace kda_chunk_bwd needs (0 on bad args): 256 for the status
 * word, then, with NS chunk slots per head (B ceil(T/32); B + ceil(T/32) with
 * cu_seqlens), the float32 chunk states and state gradients,
 * (2 NS + B) H dv dk 4 bytes, one float32 record of state-independent chunk
 * operands per slot, NS H (3 32 32 + 3 32 dk + 32 dv + dk) 4 bytes, and the
 * chunk products V_new and dU, 2 NS H 32 dv 4 bytes.
 */
size_t kda_chunk_bwd_workspace(const kda_bwd_args *args);

/*
 * Backward of the chunkwise gated delta rule: four kernels with float32
 * accumulation.  For bfloat16 inputs the chunk products run as warp-level
 * tf32 tensor-core MMAs (operands rounded to tf32); float32 inputs take exact
 * float32 products on the CUDA cores.
 */
kda_status kda_chunk_bwd(const kda_bwd_args *args, kda_stream_t stream);

/* ------------------------------------------------------------------ DPLR */

/*
 * General gated DPLR recurrence (page "Diagonal Plus Low Rank", section 2):
 *
 *     S_t = S_{t-1} Diag(alpha_t) (I - b_t a_t^T) + v_t k_t^T,   o_t = S_t q_t,
 *
 * with a_t, b_t given independently and v unscaled.  Evaluated by that
 * section's chunk form: per chunk, Gamma = exp(in-chunk cumsum g),
 * Q<- = Q*Gamma, K-> = K/Gamma, A-> = A/Gamma, B<- = B*Gamma;
 *     E = (I + (B<- A->^T * M_{-1}))^{-1},  W = E B<-,
 *     C = -E (B<- K->^T * M_{-1}) V,        X = C - W S^T,
 *     O = Q<- S^T + (Q<- K->^T * M) V + (Q<- A->^T * M) X,
 *     S <- (S + V^T K-> + X^T A->) Diag(gamma^C).
 * Layouts, ownership, stream semantics and error reporting are those of
 * kda_chunk_fwd.
 *
 * DPLR_FLAG_CLIP_GATE applies the stabilising clip of page "How to make GDN2
 * more stable", eq. (7), token by token before the recurrence:
 * Diag(alpha_t) -> min(Diag(alpha_t), 1/rho_t) with rho_t = ||I - b_t a_t^T||_2
 * from eq. (4), i.e. g -> min(g, -log rho_t) (with no gate, g = 0 is clipped).
 * It bounds every step's factor norm by 1.
 */
#define DPLR_FLAG_CLIP_GATE 1u

typedef struct {
    int B, T, H;           /* batch, sequence length (any T >= 1), heads */
    int dk, dv;            /* key head dim 64 or 128; value head dim a multiple of 32, <= 256 */
    int chunk;             /* 0 (library's choice) or 32; the result does not depend on it */
    kda_dtype dtype;       /* dtype of q, k, v, a, b and o */
    kda_gate gate_kind;
    kda_dtype g_dtype;     /* dtype of g */
    unsigned flags;        /* DPLR_FLAG_* */
    const void *q;         /* [B, T, H, dk] */
    const void *k;         /* [B, T, H, dk] */
    const void *v;         /* [B, T, H, dv] */
    const void *a;         /* [B, T, H, dk] */
    const void *b;         /* [B, T, H, dk] */
    const void *g;         /* see kda_gate; NULL iff gate_kind == KDA_GATE_NONE */
    const float *h0;       /* [B, H, dv, dk] initial state, or NULL (zero) */
    void *o;               /* [B, T, H, dv] output, dtype */
    float *ht;             /* [B, H, dv, dk] final state, or NULL (not written) */
    void *workspace;       /* device buffer, zero-filled before its first use */
    size_t workspace_bytes;
    /* Packed variable-length batches, or NULL: as in kda_fwd_args (q, k, v, a, b, g and o
       [1, T, H, d]; h0 / ht one state per sequence; B + 1 int32 device offsets).
       dplr_factor_norms reads it only to count the T H tokens of the packed batch. */
    const int32_t *cu_seqlens;
} dplr_fwd_args;

/*
 * Bytes of workspace dplr_chunk_fwd needs for these arguments (0 on bad args):
 * 256 for the status word plus one float32 record of state-independent chunk
 * operands per 32-token chunk slot, NS H (4 32 dk + 2 32 dv + dk) 4 bytes with
 * NS = B ceil(T/32) (B + ceil(T/32) with cu_seqlens).
 */
size_t dplr_chunk_fwd_workspace(const dplr_fwd_args *args);

/*
 * Chunkwise forward of the general gated DPLR recurrence.  Writes o, and ht
 * when non-NULL.  Two kernels (chunk-parallel operands, then the state scan);
 * float32 arithmetic with tf32 tensor-core products for bfloat16 inputs,
 * exact float32 products for float32 inputs; o is rounded to the input dtype.
 */
kda_status dplr_chunk_fwd(const dplr_fwd_args *args, kda_stream_t stream);

/*
 * Per-token norms of the DPLR transition factors (page "How to make GDN2
 * more stable", eqs. (4) and (12)), for every (b, t, h) of args:
 *   rho  [B, T, H] float32: ||I - b a^T||_2 by eq. (4), with
 *        eta = |a| |b| and c = a.b / (|a| |b|)  (c = 1 when eta = 0);
 *   norm [B, T, H] float32: ||Diag(alpha)(I - b a^T)||_2, the largest
 *        singular value of the full factor, for which the page gives no
 *        closed form: the largest eigenvalue of its Gram matrix
 *        (Diag(alpha^2) plus a rank-2 term) by bisection on eigenvalue
 *        counts from Haynsworth's inertia additivity, in float32;
 *   maxes [2] float32: max over all tokens of rho and of norm.
 * With DPLR_FLAG_CLIP_GATE in args->flags, norm is that of the clipped
 * factor min(Diag(alpha), 1/rho)(I - b a^T), which is at most 1.
 * Reads a, b, g, flags and the sizes B, T, H, dk of args (q, k, v, o, h0, ht,
 * dv and the workspace are not used; the pointers may be NULL).  Any of rho, norm, maxes may be NULL (not written).
 */
kda_status dplr_factor_norms(const dplr_fwd_args *args, float *rho, float *norm, float *maxes,
                             kda_stream_t stream);

/*
 * Backward of dplr_chunk_fwd: given dL/do and dL/dht, the gradients of L with
 * respect to q, k, v, a, b, g and h0.  It follows the chunk backward of page
 * "Diagonal Plus Low Rank", section 3 (dC, dV_1, dW, dE, dF, dQ<-, dB<-,
 * dK->, dA->, dV, dlog Gamma with the gamma^C row, and the dS recursion),
 * with dW taken against S_[t-1], dB from dB<-, and the state-update terms
 * V_1 dS Diag(gamma^C) and V_2 dS Diag(gamma^C) in dK-> and dA->.  With
 * DPLR_FLAG_CLIP_GATE the forward's clip is differentiated too: the gate's
 * gradient reaches g where g < -log rho and a, b through eq. (4) elsewhere.
 */
typedef struct {
    int B, T, H;           /* as dplr_fwd_args */
    int dk, dv;            /* 64 or 128 each */
    int chunk;             /* 0 (library's choice) or 16; the result does not depend on it */
    kda_dtype dtype;       /* dtype of q, k, v, a, b, grad_o and of their gradients */
    kda_gate gate_kind;
    kda_dtype g_dtype;     /* dtype of g and of grad_g */
    unsigned flags;        /* DPLR_FLAG_* */
    const void *q, *k, *v, *a, *b, *g;   /* the forward's inputs */
    const float *h0;       /* [B, H, dv, dk] or NULL */
    const void *grad_o;    /* [B, T, H, dv] dL/do */
    const float *grad_ht;  /* [B, H, dv, dk] dL/dht, or NULL (zero) */
    void *grad_q, *grad_k; /* [B, T, H, dk] out */
    void *grad_v;          /* [B, T, H, dv] out */
    void *grad_a, *grad_b; /* [B, T, H, dk] out */
    void *grad_g;          /* layout of g, out; NULL iff g is NULL */
    float *grad_h0;        /* [B, H, dv, dk] out, or NULL */
    void *workspace;       /* dplr_chunk_bwd_workspace bytes; first 256 zero-filled before first use */
    size_t workspace_bytes;
    /* Packed variable-length batches, or NULL: as in kda_bwd_args. */
    const int32_t *cu_seqlens;
} dplr_bwd_args;

/*
 * Workspace bytes for dplr_chunk_bwd (0 on bad args): 256, then, with NS chunk
 * slots per head (B ceil(T/16); B + ceil(T/16) with cu_seqlens), the float32
 * chunk states and state gradients (2 NS + B) H dv dk 4, one record of
 * state-independent chunk operands per slot, NS H (4 16 dk + 16 dv + 4 16 16 + dk) 4,
 * and the chunk products X and dC, 2 NS H 16 dv 4.
 */
size_t dplr_chunk_bwd_workspace(const dplr_bwd_args *args);

/*
 * Backward of the general gated DPLR recurrence: four kernels with float32
 * accumulation; tf32 warp-level tensor-core products for bfloat16 inputs,
 * exact float32 products for float32 inputs.
 */
kda_status dplr_chunk_bwd(const dplr_bwd_args *args, kda_stream_t stream);

/*
 * Reads the device status word that kernels set on a device-side error,
 * waits for the stream, clears the word and returns the code (KDA_OK when
 * no error was recorded).
 */
kda_status kda_status_read(void *workspace, kda_stream_t stream);

/* Static English text for a status code. */
const char *kda_status_string(kda_status status);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
