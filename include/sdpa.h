/*
 * sdpa.h — C ABI of the GB300 fused scaled-dot-product attention library (libsdpa.so).
 *
 * The operation.  For query head h of batch b, with G = Hq / Hkv and KV head g = h / G:
 *     S   = scale · Q[b,h] · K[b,g]ᵀ                 (Lq × Lkv scores)
 *     S_ij = −∞ where is_causal and j > i + c        (causal mask; c = 0 top-left,
 *                                                   c = Lkv − Lq bottom-right)
 *     P   = softmax of each row of S
 *     O[b,h]   = P · V[b,g]
 *     lse[b,h,i] = ln Σ_j exp(S_ij)                  (natural log, scale included)
 * This is the definition in the NumPy "perform" sketch of the PyTensor issue "PERF: detect
 * scaled-dot-product-attention pattern and lower to mx.fast.scaled_dot_product_attention"
 * (section "Proposed change"), with the causal flag of F.scaled_dot_product_attention
 * ("mps-flash-sdpa 0.1.0", section "Quick Start") and grouped KV heads ("[Metal] Add Flash
 * Attention VJP for training", section "Key Features").  The logsumexp is the forward's
 * second output that the backward needs ("MPS scaled_dot_product_attention (SDPA)", section
 * "Problem - Unused second output tensor").  The backward is the vector-Jacobian product:
 *     dV[b,g] = Σ_{h in group g} Pᵀ·dO[b,h]
 *     dP = dO·Vᵀ,  δ_i = Σ_d dO_id·O_id,  dS = P ∘ (dP − δ)
 *     dQ[b,h] = scale · dS·K[b,g],   dK[b,g] = scale · Σ_{h in group g} dSᵀ·Q[b,h]
 * recomputing P from the cached logsumexp ("[Metal] Add Flash Attention VJP for training",
 * sections "Implementation Notes" and "Limitations": the backward requires the forward's
 * logsumexp).
 *
 * Conventions shared by every entry point:
 *  - is_causal: SDPA_CAUSAL_NONE (0), SDPA_CAUSAL_TOP_LEFT (1: key j hidden from query i
 *    when j > i, as the is_causal flag of F.scaled_dot_product_attention), or
 *    SDPA_CAUSAL_BOTTOM_RIGHT (2: hidden when j > i + Lkv − Lq, so the last query sees
 *    every key, the alignment a query chunk at the end of a longer KV sequence needs;
 *    requires Lq <= Lkv, else SDPA_ERR_UNSUPPORTED).  Other values: SDPA_ERR_INVALID_ARG.
 *  - Layout: for sdpa_fwd, sdpa_bwd and sdpa_bwd_noalloc every tensor is a dense,
 *    contiguous row-major [B, H, L, D] array of `dtype` (H = Hq for q, out, dout, dq;
 *    H = Hkv for k, v, dk, dv); sdpa_fwd_strided and sdpa_bwd_strided take the same
 *    tensors with per-tensor strides (see there).  lse is a dense fp32 [B, Hq, Lq] array.
 *    All pointers are DEVICE pointers (or managed memory) on the current CUDA device, and
 *    must be 16-byte aligned.
 *  - Ownership: the caller allocates and owns every buffer.  The library keeps only a
 *    static device error word and host-side counters.
 *  - Execution: every call enqueues work on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and returns without synchronising, except sdpa_poll_status.  The
 *    tensor-core backward forks its dK/dV kernel onto a library-owned stream of the
 *    highest priority (one per device, created on first use) and joins it back with
 *    events, so that its dQ kernel, on `stream`, runs concurrently; work enqueued on
 *    `stream` after the call still starts only when all of the call's work is done, and
 *    stream capture follows the fork and the join.
 *  - Outputs are fully overwritten; they need no zeroing.  Inputs must not overlap
 *    outputs.
 *  - Errors: argument errors are detected on the host before anything is launched and
 *    return SDPA_ERR_INVALID_ARG or SDPA_ERR_UNSUPPORTED; a failed launch returns
 *    SDPA_ERR_CUDA.  Kernels never trap: a wait that runs out of its iteration limit sets
 *    the device error word and the kernel returns; sdpa_poll_status reports it.
 *  - Supported: dtype in {SDPA_F32, SDPA_F16, SDPA_BF16}; D in {32, 64, 96, 128, 256}
 *    (fp16/bf16 run on tensor cores at every D, fp32 on the CUDA-core tiled kernels);
 *    B, Hq, Hkv, Lq, Lkv >= 1; Hq % Hkv == 0; Hq, B <= 65535; scale finite (0 allowed).
 */
#ifndef SDPA_GB300_H
#define SDPA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDPA_F32 = 0,
  SDPA_F16 = 1,
  SDPA_BF16 = 2
} sdpa_dtype_t;

typedef enum {
  SDPA_CAUSAL_NONE = 0,
  SDPA_CAUSAL_TOP_LEFT = 1,
  SDPA_CAUSAL_BOTTOM_RIGHT = 2
} sdpa_causal_t;

typedef enum {
  SDPA_OK = 0,
  SDPA_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size, overlap, bad scale */
  SDPA_ERR_UNSUPPORTED = 2,    /* valid but unsupported dtype / head dim / shape */
  SDPA_ERR_CUDA = 3,           /* a CUDA runtime call or kernel launch failed */
  SDPA_ERR_DEVICE_TIMEOUT = 4, /* a kernel's bounded wait ran out (reported by poll) */
  SDPA_ERR_WORKSPACE = 5       /* workspace missing or smaller than required */
} sdpa_status_t;

/*
 * Forward.  Computes out = softmax(scale·q·kᵀ [causal]) · v and, when lse != NULL, the
 * per-row logsumexp.  Pass lse = NULL when no gradient will be taken: it is then neither
 * computed nor written (the "second output only when needed" of "MPS
 * scaled_dot_product_attention (SDPA)", section "Problem - Unused second output tensor").
 *   q   [B,Hq,Lq,D]  dtype, read        k, v [B,Hkv,Lkv,D] dtype, read
 *   out [B,Hq,Lq,D]  dtype, written     lse  [B,Hq,Lq] fp32, written (nullable)
 * Needs no workspace.  Returns an sdpa_status_t.
 */
int sdpa_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
             int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale, int is_causal,
             int dtype, void* stream);

/*
 * Bytes of device workspace sdpa_bwd needs for these sizes (the fp32 δ = rowsum(dO∘O)
 * vector, [B,Hq,Lq], rounded up to 256 bytes).  Returns 0 for invalid arguments.
 */
size_t sdpa_bwd_workspace_size(int B, int Hq, int Hkv, int Lq, int Lkv, int D, int dtype);

/*
 * Backward.  Given the forward's inputs, its output `out` and logsumexp `lse` (both as
 * written by sdpa_fwd with the same arguments) and the output gradient `dout`, writes
 * dq, dk, dv.  dk and dv sum over the Hq/Hkv query heads that share each KV head; every
 * KV row is owned by one thread block, so no atomics are used and results are bitwise
 * reproducible run to run.
 *   q, out, dout, dq [B,Hq,Lq,D]  dtype      k, v, dk, dv [B,Hkv,Lkv,D]  dtype
 *   lse [B,Hq,Lq] fp32 (required)
 *   workspace: device buffer of at least sdpa_bwd_workspace_size(...) bytes, 16-byte
 *   aligned, owned by the caller, contents irrelevant on entry; it must stay untouched
 *   until the work enqueued by this call has finished.
 * Returns an sdpa_status_t (SDPA_ERR_WORKSPACE if the workspace is NULL or too small).
 */
int sdpa_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
             const float* lse, void* dq, void* dk, void* dv,
             int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale, int is_causal,
             int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Strided layouts.  sdpa_fwd and sdpa_bwd take contiguous [B,H,L,D] tensors.  These two
 * calls take every [B,H,L,D] tensor with its own element strides for the batch, head and
 * row dimensions (the D elements of a row stay contiguous), so that tensors stored as
 * [B,L,H,D] (one row per token holding all heads), or views into a fused [B,L,3,H,D]
 * projection output, are read and written in place instead of being copied to [B,H,L,D]
 * first (the pages' Metal kernel pays such transposes: "mps-flash-sdpa 0.1.0", section
 * "How It Works").  The operation, the other arguments and every other rule are those of
 * sdpa_fwd / sdpa_bwd; lse and the workspace stay contiguous [B,Hq,Lq] fp32.
 *  - Each stride, in bytes, must be a positive multiple of 16 (TMA and 16-byte vector
 *    access), and the layout must not map two elements of a tensor to the same address
 *    (checked: sorted by stride, each stride covers the extent of the smaller ones).
 *    Otherwise SDPA_ERR_INVALID_ARG.
 *  - Inputs may overlap one another (q, k, v as views of one buffer); outputs may overlap
 *    nothing, as measured by each tensor's address range [base, base + extent).
 * sdpa_fwd_strided reads strides->q, k, v and writes with strides->o; sdpa_bwd_strided
 * uses all eight (o is the forward output it reads).
 */
typedef struct {
  int64_t batch, head, row; /* element strides; the D elements of a row are contiguous */
} sdpa_layout_t;
typedef struct {
  sdpa_layout_t q, k, v, o, dout, dq, dk, dv;
} sdpa_strides_t;
int sdpa_fwd_strided(const void* q, const void* k, const void* v, void* out, float* lse,
                     int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale, int is_causal,
                     int dtype, const sdpa_strides_t* strides, void* stream);
int sdpa_bwd_strided(const void* q, const void* k, const void* v, const void* out, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv,
                     int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale, int is_causal,
                     int dtype, const sdpa_strides_t* strides, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * Attention sinks.  The strided calls plus one learned logit per query head, sinks[h],
 * that joins the softmax of every row of head h as one more entry with a zero value
 * vector: it enlarges each row's normaliser but contributes nothing to O.  In the notation
 * above, with σ = sinks[h]:
 *     P_ij = exp(S_ij) / (exp(σ) + Σ_j' exp(S_ij'))      O = P · V
 *     lse[b,h,i] = ln(exp(σ) + Σ_j exp(S_ij))
 *     dσ_h = −Σ_{b,i} exp(σ − lse[b,h,i]) · δ_{b,h,i}    (δ_i = Σ_d dO_id·O_id)
 * and dQ, dK, dV keep their formulas, with P recomputed from this lse.  The pages name
 * sinks, and their gradients, only as something the Metal backward leaves to unfused
 * operations ("[Metal] Add Flash Attention VJP for training", section "Limitations"); the
 * definition here is the usual one of a per-head sink logit.  Here they are fused: the
 * forward folds σ into each row's maximum and sum after its last key tile, the backward
 * kernels are unchanged, and dσ comes from one small kernel over lse and δ that sums in a
 * fixed order (bitwise reproducible).
 *   sinks  [Hq] fp32, natural-log units like S (read; NULL = no sink, the strided call);
 *          −inf means no sink for that head; +inf and NaN are not checked (NaN
 *          propagates to the head's outputs).
 *   dsinks [Hq] fp32, written with the sum over the batch (nullable; needs sinks).
 * Pointers are device pointers, 4-byte aligned; sinks may overlap no output, dsinks
 * nothing.  The backward's lse must be the one that sdpa_fwd_sinks wrote with the same
 * sinks.  Other arguments and rules are those of sdpa_fwd_strided / sdpa_bwd_strided.
 */
int sdpa_fwd_sinks(const void* q, const void* k, const void* v, void* out, float* lse,
                   const float* sinks, int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale,
                   int is_causal, int dtype, const sdpa_strides_t* strides, void* stream);
int sdpa_bwd_sinks(const void* q, const void* k, const void* v, const void* out, const void* dout,
                   const float* lse, const float* sinks, void* dq, void* dk, void* dv, float* dsinks,
                   int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale, int is_causal,
                   int dtype, const sdpa_strides_t* strides, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * Attention masks.  The sink calls plus an optional mask M over [B, Hq, Lq, Lkv] (indexed
 * by the query head), applied to the scores before the softmax:
 *   SDPA_MASK_BOOL      bytes; a nonzero byte keeps key j for query i, zero hides it (the
 *                       boolean attn_mask convention of F.scaled_dot_product_attention)
 *   SDPA_MASK_ADDITIVE  values of `dtype`, added to S = scale·q·k (−inf hides the key)
 * It combines with is_causal and with sinks.  The pages list masks with sinks among what
 * the Metal backward leaves to unfused operations ("[Metal] Add Flash Attention VJP for
 * training", section "Limitations"), and note that the Metal forward of "mps-flash-sdpa
 * 0.1.0" (section "When MFA Dispatches vs. Falls Back") takes only all-True boolean masks
 * and hands float masks and boolean masks with False values back; here both kinds are
 * fused into every kernel, forward and backward (dQ, dK, dV; the mask itself gets no
 * gradient).
 *  - A row that sees no key at all (possible only with a mask) gets O = 0, lse = −inf and
 *    zero gradients; with a sink, the sink alone fills that row's softmax.
 *  - Layout: element strides for batch, head and row (the keys of a row are contiguous);
 *    a stride of 0 broadcasts (e.g. {0, 0, Lkv_padded} for one [Lq, Lkv] mask shared by
 *    all batches and heads, {Lkv_padded, 0, 0} for a per-batch key-padding mask).  ptr and
 *    every row must be 16-byte aligned (strides in bytes multiples of 16), and each row
 *    must be readable up to the next multiple of 16 bytes past its Lkv elements (pad
 *    the key dimension); the padding's values are never used.  Otherwise
 *    SDPA_ERR_INVALID_ARG.  The mask is read only; it may overlap inputs, not outputs.
 *  - Cost: the tiles of keys that the causal bound skips are skipped with or without a
 *    mask; a mask that hides whole tiles still has them computed.
 * mask = NULL or kind SDPA_MASK_NONE is the sink call.  sdpa_bwd_masked must get the mask
 * the forward got.
 */
typedef enum {
  SDPA_MASK_NONE = 0,
  SDPA_MASK_BOOL = 1,
  SDPA_MASK_ADDITIVE = 2
} sdpa_mask_kind_t;
typedef struct {
  const void* ptr;          /* device pointer, 16-byte aligned */
  int kind;                 /* sdpa_mask_kind_t */
  int64_t batch, head, row; /* element strides (>= 0; 0 broadcasts) */
} sdpa_mask_t;
int sdpa_fwd_masked(const void* q, const void* k, const void* v, void* out, float* lse,
                    const float* sinks, const sdpa_mask_t* mask, int B, int Hq, int Hkv, int Lq,
                    int Lkv, int D, float scale, int is_causal, int dtype,
                    const sdpa_strides_t* strides, void* stream);
int sdpa_bwd_masked(const void* q, const void* k, const void* v, const void* out, const void* dout,
                    const float* lse, const float* sinks, const sdpa_mask_t* mask, void* dq,
                    void* dk, void* dv, float* dsinks, int B, int Hq, int Hkv, int Lq, int Lkv,
                    int D, float scale, int is_causal, int dtype, const sdpa_strides_t* strides,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward without a workspace argument: sdpa_bwd for callers that cannot allocate device
 * memory.  Such callers include code running inside a host application or framework that
 * owns every device allocation and hands its plugins nothing but their inputs and outputs,
 * code on a latency-critical path that must not call cudaMalloc (which can synchronise
 * the whole device), and code that runs while its own memory pool is locked.  The pages
 * this library follows have no counterpart to this call; it exists for those callers.
 *
 * Arguments, layouts and results are those of sdpa_bwd, minus the workspace.  The fp32 δ
 * scratch that sdpa_bwd keeps in the caller's workspace lives instead in a static device
 * array of SDPA_BWD_NOALLOC_MAX_ROWS floats (4 MiB) inside this library, which every GPU
 * that loads the library holds until the process exits.  The call allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine.
 *  - Limit: B·Hq·Lq must not exceed SDPA_BWD_NOALLOC_MAX_ROWS; larger problems return
 *    SDPA_ERR_WORKSPACE before anything is launched (use sdpa_bwd with a workspace).
 *  - The first call on each device looks up the array's device address (with that device
 *    current); make that first call before any stream capture begins.  The address is
 *    kept for the life of the process: the call assumes each device's primary context
 *    (the one the CUDA runtime uses) and no cudaDeviceReset while the library is loaded.
 *  - Every call shares the one array and it keeps the previous call's contents.  The
 *    backward writes every δ it reads before reading it, so nothing needs clearing, but
 *    calls whose work overlaps on the GPU (other streams, other host threads) race on the
 *    array: order them, e.g. on a single stream.
 * Returns an sdpa_status_t.
 */
#define SDPA_BWD_NOALLOC_MAX_ROWS (1u << 20)
int sdpa_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv,
                     int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale, int is_causal,
                     int dtype, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device error word that kernels set
 * when a bounded wait gives up.  Returns SDPA_OK, SDPA_ERR_DEVICE_TIMEOUT, or
 * SDPA_ERR_CUDA if the synchronisation itself reported an error.
 */
int sdpa_poll_status(void* stream);

/* A static, human-readable name for a status code. */
const char* sdpa_status_string(int status);

/*
 * Kernel family selection, for tests and measurements.  SDPA_PATH_AUTO (the default)
 * picks by shape and dtype: the vector path when Lq <= 8, (Hq/Hkv)·Lq <= 32 and D <= 128, else the
 * tensor-core tiled path for fp16/bf16 with D in {32, 64, 96, 128, 256}, else the CUDA-core
 * tiled path (every dtype, D up to 256).
 * A forced path that cannot serve a call makes that call return SDPA_ERR_UNSUPPORTED.
 * Process-wide setting; not thread-safe against concurrent calls.
 */
typedef enum {
  SDPA_PATH_AUTO = 0,
  SDPA_PATH_TENSOR = 1,  /* TMA + tcgen05 tiled kernels (fp16/bf16, D in {32,64,96,128,256}) */
  SDPA_PATH_SIMT = 2,    /* CUDA-core (FFMA) tiled kernels, every dtype and D */
  SDPA_PATH_VECTOR = 3   /* short-query kernels (Lq <= 8, (Hq/Hkv)·Lq <= 32, D <= 128) */
} sdpa_path_t;
int sdpa_set_path(int path); /* SDPA_OK, or SDPA_ERR_INVALID_ARG for an unknown path */

/* Number of kernels this library has launched since load (host-side counter). */
uint64_t sdpa_launch_count(void);

/*
 * Per-kernel device timing, for measurements.  While enabled, every kernel the library
 * launches is bracketed by two CUDA events recorded on the launch's stream, and the
 * backward runs its dK/dV and dQ kernels one after the other on `stream` (not
 * concurrently), so that each pair of events brackets one kernel's work alone;
 * sdpa_timing_read waits for the recorded events, adds their elapsed times into
 * per-kernel totals, and returns the total milliseconds and the number of timed launches
 * of one kernel kind since the last sdpa_timing_reset.  Process-wide, guarded by a mutex.
 * sdpa_timing_enable/read return an sdpa_status_t.
 */
typedef enum {
  SDPA_KERNEL_FWD = 0,      /* tiled forward (tensor-core or CUDA-core) */
  SDPA_KERNEL_DELTA = 1,    /* δ = rowsum(dO∘O) pre-pass */
  SDPA_KERNEL_DQ = 2,       /* tiled dQ kernel */
  SDPA_KERNEL_DKDV = 3,     /* tiled dK/dV kernel */
  SDPA_KERNEL_VEC_FWD = 4,  /* short-query forward */
  SDPA_KERNEL_VEC_BWD = 5,  /* short-query backward */
  SDPA_KERNEL_SINK_GRAD = 6, /* sink-logit gradients */
  SDPA_KERNEL_COUNT = 7
} sdpa_kernel_t;
int sdpa_timing_enable(int on);
int sdpa_timing_read(int kernel, double* total_ms, uint64_t* launches);
void sdpa_timing_reset(void);

/*
 * Failure-detection test hook.  Sets the time limit of every bounded wait inside the
 * kernels launched from now on (default 2 s) and, when `on` is non-zero, makes the next
 * tensor-core forward launch withhold its first K tile, so that the block's wait for it
 * runs out: the kernel then records SDPA_ERR_DEVICE_TIMEOUT in the device error word and
 * returns (no trap, no fault), and sdpa_poll_status reports it.  Returns SDPA_OK, or
 * SDPA_ERR_INVALID_ARG if wait_limit_ns is 0.
 */
int sdpa_debug_inject_timeout(int on, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif
#endif /* SDPA_GB300_H */
