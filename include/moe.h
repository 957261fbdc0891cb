/*
 * moe.h -- C ABI of the B300 (sm_103a) top-k Mixture-of-Experts layer forward.
 *
 * The layer, as the "Mixture of Experts" lesson of AI Engineering from Scratch
 * (Phase 07, section "Concept") writes it:
 *
 *     scores = router(norm(h))                       (N tokens x E experts)
 *     top_k  = argmax_k(scores + bias)               (bias picks, never weighs)
 *     out    = h + shared(norm(h)) + sum_{e in top_k} gate_e * Expert_e(norm(h))
 *
 * with every expert a SwiGLU FFN.  Five steps run it: router + top-k + gates
 * (moe_router_topk_split after moe_router_split on tensor cores, or moe_router_topk on
 * CUDA cores), histogram + scan + permute (moe_permute; moe_permute_capacity drops
 * slots over an expert capacity; moe_permute_noalloc uses library-owned scratch),
 * grouped SwiGLU GEMMs (moe_grouped_swiglu on permuted rows, or
 * moe_grouped_swiglu_gather reading the rows through the permutation), un-permute +
 * gated combine (moe_unpermute_combine), and the +-gamma bias step (moe_bias_update).
 *
 * Conventions shared by every call
 *  - Pointers are DEVICE pointers owned by the caller unless a parameter says
 *    otherwise.  The library never allocates device memory; scratch space is
 *    passed in by the caller.
 *  - Arrays are dense, row-major, and 16-byte aligned.
 *  - Every call is asynchronous on `stream` and returns a moe_status_t.  Host-side
 *    argument checks return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED before
 *    anything is launched; a launch failure returns MOE_ERR_CUDA.  Faults detected
 *    on the device (a pipeline wait that exceeded its time limit, an expert id or a
 *    gathered token index out of range) are recorded in a per-device status word,
 *    read by moe_last_device_status().  No call traps or aborts.
 *  - No call allocates, synchronises or otherwise waits on the host (except
 *    moe_last_device_status), so a sequence of calls can be captured in a CUDA graph
 *    once each entry point has run once on the device.
 *  - Results are deterministic: the same inputs give the same bits, run to run.
 *  - The library looks up the device addresses of its two module-scope device variables
 *    (the status word, the moe_permute_noalloc scratch) once per device and keeps them
 *    for the life of the process; a cudaDeviceReset while the library is loaded
 *    invalidates them and is not supported.
 *  - Kernels are launched with programmatic dependent launch: each may start while the
 *    kernel before it on the stream drains, and waits for that kernel to complete before
 *    it touches global memory, so stream order means what it always does.  MOE_PDL=0 in
 *    the environment (read once per process) launches them plainly; results are the same.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* null/unaligned pointer, size out of range, bad id */
  MOE_ERR_UNSUPPORTED = -2, /* shape or dtype the library does not run */
  MOE_ERR_CUDA = -3,        /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_TIMEOUT = -4,     /* a device-side wait gave up (status word) */
  MOE_ERR_NAN_INPUT = -5    /* a router logit was NaN or infinite (status word) */
} moe_status_t;

typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;

/* Score function of the router.
 *  MOE_SCORE_SOFTMAX: selection on logit + bias; gates = softmax over the k chosen
 *    raw logits (lesson, "Build it", step 1).
 *  MOE_SCORE_SIGMOID: s = sigmoid(logit); selection on s + bias; gates = s_j / sum of
 *    the chosen s (the sigmoid router the handbook article names, read this way).
 *  MOE_SCORE_SQRT_SOFTPLUS: s = sqrt(ln(1 + e^logit)), read like the sigmoid router (the
 *    third router of the handbook post's question list). */
typedef enum moe_score_fn {
  MOE_SCORE_SOFTMAX = 0,
  MOE_SCORE_SIGMOID = 1,
  MOE_SCORE_SQRT_SOFTPLUS = 2
} moe_score_fn_t;

/* Largest E: 1024 for the tensor-core router, the permute and the grouped GEMM; 256 for
 * the CUDA-core fp32 router (moe_router_topk).  Largest k: 16. */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_EXPERTS_CUDA_CORE 256
#define MOE_MAX_TOPK 16

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status_t status);

/* Waits for `stream`, then returns and clears the status word of the current device.
 * The first that applies, in this order: MOE_ERR_TIMEOUT (a pipeline wait gave up),
 * MOE_ERR_INVALID_ARG (an expert id outside [0, E) reached moe_permute, or a token index
 * outside [0, N) reached moe_grouped_swiglu_gather), MOE_ERR_NAN_INPUT (a router logit
 * was NaN or infinite, so that token's gates are undefined), MOE_OK. */
moe_status_t moe_last_device_status(moe_stream_t stream);

/*
 * moe_selftest_bounded_wait -- run the failure-detection path of the library's pipelines.
 * No passage of the pages defines this call: it is a diagnostic.  Every tensor-core kernel
 * waits on its pipeline barriers with a bounded wait (about 2 s of SM cycles); when one runs
 * out, the kernel records MOE_ERR_TIMEOUT in the status word, lets the copies it started
 * land, frees its tensor memory and returns, so the context stays usable.  This call
 * launches one small kernel that waits, with the same code, on a barrier nothing arrives
 * on, using a limit of `limit_cycles` SM cycles (1000 .. the normal limit), next to a real
 * 4 KB bulk copy from `src` (a 16-byte-aligned device buffer of at least 4096 bytes) and a
 * second waiter.  Afterwards moe_last_device_status returns MOE_ERR_TIMEOUT and
 * steps_out[0] (device int32) is 15: the copy landed (1), the short wait gave up (2), the
 * second waiter left on the abort flag (4), and the kernel ended with its tensor memory
 * freed (8).  MOE_ERR_INVALID_ARG for a null or unaligned pointer or a limit out of range.
 */
moe_status_t moe_selftest_bounded_wait(const void* src, long long limit_cycles, int32_t* steps_out,
                                       moe_stream_t stream);

/* Library version, major*10000 + minor*100 + patch. */
int moe_version(void);

/*
 * moe_router_topk -- router GEMM, score function, biased top-k and gates.
 * Lesson "Build it" step 1 (router) and "Load-balancing problem" item 3 (the bias
 * changes which experts are chosen, never their gate weights); handbook article,
 * router-precision paragraph (the router runs in fp32).
 *
 *   xn        [N, D]  activations (norm(h)), MOE_BF16 or MOE_F32 (x_dtype)
 *   w_router  [E, D]  fp32 router weight
 *   bias      [E]     fp32 selection bias, or NULL for zero bias
 *   logits_out[N, E]  fp32 logits = xn . w_router^T, or NULL to skip writing them
 *   topk_idx  [N, k]  int32 chosen expert ids, in descending selection score; equal
 *                     scores are ordered by ascending id; NaN scores rank last
 *   topk_gate [N, k]  fp32 gate weights (sum to 1 per token)
 *   near_tie  [N]     uint8: 1 when the k-th and (k+1)-th selection scores differ by
 *                     less than 1e-6 (0 when k == E), or NULL
 * Requires 1 <= k <= min(E, 16), 1 <= E <= 256, D % 64 == 0, N >= 0.
 * Logits are accumulated in fp32 with per-32-element partial sums combined by
 * compensated (two-sum) addition.  (CUDA cores; see moe_router_topk_split for bf16.)
 * A NaN or infinite logit sets MOE_ERR_NAN_INPUT in the status word (the token is still
 * routed by the order rule above; its gates are undefined).
 */
moe_status_t moe_router_topk(const void* xn, moe_dtype_t x_dtype, int N, int D,
                             const float* w_router, const float* bias, int E, int k,
                             moe_score_fn_t fn, float* logits_out, int32_t* topk_idx,
                             float* topk_gate, uint8_t* near_tie, moe_stream_t stream);

/* Bytes of the split router weight moe_router_split writes: 3 * E * D bf16. */
size_t moe_router_split_bytes(int E, int D);

/*
 * moe_router_split -- write the fp32 router weight as three bf16 planes.
 * w_split [3, E, D] bf16 (plane 0 = hi, 1 = mid, 2 = lo) with w = hi + mid + lo exactly
 * for every finite w of magnitude above 2^-110 (each plane keeps the next 8 significant
 * bits).  Run once per change of w_router; moe_router_topk_split reads the planes.
 */
moe_status_t moe_router_split(const float* w_router, int E, int D, void* w_split, moe_stream_t stream);

/*
 * moe_router_topk_split -- moe_router_topk on tensor cores, for bf16 activations.
 * Same router as moe_router_topk (lesson "Build it" step 1; the handbook article's fp32
 * router): logits = xn . (hi + mid + lo)^T, every bf16 x bf16 product exact.  The three
 * planes' products are summed per 64-element slice of D in a fresh fp32 TMEM accumulator;
 * the slice partials hi + (mid + lo) are added in fp32 and folded into a two-sum
 * compensated total every 8 slices.  Short batches split D across CTAs; their partial
 * logits go to `workspace` and are added in split order.
 *   xn        [N, D] bf16
 *   w_split   [3, E, D] bf16 from moe_router_split
 *   logits_out[N, E] fp32 -- REQUIRED here (the top-k reads it back)
 *   workspace moe_router_topk_split_workspace_bytes(N, D, E) bytes (may be 0 / NULL)
 *   bias, topk_idx, topk_gate, near_tie, fn, k: as moe_router_topk.
 * Requires 1 <= k <= min(E, 16), 1 <= E <= 1024, D % 64 == 0.
 */
size_t moe_router_topk_split_workspace_bytes(int N, int D, int E);
moe_status_t moe_router_topk_split(const void* xn, int N, int D, const void* w_split,
                                   const float* bias, int E, int k, moe_score_fn_t fn,
                                   float* logits_out, int32_t* topk_idx, float* topk_gate,
                                   uint8_t* near_tie, void* workspace, size_t workspace_bytes,
                                   moe_stream_t stream);

/*
 * moe_router_topk_split_shared -- moe_router_topk_split and the shared expert's first GEMM
 * in one launch over the same 128-token tiles of xn (the router's split weight rows and the
 * shared expert's gate/up rows read against the same activation tiles, so xn comes from HBM
 * once; handbook news article, why bytes moved around the expert GEMMs matter).  Lesson
 * "Shared experts": the always-on expert's H = SiLU(xn ws_gate^T) * (xn ws_up^T).
 *   xn .. workspace_bytes   as moe_router_topk_split (the same logits, ids, gates and flags)
 *   ws_gate, ws_up [F, D]   bf16, the shared expert's gate and up projections; they must be
 *                           addressable as the two planes of one tensor (distance >= F*D*2
 *                           bytes, a multiple of 16), else MOE_ERR_UNSUPPORTED
 *   hs_out [N, F]           bf16 out: the shared expert's H, the same bits as the first GEMM of
 *                           moe_grouped_swiglu with G = 1, offsets {0, N}
 * Then moe_grouped_swiglu_shared_h runs its second GEMM in the routed experts' GEMM2 launch.
 * Requires F % 64 == 0 and the conditions of moe_router_topk_split; MOE_ERR_INVALID_ARG for
 * NULL ws_gate, ws_up or hs_out.
 */
moe_status_t moe_router_topk_split_shared(const void* xn, int N, int D, const void* w_split,
                                          const float* bias, int E, int k, moe_score_fn_t fn,
                                          float* logits_out, int32_t* topk_idx, float* topk_gate,
                                          uint8_t* near_tie, void* workspace, size_t workspace_bytes,
                                          const void* ws_gate, const void* ws_up, int F, void* hs_out,
                                          moe_stream_t stream);

/* Bytes of scratch moe_permute needs for (N, k, E). */
size_t moe_permute_workspace_bytes(int N, int k, int E);

/*
 * moe_permute -- per-expert histogram, exclusive scan and stable permutation.
 * Lesson "Build it" step 2 (count how often each expert fires) and the evaluation
 * article's per-expert routed-token histogram; the permutation groups each expert's
 * tokens into one contiguous block of rows for the grouped GEMM.
 *
 *   xn         [N, D]  rows to permute (dtype), or NULL together with x_perm
 *   topk_idx   [N, k]  int32 expert ids in [0, E) (from moe_router_topk, or replayed)
 *   counts     [E]     int32 out: number of (token, slot) pairs per expert
 *   offsets    [E + 1] int32 out: exclusive scan of counts; offsets[E] = N*k
 *   row_map    [N, k]  int32 out: permuted row of slot (n, j), or NULL
 *   perm_token [N*k]   int32 out: token of each permuted row, or NULL
 *   x_perm     [N*k, D] out: x_perm[row_map[n, j]] = xn[n], or NULL
 *   workspace  scratch of at least moe_permute_workspace_bytes(N, k, E) bytes
 * Rows of expert e occupy [offsets[e], offsets[e+1]) in slot order n*k + j (stable).
 * row_map and perm_token must be both given or both NULL; x_perm needs them.
 * An id outside [0, E) sets MOE_ERR_INVALID_ARG in the status word and is skipped.
 * moe_unpermute_combine skips slots whose row_map is -1.
 */
moe_status_t moe_permute(const void* xn, moe_dtype_t dtype, int N, int D,
                         const int32_t* topk_idx, int k, int E, int32_t* counts,
                         int32_t* offsets, int32_t* row_map, int32_t* perm_token,
                         void* x_perm, void* workspace, size_t workspace_bytes,
                         moe_stream_t stream);

/*
 * moe_expert_capacity -- slots per expert for a capacity factor C.
 * Lesson "Load-balancing problem" item 2: each expert processes at most a fixed share of
 * the batch, capacity = C * N / E tokens; read per (token, slot) assignment here:
 * ceil(C * N * k / E) slots, evaluated in double precision, capped at N * k (a capacity of
 * N * k already keeps every slot).  Host-only arithmetic; no device, no stream.
 * Returns -1 for C < 0 (or NaN), N < 0, k < 1 or E < 1.
 */
int64_t moe_expert_capacity(double capacity_factor, int N, int k, int E);

/*
 * moe_permute_capacity -- moe_permute with a per-expert capacity (token dropping).
 * Lesson "Load-balancing problem" item 2: each expert processes at most a fixed number of
 * tokens and the overflow skips the layer.  Read here per (token, slot) assignment: an
 * expert keeps the first `capacity` of its slots in slot order n*k + j; every later slot
 * gets row_map = -1, no row and no copy, so moe_unpermute_combine adds nothing for it (the
 * remaining gates are not renormalised).  For a capacity factor C use
 * capacity = moe_expert_capacity(C, N, k, E).
 *   counts   [E]     the routed demand (before dropping), which drives moe_bias_update
 *   offsets  [E + 1] exclusive scan of the kept counts min(counts, capacity)
 * Other arguments as moe_permute; perm_token / x_perm hold offsets[E] <= N*k rows.
 * capacity >= 0; capacity >= N*k keeps every slot (moe_permute itself).
 */
moe_status_t moe_permute_capacity(const void* xn, moe_dtype_t dtype, int N, int D,
                                  const int32_t* topk_idx, int k, int E, int capacity,
                                  int32_t* counts, int32_t* offsets, int32_t* row_map,
                                  int32_t* perm_token, void* x_perm, void* workspace,
                                  size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_permute_update_bias -- moe_permute_capacity, then the +-gamma bias step on the counts
 * it has just made, in the same launches (lesson "Build it" step 2: the firing counts of a
 * step drive the step's bias update; "Load-balancing problem" item 3: the bias only ever
 * changes which experts are chosen, so moving it once the step's routing is done is the
 * same as moving it after the whole forward).  Equivalent to moe_permute_capacity followed
 * by moe_bias_update(counts, E, N * k, gamma, bias, max_over_mean_out).
 *   gamma, bias [E] (fp32, in place, required), max_over_mean_out [1] (or NULL): as
 *   moe_bias_update; every other argument as moe_permute_capacity (capacity >= N * k keeps
 *   every slot).  With data-parallel replicas use moe_permute and, after summing the counts
 *   across replicas, moe_bias_update instead.
 */
moe_status_t moe_permute_update_bias(const void* xn, moe_dtype_t dtype, int N, int D,
                                     const int32_t* topk_idx, int k, int E, int capacity,
                                     int32_t* counts, int32_t* offsets, int32_t* row_map,
                                     int32_t* perm_token, void* x_perm, void* workspace,
                                     size_t workspace_bytes, float gamma, float* bias,
                                     float* max_over_mean_out, moe_stream_t stream);

/*
 * moe_permute_noalloc -- moe_permute without a caller-supplied workspace.
 * The pages have no counterpart to this call; it exists for callers that cannot
 * allocate device memory at all: a plugin handed only its input and output buffers
 * by a host framework that owns every device allocation, or code that must not take
 * the cost and device-wide synchronisation of cudaMalloc/cudaFree on its path.
 *
 * Arguments and results are those of moe_permute.  Its scratch (the per-chunk expert
 * histograms) lives in a fixed array inside the library, of
 * moe_permute_noalloc_max_scratch_bytes() bytes (256 KiB), which every GPU that loads
 * the library holds until the process exits.  A size needing more scratch than that
 * (moe_permute_workspace_bytes(N, k, E) larger than the array) is rejected with
 * MOE_ERR_UNSUPPORTED before anything is launched: the scratch is at most 128 token
 * chunks of E int32 counters, so every N is accepted while E <= 512, and at E = 1024
 * batches of at most N = 64 tokens.  No call allocates or frees memory.
 * The first call on a device looks up the array's device address once for that device
 * (a CUDA runtime query); make that first call before any stream capture.  All calls on
 * a device share the one array and nothing in it needs to start at zero; calls that
 * overlap on the GPU (on different streams without ordering) race on it and must not
 * be issued.
 */
size_t moe_permute_noalloc_max_scratch_bytes(void);
moe_status_t moe_permute_noalloc(const void* xn, moe_dtype_t dtype, int N, int D,
                                 const int32_t* topk_idx, int k, int E, int32_t* counts,
                                 int32_t* offsets, int32_t* row_map, int32_t* perm_token,
                                 void* x_perm, moe_stream_t stream);

/*
 * moe_grouped_swiglu -- every expert's SwiGLU FFN on its block of permuted rows.
 * Lesson "Concept" (each expert an independent SwiGLU FFN) and "Shared experts"
 * (call with G = 1 and offsets = {0, N} on xn for the always-on expert).
 *
 *   x_perm      [M_total, D]  rows grouped by expert (dtype)
 *   offsets     [G + 1]       DEVICE int32, non-decreasing, offsets[0] = 0,
 *                             offsets[G] <= M_total; rows of group g are
 *                             [offsets[g], offsets[g+1])
 *   w_gate,w_up [G, F, D]     gate and up projections (PyTorch Linear layout)
 *   w_down      [G, D, F]     down projection
 *   h_workspace [M_total, F]  scratch for H = SiLU(x W_gate^T) * (x W_up^T)
 *   y_perm      [M_total, D]  out: H W_down^T per row (rows past offsets[G] untouched)
 * MOE_BF16: tcgen05 tensor-core kernels, fp32 accumulation in tensor memory, H and Y
 *           rounded to bf16.  When the groups average at least 256 rows, two-CTA
 *           clusters share each 256-row tile (tcgen05 cta_group::2); otherwise one CTA
 *           per 128-row tile (M = 64 MMAs for a group's last <= 64 rows).  Both give the
 *           same bits.  The environment variable
 *           MOE_GROUPED_GEMM=pair or =single forces one of the two (read on every call).
 *           MOE_F32: CUDA-core fp32 kernels.
 * Requires D % 64 == 0, F % 64 == 0, 1 <= G.
 */
moe_status_t moe_grouped_swiglu(const void* x_perm, moe_dtype_t dtype, const int32_t* offsets,
                                int G, int M_total, int D, int F, const void* w_gate,
                                const void* w_up, const void* w_down, void* h_workspace,
                                void* y_perm, moe_stream_t stream);

/*
 * moe_grouped_swiglu_ex -- moe_grouped_swiglu on at most `max_ctas` CTAs (0 = one per
 * SM).  Same bits as moe_grouped_swiglu for any cap: each CTA walks the tile list with
 * a stride of the grid size, so a cap only shares the same tiles out among fewer CTAs
 * (a cap of 1 also rules out the CTA-pair kernel, which needs two).  SMs left over are
 * free for work on another stream.  MOE_ERR_INVALID_ARG for max_ctas < 0, otherwise the
 * argument rules and errors of moe_grouped_swiglu.
 */
moe_status_t moe_grouped_swiglu_ex(const void* x_perm, moe_dtype_t dtype, const int32_t* offsets,
                                   int G, int M_total, int D, int F, const void* w_gate,
                                   const void* w_up, const void* w_down, void* h_workspace,
                                   void* y_perm, int max_ctas, moe_stream_t stream);

/*
 * moe_grouped_swiglu_shared -- the routed experts' SwiGLU FFNs and the always-on shared
 * expert's, in the same two launches.  Lesson "Shared experts" (one expert every token
 * visits, added to the routed sum) and "Concept" (every expert a SwiGLU FFN).  The shared
 * expert's row tiles follow the routed experts' tiles in each launch's tile list, so it
 * needs no launches of its own and fills the routed tiles' last wave.  Same bits as
 * moe_grouped_swiglu (or moe_grouped_swiglu_gather) on the routed rows followed by
 * moe_grouped_swiglu with G = 1, offsets {0, N} on xn.
 *   x_perm, offsets, G, M_total, D, F, w_gate, w_up, w_down, h_workspace, y_perm:
 *                      as moe_grouped_swiglu (bf16 only)
 *   perm_token [M_total] DEVICE int32 or NULL: non-NULL gathers the routed rows from
 *                      xn[perm_token[i]] as moe_grouped_swiglu_gather does (x_perm is then
 *                      not read and may be NULL); NULL reads them from x_perm
 *   xn        [N, D]   the shared expert's rows (norm(h)); N = 0: no shared expert
 *   ws_gate, ws_up [F, D], ws_down [D, F]  the shared expert's weights (the same d_ff F)
 *   hs_workspace [N, F] scratch; shared_y [N, D] out
 * When the routed experts average 256 rows or more they run on the CTA-pair kernels first and
 * the shared expert runs alone in the one-CTA kernel.  MOE_ERR_INVALID_ARG for a non-NULL
 * perm_token with N = 0 and M_total > 0 (rows to gather, no tokens); MOE_ERR_UNSUPPORTED
 * when the shared gate and up weights cannot be addressed as the two planes of one tensor
 * map (their distance in memory below F*D*2 bytes or not a multiple of 16).
 */
moe_status_t moe_grouped_swiglu_shared(const void* x_perm, const int32_t* perm_token, const int32_t* offsets,
                                       int G, int M_total, int D, int F, const void* w_gate,
                                       const void* w_up, const void* w_down, void* h_workspace, void* y_perm,
                                       const void* xn, int N, const void* ws_gate, const void* ws_up,
                                       const void* ws_down, void* hs_workspace, void* shared_y,
                                       moe_stream_t stream);

/*
 * moe_grouped_swiglu_shared_h -- moe_grouped_swiglu_shared when hs_workspace already holds
 * the shared expert's H (from moe_router_topk_split_shared): the routed experts' two GEMMs,
 * and the shared expert's second GEMM as extra tiles of the routed GEMM2 launch.  Same
 * arguments minus ws_gate / ws_up; xn is read only when perm_token is given.  Same bits as
 * moe_grouped_swiglu_shared given the same H.
 */
moe_status_t moe_grouped_swiglu_shared_h(const void* x_perm, const int32_t* perm_token, const int32_t* offsets,
                                         int G, int M_total, int D, int F, const void* w_gate,
                                         const void* w_up, const void* w_down, void* h_workspace, void* y_perm,
                                         const void* xn, int N, const void* ws_down, void* hs_workspace,
                                         void* shared_y, moe_stream_t stream);

/*
 * moe_grouped_swiglu_gather -- moe_grouped_swiglu with the permutation folded into
 * the first GEMM: row i of expert input is read straight from xn[perm_token[i]], so
 * the permuted copy x_perm is never written.  Same arithmetic as moe_grouped_swiglu
 * on x_perm = xn[perm_token] (bit-identical H and Y).  Lesson "Concept" (experts
 * see their tokens only); the handbook news article's measurement of permute cost
 * against the expert GEMMs is why the copy is worth removing.
 *
 *   xn          [N, D]        bf16 activations (row stride D)
 *   perm_token  [M_total]     DEVICE int32 token of each permuted row, in [0, N)
 *                             for rows [0, offsets[G]) (from moe_permute)
 *   offsets, w_gate, w_up, w_down, h_workspace, y_perm: as for moe_grouped_swiglu
 * bf16 only (tcgen05 path).  Requires D % 64 == 0, F % 64 == 0, 1 <= G, N >= 1 when
 * M_total > 0; xn and every matrix 16-byte aligned.  A perm_token value outside
 * [0, N) is used as a zero row and sets MOE_ERR_INVALID_ARG in the status word
 * (moe_permute writes only valid ones).
 */
moe_status_t moe_grouped_swiglu_gather(const void* xn, int N, const int32_t* perm_token,
                                       const int32_t* offsets, int G, int M_total, int D, int F,
                                       const void* w_gate, const void* w_up, const void* w_down,
                                       void* h_workspace, void* y_perm, moe_stream_t stream);

/*
 * moe_unpermute_combine -- gather each token's k expert outputs and mix them.
 * Lesson "Concept": out = h + sum_j gate_j * Expert_j(norm(h)), plus the shared
 * expert's output with weight 1 ("Shared experts").
 *
 *   y_perm    [N*k, D]  expert outputs in permuted row order (dtype)
 *   row_map   [N, k]    int32 from moe_permute
 *   topk_gate [N, k]    fp32 gates
 *   shared_y  [N, D]    shared-expert output (dtype) or NULL
 *   residual  [N, D]    h (dtype) or NULL
 *   out       [N, D]    out (dtype)
 * The sum runs in fp32 in slot order j = 0..k-1, then adds shared_y and residual,
 * and is rounded once to dtype.
 */
moe_status_t moe_unpermute_combine(const void* y_perm, const int32_t* row_map,
                                   const float* topk_gate, int N, int k, int D,
                                   const void* shared_y, const void* residual, void* out,
                                   moe_dtype_t dtype, moe_stream_t stream);

/*
 * moe_bias_update -- the auxiliary-loss-free +-gamma step.
 * Lesson "Load-balancing problem" item 3 and "Build it" step 2: after a step, each
 * expert whose load is above the uniform target moves down by gamma, each below it
 * moves up by gamma:  bias[e] += gamma * sign(total/E - counts[e])  (sign(0) = 0),
 * evaluated exactly on integers and added in fp32.
 *
 *   counts            [E] int32 per-expert loads of the step (from moe_permute)
 *   total_assignments N*k of that step
 *   bias              [E] fp32, updated in place
 *   max_over_mean_out [1] fp32 out: max(counts) / (total/E), or NULL
 */
moe_status_t moe_bias_update(const int32_t* counts, int E, int64_t total_assignments,
                             float gamma, float* bias, float* max_over_mean_out,
                             moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
