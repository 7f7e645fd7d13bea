/*
 * coli_moe.h -- C ABI of the GB300 (sm_103a) decode-time MoE block: a device router and a
 * grouped int4 expert FFN with an on-device, fixed-order weighted reduce.
 *
 * Sources (web pages about the "colibri" int4 MoE engine), cited by page and section:
 *   [g4]     c/backend_cuda.cu commit history, commit "grouped MoE kernels were per-row-only"
 *   [router] c/backend_cuda.cu commit history, commit "First increment of the #431 plan"
 *   [tcgate] c/backend_cuda.cu commit history, commit "The TC_W4A16 branch ..."
 *   [fixes]  c/backend_cuda.cu commit history, commit "Three vendor-neutral fixes to backend_cuda.cu"
 *   [pipe]   c/backend_cuda.cu commit history, commit "GPU resident pipeline ..."
 *   [resid]  PR #434 "COLI_CUDA_RESID=1", section "What"
 *   [attn]   c/backend_cuda.cu commit history, commit "CUDA batch MLA attention, kv_b head-sharding,
 *            fused o_proj, expert-group dispatch, W4A16 kernels"
 *   [q651]   PR #651, comment "Follow-up decode experiments" (Nsight kernel shares)
 *   [tier]   PR #651 "cuda: add experimental lossless compressed expert tier"
 *
 * Conventions shared by every call:
 *  - Return value: COLI_OK (0) or a negative COLI_E_* code. A failed call leaves no CUDA error
 *    pending for the next call (the runtime error is consumed on the failure path, [fixes] 2).
 *    coli_last_error() gives a one-line description of the last failure on that context.
 *  - Pointers to activations, routes and outputs are DEVICE pointers owned by the caller; the
 *    library never frees them. Weights passed to coli_expert_upload may be host or device
 *    pointers; the library copies them and owns the copy.
 *  - Compute calls are asynchronous on the context's stream: they validate arguments on the host,
 *    enqueue kernels and return. They never synchronise and never copy to the host.
 *  - Errors found by kernels (an expert index outside the table or naming an unset entry, a
 *    non-finite activation or router score) are recorded in a per-context device error word;
 *    coli_check_error() synchronises the stream, returns that code and clears it. Kernels never
 *    trap.
 *  - Test hook: if the environment variable COLI_FAIL_AFTER=N is set when a context is created,
 *    every compute call after the first N successful ones returns COLI_E_INJECTED without
 *    launching anything ([fixes] 3). Uploads, frees, table updates and queries are never gated.
 *  - A context is used by one host thread at a time.
 */
#ifndef COLI_MOE_H
#define COLI_MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define COLI_API __attribute__((visibility("default")))
#else
#define COLI_API
#endif

#define COLI_OK 0
#define COLI_E_INVAL -1      /* bad argument (NULL, size out of range, unknown dtype/handle) */
#define COLI_E_OOM -2        /* device allocation failed */
#define COLI_E_CUDA -3       /* a CUDA runtime call or kernel launch failed */
#define COLI_E_INJECTED -4   /* COLI_FAIL_AFTER test hook fired; nothing was launched */
#define COLI_E_FORMAT -5     /* weight format rejected: odd I, odd or negative gs, shape mismatch */
#define COLI_E_NONFINITE -6  /* (device) non-finite activation or router score */
#define COLI_E_ROUTE -7      /* (device) expert index outside the table or naming an unset entry */
#define COLI_E_TIMEOUT -8    /* (device) a bounded wait inside a kernel gave up (never expected) */

#define COLI_DTYPE_F32 0     /* IEEE binary32 */
#define COLI_DTYPE_BF16 1    /* bfloat16 (upper half of a binary32) */

/* Size limits of this build (checked on the host; beyond them a call returns COLI_E_INVAL). */
#define COLI_MAX_EXPERTS 4096   /* router E and expert-table entries */
#define COLI_MAX_K 32           /* experts per token */
#define COLI_MAX_DIM 32768      /* D and I */
#define COLI_MAX_TOKENS 65536   /* S for coli_router_select */
#define COLI_MAX_GROUP_TOKENS 1024  /* S for coli_expert_group */
#define COLI_MAX_GROUP_DIM 8192     /* D (model width) for coli_expert_group */
#define COLI_MAX_ISSUES 16          /* pending coli_expert_group_issue calls per round */

typedef struct coli_ctx coli_ctx;

/* Create a context on CUDA device `device` that enqueues work on `cuda_stream` (a cudaStream_t;
 * NULL = the legacy default stream). Returns COLI_E_CUDA if the device is unusable.
 * *out is set to NULL on failure. */
COLI_API int coli_init(coli_ctx **out, int device, void *cuda_stream);

/* Release every uploaded tensor, the expert table and the workspace. NULL is ignored. */
COLI_API void coli_destroy(coli_ctx *ctx);

/* Change the stream later calls enqueue on (e.g. a stream being captured into a CUDA graph). */
COLI_API int coli_set_stream(coli_ctx *ctx, void *cuda_stream);

/* Text of the last failure on this context ("" if none). Valid until the next call. */
COLI_API const char *coli_last_error(coli_ctx *ctx);

/* COLI_E_* code of the last failure on this context (COLI_OK if none), e.g. after an upload
 * returned handle 0. */
COLI_API int coli_last_code(coli_ctx *ctx);

/* Synchronise the context's stream; return and clear the device error word (COLI_OK if clean). */
COLI_API int coli_check_error(coli_ctx *ctx);

/* Pre-size the workspace for calls up to these sizes so that no later compute call allocates.
 * Without it, a compute call that needs more workspace than the last one allocates (once). */
COLI_API int coli_reserve(coli_ctx *ctx, int max_S, int max_E, int max_K, int max_D, int max_I);

/* Per-kernel timing: when on, every kernel launch of this context is bracketed by two CUDA events
 * recorded on the context's stream (off by default). Kinds: COLI_KERNEL_ROUTER, _GATEUP, _DOWN,
 * _COMBINE, _LINEAR. coli_profile_read synchronises the stream and returns, for one kind, the summed event
 * time in milliseconds and the number of launches since the previous read of that kind. */
#define COLI_KERNEL_ROUTER 0
#define COLI_KERNEL_GATEUP 1
#define COLI_KERNEL_DOWN 2
#define COLI_KERNEL_COMBINE 3
#define COLI_KERNEL_LINEAR 4
COLI_API int coli_profile_enable(coli_ctx *ctx, int on);
COLI_API int coli_profile_read(coli_ctx *ctx, int kind, double *total_ms, long long *launches);

/*
 * Device router, [router] (and the batched router of [pipe] for S > 1):
 *   z[s,e] = sum_j Wr[e,j] * x[s,j]                 (f32 logits GEMV, f32 accumulation)
 *   score[s,e]  = 1 / (1 + exp(-z[s,e]))           (sigmoid)
 *   choice[s,e] = score[s,e] + bias[e]             (bias-augmented; bias NULL = 0)
 *   idx[s,:] = K rounds of arg-max of choice over the not-yet-chosen experts with a strict '>'
 *              comparison, so a tie goes to the lower index; slots keep the selection order
 *   w[s,k]   = score[s, idx[s,k]]                  (weights from the raw, bias-free score)
 *   top-p (0 < topp < 1): p_k = w_k / sum_{k<K} w_k; keep the shortest prefix of slots whose
 *              running sum of p_k reaches topp (at least one slot); dropped slots get idx = -1
 *              and w = 0. topp <= 0 or >= 1 disables it.
 *   norm_topk != 0: w_k <- w_k / sum of the kept w; then w_k <- w_k * routed_scale.
 *   All sums of the last three steps run in slot order in binary32.
 * x: [S x D] row-major, dtype x_dtype. Wr: [E x D] row-major f32. bias: [E] f32 or NULL.
 * Outputs (device, caller-owned): idx [S x K] int32, w [S x K] f32, n_sel [S] int32 (kept slots
 * per token) or NULL. Limits: 1 <= K <= min(E, COLI_MAX_K), E <= COLI_MAX_EXPERTS.
 * A non-finite score sets COLI_E_NONFINITE in the device error word.
 * S < 16 with E <= 1024 runs as one kernel whose CTAs publish partial logits to the context's
 * router scratch and whose first CTA selects once every partial of a token has arrived; that
 * wait is bounded (2 s), after which the call sets COLI_E_TIMEOUT and writes an empty route
 * (n_sel 0, idx -1, w 0) for the token. The logits' summation order depends on the CTA grid
 * (COLI_ROUTER_ROWS / COLI_ROUTER_PARTS at coli_init), so near-tied experts may swap across grids.
 */
COLI_API int coli_router_select(coli_ctx *ctx, const void *x, int x_dtype, int S, int D,
                       const float *Wr, const float *bias, int E, int K, float topp,
                       int norm_topk, float routed_scale, int32_t *idx, float *w, int32_t *n_sel);

/*
 * coli_router_select with a shared expert ([attn], [pipe]): the same selection and weights, and
 * then the shared expert `shared` (a table id, 0 <= shared < COLI_MAX_EXPERTS, normally >= E so it
 * is never also routed) is placed right after each token's kept slots as one more kept slot with
 * weight exactly 1 (no normalisation, no routed scale). Outputs: idx [S x (K+1)], w [S x (K+1)],
 * n_sel [S] = kept routed slots + 1; the slots after the shared one hold idx = -1 and w = 0.
 * coli_expert_group with K + 1 then runs the routed experts and the shared expert in the same
 * launches and adds the shared expert's output after the routed ones, in slot order.
 * Limits as coli_router_select, with K + 1 <= COLI_MAX_K.
 */
COLI_API int coli_router_select_shared(coli_ctx *ctx, const void *x, int x_dtype, int S, int D,
                              const float *Wr, const float *bias, int E, int K, float topp,
                              int norm_topk, float routed_scale, int shared, int32_t *idx, float *w,
                              int32_t *n_sel);

/*
 * Same computation, arguments, outputs and error behaviour as coli_router_select, but the call
 * allocates nothing: no cudaMalloc or cudaFree and no allocating library call, whatever the size.
 * The router's pages have no counterpart for this entry; it serves callers that cannot let a call
 * allocate: a server that has given all free device memory to its own caching pool, or a decode
 * loop that cannot take the stall of cudaMalloc (which may synchronise the device) or of a
 * workspace that grows (which first waits for the context's stream).
 *   - Scratch: a fixed device array of the library, one per device (2.6 MiB), holding the
 *     one-kernel router's launch counter and partial logits (S < 16) and, for S >= 16, the
 *     (score, choice) pairs and partial logits of at most 65536 (token, expert) cells; S * E
 *     above that returns COLI_E_INVAL.
 *   - The first call on a device, and again the first call in a new CUDA context there (after a
 *     device reset, say), looks up that array's address (a CUDA symbol query with the context's
 *     device current); make that first call before any stream capture.
 *   - The array's launch counter only grows, so nothing is cleared between calls and each call
 *     is one kernel launch for S < 16 (three for S >= 16).
 *   - All contexts on a device share the array: calls whose kernels may run at the same time
 *     (different streams, contexts or unordered host threads) race on it and give wrong results.
 *   - Timed by coli_profile_enable as COLI_KERNEL_ROUTER, like coli_router_select.
 */
COLI_API int coli_router_select_noalloc(coli_ctx *ctx, const void *x, int x_dtype, int S, int D,
                       const float *Wr, const float *bias, int E, int K, float topp,
                       int norm_topk, float routed_scale, int32_t *idx, float *w, int32_t *n_sel);

/*
 * Upload one int4 weight tensor W [O x I], [g4]:
 *   packed: O rows of ceil(I/2) bytes; byte m of a row holds column 2m in its low nibble and
 *           column 2m+1 in its high nibble; the stored nibble n means the value n - 8.
 *   scales: gs == 0: O floats (one per row); gs > 0: O * ceil(I/gs) floats, row-major, one per
 *           row and per run of gs columns, the last run of a row being the tail group.
 *   W[o,i] = scale(o,i) * (n(o,i) - 8).
 * gs must be 0 or even (a byte never straddles two groups); I must be even. Host or device
 * pointers; the data are copied before the call returns, so the caller may free or overwrite
 * its buffers afterwards ([fixes] 1). Returns a nonzero handle, or 0 on failure (reason in
 * coli_last_error: COLI_E_FORMAT for a rejected format, COLI_E_OOM, COLI_E_CUDA).
 */
COLI_API uint64_t coli_expert_upload(coli_ctx *ctx, const uint8_t *packed, const float *scales, int O,
                            int I, int gs);

/* Shape of an uploaded tensor: O rows, I columns and its group size gs (any output pointer may be
 * NULL). COLI_E_INVAL for an unknown handle. */
COLI_API int coli_tensor_shape(coli_ctx *ctx, uint64_t handle, int *O, int *I, int *gs);

/* Free an uploaded tensor. It must not be referenced by the expert table (COLI_E_INVAL). */
COLI_API int coli_expert_free(coli_ctx *ctx, uint64_t handle);

/* Make expert e (0 <= e < COLI_MAX_EXPERTS) the triple (gate [I x D], up [I x D], down [D x I]).
 * Shapes are checked against each other and against every other entry of the table (all
 * experts share D and I): COLI_E_FORMAT on mismatch. Handles 0,0,0 clear the entry. */
COLI_API int coli_expert_table_set(coli_ctx *ctx, int e, uint64_t gate, uint64_t up, uint64_t down);

/*
 * Grouped expert FFN with weighting and a fixed-order reduce, [tcgate] [g4] [resid]:
 *   for each token s and kept slot k < n_sel[s] (all K if n_sel is NULL), with e = idx[s,k]:
 *     g = W_gate[e] x[s],  u = W_up[e] x[s]         (int4 x activation, f32 results)
 *     h = SiLU(g) * u = g / (1 + exp(-g)) * u       (f32)
 *     y_k = W_down[e] h                            (f32)
 *   y[s,:] = resid[s,:] + sum_{k < n_sel[s]} w[s,k] * y_k, the sum over slots formed in slot order
 *   without atomics, then added to the residual (resid NULL: y = the sum).
 * x_rows, resid, y: [S x D] row-major in x_dtype (f32 or bf16; bf16 values are widened exactly
 * and y is rounded to bf16 once at the end). idx, w, n_sel: as produced by coli_router_select,
 * device pointers. Slots with idx < 0 beyond n_sel are ignored. D and I come from the table.
 * Every weight byte of an expert is read once per call however many of the S tokens chose it.
 * Kernel forms, chosen on the host:
 *   - S == 1, every expert of the table streamable (D a multiple of 1024 and at most 6144, I a
 *     multiple of 16, every group size 0 or a multiple of 32): one persistent streaming kernel that
 *     runs each kept expert's gate, up and down rows as 16-row units, then a reduce kernel chained
 *     by programmatic dependent launch (profiled as COLI_KERNEL_GATEUP and COLI_KERNEL_COMBINE).
 *     The library keeps a panel-major copy of each such down tensor for it (made at table_set).
 *     COLI_DECODE_STREAM=0 in the environment at coli_init turns this form off.
 *   - Otherwise, S == 1: a gate/up kernel and a down kernel chained by programmatic dependent
 *     launch; with COLI_DECODE_FUSED=1 in the environment at coli_init, one cooperative kernel for
 *     the whole call (profiled as COLI_KERNEL_GATEUP) where the device supports cooperative launch
 *     and I <= 4096. These two forms give bit-identical y.
 *   - S > 1: the gate/up and down kernels over every token's routes, then a slot-ordered combine;
 *     bf16 batches with enough routed rows per expert run on the tensor cores instead ([tcgate]).
 */
COLI_API int coli_expert_group(coli_ctx *ctx, const void *x_rows, int x_dtype, int S,
                      const int32_t *idx, const float *w, const int32_t *n_sel, int K,
                      const void *resid, void *y);

/*
 * Resident issue/take, [resid] "What": the expert groups of one layer are issued one by one and
 * their results stay on the device; one take joins them to the residual. Nothing is copied to the
 * host and nothing synchronises, so a whole decode layer (router, issues, take) can be captured in
 * one CUDA graph.
 *
 * coli_expert_group_issue: the routes (x_rows, idx, w, n_sel, K as for coli_expert_group) are one
 * group; its weighted, slot-ordered sum  p_j[s,:] = sum_{k < n_sel[s]} w[s,k] * y_k  (no residual)
 * goes into the context's partial-sum slot j, kept in f32 whatever x_dtype is. Returns j >= 0, the
 * issue index of this round, or a negative COLI_E_* code. Every issue of a round must have the
 * same S, x_dtype and table D (COLI_E_INVAL otherwise), and at most COLI_MAX_ISSUES may be pending.
 * The first issue of a round sizes the slot pool (COLI_MAX_ISSUES x S x D floats; it may allocate
 * and wait for the stream): call coli_reserve first, or run one round, before any stream capture.
 *
 * coli_expert_group_take: y[s,:] = resid[s,:] + (p_0 + p_1 + ... + p_{n-1})[s,:], the partial sums
 * added in issue order in binary32 and then added to the residual (resid NULL: no residual); resid
 * and y are [S x D] in the round's x_dtype, device pointers. The round ends and the next issue
 * starts a new one. COLI_E_INVAL if nothing was issued; on a launch failure the round is kept.
 * With one issue holding all of a token's routes, y is bit-identical to coli_expert_group's.
 * The take is profiled as COLI_KERNEL_COMBINE.
 */
COLI_API int coli_expert_group_issue(coli_ctx *ctx, const void *x_rows, int x_dtype, int S,
                            const int32_t *idx, const float *w, const int32_t *n_sel, int K);
COLI_API int coli_expert_group_take(coli_ctx *ctx, const void *resid, void *y);

/*
 * Dense int4 projection: the one-tensor int4 matmul that [tcgate] names quant_matmul and that
 * [q651] measures as the largest kernel share of a decode step. For S tokens,
 *   y[t, o] = resid[t, o] + sum_i W[o, i] x[t, i]
 * with W an uploaded tensor [O x I] (coli_expert_upload; it may also be in the expert table) and
 * the same int4 x activation dot product as coli_expert_group (f32 results; bf16 activations are
 * widened exactly and y is rounded to bf16 once). x [S x I], resid [S x O] or NULL, y [S x O]:
 * row-major in x_dtype, device pointers. y may be resid (in place) but must not overlap x.
 * 1 <= S <= COLI_MAX_TOKENS. Every weight byte is read from HBM once per call for the first token;
 * the other tokens' passes over W mostly hit L2. COLI_E_INVAL for a bad handle, pointer, dtype or
 * S. Profiled as COLI_KERNEL_LINEAR.
 */
COLI_API int coli_w4_linear(coli_ctx *ctx, uint64_t W, const void *x, int x_dtype, int S, const void *resid,
                            void *y);

/*
 * Expert parallelism over `world` GPUs, the device steps ([resid] reduces the device groups' partial
 * sums in a fixed order; [pipe] spreads the expert groups over the cards). Expert e belongs to rank
 * e mod world. Each rank routes every token itself (coli_router_select is deterministic), keeps its
 * own routes with coli_routes_shard, issues them (coli_expert_group_issue) and takes the partial sum
 * without a residual (coli_expert_group_take with resid NULL, f32 activations). The ranks' partial
 * rows are then gathered (a collective of the caller's choice) and summed here in rank order.
 *
 * coli_routes_shard: idx_out, w_out [S x K], n_out [S]: token t's kept slots (k < n_sel[t]; all K if
 * n_sel is NULL) whose expert e satisfies e mod world == rank, moved to the front in slot order; the
 * other slots get idx -1 and w 0. A kept slot with e < 0 or e >= COLI_MAX_EXPERTS belongs to no rank
 * and sets COLI_E_ROUTE in the device error word. 0 <= rank < world; device pointers.
 *
 * coli_partials_reduce: y = resid + (((p_0 + p_1) + p_2) + ... + p_{n-1}) element by element in
 * binary32, with parts = n consecutive [S x D] f32 partials (device) and resid (NULL: none), y in
 * dtype ([S x D], device). Against one GPU the result differs only in the grouping of the slots'
 * terms. Profiled as COLI_KERNEL_COMBINE.
 */
COLI_API int coli_routes_shard(coli_ctx *ctx, const int32_t *idx, const float *w, const int32_t *n_sel, int S,
                               int K, int rank, int world, int32_t *idx_out, float *w_out, int32_t *n_out);
COLI_API int coli_partials_reduce(coli_ctx *ctx, const float *parts, int n, int S, int D, const void *resid,
                                  int dtype, void *y);

/*
 * Compressed expert tier, the codec ([tier]: experts kept as independently decodable 4096-byte ANS
 * blocks). Our own rANS over the nibbles of a packed byte stream: a per-stream table of 16 nibble
 * frequencies (12-bit probabilities, each >= 1), 4096-byte blocks, 32 interleaved 32-bit states per
 * block renormalised with 16-bit words (one lane of a warp per state when decoding). Lossless: the
 * decoded bytes equal the input exactly. Incompressible input (uniform nibbles) comes out slightly
 * larger than it went in; the caller compares the sizes (coli_ans_info) and keeps whichever it wants.
 *
 * coli_ans_encode_host: host only, no context. Writes the encoded stream of bytes[0..n) to out
 *   (cap bytes) and its length to *out_len; COLI_E_INVAL (with *out_len set) when cap is too small.
 * coli_ans_upload: encodes n host bytes and keeps the stream on the device; returns a handle (0 on
 *   failure, reason in coli_last_error).
 * coli_ans_info: the raw and stored sizes of an uploaded stream.
 * coli_ans_decode: decodes the whole stream into out (device, raw bytes), one warp per block, on the
 *   context's stream. A stream that fails its own consistency checks sets COLI_E_FORMAT in the device
 *   error word.
 * coli_ans_free: frees an uploaded stream (after the context's stream has drained).
 */
COLI_API int coli_ans_encode_host(const uint8_t *bytes, uint64_t n, uint8_t *out, uint64_t cap, uint64_t *out_len);
COLI_API uint64_t coli_ans_upload(coli_ctx *ctx, const uint8_t *bytes, uint64_t n);
COLI_API int coli_ans_info(coli_ctx *ctx, uint64_t handle, uint64_t *raw_bytes, uint64_t *stored_bytes);
COLI_API int coli_ans_decode(coli_ctx *ctx, uint64_t handle, uint8_t *out);
COLI_API int coli_ans_free(coli_ctx *ctx, uint64_t handle);

/*
 * Compressed tier, fused block decode + GEMV ([tier], comment "Fused decode/matvec feasibility
 * result": each block is decoded on chip and its row partials computed at once, writing only small
 * partial sums instead of the raw tensor). The uploaded stream (coli_ans_upload) must hold an int4
 * tensor W [O x I] in the packed format of coli_expert_upload: O rows of I/2 bytes, so raw bytes =
 * O * I / 2. For one token,
 *   y[o] = resid[o] + sum_i W[o, i] x[i],   W[o, i] = scale(o, i) (n(o, i) - 8)
 * with scales as for coli_expert_upload (gs == 0: [O] per row; gs > 0 and even: [O x ceil(I/gs)]),
 * a device pointer the caller keeps. Arithmetic in binary32: each decoded nibble's term
 * (n - 8) x[i] (times its group's scale when gs > 0) is summed per lane, the lanes' sums in lane
 * order per (block, row), a row's blocks in block order, then times the row scale (gs == 0) and
 * plus the residual; deterministic, bit-identical from run to run. x [I], resid [O] or NULL, y [O]:
 * x_dtype (f32 or bf16, y rounded to bf16 once), device pointers. Limits: I even, 256 <= I <= 16384.
 * COLI_E_INVAL for a bad handle, shape, pointer or dtype; a stream that fails its own consistency
 * checks sets COLI_E_FORMAT in the device error word. Profiled as COLI_KERNEL_LINEAR.
 */
COLI_API int coli_ans_w4_linear(coli_ctx *ctx, uint64_t handle, const float *scales, int O, int I, int gs,
                                const void *x, int x_dtype, const void *resid, void *y);

#ifdef __cplusplus
}
#endif

#endif /* COLI_MOE_H */
