/*
 * moe_gmm.h -- C ABI of the routed-expert MoE hot path on GB300 (sm_103a).
 *
 * The library computes the routed-expert part of a Mixture-of-Experts layer:
 *
 *   topk ids --permute--> expert-contiguous rows --GMM(gate_up)--> SwiGLU
 *            --GMM(down)--> weighted top-k combine --> y
 *
 * plus every gradient of it.  Sources, cited by page title and section:
 *
 *  [GMM]         "NPU Training Operators - GMM", section "算子语义" (operator
 *                semantics: x[sum(group_list), K], weight[E, K, N],
 *                group_list, the eager per-group loop, the worked example,
 *                grad_input_e = dY_e W_e^T, grad_weight_e = X_e^T dY_e) and
 *                section "Qwen3.5 MoE 路径" (permute -> histc -> GMM gate_up ->
 *                swiglu -> GMM down -> unpermute with probs).
 *  [MegaMoE]     "MegaMoE" operator doc, "计算公式" (topkIds INT32 [T, topK],
 *                topkWeights [T, topK], SiLU, the clip value c, swiglu) and
 *                "A16W16 非量化场景" (dispatch row(i,k), Linear1, activation,
 *                Linear2, Token Combine).
 *  [PermuteGrad] "CANN ops-transformer 算子详解 MoeTokenPermuteWithRoutingMapGrad",
 *                sections 2.2-2.3 (probs and token gradients), 3 (two-phase
 *                workspace-size + execute API), 4.2-4.3 (null / invalid
 *                argument errors), 5 (empty tensors need no workspace),
 *                6.2 (per token: walk topK slots, skip -1, fp32 accumulate).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - All tensor pointers are DEVICE pointers, row-major and contiguous, and
 *    must be 16-byte aligned.  The caller allocates and owns every buffer,
 *    including the workspace; the library allocates nothing.
 *  - bf16 tensors are raw bfloat16 bits (moe_bf16).  Matmuls accumulate in
 *    fp32 and round to bf16 (nearest even) once.
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream) and never synchronises the host, except moe_read_status.
 *  - Host-side argument checks return an error before anything is launched.
 *    Errors the device finds (an expert id outside [-1, E), a negative
 *    group count, sum(group_list) larger than the rows given, a row id out of
 *    range, a pipeline wait that timed out) are written to the status word
 *    at the start of the workspace; the first error sticks until
 *    moe_workspace_init clears it.  Read it with moe_read_status.
 *  - Every workspace must be zero-initialised once (moe_workspace_init)
 *    before its first use.  Calls that share a workspace must be ordered on
 *    one stream.
 *  - Empty problems (T == 0 or M == 0) are a successful no-op.
 *  - Sizes: E <= 1024; K, N, H and I multiples of 64 for the matmuls; k <= 64.
 */
#ifndef MOE_GMM_H
#define MOE_GMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;                 /* raw bfloat16 bits */
typedef struct CUstream_st* moe_stream_t;  /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_NULLPTR = 1,      /* a required pointer is NULL */
  MOE_ERR_INVALID = 2,      /* bad size, k > E, misaligned pointer, workspace too small */
  MOE_ERR_UNSUPPORTED = 3,  /* sizes outside what the kernels handle (see above) */
  MOE_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed */
  MOE_ERR_DEVICE = 5,       /* the device found bad data (ids, counts, row ids) */
  MOE_ERR_TIMEOUT = 6,      /* a bounded pipeline wait expired inside a kernel */
  MOE_ERR_BOUNDS = 7        /* bounds-checking build only: a kernel computed an index outside
                               the tensor it was about to access and skipped the access */
} moe_status_t;

enum { MOE_EPILOGUE_NONE = 0, MOE_EPILOGUE_SWIGLU = 1 };

/* Gated activations of the gate_up product ([MegaMoE] 激活函数公式), with
 * G = first I columns, U = last I columns, G_c = min(G, c), U_c = clip(U, -c, c):
 *   swiglu      A = SiLU(G_c) * U_c
 *   swiglustep  A = min(SiLU(G), c) * U_c
 *   swigluoai   A = G_c * sigmoid(alpha * G_c) * (U_c + beta)
 *   situglu     A = beta * tanh(G / beta) * sigmoid(G) * L(U),
 *               L(U) = U, or linear_beta * tanh(U / linear_beta) when given.
 * `params` holds the first n_params entries of the pages' activation_params
 * list ([MegaMoE] 参数说明): swiglu and swiglustep [] or [clamp]; swigluoai
 * [] or [clamp, alpha, beta]; situglu [], [beta] or [beta, linear_beta].
 * Missing values take the pages' defaults: clamp none (+inf; 0 also means
 * none), alpha 1.702, swigluoai beta 1.0, situglu beta 1.0 and L(U) = U.
 * clamp must be >= 0 and not NaN, alpha and beta finite, situglu's beta and
 * linear_beta finite and > 0; otherwise MOE_ERR_INVALID.  Gradients (the
 * pages give none) are the formulas' derivatives, with every min / clip kink
 * passing the gradient. */
typedef enum {
  MOE_ACT_SWIGLU = 0,
  MOE_ACT_SWIGLUSTEP = 1,
  MOE_ACT_SWIGLUOAI = 2,
  MOE_ACT_SITUGLU = 3
} moe_act_kind_t;

typedef struct {
  int32_t kind;      /* moe_act_kind_t */
  int32_t n_params;  /* 0 .. 3 */
  float params[3];
} moe_activation_t;

/* Weight layouts ([MegaMoE] 参数说明: transposeWeight1, transposeWeight2).
 * By default each expert's weight is [K, N] (w [E, K, N]); transposed it is
 * stored [N, K] (w [E, N, K]), and its gradient is produced in the same
 * layout.  The layer takes one bit per weight. */
enum { MOE_W_TRANSPOSED = 1 };
enum { MOE_W1_TRANSPOSED = 1, MOE_W2_TRANSPOSED = 2 };

/* Bytes at the start of every workspace that hold the device status word. */
#define MOE_STATUS_BYTES 256

/* ---------------------------------------------------------------- status */

/* Zero the status block of a workspace (asynchronous on stream). */
MOE_API moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Synchronise `stream` and return the sticky device status of `ws`
 * (MOE_OK, MOE_ERR_DEVICE or MOE_ERR_TIMEOUT), or MOE_ERR_CUDA if the stream
 * itself reports an error. */
MOE_API moe_status_t moe_read_status(const void* ws, moe_stream_t stream);

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_string(moe_status_t status);

/* Failure-detection check: runs one small kernel whose pipeline wait nothing
 * ever completes, using the same bounded mbarrier wait and shared abort flag
 * as the grouped-matmul kernels.  The waiting thread gives up after
 * timeout_ns (1 us .. 10 s) and raises the abort flag; a second warp waiting
 * on another barrier stops when it sees the flag; the kernel then writes
 * MOE_ERR_TIMEOUT to the workspace's status word and returns.  Expected
 * result: moe_read_status(ws) == MOE_ERR_TIMEOUT with the CUDA context still
 * usable.  ws: at least MOE_STATUS_BYTES, zeroed by moe_workspace_init. */
MOE_API moe_status_t moe_check_wait_timeout(void* ws, size_t ws_bytes, uint64_t timeout_ns, moe_stream_t stream);

/* Bounds-check self-check: one kernel thread asks the device-side bounds
 * check about an index one past the end of a range and accesses nothing.
 * Built with MOE_BOUNDS_CHECK=1 (libmoe_gb300_bounds.so) the check records
 * MOE_ERR_BOUNDS in the workspace's status word, as it would for any index a
 * kernel derives outside the tensor it is about to access (the access is
 * then skipped); the release library has no such checks and the status stays
 * MOE_OK.  ws: at least MOE_STATUS_BYTES, zeroed by moe_workspace_init. */
MOE_API moe_status_t moe_check_bounds(void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- dispatch */

/* Workspace bytes for moe_permute. */
MOE_API size_t moe_permute_workspace_size(int64_t T, int64_t k, int64_t E);

/* Token permute (dispatch): [GMM] "Qwen3.5 MoE 路径" (permute + histc) and the
 * worked example of "算子语义"; [MegaMoE] EP Dispatch (row(i,k)).
 *
 *   x          [T, H] bf16 tokens (may be NULL together with x_perm: index-only)
 *   topk_ids   [T, k] int32 expert ids in [-1, E); -1 marks an unused slot
 *   x_perm     [T*k, H] bf16 out: rows grouped by expert; within an expert,
 *              rows follow ascending flat slot index f = t*k + j (a stable
 *              counting sort).  Only the first R = sum(group_list) rows are
 *              written.
 *   group_list [E] int64 out: rows per expert (a histogram of topk_ids)
 *   row_id_map [T*k] int32 out: flat slot -> row, -1 for unused slots
 *   sorted_flat[T*k] int32 out: row -> flat slot for rows < R, -1 after R
 */
MOE_API moe_status_t moe_permute(const moe_bf16* x, const int32_t* topk_ids,
                         int64_t T, int64_t H, int64_t k, int64_t E,
                         moe_bf16* x_perm, int64_t* group_list,
                         int32_t* row_id_map, int32_t* sorted_flat,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/* The same permute for callers that cannot allocate device memory, and so
 * cannot supply a workspace: code running where cudaMalloc is not allowed
 * (a host framework whose allocator owns all device memory, a plugin or
 * embedded runtime with a fixed memory budget, a path that must not wait on
 * the driver's allocator).  The pages have no counterpart to this entry point;
 * it exists for those callers.
 *
 * Same arguments, outputs and results as moe_permute, with no workspace:
 *   device_status  NULL, or a 4-byte-aligned device word the caller owns and
 *                  zeroes; bad ids set it to MOE_ERR_DEVICE (sticky, like the
 *                  workspace word).  A misaligned word gives MOE_ERR_INVALID.
 * Scratch: one fixed device array inside the library, 512 KiB of int32
 * counters, held by every device that loads the library until the process
 * exits.  Sizes with ceil(T*k / 1024) * E > 131072 return MOE_ERR_UNSUPPORTED.
 * The first call in each CUDA context of a device looks up that array's
 * device address (with the device current), so a context rebuilt after
 * cudaDeviceReset gets its own; make that first call before any stream
 * capture.  Each rank block of the index pass reads every chunk's counters:
 * about (T*k / 1024)^2 * E * 4 bytes of L2 reads, 8 GB at the size limit.  It calls
 * no allocator.  All calls share the array, so calls whose kernels overlap on
 * the GPU race: order them on one stream. */
MOE_API moe_status_t moe_permute_no_alloc(const moe_bf16* x, const int32_t* topk_ids,
                         int64_t T, int64_t H, int64_t k, int64_t E,
                         moe_bf16* x_perm, int64_t* group_list,
                         int32_t* row_id_map, int32_t* sorted_flat,
                         uint32_t* device_status, moe_stream_t stream);

/* ---------------------------------------------------------------- grouped matmul */

/* Workspace bytes for gmm_forward / gmm_backward: the status block plus
 * 384 KiB in which the weight-gradient kernel rewrites its TMA descriptors
 * for each group (six 256-byte slots for each of up to 256 CTAs). */
MOE_API size_t gmm_workspace_size(int64_t M, int64_t K, int64_t N, int64_t E);

/* Grouped matmul forward: [GMM] "算子语义", y[s:e] = x[s:e] @ w[g] for group g
 * owning rows [s, e) = [cumsum before g, cumsum through g) of group_list.
 *
 *   x          [M, K] bf16, rows grouped by expert (M = rows of the buffer)
 *   w          [E, K, N] bf16
 *   group_list [E] int64 counts (device); sum must be <= M, rows at and past
 *              the sum are neither read for any group nor written
 *   epilogue   MOE_EPILOGUE_NONE:   y [M, N] = the product
 *              MOE_EPILOGUE_SWIGLU: N = 2I (gate = first I columns, up = last
 *                I), y [M, I] = SiLU(min(G,c)) * clip(U,-c,c) with G, U the
 *                bf16-rounded product ([MegaMoE] 激活函数公式); h_save, if not
 *                NULL, receives the bf16 product [M, N]
 *   clip       c; 0 means no clip (+inf); must be >= 0
 */
MOE_API moe_status_t gmm_forward(const moe_bf16* x, const moe_bf16* w, const int64_t* group_list,
                         int64_t M, int64_t K, int64_t N, int64_t E,
                         int epilogue, float clip, moe_bf16* y, moe_bf16* h_save,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/* gmm_forward with a gated-activation epilogue of any kind (see
 * moe_activation_t): N = 2I (a multiple of 256), y [M, I] = Activation(G, U)
 * of the bf16-rounded product; h_save as for MOE_EPILOGUE_SWIGLU.
 * activation NULL: no epilogue, y [M, N] = the product (h_save must be NULL).
 * w_flags: 0, or MOE_W_TRANSPOSED for w stored [E, N, K].  Bad activation
 * parameters or flags -> MOE_ERR_INVALID; an unknown kind -> MOE_ERR_UNSUPPORTED. */
MOE_API moe_status_t gmm_forward_act(const moe_bf16* x, const moe_bf16* w, const int64_t* group_list,
                             int64_t M, int64_t K, int64_t N, int64_t E,
                             const moe_activation_t* activation, int w_flags, moe_bf16* y, moe_bf16* h_save,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* Dispatch fused into the gate_up grouped matmul ([MegaMoE] "算子功能": the
 * dispatch and the first expert matmul with its activation in one operator;
 * the GMM of [GMM] "算子语义" over the permuted rows of [GMM] "Qwen3.5 MoE 路径").
 * Computes gmm_forward_act(x_perm, w, ...) with an activation, where the
 * permuted rows are never stored: row r of the grouped operand is token
 * sorted_flat[r] / k of x, fetched from x by the kernel (TMA gather of four
 * rows per copy).
 *   x           [T, K] bf16 tokens
 *   sorted_flat [M] int32 from moe_permute (row -> flat slot t * k + j); rows
 *               at and past sum(group_list) are not read
 *   w           [E, K, N] bf16 (or [E, N, K] with MOE_W_TRANSPOSED), N = 2I,
 *               a multiple of 256
 *   group_list  [E] int64 counts (device), sum <= M
 *   activation  required (the gated activation of the [gate | up] product)
 *   y           [M, N/2] bf16 out
 * Workspace: gmm_workspace_size(M, K, N, E).  A slot outside [0, T*k) in the
 * rows read sets MOE_ERR_DEVICE (the row reads token 0).  128-row tiles. */
MOE_API moe_status_t gmm_forward_gather_act(const moe_bf16* x, const int32_t* sorted_flat, int64_t T, int64_t k,
                             const moe_bf16* w, const int64_t* group_list,
                             int64_t M, int64_t K, int64_t N, int64_t E,
                             const moe_activation_t* activation, int w_flags, moe_bf16* y,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* Workspace bytes for moe_expert_mlp_forward: the status block and one int32
 * readiness count per 128-row tile (T*k/128 + E of them). */
MOE_API size_t moe_expert_mlp_workspace_size(int64_t T, int64_t k, int64_t E);

/* The routed experts' MLP over the permuted tokens in one launch ([MegaMoE]
 * "算子功能": the dispatch and the two expert matmuls with the activation
 * between them as one operator; [MegaMoE] "Expert Compute" 1-3):
 *   a  = gmm_forward_gather_act(x, sorted_flat, w1, activation)    [T*k, I]
 *   y2 = gmm_forward(a, w2)                                         [T*k, H]
 * bit for bit, as one persistent kernel: its CTAs first take the gate_up
 * tiles (rows gathered from x; row r of group g is token sorted_flat[r] / k),
 * then the down tiles, each of which waits until its 128 rows of `a` are
 * stored.  The CTAs wait for one another (bounded: a wait past 4 s gives
 * MOE_ERR_TIMEOUT), so they must all be resident at once: one per SM, as
 * launched.  Rows past sum(group_list) of a and y2 are not written.
 *   x [T, H] bf16; sorted_flat [T*k] int32 and group_list [E] int64 from
 *   moe_permute; w1 [E, H, 2I], w2 [E, I, H] bf16 (H % 64 == 0, I % 128 == 0);
 *   activation required; a [T*k, I] and y2 [T*k, H] bf16 out.
 * Workspace: moe_expert_mlp_workspace_size(T, k, E).  128-row tiles. */
MOE_API moe_status_t moe_expert_mlp_forward(const moe_bf16* x, const int32_t* sorted_flat, const int64_t* group_list,
                             const moe_bf16* w1, const moe_bf16* w2, int64_t T, int64_t H, int64_t I, int64_t E,
                             int64_t k, const moe_activation_t* activation, moe_bf16* a, moe_bf16* y2,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* Workspace bytes for gmm_forward_combine: the status block, ceil(N/256)
 * int32 counts (one per 256-column slice) and an [M, N] bf16 scratch for the
 * expert outputs. */
MOE_API size_t gmm_forward_combine_workspace_size(int64_t T, int64_t k, int64_t M, int64_t N);

/* The down grouped matmul fused with the weighted top-k combine ([MegaMoE]
 * "算子功能" and "Token Combine": y_i = sum_k w_k Y_{e_ik}[row(i,k)]):
 *   Y = gmm_forward(a, w) over the groups of group_list (never returned), and
 *   y[t] = sum over j in 0..k-1 with row_id_map[t*k+j] >= 0 of
 *          topk_w[t*k+j] * Y[row_id_map[t*k+j]],
 * summed in fp32 in slot order and rounded once to bf16: the same arithmetic,
 * and so the same bits, as gmm_forward followed by moe_unpermute.  The
 * matmul's tiles are visited 256 output columns at a time; once a slice is
 * stored, the tokens are summed over it while its rows are still in L2, and
 * the rows are then dropped from L2 unwritten.  The kernel's CTAs wait for one
 * another's slices (bounded: a wait past 4 s gives MOE_ERR_TIMEOUT), so they
 * must all be resident at once: one per SM, as launched.
 *   a           [M, K] bf16, rows grouped by expert; w [E, K, N] (or [E, N, K]
 *               with MOE_W_TRANSPOSED); group_list [E] int64 counts
 *   row_id_map, sorted_flat  [T*k] / [M] int32 from moe_permute
 *   topk_w      [T, k] fp32;  y [T, N] bf16 out (tokens without a routed slot
 *               get zeros)
 * Workspace: gmm_forward_combine_workspace_size(T, k, M, N).  Out-of-range
 * rows or slots set MOE_ERR_DEVICE.  128-row tiles. */
MOE_API moe_status_t gmm_forward_combine(const moe_bf16* a, const moe_bf16* w, const int64_t* group_list,
                             const int32_t* row_id_map, const int32_t* sorted_flat, const float* topk_w,
                             int64_t T, int64_t k, int64_t M, int64_t K, int64_t N, int64_t E, int w_flags,
                             moe_bf16* y, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Grouped matmul backward: [GMM] "算子语义" backward formulas
 *   dx[s:e] = dy[s:e] @ w[g]^T            (dx [M, K], NULL to skip)
 *   dw[g]   = x[s:e]^T @ dy[s:e]          (dw [E, K, N], NULL to skip;
 *                                          an empty group gets zeros)
 *   dy [M, N] bf16 upstream gradient. */
MOE_API moe_status_t gmm_backward(const moe_bf16* x, const moe_bf16* w, const int64_t* group_list,
                          const moe_bf16* dy, int64_t M, int64_t K, int64_t N, int64_t E,
                          moe_bf16* dx, moe_bf16* dw,
                          void* ws, size_t ws_bytes, moe_stream_t stream);

/* gmm_backward with a weight layout: w_flags MOE_W_TRANSPOSED reads w as
 * [E, N, K] and writes dw as [E, N, K] (dw[g] = dy[s:e]^T @ x[s:e]). */
MOE_API moe_status_t gmm_backward_ex(const moe_bf16* x, const moe_bf16* w, const int64_t* group_list,
                          const moe_bf16* dy, int64_t M, int64_t K, int64_t N, int64_t E, int w_flags,
                          moe_bf16* dx, moe_bf16* dw,
                          void* ws, size_t ws_bytes, moe_stream_t stream);

/* The input gradient of a grouped matmul followed by the SwiGLU gradient, in
 * one pass: the memory-saving backward of "03 · grouped GEMM path" (MegaBlocks),
 * section 4.3 -- the activation gradient is taken from the saved GMM output, and
 * here inside the dX epilogue, so dA is never stored:
 *   dA[s:e] = bf16(dy[s:e] @ w[g]^T)      (not written)
 *   dh[s:e] = SwiGLU'(h[s:e], dA[s:e])    ([MegaMoE] 激活函数公式 differentiated,
 *                                           clip c as in moe_swiglu_backward)
 *   dy [M, N], w [E, K, N], h [M, 2K] (gate | up) bf16 in; dh [M, 2K] bf16 out.
 * Equal, bit for bit, to gmm_backward's dx followed by moe_swiglu_backward. */
MOE_API moe_status_t gmm_backward_dx_swiglu(const moe_bf16* dy, const moe_bf16* w, const int64_t* group_list,
                          const moe_bf16* h, int64_t M, int64_t K, int64_t N, int64_t E, float clip,
                          moe_bf16* dh, void* ws, size_t ws_bytes, moe_stream_t stream);

/* gmm_backward_dx_swiglu for any gated activation: dh = Activation'(h, dA).
 * Equal, bit for bit, to gmm_backward's dx followed by moe_activation_backward. */
MOE_API moe_status_t gmm_backward_dx_act(const moe_bf16* dy, const moe_bf16* w, const int64_t* group_list,
                          const moe_bf16* h, int64_t M, int64_t K, int64_t N, int64_t E,
                          const moe_activation_t* activation, int w_flags, moe_bf16* dh,
                          void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- combine and gradients */

/* Workspace bytes for the combine-side entry points (just the status block). */
MOE_API size_t moe_unpermute_workspace_size(void);

/* Weighted combine: [MegaMoE] Token Combine, y[t] = sum_j w[t,j] * y_perm[row(t,j)],
 * fp32 accumulation in j order, one bf16 rounding; unused slots add nothing.
 *   y_perm [T*k, H] bf16, row_id_map [T*k] int32 (from moe_permute),
 *   topk_w [T, k] fp32 (NULL means every weight is 1), y [T, H] bf16 out. */
MOE_API moe_status_t moe_unpermute(const moe_bf16* y_perm, const int32_t* row_id_map, const float* topk_w,
                           int64_t T, int64_t H, int64_t k, moe_bf16* y,
                           void* ws, size_t ws_bytes, moe_stream_t stream);

/* Gradients of the combine: [PermuteGrad] 2.2 (probs) with the combine of
 * [MegaMoE] Token Combine differentiated:
 *   dy_perm[row(t,j)] = w[t,j] * dy[t]          ([T*k, H] bf16, rows >= R untouched)
 *   dprobs[t,j]       = <dy[t], y_perm[row(t,j)]> ([T, k] fp32; 0 for unused slots) */
MOE_API moe_status_t moe_unpermute_backward(const moe_bf16* dy, const moe_bf16* y_perm,
                                    const int32_t* row_id_map, const float* topk_w,
                                    int64_t T, int64_t H, int64_t k,
                                    moe_bf16* dy_perm, float* dprobs,
                                    void* ws, size_t ws_bytes, moe_stream_t stream);

/* Token gradient of the permute: [PermuteGrad] 2.3 and 6.2, index-add of the
 * permuted rows back onto their tokens, deterministic (fixed j order, fp32):
 *   dx[t] = sum_j dx_perm[row(t,j)]   (dx [T, H] bf16) */
MOE_API moe_status_t moe_permute_backward(const moe_bf16* dx_perm, const int32_t* row_id_map,
                                  int64_t T, int64_t H, int64_t k, moe_bf16* dx,
                                  void* ws, size_t ws_bytes, moe_stream_t stream);

/* SwiGLU gradient with clip: [MegaMoE] 激活函数公式 differentiated.
 *   h [rows, 2I] bf16 pre-activation (gate | up), da [rows, I] bf16,
 *   dh [rows, 2I] bf16 out:
 *   dG = dA * U_c * SiLU'(G_c) * [G <= c],  dU = dA * SiLU(G_c) * [-c <= U <= c] */
MOE_API moe_status_t moe_swiglu_backward(const moe_bf16* h, const moe_bf16* da, int64_t rows, int64_t I,
                                 float clip, moe_bf16* dh,
                                 void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_swiglu_backward for any gated activation (moe_activation_t): the
 * derivative of its formula, [dG | dU] = Activation'(h) applied to da. */
MOE_API moe_status_t moe_activation_backward(const moe_bf16* h, const moe_bf16* da, int64_t rows, int64_t I,
                                     const moe_activation_t* activation, moe_bf16* dh,
                                     void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- whole layer */

/* Tensors the forward keeps for the backward (all device pointers, caller-owned). */
typedef struct moe_layer_saved {
  moe_bf16* x_perm;      /* [T*k, H]  permuted tokens */
  moe_bf16* h;           /* [T*k, 2I] gate_up product (pre-activation) */
  moe_bf16* a;           /* [T*k, I]  SwiGLU output */
  moe_bf16* y2;          /* [T*k, H]  down product */
  int32_t* row_id_map;   /* [T*k] */
  int32_t* sorted_flat;  /* [T*k] */
  int64_t* group_list;   /* [E] */
} moe_layer_saved_t;

/* Workspace bytes for moe_layer_forward and moe_layer_backward with these
 * sizes (one size serves both calls, with or without `saved`). */
MOE_API size_t moe_layer_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k);

/* Routed-expert layer forward ([GMM] "Qwen3.5 MoE 路径"; [MegaMoE] A16W16):
 * permute -> GMM(w1 [E, H, 2I]) with SwiGLU(clip) -> GMM(w2 [E, I, H]) -> combine.
 *   x [T, H] bf16, topk_ids [T, k] int32, topk_w [T, k] fp32, y [T, H] bf16 out.
 *   saved: NULL for inference (intermediates live in ws), or the buffers that
 *   moe_layer_backward will read.
 * Inference with T*k < 512*E (groups that average under 512 rows) fuses the
 * dispatch into gate_up and runs both expert matmuls as one launch ([MegaMoE]
 * "算子功能"): the permute's index pass, moe_expert_mlp_forward and
 * moe_unpermute, three launches (four above 1024 routed slots; with
 * transposed weights the two matmuls are gmm_forward_gather_act and
 * gmm_forward); the permuted tokens are never written to HBM.  The result is
 * bit-identical to the unfused chain (moe_permute, gmm_forward with the
 * activation, gmm_forward, moe_unpermute), which the other cases run. */
MOE_API moe_status_t moe_layer_forward(const moe_bf16* x, const int32_t* topk_ids, const float* topk_w,
                               const moe_bf16* w1, const moe_bf16* w2,
                               int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, float clip,
                               moe_bf16* y, const moe_layer_saved_t* saved,
                               void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_layer_forward with any gated activation between the two GMMs, and the
 * weights' layouts: w_flags MOE_W1_TRANSPOSED (w1 [E, 2I, H]) and / or
 * MOE_W2_TRANSPOSED (w2 [E, H, I]). */
MOE_API moe_status_t moe_layer_forward_act(const moe_bf16* x, const int32_t* topk_ids, const float* topk_w,
                               const moe_bf16* w1, const moe_bf16* w2,
                               int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                               const moe_activation_t* activation, int w_flags, moe_bf16* y,
                               const moe_layer_saved_t* saved, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Backward of moe_layer_forward (saved must be what the forward filled):
 *   dy [T, H] bf16 in; dx [T, H], dw1 [E, H, 2I], dw2 [E, I, H] bf16 and
 *   dprobs [T, k] fp32 out (any of them may be NULL except dx). */
MOE_API moe_status_t moe_layer_backward(const moe_bf16* dy, const float* topk_w,
                                const moe_bf16* w1, const moe_bf16* w2,
                                const moe_layer_saved_t* saved,
                                int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, float clip,
                                moe_bf16* dx, moe_bf16* dw1, moe_bf16* dw2, float* dprobs,
                                void* ws, size_t ws_bytes, moe_stream_t stream);

/* Backward of moe_layer_forward_act (the same activation and w_flags; dw1 and
 * dw2 are written in their weights' layouts). */
MOE_API moe_status_t moe_layer_backward_act(const moe_bf16* dy, const float* topk_w,
                                const moe_bf16* w1, const moe_bf16* w2,
                                const moe_layer_saved_t* saved,
                                int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                                const moe_activation_t* activation, int w_flags,
                                moe_bf16* dx, moe_bf16* dw1, moe_bf16* dw2, float* dprobs,
                                void* ws, size_t ws_bytes, moe_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* MOE_GMM_H */
