// The C ABI (include/moe_gmm.h): argument checks, workspace carving and the
// launch sequence of each entry point.  Host code only; kernels live in
// permute.cu, gmm.cu and combine.cu.
//
// The two-phase convention (size query, then execute with a caller-owned
// workspace on a stream) and the null / invalid argument split follow
// "CANN ops-transformer 算子详解 MoeTokenPermuteWithRoutingMapGrad", sections 3
// and 4.2-4.3; empty inputs are a no-op needing no workspace (section 5).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "moe_gmm.h"
#include "moe_mx.h"

namespace moe {

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline uint32_t* status_of(void* ws) { return static_cast<uint32_t*>(ws); }
inline uint8_t* after_status(void* ws) { return static_cast<uint8_t*>(ws) + MOE_STATUS_BYTES; }

moe_status_t check_ws(const void* ws, size_t have, size_t need) {
  if (ws == nullptr) return MOE_ERR_NULLPTR;
  if (!aligned16(ws) || have < need) return MOE_ERR_INVALID;
  return MOE_OK;
}

bool bad_clip(float clip) { return !(clip >= 0.0f) || isinf(clip); }  // NaN fails the first test

// The ABI's (activation, activation_params) pair -> Act, with the pages'
// defaults and value checks ([MegaMoE] 参数说明).
moe_status_t resolve_act(const moe_activation_t* a, Act* out) {
  if (!a) return MOE_ERR_NULLPTR;
  const int n = a->n_params;
  const float* v = a->params;
  if (n < 0 || n > 3) return MOE_ERR_INVALID;
  Act r;
  r.kind = a->kind;
  auto clamp_to = [&](float c) {  // >= 0, not NaN; 0 and +inf mean no clip
    if (c > 0.0f && !isinf(c)) r.c = c;
  };
  switch (a->kind) {
    case MOE_ACT_SWIGLU:
    case MOE_ACT_SWIGLUSTEP:
      if (n > 1 || (n == 1 && !(v[0] >= 0.0f))) return MOE_ERR_INVALID;
      if (n == 1) clamp_to(v[0]);
      break;
    case MOE_ACT_SWIGLUOAI:
      if (n != 0 && n != 3) return MOE_ERR_INVALID;
      if (n == 3) {
        if (!(v[0] >= 0.0f) || !isfinite(v[1]) || !isfinite(v[2])) return MOE_ERR_INVALID;
        clamp_to(v[0]);
        r.alpha = v[1];
        r.beta = v[2];
      }
      break;
    case MOE_ACT_SITUGLU:
      if (n > 2) return MOE_ERR_INVALID;
      if (n >= 1 && !(v[0] > 0.0f && isfinite(v[0]))) return MOE_ERR_INVALID;
      if (n == 2 && !(v[1] > 0.0f && isfinite(v[1]))) return MOE_ERR_INVALID;
      if (n >= 1) r.beta = v[0];
      if (n == 2) r.lbeta = v[1];
      break;
    default:
      return MOE_ERR_UNSUPPORTED;
  }
  *out = r;
  return MOE_OK;
}

moe_activation_t swiglu_desc(float clip) {
  moe_activation_t a = {};
  a.kind = MOE_ACT_SWIGLU;
  a.n_params = 1;
  a.params[0] = clip;
  return a;
}

size_t layer_acts_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
  const size_t R = static_cast<size_t>(T * k);
  const size_t fwd = align256(R * H * 2) + align256(R * I * 2) + align256(R * H * 2) + 2 * align256(R * 4) +
                     align256(static_cast<size_t>(E) * 8);
  const size_t bwd = align256(R * H * 2) + align256(R * 2 * I * 2);
  return fwd > bwd ? fwd : bwd;
}

moe_status_t check_gmm_dims(int64_t M, int64_t K, int64_t N, int64_t E) {
  if (M < 0 || K <= 0 || N <= 0 || E <= 0) return MOE_ERR_INVALID;
  if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (K % 64 || N % 64) return MOE_ERR_UNSUPPORTED;
  if (M > INT32_MAX || K > INT32_MAX / 2 || N > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t check_tokens(int64_t T, int64_t H, int64_t k) {
  if (T < 0 || H <= 0 || k <= 0) return MOE_ERR_INVALID;
  if (k > kMaxTopK || H % 8) return MOE_ERR_UNSUPPORTED;
  if (T * k > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace

// Argument checks of the permute, shared by moe_permute and moe_permute_no_alloc.
moe_status_t check_permute_args(const uint16_t* x, const int32_t* topk_ids, int64_t T, int64_t H, int64_t k,
                                int64_t E, const uint16_t* x_perm, const int64_t* group_list,
                                const int32_t* row_id_map, const int32_t* sorted_flat) {
  if (!group_list) return MOE_ERR_NULLPTR;
  if (T != 0 && (!topk_ids || !row_id_map || !sorted_flat)) return MOE_ERR_NULLPTR;  // T == 0: nothing to read or write
  if (T != 0 && (x == nullptr) != (x_perm == nullptr)) return MOE_ERR_NULLPTR;
  if (E <= 0 || k > E) return MOE_ERR_INVALID;
  if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  moe_status_t st = check_tokens(T, x ? H : 8, k);
  if (st != MOE_OK) return st;
  if ((x && !aligned16(x)) || (x_perm && !aligned16(x_perm))) return MOE_ERR_INVALID;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_NULLPTR: return "MOE_ERR_NULLPTR";
    case MOE_ERR_INVALID: return "MOE_ERR_INVALID";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_BOUNDS: return "MOE_ERR_BOUNDS";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (ws == nullptr) return MOE_ERR_NULLPTR;
  if (ws_bytes < MOE_STATUS_BYTES || !aligned16(ws)) return MOE_ERR_INVALID;
  return cudaMemsetAsync(ws, 0, MOE_STATUS_BYTES, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_check_wait_timeout(void* ws, size_t ws_bytes, uint64_t timeout_ns, moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_ws(ws, ws_bytes, MOE_STATUS_BYTES);
  if (st != MOE_OK) return st;
  if (timeout_ns < 1000ull || timeout_ns > 10000000000ull) return MOE_ERR_INVALID;
  return launch_wait_timeout_check(status_of(ws), timeout_ns, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_check_bounds(void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_ws(ws, ws_bytes, MOE_STATUS_BYTES);
  if (st != MOE_OK) return st;
  return launch_bounds_check(status_of(ws), reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_read_status(const void* ws, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (ws == nullptr) return MOE_ERR_NULLPTR;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status_t>(v);
}

// ------------------------------------------------------------------ dispatch
size_t moe_permute_workspace_size(int64_t T, int64_t k, int64_t E) {
  if (T <= 0 || k <= 0 || E <= 0) return MOE_STATUS_BYTES;
  return MOE_STATUS_BYTES + permute_scratch_bytes(T, k, E);
}

moe_status_t moe_permute(const moe_bf16* x, const int32_t* topk_ids, int64_t T, int64_t H, int64_t k, int64_t E,
                         moe_bf16* x_perm, int64_t* group_list, int32_t* row_id_map, int32_t* sorted_flat,
                         void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_permute_args(x, topk_ids, T, H, k, E, x_perm, group_list, row_id_map, sorted_flat);
  if (st != MOE_OK) return st;
  if ((st = check_ws(ws, ws_bytes, moe_permute_workspace_size(T, k, E))) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0)
    return cudaMemsetAsync(group_list, 0, E * sizeof(int64_t), s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  return launch_permute(x, topk_ids, T, H, k, E, x_perm, group_list, row_id_map, sorted_flat, status_of(ws),
                        after_status(ws), s);
}

// ------------------------------------------------------------------ grouped matmul
size_t gmm_workspace_size(int64_t, int64_t, int64_t, int64_t) { return MOE_STATUS_BYTES + kGmmScratchBytes; }

moe_status_t gmm_forward_act(const moe_bf16* x, const moe_bf16* w, const int64_t* group_list, int64_t M, int64_t K,
                             int64_t N, int64_t E, const moe_activation_t* activation, int w_flags, moe_bf16* y,
                             moe_bf16* h_save, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!x || !w || !group_list || !y) return MOE_ERR_NULLPTR;
  Act act;
  moe_status_t st = activation ? resolve_act(activation, &act) : MOE_OK;
  if (st != MOE_OK) return st;
  if ((st = check_gmm_dims(M, K, N, E)) != MOE_OK) return st;
  if (w_flags & ~MOE_W_TRANSPOSED) return MOE_ERR_INVALID;
  if (activation && N % 256) return MOE_ERR_UNSUPPORTED;
  if (!activation && h_save) return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (h_save && !aligned16(h_save)) ||
      (reinterpret_cast<uintptr_t>(group_list) & 7u))
    return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, gmm_workspace_size(M, K, N, E))) != MOE_OK) return st;
  if (M == 0) return MOE_OK;
  GmmLaunch how;
  how.w_transposed = (w_flags & MOE_W_TRANSPOSED) != 0;
  return launch_gmm(GMM_FWD, activation ? EPI_SWIGLU : EPI_PLAIN, x, w, group_list, M, K, N, E, act, y, h_save,
                    status_of(ws), after_status(ws), reinterpret_cast<cudaStream_t>(stream), how);
}

moe_status_t gmm_forward(const moe_bf16* x, const moe_bf16* w, const int64_t* group_list, int64_t M, int64_t K,
                         int64_t N, int64_t E, int epilogue, float clip, moe_bf16* y, moe_bf16* h_save,
                         void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (epilogue != MOE_EPILOGUE_NONE && epilogue != MOE_EPILOGUE_SWIGLU) return MOE_ERR_UNSUPPORTED;
  if (bad_clip(clip)) return MOE_ERR_INVALID;
  const moe_activation_t a = swiglu_desc(clip);
  return gmm_forward_act(x, w, group_list, M, K, N, E, epilogue == MOE_EPILOGUE_SWIGLU ? &a : nullptr, 0, y, h_save,
                         ws, ws_bytes, stream);
}

moe_status_t gmm_forward_gather_act(const moe_bf16* x, const int32_t* sorted_flat, int64_t T, int64_t k,
                                    const moe_bf16* w, const int64_t* group_list, int64_t M, int64_t K, int64_t N,
                                    int64_t E, const moe_activation_t* activation, int w_flags, moe_bf16* y,
                                    void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!x || !sorted_flat || !w || !group_list || !y || !activation) return MOE_ERR_NULLPTR;
  Act act;
  moe_status_t st = resolve_act(activation, &act);
  if (st != MOE_OK) return st;
  if ((st = check_gmm_dims(M, K, N, E)) != MOE_OK) return st;
  if ((st = check_tokens(T, K, k)) != MOE_OK) return st;
  if (w_flags & ~MOE_W_TRANSPOSED) return MOE_ERR_INVALID;
  if (N % 256) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (reinterpret_cast<uintptr_t>(group_list) & 7u) ||
      (reinterpret_cast<uintptr_t>(sorted_flat) & 3u))
    return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, gmm_workspace_size(M, K, N, E))) != MOE_OK) return st;
  if (M == 0 || T == 0) return MOE_OK;
  return launch_gmm_gather_act(x, sorted_flat, T, k, w, group_list, M, K, N, E, act, (w_flags & MOE_W_TRANSPOSED) != 0,
                               y, nullptr, 0, status_of(ws), reinterpret_cast<cudaStream_t>(stream));
}

size_t gmm_forward_combine_workspace_size(int64_t T, int64_t k, int64_t M, int64_t N) {
  (void)k;
  if (T <= 0 || M < 0 || N <= 0) return MOE_STATUS_BYTES;
  return MOE_STATUS_BYTES + fused_counter_bytes(N) + align256(static_cast<size_t>(M) * N * 2);
}

moe_status_t gmm_forward_combine(const moe_bf16* a, const moe_bf16* w, const int64_t* group_list,
                                 const int32_t* row_id_map, const int32_t* sorted_flat, const float* topk_w,
                                 int64_t T, int64_t k, int64_t M, int64_t K, int64_t N, int64_t E, int w_flags,
                                 moe_bf16* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!w || !group_list || !y) return MOE_ERR_NULLPTR;
  if (T != 0 && (!row_id_map || !topk_w)) return MOE_ERR_NULLPTR;
  if (M != 0 && (!a || !sorted_flat)) return MOE_ERR_NULLPTR;
  moe_status_t st = check_gmm_dims(M, K, N, E);
  if (st != MOE_OK) return st;
  if ((st = check_tokens(T, N, k)) != MOE_OK) return st;
  if (w_flags & ~MOE_W_TRANSPOSED) return MOE_ERR_INVALID;
  if ((a && !aligned16(a)) || !aligned16(w) || !aligned16(y) || (reinterpret_cast<uintptr_t>(group_list) & 7u) ||
      (reinterpret_cast<uintptr_t>(row_id_map) & 3u) || (reinterpret_cast<uintptr_t>(sorted_flat) & 3u) ||
      (reinterpret_cast<uintptr_t>(topk_w) & 3u))
    return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, gmm_forward_combine_workspace_size(T, k, M, N))) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0)  // no expert rows: every token's sum is empty
    return cudaMemsetAsync(y, 0, static_cast<size_t>(T) * N * 2, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  int32_t* counters = reinterpret_cast<int32_t*>(after_status(ws));
  moe_bf16* y2 = reinterpret_cast<moe_bf16*>(after_status(ws) + fused_counter_bytes(N));
  if (cudaMemsetAsync(counters, 0, fused_counter_bytes(N), s) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_gmm_combine(a, w, group_list, row_id_map, sorted_flat, topk_w, T, k, M, K, N, E,
                            (w_flags & MOE_W_TRANSPOSED) != 0, y2, counters, y, status_of(ws), s);
}

size_t moe_expert_mlp_workspace_size(int64_t T, int64_t k, int64_t E) {
  if (T <= 0 || k <= 0 || E <= 0) return MOE_STATUS_BYTES;
  return MOE_STATUS_BYTES + expert_mlp_ready_bytes(T * k, E);
}

moe_status_t moe_expert_mlp_forward(const moe_bf16* x, const int32_t* sorted_flat, const int64_t* group_list,
                                    const moe_bf16* w1, const moe_bf16* w2, int64_t T, int64_t H, int64_t I,
                                    int64_t E, int64_t k, const moe_activation_t* activation, moe_bf16* a,
                                    moe_bf16* y2, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!x || !sorted_flat || !group_list || !w1 || !w2 || !a || !y2 || !activation) return MOE_ERR_NULLPTR;
  Act act;
  moe_status_t st = resolve_act(activation, &act);
  if (st != MOE_OK) return st;
  if (E <= 0 || I <= 0 || k > E) return MOE_ERR_INVALID;
  if ((st = check_tokens(T, H, k)) != MOE_OK) return st;
  if (E > kMaxExperts || H % 64 || I % 128) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w1) || !aligned16(w2) || !aligned16(a) || !aligned16(y2) ||
      (reinterpret_cast<uintptr_t>(group_list) & 7u) || (reinterpret_cast<uintptr_t>(sorted_flat) & 3u))
    return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, moe_expert_mlp_workspace_size(T, k, E))) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* ready = reinterpret_cast<int32_t*>(after_status(ws));
  if (cudaMemsetAsync(ready, 0, expert_mlp_ready_bytes(T * k, E), s) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_expert_mlp(x, sorted_flat, w1, w2, group_list, T, H, I, E, k, act, a, y2, ready, status_of(ws), s);
}

moe_status_t gmm_backward_ex(const moe_bf16* x, const moe_bf16* w, const int64_t* group_list, const moe_bf16* dy,
                             int64_t M, int64_t K, int64_t N, int64_t E, int w_flags, moe_bf16* dx, moe_bf16* dw,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!x || !w || !group_list || !dy) return MOE_ERR_NULLPTR;
  moe_status_t st = check_gmm_dims(M, K, N, E);
  if (st != MOE_OK) return st;
  if (w_flags & ~MOE_W_TRANSPOSED) return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(w) || !aligned16(dy) || (dx && !aligned16(dx)) || (dw && !aligned16(dw)) ||
      (reinterpret_cast<uintptr_t>(group_list) & 7u))
    return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, gmm_workspace_size(M, K, N, E))) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) {
    // no rows: every group is empty, so dW is zero
    if (dw && cudaMemsetAsync(dw, 0, static_cast<size_t>(E * K * N) * 2, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  return launch_gmm_backward(x, w, group_list, dy, M, K, N, E, EPI_PLAIN, Act(), nullptr, dx, dw, status_of(ws),
                             after_status(ws), s, (w_flags & MOE_W_TRANSPOSED) != 0);
}

moe_status_t gmm_backward(const moe_bf16* x, const moe_bf16* w, const int64_t* group_list, const moe_bf16* dy,
                          int64_t M, int64_t K, int64_t N, int64_t E, moe_bf16* dx, moe_bf16* dw,
                          void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  return gmm_backward_ex(x, w, group_list, dy, M, K, N, E, 0, dx, dw, ws, ws_bytes, stream);
}

moe_status_t gmm_backward_dx_act(const moe_bf16* dy, const moe_bf16* w, const int64_t* group_list,
                                 const moe_bf16* h, int64_t M, int64_t K, int64_t N, int64_t E,
                                 const moe_activation_t* activation, int w_flags, moe_bf16* dh, void* ws,
                                 size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!dy || !w || !group_list || !h || !dh) return MOE_ERR_NULLPTR;
  Act act;
  moe_status_t st = resolve_act(activation, &act);
  if (st != MOE_OK) return st;
  if ((st = check_gmm_dims(M, K, N, E)) != MOE_OK) return st;
  if (w_flags & ~MOE_W_TRANSPOSED) return MOE_ERR_INVALID;
  if (!aligned16(dy) || !aligned16(w) || !aligned16(h) || !aligned16(dh) ||
      (reinterpret_cast<uintptr_t>(group_list) & 7u))
    return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, gmm_workspace_size(M, K, N, E))) != MOE_OK) return st;
  if (M == 0) return MOE_OK;
  GmmLaunch how;
  how.w_transposed = (w_flags & MOE_W_TRANSPOSED) != 0;
  return launch_gmm(GMM_DX, EPI_DSWIGLU, dy, w, group_list, M, K, N, E, act, dh, const_cast<moe_bf16*>(h),
                    status_of(ws), after_status(ws), reinterpret_cast<cudaStream_t>(stream), how);
}

moe_status_t gmm_backward_dx_swiglu(const moe_bf16* dy, const moe_bf16* w, const int64_t* group_list,
                                    const moe_bf16* h, int64_t M, int64_t K, int64_t N, int64_t E, float clip,
                                    moe_bf16* dh, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (bad_clip(clip)) return MOE_ERR_INVALID;
  const moe_activation_t a = swiglu_desc(clip);
  return gmm_backward_dx_act(dy, w, group_list, h, M, K, N, E, &a, 0, dh, ws, ws_bytes, stream);
}

// ------------------------------------------------------------------ combine side
size_t moe_unpermute_workspace_size(void) { return MOE_STATUS_BYTES; }

moe_status_t moe_unpermute(const moe_bf16* y_perm, const int32_t* row_id_map, const float* topk_w, int64_t T,
                           int64_t H, int64_t k, moe_bf16* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!y_perm || !row_id_map || !y) return MOE_ERR_NULLPTR;
  moe_status_t st = check_tokens(T, H, k);
  if (st != MOE_OK) return st;
  if (!aligned16(y_perm) || !aligned16(y)) return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, MOE_STATUS_BYTES)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  return launch_unpermute(y_perm, row_id_map, topk_w, T, H, k, y, status_of(ws),
                          reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_unpermute_backward(const moe_bf16* dy, const moe_bf16* y_perm, const int32_t* row_id_map,
                                    const float* topk_w, int64_t T, int64_t H, int64_t k, moe_bf16* dy_perm,
                                    float* dprobs, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!dy || !y_perm || !row_id_map || !topk_w || !dy_perm) return MOE_ERR_NULLPTR;
  moe_status_t st = check_tokens(T, H, k);
  if (st != MOE_OK) return st;
  if (!aligned16(dy) || !aligned16(y_perm) || !aligned16(dy_perm)) return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, MOE_STATUS_BYTES)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  return launch_unpermute_backward(dy, y_perm, row_id_map, topk_w, T, H, k, dy_perm, dprobs, status_of(ws),
                                   reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_permute_backward(const moe_bf16* dx_perm, const int32_t* row_id_map, int64_t T, int64_t H,
                                  int64_t k, moe_bf16* dx, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!dx_perm || !row_id_map || !dx) return MOE_ERR_NULLPTR;
  moe_status_t st = check_tokens(T, H, k);
  if (st != MOE_OK) return st;
  if (!aligned16(dx_perm) || !aligned16(dx)) return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, MOE_STATUS_BYTES)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  return launch_unpermute(dx_perm, row_id_map, nullptr, T, H, k, dx, status_of(ws),
                          reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_activation_backward(const moe_bf16* h, const moe_bf16* da, int64_t rows, int64_t I,
                                     const moe_activation_t* activation, moe_bf16* dh, void* ws, size_t ws_bytes,
                                     moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!h || !da || !dh) return MOE_ERR_NULLPTR;
  Act act;
  moe_status_t st = resolve_act(activation, &act);
  if (st != MOE_OK) return st;
  if (rows < 0 || I <= 0) return MOE_ERR_INVALID;
  if (I % 8) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(h) || !aligned16(da) || !aligned16(dh)) return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, MOE_STATUS_BYTES)) != MOE_OK) return st;
  if (rows == 0) return MOE_OK;
  return launch_act_backward(h, da, rows, I, act, dh, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_swiglu_backward(const moe_bf16* h, const moe_bf16* da, int64_t rows, int64_t I, float clip,
                                 moe_bf16* dh, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (bad_clip(clip)) return MOE_ERR_INVALID;
  const moe_activation_t a = swiglu_desc(clip);
  return moe_activation_backward(h, da, rows, I, &a, dh, ws, ws_bytes, stream);
}

// ------------------------------------------------------------------ whole layer
size_t moe_layer_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
  if (T <= 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return MOE_STATUS_BYTES;
  return MOE_STATUS_BYTES + kGmmScratchBytes + permute_scratch_bytes(T, k, E) + layer_acts_bytes(T, H, I, E, k);
}

namespace {
moe_status_t check_layer(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
  if (E <= 0 || I <= 0 || k > E) return MOE_ERR_INVALID;
  moe_status_t st = check_tokens(T, H, k);
  if (st != MOE_OK) return st;
  if (E > kMaxExperts || H % 64 || I % 128) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}
bool saved_ok(const moe_layer_saved_t* sv) {
  return sv->x_perm && sv->h && sv->a && sv->y2 && sv->row_id_map && sv->sorted_flat && sv->group_list;
}
bool saved_aligned(const moe_layer_saved_t* sv) {
  return aligned16(sv->x_perm) && aligned16(sv->h) && aligned16(sv->a) && aligned16(sv->y2) &&
         (reinterpret_cast<uintptr_t>(sv->group_list) & 7u) == 0;
}
}  // namespace

moe_status_t moe_layer_forward_act(const moe_bf16* x, const int32_t* topk_ids, const float* topk_w,
                                   const moe_bf16* w1, const moe_bf16* w2, int64_t T, int64_t H, int64_t I, int64_t E,
                                   int64_t k, const moe_activation_t* activation, int w_flags, moe_bf16* y,
                                   const moe_layer_saved_t* saved, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!x || !topk_ids || !topk_w || !w1 || !w2 || !y) return MOE_ERR_NULLPTR;
  if (saved && !saved_ok(saved)) return MOE_ERR_NULLPTR;
  Act act;
  moe_status_t st = resolve_act(activation, &act);
  if (st != MOE_OK) return st;
  if ((st = check_layer(T, H, I, E, k)) != MOE_OK) return st;
  if (w_flags & ~(MOE_W1_TRANSPOSED | MOE_W2_TRANSPOSED)) return MOE_ERR_INVALID;
  if (!aligned16(x) || !aligned16(w1) || !aligned16(w2) || !aligned16(y) || (saved && !saved_aligned(saved)))
    return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, moe_layer_workspace_size(T, H, I, E, k))) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = status_of(ws);
  uint8_t* gmm_scratch = after_status(ws);
  uint8_t* scratch = gmm_scratch + kGmmScratchBytes;
  uint8_t* acts = scratch + permute_scratch_bytes(T, k, E);
  const int64_t R = T * k;
  moe_bf16 *x_perm, *h, *a, *y2;
  int32_t *rmap, *sflat;
  int64_t* gl;
  if (saved) {
    x_perm = saved->x_perm; h = saved->h; a = saved->a; y2 = saved->y2;
    rmap = saved->row_id_map; sflat = saved->sorted_flat; gl = saved->group_list;
  } else {
    uint8_t* p = acts;
    x_perm = reinterpret_cast<moe_bf16*>(p); p += align256(R * H * 2);
    a = reinterpret_cast<moe_bf16*>(p);      p += align256(R * I * 2);
    y2 = reinterpret_cast<moe_bf16*>(p);     p += align256(R * H * 2);
    rmap = reinterpret_cast<int32_t*>(p);    p += align256(R * 4);
    sflat = reinterpret_cast<int32_t*>(p);   p += align256(R * 4);
    gl = reinterpret_cast<int64_t*>(p);
    h = nullptr;
  }
  if (!saved && R < kPairMinRowsPerGroup * E) {
    // Inference with groups that average under 512 rows (the 128-row kernel's
    // regime): the permute only ranks the slots (and zeroes the readiness
    // counts, which sit where x_perm would), then both expert matmuls run in
    // one launch whose gate_up reads its rows straight from x, so the permuted
    // tokens never make a round trip through HBM.  The combine stays its own
    // launch: the fused form (gmm_forward_combine) is slower at these sizes
    // (its column-slice order re-reads the activation from HBM).  Transposed
    // weights take the gathered gate_up and the down GMM as two launches.
    int32_t* ready = reinterpret_cast<int32_t*>(x_perm);
    const bool one_launch = w_flags == 0;
    const int64_t n_ready = one_launch ? static_cast<int64_t>(expert_mlp_ready_bytes(R, E) / sizeof(int32_t)) : 0;
    if ((st = launch_permute(nullptr, topk_ids, T, H, k, E, nullptr, gl, rmap, sflat, status, scratch, s, nullptr,
                             ready, n_ready)) != MOE_OK)
      return st;
    if (one_launch) {
      if ((st = launch_expert_mlp(x, sflat, w1, w2, gl, T, H, I, E, k, act, a, y2, ready, status, s)) != MOE_OK)
        return st;
      return launch_unpermute(y2, rmap, topk_w, T, H, k, y, status, s);
    }
    if ((st = launch_gmm_gather_act(x, sflat, T, k, w1, gl, R, H, 2 * I, E, act, (w_flags & MOE_W1_TRANSPOSED) != 0,
                                    a, nullptr, 0, status, s)) != MOE_OK)
      return st;
    GmmLaunch how2;
    how2.w_transposed = (w_flags & MOE_W2_TRANSPOSED) != 0;
    if ((st = launch_gmm(GMM_FWD, EPI_PLAIN, a, w2, gl, R, I, H, E, Act(), y2, nullptr, status, gmm_scratch, s,
                         how2)) != MOE_OK)
      return st;
    return launch_unpermute(y2, rmap, topk_w, T, H, k, y, status, s);
  }
  if ((st = launch_permute(x, topk_ids, T, H, k, E, x_perm, gl, rmap, sflat, status, scratch, s)) != MOE_OK) return st;
  GmmLaunch how1, how2;
  how1.w_transposed = (w_flags & MOE_W1_TRANSPOSED) != 0;
  how2.w_transposed = (w_flags & MOE_W2_TRANSPOSED) != 0;
  if ((st = launch_gmm(GMM_FWD, EPI_SWIGLU, x_perm, w1, gl, R, H, 2 * I, E, act, a, h, status, gmm_scratch, s,
                       how1)) != MOE_OK)
    return st;
  if ((st = launch_gmm(GMM_FWD, EPI_PLAIN, a, w2, gl, R, I, H, E, Act(), y2, nullptr, status, gmm_scratch, s,
                       how2)) != MOE_OK)
    return st;
  return launch_unpermute(y2, rmap, topk_w, T, H, k, y, status, s);
}

moe_status_t moe_layer_forward(const moe_bf16* x, const int32_t* topk_ids, const float* topk_w, const moe_bf16* w1,
                               const moe_bf16* w2, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, float clip,
                               moe_bf16* y, const moe_layer_saved_t* saved, void* ws, size_t ws_bytes,
                               moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (bad_clip(clip)) return MOE_ERR_INVALID;
  const moe_activation_t a = swiglu_desc(clip);
  return moe_layer_forward_act(x, topk_ids, topk_w, w1, w2, T, H, I, E, k, &a, 0, y, saved, ws, ws_bytes, stream);
}

moe_status_t moe_layer_backward_act(const moe_bf16* dy, const float* topk_w, const moe_bf16* w1,
                                    const moe_bf16* w2, const moe_layer_saved_t* saved, int64_t T, int64_t H,
                                    int64_t I, int64_t E, int64_t k, const moe_activation_t* activation,
                                    int w_flags, moe_bf16* dx, moe_bf16* dw1, moe_bf16* dw2, float* dprobs, void* ws,
                                    size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!dy || !topk_w || !w1 || !w2 || !saved || !dx) return MOE_ERR_NULLPTR;
  if (!saved_ok(saved)) return MOE_ERR_NULLPTR;
  Act act;
  moe_status_t st = resolve_act(activation, &act);
  if (st != MOE_OK) return st;
  if ((st = check_layer(T, H, I, E, k)) != MOE_OK) return st;
  if (w_flags & ~(MOE_W1_TRANSPOSED | MOE_W2_TRANSPOSED)) return MOE_ERR_INVALID;
  if (!aligned16(dy) || !aligned16(w1) || !aligned16(w2) || !aligned16(dx) || (dw1 && !aligned16(dw1)) ||
      (dw2 && !aligned16(dw2)) || !saved_aligned(saved))
    return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, moe_layer_workspace_size(T, H, I, E, k))) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (dw1 && cudaMemsetAsync(dw1, 0, static_cast<size_t>(E * H * 2 * I) * 2, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (dw2 && cudaMemsetAsync(dw2, 0, static_cast<size_t>(E * I * H) * 2, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  uint32_t* status = status_of(ws);
  uint8_t* gmm_scratch = after_status(ws);
  uint8_t* acts = gmm_scratch + kGmmScratchBytes + permute_scratch_bytes(T, k, E);
  const int64_t R = T * k;
  moe_bf16* dy2 = reinterpret_cast<moe_bf16*>(acts);
  moe_bf16* dh = reinterpret_cast<moe_bf16*>(acts + align256(R * H * 2));
  moe_bf16* dx_perm = dy2;  // dy2 is dead once dH and dW2 are done
  if ((st = launch_unpermute_backward(dy, saved->y2, saved->row_id_map, topk_w, T, H, k, dy2, dprobs, status, s)) !=
      MOE_OK)
    return st;
  // dH = SwiGLU'(H, dY2 @ W2^T) in one grouped matmul (dA is never stored)
  if ((st = launch_gmm_backward(saved->a, w2, saved->group_list, dy2, R, I, H, E, EPI_DSWIGLU, act, saved->h, dh,
                                dw2, status, gmm_scratch, s, (w_flags & MOE_W2_TRANSPOSED) != 0)) != MOE_OK)
    return st;
  if ((st = launch_gmm_backward(saved->x_perm, w1, saved->group_list, dh, R, H, 2 * I, E, EPI_PLAIN, Act(), nullptr,
                                dx_perm, dw1, status, gmm_scratch, s, (w_flags & MOE_W1_TRANSPOSED) != 0)) != MOE_OK)
    return st;
  return launch_unpermute(dx_perm, saved->row_id_map, nullptr, T, H, k, dx, status, s);
}

moe_status_t moe_layer_backward(const moe_bf16* dy, const float* topk_w, const moe_bf16* w1, const moe_bf16* w2,
                                const moe_layer_saved_t* saved, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                                float clip, moe_bf16* dx, moe_bf16* dw1, moe_bf16* dw2, float* dprobs, void* ws,
                                size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (bad_clip(clip)) return MOE_ERR_INVALID;
  const moe_activation_t a = swiglu_desc(clip);
  return moe_layer_backward_act(dy, topk_w, w1, w2, saved, T, H, I, E, k, &a, 0, dx, dw1, dw2, dprobs, ws, ws_bytes,
                                stream);
}

}  // extern "C"

// ------------------------------------------------------------------ MXFP8 forward (moe_mx.h)
namespace moe {
namespace {
bool bad_fmt(int32_t f) { return f != MOE_FP8_E4M3 && f != MOE_FP8_E5M2 && f != MOE_FP4_E2M1; }
// the activation's element type: the tokens' fp8 type, E4M3 after E2M1 tokens (A4W4-FP)
int32_t act_fmt(int32_t x_format) { return x_format == MOE_FP4_E2M1 ? MOE_FP8_E4M3 : x_format; }
// the 4-bit TMA map wants a 32-byte-aligned base
bool q_aligned(const void* w, int32_t f) {
  return (reinterpret_cast<uintptr_t>(w) & (f == MOE_FP4_E2M1 ? 31u : 15u)) == 0;
}

size_t layer_mx_acts_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
  const size_t R = static_cast<size_t>(T * k);
  return align256(R * H) + align256(R * H / 32) + align256(R * I) + align256(R * I / 32) + align256(R * H * 2) +
         2 * align256(R * 4) + align256(static_cast<size_t>(E) * 8);
}

moe_status_t check_mx_gmm(int64_t M, int64_t K, int64_t N, int64_t E) {
  if (M < 0 || K <= 0 || N <= 0 || E <= 0) return MOE_ERR_INVALID;
  if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (K % 128 || N % 128) return MOE_ERR_UNSUPPORTED;
  if (M > INT32_MAX || K > INT32_MAX / 2 || N > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}
}  // namespace
}  // namespace moe

extern "C" {

size_t moe_mx_quantize_workspace_size(void) { return MOE_STATUS_BYTES; }

moe_status_t moe_mx_quantize(const moe_bf16* x, int64_t rows, int64_t K, int32_t format, uint8_t* q,
                             uint8_t* scales, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (rows != 0 && (!x || !q || !scales)) return MOE_ERR_NULLPTR;
  if (rows < 0 || K <= 0 || bad_fmt(format)) return MOE_ERR_INVALID;
  if (K % 32) return MOE_ERR_UNSUPPORTED;
  if (rows != 0 && (!aligned16(x) || !aligned16(q))) return MOE_ERR_INVALID;
  moe_status_t st = check_ws(ws, ws_bytes, moe_mx_quantize_workspace_size());
  if (st != MOE_OK || rows == 0) return st;
  return launch_mx_quantize(x, rows, K, format, q, scales, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_permute_mx(const moe_bf16* x, const int32_t* topk_ids, int64_t T, int64_t H, int64_t k, int64_t E,
                            int32_t format, uint8_t* x_q, uint8_t* x_scales, int64_t* group_list,
                            int32_t* row_id_map, int32_t* sorted_flat, void* ws, size_t ws_bytes,
                            moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!group_list) return MOE_ERR_NULLPTR;
  if (T != 0 && (!x || !topk_ids || !x_q || !x_scales || !row_id_map || !sorted_flat)) return MOE_ERR_NULLPTR;
  if (E <= 0 || k > E || bad_fmt(format)) return MOE_ERR_INVALID;
  if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  moe_status_t st = check_tokens(T, H, k);
  if (st != MOE_OK) return st;
  if (H % 32) return MOE_ERR_UNSUPPORTED;
  if (T != 0 && (!aligned16(x) || !aligned16(x_q))) return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, moe_permute_workspace_size(T, k, E))) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0)
    return cudaMemsetAsync(group_list, 0, E * sizeof(int64_t), s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  const MxOut mx{format, x_q, x_scales};
  return launch_permute(x, topk_ids, T, H, k, E, nullptr, group_list, row_id_map, sorted_flat, status_of(ws),
                        after_status(ws), s, &mx);
}

size_t gmm_mx_workspace_size(int64_t, int64_t, int64_t, int64_t) { return MOE_STATUS_BYTES; }

moe_status_t gmm_forward_mx(const uint8_t* x_q, const uint8_t* x_scales, const uint8_t* w_q, const uint8_t* w_scales,
                            const int64_t* group_list, int64_t M, int64_t K, int64_t N, int64_t E, int32_t x_format,
                            int32_t w_format, const moe_activation_t* activation, moe_bf16* y, uint8_t* a_q,
                            uint8_t* a_scales, moe_bf16* h_save, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!x_q || !x_scales || !w_q || !w_scales || !group_list) return MOE_ERR_NULLPTR;
  if (activation ? (!a_q || !a_scales) : !y) return MOE_ERR_NULLPTR;
  if (bad_fmt(x_format) || bad_fmt(w_format)) return MOE_ERR_INVALID;
  Act act;
  moe_status_t st = activation ? resolve_act(activation, &act) : MOE_OK;
  if (st != MOE_OK) return st;
  if ((st = check_mx_gmm(M, K, N, E)) != MOE_OK) return st;
  if (activation && N % 256) return MOE_ERR_UNSUPPORTED;
  if (!activation && h_save) return MOE_ERR_INVALID;
  if (!q_aligned(x_q, x_format) || !aligned16(x_scales) || !q_aligned(w_q, w_format) || !aligned16(w_scales) ||
      (y && !aligned16(y)) || (a_q && !aligned16(a_q)) || (a_scales && !aligned16(a_scales)) ||
      (h_save && !aligned16(h_save)) || (reinterpret_cast<uintptr_t>(group_list) & 7u))
    return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, gmm_mx_workspace_size(M, K, N, E))) != MOE_OK) return st;
  if (M == 0) return MOE_OK;
  MxGmmArgs a{};
  a.a = x_q; a.a_sf = x_scales; a.b = w_q; a.b_sf = w_scales; a.group_list = group_list;
  a.M = M; a.K = K; a.N = N; a.E = E; a.a_fmt = x_format; a.b_fmt = w_format;
  a.act = activation ? &act : nullptr;
  a.out = y; a.aq = a_q; a.as = a_scales; a.out_fmt = act_fmt(x_format); a.h_save = h_save;
  return launch_gmm_mx(a, status_of(ws), reinterpret_cast<cudaStream_t>(stream));
}

size_t moe_layer_mx_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
  if (T <= 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return MOE_STATUS_BYTES;
  return MOE_STATUS_BYTES + permute_scratch_bytes(T, k, E) + layer_mx_acts_bytes(T, H, I, E, k);
}

moe_status_t moe_layer_forward_mx(const moe_bf16* x, const int32_t* topk_ids, const float* topk_w,
                                  const uint8_t* w1_q, const uint8_t* w1_scales, const uint8_t* w2_q,
                                  const uint8_t* w2_scales, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                                  int32_t x_format, int32_t w_format, const moe_activation_t* activation,
                                  moe_bf16* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (!x || !topk_ids || !topk_w || !w1_q || !w1_scales || !w2_q || !w2_scales || !y) return MOE_ERR_NULLPTR;
  if (bad_fmt(x_format) || bad_fmt(w_format)) return MOE_ERR_INVALID;
  Act act;
  moe_status_t st = resolve_act(activation, &act);
  if (st != MOE_OK) return st;
  if ((st = check_layer(T, H, I, E, k)) != MOE_OK) return st;
  if (H % 128) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !q_aligned(w1_q, w_format) || !aligned16(w1_scales) || !q_aligned(w2_q, w_format) ||
      !aligned16(w2_scales) || !aligned16(y))
    return MOE_ERR_INVALID;
  if ((st = check_ws(ws, ws_bytes, moe_layer_mx_workspace_size(T, H, I, E, k))) != MOE_OK) return st;
  if (!q_aligned(ws, x_format)) return MOE_ERR_INVALID;  // the packed E2M1 tokens live in ws
  if (T == 0) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = status_of(ws);
  uint8_t* scratch = after_status(ws);
  uint8_t* p = scratch + permute_scratch_bytes(T, k, E);
  const int64_t R = T * k;
  uint8_t* xq = p;                                      p += align256(R * H);
  uint8_t* xs = p;                                      p += align256(R * H / 32);
  uint8_t* aq = p;                                      p += align256(R * I);
  uint8_t* as = p;                                      p += align256(R * I / 32);
  moe_bf16* o = reinterpret_cast<moe_bf16*>(p);         p += align256(R * H * 2);
  int32_t* rmap = reinterpret_cast<int32_t*>(p);        p += align256(R * 4);
  int32_t* sflat = reinterpret_cast<int32_t*>(p);       p += align256(R * 4);
  int64_t* gl = reinterpret_cast<int64_t*>(p);
  const MxOut mx{x_format, xq, xs};
  if ((st = launch_permute(x, topk_ids, T, H, k, E, nullptr, gl, rmap, sflat, status, scratch, s, &mx)) != MOE_OK)
    return st;
  MxGmmArgs g1{};
  g1.a = xq; g1.a_sf = xs; g1.b = w1_q; g1.b_sf = w1_scales; g1.group_list = gl;
  g1.M = R; g1.K = H; g1.N = 2 * I; g1.E = E; g1.a_fmt = x_format; g1.b_fmt = w_format;
  g1.act = &act; g1.aq = aq; g1.as = as; g1.out_fmt = act_fmt(x_format);
  if ((st = launch_gmm_mx(g1, status, s)) != MOE_OK) return st;
  MxGmmArgs g2{};
  g2.a = aq; g2.a_sf = as; g2.b = w2_q; g2.b_sf = w2_scales; g2.group_list = gl;
  g2.M = R; g2.K = I; g2.N = H; g2.E = E; g2.a_fmt = act_fmt(x_format); g2.b_fmt = w_format;
  g2.out = o;
  if ((st = launch_gmm_mx(g2, status, s)) != MOE_OK) return st;
  return launch_unpermute(o, rmap, topk_w, T, H, k, y, status, s);
}

}  // extern "C"
