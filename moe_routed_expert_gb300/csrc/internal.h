// Internal launchers shared by the C ABI (abi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "moe_gmm.h"
#include "moe_mx.h"

struct CUtensorMap_st;  // cuda.h

namespace moe {

// An NVTX range named after the C-ABI function it spans (push at entry, pop
// at any return): a profiler collecting NVTX (ncu --nvtx, nsys) sees each call
// of the library as one range around its launches; without one attached the
// push and pop do nothing.
struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};
#define MOE_TRACE_CALL() ::moe::TraceRange moe_trace_range_(__func__)

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 64;

// Gated activation of the gate_up product ("MegaMoE", 激活函数公式), resolved
// from the ABI's (activation, activation_params) pair with the pages'
// defaults: swiglu SiLU(G_c) U_c; swiglustep min(SiLU(G), c) U_c; swigluoai
// G_c sigma(alpha G_c) (U_c + beta); situglu beta tanh(G / beta) sigma(G) L(U),
// L(U) = U, or lbeta tanh(U / lbeta) when lbeta > 0.  G_c = min(G, c),
// U_c = clip(U, -c, c); c = +inf when no clip is configured.
struct Act {
  int kind = MOE_ACT_SWIGLU;
  float c = __builtin_huge_valf();
  float alpha = 1.702f;
  float beta = 1.0f;
  float lbeta = 0.0f;
};
inline Act act_swiglu(float clip) {
  Act a;
  if (clip > 0.0f) a.c = clip;
  return a;
}

// Workspace layout: [status block | op scratch ...], every piece 256-byte aligned.
inline size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

int num_sms();  // SM count of the current device (cached per device)

// ---- failure-detection check (selfcheck.cu)
moe_status_t launch_wait_timeout_check(uint32_t* status, uint64_t timeout_ns, cudaStream_t s);
moe_status_t launch_bounds_check(uint32_t* status, cudaStream_t s);

// ---- MX quantisation (mx.cu): fp8 codes + E8M0 scales, 32-element groups
struct MxOut {
  int fmt;           // MOE_FP8_E4M3 / MOE_FP8_E5M2
  uint8_t* q;        // [rows, K] codes
  uint8_t* scales;   // [rows, K/32]
};
moe_status_t launch_mx_quantize(const uint16_t* x, int64_t rows, int64_t K, int fmt, uint8_t* q, uint8_t* scales,
                                cudaStream_t s);
// The permute's gather, quantising: slot f's token row of x -> row row_id_map[f].
moe_status_t launch_mx_gather(const uint16_t* x, int64_t nslots, int64_t H, int k, const int32_t* row_id_map,
                              const MxOut& out, uint32_t* status, cudaStream_t s);

// ---- dispatch (permute.cu)
// Argument checks shared by the permute entry points (abi.cu).
moe_status_t check_permute_args(const uint16_t* x, const int32_t* topk_ids, int64_t T, int64_t H, int64_t k,
                                int64_t E, const uint16_t* x_perm, const int64_t* group_list,
                                const int32_t* row_id_map, const int32_t* sorted_flat);
size_t permute_scratch_bytes(int64_t T, int64_t k, int64_t E);
// With `mx`, the gathered rows leave quantised into mx->q / mx->scales (x_perm unused).
// zero / zero_n: an int32 scratch range the index pass zeroes on the way (or none).
moe_status_t launch_permute(const uint16_t* x, const int32_t* ids, int64_t T, int64_t H, int64_t k, int64_t E,
                            uint16_t* x_perm, int64_t* group_list, int32_t* row_id_map, int32_t* sorted_flat,
                            uint32_t* status, void* scratch, cudaStream_t s, const MxOut* mx = nullptr,
                            int32_t* zero = nullptr, int64_t zero_n = 0);

// ---- combine side (combine.cu)
moe_status_t launch_unpermute(const uint16_t* y_perm, const int32_t* row_id_map, const float* topk_w,
                              int64_t T, int64_t H, int64_t k, uint16_t* y, uint32_t* status, cudaStream_t s);
moe_status_t launch_unpermute_backward(const uint16_t* dy, const uint16_t* y_perm, const int32_t* row_id_map,
                                       const float* topk_w, int64_t T, int64_t H, int64_t k,
                                       uint16_t* dy_perm, float* dprobs, uint32_t* status, cudaStream_t s);
moe_status_t launch_act_backward(const uint16_t* h, const uint16_t* da, int64_t rows, int64_t I, const Act& act,
                                 uint16_t* dh, cudaStream_t s);

// ---- TMA descriptors (tmap.cu): bf16, 128B swizzle, 64-element inner box
bool make_map_2d(::CUtensorMap_st* m, const void* base, int64_t rows, int64_t cols, int box_rows);
bool make_map_3d(::CUtensorMap_st* m, const void* base, int64_t E, int64_t K, int64_t N, int box_k);
// fp8 codes: 128-byte inner box
bool make_map_2d_u8(::CUtensorMap_st* m, const void* base, int64_t rows, int64_t cols, int box_rows);
bool make_map_3d_u8(::CUtensorMap_st* m, const void* base, int64_t E, int64_t R, int64_t C, int box_rows);
// packed 4-bit codes, expanded to the 16-byte-granule shared-memory form
bool make_map_3d_fp4(::CUtensorMap_st* m, const void* base, int64_t E, int64_t R, int64_t C, int box_rows);
bool make_map_2d_fp4(::CUtensorMap_st* m, const void* base, int64_t rows, int64_t cols, int box_rows);

// ---- grouped matmul (gmm.cu, gmm_pair.cu)
enum GmmMode { GMM_FWD = 0, GMM_DX = 1, GMM_DW = 2, GMM_BWD = 3 /* dX and dW in one launch (pairs) */ };
// Epilogues: 0 plain store; 1 (forward) SwiGLU of the [gate | up] product, H
// saved to h; 2 (dX) SwiGLU gradient: out = dH from dA = this product and the
// saved pre-activation passed in h.
enum GmmEpilogue { EPI_PLAIN = 0, EPI_SWIGLU = 1, EPI_DSWIGLU = 2 };
constexpr int64_t kPairMinRowsPerGroup = 512;
// GMM scratch in the workspace: per CTA, kMapSlots pairs of 128-byte TMA
// descriptors that the dW kernel rewrites for each group.
constexpr int kMapSlots = 6;
constexpr int kMaxGmmCtas = 256;
constexpr size_t kGmmScratchBytes = static_cast<size_t>(kMaxGmmCtas) * kMapSlots * 256;
// How a grouped matmul shares the GPU with the launch before it on the stream.
struct GmmLaunch {
  int max_ctas = 0;         // cap on the persistent grid (0: one CTA per SM)
  bool concurrent = false;  // start without waiting for the previous kernel (whose
                            // inputs must not be read) and wait for it before finishing
  bool w_transposed = false;  // FWD/DX: weights stored [E, N, K]
};
moe_status_t launch_gmm_pair(int mode, int epilogue, const uint16_t* a, const uint16_t* b, const int64_t* group_list,
                             int64_t M, int64_t K, int64_t N, int64_t E, const Act& act,
                             uint16_t* out, uint16_t* h_save, uint32_t* status, void* gmm_scratch, cudaStream_t s,
                             const GmmLaunch& how = GmmLaunch());
// dX (plain) and dW of one grouped matmul in one CTA-pair launch: each cluster
// takes tiles of one of the two, the split chosen on the device from the
// group sizes.  x [M, K], w [E, K, N] (or [E, N, K] transposed), dy [M, N].
moe_status_t launch_gmm_pair_bwd(const uint16_t* x, const uint16_t* w, const int64_t* group_list, const uint16_t* dy,
                                 int64_t M, int64_t K, int64_t N, int64_t E, uint16_t* dx, uint16_t* dw,
                                 uint32_t* status, void* gmm_scratch, cudaStream_t s, bool w_transposed);
// gmm_scratch: kGmmScratchBytes of workspace (used by dW).  h: SwiGLU forward
// output of H, or the saved H read by the SwiGLU-gradient epilogue.
moe_status_t launch_gmm(int mode, int epilogue, const uint16_t* a, const uint16_t* b, const int64_t* group_list,
                        int64_t M, int64_t K, int64_t N, int64_t E, const Act& act,
                        uint16_t* out, uint16_t* h_save, uint32_t* status, void* gmm_scratch, cudaStream_t s,
                        const GmmLaunch& how = GmmLaunch());
// Fused grouped matmuls (gmm.cu, 128-row tiles): gate_up reading its rows
// straight from the tokens x [T, K] (row r of the permuted order is token
// sorted_flat[r] / k) and writing the activation [M, N/2]; down writing the
// expert outputs to a scratch y2 [M, N] and combining each token's k rows
// into y [T, N] once the 256-column slice holding them is stored.  counters:
// fused_counter_bytes(N) of scratch, zero on entry (gate_up can zero
// n_counters of them for a down GMM that follows).
struct FusedOptions {
  bool discard = true;       // drop combined expert rows from L2 unwritten
  bool evict_first = true;   // stream the weights under an L2 evict-first policy (when experts
                             // average under 64 rows)
};
size_t fused_counter_bytes(int64_t N);
moe_status_t launch_gmm_gather_act(const uint16_t* x, const int32_t* sorted_flat, int64_t T, int64_t k,
                                   const uint16_t* w, const int64_t* group_list, int64_t M, int64_t K, int64_t N,
                                   int64_t E, const Act& act, bool w_transposed, uint16_t* out, int32_t* counters,
                                   int64_t n_counters, uint32_t* status, cudaStream_t s,
                                   const FusedOptions& opt = FusedOptions());
moe_status_t launch_gmm_combine(const uint16_t* a, const uint16_t* w, const int64_t* group_list,
                                const int32_t* row_id_map, const int32_t* sorted_flat, const float* topk_w, int64_t T,
                                int64_t k, int64_t M, int64_t K, int64_t N, int64_t E, bool w_transposed,
                                uint16_t* y2, int32_t* counters, uint16_t* y, uint32_t* status, cudaStream_t s,
                                const FusedOptions& opt = FusedOptions());
// Both expert matmuls of the inference layer in one persistent launch
// (gmm.cu): gate_up with the activation over rows gathered from x (row r is
// token sorted_flat[r] / k), then down; a [R, I] and y2 [R, H] out, R = T * k.
// Weights [E, H, 2I] and [E, I, H].  ready: expert_mlp_ready_bytes(R, E) of
// scratch, zero at launch (launch_permute can zero it).
size_t expert_mlp_ready_bytes(int64_t R, int64_t E);
moe_status_t launch_expert_mlp(const uint16_t* x, const int32_t* sorted_flat, const uint16_t* w1, const uint16_t* w2,
                               const int64_t* group_list, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                               const Act& act, uint16_t* a, uint16_t* y2, int32_t* ready, uint32_t* status,
                               cudaStream_t s);
// Block-scaled grouped matmul (gmm_mx.cu): a [M, K] fp8 with scales [M, K/32];
// b [E, N, K] fp8 with scales [E, N, K/32].  act == nullptr: bf16 out [M, N];
// else the activation of the [gate | up] halves, quantised into aq [M, N/2] /
// as [M, N/64] (element format out_fmt), h_save optional bf16 [M, N].
struct MxGmmArgs {
  const uint8_t* a;
  const uint8_t* a_sf;
  const uint8_t* b;
  const uint8_t* b_sf;
  const int64_t* group_list;
  int64_t M, K, N, E;
  int a_fmt, b_fmt;
  const Act* act;
  uint16_t* out;
  uint8_t* aq;
  uint8_t* as;
  int out_fmt;
  uint16_t* h_save;
};
moe_status_t launch_gmm_mx(const MxGmmArgs& args, uint32_t* status, cudaStream_t s);

// dX and dW of one grouped matmul (both read only inputs that exist before
// either starts): small problems run them side by side on halves of the GPU,
// large ones one after the other on all of it.  `dx_epilogue` / `h` as for
// launch_gmm's dX (plain, or the SwiGLU gradient with the saved H).  With
// w_transposed the weights are [E, N, K] and dw is written in that layout.
moe_status_t launch_gmm_backward(const uint16_t* x, const uint16_t* w, const int64_t* group_list, const uint16_t* dy,
                                 int64_t M, int64_t K, int64_t N, int64_t E, int dx_epilogue, const Act& act,
                                 const uint16_t* h, uint16_t* dx, uint16_t* dw, uint32_t* status, void* gmm_scratch,
                                 cudaStream_t s, bool w_transposed = false);

}  // namespace moe
