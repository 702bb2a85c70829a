// Combine side of the routed-expert path: weighted top-k combine (unpermute),
// its gradients, and the SwiGLU gradient.  All are HBM-bound row streams:
// 16-byte vector loads through the read-only path, fp32 accumulation in a
// fixed order (so results are deterministic), one bf16 rounding at the end.
//
//   combine       "MegaMoE", Token Combine: y_i = sum_k w_k Y_{e_ik}[row(i,k)].
//   token grad    "CANN ops-transformer 算子详解 MoeTokenPermuteWithRoutingMapGrad",
//                 2.3 and 6.2: per output token, walk its topK slots, skip -1,
//                 accumulate in fp32, cast back -- the same kernel with unit
//                 weights.
//   probs grad    the same article, 2.2, in the [T, topK] shape of its 6.3:
//                 dprobs[t,j] = <dy[t], Y[row(t,j)]>, with dY[row(t,j)] = w dy[t].
//   activation grad  "MegaMoE", 激活函数公式 (swiglu and its variants) differentiated.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"

namespace moe {
namespace {

constexpr int THREADS = 256;
constexpr int COLS_PER_BLOCK = THREADS * 8;  // 2048 bf16 per block row segment
constexpr int JB = 8;                         // slots loaded together

// Rows of the slots [j0, j0 + JB) of token t; a row outside [-1, rows_cap)
// raises MOE_ERR_DEVICE and counts as unused.  Every load is issued before
// any is checked: a check whose failure path writes the status word would
// make each load wait for the one before it.
__device__ __forceinline__ void slot_rows(const int32_t* __restrict__ row_id_map, int64_t t, int j0, int k,
                                          int64_t rows_cap, uint32_t* status, int32_t (&r)[JB]) {
#pragma unroll
  for (int jj = 0; jj < JB; ++jj) {
    const int j = j0 + jj;
    r[jj] = j < k ? row_id_map[t * k + j] : -1;
  }
  bool bad = false;
#pragma unroll
  for (int jj = 0; jj < JB; ++jj) {
    const bool b = r[jj] < -1 || r[jj] >= rows_cap;
    bad |= b;
    if (b) r[jj] = -1;
  }
  if (bad) set_status(status, MOE_ERR_DEVICE);
}

// Slots [j0, j0 + JB) of token t whose rows are r into acc, in slot order.
template <bool HAS_W>
__device__ __forceinline__ void add_slots(float (&acc)[8], const uint16_t* __restrict__ y_perm,
                                          const float* __restrict__ topk_w, const int32_t (&r)[JB], int64_t t,
                                          int j0, int k, int64_t H, int64_t col, const int32_t* __restrict__ row_id_map,
                                          int64_t rows_cap, uint32_t* status, int64_t t_next, int32_t (&r_next)[JB]) {
  uint4 v[JB];
  float w[JB];
  uint32_t live = 0;
#pragma unroll
  for (int jj = 0; jj < JB; ++jj) {
    if (r[jj] >= 0) {
      v[jj] = ld_nc_v4(y_perm + static_cast<int64_t>(r[jj]) * H + col);
      live |= 1u << jj;
    }
    w[jj] = (HAS_W && j0 + jj < k) ? topk_w[t * k + j0 + jj] : 1.0f;
  }
  if (t_next >= 0) slot_rows(row_id_map, t_next, 0, k, rows_cap, status, r_next);   // while the rows load
#pragma unroll
  for (int jj = 0; jj < JB; ++jj)
    if ((live >> jj) & 1u) add8(acc, v[jj], w[jj]);
}

// The token gradient (unit weights, large batches): grid (min(T, 3 x SMs),
// ceil(H / 2048)), three blocks per SM; each thread owns 8 consecutive columns
// and walks the tokens t = blockIdx.x, + gridDim.x, ...  The rows of the next
// token's first JB slots load while the current token's rows are in flight.
// Slots are summed in order j = 0, 1, ... as in unpermute_kernel, so both give
// the same bits.  (With the weights as well, this loop spills and is slower
// than unpermute_kernel.)
template <bool HAS_W>
__global__ void __launch_bounds__(THREADS, 3) token_sum_kernel(const uint16_t* __restrict__ y_perm,
                                                               const int32_t* __restrict__ row_id_map,
                                                               const float* __restrict__ topk_w, int64_t T, int64_t H,
                                                               int k, int64_t rows_cap, uint16_t* __restrict__ y,
                                                               uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int64_t col = static_cast<int64_t>(blockIdx.y) * COLS_PER_BLOCK + threadIdx.x * 8;
  int64_t t = blockIdx.x;
  if (col >= H || t >= T) return;
  int32_t rn[JB];
  slot_rows(row_id_map, t, 0, k, rows_cap, status, rn);
  for (; t < T; t += gridDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int32_t r[JB];
#pragma unroll
    for (int jj = 0; jj < JB; ++jj) r[jj] = rn[jj];
    const int64_t t_next = t + gridDim.x < T ? t + gridDim.x : -1;
    add_slots<HAS_W>(acc, y_perm, topk_w, r, t, 0, k, H, col, row_id_map, rows_cap, status, t_next, rn);
    for (int j0 = JB; j0 < k; j0 += JB) {   // more than JB slots: the rest without a prefetch
      int32_t rb[JB], unused[JB];
      slot_rows(row_id_map, t, j0, k, rows_cap, status, rb);
      add_slots<HAS_W>(acc, y_perm, topk_w, rb, t, j0, k, H, col, row_id_map, rows_cap, status, -1, unused);
    }
    *reinterpret_cast<uint4*>(y + t * H + col) = pack8(acc);
  }
}

// grid (min(T, 4 x SMs), ceil(H / 2048)), four blocks per SM (three without
// the weights, used for small batches only; at four it spills); each thread
// owns 8 consecutive columns and walks the tokens t = blockIdx.x,
// + gridDim.x, ...: a grid that never leaves a part-empty last wave (one block
// per token left 3.4 waves of short blocks at T=4096, and took 30.7 against
// 28.7 us there, 184 against 176 us at T=16384).  Slots are summed in order
// j = 0, 1, ...
template <bool HAS_W>
__global__ void __launch_bounds__(THREADS, HAS_W ? 4 : 3)
    unpermute_kernel(const uint16_t* __restrict__ y_perm, const int32_t* __restrict__ row_id_map,
                     const float* __restrict__ topk_w, int64_t T, int64_t H, int k, int64_t rows_cap,
                     uint16_t* __restrict__ y, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int64_t col = static_cast<int64_t>(blockIdx.y) * COLS_PER_BLOCK + threadIdx.x * 8;
  if (col >= H) return;
  bool bad = false;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < k; j0 += JB) {
      int32_t r[JB];
      float w[JB];
      uint4 v[JB];
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {   // every load first, then the checks
        const int j = j0 + jj;
        r[jj] = j < k ? row_id_map[t * k + j] : -1;
        w[jj] = (HAS_W && j < k) ? topk_w[t * k + j] : 1.0f;
      }
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {
        const bool b = r[jj] < -1 || r[jj] >= rows_cap;
        bad |= b;
        if (b) r[jj] = -1;
      }
#pragma unroll
      for (int jj = 0; jj < JB; ++jj)
        if (r[jj] >= 0) v[jj] = ld_nc_v4(y_perm + static_cast<int64_t>(r[jj]) * H + col);
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {
        if (r[jj] >= 0) add8(acc, v[jj], w[jj]);
      }
    }
    *reinterpret_cast<uint4*>(y + t * H + col) = pack8(acc);
  }
  if (bad) set_status(status, MOE_ERR_DEVICE);
}

// One block per token: writes dy_perm rows and reduces the k dot products.
__global__ void __launch_bounds__(THREADS) unpermute_backward_kernel(
    const uint16_t* __restrict__ dy, const uint16_t* __restrict__ y_perm, const int32_t* __restrict__ row_id_map,
    const float* __restrict__ topk_w, int64_t H, int k, int64_t rows_cap, uint16_t* __restrict__ dy_perm,
    float* __restrict__ dprobs, uint32_t* status) {
  __shared__ float red[THREADS / 32][JB];
  pdl_wait();
  pdl_trigger();
  const int64_t t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j0 = 0; j0 < k; j0 += JB) {
    int32_t r[JB];
    float w[JB], dot[JB];
#pragma unroll
    for (int jj = 0; jj < JB; ++jj) {   // every load first, then the checks
      const int j = j0 + jj;
      r[jj] = j < k ? row_id_map[t * k + j] : -1;
      w[jj] = (j < k && topk_w) ? topk_w[t * k + j] : 0.f;
      dot[jj] = 0.f;
    }
    bool bad = false;
#pragma unroll
    for (int jj = 0; jj < JB; ++jj) {
      const bool b = r[jj] < -1 || r[jj] >= rows_cap;
      bad |= b;
      if (b) r[jj] = -1;
    }
    if (bad && threadIdx.x == 0) set_status(status, MOE_ERR_DEVICE);
    for (int64_t col = threadIdx.x * 8; col < H; col += COLS_PER_BLOCK) {
      const uint4 g = ld_nc_v4(dy + t * H + col);
      float gf[8] = {bf16_lo(g.x), bf16_hi(g.x), bf16_lo(g.y), bf16_hi(g.y),
                     bf16_lo(g.z), bf16_hi(g.z), bf16_lo(g.w), bf16_hi(g.w)};
      uint4 v[JB];
#pragma unroll
      for (int jj = 0; jj < JB; ++jj)
        if (r[jj] >= 0) v[jj] = ld_nc_v4(y_perm + static_cast<int64_t>(r[jj]) * H + col);
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {
        if (r[jj] < 0) continue;
        float d = 0.f;
        d = fmaf(gf[0], bf16_lo(v[jj].x), d);
        d = fmaf(gf[1], bf16_hi(v[jj].x), d);
        d = fmaf(gf[2], bf16_lo(v[jj].y), d);
        d = fmaf(gf[3], bf16_hi(v[jj].y), d);
        d = fmaf(gf[4], bf16_lo(v[jj].z), d);
        d = fmaf(gf[5], bf16_hi(v[jj].z), d);
        d = fmaf(gf[6], bf16_lo(v[jj].w), d);
        d = fmaf(gf[7], bf16_hi(v[jj].w), d);
        dot[jj] += d;
        float o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = w[jj] * gf[i];
        *reinterpret_cast<uint4*>(dy_perm + static_cast<int64_t>(r[jj]) * H + col) = pack8(o);
      }
    }
    if (dprobs) {
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {
        float d = dot[jj];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        if (lane == 0) red[warp][jj] = d;
      }
      __syncthreads();
      if (threadIdx.x < JB) {
        const int j = j0 + threadIdx.x;
        float d = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < THREADS / 32; ++w8) d += red[w8][threadIdx.x];
        if (j < k) dprobs[t * k + j] = (r[threadIdx.x] >= 0) ? d : 0.f;
      }
      __syncthreads();
    }
  }
}

// Elementwise over rows x I: 8 columns per thread (gate at c, up at I + c).
__global__ void __launch_bounds__(THREADS) act_backward_kernel(const uint16_t* __restrict__ h,
                                                               const uint16_t* __restrict__ da, int64_t rows,
                                                               int64_t I, const Act act, uint16_t* __restrict__ dh) {
  pdl_wait();
  pdl_trigger();
  const int64_t per_row = I / 8;
  const int64_t items = rows * per_row;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x; it < items;
       it += static_cast<int64_t>(gridDim.x) * THREADS) {
    const int64_t r = it / per_row;
    const int64_t col = (it - r * per_row) * 8;
    const uint4 gv = ld_nc_v4(h + r * 2 * I + col);
    const uint4 uv = ld_nc_v4(h + r * 2 * I + I + col);
    const uint4 dv = ld_nc_v4(da + r * I + col);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
    const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
    float dg[8], du[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float g = (i & 1) ? bf16_hi(gw[i >> 1]) : bf16_lo(gw[i >> 1]);
      const float u = (i & 1) ? bf16_hi(uw[i >> 1]) : bf16_lo(uw[i >> 1]);
      const float d = (i & 1) ? bf16_hi(dw[i >> 1]) : bf16_lo(dw[i >> 1]);
      act_grad(g, u, d, act, dg[i], du[i]);
    }
    *reinterpret_cast<uint4*>(dh + r * 2 * I + col) = pack8(dg);
    *reinterpret_cast<uint4*>(dh + r * 2 * I + I + col) = pack8(du);
  }
}

}  // namespace

moe_status_t launch_unpermute(const uint16_t* y_perm, const int32_t* row_id_map, const float* topk_w,
                              int64_t T, int64_t H, int64_t k, uint16_t* y, uint32_t* status, cudaStream_t s) {
  const unsigned ycols = static_cast<unsigned>((H + COLS_PER_BLOCK - 1) / COLS_PER_BLOCK);
  const int64_t loop_blocks = 3 * static_cast<int64_t>(num_sms());
  const int64_t unperm_blocks = 4 * static_cast<int64_t>(num_sms());
  const dim3 grid(static_cast<unsigned>(T < unperm_blocks ? T : unperm_blocks), ycols);
  cudaError_t e;
  if (topk_w) {
    e = launch_pdl(unpermute_kernel<true>, grid, dim3(THREADS), 0, s, 1, y_perm, row_id_map, topk_w, T, H,
                   static_cast<int>(k), T * k, y, status);
  } else if (T > loop_blocks) {   // the token gradient of a large batch
    const dim3 g2(static_cast<unsigned>(loop_blocks), ycols);
    e = launch_pdl(token_sum_kernel<false>, g2, dim3(THREADS), 0, s, 1, y_perm, row_id_map,
                   static_cast<const float*>(nullptr), T, H, static_cast<int>(k), T * k, y, status);
  } else {
    e = launch_pdl(unpermute_kernel<false>, grid, dim3(THREADS), 0, s, 1, y_perm, row_id_map,
                   static_cast<const float*>(nullptr), T, H, static_cast<int>(k), T * k, y, status);
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t launch_unpermute_backward(const uint16_t* dy, const uint16_t* y_perm, const int32_t* row_id_map,
                                       const float* topk_w, int64_t T, int64_t H, int64_t k,
                                       uint16_t* dy_perm, float* dprobs, uint32_t* status, cudaStream_t s) {
  return launch_pdl(unpermute_backward_kernel, dim3(static_cast<unsigned>(T)), dim3(THREADS), 0, s, 1, dy, y_perm,
                    row_id_map, topk_w, H, static_cast<int>(k), T * k, dy_perm, dprobs, status) == cudaSuccess
             ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t launch_act_backward(const uint16_t* h, const uint16_t* da, int64_t rows, int64_t I, const Act& act,
                                 uint16_t* dh, cudaStream_t s) {
  const int64_t items = rows * (I / 8);
  int64_t blocks = (items + THREADS - 1) / THREADS;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(act_backward_kernel, dim3(static_cast<unsigned>(blocks)), dim3(THREADS), 0, s, 1, h, da, rows, I,
                    act, dh) == cudaSuccess
             ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
