// Q_MX of bf16 rows ("MegaMoE", "A8W8-FP 量化场景" and "A4W4-FP 量化场景",
// stage 1): the standalone row quantiser and the permute's quantising gather,
// which writes the rows of each expert straight into fp8 / fp4 codes and E8M0
// scales.  HBM-bound: per row, K*2 bytes read, K (fp4: K/2) + K/32 written.
//
// One warp per (row, 1024-element segment): lane l quantises group l of the
// segment from its 64 contiguous bytes, writes its 32 codes as two 16-byte
// stores (E2M1: one, two codes per byte, rows of K/2 bytes) and its scale byte
// (the warp's 32 scale bytes are contiguous).  The gather reads each token row
// once and stores its codes to all k of its permuted rows.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "mx.cuh"

namespace moe {
namespace {

constexpr int THREADS = 256;

// Quantised codes of one group, held in registers until they are stored.
template <int FMT>
struct GroupCodes {
  uint32_t c[FMT == MOE_FP4_E2M1 ? 4 : 8];
  uint32_t sc;
};

template <int FMT>
__device__ __forceinline__ void store_group(const GroupCodes<FMT>& g, uint8_t* q, uint8_t* scales, int64_t row,
                                            int64_t K, int64_t grp) {
  if constexpr (FMT == MOE_FP4_E2M1) {
    *reinterpret_cast<uint4*>(q + row * (K / 2) + grp * 16) = make_uint4(g.c[0], g.c[1], g.c[2], g.c[3]);
  } else {
    uint4* d = reinterpret_cast<uint4*>(q + row * K + grp * 32);
    d[0] = make_uint4(g.c[0], g.c[1], g.c[2], g.c[3]);
    d[1] = make_uint4(g.c[4], g.c[5], g.c[6], g.c[7]);
  }
  scales[row * (K / 32) + grp] = static_cast<uint8_t>(g.sc);
}

// Rows of x in, quantised rows out.  GATHER: x has T token rows and each is
// quantised once, then stored to the permuted row of each of its k routed
// slots (row_id_map[t*k + j], -1 for an unused slot): Q_MX of a row does not
// depend on where the row goes.
template <int FMT, bool GATHER>
__global__ void __launch_bounds__(THREADS) mx_rows_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                          const int32_t* __restrict__ row_id_map, int k,
                                                          uint8_t* __restrict__ q, uint8_t* __restrict__ scales,
                                                          uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int64_t groups = K / 32;
  const int64_t nseg = (groups + 31) / 32;
  const int64_t items = rows * nseg;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * THREADS) >> 5;
  for (int64_t item = gw; item < items; item += nw) {   // the whole warp takes each item
    const int64_t t = item / nseg;
    const int64_t grp = (item - t * nseg) * 32 + lane;
    const bool active = grp < groups;
    GroupCodes<FMT> g;
    if (active) {
      const uint16_t* src = x + t * K + grp * 32;
      float v[32];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 w = ld_nc_v4(src + 8 * u);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[8 * u + 2 * i] = bf16_lo(ws[i]);
          v[8 * u + 2 * i + 1] = bf16_hi(ws[i]);
        }
      }
      if constexpr (FMT == MOE_FP4_E2M1)
        g.sc = mx_quant32_fp4(v, g.c);
      else
        g.sc = mx_quant32<FMT>(v, g.c);
    }
    if constexpr (!GATHER) {
      if (active) store_group<FMT>(g, q, scales, t, K, grp);
    } else {
      for (int j0 = 0; j0 < k; j0 += 32) {   // lane l fetches slot j0 + l's row, then the warp walks them
        const int32_t rl = j0 + lane < k ? row_id_map[t * k + j0 + lane] : -1;
        const int n = min(32, k - j0);
        for (int jj = 0; jj < n; ++jj) {
          const int32_t r = __shfl_sync(0xffffffffu, rl, jj);
          if (r >= 0 && active && in_bounds(r, rows * k, status)) store_group<FMT>(g, q, scales, r, K, grp);
        }
      }
    }
  }
}

template <bool GATHER>
moe_status_t launch_rows(const uint16_t* x, int64_t n, int64_t K, const int32_t* row_id_map, int k, int fmt,
                         uint8_t* q, uint8_t* scales, uint32_t* status, cudaStream_t s) {
  const int64_t items = n * ((K / 32 + 31) / 32);
  int64_t blocks = (items + THREADS / 32 - 1) / (THREADS / 32);
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid(static_cast<unsigned>(blocks));
  cudaError_t e;
  if (fmt == MOE_FP8_E5M2)
    e = launch_pdl(mx_rows_kernel<MOE_FP8_E5M2, GATHER>, grid, dim3(THREADS), 0, s, 1, x, n, K, row_id_map, k, q,
                   scales, status);
  else if (fmt == MOE_FP4_E2M1)
    e = launch_pdl(mx_rows_kernel<MOE_FP4_E2M1, GATHER>, grid, dim3(THREADS), 0, s, 1, x, n, K, row_id_map, k, q,
                   scales, status);
  else
    e = launch_pdl(mx_rows_kernel<MOE_FP8_E4M3, GATHER>, grid, dim3(THREADS), 0, s, 1, x, n, K, row_id_map, k, q,
                   scales, status);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

moe_status_t launch_mx_quantize(const uint16_t* x, int64_t rows, int64_t K, int fmt, uint8_t* q, uint8_t* scales,
                                cudaStream_t s) {
  return launch_rows<false>(x, rows, K, nullptr, 1, fmt, q, scales, nullptr, s);
}

moe_status_t launch_mx_gather(const uint16_t* x, int64_t nslots, int64_t H, int k, const int32_t* row_id_map,
                              const MxOut& out, uint32_t* status, cudaStream_t s) {
  return launch_rows<true>(x, nslots / k, H, row_id_map, k, out.fmt, out.q, out.scales, status, s);
}

}  // namespace moe
