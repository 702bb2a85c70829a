// Q_MX of bf16 rows ("MegaMoE", "A8W8-FP 量化场景" and "A4W4-FP 量化场景",
// stage 1): the standalone row quantiser and the permute's quantising gather,
// which writes the rows of each expert straight into fp8 / fp4 codes and E8M0
// scales.  HBM-bound: per row, K*2 bytes read, K (fp4: K/2) + K/32 written.
//
// One warp per (row, 1024-element segment): lane l quantises group l of the
// segment from its 64 contiguous bytes, writes its 32 codes as two 16-byte
// stores (E2M1: one, two codes per byte, rows of K/2 bytes) and its scale byte
// (the warp's 32 scale bytes are contiguous).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "mx.cuh"

namespace moe {
namespace {

constexpr int THREADS = 256;

template <int FMT, bool GATHER>
__global__ void __launch_bounds__(THREADS) mx_rows_kernel(const uint16_t* __restrict__ x, int64_t nitems_rows,
                                                          int64_t K, const int32_t* __restrict__ row_id_map, int k,
                                                          uint8_t* __restrict__ q, uint8_t* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  const int64_t groups = K / 32;
  const int64_t nseg = (groups + 31) / 32;
  const int64_t items = nitems_rows * nseg;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * THREADS) >> 5;
  for (int64_t item = gw; item < items; item += nw) {
    const int64_t f = item / nseg;
    const int64_t seg = item - f * nseg;
    int64_t src_row = f, dst_row = f;
    if (GATHER) {  // f is a routed slot t*k + j: its row of the permuted output, its token's row of x
      const int32_t r = row_id_map[f];
      if (r < 0) continue;
      dst_row = r;
      src_row = f / k;
    }
    const int64_t grp = seg * 32 + lane;
    if (grp >= groups) continue;
    const uint16_t* src = x + src_row * K + grp * 32;
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
    uint32_t sc;
    if constexpr (FMT == MOE_FP4_E2M1) {
      uint32_t c[4];
      sc = mx_quant32_fp4(v, c);
      *reinterpret_cast<uint4*>(q + dst_row * (K / 2) + grp * 16) = make_uint4(c[0], c[1], c[2], c[3]);
    } else {
      uint32_t c[8];
      sc = mx_quant32<FMT>(v, c);
      uint4* d = reinterpret_cast<uint4*>(q + dst_row * K + grp * 32);
      d[0] = make_uint4(c[0], c[1], c[2], c[3]);
      d[1] = make_uint4(c[4], c[5], c[6], c[7]);
    }
    scales[dst_row * groups + grp] = static_cast<uint8_t>(sc);
  }
}

template <bool GATHER>
moe_status_t launch_rows(const uint16_t* x, int64_t n, int64_t K, const int32_t* row_id_map, int k, int fmt,
                         uint8_t* q, uint8_t* scales, cudaStream_t s) {
  const int64_t items = n * ((K / 32 + 31) / 32);
  int64_t blocks = (items + THREADS / 32 - 1) / (THREADS / 32);
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid(static_cast<unsigned>(blocks));
  cudaError_t e;
  if (fmt == MOE_FP8_E5M2)
    e = launch_pdl(mx_rows_kernel<MOE_FP8_E5M2, GATHER>, grid, dim3(THREADS), 0, s, 1, x, n, K, row_id_map, k, q,
                   scales);
  else if (fmt == MOE_FP4_E2M1)
    e = launch_pdl(mx_rows_kernel<MOE_FP4_E2M1, GATHER>, grid, dim3(THREADS), 0, s, 1, x, n, K, row_id_map, k, q,
                   scales);
  else
    e = launch_pdl(mx_rows_kernel<MOE_FP8_E4M3, GATHER>, grid, dim3(THREADS), 0, s, 1, x, n, K, row_id_map, k, q,
                   scales);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

moe_status_t launch_mx_quantize(const uint16_t* x, int64_t rows, int64_t K, int fmt, uint8_t* q, uint8_t* scales,
                                cudaStream_t s) {
  return launch_rows<false>(x, rows, K, nullptr, 1, fmt, q, scales, s);
}

moe_status_t launch_mx_gather(const uint16_t* x, int64_t nslots, int64_t H, int k, const int32_t* row_id_map,
                              const MxOut& out, cudaStream_t s) {
  return launch_rows<true>(x, nslots, H, row_id_map, k, out.fmt, out.q, out.scales, s);
}

}  // namespace moe
