// Token permute (dispatch): device histogram, exclusive scan and stable
// counting-sort scatter, then a row gather.
//
// "NPU Training Operators - GMM", section "算子语义": tokens must be laid out
// expert-contiguous with group_list holding the rows per expert (permute +
// histc in "Qwen3.5 MoE 路径"); "MegaMoE", EP Dispatch: each (token i, slot k)
// owns one row row(i,k) of its expert's block, rows stacked in a fixed order.
// The order used here is ascending flat slot f = t*k + j within an expert.
//
// Kernels (three launches, no host sync):
//   count   one block per chunk of 1024 slots: shared-memory histogram,
//           written as chunk_counts[e][chunk]; ids outside [-1, E) raise
//           MOE_ERR_DEVICE and are skipped.
//   rank    one block per chunk.  From all chunk counts, its chunk's first
//           row per expert (earlier chunks, then the exclusive scan over the
//           experts' totals; block 0 writes group_list).  Each of its 8 warps
//           owns 128 consecutive slots: per-warp expert counts -> per-warp
//           base rows; then every 32-slot step ranks equal ids with
//           __match_any_sync, which keeps the flat order (stable).  Writes
//           row_id_map and sorted_flat.
//   gather  warp per (token, 2 KB segment of its row): read once, stored to
//           the permuted row of each of the token's k slots: x_perm[row] = x[t].
//           Small batches take a warp per (slot, segment) instead, for more
//           warps in flight.
// Up to kSmallSlots slots (decode batches), one block does count, scan and
// rank (permute_small_kernel) and the gather follows: two launches instead of
// three, for index work that is all latency at that size.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"

namespace moe {
namespace {

constexpr int CHUNK = 1024;          // slots per block (count and rank)
constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;  // 8
constexpr int SUB = CHUNK / WARPS;   // 128 slots per warp in the rank kernel
constexpr int kSmallSlots = 1024;    // one-block index path up to this many slots

// Count, scan and rank of up to kSmallSlots slots in one block of 1024
// threads: a shared-memory histogram (the ids stay in shared memory), an
// exclusive scan over the experts (one per thread), then warp 0 walks the
// slots 32 at a time in flat order and ranks equal ids with __match_any_sync
// (stable), advancing a running row per expert.  Same outputs and status as
// count + rank.
__global__ void __launch_bounds__(1024) permute_small_kernel(const int32_t* __restrict__ ids, int nslots, int E,
                                                             int64_t* __restrict__ group_list,
                                                             int32_t* __restrict__ row_id_map,
                                                             int32_t* __restrict__ sorted_flat, uint32_t* status,
                                                             int32_t* zero, int64_t zero_n) {
  __shared__ int32_t cnt[kMaxExperts];
  __shared__ int32_t next_row[kMaxExperts];
  __shared__ int32_t id_sh[kSmallSlots];   // each slot's expert, -1 when unused or invalid
  __shared__ int32_t warp_sum[32];
  __shared__ int32_t R_sh;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int64_t i = tid; i < zero_n; i += 1024) zero[i] = 0;   // a scratch range the caller wants zeroed
  for (int e = tid; e < E; e += 1024) cnt[e] = 0;
  __syncthreads();
  for (int f = tid; f < nslots; f += 1024) {
    int e = ids[f];
    if (e < -1 || e >= E) {
      set_status(status, MOE_ERR_DEVICE);
      e = -1;
    } else if (e >= 0) {
      atomicAdd(&cnt[e], 1);
    }
    id_sh[f] = e;
  }
  __syncthreads();
  const int32_t v = tid < E ? cnt[tid] : 0;
  int32_t incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int32_t w = warp_sum[lane];
    int32_t wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += o;
    }
    warp_sum[lane] = wi - w;
    if (lane == 31) R_sh = wi;
  }
  __syncthreads();
  if (tid < E) {
    group_list[tid] = v;
    next_row[tid] = warp_sum[warp] + incl - v;
  }
  __syncthreads();
  if (warp == 0) {
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll 1
    for (int c = 0; c < nslots; c += 32) {
      const int f = c + lane;
      const int e = f < nslots ? id_sh[f] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0) {
        const int32_t row = next_row[e] + __popc(peers & lt);
        row_id_map[f] = row;
        if (in_bounds(row, nslots, status)) sorted_flat[row] = f;
      } else if (f < nslots) {
        row_id_map[f] = -1;
      }
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) next_row[e] += __popc(peers);
      __syncwarp();
    }
  }
  for (int r = R_sh + tid; r < nslots; r += 1024) sorted_flat[r] = -1;   // rows past R own no slot
}

__global__ void __launch_bounds__(THREADS) permute_count_kernel(const int32_t* __restrict__ ids, int64_t nslots,
                                                                int E, int nchunks, int32_t* __restrict__ chunk_counts,
                                                                uint32_t* status, int32_t* zero, int64_t zero_n) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x; i < zero_n;
       i += static_cast<int64_t>(gridDim.x) * THREADS)
    zero[i] = 0;   // a scratch range the caller wants zeroed
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += THREADS) hist[e] = 0;
  __syncthreads();
  const int64_t f0 = static_cast<int64_t>(blockIdx.x) * CHUNK;
  int e[CHUNK / THREADS];   // all loads first, then the counting
#pragma unroll
  for (int u = 0; u < CHUNK / THREADS; ++u) {
    const int64_t f = f0 + threadIdx.x + u * THREADS;
    e[u] = f < nslots ? ids[f] : -1;
  }
  bool bad = false;
#pragma unroll
  for (int u = 0; u < CHUNK / THREADS; ++u) {
    if (e[u] < -1 || e[u] >= E) bad = true;
    else if (e[u] >= 0) atomicAdd(&hist[e[u]], 1);
  }
  if (bad) set_status(status, MOE_ERR_DEVICE);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += THREADS)
    chunk_counts[static_cast<int64_t>(e) * nchunks + blockIdx.x] = hist[e];
}

// Rank kernel, one block per chunk.  It first turns the chunk counts of all
// chunks into this chunk's first row per expert: rows of expert e in earlier
// chunks plus the rows of all earlier experts (an exclusive scan over the
// experts of their totals).  Block 0 writes group_list; the blocks share the
// rows past R, which own no slot (-1 in sorted_flat).
__global__ void __launch_bounds__(THREADS) permute_rank_kernel(const int32_t* __restrict__ ids, int64_t nslots,
                                                               int E, int nchunks,
                                                               const int32_t* __restrict__ chunk_counts,
                                                               int64_t* __restrict__ group_list,
                                                               int32_t* __restrict__ row_id_map,
                                                               int32_t* __restrict__ sorted_flat, uint32_t* status) {
  extern __shared__ int32_t wbase[];  // [WARPS][E], then the chunk's first row per expert [E]
  int32_t* cbase = wbase + WARPS * E;
  __shared__ int32_t warp_sum[WARPS];
  __shared__ int32_t R_sh;
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < WARPS * E; i += THREADS) wbase[i] = 0;
  // this thread's experts: ept consecutive ones (E <= 4 x THREADS)
  const int ept = (E + THREADS - 1) / THREADS;
  int32_t tot[4] = {0, 0, 0, 0}, pre[4] = {0, 0, 0, 0};
  int32_t mine_tot = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = threadIdx.x * ept + i;
    if (i < ept && e < E) {
      const int32_t* row = chunk_counts + static_cast<int64_t>(e) * nchunks;
      for (int c0 = 0; c0 < nchunks; c0 += 8) {   // eight loads in flight at a time
        int32_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = c0 + u < nchunks ? row[c0 + u] : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          tot[i] += v[u];
          if (c0 + u < static_cast<int>(blockIdx.x)) pre[i] += v[u];
        }
      }
      mine_tot += tot[i];
    }
  }
  int32_t incl = mine_tot;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t run = 0;
    for (int w = 0; w < WARPS; ++w) {
      const int32_t v = warp_sum[w];
      warp_sum[w] = run;
      run += v;
    }
    R_sh = run;
  }
  __syncthreads();
  int32_t off = warp_sum[warp] + incl - mine_tot;   // rows of all experts before this thread's first
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = threadIdx.x * ept + i;
    if (i < ept && e < E) {
      cbase[e] = off + pre[i];
      if (blockIdx.x == 0) group_list[e] = tot[i];
      off += tot[i];
    }
  }
  for (int64_t r = R_sh + static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x; r < nslots;
       r += static_cast<int64_t>(gridDim.x) * THREADS)
    sorted_flat[r] = -1;
  __syncthreads();
  const int64_t f0 = static_cast<int64_t>(blockIdx.x) * CHUNK + warp * SUB;
  int32_t* mine = wbase + warp * E;
  // this warp's ids, loaded once for both passes (all loads in flight together)
  int ev[SUB / 32];
#pragma unroll
  for (int step = 0; step < SUB / 32; ++step) {
    const int64_t f = f0 + step * 32 + lane;
    ev[step] = f < nslots ? ids[f] : -1;
  }
#pragma unroll
  for (int step = 0; step < SUB / 32; ++step)
    if (ev[step] < -1 || ev[step] >= E) ev[step] = -1;
  // per-warp counts
#pragma unroll
  for (int step = 0; step < SUB / 32; ++step) {
    const int e = ev[step];
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // per-expert scan over the warps of this chunk, starting at the chunk's first row
  for (int e = threadIdx.x; e < E; e += THREADS) {
    int32_t run = cbase[e];
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const int32_t c = wbase[w * E + e];
      wbase[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int step = 0; step < SUB / 32; ++step) {
    const int64_t f = f0 + step * 32 + lane;
    const int e = ev[step];
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int32_t row = mine[e] + __popc(peers & lt);
      row_id_map[f] = row;
      if (in_bounds(row, nslots, status)) sorted_flat[row] = static_cast<int32_t>(f);
    } else if (f < nslots) {
      row_id_map[f] = -1;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
}

constexpr int SEG = 1024;  // bf16 elements per warp item (2 KB)

// Warp per (token, 2 KB segment of its row): the segment is read once and
// stored to the permuted row of each of the token's k slots.
__global__ void __launch_bounds__(THREADS) permute_gather_kernel(const uint16_t* __restrict__ x, int64_t T,
                                                                 int64_t H, int k,
                                                                 const int32_t* __restrict__ row_id_map,
                                                                 uint16_t* __restrict__ x_perm, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int64_t nseg = (H + SEG - 1) / SEG;
  const int64_t items = T * nseg;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * THREADS) >> 5;
  for (int64_t item = gw; item < items; item += nw) {   // the whole warp takes each item
    const int64_t t = item / nseg;
    const int64_t seg = item - t * nseg;
    const uint16_t* src = x + t * H + seg * SEG;
    const int64_t n = (H - seg * SEG) < SEG ? (H - seg * SEG) : static_cast<int64_t>(SEG);
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t c = (u * 32 + lane) * 8;
      if (c < n) v[u] = ld_nc_v4(src + c);
    }
    for (int j0 = 0; j0 < k; j0 += 32) {   // lane l fetches slot j0 + l's row, then the warp walks them
      const int32_t rl = j0 + lane < k ? row_id_map[t * k + j0 + lane] : -1;
      const int m = min(32, k - j0);
      for (int jj = 0; jj < m; ++jj) {
        const int32_t row = __shfl_sync(0xffffffffu, rl, jj);
        if (row < 0 || !in_bounds(row, T * k, status)) continue;
        uint16_t* dst = x_perm + static_cast<int64_t>(row) * H + seg * SEG;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t c = (u * 32 + lane) * 8;
          if (c < n) *reinterpret_cast<uint4*>(dst + c) = v[u];
        }
      }
    }
  }
}

// Warp per (slot, 2 KB segment): more warps than tokens, for small batches.
__global__ void __launch_bounds__(THREADS) permute_gather_slots_kernel(const uint16_t* __restrict__ x, int64_t nslots,
                                                                 int64_t H, int k,
                                                                 const int32_t* __restrict__ row_id_map,
                                                                 uint16_t* __restrict__ x_perm, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int64_t nseg = (H + SEG - 1) / SEG;
  const int64_t items = nslots * nseg;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * THREADS) >> 5;
  for (int64_t item = gw; item < items; item += nw) {
    const int64_t f = item / nseg;
    const int64_t seg = item - f * nseg;
    const int32_t row = row_id_map[f];
    if (row < 0 || !in_bounds(row, nslots, status)) continue;
    const int64_t t = f / k;
    const uint16_t* src = x + t * H + seg * SEG;
    uint16_t* dst = x_perm + static_cast<int64_t>(row) * H + seg * SEG;
    const int64_t n = (H - seg * SEG) < SEG ? (H - seg * SEG) : static_cast<int64_t>(SEG);
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t c = (u * 32 + lane) * 8;
      if (c < n) v[u] = ld_nc_v4(src + c);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t c = (u * 32 + lane) * 8;
      if (c < n) *reinterpret_cast<uint4*>(dst + c) = v[u];
    }
  }
}

}  // namespace

size_t permute_scratch_bytes(int64_t T, int64_t k, int64_t E) {
  const int64_t nslots = T * k;
  const int64_t nchunks = (nslots + CHUNK - 1) / CHUNK;
  return align256(static_cast<size_t>(nchunks * E) * sizeof(int32_t));
}

moe_status_t launch_permute(const uint16_t* x, const int32_t* ids, int64_t T, int64_t H, int64_t k, int64_t E,
                            uint16_t* x_perm, int64_t* group_list, int32_t* row_id_map, int32_t* sorted_flat,
                            uint32_t* status, void* scratch, cudaStream_t s, const MxOut* mx, int32_t* zero,
                            int64_t zero_n) {
  const int64_t nslots = T * k;
  const int nchunks = static_cast<int>((nslots + CHUNK - 1) / CHUNK);
  int32_t* chunk_counts = static_cast<int32_t*>(scratch);
  const int e = static_cast<int>(E);
  if (nslots <= kSmallSlots) {
    if (launch_pdl(permute_small_kernel, dim3(1), dim3(1024), 0, s, 1, ids, static_cast<int>(nslots), e, group_list,
                   row_id_map, sorted_flat, status, zero, zero_n) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else {
    if (launch_pdl(permute_count_kernel, dim3(nchunks), dim3(THREADS), e * sizeof(int32_t), s, 1, ids, nslots, e,
                   nchunks, chunk_counts, status, zero, zero_n) != cudaSuccess)
      return MOE_ERR_CUDA;
    const size_t rank_smem = static_cast<size_t>(WARPS + 1) * e * sizeof(int32_t);
    if (launch_pdl(permute_rank_kernel, dim3(nchunks), dim3(THREADS), rank_smem, s, 1, ids, nslots, e, nchunks,
                   static_cast<const int32_t*>(chunk_counts), group_list, row_id_map, sorted_flat, status) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (mx != nullptr && x != nullptr && H > 0) {
    if (launch_mx_gather(x, nslots, H, static_cast<int>(k), row_id_map, *mx, status, s) != MOE_OK)
      return MOE_ERR_CUDA;
  } else if (x != nullptr && x_perm != nullptr && H > 0) {
    const int64_t nseg = (H + SEG - 1) / SEG;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
    // token-major once there are enough tokens to fill the GPU's warps a few times over
    const bool by_token = T * nseg >= 4 * static_cast<int64_t>(num_sms()) * WARPS;
    const int64_t items = (by_token ? T : nslots) * nseg;
    int64_t blocks = (items + WARPS - 1) / WARPS;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const cudaError_t ge =
        by_token ? launch_pdl(permute_gather_kernel, dim3(static_cast<unsigned>(blocks)), dim3(THREADS), 0, s, 1, x,
                              T, H, static_cast<int>(k), static_cast<const int32_t*>(row_id_map), x_perm, status)
                 : launch_pdl(permute_gather_slots_kernel, dim3(static_cast<unsigned>(blocks)), dim3(THREADS), 0, s,
                              1, x, nslots, H, static_cast<int>(k), static_cast<const int32_t*>(row_id_map), x_perm,
                              status);
    if (ge != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
