// Block-scaled (MXFP8) grouped matmul on the 5th-generation tensor cores.
//
// What it computes follows "MegaMoE", "A8W8-FP 量化场景": for each expert e
// with rows [off_e, off_e + m_e) of the fp8 operand X,
//   P_e = DQ_MX(X_e) DQ_MX(W_e)^T
// with W_e = weight[e] stored [N, K] (one output channel per row) and one E8M0
// scale per 32 elements of K on both sides, as the page's MXFP constraints lay
// out weight1 / weight2 and weightScales1 / weightScales2.  The weights
// ("A8W4-FP 量化场景") and the tokens ("A4W4-FP 量化场景") may be FLOAT4_E2M1:
// packed two per byte in HBM, expanded by the TMA unit to the 16-byte-granule
// form the MMA reads, so a stage has the same shared-memory footprint and
// descriptors as with fp8.  Epilogues:
//   plain  (stage 3)  O_e = bf16(P_e);
//   ACT    (stage 2)  H = bf16(P_e) split into gate (first N/2 channels) and
//                     up (last N/2), A = Activation(G, U), then Q_MX(A): fp8
//                     codes and scales of the next matmul's operand.
//
// Design (one CTA per SM, 384 threads; 128 x 256 output tiles, K in blocks
// of 128 fp8 elements = one 128-byte swizzle row):
//   warp 0      tile producer.  Lane 0 issues the TMA copies of the A tile
//               (128 rows x 128) and the B tile (256 channels x 128) into a
//               4-stage ring; the B copies take an L2 evict-first policy when
//               the groups average under 64 rows (each weight tile is then
//               read once).
//   warps 10-11 scale producers.  Their lanes copy the stage's scales with
//               cp.async (4 bytes each: the 4 scales of one row) into the
//               stage's scale slot, in the order the tensor core reads them:
//               per 128 rows a 512-byte block in which row r's word sits at
//               word 4 (r % 32) + r / 32, and each lane's copies arrive on the
//               stage's full barrier when they land (cp.async.mbarrier.arrive),
//               so the barrier completes with the TMA bytes and all 64 lanes'
//               scales and no producer waits for its copies.  Issuing the
//               384 scale copies of a stage takes longer than issuing its
//               tile copies, so they are spread over two warps that run
//               beside the TMA thread.
//   warp 1      TMEM allocator; one thread, after the stage's full barrier and
//               a proxy fence (the scales were written by the generic proxy),
//               copies the stage's scales into TMEM
//               (tcgen05.cp 32x128b, replicated to all four lane quarters:
//               4 columns for A, 8 for B) and issues four
//               tcgen05.mma.kind::mxf8f6f4.block_scale (M=128, N=256, K=32)
//               whose scale-factor ids pick byte kk of each scale word.
//   warps 2..9  epilogue, two warps per TMEM lane quarter, each taking half
//               of the tile's columns: tcgen05.ld -> registers (bf16) ->
//               release the accumulator -> activation / Q_MX -> global stores.
//               A quarter with no row of the tile releases at once.
// TMEM: one 256-column fp32 accumulator (the scales of the stages take 48
// more columns, and a second accumulator does not fit in 512 with them); the
// epilogue releases it as soon as the tile is in registers.
// Group structure, tile order, bounded waits and the abort path are those of
// the bf16 kernel (gmm.cu).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "mx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;                     // fp8 elements (bytes) per stage row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;            // 16 KB
constexpr int B_BYTES = BN * BK;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SFA_BYTES = BM * 4;           // 4 scales per row per stage
constexpr int SFB_BYTES = BN * 4;
constexpr int SF_STAGE_BYTES = SFA_BYTES + SFB_BYTES;
constexpr int ACC_COLS = BN;
constexpr int SF_COLS = 12;                 // TMEM columns per scale slot: 4 (A) + 8 (B)
constexpr int SF_SLOTS = STAGES;            // one scale slot per stage (shared memory and TMEM)
constexpr int SF_WARPS = 2;                // warps copying the scales
constexpr int FULL_ARRIVALS = 1 + 32 * SF_WARPS;  // the TMA arrival and each scale-warp lane's copies
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int SF_WARP = 2 + EPI_WARPS;      // the first scale warp; the others follow it
constexpr int NUM_THREADS = 32 * (SF_WARP + SF_WARPS);
constexpr uint64_t kTimeoutNs = 4000000000ull;
static_assert(ACC_COLS + SF_SLOTS * SF_COLS <= TMEM_COLS, "TMEM budget");

enum { MX_PLAIN = 0, MX_ACT = 1 };

#ifndef MOE_MX_PREFETCH_MB
#define MOE_MX_PREFETCH_MB 24
#endif
constexpr int kMxPrefetchMB = MOE_MX_PREFETCH_MB;   // weight bytes prefetched into L2 before the wait

struct MxParams {
  const int64_t* group_list;
  const uint8_t* a_sf;   // [M, K/32]
  const uint8_t* b_sf;   // [E, N, K/32]
  int E;
  int64_t rows_cap;      // M
  int N;                 // channels of each expert's weight
  int sf_ld;             // K / 32
  int tile_cols;
  int kblocks;           // K / 128
  int out_cols;          // plain: N; ACT: N / 2
  uint16_t* out;         // plain: bf16 [M, N]
  uint8_t* aq;           // ACT: fp8 [M, N/2]
  uint8_t* as;           // ACT: [M, N/64]
  uint16_t* h_save;      // ACT: optional bf16 [M, N]
  uint32_t out32;        // the outputs (plain: out; ACT: aq and h_save) are 32-byte aligned, so
                         // rows are written in 32-byte pieces
  Act act;
  uint32_t idesc;
  uint32_t tx_bytes;     // bytes a stage's A and B copies deliver: E2M1 operands count their packed size
  uint32_t w_evict_first;  // weight tiles loaded under an L2 evict-first policy
  uint32_t* status;
  const uint8_t* b;      // the weight codes, for the L2 prefetch before the wait
  int64_t b_prefetch;    // bytes of b to prefetch, and of b_sf
  int64_t sf_prefetch;
};

struct __align__(16) MxSmem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full;
  uint64_t tmem_empty;
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
  int32_t bad;
  int32_t ntiles;
  int32_t grp_off[kMaxExperts + 1];    // M < 2^31 (checked by the ABI)
  int32_t grp_cnt[kMaxExperts];
  int32_t tile_start[kMaxExperts + 1];
};

// [A|B stages, 1024-aligned][scale slots][MxSmem]
constexpr size_t kSmemBytes = 1024 + STAGES * STAGE_BYTES + SF_SLOTS * SF_STAGE_BYTES + sizeof(MxSmem);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct TileInfo {
  int g;
  int64_t row0;
  int rows_valid;
  int col0;   // first output column (ACT: first activation column)
};

template <int EPI>
__device__ __forceinline__ TileInfo decode_tile(const MxSmem* sm, const MxParams& p, int t) {
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sm->tile_start[mid] <= t) lo = mid; else hi = mid;
  }
  TileInfo ti;
  const int local = t - sm->tile_start[lo];
  const int rt = local / p.tile_cols;
  const int ct = local - rt * p.tile_cols;
  ti.g = lo;
  ti.col0 = ct * (EPI == MX_ACT ? BN / 2 : BN);
  ti.row0 = sm->grp_off[lo] + static_cast<int64_t>(rt) * BM;
  ti.rows_valid = min(BM, sm->grp_cnt[lo] - rt * BM);
  return ti;
}

// One 32-byte store: a whole sector, where two 16-byte stores would each fill half of one.
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "l"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait_bounded(bar, parity, abort, kTimeoutNs) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  uint32_t dummy = 0;
  mbar_wait_bounded(bar, parity, &dummy, 200000000ull);
}

// Copy one stage's scales into a scale slot: lane l copies the words of rows
// l + 32 j of the A tile (j < 4) and of channels l + 32 j of the B tile
// (j < 8) to the tensor core's order, split in two halves of six words, one
// per scale warp (PART 0: the A words and B's j < 2; PART 1: B's j >= 2).
// Rows past M and channels past N copy zeros (their data arrive as zeros from
// the TMA unit).
template <int EPI, int PART>
__device__ __forceinline__ void copy_sf(const MxParams& p, const TileInfo& ti, int kb, int lane, uint32_t slot) {
  const int64_t ld = p.sf_ld;
  if (PART == 0) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t r = ti.row0 + lane + 32 * j;
      const bool in = r < p.rows_cap;
      cp_async4(slot + 16 * lane + 4 * j, p.a_sf + (in ? r * ld + 4 * kb : 0), in ? 4u : 0u);
    }
  }
  const uint8_t* bsf = p.b_sf + static_cast<int64_t>(ti.g) * p.N * ld + 4 * kb;
#pragma unroll
  for (int j = PART == 0 ? 0 : 2; j < (PART == 0 ? 2 : 8); ++j) {
    int n;
    if (EPI == MX_ACT)  // channels [0, 128) of the tile: gate; [128, 256): the matching up channels
      n = (j < 4 ? ti.col0 : p.out_cols + ti.col0) + lane + 32 * (j & 3);
    else
      n = ti.col0 + lane + 32 * j;
    const bool in = n < p.N;
    cp_async4(slot + SFA_BYTES + 512 * (j >> 2) + 16 * lane + 4 * (j & 3),
              in ? bsf + static_cast<int64_t>(n) * ld : p.b_sf, in ? 4u : 0u);
  }
}

// Position of the producer in its walk over (tile, K block) stages.
struct StageIter {
  int t;
  int kb;
  bool valid;
  TileInfo ti;
};

template <int EPI>
__device__ __forceinline__ void stage_iter_start(StageIter& w, const MxSmem* sm, const MxParams& p, int ntiles) {
  w.t = blockIdx.x;
  w.kb = 0;
  w.valid = w.t < ntiles;
  if (w.valid) w.ti = decode_tile<EPI>(sm, p, w.t);
}

template <int EPI>
__device__ __forceinline__ void stage_iter_next(StageIter& w, const MxSmem* sm, const MxParams& p, int ntiles) {
  if (!w.valid) return;
  if (++w.kb == p.kblocks) {
    w.kb = 0;
    w.t += gridDim.x;
    w.valid = w.t < ntiles;
    if (w.valid) w.ti = decode_tile<EPI>(sm, p, w.t);
  }
}

template <int EPI, int OUT_FMT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gmm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const MxParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sf_smem = smem + STAGES * STAGE_BYTES;
  MxSmem* sm = reinterpret_cast<MxSmem*>(sf_smem + SF_SLOTS * SF_STAGE_BYTES);
  const uint32_t stage_base = smem_u32(smem);
  const uint32_t sf_base = smem_u32(sf_smem);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;

  // ---------------------------------------------------------------- set-up
  if (tid == 0) {
    sm->bad = 0;
    sm->abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sm->full[s]), FULL_ARRIVALS);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    mbar_init(smem_u32(&sm->tmem_full), 1);
    mbar_init(smem_u32(&sm->tmem_empty), EPI_WARPS);
    mbar_init(smem_u32(&sm->drain), 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2 && p.b_prefetch > 0) {
    // While the launch before this one still runs, pull the first experts'
    // weights and their scales into L2: the first wave of tiles starts with
    // the lowest experts.  CTA b takes the b-th share, 16 KB a lane and copy.
    const int64_t share = (p.b_prefetch / gridDim.x) & ~int64_t(15);
    const uint8_t* base = p.b + share * blockIdx.x;
    for (int64_t off = static_cast<int64_t>(lane) * 16384; off < share; off += 32 * 16384)
      prefetch_l2_bulk(base + off, static_cast<uint32_t>(share - off < 16384 ? share - off : 16384));
    const int64_t sshare = (p.sf_prefetch / gridDim.x) & ~int64_t(15);
    if (lane == 0 && sshare > 0) prefetch_l2_bulk(p.b_sf + sshare * blockIdx.x, static_cast<uint32_t>(sshare));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  pdl_trigger();
  for (int e = tid; e < E; e += NUM_THREADS) {
    const int64_t c = p.group_list[e];
    if (c < 0 || c > p.rows_cap) atomicOr(&sm->bad, 1);
    sm->grp_cnt[e] = static_cast<int32_t>(c < 0 ? 0 : (c > p.rows_cap ? p.rows_cap : c));
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int lo = min(E, lane * per), hi = min(E, lo + per);
    int64_t rows = 0;
    int32_t tiles = 0;
    for (int e = lo; e < hi; ++e) {
      rows += sm->grp_cnt[e];
      tiles += ((sm->grp_cnt[e] + BM - 1) / BM) * p.tile_cols;
    }
    int64_t rows_incl = rows;
    int32_t tiles_incl = tiles;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t r2 = __shfl_up_sync(0xffffffffu, rows_incl, d);
      const int32_t t2 = __shfl_up_sync(0xffffffffu, tiles_incl, d);
      if (lane >= d) { rows_incl += r2; tiles_incl += t2; }
    }
    int64_t rb = rows_incl - rows;
    int32_t tb = tiles_incl - tiles;
    for (int e = lo; e < hi; ++e) {
      sm->grp_off[e] = static_cast<int32_t>(rb);
      sm->tile_start[e] = tb;
      rb += sm->grp_cnt[e];
      tb += ((sm->grp_cnt[e] + BM - 1) / BM) * p.tile_cols;
    }
    if (lane == 31) {
      sm->grp_off[E] = static_cast<int32_t>(rows_incl);
      sm->tile_start[E] = tiles_incl;
      sm->ntiles = tiles_incl;
      if (rows_incl > p.rows_cap) sm->bad = 1;
    }
  }
  __syncthreads();
  const uint32_t tmem_base = sm->tmem_base;
  const int ntiles = sm->bad ? 0 : sm->ntiles;   // a bad group_list: no tile, straight to teardown
  if (sm->bad && tid == 0 && blockIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE);
  volatile uint32_t* abort_flag = &sm->abort;

  if (warp == 0) {
    // ---------------------------------------------------------------- tile producer (one thread)
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      StageIter cur;
      const uint64_t pol = p.w_evict_first ? l2_policy_evict_first() : 0ull;
      stage_iter_start<EPI>(cur, sm, p, ntiles);
      while (cur.valid) {
        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
        if (!mbar_wait_bounded(smem_u32(&sm->empty[s]), ph ^ 1u, abort_flag, kTimeoutNs)) { ok = false; break; }
        const uint32_t bar = smem_u32(&sm->full[s]);
        const uint32_t a_dst = stage_base + s * STAGE_BYTES;
        const uint32_t b_dst = a_dst + A_BYTES;
        const TileInfo& ti = cur.ti;
        mbar_expect_tx(bar, p.tx_bytes);
        tma_load_2d(a_dst, &tmA, bar, cur.kb * BK, static_cast<int32_t>(ti.row0));
        // ACT: 128 gate channels, then the 128 matching up channels
        const int c1 = EPI == MX_ACT ? p.out_cols + ti.col0 : 0;
        if (p.w_evict_first) {
          tma_load_3d_hint(b_dst, &tmB, bar, cur.kb * BK, ti.col0, ti.g, pol);
          if (EPI == MX_ACT) tma_load_3d_hint(b_dst + (BN / 2) * BK, &tmB, bar, cur.kb * BK, c1, ti.g, pol);
        } else {
          tma_load_3d(b_dst, &tmB, bar, cur.kb * BK, ti.col0, ti.g);
          if (EPI == MX_ACT) tma_load_3d(b_dst + (BN / 2) * BK, &tmB, bar, cur.kb * BK, c1, ti.g);
        }
        ++it;
        stage_iter_next<EPI>(cur, sm, p, ntiles);
      }
      if (!ok) {  // copies still in flight land before the CTA exits (bounded: the scale warp may have stopped)
        const uint32_t first = it > STAGES ? it - STAGES : 0;
        for (uint32_t i = first; i < it; ++i) drain_wait(smem_u32(&sm->full[i % STAGES]), (i / STAGES) & 1u);
      }
    }
  } else if (warp >= SF_WARP) {
    // ---------------------------------------------------------------- scale producers (whole warps)
    uint32_t it = 0;
    StageIter cur;
    stage_iter_start<EPI>(cur, sm, p, ntiles);
    while (cur.valid) {
      const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
      if (!warp_wait(smem_u32(&sm->empty[s]), ph ^ 1u, abort_flag, lane)) break;
      if (warp == SF_WARP)
        copy_sf<EPI, 0>(p, cur.ti, cur.kb, lane, sf_base + s * SF_STAGE_BYTES);
      else
        copy_sf<EPI, 1>(p, cur.ti, cur.kb, lane, sf_base + s * SF_STAGE_BYTES);
      cp_async_arrive_noinc(smem_u32(&sm->full[s]));   // arrives when this lane's copies have landed
      ++it;
      stage_iter_next<EPI>(cur, sm, p, ntiles);
    }
    cp_async_wait_all();                   // no copy of this CTA outlives it
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (one thread)
    if (lane == 0) {
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++local) {
        if (!mbar_wait_bounded(smem_u32(&sm->tmem_empty), (local & 1u) ^ 1u, abort_flag, kTimeoutNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait_bounded(smem_u32(&sm->full[s]), ph, abort_flag, kTimeoutNs)) { ok = false; break; }
          tc_fence_after();
          fence_proxy_async_smem();        // the scales came through the generic proxy (cp.async)
          const uint32_t a_addr = stage_base + s * STAGE_BYTES;
          const uint32_t b_addr = a_addr + A_BYTES;
          const uint32_t sf_slot = s;
          const uint32_t sfa_smem = sf_base + sf_slot * SF_STAGE_BYTES;
          const uint32_t sf_col = tmem_base + ACC_COLS + sf_slot * SF_COLS;
          tc_cp_32x128b_x4(sf_col, smem_desc_plain(sfa_smem, 128, 128));
          tc_cp_32x128b_x4(sf_col + 4, smem_desc_plain(sfa_smem + SFA_BYTES, 128, 128));
          tc_cp_32x128b_x4(sf_col + 8, smem_desc_plain(sfa_smem + SFA_BYTES + 512, 128, 128));
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint64_t ad = smem_desc_sw128(a_addr + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b_addr + kk * 32, 16, 1024);
            tc_mma_mxf8(tmem_base, ad, bd, p.idesc | idesc_sf_ids(kk, kk), sf_col, sf_col + 4, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&sm->empty[s]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm->tmem_full));
      }
      if (!ok) {
        tc_commit(smem_u32(&sm->drain));
        drain_wait(smem_u32(&sm->drain), 0);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                   // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;         // which half of the tile's columns
    const int row_in_tile = q * 32 + lane;
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t local = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++local) {
      const TileInfo ti = decode_tile<EPI>(sm, p, t);
      const bool row_ok = row_in_tile < ti.rows_valid && in_bounds(ti.row0 + row_in_tile, p.rows_cap, p.status);
      const int64_t row = ti.row0 + row_in_tile;
      if (!warp_wait(smem_u32(&sm->tmem_full), local & 1u, abort_flag, lane)) break;
      if (q * 32 >= ti.rows_valid) {   // no row of this lane quarter is stored: release at once
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm->tmem_empty));
        continue;
      }
      tc_fence_after();
      if (EPI == MX_ACT) {
        // activation columns [64 half, 64 half + 64): gate at TMEM columns 64 half + c,
        // up at 128 + 64 half + c; held as bf16 pairs (gate low, up high)
        const int I = p.out_cols;
        uint32_t gu[64];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + 64 * half + 32 * cc, g);
          tmem_ld32(taddr + BN / 2 + 64 * half + 32 * cc, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) gu[32 * cc + i] = pack_bf16x2(__uint_as_float(g[i]), __uint_as_float(u[i]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm->tmem_empty));
        if (row_ok) {
          const int c0 = ti.col0 + 64 * half;
          uint32_t scales = 0;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            float a[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)   // H is bf16; the activation is taken on those values
              a[i] = act_forward(bf16_lo(gu[32 * cc + i]), bf16_hi(gu[32 * cc + i]), p.act);
            uint32_t c8[8];
            scales |= mx_quant32<OUT_FMT>(a, c8) << (8 * cc);
            if (p.out32) {
              st_global_v8(p.aq + row * I + c0 + 32 * cc, c8);
            } else {
              uint4* dq = reinterpret_cast<uint4*>(p.aq + row * I + c0 + 32 * cc);
              dq[0] = make_uint4(c8[0], c8[1], c8[2], c8[3]);
              dq[1] = make_uint4(c8[4], c8[5], c8[6], c8[7]);
            }
          }
          *reinterpret_cast<uint16_t*>(p.as + row * (I / 32) + c0 / 32) = static_cast<uint16_t>(scales);
          if (p.h_save) {
            uint16_t* hg = p.h_save + row * (2 * static_cast<int64_t>(I)) + c0;
#pragma unroll
            for (int v = 0; v < 4; ++v) {   // 16 columns of gate and of up at a time
              uint32_t gw[8], uw[8];
#pragma unroll
              for (int w = 0; w < 8; ++w) {
                const uint32_t p0 = gu[16 * v + 2 * w], p1 = gu[16 * v + 2 * w + 1];
                gw[w] = (p0 & 0xFFFFu) | (p1 << 16);
                uw[w] = (p0 >> 16) | (p1 & 0xFFFF0000u);
              }
              if (p.out32) {
                st_global_v8(hg + 16 * v, gw);
                st_global_v8(hg + I + 16 * v, uw);
              } else {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                  reinterpret_cast<uint4*>(hg + 16 * v)[h2] = make_uint4(gw[4 * h2], gw[4 * h2 + 1], gw[4 * h2 + 2],
                                                                         gw[4 * h2 + 3]);
                  reinterpret_cast<uint4*>(hg + I + 16 * v)[h2] = make_uint4(uw[4 * h2], uw[4 * h2 + 1],
                                                                             uw[4 * h2 + 2], uw[4 * h2 + 3]);
                }
              }
            }
          }
        }
      } else {
        uint32_t packed[64];   // this warp's 128 columns of the tile row, as bf16 pairs
#pragma unroll
        for (int cc = 0; cc < 4; cc += 2) {
          uint32_t r0[32], r1[32];
          tmem_ld32(taddr + 128 * half + 32 * cc, r0);
          tmem_ld32(taddr + 128 * half + 32 * (cc + 1), r1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            packed[16 * cc + i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
            packed[16 * (cc + 1) + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm->tmem_empty));
        if (row_ok) {
          const int c0 = ti.col0 + 128 * half;
          uint16_t* dst = p.out + row * p.out_cols + c0;
          if (p.out32) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              if (c0 + 32 * cc < p.out_cols) {
                st_global_v8(dst + 32 * cc, &packed[16 * cc]);
                st_global_v8(dst + 32 * cc + 16, &packed[16 * cc + 8]);
              }
          } else {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              if (c0 + 32 * cc < p.out_cols) {
                uint4* d = reinterpret_cast<uint4*>(dst + 32 * cc);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                  d[v] = make_uint4(packed[16 * cc + 4 * v], packed[16 * cc + 4 * v + 1], packed[16 * cc + 4 * v + 2],
                                    packed[16 * cc + 4 * v + 3]);
              }
            }
          }
        }
      }
    }
  }

  __syncthreads();
  if (sm->abort && tid == 0) set_status(p.status, MOE_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int EPI, int OUT_FMT>
moe_status_t launch_kernel(const CUtensorMap& ta, const CUtensorMap& tb, const MxParams& p, cudaStream_t s) {
  auto kern = gmm_mx_kernel<EPI, OUT_FMT>;
  static int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes)) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    configured_dev = dev;
  }
  if (launch_pdl(kern, dim3(num_sms()), dim3(NUM_THREADS), kSmemBytes, s, 1, ta, tb, p) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

moe_status_t launch_gmm_mx(const MxGmmArgs& x, uint32_t* status, cudaStream_t s) {
  MxParams p{};
  // weights streamed under an L2 evict-first policy only when experts average
  // under 64 rows (decode), as in the bf16 grouped matmul: there each weight
  // tile is read once, while larger groups read it again from L2 for each of
  // their 128-row tiles
  p.w_evict_first = x.M < 64 * x.E ? 1u : 0u;
  // the L2 prefetch before the wait (at most all of the weights), with the
  // matching share of their scales (a scale byte per 32 elements)
  {
    const int64_t elems = x.E * x.N * x.K;
    const int64_t b_bytes = x.b_fmt == MOE_FP4_E2M1 ? elems / 2 : elems;
    const int64_t budget = static_cast<int64_t>(kMxPrefetchMB) << 20;
    p.b = x.b;
    p.b_prefetch = budget < b_bytes ? budget : b_bytes;
    p.sf_prefetch = p.b_prefetch / (b_bytes / (elems / 32));
  }
  p.group_list = x.group_list;
  p.a_sf = x.a_sf;
  p.b_sf = x.b_sf;
  p.E = static_cast<int>(x.E);
  p.rows_cap = x.M;
  p.N = static_cast<int>(x.N);
  p.sf_ld = static_cast<int>(x.K / 32);
  p.kblocks = static_cast<int>(x.K / BK);
  p.status = status;
  p.idesc = idesc_mxf8(BM, BN, x.a_fmt, x.b_fmt);
  // a 4-bit map fills the same shared memory as an fp8 one but counts the packed bytes it read
  const bool a_fp4 = (x.a_fmt == MOE_FP4_E2M1), b_fp4 = (x.b_fmt == MOE_FP4_E2M1);
  p.tx_bytes = (a_fp4 ? A_BYTES / 2 : A_BYTES) + (b_fp4 ? B_BYTES / 2 : B_BYTES);
  const bool act = x.act != nullptr;
  p.out_cols = static_cast<int>(act ? x.N / 2 : x.N);
  p.tile_cols = act ? static_cast<int>((x.N / 2) / (BN / 2)) : static_cast<int>((x.N + BN - 1) / BN);
  p.out = x.out;
  p.aq = x.aq;
  p.as = x.as;
  p.h_save = x.h_save;
  const auto a32 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 31u) == 0; };
  p.out32 = (act ? a32(x.aq) && a32(x.h_save) : a32(x.out)) ? 1u : 0u;
  if (act) p.act = *x.act;
  CUtensorMap ta, tb;
  if (!(a_fp4 ? make_map_2d_fp4(&ta, x.a, x.M, x.K, BM) : make_map_2d_u8(&ta, x.a, x.M, x.K, BM)) ||
      !(b_fp4 ? make_map_3d_fp4(&tb, x.b, x.E, x.N, x.K, act ? BN / 2 : BN)
              : make_map_3d_u8(&tb, x.b, x.E, x.N, x.K, act ? BN / 2 : BN)))
    return MOE_ERR_CUDA;
  if (!act) return launch_kernel<MX_PLAIN, MOE_FP8_E4M3>(ta, tb, p, s);
  return x.out_fmt == MOE_FP8_E5M2 ? launch_kernel<MX_ACT, MOE_FP8_E5M2>(ta, tb, p, s)
                                   : launch_kernel<MX_ACT, MOE_FP8_E4M3>(ta, tb, p, s);
}

}  // namespace moe
