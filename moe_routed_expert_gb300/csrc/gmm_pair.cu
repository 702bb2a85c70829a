// Grouped matmul on CTA pairs (tcgen05 cta_group::2): forward, input gradient
// and weight gradient.
//
// Same operations as gmm.cu ("NPU Training Operators - GMM", section "算子语义":
// y_g = x_g @ W_g, dx_g = dy_g @ W_g^T over the rows of each group, and
// dW_g = x_g^T @ dy_g contracted over the group's own rows, zero for an empty
// group; the gate_up forward can end with the clipped SwiGLU of "MegaMoE",
// "激活函数公式"), laid out for GB300's paired SMs:
//
//   * a cluster of two CTAs owns a 256 x 256 output tile; CTA r loads rows
//     [128r, 128r+128) of A and columns [128r, 128r+128) of B (32 KB per 64-deep
//     stage instead of 48 KB), and one thread of the even CTA issues
//     tcgen05.mma.cta_group::2 (M=256, N=256, K=16), which reads both CTAs'
//     shared memory and writes each CTA's 128 rows into its own TMEM;
//   * both CTAs' TMA copies complete on the even CTA's stage barrier;
//     tcgen05.commit multicasts the stage release and the accumulator-ready
//     signal to both CTAs; both epilogues release the accumulator on the even
//     CTA's barrier;
//   * 5 stages of 32 KB; two 256-column fp32 accumulators (all 512 TMEM columns);
//   * the epilogue stages each warp's 32 rows x 128 columns as bf16 in
//     shared memory (XOR-swizzled 16-byte chunks, conflict-free).  A plain
//     product leaves through TMA tile stores (two 64-column boxes per warp
//     and half tile; the map clips columns past N); the rows of a group's last
//     tile that end inside a warp's 32, and the SwiGLU epilogues, are written
//     two full rows per warp instruction (coalesced), masking rows past the
//     group end and columns past N.
//   * dW contracts over each group's own rows.  For every group it starts, the
//     producer warp rewrites a copy of each TMA descriptor (base address = the
//     group's first row, row extent = the group's row count) and publishes it
//     to a per-CTA slot in the workspace, so rows past the group end arrive as
//     zeros from the TMA unit itself.
//   * tiles go to the clusters as sched.cuh describes: strided over all tiles
//     (group by group, column tile fastest), or, for a weight gradient whose
//     operands fit in L2, a run of clusters per group sized to even out the
//     groups' different contraction depths.  dW visits the groups largest
//     first: the deepest tiles start together and share their operands in L2.
// Group offsets are read on the device as in gmm.cu.  Every mbarrier wait is
// bounded; a timeout stops all roles, waits for copies in flight, frees TMEM
// and writes MOE_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "sched.cuh"

namespace moe {
namespace {

constexpr int BM = 128;                         // rows per CTA (256 per pair)
constexpr int BN = 256;                         // accumulator columns
constexpr int BNH = 128;                        // B columns held by each CTA
constexpr int BK = 64;
constexpr int STAGES = 5;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BNH * BK * 2;           // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB per CTA
constexpr int BOX_BYTES = 64 * 64 * 2;
constexpr int EPI_ROW_BYTES = 256;              // 128 bf16 columns
constexpr int EPI_WARP_BYTES = 32 * EPI_ROW_BYTES;
constexpr int EPI_BYTES = 4 * EPI_WARP_BYTES;   // 32 KB
constexpr int BOX_STAGE = 32 * 128;             // one warp's 32 rows x 64 columns, bf16
constexpr int TMEM_COLS = 2 * BN;
constexpr int NUM_THREADS = 192;
constexpr uint64_t kTimeoutNs = 4000000000ull;
// dW is scheduled by group when its operands (x and dy rows of every group)
// take at most this many bytes and at most this many groups have rows.
constexpr int64_t kByGroupMaxBytes = 64ll << 20;
constexpr int kByGroupMaxGroups = 32;
// A dW tile's epilogue takes about as long as this many 64-deep MMA blocks.
constexpr uint32_t kEpilogueBlocks = 8;
// dX and dW in one launch: relative cost of a 64-deep block of each (measured
// on GB300: about 0.31 us for dX's K-major operands, 0.36 us for dW's MN-major ones).
constexpr uint32_t kBlockCostDx = 7;
constexpr uint32_t kBlockCostDw = 8;

struct PairParams {
  const int64_t* group_list;
  int E;
  int64_t rows_cap;
  int out_rows;     // dW: rows of one expert's gradient (K)
  int out_cols;     // output columns (FWD: N or I; DX: K; DW: N)
  int tile_cols;    // column tiles
  int kblocks;      // contraction blocks of 64
  uint16_t* out;
  int64_t ld_out;
  uint16_t* h_save;
  const uint16_t* h_in;   // SwiGLU gradient: saved pre-activation [rows, 2I]
  int act_cols;     // SwiGLU: I
  Act act;          // gated activation (SwiGLU epilogues)
  uint32_t* status;
  // dW: the operands' bases and row pitches, and kMapSlots descriptor pairs per CTA
  const uint8_t* a_base;
  const uint8_t* b_base;
  int64_t a_pitch;
  int64_t b_pitch;
  uint8_t* map_slots;
  int concurrent;   // see GmmLaunch
  int wt;           // FWD/DX: each expert's weight stored transposed, [N, K]
};

struct __align__(128) PairSmem {
  uint8_t map_edit[2][128];    // dW: descriptors being rewritten (A, B)
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
  int32_t bad;
  int32_t n_empty;                     // groups without rows
  int32_t n_live;                      // groups with rows
  int32_t by_group;                    // dW: tiles scheduled by group
  int64_t units;                       // dW: contraction blocks of all tiles
  int64_t grp_off[kMaxExperts + 1];
  int32_t grp_cnt[kMaxExperts];
  int32_t order[kMaxExperts];          // visiting position -> group (dW: largest first)
  int32_t tile_start[kMaxExperts + 1]; // tile prefix over visiting positions (dW: groups with rows only)
  int32_t run_start[kMaxExperts + 1];  // dW by group: prefix over visiting positions of the cluster runs
  int32_t empty_ids[kMaxExperts];      // dW: the groups without rows
  int32_t xtile_start[kMaxExperts + 1];  // dX and dW together: dX tile prefix over the groups
  int32_t ncl_x;                       // dX and dW together, split schedule: clusters given to dX
};

constexpr size_t kSmemBytes = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + sizeof(PairSmem);
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct PairTile {
  int g;
  int64_t row0;     // FWD/DX: first row of this CTA's half; DW: first output row of it
  int rows_valid;   // rows of this CTA's half that belong to the output (may be <= 0)
  int col0;         // first output column of the pair tile (SwiGLU: first activation column)
  int kblocks;      // contraction blocks of 64
  int64_t m0;       // DW: first contraction row (the group's first row)
  int depth;        // DW: contraction rows of the group
};

// Cost of a dW tile of a group with `cnt` rows, in 64-deep blocks.
__device__ __forceinline__ uint32_t tile_cost(int cnt) {
  const uint32_t kb = (cnt + BK - 1) / BK;
  return kb > kEpilogueBlocks ? kb : kEpilogueBlocks;
}

// Tile `local` of group g (row tile major, column tile fastest) of a tile of
// mode `mode` (FWD, DX or DW), p holding that mode's sizes.
template <int EPI>
__device__ __forceinline__ PairTile decode_pair_tile(const PairSmem* sm, const PairParams& p, int mode, int g,
                                                     int local, uint32_t rank) {
  const int rt = local / p.tile_cols;
  const int ct = local - rt * p.tile_cols;
  PairTile ti;
  ti.g = g;
  const int first = rt * (2 * BM) + static_cast<int>(rank) * BM;
  ti.col0 = ct * (EPI == EPI_SWIGLU ? BN / 2 : BN);
  if (mode == GMM_DW) {
    ti.row0 = first;
    ti.rows_valid = min(BM, p.out_rows - first);
    ti.m0 = sm->grp_off[g];
    ti.depth = sm->grp_cnt[g];
    ti.kblocks = (ti.depth + BK - 1) / BK;
  } else {
    ti.row0 = sm->grp_off[g] + first;
    ti.rows_valid = min(BM, sm->grp_cnt[g] - first);
    ti.m0 = 0;
    ti.depth = 0;
    ti.kblocks = p.kblocks;
  }
  return ti;
}

// Which tiles a cluster takes (the same for every role of both CTAs): a
// strided walk over the tile prefix T of nT groups (start, start + stride,
// ...), or its run of the by-group schedule (prefix T over nT groups, cluster
// runs C).  TileRef.g is the index into T.
struct Walk {
  const int32_t* T;
  const int32_t* C;
  int nT, start, stride;
  bool by_group, none;
};

struct ClusterTiles {
  Walk k;
  TileWalk w;
  __device__ __forceinline__ explicit ClusterTiles(const Walk& k_) : k(k_) {
    if (k.by_group) walk_group_init(w, k.start, k.C, k.nT);
    else walk_strided_init(w, k.start);
    if (k.none) w.t = INT64_MAX, w.g = -1;
  }
  __device__ __forceinline__ bool next(TileRef& r) {
    if (k.none) return false;
    return k.by_group ? walk_group_next(w, k.T, r) : walk_strided_next(w, k.T, k.nT, k.stride, r);
  }
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait_bounded(bar, parity, abort, kTimeoutNs) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  uint32_t dummy = 0;
  mbar_wait_bounded(bar, parity, &dummy, 200000000ull);
}

// 32 fp32 accumulator columns of this thread's row -> bf16 -> 4 swizzled
// 16-byte chunks (chunk index c0 .. c0+3) of this thread's staging row.
__device__ __forceinline__ void stage_chunk(uint8_t* ebuf, int lane, int c0, const uint32_t (&r)[32]) {
  uint8_t* row = ebuf + lane * EPI_ROW_BYTES;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint4 q;
    q.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
    q.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
    q.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
    q.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
    const int c = (c0 + v) ^ (lane & 7);
    *reinterpret_cast<uint4*>(row + c * 16) = q;
  }
}

// The same 32 columns into the TMA store layout: two 64-column boxes of 32
// rows x 128 bytes, 16-byte chunk j of row r at (j ^ (r & 7)) (128B swizzle).
__device__ __forceinline__ void stage_box(uint8_t* ebuf, int lane, int cc, const uint32_t (&r)[32]) {
  uint8_t* row = ebuf + (cc >> 6) * BOX_STAGE + lane * 128;
  const int j0 = (cc & 63) >> 3;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint4 q;
    q.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
    q.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
    q.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
    q.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
    *reinterpret_cast<uint4*>(row + (((j0 + v) ^ (lane & 7)) * 16)) = q;
  }
}

// flush_rows for the box layout.
__device__ __forceinline__ void flush_rows_box(const uint8_t* ebuf, int lane, uint16_t* base, int64_t ld,
                                               int rows_valid, int ncols) {
  const int j = lane & 15;
  const int half = lane >> 4;
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int row = 2 * i + half;
    const uint4 v = *reinterpret_cast<const uint4*>(ebuf + (j >> 3) * BOX_STAGE + row * 128 +
                                                    (((j & 7) ^ (row & 7)) * 16));
    if (row < rows_valid && j * 8 < ncols) *reinterpret_cast<uint4*>(base + row * ld + j * 8) = v;
  }
}

// Write the warp's staged 32 rows x 128 columns: two rows per instruction,
// 16 lanes x 16 bytes per row.  Rows >= rows_valid and columns >= ncols are skipped.
__device__ __forceinline__ void flush_rows(const uint8_t* ebuf, int lane, uint16_t* base, int64_t ld, int rows_valid,
                                           int ncols) {
  const int j = lane & 15;
  const int half = lane >> 4;
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int row = 2 * i + half;
    const uint4 v = *reinterpret_cast<const uint4*>(ebuf + row * EPI_ROW_BYTES + ((j ^ (row & 7)) * 16));
    if (row < rows_valid && j * 8 < ncols) *reinterpret_cast<uint4*>(base + row * ld + j * 8) = v;
  }
}

// MODE GMM_BWD runs the dX (tmA, tmB, tmC, p) and dW (tmA2, tmB2, tmC2, pw)
// contractions of one grouped matmul in one launch: each cluster takes tiles
// of one of the two (see the schedule below).  The other modes use the first
// set only.
template <int MODE, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gmm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmA2,
                const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmC2,
                const PairParams p, const PairParams pw) {
  static_assert(MODE != GMM_BWD || EPI == EPI_PLAIN, "dX and dW together: plain epilogues only");
  constexpr bool DW_SCHED = (MODE == GMM_DW) || (MODE == GMM_BWD);   // groups visited largest first
  // the dW operands and parameters
  const PairParams& pd = (MODE == GMM_BWD) ? pw : p;
  const CUtensorMap* dwA = (MODE == GMM_BWD) ? &tmA2 : &tmA;
  const CUtensorMap* dwB = (MODE == GMM_BWD) ? &tmB2 : &tmB;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ebuf_all = smem + STAGES * STAGE_BYTES;
  PairSmem* sm = reinterpret_cast<PairSmem*>(ebuf_all + EPI_BYTES);
  const uint32_t stage_base = smem_u32(smem);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;
  const uint32_t rank = cluster_ctarank();
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(nclusters_x());

  // ---------------------------------------------------------------- set-up
  if (tid == 0) {
    sm->bad = 0;
    sm->abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sm->tmem_full[a]), 1);
      mbar_init(smem_u32(&sm->tmem_empty[a]), 8);  // 4 epilogue warps in each CTA
    }
    mbar_init(smem_u32(&sm->drain), 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (EPI == EPI_PLAIN) tma_prefetch_desc(&tmC);
    if (MODE == GMM_BWD) {
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
      tma_prefetch_desc(&tmC2);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&sm->tmem_base), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // the peer's barriers are initialised before any remote arrive or copy completion
  // Everything above touches only shared memory, TMEM and the kernel
  // parameters, so it overlaps the tail of the previous kernel on the stream.
  if (!p.concurrent) pdl_wait();
  pdl_trigger();
  for (int e = tid; e < E; e += NUM_THREADS) {
    const int64_t c = p.group_list[e];
    if (c < 0 || c > p.rows_cap) atomicOr(&sm->bad, 1);
    sm->grp_cnt[e] = static_cast<int32_t>(c < 0 ? 0 : (c > p.rows_cap ? p.rows_cap : c));
  }
  __syncthreads();
  if (DW_SCHED) {
    // largest group first (ties: lower id first)
    for (int e = tid; e < E; e += NUM_THREADS) {
      const int ce = sm->grp_cnt[e];
      int r = 0;
      for (int e2 = 0; e2 < E; ++e2) {
        const int c2 = sm->grp_cnt[e2];
        r += (c2 > ce) || (c2 == ce && e2 < e);
      }
      sm->order[r] = e;
    }
  } else {
    for (int e = tid; e < E; e += NUM_THREADS) sm->order[e] = e;
  }
  __syncthreads();
  // Prefix over the groups of rows, over visiting positions of tiles (dW:
  // groups with rows only), and the list of the groups without rows.
  const int dw_tiles = ((pd.out_rows + 2 * BM - 1) / (2 * BM)) * pd.tile_cols;
  auto tiles_of = [&](int c) -> int {
    return DW_SCHED ? (c > 0 ? dw_tiles : 0) : ((c + 2 * BM - 1) / (2 * BM)) * p.tile_cols;
  };
  auto xtiles_of = [&](int c) -> int { return ((c + 2 * BM - 1) / (2 * BM)) * p.tile_cols; };
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int lo = min(E, lane * per), hi = min(E, lo + per);
    int64_t rows = 0, units = 0;
    int32_t tiles = 0, empties = 0, xtiles = 0;
    for (int e = lo; e < hi; ++e) {
      const int c = sm->grp_cnt[e];
      const int kb = (c + BK - 1) / BK;
      rows += c;
      tiles += tiles_of(sm->grp_cnt[sm->order[e]]);
      units += static_cast<int64_t>(tiles_of(c)) * kb;
      empties += (c == 0);
      if (MODE == GMM_BWD) xtiles += xtiles_of(c);
    }
    int64_t rows_incl = rows, units_incl = units;
    int32_t tiles_incl = tiles, empties_incl = empties, xtiles_incl = xtiles;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t r2 = __shfl_up_sync(0xffffffffu, rows_incl, d);
      const int64_t u2 = __shfl_up_sync(0xffffffffu, units_incl, d);
      const int32_t t2 = __shfl_up_sync(0xffffffffu, tiles_incl, d);
      const int32_t e2 = __shfl_up_sync(0xffffffffu, empties_incl, d);
      const int32_t x2 = __shfl_up_sync(0xffffffffu, xtiles_incl, d);
      if (lane >= d) { rows_incl += r2; units_incl += u2; tiles_incl += t2; empties_incl += e2; xtiles_incl += x2; }
    }
    int64_t rb = rows_incl - rows;
    int32_t tb = tiles_incl - tiles, eb = empties_incl - empties, xb = xtiles_incl - xtiles;
    for (int e = lo; e < hi; ++e) {
      const int c = sm->grp_cnt[e];
      sm->grp_off[e] = rb;
      sm->tile_start[e] = tb;
      rb += c;
      tb += tiles_of(sm->grp_cnt[sm->order[e]]);
      if (c == 0) sm->empty_ids[eb++] = e;
      if (MODE == GMM_BWD) {
        sm->xtile_start[e] = xb;
        xb += xtiles_of(c);
      }
    }
    if (lane == 31) {
      sm->grp_off[E] = rows_incl;
      sm->tile_start[E] = tiles_incl;
      if (MODE == GMM_BWD) sm->xtile_start[E] = xtiles_incl;
      sm->n_empty = empties_incl;
      sm->n_live = E - empties_incl;
      sm->units = units_incl;
      sm->by_group = 0;
      if (rows_incl > p.rows_cap) sm->bad = 1;
    }
  }
  __syncthreads();
  if (DW_SCHED) {
    // Few groups whose operands fit in L2: warp 0 searches the smallest
    // per-cluster load L for which every group j gets a run of
    // ceil(tiles_j / floor(L / cost_j)) clusters within the grid, cost_j the
    // tile's blocks of 64 but at least kEpilogueBlocks (a tile's epilogue
    // takes about that long, and it bounds short tiles).  Two rounds of 32
    // candidates (one per lane), the first over [lb, 2 lb), lb the larger of
    // the costliest tile and the average load.  Taken when L is within 15% of
    // the average.
    // With dX and dW together, all of dX's tiles (N/64 blocks each) are one
    // more "group" after dW's, and the costs weigh a block of each by its speed.
    const int nl = sm->n_live;
    const int32_t xt = (MODE == GMM_BWD) ? sm->xtile_start[E] : 0;
    const int npos = nl + (xt > 0 ? 1 : 0);
    const int64_t units_x = static_cast<int64_t>(xt) * p.kblocks;
    const int64_t bytes = sm->grp_off[E] * (static_cast<int64_t>(pd.out_rows) + pd.out_cols) * 2;
    if (warp == 0 && !sm->bad && npos >= 1 && npos <= kByGroupMaxGroups && npos <= ncl &&
        bytes <= kByGroupMaxBytes && sm->units + units_x < (1ll << 18) && dw_tiles < (1 << 12) && xt < (1 << 12)) {
      // Lane j holds the tile count and cost of visiting position j; with the
      // groups visited largest first, positions [0, nl) are the groups with
      // rows, and position nl is dX's tiles.
      const uint32_t my_tiles = lane < nl ? static_cast<uint32_t>(dw_tiles)
                                          : (lane == nl && xt > 0 ? static_cast<uint32_t>(xt) : 0u);
      const uint32_t wdw = (MODE == GMM_BWD) ? kBlockCostDw : 1u;
      const uint32_t my_cost = lane < nl ? wdw * tile_cost(sm->grp_cnt[sm->order[lane]])
                                         : (lane == nl && xt > 0 ? kBlockCostDx * max(static_cast<uint32_t>(p.kblocks),
                                                                                      kEpilogueBlocks) : 0u);
      const uint32_t cost_max = __reduce_max_sync(0xffffffffu, my_cost);
      const uint32_t cost_sum = __reduce_add_sync(0xffffffffu, my_cost * my_tiles);
      auto need = [&](uint32_t L) -> uint32_t {  // clusters for load L (every lane takes part)
        uint32_t n = 0;
#pragma unroll 1
        for (int i = 0; i < npos; ++i)
          n += group_clusters(__shfl_sync(0xffffffffu, my_tiles, i), __shfl_sync(0xffffffffu, my_cost, i), L, ncl);
        return n;
      };
      uint32_t best = 0;
      if (cost_sum < (1u << 20)) {  // every candidate L stays below 2^21
        const uint32_t lb = max(cost_max, udiv_small(cost_sum + ncl - 1, ncl));
        uint32_t lo = lb, step = (lb + 31) / 32;
#pragma unroll 1
        for (int round = 0; round < 2; ++round) {
          const unsigned ok = __ballot_sync(0xffffffffu, need(lo + step * lane) <= static_cast<uint32_t>(ncl));
          if (ok == 0) break;
          const int f = __ffs(ok) - 1;
          best = lo + step * f;
          if (f == 0) break;
          lo = lo + step * (f - 1) + 1;
          step = (step + 30) / 31;
        }
      }
      if (best != 0 && static_cast<uint64_t>(best) * ncl * 100 <= static_cast<uint64_t>(cost_sum) * 115) {
        const int32_t runs = lane < npos ? static_cast<int32_t>(group_clusters(my_tiles, my_cost, best, ncl)) : 0;
        int32_t incl = runs;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int32_t r2 = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += r2;
        }
        const int32_t total = __shfl_sync(0xffffffffu, incl, 31);
        if (lane < npos) sm->run_start[lane] = incl - runs;
        for (int j = npos + lane; j <= E; j += 32) sm->run_start[j] = total;
        if (lane == 0) sm->by_group = 1;
      }
    }
    if (MODE == GMM_BWD && tid == 0) {
      // without the by-group schedule: the clusters split between dX and dW in
      // proportion to their blocks of 64
      const int64_t uw = sm->units;
      int nx;
      if (units_x == 0) nx = 0;
      else if (uw == 0) nx = ncl;
      else {
        nx = static_cast<int>((units_x * ncl + (units_x + uw) / 2) / (units_x + uw));  // rounded; no FP64
        nx = nx < 1 ? 1 : (nx > ncl - 1 ? ncl - 1 : nx);
      }
      sm->ncl_x = nx;
    }
    __syncthreads();
  }
  if (sm->bad && tid == 0 && blockIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE);
  const bool no_work = sm->bad != 0;  // both CTAs of the pair read the same group_list: no tiles for either

  // This cluster's tiles and their mode (both CTAs of the pair agree: they
  // read the same group_list and make the same choices).
  int mode = (MODE == GMM_BWD) ? GMM_DX : MODE;
  Walk wk;
  if (MODE == GMM_BWD) {
    const int nl = sm->n_live;
    if (sm->by_group) {
      const int xr0 = sm->run_start[nl], xr1 = sm->run_start[nl + 1];
      if (cid < xr0) {
        mode = GMM_DW;
        wk = Walk{sm->tile_start, sm->run_start, nl, cid, 0, true, no_work};
      } else {
        wk = Walk{sm->xtile_start, nullptr, E, cid - xr0, max(xr1 - xr0, 1), false, no_work || cid >= xr1};
      }
    } else {
      const int nx = sm->ncl_x;
      if (cid < nx) {
        wk = Walk{sm->xtile_start, nullptr, E, cid, nx, false, no_work};
      } else {
        mode = GMM_DW;
        wk = Walk{sm->tile_start, nullptr, E, cid - nx, ncl - nx, false, no_work};
      }
    }
  } else {
    wk = Walk{sm->tile_start, sm->run_start, E, cid, ncl, sm->by_group != 0, no_work};
  }
  const PairParams& q = (mode == GMM_DW) ? pd : p;
  const bool A_MN = (mode == GMM_DW);
  // B is MN-major (output columns contiguous) for dW (dy rows), for the forward
  // over [K, N] weights and for dX over transposed [N, K] weights.
  const bool B_MN = (mode == GMM_DW) || ((mode == GMM_FWD) != (p.wt != 0));
  const uint32_t IDESC = idesc_bf16_f32(2 * BM, BN, A_MN, B_MN);
  const CUtensorMap* mC = (MODE == GMM_BWD && mode == GMM_DW) ? &tmC2 : &tmC;
  // tile reference -> group: dW walks visit positions (largest group first), the others groups
  auto group_of = [&](const TileRef& r) -> int { return mode == GMM_DW ? sm->order[r.g] : r.g; };

  const uint32_t tmem_base = sm->tmem_base;
  volatile uint32_t* abort_flag = &sm->abort;

  if (warp == 0 && mode == GMM_DW) {
    // ---------------------------------------------------------------- dW TMA producer (both CTAs)
    // The whole warp walks the tiles (it rewrites descriptors together); lane 0 copies.
    uint8_t* slots = pd.map_slots + static_cast<size_t>(blockIdx.x) * kMapSlots * 256;
    const uint32_t edit_a = smem_u32(sm->map_edit[0]), edit_b = smem_u32(sm->map_edit[1]);
    uint32_t it = 0;
    int ok = 1, cur_g = -1, slot = -1;
    const void* map_a = nullptr;
    const void* map_b = nullptr;
    ClusterTiles tiles(wk);
    TileRef tr;
    while (ok && tiles.next(tr)) {
      const PairTile ti = decode_pair_tile<EPI>(sm, pd, GMM_DW, group_of(tr), tr.local, rank);
      if (ti.g != cur_g) {
        // a new group: descriptors whose row 0 is the group's first row and
        // whose row extent is the group's row count
        cur_g = ti.g;
        slot = (slot + 1) % kMapSlots;  // a slot is rewritten only after its copies have all landed
        uint8_t* ga = slots + slot * 256;
        uint8_t* gb = ga + 128;
        if (lane < 8) {
          reinterpret_cast<uint4*>(sm->map_edit[0])[lane] = reinterpret_cast<const uint4*>(dwA)[lane];
          reinterpret_cast<uint4*>(sm->map_edit[1])[lane] = reinterpret_cast<const uint4*>(dwB)[lane];
        }
        __syncwarp();
        if (lane == 0) {
          tmap_set_address(edit_a, reinterpret_cast<uint64_t>(pd.a_base + ti.m0 * pd.a_pitch));
          tmap_set_rows(edit_a, static_cast<uint32_t>(ti.depth));
          tmap_set_address(edit_b, reinterpret_cast<uint64_t>(pd.b_base + ti.m0 * pd.b_pitch));
          tmap_set_rows(edit_b, static_cast<uint32_t>(ti.depth));
        }
        __syncwarp();
        tmap_publish(ga, edit_a);
        tmap_publish(gb, edit_b);
        if (lane == 0) {
          tmap_acquire(ga);
          tmap_acquire(gb);
        }
        map_a = ga;
        map_b = gb;
      }
      if (lane == 0) {
        const int bcol = ti.col0 + static_cast<int>(rank) * BNH;
        for (int kb = 0; kb < ti.kblocks; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait_bounded(smem_u32(&sm->empty[s]), ph ^ 1u, abort_flag, kTimeoutNs)) { ok = 0; break; }
          const uint32_t a_dst = stage_base + s * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          const uint32_t bar_local = smem_u32(&sm->full[s]);
          const uint32_t bar = mapa_shared(bar_local, 0);
          if (rank == 0) mbar_expect_tx(bar_local, 2 * STAGE_BYTES);
#pragma unroll
          for (int i2 = 0; i2 < BM / 64; ++i2)
            tma_load_2d_pair(a_dst + i2 * BOX_BYTES, map_a, bar, static_cast<int32_t>(ti.row0) + 64 * i2, kb * BK);
#pragma unroll
          for (int j = 0; j < BNH / 64; ++j) tma_load_2d_pair(b_dst + j * BOX_BYTES, map_b, bar, bcol + 64 * j, kb * BK);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0) {  // every stage filled here must be released before the CTA may exit
      const uint32_t first = it > STAGES ? it - STAGES : 0;
      for (uint32_t i2 = first; i2 < it; ++i2) {
        if (*abort_flag) break;
        mbar_wait_bounded(smem_u32(&sm->empty[i2 % STAGES]), (i2 / STAGES) & 1u, abort_flag, kTimeoutNs);
      }
    }
  } else if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      ClusterTiles tiles(wk);
      TileRef tr;
      while (ok && tiles.next(tr)) {
        const PairTile ti = decode_pair_tile<EPI>(sm, p, mode, group_of(tr), tr.local, rank);
        for (int kb = 0; kb < ti.kblocks; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait_bounded(smem_u32(&sm->empty[s]), ph ^ 1u, abort_flag, kTimeoutNs)) { ok = false; break; }
          const uint32_t a_dst = stage_base + s * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          const uint32_t bar_local = smem_u32(&sm->full[s]);
          const uint32_t bar = mapa_shared(bar_local, 0);  // the even CTA's stage barrier
          if (rank == 0) mbar_expect_tx(bar_local, 2 * STAGE_BYTES);
          tma_load_2d_pair(a_dst, &tmA, bar, kb * BK, static_cast<int32_t>(ti.row0));
          // this CTA's 128 output columns of B: the gate or the up half with SwiGLU
          const int bcol = EPI == EPI_SWIGLU ? (rank == 0 ? ti.col0 : p.act_cols + ti.col0)
                                             : ti.col0 + static_cast<int>(rank) * BNH;
          if (B_MN) {  // weight rows hold output columns: two 64-column boxes
#pragma unroll
            for (int j = 0; j < BNH / 64; ++j)
              tma_load_3d_pair(b_dst + j * BOX_BYTES, &tmB, bar, bcol + 64 * j, kb * BK, ti.g);
          } else {     // weight rows hold the contraction: one box of 128 rows
            tma_load_3d_pair(b_dst, &tmB, bar, kb * BK, bcol, ti.g);
          }
        }
      }
      // every stage this CTA filled must be released before the CTA may exit:
      // the release is an arrival sent from the even CTA
      const uint32_t first = it > STAGES ? it - STAGES : 0;
      for (uint32_t i = first; i < it; ++i) {
        if (*abort_flag) break;
        mbar_wait_bounded(smem_u32(&sm->empty[i % STAGES]), (i / STAGES) & 1u, abort_flag, kTimeoutNs);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA, one thread)
    // A single thread waits and issues: warp-wide shuffles and syncs per stage
    // measurably delay the MMA stream.
    if (rank == 0 && lane == 0) {
      uint32_t it = 0, local = 0;
      bool ok = true;
      ClusterTiles tiles(wk);
      TileRef tr;
      while (ok && tiles.next(tr)) {
        const int kblocks = decode_pair_tile<EPI>(sm, q, mode, group_of(tr), tr.local, 0).kblocks;
        const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
        if (!mbar_wait_bounded(smem_u32(&sm->tmem_empty[acc]), aph ^ 1u, abort_flag, kTimeoutNs)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait_bounded(smem_u32(&sm->full[s]), ph, abort_flag, kTimeoutNs)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = stage_base + s * STAGE_BYTES;
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? smem_desc_sw128(a_addr + kk * 2048, BOX_BYTES, 1024)
                                     : smem_desc_sw128(a_addr + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(b_addr + kk * 2048, BOX_BYTES, 1024)
                                     : smem_desc_sw128(b_addr + kk * 32, 16, 1024);
            tc_mma_bf16_pair(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit_pair_multicast(smem_u32(&sm->empty[s]), 0x3);
        }
        if (!ok) break;
        tc_commit_pair_multicast(smem_u32(&sm->tmem_full[acc]), 0x3);
        ++local;
      }
      if (!ok) {
        tc_commit_pair_multicast(smem_u32(&sm->drain), 0x1);
        drain_wait(smem_u32(&sm->drain), 0);
      }
    }
  } else if (warp <= 5) {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int qw = warp & 3;   // TMEM lane quarter of this warp
    uint8_t* ebuf = ebuf_all + qw * EPI_WARP_BYTES;
    if (DW_SCHED && !no_work) {
      // an empty group's weight gradient is zero: one 512-byte row per instruction
      const int nz = sm->n_empty * dw_tiles;
      for (int z = cid; z < nz; z += ncl) {
        const PairTile ti = decode_pair_tile<EPI>(sm, pd, GMM_DW, sm->empty_ids[z / dw_tiles], z % dw_tiles, rank);
        uint16_t* obase = pd.out + static_cast<int64_t>(ti.g) * pd.out_rows * pd.ld_out;
        const int rows_valid = ti.rows_valid - qw * 32;
        const int ncols = min(BN, pd.out_cols - ti.col0);
        for (int r = 0; r < 32 && r < rows_valid; ++r)
          if (lane * 8 < ncols)
            *reinterpret_cast<uint4*>(obase + (ti.row0 + qw * 32 + r) * pd.ld_out + ti.col0 + lane * 8) =
                make_uint4(0, 0, 0, 0);
      }
    }
    uint32_t local = 0;
    ClusterTiles tiles(wk);
    TileRef tr;
    while (tiles.next(tr)) {
      const PairTile ti = decode_pair_tile<EPI>(sm, q, mode, group_of(tr), tr.local, rank);
      uint16_t* obase = (mode == GMM_DW) ? q.out + static_cast<int64_t>(ti.g) * q.out_rows * q.ld_out : q.out;
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      if (!warp_wait(smem_u32(&sm->tmem_full[acc]), aph, abort_flag, lane)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(qw * 32) << 16) + acc * BN;
      int rows_valid = ti.rows_valid - qw * 32;  // rows of this warp's 32 that are in the group
      const int64_t wrow0 = ti.row0 + qw * 32;
      {  // bounds-checking build: the warp's first and last rows lie in the output (dW: in the group's gradient)
        const int64_t rcap = mode == GMM_DW ? q.out_rows : q.rows_cap;
        if (rows_valid > 0 &&
            !(in_bounds(wrow0, rcap, q.status) && in_bounds(wrow0 + min(rows_valid, 32) - 1, rcap, q.status) &&
              (mode != GMM_DW || in_bounds(ti.g, q.E, q.status))))
          rows_valid = 0;
      }
      const uint32_t release = mapa_shared(smem_u32(&sm->tmem_empty[acc]), 0);
      auto release_tmem = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(release);
      };
      if (EPI == EPI_SWIGLU) {
        const int64_t ldh = 2 * static_cast<int64_t>(p.act_cols);
        // pass 1: the activation
#pragma unroll 1
        for (int cc = 0; cc < BN / 2; cc += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + cc, g);
          tmem_ld32(taddr + BN / 2 + cc, u);
          tmem_ld_wait();
          uint32_t a[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float gv = round_bf16(__uint_as_float(g[i]));  // H is stored in bf16
            const float uv = round_bf16(__uint_as_float(u[i]));
            a[i] = __float_as_uint(act_forward(gv, uv, p.act));
          }
          stage_chunk(ebuf, lane, cc / 8, a);
        }
        if (!p.h_save) release_tmem();
        __syncwarp();
        flush_rows(ebuf, lane, p.out + wrow0 * p.ld_out + ti.col0, p.ld_out, rows_valid, BN / 2);
        __syncwarp();
        if (p.h_save) {
          // passes 2 and 3: the bf16 pre-activation, gate then up
#pragma unroll 1
          for (int part = 0; part < 2; ++part) {
#pragma unroll 1
            for (int cc = 0; cc < BN / 2; cc += 32) {
              uint32_t r[32];
              tmem_ld32(taddr + part * (BN / 2) + cc, r);
              tmem_ld_wait();
              stage_chunk(ebuf, lane, cc / 8, r);
            }
            if (part == 1) release_tmem();
            __syncwarp();
            flush_rows(ebuf, lane, p.h_save + wrow0 * ldh + part * p.act_cols + ti.col0, ldh, rows_valid, BN / 2);
            __syncwarp();
          }
        }
      } else if (EPI == EPI_DSWIGLU) {
        // dH from dA (this accumulator, rounded to bf16 as a stored dA would be)
        // and the saved H: per 64 columns, the warp loads its 32 rows of gate and
        // up into shared memory (coalesced), each thread turns its row into dG
        // and dU in place, and the warp writes them back (coalesced).
        const int I = p.act_cols;
        const int64_t ldh = 2 * static_cast<int64_t>(I);
        uint8_t* gbuf = ebuf;                 // 32 rows x 128 bytes
        uint8_t* ubuf = ebuf + 32 * 128;
        const int lr = lane >> 3, lc = lane & 7;  // coalesced: 4 rows x 8 chunks per instruction
#pragma unroll 1
        for (int c64 = 0; c64 < BN / 64; ++c64) {
          const int col = ti.col0 + c64 * 64;
          const bool cols_ok = col < p.out_cols;   // warp-uniform
          if (cols_ok) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = 4 * i + lr;
              if (r < rows_valid) {
                const uint16_t* src = p.h_in + (wrow0 + r) * ldh + col + lc * 8;
                const int off = r * 128 + ((lc ^ (r & 7)) * 16);
                *reinterpret_cast<uint4*>(gbuf + off) = ld_nc_v4(src);
                *reinterpret_cast<uint4*>(ubuf + off) = ld_nc_v4(src + I);
              }
            }
          }
          __syncwarp();
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            uint32_t d[32];
            tmem_ld32(taddr + c64 * 64 + half * 32, d);
            tmem_ld_wait();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int off = lane * 128 + (((half * 4 + q4) ^ (lane & 7)) * 16);
              uint4 gv = *reinterpret_cast<const uint4*>(gbuf + off);
              uint4 uv = *reinterpret_cast<const uint4*>(ubuf + off);
              const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
              const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
              float dg[8], du[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float g = (e & 1) ? bf16_hi(gw[e >> 1]) : bf16_lo(gw[e >> 1]);
                const float u = (e & 1) ? bf16_hi(uw[e >> 1]) : bf16_lo(uw[e >> 1]);
                const float da = round_bf16(__uint_as_float(d[q4 * 8 + e]));
                act_grad(g, u, da, p.act, dg[e], du[e]);
              }
              gv.x = pack_bf16x2(dg[0], dg[1]); gv.y = pack_bf16x2(dg[2], dg[3]);
              gv.z = pack_bf16x2(dg[4], dg[5]); gv.w = pack_bf16x2(dg[6], dg[7]);
              uv.x = pack_bf16x2(du[0], du[1]); uv.y = pack_bf16x2(du[2], du[3]);
              uv.z = pack_bf16x2(du[4], du[5]); uv.w = pack_bf16x2(du[6], du[7]);
              *reinterpret_cast<uint4*>(gbuf + off) = gv;
              *reinterpret_cast<uint4*>(ubuf + off) = uv;
            }
          }
          if (c64 == BN / 64 - 1) release_tmem();
          __syncwarp();
          if (cols_ok) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = 4 * i + lr;
              if (r < rows_valid) {
                uint16_t* dst = obase + (wrow0 + r) * ldh + col + lc * 8;
                const int off = r * 128 + ((lc ^ (r & 7)) * 16);
                *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(gbuf + off);
                *reinterpret_cast<uint4*>(dst + I) = *reinterpret_cast<const uint4*>(ubuf + off);
              }
            }
          }
          __syncwarp();
        }
      } else {
        // dW rows come in whole warps (K is a multiple of 64); forward and dX
        // rows past the group end can fall inside a warp's 32.  Half 0 is
        // loaded from TMEM two 32-column chunks per wait; all of half 1 is
        // loaded (and the accumulator released) before waiting for the
        // staging buffer to be read by half 0's stores.
        const int64_t grow0 = (mode == GMM_DW) ? static_cast<int64_t>(ti.g) * q.out_rows + wrow0 : wrow0;
        auto store_half = [&](int half) {
          const int col = ti.col0 + half * (BN / 2);
          if (rows_valid >= 32) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              for (int b = 0; b < 2; ++b)
                if (col + 64 * b < q.out_cols)
                  tma_store_2d(mC, smem_u32(ebuf + b * BOX_STAGE), col + 64 * b, static_cast<int32_t>(grow0));
              bulk_commit();
            }
          } else if (rows_valid > 0) {
            __syncwarp();
            flush_rows_box(ebuf, lane, obase + wrow0 * q.ld_out + col, q.ld_out, rows_valid, q.out_cols - col);
          }
          __syncwarp();
        };
        if (lane == 0) bulk_wait_read();  // the previous tile's stores have read the staging buffer
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < BN / 2; cc += 64) {
          uint32_t r0[32], r1[32];
          tmem_ld32(taddr + cc, r0);
          tmem_ld32(taddr + cc + 32, r1);
          tmem_ld_wait();
          stage_box(ebuf, lane, cc, r0);
          stage_box(ebuf, lane, cc + 32, r1);
        }
        store_half(0);
        {
          uint32_t h[4][32];
#pragma unroll
          for (int i = 0; i < 4; ++i) tmem_ld32(taddr + BN / 2 + 32 * i, h[i]);
          tmem_ld_wait();
          release_tmem();
          if (lane == 0) bulk_wait_read();
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) stage_box(ebuf, lane, 32 * i, h[i]);
          store_half(1);
        }
      }
      ++local;
    }
    if (EPI == EPI_PLAIN && lane == 0) bulk_wait_all();  // every tile store has landed
    __syncwarp();
  }

  __syncthreads();
  if (*abort_flag) {
    // a timed-out pipeline may still have copies landing: give them time
    if (tid == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
    }
    __syncthreads();
  }
  cluster_sync_all();  // no arrival or copy targets either CTA past this point
  if (*abort_flag && tid == 0) set_status(p.status, MOE_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
  if (p.concurrent && tid == 0) pdl_wait();  // finish no earlier than the launch before this one
}

template <int MODE, int EPI>
moe_status_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const PairParams& p,
                         cudaStream_t s, int max_ctas, const CUtensorMap* ta2 = nullptr, const CUtensorMap* tb2 = nullptr,
                         const CUtensorMap* tc2 = nullptr, const PairParams* pw = nullptr) {
  auto kern = gmm_pair_kernel<MODE, EPI>;
  static int configured_dev = -1;
  static int grid = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (configured_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes)) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) return MOE_ERR_CUDA;
    grid = 2 * clusters;
    if (grid > kMaxGmmCtas) grid = kMaxGmmCtas;  // the descriptor slots cover this many CTAs
    configured_dev = dev;
  }
  const int g = (max_ctas >= 2 && max_ctas < grid) ? (max_ctas & ~1) : grid;
  if (launch_pdl(kern, dim3(g), dim3(NUM_THREADS), kSmemBytes, s, 2, ta, tb, tc, ta2 ? *ta2 : ta, tb2 ? *tb2 : tb,
                 tc2 ? *tc2 : tc, p, pw ? *pw : p) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// dW parameters and maps: a [M, Ka] and b [M, Nb] contracted over each group's
// rows into out [E, Ka, Nb].
bool setup_dw(PairParams& p, CUtensorMap& ta, CUtensorMap& tb, CUtensorMap& tc, const uint16_t* a, const uint16_t* b,
              int64_t M, int64_t Ka, int64_t Nb, int64_t E, uint16_t* out, void* gmm_scratch) {
  p.a_base = reinterpret_cast<const uint8_t*>(a);
  p.b_base = reinterpret_cast<const uint8_t*>(b);
  p.a_pitch = Ka * 2;
  p.b_pitch = Nb * 2;
  p.map_slots = static_cast<uint8_t*>(gmm_scratch);
  p.out = out;
  p.out_rows = static_cast<int>(Ka);
  p.out_cols = static_cast<int>(Nb);
  p.ld_out = Nb;
  p.tile_cols = static_cast<int>((Nb + BN - 1) / BN);
  return make_map_2d(&ta, a, M, Ka, 64) && make_map_2d(&tb, b, M, Nb, 64) && make_map_2d(&tc, out, E * Ka, Nb, 32);
}

}  // namespace

// FWD (optionally with the SwiGLU epilogue), DX and DW on CTA pairs.
moe_status_t launch_gmm_pair(int mode, int epilogue, const uint16_t* a, const uint16_t* b, const int64_t* group_list,
                             int64_t M, int64_t K, int64_t N, int64_t E, const Act& act, uint16_t* out, uint16_t* h_save,
                             uint32_t* status, void* gmm_scratch, cudaStream_t s, const GmmLaunch& how) {
  PairParams p{};
  p.concurrent = how.concurrent ? 1 : 0;
  p.wt = how.w_transposed ? 1 : 0;
  p.group_list = group_list;
  p.E = static_cast<int>(E);
  p.rows_cap = M;
  p.status = status;
  p.out = out;
  p.h_save = h_save;
  p.act = act;
  CUtensorMap ta, tb, tc;
  if (mode == GMM_FWD) {
    const bool sw = (epilogue == EPI_SWIGLU);
    p.out_cols = static_cast<int>(sw ? N / 2 : N);
    p.ld_out = p.out_cols;
    p.act_cols = static_cast<int>(N / 2);
    p.tile_cols = sw ? static_cast<int>((N / 2) / (BN / 2)) : static_cast<int>((N + BN - 1) / BN);
    p.kblocks = static_cast<int>(K / BK);
    if (!make_map_2d(&ta, a, M, K, BM) ||
        !(how.w_transposed ? make_map_3d(&tb, b, E, N, K, BNH) : make_map_3d(&tb, b, E, K, N, 64)))
      return MOE_ERR_CUDA;
    if (sw) return launch_pair<GMM_FWD, EPI_SWIGLU>(ta, tb, tb, p, s, how.max_ctas);
    if (!make_map_2d(&tc, out, M, N, 32)) return MOE_ERR_CUDA;
    return launch_pair<GMM_FWD, EPI_PLAIN>(ta, tb, tc, p, s, how.max_ctas);
  }
  if (mode == GMM_DX) {
    const bool dsw = (epilogue == EPI_DSWIGLU);
    p.out_cols = static_cast<int>(K);
    p.ld_out = dsw ? 2 * K : K;
    p.act_cols = static_cast<int>(K);
    p.h_in = h_save;
    p.tile_cols = static_cast<int>((K + BN - 1) / BN);
    p.kblocks = static_cast<int>(N / BK);
    if (!make_map_2d(&ta, a, M, N, BM) ||
        !(how.w_transposed ? make_map_3d(&tb, b, E, N, K, 64) : make_map_3d(&tb, b, E, K, N, BNH)))
      return MOE_ERR_CUDA;
    if (dsw) return launch_pair<GMM_DX, EPI_DSWIGLU>(ta, tb, tb, p, s, how.max_ctas);
    if (!make_map_2d(&tc, out, M, K, 32)) return MOE_ERR_CUDA;
    return launch_pair<GMM_DX, EPI_PLAIN>(ta, tb, tc, p, s, how.max_ctas);
  }
  // DW: a = x [M, K], b = dy [M, N]; output dw [E, K, N]
  if (gmm_scratch == nullptr) return MOE_ERR_INVALID;
  if (!setup_dw(p, ta, tb, tc, a, b, M, K, N, E, out, gmm_scratch)) return MOE_ERR_CUDA;
  return launch_pair<GMM_DW, EPI_PLAIN>(ta, tb, tc, p, s, how.max_ctas);
}

// dX and dW of one grouped matmul in one launch (plain dX epilogue).
//   dX: dy [M, N] x w -> dx [M, K] (w [E, K, N], or [E, N, K] when transposed);
//   dW: x [M, K], dy [M, N] -> dw [E, K, N] (transposed: dy, x -> dw [E, N, K]).
moe_status_t launch_gmm_pair_bwd(const uint16_t* x, const uint16_t* w, const int64_t* group_list, const uint16_t* dy,
                                 int64_t M, int64_t K, int64_t N, int64_t E, uint16_t* dx, uint16_t* dw,
                                 uint32_t* status, void* gmm_scratch, cudaStream_t s, bool w_transposed) {
  if (gmm_scratch == nullptr) return MOE_ERR_INVALID;
  PairParams p{}, pw{};
  p.wt = w_transposed ? 1 : 0;
  p.group_list = pw.group_list = group_list;
  p.E = pw.E = static_cast<int>(E);
  p.rows_cap = pw.rows_cap = M;
  p.status = pw.status = status;
  p.out = dx;
  p.out_cols = static_cast<int>(K);
  p.ld_out = K;
  p.act_cols = static_cast<int>(K);
  p.tile_cols = static_cast<int>((K + BN - 1) / BN);
  p.kblocks = static_cast<int>(N / BK);
  CUtensorMap ta, tb, tc, ta2, tb2, tc2;
  if (!make_map_2d(&ta, dy, M, N, BM) ||
      !(w_transposed ? make_map_3d(&tb, w, E, N, K, 64) : make_map_3d(&tb, w, E, K, N, BNH)) ||
      !make_map_2d(&tc, dx, M, K, 32))
    return MOE_ERR_CUDA;
  const bool ok = w_transposed ? setup_dw(pw, ta2, tb2, tc2, dy, x, M, N, K, E, dw, gmm_scratch)
                               : setup_dw(pw, ta2, tb2, tc2, x, dy, M, K, N, E, dw, gmm_scratch);
  if (!ok) return MOE_ERR_CUDA;
  return launch_pair<GMM_BWD, EPI_PLAIN>(ta, tb, tc, p, s, 0, &ta2, &tb2, &tc2, &pw);
}

}  // namespace moe
