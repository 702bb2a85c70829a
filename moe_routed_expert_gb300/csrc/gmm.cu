// Grouped matmul (GMM) on the 5th-generation tensor cores: a persistent,
// warp-specialised tcgen05 kernel with TMA-fed shared-memory stages and a
// double-buffered fp32 accumulator in TMEM.
//
// What it computes follows "NPU Training Operators - GMM", section "算子语义":
// rows of x are grouped by expert (group g owns rows [cumsum before g,
// cumsum through g) of group_list) and
//   forward   y_g  = x_g  @ W_g                 (GMM_FWD)
//   input grad dx_g = dy_g @ W_g^T              (GMM_DX)
// The gate_up forward can finish with the clipped SwiGLU of "MegaMoE",
// "激活函数公式" (gate = first I columns, up = last I), in the epilogue.
// This 128-row kernel serves groups that average under 512 rows; larger ones,
// and every weight gradient, run on CTA pairs (gmm_pair.cu).
//
// Design (one CTA per SM, 192 threads):
//   warp 0      TMA producer: 128B-swizzled tiles of A (128 x 64) and B
//               (64 x 256) into a 4-stage ring, one mbarrier pair per stage.
//   warp 1      TMEM allocator; one thread issues 4 x tcgen05.mma (M=128,
//               N=256, K=16) per stage into one of two 256-column fp32
//               accumulators; tcgen05.commit frees the stage and, after the
//               last stage, hands the accumulator to the epilogue.
//   warps 2..5  epilogue: tcgen05.ld (32 lanes x 32 columns) -> bf16 ->
//               row-masked global stores; then release the accumulator.
// The group structure is read on the device (no host sync): every CTA scans
// group_list into row offsets and a tile prefix in shared memory and maps a
// linear tile id to (group, row tile, column tile) by binary search.  Tiles
// are visited column-tile fastest so concurrent CTAs share A rows and W
// columns in L2.
// Every wait is bounded; on a timeout the kernel drains its own copies and
// MMAs, writes MOE_ERR_TIMEOUT to the status word and returns.
//
// The fused layer forward ("MegaMoE", 算子功能: dispatch, the two expert
// matmuls with the activation between them, and the combine as one operator)
// runs two variants of this kernel, and neither the permuted tokens nor the
// expert outputs ever make a round trip through HBM:
//   FUSE_GATHER   gate_up: A rows are copied straight from the tokens x,
//                 row r of a group being token sorted_flat[r] / k: gather
//                 warps copy 16-byte pieces of the tile's rows (cp.async,
//                 into the 128B-swizzled layout the MMA reads) and signal the
//                 stage barrier when they land; the
//                 weight tile still comes by TMA.  x stays in L2 (read k times).
//                 (A TMA gather4 per four rows was tried: the TMA unit's cost
//                 per row made a stage take twice as long.)  Two gather warps
//                 copy 64 rows each.
//   FUSE_COMBINE  down: tiles are visited column tile slowest, so the expert
//                 outputs of one 256-column slice stay in L2 while it lasts.
//                 Once the epilogue warps stored a tile, a signal warp counts
//                 it in for its slice (a release); four combine warps per
//                 CTA wait until a slice is complete and then sum their CTA's
//                 share of the tokens over it: a token's k rows in slot order
//                 j = 0, 1, ... with the routing weights (fp32, one bf16
//                 rounding: the same arithmetic as the standalone combine, so
//                 the same bits), two tokens per warp at a time, dropping the
//                 rows from L2 unwritten once read.  The combine of one slice
//                 overlaps the matmuls of the next.  (Per-token completion
//                 counts, a ring of finished tokens per epilogue warp, and the
//                 sums done in the epilogue itself were tried: each put
//                 dependent L2 round trips on every tile's critical path.)
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_BYTES = BN * BK * 2;        // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BOX_BYTES = 64 * 64 * 2;      // one 64 x 64 bf16 box = 8 KB
constexpr int TMEM_COLS = 2 * BN;           // two accumulators
constexpr int NUM_THREADS = 192;                 // producer, MMA, 4 epilogue warps
constexpr int GATHER_WARPS = 2;                  // FUSE_GATHER: warps copying A rows (64 rows each)
constexpr int COMBINE_WARPS = 4;                 // FUSE_COMBINE: warps summing tokens (plus one signal warp)
constexpr uint64_t kTimeoutNs = 4000000000ull;   // 4 s: far above any legal wait

struct GmmParams {
  const int64_t* group_list;
  int E;
  int64_t rows_cap;    // rows of the grouped operand (M)
  int out_cols;        // columns of the output (FWD: N, or I with SwiGLU; DX: K)
  int tile_cols;       // column tiles per row tile
  int kblocks;         // contraction blocks of 64 (FWD: K/64, DX: N/64)
  uint16_t* out;
  int64_t ld_out;
  uint16_t* h_save;    // SwiGLU: bf16 pre-activation [M, 2I] out
  const uint16_t* h_in;  // SwiGLU gradient: saved pre-activation [M, 2I] in
  int act_cols;        // SwiGLU: I
  Act act;             // gated activation (SwiGLU epilogues)
  uint32_t* status;
  int concurrent;      // see GmmLaunch
  int wt;              // each expert's weight stored transposed, [N, K]
  // fused layer forward
  const int32_t* sorted_flat;  // GATHER, COMBINE: permuted row -> flat slot t * k + j
  const int32_t* row_id_map;   // COMBINE, GATHER set-up: flat slot -> row (-1: unused)
  const float* topk_w;         // COMBINE: routing weights [T, k]
  int k;                       // slots per token
  int64_t T;                   // tokens
  uint16_t* y;                 // COMBINE: the combined output [T, out_cols]
  int32_t* counters;           // COMBINE: per column tile, epilogue warps that finished a tile of it
  int64_t n_counters;          // GATHER: counts to zero for the down GMM that follows
  int cols_slow;               // tiles visited column tile slowest
  int discard;                 // COMBINE: expert rows dropped from L2 once combined
  int w_evict_first;           // weight tiles loaded under an L2 evict-first policy
  const uint16_t* gx;          // GATHER: the tokens x [T, gx_ld]
  int64_t gx_ld;
};

enum GmmFuse { FUSE_NONE = 0, FUSE_GATHER = 1, FUSE_COMBINE = 2 };

template <int FUSE>
constexpr int threads_of() {
  return NUM_THREADS + 32 * (FUSE == FUSE_COMBINE ? COMBINE_WARPS + 1 : (FUSE == FUSE_GATHER ? GATHER_WARPS : 0));
}

struct __align__(16) GmmSmem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t stored[2];                 // FUSE_COMBINE: the epilogue warps stored an accumulator's tile
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
  int32_t bad;
  int32_t ntiles;
  int32_t row_tiles;                  // row tiles of all experts
  int64_t grp_off[kMaxExperts + 1];   // row offset of each expert (by id)
  int32_t grp_cnt[kMaxExperts];       // rows of each expert (by id)
  int32_t tile_start[kMaxExperts + 1];  // tile prefix over experts (row tiles only when cols_slow)
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + sizeof(GmmSmem);

struct TileInfo {
  int g;          // expert id
  int64_t row0;   // first row of x / dy
  int rows_valid; // rows of the tile inside the group
  int col0;       // first output column (SwiGLU: first activation column)
};

template <int MODE, int EPI>
__device__ __forceinline__ TileInfo decode_tile(const GmmSmem* sm, const GmmParams& p, int t) {
  // column tile fastest: t runs over (expert, row tile, column tile); slowest:
  // over (column tile, expert, row tile)
  int ct = 0;
  if (p.cols_slow) {
    ct = t / sm->row_tiles;
    t -= ct * sm->row_tiles;
  }
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (sm->tile_start[mid] <= t) lo = mid; else hi = mid;
  }
  TileInfo ti;
  const int g = lo;
  const int local = t - sm->tile_start[lo];
  int rt = local;
  if (!p.cols_slow) {
    rt = local / p.tile_cols;
    ct = local - rt * p.tile_cols;
  }
  ti.g = g;
  ti.col0 = ct * (EPI == EPI_SWIGLU ? BN / 2 : BN);
  ti.row0 = sm->grp_off[g] + static_cast<int64_t>(rt) * BM;
  ti.rows_valid = min(BM, sm->grp_cnt[g] - rt * BM);
  return ti;
}

// Lane 0 waits, the whole warp learns the outcome (keeps the warp converged
// for the .sync.aligned tcgen05 instructions that follow).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait_bounded(bar, parity, abort, kTimeoutNs) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Wait that ignores the abort flag: used only to drain in-flight work on the abort path.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  uint32_t dummy = 0;
  mbar_wait_bounded(bar, parity, &dummy, 200000000ull);
}

__device__ __forceinline__ void store_row32(uint16_t* dst, const uint32_t (&r)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint4 q;
    q.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
    q.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
    q.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
    q.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
    d[v] = q;
  }
}

__device__ __forceinline__ void store_row32_hint(uint16_t* dst, const uint32_t (&r)[32], uint64_t pol) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint4 q;
    q.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
    q.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
    q.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
    q.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
    st_v4_hint(dst + 8 * v, q, pol);
  }
}

// FUSE_COMBINE, in a combine warp: the sums of token ta over column slice cta
// and of token tb over slice ctb (tb < 0: none) into y, 8 columns per lane,
// each token's slots in order j = 0, 1, ... (fp32, one bf16 rounding); the
// two tokens' loads are in flight together.  Then the tokens' expert rows of
// those slices are dead: their 128-byte lines are dropped from L2 unwritten.
__device__ __forceinline__ void combine_tokens(const GmmParams& p, int64_t ta, int cta, int64_t tb, int ctb,
                                              int lane) {
  const int64_t ca = static_cast<int64_t>(cta) * BN + lane * 8;
  const int64_t cb = static_cast<int64_t>(ctb) * BN + lane * 8;
  const bool oka = ca < p.out_cols;
  const bool okb = tb >= 0 && cb < p.out_cols;
  float acca[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float accb[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  bool bad = false;
  for (int j0 = 0; j0 < p.k; j0 += 8) {
    int32_t ra[8], rb[8];
    float wa[8], wb[8];
    uint4 va[8], vb[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {   // every load first, then the checks
      const int j = j0 + jj;
      ra[jj] = j < p.k ? p.row_id_map[ta * p.k + j] : -1;
      rb[jj] = (tb >= 0 && j < p.k) ? p.row_id_map[tb * p.k + j] : -1;
      wa[jj] = j < p.k ? p.topk_w[ta * p.k + j] : 0.0f;
      wb[jj] = (tb >= 0 && j < p.k) ? p.topk_w[tb * p.k + j] : 0.0f;
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const bool ba = ra[jj] < -1 || ra[jj] >= p.rows_cap, bb = rb[jj] < -1 || rb[jj] >= p.rows_cap;
      bad |= ba || bb;
      if (ba) ra[jj] = -1;
      if (bb) rb[jj] = -1;
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      if (ra[jj] >= 0 && oka) va[jj] = ld_cg_v4(p.out + static_cast<int64_t>(ra[jj]) * p.ld_out + ca);
      if (rb[jj] >= 0 && okb) vb[jj] = ld_cg_v4(p.out + static_cast<int64_t>(rb[jj]) * p.ld_out + cb);
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      if (ra[jj] >= 0 && oka) add8(acca, va[jj], wa[jj]);
      if (rb[jj] >= 0 && okb) add8(accb, vb[jj], wb[jj]);
    }
  }
  if (oka) *reinterpret_cast<uint4*>(p.y + ta * p.out_cols + ca) = pack8(acca);
  if (okb) *reinterpret_cast<uint4*>(p.y + tb * p.out_cols + cb) = pack8(accb);
  if (p.discard) {
    __syncwarp();   // every lane holds its values: the lines may go
    // four 128-byte lines per row of a 256-column slice; the rows are read
    // first, then the lines dropped
    const int per = p.k * 4;
    for (int u0 = lane; u0 < 2 * per; u0 += 4 * 32) {   // k <= 16: one round
      int32_t r[4];
      int cl[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = u0 + 32 * u;
        const bool second = i >= per;
        const int64_t t = second ? tb : ta;
        const int ii = second ? i - per : i;
        r[u] = -1;
        cl[u] = (second ? ctb : cta) * BN + (ii & 3) * 64;
        if (i < 2 * per && t >= 0) r[u] = p.row_id_map[t * p.k + (ii >> 2)];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (r[u] >= 0 && r[u] < p.rows_cap && cl[u] < p.out_cols)
          discard_l2_line(p.out + static_cast<int64_t>(r[u]) * p.ld_out + cl[u]);
    }
  }
  if (bad) set_status(p.status, MOE_ERR_DEVICE);
}

template <int MODE, int EPI, int FUSE>
__global__ void __launch_bounds__(threads_of<FUSE>(), 1)
gmm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GmmParams p) {
  static_assert(MODE == GMM_FWD || MODE == GMM_DX, "dW runs on CTA pairs");
  static_assert(FUSE == FUSE_NONE || (MODE == GMM_FWD && (FUSE == FUSE_GATHER) == (EPI == EPI_SWIGLU)),
                "fused forms: the gate_up forward with the gather, the down forward with the combine");
  // B is MN-major (output columns contiguous) for the forward over [K, N]
  // weights and for dX over transposed [N, K] weights.
  const bool B_MN = (MODE == GMM_FWD) != (p.wt != 0);
  const uint32_t IDESC = idesc_bf16_f32(BM, BN, false, B_MN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GmmSmem* sm = reinterpret_cast<GmmSmem*>(smem + STAGES * STAGE_BYTES);
  const uint32_t stage_base = smem_u32(smem);

  constexpr int NT = threads_of<FUSE>();
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;

  // ---------------------------------------------------------------- set-up
  if (tid == 0) {
    sm->bad = 0;
    sm->abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      // with the gather, each lane of the gather warps also arrives once its
      // copies of the stage have landed
      mbar_init(smem_u32(&sm->full[s]), FUSE == FUSE_GATHER ? 1 + 32 * GATHER_WARPS : 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sm->tmem_full[a]), 1);
      // with the combine, the signal warp releases the accumulator once the
      // four epilogue warps have stored its tile (so they can never run two
      // tiles ahead of it on one barrier)
      mbar_init(smem_u32(&sm->tmem_empty[a]), FUSE == FUSE_COMBINE ? 1 : 4);
      mbar_init(smem_u32(&sm->stored[a]), 4);
    }
    mbar_init(smem_u32(&sm->drain), 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  __syncthreads();
  // Everything above touches only shared memory and the kernel parameters, so
  // it overlaps the tail of the previous kernel on the stream.
  if (!p.concurrent) pdl_wait();
  pdl_trigger();
  for (int e = tid; e < E; e += NT) {
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
    const int per_rt = p.cols_slow ? 1 : p.tile_cols;   // prefix entries per row tile
    for (int e = lo; e < hi; ++e) {
      rows += sm->grp_cnt[e];
      tiles += ((sm->grp_cnt[e] + BM - 1) / BM) * per_rt;
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
      sm->grp_off[e] = rb;
      sm->tile_start[e] = tb;
      rb += sm->grp_cnt[e];
      tb += ((sm->grp_cnt[e] + BM - 1) / BM) * per_rt;
    }
    if (lane == 31) {
      sm->grp_off[E] = rows_incl;
      sm->tile_start[E] = tiles_incl;
      sm->row_tiles = tiles_incl;
      sm->ntiles = p.cols_slow ? tiles_incl * p.tile_cols : tiles_incl;
      if (rows_incl > p.rows_cap) sm->bad = 1;
    }
  }
  __syncthreads();
  if (sm->bad) {
    if (tid == 0 && blockIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE);
    if (p.concurrent && tid == 0) pdl_wait();
    return;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm->tmem_base;
  const int ntiles = sm->ntiles;
  volatile uint32_t* abort_flag = &sm->abort;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (one thread)
    // With the gather it copies only the weight tile; the gather warps copy A.
    if (lane == 0) {
      const uint64_t pol = p.w_evict_first ? l2_policy_evict_first() : 0ull;
      const uint64_t pol_keep = FUSE == FUSE_COMBINE ? l2_policy_evict_last() : 0ull;
      auto load_b = [&](uint32_t dst, uint32_t bar, int32_t c0, int32_t c1, int32_t g) {
        if (p.w_evict_first) tma_load_3d_hint(dst, &tmB, bar, c0, c1, g, pol);
        else tma_load_3d(dst, &tmB, bar, c0, c1, g);
      };
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const TileInfo ti = decode_tile<MODE, EPI>(sm, p, t);
        for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait_bounded(smem_u32(&sm->empty[s]), ph ^ 1u, abort_flag, kTimeoutNs)) { ok = false; break; }
          const uint32_t bar = smem_u32(&sm->full[s]);
          const uint32_t a_dst = stage_base + s * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          if (FUSE == FUSE_GATHER) {
            mbar_expect_tx(bar, B_BYTES);
          } else {
            mbar_expect_tx(bar, STAGE_BYTES);
            if (FUSE == FUSE_COMBINE)   // the rows are read again for every column slice
              tma_load_2d_hint(a_dst, &tmA, bar, kb * BK, static_cast<int32_t>(ti.row0), pol_keep);
            else
              tma_load_2d(a_dst, &tmA, bar, kb * BK, static_cast<int32_t>(ti.row0));
          }
          // output columns [0, 128) and [128, 256) of the tile: the gate and the up half with SwiGLU
          const int c0 = ti.col0, c1 = EPI == EPI_SWIGLU ? p.act_cols + ti.col0 : ti.col0 + BN / 2;
          if (B_MN) {  // weight rows hold output columns: four 64-column boxes
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              load_b(b_dst + j * BOX_BYTES, bar, (j < 2 ? c0 : c1) + 64 * (j & 1), kb * BK, ti.g);
          } else if (MODE == GMM_FWD) {  // transposed weights: two boxes of 128 rows
            load_b(b_dst, bar, kb * BK, c0, ti.g);
            load_b(b_dst + (BN / 2) * 128, bar, kb * BK, c1, ti.g);
          } else {     // dX over [K, N] weights: one box of 256 rows
            load_b(b_dst, bar, kb * BK, ti.col0, ti.g);
          }
        }
      }
      if (!ok) {
        // let every copy already issued land before the CTA can exit
        const uint32_t first = it > STAGES ? it - STAGES : 0;
        for (uint32_t i = first; i < it; ++i) drain_wait(smem_u32(&sm->full[i % STAGES]), (i / STAGES) & 1u);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (one thread)
    if (lane == 0) {
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
        if (!mbar_wait_bounded(smem_u32(&sm->tmem_empty[acc]), aph ^ 1u, abort_flag, kTimeoutNs)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait_bounded(smem_u32(&sm->full[s]), ph, abort_flag, kTimeoutNs)) { ok = false; break; }
          tc_fence_after();
          if (FUSE == FUSE_GATHER) fence_proxy_async_smem();   // the cp.async rows, for the tensor core
          const uint32_t a_addr = stage_base + s * STAGE_BYTES;
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(a_addr + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(b_addr + kk * 2048, BOX_BYTES, 1024)
                                     : smem_desc_sw128(b_addr + kk * 32, 16, 1024);
            tc_mma_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&sm->empty[s]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm->tmem_full[acc]));
        ++local;
      }
      if (!ok) {
        tc_commit(smem_u32(&sm->drain));
        drain_wait(smem_u32(&sm->drain), 0);
      }
    }
  } else if (FUSE == FUSE_GATHER && warp >= NUM_THREADS / 32) {
    // ---------------------------------------------------------------- gather warps
    // Warp g copies rows [64 g, 64 g + 64) of each stage's A tile from x with
    // cp.async, 16 bytes at a time, into the 128B-swizzled K-major layout the
    // MMA reads: 8 lanes cover one row's 128 bytes, so lane l copies piece
    // l & 7 of rows 64 g + (l >> 3) + 4 i, i = 0 .. 15.  Rows past the group
    // end are not copied (the MMA's results for them are never stored).
    const int gw = warp - NUM_THREADS / 32;
    const int chunk = lane & 7;
    constexpr int ROWS = BM / GATHER_WARPS / 4;   // rows per lane
    const int64_t nslots = p.T * p.k;
    uint32_t it = 0;
    int ok = 1;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const TileInfo ti = decode_tile<MODE, EPI>(sm, p, t);
      // the source of each of this lane's rows (all loads first, then the checks)
      // the token rows under an L2 evict-last policy: each is read by its k slots' tiles while
      // the weights stream through L2 (prefill layer 0.360 -> 0.340 ms in isolation)
      const uint64_t xpol = l2_policy_evict_last();
      int32_t f[ROWS];
#pragma unroll
      for (int i = 0; i < ROWS; ++i) {
        const int r = gw * (BM / GATHER_WARPS) + (lane >> 3) + 4 * i;
        f[i] = r < ti.rows_valid && in_bounds(ti.row0 + r, p.rows_cap, p.status) ? p.sorted_flat[ti.row0 + r] : 0;
      }
      const uint16_t* src[ROWS];
      bool bad = false;
#pragma unroll
      for (int i = 0; i < ROWS; ++i) {
        const bool b = f[i] < 0 || f[i] >= nslots;
        bad |= b;
        src[i] = p.gx + static_cast<int64_t>(b ? 0 : f[i] / p.k) * p.gx_ld + chunk * 8;
      }
      if (bad) set_status(p.status, MOE_ERR_DEVICE);
      const int nrows = ti.rows_valid - gw * (BM / GATHER_WARPS) - (lane >> 3);   // rows i with 4 i < nrows
      for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
        if (lane == 0) ok = mbar_wait_bounded(smem_u32(&sm->empty[s]), ph ^ 1u, abort_flag, kTimeoutNs) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t a_dst = stage_base + s * STAGE_BYTES;
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
          const int r = gw * (BM / GATHER_WARPS) + (lane >> 3) + 4 * i;
          if (4 * i < nrows) cp_async16_hint(a_dst + r * 128 + ((chunk ^ (r & 7)) << 4), src[i] + kb * BK, xpol);
        }
        cp_async_arrive_noinc(smem_u32(&sm->full[s]));   // once this lane's copies of the stage land
      }
    }
    cp_async_wait_all();   // no copy of this thread lands after the CTA retires
  } else if (FUSE == FUSE_COMBINE && warp == NUM_THREADS / 32 + COMBINE_WARPS) {
    // ---------------------------------------------------------------- signal warp
    // Once the four epilogue warps have stored a tile of this CTA, frees its
    // accumulator and counts the tile into its column slice: the wait on their
    // arrival orders their stores before this thread's GPU-scope fence, which
    // orders them before the count (the epilogue warps never wait for their
    // stores to land).
    if (lane == 0) {
      uint32_t local = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++local) {
        const TileInfo ti = decode_tile<MODE, EPI>(sm, p, t);
        if (!mbar_wait_bounded(smem_u32(&sm->stored[local & 1u]), (local >> 1) & 1u, abort_flag, kTimeoutNs)) break;
        mbar_arrive(smem_u32(&sm->tmem_empty[local & 1u]));
        __threadfence();
        red_add_release_gpu(&p.counters[ti.col0 / BN], 1);
      }
    }
  } else if (FUSE == FUSE_COMBINE && warp >= NUM_THREADS / 32) {
    // ---------------------------------------------------------------- combine warps
    // Column slice by column slice (the tile order): once every tile of the
    // slice is stored (the signal warps count them in), this CTA sums its
    // share of the tokens, two per warp at a time.
    const int cw = warp - NUM_THREADS / 32;
    const int64_t tb0 = static_cast<int64_t>(blockIdx.x) * p.T / gridDim.x;
    const int64_t tb1 = static_cast<int64_t>(blockIdx.x + 1) * p.T / gridDim.x;
    const int need = sm->row_tiles;   // tiles per slice
    for (int ct = 0; ct < p.tile_cols; ++ct) {
      int ok = 1;
      if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(&p.counters[ct]) < need) {
          if (*abort_flag) { ok = 0; break; }
          if (globaltimer_ns() - t0 > kTimeoutNs) { *abort_flag = 1u; ok = 0; break; }
          __nanosleep(256);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      __threadfence();   // the slice's stored rows are visible to every lane's reads
      for (int64_t t = tb0 + 2 * cw; t < tb1; t += 2 * COMBINE_WARPS)
        combine_tokens(p, t, ct, t + 1 < tb1 ? t + 1 : -1, ct, lane);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;              // TMEM lane quarter of this warp
    const int row_in_tile = q * 32 + lane;
    if (FUSE == FUSE_GATHER) {
      // while the first tile's stages fill: zero the arrival counts of the down
      // GMM that follows (epilogue threads, spread over the grid)
      const int64_t nthr = static_cast<int64_t>(gridDim.x) * (NUM_THREADS - 64);
      const int64_t gthr = static_cast<int64_t>(blockIdx.x) * (NUM_THREADS - 64) + (tid - 64);
      for (int64_t i = gthr; i < p.n_counters; i += nthr) p.counters[i] = 0;
    }
    const uint64_t pol_keep = FUSE == FUSE_COMBINE ? l2_policy_evict_last() : 0ull;
    uint32_t local = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const TileInfo ti = decode_tile<MODE, EPI>(sm, p, t);
      const bool row_ok = row_in_tile < ti.rows_valid && in_bounds(ti.row0 + row_in_tile, p.rows_cap, p.status);
      const int64_t row = ti.row0 + row_in_tile;
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      if (!warp_wait(smem_u32(&sm->tmem_full[acc]), aph, abort_flag, lane)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (EPI == EPI_SWIGLU) {
#pragma unroll 1
        for (int cc = 0; cc < BN / 2; cc += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + cc, g);
          tmem_ld32(taddr + BN / 2 + cc, u);
          tmem_ld_wait();
          if (row_ok) {
            // H is stored in bf16; the activation is taken on those stored values
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              g[i] = __float_as_uint(round_bf16(__uint_as_float(g[i])));
              u[i] = __float_as_uint(round_bf16(__uint_as_float(u[i])));
            }
            if (p.h_save) {
              store_row32(p.h_save + row * (2 * p.act_cols) + ti.col0 + cc, g);
              store_row32(p.h_save + row * (2 * p.act_cols) + p.act_cols + ti.col0 + cc, u);
            }
            uint32_t a[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
              a[i] = __float_as_uint(act_forward(__uint_as_float(g[i]), __uint_as_float(u[i]), p.act));
            store_row32(p.out + row * p.ld_out + ti.col0 + cc, a);
          }
        }
      } else if (EPI == EPI_DSWIGLU) {
        // dH from dA (this accumulator, rounded to bf16) and the saved H, row by row
        const int I = p.act_cols;
        const int64_t ldh = 2 * static_cast<int64_t>(I);
#pragma unroll 1
        for (int cc = 0; cc < BN; cc += 32) {
          if (ti.col0 + cc >= p.out_cols) break;  // warp-uniform
          uint32_t d[32];
          tmem_ld32(taddr + cc, d);
          tmem_ld_wait();
          if (row_ok) {
            const uint16_t* hg = p.h_in + row * ldh + ti.col0 + cc;
            uint16_t* out = p.out + row * ldh + ti.col0 + cc;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 gv = ld_nc_v4(hg + 8 * v);
              const uint4 uv = ld_nc_v4(hg + I + 8 * v);
              const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
              const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
              float dg[8], du[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float g = (e & 1) ? bf16_hi(gw[e >> 1]) : bf16_lo(gw[e >> 1]);
                const float u = (e & 1) ? bf16_hi(uw[e >> 1]) : bf16_lo(uw[e >> 1]);
                const float da = round_bf16(__uint_as_float(d[8 * v + e]));
                act_grad(g, u, da, p.act, dg[e], du[e]);
              }
              uint4 og, ou;
              og.x = pack_bf16x2(dg[0], dg[1]); og.y = pack_bf16x2(dg[2], dg[3]);
              og.z = pack_bf16x2(dg[4], dg[5]); og.w = pack_bf16x2(dg[6], dg[7]);
              ou.x = pack_bf16x2(du[0], du[1]); ou.y = pack_bf16x2(du[2], du[3]);
              ou.z = pack_bf16x2(du[4], du[5]); ou.w = pack_bf16x2(du[6], du[7]);
              *reinterpret_cast<uint4*>(out + 8 * v) = og;
              *reinterpret_cast<uint4*>(out + I + 8 * v) = ou;
            }
          }
        }
      } else {
#pragma unroll 1
        for (int cc = 0; cc < BN; cc += 32) {
          if (ti.col0 + cc >= p.out_cols) break;  // warp-uniform
          uint32_t r[32];
          tmem_ld32(taddr + cc, r);
          tmem_ld_wait();
          if (row_ok) {
            uint16_t* dst = p.out + row * p.ld_out + ti.col0 + cc;
            if (FUSE == FUSE_COMBINE) store_row32_hint(dst, r, pol_keep);   // read again soon, by the combine
            else store_row32(dst, r);
          }
        }
        if (FUSE == FUSE_COMBINE) {
          // the signal warp frees the accumulator and counts the tile in once
          // all four warps stored it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm->stored[acc]));
        }
      }
      if (FUSE != FUSE_COMBINE) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm->tmem_empty[acc]));
      }
      ++local;
    }
  }

  __syncthreads();
  if (sm->abort && tid == 0) set_status(p.status, MOE_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (p.concurrent && tid == 0) pdl_wait();  // finish no earlier than the launch before this one
}

// ------------------------------------------------------------------ host side
template <int MODE, int EPI, int FUSE = FUSE_NONE>
moe_status_t launch_mode(const CUtensorMap& ta, const CUtensorMap& tb, const GmmParams& p, cudaStream_t s,
                         int max_ctas) {
  auto kern = gmm_kernel<MODE, EPI, FUSE>;
  constexpr int NT = threads_of<FUSE>();
  static int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes)) != cudaSuccess)
      return MOE_ERR_CUDA;
    configured_dev = dev;
  }
  const int grid = (max_ctas > 0 && max_ctas < num_sms()) ? max_ctas : num_sms();
  if (launch_pdl(kern, dim3(grid), dim3(NT), kSmemBytes, s, 1, ta, tb, p) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// ------------------------------------------------------------------ both expert matmuls in one launch
// The expert MLP of the inference layer ("MegaMoE", 算子功能: the dispatch and
// the two expert matmuls with the activation between them in one operator),
// on 128-row tiles:
//   phase 0  gate_up + activation: a[r] = act(x[sorted_flat[r] / k] W1[e]),
//            its rows gathered from the tokens x by two gather warps (cp.async),
//            as the FUSE_GATHER form does;
//   phase 1  down: y2[r] = a[r] W2[e], A by TMA.
// One persistent grid walks all phase-0 tiles, then all phase-1 tiles
// (column tile fastest within each); a CTA's tiles come in that order.  A
// phase-1 tile needs its row tile of a, i.e. all phase-0 tiles of that row
// tile: a signal warp counts each stored phase-0 tile into ready[row tile]
// (GPU-scope fence, then a release add), and the producer, before the first
// A copy of a phase-1 tile, waits (bounded) until the count is complete, then
// fences the generic and async proxies.  Phase-0 tiles never wait, and every
// CTA of the grid is resident (one per SM), so the waits end.  The weight
// tiles of the first stage are issued before that wait.  The signal warp also
// frees each accumulator once the four epilogue warps stored its tile.
constexpr int LAYER_THREADS = NUM_THREADS + 32 * GATHER_WARPS + 32;   // + gather warps + signal warp
#ifndef MOE_W1_PREFETCH_MB
#define MOE_W1_PREFETCH_MB 24
#endif
constexpr int kW1PrefetchMB = MOE_W1_PREFETCH_MB;

struct LayerParams {
  const int64_t* group_list;
  int E;
  int64_t rows_cap;            // R = T * k
  uint32_t* status;
  const uint16_t* x;           // tokens [T, H]
  int64_t H;
  int64_t T;
  int k;
  const int32_t* sorted_flat;  // [R]: permuted row -> flat slot
  int I;                       // activation columns
  int kb1, kb2;                // contraction blocks of 64: H / 64, I / 64
  int tc1, tc2;                // column tiles: I / 128 (activation), ceil(H / 256)
  uint16_t* a;                 // [R, I]
  uint16_t* y2;                // [R, H]
  int32_t* ready;              // [row tiles]: phase-0 tiles stored (zero at launch)
  Act act;
  int w_evict_first;
  const uint8_t* w1;           // gate_up weights, for the L2 prefetch before the wait
  int64_t w1_prefetch;         // bytes of w1 to prefetch (a multiple of 16 per CTA share)
};

struct LTile {
  int phase;
  int g;
  int rtg;          // row tile over all experts
  int64_t row0;
  int rows_valid;
  int col0;         // phase 0: first activation column; phase 1: first output column
};

__device__ __forceinline__ LTile decode_layer_tile(const GmmSmem* sm, const LayerParams& p, int n1, int t) {
  LTile ti;
  ti.phase = t < n1 ? 0 : 1;
  const int u = ti.phase ? t - n1 : t;
  const int tc = ti.phase ? p.tc2 : p.tc1;
  ti.rtg = u / tc;
  const int ct = u - ti.rtg * tc;
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sm->tile_start[mid] <= ti.rtg) lo = mid; else hi = mid;
  }
  const int rt = ti.rtg - sm->tile_start[lo];
  ti.g = lo;
  ti.row0 = sm->grp_off[lo] + static_cast<int64_t>(rt) * BM;
  ti.rows_valid = min(BM, sm->grp_cnt[lo] - rt * BM);
  ti.col0 = ti.phase ? ct * BN : ct * (BN / 2);
  return ti;
}

__global__ void __launch_bounds__(LAYER_THREADS, 1)
expert_mlp_kernel(const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmA2,
                  const __grid_constant__ CUtensorMap tmB2, const LayerParams p) {
  const uint32_t IDESC = idesc_bf16_f32(BM, BN, false, true);   // both weights [K, N]: MN-major B
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GmmSmem* sm = reinterpret_cast<GmmSmem*>(smem + STAGES * STAGE_BYTES);
  const uint32_t stage_base = smem_u32(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;
  constexpr int GATHER_W0 = NUM_THREADS / 32;            // first gather warp
  constexpr int SIGNAL_W = GATHER_W0 + GATHER_WARPS;     // the signal warp

  if (tid == 0) {
    sm->bad = 0;
    sm->abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1 + 32 * GATHER_WARPS);   // producer + every gather lane
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sm->tmem_full[a]), 1);
      mbar_init(smem_u32(&sm->tmem_empty[a]), 1);   // the signal warp
      mbar_init(smem_u32(&sm->stored[a]), 4);       // the epilogue warps
    }
    mbar_init(smem_u32(&sm->drain), 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmB1);
    tma_prefetch_desc(&tmA2);
    tma_prefetch_desc(&tmB2);
  }
  if (warp == 2 && p.w1_prefetch > 0) {
    // While the index pass that writes group_list still runs, pull the first
    // experts' gate_up weights into L2: the first wave of phase-0 tiles starts
    // with the lowest experts.  CTA b takes the b-th share of the first
    // w1_prefetch bytes, 16 KB a lane and copy.
    const int64_t share = (p.w1_prefetch / gridDim.x) & ~int64_t(15);
    const uint8_t* base = p.w1 + share * blockIdx.x;
    for (int64_t off = static_cast<int64_t>(lane) * 16384; off < share; off += 32 * 16384)
      prefetch_l2_bulk(base + off, static_cast<uint32_t>(share - off < 16384 ? share - off : 16384));
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  for (int e = tid; e < E; e += LAYER_THREADS) {
    const int64_t c = p.group_list[e];
    if (c < 0 || c > p.rows_cap) atomicOr(&sm->bad, 1);
    sm->grp_cnt[e] = static_cast<int32_t>(c < 0 ? 0 : (c > p.rows_cap ? p.rows_cap : c));
  }
  __syncthreads();
  if (warp == 0) {   // row offsets and the row-tile prefix over the experts
    const int per = (E + 31) / 32;
    const int lo = min(E, lane * per), hi = min(E, lo + per);
    int64_t rows = 0;
    int32_t tiles = 0;
    for (int e = lo; e < hi; ++e) {
      rows += sm->grp_cnt[e];
      tiles += (sm->grp_cnt[e] + BM - 1) / BM;
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
      sm->grp_off[e] = rb;
      sm->tile_start[e] = tb;
      rb += sm->grp_cnt[e];
      tb += (sm->grp_cnt[e] + BM - 1) / BM;
    }
    if (lane == 31) {
      sm->grp_off[E] = rows_incl;
      sm->tile_start[E] = tiles_incl;
      sm->row_tiles = tiles_incl;
      sm->ntiles = tiles_incl * (p.tc1 + p.tc2);
      if (rows_incl > p.rows_cap) sm->bad = 1;
    }
  }
  __syncthreads();
  if (sm->bad) {
    if (tid == 0 && blockIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE);
    return;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm->tmem_base;
  const int ntiles = sm->ntiles;
  const int n1 = sm->row_tiles * p.tc1;   // phase-0 tiles
  volatile uint32_t* abort_flag = &sm->abort;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer (one thread)
    if (lane == 0) {
      const uint64_t pol = p.w_evict_first ? l2_policy_evict_first() : 0ull;
      auto load_b = [&](const CUtensorMap* m, uint32_t dst, uint32_t bar, int32_t c0, int32_t c1, int32_t g) {
        if (p.w_evict_first) tma_load_3d_hint(dst, m, bar, c0, c1, g, pol);
        else tma_load_3d(dst, m, bar, c0, c1, g);
      };
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const LTile ti = decode_layer_tile(sm, p, n1, t);
        const int kbs = ti.phase ? p.kb2 : p.kb1;
        for (int kb = 0; kb < kbs; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait_bounded(smem_u32(&sm->empty[s]), ph ^ 1u, abort_flag, kTimeoutNs)) { ok = false; break; }
          const uint32_t bar = smem_u32(&sm->full[s]);
          const uint32_t a_dst = stage_base + s * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          if (ti.phase == 0) {
            mbar_expect_tx(bar, B_BYTES);   // A comes from the gather warps
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)   // gate columns [col0, col0 + 128), then the matching up columns
              load_b(&tmB1, b_dst + j * BOX_BYTES, bar, (j < 2 ? ti.col0 : p.I + ti.col0) + 64 * (j & 1), kb * BK,
                     ti.g);
          } else {
            mbar_arrive_n(bar, 32 * GATHER_WARPS);   // the gather warps' share of the stage's arrivals
            mbar_expect_tx(bar, STAGE_BYTES);
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) load_b(&tmB2, b_dst + j * BOX_BYTES, bar, ti.col0 + 64 * j, kb * BK, ti.g);
            if (kb == 0) {
              // the row tile of a must be complete: wait for its phase-0 tiles
              const uint64_t t0 = globaltimer_ns();
              while (ld_acquire_gpu(&p.ready[ti.rtg]) < p.tc1) {
                if (*abort_flag) { ok = false; break; }
                if (globaltimer_ns() - t0 > kTimeoutNs) { *abort_flag = 1u; ok = false; break; }
                __nanosleep(128);
              }
              if (!ok) {   // the stage's weight copies are in flight: the drain below waits for them
                ++it;
                break;
              }
              fence_proxy_async_global();   // the stored rows, for the TMA unit
            }
            tma_load_2d(a_dst, &tmA2, bar, kb * BK, static_cast<int32_t>(ti.row0));
          }
        }
      }
      if (!ok) {   // let every copy already issued land before the CTA can exit
        const uint32_t first = it > STAGES ? it - STAGES : 0;
        for (uint32_t i = first; i < it; ++i) drain_wait(smem_u32(&sm->full[i % STAGES]), (i / STAGES) & 1u);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (one thread)
    if (lane == 0) {
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const int kbs = t < n1 ? p.kb1 : p.kb2;
        const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
        if (!mbar_wait_bounded(smem_u32(&sm->tmem_empty[acc]), aph ^ 1u, abort_flag, kTimeoutNs)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < kbs; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait_bounded(smem_u32(&sm->full[s]), ph, abort_flag, kTimeoutNs)) { ok = false; break; }
          tc_fence_after();
          fence_proxy_async_smem();   // gathered rows came through the generic proxy
          const uint32_t a_addr = stage_base + s * STAGE_BYTES;
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(a_addr + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b_addr + kk * 2048, BOX_BYTES, 1024);
            tc_mma_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&sm->empty[s]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm->tmem_full[acc]));
        ++local;
      }
      if (!ok) {
        tc_commit(smem_u32(&sm->drain));
        drain_wait(smem_u32(&sm->drain), 0);
      }
    }
  } else if (warp >= GATHER_W0 && warp < SIGNAL_W) {
    // ---------------------------------------------------------------- gather warps (phase-0 tiles)
    // As in the FUSE_GATHER form: warp g copies rows [64 g, 64 g + 64) of A.
    const int gw = warp - GATHER_W0;
    const int chunk = lane & 7;
    constexpr int ROWS = BM / GATHER_WARPS / 4;
    const int64_t nslots = p.T * p.k;
    uint32_t it = 0;
    int ok = 1;
    for (int t = blockIdx.x; t < n1 && ok; t += gridDim.x) {   // a CTA's phase-0 tiles come first
      const LTile ti = decode_layer_tile(sm, p, n1, t);
      // the token rows under an L2 evict-last policy: each is read by its k slots' tiles while
      // the weights stream through L2 (prefill layer 0.360 -> 0.340 ms in isolation)
      const uint64_t xpol = l2_policy_evict_last();
      int32_t f[ROWS];
#pragma unroll
      for (int i = 0; i < ROWS; ++i) {
        const int r = gw * (BM / GATHER_WARPS) + (lane >> 3) + 4 * i;
        f[i] = r < ti.rows_valid && in_bounds(ti.row0 + r, p.rows_cap, p.status) ? p.sorted_flat[ti.row0 + r] : 0;
      }
      const uint16_t* src[ROWS];
      bool bad = false;
#pragma unroll
      for (int i = 0; i < ROWS; ++i) {
        const bool b = f[i] < 0 || f[i] >= nslots;
        bad |= b;
        src[i] = p.x + static_cast<int64_t>(b ? 0 : f[i] / p.k) * p.H + chunk * 8;
      }
      if (bad) set_status(p.status, MOE_ERR_DEVICE);
      const int nrows = ti.rows_valid - gw * (BM / GATHER_WARPS) - (lane >> 3);
      for (int kb = 0; kb < p.kb1; ++kb, ++it) {
        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
        if (lane == 0) ok = mbar_wait_bounded(smem_u32(&sm->empty[s]), ph ^ 1u, abort_flag, kTimeoutNs) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t a_dst = stage_base + s * STAGE_BYTES;
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
          const int r = gw * (BM / GATHER_WARPS) + (lane >> 3) + 4 * i;
          if (4 * i < nrows) cp_async16_hint(a_dst + r * 128 + ((chunk ^ (r & 7)) << 4), src[i] + kb * BK, xpol);
        }
        cp_async_arrive_noinc(smem_u32(&sm->full[s]));
      }
    }
    cp_async_wait_all();
  } else if (warp == SIGNAL_W) {
    // ---------------------------------------------------------------- signal warp
    // Frees each accumulator once its tile is stored, and counts the stored
    // phase-0 tiles into ready[] (fence, then a release add), so a phase-1
    // tile on any CTA can read the rows.
    if (lane == 0) {
      uint32_t local = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++local) {
        if (!mbar_wait_bounded(smem_u32(&sm->stored[local & 1u]), (local >> 1) & 1u, abort_flag, kTimeoutNs)) break;
        mbar_arrive(smem_u32(&sm->tmem_empty[local & 1u]));
        if (t < n1) {
          const LTile ti = decode_layer_tile(sm, p, n1, t);
          __threadfence();
          red_add_release_gpu(&p.ready[ti.rtg], 1);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    uint32_t local = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++local) {
      const LTile ti = decode_layer_tile(sm, p, n1, t);
      const bool row_ok = row_in_tile < ti.rows_valid && in_bounds(ti.row0 + row_in_tile, p.rows_cap, p.status);
      const int64_t row = ti.row0 + row_in_tile;
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      if (!warp_wait(smem_u32(&sm->tmem_full[acc]), aph, abort_flag, lane)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (ti.phase == 0) {
#pragma unroll 1
        for (int cc = 0; cc < BN / 2; cc += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + cc, g);
          tmem_ld32(taddr + BN / 2 + cc, u);
          tmem_ld_wait();
          if (row_ok) {
            uint32_t a[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)   // H is bf16; the activation is taken on those values
              a[i] = __float_as_uint(act_forward(round_bf16(__uint_as_float(g[i])), round_bf16(__uint_as_float(u[i])),
                                                 p.act));
            store_row32(p.a + row * p.I + ti.col0 + cc, a);
          }
        }
      } else {
#pragma unroll 1
        for (int cc = 0; cc < BN; cc += 32) {
          if (ti.col0 + cc >= p.H) break;   // warp-uniform
          uint32_t r[32];
          tmem_ld32(taddr + cc, r);
          tmem_ld_wait();
          if (row_ok) store_row32(p.y2 + row * p.H + ti.col0 + cc, r);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->stored[acc]));
    }
  }

  __syncthreads();
  if (sm->abort && tid == 0) set_status(p.status, MOE_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

moe_status_t launch_gmm(int mode, int epilogue, const uint16_t* a, const uint16_t* b, const int64_t* group_list,
                        int64_t M, int64_t K, int64_t N, int64_t E, const Act& act,
                        uint16_t* out, uint16_t* h_save, uint32_t* status, void* gmm_scratch, cudaStream_t s,
                        const GmmLaunch& how) {
  // a: FWD x [M,K]; DX dy [M,N]; DW x [M,K].   b: FWD/DX w [E,K,N]; DW dy [M,N].
  // CTA pairs (256 x 256 tiles) for every weight gradient, and for forward and
  // dX when groups average at least 512 rows; below that the extra padding of
  // a 256-row tile costs more than the pair saves, and the 128-row kernel here
  // runs instead.
  if (mode == GMM_DW || M >= kPairMinRowsPerGroup * E)
    return launch_gmm_pair(mode, epilogue, a, b, group_list, M, K, N, E, act, out, h_save, status, gmm_scratch, s,
                           how);
  GmmParams p{};
  p.group_list = group_list;
  p.E = static_cast<int>(E);
  p.rows_cap = M;
  p.status = status;
  p.out = out;
  p.h_save = h_save;
  p.act = act;
  p.concurrent = how.concurrent ? 1 : 0;
  p.wt = how.w_transposed ? 1 : 0;
  CUtensorMap ta, tb;
  if (mode == GMM_FWD) {
    const bool sw = (epilogue == EPI_SWIGLU);
    p.out_cols = static_cast<int>(sw ? N / 2 : N);
    p.ld_out = p.out_cols;
    p.act_cols = static_cast<int>(N / 2);
    p.tile_cols = sw ? static_cast<int>((N / 2) / (BN / 2)) : static_cast<int>((N + BN - 1) / BN);
    p.kblocks = static_cast<int>(K / BK);
    if (!make_map_2d(&ta, a, M, K, BM) ||
        !(how.w_transposed ? make_map_3d(&tb, b, E, N, K, BN / 2) : make_map_3d(&tb, b, E, K, N, 64)))
      return MOE_ERR_CUDA;
    return sw ? launch_mode<GMM_FWD, EPI_SWIGLU>(ta, tb, p, s, how.max_ctas)
              : launch_mode<GMM_FWD, EPI_PLAIN>(ta, tb, p, s, how.max_ctas);
  }
  const bool dsw = (epilogue == EPI_DSWIGLU);
  p.out_cols = static_cast<int>(K);
  p.ld_out = dsw ? 2 * K : K;
  p.act_cols = static_cast<int>(K);
  p.h_in = h_save;
  p.tile_cols = static_cast<int>((K + BN - 1) / BN);
  p.kblocks = static_cast<int>(N / BK);
  if (!make_map_2d(&ta, a, M, N, BM) ||
      !(how.w_transposed ? make_map_3d(&tb, b, E, N, K, 64) : make_map_3d(&tb, b, E, K, N, BN)))
    return MOE_ERR_CUDA;
  return dsw ? launch_mode<GMM_DX, EPI_DSWIGLU>(ta, tb, p, s, how.max_ctas)
             : launch_mode<GMM_DX, EPI_PLAIN>(ta, tb, p, s, how.max_ctas);
}

size_t fused_counter_bytes(int64_t N) { return align256(static_cast<size_t>((N + BN - 1) / BN) * sizeof(int32_t)); }

// Fused dispatch + gate_up: rows of A gathered from x [T, K] (row r of the
// permuted order is token sorted_flat[r] / k), w [E, K, N], the gated
// activation of the [gate | up] product into out [M, N/2].  With counters,
// the kernel also zeroes n_counters arrival counts for a down GMM that follows.
moe_status_t launch_gmm_gather_act(const uint16_t* x, const int32_t* sorted_flat, int64_t T, int64_t k,
                                   const uint16_t* w, const int64_t* group_list, int64_t M, int64_t K, int64_t N,
                                   int64_t E, const Act& act, bool w_transposed, uint16_t* out, int32_t* counters,
                                   int64_t n_counters, uint32_t* status, cudaStream_t s, const FusedOptions& opt) {
  GmmParams p{};
  p.group_list = group_list;
  p.E = static_cast<int>(E);
  p.rows_cap = M;
  p.status = status;
  p.act = act;
  p.sorted_flat = sorted_flat;
  p.k = static_cast<int>(k);
  p.T = T;
  p.counters = counters;
  p.n_counters = counters ? n_counters : 0;
  p.gx = x;
  p.gx_ld = K;
  p.w_evict_first = (opt.evict_first && M < 64 * E) ? 1 : 0;   // as in launch_expert_mlp
  p.wt = w_transposed ? 1 : 0;
  p.out = out;
  p.out_cols = static_cast<int>(N / 2);
  p.ld_out = N / 2;
  p.act_cols = static_cast<int>(N / 2);
  p.tile_cols = static_cast<int>((N / 2) / (BN / 2));
  p.kblocks = static_cast<int>(K / BK);
  CUtensorMap ta, tb;
  if (!make_map_2d(&ta, x, T, K, 1) ||
      !(w_transposed ? make_map_3d(&tb, w, E, N, K, BN / 2) : make_map_3d(&tb, w, E, K, N, 64)))
    return MOE_ERR_CUDA;
  return launch_mode<GMM_FWD, EPI_SWIGLU, FUSE_GATHER>(ta, tb, p, s, 0);
}

size_t expert_mlp_ready_bytes(int64_t R, int64_t E) {
  return align256(static_cast<size_t>((R + BM - 1) / BM + E) * sizeof(int32_t));
}

// Both expert matmuls in one launch (see expert_mlp_kernel): x [T, H] tokens,
// rows gathered through sorted_flat; a [R, I] and y2 [R, H] out.  ready:
// expert_mlp_ready_bytes(R, E) of scratch, zero at launch.
moe_status_t launch_expert_mlp(const uint16_t* x, const int32_t* sorted_flat, const uint16_t* w1, const uint16_t* w2,
                               const int64_t* group_list, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                               const Act& act, uint16_t* a, uint16_t* y2, int32_t* ready, uint32_t* status,
                               cudaStream_t s) {
  LayerParams p{};
  p.group_list = group_list;
  p.E = static_cast<int>(E);
  p.rows_cap = T * k;
  p.status = status;
  p.x = x;
  p.H = H;
  p.T = T;
  p.k = static_cast<int>(k);
  p.sorted_flat = sorted_flat;
  p.I = static_cast<int>(I);
  p.kb1 = static_cast<int>(H / BK);
  p.kb2 = static_cast<int>(I / BK);
  p.tc1 = static_cast<int>(I / (BN / 2));
  p.tc2 = static_cast<int>((H + BN - 1) / BN);
  p.a = a;
  p.y2 = y2;
  p.ready = ready;
  p.act = act;
  // weights streamed under an L2 evict-first policy only when experts average
  // under 64 rows: a weight tile is then read by one row tile; with more rows
  // an expert's second row tile reads it again from L2 (measured at about 128
  // rows per expert: 0.383 ms with the policy against 0.356 without; at a few
  // rows per expert 0.212 against 0.216)
  p.w_evict_first = (T * k < 64 * E) ? 1 : 0;
  // the L2 prefetch before the wait: about what HBM delivers during the index
  // pass (decode 8 us, prefill 14 us), at most all of w1
  p.w1 = reinterpret_cast<const uint8_t*>(w1);
  const int64_t w1_bytes = E * H * 2 * I * 2;
  p.w1_prefetch = (static_cast<int64_t>(kW1PrefetchMB) << 20) < w1_bytes ? (static_cast<int64_t>(kW1PrefetchMB) << 20)
                                                                           : w1_bytes;
  CUtensorMap tb1, ta2, tb2;
  if (!make_map_3d(&tb1, w1, E, H, 2 * I, 64) || !make_map_2d(&ta2, a, T * k, I, BM) ||
      !make_map_3d(&tb2, w2, E, I, H, 64))
    return MOE_ERR_CUDA;
  static int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    if (cudaFuncSetAttribute(expert_mlp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess)
      return MOE_ERR_CUDA;
    configured_dev = dev;
  }
  if (launch_pdl(expert_mlp_kernel, dim3(num_sms()), dim3(LAYER_THREADS), kSmemBytes, s, 1, tb1, ta2, tb2, p) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// Fused down + combine: a [M, K] @ w [E, K, N] into the scratch y2 [M, N],
// each token's k rows summed with the routing weights into y [T, N] once the
// column slice holding them is stored.  counters: fused_counter_bytes(N),
// zero on entry.
moe_status_t launch_gmm_combine(const uint16_t* a, const uint16_t* w, const int64_t* group_list,
                                const int32_t* row_id_map, const int32_t* sorted_flat, const float* topk_w, int64_t T,
                                int64_t k, int64_t M, int64_t K, int64_t N, int64_t E, bool w_transposed,
                                uint16_t* y2, int32_t* counters, uint16_t* y, uint32_t* status, cudaStream_t s,
                                const FusedOptions& opt) {
  GmmParams p{};
  p.group_list = group_list;
  p.E = static_cast<int>(E);
  p.rows_cap = M;
  p.status = status;
  p.sorted_flat = sorted_flat;
  p.row_id_map = row_id_map;
  p.topk_w = topk_w;
  p.k = static_cast<int>(k);
  p.T = T;
  p.counters = counters;
  p.w_evict_first = (opt.evict_first && M < 64 * E) ? 1 : 0;   // as in launch_expert_mlp
  p.wt = w_transposed ? 1 : 0;
  p.out = y2;
  p.out_cols = static_cast<int>(N);
  p.ld_out = N;
  p.tile_cols = static_cast<int>((N + BN - 1) / BN);
  p.kblocks = static_cast<int>(K / BK);
  p.y = y;
  p.cols_slow = 1;
  p.discard = opt.discard ? 1 : 0;
  CUtensorMap ta, tb;
  if (!make_map_2d(&ta, a, M, K, BM) ||
      !(w_transposed ? make_map_3d(&tb, w, E, N, K, BN / 2) : make_map_3d(&tb, w, E, K, N, 64)))
    return MOE_ERR_CUDA;
  return launch_mode<GMM_FWD, EPI_PLAIN, FUSE_COMBINE>(ta, tb, p, s, 0);
}

}  // namespace moe

namespace moe {

// dX then dW.  When dX is small (at most about four waves of 256 x 256 tiles
// on the whole GPU, counting one partial row tile per group) and its groups
// are large enough for CTA pairs, one launch does both (launch_gmm_pair_bwd).
// Other small problems run them side by side: dX on half the SMs, and dW,
// launched right behind it with programmatic serialisation, starts at once on
// the other half (it reads only inputs that exist before dX starts) and
// finishes no earlier than dX.  That hides the last partial wave and the
// prologue and epilogue of one launch.
moe_status_t launch_gmm_backward(const uint16_t* x, const uint16_t* w, const int64_t* group_list, const uint16_t* dy,
                                 int64_t M, int64_t K, int64_t N, int64_t E, int dx_epilogue, const Act& act,
                                 const uint16_t* h, uint16_t* dx, uint16_t* dw, uint32_t* status, void* gmm_scratch,
                                 cudaStream_t s, bool w_transposed) {
  GmmLaunch first, second;
  first.w_transposed = w_transposed;
  const int half = (num_sms() / 2) & ~1;
  const bool small = dx && dw && half >= 2 && (M / 256 + E) * ((K + 255) / 256) <= 4 * static_cast<int64_t>(half);
  // Small problems on CTA pairs: one launch whose clusters each take dX or dW
  // tiles, balanced on the device from the group sizes.
  if (small && dx_epilogue == EPI_PLAIN && M >= kPairMinRowsPerGroup * E)
    return launch_gmm_pair_bwd(x, w, group_list, dy, M, K, N, E, dx, dw, status, gmm_scratch, s, w_transposed);
  if (small) {
    first.max_ctas = half;
    second.max_ctas = num_sms() - half;
    second.concurrent = true;
  }
  moe_status_t st = MOE_OK;
  if (dx && (st = launch_gmm(GMM_DX, dx_epilogue, dy, w, group_list, M, K, N, E, act, dx,
                             const_cast<uint16_t*>(h), status, gmm_scratch, s, first)) != MOE_OK)
    return st;
  // dW in the weights' layout: [E, K, N] = x^T dy, or transposed [E, N, K] = dy^T x
  if (dw && (st = w_transposed ? launch_gmm(GMM_DW, EPI_PLAIN, dy, x, group_list, M, N, K, E, Act(), dw, nullptr,
                                            status, gmm_scratch, s, second)
                               : launch_gmm(GMM_DW, EPI_PLAIN, x, dy, group_list, M, K, N, E, Act(), dw, nullptr,
                                            status, gmm_scratch, s, second)) != MOE_OK)
    return st;
  return MOE_OK;
}

}  // namespace moe
