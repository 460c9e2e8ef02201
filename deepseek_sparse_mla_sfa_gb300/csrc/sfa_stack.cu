// sfa_stack.cu -- tcgen05 / TMA path of sparse MLA decode for 33-64 heads on sm_103a:
// one CTA per work unit (or per range of tiles), the two column halves of QK^T stacked
// in the M dimension.
//
// The computation is the one of "RFC: MsModeling 支持 Decode Context Parallel 仿真"
// 2.1.4.1-2.1.4.4 and "vllm-ascend PR #18870 解读" 4.3 / 4.5: for every query token,
// softmax(scale * q K^T) V over the latent rows its top-k list selects, with the
// per-head log-sum-exp, optionally restricted to one sequence shard (DCP).
//
// Why one CTA suffices at 64 heads.  The output O^T[v, heads] (512 output columns as
// four 128-lane blocks, the heads as columns) takes 4 x 64 = 256 TMEM columns.  q's
// latent part would take another 256 if its 64 heads sat in 128 lanes the usual way
// (one head per lane, 512 values = 256 bf16 pairs), leaving nothing for the scores.
// Here the latent columns are split in two halves and the halves are stacked in M:
//   * TMEM lane 32w + 16c + j holds head 16w + j with latent columns [256c, 256c + 256)
//     (w = 0..3, c = 0, 1, j = 0..15): 128 TMEM columns for all of q's latent part, and
//     each lane quadrant (the lanes one warp can read) holds 16 heads in both halves;
//   * each latent step of QK^T is one M=128, N=64 MMA whose B operand is the tile's 32
//     rows in column block j followed by the same rows in block j+4 (the gathered
//     blocks are laid out in that order, so the 64 operand rows are contiguous);
//   * a lane of half c reads its half's partial scores in columns 32c..32c+31 of the
//     128 x 64 result (the other 32 columns pair the head with the other half of a row
//     and are never read).  The rope columns (64) add into columns 0-31 with four M=128,
//     N=32 MMAs whose A operand is q's rope part in shared memory, in the rows of the
//     first-half lanes;
//   * the two lanes of a head (16 apart in one warp) each finish 16 of the tile's 32 rows:
//     one warp shuffle brings the other half's partials of those rows, another the
//     other lane's maximum, so both keep the same online softmax of the head;
//   * P.V is formed transposed, O^T[v, heads] += V^T[v, rows] P^T[rows, heads]: V^T is
//     read straight from the gathered tile (MN-major), P^T from a shared-memory tile
//     the softmax writes (K-major).
// TMEM: q latent (128 columns), two score buffers (2 x 64), O^T (256).  With q out of
// shared memory, five 36 KB stages of whole rows fit, enough to keep a gather stream
// in flight without a second CTA.
//
// Schedules.  A CTA processes a sequence of pieces, each a range of tiles of one unit
// (token, shard); every role walks the same pieces, with tile-counted barrier phases
// that run on across them, so the gather ring never drains between pieces.
//   * one unit per CTA: when units fill at most the GPU.  When they fill less than half
//     of it, a cluster of G = 2 or 4 CTAs shares each unit (CTA c takes tiles c, c + G,
//     ...) and the CTAs merge (O, m, l) over distributed shared memory at the end;
//   * balanced ranges (with the caller's workspace, when units outnumber the SMs): one
//     CTA per SM, each taking an equal range of the units' tiles in order (at most two
//     units are cut, and each cut unit is split between two neighbouring CTAs).  A cut
//     unit's two pieces each leave their unnormalised (O, m, l) in the workspace and
//     count themselves in; the second to finish merges the two into the output.  No CTA
//     ever waits for another.
//
// Warp roles (320 threads): warps 0-3 softmax, O rescale and output (warp w owns TMEM
// lane quadrant w: heads 16w..16w+15 in both column halves for the scores, output
// columns 128m + 32w + lane of block m for O^T); warps 4-7 resolve each piece's index
// list and issue the gathers (TMA tile::gather4, four rows per instruction); warp 8
// issues QK^T; warp 9 issues P.V.  Every wait is bounded; a wait that gives up records
// SFA_ERR_DEVICE_TIMEOUT and the kernel unwinds without trapping.
#include <atomic>
#include <cuda.h>
#include <string.h>

#include "sfa_internal.h"
#include "sfa_ptx.cuh"
#include "sfa_resolve.cuh"

namespace sfa {
namespace {

using namespace ptx;

constexpr int kNt = 32;              // selected rows per tile
constexpr int kStages = 5;           // gather pipeline depth
constexpr int kThreads = 320;
constexpr int kWarps = kThreads / 32;
constexpr int kProducerWarp = 4;     // warps 4..7 resolve the lists and issue the gathers
constexpr int kProducerWarps = 4;
constexpr int kQkWarp = 8;
constexpr int kPvWarp = 9;
constexpr int kNH = 64;              // padded heads: N of P.V, columns of O^T per block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P entries stay below 2^8

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kBlk = kNt * 128;                   // one 64-column SW128 block of a tile (4 KB)
constexpr int kColBlocks = 9;                     // 8 latent blocks + the rope block
constexpr int kStageBytes = kColBlocks * kBlk;    // 36 KB: whole rows
// Offset of column block j in a stage: latent blocks j and j+4 side by side (so block j's
// rows followed by block j+4's rows form one 64-row operand), the rope block last.
__host__ __device__ constexpr int blk_off(int j) {
  return j == 8 ? 8 * kBlk : (j < 4 ? 2 * j * kBlk : (2 * (j - 4) + 1) * kBlk);
}
// q's rope part as the 128-row A operand of the rope steps, SW128: for the piece of parity
// p, head 16w + j sits in row 32w + 16p + j, and the operand starts at row 16p (so its
// row 32w + j is that head; its other rows feed unread lanes: for p = 1 the last 16 rows
// run 2 KB into the lists)
constexpr int kOffQRope = kStages * kStageBytes;
constexpr int kQRopeBytes = 128 * 128;
constexpr int kOffList = kOffQRope + kQRopeBytes; // two resolved lists (pieces of either parity)
constexpr int kListCap = 64 * kNt;                // resolved rows kept at once (whole tiles)
constexpr int kOffP = kOffList + 2 * kListCap * 4;
constexpr int kPBytes = kNH * 64;                 // P^T [64 heads x 32 rows] bf16, K-major SW64 rows
constexpr int kOffMisc = kOffP + 2 * kPBytes;
// misc: per-head (m, l) [64] float2 (+0), rescale factors [64] (+512), output scales [64]
// (+768), flags (+1024: [1] abort, [2] merge), the warps' stop and rescale flags [2 tile
// parities][4 warps] (+1088, +1120), the pieces' valid entries [2 parities] (+1152), the
// TMEM address (+1160), per-warp counts (+1168)
constexpr int kMiscBytes = 1168 + 4 * kWarps;
constexpr int kOffBar = (kOffMisc + kMiscBytes + 7) / 8 * 8;
constexpr int kBarKvFull = 0, kBarKvEmpty = kBarKvFull + kStages, kBarSFull = kBarKvEmpty + kStages,
              kBarSFree = kBarSFull + 2, kBarPReady = kBarSFree + 2, kBarPFree = kBarPReady + 2,
              kBarListReady = kBarPFree + 2, kBarListFree = kBarListReady + 2, kBarQLoad = kBarListFree + 2,
              kBarQRopeFree = kBarQLoad + 2, kBarQReady = kBarQRopeFree + 2, kBarPvFinal = kBarQReady + 1,
              kBarODrained = kBarPvFinal + 1, kBarMmaFin = kBarODrained + 1, kBarMmaFin2 = kBarMmaFin + 1,
              kBarNever = kBarMmaFin2 + 1, kBarMerge = kBarNever + 1, kNumBars = kBarMerge + 1;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffQRope % 1024 == 0 && kOffP % 1024 == 0 && kBlk % 1024 == 0, "SW128 / SW64 operands: alignment");
static_assert(2 * kListCap * 4 >= 16 * 128, "the rope operand's last rows stay inside shared memory");
static_assert(kListCap % kNt == 0, "list segments hold whole tiles");

constexpr long long kDrainLimit = 1LL << 40;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColS = 128, kColO = 256;   // q latent (128), S x 2 (128), O^T (4 x 64)

struct StackParams {
  DecodeParams p;
  int num_rows;          // num_blocks * block_size (an out-of-range row used for padding)
  int balanced;          // 1: balanced tile ranges (G == 1), 0: one unit per CTA / cluster
  int unit_tiles;        // tiles a unit can have: ceil(top_k / 32)
  long long span;        // balanced: units * unit_tiles
  float* ws_part;        // balanced: unnormalised O of cut pieces [2 * grid][64 heads][512]
  float2* ws_ml;         // balanced: their (m, l) per head [2 * grid][64]
  int* ws_count;         // balanced: pieces of each unit finished [units] (zero on entry)
};

// One piece of a CTA's work: tiles k0, k0 + stride, ... (below k1) of unit `unit`.
struct Piece {
  int unit, k0, k1, stride;
  int slot;   // balanced, cut unit: this piece's workspace slot (-1: the whole unit)
};

// Number of pieces of this CTA and the kp-th of them.
__device__ __forceinline__ int piece_count(const StackParams& sp) {
  if (!sp.balanced) return 1;
  const long long P = gridDim.x, c = blockIdx.x;
  const long long b = c * sp.span / P, e = (c + 1) * sp.span / P;
  return e > b ? (int)((e - 1) / sp.unit_tiles - b / sp.unit_tiles + 1) : 0;
}
__device__ __forceinline__ Piece piece_at(const StackParams& sp, int kp, uint32_t crank, int G) {
  Piece pc;
  if (!sp.balanced) {
    pc.unit = blockIdx.x / G;
    pc.k0 = (int)crank;
    pc.k1 = 0x7fffffff;
    pc.stride = G;
    pc.slot = -1;
    return pc;
  }
  const long long P = gridDim.x, c = blockIdx.x, T = sp.unit_tiles;
  const long long b = c * sp.span / P, e = (c + 1) * sp.span / P;
  const long long u = b / T + kp;
  pc.unit = (int)u;
  pc.k0 = (int)((b > u * T ? b : u * T) - u * T);
  pc.k1 = (int)((e < (u + 1) * T ? e : (u + 1) * T) - u * T);
  pc.stride = 1;
  // a cut unit has two pieces: its head (k0 == 0) ends this CTA's range, its tail
  // (k1 == T) starts it
  pc.slot = (pc.k0 == 0 && pc.k1 == T) ? -1 : (pc.k0 == 0 ? (int)(2 * c + 1) : (int)(2 * c));
  return pc;
}
// tiles of a piece, given the unit's valid entries
__device__ __forceinline__ int piece_tiles(const Piece& pc, int total) {
  const int n = (total + kNt - 1) / kNt;
  const int hi = n < pc.k1 ? n : pc.k1;
  return hi > pc.k0 ? (hi - pc.k0 + pc.stride - 1) / pc.stride : 0;
}
// the selection of one unit: token t, shard r
struct UnitSel {
  int t, r, bt_row;
  ShardSel sel;
  const int32_t* idx;
};
__device__ __forceinline__ UnitSel unit_sel(const DecodeParams& p, int unit) {
  UnitSel us;
  const int T = p.B * p.Q;
  // units go out last shard first (the heaviest shards of a sparse selection start first)
  us.t = unit % T;
  us.r = p.n_splits - 1 - unit / T;
  const int b = us.t / p.Q, qi = us.t % p.Q;
  const int seq_len = p.seq_lens[b];
  const int L = seq_len - (p.Q - 1 - qi);
  us.sel = shard_sel(seq_len, L, us.r, p.n_splits, p.interleave);
  us.bt_row = p.bt_per_token ? us.t : b;
  us.idx = p.topk_idx + (size_t)us.t * p.top_k;
  return us;
}

// Resolves the selection of one unit into lst: its entries that resolve to a cache row,
// in list order, as rows (the first kListCap of them); returns how many there are.  The
// four producer warps call it together (warp pw); invalid block-table entries are
// reported when `report` is set.  Each warp brings its own `ok_in`; all_ok is their
// conjunction, the same in every producer warp, so that they leave their loop together.
template <bool kInterleaved>
__device__ int resolve_unit(const DecodeParams& p, const UnitSel& us, int* lst, int* wcount, int pw, int lane,
                            bool report, bool ok_in, bool& all_ok) {
  constexpr int kRounds = 16;   // entries a lane keeps between the two passes
  const int chunk = ((p.top_k + kProducerWarps * 32 - 1) / (kProducerWarps * 32)) * 32;
  const int c_begin = min(pw * chunk, p.top_k), c_end = min(c_begin + chunk, p.top_k);
  const bool one_round = chunk <= kRounds * 32;
  int row_r[kRounds];
  int cnt = 0;
  if (one_round) {
    int pos[kRounds], blkv[kRounds];
#pragma unroll
    for (int k = 0; k < kRounds; ++k) {
      const int j = c_begin + 32 * k + lane;
      pos[k] = j < c_end ? __ldg(us.idx + j) : -1;
    }
#pragma unroll
    for (int k = 0; k < kRounds; ++k) {
      const bool in = us.sel.has_fixed<kInterleaved>(pos[k]);
      const int blk = in ? pos[k] / p.block_size : 0;
      blkv[k] = in && blk < p.max_blocks ? __ldg(p.block_table + (size_t)us.bt_row * p.max_blocks + blk) : -2;
      if (!in) blkv[k] = -3;
    }
#pragma unroll
    for (int k = 0; k < kRounds; ++k) {
      row_r[k] = -1;
      if (blkv[k] == -3) continue;
      if (blkv[k] < 0 || blkv[k] >= p.num_blocks) {
        if (report) report_status(p.status, kStatusBadBlock);
      } else {
        ++cnt;
        row_r[k] = blkv[k] * p.block_size + pos[k] % p.block_size;
      }
    }
  } else {
    for (int j0 = c_begin; j0 < c_end; j0 += 32) {
      const int j = j0 + lane;
      cnt += (j < c_end && resolve_row<kInterleaved>(p, us.bt_row, __ldg(us.idx + j), us.sel, report) >= 0) ? 1 : 0;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if (lane == 0) {
    wcount[pw] = cnt;
    wcount[kProducerWarps + pw] = ok_in ? 1 : 0;
  }
  named_barrier(6, kProducerWarps * 32);   // every producer warp's count is published
  all_ok = wcount[kProducerWarps] && wcount[kProducerWarps + 1] && wcount[kProducerWarps + 2] &&
           wcount[kProducerWarps + 3];
  int total = 0, off = 0;
#pragma unroll
  for (int w = 0; w < kProducerWarps; ++w) {
    const int c = wcount[w];
    if (w < pw) off += c;
    total += c;
  }
  if (one_round) {
#pragma unroll
    for (int k = 0; k < kRounds; ++k) {
      const unsigned mask = __ballot_sync(0xffffffffu, row_r[k] >= 0);
      const int o = off + __popc(mask & lanemask_lt());
      if (row_r[k] >= 0 && o < kListCap) lst[o] = row_r[k];
      off += __popc(mask);
    }
  } else {
    for (int j0 = c_begin; j0 < c_end && off < kListCap; j0 += 32) {
      const int j = j0 + lane;
      const int row = j < c_end ? resolve_row<kInterleaved>(p, us.bt_row, __ldg(us.idx + j), us.sel, false) : -1;
      const unsigned mask = __ballot_sync(0xffffffffu, row >= 0);
      const int o = off + __popc(mask & lanemask_lt());
      if (row >= 0 && o < kListCap) lst[o] = row;
      off += __popc(mask);
    }
  }
  named_barrier(6, kProducerWarps * 32);   // the list is complete (and the counts may be reused)
  return total;
}

// kInterleaved: shard layout.
template <bool kInterleaved>
__global__ void __launch_bounds__(kThreads, 1)
    decode_stack_kernel(const __grid_constant__ CUtensorMap tmap_rows, const __grid_constant__ CUtensorMap tmap_qrope,
                        const __grid_constant__ CUtensorMap tmap_out, const StackParams sp) {
  const DecodeParams& p = sp.p;
  extern __shared__ char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  int* list_s = reinterpret_cast<int*>(smem + kOffList);
  float2* ml_s = reinterpret_cast<float2*>(smem + kOffMisc);                   // [64] (m, l)
  float* alpha_s = reinterpret_cast<float*>(smem + kOffMisc + 512);           // [64]
  float* scale_s = reinterpret_cast<float*>(smem + kOffMisc + 768);           // [64]
  volatile int* flags_s = reinterpret_cast<volatile int*>(smem + kOffMisc + 1024);
  volatile int* stop_s = reinterpret_cast<volatile int*>(smem + kOffMisc + 1088);   // [2][4]
  volatile int* mv_s = reinterpret_cast<volatile int*>(smem + kOffMisc + 1120);     // [2][4]
  volatile int* totals_s = reinterpret_cast<volatile int*>(smem + kOffMisc + 1152); // [2]
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + kOffMisc + 1160);
  int* wcount_s = reinterpret_cast<int*>(smem + kOffMisc + 1168);             // [kWarps]
  volatile int* abort_s = flags_s + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  uint32_t G;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(G));
  const int T = p.B * p.Q;
  const int n_pieces = piece_count(sp);
  const long long wl = p.wait_limit;

  // ---- set-up ----------------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[kBarKvFull + s], kProducerWarps);
      mbar_init(&bars[kBarKvEmpty + s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars[kBarSFull + x], 1);       // QK^T of the tile in this score buffer done
      mbar_init(&bars[kBarSFree + x], 4);       // the four softmax warps read this score buffer
      mbar_init(&bars[kBarPReady + x], 4);      // P in this buffer and O rescaled (one arrival per warp 0-3)
      mbar_init(&bars[kBarPFree + x], 1);       // P.V has read this buffer's P (and updated O)
      mbar_init(&bars[kBarListReady + x], kProducerWarps);   // a piece's list and valid count are ready
      mbar_init(&bars[kBarListFree + x], 6);    // QK^T, P.V and the four softmax warps read the count
      mbar_init(&bars[kBarQLoad + x], 1);       // a piece's q rope rows landed
      mbar_init(&bars[kBarQRopeFree + x], 1);   // QK^T is done with a piece's q rope rows
    }
    mbar_init(&bars[kBarQReady], 4);            // a piece's q latent part is in TMEM (warps 0-3)
    mbar_init(&bars[kBarPvFinal], 1);           // a piece's last P.V has completed
    mbar_init(&bars[kBarODrained], 4);          // warps 0-3 have read a piece's O from TMEM
    mbar_init(&bars[kBarMmaFin], 1);
    mbar_init(&bars[kBarMmaFin2], 1);
    mbar_init(&bars[kBarNever], 1);             // nothing arrives: the stall test hook waits on it
    mbar_init(&bars[kBarMerge], 1);             // the other piece of a cut unit has landed (bulk copies)
    for (int k = 0; k < 8; ++k) flags_s[k] = 0;
    fence_barrier_init();
    if (n_pieces > 0) {
      // the first piece's q rope rows (parity 0), while every warp resolves its list
      mbar_arrive_expect_tx(&bars[kBarQLoad], 4u * 16u * 128u);
      const int t0 = piece_at(sp, 0, crank, (int)G).unit % T;
      for (int w = 0; w < 4; ++w)
        tma_load_3d(smem_u32(smem + kOffQRope + 32 * w * 128), &tmap_qrope, 512, 16 * w, t0, &bars[kBarQLoad]);
    }
  }
  if (warp == 0) {
    tmem_alloc(tmem_base_s, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmap_rows);
    prefetch_tmap(&tmap_qrope);
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&tmap_out);
  // ---- the first piece's list: every warp resolves a chunk (the later pieces' lists are
  // the producer warps' work) ------------------------------------------------------------
  // (its selection is kept: computing it again would load seq_lens on the critical path)
  const UnitSel us_first = unit_sel(p, piece_at(sp, 0, crank, (int)G).unit);
  if (n_pieces > 0) {
    const UnitSel& us = us_first;
    const int chunk = ((p.top_k + kWarps * 32 - 1) / (kWarps * 32)) * 32;
    const int c_begin = min(warp * chunk, p.top_k), c_end = min(c_begin + chunk, p.top_k);
    const bool one_round = chunk <= 8 * 32;
    int row_r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) row_r[k] = -1;
    int cnt = resolve_chunk<kInterleaved>(p, us.idx, c_begin, c_end, lane, us.sel, us.bt_row, crank == 0, row_r);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0) wcount_s[warp] = cnt;
    __syncthreads();
    int total = 0, off = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = wcount_s[w];
      if (w < warp) off += c;
      total += c;
    }
    if (one_round) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const unsigned mask = __ballot_sync(0xffffffffu, row_r[k] >= 0);
        const int o = off + __popc(mask & lanemask_lt());
        if (row_r[k] >= 0 && o < kListCap) list_s[o] = row_r[k];
        off += __popc(mask);
      }
    } else {
      for (int j0 = c_begin; j0 < c_end && off < kListCap; j0 += 32) {
        const int j = j0 + lane;
        const int row = j < c_end ? resolve_row<kInterleaved>(p, us.bt_row, __ldg(us.idx + j), us.sel, false) : -1;
        const unsigned mask = __ballot_sync(0xffffffffu, row >= 0);
        const int o = off + __popc(mask & lanemask_lt());
        if (row >= 0 && o < kListCap) list_s[o] = row;
        off += __popc(mask);
      }
    }
    if (threadIdx.x == 0) totals_s[0] = total;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;

  auto fail = [&](void) {
    report_status(p.status, kStatusTimeout);
    *abort_s = 1;
  };
  auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, wl));
  };

  // warps 0-3: lane 16c + j of warp w serves head 16w + j and latent column half c; it
  // keeps the head's running max (log2 units; the same in the head's two lanes) and its
  // share of the running sum (the two lanes' shares are added at the end of a piece)
  float m_ref = -INFINITY, l_part = 0.f;
  int last_cnt = 0;   // tiles of the last piece (one-unit schedule: the only one)
  const int half = (lane >> 4) & 1;
  const int head = 16 * (warp & 3) + (lane & 15);
  if (warp < 4) {
    // =================== softmax, O rescale and the pieces' output (warps 0-3) =======
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const float c_scale = p.scale * kLog2e;
    // |scale| in log2 units, at least 1e-30: masked scores are -inf, and -inf times a zero
    // scale would be NaN.  For a zero scale every valid weight still rounds to exactly 1
    // (|scores * 1e-30| is far below one ulp of 1), the uniform average the definition gives.
    const float c_abs = fmaxf(fabsf(c_scale), 1e-30f);
    const int row0 = 16 * half;         // this lane finishes tile rows row0 .. row0 + 15
    // q's latent columns [256 half, 256 half + 256) of head `head` of token t into this lane
    // as bf16 pairs (the A operand of the latent steps; heads past h are zeros), then QReady
    auto load_q = [&](int t) {
      const bool have = head < p.h;
      const uint4* qsrc =
          reinterpret_cast<const uint4*>(p.q + ((size_t)t * p.h + (have ? head : 0)) * kDQK + 256 * half);
#pragma unroll 1
      for (int c64 = 0; c64 < 2; ++c64) {   // 64 TMEM columns (128 latent values) per round
        uint4 x[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) x[k] = have ? __ldg(qsrc + 16 * c64 + k) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t v[16];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[4 * k] = x[4 * u + k].x; v[4 * k + 1] = x[4 * u + k].y;
            v[4 * k + 2] = x[4 * u + k].z; v[4 * k + 3] = x[4 * u + k].w;
          }
          tmem_st16(lane_base + kColQ + 64 * c64 + 16 * u, v);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarQReady]);
    };
    // Each warp waits for its tile itself.  A wait that gives up marks the warp bad; the
    // warps publish that at barrier B, and all four leave together after barrier B of the
    // same tile.
    bool bad = false, stopped = false;
    int n = 0;         // tiles processed so far (all pieces): the phases of the tile barriers
    int q_for = -1;    // the piece whose q is in TMEM
    for (int kp = 0; kp < n_pieces && !stopped; ++kp) {
      const Piece pc = piece_at(sp, kp, crank, (int)G);
      const UnitSel us = kp == 0 ? us_first : unit_sel(p, pc.unit);
      const int par = kp & 1;
      // (the first piece's list is complete since the start of the kernel)
      if (kp > 0 && !bad && !wait_warp(&bars[kBarListReady + par], (kp >> 1) & 1)) { fail(); bad = true; }
      const int total = totals_s[par];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarListFree + par]);
      const int cnt = piece_tiles(pc, total);
      last_cnt = cnt;
      if (q_for != kp) {
        load_q(us.t);
        q_for = kp;
      }
      m_ref = -INFINITY;
      l_part = 0.f;
      for (int i = 0; i < cnt; ++i, ++n) {
        const int bb = n & 1;
        if (!bad && !wait_warp(&bars[kBarSFull + bb], (n >> 1) & 1)) { fail(); bad = true; }
        // P buffer bb is free once P.V of tile n-2 has read it
        if (!bad && n >= 2 && !wait_warp(&bars[kBarPFree + bb], ((n >> 1) - 1) & 1)) { fail(); bad = true; }
        tc_fence_after();
        // The tile's 64 score columns of this quadrant: a first-half lane's partials are in
        // columns 0-31 (rows 0-31), a second-half lane's in columns 32-63.  Each lane keeps
        // its half's partials of its own 16 rows and passes those of the other 16 rows to the
        // head's other lane.
        float s[16];
        {
          uint32_t c0[16], c1[16], c2[16], c3[16];
          const uint32_t sb = lane_base + kColS + 64 * bb;
          tmem_ld16(sb, c0);
          tmem_ld16(sb + 16, c1);
          tmem_ld16(sb + 32, c2);
          tmem_ld16(sb + 48, c3);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kBarSFree + bb]);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float own = __uint_as_float(half ? c3[j] : c0[j]);
            const float other = __shfl_xor_sync(0xffffffffu, __uint_as_float(half ? c2[j] : c1[j]), 16);
            s[j] = own + other;
          }
        }
        // The piece's last scores are read, so every QK^T of the piece has completed: the
        // next piece's q goes to TMEM now and its first QK^T need not wait for this piece's
        // softmax and output.
        if (i == cnt - 1 && kp + 1 < n_pieces) {
          load_q(piece_at(sp, kp + 1, crank, (int)G).unit % T);   // (the token: no load)
          q_for = kp + 1;
        }
        const int g = pc.k0 + i * pc.stride;   // the unit's tile index
        const int nvalid = min(kNt, total - kNt * g);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float x = s[j];
          if (c_scale < 0.f) x = -x;   // keep max(s) * |c| == max(s * c) for a negative scale
          s[j] = (row0 + j >= nvalid || head >= p.h) ? -INFINITY : x;
        }
        float mx = s[0];
#pragma unroll
        for (int j = 1; j < 16; ++j) mx = fmaxf(mx, s[j]);
        // the tile max of the head: fmaxf is exact and symmetric, both lanes see the same
        const float mt = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16)) * c_abs;
        float m_new = m_ref;
        if (head < p.h && (i == 0 || mt > m_ref + kRescaleThreshold)) m_new = fmaxf(mt, m_ref);
        const float alpha = (i == 0 || head >= p.h) ? 1.f : ex2(m_ref - m_new);
        const bool moved = __any_sync(0xffffffffu, i > 0 && m_new != m_ref);
        m_ref = m_new;
        uint32_t pk[8];
        float sm = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float e0 = head < p.h ? ex2(fmaf(s[2 * j], c_abs, -m_new)) : 0.f;
          const float e1 = head < p.h ? ex2(fmaf(s[2 * j + 1], c_abs, -m_new)) : 0.f;
          sm += e0 + e1;
          pk[j] = pack_bf16(e0, e1);
        }
        l_part = l_part * alpha + sm;
        {
          // this head's row of P^T (64 bytes, K-major SW64), tile rows row0..row0+15 = 16-byte
          // chunks 2 half and 2 half + 1, whose positions the swizzle permutes by the row
          char* p_row = smem + kOffP + bb * kPBytes + head * 64;
#pragma unroll
          for (int u = 0; u < 2; ++u)
            *reinterpret_cast<uint4*>(p_row + (((2 * half + u) ^ ((head >> 1) & 3)) << 4)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          fence_proxy_async_smem();
        }
        if (lane == 0) {
          stop_s[4 * bb + warp] = bad ? 1 : 0;
          mv_s[4 * bb + warp] = moved ? 1 : 0;
        }
        named_barrier(2, 128);   // B: whether any warp gave up, and whether any head's max moved
        if (stop_s[4 * bb] | stop_s[4 * bb + 1] | stop_s[4 * bb + 2] | stop_s[4 * bb + 3]) {
          stopped = true;
          break;
        }
        if (mv_s[4 * bb] | mv_s[4 * bb + 1] | mv_s[4 * bb + 2] | mv_s[4 * bb + 3]) {
          // Rare: some head's reference max moved by more than the threshold.  Every warp
          // rescales its output-column lanes of O for all heads, once P.V of the previous
          // tile has completed.  (Tile n+1 waits on the same phase of that buffer again: it
          // cannot have moved on, P.V of tile n+1 is not issued yet.)
          if (lane < 16) alpha_s[head] = alpha;
          if (!bad && !wait_warp(&bars[kBarPFree + (bb ^ 1)], ((n - 1) >> 1) & 1)) { fail(); bad = true; }
          named_barrier(3, 128);   // C: the factors are published
          if (!bad) {
            tc_fence_after();
            // O^T lane v holds output column v of every head: scale column hh by alpha[hh]
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
#pragma unroll
              for (int c16 = 0; c16 < kNH / 16; ++c16) {
                uint32_t o[16];
                tmem_ld16(lane_base + kColO + kNH * m + 16 * c16, o);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha_s[16 * c16 + k]);
                tmem_st16(lane_base + kColO + kNH * m + 16 * c16, o);
              }
            }
            tmem_st_wait();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarPReady + bb]);
      }
      if (stopped || !sp.balanced) break;
      // ---- the piece's output (balanced schedule) -----------------------------------
      bool have = false;
      if (!bad) {
        // P.V arrives on PvFinal once per piece (an empty piece too)
        if (wait_warp(&bars[kBarPvFinal], kp & 1)) have = cnt > 0;
        else { fail(); bad = true; }
      }
      tc_fence_after();
      const float l_sum = l_part + __shfl_xor_sync(0xffffffffu, l_part, 16);
      const float m_h = (have && head < p.h) ? m_ref : -INFINITY;
      const float l_h = (have && head < p.h) ? l_sum : 0.f;
      const int v = warp * 32 + lane;   // output column v of each 128-column block
      const size_t out_row = ((size_t)us.r * T + us.t) * p.h;   // the unit's first (token, head) row
      if (pc.slot < 0) {
        // the whole unit: normalise and write the output and lse
        if (lane < 16) {
          scale_s[head] = l_h > 0.f ? 1.f / l_h : 0.f;
          if (head < p.h && !*abort_s) p.lse[out_row + head] = l_h > 0.f ? (m_h + __log2f(l_h)) * kLn2 : -INFINITY;
        }
        named_barrier(2, 128);
        // the heads' output scales in registers: read from shared memory between the global
        // stores below, each would wait for the stores before it
        float sc[kNH];
#pragma unroll
        for (int hh = 0; hh < kNH; ++hh) sc[hh] = scale_s[hh];
        named_barrier(2, 128);   // the scales are read before the next piece can change them
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
          uint32_t o[kNH];
          if (have) {
#pragma unroll
            for (int c16 = 0; c16 < kNH / 16; ++c16)
              tmem_ld16(lane_base + kColO + kNH * m + 16 * c16, *reinterpret_cast<uint32_t(*)[16]>(&o[16 * c16]));
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int k = 0; k < kNH; ++k) o[k] = 0u;
          }
          if (!*abort_s) {
#pragma unroll
            for (int hh = 0; hh < kNH; ++hh)
              if (hh < p.h) p.out[(out_row + hh) * kDV + 128 * m + v] = __uint_as_float(o[hh]) * sc[hh];
          }
        }
      } else {
        // ---- a cut unit -----------------------------------------------------------
        // Its head piece (tiles from 0) is the last piece of CTA c, in slot 2c + 1; its
        // tail piece (tiles up to the end) is the first piece of CTA c + 1, in slot
        // 2(c + 1).  The unit's counter takes the tail once, when its partial result is in
        // the workspace, and the head once on arrival and once more if the head has to leave
        // its own partial there.  Exactly one of the two merges:
        //   tail, then head arrives:           the head reads 1 and merges;
        //   head arrives, tail, head again:    the head reads 0, then 2, and merges;
        //   head arrives, head again, tail:    the tail reads 2 and merges.
        const bool is_head = pc.k0 == 0;
        const int other = is_head ? pc.slot + 1 : pc.slot - 1;
        float* part = sp.ws_part + (size_t)pc.slot * kNH * kDV;
        const float* opart = sp.ws_part + (size_t)other * kNH * kDV;
        auto write_partial = [&]() {
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
            uint32_t o[kNH];
            if (have) {
#pragma unroll
              for (int c16 = 0; c16 < kNH / 16; ++c16)
                tmem_ld16(lane_base + kColO + kNH * m + 16 * c16, *reinterpret_cast<uint32_t(*)[16]>(&o[16 * c16]));
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int k = 0; k < kNH; ++k) o[k] = 0u;
            }
#pragma unroll
            for (int hh = 0; hh < kNH; ++hh)
              if (hh < p.h) part[hh * kDV + 128 * m + v] = __uint_as_float(o[hh]);
          }
          if (lane < 16) sp.ws_ml[pc.slot * kNH + head] = make_float2(m_h, l_h);
        };
        // the merged lse, and the two pieces' weights in alpha_s (this piece) and scale_s
        auto merge_weights = [&]() {
          if (lane < 16) {
            const float2 ot = __ldcg(&sp.ws_ml[other * kNH + head]);
            const float M = fmaxf(m_h, ot.x);
            const float wa = m_h == -INFINITY ? 0.f : ex2(m_h - M);
            const float wo = ot.x == -INFINITY ? 0.f : ex2(ot.x - M);
            const float L = l_h * wa + ot.y * wo;
            alpha_s[head] = L > 0.f ? wa / L : 0.f;
            scale_s[head] = L > 0.f ? wo / L : 0.f;
            if (head < p.h && !*abort_s) p.lse[out_row + head] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
          }
          named_barrier(2, 128);
        };
        if (is_head) {
          if (threadIdx.x == 0) {
            flags_s[2] = atomicAdd(&sp.ws_count[pc.unit], 1);
            __threadfence();
          }
          named_barrier(2, 128);
          bool merge = flags_s[2] == 1;
          if (!merge) {
            write_partial();
            __threadfence();
            named_barrier(2, 128);   // every warp's share of the partial result is written
            if (threadIdx.x == 0) {
              flags_s[2] = atomicAdd(&sp.ws_count[pc.unit], 1);
              __threadfence();
            }
            named_barrier(2, 128);
            merge = flags_s[2] == 2;
          }
          if (merge) {
            // This CTA has no further piece, so its stages are idle: the tail's rows come in
            // by bulk copies, and this piece's O is still in TMEM.
            if (threadIdx.x == 0) {
              // The tail's partial was written by another CTA's generic-proxy stores and is
              // now visible to this thread (the counter's fences); the bulk copies read it
              // through the async proxy, which a proxy fence orders after that.
              asm volatile("fence.proxy.async.global;" ::: "memory");
              const uint32_t bytes = (uint32_t)p.h * kDV * 4;
              mbar_arrive_expect_tx(&bars[kBarMerge], bytes);
              for (uint32_t o = 0; o < bytes; o += 32768u)
                bulk_load_g2s(smem_u32(smem) + o, reinterpret_cast<const char*>(opart) + o,
                              bytes - o < 32768u ? bytes - o : 32768u, &bars[kBarMerge]);
            }
            merge_weights();
            if (!wait_warp(&bars[kBarMerge], 0)) fail();   // a CTA merges at most once, from its last piece
            const float* tail_s = reinterpret_cast<const float*>(smem);
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
              uint32_t o[kNH];
              if (have) {
#pragma unroll
                for (int c16 = 0; c16 < kNH / 16; ++c16)
                  tmem_ld16(lane_base + kColO + kNH * m + 16 * c16, *reinterpret_cast<uint32_t(*)[16]>(&o[16 * c16]));
                tmem_ld_wait();
              } else {
#pragma unroll
                for (int k = 0; k < kNH; ++k) o[k] = 0u;
              }
#pragma unroll
              for (int c16 = 0; c16 < kNH / 16; ++c16) {
                // each chunk's operands are read before its stores
                float wa[16], wo[16], tv[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                  wa[k] = alpha_s[16 * c16 + k];
                  wo[k] = scale_s[16 * c16 + k];
                  tv[k] = tail_s[(16 * c16 + k) * kDV + 128 * m + v];
                }
                if (!*abort_s) {
#pragma unroll
                  for (int k = 0; k < 16; ++k)
                    if (16 * c16 + k < p.h)
                      p.out[(out_row + 16 * c16 + k) * kDV + 128 * m + v] =
                          __uint_as_float(o[16 * c16 + k]) * wa[k] + tv[k] * wo[k];
                }
              }
            }
            if (threadIdx.x == 0) sp.ws_count[pc.unit] = 0;   // back to zero for the next call
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kBarODrained]);
        } else {
          write_partial();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kBarODrained]);   // this piece's O has been read
          __threadfence();
          named_barrier(2, 128);   // every warp's share of the partial result is written
          if (threadIdx.x == 0) {
            flags_s[2] = atomicAdd(&sp.ws_count[pc.unit], 1);
            __threadfence();
          }
          named_barrier(2, 128);
          if (flags_s[2] == 2) {
            // rare: the head piece finished first; both partials come from the workspace
            merge_weights();
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
#pragma unroll 1
              for (int c16 = 0; c16 < kNH / 16; ++c16) {
                float wa[16], wo[16], va[16], vo[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                  const size_t e = (size_t)(16 * c16 + k) * kDV + 128 * m + v;
                  wa[k] = alpha_s[16 * c16 + k];
                  wo[k] = scale_s[16 * c16 + k];
                  va[k] = 16 * c16 + k < p.h ? __ldcg(part + e) : 0.f;
                  vo[k] = 16 * c16 + k < p.h ? __ldcg(opart + e) : 0.f;
                }
                if (!*abort_s) {
#pragma unroll
                  for (int k = 0; k < 16; ++k)
                    if (16 * c16 + k < p.h)
                      p.out[(out_row + 16 * c16 + k) * kDV + 128 * m + v] = va[k] * wa[k] + vo[k] * wo[k];
                }
              }
            }
            if (threadIdx.x == 0) sp.ws_count[pc.unit] = 0;   // back to zero for the next call
          }
        }
        // the merge weights are read before the next piece can change them
        named_barrier(2, 128);
        continue;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarODrained]);   // this piece's O has been read
    }
  } else if (warp < kProducerWarp + kProducerWarps) {
    // =================== index resolution and gathers (warps 4-7) ======================
    // Producer warp pw resolves its share of each piece's list, then issues the gathers of
    // row groups g = pw, pw + 4 of each tile (4 rows each, all nine 64-column blocks): 18
    // per tile, one per lane.
    const int pw = warp - kProducerWarp;
    int n = 0;   // tiles gathered so far (all pieces)
    bool ok = true;
    int rope_loads[2] = {1, 0};   // q rope loads issued per parity (the first at set-up)
    // The four producer warps meet at named barriers in every resolution, so they leave
    // this loop together: at the resolution of the first piece after any of them (or any
    // other role) gave up.
    for (int kp = 0; kp < n_pieces; ++kp) {
      const Piece pc = piece_at(sp, kp, crank, (int)G);
      const UnitSel us = kp == 0 ? us_first : unit_sel(p, pc.unit);
      const int par = kp & 1;
      int* lst = list_s + par * kListCap;
      bool wok = ok && !*abort_s;
      // the other roles have read the valid count of piece kp-2 (the same parity)
      if (wok && kp >= 2 && !(wok = wait_warp(&bars[kBarListFree + par], ((kp >> 1) - 1) & 1))) ok = false;
      bool go = true;
      const int total = kp == 0 ? totals_s[0]
                                : resolve_unit<kInterleaved>(p, us, lst, wcount_s, pw, lane, crank == 0, wok, go);
      if (!go) {
        ok = false;
        break;
      }
      if (kp > 0 && pw == 0 && lane == 0) {
        totals_s[par] = total;
        // q's rope rows of this piece's token, once QK^T of piece kp-2 is done with them
        if (kp < 2 || mbar_wait(&bars[kBarQRopeFree + par], ((kp >> 1) - 1) & 1, wl)) {
          ++rope_loads[par];
          mbar_arrive_expect_tx(&bars[kBarQLoad + par], 4u * 16u * 128u);
          for (int w = 0; w < 4; ++w)
            tma_load_3d(smem_u32(smem + kOffQRope + (32 * w + 16 * par) * 128), &tmap_qrope, 512, 16 * w, us.t,
                        &bars[kBarQLoad + par]);
        } else {
          fail();   // the others stop at the next resolution
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarListReady + par]);
      const int cnt = piece_tiles(pc, total);
      int seg = 0;
      for (int i = 0; i < cnt && !*abort_s; ++i, ++n) {
        const int s = n % kStages;
        if (n >= kStages && !(ok = wait_warp(&bars[kBarKvEmpty + s], ((n / kStages) - 1) & 1))) break;
        const int first = kNt * (pc.k0 + i * pc.stride);
        if (first >= (seg + 1) * kListCap) {
          // rare (more valid entries than the list holds): this warp re-resolves the
          // entries of its own row groups for the segment that holds this tile
          seg = first / kListCap;
          int ord = 0;
          for (int j0 = 0; j0 < p.top_k; j0 += 32) {
            const int j = j0 + lane;
            const int row = j < p.top_k ? resolve_row<kInterleaved>(p, us.bt_row, __ldg(us.idx + j), us.sel, false) : -1;
            const unsigned mask = __ballot_sync(0xffffffffu, row >= 0);
            const int o = ord + __popc(mask & lanemask_lt()) - seg * kListCap;
            if (row >= 0 && o >= 0 && o < kListCap && ((o % kNt) / 4) % kProducerWarps == pw) lst[o] = row;
            ord += __popc(mask);
          }
          __syncwarp();
        }
        char* st = smem + s * kStageBytes;
        if (lane == 0) mbar_arrive_expect_tx(&bars[kBarKvFull + s], kStageBytes / kProducerWarps);
        __syncwarp();
        constexpr int kGroupsPerWarp = kNt / 4 / kProducerWarps;   // 2
        if (lane < kColBlocks * kGroupsPerWarp) {
          const int g = pw + kProducerWarps * (lane / kColBlocks), jb = lane % kColBlocks;
          int rr[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int e = first + 4 * g + k;
            rr[k] = e < total ? lst[e - seg * kListCap] : sp.num_rows;   // past the end: zero fill
          }
          tma_gather4(smem_u32(st + blk_off(jb) + g * 512), &tmap_rows, 64 * jb, rr[0], rr[1], rr[2], rr[3],
                      &bars[kBarKvFull + s]);
        }
        __syncwarp();
      }
    }
    if (!ok) fail();
    // no gather or q rope load of this CTA may still be landing in shared memory at exit
    for (int k = n > kStages ? n - kStages : 0; k < n; ++k)
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarKvFull + k % kStages], (k / kStages) & 1, kDrainLimit)))
        report_status(p.status, kStatusTimeout);
    if (pw == 0 && lane == 0)
      for (int x = 0; x < 2; ++x)
        if (rope_loads[x] > 0 && !mbar_wait(&bars[kBarQLoad + x], (rope_loads[x] - 1) & 1, kDrainLimit))
          report_status(p.status, kStatusTimeout);
  } else if (warp == kQkWarp || warp == kPvWarp) {
    // =================== tcgen05 MMA issue: QK^T (warp 8) and P.V (warp 9) ========
    if (lane == 0) {
      bool ok = true;
      int n = 0;   // tiles so far (all pieces)
      if (warp == kQkWarp) {
        // test hook: a wait that cannot complete, so the wait limit runs out
        ok = !p.stall || mbar_wait(&bars[kBarNever], 0, wl);
        // latent steps: M = 128 (two column halves of 64 heads), N = 64 (block j's rows,
        // then block j+4's); rope steps: M = 128 (the piece's q rope rows), N = 32
        const uint32_t id_lat = idesc_bf16(128, 2 * kNt, 0, 0);
        const uint32_t id_rope = idesc_bf16(128, kNt, 0, 0);
        for (int kp = 0; ok && kp < n_pieces && !*abort_s; ++kp) {
          const Piece pc = piece_at(sp, kp, crank, (int)G);
          const int par = kp & 1;
          if (kp > 0 && !(ok = mbar_wait(&bars[kBarListReady + par], (kp >> 1) & 1, wl))) break;
          const int cnt = piece_tiles(pc, totals_s[par]);
          mbar_arrive(&bars[kBarListFree + par]);
          // this piece's q: rope rows in shared memory, latent part in TMEM
          if (!(ok = mbar_wait(&bars[kBarQLoad + par], (kp >> 1) & 1, wl))) break;
          if (!(ok = mbar_wait(&bars[kBarQReady], kp & 1, wl))) break;
          tc_fence_after();
          const uint32_t qrope = smem_u32(smem + kOffQRope + 16 * 128 * par);
          for (int i = 0; i < cnt; ++i, ++n) {
            const int s = n % kStages, bb = n & 1;
            if (!(ok = mbar_wait(&bars[kBarKvFull + s], (n / kStages) & 1, wl))) break;
            // the score buffer is free once the softmax has read tile n-2 from it
            if (n >= 2 && !(ok = mbar_wait(&bars[kBarSFree + bb], ((n >> 1) - 1) & 1, wl))) break;
            tc_fence_after();
            const uint32_t st = smem_u32(smem + s * kStageBytes);
            const uint32_t d = tmem + kColS + 64 * bb;
#pragma unroll
            for (int k = 0; k < 16; ++k)
              mma_ts(d, tmem + kColQ + 8 * k,
                     smem_desc(st + blk_off(k >> 2) + (k & 3) * 32, 16, 1024, kSwizzle128), id_lat, k > 0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(d, smem_desc(qrope + 32 * k, 16, 1024, kSwizzle128),
                     smem_desc(st + blk_off(8) + 32 * k, 16, 1024, kSwizzle128), id_rope, 1);
            mma_commit(&bars[kBarSFull + bb]);
          }
          if (!ok) break;
          // the piece's q rope rows may be overwritten once its last QK^T has completed
          if (cnt > 0) mma_commit(&bars[kBarQRopeFree + par]);
          else mbar_arrive(&bars[kBarQRopeFree + par]);
        }
      } else {
        // A = V^T: output columns 128m..128m+127 (latent blocks 2m, 2m+1, 8 KB apart in
        // the stage) of 16 tile rows, MN-major; B = P^T: 64 heads x 16 rows, K-major SW64.
        // The four output blocks are independent accumulators: issuing them between the two
        // steps of each keeps dependent MMAs apart.
        const uint32_t id_pv = idesc_bf16(128, kNH, 1, 0);
        const uint32_t pt = smem_u32(smem + kOffP);
        static_assert(blk_off(1) - blk_off(0) == 2 * kBlk && blk_off(3) - blk_off(2) == 2 * kBlk &&
                          blk_off(5) - blk_off(4) == 2 * kBlk && blk_off(7) - blk_off(6) == 2 * kBlk,
                      "the two blocks of an output block sit 2 kBlk apart");
        for (int kp = 0; ok && kp < n_pieces && !*abort_s; ++kp) {
          const Piece pc = piece_at(sp, kp, crank, (int)G);
          const int par = kp & 1;
          if (kp > 0 && !(ok = mbar_wait(&bars[kBarListReady + par], (kp >> 1) & 1, wl))) break;
          const int cnt = piece_tiles(pc, totals_s[par]);
          mbar_arrive(&bars[kBarListFree + par]);
          // O holds the previous piece's result until the softmax warps have read it
          if (kp >= 1 && !(ok = mbar_wait(&bars[kBarODrained], (kp - 1) & 1, wl))) break;
          tc_fence_after();
          for (int i = 0; i < cnt; ++i, ++n) {
            const int s = n % kStages, bb = n & 1;
            if (!(ok = mbar_wait(&bars[kBarPReady + bb], (n >> 1) & 1, wl))) break;
            tc_fence_after();
            const uint32_t st = smem_u32(smem + s * kStageBytes);
            const uint32_t ptb = pt + bb * kPBytes;
#pragma unroll
            for (int k = 0; k < kNt / 16; ++k)
#pragma unroll
              for (int m = 0; m < 4; ++m)
                mma_ss(tmem + kColO + kNH * m, smem_desc(st + blk_off(2 * m) + 2048 * k, 2 * kBlk, 1024, kSwizzle128),
                       smem_desc(ptb + 32 * k, 16, 512, kSwizzle64), id_pv, (i > 0 || k > 0) ? 1u : 0u);
            mma_commit(&bars[kBarKvEmpty + s]);
            mma_commit(&bars[kBarPFree + bb]);
          }
          if (!ok) break;
          if (cnt > 0) mma_commit(&bars[kBarPvFinal]);
          else mbar_arrive(&bars[kBarPvFinal]);
        }
      }
      if (!ok) fail();
      // every MMA this thread issued has completed before TMEM is released
      uint64_t* fin_bar = &bars[warp == kQkWarp ? kBarMmaFin : kBarMmaFin2];
      mma_commit(fin_bar);
      if (!mbar_wait(fin_bar, 0, kDrainLimit)) report_status(p.status, kStatusTimeout);
    }
  }

  // ---- one-unit schedule: merge of the cluster's partial results and the output ----
  // Every thread of every CTA of the cluster reaches both cluster barriers.
  __syncwarp();
  if (!sp.balanced) {
  const int t = us_first.t, r = us_first.r;
  bool have_o = false;
  if (warp < 4) {
    if (last_cnt > 0 && !*abort_s) {
      have_o = wait_warp(&bars[kBarPvFinal], 0);
      if (!have_o) fail();
    }
    // the head's sum is its two lanes' shares
    const float l_sum = l_part + __shfl_xor_sync(0xffffffffu, l_part, 16);
    if (lane < 16) ml_s[head] = (have_o && head < p.h) ? make_float2(m_ref, l_sum) : make_float2(-INFINITY, 0.f);
  }
  tc_fence_before();
  cluster_sync();   // every CTA's (m, l) is published
  tc_fence_after();
  if (warp < 4 && lane < 16) {
    // head `head`: the merged max M, total sum L and this CTA's weight exp2(m - M) / L
    float M = -INFINITY;
    for (uint32_t c = 0; c < G; ++c) {
      float mc;
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(mc) : "r"(mapa(&ml_s[head], c) + 0u));
      M = fmaxf(M, mc);
    }
    float Lsum = 0.f;
    for (uint32_t c = 0; c < G; ++c) {
      float mc, lc;
      const uint32_t a = mapa(&ml_s[head], c);
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(mc) : "r"(a));
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(lc) : "r"(a + 4u));
      if (mc != -INFINITY) Lsum += ex2(mc - M) * lc;
    }
    const float mine = ml_s[head].x;
    scale_s[head] = (Lsum > 0.f && mine != -INFINITY) ? ex2(mine - M) / Lsum : 0.f;
    if (crank == 0 && head < p.h && !*abort_s)
      p.lse[((size_t)r * T + t) * p.h + head] = Lsum > 0.f ? (M + __log2f(Lsum)) * kLn2 : -INFINITY;
  }
  const int v = warp * 32 + lane;   // TMEM lane of warps 0-3: output column v of each 128-column block
  // The output leaves through TMA tensor stores of 32-column x h-head boxes staged in the
  // idle stages: box (m, c) holds output columns 128m + 32c .. +31 of every head, one
  // 128-byte SW128 row per head, so warp c of the softmax warps fills box (m, c) with one
  // conflict-free 128-byte row store per head.
  auto stage_box = [&](char* box, int hh, float x) {
    *reinterpret_cast<float*>(box + hh * 128 + ((((lane >> 2) ^ (hh & 7)) << 4) | ((lane & 3) << 2))) = x;
  };
  const int out_tok = r * T + t;   // token row of out (or of the shard's partials)
  // the merge buffer (G > 1, in the idle stages): for block m, owner m % G, slot of source
  // CTA c: recv[((c * (4 / G) + m / G) * 128 + v) * 64 + hh], 16-byte chunks swizzled by v;
  // the owner's boxes follow it
  float* recv = reinterpret_cast<float*>(smem);
  const int blocks_per = 4 / (int)G;
  char* staging = smem + (G == 1 ? 0 : 4 * 128 * kNH * 4);
  static_assert(4 * 128 * kNH * 4 + 2 * 4 * kNH * 128 <= kOffList, "merge buffer and boxes stay below the lists");
  if (warp < 4) {
    named_barrier(2, 128);
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    // the heads' output scales in registers: read from shared memory between the staging
    // stores below, each would wait for the stores before it
    float sc[kNH];
#pragma unroll
    for (int hh = 0; hh < kNH; ++hh) sc[hh] = scale_s[hh];
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
      uint32_t o[kNH];
      if (have_o) {
#pragma unroll
        for (int c16 = 0; c16 < kNH / 16; ++c16)
          tmem_ld16(lane_base + kColO + kNH * m + 16 * c16, *reinterpret_cast<uint32_t(*)[16]>(&o[16 * c16]));
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int k = 0; k < kNH; ++k) o[k] = 0u;
      }
      if (G == 1) {
        if (!*abort_s) {
          char* box = staging + (4 * m + warp) * (kNH * 128);
#pragma unroll
          for (int hh = 0; hh < kNH; ++hh) stage_box(box, hh, __uint_as_float(o[hh]) * sc[hh]);
        }
        continue;
      }
      const uint32_t owner = (uint32_t)m % G;
      float* slot = recv + ((size_t)(crank * blocks_per + m / (int)G) * 128 + v) * kNH;
      const uint32_t dst = mapa(slot, owner);
#pragma unroll
      for (int c4 = 0; c4 < kNH / 4; ++c4) {
        const int sw = c4 ^ (v & (kNH / 4 - 1));
        st_cluster_v4(dst + 16u * sw, __float_as_uint(__uint_as_float(o[4 * c4]) * sc[4 * c4]),
                      __float_as_uint(__uint_as_float(o[4 * c4 + 1]) * sc[4 * c4 + 1]),
                      __float_as_uint(__uint_as_float(o[4 * c4 + 2]) * sc[4 * c4 + 2]),
                      __float_as_uint(__uint_as_float(o[4 * c4 + 3]) * sc[4 * c4 + 3]));
      }
    }
    if (G == 1) {
      fence_proxy_async_smem();
      named_barrier(2, 128);   // every box is staged
      if (threadIdx.x == 0 && !*abort_s) {
        for (int b = 0; b < 16; ++b)
          tma_store_3d(&tmap_out, smem_u32(staging + b * (kNH * 128)), 32 * b, 0, out_tok);
        bulk_commit_group();
        bulk_wait_read<0>();   // shared memory may be released once read; the writes finish with the grid
      }
    }
  }
  tc_fence_before();
  cluster_sync();   // every CTA's scaled partial O has landed with its owner
  tc_fence_after();
  if (G > 1 && warp < 4) {
    // this CTA's output blocks: the sum of the G scaled partials, staged as boxes
    int nb = 0;
    for (int m = (int)crank; m < 4; m += (int)G, ++nb) {
      float acc[kNH];
#pragma unroll
      for (int k = 0; k < kNH; ++k) acc[k] = 0.f;
      for (uint32_t c = 0; c < G; ++c) {
        const float* slot = recv + ((size_t)(c * blocks_per + m / (int)G) * 128 + v) * kNH;
#pragma unroll
        for (int c4 = 0; c4 < kNH / 4; ++c4) {
          const float4 x = *reinterpret_cast<const float4*>(slot + 4 * (c4 ^ (v & (kNH / 4 - 1))));
          acc[4 * c4] += x.x; acc[4 * c4 + 1] += x.y; acc[4 * c4 + 2] += x.z; acc[4 * c4 + 3] += x.w;
        }
      }
      char* box = staging + (4 * nb + warp) * (kNH * 128);
#pragma unroll
      for (int hh = 0; hh < kNH; ++hh) stage_box(box, hh, acc[hh]);
    }
    fence_proxy_async_smem();
    named_barrier(2, 128);   // every owned box is staged
    if (threadIdx.x == 0 && !*abort_s) {
      int k = 0;
      for (int m = (int)crank; m < 4; m += (int)G, ++k)
        for (int c = 0; c < 4; ++c)
          tma_store_3d(&tmap_out, smem_u32(staging + (4 * k + c) * (kNH * 128)), 128 * m + 32 * c, 0, out_tok);
      bulk_commit_group();
      bulk_wait_read<0>();
    }
  }
  }

  // ---- teardown ------------------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <bool kIL>
constexpr auto stack_kernel() {
  return decode_stack_kernel<kIL>;
}

}  // namespace

bool stack_supports(int h) { return h > 32 && h <= kNH; }

size_t stack_workspace_bytes(long long units, int h, int top_k, int n_sms) {
  if (!stack_supports(h) || top_k <= 0 || n_sms <= 0 || units <= n_sms) return 0;
  auto a256 = [](size_t x) { return (x + 255) / 256 * 256; };
  return a256((size_t)2 * n_sms * kNH * kDV * 4) + a256((size_t)2 * n_sms * kNH * sizeof(float2)) +
         a256((size_t)units * 4);
}

cudaError_t prepare_decode_stack() {
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    for (auto kernel : {stack_kernel<false>(), stack_kernel<true>()}) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
    }
    attr_set[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

cudaError_t launch_decode_stack(const DecodeParams& p, const CUtensorMap& rows_map, const CUtensorMap& qrope_map,
                                const CUtensorMap& out_map, int n_sms, cudaStream_t stream) {
  const long long T = (long long)p.B * p.Q;
  const long long units = T * p.n_splits;
  if (units == 0) return cudaSuccess;
  const long long num_rows = (long long)p.num_blocks * p.block_size;
  cudaError_t e = prepare_decode_stack();
  if (e != cudaSuccess) return e;
  // balanced ranges of tiles when the caller's workspace allows it (and units outnumber
  // the SMs), else one unit per CTA or per cluster
  const size_t need = stack_workspace_bytes(units, p.h, p.top_k, n_sms);
  const bool balanced = need > 0 && p.workspace && p.workspace_bytes >= need &&
                        (reinterpret_cast<uintptr_t>(p.workspace) & 255) == 0;
  const int G = balanced ? 1 : narrow_cluster_size(units, n_sms);
  if (!stack_supports(p.h) || num_rows >= 0x7fffffffLL || units * G > 0x7fffffffLL) return cudaErrorInvalidValue;
  StackParams sp;
  memset(&sp, 0, sizeof sp);
  sp.p = p;
  sp.num_rows = (int)num_rows;
  long long grid = units * G;
  if (balanced) {
    auto a256 = [](size_t x) { return (x + 255) / 256 * 256; };
    char* ws = static_cast<char*>(p.workspace);
    sp.balanced = 1;
    sp.unit_tiles = (p.top_k + kNt - 1) / kNt;
    sp.span = units * sp.unit_tiles;
    sp.ws_part = reinterpret_cast<float*>(ws);
    sp.ws_ml = reinterpret_cast<float2*>(ws + a256((size_t)2 * n_sms * kNH * kDV * 4));
    sp.ws_count = reinterpret_cast<int*>(ws + a256((size_t)2 * n_sms * kNH * kDV * 4) +
                                         a256((size_t)2 * n_sms * kNH * sizeof(float2)));
    grid = n_sms;
    // the per-unit piece counters start at zero (a merge puts its unit's back to zero; this
    // also clears what an aborted call may have left)
    e = cudaMemsetAsync(sp.ws_count, 0, (size_t)units * 4, stream);
    if (e != cudaSuccess) return e;
  }
  const bool il = p.interleave > 0 && p.n_splits > 1;
  auto kernel = il ? stack_kernel<true>() : stack_kernel<false>();
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, rows_map, qrope_map, out_map, sp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace sfa
