// sfa_narrow.cu -- tcgen05 / TMA path of sparse MLA decode for small head counts
// (h <= 32) on sm_103a.
//
// The computation is the one of "RFC: MsModeling 支持 Decode Context Parallel 仿真"
// 2.1.4.1-2.1.4.4 and "vllm-ascend PR #18870 解读" 4.3 / 4.5: for every query token,
// softmax(scale * q K^T) V over the latent rows its top-k list selects, with the
// per-head log-sum-exp, optionally restricted to one sequence shard (DCP).
//
// With few heads the step is a gather of 1152-byte rows with little arithmetic per
// byte, so one CTA holds everything a unit needs and nothing crosses between CTAs
// per tile:
//   * each CTA gathers whole rows (all 576 columns) of its tiles of the unit;
//   * QK^T: S[heads, rows] with the heads as M (padded to 128, q's latent part in
//     TMEM, its rope part in shared memory) and 48 rows as N, so the online softmax
//     keeps one thread per head;
//   * P.V is formed transposed, O^T[v, heads] += V^T[v, rows] P^T[rows, heads]: M is
//     128 output columns (four blocks cover the 512), N the padded head count, K the
//     48 rows.  V^T is read straight from the gathered tile (MN-major operand) and
//     P^T from a small shared-memory tile the softmax writes (K-major operand), so O
//     takes only 4 x N columns of TMEM.
// When a batch has fewer units (token, shard) than half the SMs, a cluster of G = 2
// or 4 CTAs shares each unit: CTA c takes tiles c, c + G, ... with its own online
// softmax, and at the end the CTAs merge their (O, m, l) over distributed shared
// memory, each finishing a quarter or half of the output columns.
//
// Warp roles (320 threads): warp 0 softmax (lane = head); warps 0-3 rescale O and
// write the output (warp w owns TMEM lanes 32w..32w+31, i.e. output columns
// 128m + 32w + lane of block m); warps 4-7 gathers (TMA tile::gather4, four rows per
// instruction); warp 8 issues QK^T; warp 9 issues P.V.  Every wait is bounded; a wait
// that gives up records SFA_ERR_DEVICE_TIMEOUT and the kernel unwinds without trapping.
#include <atomic>
#include <cuda.h>
#include <string.h>

#include "sfa_internal.h"
#include "sfa_ptx.cuh"
#include "sfa_resolve.cuh"

namespace sfa {
namespace {

using namespace ptx;

constexpr int kNt = 48;              // selected rows per tile: N of QK^T, K of P.V
constexpr int kStages = 3;           // gather pipeline depth
constexpr int kThreads = 320;
constexpr int kWarps = kThreads / 32;
constexpr int kProducerWarp = 4;     // warps 4..7 issue the gathers
constexpr int kProducerWarps = 4;
constexpr int kQkWarp = 8;
constexpr int kPvWarp = 9;
constexpr int kMaxNarrowHeads = 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P entries stay below 2^8

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kBlk = kNt * 128;                   // one 64-column SW128 block of a tile (6 KB)
constexpr int kColBlocks = 9;                     // 8 latent blocks + the rope block
constexpr int kStageBytes = kColBlocks * kBlk;    // 54 KB: whole rows
constexpr int kOffQRope = kStages * kStageBytes;
constexpr int kQRopeBytes = 128 * 128;            // q rope [128 padded heads x 64] bf16, SW128
constexpr int kOffP = kOffQRope + kQRopeBytes;
constexpr int kPBytes = kMaxNarrowHeads * 128;    // P^T [heads x 48 rows] bf16, K-major SW128 rows
constexpr int kPBuffers = 2;                      // tile i's P in buffer i % 2
constexpr int kOffList = kOffP + kPBuffers * kPBytes;
constexpr int kListCap = 43 * kNt;                // resolved rows kept at once (whole tiles)
constexpr int kOffMisc = kOffList + kListCap * 4;
// misc: per-head (m, l) [32] float2 (+0), rescale factors [32] (+256), the warps' partial
// maxima [2 tile parities][4 warps][32] (+384), output scales [32] (+1408), the warps'
// partial sums [4][32] (+1536), flags (+2048: [0] rescale, [1] abort, [2] stop), the TMEM
// address (+2064), per-warp counts (+2112)
constexpr int kMiscBytes = 2112 + 4 * kWarps;
constexpr int kOffBar = (kOffMisc + kMiscBytes + 7) / 8 * 8;
constexpr int kBarKvFull = 0, kBarKvEmpty = kBarKvFull + kStages, kBarQLoad = kBarKvEmpty + kStages,
              kBarQReady = kBarQLoad + 1, kBarSFull = kBarQReady + 1, kBarSFree = kBarSFull + 2,
              kBarPReady = kBarSFree + 2, kBarPFree = kBarPReady + 2, kBarPvFinal = kBarPFree + 2,
              kBarMmaFin = kBarPvFinal + 1, kBarMmaFin2 = kBarMmaFin + 1, kBarNever = kBarMmaFin2 + 1,
              kNumBars = kBarNever + 1;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffQRope % 1024 == 0 && kOffP % 1024 == 0 && kBlk % 1024 == 0, "SW128 operands: 1024-byte alignment");
static_assert(kListCap % kNt == 0, "list segments hold whole tiles");
// the merge receives every CTA's scaled O^T for 4 blocks x 128 columns in the idle stages
static_assert(4 * 128 * kMaxNarrowHeads * 4 <= kStages * kStageBytes, "merge buffer fits in the stages");

constexpr long long kDrainLimit = 1LL << 40;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColS = 256, kColO = 384;   // q latent (256), S x 2 (128), O^T (4 x NH)

struct NarrowParams {
  DecodeParams p;
  int num_rows;   // num_blocks * block_size (an out-of-range row used for padding)
  int q_rows;     // heads per q box: h
};

// NH: padded head count (16 or 32), the N of P.V.  kInterleaved: shard layout.
template <int NH, bool kInterleaved>
__global__ void __launch_bounds__(kThreads, 1)
    decode_narrow_kernel(const __grid_constant__ CUtensorMap tmap_rows, const __grid_constant__ CUtensorMap tmap_qrope,
                         const NarrowParams np) {
  static_assert(NH == 16 || NH == 32, "padded head count");
  const DecodeParams& p = np.p;
  extern __shared__ char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  int* list_s = reinterpret_cast<int*>(smem + kOffList);
  float2* ml_s = reinterpret_cast<float2*>(smem + kOffMisc);                   // [32] (m, l)
  float* alpha_s = reinterpret_cast<float*>(smem + kOffMisc + 256);           // [32]
  float* mxs_base = reinterpret_cast<float*>(smem + kOffMisc + 384);          // [2][4][32]
  float* scale_s = reinterpret_cast<float*>(smem + kOffMisc + 1408);          // [32]
  float* lpart_s = reinterpret_cast<float*>(smem + kOffMisc + 1536);          // [4][32]
  volatile int* flags_s = reinterpret_cast<volatile int*>(smem + kOffMisc + 2048);
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + kOffMisc + 2064);
  int* wcount_s = reinterpret_cast<int*>(smem + kOffMisc + 2112);             // [kWarps]
  volatile int* abort_s = flags_s + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  uint32_t G;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(G));
  const int unit = blockIdx.x / G;
  const int T = p.B * p.Q;
  // units go out last shard first (the heaviest shards of a sparse selection start first)
  const int t = unit % T, r = p.n_splits - 1 - unit / T;
  const int b = t / p.Q, qi = t % p.Q;
  const int seq_len = p.seq_lens[b];
  const int L = seq_len - (p.Q - 1 - qi);
  const ShardSel sel = shard_sel(seq_len, L, r, p.n_splits, p.interleave);
  const int bt_row = p.bt_per_token ? t : b;
  const int32_t* idx = p.topk_idx + (size_t)t * p.top_k;
  const long long wl = p.wait_limit;

  // ---- set-up ----------------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[kBarKvFull + s], kProducerWarps);
      mbar_init(&bars[kBarKvEmpty + s], 1);
    }
    mbar_init(&bars[kBarQLoad], 1);
    mbar_init(&bars[kBarQReady], 4);        // one arrival per warp 0-3 (each holds a copy of q)
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars[kBarSFull + x], 1);   // QK^T of the tile in this score buffer done
      mbar_init(&bars[kBarSFree + x], 4);   // the four softmax warps read this score buffer
    }
    for (int x = 0; x < kPBuffers; ++x) {
      mbar_init(&bars[kBarPReady + x], 4);  // P in this buffer and O rescaled (one arrival per warp 0-3)
      mbar_init(&bars[kBarPFree + x], 1);   // P.V has read this buffer's P (and updated O)
    }
    mbar_init(&bars[kBarPvFinal], 1);
    mbar_init(&bars[kBarMmaFin], 1);
    mbar_init(&bars[kBarMmaFin2], 1);
    mbar_init(&bars[kBarNever], 1);         // nothing arrives: the stall test hook waits on it
    flags_s[0] = 0;
    flags_s[2] = 0;
    *abort_s = 0;
    fence_barrier_init();
    // q's rope columns of this token as the shared-memory A operand of the rope steps, in
    // each 32-row group (rows 32w + head), matching the four copies of q in TMEM
    mbar_arrive_expect_tx(&bars[kBarQLoad], (uint32_t)(4 * np.q_rows * 128));
    for (int w = 0; w < 4; ++w)
      tma_load_3d(smem_u32(smem + kOffQRope + w * 32 * 128), &tmap_qrope, 512, 0, t, &bars[kBarQLoad]);
  }
  if (warp == 0) {
    tmem_alloc(tmem_base_s, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) prefetch_tmap(&tmap_rows);

  // ---- index resolution: count per warp chunk, then ordered compaction into smem ----
  const int chunk = ((p.top_k + kWarps * 32 - 1) / (kWarps * 32)) * 32;
  const int c_begin = min(warp * chunk, p.top_k), c_end = min(c_begin + chunk, p.top_k);
  const bool one_round = chunk <= 8 * 32;
  int row_r[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) row_r[k] = -1;
  {
    int cnt = resolve_chunk<kInterleaved>(p, idx, c_begin, c_end, lane, sel, bt_row, crank == 0, row_r);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0) wcount_s[warp] = cnt;
  }
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
      const int row = j < c_end ? resolve_row<kInterleaved>(p, bt_row, __ldg(idx + j), sel, false) : -1;
      const unsigned mask = __ballot_sync(0xffffffffu, row >= 0);
      const int o = off + __popc(mask & lanemask_lt());
      if (row >= 0 && o < kListCap) list_s[o] = row;
      off += __popc(mask);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;
  const int n_tiles = (total + kNt - 1) / kNt;                              // tiles of the unit
  const int n_local = n_tiles > (int)crank ? (n_tiles - (int)crank + (int)G - 1) / (int)G : 0;   // this CTA's

  auto fail = [&](void) {
    report_status(p.status, kStatusTimeout);
    *abort_s = 1;
  };
  auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, wl));
  };

  // warps 0-3: running max of head `lane` (log2 units, the same in every warp) and this
  // warp's share of its running sum (the four shares are added at the end)
  float m_ref = -INFINITY, l_part = 0.f;
  if (warp < 4) {
    // =================== softmax and O rescale (warps 0-3) ==========================
    // q's rows are replicated in the four TMEM lane quadrants (and the four 32-row groups
    // of the rope operand), so every warp sees every head's scores; warp w takes tile
    // columns 12w..12w+11.
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int head = lane;
    {
      // q's latent columns of head `lane` into this warp's quadrant as bf16 pairs (the A
      // operand of the latent steps of QK^T); lanes past h hold zeros
      const bool have = lane < p.h;
      const uint4* qsrc = reinterpret_cast<const uint4*>(p.q + ((size_t)t * p.h + (have ? lane : 0)) * kDQK);
#pragma unroll 1
      for (int c64 = 0; c64 < 4; ++c64) {   // 64 columns (128 latent values) per round
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
    }
    const float c_scale = p.scale * kLog2e;
    // |scale| in log2 units, at least 1e-30: masked scores are -inf, and -inf times a zero
    // scale would be NaN.  For a zero scale every valid weight still rounds to exactly 1
    // (|scores * 1e-30| is far below one ulp of 1), the uniform average the definition gives.
    const float c_abs = fmaxf(fabsf(c_scale), 1e-30f);
    constexpr int kCols = kNt / 4;   // tile columns per warp
    const int col0 = warp * kCols;
    // Warps 0-3 leave the tile loop together: warp 0 alone reads the abort flag at the top
    // of each tile and publishes the decision before the barrier the others wait at.
    for (int i = 0; i < n_local; ++i) {
      const int bb = i & 1;
      if (warp == 0) {
        bool go = !*abort_s;
        if (go && !wait_warp(&bars[kBarSFull + bb], (i >> 1) & 1)) { fail(); go = false; }
        // P buffer bb is free once P.V of tile i-2 has read it
        if (go && i >= 2 && !wait_warp(&bars[kBarPFree + bb], ((i >> 1) - 1) & 1)) { fail(); go = false; }
        if (lane == 0) flags_s[2] = go ? 0 : 1;
      }
      named_barrier(1, 128);   // A: the scores of tile i are in TMEM and P buffer bb is free
      if (flags_s[2]) break;
      tc_fence_after();
      uint32_t v[16];
      tmem_ld16(lane_base + kColS + 64 * bb + col0, v);   // columns col0 .. col0+11 used
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarSFree + bb]);
      float s[kCols];
      const int g = (int)crank + (int)G * i;   // the unit's tile index
      const int nvalid = min(kNt, total - kNt * g);
#pragma unroll
      for (int j = 0; j < kCols; ++j) {
        float x = __uint_as_float(v[j]);
        if (c_scale < 0.f) x = -x;   // keep max(s) * |c| == max(s * c) for a negative scale
        s[j] = (col0 + j >= nvalid || head >= p.h) ? -INFINITY : x;
      }
      float mx = s[0];
#pragma unroll
      for (int j = 1; j < kCols; ++j) mx = fmaxf(mx, s[j]);
      float* mx_s = mxs_base + 128 * bb;   // [4 warps][32 heads] of this tile parity
      mx_s[warp * 32 + lane] = mx;
      named_barrier(2, 128);   // B: every warp's partial max of tile i is published
      const float mt = fmaxf(fmaxf(mx_s[lane], mx_s[32 + lane]), fmaxf(mx_s[64 + lane], mx_s[96 + lane])) * c_abs;
      float m_new = m_ref;
      if (head < p.h && (i == 0 || mt > m_ref + kRescaleThreshold)) m_new = fmaxf(mt, m_ref);
      const float alpha = (i == 0 || head >= p.h) ? 1.f : ex2(m_ref - m_new);
      m_ref = m_new;
      uint32_t pk[kCols / 2];
      float sm = 0.f;
#pragma unroll
      for (int j = 0; j < kCols / 2; ++j) {
        const float e0 = head < p.h ? ex2(fmaf(s[2 * j], c_abs, -m_new)) : 0.f;
        const float e1 = head < p.h ? ex2(fmaf(s[2 * j + 1], c_abs, -m_new)) : 0.f;
        sm += e0 + e1;
        pk[j] = pack_bf16(e0, e1);
      }
      l_part = l_part * alpha + sm;
      if (lane < NH) {
        // this head's row of P^T, tile columns col0..col0+11 = bytes 24w..24w+23 of the
        // K-major SW128 row: three 8-byte pieces, none crossing a 16-byte chunk
        char* p_row = smem + kOffP + bb * kPBytes + head * 128;
#pragma unroll
        for (int u = 0; u < 3; ++u) {
          const int byte = 2 * col0 + 8 * u;
          *reinterpret_cast<uint2*>(p_row + ((((byte >> 4) ^ (head & 7)) << 4) | (byte & 15))) =
              make_uint2(pk[2 * u], pk[2 * u + 1]);
        }
        fence_proxy_async_smem();
      }
      if (warp == 0) {
        // O is rescaled (rarely: the reference max moves only by more than the threshold)
        // once P.V of the previous tile has completed.  (Tile i+1 waits on the same phase
        // of that buffer again: it cannot have moved on, P.V of tile i+1 is not issued yet.)
        const bool resc = __any_sync(0xffffffffu, alpha != 1.f);
        if (resc && i >= 1 && !wait_warp(&bars[kBarPFree + (bb ^ 1)], ((i - 1) >> 1) & 1)) fail();
        if (lane < NH) alpha_s[lane] = alpha;
        if (lane == 0) flags_s[0] = resc ? 1 : 0;
      }
      named_barrier(3, 128);   // C: whether O is rescaled, and by what
      if (flags_s[0] && !*abort_s) {
        tc_fence_after();
        // O^T lane v holds output column v of every head: scale column hh by alpha[hh]
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int c16 = 0; c16 < NH / 16; ++c16) {
            uint32_t o[16];
            tmem_ld16(lane_base + kColO + NH * m + 16 * c16, o);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha_s[16 * c16 + k]);
            tmem_st16(lane_base + kColO + NH * m + 16 * c16, o);
          }
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarPReady + bb]);
    }
  } else if (warp < kProducerWarp + kProducerWarps) {
    // =================== gathers ===================================================
    // Producer warp pw issues the gathers of row groups g = pw, pw + 4, pw + 8 of each
    // of its tiles (4 rows each, all nine 64-column blocks): 27 per tile, one per lane.
    const int pw = warp - kProducerWarp;
    int seg = 0;
    int n = 0;
    bool ok = true;
    for (; n < n_local && !*abort_s; ++n) {
      const int s = n % kStages;
      if (n >= kStages && !(ok = wait_warp(&bars[kBarKvEmpty + s], ((n / kStages) - 1) & 1))) break;
      const int first = kNt * ((int)crank + (int)G * n);
      if (first >= (seg + 1) * kListCap) {
        // rare (more valid entries than the list holds): this warp re-resolves the
        // entries of its own row groups for the segment that holds this tile
        seg = first / kListCap;
        int ord = 0;
        for (int j0 = 0; j0 < p.top_k; j0 += 32) {
          const int j = j0 + lane;
          const int row = j < p.top_k ? resolve_row<kInterleaved>(p, bt_row, __ldg(idx + j), sel, false) : -1;
          const unsigned mask = __ballot_sync(0xffffffffu, row >= 0);
          const int o = ord + __popc(mask & lanemask_lt()) - seg * kListCap;
          if (row >= 0 && o >= 0 && o < kListCap && ((o % kNt) / 4) % kProducerWarps == pw) list_s[o] = row;
          ord += __popc(mask);
        }
        __syncwarp();
      }
      char* st = smem + s * kStageBytes;
      if (lane == 0) mbar_arrive_expect_tx(&bars[kBarKvFull + s], kStageBytes / kProducerWarps);
      __syncwarp();
      constexpr int kGroupsPerWarp = kNt / 4 / kProducerWarps;   // 3
      if (lane < kColBlocks * kGroupsPerWarp) {
        const int g = pw + kProducerWarps * (lane / kColBlocks), j = lane % kColBlocks;
        int rr[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int e = first + 4 * g + k;
          rr[k] = e < total ? list_s[e - seg * kListCap] : np.num_rows;   // past the end: zero fill
        }
        tma_gather4(smem_u32(st + j * kBlk + g * 512), &tmap_rows, 64 * j, rr[0], rr[1], rr[2], rr[3],
                    &bars[kBarKvFull + s]);
      }
      __syncwarp();
    }
    if (!ok) fail();
    // no gather of this CTA may still be landing in shared memory at exit
    for (int k = n > kStages ? n - kStages : 0; k < n; ++k)
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarKvFull + k % kStages], (k / kStages) & 1, kDrainLimit)))
        report_status(p.status, kStatusTimeout);
  } else if (warp == kQkWarp || warp == kPvWarp) {
    // =================== tcgen05 MMA issue: QK^T (warp 8) and P.V (warp 9) ========
    // q's rope load must have landed before the CTA exits, whatever happens below
    bool q_landed = false;
    if (lane == 0 && n_local > 0) {
      bool ok = true;
      if (warp == kQkWarp) {
        // test hook: a wait that cannot complete, so the wait limit runs out
        ok = !p.stall || mbar_wait(&bars[kBarNever], 0, wl);
        ok = ok && (q_landed = mbar_wait(&bars[kBarQLoad], 0, wl)) && mbar_wait(&bars[kBarQReady], 0, wl);
        tc_fence_after();
        const uint32_t id_qk = idesc_bf16(128, kNt, 0, 0);
        const uint32_t qrope = smem_u32(smem + kOffQRope);
        for (int n = 0; ok && n < n_local && !*abort_s; ++n) {
          const int s = n % kStages, bb = n & 1;
          if (!(ok = mbar_wait(&bars[kBarKvFull + s], (n / kStages) & 1, wl))) break;
          // the score buffer is free once the softmax has read tile n-2 from it
          if (n >= 2 && !(ok = mbar_wait(&bars[kBarSFree + bb], ((n >> 1) - 1) & 1, wl))) break;
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * kStageBytes);
          const uint32_t d = tmem + kColS + 64 * bb;
#pragma unroll
          for (int k = 0; k < 32; ++k)
            mma_ts(d, tmem + kColQ + 8 * k, smem_desc(st + (k >> 2) * kBlk + (k & 3) * 32, 16, 1024, kSwizzle128),
                   id_qk, k > 0);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(d, smem_desc(qrope + 32 * k, 16, 1024, kSwizzle128),
                   smem_desc(st + 8 * kBlk + 32 * k, 16, 1024, kSwizzle128), id_qk, 1);
          mma_commit(&bars[kBarSFull + bb]);
        }
      } else {
        // A = V^T: output columns 128m..128m+127 (latent blocks 2m, 2m+1) of 16 tile rows,
        // MN-major; B = P^T: NH heads x 16 rows, K-major
        const uint32_t id_pv = idesc_bf16(128, NH, 1, 0);
        const uint32_t pt = smem_u32(smem + kOffP);
        for (int n = 0; ok && n < n_local && !*abort_s; ++n) {
          const int s = n % kStages, bb = n & 1;
          if (!(ok = mbar_wait(&bars[kBarPReady + bb], (n >> 1) & 1, wl))) break;
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * kStageBytes);
          const uint32_t ptb = pt + bb * kPBytes;
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int k = 0; k < kNt / 16; ++k)
              mma_ss(tmem + kColO + NH * m, smem_desc(st + 2 * m * kBlk + 2048 * k, kBlk, 1024, kSwizzle128),
                     smem_desc(ptb + 32 * k, 16, 1024, kSwizzle128), id_pv, (n > 0 || k > 0) ? 1u : 0u);
          mma_commit(&bars[kBarKvEmpty + s]);
          mma_commit(&bars[kBarPFree + bb]);
          if (n == n_local - 1) mma_commit(&bars[kBarPvFinal]);
        }
      }
      if (!ok) fail();
      // every MMA this thread issued has completed before TMEM is released
      uint64_t* fin_bar = &bars[warp == kQkWarp ? kBarMmaFin : kBarMmaFin2];
      mma_commit(fin_bar);
      if (!mbar_wait(fin_bar, 0, kDrainLimit)) report_status(p.status, kStatusTimeout);
    }
    if (warp == kQkWarp && lane == 0 && !q_landed && !mbar_wait(&bars[kBarQLoad], 0, kDrainLimit))
      report_status(p.status, kStatusTimeout);
  }

  // ---- merge of the cluster's partial results and the output ---------------------
  // Every thread of every CTA of the cluster reaches both cluster barriers.
  __syncwarp();
  bool have_o = false;
  if (warp < 4) {
    if (n_local > 0 && !*abort_s) {
      have_o = wait_warp(&bars[kBarPvFinal], 0);
      if (!have_o) fail();
    }
    lpart_s[warp * 32 + lane] = l_part;
    named_barrier(2, 128);
    if (warp == 0) {
      const float l_sum = (lpart_s[lane] + lpart_s[32 + lane]) + (lpart_s[64 + lane] + lpart_s[96 + lane]);
      ml_s[lane] = (have_o && lane < p.h) ? make_float2(m_ref, l_sum) : make_float2(-INFINITY, 0.f);
    }
  }
  tc_fence_before();
  cluster_sync();   // every CTA's (m, l) is published
  tc_fence_after();
  if (warp == 0) {
    // head `lane`: the merged max M, total sum L and this CTA's weight exp2(m - M) / L
    float M = -INFINITY;
    for (uint32_t c = 0; c < G; ++c) {
      float mc;
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(mc) : "r"(mapa(&ml_s[lane], c) + 0u));
      M = fmaxf(M, mc);
    }
    float Lsum = 0.f;
    for (uint32_t c = 0; c < G; ++c) {
      float mc, lc;
      const uint32_t a = mapa(&ml_s[lane], c);
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(mc) : "r"(a));
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(lc) : "r"(a + 4u));
      if (mc != -INFINITY) Lsum += ex2(mc - M) * lc;
    }
    const float mine = ml_s[lane].x;
    scale_s[lane] = (Lsum > 0.f && mine != -INFINITY) ? ex2(mine - M) / Lsum : 0.f;
    if (crank == 0 && lane < p.h && !*abort_s)
      p.lse[((size_t)r * T + t) * p.h + lane] = Lsum > 0.f ? (M + __log2f(Lsum)) * kLn2 : -INFINITY;
  }
  // the merge buffer (in the idle stages): for block m, owner m % G, slot of source CTA c:
  //   recv[((c * (4 / G) + m / G) * 128 + v) * NH + hh], 16-byte chunks swizzled by v
  float* recv = reinterpret_cast<float*>(smem);
  const int blocks_per = 4 / (int)G;
  if (warp < 4) {
    named_barrier(2, 128);
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int v = warp * 32 + lane;   // TMEM lane: output column v of each 128-column block
    // the heads' output scales in registers: read from shared memory between the stores
    // below, each would wait for the stores before it
    float sc[NH];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) sc[hh] = scale_s[hh];
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
      uint32_t o[NH];
      if (have_o) {
#pragma unroll
        for (int c16 = 0; c16 < NH / 16; ++c16) tmem_ld16(lane_base + kColO + NH * m + 16 * c16,
                                                          *reinterpret_cast<uint32_t(*)[16]>(&o[16 * c16]));
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int k = 0; k < NH; ++k) o[k] = 0u;
      }
      const uint32_t owner = (uint32_t)m % G;
      float* slot = recv + ((size_t)(crank * blocks_per + m / (int)G) * 128 + v) * NH;
      const uint32_t dst = mapa(slot, owner);
#pragma unroll
      for (int c4 = 0; c4 < NH / 4; ++c4) {
        const int sw = c4 ^ (v & (NH / 4 - 1));
        st_cluster_v4(dst + 16u * sw, __float_as_uint(__uint_as_float(o[4 * c4]) * sc[4 * c4]),
                      __float_as_uint(__uint_as_float(o[4 * c4 + 1]) * sc[4 * c4 + 1]),
                      __float_as_uint(__uint_as_float(o[4 * c4 + 2]) * sc[4 * c4 + 2]),
                      __float_as_uint(__uint_as_float(o[4 * c4 + 3]) * sc[4 * c4 + 3]));
      }
    }
  }
  tc_fence_before();
  cluster_sync();   // every CTA's scaled partial O has landed with its owner
  tc_fence_after();
  if (warp < 4 && !*abort_s) {
    // this CTA's output blocks: the sum of the G scaled partials; one coalesced 128-byte
    // row segment per (head, warp) store
    const int v = warp * 32 + lane;
    float* outp = p.out + ((size_t)r * T + t) * p.h * kDV;
    for (int m = (int)crank; m < 4; m += (int)G) {
      float acc[NH];
#pragma unroll
      for (int k = 0; k < NH; ++k) acc[k] = 0.f;
      for (uint32_t c = 0; c < G; ++c) {
        const float* slot = recv + ((size_t)(c * blocks_per + m / (int)G) * 128 + v) * NH;
#pragma unroll
        for (int c4 = 0; c4 < NH / 4; ++c4) {
          const float4 x = *reinterpret_cast<const float4*>(slot + 4 * (c4 ^ (v & (NH / 4 - 1))));
          acc[4 * c4] += x.x; acc[4 * c4 + 1] += x.y; acc[4 * c4 + 2] += x.z; acc[4 * c4 + 3] += x.w;
        }
      }
#pragma unroll
      for (int hh = 0; hh < NH; ++hh)
        if (hh < p.h) outp[(size_t)hh * kDV + 128 * m + v] = acc[hh];
    }
  }

  // ---- teardown ------------------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int NH, bool kIL>
constexpr auto narrow_kernel() {
  return decode_narrow_kernel<NH, kIL>;
}

}  // namespace

// SM count of the current device, looked up once per device
int device_sm_count() {
  static std::atomic<int> n_sms[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  int n = n_sms[dev].load(std::memory_order_acquire);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    n_sms[dev].store(n, std::memory_order_release);
  }
  return n;
}

bool narrow_supports(int h) { return h >= 1 && h <= kMaxNarrowHeads; }

int narrow_cluster_size(long long units, int n_sms) {
  // share a unit between 2 or 4 CTAs while the units alone fill less than half the GPU
  int G = 1;
  while (G < 4 && units * G * 2 <= n_sms) G *= 2;
  return G;
}

cudaError_t prepare_decode_narrow() {
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    for (auto kernel : {narrow_kernel<16, false>(), narrow_kernel<16, true>(), narrow_kernel<32, false>(),
                        narrow_kernel<32, true>()}) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
      if (e != cudaSuccess) return e;
    }
    attr_set[dev].store(true, std::memory_order_release);
  }
  (void)device_sm_count();
  return cudaSuccess;
}

cudaError_t launch_decode_narrow(const DecodeParams& p, const CUtensorMap& rows_map, const CUtensorMap& qrope_map,
                                 cudaStream_t stream) {
  const long long T = (long long)p.B * p.Q;
  const long long units = T * p.n_splits;
  if (units == 0) return cudaSuccess;
  const long long num_rows = (long long)p.num_blocks * p.block_size;
  cudaError_t e = prepare_decode_narrow();
  if (e != cudaSuccess) return e;
  const int G = narrow_cluster_size(units, device_sm_count());
  if (num_rows >= 0x7fffffffLL || units * G > 0x7fffffffLL) return cudaErrorInvalidValue;
  NarrowParams np;
  np.p = p;
  np.num_rows = (int)num_rows;
  np.q_rows = p.h;
  const bool il = p.interleave > 0 && p.n_splits > 1;
  auto kernel = p.h <= 16 ? (il ? narrow_kernel<16, true>() : narrow_kernel<16, false>())
                          : (il ? narrow_kernel<32, true>() : narrow_kernel<32, false>());
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)(units * G), 1, 1);
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
  e = cudaLaunchKernelEx(&cfg, kernel, rows_map, qrope_map, np);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace sfa
