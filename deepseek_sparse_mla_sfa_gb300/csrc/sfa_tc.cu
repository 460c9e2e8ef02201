// sfa_tc.cu -- tcgen05 / TMA path of sparse MLA decode on sm_103a.
//
// The computation is the one of "RFC: MsModeling 支持 Decode Context Parallel 仿真"
// 2.1.4.1-2.1.4.4 and "vllm-ascend PR #18870 解读" 4.3 / 4.5: for every query token,
// softmax(scale * q K^T) V over the latent rows its top-k list selects, with the
// per-head log-sum-exp, optionally restricted to one sequence shard (DCP).
//
// Layout of the work.  One work unit = (query token, shard).  Two CTAs of a
// cluster share a unit and all of its 128 (padded) heads:
//   * the QK^T contraction is split by columns: CTA c holds q's latent columns
//     [256c, 256c+256) in TMEM (A operand) and rope columns [512+32c, 544+32c) in
//     shared memory, and gathers exactly those columns of each selected row;
//   * each CTA sends the other its partial scores for all heads through
//     distributed shared memory; both then hold the full scores S = S_0 + S_1
//     (the same fp32 sums in both CTAs) and run the same online softmax, so their
//     probabilities, running max and sum agree bit for bit without exchanging them;
//   * P.V is split by output columns: CTA c owns out[:, 256c : 256c+256), which
//     are the latent columns it already holds (V is the latent part of the row).
//     P (bf16 pairs) overwrites the tile's partial scores in its TMEM score buffer
//     and is the TMEM (A) operand of P.V; the buffer takes the next QK^T once
//     P.V has read it.
// Each CTA therefore reads 576 of the 1152 bytes of every selected row, once.
// TMEM per CTA: O [128 heads x 256] fp32 (cols 0-255), q latent part (256-383,
// bf16 pairs), two score / probability buffers of 64 rows (384-511).  q arrives by
// TMA at kernel start: its latent half lands in the (still idle) exchange buffers,
// from where the softmax warps move it into TMEM, and its rope part lands in place
// as the shared-memory operand of the rope columns of QK^T.
//
// Warp roles (448 threads): warps 0-3 softmax / rescale / epilogue (warp w owns
// TMEM lanes 32w..32w+31 = heads 32w..32w+31), warps 4-7 gathers (TMA, twenty
// lanes each), warp 8 issues QK^T, warp 9 issues P.V, warps 10-13 send each tile's
// partial scores to the peer as soon as QK^T has produced them (warp w serves TMEM
// lane quadrant w % 4).  Every wait is bounded; a wait that gives up records
// SFA_ERR_DEVICE_TIMEOUT and the kernel unwinds without trapping.
//
// Ordering of the score exchange.  A sender copies its partials to the peer with
// cp.async.bulk shared::cluster copies, which complete only on the peer's mbarrier
// (mbarrier::complete_tx); the bulk async-group operations (commit_group /
// wait_group.read) track only copies that complete through a bulk async-group, so
// they say nothing about when such a copy has read its source.  Each 16-head slot
// of the staging area is therefore written once per tile, and rewritten for tile j
// only after the peer's softmax warps have arrived on our XFree barrier for tile j:
// they do so after reading tile j-1 from their X buffer, which they do only once
// every copy of tile j-1 has landed there, i.e. once every source slot has been read.
// A softmax warp that gives up waiting still lets the copy of the tile it was
// waiting for land (a time-capped drain) before the CTA exits.
#include <atomic>
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "sfa_internal.h"
#include "sfa_ptx.cuh"
#include "sfa_resolve.cuh"

namespace sfa {
namespace {

using namespace ptx;

constexpr int kNt = 64;          // selected rows per tile
constexpr int kStages = 4;       // gather pipeline depth
constexpr int kHeads = 128;      // heads per unit (padded)
constexpr int kThreads = 448;
constexpr int kWarps = kThreads / 32;
constexpr int kProducerWarp = 4;  // warps 4..7 issue the gathers (twenty lanes each)
constexpr int kProducerWarps = 4;
constexpr int kMmaWarp = 8;        // issues QK^T
constexpr int kPvWarp = 9;         // issues P.V
constexpr int kSendWarp = 10;      // warps 10..13 send partial scores
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P entries stay below 2^8

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kLatBlk = kNt * 128;                      // one 64-column SW128 block of a tile
constexpr int kRopeBlk = kNt * 64;                      // the 32-column SW64 rope block
constexpr int kStageBytes = 4 * kLatBlk + kRopeBlk;     // 36 KB
constexpr int kOffQRope = kStages * kStageBytes;
constexpr int kQRopeBytes = kHeads * 64;
constexpr int kOffX = kOffQRope + kQRopeBytes;
constexpr int kXBytes = kHeads * kNt * 4;               // partial scores [128 heads x 64 rows] fp32
constexpr int kXWarpBytes = kXBytes / 4;                // the 32 heads of one warp
constexpr int kXHalfBytes = kXWarpBytes / 2;            // 16 heads: one staging slot / bulk copy
// outgoing partials: one slot per 16 heads, so no slot is rewritten while a copy of the
// same tile may still be reading it
constexpr int kOffXStage = kOffX + kXBytes;
constexpr int kXStageBytes = kXBytes;
constexpr int kQBox = kHeads * 128;                     // one 64-column SW128 box of q's latent half
constexpr int kOutBox = kHeads * 128;                   // one 32-column SW128 box of out (fp32)
static_assert(8 * kOutBox <= kStages * kStageBytes, "out is staged in the gather stages");
static_assert(4 * kQBox == kXBytes + kXStageBytes, "q's latent half fills X and the staging slots");
static_assert(kOffX % 1024 == 0, "SW128 boxes need 1024-byte alignment");
constexpr int kOffList = kOffXStage + kXStageBytes;
constexpr int kListCap = 2048;                          // resolved rows kept at once (multiple of kNt)
constexpr int kOffBar = kOffList + kListCap * 4;
// barriers
constexpr int kBarKvFull = 0, kBarKvEmpty = kBarKvFull + kStages, kBarQReady = kBarKvEmpty + kStages,
              kBarSFull = kBarQReady + 1, kBarSpFree = kBarSFull + 2, kBarOReady = kBarSpFree + 2,
              kBarSFree = kBarOReady + 2, kBarXFull = kBarSFree + 2, kBarXFree = kBarXFull + 1,
              kBarPvDone = kBarXFree + 1, kBarPvFinal = kBarPvDone + 1, kBarMmaFin = kBarPvFinal + 1,
              kBarMmaFin2 = kBarMmaFin + 1, kBarQLoad = kBarMmaFin2 + 1, kBarNever = kBarQLoad + 1,
              kNumBars = kBarNever + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 128 + 1024;        // + alignment slack
static_assert(8 + 4 * kWarps <= 128, "misc area");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kStageBytes % 1024 == 0, "stages must stay 1024-byte aligned");
static_assert(kListCap % kNt == 0, "list segments hold whole tiles");

// waits for this CTA's own copies / MMAs still in flight at exit use their own
// (time-capped) limit, independent of the pipeline-wait cap
constexpr long long kDrainLimit = 1LL << 40;
constexpr uint64_t kDrainCapNs = 5000000ull;   // 5 ms: copies in flight land within microseconds

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColQ = 256, kColS = 384;
constexpr uint32_t kStageTx = kStageBytes;  // bytes a full tile delivers (OOB rows are zero-filled)

struct TcParams {
  DecodeParams p;
  int num_rows;  // num_blocks * block_size (== out-of-range row used for padding)
  int q_rows;    // heads per q box: min(h, 128)
};

// kInterleaved: the shards are interleaved (interleave size > 0 and more than one shard);
// the layout is fixed per instantiation so that no selection test branches on it.
template <bool kInterleaved>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_lat,
                     const __grid_constant__ CUtensorMap tmap_rope,
                     const __grid_constant__ CUtensorMap tmap_qlat,
                     const __grid_constant__ CUtensorMap tmap_qrope,
                     const __grid_constant__ CUtensorMap tmap_out, const TcParams tp) {
  const DecodeParams& p = tp.p;
  extern __shared__ char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  int* list_s = reinterpret_cast<int*>(smem + kOffList);
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* wcount_s = reinterpret_cast<int*>(smem + kOffMisc + 8);   // [kWarps]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();   // which half of the columns
  const uint32_t peer = crank ^ 1u;
  const int unit = blockIdx.x >> 1;
  const int T = p.B * p.Q;
  // Units go out last shard first: a sequence's most recent positions, where a sparse
  // selection usually concentrates, are its last shard, so the heaviest units start in
  // the first wave and the light ones fill in behind them.
  const int t = unit % T, r = p.n_splits - 1 - unit / T;
  const int b = t / p.Q, qi = t % p.Q;
  const int seq_len = p.seq_lens[b];
  const int L = seq_len - (p.Q - 1 - qi);
  const ShardSel sel = shard_sel(seq_len, L, r, p.n_splits, p.interleave);
  const int bt_row = p.bt_per_token ? t : b;   // block-table row of this unit
  const int32_t* idx = p.topk_idx + (size_t)t * p.top_k;
  const long long wl = p.wait_limit;

  // ---- set-up: barriers, TMEM ------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[kBarKvFull + s], kProducerWarps);
      mbar_init(&bars[kBarKvEmpty + s], 1);
    }
    mbar_init(&bars[kBarQReady], 128);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars[kBarSFull + x], 1);     // QK^T of the tile in this score buffer done
      mbar_init(&bars[kBarSpFree + x], 4);    // the 4 sender warps read this buffer's partials
      mbar_init(&bars[kBarOReady + x], 128);  // probabilities in this buffer and O rescaled
      mbar_init(&bars[kBarSFree + x], 1);     // P.V has read the probabilities: buffer free
    }
    mbar_init(&bars[kBarXFull], 1);           // arming arrival + the peer's 4 x 8 KB of partials
    mbar_init(&bars[kBarXFree], 4);           // the peer's 4 softmax warps read our partials (phase
                                              // 0: they have moved their q out of their buffers)
    mbar_init(&bars[kBarPvDone], 1);
    mbar_init(&bars[kBarPvFinal], 1);         // the last P.V of the unit has completed
    mbar_init(&bars[kBarMmaFin], 1);
    mbar_init(&bars[kBarMmaFin2], 1);
    mbar_init(&bars[kBarQLoad], 1);
    mbar_init(&bars[kBarNever], 1);           // nothing arrives: the stall test hook waits on it
    *abort_s = 0;
    fence_barrier_init();
    // q of this token: latent columns [256c, 256c+256) as four SW128 boxes into the
    // exchange buffers, rope columns [512+32c, +32) as one SW64 box into qrope
    mbar_arrive_expect_tx(&bars[kBarQLoad], (uint32_t)(tp.q_rows * (4 * 128 + 64)));
    for (int j = 0; j < 4; ++j)
      tma_load_3d(smem_u32(smem + kOffX + j * kQBox), &tmap_qlat, 256 * crank + 64 * j, 0, t, &bars[kBarQLoad]);
    tma_load_3d(smem_u32(smem + kOffQRope), &tmap_qrope, 512 + 32 * crank, 0, t, &bars[kBarQLoad]);
  }
  if (warp == 0) {
    tmem_alloc(tmem_base_s, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= kProducerWarp && warp < kProducerWarp + kProducerWarps && lane == 0) {
    prefetch_tmap(&tmap_lat);
    prefetch_tmap(&tmap_rope);
  }

  // ---- index resolution: count per warp chunk, then ordered compaction into smem ----
  // A warp's chunk of the list is resolved 8 entries per lane at a time.  When the chunk
  // fits in one such round (top_k <= 8 * kThreads), the resolved rows stay in registers
  // for the ordered write; otherwise the write pass resolves them again.
  const int chunk = ((p.top_k + kWarps * 32 - 1) / (kWarps * 32)) * 32;
  const int c_begin = min(warp * chunk, p.top_k), c_end = min(c_begin + chunk, p.top_k);
  const bool one_round = chunk <= 8 * 32;
  int row_r[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) row_r[k] = -1;   // warps with an empty chunk write nothing
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
  cluster_sync();  // both CTAs' barriers are initialised before any remote access
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;
  const int n_tiles = (total + kNt - 1) / kNt;
  // partial scores cross between the CTAs in 16-head slots; only slots holding real
  // heads (h of the padded 128) are sent
  const uint32_t x_bytes = (uint32_t)((p.h + 15) / 16) * kXHalfBytes;

  auto fail = [&](void) {
    report_status(p.status, kStatusTimeout);
    *abort_s = 1;
  };
  // waits executed by a whole warp give the same answer on every lane
  auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, wl));
  };
  auto wait_warp_cluster = [&](uint64_t* bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait<true>(bar, parity, wl));
  };

  char* qrope = smem + kOffQRope;

  if (warp < 4) {
    // =================== softmax / rescale / epilogue warps =====================
    const int head = warp * 32 + lane;
    const bool head_ok = head < p.h;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);

    const uint32_t xfree_peer = mapa(&bars[kBarXFree], peer);
    // q's latent half: from the SW128 boxes in the exchange buffers into TMEM (bf16
    // pairs); every softmax warp is done with those buffers before any of them reuses
    // its slice, and the peer may write into ours once all four warps have arrived
    {
      bool qok = wait_warp(&bars[kBarQLoad], 0);
      if (!qok) {
        fail();
        // the q load must land before this CTA can exit
        if (warp == 0 && lane == 0 && !mbar_wait(&bars[kBarQLoad], 0, kDrainLimit))
          report_status(p.status, kStatusTimeout);
        __syncwarp();
      }
      const bool have = qok && head < tp.q_rows;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v[16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int ch = 4 * hh + c;
            const uint4 x = have ? *reinterpret_cast<const uint4*>(smem + kOffX + j * kQBox + head * 128 +
                                                                   ((ch ^ (head & 7)) * 16))
                                 : make_uint4(0, 0, 0, 0);
            v[4 * c] = x.x; v[4 * c + 1] = x.y; v[4 * c + 2] = x.z; v[4 * c + 3] = x.w;
          }
          tmem_st16(lane_base + kColQ + 32 * j + 16 * hh, v);
        }
      }
      if (head >= tp.q_rows) {   // heads past h: zero rope row (the box stops at h)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4*>(qrope + head * 64 + ((k ^ ((head >> 1) & 3)) * 16)) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      tmem_st_wait();
      tc_fence_before();
      named_barrier(1, 128);
      if (lane == 0) mbar_arrive_remote_relaxed(xfree_peer);
      mbar_arrive(&bars[kBarQReady]);
    }

    const float c_scale = p.scale * kLog2e;
    // |scale| in log2 units, at least 1e-30: masked scores are -inf, and -inf times a zero
    // scale would be NaN.  For a zero scale every valid weight still rounds to exactly 1
    // (|scores * 1e-30| is far below one ulp of 1), the uniform average the definition gives.
    const float c_abs = fmaxf(fabsf(c_scale), 1e-30f);
    const char* xin = smem + kOffX + head * 256;   // the peer's partial scores of this head

    float m_ref = -INFINITY, l_sum = 0.f;  // running max (log2 units) and sum of this head
    if (warp == 0 && lane == 0 && n_tiles > 0) mbar_arrive_expect_tx(&bars[kBarXFull], x_bytes);
    int x_seen = 0;   // tiles whose partials from the peer have landed in X
    for (int i = 0; i < n_tiles && !*abort_s; ++i) {
      const int bb = i & 1;
      // full scores of tile i = our partials (in this tile's TMEM score buffer) + the
      // peer's (in X); both CTAs form the same fp32 sums.
      if (!wait_warp(&bars[kBarSFull + bb], (i >> 1) & 1)) { fail(); break; }
      tc_fence_after();
      uint32_t v[4][16];
#pragma unroll
      for (int c4 = 0; c4 < kNt / 16; ++c4) tmem_ld16(lane_base + kColS + kNt * bb + 16 * c4, v[c4]);
      tmem_ld_wait();
      if (!wait_warp_cluster(&bars[kBarXFull], i & 1)) { fail(); break; }
      x_seen = i + 1;
      if (warp == 0 && lane == 0 && i + 1 < n_tiles) mbar_arrive_expect_tx(&bars[kBarXFull], x_bytes);
      float s[kNt];
#pragma unroll
      for (int k = 0; k < kNt / 4; ++k) {
        const float4 x = *reinterpret_cast<const float4*>(xin + ((k ^ (head & 15)) * 16));
        s[4 * k] = __uint_as_float(v[k >> 2][4 * (k & 3)]) + x.x;
        s[4 * k + 1] = __uint_as_float(v[k >> 2][4 * (k & 3) + 1]) + x.y;
        s[4 * k + 2] = __uint_as_float(v[k >> 2][4 * (k & 3) + 2]) + x.z;
        s[4 * k + 3] = __uint_as_float(v[k >> 2][4 * (k & 3) + 3]) + x.w;
      }
      if (head >= p.h) {   // padding head: its slot may not have been sent
#pragma unroll
        for (int j = 0; j < kNt; ++j) s[j] = 0.f;
      }
      // our reads of the peer's partials are complete: a relaxed arrive tells the peer
      // it may overwrite X with the next tile
      __syncwarp();
      if (lane == 0) mbar_arrive_remote_relaxed(xfree_peer);
      // online softmax in log2 units; the reference max only moves when it grows past
      // the threshold, so O is rarely rescaled
      const int nvalid = min(kNt, total - kNt * i);
      if (c_scale < 0.f) {   // keep max(s) * |c| == max(s * c) for a negative scale
#pragma unroll
        for (int j = 0; j < kNt; ++j) s[j] = -s[j];
      }
      if (nvalid < kNt) {
#pragma unroll
        for (int j = 0; j < kNt; ++j)
          if (j >= nvalid) s[j] = -INFINITY;
      }
      float mx[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) mx[j] = fmaxf(fmaxf(s[4 * j], s[4 * j + 1]), fmaxf(s[4 * j + 2], s[4 * j + 3]));
#pragma unroll
      for (int w2 = 8; w2 > 0; w2 >>= 1)
#pragma unroll
        for (int j = 0; j < w2; ++j) mx[j] = fmaxf(mx[j], mx[j + w2]);
      const float mt = mx[0] * c_abs;
      float m_new = m_ref;
      if (i == 0 || mt > m_ref + kRescaleThreshold) m_new = fmaxf(mt, m_ref);
      const float alpha = i == 0 ? 1.f : ex2(m_ref - m_new);
      m_ref = m_new;
      uint32_t pk[kNt / 2];
      float sm[16];
#pragma unroll
      for (int j = 0; j < kNt / 2; ++j) {
        const float e0 = ex2(fmaf(s[2 * j], c_abs, -m_new));
        const float e1 = ex2(fmaf(s[2 * j + 1], c_abs, -m_new));
        if (j < 16) sm[j] = e0 + e1; else sm[j - 16] += e0 + e1;
        pk[j] = pack_bf16(e0, e1);
      }
#pragma unroll
      for (int w2 = 8; w2 > 0; w2 >>= 1)
#pragma unroll
        for (int j = 0; j < w2; ++j) sm[j] += sm[j + w2];
      l_sum = l_sum * alpha + sm[0];
      // probabilities (bf16 pairs) replace the partial scores in this tile's TMEM
      // buffer once the sender warps have read them; P.V takes them from there
      if (!wait_warp(&bars[kBarSpFree + bb], (i >> 1) & 1)) { fail(); break; }
      tc_fence_after();
      tmem_st16(lane_base + kColS + kNt * bb, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
      tmem_st16(lane_base + kColS + kNt * bb + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
      // O may be rescaled once P.V of the previous tile has completed
      if (i >= 1) {
        if (!wait_warp(&bars[kBarPvDone], (i - 1) & 1)) { fail(); break; }
        tc_fence_after();
      }
      // rescale this warp's O rows if any of its heads' reference max moved
      if (i >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c16 = 0; c16 < 256 / 16; ++c16) {
          uint32_t v[16];
          tmem_ld16(lane_base + kColO + 16 * c16, v);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
          tmem_st16(lane_base + kColO + 16 * c16, v);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[kBarOReady + bb]);
    }

    // A softmax warp that gave up may leave the peer's copies of one more tile in
    // flight into X (the peer sends tile j once we have read tile j-1): let them land,
    // for at most a few milliseconds, before this CTA can exit.
    if (*abort_s && warp == 0 && lane == 0 && x_seen < n_tiles)
      (void)mbar_wait<true>(&bars[kBarXFull], x_seen & 1, kDrainLimit, kDrainCapNs);

    // ---- epilogue: out = O / l for this CTA's 256 columns; lse from CTA 0 --------
    // The normalised rows are staged in the (idle) gather stages as eight SW128 boxes
    // of 32 columns and written by TMA, one 16 KB box per store.  Every softmax warp
    // reaches the named barrier, whatever happened before; the stores are issued only
    // when no wait of this CTA gave up.
    const bool aborted = *abort_s;
    bool have_o = false;
    if (n_tiles > 0 && !aborted) {
      // a dedicated one-phase barrier: pv_done may still be two phases behind here
      have_o = wait_warp(&bars[kBarPvFinal], 0);
      if (!have_o) fail();
    }
    if (have_o || n_tiles == 0) {
      tc_fence_after();
      const float inv = n_tiles > 0 ? 1.f / l_sum : 0.f;
#pragma unroll 1
      for (int c64 = 0; c64 < 256 / 64; ++c64) {   // 64 columns per round: four TMEM loads in flight
        uint32_t v[4][16];
        if (n_tiles > 0) {
#pragma unroll
          for (int u = 0; u < 4; ++u) tmem_ld16(lane_base + kColO + 64 * c64 + 16 * u, v[u]);
          tmem_ld_wait();
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c16 = 4 * c64 + u;
          char* box = smem + (c16 >> 1) * kOutBox + head * 128;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int ch = 4 * (c16 & 1) + k;
            const float4 o = n_tiles > 0 ? make_float4(__uint_as_float(v[u][4 * k]) * inv, __uint_as_float(v[u][4 * k + 1]) * inv,
                                                       __uint_as_float(v[u][4 * k + 2]) * inv, __uint_as_float(v[u][4 * k + 3]) * inv)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(box + ((ch ^ (head & 7)) * 16)) = o;
          }
        }
      }
      if (crank == 0 && head_ok)
        p.lse[((size_t)r * T + t) * p.h + head] = n_tiles > 0 ? (m_ref + __log2f(l_sum)) * kLn2 : -INFINITY;
      fence_proxy_async_smem();
    }
    named_barrier(2, 128);
    if (warp == 0 && lane == 0 && !*abort_s) {
      for (int b = 0; b < 8; ++b) tma_store_3d(&tmap_out, smem_u32(smem + b * kOutBox), 256 * crank + 32 * b, 0, r * T + t);
      bulk_commit_group();
      bulk_wait_read<0>();   // shared memory may be released once read; the writes finish with the grid
    }
    __syncwarp();
  } else if (warp < kProducerWarp + kProducerWarps) {
    // =================== gathers ===================================================
    // Producer warp pw issues the gathers of row groups g = pw, pw+4, .. (4 rows each)
    // of every tile, twenty per tile, one per lane in a single instruction: issue from
    // several warps and several lanes keeps the gather engine busiest.
    const int pw = warp - kProducerWarp;
    int seg = 0;   // which kListCap-row segment of the resolved list is in list_s
    int n = 0;
    bool ok = true;
    for (; n < n_tiles && !*abort_s; ++n) {
      const int s = n % kStages;
      if (n >= kStages && !(ok = wait_warp(&bars[kBarKvEmpty + s], ((n / kStages) - 1) & 1))) break;
      const int first = kNt * n;
      if (first >= (seg + 1) * kListCap) {
        // rare (more than kListCap valid entries): this warp re-resolves the entries of
        // its own row groups for the next segment (disjoint writes, no cross-warp sync)
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
      // one gather per lane: lane l takes column block l % 5 (four latent blocks, then
      // the rope block) of the warp's row group l / 5, so the warp issues its twenty
      // gathers of the tile as one instruction
      char* st = smem + s * kStageBytes;
      if (lane == 0) mbar_arrive_expect_tx(&bars[kBarKvFull + s], kStageTx / kProducerWarps);
      __syncwarp();
      constexpr int kGroupsPerWarp = kNt / 4 / kProducerWarps;
      if (lane < 5 * kGroupsPerWarp) {
        const int g = pw + kProducerWarps * (lane / 5), j = lane % 5;
        int rr[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int e = first + 4 * g + k;
          rr[k] = e < total ? list_s[e - seg * kListCap] : tp.num_rows;   // past the end: zero fill
        }
        if (j < 4)
          tma_gather4(smem_u32(st + j * kLatBlk + g * 4 * 128), &tmap_lat, 256 * crank + 64 * j, rr[0], rr[1], rr[2],
                      rr[3], &bars[kBarKvFull + s]);
        else
          tma_gather4(smem_u32(st + 4 * kLatBlk + g * 4 * 64), &tmap_rope, 512 + 32 * crank, rr[0], rr[1], rr[2], rr[3],
                      &bars[kBarKvFull + s]);
      }
      __syncwarp();
    }
    if (!ok) fail();
    // no gather of this CTA may still be landing in shared memory at exit
    for (int k = n > kStages ? n - kStages : 0; k < n; ++k)
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarKvFull + k % kStages], (k / kStages) & 1, kDrainLimit)))
        report_status(p.status, kStatusTimeout);
  } else if (warp >= kSendWarp) {
    // =================== partial-score senders =====================================
    // Sender warp w serves TMEM lane quadrant w % 4 (heads 32(w%4) .. +31): for every
    // tile it loads our partial scores from the TMEM score buffer, stages them (lane l
    // in the slot of heads 16(l/16) .. +15) and copies each slot holding real heads into
    // the peer's X buffer as soon as QK^T is done.
    const int qd = warp & 3;
    const int head = qd * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
    char* xout_warp = smem + kOffXStage + qd * kXWarpBytes;
    char* xout = xout_warp + lane * 256;   // this lane's staging row
    const uint32_t xdst_warp = mapa(smem + kOffX + qd * kXWarpBytes, peer);
    const uint32_t xfull_peer = mapa(&bars[kBarXFull], peer);
    const int n_half = min(2, max(0, (p.h - 32 * qd + 15) / 16));   // this warp's 16-head slots with real heads
    // the staging rows held q until the softmax warps moved it into TMEM
    bool ok = n_tiles == 0 || wait_warp(&bars[kBarQReady], 0);
    for (int j = 0; ok && j < n_tiles && !*abort_s; ++j) {
      const int bj = j & 1;
      if (!(ok = wait_warp(&bars[kBarSFull + bj], (j >> 1) & 1))) break;
      tc_fence_after();
      uint32_t v[4][16];
#pragma unroll
      for (int c4 = 0; c4 < kNt / 16; ++c4) tmem_ld16(lane_base + kColS + kNt * bj + 16 * c4, v[c4]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarSpFree + bj]);   // the softmax may overwrite the buffer with P
      if (n_half == 0) continue;   // only padding heads in this quadrant
      // The peer has read tile j-1 from its X buffer (phase 0: moved its q out of it), so
      // every copy of tile j-1 has landed there and has read its source slot.
      if (!(ok = wait_warp_cluster(&bars[kBarXFree], j & 1))) break;
      if ((lane >> 4) < n_half) {
#pragma unroll
        for (int k = 0; k < 16; ++k)
          *reinterpret_cast<uint4*>(xout + ((k ^ (head & 15)) * 16)) =
              make_uint4(v[k >> 2][4 * (k & 3)], v[k >> 2][4 * (k & 3) + 1], v[k >> 2][4 * (k & 3) + 2],
                         v[k >> 2][4 * (k & 3) + 3]);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0)
        for (int hh = 0; hh < n_half; ++hh)
          bulk_copy_s2cluster(xdst_warp + hh * kXHalfBytes, xout_warp + hh * kXHalfBytes, kXHalfBytes, xfull_peer);
      __syncwarp();
    }
    if (!ok) fail();
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // =================== tcgen05 MMA issue: QK^T (warp 8) and P.V (warp 9) ========
    if (lane == 0 && n_tiles > 0) {
      bool ok = true;
      if (warp == kMmaWarp) {
        // test hook: a wait that cannot complete, so the wait limit runs out
        ok = !p.stall || mbar_wait(&bars[kBarNever], 0, wl);
        ok = ok && mbar_wait(&bars[kBarQReady], 0, wl);
        tc_fence_after();
        const uint32_t id_qk = idesc_bf16(128, kNt, 0, 0);
        const uint32_t qrope_a = smem_u32(qrope);
        for (int n = 0; ok && n < n_tiles && !*abort_s; ++n) {
          const int s = n % kStages, bb = n & 1;
          if (!(ok = mbar_wait(&bars[kBarKvFull + s], (n / kStages) & 1, wl))) break;
          // the score buffer is free once P.V has read tile n-2's probabilities from it
          if (n >= 2 && !(ok = mbar_wait(&bars[kBarSFree + bb], ((n >> 1) - 1) & 1, wl))) break;
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * kStageBytes);
          const uint32_t d = tmem + kColS + kNt * bb;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            mma_ts(d, tmem + kColQ + 8 * k,
                   smem_desc(st + (k >> 2) * kLatBlk + (k & 3) * 32, 16, 1024, kSwizzle128), id_qk, k > 0);
#pragma unroll
          for (int k = 0; k < 2; ++k)
            mma_ss(d, smem_desc(qrope_a + 32 * k, 16, 512, kSwizzle64),
                   smem_desc(st + 4 * kLatBlk + 32 * k, 16, 512, kSwizzle64), id_qk, 1);
          mma_commit(&bars[kBarSFull + bb]);
        }
      } else {
        const uint32_t id_pv = idesc_bf16(128, 256, 0, 1);
        for (int n = 0; ok && n < n_tiles && !*abort_s; ++n) {
          const int s = n % kStages, bb = n & 1;
          if (!(ok = mbar_wait(&bars[kBarOReady + bb], (n >> 1) & 1, wl))) break;
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * kStageBytes);
          // A = P [128 heads x 64 rows] bf16 pairs in TMEM, 16 rows (8 columns) per step
#pragma unroll
          for (int k = 0; k < kNt / 16; ++k)
            mma_ts(tmem + kColO, tmem + kColS + kNt * bb + 8 * k,
                   smem_desc(st + 2048 * k, kLatBlk, 1024, kSwizzle128), id_pv, (n > 0 || k > 0) ? 1u : 0u);
          mma_commit(&bars[kBarKvEmpty + s]);
          mma_commit(&bars[kBarSFree + bb]);
          mma_commit(&bars[kBarPvDone]);
          if (n == n_tiles - 1) mma_commit(&bars[kBarPvFinal]);
        }
      }
      if (!ok) fail();
      // every MMA this thread issued has completed before TMEM is released
      uint64_t* fin_bar = &bars[warp == kMmaWarp ? kBarMmaFin : kBarMmaFin2];
      mma_commit(fin_bar);
      if (!mbar_wait(fin_bar, 0, kDrainLimit)) report_status(p.status, kStatusTimeout);
    }
  }

  // ---- teardown: all DSMEM traffic of both CTAs is over before either exits -----
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Encoded tensor maps, remembered per host thread: a serving loop passes the same cache,
// staging and output buffers every step, so encoding happens once per buffer layout.
struct MapKey {
  uint64_t f[14];
  bool operator==(const MapKey& o) const { return memcmp(f, o.f, sizeof f) == 0; }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};
constexpr int kMapCache = 32;
thread_local MapEntry t_maps[kMapCache];
thread_local int t_maps_next = 0;

bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw, CUtensorMapL2promotion l2) {
  MapKey k;
  memset(&k, 0, sizeof k);
  k.f[0] = (uint64_t)dt | ((uint64_t)rank << 8) | ((uint64_t)sw << 16) | ((uint64_t)l2 << 24);
  k.f[1] = reinterpret_cast<uint64_t>(base);
  for (int i = 0; i < rank; ++i) {
    k.f[2 + i] = dims[i];
    k.f[5 + i] = box[i];
    if (i + 1 < rank) k.f[8 + i] = strides[i];
  }
  for (int e = 0; e < kMapCache; ++e)
    if (t_maps[e].used && t_maps[e].key == k) {
      *m = t_maps[e].map;
      return true;
    }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  if (fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
         l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  MapEntry& slot = t_maps[t_maps_next];
  t_maps_next = (t_maps_next + 1) % kMapCache;
  slot.key = k;
  slot.map = *m;
  slot.used = true;
  return true;
}

// q [T, h, 576] as a 3D tensor (columns, heads, tokens); one box = box_cols columns of
// q_rows heads of one token
bool make_q_map(CUtensorMap* m, const void* q, int h, long long T, int q_rows, int box_cols, CUtensorMapSwizzle sw) {
  cuuint64_t dims[3] = {(cuuint64_t)kDQK, (cuuint64_t)h, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)kDQK * 2, (cuuint64_t)h * kDQK * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)q_rows, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

// out [n_tok, h, 512] fp32 as a 3D tensor; one box = 32 columns of q_rows heads of one token
bool make_out_map(CUtensorMap* m, float* out, int h, long long n_tok, int q_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)kDV, (cuuint64_t)h, (cuuint64_t)n_tok};
  cuuint64_t strides[2] = {(cuuint64_t)kDV * 4, (cuuint64_t)h * kDV * 4};
  cuuint32_t box[3] = {32, (cuuint32_t)q_rows, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// the cache as [num_rows, 576] rows; one box = box_cols columns of one row (gathered four at a time)
bool make_row_map(CUtensorMap* m, const void* kv, int num_rows, int box_cols, CUtensorMapSwizzle sw) {
  cuuint64_t dims[2] = {(cuuint64_t)kDQK, (cuuint64_t)num_rows};
  cuuint64_t strides[1] = {(cuuint64_t)kDQK * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv, dims, strides, box, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

}  // namespace

bool tc_supports(int h, int block_size) {
  (void)block_size;
  return h >= 1 && h <= kHeads;
}

bool tc_supports_ptrs(const void* q, const void* kv, const void* out) {
  // tensor maps want 16-byte aligned base addresses
  return ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv) | reinterpret_cast<uintptr_t>(out)) & 15) == 0;
}

size_t tc_workspace_bytes(int T, int h, int top_k, int n_splits) {
  // only the stacked-half kernel uses scratch: its balanced schedule
  return stack_workspace_bytes((long long)T * n_splits, h, top_k, device_sm_count());
}

int tc_launches(int T, int h, int top_k, int n_splits) {
  (void)T; (void)h; (void)top_k; (void)n_splits;
  return 1;
}

cudaError_t prepare_decode_tc() {
  static std::atomic<bool> attr_set[64];   // per device: set once (a repeat is harmless)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    for (auto kernel : {decode_tc_kernel<false>, decode_tc_kernel<true>}) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
    }
    attr_set[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

cudaError_t launch_decode_tc(const DecodeParams& p, int kernel_id, cudaStream_t stream) {
  const long long T = (long long)p.B * p.Q;
  const long long units = T * p.n_splits;
  if (units == 0) return cudaSuccess;
  const long long num_rows = (long long)p.num_blocks * p.block_size;
  if (num_rows >= 0x7fffffffLL || 2 * units > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (kernel_id == 2 || kernel_id == 3) {
    // whole rows as nine 64-column SW128 boxes from one map; q's rope columns as one box
    CUtensorMap rows, qrope;
    // (the stacked-half kernel loads q's rope rows 16 heads at a time)
    const bool ok_h = kernel_id == 2 ? narrow_supports(p.h) : stack_supports(p.h);
    if (!ok_h || !make_row_map(&rows, p.kv, (int)num_rows, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_q_map(&qrope, p.q, p.h, T, kernel_id == 2 ? p.h : 16, 64, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (kernel_id == 2) return launch_decode_narrow(p, rows, qrope, stream);
    CUtensorMap omap;
    if (!make_out_map(&omap, p.out, p.h, T * p.n_splits, p.h)) return cudaErrorInvalidValue;
    return launch_decode_stack(p, rows, qrope, omap, device_sm_count(), stream);
  }
  TcParams tp;
  tp.p = p;
  tp.num_rows = (int)num_rows;
  tp.q_rows = p.h < kHeads ? p.h : kHeads;
  CUtensorMap lat, rope, qlat, qrope, omap;
  if (!make_row_map(&lat, p.kv, (int)num_rows, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_row_map(&rope, p.kv, (int)num_rows, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_q_map(&qlat, p.q, p.h, T, tp.q_rows, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_q_map(&qrope, p.q, p.h, T, tp.q_rows, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_out_map(&omap, p.out, p.h, T * p.n_splits, tp.q_rows))
    return cudaErrorInvalidValue;
  const bool il = p.interleave > 0 && p.n_splits > 1;
  auto kernel = il ? decode_tc_kernel<true> : decode_tc_kernel<false>;
  cudaError_t e = prepare_decode_tc();
  if (e != cudaSuccess) return e;
  kernel<<<(unsigned)(2 * units), kThreads, kSmemBytes, stream>>>(lat, rope, qlat, qrope, omap, tp);
  return cudaGetLastError();
}

}  // namespace sfa
