// sfa_topk.cu -- indexer top-k selection: for each query token, the k cache positions
// with the largest indexer scores, i.e. the list that sparse attention then visits
// ("vllm-ascend PR #18870 解读", 4.5: only the top-2048 positions the indexer chose are
// attended, not the whole history).
//
// Order: IEEE 754 totalOrder of the fp32 scores, larger first; equal scores are taken
// lower position first.  Output: the chosen positions in ascending order, then -1.
//
// One cluster of C CTAs (C = 1..8, C = 1 for rows of up to 32K positions) of 512 threads
// per query token; CTA r of the cluster takes the contiguous chunk [r*chunk, (r+1)*chunk) of
// the token's candidate range, as 32-bit keys whose unsigned order is the totalOrder of
// the scores.  Two ways to the same list:
//
// Sampled threshold (tried first).  Each CTA copies its chunk to shared memory (cp.async,
// no registers held) and, from two scores per thread of the first copies to land,
// estimates a key threshold tau below which the k-th largest key of the row almost surely
// does not lie.  Each lane then lists, in position order, the keys of its own contiguous
// run that reach tau (one compare a key on the raw bits; a warp scan orders the lanes).
// After one cluster barrier every CTA copies all the lists into one array (16-byte
// distributed-shared-memory reads), checks that at least k of the keys reach the largest
// threshold of the cluster (else the estimate was too high, and the cluster runs the sweep
// below), and finds the k-th largest key in that array by radix passes whose 13-bit digits
// span only the keys' actual range (one or two passes for typical scores).  Each CTA then
// writes its own chosen positions.
//
// Sweep (the fallback).  Each CTA stages its chunk in shared memory:
//   * Radix select in three passes (11, 11 and 10 key bits from the top).  Pass 0 counts
//     every key into a shared-memory histogram; the keys that fall in the chosen bin are
//     then copied to a short candidate list, which passes 1 and 2 scan instead of the
//     whole chunk.  With C > 1 the cluster sums each pass's histograms over distributed
//     shared memory, and every CTA finds the same bin.  A pass whose bin must be taken
//     whole ends the search early.
//   * Ordered compaction: each warp owns a contiguous run of the chunk; ballots give the
//     order within a warp, a block scan of the warps' (above, equal) counts and the
//     totals of lower-ranked CTAs give each warp its base, so every chosen position
//     knows its output index and the list comes out sorted without a sort.
// No wait in this kernel spins: the only synchronisation is block and cluster barriers.
#include <atomic>
#include "sfa_internal.h"
#include "sfa_ptx.cuh"

namespace sfa {
namespace {

using namespace ptx;

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kMaxBins = 2048;
constexpr int kPasses = 3;
constexpr int kCandCap = 8192;                // candidates kept after pass 0 (32 KB)
constexpr int kCandPerWarp = kCandCap / kTkWarps;
constexpr int kChunkUnit = 128 * kTkWarps;    // chunks are whole 128-key steps of every warp
static_assert(kTopkChunkMax % kChunkUnit == 0, "a chunk splits into whole warp runs");
static_assert(kMaxBins / kTkThreads == 2 || kMaxBins / kTkThreads == 4,
              "sweep bins: 2 or 4 a thread in an 11-bit pass, half that in the 10-bit one");
// sampled threshold: 13-bit digits; a warp sums a slice of kSlice bins
constexpr int kDigitBits = 13;
constexpr int kDigitBins = 1 << kDigitBits;
constexpr int kSlice = kDigitBins / kTkWarps;
constexpr int kBinsPerLane = kSlice / 32;
constexpr int kMaxSteps = kTopkChunkMax / kTkWarps / 128;   // 16-byte copies a thread
static_assert(kBinsPerLane == 8 || kBinsPerLane == 16, "a lane's bins are 2 or 4 16-byte vectors");
static_assert(kPasses * kMaxBins <= kDigitBins, "the sweep's histograms fit the sampled path's");

// dynamic shared memory: keys | candidate keys | candidate positions | histograms
// (the sampled path stages the chunk's raw score bits in the key area and then gathers the
// cluster's candidate keys there; its histogram area is one 8192-bin histogram, zeroed
// again after each use; the sweep's, three 2048-bin histograms)
__host__ __device__ constexpr int kOffCand(int chunk) { return chunk * 4; }
__host__ __device__ constexpr int kOffCpos(int chunk) { return chunk * 4 + kCandCap * 4; }
__host__ __device__ constexpr int kOffHist(int chunk) { return chunk * 4 + 2 * kCandCap * 4; }
__host__ __device__ constexpr int topk_smem_bytes(int chunk) { return kOffHist(chunk) + kDigitBins * 4; }

struct TopkParams {
  const float* scores;
  long long row_stride;
  const int32_t* seq_lens;
  int Q, S, k, chunk;
  int32_t* out;
};

// unsigned order of the keys == IEEE 754 totalOrder of the floats (the usual radix-sort
// key for floats: negatives have every bit flipped, non-negatives only the sign bit)
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void ld_cluster_v2(uint32_t addr, uint32_t& a, uint32_t& b) {
  asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr) : "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ int pass_width(int pass) { return pass < 2 ? 11 : 10; }

// Exclusive warp scan of one value per lane; also returns the warp's total.
__device__ __forceinline__ uint32_t warp_exclusive_scan(uint32_t v, uint32_t& total) {
  const int lane = threadIdx.x & 31;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  total = __shfl_sync(0xffffffffu, inc, 31);
  return inc - v;
}

// Exclusive block scan of one value per thread (in thread order); also returns the total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* wsum, uint32_t& total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t x = lane < kTkWarps ? wsum[lane] : 0u;
    uint32_t y = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += n;
    }
    if (lane < kTkWarps) wsum[lane] = y - x;
    if (lane == 31) wsum[32] = y;
  }
  __syncthreads();
  total = wsum[32];
  const uint32_t r = wsum[warp] + inc - v;
  __syncthreads();   // wsum is reused by the next scan
  return r;
}

// 16-byte global -> shared copy through L2 (cp.async): `bytes` (0..16) read, the rest zeroed
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(__cvta_generic_to_global(gsrc)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Block-shared state of both paths.  Static shared memory has the same offsets in every
// CTA, so the cluster reads its peers' fields through mapa.
struct TkShared {
  uint4 meta;                            // sampled path: (tau, some list overflowed, candidates, 0)
  uint2 wcp[kTkWarps];                   // sampled path: (candidates, those of lower warps) a warp
  uint32_t wsum[33];                     // block scan scratch
  uint32_t wg[kTkWarps], we[kTkWarps];   // per-warp (above, equal) counts
  uint32_t sel[3];                       // chosen bin, keys still needed, keys in the bin
  uint32_t wcand[kTkWarps];              // sweep: candidates each warp listed
  uint32_t ncand_over;                   // some warp listed more than it keeps
  uint32_t cta_tot[2];                   // sweep: this CTA's (above, equal) totals
  uint32_t kmax;                         // sampled path: largest candidate key of the cluster
  uint32_t lower[2];                     // sampled path: (above, within) keys of lower CTAs
};

// The token and chunk one CTA serves.
struct TkRow {
  uint32_t C, cr;   // CTAs per token, this CTA's rank
  int t, L;         // token, causal length of its row
  int lo, n_here;   // chunk start, valid keys of the chunk
};

// Where bin b of the sampled path's histogram lives: thread t reads its kBinsPerLane bins as
// V = kBinsPerLane / 4 16-byte vectors, and the XOR of the vector slot (b >> 2) % V with
// (b >> 5) % V spreads the 8 lanes of each 16-byte access phase over all 32 banks
// (unswizzled, those lanes' vectors sit 16 * V bytes apart and share 8 / V bank groups).
constexpr uint32_t kVecMask = kBinsPerLane / 4 - 1;
__device__ __forceinline__ uint32_t hslot(uint32_t b) { return b ^ (((b >> 5) & kVecMask) << 2); }

// Over the kDigitBins-bin histogram, find the bin at which the count from the top bin down
// first reaches `need` (1 <= need): thread t holds bins [kBinsPerLane*t, kBinsPerLane*(t+1))
// and warp w the slice [kSlice*w, kSlice*(w+1)).  Every warp learns the slice totals through
// one barrier and the count above its own slice with one reduction; the warp whose slice
// holds the crossing finds the thread (a suffix scan) and that thread the bin, recording
// (bin, need left within it, its count) in sel.  sel[0] = ~0 when the total is below need.
// Each thread zeroes its bins once it holds them, so the histogram is clear for the next
// count when this returns.  Returns the histogram's total.  Two barriers; sel is readable on
// return; wsum is reused, so the caller puts a barrier between this call's return and the
// next call.
__device__ __forceinline__ uint32_t find_from_top(uint32_t* hist, uint32_t need, uint32_t* wsum,
                                                  uint32_t* sel) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t c[kBinsPerLane];   // this thread's bins, ascending
  // logical vector v sits in physical slot v ^ (hslot's XOR for this thread's bins)
  const int vx = (int)(((uint32_t)(kBinsPerLane * tid) >> 5) & kVecMask);
#pragma unroll
  for (int v = 0; v < kBinsPerLane / 4; ++v) {
    uint4* h4 = reinterpret_cast<uint4*>(hist + kBinsPerLane * tid + 4 * (v ^ vx));
    const uint4 x = *h4;
    *h4 = make_uint4(0u, 0u, 0u, 0u);
    c[4 * v] = x.x;
    c[4 * v + 1] = x.y;
    c[4 * v + 2] = x.z;
    c[4 * v + 3] = x.w;
  }
  uint32_t ts = 0u;
#pragma unroll
  for (int q = 0; q < kBinsPerLane; ++q) ts += c[q];
  const uint32_t ws = __reduce_add_sync(0xffffffffu, ts);
  if (lane == 0) wsum[warp] = ws;
  __syncthreads();
  const uint32_t x = lane < kTkWarps ? wsum[lane] : 0u;
  const uint32_t total = __reduce_add_sync(0xffffffffu, x);
  const uint32_t above = __reduce_add_sync(0xffffffffu, lane > warp ? x : 0u);   // higher slices
  if (tid == 0 && need > total) sel[0] = ~0u;
  if (above < need && need <= above + ws) {
    // suffix sums within the warp: keys in this lane's bins and those of higher lanes
    uint32_t suf = ts;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += n;
    }
    if (above + suf - ts < need && need <= above + suf) {
      uint32_t acc = above + suf - ts;   // keys above this thread's top bin
#pragma unroll
      for (int q = kBinsPerLane - 1; q >= 0; --q) {
        if (acc < need && need <= acc + c[q]) {
          sel[0] = (uint32_t)(kBinsPerLane * tid + q);
          sel[1] = need - acc;
          sel[2] = c[q];
        }
        acc += c[q];
      }
    }
  }
  __syncthreads();
  return total;
}

__device__ __forceinline__ void zero_hist(uint32_t* hist) {
#pragma unroll
  for (int x = 4 * (int)threadIdx.x; x < kDigitBins; x += 4 * kTkThreads)
    *reinterpret_cast<uint4*>(hist + x) = make_uint4(0u, 0u, 0u, 0u);
}

// Where the staged copy of 16-byte block b of a warp's run lives (in 16-byte blocks from the
// run's start): XOR of the block's low 3 bits with the next 3.  The copies (lane l of step u
// writes block 32u + l) and the listing's reads (lane L reads blocks L*G .. L*G+G-1, G
// blocks a lane) then spread each 8-lane access phase over all 32 banks (2 ways for G = 16).
__device__ __forceinline__ int stage_slot(int b) { return b ^ ((b >> 3) & 7); }

// List, in position order, the staged keys of one warp's run that pass (kSigned ? (int)b >=
// (int)thr : b <= thr) -- the form order_key(b) >= tau takes for tau at or above
// order_key(+0) (thr = tau ^ 0x80000000) and below it (thr = ~tau).  Lane L holds the 4G
// contiguous keys of blocks L*G .. L*G+G-1 (positions pos0 + 0 .. 4G-1), of which the first
// nv are in the chunk; a warp scan of the lanes' counts orders the lists.  Keeps the first
// kCandPerWarp as (raw bits, position); returns how many pass.
template <bool kSigned>
__device__ __forceinline__ uint32_t list_run(const uint32_t* run, int G, int nv, uint32_t thr, uint32_t pos0,
                                             uint32_t* my_cand, uint32_t* my_cpos) {
  const int lane = threadIdx.x & 31;
  static_assert(kMaxSteps <= 16, "a lane's keys fit two 32-bit masks");
  uint32_t m[2] = {0u, 0u};   // bit k: the lane's key k passes
#pragma unroll
  for (int v = 0; v < kMaxSteps; ++v) {
    if (v < G) {
      const uint4 b = *reinterpret_cast<const uint4*>(run + 4 * stage_slot(lane * G + v));
      uint32_t mk;
      if (kSigned)
        mk = ((int)b.x >= (int)thr ? 1u : 0u) | ((int)b.y >= (int)thr ? 2u : 0u) |
             ((int)b.z >= (int)thr ? 4u : 0u) | ((int)b.w >= (int)thr ? 8u : 0u);
      else
        mk = (b.x <= thr ? 1u : 0u) | (b.y <= thr ? 2u : 0u) | (b.z <= thr ? 4u : 0u) | (b.w <= thr ? 8u : 0u);
      m[v >> 3] |= mk << (4 * (v & 7));
    }
  }
  if (nv < 32) {   // keys from nv on lie past the chunk's valid end
    m[0] &= nv > 0 ? (1u << nv) - 1u : 0u;
    m[1] = 0u;
  } else if (nv < 64) {
    m[1] &= (1u << (nv - 32)) - 1u;
  }
  uint32_t tot;
  uint32_t o = warp_exclusive_scan((uint32_t)(__popc(m[0]) + __popc(m[1])), tot);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t mm = m[h];
    while (mm) {
      const int k = 32 * h + __ffs(mm) - 1;
      mm &= mm - 1u;
      if (o < (uint32_t)kCandPerWarp) {
        my_cand[o] = run[4 * stage_slot(lane * G + (k >> 2)) + (k & 3)];
        my_cpos[o] = pos0 + (uint32_t)k;
      }
      ++o;
    }
  }
  return tot;
}

// The sampled-threshold path.  Returns true with this CTA's share of the token's list
// written; false, the same in every CTA of the cluster, when the cluster has to run the
// sweep.  Either way the CTA has arrived on a cluster barrier (C > 1) that the caller
// waits on: with false, before the sweep reuses the lists that peers read.
__device__ __forceinline__ bool sampled_select(const TopkParams& p, const TkRow& r, TkShared& sh) {
  extern __shared__ __align__(16) uint32_t tk_smem[];
  uint32_t* kbuf = tk_smem;   // the chunk's raw score bits, then every CTA's candidate keys
  // cand / cpos: warp w's list (raw score bits, position) in its kCandPerWarp slot
  uint32_t* cand = tk_smem + kOffCand(p.chunk) / 4;
  uint32_t* cpos = tk_smem + kOffCpos(p.chunk) / 4;
  uint32_t* hist = tk_smem + kOffHist(p.chunk) / 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = p.chunk / kTkWarps;               // warp w's run: keys [w*seg, (w+1)*seg)
  const int w0 = warp * seg, w1 = min(w0 + seg, r.n_here);
  const int steps = (seg + 127) / 128;
  uint32_t* my_cand = cand + warp * kCandPerWarp;
  uint32_t* my_cpos = cpos + warp * kCandPerWarp;

  // ---- stage the run: step u, lane l copies block 32u + l (keys w0 + 128u + 4l + 0..3) to
  // its stage_slot; step 0 is a group of its own, so the sample can go ahead while the rest
  // is in flight
  {
    const float* wrow = p.scores + (size_t)r.t * p.row_stride + r.lo + w0;
#pragma unroll
    for (int u = 0; u < kMaxSteps; ++u) {
      const int j = 128 * u + 4 * lane, rem = w1 - (w0 + j);
      if (u < steps && rem > 0)
        cp_async16(kbuf + w0 + 4 * stage_slot(32 * u + lane), wrow + j, rem >= 4 ? 16u : 4u * (uint32_t)rem);
      if (u == 0) cp_async_commit();
    }
    cp_async_commit();
  }
  zero_hist(hist);
  if (tid == 0) {
    sh.ncand_over = 0u;
    sh.kmax = 0u;
    sh.lower[0] = sh.lower[1] = 0u;
  }
  __syncthreads();

  // Of n_s iid samples, about n_s*k/L reach the row's k-th largest key.  tau is the lower
  // edge of the bin holding the m-th largest sample, m = that mean x 1.25 + 3 standard
  // deviations + 4, so that tau lies above the k-th largest key only for rows whose
  // chunks differ in distribution (the cluster then runs the sweep).  With fewer than m
  // samples, tau = 0: every key is a candidate.  n_s counts the samples taken below: keys
  // 0 and 2 of each lane's first copy that lie in the chunk.
  uint32_t m;
  {
    const int len = lane < kTkWarps ? max(0, min(seg, r.n_here - lane * seg)) : 0;   // warp `lane`'s run
    const int n_s = (int)__reduce_add_sync(0xffffffffu, (uint32_t)(min(32, (len + 3) / 4) + min(32, (len + 1) / 4)));
    const float mean = (float)n_s * __fdividef((float)p.k, (float)r.L);
    m = (uint32_t)ceilf(1.25f * mean + 3.f * (mean > 0.f ? mean * rsqrtf(mean) : 0.f) + 4.f);
  }

  // ---- the threshold, from keys 0 and 2 of each thread's first copy (13-bit digits: bins
  // of 2^19 keys)
  cp_async_wait<1>();
  {
    const uint32_t* blk = kbuf + w0 + 4 * stage_slot(lane);   // this lane's own step-0 copy
    if (w0 + 4 * lane < w1) atomicAdd(&hist[hslot(order_key(blk[0]) >> (32 - kDigitBits))], 1u);
    if (w0 + 4 * lane + 2 < w1) atomicAdd(&hist[hslot(order_key(blk[2]) >> (32 - kDigitBits))], 1u);
  }
  __syncthreads();
  find_from_top(hist, m, sh.wsum, sh.sel);   // leaves the histogram zeroed for the select
  const uint32_t tau = sh.sel[0] == ~0u ? 0u : sh.sel[0] << (32 - kDigitBits);

  // ---- list the keys at or above tau in position order, one compare a key on the raw
  // bits: for tau >= order_key(+0) no negative score passes and a non-negative one passes
  // when its bits, as a signed int, reach tau's bits under the sign; below it every
  // non-negative score passes and a negative one when its bits, unsigned, are <= ~tau.
  cp_async_wait<0>();
  __syncwarp();   // the listing reads the whole warp's copies
  uint32_t n_w;
  {
    const int nv = w1 - (w0 + 4 * steps * lane);   // the lane's keys in the chunk (may be <= 0)
    const uint32_t pos0 = (uint32_t)(r.lo + w0 + 4 * steps * lane);
    if (tau >= 0x80000000u)
      n_w = list_run<true>(kbuf + w0, steps, nv, tau ^ 0x80000000u, pos0, my_cand, my_cpos);
    else
      n_w = list_run<false>(kbuf + w0, steps, nv, ~tau, pos0, my_cand, my_cpos);
  }
  if (lane == 0) {
    sh.wcp[warp].x = n_w;
    if (n_w > (uint32_t)kCandPerWarp) sh.ncand_over = 1u;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t tot;
    const uint32_t ex = warp_exclusive_scan(lane < kTkWarps ? sh.wcp[lane].x : 0u, tot);
    if (lane < kTkWarps) sh.wcp[lane].y = ex;
    if (lane == 0) sh.meta = make_uint4(tau, sh.ncand_over, tot, 0u);
  }
  if (r.C > 1) cluster_sync(); else __syncthreads();   // every CTA's lists and counts are out

  // ---- the cluster's view: lane q of each warp reads CTA q's summary and this warp's slot
  uint4 mq = make_uint4(0u, 0u, 0u, 0u);
  uint4 cq = make_uint4(0u, 0u, 0u, 0u);
  if (lane < (int)r.C) {
    mq = ld_cluster_v4(mapa(&sh.meta, (uint32_t)lane));
    ld_cluster_v2(mapa(&sh.wcp[warp], (uint32_t)lane), cq.x, cq.y);
  }
  const uint32_t tau_max = __reduce_max_sync(0xffffffffu, mq.x);
  const uint32_t over = __reduce_or_sync(0xffffffffu, mq.y);
  uint32_t n_tot;
  const uint32_t off_q = warp_exclusive_scan(mq.z, n_tot);   // where CTA `lane`'s keys go
  const uint32_t off_me = __shfl_sync(0xffffffffu, off_q, (int)r.cr);
  if (over || n_tot > (uint32_t)p.chunk) {   // a list overflowed, or they do not fit kbuf
    if (r.C > 1) cluster_arrive();
    return false;
  }

  // ---- every CTA's keys into kbuf, in rank order; warp w copies warp w's list of each CTA
  {
    uint32_t lmax = 0u;
    for (int q = 0; q < (int)r.C; ++q) {
      const uint32_t cnt = __shfl_sync(0xffffffffu, cq.x, q);
      uint32_t* dst = kbuf + __shfl_sync(0xffffffffu, off_q, q) + __shfl_sync(0xffffffffu, cq.y, q);
      if (q == (int)r.cr) {
        for (uint32_t i = lane; i < cnt; i += 32) {
          const uint32_t key = order_key(my_cand[i]);
          dst[i] = key;
          lmax = max(lmax, key);
        }
      } else {
        // 16-byte reads of the peer's slot; a slot holds kCandPerWarp (a multiple of 4) keys
        const uint32_t src = mapa(my_cand, (uint32_t)q);
        for (uint32_t i = 4 * lane; i < cnt; i += 128) {
          const uint4 kk = ld_cluster_v4(src + 4u * i);
          const uint32_t k4[4] = {order_key(kk.x), order_key(kk.y), order_key(kk.z), order_key(kk.w)};
#pragma unroll
          for (int x = 0; x < 4; ++x)
            if (i + x < cnt) {
              dst[i + x] = k4[x];
              lmax = max(lmax, k4[x]);
            }
        }
      }
    }
    lmax = __reduce_max_sync(0xffffffffu, lmax);
    if (lane == 0) atomicMax(&sh.kmax, lmax);
  }
  if (r.C > 1) cluster_arrive();   // this CTA's reads of its peers are done
  __syncthreads();

  // ---- the k-th largest of the keys at or above tau_max: radix passes over [base, hi]
  // with 13-bit digits of (key - base) >> s, s set by the range (<= 3 passes, 1-2 typical)
  uint32_t base = tau_max, hi = sh.kmax, krem = (uint32_t)p.k;
  if (hi < base) return false;   // no key reaches tau_max
  uint32_t lo_t = 0u, hi_t = 0u;   // keys above hi_t are chosen, and the first krem in [lo_t, hi_t]
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const uint32_t range = hi - base;
    const int nbits = range ? 32 - __clz((int)range) : 0;
    const int s = nbits > kDigitBits ? nbits - kDigitBits : 0;
    for (uint32_t i = 4 * tid; i < n_tot; i += 4 * kTkThreads) {   // kbuf is 16-byte aligned
      const uint4 k4 = *reinterpret_cast<const uint4*>(kbuf + i);
      const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
        if (i + x < n_tot && kk[x] >= base && kk[x] <= hi) atomicAdd(&hist[hslot((kk[x] - base) >> s)], 1u);
    }
    __syncthreads();
    // bins above (hi - base) >> s stay zero; the call leaves every bin zero for the next pass
    const uint32_t tot = find_from_top(hist, krem, sh.wsum, sh.sel);
    if (tot < krem) return false;   // pass 0 only: fewer than k keys reach tau_max
    const uint32_t bin = sh.sel[0], need = sh.sel[1], inbin = sh.sel[2];
    const uint32_t nbase = base + (bin << s);
    const uint32_t nhi = min(hi, nbase + ((1u << s) - 1u));
    krem = need;
    if (s == 0 || inbin == need) {   // one key value, or a bin taken whole
      lo_t = nbase;
      hi_t = nhi;
      break;
    }
    base = nbase;
    hi = nhi;
  }

  // ---- output: each warp's chosen positions at their ranks in the token's list
  {
    uint32_t g = 0u, e = 0u;   // keys of lower-ranked CTAs above hi_t / within [lo_t, hi_t]
    for (uint32_t i = 4 * tid; i < off_me; i += 4 * kTkThreads) {
      const uint4 k4 = *reinterpret_cast<const uint4*>(kbuf + i);
      const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        g += (i + x < off_me && kk[x] > hi_t) ? 1u : 0u;
        e += (i + x < off_me && kk[x] >= lo_t && kk[x] <= hi_t) ? 1u : 0u;
      }
    }
    g = __reduce_add_sync(0xffffffffu, g);
    e = __reduce_add_sync(0xffffffffu, e);
    if (lane == 0 && (g | e)) {
      atomicAdd(&sh.lower[0], g);
      atomicAdd(&sh.lower[1], e);
    }
  }
  const uint32_t nc = sh.wcp[warp].x;
  {
    uint32_t n_gt = 0u, n_eq = 0u;
    for (uint32_t i0 = 0; i0 < nc; i0 += 32) {
      const uint32_t i = i0 + lane;
      const uint32_t key = i < nc ? order_key(my_cand[i]) : 0u;
      n_gt += (uint32_t)__popc(__ballot_sync(0xffffffffu, i < nc && key > hi_t));
      n_eq += (uint32_t)__popc(__ballot_sync(0xffffffffu, i < nc && key >= lo_t && key <= hi_t));
    }
    if (lane == 0) {
      sh.wg[warp] = n_gt;
      sh.we[warp] = n_eq;
    }
  }
  __syncthreads();
  uint32_t g, q;
  {
    uint32_t tg, te;
    const uint32_t xg = warp_exclusive_scan(lane < kTkWarps ? sh.wg[lane] : 0u, tg);
    const uint32_t xe = warp_exclusive_scan(lane < kTkWarps ? sh.we[lane] : 0u, te);
    g = sh.lower[0] + __shfl_sync(0xffffffffu, xg, warp);
    q = sh.lower[1] + __shfl_sync(0xffffffffu, xe, warp);
  }
  int32_t* orow = p.out + (size_t)r.t * p.k;
  for (uint32_t i0 = 0; i0 < nc; i0 += 32) {
    const uint32_t i = i0 + lane;
    const uint32_t key = i < nc ? order_key(my_cand[i]) : 0u;
    const bool gsel = i < nc && key > hi_t;
    const bool e = i < nc && key >= lo_t && key <= hi_t;
    const unsigned mg = __ballot_sync(0xffffffffu, gsel), me = __ballot_sync(0xffffffffu, e);
    const uint32_t lt = lanemask_lt();
    const uint32_t gb = g + (uint32_t)__popc(mg & lt), eb = q + (uint32_t)__popc(me & lt);
    // the output index is below k by construction; the bound only keeps a fault out
    if (gsel) {
      const uint32_t o = gb + min(eb, krem);
      if (o < (uint32_t)p.k) orow[o] = (int32_t)my_cpos[i];
    } else if (e && eb < krem) {
      const uint32_t o = gb + eb;
      if (o < (uint32_t)p.k) orow[o] = (int32_t)my_cpos[i];
    }
    g += (uint32_t)__popc(mg);
    q += (uint32_t)__popc(me);
  }
  if (r.C > 1) cluster_wait();
  return true;
}

// The sweep: stage the whole chunk in shared memory, radix-select over it (or over the
// warps' candidate lists), then the ordered compaction.  Also serves take_all rows.
__device__ __forceinline__ void sweep_select(const TopkParams& p, const TkRow& row, const bool take_all,
                                             TkShared& sh) {
  extern __shared__ __align__(16) uint32_t tk_smem[];
  uint32_t* keys = tk_smem;
  uint32_t* cand = tk_smem + kOffCand(p.chunk) / 4;
  uint32_t* cpos = tk_smem + kOffCpos(p.chunk) / 4;
  uint32_t* hist = tk_smem + kOffHist(p.chunk) / 4;   // [kPasses][kMaxBins]
  uint32_t* wsum = sh.wsum;
  uint32_t* wg_s = sh.wg;
  uint32_t* we_s = sh.we;
  uint32_t* sel_s = sh.sel;
  uint32_t* wcand_s = sh.wcand;
  uint32_t& ncand_over_s = sh.ncand_over;
  uint32_t* cta_tot = sh.cta_tot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t C = row.C, cr = row.cr;
  const int t = row.t, L = row.L, lo = row.lo, n_here = row.n_here;

  for (int x = tid; x < kPasses * kMaxBins; x += kTkThreads) hist[x] = 0u;
  if (tid == 0) ncand_over_s = 0u;

  // ---- stage the chunk and count pass 0 --------------------------------------------
  // A chunk is at most 64 keys a thread: all of a thread's 16-byte loads are in flight
  // at once, and each key is counted into the pass-0 histogram (top 11 bits) as it is
  // converted and stored.
  {
    constexpr int kUnroll = kTopkChunkMax / (4 * kTkThreads);
    static_assert(kTopkChunkMax == 4 * kTkThreads * kUnroll, "one round of loads covers a chunk");
    const float* row = p.scores + (size_t)t * p.row_stride + lo;
    float4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = 4 * tid + 4 * kTkThreads * u;
      v[u] = j < n_here ? __ldg(reinterpret_cast<const float4*>(row + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();   // the histograms are zeroed before any count lands
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = 4 * tid + 4 * kTkThreads * u;
      if (j < n_here) {
        const uint4 kv = make_uint4(order_key(__float_as_uint(v[u].x)), order_key(__float_as_uint(v[u].y)),
                                    order_key(__float_as_uint(v[u].z)), order_key(__float_as_uint(v[u].w)));
        *reinterpret_cast<uint4*>(keys + j) = kv;
        if (!take_all) {
          atomicAdd(&hist[kv.x >> 21], 1u);
          if (j + 1 < n_here) atomicAdd(&hist[kv.y >> 21], 1u);
          if (j + 2 < n_here) atomicAdd(&hist[kv.z >> 21], 1u);
          if (j + 3 < n_here) atomicAdd(&hist[kv.w >> 21], 1u);
        }
      }
    }
  }
  __syncthreads();

  // ---- radix select ---------------------------------------------------------------
  // Warp w owns keys [w*seg, (w+1)*seg) of the chunk for the sweeps that keep position
  // order; a lane takes 4 consecutive keys of each 128-key step (one 16-byte load).
  const int seg = p.chunk / kTkWarps;
  const int w0 = warp * seg, w1 = min(w0 + seg, n_here);
  uint32_t prefix = 0;               // key bits above `shift` of the k-th largest key
  int shift = 32;
  uint32_t krem = (uint32_t)p.k;     // keys still to take at or below the prefix
  bool use_cand = false;             // passes 1-2 scan the warps' candidate lists
  uint32_t* my_cand = cand + warp * kCandPerWarp;
  uint32_t* my_cpos = cpos + warp * kCandPerWarp;
#pragma unroll 1
  for (int pass = 0; pass < kPasses && !take_all; ++pass) {
    const int width = pass_width(pass);
    const int nshift = shift - width;
    const uint32_t mask = (1u << width) - 1u;
    uint32_t* h = hist + pass * kMaxBins;
    if (pass == 0) {
      // counted while staging (top 11 bits: nshift == 21)
    } else if (use_cand) {
      const int nc = (int)wcand_s[warp];
      for (int j = lane; j < nc; j += 32) {
        const uint32_t key = my_cand[j];
        if ((key >> shift) == prefix) atomicAdd(&h[(key >> nshift) & mask], 1u);
      }
    } else {
      for (int j = tid; j < n_here; j += kTkThreads) {
        const uint32_t key = keys[j];
        if ((key >> shift) == prefix) atomicAdd(&h[(key >> nshift) & mask], 1u);
      }
    }
    if (C > 1) cluster_sync(); else __syncthreads();   // this pass's histograms are complete
    // thread tid owns bins lowest + per-1 down to lowest: descending bins in thread order;
    // with C > 1 the cluster's counts of those bins, one load per CTA, all in flight
    const int nb = 1 << width, per = nb / kTkThreads;   // 4 or 2 bins, half that in the 10-bit pass
    const int lowest = nb - per * (tid + 1);
    uint32_t c[4] = {0u, 0u, 0u, 0u};   // c[u]: bin lowest + per-1-u
    if (C == 1) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (u < per) c[u] = h[lowest + per - 1 - u];
    } else {
#pragma unroll
      for (int r0 = 0; r0 < 8; r0 += 4) {
        uint4 va[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          va[r] = make_uint4(0u, 0u, 0u, 0u);
          if (r0 + r < (int)C) {
            const uint32_t a = mapa(&h[lowest], (uint32_t)(r0 + r));
            if (per == 4)
              va[r] = ld_cluster_v4(a);
            else if (per == 2)
              ld_cluster_v2(a, va[r].x, va[r].y);
            else
              va[r].x = ld_cluster_u32(a);
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (per == 4) {
            c[0] += va[r].w;
            c[1] += va[r].z;
            c[2] += va[r].y;
            c[3] += va[r].x;
          } else if (per == 2) {
            c[0] += va[r].y;
            c[1] += va[r].x;
          } else {
            c[0] += va[r].x;
          }
        }
      }
    }
    uint32_t tot;
    uint32_t above = block_exclusive_scan(c[0] + c[1] + c[2] + c[3], wsum, tot);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (u < per && above < krem && krem <= above + c[u]) {
        sel_s[0] = (uint32_t)(lowest + per - 1 - u);
        sel_s[1] = krem - above;
        sel_s[2] = c[u];
      }
      above += c[u];
    }
    __syncthreads();
    prefix = (prefix << width) | sel_s[0];
    krem = sel_s[1];
    shift = nshift;
    const bool whole_bin = sel_s[2] == krem;
    if (pass == 0) {
      // each warp lists, in position order, the keys of its run whose top digit is at
      // least the chosen bin's -- every key that can still be chosen -- with their
      // positions.  Passes 1-2 and the output only look at these.  A warp with more than
      // kCandPerWarp of them sends every warp back to the whole chunk.
      uint32_t n = 0;
      for (int j0 = w0; j0 < w1; j0 += 32) {
        const int j = j0 + lane;
        const uint32_t key = j < w1 ? keys[j] : 0u;
        const bool in = j < w1 && (key >> shift) >= prefix;
        const unsigned m = __ballot_sync(0xffffffffu, in);
        const uint32_t o = n + (uint32_t)__popc(m & lanemask_lt());
        if (in && o < (uint32_t)kCandPerWarp) {
          my_cand[o] = key;
          my_cpos[o] = (uint32_t)(lo + j);
        }
        n += (uint32_t)__popc(m);
      }
      if (lane == 0) wcand_s[warp] = n;
      if (lane == 0 && n > (uint32_t)kCandPerWarp) ncand_over_s = 1u;
      __syncthreads();
      use_cand = ncand_over_s == 0u;
    }
    __syncthreads();   // sel_s is rewritten by the next pass
    if (whole_bin) break;
  }

  // ---- ordered compaction -----------------------------------------------------------
  // above: key bits over `shift` greater than the prefix; equal: the same bits; the
  // first `krem` equal keys in position order are taken.  With the candidate lists (in
  // position order) the warps count from those; otherwise each warp stages its chosen
  // and tied positions, in order, over the start of its own run of keys (a write never
  // overtakes the reads of the same step), tagging ties in bit 31.
  uint32_t n_st = 0, n_gt = 0, n_eq = 0;
  if (use_cand) {
    const uint32_t nc = wcand_s[warp];
    for (uint32_t i0 = 0; i0 < nc; i0 += 32) {
      const uint32_t i = i0 + lane;
      const uint32_t kb = i < nc ? my_cand[i] >> shift : 0u;
      n_gt += (uint32_t)__popc(__ballot_sync(0xffffffffu, i < nc && kb > prefix));
      n_eq += (uint32_t)__popc(__ballot_sync(0xffffffffu, i < nc && kb == prefix));
    }
  } else {
    for (int j0 = w0; j0 < w1; j0 += 128) {
      const int j = j0 + 4 * lane;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (j < w1) v = *reinterpret_cast<const uint4*>(keys + j);
      const uint32_t kv[4] = {v.x, v.y, v.z, v.w};
      uint32_t gbits = 0, ebits = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (j + u >= w1) continue;
        if (take_all) {
          gbits |= 1u << u;
        } else {
          const uint32_t kb = kv[u] >> shift;
          if (kb > prefix) gbits |= 1u << u;
          if (kb == prefix) ebits |= 1u << u;
        }
      }
      const uint32_t ng = (uint32_t)__popc(gbits), ne = (uint32_t)__popc(ebits);
      uint32_t tot_step;
      // packed (equal << 16 | above) counts: at most 128 of each per step
      const uint32_t off = warp_exclusive_scan(ng | (ne << 16), tot_step);
      uint32_t o = n_st + (off & 0xFFFFu) + (off >> 16);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool g = gbits & (1u << u), e = ebits & (1u << u);
        if (g || e) {
          keys[w0 + o] = (uint32_t)(lo + j + u) | (e ? 0x80000000u : 0u);
          ++o;
        }
      }
      n_gt += tot_step & 0xFFFFu;
      n_eq += tot_step >> 16;
      n_st += (tot_step & 0xFFFFu) + (tot_step >> 16);
    }
  }
  if (lane == 0) {
    wg_s[warp] = n_gt;
    we_s[warp] = n_eq;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t xg = lane < kTkWarps ? wg_s[lane] : 0u, xe = lane < kTkWarps ? we_s[lane] : 0u;
    uint32_t yg = xg, ye = xe;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t ng = __shfl_up_sync(0xffffffffu, yg, o), ne = __shfl_up_sync(0xffffffffu, ye, o);
      if (lane >= o) {
        yg += ng;
        ye += ne;
      }
    }
    if (lane < kTkWarps) {
      wg_s[lane] = yg - xg;
      we_s[lane] = ye - xe;
    }
    if (lane == 31) {
      cta_tot[0] = yg;
      cta_tot[1] = ye;
    }
  }
  uint32_t gbase = 0, ebase = 0;   // keys above / equal in lower-ranked CTAs
  if (C > 1) {
    cluster_sync();   // every CTA's totals are visible
    uint32_t xg[8], xe[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < (int)cr) {
        xg[r] = ld_cluster_u32(mapa(&cta_tot[0], (uint32_t)r));
        xe[r] = ld_cluster_u32(mapa(&cta_tot[1], (uint32_t)r));
      }
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < (int)cr) {
        gbase += xg[r];
        ebase += xe[r];
      }
    // the last read of another CTA's shared memory is done; the matching wait comes
    // after the writes, so no CTA leaves while a peer still reads its totals
    cluster_arrive();
  } else {
    __syncthreads();
  }
  // copy each warp's staged positions to the output: above-threshold positions all go,
  // ties while their rank is below krem
  int32_t* orow = p.out + (size_t)t * p.k;
  {
    uint32_t g = gbase + wg_s[warp], q = ebase + we_s[warp];
    const uint32_t n_items = use_cand ? wcand_s[warp] : n_st;
    for (uint32_t i0 = 0; i0 < n_items; i0 += 32) {
      const uint32_t i = i0 + lane;
      bool e, gsel;
      uint32_t item;
      if (use_cand) {
        const uint32_t kb = i < n_items ? my_cand[i] >> shift : 0u;
        gsel = i < n_items && kb > prefix;
        e = i < n_items && kb == prefix;
        item = i < n_items ? my_cpos[i] : 0u;
      } else {
        item = i < n_items ? keys[w0 + i] : 0u;
        e = i < n_items && (item >> 31);
        gsel = i < n_items && !(item >> 31);
      }
      const unsigned mg = __ballot_sync(0xffffffffu, gsel), me = __ballot_sync(0xffffffffu, e);
      const uint32_t lt = lanemask_lt();
      const uint32_t gb = g + (uint32_t)__popc(mg & lt), eb = q + (uint32_t)__popc(me & lt);
      const int32_t pos = (int32_t)(item & 0x7FFFFFFFu);
      // the output index is below k by construction; the bound only keeps a fault out
      if (gsel) {
        const uint32_t o = gb + min(eb, krem);
        if (o < (uint32_t)p.k) orow[o] = pos;
      } else if (e && eb < krem) {
        const uint32_t o = gb + eb;
        if (o < (uint32_t)p.k) orow[o] = pos;
      }
      g += __popc(mg);
      q += __popc(me);
    }
  }
  const int n_sel = take_all ? L : p.k;
  for (int j = n_sel + (int)cr * kTkThreads + tid; j < p.k; j += (int)C * kTkThreads) orow[j] = -1;
  if (C > 1) cluster_wait();
}

__global__ void __launch_bounds__(kTkThreads, 1) topk_kernel(const TopkParams p) {
  __shared__ TkShared sh;
  TkRow r;
  r.C = cluster_nctarank();
  r.cr = cluster_ctarank();
  r.t = (int)(blockIdx.x / r.C);
  int L = p.S;
  if (p.seq_lens) {
    const int b = r.t / p.Q, i = r.t % p.Q;
    const long long causal = (long long)p.seq_lens[b] - (p.Q - 1 - i);
    if (causal < L) L = causal > 0 ? (int)causal : 0;
  }
  r.L = L;
  r.lo = (int)r.cr * p.chunk;
  r.n_here = max(0, min(p.chunk, L - r.lo));
  const bool take_all = L <= p.k;   // every candidate is chosen: no search
  if (!take_all) {
    if (sampled_select(p, r, sh)) return;
    // the sampled threshold failed in this cluster: the sweep, once the peers are done
    // reading this CTA's lists
    if (r.C > 1) cluster_wait(); else __syncthreads();
  }
  sweep_select(p, r, take_all, sh);
}

int sm_count() {
  static std::atomic<int> cached[64];   // per device, 0 until first asked
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace

void topk_plan(int T, int S, int n_sms, int& C, int& chunk, int& threads) {
  // as few CTAs per token as hold the row (32K positions each), doubled while the grid
  // would fill less than half of the GPU and the chunks stay at least 4K positions
  C = (S + kTopkChunkMax - 1) / kTopkChunkMax;
  if (C < 1) C = 1;
  if (C > 8) C = 8;
  while (2 * C <= 8 && 2LL * T * C <= n_sms && (S + 2 * C - 1) / (2 * C) >= 4096) C *= 2;
  const int per = (S + C - 1) / C;
  chunk = ((per + kChunkUnit - 1) / kChunkUnit) * kChunkUnit;
  if (chunk < kChunkUnit) chunk = kChunkUnit;
  threads = kTkThreads;
}

cudaError_t launch_topk(const float* scores, long long row_stride, const int32_t* seq_lens, int B, int Q, int S,
                        int k, int32_t* out, cudaStream_t stream) {
  const int T = B * Q;
  if (T == 0) return cudaSuccess;
  int C = 1, chunk = 0, threads = 0;
  topk_plan(T, S, sm_count(), C, chunk, threads);
  TopkParams p;
  p.scores = scores;
  p.row_stride = row_stride;
  p.seq_lens = seq_lens;
  p.Q = Q;
  p.S = S;
  p.k = k;
  p.chunk = chunk;
  p.out = out;
  static std::atomic<bool> attr_set[64];   // per device: set once (a repeat is harmless)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         topk_smem_bytes(kTopkChunkMax));
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(T * C));
  cfg.blockDim = dim3(kTkThreads);
  cfg.dynamicSmemBytes = (size_t)topk_smem_bytes(chunk);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel, p);
}

}  // namespace sfa
