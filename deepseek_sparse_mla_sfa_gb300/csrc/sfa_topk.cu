// sfa_topk.cu -- indexer top-k selection: for each query token, the k cache positions
// with the largest indexer scores, i.e. the list that sparse attention then visits
// ("vllm-ascend PR #18870 解读", 4.5: only the top-2048 positions the indexer chose are
// attended, not the whole history).
//
// Order: IEEE 754 totalOrder of the fp32 scores, larger first; equal scores are taken
// lower position first.  Output: the chosen positions in ascending order, then -1.
//
// One cluster of C CTAs (C = 1..8, C = 1 for rows of up to 32K positions) per query
// token; CTA r of the cluster stages the contiguous chunk [r*chunk, (r+1)*chunk) of the
// token's candidate range in shared memory, as 32-bit keys whose unsigned order is the
// totalOrder of the scores.
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

constexpr int kTkThreads = 1024;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kMaxBins = 2048;
constexpr int kPasses = 3;
constexpr int kPer = kMaxBins / kTkThreads;   // histogram bins per thread in an 11-bit pass
constexpr int kCandCap = 8192;                // candidates kept after pass 0 (32 KB)
constexpr int kCandPerWarp = kCandCap / kTkWarps;
static_assert(kPer == 2, "bin ownership below assumes two bins per thread");
static_assert(kTopkChunkMax % (32 * kTkWarps) == 0, "a chunk splits into whole warp runs");

// dynamic shared memory: keys | candidate keys | candidate positions | histograms
__host__ __device__ constexpr int kOffCand(int chunk) { return chunk * 4; }
__host__ __device__ constexpr int kOffCpos(int chunk) { return chunk * 4 + kCandCap * 4; }
__host__ __device__ constexpr int kOffHist(int chunk) { return chunk * 4 + 2 * kCandCap * 4; }
__host__ __device__ constexpr int topk_smem_bytes(int chunk) { return kOffHist(chunk) + kPasses * kMaxBins * 4; }

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
    const uint32_t x = wsum[lane];
    uint32_t y = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += n;
    }
    wsum[lane] = y - x;
    if (lane == 31) wsum[32] = y;
  }
  __syncthreads();
  total = wsum[32];
  const uint32_t r = wsum[warp] + inc - v;
  __syncthreads();   // wsum is reused by the next scan
  return r;
}

__global__ void __launch_bounds__(kTkThreads, 1) topk_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint32_t tk_smem[];
  uint32_t* keys = tk_smem;
  uint32_t* cand = tk_smem + kOffCand(p.chunk) / 4;
  uint32_t* cpos = tk_smem + kOffCpos(p.chunk) / 4;
  uint32_t* hist = tk_smem + kOffHist(p.chunk) / 4;   // [kPasses][kMaxBins]
  __shared__ uint32_t wsum[33];
  __shared__ uint32_t wg_s[kTkWarps], we_s[kTkWarps];   // per-warp (above, equal) counts, then bases
  __shared__ uint32_t sel_s[3];                         // chosen bin, keys still needed, keys in the bin
  __shared__ uint32_t wcand_s[kTkWarps];               // candidates each warp listed
  __shared__ uint32_t ncand_over_s;                     // some warp listed more than it keeps
  __shared__ uint32_t cta_tot[2];                       // this CTA's (above, equal) totals

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t C = cluster_nctarank(), cr = cluster_ctarank();
  const int t = (int)(blockIdx.x / C);

  int L = p.S;
  if (p.seq_lens) {
    const int b = t / p.Q, i = t % p.Q;
    const long long causal = (long long)p.seq_lens[b] - (p.Q - 1 - i);
    if (causal < L) L = causal > 0 ? (int)causal : 0;
  }
  const bool take_all = L <= p.k;   // every candidate is chosen: no search
  const int lo = (int)cr * p.chunk;
  const int n_here = max(0, min(p.chunk, L - lo));   // valid keys of this CTA: keys[0, n_here)

  for (int x = tid; x < kPasses * kMaxBins; x += kTkThreads) hist[x] = 0u;
  if (tid == 0) ncand_over_s = 0u;

  // ---- stage the chunk and count pass 0 --------------------------------------------
  // A chunk is at most 32 keys a thread: all of a thread's 16-byte loads are in flight
  // at once, and each key is counted into the pass-0 histogram (top 11 bits) as it is
  // converted and stored.
  {
    static_assert(kTopkChunkMax <= 4 * kTkThreads * 8, "one round of 8 loads covers a chunk");
    const float* row = p.scores + (size_t)t * p.row_stride + lo;
    constexpr int kUnroll = 8;
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
    // thread tid owns bins nb-1-per*tid-u (u < per): descending bins in thread order;
    // with C > 1 the cluster's counts of those bins, one load per CTA, all in flight
    const int nb = 1 << width, per = nb / kTkThreads;   // 2, or 1 for the 10-bit pass
    uint32_t c0 = 0u, c1 = 0u;   // bins nb-1-per*tid and nb-2-2*tid
    const int lowest = nb - per * (tid + 1);
    if (C == 1) {
      if (per == 2) {
        c0 = h[lowest + 1];
        c1 = h[lowest];
      } else {
        c0 = h[lowest];
      }
    } else {
#pragma unroll
      for (int r0 = 0; r0 < 8; r0 += 4) {
        uint32_t va[4], vb[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          va[r] = vb[r] = 0u;
          if (r0 + r < (int)C) {
            const uint32_t a = mapa(&h[lowest], (uint32_t)(r0 + r));
            if (per == 2)
              ld_cluster_v2(a, va[r], vb[r]);
            else
              vb[r] = ld_cluster_u32(a);
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          c0 += vb[r];
          c1 += va[r];
        }
      }
      if (per == 1) c1 = 0u;
    }
    uint32_t tot;
    const uint32_t above = block_exclusive_scan(c0 + c1, wsum, tot);
    if (above < krem && krem <= above + c0) {
      sel_s[0] = (uint32_t)(nb - 1 - per * tid);
      sel_s[1] = krem - above;
      sel_s[2] = c0;
    } else if (per == 2 && above + c0 < krem && krem <= above + c0 + c1) {
      sel_s[0] = (uint32_t)(nb - 2 - 2 * tid);
      sel_s[1] = krem - above - c0;
      sel_s[2] = c1;
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
    const uint32_t xg = wg_s[lane], xe = we_s[lane];
    uint32_t yg = xg, ye = xe;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t ng = __shfl_up_sync(0xffffffffu, yg, o), ne = __shfl_up_sync(0xffffffffu, ye, o);
      if (lane >= o) {
        yg += ng;
        ye += ne;
      }
    }
    wg_s[lane] = yg - xg;
    we_s[lane] = ye - xe;
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
  while (C < 8 && 2LL * T * C <= n_sms && (S + 2 * C - 1) / (2 * C) >= 4096) C *= 2;
  const int per = (S + C - 1) / C;
  const int unit = 32 * kTkWarps;
  chunk = ((per + unit - 1) / unit) * unit;
  if (chunk < unit) chunk = unit;
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
