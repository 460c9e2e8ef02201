// sfa_topk.cu -- indexer top-k selection: for each query token, the k cache positions
// with the largest indexer scores, i.e. the list that sparse attention then visits
// ("vllm-ascend PR #18870 解读", 4.5: only the top-2048 positions the indexer chose are
// attended, not the whole history).
//
// Order: IEEE 754 totalOrder of the fp32 scores, larger first; equal scores are taken
// lower position first.  Output: the chosen positions in ascending order, then -1.
//
// One cluster of C CTAs (C = 1..8) per query token; CTA r of the cluster holds the
// contiguous chunk [r*chunk, (r+1)*chunk) of the token's candidate range in registers,
// as 32-bit keys whose unsigned order is the totalOrder of the scores.
//   * Radix select in three passes (11, 11 and 10 key bits from the top).  In each pass
//     every CTA counts its keys that still carry the chosen prefix into a shared-memory
//     histogram; the cluster sums the histograms over distributed shared memory and every
//     CTA finds the same bin, the one holding the k-th largest key.  A pass whose bin
//     must be taken whole ends the search early.
//   * Ordered compaction: per-thread counts of keys above the threshold and equal to it
//     go through a block scan; the totals of lower-ranked CTAs of the cluster give each
//     CTA its base; each chosen position then knows its output index.
// No wait in this kernel spins: the only synchronisation is block and cluster barriers.
#include "sfa_internal.h"
#include "sfa_ptx.cuh"

namespace sfa {
namespace {

using namespace ptx;

constexpr int kMaxBins = 2048;
constexpr int kPasses = 3;
// Chunks of up to kSmallChunk positions run as 512-thread CTAs (two per SM); longer
// chunks as 1024-thread CTAs, so that a thread holds at most 32 keys.
constexpr int kSmallThreads = 512;
constexpr int kSmallChunk = 16 * kSmallThreads;

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
// `n` (1, 2 or 4) consecutive words of another CTA's shared memory into v[0..n)
__device__ __forceinline__ void ld_cluster_vec(uint32_t addr, int n, uint32_t* v) {
  if (n == 4)
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "r"(addr)
                 : "memory");
  else if (n == 2)
    asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "r"(addr) : "memory");
  else
    v[0] = ld_cluster_u32(addr);
}

__device__ __forceinline__ int pass_width(int pass) { return pass < 2 ? 11 : 10; }

template <int NT, int KPT>
__global__ void __launch_bounds__(NT, 1024 / NT) topk_kernel(const TopkParams p) {
  constexpr int kTkThreads = NT;
  constexpr int kTkWarps = NT / 32;
  static_assert(kTkWarps <= 32, "one warp scans the per-warp totals");
  constexpr int kSlab = 4 * NT;                   // positions covered by one float4 load per thread
  constexpr int kMaxPer = kMaxBins / NT;          // histogram bins per thread in the widest pass
  static_assert(kMaxPer == 2 || kMaxPer == 4, "bins per thread load as one vector");
  constexpr int kSlabs = KPT / 4;
  __shared__ __align__(16) uint32_t hist[kPasses][kMaxBins];   // vector loads of 1, 2 or 4 bins
  __shared__ uint32_t wtot[kSlabs][kTkWarps];   // warp totals of the packed counts
  __shared__ uint32_t slab_off[kSlabs];
  __shared__ uint32_t wsum[kTkWarps];
  __shared__ uint32_t sel_s[3];                 // chosen bin, keys still needed, keys in the bin
  __shared__ uint32_t cta_tot;                  // this CTA's (above << 16 | equal) total

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
  const int hi = min(lo + p.chunk, L);

  for (int x = tid; x < kPasses * kMaxBins; x += kTkThreads) (&hist[0][0])[x] = 0;

  // this thread's keys: slab j holds positions lo + kSlab*j + 4*tid + (0..3)
  uint32_t key[KPT];
  const float* row = p.scores + (size_t)t * p.row_stride;
#pragma unroll
  for (int j = 0; j < kSlabs; ++j) {
    const int base = lo + kSlab * j + 4 * tid;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (base < hi) v = __ldg(reinterpret_cast<const float4*>(row + base));
    key[4 * j] = order_key(__float_as_uint(v.x));
    key[4 * j + 1] = order_key(__float_as_uint(v.y));
    key[4 * j + 2] = order_key(__float_as_uint(v.z));
    key[4 * j + 3] = order_key(__float_as_uint(v.w));
  }
  auto valid = [&](int e) { return lo + kSlab * (e >> 2) + 4 * tid + (e & 3) < hi; };
  __syncthreads();

  // ---- radix select ---------------------------------------------------------------
  uint32_t prefix = 0;   // key bits above `shift` of the k-th largest key
  int shift = 32;
  uint32_t krem = (uint32_t)p.k;   // keys still to take at or below the prefix
#pragma unroll 1
  for (int pass = 0; pass < kPasses && !take_all; ++pass) {
    const int width = pass_width(pass);
    const int nshift = shift - width;
    const uint32_t mask = (1u << width) - 1u;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      const bool match = pass == 0 || (key[e] >> shift) == prefix;
      if (valid(e) && match) atomicAdd(&hist[pass][(key[e] >> nshift) & mask], 1u);
    }
    cluster_sync();   // every CTA's histogram of this pass is complete and visible
    // thread tid owns bins nb-1-per*tid-u (u < per): descending bins in thread order.
    // The cluster's counts of those bins: one load per CTA, all in flight together.
    const int nb = 1 << width, per = nb / kTkThreads;   // kMaxPer, or half of it for 10 bits
    uint32_t c[kMaxPer];
#pragma unroll
    for (int u = 0; u < kMaxPer; ++u) c[u] = 0u;
    {
      const uint32_t* own = &hist[pass][nb - per * (tid + 1)];   // the lowest of the thread's bins
#pragma unroll
      for (int r0 = 0; r0 < 8; r0 += 4) {   // four CTAs' loads in flight at a time
        uint32_t v[4][kMaxPer];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
#pragma unroll
          for (int u = 0; u < kMaxPer; ++u) v[r][u] = 0u;
          if (r0 + r < (int)C) ld_cluster_vec(mapa(own, (uint32_t)(r0 + r)), per, v[r]);
        }
        // bin nb-1-per*tid-u is word per-1-u of the vector (per is kMaxPer or half of it)
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int u = 0; u < kMaxPer; ++u) {
            if (per == kMaxPer) {
              c[u] += v[r][kMaxPer - 1 - u];
            } else if (u < kMaxPer / 2) {
              c[u] += v[r][kMaxPer / 2 - 1 - u];
            }
          }
      }
    }
    // exclusive block scan of the per-thread sums: keys in higher bins than this thread's
    uint32_t s = 0;
#pragma unroll
    for (int u = 0; u < kMaxPer; ++u) s += c[u];
    uint32_t inc = s;
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
    }
    __syncthreads();
    uint32_t above = wsum[warp] + inc - s;
#pragma unroll
    for (int u = 0; u < kMaxPer; ++u) {
      if (u >= per) break;
      if (above < krem && krem <= above + c[u]) {
        sel_s[0] = (uint32_t)(nb - 1 - per * tid - u);
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
    __syncthreads();   // sel_s and wsum are rewritten by the next pass
    if (whole_bin) break;
  }

  // ---- ordered compaction -----------------------------------------------------------
  // above: key bits over `shift` greater than the prefix; equal: the same bits; the
  // first `krem` equal keys in position order are taken
  auto cls = [&](int e, bool& gt, bool& eq) {
    gt = false;
    eq = false;
    if (!valid(e)) return;
    if (take_all) {
      gt = true;
      return;
    }
    const uint32_t kb = key[e] >> shift;
    gt = kb > prefix;
    eq = kb == prefix;
  };
  uint32_t cnt[kSlabs];
#pragma unroll
  for (int j = 0; j < kSlabs; ++j) {
    uint32_t v = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      bool gt, eq;
      cls(4 * j + u, gt, eq);
      v += (gt ? 0x10000u : 0u) + (eq ? 1u : 0u);
    }
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    if (lane == 31) wtot[j][warp] = inc;
    cnt[j] = inc - v;   // exclusive within the warp
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t run = 0;
#pragma unroll
    for (int j = 0; j < kSlabs; ++j) {
      const uint32_t x = lane < kTkWarps ? wtot[j][lane] : 0u;
      uint32_t y = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) y += n;
      }
      if (lane < kTkWarps) wtot[j][lane] = y - x;
      if (lane == 0) slab_off[j] = run;
      run += __shfl_sync(0xffffffffu, y, 31);
    }
    if (lane == 0) cta_tot = run;
  }
  cluster_sync();   // slab offsets, warp prefixes and every CTA's total are visible
  uint32_t gbase = 0, ebase = 0;   // keys above / equal in lower-ranked CTAs
  {
    uint32_t x[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < (int)cr) x[r] = ld_cluster_u32(mapa(&cta_tot, (uint32_t)r));
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < (int)cr) {
        gbase += x[r] >> 16;
        ebase += x[r] & 0xFFFFu;
      }
  }
  // the last read of another CTA's shared memory is done; the matching wait comes after
  // the writes, so no CTA leaves while a peer still reads its totals
  cluster_arrive();
  int32_t* orow = p.out + (size_t)t * p.k;
#pragma unroll
  for (int j = 0; j < kSlabs; ++j) {
    const uint32_t b = slab_off[j] + wtot[j][warp] + cnt[j];
    uint32_t g = gbase + (b >> 16), q = ebase + (b & 0xFFFFu);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      bool gt, eq;
      cls(4 * j + u, gt, eq);
      const int pos = lo + kSlab * j + 4 * tid + u;
      // the output index is below k by construction; the bound only keeps a fault out
      if (gt) {
        const uint32_t o = g + min(q, krem);
        if (o < (uint32_t)p.k) orow[o] = pos;
        ++g;
      } else if (eq) {
        if (q < krem && g + q < (uint32_t)p.k) orow[g + q] = pos;
        ++q;
      }
    }
  }
  const int n_sel = take_all ? L : p.k;
  for (int j = n_sel + (int)cr * kTkThreads + tid; j < p.k; j += (int)C * kTkThreads) orow[j] = -1;
  cluster_wait();
}

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int NT, int KPT>
cudaError_t launch_kpt(const TopkParams& p, int T, int C, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(T * C));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel<NT, KPT>, p);
}

}  // namespace

void topk_plan(int T, int S, int n_sms, int& C, int& chunk, int& threads) {
  // at most kSmallChunk positions per CTA where 8 CTAs per token allow it, then more CTAs
  // per token while the grid is smaller than the GPU (chunks of at least 2048 positions)
  C = 1;
  while (C < 8 && (long long)C * kSmallChunk < S) C *= 2;
  while (C < 8 && (long long)T * C < n_sms && (S + 2 * C - 1) / (2 * C) >= 4 * kSmallThreads) C *= 2;
  const int per = (S + C - 1) / C;
  threads = per <= kSmallChunk ? kSmallThreads : 2 * kSmallThreads;
  const int slab = 4 * threads;
  chunk = ((per + slab - 1) / slab) * slab;
  if (chunk < slab) chunk = slab;
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
  if (threads == kSmallThreads) {
    if (chunk <= 4 * kSmallThreads) return launch_kpt<kSmallThreads, 4>(p, T, C, stream);
    if (chunk <= 8 * kSmallThreads) return launch_kpt<kSmallThreads, 8>(p, T, C, stream);
    return launch_kpt<kSmallThreads, 16>(p, T, C, stream);
  }
  if (chunk <= 32 * kSmallThreads) return launch_kpt<2 * kSmallThreads, 16>(p, T, C, stream);
  return launch_kpt<2 * kSmallThreads, 32>(p, T, C, stream);
}

}  // namespace sfa
