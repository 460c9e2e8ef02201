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

constexpr int kTkThreads = 1024;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kSlab = 4 * kTkThreads;   // positions covered by one float4 load per thread
constexpr int kMaxBins = 2048;
constexpr int kPasses = 3;

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

__device__ __forceinline__ int pass_width(int pass) { return pass < 2 ? 11 : 10; }

template <int KPT>
__global__ void __launch_bounds__(kTkThreads, 1) topk_kernel(const TopkParams p) {
  constexpr int kSlabs = KPT / 4;
  __shared__ uint32_t hist[kPasses][kMaxBins];
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
    // thread tid owns bins nb-1-per*tid-u (u < per): descending bins in thread order
    const int nb = 1 << width, per = nb / kTkThreads;
    uint32_t c[2] = {0u, 0u};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u >= per) break;
      const int bin = nb - 1 - per * tid - u;
      for (uint32_t r = 0; r < C; ++r) c[u] += ld_cluster_u32(mapa(&hist[pass][bin], r));
    }
    // exclusive block scan of the per-thread sums: keys in higher bins than this thread's
    uint32_t s = c[0] + c[1], inc = s;
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
    }
    __syncthreads();
    uint32_t above = wsum[warp] + inc - s;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
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
      const uint32_t x = wtot[j][lane];
      uint32_t y = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) y += n;
      }
      wtot[j][lane] = y - x;
      if (lane == 0) slab_off[j] = run;
      run += __shfl_sync(0xffffffffu, y, 31);
    }
    if (lane == 0) cta_tot = run;
  }
  cluster_sync();   // slab offsets, warp prefixes and every CTA's total are visible
  uint32_t gbase = 0, ebase = 0;   // keys above / equal in lower-ranked CTAs
  for (uint32_t r = 0; r < cr; ++r) {
    const uint32_t x = ld_cluster_u32(mapa(&cta_tot, r));
    gbase += x >> 16;
    ebase += x & 0xFFFFu;
  }
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
      if (gt) {
        orow[g + min(q, krem)] = pos;
        ++g;
      } else if (eq) {
        if (q < krem) orow[g + q] = pos;
        ++q;
      }
    }
  }
  const int n_sel = take_all ? L : p.k;
  for (int j = n_sel + (int)cr * kTkThreads + tid; j < p.k; j += (int)C * kTkThreads) orow[j] = -1;
  cluster_sync();   // no CTA leaves while another still reads its shared memory
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

template <int KPT>
cudaError_t launch_kpt(const TopkParams& p, int T, int C, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(T * C));
  cfg.blockDim = dim3(kTkThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel<KPT>, p);
}

}  // namespace

void topk_plan(int T, int S, int n_sms, int& C, int& chunk) {
  // up to 16K positions per CTA where 8 CTAs allow it (32 keys a thread spill registers),
  // then more CTAs per token while the grid is smaller than the GPU
  C = 1;
  while (C < 8 && (long long)C * (kTopkChunkMax / 2) < S) C *= 2;
  while (C < 8 && (long long)T * C < n_sms && (S + 2 * C - 1) / (2 * C) >= kSlab) C *= 2;
  const int per = (S + C - 1) / C;
  chunk = ((per + kSlab - 1) / kSlab) * kSlab;
  if (chunk < kSlab) chunk = kSlab;
}

cudaError_t launch_topk(const float* scores, long long row_stride, const int32_t* seq_lens, int B, int Q, int S,
                        int k, int32_t* out, cudaStream_t stream) {
  const int T = B * Q;
  if (T == 0) return cudaSuccess;
  int C = 1, chunk = kSlab;
  topk_plan(T, S, sm_count(), C, chunk);
  TopkParams p;
  p.scores = scores;
  p.row_stride = row_stride;
  p.seq_lens = seq_lens;
  p.Q = Q;
  p.S = S;
  p.k = k;
  p.chunk = chunk;
  p.out = out;
  if (chunk <= 4 * kTkThreads) return launch_kpt<4>(p, T, C, stream);
  if (chunk <= 8 * kTkThreads) return launch_kpt<8>(p, T, C, stream);
  if (chunk <= 16 * kTkThreads) return launch_kpt<16>(p, T, C, stream);
  return launch_kpt<32>(p, T, C, stream);
}

}  // namespace sfa
