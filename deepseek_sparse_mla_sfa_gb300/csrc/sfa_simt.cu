// sfa_simt.cu -- general CUDA-core path of sparse MLA decode.
//
// Handles every supported shape (1 <= h <= 128, any block size); the tcgen05
// path takes the shapes it supports.  One CTA per (query token, shard, group of
// 8 heads); its 4 warps take the token's selected entries round-robin, each
// keeping an online softmax (running max m, sum l, unnormalised output) per
// head, and the warps' states are combined at the end.  This is the plain
// definition of "RFC: MsModeling 支持 Decode Context Parallel 仿真" 2.1.4.2 /
// "vllm-ascend PR #18870 解读" 4.5 (softmax(q K^T scale) V over the selected rows
// of the paged latent cache, with the per-head log-sum-exp).
#include <atomic>
#include "sfa_internal.h"

namespace sfa {
namespace {

constexpr int kHG = 8;      // heads per CTA
constexpr int kWarps = 4;   // warps per CTA
constexpr int kQKPerLane = kDQK / 64;  // 9 bf16x2 pairs per lane cover 576 columns
constexpr int kVPerLane = kDV / 64;    // 8 of them are the latent (V) columns

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kWarps * 32) decode_simt_kernel(DecodeParams p) {
  extern __shared__ float smem[];
  float* q_s = smem;                                  // [kHG][576]
  float* o_s = q_s + kHG * kDQK;                      // [kWarps][kHG][512]
  float* m_s = o_s + kWarps * kHG * kDV;              // [kWarps][kHG]
  float* l_s = m_s + kWarps * kHG;                    // [kWarps][kHG]

  const int t = blockIdx.x, r = blockIdx.y, g = blockIdx.z;
  const int T = p.B * p.Q;
  const int h0 = g * kHG;
  const int nh = min(kHG, p.h - h0);
  const int b = t / p.Q, i = t % p.Q;
  const int seq_len = p.seq_lens[b];
  const int L = seq_len - (p.Q - 1 - i);
  const ShardSel sel = shard_sel(seq_len, L, r, p.n_splits, p.interleave);
  const int bt_row = p.bt_per_token ? t : b;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int x = threadIdx.x; x < kHG * kDQK; x += blockDim.x) {
    int hh = x / kDQK, d = x % kDQK;
    q_s[x] = hh < nh ? __bfloat162float(p.q[((size_t)t * p.h + h0 + hh) * kDQK + d]) : 0.f;
  }
  __syncthreads();

  float m[kHG], l[kHG], o[kHG][2 * kVPerLane];
#pragma unroll
  for (int hh = 0; hh < kHG; ++hh) {
    m[hh] = -INFINITY;
    l[hh] = 0.f;
#pragma unroll
    for (int c = 0; c < 2 * kVPerLane; ++c) o[hh][c] = 0.f;
  }

  const int32_t* idx = p.topk_idx + (size_t)t * p.top_k;
  for (int j = warp; j < p.top_k; j += kWarps) {
    const int pos = idx[j];
    if (!sel.has(pos)) continue;
    const int blk = pos / p.block_size;
    const int phys = blk < p.max_blocks ? p.block_table[(size_t)bt_row * p.max_blocks + blk] : -1;
    if (phys < 0 || phys >= p.num_blocks) {
      if (lane == 0) report_status(p.status, kStatusBadBlock);
      continue;
    }
    const __nv_bfloat162* row = reinterpret_cast<const __nv_bfloat162*>(
        p.kv + ((size_t)phys * p.block_size + pos % p.block_size) * kDQK);
    // lane holds columns 2*lane + 64*k and 2*lane + 1 + 64*k, k = 0..8
    float kx[2 * kQKPerLane];
#pragma unroll
    for (int k = 0; k < kQKPerLane; ++k) {
      float2 f = __bfloat1622float2(row[lane + 32 * k]);
      kx[2 * k] = f.x;
      kx[2 * k + 1] = f.y;
    }
#pragma unroll
    for (int hh = 0; hh < kHG; ++hh) {
      if (hh >= nh) break;
      const float* qh = q_s + hh * kDQK;
      float part = 0.f;
#pragma unroll
      for (int k = 0; k < kQKPerLane; ++k)
        part += qh[2 * lane + 64 * k] * kx[2 * k] + qh[2 * lane + 1 + 64 * k] * kx[2 * k + 1];
      const float s = warp_sum(part) * p.scale;
      const float m_new = fmaxf(m[hh], s);
      const float alpha = __expf(m[hh] - m_new);
      const float e = __expf(s - m_new);
      l[hh] = l[hh] * alpha + e;
#pragma unroll
      for (int c = 0; c < 2 * kVPerLane; ++c) o[hh][c] = o[hh][c] * alpha + e * kx[c];
      m[hh] = m_new;
    }
  }

  // combine the warps' online-softmax states
#pragma unroll
  for (int hh = 0; hh < kHG; ++hh) {
#pragma unroll
    for (int k = 0; k < kVPerLane; ++k) {
      o_s[(warp * kHG + hh) * kDV + 2 * lane + 64 * k] = o[hh][2 * k];
      o_s[(warp * kHG + hh) * kDV + 2 * lane + 1 + 64 * k] = o[hh][2 * k + 1];
    }
    if (lane == 0) {
      m_s[warp * kHG + hh] = m[hh];
      l_s[warp * kHG + hh] = l[hh];
    }
  }
  __syncthreads();

  float* out = p.out + ((size_t)r * T + t) * p.h * kDV;
  float* lse = p.lse + ((size_t)r * T + t) * p.h;
  for (int x = threadIdx.x; x < nh * kDV; x += blockDim.x) {
    const int hh = x / kDV, c = x % kDV;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, m_s[w * kHG + hh]);
    float val = 0.f, lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float sc = __expf(m_s[w * kHG + hh] - M);
        lsum += l_s[w * kHG + hh] * sc;
        val += o_s[(w * kHG + hh) * kDV + c] * sc;
      }
      val /= lsum;
    }
    out[(size_t)(h0 + hh) * kDV + c] = val;
    if (c == 0) lse[h0 + hh] = M == -INFINITY ? -INFINITY : M + logf(lsum);
  }
}

}  // namespace

constexpr size_t kSmemSimt = sizeof(float) * (kHG * kDQK + kWarps * kHG * kDV + 2 * kWarps * kHG);

cudaError_t prepare_decode_simt() {
  static std::atomic<bool> attr_set[64];   // per device: set once (a repeat is harmless)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemSimt);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

cudaError_t launch_decode_simt(const DecodeParams& p, cudaStream_t stream) {
  const int T = p.B * p.Q;
  if (T == 0) return cudaSuccess;
  const size_t smem = kSmemSimt;
  cudaError_t e = prepare_decode_simt();
  if (e != cudaSuccess) return e;
  dim3 grid(T, p.n_splits, (p.h + kHG - 1) / kHG);
  decode_simt_kernel<<<grid, kWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace sfa
