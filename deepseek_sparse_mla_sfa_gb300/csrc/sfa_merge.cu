// sfa_merge.cu -- online-softmax merge of per-shard (out, lse) partials.
//
// "RFC: MsModeling 支持 Decode Context Parallel 仿真" 1.1 / 2.1.1: after the
// all-to-all of (output ⊕ lse) each rank rebuilds the full output with a local
// online-softmax merge; 2.1.4.3: the partials travel in fp32.  Here the shards
// are all on one GPU and the merge is a streaming kernel: one warp per output
// row, the n lse values spread over the lanes, 16-byte loads of the partial
// rows, one pass over the data.
#include "sfa_internal.h"

namespace sfa {
namespace {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// n <= 64: lane holds shards `lane` and `lane + 32`.
template <bool kVec4>
__global__ void __launch_bounds__(256) lse_merge_kernel(const float* __restrict__ out_part,
                                                        const float* __restrict__ lse_part, int n,
                                                        int rows, int dv, float* __restrict__ out,
                                                        float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  const long long stride = (long long)gridDim.x * warps_per_block;
  for (long long row = (long long)blockIdx.x * warps_per_block + (threadIdx.x >> 5); row < rows;
       row += stride) {
    const float l0 = lane < n ? lse_part[(size_t)lane * rows + row] : -INFINITY;
    const float l1 = lane + 32 < n ? lse_part[(size_t)(lane + 32) * rows + row] : -INFINITY;
    const float M = warp_max(fmaxf(l0, l1));
    float* orow = out + (size_t)row * dv;
    if (M == -INFINITY) {
      for (int c = lane; c < dv; c += 32) orow[c] = 0.f;
      if (lane == 0) lse[row] = -INFINITY;
      continue;
    }
    const float Z = warp_sum((lane < n ? expf(l0 - M) : 0.f) + (lane + 32 < n ? expf(l1 - M) : 0.f));
    const float L = M + logf(Z);
    // weight of shard r: exp(lse_r - L) (exactly 0 for an empty shard)
    const float w0 = lane < n ? expf(l0 - L) : 0.f;
    const float w1 = lane + 32 < n ? expf(l1 - L) : 0.f;
    // The column loops run the same trip count on every lane (the weight of shard r comes
    // from lane r % 32 by a full-warp shuffle); each lane bounds its own column.
    if (kVec4) {
      const int dv4 = dv >> 2;
      for (int c0 = 0; c0 < dv4; c0 += 32) {
        const int c = c0 + lane;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < n; ++r) {
          const float w = __shfl_sync(0xffffffffu, r < 32 ? w0 : w1, r & 31);
          if (w == 0.f || c >= dv4) continue;
          const float4 v =
              __ldg(reinterpret_cast<const float4*>(out_part + ((size_t)r * rows + row) * dv) + c);
          acc.x += w * v.x;
          acc.y += w * v.y;
          acc.z += w * v.z;
          acc.w += w * v.w;
        }
        if (c < dv4) reinterpret_cast<float4*>(orow)[c] = acc;
      }
    } else {
      for (int c0 = 0; c0 < dv; c0 += 32) {
        const int c = c0 + lane;
        float acc = 0.f;
        for (int r = 0; r < n; ++r) {
          const float w = __shfl_sync(0xffffffffu, r < 32 ? w0 : w1, r & 31);
          if (w == 0.f || c >= dv) continue;
          acc += w * out_part[((size_t)r * rows + row) * dv + c];
        }
        if (c < dv) orow[c] = acc;
      }
    }
    if (lane == 0) lse[row] = L;
  }
}

// n <= 8 shards of 512-wide rows: a lane owns 16-byte columns lane + 32j (j < 4) of the
// row.  All of its partial loads go out together with the lse loads, in two rounds of 16,
// so the weights are computed while the rows are in flight instead of before.
constexpr int kFastShards = 8;
constexpr int kFastCols4 = 512 / 4 / 32;   // float4 columns per lane

__global__ void __launch_bounds__(256) lse_merge_fast_kernel(const float* __restrict__ out_part,
                                                             const float* __restrict__ lse_part, int n,
                                                             int rows, float* __restrict__ out,
                                                             float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  const long long stride = (long long)gridDim.x * warps_per_block;
  const size_t rstride4 = (size_t)rows * 512 / 4;   // float4s between shards
  for (long long row = (long long)blockIdx.x * warps_per_block + (threadIdx.x >> 5); row < rows;
       row += stride) {
    const float lv = lane < n ? lse_part[(size_t)lane * rows + row] : -INFINITY;
    const float4* base = reinterpret_cast<const float4*>(out_part + (size_t)row * 512) + lane;
    float4 acc[kFastCols4];
    float w = 0.f, L = -INFINITY;
    bool empty = false;
#pragma unroll
    for (int j0 = 0; j0 < kFastCols4; j0 += 2) {
      float4 v[2][kFastShards];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int u = 0; u < kFastShards; ++u)
          v[jj][u] = u < n ? __ldg(base + (size_t)u * rstride4 + 32 * (j0 + jj)) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (j0 == 0) {   // the weights, while the first round of rows is in flight
        const float M = warp_max(lv);
        empty = M == -INFINITY;
        if (!empty) {
          const float Z = warp_sum(lane < n ? expf(lv - M) : 0.f);
          L = M + logf(Z);
          w = lane < n ? expf(lv - L) : 0.f;   // exactly 0 for an empty shard
        }
      }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kFastShards; ++u) {
          const float wu = __shfl_sync(0xffffffffu, w, u);
          if (u < n && wu != 0.f) {
            a.x += wu * v[jj][u].x;
            a.y += wu * v[jj][u].y;
            a.z += wu * v[jj][u].z;
            a.w += wu * v[jj][u].w;
          }
        }
        acc[j0 + jj] = a;
      }
    }
    float4* orow = reinterpret_cast<float4*>(out + (size_t)row * 512) + lane;
#pragma unroll
    for (int j = 0; j < kFastCols4; ++j) orow[32 * j] = empty ? make_float4(0.f, 0.f, 0.f, 0.f) : acc[j];
    if (lane == 0) lse[row] = empty ? -INFINITY : L;
  }
}

}  // namespace

cudaError_t launch_lse_merge(const float* out_part, const float* lse_part, int n_splits, int rows,
                             int dv, float* out, float* lse, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // small blocks (one warp a row, two rows a block) spread the rows evenly over the SMs:
  // with eight-warp blocks a short merge gave some SMs a third more rows than others
  const int warps_per_block = 2;
  long long blocks = ((long long)rows + warps_per_block - 1) / warps_per_block;
  const long long cap = (long long)sms * 32;   // resident 64-thread blocks per SM
  if (blocks > cap) blocks = cap;
  const bool vec4 = (dv % 4) == 0;
  const bool fast = dv == 512 && n_splits <= kFastShards && (reinterpret_cast<uintptr_t>(out_part) % 16) == 0 &&
                    (reinterpret_cast<uintptr_t>(out) % 16) == 0;
  if (fast)
    lse_merge_fast_kernel<<<(int)blocks, warps_per_block * 32, 0, stream>>>(out_part, lse_part, n_splits, rows,
                                                                            out, lse);
  else if (vec4)
    lse_merge_kernel<true><<<(int)blocks, warps_per_block * 32, 0, stream>>>(
        out_part, lse_part, n_splits, rows, dv, out, lse);
  else
    lse_merge_kernel<false><<<(int)blocks, warps_per_block * 32, 0, stream>>>(
        out_part, lse_part, n_splits, rows, dv, out, lse);
  return cudaGetLastError();
}

}  // namespace sfa
