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
    if (kVec4) {
      const int dv4 = dv >> 2;
      for (int c = lane; c < dv4; c += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < n; ++r) {
          const float w = __shfl_sync(0xffffffffu, r < 32 ? w0 : w1, r & 31);
          if (w == 0.f) continue;
          const float4 v =
              __ldg(reinterpret_cast<const float4*>(out_part + ((size_t)r * rows + row) * dv) + c);
          acc.x += w * v.x;
          acc.y += w * v.y;
          acc.z += w * v.z;
          acc.w += w * v.w;
        }
        reinterpret_cast<float4*>(orow)[c] = acc;
      }
    } else {
      for (int c = lane; c < dv; c += 32) {
        float acc = 0.f;
        for (int r = 0; r < n; ++r) {
          const float w = __shfl_sync(0xffffffffu, r < 32 ? w0 : w1, r & 31);
          if (w == 0.f) continue;
          acc += w * out_part[((size_t)r * rows + row) * dv + c];
        }
        orow[c] = acc;
      }
    }
    if (lane == 0) lse[row] = L;
  }
}

}  // namespace

cudaError_t launch_lse_merge(const float* out_part, const float* lse_part, int n_splits, int rows,
                             int dv, float* out, float* lse, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int warps_per_block = 8;
  long long blocks = ((long long)rows + warps_per_block - 1) / warps_per_block;
  const long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  const bool vec4 = (dv % 4) == 0;
  if (vec4)
    lse_merge_kernel<true><<<(int)blocks, warps_per_block * 32, 0, stream>>>(
        out_part, lse_part, n_splits, rows, dv, out, lse);
  else
    lse_merge_kernel<false><<<(int)blocks, warps_per_block * 32, 0, stream>>>(
        out_part, lse_part, n_splits, rows, dv, out, lse);
  return cudaGetLastError();
}

}  // namespace sfa
