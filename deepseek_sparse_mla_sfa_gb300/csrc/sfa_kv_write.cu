// sfa_kv_write.cu -- the latent-cache write: each new token's 1152-byte latent row goes
// to the cache slot slot_mapping[t] (the slot_mapping scatter of the fused pre-attention
// op: "RFC: MsModeling 支持 Decode Context Parallel 仿真", 2.1.4.1 and 1.3).
//
// One warp per token moves the row as 72 coalesced 16-byte words.  A negative slot is
// padding.  A slot past the cache writes nothing and sets the device status word.
#include "sfa_internal.h"

namespace sfa {
namespace {

constexpr int kRowWords = kDQK * 2 / 16;   // 72 x 16 bytes per latent row

__global__ void __launch_bounds__(256) kv_write_kernel(uint4* __restrict__ kv, long long num_slots,
                                                       const int32_t* __restrict__ slot_mapping,
                                                       const uint4* __restrict__ rows, int T, int* status) {
  const int t = (int)((blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const long long slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (lane == 0) report_status(status, kStatusBadBlock);
    return;
  }
  const uint4* src = rows + (size_t)t * kRowWords;
  uint4* dst = kv + (size_t)slot * kRowWords;
  for (int w = lane; w < kRowWords; w += 32) dst[w] = __ldg(src + w);
}

}  // namespace

cudaError_t launch_kv_write(void* kv, long long num_slots, const int32_t* slot_mapping, const void* rows, int T,
                            int* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int warps_per_block = 8;
  const unsigned grid = (unsigned)((T + warps_per_block - 1) / warps_per_block);
  kv_write_kernel<<<grid, 32 * warps_per_block, 0, stream>>>(static_cast<uint4*>(kv), num_slots, slot_mapping,
                                                               static_cast<const uint4*>(rows), T, status);
  return cudaGetLastError();
}

}  // namespace sfa
