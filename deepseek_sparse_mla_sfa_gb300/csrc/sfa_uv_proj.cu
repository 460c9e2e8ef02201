// sfa_uv_proj.cu -- the W_UV up-projection that follows sparse MLA attention:
//   y[t, h, v] = sum_{c < 512} out[t, h, c] * W_UV[h, c, v],   v < 128
// (MLA attends in the 512-wide latent space; W_UV, derived from kv_b_proj, takes each
// head's latent output to its 128-wide value space: "RFC: Context Parallel Modeling for
// DeepSeek-Style Attention", 3.5).
//
// One CTA of 512 threads per (head, 64 query tokens) runs one tcgen05 contraction with
//   M = 128 output dims  (A = W_UV[h] as [v, c], loaded by TMA as an MN-major SW128 tile),
//   N = 64 tokens        (B = out[t0:t0+64, h, :] rounded to bf16 by the CTA's threads
//                         into a K-major SW128 tile),
//   K = 512              (32 MMAs of K = 16, fp32 accumulation in TMEM),
// and writes y in bf16.  Every wait is bounded; a wait that gives up records
// SFA_ERR_DEVICE_TIMEOUT and the CTA skips its stores.
#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "sfa_internal.h"
#include "sfa_ptx.cuh"

namespace sfa {
namespace {

using namespace ptx;

constexpr int kTok = 64;                  // tokens per CTA (MMA N)
constexpr int kVd = 128;                  // value head dim (MMA M)
constexpr int kC = kDV;                   // latent width (MMA K)
constexpr int kThreadsUV = 512;           // 16 warps: the whole out tile is in flight at once
constexpr int kWBlk = kC * 128;           // one 64-wide v block of W_UV[h]: 512 rows x 128 B
constexpr int kWBytes = 2 * kWBlk;        // 128 KB
constexpr int kOBlk = kTok * 128;         // one 64-column K block of the bf16 out tile
constexpr int kOBytes = (kC / 64) * kOBlk;   // 64 KB
constexpr int kSmemUV = kWBytes + kOBytes + 64 + 1024;   // + barriers and the TMEM address
constexpr long long kDrainLimitUV = 1LL << 40;

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreadsUV, 1)
    uv_proj_kernel(const __grid_constant__ CUtensorMap tmap_w, const float* __restrict__ out,
                   __nv_bfloat16* __restrict__ y, int T, int h, long long wait_limit, int stall, int* status) {
  extern __shared__ char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  char* w_s = smem;
  char* o_s = smem + kWBytes;
  // [0] W landed, [1] MMAs done, [2] never completed (the stall test hook waits on it)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWBytes + kOBytes);
  uint32_t* tmem_s = reinterpret_cast<uint32_t*>(bars + 3);
  const int head = blockIdx.y, t0 = blockIdx.x * kTok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 1);
    fence_barrier_init();
    // W_UV[h] as two 64-wide v blocks, each 512 rows of c (two 256-row boxes)
    mbar_arrive_expect_tx(&bars[0], kWBytes);
    for (int vb = 0; vb < 2; ++vb)
      for (int ch = 0; ch < 2; ++ch)
        tma_load_3d(smem_u32(w_s + vb * kWBlk + ch * (kWBlk / 2)), &tmap_w, 64 * vb, 256 * ch, head, &bars[0]);
  }
  if (warp == 0) {
    tmem_alloc(tmem_s, kTok);
    tmem_relinquish();
  }
  // out tile: token rows, 64 chunks of 8 columns each, rounded to bf16 into the K-major
  // SW128 layout (K block c / 64, chunk (c % 64) / 8 swizzled by the row).  Eight chunks
  // per thread are loaded before any is converted, so 16 loads per thread are in flight.
  constexpr int kChunks = kTok * (kC / 8);
  constexpr int kUnroll = 8;
  static_assert(kChunks % (kThreadsUV * kUnroll) == 0, "whole rounds");
#pragma unroll 1
  for (int i0 = threadIdx.x; i0 < kChunks; i0 += kThreadsUV * kUnroll) {
    float4 a[kUnroll], b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * kThreadsUV;
      const int tt = i / (kC / 8), ch = i % (kC / 8);
      const int t = t0 + tt;
      a[u] = b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < T) {
        const float4* src = reinterpret_cast<const float4*>(out + ((size_t)t * h + head) * kC + ch * 8);
        a[u] = __ldg(src);
        b[u] = __ldg(src + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * kThreadsUV;
      const int tt = i / (kC / 8), ch = i % (kC / 8);
      *reinterpret_cast<uint4*>(o_s + (ch >> 3) * kOBlk + tt * 128 + (((ch & 7) ^ (tt & 7)) * 16)) =
          make_uint4(pack2(a[u].x, a[u].y), pack2(a[u].z, a[u].w), pack2(b[u].x, b[u].y), pack2(b[u].z, b[u].w));
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_s;

  bool issued = false;
  if (threadIdx.x == 0) {
    if ((!stall || mbar_wait(&bars[2], 0, wait_limit)) && mbar_wait(&bars[0], 0, wait_limit)) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(kVd, kTok, 1, 0);   // A MN-major (v contiguous), B K-major
      const uint32_t wa = smem_u32(w_s), ob = smem_u32(o_s);
#pragma unroll
      for (int k = 0; k < kC / 16; ++k)
        mma_ss(tmem, smem_desc(wa + 2048 * k, kWBlk, 1024, kSwizzle128),
               smem_desc(ob + (k >> 2) * kOBlk + (k & 3) * 32, 16, 1024, kSwizzle128), id, k > 0 ? 1u : 0u);
      mma_commit(&bars[1]);
      issued = true;
    } else {
      report_status(status, kStatusTimeout);
    }
  }
  // epilogue: warp w holds output dims 32(w%4)..+31 (TMEM lanes) for tokens
  // 16(w/4)..+15 of the tile
  const bool done = __all_sync(0xffffffffu, mbar_wait(&bars[1], 0, wait_limit));
  tc_fence_after();
  if (done) {
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int v = (warp & 3) * 32 + lane;
#pragma unroll 1
    for (int c16 = warp >> 2; c16 < (warp >> 2) + 1; ++c16) {
      uint32_t r[16];
      tmem_ld16(lane_base + 16 * c16, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = t0 + 16 * c16 + j;
        if (t < T) y[((size_t)t * h + head) * kVd + v] = __float2bfloat16_rn(__uint_as_float(r[j]));
      }
    }
  } else if (threadIdx.x == 0) {
    report_status(status, kStatusTimeout);
  }
  // nothing of this CTA may still be in flight at exit: the W load and the MMAs
  if (threadIdx.x == 0) {
    if (!issued && !mbar_wait(&bars[0], 0, kDrainLimitUV)) report_status(status, kStatusTimeout);
    if (issued && !mbar_wait(&bars[1], 0, kDrainLimitUV)) report_status(status, kStatusTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTok);
}

typedef CUresult (*EncodeTiledFnUV)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnUV encode_fn_uv() {
  static std::once_flag once;
  static EncodeTiledFnUV fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnUV>(ptr);
  });
  return fn;
}

}  // namespace

cudaError_t launch_uv_proj(const float* out, const void* w_uv, void* y, int T, int h, long long wait_limit,
                           int stall, int* status, cudaStream_t stream) {
  if (T == 0 || h == 0) return cudaSuccess;
  EncodeTiledFnUV fn = encode_fn_uv();
  if (!fn) return cudaErrorInvalidValue;
  // W_UV [h, 512, 128] bf16 as (v, c, head); one box = 64 v x 256 c of one head
  CUtensorMap wmap;
  cuuint64_t dims[3] = {(cuuint64_t)kVd, (cuuint64_t)kC, (cuuint64_t)h};
  cuuint64_t strides[2] = {(cuuint64_t)kVd * 2, (cuuint64_t)kC * kVd * 2};
  cuuint32_t box[3] = {64, 256, 1};
  cuuint32_t es[3] = {1, 1, 1};
  if (fn(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w_uv), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[64];   // per device: set once (a repeat is harmless)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(uv_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemUV);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const dim3 grid((unsigned)((T + kTok - 1) / kTok), (unsigned)h);
  uv_proj_kernel<<<grid, kThreadsUV, kSmemUV, stream>>>(wmap, out, static_cast<__nv_bfloat16*>(y), T, h, wait_limit,
                                                        stall, status);
  return cudaGetLastError();
}

}  // namespace sfa
