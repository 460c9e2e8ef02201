// sfa_resolve.cuh -- device helpers shared by the tcgen05 decode kernels: resolving a
// token's selected positions to cache rows through the block table ("RFC: MsModeling
// 支持 Decode Context Parallel 仿真" 2.1.4.1: a position p of sequence b lives in row
// block_table[b, p / block_size] * block_size + p % block_size), and small arithmetic
// helpers of the online softmax.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "sfa_internal.h"

namespace sfa {

__device__ __forceinline__ int lanemask_lt() {
  int m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// 2^x on the special-function unit (inputs <= 8 here; -inf gives 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Physical cache row of selected entry `pos`, or -1 when the entry is padding for
// this shard (or its block-table entry is invalid, which is reported).
template <bool kInterleaved>
__device__ __forceinline__ int resolve_row(const DecodeParams& p, int bt_row, int pos, const ShardSel& sel,
                                           bool report) {
  if (!sel.has_fixed<kInterleaved>(pos)) return -1;
  const int blk = pos / p.block_size;
  const int phys = blk < p.max_blocks ? p.block_table[(size_t)bt_row * p.max_blocks + blk] : -1;
  if (phys < 0 || phys >= p.num_blocks) {
    if (report) report_status(p.status, kStatusBadBlock);
    return -1;
  }
  return phys * p.block_size + pos % p.block_size;
}

// One lane's share of a warp's chunk [c_begin, c_end) of the selected list, 8 entries
// per lane per round: counts the entries that resolve to a cache row of this unit and
// leaves the last round's rows in row_r (-1 for entries that do not).  The layout of the
// shards is a template argument so that the loop carries no per-entry branch on it.
template <bool kInterleaved>
__device__ __forceinline__ int resolve_chunk(const DecodeParams& p, const int32_t* idx, int c_begin, int c_end,
                                             int lane, const ShardSel& sel, int bt_row, bool report,
                                             int (&row_r)[8]) {
  int cnt = 0;
  for (int j0 = c_begin; j0 < c_end; j0 += 32 * 8) {
    int pos[8], blkv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int j = j0 + 32 * k + lane;
      pos[k] = j < c_end ? __ldg(idx + j) : -1;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const bool in = sel.has_fixed<kInterleaved>(pos[k]);
      const int blk = in ? pos[k] / p.block_size : 0;
      blkv[k] = in && blk < p.max_blocks ? __ldg(p.block_table + (size_t)bt_row * p.max_blocks + blk) : -2;
      if (!in) blkv[k] = -3;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      row_r[k] = -1;
      if (blkv[k] == -3) continue;
      if (blkv[k] < 0 || blkv[k] >= p.num_blocks) {
        if (report) report_status(p.status, kStatusBadBlock);
      } else {
        ++cnt;
        row_r[k] = blkv[k] * p.block_size + pos[k] % p.block_size;
      }
    }
  }
  return cnt;
}

}  // namespace sfa
