// (expert, token)-sorted expert maps of the top-K choices: device helpers
// shared by the stand-alone maps kernels and the fused decode forward.
//
// The T K choices are ordered by expert, then token (a token picks an expert
// at most once).  A choice's permuted row is
//   offset[e] + (choices of e by earlier tokens),
// and the tokens of a tile of 32 that chose e are the set bits of one 32-bit
// mask per expert, built with shared-memory atomicOr, so the count among
// earlier tokens of the tile is a popcount of the mask below the token's bit.
#pragma once

#include "router_common.cuh"

namespace moe_router {

// Exclusive prefix sums of v[0..n) in place (shared memory); every thread of
// the block (a multiple of 32 threads, at most 1024) calls it.  Thread i owns
// the contiguous run i*per .. i*per+per-1.  tmp: blockDim.x / 32 + 1 ints of
// shared memory.  Returns the total.
__device__ __forceinline__ int block_exclusive_scan(int* v, int n, int* tmp) {
  const int nthreads = blockDim.x;
  const int per = (n + nthreads - 1) / nthreads;
  const int b0 = threadIdx.x * per;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int local = 0;
  for (int i = 0; i < per; ++i)
    if (b0 + i < n) local += v[b0 + i];
  int x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  const int W = nthreads / 32;
  if (warp == 0) {
    const int w = lane < W ? tmp[lane] : 0;
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < W) tmp[lane] = s - w;
    if (lane == W - 1) tmp[W] = s;
  }
  __syncthreads();
  int run = tmp[warp] + x - local;
  for (int i = 0; i < per; ++i) {
    if (b0 + i < n) {
      const int c = v[b0 + i];
      v[b0 + i] = run;
      run += c;
    }
  }
  const int total = tmp[W];
  __syncthreads();
  return total;
}

// Maps of at most 32 tokens in one block (the fused decode forward).  idx:
// the block's own compact indices ([T, ld_i], written before a
// __syncthreads); smem: 2 E + blockDim.x / 32 + 1 ints.
__device__ __forceinline__ void expert_maps_block(const int32_t* idx, long long ld_i, int T,
                                                  int E, int K, int* smem, int32_t* offsets,
                                                  int32_t* p2u, int32_t* u2p, int32_t* pexp) {
  uint32_t* mask = reinterpret_cast<uint32_t*>(smem);  // [E]: tokens that chose e
  int* off = smem + E;                                 // [E]
  int* tmp = smem + 2 * E;
  const int n = T * K;
  const int nthreads = blockDim.x;
  for (int e = threadIdx.x; e < E; e += nthreads) mask[e] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += nthreads) {
    const int t = i / K, k = i - t * K;
    atomicOr(&mask[idx[t * ld_i + k]], 1u << t);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += nthreads) off[e] = __popc(mask[e]);
  __syncthreads();
  const int total = block_exclusive_scan(off, E, tmp);
  for (int e = threadIdx.x; e <= E; e += nthreads) offsets[e] = e < E ? off[e] : total;
  for (int i = threadIdx.x; i < n; i += nthreads) {
    const int t = i / K, k = i - t * K;
    const int e = idx[t * ld_i + k];
    const int p = off[e] + __popc(mask[e] & ((1u << t) - 1u));
    p2u[p] = t + k * T;
    u2p[t + k * T] = p;
    pexp[p] = e;
  }
}

}  // namespace moe_router
