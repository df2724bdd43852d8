// (expert, token)-sorted expert maps from [T, K] expert indices (stand-alone
// kernels).  Declarations and contracts: moe_router.h.
//
// Three launches, deterministic (no global atomics):
//   1  count: a block takes 256 tokens (a warp per 32); every warp builds one
//      32-bit token mask per expert in shared memory; the block writes its
//      per-expert counts (popcounts summed over its warps).
//   2  column prefix: per expert, the counts of the blocks before each block
//      (in place) and the expert's total.
//   3  scatter: every block rebuilds its masks, scans the totals into the
//      expert offsets, and places each choice at
//        offset[e] + (earlier blocks) + (earlier warps) + (earlier lanes),
//      the last two from the masks.
#include <climits>
#include <cstddef>
#include <cstdint>

#include "moe_router.h"
#include "router_maps.cuh"

namespace moe_router {

constexpr int kMapsThreads = 256;
constexpr int kMapsWarps = kMapsThreads / 32;

__host__ __device__ inline int maps_blocks(int T) { return (T + kMapsThreads - 1) / kMapsThreads; }

// Token masks of the block's warps: masks[w * E + e] bit l = token
// blockIdx.x * 256 + 32 w + l chose expert e.  Entries outside [0, E) are
// left out.
__device__ __forceinline__ void build_masks(const int32_t* __restrict__ idx, long long ld, int T,
                                            int E, int K, uint32_t* masks) {
  for (int i = threadIdx.x; i < kMapsWarps * E; i += kMapsThreads) masks[i] = 0u;
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kMapsThreads + threadIdx.x;
  if (t < T) {
    const int32_t* row = idx + static_cast<size_t>(t) * ld;
    for (int k = 0; k < K; ++k) {
      const int e = row[k];
      if (e >= 0 && e < E) atomicOr(&masks[w * E + e], 1u << lane);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kMapsThreads)
maps_count_kernel(const int32_t* __restrict__ idx, long long ld, int T, int E, int K,
                  int* __restrict__ counts) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* masks = reinterpret_cast<uint32_t*>(smem);
  build_masks(idx, ld, T, E, K, masks);
  for (int e = threadIdx.x; e < E; e += kMapsThreads) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kMapsWarps; ++w) c += __popc(masks[w * E + e]);
    counts[static_cast<size_t>(blockIdx.x) * E + e] = c;
  }
}

__global__ void __launch_bounds__(kMapsThreads)
maps_colscan_kernel(int* __restrict__ counts, int nb, int E, int* __restrict__ totals) {
  const int e = blockIdx.x * kMapsThreads + threadIdx.x;
  if (e >= E) return;
  int run = 0;
#pragma unroll 4
  for (int b = 0; b < nb; ++b) {
    const size_t i = static_cast<size_t>(b) * E + e;
    const int c = counts[i];
    counts[i] = run;
    run += c;
  }
  totals[e] = run;
}

__global__ void __launch_bounds__(kMapsThreads)
maps_scatter_kernel(const int32_t* __restrict__ idx, long long ld, int T, int E, int K,
                    const int* __restrict__ colbase, const int* __restrict__ totals,
                    int32_t* __restrict__ offsets, int32_t* __restrict__ p2u,
                    int32_t* __restrict__ u2p, int32_t* __restrict__ pexp) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* masks = reinterpret_cast<uint32_t*>(smem);
  int* off = reinterpret_cast<int*>(masks + kMapsWarps * E);
  int* tmp = off + E;
  for (int e = threadIdx.x; e < E; e += kMapsThreads) off[e] = totals[e];
  build_masks(idx, ld, T, E, K, masks);  // its barriers also publish off[]
  const int total = block_exclusive_scan<kMapsThreads>(off, E, tmp);
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += kMapsThreads) offsets[e] = e < E ? off[e] : total;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kMapsThreads + threadIdx.x;
  if (t >= T) return;
  const int32_t* row = idx + static_cast<size_t>(t) * ld;
  const int* base = colbase + static_cast<size_t>(blockIdx.x) * E;
  const uint32_t below = (1u << lane) - 1u;
  for (int k = 0; k < K; ++k) {
    const int e = row[k];
    const int u = t + k * T;
    if (e < 0 || e >= E) {
      u2p[u] = -1;
      continue;
    }
    int p = off[e] + base[e] + __popc(masks[w * E + e] & below);
    for (int v = 0; v < w; ++v) p += __popc(masks[v * E + e]);
    p2u[p] = u;
    u2p[u] = p;
    pexp[p] = e;
  }
}

size_t maps_smem_count(int E) { return static_cast<size_t>(kMapsWarps) * E * 4; }
size_t maps_smem_scatter(int E) {
  return static_cast<size_t>(kMapsWarps) * E * 4 + static_cast<size_t>(E) * 4 +
         (kMapsWarps + 1) * 4;
}

// workspace: nb rows of E ints (counts, then column prefixes), then E totals
size_t maps_workspace_bytes(int T, int E) {
  return (static_cast<size_t>(maps_blocks(T)) + 1) * static_cast<size_t>(E) * 4u;
}

int maps_check(int T, int E, int K, int ld) {
  if (T < 0 || E < 1 || K < 1 || K > E || ld < K) return MR_ERR_INVALID;
  if (static_cast<long long>(T) * static_cast<long long>(E) > INT_MAX) return MR_ERR_INVALID;
  if (E > MR_MAX_EXPERTS || K > MR_MAX_TOPK) return MR_ERR_UNSUPPORTED;
  return MR_OK;
}

// The three launches; arguments checked by the caller.
int launch_expert_maps(const int32_t* idx, long long ld, int T, int E, int K, int32_t* offsets,
                       int32_t* p2u, int32_t* u2p, int32_t* pexp, void* workspace,
                       cudaStream_t st) {
  const int nb = maps_blocks(T);
  int* counts = static_cast<int*>(workspace);
  int* totals = counts + static_cast<size_t>(nb) * E;
  const size_t s1 = maps_smem_count(E), s3 = maps_smem_scatter(E);
  if (s1 > 48 * 1024 && cudaFuncSetAttribute(maps_count_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(s1)) != cudaSuccess)
    return MR_ERR_CUDA;
  if (s3 > 48 * 1024 && cudaFuncSetAttribute(maps_scatter_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(s3)) != cudaSuccess)
    return MR_ERR_CUDA;
  maps_count_kernel<<<nb, kMapsThreads, s1, st>>>(idx, ld, T, E, K, counts);
  maps_colscan_kernel<<<(E + kMapsThreads - 1) / kMapsThreads, kMapsThreads, 0, st>>>(
      counts, nb, E, totals);
  maps_scatter_kernel<<<nb, kMapsThreads, s3, st>>>(idx, ld, T, E, K, counts, totals, offsets,
                                                    p2u, u2p, pexp);
  return cudaGetLastError() == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

}  // namespace moe_router

using namespace moe_router;

extern "C" {

size_t router_expert_maps_workspace_bytes(int T, int E) {
  if (T <= 0 || E <= 0) return 0;
  return maps_workspace_bytes(T, E);
}

int router_expert_maps(const int32_t* topk_indices, int ld_indices, int T, int E, int K,
                       int32_t* expert_first_token_offset, int32_t* permuted_to_unpermuted,
                       int32_t* unpermuted_to_permuted, int32_t* permuted_experts,
                       void* workspace, size_t workspace_bytes, mr_stream_t stream) {
  const int rc = maps_check(T, E, K, ld_indices);
  if (rc != MR_OK) return rc;
  if (T == 0) return MR_OK;
  if (topk_indices == nullptr || expert_first_token_offset == nullptr ||
      permuted_to_unpermuted == nullptr || unpermuted_to_permuted == nullptr ||
      permuted_experts == nullptr || workspace == nullptr)
    return MR_ERR_INVALID;
  if (workspace_bytes < maps_workspace_bytes(T, E) ||
      (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
    return MR_ERR_INVALID;
  return launch_expert_maps(topk_indices, ld_indices, T, E, K, expert_first_token_offset,
                            permuted_to_unpermuted, unpermuted_to_permuted, permuted_experts,
                            workspace, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
