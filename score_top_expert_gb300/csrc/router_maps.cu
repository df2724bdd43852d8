// (expert, token)-sorted expert maps from [T, K] expert indices (stand-alone
// kernels).  Declarations and contracts: moe_router.h.
//
// Three launches, deterministic (no global atomics):
//   1  count: a block takes a tile of 64 tokens (a thread per token and per
//      quarter of its K choices); it builds one 64-bit token mask per
//      expert in shared memory and writes its per-expert counts (popcounts).
//   2  column prefix: per expert (a lane each), the counts of the tiles
//      before each tile (in place; 8 warps split the tiles, then add the
//      sums of the warps before them) and the expert's total; the last
//      block to finish (a counter in the workspace, zeroed by launch 1)
//      scans the totals into the expert offsets.
//   3  scatter: every block rebuilds its masks and places each choice at
//        offset[e] + (earlier tiles) + popcount(mask[e] below its token).
// When every tile's block fits on the GPU at once, the three phases run as
// one cooperative launch instead (after a one-block kernel that zeroes the
// barrier's counter), separated by a grid barrier (bounded in time like
// every wait of this library); the scatter reuses the masks of phase 1 from
// shared memory and each thread's choices from its registers, and adds the
// tile's column prefixes to the offsets in shared memory once per block.
#include <climits>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "moe_router.h"
#include "router_launch.cuh"
#include "router_maps.cuh"
#include "router_tma.cuh"

namespace moe_router {

constexpr int kMapsThreads = 256;
constexpr int kMapsTile = 64;                           // tokens per block
constexpr int kMapsSlots = kMapsThreads / kMapsTile;    // threads per token

__host__ __device__ inline int maps_blocks(int T) { return (T + kMapsTile - 1) / kMapsTile; }

constexpr int kMapsPerThread = (MR_MAX_TOPK + kMapsSlots - 1) / kMapsSlots;

// The choices k = slot, slot + 4, ... of token t, all loads issued before any
// use; -1 past K.
__device__ __forceinline__ void load_choices(const int32_t* __restrict__ idx, long long ld, int t,
                                             int K, int slot, int (&e)[kMapsPerThread]) {
  const int32_t* row = idx + static_cast<size_t>(t) * ld;
#pragma unroll
  for (int j = 0; j < kMapsPerThread; ++j) {
    const int k = slot + j * kMapsSlots;
    e[j] = k < K ? row[k] : -1;
  }
}

// masks[e] bit l: token blockIdx.x * 64 + l chose expert e.  Entries outside
// [0, E) are left out.
__device__ __forceinline__ void build_masks(const int32_t* __restrict__ idx, long long ld, int T,
                                            int E, int K, unsigned long long* masks) {
  for (int e = threadIdx.x; e < E; e += kMapsThreads) masks[e] = 0ull;
  __syncthreads();
  const int tl = threadIdx.x & (kMapsTile - 1), slot = threadIdx.x / kMapsTile;
  const int t = blockIdx.x * kMapsTile + tl;
  if (t < T) {
    int e[kMapsPerThread];
    load_choices(idx, ld, t, K, slot, e);
#pragma unroll
    for (int j = 0; j < kMapsPerThread; ++j)
      if (e[j] >= 0 && e[j] < E) atomicOr(&masks[e[j]], 1ull << tl);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kMapsThreads)
maps_count_kernel(const int32_t* __restrict__ idx, long long ld, int T, int E, int K,
                  int* __restrict__ counts, unsigned int* __restrict__ counter) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem[];
  if (blockIdx.x == 0 && threadIdx.x == 0) *counter = 0u;
  unsigned long long* masks = reinterpret_cast<unsigned long long*>(smem);
  build_masks(idx, ld, T, E, K, masks);
  for (int e = threadIdx.x; e < E; e += kMapsThreads)
    counts[static_cast<size_t>(blockIdx.x) * E + e] = __popcll(masks[e]);
}

__global__ void __launch_bounds__(kMapsThreads)
maps_colscan_kernel(int* __restrict__ counts, int nb, int E, int* __restrict__ totals,
                    unsigned int* __restrict__ counter, int32_t* __restrict__ offsets) {
  pdl_enter();
  constexpr int W = kMapsThreads / 32;
  constexpr int kBatch = 8;  // loads issued before the stores that depend on them
  __shared__ int wsum[W][32];
  __shared__ bool last;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const int per = (nb + W - 1) / W;
  const int b0 = w * per, b1 = min(nb, b0 + per);
  int run = 0;
  if (e < E) {
    for (int b = b0; b < b1; b += kBatch) {
      int c[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        c[j] = b + j < b1 ? counts[static_cast<size_t>(b + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (b + j < b1) counts[static_cast<size_t>(b + j) * E + e] = run;
        run += c[j];
      }
    }
  }
  wsum[w][lane] = run;
  __syncthreads();
  int base = 0;
  for (int v = 0; v < w; ++v) base += wsum[v][lane];
  if (e < E) {
    if (base != 0) {
      for (int b = b0; b < b1; b += kBatch) {
        int c[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
          c[j] = b + j < b1 ? counts[static_cast<size_t>(b + j) * E + e] : 0;
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
          if (b + j < b1) counts[static_cast<size_t>(b + j) * E + e] = c[j] + base;
      }
    }
    if (w == W - 1) totals[e] = base + run;
  }
  // the last block scans the experts' totals into their offsets
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last = atomicAdd(counter, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  extern __shared__ __align__(16) unsigned char smem[];
  int* off = reinterpret_cast<int*>(smem);
  int* tmp = off + E;
  for (int i = threadIdx.x; i < E; i += kMapsThreads) off[i] = __ldcg(totals + i);
  __syncthreads();
  const int total = block_exclusive_scan(off, E, tmp);
  for (int i = threadIdx.x; i <= E; i += kMapsThreads) offsets[i] = i < E ? off[i] : total;
}

__global__ void __launch_bounds__(kMapsThreads)
maps_scatter_kernel(const int32_t* __restrict__ idx, long long ld, int T, int E, int K,
                    const int* __restrict__ colbase, const int32_t* __restrict__ offsets,
                    int32_t* __restrict__ p2u, int32_t* __restrict__ u2p,
                    int32_t* __restrict__ pexp) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned long long* masks = reinterpret_cast<unsigned long long*>(smem);
  build_masks(idx, ld, T, E, K, masks);
  const int tl = threadIdx.x & (kMapsTile - 1), slot = threadIdx.x / kMapsTile;
  const int t = blockIdx.x * kMapsTile + tl;
  if (t >= T) return;
  const int* base = colbase + static_cast<size_t>(blockIdx.x) * E;
  const unsigned long long below = (1ull << tl) - 1ull;
  int ch[kMapsPerThread];
  load_choices(idx, ld, t, K, slot, ch);
  int pos[kMapsPerThread];
#pragma unroll
  for (int j = 0; j < kMapsPerThread; ++j) {  // gathers issued before any use
    const int e = ch[j];
    pos[j] = (e >= 0 && e < E) ? offsets[e] + base[e] : -1;
  }
#pragma unroll
  for (int j = 0; j < kMapsPerThread; ++j) {
    const int k = slot + j * kMapsSlots;
    if (k >= K) break;
    const int e = ch[j];
    const int u = t + k * T;
    if (pos[j] < 0) {
      u2p[u] = -1;
      continue;
    }
    const int p = pos[j] + __popcll(masks[e] & below);
    p2u[p] = u;
    u2p[u] = p;
    pexp[p] = e;
  }
}

// Grid-wide barrier of a cooperative launch (every block resident): the
// blocks add their arrivals to a counter zeroed before the launch; barrier
// number `gen` (1, 2, ...) is passed when the counter reaches gen blocks per
// block of the grid.  The wait gives up after kWaitLimitNs and records the
// timeout in the status word; every thread of the block returns the verdict.
__device__ __forceinline__ bool grid_barrier(unsigned int* count, unsigned int gen, int* status,
                                             int* verdict) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(count, 1u);
    const unsigned int target = gen * gridDim.x;
    int ok = 1;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
      if (v >= target) break;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicExch(status, kDeviceWaitTimeout);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    *verdict = ok;
  }
  __syncthreads();
  return *verdict != 0;
}

__global__ void __launch_bounds__(kMapsThreads, 3)
maps_fused_kernel(const int32_t* __restrict__ idx, long long ld, int T, int E, int K,
                  int* __restrict__ counts, int* __restrict__ totals,
                  unsigned int* __restrict__ barrier, int* __restrict__ status,
                  int32_t* __restrict__ offsets, int32_t* __restrict__ p2u,
                  int32_t* __restrict__ u2p, int32_t* __restrict__ pexp) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned long long* masks = reinterpret_cast<unsigned long long*>(smem);
  int* off = reinterpret_cast<int*>(masks + E);
  int* verdict = off + E;  // the barrier verdict
  int* tmp = verdict + 4;  // scan slots / per-warp prefix sums (8 x 32 ints)
  const int nb = gridDim.x;

  // ---- 1: this tile's choices (kept in registers for the scatter), masks
  //      and counts (the choice loads overlap the zeroing of the masks) ------
  const int tl = threadIdx.x & (kMapsTile - 1), slot = threadIdx.x / kMapsTile;
  const int t = blockIdx.x * kMapsTile + tl;
  int ch[kMapsPerThread];
  if (t < T) {
    load_choices(idx, ld, t, K, slot, ch);
  } else {
#pragma unroll
    for (int j = 0; j < kMapsPerThread; ++j) ch[j] = -1;
  }
  for (int e = threadIdx.x; e < E; e += kMapsThreads) masks[e] = 0ull;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kMapsPerThread; ++j)
    if (ch[j] >= 0 && ch[j] < E) atomicOr(&masks[ch[j]], 1ull << tl);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kMapsThreads)
    counts[static_cast<size_t>(blockIdx.x) * E + e] = __popcll(masks[e]);
  if (!grid_barrier(barrier, 1u, status, verdict)) return;

  // ---- 2: column prefixes: blocks take groups of 32 experts (a lane each),
  //      the 8 warps split the tiles (coalesced 128-byte rows); a warp sums
  //      its tiles' counts, then, after the sums of the warps before it,
  //      writes their exclusive prefixes (each pass loads 16 tiles at once) -
  {
    constexpr int W = kMapsThreads / 32;
    constexpr int B = 16;  // loads in flight per lane
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int* wsum = tmp;  // W x 32 ints, past the scan slots (sized in maps_smem_fused)
    const int per = (nb + W - 1) / W;
    const int b0 = min(nb, w * per), b1 = min(nb, b0 + per);
    for (int grp = blockIdx.x; grp * 32 < E; grp += nb) {
      const int e = grp * 32 + lane;
      int sum = 0;
      if (e < E) {
        for (int b = b0; b < b1; b += B) {
          int c[B];
#pragma unroll
          for (int j = 0; j < B; ++j)
            c[j] = b + j < b1 ? __ldcg(counts + static_cast<size_t>(b + j) * E + e) : 0;
#pragma unroll
          for (int j = 0; j < B; ++j) sum += c[j];
        }
      }
      wsum[w * 32 + lane] = sum;
      __syncthreads();
      int run = 0;
      for (int v = 0; v < w; ++v) run += wsum[v * 32 + lane];
      if (e < E) {
        if (w == W - 1) totals[e] = run + sum;
        for (int b = b0; b < b1; b += B) {
          int c[B];
#pragma unroll
          for (int j = 0; j < B; ++j)
            c[j] = b + j < b1 ? __ldcg(counts + static_cast<size_t>(b + j) * E + e) : 0;
#pragma unroll
          for (int j = 0; j < B; ++j) {
            if (b + j < b1) __stcg(counts + static_cast<size_t>(b + j) * E + e, run);
            run += c[j];
          }
        }
      }
      __syncthreads();
    }
  }
  if (!grid_barrier(barrier, 2u, status, verdict)) return;

  // ---- 3: offsets (every block), then this tile's scatter -------------------
  for (int e = threadIdx.x; e < E; e += kMapsThreads) off[e] = __ldcg(totals + e);
  __syncthreads();
  const int total = block_exclusive_scan(off, E, tmp);
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += kMapsThreads) offsets[e] = e < E ? off[e] : total;
  // each expert's first row for this tile: its offset plus the earlier tiles'
  // choices (the same thread reads off[e] above and updates it here)
  const int* base = counts + static_cast<size_t>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += kMapsThreads) off[e] += __ldcg(base + e);
  __syncthreads();
  if (t >= T) return;
  const unsigned long long below = (1ull << tl) - 1ull;
#pragma unroll
  for (int j = 0; j < kMapsPerThread; ++j) {
    const int k = slot + j * kMapsSlots;
    if (k >= K) break;
    const int e = ch[j];
    const int u = t + k * T;
    if (e < 0 || e >= E) {
      u2p[u] = -1;
      continue;
    }
    const int p = off[e] + __popcll(masks[e] & below);
    p2u[p] = u;
    u2p[u] = p;
    pexp[p] = e;
  }
}

size_t maps_smem_fused(int E) {
  return static_cast<size_t>(E) * 12 + 16 + (kMapsThreads / 32) * 32 * 4;
}

// Blocks of the fused kernel that fit on the current device at once (0 if
// cooperative launches are not available); cached per device and E.
int maps_fused_capacity(int E) {
  constexpr int kDevs = 64;
  static std::mutex mu;
  static int cache_E[kDevs] = {0};
  static int cache_n[kDevs] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache_E[dev] == E) return cache_n[dev];
  int coop = 0, sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, maps_fused_kernel, kMapsThreads,
                                                    maps_smem_fused(E)) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  const int n = coop ? per_sm * sms : 0;
  cache_n[dev] = n;
  cache_E[dev] = E;
  return n;
}

size_t maps_smem_count(int E) { return static_cast<size_t>(E) * 8; }
size_t maps_smem_colscan(int E) {
  return static_cast<size_t>(E) * 4 + (kMapsThreads / 32 + 1) * 4;
}
size_t maps_smem_scatter(int E) { return static_cast<size_t>(E) * 8; }

// workspace: nb rows of E ints (counts, then column prefixes), E totals,
// and the completion counter
size_t maps_workspace_bytes(int T, int E) {
  return (static_cast<size_t>(maps_blocks(T)) + 1) * static_cast<size_t>(E) * 4u + 16u;
}

int maps_check(int T, int E, int K, int ld) {
  if (T < 0 || E < 1 || K < 1 || K > E || ld < K) return MR_ERR_INVALID;
  if (static_cast<long long>(T) * static_cast<long long>(E) > INT_MAX) return MR_ERR_INVALID;
  if (E > MR_MAX_EXPERTS || K > MR_MAX_TOPK) return MR_ERR_UNSUPPORTED;
  return MR_OK;
}

// The maps on the stream: one cooperative launch when every tile's block
// fits on the GPU at once, else the three launches; arguments checked by the
// caller.
int launch_expert_maps(const int32_t* idx, long long ld, int T, int E, int K, int32_t* offsets,
                       int32_t* p2u, int32_t* u2p, int32_t* pexp, void* workspace,
                       cudaStream_t st) {
  const int nb = maps_blocks(T);
  int* counts = static_cast<int*>(workspace);
  int* totals = counts + static_cast<size_t>(nb) * E;
  unsigned int* counter = reinterpret_cast<unsigned int*>(totals + E);
  int* status = device_status_word();
  if (status != nullptr && nb <= maps_fused_capacity(E)) {
    // one cooperative launch: every tile's block is resident
    if (launch_zero_words(counter, 1, st) != cudaSuccess) return MR_ERR_CUDA;
    void* args[] = {&idx, &ld, &T, &E, &K, &counts, &totals, &counter, &status,
                    &offsets, &p2u, &u2p, &pexp};
    const cudaError_t e = cudaLaunchCooperativeKernel(
        reinterpret_cast<const void*>(maps_fused_kernel), dim3(nb), dim3(kMapsThreads), args,
        maps_smem_fused(E), st);
    if (e == cudaSuccess) return MR_OK;
    (void)cudaGetLastError();  // not launched: take the three launches below
  }
  // shared memory: at most 18 KB (E <= 2304), no opt-in needed
  cudaError_t e = launch_kernel(maps_count_kernel, dim3(nb), dim3(kMapsThreads),
                                maps_smem_count(E), st, idx, ld, T, E, K, counts, counter);
  if (e == cudaSuccess)
    e = launch_kernel(maps_colscan_kernel, dim3((E + 31) / 32), dim3(kMapsThreads),
                      maps_smem_colscan(E), st, counts, nb, E, totals, counter, offsets);
  if (e == cudaSuccess)
    e = launch_kernel(maps_scatter_kernel, dim3(nb), dim3(kMapsThreads), maps_smem_scatter(E),
                      st, idx, ld, T, E, K, static_cast<const int*>(counts),
                      static_cast<const int32_t*>(offsets), p2u, u2p, pexp);
  if (e != cudaSuccess) return MR_ERR_CUDA;
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
