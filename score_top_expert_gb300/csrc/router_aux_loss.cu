// Load-balancing aux loss over the aux-score forward's outputs, and its
// backward.  Declarations and contracts: moe_router.h.
//
// Forward: one launch, deterministic (fixed summation orders, compensated
// fp32 sums, no floating-point atomics).  The grid is B row ranges x G
// column groups of 128 experts (32 with scalar rows), B chosen so that the
// grid is one wave of three blocks on each SM (at most 64 ranges):
//   1  block (b, g): lane l owns the four experts of chunk 32 g + l, warp w
//      the rows w, w + 8, ... of range b (eight rows' loads in flight); the
//      8 warps combine in order and the block writes its partial row;
//   2  the last block of group g to finish (a counter per group, arrived on
//      with one acquire-release atomic) adds the B partial rows of its
//      experts (all of a warp's rows loaded at once), writes
//      tokens_per_expert and the group's share of
//        loss = coeff E / (K T^2) * sum_e (sum_t q_te) * tokens_e;
//   3  the last group to finish adds the shares in group order.
// The counters are zeroed by a one-block kernel on the stream before the
// launch.
// Backward: grad[t, e] = grad_loss * coeff E / (K T^2) * tokens_e, a pure
// streaming write (blocks stride over rows, threads over 16-byte chunks).
#include <atomic>
#include <climits>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "moe_router.h"
#include "router_common.cuh"

namespace moe_router {

constexpr int kAuxThreads = 256;
constexpr int kAuxWarps = kAuxThreads / 32;
constexpr int kAuxMaxBlocks = 64;  // row ranges (partial rows)
// Blocks a forward launch aims for: one wave of three blocks on each of the
// 152 SMs of a GB300 (fixed, so the summation order does not depend on the
// GPU).
constexpr int kAuxBlocksPerSm = 3;
constexpr int kAuxTargetBlocks = kAuxBlocksPerSm * 152;

__host__ __device__ inline int aux_blocks(int T) { return T < kAuxMaxBlocks ? T : kAuxMaxBlocks; }

// workspace: B rows of E float partial score sums, then B rows of E int
// counts, then the column groups' shares (fp32) and the completion counters
constexpr int kAuxSlots = 128;  // >= MR_MAX_EXPERTS / 32 + 1
constexpr size_t kAuxTailBytes = kAuxSlots * sizeof(float) + kAuxSlots * sizeof(int) + 16;
static_assert(kAuxSlots >= MR_MAX_EXPERTS / 32 + 1, "share and counter slots");

__host__ __device__ inline size_t aux_workspace_bytes(int T, int E) {
  return static_cast<size_t>(aux_blocks(T)) * static_cast<size_t>(E) * 8u + kAuxTailBytes;
}

struct AuxScratch {
  float* part_q;
  int* part_n;
  float* shares;            // one per column group
  unsigned int* counters;   // one per column group, then one for the groups
};

__host__ __device__ inline AuxScratch aux_scratch(void* base, int nb, int E) {
  AuxScratch s;
  s.part_q = static_cast<float*>(base);
  s.part_n = reinterpret_cast<int*>(s.part_q + static_cast<size_t>(nb) * E);
  s.shares = reinterpret_cast<float*>(s.part_n + static_cast<size_t>(nb) * E);
  s.counters = reinterpret_cast<unsigned int*>(s.shares + kAuxSlots);
  return s;
}

// Arrival on a completion counter: one acquire-release atomic add at GPU
// scope.  The release publishes the block's earlier writes (ordered before
// it by the block barrier that precedes the call); the acquire lets the
// block that arrives last read every other block's writes (the rest of its
// threads after the next block barrier).  Returns the previous count.
__device__ __forceinline__ unsigned int arrive_acq_rel(unsigned int* counter) {
  unsigned int old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
               : "=r"(old) : "l"(counter) : "memory");
  return old;
}

// Compensated (Kahan) fp32 addition: sum - c carries the running total.
__device__ __forceinline__ void kahan_add(float& sum, float& c, float v) {
  const float y = v - c;
  const float t = sum + y;
  c = (t - sum) - y;
  sum = t;
}

// Experts a lane owns: four consecutive ones (VEC: one float4 of q and four
// map bytes per row) or one.
template <bool VEC>
struct AuxLane {
  static constexpr int N = VEC ? 4 : 1;
  float q[N], c[N];
  int n[N];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < N; ++i) { q[i] = 0.0f; c[i] = 0.0f; n[i] = 0; }
  }
};

template <bool VEC>
__device__ __forceinline__ void aux_load(const float* __restrict__ q, const uint8_t* __restrict__ map,
                                         size_t off, float (&v)[AuxLane<VEC>::N], uint32_t& m) {
  if constexpr (VEC) {
    const float4 t = __ldcs(reinterpret_cast<const float4*>(q + off));
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    m = __ldcs(reinterpret_cast<const unsigned int*>(map + off));
  } else {
    v[0] = __ldcs(q + off);
    m = __ldcs(map + off);
  }
}

// Three blocks per SM (at most 80 registers a thread: the partial-row phase
// holds eight partial rows per lane in flight).
template <bool VEC>
__global__ void __launch_bounds__(kAuxThreads, kAuxBlocksPerSm)
aux_loss_kernel(const float* __restrict__ q, const uint8_t* __restrict__ map, int T, int E,
                int rows_per_block, float scale, AuxScratch ws, float* __restrict__ loss,
                int32_t* __restrict__ tokens) {
  pdl_enter();
  constexpr int N = AuxLane<VEC>::N;
  constexpr int kBatch = 8;   // rows whose loads precede any use
  constexpr int kBatch2 = 4;  // partial rows whose loads precede any use
  __shared__ float sq[kAuxWarps][32][N];  // per warp: sums (compensation folded in)
  __shared__ int sn[kAuxWarps][32][N];
  __shared__ bool last;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int b = blockIdx.x, g = blockIdx.y;
  const int e0 = (g * 32 + lane) * N;  // first expert of the lane
  const bool mine = e0 < E;
  const int nb = gridDim.x;

  // ---- 1: this block's rows -------------------------------------------------
  const int r0 = b * rows_per_block;
  const int r1 = min(T, r0 + rows_per_block);
  AuxLane<VEC> acc;
  acc.zero();
  if (mine) {
    for (int r = r0 + w; r < r1; r += kAuxWarps * kBatch) {
      float v[kBatch][N];
      uint32_t m[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int rj = r + j * kAuxWarps;
        if (rj < r1) {
          aux_load<VEC>(q, map, static_cast<size_t>(rj) * E + e0, v[j], m[j]);
        } else {
#pragma unroll
          for (int i = 0; i < N; ++i) v[j][i] = 0.0f;
          m[j] = 0u;
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
#pragma unroll
        for (int i = 0; i < N; ++i) {
          acc.q[i] += v[j][i];
          acc.n[i] += ((m[j] >> (8 * i)) & 0xffu) != 0;
        }
    }
  }
#pragma unroll
  for (int i = 0; i < N; ++i) { sq[w][lane][i] = acc.q[i]; sn[w][lane][i] = acc.n[i]; }
  __syncthreads();
  if (w == 0 && mine) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      float s = 0.0f, c = 0.0f;
      int n = 0;
#pragma unroll
      for (int v = 0; v < kAuxWarps; ++v) {
        kahan_add(s, c, sq[v][lane][i]);
        n += sn[v][lane][i];
      }
      acc.q[i] = s - c;
      acc.n[i] = n;
    }
    const size_t o = static_cast<size_t>(b) * E + e0;
    if constexpr (VEC) {  // E % 4 == 0: the lane's four experts all exist
      __stcg(reinterpret_cast<float4*>(ws.part_q + o),
             make_float4(acc.q[0], acc.q[1], acc.q[2], acc.q[3]));
      __stcg(reinterpret_cast<int4*>(ws.part_n + o),
             make_int4(acc.n[0], acc.n[1], acc.n[2], acc.n[3]));
    } else {
      ws.part_q[o] = acc.q[0];
      ws.part_n[o] = acc.n[0];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    last = arrive_acq_rel(&ws.counters[g]) == static_cast<unsigned>(nb) - 1u;
  }
  __syncthreads();
  if (!last) return;

  // ---- 2: the last block of group g adds the partial rows -------------------
  acc.zero();
  if constexpr (VEC) {
    // a warp's partial rows w, w + 8, ... (nb <= kAuxMaxBlocks: one batch),
    // added in that order
    constexpr int R = (kAuxMaxBlocks + kAuxWarps - 1) / kAuxWarps;
    if (mine) {
      float4 pq[R];
      int4 pn[R];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int bj = w + j * kAuxWarps;
        const size_t o = static_cast<size_t>(bj) * E + e0;
        pq[j] = bj < nb ? __ldcg(reinterpret_cast<const float4*>(ws.part_q + o))
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        pn[j] = bj < nb ? __ldcg(reinterpret_cast<const int4*>(ws.part_n + o))
                        : make_int4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (w + j * kAuxWarps < nb) {
          kahan_add(acc.q[0], acc.c[0], pq[j].x);
          kahan_add(acc.q[1], acc.c[1], pq[j].y);
          kahan_add(acc.q[2], acc.c[2], pq[j].z);
          kahan_add(acc.q[3], acc.c[3], pq[j].w);
          acc.n[0] += pn[j].x;
          acc.n[1] += pn[j].y;
          acc.n[2] += pn[j].z;
          acc.n[3] += pn[j].w;
        }
      }
    }
  } else if (mine) {
    for (int pb = w; pb < nb; pb += kAuxWarps * kBatch2) {
      float pq[kBatch2][N];
      int pn[kBatch2][N];
#pragma unroll
      for (int j = 0; j < kBatch2; ++j) {
        const int bj = pb + j * kAuxWarps;
#pragma unroll
        for (int i = 0; i < N; ++i) {
          const bool ok = bj < nb && e0 + i < E;
          const size_t o = static_cast<size_t>(bj) * E + e0 + i;
          pq[j][i] = ok ? __ldcg(ws.part_q + o) : 0.0f;
          pn[j][i] = ok ? __ldcg(ws.part_n + o) : 0;
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch2; ++j)
#pragma unroll
        for (int i = 0; i < N; ++i) {
          kahan_add(acc.q[i], acc.c[i], pq[j][i]);
          acc.n[i] += pn[j][i];
        }
    }
  }
#pragma unroll
  for (int i = 0; i < N; ++i) {
    sq[w][lane][i] = acc.q[i] - acc.c[i];
    sn[w][lane][i] = acc.n[i];
  }
  __syncthreads();
  if (w == 0) {
    float term = 0.0f;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      float s = 0.0f, c = 0.0f;
      int n = 0;
#pragma unroll
      for (int v = 0; v < kAuxWarps; ++v) {
        kahan_add(s, c, sq[v][lane][i]);
        n += sn[v][lane][i];
      }
      const int e = e0 + i;
      if (e < E) {
        tokens[e] = n;
        term += (s - c) * static_cast<float>(n);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
    if (lane == 0) {
      ws.shares[g] = term;
      last = arrive_acq_rel(&ws.counters[gridDim.y]) == gridDim.y - 1u;
    }
  }
  __syncthreads();

  // ---- 3: the last group adds the shares in order ---------------------------
  // (warp 0 loads them all at once and every lane adds them in group order)
  if (last && w == 0) {
    const int G = static_cast<int>(gridDim.y);
    float total = 0.0f, comp = 0.0f;
    for (int c0 = 0; c0 < G; c0 += 32) {
      const float sh = c0 + lane < G ? __ldcg(ws.shares + c0 + lane) : 0.0f;
      const int m = G - c0 < 32 ? G - c0 : 32;
      for (int j = 0; j < m; ++j) kahan_add(total, comp, __shfl_sync(0xffffffffu, sh, j));
    }
    if (lane == 0) loss[0] = scale * (total - comp);
  }
}

template <bool VEC>
__global__ void __launch_bounds__(256)
aux_loss_bwd_kernel(const float* __restrict__ grad_loss, const int32_t* __restrict__ tokens,
                    int T, int E, float scale, float* __restrict__ grad) {
  pdl_enter();
  const float gl = grad_loss[0] * scale;
  for (int row = blockIdx.x; row < T; row += gridDim.x) {
    float* out = grad + static_cast<size_t>(row) * E;
    if constexpr (VEC) {  // E % 4 == 0, 16-byte aligned rows
      for (int c = threadIdx.x; c < (E >> 2); c += blockDim.x) {
        const int4 tk = reinterpret_cast<const int4*>(tokens)[c];
        __stcs(reinterpret_cast<float4*>(out) + c,
               make_float4(gl * tk.x, gl * tk.y, gl * tk.z, gl * tk.w));
      }
    } else {
      for (int e = threadIdx.x; e < E; e += blockDim.x)
        __stcs(out + e, gl * static_cast<float>(tokens[e]));
    }
  }
}

namespace {

int aux_check(int T, int E, int K) {
  if (T < 0 || E < 1 || K < 1 || K > E) return MR_ERR_INVALID;
  if (static_cast<long long>(T) * static_cast<long long>(E) > INT_MAX) return MR_ERR_INVALID;
  if (E > MR_MAX_EXPERTS) return MR_ERR_UNSUPPORTED;
  return MR_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

// The forward with its partial rows in the scratch at `scratch` (at least
// aux_workspace_bytes(T, E) bytes, 16-byte aligned): a one-block kernel that
// zeroes the completion counters, then the forward.  The number of row
// ranges depends on T, E and the row layout only, so both entry points (and
// every GPU) sum in the same order.
int launch_aux_loss(const float* q, const uint8_t* map, int T, int E, int K, float coeff,
                    float* loss, int32_t* tokens, void* scratch, cudaStream_t st) {
  const bool vec = E % 4 == 0 && aligned16(q) && (reinterpret_cast<uintptr_t>(map) & 3u) == 0;
  const int per_group = vec ? 128 : 32;
  const int groups = (E + per_group - 1) / per_group;
  int nb = kAuxTargetBlocks / groups;
  if (nb < 1) nb = 1;
  if (nb > aux_blocks(T)) nb = aux_blocks(T);
  const int rows = (T + nb - 1) / nb;
  const AuxScratch ws = aux_scratch(scratch, nb, E);
  const float scale = static_cast<float>(static_cast<double>(coeff) * E /
                                         (static_cast<double>(K) * T * static_cast<double>(T)));
  if (launch_zero_words(ws.counters, groups + 1, st) != cudaSuccess) return MR_ERR_CUDA;
  const dim3 grid(nb, groups);
  const cudaError_t e =
      vec ? launch_kernel(aux_loss_kernel<true>, grid, dim3(kAuxThreads), 0, st, q, map, T, E,
                          rows, scale, ws, loss, tokens)
          : launch_kernel(aux_loss_kernel<false>, grid, dim3(kAuxThreads), 0, st, q, map, T, E,
                          rows, scale, ws, loss, tokens);
  return e == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

}  // namespace

// Allocation-free forward: the column partials live in this file-scope
// array instead of a caller workspace.  Its size is fixed: up to
// kNoAllocBlocks partial rows of MR_MAX_EXPERTS floats plus as many ints,
// and the final blocks' shares and counter.
// Every GPU that loads the library holds it until the process exits.
constexpr int kNoAllocBlocks = MR_AUX_LOSS_NOALLOC_BLOCKS;
static_assert(MR_AUX_LOSS_NOALLOC_SCRATCH_BYTES ==
                  static_cast<size_t>(kNoAllocBlocks) * MR_MAX_EXPERTS * 8u + kAuxTailBytes,
              "scratch size stated in the header");
static __device__ __align__(256) unsigned char
    g_aux_noalloc_scratch[MR_AUX_LOSS_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::atomic<void*> g_noalloc_ptr[kNoAllocMaxDevices];
std::mutex g_noalloc_setup;

// Device address of the scratch array on the current device.  In host code
// g_aux_noalloc_scratch names a host-side stand-in, so the address comes
// from the runtime, once per device, with that device current.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return MR_ERR_CUDA;
  }
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MR_ERR_UNSUPPORTED;
  void* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_noalloc_setup);
    p = g_noalloc_ptr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      if (cudaGetSymbolAddress(&p, g_aux_noalloc_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return MR_ERR_CUDA;
      }
      g_noalloc_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return MR_OK;
}

}  // namespace
}  // namespace moe_router

using namespace moe_router;

extern "C" {

size_t router_aux_loss_workspace_bytes(int T, int E) {
  if (T <= 0 || E <= 0) return 0;
  return aux_workspace_bytes(T, E);
}

int router_aux_loss_fwd(const float* aux_scores, const uint8_t* routing_map, int T, int E, int K,
                        float coeff, float* loss, int32_t* tokens_per_expert, void* workspace,
                        size_t workspace_bytes, mr_stream_t stream) {
  const int rc = aux_check(T, E, K);
  if (rc != MR_OK) return rc;
  if (T == 0) return MR_OK;
  if (aux_scores == nullptr || routing_map == nullptr || loss == nullptr ||
      tokens_per_expert == nullptr || workspace == nullptr)
    return MR_ERR_INVALID;
  if (workspace_bytes < aux_workspace_bytes(T, E) || !aligned16(workspace)) return MR_ERR_INVALID;
  return launch_aux_loss(aux_scores, routing_map, T, E, K, coeff, loss, tokens_per_expert,
                         workspace, reinterpret_cast<cudaStream_t>(stream));
}

int router_aux_loss_bwd(const float* grad_loss, const int32_t* tokens_per_expert, int T, int E,
                        int K, float coeff, float* grad_aux_scores, mr_stream_t stream) {
  const int rc = aux_check(T, E, K);
  if (rc != MR_OK) return rc;
  if (T == 0) return MR_OK;
  if (grad_loss == nullptr || tokens_per_expert == nullptr || grad_aux_scores == nullptr)
    return MR_ERR_INVALID;
  const float scale = static_cast<float>(static_cast<double>(coeff) * E /
                                         (static_cast<double>(K) * T * static_cast<double>(T)));
  const int sms = sm_count();
  if (sms <= 0) return MR_ERR_CUDA;
  const bool vec = E % 4 == 0 && aligned16(grad_aux_scores) && aligned16(tokens_per_expert);
  long long blocks = T;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const dim3 g(static_cast<unsigned>(blocks));
  const cudaError_t e =
      vec ? launch_kernel(aux_loss_bwd_kernel<true>, g, dim3(256), 0, st, grad_loss,
                          tokens_per_expert, T, E, scale, grad_aux_scores)
          : launch_kernel(aux_loss_bwd_kernel<false>, g, dim3(256), 0, st, grad_loss,
                          tokens_per_expert, T, E, scale, grad_aux_scores);
  if (e != cudaSuccess) return MR_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

// The same launches as router_aux_loss_fwd (the same number of partial
// rows, at most aux_blocks(T) <= kNoAllocBlocks).  Every partial the launch
// reads is written by its own blocks, and the call zeroes the completion
// counters first, so nothing in the scratch has to start at zero and a
// previous call's contents are never read.
int router_aux_loss_fwd_noalloc(const float* aux_scores, const uint8_t* routing_map, int T, int E,
                                int K, float coeff, float* loss, int32_t* tokens_per_expert,
                                mr_stream_t stream) {
  const int rc = aux_check(T, E, K);
  if (rc != MR_OK) return rc;
  static_assert(kAuxMaxBlocks <= kNoAllocBlocks, "partial rows of the scratch array");
  // Cannot fire while aux_check caps E at MR_MAX_EXPERTS (the array is sized
  // for that E and kNoAllocBlocks rows); kept as a guard should either limit
  // change.
  if (aux_workspace_bytes(T, E) > sizeof(g_aux_noalloc_scratch)) return MR_ERR_UNSUPPORTED;
  if (T == 0) return MR_OK;
  if (aux_scores == nullptr || routing_map == nullptr || loss == nullptr ||
      tokens_per_expert == nullptr)
    return MR_ERR_INVALID;
  void* scratch = nullptr;
  const int sc = noalloc_scratch(&scratch);
  if (sc != MR_OK) return sc;
  return launch_aux_loss(aux_scores, routing_map, T, E, K, coeff, loss, tokens_per_expert,
                         scratch, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
