// Load-balancing aux loss over the aux-score forward's outputs, and its
// backward.  Declarations and contracts: moe_router.h.
//
// Forward, two launches, deterministic (no atomics):
//   1  B blocks split the T rows; each thread owns experts e = t, t + 256,
//      ... and sums q[t, e] and map[t, e] over its block's rows (coalesced
//      row reads); the block writes its column partials to the workspace.
//   2  one block adds the B partials of every expert in a fixed order (in
//      double), writes tokens_per_expert, and reduces
//      loss = coeff E / (K T^2) * sum_e (sum_t q_te) * tokens_e.
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
constexpr int kAuxMaxBlocks = 256;
constexpr int kAuxCols = (MR_MAX_EXPERTS + kAuxThreads - 1) / kAuxThreads;  // per thread

__host__ __device__ inline int aux_blocks(int T) { return T < kAuxMaxBlocks ? T : kAuxMaxBlocks; }

// workspace: B rows of E float partial score sums, then B rows of E int counts
__host__ __device__ inline size_t aux_workspace_bytes(int T, int E) {
  return static_cast<size_t>(aux_blocks(T)) * static_cast<size_t>(E) * 8u;
}

__global__ void __launch_bounds__(kAuxThreads)
aux_loss_partial_kernel(const float* __restrict__ q, const uint8_t* __restrict__ map, int T,
                        int E, int rows_per_block, float* __restrict__ part_q,
                        int* __restrict__ part_n) {
  const int b = blockIdx.x;
  const int r0 = b * rows_per_block;
  const int r1 = min(T, r0 + rows_per_block);
  float acc_q[kAuxCols];
  int acc_n[kAuxCols];
#pragma unroll
  for (int i = 0; i < kAuxCols; ++i) { acc_q[i] = 0.0f; acc_n[i] = 0; }
#pragma unroll 2
  for (int r = r0; r < r1; ++r) {
    const size_t off = static_cast<size_t>(r) * static_cast<size_t>(E);
#pragma unroll
    for (int i = 0; i < kAuxCols; ++i) {
      const int e = threadIdx.x + kAuxThreads * i;
      if (e < E) {
        acc_q[i] += __ldcs(q + off + e);
        acc_n[i] += __ldcs(map + off + e) != 0;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kAuxCols; ++i) {
    const int e = threadIdx.x + kAuxThreads * i;
    if (e < E) {
      part_q[static_cast<size_t>(b) * E + e] = acc_q[i];
      part_n[static_cast<size_t>(b) * E + e] = acc_n[i];
    }
  }
}

__global__ void __launch_bounds__(kAuxThreads)
aux_loss_final_kernel(const float* __restrict__ part_q, const int* __restrict__ part_n,
                      int nblocks, int T, int E, int K, float coeff, float* __restrict__ loss,
                      int32_t* __restrict__ tokens) {
  __shared__ double red[kAuxThreads / 32];
  double term = 0.0;
  for (int e = threadIdx.x; e < E; e += kAuxThreads) {
    double cq = 0.0;
    long long cn = 0;
    for (int b = 0; b < nblocks; ++b) {
      cq += static_cast<double>(part_q[static_cast<size_t>(b) * E + e]);
      cn += part_n[static_cast<size_t>(b) * E + e];
    }
    tokens[e] = static_cast<int32_t>(cn);
    term += cq * static_cast<double>(cn);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = term;
  __syncthreads();
  if (threadIdx.x == 0) {
    double total = 0.0;
    for (int w = 0; w < kAuxThreads / 32; ++w) total += red[w];
    const double c = static_cast<double>(coeff) * E /
                     (static_cast<double>(K) * static_cast<double>(T) * static_cast<double>(T));
    loss[0] = static_cast<float>(c * total);
  }
}

template <bool VEC>
__global__ void __launch_bounds__(256)
aux_loss_bwd_kernel(const float* __restrict__ grad_loss, const int32_t* __restrict__ tokens,
                    int T, int E, float scale, float* __restrict__ grad) {
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

}  // namespace

// Allocation-free forward: the column partials live in this file-scope
// array instead of a caller workspace.  Its size is fixed: up to
// kNoAllocBlocks partial rows of MR_MAX_EXPERTS floats plus as many ints.
// Every GPU that loads the library holds it until the process exits.
constexpr int kNoAllocBlocks = MR_AUX_LOSS_NOALLOC_BLOCKS;
static_assert(MR_AUX_LOSS_NOALLOC_SCRATCH_BYTES ==
                  static_cast<size_t>(kNoAllocBlocks) * MR_MAX_EXPERTS * 8u,
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
  const int nb = aux_blocks(T);
  const int rows = (T + nb - 1) / nb;
  float* part_q = static_cast<float*>(workspace);
  int* part_n = reinterpret_cast<int*>(part_q + static_cast<size_t>(nb) * E);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  aux_loss_partial_kernel<<<nb, kAuxThreads, 0, st>>>(aux_scores, routing_map, T, E, rows, part_q,
                                                      part_n);
  aux_loss_final_kernel<<<1, kAuxThreads, 0, st>>>(part_q, part_n, nb, T, E, K, coeff, loss,
                                                   tokens_per_expert);
  return cudaGetLastError() == cudaSuccess ? MR_OK : MR_ERR_CUDA;
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
  if (vec)
    aux_loss_bwd_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        grad_loss, tokens_per_expert, T, E, scale, grad_aux_scores);
  else
    aux_loss_bwd_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        grad_loss, tokens_per_expert, T, E, scale, grad_aux_scores);
  return cudaGetLastError() == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

// Same two kernels as router_aux_loss_fwd, with at most kNoAllocBlocks
// partial rows.  Every partial the second kernel reads is written by the
// first kernel of the same call, so nothing in the scratch has to start at
// zero and a previous call's contents are never read.
int router_aux_loss_fwd_noalloc(const float* aux_scores, const uint8_t* routing_map, int T, int E,
                                int K, float coeff, float* loss, int32_t* tokens_per_expert,
                                mr_stream_t stream) {
  const int rc = aux_check(T, E, K);
  if (rc != MR_OK) return rc;
  const int nb = T < kNoAllocBlocks ? T : kNoAllocBlocks;
  if (static_cast<size_t>(nb) * static_cast<size_t>(E) * 8u > sizeof(g_aux_noalloc_scratch))
    return MR_ERR_UNSUPPORTED;
  if (T == 0) return MR_OK;
  if (aux_scores == nullptr || routing_map == nullptr || loss == nullptr ||
      tokens_per_expert == nullptr)
    return MR_ERR_INVALID;
  void* scratch = nullptr;
  const int sc = noalloc_scratch(&scratch);
  if (sc != MR_OK) return sc;
  const int rows = (T + nb - 1) / nb;
  float* part_q = static_cast<float*>(scratch);
  int* part_n = reinterpret_cast<int*>(part_q + static_cast<size_t>(nb) * E);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  aux_loss_partial_kernel<<<nb, kAuxThreads, 0, st>>>(aux_scores, routing_map, T, E, rows, part_q,
                                                      part_n);
  aux_loss_final_kernel<<<1, kAuxThreads, 0, st>>>(part_q, part_n, nb, T, E, K, coeff, loss,
                                                   tokens_per_expert);
  return cudaGetLastError() == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

}  // extern "C"
