// Load-balancing aux loss over the aux-score forward's outputs, and its
// backward.  Declarations and contracts: moe_router.h.
//
// Forward, two launches, deterministic (no floating-point atomics):
//   1  B blocks split the T rows; each thread owns four consecutive experts
//      (one float4 of q, four map bytes per row; unaligned rows: experts
//      e = t, t + 256, ...) and sums q[t, e] and map[t, e] over its block's
//      rows (coalesced row reads); the block writes its column partials to
//      the workspace.
//   2  E / 32 blocks, a lane per expert: the block's 8 warps add the B
//      partials of its 32 experts (warp w takes partial rows w, w + 8, ...,
//      coalesced; compensated fp32 sums), combine them in a fixed order,
//      write tokens_per_expert and the block's share (in double) of
//        loss = coeff E / (K T^2) * sum_e (sum_t q_te) * tokens_e;
//      the last block to finish (a counter in the workspace, zeroed by
//      launch 1) adds the shares in block order and writes the loss.
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

// workspace: B rows of E float partial score sums, then B rows of E int
// counts, then the final blocks' shares (doubles) and the completion counter
constexpr int kAuxFinalExperts = 32;  // experts per final block (a lane each)
constexpr int kAuxShareSlots = 128;   // >= MR_MAX_EXPERTS / kAuxFinalExperts
constexpr size_t kAuxTailBytes = kAuxShareSlots * sizeof(double) + 16;
static_assert(kAuxShareSlots * kAuxFinalExperts >= MR_MAX_EXPERTS, "share slots");

__host__ __device__ inline size_t aux_workspace_bytes(int T, int E) {
  return static_cast<size_t>(aux_blocks(T)) * static_cast<size_t>(E) * 8u + kAuxTailBytes;
}

struct AuxScratch {
  float* part_q;
  int* part_n;
  double* shares;
  unsigned int* counter;
};

__host__ __device__ inline AuxScratch aux_scratch(void* base, int nb, int E) {
  AuxScratch s;
  s.part_q = static_cast<float*>(base);
  s.part_n = reinterpret_cast<int*>(s.part_q + static_cast<size_t>(nb) * E);
  s.shares = reinterpret_cast<double*>(s.part_n + static_cast<size_t>(nb) * E);
  s.counter = reinterpret_cast<unsigned int*>(s.shares + kAuxShareSlots);
  return s;
}

__global__ void __launch_bounds__(kAuxThreads)
aux_loss_partial_kernel(const float* __restrict__ q, const uint8_t* __restrict__ map, int T,
                        int E, int rows_per_block, AuxScratch ws) {
  const int b = blockIdx.x;
  if (b == 0 && threadIdx.x == 0) *ws.counter = 0u;
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
      ws.part_q[static_cast<size_t>(b) * E + e] = acc_q[i];
      ws.part_n[static_cast<size_t>(b) * E + e] = acc_n[i];
    }
  }
}

// Vector form of the partial sums (E % 4 == 0, 16-byte aligned q): thread
// (blockIdx.y, threadIdx.x) owns the four experts of chunk
// blockIdx.y * 256 + threadIdx.x and reads one float4 of q and four map
// bytes per row, eight rows in flight.
__global__ void __launch_bounds__(kAuxThreads)
aux_loss_partial_vec_kernel(const float* __restrict__ q, const uint8_t* __restrict__ map, int T,
                            int E, int rows_per_block, AuxScratch ws) {
  const int b = blockIdx.x;
  if (b == 0 && blockIdx.y == 0 && threadIdx.x == 0) *ws.counter = 0u;
  const int c = blockIdx.y * kAuxThreads + threadIdx.x;
  if (4 * c >= E) return;
  const int r0 = b * rows_per_block;
  const int r1 = min(T, r0 + rows_per_block);
  float4 aq = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  int n0 = 0, n1 = 0, n2 = 0, n3 = 0;
  const float4* q4 = reinterpret_cast<const float4*>(q);
  const uint32_t* m4 = reinterpret_cast<const uint32_t*>(map);
  const size_t stride = static_cast<size_t>(E) >> 2;
#pragma unroll 8
  for (int r = r0; r < r1; ++r) {
    const size_t i = static_cast<size_t>(r) * stride + c;
    const float4 v = __ldcs(q4 + i);
    const uint32_t m = __ldcs(m4 + i);
    aq.x += v.x; aq.y += v.y; aq.z += v.z; aq.w += v.w;
    n0 += (m & 0xffu) != 0;
    n1 += (m & 0xff00u) != 0;
    n2 += (m & 0xff0000u) != 0;
    n3 += (m & 0xff000000u) != 0;
  }
  const size_t o = static_cast<size_t>(b) * E + 4 * c;
  *reinterpret_cast<float4*>(ws.part_q + o) = aq;
  *reinterpret_cast<int4*>(ws.part_n + o) = make_int4(n0, n1, n2, n3);
}

// Compensated (Kahan) fp32 addition: sum + c carries the running total.
__device__ __forceinline__ void kahan_add(float& sum, float& c, float v) {
  const float y = v - c;
  const float t = sum + y;
  c = (t - sum) - y;
  sum = t;
}

__global__ void __launch_bounds__(kAuxThreads)
aux_loss_final_kernel(AuxScratch ws, int nblocks, int T, int E, int K, float coeff,
                      float* __restrict__ loss, int32_t* __restrict__ tokens) {
  constexpr int W = kAuxThreads / 32;
  __shared__ float sq[W][32];
  __shared__ float sc[W][32];
  __shared__ int sn[W][32];
  __shared__ bool last;
  __shared__ double sh[kAuxShareSlots];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int e = blockIdx.x * kAuxFinalExperts + lane;
  // per expert: the partials of rows w, w + 8, ... (fp32, compensated; the
  // fp64 pipe of this part is far too narrow for a per-partial double add)
  float cq = 0.0f, cc = 0.0f;
  int cn = 0;
  if (e < E) {
#pragma unroll 8
    for (int b = w; b < nblocks; b += W) {
      kahan_add(cq, cc, ws.part_q[static_cast<size_t>(b) * E + e]);
      cn += ws.part_n[static_cast<size_t>(b) * E + e];
    }
  }
  sq[w][lane] = cq;
  sc[w][lane] = cc;
  sn[w][lane] = cn;
  __syncthreads();
  if (w == 0) {
    float colq = 0.0f, colc = 0.0f;
    int coln = 0;
#pragma unroll
    for (int v = 0; v < W; ++v) {
      kahan_add(colq, colc, sq[v][lane]);
      kahan_add(colq, colc, -sc[v][lane]);
      coln += sn[v][lane];
    }
    double term = 0.0;
    if (e < E) {
      tokens[e] = coln;
      term = (static_cast<double>(colq) - static_cast<double>(colc)) * static_cast<double>(coln);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
    if (lane == 0) {
      ws.shares[blockIdx.x] = term;
      __threadfence();
      last = atomicAdd(ws.counter, 1u) == gridDim.x - 1;
    }
  }
  __syncthreads();
  if (!last) return;
  // the last block: read every block's share at once, add them in order
  __threadfence();
  for (int j = threadIdx.x; j < static_cast<int>(gridDim.x); j += kAuxThreads)
    sh[j] = __ldcg(ws.shares + j);
  __syncthreads();
  if (threadIdx.x == 0) {
    double total = 0.0;
    for (int j = 0; j < static_cast<int>(gridDim.x); ++j) total += sh[j];
    const double c = static_cast<double>(coeff) * E /
                     (static_cast<double>(K) * static_cast<double>(T) * static_cast<double>(T));
    loss[0] = static_cast<float>(c * total);
    *ws.counter = 0u;
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

// The two forward launches over nb partial rows in the scratch ws.
int launch_aux_loss(const float* q, const uint8_t* map, int T, int E, int K, float coeff,
                    float* loss, int32_t* tokens, const AuxScratch& ws, int nb, cudaStream_t st) {
  const int rows = (T + nb - 1) / nb;
  // the vector form also needs 16-byte aligned partial rows (E % 4 == 0
  // keeps every row of the scratch aligned when its base is)
  if (E % 4 == 0 && aligned16(q) && (reinterpret_cast<uintptr_t>(map) & 3u) == 0 &&
      aligned16(ws.part_q)) {
    const dim3 grid(nb, (E / 4 + kAuxThreads - 1) / kAuxThreads);
    aux_loss_partial_vec_kernel<<<grid, kAuxThreads, 0, st>>>(q, map, T, E, rows, ws);
  } else {
    aux_loss_partial_kernel<<<nb, kAuxThreads, 0, st>>>(q, map, T, E, rows, ws);
  }
  const int nfinal = (E + kAuxFinalExperts - 1) / kAuxFinalExperts;
  aux_loss_final_kernel<<<nfinal, kAuxThreads, 0, st>>>(ws, nb, T, E, K, coeff, loss, tokens);
  return cudaGetLastError() == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

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
  const int nb = aux_blocks(T);
  return launch_aux_loss(aux_scores, routing_map, T, E, K, coeff, loss, tokens_per_expert,
                         aux_scratch(workspace, nb, E), nb,
                         reinterpret_cast<cudaStream_t>(stream));
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
// first kernel of the same call, which also zeroes the completion counter,
// so nothing in the scratch has to start at zero and a previous call's
// contents are never read.
int router_aux_loss_fwd_noalloc(const float* aux_scores, const uint8_t* routing_map, int T, int E,
                                int K, float coeff, float* loss, int32_t* tokens_per_expert,
                                mr_stream_t stream) {
  const int rc = aux_check(T, E, K);
  if (rc != MR_OK) return rc;
  const int nb = T < kNoAllocBlocks ? T : kNoAllocBlocks;
  if (static_cast<size_t>(nb) * static_cast<size_t>(E) * 8u + kAuxTailBytes >
      sizeof(g_aux_noalloc_scratch))
    return MR_ERR_UNSUPPORTED;
  if (T == 0) return MR_OK;
  if (aux_scores == nullptr || routing_map == nullptr || loss == nullptr ||
      tokens_per_expert == nullptr)
    return MR_ERR_INVALID;
  void* scratch = nullptr;
  const int sc = noalloc_scratch(&scratch);
  if (sc != MR_OK) return sc;
  return launch_aux_loss(aux_scores, routing_map, T, E, K, coeff, loss, tokens_per_expert,
                         aux_scratch(scratch, nb, E), nb, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
