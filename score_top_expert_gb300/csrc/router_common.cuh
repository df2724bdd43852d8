// Device helpers shared by the router kernels: element loads/stores in the
// logits dtype, order-preserving float keys and reductions over a "segment"
// (the SEG consecutive lanes of a warp that own one token row).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdlib>
#include <cstring>
#include <utility>

#include "moe_router.h"

namespace moe_router {

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every router kernel is launched with
// programmatic stream serialization (unless MOE_ROUTER_PDL=0), so that its
// blocks may be scheduled while the previous kernel in the stream drains;
// each kernel waits in pdl_wait(), before its first global memory access,
// until that kernel has completed and its writes are visible.  No-op for a
// plain launch.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Kernel entry: wait for the previous kernel only.  The next kernel is let
// in as this one's blocks exit (no early trigger: a persistent kernel's
// dependents would otherwise sit resident beside it).
__device__ __forceinline__ void pdl_enter() { pdl_wait(); }

inline bool pdl_enabled() {
  static const bool on = [] {
    const char* env = std::getenv("MOE_ROUTER_PDL");
    return env == nullptr || std::strcmp(env, "0") != 0;
  }();
  return on;
}

// Launch `kern` on `st` (with programmatic stream serialization when
// enabled); returns the launch status.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Zeroes n words at p (one block of up to 1024 threads, n <= 1024).  Calls
// that need zeroed counters launch it instead of a memset: in a stream or a
// CUDA graph a memset costs several times a kernel launch between two
// kernels, and unlike a memset this launch takes part in the programmatic
// serialization above.
template <typename Word>
__global__ void zero_words_kernel(Word* __restrict__ p, int n) {
  pdl_enter();
  if (static_cast<int>(threadIdx.x) < n) p[threadIdx.x] = Word(0);
}

template <typename Word>
cudaError_t launch_zero_words(Word* p, int n, cudaStream_t st) {
  if (n < 1 || n > 1024) return cudaErrorInvalidValue;
  const unsigned threads = static_cast<unsigned>((n + 31) / 32 * 32);
  return launch_kernel(zero_words_kernel<Word>, dim3(1), dim3(threads), 0, st, p, n);
}

// SF_SOFTMAX_POST scores like softmax (over all E) and renormalises the
// selected probabilities like sigmoid (the softmax of the selected logits).
enum { SF_SOFTMAX = 0, SF_SIGMOID = 1, SF_SOFTMAX_POST = 2 };
enum { DT_F32 = 0, DT_BF16 = 1 };

// ---------------------------------------------------------------------------
// keys: float -> uint32 with the same order (a numeric compare); -0.0 and
// +0.0 map to the same key.  Finite floats map to keys >= 0x00800000, so key
// 0 is below every real expert and marks "not selectable".
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Total order used for the top-K: larger key first, then lower index.
__device__ __forceinline__ unsigned long long pack_key(uint32_t key, int idx) {
  return (static_cast<unsigned long long>(key) << 32) |
         static_cast<unsigned long long>(~static_cast<uint32_t>(idx));
}

// ---------------------------------------------------------------------------
// score functions in fp32
//
// e^t is computed as 2^(t log2 e) with the hardware base-2 exponential
// (ex2.approx, about 2 ulp).  For softmax the argument is one FFMA,
// x * log2e - max * log2e: the rounding of max * log2e scales every e of the
// row by the same factor, which cancels in the normalisation, and the
// rounding of the FFMA itself costs at most |x - max| * 2^-24 relative, which
// is negligible where e is not.  The sigmoid takes the hardware reciprocal
// (rcp.approx, about 1 ulp) of 1 + e^-x; it saturates correctly to 0 and 1.
// ---------------------------------------------------------------------------
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float t) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
  return y;
}

__device__ __forceinline__ float rcp_approx(float t) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
  return y;
}

// exp(x - max) given max_l2e = max * log2e
__device__ __forceinline__ float exp_shifted(float x, float max_l2e) {
  return ex2_approx(fmaf(x, kLog2e, -max_l2e));
}

__device__ __forceinline__ float sigmoid_f32(float x) {
  return rcp_approx(1.0f + ex2_approx(-x * kLog2e));
}

// ---------------------------------------------------------------------------
// four consecutive elements of a row.  VEC: one 16-byte (fp32) or 8-byte
// (bf16) access, caller guarantees alignment and e0 + 3 < E.  Otherwise
// element-wise with a bound check per element.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

template <int DT, bool VEC>
__device__ __forceinline__ void load4(const void* base, size_t off, int e0, int E,
                                      float (&v)[4]) {
  if constexpr (DT == DT_F32) {
    const float* p = static_cast<const float*>(base) + off + e0;
    if constexpr (VEC) {
      const float4 t = __ldcs(reinterpret_cast<const float4*>(p));
      v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = (e0 + u < E) ? __ldcs(p + u) : 0.0f;
    }
  } else {
    const unsigned short* p = static_cast<const unsigned short*>(base) + off + e0;
    if constexpr (VEC) {
      const uint2 t = __ldcs(reinterpret_cast<const uint2*>(p));
      v[0] = __uint_as_float(t.x << 16);
      v[1] = __uint_as_float(t.x & 0xffff0000u);
      v[2] = __uint_as_float(t.y << 16);
      v[3] = __uint_as_float(t.y & 0xffff0000u);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[u] = (e0 + u < E) ? bf16_bits_to_f32(__ldcs(p + u)) : 0.0f;
    }
  }
}

template <bool VEC>
__device__ __forceinline__ void load4_f32(const float* base, size_t off, int e0, int E,
                                          float (&v)[4]) {
  load4<DT_F32, VEC>(base, off, e0, E, v);
}

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(f)));
}

template <int DT, bool VEC>
__device__ __forceinline__ void store4(void* base, size_t off, int e0, int E,
                                       const float (&v)[4]) {
  if constexpr (DT == DT_F32) {
    float* p = static_cast<float*>(base) + off + e0;
    if constexpr (VEC) {
      __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (e0 + u < E) __stcs(p + u, v[u]);
    }
  } else {
    unsigned short* p = static_cast<unsigned short*>(base) + off + e0;
    if constexpr (VEC) {
      uint2 t;
      t.x = f32_to_bf16_bits(v[0]) | (f32_to_bf16_bits(v[1]) << 16);
      t.y = f32_to_bf16_bits(v[2]) | (f32_to_bf16_bits(v[3]) << 16);
      __stcs(reinterpret_cast<uint2*>(p), t);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (e0 + u < E) __stcs(p + u, static_cast<unsigned short>(f32_to_bf16_bits(v[u])));
    }
  }
}

template <bool VEC>
__device__ __forceinline__ void store4_f32(float* base, size_t off, int e0, int E,
                                           const float (&v)[4]) {
  store4<DT_F32, VEC>(base, off, e0, E, v);
}

// routing-map bytes (0/1) of four consecutive experts
template <bool VEC>
__device__ __forceinline__ void store_map4(uint8_t* base, size_t off, int e0, int E,
                                           const bool (&m)[4]) {
  uint8_t* p = base + off + e0;
  if constexpr (VEC) {
    const uint32_t w = (m[0] ? 1u : 0u) | (m[1] ? 1u << 8 : 0u) |
                       (m[2] ? 1u << 16 : 0u) | (m[3] ? 1u << 24 : 0u);
    __stcs(reinterpret_cast<unsigned int*>(p), w);
  } else {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (e0 + u < E) p[u] = m[u] ? 1 : 0;
  }
}

template <bool VEC>
__device__ __forceinline__ void load_map4(const uint8_t* base, size_t off, int e0, int E,
                                          bool (&m)[4]) {
  const uint8_t* p = base + off + e0;
  if constexpr (VEC) {
    const uint32_t w = __ldcs(reinterpret_cast<const unsigned int*>(p));
    m[0] = (w & 0xffu) != 0; m[1] = (w & 0xff00u) != 0;
    m[2] = (w & 0xff0000u) != 0; m[3] = (w & 0xff000000u) != 0;
  } else {
#pragma unroll
    for (int u = 0; u < 4; ++u) m[u] = (e0 + u < E) ? (__ldcs(p + u) != 0) : false;
  }
}

// ---------------------------------------------------------------------------
// segment reductions: SEG (8, 16 or 32) aligned lanes of one warp
// ---------------------------------------------------------------------------
template <int SEG>
__device__ __forceinline__ unsigned seg_mask() {
  if constexpr (SEG == 32) {
    return 0xffffffffu;
  } else {
    return ((1u << SEG) - 1u) << ((threadIdx.x & 31u) & ~static_cast<unsigned>(SEG - 1));
  }
}

template <int SEG>
__device__ __forceinline__ float seg_max(float v) {
  const unsigned m = seg_mask<SEG>();
#pragma unroll
  for (int o = SEG / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(m, v, o));
  return v;
}

// Butterfly sum: every lane ends with the same (bitwise) total.
template <int SEG>
__device__ __forceinline__ float seg_sum(float v) {
  const unsigned m = seg_mask<SEG>();
#pragma unroll
  for (int o = SEG / 2; o > 0; o >>= 1) v += __shfl_xor_sync(m, v, o);
  return v;
}

template <int SEG>
__device__ __forceinline__ int seg_sum_int(int v) {
  const unsigned m = seg_mask<SEG>();
#pragma unroll
  for (int o = SEG / 2; o > 0; o >>= 1) v += __shfl_xor_sync(m, v, o);
  return v;
}

template <int SEG>
__device__ __forceinline__ int seg_exclusive_scan(int v) {
  const unsigned m = seg_mask<SEG>();
  const int li = threadIdx.x & (SEG - 1);
  int incl = v;
#pragma unroll
  for (int o = 1; o < SEG; o <<= 1) {
    const int t = __shfl_up_sync(m, incl, o, SEG);
    if (li >= o) incl += t;
  }
  return incl - v;
}

template <int SEG>
__device__ __forceinline__ int seg_count(bool p) {
  const unsigned m = seg_mask<SEG>();
  return __popc(__ballot_sync(m, p) & m);
}

}  // namespace moe_router
