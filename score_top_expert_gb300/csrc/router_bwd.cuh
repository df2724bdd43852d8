// Router backwards: two passes over a row held in registers.
//
// A row is owned by RL = SEG * W lanes (SEG lanes of one warp when W == 1,
// or W whole warps).  Lane rl of the row holds chunks j = 0..NC-1, chunk j
// being the four consecutive experts 4 * (rl + RL * j) .. +3.
// Pass 1 reduces two row sums (register accumulation, then a butterfly over
// the segment, then, for W > 1, the W warp partials through shared memory
// behind a named barrier); pass 2 writes the per-element gradient.
//
// OP 0, top-K (g = grad_probs, m = routing_map, s = saved scores):
//   softmax: D = c sum m g s;             gx = s (c m g - D)
//   sigmoid: S = sum m s, D = sum m g s;  gx = m (c / S)(g - D / S) s (1 - s)
//   post-softmax (p = c m s / S, s the full softmax):
//            S = sum m s, D = sum m g s;  gx = m (c / S)(g - D / S) s
// OP 1, aux scores (g = grad_scores):
//   softmax (saved q):     A = sum g q;             gx = q (g - A)
//   sigmoid (saved sig):   Z = sum sig, B = sum g sig;
//                          gx = (g - B / Z) / Z * sig (1 - sig)
#pragma once

#include "router_common.cuh"

namespace moe_router {

struct BwdArgs {
  const void* grad;      // OP 0: [T,E] dtype; OP 1: [T,E] float
  const uint8_t* map;    // OP 0 only
  const float* saved;    // [T,E] float
  void* grad_logits;     // [T,E] dtype
  int T, E;
  float scaling;
};

template <int SEG, int W>
struct BwdShape {
  static constexpr int RL = SEG * W;                          // lanes per row
  static constexpr int RPB = (256 / RL) > 0 ? (256 / RL) : 1;  // rows per block
  static constexpr int THREADS = RL * RPB;
};

template <int SF, int DT, int SEG, int W, int NC, bool VEC, int OP>
__global__ void __launch_bounds__(BwdShape<SEG, W>::THREADS)
router_bwd_kernel(const BwdArgs a) {
  pdl_enter();
  using S = BwdShape<SEG, W>;
  constexpr int RL = S::RL;
  static_assert(W == 1 || SEG == 32, "multi-warp rows use whole warps");
  __shared__ float red[S::RPB][W][2];

  const int rg = threadIdx.x / RL;          // row group in the block
  const int rl = threadIdx.x % RL;          // lane in the row
  const int row = blockIdx.x * S::RPB + rg;
  const bool active = row < a.T;
  const int E = a.E;
  const size_t off = static_cast<size_t>(active ? row : 0) * static_cast<size_t>(E);

  auto chunk_ok = [&](int j) { return active && 4 * (rl + RL * j) < E; };

  float g[NC][4], v[NC][4];
  bool m[NC][4];
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const int e0 = 4 * (rl + RL * j);
    if (chunk_ok(j)) {
      if constexpr (OP == 0) {
        load4<DT, VEC>(a.grad, off, e0, E, g[j]);
        load_map4<VEC>(a.map, off, e0, E, m[j]);
      } else {
        load4_f32<VEC>(static_cast<const float*>(a.grad), off, e0, E, g[j]);
      }
      load4_f32<VEC>(a.saved, off, e0, E, v[j]);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) { g[j][u] = 0.0f; v[j][u] = 0.0f; m[j][u] = false; }
    }
    if constexpr (OP == 1) {
#pragma unroll
      for (int u = 0; u < 4; ++u) m[j][u] = false;
    }
  }

  // ---- pass 1: two row sums -------------------------------------------------
  float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
  for (int j = 0; j < NC; ++j)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if constexpr (OP == 0) {
        // elements past E were zero-filled: no contribution
        const float ms = m[j][u] ? v[j][u] : 0.0f;
        if constexpr (SF == SF_SOFTMAX) {
          p0 = fmaf(ms, g[j][u], p0);
        } else {
          p0 += ms;
          p1 = fmaf(ms, g[j][u], p1);
        }
      } else {
        if constexpr (SF == SF_SOFTMAX) {
          p0 = fmaf(g[j][u], v[j][u], p0);
        } else {
          p0 += v[j][u];
          p1 = fmaf(g[j][u], v[j][u], p1);
        }
      }
    }
  p0 = seg_sum<SEG>(p0);
  p1 = seg_sum<SEG>(p1);
  if constexpr (W > 1) {
    const int w = rl / 32;
    if ((rl & 31) == 0) { red[rg][w][0] = p0; red[rg][w][1] = p1; }
    asm volatile("bar.sync %0, %1;" ::"r"(1 + rg), "r"(RL) : "memory");
    p0 = 0.0f; p1 = 0.0f;
#pragma unroll
    for (int i = 0; i < W; ++i) { p0 += red[rg][i][0]; p1 += red[rg][i][1]; }
  }

  // ---- pass 2: per-element gradient -----------------------------------------
  const float c = a.scaling;
  float k0 = 0.0f, k1 = 0.0f;
  if constexpr (OP == 0 && SF == SF_SOFTMAX) {
    k0 = c * p0;                       // D
  } else if constexpr (OP == 0) {
    k0 = c / p0;                       // c / S
    k1 = p1 / p0;                      // D / S
  } else if constexpr (SF == SF_SOFTMAX) {
    k0 = p0;                           // A
  } else {
    k0 = 1.0f / p0;                    // 1 / Z
    k1 = p1 * k0;                      // B / Z
  }
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    if (!chunk_ok(j)) continue;
    float gx[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float s = v[j][u];
      if constexpr (OP == 0 && SF == SF_SOFTMAX) {
        gx[u] = s * ((m[j][u] ? c * g[j][u] : 0.0f) - k0);
      } else if constexpr (OP == 0 && SF == SF_SIGMOID) {
        gx[u] = m[j][u] ? k0 * (g[j][u] - k1) * (s * (1.0f - s)) : 0.0f;
      } else if constexpr (OP == 0) {  // post-softmax
        gx[u] = m[j][u] ? k0 * (g[j][u] - k1) * s : 0.0f;
      } else if constexpr (SF == SF_SOFTMAX) {
        gx[u] = s * (g[j][u] - k0);
      } else {
        gx[u] = (g[j][u] - k1) * k0 * (s * (1.0f - s));
      }
    }
    store4<DT, VEC>(a.grad_logits, off, 4 * (rl + RL * j), E, gx);
  }
}

}  // namespace moe_router
