// Router forward, shared-memory staged path (no bias, no groups).
//
// Each warp owns one token row at a time and walks the rows of the batch
// persistently (row, row + all warps, ...).  Rows arrive in shared memory by
// one bulk copy each, double-buffered: while the warp works on row r from one
// stage, the copy of its next row fills the other, so every warp keeps a row
// in flight without holding it in registers.
//
// Per row (lane l holds chunks c = l + 32 j, four consecutive experts each):
//   A  logits -> row max and two half maxima per lane (64 group maxima)
//      -> lower bound on the K-th largest logit (16-step ballot search)
//   B  count of logits >= bound
//   C  scores: softmax e = exp(x - max) (row sum) or sigmoid s; written back
//      to shared memory (over the logits for fp32, to a work row for bf16);
//      logits >= bound are compacted as (ordered key << 32 | ~index) words
//   -  exact rank among the candidates; the K selected set their bits in a
//      per-row bitmask.  A row with more candidates than the buffer holds
//      (many equal logits) instead walks the distinct logits down from the
//      maximum, one pass each, to the K-th largest (a bitwise search after
//      eight values), takes the tied ones in index order by a prefix count,
//      and marks the bitmask before pass C.
//   D  outputs from the stored scores and the bitmask: probs, map, scores
//      (top-K) or q, map, intermediate (aux scores).
// Keying on the logit is exact: softmax and sigmoid are strictly increasing.
#pragma once

#include "router_common.cuh"
#include "router_fwd.cuh"
#include "router_tma.cuh"

namespace moe_router {

// Byte offsets inside one warp's slice of shared memory (set on the host).
struct StagedLayout {
  int stage_bytes;  // one row of logits, rounded up to 128
  int work_off;     // bf16 rows: fp32 scores of the current row
  int cand_off;     // kCandPerLane * 32 packed candidate words
  int cand_s_off;   // their scores (sigmoid top-K)
  int mask_off;     // ceil(E / 32) selection words
  int bar_off;      // two mbarriers
  int warp_bytes;   // slice size, multiple of 128
};

constexpr int kStagedMaxWarps = 12;

__device__ __forceinline__ float4 lds_f4(const void* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

__device__ __forceinline__ uint2 lds_u2(const void* p) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_addr(p)));
  return v;
}

__device__ __forceinline__ void sts_f4(void* p, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
               ::"r"(smem_addr(p)), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

template <int DT>
__device__ __forceinline__ void stage_x(const unsigned char* stage, int c, float (&x)[4]) {
  if constexpr (DT == DT_F32) {
    const float4 t = lds_f4(stage + 16 * c);
    x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
  } else {
    const uint2 t = lds_u2(stage + 8 * c);
    x[0] = __uint_as_float(t.x << 16);
    x[1] = __uint_as_float(t.x & 0xffff0000u);
    x[2] = __uint_as_float(t.y << 16);
    x[3] = __uint_as_float(t.y & 0xffff0000u);
  }
}

// Rank of each owned candidate among all `total` candidates (NOWN per lane).
template <int NOWN>
__device__ __forceinline__ void rank_candidates(const unsigned long long* cand, int total,
                                                int lane, int K, uint32_t* selmask,
                                                const float* cand_s, float& part) {
  unsigned long long own[NOWN];
  int rank[NOWN];
#pragma unroll
  for (int r = 0; r < NOWN; ++r) {
    own[r] = (r * 32 + lane < total) ? cand[r * 32 + lane] : ~0ull;
    rank[r] = 0;
  }
#pragma unroll 4
  for (int c = 0; c < total; ++c) {
    const unsigned long long w = cand[c];
#pragma unroll
    for (int r = 0; r < NOWN; ++r) rank[r] += w > own[r];
  }
#pragma unroll
  for (int r = 0; r < NOWN; ++r) {
    if (r * 32 + lane < total && rank[r] < K) {
      const uint32_t idx = ~static_cast<uint32_t>(own[r]);
      atomicOr(&selmask[idx >> 5], 1u << (idx & 31));
      if (cand_s != nullptr) part += cand_s[r * 32 + lane];
    }
  }
}

template <int SF, int DT, int NC, int OP>
__global__ void __launch_bounds__(kStagedMaxWarps * 32)
router_fwd_staged_kernel(const FwdArgs a, const StagedLayout L, int* status) {
  constexpr int CAP = kCandPerLane * 32;
  constexpr int D = DT == DT_F32 ? 4 : 2;
  constexpr bool kSigTopk = (OP == 0 && SF == SF_SIGMOID);
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  unsigned char* base = smem + warp * L.warp_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bar_off);
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(base + L.cand_off);
  float* cand_s = reinterpret_cast<float*>(base + L.cand_s_off);
  uint32_t* selmask = reinterpret_cast<uint32_t*>(base + L.mask_off);

  const int E = a.E, K = a.K, T = a.T;
  const int nchunks = E >> 2;
  const int nwords = (E + 31) >> 5;
  const uint32_t row_bytes = static_cast<uint32_t>(E) * D;
  const int nwarps = gridDim.x * wpb;
  const unsigned char* src = static_cast<const unsigned char*>(a.logits);

  if (lane == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncwarp();

  int row = blockIdx.x * wpb + warp;
  if (lane == 0) {
    if (row < T) bulk_load(base, src + static_cast<size_t>(row) * row_bytes, row_bytes, &bars[0]);
    if (row + nwarps < T)
      bulk_load(base + L.stage_bytes, src + static_cast<size_t>(row + nwarps) * row_bytes,
                row_bytes, &bars[1]);
  }

  uint32_t phase = 0;
  for (int it = 0; row < T; ++it, row += nwarps) {
    const int b = it & 1;
    bool ok = mbar_wait_bounded(&bars[b], (phase >> b) & 1u);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      // record the failure, let the other stage's copy (if any) land, leave
      if (lane == 0) {
        atomicExch(status, kDeviceWaitTimeout);
        if (row + nwarps < T) mbar_wait_bounded(&bars[b ^ 1], (phase >> (b ^ 1)) & 1u);
      }
      __syncwarp();
      return;
    }
    phase ^= 1u << b;
    unsigned char* stage = base + b * L.stage_bytes;
    float* work = (DT == DT_F32) ? reinterpret_cast<float*>(stage)
                                 : reinterpret_cast<float*>(base + L.work_off);
    const size_t off = static_cast<size_t>(row) * static_cast<size_t>(E);

    for (int w = lane; w < nwords; w += 32) selmask[w] = 0u;

    // ---- A: maxima -------------------------------------------------------------
    float hm[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = lane + 32 * j;
      if (c < nchunks) {
        float x[4];
        stage_x<DT>(stage, c, x);
        const float m4 = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        hm[half_of<NC>(j, 0)] = fmaxf(hm[half_of<NC>(j, 0)], m4);
      }
    }
    float row_max = 0.0f;
    if constexpr (SF == SF_SOFTMAX) row_max = seg_max<32>(fmaxf(hm[0], hm[1]));
    uint32_t gmax[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) gmax[h] = hm[h] == -INFINITY ? 0u : ordered_key(hm[h]);
    uint32_t bound = 0;
#pragma unroll
    for (int bit = 31; bit >= 16; --bit) {
      const uint32_t c = bound | (1u << bit);
      if (seg_count<32>(gmax[0] >= c) + seg_count<32>(gmax[1] >= c) >= K) bound = c;
    }
    const float tf = bound < 0x00800000u ? -INFINITY : key_to_float(bound);

    // ---- B: candidate count --------------------------------------------------------
    int cnt0 = 0, cnt1 = 0;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = lane + 32 * j;
      if (c < nchunks) {
        float x[4];
        stage_x<DT>(stage, c, x);
        const int n = (x[0] >= tf) + (x[1] >= tf) + (x[2] >= tf) + (x[3] >= tf);
        if (j & 1) cnt1 += n; else cnt0 += n;
      }
    }
    const int my_cnt = cnt0 + cnt1;
    const int total = seg_sum_int<32>(my_cnt);
    const bool fast = total <= CAP;

    float part = 0.0f;  // sum of selected scores (sigmoid top-K)
    if (!fast) {
      // more candidates than the buffer holds: many equal logits.  Find the
      // K-th largest logit tk by walking the distinct values down from the
      // maximum, then the need-th lowest index among the logits equal to it.
      float v = seg_max<32>(fmaxf(hm[0], hm[1]));
      int above = 0;      // logits > v
      bool found = false;
#pragma unroll 1
      for (int round = 0; round < 8 && !found; ++round) {
        int eq = 0;
        float below = -INFINITY;
#pragma unroll 1
        for (int j = 0; j < NC; ++j) {
          const int c = lane + 32 * j;
          if (c < nchunks) {
            float x[4];
            stage_x<DT>(stage, c, x);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              eq += x[u] == v;
              if (x[u] < v) below = fmaxf(below, x[u]);
            }
          }
        }
        eq = seg_sum_int<32>(eq);
        below = seg_max<32>(below);
        if (above + eq >= K) found = true;
        else { above += eq; v = below; }
      }
      if (!found) {
        // general case: bitwise search for the K-th largest key
        uint32_t tk = 0;
#pragma unroll 1
        for (int bit = 31; bit >= 0; --bit) {
          const uint32_t cb = tk | (1u << bit);
          int n = 0;
#pragma unroll 1
          for (int j = 0; j < NC; ++j) {
            const int c = lane + 32 * j;
            if (c < nchunks) {
              float x[4];
              stage_x<DT>(stage, c, x);
#pragma unroll
              for (int u = 0; u < 4; ++u) n += ordered_key(x[u]) >= cb;
            }
          }
          if (seg_sum_int<32>(n) >= K) tk = cb;
        }
        v = key_to_float(tk);
        int gt = 0;
#pragma unroll 1
        for (int j = 0; j < NC; ++j) {
          const int c = lane + 32 * j;
          if (c < nchunks) {
            float x[4];
            stage_x<DT>(stage, c, x);
#pragma unroll
            for (int u = 0; u < 4; ++u) gt += x[u] > v;
          }
        }
        above = seg_sum_int<32>(gt);
      }
      // need-th lowest index among the logits equal to v: chunks in index
      // order (chunk c covers experts 4c..4c+3), prefix counts across lanes
      const int need = K - above;
      int ti = -1, run = 0;
#pragma unroll 1
      for (int j = 0; j < NC && ti < 0; ++j) {
        const int c = lane + 32 * j;
        float x[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (c < nchunks) stage_x<DT>(stage, c, x);
        const int e = (x[0] == v) + (x[1] == v) + (x[2] == v) + (x[3] == v);
        const int excl = seg_exclusive_scan<32>(e);
        const int tot = __shfl_sync(0xffffffffu, excl + e, 31);
        int mine = -1;
        if (run + excl < need && run + excl + e >= need) {
          int left = need - run - excl;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (x[u] == v && --left == 0 && mine < 0) mine = 4 * c + u;
        }
        const unsigned who = __ballot_sync(0xffffffffu, mine >= 0);
        if (who) ti = __shfl_sync(0xffffffffu, mine, __ffs(who) - 1);
        run += tot;
      }
      __syncwarp();
      // mark the selection: logits > v, and the equal ones up to index ti
#pragma unroll 1
      for (int j = 0; j < NC; ++j) {
        const int c = lane + 32 * j;
        if (c < nchunks) {
          float x[4];
          stage_x<DT>(stage, c, x);
          uint32_t bits = 0;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (x[u] > v || (x[u] == v && 4 * c + u <= ti)) {
              bits |= 1u << u;
              if constexpr (kSigTopk) part += sigmoid_f32(x[u]);
            }
          }
          if (bits) atomicOr(&selmask[c >> 3], bits << (4 * (c & 7)));
        }
      }
    }

    // ---- C: scores (and the candidates) -----------------------------------------------
    int pos = fast ? seg_exclusive_scan<32>(my_cnt) : 0;
    float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = lane + 32 * j;
      if (c < nchunks) {
        float x[4], s[4];
        stage_x<DT>(stage, c, x);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if constexpr (SF == SF_SOFTMAX) s[u] = expf(x[u] - row_max);
          else s[u] = sigmoid_f32(x[u]);
        }
        if constexpr (SF == SF_SOFTMAX || OP == 1) {
          const float add = (s[0] + s[1]) + (s[2] + s[3]);
          if (j & 1) sum1 += add; else sum0 += add;
        }
        sts_f4(work + 4 * c, make_float4(s[0], s[1], s[2], s[3]));
        if (fast) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (x[u] >= tf) {
              cand[pos] = pack_key(ordered_key(x[u]), 4 * c + u);
              if constexpr (kSigTopk) cand_s[pos] = s[u];
              ++pos;
            }
          }
        }
      }
    }
    __syncwarp();
    if (fast) {
      const int nown = (total + 31) >> 5;
      const float* cs = kSigTopk ? cand_s : nullptr;
      if (nown <= 1) rank_candidates<1>(cand, total, lane, K, selmask, cs, part);
      else if (nown == 2) rank_candidates<2>(cand, total, lane, K, selmask, cs, part);
      else if (nown == 3) rank_candidates<3>(cand, total, lane, K, selmask, cs, part);
      else rank_candidates<4>(cand, total, lane, K, selmask, cs, part);
    }
    float inv = 1.0f;
    if constexpr (SF == SF_SOFTMAX || OP == 1) inv = 1.0f / seg_sum<32>(sum0 + sum1);
    float pf = a.scaling;
    if constexpr (kSigTopk) pf = a.scaling / seg_sum<32>(part);
    __syncwarp();

    // ---- D: outputs ----------------------------------------------------------------------
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = lane + 32 * j;
      if (c < nchunks) {
        const float4 w = lds_f4(work + 4 * c);
        const uint32_t bits = (selmask[c >> 3] >> (4 * (c & 7))) & 0xfu;
        float s[4] = {w.x, w.y, w.z, w.w};
        if constexpr (SF == SF_SOFTMAX) {
#pragma unroll
          for (int u = 0; u < 4; ++u) s[u] *= inv;
        }
        const uint32_t mapw = (bits * 0x00204081u) & 0x01010101u;
        __stcs(reinterpret_cast<unsigned int*>(a.map + off + 4 * c), mapw);
        if constexpr (OP == 0) {
          float p[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) p[u] = (bits & (1u << u)) ? s[u] * pf : 0.0f;
          store4<DT, true>(a.probs, off, 4 * c, E, p);
          store4_f32<true>(a.scores, off, 4 * c, E, s);
        } else {
          if constexpr (SF == SF_SOFTMAX) {
            store4_f32<true>(a.scores, off, 4 * c, E, s);
            if (a.intermediate != nullptr) store4_f32<true>(a.intermediate, off, 4 * c, E, s);
          } else {
            float q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) q[u] = s[u] * inv;
            store4_f32<true>(a.scores, off, 4 * c, E, q);
            store4_f32<true>(a.intermediate, off, 4 * c, E, s);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      const int nr = row + 2 * nwarps;
      if (nr < T) {
        fence_proxy_async_smem();
        bulk_load(stage, src + static_cast<size_t>(nr) * row_bytes, row_bytes, &bars[b]);
      }
    }
  }
}

}  // namespace moe_router
