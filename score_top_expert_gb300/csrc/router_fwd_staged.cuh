// Router forward, shared-memory staged path (no bias, no groups).
//
// Each warp owns one token row at a time and walks the rows of the batch
// persistently (row, row + all warps, ...).  Rows arrive in shared memory by
// one bulk copy each, double-buffered: while the warp works on row r from one
// stage, the copy of its next row fills the other, so every warp keeps a row
// in flight without holding it in registers.
//
// Per row (lane l holds chunks c = l + 32 j, four consecutive experts each):
//   1  row max and two half maxima per lane (64 group maxima); if the warp
//      carries a threshold from its previous row, each lane also marks its
//      logits >= that threshold in a candidate bit mask (branch-free).  The
//      speculation is kept only if it yields at least K and at most 128
//      candidates, which makes it exact: every top-K logit is a candidate.
//   2  otherwise: a lower bound on the K-th largest logit from the 64 group
//      maxima (the K-th largest of them, rounded down to 16 high bits; a
//      16-step search) and a second pass marking logits >= the bound.
//   3  the marked logits are compacted as (ordered key << 32 | ~index) words
//      (ffs over each lane's mask, lanes in order by a prefix count); each
//      word's exact rank among them selects the K best, which set their bits
//      in a per-row bitmask.  The candidate ranked about 1.5 K gives the next
//      row's threshold.  A row with more than 128 candidates (many equal
//      logits) instead walks the distinct logits down from the maximum, one
//      pass each, to the K-th largest (a bitwise search after eight values),
//      takes the tied ones in index order by a prefix count, and marks the
//      bitmask directly.
//   4  scores: softmax e = exp(x - max) and the row sum, or sigmoid s; fp32
//      rows store them over their logits (bf16 rows recompute them in 5).
//   5  outputs from the scores and the bitmask: probs, map, scores (top-K)
//      or q, map, intermediate (aux scores).
// Keying on the logit is exact: softmax and sigmoid are strictly increasing.
#pragma once

#include "router_common.cuh"
#include "router_fwd.cuh"
#include "router_tma.cuh"

namespace moe_router {

// Byte offsets inside one warp's slice of shared memory (set on the host).
// A stage holds one row padded to the full chunk grid (32 * NC chunks), so
// every lane reads every chunk without a bound check; the padding is never
// written by the copy and is masked out when the row is not full.
struct StagedLayout {
  int stage_bytes;  // 32 * NC chunks of 4 logits
  int cand_off;     // kCandPerLane * 32 packed candidate words
  int mask_off;     // selection words, one bit per expert of the padded row
  int bar_off;      // two mbarriers and one 32-bit slot
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

template <int DT>
__device__ __forceinline__ float stage_x1(const unsigned char* stage, int idx) {
  if constexpr (DT == DT_F32) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(smem_addr(stage + 4 * idx)));
    return v;
  } else {
    unsigned short h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(smem_addr(stage + 2 * idx)));
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
}

// Candidate mask of one lane: bit 4 j + u marks element u of chunk j.
template <int NC>
struct CandMask {
  static constexpr int W = (4 * NC + 31) / 32;
  uint32_t w[W];
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int i = 0; i < W; ++i) w[i] = 0u;
  }
  __device__ __forceinline__ void mark(int bit, bool on) {
    if (on) w[bit >> 5] |= 1u << (bit & 31);
  }
  __device__ __forceinline__ int count() const {
    int n = 0;
#pragma unroll
    for (int i = 0; i < W; ++i) n += __popc(w[i]);
    return n;
  }
};

// Compact the marked logits of the lane into cand[pos...] as packed words.
template <int DT, int NC>
__device__ __forceinline__ void compact_marked(const unsigned char* stage, const CandMask<NC>& m,
                                               int pos, int lane, unsigned long long* cand) {
#pragma unroll
  for (int i = 0; i < CandMask<NC>::W; ++i) {
    uint32_t bits = m.w[i];
    while (bits) {
      const int b = 32 * i + __ffs(bits) - 1;
      bits &= bits - 1;
      const int idx = 4 * (lane + 32 * (b >> 2)) + (b & 3);
      cand[pos++] = pack_key(ordered_key(stage_x1<DT>(stage, idx)), idx);
    }
  }
}

// Rank of each owned candidate among all `total` candidates (NOWN per lane):
// the K best set their selection bits; the one ranked `target` publishes its
// key as the next row's threshold; sigmoid rows sum their selected scores.
template <int NOWN, bool SIG>
__device__ __forceinline__ void rank_candidates(const unsigned long long* cand, int total,
                                                int lane, int K, int target, uint32_t* selmask,
                                                uint32_t* next_key, float& part) {
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
    if (r * 32 + lane < total) {
      if (rank[r] < K) {
        const uint32_t idx = ~static_cast<uint32_t>(own[r]);
        atomicOr(&selmask[idx >> 5], 1u << (idx & 31));
        if constexpr (SIG) part += sigmoid_f32(key_to_float(static_cast<uint32_t>(own[r] >> 32)));
      }
      if (rank[r] == target) *next_key = static_cast<uint32_t>(own[r] >> 32);
    }
  }
}

template <int SF, int DT, int NC, int OP, bool FULL>
__global__ void __launch_bounds__(kStagedMaxWarps * 32)
router_fwd_staged_kernel(const FwdArgs a, const StagedLayout L, int* status) {
  constexpr int CAP = kCandPerLane * 32;
  constexpr int D = DT == DT_F32 ? 4 : 2;
  constexpr bool kSigTopk = (OP == 0 && SF == SF_SIGMOID);
  constexpr bool kStore = (DT == DT_F32);       // scores kept over the fp32 logits
  constexpr bool kNeedSum = (SF == SF_SOFTMAX || OP == 1);
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  unsigned char* base = smem + warp * L.warp_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bar_off);
  uint32_t* next_key = reinterpret_cast<uint32_t*>(bars + 2);
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(base + L.cand_off);
  uint32_t* selmask = reinterpret_cast<uint32_t*>(base + L.mask_off);

  const int E = a.E, K = a.K, T = a.T;
  const int nchunks = E >> 2;
  const uint32_t row_bytes = static_cast<uint32_t>(E) * D;
  const int nwarps = gridDim.x * wpb;
  const unsigned char* src = static_cast<const unsigned char*>(a.logits);
  const int target = K - 1 + (K / 2 > 4 ? K / 2 : 4);  // rank giving the next threshold

  // logits of chunk j; padding chunks of a partial row read as -inf
  auto load_x = [&](const unsigned char* stage, int j, float (&x)[4]) {
    const int c = lane + 32 * j;
    stage_x<DT>(stage, c, x);
    if constexpr (!FULL) {
      const bool ok = c < nchunks;
#pragma unroll
      for (int u = 0; u < 4; ++u) x[u] = ok ? x[u] : -INFINITY;
    }
  };

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

  bool have_spec = false;  // a threshold carried over from the previous row
  float spec_t = 0.0f;
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
    const size_t off = static_cast<size_t>(row) * static_cast<size_t>(E);

#pragma unroll
    for (int w = lane; w < NC * 4; w += 32) selmask[w] = 0u;

    // ---- 1: maxima, speculative candidate mask -------------------------------------
    float hm[2] = {-INFINITY, -INFINITY};
    CandMask<NC> cm;
    cm.clear();
    const float ts = have_spec ? spec_t : INFINITY;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      float x[4];
      load_x(stage, j, x);
      const float m4 = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      hm[half_of<NC>(j, 0)] = fmaxf(hm[half_of<NC>(j, 0)], m4);
#pragma unroll
      for (int u = 0; u < 4; ++u) cm.mark(4 * j + u, x[u] >= ts);
    }
    const float row_max = seg_max<32>(fmaxf(hm[0], hm[1]));
    int cnt = cm.count();
    int total = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(cnt)));
    bool cand_ok = have_spec && total >= K && total <= CAP;

    // ---- 2: bound from the group maxima ---------------------------------------------
    if (!cand_ok) {
      uint32_t gmax[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) gmax[h] = hm[h] == -INFINITY ? 0u : ordered_key(hm[h]);
      uint32_t bound = 0;
#pragma unroll
      for (int bit = 31; bit >= 16; --bit) {
        const uint32_t cb = bound | (1u << bit);
        const unsigned n = __reduce_add_sync(
            0xffffffffu, static_cast<unsigned>((gmax[0] >= cb) + (gmax[1] >= cb)));
        if (static_cast<int>(n) >= K) bound = cb;
      }
      // lowest finite float when the bound says nothing: padding (-inf) stays out
      const float tf = bound < 0x00800000u ? -3.402823466e38f : key_to_float(bound);
      cm.clear();
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        float x[4];
        load_x(stage, j, x);
#pragma unroll
        for (int u = 0; u < 4; ++u) cm.mark(4 * j + u, x[u] >= tf);
      }
      cnt = cm.count();
      total = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(cnt)));
      cand_ok = total <= CAP;
    }

    // ---- 3: exact selection ----------------------------------------------------------
    float part = 0.0f;  // sum of the selected scores (sigmoid top-K)
    if (cand_ok) {
      compact_marked<DT, NC>(stage, cm, seg_exclusive_scan<32>(cnt), lane, cand);
      __syncwarp();
      const int nown = (total + 31) >> 5;
      const int tgt = target < total - 1 ? target : total - 1;
      if (nown <= 1) rank_candidates<1, kSigTopk>(cand, total, lane, K, tgt, selmask, next_key, part);
      else if (nown == 2) rank_candidates<2, kSigTopk>(cand, total, lane, K, tgt, selmask, next_key, part);
      else if (nown == 3) rank_candidates<3, kSigTopk>(cand, total, lane, K, tgt, selmask, next_key, part);
      else rank_candidates<4, kSigTopk>(cand, total, lane, K, tgt, selmask, next_key, part);
      __syncwarp();
      spec_t = key_to_float(*next_key);
      have_spec = true;
    } else {
      // more candidates than the buffer holds: many equal logits.  Walk the
      // distinct values down from the maximum to the K-th largest logit v.
      float v = row_max;
      int above = 0;      // logits > v
      bool found = false;
#pragma unroll 1
      for (int round = 0; round < 8 && !found; ++round) {
        int eq = 0;
        float below = -INFINITY;
#pragma unroll 1
        for (int j = 0; j < NC; ++j) {
          float x[4];
          load_x(stage, j, x);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            eq += x[u] == v;
            if (x[u] < v) below = fmaxf(below, x[u]);
          }
        }
        eq = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(eq)));
        below = seg_max<32>(below);
        if (above + eq >= K) found = true;
        else { above += eq; v = below; }
      }
      if (!found) {
        // general case: bitwise search for the K-th largest key (padding is
        // -inf, below every finite logit, and K <= E keeps it out)
        uint32_t tk = 0;
#pragma unroll 1
        for (int bit = 31; bit >= 0; --bit) {
          const uint32_t cb = tk | (1u << bit);
          int n = 0;
#pragma unroll 1
          for (int j = 0; j < NC; ++j) {
            float x[4];
            load_x(stage, j, x);
#pragma unroll
            for (int u = 0; u < 4; ++u) n += ordered_key(x[u]) >= cb;
          }
          if (static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(n))) >= K)
            tk = cb;
        }
        v = key_to_float(tk);
        int gt = 0;
#pragma unroll 1
        for (int j = 0; j < NC; ++j) {
          float x[4];
          load_x(stage, j, x);
#pragma unroll
          for (int u = 0; u < 4; ++u) gt += x[u] > v;
        }
        above = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(gt)));
      }
      // need-th lowest index among the logits equal to v: chunks in index
      // order (chunk c covers experts 4c..4c+3), prefix counts across lanes
      const int need = K - above;
      int ti = -1, run = 0;
#pragma unroll 1
      for (int j = 0; j < NC && ti < 0; ++j) {
        const int c = lane + 32 * j;
        float x[4];
        load_x(stage, j, x);
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
        float x[4];
        load_x(stage, j, x);
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
      have_spec = false;
    }

    // ---- 4: scores ----------------------------------------------------------------------
    const float max_l2e = row_max * kLog2e;
    float inv = 1.0f;
    if constexpr (kNeedSum || kStore) {
      float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        float x[4], s[4];
        load_x(stage, j, x);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if constexpr (SF == SF_SOFTMAX) s[u] = exp_shifted(x[u], max_l2e);
          else s[u] = sigmoid_f32(x[u]);
        }
        if constexpr (kNeedSum) {
          const float add = (s[0] + s[1]) + (s[2] + s[3]);
          if (j & 1) sum1 += add; else sum0 += add;
        }
        if constexpr (kStore)
          sts_f4(stage + 16 * (lane + 32 * j), make_float4(s[0], s[1], s[2], s[3]));
      }
      if constexpr (kNeedSum) inv = 1.0f / seg_sum<32>(sum0 + sum1);
    }
    float pf = a.scaling;
    if constexpr (kSigTopk) pf = a.scaling / seg_sum<32>(part);
    else if constexpr (SF == SF_SOFTMAX && OP == 0) pf = a.scaling * inv;
    __syncwarp();

    // ---- 5: outputs -----------------------------------------------------------------------
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = lane + 32 * j;
      if (FULL || c < nchunks) {
        float w[4];  // e (softmax) or s (sigmoid)
        if constexpr (kStore) {
          const float4 t = lds_f4(stage + 16 * c);
          w[0] = t.x; w[1] = t.y; w[2] = t.z; w[3] = t.w;
        } else {
          float x[4];
          stage_x<DT>(stage, c, x);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if constexpr (SF == SF_SOFTMAX) w[u] = exp_shifted(x[u], max_l2e);
            else w[u] = sigmoid_f32(x[u]);
          }
        }
        const uint32_t bits = (selmask[c >> 3] >> (4 * (c & 7))) & 0xfu;
        const uint32_t mapw = (bits * 0x00204081u) & 0x01010101u;
        __stcs(reinterpret_cast<unsigned int*>(a.map + off + 4 * c), mapw);
        float s[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) s[u] = (SF == SF_SOFTMAX) ? w[u] * inv : w[u];
        if constexpr (OP == 0) {
          float p[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) p[u] = (bits & (1u << u)) ? w[u] * pf : 0.0f;
          store4<DT, true>(a.probs, off, 4 * c, E, p);
          store4_f32<true>(a.scores, off, 4 * c, E, s);
        } else if constexpr (SF == SF_SOFTMAX) {
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
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const int nr = row + 2 * nwarps;
      if (nr < T) bulk_load(stage, src + static_cast<size_t>(nr) * row_bytes, row_bytes, &bars[b]);
    }
  }
}

}  // namespace moe_router
