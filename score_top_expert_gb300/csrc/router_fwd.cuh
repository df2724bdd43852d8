// Router forward, segment-per-token path.
//
// One token row is owned by a segment of SEG lanes (8, 16 or 32) of a warp,
// so a warp routes 32/SEG tokens at once.  Lane li of the segment holds
// chunks j = 0..NC-1 of the row in registers, chunk j being the four
// consecutive experts 4*(li + SEG*j) .. +3 (one 16-byte load for fp32, one
// 8-byte load for bf16; consecutive lanes read consecutive chunks, so each
// warp access is fully coalesced).
//
// Selection (top-K with ties to the lower index) works on 64-bit packed
// words (ordered float key << 32 | ~index): the K-th largest word W splits
// the row exactly into selected (word >= W) and not.  W is found in three
// steps, all inside the segment:
//   1. lower bound.  Each lane takes the maxima of two halves of its chunks:
//      2*SEG disjoint groups.  If t is the K-th largest group maximum, at
//      least K keys are >= t; the bound is t rounded down to its 16 high
//      bits (a 16-step ballot search).
//   2. candidates.  Keys >= the bound (about 1.5 K for random rows) are
//      compacted into shared memory (at most 4 per lane).
//   3. exact rank.  Each candidate counts the candidates above it; the one
//      with rank K-1 is W.
// Rows with more candidates than the buffer holds (many equal keys) walk the
// distinct keys down from the largest (one pass each) to the K-th largest
// key, falling back to a bitwise search after eight distinct values; the
// index part of W then comes from an ordered prefix count of the equal keys.
//
// KM (key mode) 0: no bias, no groups.  The key is the raw logit: softmax and
//   sigmoid are strictly increasing, so the order is the order of the scores,
//   exactly; the scores are recomputed in the output pass.
// KM 1: bias and/or groups.  The key is s + bias in fp32, kept in registers;
//   groups (contiguous, E / num_groups experts) score the sum of their
//   per_group largest keys and all but the group_topk best are masked out.
//
// OP 0: top-K router (probs, routing_map, scores).
// OP 1: aux-loss scores (scores = q, routing_map, intermediate = sigmoid).
// OP 2: top-K router with compact outputs: per row the K selected experts in
//   rank order (key descending, index ascending) with their probabilities,
//   and the expanded row k T + t of each; probs, map and scores are written
//   too where their pointers are set.
#pragma once

#include "router_common.cuh"

namespace moe_router {

struct FwdArgs {
  const void* logits;
  const float* bias;      // [E] or null (OP 0, KM 1 only)
  void* probs;            // OP 0: [T,E] dtype
  uint8_t* map;           // [T,E]
  float* scores;          // [T,E]: OP 0 s, OP 1 q
  float* intermediate;    // OP 1: [T,E] sigmoid (may be null for softmax)
  float* topk_w;          // OP 2: [T, ld_w] probabilities in rank order
  int32_t* topk_i;        // OP 2: [T, ld_i] expert indices in rank order
  int32_t* tei;           // OP 2: [T, K] expanded rows k T + t, or null
  long long ld_w, ld_i;   // OP 2: row strides (elements) of topk_w / topk_i
  int32_t* maps_offsets;  // staged OP 3: [E+1] first permuted row of each expert
  int32_t* maps_p2u;      // staged OP 3: [T K] expanded row of each permuted row
  int32_t* maps_u2p;      // staged OP 3: [T K] permuted row of each expanded row
  int32_t* maps_pexp;     // staged OP 3: [T K] expert of each permuted row
  int T, E, K;
  int num_groups;         // > 1 only when grouping is on (KM 1)
  int group_topk;
  int group_size;         // E / num_groups
  int per_group;          // K / group_topk
  int lanes_per_group;    // power of two, SEG / lanes_per_group >= 1
  int group_chunk_lanes;  // staged path: lanes holding one group (group_size / 4,
                          // a power of two <= 32) when groups align with chunks
                          // and per_group <= 4; else 0 (shared-memory scan)
  float inv_group_size;   // 1 / group_size (exact enough for idx < 4096)
  int spec_target;        // staged path: the candidate rank whose key becomes the
                          // next row's speculative threshold (>= K - 1)
  float scaling;
};

constexpr int kFwdThreads = 256;
constexpr int kCandPerLane = 4;
constexpr int kMaxGroups = 32;
constexpr int kTopMRegs = 4;  // grouped top-M sums up to this M use an insertion list

// Compact outputs of one row (OP 2): rank every selected word among the K
// selected words of the segment's list (K <= MR_MAX_TOPK) and write position
// rank of the row.  words[i] = (ordered key << 32 | ~index), p[i] its weight.
template <int SEG>
__device__ __forceinline__ void write_compact_row(const FwdArgs& a, int row, int li,
                                                  const unsigned long long* words,
                                                  const float* p) {
  constexpr int kPerLane = (MR_MAX_TOPK + SEG - 1) / SEG;
  const int K = a.K;
#pragma unroll
  for (int r = 0; r < kPerLane; ++r) {
    const int i = r * SEG + li;
    if (i < K) {
      const unsigned long long w = words[i];
      int rank = 0;
#pragma unroll 4
      for (int c = 0; c < K; ++c) rank += words[c] > w;
      const size_t t = static_cast<size_t>(row);
      a.topk_w[t * a.ld_w + rank] = p[i];
      a.topk_i[t * a.ld_i + rank] = static_cast<int32_t>(~static_cast<uint32_t>(w));
      if (a.tei != nullptr) a.tei[t * K + rank] = rank * a.T + row;
    }
  }
}

template <int SEG>
struct FwdSegSmem {
  unsigned long long cand[kCandPerLane * SEG];
  float cand_s[kCandPerLane * SEG];
  unsigned long long thr;
  float gs[kMaxGroups];
  int kept[kMaxGroups];
};

template <int SEG>
__host__ __device__ constexpr size_t fwd_smem_bytes_static() {
  return sizeof(FwdSegSmem<SEG>) * (kFwdThreads / SEG);
}

// Which of the two halves of a lane's chunks an element belongs to.
template <int NC>
__device__ __forceinline__ int half_of(int j, int u) {
  if constexpr (NC >= 2) return j >= NC / 2 ? 1 : 0;
  else return u >= 2 ? 1 : 0;
}

// Sum of the M largest keys of each expert group, for the group-limited
// pre-selection; writes the groups' scores to gs[] and their kept flags to
// kept[] (both in shared memory, num_groups entries).
template <int SEG>
__device__ __forceinline__ void group_select(const FwdArgs& a, const float* rowkeys,
                                             float* gs_out, int* kept_out) {
  const unsigned smask = seg_mask<SEG>();
  const int li = threadIdx.x & (SEG - 1);
  const int G = a.num_groups, Eg = a.group_size, M = a.per_group;
  const int L = a.lanes_per_group;       // lanes sharing one group
  const int per_pass = SEG / L;          // groups handled per pass
  for (int gbase = 0; gbase < G; gbase += per_pass) {
    const int g = gbase + li / L;
    const int r = li & (L - 1);
    const bool act = g < G;
    float gsum;
    if (M <= kTopMRegs) {
      float top[kTopMRegs];
#pragma unroll
      for (int i = 0; i < kTopMRegs; ++i) top[i] = -INFINITY;
      if (act) {
        for (int e = r; e < Eg; e += L) {
          float w = rowkeys[g * Eg + e];
#pragma unroll
          for (int i = 0; i < kTopMRegs; ++i) {
            if (i < M) {
              const float hi = fmaxf(top[i], w);
              w = fminf(top[i], w);
              top[i] = hi;
            }
          }
        }
      }
      for (int o = L / 2; o > 0; o >>= 1) {
        float other[kTopMRegs];
#pragma unroll
        for (int i = 0; i < kTopMRegs; ++i) other[i] = __shfl_xor_sync(smask, top[i], o);
#pragma unroll
        for (int k = 0; k < kTopMRegs; ++k) {
          float w = other[k];
#pragma unroll
          for (int i = 0; i < kTopMRegs; ++i) {
            if (i < M) {
              const float hi = fmaxf(top[i], w);
              w = fminf(top[i], w);
              top[i] = hi;
            }
          }
        }
      }
      gsum = 0.0f;
#pragma unroll
      for (int i = 0; i < kTopMRegs; ++i)
        if (i < M) gsum += top[i];
    } else {
      // exact M-th largest key of the group by a 32-step search, then
      // sum(keys above it) + (M - count above) * (M-th key)
      uint32_t t = 0;
      for (int bit = 31; bit >= 0; --bit) {
        const uint32_t c = t | (1u << bit);
        int n = 0;
        if (act)
          for (int e = r; e < Eg; e += L) n += ordered_key(rowkeys[g * Eg + e]) >= c;
        for (int o = L / 2; o > 0; o >>= 1) n += __shfl_xor_sync(smask, n, o);
        if (n >= M) t = c;
      }
      float above = 0.0f;
      int n_above = 0;
      if (act)
        for (int e = r; e < Eg; e += L) {
          const float w = rowkeys[g * Eg + e];
          if (ordered_key(w) > t) { above += w; ++n_above; }
        }
      for (int o = L / 2; o > 0; o >>= 1) {
        above += __shfl_xor_sync(smask, above, o);
        n_above += __shfl_xor_sync(smask, n_above, o);
      }
      gsum = above + static_cast<float>(M - n_above) * key_to_float(t);
    }
    if (act && r == 0) gs_out[g] = gsum;
  }
  __syncwarp(smask);
  for (int g = li; g < G; g += SEG) {
    const float mine = gs_out[g];
    int rank = 0;
    for (int h = 0; h < G; ++h) {
      const float o = gs_out[h];
      rank += (o > mine) || (o == mine && h < g);
    }
    kept_out[g] = rank < a.group_topk;
  }
  __syncwarp(smask);
}

template <int SF, int DT, int SEG, int NC, bool VEC, int KM, int OP>
__global__ void __launch_bounds__(kFwdThreads)
router_fwd_seg_kernel(const FwdArgs a) {
  pdl_enter();
  constexpr int SEGS_PER_BLOCK = kFwdThreads / SEG;
  constexpr int CAP = kCandPerLane * SEG;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  FwdSegSmem<SEG>* segs = reinterpret_cast<FwdSegSmem<SEG>*>(smem_raw);
  const int seg_id = threadIdx.x / SEG;
  FwdSegSmem<SEG>& sm = segs[seg_id];
  const unsigned smask = seg_mask<SEG>();
  const int li = threadIdx.x & (SEG - 1);

  const int E = a.E;
  const int K = a.K;
  const int row = blockIdx.x * SEGS_PER_BLOCK + seg_id;
  const bool active = row < a.T;
  const size_t off = static_cast<size_t>(active ? row : 0) * static_cast<size_t>(E);

  auto chunk_ok = [&](int j) { return active && 4 * (li + SEG * j) < E; };
  auto elem_ok = [&](int j, int u) {
    return chunk_ok(j) && (VEC || 4 * (li + SEG * j) + u < E);
  };

  // ---- load the row -------------------------------------------------------
  float v[NC][4];
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    if (chunk_ok(j)) {
      load4<DT, VEC>(a.logits, off, 4 * (li + SEG * j), E, v[j]);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) v[j][u] = 0.0f;
    }
  }

  // ---- score prerequisites: row max and sums ------------------------------
  float hmax[2] = {-INFINITY, -INFINITY};  // per-half maxima of the logits
#pragma unroll
  for (int j = 0; j < NC; ++j)
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (elem_ok(j, u)) hmax[half_of<NC>(j, u)] = fmaxf(hmax[half_of<NC>(j, u)], v[j][u]);

  float row_max = 0.0f, inv_sum = 1.0f;
  if constexpr (SF != SF_SIGMOID) {
    row_max = seg_max<SEG>(fmaxf(hmax[0], hmax[1])) * kLog2e;
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < NC; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (elem_ok(j, u)) {
          const float e = exp_shifted(v[j][u], row_max);
          if constexpr (KM == 1) v[j][u] = e;
          sum += e;
        }
    inv_sum = 1.0f / seg_sum<SEG>(sum);
  } else if constexpr (OP == 1) {
    // aux sigmoid: q = sigmoid / sum of sigmoids over the row
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < NC; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (elem_ok(j, u)) sum += sigmoid_f32(v[j][u]);
    inv_sum = 1.0f / seg_sum<SEG>(sum);
  }

  // ---- keys ---------------------------------------------------------------
  // KM 0: key = ordered(logit); the group maxima are the half maxima.
  // KM 1: v becomes the score s, kk the ordered key of s + bias (0 = masked).
  uint32_t kk[KM == 1 ? NC : 1][4];
  uint32_t gmax[2];
  if constexpr (KM == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) gmax[h] = hmax[h] == -INFINITY ? 0u : ordered_key(hmax[h]);
  } else {
    const bool has_bias = a.bias != nullptr;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      float b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (has_bias && chunk_ok(j)) load4_f32<VEC>(a.bias, 0, 4 * (li + SEG * j), E, b);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if constexpr (SF != SF_SIGMOID) v[j][u] *= inv_sum;
        else v[j][u] = sigmoid_f32(v[j][u]);
        kk[j][u] = elem_ok(j, u) ? ordered_key(v[j][u] + b[u]) : 0u;
      }
    }
    if (a.num_groups > 1) {
      // group-limited pre-selection over the keys s + bias, staged in shared memory
      float* rowkeys = reinterpret_cast<float*>(segs + SEGS_PER_BLOCK) + seg_id * E;
#pragma unroll
      for (int j = 0; j < NC; ++j)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (elem_ok(j, u)) rowkeys[4 * (li + SEG * j) + u] = key_to_float(kk[j][u]);
      __syncwarp(smask);
      group_select<SEG>(a, rowkeys, sm.gs, sm.kept);
#pragma unroll
      for (int j = 0; j < NC; ++j)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int idx = 4 * (li + SEG * j) + u;
          if (elem_ok(j, u)) {
            const int g = static_cast<int>((static_cast<float>(idx) + 0.5f) * a.inv_group_size);
            if (!sm.kept[g]) kk[j][u] = 0u;
          }
        }
    }
    gmax[0] = gmax[1] = 0u;
#pragma unroll
    for (int j = 0; j < NC; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u) gmax[half_of<NC>(j, u)] = max(gmax[half_of<NC>(j, u)], kk[j][u]);
  }

  auto key_at = [&](int j, int u) -> uint32_t {
    if constexpr (KM == 0) return elem_ok(j, u) ? ordered_key(v[j][u]) : 0u;
    else return kk[j][u];
  };
  auto score_at = [&](int j, int u) -> float {  // the score s of the element
    if constexpr (KM == 1) return v[j][u];
    else if constexpr (SF != SF_SIGMOID) return exp_shifted(v[j][u], row_max) * inv_sum;
    else return sigmoid_f32(v[j][u]);
  };

  // ---- 1. lower bound on the K-th largest key ------------------------------
  uint32_t bound = 0;
#pragma unroll
  for (int bit = 31; bit >= 16; --bit) {
    const uint32_t c = bound | (1u << bit);
    const int n = seg_count<SEG>(gmax[0] >= c) + seg_count<SEG>(gmax[1] >= c);
    if (n >= K) bound = c;
  }
  if (bound == 0) bound = 1;

  // ---- 2. candidates ------------------------------------------------------
  int my_cnt = 0;
#pragma unroll
  for (int j = 0; j < NC; ++j)
#pragma unroll
    for (int u = 0; u < 4; ++u) my_cnt += key_at(j, u) >= bound;
  const int total = seg_sum_int<SEG>(my_cnt);

  unsigned long long thr = 0ull;  // the K-th largest packed word of the row
  float sel_sum = 0.0f;           // sum of s over the selected (sigmoid top-K)
  constexpr bool kNeedSelSum = (OP != 1 && SF != SF_SOFTMAX);  // renormalised probs
  if (total <= CAP) {
    int pos = seg_exclusive_scan<SEG>(my_cnt);
#pragma unroll
    for (int j = 0; j < NC; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t k = key_at(j, u);
        if (k >= bound) {
          sm.cand[pos] = pack_key(k, 4 * (li + SEG * j) + u);
          if constexpr (kNeedSelSum) sm.cand_s[pos] = score_at(j, u);
          ++pos;
        }
      }
    if (li == 0) sm.thr = 0ull;
    __syncwarp(smask);
    // ---- 3. exact rank among the candidates -------------------------------
    unsigned long long own[kCandPerLane];
    int rank[kCandPerLane];
#pragma unroll
    for (int r = 0; r < kCandPerLane; ++r) {
      own[r] = (r * SEG + li < total) ? sm.cand[r * SEG + li] : 0ull;
      rank[r] = 0;
    }
    for (int c = 0; c < total; ++c) {
      const unsigned long long w = sm.cand[c];
#pragma unroll
      for (int r = 0; r < kCandPerLane; ++r) rank[r] += w > own[r];
    }
    float part = 0.0f;
#pragma unroll
    for (int r = 0; r < kCandPerLane; ++r) {
      if (r * SEG + li < total) {
        if (rank[r] == K - 1) sm.thr = own[r];
        if constexpr (kNeedSelSum)
          if (rank[r] < K) part += sm.cand_s[r * SEG + li];
      }
    }
    if constexpr (kNeedSelSum) sel_sum = seg_sum<SEG>(part);
    __syncwarp(smask);
    thr = sm.thr;
    __syncwarp(smask);
  } else {
    // more candidates than the buffer holds: many equal keys.  Walk the
    // distinct keys down from the largest until K are covered (one pass per
    // distinct value), else search the K-th largest key bit by bit.
    uint32_t tk = max(gmax[0], gmax[1]);
#pragma unroll
    for (int o = SEG / 2; o > 0; o >>= 1) tk = max(tk, __shfl_xor_sync(smask, tk, o));
    int above = 0;
    bool found = false;
#pragma unroll 1
    for (int round = 0; round < 8 && !found; ++round) {
      int eq = 0;
      uint32_t below = 0;
#pragma unroll
      for (int j = 0; j < NC; ++j)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t k = key_at(j, u);
          eq += k == tk;
          if (k < tk) below = max(below, k);
        }
      eq = seg_sum_int<SEG>(eq);
#pragma unroll
      for (int o = SEG / 2; o > 0; o >>= 1) below = max(below, __shfl_xor_sync(smask, below, o));
      if (above + eq >= K) found = true;
      else { above += eq; tk = below; }
    }
    if (!found) {
      tk = 0;
#pragma unroll 1
      for (int bit = 31; bit >= 0; --bit) {
        const uint32_t c = tk | (1u << bit);
        int n = 0;
#pragma unroll
        for (int j = 0; j < NC; ++j)
#pragma unroll
          for (int u = 0; u < 4; ++u) n += key_at(j, u) >= c;
        if (seg_sum_int<SEG>(n) >= K) tk = c;
      }
      int gt = 0;
#pragma unroll
      for (int j = 0; j < NC; ++j)
#pragma unroll
        for (int u = 0; u < 4; ++u) gt += key_at(j, u) > tk;
      above = seg_sum_int<SEG>(gt);
    }
    // the need-th lowest index among the keys equal to tk: chunks in index
    // order, prefix counts across the segment's lanes
    const int need = K - above;
    int ti = -1, run = 0;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      if (ti >= 0) break;
      int e = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) e += key_at(j, u) == tk;
      const int excl = seg_exclusive_scan<SEG>(e);
      const int tot = __shfl_sync(smask, excl + e, SEG - 1, SEG);
      int mine = -1;
      if (run + excl < need && run + excl + e >= need) {
        int left = need - run - excl;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (key_at(j, u) == tk && --left == 0 && mine < 0) mine = 4 * (li + SEG * j) + u;
      }
      const unsigned who = __ballot_sync(smask, mine >= 0) & smask;
      if (who) ti = __shfl_sync(smask, mine, __ffs(who) - 1);
      run += tot;
    }
    thr = pack_key(tk, ti);
    if constexpr (kNeedSelSum) {
      float part = 0.0f;
#pragma unroll
      for (int j = 0; j < NC; ++j)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (key_at(j, u) != 0u && pack_key(key_at(j, u), 4 * (li + SEG * j) + u) >= thr)
            part += score_at(j, u);
      sel_sum = seg_sum<SEG>(part);
    }
  }

  // ---- outputs --------------------------------------------------------------
  const uint32_t tk = static_cast<uint32_t>(thr >> 32);
  const int ti = static_cast<int>(~static_cast<uint32_t>(thr));
  const float tkf = key_to_float(tk);
  float pf = a.scaling;
  if constexpr (kNeedSelSum) pf = a.scaling / sel_sum;
  auto selected = [&](int j, int u) -> bool {
    const int e = 4 * (li + SEG * j) + u;
    if constexpr (KM == 0) return (v[j][u] > tkf) || (v[j][u] == tkf && e <= ti);
    else return (kk[j][u] > tk) || (kk[j][u] == tk && kk[j][u] != 0u && e <= ti);
  };
  if constexpr (OP == 2) {
    // the K selected words and weights, gathered in lane order into the
    // segment's list, then ranked
    unsigned char* extra = reinterpret_cast<unsigned char*>(segs + SEGS_PER_BLOCK);
    if (a.num_groups > 1) extra += static_cast<size_t>(SEGS_PER_BLOCK) * E * sizeof(float);
    unsigned long long* words =
        reinterpret_cast<unsigned long long*>(extra) + seg_id * MR_MAX_TOPK;
    float* wp = reinterpret_cast<float*>(reinterpret_cast<unsigned long long*>(extra) +
                                         SEGS_PER_BLOCK * MR_MAX_TOPK) +
                seg_id * MR_MAX_TOPK;
    int nsel = 0;
#pragma unroll
    for (int j = 0; j < NC; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u) nsel += elem_ok(j, u) && selected(j, u);
    int pos = seg_exclusive_scan<SEG>(nsel);
#pragma unroll
    for (int j = 0; j < NC; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (elem_ok(j, u) && selected(j, u)) {
          words[pos] = pack_key(key_at(j, u), 4 * (li + SEG * j) + u);
          wp[pos] = score_at(j, u) * pf;
          ++pos;
        }
    __syncwarp(smask);
    if (active) write_compact_row<SEG>(a, row, li, words, wp);
    if (a.map == nullptr && a.probs == nullptr && a.scores == nullptr) return;
  }
  const bool dense = OP < 2 || a.map != nullptr || a.probs != nullptr || a.scores != nullptr;
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    if (!dense || !chunk_ok(j)) continue;
    const int e0 = 4 * (li + SEG * j);
    bool m[4];
    float s[4], p[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      m[u] = selected(j, u);
      s[u] = score_at(j, u);
      p[u] = m[u] ? s[u] * pf : 0.0f;
    }
    if (OP < 2 || a.map != nullptr) store_map4<VEC>(a.map, off, e0, E, m);
    if constexpr (OP != 1) {
      if (OP == 0 || a.probs != nullptr) store4<DT, VEC>(a.probs, off, e0, E, p);
      if (OP == 0 || a.scores != nullptr) store4_f32<VEC>(a.scores, off, e0, E, s);
    } else {
      float q[4];
      if constexpr (SF == SF_SOFTMAX) {
#pragma unroll
        for (int u = 0; u < 4; ++u) q[u] = s[u];
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) q[u] = s[u] * inv_sum;
      }
      store4_f32<VEC>(a.scores, off, e0, E, q);
      if (a.intermediate != nullptr) store4_f32<VEC>(a.intermediate, off, e0, E, s);
    }
  }
}

}  // namespace moe_router
