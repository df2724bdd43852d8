// Router forward, shared-memory staged path.
//
// A segment of SEG lanes (32 in this build; the code also takes 16, a warp
// then holding 32 / SEG segments) owns one token row at a time and walks the
// rows of the batch persistently (row, row + all segments, ...).  Rows arrive in shared memory by one bulk copy
// each, double-buffered: while the segment works on row r from one stage, the
// copy of its next row fills the other, so every segment keeps a row in
// flight without holding it in registers.  Segments only synchronise among
// their own lanes, so the segments of a warp may take different paths.
// Batches larger than the resident warps (logit keys, OP 0 to 2) launch
// instead one one-warp block per row; a running warp takes over the rows of
// blocks that have not started yet (cluster launch control), one request
// ahead, so the rows go to whichever warps finish first and the batch's
// tail stays short.  When such a launch writes compact outputs only, a warp
// may keep one stage instead of two: the row's logits are last needed for
// its candidates and its row sum, so the stage is refilled with the next
// row right then, and that copy lands while the candidates are ranked and
// the K outputs written (each selected logit is read back from its packed
// key).  Fewer bytes per warp keep more warps resident.
//
// Per row (lane l of the segment holds chunks c = l + SEG j, four consecutive
// experts each):
//   1  row max and two half maxima per lane (2 SEG group maxima); if the
//      segment carries a threshold from its previous row, each lane also
//      marks its logits >= that threshold in a candidate bit mask (branch-free).
//      The speculation is kept only if it yields at least K and at most 4 SEG
//      candidates, which makes it exact: every top-K logit is a candidate.
//   2  otherwise: a lower bound on the K-th largest logit from the 2 SEG group
//      maxima (the K-th largest of them, rounded down to 16 high bits; a
//      16-step search) and a second pass marking logits >= the bound.
//   3  the marked logits are compacted as (ordered key << 32 | ~index) words
//      (ffs over each lane's mask, lanes in order by a prefix count); each
//      word's exact rank among them selects the K best, which set their bits
//      in a per-row bitmask.  The candidate ranked about 1.5 K gives the next
//      row's threshold.  A row with more than 4 SEG logits at the bound
//      narrows the threshold by a binary search on the key (one counting pass
//      per step, stopping at K..4 SEG candidates); when the search closes on
//      a single key that still holds too many, that key is tied: the tied
//      logits are taken in index order by a prefix count and marked directly
//      (so is a row whose maximum alone is tied K times).
//   4  scores: softmax e = exp(x - max) and the row sum, or sigmoid s; fp32
//      rows store them over their logits (bf16 rows recompute them in 5).
//   5  outputs from the scores and the bitmask: probs, map, scores (top-K)
//      or q, map, intermediate (aux scores).  Compact outputs (OP 2) gather
//      the K selected (key, ~index) words into the candidate buffer, rank
//      them, and write the row's K weights, indices and expanded rows; the
//      dense outputs follow only where their pointers are set, and the
//      logits stay in the stage (scores are recomputed, not stored).  OP 3
//      (a batch that fits one block: decode) then builds the batch's
//      (expert, token)-sorted expert maps in the block after the last row.
// Keying on the logit is exact: softmax and sigmoid are strictly increasing.
//
// Key mode KM 1 (top-K with a bias and/or groups): before pass 1 the row's
// keys s + bias are built in a per-warp fp32 key row (the bias sits in shared
// memory once per block); with groups, a group scores the sum of its
// per_group largest keys, and the keys of every group outside the
// group_topk best are set to -inf.  Passes 1-3 then select on that key row
// exactly as KM 0 selects on the logits; the scores are recomputed from the
// logits in pass 5.
#pragma once

#include "router_common.cuh"
#include "router_fwd.cuh"
#include "router_maps.cuh"
#include "router_tma.cuh"

namespace moe_router {

// Byte offsets inside one segment's slice of shared memory (set on the host).
// A stage holds one row padded to the full chunk grid (SEG * NC chunks), so
// every lane reads every chunk without a bound check; the padding is never
// written by the copy and is masked out when the row is not full.
struct StagedLayout {
  int head_bytes;   // KM 1: the block's bias row (fp32, padded), before the slices
  int work_off;     // KM 1: the row's keys (fp32, padded)
  int grp_off;      // KM 1: group scores and kept flags (32 + 32 words)
  int stage_bytes;  // SEG * NC chunks of 4 logits
  int cand_off;     // kCandPerLane * SEG packed candidate words
  int sorted_off;   // OP 2, 3: the K selected words by rank (MR_MAX_TOPK words)
  int sel_off;      // the K selected scores by rank (MR_MAX_TOPK floats)
  int mask_off;     // selection words, one bit per expert of the padded row
  int bar_off;      // two mbarriers, one 32-bit slot, and for stealing launches
                    // a third mbarrier (at +24) and a 16-byte response (at +32)
  int seg_bytes;    // slice size, multiple of 128
  int steal;        // 1: one-warp blocks, one row each, that take over the rows
                    // of blocks not yet started (cluster launch control)
  int one_stage;    // 1 (stealing launches of compact-only outputs): one stage,
                    // refilled as soon as the row's candidates and sum are taken
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

// Sum over the segment's lanes (one warp reduction when SEG == 32).
template <int SEG>
__device__ __forceinline__ int seg_reduce_add(int v) {
  if constexpr (SEG == 32) {
    return static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(v)));
  } else {
    return seg_sum_int<SEG>(v);
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
template <int DT, int SEG, int NC>
__device__ __forceinline__ void compact_marked(const unsigned char* stage, const CandMask<NC>& m,
                                               int pos, int li, unsigned long long* cand) {
#pragma unroll
  for (int i = 0; i < CandMask<NC>::W; ++i) {
    uint32_t bits = m.w[i];
    while (bits) {
      const int b = 32 * i + __ffs(bits) - 1;
      bits &= bits - 1;
      const int idx = 4 * (li + SEG * (b >> 2)) + (b & 3);
      cand[pos++] = pack_key(ordered_key(stage_x1<DT>(stage, idx)), idx);
    }
  }
}

// Rank of each owned candidate among all `total` candidates (NOWN per lane):
// the K best set their selection bits (and, with SORTED, take their place in
// sorted[rank]); the one ranked `target` publishes its key as the next row's
// threshold.  With SIG (top-K renormalised over the selected), each selected
// candidate's score goes to sel_scores[rank], so that the row sums them in
// rank order whatever the candidates' layout.
// With TRY32 (fp32 rows, where equal logits are rare) the rank first counts
// the candidates with a larger 32-bit key (one compare per pair); when keys
// repeat, the ranks of the tied candidates coincide and no longer sum to
// 0 + 1 + ... + (total - 1), and the rank is recounted on the full
// (key, ~index) words, which is what bf16 rows do directly.
template <int SEG, int NOWN, bool SIG, bool TRY32, bool SORTED, class ScoreOf>
__device__ __forceinline__ void rank_candidates(const unsigned long long* cand, int total,
                                                int li, int K, int target, uint32_t* selmask,
                                                uint32_t* next_key, float* sel_scores,
                                                const ScoreOf& score_of,
                                                unsigned long long* sorted) {
  const uint32_t* hi_words = reinterpret_cast<const uint32_t*>(cand) + 1;  // keys
  unsigned long long own[NOWN];
  int rank[NOWN];
  int rsum = 0;
#pragma unroll
  for (int r = 0; r < NOWN; ++r) {
    own[r] = (r * SEG + li < total) ? cand[r * SEG + li] : ~0ull;
    rank[r] = 0;
  }
  if constexpr (TRY32) {
#pragma unroll 4
    for (int c = 0; c < total; ++c) {
      const uint32_t w = hi_words[2 * c];
#pragma unroll
      for (int r = 0; r < NOWN; ++r) rank[r] += w > static_cast<uint32_t>(own[r] >> 32);
    }
#pragma unroll
    for (int r = 0; r < NOWN; ++r) rsum += (r * SEG + li < total) ? rank[r] : 0;
  }
  if (!TRY32 || seg_reduce_add<SEG>(rsum) != total * (total - 1) / 2) {
#pragma unroll
    for (int r = 0; r < NOWN; ++r) rank[r] = 0;
#pragma unroll 4
    for (int c = 0; c < total; ++c) {
      const unsigned long long w = cand[c];
#pragma unroll
      for (int r = 0; r < NOWN; ++r) rank[r] += w > own[r];
    }
  }
#pragma unroll
  for (int r = 0; r < NOWN; ++r) {
    if (r * SEG + li < total) {
      if (rank[r] < K) {
        const uint32_t idx = ~static_cast<uint32_t>(own[r]);
        atomicOr(&selmask[idx >> 5], 1u << (idx & 31));
        if constexpr (SORTED) sorted[rank[r]] = own[r];
        if constexpr (SIG)
          sel_scores[rank[r]] = score_of(static_cast<int>(idx), static_cast<uint32_t>(own[r] >> 32));
      }
      if (rank[r] == target) *next_key = static_cast<uint32_t>(own[r] >> 32);
    }
  }
}

// Registers of the 18-chunk logit-keyed kernels are capped: bf16 at 128, so that they
// keep 16 warps per SM (their shared memory would allow 21; uncapped they need 160);
// the fp32 compact kernel at 120, so that its one-stage launch keeps 17 (it uses 114;
// uncapped, 168).
template <int DT, int NC, int KM, int OP>
constexpr int staged_max_regs() {
  if (NC == 18 && KM == 0 && DT == DT_BF16) return 128;
  if (NC == 18 && KM == 0 && OP == 2) return 120;
  return 168;
}

template <int SF, int DT, int SEG, int NC, int OP, bool FULL, int KM>
__global__ void __launch_bounds__(kStagedMaxWarps * 32) __maxnreg__((staged_max_regs<DT, NC, KM, OP>()))
router_fwd_staged_kernel(const FwdArgs a, const StagedLayout L, int* status) {
  pdl_enter();
  constexpr int CAP = kCandPerLane * SEG;
  constexpr int RPW = 32 / SEG;                 // rows (segments) per warp
  constexpr int D = DT == DT_F32 ? 4 : 2;
  constexpr bool kSigTopk = (OP != 1 && SF != SF_SOFTMAX);  // probs renormalised over the K
  // scores kept over the fp32 logits (not with compact outputs, which read
  // the logits after pass 4)
  constexpr bool kStore = (DT == DT_F32 && KM == 0 && OP < 2);
  constexpr bool kNeedSum = (SF != SF_SIGMOID || OP == 1) && KM == 0;
  constexpr int KDT = KM == 0 ? DT : DT_F32;  // type of the selection keys
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31;
  const int li = lane & (SEG - 1);
  const int seg = (threadIdx.x >> 5) * RPW + lane / SEG;  // segment in the block
  const int spb = (blockDim.x >> 5) * RPW;                // segments per block
  const unsigned smask = seg_mask<SEG>();
  unsigned char* base = smem + L.head_bytes + seg * L.seg_bytes;
  float* bias_s = reinterpret_cast<float*>(smem);           // KM 1
  float* work = reinterpret_cast<float*>(base + L.work_off);  // KM 1
  float* gs = reinterpret_cast<float*>(base + L.grp_off);     // KM 1, grouped
  int* kept = reinterpret_cast<int*>(gs + kMaxGroups);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bar_off);
  uint32_t* next_key = reinterpret_cast<uint32_t*>(bars + 2);
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(base + L.cand_off);
  uint32_t* selmask = reinterpret_cast<uint32_t*>(base + L.mask_off);
  unsigned long long* sorted_sel =
      reinterpret_cast<unsigned long long*>(base + L.sorted_off);  // OP 2, 3
  float* sel_scores = reinterpret_cast<float*>(base + L.sel_off);  // renormalising top-K

  const int E = a.E, K = a.K, T = a.T;
  const int nchunks = E >> 2;
  const uint32_t row_bytes = static_cast<uint32_t>(E) * D;
  const int nsegs = gridDim.x * spb;
  const unsigned char* src = static_cast<const unsigned char*>(a.logits);
  const int target = a.spec_target;  // rank giving the next row's threshold

  // logits (KM 0) or keys (KM 1) of chunk j; padding chunks of a partial
  // row read as -inf
  auto load_x = [&](const unsigned char* stage, int j, float (&x)[4]) {
    if constexpr (KM == 1) {
      const float4 t = lds_f4(reinterpret_cast<const unsigned char*>(work) + 16 * (li + SEG * j));
      x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
      return;
    }
    const int c = li + SEG * j;
    stage_x<DT>(stage, c, x);
    if constexpr (!FULL) {
      const bool ok = c < nchunks;
#pragma unroll
      for (int u = 0; u < 4; ++u) x[u] = ok ? x[u] : -INFINITY;
    }
  };

  if constexpr (KM == 1) {
    for (int i = threadIdx.x; i < 4 * SEG * NC; i += blockDim.x)
      bias_s[i] = (a.bias != nullptr && i < E) ? a.bias[i] : 0.0f;
    __syncthreads();
  }
  // Stealing launches (one row per one-warp block, whole rows per warp): the
  // warp's next rows are those of blocks it cancels before they start, one
  // request in flight, so rows go to whichever warps finish first.
  constexpr bool kCanSteal = SEG == 32 && KM == 0 && OP <= 2;
  const bool steal = kCanSteal && L.steal != 0;
  constexpr bool kCanOne = kCanSteal && OP == 2 && NC == 18;  // as the host launches it
  const bool one = kCanOne && steal && L.one_stage != 0;
  uint64_t* clc_bar = bars + 3;
  unsigned char* clc_resp = reinterpret_cast<unsigned char*>(bars) + 32;
  uint32_t clc_phase = 0;
  if (li == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    if (steal) mbar_init(clc_bar, 1);
    fence_mbar_init();
  }
  __syncwarp(smask);

  const int row0 = blockIdx.x * spb + seg;
  if (li == 0) {
    if (row0 < T)
      bulk_load(base, src + static_cast<size_t>(row0) * row_bytes, row_bytes, &bars[0]);
    if (!one && row0 + nsegs < T)
      bulk_load(base + L.stage_bytes, src + static_cast<size_t>(row0 + nsegs) * row_bytes,
                row_bytes, &bars[1]);
    if (steal && row0 < T) clc_request(clc_resp, clc_bar);
  }
  int cur = row0, nxt = -1;  // stealing: this row and the next (-1: none)
  bool pending = false;      // stealing: a request is in flight
  if (one) {
    pending = row0 < T;  // answered when the first row releases the stage
  } else if (steal && row0 < T) {
    const bool got = mbar_wait_bounded(clc_bar, clc_phase);
    clc_phase ^= 1u;
    if (got) nxt = clc_cancelled_x(clc_resp);
    else if (li == 0) atomicExch(status, kDeviceWaitTimeout);
    fence_proxy_async_smem();
    __syncwarp();
    if (nxt >= 0) {
      pending = true;
      if (li == 0) {
        bulk_load(base + L.stage_bytes, src + static_cast<size_t>(nxt) * row_bytes, row_bytes,
                  &bars[1]);
        clc_request(clc_resp, clc_bar);
      }
    }
  }

  // One-stage launches: the row the request in flight took over (if any) goes
  // into the stage just released, and the next request is made; returns
  // that row, or -1.
  auto refill_one = [&](unsigned char* stage) -> int {
    int nn = -1;
    if (pending) {
      const bool got = mbar_wait_bounded(clc_bar, clc_phase);
      clc_phase ^= 1u;
      if (got) nn = clc_cancelled_x(clc_resp);
      else if (li == 0) atomicExch(status, kDeviceWaitTimeout);
      pending = nn >= 0;
    }
    fence_proxy_async_smem();  // every lane's reads of the stage and the response
    __syncwarp();
    if (li == 0 && nn >= 0) {
      bulk_load(stage, src + static_cast<size_t>(nn) * row_bytes, row_bytes, &bars[0]);
      clc_request(clc_resp, clc_bar);
    }
    return nn;
  };

  // The loop is uniform over the warp: the segments of a warp process rows
  // in step and meet at full-warp barriers after the copy wait and after the
  // selection, so that their paths reconverge.
  bool failed = false;     // a bounded wait gave up (OP 3 leaves the loop)
  bool have_spec = false;  // a threshold carried over from the previous row
  float spec_t = 0.0f;
  uint32_t phase = 0;
  for (int it = 0;; ++it) {
    const int row = steal ? cur : row0 + it * nsegs;
    const bool active = row >= 0 && row < T;
    if (!__any_sync(0xffffffffu, active)) break;
    const int b = one ? 0 : (it & 1);
    bool ok = true;
    if (active) ok = mbar_wait_bounded(&bars[b], (phase >> b) & 1u);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      // record the failure, let the other stage's copy (if any) land, leave
      if (active && li == 0) {
        atomicExch(status, kDeviceWaitTimeout);
        if (!one && (steal ? nxt >= 0 : row + nsegs < T))
          mbar_wait_bounded(&bars[b ^ 1], (phase >> (b ^ 1)) & 1u);
        if (pending) mbar_wait_bounded(clc_bar, clc_phase);
      }
      __syncwarp();
      if constexpr (OP == 3) {  // the block meets once more below
        failed = true;
        break;
      } else {
        return;
      }
    }
    if (!active) {  // this segment has no row left; its partner still has one
      __syncwarp();
      __syncwarp();
      continue;
    }
    phase ^= 1u << b;
    unsigned char* stage = base + b * L.stage_bytes;
    const size_t off = static_cast<size_t>(row) * static_cast<size_t>(E);

#pragma unroll
    for (int w = li; w < NC * SEG / 8; w += SEG) selmask[w] = 0u;

    // ---- 0 (KM 1): keys s + bias, group mask ------------------------------------------
    float xmax_l2e = 0.0f;  // KM 1 softmax: row max of the logits * log2e
    float xinv = 1.0f;      // KM 1 softmax: 1 / row sum of exp
    if constexpr (KM == 1) {
      auto logits_of = [&](int j, float (&x)[4]) {
        const int c = li + SEG * j;
        stage_x<DT>(stage, c, x);
        if constexpr (!FULL) {
          const bool okc = c < nchunks;
#pragma unroll
          for (int u = 0; u < 4; ++u) x[u] = okc ? x[u] : -INFINITY;
        }
      };
      if constexpr (SF != SF_SIGMOID) {
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          float x[4];
          logits_of(j, x);
          mx = fmaxf(mx, fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])));
        }
        xmax_l2e = seg_max<SEG>(mx) * kLog2e;
        float sm0 = 0.0f, sm1 = 0.0f;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          float x[4];
          logits_of(j, x);
          const float add = (exp_shifted(x[0], xmax_l2e) + exp_shifted(x[1], xmax_l2e)) +
                            (exp_shifted(x[2], xmax_l2e) + exp_shifted(x[3], xmax_l2e));
          if (j & 1) sm1 += add; else sm0 += add;
        }
        xinv = 1.0f / seg_sum<SEG>(sm0 + sm1);
      }
      // groups that align with chunks: a group is L = group_size / 4 lanes of
      // one chunk column j; its top-M sum is a butterfly merge of the lanes'
      // top-M lists in registers
      const int L = a.group_chunk_lanes;
      const bool fast_groups = a.num_groups > 1 && L > 0;
      const int M = a.per_group;
      float gsum[NC];
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        const int c = li + SEG * j;
        float x[4], k[4];
        logits_of(j, x);
        const float4 bv = lds_f4(bias_s + 4 * c);
        const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float sc = (SF != SF_SIGMOID) ? exp_shifted(x[u], xmax_l2e) * xinv : sigmoid_f32(x[u]);
          k[u] = (FULL || c < nchunks) ? sc + bb[u] : -INFINITY;
        }
        sts_f4(work + 4 * c, make_float4(k[0], k[1], k[2], k[3]));
        if (fast_groups && M <= 2) {
          // top-2 pair (t0 >= t1); M == 1 uses t0 only
          float t0 = fmaxf(fmaxf(k[0], k[1]), fmaxf(k[2], k[3]));
          float t1 = fmaxf(fmaxf(fminf(k[0], k[1]), fminf(k[2], k[3])),
                           fminf(fmaxf(k[0], k[1]), fmaxf(k[2], k[3])));
          for (int o = L / 2; o > 0; o >>= 1) {
            const float p0 = __shfl_xor_sync(smask, t0, o);
            const float p1 = __shfl_xor_sync(smask, t1, o);
            t1 = fmaxf(fminf(t0, p0), fmaxf(t1, p1));
            t0 = fmaxf(t0, p0);
          }
          gsum[j] = M == 1 ? t0 : t0 + t1;
        } else if (fast_groups) {
          float top[kTopMRegs];
#pragma unroll
          for (int i = 0; i < kTopMRegs; ++i) top[i] = -INFINITY;
          auto insert = [&](float w) {
#pragma unroll
            for (int i = 0; i < kTopMRegs; ++i) {
              if (i < M) {
                const float hi = fmaxf(top[i], w);
                w = fminf(top[i], w);
                top[i] = hi;
              }
            }
          };
#pragma unroll
          for (int u = 0; u < 4; ++u) insert(k[u]);
          for (int o = L / 2; o > 0; o >>= 1) {
            float other[kTopMRegs];
#pragma unroll
            for (int i = 0; i < kTopMRegs; ++i) other[i] = __shfl_xor_sync(smask, top[i], o);
#pragma unroll
            for (int i = 0; i < kTopMRegs; ++i) insert(other[i]);
          }
          float g = 0.0f;
#pragma unroll
          for (int i = 0; i < kTopMRegs; ++i)
            if (i < M) g += top[i];
          gsum[j] = g;
        }
      }
      if (fast_groups) {
        // rank every group against all others (ties: lower group index) by
        // reading each group's score from its first lane; drop the keys of
        // groups outside the group_topk best
        const int gpj = SEG / L;  // groups per chunk column
        int grank[NC];
#pragma unroll
        for (int j = 0; j < NC; ++j) grank[j] = 0;
#pragma unroll
        for (int jj = 0; jj < NC; ++jj) {
          for (int q = 0; q < gpj; ++q) {
            const int h = jj * gpj + q;
            const float hv = __shfl_sync(smask, gsum[jj], q * L);
            if (h < a.num_groups) {
#pragma unroll
              for (int j = 0; j < NC; ++j) {
                const int g = j * gpj + li / L;
                grank[j] += (hv > gsum[j]) || (hv == gsum[j] && h < g);
              }
            }
          }
        }
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          const int g = j * gpj + li / L;
          if (g < a.num_groups && grank[j] >= a.group_topk)
            sts_f4(work + 4 * (li + SEG * j),
                   make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY));
        }
      } else if (a.num_groups > 1) {
        __syncwarp(smask);
        group_select<SEG>(a, work, gs, kept);
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          const int c = li + SEG * j;
          if (FULL || c < nchunks) {
            float4 t = lds_f4(work + 4 * c);
            float k[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int g = static_cast<int>((static_cast<float>(4 * c + u) + 0.5f) * a.inv_group_size);
              if (!kept[g]) k[u] = -INFINITY;
            }
            sts_f4(work + 4 * c, make_float4(k[0], k[1], k[2], k[3]));
          }
        }
      }
      __syncwarp(smask);
    }

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
      if (have_spec) {
#pragma unroll
        for (int u = 0; u < 4; ++u) cm.mark(4 * j + u, x[u] >= ts);
      }
    }
    const float row_max = seg_max<SEG>(fmaxf(hm[0], hm[1]));
    int cnt = cm.count();
    int total = seg_reduce_add<SEG>(cnt);
    bool cand_ok = have_spec && total >= K && total <= CAP;

    // ---- 2: bound from the group maxima ---------------------------------------------
    uint32_t lo_key = 0;  // a key with more than CAP logits at or above it
    if (!cand_ok) {
      uint32_t gmax[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) gmax[h] = hm[h] == -INFINITY ? 0u : ordered_key(hm[h]);
      uint32_t bound = 0;
#pragma unroll
      for (int bit = 31; bit >= 16; --bit) {
        const uint32_t cb = bound | (1u << bit);
        int n;
        if constexpr (SEG == 32) n = seg_reduce_add<32>((gmax[0] >= cb) + (gmax[1] >= cb));
        else n = seg_count<SEG>(gmax[0] >= cb) + seg_count<SEG>(gmax[1] >= cb);
        if (n >= K) bound = cb;
      }
      // lowest finite float when the bound says nothing: padding (-inf) stays out
      if (bound < 0x00800000u) bound = 0x00800000u;
      lo_key = bound;
      const float tf = key_to_float(bound);
      cm.clear();
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        float x[4];
        load_x(stage, j, x);
#pragma unroll
        for (int u = 0; u < 4; ++u) cm.mark(4 * j + u, x[u] >= tf);
      }
      cnt = cm.count();
      total = seg_reduce_add<SEG>(cnt);
      cand_ok = total <= CAP;
    }

    // ---- 4 (as a step): scores e = exp(x - max) or s, their row sum -----------------
    const float max_l2e = KM == 1 ? xmax_l2e : row_max * kLog2e;
    float inv = xinv;
    auto score_pass = [&]() {
      if constexpr (kNeedSum || kStore) {
        float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          float x[4], s[4];
          load_x(stage, j, x);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if constexpr (SF != SF_SIGMOID) s[u] = exp_shifted(x[u], max_l2e);
            else s[u] = sigmoid_f32(x[u]);
          }
          if constexpr (kNeedSum) {
            const float add = (s[0] + s[1]) + (s[2] + s[3]);
            if (j & 1) sum1 += add; else sum0 += add;
          }
          if constexpr (kStore)
            sts_f4(stage + 16 * (li + SEG * j), make_float4(s[0], s[1], s[2], s[3]));
        }
        if constexpr (kNeedSum) inv = 1.0f / seg_sum<SEG>(sum0 + sum1);
      }
    };
    bool released = false;  // one-stage: the stage holds the next row already
    int next_one = -1;      // one-stage: that row

    // ---- 3: exact selection ----------------------------------------------------------
    float part = 0.0f;  // sum of the selected scores (sigmoid top-K)
    bool tie_row = false;
    bool sorted_row = false;  // OP 2, 3: the K selected words sit in sorted_sel by rank
    float v = row_max;    // tied rows: the K-th largest logit
    int above = 0;        // tied rows: logits > v
    if (!cand_ok) {
      // more than CAP logits reach the bound.  Either the maximum alone is
      // tied K times, or a binary search on the key between the bound and
      // the maximum finds a threshold with K..CAP logits above it; if the
      // search closes on one key that still holds more, that key is tied.
      int eq = 0;
#pragma unroll 1
      for (int j = 0; j < NC; ++j) {
        float x[4];
        load_x(stage, j, x);
        eq += (x[0] == v) + (x[1] == v) + (x[2] == v) + (x[3] == v);
      }
      eq = seg_reduce_add<SEG>(eq);
      if (eq >= K) {
        tie_row = true;
      } else {
        uint32_t lo = lo_key, hi = ordered_key(row_max) + 1u;
        int n_hi = 0;
#pragma unroll 1
        while (hi - lo > 1u) {
          const uint32_t mid = lo + (hi - lo) / 2u;
          const float tm = key_to_float(mid);
          int n = 0;
#pragma unroll 1
          for (int j = 0; j < NC; ++j) {
            float x[4];
            load_x(stage, j, x);
            n += (x[0] >= tm) + (x[1] >= tm) + (x[2] >= tm) + (x[3] >= tm);
          }
          n = seg_reduce_add<SEG>(n);
          if (n > CAP) {
            lo = mid;
          } else if (n < K) {
            hi = mid;
            n_hi = n;
          } else {
            lo = mid;
            cand_ok = true;
            break;
          }
        }
        if (cand_ok) {
          const float tm = key_to_float(lo);
          cm.clear();
#pragma unroll
          for (int j = 0; j < NC; ++j) {
            float x[4];
            load_x(stage, j, x);
#pragma unroll
            for (int u = 0; u < 4; ++u) cm.mark(4 * j + u, x[u] >= tm);
          }
          cnt = cm.count();
          total = seg_reduce_add<SEG>(cnt);
        } else {
          tie_row = true;
          v = key_to_float(lo);
          above = n_hi;
        }
      }
    }
    // the unnormalised score of a selected candidate (renormalising top-K
    // sums them): sigmoid s, or e = exp(x - max) for the post-softmax
    const float sel_max_l2e = KM == 1 ? xmax_l2e : row_max * kLog2e;
    auto score_of = [&](int idx, uint32_t key) -> float {
      const float x = KM == 1 ? stage_x1<DT>(stage, idx) : key_to_float(key);
      if constexpr (SF == SF_SIGMOID) return sigmoid_f32(x);
      else return exp_shifted(x, sel_max_l2e);
    };
    if (cand_ok) {
      compact_marked<KDT, SEG, NC>(KM == 1 ? reinterpret_cast<const unsigned char*>(work) : stage,
                                   cm, seg_exclusive_scan<SEG>(cnt), li, cand);
      __syncwarp(smask);
      if constexpr (kCanOne) {
        if (one) {  // the stage's last use is the row sum: take it now, refill
          score_pass();
          next_one = refill_one(stage);
          released = true;
        }
      }
      const int nown = (total + SEG - 1) / SEG;
      const int tgt = target < total - 1 ? target : total - 1;
      if (nown <= 1)
        rank_candidates<SEG, 1, kSigTopk, DT == DT_F32, (OP >= 2)>(cand, total, li, K, tgt, selmask, next_key, sel_scores, score_of, sorted_sel);
      else if (nown == 2)
        rank_candidates<SEG, 2, kSigTopk, DT == DT_F32, (OP >= 2)>(cand, total, li, K, tgt, selmask, next_key, sel_scores, score_of, sorted_sel);
      else if (nown == 3)
        rank_candidates<SEG, 3, kSigTopk, DT == DT_F32, (OP >= 2)>(cand, total, li, K, tgt, selmask, next_key, sel_scores, score_of, sorted_sel);
      else
        rank_candidates<SEG, 4, kSigTopk, DT == DT_F32, (OP >= 2)>(cand, total, li, K, tgt, selmask, next_key, sel_scores, score_of, sorted_sel);
      __syncwarp(smask);
      if constexpr (kSigTopk) {  // the selected scores in rank order
        for (int r = li; r < K; r += SEG) part += sel_scores[r];
      }
      spec_t = key_to_float(*next_key);
      have_spec = true;
      sorted_row = true;
    } else if (tie_row) {
      // need-th lowest index among the logits equal to v: chunks in index
      // order (chunk c covers experts 4c..4c+3), prefix counts across lanes
      const int need = K - above;
      int ti = -1, run = 0;
#pragma unroll 1
      for (int j = 0; j < NC && ti < 0; ++j) {
        const int c = li + SEG * j;
        float x[4];
        load_x(stage, j, x);
        const int e = (x[0] == v) + (x[1] == v) + (x[2] == v) + (x[3] == v);
        const int excl = seg_exclusive_scan<SEG>(e);
        const int tot = __shfl_sync(smask, excl + e, SEG - 1, SEG);
        int mine = -1;
        if (run + excl < need && run + excl + e >= need) {
          int left = need - run - excl;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (x[u] == v && --left == 0 && mine < 0) mine = 4 * c + u;
        }
        const unsigned who = __ballot_sync(smask, mine >= 0) & smask;
        if (who) ti = __shfl_sync(smask, mine, __ffs(who) - 1);
        run += tot;
      }
      __syncwarp(smask);
      // mark the selection: logits > v, and the equal ones up to index ti
#pragma unroll 1
      for (int j = 0; j < NC; ++j) {
        const int c = li + SEG * j;
        float x[4];
        load_x(stage, j, x);
        uint32_t bits = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (x[u] > v || (x[u] == v && 4 * c + u <= ti)) {
            bits |= 1u << u;
            if constexpr (kSigTopk) part += score_of(4 * c + u, ordered_key(x[u]));
          }
        }
        if (bits) atomicOr(&selmask[c >> 3], bits << (4 * (c & 7)));
      }
      have_spec = false;
    }

    __syncwarp(0xffffffffu);  // reconverge the segments of the warp

    // ---- 4: scores ----------------------------------------------------------------------
    if (!released) score_pass();
    float pf = a.scaling;
    if constexpr (kSigTopk) pf = a.scaling / seg_sum<SEG>(part);
    else if constexpr (SF == SF_SOFTMAX && OP != 1) pf = a.scaling * inv;
    __syncwarp(smask);

    bool dense = true;  // OP 2, 3: dense outputs requested
    if constexpr (OP >= 2) {
      if (sorted_row) {
        // ---- compact outputs, ranks known: the K selected words by rank ----
        constexpr int kPerLane = (MR_MAX_TOPK + SEG - 1) / SEG;
        const size_t t = static_cast<size_t>(row);
#pragma unroll
        for (int r = 0; r < kPerLane; ++r) {
          const int k = r * SEG + li;
          if (k < K) {
            const unsigned long long w = sorted_sel[k];
            const int idx = static_cast<int>(~static_cast<uint32_t>(w));
            // the logit itself: its ordered key (logit keys), else the stage
            const float x = KM == 0 ? key_to_float(static_cast<uint32_t>(w >> 32))
                                    : stage_x1<DT>(stage, idx);
            const float wt = (SF != SF_SIGMOID) ? exp_shifted(x, max_l2e) : sigmoid_f32(x);
            a.topk_w[t * a.ld_w + k] = wt * pf;
            a.topk_i[t * a.ld_i + k] = idx;
            if (a.tei != nullptr) a.tei[t * K + k] = k * T + row;
          }
        }
      } else {
      // ---- compact outputs: gather the K selected words (lane order), rank ----
      CandMask<NC> sel;  // the lane's selected experts, bit 4 j + u
      sel.clear();
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        const int c = li + SEG * j;
        if (FULL || c < nchunks)
          sel.w[(4 * j) >> 5] |= ((selmask[c >> 3] >> (4 * (c & 7))) & 0xfu) << ((4 * j) & 31);
      }
      int pos = seg_exclusive_scan<SEG>(sel.count());
      float* cand_p = reinterpret_cast<float*>(cand + MR_MAX_TOPK);
#pragma unroll
      for (int i = 0; i < CandMask<NC>::W; ++i) {
        uint32_t bits = sel.w[i];
#pragma unroll 1
        while (bits) {
          const int b = 32 * i + __ffs(bits) - 1;
          bits &= bits - 1;
          const int idx = 4 * (li + SEG * (b >> 2)) + (b & 3);
          const float x = stage_x1<DT>(stage, idx);
          const float key = KM == 1 ? work[idx] : x;
          const float w = (SF != SF_SIGMOID) ? exp_shifted(x, max_l2e) : sigmoid_f32(x);
          cand[pos] = pack_key(ordered_key(key), idx);
          cand_p[pos] = w * pf;
          ++pos;
        }
      }
      __syncwarp(smask);
      write_compact_row<SEG>(a, row, li, cand, cand_p);
      }
      dense = !released && (a.map != nullptr || a.probs != nullptr || a.scores != nullptr);
    }

    // ---- 5: outputs -----------------------------------------------------------------------
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = li + SEG * j;
      if (dense && (FULL || c < nchunks)) {
        float w[4];  // e (softmax) or s (sigmoid)
        if constexpr (kStore) {
          const float4 t = lds_f4(stage + 16 * c);
          w[0] = t.x; w[1] = t.y; w[2] = t.z; w[3] = t.w;
        } else {
          float x[4];
          stage_x<DT>(stage, c, x);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if constexpr (SF != SF_SIGMOID) w[u] = exp_shifted(x[u], max_l2e);
            else w[u] = sigmoid_f32(x[u]);
          }
        }
        const uint32_t bits = (selmask[c >> 3] >> (4 * (c & 7))) & 0xfu;
        const uint32_t mapw = (bits * 0x00204081u) & 0x01010101u;
        if (OP < 2 || a.map != nullptr)
          __stcs(reinterpret_cast<unsigned int*>(a.map + off + 4 * c), mapw);
        float s[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) s[u] = (SF != SF_SIGMOID) ? w[u] * inv : w[u];
        if constexpr (OP != 1) {
          float p[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) p[u] = (bits & (1u << u)) ? w[u] * pf : 0.0f;
          if (OP == 0 || a.probs != nullptr) store4<DT, true>(a.probs, off, 4 * c, E, p);
          if (OP == 0 || a.scores != nullptr) store4_f32<true>(a.scores, off, 4 * c, E, s);
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
    __syncwarp(0xffffffffu);
    if (one) {
      if (!released) next_one = refill_one(stage);
      cur = next_one;
    } else if (steal) {
      // the row after next: the one the request in flight took, if any
      int nn = -1;
      if (pending) {
        const bool got = mbar_wait_bounded(clc_bar, clc_phase);
        clc_phase ^= 1u;
        if (got) nn = clc_cancelled_x(clc_resp);
        else if (li == 0) atomicExch(status, kDeviceWaitTimeout);
        fence_proxy_async_smem();  // every lane has read the response
        __syncwarp();
        pending = nn >= 0;
        if (li == 0 && pending) {
          bulk_load(stage, src + static_cast<size_t>(nn) * row_bytes, row_bytes, &bars[b]);
          clc_request(clc_resp, clc_bar);
        }
      }
      cur = nxt;
      nxt = nn;
    } else if (li == 0) {
      const int nr = row + 2 * nsegs;
      if (nr < T) bulk_load(stage, src + static_cast<size_t>(nr) * row_bytes, row_bytes, &bars[b]);
    }
  }
  if constexpr (OP == 3) {
    // the whole batch is this block's (one launch of one block): its compact
    // indices are written; the maps region follows the segments' slices
    if (!__syncthreads_or(failed)) {
      int* maps_smem = reinterpret_cast<int*>(smem + L.head_bytes + spb * L.seg_bytes);
      expert_maps_block(a.topk_i, a.ld_i, T, E, K, maps_smem, a.maps_offsets, a.maps_p2u,
                        a.maps_u2p, a.maps_pexp);
    }
  }
}

}  // namespace moe_router
