// Router forward for rows of at most 512 experts, each row held in the
// registers of one warp (top-K router and aux scores; the top-K router also
// with an expert bias and with groups that align with 4-expert chunks).
//
// A warp owns one token row at a time and walks the rows of the batch
// persistently (row, row + all warps, ...).  Rows arrive in shared memory by
// one bulk copy each into two stages per warp; as soon as a row is in
// registers its stage is refilled with the row two steps ahead, so every
// warp keeps two rows in flight.  Lane l holds chunks c = l + 32 j (j < NC)
// of the row, chunk c being experts 4c .. 4c + 3.
//
// Per row:
//   1  row maximum (a warp max-reduction of ordered keys) and each lane's two
//      half maxima (64 disjoint group maxima);
//   2  scores: softmax e = exp(x - max) with the row sum, or sigmoid s,
//      kept in registers;
//   3  a threshold t with K <= n <= 128 logits at or above it: the previous
//      row's threshold when it verifies, else a lower bound from the group
//      maxima (if K of them reach t, so do K logits) found by bisection on
//      the value; rows where neither works take step 5 over the whole row;
//   4  the logits >= t are compacted into shared memory (a prefix count
//      gives each lane its slots), each lane takes up to four of them back
//      into registers, and a bisection on the ordered key, counting
//      candidates with one warp reduction per step, finds the largest key
//      with exactly K logits at or above it.  A bisection that closes on a
//      single key with more than K logits at or above it has found a tie:
//      the logits above that key are taken, and the equal ones in index
//      order up to K by a prefix count;
//   5  (no usable t) the same bisection counting over the whole row;
//   6  outputs straight from registers: probs, map and scores (top-K), or
//      q, map and the sigmoid (aux scores).  Compact outputs (OP 2) gather
//      the K selected (key, ~index) words into shared memory, rank them
//      among themselves and write the row's K weights, indices and expanded
//      rows by rank; the dense outputs follow only where their pointers are
//      set.
// Key mode KM 0 (no bias, no groups) selects on the logit, which is exact:
// softmax and sigmoid are strictly increasing.  KM 1 selects on the fp32 key
// s + bias, built in registers after step 2; with groups, a group scores the
// sum of its per_group largest keys (a butterfly over the lanes holding the
// group), and the keys of every group outside the group_topk best are set to
// -inf before step 3.  Ties go to the lower expert index (and, among groups,
// to the lower group index).
#pragma once

#include <climits>
#include <type_traits>

#include "router_common.cuh"
#include "router_fwd.cuh"
#include "router_tma.cuh"

namespace moe_router {

// Byte offsets inside one warp's slice of shared memory (set on the host).
struct RegLayout {
  int stage_bytes;  // 32 * NC chunks of four logits (one padded row)
  int cand_off;     // kRegCap candidate logits (fp32)
  int grp_off;      // KM 1 groups: kMaxGroups packed group words (8 bytes each)
  int bar_off;      // two mbarriers
  int warp_bytes;   // slice size, multiple of 128
};

constexpr int kRegMaxWarps = 16;
constexpr int kRegCap = 128;   // candidates one row may carry into the bisection
constexpr int kRegBoundSlack = 8;  // group maxima above K the bound may leave
constexpr int kRegBoundSteps = 12;

// Ordered keys restricted to the precision of the logits: bf16 rows bisect
// on the 16 high bits (every bf16 value is one 16-bit key), fp32 rows on all
// 32.  to_float(k) is the smallest logit value with key k.
template <int DT>
struct RowKey {
  static constexpr int SH = DT == DT_F32 ? 0 : 16;
  __device__ __forceinline__ static uint32_t of(float f) { return ordered_key(f) >> SH; }
  __device__ __forceinline__ static float to_float(uint32_t k) {
    if constexpr (SH == 0) {
      return key_to_float(k);
    } else {
      return key_to_float((k << 16) | ((k & 0x8000u) ? 0u : 0xffffu));
    }
  }
  // key of the lowest finite logit (-FLT_MAX, or the lowest bf16 value)
  __device__ __forceinline__ static uint32_t lowest() { return SH == 0 ? 0x00800000u : 0x0080u; }
};

__device__ __forceinline__ int warp_add(int v) {
  return static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(v)));
}

// Load one chunk of four logits from a stage.
template <int DT>
__device__ __forceinline__ void stage_chunk(const unsigned char* stage, int c, float* x) {
  if constexpr (DT == DT_F32) {
    float4 t;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(t.x), "=f"(t.y), "=f"(t.z), "=f"(t.w)
                 : "r"(smem_addr(stage + 16 * c)));
    x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
  } else {
    uint32_t lo, hi;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(lo), "=r"(hi)
                 : "r"(smem_addr(stage + 8 * c)));
    x[0] = __uint_as_float(lo << 16);
    x[1] = __uint_as_float(lo & 0xffff0000u);
    x[2] = __uint_as_float(hi << 16);
    x[3] = __uint_as_float(hi & 0xffff0000u);
  }
}

// KM 1 groups that align with 4-expert chunks: group g is the
// a.group_chunk_lanes = Lg consecutive chunks Lg g .. Lg g + Lg - 1 (Lg a
// power of two <= 32, so one chunk column j holds 32 / Lg whole groups); its
// score is the sum of its per_group (<= kTopMRegs) largest keys, merged over
// its Lg lanes by a butterfly.  Ranking: the first lane of each group
// publishes the packed word (ordered score key << 32 | ~group) in the warp's
// slots `gw`, each lane of a group counts the larger words among every Lg-th
// group, and a butterfly over the group's lanes sums the counts (ties between
// scores go to the lower group index).  The keys of groups ranked group_topk
// or lower become -inf.
template <int NC>
__device__ __forceinline__ void group_mask(const FwdArgs& a, int lane, float (&sk)[4 * NC],
                                           unsigned long long* gw) {
  constexpr unsigned kFull = 0xffffffffu;
  const int Lg = a.group_chunk_lanes;
  const int M = a.per_group;
  const int G = a.num_groups;
  const int gpj = 32 / Lg;  // groups per chunk column
  float gsum[NC];
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const float* k = &sk[4 * j];
    if (M <= 2) {
      // top-2 pair (t0 >= t1); M == 1 uses t0 only
      float t0 = fmaxf(fmaxf(k[0], k[1]), fmaxf(k[2], k[3]));
      float t1 = fmaxf(fmaxf(fminf(k[0], k[1]), fminf(k[2], k[3])),
                       fminf(fmaxf(k[0], k[1]), fmaxf(k[2], k[3])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        if (o < Lg) {
          const float p0 = __shfl_xor_sync(kFull, t0, o);
          const float p1 = __shfl_xor_sync(kFull, t1, o);
          t1 = fmaxf(fminf(t0, p0), fmaxf(t1, p1));
          t0 = fmaxf(t0, p0);
        }
      }
      gsum[j] = M == 1 ? t0 : t0 + t1;
    } else {
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
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        if (o < Lg) {
          float other[kTopMRegs];
#pragma unroll
          for (int i = 0; i < kTopMRegs; ++i) other[i] = __shfl_xor_sync(kFull, top[i], o);
#pragma unroll
          for (int i = 0; i < kTopMRegs; ++i) insert(other[i]);
        }
      }
      float g = 0.0f;
#pragma unroll
      for (int i = 0; i < kTopMRegs; ++i)
        if (i < M) g += top[i];
      gsum[j] = g;
    }
  }
  unsigned long long word[NC];
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const int g = j * gpj + lane / Lg;
    word[j] = pack_key(ordered_key(gsum[j]), g);
    if ((lane & (Lg - 1)) == 0 && g < G) gw[g] = word[j];
  }
  __syncwarp();
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    int r = 0;
    for (int h = lane & (Lg - 1); h < G; h += Lg) r += gw[h] > word[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      if (o < Lg) r += __shfl_xor_sync(kFull, r, o);
    const int g = j * gpj + lane / Lg;
    if (g < G && r >= a.group_topk) {
#pragma unroll
      for (int u = 0; u < 4; ++u) sk[4 * j + u] = -INFINITY;
    }
  }
  __syncwarp();  // the slots are free again
}

// Registers per thread: 64 keeps 32 warps per SM; the compact-output kernels
// at 512 experts get 80 (25 warps), which spills much less, except fp32 rows
// of exactly 512 experts without bias or groups, which fit 64.  Rows of at
// most 256 experts without bias or groups get 48 (42 warps): at 8192 x 256,
// K = 8, the top-K forward took 6.46 against 6.57 us (fp32 softmax) and 6.53
// against 7.01 us (bf16 sigmoid), with a few bytes of spills in the aux-score
// kernels only.
template <int NC, int OP, int KM, bool FULL, int DT>
constexpr int reg_max_regs() {
  if (NC == 2 && KM == 0) return 48;
  return (NC == 4 && OP == 2 && !(KM == 0 && FULL && DT == DT_F32)) ? 80 : 64;
}

template <int SF, int DT, int NC, int OP, bool FULL, int KM>
__global__ void __launch_bounds__(kRegMaxWarps * 32) __maxnreg__((reg_max_regs<NC, OP, KM, FULL, DT>()))
router_fwd_reg_kernel(const FwdArgs a, const RegLayout L, int* status) {
  pdl_enter();
  static_assert(NC == 2 || NC == 4, "rows of up to 256 or 512 experts");
  static_assert(KM == 0 || OP != 1, "bias and groups: top-K router only");
  static_assert(OP <= 2, "dense top-K (0), aux scores (1), compact top-K (2)");
  constexpr int N = 4 * NC;  // logits per lane
  constexpr int D = DT == DT_F32 ? 4 : 2;
  constexpr unsigned kFull = 0xffffffffu;
  using RK = RowKey<KM == 1 ? DT_F32 : DT>;  // keys s + bias are fp32 values
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  unsigned char* base = smem + warp * L.warp_bytes;
  float* cand = reinterpret_cast<float*>(base + L.cand_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bar_off);

  const int E = a.E, K = a.K, T = a.T;
  const int nchunks = E >> 2;
  const uint32_t row_bytes = static_cast<uint32_t>(E) * D;
  const int nwarps = gridDim.x * wpb;
  const unsigned char* src = static_cast<const unsigned char*>(a.logits);

  if (lane == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const int row0 = blockIdx.x * wpb + warp;
  if (lane == 0) {
    if (row0 < T)
      bulk_load(base, src + static_cast<size_t>(row0) * row_bytes, row_bytes, &bars[0]);
    if (row0 + nwarps < T)
      bulk_load(base + L.stage_bytes, src + static_cast<size_t>(row0 + nwarps) * row_bytes,
                row_bytes, &bars[1]);
  }

  bool have_spec = false;  // an estimate carried over from the previous row
  float spec_t = 0.0f;
  uint32_t phase = 0;
#pragma unroll 1
  for (int it = 0;; ++it) {
    const int row = row0 + it * nwarps;
    if (row >= T) break;  // uniform over the warp
    const int b = it & 1;
    if (!__all_sync(kFull, mbar_wait_bounded(&bars[b], (phase >> b) & 1u))) {
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

    // ---- 1: the row in registers, maxima; the stage takes the next row ----------
    float x[N];
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = lane + 32 * j;
      stage_chunk<DT>(stage, c, &x[4 * j]);
      if constexpr (!FULL) {
        if (c >= nchunks) {
#pragma unroll
          for (int u = 0; u < 4; ++u) x[4 * j + u] = -INFINITY;
        }
      }
    }
    // half maxima of the lane (64 group maxima of the row)
    auto half_maxima = [&](const float (&v)[N], float (&hm)[2]) {
      hm[0] = hm[1] = -INFINITY;
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        const float m4 = fmaxf(fmaxf(v[4 * j], v[4 * j + 1]), fmaxf(v[4 * j + 2], v[4 * j + 3]));
        hm[j < NC / 2 ? 0 : 1] = fmaxf(hm[j < NC / 2 ? 0 : 1], m4);
      }
    };
    float hm[2];
    half_maxima(x, hm);
    // every real row has a finite maximum (padding is -inf, inputs are finite)
    const float xmax =
        key_to_float(__reduce_max_sync(kFull, ordered_key(fmaxf(hm[0], hm[1]))));
    // the maximum consumed every logit read from the stage: refill it
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const int nr = row + 2 * nwarps;
      if (nr < T) bulk_load(stage, src + static_cast<size_t>(nr) * row_bytes, row_bytes, &bars[b]);
    }
    const size_t off = static_cast<size_t>(row) * static_cast<size_t>(E);

    // ---- 2: scores and their row sum ----------------------------------------------
    const float max_l2e = xmax * kLog2e;
    float w[N];  // softmax: e = exp(x - max); sigmoid: s (padding: exactly 0)
    // summed in the staged forward's order (pairs within a chunk, chunks
    // alternating between two sums, then the butterfly), so that the scores
    // are bit for bit those of the other forward paths
    float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = 4 * j + u;
        if constexpr (SF != SF_SIGMOID) w[k] = exp_shifted(x[k], max_l2e);
        else w[k] = sigmoid_f32(x[k]);
      }
      const float add = (w[4 * j] + w[4 * j + 1]) + (w[4 * j + 2] + w[4 * j + 3]);
      if (j & 1) sum1 += add; else sum0 += add;
    }
    constexpr bool kNeedSum = SF != SF_SIGMOID || OP == 1;
    float inv = 1.0f;
    if constexpr (kNeedSum) inv = 1.0f / seg_sum<32>(sum0 + sum1);

    // ---- 2b: selection keys: the logits (KM 0), or s + bias with groups (KM 1) ----
    float sk[N];
    float row_max = xmax;  // largest selection key of the row
    if constexpr (KM == 0) {
#pragma unroll
      for (int k = 0; k < N; ++k) sk[k] = x[k];
    } else {
      // the bias (16-byte aligned, read through the cache: the same E floats
      // for every row)
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        const int c = lane + 32 * j;
        float4 b4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (a.bias != nullptr && (FULL || c < nchunks))
          b4 = __ldg(reinterpret_cast<const float4*>(a.bias) + c);
        const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int k = 4 * j + u;
          sk[k] = x[k] == -INFINITY ? -INFINITY
                                    : ((SF != SF_SIGMOID) ? w[k] * inv : w[k]) + bb[u];
        }
      }
      if (a.num_groups > 1)
        group_mask<NC>(a, lane, sk, reinterpret_cast<unsigned long long*>(base + L.grp_off));
      half_maxima(sk, hm);
      row_max = key_to_float(__reduce_max_sync(kFull, ordered_key(fmaxf(hm[0], hm[1]))));
    }

    // ---- 3: a candidate threshold ---------------------------------------------------
    auto count_ge = [&](float t) {
      int c = 0;
#pragma unroll
      for (int k = 0; k < N; ++k) c += sk[k] >= t;
      return c;
    };
    float t = 0.0f;
    int cnt = 0, n = 0;
    bool ok = false;
    if (have_spec) {
      t = spec_t;
      cnt = count_ge(t);
      n = warp_add(cnt);
      ok = n >= K && n <= kRegCap;
    }
    if (!ok) {
      // bisection on the value between the smallest finite group maximum
      // (every real group at or above it) and the row maximum; any value
      // with K group maxima at or above it has K logits at or above it
      const float g0 = hm[0] == -INFINITY ? INFINITY : hm[0];  // padding groups left out
      const float g1 = hm[1] == -INFINITY ? INFINITY : hm[1];
      const float gl = fminf(g0, g1);
      const float gmin = key_to_float(
          __reduce_min_sync(kFull, gl == INFINITY ? 0xffffffffu : ordered_key(gl)));
      int gn = warp_add((hm[0] != -INFINITY) + (hm[1] != -INFINITY));
      if (gn >= K) {
        float blo = gmin, bhi = row_max;
#pragma unroll 1
        for (int s = 0; s < kRegBoundSteps && gn > K + kRegBoundSlack; ++s) {
          const float mid = 0.5f * blo + 0.5f * bhi;
          if (mid == blo || mid == bhi) break;
          const int c = warp_add((hm[0] >= mid) + (hm[1] >= mid));
          if (c >= K) {
            blo = mid;
            gn = c;
          } else {
            bhi = mid;
          }
        }
        t = blo;
        cnt = count_ge(t);
        n = warp_add(cnt);
        ok = n <= kRegCap;  // n >= K holds by construction
      }
    }

    // ---- 4 / 5: exact K-th largest key by bisection -------------------------------
    uint32_t lo, hi = RK::of(row_max) + 1u;
    int n_lo;
    // count_at(m): this lane's keys at or above key m
    auto bisect = [&](auto count_at) {
#pragma unroll 1
      while (n_lo != K && hi - lo > 1u) {
        const uint32_t mid = lo + ((hi - lo) >> 1);
        const int c = warp_add(count_at(mid));
        if (c >= K) {
          lo = mid;
          n_lo = c;
        } else {
          hi = mid;
        }
      }
    };
    float o[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // this lane's candidates
    if (ok) {
      // compact the candidates: the lane's logits >= t go to its slots
      int pos = seg_exclusive_scan<32>(cnt);
#pragma unroll
      for (int k = 0; k < N; ++k) {
        if (sk[k] >= t) cand[pos++] = sk[k];
      }
      __syncwarp();
      auto slot = [&](int r) { return 32 * r + lane < n ? cand[32 * r + lane] : -INFINITY; };
      // the smallest key whose value is >= t: the logits at or above it are
      // exactly the n candidates (t need not lie on the key grid of bf16 rows)
      lo = RK::of(t);
      if (RK::to_float(lo) < t) ++lo;
      n_lo = n;
      // the bisection compares keys (x >= to_float(m) exactly when
      // RK::of(x) >= m; an empty slot's -inf keys below every finite one)
      if (n <= 32) {
        o[0] = slot(0);
        __syncwarp();  // the slots are free again (the next row writes them)
        const uint32_t k0 = RK::of(o[0]);
        bisect([&](uint32_t m) { return static_cast<int>(k0 >= m); });
      } else if (n <= 64) {
        o[0] = slot(0);
        o[1] = slot(1);
        __syncwarp();
        const uint32_t k0 = RK::of(o[0]), k1 = RK::of(o[1]);
        bisect([&](uint32_t m) { return (k0 >= m) + (k1 >= m); });
      } else {
#pragma unroll
        for (int r = 0; r < 4; ++r) o[r] = slot(r);
        __syncwarp();
        uint32_t k[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) k[r] = RK::of(o[r]);
        bisect([&](uint32_t m) { return (k[0] >= m) + (k[1] >= m) + (k[2] >= m) + (k[3] >= m); });
      }
    } else {
      lo = RK::lowest();
      n_lo = E;  // every real logit is finite
      bisect([&](uint32_t m) { return count_ge(RK::to_float(m)); });
    }
    const float v = RK::to_float(lo);
    int ti = INT_MAX;  // selected: x > v, or x == v with index <= ti
    if (n_lo != K) {
      // tie at v: n_hi logits above it (those at or above the next key); the
      // (K - n_hi)-th equal one in index order (chunk j covers experts
      // 128 j .. 128 j + 127 in lane order)
      const float above = RK::to_float(hi);
      const int n_hi = ok ? warp_add((o[0] >= above) + (o[1] >= above) + (o[2] >= above) +
                                     (o[3] >= above))
                          : warp_add(count_ge(above));
      const int need = K - n_hi;
      int run = 0;
      ti = -1;
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        int e = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) e += sk[4 * j + u] == v;
        const int excl = seg_exclusive_scan<32>(e);
        const int tot = __shfl_sync(kFull, excl + e, 31);
        int mine = -1;
        if (run + excl < need && run + excl + e >= need) {
          int left = need - run - excl;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (sk[4 * j + u] == v && --left == 0 && mine < 0) mine = 4 * (lane + 32 * j) + u;
        }
        const unsigned who = __ballot_sync(kFull, mine >= 0);
        if (who) {
          ti = __shfl_sync(kFull, mine, __ffs(who) - 1);
          break;
        }
        run += tot;
      }
    }

    // the next row starts from this row's candidate threshold
    spec_t = t;
    have_spec = ok;

    // ---- 6: outputs -----------------------------------------------------------------
    // score k: compact outputs without bias or groups (OP 2, KM 0) recompute
    // it from the logit (the same instructions, so the same bits), which
    // frees the scores' registers after the row sum (the empty asm keeps the
    // compiler from reusing the first computation instead)
    auto wv = [&](int k) -> float {
      if constexpr (OP == 2 && KM == 0) {
        float xk = x[k];
        asm("" : "+f"(xk));
        if constexpr (SF != SF_SIGMOID) return exp_shifted(xk, max_l2e);
        else return sigmoid_f32(xk);
      } else {
        return w[k];
      }
    };
    auto emit = [&](auto tie_tag) {
      constexpr bool kTie = decltype(tie_tag)::value;
      auto sel = [&](int k, int idx) -> bool {
        if constexpr (kTie) return sk[k] > v || (sk[k] == v && idx <= ti);
        else return sk[k] >= v;
      };
      [[maybe_unused]] float pf = a.scaling;  // probs factor (top-K router only)
      if constexpr (OP != 1 && SF != SF_SOFTMAX) {
        // renormalised over the selected: c / sum of their scores
        float part = 0.0f;
#pragma unroll
        for (int k = 0; k < N; ++k)
          if (sel(k, 4 * (lane + 32 * (k >> 2)) + (k & 3))) part += wv(k);
        pf = a.scaling / seg_sum<32>(part);
      } else if constexpr (OP != 1) {
        pf = a.scaling * inv;
      }
      // dense outputs straight from registers
      auto dense_outputs = [&]() {
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          const int c = lane + 32 * j;
          if (FULL || c < nchunks) {
            bool m[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) m[u] = sel(4 * j + u, 4 * c + u);
            if (OP != 2 || a.map != nullptr) store_map4<true>(a.map, off, 4 * c, E, m);
            float s[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) s[u] = (SF != SF_SIGMOID) ? wv(4 * j + u) * inv : wv(4 * j + u);
            if constexpr (OP != 1) {
              float p[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) p[u] = m[u] ? wv(4 * j + u) * pf : 0.0f;
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
      };
      if constexpr (OP == 2) {
        // compact outputs: the K selected (key, ~index) words and their
        // weights go to the warp's slots by a prefix count, each word's rank
        // among them is counted (on the 32-bit key first; when keys repeat the
        // ranks no longer sum to 0 + 1 + ... + K - 1 and they are recounted on
        // the whole words), and position rank of the row takes the expert
        unsigned long long* wd = reinterpret_cast<unsigned long long*>(cand);
        float* wt = reinterpret_cast<float*>(wd + MR_MAX_TOPK);
        int sc = 0;
#pragma unroll
        for (int k = 0; k < N; ++k) sc += sel(k, 4 * (lane + 32 * (k >> 2)) + (k & 3));
        int pos = seg_exclusive_scan<32>(sc);
#pragma unroll
        for (int k = 0; k < N; ++k) {
          const int idx = 4 * (lane + 32 * (k >> 2)) + (k & 3);
          if (sel(k, idx)) {
            wd[pos] = pack_key(ordered_key(sk[k]), idx);
            wt[pos] = wv(k) * pf;
            ++pos;
          }
        }
        // the dense outputs, when asked for, before the ranking: the row's
        // registers are then free for it
        if (a.map != nullptr || a.probs != nullptr || a.scores != nullptr) dense_outputs();
        __syncwarp();
        const uint32_t* hi_words = reinterpret_cast<const uint32_t*>(wd) + 1;  // keys
        const int i1 = lane + 32;
        const unsigned long long w0 = lane < K ? wd[lane] : 0ull;
        const unsigned long long w1 = i1 < K ? wd[i1] : 0ull;
        const uint32_t k0 = static_cast<uint32_t>(w0 >> 32), k1 = static_cast<uint32_t>(w1 >> 32);
        int r0 = 0, r1 = 0;
#pragma unroll 4
        for (int q = 0; q < K; ++q) {
          const uint32_t kq = hi_words[2 * q];
          r0 += kq > k0;
          r1 += kq > k1;
        }
        const int rs = (lane < K ? r0 : 0) + (i1 < K ? r1 : 0);
        if (warp_add(rs) != K * (K - 1) / 2) {
          r0 = r1 = 0;
#pragma unroll 4
          for (int q = 0; q < K; ++q) {
            const unsigned long long wq = wd[q];
            r0 += wq > w0;
            r1 += wq > w1;
          }
        }
        const size_t t = static_cast<size_t>(row);
        if (lane < K) {
          a.topk_w[t * a.ld_w + r0] = wt[lane];
          a.topk_i[t * a.ld_i + r0] = static_cast<int>(~static_cast<uint32_t>(w0));
          if (a.tei != nullptr) a.tei[t * K + r0] = r0 * T + row;
        }
        if (i1 < K) {
          a.topk_w[t * a.ld_w + r1] = wt[i1];
          a.topk_i[t * a.ld_i + r1] = static_cast<int>(~static_cast<uint32_t>(w1));
          if (a.tei != nullptr) a.tei[t * K + r1] = r1 * T + row;
        }
        __syncwarp();  // the slots are free again
      }
      if constexpr (OP != 2) dense_outputs();
    };
    if (ti == INT_MAX) emit(std::false_type{});
    else emit(std::true_type{});
  }
}

}  // namespace moe_router
