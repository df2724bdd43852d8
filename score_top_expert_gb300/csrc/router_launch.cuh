// Host-side launch of the router kernel templates: one function per
// (score function, dtype) that maps a runtime configuration onto the
// compiled instantiations.  Each .cu file instantiates one pair, so the
// instantiations compile in parallel.
#pragma once

#include <atomic>

#include "router_bwd.cuh"
#include "router_fwd.cuh"
#include "router_fwd_reg.cuh"
#include "router_fwd_staged.cuh"

namespace moe_router {

// Allow `kern` the dynamic shared memory `smem` (above the 48 KB default
// only), once per device and size: `granted` is the calling launcher's own
// record (one per kernel instantiation), the largest size set per device.
constexpr int kSmemDevs = 64;
template <typename Kern>
cudaError_t allow_smem(Kern kern, size_t smem, std::atomic<int>* granted) {
  if (smem <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const bool cached = dev >= 0 && dev < kSmemDevs;
  if (cached && granted[dev].load(std::memory_order_relaxed) >= static_cast<int>(smem))
    return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess && cached) {
    int cur = granted[dev].load(std::memory_order_relaxed);
    while (cur < static_cast<int>(smem) &&
           !granted[dev].compare_exchange_weak(cur, static_cast<int>(smem))) {
    }
  }
  return e;
}

// Forward configuration chosen by the C ABI layer.
struct FwdConfig {
  int seg;     // lanes per row: 8, 16, 32
  int nc;      // chunks of 4 experts per lane
  bool vec;    // aligned 16-byte rows
  int km;      // key mode (0: key = logit; 1: key = s + bias, optional groups)
  int op;      // 0 top-K router, 1 aux scores, 2 top-K with compact outputs
  size_t extra_smem;  // grouped: rows of keys staged in shared memory
};

struct BwdConfig {
  int seg, w, nc;
  bool vec;
  int op;
};

// compiled (SEG, NC) pairs of the forward; scalar rows use SEG 32, NC 18
#define MR_FWD_VEC_CONFIGS(X) \
  X(8, 2) X(8, 4) X(8, 8) X(16, 4) X(16, 8) X(32, 2) X(32, 4) X(32, 8) X(32, 18)

// compiled (SEG, W, NC) triples of the backwards (vector and scalar rows)
#define MR_BWD_CONFIGS(X)                                                      \
  X(8, 1, 2) X(16, 1, 4) X(32, 1, 2) X(32, 1, 4) X(32, 2, 1) X(32, 2, 2) X(32, 2, 4) \
  X(32, 4, 1) X(32, 4, 2) X(32, 3, 6) X(32, 6, 3) X(32, 9, 2)

template <int SF, int DT, int SEG, int NC, bool VEC, int KM, int OP>
cudaError_t launch_fwd_inst(const FwdArgs& a, const FwdConfig& c, cudaStream_t st) {
  auto kern = router_fwd_seg_kernel<SF, DT, SEG, NC, VEC, KM, OP>;
  constexpr int kSegsPerBlock = kFwdThreads / SEG;
  const size_t smem = fwd_smem_bytes_static<SEG>() + c.extra_smem;
  static std::atomic<int> granted[kSmemDevs];  // this kernel's record
  const cudaError_t se = allow_smem(kern, smem, granted);
  if (se != cudaSuccess) return se;
  const unsigned grid = static_cast<unsigned>((a.T + kSegsPerBlock - 1) / kSegsPerBlock);
  return launch_kernel(kern, dim3(grid), dim3(kFwdThreads), smem, st, a);
}

// MODE 0 instantiates the top-K (OP 0) and aux (OP 1) forwards, MODE 2 the
// compact-output router (OP 2); the modes live in separate translation
// units.
template <int SF, int DT, int SEG, int NC, bool VEC, int MODE>
cudaError_t launch_fwd_mode(const FwdArgs& a, const FwdConfig& c, cudaStream_t st) {
  if constexpr (MODE == 2) {
    return c.km == 1 ? launch_fwd_inst<SF, DT, SEG, NC, VEC, 1, MODE>(a, c, st)
                     : launch_fwd_inst<SF, DT, SEG, NC, VEC, 0, MODE>(a, c, st);
  } else {
    if constexpr (SF != SF_SOFTMAX_POST) {  // aux scores take softmax or sigmoid only
      if (c.op == 1) return launch_fwd_inst<SF, DT, SEG, NC, VEC, 0, 1>(a, c, st);
    }
    if (c.km == 1) return launch_fwd_inst<SF, DT, SEG, NC, VEC, 1, 0>(a, c, st);
    return launch_fwd_inst<SF, DT, SEG, NC, VEC, 0, 0>(a, c, st);
  }
}

template <int SF, int DT, int MODE = 0>
cudaError_t launch_fwd(const FwdArgs& a, const FwdConfig& c, cudaStream_t st) {
  if (!c.vec) {
    if (c.seg == 32 && c.nc == 18) return launch_fwd_mode<SF, DT, 32, 18, false, MODE>(a, c, st);
    return cudaErrorInvalidConfiguration;
  }
#define MR_FWD_CASE(S, N) \
  if (c.seg == S && c.nc == N) return launch_fwd_mode<SF, DT, S, N, true, MODE>(a, c, st);
  MR_FWD_VEC_CONFIGS(MR_FWD_CASE)
#undef MR_FWD_CASE
  return cudaErrorInvalidConfiguration;
}

template <int SF, int DT, int SEG, int W, int NC, bool VEC, int OP>
cudaError_t launch_bwd_inst(const BwdArgs& a, cudaStream_t st) {
  using S = BwdShape<SEG, W>;
  const unsigned grid = static_cast<unsigned>((a.T + S::RPB - 1) / S::RPB);
  return launch_kernel(router_bwd_kernel<SF, DT, SEG, W, NC, VEC, OP>, dim3(grid),
                       dim3(S::THREADS), 0, st, a);
}

template <int SF, int DT>
cudaError_t launch_bwd(const BwdArgs& a, const BwdConfig& c, cudaStream_t st) {
#define MR_BWD_CASE(S, W, N)                                                     \
  if (c.seg == S && c.w == W && c.nc == N) {                                     \
    if constexpr (SF == SF_SOFTMAX_POST) {                                       \
      return c.vec ? launch_bwd_inst<SF, DT, S, W, N, true, 0>(a, st)            \
                   : launch_bwd_inst<SF, DT, S, W, N, false, 0>(a, st);          \
    } else {                                                                     \
      if (c.vec) {                                                               \
        return c.op == 0 ? launch_bwd_inst<SF, DT, S, W, N, true, 0>(a, st)      \
                         : launch_bwd_inst<SF, DT, S, W, N, true, 1>(a, st);     \
      }                                                                          \
      return c.op == 0 ? launch_bwd_inst<SF, DT, S, W, N, false, 0>(a, st)       \
                       : launch_bwd_inst<SF, DT, S, W, N, false, 1>(a, st);      \
    }                                                                            \
  }
  MR_BWD_CONFIGS(MR_BWD_CASE)
#undef MR_BWD_CASE
  return cudaErrorInvalidConfiguration;
}

// Staged forward: segment shape, warps per block, the per-segment slice and
// the grid cap.
struct StagedPlan {
  StagedLayout layout;
  int warps_per_block;
  int max_blocks;  // resident blocks per SM x SMs
  int seg;         // lanes per row (32 in this build)
  int nc;          // chunks of 4 experts per lane
  int op;
  int km;          // key mode: 0 logits, 1 s + bias (and groups), top-K only
  bool full;       // E == 4 * seg * nc: no padding chunks
  int tail_bytes;  // after the slices: the block's expert maps (op 3)
  int steal_blocks;  // resident one-warp blocks of the stealing launch (0: none);
                     // batches of more rows than that launch it
  StagedLayout layout1;  // compact-only outputs: the one-stage slice
  int steal_blocks1;     // resident one-stage blocks (0: not used); compact-only
                         // batches of more rows than that launch them
};

// compiled (SEG, NC) pairs of the staged forward
#define MR_STAGED_SHAPES(X) X(32, 2) X(32, 4) X(32, 8) X(32, 18)

template <int SF, int DT, int SEG, int NC, int OP, bool FULL, int KM>
cudaError_t launch_staged_inst(const FwdArgs& a, const StagedPlan& p, int* status,
                               cudaStream_t st) {
  auto kern = router_fwd_staged_kernel<SF, DT, SEG, NC, OP, FULL, KM>;
  const size_t smem = p.layout.head_bytes +
                      static_cast<size_t>(p.warps_per_block) * (32 / SEG) * p.layout.seg_bytes +
                      p.tail_bytes;
  static std::atomic<int> granted[kSmemDevs];  // this kernel's record
  const cudaError_t se = allow_smem(kern, smem, granted);
  if (se != cudaSuccess) return se;
  if constexpr (SEG == 32 && KM == 0 && OP <= 2) {
    // more rows than resident warps: one one-warp block per row, the warps
    // taking over the rows of blocks not yet started
    if constexpr (OP == 2) {
      const bool compact_only = a.map == nullptr && a.probs == nullptr && a.scores == nullptr;
      if (compact_only && p.steal_blocks1 > 0 && a.T > p.steal_blocks1) {
        StagedLayout L = p.layout1;
        L.steal = 1;
        return launch_kernel(kern, dim3(static_cast<unsigned>(a.T)), dim3(32),
                             static_cast<size_t>(L.head_bytes) + L.seg_bytes, st, a, L, status);
      }
    }
    if (p.steal_blocks > 0 && a.T > p.steal_blocks) {
      StagedLayout L = p.layout;
      L.steal = 1;
      return launch_kernel(kern, dim3(static_cast<unsigned>(a.T)), dim3(32),
                           static_cast<size_t>(L.head_bytes) + L.seg_bytes, st, a, L, status);
    }
  }
  // Rows go round-robin over all resident segments.  When they take more
  // than one round, use the fewest blocks that still need the same number of
  // rounds, so that every segment carries the same number of rows (no
  // half-empty last round).
  const long long rows_per_block = static_cast<long long>(p.warps_per_block) * (32 / SEG);
  const long long need = (static_cast<long long>(a.T) + rows_per_block - 1) / rows_per_block;
  long long blocks = need;
  if (need > p.max_blocks) {
    const long long rounds = (need + p.max_blocks - 1) / p.max_blocks;
    blocks = (need + rounds - 1) / rounds;
  }
  const unsigned grid = static_cast<unsigned>(blocks);
  return launch_kernel(kern, dim3(grid), dim3(p.warps_per_block * 32), smem, st, a, p.layout,
                       status);
}

// Resident blocks per SM of one staged instantiation (occupancy query).
template <int SF, int DT, int SEG, int NC, int OP, bool FULL, int KM>
int staged_blocks_per_sm(int warps_per_block, size_t smem) {
  auto kern = router_fwd_staged_kernel<SF, DT, SEG, NC, OP, FULL, KM>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, warps_per_block * 32, smem) !=
      cudaSuccess)
    return 0;
  return n;
}

// MODE 0: top-K (OP 0) and aux (OP 1); MODE 2: compact outputs (OP 2);
// MODE 3: compact outputs and expert maps of a one-block batch (OP 3).
template <int SF, int DT, int MODE = 0>
cudaError_t launch_staged(const FwdArgs& a, const StagedPlan& p, int* status, cudaStream_t st) {
#define MR_STAGED_CASE(S, N)                                                               \
  if (p.seg == S && p.nc == N) {                                                           \
    if constexpr (MODE >= 2) {                                                             \
      if (p.km == 1)                                                                       \
        return p.full ? launch_staged_inst<SF, DT, S, N, MODE, true, 1>(a, p, status, st)  \
                      : launch_staged_inst<SF, DT, S, N, MODE, false, 1>(a, p, status, st);\
      return p.full ? launch_staged_inst<SF, DT, S, N, MODE, true, 0>(a, p, status, st)    \
                    : launch_staged_inst<SF, DT, S, N, MODE, false, 0>(a, p, status, st);  \
    } else {                                                                               \
      if constexpr (SF != SF_SOFTMAX_POST) {                                               \
        if (p.op == 1)                                                                     \
          return p.full ? launch_staged_inst<SF, DT, S, N, 1, true, 0>(a, p, status, st)   \
                        : launch_staged_inst<SF, DT, S, N, 1, false, 0>(a, p, status, st); \
      }                                                                                    \
      if (p.km == 1)                                                                       \
        return p.full ? launch_staged_inst<SF, DT, S, N, 0, true, 1>(a, p, status, st)     \
                      : launch_staged_inst<SF, DT, S, N, 0, false, 1>(a, p, status, st);   \
      return p.full ? launch_staged_inst<SF, DT, S, N, 0, true, 0>(a, p, status, st)       \
                    : launch_staged_inst<SF, DT, S, N, 0, false, 0>(a, p, status, st);     \
    }                                                                                      \
  }
  MR_STAGED_SHAPES(MR_STAGED_CASE)
#undef MR_STAGED_CASE
  return cudaErrorInvalidConfiguration;
}

template <int SF, int DT, int MODE = 0>
int staged_occupancy(const StagedPlan& p) {
  const size_t smem = p.layout.head_bytes +
      static_cast<size_t>(p.warps_per_block) * (32 / p.seg) * p.layout.seg_bytes + p.tail_bytes;
#define MR_STAGED_OCC(S, N)                                                                \
  if (p.seg == S && p.nc == N) {                                                           \
    const int w = p.warps_per_block;                                                       \
    if constexpr (MODE >= 2) {                                                             \
      if (p.km == 1)                                                                       \
        return p.full ? staged_blocks_per_sm<SF, DT, S, N, MODE, true, 1>(w, smem)         \
                      : staged_blocks_per_sm<SF, DT, S, N, MODE, false, 1>(w, smem);       \
      return p.full ? staged_blocks_per_sm<SF, DT, S, N, MODE, true, 0>(w, smem)           \
                    : staged_blocks_per_sm<SF, DT, S, N, MODE, false, 0>(w, smem);         \
    } else {                                                                               \
      if constexpr (SF != SF_SOFTMAX_POST) {                                               \
        if (p.op == 1)                                                                     \
          return p.full ? staged_blocks_per_sm<SF, DT, S, N, 1, true, 0>(w, smem)          \
                        : staged_blocks_per_sm<SF, DT, S, N, 1, false, 0>(w, smem);        \
      }                                                                                    \
      if (p.km == 1)                                                                       \
        return p.full ? staged_blocks_per_sm<SF, DT, S, N, 0, true, 1>(w, smem)            \
                      : staged_blocks_per_sm<SF, DT, S, N, 0, false, 1>(w, smem);          \
      return p.full ? staged_blocks_per_sm<SF, DT, S, N, 0, true, 0>(w, smem)              \
                    : staged_blocks_per_sm<SF, DT, S, N, 0, false, 0>(w, smem);            \
    }                                                                                      \
  }
  MR_STAGED_SHAPES(MR_STAGED_OCC)
#undef MR_STAGED_OCC
  return 0;
}

// Register-resident forward (rows of up to 512 experts; OP 0 and 2 with key
// mode 0 or 1, OP 1 with key mode 0): warps per block and the grid cap.
struct RegPlan {
  RegLayout layout;
  int warps_per_block;
  int max_blocks;  // resident blocks per SM x SMs
  int nc;          // chunks of 4 experts per lane (2 or 4)
  int op;          // 0 top-K router, 1 aux scores, 2 compact top-K outputs
  int km;          // key mode: 0 logits, 1 s + bias (and aligned groups)
  bool full;       // E == 128 * nc
};

template <int SF, int DT, int NC, int OP, bool FULL, int KM>
cudaError_t launch_reg_inst(const FwdArgs& a, const RegPlan& p, int* status, cudaStream_t st) {
  auto kern = router_fwd_reg_kernel<SF, DT, NC, OP, FULL, KM>;
  const size_t smem = static_cast<size_t>(p.warps_per_block) * p.layout.warp_bytes;
  static std::atomic<int> granted[kSmemDevs];  // this kernel's record
  const cudaError_t se = allow_smem(kern, smem, granted);
  if (se != cudaSuccess) return se;
  // rows go round-robin over the resident warps: one block per row group, or
  // every resident slot when the rows outnumber them (more warps in flight
  // measured faster than equal rounds with fewer: 9.5 against 9.8 us for the
  // 8192 x 512 aux forward)
  const long long need = (static_cast<long long>(a.T) + p.warps_per_block - 1) / p.warps_per_block;
  const long long blocks = need < p.max_blocks ? need : p.max_blocks;
  return launch_kernel(kern, dim3(static_cast<unsigned>(blocks)), dim3(p.warps_per_block * 32),
                       smem, st, a, p.layout, status);
}

template <int SF, int DT, int NC, int OP, bool FULL, int KM>
int reg_blocks_per_sm(int warps_per_block, size_t smem) {
  auto kern = router_fwd_reg_kernel<SF, DT, NC, OP, FULL, KM>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, warps_per_block * 32, smem) !=
      cudaSuccess)
    return 0;
  return n;
}

// OCC false: launch; true: resident blocks per SM (returned through *occ).
// MODE 0: top-K (OP 0) and aux (OP 1); MODE 2: compact outputs (OP 2); the
// modes live in separate translation units.
template <int SF, int DT, bool OCC, int MODE = 0>
cudaError_t reg_dispatch(const FwdArgs& a, const RegPlan& p, int* status, cudaStream_t st,
                         int* occ) {
  const size_t smem = static_cast<size_t>(p.warps_per_block) * p.layout.warp_bytes;
#define MR_REG_CASE(N, O, F, M)                                                      \
  if (p.nc == N && p.op == O && p.full == F && p.km == M) {                          \
    if constexpr (OCC) {                                                             \
      *occ = reg_blocks_per_sm<SF, DT, N, O, F, M>(p.warps_per_block, smem);         \
      return cudaSuccess;                                                            \
    } else {                                                                         \
      return launch_reg_inst<SF, DT, N, O, F, M>(a, p, status, st);                  \
    }                                                                                \
  }
  if constexpr (MODE == 2) {
    MR_REG_CASE(2, 2, true, 0) MR_REG_CASE(2, 2, false, 0) MR_REG_CASE(4, 2, true, 0)
    MR_REG_CASE(4, 2, false, 0)
    MR_REG_CASE(2, 2, true, 1) MR_REG_CASE(2, 2, false, 1) MR_REG_CASE(4, 2, true, 1)
    MR_REG_CASE(4, 2, false, 1)
  } else {
    MR_REG_CASE(2, 0, true, 0) MR_REG_CASE(2, 0, false, 0) MR_REG_CASE(4, 0, true, 0)
    MR_REG_CASE(4, 0, false, 0)
    MR_REG_CASE(2, 0, true, 1) MR_REG_CASE(2, 0, false, 1) MR_REG_CASE(4, 0, true, 1)
    MR_REG_CASE(4, 0, false, 1)
    if constexpr (SF != SF_SOFTMAX_POST) {  // aux scores take softmax or sigmoid only
      MR_REG_CASE(2, 1, true, 0) MR_REG_CASE(2, 1, false, 0) MR_REG_CASE(4, 1, true, 0)
      MR_REG_CASE(4, 1, false, 0)
    }
  }
#undef MR_REG_CASE
  return cudaErrorInvalidConfiguration;
}

#define MR_DECLARE_REG(NAME)                                                           \
  cudaError_t launch_reg_##NAME(const FwdArgs&, const RegPlan&, int*, cudaStream_t);   \
  int occupancy_reg_##NAME(const RegPlan&);                                            \
  cudaError_t launch_reg_compact_##NAME(const FwdArgs&, const RegPlan&, int*, cudaStream_t); \
  int occupancy_reg_compact_##NAME(const RegPlan&);
MR_DECLARE_REG(softmax_f32)
MR_DECLARE_REG(softmax_bf16)
MR_DECLARE_REG(sigmoid_f32)
MR_DECLARE_REG(sigmoid_bf16)
MR_DECLARE_REG(softmaxpost_f32)
MR_DECLARE_REG(softmaxpost_bf16)
#undef MR_DECLARE_REG

// One (score function, dtype) pair per translation unit.
cudaError_t launch_staged_softmax_f32(const FwdArgs&, const StagedPlan&, int*, cudaStream_t);
cudaError_t launch_staged_softmax_bf16(const FwdArgs&, const StagedPlan&, int*, cudaStream_t);
cudaError_t launch_staged_sigmoid_f32(const FwdArgs&, const StagedPlan&, int*, cudaStream_t);
cudaError_t launch_staged_sigmoid_bf16(const FwdArgs&, const StagedPlan&, int*, cudaStream_t);
int occupancy_staged_softmax_f32(const StagedPlan&);
int occupancy_staged_softmax_bf16(const StagedPlan&);
int occupancy_staged_sigmoid_f32(const StagedPlan&);
int occupancy_staged_sigmoid_bf16(const StagedPlan&);

cudaError_t launch_fwd_softmax_f32(const FwdArgs&, const FwdConfig&, cudaStream_t);
cudaError_t launch_fwd_softmaxpost_f32(const FwdArgs&, const FwdConfig&, cudaStream_t);
cudaError_t launch_fwd_softmaxpost_bf16(const FwdArgs&, const FwdConfig&, cudaStream_t);
cudaError_t launch_staged_softmaxpost_f32(const FwdArgs&, const StagedPlan&, int*, cudaStream_t);
cudaError_t launch_staged_softmaxpost_bf16(const FwdArgs&, const StagedPlan&, int*, cudaStream_t);
int occupancy_staged_softmaxpost_f32(const StagedPlan&);
int occupancy_staged_softmaxpost_bf16(const StagedPlan&);
cudaError_t launch_fwd_softmax_bf16(const FwdArgs&, const FwdConfig&, cudaStream_t);
cudaError_t launch_fwd_sigmoid_f32(const FwdArgs&, const FwdConfig&, cudaStream_t);
cudaError_t launch_fwd_sigmoid_bf16(const FwdArgs&, const FwdConfig&, cudaStream_t);
cudaError_t launch_bwd_any(int sf, int dt, const BwdArgs&, const BwdConfig&, cudaStream_t);

// Compact-output router (OP 2), both paths, one (score function, dtype)
// pair per translation unit.
#define MR_DECLARE_COMPACT(NAME)                                                     \
  cudaError_t launch_fwd_compact_##NAME(const FwdArgs&, const FwdConfig&, cudaStream_t); \
  cudaError_t launch_staged_compact_##NAME(const FwdArgs&, const StagedPlan&, int*,    \
                                           cudaStream_t);                              \
  int occupancy_staged_compact_##NAME(const StagedPlan&);
MR_DECLARE_COMPACT(softmax_f32)
MR_DECLARE_COMPACT(softmax_bf16)
MR_DECLARE_COMPACT(sigmoid_f32)
MR_DECLARE_COMPACT(sigmoid_bf16)
MR_DECLARE_COMPACT(softmaxpost_f32)
MR_DECLARE_COMPACT(softmaxpost_bf16)
#undef MR_DECLARE_COMPACT

// Fused decode router with expert maps (OP 3, staged path, one block).
#define MR_DECLARE_MAPS(NAME)                                                          \
  cudaError_t launch_staged_maps_##NAME(const FwdArgs&, const StagedPlan&, int*,       \
                                        cudaStream_t);                                 \
  int occupancy_staged_maps_##NAME(const StagedPlan&);
MR_DECLARE_MAPS(softmax_f32)
MR_DECLARE_MAPS(softmax_bf16)
MR_DECLARE_MAPS(sigmoid_f32)
MR_DECLARE_MAPS(sigmoid_bf16)
MR_DECLARE_MAPS(softmaxpost_f32)
MR_DECLARE_MAPS(softmaxpost_bf16)
#undef MR_DECLARE_MAPS

// Device address of the library's status word on the current device
// (bounded waits that give up record it there); nullptr if unavailable.
int* device_status_word();

// Stand-alone expert maps (one cooperative launch, or three) and their
// workspace size.
size_t maps_workspace_bytes(int T, int E);
int launch_expert_maps(const int32_t* idx, long long ld, int T, int E, int K, int32_t* offsets,
                       int32_t* p2u, int32_t* u2p, int32_t* pexp, void* workspace,
                       cudaStream_t st);

}  // namespace moe_router
