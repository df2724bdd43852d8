// C ABI of the router library: argument checks, kernel-path choice, launch.
// Declarations and the contract of every entry point are in moe_router.h.
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "moe_router.h"
#include "router_launch.cuh"

using namespace moe_router;

// Status word the kernels write when a bounded wait gives up (one per device).
__device__ int g_mr_device_status;

// Diagnostic: one warp waits, with a bounded wait, for an mbarrier phase
// that nothing completes; the wait gives up after limit_ns and the status
// word records the timeout, exactly as a router kernel does when a bulk copy
// never lands.
__global__ void selftest_bounded_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar, 0u, limit_ns));
  if (!ok && threadIdx.x == 0) atomicExch(status, kDeviceWaitTimeout);
}

namespace {

constexpr int kVersion = 100;

std::atomic<int> g_path{-1};       // -1: not yet read from the environment
std::atomic<int> g_fwd_lanes{0};   // 0: automatic

int current_path() {
  int p = g_path.load(std::memory_order_relaxed);
  if (p >= 0) return p;
  p = MR_PATH_AUTO;
  if (const char* env = std::getenv("MOE_ROUTER_FORCE_PATH")) {
    if (std::strcmp(env, "segment") == 0) p = MR_PATH_SEGMENT;
    else if (std::strcmp(env, "staged") == 0) p = MR_PATH_STAGED;
    else if (std::strcmp(env, "register") == 0) p = MR_PATH_REGISTER;
  }
  int expected = -1;
  g_path.compare_exchange_strong(expected, p);
  return g_path.load(std::memory_order_relaxed);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- per-device facts, read once -------------------------------------------
constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool ready;
  int sms;
  int smem_per_sm;
  int smem_per_block;
  int* status;  // device address of g_mr_device_status
};
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

bool device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               dev) != cudaSuccess ||
        cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_mr_device_status) !=
            cudaSuccess)
      return false;
    d.ready = true;
  }
  *out = d;
  return true;
}

}  // namespace

int* moe_router::device_status_word() {
  DeviceInfo di{};
  return device_info(&di) ? di.status : nullptr;
}

namespace {

// ---- staged forward plans, computed once per (device, shape) ----------------
struct PlanKey {
  int dev, sf, dt, op, km, E, K;
};
struct PlanEntry {
  PlanKey key;
  StagedPlan plan;
  bool valid;
};
constexpr int kPlanCache = 256;
PlanEntry g_plans[kPlanCache];
int g_nplans = 0;

int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Lanes per row and chunks per lane of the staged forward.  (16-lane
// segments, two rows per warp, measured slower at 256 and 512 experts: the
// two rows of a warp take different selection paths and wait for each
// other.)
void staged_shape(int E, int /*K*/, int* seg, int* nc) {
  *seg = 32;
  *nc = E <= 256 ? 2 : (E <= 512 ? 4 : (E <= 1024 ? 8 : 18));
}

StagedLayout staged_layout(int seg, int nc, int dt, int km, int op, int stages) {
  StagedLayout L{};
  const int d = dt == MR_F32 ? 4 : 2;
  L.head_bytes = km == 1 ? round_up(4 * seg * nc * 4, 128) : 0;  // the bias row
  L.stage_bytes = 4 * seg * nc * d;  // seg * nc chunks of four logits
  int off = stages * L.stage_bytes;
  if (km == 1) {
    L.work_off = off;
    off += 4 * seg * nc * 4;  // keys
    L.grp_off = off;
    off += 2 * kMaxGroups * 4;
  }
  L.cand_off = off;
  off += kCandPerLane * seg * 8;
  L.mask_off = off;
  off += round_up(seg * nc / 2, 16);  // one bit per padded expert
  if (op >= 2) {  // compact outputs: the K selected words by rank
    L.sorted_off = off;
    off += MR_MAX_TOPK * 8;
  }
  L.sel_off = off;  // renormalising top-K: the K selected scores by rank
  off += MR_MAX_TOPK * 4;
  L.bar_off = round_up(off, 16);
  off = L.bar_off + 48;
  L.seg_bytes = round_up(off, 128);
  L.steal = 0;
  L.one_stage = stages == 1 ? 1 : 0;
  return L;
}

int occupancy_any(int sf, int dt, const StagedPlan& p) {
  if (p.op == 3) {
    if (sf == MR_SOFTMAX)
      return dt == MR_F32 ? occupancy_staged_maps_softmax_f32(p)
                          : occupancy_staged_maps_softmax_bf16(p);
    if (sf == MR_SOFTMAX_POST)
      return dt == MR_F32 ? occupancy_staged_maps_softmaxpost_f32(p)
                          : occupancy_staged_maps_softmaxpost_bf16(p);
    return dt == MR_F32 ? occupancy_staged_maps_sigmoid_f32(p)
                        : occupancy_staged_maps_sigmoid_bf16(p);
  }
  if (p.op == 2) {
    if (sf == MR_SOFTMAX)
      return dt == MR_F32 ? occupancy_staged_compact_softmax_f32(p)
                          : occupancy_staged_compact_softmax_bf16(p);
    if (sf == MR_SOFTMAX_POST)
      return dt == MR_F32 ? occupancy_staged_compact_softmaxpost_f32(p)
                          : occupancy_staged_compact_softmaxpost_bf16(p);
    return dt == MR_F32 ? occupancy_staged_compact_sigmoid_f32(p)
                        : occupancy_staged_compact_sigmoid_bf16(p);
  }
  if (sf == MR_SOFTMAX)
    return dt == MR_F32 ? occupancy_staged_softmax_f32(p) : occupancy_staged_softmax_bf16(p);
  if (sf == MR_SOFTMAX_POST)
    return dt == MR_F32 ? occupancy_staged_softmaxpost_f32(p)
                        : occupancy_staged_softmaxpost_bf16(p);
  return dt == MR_F32 ? occupancy_staged_sigmoid_f32(p) : occupancy_staged_sigmoid_bf16(p);
}

// Warps per block that keep the most warps resident per SM (shared memory is
// the limit: one slice per warp).
bool staged_plan(const DeviceInfo& di, int sf, int dt, int op, int km, int E, int K,
                 StagedPlan* out) {
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_nplans; ++i) {
      const PlanKey& k = g_plans[i].key;
      if (k.dev == dev && k.sf == sf && k.dt == dt && k.op == op && k.km == km && k.E == E &&
          k.K == K) {
        *out = g_plans[i].plan;
        return g_plans[i].valid;
      }
    }
  }
  StagedPlan p{};
  staged_shape(E, K, &p.seg, &p.nc);
  p.full = E == 4 * p.seg * p.nc;
  p.layout = staged_layout(p.seg, p.nc, dt, km, op, 2);
  p.op = op;
  p.km = km;
  p.tail_bytes = op == 3 ? (2 * E + 16) * 4 : 0;  // the block's expert maps
  const int warp_bytes = (32 / p.seg) * p.layout.seg_bytes;
  int best_warps = 0;
  // tuning override: MOE_ROUTER_STAGED_WARPS caps the resident warps per SM
  int cap_warps = 64;
  if (const char* env = std::getenv("MOE_ROUTER_STAGED_WARPS")) {
    const int v = std::atoi(env);
    if (v > 0) cap_warps = v;
  }
  for (int w = 1; w <= kStagedMaxWarps; ++w) {
    const int smem = p.layout.head_bytes + w * warp_bytes + p.tail_bytes;
    if (smem > di.smem_per_block) break;
    int blocks = di.smem_per_sm / (smem + 1024);
    blocks = blocks < 2048 / (32 * w) ? blocks : 2048 / (32 * w);
    blocks = blocks < 32 ? blocks : 32;
    if (blocks * w > cap_warps) blocks = cap_warps / w;
    if (blocks > 0 && blocks * w >= best_warps) {
      best_warps = blocks * w;
      p.warps_per_block = w;
    }
  }
  bool valid = best_warps > 0;
  if (valid) {
    int per_sm = occupancy_any(sf, dt, p);
    if (per_sm * p.warps_per_block > cap_warps) per_sm = cap_warps / p.warps_per_block;
    valid = per_sm > 0;
    p.max_blocks = per_sm * di.sms;
  }
  // the stealing launch (one-warp blocks, logit keys, OP 0 to 2): how many
  // such blocks are resident at once (tuning override MOE_ROUTER_STEAL=0)
  p.steal_blocks = 0;
  static const bool steal_on = [] {
    const char* env = std::getenv("MOE_ROUTER_STEAL");
    return env == nullptr || std::strcmp(env, "0") != 0;
  }();
  if (valid && steal_on && p.seg == 32 && km == 0 && op <= 2) {
    StagedPlan one = p;
    one.warps_per_block = 1;
    int per_sm = occupancy_any(sf, dt, one);
    if (per_sm > cap_warps) per_sm = cap_warps;
    p.steal_blocks = per_sm * di.sms;
  }
  // compact-only outputs of 18-chunk rows take one stage per warp (refilled
  // once the row's candidates and sum are taken) when that keeps more warps
  // resident: at 8192x2304, K = 36, fp32, 17 warps per SM instead of 11 and
  // 22.9 against 27.6 us.  At 512 experts it measured slower (12.9 against
  // 12.1 us): there the second stage's prefetch is worth more.
  p.steal_blocks1 = 0;
  if (p.steal_blocks > 0 && op == 2 && p.nc == 18) {
    StagedPlan one = p;
    one.layout = staged_layout(p.seg, p.nc, dt, km, op, 1);
    one.warps_per_block = 1;
    int per_sm = occupancy_any(sf, dt, one);
    if (per_sm > cap_warps) per_sm = cap_warps;
    if (per_sm * di.sms > p.steal_blocks) {
      p.layout1 = one.layout;
      p.steal_blocks1 = per_sm * di.sms;
    }
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_nplans < kPlanCache)
    g_plans[g_nplans++] = PlanEntry{{dev, sf, dt, op, km, E, K}, p, valid};
  *out = p;
  return valid;
}

bool staged_shape_ok(int E, int dt) {
  return E % 4 == 0 && (dt == MR_F32 || E % 8 == 0) && E <= 2304;
}

// The staged path serves every aligned row shape unless a path is forced,
// except batches of 8192 or more rows of fewer than 128 experts, where the
// register-resident segment path measured faster (T = 16384, E = 64:
// 16.6 us against 18.9 us; at T <= 4096 the staged path is 2 to 4 times
// faster, its single-row latency being 3 us against 7).
bool use_staged(int E, int dt, bool aligned, int T) {
  if (!aligned || !staged_shape_ok(E, dt)) return false;
  const int path = current_path();
  if (path == MR_PATH_SEGMENT) return false;
  if (path == MR_PATH_STAGED) return true;
  return E >= 128 || T < 8192;
}

// ---- register-resident forward plans, computed once per (device, shape) -----
struct RegPlanEntry {
  PlanKey key;
  RegPlan plan;
  bool valid;
};
RegPlanEntry g_reg_plans[kPlanCache];
int g_nreg_plans = 0;

RegLayout reg_layout(int nc, int dt) {
  RegLayout L{};
  const int d = dt == MR_F32 ? 4 : 2;
  L.stage_bytes = 4 * 32 * nc * d;  // one padded row
  L.cand_off = 2 * L.stage_bytes;
  L.grp_off = round_up(L.cand_off + kRegCap * 4, 16);
  L.bar_off = L.grp_off + kMaxGroups * 8;
  L.warp_bytes = round_up(L.bar_off + 16, 128);
  return L;
}

int occupancy_reg_any(int sf, int dt, const RegPlan& p) {
  if (p.op == 2) {
    if (sf == MR_SOFTMAX)
      return dt == MR_F32 ? occupancy_reg_compact_softmax_f32(p)
                          : occupancy_reg_compact_softmax_bf16(p);
    if (sf == MR_SOFTMAX_POST)
      return dt == MR_F32 ? occupancy_reg_compact_softmaxpost_f32(p)
                          : occupancy_reg_compact_softmaxpost_bf16(p);
    return dt == MR_F32 ? occupancy_reg_compact_sigmoid_f32(p)
                        : occupancy_reg_compact_sigmoid_bf16(p);
  }
  if (sf == MR_SOFTMAX)
    return dt == MR_F32 ? occupancy_reg_softmax_f32(p) : occupancy_reg_softmax_bf16(p);
  if (sf == MR_SOFTMAX_POST)
    return dt == MR_F32 ? occupancy_reg_softmaxpost_f32(p) : occupancy_reg_softmaxpost_bf16(p);
  return dt == MR_F32 ? occupancy_reg_sigmoid_f32(p) : occupancy_reg_sigmoid_bf16(p);
}

// Warps per block that keep the most warps resident per SM (fewer per block
// on a tie: finer grid balance).
bool reg_plan(const DeviceInfo& di, int sf, int dt, int op, int km, int E, RegPlan* out) {
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_nreg_plans; ++i) {
      const PlanKey& k = g_reg_plans[i].key;
      if (k.dev == dev && k.sf == sf && k.dt == dt && k.op == op && k.km == km && k.E == E) {
        *out = g_reg_plans[i].plan;
        return g_reg_plans[i].valid;
      }
    }
  }
  RegPlan p{};
  p.nc = E <= 256 ? 2 : 4;
  p.full = E == 128 * p.nc;
  p.op = op;
  p.km = km;
  p.layout = reg_layout(p.nc, dt);
  int best_warps = 0, best_per_sm = 0;
  for (int w = 2; w <= kRegMaxWarps; w += 2) {
    if (static_cast<long long>(w) * p.layout.warp_bytes > di.smem_per_block) break;
    RegPlan q = p;
    q.warps_per_block = w;
    const int per_sm = occupancy_reg_any(sf, dt, q);
    if (per_sm * w > best_warps) {
      best_warps = per_sm * w;
      best_per_sm = per_sm;
      p.warps_per_block = w;
    }
  }
  const bool valid = best_warps > 0;
  p.max_blocks = best_per_sm * di.sms;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_nreg_plans < kPlanCache)
    g_reg_plans[g_nreg_plans++] = RegPlanEntry{{dev, sf, dt, op, km, E, 0}, p, valid};
  *out = p;
  return valid;
}

// The register-resident forward serves the top-K router with dense (op 0) or
// compact (op 2) outputs, with or without bias (groups only when they align
// with 4-expert chunks and sum at most kTopMRegs keys), and the aux scores
// (op 1) for aligned rows of at most 512 experts.  The automatic choice
// takes it wherever it would take the staged path, except for compact
// outputs without bias or groups: there the staged path's candidate ranking
// already orders the selection (8192 x 512, K = 22: 11.8 us against 14.0
// steady state; with bias and groups at 16384 x 256 the register path takes
// 18.9 us against 25.0).
bool use_reg(int E, int dt, bool aligned, int T, int km, int op, bool groups_ok = true) {
  if (op > 2 || (km == 1 && (op == 1 || !groups_ok)) || E > 512 || !aligned ||
      !staged_shape_ok(E, dt))
    return false;
  const int path = current_path();
  if (path == MR_PATH_SEGMENT || path == MR_PATH_STAGED) return false;
  if (path == MR_PATH_REGISTER) return true;
  if (op == 2 && km == 0) return false;
  return E >= 128 || T < 8192;
}

int launch_reg_any(int sf, int dt, const FwdArgs& a, int op, int km, cudaStream_t st) {
  DeviceInfo di{};
  if (!device_info(&di)) return MR_ERR_CUDA;
  RegPlan p{};
  if (!reg_plan(di, sf, dt, op, km, a.E, &p)) return MR_ERR_CUDA;
  cudaError_t e;
  if (op == 2) {
    if (sf == MR_SOFTMAX)
      e = dt == MR_F32 ? launch_reg_compact_softmax_f32(a, p, di.status, st)
                       : launch_reg_compact_softmax_bf16(a, p, di.status, st);
    else if (sf == MR_SOFTMAX_POST)
      e = dt == MR_F32 ? launch_reg_compact_softmaxpost_f32(a, p, di.status, st)
                       : launch_reg_compact_softmaxpost_bf16(a, p, di.status, st);
    else
      e = dt == MR_F32 ? launch_reg_compact_sigmoid_f32(a, p, di.status, st)
                       : launch_reg_compact_sigmoid_bf16(a, p, di.status, st);
    return e == cudaSuccess ? MR_OK : MR_ERR_CUDA;
  }
  if (sf == MR_SOFTMAX)
    e = dt == MR_F32 ? launch_reg_softmax_f32(a, p, di.status, st)
                     : launch_reg_softmax_bf16(a, p, di.status, st);
  else if (sf == MR_SOFTMAX_POST)
    e = dt == MR_F32 ? launch_reg_softmaxpost_f32(a, p, di.status, st)
                     : launch_reg_softmaxpost_bf16(a, p, di.status, st);
  else
    e = dt == MR_F32 ? launch_reg_sigmoid_f32(a, p, di.status, st)
                     : launch_reg_sigmoid_bf16(a, p, di.status, st);
  return e == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

int launch_staged_any(int sf, int dt, const FwdArgs& a, int op, int km, cudaStream_t st) {
  DeviceInfo di{};
  if (!device_info(&di)) return MR_ERR_CUDA;
  StagedPlan p{};
  if (!staged_plan(di, sf, dt, op, km, a.E, a.K, &p)) return MR_ERR_CUDA;
  if (op == 3 && a.T > p.warps_per_block * (32 / p.seg)) return MR_ERR_UNSUPPORTED;
  cudaError_t e;
  if (op == 3) {
    if (sf == MR_SOFTMAX)
      e = dt == MR_F32 ? launch_staged_maps_softmax_f32(a, p, di.status, st)
                       : launch_staged_maps_softmax_bf16(a, p, di.status, st);
    else if (sf == MR_SOFTMAX_POST)
      e = dt == MR_F32 ? launch_staged_maps_softmaxpost_f32(a, p, di.status, st)
                       : launch_staged_maps_softmaxpost_bf16(a, p, di.status, st);
    else
      e = dt == MR_F32 ? launch_staged_maps_sigmoid_f32(a, p, di.status, st)
                       : launch_staged_maps_sigmoid_bf16(a, p, di.status, st);
  } else if (op == 2) {
    if (sf == MR_SOFTMAX)
      e = dt == MR_F32 ? launch_staged_compact_softmax_f32(a, p, di.status, st)
                       : launch_staged_compact_softmax_bf16(a, p, di.status, st);
    else if (sf == MR_SOFTMAX_POST)
      e = dt == MR_F32 ? launch_staged_compact_softmaxpost_f32(a, p, di.status, st)
                       : launch_staged_compact_softmaxpost_bf16(a, p, di.status, st);
    else
      e = dt == MR_F32 ? launch_staged_compact_sigmoid_f32(a, p, di.status, st)
                       : launch_staged_compact_sigmoid_bf16(a, p, di.status, st);
  } else if (sf == MR_SOFTMAX) {
    e = dt == MR_F32 ? launch_staged_softmax_f32(a, p, di.status, st)
                     : launch_staged_softmax_bf16(a, p, di.status, st);
  } else if (sf == MR_SOFTMAX_POST) {
    e = dt == MR_F32 ? launch_staged_softmaxpost_f32(a, p, di.status, st)
                     : launch_staged_softmaxpost_bf16(a, p, di.status, st);
  } else {
    e = dt == MR_F32 ? launch_staged_sigmoid_f32(a, p, di.status, st)
                     : launch_staged_sigmoid_bf16(a, p, di.status, st);
  }
  return e == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

// Candidate rank whose key becomes the staged forward's next speculative
// threshold: K - 1 plus a margin (max(K / 2, 4) unless the tuning variable
// MOE_ROUTER_SPEC_MARGIN gives one).  A larger margin makes the next row's
// speculation fail less often (fewer than K candidates) but ranks more
// candidates per row.
int spec_target(int K) {
  static const int env_margin = [] {
    const char* env = std::getenv("MOE_ROUTER_SPEC_MARGIN");
    const int v = env != nullptr ? std::atoi(env) : -1;
    return v >= 0 ? v : -1;
  }();
  const int margin = env_margin >= 0 ? env_margin : (K / 2 > 4 ? K / 2 : 4);
  return K - 1 + margin;
}

int check_shape(int dtype, int T, int E, int K, int sf) {
  if (dtype != MR_F32 && dtype != MR_BF16) return MR_ERR_INVALID;
  if (sf != MR_SOFTMAX && sf != MR_SIGMOID && sf != MR_SOFTMAX_POST) return MR_ERR_INVALID;
  if (T < 0 || E < 1 || K < 1 || K > E) return MR_ERR_INVALID;
  if (static_cast<long long>(T) * static_cast<long long>(E) > INT_MAX) return MR_ERR_INVALID;
  if (E > MR_MAX_EXPERTS || K > MR_MAX_TOPK) return MR_ERR_UNSUPPORTED;
  return MR_OK;
}

int check_groups(int E, int K, int num_groups, int group_topk) {
  if (num_groups < 0) return MR_ERR_INVALID;
  if (num_groups <= 1) return MR_OK;
  if (E % num_groups != 0) return MR_ERR_INVALID;
  if (group_topk < 1 || group_topk > num_groups) return MR_ERR_INVALID;
  if (K % group_topk != 0) return MR_ERR_INVALID;
  if (K / group_topk > E / num_groups) return MR_ERR_INVALID;
  if (num_groups > MR_MAX_GROUPS) return MR_ERR_UNSUPPORTED;
  return MR_OK;
}

// Lanes per row and chunks per lane of the segment forward.  The lower bound
// needs 2 * lanes >= K disjoint groups; fewer lanes per row share the per-row
// selection work among fewer lanes and route more rows per warp.
bool choose_fwd(int E, int K, bool vec, FwdConfig* c) {
  const int chunks = (E + 3) / 4;
  if (!vec) {
    c->seg = 32;
    c->nc = 18;
    return chunks <= 32 * 18;
  }
  struct Opt { int seg, nc; };
  static const Opt opts[] = {{8, 2}, {8, 4}, {8, 8}, {16, 4}, {16, 8},
                             {32, 2}, {32, 4}, {32, 8}, {32, 18}};
  const int forced = g_fwd_lanes.load(std::memory_order_relaxed);
  for (const Opt& o : opts) {
    if (forced != 0 && o.seg != forced) continue;
    if (2 * o.seg < K) continue;
    if (o.seg * o.nc >= chunks) {
      c->seg = o.seg;
      c->nc = o.nc;
      return true;
    }
  }
  if (forced != 0) {  // the forced width cannot hold this row: automatic choice
    for (const Opt& o : opts) {
      if (2 * o.seg < K) continue;
      if (o.seg * o.nc >= chunks) { c->seg = o.seg; c->nc = o.nc; return true; }
    }
  }
  return false;
}

// Lanes x warps x chunks per row of the two-pass backwards (measured best
// per row size: more warps per row at large E keep more loads in flight).
// The softmax top-K backward of a 2304-expert row fits 7 blocks of 9 warps
// per SM (32 registers a thread); the sigmoid and post-softmax ones need 48
// and fit only 4 such blocks, so they take the aux shapes, 6 warps of 3
// chunks at that size (6 blocks per SM): 34.3 us against 40.5 us at
// 8192 x 2304, where the softmax one takes 32.9 us at 9 x 2 and 35.5 at 6 x 3.
bool choose_bwd(int E, int op, int sf, BwdConfig* c) {
  const int chunks = (E + 3) / 4;
  struct Opt { int seg, w, nc; };
  static const Opt all[] = {{8, 1, 2}, {16, 1, 4}, {32, 1, 2}, {32, 1, 4}, {32, 2, 1},
                            {32, 2, 2}, {32, 2, 4}, {32, 4, 1}, {32, 4, 2}, {32, 3, 6},
                            {32, 6, 3}, {32, 9, 2}};
  // tuning override: MOE_ROUTER_BWD_SHAPE="lanes,warps,chunks" (a compiled
  // shape that holds the row), else the table below
  if (const char* env = std::getenv("MOE_ROUTER_BWD_SHAPE")) {
    int sg = 0, w = 0, nc = 0;
    if (std::sscanf(env, "%d,%d,%d", &sg, &w, &nc) == 3) {
      for (const Opt& o : all) {
        if (o.seg == sg && o.w == w && o.nc == nc && o.seg * o.w * o.nc >= chunks) {
          c->seg = sg; c->w = w; c->nc = nc;
          return true;
        }
      }
    }
  }
  static const Opt opts_topk[] = {{8, 1, 2}, {32, 1, 2}, {32, 1, 4}, {32, 2, 4}, {32, 9, 2}};
  static const Opt opts_aux[] = {{8, 1, 2}, {32, 1, 2}, {32, 1, 4}, {32, 2, 4}, {32, 6, 3}};
  const bool topk_shapes = op == 0 && sf == MR_SOFTMAX;
  for (const Opt& o : (topk_shapes ? opts_topk : opts_aux)) {
    if (o.seg * o.w * o.nc >= chunks) {
      c->seg = o.seg; c->w = o.w; c->nc = o.nc;
      return true;
    }
  }
  return false;
}

int launch_fwd_any(int sf, int dt, const FwdArgs& a, const FwdConfig& c, cudaStream_t st) {
  cudaError_t e;
  if (c.op == 2) {
    if (sf == MR_SOFTMAX)
      e = dt == MR_F32 ? launch_fwd_compact_softmax_f32(a, c, st)
                       : launch_fwd_compact_softmax_bf16(a, c, st);
    else if (sf == MR_SOFTMAX_POST)
      e = dt == MR_F32 ? launch_fwd_compact_softmaxpost_f32(a, c, st)
                       : launch_fwd_compact_softmaxpost_bf16(a, c, st);
    else
      e = dt == MR_F32 ? launch_fwd_compact_sigmoid_f32(a, c, st)
                       : launch_fwd_compact_sigmoid_bf16(a, c, st);
  } else if (sf == MR_SOFTMAX) {
    e = dt == MR_F32 ? launch_fwd_softmax_f32(a, c, st) : launch_fwd_softmax_bf16(a, c, st);
  } else if (sf == MR_SOFTMAX_POST) {
    e = dt == MR_F32 ? launch_fwd_softmaxpost_f32(a, c, st)
                     : launch_fwd_softmaxpost_bf16(a, c, st);
  } else {
    e = dt == MR_F32 ? launch_fwd_sigmoid_f32(a, c, st) : launch_fwd_sigmoid_bf16(a, c, st);
  }
  return e == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

// Expert-map outputs of the fused decode router (op 3).
struct MapsOut {
  int32_t* offsets;
  int32_t* p2u;
  int32_t* u2p;
  int32_t* pexp;
};

// Rows of the fused decode router (op 3): one block of the staged path.
constexpr int kFusedMapsMaxTokens = 8;

// The top-K router forward behind router_topk_fwd (op 0: dense outputs),
// router_topk_fwd_compact (op 2: compact outputs, dense ones optional) and
// the fused decode router_topk_fwd_maps (op 3: op 2 + expert maps, one block
// of the staged path; MR_ERR_UNSUPPORTED when the batch does not qualify);
// arguments already checked.
int topk_fwd_launch(int op, const void* logits, int dtype, int T, int E, int K, int score_func,
                    int num_groups, int group_topk, float scaling_factor,
                    const float* expert_bias, void* probs, uint8_t* routing_map, float* scores,
                    float* topk_w, long long ld_w, int32_t* topk_i, long long ld_i,
                    int32_t* tei, mr_stream_t stream, const MapsOut* maps = nullptr) {
  auto aligned_or_null = [](const void* p) { return p == nullptr || aligned16(p); };
  const bool grouped = num_groups > 1;
  const bool vec = (E % 4 == 0) && aligned16(logits) && aligned_or_null(probs) &&
                   aligned_or_null(routing_map) && aligned_or_null(scores) &&
                   aligned_or_null(expert_bias);
  const int km = (expert_bias != nullptr || grouped) ? 1 : 0;
  const bool staged = op == 3 ? (vec && staged_shape_ok(E, dtype)) : use_staged(E, dtype, vec, T);
  if (op == 3 && (!staged || T > kFusedMapsMaxTokens)) return MR_ERR_UNSUPPORTED;
  FwdConfig c{};
  if (!staged && !choose_fwd(E, K, vec, &c)) return MR_ERR_UNSUPPORTED;
  c.vec = vec;
  c.op = op;
  c.km = km;
  c.extra_smem = (grouped && !staged)
                     ? static_cast<size_t>(kFwdThreads / c.seg) * E * sizeof(float)
                     : 0;
  if (op == 2 && !staged)  // per segment: K selected words and weights
    c.extra_smem += static_cast<size_t>(kFwdThreads / c.seg) * MR_MAX_TOPK * 12;

  FwdArgs a{};
  a.logits = logits;
  a.bias = expert_bias;
  a.probs = probs;
  a.map = routing_map;
  a.scores = scores;
  a.intermediate = nullptr;
  a.topk_w = topk_w;
  a.topk_i = topk_i;
  a.tei = tei;
  a.ld_w = ld_w;
  a.ld_i = ld_i;
  if (maps != nullptr) {
    a.maps_offsets = maps->offsets;
    a.maps_p2u = maps->p2u;
    a.maps_u2p = maps->u2p;
    a.maps_pexp = maps->pexp;
  }
  a.T = T; a.E = E; a.K = K;
  a.spec_target = spec_target(K);
  a.scaling = scaling_factor;
  a.num_groups = grouped ? num_groups : 0;
  a.group_topk = grouped ? group_topk : 0;
  // groups of a power-of-two number of 4-expert chunks (at most a warp) with
  // at most kTopMRegs keys summed are scored in registers on the staged and
  // register paths; the register path takes no other groups
  bool chunk_groups = false;
  if (grouped) {
    a.group_size = E / num_groups;
    a.per_group = K / group_topk;
    a.inv_group_size = 1.0f / static_cast<float>(a.group_size);
    const int gl = a.group_size / 4;
    chunk_groups = a.group_size % 4 == 0 && gl >= 1 && gl <= 32 && (gl & (gl - 1)) == 0 &&
                   a.per_group <= kTopMRegs;
  }
  const bool reg = use_reg(E, dtype, vec, T, km, op, !grouped || chunk_groups);
  if (grouped) {
    const bool lanes32 = staged || reg;
    const int lanes = lanes32 ? 32 : c.seg;
    int lpg = 1;
    while (lpg * 2 * num_groups <= lanes) lpg *= 2;
    a.lanes_per_group = lpg;
    a.group_chunk_lanes = (lanes32 && chunk_groups) ? a.group_size / 4 : 0;
  }
  if (reg)
    return launch_reg_any(score_func, dtype, a, op, km, reinterpret_cast<cudaStream_t>(stream));
  if (staged)
    return launch_staged_any(score_func, dtype, a, op, km, reinterpret_cast<cudaStream_t>(stream));
  return launch_fwd_any(score_func, dtype, a, c, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int router_topk_fwd(const void* logits, mr_dtype dtype, int T, int E, int K,
                    mr_score_func score_func, int num_groups, int group_topk,
                    float scaling_factor, const float* expert_bias, void* probs,
                    uint8_t* routing_map, float* scores, mr_stream_t stream) {
  int rc = check_shape(dtype, T, E, K, score_func);
  if (rc != MR_OK) return rc;
  rc = check_groups(E, K, num_groups, group_topk);
  if (rc != MR_OK) return rc;
  if (T > 0 && (logits == nullptr || probs == nullptr || routing_map == nullptr ||
                scores == nullptr))
    return MR_ERR_INVALID;
  if (T == 0) return MR_OK;
  return topk_fwd_launch(0, logits, dtype, T, E, K, score_func, num_groups, group_topk,
                         scaling_factor, expert_bias, probs, routing_map, scores, nullptr, 0,
                         nullptr, 0, nullptr, stream);
}

int router_topk_fwd_compact(const void* logits, mr_dtype dtype, int T, int E, int K,
                            mr_score_func score_func, int num_groups, int group_topk,
                            float scaling_factor, const float* expert_bias,
                            float* topk_weights, int ld_weights, int32_t* topk_indices,
                            int ld_indices, int32_t* token_expert_indices, void* probs,
                            uint8_t* routing_map, float* scores, mr_stream_t stream) {
  int rc = check_shape(dtype, T, E, K, score_func);
  if (rc != MR_OK) return rc;
  rc = check_groups(E, K, num_groups, group_topk);
  if (rc != MR_OK) return rc;
  if (ld_weights < K || ld_indices < K) return MR_ERR_INVALID;
  if (T > 0 && (logits == nullptr || topk_weights == nullptr || topk_indices == nullptr))
    return MR_ERR_INVALID;
  if (T == 0) return MR_OK;
  return topk_fwd_launch(2, logits, dtype, T, E, K, score_func, num_groups, group_topk,
                         scaling_factor, expert_bias, probs, routing_map, scores, topk_weights,
                         ld_weights, topk_indices, ld_indices, token_expert_indices, stream);
}

int router_topk_fwd_maps(const void* logits, mr_dtype dtype, int T, int E, int K,
                         mr_score_func score_func, int num_groups, int group_topk,
                         float scaling_factor, const float* expert_bias, float* topk_weights,
                         int ld_weights, int32_t* topk_indices, int ld_indices,
                         int32_t* token_expert_indices, int32_t* expert_first_token_offset,
                         int32_t* permuted_to_unpermuted, int32_t* unpermuted_to_permuted,
                         int32_t* permuted_experts, void* workspace, size_t workspace_bytes,
                         mr_stream_t stream) {
  int rc = check_shape(dtype, T, E, K, score_func);
  if (rc != MR_OK) return rc;
  rc = check_groups(E, K, num_groups, group_topk);
  if (rc != MR_OK) return rc;
  if (ld_weights < K || ld_indices < K) return MR_ERR_INVALID;
  if (T == 0) return MR_OK;
  if (logits == nullptr || topk_weights == nullptr || topk_indices == nullptr ||
      expert_first_token_offset == nullptr || permuted_to_unpermuted == nullptr ||
      unpermuted_to_permuted == nullptr || permuted_experts == nullptr)
    return MR_ERR_INVALID;
  const MapsOut maps{expert_first_token_offset, permuted_to_unpermuted, unpermuted_to_permuted,
                     permuted_experts};
  if (T <= kFusedMapsMaxTokens) {
    rc = topk_fwd_launch(3, logits, dtype, T, E, K, score_func, num_groups, group_topk,
                         scaling_factor, expert_bias, nullptr, nullptr, nullptr, topk_weights,
                         ld_weights, topk_indices, ld_indices, token_expert_indices, stream,
                         &maps);
    if (rc != MR_ERR_UNSUPPORTED) return rc;  // else: the composed launches below
  }
  if (workspace == nullptr || workspace_bytes < maps_workspace_bytes(T, E) ||
      (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
    return MR_ERR_INVALID;
  rc = topk_fwd_launch(2, logits, dtype, T, E, K, score_func, num_groups, group_topk,
                       scaling_factor, expert_bias, nullptr, nullptr, nullptr, topk_weights,
                       ld_weights, topk_indices, ld_indices, token_expert_indices, stream);
  if (rc != MR_OK) return rc;
  return launch_expert_maps(topk_indices, ld_indices, T, E, K, expert_first_token_offset,
                            permuted_to_unpermuted, unpermuted_to_permuted, permuted_experts,
                            workspace, reinterpret_cast<cudaStream_t>(stream));
}

int router_topk_bwd(const void* grad_probs, const uint8_t* routing_map,
                    const float* scores, mr_dtype dtype, int T, int E, int K,
                    mr_score_func score_func, float scaling_factor,
                    void* grad_logits, mr_stream_t stream) {
  const int rc = check_shape(dtype, T, E, K, score_func);
  if (rc != MR_OK) return rc;
  if (T > 0 && (grad_probs == nullptr || routing_map == nullptr || scores == nullptr ||
                grad_logits == nullptr))
    return MR_ERR_INVALID;
  if (T == 0) return MR_OK;
  BwdConfig c{};
  if (!choose_bwd(E, 0, score_func, &c)) return MR_ERR_UNSUPPORTED;
  c.vec = (E % 4 == 0) && aligned16(grad_probs) && aligned16(routing_map) &&
          aligned16(scores) && aligned16(grad_logits);
  c.op = 0;
  BwdArgs a{};
  a.grad = grad_probs;
  a.map = routing_map;
  a.saved = scores;
  a.grad_logits = grad_logits;
  a.T = T; a.E = E;
  a.scaling = scaling_factor;
  const cudaError_t e = launch_bwd_any(score_func, dtype, a, c,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

int router_aux_scores_fwd(const void* logits, mr_dtype dtype, int T, int E, int K,
                          mr_score_func score_func, float* scores,
                          uint8_t* routing_map, float* intermediate,
                          mr_stream_t stream) {
  const int rc = check_shape(dtype, T, E, K, score_func);
  if (rc != MR_OK) return rc;
  if (score_func == MR_SOFTMAX_POST) return MR_ERR_INVALID;  // aux scores: softmax or sigmoid
  if (T > 0 && (logits == nullptr || scores == nullptr || routing_map == nullptr ||
                (score_func == MR_SIGMOID && intermediate == nullptr)))
    return MR_ERR_INVALID;
  if (T == 0) return MR_OK;
  const bool vec = (E % 4 == 0) && aligned16(logits) && aligned16(scores) &&
                   aligned16(routing_map) &&
                   (intermediate == nullptr || aligned16(intermediate));
  FwdArgs a{};
  a.logits = logits;
  a.map = routing_map;
  a.scores = scores;
  a.intermediate = intermediate;
  a.T = T; a.E = E; a.K = K;
  a.spec_target = spec_target(K);
  a.scaling = 1.0f;
  if (use_reg(E, dtype, vec, T, 0, 1))
    return launch_reg_any(score_func, dtype, a, 1, 0, reinterpret_cast<cudaStream_t>(stream));
  if (use_staged(E, dtype, vec, T))
    return launch_staged_any(score_func, dtype, a, 1, 0, reinterpret_cast<cudaStream_t>(stream));
  FwdConfig c{};
  if (!choose_fwd(E, K, vec, &c)) return MR_ERR_UNSUPPORTED;
  c.vec = vec;
  c.op = 1;
  c.km = 0;
  c.extra_smem = 0;
  return launch_fwd_any(score_func, dtype, a, c, reinterpret_cast<cudaStream_t>(stream));
}

int router_aux_scores_bwd(const float* grad_scores, const float* saved, mr_dtype dtype,
                          int T, int E, int K, mr_score_func score_func,
                          void* grad_logits, mr_stream_t stream) {
  const int rc = check_shape(dtype, T, E, K, score_func);
  if (rc != MR_OK) return rc;
  if (score_func == MR_SOFTMAX_POST) return MR_ERR_INVALID;
  if (T > 0 && (grad_scores == nullptr || saved == nullptr || grad_logits == nullptr))
    return MR_ERR_INVALID;
  if (T == 0) return MR_OK;
  BwdConfig c{};
  if (!choose_bwd(E, 1, score_func, &c)) return MR_ERR_UNSUPPORTED;
  c.vec = (E % 4 == 0) && aligned16(grad_scores) && aligned16(saved) &&
          aligned16(grad_logits);
  c.op = 1;
  BwdArgs a{};
  a.grad = grad_scores;
  a.map = nullptr;
  a.saved = saved;
  a.grad_logits = grad_logits;
  a.T = T; a.E = E;
  a.scaling = 1.0f;
  const cudaError_t e = launch_bwd_any(score_func, dtype, a, c,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

const char* moe_router_strerror(int code) {
  switch (code) {
    case MR_OK: return "success";
    case MR_ERR_INVALID: return "invalid argument";
    case MR_ERR_UNSUPPORTED: return "unsupported size (beyond this build's limits)";
    case MR_ERR_CUDA: return "CUDA launch or runtime error";
    default: return "unknown status code";
  }
}

int moe_router_force_path(int path) {
  if (path != MR_PATH_AUTO && path != MR_PATH_SEGMENT && path != MR_PATH_STAGED &&
      path != MR_PATH_REGISTER)
    return MR_ERR_INVALID;
  const int prev = current_path();
  g_path.store(path, std::memory_order_relaxed);
  return prev;
}

int moe_router_force_fwd_lanes(int lanes) {
  if (lanes != 0 && lanes != 8 && lanes != 16 && lanes != 32) return MR_ERR_INVALID;
  return g_fwd_lanes.exchange(lanes, std::memory_order_relaxed);
}

int moe_router_device_status(int* status) {
  if (status == nullptr) return MR_ERR_INVALID;
  DeviceInfo di{};
  if (!device_info(&di)) return MR_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, di.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MR_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(di.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return MR_ERR_CUDA;
  }
  *status = v;
  return MR_OK;
}

int moe_router_selftest_bounded_wait(unsigned timeout_us, mr_stream_t stream) {
  if (timeout_us == 0 || timeout_us > 1000000u) return MR_ERR_INVALID;
  DeviceInfo di{};
  if (!device_info(&di)) return MR_ERR_CUDA;
  selftest_bounded_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      di.status, 1000ull * timeout_us);
  return cudaGetLastError() == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

int moe_router_version(void) { return kVersion; }

}  // extern "C"
