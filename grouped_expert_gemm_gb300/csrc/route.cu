// Router: top-k selection over fp32 logits with softmax-over-selected gates, or
// DeepSeek-V3 group-limited sigmoid routing.
//
// [M6.2] 0x06L1 (family table), 0x06A-0x06D and 0x06I (V3 group rule and gate).
//
// Three kernels.  route_quarter_kernel (softmax batches of tens of thousands of
// tokens with E = 128, 256, 384 or 512) gives each token four lanes.
// route_rank_kernel (the other softmax batches, and grouped routers whose expert
// groups span whole lanes) gives each token a warp and selects by threshold and
// rank, see route_token in route_dev.cuh.  route_kernel (the remaining grouped
// shapes) gives lane l the experts 32*i + l and runs k rounds of a warp
// all-reduce of 64-bit keys (orderable score bits << 32 | ~expert), so the
// maximum key is the highest score and, among equal scores, the lowest expert
// index.  In all three, +0.0 and -0.0 tie, NaN logits are reported and rank
// below every number, and the softmax normaliser is summed in slot order: the
// first two give bit-identical ids and gates.
#include "route_dev.cuh"
#include "tma.cuh"

#include <atomic>
#include <mutex>

namespace moe {
namespace {

constexpr int kTokensPerBlock = 8;

template <int VPL, bool GROUPED>
__global__ void __launch_bounds__(kTokensPerBlock * 32)
route_kernel(int T, int E, int k, int n_group, int topk_group, float route_scale,
             const float* __restrict__ logits, const float* __restrict__ sel_bias,
             int32_t* __restrict__ topk_ids, float* __restrict__ gates,
             uint32_t* __restrict__ dev_status, const int32_t* __restrict__ valid, bool early) {
  pdl_wait_then_trigger(early);
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTokensPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  if (valid != nullptr && t >= __ldg(valid)) {
    // padding slot of a fixed token bucket: no expert identity, zero gate
    if (lane < k) {
      topk_ids[static_cast<int64_t>(t) * k + lane] = MOE_ROUTE_MASKED;
      gates[static_cast<int64_t>(t) * k + lane] = 0.0f;
    }
    return;
  }
  const float* row = logits + static_cast<int64_t>(t) * E;

  float sel[VPL];  // selection score: the logit, or the corrected sigmoid s~
  float aff[VPL];  // gate source (V3: original affinity s)
  uint32_t taken = 0;
  bool saw_nan = false;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = i * 32 + lane;
    float z = -INFINITY;
    if (e < E) {
      z = __ldg(row + e);
      if (z != z) { saw_nan = true; z = -INFINITY; }
    } else {
      taken |= 1u << i;
    }
    if (GROUPED) {
      aff[i] = sigmoid_det(z);
      const float b = (sel_bias != nullptr && e < E) ? __ldg(sel_bias + e) : 0.0f;
      sel[i] = __fadd_rn(aff[i], b);
    } else {
      sel[i] = z;
      aff[i] = 0.0f;
    }
  }
  if (__any_sync(0xFFFFFFFFu, saw_nan) && lane == 0) report(dev_status, MOE_DEV_NONFINITE_LOGIT);

  if (GROUPED) {
    // Group score: sum of the two largest corrected scores of each contiguous group.
    const int gs = E / n_group;
    int grp[VPL];  // group of each of this lane's experts (one division each)
#pragma unroll
    for (int i = 0; i < VPL; ++i) grp[i] = (i * 32 + lane) / gs;
    float my_gscore = -INFINITY;
    for (int g = 0; g < n_group; ++g) {
      float b1 = -INFINITY, b2 = -INFINITY;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = i * 32 + lane;
        if (e < E && grp[i] == g) {
          const float v = sel[i];
          if (v > b1) { b2 = b1; b1 = v; } else if (v > b2) { b2 = v; }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float o1 = __shfl_xor_sync(0xFFFFFFFFu, b1, o);
        const float o2 = __shfl_xor_sync(0xFFFFFFFFu, b2, o);
        const float n1 = fmaxf(b1, o1);
        const float n2 = fmaxf(fminf(b1, o1), fmaxf(b2, o2));
        b1 = n1; b2 = n2;
      }
      if (lane == g) my_gscore = __fadd_rn(b1, b2);
    }
    // Keep the topk_group best groups (ties to the lower group index).
    uint32_t keep = 0;
    uint64_t gkey = lane < n_group ? make_key(my_gscore, lane) : 0ull;
    for (int r = 0; r < topk_group; ++r) {
      const uint64_t best = warp_max_u64(gkey);
      const int g = key_expert(best);
      keep |= 1u << g;
      if (lane == g) gkey = 0ull;
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = i * 32 + lane;
      if (e < E && !((keep >> grp[i]) & 1u)) taken |= 1u << i;
    }
  }

  // k rounds of warp arg-max over orderable 32-bit scores built once; lane j keeps
  // the j-th winner.  A round takes the lane maxima by a tree, the warp maximum,
  // then the lowest expert index holding it (a lane's experts i*32 + lane grow
  // with i, so its first slot at the maximum is its lowest): the order is score
  // descending, ties to the lower expert.  A taken expert's score is 0, below
  // every live score (the orderable bits of a number or -inf are never 0).
  uint32_t ob[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) ob[i] = ((taken >> i) & 1u) ? 0u : ord_bits(sel[i]);
  int my_id = 0;
  float my_sel = 0.0f, my_aff = 0.0f, top_sel = 0.0f;
  for (int j = 0; j < k; ++j) {
    uint32_t t[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) t[i] = ob[i];
#pragma unroll
    for (int w = 1; w < VPL; w <<= 1)
#pragma unroll
      for (int i = 0; i + w < VPL; i += 2 * w) t[i] = max(t[i], t[i + w]);
    const uint32_t gm = __reduce_max_sync(0xFFFFFFFFu, t[0]);
    uint32_t cand = 0xFFFFFFFFu;
#pragma unroll
    for (int i = VPL - 1; i >= 0; --i)
      if (ob[i] == gm) cand = static_cast<uint32_t>(i * 32 + lane);
    const int e = static_cast<int>(__reduce_min_sync(0xFFFFFFFFu, cand));
    const int owner = e & 31, slot = e >> 5;
    float a = 0.0f;
    if (lane == owner) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        if (i == slot) {
          ob[i] = 0u;
          if (GROUPED) a = aff[i];
        }
      }
    }
    if (GROUPED) a = __shfl_sync(0xFFFFFFFFu, a, owner);
    const float v = ord_to_float(gm);
    if (j == 0) top_sel = v;
    if (lane == j) { my_id = e; my_sel = v; my_aff = a; }
  }

  float g;
  if (GROUPED) {
    const float s = warp_sum(lane < k ? my_aff : 0.0f);
    g = route_scale * my_aff / s;
  } else {
    const float ex = lane < k ? expf(my_sel - top_sel) : 0.0f;
    const float s = warp_sum(ex);
    g = ex / s;
  }
  if (lane < k) {
    topk_ids[static_cast<int64_t>(t) * k + lane] = my_id;
    gates[static_cast<int64_t>(t) * k + lane] = g;
  }
  if (!early) pdl_trigger();
}

// ---- threshold-and-rank router ---------------------------------------------
//
// One warp per token at a time, in a grid-stride loop that loads the next
// token's row while it selects the current one.  Lane l holds the VPL
// consecutive experts l*VPL .. l*VPL + VPL - 1 (16-byte loads when the row
// allows), so a contiguous group of experts spans whole lanes.
//
// Selection without k serial arg-max rounds: theta = the k-th largest of the 32
// lane maxima (counted with multiplicity) is a lower bound of the k-th largest
// score, since the k lanes holding those maxima hold k scores >= theta.  Every
// score >= theta is a candidate; usually a dozen or two remain.  With at most 32
// candidates each lane takes one (64-bit key: orderable score bits, then the
// complement of the expert index) and its slot is the number of larger keys,
// which orders by score descending with ties to the lower expert.  More than 32
// candidates (heavy ties) fall back to k arg-max rounds.
constexpr int kRouteWarps = 8;

struct RouteArgs {
  int T, E, k, n_group, topk_group;
  float route_scale;
  const float* logits;
  const float* sel_bias;
  int32_t* topk_ids;
  float* gates;
  uint32_t* dev_status;
  const int32_t* valid;
};

template <int VPL, bool GROUPED, bool VEC>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_rank_kernel(RouteArgs a, bool early) {
  __shared__ RouteSmem<VPL, GROUPED> s_route[kRouteWarps];
  pdl_wait_then_trigger(early);
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int nwarps = gridDim.x * kRouteWarps;
  const int E = a.E, k = a.k;
  const int valid = a.valid != nullptr ? min(max(__ldg(a.valid), 0), a.T) : a.T;
  float bias[VPL];
#pragma unroll
  for (int c = 0; c < VPL; ++c) {
    const int e = lane * VPL + c;
    bias[c] = (GROUPED && a.sel_bias != nullptr && e < E) ? __ldg(a.sel_bias + e) : 0.f;
  }
  int t = blockIdx.x * kRouteWarps + wib;
  float cur[VPL];
  if (t < valid) load_row<VPL, VEC>(a.logits + static_cast<int64_t>(t) * E, E, lane, cur);
  bool saw_nan = false;
  for (; t < a.T; t += nwarps) {
    const int tn = t + nwarps;
    float nxt[VPL];
    if (tn < valid) load_row<VPL, VEC>(a.logits + static_cast<int64_t>(tn) * E, E, lane, nxt);
    int32_t* ids_t = a.topk_ids + static_cast<int64_t>(t) * k;
    float* gates_t = a.gates + static_cast<int64_t>(t) * k;
    if (t >= valid) {
      // padding slot of a fixed token bucket: no expert identity, zero gate
      if (lane < k) { ids_t[lane] = MOE_ROUTE_MASKED; gates_t[lane] = 0.0f; }
      continue;
    }
    const RouteLane r = route_token<VPL, GROUPED>(cur, bias, lane, E, k, a.n_group,
                                                  a.topk_group, a.route_scale, s_route[wib],
                                                  saw_nan);
    if (r.slot >= 0) {
      ids_t[r.slot] = r.id;
      gates_t[r.slot] = r.gate;
    }
#pragma unroll
    for (int c = 0; c < VPL; ++c) cur[c] = nxt[c];
  }
  if (__any_sync(0xFFFFFFFFu, saw_nan) && lane == 0) report(a.dev_status, MOE_DEV_NONFINITE_LOGIT);
  if (!early) pdl_trigger();
}

// Resident blocks per SM of a route_rank_kernel instance, read once per device.
template <int VPL, bool GROUPED, bool VEC>
int route_rank_grid(int T) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> occ[kMaxDev] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  int per_sm = (dev >= 0 && dev < kMaxDev) ? occ[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, route_rank_kernel<VPL, GROUPED, VEC>, kRouteWarps * 32, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    if (dev >= 0 && dev < kMaxDev) occ[dev].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t need = ceil_div(T, kRouteWarps);
  const int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
  return static_cast<int>(need < cap ? need : cap);
}

template <int VPL, bool GROUPED, bool VEC>
void launch_rank(const RouteArgs& a, cudaStream_t s) {
  const int grid = route_rank_grid<VPL, GROUPED, VEC>(a.T);
  launch(route_rank_kernel<VPL, GROUPED, VEC>, dim3(grid), dim3(kRouteWarps * 32), 0, s, a,
         one_wave(grid));
}

// ---- quarter-row router (large softmax batches) --------------------------------
//
// For batches far larger than the GPU (tens of thousands of tokens) the router
// is a stream of logits, and the warp-per-token kernel spends hundreds of warp
// instructions per token on warp-wide steps.  Here four lanes select one token,
// each lane a quarter of its row.  A warp takes 8 consecutive tokens at a time:
// their rows arrive by 2-D TMA boxes (8 rows x 32 experts, 128-byte swizzle) in
// one of the warp's two 12 KB (E = 384) stages, so the next batch's rows arrive
// while the current one is selected (9 warps share an SM).  Lane 4r + h holds row
// r's boxes h, h + 4, ...; the parts read their chunks in different orders so no
// two lanes of a phase meet in a bank.  For k <= 8 (quarter_select_fast):
//   1. each lane takes the maxima of the 8 chunks of its quarter; theta, the 8th
//      largest of the row's 32, is a lower bound of its k-th largest score (the
//      8 chunks holding those maxima hold 8 scores >= theta);
//   2. exactly 8 chunks reach theta (else the general selection below), and every
//      score not below theta lies in them: the row's four lanes scan two each and
//      write those scores (at most 16, else the general selection) as orderable
//      64-bit keys into the row's 16 shared-memory slots;
//   3. a bitonic network over the four lanes sorts the slots, and the gates are
//      formed exactly as the warp router does (exp against the top score, the
//      normaliser summed in the warp's slot-order butterfly).
// The general selection (any k <= 16, NaN logits, ties at theta) takes theta
// from 16 chunk maxima, inserts every score of its quarter not below theta into a
// per-lane sorted list of KS keys and merges the four lists with shuffles.
// Selection, ids and gates are identical to the warp router's either way.
constexpr int kQuarter = 4;                       // lanes per token
constexpr int kQuarterRows = 32 / kQuarter;       // tokens per warp batch
constexpr int kQuarterWarps = 16;                 // warps per block, at most

template <int NM, int KS>
struct QuarterRouter {
  static constexpr int kBoxBytes = kQuarterRows * 128;       // 1 KB: 8 rows x 32 fp32
  static constexpr int kStage = NM * kBoxBytes;              // one warp's rows
  // the fast selection's 16 candidate slots per row (the general selection merges
  // in the stage it has just read)
  static constexpr int kLists = KS == 8 ? kQuarterRows * 16 * 8 : 0;
  static constexpr int kStages = 2;                          // the next batch in flight
  static constexpr int kWarpBytes = ((kStages * kStage + kLists) + 1023) & ~1023;
  static constexpr int kFit = (227 * 1024 - 1024) / kWarpBytes;
  static constexpr int kWarps = kFit < kQuarterWarps ? kFit : kQuarterWarps;
  static constexpr int kSmem = 1024 + kWarps * kWarpBytes;
  static_assert(NM % kQuarter == 0, "whole boxes per quarter");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds_f1(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// All ones when v is not below th (or either is NaN), else zero.
__device__ __forceinline__ uint32_t not_below(float v, float th) {
  uint32_t r;
  asm("set.geu.u32.f32 %0, %1, %2;" : "=r"(r) : "f"(v), "f"(th));
  return r;
}

// Sorts 8 values descending in place (a 19-comparator network).
__device__ __forceinline__ void sort8_desc(float* x) {
  auto ce = [&](int i, int j) {
    const float hi = fmaxf(x[i], x[j]), lo = fminf(x[i], x[j]);
    x[i] = hi;
    x[j] = lo;
  };
  ce(0, 2); ce(1, 3); ce(4, 6); ce(5, 7);
  ce(0, 4); ce(1, 5); ce(2, 6); ce(3, 7);
  ce(0, 1); ce(2, 3); ce(4, 5); ce(6, 7);
  ce(2, 4); ce(3, 5);
  ce(1, 4); ce(3, 6);
  ce(1, 2); ce(3, 4); ce(5, 6);
}

// Insert (key, e) into keys sorted descending; an equal key stays ahead (the
// candidates arrive in expert order, so ties keep the lower expert first).
template <int KS>
__device__ __forceinline__ void key_insert(uint32_t (&tk)[KS], int (&ti)[KS], uint32_t key, int e) {
#pragma unroll
  for (int j = KS - 1; j > 0; --j) {
    const bool sh = key > tk[j - 1];
    const bool here = key > tk[j];
    ti[j] = sh ? ti[j - 1] : (here ? e : ti[j]);
    tk[j] = sh ? tk[j - 1] : (here ? key : tk[j]);
  }
  if (key > tk[0]) { tk[0] = key; ti[0] = e; }
}

// Bitonic merge network for 8 values that form a bitonic sequence: sorts them
// descending in place.
__device__ __forceinline__ void bitonic8_desc(float* x) {
  auto ce = [&](int i, int j) {
    const float hi = fmaxf(x[i], x[j]), lo = fminf(x[i], x[j]);
    x[i] = hi;
    x[j] = lo;
  };
  ce(0, 4); ce(1, 5); ce(2, 6); ce(3, 7);
  ce(0, 2); ce(1, 3); ce(4, 6); ce(5, 7);
  ce(0, 1); ce(2, 3); ce(4, 5); ce(6, 7);
}

// Maxima that propagate NaN: a NaN among the inputs gives NaN.
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float max2_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Compare-exchange of two 64-bit selection keys, the larger first.
__device__ __forceinline__ void ce_desc(uint64_t& a, uint64_t& b) {
  const bool sw = b > a;
  const uint64_t hi = sw ? b : a;
  b = sw ? a : b;
  a = hi;
}

// The larger (keep_max) or the smaller of a lane's key and its partner's.
__device__ __forceinline__ uint64_t keep_key(uint64_t own, uint64_t other, bool keep_max) {
  return ((own > other) == keep_max) ? own : other;
}

// Shared-memory address of float4 p (0 .. 8 * NM / 4 - 1, in the order part hp reads
// its quarter) of row r: box hp + 4 * (p / 8), logical 16-byte column (p % 8) ^ 2hp,
// stored at column ((p % 8) ^ 2hp) ^ (r % 8) by the copy's 128-byte swizzle.  The
// column's first expert is 32 * box + 4 * column.
__device__ __forceinline__ uint32_t quarter_f4(uint32_t stage, int r, int hp, int p, int& e0) {
  const int b = hp + kQuarter * (p >> 3), cc = (p & 7) ^ (2 * hp);
  e0 = 32 * b + 4 * cc;
  return stage + static_cast<uint32_t>(b * kQuarterRows * 128 + r * 128 + ((cc ^ (r & 7)) << 4));
}

// The general selection (any k <= KS, NaN logits, ties): theta from the row's 16
// chunk maxima (4 per lane, NaN ignored), every candidate of the lane's quarter
// inserted in expert order into a sorted list of KS keys, the four lists merged
// through the stage's first KS KB once its rows have been read.  Leaves the row's
// top KS keys and experts, sorted, in tk/ti of all four lanes; issue_next() runs
// after the merge, when the stage is free.
template <int NM, int KS, class F>
__device__ __forceinline__ void quarter_select_general(uint32_t stage, const uint32_t (&slot)[8],
                                                       int lane, int r,
                                                       int h, bool live, bool& saw_nan,
                                                       uint32_t (&tk)[KS], int (&ti)[KS],
                                                       F&& issue_next) {
  using R = QuarterRouter<NM, KS>;
  constexpr int kPer = NM / kQuarter;  // boxes of one quarter
  // 1. maxima of this quarter's 4 chunks (NaN ignored: an all-NaN chunk is -inf),
  //    then the row's 16 from the other quarters
  float cm[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) cm[j] = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t bx = stage + static_cast<uint32_t>((h + kQuarter * i) * R::kBoxBytes);
    float4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = lds_f4(bx + slot[c]);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int j = (8 * i + c) / (2 * kPer);  // 4 chunks of 2 * kPer float4 each
      cm[j] = fmaxf(cm[j], fmaxf(fmaxf(v[c].x, v[c].y), fmaxf(v[c].z, v[c].w)));
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) cm[4 + j] = __shfl_xor_sync(0xFFFFFFFFu, cm[j], 1);
#pragma unroll
  for (int j = 0; j < 8; ++j) cm[8 + j] = __shfl_xor_sync(0xFFFFFFFFu, cm[j], 2);
  // theta, a lower bound of the row's k-th largest score: with KS = 8 (k <= 8) the
  // 8th largest chunk maximum (the two sorted halves' pairwise maxima are the top
  // 8, theta their minimum); with KS = 16 the smallest of the 16
  float th;
  if (KS == 8) {
    sort8_desc(cm);
    sort8_desc(cm + 8);
    th = fmaxf(cm[0], cm[15]);
#pragma unroll
    for (int j = 1; j < 8; ++j) th = fminf(th, fmaxf(cm[j], cm[15 - j]));
  } else {
    th = cm[0];
#pragma unroll
    for (int j = 1; j < 16; ++j) th = fminf(th, cm[j]);
  }
  // (a warp barrier orders the shared memory: the second pass reloads the rows
  // instead of keeping the first pass's values live across the sort)
  __syncwarp();
  // 2. this quarter's candidates (not below theta; a NaN compares unordered), in
  //    expert order, into a sorted list
  uint32_t msk[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t bx = stage + static_cast<uint32_t>((h + kQuarter * i) * R::kBoxBytes);
    uint32_t m = 0u;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 v = lds_f4(bx + slot[c]);
      const int sh = 4 * (c ^ (2 * h));
      m |= (not_below(v.x, th) & (1u << sh)) | (not_below(v.y, th) & (2u << sh)) |
           (not_below(v.z, th) & (4u << sh)) | (not_below(v.w, th) & (8u << sh));
    }
    msk[i] = m;
  }
#pragma unroll
  for (int j = 0; j < KS; ++j) { tk[j] = 0u; ti[j] = 0; }
  {
    int i = 0;
    uint32_t m = msk[0];
    for (;;) {
      while (m == 0u && i + 1 < kPer) {  // the next box with candidates
        ++i;
#pragma unroll
        for (int ii = 1; ii < kPer; ++ii) m = ii == i ? msk[ii] : m;
      }
      if (m == 0u) break;
      const int e = __ffs(m) - 1;
      m &= m - 1u;
      const int b = h + kQuarter * i;
      float v = lds_f1(stage + static_cast<uint32_t>(b * R::kBoxBytes + r * 128 +
                                                     ((((e >> 2) ^ (r & 7)) & 7) << 4) + ((e & 3) << 2)));
      if (v != v) { saw_nan |= live; v = -INFINITY; }
      key_insert<KS>(tk, ti, ord_bits(v), 32 * b + e);
    }
  }
  // 3. each lane's list to shared memory over the read rows (entry-major: entry j
  //    of lane l at j * 32 + l), where the merge reads a lane's next entry
  const uint32_t lists = stage;
  __syncwarp();
#pragma unroll
  for (int j = 0; j < KS; ++j)
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(lists + static_cast<uint32_t>((j * 32 + lane) * 8)),
                 "r"(tk[j]), "r"(static_cast<uint32_t>(ti[j])) : "memory");
  __syncwarp();
  // merge: KS rounds; in each, the row's four lanes agree (two shuffle steps) on the
  // best head -- larger key, then the lower expert -- and its lane advances
  int pos = 0;
  uint32_t hk = tk[0];
  int hi = ti[0];
#pragma unroll
  for (int j = 0; j < KS; ++j) {
    uint32_t bk = hk;
    int bi = hi, bl = h;
#pragma unroll
    for (int o = 1; o < kQuarter; o <<= 1) {
      const uint32_t ok = __shfl_xor_sync(0xFFFFFFFFu, bk, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      const int ol = __shfl_xor_sync(0xFFFFFFFFu, bl, o);
      const bool better = ok > bk || (ok == bk && oi < bi);
      bk = better ? ok : bk;
      bi = better ? oi : bi;
      bl = better ? ol : bl;
    }
    tk[j] = bk;
    ti[j] = bi;
    if (bl == h && j + 1 < KS) {  // this lane's head was taken: the next entry
      ++pos;
      uint32_t kk = 0u, ii = 0u;
      if (pos < KS)
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(kk), "=r"(ii)
                     : "r"(lists + static_cast<uint32_t>((pos * 32 + lane) * 8)) : "memory");
      hk = kk;
      hi = static_cast<int>(ii);
    }
  }
  // the lists were written through the generic proxy; the copy into the same
  // bytes goes through the async proxy
  __syncwarp();
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  issue_next();
}

// The selection for k <= 8 on rows without NaN.  theta = the 8th largest of the
// row's 32 chunk maxima (8 per lane) bounds the k-th largest score from below; when
// exactly 8 chunks reach it, every score not below theta lies in those 8, and the
// row's four lanes scan two of them each (the 1st and 5th, 2nd and 6th, ... in chunk
// order), so a lane reads a quarter of what it would scan in its own quarter.  The
// candidates (at most 16 per row) go as 64-bit keys -- orderable score bits, then
// the complement of the expert, so larger means the higher score and, among equal
// scores, the lower expert -- into the row's 16 slots in shared memory, 4 per lane,
// and a bitonic network over the four lanes sorts them.  Returns false, having
// written nothing, when a live row of the batch holds a NaN, more than 8 chunks
// reach theta (a tie at theta) or more than 16 scores do; otherwise lane h < 2 of
// each row holds the row's ranks 4h .. 4h + 3 in key[], and issue_next() has run.
template <int NM, class F>
__device__ __forceinline__ bool quarter_select_fast(uint32_t stage, uint32_t lists,
                                                    const uint32_t (&slot)[8], int r, int h,
                                                    bool live, uint64_t (&key)[4],
                                                    F&& issue_next) {
  constexpr int kPer = NM / kQuarter;  // boxes of one quarter
  constexpr int kF = kPer;             // float4 per chunk: a quarter is 8 chunks
  constexpr unsigned kAll = 0xFFFFFFFFu;
  // 1. this quarter's 8 chunk maxima (a NaN anywhere in a chunk gives NaN)
  float cm[8];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t bx = stage + static_cast<uint32_t>((h + kQuarter * i) * kQuarterRows * 128);
    float4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = lds_f4(bx + slot[c]);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int p = 8 * i + c, j = p / kF;
      const float m = max3_nan(v[c].x, v[c].y, v[c].z);
      if (p % kF == 0)
        cm[j] = max2_nan(m, v[c].w);
      else
        cm[j] = max3_nan(cm[j], m, v[c].w);
    }
  }
  bool nan_row = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) nan_row |= cm[j] != cm[j];
  if (__any_sync(kAll, live && nan_row)) return false;
  // 2. theta: this lane's 8 maxima sorted, the top 8 of each lane pair (half-cleaner
  //    of the two sorted lists, then a bitonic merge), and the smallest of the top 8
  //    over the two pairs
  float w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = cm[j];
  sort8_desc(w);
  {
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = __shfl_xor_sync(kAll, w[7 - j], 1);
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = fmaxf(w[j], o[j]);
    bitonic8_desc(w);
  }
  float th;
  {
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = __shfl_xor_sync(kAll, w[7 - j], 2);
    th = fmaxf(w[0], o[0]);
#pragma unroll
    for (int j = 1; j < 8; ++j) th = fminf(th, fmaxf(w[j], o[j]));
  }
  // 3. the row's chunks that reach theta, as a mask over chunk ids 8 * part + chunk
  uint32_t qm = 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) qm |= (cm[j] >= th ? 1u : 0u) << j;
  qm <<= 8 * h;
  qm |= __shfl_xor_sync(kAll, qm, 1);
  qm |= __shfl_xor_sync(kAll, qm, 2);
  if (__any_sync(kAll, live && __popc(qm) != 8)) return false;
  // lane h takes the row's qualifying chunks h and h + 4 (rows that are not live
  // read two of their own chunks and keep nothing)
  uint32_t wm = qm;
#pragma unroll
  for (int s = 0; s < 3; ++s)
    if (s < h) wm &= wm - 1u;
  const int c0 = live ? __ffs(wm) - 1 : 8 * h;
#pragma unroll
  for (int s = 0; s < 4; ++s) wm &= wm - 1u;
  const int c1 = live ? __ffs(wm) - 1 : 8 * h + 1;
  // 4. their candidates: bit 16 * (second chunk) + 4 * float4 + component
  uint32_t lm = 0u;
#pragma unroll
  for (int u2 = 0; u2 < 2; ++u2) {
    const int cid = u2 ? c1 : c0;
#pragma unroll
    for (int u = 0; u < kF; ++u) {
      int e0;
      const float4 v = lds_f4(quarter_f4(stage, r, cid >> 3, kF * (cid & 7) + u, e0));
      const int sh = 16 * u2 + 4 * u;
      lm |= (not_below(v.x, th) & (1u << sh)) | (not_below(v.y, th) & (2u << sh)) |
            (not_below(v.z, th) & (4u << sh)) | (not_below(v.w, th) & (8u << sh));
    }
  }
  if (!live) lm = 0u;
  // 5. the row's candidate count and this lane's first slot (the lanes before it)
  const int cnt = __popc(lm);
  const int s1 = __shfl_xor_sync(kAll, cnt, 1);
  const int s2 = __shfl_xor_sync(kAll, cnt + s1, 2);
  const int ct = cnt + s1 + s2;
  if (__any_sync(kAll, ct > 16)) return false;
  int n = ((h & 1) ? s1 : 0) + ((h & 2) ? s2 : 0);
  const uint32_t row_slots = lists + static_cast<uint32_t>(r * 128);
  while (lm != 0u) {
    const int s = __ffs(lm) - 1;
    lm &= lm - 1u;
    const int cid = (s >> 4) ? c1 : c0;
    int e0;
    const uint32_t a = quarter_f4(stage, r, cid >> 3, kF * (cid & 7) + ((s >> 2) & 3), e0);
    const float v = lds_f1(a + static_cast<uint32_t>((s & 3) << 2));
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(row_slots + static_cast<uint32_t>(8 * n)),
                 "r"(0xFFFFFFFFu - static_cast<uint32_t>(e0 + (s & 3))), "r"(ord_bits(v)) : "memory");
    ++n;
  }
  __syncwarp();
  issue_next();  // the staged rows are free
  // 6. this lane's 4 slots (slots past the row's count are empty: key 0, below any
  //    score's key), then the bitonic network over the row's 16
  {
    uint32_t q[8];
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3])
                 : "r"(row_slots + static_cast<uint32_t>(32 * h)) : "memory");
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7])
                 : "r"(row_slots + static_cast<uint32_t>(32 * h + 16)) : "memory");
#pragma unroll
    for (int s = 0; s < 4; ++s)
      key[s] = 4 * h + s < ct ? (static_cast<uint64_t>(q[2 * s + 1]) << 32) | q[2 * s] : 0ull;
  }
  // each lane's 4 sorted
  ce_desc(key[0], key[1]); ce_desc(key[2], key[3]);
  ce_desc(key[0], key[2]); ce_desc(key[1], key[3]);
  ce_desc(key[1], key[2]);
  // lane pairs: half-cleaner of the two sorted 4s (the even lane keeps the larger
  // half), then each half sorted
  {
    uint64_t o[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) o[s] = __shfl_xor_sync(kAll, key[3 - s], 1);
#pragma unroll
    for (int s = 0; s < 4; ++s) key[s] = keep_key(key[s], o[s], (h & 1) == 0);
    ce_desc(key[0], key[2]); ce_desc(key[1], key[3]);
    ce_desc(key[0], key[1]); ce_desc(key[2], key[3]);
  }
  // the row: the top 8 of the two sorted 8s (lanes 0-1 against lanes 3-2), then
  // sorted across lanes 0 and 1
  {
    uint64_t o[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) o[s] = __shfl_xor_sync(kAll, key[3 - s], 3);
#pragma unroll
    for (int s = 0; s < 4; ++s) key[s] = keep_key(key[s], o[s], h < 2);
#pragma unroll
    for (int s = 0; s < 4; ++s) o[s] = __shfl_xor_sync(kAll, key[s], 1);
#pragma unroll
    for (int s = 0; s < 4; ++s) key[s] = keep_key(key[s], o[s], (h & 1) == 0);
    ce_desc(key[0], key[2]); ce_desc(key[1], key[3]);
    ce_desc(key[0], key[1]); ce_desc(key[2], key[3]);
  }
  return true;
}

template <int NM, int KS>  // E = 32 * NM experts; k <= KS
__global__ void __launch_bounds__(QuarterRouter<NM, KS>::kWarps * 32, 1)
route_quarter_kernel(const __grid_constant__ CUtensorMap map, RouteArgs a, bool early) {
  using R = QuarterRouter<NM, KS>;
  constexpr unsigned kAll = 0xFFFFFFFFu;
  extern __shared__ unsigned char q_raw[];
  __shared__ uint64_t bar[R::kWarps * R::kStages];
  __shared__ int abort_flag;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int r = lane / kQuarter, h = lane % kQuarter;
  const uint32_t base = ((smem_u32(q_raw) + 1023u) & ~1023u) + static_cast<uint32_t>(w * R::kWarpBytes);
  const uint32_t lists = base + R::kStages * R::kStage;
  if (threadIdx.x == 0) {
    for (int i = 0; i < R::kWarps * R::kStages; ++i) mbar_init(smem_u32(&bar[i]), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map)) : "memory");
  }
  __syncthreads();
  pdl_wait_then_trigger(early);
  const int k = a.k;
  const int valid = a.valid != nullptr ? min(max(__ldg(a.valid), 0), a.T) : a.T;
  const int n_batches = static_cast<int>(ceil_div(a.T, kQuarterRows));
  // Logical chunk c of this lane's box rows sits at physical slot c ^ (r & 7) (the
  // copy's swizzle); part h walks its chunks in the order c ^ 2h, so the 8 lanes of
  // a phase (2 rows x 4 parts) read 8 different bank groups.
  uint32_t slot[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) slot[c] = static_cast<uint32_t>(r * 128 + (((c ^ (2 * h)) ^ (r & 7)) << 4));
  // A warp's batches alternate between its two stages, so the next batch's rows
  // arrive while the current one is selected; rows past T are zero-filled by the copy.
  // pend bit s: a copy into stage s is in flight; ph bit s: the parity of its phase.
  auto issue = [&](int st, int batch) {
    if (lane == 0) {
      const uint32_t ba = smem_u32(&bar[w * R::kStages + st]);
      mbar_arrive_expect_tx(ba, R::kStage);
#pragma unroll
      for (int b = 0; b < NM; ++b)
        tma_load_2d(base + static_cast<uint32_t>(st * R::kStage + b * R::kBoxBytes), &map, ba, b * 32,
                    batch * kQuarterRows);
    }
  };
  const int stride = gridDim.x * R::kWarps, first = blockIdx.x * R::kWarps + w;
  uint32_t pend = 0u, ph = 0u;
  bool saw_nan = false;
  for (int st = 0; st < R::kStages; ++st)
    if (first + st * stride < n_batches) { issue(st, first + st * stride); pend |= 1u << st; }
  int it = 0;
  for (int bt = first; bt < n_batches; bt += stride, ++it) {
    const int t0 = bt * kQuarterRows, t = t0 + r;
    const int st = it % R::kStages;
    const uint32_t stage = base + static_cast<uint32_t>(st * R::kStage);
    if (!__all_sync(kAll, wait_bounded(smem_u32(&bar[w * R::kStages + st]), (ph >> st) & 1u,
                                       &abort_flag, a.dev_status)))
      break;
    pend &= ~(1u << st);
    ph ^= 1u << st;
    const bool live = t < valid;  // every lane works; only live rows are written
    // the batch after next into this stage, as soon as this batch's rows are no
    // longer read
    auto issue_next = [&]() {
      const int nb = bt + R::kStages * stride;
      if (nb < n_batches) { issue(st, nb); pend |= 1u << st; }
    };
    int32_t* ids_t = a.topk_ids + static_cast<int64_t>(t) * k;
    float* gates_t = a.gates + static_cast<int64_t>(t) * k;
    if constexpr (KS == 8) {
      uint64_t key[4];
      if (!quarter_select_fast<NM>(stage, lists, slot, r, h, live, key, issue_next)) {
        uint32_t tk[8];
        int ti[8];
        quarter_select_general<NM, 8>(stage, slot, lane, r, h, live, saw_nan, tk, ti, issue_next);
        const bool odd = (h & 1) != 0;  // lane h < 2 holds ranks 4h .. 4h + 3
#pragma unroll
        for (int s = 0; s < 4; ++s)
          key[s] = (static_cast<uint64_t>(odd ? tk[4 + s] : tk[s]) << 32) |
                   (0xFFFFFFFFu - static_cast<uint32_t>(odd ? ti[4 + s] : ti[s]));
      }
      // gates: lane h takes ranks j0 = 4 (h % 2) + 2 (h / 2) and j0 + 1 (lanes 2 and 3
      // from lanes 0 and 1), exp against the top score, and the normaliser in the warp
      // router's slot order ((e0 + e4) + (e2 + e6)) + ((e1 + e5) + (e3 + e7)): the
      // xor-1 partner holds the rank 4 apart, the xor-2 partner the rank 2 apart
      const float top = ord_to_float(__shfl_sync(kAll, static_cast<uint32_t>(key[0] >> 32), lane & ~3));
      const bool far = h >= 2;
      const uint64_t f2 = __shfl_xor_sync(kAll, key[2], 2), f3 = __shfl_xor_sync(kAll, key[3], 2);
      const uint64_t ka = far ? f2 : key[0], kb = far ? f3 : key[1];
      const int j0 = 4 * (h & 1) + 2 * (h >> 1);
      const float ea = j0 < k ? expf(ord_to_float(static_cast<uint32_t>(ka >> 32)) - top) : 0.0f;
      const float eb = j0 + 1 < k ? expf(ord_to_float(static_cast<uint32_t>(kb >> 32)) - top) : 0.0f;
      const float pa = ea + __shfl_xor_sync(kAll, ea, 1), pb = eb + __shfl_xor_sync(kAll, eb, 1);
      const float ssum = (pa + __shfl_xor_sync(kAll, pa, 2)) + (pb + __shfl_xor_sync(kAll, pb, 2));
      if (live) {
        if (j0 < k) {
          ids_t[j0] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(ka));
          gates_t[j0] = ea / ssum;
        }
        if (j0 + 1 < k) {
          ids_t[j0 + 1] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(kb));
          gates_t[j0 + 1] = eb / ssum;
        }
      } else if (t < a.T) {
        // padding slot of a fixed token bucket: no expert identity, zero gate
        for (int j = h; j < k; j += kQuarter) { ids_t[j] = MOE_ROUTE_MASKED; gates_t[j] = 0.0f; }
      }
    } else {
      uint32_t tk[KS];
      int ti[KS];
      quarter_select_general<NM, KS>(stage, slot, lane, r, h, live, saw_nan, tk, ti, issue_next);
      // gates: exp against the top score; the normaliser in the warp's order; each of
      // the row's lanes divides and stores the slots j = h, h + 4, ...
      const float top = ord_to_float(tk[0]);
      float ex[KS];
#pragma unroll
      for (int j = 0; j < KS; ++j) ex[j] = j < k ? expf(ord_to_float(tk[j]) - top) : 0.0f;
      float wv[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) wv[j] = j < KS ? ex[j < KS ? j : 0] : 0.0f;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1)
#pragma unroll
        for (int ii = 0; ii < o; ++ii) wv[ii] = wv[ii] + wv[ii + o];
      const float ssum = wv[0];
      if (live) {
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          if (j % kQuarter == h && j < k) {
            ids_t[j] = ti[j];
            gates_t[j] = ex[j] / ssum;
          }
        }
      } else if (t < a.T) {
        // padding slot of a fixed token bucket: no expert identity, zero gate
        for (int j = h; j < k; j += kQuarter) { ids_t[j] = MOE_ROUTE_MASKED; gates_t[j] = 0.0f; }
      }
    }
    __syncwarp();  // every lane is done with the stage and the lists before the refill
  }
  if (lane == 0)  // copies still in flight after a timeout
    for (int st = 0; st < R::kStages; ++st)
      if (pend & (1u << st)) wait_drain(smem_u32(&bar[w * R::kStages + st]), (ph >> st) & 1u);
  if (__any_sync(kAll, saw_nan) && lane == 0) report(a.dev_status, MOE_DEV_NONFINITE_LOGIT);
  if (!early) pdl_trigger();
}

// The logits as a 2-D TMA view [T, E] fp32, boxes of 32 experts x 8 rows with the
// 128-byte swizzle, kept in a small cache (an encoding depends only on these values).
bool lane_map(CUtensorMap* out, const float* logits, int T, int E) {
  struct Entry {
    const float* p;
    int T, E;
    CUtensorMap map;
  };
  constexpr int kCache = 8;
  static Entry cache[kCache];
  static int used = 0, next = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].p == logits && cache[i].T == T && cache[i].E == E) { *out = cache[i].map; return true; }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(E), static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(E) * 4};
  const cuuint32_t box[2] = {32, kQuarterRows};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(logits), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache[next] = Entry{logits, T, E, m};
  next = (next + 1) % kCache;
  if (used < kCache) ++used;
  *out = m;
  return true;
}

template <int NM, int KS>
moe_status launch_lane(const RouteArgs& a, const CUtensorMap& map, cudaStream_t s) {
  using R = QuarterRouter<NM, KS>;
  auto kern = route_quarter_kernel<NM, KS>;
  constexpr int kMaxDev = 64;
  static std::atomic<int> ready[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MOE_ERR_CUDA;
  if (!ready[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, R::kSmem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    ready[dev].store(1, std::memory_order_relaxed);
  }
  const int64_t batches = ceil_div(a.T, kQuarterRows);
  const int64_t need = ceil_div(batches, R::kWarps);
  const int grid = static_cast<int>(need < sm_count() ? need : sm_count());
  launch(kern, dim3(grid), dim3(R::kWarps * 32), R::kSmem, s, map, a, one_wave(grid));
  return launch_status();
}

// The quarter-row router takes softmax batches of at least two 8-token batches per
// warp of a full wave (below that the warp-per-token kernel has more parallelism
// and the lower latency), E = 32 * NM with NM in {4, 8, 12, 16}, 16-byte aligned rows.
bool lane_shape(int T, int E, int k, const float* logits) {
  const int nm = E / 32;
  if (E % 32 != 0 || (nm != 4 && nm != 8 && nm != 12 && nm != 16) || k > 16) return false;
  if (!aligned16(logits)) return false;
  return static_cast<int64_t>(T) >= static_cast<int64_t>(2) * kQuarterRows * kQuarterWarps * sm_count();
}

moe_status launch_lane_any(const RouteArgs& a, cudaStream_t s, bool* done) {
  *done = false;
  CUtensorMap map;
  if (!lane_map(&map, a.logits, a.T, a.E)) return MOE_OK;  // the warp router instead
  *done = true;
  const bool k8 = a.k <= 8;
  switch (a.E / 32) {
    case 4: return k8 ? launch_lane<4, 8>(a, map, s) : launch_lane<4, 16>(a, map, s);
    case 8: return k8 ? launch_lane<8, 8>(a, map, s) : launch_lane<8, 16>(a, map, s);
    case 12: return k8 ? launch_lane<12, 8>(a, map, s) : launch_lane<12, 16>(a, map, s);
    default: return k8 ? launch_lane<16, 8>(a, map, s) : launch_lane<16, 16>(a, map, s);
  }
}

// Lanes per expert group of the rank kernel's layout when groups span whole
// lanes in a power of two, else 0 (the grouped router then takes the one-slot-
// per-lane kernel above).
inline int lanes_per_group(int E, int n_group, int vpl) {
  const int gs = E / n_group;
  if (gs % vpl != 0) return 0;
  const int lpg = gs / vpl;
  return (lpg > 0 && lpg <= 32 && (lpg & (lpg - 1)) == 0) ? lpg : 0;
}

template <bool GROUPED>
moe_status launch_route(const moe_route_params* p, const float* logits, const float* sel_bias,
                        int32_t* ids, float* gates, uint32_t* st, cudaStream_t s,
                        const int32_t* valid) {
  int vpl = static_cast<int>(ceil_div(p->E, 32));
  vpl = vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : vpl <= 12 ? 12 : 16;
  if (!GROUPED || lanes_per_group(p->E, p->n_group, vpl) > 0) {
    const RouteArgs a{p->T, p->E, p->k, p->n_group, p->topk_group, p->route_scale, logits,
                      sel_bias, ids, gates, st, valid};
    if (!GROUPED && lane_shape(p->T, p->E, p->k, logits)) {
      bool done = false;
      const moe_status r = launch_lane_any(a, s, &done);
      if (done) return r;
    }
    const bool vec = vpl % 4 == 0 && p->E % 4 == 0 && aligned16(logits);
#define MOE_RANK_CASE(V)                                                   \
  do {                                                                     \
    if (vec) launch_rank<V, GROUPED, true>(a, s);                          \
    else launch_rank<V, GROUPED, false>(a, s);                             \
  } while (0)
    switch (vpl) {
      case 1: launch_rank<1, GROUPED, false>(a, s); break;
      case 2: launch_rank<2, GROUPED, false>(a, s); break;
      case 4: MOE_RANK_CASE(4); break;
      case 8: MOE_RANK_CASE(8); break;
      case 12: MOE_RANK_CASE(12); break;
      default: MOE_RANK_CASE(16); break;
    }
#undef MOE_RANK_CASE
    return launch_status();
  }
  const dim3 grid(static_cast<unsigned>(ceil_div(p->T, kTokensPerBlock)));
  const dim3 block(kTokensPerBlock * 32);
  const bool early = one_wave(grid.x);
#define MOE_ROUTE_CASE(V)                                                                \
  launch(route_kernel<V, GROUPED>, grid, block, 0, s, p->T, p->E, p->k, p->n_group,        \
         p->topk_group, p->route_scale, logits, sel_bias, ids, gates, st, valid, early)
  if (vpl <= 1) MOE_ROUTE_CASE(1);
  else if (vpl <= 2) MOE_ROUTE_CASE(2);
  else if (vpl <= 4) MOE_ROUTE_CASE(4);
  else if (vpl <= 8) MOE_ROUTE_CASE(8);
  else if (vpl <= 12) MOE_ROUTE_CASE(12);
  else MOE_ROUTE_CASE(16);
#undef MOE_ROUTE_CASE
  return launch_status();
}

__global__ void sigmoid_det_kernel(int64_t n, const float* __restrict__ z, float* __restrict__ s) {
  pdl_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    s[i] = sigmoid_det(z[i]);
  pdl_trigger();
}

// Decode bucket staging: the step's logits and token rows into rows [0, T) of
// the bucket's stable buffers, and the real token count into its device int32.
// One grid-stride pass over both copies (16-byte units where both sides allow).
__global__ void bucket_stage_kernel(int T, int64_t n_logit_vec, int64_t n_logit,
                                    int64_t n_x_vec, const float4* __restrict__ logits_v,
                                    const float* __restrict__ logits, float4* __restrict__ dst_v,
                                    float* __restrict__ dst, const uint4* __restrict__ x,
                                    uint4* __restrict__ x_dst, int32_t* __restrict__ valid) {
  pdl_wait();  // the previous step's kernels may still read the stable buffers
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  for (int64_t i = i0; i < n_logit_vec; i += stride) dst_v[i] = __ldg(logits_v + i);
  for (int64_t i = n_logit_vec * 4 + i0; i < n_logit; i += stride) dst[i] = __ldg(logits + i);
  for (int64_t i = i0; i < n_x_vec; i += stride) x_dst[i] = __ldg(x + i);
  if (i0 == 0) *valid = T;
  pdl_trigger();
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API moe_status moe_bucket_stage(int32_t T, int32_t E, int32_t d, const float* logits,
                                    const moe_bf16* x, float* logits_dst, moe_bf16* x_dst,
                                    int32_t* valid_tokens, moe_stream_t stream) {
  if (T < 0 || E <= 0 || d <= 0 || valid_tokens == nullptr) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (logits == nullptr || x == nullptr || logits_dst == nullptr || x_dst == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (d % 8 != 0 || (T > 0 && (!aligned16(x) || !aligned16(x_dst)))) return MOE_ERR_UNSUPPORTED;
  const int64_t n_logit = static_cast<int64_t>(T) * E;
  const bool vec = aligned16(logits) && aligned16(logits_dst);
  const int64_t n_logit_vec = vec ? n_logit / 4 : 0;
  const int64_t n_x_vec = static_cast<int64_t>(T) * d / 8;
  const int64_t work = n_logit_vec + (n_logit - 4 * n_logit_vec) + n_x_vec;
  int64_t blocks = ceil_div(work > 0 ? work : 1, 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  launch(bucket_stage_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
         as_cuda(stream), T, n_logit_vec, n_logit, n_x_vec,
         reinterpret_cast<const float4*>(logits), logits, reinterpret_cast<float4*>(logits_dst),
         logits_dst, reinterpret_cast<const uint4*>(x), reinterpret_cast<uint4*>(x_dst),
         valid_tokens);
  return launch_status();
}

static moe_status route_impl(const moe_route_params* p, const int32_t* valid, const float* logits,
                             const float* sel_bias, int32_t* topk_ids, float* gates,
                             uint32_t* dev_status, moe_stream_t stream) {
  if (p == nullptr || logits == nullptr || topk_ids == nullptr || gates == nullptr)
    return p && p->T == 0 ? MOE_OK : MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->E <= 0 || p->k <= 0 || p->k > p->E) return MOE_ERR_INVALID_ARG;
  if (p->E > 512 || p->k > 16) return MOE_ERR_UNSUPPORTED;
  if (p->T == 0) return MOE_OK;
  if (p->score_fn == MOE_SCORE_SOFTMAX) {
    if (sel_bias != nullptr) return MOE_ERR_INVALID_ARG;
    return launch_route<false>(p, logits, nullptr, topk_ids, gates, dev_status, as_cuda(stream),
                               valid);
  }
  if (p->score_fn != MOE_SCORE_SIGMOID_GROUP) return MOE_ERR_INVALID_ARG;
  if (p->n_group <= 0 || p->topk_group <= 0 || p->topk_group > p->n_group ||
      p->E % p->n_group != 0)
    return MOE_ERR_INVALID_ARG;
  if (p->n_group > 32 || p->E / p->n_group < 2 || p->topk_group * (p->E / p->n_group) < p->k)
    return MOE_ERR_UNSUPPORTED;
  return launch_route<true>(p, logits, sel_bias, topk_ids, gates, dev_status, as_cuda(stream),
                            valid);
}

MOE_API moe_status moe_route(const moe_route_params* p, const float* logits,
                             const float* sel_bias, int32_t* topk_ids, float* gates,
                             uint32_t* dev_status, moe_stream_t stream) {
  return route_impl(p, nullptr, logits, sel_bias, topk_ids, gates, dev_status, stream);
}

MOE_API moe_status moe_route_bucket(const moe_route_params* p, const int32_t* valid_tokens,
                                    const float* logits, const float* sel_bias,
                                    int32_t* topk_ids, float* gates, uint32_t* dev_status,
                                    moe_stream_t stream) {
  if (valid_tokens == nullptr) return MOE_ERR_INVALID_ARG;
  return route_impl(p, valid_tokens, logits, sel_bias, topk_ids, gates, dev_status, stream);
}

MOE_API moe_status moe_sigmoid_det(int64_t n, const float* z, float* s, moe_stream_t stream) {
  if (n < 0 || (n > 0 && (z == nullptr || s == nullptr))) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  const int64_t blocks = ceil_div(n, 256);
  launch(sigmoid_det_kernel, dim3(static_cast<unsigned>(blocks < 152 * 64 ? blocks : 152 * 64)),
         dim3(256), 0, as_cuda(stream), n, z, s);
  return launch_status();
}
