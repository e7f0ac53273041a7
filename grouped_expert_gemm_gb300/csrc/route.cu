// Router: top-k selection over fp32 logits with softmax-over-selected gates, or
// DeepSeek-V3 group-limited sigmoid routing.
//
// [M6.2] 0x06L1 (family table), 0x06A-0x06D and 0x06I (V3 group rule and gate).
//
// One warp owns one token.  Lane l holds experts e = 32*i + l (coalesced 128-byte
// row segments per load).  Each selection round is a warp all-reduce of 64-bit
// keys (orderable score bits << 32 | ~expert), so the maximum key is the highest
// score and, among equal scores, the lowest expert index; +0.0 and -0.0 are
// folded together first so they tie.  NaN logits are reported and replaced by
// -inf, which ranks below every number.
#include "common.cuh"

#include <atomic>

namespace moe {
namespace {

// ---- deterministic fp32 sigmoid -------------------------------------------
// e^x: Cody-Waite reduction with ln2 split at 16 significant bits, degree-7
// Taylor polynomial of e^r in Horner form, scale by 2^n from exponent bits.
// Every step is an explicitly rounded single fp32 operation (no contraction),
// so a host implementation of the same steps gets identical bits.
__device__ __forceinline__ float exp_det(float x) {
  x = fminf(fmaxf(x, -87.0f), 87.0f);
  const float n = rintf(__fmul_rn(x, 0x1.715476p+0f));                 // x * log2(e)
  const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(n, 0x1.62e4p-1f)),  // - n * ln2_hi
                            __fmul_rn(n, 0x1.7f7d1cp-20f));            // - n * ln2_lo
  float p = 0x1.a01a02p-13f;                                           // 1/7!
  p = __fadd_rn(__fmul_rn(p, r), 0x1.6c16c2p-10f);                     // 1/6!
  p = __fadd_rn(__fmul_rn(p, r), 0x1.111112p-7f);                      // 1/5!
  p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-5f);                      // 1/4!
  p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-3f);                      // 1/3!
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);                                // 1/2!
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);                                // 1/1!
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);                                // 1/0!
  const float two_n = __uint_as_float(static_cast<uint32_t>(static_cast<int>(n) + 127) << 23);
  return __fmul_rn(p, two_n);
}

__device__ __forceinline__ float sigmoid_det(float z) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, exp_det(-z)));
}

// Orderable bits of a float: unsigned comparison of the result follows float order.
__device__ __forceinline__ uint32_t ord_bits(float v) {
  if (v == 0.0f) v = 0.0f;  // fold -0.0 into +0.0
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float ord_to_float(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

__device__ __forceinline__ uint64_t make_key(float v, int e) {
  return (static_cast<uint64_t>(ord_bits(v)) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - e);
}

__device__ __forceinline__ int key_expert(uint64_t key) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}

// Warp maximum of 64-bit keys with two 32-bit reductions: the high words first,
// then the low words of the lanes that hold the maximal high word.
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
  const uint32_t hi = static_cast<uint32_t>(v >> 32);
  const uint32_t mhi = __reduce_max_sync(0xFFFFFFFFu, hi);
  const uint32_t lo = hi == mhi ? static_cast<uint32_t>(v) : 0u;
  const uint32_t mlo = __reduce_max_sync(0xFFFFFFFFu, lo);
  return (static_cast<uint64_t>(mhi) << 32) | mlo;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

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

template <int VPL, bool VEC>
__device__ __forceinline__ void load_row(const float* __restrict__ row, int E, int lane,
                                         float (&v)[VPL]) {
  const int e0 = lane * VPL;
  if (VEC) {
#pragma unroll
    for (int q = 0; q < VPL / 4; ++q) {
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e0 + 4 * q < E) f = __ldg(reinterpret_cast<const float4*>(row + e0) + q);
      v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int c = 0; c < VPL; ++c) v[c] = e0 + c < E ? __ldg(row + e0 + c) : 0.f;
  }
}

template <int VPL, bool GROUPED, bool VEC>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_rank_kernel(RouteArgs a, bool early) {
  __shared__ uint64_t s_key[kRouteWarps][32];
  __shared__ float s_aff[kRouteWarps][32];
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
    // selection keys: 0 marks "not selectable" (the orderable bits of a number or
    // -inf are never 0)
    uint32_t u[VPL];
    float aff[VPL];
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
      const int e = lane * VPL + c;
      float z = cur[c];
      if (z != z) { saw_nan = true; z = -INFINITY; }
      float sel = z;
      aff[c] = 0.f;
      if (GROUPED) {
        aff[c] = sigmoid_det(z);
        sel = __fadd_rn(aff[c], bias[c]);
      }
      cur[c] = sel;
      u[c] = e < E ? ord_bits(sel) : 0u;
    }
    if (GROUPED) {
      // group score: the sum of the two largest corrected scores of the group's
      // gs / VPL lanes (a power of two), then the topk_group best groups
      // (ties to the lower group), each lane ranking its own group by counting
      const int gs = E / a.n_group, lpg = gs / VPL;
      float b1 = -INFINITY, b2 = -INFINITY;
#pragma unroll
      for (int c = 0; c < VPL; ++c) {
        if (lane * VPL + c < E) {
          const float v = cur[c];
          if (v > b1) { b2 = b1; b1 = v; } else if (v > b2) { b2 = v; }
        }
      }
      for (int o = 1; o < lpg; o <<= 1) {
        const float o1 = __shfl_xor_sync(0xFFFFFFFFu, b1, o);
        const float o2 = __shfl_xor_sync(0xFFFFFFFFu, b2, o);
        const float n1 = fmaxf(b1, o1);
        const float n2 = fmaxf(fminf(b1, o1), fmaxf(b2, o2));
        b1 = n1; b2 = n2;
      }
      const float gsc = __fadd_rn(b1, b2);
      const int g = lane / lpg;
      int grank = 0;
      for (int h = 0; h < a.n_group; ++h) {
        const float sh = __shfl_sync(0xFFFFFFFFu, gsc, h * lpg);
        grank += (sh > gsc) || (sh == gsc && h < g);
      }
      if (lane * VPL >= E || grank >= a.topk_group) {
#pragma unroll
        for (int c = 0; c < VPL; ++c) u[c] = 0u;
      }
    }
    // theta: the k-th largest lane maximum, with multiplicity; when fewer than k
    // lanes hold a selectable score, every selectable score is a candidate
    uint32_t m = u[0];
#pragma unroll
    for (int c = 1; c < VPL; ++c) m = max(m, u[c]);
    uint32_t theta = 1u, top = 0u;
    for (int r = 0; r < k; ++r) {
      const uint32_t M = __reduce_max_sync(0xFFFFFFFFu, m);
      if (r == 0) top = M;
      if (M == 0u) { theta = 1u; break; }
      theta = M;
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, m == M);
      if (lane == __ffs(bal) - 1) m = 0u;
    }
    uint32_t cmask = 0;
#pragma unroll
    for (int c = 0; c < VPL; ++c) cmask |= (u[c] >= theta ? 1u : 0u) << c;
    const int n = __popc(cmask);
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const int C = __shfl_sync(0xFFFFFFFFu, incl, 31);
    // what this lane ends with: slot `my_slot` (or -1) holding expert my_id
    int my_slot = -1, my_id = 0;
    float my_val = 0.f, my_aff = 0.f;
    if (C <= 32) {
      int p = incl - n;
#pragma unroll
      for (int c = 0; c < VPL; ++c) {
        if ((cmask >> c) & 1u) {
          const int e = lane * VPL + c;
          s_key[wib][p] = (static_cast<uint64_t>(u[c]) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e));
          s_aff[wib][p] = aff[c];
          ++p;
        }
      }
      __syncwarp();
      const uint64_t mine = lane < C ? s_key[wib][lane] : 0ull;
      int rank = 0;
      for (int i = 0; i < C; ++i) rank += s_key[wib][i] > mine;
      if (lane < C && rank < k) {
        my_slot = rank;
        my_id = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(mine));
        my_val = ord_to_float(static_cast<uint32_t>(mine >> 32));
        my_aff = s_aff[wib][lane];
      }
      __syncwarp();
    } else {
      // heavy ties: k rounds of warp arg-max (lowest expert among equal scores)
      for (int j = 0; j < k; ++j) {
        uint32_t lm = u[0];
#pragma unroll
        for (int c = 1; c < VPL; ++c) lm = max(lm, u[c]);
        const uint32_t gm = __reduce_max_sync(0xFFFFFFFFu, lm);
        uint32_t cand = 0xFFFFFFFFu;
#pragma unroll
        for (int c = VPL - 1; c >= 0; --c)
          if (u[c] == gm) cand = static_cast<uint32_t>(lane * VPL + c);
        const int e = static_cast<int>(__reduce_min_sync(0xFFFFFFFFu, cand));
        const int owner = e / VPL, slot = e - owner * VPL;
        float av = 0.f;
        if (lane == owner) {
#pragma unroll
          for (int c = 0; c < VPL; ++c)
            if (c == slot) { u[c] = 0u; av = aff[c]; }
        }
        av = __shfl_sync(0xFFFFFFFFu, av, owner);
        if (lane == j) { my_slot = j; my_id = e; my_val = ord_to_float(gm); my_aff = av; }
      }
    }
    float g;
    if (GROUPED) {
      const float s = warp_sum(my_slot >= 0 ? my_aff : 0.0f);
      g = a.route_scale * my_aff / s;
    } else {
      const float ex = my_slot >= 0 ? expf(my_val - ord_to_float(top)) : 0.0f;
      const float s = warp_sum(ex);
      g = ex / s;
    }
    if (my_slot >= 0) {
      ids_t[my_slot] = my_id;
      gates_t[my_slot] = g;
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
