// Router: top-k selection over fp32 logits with softmax-over-selected gates, or
// DeepSeek-V3 group-limited sigmoid routing.
//
// [M6.2] 0x06L1 (family table), 0x06A-0x06D and 0x06I (V3 group rule and gate).
//
// Two kernels.  route_rank_kernel (every softmax router, and grouped routers
// whose expert groups span whole lanes) selects by threshold and rank, see
// route_token in route_dev.cuh.  route_kernel (the remaining grouped shapes)
// gives lane l the experts 32*i + l and runs k rounds of a warp all-reduce of
// 64-bit keys (orderable score bits << 32 | ~expert), so the maximum key is the
// highest score and, among equal scores, the lowest expert index.  In both,
// +0.0 and -0.0 tie, and NaN logits are reported and rank below every number.
#include "route_dev.cuh"

#include <atomic>

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
