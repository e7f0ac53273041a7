// Device-side pieces of the router shared by the routing kernels and the
// one-launch decode layer: the deterministic sigmoid, orderable score bits,
// warp reductions, row loads and the selection of one token by one warp.
#pragma once

#include "common.cuh"

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

// 1 / (1 + e^-z) with one correctly rounded reciprocal (the same value as a
// correctly rounded division of 1 by the sum).
__device__ __forceinline__ float sigmoid_det(float z) {
  return __frcp_rn(__fadd_rn(1.0f, exp_det(-z)));
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

// Per-warp shared scratch of the selection: the row's scores (and, grouped, the
// affinities) by expert, the candidates' keys and affinities, then the selected
// terms of the gate normaliser by slot.
template <int VPL, bool GROUPED>
struct RouteSmem {
  __align__(16) float val[32 * VPL];
  __align__(16) float aff[GROUPED ? 32 * VPL : 4];
  uint64_t key[32];
  float kaff[32];
};

// Store a lane's VPL values at v[lane * VPL] (16-byte stores when VPL % 4 == 0:
// eight lanes 48 or more bytes apart fall on distinct banks).
template <int VPL>
__device__ __forceinline__ void stage_lane(float* v, int lane, const float (&x)[VPL]) {
  if (VPL % 4 == 0) {
#pragma unroll
    for (int q = 0; q < VPL / 4; ++q)
      reinterpret_cast<float4*>(v + lane * VPL)[q] =
          make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
  } else {
#pragma unroll
    for (int c = 0; c < VPL; ++c) v[lane * VPL + c] = x[c];
  }
}

// What one lane holds after selecting one token: slot (-1: none), expert, gate.
struct RouteLane {
  int slot, id;
  float gate;
};

// Selection of one token by one warp from its scores in registers: lane l holds
// experts l*VPL .. l*VPL + VPL - 1 in z (raw logits).  Every lane of the warp
// calls it.  Scores are compared as floats (+0 and -0 tie); NaN logits are
// reported through saw_nan and rank below every number.
template <int VPL, bool GROUPED>
__device__ __forceinline__ RouteLane route_token(const float (&z)[VPL], const float (&bias)[VPL],
                                                 int lane, int E, int k, int n_group,
                                                 int topk_group, float route_scale,
                                                 RouteSmem<VPL, GROUPED>& sm,
                                                 bool& saw_nan) {
  const int nv = min(max(E - lane * VPL, 0), VPL);  // this lane's experts that exist
  float sel[VPL], aff[VPL];
  if (GROUPED) {
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
      float v = z[c];
      if (v != v) { saw_nan = true; v = -INFINITY; }
      aff[c] = sigmoid_det(v);
      sel[c] = __fadd_rn(aff[c], bias[c]);
    }
  } else {
    float sum = 0.f;  // NaN iff a NaN logit (or +inf beside -inf): then the exact check
#pragma unroll
    for (int c = 0; c < VPL; ++c) { sel[c] = z[c]; sum += z[c]; aff[c] = 0.f; }
    if (__any_sync(0xFFFFFFFFu, sum != sum)) {
#pragma unroll
      for (int c = 0; c < VPL; ++c)
        if (sel[c] != sel[c]) { saw_nan = true; sel[c] = -INFINITY; }
    }
  }
  if (nv < VPL) {
#pragma unroll
    for (int c = 0; c < VPL; ++c)
      if (c >= nv) sel[c] = -INFINITY;
  }
  uint32_t live = nv >= 32 ? 0xFFFFFFFFu : (1u << nv) - 1u;  // selectable slots
  if (GROUPED) {
    // group score: the sum of the two largest corrected scores of the group's
    // gs / VPL lanes (a power of two), then the topk_group best groups (ties to
    // the lower group), each lane ranking its own group by counting
    const int lpg = (E / n_group) / VPL;
    float b1 = -INFINITY, b2 = -INFINITY;
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
      const float v = sel[c];
      if (v > b1) { b2 = b1; b1 = v; } else if (v > b2) { b2 = v; }
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
    for (int h = 0; h < n_group; ++h) {
      const float sh = __shfl_sync(0xFFFFFFFFu, gsc, h * lpg);
      grank += (sh > gsc) || (sh == gsc && h < g);
    }
    if (grank >= topk_group) live = 0u;
  }
  // theta: the k-th largest lane maximum with multiplicity, over lanes holding a
  // selectable score; with fewer such lanes every selectable score is a candidate
  float m = sel[0];
#pragma unroll
  for (int c = 1; c < VPL; ++c) m = fmaxf(m, sel[c]);
  uint32_t um = live ? ord_bits(m) : 0u;  // the orderable bits of a number or -inf are never 0
  uint32_t th_u = 0u, top_u = 0u;
  for (int r = 0; r < k; ++r) {
    const uint32_t M = __reduce_max_sync(0xFFFFFFFFu, um);
    if (r == 0) top_u = M;
    if (M == 0u) { th_u = 0u; break; }
    th_u = M;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, um == M);
    if (lane == __ffs(bal) - 1) um = 0u;
  }
  const float th = th_u ? ord_to_float(th_u) : -INFINITY;
  uint32_t cm = 0u;
#pragma unroll
  for (int c = 0; c < VPL; ++c) cm |= (sel[c] >= th ? 1u : 0u) << c;
  cm &= live;
  const int n = __popc(cm);
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  const int C = __shfl_sync(0xFFFFFFFFu, incl, 31);
  RouteLane out{-1, 0, 0.f};
  float my_val = 0.f, my_aff = 0.f;
  if (C <= 32) {
    // one candidate per lane, its slot the number of larger keys (score, then the
    // complement of the expert index)
    stage_lane<VPL>(sm.val, lane, sel);
    if (GROUPED) stage_lane<VPL>(sm.aff, lane, aff);
    __syncwarp();
    int p = incl - n;
    while (cm) {
      const int c = __ffs(cm) - 1;
      cm &= cm - 1u;
      const int e = lane * VPL + c;
      sm.key[p] = (static_cast<uint64_t>(ord_bits(sm.val[e])) << 32) |
                  (0xFFFFFFFFu - static_cast<uint32_t>(e));
      if (GROUPED) sm.kaff[p] = sm.aff[e];
      ++p;
    }
    __syncwarp();
    const uint64_t mine = lane < C ? sm.key[lane] : 0ull;
    int rank = 0;
    for (int i = 0; i < C; ++i) rank += sm.key[i] > mine;
    if (lane < C && rank < k) {
      out.slot = rank;
      out.id = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(mine));
      my_val = ord_to_float(static_cast<uint32_t>(mine >> 32));
      if (GROUPED) my_aff = sm.kaff[lane];
    }
    __syncwarp();
  } else {
    // heavy ties: k rounds of warp arg-max (lowest expert among equal scores)
    uint32_t u[VPL];
#pragma unroll
    for (int c = 0; c < VPL; ++c) u[c] = ((live >> c) & 1u) ? ord_bits(sel[c]) : 0u;
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
      if (lane == j) { out.slot = j; out.id = e; my_val = ord_to_float(gm); my_aff = av; }
    }
  }
  // the normaliser: the selected terms summed in slot order (slot j's term at lane j,
  // then the warp's xor butterfly), so every router kernel forms the same sum
  const float term = out.slot < 0 ? 0.0f
                     : GROUPED    ? my_aff
                                  : expf(my_val - ord_to_float(top_u));
  __syncwarp();
  if (out.slot >= 0) sm.kaff[out.slot] = term;
  __syncwarp();
  const float s = warp_sum(lane < k ? sm.kaff[lane] : 0.0f);
  __syncwarp();  // kaff is free for the next token
  out.gate = GROUPED ? route_scale * my_aff / s : term / s;
  return out;
}

}  // namespace
}  // namespace moe
