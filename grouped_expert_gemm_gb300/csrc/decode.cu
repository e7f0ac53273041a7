// One-launch MoE layer for small batches (decode steps of a few tokens).
//
// The whole layer of [M6.6] 0x03 and 0x04 -- route, admission and count/prefix,
// permutation with both maps, SwiGLU over the expert segments, gate-weighted
// fp32 combine -- as one kernel, for T*k <= 64 routes.  At that size the layer
// is a stream of the touched experts' weights (one-token decode: 8 experts x
// 4.7 MB); split into six kernels it is bound by their launch gaps and first
// loads instead, and each GEMM pass keeps only part of the SMs streaming.
//
// Every CTA first routes all T tokens and builds the permutation in shared
// memory on its own (a few KB of logits; identical results in every CTA, so no
// grid-wide step is needed).  CTA 0 writes the routing and the maps out.  A
// segment's rows are cut into row groups of up to four.  One producer warp per
// CTA then claims work units from a global counter, in this order:
//   gate/up units  (row group, 64 columns of I): all d rows of W_gate and W_up
//   down units     (row group, 64 columns of d): all I rows of W_down
// and streams each unit's weight boxes (256 rows x 128 bytes) with TMA into a
// ring of shared-memory stages, running ahead of the eight consumer warps.  The
// consumers multiply on CUDA cores (a row group holds a row or two here: the
// tensor cores would pad it to 128) and, with the whole K range in one CTA,
// reduce in a fixed order and write H (SiLU epilogue) or y (bf16) directly: no
// partial sums leave the CTA and the result is deterministic.  A down unit
// waits, with a bounded wait, until its row group's H is complete: every unit
// it can wait on was claimed before it by a running CTA, and a CTA consumes its
// units in claim order with all gate/up units before any down unit, so the
// wait always ends.  The CTA that completes the last row group of a column
// block of y forms that block of the combined output for every token.
// Counters live in the caller's workspace, zero before a call and zeroed again
// by the last CTA to finish, so the call can be replayed from a CUDA graph.
#include "route_dev.cuh"
#include "tma.cuh"

#include <atomic>
#include <mutex>

namespace moe {
namespace {

constexpr int kConsumers = 256;               // eight consumer warps
constexpr int kProducerWarp = kConsumers / 32;
constexpr int kSignalWarp = kProducerWarp + 1;
constexpr int kDecThreads = kConsumers + 64;  // plus the producer and the signal warp
constexpr int kDecWarps = kConsumers / 32;    // warps that route tokens
constexpr int kDecMaxRoutes = 64;  // T*k
constexpr int kDecMaxT = 16;
constexpr int kDecMaxTd = 16384;   // T*d: the token rows staged in shared memory
constexpr int kDecMaxE = 512;
constexpr int kCols = 64;          // columns of a unit: 128 bytes of bf16 per weight row
constexpr int kCG = kCols / 8;     // 16-byte column groups of a weight row
constexpr int kKLanes = kConsumers / kCG;  // weight rows read side by side (32)
constexpr int kKSlice = 128;       // weight rows per box
constexpr int kKIter = kKSlice / kKLanes;  // weight rows per thread per box (4)
constexpr int kRG = 4;             // rows of a row group (accumulated together)
constexpr int kDecMaxI = 2048;     // the H rows of a row group staged in shared memory
constexpr int kMaxStages = 8;      // shared-memory ring of weight boxes (fewer if it must)
constexpr int kStageBytes = kKSlice * kCols * 2;  // 16 KB
constexpr int kSigSlots = 4;       // finished units waiting for the signal warp
constexpr int kMaxSplit = 4;       // row slices of d a gate/up unit may be cut into
constexpr int kSplitBlocks = 512;  // (row group, column block) pairs that may be cut
constexpr int kConsumerBar = 1;    // named barrier of the consumer warps

struct DecodeArgs {
  int T, E, k, d, I, capacity, n_group, topk_group;
  float route_scale;
  const int32_t* valid;
  const float* logits;
  const float* sel_bias;
  const uint16_t* x;
  int32_t* topk_ids;
  float* gates;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_to_route;
  int32_t* route_to_row;
  int32_t* n_dropped;
  uint16_t* x_perm;
  uint16_t* h;
  uint16_t* y;
  float* out;
  uint32_t* ctr;  // counters (CtrLayout)
  float* part;    // partial G and U of cut gate/up units
  uint32_t* dev_status;
};

// The three weight tensors as 2-D TMA views: W_gate and W_up as [E*d, I], W_down
// as [E*I, d], boxes of 256 rows x 64 columns.
struct DecodeMaps {
  CUtensorMap wg, wu, wd;
};

// Counter layout in the workspace (32-bit words): unit claims, finished CTAs,
// completed gate/up units per row group, completed row groups per column block of y.
struct CtrLayout {
  int n_ci, n_cd;  // column blocks of I and of d
  __host__ __device__ static int claim() { return 0; }
  __host__ __device__ static int done() { return 1; }
  __host__ __device__ static int h_ready() { return 2; }                 // [64]
  __host__ __device__ int y_ready() const { return 2 + kDecMaxRoutes; }  // [n_cd]
  __host__ __device__ int gu_fin() const { return y_ready() + n_cd; }    // [64 * n_ci]
  __host__ __device__ int words() const { return gu_fin() + kDecMaxRoutes * n_ci; }
};

// Workspace bytes of the counters (the fp32 partial sums of cut gate/up units follow).
__host__ __device__ inline size_t ctr_bytes(const CtrLayout& L) {
  return (static_cast<size_t>(L.words()) * 4 + 255) & ~size_t(255);
}
// One cut part's partial G and U: [kRG rows][2][kCols] fp32.
constexpr int kPartFloats = kRG * 2 * kCols;

__host__ __device__ inline int n_slices(int rows) { return (rows + kKSlice - 1) / kKSlice; }

// Shared memory of one CTA other than the ring of weight boxes.
template <int VPL, bool GROUPED>
struct DecodeRest {
  union {
    RouteSmem<VPL, GROUPED> route[kDecWarps];
    float red[kRG][kConsumers / 32][2][kCols];  // per-warp sums of a unit
  } u;
  __align__(16) uint16_t xs[kDecMaxTd];                  // token rows [T, d]
  __align__(16) uint16_t hs[kRG * kDecMaxI];             // H rows of the current down unit
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t sig_full[kSigSlots], sig_empty[kSigSlots];
  int32_t stage_unit[kMaxStages];  // unit of the box (at a unit's first box); -1: no more units
  int32_t pending[kMaxStages];     // a TMA box issued and not yet waited for (its parity + 1)
  int32_t sig_unit[kSigSlots];     // finished unit handed to the signal warp; -1: stop
  int32_t ids[kDecMaxRoutes];
  float gates[kDecMaxRoutes];
  int32_t r2row[kDecMaxRoutes];                 // route -> row (-1 dropped/padding)
  int32_t row2r[kDecMaxRoutes];                 // row -> route
  int32_t cnt[kDecMaxE];                        // demand, then admitted counts
  int32_t off[kDecMaxE + 1];
  int32_t rg_e[kDecMaxRoutes], rg_b[kDecMaxRoutes], rg_n[kDecMaxRoutes];  // row groups
  int32_t n_rg, n_drop, flag, cur, first_unit, nsplit;
  int abort;
};

// Ring stages that fit beside the rest of the shared memory (at most kMaxStages).
template <int VPL, bool GROUPED>
constexpr int ring_stages() {
  constexpr size_t budget = 227 * 1024 - 256;
  constexpr size_t rest = (sizeof(DecodeRest<VPL, GROUPED>) + 127) & ~size_t(127);
  constexpr size_t n = (budget - rest) / kStageBytes;
  return n >= kMaxStages ? kMaxStages : static_cast<int>(n);
}

// Shared memory of one CTA: the rest, then the ring of weight boxes (TMA
// destinations, 128-byte aligned).
template <int VPL, bool GROUPED>
struct DecodeSmem : DecodeRest<VPL, GROUPED> {
  static constexpr int kStages = ring_stages<VPL, GROUPED>();
  __align__(128) uint8_t ring[kStages][kStageBytes];
};

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Counter increment that publishes the CTA's earlier global writes: called by one
// thread after a barrier of the writers (cumulative release at GPU scope).
__device__ __forceinline__ uint32_t add_release(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void fence_acquire() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kConsumerBar), "n"(kConsumers) : "memory");
}

// Barrier of the consumer warps that also returns the AND of every consumer's v
// (the others pass true, so thread 0's decision reaches all of them at once).
__device__ __forceinline__ bool consumer_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kConsumerBar), "n"(kConsumers)
      : "memory");
  return r != 0;
}

// Bounded wait of one thread until *p >= target; false if it gave up.
__device__ bool wait_at_least(const uint32_t* p, uint32_t target) {
  constexpr uint64_t kLimitNs = 1000000000ull;  // one second
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire(p) < target) {
    if (global_timer_ns() - t0 > kLimitNs) return false;
    __nanosleep(64);
  }
  return true;
}

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// The CTA's own copy of routing and permutation for all T tokens.
template <int VPL, bool GROUPED, bool VEC>
__device__ void decode_prologue(const DecodeArgs& a, DecodeSmem<VPL, GROUPED>& s, int valid) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int T = a.T, E = a.E, k = a.k, R = T * k;
  // the token rows (the permuted copy and the gate/up units read them from here),
  // loaded first: they do not depend on the routing
  {
    const int n16 = valid * a.d / 8;
    for (int i = tid; i < n16; i += kDecThreads)
      reinterpret_cast<uint4*>(s.xs)[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
  }
  // 1. routing: one consumer warp per token
  if (w < kDecWarps) {
    float bias[VPL];
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
      const int e = lane * VPL + c;
      bias[c] = (GROUPED && a.sel_bias != nullptr && e < E) ? __ldg(a.sel_bias + e) : 0.f;
    }
    bool saw_nan = false;
    for (int t = w; t < T; t += kDecWarps) {
      if (t >= valid) {
        if (lane < k) { s.ids[t * k + lane] = MOE_ROUTE_MASKED; s.gates[t * k + lane] = 0.f; }
        continue;
      }
      float z[VPL];
      load_row<VPL, VEC>(a.logits + static_cast<int64_t>(t) * E, E, lane, z);
      const RouteLane r = route_token<VPL, GROUPED>(z, bias, lane, E, k, a.n_group,
                                                    a.topk_group, a.route_scale, s.u.route[w],
                                                    saw_nan);
      if (r.slot >= 0) { s.ids[t * k + r.slot] = r.id; s.gates[t * k + r.slot] = r.gate; }
    }
    if (blockIdx.x == 0 && __any_sync(0xFFFFFFFFu, saw_nan) && lane == 0)
      report(a.dev_status, MOE_DEV_NONFINITE_LOGIT);
  }
  for (int e = tid; e < E; e += kDecThreads) s.cnt[e] = 0;
  __syncthreads();
  // 2. admission in route-id order: demand per expert, then each route's ordinal
  if (tid < R) {
    const int e = s.ids[tid];
    if (e >= 0) atomicAdd(&s.cnt[e], 1);
  }
  __syncthreads();
  if (w == 0) {
    // admitted counts, drops, offsets with sentinel and the row groups of the
    // segments: lane l takes experts [l*per, (l+1)*per), then a warp scan
    const int per = (E + 31) / 32, e0 = lane * per, e1 = min(E, e0 + per);
    int acc = 0, drops = 0, ng = 0;
    for (int e = e0; e < e1; ++e) {
      const int n = s.cnt[e];
      const int c = a.capacity < 0 ? n : min(n, a.capacity);
      drops += n - c;
      acc += c;
      ng += (c + kRG - 1) / kRG;
    }
    int acc_x = acc, ng_x = ng;  // inclusive scans over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int va = __shfl_up_sync(0xFFFFFFFFu, acc_x, o);
      const int vg = __shfl_up_sync(0xFFFFFFFFu, ng_x, o);
      if (lane >= o) { acc_x += va; ng_x += vg; }
    }
    int off = acc_x - acc, g = ng_x - ng;
    for (int e = e0; e < e1; ++e) {
      const int n = s.cnt[e];
      const int c = a.capacity < 0 ? n : min(n, a.capacity);
      s.off[e] = off;
      s.cnt[e] = c;
      for (int r = 0; r < c; r += kRG) {
        s.rg_e[g] = e;
        s.rg_b[g] = off + r;
        s.rg_n[g] = min(kRG, c - r);
        ++g;
      }
      off += c;
    }
    drops = __reduce_add_sync(0xFFFFFFFFu, drops);
    if (lane == 31) { s.off[E] = acc_x; s.n_rg = ng_x; s.n_drop = drops; }
  }
  __syncthreads();
  if (tid < R) {
    const int e = s.ids[tid];
    int row = -1;
    if (e >= 0) {
      int ord = 0;
      for (int q = 0; q < tid; ++q) ord += s.ids[q] == e;
      if (ord < s.cnt[e]) row = s.off[e] + ord;
    }
    s.r2row[tid] = row;
    if (row >= 0) s.row2r[row] = tid;
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    if (tid < R) {
      a.topk_ids[tid] = s.ids[tid];
      a.gates[tid] = s.gates[tid];
      a.route_to_row[tid] = s.r2row[tid];
      if (tid < s.off[E]) a.row_to_route[tid] = s.row2r[tid];
    }
    for (int e = tid; e < E; e += kDecThreads) { a.counts[e] = s.cnt[e]; a.offsets[e] = s.off[e]; }
    if (tid == 0) { a.offsets[E] = s.off[E]; *a.n_dropped = s.n_drop; }
  }
  // the permuted copy of the token rows, spread over the CTAs
  if (a.x_perm != nullptr) {
    const int chunks = a.d / 8;
    for (int row = blockIdx.x; row < s.off[E]; row += gridDim.x) {
      const int t = s.row2r[row] / k;
      for (int c = tid; c < chunks; c += kDecThreads)
        reinterpret_cast<uint4*>(a.x_perm + static_cast<int64_t>(row) * a.d)[c] =
            reinterpret_cast<const uint4*>(s.xs + t * a.d)[c];
    }
  }
}

// ---- work units ----------------------------------------------------------------
// Gate/up unit u < n_gu: row group q, column block cb of I, part p of nsplit
// (rows [p, p+1) * d / nsplit of W_gate and W_up; nsplit > 1 only when the row
// groups are too few to give every SM its own units).  Down unit u >= n_gu: row
// group q, column block cb of d, all I rows of W_down.
struct Unit {
  int q, cb, part;
  bool gu;
};
__device__ __forceinline__ Unit unit_of(int u, int n_gu, int n_ci, int n_cd, int nsplit) {
  if (u < n_gu) return Unit{u / (n_ci * nsplit), (u / nsplit) % n_ci, u % nsplit, true};
  const int v = u - n_gu;
  return Unit{v / n_cd, v % n_cd, 0, false};
}

// ---- producer warp: claims units in order and streams their weight boxes ------
// A gate/up unit is the boxes W_gate[ks], W_up[ks] of its row slices (pairs of
// stages); a down unit is W_down[ks] for ks = 0 .. I/256, issued once its row
// group's H is complete (checked once per row group: counts only grow).  The next
// unit is claimed while the current one is issued.  Lane 0 claims and issues;
// the warp stays converged.
template <int VPL, bool GROUPED>
__device__ void producer(const DecodeArgs& a, const DecodeMaps& m, DecodeSmem<VPL, GROUPED>& s,
                         int n_ci, int n_cd, int n_gu, int n_all, int nsplit) {
  constexpr int NS = DecodeSmem<VPL, GROUPED>::kStages;
  const int lane = threadIdx.x & 31;
  const int nks_d = n_slices(a.d), nks_i = n_slices(a.I), per_part = nks_d / nsplit;
  int st = 0;
  uint32_t ph = 0;
  uint64_t ready = 0;  // row groups whose H this CTA has seen complete
  int u = s.first_unit, nxt = 0;  // the first unit was claimed before the prologue
  if (lane == 0 && u < n_all) nxt = static_cast<int>(atomicAdd(a.ctr + CtrLayout::claim(), 1u));
  nxt = __shfl_sync(0xFFFFFFFFu, nxt, 0);
  for (;;) {
    const bool more = u < n_all;
    bool ok = true;
    if (lane == 0) {
      Unit un{0, 0, 0, true};
      if (more) un = unit_of(u, n_gu, n_ci, n_cd, nsplit);
      if (more && !un.gu && !((ready >> un.q) & 1ull)) {
        ok = !*reinterpret_cast<volatile int*>(&s.abort) &&
             wait_at_least(a.ctr + CtrLayout::h_ready() + un.q, static_cast<uint32_t>(n_ci));
        if (!ok) { report(a.dev_status, MOE_DEV_TIMEOUT); s.abort = 1; }
        ready |= 1ull << un.q;
      }
      const int e = more ? s.rg_e[un.q] : 0;
      const int boxes = !more ? 1 : (un.gu ? 2 * per_part : nks_i);
      for (int bx = 0; bx < boxes && ok; ++bx) {
        ok = wait_bounded(smem_u32(&s.empty[st]), ph ^ 1u, &s.abort, a.dev_status);
        if (!ok) break;
        if (!more) {
          s.stage_unit[st] = -1;
          mbar_arrive(smem_u32(&s.full[st]));  // completes the phase without data
          break;
        }
        s.stage_unit[st] = u;
        s.pending[st] = static_cast<int>(ph) + 1;
        mbar_arrive_expect_tx(smem_u32(&s.full[st]), kStageBytes);
        const CUtensorMap* map = un.gu ? ((bx & 1) ? &m.wu : &m.wg) : &m.wd;
        const int row0 = un.gu ? e * a.d + (un.part * per_part + (bx >> 1)) * kKSlice
                               : e * a.I + bx * kKSlice;
        tma_load_2d(smem_u32(s.ring[st]), map, smem_u32(&s.full[st]), un.cb * kCols, row0);
        if (++st == NS) { st = 0; ph ^= 1u; }
      }
      if (ok && more && *reinterpret_cast<volatile int*>(&s.abort)) ok = false;
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
    if (!ok || !more) return;
    // the claimed-ahead unit becomes current; claim the one after it
    u = nxt;
    if (lane == 0 && u < n_all) nxt = static_cast<int>(atomicAdd(a.ctr + CtrLayout::claim(), 1u));
    nxt = __shfl_sync(0xFFFFFFFFu, nxt, 0);
  }
}

// Consumer thread 0 waits (bounded) on `count` consecutive ring stages from (st, ph),
// then tells the other consumers through a reducing barrier: every consumer
// thread takes the same decision at the same point, so a named barrier is never
// left waiting for a thread that gave up.  Returns false when the CTA stops.
template <int NS>
__device__ __forceinline__ bool take_stages(uint64_t* bars, int32_t* pending, int st, uint32_t ph,
                                            int count, int* abort, uint32_t* dev_status) {
  bool ok = true;
  if (threadIdx.x == 0) {
    ok = !*reinterpret_cast<volatile int*>(abort);
    for (int i = 0; i < count && ok; ++i) {
      ok = wait_bounded(smem_u32(&bars[st]), ph, abort, dev_status);
      if (ok) pending[st] = 0;
      if (++st == NS) { st = 0; ph ^= 1u; }
    }
  }
  return consumer_and(ok);
}

// Hand a stage back to the producer: one arrival per consumer warp, after the
// warp's last read of it.
__device__ __forceinline__ void release_stage(uint64_t* empty) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(empty));
}

// Per-warp reduction of acc[c] (this thread's weight rows, columns cg*8 + c) over
// the warp's weight-row lanes (the lane bits above the column group), in a fixed
// order; lanes 0 .. kCG-1 then hold the warp's sums for columns lane*8 .. lane*8+7.
__device__ __forceinline__ void warp_rows_sum(float (&acc)[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
#pragma unroll
    for (int o = kCG; o < 32; o <<= 1) acc[c] += __shfl_xor_sync(0xFFFFFFFFu, acc[c], o);
}

// One W_gate / W_up box pair for N rows: this thread's weight rows k0 + kl + 64 i,
// columns cg*8 .. cg*8+7 (the box pointers are offset by cg already).  Rows of the
// box past this expert's d rows (the next expert's, or the zero fill past the
// tensor) meet a zero activation.
template <int N>
__device__ __forceinline__ void gu_box(const uint8_t* wgs, const uint8_t* wus,
                                       const uint16_t* const (&xr)[kRG], int k0, int kl, int d,
                                       float (&ag)[kRG][8], float (&au)[kRG][8]) {
#pragma unroll
  for (int i = 0; i < kKIter; ++i) {
    const int row = kl + kKLanes * i, kr = k0 + row;
    float fg[8], fu[8];
    unpack8(lds128(wgs + row * (kCols * 2)), fg);
    unpack8(lds128(wus + row * (kCols * 2)), fu);
#pragma unroll
    for (int r = 0; r < N; ++r) {
      const float xv = kr < d ? bf16f(xr[r][kr]) : 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        ag[r][c] = fmaf(xv, fg[c], ag[r][c]);
        au[r][c] = fmaf(xv, fu[c], au[r][c]);
      }
    }
  }
}

// One W_down box for N rows of H staged in hs ([kRG][I]); rows past I (the next
// expert's) meet a zero activation.
template <int N>
__device__ __forceinline__ void dn_box(const uint8_t* wds, const uint16_t* hs, int k0, int kl,
                                       int I, float (&ay)[kRG][8]) {
#pragma unroll
  for (int i = 0; i < kKIter; ++i) {
    const int row = kl + kKLanes * i, kr = k0 + row;
    float f[8];
    unpack8(lds128(wds + row * (kCols * 2)), f);
#pragma unroll
    for (int r = 0; r < N; ++r) {
      const float hv = kr < I ? bf16f(hs[r * I + kr]) : 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) ay[r][c] = fmaf(hv, f[c], ay[r][c]);
    }
  }
}

// Consumers: hand a finished unit (its outputs written) to the signal warp.
template <int VPL, bool GROUPED>
__device__ __forceinline__ bool hand_over(const DecodeArgs& a, DecodeSmem<VPL, GROUPED>& s,
                                          int unit, int& sig, uint32_t& sph) {
  consumer_sync();  // every consumer's writes of the unit's outputs are issued
  bool ok = true;
  if (threadIdx.x == 0) {
    ok = wait_bounded(smem_u32(&s.sig_empty[sig]), sph ^ 1u, &s.abort, a.dev_status);
    if (ok) {
      s.sig_unit[sig] = unit;
      mbar_arrive(smem_u32(&s.sig_full[sig]));  // releases the CTA's writes before it
    }
  }
  if (++sig == kSigSlots) { sig = 0; sph ^= 1u; }
  return consumer_and(ok);
}

// Consumers: one gate/up unit.  Uncut, it writes H for its rows and columns; cut,
// it writes its part's fp32 partial G and U and the signal warp forms H.
template <int VPL, bool GROUPED>
__device__ bool gate_up_unit(const DecodeArgs& a, DecodeSmem<VPL, GROUPED>& s, const Unit& un,
                             int n_ci, int nsplit, int& st, uint32_t& ph) {
  constexpr int NS = DecodeSmem<VPL, GROUPED>::kStages;
  const int tid = threadIdx.x, kl = tid / kCG, cg = tid % kCG, lane = tid & 31, w = tid >> 5;
  const int b = s.rg_b[un.q], n = s.rg_n[un.q], col0 = un.cb * kCols;
  const int per_part = n_slices(a.d) / nsplit;
  float ag[kRG][8], au[kRG][8];
  const uint16_t* xr[kRG];
#pragma unroll
  for (int r = 0; r < kRG; ++r) {
    xr[r] = s.xs + (s.row2r[b + min(r, n - 1)] / a.k) * a.d;
#pragma unroll
    for (int c = 0; c < 8; ++c) { ag[r][c] = 0.f; au[r][c] = 0.f; }
  }
  for (int j = 0; j < per_part; ++j) {
    if (!take_stages<NS>(s.full, s.pending, st, ph, 2, &s.abort, a.dev_status)) return false;
    const int sg = st, su = st + 1 == NS ? 0 : st + 1;
    const uint8_t* wgs = s.ring[sg] + cg * 16;
    const uint8_t* wus = s.ring[su] + cg * 16;
    const int k0 = (un.part * per_part + j) * kKSlice;
    switch (n) {
      case 1: gu_box<1>(wgs, wus, xr, k0, kl, a.d, ag, au); break;
      case 2: gu_box<2>(wgs, wus, xr, k0, kl, a.d, ag, au); break;
      case 3: gu_box<3>(wgs, wus, xr, k0, kl, a.d, ag, au); break;
      default: gu_box<4>(wgs, wus, xr, k0, kl, a.d, ag, au); break;
    }
    release_stage(&s.empty[sg]);
    release_stage(&s.empty[su]);
    st = su + 1 == NS ? 0 : su + 1;
    if (su + 1 == NS || sg + 1 == NS) ph ^= 1u;
  }
  // sums over the weight-row lanes: within each warp, then across the warps in order
#pragma unroll
  for (int r = 0; r < kRG; ++r) {
    if (r < n) {
      warp_rows_sum(ag[r]);
      warp_rows_sum(au[r]);
      if (lane < kCG) {
        float4* dg = reinterpret_cast<float4*>(&s.u.red[r][w][0][cg * 8]);
        float4* du = reinterpret_cast<float4*>(&s.u.red[r][w][1][cg * 8]);
        dg[0] = make_float4(ag[r][0], ag[r][1], ag[r][2], ag[r][3]);
        dg[1] = make_float4(ag[r][4], ag[r][5], ag[r][6], ag[r][7]);
        du[0] = make_float4(au[r][0], au[r][1], au[r][2], au[r][3]);
        du[1] = make_float4(au[r][4], au[r][5], au[r][6], au[r][7]);
      }
    }
  }
  consumer_sync();
  // thread -> (row, two columns)
  const int r = tid / (kCols / 2), c2 = (tid % (kCols / 2)) * 2;
  if (r < n) {
    float g[2] = {0.f, 0.f}, u[2] = {0.f, 0.f};
#pragma unroll
    for (int ww = 0; ww < kConsumers / 32; ++ww) {
      g[0] += s.u.red[r][ww][0][c2]; g[1] += s.u.red[r][ww][0][c2 + 1];
      u[0] += s.u.red[r][ww][1][c2]; u[1] += s.u.red[r][ww][1][c2 + 1];
    }
    if (nsplit == 1) {
      float hv[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) hv[i] = __fdividef(g[i], 1.0f + __expf(-g[i])) * u[i];
      *reinterpret_cast<uint32_t*>(a.h + static_cast<int64_t>(b + r) * a.I + col0 + c2) =
          pack_bf16x2(hv[0], hv[1]);
    } else {
      float* pp = a.part + (static_cast<int64_t>(un.q * n_ci + un.cb) * nsplit + un.part) * kPartFloats;
      *reinterpret_cast<float2*>(pp + (r * 2 + 0) * kCols + c2) = make_float2(g[0], g[1]);
      *reinterpret_cast<float2*>(pp + (r * 2 + 1) * kCols + c2) = make_float2(u[0], u[1]);
    }
  }
  return true;
}

// Consumers: one down unit (row group q, columns cb*64 .. cb*64+63 of d).
template <int VPL, bool GROUPED>
__device__ bool down_unit(const DecodeArgs& a, DecodeSmem<VPL, GROUPED>& s, const Unit& un,
                          int& st, uint32_t& ph) {
  constexpr int NS = DecodeSmem<VPL, GROUPED>::kStages;
  const int tid = threadIdx.x, kl = tid / kCG, cg = tid % kCG, lane = tid & 31, w = tid >> 5;
  const int b = s.rg_b[un.q], n = s.rg_n[un.q];
  const int nks = n_slices(a.I), col0 = un.cb * kCols;
  float ay[kRG][8];
#pragma unroll
  for (int r = 0; r < kRG; ++r)
#pragma unroll
    for (int c = 0; c < 8; ++c) ay[r][c] = 0.f;
  // the row group's H rows into shared memory, one L2 round trip per unit (H was
  // written by other CTAs; the producer saw it complete before issuing the unit)
  for (int i = tid; i < n * (a.I / 8); i += kConsumers)
    reinterpret_cast<uint4*>(s.hs)[i] =
        __ldcg(reinterpret_cast<const uint4*>(a.h + static_cast<int64_t>(b) * a.I) + i);
  consumer_sync();
  for (int ks = 0; ks < nks; ++ks) {
    if (!take_stages<NS>(s.full, s.pending, st, ph, 1, &s.abort, a.dev_status)) return false;
    const uint8_t* wds = s.ring[st] + cg * 16;
    const int k0 = ks * kKSlice;
    switch (n) {
      case 1: dn_box<1>(wds, s.hs, k0, kl, a.I, ay); break;
      case 2: dn_box<2>(wds, s.hs, k0, kl, a.I, ay); break;
      case 3: dn_box<3>(wds, s.hs, k0, kl, a.I, ay); break;
      default: dn_box<4>(wds, s.hs, k0, kl, a.I, ay); break;
    }
    release_stage(&s.empty[st]);
    if (++st == NS) { st = 0; ph ^= 1u; }
  }
#pragma unroll
  for (int r = 0; r < kRG; ++r) {
    if (r < n) {
      warp_rows_sum(ay[r]);
      if (lane < kCG) {
        float4* dy = reinterpret_cast<float4*>(&s.u.red[r][w][0][cg * 8]);
        dy[0] = make_float4(ay[r][0], ay[r][1], ay[r][2], ay[r][3]);
        dy[1] = make_float4(ay[r][4], ay[r][5], ay[r][6], ay[r][7]);
      }
    }
  }
  consumer_sync();
  const int r = tid / (kCols / 2), c2 = (tid % (kCols / 2)) * 2;
  if (r < n) {
    float v[2] = {0.f, 0.f};
#pragma unroll
    for (int ww = 0; ww < kConsumers / 32; ++ww) {
      v[0] += s.u.red[r][ww][0][c2];
      v[1] += s.u.red[r][ww][0][c2 + 1];
    }
    *reinterpret_cast<uint32_t*>(a.y + static_cast<int64_t>(b + r) * a.d + col0 + c2) =
        pack_bf16x2(v[0], v[1]);
  }
  return true;
}

// ---- consumers: take the units in the ring's order ------------------------------
template <int VPL, bool GROUPED>
__device__ void consumer(const DecodeArgs& a, DecodeSmem<VPL, GROUPED>& s, int n_ci, int n_cd,
                         int n_gu, int nsplit) {
  int st = 0, sig = 0;
  uint32_t ph = 0, sph = 0;
  for (;;) {
    // the unit of the next box: thread 0 looks, the others follow
    if (threadIdx.x == 0) {
      int code = -1;
      if (!*reinterpret_cast<volatile int*>(&s.abort) &&
          wait_bounded(smem_u32(&s.full[st]), ph, &s.abort, a.dev_status))
        code = s.stage_unit[st];
      s.cur = code;
    }
    consumer_sync();
    const int u = s.cur;
    consumer_sync();  // every consumer has read s.cur before thread 0 writes it again
    bool ok = u >= 0;
    if (ok) {
      const Unit un = unit_of(u, n_gu, n_ci, n_cd, nsplit);
      ok = un.gu ? gate_up_unit(a, s, un, n_ci, nsplit, st, ph) : down_unit(a, s, un, st, ph);
    }
    // the finished unit, or the end (-1), to the signal warp
    if (!hand_over(a, s, ok ? u : -1, sig, sph) || !ok) return;
  }
}

// ---- signal warp: publishes finished units and finishes the cut ones ----------
// Uncut gate/up unit: one more complete column block of its row group's H.  Cut
// gate/up unit: the part that completes its (row group, column block) sums the
// parts' partial G and U in part order, writes H and counts the column block.
// Down unit: one more row group of its column block of y; the unit that completes
// the column block combines it for every token, in slot order in fp32 like
// moe_combine (padding slots of a bucket get zeros).  Every increment releases
// the writes before it (the consumers' writes are ordered before the hand-over).
template <int VPL, bool GROUPED>
__device__ void signaller(const DecodeArgs& a, DecodeSmem<VPL, GROUPED>& s, int n_ci, int n_cd,
                          int n_gu, int nsplit, int valid) {
  const int lane = threadIdx.x & 31;
  const CtrLayout L{n_ci, n_cd};
  int sig = 0;
  uint32_t sph = 0;
  for (;;) {
    int u = -1;
    if (lane == 0) {
      if (wait_bounded(smem_u32(&s.sig_full[sig]), sph, &s.abort, a.dev_status))
        u = s.sig_unit[sig];
    }
    u = __shfl_sync(0xFFFFFFFFu, u, 0);
    if (u < 0) return;
    const Unit un = unit_of(u, n_gu, n_ci, n_cd, nsplit);
    bool last = false;
    if (lane == 0) {
      if (un.gu && nsplit == 1) {
        add_release(a.ctr + CtrLayout::h_ready() + un.q, 1u);
      } else {
        const uint32_t target = un.gu ? static_cast<uint32_t>(nsplit - 1)
                                      : static_cast<uint32_t>(s.n_rg - 1);
        uint32_t* c = un.gu ? a.ctr + L.gu_fin() + un.q * n_ci + un.cb : a.ctr + L.y_ready() + un.cb;
        last = add_release(c, 1u) == target;
        if (last) fence_acquire();
      }
    }
    last = __shfl_sync(0xFFFFFFFFu, last ? 1 : 0, 0) != 0;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.sig_empty[sig]));
    if (++sig == kSigSlots) { sig = 0; sph ^= 1u; }
    if (!last) continue;
    const int col0 = un.cb * kCols;
    if (un.gu) {
      // H of this (row group, column block): lane -> column
      const int b = s.rg_b[un.q], n = s.rg_n[un.q];
      const float* pp = a.part + static_cast<int64_t>(un.q * n_ci + un.cb) * nsplit * kPartFloats;
      for (int i = lane; i < n * kCols; i += 32) {
        const int r = i / kCols, c = i % kCols;
        float g = 0.f, uu = 0.f;
        for (int p = 0; p < nsplit; ++p) {
          g += __ldcg(pp + p * kPartFloats + (r * 2 + 0) * kCols + c);
          uu += __ldcg(pp + p * kPartFloats + (r * 2 + 1) * kCols + c);
        }
        const float hv = __fdividef(g, 1.0f + __expf(-g)) * uu;
        const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
        a.h[static_cast<int64_t>(b + r) * a.I + col0 + c] = *reinterpret_cast<const uint16_t*>(&hb);
      }
      __syncwarp();
      if (lane == 0) add_release(a.ctr + CtrLayout::h_ready() + un.q, 1u);
      continue;
    }
    for (int q2 = lane; q2 < a.T * (kCols / 2); q2 += 32) {
      const int t = q2 / (kCols / 2), c2 = (q2 % (kCols / 2)) * 2;
      float acc[2] = {0.f, 0.f};
      if (t < valid) {
        for (int j = 0; j < a.k; ++j) {
          const int row = s.r2row[t * a.k + j];
          if (row < 0) continue;
          const uint32_t yv = __ldcg(reinterpret_cast<const unsigned int*>(
              a.y + static_cast<int64_t>(row) * a.d + col0 + c2));
          const float g = s.gates[t * a.k + j];
          acc[0] = fmaf(g, __uint_as_float(yv << 16), acc[0]);
          acc[1] = fmaf(g, __uint_as_float(yv & 0xFFFF0000u), acc[1]);
        }
      }
      *reinterpret_cast<float2*>(a.out + static_cast<int64_t>(t) * a.d + col0 + c2) =
          make_float2(acc[0], acc[1]);
    }
  }
}

template <int VPL, bool GROUPED, bool VEC>
__global__ void __launch_bounds__(kDecThreads, 1)
decode_kernel(DecodeArgs a, const __grid_constant__ DecodeMaps maps) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto& s = *reinterpret_cast<DecodeSmem<VPL, GROUPED>*>(smem_raw);
  constexpr int NS = DecodeSmem<VPL, GROUPED>::kStages;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == kConsumers) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&s.full[i]), 1);
      mbar_init(smem_u32(&s.empty[i]), kConsumers / 32);
      s.pending[i] = 0;
    }
    for (int i = 0; i < kSigSlots; ++i) {
      mbar_init(smem_u32(&s.sig_full[i]), 1);
      mbar_init(smem_u32(&s.sig_empty[i]), 1);
    }
    s.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.wg)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.wu)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.wd)) : "memory");
  }
  pdl_wait();
  // the first unit is claimed now, its latency hidden behind the prologue
  if (tid == kConsumers) s.first_unit = static_cast<int>(atomicAdd(a.ctr + CtrLayout::claim(), 1u));
  const int valid = a.valid != nullptr ? min(max(__ldg(a.valid), 0), a.T) : a.T;
  decode_prologue<VPL, GROUPED, VEC>(a, s, valid);
  __syncthreads();
  const int n_ci = a.I / kCols, n_cd = a.d / kCols;
  const CtrLayout L{n_ci, n_cd};
  const int n_rg = s.n_rg;
  // cut the gate/up units along d while they are too few to give every SM two
  int nsplit = 1;
  const int nks_d = n_slices(a.d);
  while (nsplit < kMaxSplit && n_rg * n_ci <= kSplitBlocks &&
         n_rg * n_ci * nsplit < 2 * static_cast<int>(gridDim.x) && nks_d % (2 * nsplit) == 0)
    nsplit *= 2;
  const int n_gu = n_rg * n_ci * nsplit, n_all = n_gu + n_rg * n_cd;
  // no live route: the output is all zeros (no combine runs)
  if (n_rg == 0 && blockIdx.x == 0) {
    for (int i = tid; i < a.T * a.d; i += kDecThreads) a.out[i] = 0.f;
  }
  if (warp == kProducerWarp) producer(a, maps, s, n_ci, n_cd, n_gu, n_all, nsplit);
  else if (warp == kSignalWarp) signaller(a, s, n_ci, n_cd, n_gu, nsplit, valid);
  else consumer(a, s, n_ci, n_cd, n_gu, nsplit);
  __syncthreads();
  // after an abort, let the copies already issued land before the CTA exits
  if (s.abort && tid == kConsumers) {
    for (int i = 0; i < NS; ++i)
      if (s.pending[i]) wait_drain(smem_u32(&s.full[i]), static_cast<uint32_t>(s.pending[i] - 1));
  }
  pdl_trigger();
  // the last CTA to finish leaves the counters zero for the next call
  if (tid == 0) {
    __threadfence();
    s.flag = atomicAdd(a.ctr + CtrLayout::done(), 1u) == gridDim.x - 1;
    if (s.flag) __threadfence();
  }
  __syncthreads();
  if (s.flag) {
    for (int i = tid; i < L.words(); i += kDecThreads) a.ctr[i] = 0u;
  }
}

// 2-D view [rows, cols] of a bf16 tensor with 256 x 64 boxes, no swizzle.
bool decode_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {kCols, kKSlice};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded maps of one (W_gate, W_up, W_down, E, d, I), kept in a small cache (an
// encoding depends only on those values).
bool decode_maps(DecodeMaps* out, const void* wg, const void* wu, const void* wd, int E, int d,
                 int I) {
  struct Entry {
    const void *wg, *wu, *wd;
    int E, d, I;
    DecodeMaps maps;
  };
  constexpr int kCache = 16;
  static Entry cache[kCache];
  static int used = 0, next = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i) {
    const Entry& e = cache[i];
    if (e.wg == wg && e.wu == wu && e.wd == wd && e.E == E && e.d == d && e.I == I) {
      *out = e.maps;
      return true;
    }
  }
  DecodeMaps mp;
  if (!decode_map(&mp.wg, wg, static_cast<uint64_t>(E) * d, I) ||
      !decode_map(&mp.wu, wu, static_cast<uint64_t>(E) * d, I) ||
      !decode_map(&mp.wd, wd, static_cast<uint64_t>(E) * I, d))
    return false;
  cache[next] = Entry{wg, wu, wd, E, d, I, mp};
  next = (next + 1) % kCache;
  if (used < kCache) ++used;
  *out = mp;
  return true;
}

template <int VPL, bool GROUPED, bool VEC>
moe_status launch_decode(const DecodeArgs& a, const DecodeMaps& maps, cudaStream_t st) {
  auto kern = decode_kernel<VPL, GROUPED, VEC>;
  constexpr size_t smem = sizeof(DecodeSmem<VPL, GROUPED>);
  static_assert(smem <= 227 * 1024, "decode kernel shared memory");
  constexpr int kMaxDev = 64;
  static std::atomic<int> ready[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MOE_ERR_CUDA;
  if (!ready[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
    ready[dev].store(1, std::memory_order_relaxed);
  }
  // one CTA per SM: every CTA is resident at once
  launch(kern, dim3(sm_count()), dim3(kDecThreads), smem, st, a, maps);
  return launch_status();
}

}  // namespace
}  // namespace moe

using namespace moe;

static bool decode_shape_ok(int32_t T, int32_t d, int32_t E, int32_t k, int32_t I) {
  return T >= 1 && T <= kDecMaxT && k >= 1 && k <= 16 && T * k <= kDecMaxRoutes && E >= 1 &&
         E <= kDecMaxE && k <= E && d >= 64 && d % 64 == 0 && I >= 64 && I % 64 == 0 &&
         I <= kDecMaxI && T * d <= kDecMaxTd &&
         static_cast<int64_t>(E) * (d > I ? d : I) < (1ll << 31);
}

MOE_API size_t moe_decode_workspace_size(int32_t T, int32_t d, int32_t E, int32_t k, int32_t I) {
  if (!decode_shape_ok(T, d, E, k, I)) return 0;
  const CtrLayout L{I / kCols, d / kCols};
  return ctr_bytes(L) + static_cast<size_t>(kSplitBlocks) * kMaxSplit * kPartFloats * 4;
}

MOE_API moe_status moe_decode_layer(const moe_route_params* p, int32_t d, int32_t I,
                                    int32_t capacity, const int32_t* valid_tokens,
                                    const float* logits, const float* sel_bias,
                                    const moe_bf16* x, const moe_bf16* w_gate,
                                    const moe_bf16* w_up, const moe_bf16* w_down,
                                    int32_t* topk_ids, float* gates, int32_t* counts,
                                    int32_t* offsets, int32_t* row_to_route,
                                    int32_t* route_to_row, int32_t* n_dropped, moe_bf16* x_perm,
                                    moe_bf16* h, moe_bf16* y, float* out, void* ws,
                                    size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream) {
  if (p == nullptr || logits == nullptr || x == nullptr || w_gate == nullptr ||
      w_up == nullptr || w_down == nullptr || topk_ids == nullptr || gates == nullptr ||
      counts == nullptr || offsets == nullptr || row_to_route == nullptr ||
      route_to_row == nullptr || n_dropped == nullptr || h == nullptr || y == nullptr ||
      out == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  const int32_t T = p->T, E = p->E, k = p->k;
  if (T < 1 || E <= 0 || k <= 0 || k > E || d <= 0 || I <= 0 || capacity < -1)
    return MOE_ERR_INVALID_ARG;
  if (!decode_shape_ok(T, d, E, k, I)) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(h) || !aligned16(y) || !aligned16(out) || !aligned16(ws) ||
      (x_perm != nullptr && !aligned16(x_perm)))
    return MOE_ERR_UNSUPPORTED;
  if (ws_bytes < moe_decode_workspace_size(T, d, E, k, I)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  int vpl = static_cast<int>(ceil_div(E, 32));
  vpl = vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : vpl <= 12 ? 12 : 16;
  bool grouped = false;
  if (p->score_fn == MOE_SCORE_SOFTMAX) {
    if (sel_bias != nullptr) return MOE_ERR_INVALID_ARG;
  } else if (p->score_fn == MOE_SCORE_SIGMOID_GROUP) {
    if (p->n_group <= 0 || p->topk_group <= 0 || p->topk_group > p->n_group ||
        E % p->n_group != 0)
      return MOE_ERR_INVALID_ARG;
    if (p->n_group > 32 || E / p->n_group < 2 || p->topk_group * (E / p->n_group) < k)
      return MOE_ERR_UNSUPPORTED;
    const int gs = E / p->n_group;
    if (gs % vpl != 0) return MOE_ERR_UNSUPPORTED;
    const int lpg = gs / vpl;
    if (lpg > 32 || (lpg & (lpg - 1)) != 0) return MOE_ERR_UNSUPPORTED;
    grouped = true;
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  DecodeMaps maps;
  if (!decode_maps(&maps, w_gate, w_up, w_down, E, d, I)) return MOE_ERR_CUDA;
  const CtrLayout L{I / kCols, d / kCols};
  DecodeArgs a{T, E, k, d, I, capacity, p->n_group, p->topk_group, p->route_scale,
               valid_tokens, logits, sel_bias, x, topk_ids, gates, counts, offsets,
               row_to_route, route_to_row, n_dropped, x_perm, h, y, out,
               static_cast<uint32_t*>(ws),
               reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ctr_bytes(L)), dev_status};
  const bool vec = vpl % 4 == 0 && E % 4 == 0 && aligned16(logits);
  const cudaStream_t st = as_cuda(stream);
#define MOE_DEC(V, G)                                                                  \
  return vec ? launch_decode<V, G, true>(a, maps, st) : launch_decode<V, G, false>(a, maps, st)
#define MOE_DEC_SCALAR(V, G) return launch_decode<V, G, false>(a, maps, st)
  if (grouped) {
    switch (vpl) {
      case 1: MOE_DEC_SCALAR(1, true);
      case 2: MOE_DEC_SCALAR(2, true);
      case 4: MOE_DEC(4, true);
      case 8: MOE_DEC(8, true);
      case 12: MOE_DEC(12, true);
      default: MOE_DEC(16, true);
    }
  }
  switch (vpl) {
    case 1: MOE_DEC_SCALAR(1, false);
    case 2: MOE_DEC_SCALAR(2, false);
    case 4: MOE_DEC(4, false);
    case 8: MOE_DEC(8, false);
    case 12: MOE_DEC(12, false);
    default: MOE_DEC(16, false);
  }
#undef MOE_DEC
#undef MOE_DEC_SCALAR
}
