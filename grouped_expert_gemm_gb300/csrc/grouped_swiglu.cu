// Grouped SwiGLU expert GEMM over ragged row segments on the 5th-generation
// tensor cores (tcgen05.mma, fp32 accumulators in tensor memory, operands
// staged by TMA with 128-byte swizzle).
//
// [M6.6] 0x04A "The Frozen Six-Segment Input": E(X) = (SiLU(X Wg) * (X Wu)) W2,
// F = 6 n d d_ff.  0x04C "Variable Grouped GEMM": one launch, exact row count
// per problem (no capacity padding reaches the output), a per-problem
// descriptor read on the device.
//
// Two persistent passes:
//   gate/up (SWIGLU): per tile, one MMA chain over N = [BN gate | BN up]
//     columns computes [G | U] = X [Wg | Wu] into tensor memory; the epilogue
//     writes H = bf16(SiLU(G) * U).
//   down:             per tile, Y = bf16(H Wd).
//
// Two kernel shapes share the scheduling and the epilogue:
//   * pair kernel (cta_group::2): a cluster of two CTAs on an SM pair computes a
//     256-row tile with N = 256; each CTA stages its own 128 rows of A and half
//     of the 256 B columns (6 stages of 32 KB), the leader CTA issues
//     tcgen05.mma.cta_group::2 and multicasts the stage/accumulator commits to
//     both CTAs, and each CTA's epilogue drains its own 128 accumulator rows.
//     Per SM this moves a third less operand data from L2 than the single-CTA
//     shape and fetches each weight tile once per 256 rows.
//   * single-CTA kernel (cta_group::1): a 128-row tile with N = 64..256, 4
//     stages; used where the pair shape does not divide the problem.
//
// Roles inside a CTA (192 threads, one CTA per SM):
//   warp 0      TMA producer: A tile [128 x 64] (K-major) and B atoms
//               [64 (K) x 64 (N)] (N-major: the weights are stored [K, N]).
//   warp 1      allocates tensor memory; lane 0 issues tcgen05.mma and commits.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, SwiGLU or conversion,
//               bf16 stores of the rows that belong to the segment.
// Two accumulator buffers let the epilogue of tile i overlap the MMAs of tile i+1.
//
// Tiles are enumerated per segment (n-block outer, m-block inner) from the
// device-resident segment table, so no host synchronisation is needed and
// consecutive tiles on neighbouring SMs share the same weight columns in L2.
// Rows of a partial m-block that belong to the next segment (or lie past the
// end of the tensor, zero-filled by TMA) are computed but never stored.
//
// Every wait is bounded: after kWaitLimitNs without progress the CTA reports
// MOE_DEV_TIMEOUT, stops all roles, waits (bounded) for its own copies and
// MMAs in flight, frees its tensor memory and returns.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;          // rows per tile (MMA M)
constexpr int kBK = 64;           // K per stage: one 128-byte swizzle row of bf16
constexpr int kUmmaK = 16;        // K per tcgen05.mma (kind::f16)
constexpr int kThreads = 192;
constexpr int kMaxSeg = 1024;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s without progress = broken pipeline

constexpr int kABytes = kBM * kBK * 2;        // 16 KB
constexpr int kAtomBytes = kBK * 64 * 2;      // 8 KB: [64 K rows][64 N cols]

constexpr int kStagesPair = 6;
constexpr int kPairAtoms = 2;                     // B atoms per CTA in the pair kernel
constexpr int kPairStageBytes = kABytes + kPairAtoms * kAtomBytes;  // 32 KB
constexpr int kPairSmemBytes = 1024 + kStagesPair * kPairStageBytes + 256 + (3 * kMaxSeg + 16) * 4;

template <int N_ATOMS>
struct Geometry {
  static constexpr int kN = 64 * N_ATOMS;                  // MMA N
  static constexpr int kStageBytes = kABytes + N_ATOMS * kAtomBytes;
  // As many stages as fit the same ~192 KB: narrower tiles keep more loads in flight.
  static constexpr int kStages = N_ATOMS >= 4 ? 4 : (N_ATOMS == 2 ? 6 : 8);
  static constexpr int kTmemCols = 2 * kN;                 // two accumulator buffers
  static constexpr int kTmemAlloc = kTmemCols <= 32 ? 32 : kTmemCols <= 64 ? 64 : kTmemCols <= 128 ? 128 : kTmemCols <= 256 ? 256 : 512;
  static constexpr int kSmemBytes = 1024 /*align slack*/ + kStages * kStageBytes +
                                    (2 * kStages + 5) * 8 /*barriers*/ + (3 * kMaxSeg + 16) * 4;
};

struct GemmArgs {
  const int32_t* seg_begin;
  const int32_t* seg_count;
  int n_seg;
  int K;         // reduction width
  int N;         // output columns per segment
  int max_rows;
  uint16_t* out; // [max_rows, N] bf16 bits
  uint32_t* dev_status;
  int m_outer;   // tile order inside a segment: 0 = n-block outer, 1 = m-block outer
};

// ------------------------------ PTX wrappers -------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `parity` to complete.  Returns false when the
// CTA is aborting (another role gave up) or when this wait itself times out.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             uint32_t* dev_status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((i & 255u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      report(dev_status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
}

// Short bounded wait used only while tearing down after an abort.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > 100000000ull) return;  // 100 ms
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c_inner, int32_t c_outer) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c_inner), "r"(c_outer)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, A K-major,
// B N-major, M = m, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// ---- CTA-pair (cluster of two) forms ----

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of `local` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at the same offset in every CTA of `mask` once all
// prior tcgen05 operations of this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// TMA tile load into this CTA's shared memory whose completion is counted on an
// mbarrier that may live in the peer CTA (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c_inner,
                                                 int32_t c_outer) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c_inner), "r"(c_outer)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// Spin for about `ns` nanoseconds (drain window for copies whose completion
// lands on another CTA's barrier).
__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

// ------------------------------ scheduling ---------------------------------

struct Tile {
  int seg, row0, rows, n0;
};

// tile_start[q] = first tile of segment q (exclusive scan of its tile count).
// Inside a segment the tiles run n-block outer / m-block inner (neighbouring
// CTAs share one weight tile and walk the segment's rows), or, with m_outer,
// m-block outer / n-block inner (neighbouring CTAs share one block of rows and
// walk the expert's weight columns).  m-blocks have `bm` rows.
__device__ __forceinline__ Tile tile_of(int t, const int* tile_start, const int* s_begin,
                                        const int* s_count, int n_seg, int bm, int bn_out,
                                        int n_blocks, int m_outer) {
  int lo = 0, hi = n_seg - 1;
  while (lo < hi) {  // last q with tile_start[q] <= t
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int q = lo;
  const int local = t - tile_start[q];
  const int m_blocks = (s_count[q] + bm - 1) / bm;
  const int nb = m_outer ? local % n_blocks : local / m_blocks;
  const int mb = m_outer ? local / n_blocks : local % m_blocks;
  Tile tl;
  tl.seg = q;
  tl.row0 = s_begin[q] + mb * bm;
  tl.rows = min(bm, s_count[q] - mb * bm);
  tl.n0 = nb * bn_out;
  return tl;
}

// Segment table in shared memory, built by threads 64..191 (each owns a run of
// up to 8 consecutive segments): bad segments are reported and treated as
// empty; s_tile_start[q] is the exclusive scan of the tile counts and
// s_tile_start[n_seg] the total.
__device__ __forceinline__ void build_segment_table(const GemmArgs& args, int bm, int n_blocks,
                                                    int* s_begin, int* s_count, int* s_tile_start,
                                                    int* warp_tot) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x - 64;
  const int n_seg = args.n_seg;
  const int per = (n_seg + 127) / 128;
  const int q0 = tid * per, q1 = min(n_seg, q0 + per);
  int local = 0;
  for (int q = q0; q < q1; ++q) {
    int b = __ldg(args.seg_begin + q), c = __ldg(args.seg_count + q);
    if (c < 0 || b < 0 || static_cast<int64_t>(b) + c > args.max_rows) {
      if (c != 0) report(args.dev_status, MOE_DEV_BAD_ROW);
      b = 0;
      c = 0;
    }
    s_begin[q] = b;
    s_count[q] = c;
    local += ((c + bm - 1) / bm) * n_blocks;
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp - 2] = incl;
  asm volatile("bar.sync 1, 128;" ::: "memory");
  int before = 0;
  for (int w = 2; w < warp; ++w) before += warp_tot[w - 2];
  const int total_all = warp_tot[0] + warp_tot[1] + warp_tot[2] + warp_tot[3];
  int run = before + incl - local;
  for (int q = q0; q < q1; ++q) {
    s_tile_start[q] = run;
    run += ((s_count[q] + bm - 1) / bm) * n_blocks;
  }
  if (tid == 127) s_tile_start[n_seg] = total_all;
}

// Epilogue of one tile for the calling thread's accumulator row: `taddr`
// addresses this warp's TMEM lane quadrant at the tile's first column.  BN_OUT
// output columns; for SWIGLU the gate accumulators are columns [0, BN_OUT) and
// the up accumulators [BN_OUT, 2*BN_OUT).  All lanes execute the tensor-memory
// loads (.sync.aligned); only live rows compute and store.
template <int BN_OUT, bool SWIGLU>
__device__ __forceinline__ void epilogue_row(uint32_t taddr, bool live, uint16_t* orow) {
  if constexpr (SWIGLU) {
#pragma unroll 1
    for (int c = 0; c < BN_OUT; c += 32) {
      uint32_t g[32], u[32];
      tmem_ld32(taddr + c, g);
      tmem_ld32(taddr + BN_OUT + c, u);
      tmem_ld_wait();
      if (live) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float h2[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float gv = __uint_as_float(g[2 * i + h]);
            const float uv = __uint_as_float(u[2 * i + h]);
            // SiLU(g) * u with the fast exp and division: measured 6 % faster on the
            // weight-streaming decode shape than expf + IEEE division, and H still
            // rounds to the same bf16 value in all but ~0.2 % of elements.
            h2[h] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
          }
          pk[i] = pack_bf16x2(h2[0], h2[1]);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < BN_OUT; c += 32) {
      uint32_t v[32];
      tmem_ld32(taddr + c, v);
      tmem_ld_wait();
      if (live) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
  }
}

// Shared-memory carve-up common to both kernels, after the stage buffers.
struct Smem {
  uint64_t* bars;
  volatile int* abort_flag;
  uint32_t* tmem_slot;
  int* warp_tot;
  int* s_tile_start;
  int* s_begin;
  int* s_count;
};

__device__ __forceinline__ Smem carve(uint8_t* after_stages, int n_bars) {
  Smem m;
  m.bars = reinterpret_cast<uint64_t*>(after_stages);
  int* misc = reinterpret_cast<int*>(m.bars + n_bars);
  m.abort_flag = misc;
  m.tmem_slot = reinterpret_cast<uint32_t*>(misc + 1);
  m.warp_tot = misc + 4;
  m.s_tile_start = misc + 8;
  m.s_begin = m.s_tile_start + kMaxSeg + 1;
  m.s_count = m.s_begin + kMaxSeg;
  return m;
}

// ------------------------- single-CTA kernel --------------------------------

template <int N_ATOMS, bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b0,
                    const __grid_constant__ CUtensorMap tmap_b1, const GemmArgs args) {
  using G = Geometry<N_ATOMS>;
  constexpr int kStages = G::kStages;
  constexpr int kN = G::kN;
  constexpr int kBnOut = SWIGLU ? kN / 2 : kN;  // output columns per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // bars: full[S], empty[S], tmem_full[2], tmem_empty[2], drain
  const Smem sm = carve(stage_base + kStages * G::kStageBytes, 2 * kStages + 5);
  uint64_t* bars = sm.bars;
  volatile int* abort_flag = sm.abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_seg = args.n_seg;
  const int n_blocks = args.N / kBnOut;
  const int k_steps = args.K / kBK;

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };
  auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * kStages + b); };
  auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * kStages + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * kStages + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b0)) : "memory");
    if (SWIGLU)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b1)) : "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(sm.tmem_slot), G::kTmemAlloc);
  pdl_wait();  // everything above is local; global data only from here on
  if (threadIdx.x >= 64)
    build_segment_table(args, kBM, n_blocks, sm.s_begin, sm.s_count, sm.s_tile_start, sm.warp_tot);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;
  const int total_tiles = sm.s_tile_start[n_seg];

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const Tile tl = tile_of(t, sm.s_tile_start, sm.s_begin, sm.s_count, n_seg, kBM, kBnOut, n_blocks,
                              args.m_outer);
        const int b_row0 = tl.seg * args.K;
        for (int ks = 0; ks < k_steps; ++ks) {
          if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, args.dev_status)) { ok = false; break; }
          const uint32_t st = smem_u32(stage_base + s * G::kStageBytes);
          mbar_arrive_expect_tx(full_bar(s), G::kStageBytes);
          tma_load_2d(st, &tmap_a, full_bar(s), ks * kBK, tl.row0);
#pragma unroll
          for (int a = 0; a < N_ATOMS; ++a) {
            const uint32_t dst = st + kABytes + a * kAtomBytes;
            if constexpr (SWIGLU) {
              const int half = N_ATOMS / 2;
              const CUtensorMap* m = a < half ? &tmap_b0 : &tmap_b1;
              const int col = tl.n0 + (a % half) * 64;
              tma_load_2d(dst, m, full_bar(s), col, b_row0 + ks * kBK);
            } else {
              tma_load_2d(dst, &tmap_b0, full_bar(s), tl.n0 + a * 64, b_row0 + ks * kBK);
            }
          }
          if (++s == kStages) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {
        // Let the copies this thread issued land before the CTA goes away: the
        // last kStages fills precede (s, ph) in issue order.
        int ss = s;
        uint32_t pp = ph;
        for (int i = 0; i < kStages; ++i) {
          if (--ss < 0) { ss = kStages - 1; pp ^= 1u; }
          wait_drain(full_bar(ss), pp);
        }
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, kN);
      int s = 0;
      uint32_t ph = 0;
      int buf = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      bool issued_any = false;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        if (!wait_bounded(tempty_bar(buf), acc_ph ^ 1u, abort_flag, args.dev_status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kN);
        for (int ks = 0; ks < k_steps; ++ks) {
          if (!wait_bounded(full_bar(s), ph, abort_flag, args.dev_status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stage_base + s * G::kStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
            // A: K-major, advance 16 elements = 32 bytes inside the swizzle row.
            const uint64_t ad = smem_desc_sw128(a_addr + kk * kUmmaK * 2, 16, 1024);
            // B: N-major, advance 16 K rows = 2048 bytes; atoms of 64 columns
            // are kAtomBytes apart (LBO), 8-row K groups 1024 bytes apart (SBO).
            const uint64_t bd = smem_desc_sw128(b_addr + kk * kUmmaK * 128, kAtomBytes, 1024);
            mma_bf16(d_tmem, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
          }
          issued_any = true;
          mma_commit(empty_bar(s));  // frees this stage once its MMAs have read it
          if (++s == kStages) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(tfull_bar(buf));  // accumulator ready for the epilogue
        if (++buf == 2) { buf = 0; acc_ph ^= 1u; }
      }
      if (!ok && issued_any) {
        // All MMAs issued so far must finish before tensor memory is freed.
        mma_commit(drain_bar);
        wait_drain(drain_bar, 0);
      }
    }
  } else {
    // ======================= epilogue (warps 2..5) =======================
    const int quad = warp & 3;            // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;       // accumulator row owned by this thread
    int buf = 0;
    uint32_t acc_ph = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
      const Tile tl = tile_of(t, sm.s_tile_start, sm.s_begin, sm.s_count, n_seg, kBM, kBnOut, n_blocks,
                              args.m_outer);
      if (!wait_bounded(tfull_bar(buf), acc_ph, abort_flag, args.dev_status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(buf * kN);
      const bool live = r < tl.rows;
      uint16_t* orow = args.out + static_cast<int64_t>(tl.row0 + (live ? r : 0)) * args.N + tl.n0;
      epilogue_row<kBnOut, SWIGLU>(taddr, live, orow);
      tc_fence_before();
      mbar_arrive(tempty_bar(buf));
      if (++buf == 2) { buf = 0; acc_ph ^= 1u; }
    }
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, G::kTmemAlloc);
  }
  pdl_trigger();
}

// ------------------------- CTA-pair kernel ----------------------------------
//
// A cluster of two CTAs (ranks 0 and 1) computes a tile of 2*kBM = 256 rows and
// N = 256 accumulator columns.  Rank r stages rows [row0 + 128 r, +128) of A and
// the r-th half (128 columns) of the B tile in its own shared memory; for the
// gate/up pass rank 0 holds the 128 gate columns and rank 1 the 128 up columns,
// so the accumulator of either rank is [G | U] for its own 128 rows.  Barriers:
//   full[s]      leader only: the leader's expect_tx covers both ranks' bytes,
//                and each rank's TMA completes its bytes on the leader's barrier;
//   empty[s]     both ranks: the leader's commit is multicast to both;
//   tfull[b]     both ranks: multicast commit after a tile's last MMA;
//   tempty[b]    leader only: one arrival per epilogue warp of both ranks (8).
template <bool SWIGLU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b0,
                         const __grid_constant__ CUtensorMap tmap_b1, const GemmArgs args) {
  constexpr int kN = 2 * kPairAtoms * 64;        // 256 accumulator columns
  constexpr int kBnOut = SWIGLU ? kN / 2 : kN;   // output columns per tile
  constexpr int kPairBM = 2 * kBM;               // rows per tile
  constexpr int kTmemAlloc = 2 * kN;             // two accumulator buffers = 512
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Smem sm = carve(stage_base + kStagesPair * kPairStageBytes, 2 * kStagesPair + 5);
  uint64_t* bars = sm.bars;
  volatile int* abort_flag = sm.abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cid = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int n_seg = args.n_seg;
  const int n_blocks = args.N / kBnOut;
  const int k_steps = args.K / kBK;

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kStagesPair + s); };
  auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * kStagesPair + b); };
  auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * kStagesPair + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * kStagesPair + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesPair; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 8);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b0)) : "memory");
    if (SWIGLU)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b1)) : "memory");
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(sm.tmem_slot), kTmemAlloc);
  pdl_wait();  // everything above is local; global data only from here on
  if (threadIdx.x >= 64)
    build_segment_table(args, kPairBM, n_blocks, sm.s_begin, sm.s_count, sm.s_tile_start,
                        sm.warp_tot);
  // Both ranks' barriers are initialised and their tensor memory allocated
  // before any rank signals the other.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;
  const int total_tiles = sm.s_tile_start[n_seg];

  if (warp == 0) {
    // ======================= TMA producer (both ranks) =======================
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      bool issued_any = false;
      for (int t = cid; t < total_tiles && ok; t += n_clusters) {
        const Tile tl = tile_of(t, sm.s_tile_start, sm.s_begin, sm.s_count, n_seg, kPairBM, kBnOut,
                              n_blocks, args.m_outer);
        const int b_row0 = tl.seg * args.K;
        for (int ks = 0; ks < k_steps; ++ks) {
          if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, args.dev_status)) { ok = false; break; }
          const uint32_t full_leader = map_to_rank(full_bar(s), 0);
          if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * kPairStageBytes);
          const uint32_t st = smem_u32(stage_base + s * kPairStageBytes);
          tma_load_2d_pair(st, &tmap_a, full_leader, ks * kBK, tl.row0 + static_cast<int>(rank) * kBM);
#pragma unroll
          for (int a = 0; a < kPairAtoms; ++a) {
            const uint32_t dst = st + kABytes + a * kAtomBytes;
            if constexpr (SWIGLU) {
              tma_load_2d_pair(dst, leader ? &tmap_b0 : &tmap_b1, full_leader, tl.n0 + a * 64,
                               b_row0 + ks * kBK);
            } else {
              tma_load_2d_pair(dst, &tmap_b0, full_leader,
                               tl.n0 + static_cast<int>(rank) * (kPairAtoms * 64) + a * 64,
                               b_row0 + ks * kBK);
            }
          }
          issued_any = true;
          if (++s == kStagesPair) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok && issued_any) {
        if (leader) {
          int ss = s;
          uint32_t pp = ph;
          for (int i = 0; i < kStagesPair; ++i) {
            if (--ss < 0) { ss = kStagesPair - 1; pp ^= 1u; }
            wait_drain(full_bar(ss), pp);
          }
        } else {
          // This rank's completions land on the leader's barriers: give its
          // copies in flight a fixed window to land.
          spin_ns(2000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer (leader only) =======================
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_bf16(kPairBM, kN);
      int s = 0;
      uint32_t ph = 0;
      int buf = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      bool issued_any = false;
      for (int t = cid; t < total_tiles && ok; t += n_clusters) {
        if (!wait_bounded(tempty_bar(buf), acc_ph ^ 1u, abort_flag, args.dev_status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kN);
        for (int ks = 0; ks < k_steps; ++ks) {
          if (!wait_bounded(full_bar(s), ph, abort_flag, args.dev_status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stage_base + s * kPairStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
            const uint64_t ad = smem_desc_sw128(a_addr + kk * kUmmaK * 2, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b_addr + kk * kUmmaK * 128, kAtomBytes, 1024);
            mma_bf16_pair(d_tmem, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
          }
          issued_any = true;
          mma_commit_pair(empty_bar(s), 0x3);  // frees stage s in both ranks
          if (++s == kStagesPair) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit_pair(tfull_bar(buf), 0x3);  // both ranks' accumulators ready
        if (++buf == 2) { buf = 0; acc_ph ^= 1u; }
      }
      if (!ok && issued_any) {
        mma_commit_pair(drain_bar, 0x1);
        wait_drain(drain_bar, 0);
      }
    }
  } else {
    // ======================= epilogue (warps 2..5, both ranks) ===============
    const int quad = warp & 3;
    const int r = quad * 32 + lane;                        // row within this rank's half
    const int tile_r = static_cast<int>(rank) * kBM + r;   // row within the 256-row tile
    int buf = 0;
    uint32_t acc_ph = 0;
    for (int t = cid; t < total_tiles; t += n_clusters) {
      const Tile tl = tile_of(t, sm.s_tile_start, sm.s_begin, sm.s_count, n_seg, kPairBM, kBnOut,
                              n_blocks, args.m_outer);
      if (!wait_bounded(tfull_bar(buf), acc_ph, abort_flag, args.dev_status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(buf * kN);
      const bool live = tile_r < tl.rows;
      uint16_t* orow =
          args.out + static_cast<int64_t>(tl.row0 + (live ? tile_r : 0)) * args.N + tl.n0;
      epilogue_row<kBnOut, SWIGLU>(taddr, live, orow);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(buf), 0));
      if (++buf == 2) { buf = 0; acc_ph ^= 1u; }
    }
  }

  // ---- teardown: no rank leaves while the other may still touch its memory ----
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, kTmemAlloc);
  }
  pdl_trigger();
}

// ------------------------------ host side ----------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box [box_rows, 64], 128B swizzle.
// An encoded map depends only on (address, rows, cols, box rows), so encodings
// are kept in a small cache keyed by exactly those values: a hit is always a
// valid map, whatever the caller did with the memory in between.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  struct Entry {
    const void* base;
    uint64_t rows, cols;
    uint32_t box_rows;
    CUtensorMap map;
  };
  constexpr int kCache = 64;
  static Entry cache[kCache];
  static int used = 0, next = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i) {
      const Entry& e = cache[i];
      if (e.base == base && e.rows == rows && e.cols == cols && e.box_rows == box_rows) {
        *m = e.map;
        return true;
      }
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(mu);
  Entry& e = cache[next];
  e = Entry{base, rows, cols, box_rows, *m};
  next = (next + 1) % kCache;
  if (used < kCache) ++used;
  return true;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int N_ATOMS, bool SWIGLU>
moe_status launch_gemm(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                       const GemmArgs& args, cudaStream_t s) {
  using G = Geometry<N_ATOMS>;
  auto kern = grouped_gemm_kernel<N_ATOMS, SWIGLU>;
  // The shared-memory opt-in and the SM count are per device: set/read once.
  constexpr int kMaxDev = 64;
  static int sms[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MOE_ERR_CUDA;
  int n_sm;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (sms[dev] == 0) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               G::kSmemBytes) != cudaSuccess)
        return MOE_ERR_CUDA;
      sms[dev] = num_sms();
    }
    n_sm = sms[dev];
  }
  launch(kern, dim3(n_sm), dim3(kThreads), G::kSmemBytes, s, a, b0, b1, args);
  return launch_status();
}

// The pair kernel runs as many two-CTA clusters as can be resident at once
// (queried once per device), each looping over its share of the tiles.
template <bool SWIGLU>
moe_status launch_gemm_pair(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                            const GemmArgs& args, cudaStream_t s) {
  auto kern = grouped_gemm_pair_kernel<SWIGLU>;
  constexpr int kMaxDev = 64;
  static int grid[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MOE_ERR_CUDA;
  int g;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (grid[dev] == 0) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kPairSmemBytes) != cudaSuccess)
        return MOE_ERR_CUDA;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(num_sms() & ~1));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kPairSmemBytes;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0)
        clusters = num_sms() / 2;
      cudaGetLastError();
      grid[dev] = 2 * clusters;
    }
    g = grid[dev];
  }
  launch(kern, dim3(g), dim3(kThreads), kPairSmemBytes, s, a, b0, b1, args);
  return launch_status();
}

// The pair kernel stages 256 rows of A per tile.  When segments average fewer
// than 128 rows (decode-sized batches) most of those rows belong to other
// segments, and the single-CTA kernel, which stages half as many A rows for
// the same weight columns, streams the weights faster (measured: 117.5 vs
// 128.3 us for the gate/up pass at T=128, E=128, top-8).
// Tile order that keeps HBM re-reads down.  With n-block outer, a segment's
// rows of A are re-read once per n-block unless they stay in L2; with m-block
// outer, the expert's B columns are re-read once per m-block unless they stay in
// L2.  Rows-inner (n-block outer) is the default; m-block outer is chosen when
// an average segment of A is too large for L2 while one expert's B fits
// (e.g. 29 K rows x 3072 of A against 18.9 MB of gate+up weights).
int choose_m_outer(int32_t n_seg, int32_t max_rows, int32_t K, int64_t b_cols_per_seg) {
  constexpr int64_t kL2Budget = 48ll << 20;  // of the 129 MB L2, leaving room for concurrency
  const int64_t a_seg = static_cast<int64_t>(max_rows) / n_seg * K * 2;
  const int64_t b_seg = static_cast<int64_t>(K) * b_cols_per_seg * 2;
  return (a_seg > kL2Budget && b_seg <= kL2Budget) ? 1 : 0;
}

bool pair_shape(int32_t n_seg, int32_t max_rows) {
  return static_cast<int64_t>(max_rows) >= static_cast<int64_t>(kBM) * n_seg;
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API size_t moe_grouped_swiglu_workspace_size(int32_t max_rows, int32_t I) {
  if (max_rows <= 0 || I <= 0) return 256;
  return static_cast<size_t>(max_rows) * I * 2 + 256;
}

static moe_status check_common(int32_t n_seg, int32_t K, int32_t N, int32_t max_rows) {
  if (n_seg <= 0 || K <= 0 || N <= 0 || max_rows < 0) return MOE_ERR_INVALID_ARG;
  if (K % 64 != 0 || N % 64 != 0 || K > 65536 || N > 65536 || n_seg > kMaxSeg)
    return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(n_seg) * K >= (int64_t(1) << 31) ||
      static_cast<int64_t>(n_seg) * N >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

MOE_API moe_status moe_grouped_gate_up(int32_t n_seg, int32_t d, int32_t I, int32_t max_rows,
                                       const moe_bf16* x, const int32_t* seg_begin,
                                       const int32_t* seg_count, const moe_bf16* w_gate,
                                       const moe_bf16* w_up, moe_bf16* h, uint32_t* dev_status,
                                       moe_stream_t stream) {
  moe_status st = check_common(n_seg, d, I, max_rows);
  if (st != MOE_OK || max_rows == 0) return st;
  if (x == nullptr || seg_begin == nullptr || seg_count == nullptr || w_gate == nullptr ||
      w_up == nullptr || h == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(h) || !aligned16(w_gate) || !aligned16(w_up))
    return MOE_ERR_UNSUPPORTED;
  CUtensorMap m_x, m_wg, m_wu;
  if (!make_map(&m_x, x, max_rows, d, kBM) || !make_map(&m_wg, w_gate, int64_t(n_seg) * d, I, kBK) ||
      !make_map(&m_wu, w_up, int64_t(n_seg) * d, I, kBK))
    return MOE_ERR_CUDA;
  GemmArgs a{seg_begin, seg_count, n_seg, d, I, max_rows, reinterpret_cast<uint16_t*>(h),
             dev_status, choose_m_outer(n_seg, max_rows, d, 2 * static_cast<int64_t>(I))};
  cudaStream_t s = as_cuda(stream);
  if (I % 128 == 0) {
    return pair_shape(n_seg, max_rows) ? launch_gemm_pair<true>(m_x, m_wg, m_wu, a, s)
                                       : launch_gemm<4, true>(m_x, m_wg, m_wu, a, s);
  }
  return launch_gemm<2, true>(m_x, m_wg, m_wu, a, s);
}

MOE_API moe_status moe_grouped_down(int32_t n_seg, int32_t I, int32_t d, int32_t max_rows,
                                    const moe_bf16* h, const int32_t* seg_begin,
                                    const int32_t* seg_count, const moe_bf16* w_down, moe_bf16* y,
                                    uint32_t* dev_status, moe_stream_t stream) {
  moe_status st = check_common(n_seg, I, d, max_rows);
  if (st != MOE_OK || max_rows == 0) return st;
  if (h == nullptr || seg_begin == nullptr || seg_count == nullptr || w_down == nullptr ||
      y == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(y) || !aligned16(w_down)) return MOE_ERR_UNSUPPORTED;
  CUtensorMap m_h, m_wd;
  if (!make_map(&m_h, h, max_rows, I, kBM) || !make_map(&m_wd, w_down, int64_t(n_seg) * I, d, kBK))
    return MOE_ERR_CUDA;
  GemmArgs a{seg_begin, seg_count, n_seg, I, d, max_rows, reinterpret_cast<uint16_t*>(y),
             dev_status, choose_m_outer(n_seg, max_rows, I, d)};
  cudaStream_t s = as_cuda(stream);
  // The widest output tile the width allows (narrower tiles for one-token decode were
  // measured slower: the few tiles there are bound by pipeline latency, not SM count).
  if (d % 256 == 0) {
    return pair_shape(n_seg, max_rows) ? launch_gemm_pair<false>(m_h, m_wd, m_wd, a, s)
                                       : launch_gemm<4, false>(m_h, m_wd, m_wd, a, s);
  }
  if (d % 128 == 0) return launch_gemm<2, false>(m_h, m_wd, m_wd, a, s);
  return launch_gemm<1, false>(m_h, m_wd, m_wd, a, s);
}

MOE_API moe_status moe_grouped_swiglu(int32_t n_seg, int32_t d, int32_t I, int32_t max_rows,
                                      const moe_bf16* x, const int32_t* seg_begin,
                                      const int32_t* seg_count, const moe_bf16* w_gate,
                                      const moe_bf16* w_up, const moe_bf16* w_down, moe_bf16* y,
                                      void* ws, size_t ws_bytes, uint32_t* dev_status,
                                      moe_stream_t stream) {
  moe_status st = check_common(n_seg, d, I, max_rows);
  if (st != MOE_OK || max_rows == 0) return st;
  if (x == nullptr || seg_begin == nullptr || seg_count == nullptr || w_gate == nullptr ||
      w_up == nullptr || w_down == nullptr || y == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(ws) || !aligned16(w_gate) ||
      !aligned16(w_up) || !aligned16(w_down))
    return MOE_ERR_UNSUPPORTED;
  if (ws_bytes < moe_grouped_swiglu_workspace_size(max_rows, I)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe_bf16* h = static_cast<moe_bf16*>(ws);
  st = moe_grouped_gate_up(n_seg, d, I, max_rows, x, seg_begin, seg_count, w_gate, w_up, h,
                           dev_status, stream);
  if (st != MOE_OK) return st;
  return moe_grouped_down(n_seg, I, d, max_rows, h, seg_begin, seg_count, w_down, y, dev_status,
                          stream);
}
