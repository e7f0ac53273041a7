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
// FP8 dispatch payload ([M6.6] 0x0AB-0x0AC): with an E4M3 A operand (gate/up
// pass only) TMA stages the [128 x 64] E4M3 tile (8 KB instead of 16 KB) and
// four more warps (6..9, 320 threads) dequantize it with each row's fp32 scale
// into the bf16 A tile the MMA reads, so the expert input never exists as bf16
// in HBM.
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

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "tma.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;          // rows per tile (MMA M)
constexpr int kBK = 64;           // K per stage: one 128-byte swizzle row of bf16
constexpr int kUmmaK = 16;        // K per tcgen05.mma (kind::f16)
constexpr int kMaxSeg = 1024;

constexpr int kABytes = kBM * kBK * 2;        // 16 KB
constexpr int kAtomBytes = kBK * 64 * 2;      // 8 KB: [64 K rows][64 N cols]
constexpr int kRawBytes = kBM * kBK;          // 8 KB: [128 rows][64 E4M3 codes]

constexpr int kPairAtoms = 2;                     // B atoms per CTA in the pair kernel

// Stage (TMA slot) layout.  bf16 A operand: [A tile 16 KB][N_ATOMS B atoms].
// E4M3 A operand: [N_ATOMS B atoms][E4M3 A tile 8 KB]; the converter warps write
// the bf16 A operand into tensor memory -- kASlots slots of 32 columns after the
// accumulators -- where the MMA reads it, so it costs no shared-memory traffic.
// Where the A slots do not fit beside two accumulator buffers (N = 256) there is
// one.  With an E4M3 operand both ring sizes are even: stage n, TMA slot
// n % kStages and A slot n % kASlots then always belong to converter group
// n % 2, so every barrier a converter group waits on is one whose phases only
// that group observes, in order (a parity wait cannot tell a phase from the one
// two phases later).
constexpr int kTmemCols = 512;
constexpr int kASlotCols = kBK / 2;  // 64 bf16 of a row = 32 columns

// SMALLA (bf16 A, boxes of at most 32 rows): the A slot holds only the 32 rows
// TMA stages (4 KB), so more stages fit; the MMA still reads 128 rows from the
// slot's start, the rows past 32 falling on the same stage's B atoms -- finite
// data whose accumulator rows are never stored.
constexpr int kSmallABytes = 32 * kBK * 2;  // 4 KB
constexpr int kFixedSmem = 1024 + (3 * kMaxSeg + 16) * 4 + 64 * 8;  // alignment, tables, barriers

// KS = K per stage.  Deep stages (KS = 128, small-A bf16 only) stage each B atom as
// one [128 K x 64 N] box and the A rows as two [rows x 64 K] boxes: half as many
// TMA boxes per byte of weights, which streams them faster when a pass has few
// tiles (one-token decode: 44 -> 67 GB/s per SM in a producer-only measurement).
template <int N_ATOMS, bool FP8A = false, bool SMALLA = false, int KS = kBK>
struct Geometry {
  static constexpr int kN = 64 * N_ATOMS;                  // MMA N
  static constexpr int kAtom = KS * 64 * 2;                // one B atom box [KS x 64]
  static constexpr int kABoxes = KS / kBK;                 // A boxes per stage
  static constexpr int kABoxSlot = SMALLA ? kSmallABytes : kABytes;  // bytes per A box slot
  static constexpr int kASlotBytes = kABoxSlot * kABoxes;
  static constexpr int kBOff = FP8A ? 0 : kASlotBytes;     // B atoms in a TMA slot
  static constexpr int kRawOff = N_ATOMS * kAtom;          // E4M3 tile in a TMA slot
  static constexpr int kStageBytes = N_ATOMS * kAtom + (FP8A ? kRawBytes : kASlotBytes);
  // As many stages as fit the shared memory: narrower tiles keep more loads in flight.
  static constexpr int kSmallAStages = (227 * 1024 - kFixedSmem) / kStageBytes;
  static constexpr int kStages = SMALLA ? (kSmallAStages > 12 ? 12 : kSmallAStages)
                                 : FP8A ? (N_ATOMS >= 4 ? 4 : 8)
                                        : (N_ATOMS >= 4 ? 4 : (N_ATOMS == 2 ? 6 : 8));
  static constexpr int kASlots = FP8A ? 8 : 0;
  static constexpr int kAccBufs = 2 * kN + kASlots * kASlotCols <= kTmemCols ? 2 : 1;
  static constexpr int kACol = kAccBufs * kN;              // first column of the A slots
  static constexpr int kTmemUsed = kACol + kASlots * kASlotCols;
  static constexpr int kTmemAlloc = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128 : kTmemUsed <= 256 ? 256 : 512;
  // full[S], empty[S], tfull[2], tempty[2], drain, (FP8A) afull[A], aempty[A]
  static constexpr int kBars = 2 * kStages + 5 + 2 * kASlots;
  static constexpr int kThreads = FP8A ? 448 : 192;        // + 8 converter warps
  static constexpr int kSmemBytes = 1024 /*align slack*/ + kStages * kStageBytes +
                                    kBars * 8 /*barriers*/ + (3 * kMaxSeg + 16) * 4;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kTmemUsed <= kTmemCols, "tensor memory");
  static_assert(!FP8A || (kStages % 2 == 0 && kASlots % 2 == 0), "even rings");
  static_assert(kRawOff % 1024 == 0 && kStageBytes % 1024 == 0, "swizzle alignment");
  static_assert(!(FP8A && SMALLA), "the E4M3 loader has its own slot layout");
  static_assert(!SMALLA || kStageBytes >= kABytes + (kABoxes - 1) * kABoxSlot,
                "the MMA's 128 A rows stay inside the stage");
  static_assert(KS == kBK || (KS == 2 * kBK && SMALLA && !FP8A), "deep stages: small-A bf16");
};

// Pair kernel, per CTA: TMA slot [A bf16 tile 16 KB][2 B atoms 16 KB], or with an
// E4M3 A operand [2 B atoms 16 KB][E4M3 A tile 8 KB] and A slots in tensor memory
// after a single accumulator buffer.
template <bool FP8A = false>
struct PairGeometry {
  static constexpr int kN = 2 * kPairAtoms * 64;           // 256 accumulator columns
  static constexpr int kBOff = FP8A ? 0 : kABytes;
  static constexpr int kRawOff = kPairAtoms * kAtomBytes;
  static constexpr int kStageBytes = kPairAtoms * kAtomBytes + (FP8A ? kRawBytes : kABytes);
  static constexpr int kStages = FP8A ? 8 : 6;
  static constexpr int kASlots = FP8A ? 8 : 0;
  static constexpr int kAccBufs = FP8A ? 1 : 2;
  static constexpr int kACol = kAccBufs * kN;
  static constexpr int kTmemAlloc = 512;
  // full, empty, tfull[2], tempty[2], drain, (FP8A) raw[S], afull[A], aempty[A]
  static constexpr int kBars = 2 * kStages + 5 + (FP8A ? kStages + 2 * kASlots : 0);
  static constexpr int kThreads = FP8A ? 448 : 192;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBars * 8 +
                                    (3 * kMaxSeg + 16) * 4;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kACol + kASlots * kASlotCols <= kTmemAlloc, "tensor memory");
  static_assert(!FP8A || (kStages % 2 == 0 && kASlots % 2 == 0), "even rings");
  static_assert(kRawOff % 1024 == 0 && kStageBytes % 1024 == 0, "swizzle alignment");
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
  // E4M3 A operand only: fp32 scales [max_rows, n_groups], one per group_k
  // consecutive K values of a row.
  const float* scales;
  int n_groups;
  int group_k;
  // Single-CTA kernel: rows per tile (the height of the A box TMA stages: 128, or
  // 16..64 when experts hold few rows; the MMA still runs M = 128 and the rows
  // past the box are never stored) and the A bytes one stage's TMA delivers.
  int bm;
  int a_box_bytes;
  // Gathered A rows (bf16 gate/up only; nullptr otherwise): row i of the expert
  // row space is token row gather[i] / gather_k of the [gather_T, K] tensor the A
  // map describes (one-row boxes), loaded four rows per TMA gather.
  const int32_t* gather;
  int gather_k;
  int gather_T;
  // bf16 down pass (single-CTA kernel) issued right after this library's gate/up
  // pass on the same stream and segment table: the segment table and the first
  // tile's weight atoms are read before waiting for the gate/up pass (see
  // moe_grouped_down_chained).
  int chained;
};

// ------------------------------ PTX wrappers -------------------------------

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

// This thread's TMEM lane, 32 consecutive 32-bit columns from `taddr` (the
// warp's lane quadrant is in the address).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D (+)= A B with the A operand in tensor memory (rows = lanes, two K-consecutive
// bf16 per 32-bit column) and B in shared memory.
__device__ __forceinline__ void mma_bf16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
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

__device__ __forceinline__ void mma_bf16_pair_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
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

// Four rows (r0..r3) x 64 columns from column c_inner of a map with one-row boxes,
// landing as four consecutive 128-byte rows at dst (with the map's swizzle).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c_inner, const int (&r)[4]) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c_inner), "r"(r[0]), "r"(r[1]),
      "r"(r[2]), "r"(r[3])
      : "memory");
}

__device__ __forceinline__ void tma_gather4_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c_inner,
                                                 const int (&r)[4]) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4"
      ".mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c_inner), "r"(r[0]),
      "r"(r[1]), "r"(r[2]), "r"(r[3])
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

// Token rows of the four A rows 4*lane .. 4*lane+3 of a gathered box whose first
// row is `row0` of the expert row space and whose first `live` rows belong to the
// segment.  Rows past `live` (the ragged tail) load token 0: they are computed
// but never stored.  A map entry outside the routes is reported and reads token 0.
__device__ __forceinline__ void gather_tokens(const GemmArgs& a, int row0, int live, int lane,
                                              int (&tok)[4]) {
  const int n_routes = a.gather_T * a.gather_k;
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = 4 * lane + j;
    int t = 0;
    if (i < live) {
      const int r = __ldg(a.gather + row0 + i);
      if (r >= 0 && r < n_routes) t = r / a.gather_k; else bad = true;
    }
    tok[j] = t;
  }
  if (bad) report(a.dev_status, MOE_DEV_BAD_ROW);
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

// E4M3 A operand.  Two groups of four converter warps take the stages in turn
// (stage n goes to group n % 2), so the hand-over of one stage overlaps the
// conversion of the next.  Thread lane of converter warp w converts row
// r = 32 (w % 4) + lane -- the tensor-memory lane its warp may access -- of the
// staged [128 x 64] E4M3 tile (TMA layout with 64-byte swizzle: 16-byte chunk c
// of row r at chunk c ^ ((r >> 1) & 3)): each value becomes
// bf16(fp32(decode(code) * scale of its row and group)), two K-consecutive
// values per 32-bit column of the row's lane in A slot n % kASlots.  Per stage:
// wait for the E4M3 tile (raw barrier n % kStages) and for the MMA to have
// released the A slot, convert, store to tensor memory, wait for the stores,
// then one arrival per warp on the slot's afull barrier.  Scales are loaded one
// own stage ahead (the first one of a tile during the previous tile).
constexpr int kConvGroups = 2;

template <int kStages, int kStageBytes, int kRawOff, int kASlots>
__device__ __forceinline__ void convert_a_tiles(uint8_t* stage_base, uint32_t tmem_a0, int ct,
                                                int lane, int t0, int t_step, int total_tiles,
                                                int k_steps, int bm, int row_off,
                                                const GemmArgs& args, const Smem& sm,
                                                int n_blocks, int bn_out, uint32_t raw_bar0,
                                                uint32_t afull_bar0, uint32_t aempty_bar0,
                                                volatile int* abort_flag) {
  const int quad = (ct >> 5) & 3;  // converter warps start at warp 6: (6 + i) & 3 == (2 + i) & 3
  const int r = ((quad + 2) & 3) * 32 + lane;  // = 32 * (warp % 4) + lane
  const int grp = ct >> 7;         // converter group
  const uint32_t tmem_row = tmem_a0 + (static_cast<uint32_t>(r & ~31) << 16);
  const int ng = args.n_groups;
  auto scale_row = [&](int t) {
    const Tile tl = tile_of(t, sm.s_tile_start, sm.s_begin, sm.s_count, args.n_seg, bm, bn_out,
                            n_blocks, args.m_outer);
    // rows past the tensor (zero-filled by TMA) read the last row's scale: unused
    const int row = min(tl.row0 + row_off + r, args.max_rows - 1);
    return args.scales + static_cast<int64_t>(row) * ng;
  };
  auto scale_at = [&](const float* row, int ks) { return __ldg(row + (ks * kBK) / args.group_k); };
  // first k-step of a tile that belongs to this group, given the tile's first stage index
  auto first_own = [&](int n_base) {
    const int k0 = (grp - n_base) % kConvGroups;
    return k0 < 0 ? k0 + kConvGroups : k0;
  };
  const int swz_in = (r >> 1) & 3;
  int n_base = 0;  // stage index (over all of this CTA's tiles) of the tile's k-step 0
  int t = t0;
  const float* next_row = nullptr;
  float next_first = 1.0f;
  if (t < total_tiles) {
    next_row = scale_row(t);
    if (first_own(0) < k_steps) next_first = scale_at(next_row, first_own(0));
  }
  for (; t < total_tiles; t += t_step, n_base += k_steps) {
    const float* srow = next_row;
    float sc = next_first;
    if (t + t_step < total_tiles) {
      next_row = scale_row(t + t_step);
      const int k0 = first_own(n_base + k_steps);
      if (k0 < k_steps) next_first = scale_at(next_row, k0);
    }
    for (int ks = first_own(n_base); ks < k_steps; ks += kConvGroups) {
      const int n = n_base + ks;
      const int s = n % kStages, a = n % kASlots;
      const float sc_next = ks + kConvGroups < k_steps ? scale_at(srow, ks + kConvGroups) : 0.0f;
      // every exit is warp-uniform: the tensor-memory stores below are .sync.aligned
      if (!__all_sync(0xFFFFFFFFu, wait_bounded(raw_bar0 + 8 * s,
                                                static_cast<uint32_t>(n / kStages) & 1u,
                                                abort_flag, args.dev_status)))
        return;
      const uint8_t* raw = stage_base + s * kStageBytes + kRawOff + r * 64;
      uint32_t col[kASlotCols];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(raw + ((c ^ swz_in) << 4));
        uint4 lo, hi;
        dequant16(v, sc, lo, hi);
        col[8 * c + 0] = lo.x; col[8 * c + 1] = lo.y; col[8 * c + 2] = lo.z; col[8 * c + 3] = lo.w;
        col[8 * c + 4] = hi.x; col[8 * c + 5] = hi.y; col[8 * c + 6] = hi.z; col[8 * c + 7] = hi.w;
      }
      // the MMAs that read this slot's previous contents must have completed
      if (!__all_sync(0xFFFFFFFFu,
                      wait_bounded(aempty_bar0 + 8 * a, (static_cast<uint32_t>(n / kASlots) & 1u) ^ 1u,
                                   abort_flag, args.dev_status)))
        return;
      tc_fence_after();
      tmem_st32(tmem_row + static_cast<uint32_t>(a * kASlotCols), col);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(afull_bar0 + 8 * a);
      sc = sc_next;
    }
  }
}

// Pair kernel, rank 1: one thread forwards each completed local afull[a] phase
// to the leader's afull[a] barrier, whose thread issues the MMAs that read this
// rank's A slot.  The arrival is relaxed: by the time this thread has acquired
// the local phase, every converter warp has waited for its tensor-memory stores
// to complete (tcgen05.wait::st) and fenced them before its release, so the
// slot's contents are in place before the signal leaves this CTA.  (A release
// at cluster scope per stage measured about 1,500 cycles and paced the whole
// pipeline.)
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ bool forward_conversions(int n_stages_total, int slots,
                                                    uint32_t local_bar0, volatile int* abort_flag,
                                                    uint32_t* dev_status) {
  for (int n = 0; n < n_stages_total; ++n) {
    const int a = n % slots;
    if (!wait_bounded(local_bar0 + 8 * a, static_cast<uint32_t>(n / slots) & 1u, abort_flag,
                      dev_status))
      return false;
    mbar_arrive_remote_relaxed(map_to_rank(local_bar0 + 8 * a, 0));
  }
  return true;
}

// ------------------------- single-CTA kernel --------------------------------

template <int N_ATOMS, bool SWIGLU, bool FP8A, bool SMALLA, int KS>
__global__ void __launch_bounds__(Geometry<N_ATOMS, FP8A, SMALLA, KS>::kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b0,
                    const __grid_constant__ CUtensorMap tmap_b1, const GemmArgs args) {
  using G = Geometry<N_ATOMS, FP8A, SMALLA, KS>;
  constexpr int kStages = G::kStages;
  constexpr int kASlots = G::kASlots;
  constexpr int kAccBufs = G::kAccBufs;
  constexpr int kN = G::kN;
  constexpr int kBnOut = SWIGLU ? kN / 2 : kN;  // output columns per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // bars: full[S], empty[S], tmem_full[2], tmem_empty[2], drain, (FP8A) afull[A], aempty[A]
  const Smem sm = carve(stage_base + kStages * G::kStageBytes, G::kBars);
  uint64_t* bars = sm.bars;
  volatile int* abort_flag = sm.abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_seg = args.n_seg;
  const int n_blocks = args.N / kBnOut;
  const int k_steps = args.K / KS;
  const int stage_tx = G::kABoxes * args.a_box_bytes + N_ATOMS * G::kAtom;

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };
  auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * kStages + b); };
  auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * kStages + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * kStages + 4);
  auto afull_bar = [&](int a) { return smem_u32(bars + 2 * kStages + 5 + a); };
  auto aempty_bar = [&](int a) { return smem_u32(bars + 2 * kStages + 5 + kASlots + a); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < kASlots; ++a) {
      mbar_init(afull_bar(a), 4);  // one arrival per warp of the converting group
      mbar_init(aempty_bar(a), 1);
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
  // Everything above is local; global data only after the wait.  A chained down
  // pass reads only data written before the gate/up pass began (the segment table,
  // the weights) until its producer waits, just before its first A load; its other
  // warps touch no global data the gate/up pass writes.  The gate/up pass lets its
  // dependents launch right after its own wait: its grid is one CTA per SM, all
  // resident by then, and a chained down pass then stages weights on the SMs the
  // gate/up tiles leave idle or free first.
  const bool chained = !SWIGLU && !FP8A && args.chained != 0;
  if (!chained) pdl_wait();
  if (SWIGLU) pdl_trigger();
  if (threadIdx.x >= 64 && threadIdx.x < 192)
    build_segment_table(args, args.bm, n_blocks, sm.s_begin, sm.s_count, sm.s_tile_start, sm.warp_tot);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;
  const int total_tiles = sm.s_tile_start[n_seg];

  bool gathered = false;
  if constexpr (SWIGLU && !FP8A && KS == kBK) gathered = args.gather != nullptr;
  if (warp == 0 && gathered) {
    // ============ TMA producer, A rows gathered from token order ============
    // The whole warp: lane 0 waits and arms the stage, lanes 0 .. bm/4-1 each
    // gather four A rows (512 bytes at offset 512 * lane of the A tile), lane 0
    // loads the B atoms.
    if constexpr (SWIGLU && !FP8A && KS == kBK) {
      const int lanes_a = args.bm / 4;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const Tile tl = tile_of(t, sm.s_tile_start, sm.s_begin, sm.s_count, n_seg, args.bm,
                                kBnOut, n_blocks, args.m_outer);
        int tok[4];
        gather_tokens(args, tl.row0, tl.rows, lane, tok);
        const int b_row0 = tl.seg * args.K;
        for (int ks = 0; ks < k_steps; ++ks) {
          bool w = true;
          if (lane == 0) w = wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, args.dev_status);
          if (!__shfl_sync(0xFFFFFFFFu, w, 0)) { ok = false; break; }
          const uint32_t st = smem_u32(stage_base + s * G::kStageBytes);
          if (lane == 0)
            mbar_arrive_expect_tx(full_bar(s), args.a_box_bytes + N_ATOMS * kAtomBytes);
          __syncwarp();
          if (lane < lanes_a) tma_gather4(st + lane * 512, &tmap_a, full_bar(s), ks * kBK, tok);
          if (lane == 0) {
            constexpr int half = N_ATOMS / 2;
#pragma unroll
            for (int a = 0; a < N_ATOMS; ++a)
              tma_load_2d(st + G::kBOff + a * kAtomBytes, a < half ? &tmap_b0 : &tmap_b1,
                          full_bar(s), tl.n0 + (a % half) * 64, b_row0 + ks * kBK);
          }
          if (++s == kStages) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok && lane == 0) {
        int ss = s;
        uint32_t pp = ph;
        for (int i = 0; i < kStages; ++i) {
          if (--ss < 0) { ss = kStages - 1; pp ^= 1u; }
          wait_drain(full_bar(ss), pp);
        }
      }
    }
  } else if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      int staged = 0;  // k-steps of the first tile whose weight atoms precede the wait
      if (chained) {
        if (static_cast<int>(blockIdx.x) < total_tiles) {
          const Tile tl = tile_of(blockIdx.x, sm.s_tile_start, sm.s_begin, sm.s_count, n_seg,
                                  args.bm, kBnOut, n_blocks, args.m_outer);
          const int b_row0 = tl.seg * args.K;
          staged = min(kStages, k_steps);
          for (int ks = 0; ks < staged; ++ks) {  // the ring's first round: all slots free
            const uint32_t st = smem_u32(stage_base + ks * G::kStageBytes);
            mbar_arrive_expect_tx(full_bar(ks), stage_tx);
#pragma unroll
            for (int a = 0; a < N_ATOMS; ++a)
              tma_load_2d(st + G::kBOff + a * G::kAtom, &tmap_b0, full_bar(ks), tl.n0 + a * 64,
                          b_row0 + ks * KS);
          }
        }
        pdl_wait();  // the A rows (H) are the gate/up pass's output
      }
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const Tile tl = tile_of(t, sm.s_tile_start, sm.s_begin, sm.s_count, n_seg, args.bm, kBnOut,
                                n_blocks, args.m_outer);
        const int b_row0 = tl.seg * args.K;
        for (int ks = 0; ks < k_steps; ++ks) {
          const bool pre = t == static_cast<int>(blockIdx.x) && ks < staged;
          const uint32_t st = smem_u32(stage_base + s * G::kStageBytes);
          if (!pre) {
            if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, args.dev_status)) { ok = false; break; }
            mbar_arrive_expect_tx(full_bar(s), stage_tx);
          }
          // A: the bf16 tile (KS / 64 boxes), or the E4M3 tile for the converter warps
#pragma unroll
          for (int h = 0; h < G::kABoxes; ++h)
            tma_load_2d(FP8A ? st + G::kRawOff : st + h * G::kABoxSlot, &tmap_a, full_bar(s),
                        ks * KS + h * kBK, tl.row0);
          if (pre) {  // its weight atoms are already on their way
            if (++s == kStages) { s = 0; ph ^= 1u; }
            continue;
          }
#pragma unroll
          for (int a = 0; a < N_ATOMS; ++a) {
            const uint32_t dst = st + G::kBOff + a * G::kAtom;
            if constexpr (SWIGLU) {
              const int half = N_ATOMS / 2;
              const CUtensorMap* m = a < half ? &tmap_b0 : &tmap_b1;
              const int col = tl.n0 + (a % half) * 64;
              tma_load_2d(dst, m, full_bar(s), col, b_row0 + ks * KS);
            } else {
              tma_load_2d(dst, &tmap_b0, full_bar(s), tl.n0 + a * 64, b_row0 + ks * KS);
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
      int s = 0, a = 0;
      uint32_t ph = 0, aph = 0;
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
          if (FP8A && !wait_bounded(afull_bar(a), aph, abort_flag, args.dev_status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = smem_u32(stage_base + s * G::kStageBytes);
          const uint32_t b_addr = st + G::kBOff;
#pragma unroll
          for (int kk = 0; kk < KS / kUmmaK; ++kk) {
            // B: N-major, advance 16 K rows = 2048 bytes; atoms of 64 columns
            // are G::kAtom apart (LBO), 8-row K groups 1024 bytes apart (SBO).
            const uint64_t bd = smem_desc_sw128(b_addr + kk * kUmmaK * 128, G::kAtom, 1024);
            if constexpr (FP8A) {
              // A in tensor memory: 16 K values = 8 columns of slot a
              const uint32_t ta = tmem_base + static_cast<uint32_t>(G::kACol + a * kASlotCols + kk * (kUmmaK / 2));
              mma_bf16_ta(d_tmem, ta, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
            } else {
              // A: K-major, advance 16 elements = 32 bytes inside the swizzle row
              // of the stage's (kk / 4)-th A box.
              constexpr int kPerBox = kBK / kUmmaK;
              const uint64_t ad = smem_desc_sw128(
                  st + (kk / kPerBox) * G::kABoxSlot + (kk % kPerBox) * kUmmaK * 2, 16, 1024);
              mma_bf16(d_tmem, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
            }
          }
          issued_any = true;
          mma_commit(empty_bar(s));  // frees this stage once its MMAs have read it
          if (++s == kStages) { s = 0; ph ^= 1u; }
          if constexpr (FP8A) {
            mma_commit(aempty_bar(a));  // and the converted A slot
            if (++a == kASlots) { a = 0; aph ^= 1u; }
          }
        }
        if (!ok) break;
        mma_commit(tfull_bar(buf));  // accumulator ready for the epilogue
        if (++buf == kAccBufs) { buf = 0; acc_ph ^= 1u; }
      }
      if (!ok && issued_any) {
        // All MMAs issued so far must finish before tensor memory is freed.
        mma_commit(drain_bar);
        wait_drain(drain_bar, 0);
      }
    }
  } else if (warp < 6) {
    // ======================= epilogue (warps 2..5) =======================
    const int quad = warp & 3;            // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;       // accumulator row owned by this thread
    int buf = 0;
    uint32_t acc_ph = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
      const Tile tl = tile_of(t, sm.s_tile_start, sm.s_begin, sm.s_count, n_seg, args.bm, kBnOut,
                              n_blocks, args.m_outer);
      // warp-uniform exit: the tensor-memory loads below are .sync.aligned
      if (!__all_sync(0xFFFFFFFFu, wait_bounded(tfull_bar(buf), acc_ph, abort_flag, args.dev_status)))
        break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(buf * kN);
      const bool live = r < tl.rows;
      uint16_t* orow = args.out + static_cast<int64_t>(tl.row0 + (live ? r : 0)) * args.N + tl.n0;
      epilogue_row<kBnOut, SWIGLU>(taddr, live, orow);
      tc_fence_before();
      mbar_arrive(tempty_bar(buf));
      if (++buf == kAccBufs) { buf = 0; acc_ph ^= 1u; }
    }
  } else if constexpr (FP8A) {
    // ================ E4M3 -> bf16 converter (warps 6..13) ================
    convert_a_tiles<kStages, G::kStageBytes, G::kRawOff, kASlots>(
        stage_base, tmem_base + G::kACol, threadIdx.x - 192, lane, blockIdx.x, gridDim.x,
        total_tiles, k_steps, args.bm, 0, args, sm, n_blocks, kBnOut, full_bar(0), afull_bar(0),
        aempty_bar(0), abort_flag);
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
//                and each rank's TMA completes its bytes on the leader's barrier
//                (with an E4M3 A operand: the B bytes only);
//   empty[s]     both ranks: the leader's commit is multicast to both;
//   raw[s]       E4M3 A only, both ranks: the rank's own E4M3 tile has landed;
//   afull[a]     E4M3 A only: the rank's bf16 A slot a is written (4 converter
//                warps); the leader's also counts one arrival forwarded by rank 1;
//   aempty[a]    E4M3 A only, both ranks: multicast commit, slot a free again;
//   tfull[b]     both ranks: multicast commit after a tile's last MMA;
//   tempty[b]    leader only: one arrival per epilogue warp of both ranks (8).
template <bool SWIGLU, bool FP8A>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairGeometry<FP8A>::kThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b0,
                         const __grid_constant__ CUtensorMap tmap_b1, const GemmArgs args) {
  using PG = PairGeometry<FP8A>;
  constexpr int kStagesPair = PG::kStages;
  constexpr int kPairStageBytes = PG::kStageBytes;
  constexpr int kASlots = PG::kASlots;
  constexpr int kAccBufs = PG::kAccBufs;
  constexpr int kN = PG::kN;                     // 256 accumulator columns
  constexpr int kBnOut = SWIGLU ? kN / 2 : kN;   // output columns per tile
  constexpr int kPairBM = 2 * kBM;               // rows per tile
  constexpr int kTmemAlloc = PG::kTmemAlloc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Smem sm = carve(stage_base + kStagesPair * kPairStageBytes, PG::kBars);
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
  auto raw_bar = [&](int s) { return smem_u32(bars + 2 * kStagesPair + 5 + s); };
  auto afull_bar = [&](int a) { return smem_u32(bars + 3 * kStagesPair + 5 + a); };
  auto aempty_bar = [&](int a) { return smem_u32(bars + 3 * kStagesPair + 5 + kASlots + a); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesPair; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      if (FP8A) mbar_init(raw_bar(s), 1);
    }
    for (int a = 0; a < kASlots; ++a) {
      // leader: its own 4 converter arrivals + 1 forwarded from rank 1; rank 1: 4
      mbar_init(afull_bar(a), leader ? 5 : 4);
      mbar_init(aempty_bar(a), 1);
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
  if (threadIdx.x >= 64 && threadIdx.x < 192)
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

  bool gathered = false;
  if constexpr (SWIGLU && !FP8A) gathered = args.gather != nullptr;
  if (warp == 0 && gathered) {
    // ==== TMA producer (both ranks), A rows gathered from token order ====
    // Every lane gathers four of this rank's 128 A rows (512 bytes at offset
    // 512 * lane of its A tile); lane 0 waits, the leader's lane 0 arms the stage
    // for both ranks' bytes, and lane 0 loads this rank's B atoms.
    if constexpr (SWIGLU && !FP8A) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      bool issued_any = false;
      for (int t = cid; t < total_tiles && ok; t += n_clusters) {
        const Tile tl = tile_of(t, sm.s_tile_start, sm.s_begin, sm.s_count, n_seg, kPairBM,
                                kBnOut, n_blocks, args.m_outer);
        const int my_row0 = tl.row0 + static_cast<int>(rank) * kBM;
        const int my_live = min(max(tl.rows - static_cast<int>(rank) * kBM, 0), kBM);
        int tok[4];
        gather_tokens(args, my_row0, my_live, lane, tok);
        const int b_row0 = tl.seg * args.K;
        for (int ks = 0; ks < k_steps; ++ks) {
          bool w = true;
          if (lane == 0) w = wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, args.dev_status);
          if (!__shfl_sync(0xFFFFFFFFu, w, 0)) { ok = false; break; }
          const uint32_t full_leader = map_to_rank(full_bar(s), 0);
          const uint32_t st = smem_u32(stage_base + s * kPairStageBytes);
          if (leader && lane == 0) mbar_arrive_expect_tx(full_bar(s), 2 * kPairStageBytes);
          __syncwarp();
          tma_gather4_pair(st + lane * 512, &tmap_a, full_leader, ks * kBK, tok);
          if (lane == 0) {
#pragma unroll
            for (int a = 0; a < kPairAtoms; ++a)
              tma_load_2d_pair(st + PG::kBOff + a * kAtomBytes, leader ? &tmap_b0 : &tmap_b1,
                               full_leader, tl.n0 + a * 64, b_row0 + ks * kBK);
          }
          issued_any = true;
          if (++s == kStagesPair) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok && issued_any && lane == 0) {
        if (leader) {
          int ss = s;
          uint32_t pp = ph;
          for (int i = 0; i < kStagesPair; ++i) {
            if (--ss < 0) { ss = kStagesPair - 1; pp ^= 1u; }
            wait_drain(full_bar(ss), pp);
          }
        } else {
          spin_ns(2000000ull);  // this rank's copies complete on the leader's barriers
        }
      }
    }
  } else if (warp == 0) {
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
          const uint32_t st = smem_u32(stage_base + s * kPairStageBytes);
          if constexpr (FP8A) {
            // this rank's E4M3 rows land on its own raw barrier; B on the leader's
            if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * kPairAtoms * kAtomBytes);
            mbar_arrive_expect_tx(raw_bar(s), kRawBytes);
            tma_load_2d(st + PG::kRawOff, &tmap_a, raw_bar(s), ks * kBK,
                        tl.row0 + static_cast<int>(rank) * kBM);
          } else {
            if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * kPairStageBytes);
            tma_load_2d_pair(st, &tmap_a, full_leader, ks * kBK,
                             tl.row0 + static_cast<int>(rank) * kBM);
          }
#pragma unroll
          for (int a = 0; a < kPairAtoms; ++a) {
            const uint32_t dst = st + PG::kBOff + a * kAtomBytes;
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
        if (FP8A) {  // this rank's own E4M3 copies
          int ss = s;
          uint32_t pp = ph;
          for (int i = 0; i < kStagesPair; ++i) {
            if (--ss < 0) { ss = kStagesPair - 1; pp ^= 1u; }
            wait_drain(raw_bar(ss), pp);
          }
        }
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
      int s = 0, a = 0;
      uint32_t ph = 0, aph = 0;
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
          if (FP8A && !wait_bounded<true>(afull_bar(a), aph, abort_flag, args.dev_status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = smem_u32(stage_base + s * kPairStageBytes);
          const uint32_t b_addr = st + PG::kBOff;
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
            const uint64_t bd = smem_desc_sw128(b_addr + kk * kUmmaK * 128, kAtomBytes, 1024);
            if constexpr (FP8A) {
              // A in tensor memory, each rank's 128 rows in its own lanes
              const uint32_t ta = tmem_base + static_cast<uint32_t>(PG::kACol + a * kASlotCols + kk * (kUmmaK / 2));
              mma_bf16_pair_ta(d_tmem, ta, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
            } else {
              const uint64_t ad = smem_desc_sw128(st + kk * kUmmaK * 2, 16, 1024);
              mma_bf16_pair(d_tmem, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
            }
          }
          issued_any = true;
          mma_commit_pair(empty_bar(s), 0x3);  // frees stage s in both ranks
          if (++s == kStagesPair) { s = 0; ph ^= 1u; }
          if constexpr (FP8A) {
            mma_commit_pair(aempty_bar(a), 0x3);  // and A slot a in both ranks
            if (++a == kASlots) { a = 0; aph ^= 1u; }
          }
        }
        if (!ok) break;
        mma_commit_pair(tfull_bar(buf), 0x3);  // both ranks' accumulators ready
        if (++buf == kAccBufs) { buf = 0; acc_ph ^= 1u; }
      }
      if (!ok && issued_any) {
        mma_commit_pair(drain_bar, 0x1);
        wait_drain(drain_bar, 0);
      }
    } else if (FP8A && lane == 0) {
      // rank 1: forward its converted A slots to the leader
      const int my_tiles = cid < total_tiles ? (total_tiles - cid + n_clusters - 1) / n_clusters : 0;
      forward_conversions(my_tiles * k_steps, kASlots, afull_bar(0), abort_flag, args.dev_status);
    }
  } else if (warp < 6) {
    // ======================= epilogue (warps 2..5, both ranks) ===============
    const int quad = warp & 3;
    const int r = quad * 32 + lane;                        // row within this rank's half
    const int tile_r = static_cast<int>(rank) * kBM + r;   // row within the 256-row tile
    int buf = 0;
    uint32_t acc_ph = 0;
    for (int t = cid; t < total_tiles; t += n_clusters) {
      const Tile tl = tile_of(t, sm.s_tile_start, sm.s_begin, sm.s_count, n_seg, kPairBM, kBnOut,
                              n_blocks, args.m_outer);
      // warp-uniform exit: the tensor-memory loads below are .sync.aligned
      if (!__all_sync(0xFFFFFFFFu, wait_bounded(tfull_bar(buf), acc_ph, abort_flag, args.dev_status)))
        break;
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
      if (++buf == kAccBufs) { buf = 0; acc_ph ^= 1u; }
    }
  } else if constexpr (FP8A) {
    // ============ E4M3 -> bf16 converter (warps 6..13, both ranks) ============
    convert_a_tiles<kStagesPair, kPairStageBytes, PG::kRawOff, kASlots>(
        stage_base, tmem_base + PG::kACol, threadIdx.x - 192, lane, cid, n_clusters, total_tiles,
        k_steps, kPairBM, static_cast<int>(rank) * kBM, args, sm, n_blocks, kBnOut, raw_bar(0),
        afull_bar(0), aempty_bar(0), abort_flag);
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

// ------------------- both passes in one persistent launch ---------------------
//
// Decode-sized batches (row boxes of at most 32 rows, d and I multiples of 128) can
// run the gate/up and the down pass as one launch of the narrow single-CTA tiles
// with 128-K stages.  The units are the gate/up tiles, then the down tiles, dealt
// round robin to one CTA per SM.  A CTA's producer streams a down tile's weights
// into the stage ring right behind its own gate/up weights (or at once, on an SM
// without a gate/up tile) and waits only before the tile's H rows, until every
// gate/up tile of the tile's expert has stored its H columns.  The weights of the
// two passes so stream back to back, with no kernel boundary between them.
// Per expert q, two counters in `sync` (all zero before a launch, all zero after it):
// sync[q] counts, four per tile (one release add per epilogue warp after its lanes'
// stores), the gate/up tiles that stored their H columns, sync[n_seg + q] the stored
// down tiles; the last count of q's down tiles resets both.  A down tile waits only on gate/up tiles, which
// come before every down tile in every CTA's order and wait on nothing, and every
// CTA is resident (one per SM), so each wait ends; it is bounded all the same.
__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Spin (bounded) until *c >= need; false when the CTA is aborting or the wait times out.
__device__ __forceinline__ bool wait_count(const int32_t* c, int need, volatile int* abort_flag,
                                           uint32_t* dev_status) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (ld_acquire_gpu(c) >= need) return true;
    if (*abort_flag) return false;
    if ((i & 255u) == 255u && global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      report(dev_status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
}

// Down tile t of the one-launch kernel: the same segment order as the gate/up tiles
// (whose table counts n_blocks_gu tiles per m-block), n_blocks_dn tiles per m-block.
__device__ __forceinline__ Tile down_tile_of(int t, const int* tile_start_gu, const int* s_begin,
                                             const int* s_count, int n_seg, int bm, int n_blocks_gu,
                                             int n_blocks_dn) {
  int lo = 0, hi = n_seg - 1;
  while (lo < hi) {  // last q whose first down tile is at or before t
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start_gu[mid] / n_blocks_gu * n_blocks_dn <= t) lo = mid; else hi = mid - 1;
  }
  const int q = lo;
  const int local = t - tile_start_gu[q] / n_blocks_gu * n_blocks_dn;
  const int m_blocks = (s_count[q] + bm - 1) / bm;
  const int nb = local / m_blocks, mb = local % m_blocks;
  Tile tl;
  tl.seg = q;
  tl.row0 = s_begin[q] + mb * bm;
  tl.rows = min(bm, s_count[q] - mb * bm);
  tl.n0 = nb * 128;
  return tl;
}

__global__ void __launch_bounds__(192, 1)
grouped_swiglu_onepass_kernel(const __grid_constant__ CUtensorMap tmap_x,
                              const __grid_constant__ CUtensorMap tmap_wg,
                              const __grid_constant__ CUtensorMap tmap_wu,
                              const __grid_constant__ CUtensorMap tmap_h,
                              const __grid_constant__ CUtensorMap tmap_wd, const GemmArgs args,
                              uint16_t* __restrict__ y, int32_t* __restrict__ sync) {
  using G = Geometry<2, false, true, 2 * kBK>;
  constexpr int KS = 2 * kBK;
  constexpr int kStages = G::kStages;
  constexpr int kN = G::kN;  // 128 accumulator columns in both passes
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Smem sm = carve(stage_base + kStages * G::kStageBytes, G::kBars);
  uint64_t* bars = sm.bars;
  volatile int* abort_flag = sm.abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_seg = args.n_seg;
  const int d = args.K, I = args.N;                        // gate/up: K = d, N = I
  const int nb_gu = I / 64, nb_dn = d / 128;               // tiles per m-block
  const int ks_gu = d / KS, ks_dn = I / KS;                // k-steps per tile
  const int stage_tx = G::kABoxes * args.a_box_bytes + 2 * G::kAtom;

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
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_wg)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_wu)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_h)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_wd)) : "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(sm.tmem_slot), G::kTmemAlloc);
  // everything above is local; global data only after the wait (one CTA per SM, all
  // resident, so the dependents may launch right away)
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x >= 64 && threadIdx.x < 192)
    build_segment_table(args, args.bm, nb_gu, sm.s_begin, sm.s_count, sm.s_tile_start, sm.warp_tot);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;
  const int total_gu = sm.s_tile_start[n_seg];
  const int total = total_gu + total_gu / nb_gu * nb_dn;
  auto unit_tile = [&](int u) {
    return u < total_gu ? tile_of(u, sm.s_tile_start, sm.s_begin, sm.s_count, n_seg, args.bm, 64,
                                  nb_gu, 0)
                        : down_tile_of(u - total_gu, sm.s_tile_start, sm.s_begin, sm.s_count,
                                       n_seg, args.bm, nb_gu, nb_dn);
  };

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Tile tl = unit_tile(u);
        if (u < total_gu) {
          const int b_row0 = tl.seg * d;
          for (int ks = 0; ks < ks_gu; ++ks) {
            if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, args.dev_status)) { ok = false; break; }
            const uint32_t st = smem_u32(stage_base + s * G::kStageBytes);
            mbar_arrive_expect_tx(full_bar(s), stage_tx);
#pragma unroll
            for (int hb = 0; hb < G::kABoxes; ++hb)
              tma_load_2d(st + hb * G::kABoxSlot, &tmap_x, full_bar(s), ks * KS + hb * kBK, tl.row0);
            tma_load_2d(st + G::kBOff, &tmap_wg, full_bar(s), tl.n0, b_row0 + ks * KS);
            tma_load_2d(st + G::kBOff + G::kAtom, &tmap_wu, full_bar(s), tl.n0, b_row0 + ks * KS);
            if (++s == kStages) { s = 0; ph ^= 1u; }
          }
        } else {
          // the weights of the first stages at once, the H rows once the expert's
          // gate/up tiles have stored them
          const int b_row0 = tl.seg * I;
          const int staged = ks_dn < kStages ? ks_dn : kStages;
          const int s0 = s;
          for (int ks = 0; ks < staged && ok; ++ks) {
            if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, args.dev_status)) { ok = false; break; }
            const uint32_t st = smem_u32(stage_base + s * G::kStageBytes);
            mbar_arrive_expect_tx(full_bar(s), stage_tx);
            tma_load_2d(st + G::kBOff, &tmap_wd, full_bar(s), tl.n0, b_row0 + ks * KS);
            tma_load_2d(st + G::kBOff + G::kAtom, &tmap_wd, full_bar(s), tl.n0 + 64, b_row0 + ks * KS);
            if (++s == kStages) { s = 0; ph ^= 1u; }
          }
          if (!ok) break;
          const int need = 4 * ((sm.s_count[tl.seg] + args.bm - 1) / args.bm) * nb_gu;
          if (!wait_count(sync + tl.seg, need, abort_flag, args.dev_status)) { ok = false; break; }
          // H was stored by other SMs through the generic proxy; the copies read it
          // through the async proxy
          asm volatile("fence.proxy.async.global;" ::: "memory");
          for (int ks = 0; ks < staged; ++ks) {
            const int ss = (s0 + ks) % kStages;
            const uint32_t st = smem_u32(stage_base + ss * G::kStageBytes);
#pragma unroll
            for (int hb = 0; hb < G::kABoxes; ++hb)
              tma_load_2d(st + hb * G::kABoxSlot, &tmap_h, full_bar(ss), ks * KS + hb * kBK, tl.row0);
          }
          for (int ks = staged; ks < ks_dn; ++ks) {
            if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, args.dev_status)) { ok = false; break; }
            const uint32_t st = smem_u32(stage_base + s * G::kStageBytes);
            mbar_arrive_expect_tx(full_bar(s), stage_tx);
#pragma unroll
            for (int hb = 0; hb < G::kABoxes; ++hb)
              tma_load_2d(st + hb * G::kABoxSlot, &tmap_h, full_bar(s), ks * KS + hb * kBK, tl.row0);
            tma_load_2d(st + G::kBOff, &tmap_wd, full_bar(s), tl.n0, b_row0 + ks * KS);
            tma_load_2d(st + G::kBOff + G::kAtom, &tmap_wd, full_bar(s), tl.n0 + 64, b_row0 + ks * KS);
            if (++s == kStages) { s = 0; ph ^= 1u; }
          }
        }
      }
      if (!ok) {
        // the copies this thread issued land (or time out) before the CTA goes away
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
      constexpr int kPerBox = kBK / kUmmaK;
      int s = 0, buf = 0;
      uint32_t ph = 0, acc_ph = 0;
      bool ok = true, issued_any = false;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const int k_steps = u < total_gu ? ks_gu : ks_dn;
        if (!wait_bounded(tempty_bar(buf), acc_ph ^ 1u, abort_flag, args.dev_status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kN);
        for (int ks = 0; ks < k_steps; ++ks) {
          if (!wait_bounded(full_bar(s), ph, abort_flag, args.dev_status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = smem_u32(stage_base + s * G::kStageBytes);
#pragma unroll
          for (int kk = 0; kk < KS / kUmmaK; ++kk) {
            const uint64_t bd = smem_desc_sw128(st + G::kBOff + kk * kUmmaK * 128, G::kAtom, 1024);
            const uint64_t ad = smem_desc_sw128(
                st + (kk / kPerBox) * G::kABoxSlot + (kk % kPerBox) * kUmmaK * 2, 16, 1024);
            mma_bf16(d_tmem, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
          }
          issued_any = true;
          mma_commit(empty_bar(s));
          if (++s == kStages) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(tfull_bar(buf));
        if (++buf == 2) { buf = 0; acc_ph ^= 1u; }
      }
      if (!ok && issued_any) {
        mma_commit(drain_bar);
        wait_drain(drain_bar, 0);
      }
    }
  } else {
    // =========== epilogue (warps 2..5): H with SwiGLU, or y; then the count ===========
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    int buf = 0;
    uint32_t acc_ph = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const Tile tl = unit_tile(u);
      const bool gu = u < total_gu;
      if (!__all_sync(0xFFFFFFFFu, wait_bounded(tfull_bar(buf), acc_ph, abort_flag, args.dev_status)))
        break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(buf * kN);
      const bool live = r < tl.rows;
      const int row = tl.row0 + (live ? r : 0);
      if (gu)
        epilogue_row<64, true>(taddr, live, args.out + static_cast<int64_t>(row) * I + tl.n0);
      else
        epilogue_row<128, false>(taddr, live, y + static_cast<int64_t>(row) * d + tl.n0);
      tc_fence_before();
      mbar_arrive(tempty_bar(buf));
      if (++buf == 2) { buf = 0; acc_ph ^= 1u; }
      // each epilogue warp counts its own quarter of the tile once its lanes' stores
      // are visible GPU-wide (no barrier across the warps: a warp that leaves the loop
      // on an abort holds up no other)
      __threadfence();
      __syncwarp();
      if (lane == 0) {
        if (gu) {
          red_release_gpu_add(sync + tl.seg, 1);
        } else {
          const int m_blocks = (sm.s_count[tl.seg] + args.bm - 1) / args.bm;
          if (atomicAdd(sync + n_seg + tl.seg, 1) == 4 * m_blocks * nb_dn - 1) {
            // the expert's last down count: every down tile of the expert has passed
            // its wait, so both counts return to zero for the next launch
            sync[tl.seg] = 0;
            sync[n_seg + tl.seg] = 0;
          }
        }
      }
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

// ------------------------------ host side ----------------------------------

// 2-D tensor [rows, cols] (cols contiguous) with a box of [box_rows, 64]
// elements: bf16 with 128-byte swizzle, or (fp8) bytes with 64-byte swizzle.
// An encoded map depends only on (address, rows, cols, box rows, element type),
// so encodings are kept in a small cache keyed by exactly those values: a hit is
// always a valid map, whatever the caller did with the memory in between.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
              bool fp8 = false) {
  struct Entry {
    const void* base;
    uint64_t rows, cols;
    uint32_t box_rows;
    bool fp8;
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
      if (e.base == base && e.rows == rows && e.cols == cols && e.box_rows == box_rows &&
          e.fp8 == fp8) {
        *m = e.map;
        return true;
      }
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (fp8 ? 1 : 2)};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         fp8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(mu);
  Entry& e = cache[next];
  e = Entry{base, rows, cols, box_rows, fp8, *m};
  next = (next + 1) % kCache;
  if (used < kCache) ++used;
  return true;
}

// SM count of the current device, read once per device (each entry is written
// with the same value by whichever host thread gets there first).
int num_sms() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev] = {};
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDev) {
    n = cache[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  n = n > 0 ? n : 1;
  if (dev >= 0 && dev < kMaxDev) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int N_ATOMS, bool SWIGLU, bool FP8A = false, bool SMALLA = false, int KS = kBK>
moe_status launch_gemm_shape(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                             const GemmArgs& args, cudaStream_t s) {
  using G = Geometry<N_ATOMS, FP8A, SMALLA, KS>;
  auto kern = grouped_gemm_kernel<N_ATOMS, SWIGLU, FP8A, SMALLA, KS>;
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
  launch(kern, dim3(n_sm), dim3(G::kThreads), G::kSmemBytes, s, a, b0, b1, args);
  return launch_status();
}

// Single-CTA launch: the small-A slot layout (deeper pipeline) when the row
// boxes hold at most 32 rows, the A operand is bf16 and a stage (at least two B
// atoms) covers the 128 rows the MMA reads; with `deep` (weight maps of 128-row
// boxes, see deep_stages; two B atoms per stage only) its stages take 128 K each.
template <int N_ATOMS, bool SWIGLU, bool FP8A = false>
moe_status launch_gemm(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                       const GemmArgs& args, cudaStream_t s, bool deep = false) {
  if constexpr (!FP8A && N_ATOMS == 2) {
    if (deep) return launch_gemm_shape<N_ATOMS, SWIGLU, false, true, 2 * kBK>(a, b0, b1, args, s);
  }
  if (deep) return MOE_ERR_UNSUPPORTED;  // maps of 128-row boxes need the deep kernel
  if constexpr (!FP8A && N_ATOMS >= 2) {
    if (args.bm <= 32) return launch_gemm_shape<N_ATOMS, SWIGLU, false, true>(a, b0, b1, args, s);
  }
  return launch_gemm_shape<N_ATOMS, SWIGLU, FP8A, false>(a, b0, b1, args, s);
}

// The pair kernel runs as many two-CTA clusters as can be resident at once
// (queried once per device), each looping over its share of the tiles.
template <bool SWIGLU, bool FP8A = false>
moe_status launch_gemm_pair(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                            const GemmArgs& args, cudaStream_t s) {
  using PG = PairGeometry<FP8A>;
  auto kern = grouped_gemm_pair_kernel<SWIGLU, FP8A>;
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
                               PG::kSmemBytes) != cudaSuccess)
        return MOE_ERR_CUDA;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(num_sms() & ~1));
      cfg.blockDim = dim3(PG::kThreads);
      cfg.dynamicSmemBytes = PG::kSmemBytes;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0)
        clusters = num_sms() / 2;
      cudaGetLastError();
      grid[dev] = 2 * clusters;
    }
    g = grid[dev];
  }
  launch(kern, dim3(g), dim3(PG::kThreads), PG::kSmemBytes, s, a, b0, b1, args);
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

// Rows per single-CTA tile.  Decode-sized batches leave most of a 128-row A box
// empty (one token touches k experts with one row each), and staging it costs
// L2 traffic and TMA time beside the weights being streamed: the box height
// follows four times the average rows per segment, at least 16.
int choose_bm(int32_t n_seg, int32_t max_rows) {
  const int64_t four_avg = 4 * static_cast<int64_t>(max_rows) / (n_seg > 0 ? n_seg : 1);
  return four_avg <= 16 ? 16 : four_avg <= 32 ? 32 : four_avg <= 64 ? 64 : kBM;
}

// Single-CTA tile width: the wide tiles (gate/up 2 x 128 columns, down 256) or
// the narrow ones (half as wide), whichever leaves the busiest CTA less to do.
// With at most min(n_seg, max_rows) experts holding rows and wide_blocks wide
// tiles per expert, the wide tiles take ceil(n / SMs) rounds per CTA and the
// narrow ones ceil(2n / SMs) rounds of about 0.6 of a wide tile's time (half the
// columns with the same per-tile start-up).  Measured on decode (E = 128, top-8,
// d = 2048, I = 768), narrow against wide, µs per step: gate/up T = 1 narrow
// (the pass 18.4 against 20.5), T = 2 wide (43.7 against 47.7), T = 4 narrow
// (64.2 against 66.2), T >= 8 wide (T = 128: 182.7 against 187.5); down T = 1
// narrow (37.5 against 38.6), T = 2 wide (51.8 against 53.3).
bool wide_tiles(int32_t n_seg, int32_t max_rows, int64_t wide_blocks) {
  const int sms = num_sms();
  const int64_t touched = n_seg < max_rows ? n_seg : max_rows;
  const int64_t n_wide = touched * wide_blocks;
  const int64_t rounds_wide = ceil_div(n_wide, sms), rounds_narrow = ceil_div(2 * n_wide, sms);
  return 10 * rounds_wide <= 6 * rounds_narrow;
}

bool wide_gate_up(int32_t n_seg, int32_t max_rows, int32_t I) {
  return I % 128 == 0 && wide_tiles(n_seg, max_rows, I / 128);
}

// Deep stages (128 K per stage, weight boxes of 128 rows) for the small-A
// single-CTA kernel with two B atoms per stage (the narrow tiles): bf16 rows staged
// by tile loads (not gathered) and K a multiple of 128.  (With four atoms a deep
// stage is 72 KB and only two fit the shared memory.)
bool deep_stages(bool pair, int bm, bool gathered, int32_t K, bool narrow) {
  return !pair && bm <= 32 && !gathered && K % (2 * kBK) == 0 && narrow;
}

bool pair_shape(int32_t n_seg, int32_t max_rows) {
  return static_cast<int64_t>(max_rows) >= static_cast<int64_t>(kBM) * n_seg;
}

// One warp; lane 0 waits, with the pipelines' bounded wait, on a barrier whose
// phase never completes (nothing arrives), so the wait gives up after limit_ns.
__global__ void __launch_bounds__(32) wait_timeout_selftest(uint64_t limit_ns, uint32_t* dev_status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  if (threadIdx.x == 0) wait_bounded(smem_u32(&bar), 0, &abort_flag, dev_status, limit_ns);
  __syncwarp();
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

// The bf16 gate/up pass.  With gather == nullptr the A rows are rows [0, max_rows)
// of x; otherwise row i is x[gather[i] / k] of the token rows x [T, d].
static moe_status gate_up_impl(int32_t n_seg, int32_t d, int32_t I, int32_t max_rows,
                               const moe_bf16* x, int32_t T, int32_t k, const int32_t* gather,
                               const int32_t* seg_begin, const int32_t* seg_count,
                               const moe_bf16* w_gate, const moe_bf16* w_up, moe_bf16* h,
                               uint32_t* dev_status, moe_stream_t stream) {
  const bool pair = I % 128 == 0 && pair_shape(n_seg, max_rows);
  const int bm = pair ? kBM : choose_bm(n_seg, max_rows);
  CUtensorMap m_x, m_wg, m_wu;
  const bool wide = !pair && wide_gate_up(n_seg, max_rows, I);
  const bool deep = deep_stages(pair, bm, gather != nullptr, d, !wide);
  const uint32_t b_rows = deep ? 2 * kBK : kBK;
  const bool x_ok = gather == nullptr ? make_map(&m_x, x, max_rows, d, bm)
                                      : make_map(&m_x, x, T, d, 1);  // one-row boxes
  if (!x_ok || !make_map(&m_wg, w_gate, int64_t(n_seg) * d, I, b_rows) ||
      !make_map(&m_wu, w_up, int64_t(n_seg) * d, I, b_rows))
    return MOE_ERR_CUDA;
  GemmArgs a{seg_begin, seg_count, n_seg, d, I, max_rows, reinterpret_cast<uint16_t*>(h),
             dev_status, choose_m_outer(n_seg, max_rows, d, 2 * static_cast<int64_t>(I)),
             nullptr, 0, 0, bm, bm * kBK * 2, gather, k, T};
  cudaStream_t s = as_cuda(stream);
  if (pair) return launch_gemm_pair<true>(m_x, m_wg, m_wu, a, s);
  if (wide) return launch_gemm<4, true>(m_x, m_wg, m_wu, a, s);
  return launch_gemm<2, true>(m_x, m_wg, m_wu, a, s, deep);
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
  return gate_up_impl(n_seg, d, I, max_rows, x, 0, 1, nullptr, seg_begin, seg_count, w_gate,
                      w_up, h, dev_status, stream);
}

MOE_API moe_status moe_grouped_gate_up_gather(int32_t n_seg, int32_t d, int32_t I,
                                              int32_t max_rows, int32_t T, int32_t k,
                                              const moe_bf16* x, const int32_t* row_to_route,
                                              const int32_t* seg_begin, const int32_t* seg_count,
                                              const moe_bf16* w_gate, const moe_bf16* w_up,
                                              moe_bf16* h, uint32_t* dev_status,
                                              moe_stream_t stream) {
  moe_status st = check_common(n_seg, d, I, max_rows);
  if (st != MOE_OK) return st;
  if (T < 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  if (max_rows == 0) return MOE_OK;
  if (T == 0 || x == nullptr || row_to_route == nullptr || seg_begin == nullptr ||
      seg_count == nullptr || w_gate == nullptr || w_up == nullptr || h == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(h) || !aligned16(w_gate) || !aligned16(w_up))
    return MOE_ERR_UNSUPPORTED;
  return gate_up_impl(n_seg, d, I, max_rows, x, T, k, row_to_route, seg_begin, seg_count, w_gate,
                      w_up, h, dev_status, stream);
}

MOE_API moe_status moe_grouped_gate_up_fp8(int32_t n_seg, int32_t d, int32_t I, int32_t max_rows,
                                           int32_t group, const moe_fp8* xq, const float* scales,
                                           const int32_t* seg_begin, const int32_t* seg_count,
                                           const moe_bf16* w_gate, const moe_bf16* w_up,
                                           moe_bf16* h, uint32_t* dev_status,
                                           moe_stream_t stream) {
  moe_status st = check_common(n_seg, d, I, max_rows);
  if (st != MOE_OK) return st;
  if (group != MOE_SCALE_ROW && group != MOE_SCALE_BLOCK128) return MOE_ERR_INVALID_ARG;
  if (max_rows == 0) return MOE_OK;
  if (xq == nullptr || scales == nullptr || seg_begin == nullptr || seg_count == nullptr ||
      w_gate == nullptr || w_up == nullptr || h == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(xq) || !aligned16(h) || !aligned16(w_gate) || !aligned16(w_up) ||
      (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
    return MOE_ERR_UNSUPPORTED;
  // the same kernel shapes and tile heights as the bf16 operand
  const bool pair = I % 128 == 0 && pair_shape(n_seg, max_rows);
  const int bm = pair ? kBM : choose_bm(n_seg, max_rows);
  CUtensorMap m_x, m_wg, m_wu;
  if (!make_map(&m_x, xq, max_rows, d, bm, true) ||
      !make_map(&m_wg, w_gate, int64_t(n_seg) * d, I, kBK) ||
      !make_map(&m_wu, w_up, int64_t(n_seg) * d, I, kBK))
    return MOE_ERR_CUDA;
  const int n_groups = group == MOE_SCALE_ROW ? 1 : static_cast<int>(ceil_div(d, 128));
  GemmArgs a{seg_begin, seg_count, n_seg, d, I, max_rows, reinterpret_cast<uint16_t*>(h),
             dev_status, choose_m_outer(n_seg, max_rows, d, 2 * static_cast<int64_t>(I)),
             scales, n_groups, group == MOE_SCALE_ROW ? d : 128, bm, bm * kBK};
  cudaStream_t s = as_cuda(stream);
  if (pair) return launch_gemm_pair<true, true>(m_x, m_wg, m_wu, a, s);
  if (wide_gate_up(n_seg, max_rows, I)) return launch_gemm<4, true, true>(m_x, m_wg, m_wu, a, s);
  return launch_gemm<2, true, true>(m_x, m_wg, m_wu, a, s);
}

static moe_status down_impl(int32_t n_seg, int32_t I, int32_t d, int32_t max_rows,
                            const moe_bf16* h, const int32_t* seg_begin, const int32_t* seg_count,
                            const moe_bf16* w_down, moe_bf16* y, uint32_t* dev_status,
                            moe_stream_t stream, int chained) {
  moe_status st = check_common(n_seg, I, d, max_rows);
  if (st != MOE_OK || max_rows == 0) return st;
  if (h == nullptr || seg_begin == nullptr || seg_count == nullptr || w_down == nullptr ||
      y == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(y) || !aligned16(w_down)) return MOE_ERR_UNSUPPORTED;
  const bool pair = d % 256 == 0 && pair_shape(n_seg, max_rows);
  const int bm = pair ? kBM : choose_bm(n_seg, max_rows);
  const bool wide = !pair && d % 256 == 0 && wide_tiles(n_seg, max_rows, d / 256);
  const bool deep = deep_stages(pair, bm, false, I, !wide && d % 128 == 0);
  CUtensorMap m_h, m_wd;
  if (!make_map(&m_h, h, max_rows, I, bm) ||
      !make_map(&m_wd, w_down, int64_t(n_seg) * I, d, deep ? 2 * kBK : kBK))
    return MOE_ERR_CUDA;
  GemmArgs a{seg_begin, seg_count, n_seg, I, d, max_rows, reinterpret_cast<uint16_t*>(y),
             dev_status, choose_m_outer(n_seg, max_rows, I, d), nullptr, 0, 0, bm, bm * kBK * 2,
             nullptr, 0, 0, chained};
  cudaStream_t s = as_cuda(stream);
  if (pair) return launch_gemm_pair<false>(m_h, m_wd, m_wd, a, s);
  if (wide) return launch_gemm<4, false>(m_h, m_wd, m_wd, a, s);
  if (d % 128 == 0) return launch_gemm<2, false>(m_h, m_wd, m_wd, a, s, deep);
  return launch_gemm<1, false>(m_h, m_wd, m_wd, a, s);
}

MOE_API moe_status moe_grouped_down(int32_t n_seg, int32_t I, int32_t d, int32_t max_rows,
                                    const moe_bf16* h, const int32_t* seg_begin,
                                    const int32_t* seg_count, const moe_bf16* w_down, moe_bf16* y,
                                    uint32_t* dev_status, moe_stream_t stream) {
  return down_impl(n_seg, I, d, max_rows, h, seg_begin, seg_count, w_down, y, dev_status, stream,
                   0);
}

MOE_API moe_status moe_grouped_down_chained(int32_t n_seg, int32_t I, int32_t d, int32_t max_rows,
                                            const moe_bf16* h, const int32_t* seg_begin,
                                            const int32_t* seg_count, const moe_bf16* w_down,
                                            moe_bf16* y, uint32_t* dev_status,
                                            moe_stream_t stream) {
  return down_impl(n_seg, I, d, max_rows, h, seg_begin, seg_count, w_down, y, dev_status, stream,
                   1);
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
  return moe_grouped_down_chained(n_seg, I, d, max_rows, h, seg_begin, seg_count, w_down, y,
                                  dev_status, stream);
}

// Whether moe_grouped_swiglu_onepass runs as one launch: the row boxes hold at most 32
// rows, d and I are multiples of 128, and the two-launch gate/up pass would take the
// narrow tiles too (measured on the decode shape, µs per step, two launches against one:
// T = 1 33.84 against 32.73, T = 4 61.05 against 59.0; where the gate/up pass takes the
// wide tiles the one launch, narrow only, lost: T = 2 42.7 against 45.9, T = 8 77.8
// against 78.6).
static bool onepass_taken(int32_t n_seg, int32_t d, int32_t I, int32_t max_rows) {
  if (n_seg <= 0 || max_rows <= 0 || pair_shape(n_seg, max_rows)) return false;
  return choose_bm(n_seg, max_rows) <= 32 && d % (2 * kBK) == 0 && I % (2 * kBK) == 0 &&
         !wide_gate_up(n_seg, max_rows, I);
}

MOE_API int32_t moe_grouped_swiglu_onepass_taken(int32_t n_seg, int32_t d, int32_t I,
                                                 int32_t max_rows) {
  return onepass_taken(n_seg, d, I, max_rows) ? 1 : 0;
}

// One launch for both passes when onepass_taken; the two launches otherwise.
MOE_API moe_status moe_grouped_swiglu_onepass(int32_t n_seg, int32_t d, int32_t I,
                                              int32_t max_rows, const moe_bf16* x,
                                              const int32_t* seg_begin, const int32_t* seg_count,
                                              const moe_bf16* w_gate, const moe_bf16* w_up,
                                              const moe_bf16* w_down, moe_bf16* h, moe_bf16* y,
                                              int32_t* sync, uint32_t* dev_status,
                                              moe_stream_t stream) {
  moe_status st = check_common(n_seg, d, I, max_rows);
  if (st == MOE_OK) st = check_common(n_seg, I, d, max_rows);
  if (st != MOE_OK || max_rows == 0) return st;
  if (x == nullptr || seg_begin == nullptr || seg_count == nullptr || w_gate == nullptr ||
      w_up == nullptr || w_down == nullptr || h == nullptr || y == nullptr || sync == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(h) || !aligned16(y) || !aligned16(w_gate) ||
      !aligned16(w_up) || !aligned16(w_down) || (reinterpret_cast<uintptr_t>(sync) & 3u) != 0)
    return MOE_ERR_UNSUPPORTED;
  const int bm = choose_bm(n_seg, max_rows);
  if (!onepass_taken(n_seg, d, I, max_rows)) {
    st = moe_grouped_gate_up(n_seg, d, I, max_rows, x, seg_begin, seg_count, w_gate, w_up, h,
                             dev_status, stream);
    if (st != MOE_OK) return st;
    return moe_grouped_down_chained(n_seg, I, d, max_rows, h, seg_begin, seg_count, w_down, y,
                                    dev_status, stream);
  }
  using G = Geometry<2, false, true, 2 * kBK>;
  CUtensorMap m_x, m_wg, m_wu, m_h, m_wd;
  if (!make_map(&m_x, x, max_rows, d, bm) ||
      !make_map(&m_wg, w_gate, int64_t(n_seg) * d, I, 2 * kBK) ||
      !make_map(&m_wu, w_up, int64_t(n_seg) * d, I, 2 * kBK) ||
      !make_map(&m_h, h, max_rows, I, bm) ||
      !make_map(&m_wd, w_down, int64_t(n_seg) * I, d, 2 * kBK))
    return MOE_ERR_CUDA;
  GemmArgs a{seg_begin, seg_count, n_seg, d, I, max_rows, reinterpret_cast<uint16_t*>(h),
             dev_status, 0, nullptr, 0, 0, bm, bm * kBK * 2, nullptr, 0, 0, 0};
  constexpr int kMaxDev = 64;
  static std::atomic<int> ready[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MOE_ERR_CUDA;
  if (!ready[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(grouped_swiglu_onepass_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes) != cudaSuccess)
      return MOE_ERR_CUDA;
    ready[dev].store(1, std::memory_order_relaxed);
  }
  launch(grouped_swiglu_onepass_kernel, dim3(num_sms()), dim3(G::kThreads), G::kSmemBytes,
         as_cuda(stream), m_x, m_wg, m_wu, m_h, m_wd, a, reinterpret_cast<uint16_t*>(y), sync);
  return launch_status();
}

MOE_API moe_status moe_debug_wait_timeout(int64_t limit_ns, uint32_t* dev_status,
                                          moe_stream_t stream) {
  if (dev_status == nullptr || limit_ns < 1 || limit_ns > 1000000000ll) return MOE_ERR_INVALID_ARG;
  wait_timeout_selftest<<<1, 32, 0, as_cuda(stream)>>>(static_cast<uint64_t>(limit_ns), dev_status);
  return launch_status();
}
