// Permute: capacity admission, per-expert count, exclusive prefix, stable
// expert-major scatter of route ids with the exact inverse map, and the bf16
// row gather x_perm[row] = x[token].
//
// [M6.2] 0x03B "Count, Prefix, Permute": c_e, o_{e+1} = o_e + c_e, pi = stable
// order by (expert, route id), inverse pi^-1[pi[j]] = j.  [M6.6] 0x03B: the
// sentinel offset o_E is part of the contract.  Admission (which routes an
// expert of capacity C keeps) takes routes in route id order.
//
// Three launches, no host synchronisation and no inter-block waiting:
//   1. permute_hist  one block per tile of consecutive routes (at most 128
//                    tiles): per-tile expert histogram -> ws hist[tile][E].
//                    Skipped when there is a single tile: its block counts itself.
//   2. permute_rank  one block per tile.  Each block reads the whole (small)
//                    histogram matrix with independent loads to get its tile's
//                    first ordinal per expert and every expert's total, hence
//                    the admitted counts and the offsets (block 0 writes them);
//                    then stable in-tile ranks (warp sub-ranges in route order,
//                    __match_any_sync + popc within 32 routes) give each route
//                    its ordinal, its row and both maps.
//   3. permute_copy  token-major row copy over many blocks: every token row is
//                    read once and written to its admitted rows with 16-byte
//                    accesses.  Skipped when the caller wants the maps only (the
//                    gate/up pass can gather the rows itself).  With at most 16
//                    routes (one or two tokens at top-8) the rank block copies
//                    the rows itself after ranking, and this launch is left out
//                    (one-token decode 36.9 -> 35.7 us per step; at 32 or 64
//                    routes one block copying was slower than the copy kernel).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kHistThreads = 256;
constexpr int kRankThreads = 512;  // one thread per expert (E <= 512)
constexpr int kRankWarps = kRankThreads / 32;
constexpr int kMinTileRoutes = 2048;
constexpr int kMaxTiles = 128;
constexpr int kCopyThreads = 256;

// Routes of the first min(*valid, T) tokens (all T*k routes without a valid count).
__device__ __forceinline__ int valid_routes(int R, int k, const int32_t* __restrict__ valid) {
  if (valid == nullptr) return R;
  const int v = __ldg(valid);
  return v <= 0 ? 0 : min(R, v * k);
}

struct PermTiling {
  int routes_per_tile;
  int n_tiles;
};

// Routes up to which the rank block also copies the rows (a single tile).
constexpr int kFusedCopyRoutes = 16;
inline bool fuse_row_copy(int64_t R) { return R <= kFusedCopyRoutes; }

PermTiling permute_tiling(int64_t R) {
  PermTiling p;
  int64_t rpt = ceil_div(R, kMaxTiles);
  if (rpt < kMinTileRoutes) rpt = kMinTileRoutes;
  p.routes_per_tile = static_cast<int>(rpt);
  p.n_tiles = R > 0 ? static_cast<int>(ceil_div(R, rpt)) : 0;
  return p;
}

__global__ void __launch_bounds__(kHistThreads)
permute_hist(int R, int E, int k, int routes_per_tile, const int32_t* __restrict__ ids,
             int32_t* __restrict__ hist, uint32_t* __restrict__ dev_status,
             const int32_t* __restrict__ valid, bool early) {
  extern __shared__ int32_t sh[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  pdl_wait_then_trigger(early);
  __syncthreads();
  const int R_live = valid_routes(R, k, valid);
  const int r0 = blockIdx.x * routes_per_tile;
  const int r1 = min(R_live, r0 + routes_per_tile);
  bool bad = false;
  for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    const int e = __ldg(ids + r);
    if (e >= 0 && e < E) atomicAdd(&sh[e], 1); else bad = true;
  }
  if (bad) report(dev_status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  int32_t* out = hist + static_cast<int64_t>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) out[e] = sh[e];
  if (!early) pdl_trigger();
}

__global__ void __launch_bounds__(kRankThreads)
permute_rank(int R, int E, int k, int routes_per_tile, int n_tiles, int capacity,
             const int32_t* __restrict__ ids, const int32_t* __restrict__ hist,
             int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
             int32_t* __restrict__ n_dropped, int32_t* __restrict__ row_to_route,
             int32_t* __restrict__ route_to_row, uint32_t* __restrict__ dev_status,
             const int32_t* __restrict__ valid, bool early, const uint4* __restrict__ x,
             uint4* __restrict__ x_perm, int chunks, int G, const float* __restrict__ scales,
             float* __restrict__ scales_perm) {
  extern __shared__ int32_t sh[];
  int32_t* cnt = sh;                    // [kRankWarps][E]
  int32_t* off = cnt + kRankWarps * E;  // [E]
  __shared__ int32_t warp_tot[kRankWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int tile = blockIdx.x;

  for (int i = threadIdx.x; i < kRankWarps * E; i += blockDim.x) cnt[i] = 0;
  if (x_perm != nullptr) {
    // the block copies the token rows itself (a handful of tokens): they do not
    // depend on the routes, so their first read from HBM overlaps the router
    const char* xb = reinterpret_cast<const char*>(x);
    const int64_t bytes = static_cast<int64_t>(R / k) * chunks * 16;
    for (int64_t o = static_cast<int64_t>(threadIdx.x) * 128; o < bytes; o += 128 * kRankThreads)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(xb + o));
  }
  pdl_wait_then_trigger(early);
  __syncthreads();
  // Routes at or past R_live belong to masked padding tokens of a fixed bucket:
  // they are neither counted, admitted nor dropped, and map to row -1.
  const int R_live = valid_routes(R, k, valid);
  const int r0 = tile * routes_per_tile;
  const int r1 = min(R_live, r0 + routes_per_tile);
  const int sub = (max(r1 - r0, 0) + kRankWarps - 1) / kRankWarps;
  const int s0 = r0 + w * sub, s1 = min(r1, s0 + sub);
  for (int r = max(r0, R_live) + threadIdx.x; r < min(R, r0 + routes_per_tile); r += blockDim.x)
    route_to_row[r] = -1;
  // per-warp expert counts of the warp's contiguous sub-range
  for (int r = s0 + lane; r < s1; r += 32) {
    const int ee = __ldg(ids + r);
    if (ee >= 0 && ee < E) atomicAdd(&cnt[w * E + ee], 1);
  }
  __syncthreads();
  // 1. this tile's first ordinal per expert, every expert's total, admitted counts
  //    (from the histogram of all tiles, or, with no histogram (hist == nullptr,
  //    a single tile), from this block's own counts)
  const int e = threadIdx.x;
  int32_t base = 0, total = 0;
  if (e < E && hist == nullptr) {
    for (int ww = 0; ww < kRankWarps; ++ww) total += cnt[ww * E + e];
  } else if (e < E) {
    int t = 0;
    for (; t + 8 <= n_tiles; t += 8) {
      int32_t v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __ldg(hist + static_cast<int64_t>(t + i) * E + e);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        base += (t + i < tile) ? v[i] : 0;
        total += v[i];
      }
    }
    for (; t < n_tiles; ++t) {
      const int32_t v = __ldg(hist + static_cast<int64_t>(t) * E + e);
      base += (t < tile) ? v : 0;
      total += v;
    }
  }
  const int32_t c = (e < E) ? (capacity < 0 ? total : min(total, capacity)) : 0;
  // 2. offsets: block-wide exclusive scan of the admitted counts
  int32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  int32_t before = 0;
  for (int i = 0; i < w; ++i) before += warp_tot[i];
  if (e < E) {
    off[e] = before + incl - c;
    if (tile == 0) {
      counts[e] = c;
      offsets[e] = before + incl - c;
      if (e == E - 1) {
        offsets[E] = before + incl;
        *n_dropped = R_live - (before + incl);
      }
    }
  }
  // 3. each warp's first ordinal per expert: tile base + earlier warps
  if (e < E) {
    int32_t run = base;
    for (int ww = 0; ww < kRankWarps; ++ww) {
      const int32_t v = cnt[ww * E + e];
      cnt[ww * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  // 4. stable ranks, 32 routes at a time in route order
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int c0 = s0; c0 < s1; c0 += 32) {
    const int r = c0 + lane;
    int ee = -1;
    if (r < s1) {
      ee = __ldg(ids + r);
      if (ee < 0 || ee >= E) {  // invalid id: its own group, never admitted
        ee = -2;
        if (hist == nullptr) report(dev_status, MOE_DEV_BAD_EXPERT_ID);
      }
    }
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, ee);
    int32_t ordinal = 0;
    if (ee >= 0) ordinal = cnt[w * E + ee] + __popc(peers & lt_mask);
    __syncwarp();
    if (ee >= 0 && (peers & lt_mask) == 0) cnt[w * E + ee] += __popc(peers);
    __syncwarp();
    if (r < s1) {
      int32_t row = -1;
      if (ee >= 0 && (capacity < 0 || ordinal < capacity)) {
        row = off[ee] + ordinal;
        row_to_route[row] = r;
      }
      route_to_row[r] = row;
    }
  }
  if (x_perm != nullptr) {
    // 5. the row copy, in this block when every route is in this one tile and there
    //    are few (a handful of tokens): one warp per admitted row, whose route this
    //    block has just written (visible to the block after the barrier)
    __syncthreads();
    int32_t n_rows = 0;
    for (int i = 0; i < kRankWarps; ++i) n_rows += warp_tot[i];
    for (int row = w; row < n_rows; row += kRankWarps) {
      const int t = row_to_route[row] / k;
      const uint4* src = x + static_cast<int64_t>(t) * chunks;
      uint4* dst = x_perm + static_cast<int64_t>(row) * chunks;
      for (int c = lane; c < chunks; c += 32) dst[c] = __ldg(src + c);
      for (int g = lane; g < G; g += 32)
        scales_perm[static_cast<int64_t>(row) * G + g] = __ldg(scales + static_cast<int64_t>(t) * G + g);
    }
  }
  if (!early) pdl_trigger();
}

// One warp per (token, column part): read the part of the row once, store it to
// each admitted row (and, with SCALES, part 0 copies the row's G fp32 scales to
// the same rows of scales_perm).  `parts` > 1 splits rows into column ranges
// when there are too few tokens to give every SM work (decode).
template <bool SCALES>
__global__ void __launch_bounds__(kCopyThreads)
permute_copy(int T, int k, int chunks, int parts, const int32_t* __restrict__ route_to_row,
             const uint4* __restrict__ x, uint4* __restrict__ x_perm,
             const int32_t* __restrict__ valid, int G, const float* __restrict__ scales,
             float* __restrict__ scales_perm, bool early) {
  pdl_wait_then_trigger(early);
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int T_live = valid_routes(T, 1, valid);
  const int per = (chunks + parts - 1) / parts;
  const int64_t units = static_cast<int64_t>(T_live) * parts;
  for (int64_t u0 = static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5); u0 < units;
       u0 += static_cast<int64_t>(gridDim.x) * warps) {
    const int t = static_cast<int>(u0 / parts), part = static_cast<int>(u0 % parts);
    const int c_lo = part * per, c_hi = min(chunks, c_lo + per);
    const int32_t my_row = lane < k ? __ldg(route_to_row + static_cast<int64_t>(t) * k + lane) : -1;
    const uint4* src = x + static_cast<int64_t>(t) * chunks;
    // The chunk loop runs uniformly over the warp (lanes past the range end only
    // skip their accesses) because its body broadcasts rows with __shfl_sync.
    for (int cb = c_lo; cb < c_hi; cb += 32 * 4) {
      const int c = cb + lane;
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + 32 * u < c_hi) v[u] = __ldg(src + c + 32 * u);
      for (int j = 0; j < k; ++j) {
        const int32_t row = __shfl_sync(0xFFFFFFFFu, my_row, j);
        if (row < 0) continue;
        uint4* dst = x_perm + static_cast<int64_t>(row) * chunks;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (c + 32 * u < c_hi) dst[c + 32 * u] = v[u];
      }
    }
    if constexpr (SCALES) {
      if (part != 0) continue;
      const float* src_s = scales + static_cast<int64_t>(t) * G;
      for (int j = 0; j < k; ++j) {
        const int32_t row = __shfl_sync(0xFFFFFFFFu, my_row, j);
        if (row < 0) continue;
        for (int g = lane; g < G; g += 32)
          scales_perm[static_cast<int64_t>(row) * G + g] = __ldg(src_s + g);
      }
    }
  }
  if (!early) pdl_trigger();
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API size_t moe_permute_workspace_size(int32_t T, int32_t k, int32_t E) {
  if (T <= 0 || k <= 0 || E <= 0) return 256;
  const PermTiling tl = permute_tiling(static_cast<int64_t>(T) * k);
  Carver c;
  c.take<int32_t>(static_cast<size_t>(tl.n_tiles) * E);
  return c.off + 256;
}

// Payload rows are row_bytes long (a multiple of 16); with scales != nullptr each
// row also carries G fp32 scales, copied to the same rows of scales_perm.
static moe_status permute_impl(int32_t T, int64_t row_bytes, int32_t E, int32_t k,
                               int32_t capacity, const int32_t* valid, const int32_t* topk_ids,
                               const void* x, void* x_perm, int32_t G, const float* scales,
                               float* scales_perm, int32_t* counts, int32_t* offsets,
                               int32_t* row_to_route, int32_t* route_to_row, int32_t* n_dropped,
                               void* ws, size_t ws_bytes, uint32_t* dev_status,
                               moe_stream_t stream) {
  if (T < 0 || row_bytes <= 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > 512 || k > 16 || row_bytes % 16 != 0 || row_bytes > (int64_t(1) << 24) ||
      static_cast<int64_t>(T) * k >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  if (T > 0 && G > 0 && (scales == nullptr || scales_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if (counts == nullptr || offsets == nullptr || n_dropped == nullptr) return MOE_ERR_INVALID_ARG;
  // x and x_perm both NULL (no scales): the maps only, no row copy
  const bool maps_only = x == nullptr && x_perm == nullptr && G == 0;
  if (T > 0 && (topk_ids == nullptr || row_to_route == nullptr || route_to_row == nullptr ||
                ws == nullptr || (!maps_only && (x == nullptr || x_perm == nullptr))))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && !maps_only && (!aligned16(x) || !aligned16(x_perm))) return MOE_ERR_UNSUPPORTED;
  if (ws_bytes < moe_permute_workspace_size(T, k, E)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = as_cuda(stream);
  const int R = T * k;
  const PermTiling tl = permute_tiling(R);
  int32_t* hist = static_cast<int32_t*>(ws);
  const size_t rank_smem = (static_cast<size_t>(kRankWarps) * E + E) * sizeof(int32_t);
  if (R == 0) {
    // No routes: one rank block with no tiles writes empty counts and offsets.
    launch(permute_rank, dim3(1), dim3(kRankThreads), rank_smem, s, 0, E, k, 1, 0, capacity,
           topk_ids, static_cast<const int32_t*>(nullptr), counts, offsets, n_dropped,
           row_to_route, route_to_row, dev_status, static_cast<const int32_t*>(nullptr), true,
           static_cast<const uint4*>(nullptr), static_cast<uint4*>(nullptr), 0, 0,
           static_cast<const float*>(nullptr), static_cast<float*>(nullptr));
    return launch_status();
  }
  if (tl.n_tiles > 1)
    launch(permute_hist, dim3(tl.n_tiles), dim3(kHistThreads), E * sizeof(int32_t), s, R, E, k,
           tl.routes_per_tile, topk_ids, hist, dev_status, valid, one_wave(tl.n_tiles));
  const int chunks = static_cast<int>(row_bytes / 16);
  // A handful of tokens: the rank block copies the rows itself (one launch less).
  const bool fused_copy = !maps_only && fuse_row_copy(R);
  launch(permute_rank, dim3(tl.n_tiles), dim3(kRankThreads), rank_smem, s, R, E, k,
         tl.routes_per_tile, tl.n_tiles, capacity, topk_ids,
         static_cast<const int32_t*>(tl.n_tiles > 1 ? hist : nullptr), counts, offsets, n_dropped,
         row_to_route, route_to_row, dev_status, valid, one_wave(tl.n_tiles),
         static_cast<const uint4*>(fused_copy ? x : nullptr),
         static_cast<uint4*>(fused_copy ? x_perm : nullptr), chunks, fused_copy ? G : 0, scales,
         scales_perm);
  if (maps_only || fused_copy) return launch_status();
  const int warps = kCopyThreads / 32;
  // Column parts: enough warps for every SM when tokens are few, at least 64
  // chunks (1 KB) per part.
  int parts = 1;
  while (static_cast<int64_t>(T) * parts * 2 <= 152 * warps && chunks / (parts * 2) >= 64)
    parts *= 2;
  int64_t blocks = ceil_div(static_cast<int64_t>(T) * parts, warps);
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (scales == nullptr)
    launch(permute_copy<false>, dim3(static_cast<unsigned>(blocks)), dim3(kCopyThreads), 0, s, T,
           k, chunks, parts, static_cast<const int32_t*>(route_to_row),
           static_cast<const uint4*>(x), static_cast<uint4*>(x_perm), valid, 0, scales,
           scales_perm, one_wave(blocks));
  else
    launch(permute_copy<true>, dim3(static_cast<unsigned>(blocks)), dim3(kCopyThreads), 0, s, T, k,
           chunks, parts, static_cast<const int32_t*>(route_to_row), static_cast<const uint4*>(x),
           static_cast<uint4*>(x_perm), valid, G, scales, scales_perm, one_wave(blocks));
  return launch_status();
}

MOE_API moe_status moe_permute(int32_t T, int32_t d, int32_t E, int32_t k, int32_t capacity,
                               const int32_t* topk_ids, const moe_bf16* x, moe_bf16* x_perm,
                               int32_t* counts, int32_t* offsets, int32_t* row_to_route,
                               int32_t* route_to_row, int32_t* n_dropped, void* ws,
                               size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream) {
  if (d <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  return permute_impl(T, int64_t(d) * 2, E, k, capacity, nullptr, topk_ids, x, x_perm, 0, nullptr,
                      nullptr, counts, offsets, row_to_route, route_to_row, n_dropped, ws,
                      ws_bytes, dev_status, stream);
}

MOE_API moe_status moe_permute_fp8(int32_t T, int32_t d, int32_t E, int32_t k, int32_t capacity,
                                   int32_t group, const int32_t* topk_ids, const moe_fp8* q,
                                   const float* scales, moe_fp8* q_perm, float* scales_perm,
                                   int32_t* counts, int32_t* offsets, int32_t* row_to_route,
                                   int32_t* route_to_row, int32_t* n_dropped, void* ws,
                                   size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream) {
  if (d <= 0 || (group != MOE_SCALE_ROW && group != MOE_SCALE_BLOCK128)) return MOE_ERR_INVALID_ARG;
  if (d % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && (reinterpret_cast<uintptr_t>(scales) & 3u || reinterpret_cast<uintptr_t>(scales_perm) & 3u))
    return MOE_ERR_UNSUPPORTED;
  const int32_t G = group == MOE_SCALE_ROW ? 1 : static_cast<int32_t>(ceil_div(d, 128));
  return permute_impl(T, d, E, k, capacity, nullptr, topk_ids, q, q_perm, G, scales, scales_perm,
                      counts, offsets, row_to_route, route_to_row, n_dropped, ws, ws_bytes,
                      dev_status, stream);
}

MOE_API moe_status moe_permute_bucket(int32_t T, int32_t d, int32_t E, int32_t k, int32_t capacity,
                                      const int32_t* valid_tokens, const int32_t* topk_ids,
                                      const moe_bf16* x, moe_bf16* x_perm, int32_t* counts,
                                      int32_t* offsets, int32_t* row_to_route,
                                      int32_t* route_to_row, int32_t* n_dropped, void* ws,
                                      size_t ws_bytes, uint32_t* dev_status,
                                      moe_stream_t stream) {
  if (valid_tokens == nullptr || d <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  return permute_impl(T, int64_t(d) * 2, E, k, capacity, valid_tokens, topk_ids, x, x_perm, 0,
                      nullptr, nullptr, counts, offsets, row_to_route, route_to_row, n_dropped, ws,
                      ws_bytes, dev_status, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of moe_permute.
//
// Some callers cannot call cudaMalloc and have no workspace to hand over: for
// example an inference runtime's plugin hook that may only enqueue work on the
// stream it is given, or a latency-critical serving loop where an allocation
// could synchronise the device or break a fixed memory budget.  For them the
// per-tile histogram lives in a fixed file-scope device array instead of a
// caller workspace.  The array is part of the library image: every GPU that
// loads the library holds it until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 10;  // 64 KiB
static __device__ __align__(256) uint8_t g_permute_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device, looked up once per
// device (in host code the array's name is only a host-side stand-in).  The
// cached address lives as long as the process; cudaDeviceReset unloads the module
// on that device, after which the array may be placed elsewhere, so this entry
// point is not for use after a device reset.
moe_status static_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

MOE_API moe_status moe_permute_noalloc(int32_t T, int32_t d, int32_t E, int32_t k,
                                       int32_t capacity, const int32_t* topk_ids,
                                       const moe_bf16* x, moe_bf16* x_perm, int32_t* counts,
                                       int32_t* offsets, int32_t* row_to_route,
                                       int32_t* route_to_row, int32_t* n_dropped,
                                       uint32_t* dev_status, moe_stream_t stream) {
  if (T < 0 || k <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (moe_permute_workspace_size(T, k, E) > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const moe_status st = static_scratch(&scratch);
  if (st != MOE_OK) return st;
  return moe_permute(T, d, E, k, capacity, topk_ids, x, x_perm, counts, offsets, row_to_route,
                     route_to_row, n_dropped, scratch, kStaticScratchBytes, dev_status, stream);
}
