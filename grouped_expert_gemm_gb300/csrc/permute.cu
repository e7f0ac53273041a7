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
//   1. permute_hist   one block per tile of consecutive tokens: per-tile
//                     expert histogram -> ws hist[tile][E]
//   2. permute_scan   one block: per expert an exclusive scan over tiles (the
//                     tile's first ordinal), admitted counts, offsets, drops
//   3. permute_scatter one block per tile: stable in-tile ranks (warp sub-ranges
//                     in order, __match_any_sync + popc within 32 routes),
//                     ordinal -> row, both maps, then a token-major row copy
//                     that reads every token row once and writes its admitted
//                     copies with 16-byte accesses.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kPermThreads = 256;
constexpr int kPermWarps = kPermThreads / 32;
constexpr int kMaxTileRoutes = 4096;

struct PermTiling {
  int tokens_per_tile;
  int n_tiles;
};

PermTiling permute_tiling(int T, int k) {
  PermTiling p;
  // Aim for about two tiles per SM so the row copy fills the GPU.
  int64_t tpt = ceil_div(T, 2 * 152);
  if (tpt < 1) tpt = 1;
  if (tpt * k > kMaxTileRoutes) tpt = kMaxTileRoutes / k;
  p.tokens_per_tile = static_cast<int>(tpt);
  p.n_tiles = static_cast<int>(ceil_div(T, tpt));
  return p;
}

__global__ void __launch_bounds__(kPermThreads)
permute_hist(int R, int E, int routes_per_tile, const int32_t* __restrict__ ids,
             int32_t* __restrict__ hist, uint32_t* __restrict__ dev_status) {
  extern __shared__ int32_t sh[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int r0 = blockIdx.x * routes_per_tile;
  const int r1 = min(R, r0 + routes_per_tile);
  bool bad = false;
  for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    const int e = __ldg(ids + r);
    if (e >= 0 && e < E) atomicAdd(&sh[e], 1); else bad = true;
  }
  if (bad) report(dev_status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  int32_t* out = hist + static_cast<int64_t>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) out[e] = sh[e];
}

__global__ void __launch_bounds__(512)
permute_scan(int R, int E, int n_tiles, int capacity, int32_t* __restrict__ hist,
             int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
             int32_t* __restrict__ n_dropped) {
  __shared__ int32_t warp_tot[16];
  const int e = threadIdx.x;
  int32_t run = 0;
  if (e < E) {
    int t = 0;
    for (; t + 4 <= n_tiles; t += 4) {
      const int64_t b = static_cast<int64_t>(t) * E + e;
      const int32_t v0 = hist[b], v1 = hist[b + E], v2 = hist[b + 2 * E], v3 = hist[b + 3 * E];
      hist[b] = run; run += v0;
      hist[b + E] = run; run += v1;
      hist[b + 2 * E] = run; run += v2;
      hist[b + 3 * E] = run; run += v3;
    }
    for (; t < n_tiles; ++t) {
      const int64_t b = static_cast<int64_t>(t) * E + e;
      const int32_t v = hist[b];
      hist[b] = run;
      run += v;
    }
  }
  const int32_t c = (e < E) ? (capacity < 0 ? run : min(run, capacity)) : 0;
  // Block-wide exclusive scan of c over experts.
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
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
    counts[e] = c;
    offsets[e] = before + incl - c;
  }
  if (e == E - 1) {
    offsets[E] = before + incl;
    *n_dropped = R - (before + incl);
  }
}

__global__ void __launch_bounds__(kPermThreads)
permute_scatter(int T, int d, int E, int k, int tokens_per_tile, int capacity,
                const int32_t* __restrict__ ids, const int32_t* __restrict__ tile_base,
                const int32_t* __restrict__ offsets, const uint4* __restrict__ x,
                uint4* __restrict__ x_perm, int32_t* __restrict__ row_to_route,
                int32_t* __restrict__ route_to_row) {
  extern __shared__ int32_t sh[];
  int32_t* cnt = sh;                        // [kPermWarps][E]
  int32_t* off = cnt + kPermWarps * E;      // [E]
  int32_t* rows = off + E;                  // [routes in tile]
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int t0 = blockIdx.x * tokens_per_tile;
  const int t1 = min(T, t0 + tokens_per_tile);
  const int r0 = t0 * k, r1 = t1 * k, nr = r1 - r0;
  const int sub = (nr + kPermWarps - 1) / kPermWarps;
  const int s0 = r0 + w * sub, s1 = min(r1, s0 + sub);

  for (int i = threadIdx.x; i < kPermWarps * E; i += blockDim.x) cnt[i] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) off[e] = __ldg(offsets + e);
  __syncthreads();
  // 1. per-warp expert counts of the warp's contiguous sub-range
  for (int r = s0 + lane; r < s1; r += 32) {
    const int e = __ldg(ids + r);
    if (e >= 0 && e < E) atomicAdd(&cnt[w * E + e], 1);
  }
  __syncthreads();
  // 2. turn counts into each warp's first ordinal: tile base + earlier warps
  const int32_t* base = tile_base + static_cast<int64_t>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = __ldg(base + e);
    for (int ww = 0; ww < kPermWarps; ++ww) {
      const int32_t v = cnt[ww * E + e];
      cnt[ww * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  // 3. stable ranks, 32 routes at a time in route order
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int c0 = s0; c0 < s1; c0 += 32) {
    const int r = c0 + lane;
    int e = -1;
    if (r < s1) {
      e = __ldg(ids + r);
      if (e < 0 || e >= E) e = -2;  // invalid id: its own group, never admitted
    }
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
    int32_t ordinal = 0;
    if (e >= 0) ordinal = cnt[w * E + e] + __popc(peers & lt_mask);
    __syncwarp();
    if (e >= 0 && (peers & lt_mask) == 0) cnt[w * E + e] += __popc(peers);
    __syncwarp();
    if (r < s1) {
      int32_t row = -1;
      if (e >= 0 && (capacity < 0 || ordinal < capacity)) {
        row = off[e] + ordinal;
        row_to_route[row] = r;
      }
      route_to_row[r] = row;
      rows[r - r0] = row;
    }
  }
  __syncthreads();
  // 4. token-major row copy: each token row is read once
  const int chunks = d >> 3;  // 16-byte chunks per row
  for (int t = t0 + w; t < t1; t += kPermWarps) {
    const uint4* src = x + static_cast<int64_t>(t) * chunks;
    const int32_t* trow = rows + (t - t0) * k;
    for (int c = lane; c < chunks; c += 32) {
      const uint4 v = __ldg(src + c);
      for (int j = 0; j < k; ++j) {
        const int32_t row = trow[j];
        if (row >= 0) x_perm[static_cast<int64_t>(row) * chunks + c] = v;
      }
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API size_t moe_permute_workspace_size(int32_t T, int32_t k, int32_t E) {
  if (T <= 0 || k <= 0 || E <= 0) return 256;
  const PermTiling tl = permute_tiling(T, k);
  Carver c;
  c.take<int32_t>(static_cast<size_t>(tl.n_tiles) * E);
  return c.off + 256;
}

MOE_API moe_status moe_permute(int32_t T, int32_t d, int32_t E, int32_t k, int32_t capacity,
                               const int32_t* topk_ids, const moe_bf16* x, moe_bf16* x_perm,
                               int32_t* counts, int32_t* offsets, int32_t* row_to_route,
                               int32_t* route_to_row, int32_t* n_dropped, void* ws,
                               size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > 512 || k > 16 || d % 8 != 0 || static_cast<int64_t>(T) * k >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  if (counts == nullptr || offsets == nullptr || n_dropped == nullptr) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (topk_ids == nullptr || x == nullptr || x_perm == nullptr ||
                row_to_route == nullptr || route_to_row == nullptr || ws == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned16(x) || !aligned16(x_perm))) return MOE_ERR_UNSUPPORTED;
  if (ws_bytes < moe_permute_workspace_size(T, k, E)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = as_cuda(stream);
  const int R = T * k;
  if (T == 0) {
    // No routes: empty segments.  The scan kernel with zero tiles writes them.
    permute_scan<<<1, 512, 0, s>>>(0, E, 0, capacity, nullptr, counts, offsets, n_dropped);
    return launch_status();
  }
  const PermTiling tl = permute_tiling(T, k);
  Carver c;
  int32_t* hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) +
                                             c.take<int32_t>(static_cast<size_t>(tl.n_tiles) * E));
  const int rpt = tl.tokens_per_tile * k;
  permute_hist<<<tl.n_tiles, kPermThreads, E * sizeof(int32_t), s>>>(R, E, rpt, topk_ids, hist,
                                                                   dev_status);
  permute_scan<<<1, 512, 0, s>>>(R, E, tl.n_tiles, capacity, hist, counts, offsets, n_dropped);
  const size_t smem = (static_cast<size_t>(kPermWarps) * E + E + rpt) * sizeof(int32_t);
  permute_scatter<<<tl.n_tiles, kPermThreads, smem, s>>>(
      T, d, E, k, tl.tokens_per_tile, capacity, topk_ids, hist, offsets,
      reinterpret_cast<const uint4*>(x), reinterpret_cast<uint4*>(x_perm), row_to_route,
      route_to_row);
  return launch_status();
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

constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB
static __device__ __align__(256) uint8_t g_permute_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device, looked up once per
// device (in host code the array's name is only a host-side stand-in).
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
