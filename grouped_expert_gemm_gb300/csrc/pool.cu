// Static-shape pooled-wave layout, kept in memory (no communication).
//
// [POOL] "Fixed pooled-wave all-to-all for the 8-of-384 MoE":
//   02 "One pool for each destination GPU": expert e belongs to destination
//      e / L as local expert e % L; 64 fixed destination pools per wave; the
//      first full-width row carries the packed local expert ids.
//   03 "Static shapes from send to combine": [n_dest, pool_cap + 1, d] pools,
//      receiver compact [n_local, local_cap, d], fixed source order.
//   04 "Capacity and memory": extra sender rows and rows above the receiver
//      capacity are dropped, counted separately.
//
// Both sides use the same three-launch stable ranking as the permute step
// (tile histogram -> per-key scan over tiles -> in-tile stable ranks with
// __match_any_sync), keyed by destination on the sender and by the local id
// read from the header row on the receiver.  Payload rows move as 16-byte
// chunks, each source row read once.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxTileItems = 4096;

int tile_items(int64_t n_items, int granule) {
  // about two tiles per SM, whole granules (tokens) per tile
  int64_t per = ceil_div(ceil_div(n_items, granule), 2 * 152) * granule;
  if (per < granule) per = granule;
  const int64_t cap = (kMaxTileItems / granule) * granule;
  if (per > cap) per = cap;
  return static_cast<int>(per);
}

// ------------------------------- sender -----------------------------------

__global__ void __launch_bounds__(kThreads)
pack_hist(int R, int n_dest, int L, int items_per_tile, const int32_t* __restrict__ ids,
          int32_t* __restrict__ hist, uint32_t* __restrict__ dev_status) {
  extern __shared__ int32_t sh[];
  for (int i = threadIdx.x; i < n_dest; i += blockDim.x) sh[i] = 0;
  pdl_wait();
  __syncthreads();
  const int r0 = blockIdx.x * items_per_tile, r1 = min(R, r0 + items_per_tile);
  bool bad = false;
  for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    const int e = __ldg(ids + r);
    if (e >= 0 && e < n_dest * L) atomicAdd(&sh[e / L], 1); else bad = true;
  }
  if (bad) report(dev_status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  for (int i = threadIdx.x; i < n_dest; i += blockDim.x)
    hist[static_cast<int64_t>(blockIdx.x) * n_dest + i] = sh[i];
  pdl_trigger();
}

__device__ __forceinline__ int block_sum_512(int v, int* scratch) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  int tot = 0;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) tot += scratch[i];
  return tot;
}

// In-place exclusive scan down the columns of hist [n_tiles][n_cols] (row-major),
// column totals to tot[n_cols] (shared memory); every thread of the block calls it.
// G threads (a power of two, at most a warp) share a column: each sums its slice of
// the tiles with batched independent loads, the group scans the slice sums with
// shuffles, and each thread rewrites its slice -- a chain of n_tiles / G loads
// instead of n_tiles dependent ones.
constexpr int kScanBatch = 8;

__device__ void scan_columns(int n_cols, int n_tiles, int32_t* __restrict__ hist, int32_t* tot) {
  const int nthr = blockDim.x;
  int G = 1;
  while (G < 32 && n_cols * G * 2 <= nthr) G *= 2;
  const int per_pass = nthr / G;
  const int m = threadIdx.x % G, cl = threadIdx.x / G;
  const int t0 = static_cast<int>(static_cast<int64_t>(n_tiles) * m / G);
  const int t1 = static_cast<int>(static_cast<int64_t>(n_tiles) * (m + 1) / G);
  for (int c0 = 0; c0 < n_cols; c0 += per_pass) {
    const int c = c0 + cl;
    const bool live = c < n_cols;
    int sum = 0;
    if (live) {
      for (int t = t0; t < t1; t += kScanBatch) {
        int32_t v[kScanBatch];
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j)
          v[j] = t + j < t1 ? hist[static_cast<int64_t>(t + j) * n_cols + c] : 0;
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j) sum += v[j];
      }
    }
    int incl = sum;
    for (int o = 1; o < G; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o, G);
      if (m >= o) incl += n;
    }
    const int total = __shfl_sync(0xFFFFFFFFu, incl, G - 1, G);
    if (live) {
      int run = incl - sum;
      for (int t = t0; t < t1; t += kScanBatch) {
        int32_t v[kScanBatch];
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j)
          v[j] = t + j < t1 ? hist[static_cast<int64_t>(t + j) * n_cols + c] : 0;
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j) {
          if (t + j < t1) hist[static_cast<int64_t>(t + j) * n_cols + c] = run;
          run += v[j];
        }
      }
      if (m == 0) tot[c] = total;
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(512)
pack_scan(int n_dest, int n_tiles, int n_waves, int pool_cap, int policy, int wave,
          int32_t* __restrict__ hist, int32_t* __restrict__ pool_fill,
          int32_t* __restrict__ sender_drops) {
  pdl_wait();
  __shared__ int scratch[16];
  __shared__ int32_t tot[512];  // n_dest <= 512
  scan_columns(n_dest, n_tiles, hist, tot);
  const int D = threadIdx.x;
  const int32_t run = D < n_dest ? tot[D] : 0;
  int in_wave = 0;
  if (D < n_dest) {
    if (policy == MOE_WAVE_STRIPE)
      in_wave = run > wave ? (run - wave + n_waves - 1) / n_waves : 0;
    else
      in_wave = (D % n_waves == wave) ? run : 0;
  }
  const int fill = min(in_wave, pool_cap);
  if (D < n_dest) pool_fill[D] = fill;
  const int drops = block_sum_512(in_wave - fill, scratch);
  if (threadIdx.x == 0) *sender_drops = drops;
  pdl_trigger();
}

__global__ void __launch_bounds__(kThreads)
pack_scatter(int T, int d, int k, int n_dest, int L, int n_waves, int pool_cap, int policy,
             int wave, int tokens_per_tile, const int32_t* __restrict__ ids,
             const int32_t* __restrict__ tile_base, const int32_t* __restrict__ pool_fill,
             const uint4* __restrict__ x, uint4* __restrict__ pools,
             uint16_t* __restrict__ pools_u16, int32_t* __restrict__ route_to_poolrow) {
  pdl_wait();
  extern __shared__ int32_t sh[];
  int32_t* cnt = sh;                    // [kWarps][n_dest]
  int64_t* rows = reinterpret_cast<int64_t*>(cnt + ((kWarps * n_dest + 1) & ~1));  // [tile routes]
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t pool_rows = pool_cap + 1;
  // Header elements past each pool's fill are EMPTY (grid-stride over all pools).
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       i < static_cast<int64_t>(n_dest) * d; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int D = static_cast<int>(i / d), c = static_cast<int>(i % d);
    if (c >= __ldg(pool_fill + D)) pools_u16[D * pool_rows * d + c] = MOE_POOL_EMPTY;
  }
  const int t0 = blockIdx.x * tokens_per_tile, t1 = min(T, t0 + tokens_per_tile);
  const int r0 = t0 * k, r1 = t1 * k, nr = r1 - r0;
  const int sub = (nr + kWarps - 1) / kWarps;
  const int s0 = r0 + w * sub, s1 = min(r1, s0 + sub);
  const int E = n_dest * L;
  for (int i = threadIdx.x; i < kWarps * n_dest; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  for (int r = s0 + lane; r < s1; r += 32) {
    const int e = __ldg(ids + r);
    if (e >= 0 && e < E) atomicAdd(&cnt[w * n_dest + e / L], 1);
  }
  __syncthreads();
  const int32_t* base = tile_base + static_cast<int64_t>(blockIdx.x) * n_dest;
  for (int D = threadIdx.x; D < n_dest; D += blockDim.x) {
    int32_t run = __ldg(base + D);
    for (int ww = 0; ww < kWarps; ++ww) {
      const int32_t v = cnt[ww * n_dest + D];
      cnt[ww * n_dest + D] = run;
      run += v;
    }
  }
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
  for (int c0 = s0; c0 < s1; c0 += 32) {
    const int r = c0 + lane;
    int e = -1, D = -1;
    if (r < s1) {
      e = __ldg(ids + r);
      D = (e >= 0 && e < E) ? e / L : -2;
    }
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, D);
    int32_t j = 0;
    if (D >= 0) j = cnt[w * n_dest + D] + __popc(peers & lt);
    __syncwarp();
    if (D >= 0 && (peers & lt) == 0) cnt[w * n_dest + D] += __popc(peers);
    __syncwarp();
    if (r < s1) {
      int64_t dst = -1;
      int32_t map = -1;
      if (D >= 0) {
        const int wv = policy == MOE_WAVE_STRIPE ? j % n_waves : D % n_waves;
        const int row = policy == MOE_WAVE_STRIPE ? j / n_waves : j;
        if (wv == wave && row < pool_cap) {
          map = D * pool_cap + row;
          dst = D * pool_rows + 1 + row;
          pools_u16[D * pool_rows * d + row] = static_cast<uint16_t>(e % L);
        }
      }
      route_to_poolrow[r] = map;
      rows[r - r0] = dst;
    }
  }
  __syncthreads();
  // Token-major copy: each token row is read once (four 16-byte loads in flight
  // per lane) and written to each of its rows placed in this wave.
  const int chunks = d >> 3;
  for (int t = t0 + w; t < t1; t += kWarps) {
    const int64_t* trow = rows + (t - t0) * k;
    bool any = false;
    for (int jj = 0; jj < k; ++jj) any |= trow[jj] >= 0;
    if (!any) continue;
    const uint4* src = x + static_cast<int64_t>(t) * chunks;
    for (int cb = 0; cb < chunks; cb += 32 * 4) {
      const int c = cb + lane;
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + 32 * u < chunks) v[u] = __ldg(src + c + 32 * u);
      for (int jj = 0; jj < k; ++jj) {
        const int64_t dst = trow[jj];
        if (dst < 0) continue;
        uint4* o = pools + dst * chunks;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (c + 32 * u < chunks) o[c + 32 * u] = v[u];
      }
    }
  }
  pdl_trigger();
}

// ------------------------------ receiver ----------------------------------

// Visit position i of the receiver -> pool row (source * pool_cap + row): sources
// from `first` on (the per-receiver rotation; 0 = fixed source order), rows up.
__device__ __forceinline__ int64_t visit_to_poolrow(int64_t i, int pool_cap, int n_src, int first) {
  const int64_t s = i / pool_cap + first;
  return (s >= n_src ? s - n_src : s) * pool_cap + i % pool_cap;
}

__device__ __forceinline__ int header_key(const uint16_t* __restrict__ pools_u16, int64_t i,
                                          int pool_cap, int d, int n_local, bool* bad) {
  const int64_t s = i / pool_cap, r = i % pool_cap;
  const int h = __ldg(pools_u16 + s * (pool_cap + 1) * d + r);
  if (h == MOE_POOL_EMPTY) return -1;
  if (h >= n_local) { *bad = true; return -1; }
  return h;
}

__global__ void __launch_bounds__(kThreads)
compact_hist(int64_t n_items, int pool_cap, int d, int n_local, int items_per_tile, int n_src,
             int first, const uint16_t* __restrict__ pools_u16, int32_t* __restrict__ hist,
             uint32_t* __restrict__ dev_status) {
  extern __shared__ int32_t sh[];
  for (int i = threadIdx.x; i < n_local; i += blockDim.x) sh[i] = 0;
  pdl_wait();
  __syncthreads();
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * items_per_tile;
  const int64_t i1 = min(n_items, i0 + items_per_tile);
  bool bad = false;
  for (int64_t i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const int l = header_key(pools_u16, visit_to_poolrow(i, pool_cap, n_src, first), pool_cap, d,
                             n_local, &bad);
    if (l >= 0) atomicAdd(&sh[l], 1);
  }
  if (bad) report(dev_status, MOE_DEV_BAD_HEADER_ID);
  __syncthreads();
  for (int i = threadIdx.x; i < n_local; i += blockDim.x)
    hist[static_cast<int64_t>(blockIdx.x) * n_local + i] = sh[i];
  pdl_trigger();
}

__global__ void __launch_bounds__(512)
compact_scan(int n_local, int n_tiles, int local_cap, int32_t* __restrict__ hist,
             int32_t* __restrict__ local_counts, int32_t* __restrict__ receiver_drops) {
  pdl_wait();
  __shared__ int scratch[16];
  extern __shared__ int32_t tot[];  // [n_local]
  scan_columns(n_local, n_tiles, hist, tot);
  int drops_total = 0;
  for (int l0 = 0; l0 < n_local; l0 += blockDim.x) {
    const int l = l0 + threadIdx.x;
    const int32_t run = l < n_local ? tot[l] : 0;
    if (l < n_local) local_counts[l] = min(run, local_cap);
    drops_total += block_sum_512(l < n_local ? run - min(run, local_cap) : 0, scratch);
    __syncthreads();
  }
  if (threadIdx.x == 0) *receiver_drops = drops_total;
  pdl_trigger();
}

__global__ void __launch_bounds__(kThreads)
compact_scatter(int64_t n_items, int pool_cap, int d, int n_local, int local_cap,
                int items_per_tile, int n_src, int first, const uint16_t* __restrict__ pools_u16,
                const uint4* __restrict__ pools, const int32_t* __restrict__ tile_base,
                uint4* __restrict__ compact, int32_t* __restrict__ poolrow_to_row) {
  pdl_wait();
  extern __shared__ int32_t sh[];
  int32_t* cnt = sh;                    // [kWarps][n_local]
  int32_t* rows = cnt + kWarps * n_local;  // [items in tile]
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * items_per_tile;
  const int64_t i1 = min(n_items, i0 + items_per_tile);
  const int64_t nr = i1 - i0;
  const int64_t sub = (nr + kWarps - 1) / kWarps;
  const int64_t s0 = i0 + w * sub, s1 = min(i1, s0 + sub);
  for (int i = threadIdx.x; i < kWarps * n_local; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  bool bad = false;
  for (int64_t i = s0 + lane; i < s1; i += 32) {
    const int l = header_key(pools_u16, visit_to_poolrow(i, pool_cap, n_src, first), pool_cap, d,
                             n_local, &bad);
    if (l >= 0) atomicAdd(&cnt[w * n_local + l], 1);
  }
  __syncthreads();
  const int32_t* base = tile_base + static_cast<int64_t>(blockIdx.x) * n_local;
  for (int l = threadIdx.x; l < n_local; l += blockDim.x) {
    int32_t run = __ldg(base + l);
    for (int ww = 0; ww < kWarps; ++ww) {
      const int32_t v = cnt[ww * n_local + l];
      cnt[ww * n_local + l] = run;
      run += v;
    }
  }
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
  for (int64_t c0 = s0; c0 < s1; c0 += 32) {
    const int64_t i = c0 + lane;
    const int64_t pr = visit_to_poolrow(i, pool_cap, n_src, first);
    int l = -2;
    if (i < s1) l = header_key(pools_u16, pr, pool_cap, d, n_local, &bad);
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, l);
    int32_t o = 0;
    if (l >= 0) o = cnt[w * n_local + l] + __popc(peers & lt);
    __syncwarp();
    if (l >= 0 && (peers & lt) == 0) cnt[w * n_local + l] += __popc(peers);
    __syncwarp();
    if (i < s1) {
      const int32_t row = (l >= 0 && o < local_cap) ? l * local_cap + o : -1;
      poolrow_to_row[pr] = row;
      rows[i - i0] = row;
    }
  }
  __syncthreads();
  // Row copy, one warp per kept row, four 16-byte loads in flight per lane.
  const int chunks = d >> 3;
  for (int64_t i = i0 + w; i < i1; i += kWarps) {
    const int32_t row = rows[i - i0];
    if (row < 0) continue;
    const int64_t pr = visit_to_poolrow(i, pool_cap, n_src, first);
    const int64_t s = pr / pool_cap, r = pr % pool_cap;
    const uint4* src = pools + (s * (pool_cap + 1) + 1 + r) * chunks;
    uint4* dst = compact + static_cast<int64_t>(row) * chunks;
    for (int cb = 0; cb < chunks; cb += 32 * 4) {
      const int c = cb + lane;
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + 32 * u < chunks) v[u] = __ldg(src + c + 32 * u);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + 32 * u < chunks) dst[c + 32 * u] = v[u];
    }
  }
  pdl_trigger();
}

__global__ void compose_kernel(int64_t n, const int32_t* __restrict__ a,
                               const int32_t* __restrict__ b, int64_t b_len,
                               int32_t* __restrict__ out, uint32_t* __restrict__ dev_status) {
  pdl_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t v = __ldg(a + i);
    int32_t r = -1;
    if (v >= 0) {
      if (v < b_len) r = __ldg(b + v); else report(dev_status, MOE_DEV_BAD_ROW);
    }
    out[i] = r;
  }
  pdl_trigger();
}

}  // namespace
}  // namespace moe

using namespace moe;

static bool pool_params_ok(const moe_pool_params* p) {
  return p != nullptr && p->n_dest > 0 && p->local_per_dest > 0 && p->n_waves > 0 &&
         p->pool_cap > 0 && (p->wave_policy == MOE_WAVE_STRIPE || p->wave_policy == MOE_WAVE_DESTMOD);
}

MOE_API size_t moe_pool_pack_workspace_size(const moe_pool_params* p, int32_t T, int32_t k) {
  if (!pool_params_ok(p) || T <= 0 || k <= 0) return 256;
  const int per = tile_items(static_cast<int64_t>(T) * k, k);
  const int64_t n_tiles = ceil_div(static_cast<int64_t>(T) * k, per);
  Carver c;
  c.take<int32_t>(static_cast<size_t>(n_tiles) * p->n_dest);
  return c.off + 256;
}

MOE_API moe_status moe_pool_pack(const moe_pool_params* p, int32_t T, int32_t d, int32_t k,
                                 int32_t wave, const int32_t* topk_ids, const moe_bf16* x,
                                 moe_bf16* pools, int32_t* route_to_poolrow, int32_t* pool_fill,
                                 int32_t* sender_drops, void* ws, size_t ws_bytes,
                                 uint32_t* dev_status, moe_stream_t stream) {
  if (!pool_params_ok(p) || T < 0 || d <= 0 || k <= 0 || wave < 0 || wave >= p->n_waves)
    return MOE_ERR_INVALID_ARG;
  if (k > 16 || d % 8 != 0 || p->pool_cap > d || p->local_per_dest > 65534 ||
      static_cast<int64_t>(p->n_dest) * p->local_per_dest > 512 || p->n_dest > 512 ||
      static_cast<int64_t>(T) * k >= (int64_t(1) << 31) ||
      static_cast<int64_t>(p->n_dest) * p->pool_cap >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  if (pools == nullptr || pool_fill == nullptr || sender_drops == nullptr ||
      (T > 0 && (topk_ids == nullptr || x == nullptr || route_to_poolrow == nullptr ||
                 ws == nullptr)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(pools) || (T > 0 && !aligned16(x))) return MOE_ERR_UNSUPPORTED;
  if (ws_bytes < moe_pool_pack_workspace_size(p, T, k)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = as_cuda(stream);
  const int64_t R = static_cast<int64_t>(T) * k;
  const int per = T > 0 ? tile_items(R, k) : k;
  const int n_tiles = T > 0 ? static_cast<int>(ceil_div(R, per)) : 0;
  int32_t* hist = static_cast<int32_t*>(ws);
  if (n_tiles > 0)
    launch(pack_hist, dim3(n_tiles), dim3(kThreads), p->n_dest * sizeof(int32_t), s,
           static_cast<int>(R), p->n_dest, p->local_per_dest, per, topk_ids, hist, dev_status);
  launch(pack_scan, dim3(1), dim3(512), 0, s, p->n_dest, n_tiles, p->n_waves, p->pool_cap,
         p->wave_policy, wave, hist, pool_fill, sender_drops);
  const size_t smem = ((kWarps * p->n_dest + 1) & ~1) * sizeof(int32_t) + per * sizeof(int64_t);
  launch(pack_scatter, dim3(n_tiles > 0 ? n_tiles : 1), dim3(kThreads), smem, s, T, d, k,
         p->n_dest, p->local_per_dest, p->n_waves, p->pool_cap, p->wave_policy, wave, per / k,
         topk_ids, static_cast<const int32_t*>(hist), static_cast<const int32_t*>(pool_fill),
         reinterpret_cast<const uint4*>(x), reinterpret_cast<uint4*>(pools),
         reinterpret_cast<uint16_t*>(pools), route_to_poolrow);
  return launch_status();
}

MOE_API size_t moe_pool_compact_workspace_size(int32_t n_src, int32_t pool_cap, int32_t n_local) {
  if (n_src <= 0 || pool_cap <= 0 || n_local <= 0) return 256;
  const int64_t n_items = static_cast<int64_t>(n_src) * pool_cap;
  const int per = tile_items(n_items, 32);
  Carver c;
  c.take<int32_t>(static_cast<size_t>(ceil_div(n_items, per)) * n_local);
  return c.off + 256;
}

MOE_API moe_status moe_pool_compact_rotated(int32_t n_src, int32_t pool_cap, int32_t d,
                                            int32_t n_local, int32_t local_cap,
                                            int32_t first_source, const moe_bf16* pools,
                                            moe_bf16* compact, int32_t* local_counts,
                                            int32_t* poolrow_to_row, int32_t* receiver_drops,
                                            void* ws, size_t ws_bytes, uint32_t* dev_status,
                                            moe_stream_t stream) {
  if (n_src <= 0 || pool_cap <= 0 || d <= 0 || n_local <= 0 || local_cap < 0 ||
      first_source < 0 || first_source >= n_src)
    return MOE_ERR_INVALID_ARG;
  if (d % 8 != 0 || pool_cap > d || n_local > 65534 || n_local > 4096 ||
      static_cast<int64_t>(n_src) * pool_cap >= (int64_t(1) << 31) ||
      static_cast<int64_t>(n_local) * local_cap >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  if (pools == nullptr || local_counts == nullptr || poolrow_to_row == nullptr ||
      receiver_drops == nullptr || ws == nullptr || (compact == nullptr && local_cap > 0))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(pools) || (compact != nullptr && !aligned16(compact))) return MOE_ERR_UNSUPPORTED;
  if (ws_bytes < moe_pool_compact_workspace_size(n_src, pool_cap, n_local))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = as_cuda(stream);
  const int64_t n_items = static_cast<int64_t>(n_src) * pool_cap;
  const int per = tile_items(n_items, 32);
  const int n_tiles = static_cast<int>(ceil_div(n_items, per));
  int32_t* hist = static_cast<int32_t*>(ws);
  const uint16_t* hdr = reinterpret_cast<const uint16_t*>(pools);
  launch(compact_hist, dim3(n_tiles), dim3(kThreads), n_local * sizeof(int32_t), s, n_items,
         pool_cap, d, n_local, per, n_src, first_source, hdr, hist, dev_status);
  launch(compact_scan, dim3(1), dim3(512), n_local * sizeof(int32_t), s, n_local, n_tiles,
         local_cap, hist, local_counts, receiver_drops);
  const size_t smem = (static_cast<size_t>(kWarps) * n_local + per) * sizeof(int32_t);
  launch(compact_scatter, dim3(n_tiles), dim3(kThreads), smem, s, n_items, pool_cap, d, n_local,
         local_cap, per, n_src, first_source, hdr, reinterpret_cast<const uint4*>(pools),
         static_cast<const int32_t*>(hist), reinterpret_cast<uint4*>(compact), poolrow_to_row);
  return launch_status();
}

MOE_API moe_status moe_pool_compact(int32_t n_src, int32_t pool_cap, int32_t d, int32_t n_local,
                                    int32_t local_cap, const moe_bf16* pools, moe_bf16* compact,
                                    int32_t* local_counts, int32_t* poolrow_to_row,
                                    int32_t* receiver_drops, void* ws, size_t ws_bytes,
                                    uint32_t* dev_status, moe_stream_t stream) {
  return moe_pool_compact_rotated(n_src, pool_cap, d, n_local, local_cap, 0, pools, compact,
                                  local_counts, poolrow_to_row, receiver_drops, ws, ws_bytes,
                                  dev_status, stream);
}

MOE_API moe_status moe_compose_map(int64_t n, const int32_t* a, const int32_t* b, int64_t b_len,
                                   int32_t* out, uint32_t* dev_status, moe_stream_t stream) {
  if (n < 0 || b_len < 0) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (a == nullptr || out == nullptr || (b == nullptr && b_len > 0)) return MOE_ERR_INVALID_ARG;
  const int64_t blocks = ceil_div(n, 256);
  launch(compose_kernel, dim3(static_cast<unsigned>(blocks < 152 * 32 ? blocks : 152 * 32)),
         dim3(256), 0, as_cuda(stream), n, a, b, b_len, out, dev_status);
  return launch_status();
}
