// Debug validators of the permutation and pooled-layout maps: each reads what a
// permute / pool call wrote and sets MOE_DEV_BAD_MAP in the caller's status word
// when an invariant fails.
//
// [M6.6] 0x0CD "Route And Combine Assertions", [M6.2] 0x03B / [M6.6] 0x03B,
// 0x03C3: counts and offsets with their sentinel,
// the stable expert-major order, the inverse map (pi^-1[pi[j]] = j: one row per
// accepted route and one route per row), accepted + dropped = T*k, and with a
// capacity C a route dropped only when its expert already holds C routes of
// smaller id.  [POOL] 02-05: header ids and fills, one route per filled pool
// row; pool rows to compact rows one to one, in (source, row) order.
//
// The permutation carries both directions of its map, so every check reads one
// entry and the entries it points at.  The pooled maps go one way only
// (route -> pool row, pool row -> compact row): their inverse is rebuilt in the
// caller's workspace (one compare-and-swap per mapped entry, a second writer to
// the same target is a violation), then read back per target row.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kValThreads = 256;

__device__ __forceinline__ int live_routes(int R, int k, const int32_t* valid) {
  if (valid == nullptr) return R;
  const int v = __ldg(valid);
  return v <= 0 ? 0 : min(R, v * k);
}

__device__ __forceinline__ void flag_if(bool bad, uint32_t* st) {
  if (bad) report(st, MOE_DEV_BAD_MAP);
}

// ---- permutation ------------------------------------------------------------

// counts / offsets / sentinel / conservation (one block).
__global__ void __launch_bounds__(kValThreads)
validate_counts_kernel(int R, int E, int k, int capacity, const int32_t* __restrict__ valid,
                       const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
                       const int32_t* __restrict__ n_dropped, uint32_t* __restrict__ st) {
  pdl_wait();
  bool bad = false;
  if (threadIdx.x == 0) {
    const int acc = __ldg(offsets + E);
    const int drop = __ldg(n_dropped);
    bad = __ldg(offsets) != 0 || acc < 0 || drop < 0 || acc + drop != live_routes(R, k, valid) ||
          (capacity < 0 && drop != 0);
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = __ldg(counts + e);
    if (c < 0 || __ldg(offsets + e + 1) - __ldg(offsets + e) != c) bad = true;
    if (capacity >= 0 && c > capacity) bad = true;
  }
  flag_if(bad, st);
  pdl_trigger();
}

// Thread i checks route i (its row and the way back) and row i (its route and
// the way back, and the order against row i + 1).
__global__ void __launch_bounds__(kValThreads)
validate_maps_kernel(int R, int E, int k, int capacity, const int32_t* __restrict__ valid,
                     const int32_t* __restrict__ ids, const int32_t* __restrict__ counts,
                     const int32_t* __restrict__ offsets, const int32_t* __restrict__ row_to_route,
                     const int32_t* __restrict__ route_to_row, uint32_t* __restrict__ st) {
  pdl_wait();
  const int R_live = live_routes(R, k, valid);
  const int acc = __ldg(offsets + E);
  bool bad = acc < 0 || acc > R_live;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; !bad && i < R; i += gridDim.x * blockDim.x) {
    const int row = __ldg(route_to_row + i);
    if (i >= R_live) {
      bad = row != -1;  // padding routes map nowhere
    } else {
      const int e = __ldg(ids + i);
      const bool known = e >= 0 && e < E;
      if (row >= 0) {
        bad = !known || row >= acc || __ldg(row_to_route + row) != i ||
              row < __ldg(offsets + e) || row >= __ldg(offsets + e + 1);
      } else if (row == -1) {
        // dropped: the expert is full, with routes of smaller id only
        if (known) {
          const int c = __ldg(counts + e), o = __ldg(offsets + e + 1);
          bad = capacity < 0 || c != capacity ||
                (c > 0 && (o < 1 || o > acc || __ldg(row_to_route + o - 1) > i));
        }
      } else {
        bad = true;
      }
    }
    if (!bad && i < acc) {
      const int r = __ldg(row_to_route + i);
      if (r < 0 || r >= R_live || __ldg(route_to_row + r) != i) {
        bad = true;
      } else if (i + 1 < acc) {
        const int e = __ldg(ids + r);  // a mapped route has a known expert (checked above)
        if (e >= 0 && e < E && i + 1 < __ldg(offsets + e + 1))
          bad = __ldg(row_to_route + i + 1) <= r;  // stable: ids increase along a segment
      }
    }
  }
  flag_if(bad, st);
  pdl_trigger();
}

// ---- inverse of a one-way map in the workspace ------------------------------

__global__ void __launch_bounds__(kValThreads) fill_minus_one(int64_t n, int32_t* __restrict__ a) {
  pdl_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    a[i] = -1;
  pdl_trigger();
}

// Record source i as the preimage of `target`; false when another source holds it.
__device__ __forceinline__ bool claim(int32_t* inv, int64_t target, int32_t i) {
  return atomicCAS(inv + target, -1, i) == -1;
}

// Target rows [0, n_owner * cap): row j < fill of its owner has exactly one
// preimage, the preimages increase along the row index (stable order), rows at
// or past the fill have none.  Returns true on a violation.  Every index is
// bounded by the target space whatever the (possibly corrupted) fills hold.
__device__ __forceinline__ bool check_targets(int64_t q, int cap, const int32_t* fill,
                                              const int32_t* inv) {
  const int owner = static_cast<int>(q / cap), j = static_cast<int>(q % cap);
  const int f = min(__ldg(fill + owner), cap);  // a fill above cap is flagged by its owner's check
  const int src = inv[q];
  if (j >= f) return src != -1;
  if (src < 0) return true;
  return j + 1 < f && inv[q + 1] <= src;
}

// ---- pooled layout: sender pools of one wave ---------------------------------

__device__ __forceinline__ uint16_t header_at(const uint16_t* pools, int pool_cap, int d, int D,
                                              int r) {
  return __ldg(pools + static_cast<int64_t>(D) * (pool_cap + 1) * d + r);
}

// Fills and headers (one warp per destination); routes claim their pool rows.
__global__ void __launch_bounds__(kValThreads)
validate_pack_kernel(int R, int n_dest, int L, int pool_cap, int d,
                     const int32_t* __restrict__ ids, const uint16_t* __restrict__ pools,
                     const int32_t* __restrict__ route_to_poolrow,
                     const int32_t* __restrict__ fill, int32_t* inv, uint32_t* __restrict__ st) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  bool bad = false;
  for (int D = blockIdx.x * warps + (threadIdx.x >> 5); D < n_dest; D += gridDim.x * warps) {
    const int f = __ldg(fill + D);
    if (f < 0 || f > pool_cap) { bad = true; continue; }
    for (int r = lane; r < d; r += 32) {
      const uint16_t h = header_at(pools, pool_cap, d, D, r);
      if (r < f ? h >= L : h != MOE_POOL_EMPTY) bad = true;
    }
  }
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < R; r += gridDim.x * blockDim.x) {
    const int p = __ldg(route_to_poolrow + r);
    if (p < 0) {
      if (p != -1) bad = true;
      continue;
    }
    const int e = __ldg(ids + r);
    const int D = p / pool_cap, row = p % pool_cap;
    if (e < 0 || e >= n_dest * L || D != e / L || row >= __ldg(fill + D) ||
        header_at(pools, pool_cap, d, D, row) != e % L || !claim(inv, p, r))
      bad = true;
  }
  flag_if(bad, st);
  pdl_trigger();
}

// ---- pooled layout: receiver compact of one wave ----------------------------

// Visit position of pool row i (source s = i / pool_cap) for a receiver whose
// visit starts at source `first`: the order in which compact rows are assigned.
__device__ __forceinline__ int visit_pos(int i, int pool_cap, int n_src, int first) {
  const int s = i / pool_cap - first;
  return (s < 0 ? s + n_src : s) * pool_cap + i % pool_cap;
}

__global__ void __launch_bounds__(kValThreads)
validate_compact_kernel(int n_src, int pool_cap, int d, int n_local, int local_cap, int first,
                        const uint16_t* __restrict__ pools, const int32_t* __restrict__ counts,
                        const int32_t* __restrict__ poolrow_to_row, int32_t* inv,
                        uint32_t* __restrict__ st) {
  pdl_wait();
  bool bad = false;
  for (int l = blockIdx.x * blockDim.x + threadIdx.x; l < n_local; l += gridDim.x * blockDim.x) {
    const int c = __ldg(counts + l);
    if (c < 0 || c > local_cap) bad = true;
  }
  const int n_rows = n_src * pool_cap;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_rows; i += gridDim.x * blockDim.x) {
    const int s = i / pool_cap, r = i % pool_cap;
    const uint16_t h = header_at(pools, pool_cap, d, s, r);
    const int q = __ldg(poolrow_to_row + i);
    if (q == -1) continue;  // empty, invalid header or receiver drop: checked below
    if (h >= n_local || q < 0 || q / local_cap != h || q % local_cap >= __ldg(counts + h) ||
        !claim(inv, q, visit_pos(i, pool_cap, n_src, first)))
      bad = true;
  }
  flag_if(bad, st);
  pdl_trigger();
}

// A receiver drop (a row with a valid header mapped to -1) needs its expert full
// with rows that came earlier in the receiver's visiting order.
__global__ void __launch_bounds__(kValThreads)
validate_compact_drops_kernel(int n_src, int pool_cap, int d, int n_local, int local_cap, int first,
                              const uint16_t* __restrict__ pools,
                              const int32_t* __restrict__ counts,
                              const int32_t* __restrict__ poolrow_to_row, const int32_t* inv,
                              uint32_t* __restrict__ st) {
  pdl_wait();
  bool bad = false;
  const int n_rows = n_src * pool_cap;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_rows; i += gridDim.x * blockDim.x) {
    const uint16_t h = header_at(pools, pool_cap, d, i / pool_cap, i % pool_cap);
    if (h >= n_local || __ldg(poolrow_to_row + i) != -1) continue;
    const int c = __ldg(counts + h);
    if (c != local_cap ||
        (c > 0 && inv[static_cast<int64_t>(h) * local_cap + c - 1] > visit_pos(i, pool_cap, n_src, first)))
      bad = true;
  }
  flag_if(bad, st);
  pdl_trigger();
}

__global__ void __launch_bounds__(kValThreads)
validate_targets_kernel(int64_t n_targets, int cap, const int32_t* __restrict__ fill,
                        const int32_t* inv, uint32_t* __restrict__ st) {
  pdl_wait();
  bool bad = false;
  for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; q < n_targets;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x)
    if (check_targets(q, cap, fill, inv)) bad = true;
  flag_if(bad, st);
  pdl_trigger();
}

unsigned grid_of(int64_t n) {
  int64_t b = ceil_div(n, kValThreads);
  if (b > 152 * 8) b = 152 * 8;
  return static_cast<unsigned>(b < 1 ? 1 : b);
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API moe_status moe_validate_permutation(int32_t T, int32_t E, int32_t k, int32_t capacity,
                                            const int32_t* valid_tokens, const int32_t* topk_ids,
                                            const int32_t* counts, const int32_t* offsets,
                                            const int32_t* row_to_route,
                                            const int32_t* route_to_row,
                                            const int32_t* n_dropped, uint32_t* dev_status,
                                            moe_stream_t stream) {
  if (T < 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > 512 || k > 16 || static_cast<int64_t>(T) * k >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  if (dev_status == nullptr || counts == nullptr || offsets == nullptr || n_dropped == nullptr)
    return MOE_ERR_INVALID_ARG;
  const int R = T * k;
  if (R > 0 && (topk_ids == nullptr || row_to_route == nullptr || route_to_row == nullptr))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_cuda(stream);
  launch(validate_counts_kernel, dim3(1), dim3(kValThreads), 0, s, R, E, k, capacity, valid_tokens,
         counts, offsets, n_dropped, dev_status);
  if (R > 0)
    launch(validate_maps_kernel, dim3(grid_of(R)), dim3(kValThreads), 0, s, R, E, k, capacity,
           valid_tokens, topk_ids, counts, offsets, row_to_route, route_to_row, dev_status);
  return launch_status();
}

MOE_API size_t moe_validate_pools_workspace_size(const moe_pool_params* p) {
  if (p == nullptr || p->n_dest <= 0 || p->pool_cap <= 0) return 0;
  return static_cast<size_t>(p->n_dest) * p->pool_cap * sizeof(int32_t);
}

MOE_API moe_status moe_validate_pools(const moe_pool_params* p, int32_t T, int32_t d, int32_t k,
                                      const int32_t* topk_ids, const moe_bf16* pools,
                                      const int32_t* route_to_poolrow, const int32_t* pool_fill,
                                      void* ws, size_t ws_bytes, uint32_t* dev_status,
                                      moe_stream_t stream) {
  if (p == nullptr || T < 0 || d <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (p->n_dest <= 0 || p->local_per_dest <= 0 || p->pool_cap <= 0) return MOE_ERR_INVALID_ARG;
  if (p->pool_cap > d || p->local_per_dest > 65534 ||
      static_cast<int64_t>(p->n_dest) * p->local_per_dest > 512 || k > 16 ||
      static_cast<int64_t>(T) * k >= (int64_t(1) << 31) ||
      static_cast<int64_t>(p->n_dest) * p->pool_cap >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  if (dev_status == nullptr || pools == nullptr || pool_fill == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_validate_pools_workspace_size(p)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int R = T * k;
  if (R > 0 && (topk_ids == nullptr || route_to_poolrow == nullptr)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_cuda(stream);
  int32_t* inv = static_cast<int32_t*>(ws);
  const int64_t n_targets = static_cast<int64_t>(p->n_dest) * p->pool_cap;
  launch(fill_minus_one, dim3(grid_of(n_targets)), dim3(kValThreads), 0, s, n_targets, inv);
  const int64_t work = R > int64_t(p->n_dest) * 32 ? R : int64_t(p->n_dest) * 32;
  launch(validate_pack_kernel, dim3(grid_of(work)), dim3(kValThreads), 0, s, R, p->n_dest,
         p->local_per_dest, p->pool_cap, d, topk_ids, pools, route_to_poolrow, pool_fill, inv,
         dev_status);
  launch(validate_targets_kernel, dim3(grid_of(n_targets)), dim3(kValThreads), 0, s, n_targets,
         p->pool_cap, pool_fill, static_cast<const int32_t*>(inv), dev_status);
  return launch_status();
}

MOE_API size_t moe_validate_compact_workspace_size(int32_t n_local, int32_t local_cap) {
  if (n_local <= 0 || local_cap <= 0) return 0;
  return static_cast<size_t>(n_local) * local_cap * sizeof(int32_t);
}

MOE_API moe_status moe_validate_compact(int32_t n_src, int32_t pool_cap, int32_t d,
                                        int32_t n_local, int32_t local_cap, int32_t first_source,
                                        const moe_bf16* pools, const int32_t* local_counts,
                                        const int32_t* poolrow_to_row, void* ws, size_t ws_bytes,
                                        uint32_t* dev_status, moe_stream_t stream) {
  if (n_src <= 0 || pool_cap <= 0 || d <= 0 || n_local <= 0 || local_cap <= 0 ||
      first_source < 0 || first_source >= n_src)
    return MOE_ERR_INVALID_ARG;
  if (pool_cap > d || n_local > 65534 ||
      static_cast<int64_t>(n_src) * pool_cap >= (int64_t(1) << 31) ||
      static_cast<int64_t>(n_local) * local_cap >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  if (pools == nullptr || local_counts == nullptr || poolrow_to_row == nullptr || ws == nullptr ||
      dev_status == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_validate_compact_workspace_size(n_local, local_cap))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = as_cuda(stream);
  int32_t* inv = static_cast<int32_t*>(ws);
  const int64_t n_targets = static_cast<int64_t>(n_local) * local_cap;
  const int64_t n_rows = static_cast<int64_t>(n_src) * pool_cap;
  const uint16_t* pl = reinterpret_cast<const uint16_t*>(pools);
  launch(fill_minus_one, dim3(grid_of(n_targets)), dim3(kValThreads), 0, s, n_targets, inv);
  launch(validate_compact_kernel, dim3(grid_of(n_rows > n_local ? n_rows : n_local)),
         dim3(kValThreads), 0, s, n_src, pool_cap, d, n_local, local_cap, first_source, pl,
         local_counts, poolrow_to_row, inv, dev_status);
  launch(validate_compact_drops_kernel, dim3(grid_of(n_rows)), dim3(kValThreads), 0, s, n_src,
         pool_cap, d, n_local, local_cap, first_source, pl, local_counts, poolrow_to_row,
         static_cast<const int32_t*>(inv), dev_status);
  launch(validate_targets_kernel, dim3(grid_of(n_targets)), dim3(kValThreads), 0, s, n_targets,
         local_cap, local_counts, static_cast<const int32_t*>(inv), dev_status);
  return launch_status();
}
