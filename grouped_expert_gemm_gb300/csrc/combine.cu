// Combine: gate-weighted scatter-add of expert output rows back to token order.
//
// [M6.6] 0x03C3 "Round-Trip Identity And Weighted Combine" and 0x0CD; [M6.2]
// 0x03C: out[t] = sum over the token's surviving routes of g_r * z_r, with the
// gate applied once, after the expert ([M6.6] 0x0AE), and fp32 accumulation of
// bf16 returned rows.  [POOL] 03: waves add into one fp32 accumulator
// (accumulate != 0).
//
// One block owns one token at a time (grid-stride over tokens; with few tokens,
// one column part of a token).  The token's k row indices and gates are staged
// once in shared memory; each thread then
// handles 16-byte column chunks, issuing all k (up to KMAX) independent 16-byte
// loads of y for UNROLL chunks before using them, sums in fp32 in slot order,
// and writes two 16-byte fp32 stores per chunk.  No atomics: each output element
// has exactly one writer, so the result is deterministic.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kCombThreads = 128;

template <int KMAX>
__global__ void __launch_bounds__(kCombThreads)
combine_kernel(int T, int k, int chunks, int parts, const uint4* __restrict__ y, int64_t y_rows,
               const int32_t* __restrict__ route_to_row, const float* __restrict__ gates,
               const uint4* __restrict__ shared_y, int accumulate, float4* __restrict__ out,
               uint32_t* __restrict__ dev_status, const int32_t* __restrict__ valid, bool early) {
  pdl_wait_then_trigger(early);
  constexpr int UNROLL = KMAX >= 8 ? 1 : (KMAX >= 4 ? 2 : 4);
  __shared__ int32_t s_row[KMAX];
  __shared__ float s_gate[KMAX];
  const int64_t T_live = valid == nullptr ? T : min(static_cast<int64_t>(T),
                                                    static_cast<int64_t>(max(__ldg(valid), 0)));
  // Padding slots of a fixed token bucket get a zero output (left as they are
  // when accumulating): they never receive a routed contribution.
  for (int64_t t = T_live + blockIdx.x; t < T; t += gridDim.x) {
    if (accumulate) break;
    for (int c = threadIdx.x; c < chunks; c += kCombThreads) {
      out[(t * chunks + c) * 2] = make_float4(0.f, 0.f, 0.f, 0.f);
      out[(t * chunks + c) * 2 + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // A block owns one (token, column part) unit at a time; parts > 1 only when
  // there are too few tokens to give every SM work.
  const int per = (chunks + parts - 1) / parts;
  for (int64_t u0 = blockIdx.x; u0 < T_live * parts; u0 += gridDim.x) {
    const int64_t t = u0 / parts;
    const int c_lo = static_cast<int>(u0 % parts) * per, c_hi = min(chunks, c_lo + per);
    if (threadIdx.x < KMAX) {
      int32_t r = -1;
      float g = 0.0f;
      if (threadIdx.x < k) {
        r = __ldg(route_to_row + t * k + threadIdx.x);
        g = gates != nullptr ? __ldg(gates + t * k + threadIdx.x) : 1.0f;
        if (r >= 0 && r >= y_rows) {
          report(dev_status, MOE_DEV_BAD_ROW);
          r = -1;
        }
      }
      s_row[threadIdx.x] = r;
      s_gate[threadIdx.x] = g;
    }
    __syncthreads();
    for (int c0 = c_lo + threadIdx.x; c0 < c_hi; c0 += kCombThreads * UNROLL) {
      uint4 v[UNROLL][KMAX];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int c = c0 + u * kCombThreads;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (c < c_hi && s_row[j] >= 0)
            v[u][j] = __ldg(y + static_cast<int64_t>(s_row[j]) * chunks + c);
      }
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int c = c0 + u * kCombThreads;
        if (c >= c_hi) continue;
        float acc[8];
        float4* o = out + (t * chunks + c) * 2;
        if (accumulate) {
          const float4 a = o[0], b = o[1];
          acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
          acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        }
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (s_row[j] >= 0) {
            float f[8];
            unpack8(v[u][j], f);
            const float g = s_gate[j];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, f[i], acc[i]);
          }
        }
        if (shared_y != nullptr) {
          float f[8];
          unpack8(__ldg(shared_y + t * chunks + c), f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] += f[i];
        }
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      }
    }
    __syncthreads();
  }
  if (!early) pdl_trigger();
}

}  // namespace
}  // namespace moe

using namespace moe;

// Shared by moe_combine (gates given) and moe_unpermute_grad (unit gates).
static moe_status combine_impl(int32_t T, int32_t k, int32_t d, const moe_bf16* y, int64_t y_rows,
                               const int32_t* route_to_row, const float* gates,
                               const moe_bf16* shared_y, int32_t accumulate, float* out,
                               uint32_t* dev_status, moe_stream_t stream,
                               const int32_t* valid = nullptr);

MOE_API moe_status moe_combine(int32_t T, int32_t k, int32_t d, const moe_bf16* y, int64_t y_rows,
                               const int32_t* route_to_row, const float* gates,
                               const moe_bf16* shared_y, int32_t accumulate, float* out,
                               uint32_t* dev_status, moe_stream_t stream) {
  if (T > 0 && gates == nullptr) return MOE_ERR_INVALID_ARG;
  return combine_impl(T, k, d, y, y_rows, route_to_row, gates, shared_y, accumulate, out,
                      dev_status, stream);
}

MOE_API moe_status moe_combine_bucket(int32_t T, int32_t k, int32_t d, const int32_t* valid_tokens,
                                      const moe_bf16* y, int64_t y_rows,
                                      const int32_t* route_to_row, const float* gates,
                                      const moe_bf16* shared_y, int32_t accumulate, float* out,
                                      uint32_t* dev_status, moe_stream_t stream) {
  if (valid_tokens == nullptr || (T > 0 && gates == nullptr)) return MOE_ERR_INVALID_ARG;
  return combine_impl(T, k, d, y, y_rows, route_to_row, gates, shared_y, accumulate, out,
                      dev_status, stream, valid_tokens);
}

MOE_API moe_status moe_unpermute_grad(int32_t T, int32_t k, int32_t d, const moe_bf16* dx_perm,
                                      int64_t rows, const int32_t* route_to_row, float* dx,
                                      int32_t accumulate, uint32_t* dev_status,
                                      moe_stream_t stream) {
  return combine_impl(T, k, d, dx_perm, rows, route_to_row, nullptr, nullptr, accumulate, dx,
                      dev_status, stream);
}

static moe_status combine_impl(int32_t T, int32_t k, int32_t d, const moe_bf16* y, int64_t y_rows,
                               const int32_t* route_to_row, const float* gates,
                               const moe_bf16* shared_y, int32_t accumulate, float* out,
                               uint32_t* dev_status, moe_stream_t stream, const int32_t* valid) {
  if (T < 0 || k <= 0 || d <= 0 || y_rows < 0) return MOE_ERR_INVALID_ARG;
  if (k > 16 || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (out == nullptr || route_to_row == nullptr || (y == nullptr && y_rows > 0))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(out) || (y != nullptr && !aligned16(y)) ||
      (shared_y != nullptr && !aligned16(shared_y)))
    return MOE_ERR_UNSUPPORTED;
  const int chunks = d / 8;
  cudaStream_t s = as_cuda(stream);
  // Column parts while that still leaves a chunk per thread and fewer than two
  // blocks per SM would otherwise have work (decode).
  int parts = 1;
  while (static_cast<int64_t>(T) * parts * 2 <= 152 * 2 && chunks / (parts * 2) >= kCombThreads)
    parts *= 2;
  const int64_t units = static_cast<int64_t>(T) * parts;
  const unsigned grid = static_cast<unsigned>(units < 152 * 24 ? units : 152 * 24);
#define MOE_COMBINE_CASE(K)                                                                 \
  launch(combine_kernel<K>, dim3(grid), dim3(kCombThreads), 0, s, T, k, chunks, parts,        \
         reinterpret_cast<const uint4*>(y), y_rows, route_to_row, gates,                      \
         reinterpret_cast<const uint4*>(shared_y), static_cast<int>(accumulate),              \
         reinterpret_cast<float4*>(out), dev_status, valid, one_wave(grid))
  if (k <= 1) MOE_COMBINE_CASE(1);
  else if (k <= 2) MOE_COMBINE_CASE(2);
  else if (k <= 4) MOE_COMBINE_CASE(4);
  else if (k <= 8) MOE_COMBINE_CASE(8);
  else MOE_COMBINE_CASE(16);
#undef MOE_COMBINE_CASE
  return launch_status();
}
