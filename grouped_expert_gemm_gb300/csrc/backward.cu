// Backward of the weighted combine (the reverse of the semantic transpose).
//
// [M6.2] 0x03D "Backward Is The Reverse Semantic Transpose": with upstream
// gradient dout[t] of out[t] = sum_j g[t,j] * y[row(t,j)],
//   dy[row(t,j)]  = g[t,j] * dout[t]        (bf16, the expert output gradient)
//   dgates[t,j]   = <dout[t], y[row(t,j)]>   (fp32)
// and the route-input gradients return to their tokens through the saved
// inverse map (moe_unpermute_grad, the combine kernel with unit gates).
//
// One block owns one token at a time: the token's k rows and gates are staged
// in shared memory; each thread walks 16-byte column chunks, loads dout once
// and each accepted route's y chunk once (all loads of a chunk issued before
// use), writes the scaled dy chunk and keeps per-slot partial dot products in
// fp32, which are reduced across the block at the end of the token.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kBwdThreads = 128;
constexpr int kBwdWarps = kBwdThreads / 32;

template <int KMAX>
__global__ void __launch_bounds__(kBwdThreads)
combine_backward_kernel(int T, int k, int chunks, const float4* __restrict__ dout,
                        const uint4* __restrict__ y, int64_t y_rows,
                        const int32_t* __restrict__ route_to_row, const float* __restrict__ gates,
                        uint4* __restrict__ dy, float* __restrict__ dgates,
                        uint32_t* __restrict__ dev_status) {
  pdl_wait();
  __shared__ int32_t s_row[KMAX];
  __shared__ float s_gate[KMAX];
  __shared__ float s_dot[kBwdWarps][KMAX];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    if (threadIdx.x < KMAX) {
      int32_t r = -1;
      float g = 0.0f;
      if (threadIdx.x < k) {
        r = __ldg(route_to_row + t * k + threadIdx.x);
        g = __ldg(gates + t * k + threadIdx.x);
        if (r >= 0 && r >= y_rows) {
          report(dev_status, MOE_DEV_BAD_ROW);
          r = -1;
        }
      }
      s_row[threadIdx.x] = r;
      s_gate[threadIdx.x] = g;
    }
    __syncthreads();
    float dot[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) dot[j] = 0.0f;
    for (int c = threadIdx.x; c < chunks; c += kBwdThreads) {
      const float4 a = __ldg(dout + (t * chunks + c) * 2);
      const float4 b = __ldg(dout + (t * chunks + c) * 2 + 1);
      const float o[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint4 v[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (s_row[j] >= 0) v[j] = __ldg(y + static_cast<int64_t>(s_row[j]) * chunks + c);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (s_row[j] < 0) continue;
        float f[8];
        unpack8(v[j], f);
        float acc = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = fmaf(o[i], f[i], acc);
        dot[j] += acc;
        const float g = s_gate[j];
        dy[static_cast<int64_t>(s_row[j]) * chunks + c] =
            make_uint4(pack_bf16x2(g * o[0], g * o[1]), pack_bf16x2(g * o[2], g * o[3]),
                       pack_bf16x2(g * o[4], g * o[5]), pack_bf16x2(g * o[6], g * o[7]));
      }
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      float v = dot[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      if (lane == 0) s_dot[w][j] = v;
    }
    __syncthreads();
    if (threadIdx.x < k) {
      float sum = 0.0f;
      for (int ww = 0; ww < kBwdWarps; ++ww) sum += s_dot[ww][threadIdx.x];
      dgates[t * k + threadIdx.x] = s_row[threadIdx.x] >= 0 ? sum : 0.0f;
    }
    __syncthreads();
  }
  pdl_trigger();
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API moe_status moe_combine_backward(int32_t T, int32_t k, int32_t d, const float* dout,
                                        const moe_bf16* y, int64_t y_rows,
                                        const int32_t* route_to_row, const float* gates,
                                        moe_bf16* dy, float* dgates, uint32_t* dev_status,
                                        moe_stream_t stream) {
  if (T < 0 || k <= 0 || d <= 0 || y_rows < 0) return MOE_ERR_INVALID_ARG;
  if (k > 16 || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (dout == nullptr || route_to_row == nullptr || gates == nullptr || dgates == nullptr ||
      ((y == nullptr || dy == nullptr) && y_rows > 0))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(dout) || (y != nullptr && !aligned16(y)) || (dy != nullptr && !aligned16(dy)))
    return MOE_ERR_UNSUPPORTED;
  const int chunks = d / 8;
  cudaStream_t s = as_cuda(stream);
  const dim3 grid(static_cast<unsigned>(T < 152 * 24 ? T : 152 * 24));
#define MOE_BWD_CASE(K)                                                                      \
  launch(combine_backward_kernel<K>, grid, dim3(kBwdThreads), 0, s, T, k, chunks,           \
         reinterpret_cast<const float4*>(dout), reinterpret_cast<const uint4*>(y), y_rows,  \
         route_to_row, gates, reinterpret_cast<uint4*>(dy), dgates, dev_status)
  if (k <= 2) MOE_BWD_CASE(2);
  else if (k <= 4) MOE_BWD_CASE(4);
  else if (k <= 8) MOE_BWD_CASE(8);
  else MOE_BWD_CASE(16);
#undef MOE_BWD_CASE
  return launch_status();
}
