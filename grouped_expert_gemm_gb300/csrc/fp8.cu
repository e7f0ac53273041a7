// FP8 dispatch payload: E4M3 quantization with fp32 scales (one per row or one
// per 128 values of a row), its inverse, and the logical payload ledger.
//
// [M6.6] 0x0AB "Deriving BF16 And FP8 Payloads" (byte formulas), 0x0AC "Scale
// Tensor Ownership And Row Trace" (data and scales are one pair), 0x0AE (the
// dispatch activation may be BF16 or FP8 plus FP32 scales).
//
// One warp per row, 16-byte accesses.  Whole-row scales take two passes over
// the row (the largest magnitude first, then the codes; the second read hits
// L1/L2); 128-value groups are handled by half-warps in one pass (16 lanes x 8
// values = one group).  Every quotient is an IEEE-rounded fp32 division and the
// E4M3 conversion rounds to nearest even with saturation, so the codes are a
// deterministic function of the bf16 input.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kQThreads = 256;
constexpr int kQUnroll = 4;  // 16-byte loads in flight per lane
constexpr float kE4M3Max = 448.0f;
constexpr uint32_t kAbsInf = 0x7F800000u;

// Largest |x| bit pattern of 8 bf16 values (as fp32 bits: for non-negative
// values the integer order of the bits is the numeric order, NaN above Inf).
__device__ __forceinline__ uint32_t amax_bits8(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = max(m, (w[i] << 16) & 0x7FFFFFFFu);
    m = max(m, w[i] & 0x7FFF0000u);
  }
  return m;
}

__device__ __forceinline__ float scale_of(uint32_t amax) {
  return amax == 0 ? 1.0f : __fdiv_rn(__uint_as_float(amax), kE4M3Max);
}

// 8 bf16 values -> 8 E4M3 codes (byte order = element order).
__device__ __forceinline__ uint2 quant8(const uint4& v, float s) {
  float f[8];
  unpack8(v, f);
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    p[i] = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(f[2 * i], s), __fdiv_rn(f[2 * i + 1], s)),
                                    __NV_SATFINITE, __NV_E4M3);
  return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

template <bool ROW>
__global__ void __launch_bounds__(kQThreads)
quantize_kernel(int64_t n, int d, int G, const uint4* __restrict__ x, uint2* __restrict__ q,
                float* __restrict__ scales, uint32_t* __restrict__ dev_status) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int chunks = d / 8;  // 8 values per 16-byte chunk
  bool bad = false;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5); row < n;
       row += static_cast<int64_t>(gridDim.x) * warps) {
    const uint4* xr = x + row * chunks;
    uint2* qr = q + row * chunks;
    if constexpr (ROW) {
      // largest magnitude first (four 16-byte loads in flight per lane), then the codes
      uint32_t m = 0;
      for (int cb = 0; cb < chunks; cb += 32 * kQUnroll) {
        uint4 v[kQUnroll];
#pragma unroll
        for (int u = 0; u < kQUnroll; ++u) {
          const int c = cb + u * 32 + lane;
          v[u] = c < chunks ? __ldg(xr + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kQUnroll; ++u) m = max(m, amax_bits8(v[u]));
      }
      m = __reduce_max_sync(0xFFFFFFFFu, m);
      if (m >= kAbsInf) bad = true;
      const float s = scale_of(m);
      if (lane == 0) scales[row] = s;
      for (int cb = 0; cb < chunks; cb += 32 * kQUnroll) {
        uint4 v[kQUnroll];
#pragma unroll
        for (int u = 0; u < kQUnroll; ++u) {
          const int c = cb + u * 32 + lane;
          if (c < chunks) v[u] = __ldg(xr + c);
        }
#pragma unroll
        for (int u = 0; u < kQUnroll; ++u) {
          const int c = cb + u * 32 + lane;
          if (c < chunks) qr[c] = quant8(v[u], s);
        }
      }
    } else {
      // Half-warp h of sub-iteration u owns group 2*(cb/32 + u) + h (chunks 16g .. 16g+15).
      for (int cb = 0; cb < chunks; cb += 32 * kQUnroll) {
        uint4 v[kQUnroll];
#pragma unroll
        for (int u = 0; u < kQUnroll; ++u) {
          const int c = cb + u * 32 + lane;
          v[u] = c < chunks ? __ldg(xr + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kQUnroll; ++u) {
          const int c = cb + u * 32 + lane;
          const bool live = c < chunks;
          uint32_t m = amax_bits8(v[u]);
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
          if (m >= kAbsInf && live) bad = true;
          const float s = scale_of(m);
          if (live && (c & 15) == 0) scales[row * G + (c >> 4)] = s;
          if (live) qr[c] = quant8(v[u], s);
        }
      }
    }
  }
  if (bad) report(dev_status, MOE_DEV_NONFINITE_INPUT);
  pdl_trigger();
}

// One warp per row, kDqUnroll 16-code chunks in flight per lane.  A chunk's
// scale is the row's (one group) or that of its 128-value group (chunk c / 8).
constexpr int kDqUnroll = 4;

__global__ void __launch_bounds__(kQThreads)
dequantize_kernel(int64_t n, int d, int G, const uint4* __restrict__ q,
                  const float* __restrict__ scales, uint4* __restrict__ x) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int per_row = d / 16;  // 16 codes per chunk
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5); row < n;
       row += static_cast<int64_t>(gridDim.x) * warps) {
    const uint4* qr = q + row * per_row;
    uint4* xr = x + row * per_row * 2;
    const float* sr = scales + row * G;
    for (int cb = 0; cb < per_row; cb += 32 * kDqUnroll) {
      uint4 v[kDqUnroll];
      float sc[kDqUnroll];
#pragma unroll
      for (int u = 0; u < kDqUnroll; ++u) {
        const int c = cb + u * 32 + lane;
        if (c < per_row) {
          v[u] = __ldg(qr + c);
          sc[u] = __ldg(sr + (G == 1 ? 0 : (c >> 3)));
        }
      }
#pragma unroll
      for (int u = 0; u < kDqUnroll; ++u) {
        const int c = cb + u * 32 + lane;
        if (c < per_row) {
          uint4 lo, hi;
          dequant16(v[u], sc[u], lo, hi);
          xr[2 * c] = lo;
          xr[2 * c + 1] = hi;
        }
      }
    }
  }
  pdl_trigger();
}

int64_t n_groups(int32_t d, int32_t group) { return group == 0 ? 1 : ceil_div(d, group); }

moe_status check_fp8_shape(int64_t n, int32_t d, int32_t group) {
  if (n < 0 || d <= 0) return MOE_ERR_INVALID_ARG;
  if (group != MOE_SCALE_ROW && group != MOE_SCALE_BLOCK128) return MOE_ERR_INVALID_ARG;
  if (d % 16 != 0 || d > (1 << 20)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

unsigned grid_for(int64_t work_items, int per_block) {
  int64_t b = ceil_div(work_items, per_block);
  if (b > 152 * 16) b = 152 * 16;
  return static_cast<unsigned>(b < 1 ? 1 : b);
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API int64_t moe_payload_bytes(int64_t rows, int32_t d, int32_t payload) {
  if (rows < 0 || d < 1) return -1;
  switch (payload) {
    case MOE_PAYLOAD_BF16: return rows * d * 2;
    case MOE_PAYLOAD_FP8_ROW: return rows * d + rows * 4;
    case MOE_PAYLOAD_FP8_BLOCK128: return rows * d + rows * ceil_div(d, 128) * 4;
    default: return -1;
  }
}

MOE_API moe_status moe_quantize_fp8(int64_t n, int32_t d, int32_t group, const moe_bf16* x,
                                    moe_fp8* q, float* scales, uint32_t* dev_status,
                                    moe_stream_t stream) {
  moe_status st = check_fp8_shape(n, d, group);
  if (st != MOE_OK || n == 0) return st;
  if (x == nullptr || q == nullptr || scales == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
    return MOE_ERR_UNSUPPORTED;
  const int G = static_cast<int>(n_groups(d, group));
  const unsigned grid = grid_for(n, kQThreads / 32);
  cudaStream_t s = as_cuda(stream);
  if (group == MOE_SCALE_ROW)
    launch(quantize_kernel<true>, dim3(grid), dim3(kQThreads), 0, s, n, d, G,
           reinterpret_cast<const uint4*>(x), reinterpret_cast<uint2*>(q), scales, dev_status);
  else
    launch(quantize_kernel<false>, dim3(grid), dim3(kQThreads), 0, s, n, d, G,
           reinterpret_cast<const uint4*>(x), reinterpret_cast<uint2*>(q), scales, dev_status);
  return launch_status();
}

MOE_API moe_status moe_dequantize_fp8(int64_t n, int32_t d, int32_t group, const moe_fp8* q,
                                      const float* scales, moe_bf16* x, moe_stream_t stream) {
  moe_status st = check_fp8_shape(n, d, group);
  if (st != MOE_OK || n == 0) return st;
  if (x == nullptr || q == nullptr || scales == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
    return MOE_ERR_UNSUPPORTED;
  const int G = static_cast<int>(n_groups(d, group));
  launch(dequantize_kernel, dim3(grid_for(n, kQThreads / 32)), dim3(kQThreads), 0, as_cuda(stream),
         n, d, G, reinterpret_cast<const uint4*>(q), scales, reinterpret_cast<uint4*>(x));
  return launch_status();
}
