// Shared device/host helpers of the MoE hot-path library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

constexpr int kWarp = 32;

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline cudaStream_t as_cuda(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch-error check used at the end of every entry point.
inline moe_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation.  Before its first global-memory access a
// kernel waits until the previous kernel has completed and its writes are
// visible (pdl_wait); when a block has finished its work it lets the next
// kernel of the stream start launching (pdl_trigger).  So the next kernel's
// launch and purely local set-up (shared memory, mbarriers, tensor memory,
// tensor-map prefetch) overlap the tail of the previous one, no data access
// ever does, and no waiting block sits beside a kernel's main work (triggering
// at entry instead slowed the pooled pack copy by 43 %).  Without the launch
// attribute both are no-ops.
//
// The exception is a kernel whose grid fits one wave (no more blocks than SMs):
// it triggers right after its own wait (pdl_wait_then_trigger).  Dependents can
// launch only once every block of the grid has triggered, so by then all of its
// blocks are resident and none can be kept waiting for a slot; the dependents'
// launch latency then hides behind its work instead of following its last block
// (one-token decode 39.0 -> 37.5 us per step, the 256-token tiny layer
// 25.2 -> 23.1 us).
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Wait for the previous kernel; then, with `early`, let the dependents launch.
// A kernel calling this ends with `if (!early) pdl_trigger();`.
__device__ __forceinline__ void pdl_wait_then_trigger(bool early) {
  pdl_wait();
  if (early) pdl_trigger();
}

// SM count of the current device, read once per device.
inline int sm_count() {
  constexpr int kMaxDev = 64;
  static int cache[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

// A grid of at most one block per SM is resident all at once.
inline bool one_wave(int64_t blocks) { return blocks <= sm_count(); }

template <typename... KArgs, typename... Args>
inline void launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                   Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ void report(uint32_t* dev_status, uint32_t bits) {
  if (dev_status != nullptr) atomicOr(dev_status, bits);
}

// Workspace carving: 256-byte aligned sub-buffers.
struct Carver {
  size_t off = 0;
  template <typename T>
  size_t take(size_t count) {
    size_t o = (off + 255) & ~size_t(255);
    off = o + count * sizeof(T);
    return o;
  }
};

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Unpack 8 bf16 held in a uint4 into 8 floats (element order preserved).
__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
  f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xFFFF0000u);
  f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xFFFF0000u);
  f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

// Pack two floats into bf16x2 with round-to-nearest-even (lo element first).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// E4M3 decoding by bit placement: a code's 7 magnitude bits moved to fp32 bits
// 20..26 (its 4 exponent bits become the low bits of the fp32 exponent field,
// its 3 mantissa bits the top of the fp32 mantissa) and its sign to bit 31 give
// exactly decode(code) * 2^-120 -- for subnormal codes too, since both formats
// continue their smallest binade linearly.  Multiplying by 2^120 is then exact,
// and the multiply by the scale is the one rounding of decode(code) * s to fp32.
// (NaN codes 0x7F / 0xFF, which moe_quantize_fp8 produces only from non-finite
// input, come out as +-480 * s.)  Four codes of one word at a time, two fp32
// lanes per multiply.
__device__ __forceinline__ void dequant4(uint32_t w, float s, uint32_t& bf01, uint32_t& bf23) {
  const float2 two120 = make_float2(0x1p120f, 0x1p120f);
  const float2 sc = make_float2(s, s);
  float2 a, b;
  a.x = __uint_as_float(((w << 24) & 0x80000000u) | ((w << 20) & 0x07F00000u));
  a.y = __uint_as_float(((w << 16) & 0x80000000u) | ((w << 12) & 0x07F00000u));
  b.x = __uint_as_float(((w << 8) & 0x80000000u) | ((w << 4) & 0x07F00000u));
  b.y = __uint_as_float((w & 0x80000000u) | ((w >> 4) & 0x07F00000u));
  a = __fmul2_rn(__fmul2_rn(a, two120), sc);
  b = __fmul2_rn(__fmul2_rn(b, two120), sc);
  bf01 = pack_bf16x2(a.x, a.y);
  bf23 = pack_bf16x2(b.x, b.y);
}

// 16 E4M3 codes (one uint4, element order = byte order) -> 16 bf16 in two uint4,
// each bf16(fp32(decode(code) * s)).
__device__ __forceinline__ void dequant16(const uint4& v, float s, uint4& lo, uint4& hi) {
  dequant4(v.x, s, lo.x, lo.y);
  dequant4(v.y, s, lo.z, lo.w);
  dequant4(v.z, s, hi.x, hi.y);
  dequant4(v.w, s, hi.z, hi.w);
}

}  // namespace moe
