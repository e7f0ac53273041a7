// Load telemetry and the delayed bias controller on device.
//
// [M6.2] 0x01I (skew summaries of a count vector n over U units, mu = R / U):
//   CV^2 = mean((n - mu)^2) / mu^2, rho_max = max n / mu, with q = n / R and
//   0 log 0 = 0: H_norm = -sum q log q / log U, E_eff = exp(-sum q log q),
//   MaxVio = (max n - mu) / mu (0x06J2).
// [M6.2] 0x01I demand n_e (routes that chose expert e, before any capacity):
//   a shared-memory histogram per block over a slice of the routes, merged with
//   one global atomic per non-empty bin.
// [M6.2] 0x06E and 0x06J1-0x06J3 (the controller acts on the counts of the
// batch just routed): b_e <- b_e + u * sign(mean c - c_e), or with the
// proportional rule b_e <- b_e + u * (mean c - c_e).
//
// One block of 256 threads: fp64 block reductions over the count vector.  The
// bias increment is formed in fp64 and rounded to fp32 once, then added with one
// fp32 rounding, so the result is reproducible bit for bit.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kTelThreads = 256;

__device__ double block_sum(double v, double* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  double t = 0.0;
  for (int i = 0; i < kTelThreads / 32; ++i) t += sh[i];
  return t;
}

__device__ double block_max(double v, double* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  double t = sh[0];
  for (int i = 1; i < kTelThreads / 32; ++i) t = fmax(t, sh[i]);
  return t;
}

__global__ void __launch_bounds__(kTelThreads)
load_stats_kernel(int U, const int32_t* __restrict__ counts, double* __restrict__ stats) {
  pdl_wait();
  __shared__ double sh[kTelThreads / 32];
  double r = 0.0, mx = 0.0;
  for (int u = threadIdx.x; u < U; u += kTelThreads) {
    const double n = static_cast<double>(max(__ldg(counts + u), 0));
    r += n;
    mx = fmax(mx, n);
  }
  const double R = block_sum(r, sh);
  const double M = block_max(mx, sh);
  double out[5] = {0.0, 0.0, 0.0, 0.0, 0.0};
  if (R > 0.0) {
    const double mu = R / U;
    double dev = 0.0, ent = 0.0;
    for (int u = threadIdx.x; u < U; u += kTelThreads) {
      const double n = static_cast<double>(max(__ldg(counts + u), 0));
      dev += (n - mu) * (n - mu);
      if (n > 0.0) {
        const double q = n / R;
        ent -= q * log(q);
      }
    }
    const double D = block_sum(dev, sh);
    const double H = block_sum(ent, sh);
    out[0] = (D / U) / (mu * mu);
    out[1] = M / mu;
    out[2] = U > 1 ? H / log(static_cast<double>(U)) : 0.0;
    out[3] = exp(H);
    out[4] = (M - mu) / mu;
  }
  if (threadIdx.x < 5) stats[threadIdx.x] = out[threadIdx.x];
  pdl_trigger();
}

__global__ void __launch_bounds__(kTelThreads)
bias_update_kernel(int E, const int32_t* __restrict__ counts, float* __restrict__ bias, float u,
                   int rule) {
  pdl_wait();
  __shared__ double sh[kTelThreads / 32];
  double r = 0.0;
  for (int e = threadIdx.x; e < E; e += kTelThreads) r += static_cast<double>(__ldg(counts + e));
  const double mean = block_sum(r, sh) / E;
  for (int e = threadIdx.x; e < E; e += kTelThreads) {
    const double err = mean - static_cast<double>(__ldg(counts + e));
    const double step = rule == MOE_BIAS_SIGN ? (err > 0.0 ? 1.0 : (err < 0.0 ? -1.0 : 0.0)) : err;
    const float inc = __double2float_rn(static_cast<double>(u) * step);
    bias[e] = __fadd_rn(bias[e], inc);
  }
  pdl_trigger();
}

constexpr int kDemandThreads = 256;
constexpr int kDemandRoutesPerBlock = 2048;

__global__ void __launch_bounds__(kDemandThreads)
demand_kernel(int R, int E, int k, const int32_t* __restrict__ valid,
              const int32_t* __restrict__ ids, int32_t* __restrict__ demand,
              uint32_t* __restrict__ dev_status) {
  __shared__ int32_t hist[512];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  pdl_wait();
  __syncthreads();
  int R_live = R;
  if (valid != nullptr) {
    const int v = __ldg(valid);
    R_live = v <= 0 ? 0 : min(R, v * k);
  }
  bool bad = false;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kDemandRoutesPerBlock;
  const int64_t r1 = min(static_cast<int64_t>(R_live), r0 + kDemandRoutesPerBlock);
  for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    const int e = __ldg(ids + r);
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else if (e != MOE_ROUTE_MASKED) bad = true;
  }
  if (bad) report(dev_status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (hist[e] != 0) atomicAdd(demand + e, hist[e]);
  pdl_trigger();
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API moe_status moe_expert_demand(int32_t T, int32_t k, int32_t E, const int32_t* valid_tokens,
                                     const int32_t* topk_ids, int32_t* demand,
                                     uint32_t* dev_status, moe_stream_t stream) {
  if (T < 0 || k <= 0 || E <= 0 || demand == nullptr) return MOE_ERR_INVALID_ARG;
  if (E > 512 || static_cast<int64_t>(T) * k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  const int R = T * k;
  if (R > 0 && topk_ids == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_cuda(stream);
  if (cudaMemsetAsync(demand, 0, static_cast<size_t>(E) * sizeof(int32_t), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (R == 0) return MOE_OK;
  launch(demand_kernel, dim3(static_cast<unsigned>(ceil_div(R, kDemandRoutesPerBlock))),
         dim3(kDemandThreads), 0, s, R, E, k, valid_tokens, topk_ids, demand, dev_status);
  return launch_status();
}

MOE_API moe_status moe_load_stats(int32_t U, const int32_t* counts, double* stats,
                                  moe_stream_t stream) {
  if (U <= 0 || counts == nullptr || stats == nullptr) return MOE_ERR_INVALID_ARG;
  launch(load_stats_kernel, dim3(1), dim3(kTelThreads), 0, as_cuda(stream), U, counts, stats);
  return launch_status();
}

MOE_API moe_status moe_bias_update(int32_t E, const int32_t* counts, float* bias, float u,
                                   int32_t rule, moe_stream_t stream) {
  if (E <= 0 || counts == nullptr || bias == nullptr) return MOE_ERR_INVALID_ARG;
  if (rule != MOE_BIAS_SIGN && rule != MOE_BIAS_PROPORTIONAL) return MOE_ERR_INVALID_ARG;
  launch(bias_update_kernel, dim3(1), dim3(kTelThreads), 0, as_cuda(stream), E, counts, bias, u,
         static_cast<int>(rule));
  return launch_status();
}
