// Library-level entry points of the C ABI: version, status strings, capacity.
#include "common.cuh"

MOE_API int32_t moe_version(void) { return 100; /* 0.1.0 */ }

MOE_API const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA launch or driver call failed";
    default: return "unknown status";
  }
}

// ceil(cf_num * assignments / (cf_den * slots)), exact in 128-bit integers.
// [M6.2] 0x01C: C = ceil(c_f * T * k / E).  [POOL] 04: the sender pool and
// receiver array capacities use the same rule with slots = n_dest * n_waves and
// n_local * n_waves.
MOE_API int64_t moe_capacity(int64_t cf_num, int64_t cf_den, int64_t assignments, int64_t slots) {
  if (cf_num < 0 || cf_den <= 0 || assignments < 0 || slots <= 0) return -1;
  const __int128 num = static_cast<__int128>(cf_num) * assignments;
  const __int128 den = static_cast<__int128>(cf_den) * slots;
  const __int128 q = (num + den - 1) / den;
  if (q > static_cast<__int128>(INT64_MAX)) return -1;
  return static_cast<int64_t>(q);
}
