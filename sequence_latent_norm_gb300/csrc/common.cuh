// Shared device helpers of the LAGA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define LAGA_DEVINL __device__ __forceinline__

namespace laga {

// Internal ("canonical") head dimensions every tensor-core kernel is built
// for: the DeepSeek-V3 dims of the page's evaluation (Section 4.1).  Smaller
// problem dims are zero-padded up to these by the prologue kernels; zero
// columns add exact zeros to every dot product, so results are unchanged.
constexpr int DN = 128;          // d_nope
constexpr int DR = 64;           // d_rope
constexpr int DV = 128;          // d_v
constexpr int DKV = 512;         // d_kv
constexpr int DQK = DN + DR;     // 192
constexpr int DH = DN + DV;      // 256: one head's [k_nope | v] columns

// Error codes written to the device error word (mirrors laga_status).
constexpr int DEV_ERR_TIMEOUT = 6;

LAGA_DEVINL float to_f32(float x) { return x; }
LAGA_DEVINL float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> LAGA_DEVINL T from_f32(float x);
template <> LAGA_DEVINL float from_f32<float>(float x) { return x; }
template <> LAGA_DEVINL __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

LAGA_DEVINL float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Layout of the per-head K/V tensor [.., 256]: element (b, s, h, e) sits at
// b*sb + s*ss + h*sh + e.  Token-major (LAGA) and head-major (explicit form)
// differ only in these strides.
struct KVLayout {
  long long sb, ss, sh;
  LAGA_DEVINL long long at(int b, int s, int h) const { return b * sb + s * ss + h * sh; }
};

}  // namespace laga
