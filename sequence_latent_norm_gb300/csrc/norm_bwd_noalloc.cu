// LayerNorm + RoPE backward (the a7 step) for callers that cannot allocate
// device memory.
//
// Some callers cannot hand this library a scratch buffer.  Examples: a
// runtime that reserves the whole device up front for its own pool and
// forbids any further cudaMalloc while a step runs, or an embedding that
// only owns the tensors it passes in.  The regular backward needs a
// caller-provided workspace, including the partial sums of dgamma.  This
// entry point keeps that scratch in a fixed-size array of this library's
// own device memory instead, so it calls no cudaMalloc, cudaFree or
// allocating library routine.
//
// The scratch (kParts x 512 fp32 = 592 KiB) exists once per device that
// loads the library and lives until the process exits.  Every call shares
// it, so two calls whose kernels overlap on the GPU (different streams, no
// ordering between them) race on it.  Each call overwrites every partial
// row it later reads, so nothing is carried over from the previous call and
// nothing has to be cleared.
#include <mutex>

#include "../../include/laga.h"
#include "common.cuh"
#include "plan.h"

namespace laga {
namespace {

constexpr int kParts = 296;   // dgamma partial rows (blocks of the first kernel)
constexpr int kCols = 512;    // largest d_kv the scratch holds
constexpr int kWarps = 8;

static __device__ __align__(256) float g_noalloc_dgamma_part[kParts * kCols];

// Device address of the scratch for each device, looked up on the first
// call made with that device current.
constexpr int kMaxDev = 64;
float* g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;

laga_status scratch_on_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return LAGA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_dgamma_part) != cudaSuccess) return LAGA_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return LAGA_OK;
}

// One warp per token: recompute the norm statistics of the latent,
// dx = rstd (g - mean(g) - xhat mean(g xhat)) with g = dL * gamma (no
// mean(g) term for the RMS variant, whose mean is 0), the
// block's dgamma partial sums, and the k_pe gradient summed over heads in
// head order and rotated back.
template <typename T>
__global__ void __launch_bounds__(256) noalloc_norm_rope_bwd_kernel(
    const T* __restrict__ c, const float* __restrict__ gamma, const float* __restrict__ cosT,
    const float* __restrict__ sinT, const float* __restrict__ dL,
    const float* __restrict__ dkpe_h, int B, int S, int H, int dr, int dkv, float eps, int rms,
    float* __restrict__ dc, float* __restrict__ part) {
  __shared__ float red[kWarps][kCols];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float dg[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) dg[i] = 0.f;
  const long long tokens = (long long)B * S;
  const int half = dr >> 1;
  for (long long tok = (long long)blockIdx.x * kWarps + warp; tok < tokens;
       tok += (long long)gridDim.x * kWarps) {
    const T* crow = c + tok * (dkv + dr);
    float x[16];
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int col = lane + 32 * i;
      x[i] = col < dkv ? to_f32(crow[col]) : 0.f;
      sum += x[i];
    }
    const float mu = rms ? 0.f : warp_sum(sum) / dkv;   // RMS variant: no centring
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int col = lane + 32 * i;
      const float d = col < dkv ? x[i] - mu : 0.f;
      sq += d * d;
    }
    const float rs = 1.0f / sqrtf(warp_sum(sq) / dkv + eps);
    const float* gL = dL + tok * dkv;
    float xh[16], g[16];
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int col = lane + 32 * i;
      const bool ok = col < dkv;
      xh[i] = ok ? (x[i] - mu) * rs : 0.f;
      const float d = ok ? gL[col] : 0.f;
      g[i] = ok ? d * gamma[col] : 0.f;
      dg[i] += d * xh[i];
      s1 += g[i];
      s2 += g[i] * xh[i];
    }
    const float m1 = rms ? 0.f : warp_sum(s1) / dkv, m2 = warp_sum(s2) / dkv;
    float* drow = dc + tok * (dkv + dr);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int col = lane + 32 * i;
      if (col < dkv) drow[col] = rs * (g[i] - m1 - xh[i] * m2);
    }
    if (lane < half) {
      const int s = (int)(tok % S);
      float a = 0.f, b = 0.f;
      for (int h = 0; h < H; ++h) {
        const float* src = dkpe_h + (tok * H + h) * dr;
        a += src[lane];
        b += src[lane + half];
      }
      const float cs = cosT[(long long)s * half + lane], sn = sinT[(long long)s * half + lane];
      drow[dkv + lane] = a * cs + b * sn;
      drow[dkv + lane + half] = b * cs - a * sn;
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) red[warp][lane + 32 * i] = dg[i];
  __syncthreads();
  for (int col = threadIdx.x; col < kCols; col += 256) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += red[w][col];
    part[(long long)blockIdx.x * kCols + col] = t;  // every row and column rewritten
  }
}

__global__ void noalloc_dgamma_reduce_kernel(const float* __restrict__ part, int dkv,
                                             float* __restrict__ dgamma) {
  const int col = blockIdx.x * blockDim.x + threadIdx.x;
  if (col >= dkv) return;
  float t = 0.f;
  for (int p = 0; p < kParts; ++p) t += part[(long long)p * kCols + col];
  dgamma[col] = t;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace laga

using namespace laga;

extern "C" laga_status laga_norm_rope_bwd_noalloc(const laga_dims* dims, const void* c,
                                                  const float* gamma, const float* cos,
                                                  const float* sin, const float* d_latent,
                                                  const float* d_kpe_rot, float* dc,
                                                  float* dgamma, void* stream) {
  if (dims && dims->d_kv > kCols) return LAGA_ERR_WORKSPACE;  // beyond the static scratch
  Plan p;
  laga_status s = make_plan(dims, &p);
  if (s != LAGA_OK) return s;
  const void* ptrs[] = {c, gamma, cos, sin, d_latent, d_kpe_rot, dc, dgamma};
  for (const void* ptr : ptrs)
    if (!ptr) return LAGA_ERR_ARG;
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return LAGA_ERR_ALIGN;
  float* part = nullptr;
  if ((s = scratch_on_current_device(&part)) != LAGA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.fp32)
    noalloc_norm_rope_bwd_kernel<float><<<kParts, 256, 0, st>>>(
        static_cast<const float*>(c), gamma, cos, sin, d_latent, d_kpe_rot, p.B, p.S, p.H, p.dr,
        p.dkv, p.d.ln_eps, (int)p.rms, dc, part);
  else
    noalloc_norm_rope_bwd_kernel<__nv_bfloat16><<<kParts, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(c), gamma, cos, sin, d_latent, d_kpe_rot, p.B, p.S, p.H,
        p.dr, p.dkv, p.d.ln_eps, (int)p.rms, dc, part);
  if (cudaGetLastError() != cudaSuccess) return LAGA_ERR_CUDA;
  noalloc_dgamma_reduce_kernel<<<(p.dkv + 127) / 128, 128, 0, st>>>(part, p.dkv, dgamma);
  return cudaGetLastError() == cudaSuccess ? LAGA_OK : LAGA_ERR_CUDA;
}
