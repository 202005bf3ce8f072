// a4/a5 causal MLA attention, forward and backward (Algorithm 1 step 5,
// Section 5.2).  scores = (q_nope||q_rope)(k_nope||k_pe)^T * scale with the
// RoPE'd k_pe shared by all heads; out = softmax(scores) v.
//
// Straightforward tiled kernels (64x64 tiles, fp32 in shared memory).  The
// backward is split in a key-stationary dK/dV pass and a query-stationary dQ
// pass so that every sum is taken in a fixed order (no atomics).
#include "common.cuh"
#include "kernels.h"

namespace laga {
namespace {

constexpr int BT = 64;          // query / key tile
constexpr int QS = DQK + 1;     // padded smem row strides (floats)
constexpr int VS = DV + 1;
constexpr int PS = BT + 1;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

struct AttnArgs {
  Views v;
  int B, S, H;
  float scale;
  const float* lse;     // [B,H,S]
  float* lse_out;
  const float* delta;   // [B,H,S]
  __nv_bfloat16* dkv;   // same layout as kv
  float* dkpe;          // [R,64]
  float* dq;            // [R,192]
};

LAGA_DEVINL long long rowid(int b, int s, int h, int S, int H) {
  return ((long long)b * S + s) * H + h;
}

// Q (or any [q_nope | q_rope_rot]) tile of 64 rows into smem as fp32.
LAGA_DEVINL void load_q_tile(float* Qs, const AttnArgs& a, int b, int h, int r0) {
  for (int i = threadIdx.x; i < BT * DQK; i += blockDim.x) {
    int rr = i / DQK, d = i % DQK, s = r0 + rr;
    float val = 0.f;
    if (s < a.S) {
      long long row = rowid(b, s, h, a.S, a.H);
      val = d < DN ? __bfloat162float(a.v.qn[row * a.v.qn_ld + d])
                   : __bfloat162float(a.v.qr[row * DR + d - DN]);
    }
    Qs[rr * QS + d] = val;
  }
}

LAGA_DEVINL void load_k_tile(float* Ks, const AttnArgs& a, int b, int h, int k0) {
  for (int i = threadIdx.x; i < BT * DQK; i += blockDim.x) {
    int rr = i / DQK, d = i % DQK, s = k0 + rr;
    float val = 0.f;
    if (s < a.S) {
      val = d < DN ? __bfloat162float(a.v.kv[b * a.v.kv_sb + s * a.v.kv_ss + h * a.v.kv_sh + d])
                   : __bfloat162float(a.v.kpe[((long long)b * a.S + s) * DR + d - DN]);
    }
    Ks[rr * QS + d] = val;
  }
}

LAGA_DEVINL void load_v_tile(float* Vs, const AttnArgs& a, int b, int h, int k0) {
  for (int i = threadIdx.x; i < BT * DV; i += blockDim.x) {
    int rr = i / DV, d = i % DV, s = k0 + rr;
    Vs[rr * VS + d] = s < a.S ? __bfloat162float(a.v.kv[b * a.v.kv_sb + s * a.v.kv_ss +
                                                         h * a.v.kv_sh + DN + d])
                              : 0.f;
  }
}

LAGA_DEVINL void load_do_tile(float* Ds, const AttnArgs& a, int b, int h, int r0) {
  for (int i = threadIdx.x; i < BT * DV; i += blockDim.x) {
    int rr = i / DV, d = i % DV, s = r0 + rr;
    Ds[rr * VS + d] = s < a.S ? __bfloat162float(a.v.dO[rowid(b, s, h, a.S, a.H) * DV + d]) : 0.f;
  }
}

// grid (q tiles, H, B); thread t: row t/4, column quarter t%4.
__global__ void __launch_bounds__(256) attn_fwd_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Ks = Qs + BT * QS;
  float* Vs = Ks + BT * QS;
  float* Ps = Vs + BT * VS;
  const int qt = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int r = threadIdx.x >> 2, qd = threadIdx.x & 3;
  const int q0 = qt * BT, qi = q0 + r;
  load_q_tile(Qs, a, b, h, q0);
  const float sl2 = a.scale * LOG2E;
  float m = -INFINITY, l = 0.f, acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  for (int kt = 0; kt <= qt; ++kt) {
    __syncthreads();
    load_k_tile(Ks, a, b, h, kt * BT);
    load_v_tile(Vs, a, b, h, kt * BT);
    __syncthreads();
    float s[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) s[j] = 0.f;
    for (int d = 0; d < DQK; ++d) {
      float qv = Qs[r * QS + d];
#pragma unroll
      for (int j = 0; j < 16; ++j) s[j] = fmaf(qv, Ks[(qd + 4 * j) * QS + d], s[j]);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      int key = kt * BT + qd + 4 * j;
      s[j] = (key <= qi && key < a.S) ? s[j] * sl2 : -INFINITY;
      mx = fmaxf(mx, s[j]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m, mx);
    const float alpha = exp2f(m - mn);
    float ps = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float pj = exp2f(s[j] - mn);
      ps += pj;
      Ps[r * PS + qd + 4 * j] = pj;
    }
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    l = l * alpha + ps;
    m = mn;
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] *= alpha;
    __syncthreads();
    for (int cc = 0; cc < BT; ++cc) {
      float pv = Ps[r * PS + cc];
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = fmaf(pv, Vs[cc * VS + qd + 4 * i], acc[i]);
    }
  }
  if (qi < a.S) {
    long long row = rowid(b, qi, h, a.S, a.H);
    const float inv = 1.0f / l;
#pragma unroll
    for (int i = 0; i < 32; ++i) a.v.O[row * DV + qd + 4 * i] = __float2bfloat16_rn(acc[i] * inv);
    if (qd == 0) a.lse_out[((long long)b * a.H + h) * a.S + qi] = (m + log2f(l)) * LN2;
  }
}

// Key-stationary pass: grid (key tiles, H, B); thread t: key row t/4.
__global__ void __launch_bounds__(256) attn_bwd_dkdv_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  float* Ks = sm;
  float* Vs = Ks + BT * QS;
  float* Qs = Vs + BT * VS;
  float* Ds = Qs + BT * QS;
  float* Ps = Ds + BT * VS;
  float* dSs = Ps + BT * PS;
  float* lse2 = dSs + BT * PS;
  float* dlt = lse2 + BT;
  const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int r = threadIdx.x >> 2, qd = threadIdx.x & 3;
  const int k0 = kt * BT, key = k0 + r;
  const int nqt = (a.S + BT - 1) / BT;
  load_k_tile(Ks, a, b, h, k0);
  load_v_tile(Vs, a, b, h, k0);
  const float sl2 = a.scale * LOG2E;
  float dk[48], dv[32];
#pragma unroll
  for (int i = 0; i < 48; ++i) dk[i] = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) dv[i] = 0.f;
  for (int qt = kt; qt < nqt; ++qt) {
    const int q0 = qt * BT;
    __syncthreads();
    load_q_tile(Qs, a, b, h, q0);
    load_do_tile(Ds, a, b, h, q0);
    if (threadIdx.x < BT) {
      int s = q0 + threadIdx.x;
      long long li = ((long long)b * a.H + h) * a.S + s;
      lse2[threadIdx.x] = s < a.S ? a.lse[li] * LOG2E : 0.f;
      dlt[threadIdx.x] = s < a.S ? a.delta[li] : 0.f;
    }
    __syncthreads();
    float s[16], dp[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) { s[j] = 0.f; dp[j] = 0.f; }
    for (int d = 0; d < DQK; ++d) {
      float kv = Ks[r * QS + d];
#pragma unroll
      for (int j = 0; j < 16; ++j) s[j] = fmaf(kv, Qs[(qd + 4 * j) * QS + d], s[j]);
    }
    for (int d = 0; d < DV; ++d) {
      float vv = Vs[r * VS + d];
#pragma unroll
      for (int j = 0; j < 16; ++j) dp[j] = fmaf(vv, Ds[(qd + 4 * j) * VS + d], dp[j]);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      int c = qd + 4 * j, q = q0 + c;
      bool ok = q >= key && q < a.S && key < a.S;
      float pj = ok ? exp2f(s[j] * sl2 - lse2[c]) : 0.f;
      Ps[r * PS + c] = pj;
      dSs[r * PS + c] = pj * (dp[j] - dlt[c]);
    }
    __syncthreads();
    for (int c = 0; c < BT; ++c) {
      float pv = Ps[r * PS + c], ds = dSs[r * PS + c];
#pragma unroll
      for (int i = 0; i < 32; ++i) dv[i] = fmaf(pv, Ds[c * VS + qd + 4 * i], dv[i]);
#pragma unroll
      for (int i = 0; i < 48; ++i) dk[i] = fmaf(ds, Qs[c * QS + qd + 4 * i], dk[i]);
    }
  }
  if (key < a.S) {
    long long base = b * a.v.kv_sb + key * a.v.kv_ss + h * a.v.kv_sh;
    long long row = rowid(b, key, h, a.S, a.H);
#pragma unroll
    for (int i = 0; i < 48; ++i) {
      int d = qd + 4 * i;
      float val = dk[i] * a.scale;
      if (d < DN) a.dkv[base + d] = __float2bfloat16_rn(val);
      else a.dkpe[row * DR + d - DN] = val;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) a.dkv[base + DN + qd + 4 * i] = __float2bfloat16_rn(dv[i]);
  }
}

// Query-stationary pass: grid (q tiles, H, B); thread t: query row t/4.
__global__ void __launch_bounds__(256) attn_bwd_dq_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Ds = Qs + BT * QS;
  float* Ks = Ds + BT * VS;
  float* Vs = Ks + BT * QS;
  float* dSs = Vs + BT * VS;
  const int qt = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int r = threadIdx.x >> 2, qd = threadIdx.x & 3;
  const int q0 = qt * BT, qi = q0 + r;
  load_q_tile(Qs, a, b, h, q0);
  load_do_tile(Ds, a, b, h, q0);
  const float sl2 = a.scale * LOG2E;
  float my_lse2 = 0.f, my_dlt = 0.f;
  if (qi < a.S) {
    long long li = ((long long)b * a.H + h) * a.S + qi;
    my_lse2 = a.lse[li] * LOG2E;
    my_dlt = a.delta[li];
  }
  float dq[48];
#pragma unroll
  for (int i = 0; i < 48; ++i) dq[i] = 0.f;
  for (int kt = 0; kt <= qt; ++kt) {
    __syncthreads();
    load_k_tile(Ks, a, b, h, kt * BT);
    load_v_tile(Vs, a, b, h, kt * BT);
    __syncthreads();
    float s[16], dp[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) { s[j] = 0.f; dp[j] = 0.f; }
    for (int d = 0; d < DQK; ++d) {
      float qv = Qs[r * QS + d];
#pragma unroll
      for (int j = 0; j < 16; ++j) s[j] = fmaf(qv, Ks[(qd + 4 * j) * QS + d], s[j]);
    }
    for (int d = 0; d < DV; ++d) {
      float gv = Ds[r * VS + d];
#pragma unroll
      for (int j = 0; j < 16; ++j) dp[j] = fmaf(gv, Vs[(qd + 4 * j) * VS + d], dp[j]);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      int c = qd + 4 * j, key = kt * BT + c;
      bool ok = key <= qi && key < a.S && qi < a.S;
      float pj = ok ? exp2f(s[j] * sl2 - my_lse2) : 0.f;
      dSs[r * PS + c] = pj * (dp[j] - my_dlt);
    }
    __syncthreads();
    for (int c = 0; c < BT; ++c) {
      float ds = dSs[r * PS + c];
#pragma unroll
      for (int i = 0; i < 48; ++i) dq[i] = fmaf(ds, Ks[c * QS + qd + 4 * i], dq[i]);
    }
  }
  if (qi < a.S) {
    long long row = rowid(b, qi, h, a.S, a.H);
#pragma unroll
    for (int i = 0; i < 48; ++i) a.dq[row * DQK + qd + 4 * i] = dq[i] * a.scale;
  }
}

AttnArgs make_args(const Plan& p, const Ptrs& x) {
  AttnArgs a{};
  a.v = make_views(p, x);
  a.B = p.B; a.S = p.S; a.H = p.H;
  a.scale = p.scale;
  return a;
}

}  // namespace

cudaError_t launch_attn_fwd(const Plan& p, const Ptrs& x, cudaStream_t st) {
  AttnArgs a = make_args(p, x);
  a.lse_out = x.lse;
  const size_t smem = sizeof(float) * (2 * BT * QS + BT * VS + BT * PS);
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.S + BT - 1) / BT, p.H, p.B);
  LaunchScope ls_("attn_fwd", st);
  attn_fwd_kernel<<<grid, 256, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const Plan& p, const Ptrs& x, cudaStream_t st) {
  AttnArgs a = make_args(p, x);
  a.lse = x.lse;
  a.delta = x.buf<float>(p, T_DELTA);
  a.dkv = x.buf<__nv_bfloat16>(p, T_DKV);
  a.dkpe = x.buf<float>(p, T_DKPE);
  a.dq = x.buf<float>(p, T_DQ);
  dim3 grid((p.S + BT - 1) / BT, p.H, p.B);
  const size_t smem1 = sizeof(float) * (2 * BT * QS + 2 * BT * VS + 2 * BT * PS + 2 * BT);
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
  if (e != cudaSuccess) return e;
  {
    LaunchScope ls_("attn_bwd_dkdv", st);
    attn_bwd_dkdv_kernel<<<grid, 256, smem1, st>>>(a);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t smem2 = sizeof(float) * (2 * BT * QS + 2 * BT * VS + BT * PS);
  e = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem2);
  if (e != cudaSuccess) return e;
  LaunchScope ls_("attn_bwd_dq", st);
  attn_bwd_dq_kernel<<<grid, 256, smem2, st>>>(a);
  return cudaGetLastError();
}

}  // namespace laga
