// HBM-bound kernels around the tensor-core work:
//   prep_fwd   a1 latent LayerNorm + a2 RoPE of k_pe and q_rope (and, for
//              non-canonical dims or fp32 I/O, the padded bf16 q_nope copy)
//   bwd_pre    delta = rowsum(dO * O) of the attention backward
//   norm_bwd   a7 LayerNorm backward and the RoPE backward of k_pe -> dc
//   dq_final   inverse RoPE of the rope band of dq, cast to the I/O dtype
// Paper: Section 2.1 (kv = W_kv_b LN(latent), decoupled k_pe band),
// Algorithm 1 step 1, Section 5.2 (backward), Section 5.3 (RoPE band).
#include "common.cuh"
#include "kernels.h"

namespace laga {

namespace {

constexpr int WARPS = 8;  // warps per block of the per-token kernels

template <typename T>
__global__ void __launch_bounds__(256) pad_w_kernel(const T* __restrict__ w, long long w_ld,
                                                    int col0, int H, int dn, int dv, int dkv,
                                                    __nv_bfloat16* __restrict__ wc) {
  // wc[k][h*256 + e]: e < 128 -> k_nope column e, e >= 128 -> v column e-128
  long long n = (long long)512 * H * 256;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n; i += (long long)gridDim.x * 256) {
    int k = (int)(i / (H * 256));
    int col = (int)(i % (H * 256));
    int h = col / 256, e = col % 256;
    float v = 0.f;
    if (k < dkv) {
      if (e < 128 && e < dn) v = to_f32(w[k * w_ld + col0 + (long long)h * (dn + dv) + e]);
      if (e >= 128 && e - 128 < dv) v = to_f32(w[k * w_ld + col0 + (long long)h * (dn + dv) + dn + e - 128]);
    }
    wc[i] = __float2bfloat16_rn(v);
  }
}

// One warp per token: LayerNorm of the latent (lane owns columns lane+32i),
// RoPE of k_pe and of every head's q_rope (lane owns pair (i, i+dr/2)).
template <typename T>
__global__ void __launch_bounds__(256) prep_fwd_kernel(
    const T* __restrict__ q, const T* __restrict__ c, const float* __restrict__ gamma,
    const float* __restrict__ cosT, const float* __restrict__ sinT, int B, int S, int H, int dn,
    int dr, int dkv, float eps, __nv_bfloat16* __restrict__ L, float* __restrict__ mean_o,
    float* __restrict__ rstd_o, __nv_bfloat16* __restrict__ kpe, __nv_bfloat16* __restrict__ qr,
    __nv_bfloat16* __restrict__ qn_pad) {
  const int lane = threadIdx.x & 31;
  const long long tok = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (tok >= (long long)B * S) return;
  const int s = (int)(tok % S);
  const T* crow = c + tok * (dkv + dr);
  float x[16];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    int col = lane + 32 * i;
    x[i] = col < dkv ? to_f32(crow[col]) : 0.f;
    sum += x[i];
  }
  const float mu = warp_sum(sum) / dkv;
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    int col = lane + 32 * i;
    float dlt = col < dkv ? x[i] - mu : 0.f;
    sq += dlt * dlt;
  }
  const float var = warp_sum(sq) / dkv;
  const float rstd = 1.0f / sqrtf(var + eps);
  __nv_bfloat16* Lrow = L + tok * 512;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    int col = lane + 32 * i;
    float v = col < dkv ? (x[i] - mu) * rstd * gamma[col] : 0.f;
    Lrow[col] = __float2bfloat16_rn(v);
  }
  if (lane == 0) { mean_o[tok] = mu; rstd_o[tok] = rstd; }
  const int half = dr >> 1;
  const float cs = lane < half ? cosT[(long long)s * half + lane] : 1.f;
  const float sn = lane < half ? sinT[(long long)s * half + lane] : 0.f;
  {
    const T* kp = crow + dkv;
    float a = lane < half ? to_f32(kp[lane]) : 0.f;
    float b = lane < half ? to_f32(kp[lane + half]) : 0.f;
    __nv_bfloat16* ko = kpe + tok * 64;
    if (lane < half) {
      ko[lane] = __float2bfloat16_rn(a * cs - b * sn);
      ko[lane + half] = __float2bfloat16_rn(b * cs + a * sn);
    }
    for (int e = 2 * half + lane; e < 64; e += 32) ko[e] = __float2bfloat16_rn(0.f);
  }
  for (int h = 0; h < H; ++h) {
    const long long row = tok * H + h;
    const T* qrow = q + row * (dn + dr);
    __nv_bfloat16* qo = qr + row * 64;
    if (lane < half) {
      float a = to_f32(qrow[dn + lane]);
      float b = to_f32(qrow[dn + lane + half]);
      qo[lane] = __float2bfloat16_rn(a * cs - b * sn);
      qo[lane + half] = __float2bfloat16_rn(b * cs + a * sn);
    }
    for (int e = 2 * half + lane; e < 64; e += 32) qo[e] = __float2bfloat16_rn(0.f);
    if (qn_pad) {
      __nv_bfloat16* qp = qn_pad + row * 128;
      for (int e = lane; e < 128; e += 32)
        qp[e] = __float2bfloat16_rn(e < dn ? to_f32(qrow[e]) : 0.f);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) unpad_o_kernel(const __nv_bfloat16* __restrict__ oc,
                                                      long long R, int dv, T* __restrict__ o) {
  long long n = R * dv;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n; i += (long long)gridDim.x * 256) {
    long long r = i / dv;
    int e = (int)(i % dv);
    o[i] = from_f32<T>(__bfloat162float(oc[r * 128 + e]));
  }
}

// One warp per (token, head) row: delta = sum_d dO*O over the true d_v,
// plus the padded bf16 dO copy when the dims are not canonical.
template <typename T>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const T* __restrict__ o,
                                                      const T* __restrict__ d_o, int B, int S,
                                                      int H, int dv, float* __restrict__ delta,
                                                      __nv_bfloat16* __restrict__ do_pad,
                                                      int* __restrict__ sem, int n_sem,
                                                      const float* __restrict__ lse,
                                                      float* __restrict__ lse2, int s_pad) {
  const int lane = threadIdx.x & 31;
  // the attention backward's semaphores and work counter start at zero
  for (int i = blockIdx.x * 256 + threadIdx.x; i < n_sem; i += gridDim.x * 256) sem[i] = 0;
  const long long row = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (row >= (long long)B * S * H) return;
  const T* orow = o + row * dv;
  const T* grow = d_o + row * dv;
  float acc = 0.f;
  for (int e = lane; e < dv; e += 32) acc += to_f32(orow[e]) * to_f32(grow[e]);
  acc = warp_sum(acc);
  const int h = (int)(row % H);
  const long long tok = row / H;
  const int b = (int)(tok / S), s = (int)(tok % S);
  if (lane == 0) {
    const long long pr = ((long long)b * H + h) * s_pad + s;
    delta[pr] = acc;
    lse2[pr] = lse[((long long)b * H + h) * S + s] * 1.4426950408889634f;
  }
  if (do_pad) {
    for (int e = lane; e < 128; e += 32)
      do_pad[row * 128 + e] = __float2bfloat16_rn(e < dv ? to_f32(grow[e]) : 0.f);
  }
}

// dq in the raw frame: nope band copied, rope band rotated back (R^T).
template <typename T>
__global__ void __launch_bounds__(256) dq_final_kernel(const float* __restrict__ dqr, int B, int S,
                                                       int H, int dn, int dr,
                                                       const float* __restrict__ cosT,
                                                       const float* __restrict__ sinT,
                                                       T* __restrict__ dq) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (row >= (long long)B * S * H) return;
  const int s = (int)((row / H) % S);
  const float* src = dqr + row * 192;
  T* dst = dq + row * (dn + dr);
  for (int e = lane; e < dn; e += 32) dst[e] = from_f32<T>(src[e]);
  const int half = dr >> 1;
  if (lane < half) {
    float cs = cosT[(long long)s * half + lane], sn = sinT[(long long)s * half + lane];
    float a = src[128 + lane], b = src[128 + lane + half];
    dst[dn + lane] = from_f32<T>(a * cs + b * sn);
    dst[dn + lane + half] = from_f32<T>(b * cs - a * sn);
  }
}

// a7: one warp per token.  dx = rstd (g - mean(g) - xhat mean(g xhat)) with
// g = dL*gamma; dgamma partial sums per block in a fixed token order; the
// k_pe gradient summed over heads in head order, then rotated back (R^T).
template <typename T>
__global__ void __launch_bounds__(256) norm_bwd_kernel(
    const float* __restrict__ dL, const T* __restrict__ c, const float* __restrict__ mean,
    const float* __restrict__ rstd, const float* __restrict__ gamma,
    const float* __restrict__ dkpe_h, const float* __restrict__ cosT,
    const float* __restrict__ sinT, int B, int S, int H, int dr, int dkv,
    float* __restrict__ dc, float* __restrict__ dg_part) {
  __shared__ float red[WARPS][512];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float dg[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) dg[i] = 0.f;
  const long long T_ = (long long)B * S;
  const int half = dr >> 1;
  for (long long tok = (long long)blockIdx.x * WARPS + warp; tok < T_;
       tok += (long long)gridDim.x * WARPS) {
    const T* crow = c + tok * (dkv + dr);
    const float* gL = dL + tok * 512;
    const float mu = mean[tok], rs = rstd[tok];
    float xh[16], g[16];
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      int col = lane + 32 * i;
      bool ok = col < dkv;
      xh[i] = ok ? (to_f32(crow[col]) - mu) * rs : 0.f;
      float d = ok ? gL[col] : 0.f;
      g[i] = ok ? d * gamma[col] : 0.f;
      dg[i] += d * xh[i];
      s1 += g[i];
      s2 += g[i] * xh[i];
    }
    const float m1 = warp_sum(s1) / dkv, m2 = warp_sum(s2) / dkv;
    float* drow = dc + tok * (dkv + dr);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      int col = lane + 32 * i;
      if (col < dkv) drow[col] = rs * (g[i] - m1 - xh[i] * m2);
    }
    if (lane < half) {
      const int s = (int)(tok % S);
      float a = 0.f, b = 0.f;
      for (int h = 0; h < H; ++h) {
        const float* src = dkpe_h + (tok * H + h) * 64;
        a += src[lane];
        b += src[lane + half];
      }
      float cs = cosT[(long long)s * half + lane], sn = sinT[(long long)s * half + lane];
      drow[dkv + lane] = a * cs + b * sn;
      drow[dkv + lane + half] = b * cs - a * sn;
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) red[warp][lane + 32 * i] = dg[i];
  __syncthreads();
  for (int col = threadIdx.x; col < 512; col += 256) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) t += red[w][col];
    dg_part[(long long)blockIdx.x * 512 + col] = t;
  }
}

__global__ void dgamma_reduce_kernel(const float* __restrict__ part, int nparts, int dkv,
                                     float* __restrict__ dgamma) {
  int col = blockIdx.x * blockDim.x + threadIdx.x;
  if (col >= dkv) return;
  float t = 0.f;
  for (int p = 0; p < nparts; ++p) t += part[(long long)p * 512 + col];
  dgamma[col] = t;
}

__global__ void __launch_bounds__(256) unpad_dw_kernel(const float* __restrict__ dwc, int H, int dn,
                                                       int dv, int dkv, float* __restrict__ dw) {
  const int dh = dn + dv;
  long long n = (long long)dkv * H * dh;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n; i += (long long)gridDim.x * 256) {
    int k = (int)(i / (H * dh));
    int col = (int)(i % (H * dh));
    int h = col / dh, e = col % dh;
    int ec = e < dn ? e : 128 + (e - dn);
    dw[i] = dwc[(long long)k * H * 256 + h * 256 + ec];
  }
}

inline int grid_for(long long n, int per_block) {
  long long g = (n + per_block - 1) / per_block;
  return (int)(g < 1 ? 1 : g);
}
inline int grid_stride(long long n) {
  long long g = (n + 255) / 256;
  return (int)(g > 152 * 16 ? 152 * 16 : (g < 1 ? 1 : g));
}

}  // namespace

cudaError_t launch_pad_w(const Plan& p, const Ptrs& x, cudaStream_t st) {
  LaunchScope ls_("pad_w", st);
  const long long w_ld = (long long)p.d.n_h_total * (p.dn + p.dv);
  const int col0 = p.d.head_offset * (p.dn + p.dv);
  auto* wc = x.buf<__nv_bfloat16>(p, W_WC);
  const int g = grid_stride((long long)512 * p.H * 256);
  if (p.fp32)
    pad_w_kernel<float><<<g, 256, 0, st>>>((const float*)x.w, w_ld, col0, p.H, p.dn, p.dv, p.dkv, wc);
  else
    pad_w_kernel<__nv_bfloat16><<<g, 256, 0, st>>>((const __nv_bfloat16*)x.w, w_ld, col0, p.H, p.dn,
                                                   p.dv, p.dkv, wc);
  return cudaGetLastError();
}

cudaError_t launch_prep_fwd(const Plan& p, const Ptrs& x, cudaStream_t st) {
  LaunchScope ls_("prep_fwd", st);
  const int g = grid_for(p.tokens(), WARPS);
  __nv_bfloat16* qn = p.canonical ? nullptr : x.buf<__nv_bfloat16>(p, W_QN);
  auto* L = x.buf<__nv_bfloat16>(p, W_L);
  auto* kpe = x.buf<__nv_bfloat16>(p, W_KPE);
  auto* qr = x.buf<__nv_bfloat16>(p, W_QR);
  float* mean = x.buf<float>(p, W_MEAN);
  float* rstd = x.buf<float>(p, W_RSTD);
  if (p.fp32)
    prep_fwd_kernel<float><<<g, 256, 0, st>>>((const float*)x.q, (const float*)x.c, x.gamma, x.cos,
                                              x.sin, p.B, p.S, p.H, p.dn, p.dr, p.dkv, p.d.ln_eps,
                                              L, mean, rstd, kpe, qr, qn);
  else
    prep_fwd_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(
        (const __nv_bfloat16*)x.q, (const __nv_bfloat16*)x.c, x.gamma, x.cos, x.sin, p.B, p.S, p.H,
        p.dn, p.dr, p.dkv, p.d.ln_eps, L, mean, rstd, kpe, qr, qn);
  return cudaGetLastError();
}

cudaError_t launch_unpad_o(const Plan& p, const Ptrs& x, cudaStream_t st) {
  LaunchScope ls_("unpad_o", st);
  const auto* oc = x.buf<__nv_bfloat16>(p, W_OC);
  const int g = grid_stride(p.rows() * p.dv);
  if (p.fp32)
    unpad_o_kernel<float><<<g, 256, 0, st>>>(oc, p.rows(), p.dv, (float*)x.o);
  else
    unpad_o_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(oc, p.rows(), p.dv, (__nv_bfloat16*)x.o);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const Plan& p, const Ptrs& x, cudaStream_t st) {
  LaunchScope ls_("bwd_pre", st);
  const int g = grid_for(p.rows(), WARPS);
  float* delta = x.buf<float>(p, T_DELTA);
  __nv_bfloat16* dop = p.canonical ? nullptr : x.buf<__nv_bfloat16>(p, T_DOC);
  int* sem = x.buf<int>(p, T_SEM);
  float* lse2 = x.buf<float>(p, T_LSE2);
  const int n_sem = (int)(p.len[T_SEM] / 4);
  if (p.fp32)
    bwd_pre_kernel<float><<<g, 256, 0, st>>>((const float*)x.o, (const float*)x.d_o, p.B, p.S, p.H,
                                             p.dv, delta, dop, sem, n_sem, x.lse, lse2,
                                             (int)p.s_pad());
  else
    bwd_pre_kernel<__nv_bfloat16><<<g, 256, 0, st>>>((const __nv_bfloat16*)x.o,
                                                     (const __nv_bfloat16*)x.d_o, p.B, p.S, p.H,
                                                     p.dv, delta, dop, sem, n_sem, x.lse, lse2,
                                             (int)p.s_pad());
  return cudaGetLastError();
}

cudaError_t launch_dq_finalize(const Plan& p, const Ptrs& x, cudaStream_t st) {
  LaunchScope ls_("dq_final", st);
  const int g = grid_for(p.rows(), WARPS);
  const float* dqr = x.buf<float>(p, T_DQ);
  if (p.fp32)
    dq_final_kernel<float><<<g, 256, 0, st>>>(dqr, p.B, p.S, p.H, p.dn, p.dr, x.cos, x.sin,
                                              (float*)x.dq);
  else
    dq_final_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(dqr, p.B, p.S, p.H, p.dn, p.dr, x.cos, x.sin,
                                                      (__nv_bfloat16*)x.dq);
  return cudaGetLastError();
}

cudaError_t launch_norm_bwd(const Plan& p, const Ptrs& x, const float* dL, cudaStream_t st) {
  const float* dk = x.buf<float>(p, T_DKPE);
  float* part = x.buf<float>(p, T_DGP);
  {
  LaunchScope ls_("norm_bwd", st);
  if (p.fp32)
    norm_bwd_kernel<float><<<NGP, 256, 0, st>>>(dL, (const float*)x.c, x.buf<float>(p, W_MEAN),
                                                x.buf<float>(p, W_RSTD), x.gamma, dk, x.cos, x.sin,
                                                p.B, p.S, p.H, p.dr, p.dkv, x.dc, part);
  else
    norm_bwd_kernel<__nv_bfloat16><<<NGP, 256, 0, st>>>(
        dL, (const __nv_bfloat16*)x.c, x.buf<float>(p, W_MEAN), x.buf<float>(p, W_RSTD), x.gamma,
        dk, x.cos, x.sin, p.B, p.S, p.H, p.dr, p.dkv, x.dc, part);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  LaunchScope ls2_("dgamma_reduce", st);
  dgamma_reduce_kernel<<<(p.dkv + 127) / 128, 128, 0, st>>>(part, NGP, p.dkv, x.dgamma);
  return cudaGetLastError();
}

cudaError_t launch_unpad_dw(const Plan& p, const Ptrs& x, cudaStream_t st) {
  LaunchScope ls_("unpad_dw", st);
  const int g = grid_stride((long long)p.dkv * p.H * (p.dn + p.dv));
  unpad_dw_kernel<<<g, 256, 0, st>>>(x.buf<float>(p, T_DWC), p.H, p.dn, p.dv, p.dkv, x.dw);
  return cudaGetLastError();
}

}  // namespace laga
