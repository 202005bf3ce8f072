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
    int dr, int dkv, float eps, int rms, __nv_bfloat16* __restrict__ L, float* __restrict__ mean_o,
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
  const float mu = rms ? 0.f : warp_sum(sum) / dkv;   // RMS variant: no centring
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
                                                      const float* __restrict__ lse,
                                                      float* __restrict__ lse2, int s_pad) {
  const int lane = threadIdx.x & 31;
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
    const float* __restrict__ sinT, int B, int S, int H, int dr, int dkv, int rms,
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
    // the RMS variant has no centring, so no mean(g) term
    const float m1 = rms ? 0.f : warp_sum(s1) / dkv, m2 = warp_sum(s2) / dkv;
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

// dgamma[col] = sum over the NGP partial rows, in a fixed order: warp w of a
// block sums its contiguous chunk of rows in row order (all loads issued
// first), then the chunk sums are added in warp order.  32 columns per block.
constexpr int DG_WARPS = 16, DG_CHUNK = 32;
static_assert(NGP <= DG_WARPS * DG_CHUNK, "dgamma chunks");
__global__ void __launch_bounds__(DG_WARPS * 32) dgamma_reduce_kernel(
    const float* __restrict__ part, int nparts, int dkv, float* __restrict__ dgamma) {
  __shared__ float red[DG_WARPS][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int col = blockIdx.x * 32 + lane;
  const int per = (nparts + DG_WARPS - 1) / DG_WARPS;
  const int p0 = warp * per, cnt = max(0, min(per, nparts - p0));
  float v[DG_CHUNK];
#pragma unroll
  for (int i = 0; i < DG_CHUNK; ++i)
    v[i] = (col < dkv && i < cnt) ? part[(long long)(p0 + i) * 512 + col] : 0.f;
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < DG_CHUNK; ++i)
    if (i < cnt) t += v[i];
  red[warp][lane] = t;
  __syncthreads();
  if (warp == 0 && col < dkv) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < DG_WARPS; ++w) s += red[w][lane];
    dgamma[col] = s;
  }
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

// ---------------------------------------------------------------------------
// Canonical dims (d_kv 512, d_rope 64, d_nope = d_v = 128) with bf16 I/O:
// the same steps with 16-byte accesses.  A lane owns eight consecutive
// elements (one 16-byte chunk); the rotate-half partner of chunk c is c + 4.

LAGA_DEVINL void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 t = __bfloat1622float2(h[k]);
    f[2 * k] = t.x;
    f[2 * k + 1] = t.y;
  }
}
LAGA_DEVINL uint4 f32x8_to_bf16(const float (&f)[8]) {
  uint4 v;
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __nv_bfloat162 t = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
    w[k] = *reinterpret_cast<uint32_t*>(&t);
  }
  return v;
}
LAGA_DEVINL void load_f32x8(const float* p, float (&f)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// Rotate the pair (chunk c, chunk c+4) of a 64-wide band by position s:
// x'[i] = x[i] cos - x[i+32] sin, x'[i+32] = x[i+32] cos + x[i] sin.
LAGA_DEVINL void rope_chunk_pair(const __nv_bfloat16* src, __nv_bfloat16* dst, int c,
                                 const float* cs_row, const float* sn_row) {
  float a[8], b[8], cs[8], sn[8];
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + 8 * c), a);
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + 32 + 8 * c), b);
  load_f32x8(cs_row + 8 * c, cs);
  load_f32x8(sn_row + 8 * c, sn);
  float x[8], y[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    x[k] = a[k] * cs[k] - b[k] * sn[k];
    y[k] = b[k] * cs[k] + a[k] * sn[k];
  }
  *reinterpret_cast<uint4*>(dst + 8 * c) = f32x8_to_bf16(x);
  *reinterpret_cast<uint4*>(dst + 32 + 8 * c) = f32x8_to_bf16(y);
}

// a1 + a2, one warp per token.
__global__ void __launch_bounds__(256) prep_fwd_v_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ c,
    const float* __restrict__ gamma, const float* __restrict__ cosT,
    const float* __restrict__ sinT, int S, int H, long long tokens, float eps, int rms,
    __nv_bfloat16* __restrict__ L, float* __restrict__ mean_o, float* __restrict__ rstd_o,
    __nv_bfloat16* __restrict__ kpe, __nv_bfloat16* __restrict__ qr) {
  const int lane = threadIdx.x & 31;
  const long long tok = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (tok >= tokens) return;
  const int s = (int)(tok % S);
  const __nv_bfloat16* crow = c + tok * 576;
  float x[2][8];
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(crow + 8 * lane), x[0]);
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(crow + 256 + 8 * lane), x[1]);
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) sum += x[0][k] + x[1][k];
  const float mu = rms ? 0.f : warp_sum(sum) * (1.0f / 512);   // RMS variant: no centring
  float sq = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float d0 = x[0][k] - mu, d1 = x[1][k] - mu;
    sq += d0 * d0 + d1 * d1;
  }
  const float rstd = 1.0f / sqrtf(warp_sum(sq) * (1.0f / 512) + eps);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int col = 256 * hh + 8 * lane;
    float g[8], y[8];
    load_f32x8(gamma + col, g);
#pragma unroll
    for (int k = 0; k < 8; ++k) y[k] = (x[hh][k] - mu) * rstd * g[k];
    *reinterpret_cast<uint4*>(L + tok * 512 + col) = f32x8_to_bf16(y);
  }
  if (lane == 0) { mean_o[tok] = mu; rstd_o[tok] = rstd; }
  const float* cs_row = cosT + (long long)s * 32;
  const float* sn_row = sinT + (long long)s * 32;
  if (lane < 4) rope_chunk_pair(crow + 512, kpe + tok * 64, lane, cs_row, sn_row);
  // every head's q_rope: 4 chunk pairs per head
  for (int task = lane; task < 4 * H; task += 32) {
    const int h = task >> 2, cc = task & 3;
    const long long row = tok * H + h;
    rope_chunk_pair(q + row * 192 + 128, qr + row * 64, cc, cs_row, sn_row);
  }
}

// delta = rowsum(dO * O): a half-warp per (token, head) row of 128, PRE_ROWS
// rows per half-warp, all loads issued before any use.  Row k of a block is
// blockIdx.x * 16 * PRE_ROWS + k * 16 + (half-warp), so each load instruction
// of the block covers 16 consecutive rows.
constexpr int PRE_ROWS = 4;
__global__ void __launch_bounds__(256) bwd_pre_v_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ d_o, int S, int H,
    long long rows, float* __restrict__ delta,
    const float* __restrict__ lse, float* __restrict__ lse2, int s_pad) {
  const int sub = threadIdx.x & 15;
  const long long base = (long long)blockIdx.x * 16 * PRE_ROWS + (threadIdx.x >> 4);
  uint4 ov[PRE_ROWS], gv[PRE_ROWS];
  float lz[PRE_ROWS];
  long long pr[PRE_ROWS];
#pragma unroll
  for (int k = 0; k < PRE_ROWS; ++k) {
    const long long row = base + 16 * k;
    ov[k] = gv[k] = make_uint4(0u, 0u, 0u, 0u);
    lz[k] = 0.f;
    pr[k] = -1;
    if (row < rows) {
      ov[k] = *reinterpret_cast<const uint4*>(o + row * 128 + 8 * sub);
      gv[k] = *reinterpret_cast<const uint4*>(d_o + row * 128 + 8 * sub);
      if (sub == 0) {
        const int h = (int)(row % H);
        const long long tok = row / H;
        const int b = (int)(tok / S), s = (int)(tok % S);
        pr[k] = ((long long)b * H + h) * s_pad + s;
        lz[k] = lse[((long long)b * H + h) * S + s];
      }
    }
  }
#pragma unroll
  for (int k = 0; k < PRE_ROWS; ++k) {
    float a[8], g[8];
    bf16x8_to_f32(ov[k], a);
    bf16x8_to_f32(gv[k], g);
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc += a[j] * g[j];
#pragma unroll
    for (int m = 8; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (pr[k] >= 0) {
      delta[pr[k]] = acc;
      lse2[pr[k]] = lz[k] * 1.4426950408889634f;
    }
  }
}

// dq in the raw frame: the nope band cast, the rope band rotated back (R^T).
// A warp takes DQ_ROWS rows and issues all of their loads before any store.
constexpr int DQ_ROWS = 4;
__global__ void __launch_bounds__(256) dq_final_v_kernel(const float* __restrict__ dqr, int S,
                                                         int H, long long rows,
                                                         const float* __restrict__ cosT,
                                                         const float* __restrict__ sinT,
                                                         __nv_bfloat16* __restrict__ dq) {
  const int lane = threadIdx.x & 31;
  const long long row0 = ((long long)blockIdx.x * WARPS + (threadIdx.x >> 5)) * DQ_ROWS;
  float4 nope[DQ_ROWS];
  float a[DQ_ROWS], b[DQ_ROWS], cs[DQ_ROWS], sn[DQ_ROWS];
#pragma unroll
  for (int k = 0; k < DQ_ROWS; ++k) {
    const long long row = row0 + k;
    if (row < rows) {
      const float* src = dqr + row * 192;
      const int s = (int)((row / H) % S);
      nope[k] = *reinterpret_cast<const float4*>(src + 4 * lane);
      a[k] = src[128 + lane];
      b[k] = src[160 + lane];
      cs[k] = cosT[(long long)s * 32 + lane];
      sn[k] = sinT[(long long)s * 32 + lane];
    }
  }
#pragma unroll
  for (int k = 0; k < DQ_ROWS; ++k) {
    const long long row = row0 + k;
    if (row < rows) {
      __nv_bfloat16* dst = dq + row * 192;
      __nv_bfloat162 lo = __floats2bfloat162_rn(nope[k].x, nope[k].y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(nope[k].z, nope[k].w);
      uint2 w;
      w.x = *reinterpret_cast<uint32_t*>(&lo);
      w.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(dst + 4 * lane) = w;
      dst[128 + lane] = __float2bfloat16_rn(a[k] * cs[k] + b[k] * sn[k]);
      dst[160 + lane] = __float2bfloat16_rn(b[k] * cs[k] - a[k] * sn[k]);
    }
  }
}

// a7, one warp per token; a lane owns latent columns 8*lane.. and
// 256 + 8*lane.., and the k_pe column pair (2*lane, 2*lane+1) of the sum
// over heads (taken in head order).
__global__ void __launch_bounds__(256) norm_bwd_v_kernel(
    const float* __restrict__ dL, const __nv_bfloat16* __restrict__ c,
    const float* __restrict__ mean, const float* __restrict__ rstd,
    const float* __restrict__ gamma, const float* __restrict__ dkpe_h,
    const float* __restrict__ cosT, const float* __restrict__ sinT, int S, int H,
    long long tokens, int rms, float* __restrict__ dc, float* __restrict__ dg_part) {
  __shared__ float red[WARPS][512];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float gm[2][8], dg[2][8];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    load_f32x8(gamma + 256 * hh + 8 * lane, gm[hh]);
#pragma unroll
    for (int k = 0; k < 8; ++k) dg[hh][k] = 0.f;
  }
  for (long long tok = (long long)blockIdx.x * WARPS + warp; tok < tokens;
       tok += (long long)gridDim.x * WARPS) {
    const __nv_bfloat16* crow = c + tok * 576;
    // all loads first: the latent and dL rows, the row statistics and the
    // first KP_PRE heads' k_pe gradients, so their latencies overlap
    uint4 cv[2];
    float dv[2][8];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      cv[hh] = *reinterpret_cast<const uint4*>(crow + 256 * hh + 8 * lane);
      load_f32x8(dL + tok * 512 + 256 * hh + 8 * lane, dv[hh]);
    }
    const float mu = mean[tok], rs = rstd[tok];
    constexpr int KP_PRE = 16;
    float2 kp[KP_PRE];
#pragma unroll
    for (int h = 0; h < KP_PRE; ++h)
      kp[h] = h < H ? *reinterpret_cast<const float2*>(dkpe_h + (tok * H + h) * 64 + 2 * lane)
                    : make_float2(0.f, 0.f);
    float xh[2][8], g[2][8];
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float xv[8];
      const float* d = dv[hh];
      bf16x8_to_f32(cv[hh], xv);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        xh[hh][k] = (xv[k] - mu) * rs;
        g[hh][k] = d[k] * gm[hh][k];
        dg[hh][k] += d[k] * xh[hh][k];
        s1 += g[hh][k];
        s2 += g[hh][k] * xh[hh][k];
      }
    }
    // the RMS variant has no centring, so no mean(g) term
    const float m1 = rms ? 0.f : warp_sum(s1) * (1.0f / 512), m2 = warp_sum(s2) * (1.0f / 512);
    float* drow = dc + tok * 576;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float r[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) r[k] = rs * (g[hh][k] - m1 - xh[hh][k] * m2);
      float* dst = drow + 256 * hh + 8 * lane;
      *reinterpret_cast<float4*>(dst) = make_float4(r[0], r[1], r[2], r[3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(r[4], r[5], r[6], r[7]);
    }
    // sum over heads of the per-head k_pe gradient, columns 2*lane, 2*lane+1
    // (in head order)
    float2 a = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < KP_PRE; ++h) {
      if (h < H) {
        a.x += kp[h].x;
        a.y += kp[h].y;
      }
    }
    for (int h = KP_PRE; h < H; ++h) {
      const float2 v = *reinterpret_cast<const float2*>(dkpe_h + (tok * H + h) * 64 + 2 * lane);
      a.x += v.x;
      a.y += v.y;
    }
    // rotate back: lanes < 16 hold x[i], lanes >= 16 hold x[i + 32]
    float2 pb;
    pb.x = __shfl_xor_sync(0xffffffffu, a.x, 16);
    pb.y = __shfl_xor_sync(0xffffffffu, a.y, 16);
    const int s = (int)(tok % S), i = 2 * (lane & 15);
    const float2 cs = *reinterpret_cast<const float2*>(cosT + (long long)s * 32 + i);
    const float2 sn = *reinterpret_cast<const float2*>(sinT + (long long)s * 32 + i);
    float2 out;
    if (lane < 16) {
      out.x = a.x * cs.x + pb.x * sn.x;
      out.y = a.y * cs.y + pb.y * sn.y;
    } else {
      out.x = a.x * cs.x - pb.x * sn.x;
      out.y = a.y * cs.y - pb.y * sn.y;
    }
    *reinterpret_cast<float2*>(drow + 512 + 2 * lane) = out;
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int k = 0; k < 8; ++k) red[warp][256 * hh + 8 * lane + k] = dg[hh][k];
  __syncthreads();
  for (int col = threadIdx.x; col < 512; col += 256) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) t += red[w][col];
    dg_part[(long long)blockIdx.x * 512 + col] = t;
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
  if (p.canonical)
    prep_fwd_v_kernel<<<g, 256, 0, st>>>((const __nv_bfloat16*)x.q, (const __nv_bfloat16*)x.c,
                                         x.gamma, x.cos, x.sin, p.S, p.H, p.tokens(), p.d.ln_eps,
                                         (int)p.rms, L, mean, rstd, kpe, qr);
  else if (p.fp32)
    prep_fwd_kernel<float><<<g, 256, 0, st>>>((const float*)x.q, (const float*)x.c, x.gamma, x.cos,
                                              x.sin, p.B, p.S, p.H, p.dn, p.dr, p.dkv, p.d.ln_eps,
                                              (int)p.rms, L, mean, rstd, kpe, qr, qn);
  else
    prep_fwd_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(
        (const __nv_bfloat16*)x.q, (const __nv_bfloat16*)x.c, x.gamma, x.cos, x.sin, p.B, p.S, p.H,
        p.dn, p.dr, p.dkv, p.d.ln_eps, (int)p.rms, L, mean, rstd, kpe, qr, qn);
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
  float* lse2 = x.buf<float>(p, T_LSE2);
  if (p.canonical)
    bwd_pre_v_kernel<<<grid_for(p.rows(), 16 * PRE_ROWS), 256, 0, st>>>(
        (const __nv_bfloat16*)x.o, (const __nv_bfloat16*)x.d_o, p.S, p.H, p.rows(), delta,
        x.lse, lse2, (int)p.s_pad());
  else if (p.fp32)
    bwd_pre_kernel<float><<<g, 256, 0, st>>>((const float*)x.o, (const float*)x.d_o, p.B, p.S, p.H,
                                             p.dv, delta, dop, x.lse, lse2,
                                             (int)p.s_pad());
  else
    bwd_pre_kernel<__nv_bfloat16><<<g, 256, 0, st>>>((const __nv_bfloat16*)x.o,
                                                     (const __nv_bfloat16*)x.d_o, p.B, p.S, p.H,
                                                     p.dv, delta, dop, x.lse, lse2,
                                             (int)p.s_pad());
  return cudaGetLastError();
}

cudaError_t launch_dq_finalize(const Plan& p, const Ptrs& x, cudaStream_t st) {
  LaunchScope ls_("dq_final", st);
  const int g = grid_for(p.rows(), WARPS);
  const float* dqr = x.buf<float>(p, T_DQ);
  if (p.canonical)
    dq_final_v_kernel<<<grid_for(p.rows(), WARPS * DQ_ROWS), 256, 0, st>>>(
        dqr, p.S, p.H, p.rows(), x.cos, x.sin, (__nv_bfloat16*)x.dq);
  else if (p.fp32)
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
  if (p.canonical)
    norm_bwd_v_kernel<<<NGP, 256, 0, st>>>(dL, (const __nv_bfloat16*)x.c, x.buf<float>(p, W_MEAN),
                                           x.buf<float>(p, W_RSTD), x.gamma, dk, x.cos, x.sin, p.S,
                                           p.H, p.tokens(), (int)p.rms, x.dc, part);
  else if (p.fp32)
    norm_bwd_kernel<float><<<NGP, 256, 0, st>>>(dL, (const float*)x.c, x.buf<float>(p, W_MEAN),
                                                x.buf<float>(p, W_RSTD), x.gamma, dk, x.cos, x.sin,
                                                p.B, p.S, p.H, p.dr, p.dkv, (int)p.rms, x.dc, part);
  else
    norm_bwd_kernel<__nv_bfloat16><<<NGP, 256, 0, st>>>(
        dL, (const __nv_bfloat16*)x.c, x.buf<float>(p, W_MEAN), x.buf<float>(p, W_RSTD), x.gamma,
        dk, x.cos, x.sin, p.B, p.S, p.H, p.dr, p.dkv, (int)p.rms, x.dc, part);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  LaunchScope ls2_("dgamma_reduce", st);
  dgamma_reduce_kernel<<<(p.dkv + 31) / 32, DG_WARPS * 32, 0, st>>>(part, NGP, p.dkv, x.dgamma);
  return cudaGetLastError();
}

cudaError_t launch_unpad_dw(const Plan& p, const Ptrs& x, cudaStream_t st) {
  LaunchScope ls_("unpad_dw", st);
  const int g = grid_stride((long long)p.dkv * p.H * (p.dn + p.dv));
  unpad_dw_kernel<<<g, 256, 0, st>>>(x.buf<float>(p, T_DWC), p.H, p.dn, p.dv, p.dkv, x.dw);
  return cudaGetLastError();
}

}  // namespace laga
