// Absorbed form B2 (Section 3.2, Figure 2): the inference-side absorb trick
// ported to training, built only as the memory-trap contrast of LAGA.
//   q_abs[t,h,:] = W^k[h] q_nope[t,h]            (n_h * d_kv per token)
//   s_ij = (q_abs_i . L_j + q_rope_i . k_pe_j) * scale
//   o_lat_i = sum_j softmax_j(s_i) L_j           (latent accumulator, n_h * d_kv)
//   O_i = W^v[h]^T o_lat_i                       (un-absorb)
// and the backward of all of it.  Straightforward fp32-accumulating tiled
// kernels (performance is not the point of this form); every sum is taken
// in a fixed order, so results are deterministic.
#include "common.cuh"
#include "kernels.h"

namespace laga {
namespace {

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// ---------------------------------------------------------------- batched GEMM
// C[z](m, n) = sum_k A[z](m, k) B[z](k, n), element (z, i, j) of X at
// X + z*sXz + i*sXi + j*sXj.  fp32 accumulation, K ascending.
struct Mat {
  long long sz, si, sj;
};

template <typename TA, typename TB, typename TC>
__global__ void __launch_bounds__(256) bgemm_kernel(int M, int N, int K, const TA* __restrict__ A,
                                                    Mat a, const TB* __restrict__ B, Mat bm,
                                                    TC* __restrict__ C, Mat c) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int z = blockIdx.z;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const long long m0 = (long long)blockIdx.y * 64, n0 = (long long)blockIdx.x * 64;
  const TA* Az = A + z * a.sz;
  const TB* Bz = B + z * bm.sz;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 64 * 16; i += 256) {
      const int mm = i % 64, kk = i / 64;
      const long long gm = m0 + mm, gn = n0 + mm;
      const int gk = k0 + kk;
      As[kk][mm] = (gm < M && gk < K) ? to_f32(Az[gm * a.si + gk * a.sj]) : 0.f;
      Bs[kk][mm] = (gn < N && gk < K) ? to_f32(Bz[gk * bm.si + gn * bm.sj]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  TC* Cz = C + z * c.sz;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long gm = m0 + ty * 4 + i, gn = n0 + tx * 4 + j;
      if (gm < M && gn < N) Cz[gm * c.si + gn * c.sj] = from_f32<TC>(acc[i][j]);
    }
}

template <typename TA, typename TB, typename TC>
cudaError_t bgemm(const char* name, int Z, int M, int N, int K, const TA* A, Mat a, const TB* B,
                  Mat b, TC* C, Mat c, cudaStream_t st) {
  LaunchScope ls_(name, st);
  dim3 grid((N + 63) / 64, (M + 63) / 64, Z);
  bgemm_kernel<TA, TB, TC><<<grid, 256, 0, st>>>(M, N, K, A, a, B, b, C, c);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- latent attention
// Tiles of 32 rows; 256 threads, 8 per row.  Key rows are [L (512) | k_pe_rot (64)].
constexpr int AT = 32;
constexpr int DQA = DKV + DR;      // 576
constexpr int QS = DQA + 1;        // smem row strides (floats)
constexpr int LS = DKV + 1;
constexpr int PS = AT + 1;

struct LatArgs {
  int B, S, H;
  float scale;
  const __nv_bfloat16* qabs;   // [R, 512]
  const __nv_bfloat16* qr;     // [R, 64]
  const __nv_bfloat16* L;      // [T, 512]
  const __nv_bfloat16* kpe;    // [T, 64]
  __nv_bfloat16* olat;         // [R, 512]
  float* lse;                  // [B, H, S] natural log
  const float* lse2;           // [B*H, Sp] LSE * log2(e)
  const float* delta;          // [B*H, Sp]
  long long s_pad;
  const __nv_bfloat16* dolat;  // [R, 512]
  float* dqabs;                // [R, 512]
  float* dq;                   // [R, 192]: rope band written at 128..191
  float* dL;                   // [T, 512]
  float* dkpe;                 // [R, 64]
};

LAGA_DEVINL long long rid(const LatArgs& a, int b, int s, int h) {
  return ((long long)b * a.S + s) * a.H + h;
}

// rows r0.. of (q_abs | q_rope_rot) for head h
LAGA_DEVINL void load_q(float* Qs, const LatArgs& a, int b, int h, int r0) {
  for (int i = threadIdx.x; i < AT * DQA; i += blockDim.x) {
    const int rr = i / DQA, d = i % DQA, s = r0 + rr;
    float v = 0.f;
    if (s < a.S) {
      const long long row = rid(a, b, s, h);
      v = d < DKV ? __bfloat162float(a.qabs[row * DKV + d]) : __bfloat162float(a.qr[row * DR + d - DKV]);
    }
    Qs[rr * QS + d] = v;
  }
}
// key rows k0.. of (L | k_pe_rot)
LAGA_DEVINL void load_k(float* Ks, const LatArgs& a, int b, int k0) {
  for (int i = threadIdx.x; i < AT * DQA; i += blockDim.x) {
    const int rr = i / DQA, d = i % DQA, s = k0 + rr;
    float v = 0.f;
    if (s < a.S) {
      const long long tok = (long long)b * a.S + s;
      v = d < DKV ? __bfloat162float(a.L[tok * DKV + d]) : __bfloat162float(a.kpe[tok * DR + d - DKV]);
    }
    Ks[rr * QS + d] = v;
  }
}
LAGA_DEVINL void load_dol(float* Ds, const LatArgs& a, int b, int h, int r0) {
  for (int i = threadIdx.x; i < AT * DKV; i += blockDim.x) {
    const int rr = i / DKV, d = i % DKV, s = r0 + rr;
    Ds[rr * LS + d] = s < a.S ? __bfloat162float(a.dolat[rid(a, b, s, h) * DKV + d]) : 0.f;
  }
}

// grid (q tiles, H, B)
__global__ void __launch_bounds__(256) lat_fwd_kernel(LatArgs a) {
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Ks = Qs + AT * QS;
  float* Ps = Ks + AT * QS;
  const int qt = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int r = threadIdx.x >> 3, sub = threadIdx.x & 7;
  const int q0 = qt * AT, qi = q0 + r;
  load_q(Qs, a, b, h, q0);
  const float sl2 = a.scale * LOG2E;
  float m = -INFINITY, l = 0.f, acc[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) acc[i] = 0.f;
  for (int kt = 0; kt <= qt; ++kt) {
    __syncthreads();
    load_k(Ks, a, b, kt * AT);
    __syncthreads();
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    for (int d = 0; d < DQA; ++d) {
      const float qv = Qs[r * QS + d];
#pragma unroll
      for (int c = 0; c < 4; ++c) s[c] = fmaf(qv, Ks[(sub + 8 * c) * QS + d], s[c]);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int key = kt * AT + sub + 8 * c;
      s[c] = (key <= qi && key < a.S) ? s[c] * sl2 : -INFINITY;
      mx = fmaxf(mx, s[c]);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float mn = fmaxf(m, mx), alpha = exp2f(m - mn);
    float ps = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float p = exp2f(s[c] - mn);
      ps += p;
      Ps[r * PS + sub + 8 * c] = p;
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    l = l * alpha + ps;
    m = mn;
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] *= alpha;
    __syncthreads();
    for (int cc = 0; cc < AT; ++cc) {
      const float p = Ps[r * PS + cc];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = fmaf(p, Ks[cc * QS + sub + 8 * i], acc[i]);  // V = L
    }
  }
  if (qi < a.S) {
    const long long row = rid(a, b, qi, h);
    const float inv = 1.f / l;
#pragma unroll
    for (int i = 0; i < 64; ++i) a.olat[row * DKV + sub + 8 * i] = __float2bfloat16_rn(acc[i] * inv);
    if (sub == 0) a.lse[((long long)b * a.H + h) * a.S + qi] = (m + log2f(l)) * LN2;
  }
}

// query-stationary: dq_abs_i = scale sum_j dS_ij L_j, dq_rope_i = scale sum_j dS_ij k_pe_j
__global__ void __launch_bounds__(256) lat_bwd_dq_kernel(LatArgs a) {
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Ds = Qs + AT * QS;
  float* Ks = Ds + AT * LS;
  float* Ss = Ks + AT * QS;
  const int qt = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int r = threadIdx.x >> 3, sub = threadIdx.x & 7;
  const int q0 = qt * AT, qi = q0 + r;
  load_q(Qs, a, b, h, q0);
  load_dol(Ds, a, b, h, q0);
  const float sl2 = a.scale * LOG2E;
  float my_l2 = 0.f, my_dl = 0.f;
  if (qi < a.S) {
    const long long pr = ((long long)b * a.H + h) * a.s_pad + qi;
    my_l2 = a.lse2[pr];
    my_dl = a.delta[pr];
  }
  float acc[72];   // 64 latent + 8 rope columns
#pragma unroll
  for (int i = 0; i < 72; ++i) acc[i] = 0.f;
  for (int kt = 0; kt <= qt; ++kt) {
    __syncthreads();
    load_k(Ks, a, b, kt * AT);
    __syncthreads();
    float s[4] = {0.f, 0.f, 0.f, 0.f}, dp[4] = {0.f, 0.f, 0.f, 0.f};
    for (int d = 0; d < DQA; ++d) {
      const float qv = Qs[r * QS + d];
      const float gv = d < DKV ? Ds[r * LS + d] : 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float kv = Ks[(sub + 8 * c) * QS + d];
        s[c] = fmaf(qv, kv, s[c]);
        dp[c] = fmaf(gv, kv, dp[c]);   // dP = dO_lat . V with V = L
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int key = kt * AT + sub + 8 * c;
      const bool ok = key <= qi && key < a.S && qi < a.S;
      const float p = ok ? exp2f(s[c] * sl2 - my_l2) : 0.f;
      Ss[r * PS + sub + 8 * c] = p * (dp[c] - my_dl) * a.scale;
    }
    __syncthreads();
    for (int cc = 0; cc < AT; ++cc) {
      const float ds = Ss[r * PS + cc];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = fmaf(ds, Ks[cc * QS + sub + 8 * i], acc[i]);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[64 + i] = fmaf(ds, Ks[cc * QS + DKV + sub + 8 * i], acc[64 + i]);
    }
  }
  if (qi < a.S) {
    const long long row = rid(a, b, qi, h);
#pragma unroll
    for (int i = 0; i < 64; ++i) a.dqabs[row * DKV + sub + 8 * i] = acc[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) a.dq[row * DQK + DN + sub + 8 * i] = acc[64 + i];
  }
}

// key-stationary over all heads: dL_j = sum_h sum_i (scale dS_ij q_abs_i + P_ij dO_lat_i),
// dk_pe_{j,h} = scale sum_i dS_ij q_rope_i.  grid (key tiles, B)
__global__ void __launch_bounds__(256) lat_bwd_dk_kernel(LatArgs a) {
  extern __shared__ float sm[];
  float* Ks = sm;
  float* Qs = Ks + AT * QS;
  float* Ds = Qs + AT * QS;
  float* Ps = Ds + AT * LS;
  float* Ss = Ps + AT * PS;
  float* l2s = Ss + AT * PS;
  float* dls = l2s + AT;
  const int kt = blockIdx.x, b = blockIdx.y;
  const int r = threadIdx.x >> 3, sub = threadIdx.x & 7;
  const int k0 = kt * AT, key = k0 + r;
  const int nqt = (a.S + AT - 1) / AT;
  load_k(Ks, a, b, k0);
  const float sl2 = a.scale * LOG2E;
  float dl[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) dl[i] = 0.f;
  for (int h = 0; h < a.H; ++h) {
    float dk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) dk[i] = 0.f;
    for (int qt = kt; qt < nqt; ++qt) {
      const int q0 = qt * AT;
      __syncthreads();
      load_q(Qs, a, b, h, q0);
      load_dol(Ds, a, b, h, q0);
      if (threadIdx.x < AT) {
        const int s = q0 + threadIdx.x;
        const long long pr = ((long long)b * a.H + h) * a.s_pad + s;
        l2s[threadIdx.x] = s < a.S ? a.lse2[pr] : 0.f;
        dls[threadIdx.x] = s < a.S ? a.delta[pr] : 0.f;
      }
      __syncthreads();
      float s[4] = {0.f, 0.f, 0.f, 0.f}, dp[4] = {0.f, 0.f, 0.f, 0.f};
      for (int d = 0; d < DQA; ++d) {
        const float kv = Ks[r * QS + d];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          s[c] = fmaf(kv, Qs[(sub + 8 * c) * QS + d], s[c]);
          if (d < DKV) dp[c] = fmaf(kv, Ds[(sub + 8 * c) * LS + d], dp[c]);
        }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int col = sub + 8 * c, q = q0 + col;
        const bool ok = q >= key && q < a.S && key < a.S;
        const float p = ok ? exp2f(s[c] * sl2 - l2s[col]) : 0.f;
        Ps[r * PS + col] = p;
        Ss[r * PS + col] = p * (dp[c] - dls[col]) * a.scale;
      }
      __syncthreads();
      for (int cc = 0; cc < AT; ++cc) {
        const float p = Ps[r * PS + cc], ds = Ss[r * PS + cc];
#pragma unroll
        for (int i = 0; i < 64; ++i)
          dl[i] = fmaf(ds, Qs[cc * QS + sub + 8 * i], fmaf(p, Ds[cc * LS + sub + 8 * i], dl[i]));
#pragma unroll
        for (int i = 0; i < 8; ++i) dk[i] = fmaf(ds, Qs[cc * QS + DKV + sub + 8 * i], dk[i]);
      }
    }
    if (key < a.S) {
      const long long row = rid(a, b, key, h);
#pragma unroll
      for (int i = 0; i < 8; ++i) a.dkpe[row * DR + sub + 8 * i] = dk[i];
    }
  }
  if (key < a.S) {
    const long long tok = (long long)b * a.S + key;
#pragma unroll
    for (int i = 0; i < 64; ++i) a.dL[tok * DKV + sub + 8 * i] = dl[i];
  }
}

LatArgs lat_args(const Plan& p, const Ptrs& x) {
  LatArgs a{};
  a.B = p.B; a.S = p.S; a.H = p.H;
  a.scale = p.scale;
  a.qabs = x.buf<__nv_bfloat16>(p, W_QABS);
  a.qr = x.buf<__nv_bfloat16>(p, W_QR);
  a.L = x.buf<__nv_bfloat16>(p, W_L);
  a.kpe = x.buf<__nv_bfloat16>(p, W_KPE);
  a.olat = x.buf<__nv_bfloat16>(p, W_OLAT);
  a.lse = x.lse;
  a.s_pad = p.s_pad();
  if (x.ws_bwd) {
    a.lse2 = x.buf<float>(p, T_LSE2);
    a.delta = x.buf<float>(p, T_DELTA);
    a.dolat = x.buf<__nv_bfloat16>(p, T_DOLAT);
    a.dqabs = x.buf<float>(p, T_DQABS);
    a.dq = x.buf<float>(p, T_DQ);
    a.dL = x.buf<float>(p, T_DL);
    a.dkpe = x.buf<float>(p, T_DKPE);
  }
  return a;
}

cudaError_t set_smem(const void* f, size_t bytes) {
  return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_absorbed_fwd(const Plan& p, const Ptrs& x, cudaStream_t st) {
  Views v = make_views(p, x);
  const long long H = p.H, T = p.tokens();
  __nv_bfloat16* qabs = x.buf<__nv_bfloat16>(p, W_QABS);
  cudaError_t e;
  // q_abs[t,h,k] = sum_e q_nope[t,h,e] W[k, h*256 + e]      (z = h)
  e = bgemm("abs_qabs", p.H, (int)T, DKV, DN, v.qn, Mat{v.qn_ld, H * v.qn_ld, 1}, v.W,
            Mat{DH, 1, v.w_ld}, qabs, Mat{DKV, H * DKV, 1}, st);
  if (e != cudaSuccess) return e;
  LatArgs a = lat_args(p, x);
  const size_t smem = sizeof(float) * (2 * AT * QS + AT * PS);
  if ((e = set_smem((const void*)lat_fwd_kernel, smem)) != cudaSuccess) return e;
  {
    LaunchScope ls_("abs_lat_fwd", st);
    lat_fwd_kernel<<<dim3((p.S + AT - 1) / AT, p.H, p.B), 256, smem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // O[t,h,d] = sum_k o_lat[t,h,k] W[k, h*256 + 128 + d]     (z = h)
  return bgemm("abs_unabsorb", p.H, (int)T, DV, DKV, a.olat, Mat{DKV, H * DKV, 1}, v.W + DN,
               Mat{DH, v.w_ld, 1}, v.O, Mat{DV, H * DV, 1}, st);
}

cudaError_t launch_absorbed_bwd(const Plan& p, const Ptrs& x, cudaStream_t st) {
  Views v = make_views(p, x);
  const long long H = p.H, T = p.tokens();
  LatArgs a = lat_args(p, x);
  float* dw = p.canonical ? x.dw : x.buf<float>(p, T_DWC);
  __nv_bfloat16* dolat = x.buf<__nv_bfloat16>(p, T_DOLAT);
  cudaError_t e;
  // dO_lat[t,h,k] = sum_d dO[t,h,d] W[k, h*256 + 128 + d]
  e = bgemm("abs_dolat", p.H, (int)T, DKV, DV, v.dO, Mat{DV, H * DV, 1}, v.W + DN,
            Mat{DH, 1, v.w_ld}, dolat, Mat{DKV, H * DKV, 1}, st);
  if (e != cudaSuccess) return e;
  // dW^v[k, h*256 + 128 + d] = sum_t o_lat[t,h,k] dO[t,h,d]
  e = bgemm("abs_dwv", p.H, DKV, DV, (int)T, a.olat, Mat{DKV, 1, H * DKV}, v.dO,
            Mat{DV, H * DV, 1}, dw + DN, Mat{DH, H * DH, 1}, st);
  if (e != cudaSuccess) return e;
  const size_t smem_q = sizeof(float) * (2 * AT * QS + AT * LS + AT * PS);
  const size_t smem_k = sizeof(float) * (2 * AT * QS + AT * LS + 2 * AT * PS + 2 * AT);
  if ((e = set_smem((const void*)lat_bwd_dq_kernel, smem_q)) != cudaSuccess) return e;
  if ((e = set_smem((const void*)lat_bwd_dk_kernel, smem_k)) != cudaSuccess) return e;
  {
    LaunchScope ls_("abs_lat_bwd_dq", st);
    lat_bwd_dq_kernel<<<dim3((p.S + AT - 1) / AT, p.H, p.B), 256, smem_q, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    LaunchScope ls_("abs_lat_bwd_dk", st);
    lat_bwd_dk_kernel<<<dim3((p.S + AT - 1) / AT, p.B), 256, smem_k, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // dW^k[k, h*256 + e] = sum_t dq_abs[t,h,k] q_nope[t,h,e]
  e = bgemm("abs_dwk", p.H, DKV, DN, (int)T, a.dqabs, Mat{DKV, 1, H * DKV}, v.qn,
            Mat{v.qn_ld, H * v.qn_ld, 1}, dw, Mat{DH, H * DH, 1}, st);
  if (e != cudaSuccess) return e;
  // dq_nope[t,h,e] = sum_k dq_abs[t,h,k] W[k, h*256 + e]   -> columns 0..127 of the dq accumulator
  return bgemm("abs_dqnope", p.H, (int)T, DN, DKV, a.dqabs, Mat{DKV, H * DKV, 1}, v.W,
               Mat{DH, v.w_ld, 1}, a.dq, Mat{DQK, H * DQK, 1}, st);
}

}  // namespace laga
