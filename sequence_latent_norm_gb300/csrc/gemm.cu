// a3 head-shard up-projection KV = L . W_kv_b[:, shard] (Algorithm 1 step 4,
// Section 5.1: k_nope[i,t] = W^k[i] L[t], v[i,t] = W^v[i] L[t]) and its
// backward (Section 5.2): dW_shard = L^T dKV, dL = dKV W_shard^T.
//
// Generic fp32-accumulating tiled GEMM over accessor functors.  Each output
// element is one dot product over K taken in ascending K order, independent
// of the tensor layouts, so the token-major (LAGA) and head-major (explicit)
// K/V layouts give bit-identical results.
#include "common.cuh"
#include "kernels.h"

namespace laga {
namespace {

struct RowBF {  // (r, c) -> p[r*ld + c]
  const __nv_bfloat16* p;
  long long ld;
  LAGA_DEVINL float operator()(long long r, long long c) const { return __bfloat162float(p[r * ld + c]); }
};
struct ColBF {  // (r, c) -> p[c*ld + r]
  const __nv_bfloat16* p;
  long long ld;
  LAGA_DEVINL float operator()(long long r, long long c) const { return __bfloat162float(p[c * ld + r]); }
};
struct KVMat {  // (token, column) of a per-head [.., 256] tensor
  const __nv_bfloat16* p;
  int S;
  long long sb, ss, sh;
  LAGA_DEVINL float operator()(long long tok, long long col) const {
    long long b = tok / S, s = tok % S, h = col >> 8, e = col & 255;
    return __bfloat162float(p[b * sb + s * ss + h * sh + e]);
  }
};
struct StoreKV {
  __nv_bfloat16* p;
  int S;
  long long sb, ss, sh;
  LAGA_DEVINL void operator()(long long tok, long long col, float v) const {
    long long b = tok / S, s = tok % S, h = col >> 8, e = col & 255;
    p[b * sb + s * ss + h * sh + e] = __float2bfloat16_rn(v);
  }
};
struct StoreF32 {
  float* p;
  long long ld;
  LAGA_DEVINL void operator()(long long r, long long c, float v) const { p[r * ld + c] = v; }
};

constexpr int TM = 64, TN = 64, TK = 16;

template <class AF, class BF, class CF>
__global__ void __launch_bounds__(256) gemm_simt_kernel(long long M, long long N, long long K,
                                                        AF A, BF B, CF C) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const long long m0 = (long long)blockIdx.y * TM, n0 = (long long)blockIdx.x * TN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (long long k0 = 0; k0 < K; k0 += TK) {
    for (int i = threadIdx.x; i < TM * TK; i += 256) {
      int mm = i % TM, kk = i / TM;
      long long gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < M && gk < K) ? A(gm, gk) : 0.f;
      long long gn = n0 + mm;
      Bs[kk][mm] = (gn < N && gk < K) ? B(gk, gn) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      long long gm = m0 + ty * 4 + i, gn = n0 + tx * 4 + j;
      if (gm < M && gn < N) C(gm, gn, acc[i][j]);
    }
}

template <class AF, class BF, class CF>
cudaError_t run_gemm(const char* name, long long M, long long N, long long K, AF A, BF B, CF C,
                     cudaStream_t st) {
  LaunchScope ls_(name, st);
  dim3 grid((unsigned)((N + TN - 1) / TN), (unsigned)((M + TM - 1) / TM));
  gemm_simt_kernel<<<grid, 256, 0, st>>>(M, N, K, A, B, C);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_upproj(const Plan& p, const Ptrs& x, cudaStream_t st) {
  Views v = make_views(p, x);
  return run_gemm("upproj", p.tokens(), (long long)p.H * 256, 512, RowBF{v.L, 512}, RowBF{v.W, v.w_ld},
                  StoreKV{v.kv, p.S, v.kv_sb, v.kv_ss, v.kv_sh}, st);
}

cudaError_t launch_upproj_bwd(const Plan& p, const Ptrs& x, cudaStream_t st) {
  Views v = make_views(p, x);
  const __nv_bfloat16* dkv = x.buf<__nv_bfloat16>(p, T_DKV);
  float* dw = p.canonical ? x.dw : x.buf<float>(p, T_DWC);
  cudaError_t e = run_gemm("upproj_dw", 512, (long long)p.H * 256, p.tokens(), ColBF{v.L, 512},
                           KVMat{dkv, p.S, v.kv_sb, v.kv_ss, v.kv_sh},
                           StoreF32{dw, (long long)p.H * 256}, st);
  if (e != cudaSuccess) return e;
  return run_gemm("upproj_dl", p.tokens(), 512, (long long)p.H * 256, KVMat{dkv, p.S, v.kv_sb, v.kv_ss, v.kv_sh},
                  ColBF{v.W, v.w_ld}, StoreF32{x.buf<float>(p, T_DL), 512}, st);
}

}  // namespace laga
