// a3 head-shard up-projection and its backward on the tensor cores
// (Algorithm 1 step 4; Section 5.1 k_nope[i,t] = W^k[i] L[t],
// v[i,t] = W^v[i] L[t]; Section 5.2 W_kv_b gradient shard):
//   UP   KV[t, h, :]  = L[t, :] . W[:, h*256 : h*256+256]        M=tokens N=256/head K=512
//   DL   dL[t, :]     = sum_h dKV[t, h, :] . W[:, h-cols]^T       M=tokens N=512      K=H*256
//   DW   dW[:, h-cols] = sum_t L[t, :]^T dKV[t, h, :]             M=512    N=256/head K=tokens
// One CTA per 128 x 256 output tile, two CTAs per SM (each one's prologue and
// epilogue overlap the other's main loop); 6 warps: warp 0 TMA producer
// (2-stage ring), warp 1 TMEM allocator + MMA issuer (M128 N256 K16 steps,
// fp32 accumulator in 256 TMEM columns), warps 2-5 epilogue (TMEM ->
// registers -> swizzled tiles in the idle ring -> TMA tensor stores).  DW splits the token reduction into a fixed number of chunks whose
// fp32 partial tiles are summed afterwards in chunk order, so every run adds
// in the same order.  Each output element is one accumulation over K in
// ascending K-step order whatever the K/V layout, which keeps the
// token-major (LAGA) and head-major (explicit) layouts bit-identical.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace laga {
namespace {
using namespace sm100;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 2;   // two CTAs per SM
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
constexpr int THREADS = 192;
constexpr int BOX8K = 64 * 64 * 2;

enum Mode { UP = 0, DL = 1, DW = 2 };

struct GemmMaps {
  CUtensorMap a, b;
  CUtensorMap o;      // output: UP KV, 64 x 128 bf16 boxes; DL / DW fp32, 32 x 32 boxes
};
struct GemmParams {
  int S, H, B;
  int k_steps;        // K steps handled by one CTA
  int k_steps_total;  // DW: token steps over all batches
  // outputs
  __nv_bfloat16* kv; long long kv_sb, kv_ss, kv_sh;   // UP
  float* out; long long out_ld;                        // DL: dL; DW: dW (or partials)
  long long split_stride;                              // DW: elements between split partials
  int* err;
};

template <int MODE>
LAGA_DEVINL void load_stage(const GemmMaps& tm, uint8_t* a_dst, uint8_t* b_dst, uint64_t* bar,
                            int kstep, int m0, int n_tile, int b_idx, const GemmParams& p) {
  if (MODE == UP) {
    tma_load_3d(a_dst, &tm.a, bar, kstep * BK, m0, b_idx);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      tma_load_2d(b_dst + i * BOX8K, &tm.b, bar, n_tile * BN + i * 64, kstep * BK);
  } else if (MODE == DL) {
    const int h = kstep >> 2, e0 = (kstep & 3) * 64;
    tma_load_4d(a_dst, &tm.a, bar, e0, m0, h, b_idx);
    tma_load_2d(b_dst, &tm.b, bar, kstep * BK, n_tile * BN);
  } else {
    // K index = token: step -> (batch, 64-token chunk)
    const int chunks = (p.S + 63) / 64;
    const int bb = kstep / chunks, s0 = (kstep % chunks) * 64;
    tma_load_3d(a_dst, &tm.a, bar, m0, s0, bb);
    tma_load_3d(a_dst + BOX8K, &tm.a, bar, m0 + 64, s0, bb);
#pragma unroll
    for (int i = 0; i < 4; ++i) tma_load_4d(b_dst + i * BOX8K, &tm.b, bar, i * 64, s0, n_tile, bb);
  }
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 2)
    gemm_tc_kernel(const __grid_constant__ GemmMaps tm, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_full[STAGES], bar_empty[STAGES], bar_done;
  __shared__ uint32_t tmem_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tile = blockIdx.x;
  const int m_tile = blockIdx.y;
  const int zz = blockIdx.z;  // UP/DL: batch; DW: split
  const int m0 = m_tile * BM;
  const int b_idx = MODE == DW ? 0 : zz;
  const int k_first = MODE == DW ? zz * p.k_steps : 0;
  const int k_count = MODE == DW ? max(0, min(p.k_steps, p.k_steps_total - k_first)) : p.k_steps;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
    }
    mbar_init(&bar_done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_sh, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;
  bool staged = false;   // UP: this epilogue thread staged its row of the tile

  if (warp == 0) {
    if (lane == 0) {
      for (int k = 0; k < k_count; ++k) {
        const int st = k % STAGES;
        if (k >= STAGES && !mbar_wait(&bar_empty[st], ((k / STAGES) - 1) & 1, p.err)) break;
        uint8_t* a_dst = sm + st * STAGE_BYTES;
        mbar_arrive_expect_tx(&bar_full[st], STAGE_BYTES);
        load_stage<MODE>(tm, a_dst, a_dst + A_BYTES, &bar_full[st], k_first + k, m0, n_tile,
                         b_idx, p);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, BN, MODE == DW, MODE != DL);
      for (int k = 0; k < k_count; ++k) {
        const int st = k % STAGES;
        if (!mbar_wait(&bar_full[st], (k / STAGES) & 1, p.err)) break;
        tc_fence_after();
        const uint32_t a = smem_u32(sm + st * STAGE_BYTES);
        const uint32_t bsm = a + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = MODE == DW ? sdesc_sw128(a + kk * 2048, BOX8K, 1024)
                                         : sdesc_sw128(a + kk * 32, 16, 1024);
          const uint64_t bd = MODE == DL ? sdesc_sw128(bsm + kk * 32, 16, 1024)
                                         : sdesc_sw128(bsm + kk * 2048, BOX8K, 1024);
          mma_ss(tmem, ad, bd, idesc, (k > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bar_empty[st]);
      }
      mma_commit(&bar_done);
    }
  } else {
    // epilogue warps 2..5: TMEM lane quadrant = warp % 4
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const bool have = k_count > 0;
    if (mbar_wait(&bar_done, 0, p.err)) {
      staged = true;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t u[32];
        if (have) {
          tmem_ld32(tmem_addr(tmem, q, c * 32), u);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) u[k] = 0u;
        }
        if (MODE == UP) {
          // staged in the idle ring as four 128 x 64 swizzled boxes, written
          // by TMA after the final barrier (rows past the sequence clipped)
          uint8_t* box = sm + (c >> 1) * (BM * 128) + r * 128;
          const int k0 = (c & 1) * 4;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(u[8 * g]), __uint_as_float(u[8 * g + 1]));
            w.y = pack_bf16(__uint_as_float(u[8 * g + 2]), __uint_as_float(u[8 * g + 3]));
            w.z = pack_bf16(__uint_as_float(u[8 * g + 4]), __uint_as_float(u[8 * g + 5]));
            w.w = pack_bf16(__uint_as_float(u[8 * g + 6]), __uint_as_float(u[8 * g + 7]));
            *reinterpret_cast<uint4*>(box + (((k0 + g) ^ (r & 7)) << 4)) = w;
          }
        } else {
          // fp32 output: each epilogue warp stages its own 32 rows, four
          // 32 x 32 swizzled boxes at a time, and lane 0 stores them by TMA
          // (rows past the output are clipped there); no block barrier
          uint8_t* wst = sm + q * 16384 + (c & 3) * 4096 + lane * 128;
#pragma unroll
          for (int g = 0; g < 8; ++g)
            *reinterpret_cast<float4*>(wst + ((g ^ (lane & 7)) << 4)) =
                make_float4(__uint_as_float(u[4 * g]), __uint_as_float(u[4 * g + 1]),
                            __uint_as_float(u[4 * g + 2]), __uint_as_float(u[4 * g + 3]));
          if ((c & 3) == 3) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                tma_store_3d(&tm.o, sm + q * 16384 + cc * 4096, n_tile * BN + (c - 3 + cc) * 32,
                             m0 + q * 32, zz);
              bulk_commit();
              bulk_wait_read0();
            }
            __syncwarp();
          }
        }
      }
    }
  }
  if (MODE == UP && warp >= 2) fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (MODE == UP && threadIdx.x == 64 && staged) {
#pragma unroll
    for (int bx = 0; bx < BN / 64; ++bx)
      tma_store_4d(&tm.o, sm + bx * (BM * 128), bx * 64, m0, n_tile, zz);
    bulk_commit();
    bulk_wait_read0();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Sum of the DW split partials in split order.
__global__ void __launch_bounds__(256) split_reduce_kernel(const float4* __restrict__ part,
                                                           long long n4, int splits,
                                                           long long stride4,
                                                           float4* __restrict__ out) {
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n4; i += (long long)gridDim.x * 256) {
    float4 acc = part[i];
    for (int z = 1; z < splits; ++z) {
      const float4 v = part[z * stride4 + i];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    out[i] = acc;
  }
}

template <int MODE>
cudaError_t launch(const char* name, const GemmMaps& tm, const GemmParams& prm, dim3 grid,
                   cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  LaunchScope ls_(name, st);
  gemm_tc_kernel<MODE><<<grid, THREADS, SMEM_BYTES, st>>>(tm, prm);
  return cudaGetLastError();
}

cudaError_t kv_map(CUtensorMap* m, const Plan& p, const Views& v, const __nv_bfloat16* base,
                   uint32_t rows) {
  uint64_t dims[4] = {256, (uint64_t)p.S, (uint64_t)p.H, (uint64_t)p.B};
  uint64_t str[3] = {(uint64_t)v.kv_ss * 2, (uint64_t)v.kv_sh * 2, (uint64_t)v.kv_sb * 2};
  uint32_t box[4] = {64, rows, 1, 1};
  return make_tmap_bf16(m, base, 4, dims, str, box);
}

}  // namespace

cudaError_t launch_upproj(const Plan& p, const Ptrs& x, cudaStream_t st) {
  Views v = make_views(p, x);
  GemmMaps tm;
  cudaError_t e;
  {
    uint64_t dims[3] = {512, (uint64_t)p.S, (uint64_t)p.B}, str[2] = {1024, (uint64_t)p.S * 1024};
    uint32_t box[3] = {64, 128, 1};
    if ((e = make_tmap_bf16(&tm.a, v.L, 3, dims, str, box)) != cudaSuccess) return e;
  }
  {
    uint64_t dims[2] = {(uint64_t)p.H * 256, 512}, str[1] = {(uint64_t)v.w_ld * 2};
    uint32_t box[2] = {64, 64};
    if ((e = make_tmap_bf16(&tm.b, v.W, 2, dims, str, box)) != cudaSuccess) return e;
  }
  if ((e = kv_map(&tm.o, p, v, v.kv, 128)) != cudaSuccess) return e;
  GemmParams prm{};
  prm.S = p.S; prm.H = p.H; prm.B = p.B;
  prm.k_steps = 512 / BK;
  prm.kv = v.kv; prm.kv_sb = v.kv_sb; prm.kv_ss = v.kv_ss; prm.kv_sh = v.kv_sh;
  prm.err = x.err;
  dim3 grid(p.H, (p.S + BM - 1) / BM, p.B);
  return launch<UP>("upproj", tm, prm, grid, st);
}

cudaError_t launch_upproj_bwd(const Plan& p, const Ptrs& x, cudaStream_t st) {
  Views v = make_views(p, x);
  const __nv_bfloat16* dkv = x.buf<__nv_bfloat16>(p, T_DKV);
  cudaError_t e;
  // ---- dW = L^T dKV (split over tokens, partials summed in split order)
  {
    GemmMaps tm;
    {
      uint64_t dims[3] = {512, (uint64_t)p.S, (uint64_t)p.B}, str[2] = {1024, (uint64_t)p.S * 1024};
      uint32_t box[3] = {64, 64, 1};
      if ((e = make_tmap_bf16(&tm.a, v.L, 3, dims, str, box)) != cudaSuccess) return e;
    }
    if ((e = kv_map(&tm.b, p, v, dkv, 64)) != cudaSuccess) return e;
    const int splits = dw_splits(p.H);
    const int total = p.B * ((p.S + 63) / 64);
    GemmParams prm{};
    prm.S = p.S; prm.H = p.H; prm.B = p.B;
    prm.k_steps_total = total;
    prm.k_steps = (total + splits - 1) / splits;
    float* dw = p.canonical ? x.dw : x.buf<float>(p, T_DWC);
    prm.out = splits > 1 ? x.buf<float>(p, T_DWP) : dw;
    prm.out_ld = (long long)p.H * 256;
    prm.split_stride = 512LL * p.H * 256;
    {
      uint64_t dims[3] = {(uint64_t)prm.out_ld, 512, (uint64_t)splits};
      uint64_t str[2] = {(uint64_t)prm.out_ld * 4, (uint64_t)prm.split_stride * 4};
      uint32_t box[3] = {32, 32, 1};
      if ((e = make_tmap_f32(&tm.o, prm.out, 3, dims, str, box, true)) != cudaSuccess) return e;
    }
    prm.err = x.err;
    dim3 grid(p.H, 512 / BM, splits);
    if ((e = launch<DW>("upproj_dw", tm, prm, grid, st)) != cudaSuccess) return e;
    if (splits > 1) {
      const long long n4 = prm.split_stride / 4;
      LaunchScope ls_("dw_split_reduce", st);
      split_reduce_kernel<<<152 * 8, 256, 0, st>>>(reinterpret_cast<const float4*>(prm.out), n4,
                                                   splits, n4, reinterpret_cast<float4*>(dw));
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  // ---- dL = dKV W^T
  {
    GemmMaps tm;
    if ((e = kv_map(&tm.a, p, v, dkv, 128)) != cudaSuccess) return e;
    {
      uint64_t dims[2] = {(uint64_t)p.H * 256, 512}, str[1] = {(uint64_t)v.w_ld * 2};
      uint32_t box[2] = {64, 256};
      if ((e = make_tmap_bf16(&tm.b, v.W, 2, dims, str, box)) != cudaSuccess) return e;
    }
    GemmParams prm{};
    prm.S = p.S; prm.H = p.H; prm.B = p.B;
    prm.k_steps = p.H * 4;
    prm.out = x.buf<float>(p, T_DL);
    prm.out_ld = 512;
    {
      uint64_t dims[3] = {512, (uint64_t)p.S, (uint64_t)p.B}, str[2] = {512 * 4, (uint64_t)p.S * 512 * 4};
      uint32_t box[3] = {32, 32, 1};
      if ((e = make_tmap_f32(&tm.o, prm.out, 3, dims, str, box, true)) != cudaSuccess) return e;
    }
    prm.err = x.err;
    dim3 grid(2, (p.S + BM - 1) / BM, p.B);
    return launch<DL>("upproj_dl", tm, prm, grid, st);
  }
}

}  // namespace laga
