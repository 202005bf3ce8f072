// a5 causal MLA attention backward on the 5th-generation tensor cores
// (Section 5.2).  With P = exp(s - LSE), delta = rowsum(dO * O):
//   dV = P^T dO,  dP = dO V^T,  dS = P (dP - delta) * scale,
//   dQ = dS K,    dK = dS^T Q   (the k_pe band of dK kept per head).
//
// One CTA per (128-key tile j, head h, batch b), taken from a global work
// counter in order of increasing j (longest first).  It walks the query
// tiles i = j .. last.  10 warps:
//   warps 0-3  "softmax": thread r owns key row r.  Reads S^T = K Q_i^T and
//              dP^T = V dO_i^T rows from TMEM, forms P^T (bf16, written back
//              into the S^T columns for the TMEM-operand MMA) and
//              dS^T * scale (bf16, written to shared memory, 128-byte
//              swizzled, for the shared-memory-operand MMAs).
//   warps 4-7  "dQ": read dQ_i = dS K_j (query rows) and the k_pe part of
//              dK_j for this i (key rows) from TMEM; add dQ_i into the fp32
//              dQ accumulator in global memory in a fixed order (key tile
//              0, 1, 2, ... through a per-(b,h,i) semaphore), so every run
//              sums identically; keep the k_pe part of dK in registers.
//   warp 8     TMA producer: K_j, V_j once; Q_i, dO_i, LSE_i, delta_i per i.
//   warp 9     TMEM allocator and MMA issuer.
// TMEM columns: dV [0,128), dK_nope [128,256), S^T -> P^T [256,384),
// dP^T [384,512); after the softmax warps are done: dK_rope_i [256,320),
// dQ_i [320,512).
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace laga {
namespace {
using namespace sm100;

constexpr int BT = 128;                  // key tile = query tile
constexpr int BOX = 128 * 64 * 2;        // 16 KB
constexpr int K_OFF = 0;                 // K_j: 3 boxes
constexpr int V_OFF = 3 * BOX;           // V_j: 2 boxes
constexpr int Q_OFF = 5 * BOX;           // Q_i: 3 boxes
constexpr int DO_OFF = 8 * BOX;          // dO_i: 2 boxes
constexpr int DS_OFF = 10 * BOX;         // dS^T: 2 boxes
constexpr int LSE_OFF = 12 * BOX;        // 128 fp32
constexpr int DLT_OFF = LSE_OFF + 512;   // 128 fp32
constexpr int SMEM_BYTES = DLT_OFF + 512 + 1024;
constexpr int THREADS = 320;
constexpr uint32_t TMEM_COLS = 512;
constexpr int C_DV = 0, C_DK = 128, C_S = 256, C_DP = 384, C_DKR = 256, C_DQ = 320;
constexpr uint32_t KV_BYTES = 5 * BOX;
constexpr uint32_t QDO_BYTES = 5 * BOX + 1024;
constexpr uint32_t kSpinPolls = 1u << 24;

struct BwdMaps {
  CUtensorMap qn, qr, kv, kpe, dO, lse, dlt;
};
struct BwdParams {
  int S, H, B, n_t;
  float sl2;                 // scale * log2(e)
  float scale;
  __nv_bfloat16* dkv;        // per-head [.., 256]
  long long kv_sb, kv_ss, kv_sh;
  float* dkpe;               // [R, 64]
  float* dq;                 // [R, 192] fp32 accumulator
  int* sem;                  // [B*H*n_t] ordered-dQ semaphores (zeroed per call)
  int* counter;              // work counter (zeroed per call)
  int* err;
};

// Row r of a [128 x 128] bf16 tile stored as two 128-byte-swizzled boxes of
// 64 columns: 16-byte chunk c (8 bf16) of the row.
LAGA_DEVINL uint32_t sw_chunk_off(int r, int c) {
  return (uint32_t)((c >> 3) * BOX + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_tc_kernel(const __grid_constant__ BwdMaps tm, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_kv, bar_qdo, bar_qdo_free, bar_s, bar_p, bar_dq, bar_tfree, bar_fin;
  __shared__ uint32_t tmem_sh;
  __shared__ int item_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    item_sh = atomicAdd(p.counter, 1);
    mbar_init(&bar_kv, 1);
    mbar_init(&bar_qdo, 1);
    mbar_init(&bar_qdo_free, 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_p, 4);
    mbar_init(&bar_dq, 1);
    mbar_init(&bar_tfree, 4);
    mbar_init(&bar_fin, 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&tmem_sh, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;
  const int per = p.H * p.B;
  const int item = item_sh;
  const int j = item / per;
  const int h = (item % per) % p.H;
  const int b = (item % per) / p.H;
  const int k0 = j * BT;
  const int n_i = p.n_t - j;   // query tiles j .. n_t-1

  if (warp == 8) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar_kv, KV_BYTES);
      tma_load_4d(sm + K_OFF, &tm.kv, &bar_kv, 0, k0, h, b);
      tma_load_4d(sm + K_OFF + BOX, &tm.kv, &bar_kv, 64, k0, h, b);
      tma_load_3d(sm + K_OFF + 2 * BOX, &tm.kpe, &bar_kv, 0, k0, b);
      tma_load_4d(sm + V_OFF, &tm.kv, &bar_kv, 128, k0, h, b);
      tma_load_4d(sm + V_OFF + BOX, &tm.kv, &bar_kv, 192, k0, h, b);
      for (int t = 0; t < n_i; ++t) {
        const int q0 = (j + t) * BT;
        if (t > 0 && !mbar_wait(&bar_qdo_free, (t - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&bar_qdo, QDO_BYTES);
        tma_load_4d(sm + Q_OFF, &tm.qn, &bar_qdo, 0, h, q0, b);
        tma_load_4d(sm + Q_OFF + BOX, &tm.qn, &bar_qdo, 64, h, q0, b);
        tma_load_4d(sm + Q_OFF + 2 * BOX, &tm.qr, &bar_qdo, 0, h, q0, b);
        tma_load_4d(sm + DO_OFF, &tm.dO, &bar_qdo, 0, h, q0, b);
        tma_load_4d(sm + DO_OFF + BOX, &tm.dO, &bar_qdo, 64, h, q0, b);
        tma_load_2d(sm + LSE_OFF, &tm.lse, &bar_qdo, q0, b * p.H + h);
        tma_load_2d(sm + DLT_OFF, &tm.dlt, &bar_qdo, q0, b * p.H + h);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idST = idesc_bf16(128, 128, 0, 0);
      const uint32_t idDV = idesc_bf16(128, 128, 0, 1);
      const uint32_t idDKn = idesc_bf16(128, 128, 0, 1);
      const uint32_t idDKr = idesc_bf16(128, 64, 0, 1);
      const uint32_t idDQ = idesc_bf16(128, 192, 1, 1);
      const uint32_t kb = smem_u32(sm + K_OFF), vb = smem_u32(sm + V_OFF);
      const uint32_t qb = smem_u32(sm + Q_OFF), gb = smem_u32(sm + DO_OFF);
      const uint32_t sb = smem_u32(sm + DS_OFF);
      bool ok = mbar_wait(&bar_kv, 0, p.err);
      for (int t = 0; ok && t < n_i; ++t) {
        if (!mbar_wait(&bar_qdo, t & 1, p.err)) break;
        if (t > 0 && !mbar_wait(&bar_tfree, (t - 1) & 1, p.err)) break;
        tc_fence_after();
        // S^T = K Q^T (12 K-steps over d = 192), dP^T = V dO^T (8 over d_v)
#pragma unroll
        for (int s = 0; s < 12; ++s) {
          const uint32_t off = (s >> 2) * BOX + (s & 3) * 32;
          mma_ss(tmem + C_S, sdesc_sw128(kb + off, 16, 1024), sdesc_sw128(qb + off, 16, 1024),
                 idST, s > 0);
        }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t off = (s >> 2) * BOX + (s & 3) * 32;
          mma_ss(tmem + C_DP, sdesc_sw128(vb + off, 16, 1024), sdesc_sw128(gb + off, 16, 1024),
                 idST, s > 0);
        }
        mma_commit(&bar_s);
        if (!mbar_wait(&bar_p, t & 1, p.err)) break;
        tc_fence_after();
        // dV += P^T dO (P^T from TMEM), dK_nope += dS^T Q_nope, dK_rope_i = dS^T Q_rope
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ts(tmem + C_DV, tmem + C_S + s * 8, sdesc_sw128(gb + s * 2048, BOX, 1024), idDV,
                 (t > 0 || s > 0) ? 1u : 0u);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint64_t ad = sdesc_sw128(sb + (s >> 2) * BOX + (s & 3) * 32, 16, 1024);
          mma_ss(tmem + C_DK, ad, sdesc_sw128(qb + s * 2048, BOX, 1024), idDKn,
                 (t > 0 || s > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint64_t ad = sdesc_sw128(sb + (s >> 2) * BOX + (s & 3) * 32, 16, 1024);
          mma_ss(tmem + C_DKR, ad, sdesc_sw128(qb + 2 * BOX + s * 2048, BOX, 1024), idDKr, s > 0);
        }
        mma_commit(&bar_qdo_free);
        // dQ_i = dS K (dS read MN-major from the dS^T tile, K MN-major)
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ss(tmem + C_DQ, sdesc_sw128(sb + s * 2048, BOX, 1024),
                 sdesc_sw128(kb + s * 2048, BOX, 1024), idDQ, s > 0);
        mma_commit(&bar_dq);
      }
      mma_commit(&bar_fin);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------- softmax
    const int r = threadIdx.x;          // key row
    const int key = k0 + r;
    const float* lse_s = reinterpret_cast<const float*>(sm + LSE_OFF);
    const float* dlt_s = reinterpret_cast<const float*>(sm + DLT_OFF);
    uint8_t* ds_tile = sm + DS_OFF;
    for (int t = 0; t < n_i; ++t) {
      const int q0 = (j + t) * BT;
      if (!mbar_wait(&bar_s, t & 1, p.err)) break;
      tc_fence_after();
      // valid q columns for this key row: q >= key (causal), q < S
      const int qlo = key - q0;          // first valid column (may be <= 0)
      const int qhi = p.S - q0;          // columns >= qhi are past the sequence
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t us[32], ud[32];
        tmem_ld32(tmem_addr(tmem, warp, C_S + c * 32), us);
        tmem_ld32(tmem_addr(tmem, warp, C_DP + c * 32), ud);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float pv[2], dv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int col = c * 32 + 2 * k + e;
            const bool ok = col >= qlo && col < qhi && key < p.S;
            const float pp =
                ok ? exp2f(fmaf(__uint_as_float(us[2 * k + e]), p.sl2, -lse_s[col])) : 0.f;
            pv[e] = pp;
            dv[e] = pp * (__uint_as_float(ud[2 * k + e]) - dlt_s[col]) * p.scale;
          }
          pk[k] = pack_bf16(pv[0], pv[1]);
          dk[k] = pack_bf16(dv[0], dv[1]);
        }
        tmem_st16(tmem_addr(tmem, warp, C_S + c * 16), pk);
        // dS^T row r, q columns c*32 .. c*32+31 = 16-byte chunks 4c .. 4c+3
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 v = make_uint4(dk[4 * k], dk[4 * k + 1], dk[4 * k + 2], dk[4 * k + 3]);
          *reinterpret_cast<uint4*>(ds_tile + sw_chunk_off(r, 4 * c + k)) = v;
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p);
    }
    // dK_nope, dV epilogue
    if (mbar_wait(&bar_fin, 0, p.err)) {
      tc_fence_after();
      __nv_bfloat16* dst = p.dkv + b * p.kv_sb + (long long)key * p.kv_ss + h * p.kv_sh;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t u[32];
        // columns 0..127 of dkv <- dK_nope (TMEM 128..255); 128..255 <- dV (TMEM 0..127)
        const int tc = c < 4 ? C_DK + c * 32 : C_DV + (c - 4) * 32;
        tmem_ld32(tmem_addr(tmem, warp, tc), u);
        if (key < p.S) {
          uint4 v4[4];
          uint32_t* w = reinterpret_cast<uint32_t*>(v4);
#pragma unroll
          for (int k = 0; k < 16; ++k)
            w[k] = pack_bf16(__uint_as_float(u[2 * k]), __uint_as_float(u[2 * k + 1]));
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) d4[k] = v4[k];
        }
      }
    }
  } else {
    // ------------------------------------------------------------- dQ warps 4..7
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;       // TMEM lane: query row (dQ), key row (dK_rope)
    const int key = k0 + r;
    float acc[64];
#pragma unroll
    for (int k = 0; k < 64; ++k) acc[k] = 0.f;
    for (int t = 0; t < n_i; ++t) {
      const int i = j + t;
      const int q = i * BT + r;
      if (!mbar_wait(&bar_dq, t & 1, p.err)) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem_addr(tmem, q4, C_DKR + c * 32), u);
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[c * 32 + k] += __uint_as_float(u[k]);
      }
      // wait for this (b, h, i) tile's turn: key tiles add in order 0, 1, ..., i
      int* sem = p.sem + ((long long)b * p.H + h) * p.n_t + i;
      if (threadIdx.x == 128) {
        uint32_t n = 0;
        while (ld_acquire_gpu(sem) != j) {
          if (++n > kSpinPolls) {
            atomicExch(p.err, DEV_ERR_TIMEOUT);
            break;
          }
          if (n > 32) __nanosleep(128);
        }
      }
      named_bar_sync(1, 128);
      float* dq_row = p.dq + (((long long)b * p.S + q) * p.H + h) * DQK;
#pragma unroll 1
      for (int c = 0; c < 6; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem_addr(tmem, q4, C_DQ + c * 32), u);
        if (q < p.S) {
          float4* d4 = reinterpret_cast<float4*>(dq_row + c * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float4 v = make_float4(__uint_as_float(u[4 * k]), __uint_as_float(u[4 * k + 1]),
                                   __uint_as_float(u[4 * k + 2]), __uint_as_float(u[4 * k + 3]));
            if (j == 0) {
              __stcg(d4 + k, v);
            } else {
              float4 o = __ldcg(d4 + k);
              o.x += v.x; o.y += v.y; o.z += v.z; o.w += v.w;
              __stcg(d4 + k, o);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_tfree);
      __threadfence();
      named_bar_sync(1, 128);
      if (threadIdx.x == 128) st_release_gpu(sem, j + 1);
    }
    if (key < p.S) {
      float* dst = p.dkpe + (((long long)b * p.S + key) * p.H + h) * DR;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        reinterpret_cast<float4*>(dst)[k] =
            make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_attn_bwd(const Plan& p, const Ptrs& x, cudaStream_t st) {
  Views v = make_views(p, x);
  const uint64_t S = p.S, H = p.H, B = p.B;
  BwdMaps tm;
  cudaError_t e;
  {
    const uint64_t ld = (uint64_t)v.qn_ld * 2;
    uint64_t dims[4] = {128, H, S, B}, str[3] = {ld, H * ld, S * H * ld};
    uint32_t box[4] = {64, 1, 128, 1};
    if ((e = make_tmap_bf16(&tm.qn, v.qn, 4, dims, str, box)) != cudaSuccess) return e;
  }
  {
    uint64_t dims[4] = {64, H, S, B}, str[3] = {128, H * 128, S * H * 128};
    uint32_t box[4] = {64, 1, 128, 1};
    if ((e = make_tmap_bf16(&tm.qr, v.qr, 4, dims, str, box)) != cudaSuccess) return e;
  }
  {
    uint64_t dims[4] = {128, H, S, B}, str[3] = {256, H * 256, S * H * 256};
    uint32_t box[4] = {64, 1, 128, 1};
    if ((e = make_tmap_bf16(&tm.dO, v.dO, 4, dims, str, box)) != cudaSuccess) return e;
  }
  {
    uint64_t dims[4] = {256, S, H, B};
    uint64_t str[3] = {(uint64_t)v.kv_ss * 2, (uint64_t)v.kv_sh * 2, (uint64_t)v.kv_sb * 2};
    uint32_t box[4] = {64, 128, 1, 1};
    if ((e = make_tmap_bf16(&tm.kv, v.kv, 4, dims, str, box)) != cudaSuccess) return e;
  }
  {
    uint64_t dims[3] = {64, S, B}, str[2] = {128, S * 128};
    uint32_t box[3] = {64, 128, 1};
    if ((e = make_tmap_bf16(&tm.kpe, v.kpe, 3, dims, str, box)) != cudaSuccess) return e;
  }
  {
    // rows padded to a multiple of 128 floats; extent S so TMA zero-fills the tail
    uint64_t dims[2] = {S, B * H}, str[1] = {(uint64_t)p.s_pad() * 4};
    uint32_t box[2] = {128, 1};
    if ((e = make_tmap_f32(&tm.lse, x.buf<float>(p, T_LSE2), 2, dims, str, box)) != cudaSuccess)
      return e;
    if ((e = make_tmap_f32(&tm.dlt, x.buf<float>(p, T_DELTA), 2, dims, str, box)) != cudaSuccess)
      return e;
  }
  BwdParams prm;
  prm.S = p.S;
  prm.H = p.H;
  prm.B = p.B;
  prm.n_t = (p.S + BT - 1) / BT;
  prm.sl2 = p.scale * 1.4426950408889634f;
  prm.scale = p.scale;
  prm.dkv = x.buf<__nv_bfloat16>(p, T_DKV);
  prm.kv_sb = v.kv_sb;
  prm.kv_ss = v.kv_ss;
  prm.kv_sh = v.kv_sh;
  prm.dkpe = x.buf<float>(p, T_DKPE);
  prm.dq = x.buf<float>(p, T_DQ);
  prm.sem = x.buf<int>(p, T_SEM);
  prm.counter = prm.sem + (long long)p.B * p.H * prm.n_t;
  prm.err = x.err;
  e = cudaFuncSetAttribute(attn_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)prm.n_t * p.H * p.B;
  LaunchScope ls_("attn_bwd", st);
  attn_bwd_tc_kernel<<<(unsigned)grid, THREADS, SMEM_BYTES, st>>>(tm, prm);
  return cudaGetLastError();
}

}  // namespace laga
