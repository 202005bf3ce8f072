// a5, query-stationary half of the causal MLA attention backward: dQ
// (Section 5.2).  With P = exp(s - LSE), delta = rowsum(dO * O):
//   dP = dO V^T,  dS = P (dP - delta) * scale,  dQ = dS K
// over the key tiles j = 0 .. i of query tile i, in the rotated frame
// (columns 0-127 against k_nope, 128-191 against k_pe).  The key-stationary
// kernel (attn_bwd_kv.cu) recomputes the same P and dS for dK and dV, so no
// partial dQ is ever exchanged between CTAs: every element of dQ is one
// fixed-order accumulation in TMEM, stored once.
//
// One CTA per (128-query tile i, head h, batch b), longest (largest i)
// first.  10 warps:
//   warps 0-7  compute.  Warp w owns TMEM lane quadrant w%4 (query rows) and
//              column half w/4 (key columns).  It reads S_ij into registers
//              as P (freeing the S columns for S_i,j+1), then reads dP_ij and
//              writes dS_ij / scale as bf16 pairs packed into its own dP
//              columns, the TMEM operand of the dQ MMA (dQ is scaled in the
//              epilogue).
//              First they place q_nope_i in TMEM as packed bf16 pairs, the
//              TMEM A operand of the first 8 K-steps of S.
//   warp 8     TMA producer: q_rope_i and dO_i once; K_j in a ring of three
//              buffers, so K_{j+2} loads while dQ of tile j-1 is the last
//              reader of its buffer; V_j single-buffered.
//   warp 9     TMEM allocator and MMA issuer.  Per j: S_i,j+1 as soon as S_ij
//              is read, then dQ += dS_ij K_j and dP_i,j+1.
// TMEM columns: S [0,128), dP [128,256) with dS in [128,160) and [192,224),
// dQ [256,448), q_nope [448,512).  Every mbarrier is waited phase by phase,
// so parity waits are exact.
// Epilogue: for the canonical bf16 layout the kernel writes the final dq,
// rotating the k_pe band back by the row's position; otherwise it writes
// fp32 rotated-frame rows that dq_final converts.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace laga {
namespace {
using namespace sm100;

constexpr int BT = 128;                  // query tile = key tile
constexpr int BOX = 128 * 64 * 2;        // 16 KB
constexpr int QR_OFF = 0;                // q_rope_i: 1 box
constexpr int DO_OFF = BOX;              // dO_i: 2 boxes
constexpr int K_OFF = 3 * BOX;           // K_j: ring of three buffers of 3 boxes (k_nope | k_pe)
constexpr int K_BUFS = 3;
constexpr int V_OFF = 12 * BOX;          // V_j: 2 boxes
constexpr int SMEM_BYTES = 14 * BOX + 1024;   // + slack to align the base
constexpr int THREADS = 320;
constexpr int N_COMPUTE = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr int C_S = 0, C_DP = 128, C_DQ = 256, C_QN = 448;
constexpr uint32_t QO_BYTES = 3 * BOX;
constexpr uint32_t K_BYTES = 3 * BOX;
constexpr uint32_t V_BYTES = 2 * BOX;

struct DqMaps {
  CUtensorMap qr, kv, kpe, dO;
  CUtensorMap dq;            // final bf16 dq [B, S, H, 192], 64 x 128 boxes (canonical dims)
};
struct DqParams {
  int S, H, B, n_t, s_pad;
  const __nv_bfloat16* qn;   // q_nope rows
  long long qn_ld;
  float sl2;                 // scale * log2(e)
  float scale;
  const float* lse2;         // [B*H, s_pad]  LSE * log2(e)
  const float* delta;        // [B*H, s_pad]
  float* dq;                 // [B, S, H, 192] fp32, rotated frame (when dq_out is null)
  __nv_bfloat16* dq_out;     // [B, S, H, 192] bf16 final dq, or null
  const float* cosT;         // [S, 32]
  const float* sinT;         // [S, 32]
  int* err;
};

// TMEM column of the K-step s (16 key columns) of the packed dS tile:
// key columns 0-63 are packed into [C_DP, C_DP+32), 64-127 into
// [C_DP+64, C_DP+96).
LAGA_DEVINL uint32_t ds_col(int s) { return s < 4 ? C_DP + 8 * s : C_DP + 64 + 8 * (s - 4); }

__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ DqMaps tm, const DqParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_qo, bar_k_full[K_BUFS], bar_k_free[K_BUFS], bar_v_full, bar_v_free;
  __shared__ uint64_t bar_qn, bar_s, bar_dp, bar_a, bar_ds, bar_fin;
  __shared__ uint32_t tmem_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bar_qo, 1);
    for (int k = 0; k < K_BUFS; ++k) {
      mbar_init(&bar_k_full[k], 1);
      mbar_init(&bar_k_free[k], 1);
    }
    mbar_init(&bar_v_full, 1);
    mbar_init(&bar_v_free, 1);
    mbar_init(&bar_qn, N_COMPUTE);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_a, N_COMPUTE);
    mbar_init(&bar_ds, N_COMPUTE);
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
  bool stored = false;   // this thread staged its part of the final dq tile
  const int per = p.H * p.B;
  const int i = p.n_t - 1 - (int)(blockIdx.x / per);   // largest query tiles first
  const int h = (int)(blockIdx.x % per) % p.H;
  const int b = (int)(blockIdx.x % per) / p.H;
  const int q0 = i * BT;
  const int n_j = i + 1;                                 // key tiles 0 .. i

  if (warp == 8) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar_qo, QO_BYTES);
      tma_load_4d(sm + QR_OFF, &tm.qr, &bar_qo, 0, h, q0, b);
      tma_load_4d(sm + DO_OFF, &tm.dO, &bar_qo, 0, h, q0, b);
      tma_load_4d(sm + DO_OFF + BOX, &tm.dO, &bar_qo, 64, h, q0, b);
      for (int j = 0; j < n_j; ++j) {
        const int k0 = j * BT;
        const int kb = j % K_BUFS;
        // K_j into buffer j%3 once dQ of tile j-3 has read it
        if (j >= K_BUFS && !mbar_wait(&bar_k_free[kb], (j / K_BUFS - 1) & 1, p.err)) break;
        uint8_t* kd = sm + K_OFF + kb * 3 * BOX;
        mbar_arrive_expect_tx(&bar_k_full[kb], K_BYTES);
        tma_load_4d(kd, &tm.kv, &bar_k_full[kb], 0, k0, h, b);
        tma_load_4d(kd + BOX, &tm.kv, &bar_k_full[kb], 64, k0, h, b);
        tma_load_3d(kd + 2 * BOX, &tm.kpe, &bar_k_full[kb], 0, k0, b);
        // V_j once dP of tile j-1 has read V_{j-1}
        if (j > 0 && !mbar_wait(&bar_v_free, (j - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&bar_v_full, V_BYTES);
        tma_load_4d(sm + V_OFF, &tm.kv, &bar_v_full, 128, k0, h, b);
        tma_load_4d(sm + V_OFF + BOX, &tm.kv, &bar_v_full, 192, k0, h, b);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16(128, 128, 0, 0);
      const uint32_t idQ = idesc_bf16(128, 192, 0, 1);
      const uint32_t qrlo = sdesc_lo(smem_u32(sm + QR_OFF), 16);
      const uint32_t glo = sdesc_lo(smem_u32(sm + DO_OFF), 16);
      const uint32_t vlo = sdesc_lo(smem_u32(sm + V_OFF), 16);
      // S_ij = Q_i K_j^T (12 K-steps over d = 192): q_nope from TMEM for
      // the first 8, q_rope from shared memory for the last 4
      auto issue_s = [&](int j) -> bool {
        if (!mbar_wait(&bar_k_full[j % K_BUFS], (j / K_BUFS) & 1, p.err)) return false;
        tc_fence_after();
        const uint32_t klo = sdesc_lo(smem_u32(sm + K_OFF + (j % K_BUFS) * 3 * BOX), 16);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t off = ((s >> 2) * BOX + (s & 3) * 32) >> 4;
          mma_ts(tmem + C_S, tmem + C_QN + 8 * s, sdesc_make(klo + off), idS, s > 0);
        }
#pragma unroll
        for (int s = 0; s < 4; ++s)
          mma_ss(tmem + C_S, sdesc_make(qrlo + ((s * 32) >> 4)),
                 sdesc_make(klo + ((2 * BOX + s * 32) >> 4)), idS, 1u);
        mma_commit(&bar_s);
        return true;
      };
      // dP_ij = dO_i V_j^T (8 K-steps over d_v); afterwards V_j is free
      auto issue_dp = [&](int j) -> bool {
        if (!mbar_wait(&bar_v_full, j & 1, p.err)) return false;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t off = ((s >> 2) * BOX + (s & 3) * 32) >> 4;
          mma_ss(tmem + C_DP, sdesc_make(glo + off), sdesc_make(vlo + off), idS, s > 0);
        }
        mma_commit(&bar_dp);
        mma_commit(&bar_v_free);
        return true;
      };
      bool ok = mbar_wait(&bar_qo, 0, p.err) && mbar_wait(&bar_qn, 0, p.err) && issue_s(0) &&
                issue_dp(0);
      for (int j = 0; ok && j < n_j; ++j) {
        // S columns are free once every compute warp has read S_ij
        if (!mbar_wait(&bar_a, j & 1, p.err)) break;
        if (j + 1 < n_j && !issue_s(j + 1)) break;
        // dQ += dS_ij K_j (dS from TMEM, K_j as the N-major B operand)
        if (!mbar_wait(&bar_ds, j & 1, p.err)) break;
        tc_fence_after();
        const uint32_t kmn = sdesc_lo(smem_u32(sm + K_OFF + (j % K_BUFS) * 3 * BOX), BOX);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ts(tmem + C_DQ, tmem + ds_col(s), sdesc_make(kmn + s * (2048 >> 4)), idQ,
                 (j > 0 || s > 0) ? 1u : 0u);
        mma_commit(&bar_k_free[j % K_BUFS]);
        // dP_i,j+1 overwrites dS_ij only after the dQ MMAs above have read it
        if (j + 1 < n_j && !issue_dp(j + 1)) break;
      }
      mma_commit(&bar_fin);
    }
  } else {
    // ------------------------------------------------------------- compute warps 0..7
    const int qd = warp & 3;            // TMEM lane quadrant
    const int ch = warp >> 2;           // column half
    const int r = qd * 32 + lane;       // TMEM lane: query row
    const int query = q0 + r;
    const bool q_ok = query < p.S;
    const long long lrow = (long long)(b * p.H + h) * p.s_pad + query;
    const float lse_r = q_ok ? p.lse2[lrow] : 0.f;
    const float dlt_r = q_ok ? p.delta[lrow] : 0.f;
    {
      // q_nope row -> TMEM [448 + 32*half, +32): dims 64*half .. +63 as bf16
      // pairs, zero past the sequence
      uint32_t w[32];
      if (q_ok) {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.qn + (((long long)b * p.S + query) * p.H + h) * p.qn_ld + ch * 64);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v4 = src[k];
          w[4 * k] = v4.x; w[4 * k + 1] = v4.y; w[4 * k + 2] = v4.z; w[4 * k + 3] = v4.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) w[k] = 0u;
      }
      tmem_st16(tmem_addr(tmem, qd, C_QN + ch * 32), *reinterpret_cast<const uint32_t(*)[16]>(w));
      tmem_st16(tmem_addr(tmem, qd, C_QN + ch * 32 + 16),
                *reinterpret_cast<const uint32_t(*)[16]>(w + 16));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_qn);
    }
    bool ok = true;
    for (int j = 0; j < n_j; ++j) {
      const int k0 = j * BT;
      const int kmax = query - k0;      // last valid key column (causal)
      // ---- P_ij = exp2(S_ij * scale * log2e - LSE * log2e)
      if (!mbar_wait(&bar_s, j & 1, p.err)) { ok = false; break; }
      tc_fence_after();
      float pv[64];
      // key tiles before the diagonal need no mask when the query tile
      // ends inside the sequence
      const bool full = j < i && q0 + BT <= p.S;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t us[32];
        tmem_ld32(tmem_addr(tmem, qd, C_S + ch * 64 + c * 32), us);
        if (full) {
#pragma unroll
          for (int k = 0; k < 32; ++k) pv[c * 32 + k] = ex2(fmaf(__uint_as_float(us[k]), p.sl2, -lse_r));
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const int col = ch * 64 + c * 32 + k;
            pv[c * 32 + k] =
                q_ok && col <= kmax ? ex2(fmaf(__uint_as_float(us[k]), p.sl2, -lse_r)) : 0.f;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_a);
      // ---- dS_ij / scale = P_ij (dP_ij - delta), packed into this warp's
      //      own dP columns once it has read them (dQ is scaled once, in the
      //      epilogue)
      if (!mbar_wait(&bar_dp, j & 1, p.err)) { ok = false; break; }
      tc_fence_after();
      // chunk c reads columns [32c, 32c+32) and writes [16c, 16c+16): the
      // second read is of columns the first write leaves alone
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t ud[32], dk[16];
        tmem_ld32(tmem_addr(tmem, qd, C_DP + ch * 64 + c * 32), ud);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float d0 = pv[c * 32 + 2 * k] * (__uint_as_float(ud[2 * k]) - dlt_r);
          const float d1 = pv[c * 32 + 2 * k + 1] * (__uint_as_float(ud[2 * k + 1]) - dlt_r);
          dk[k] = pack_bf16(d0, d1);
        }
        tmem_st16(tmem_addr(tmem, qd, C_DP + ch * 64 + c * 16), dk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ds);
    }
    // ---- epilogue: this thread's query row, half of its 192 dQ columns
    if (ok && mbar_wait(&bar_fin, 0, p.err)) {
      tc_fence_after();
      const long long row = ((long long)b * p.S + query) * p.H + h;
      if (p.dq_out) {
        // Final bf16 dq.  The k_pe band [128,192) lies wholly in half 1; it
        // is rotated back by the row's position (the adjoint of the forward
        // rotate-half RoPE): a' = a cos + b sin, b' = b cos - a sin for the
        // pairs (128+k, 160+k).  The tile is staged in the (now idle) K ring
        // as three 128 x 64 boxes with 128-byte swizzling and written by TMA
        // after the final barrier; rows past the sequence are clipped there.
        uint8_t* stage = sm + K_OFF;
        // 32 columns starting at c0 (a multiple of 32) of this thread's row
        auto stage32 = [&](int c0, const float* v) {
          uint8_t* box = stage + (c0 >> 6) * BOX + r * 128;
          const int k0 = (c0 & 63) >> 3;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 w;
            w.x = pack_bf16(v[8 * g], v[8 * g + 1]);
            w.y = pack_bf16(v[8 * g + 2], v[8 * g + 3]);
            w.z = pack_bf16(v[8 * g + 4], v[8 * g + 5]);
            w.w = pack_bf16(v[8 * g + 6], v[8 * g + 7]);
            *reinterpret_cast<uint4*>(box + (((k0 + g) ^ (r & 7)) << 4)) = w;
          }
        };
        const float sc = p.scale;
        {
          uint32_t u[32];
          float v[32];
          tmem_ld32(tmem_addr(tmem, qd, C_DQ + ch * 96), u);
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = sc * __uint_as_float(u[k]);
          stage32(ch * 96, v);
        }
        if (ch == 0) {
#pragma unroll 1
          for (int c = 1; c < 3; ++c) {
            uint32_t u[32];
            float v[32];
            tmem_ld32(tmem_addr(tmem, qd, C_DQ + c * 32), u);
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = sc * __uint_as_float(u[k]);
            stage32(c * 32, v);
          }
        } else {
          uint32_t ua[32], ub[32];
          tmem_ld32(tmem_addr(tmem, qd, C_DQ + 128), ua);
          tmem_ld32(tmem_addr(tmem, qd, C_DQ + 160), ub);
          float ra[32], rb[32];
          const long long pos = q_ok ? query : 0;
          const float4* c4 = reinterpret_cast<const float4*>(p.cosT + pos * 32);
          const float4* s4 = reinterpret_cast<const float4*>(p.sinT + pos * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 cv = c4[k], sv = s4[k];
            const float cs[4] = {cv.x, cv.y, cv.z, cv.w}, sn[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float av = sc * __uint_as_float(ua[4 * k + e]);
              const float bv = sc * __uint_as_float(ub[4 * k + e]);
              ra[4 * k + e] = av * cs[e] + bv * sn[e];
              rb[4 * k + e] = bv * cs[e] - av * sn[e];
            }
          }
          stage32(128, ra);
          stage32(160, rb);
        }
        fence_proxy_async_smem();
        stored = true;
      } else {
        float* dst = p.dq + row * 192 + ch * 96;
#pragma unroll 1
        for (int c = 0; c < 3; ++c) {
          uint32_t u[32];
          tmem_ld32(tmem_addr(tmem, qd, C_DQ + ch * 96 + c * 32), u);
          if (q_ok) {
            float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              d4[k] = make_float4(p.scale * __uint_as_float(u[4 * k]),
                                  p.scale * __uint_as_float(u[4 * k + 1]),
                                  p.scale * __uint_as_float(u[4 * k + 2]),
                                  p.scale * __uint_as_float(u[4 * k + 3]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && stored) {
    // the staged dq tile: columns [0,64), [64,128), [128,192)
#pragma unroll
    for (int bx = 0; bx < 3; ++bx) tma_store_4d(&tm.dq, sm + K_OFF + bx * BOX, bx * 64, h, q0, b);
    bulk_commit();
    bulk_wait_read0();
  }
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_attn_bwd_dq(const Plan& p, const Ptrs& x, cudaStream_t st) {
  Views v = make_views(p, x);
  const uint64_t S = p.S, H = p.H, B = p.B;
  DqMaps tm;
  cudaError_t e;
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
  if (p.canonical) {
    uint64_t dims[4] = {192, H, S, B}, str[3] = {192 * 2, H * 192 * 2, S * H * 192 * 2};
    uint32_t box[4] = {64, 1, 128, 1};
    if ((e = make_tmap_bf16(&tm.dq, x.dq, 4, dims, str, box)) != cudaSuccess) return e;
  }
  DqParams prm;
  prm.S = p.S;
  prm.H = p.H;
  prm.B = p.B;
  prm.n_t = (p.S + BT - 1) / BT;
  prm.s_pad = (int)p.s_pad();
  prm.qn = v.qn;
  prm.qn_ld = v.qn_ld;
  prm.sl2 = p.scale * 1.4426950408889634f;
  prm.scale = p.scale;
  prm.lse2 = x.buf<float>(p, T_LSE2);
  prm.delta = x.buf<float>(p, T_DELTA);
  // canonical dims: the kernel writes the final bf16 dq itself; otherwise
  // fp32 rotated-frame rows for dq_final
  prm.dq = p.canonical ? nullptr : x.buf<float>(p, T_DQ);
  prm.dq_out = p.canonical ? static_cast<__nv_bfloat16*>(x.dq) : nullptr;
  prm.cosT = x.cos;
  prm.sinT = x.sin;
  prm.err = x.err;
  e = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)prm.n_t * p.H * p.B;
  LaunchScope ls_("attn_bwd_dq", st);
  attn_bwd_dq_kernel<<<(unsigned)grid, THREADS, SMEM_BYTES, st>>>(tm, prm);
  return cudaGetLastError();
}

}  // namespace laga
