// a5 causal MLA attention backward on the 5th-generation tensor cores
// (Section 5.2).  With P = exp(s - LSE), delta = rowsum(dO * O):
//   dV = P^T dO,  dP = dO V^T,  dS = P (dP - delta) * scale,
//   dQ = dS K,    dK = dS^T Q   (the k_pe band of dK kept per head).
//
// One CTA per (128-key tile j, head h, batch b), taken from a global work
// counter in order of increasing j (longest first); it walks the query
// tiles i = last .. j.  11 warps:
//   warps 0-7  compute.  Warp w owns TMEM lane quadrant w%4 (key rows for
//              S^T, dP^T, dK; query rows for dQ) and column half w/4.
//              Phase A: S^T -> P^T (bf16 into TMEM for the TMEM-operand
//              MMA of dV).  Phase B: dP^T -> dS^T * scale (bf16 into shared
//              memory, 128-byte swizzled).  Phase C: copy dQ_i and this
//              tile's k_pe part of dK out of TMEM into registers, free the
//              columns, and write dQ_i as three 64-column fp32 chunks into
//              128-byte-swizzled staging tiles: the staging buffer (chunks 0
//              and 2) and the dS^T tile (chunk 1; dead between the dQ MMA and
//              the next phase B).
//   warp 10    dQ reducer: adds the staged chunks into the fp32 dQ
//              accumulator in global memory with TMA tensor reduce-adds (a
//              store for key tile 0), in a fixed order -- key tile 0, 1, 2,
//              ... through a per-(b,h,i) semaphore -- so every run sums
//              identically, and hands the staging tiles back.
//   warp 8     TMA producer: K_j, V_j once; per i: Q_i, dO_i, LSE_i, delta_i.
//   warp 9     TMEM allocator and MMA issuer.
// TMEM columns: dV [0,128), dK_nope [128,256), S^T [256,384) with P^T in
// [256,288) and [320,352), dP^T [384,512); after the softmax phases the
// k_pe part of dK for this i goes to [256,320) and dQ_i to [320,512).
// Every mbarrier is waited phase by phase, so parity waits are exact.
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
constexpr int DS_OFF = 8 * BOX;          // dS^T: 2 boxes
constexpr int DO_OFF = 10 * BOX;         // dO_i: 2 boxes
constexpr int ST_OFF = 12 * BOX;         // dQ staging: 2 boxes of [128 rows x 32 fp32]
                                         // (the dS^T tile is the second staging buffer)
constexpr int LD_OFF = 14 * BOX;         // LSE 512 B + delta 512 B
constexpr int BAR_OFF = LD_OFF + 1024;   // mbarriers, TMEM address, work item
constexpr int SMEM_BYTES = BAR_OFF + 256;  // 230656 B: within the 227 KiB per block
constexpr int THREADS = 352;
constexpr int N_COMPUTE = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr int C_DV = 0, C_DK = 128, C_S = 256, C_DP = 384, C_DKR = 256, C_DQ = 320;
constexpr uint32_t KV_BYTES = 5 * BOX;
constexpr uint32_t Q_BYTES = 3 * BOX;
constexpr uint32_t DO_BYTES = 2 * BOX + 1024;   // dO_i + LSE_i + delta_i
constexpr uint32_t kSemPolls = 1u << 24;

struct BwdMaps {
  CUtensorMap qn, qr, kv, kpe, dO, lse, dlt, dq;
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

// Publish a key tile's TMA reduce-adds into one dQ tile: once they are
// performed (the caller waits for their bulk groups), order them before the
// release and hand the turn to key tile j + 1 (`next`).
LAGA_DEVINL void release_dq(int* sem, int next) {
  fence_proxy_async_global();
  __threadfence();
  st_release_gpu(sem, next);
}

// TMEM column of the P^T K-step s (16 query columns): the first 64 query
// columns are packed at [256,288), the last 64 at [320,352).
LAGA_DEVINL uint32_t pt_col(int s) { return s < 4 ? C_S + 8 * s : C_S + 64 + 8 * (s - 4); }

__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_tc_kernel(const __grid_constant__ BwdMaps tm, const BwdParams p) {
  // The whole budget is used, so there is no room to align the dynamic
  // region by hand: it must start on a 1024-byte boundary (it does when the
  // kernel has no static shared memory).  Otherwise record the error and
  // leave before touching shared memory.
  extern __shared__ __align__(1024) uint8_t sm[];
  if (smem_u32(sm) & 1023u) {
    if (threadIdx.x == 0) atomicExch(p.err, 4);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + BAR_OFF);
  uint64_t& bar_kv = bars[0];
  uint64_t& bar_q_full = bars[1];
  uint64_t& bar_q_free = bars[2];
  uint64_t& bar_do_full = bars[3];
  uint64_t& bar_do_free = bars[4];
  uint64_t& bar_s = bars[7];
  uint64_t& bar_dp = bars[8];
  uint64_t& bar_p = bars[9];
  uint64_t& bar_ds = bars[10];
  uint64_t& bar_dq = bars[11];
  uint64_t& bar_tfree = bars[12];
  uint64_t& bar_fin = bars[13];
  // staged dQ chunk m is ready (8 arrivals).  One barrier per chunk: a warp
  // may arrive for chunk m+1 before another has arrived for chunk m.
  uint64_t* bar_stg_full = bars + 14;  // [3]
  uint64_t& bar_a_free = bars[17];     // the staging buffer may be rewritten
  uint64_t& bar_b_free = bars[18];     // the dS^T tile may be rewritten
  uint32_t& tmem_sh = *reinterpret_cast<uint32_t*>(sm + BAR_OFF + 192);
  int& item_sh = *reinterpret_cast<int*>(sm + BAR_OFF + 196);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    item_sh = atomicAdd(p.counter, 1);
    mbar_init(&bar_kv, 1);
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_free, 1);
    mbar_init(&bar_do_full, 1);
    mbar_init(&bar_do_free, 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_p, N_COMPUTE);
    mbar_init(&bar_ds, N_COMPUTE);
    mbar_init(&bar_dq, 1);
    mbar_init(&bar_tfree, N_COMPUTE);
    mbar_init(&bar_fin, 1);
    for (int m = 0; m < 3; ++m) mbar_init(&bar_stg_full[m], N_COMPUTE);
    mbar_init(&bar_a_free, 1);
    mbar_init(&bar_b_free, 1);
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
  // query tiles last .. j, the diagonal last: a CTA started later reaches
  // every tile after the CTAs of lower key tiles started before it, which is
  // the order the dQ adds must take
  const int n_i = p.n_t - j;

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
        const int q0 = (p.n_t - 1 - t) * BT;
        // Q_i, dO_i, LSE_i and delta_i are free once tile i-1's dK MMAs ran
        if (t > 0 && !mbar_wait(&bar_q_free, (t - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&bar_do_full, DO_BYTES);
        tma_load_4d(sm + DO_OFF, &tm.dO, &bar_do_full, 0, h, q0, b);
        tma_load_4d(sm + DO_OFF + BOX, &tm.dO, &bar_do_full, 64, h, q0, b);
        tma_load_2d(sm + LD_OFF, &tm.lse, &bar_do_full, q0, b * p.H + h);
        tma_load_2d(sm + LD_OFF + 512, &tm.dlt, &bar_do_full, q0, b * p.H + h);
        mbar_arrive_expect_tx(&bar_q_full, Q_BYTES);
        tma_load_4d(sm + Q_OFF, &tm.qn, &bar_q_full, 0, h, q0, b);
        tma_load_4d(sm + Q_OFF + BOX, &tm.qn, &bar_q_full, 64, h, q0, b);
        tma_load_4d(sm + Q_OFF + 2 * BOX, &tm.qr, &bar_q_full, 0, h, q0, b);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idST = idesc_bf16(128, 128, 0, 0);
      const uint32_t idMN = idesc_bf16(128, 128, 0, 1);
      const uint32_t idDKr = idesc_bf16(128, 64, 0, 1);
      const uint32_t idDQ = idesc_bf16(128, 192, 1, 1);
      const uint32_t kb = smem_u32(sm + K_OFF), vb = smem_u32(sm + V_OFF);
      const uint32_t qb = smem_u32(sm + Q_OFF), sb = smem_u32(sm + DS_OFF);
      bool ok = mbar_wait(&bar_kv, 0, p.err);
      const uint32_t gb = smem_u32(sm + DO_OFF);
      for (int t = 0; ok && t < n_i; ++t) {
        if (!mbar_wait(&bar_q_full, t & 1, p.err)) break;
        if (!mbar_wait(&bar_do_full, t & 1, p.err)) break;
        if (t > 0 && !mbar_wait(&bar_tfree, (t - 1) & 1, p.err)) break;
        tc_fence_after();
        // S^T = K Q^T (12 K-steps over d = 192)
#pragma unroll
        for (int s = 0; s < 12; ++s) {
          const uint32_t off = (s >> 2) * BOX + (s & 3) * 32;
          mma_ss(tmem + C_S, sdesc_sw128(kb + off, 16, 1024), sdesc_sw128(qb + off, 16, 1024),
                 idST, s > 0);
        }
        mma_commit(&bar_s);
        // dP^T = V dO^T (8 K-steps over d_v)
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t off = (s >> 2) * BOX + (s & 3) * 32;
          mma_ss(tmem + C_DP, sdesc_sw128(vb + off, 16, 1024), sdesc_sw128(gb + off, 16, 1024),
                 idST, s > 0);
        }
        mma_commit(&bar_dp);
        // dV += P^T dO (P^T from TMEM)
        if (!mbar_wait(&bar_p, t & 1, p.err)) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ts(tmem + C_DV, tmem + pt_col(s), sdesc_sw128(gb + s * 2048, BOX, 1024), idMN,
                 (t > 0 || s > 0) ? 1u : 0u);
        // dK_nope += dS^T Q_nope, dK_rope_i = dS^T Q_rope
        if (!mbar_wait(&bar_ds, t & 1, p.err)) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint64_t ad = sdesc_sw128(sb + (s >> 2) * BOX + (s & 3) * 32, 16, 1024);
          mma_ss(tmem + C_DK, ad, sdesc_sw128(qb + s * 2048, BOX, 1024), idMN,
                 (t > 0 || s > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint64_t ad = sdesc_sw128(sb + (s >> 2) * BOX + (s & 3) * 32, 16, 1024);
          mma_ss(tmem + C_DKR, ad, sdesc_sw128(qb + 2 * BOX + s * 2048, BOX, 1024), idDKr, s > 0);
        }
        mma_commit(&bar_q_free);
        // dQ_i = dS K (dS read MN-major from the dS^T tile, K MN-major)
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ss(tmem + C_DQ, sdesc_sw128(sb + s * 2048, BOX, 1024),
                 sdesc_sw128(kb + s * 2048, BOX, 1024), idDQ, s > 0);
        mma_commit(&bar_dq);
      }
      mma_commit(&bar_fin);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------- dQ reducer
    if (lane == 0) {
      for (int t = 0; t < n_i; ++t) {
        const int i = p.n_t - 1 - t, q0 = i * BT;
        int* sem = p.sem + ((long long)b * p.H + h) * p.n_t + i;
        uint32_t n = 0;
        while (ld_acquire_gpu(sem) != j) {   // key tiles add in order 0, 1, ..., i
          if (++n > kSemPolls) {
            atomicExch(p.err, DEV_ERR_TIMEOUT);
            break;
          }
          if (n > 4096) __nanosleep(64);
        }
        fence_proxy_async_global();
        bool ok = true;
        for (int m = 0; m < 3; ++m) {
          if (!(ok = mbar_wait(&bar_stg_full[m], t & 1, p.err))) break;
          const int sbase = (m == 1) ? DS_OFF : ST_OFF;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const void* src = sm + sbase + hb * BOX;
            const int c0 = 32 * (2 * m + hb);
            if (j == 0) tma_store_4d(&tm.dq, src, c0, h, q0, b);
            else tma_reduce_add_4d(&tm.dq, src, c0, h, q0, b);
          }
          bulk_commit();
          if (m == 1) {                    // chunk 0 read: staging buffer reusable
            bulk_wait_read1();
            mbar_arrive(&bar_a_free);
          }
        }
        bulk_wait_read1();                 // chunk 1 read: the dS^T tile is free
        mbar_arrive(&bar_b_free);
        bulk_wait_read0();                 // chunk 2 read: the staging buffer is free
        mbar_arrive(&bar_a_free);
        if (!ok) break;
        // pass the turn on as soon as this tile's adds are performed: the
        // next key tile's CTA is usually already waiting for it
        bulk_wait0();
        release_dq(sem, j + 1);
      }
    }
  } else {
    // ------------------------------------------------------------- compute warps 0..7
    const int qd = warp & 3;            // TMEM lane quadrant
    const int ch = warp >> 2;           // column half
    const int r = qd * 32 + lane;       // TMEM lane: key row (S^T, dP^T, dK), query row (dQ)
    const int key = k0 + r;
    uint8_t* ds_tile = sm + DS_OFF;
    float acc[32];                      // this thread's 32 columns of the k_pe part of dK
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] = 0.f;
    for (int t = 0; t < n_i; ++t) {
      const int i = p.n_t - 1 - t, q0 = i * BT;
      const float* lse_s = reinterpret_cast<const float*>(sm + LD_OFF);
      const float* dlt_s = lse_s + 128;
      const int qlo = key - q0;         // first valid query column (causal)
      const int qhi = p.S - q0;         // columns >= qhi are past the sequence
      const bool key_ok = key < p.S;
      // ---- phase A: P^T = exp2(S^T * scale * log2e - LSE * log2e)
      if (!mbar_wait(&bar_s, t & 1, p.err)) break;
      tc_fence_after();
      float pv[64];
      // query tiles after the diagonal that end inside the sequence need no mask
      const bool full = i > j && q0 + BT <= p.S && k0 + BT <= p.S;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t us[32];
        tmem_ld32(tmem_addr(tmem, qd, C_S + ch * 64 + c * 32), us);
        uint32_t pk[16];
        if (full) {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            pv[c * 32 + k] =
                ex2(fmaf(__uint_as_float(us[k]), p.sl2, -lse_s[ch * 64 + c * 32 + k]));
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const int col = ch * 64 + c * 32 + k;
            const bool ok = key_ok && col >= qlo && col < qhi;
            pv[c * 32 + k] = ok ? ex2(fmaf(__uint_as_float(us[k]), p.sl2, -lse_s[col])) : 0.f;
          }
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) pk[k] = pack_bf16(pv[c * 32 + 2 * k], pv[c * 32 + 2 * k + 1]);
        tmem_st16(tmem_addr(tmem, qd, C_S + ch * 64 + c * 16), pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p);
      // ---- phase B: dS^T = P^T (dP^T - delta) * scale -> shared memory
      // (the previous tile's dQ chunk 1 was staged in the dS^T tile)
      if (t > 0 && !mbar_wait(&bar_b_free, (t - 1) & 1, p.err)) break;
      if (!mbar_wait(&bar_dp, t & 1, p.err)) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t ud[32];
        tmem_ld32(tmem_addr(tmem, qd, C_DP + ch * 64 + c * 32), ud);
        uint32_t dk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int col = ch * 64 + c * 32 + 2 * k;
          const float d0 = pv[c * 32 + 2 * k] * (__uint_as_float(ud[2 * k]) - dlt_s[col]) * p.scale;
          const float d1 =
              pv[c * 32 + 2 * k + 1] * (__uint_as_float(ud[2 * k + 1]) - dlt_s[col + 1]) * p.scale;
          dk[k] = pack_bf16(d0, d1);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = make_uint4(dk[4 * k], dk[4 * k + 1], dk[4 * k + 2], dk[4 * k + 3]);
          *reinterpret_cast<uint4*>(ds_tile + sw_chunk_off(r, ch * 8 + c * 4 + k)) = v;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ds);
      // ---- phase C: dQ_i and the k_pe part of dK out of TMEM
      if (!mbar_wait(&bar_dq, t & 1, p.err)) break;
      tc_fence_after();
      {
        uint32_t u[32];
        tmem_ld32(tmem_addr(tmem, qd, C_DKR + ch * 32), u);
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[k] += __uint_as_float(u[k]);
      }
      // this thread holds dQ columns 32*(2m + ch) .. +32 for m = 0, 1, 2
      float dqv[96];
#pragma unroll
      for (int m = 0; m < 3; ++m) {
        uint32_t u[32];
        tmem_ld32(tmem_addr(tmem, qd, C_DQ + 32 * (2 * m + ch)), u);
#pragma unroll
        for (int k = 0; k < 32; ++k) dqv[m * 32 + k] = __uint_as_float(u[k]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_tfree);
      // ---- stage dQ_i for the reducer: chunks 0, 2 -> staging buffer,
      //      chunk 1 -> dS^T tile (free: its MMAs completed with dQ_i)
#pragma unroll
      for (int m = 0; m < 3; ++m) {
        const int sbase = (m == 1) ? DS_OFF : ST_OFF;
        if (m == 0 && t > 0 && !mbar_wait(&bar_a_free, (2 * t - 1) & 1, p.err)) break;
        if (m == 2 && !mbar_wait(&bar_a_free, (2 * t) & 1, p.err)) break;
        uint8_t* stage = sm + sbase + ch * BOX;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const float4 v = make_float4(dqv[m * 32 + 4 * cc], dqv[m * 32 + 4 * cc + 1],
                                       dqv[m * 32 + 4 * cc + 2], dqv[m * 32 + 4 * cc + 3]);
          *reinterpret_cast<float4*>(stage + r * 128 + ((cc ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_stg_full[m]);
      }
    }
    // ---- epilogue: dK_nope (half 0) or dV (half 1) rows, k_pe part of dK
    if (mbar_wait(&bar_fin, 0, p.err)) {
      tc_fence_after();
      __nv_bfloat16* dst = p.dkv + b * p.kv_sb + (long long)key * p.kv_ss + h * p.kv_sh + ch * 128;
      const int src = ch == 0 ? C_DK : C_DV;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem_addr(tmem, qd, src + c * 32), u);
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
      if (key < p.S) {
        float4* d4 = reinterpret_cast<float4*>(p.dkpe + (((long long)b * p.S + key) * p.H + h) * DR +
                                               ch * 32);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          d4[k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
      }
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
  {
    // fp32 dQ accumulator [B,S,H,192]; 32-float boxes, 128-byte swizzled
    uint64_t dims[4] = {192, H, S, B}, str[3] = {192 * 4, H * 192 * 4, S * H * 192 * 4};
    uint32_t box[4] = {32, 1, 128, 1};
    if ((e = make_tmap_f32(&tm.dq, x.buf<float>(p, T_DQ), 4, dims, str, box, true)) != cudaSuccess)
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
