// a5, key-stationary half of the causal MLA attention backward: dK and dV
// (Section 5.2).  With P = exp(s - LSE), delta = rowsum(dO * O):
//   dV = P^T dO,  dP^T = V dO^T,  dS^T = P^T (dP^T - delta) * scale,
//   dK = dS^T Q   (the k_pe band of dK kept per head).
// dQ = dS K is the query-stationary kernel's (attn_bwd_dq.cu); with no dQ
// here, neither P^T nor dS^T ever leaves TMEM and nothing is reduced across
// CTAs, so every output element is one fixed-order accumulation.
//
// One CTA per (128-key tile j, head h, batch b), longest (smallest j)
// first; it walks the query tiles i = j .. last.  20 warps:
//   warps 0-15 compute.  Warp w owns TMEM lane quadrant w%4 (32 key rows)
//              and column group g = w/4: query columns [16g, 16g+16) and
//              [64+16g, 64+16g+16).  Phase A: S^T -> P^T (bf16 pairs packed
//              into the first 64 S^T columns, the TMEM operand of dV).
//              Phase B: dP^T -> dS^T / scale (packed into the first 64 dP^T
//              columns, the TMEM operand of dK; dK is scaled in the
//              epilogue).  Then it adds this tile's k_pe part of dK from
//              TMEM into registers.  Four warps per SMSP hide the latency of
//              the phases' TMEM and shared-memory loads.
//   warp 16    TMA producer: K_j, V_j once; per i: Q_i with LSE_i and
//              delta_i (double-buffered), dO_i.
//   warp 17    TMEM allocator and MMA issuer.  Per i: dP^T_i, dV, the
//              k_nope steps of S^T_{i+1} (overlapping phase B), the k_pe
//              part of dK, the k_pe steps of S^T_{i+1}, dK_nope.
//   warps 18-19 idle (they complete warpgroup 4 for the register split).
// TMEM columns: dV [0,128), dK_nope [128,256), S^T [256,384) with P^T in
// [256,320), dP^T [384,512) with dS^T in [384,448); the k_pe part of dK
// for tile i goes to [448,512), the dP^T columns phase B has read and left
// free.  Every mbarrier is waited phase by phase, so parity waits are exact.
//
// Fused form (the up-projection fused into the attention backward, the
// LAGA page's Section 4.7 and Section 8 future work): instead of loading
// k_nope_j and v_j, the CTA rebuilds them, [k_nope | v]_j = L_j W_h
// (M 128 keys, N 256, K 512), before its walk.  The producer streams L_j and
// W_h in eight 64-wide K chunks through four buffers idle until the walk
// (the Q, K_j, V_j and dO_i boxes), the issuer accumulates into TMEM
// [256,512) (the S^T and dP^T columns, unused until the walk), and the
// compute warps round the tile to
// bf16 into the K_j / V_j boxes -- the rounding the up-projection GEMM
// applies -- from which the producer also stores it to HBM for the dQ
// kernel.  The walk is unchanged.  Per CTA that is 33.5 MFLOP and 384 KB of
// L2 reads, once per key tile: 1x the up-projection in total.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace laga {
namespace {
using namespace sm100;

constexpr int BT = 128;                  // key tile = query tile
constexpr int BOX = 128 * 64 * 2;        // 16 KB
constexpr int K_OFF = 0;                 // K_j: 3 boxes (k_nope | k_pe)
constexpr int V_OFF = 3 * BOX;           // V_j: 2 boxes
constexpr int Q_OFF = 5 * BOX;           // Q_i: two buffers of 3 boxes
constexpr int DO_OFF = 11 * BOX;         // dO_i: 2 boxes
constexpr int LD_OFF = 13 * BOX;         // 2 x (LSE 512 B + delta 512 B)
constexpr int SMEM_BYTES = LD_OFF + 2048 + 1024;   // + slack to align the base
constexpr int THREADS = 640;   // 20 warps: 5 whole warpgroups for setmaxnreg
constexpr int N_COMPUTE = 16;
constexpr int W_PROD = 16, W_MMA = 17;  // warps 18-19 complete warpgroup 4
constexpr uint32_t TMEM_COLS = 512;
constexpr int C_DV = 0, C_DK = 128, C_S = 256, C_DP = 384, C_DKR = C_DP + 64;
constexpr uint32_t KV_BYTES = 5 * BOX;
constexpr uint32_t Q_BYTES = 3 * BOX + 1024;    // Q_i + LSE_i + delta_i
constexpr uint32_t DO_BYTES = 2 * BOX;
constexpr int NCH = 512 / 64;            // fused form: K chunks of the rebuild
constexpr int NST = 4;                   // fused form: chunk buffers
constexpr int WBOX = 64 * 64 * 2;        // one 64 x 64 box of W_h (MN-major)
// Buffers of the rebuild's chunks (an L box, and four W boxes of 8 KB in a
// row), in regions idle until the walk: the two Q buffers, the K_j boxes
// (the k_pe box is loaded after the rebuild) and the V_j / dO_i boxes.
LAGA_DEVINL int chunk_a(int st) {
  return st == 0 ? Q_OFF : st == 1 ? Q_OFF + 3 * BOX : st == 2 ? K_OFF + 2 * BOX : DO_OFF;
}
LAGA_DEVINL int chunk_b(int st) {
  return st == 0 ? Q_OFF + BOX : st == 1 ? Q_OFF + 4 * BOX : st == 2 ? K_OFF : V_OFF;
}

struct KvMaps {
  CUtensorMap qn, qr, kv, kpe, dO, lse, dlt;   // fused form: kv is the store map of the rebuilt K/V
  CUtensorMap lat, w;        // fused form: L rows (64 x 128 boxes), W_h (64 x 64 boxes)
  CUtensorMap dkv;           // dK_nope | dV rows, 64 x 128 bf16 boxes
  CUtensorMap dkpe;          // per-head k_pe part of dK, 32 x 128 fp32 boxes
};
struct KvParams {
  int S, H, B, n_t;
  float sl2;                 // scale * log2(e)
  float scale;
  __nv_bfloat16* dkv;        // per-head [.., 256]
  long long kv_sb, kv_ss, kv_sh;
  float* dkpe;               // [R, 64]
  int* err;
};

// Column group g of the compute warps owns query columns [16g, 16g+16)
// (piece 0) and [64+16g, 64+16g+16) (piece 1).  Both packed tiles use the
// same layout: the 8 bf16 pairs of piece p of group g land at base + 16g +
// 8p, inside columns the group's own warp read with piece 0, so the packed
// tile fills [base, base+64) and [base+64, base+128) is left free.
// TMEM column of the K-step s (16 query columns) of a packed tile:
LAGA_DEVINL uint32_t packed_col(int base, int s) {
  return s < 4 ? base + 16 * s : base + 16 * (s - 4) + 8;
}

// 64 columns of an fp32 TMEM tile (this thread's row r, lane quadrant qd),
// times f, as bf16 into one 64-column 128-byte swizzled box.
LAGA_DEVINL void stage64(uint32_t tmem, int qd, int r, int col, float f, uint8_t* box) {
  uint8_t* row = box + r * 128;
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    uint32_t u[32];
    tmem_ld32(tmem_addr(tmem, qd, col + 32 * c), u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint4 w;
      w.x = pack_bf16(f * __uint_as_float(u[8 * k]), f * __uint_as_float(u[8 * k + 1]));
      w.y = pack_bf16(f * __uint_as_float(u[8 * k + 2]), f * __uint_as_float(u[8 * k + 3]));
      w.z = pack_bf16(f * __uint_as_float(u[8 * k + 4]), f * __uint_as_float(u[8 * k + 5]));
      w.w = pack_bf16(f * __uint_as_float(u[8 * k + 6]), f * __uint_as_float(u[8 * k + 7]));
      *reinterpret_cast<uint4*>(row + (((4 * c + k) ^ (r & 7)) << 4)) = w;
    }
  }
}

template <bool FUSED>
__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_kv_kernel(const __grid_constant__ KvMaps tm, const KvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_kv, bar_q_full[2], bar_q_free[2], bar_do_full, bar_do_free;
  __shared__ uint64_t bar_s, bar_dp, bar_p, bar_ds, bar_dkr, bar_tfree, bar_fin;
  __shared__ uint64_t bar_pfull[NST], bar_pfree[NST], bar_kvacc, bar_kvready;   // fused form
  __shared__ uint32_t tmem_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bar_kv, 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bar_q_full[k], 1);
      mbar_init(&bar_q_free[k], 1);
    }
    mbar_init(&bar_do_full, 1);
    mbar_init(&bar_do_free, 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_p, N_COMPUTE);
    mbar_init(&bar_ds, N_COMPUTE);
    mbar_init(&bar_dkr, 1);
    mbar_init(&bar_tfree, N_COMPUTE);
    mbar_init(&bar_fin, 1);
    for (int k = 0; k < NST; ++k) {
      mbar_init(&bar_pfull[k], 1);
      mbar_init(&bar_pfree[k], 1);
    }
    mbar_init(&bar_kvacc, 1);
    mbar_init(&bar_kvready, N_COMPUTE);
    fence_barrier_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(&tmem_sh, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;
  bool stored = false;   // this thread staged its rows of the dK / dV tile
  const int per = p.H * p.B;
  const int j = (int)(blockIdx.x / per);   // smallest key tiles (longest walks) first
  const int h = (int)(blockIdx.x % per) % p.H;
  const int b = (int)(blockIdx.x % per) / p.H;
  const int k0 = j * BT;
  const int n_i = p.n_t - j;              // query tiles j .. n_t-1
  // 96 registers a thread at launch (20 warps).  Warpgroup 4 (producer,
  // MMA issuer, two idle warps) drops to 64, the four compute warpgroups
  // rise to 104: 128 * (4 * 104 + 64) = 61440 <= 640 * 96.
  if (warp >= W_PROD) {
  reg_shrink<64>();
  if (warp == W_PROD) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      bool ok = true;
      if (FUSED) {
        // k_nope_j and v_j are rebuilt from L_j and W_h, streamed in K
        // chunks through four idle buffers
        for (int c = 0; c < NCH; ++c) {
          const int st = c % NST;
          if (c >= NST && !mbar_wait(&bar_pfree[st], ((c / NST) - 1) & 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar_pfull[st], 3 * BOX);
          tma_load_3d(sm + chunk_a(st), &tm.lat, &bar_pfull[st], c * 64, k0, b);
#pragma unroll
          for (int n = 0; n < 4; ++n)
            tma_load_2d(sm + chunk_b(st) + n * WBOX, &tm.w, &bar_pfull[st], h * 256 + n * 64,
                        c * 64);
        }
        // the rebuild's MMAs have read every buffer before the walk's
        // operands and the k_pe band of K_j land there
        for (int st = 0; ok && st < NST; ++st)
          ok = mbar_wait(&bar_pfree[st], ((NCH / NST) - 1) & 1, p.err);
        if (ok) {
          mbar_arrive_expect_tx(&bar_kv, BOX);
          tma_load_3d(sm + K_OFF + 2 * BOX, &tm.kpe, &bar_kv, 0, k0, b);
        }
      } else {
        mbar_arrive_expect_tx(&bar_kv, KV_BYTES);
        tma_load_4d(sm + K_OFF, &tm.kv, &bar_kv, 0, k0, h, b);
        tma_load_4d(sm + K_OFF + BOX, &tm.kv, &bar_kv, 64, k0, h, b);
        tma_load_3d(sm + K_OFF + 2 * BOX, &tm.kpe, &bar_kv, 0, k0, b);
        tma_load_4d(sm + V_OFF, &tm.kv, &bar_kv, 128, k0, h, b);
        tma_load_4d(sm + V_OFF + BOX, &tm.kv, &bar_kv, 192, k0, h, b);
      }
      for (int t = 0; ok && t < n_i; ++t) {
        const int q0 = (j + t) * BT;
        const int qb = t & 1;
        // Q_i, LSE_i, delta_i into buffer i%2 once the dK MMAs of tile i-2
        // have read it (phase B of i-2 has read LSE and delta before those)
        if (t >= 2 && !mbar_wait(&bar_q_free[qb], ((t >> 1) - 1) & 1, p.err)) break;
        uint8_t* qd = sm + Q_OFF + qb * 3 * BOX;
        uint8_t* ld = sm + LD_OFF + qb * 1024;
        mbar_arrive_expect_tx(&bar_q_full[qb], Q_BYTES);
        tma_load_4d(qd, &tm.qn, &bar_q_full[qb], 0, h, q0, b);
        tma_load_4d(qd + BOX, &tm.qn, &bar_q_full[qb], 64, h, q0, b);
        tma_load_4d(qd + 2 * BOX, &tm.qr, &bar_q_full[qb], 0, h, q0, b);
        tma_load_2d(ld, &tm.lse, &bar_q_full[qb], q0, b * p.H + h);
        tma_load_2d(ld + 512, &tm.dlt, &bar_q_full[qb], q0, b * p.H + h);
        // dO_i once dV_{i-1} has read dO_{i-1}
        if (t > 0 && !mbar_wait(&bar_do_free, (t - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&bar_do_full, DO_BYTES);
        tma_load_4d(sm + DO_OFF, &tm.dO, &bar_do_full, 0, h, q0, b);
        tma_load_4d(sm + DO_OFF + BOX, &tm.dO, &bar_do_full, 64, h, q0, b);
        if (FUSED && t == 0) {
          // the rebuilt k_nope_j | v_j to HBM, where the dQ kernel reads it;
          // the boxes stay unchanged for the rest of the CTA
          if (!mbar_wait(&bar_kvready, 0, p.err)) break;
#pragma unroll
          for (int bx = 0; bx < 2; ++bx) {
            tma_store_4d(&tm.kv, sm + K_OFF + bx * BOX, bx * 64, k0, h, b);
            tma_store_4d(&tm.kv, sm + V_OFF + bx * BOX, 128 + bx * 64, k0, h, b);
          }
          bulk_commit();
        }
      }
      if (FUSED) bulk_wait0();
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idST = idesc_bf16(128, 128, 0, 0);
      const uint32_t idMN = idesc_bf16(128, 128, 0, 1);
      const uint32_t idDKr = idesc_bf16(128, 64, 0, 1);
      const uint32_t klo = sdesc_lo(smem_u32(sm + K_OFF), 16);
      const uint32_t vlo = sdesc_lo(smem_u32(sm + V_OFF), 16);
      const uint32_t glo = sdesc_lo(smem_u32(sm + DO_OFF), 16);      // dO K-major (dP^T)
      const uint32_t glo_mn = sdesc_lo(smem_u32(sm + DO_OFF), BOX);  // dO MN-major (dV)
      // S^T_i = K Q_i^T (12 K-steps over d = 192) into [256,384), in two
      // parts: the 8 k_nope steps, then the 4 k_pe steps and the commit
      auto issue_s_nope = [&](int t) -> bool {
        if (!mbar_wait(&bar_q_full[t & 1], (t >> 1) & 1, p.err)) return false;
        tc_fence_after();
        const uint32_t qlo = sdesc_lo(smem_u32(sm + Q_OFF + (t & 1) * 3 * BOX), 16);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t off = ((s >> 2) * BOX + (s & 3) * 32) >> 4;
          mma_ss(tmem + C_S, sdesc_make(klo + off), sdesc_make(qlo + off), idST, s > 0);
        }
        return true;
      };
      auto issue_s_rope = [&](int t) {
        const uint32_t qlo = sdesc_lo(smem_u32(sm + Q_OFF + (t & 1) * 3 * BOX), 16);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint32_t off = (2 * BOX + s * 32) >> 4;
          mma_ss(tmem + C_S, sdesc_make(klo + off), sdesc_make(qlo + off), idST, 1u);
        }
        mma_commit(&bar_s);
      };
      bool ok = true;
      if (FUSED) {
        // [k_nope | v]_j = L_j W_h into [256,512): 8 chunks x 4 K-steps
        const uint32_t idUP = idesc_bf16(128, 256, 0, 1);
        for (int c = 0; c < NCH; ++c) {
          const int st = c % NST;
          if (!mbar_wait(&bar_pfull[st], (c / NST) & 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t alo = sdesc_lo(smem_u32(sm + chunk_a(st)), 16);
          const uint32_t blo = sdesc_lo(smem_u32(sm + chunk_b(st)), WBOX);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem + C_S, sdesc_make(alo + kk * (32 >> 4)),
                   sdesc_make(blo + kk * (2048 >> 4)), idUP, (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar_pfree[st]);
        }
        if (ok) mma_commit(&bar_kvacc);
        // the compute warps have read the accumulator and written K_j, V_j
        ok = ok && mbar_wait(&bar_kvready, 0, p.err);
      }
      ok = ok && mbar_wait(&bar_kv, 0, p.err) && issue_s_nope(0);
      if (ok) issue_s_rope(0);
      for (int t = 0; ok && t < n_i; ++t) {
        const uint32_t qlo_mn = sdesc_lo(smem_u32(sm + Q_OFF + (t & 1) * 3 * BOX), BOX);
        const bool next = t + 1 < n_i;
        // dP^T = V dO^T (8 K-steps over d_v) into [384,512): dS^T of tile
        // i-1 there was read by the dK MMAs issued before, and the k_pe part
        // of dK of tile i-1 has been read out once tfree completes
        if (!mbar_wait(&bar_do_full, t & 1, p.err)) break;
        if (t > 0 && !mbar_wait(&bar_tfree, (t - 1) & 1, p.err)) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t off = ((s >> 2) * BOX + (s & 3) * 32) >> 4;
          mma_ss(tmem + C_DP, sdesc_make(vlo + off), sdesc_make(glo + off), idST, s > 0);
        }
        mma_commit(&bar_dp);
        // dV += P^T dO (P^T from TMEM); afterwards dO_i is no longer read
        if (!mbar_wait(&bar_p, t & 1, p.err)) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ts(tmem + C_DV, tmem + packed_col(C_S, s), sdesc_make(glo_mn + s * (2048 >> 4)),
                 idMN, (t > 0 || s > 0) ? 1u : 0u);
        mma_commit(&bar_do_free);
        // S^T_{i+1} overwrites P^T_i only after the dV MMAs above read it.
        // Its k_nope steps keep the pipe busy until dS^T_i is ready; the
        // k_pe part of dK for tile i goes ahead of its k_pe steps, so the
        // compute warps can read it out while the rest of the pipe runs
        // (issuing all of S^T_{i+1} first was measured slower).
        if (next && !issue_s_nope(t + 1)) break;
        if (!mbar_wait(&bar_ds, t & 1, p.err)) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ts(tmem + C_DKR, tmem + packed_col(C_DP, s),
                 sdesc_make(qlo_mn + ((2 * BOX + s * 2048) >> 4)), idDKr, s > 0);
        mma_commit(&bar_dkr);
        if (next) issue_s_rope(t + 1);
        // dK_nope += dS^T Q_nope
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ts(tmem + C_DK, tmem + packed_col(C_DP, s), sdesc_make(qlo_mn + s * (2048 >> 4)),
                 idMN, (t > 0 || s > 0) ? 1u : 0u);
        mma_commit(&bar_q_free[t & 1]);
      }
      mma_commit(&bar_fin);
    }
  }
  } else {
    reg_grow<104>();
    // ------------------------------------------------------------- compute warps 0..15
    const int qd = warp & 3;            // TMEM lane quadrant
    const int g = warp >> 2;            // column group (see packed_col)
    const int r = qd * 32 + lane;       // TMEM lane: key row
    const int key = k0 + r;
    const bool key_ok = key < p.S;
    float acc[16];                      // this thread's 16 columns of the k_pe part of dK
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;
    bool live = true;
    if (FUSED) {
      // the rebuilt k_nope_j (groups 0-1) or v_j (groups 2-3) rows, 64
      // columns a group, rounded to bf16 into the K_j / V_j boxes
      live = mbar_wait(&bar_kvacc, 0, p.err);
      if (live) {
        tc_fence_after();
        stage64(tmem, qd, r, C_S + 64 * g, 1.f,
                sm + (g < 2 ? K_OFF + g * BOX : V_OFF + (g - 2) * BOX));
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_kvready);
      }
    }
    for (int t = 0; live && t < n_i; ++t) {
      const int i = j + t, q0 = i * BT;
      const float* lse_s = reinterpret_cast<const float*>(sm + LD_OFF + (t & 1) * 1024);
      const float* dlt_s = lse_s + 128;
      const int qlo = key - q0;         // first valid query column (causal)
      const int qhi = p.S - q0;         // columns >= qhi are past the sequence
      // ---- phase A: P^T = exp2(S^T * scale * log2e - LSE * log2e)
      if (!mbar_wait(&bar_q_full[t & 1], (t >> 1) & 1, p.err)) break;   // LSE_i, delta_i
      if (!mbar_wait(&bar_s, t & 1, p.err)) break;
      tc_fence_after();
      float pv[32];
      // query tiles after the diagonal that end inside the sequence need no mask
      const bool full = t > 0 && q0 + BT <= p.S && k0 + BT <= p.S;
      // both pieces' scores in one TMEM round trip
      uint32_t usa[32];
      tmem_ld16x2(tmem_addr(tmem, qd, C_S + 16 * g), tmem_addr(tmem, qd, C_S + 64 + 16 * g), usa);
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        const int col0 = 64 * pc + 16 * g;
        const uint32_t* us = usa + 16 * pc;
        if (full) {
          // the piece's LSE values first: shared-memory loads wait behind
          // the tensor core's operand reads, so none may sit between the
          // exponentials
          const float4* l4 = reinterpret_cast<const float4*>(lse_s + col0);
          float4 lz[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) lz[k] = l4[k];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float* o = pv + 16 * pc + 4 * k;
            o[0] = ex2(fmaf(__uint_as_float(us[4 * k]), p.sl2, -lz[k].x));
            o[1] = ex2(fmaf(__uint_as_float(us[4 * k + 1]), p.sl2, -lz[k].y));
            o[2] = ex2(fmaf(__uint_as_float(us[4 * k + 2]), p.sl2, -lz[k].z));
            o[3] = ex2(fmaf(__uint_as_float(us[4 * k + 3]), p.sl2, -lz[k].w));
          }
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int col = col0 + k;
            const bool ok = key_ok && col >= qlo && col < qhi;
            pv[16 * pc + k] = ok ? ex2(fmaf(__uint_as_float(us[k]), p.sl2, -lse_s[col])) : 0.f;
          }
        }
        uint32_t pk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) pk[k] = pack_bf16(pv[16 * pc + 2 * k], pv[16 * pc + 2 * k + 1]);
        tmem_st8(tmem_addr(tmem, qd, C_S + 16 * g + 8 * pc), pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p);
      // ---- phase B: dS^T / scale = P^T (dP^T - delta), packed like P^T
      //      into the first 64 dP^T columns (dK is scaled in the epilogue)
      if (!mbar_wait(&bar_dp, t & 1, p.err)) break;
      tc_fence_after();
      uint32_t uda[32];
      tmem_ld16x2(tmem_addr(tmem, qd, C_DP + 16 * g), tmem_addr(tmem, qd, C_DP + 64 + 16 * g), uda);
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        const int col0 = 64 * pc + 16 * g;
        // the piece's delta values first (see phase A)
        const float4* d4 = reinterpret_cast<const float4*>(dlt_s + col0);
        float4 dz[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) dz[k] = d4[k];
        uint32_t dk[8];
        const uint32_t* ud = uda + 16 * pc;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 dl = dz[k];
          const float* u = reinterpret_cast<const float*>(ud) + 4 * k;
          const float* pk = pv + 16 * pc + 4 * k;
          dk[2 * k] = pack_bf16(pk[0] * (u[0] - dl.x), pk[1] * (u[1] - dl.y));
          dk[2 * k + 1] = pack_bf16(pk[2] * (u[2] - dl.z), pk[3] * (u[3] - dl.w));
        }
        tmem_st8(tmem_addr(tmem, qd, C_DP + 16 * g + 8 * pc), dk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ds);
      // ---- the k_pe part of dK for this query tile, out of [448,512)
      if (!mbar_wait(&bar_dkr, t & 1, p.err)) break;
      tc_fence_after();
      {
        uint32_t u[16];
        tmem_ld16(tmem_addr(tmem, qd, C_DKR + 16 * g), u);
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] += __uint_as_float(u[k]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_tfree);
    }
    // ---- epilogue: dK_nope (groups 0-1, scaled) or dV (groups 2-3) rows as
    //      bf16, 64 columns a group, and the k_pe part of dK, scaled, as
    //      fp32; staged in the idle Q buffers as 128-byte swizzled boxes
    //      (four 64-column bf16 boxes, two 32-column fp32 boxes) and written
    //      by TMA after the final barrier; rows past the sequence are
    //      clipped there
    if (mbar_wait(&bar_fin, 0, p.err)) {
      tc_fence_after();
      stage64(tmem, qd, r, g < 2 ? C_DK + 64 * g : C_DV + 64 * (g - 2), g < 2 ? p.scale : 1.f,
              sm + Q_OFF + g * BOX);
      uint8_t* box = sm + Q_OFF + (4 + (g >> 1)) * BOX + r * 128;
      const float sc = p.scale;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        *reinterpret_cast<float4*>(box + ((((g & 1) * 4 + k) ^ (r & 7)) << 4)) =
            make_float4(sc * acc[4 * k], sc * acc[4 * k + 1], sc * acc[4 * k + 2],
                        sc * acc[4 * k + 3]);
      fence_proxy_async_smem();
      stored = true;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && stored) {
#pragma unroll
    for (int bx = 0; bx < 4; ++bx) tma_store_4d(&tm.dkv, sm + Q_OFF + bx * BOX, bx * 64, k0, h, b);
#pragma unroll
    for (int cx = 0; cx < 2; ++cx)
      tma_store_4d(&tm.dkpe, sm + Q_OFF + (4 + cx) * BOX, cx * 32, h, k0, b);
    bulk_commit();
    bulk_wait_read0();
  }
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_attn_bwd_kv(const Plan& p, const Ptrs& x, cudaStream_t st) {
  Views v = make_views(p, x);
  const uint64_t S = p.S, H = p.H, B = p.B;
  KvMaps tm;
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
    uint64_t dims[4] = {256, S, H, B};
    uint64_t str[3] = {(uint64_t)v.kv_ss * 2, (uint64_t)v.kv_sh * 2, (uint64_t)v.kv_sb * 2};
    uint32_t box[4] = {64, 128, 1, 1};
    if ((e = make_tmap_bf16(&tm.dkv, x.buf<__nv_bfloat16>(p, T_DKV), 4, dims, str, box)) != cudaSuccess)
      return e;
  }
  {
    uint64_t dims[4] = {64, H, S, B}, str[3] = {64 * 4, H * 64 * 4, S * H * 64 * 4};
    uint32_t box[4] = {32, 1, 128, 1};
    if ((e = make_tmap_f32(&tm.dkpe, x.buf<float>(p, T_DKPE), 4, dims, str, box, true)) != cudaSuccess)
      return e;
  }
  if (p.fused) {
    {
      uint64_t dims[3] = {512, S, B}, str[2] = {1024, S * 1024};
      uint32_t box[3] = {64, 128, 1};
      if ((e = make_tmap_bf16(&tm.lat, v.L, 3, dims, str, box)) != cudaSuccess) return e;
    }
    {
      uint64_t dims[2] = {H * 256, 512}, str[1] = {(uint64_t)v.w_ld * 2};
      uint32_t box[2] = {64, 64};
      if ((e = make_tmap_bf16(&tm.w, v.W, 2, dims, str, box)) != cudaSuccess) return e;
    }
  } else {
    tm.lat = tm.kv;   // unused
    tm.w = tm.kv;
  }
  KvParams prm;
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
  prm.err = x.err;
  auto* kernel = p.fused ? attn_bwd_kv_kernel<true> : attn_bwd_kv_kernel<false>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)prm.n_t * p.H * p.B;
  LaunchScope ls_(p.fused ? "attn_bwd_dkdv_fused" : "attn_bwd_dkdv", st);
  kernel<<<(unsigned)grid, THREADS, SMEM_BYTES, st>>>(tm, prm);
  return cudaGetLastError();
}

}  // namespace laga
