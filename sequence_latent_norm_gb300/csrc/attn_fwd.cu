// a4 causal MLA attention forward on the 5th-generation tensor cores
// (Algorithm 1 step 5: scores = (q_nope||q_rope)(k_nope||k_pe)^T / sqrt(d),
// out = softmax(scores) v; Section 5.3: k_pe shared by all heads).
//
// One CTA per (128-row query tile, head, batch), 12 warps:
//   warps 0-7  softmax: warp w owns query rows 32*(w%4) .. +32 (TMEM lanes)
//              and key-column half w/4 of every score tile.  A thread reads
//              its 64 scores of S_j from TMEM, applies the causal mask on
//              the diagonal tile, takes the row max together with the
//              partner warp that holds the other half of the row (through
//              shared memory and an mbarrier), keeps the running max m
//              (base-2 domain) and its half of the sum l, writes
//              P_j = exp2(s*scale*log2e - m) as bf16 back into its own
//              TMEM columns, and rescales its half of the O accumulator only
//              when the row max grows by more than 2^8 (exact either way: O
//              and l carry the same stale max).
//   warp 8     TMA producer of Q once (q_nope | RoPE'd q_rope, 3 boxes) and
//              per key tile K_j (k_nope | k_pe, 3 boxes) into a two-stage
//              ring; warp 10 the same for V_j (2 boxes).
//   warp 9     TMEM allocator and issuer of the score MMAs: S_j = Q K_j^T
//              (12 K-steps) into S buffer j%3, once P_{j-3} V_{j-3} has
//              consumed that buffer, so the tensor core works on the next
//              tile while the softmax warps handle this one.
//   warp 11    issuer of O += P_j V_j (8 K-steps, P from TMEM) once the
//              softmax warps have written P_j.  One thread can issue a
//              tcgen05.mma only every ~50 clocks, close to the 64 clocks an
//              N=128 MMA takes, and every barrier wait on the issuing
//              thread would leave the tensor core idle; two issuers keep
//              it fed while each waits on its own barriers.
// Epilogue: the rows of O, divided by l, are staged as bf16 in the idle Q tile (two 128 x 64
// swizzled boxes) and written by TMA stores after the final barrier.
// TMEM columns: S/P triple buffer [0,384) (P of key columns 0-63 packed into
// the first 32 columns of a buffer, of 64-127 into columns 64-95), O
// [384,512).  With three buffers, S_{j+2} can be issued while P_j V_j is
// still pending, so the score MMAs of later tiles run during softmax j.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace laga {
namespace {
using namespace sm100;

constexpr int BM = 128;                 // query rows per tile
constexpr int BN = 128;                 // keys per tile
constexpr int BOX = 128 * 64 * 2;       // one [128 rows x 64 bf16] box = 16 KB
constexpr int Q_BYTES = 3 * BOX;
constexpr int K_BYTES = 3 * BOX;
constexpr int V_BYTES = 2 * BOX;
constexpr int SMEM_BYTES = Q_BYTES + 2 * (K_BYTES + V_BYTES) + 1024;
constexpr int THREADS = 384;
constexpr int N_SOFTMAX = 8;
constexpr int W_PROD = 8, W_MMA = 9, W_VPROD = 10, W_PV = 11;
constexpr uint32_t TMEM_COLS = 512;
constexpr int NSB = 3;                  // S/P buffers in TMEM
constexpr int O_COL = NSB * BN;         // 384
constexpr float RESCALE_LOG2 = 8.0f;
constexpr float LN2 = 0.6931471805599453f;

struct FwdMaps {
  CUtensorMap qn, qr, kv, kpe;
  CUtensorMap o;            // O [B, S, H, 128] bf16, 64 x 128 boxes
};
struct FwdParams {
  int S, H, B, n_qt;
  float sl2;              // softmax scale * log2(e)
  __nv_bfloat16* O;       // [B,S,H,128]
  float* lse;             // [B,H,S]
  int* err;
};

__global__ void __launch_bounds__(THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ FwdMaps tm, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* Qs = sm;
  uint8_t* Ks = sm + Q_BYTES;
  uint8_t* Vs = Ks + 2 * K_BYTES;
  // Per S buffer b = j % 3 (phase parity (j / 3) & 1): bar_s[b], S_j in
  // TMEM (so K stage j % 2 has been read); bar_p[b], P_j written; bar_ve[b],
  // P_j V_j done (so S buffer b and V stage j % 2 are free, and O holds
  // every product up to tile j).  Per K/V ring stage j % 2: bar_kf, bar_vf.
  __shared__ uint64_t bar_q, bar_kf[2], bar_vf[2], bar_ve[NSB], bar_s[NSB], bar_p[NSB];
  // row-max exchange between the two warps of a query-row quadrant, per S
  // buffer; the final row-sum exchange
  __shared__ uint64_t bar_mx[4][NSB], bar_lx[4];
  __shared__ float red_mx[NSB][2][BM], red_l[2][BM];
  __shared__ uint32_t tmem_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = p.H * p.B;
  const int qt = p.n_qt - 1 - (int)(blockIdx.x / per);   // longest query tiles first
  const int h = (int)(blockIdx.x % per) % p.H;
  const int b = (int)(blockIdx.x % per) / p.H;
  const int q0 = qt * BM;
  const int n_kt = qt + 1;

  if (threadIdx.x == 0) {
    mbar_init(&bar_q, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_kf[i], 1);
      mbar_init(&bar_vf[i], 1);
    }
    for (int i = 0; i < NSB; ++i) {
      mbar_init(&bar_ve[i], 1);
      mbar_init(&bar_s[i], 1);
      mbar_init(&bar_p[i], N_SOFTMAX);
    }
    for (int q = 0; q < 4; ++q) {
      for (int i = 0; i < NSB; ++i) mbar_init(&bar_mx[q][i], 2);
      mbar_init(&bar_lx[q], 2);
    }
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
  bool stored = false;   // this thread staged its half row of the O tile

  if (warp == W_PROD) {
    // Q, then K_j into its ring stage as soon as S_{j-2} has read it
    if (lane == 0) {
      tma_prefetch_desc(&tm.qn);
      tma_prefetch_desc(&tm.kv);
      mbar_arrive_expect_tx(&bar_q, Q_BYTES);
      tma_load_4d(Qs, &tm.qn, &bar_q, 0, h, q0, b);
      tma_load_4d(Qs + BOX, &tm.qn, &bar_q, 64, h, q0, b);
      tma_load_4d(Qs + 2 * BOX, &tm.qr, &bar_q, 0, h, q0, b);
      for (int j = 0; j < n_kt; ++j) {
        const int st = j & 1;
        const int k0 = j * BN;
        // stage st is free once S_{j-2} is done
        if (j >= 2 && !mbar_wait(&bar_s[(j - 2) % NSB], ((j - 2) / NSB) & 1, p.err)) break;
        uint8_t* kd = Ks + st * K_BYTES;
        mbar_arrive_expect_tx(&bar_kf[st], K_BYTES);
        tma_load_4d(kd, &tm.kv, &bar_kf[st], 0, k0, h, b);
        tma_load_4d(kd + BOX, &tm.kv, &bar_kf[st], 64, k0, h, b);
        tma_load_3d(kd + 2 * BOX, &tm.kpe, &bar_kf[st], 0, k0, b);
      }
    }
  } else if (warp == W_VPROD) {
    // V_j into its ring stage as soon as P_{j-2} V_{j-2} has read it (its
    // own warp, so a late V stage never holds back the next K load)
    if (lane == 0) {
      for (int j = 0; j < n_kt; ++j) {
        const int st = j & 1;
        // stage st is free once P_{j-2} V_{j-2} is done
        if (j >= 2 && !mbar_wait(&bar_ve[(j - 2) % NSB], ((j - 2) / NSB) & 1, p.err)) break;
        uint8_t* vd = Vs + st * V_BYTES;
        mbar_arrive_expect_tx(&bar_vf[st], V_BYTES);
        tma_load_4d(vd, &tm.kv, &bar_vf[st], 128, j * BN, h, b);
        tma_load_4d(vd + BOX, &tm.kv, &bar_vf[st], 192, j * BN, h, b);
      }
    }
  } else if (warp == W_MMA) {
    // score MMAs: S_j into buffer j%3 once K_j has landed and P_{j-3} V_{j-3}
    // (issued by warp W_PV) has read the buffer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16(BM, BN, 0, 0);
      const uint32_t qlo = sdesc_lo(smem_u32(Qs), 16);
      bool ok = mbar_wait(&bar_q, 0, p.err);
      for (int j = 0; ok && j < n_kt; ++j) {
        const int sb = j % NSB, st = j & 1;
        if (j >= NSB && !mbar_wait(&bar_ve[sb], ((j - NSB) / NSB) & 1, p.err)) break;
        if (!mbar_wait(&bar_kf[st], (j >> 1) & 1, p.err)) break;
        tc_fence_after();
        const uint32_t klo = sdesc_lo(smem_u32(Ks + st * K_BYTES), 16);
        const uint32_t d = tmem + sb * BN;
#pragma unroll
        for (int s = 0; s < 12; ++s) {
          const uint32_t off = ((s >> 2) * BOX + (s & 3) * 32) >> 4;
          mma_ss(d, sdesc_make(qlo + off), sdesc_make(klo + off), idS, s > 0);
        }
        mma_commit(&bar_s[sb]);
      }
    }
  } else if (warp == W_PV) {
    // O += P_j V_j once the softmax warps have written P_j and V_j has landed
    if (lane == 0) {
      const uint32_t idO = idesc_bf16(BM, 128, 0, 1);
      for (int j = 0; j < n_kt; ++j) {
        const int sb = j % NSB, st = j & 1;
        if (!mbar_wait(&bar_p[sb], (j / NSB) & 1, p.err)) break;
        if (!mbar_wait(&bar_vf[st], (j >> 1) & 1, p.err)) break;
        tc_fence_after();
        const uint32_t vlo = sdesc_lo(smem_u32(Vs + st * V_BYTES), BOX);
        const uint32_t pa = tmem + sb * BN;
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ts(tmem + O_COL, pa + (s < 4 ? 8 * s : 64 + 8 * (s - 4)),
                 sdesc_make(vlo + s * (2048 >> 4)), idO, (j > 0 || s > 0) ? 1u : 0u);
        mma_commit(&bar_ve[sb]);
      }
    }
  } else {
    // ---------------------------------------------------------- softmax warps
    const int qd = warp & 3;            // TMEM lane quadrant = query rows
    const int ch = warp >> 2;           // key-column half
    const int r = qd * 32 + lane;
    const int qi = q0 + r;
    float m = -INFINITY, l = 0.f;       // l: this half's part of the row sum
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      const int st = j % NSB;   // S buffer
      if (!mbar_wait(&bar_s[st], (j / NSB) & 1, p.err)) { ok = false; break; }
      tc_fence_after();
      float s[64];
      {
        uint32_t u[64];
        tmem_ld64(tmem_addr(tmem, qd, st * BN + ch * 64), u);
#pragma unroll
        for (int k = 0; k < 64; ++k) s[k] = __uint_as_float(u[k]);
      }
      if (j == n_kt - 1) {  // diagonal tile: key k0+c visible iff c <= r and k0+c < S
        const int lim = min(r, p.S - 1 - j * BN) - ch * 64;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c > lim) s[c] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) mx = fmaxf(mx, s[c]);
      // row max over both halves
      red_mx[st][ch][r] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_mx[qd][st]);
      if (!mbar_wait(&bar_mx[qd][st], (j / NSB) & 1, p.err)) { ok = false; break; }
      mx = fmaxf(mx, red_mx[st][ch ^ 1][r]) * p.sl2;
      const float m_new = (mx > m + RESCALE_LOG2) ? mx : m;
      const float alpha = ex2(m - m_new);
      const bool need = j > 0 && m_new != m;
      if (__any_sync(0xffffffffu, need)) {
        // O must hold P_{j-1} V_{j-1} before it is rescaled in place.
        if (!mbar_wait(&bar_ve[(j - 1) % NSB], ((j - 1) / NSB) & 1, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = O_COL + ch * 64 + c * 32;
          uint32_t u[32];
          tmem_ld32(tmem_addr(tmem, qd, col), u);
          uint32_t lo[16], hi[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            lo[k] = __float_as_uint(__uint_as_float(u[k]) * alpha);
            hi[k] = __float_as_uint(__uint_as_float(u[16 + k]) * alpha);
          }
          tmem_st16(tmem_addr(tmem, qd, col), lo);
          tmem_st16(tmem_addr(tmem, qd, col + 16), hi);
        }
      }
      m = m_new;
      float rs = 0.f;
      const float negm = -m;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float a = ex2(fmaf(s[c * 32 + 2 * k], p.sl2, negm));
          const float bb = ex2(fmaf(s[c * 32 + 2 * k + 1], p.sl2, negm));
          rs += a + bb;
          pk[k] = pack_bf16(a, bb);
        }
        // P of this half packed into the first 32 of its own 64 S columns
        tmem_st16(tmem_addr(tmem, qd, st * BN + ch * 64 + c * 16), pk);
      }
      l = l * alpha + rs;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p[st]);
    }
    // ---------------------------------------------------------- epilogue
    // O is complete once P V of the last tile is done (each stage barrier
    // is waited for its own latest phase, so the parity test is exact)
    // (the PV warp's last commit covers every earlier product too)
    if (ok) ok = mbar_wait(&bar_ve[(n_kt - 1) % NSB], ((n_kt - 1) / NSB) & 1, p.err);
    if (ok) {
      red_l[ch][r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_lx[qd]);
      ok = mbar_wait(&bar_lx[qd], 0, p.err);
    }
    if (ok) {
      tc_fence_after();
      const float lt = l + red_l[ch ^ 1][r];
      const float inv = 1.0f / lt;
      // O rows staged in the (now idle) Q tile as two 128 x 64 swizzled
      // boxes and written by TMA after the final barrier; rows past the
      // sequence are clipped there
      uint8_t* box = Qs + ch * BOX + r * 128;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem_addr(tmem, qd, O_COL + ch * 64 + c * 32), u);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(u[8 * g]) * inv, __uint_as_float(u[8 * g + 1]) * inv);
          w.y = pack_bf16(__uint_as_float(u[8 * g + 2]) * inv, __uint_as_float(u[8 * g + 3]) * inv);
          w.z = pack_bf16(__uint_as_float(u[8 * g + 4]) * inv, __uint_as_float(u[8 * g + 5]) * inv);
          w.w = pack_bf16(__uint_as_float(u[8 * g + 6]) * inv, __uint_as_float(u[8 * g + 7]) * inv);
          *reinterpret_cast<uint4*>(box + (((c * 4 + g) ^ (r & 7)) << 4)) = w;
        }
      }
      fence_proxy_async_smem();
      stored = true;
      if (ch == 0 && qi < p.S) p.lse[((long long)b * p.H + h) * p.S + qi] = (m + log2f(lt)) * LN2;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && stored) {
    tma_store_4d(&tm.o, Qs, 0, h, q0, b);
    tma_store_4d(&tm.o, Qs + BOX, 64, h, q0, b);
    bulk_commit();
    bulk_wait_read0();
  }
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_attn_fwd(const Plan& p, const Ptrs& x, cudaStream_t st) {
  Views v = make_views(p, x);
  const uint64_t S = p.S, H = p.H, B = p.B;
  FwdMaps tm;
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
    uint64_t dims[4] = {128, H, S, B}, str[3] = {128 * 2, H * 128 * 2, S * H * 128 * 2};
    uint32_t box[4] = {64, 1, 128, 1};
    if ((e = make_tmap_bf16(&tm.o, v.O, 4, dims, str, box)) != cudaSuccess) return e;
  }
  FwdParams prm;
  prm.S = p.S;
  prm.H = p.H;
  prm.B = p.B;
  prm.n_qt = (p.S + BM - 1) / BM;
  prm.sl2 = p.scale * 1.4426950408889634f;
  prm.O = v.O;
  prm.lse = x.lse;
  prm.err = x.err;
  e = cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)prm.n_qt * p.H * p.B;
  LaunchScope ls_("attn_fwd", st);
  attn_fwd_tc_kernel<<<(unsigned)grid, THREADS, SMEM_BYTES, st>>>(tm, prm);
  return cudaGetLastError();
}

}  // namespace laga
