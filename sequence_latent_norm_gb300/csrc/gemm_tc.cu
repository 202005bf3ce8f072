// a3 head-shard up-projection and its backward on the tensor cores
// (Algorithm 1 step 4; Section 5.1 k_nope[i,t] = W^k[i] L[t],
// v[i,t] = W^v[i] L[t]; Section 5.2 W_kv_b gradient shard):
//   UP   KV[t, h, :]  = L[t, :] . W[:, h*256 : h*256+256]        M=tokens N=256/head K=512
//   DL   dL[t, :]     = sum_h dKV[t, h, :] . W[:, h-cols]^T       M=tokens N=512      K=H*256
//   DW   dW[:, h-cols] = sum_t L[t, :]^T dKV[t, h, :]             M=512    N=256/head K=tokens
// Persistent pairs of CTAs (two-CTA clusters, cta_group::2), one pair per
// two SMs, each walking 256 x 256 output tiles in a fixed stride; 6 warps:
// warp 0 TMA producer (a ring of this CTA's 128 A rows and 128 B columns per
// 64-wide K step), warp 1 TMEM allocator and, in rank 0, the MMA issuer (M256
// N256 K16 pair steps into one of two 256-column fp32 accumulators in each
// CTA's TMEM), warps 2-5 epilogue (TMEM -> registers -> swizzled 32-row boxes
// in per-warp store slots -> TMA tensor stores), draining one accumulator
// while the MMAs fill the other.  DW splits the token reduction into a fixed
// number of chunks whose
// fp32 partial tiles are summed afterwards in chunk order, so every run adds
// in the same order.  Each output element is one accumulation over K in
// ascending K-step order whatever the K/V layout, which keeps the
// token-major (LAGA) and head-major (explicit) layouts bit-identical.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace laga {
namespace {
using namespace sm100;

// A pair of CTAs (a cluster of two, on two SMs) owns a 256 x 256 output
// tile at a time: CTA rank r holds rows r*128 .. r*128+127 of A and columns
// r*128 .. r*128+127 of B's N in its own shared memory, rank 0 issues the
// M = 256 pair MMAs, and each CTA's TMEM receives its own 128 x 256
// accumulator.  Per SM that is 32 KB of operand ingress per 4 MMA-equivalents
// instead of 48 KB for a lone 128 x 256 tile.  The pairs are persistent (one
// per two SMs, walking the tiles in a fixed stride) and keep two accumulators,
// so one tile's epilogue drains while the next tile's MMAs run.
constexpr int BM = 128, BN = 256, BK = 64;   // per CTA rows; per pair columns
constexpr int BN_CTA = BN / 2;
constexpr int A_BYTES = BM * BK * 2;       // 16 KB
constexpr int B_BYTES = BN_CTA * BK * 2;   // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_BOX = 32 * 128;          // one 32-row x 128-byte store box
constexpr int SMEM_BYTES = 5 * STAGE_BYTES + 4 * 4 * EPI_BOX + 1024;
// Ring stages and store slots per epilogue warp in those bytes: UP has a
// short K loop and a busy epilogue (5 stages, 4 slots); DL and DW drain an
// accumulator rarely and wait on operand loads more (6 stages, 2 slots).
template <int MODE>
struct Shape {
  static constexpr int STAGES = MODE == 0 ? 5 : 6;
  static constexpr int EPI_BUFS = MODE == 0 ? 4 : 2;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static_assert(RING_BYTES + 4 * EPI_BUFS * EPI_BOX + 1024 <= SMEM_BYTES, "shared memory");
};
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;          // two 256-column accumulators
constexpr int BOX8K = 64 * 64 * 2;

enum Mode { UP = 0, DL = 1, DW = 2 };

struct GemmMaps {
  CUtensorMap a, b;
  CUtensorMap o;      // output: UP KV, 64 x 32 bf16 boxes; DL / DW fp32, 32 x 32 boxes
};
struct GemmParams {
  int S, H, B;
  int m_rows;         // rows of the output (UP/DL: tokens per batch; DW: d_kv)
  int m_pairs, n_tiles, tiles;   // tile grid: row pairs x N tiles x z
  int k_steps;        // K steps of one tile
  int k_steps_total;  // DW: token steps over all batches
  int* err;
};

struct TileIdx {
  int mp, n, z;
};
// Tile t of a launch.  DL: the N tile runs fastest, so the two N tiles of
// one row pair run side by side and share the dKV rows they stream through
// L2; UP and DW: the row pair runs fastest (DW's two row pairs share the
// dKV slice of one head and split).
template <int MODE>
LAGA_DEVINL TileIdx tile_of(const GemmParams& p, int t) {
  TileIdx r;
  if (MODE == DL) {
    r.n = t % p.n_tiles;
    const int rest = t / p.n_tiles;
    r.mp = rest % p.m_pairs;
    r.z = rest / p.m_pairs;
  } else {
    r.mp = t % p.m_pairs;
    const int rest = t / p.m_pairs;
    r.n = rest % p.n_tiles;
    r.z = rest / p.n_tiles;
  }
  return r;
}
// K steps of a tile (DW: its split's share of the token steps)
template <int MODE>
LAGA_DEVINL int tile_k_first(const GemmParams& p, const TileIdx& t) {
  return MODE == DW ? t.z * p.k_steps : 0;
}
template <int MODE>
LAGA_DEVINL int tile_k_count(const GemmParams& p, const TileIdx& t) {
  return MODE == DW ? max(0, min(p.k_steps, p.k_steps_total - t.z * p.k_steps)) : p.k_steps;
}

// One K step of this CTA's operands: its 128 A rows and its 128 B columns.
// Completion is counted on rank 0's `full` barrier (`bar`, a cluster address).
template <int MODE>
LAGA_DEVINL void load_stage(const GemmMaps& tm, uint8_t* a_dst, uint8_t* b_dst, uint32_t bar,
                            int kstep, int m0, int n0, int n_tile, int b_idx, const GemmParams& p) {
  if (MODE == UP) {
    tma_load_3d_pair(a_dst, &tm.a, bar, kstep * BK, m0, b_idx);
#pragma unroll
    for (int i = 0; i < 2; ++i)
      tma_load_2d_pair(b_dst + i * BOX8K, &tm.b, bar, n0 + i * 64, kstep * BK);
  } else if (MODE == DL) {
    const int h = kstep >> 2, e0 = (kstep & 3) * 64;
    tma_load_4d_pair(a_dst, &tm.a, bar, e0, m0, h, b_idx);
    tma_load_2d_pair(b_dst, &tm.b, bar, kstep * BK, n0);
  } else {
    // K index = token: step -> (batch, 64-token chunk)
    const int chunks = (p.S + 63) / 64;
    const int bb = kstep / chunks, s0 = (kstep % chunks) * 64;
    tma_load_3d_pair(a_dst, &tm.a, bar, m0, s0, bb);
    tma_load_3d_pair(a_dst + BOX8K, &tm.a, bar, m0 + 64, s0, bb);
    const int c0 = n0 - n_tile * BN;   // this CTA's column half within the head
#pragma unroll
    for (int i = 0; i < 2; ++i)
      tma_load_4d_pair(b_dst + i * BOX8K, &tm.b, bar, c0 + i * 64, s0, n_tile, bb);
  }
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ GemmMaps tm, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  // full: rank 0's, counts both CTAs' bytes; empty: each CTA's, freed by the
  // pair MMAs' commit; acc_full: each CTA's, one accumulator complete;
  // acc_empty: rank 0's, one arrival per epilogue warp of either CTA
  constexpr int STAGES = Shape<MODE>::STAGES, EPI_BUFS = Shape<MODE>::EPI_BUFS;
  constexpr int RING_BYTES = Shape<MODE>::RING_BYTES;
  __shared__ uint64_t bar_full[STAGES], bar_empty[STAGES], bar_acc_full[2], bar_acc_empty[2];
  __shared__ uint32_t tmem_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // = blockIdx.x & 1
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  if (threadIdx.x == 32) {
    tma_prefetch_desc(&tm.a);
    tma_prefetch_desc(&tm.b);
    tma_prefetch_desc(&tm.o);
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_acc_full[i], 1);
      mbar_init(&bar_acc_empty[i], 8);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_sh, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers initialised before any load signals them
  tc_fence_after();
  const uint32_t tmem = tmem_sh;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = pair; t < p.tiles && ok; t += n_pairs) {
        const TileIdx ti = tile_of<MODE>(p, t);
        const int m0 = (ti.mp * 2 + (int)rank) * BM;
        const int n0 = ti.n * BN + (int)rank * BN_CTA;
        const int k_first = tile_k_first<MODE>(p, ti), k_count = tile_k_count<MODE>(p, ti);
        for (int k = 0; k < k_count; ++k, ++it) {
          const int st = it % STAGES;
          if (it >= STAGES && !mbar_wait(&bar_empty[st], ((it / STAGES) - 1) & 1, p.err)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = sm + st * STAGE_BYTES;
          if (rank == 0) mbar_arrive_expect_tx(&bar_full[st], 2 * STAGE_BYTES);
          load_stage<MODE>(tm, a_dst, a_dst + A_BYTES, smem_cluster_addr(&bar_full[st], 0),
                           k_first + k, m0, n0, ti.n, MODE == DW ? 0 : ti.z, p);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = idesc_bf16(2 * BM, BN, MODE == DW, MODE != DL);
      uint32_t it = 0;
      bool ok = true;
      int j = 0;
      for (int t = pair; t < p.tiles && ok; t += n_pairs, ++j) {
        const int buf = j & 1;
        if (j >= 2 && !mbar_wait_cluster(&bar_acc_empty[buf], ((j >> 1) - 1) & 1, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * BN);
        const int k_count = tile_k_count<MODE>(p, tile_of<MODE>(p, t));
        for (int k = 0; k < k_count; ++k, ++it) {
          const int st = it % STAGES;
          if (!mbar_wait(&bar_full[st], (it / STAGES) & 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(sm + st * STAGE_BYTES);
          const uint32_t bsm = a + A_BYTES;
          const uint32_t alo = MODE == DW ? sdesc_lo(a, BOX8K) : sdesc_lo(a, 16);
          const uint32_t blo = MODE == DL ? sdesc_lo(bsm, 16) : sdesc_lo(bsm, BOX8K);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = sdesc_make(alo + (MODE == DW ? kk * (2048 >> 4) : kk * (32 >> 4)));
            const uint64_t bd = sdesc_make(blo + (MODE == DL ? kk * (32 >> 4) : kk * (2048 >> 4)));
            mma_ss_pair(d, ad, bd, idesc, (k > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_pair(&bar_empty[st]);
        }
        mma_commit_pair(&bar_acc_full[buf]);
      }
    }
  } else {
    // epilogue warps 2..5: TMEM lane quadrant q = warp % 4 = this warp's 32
    // rows; each output box (32 rows x 128 B, 128-byte swizzled) is staged in
    // one of this warp's EPI_BUFS slots and stored by TMA from lane 0
    const int q = warp & 3;
    uint8_t* stg = sm + RING_BYTES + q * (EPI_BUFS * EPI_BOX);
    int nbox = 0;
    int j = 0;
    for (int t = pair; t < p.tiles; t += n_pairs, ++j) {
      const int buf = j & 1;
      if (!mbar_wait(&bar_acc_full[buf], (j >> 1) & 1, p.err)) break;
      tc_fence_after();
      const TileIdx ti = tile_of<MODE>(p, t);
      const int m0 = (ti.mp * 2 + (int)rank) * BM;
      const int row0 = m0 + q * 32;
      const bool have = tile_k_count<MODE>(p, ti) > 0;
      const bool rows_in = row0 < p.m_rows;   // rows past the output are clipped by TMA
      const uint32_t d = tmem + (uint32_t)(buf * BN);
      constexpr int COLS = MODE == UP ? 64 : 32;   // output columns per box
#pragma unroll 1
      for (int bx = 0; bx < BN / COLS; ++bx, ++nbox) {
        uint32_t u[COLS];
#pragma unroll
        for (int h = 0; h < COLS / 32; ++h) {
          if (have) {
            tmem_ld32(tmem_addr(d, q, bx * COLS + h * 32), *reinterpret_cast<uint32_t(*)[32]>(u + 32 * h));
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) u[32 * h + k] = 0u;
          }
        }
        uint8_t* slot = stg + (nbox % EPI_BUFS) * EPI_BOX;
        // the store that last read this slot is done
        if (lane == 0) bulk_wait_read<EPI_BUFS - 1>();
        __syncwarp();
        uint8_t* row = slot + lane * 128;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          uint4 w;
          if (MODE == UP) {
            w.x = pack_bf16(__uint_as_float(u[8 * g]), __uint_as_float(u[8 * g + 1]));
            w.y = pack_bf16(__uint_as_float(u[8 * g + 2]), __uint_as_float(u[8 * g + 3]));
            w.z = pack_bf16(__uint_as_float(u[8 * g + 4]), __uint_as_float(u[8 * g + 5]));
            w.w = pack_bf16(__uint_as_float(u[8 * g + 6]), __uint_as_float(u[8 * g + 7]));
          } else {
            w = make_uint4(u[4 * g], u[4 * g + 1], u[4 * g + 2], u[4 * g + 3]);
          }
          *reinterpret_cast<uint4*>(row + ((g ^ (lane & 7)) << 4)) = w;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (rows_in) {
            if (MODE == UP)
              tma_store_4d(&tm.o, slot, bx * 64, row0, ti.n, ti.z);
            else
              tma_store_3d(&tm.o, slot, ti.n * BN + bx * 32, row0, ti.z);
          }
          bulk_commit();
        }
      }
      // this warp's rows of the accumulator are read: rank 0 may reuse it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(smem_cluster_addr(&bar_acc_empty[buf], 0));
    }
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
  }
  // neither CTA leaves (or frees its TMEM) while the pair's MMAs may still
  // read its shared memory, write its accumulators or arrive on its barriers
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
  cluster_sync();
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
cudaError_t launch(const char* name, const GemmMaps& tm, GemmParams prm, int m_pairs, int n_tiles,
                   int z_count, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  prm.m_pairs = m_pairs;
  prm.n_tiles = n_tiles;
  prm.tiles = m_pairs * n_tiles * z_count;
  const int pairs = std::max(1, std::min(prm.tiles, sms / 2));   // one pair per two SMs
  LaunchScope ls_(name, st);
  gemm_tc_kernel<MODE><<<dim3(2 * pairs), THREADS, SMEM_BYTES, st>>>(tm, prm);
  return cudaGetLastError();
}

cudaError_t kv_map(CUtensorMap* m, const Plan& p, const Views& v, const __nv_bfloat16* base,
                   uint32_t rows) {
  uint64_t dims[4] = {256, (uint64_t)p.S, (uint64_t)p.H, (uint64_t)p.B};
  uint64_t str[3] = {(uint64_t)v.kv_ss * 2, (uint64_t)v.kv_sh * 2, (uint64_t)v.kv_sb * 2};
  uint32_t box[4] = {64, rows, 1, 1};
  return make_tmap_bf16(m, base, 4, dims, str, box);
}

// pairs of 128-row tiles covering `rows`
int row_pairs(int rows) { return (((rows + BM - 1) / BM) + 1) / 2; }

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
  if ((e = kv_map(&tm.o, p, v, v.kv, 32)) != cudaSuccess) return e;
  GemmParams prm{};
  prm.S = p.S; prm.H = p.H; prm.B = p.B;
  prm.m_rows = p.S;
  prm.k_steps = 512 / BK;
  prm.err = x.err;
  return launch<UP>("upproj", tm, prm, row_pairs(p.S), p.H, p.B, st);
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
    const int total = p.B * ((p.S + 63) / 64);
    const int splits = dw_splits(p.H, total);
    GemmParams prm{};
    prm.S = p.S; prm.H = p.H; prm.B = p.B;
    prm.m_rows = 512;
    prm.k_steps_total = total;
    prm.k_steps = (total + splits - 1) / splits;
    float* dw = p.canonical ? x.dw : x.buf<float>(p, T_DWC);
    float* out = splits > 1 ? x.buf<float>(p, T_DWP) : dw;
    const long long out_ld = (long long)p.H * 256, split_stride = 512LL * p.H * 256;
    {
      uint64_t dims[3] = {(uint64_t)out_ld, 512, (uint64_t)splits};
      uint64_t str[2] = {(uint64_t)out_ld * 4, (uint64_t)split_stride * 4};
      uint32_t box[3] = {32, 32, 1};
      if ((e = make_tmap_f32(&tm.o, out, 3, dims, str, box, true)) != cudaSuccess) return e;
    }
    prm.err = x.err;
    if ((e = launch<DW>("upproj_dw", tm, prm, row_pairs(512), p.H, splits, st)) != cudaSuccess)
      return e;
    if (splits > 1) {
      const long long n4 = split_stride / 4;
      LaunchScope ls_("dw_split_reduce", st);
      split_reduce_kernel<<<152 * 8, 256, 0, st>>>(reinterpret_cast<const float4*>(out), n4,
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
      uint32_t box[2] = {64, BN_CTA};
      if ((e = make_tmap_bf16(&tm.b, v.W, 2, dims, str, box)) != cudaSuccess) return e;
    }
    GemmParams prm{};
    prm.S = p.S; prm.H = p.H; prm.B = p.B;
    prm.m_rows = p.S;
    prm.k_steps = p.H * 4;
    float* out = x.buf<float>(p, T_DL);
    {
      uint64_t dims[3] = {512, (uint64_t)p.S, (uint64_t)p.B}, str[2] = {512 * 4, (uint64_t)p.S * 512 * 4};
      uint32_t box[3] = {32, 32, 1};
      if ((e = make_tmap_f32(&tm.o, out, 3, dims, str, box, true)) != cudaSuccess) return e;
    }
    prm.err = x.err;
    return launch<DL>("upproj_dl", tm, prm, row_pairs(p.S), 512 / BN, p.B, st);
  }
}

}  // namespace laga
