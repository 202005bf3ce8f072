// Diagnostic: the issue rate of tcgen05.mma (kind::f16, bf16 operands, fp32
// TMEM accumulator, M = 128, K = 16) on every SM, for one instruction shape
// and one interleaving of accumulators.  It measures what bounds the
// attention kernels: how many SM clocks one MMA of a given N costs when a
// single thread issues a long stream of them, either all into one
// accumulator (a dependent chain) or round-robin over several independent
// accumulators (as the kernels interleave S, dP, dV and dK).  Not part of
// the LAGA compute; the paper has no counterpart.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace laga {
namespace {
using namespace sm100;

constexpr int A_BYTES = 128 * 128;        // 128 rows x 64 bf16 (one swizzle box)
constexpr int B_BYTES = 4 * 128 * 128;    // four 128-row boxes (N up to 256, either major)
constexpr int BG_OFF = A_BYTES + B_BYTES; // shared-memory stores of the background warps
constexpr int BG_BYTES = 32 * 1024;
// more than half of an SM's shared memory, so that exactly one CTA runs per SM
constexpr int SMEM = 120 * 1024;
constexpr int A_TMEM_COL = 496;           // A operand of the TMEM form: 16 columns
constexpr int BG_TMEM_COL = 448;          // columns the background TMEM loads read
__device__ int g_diag_err;                // bounded waits of this diagnostic give up here
__device__ __align__(128) uint8_t g_diag_src[64 * 1024];   // source of the background bulk copies

// Instructions are issued in fully unrolled blocks of UNR (a multiple of
// every run * n_acc pattern used), with every operand descriptor and
// accumulator address computed before the timed loop, so that the issuing
// thread spends no time between MMAs.
constexpr int UNR = 48;

// FORM 0: A and B in shared memory; 1: A in TMEM; 2: alternating 0 and 1.
// BMN: B is MN-major (N in 64-wide boxes 16 KB apart) instead of K-major.
// BG: while the MMAs run, warps 1-7 (warp 4 shares the issuing warp's
// scheduler) 0: idle; 1: stream tcgen05.ld from
// other TMEM columns; 2: stream 16-byte shared-memory stores; 3: warp 1
// streams 16 KB bulk copies (the TMA engine) from global into shared
// memory, two in flight; 4: stream TMEM stores; 5: exponentials and FMAs
// in registers.
// Instruction k goes to accumulator (k / run) % n_acc at column acc * n.
template <int FORM, int BMN, int BG>
__global__ void __launch_bounds__(256, 1)
    diag_mma_kernel(int n, int n_acc, int run, int n_blocks, int rnd, int bg_clk, int two,
                    unsigned long long* cycles, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar, bar2, bg_bar[2];
  __shared__ uint32_t tmem_sh;
  __shared__ volatile int stop;
  __shared__ float sink[8];
  __shared__ unsigned long long bg_cycles;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // operands: small repeating values, or (rnd) values spread like N(0,1)
  // draws (a sum of four uniform hashes), whose bit patterns toggle like
  // real activations
  for (int i = threadIdx.x; i < (A_BYTES + B_BYTES) / 2; i += blockDim.x) {
    float v = 0.001f * (float)(i % 7);
    if (rnd) {
      uint32_t hsh = (uint32_t)i * 2654435761u + blockIdx.x * 40503u;
      float u = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        hsh ^= hsh >> 15; hsh *= 2246822519u; hsh ^= hsh >> 13;
        u += (float)(hsh & 0xffffu) * (1.0f / 65536.0f);
      }
      v = (u - 2.0f) * 1.7320508f;
    }
    reinterpret_cast<__nv_bfloat16*>(sm)[i] = __float2bfloat16_rn(v);
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init(&bar2, 1);
    mbar_init(&bg_bar[0], 1);
    mbar_init(&bg_bar[1], 1);
    fence_barrier_init();
    stop = 0;
    bg_cycles = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_sh, 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;
  {
    uint32_t z[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) z[k] = rnd ? 0xbf803f80u ^ (uint32_t)(k * 0x00110011u) : 0x3c003c00u;
    if (warp < 4) {
      tmem_st16(tmem_addr(tmem, warp, A_TMEM_COL), z);
      tmem_wait_st();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int issuer = threadIdx.x >> 5;   // with `two`, lane 0 of warps 0 and 1 both issue
  if (threadIdx.x == 0 || (two && threadIdx.x == 32)) {
    const uint32_t id = idesc_bf16(128, n, 0, BMN);
    const uint32_t ab = smem_u32(sm), bb = smem_u32(sm + A_BYTES);
    uint64_t ad[4], bd[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ad[k] = sdesc_sw128(ab + 32 * k, 16, 1024);
      bd[k] = BMN ? sdesc_sw128(bb + 2048 * k, 128 * 128, 1024) : sdesc_sw128(bb + 32 * k, 16, 1024);
    }
    uint32_t d[UNR];
#pragma unroll
    for (int k = 0; k < UNR; ++k)
      d[k] = tmem + (uint32_t)(((k / run) % n_acc) * n + issuer * n_acc * n);
    const uint32_t at0 = tmem + A_TMEM_COL, at1 = at0 + 8;
    const unsigned long long t0 = clock64();
    const int my_blocks = two ? n_blocks / 2 : n_blocks;
    for (int blk = 0; blk < my_blocks; ++blk) {
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        const bool ts = FORM == 1 || (FORM == 2 && (k & 1));
        if (ts)
          mma_ts(d[k], (k & 1) ? at1 : at0, bd[k & 3], id, 1u);
        else
          mma_ss(d[k], ad[k & 3], bd[k & 3], id, 1u);
      }
    }
    mma_commit(issuer == 0 ? &bar : &bar2);
    bool ok = mbar_wait(issuer == 0 ? &bar : &bar2, 0, err);
    if (two && issuer == 0) ok = mbar_wait(&bar2, 0, err) && ok;
    const unsigned long long t1 = clock64();
    if (issuer == 0) {
      if (!bg_clk) cycles[blockIdx.x] = ok ? t1 - t0 : 0ull;
      stop = 1;
    }
  } else if (BG == 3 && warp == 1) {
    // background bulk copies until the MMAs are done (bounded)
    if (lane == 0) {
      uint32_t issued[2] = {0u, 0u};
      for (uint32_t it = 0; it < (1u << 20) && !stop; ++it) {
        const int k = it & 1;
        if (issued[k] && !mbar_wait(&bg_bar[k], (issued[k] - 1) & 1, err)) break;
        mbar_arrive_expect_tx(&bg_bar[k], 16384);
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
            ::"r"(smem_u32(sm + BG_OFF + k * 16384)), "l"(g_diag_src + k * 16384), "r"(16384),
            "r"(smem_u32(&bg_bar[k]))
            : "memory");
        ++issued[k];
      }
      for (int k = 0; k < 2; ++k)
        if (issued[k]) mbar_wait(&bg_bar[k], (issued[k] - 1) & 1, err);
    }
  } else if (BG == 6 && warp > 0) {
    // background broadcast shared-memory loads (every lane reads the same
    // 16 bytes), the pattern of per-column softmax statistics
    const float4* src = reinterpret_cast<const float4*>(sm + BG_OFF + ((warp - 1) & 3) * 8192);
    float acc = 0.f;
    const unsigned long long b0 = clock64();
    uint32_t nops = 0;
    for (uint32_t it = 0; it < (1u << 22) && !stop; ++it, ++nops) {
      const float4 v = src[(it * 7u + (uint32_t)(acc > 1e30f)) & 511];
      acc += v.x + v.y + v.z + v.w;
    }
    if (lane == 0) sink[warp] = acc;
    if (bg_clk && warp == 1 && lane == 0 && nops > 0) bg_cycles = (clock64() - b0) / nops;
  } else if (BG == 5 && warp > 0) {
    // background exponentials and FMAs, the mix of a softmax, until the
    // MMAs are done
    float x[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) x[k] = 0.001f * (float)(lane + k);
    for (uint32_t it = 0; it < (1u << 22) && !stop; ++it) {
#pragma unroll
      for (int k = 0; k < 16; ++k) x[k] = ex2(fmaf(x[k], -0.75f, 0.25f));
    }
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) acc += x[k];
    if (lane == 0) sink[warp] = acc;
  } else if (BG == 4 && warp > 0) {
    // background TMEM stores (and their completion waits) until the MMAs are done
    uint32_t v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = 0x3f803f80u + (uint32_t)k;
    for (uint32_t it = 0; it < (1u << 22) && !stop; ++it) {
      v[it & 15] += 1u;
      tmem_st16(tmem_addr(tmem, warp & 3, BG_TMEM_COL + (int)(it & 1) * 16), v);
      tmem_wait_st();
    }
  } else if ((BG == 1 || BG == 2) && warp > 0) {
    // background traffic until the MMAs are done (bounded)
    float acc = 0.f;
    const unsigned long long b0 = clock64();
    uint32_t nops = 0;
    for (uint32_t it = 0; it < (1u << 22) && !stop; ++it, ++nops) {
      if (BG == 1) {
        uint32_t u[32];
        tmem_ld32(tmem_addr(tmem, warp & 3, BG_TMEM_COL), u);
        acc += __uint_as_float(u[it & 31]);
      } else {
        uint4* dst = reinterpret_cast<uint4*>(sm + BG_OFF + ((warp - 1) & 3) * 8192);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          dst[(k * 32 + lane + (int)(it & 3) * 128) & 511] = make_uint4(it, k, lane, warp);
      }
    }
    if (lane == 0) sink[warp] = acc;
    // with `bg_clk`, warp 1 reports the mean clocks of one of its operations
    if (bg_clk && warp == 1 && lane == 0 && nops > 0) bg_cycles = (clock64() - b0) / nops;
  }
  tc_fence_before();
  __syncthreads();
  if (bg_clk && threadIdx.x == 0) cycles[blockIdx.x] = bg_cycles;
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int FORM, int BMN, int BG>
cudaError_t launch_diag(int n, int n_acc, int run, int n_blocks, int rnd, int bg_clk, int two,
                        int n_cta,
                        unsigned long long* cycles, int* err, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(diag_mma_kernel<FORM, BMN, BG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  diag_mma_kernel<FORM, BMN, BG><<<n_cta, 256, SMEM, st>>>(n, n_acc, run, n_blocks, rnd, bg_clk,
                                                           two, cycles, err);
  return cudaGetLastError();
}

template <int FORM, int BMN>
cudaError_t launch_diag_bg(int bg, int n, int n_acc, int run, int n_blocks, int rnd, int bg_clk,
                           int two, int n_cta,
                           unsigned long long* cycles, int* err, cudaStream_t st) {
  if (bg == 1)
    return launch_diag<FORM, BMN, 1>(n, n_acc, run, n_blocks, rnd, bg_clk, two, n_cta, cycles, err, st);
  if (bg == 2)
    return launch_diag<FORM, BMN, 2>(n, n_acc, run, n_blocks, rnd, bg_clk, two, n_cta, cycles, err, st);
  if (bg == 3)
    return launch_diag<FORM, BMN, 3>(n, n_acc, run, n_blocks, rnd, bg_clk, two, n_cta, cycles, err, st);
  if (bg == 4)
    return launch_diag<FORM, BMN, 4>(n, n_acc, run, n_blocks, rnd, bg_clk, two, n_cta, cycles, err, st);
  if (bg == 5)
    return launch_diag<FORM, BMN, 5>(n, n_acc, run, n_blocks, rnd, bg_clk, two, n_cta, cycles, err, st);
  if (bg == 6)
    return launch_diag<FORM, BMN, 6>(n, n_acc, run, n_blocks, rnd, bg_clk, two, n_cta, cycles, err, st);
  return launch_diag<FORM, BMN, 0>(n, n_acc, run, n_blocks, rnd, bg_clk, two, n_cta, cycles, err, st);
}

template <int FORM>
cudaError_t launch_diag_form(int bmn, int bg, int n, int n_acc, int run, int n_blocks, int rnd,
                             int bg_clk, int two, int n_cta, unsigned long long* cycles,
                             int* err, cudaStream_t st) {
  return bmn ? launch_diag_bg<FORM, 1>(bg, n, n_acc, run, n_blocks, rnd, bg_clk, two, n_cta, cycles, err,
                                       st)
             : launch_diag_bg<FORM, 0>(bg, n, n_acc, run, n_blocks, rnd, bg_clk, two, n_cta, cycles, err,
                                       st);
}

}  // namespace
}  // namespace laga

extern "C" laga_status laga_diag_mma_rate(int form, int n, int n_acc, int run, int n_instr,
                                          int n_cta, unsigned long long* cycles, void* stream) {
  using namespace laga;
  const int op = form & 3, bmn = (form >> 2) & 1, bg = (form >> 3) & 7, rnd = (form >> 6) & 1;
  const int bg_clk = (form >> 7) & 1, two = (form >> 8) & 1;
  if (form < 0 || form >= 512 || (two && bg != 0) || bg > 6 || (bg_clk && bg != 1 && bg != 2 && bg != 6) || op > 2 || n < 16 || n > 256 || n % 16 != 0 ||
      n_acc < 1 || run < 1 || n_instr < 1 || n_instr > (1 << 20) || n_cta < 1 || n_cta > 4096 ||
      !cycles)
    return LAGA_ERR_ARG;
  if (bmn && n % 64 != 0) return LAGA_ERR_ARG;
  const int cols = (bg == 1 || bg == 4) ? BG_TMEM_COL : (op == 0 ? 512 : A_TMEM_COL);
  if ((two + 1) * n_acc * n > cols || n_instr % ((two + 1) * UNR) != 0 ||
      UNR % (n_acc * run) != 0)
    return LAGA_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(cycles) & 7u) != 0) return LAGA_ERR_ALIGN;
  void* err = nullptr;
  if (cudaGetSymbolAddress(&err, g_diag_err) != cudaSuccess) return LAGA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int nb = n_instr / UNR;
  int* ew = static_cast<int*>(err);
  cudaError_t e =
      op == 0   ? launch_diag_form<0>(bmn, bg, n, n_acc, run, nb, rnd, bg_clk, two, n_cta, cycles, ew, st)
      : op == 1 ? launch_diag_form<1>(bmn, bg, n, n_acc, run, nb, rnd, bg_clk, two, n_cta, cycles, ew, st)
                : launch_diag_form<2>(bmn, bg, n, n_acc, run, nb, rnd, bg_clk, two, n_cta, cycles, ew, st);
  return e == cudaSuccess ? LAGA_OK : LAGA_ERR_CUDA;
}
