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
constexpr int B_BYTES = 256 * 128;        // up to 256 rows x 64 bf16
// more than half of an SM's shared memory, so that exactly one CTA runs per SM
constexpr int SMEM = 120 * 1024;
constexpr int A_TMEM_COL = 496;           // A operand of the TMEM form: 16 columns
__device__ int g_diag_err;                // bounded waits of this diagnostic give up here

// Instructions are issued in fully unrolled blocks of UNR (a multiple of
// every run * n_acc pattern used), with every operand descriptor and
// accumulator address computed before the timed loop, so that the issuing
// thread spends no time between MMAs.
constexpr int UNR = 48;

// FORM 0: A and B in shared memory; 1: A in TMEM; 2: alternating 0 and 1.
// Instruction k goes to accumulator (k / run) % n_acc at column acc * n.
template <int FORM>
__global__ void __launch_bounds__(128, 1)
    diag_mma_kernel(int n, int n_acc, int run, int n_blocks, unsigned long long* cycles,
                    int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_sh;
  const int warp = threadIdx.x >> 5;
  // operands: small finite bf16 values (the rate does not depend on them)
  for (int i = threadIdx.x; i < (A_BYTES + B_BYTES) / 2; i += blockDim.x)
    reinterpret_cast<__nv_bfloat16*>(sm)[i] = __float2bfloat16_rn(0.001f * (float)(i % 7));
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
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
    for (int k = 0; k < 16; ++k) z[k] = 0x3c003c00u;   // bf16 pairs of small values
    tmem_st16(tmem_addr(tmem, warp, A_TMEM_COL), z);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t id = idesc_bf16(128, n, 0, 0);
    const uint32_t ab = smem_u32(sm), bb = smem_u32(sm + A_BYTES);
    uint64_t ad[4], bd[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ad[k] = sdesc_sw128(ab + 32 * k, 16, 1024);
      bd[k] = sdesc_sw128(bb + 32 * k, 16, 1024);
    }
    uint32_t d[UNR];
#pragma unroll
    for (int k = 0; k < UNR; ++k) d[k] = tmem + (uint32_t)(((k / run) % n_acc) * n);
    const uint32_t at0 = tmem + A_TMEM_COL, at1 = at0 + 8;
    const unsigned long long t0 = clock64();
    for (int blk = 0; blk < n_blocks; ++blk) {
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        const bool ts = FORM == 1 || (FORM == 2 && (k & 1));
        if (ts)
          mma_ts(d[k], (k & 1) ? at1 : at0, bd[k & 3], id, 1u);
        else
          mma_ss(d[k], ad[k & 3], bd[k & 3], id, 1u);
      }
    }
    mma_commit(&bar);
    const bool ok = mbar_wait(&bar, 0, err);
    const unsigned long long t1 = clock64();
    cycles[blockIdx.x] = ok ? t1 - t0 : 0ull;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int FORM>
cudaError_t launch_diag(int n, int n_acc, int run, int n_blocks, int n_cta,
                        unsigned long long* cycles, int* err, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(diag_mma_kernel<FORM>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  diag_mma_kernel<FORM><<<n_cta, 128, SMEM, st>>>(n, n_acc, run, n_blocks, cycles, err);
  return cudaGetLastError();
}

}  // namespace
}  // namespace laga

extern "C" laga_status laga_diag_mma_rate(int form, int n, int n_acc, int run, int n_instr,
                                          int n_cta, unsigned long long* cycles, void* stream) {
  using namespace laga;
  if (form < 0 || form > 2 || n < 16 || n > 256 || n % 16 != 0 || n_acc < 1 || run < 1 ||
      n_instr < 1 || n_instr > (1 << 20) || n_cta < 1 || n_cta > 4096 || !cycles)
    return LAGA_ERR_ARG;
  if (n_acc * n > (form == 0 ? 512 : A_TMEM_COL) || n_instr % UNR != 0 ||
      UNR % (n_acc * run) != 0)
    return LAGA_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(cycles) & 7u) != 0) return LAGA_ERR_ALIGN;
  void* err = nullptr;
  if (cudaGetSymbolAddress(&err, g_diag_err) != cudaSuccess) return LAGA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int nb = n_instr / UNR;
  int* ew = static_cast<int*>(err);
  cudaError_t e = form == 0   ? launch_diag<0>(n, n_acc, run, nb, n_cta, cycles, ew, st)
                  : form == 1 ? launch_diag<1>(n, n_acc, run, nb, n_cta, cycles, ew, st)
                              : launch_diag<2>(n, n_acc, run, nb, n_cta, cycles, ew, st);
  return e == cudaSuccess ? LAGA_OK : LAGA_ERR_CUDA;
}
