// Host-side launchers of the LAGA kernels (one per .cu translation unit).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "plan.h"

namespace laga {

// Every pointer one call touches: the caller's tensors and both workspaces.
struct Ptrs {
  const void* q = nullptr;
  const void* c = nullptr;
  const void* w = nullptr;
  const float* gamma = nullptr;
  const float* cos = nullptr;
  const float* sin = nullptr;
  void* o = nullptr;
  float* lse = nullptr;
  const void* d_o = nullptr;
  void* dq = nullptr;
  float* dc = nullptr;
  float* dw = nullptr;
  float* dgamma = nullptr;
  unsigned char* ws_saved = nullptr;
  unsigned char* ws_bwd = nullptr;
  unsigned char* ws_fwd = nullptr;   // forward scratch (fused form)
  int* err = nullptr;  // device error word

  template <typename T>
  T* buf(const Plan& p, int id) const {
    unsigned char* base = id < N_SAVED ? ws_saved : (id < N_BWD_END ? ws_bwd : ws_fwd);
    return reinterpret_cast<T*>(base + p.off[id]);
  }
};

// Bracket one kernel launch: counts it for laga_last_launch_count() and,
// while profiling is on, records CUDA events on `st` around it.
struct LaunchScope {
  LaunchScope(const char* name, cudaStream_t st);
  ~LaunchScope();
  const char* name;
  cudaStream_t st;
  int slot;
};

// prep.cu: HBM-bound prologue / epilogue kernels.
cudaError_t launch_pad_w(const Plan& p, const Ptrs& x, cudaStream_t st);
cudaError_t launch_prep_fwd(const Plan& p, const Ptrs& x, cudaStream_t st);
cudaError_t launch_unpad_o(const Plan& p, const Ptrs& x, cudaStream_t st);
cudaError_t launch_bwd_pre(const Plan& p, const Ptrs& x, cudaStream_t st);
cudaError_t launch_dq_finalize(const Plan& p, const Ptrs& x, cudaStream_t st);
cudaError_t launch_norm_bwd(const Plan& p, const Ptrs& x, const float* dL, cudaStream_t st);
cudaError_t launch_unpad_dw(const Plan& p, const Ptrs& x, cudaStream_t st);

// gemm.cu: the up-projection and its two backward GEMMs.
cudaError_t launch_upproj(const Plan& p, const Ptrs& x, cudaStream_t st);
cudaError_t launch_upproj_bwd(const Plan& p, const Ptrs& x, cudaStream_t st);

// absorbed.cu: the absorbed-form contrast path (attention over the latent).
cudaError_t launch_absorbed_fwd(const Plan& p, const Ptrs& x, cudaStream_t st);
cudaError_t launch_absorbed_bwd(const Plan& p, const Ptrs& x, cudaStream_t st);

// attn_fwd.cu: causal attention forward.  attn_bwd_kv.cu / attn_bwd_dq.cu:
// its backward, split into a key-stationary dK/dV kernel and a
// query-stationary dQ kernel.
cudaError_t launch_attn_fwd(const Plan& p, const Ptrs& x, cudaStream_t st);
cudaError_t launch_attn_bwd_kv(const Plan& p, const Ptrs& x, cudaStream_t st);
cudaError_t launch_attn_bwd_dq(const Plan& p, const Ptrs& x, cudaStream_t st);

// Pointers and strides the kernels share, derived from the plan.
struct Views {
  const __nv_bfloat16* qn;  long long qn_ld;   // q_nope rows
  const __nv_bfloat16* qr;                      // [R, 64]
  const __nv_bfloat16* L;                       // [T, 512]
  const __nv_bfloat16* kpe;                     // [T, 64]
  const __nv_bfloat16* W;   long long w_ld;     // shard [512, H*256]
  __nv_bfloat16* kv;                            // per-head [.., 256]
  long long kv_sb, kv_ss, kv_sh;                // kv element strides
  __nv_bfloat16* O;                             // [R, 128] canonical O
  const __nv_bfloat16* dO;                      // [R, 128] canonical dO
};
Views make_views(const Plan& p, const Ptrs& x);

}  // namespace laga
