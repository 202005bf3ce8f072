// C ABI of the library (declared in include/laga.h): argument checks, the
// workspace plan and the launch sequence of each pass.
#include <mutex>
#include <nvtx3/nvToolsExt.h>
#include <string.h>
#include <utility>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace laga {

namespace {
thread_local int t_launches = 0;
__device__ int g_err_word;  // one per device: a bounded wait that gave up writes here
constexpr int kMaxDev = 64;
int* g_err_ptr[kMaxDev] = {};
std::mutex g_err_mu;

laga_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LAGA_OK : LAGA_ERR_CUDA; }

// Device address of the error word on the current device (looked up once).
laga_status err_word(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return LAGA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return LAGA_ERR_CUDA;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_err_ptr[dev];
  return LAGA_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

// An NVTX range around one whole entry-point call.
struct NvtxCall {
  explicit NvtxCall(const char* n) { nvtxRangePushA(n); }
  ~NvtxCall() { nvtxRangePop(); }
};

// ----------------------------------------------------------- launch records
namespace {
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_pending;
std::vector<cudaEvent_t> g_prof_pool;
std::vector<std::pair<const char*, std::pair<double, int>>> g_prof_acc;

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

// Every launch is also an NVTX range named after its kernel (host side: the
// enqueue), which a profiler attached to the process shows on its timeline;
// without one the push and pop are a check of a null hook.
LaunchScope::LaunchScope(const char* n, cudaStream_t s) : name(n), st(s), slot(-1) {
  ++t_launches;
  nvtxRangePushA(n);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) return;
  cudaEvent_t a = prof_event(), b = prof_event();
  if (!a || !b) return;
  cudaEventRecord(a, st);
  g_prof_pending.push_back({name, a, b});
  slot = (int)g_prof_pending.size() - 1;
}

LaunchScope::~LaunchScope() {
  if (slot >= 0) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (slot < (int)g_prof_pending.size()) cudaEventRecord(g_prof_pending[slot].b, st);
  }
  nvtxRangePop();
}

Views make_views(const Plan& p, const Ptrs& x) {
  Views v{};
  if (p.canonical) {
    v.qn = static_cast<const __nv_bfloat16*>(x.q);
    v.qn_ld = DQK;
    v.W = static_cast<const __nv_bfloat16*>(x.w) + (long long)p.d.head_offset * DH;
    v.w_ld = (long long)p.d.n_h_total * DH;
    v.O = static_cast<__nv_bfloat16*>(x.o);
    v.dO = static_cast<const __nv_bfloat16*>(x.d_o);
  } else {
    v.qn = x.buf<__nv_bfloat16>(p, W_QN);
    v.qn_ld = DN;
    v.W = x.buf<__nv_bfloat16>(p, W_WC);
    v.w_ld = (long long)p.H * DH;
    v.O = x.buf<__nv_bfloat16>(p, W_OC);
    v.dO = x.ws_bwd ? x.buf<__nv_bfloat16>(p, T_DOC) : nullptr;
  }
  v.qr = x.buf<__nv_bfloat16>(p, W_QR);
  v.L = x.buf<__nv_bfloat16>(p, W_L);
  v.kpe = x.buf<__nv_bfloat16>(p, W_KPE);
  // The fused form keeps no K/V between the passes: the forward's lives in
  // its scratch, the backward's is rebuilt by the dK/dV kernel.
  v.kv = !p.fused ? x.buf<__nv_bfloat16>(p, W_KV)
                  : x.buf<__nv_bfloat16>(p, x.ws_bwd ? T_KV : F_KV);
  const long long S = p.S, H = p.H;
  if (p.d.form == LAGA_FORM_EXPLICIT) {  // head-major [B, H, S, 256]
    v.kv_sb = H * S * DH; v.kv_ss = DH; v.kv_sh = S * DH;
  } else {                               // token-major [B, S, H, 256]
    v.kv_sb = S * H * DH; v.kv_ss = H * DH; v.kv_sh = DH;
  }
  return v;
}

}  // namespace laga

using namespace laga;

// One thread waits, with a short bound (2^16 polls, ~17 ms), on an mbarrier
// that nothing arrives on, then records the timeout code in the device error
// word -- the same path every kernel's bounded waits take.
static __global__ void selftest_wait_timeout_kernel(int* err) {
  __shared__ uint64_t bar;
  laga::sm100::mbar_init(&bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  for (uint32_t i = 0; i < (1u << 16); ++i) {
    if (laga::sm100::mbar_try_wait(&bar, 0)) return;
    __nanosleep(256);
  }
  atomicExch(err, laga::DEV_ERR_TIMEOUT);
}


extern "C" {

size_t laga_workspace_bytes(const laga_dims* dims, int pass) {
  Plan p;
  if (make_plan(dims, &p) != LAGA_OK) return 0;
  if (pass == LAGA_WS_SAVED) return p.saved_bytes;
  if (pass == LAGA_WS_BWD) return p.bwd_bytes;
  if (pass == LAGA_WS_FWD) return p.fwd_bytes;
  return 0;
}

laga_status laga_workspace_tensor(const laga_dims* dims, int pass, int index, const char** name,
                                  size_t* offset, size_t* bytes) {
  Plan p;
  laga_status s = make_plan(dims, &p);
  if (s != LAGA_OK) return s;
  if (!name || !offset || !bytes || index < 0) return LAGA_ERR_ARG;
  const int lo = pass == LAGA_WS_SAVED ? 0
                 : pass == LAGA_WS_BWD ? N_SAVED
                 : pass == LAGA_WS_FWD ? N_BWD_END : -1;
  const int hi = pass == LAGA_WS_SAVED ? N_SAVED : pass == LAGA_WS_BWD ? N_BWD_END : N_BUF;
  if (lo < 0) return LAGA_ERR_ARG;
  int k = -1;
  for (int i = lo; i < hi; ++i) {
    if (p.len[i] == 0) continue;
    if (++k == index) {
      *name = kBufName[i];
      *offset = p.off[i];
      *bytes = p.len[i];
      return LAGA_OK;
    }
  }
  return LAGA_ERR_ARG;
}

laga_status laga_fwd_scratch(const laga_dims* dims, const void* q, const void* c,
                             const void* w_kvb, const float* gamma, const float* cos,
                             const float* sin, void* o, float* lse, void* ws_saved,
                             size_t saved_bytes, void* ws_fwd, size_t fwd_bytes, void* stream) {
  NvtxCall range_("laga_fwd");
  t_launches = 0;
  Plan p;
  laga_status s = make_plan(dims, &p);
  if (s != LAGA_OK) return s;
  const bool absorbed = p.d.form == LAGA_FORM_ABSORBED;
  const void* ptrs[] = {q, c, w_kvb, gamma, cos, sin, o, lse, ws_saved};
  for (const void* ptr : ptrs)
    if (!ptr) return LAGA_ERR_ARG;
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return LAGA_ERR_ALIGN;
  if (ws_fwd && !aligned16(ws_fwd)) return LAGA_ERR_ALIGN;
  if (saved_bytes < p.saved_bytes) return LAGA_ERR_WORKSPACE;
  if (p.fwd_bytes > 0 && (!ws_fwd || fwd_bytes < p.fwd_bytes)) return LAGA_ERR_WORKSPACE;
  Ptrs x;
  x.q = q; x.c = c; x.w = w_kvb; x.gamma = gamma; x.cos = cos; x.sin = sin;
  x.o = o; x.lse = lse;
  x.ws_saved = static_cast<unsigned char*>(ws_saved);
  x.ws_fwd = static_cast<unsigned char*>(ws_fwd);
  if ((s = err_word(&x.err)) != LAGA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (!p.canonical) e = launch_pad_w(p, x, st);
  if (e == cudaSuccess) e = launch_prep_fwd(p, x, st);
  if (absorbed) {
    if (e == cudaSuccess) e = launch_absorbed_fwd(p, x, st);
  } else {
    if (e == cudaSuccess) e = launch_upproj(p, x, st);
    if (e == cudaSuccess) e = launch_attn_fwd(p, x, st);
  }
  if (e == cudaSuccess && !p.canonical) e = launch_unpad_o(p, x, st);
  return cuda_status(e);
}

laga_status laga_fwd(const laga_dims* dims, const void* q, const void* c, const void* w_kvb,
                     const float* gamma, const float* cos, const float* sin, void* o, float* lse,
                     void* ws_saved, size_t saved_bytes, void* stream) {
  return laga_fwd_scratch(dims, q, c, w_kvb, gamma, cos, sin, o, lse, ws_saved, saved_bytes,
                          nullptr, 0, stream);
}

// The backward of one shard.  `aux` is either `st` (everything in stream
// order on the caller's stream) or a second stream of the caller's, forked
// from `st` with `fork` and joined back with `join`: the dQ kernel, which
// nothing after it reads on canonical dims, then runs beside the dK/dV
// kernel, and the up-projection and norm backward (which need only dK/dV)
// fill the dQ kernel's last wave.
static laga_status bwd_impl(const laga_dims* dims, const void* q, const void* c,
                            const void* w_kvb, const float* gamma, const float* cos,
                            const float* sin, const void* o, const float* lse, const void* d_o,
                            void* dq, float* dc, float* dw, float* dgamma, const void* ws_saved,
                            size_t saved_bytes, void* ws_bwd, size_t bwd_bytes, cudaStream_t st,
                            cudaStream_t aux, cudaEvent_t fork_ev, cudaEvent_t join_ev) {
  NvtxCall range_("laga_bwd");
  t_launches = 0;
  Plan p;
  laga_status s = make_plan(dims, &p);
  if (s != LAGA_OK) return s;
  const bool absorbed = p.d.form == LAGA_FORM_ABSORBED;
  const void* ptrs[] = {q, c, w_kvb, gamma, cos, sin, o, lse, d_o, dq, dc, dw, dgamma,
                        ws_saved, ws_bwd};
  for (const void* ptr : ptrs)
    if (!ptr) return LAGA_ERR_ARG;
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return LAGA_ERR_ALIGN;
  if (saved_bytes < p.saved_bytes || bwd_bytes < p.bwd_bytes) return LAGA_ERR_WORKSPACE;
  Ptrs x;
  x.q = q; x.c = c; x.w = w_kvb; x.gamma = gamma; x.cos = cos; x.sin = sin;
  x.o = const_cast<void*>(o); x.lse = const_cast<float*>(lse); x.d_o = d_o;
  x.dq = dq; x.dc = dc; x.dw = dw; x.dgamma = dgamma;
  x.ws_saved = static_cast<unsigned char*>(const_cast<void*>(ws_saved));
  x.ws_bwd = static_cast<unsigned char*>(ws_bwd);
  if ((s = err_word(&x.err)) != LAGA_OK) return s;
  // With per-kernel profiling on, every kernel runs in turn on `st` so that
  // each kernel's events time it alone.
  const bool fork = !absorbed && !p.fused && aux != st && !g_prof_on;
  cudaError_t e = launch_bwd_pre(p, x, st);
  if (absorbed) {
    if (e == cudaSuccess) e = launch_absorbed_bwd(p, x, st);
    if (e == cudaSuccess) e = launch_dq_finalize(p, x, st);
  } else {
    cudaStream_t dq_st = st;
    if (fork) {
      if (e == cudaSuccess) e = cudaEventRecord(fork_ev, st);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(aux, fork_ev, 0);
      dq_st = aux;
    }
    if (e == cudaSuccess) e = launch_attn_bwd_kv(p, x, st);
    if (e == cudaSuccess) e = launch_attn_bwd_dq(p, x, dq_st);   // canonical: writes dq itself
    if (fork && e == cudaSuccess) e = cudaEventRecord(join_ev, aux);
    if (!p.canonical) {
      if (fork && e == cudaSuccess) e = cudaStreamWaitEvent(st, join_ev, 0);
      if (e == cudaSuccess) e = launch_dq_finalize(p, x, st);
    }
    if (e == cudaSuccess) e = launch_upproj_bwd(p, x, st);
  }
  if (e == cudaSuccess && !p.canonical) e = launch_unpad_dw(p, x, st);
  if (e == cudaSuccess) e = launch_norm_bwd(p, x, x.buf<float>(p, T_DL), st);
  if (fork && p.canonical && e == cudaSuccess) e = cudaStreamWaitEvent(st, join_ev, 0);
  return cuda_status(e);
}

laga_status laga_bwd(const laga_dims* dims, const void* q, const void* c, const void* w_kvb,
                     const float* gamma, const float* cos, const float* sin, const void* o,
                     const float* lse, const void* d_o, void* dq, float* dc, float* dw,
                     float* dgamma, const void* ws_saved, size_t saved_bytes, void* ws_bwd,
                     size_t bwd_bytes, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return bwd_impl(dims, q, c, w_kvb, gamma, cos, sin, o, lse, d_o, dq, dc, dw, dgamma, ws_saved,
                  saved_bytes, ws_bwd, bwd_bytes, st, st, nullptr, nullptr);
}

laga_status laga_bwd_overlap(const laga_dims* dims, const void* q, const void* c,
                             const void* w_kvb, const float* gamma, const float* cos,
                             const float* sin, const void* o, const float* lse, const void* d_o,
                             void* dq, float* dc, float* dw, float* dgamma, const void* ws_saved,
                             size_t saved_bytes, void* ws_bwd, size_t bwd_bytes, void* stream,
                             void* aux_stream, void* fork_event, void* join_event) {
  if (!fork_event || !join_event || aux_stream == stream) return LAGA_ERR_ARG;
  return bwd_impl(dims, q, c, w_kvb, gamma, cos, sin, o, lse, d_o, dq, dc, dw, dgamma, ws_saved,
                  saved_bytes, ws_bwd, bwd_bytes, static_cast<cudaStream_t>(stream),
                  static_cast<cudaStream_t>(aux_stream), static_cast<cudaEvent_t>(fork_event),
                  static_cast<cudaEvent_t>(join_event));
}

laga_status laga_selftest_wait_timeout(void* stream) {
  int* w = nullptr;
  laga_status s = err_word(&w);
  if (s != LAGA_OK) return s;
  selftest_wait_timeout_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(w);
  return cudaGetLastError() == cudaSuccess ? LAGA_OK : LAGA_ERR_CUDA;
}

laga_status laga_sync_check(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return LAGA_ERR_CUDA;
  int* w = nullptr;
  laga_status s = err_word(&w);
  if (s != LAGA_OK) return s;
  int v = 0;
  if (cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LAGA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return LAGA_ERR_CUDA;
    return static_cast<laga_status>(v);
  }
  return LAGA_OK;
}

const char* laga_status_string(laga_status status) {
  switch (status) {
    case LAGA_OK: return "ok";
    case LAGA_ERR_ARG: return "invalid argument";
    case LAGA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case LAGA_ERR_WORKSPACE: return "workspace too small";
    case LAGA_ERR_UNSUPPORTED: return "unsupported configuration";
    case LAGA_ERR_CUDA: return "CUDA error";
    case LAGA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int laga_last_launch_count(void) { return t_launches; }

void laga_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
}

void laga_profile_reset(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof_pending) {
    cudaEventSynchronize(r.b);
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_pending.clear();
  g_prof_acc.clear();
}

int laga_profile_read(const char** names, double* total_ms, int* launches, int max) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      bool found = false;
      for (auto& acc : g_prof_acc)
        if (strcmp(acc.first, r.name) == 0) {
          acc.second.first += ms;
          acc.second.second += 1;
          found = true;
          break;
        }
      if (!found) g_prof_acc.push_back({r.name, {(double)ms, 1}});
    }
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_pending.clear();
  const int n = (int)g_prof_acc.size();
  for (int i = 0; i < n && i < max; ++i) {
    if (names) names[i] = g_prof_acc[i].first;
    if (total_ms) total_ms[i] = g_prof_acc[i].second.first;
    if (launches) launches[i] = g_prof_acc[i].second.second;
  }
  return n;
}

}  // extern "C"
