// Host-side plan of one laga_fwd / laga_bwd call: validated dims and the
// byte layout of both workspaces.  Pure host code (no CUDA calls), so the
// accounting entry points work without a GPU.
#pragma once

#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/laga.h"

namespace laga {

enum BufId {
  // saved by the forward (LAGA_WS_SAVED)
  W_L = 0,      // bf16 [B*S, 512]      normalised latent, L = LN(x)*gamma
  W_MEAN,       // fp32 [B*S]           LayerNorm mean
  W_RSTD,       // fp32 [B*S]           LayerNorm 1/sqrt(var + eps)
  W_KPE,        // bf16 [B*S, 64]       RoPE'd k_pe (shared by all heads)
  W_QR,         // bf16 [B*S*H, 64]     RoPE'd q_rope
  W_KV,         // bf16 [B*S*H, 256]    k_nope | v per head (LAGA/explicit; not
                //                      kept by the fused form)
  W_QABS,       // bf16 [B*S*H, 512]    q_absorbed (absorbed form)
  W_OLAT,       // bf16 [B*S*H, 512]    latent accumulator (absorbed form)
  W_QN,         // bf16 [B*S*H, 128]    padded q_nope (non-canonical dims / fp32)
  W_WC,         // bf16 [512, H*256]    padded W_kv_b shard
  W_OC,         // bf16 [B*S*H, 128]    padded O
  N_SAVED,
  // transient of the backward (LAGA_WS_BWD)
  T_DELTA = N_SAVED,  // fp32 [B*H, Sp]  rowsum(dO * O), rows padded to Sp = ceil128(S)
  T_LSE2,       // fp32 [B*H, Sp]       LSE * log2(e) in the same padded rows
  T_DOC,        // bf16 [B*S*H, 128]    padded / converted dO
  T_DQ,         // fp32 [B*S*H, 192]    dq in the rotated frame
  T_DKV,        // bf16 [B*S*H, 256]    dk_nope | dv per head
  T_DKPE,       // fp32 [B*S*H, 64]     per-head dk_pe (rotated frame)
  T_DL,         // fp32 [B*S, 512]      gradient of L
  T_DGP,        // fp32 [NGP, 512]      dgamma partial sums
  T_DWC,        // fp32 [512, H*256]    padded dW shard
  T_DOLAT,      // bf16 [B*S*H, 512]    dO up-projected to the latent (absorbed)
  T_DQABS,      // fp32 [B*S*H, 512]    gradient of q_absorbed (absorbed)
  T_DWP,        // fp32 [splits, 512, H*256] split-K partials of dW
  T_KV,         // bf16 [B*S*H, 256]    fused form: K/V rebuilt by the dK/dV kernel
  N_BWD_END,
  // transient of the forward (LAGA_WS_FWD)
  F_KV = N_BWD_END,  // bf16 [B*S*H, 256] fused form: the forward's K/V
  N_BUF
};

// Number of dgamma partial rows (fixed, so the reduction order is fixed).
constexpr int NGP = 296;

struct Plan {
  laga_dims d{};
  int B = 0, S = 0, H = 0, dn = 0, dr = 0, dv = 0, dkv = 0;
  bool canonical = false;   // dims are 128/64/128/512 and I/O is bf16
  bool fp32 = false;
  bool rms = false;         // RMS variant of the latent norm (no mean subtraction)
  bool fused = false;       // LAGA_FORM_LAGA_FUSED: K/V rebuilt in the dK/dV kernel
  float scale = 0.f;
  size_t off[N_BUF] = {};
  size_t len[N_BUF] = {};
  size_t saved_bytes = 0, bwd_bytes = 0, fwd_bytes = 0;

  long long tokens() const { return (long long)B * S; }
  long long rows() const { return (long long)B * S * H; }  // (token, head) rows
  long long s_pad() const { return (S + 127) / 128 * 128; }  // padded row length
};

static const char* const kBufName[N_BUF] = {
    "L", "ln_mean", "ln_rstd", "k_pe_rot", "q_rope_rot", "kv", "q_absorbed", "o_latent",
    "q_nope_padded", "w_kvb_padded", "o_padded",
    "delta", "lse_log2", "dO_padded", "dq_rot", "dkv", "dk_pe_heads", "dL", "dgamma_partials",
    "dw_padded", "dO_latent", "dq_absorbed", "dw_split_partials", "kv_rebuilt", "kv"};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Token-reduction splits of the dW GEMM (at most 8).  Its CTA pairs (76 on
// 152 SMs) run 2*H*s output tiles of ceil(steps/s) 64-token steps each, and
// every split past the first writes and re-reads an fp32 partial of the
// shard's dW (8 MB at 16 heads, costed as ~7 token steps of MMA time).  The
// count minimising waves x steps + partial traffic depends on the dims only,
// so the summation order is fixed.
inline int dw_splits(int H, int token_steps) {
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= 8; ++s) {
    const long long waves = (2LL * H * s + 75) / 76;
    const long long steps = (token_steps + s - 1) / s;
    const long long cost = 16 * waves * steps + (s > 1 ? 7LL * s * H : 0);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// Validate dims; returns LAGA_OK or the error and fills the plan.
inline laga_status make_plan(const laga_dims* dims, Plan* p) {
  if (!dims || !p) return LAGA_ERR_ARG;
  const laga_dims& d = *dims;
  if (d.B < 1 || d.S < 1 || d.n_h_shard < 1 || d.n_h_total < 1 || d.head_offset < 0 ||
      d.head_offset + d.n_h_shard > d.n_h_total)
    return LAGA_ERR_ARG;
  if (d.d_nope < 16 || d.d_nope > 128 || d.d_nope % 16 || d.d_v < 16 || d.d_v > 128 ||
      d.d_v % 16 || d.d_kv < 16 || d.d_kv > 512 || d.d_kv % 16 || d.d_rope < 2 ||
      d.d_rope > 64 || d.d_rope % 2)
    return LAGA_ERR_ARG;
  if (!(d.scale >= 0.f) || !(d.ln_eps > 0.f)) return LAGA_ERR_ARG;
  if (d.io_dtype != LAGA_BF16 && d.io_dtype != LAGA_FP32) return LAGA_ERR_ARG;
  if (d.form != LAGA_FORM_LAGA && d.form != LAGA_FORM_EXPLICIT && d.form != LAGA_FORM_ABSORBED &&
      d.form != LAGA_FORM_LAGA_FUSED)
    return LAGA_ERR_ARG;
  if (d.norm != LAGA_NORM_LAYER && d.norm != LAGA_NORM_RMS) return LAGA_ERR_ARG;
  if (d.causal != 1) return LAGA_ERR_UNSUPPORTED;
  // Keep every element index inside 32-bit row counts times 64-bit strides.
  if ((long long)d.B * d.S * d.n_h_shard > (1LL << 31) - 1) return LAGA_ERR_ARG;

  p->d = d;
  p->B = d.B; p->S = d.S; p->H = d.n_h_shard;
  p->dn = d.d_nope; p->dr = d.d_rope; p->dv = d.d_v; p->dkv = d.d_kv;
  p->fp32 = d.io_dtype == LAGA_FP32;
  p->rms = d.norm == LAGA_NORM_RMS;
  p->fused = d.form == LAGA_FORM_LAGA_FUSED;
  p->canonical = !p->fp32 && d.d_nope == 128 && d.d_rope == 64 && d.d_v == 128 && d.d_kv == 512;
  p->scale = d.scale > 0.f ? d.scale : 1.0f / sqrtf((float)(d.d_nope + d.d_rope));

  const size_t T = (size_t)p->tokens(), R = (size_t)p->rows(), H = (size_t)p->H;
  const bool absorbed = d.form == LAGA_FORM_ABSORBED;
  for (int i = 0; i < N_BUF; ++i) p->len[i] = 0;
  p->len[W_L] = T * 512 * 2;
  p->len[W_MEAN] = T * 4;
  p->len[W_RSTD] = T * 4;
  p->len[W_KPE] = T * 64 * 2;
  p->len[W_QR] = R * 64 * 2;
  if (!absorbed && !p->fused) p->len[W_KV] = R * 256 * 2;
  if (absorbed) { p->len[W_QABS] = R * 512 * 2; p->len[W_OLAT] = R * 512 * 2; }
  if (!p->canonical) {
    p->len[W_QN] = R * 128 * 2;
    p->len[W_WC] = (size_t)512 * H * 256 * 2;
    p->len[W_OC] = R * 128 * 2;
  }
  p->len[T_DELTA] = (size_t)p->B * H * p->s_pad() * 4;
  p->len[T_LSE2] = (size_t)p->B * H * p->s_pad() * 4;
  if (!p->canonical) p->len[T_DOC] = R * 128 * 2;
  if (absorbed || !p->canonical) p->len[T_DQ] = R * 192 * 4;
  if (!absorbed) p->len[T_DKV] = R * 256 * 2;
  p->len[T_DKPE] = R * 64 * 4;
  p->len[T_DL] = T * 512 * 4;
  p->len[T_DGP] = (size_t)NGP * 512 * 4;
  if (!p->canonical) p->len[T_DWC] = (size_t)512 * H * 256 * 4;
  if (absorbed) {
    p->len[T_DOLAT] = R * 512 * 2;
    p->len[T_DQABS] = R * 512 * 4;
  }
  const int splits = dw_splits(p->H, p->B * ((p->S + 63) / 64));
  if (!absorbed && splits > 1) p->len[T_DWP] = (size_t)splits * 512 * H * 256 * 4;
  if (p->fused) {
    p->len[T_KV] = R * 256 * 2;
    p->len[F_KV] = R * 256 * 2;
  }
  size_t o = 0;
  for (int i = 0; i < N_SAVED; ++i) { p->off[i] = o; o = align_up(o + p->len[i], 1024); }
  p->saved_bytes = o;
  o = 0;
  for (int i = N_SAVED; i < N_BWD_END; ++i) { p->off[i] = o; o = align_up(o + p->len[i], 1024); }
  p->bwd_bytes = o;
  o = 0;
  for (int i = N_BWD_END; i < N_BUF; ++i) { p->off[i] = o; o = align_up(o + p->len[i], 1024); }
  p->fwd_bytes = o;
  return LAGA_OK;
}

}  // namespace laga
