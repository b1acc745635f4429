// Latency-path draft block for one sequence (B = 1): a persistent kernel of one CTA per SM
// in which every weight slice and the attended shared K stay resident in shared memory for
// the whole block, and CTAs exchange vectors through "mailboxes" instead of grid barriers.
//
// Data flow of one drafter step (every GEMV is split by output rows over the N CTAs; every
// CTA keeps its own copy of the residual stream x and recomputes the norms):
//   PRE   gather the previous step's argmax keys -> token; e = embed row; gather h';
//         x0[rows] = W_pre [h ; e]                                      -> mailbox x0
//   per block l:
//     Q    gather x0 (l=0) or dn (l>0: x = lambda(x + norm(dn))); a = norm(x);
//          q[rows] = W_q a                                              -> mailbox q
//     ATT  gather q; q_norm + RoPE for all heads; softmax partial over this CTA's keys
//          (scores, max, exp-sum, weighted key sum)                     -> mailbox part
//     CMB  gather the partials of this CTA's output dims from all CTAs; combine -> o[dims]
//     O    gather o; o'[rows] = W_o o                                   -> mailbox o'
//     GU   gather o'; x += norm(o'); f = norm(x); m[rows] = gelu(W_g f) * W_u f -> mailbox m
//     DN   gather m; dn[rows] = W_d m                                   -> mailbox dn
//   HEAD  gather dn; x = lambda(x + norm(dn)); y = output_norm(x);
//         h'[rows] = W_post y (hidden output)                           -> mailbox h'
//         centroid logits[rows] = Cent y                                -> mailbox cent
//   TOPK  gather all centroid logits; top_k by radix select (every CTA, same result)
//   GATHER this CTA's token_ordering offsets of the selected centroids -> candidate rows;
//         logits; local (value, id) max; L2 prefetch of that token's embedding row
//                                                                       -> mailbox key
// A mailbox word is (epoch << 32 | fp32 bits): a reader polls until the word carries the
// epoch of the exchange it waits for, so no separate flag or fence is needed, and words
// left by earlier exchanges can never be mistaken for new ones.
#pragma once

#include "mtp_common.cuh"
#include "mtp.h"

namespace mtp {
namespace ll {

constexpr int kT = 512;
constexpr int kW = kT / 32;
constexpr int kMaxL = 8;
constexpr int kMaxSections = 2 + 5 * kMaxL + 4;
constexpr int kExPerStep = 64;  // mailbox epochs reserved per drafter step

typedef __nv_bfloat16 bf16;

struct Range {
  int lo, hi;
};
__host__ __device__ inline Range split(int R, int N, int c) {
  const long long lo = static_cast<long long>(R) * c / N, hi = static_cast<long long>(R) * (c + 1) / N;
  return Range{static_cast<int>(lo), static_cast<int>(hi)};
}
__host__ __device__ inline int split_max(int R, int N) { return (R + N - 1) / N; }
__host__ __device__ inline int align16(int v) { return (v + 15) & ~15; }

struct Params {
  int N;  // CTAs
  int bb, H, nl, nh, nkv, F, V, C, topk, vsc, W;
  int d[2];
  float scale[2], theta[2], eps;
  int ltype[kMaxL];
  float lambda[kMaxL];
  const bf16 *pre, *post, *temb, *cent, *tgt;
  const float* out_norm;
  const int* ord;
  const bf16 *q[kMaxL], *o[kMaxL], *gate[kMaxL], *up[kMaxL], *down[kMaxL];
  const float *q_norm[kMaxL], *attn_norm[kMaxL], *post_attn_norm[kMaxL], *ffn_norm[kMaxL], *post_ffn_norm[kMaxL];
  const bf16* k[2];
  const bf16* v[2];
  const int* ctx_len[2];
  long long sb[2], st[2];
  int kv_max[2];
  bool has_type[2];
  const bf16* hidden_in;
  const int* tok_in;
  const int* pos;
  int* out_tokens;
  float* out_hidden;
  int n_draft;
  // mailboxes
  unsigned long long *mb_x0, *mb_q, *mb_part, *mb_o, *mb_op, *mb_m, *mb_dn, *mb_h, *mb_cent, *mb_key;
  unsigned epoch_base;
  int* status;
  unsigned* abort_flag;
  long long spin_limit;
};

// ------------------------------------------------------------------ shared-memory layout

// Resident sections, in the order the phases first need them. Each section is sized for the
// largest share any CTA owns, so the offsets are the same in every CTA.
enum Sec { S_PRE = 0, S_LAYER = 1, S_POST = 1 + 5 * kMaxL, S_CENT, S_KF, S_KS, S_COUNT };
__host__ __device__ inline int sec_q(int l) { return S_LAYER + 5 * l; }
__host__ __device__ inline int sec_o(int l) { return S_LAYER + 5 * l + 1; }
__host__ __device__ inline int sec_g(int l) { return S_LAYER + 5 * l + 2; }
__host__ __device__ inline int sec_u(int l) { return S_LAYER + 5 * l + 3; }
__host__ __device__ inline int sec_d(int l) { return S_LAYER + 5 * l + 4; }

struct Layout {
  int sec_off[S_COUNT];
  int sec_bytes[S_COUNT];
  int ord_off, ord_count;       // token_ordering columns: [offsets][C] int32
  int r1_off, r1_floats;        // scratch 1: u / m / centroid logits
  int r2_off, r2_floats;        // scratch 2: q / o
  int x_off, t_off, a_off;      // [H] each
  int sc_off, sc_count;         // attention scores [keys][nh]
  int red_off, hist_off, sel_off, mbar_off;
  int cs_off, cs_half;          // RoPE (cos, sin): [2 types][cs_half] float2
  int g_off;                    // staged q_norm gains
  int total;
  int keys_f, keys_s;           // max keys per CTA of each attention type
  int offs_per_cta;             // token_ordering offsets per CTA
};

__host__ __device__ inline Layout make_layout(const Params& p) {
  Layout L{};
  const int N = p.N;
  int off = 0;
  auto put = [&](int s, int bytes) {
    L.sec_off[s] = off;
    L.sec_bytes[s] = align16(bytes);
    off += L.sec_bytes[s];
  };
  for (int s = 0; s < S_COUNT; ++s) { L.sec_off[s] = 0; L.sec_bytes[s] = 0; }
  put(S_PRE, split_max(p.H, N) * 2 * p.bb * 2);
  int dmax = 0;
  for (int l = 0; l < p.nl; ++l) {
    const int d = p.d[p.ltype[l]];
    dmax = d > dmax ? d : dmax;
    put(sec_q(l), split_max(p.nh * d, N) * p.H * 2);
    put(sec_o(l), split_max(p.H, N) * p.nh * d * 2);
    put(sec_g(l), split_max(p.F, N) * p.H * 2);
    put(sec_u(l), split_max(p.F, N) * p.H * 2);
    put(sec_d(l), split_max(p.H, N) * p.F * 2);
  }
  put(S_POST, split_max(p.bb, N) * p.H * 2);
  put(S_CENT, split_max(p.C, N) * p.H * 2);
  L.keys_f = p.has_type[1] ? split_max(p.kv_max[1], N) : 0;
  const int wmax = p.kv_max[0] < p.W ? p.kv_max[0] : p.W;
  L.keys_s = p.has_type[0] ? split_max(wmax, N) : 0;
  put(S_KF, L.keys_f * p.nkv * p.d[1] * 2);
  put(S_KS, L.keys_s * p.nkv * p.d[0] * 2);
  L.offs_per_cta = split_max(p.vsc, N);
  L.ord_off = off;
  L.ord_count = L.offs_per_cta * p.C;
  off += align16(L.ord_count * 4);
  int r1 = 2 * p.bb > p.F ? (2 * p.bb > p.C ? 2 * p.bb : p.C) : (p.F > p.C ? p.F : p.C);
  for (int l = 0; l < p.nl; ++l) {  // attention combine: N sources x (2 per head touched + dims)
    const int d = p.d[p.ltype[l]];
    const int nd = split_max(p.nh * d, N);
    const int cmb = N * (2 * (nd / d + 2) + nd);
    r1 = cmb > r1 ? cmb : r1;
  }
  L.r1_off = off;
  L.r1_floats = r1;
  off += align16(r1 * 4);
  L.r2_off = off;
  L.r2_floats = p.nh * dmax;
  off += align16(L.r2_floats * 4);
  L.x_off = off;
  off += align16(p.H * 4);
  L.t_off = off;
  off += align16(p.H * 4);
  L.a_off = off;
  off += align16(p.H * 4);
  const int kmax = L.keys_f > L.keys_s ? L.keys_f : L.keys_s;
  L.sc_off = off;
  L.sc_count = (kmax > 0 ? kmax : 1) * p.nh;
  off += align16(L.sc_count * 4);
  L.red_off = off;
  off += align16(128 * 4);   // [0,64) general, [64,72) q-norm factors, [80,88) max, [96,104) exp-sum
  L.hist_off = off;
  off += align16(260 * 4);
  L.sel_off = off;
  off += align16(64 * 4);
  L.g_off = off;             // staged gain vector (q_norm) [dmax]
  off += align16(dmax * 4);
  L.mbar_off = off;
  off += align16(S_COUNT * 8);
  L.cs_half = dmax / 2 > 1 ? dmax / 2 : 1;
  L.cs_off = off;
  off += 2 * L.cs_half * 8;
  L.total = align16(off);
  return L;
}

// Number of mailbox words each exchange needs (host sizing).
struct MailboxSizes {
  long long x0, q, part, o, op, m, dn, h, cent, key;
};
__host__ __device__ inline MailboxSizes mailbox_sizes(const Params& p) {
  int dmax = 0;
  for (int l = 0; l < p.nl; ++l) dmax = p.d[p.ltype[l]] > dmax ? p.d[p.ltype[l]] : dmax;
  MailboxSizes m;
  m.x0 = p.H;
  m.q = static_cast<long long>(p.nh) * dmax;
  m.part = static_cast<long long>(p.N) * p.nh * (dmax + 2);
  m.o = static_cast<long long>(p.nh) * dmax;
  m.op = p.H;
  m.m = p.F;
  m.dn = p.H;
  m.h = p.bb;
  m.cent = p.C;
  m.key = 2LL * p.N;   // (ordered value, id) per CTA
  return m;
}

}  // namespace ll
}  // namespace mtp
