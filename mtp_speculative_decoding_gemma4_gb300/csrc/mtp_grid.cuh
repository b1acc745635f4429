// Grid draft block for one sequence (B = 1): one persistent launch over every co-resident
// thread-block cluster of the GPU. Every projection is split over all CTAs (by output rows,
// or by input columns where the next step is a reduction), the split weights and the
// attended shared K stay in shared memory for the whole draft block, and the residual stream
// is replicated in the registers of every warp (H = 32 lanes x EPL elements), so norms need
// no block barrier.
//
// Data flow of one drafter step (Gemma 4 Multi-Token Prediction (MTP) drafter, "What it is"
// and "Tensor schema"; Gemma 4 Assistant tensor inventory, "Centroid / ordered embeddings LM
// head", steps 1-4). "AR" is an all-reduce of an H-vector, "AG" an all-gather:
//   PRE   partial x0 = W_pre[:, my h cols] h'[my cols] + W_pre[:, my e cols] embed(tok)[my cols]
//                                                                       AR -> x0
//   per block l:
//     Q    a = norm(x); q[my rows] = W_q[my rows] a                     AG q (attention CTAs)
//     ATT  (attention CTAs) q_norm + RoPE of every head; softmax partial over my keys
//          (max, exp-sum, weighted key sum; V = K)                      -> owners of q's dims
//     O    combine the partials of my dims -> o[my dims];
//          partial o' = W_o[:, my dims] o[my dims]                      AR -> o'
//     MLP  x += norm(o'); f = norm(x); m[my rows] = gelu(W_g f) * W_u f;
//          partial dn = W_d[:, my rows] m[my rows]                      AR -> dn
//          x = lambda (x + norm(dn))
//   HEAD  y = norm(x); h'[my rows] = W_post y (kept for the next step's PRE);
//         centroid logits[my rows] = Cent y                             AG logits
//         top_k (every CTA, same result, ties to the lower index); my share of the k*vsc
//         candidate rows of the token_ordering-order token_embd copy; local argmax
//                                                                       AG keys -> token
// An AR is a reduce-scatter over the cluster's distributed shared memory (st.async), a
// gather of this CTA's slice from every cluster through global memory, and an all-gather of
// the slices over distributed shared memory. Global exchanges use 64-bit mailbox words
// (epoch << 32 | 32-bit payload): a reader polls until a word carries the epoch of the
// exchange it waits for, so no flag or fence is needed and words of earlier exchanges or
// launches are never mistaken for new ones.
#pragma once

#include "mtp_common.cuh"
#include "mtp.h"

namespace mtp {
namespace gr {

constexpr int kLgT = 8;
constexpr int kT = 1 << kLgT;      // threads per CTA (few enough for 255 registers each: no spills)
constexpr int kW = kT / 32;        // warps per CTA
constexpr int kMaxL = 8;
constexpr int kMaxS = 16;          // largest cluster
constexpr int kMaxEx = 3 + 4 * kMaxL;
constexpr int kExPerStep = 64;     // mailbox epochs reserved per drafter step
constexpr int kMaxHeads = 16;
constexpr int kMaxGroup = 8;       // query heads per KV head
constexpr int kKeysPerCta = 8;     // fewest attended keys per attention CTA (when CTAs are available)
constexpr int kMaxTopK = 64;

typedef __nv_bfloat16 bf16;

struct Range {
  int lo, hi;
};
__host__ __device__ inline Range split(int R, int N, int c) {
  const long long lo = static_cast<long long>(R) * c / N, hi = static_cast<long long>(R) * (c + 1) / N;
  return Range{static_cast<int>(lo), static_cast<int>(hi)};
}
__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int al16(int v) { return (v + 15) & ~15; }
__host__ __device__ inline int max3(int a, int b, int c) { return a > b ? (a > c ? a : c) : (b > c ? b : c); }
__host__ __device__ inline int even(int v) { return (v + 1) & ~1; }

// Exchange indices within a step: 0 PRE AR; per block l: Q AG, ATT, O AR, DN AR; CENT AG; KEY AG.
__host__ __device__ inline int ex_q(int l) { return 1 + 4 * l; }
__host__ __device__ inline int ex_att(int l) { return 2 + 4 * l; }
__host__ __device__ inline int ex_o(int l) { return 3 + 4 * l; }
__host__ __device__ inline int ex_dn(int l) { return 4 + 4 * l; }
__host__ __device__ inline int ex_cent(int nl) { return 1 + 4 * nl; }
__host__ __device__ inline int ex_key(int nl) { return 2 + 4 * nl; }
__host__ __device__ inline int ex_count(int nl) { return 3 + 4 * nl; }

// Shared-memory layout. The weight sections come first, in the order of the per-CTA image
// (one bulk copy per group: pre + post, each block, centroids); every section is sized for
// the largest share any CTA holds, so offsets are the same in every CTA.
struct Layout {
  int kc;               // pre columns (of each half) / post rows per CTA
  int kcp;              // kc rounded up to even (row pitch of the pre sections)
  int nq[kMaxL];        // q rows = o columns per CTA
  int nqp[kMaxL];       // even pitch of the o section
  int nf, nfp;          // gate/up rows = down columns per CTA (and pitch)
  int ncent;            // centroid rows per CTA
  int pre, post, q[kMaxL], o[kMaxL], g[kMaxL], u[kMaxL], dn[kMaxL], cent;
  int grp_off[kMaxL + 2], grp_bytes[kMaxL + 2];
  int img_bytes;
  int kbuf, kbuf_bytes; // K rows of the resident attention types [kslots][nkv * d]: both at once
                        // (type t at kbuf + koff[t]) or one type at a time (koff 0)
  int koff[2];
  int ubuf, u_words;    // gather scratch (fp32)
  int qs;               // general attention: normed, rotated, scaled q [nh * dmax]; combine:
                        // per-head source weights; head: top-k candidates
  int cand_cap;         // top-k candidates the qs region holds
  int sc, ksl;          // scores / probabilities: [nh][ksl] (general attention) or [key][nh]
                        // (four-head form); ksl: largest key share
  int hc;               // h' share [kc] (fp32, carried to the next step)
  int vs;               // partial H-vector of an AR [H] (fp32)
  int xs;               // result of the last AR [H]
  int ms;               // gelu(gate) * up of my rows [nf]
  int cs;               // RoPE (cos, sin) [d_s / 2 + d_f / 2] float2 (lane-major for the
                        // four-head form's head dim)
  int rs, ag;           // AR receive buffers [2][H] each
  int vh;               // PRE partial over the h columns [H] (computed before the token is known)
  int red;              // 64 floats: attention ([h] q_norm factor, [16 + h] max, [32 + h]
                        // exp-sum), combine ([0, nq) o values, [48, 64) head denominators),
                        // top-k and prefix-sum warp totals
  int keys;             // [kW] u64 warp keys
  int gmax;             // top-k: [kMaxTopK] u64 group maxima, then ranks ([2][128] or [cand_cap] int)
  int sel;              // [kMaxTopK] selected centroids
  int bars;             // mbarriers: load groups (nl + 2), K, RS[2], AG[2]
  int total;
};

struct Params {
  int N, S, G;  // CTAs, cluster size, clusters
  int bb, H, nl, nh, nkv, F, V, C, topk, vsc, W;
  int d[2];
  float scale[2], theta[2], eps;
  int ltype[kMaxL];
  float lambda[kMaxL];
  int A[2];      // attention CTAs of each attention type
  int kres[2];   // 1: the CTA's keys of the type are bulk-copied into the shared K region before the
                 // first block of that type (the region holds one type at a time); 0: read from global
  int kslots[2]; // largest key share of an attention CTA (shared-memory rows / score slots)
  int kboth;     // 1: the resident types' keys are loaded once, side by side, for the whole launch
  int has_type[2];
  int lg_d[2], lg_hs, lg_vsc;  // log2 of the head dims, of H / S and of vsc (all powers of two)
  int tk_lg_per, tk_lg_tpg;    // top-k tiling: log2 of keys per thread and of threads per group (-1: untiled)
  // weights: per-CTA images [N][img_bytes] in the shared-memory layout (made at init)
  const unsigned char* img;
  long long img_bytes;
  const bf16* tgt;       // target input embedding table [V][bb]
  const bf16* temb_ord;  // token_embd rows in token_ordering order [V][H]
  const int* ord;        // token_ordering [V]
  const float* out_norm;
  const double* inv_freq;  // RoPE inverse frequencies [2][dmax / 2] (fp64, made at init)
  const float *q_norm[kMaxL], *attn_norm[kMaxL], *post_attn_norm[kMaxL], *ffn_norm[kMaxL], *post_ffn_norm[kMaxL];
  // shared K per attention type (V = K), sequence 0
  const bf16* k[2];
  const int* ctx_len[2];
  long long st[2];  // elements between tokens
  int kv_max[2];
  // call
  const bf16* hidden_in;
  const int* tok_in;
  const int* pos;
  int* out_tokens;
  float* out_hidden;
  int n_draft;
  // exchanges
  unsigned long long* mb;
  long long mb_words;           // mailbox words of the launch (both step parities)
  long long ex_off[2][kMaxEx];  // word offset of each exchange's mailbox region, by step parity
  unsigned epoch_base;
  int* status;
  unsigned* abort_flag;
  long long spin_limit;
  int dbg_skip;  // testing: CTA dbg_skip - 1 does not publish its words of the first exchange
  Layout L;      // shared-memory layout (host-computed)
};

__host__ __device__ inline int max_qd(const Params& p) {
  int m = 0;
  for (int l = 0; l < p.nl; ++l) m = p.nh * p.d[p.ltype[l]] > m ? p.nh * p.d[p.ltype[l]] : m;
  return m;
}
__host__ __device__ inline int max_d(const Params& p) {
  int m = 0;
  for (int l = 0; l < p.nl; ++l) m = p.d[p.ltype[l]] > m ? p.d[p.ltype[l]] : m;
  return m;
}

// Heads touched by a dim range [lo, hi) of the flattened q of head dim d.
__host__ __device__ inline int heads_touched(int lo, int hi, int d) { return hi > lo ? (hi - 1) / d - lo / d + 1 : 0; }

// Host only (loops over every CTA's share).
inline Layout make_layout(const Params& p) {
  Layout L{};
  const int N = p.N, H = p.H;
  L.kc = cdiv(p.bb, N);
  L.kcp = even(L.kc);
  L.nf = cdiv(p.F, N);
  L.nfp = even(L.nf);
  L.ncent = cdiv(p.C, N);
  int off = 0;
  L.grp_off[0] = off;
  L.pre = off;
  off += al16(2 * H * L.kcp * 2);
  L.post = off;
  off += al16(L.kc * H * 2);
  L.grp_bytes[0] = off - L.grp_off[0];
  for (int l = 0; l < p.nl; ++l) {
    const int QD = p.nh * p.d[p.ltype[l]];
    L.nq[l] = cdiv(QD, N);
    L.nqp[l] = even(L.nq[l]);
    L.grp_off[1 + l] = off;
    L.q[l] = off;
    off += al16(L.nq[l] * H * 2);
    L.o[l] = off;
    off += al16(H * L.nqp[l] * 2);
    L.g[l] = off;
    off += al16(L.nf * H * 2);
    L.u[l] = off;
    off += al16(L.nf * H * 2);
    L.dn[l] = off;
    off += al16(H * L.nfp * 2);
    L.grp_bytes[1 + l] = off - L.grp_off[1 + l];
  }
  L.grp_off[1 + p.nl] = off;
  L.cent = off;
  off += al16(L.ncent * H * 2);
  L.grp_bytes[1 + p.nl] = off - L.grp_off[1 + p.nl];
  L.img_bytes = off;
  L.kbuf = off;
  L.kbuf_bytes = 0;
  L.koff[0] = L.koff[1] = 0;
  for (int t = 0; t < 2; ++t) {
    if (!p.has_type[t] || !p.kres[t]) continue;
    const int b = p.kslots[t] * p.nkv * p.d[t] * 2;
    if (p.kboth) {
      L.koff[t] = L.kbuf_bytes;
      L.kbuf_bytes += al16(b);
    } else if (b > L.kbuf_bytes) {
      L.kbuf_bytes = b;
    }
  }
  off += al16(L.kbuf_bytes);
  // gather scratch: q (max QD), centroid logits (C), attention partials of my dims
  // (A x (nq + 2 x heads touched)), AR slices (G x H / S), argmax keys (2N)
  int uw = max_qd(p);
  uw = p.C > uw ? p.C : uw;
  for (int l = 0; l < p.nl; ++l) {
    const int t = p.ltype[l], d = p.d[t];
    int ht = 0;
    for (int c = 0; c < N; ++c) {
      const Range r = split(p.nh * d, N, c);
      const int h = heads_touched(r.lo, r.hi, d);
      ht = h > ht ? h : ht;
    }
    const int w = p.A[t] * (L.nq[l] + 2 * ht);
    uw = w > uw ? w : uw;
  }
  uw = p.G * (H / p.S) > uw ? p.G * (H / p.S) : uw;
  uw = 2 * N > uw ? 2 * N : uw;
  L.u_words = uw;
  L.ubuf = off;
  off += al16(uw * 4);
  L.qs = off;
  L.cand_cap = max_qd(p) * 4 / 12 < kT ? max_qd(p) * 4 / 12 : kT;  // top-k candidates: int + u64 each
  off += al16(max_qd(p) * 4);
  int ks = 1;
  for (int t = 0; t < 2; ++t)
    if (p.has_type[t] && p.kslots[t] > ks) ks = p.kslots[t];
  L.sc = off;
  L.ksl = ks;
  off += al16(p.nh * ks * 4);
  L.hc = off;
  off += al16(L.kc * 4);
  L.vs = off;
  off += al16(H * 4);
  L.xs = off;
  off += al16(H * 4);
  L.vh = off;
  off += al16(H * 4);
  L.ms = off;
  off += al16(L.nf * 4);
  L.cs = off;
  off += al16((p.d[0] / 2 + p.d[1] / 2 + 1) * 8);
  L.rs = off;
  off += al16(2 * H * 4);
  L.ag = off;
  off += al16(2 * H * 4);
  L.red = off;
  off += al16(64 * 4);
  L.keys = off;
  off += al16(kW * 8);
  L.gmax = off;
  off += al16(max3(kMaxTopK * 8, 2 * 128 * 4, L.cand_cap * 4));  // group maxima, then ranks
  L.sel = off;
  off += al16(kMaxTopK * 4);
  L.bars = off;
  off += al16((p.nl + 2 + 1 + 4) * 8);
  L.total = al16(off);
  return L;
}

// Mailbox words of one exchange (one step parity).
__host__ inline long long ex_words(const Params& p, int x) {
  if (x == 0) return static_cast<long long>(p.G) * p.H;
  if (x == ex_cent(p.nl)) return p.C;
  if (x == ex_key(p.nl)) return 2LL * p.N;
  const int l = (x - 1) / 4, kind = (x - 1) % 4;
  const int t = p.ltype[l], d = p.d[t];
  if (kind == 0) return static_cast<long long>(p.nh) * d;
  if (kind == 1) return static_cast<long long>(p.A[t]) * p.nh * (d + 2);
  return static_cast<long long>(p.G) * p.H;
}

}  // namespace gr
}  // namespace mtp
