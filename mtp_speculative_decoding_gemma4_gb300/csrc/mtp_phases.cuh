// Phases of one drafter step, as device functions that loop over work items
// (item = cta; item < n_items; item += ncta). The same code runs as one kernel launch per
// phase (ncta = number of items) or inside the persistent draft-block kernel with a grid
// barrier between phases.
//
// Step structure (Gemma 4 Multi-Token Prediction (MTP) drafter, "What it is" and "Tensor
// schema"; Gemma 4 Assistant tensor inventory, "Centroid / ordered embeddings LM head"):
//   PRE    x = W_pre [h ; embed(tok)]                      (staging gathers the embed row)
//   per block l:
//     Q    a = norm(x); q = W_q a                          (staging applies the previous
//                                                           block's post-FFN residual)
//     ATT  split-KV partial softmax of each head over the shared K (V = K)
//     CMB  combine the splits -> o (attention output)
//     O    W_o o
//     GU   x += norm(W_o o); f = norm(x); gate, up = W_gate f, W_up f
//     DN   m = gelu_tanh(gate) * up; W_down m
//   HEAD1  x = lambda (x + norm(W_down m)); y = output_norm(x);
//          h' = W_post y (output + the hidden of the next step); centroid logits
// Weights, K and embeddings are read in the model dtype; every activation is fp32 and
// is never rounded to a narrower type.
//   TOPK   top_k centroids per sequence
//   GATHER sparse logits over the selected clusters' token_ordering ids + argmax
//   DENSE  (dense tied head) logits over all rows of token_embd + argmax
#pragma once

#include <cstddef>

#include "mtp_common.cuh"
#include "mtp_stage.cuh"
#include "mtp.h"

namespace mtp {

constexpr int kMaxLayers = 8;
constexpr int kBG = 8;          // largest GEMV batch group
constexpr int kGemvInBudget = 96 * 1024;  // shared-memory bytes for a batch group's inputs
constexpr int kDenseBG = 32;    // sequences per dense-head batch group
constexpr int kGatherPerItem = 32 * kWarps;  // candidates per gather item (32 per warp)
constexpr int kDenseRowsPerItem = 256;
constexpr int kCmbDims = 64;    // head dims per combine item

struct LayerP {
  const void *q, *o, *gate, *up, *down;
  const float *q_norm, *attn_norm, *post_attn_norm, *ffn_norm, *post_ffn_norm;
  float lambda;
  int type;  // 0 sliding, 1 full
};

struct KvP {
  const void* k;
  const void* v;
  const int* ctx_len;
  long long sb, st;
  int max_ctx;
  int pad_;  // explicit: Params is compared bytewise by the graph cache
};

struct ShapeP {
  int B, bb, H, nl, nh, nkv, F, V, C, topk, vsc, W, ordered;
  int d[2];
  int nsplit[2];
  float scale[2];
  float theta[2];
  float eps;
  int ncta_hint;  // CTA count the work decomposition is sized for
  int head_dd;    // sparse head cluster-major (each selected centroid's rows read once per step)
  int nsm;        // SMs of the device
  int pad_;       // explicit: Params is compared bytewise by the graph cache
};

struct WsP {
  float* x[2];                 // [B][H] residual stream, ping-pong
  float* qraw;                 // [B][nh*dmax]
  float* part_ml;              // [B][nh][nsplit_max][2]
  float* part_acc;             // [B][nh][nsplit_max][dmax]
  float* o;                    // [B][nh*dmax] attention output
  float* ao;                   // [B][H]
  float* gate;                 // [B][F]
  float* up;                   // [B][F]
  float* dn;                   // [B][H]
  float* y;                    // [B][H] final normed hidden state
  float* h_cur;                // [B][bb] hidden state of the next draft step
  float* cl;                   // [B][C]
  int* sel;                    // [B][topk]
  unsigned long long* best;    // [B]
  float* lmin;                 // [B] smallest candidate logit (the min(selected) - 1 mask)
  float2* cs;                  // [B][2][dmax/2] RoPE (cos, sin)
  unsigned int* bar;           // grid barrier counter
  int* status;                 // device status word (0 = ok)
  int nsplit_max, dmax;
};

struct Params {
  ShapeP s;
  WsP w;
  const void *pre, *post, *temb, *cent, *tgt;
  const void* temb_ord;  // token_embd rows in token_ordering order [V][H] (cluster-major head)
  const float* out_norm;
  const int* ord;
  LayerP L[kMaxLayers];
  KvP kv[2];
  const void* hidden_in;
  const int* tok_in;
  const int* pos;
  int* out_tokens;     // [B][n_draft] (draft block) or [B] (head entry)
  float* out_hidden;   // [B][n_draft][bb] or null
  int n_draft;
  int pad0_;
  const float* y_in;   // head entry: [B][H]
  float* out_logits;   // head entry: [B][V] or null
  int* out_centroids;  // head entry: [B][topk] or null
  int mask_mode;       // head entry: unselected logits -1e30 (MTP_MASK_NEG_1E30) or min - 1
  int check_ids;       // head entry: skip candidate rows whose token_ordering id is outside
                       // [0, V) (the allocation-free entry, whose ordering is not validated)
  long long spin_limit;  // bounded grid-barrier wait (clock64 cycles)
  int dbg_skip;          // testing only: CTA dbg_skip - 1 of the persistent kernel does not
                         // arrive at its first grid barrier, so that barrier times out (0: off)
  int pad1_;
  // Tensor-core path: when set, a GEMV phase only stages its inputs and writes them as three
  // bf16 terms [3][tc_bp][K_in] (hi, mid, lo of every fp32 input) for the tcgen05 GEMMs.
  __nv_bfloat16* tc_xs;
  int tc_bp;
  int pad2_;
};
// The graph cache compares whole Params objects with memcmp: no member may be followed by
// compiler padding, whose bytes a copy need not preserve.
static_assert(sizeof(KvP) == 3 * sizeof(void*) + 2 * sizeof(long long) + 2 * sizeof(int), "KvP padding");
static_assert(sizeof(ShapeP) % 8 == 0 && offsetof(Params, w) == sizeof(ShapeP), "ShapeP padding");
static_assert(offsetof(Params, y_in) == offsetof(Params, n_draft) + 8, "Params padding after n_draft");
static_assert(offsetof(Params, spin_limit) == offsetof(Params, mask_mode) + 8, "Params padding after mask_mode");
static_assert(offsetof(Params, tc_xs) == offsetof(Params, dbg_skip) + 8, "Params padding after dbg_skip");
static_assert(sizeof(Params) == offsetof(Params, tc_bp) + 8, "Params trailing padding");

// ---------------------------------------------------------------- GEMV machinery

struct GemvJob {
  const void* W;
  int R, K, ks;          // rows, columns, warps splitting K
  float* out;            // result [b*ldo + r] (may be null)
  long long ldo;
  float* out2;           // second copy [b*ld2 + r] (may be null)
  long long ld2;
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Sequences staged together by a GEMV phase whose input vectors have K_in elements.
__host__ __device__ inline int gemv_group(int B, int K_in) {
  int g = kGemvInBudget / (K_in * 4);
  g = g < 1 ? 1 : g;
  g = g < kBG ? g : kBG;
  return g < B ? g : B;
}

// Warps per row so that the phase has about ncta_hint items.
__host__ __device__ inline int choose_ks(int R, int ngroups, int ncta_hint) {
  int ks = 1;
  while (ks < kWarps && ceil_div(R * ks, kWarps) * ngroups < ncta_hint) ks *= 2;
  return ks;
}

__host__ __device__ inline int gemv_tiles(const GemvJob& j) { return ceil_div(j.R, kWarps / j.ks); }

// V consecutive fp32 values from shared memory.
template <int V>
__device__ inline void load_fvec(const float* p, float* out) {
#pragma unroll
  for (int i = 0; i < V; i += 4) {
    const float4 f = *reinterpret_cast<const float4*>(p + i);
    out[i] = f.x; out[i + 1] = f.y; out[i + 2] = f.z; out[i + 3] = f.w;
  }
}

template <typename WT>
__device__ inline void gemv_tile(const GemvJob& j, int tile, const float* in_s, int ld_in, int b0, int nb,
                                 float* red) {
  constexpr int V = Elem<WT>::kVec;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rpt = kWarps / j.ks;
  const int roff = warp / j.ks, kp = warp % j.ks;
  const int r = tile * rpt + roff;
  const int seg = ceil_div(ceil_div(j.K, j.ks), V) * V;
  const int k0 = kp * seg, k1 = min(j.K, k0 + seg);
  float acc[kBG];
#pragma unroll
  for (int b = 0; b < kBG; ++b) acc[b] = 0.f;
  if (r < j.R) {
    const WT* wr = static_cast<const WT*>(j.W) + static_cast<size_t>(r) * j.K;
    for (int k = k0 + lane * V; k < k1; k += 32 * V) {
      float w[V];
      load_vec_stream(wr + k, w);
#pragma unroll
      for (int b = 0; b < kBG; ++b) {
        if (b < nb) {
          float xv[V];
          load_fvec<V>(in_s + b * ld_in + k, xv);
#pragma unroll
          for (int v = 0; v < V; ++v) acc[b] = fmaf(w[v], xv[v], acc[b]);
        }
      }
    }
  }
#pragma unroll
  for (int b = 0; b < kBG; ++b) acc[b] = warp_sum(acc[b]);
  if (lane == 0) {
#pragma unroll
    for (int b = 0; b < kBG; ++b) red[warp * kBG + b] = acc[b];
  }
  __syncthreads();
  for (int t = threadIdx.x; t < rpt * nb; t += kThreads) {
    const int ro = t / nb, b = t % nb;
    const int row = tile * rpt + ro;
    if (row < j.R) {
      float s = 0.f;
      for (int q = 0; q < j.ks; ++q) s += red[(ro * j.ks + q) * kBG + b];
      if (j.out) j.out[(b0 + b) * j.ldo + row] = s;
      if (j.out2) j.out2[(b0 + b) * j.ld2 + row] = s;
    }
  }
  __syncthreads();
}

// Shared-memory layout of a GEMV phase: fp32 inputs [nbg][K_in], reduction scratch
// [kWarps][kBG] floats, staging scratch [2][H] floats (residual vectors).
struct GemvSmem {
  int in_bytes, red_off, scr_off, total;
};
__host__ __device__ inline GemvSmem gemv_smem(int K_in, int nbg, int max_vec) {
  GemvSmem g;
  g.in_bytes = ((nbg * K_in * 4 + 15) / 16) * 16;
  g.red_off = g.in_bytes;
  g.scr_off = g.red_off + kWarps * kBG * 4;
  g.total = g.scr_off + 2 * max_vec * 4 + 64;
  return g;
}

// Runs the GEMV jobs of one phase. `stage(b0, nb, in_s, scr, red, writer)` fills the
// inputs of a batch group; `writer` is true in exactly one CTA per group.
template <typename WT, typename Stage>
__device__ void gemv_phase(const Params& p, const GemvJob* jobs, int njobs, int K_in, Stage stage,
                           int cta, int ncta, char* smem) {
  // staging for the tensor-core GEMMs: one sequence per CTA (the most parallel split)
  const int nbg = p.tc_xs ? 1 : gemv_group(p.s.B, K_in);
  const GemvSmem L = gemv_smem(K_in, nbg, p.s.H);
  float* in_s = reinterpret_cast<float*>(smem);
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  float* scr = reinterpret_cast<float*>(smem + L.scr_off);
  const int ngroups = ceil_div(p.s.B, nbg);
  if (p.tc_xs) {
    // staging only: one CTA per batch group, inputs split into exact bf16 terms
    for (int g = cta; g < ngroups; g += ncta) {
      const int b0 = g * nbg, nb = min(nbg, p.s.B - b0);
      __syncthreads();
      stage(b0, nb, in_s, K_in, scr, red, true);
      __syncthreads();
      for (int i = threadIdx.x; i < nb * K_in; i += kThreads) {
        const int b = i / K_in, k = i % K_in;
        stage_terms(p.tc_xs, p.tc_bp, K_in, b0 + b, k, in_s[b * K_in + k]);
      }
    }
    return;
  }
  int tiles = 0;
  for (int q = 0; q < njobs; ++q) tiles += gemv_tiles(jobs[q]);
  const int n_items = ngroups * tiles;
  int staged = -1;
  for (int item = cta; item < n_items; item += ncta) {
    const int g = item / tiles;
    int t = item % tiles;
    const int b0 = g * nbg, nb = min(nbg, p.s.B - b0);
    if (g != staged) {
      __syncthreads();
      stage(b0, nb, in_s, K_in, scr, red, t == 0);
      __syncthreads();
      staged = g;
    }
    int q = 0;
    while (t >= gemv_tiles(jobs[q])) { t -= gemv_tiles(jobs[q]); ++q; }
    gemv_tile<WT>(jobs[q], t, in_s, K_in, b0, nb, red);
  }
}

// ---------------------------------------------------------------- staging helpers

// Residual update used by the post-attention / post-FFN sandwich norms:
// xs = lambda * (x + norm(v) * g). `xs` and `v_s` are shared-memory fp32 vectors.
__device__ inline void residual_update(float* xs, const float* x, float* v_s, const float* v,
                                       const float* g, float lambda, int n, float eps, float* red) {
  for (int i = threadIdx.x; i < n; i += kThreads) v_s[i] = v[i];
  __syncthreads();
  const float r = rms_factor(v_s, n, eps, red);
  for (int i = threadIdx.x; i < n; i += kThreads) xs[i] = lambda * (x[i] + v_s[i] * r * g[i]);
  __syncthreads();
}

// dst = xs * rms_factor(xs) * g (projection input; stays fp32).
__device__ inline void norm_to_input(float* dst, const float* xs, const float* g, int n, float eps, float* red) {
  const float r = rms_factor(xs, n, eps, red);
  for (int i = threadIdx.x; i < n; i += kThreads) dst[i] = xs[i] * r * g[i];
}

// n values of type T (multiple of the 16-byte vector) -> fp32 in shared memory.
template <typename T>
__device__ inline void load_to_f32(float* dst, const T* src, int n) {
  constexpr int V = Elem<T>::kVec;
  for (int i = threadIdx.x * V; i < n; i += kThreads * V) {
    float v[V];
    load_vec(src + i, v);
#pragma unroll
    for (int e = 0; e < V; ++e) dst[i + e] = v[e];
  }
}

// ---------------------------------------------------------------- PRE

template <typename WT>
__device__ void phase_pre(const Params& p, int step, int par, int cta, int ncta, char* smem) {
  const int bb = p.s.bb;
  GemvJob j{p.pre, p.s.H, 2 * bb, choose_ks(p.s.H, ceil_div(p.s.B, gemv_group(p.s.B, 2 * bb)), p.s.ncta_hint),
            p.w.x[par], p.s.H, nullptr, 0};
  auto stage = [&](int b0, int nb, float* in_s, int ld, float*, float*, bool writer) {
    for (int b = 0; b < nb; ++b) {
      const int bi = b0 + b;
      int tok = step == 0 ? p.tok_in[bi] : key_id(p.w.best[bi]);
      if (writer && step > 0 && threadIdx.x == 0) p.out_tokens[bi * p.n_draft + step - 1] = tok;
      if (tok < 0 || tok >= p.s.V) {  // an out-of-range caller token reads row 0 and is reported
        if (writer && threadIdx.x == 0) atomicExch(p.w.status, static_cast<int>(MTP_ERR_INVALID_ARG));
        tok = 0;
      }
      if (step == 0)
        load_to_f32<WT>(in_s + b * ld, static_cast<const WT*>(p.hidden_in) + static_cast<size_t>(bi) * bb, bb);
      else
        load_to_f32<float>(in_s + b * ld, p.w.h_cur + static_cast<size_t>(bi) * bb, bb);
      load_to_f32<WT>(in_s + b * ld + bb, static_cast<const WT*>(p.tgt) + static_cast<size_t>(tok) * bb, bb);
    }
  };
  gemv_phase<WT>(p, &j, 1, 2 * bb, stage, cta, ncta, smem);
}

// ---------------------------------------------------------------- Q

template <typename WT>
__device__ void phase_q(const Params& p, int l, int par, int cta, int ncta, char* smem) {
  const LayerP& L = p.L[l];
  const int d = p.s.d[L.type], H = p.s.H;
  GemvJob j{L.q, p.s.nh * d, H, choose_ks(p.s.nh * d, ceil_div(p.s.B, gemv_group(p.s.B, H)), p.s.ncta_hint),
            p.w.qraw, static_cast<long long>(p.s.nh) * p.w.dmax, nullptr, 0};
  auto stage = [&](int b0, int nb, float* in_s, int ld, float* scr, float* red, bool writer) {
    float* xs = scr;
    float* vs = scr + p.s.H;
    for (int b = 0; b < nb; ++b) {
      const int bi = b0 + b;
      const float* x = p.w.x[par] + static_cast<size_t>(bi) * H;
      if (l == 0) {
        for (int i = threadIdx.x; i < H; i += kThreads) xs[i] = x[i];
        __syncthreads();
        if (writer && threadIdx.x == 0) p.w.best[bi] = 0ull;
      } else {
        const LayerP& P = p.L[l - 1];
        residual_update(xs, x, vs, p.w.dn + static_cast<size_t>(bi) * H, P.post_ffn_norm, P.lambda, H,
                        p.s.eps, red);
        if (writer)
          for (int i = threadIdx.x; i < H; i += kThreads) p.w.x[par ^ 1][static_cast<size_t>(bi) * H + i] = xs[i];
      }
      norm_to_input(in_s + b * ld, xs, L.attn_norm, H, p.s.eps, red);
      __syncthreads();
    }
  };
  gemv_phase<WT>(p, &j, 1, H, stage, cta, ncta, smem);
}

// ---------------------------------------------------------------- ATT

// Warp geometry of the attention phase for head dim D, HPG query heads per KV head and
// model dtype WT. One warp owns one (sequence, KV head, split) item and walks its keys in
// blocks of KB. Every lane owns NVEC 16-byte vectors of a key row (LPK lanes cover one row,
// KPL rows sit side by side in the warp); each lane streams R rows per block into a private
// shared-memory ring with cp.async, so nothing of the block waits on another lane.
template <typename WT, int D, int HPG>
struct AttGeom {
  static constexpr int VE = 16 / static_cast<int>(sizeof(WT));  // elements per 16-byte vector
  static constexpr int VPK = D / VE;                             // vectors per key row
  static constexpr int LPK0 = VPK < 32 ? VPK : 32;
  static constexpr int LPK = LPK0 < HPG ? HPG : LPK0;            // lanes per row (>= HPG)
  static constexpr int NVEC = VPK > LPK ? VPK / LPK : 1;         // vectors per lane per row
  static constexpr int KPL = 32 / LPK;                           // rows per warp load
  static constexpr int RA = LPK / HPG, RB = 8 / NVEC;
  static constexpr int R = RA < RB ? RA : RB;                    // rows per lane per block
  static constexpr int KB = R * KPL;                             // keys per block
  static constexpr int NVAL = R * HPG;                           // (row, head) scores per lane group
  static constexpr int DUP = LPK / NVAL;                         // lanes holding the same score
  static constexpr int S = 3;                                    // ring stages (2 blocks ahead)
  static constexpr int kStageBytes = R * NVEC * 32 * 16;
  static constexpr int kWarpBytes = S * kStageBytes;
  static_assert(VPK >= 1 && (VPK & (VPK - 1)) == 0, "head dim must be a power-of-two multiple of a vector");
  static_assert(R >= 1 && NVAL <= LPK, "one score per lane group");
};

// Reduce-scatter over the lanes `O, O/2, .., 1` apart: N values per lane in, and lane i ends
// with the full sum of value (i mod 2*O) / (2*O / N) in v[0] (the halving steps come first).
template <int N, int O>
__device__ __forceinline__ void reduce_scatter(float* v, int lane) {
  if constexpr (O > 0) {
    if constexpr (N > 1) {
      constexpr int h = N / 2;
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < h; ++i) {
        const float send = up ? v[i] : v[i + h];
        const float keep = up ? v[i + h] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      reduce_scatter<h, O / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      reduce_scatter<1, O / 2>(v, lane);
    }
  }
}

__device__ __forceinline__ void cp_async16(unsigned dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void vec_to_f32(const uint4& u, float* out) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}
// One staged 16-byte vector of a K row from the ring as fp32 (zeros on lanes without dims).
template <typename WT, int VE>
__device__ __forceinline__ void ld_row_vec(bool has, unsigned addr, float* out) {
  if (!has) {
#pragma unroll
    for (int e = 0; e < VE; ++e) out[e] = 0.f;
    return;
  }
  uint4 u;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w) : "r"(addr));
  if constexpr (sizeof(WT) == 2) {
    vec_to_f32(u, out);
  } else {
    out[0] = __uint_as_float(u.x);
    out[1] = __uint_as_float(u.y);
    out[2] = __uint_as_float(u.z);
    out[3] = __uint_as_float(u.w);
  }
}

// Split-KV attention partials of one (sequence b, KV head g, split c) item, run by one warp.
// The HPG query heads of the group read the same K rows; V = K unless a separate V is given.
// Writes, per head, the unnormalised sum of p_j v_j over the split's keys with the running
// max m and the sum of p_j (Gemma 4 MTP drafter, "What it is": the drafter's queries attend
// the target's shared K, values equal to the keys).
template <typename WT, int D, int HPG>
__device__ void att_warp_item(const Params& p, int l, int b, int g, int c, char* wsm) {
  using G = AttGeom<WT, D, HPG>;
  constexpr int VE = G::VE, LPK = G::LPK, NVEC = G::NVEC, R = G::R, KB = G::KB, NVAL = G::NVAL,
                DUP = G::DUP, S = G::S;
  constexpr int QE = NVEC * VE;  // head dims a lane owns
  const LayerP& L = p.L[l];
  const int t = L.type;
  const KvP& kv = p.kv[t];
  const int lane = threadIdx.x & 31;
  const int dg = lane % LPK, ks = lane / LPK;
  // lanes past the row hold no dims (only when HPG exceeds the vectors of a row)
  const bool has = G::VPK >= LPK || dg < G::VPK;
  const int half = D / 2;

  // q heads of the group: q_norm, then RoPE at the constant position, for the dims this lane
  // owns: dims (dg + v*LPK)*VE + e.
  float q[HPG][QE];
  {
    const float2* cs = p.w.cs + (static_cast<size_t>(b) * 2 + t) * (p.w.dmax / 2);
#pragma unroll
    for (int hh = 0; hh < HPG; ++hh) {
      const float* qr = p.w.qraw + static_cast<size_t>(b) * p.s.nh * p.w.dmax + static_cast<size_t>(g * HPG + hh) * D;
      float ss = 0.f;
#pragma unroll
      for (int v = 0; v < NVEC; ++v)
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const float x = has ? qr[(dg + v * LPK) * VE + e] : 0.f;
          ss = fmaf(x, x, ss);
        }
#pragma unroll
      for (int o = LPK / 2; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float rf = rsqrtf(ss / D + p.s.eps);
#pragma unroll
      for (int v = 0; v < NVEC; ++v)
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const int i = (dg + v * LPK) * VE + e;
          float out = 0.f;
          if (has) {
            const int ip = i < half ? i + half : i - half;  // RoPE partner
            const float a = qr[i] * rf * L.q_norm[i];
            const float bq = qr[ip] * rf * L.q_norm[ip];
            const float2 r = cs[i < half ? i : ip];
            out = i < half ? a * r.x - bq * r.y : a * r.x + bq * r.y;
          }
          q[hh][v * VE + e] = out;
        }
    }
  }

  const int Lb = min(max(kv.ctx_len[b], 0), kv.max_ctx);  // never read past the buffer
  const int lo = t == 0 ? max(0, Lb - p.s.W) : 0, hi = Lb;
  const int nsp = p.s.nsplit[t];
  const int chunk = ceil_div(max(hi - lo, 0), nsp);
  const int j0 = lo + c * chunk, j1 = min(hi, j0 + chunk);
  const float scale = p.s.scale[t];
  const int nblk = j1 > j0 ? ceil_div(j1 - j0, KB) : 0;

  const WT* kb = static_cast<const WT*>(kv.k) + static_cast<size_t>(b) * kv.sb + static_cast<size_t>(g) * D;
  const WT* vb = kv.v ? static_cast<const WT*>(kv.v) + static_cast<size_t>(b) * kv.sb + static_cast<size_t>(g) * D
                      : nullptr;
  const unsigned ring = static_cast<unsigned>(__cvta_generic_to_shared(wsm));
  // block i -> stage i % S: rows ks*R + r of the block, this lane's vectors
  auto issue = [&](int i) {
    if (i < nblk && has) {
      const int st = i % S;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int key = j0 + i * KB + ks * R + r;
        const bool ok = key < j1;
        const WT* row = kb + static_cast<size_t>(ok ? key : j0) * kv.st;
#pragma unroll
        for (int v = 0; v < NVEC; ++v)
          cp_async16(ring + (((st * R + r) * NVEC + v) * 32 + lane) * 16, row + (dg + v * LPK) * VE, ok ? 16 : 0);
      }
    }
    cp_async_commit();  // one group per block index, empty or not
  };

  // score index of this lane after the reduce-scatter: head my_h, row my_r of its sub-slot
  const int my_idx = (lane % LPK) / DUP;
  const int my_h = my_idx / R, my_r = my_idx % R;
  float m[HPG], acc[HPG][QE];
#pragma unroll
  for (int hh = 0; hh < HPG; ++hh) {
    m[hh] = -INFINITY;
#pragma unroll
    for (int e = 0; e < QE; ++e) acc[hh][e] = 0.f;
  }
  float lsum = 0.f;  // sum of p over this lane's (head, row) scores

#pragma unroll
  for (int i = 0; i < S - 1; ++i) issue(i);
  for (int i = 0; i < nblk; ++i) {
    issue(i + S - 1);
    cp_async_wait<S - 1>();
    const unsigned stage = ring + (i % S) * (R * NVEC * 32 * 16);
    const int base = j0 + i * KB;
    // scores of (head, row) pairs, partial over this lane's dims
    float sc[NVAL];
#pragma unroll
    for (int n = 0; n < NVAL; ++n) sc[n] = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int v = 0; v < NVEC; ++v) {
        float kf[VE];
        ld_row_vec<WT, VE>(has, stage + ((r * NVEC + v) * 32 + lane) * 16, kf);
#pragma unroll
        for (int hh = 0; hh < HPG; ++hh)
#pragma unroll
          for (int e = 0; e < VE; ++e) sc[hh * R + r] = fmaf(q[hh][v * VE + e], kf[e], sc[hh * R + r]);
      }
    reduce_scatter<NVAL, LPK / 2>(sc, lane);
    float s = sc[0] * scale;
    if (base + ks * R + my_r >= j1) s = -INFINITY;
    // block max of each head: over its rows, its duplicate lanes and the sub-slots
    float bm = s;
#pragma unroll
    for (int o = 1; o < R * DUP; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
    float corr[HPG], m_me = 0.f, corr_me = 0.f;
#pragma unroll
    for (int hh = 0; hh < HPG; ++hh) {
      const float mn = fmaxf(m[hh], __shfl_sync(0xffffffffu, bm, hh * R * DUP));
      corr[hh] = expf(m[hh] - mn);  // 0 on the first block (m = -inf, mn finite)
      m[hh] = mn;
      if (hh == my_h) {
        m_me = mn;
        corr_me = corr[hh];
      }
    }
    const float pw = expf(s - m_me);  // 0 for keys past the split
    lsum = lsum * corr_me + pw;
#pragma unroll
    for (int hh = 0; hh < HPG; ++hh)
#pragma unroll
      for (int e = 0; e < QE; ++e) acc[hh][e] *= corr[hh];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float pr[HPG];
#pragma unroll
      for (int hh = 0; hh < HPG; ++hh) pr[hh] = __shfl_sync(0xffffffffu, pw, ks * LPK + (hh * R + r) * DUP);
      const int key = base + ks * R + r;
#pragma unroll
      for (int v = 0; v < NVEC; ++v) {
        float kf[VE];
        if (vb) {
          if (has && key < j1)
            load_vec(vb + static_cast<size_t>(key) * kv.st + (dg + v * LPK) * VE, kf);
          else
#pragma unroll
            for (int e = 0; e < VE; ++e) kf[e] = 0.f;
        } else {
          ld_row_vec<WT, VE>(has, stage + ((r * NVEC + v) * 32 + lane) * 16, kf);
        }
#pragma unroll
        for (int hh = 0; hh < HPG; ++hh)
#pragma unroll
          for (int e = 0; e < VE; ++e) acc[hh][v * VE + e] = fmaf(pr[hh], kf[e], acc[hh][v * VE + e]);
      }
    }
  }
  cp_async_wait<0>();

  // sub-slots hold disjoint rows of the same dims: add them up
#pragma unroll
  for (int o = LPK; o < 32; o <<= 1)
#pragma unroll
    for (int hh = 0; hh < HPG; ++hh)
#pragma unroll
      for (int e = 0; e < QE; ++e) acc[hh][e] += __shfl_xor_sync(0xffffffffu, acc[hh][e], o);
  const bool first_dup = (lane % LPK) % DUP == 0;
#pragma unroll
  for (int hh = 0; hh < HPG; ++hh) {
    const float den = warp_sum(first_dup && my_h == hh ? lsum : 0.f);
    const size_t slot = (static_cast<size_t>(b) * p.s.nh + g * HPG + hh) * p.w.nsplit_max + c;
    if (ks == 0 && has) {
      float* dst = p.w.part_acc + slot * p.w.dmax;
#pragma unroll
      for (int v = 0; v < NVEC; ++v)
#pragma unroll
        for (int e = 0; e < VE; e += 4)
          *reinterpret_cast<float4*>(dst + (dg + v * LPK) * VE + e) =
              make_float4(acc[hh][v * VE + e], acc[hh][v * VE + e + 1], acc[hh][v * VE + e + 2], acc[hh][v * VE + e + 3]);
    }
    if (lane == 0) {
      p.w.part_ml[slot * 2] = m[hh];
      p.w.part_ml[slot * 2 + 1] = den;
    }
  }
}

#define MTP_ATT_CASES                                                                       \
  MTP_ATT_CASE(32, 1) MTP_ATT_CASE(32, 2) MTP_ATT_CASE(32, 4) MTP_ATT_CASE(32, 8)           \
  MTP_ATT_CASE(64, 1) MTP_ATT_CASE(64, 2) MTP_ATT_CASE(64, 4) MTP_ATT_CASE(64, 8)           \
  MTP_ATT_CASE(128, 1) MTP_ATT_CASE(128, 2) MTP_ATT_CASE(128, 4) MTP_ATT_CASE(128, 8)       \
  MTP_ATT_CASE(256, 1) MTP_ATT_CASE(256, 2) MTP_ATT_CASE(256, 4) MTP_ATT_CASE(256, 8)       \
  MTP_ATT_CASE(512, 1) MTP_ATT_CASE(512, 2) MTP_ATT_CASE(512, 4)

// Shared memory of the attention phase: one cp.async ring per warp (0: unsupported shape).
template <typename WT>
__host__ __device__ inline int att_smem_bytes(int D, int HPG) {
#define MTP_ATT_CASE(DD, HH) \
  if (D == DD && HPG == HH) return kWarps * AttGeom<WT, DD, HH>::kWarpBytes;
  MTP_ATT_CASES
#undef MTP_ATT_CASE
  return 0;
}

template <typename WT, int D, int HPG>
__device__ void att_phase_t(const Params& p, int l, int cta, int ncta, char* smem) {
  const int t = p.L[l].type;
  const int nsp = p.s.nsplit[t];
  const int n_items = p.s.B * p.s.nkv * nsp;
  const int warp = threadIdx.x >> 5;
  char* wsm = smem + warp * AttGeom<WT, D, HPG>::kWarpBytes;
  for (int item = cta * kWarps + warp; item < n_items; item += ncta * kWarps) {
    const int c = item % nsp;
    const int g = (item / nsp) % p.s.nkv;
    const int b = item / (nsp * p.s.nkv);
    att_warp_item<WT, D, HPG>(p, l, b, g, c, wsm);
  }
}

// Items of the attention phase are warps: B * n_kv_head * nsplit of them.
template <typename WT>
__device__ void phase_att(const Params& p, int l, int cta, int ncta, char* smem) {
  const int D = p.s.d[p.L[l].type];
  const int hpg = p.s.nh / p.s.nkv;
#define MTP_ATT_CASE(DD, HH) \
  if (D == DD && hpg == HH) { att_phase_t<WT, DD, HH>(p, l, cta, ncta, smem); return; }
  MTP_ATT_CASES
#undef MTP_ATT_CASE
}

// ---------------------------------------------------------------- CMB

template <typename WT>
__device__ void phase_cmb(const Params& p, int l, int cta, int ncta, char* smem) {
  const int t = p.L[l].type;
  const int D = p.s.d[t], nsp = p.s.nsplit[t];
  const int ndc = ceil_div(D, kCmbDims);
  const int n_items = p.s.B * p.s.nh * ndc;
  constexpr int kGroups = kThreads / kCmbDims;
  float* sm = reinterpret_cast<float*>(smem);        // [kGroups][kCmbDims] num, then den
  for (int item = cta; item < n_items; item += ncta) {
    const int dc = item % ndc;
    const int h = (item / ndc) % p.s.nh;
    const int b = item / (ndc * p.s.nh);
    const size_t base = (static_cast<size_t>(b) * p.s.nh + h) * p.w.nsplit_max;
    float M = -INFINITY;
    for (int c = 0; c < nsp; ++c) M = fmaxf(M, p.w.part_ml[(base + c) * 2]);
    const int i = dc * kCmbDims + (threadIdx.x % kCmbDims);
    const int grp = threadIdx.x / kCmbDims;
    float num = 0.f, den = 0.f;
    if (M != -INFINITY && i < D) {
      for (int c = grp; c < nsp; c += kGroups) {
        const float f = expf(p.w.part_ml[(base + c) * 2] - M);
        num += f * p.w.part_acc[(base + c) * p.w.dmax + i];
        den += f * p.w.part_ml[(base + c) * 2 + 1];
      }
    }
    sm[grp * kCmbDims + (threadIdx.x % kCmbDims)] = num;
    sm[(kGroups + grp) * kCmbDims + (threadIdx.x % kCmbDims)] = den;
    __syncthreads();
    if (grp == 0 && i < D) {
      float n = 0.f, dd = 0.f;
      for (int q = 0; q < kGroups; ++q) {
        n += sm[q * kCmbDims + threadIdx.x];
        dd += sm[(kGroups + q) * kCmbDims + threadIdx.x];
      }
      const float o = dd > 0.f ? n / dd : 0.f;
      if (p.tc_xs)  // tensor-core path: straight into the O projection's staged operand
        stage_terms(p.tc_xs, p.tc_bp, p.s.nh * D, b, h * D + i, o);
      else
        p.w.o[(static_cast<size_t>(b) * p.s.nh + h) * D + i] = o;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- O

template <typename WT>
__device__ void phase_o(const Params& p, int l, int cta, int ncta, char* smem) {
  const LayerP& L = p.L[l];
  const int K = p.s.nh * p.s.d[L.type];
  GemvJob j{L.o, p.s.H, K, choose_ks(p.s.H, ceil_div(p.s.B, gemv_group(p.s.B, K)), p.s.ncta_hint), p.w.ao,
            p.s.H, nullptr, 0};
  auto stage = [&](int b0, int nb, float* in_s, int ld, float*, float*, bool) {
    for (int b = 0; b < nb; ++b) load_to_f32<float>(in_s + b * ld, p.w.o + static_cast<size_t>(b0 + b) * K, K);
  };
  gemv_phase<WT>(p, &j, 1, K, stage, cta, ncta, smem);
}

// ---------------------------------------------------------------- GU

template <typename WT>
__device__ void phase_gu(const Params& p, int l, int par, int cta, int ncta, char* smem) {
  const LayerP& L = p.L[l];
  const int H = p.s.H, F = p.s.F;
  const int ks = choose_ks(2 * F, ceil_div(p.s.B, gemv_group(p.s.B, H)), p.s.ncta_hint);
  GemvJob j[2] = {{L.gate, F, H, ks, p.w.gate, F, nullptr, 0}, {L.up, F, H, ks, p.w.up, F, nullptr, 0}};
  auto stage = [&](int b0, int nb, float* in_s, int ld, float* scr, float* red, bool writer) {
    float* xs = scr;
    float* vs = scr + p.s.H;
    for (int b = 0; b < nb; ++b) {
      const int bi = b0 + b;
      residual_update(xs, p.w.x[par] + static_cast<size_t>(bi) * H, vs, p.w.ao + static_cast<size_t>(bi) * H,
                      L.post_attn_norm, 1.0f, H, p.s.eps, red);
      if (writer)
        for (int i = threadIdx.x; i < H; i += kThreads) p.w.x[par ^ 1][static_cast<size_t>(bi) * H + i] = xs[i];
      norm_to_input(in_s + b * ld, xs, L.ffn_norm, H, p.s.eps, red);
      __syncthreads();
    }
  };
  gemv_phase<WT>(p, j, 2, H, stage, cta, ncta, smem);
}

// ---------------------------------------------------------------- DN

template <typename WT>
__device__ void phase_dn(const Params& p, int l, int cta, int ncta, char* smem) {
  const LayerP& L = p.L[l];
  const int H = p.s.H, F = p.s.F;
  GemvJob j{L.down, H, F, choose_ks(H, ceil_div(p.s.B, gemv_group(p.s.B, F)), p.s.ncta_hint), p.w.dn, H, nullptr,
            0};
  auto stage = [&](int b0, int nb, float* in_s, int ld, float*, float*, bool) {
    for (int b = 0; b < nb; ++b) {
      const float* gt = p.w.gate + static_cast<size_t>(b0 + b) * F;
      const float* up = p.w.up + static_cast<size_t>(b0 + b) * F;
      for (int i = threadIdx.x; i < F; i += kThreads) in_s[b * ld + i] = gelu_tanh(gt[i]) * up[i];
    }
  };
  gemv_phase<WT>(p, &j, 1, F, stage, cta, ncta, smem);
}

// ---------------------------------------------------------------- HEAD1

template <typename WT>
__device__ void phase_head1(const Params& p, int step, int par, int cta, int ncta, char* smem) {
  const int H = p.s.H, bb = p.s.bb;
  const int ngroups = ceil_div(p.s.B, gemv_group(p.s.B, H));
  const int rows = bb + (p.s.ordered ? p.s.C : 0);
  const int ks = choose_ks(rows, ngroups, p.s.ncta_hint);
  float* hout = p.out_hidden ? p.out_hidden + static_cast<size_t>(step) * bb : nullptr;
  const long long ldo = static_cast<long long>(p.n_draft) * bb;
  GemvJob j[2] = {{p.post, bb, H, ks, hout, ldo, p.w.h_cur, bb}, {p.cent, p.s.C, H, ks, p.w.cl, p.s.C, nullptr, 0}};
  const LayerP& P = p.L[p.s.nl - 1];
  auto stage = [&](int b0, int nb, float* in_s, int ld, float* scr, float* red, bool writer) {
    float* xs = scr;
    float* vs = scr + p.s.H;
    for (int b = 0; b < nb; ++b) {
      const int bi = b0 + b;
      residual_update(xs, p.w.x[par] + static_cast<size_t>(bi) * H, vs, p.w.dn + static_cast<size_t>(bi) * H,
                      P.post_ffn_norm, P.lambda, H, p.s.eps, red);
      norm_to_input(in_s + b * ld, xs, p.out_norm, H, p.s.eps, red);
      __syncthreads();
      if (writer)
        for (int i = threadIdx.x; i < H; i += kThreads) p.w.y[static_cast<size_t>(bi) * H + i] = in_s[b * ld + i];
    }
  };
  gemv_phase<WT>(p, j, p.s.ordered ? 2 : 1, H, stage, cta, ncta, smem);
}

// Head entry point: y given by the caller; only the centroid logits are computed here.
template <typename WT>
__device__ void phase_head_entry(const Params& p, int cta, int ncta, char* smem) {
  const int H = p.s.H;
  const int nbg = gemv_group(p.s.B, H);
  const int ngroups = ceil_div(p.s.B, nbg);
  GemvJob j{p.cent, p.s.C, H, choose_ks(p.s.C, ngroups, p.s.ncta_hint), p.w.cl, p.s.C, nullptr, 0};
  auto stage = [&](int b0, int nb, float* in_s, int ld, float*, float*, bool writer) {
    for (int b = 0; b < nb; ++b) {
      const int bi = b0 + b;
      for (int i = threadIdx.x; i < H; i += kThreads) {
        const float v = p.y_in[static_cast<size_t>(bi) * H + i];
        in_s[b * ld + i] = v;
        if (writer) p.w.y[static_cast<size_t>(bi) * H + i] = v;
      }
      if (writer && threadIdx.x == 0) p.w.best[bi] = 0ull;
    }
  };
  if (p.s.ordered) {
    gemv_phase<WT>(p, &j, 1, H, stage, cta, ncta, smem);
  } else {
    // dense head: only stage y (one CTA per group writes it)
    float* in_s = reinterpret_cast<float*>(smem);
    for (int g = cta; g < ngroups; g += ncta) {
      const int b0 = g * nbg, nb = min(nbg, p.s.B - b0);
      stage(b0, nb, in_s, H, nullptr, nullptr, true);
    }
  }
}

// ---------------------------------------------------------------- TOPK

// One in-lane compare-exchange stage (partner slot j + S) of the warp sort below.
template <int P, int S>
__device__ __forceinline__ void sort_stage_lane(unsigned long long (&v)[P], int lane, int size) {
#pragma unroll
  for (int j = 0; j < P; ++j) {
    if ((j & S) == 0) {
      const bool desc = ((lane * P + j) & size) == 0;
      const unsigned long long a = v[j], c = v[j + S];
      if ((a < c) == desc) {
        v[j] = c;
        v[j + S] = a;
      }
    }
  }
}

// Bitonic sort of the 32*P keys of a warp, descending; key lane*P + j sits in v[j] of `lane`.
// The stage loops stay rolled (a compact kernel); only the per-slot work is unrolled.
template <int P>
__device__ __forceinline__ void warp_sort_desc(unsigned long long (&v)[P], int lane) {
  static_assert(P == 1 || P == 2 || P == 4 || P == 8, "slots per lane");
#pragma unroll 1
  for (int size = 2; size <= 32 * P; size <<= 1) {
#pragma unroll 1
    for (int stride = size / 2; stride > 0; stride >>= 1) {
      if (stride >= P) {  // partner in lane ^ (stride / P), same slot
        const bool upper = (lane & (stride / P)) != 0;
#pragma unroll
        for (int j = 0; j < P; ++j) {
          const bool desc = ((lane * P + j) & size) == 0;
          const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[j], stride / P);
          const bool keep_max = desc != upper;
          v[j] = keep_max ? (o > v[j] ? o : v[j]) : (o < v[j] ? o : v[j]);
        }
      } else if constexpr (P > 1) {  // partner in the same lane
        if (P > 4 && stride == 4) sort_stage_lane<P, (P > 4 ? 4 : 1)>(v, lane, size);
        else if (P > 2 && stride == 2) sort_stage_lane<P, (P > 2 ? 2 : 1)>(v, lane, size);
        else sort_stage_lane<P, 1>(v, lane, size);
      }
    }
  }
}

constexpr int kTopkP = 8, kTopkChunk = 32 * kTopkP;  // keys per warp sort
__host__ __device__ inline int topk_keep(int k) {
  int t = 1;
  while (t < k) t <<= 1;
  return t;
}
__host__ __device__ inline int topk_smem_bytes(int C, int k) {
  return 2 * ((C + kTopkChunk - 1) / kTopkChunk) * topk_keep(k) * 8;
}

// Top-k centroids of one sequence, best first: every warp sorts chunks of 256 (value, index)
// keys in registers and keeps each chunk's best T (the power of two >= k); the kept lists
// are reduced the same way until one chunk is left, whose first k keys are the answer.
template <typename WT>
__device__ void phase_topk(const Params& p, int cta, int ncta, char* smem) {
  constexpr int P = kTopkP, CH = kTopkChunk;
  const int C = p.s.C, k = p.s.topk, T = topk_keep(k);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch1 = ceil_div(C, CH);
  unsigned long long* la = reinterpret_cast<unsigned long long*>(smem);  // [nch1 * T]
  unsigned long long* lb = la + nch1 * T;                                 // [nch1 * T]
  for (int b = cta; b < p.s.B; b += ncta) {
    const float* cl = p.w.cl + static_cast<size_t>(b) * C;
    for (int ch = warp; ch < nch1; ch += kWarps) {
      unsigned long long v[P];
#pragma unroll
      for (int j = 0; j < P; ++j) {
        const int i = ch * CH + lane * P + j;
        v[j] = i < C ? argmax_key(cl[i], i) : 0ull;
      }
      warp_sort_desc<P>(v, lane);
#pragma unroll
      for (int j = 0; j < P; ++j)
        if (lane * P + j < T) la[ch * T + lane * P + j] = v[j];
    }
    __syncthreads();
    unsigned long long *src = la, *dst = lb;
    int m = nch1 * T;
    while (m > CH) {
      const int nch = ceil_div(m, CH);
      for (int ch = warp; ch < nch; ch += kWarps) {
        unsigned long long v[P];
#pragma unroll
        for (int j = 0; j < P; ++j) {
          const int i = ch * CH + lane * P + j;
          v[j] = i < m ? src[i] : 0ull;
        }
        warp_sort_desc<P>(v, lane);
#pragma unroll
        for (int j = 0; j < P; ++j)
          if (lane * P + j < T) dst[ch * T + lane * P + j] = v[j];
      }
      __syncthreads();
      m = nch * T;
      unsigned long long* t = src;
      src = dst;
      dst = t;
    }
    if (warp == 0) {
      unsigned long long v[P];
#pragma unroll
      for (int j = 0; j < P; ++j) {
        const int i = lane * P + j;
        v[j] = i < m ? src[i] : 0ull;
      }
      warp_sort_desc<P>(v, lane);
#pragma unroll
      for (int j = 0; j < P; ++j) {
        const int i = lane * P + j;
        if (i < k) {
          const int id = key_id(v[j]);
          p.w.sel[b * k + i] = id;
          if (p.out_centroids) p.out_centroids[b * k + i] = id;
        }
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- GATHER

// Sparse logits over the selected clusters' candidates (ids from token_ordering) and their
// argmax. A warp scores 32 candidates: lane i fetches candidate i's id, every lane reads its
// slice of all 32 rows (loads of several rows in flight), and a reduce-scatter leaves row
// i's logit in lane i.
template <typename WT>
__device__ void phase_gather(const Params& p, int cta, int ncta, char* smem) {
  constexpr int V = Elem<WT>::kVec;
  constexpr int kRowsInFlight = 8;
  const int H = p.s.H, vsc = p.s.vsc;
  const int ncand = p.s.topk * vsc;
  const int per_b = ceil_div(ncand, kGatherPerItem);
  const int n_items = p.s.B * per_b;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* ys = reinterpret_cast<float*>(smem);                         // [H]
  unsigned long long* wbest = reinterpret_cast<unsigned long long*>(ys + H + 2);  // [kWarps]
  int staged = -1;
  for (int item = cta; item < n_items; item += ncta) {
    const int b = item / per_b, ci = item % per_b;
    if (b != staged) {
      __syncthreads();
      for (int i = threadIdx.x; i < H; i += kThreads) ys[i] = p.w.y[static_cast<size_t>(b) * H + i];
      __syncthreads();
      staged = b;
    }
    unsigned long long best = 0ull;
    const int c0 = ci * kGatherPerItem + warp * 32;
    if (c0 < ncand) {
      const int cand = c0 + lane;
      const bool valid = cand < ncand;
      const int cc = valid ? cand : c0;  // rows past the end re-read the first one
      const int cent = p.w.sel[b * p.s.topk + cc / vsc];
      const int id_raw = p.ord[cent * vsc + cc % vsc];
      // the allocation-free entry does not validate the ordering: an id outside [0, V) is
      // skipped (row 0 is read in its place and its logit discarded)
      const bool id_ok = !p.check_ids || static_cast<unsigned>(id_raw) < static_cast<unsigned>(p.s.V);
      const int id = id_ok ? id_raw : 0;
      float sc[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) sc[r] = 0.f;
#pragma unroll
      for (int r0 = 0; r0 < 32; r0 += kRowsInFlight) {
        const WT* rows[kRowsInFlight];
#pragma unroll
        for (int rr = 0; rr < kRowsInFlight; ++rr)
          rows[rr] = static_cast<const WT*>(p.temb) + static_cast<size_t>(__shfl_sync(0xffffffffu, id, r0 + rr)) * H;
        for (int k = lane * V; k < H; k += 32 * V) {
          float w[kRowsInFlight][V];
#pragma unroll
          for (int rr = 0; rr < kRowsInFlight; ++rr) load_vec_stream(rows[rr] + k, w[rr]);
#pragma unroll
          for (int rr = 0; rr < kRowsInFlight; ++rr)
#pragma unroll
            for (int v = 0; v < V; ++v) sc[r0 + rr] = fmaf(w[rr][v], ys[k + v], sc[r0 + rr]);
        }
      }
      reduce_scatter<32, 16>(sc, lane);  // lane i: the logit of candidate c0 + i
      if (valid && id_ok) {
        if (p.out_logits) p.out_logits[static_cast<size_t>(b) * p.s.V + id] = sc[0];
        best = argmax_key(sc[0], id);
      }
      best = warp_max_u64(best);
    }
    if (lane == 0) wbest[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kWarps; ++w) m = wbest[w] > m ? wbest[w] : m;
      atomicMax(&p.w.best[b], m);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- MASK (min(selected) - 1)

// Smallest logit among each sequence's candidates (the entries the gather scattered into its
// materialised row), for the mask variant that fills the other entries with that minus one
// ("Gemma 4 Assistant 使用指南" section 五, use_ordered_embeddings step 3; the -1e30 fill
// of "Gemma 4 Assistant tensor inventory", "Centroid / ordered embeddings LM head" step 5,
// names it as the MLX alternative).
template <typename WT>
__device__ void phase_cand_min(const Params& p, int cta, int ncta, char* smem) {
  const int vsc = p.s.vsc, k = p.s.topk, ncand = k * vsc;
  float* red = reinterpret_cast<float*>(smem);  // [kWarps]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int b = cta; b < p.s.B; b += ncta) {
    float m = INFINITY;
    for (int c = threadIdx.x; c < ncand; c += kThreads) {
      const int cent = p.w.sel[b * k + c / vsc];
      const int id = p.ord[cent * vsc + c % vsc];
      m = fminf(m, p.out_logits[static_cast<size_t>(b) * p.s.V + id]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fminf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float mm = red[0];
      for (int w = 1; w < kWarps; ++w) mm = fminf(mm, red[w]);
      p.w.lmin[b] = mm;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- DENSE

// Dense tied head: all V logits of up to 32 sequences per pass; lane b ends a row with the
// logit of sequence b (transposing butterfly reduction) and keeps its running argmax.
template <typename WT>
__device__ void phase_dense(const Params& p, int cta, int ncta, char* smem) {
  constexpr int V = Elem<WT>::kVec;
  const int H = p.s.H;
  const int ngroups = ceil_div(p.s.B, kDenseBG);
  const int row_items = ceil_div(p.s.V, kDenseRowsPerItem);
  const int n_items = ngroups * row_items;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* ys = reinterpret_cast<float*>(smem);  // [kDenseBG][H]
  unsigned long long* wbest = reinterpret_cast<unsigned long long*>(smem + kDenseBG * H * 4);
  int staged = -1;
  for (int item = cta; item < n_items; item += ncta) {
    const int g = item / row_items, ri = item % row_items;
    const int b0 = g * kDenseBG, nb = min(kDenseBG, p.s.B - b0);
    if (g != staged) {
      __syncthreads();
      for (int i = threadIdx.x; i < kDenseBG * H; i += kThreads) {
        const int b = i / H;
        ys[i] = b < nb ? p.w.y[static_cast<size_t>(b0 + b) * H + (i % H)] : 0.f;
      }
      __syncthreads();
      staged = g;
    }
    unsigned long long best = 0ull;
    const int r0 = ri * kDenseRowsPerItem;
    for (int rr = warp; rr < kDenseRowsPerItem; rr += kWarps) {
      const int row = r0 + rr;
      if (row >= p.s.V) break;
      const WT* wr = static_cast<const WT*>(p.temb) + static_cast<size_t>(row) * H;
      float acc[kDenseBG];
#pragma unroll
      for (int b = 0; b < kDenseBG; ++b) acc[b] = 0.f;
      for (int k = lane * V; k < H; k += 32 * V) {
        float w[V];
        load_vec_stream(wr + k, w);
#pragma unroll
        for (int b = 0; b < kDenseBG; ++b) {
          float yv[V];
          load_fvec<V>(ys + b * H + k, yv);
#pragma unroll
          for (int v = 0; v < V; ++v) acc[b] = fmaf(w[v], yv[v], acc[b]);
        }
      }
      // transposing butterfly: after it, acc[0] of lane l is the row's logit for sequence l
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
          const float send = upper ? acc[i] : acc[i + off];
          const float keep = upper ? acc[i + off] : acc[i];
          acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      if (lane < nb) {
        if (p.out_logits) p.out_logits[static_cast<size_t>(b0 + lane) * p.s.V + row] = acc[0];
        const unsigned long long key = argmax_key(acc[0], row);
        best = key > best ? key : best;
      }
    }
    wbest[warp * 32 + lane] = best;
    __syncthreads();
    if (threadIdx.x < nb) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kWarps; ++w) m = wbest[w * 32 + threadIdx.x] > m ? wbest[w * 32 + threadIdx.x] : m;
      atomicMax(&p.w.best[b0 + threadIdx.x], m);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- small phases

// RoPE (cos, sin) of the constant position, per sequence and layer type, angles in fp64.
__device__ inline void phase_rope(const Params& p, int cta, int ncta) {
  for (int b = cta; b < p.s.B; b += ncta) {
    const int pos = p.pos[b];
    for (int t = 0; t < 2; ++t) {
      const int d = p.s.d[t];
      const double theta = p.s.theta[t];
      for (int i = threadIdx.x; i < d / 2; i += kThreads) {
        float2 v = make_float2(1.f, 0.f);
        if (theta != 0.0) {
          const double ang = static_cast<double>(pos) * pow(theta, -2.0 * i / d);
          double sv, cv;
          sincos(ang, &sv, &cv);
          v = make_float2(static_cast<float>(cv), static_cast<float>(sv));
        }
        p.w.cs[(static_cast<size_t>(b) * 2 + t) * (p.w.dmax / 2) + i] = v;
      }
    }
  }
}

// Tokens of the last drafted step (earlier steps are written by the next PRE phase).
__device__ inline void phase_fin(const Params& p, int out_stride, int out_col, int cta, int ncta) {
  if (cta != 0) return;
  for (int b = threadIdx.x; b < p.s.B; b += kThreads) p.out_tokens[b * out_stride + out_col] = key_id(p.w.best[b]);
}

// ---------------------------------------------------------------- item counts (host + device)

__host__ __device__ inline int gemv_items(int R, int B, int K_in, int ncta_hint) {
  const int ng = ceil_div(B, gemv_group(B, K_in));
  const int ks = choose_ks(R, ng, ncta_hint);
  return ng * ceil_div(R, kWarps / ks);
}

}  // namespace mtp
