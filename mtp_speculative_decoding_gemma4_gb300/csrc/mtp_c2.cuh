// Streamed-tile cluster draft block for one sequence (B = 1). One thread-block cluster of kNC
// CTAs (one per SM) runs the whole drafter step; every projection runs on tensor cores
// (mma.m16n8k16, bf16 weights x the fp32 activation split into three exact bf16 terms).
//
// Weights: packed once at init into one contiguous stream per CTA holding, in the order the
// step consumes them, the CTA's rows of every matrix as 16x16 A-fragment tiles laid out so
// that each ring slot is one bulk copy and compute warp w always owns the same (row tile,
// k part) of a section (see WSec). A producer warp streams the sections of every step, and
// the CTA's share of the shared K (row copies issued by its 32 lanes at a padded pitch),
// through a ring of kSlots shared-memory slots (full / empty mbarriers).
//
// Exchanges stay inside the cluster: values go from registers straight into every peer's
// receive buffer with st.async, counted on the receiver's mbarrier (armed with the byte
// count it expects). Vectors that feed a projection travel as their three bf16 terms, so
// the receiver's tensor cores read them without another pass. Receive buffers alternate
// between two sets; the post-projected hidden state of step t goes to a separate buffer
// (the next step's pre_projection input) with its own mbarrier, off the critical path.
//
// Step (rows of every projection split over the kNC CTAs; every CTA keeps the residual x):
//   PRE   u = [h ; embed(token)] (terms); x0 rows = W_pre u              -> all-gather x0
//   per block l:
//     a = attn_norm(x); Q rows                                           -> all-gather q
//     q_norm + RoPE; attention over this CTA's keys (online softmax over chunks of K slots)
//                                                 -> partial sums to the owner of each dim
//     owners combine the kNC partials                                    -> all-gather o
//     O rows                                                             -> all-gather o'
//     x += post_attn_norm(o'); f = ffn_norm(x); gate / up rows; m = gelu(gate) * up
//                                                                        -> all-gather m
//     down rows                                                          -> all-gather dn
//     x = layer_scalar * (x + post_ffn_norm(dn))
//   HEAD  y = output_norm(x); centroid rows -> local top-k            -> all-gather lists
//         post rows -> h' (next step's input, output)
//         merge of the lists -> selected centroids; this CTA's clusters' rows of the
//         cluster-ordered token_embd -> local best (logit, id)         -> all-gather keys
#pragma once

#include "mtp_common.cuh"
#include "mtp.h"

namespace mtp {
namespace c2 {

constexpr int kNC = 16;             // CTAs per cluster
constexpr int kCW = 16;             // compute warps per CTA
constexpr int kCT = kCW * 32;       // compute threads
constexpr int kT = kCT + 32;        // + the producer warp
constexpr int kSlots = 4;           // ring slots
constexpr int kSlotBytes = 32768;   // largest weight payload of a slot
constexpr int kSlotStride = kSlotBytes + 512;  // K slots: kKps rows at (row + 16 bytes)
constexpr int kKps = 32;            // keys per K slot: one row copy per producer lane
constexpr int kTile = 512;          // bytes of one 16x16 bf16 A-fragment tile
constexpr int kMaxL = 8;
constexpr int kAttMT = 2;           // weighted-sum tiles (16 dims of one KV head) per warp
constexpr int kMaxSeq = 1 + 6 * kMaxL + 2;

typedef __nv_bfloat16 bf16;

struct Range {
  int lo, hi;
};
__host__ __device__ inline Range split(int R, int N, int c) {
  const long long lo = static_cast<long long>(R) * c / N, hi = static_cast<long long>(R) * (c + 1) / N;
  return Range{static_cast<int>(lo), static_cast<int>(hi)};
}
__host__ __device__ inline int split_max(int R, int N) { return (R + N - 1) / N; }
__host__ __device__ inline int al16(int v) { return (v + 15) & ~15; }
__host__ __device__ inline int imax(int a, int b) { return a > b ? a : b; }

// One weight section of CTA r: its rows [lo, lo + rows) of an R x K matrix, padded to RT row
// tiles of 16, and KT k tiles. The K range is cut into P parts; compute warp w < RT * P owns
// row tile w % RT and part w / RT, and finds 4 consecutive k tiles of its part in every slot:
// tile (slot s, warp w, j < 4) of the stream is row tile w % RT at k tile
// (w / RT) * (KT / P) + 4 s + j. nsl slots of slot_bytes each.
struct WSec {
  int lo, rows, RT, P, KT, nsl, slot_bytes;
};
__host__ __device__ inline WSec wsec(int R, int K, int r) {
  WSec s;
  const Range g = split(R, kNC, r);
  s.lo = g.lo;
  s.rows = g.hi - g.lo;
  s.RT = (s.rows + 15) / 16;
  s.KT = K / 16;
  int P = 1;
  if (s.RT > 0)
    while (2 * P * s.RT <= kCW && s.KT % (8 * P) == 0) P *= 2;
  s.P = P;
  s.nsl = s.RT > 0 ? s.KT / (4 * P) : 0;
  s.slot_bytes = 4 * s.RT * P * kTile;
  return s;
}
__host__ __device__ inline long long wsec_bytes(const WSec& s) {
  return static_cast<long long>(s.RT) * s.KT * kTile;
}

struct Params {
  int bb, H, nl, nh, nkv, F, V, C, topk, vsc, W;
  int d[2];
  float scale[2], theta[2], eps;
  int ltype[kMaxL];
  float lambda[kMaxL];
  const bf16* wstream;      // packed weight tiles: the streams of CTAs 0..kNC-1 back to back
  const bf16* tgt;          // the target's input embedding [V][bb]
  const bf16* temb_ord;     // token_embd rows in token_ordering order [V][H]
  const int* ord;           // token_ordering [C][vsc]
  const float* out_norm;
  const float *q_norm[kMaxL], *attn_norm[kMaxL], *post_attn_norm[kMaxL], *ffn_norm[kMaxL], *post_ffn_norm[kMaxL];
  const bf16* k[2];
  const int* ctx_len[2];
  long long st[2];
  int kv_max[2];
  bool has_type[2];
  const bf16* hidden_in;
  const int* tok_in;
  const int* pos;
  int* out_tokens;
  float* out_hidden;
  int n_draft;
  int* status;
  unsigned* abort_flag;
  long long spin_limit;
  int dbg_skip;  // testing: CTA dbg_skip - 1 sends none of its rows in the launch's first exchange
};

// The projection of step-sequence entry `idx` (R rows x K): 0 PRE | per block l: 1+6l Q,
// 2+6l the K rows (no weights), 3+6l O, 4+6l gate, 5+6l up, 6+6l down | CENT | POST.
__host__ __device__ inline bool seq_is_k(const Params& p, int idx) {
  return idx >= 1 && idx < 1 + 6 * p.nl && (idx - 1) % 6 == 1;
}
__host__ __device__ inline void seq_shape(const Params& p, int idx, int& R, int& K) {
  R = K = 0;
  if (idx == 0) {
    R = p.H;
    K = 2 * p.bb;
  } else if (idx == 1 + 6 * p.nl) {
    R = p.C;
    K = p.H;
  } else if (idx == 2 + 6 * p.nl) {
    R = p.bb;
    K = p.H;
  } else {
    const int l = (idx - 1) / 6, what = (idx - 1) % 6, QD = p.nh * p.d[p.ltype[l]];
    switch (what) {
      case 0: R = QD; K = p.H; break;
      case 2: R = p.H; K = QD; break;
      case 3:
      case 4: R = p.F; K = p.H; break;
      case 5: R = p.H; K = p.F; break;
      default: break;
    }
  }
}
__host__ __device__ inline int seq_count(const Params& p) { return 3 + 6 * p.nl; }
// Bytes of CTA r's stream (one step).
__host__ __device__ inline long long stream_bytes(const Params& p, int r) {
  long long b = 0;
  for (int i = 0; i < seq_count(p); ++i) {
    if (seq_is_k(p, i)) continue;
    int R, K;
    seq_shape(p, i, R, K);
    b += wsec_bytes(wsec(R, K, r));
  }
  return b;
}

// An entry of a CTA's step sequence as the kernel keeps it (shared memory).
struct SecE {
  const char* src;     // weights: this section of the CTA's stream; K: the CTA's first key row
  long long stride;    // K: bytes between key rows
  WSec w;              // weights
  int kind;            // 0 weights, 1 K rows
  int nkeys, row_bytes, pitch;  // K rows
};

// Shared-memory layout (bytes), the same in every CTA.
struct Layout {
  int ring, xs, xs_bytes, u, t, x, y, part, sp, pt, red, cs, cs_off1, nrm, nrm_stride, keys, lk, selc, tab, bars, total;
};
__host__ __device__ inline Layout make_layout(const Params& p) {
  Layout L{};
  int dmax = 0;
  for (int l = 0; l < p.nl; ++l) dmax = imax(dmax, p.d[p.ltype[l]]);
  const int QD = p.nh * dmax, dpo = QD / kNC;
  int xs = p.H * 4;
  xs = imax(xs, QD * 4);
  xs = imax(xs, kNC * (2 + dpo) * 4);
  xs = imax(xs, 3 * (QD + 8) * 2);
  xs = imax(xs, 3 * (p.F + 8) * 2);
  xs = imax(xs, kNC * p.topk * 8);
  xs = imax(xs, kNC * 8);
  int off = 0;
  L.ring = off;  off += kSlots * kSlotStride;
  L.xs_bytes = al16(xs);
  L.xs = off;    off += 2 * L.xs_bytes;
  L.u = off;     off += al16(imax(3 * (2 * p.bb + 8) * 2, 3 * p.nh * (dmax + 8) * 2));
  L.t = off;     off += al16(3 * (p.H + 8) * 2);
  L.x = off;     off += al16(p.H * 4);
  L.y = off;     off += al16(p.H * 4);
  L.part = off;  off += 2 * kCW * 16 * 4;
  // score partials: (dim part, key) pairs <= kCW key tiles of 16 keys; the merge's two lists
  L.sp = off;    off += al16(imax(kCW * 16 * p.nh * 4, 2 * (kNC / 2) * p.topk * 8));
  L.pt = off;    off += al16(3 * p.nh * (kSlots * kKps + 8) * 2);
  L.red = off;   off += 128 * 4;
  const int h0 = p.has_type[0] ? p.d[0] / 2 : 0, h1 = p.has_type[1] ? p.d[1] / 2 : 0;
  L.cs_off1 = h0;
  L.cs = off;    off += al16((h0 + h1) * 8);
  L.nrm_stride = 4 * p.H + dmax;
  L.nrm = off;   off += al16((p.nl * L.nrm_stride + p.H) * 4);
  L.keys = off;  off += al16(split_max(p.C, kNC) * 8);
  L.lk = off;    off += al16(imax(p.topk, kCW) * 8);
  L.selc = off;  off += al16(64 * 4);
  L.tab = off;   off += al16(kMaxSeq * static_cast<int>(sizeof(SecE)));
  L.bars = off;  off += (2 * kSlots + 3) * 8;
  L.total = al16(off);
  return L;
}

}  // namespace c2
}  // namespace mtp
