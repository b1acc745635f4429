// Cluster-path draft block for one sequence (B = 1): the whole drafter step runs inside one
// thread-block cluster of NC CTAs (one per SM). In every CTA a producer warp streams the
// CTA's row-slices of each weight matrix and its share of the shared K, in the order the
// step consumes them, through a ring of shared-memory slots filled by TMA bulk copies
// (full / empty mbarriers); kCW compute warps consume the slots. Vectors are exchanged
// inside the cluster only: each CTA writes its slice into every CTA's receive buffer with
// st.async, whose bytes complete on the receiver's mbarrier (armed by the receiver with the
// byte count it expects); receive buffers and their mbarriers alternate between two sets.
//
// Step (rows of every GEMV split over the NC CTAs; every CTA keeps its own residual x):
//   PRE   token from the last exchange; u = [h ; embed(token)]; x0[rows] = W_pre u  -> all x0
//   per block: Q rows -> all q; q_norm + RoPE; attention over this CTA's keys (online
//     softmax over the streamed K chunks) -> partials to the owner of each output dim;
//     owners combine -> all o; O rows -> all o'; x += norm(o'); f = norm(x);
//     gate/up rows -> m rows -> all m; W_down rows -> all dn; x = lambda (x + norm(dn))
//   HEAD  y = output_norm(x); centroid rows -> local top-k; post rows -> h';
//         exchange (h', local top-k lists); rank merge -> selected centroids; this CTA's
//         selected clusters' rows of the cluster-ordered token_embd copy -> logits ->
//         local argmax -> exchange keys -> next token
#pragma once

#include "mtp_common.cuh"
#include "mtp.h"

namespace mtp {
namespace clk {

constexpr int kNC = 16;            // CTAs per cluster
// compute warps (a multiple of 4). Nine warps per CTA leave each scheduler at most three, so
// a thread may hold 168 registers; measured on the E2B shape, 8 compute warps beat 4, 12 and
// 16 (fewer spills and cheaper barriers outweigh the lost parallelism).
constexpr int kCW = 8;
constexpr int kCT = kCW * 32;      // compute threads
constexpr int kT = kCT + 32;       // + one producer warp
static_assert(kCW % 4 == 0, "the tensor-core GEMV splits k over groups of four warps");
constexpr int kSlots = 4;
constexpr int kSlotBytes = 32768;  // payload of a weight slot
// Slots are kSlotPad bytes longer than their weight payload so that 32 K rows of d = 512 fit
// at a padded pitch (row + 16 bytes: 8 rows at the same column fall in distinct banks).
constexpr int kSlotPad = 512;
constexpr int kSlotStride = kSlotBytes + kSlotPad;
constexpr int kMaxL = 8;
constexpr int kXchFloats = 4096;   // floats per receive buffer

typedef __nv_bfloat16 bf16;

struct Range {
  int lo, hi;
};
__host__ __device__ inline Range split(int R, int N, int c) {
  const long long lo = static_cast<long long>(R) * c / N, hi = static_cast<long long>(R) * (c + 1) / N;
  return Range{static_cast<int>(lo), static_cast<int>(hi)};
}
__host__ __device__ inline int split_max(int R, int N) { return (R + N - 1) / N; }

struct Params {
  int bb, H, nl, nh, nkv, F, V, C, topk, vsc, W;
  int d[2];
  float scale[2], theta[2], eps;
  int ltype[kMaxL];
  float lambda[kMaxL];
  const bf16 *pre, *post, *cent, *tgt;
  const bf16* temb_ord;     // token_embd rows in token_ordering order [V][H]
  // Matrices with hidden-wide rows (Q, gate, up, centroids, post_projection), re-laid out
  // once at init for the tensor cores: per CTA of the cluster, its rows padded to a multiple
  // of 16, as 16x16 tiles (row tile major, k tile minor) of 512 bytes each in mma.m16n8k16
  // A-fragment order. Used when `mma` is set.
  bool mma;
  const bf16 *pk_q[kMaxL], *pk_gate[kMaxL], *pk_up[kMaxL], *pk_cent, *pk_post;
  const float* out_norm;
  const int* ord;
  const bf16 *q[kMaxL], *o[kMaxL], *gate[kMaxL], *up[kMaxL], *down[kMaxL];
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
};

// GEMV work split inside one ring slot of `rpc` rows: tasks are (row quad, k slice) pairs for
// the compute warps; rows wider than one slot's share get split along k so that every warp
// has a task. Number of k slices:
__host__ __device__ inline int gemv_ns(int rpc) {
  const int nq = (rpc + 3) / 4;
  if (nq >= kCW) return 1;
  int ns = 1;
  while (ns * 2 * nq <= kCW) ns *= 2;
  return ns;
}
__host__ __device__ inline int rows_per_slot(int row_bytes) {
  const int r = row_bytes > 0 ? kSlotBytes / row_bytes : 1;
  return r < 1 ? 1 : r;
}
// Floats of k-split partial sums a GEMV section of R rows (split over the cluster) of
// row_bytes-wide rows needs.
__host__ __device__ inline int gemv_part_floats(int R, int row_bytes) {
  const int ns = gemv_ns(rows_per_slot(row_bytes));
  return ns > 1 ? ns * split_max(R, kNC) : 0;
}
constexpr int kQkSlices = 2;  // most k slices of the attention score pass
constexpr int kMaxKeysPerSlot = 128;
// Keys per ring slot for K rows of row_bytes (bounded so that the score buffer stays small).
__host__ __device__ inline int keys_per_slot(int row_bytes) {
  const int r = rows_per_slot(row_bytes);
  return r < kMaxKeysPerSlot ? r : kMaxKeysPerSlot;
}

// Keys per slot of a K section at the padded pitch of the tensor-core attention (a multiple of
// the 16-key MMA tile).
__host__ __device__ inline int keys_per_slot_mma(int row_bytes) {
  const int r = kSlotStride / (row_bytes + 16) / 16 * 16;
  return r < kMaxKeysPerSlot ? r : kMaxKeysPerSlot;
}
// The tensor-core attention (one KV head and at most 4 query heads, q as three bf16 terms of
// every head in a receive buffer, at most four (head, dim-pair) items per thread in its q
// set-up, 16-key tiles, at most 4 dim tiles of 16 per compute warp).
__host__ __device__ inline bool att_mma_ok(const Params& p) {
  if (!p.mma || p.nkv != 1 || p.nh < 1 || p.nh > 4) return false;
  for (int t = 0; t < 2; ++t) {
    if (!p.has_type[t]) continue;
    const int d = p.d[t];
    if (d % 16 || d < 16 || d > 16 * 4 * kCW || p.nh * d > 2048 || 3 * p.nh * (d + 8) * 2 > kXchFloats * 4 ||
        keys_per_slot_mma(d * 2) < 16)
      return false;
  }
  return true;
}

// Packed tile layout of a matrix with R rows split over the cluster (see Params::pk_q):
// CTA r's rows padded to 16 and the number of 512-byte tiles before its block.
__host__ __device__ inline int padded_rows(int R, int r) {
  const Range g = split(R, kNC, r);
  return (g.hi - g.lo + 15) / 16 * 16;
}
__host__ __device__ inline long long tiles_before(int R, int K, int r) {
  long long t = 0;
  for (int i = 0; i < r; ++i) t += static_cast<long long>(padded_rows(R, i) / 16) * (K / 16);
  return t;
}
constexpr int kTileBytes = 512;

// One section of a CTA's weight / K stream: rows [0, nrows) of `row_bytes` each, row i at
// src + i*stride; rpc rows per ring slot. Packed sections (tensor-core tiles) stream tiles as
// rows and carry their k tiles per row tile and real row count (else both 0).
struct Sec {
  const char* src;
  long long stride;
  int row_bytes, nrows, rpc;
  int kt, rrows;
  int pitch;  // bytes between rows in the slot (row_bytes, or padded K rows)
};
constexpr int kMaxSec = 1 + 6 * kMaxL + 2;  // PRE | 6 per block | CENT | POST

// Shared-memory layout (bytes), identical in every CTA.
struct Layout {
  int ring, xch0, xch1, u, x, a, rows, gt, ut, part, xt, sc, red, cs, lk, ids, tab, nrm, bars, total;
  int nrm_stride;  // floats of norm gains per block: attn, post_attn, ffn, post_ffn (H each), q_norm (dmax)
  int cs_off1;  // float2 index of the full-attention RoPE table inside cs
};
__host__ __device__ inline int al16(int v) { return (v + 15) & ~15; }
__host__ __device__ inline int imax(int a, int b) { return a > b ? a : b; }
__host__ __device__ inline Layout make_layout(const Params& p) {
  Layout L{};
  int off = 0;
  int dmax = 0, dmin = 1 << 30;
  for (int l = 0; l < p.nl; ++l) {
    dmax = imax(dmax, p.d[p.ltype[l]]);
    dmin = p.d[p.ltype[l]] < dmin ? p.d[p.ltype[l]] : dmin;
  }
  if (dmin <= 0) dmin = 1;
  L.ring = off;  off += kSlots * kSlotStride;
  L.xch0 = off;  off += kXchFloats * 4;
  L.xch1 = off;  off += kXchFloats * 4;  // must directly follow xch0
  L.u = off;     off += al16(2 * p.bb * 4);
  L.x = off;     off += al16(p.H * 4);
  L.a = off;     off += al16(p.H * 4);
  int rmax = imax(imax(split_max(p.bb, kNC), split_max(p.C, kNC)), split_max(p.F, kNC));
  rmax = imax(rmax, split_max(p.H, kNC));
  // also stages the attention sums of every output dim and the (max, sum) of every head
  rmax = imax(rmax, p.nh * dmax + 2 * p.nh);
  L.rows = off;  off += al16(rmax * 4);
  const int gmax = imax(imax(split_max(p.F, kNC), split_max(p.C, kNC)), 2 * p.topk);
  L.gt = off;    off += al16(gmax * 4);        // gate rows / centroid logits / staged keys
  L.ut = off;    off += al16(split_max(p.F, kNC) * 4);
  int part = imax(gemv_part_floats(p.H, 2 * p.bb * 2), gemv_part_floats(p.bb, p.H * 2));
  part = imax(part, imax(gemv_part_floats(p.F, p.H * 2), gemv_part_floats(p.H, p.F * 2)));
  part = imax(part, gemv_part_floats(p.C, p.H * 2));
  for (int l = 0; l < p.nl; ++l) {
    const int QD = p.nh * p.d[p.ltype[l]];
    part = imax(part, imax(gemv_part_floats(QD, p.H * 2), gemv_part_floats(p.H, QD * 2)));
  }
  // k-quarter partials of the tensor-core GEMVs: 4 x padded rows of the largest section
  int pr = imax(imax(split_max(p.nh * dmax, kNC), split_max(p.F, kNC)), imax(split_max(p.C, kNC), split_max(p.bb, kNC)));
  part = imax(part, 4 * ((pr + 15) / 16 * 16));
  const bool amma = att_mma_ok(p);
  // tensor-core attention: probabilities of a slot of keys as three bf16 terms per head
  if (amma) part = imax(part, (3 * p.nh * (keys_per_slot_mma(dmin * 2) + 8) * 2 + 3) / 4);
  L.part = off;  off += al16(part * 4);
  L.xt = off;    off += al16(4 * (p.H + 8) * 2);  // bf16 hi / mid / lo terms of a GEMV input + a zero row (pitch H + 8)
  // two alternating buffers of score partials (up to kQkSlices k slices) for one slot of keys;
  // also holds the combine weights, the centroid keys and the candidate lists of the head
  int scf = 2 * kQkSlices * keys_per_slot(p.nkv * dmin * 2) * p.nh;
  if (amma) scf = imax(scf, 4 * keys_per_slot_mma(dmin * 2) * p.nh);  // 4 k-quarter score partials
  scf = imax(scf, imax(kNC * p.nh, 2 * split_max(p.C, kNC)));
  scf = imax(scf, 2 * kNC * p.topk);  // 64-bit candidate lists of the top-k merge
  L.sc = off;    off += al16(scf * 4);
  L.red = off;   off += 128 * 4;
  const int h0 = p.has_type[0] ? p.d[0] / 2 : 0, h1 = p.has_type[1] ? p.d[1] / 2 : 0;
  L.cs_off1 = h0;
  L.cs = off;    off += al16((h0 + h1) * 8);   // RoPE (cos, sin) of the sliding, then full, head_dim
  L.lk = off;    off += al16(64 * 8);          // local top-k keys / per-warp best keys
  L.ids = off;   off += al16(64 * 4);          // selected centroids
  L.tab = off;   off += al16(kMaxSec * static_cast<int>(sizeof(Sec)));  // this CTA's stream sections
  L.nrm_stride = 4 * p.H + dmax;
  L.nrm = off;   off += al16((p.nl * L.nrm_stride + p.H) * 4);  // all norm gains, then output_norm
  L.bars = off;  off += (2 * kSlots + 2) * 8;
  L.total = al16(off);
  return L;
}

}  // namespace clk
}  // namespace mtp
