// C ABI of libmtp (include/mtp.h): argument validation, workspace ownership and dispatch
// to the drafter-step kernels.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "mtp.h"
#include "mtp_launch.h"
#include "mtp_c2.cuh"
#include "mtp_grid.cuh"
#include "mtp_tc.cuh"
#include "mtp_phases.cuh"

struct mtp_handle {
  mtp_config cfg;
  mtp_weights w;
  const void* target_embed;
  int device;
  int num_sms;
  int path;
  int mask_mode;  // materialised rows of the centroid head: MTP_MASK_NEG_1E30 / MIN_MINUS_ONE
  int head_mode;  // sparse head traversal: MTP_HEAD_AUTO / PER_SEQUENCE / CLUSTER_MAJOR
  // testing only (mtp_set_debug): a CTA that skips its first grid-barrier arrival, and a
  // shorter bound for device waits (0: the defaults)
  int dbg_skip;
  long long dbg_spin;
  int dmax;
  int nsplit_max;
  void* ws;
  size_t ws_bytes;
  mtp::WsP wsp;
  // abort word of the single-sequence paths (a bounded wait that gives up raises it)
  unsigned* abort_word;
  // token_embd in token_ordering order (the rows of one centroid contiguous): single-sequence
  // paths and the cluster-major head
  void* temb_ord;
  // streamed-tile cluster path (one sequence): availability and the packed weight streams
  int c2_ok;
  void* c2_stream;
  // grid path (one sequence): availability, the planned parameters (host), the per-CTA weight
  // images, the mailboxes and the next epoch
  int gr_ok;
  mtp::gr::Params* gr;
  void* gr_img;
  unsigned long long* gr_mb;
  long long gr_mb_words;
  double* gr_inv;  // RoPE inverse frequencies of both attention types (fp64)
  unsigned gr_epoch;
  // tensor-core phase path (batches of 2..tc::kMaxB): tensor maps (64-byte aligned host memory) and
  // the staging buffer of the input terms
  mtp::TcPlan* tc;
  void* tc_mem;
  void* tc_wmem;  // the stacked weight copies of the tensor-core path
  // multi-launch paths: the draft block of the last argument set as an instantiated CUDA
  // graph, replayed on an internal stream ordered after / before the caller's stream by
  // events; a call with different arguments captures again
  struct {
    int valid, path;
    mtp::Params key;
    cudaGraphExec_t exec;
    cudaStream_t cs;
    cudaEvent_t ev_in, ev_out;
  } gc;
};

namespace mtp {

static thread_local char g_err[1024] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

}  // namespace mtp

using mtp::set_error;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_fail(const char* what, cudaError_t e) {
  set_error("%s: %s", what, cudaGetErrorString(e));
  return MTP_ERR_CUDA;
}

bool has_type(const mtp_config& c, int t) {
  for (int l = 0; l < c.n_layers; ++l)
    if (c.layer_type[l] == t) return true;
  return false;
}

int validate_config(const mtp_config& c) {
  if (c.n_layers < 1 || c.n_layers > MTP_MAX_LAYERS) {
    set_error("n_layers=%d outside [1, %d]", c.n_layers, MTP_MAX_LAYERS);
    return MTP_ERR_INVALID_ARG;
  }
  if (c.dtype != MTP_DTYPE_BF16 && c.dtype != MTP_DTYPE_F32) {
    set_error("dtype=%d is neither BF16 nor F32", c.dtype);
    return MTP_ERR_INVALID_ARG;
  }
  if (c.backbone <= 0 || c.hidden <= 0 || c.n_head <= 0 || c.n_kv_head <= 0 || c.ffn <= 0 || c.vocab <= 0 ||
      c.max_batch <= 0 || c.max_ctx <= 0) {
    set_error("non-positive size in config");
    return MTP_ERR_INVALID_ARG;
  }
  for (int l = 0; l < c.n_layers; ++l)
    if (c.layer_type[l] > 1) {
      set_error("layer_type[%d]=%d is neither sliding (0) nor full (1)", l, c.layer_type[l]);
      return MTP_ERR_INVALID_ARG;
    }
  if (!(c.rms_eps >= 0.f) || !(c.attn_scale >= 0.f) || !(c.rope_theta_swa >= 0.f) || !(c.rope_theta_full >= 0.f)) {
    set_error("rms_eps, attn_scale and rope thetas must be >= 0");
    return MTP_ERR_INVALID_ARG;
  }
  const int vec = c.dtype == MTP_DTYPE_BF16 ? 8 : 4;
  if (c.hidden % vec || c.backbone % vec || c.ffn % vec) {
    set_error("hidden, backbone and ffn must be multiples of %d", vec);
    return MTP_ERR_UNSUPPORTED_SHAPE;
  }
  if (c.n_head % c.n_kv_head) {
    set_error("n_head=%d is not a multiple of n_kv_head=%d", c.n_head, c.n_kv_head);
    return MTP_ERR_UNSUPPORTED_SHAPE;
  }
  const int hpg = c.n_head / c.n_kv_head;
  for (int t = 0; t < 2; ++t) {
    if (!has_type(c, t)) continue;
    const int d = t ? c.head_dim_full : c.head_dim_swa;
    const bool d_ok = d == 32 || d == 64 || d == 128 || d == 256 || d == 512;
    const bool h_ok = hpg == 1 || hpg == 2 || hpg == 4 || (hpg == 8 && d <= 256);
    if (!d_ok || !h_ok) {
      set_error("attention shape head_dim=%d, heads per KV head=%d not supported", d, hpg);
      return MTP_ERR_UNSUPPORTED_SHAPE;
    }
  }
  if (has_type(c, 0) && c.window < 1) {
    set_error("sliding layers need window >= 1 (got %d)", c.window);
    return MTP_ERR_INVALID_ARG;
  }
  if (c.use_ordered_embeddings) {
    if (c.n_centroids <= 0 || c.top_k <= 0 || c.top_k > 64 || c.top_k > c.n_centroids || c.n_centroids > 8192) {
      set_error("centroid head needs 0 < top_k <= min(64, n_centroids), n_centroids <= 8192");
      return MTP_ERR_UNSUPPORTED_SHAPE;
    }
    if (c.vocab % c.n_centroids) {
      set_error("vocab=%d is not a multiple of n_centroids=%d", c.vocab, c.n_centroids);
      return MTP_ERR_BAD_ORDERING;
    }
  } else {
    if (c.hidden % (32 * vec)) {
      set_error("dense head needs hidden to be a multiple of %d", 32 * vec);
      return MTP_ERR_UNSUPPORTED_SHAPE;
    }
  }
  return MTP_OK;
}

int validate_weights(const mtp_config& c, const mtp_weights& w, const void* target_embed) {
  const void* mats[] = {w.pre_proj, w.post_proj, w.token_embd, w.out_norm, target_embed};
  for (const void* m : mats)
    if (!m || !aligned16(m)) {
      set_error("pre_proj, post_proj, token_embd, out_norm and target_embed must be non-NULL, 16-byte aligned");
      return MTP_ERR_INVALID_ARG;
    }
  if (c.use_ordered_embeddings && (!w.centroids || !aligned16(w.centroids) || !w.token_ordering)) {
    set_error("centroid head needs centroids (16-byte aligned) and token_ordering");
    return MTP_ERR_INVALID_ARG;
  }
  for (int l = 0; l < c.n_layers; ++l) {
    const mtp_layer_weights& L = w.layer[l];
    const void* ptrs[] = {L.q, L.o, L.gate, L.up, L.down, L.q_norm, L.attn_norm, L.post_attn_norm, L.ffn_norm,
                          L.post_ffn_norm};
    for (const void* p : ptrs)
      if (!p || !aligned16(p)) {
        set_error("layer %d: weight pointer NULL or not 16-byte aligned", l);
        return MTP_ERR_INVALID_ARG;
      }
  }
  return MTP_OK;
}

int check_ordering(const mtp_config& c, const int32_t* ord) {
  std::vector<int32_t> h(c.vocab);
  cudaError_t e = cudaMemcpy(h.data(), ord, sizeof(int32_t) * c.vocab, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail("reading token_ordering", e);
  std::vector<unsigned char> seen(c.vocab, 0);
  for (int i = 0; i < c.vocab; ++i) {
    const int32_t v = h[i];
    if (v < 0 || v >= c.vocab || seen[v]) {
      set_error("token_ordering is not a permutation of 0..%d (entry %d = %d)", c.vocab - 1, i, v);
      return MTP_ERR_BAD_ORDERING;
    }
    seen[v] = 1;
  }
  return MTP_OK;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Tensor maps and staging buffer of the tensor-core phase path; leaves h->tc NULL when the
// configuration or the device does not allow it.
int build_tc(mtp_handle* h) {
  const mtp_config& c = h->cfg;
  h->tc = nullptr;
  h->tc_mem = nullptr;
  h->tc_wmem = nullptr;
  if (c.dtype != MTP_DTYPE_BF16 || c.max_batch < 2 || c.max_batch > mtp::tc::kMaxB || !mtp::tc_available()) return MTP_OK;
  const int bb = c.backbone, H = c.hidden, F = c.ffn;
  int qd[2] = {0, 0};
  for (int t = 0; t < 2; ++t) qd[t] = has_type(c, t) ? c.n_head * (t ? c.head_dim_full : c.head_dim_swa) : 0;
  const int ks[] = {2 * bb, H, F, qd[0], qd[1]};
  int kmax = 0;
  for (int k : ks) {
    if (k % mtp::tc::kKStage) return MTP_OK;
    kmax = k > kmax ? k : kmax;
  }
  void* mem = nullptr;
  if (posix_memalign(&mem, 64, sizeof(mtp::TcPlan)) != 0 || !mem) return MTP_OK;
  memset(mem, 0, sizeof(mtp::TcPlan));
  mtp::TcPlan* plan = static_cast<mtp::TcPlan*>(mem);
  plan->bp = (c.max_batch + 31) / 32 * 32;
  const size_t xs_bytes = static_cast<size_t>(3) * plan->bp * kmax * 2;
  cudaError_t e = cudaMalloc(&h->tc_mem, xs_bytes);
  if (e == cudaSuccess) e = cudaMemset(h->tc_mem, 0, xs_bytes);
  if (e != cudaSuccess) {
    free(mem);
    h->tc_mem = nullptr;
    return cuda_fail("allocating the tensor-core staging buffer", e);
  }
  plan->xs = static_cast<__nv_bfloat16*>(h->tc_mem);
  int rc = MTP_OK;
  auto wmap = [&](CUtensorMap* m, const void* W, int R, int K) {
    if (!rc) rc = mtp::tc_make_map(m, W, R, K, K, mtp::tc::kM);
  };
  auto xmap = [&](CUtensorMap* m, int K) {
    if (!rc && K > 0) rc = mtp::tc_make_map(m, plan->xs, 3 * plan->bp, K, K, 3 * plan->bp);
  };
  wmap(&plan->pre, h->w.pre_proj, H, 2 * bb);
  wmap(&plan->post, h->w.post_proj, bb, H);
  if (c.use_ordered_embeddings) wmap(&plan->cent, h->w.centroids, c.n_centroids, H);
  else wmap(&plan->temb, h->w.token_embd, c.vocab, H);
  for (int l = 0; l < c.n_layers; ++l) {
    const mtp_layer_weights& L = h->w.layer[l];
    const int q = qd[c.layer_type[l]];
    wmap(&plan->q[l], L.q, q, H);
    wmap(&plan->o[l], L.o, H, q);
    wmap(&plan->gate[l], L.gate, F, H);
    wmap(&plan->up[l], L.up, F, H);
    wmap(&plan->down[l], L.down, H, F);
  }
  xmap(&plan->xs_pre, 2 * bb);
  xmap(&plan->xs_h, H);
  xmap(&plan->xs_f, F);
  xmap(&plan->xs_o[0], qd[0]);
  xmap(&plan->xs_o[1], qd[1]);
  // stacked copies (made once, like the other per-handle weight copies): per layer [gate ; up]
  // interleaved in 64-row blocks for the gated-GELU epilogue, with its own staging buffer for
  // the down projection's operand (the gate / up GEMM still reads the shared one); and
  // [post_proj ; centroids], whose first block is a whole number of 128-row tiles
  const size_t row = static_cast<size_t>(H) * 2;
  const int C = c.use_ordered_embeddings ? c.n_centroids : 0;
  plan->gu_ok = F % 64 == 0;
  plan->postc_ok = C > 0 && bb % mtp::tc::kM == 0;
  const size_t gu_bytes = plan->gu_ok ? 2 * static_cast<size_t>(F) * row : 0;
  const size_t xsf_bytes = plan->gu_ok ? static_cast<size_t>(3) * plan->bp * F * 2 : 0;
  const size_t pc_bytes = plan->postc_ok ? static_cast<size_t>(bb + C) * row : 0;
  const size_t wbytes = xsf_bytes + gu_bytes * c.n_layers + pc_bytes;
  if (!rc && wbytes) {
    cudaError_t ew = cudaMalloc(&h->tc_wmem, wbytes);
    char* wb = static_cast<char*>(h->tc_wmem);
    if (ew == cudaSuccess && plan->gu_ok) {
      plan->xs_glu = reinterpret_cast<__nv_bfloat16*>(wb);
      ew = cudaMemset(wb, 0, xsf_bytes);
      if (ew == cudaSuccess && !rc) rc = mtp::tc_make_map(&plan->xs_f2, wb, 3 * plan->bp, F, F, 3 * plan->bp);
    }
    for (int l = 0; ew == cudaSuccess && plan->gu_ok && l < c.n_layers; ++l) {
      char* d = wb + xsf_bytes + l * gu_bytes;
      const size_t blk = 64 * row;  // 64 rows
      ew = cudaMemcpy2D(d, 2 * blk, h->w.layer[l].gate, blk, blk, F / 64, cudaMemcpyDeviceToDevice);
      if (ew == cudaSuccess)
        ew = cudaMemcpy2D(d + blk, 2 * blk, h->w.layer[l].up, blk, blk, F / 64, cudaMemcpyDeviceToDevice);
      wmap(&plan->gu[l], d, 2 * F, H);
    }
    if (ew == cudaSuccess && plan->postc_ok) {
      char* d = wb + xsf_bytes + gu_bytes * c.n_layers;
      ew = cudaMemcpy(d, h->w.post_proj, bb * row, cudaMemcpyDeviceToDevice);
      if (ew == cudaSuccess) ew = cudaMemcpy(d + bb * row, h->w.centroids, C * row, cudaMemcpyDeviceToDevice);
      wmap(&plan->postc, d, bb + C, H);
    }
    if (ew != cudaSuccess && !rc) rc = cuda_fail("copying the stacked tensor-core weights", ew);
  }
  if (rc) {
    cudaFree(h->tc_mem);
    h->tc_mem = nullptr;
    if (h->tc_wmem) cudaFree(h->tc_wmem);
    h->tc_wmem = nullptr;
    free(mem);
    return rc;
  }
  h->tc = plan;
  return MTP_OK;
}

// Streamed-tile cluster-path parameters that depend only on the handle.
mtp::c2::Params c2_template(const mtp_handle* h, int kv_max) {
  const mtp_config& c = h->cfg;
  mtp::c2::Params p;
  memset(&p, 0, sizeof(p));
  p.bb = c.backbone;
  p.H = c.hidden;
  p.nl = c.n_layers;
  p.nh = c.n_head;
  p.nkv = c.n_kv_head;
  p.F = c.ffn;
  p.V = c.vocab;
  p.C = c.n_centroids;
  p.topk = c.top_k;
  p.vsc = c.use_ordered_embeddings && c.n_centroids > 0 ? c.vocab / c.n_centroids : 0;
  p.W = c.window;
  p.d[0] = c.head_dim_swa;
  p.d[1] = c.head_dim_full;
  for (int t = 0; t < 2; ++t) {
    const int d = p.d[t] > 0 ? p.d[t] : 1;
    p.scale[t] = c.attn_scale > 0.f ? c.attn_scale : 1.0f / sqrtf(static_cast<float>(d));
  }
  p.theta[0] = c.rope_theta_swa;
  p.theta[1] = c.rope_theta_full;
  p.eps = c.rms_eps;
  typedef const __nv_bfloat16* cb;
  p.wstream = static_cast<cb>(h->c2_stream);
  p.tgt = static_cast<cb>(h->target_embed);
  p.temb_ord = static_cast<cb>(h->temb_ord);
  p.out_norm = h->w.out_norm;
  p.ord = h->w.token_ordering;
  for (int l = 0; l < c.n_layers; ++l) {
    const mtp_layer_weights& L = h->w.layer[l];
    p.ltype[l] = c.layer_type[l];
    p.lambda[l] = L.layer_scalar;
    p.q_norm[l] = L.q_norm;
    p.attn_norm[l] = L.attn_norm;
    p.post_attn_norm[l] = L.post_attn_norm;
    p.ffn_norm[l] = L.ffn_norm;
    p.post_ffn_norm[l] = L.post_ffn_norm;
  }
  for (int t = 0; t < 2; ++t) {
    p.has_type[t] = has_type(c, t);
    p.kv_max[t] = kv_max;
    p.st[t] = static_cast<long long>(c.n_kv_head) * (t ? c.head_dim_full : c.head_dim_swa);
  }
  p.spin_limit = 4000000000LL;  // ~2 s at 2 GHz
  return p;
}

// Whether the streamed-tile cluster path can run this configuration on this device.
bool c2_supported(const mtp_handle* h) {
  const mtp_config& c = h->cfg;
  if (c.dtype != MTP_DTYPE_BF16 || !c.use_ordered_embeddings) return false;
  const mtp::c2::Params p = c2_template(h, c.max_ctx);
  const int smem = mtp::c2_smem_bytes(p);
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (smem <= 0 || smem > optin) return false;
  return mtp::c2_capacity(smem) >= 1;
}

// Packs every projection of the drafter into the per-CTA weight streams of the streamed-tile
// cluster path (h->c2_stream).
int build_c2_stream(mtp_handle* h) {
  const mtp_config& c = h->cfg;
  const mtp::c2::Params p = c2_template(h, c.max_ctx);
  const void* mats[mtp::c2::kMaxSeq] = {};
  mats[0] = h->w.pre_proj;
  for (int l = 0; l < c.n_layers; ++l) {
    const mtp_layer_weights& L = h->w.layer[l];
    mats[1 + 6 * l] = L.q;
    mats[3 + 6 * l] = L.o;
    mats[4 + 6 * l] = L.gate;
    mats[5 + 6 * l] = L.up;
    mats[6 + 6 * l] = L.down;
  }
  mats[1 + 6 * c.n_layers] = h->w.centroids;
  mats[2 + 6 * c.n_layers] = h->w.post_proj;
  const size_t bytes = static_cast<size_t>(mtp::c2_stream_total(p));
  cudaError_t e = cudaMalloc(&h->c2_stream, bytes);
  if (e != cudaSuccess) {
    h->c2_stream = nullptr;
    return cuda_fail("allocating the streamed weight tiles", e);
  }
  int rc = mtp::c2_pack_all(p, mats, h->c2_stream, 0);
  e = rc ? cudaErrorUnknown : cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(h->c2_stream);
    h->c2_stream = nullptr;
    return rc ? rc : cuda_fail("packing the streamed weight tiles", e);
  }
  return MTP_OK;
}

// Grid-path parameters that depend only on the handle (shapes, weights), for K of up to
// kv_max keys.
mtp::gr::Params gr_template(const mtp_handle* h, int kv_max) {
  const mtp_config& c = h->cfg;
  mtp::gr::Params p;
  memset(&p, 0, sizeof(p));
  p.bb = c.backbone;
  p.H = c.hidden;
  p.nl = c.n_layers;
  p.nh = c.n_head;
  p.nkv = c.n_kv_head;
  p.F = c.ffn;
  p.V = c.vocab;
  p.C = c.n_centroids;
  p.topk = c.top_k;
  p.vsc = c.use_ordered_embeddings && c.n_centroids > 0 ? c.vocab / c.n_centroids : 0;
  p.W = c.window;
  p.d[0] = c.head_dim_swa;
  p.d[1] = c.head_dim_full;
  for (int t = 0; t < 2; ++t) {
    const int d = p.d[t] > 0 ? p.d[t] : 1;
    p.scale[t] = c.attn_scale > 0.f ? c.attn_scale : 1.0f / sqrtf(static_cast<float>(d));
  }
  p.theta[0] = c.rope_theta_swa;
  p.theta[1] = c.rope_theta_full;
  p.eps = c.rms_eps;
  typedef const __nv_bfloat16* cb;
  p.tgt = static_cast<cb>(h->target_embed);
  p.temb_ord = static_cast<cb>(h->temb_ord);
  p.out_norm = h->w.out_norm;
  p.ord = h->w.token_ordering;
  for (int l = 0; l < c.n_layers; ++l) {
    const mtp_layer_weights& L = h->w.layer[l];
    p.ltype[l] = c.layer_type[l];
    p.lambda[l] = L.layer_scalar;
    p.q_norm[l] = L.q_norm;
    p.attn_norm[l] = L.attn_norm;
    p.post_attn_norm[l] = L.post_attn_norm;
    p.ffn_norm[l] = L.ffn_norm;
    p.post_ffn_norm[l] = L.post_ffn_norm;
  }
  for (int t = 0; t < 2; ++t) {
    p.has_type[t] = has_type(c, t) ? 1 : 0;
    p.kv_max[t] = kv_max;
    p.st[t] = static_cast<long long>(c.n_kv_head) * (t ? c.head_dim_full : c.head_dim_swa);
  }
  p.spin_limit = 4000000000LL;  // ~2 s at 2 GHz
  return p;
}

// Plans the grid path for this handle and, when it fits, packs the per-CTA weight images and
// allocates the mailboxes (h->gr_ok stays 0 otherwise, and the other paths serve B = 1).
int build_gr(mtp_handle* h) {
  const mtp_config& c = h->cfg;
  h->gr_ok = 0;
  if (c.dtype != MTP_DTYPE_BF16 || !c.use_ordered_embeddings || !h->temb_ord) return MTP_OK;
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device) != cudaSuccess) {
    cudaGetLastError();
    return MTP_OK;
  }
  mtp::gr::Params* p = static_cast<mtp::gr::Params*>(malloc(sizeof(mtp::gr::Params)));
  if (!p) return MTP_OK;
  *p = gr_template(h, c.max_ctx);
  if (mtp::gr_plan(*p, optin) <= 0) {
    free(p);
    return MTP_OK;
  }
  h->gr = p;
  const size_t img = static_cast<size_t>(mtp::gr_image_total(*p));
  h->gr_mb_words = mtp::gr_mailboxes(*p);
  cudaError_t e = cudaMalloc(&h->gr_img, img);
  if (e == cudaSuccess) e = cudaMemset(h->gr_img, 0, img);
  if (e == cudaSuccess) e = cudaMalloc(&h->gr_mb, static_cast<size_t>(h->gr_mb_words) * 8);
  if (e == cudaSuccess) e = cudaMemset(h->gr_mb, 0, static_cast<size_t>(h->gr_mb_words) * 8);
  if (e != cudaSuccess) return cuda_fail("allocating the grid path's weight images and mailboxes", e);
  const void *q[MTP_MAX_LAYERS], *o[MTP_MAX_LAYERS], *g[MTP_MAX_LAYERS], *u[MTP_MAX_LAYERS], *d[MTP_MAX_LAYERS];
  for (int l = 0; l < c.n_layers; ++l) {
    q[l] = h->w.layer[l].q;
    o[l] = h->w.layer[l].o;
    g[l] = h->w.layer[l].gate;
    u[l] = h->w.layer[l].up;
    d[l] = h->w.layer[l].down;
  }
  // RoPE inverse frequencies theta^(-2i/d) of both types, formed once in fp64 (0: no rotation)
  {
    const int h0 = c.head_dim_swa / 2, h1 = c.head_dim_full / 2, hm = h0 > h1 ? h0 : h1;
    std::vector<double> inv(2 * static_cast<size_t>(hm > 0 ? hm : 1), 0.0);
    const float th[2] = {c.rope_theta_swa, c.rope_theta_full};
    const int dd[2] = {c.head_dim_swa, c.head_dim_full};
    for (int t = 0; t < 2; ++t)
      for (int i = 0; i < dd[t] / 2; ++i)
        inv[t * hm + i] = th[t] > 0.f ? std::pow(static_cast<double>(th[t]), -2.0 * i / dd[t]) : 0.0;
    e = cudaMalloc(&h->gr_inv, inv.size() * sizeof(double));
    if (e == cudaSuccess) e = cudaMemcpy(h->gr_inv, inv.data(), inv.size() * sizeof(double), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail("storing the RoPE frequencies", e);
    p->inv_freq = h->gr_inv;
  }
  int rc = mtp::gr_pack(*p, h->w.pre_proj, h->w.post_proj, h->w.centroids, q, o, g, u, d,
                        static_cast<unsigned char*>(h->gr_img), 0);
  if (rc) return rc;
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail("packing the grid path's weight images", e);
  p->img = static_cast<const unsigned char*>(h->gr_img);
  p->img_bytes = p->L.img_bytes;
  p->mb = h->gr_mb;
  p->mb_words = h->gr_mb_words;
  h->gr_epoch = 64u;
  h->gr_ok = 1;
  return MTP_OK;
}

// Carves the workspace out of one allocation (sizes for max_batch sequences).
size_t layout_ws(mtp_handle* h, char* base) {
  const mtp_config& c = h->cfg;
  const size_t B = c.max_batch, H = c.hidden, bb = c.backbone, F = c.ffn;
  const size_t nh = c.n_head, dmax = h->dmax, ns = h->nsplit_max;
  const size_t C = c.use_ordered_embeddings ? c.n_centroids : 1, k = c.use_ordered_embeddings ? c.top_k : 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off = align256(off + bytes);
    return static_cast<void*>(p);
  };
  mtp::WsP& w = h->wsp;
  w.x[0] = static_cast<float*>(take(4 * B * H));
  w.x[1] = static_cast<float*>(take(4 * B * H));
  w.qraw = static_cast<float*>(take(4 * B * nh * dmax));
  w.part_ml = static_cast<float*>(take(4 * B * nh * ns * 2));
  w.part_acc = static_cast<float*>(take(4 * B * nh * ns * dmax));
  w.o = static_cast<float*>(take(4 * B * nh * dmax));
  w.ao = static_cast<float*>(take(4 * B * H));
  w.gate = static_cast<float*>(take(4 * B * F));
  w.up = static_cast<float*>(take(4 * B * F));
  w.dn = static_cast<float*>(take(4 * B * H));
  w.y = static_cast<float*>(take(4 * B * H));
  w.h_cur = static_cast<float*>(take(4 * B * bb));
  w.cl = static_cast<float*>(take(4 * B * C));
  w.sel = static_cast<int*>(take(4 * B * k));
  w.best = static_cast<unsigned long long*>(take(8 * B));
  w.lmin = static_cast<float*>(take(4 * B));
  w.cs = static_cast<float2*>(take(8 * B * 2 * (dmax / 2)));
  w.bar = static_cast<unsigned int*>(take(16));
  w.status = static_cast<int*>(take(16));
  h->abort_word = static_cast<unsigned*>(take(16));
  w.nsplit_max = static_cast<int>(ns);
  w.dmax = static_cast<int>(dmax);
  return off;
}

// Splits of the shared-K range per attention item. An item is one warp; the splits fill
// `slots` warps (one wave) with at least 16 keys per split.
int choose_nsplit(int B, int nkv, int keys, int slots, int cap) {
  int ns = slots / (B * nkv);
  const int by_len = (keys + 15) / 16;
  if (ns > by_len) ns = by_len;
  if (ns > cap) ns = cap;
  return ns < 1 ? 1 : ns;
}

// Upper bound of the keys one sequence attends in a layer of type t.
int attended_keys(const mtp_config& c, const mtp_kv* kv, int t) {
  if (!kv) return 1;
  return t == 0 && c.window < kv->max_ctx ? c.window : kv->max_ctx;
}

int check_kv(const mtp_config& c, const mtp_kv* kv, int t, int max_ctx, const char* name) {
  if (!kv || !kv->k || !kv->ctx_len) {
    set_error("%s shared K is required (a %s layer exists) and must have k and ctx_len", name, name);
    return MTP_ERR_INVALID_ARG;
  }
  const int d = t ? c.head_dim_full : c.head_dim_swa;
  const int vec = c.dtype == MTP_DTYPE_BF16 ? 8 : 4;
  if (!aligned16(kv->k) || (kv->v && !aligned16(kv->v)) || kv->stride_t < static_cast<int64_t>(c.n_kv_head) * d ||
      kv->stride_t % vec || kv->stride_b % vec || kv->stride_b < 0) {
    set_error("%s K/V: pointers must be 16-byte aligned, stride_t >= n_kv_head*head_dim and strides multiples of %d",
              name, vec);
    return MTP_ERR_INVALID_ARG;
  }
  if (kv->max_ctx < 1 || kv->max_ctx > max_ctx) {
    set_error("%s max_ctx=%d outside [1, %d]", name, kv->max_ctx, max_ctx);
    return MTP_ERR_INVALID_ARG;
  }
  return MTP_OK;
}

mtp::Params base_params(const mtp_handle* h, int B) {
  const mtp_config& c = h->cfg;
  mtp::Params p;
  memset(&p, 0, sizeof(p));
  mtp::ShapeP& s = p.s;
  s.B = B;
  s.bb = c.backbone;
  s.H = c.hidden;
  s.nl = c.n_layers;
  s.nh = c.n_head;
  s.nkv = c.n_kv_head;
  s.F = c.ffn;
  s.V = c.vocab;
  s.ordered = c.use_ordered_embeddings ? 1 : 0;
  s.C = s.ordered ? c.n_centroids : 0;
  s.topk = s.ordered ? c.top_k : 0;
  s.vsc = s.ordered ? c.vocab / c.n_centroids : 0;
  s.nsm = h->num_sms;
  s.W = c.window;
  s.d[0] = c.head_dim_swa;
  s.d[1] = c.head_dim_full;
  for (int t = 0; t < 2; ++t) {
    const int d = s.d[t] > 0 ? s.d[t] : 1;
    s.scale[t] = c.attn_scale > 0.f ? c.attn_scale : 1.0f / sqrtf(static_cast<float>(d));
  }
  s.theta[0] = c.rope_theta_swa;
  s.theta[1] = c.rope_theta_full;
  s.eps = c.rms_eps;
  p.w = h->wsp;
  p.pre = h->w.pre_proj;
  p.post = h->w.post_proj;
  p.temb = h->w.token_embd;
  p.cent = h->w.centroids;
  p.tgt = h->target_embed;
  p.out_norm = h->w.out_norm;
  p.ord = h->w.token_ordering;
  for (int l = 0; l < c.n_layers; ++l) {
    const mtp_layer_weights& L = h->w.layer[l];
    mtp::LayerP& P = p.L[l];
    P.q = L.q;
    P.o = L.o;
    P.gate = L.gate;
    P.up = L.up;
    P.down = L.down;
    P.q_norm = L.q_norm;
    P.attn_norm = L.attn_norm;
    P.post_attn_norm = L.post_attn_norm;
    P.ffn_norm = L.ffn_norm;
    P.post_ffn_norm = L.post_ffn_norm;
    P.lambda = L.layer_scalar;
    P.type = c.layer_type[l];
  }
  p.temb_ord = h->temb_ord;
  p.spin_limit = h->dbg_spin > 0 ? h->dbg_spin : 4000000000LL;  // ~2 s at 2 GHz
  p.dbg_skip = h->dbg_skip;
  // automatic: per sequence. The rows that several sequences select are then re-read from L2
  // rather than HBM (the step's DRAM bytes match the cluster-major traversal's), and the
  // per-sequence gather keeps more loads in flight than the chunked cluster-major stream.
  s.head_dd = s.ordered && h->head_mode == MTP_HEAD_CLUSTER_MAJOR &&
              mtp::head_cm_supported(p, c.dtype == MTP_DTYPE_BF16 ? 2 : 4);
  return p;
}

// Frees every device and host allocation of a handle, also of one only partly built (its
// fields stay NULL until allocated), and the handle itself.
void release_handle(mtp_handle* h) {
  if (h->ws) cudaFree(h->ws);
  if (h->temb_ord) cudaFree(h->temb_ord);
  if (h->c2_stream) cudaFree(h->c2_stream);
  if (h->gr_img) cudaFree(h->gr_img);
  if (h->gr_mb) cudaFree(h->gr_mb);
  if (h->gr_inv) cudaFree(h->gr_inv);
  if (h->gr) free(h->gr);
  if (h->tc_mem) cudaFree(h->tc_mem);
  if (h->tc_wmem) cudaFree(h->tc_wmem);
  if (h->tc) free(h->tc);
  free(h);
}

int set_device(const mtp_handle* h) {
  cudaError_t e = cudaSetDevice(h->device);
  return e == cudaSuccess ? MTP_OK : cuda_fail("cudaSetDevice", e);
}

}  // namespace

// Runs a multi-launch draft block through the handle's graph cache: replays the instantiated
// graph when the parameters (every pointer and size the launches take) equal the cached
// ones, else captures run() on the internal stream and instantiates it. Falls back to
// direct launches on the caller's stream when graphs are not available.
template <typename Run>
int run_graph_cached(mtp_handle* h, int path, const mtp::Params& p, cudaStream_t st, Run run) {
  auto& G = h->gc;
  if (!G.cs) return run(st);
  if (!G.valid || G.path != path || memcmp(&G.key, &p, sizeof(p)) != 0) {
    if (G.valid) {
      cudaGraphExecDestroy(G.exec);
      G.valid = 0;
    }
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamBeginCapture(G.cs, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail("beginning the draft-block graph capture", e);
    const int rc = run(G.cs);
    e = cudaStreamEndCapture(G.cs, &graph);
    if (rc) {
      if (graph) cudaGraphDestroy(graph);
      cudaGetLastError();
      return rc;
    }
    if (e != cudaSuccess) return cuda_fail("ending the draft-block graph capture", e);
    e = cudaGraphInstantiate(&G.exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return cuda_fail("instantiating the draft-block graph", e);
    memcpy(&G.key, &p, sizeof(p));
    G.path = path;
    G.valid = 1;
  }
  cudaError_t e = cudaEventRecord(G.ev_in, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(G.cs, G.ev_in, 0);
  if (e == cudaSuccess) e = cudaGraphLaunch(G.exec, G.cs);
  if (e == cudaSuccess) e = cudaEventRecord(G.ev_out, G.cs);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, G.ev_out, 0);
  if (e != cudaSuccess) return cuda_fail("launching the draft-block graph", e);
  return MTP_OK;
}

extern "C" {

const char* mtp_last_error(void) { return mtp::g_err; }

int mtp_init_weights(const mtp_config* config, const mtp_weights* weights, const void* target_embed, mtp_handle** out) {
  mtp::g_err[0] = 0;
  if (!config || !weights || !out) {
    set_error("config, weights and out must be non-NULL");
    return MTP_ERR_INVALID_ARG;
  }
  *out = nullptr;
  int rc = validate_config(*config);
  if (rc) return rc;
  rc = validate_weights(*config, *weights, target_embed);
  if (rc) return rc;
  mtp_handle* h = static_cast<mtp_handle*>(calloc(1, sizeof(mtp_handle)));
  if (!h) {
    set_error("out of host memory");
    return MTP_ERR_INVALID_ARG;
  }
  h->cfg = *config;
  h->w = *weights;
  h->target_embed = target_embed;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) {
    free(h);
    return cuda_fail("querying the device", e);
  }
  if (config->use_ordered_embeddings) {
    rc = check_ordering(*config, weights->token_ordering);
    if (rc) {
      free(h);
      return rc;
    }
  }
  int dmax = 2;
  for (int l = 0; l < config->n_layers; ++l) {
    const int d = config->layer_type[l] ? config->head_dim_full : config->head_dim_swa;
    dmax = d > dmax ? d : dmax;
  }
  h->dmax = dmax;
  int ns = (config->max_ctx + 31) / 32;
  if (ns > 4 * h->num_sms) ns = 4 * h->num_sms;
  h->nsplit_max = ns < 1 ? 1 : ns;
  h->c2_ok = c2_supported(h) ? 1 : 0;
  h->temb_ord = nullptr;
  h->c2_stream = nullptr;
  h->ws_bytes = layout_ws(h, nullptr);
  e = cudaMalloc(&h->ws, h->ws_bytes);
  if (e != cudaSuccess) {
    free(h);
    return cuda_fail("allocating the workspace", e);
  }
  layout_ws(h, static_cast<char*>(h->ws));
  rc = build_tc(h);
  if (rc) {
    release_handle(h);
    return rc;
  }
  e = cudaMemset(h->ws, 0, h->ws_bytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    release_handle(h);
    return cuda_fail("clearing the workspace", e);
  }
  const int row_bytes = config->hidden * (config->dtype == MTP_DTYPE_BF16 ? 2 : 4);
  if (config->use_ordered_embeddings && row_bytes % 16 == 0) {
    // the cluster paths and the cluster-major head read token_embd rows in token_ordering
    // order (one contiguous block of vocab / n_centroids rows per centroid): a copy made once
    const size_t bytes = static_cast<size_t>(config->vocab) * row_bytes;
    e = cudaMalloc(&h->temb_ord, bytes);
    if (e == cudaSuccess) {
      rc = mtp::reorder_rows(weights->token_embd, weights->token_ordering, h->temb_ord, config->vocab, row_bytes,
                             0);
      e = rc ? cudaErrorUnknown : cudaDeviceSynchronize();
    }
    if (e != cudaSuccess) {
      release_handle(h);
      return rc ? rc : cuda_fail("building the cluster-ordered token_embd copy", e);
    }
  }
  if (!h->temb_ord) h->c2_ok = 0;
  rc = build_gr(h);
  if (rc) {
    release_handle(h);
    return rc;
  }
  // the streamed cluster path's weight streams: now when it is the automatic one-sequence
  // path (no grid plan), else when mtp_set_path first selects it
  if (h->c2_ok && !h->gr_ok) {
    rc = build_c2_stream(h);
    if (rc) {
      release_handle(h);
      return rc;
    }
  }
  // the graph cache's stream and events (graphs are skipped when they cannot be created)
  if (cudaStreamCreateWithFlags(&h->gc.cs, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->gc.ev_in, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->gc.ev_out, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    if (h->gc.ev_in) cudaEventDestroy(h->gc.ev_in);
    if (h->gc.cs) cudaStreamDestroy(h->gc.cs);
    h->gc.cs = nullptr;
    h->gc.ev_in = h->gc.ev_out = nullptr;
  }
  *out = h;
  return MTP_OK;
}

int mtp_draft_block(mtp_handle* h, const void* hidden, const int32_t* last_token, const mtp_kv* kv_sliding,
                    const mtp_kv* kv_full, const int32_t* pos, int32_t B, int32_t n_draft, int32_t* out_tokens,
                    float* out_hidden, void* stream) {
  mtp::g_err[0] = 0;
  if (!h) {
    set_error("handle is NULL");
    return MTP_ERR_INVALID_ARG;
  }
  const mtp_config& c = h->cfg;
  if (!hidden || !last_token || !pos || !out_tokens) {
    set_error("hidden, last_token, pos and out_tokens must be non-NULL");
    return MTP_ERR_INVALID_ARG;
  }
  if (!aligned16(hidden)) {
    set_error("hidden must be 16-byte aligned");
    return MTP_ERR_INVALID_ARG;
  }
  if (B < 1 || B > c.max_batch) {
    set_error("B=%d outside [1, max_batch=%d]", B, c.max_batch);
    return MTP_ERR_INVALID_ARG;
  }
  if (n_draft < 1 || n_draft > 1024) {
    set_error("n_draft=%d outside [1, 1024]", n_draft);
    return MTP_ERR_INVALID_ARG;
  }
  int rc;
  if (has_type(c, 0) && (rc = check_kv(c, kv_sliding, 0, c.max_ctx, "sliding"))) return rc;
  if (has_type(c, 1) && (rc = check_kv(c, kv_full, 1, c.max_ctx, "full"))) return rc;
  if ((rc = set_device(h))) return rc;
  mtp::Params p = base_params(h, B);
  p.hidden_in = hidden;
  p.tok_in = last_token;
  p.pos = pos;
  p.out_tokens = out_tokens;
  p.out_hidden = out_hidden;
  p.n_draft = n_draft;
  const mtp_kv* kvs[2] = {kv_sliding, kv_full};
  for (int t = 0; t < 2; ++t) {
    if (!has_type(c, t)) continue;
    p.kv[t].k = kvs[t]->k;
    p.kv[t].v = kvs[t]->v;
    p.kv[t].ctx_len = kvs[t]->ctx_len;
    p.kv[t].sb = kvs[t]->stride_b;
    p.kv[t].st = kvs[t]->stride_t;
    p.kv[t].max_ctx = kvs[t]->max_ctx;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf16 = c.dtype == MTP_DTYPE_BF16;
  int path = h->path;
  if (path == 7 || (path == 0 && B == 1 && h->gr_ok)) {
    if (!h->gr_ok || B != 1) {
      set_error("the grid path runs one sequence of a supported shape (B=%d, available=%d)", B, h->gr_ok);
      return MTP_ERR_UNSUPPORTED_SHAPE;
    }
    mtp::gr::Params& gp = *h->gr;
    for (int t = 0; t < 2; ++t) {
      if (!gp.has_type[t]) continue;
      if (kvs[t]->v && kvs[t]->v != kvs[t]->k) {
        set_error("the grid path reads V = K (attention_k_eq_v); pass v = NULL or v = k");
        return MTP_ERR_UNSUPPORTED_SHAPE;
      }
      if ((reinterpret_cast<uintptr_t>(kvs[t]->k) & 15) != 0 || (kvs[t]->stride_t * 2) % 16 != 0) {
        set_error("the grid path needs 16-byte aligned K rows");
        return MTP_ERR_UNSUPPORTED_SHAPE;
      }
      gp.k[t] = static_cast<const __nv_bfloat16*>(kvs[t]->k);
      gp.ctx_len[t] = kvs[t]->ctx_len;
      gp.st[t] = kvs[t]->stride_t;
      gp.kv_max[t] = kvs[t]->max_ctx;
    }
    gp.hidden_in = static_cast<const __nv_bfloat16*>(hidden);
    gp.tok_in = last_token;
    gp.pos = pos;
    gp.out_tokens = out_tokens;
    gp.out_hidden = out_hidden;
    gp.n_draft = n_draft;
    gp.status = h->wsp.status;
    gp.abort_flag = h->abort_word;
    gp.spin_limit = h->dbg_spin > 0 ? h->dbg_spin : 4000000000LL;
    gp.dbg_skip = h->dbg_skip;
    const unsigned need = static_cast<unsigned>(n_draft + 1) * mtp::gr::kExPerStep;
    if (h->gr_epoch > 0xF0000000u - need) {
      // epochs wrap: clear the mailboxes and the abort word (which holds the epoch base of a
      // launch that gave up) so that no old word can match a new epoch
      cudaError_t e = cudaMemsetAsync(h->gr_mb, 0, static_cast<size_t>(h->gr_mb_words) * 8, st);
      if (e == cudaSuccess) e = cudaMemsetAsync(h->abort_word, 0, sizeof(unsigned), st);
      if (e != cudaSuccess) return cuda_fail("clearing the grid path's mailboxes", e);
      h->gr_epoch = 64u;
    }
    gp.epoch_base = h->gr_epoch;
    h->gr_epoch += need;
    return mtp::run_gr(gp, st);
  }
  if (path == 6 || (path == 0 && B == 1 && h->c2_ok)) {
    if (!h->c2_ok || !h->c2_stream || B != 1) {
      set_error("the streamed cluster path runs one sequence of a supported shape (B=%d, available=%d)", B, h->c2_ok);
      return MTP_ERR_UNSUPPORTED_SHAPE;
    }
    const int kvm = has_type(c, 1) ? kv_full->max_ctx : kv_sliding->max_ctx;
    mtp::c2::Params cp = c2_template(h, kvm);
    for (int t = 0; t < 2; ++t) {
      if (!cp.has_type[t]) continue;
      if (kvs[t]->v && kvs[t]->v != kvs[t]->k) {
        set_error("the streamed cluster path reads V = K (attention_k_eq_v); pass v = NULL or v = k");
        return MTP_ERR_UNSUPPORTED_SHAPE;
      }
      cp.k[t] = static_cast<const __nv_bfloat16*>(kvs[t]->k);
      cp.ctx_len[t] = kvs[t]->ctx_len;
      cp.st[t] = kvs[t]->stride_t;
      cp.kv_max[t] = kvs[t]->max_ctx;
      if ((reinterpret_cast<uintptr_t>(kvs[t]->k) & 15) != 0) {
        set_error("the streamed cluster path needs 16-byte aligned K rows");
        return MTP_ERR_UNSUPPORTED_SHAPE;
      }
    }
    cp.hidden_in = static_cast<const __nv_bfloat16*>(hidden);
    cp.tok_in = last_token;
    cp.pos = pos;
    cp.out_tokens = out_tokens;
    cp.out_hidden = out_hidden;
    cp.n_draft = n_draft;
    cp.status = h->wsp.status;
    cp.abort_flag = h->abort_word;
    cp.spin_limit = h->dbg_spin > 0 ? h->dbg_spin : 4000000000LL;
    cp.dbg_skip = h->dbg_skip;
    const int smem = mtp::c2_smem_bytes(cp);
    if (smem <= 0 || (reinterpret_cast<uintptr_t>(hidden) & 15) != 0) {
      set_error("streamed cluster path: shape, K stride or hidden alignment not supported for this call");
      return MTP_ERR_UNSUPPORTED_SHAPE;
    }
    cudaError_t e = cudaMemsetAsync(h->abort_word, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return cuda_fail("clearing the abort word", e);
    return mtp::run_c2(cp, smem, st);
  }
  const int ncta = h->num_sms;
  if (path == 5 || (path == 0 && B >= 2 && h->tc)) {
    if (!h->tc) {
      set_error("the tensor-core path needs a bf16 drafter with max_batch in [2, %d] on this device", mtp::tc::kMaxB);
      return MTP_ERR_UNSUPPORTED_SHAPE;
    }
    p.s.ncta_hint = 2 * h->num_sms;
    // the tensor-core attention runs one CTA per (sequence, KV head, split): splits for about
    // two waves of CTAs at the number of them that fit an SM's shared memory
    for (int t = 0; t < 2; ++t) {
      if (!has_type(c, t)) {
        p.s.nsplit[t] = 1;
        continue;
      }
      const int d = t ? c.head_dim_full : c.head_dim_swa;
      const int sm = mtp::att_tc_smem(d, c.n_kv_head > 0 ? c.n_head / c.n_kv_head : 0);
      const int per_sm = sm > 0 ? (232448 / sm > 0 ? 232448 / sm : 1) : mtp::kWarps;
      p.s.nsplit[t] = choose_nsplit(B, c.n_kv_head, attended_keys(c, kvs[t], t), 2 * per_sm * h->num_sms,
                                    h->nsplit_max);
    }
    return run_graph_cached(h, 5, p, st, [&](cudaStream_t s2) { return mtp::run_phases_tc_bf16(p, *h->tc, s2); });
  }
  if (path != 1) {
    p.s.ncta_hint = ncta;
    for (int t = 0; t < 2; ++t)
      p.s.nsplit[t] = has_type(c, t) ? choose_nsplit(B, c.n_kv_head, attended_keys(c, kvs[t], t), mtp::kWarps * ncta,
                                                     h->nsplit_max) : 1;
    const int cap = bf16 ? mtp::persistent_capacity_bf16(p, h->num_sms) : mtp::persistent_capacity_f32(p, h->num_sms);
    if (cap >= ncta) {
      // the persistent kernel keeps the per-sequence gather: the cluster-major head reads the
      // top-k phase's lists with bulk copies, which want a kernel boundary after those writes
      p.s.head_dd = 0;
      return bf16 ? mtp::run_persistent_bf16(p, st) : mtp::run_persistent_f32(p, st);
    }
    if (path == 2) {
      set_error("persistent draft-block kernel cannot be co-resident for this shape");
      return MTP_ERR_UNSUPPORTED_SHAPE;
    }
  }
  p.s.ncta_hint = 2 * h->num_sms;
  for (int t = 0; t < 2; ++t)
    p.s.nsplit[t] = has_type(c, t) ? choose_nsplit(B, c.n_kv_head, attended_keys(c, kvs[t], t), mtp::kWarps * h->num_sms,
                                                   h->nsplit_max) : 1;
  return run_graph_cached(h, 1, p, st,
                          [&](cudaStream_t s2) { return bf16 ? mtp::run_phases_bf16(p, s2) : mtp::run_phases_f32(p, s2); });
}

int mtp_centroid_head(mtp_handle* h, const float* y, int32_t B, float* out_logits, int32_t* out_token,
                      int32_t* out_centroids, void* stream) {
  mtp::g_err[0] = 0;
  if (!h || !y || !out_token) {
    set_error("handle, y and out_token must be non-NULL");
    return MTP_ERR_INVALID_ARG;
  }
  const mtp_config& c = h->cfg;
  if (B < 1 || B > c.max_batch) {
    set_error("B=%d outside [1, max_batch=%d]", B, c.max_batch);
    return MTP_ERR_INVALID_ARG;
  }
  if (!c.use_ordered_embeddings && out_centroids) {
    set_error("out_centroids must be NULL for the dense head");
    return MTP_ERR_INVALID_ARG;
  }
  int rc;
  if ((rc = set_device(h))) return rc;
  mtp::Params p = base_params(h, B);
  p.s.ncta_hint = 2 * h->num_sms;
  p.y_in = y;
  p.out_logits = out_logits;
  p.out_tokens = out_token;
  p.out_centroids = out_centroids;
  p.mask_mode = h->mask_mode;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return c.dtype == MTP_DTYPE_BF16 ? mtp::run_head_bf16(p, st) : mtp::run_head_f32(p, st);
}

int mtp_set_logit_mask(mtp_handle* h, int32_t mode) {
  mtp::g_err[0] = 0;
  if (!h || (mode != MTP_MASK_NEG_1E30 && mode != MTP_MASK_MIN_MINUS_ONE)) {
    set_error("need a handle and mode MTP_MASK_NEG_1E30 (0) or MTP_MASK_MIN_MINUS_ONE (1), got %d", mode);
    return MTP_ERR_INVALID_ARG;
  }
  h->mask_mode = mode;
  return MTP_OK;
}

int mtp_set_sparse_head(mtp_handle* h, int32_t mode) {
  mtp::g_err[0] = 0;
  if (!h || mode < MTP_HEAD_AUTO || mode > MTP_HEAD_CLUSTER_MAJOR) {
    set_error("need a handle and mode MTP_HEAD_AUTO (0), MTP_HEAD_PER_SEQUENCE (1) or MTP_HEAD_CLUSTER_MAJOR (2), got %d",
              mode);
    return MTP_ERR_INVALID_ARG;
  }
  h->head_mode = mode;
  return MTP_OK;
}

int mtp_set_debug(mtp_handle* h, int32_t skip_arrival_cta, int64_t spin_limit_cycles) {
  mtp::g_err[0] = 0;
  if (!h || skip_arrival_cta < -1 || spin_limit_cycles < 0) {
    set_error("need a handle, skip_arrival_cta >= -1 and spin_limit_cycles >= 0");
    return MTP_ERR_INVALID_ARG;
  }
  h->dbg_skip = skip_arrival_cta + 1;
  h->dbg_spin = spin_limit_cycles;
  return MTP_OK;
}

int mtp_verify_greedy(const void* target_logits, const int32_t* draft, int32_t B, int32_t n, int32_t V,
                      int32_t* accept_len, int32_t* out_tokens, void* stream) {
  mtp::g_err[0] = 0;
  if (!target_logits || !accept_len || !out_tokens || (n > 0 && !draft)) {
    set_error("target_logits, draft (n > 0), accept_len and out_tokens must be non-NULL");
    return MTP_ERR_INVALID_ARG;
  }
  if (B < 1 || n < 0 || V < 1 || V % 8 || !aligned16(target_logits)) {
    set_error("need B >= 1, n >= 0, V >= 1 with V %% 8 == 0 and 16-byte aligned logits (B=%d n=%d V=%d)", B, n, V);
    return MTP_ERR_INVALID_ARG;
  }
  return mtp::run_verify(target_logits, draft, B, n, V, accept_len, out_tokens, static_cast<cudaStream_t>(stream));
}

int mtp_verify_sample(const void* target_logits, const int32_t* draft, int32_t B, int32_t n, int32_t V,
                      float temperature, const float* u_accept, const float* u_sample, int32_t* accept_len,
                      int32_t* out_tokens, void* stream) {
  mtp::g_err[0] = 0;
  if (!target_logits || !accept_len || !out_tokens || (n > 0 && (!draft || !u_accept)) || !u_sample) {
    set_error("target_logits, draft and u_accept (n > 0), u_sample, accept_len and out_tokens must be non-NULL");
    return MTP_ERR_INVALID_ARG;
  }
  if (B < 1 || n < 0 || V < 1 || V % 8 || !aligned16(target_logits) || !(temperature >= 0.f) ||
      temperature > 3.0e38f) {
    set_error("need B >= 1, n >= 0, V >= 1 with V %% 8 == 0, 16-byte aligned logits and a finite temperature >= 0 "
              "(B=%d n=%d V=%d T=%g)", B, n, V, static_cast<double>(temperature));
    return MTP_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (temperature == 0.f) return mtp::run_verify(target_logits, draft, B, n, V, accept_len, out_tokens, st);
  return mtp::run_verify_sample(target_logits, draft, B, n, V, temperature, u_accept, u_sample, accept_len, out_tokens,
                                st);
}

int mtp_get_status(mtp_handle* h) {
  mtp::g_err[0] = 0;
  if (!h) {
    set_error("handle is NULL");
    return MTP_ERR_INVALID_ARG;
  }
  int rc;
  if ((rc = set_device(h))) return rc;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail("device synchronisation", e);
  int status = 0;
  e = cudaMemcpy(&status, h->wsp.status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail("reading the status word", e);
  if (status != 0) {
    e = cudaMemset(h->wsp.status, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail("clearing the status word", e);
    set_error("a device-side wait timed out (status %d)", status);
  }
  return status;
}

int mtp_set_path(mtp_handle* h, int32_t path) {
  mtp::g_err[0] = 0;
  if (!h || path < 0 || path > 7 || path == 3 || path == 4) {
    set_error("need a handle and path in {0, 1, 2, 5, 6, 7}");
    return MTP_ERR_INVALID_ARG;
  }
  if (path == 6 && h->c2_ok && !h->c2_stream) {
    cudaSetDevice(h->device);
    const int rc = build_c2_stream(h);  // allocates and packs once; synchronises
    if (rc) return rc;
  }
  h->path = path;
  return MTP_OK;
}

void mtp_destroy(mtp_handle* h) {
  if (!h) return;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  if (h->gc.valid) cudaGraphExecDestroy(h->gc.exec);
  if (h->gc.ev_in) cudaEventDestroy(h->gc.ev_in);
  if (h->gc.ev_out) cudaEventDestroy(h->gc.ev_out);
  if (h->gc.cs) cudaStreamDestroy(h->gc.cs);
  release_handle(h);
}

}  // extern "C"
