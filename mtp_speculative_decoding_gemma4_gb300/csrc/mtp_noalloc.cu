// mtp_centroid_head_noalloc: the centroid LM head for callers that cannot allocate device
// memory. It runs the same head kernels as mtp_centroid_head, but takes the head's tensors
// as plain pointers (no handle, whose creation allocates a workspace) and keeps its scratch
// (centroid logits, selected centroids, per-sequence argmax keys, a copy of y) in one
// file-scope device array instead of memory from cudaMalloc.
#include <cstring>
#include <mutex>

#include "mtp.h"
#include "mtp_launch.h"
#include "mtp_phases.cuh"

namespace {

constexpr size_t kScratchBytes = MTP_NOALLOC_SCRATCH_BYTES;

// Shared by every call on a device and held by every GPU that loads the library until the
// process exits. Calls that overlap on the GPU race on it.
static __device__ __align__(256) unsigned char g_head_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_head_scratch on the current device; resolved once per device (the
// host-side symbol is only a stand-in and must never be handed to a kernel).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    mtp::set_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    mtp::set_error("device ordinal %d beyond the %d devices this entry point tracks", dev, kMaxDevices);
    return MTP_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_head_scratch);
    if (e != cudaSuccess || !p) {
      mtp::set_error("cudaGetSymbolAddress(g_head_scratch): %s", cudaGetErrorString(e));
      return MTP_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MTP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

}  // namespace

extern "C" MTP_API int mtp_centroid_head_noalloc(const float* y, const void* centroids,
                                                 const int32_t* token_ordering, const void* token_embd,
                                                 int32_t dtype, int32_t B, int32_t hidden, int32_t n_centroids,
                                                 int32_t top_k, int32_t vocab, float* out_logits,
                                                 int32_t* out_token, int32_t* out_centroids, void* stream) {
  mtp::set_error("%s", "");
  if (!y || !centroids || !token_ordering || !token_embd || !out_token) {
    mtp::set_error("y, centroids, token_ordering, token_embd and out_token must be non-NULL");
    return MTP_ERR_INVALID_ARG;
  }
  if (!aligned16(y) || !aligned16(centroids) || !aligned16(token_embd)) {
    mtp::set_error("y, centroids and token_embd must be 16-byte aligned");
    return MTP_ERR_INVALID_ARG;
  }
  if (dtype != MTP_DTYPE_BF16 && dtype != MTP_DTYPE_F32) {
    mtp::set_error("dtype=%d is neither BF16 nor F32", dtype);
    return MTP_ERR_INVALID_ARG;
  }
  const int vec = dtype == MTP_DTYPE_BF16 ? 8 : 4;
  if (B < 1 || hidden < vec || hidden % vec || n_centroids < 1 || n_centroids > 8192 || top_k < 1 || top_k > 64 ||
      top_k > n_centroids || vocab < 1) {
    mtp::set_error("need B >= 1, hidden a positive multiple of %d, 1 <= top_k <= min(64, n_centroids), "
                   "n_centroids <= 8192 (B=%d hidden=%d C=%d k=%d)", vec, B, hidden, n_centroids, top_k);
    return MTP_ERR_INVALID_ARG;
  }
  if (vocab % n_centroids) {
    mtp::set_error("vocab=%d is not a multiple of n_centroids=%d", vocab, n_centroids);
    return MTP_ERR_BAD_ORDERING;
  }
  // scratch layout: centroid logits [B][C], selected [B][k], argmax keys [B], y copy [B][H]
  const size_t cl_b = round256(4ull * B * n_centroids), sel_b = round256(4ull * B * top_k),
               best_b = round256(8ull * B), y_b = round256(4ull * B * hidden);
  const size_t need = cl_b + sel_b + best_b + y_b;
  if (need > kScratchBytes) {
    mtp::set_error("B=%d, n_centroids=%d, top_k=%d, hidden=%d need %zu bytes of scratch; this entry point's static "
                   "scratch holds %zu bytes", B, n_centroids, top_k, hidden, need, kScratchBytes);
    return MTP_ERR_INVALID_ARG;
  }
  void* base = nullptr;
  int rc = scratch_address(&base);
  if (rc) return rc;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    mtp::set_error("querying the device: %s", cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }

  mtp::Params p;
  memset(&p, 0, sizeof(p));
  mtp::ShapeP& s = p.s;
  s.B = B;
  s.H = hidden;
  s.bb = hidden;
  s.F = hidden;
  s.nl = 0;
  s.nh = 1;
  s.nkv = 1;
  s.d[0] = s.d[1] = 32;
  s.V = vocab;
  s.C = n_centroids;
  s.topk = top_k;
  s.vsc = vocab / n_centroids;
  s.ordered = 1;
  s.ncta_hint = 2 * sms;
  char* sc = static_cast<char*>(base);
  p.w.cl = reinterpret_cast<float*>(sc);
  p.w.sel = reinterpret_cast<int*>(sc + cl_b);
  p.w.best = reinterpret_cast<unsigned long long*>(sc + cl_b + sel_b);
  p.w.y = reinterpret_cast<float*>(sc + cl_b + sel_b + best_b);
  p.w.dmax = 32;
  p.w.nsplit_max = 1;
  p.cent = centroids;
  p.ord = token_ordering;
  p.temb = token_embd;
  p.y_in = y;
  p.out_logits = out_logits;
  p.out_tokens = out_token;
  p.out_centroids = out_centroids;
  // token_ordering is not validated here (a permutation check would need scratch of V
  // entries): the gather skips any id outside [0, vocab) instead of reading or writing out
  // of bounds
  p.check_ids = 1;
  // the argmax keys must start at zero: the head-entry phase clears them before use
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return dtype == MTP_DTYPE_BF16 ? mtp::run_head_bf16(p, st) : mtp::run_head_f32(p, st);
}
