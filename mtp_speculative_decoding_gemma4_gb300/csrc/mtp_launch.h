// Internal interface between the C ABI (mtp_api.cu) and the dtype-specific kernel
// translation units (mtp_bf16.cu, mtp_f32.cu, mtp_c2.cu, mtp_grid.cu, mtp_tc.cu, mtp_verify.cu, ...).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mtp.h"

namespace mtp {

struct Params;
namespace c2 {
struct Params;
}
namespace gr {
struct Params;
}

// Records the calling thread's last error text (printf-style).
void set_error(const char* fmt, ...);

int run_phases_bf16(const Params& p, cudaStream_t st);
int run_persistent_bf16(const Params& p, cudaStream_t st);
int persistent_capacity_bf16(const Params& p, int num_sms);
int run_head_bf16(const Params& p, cudaStream_t st);

int run_phases_f32(const Params& p, cudaStream_t st);
int run_persistent_f32(const Params& p, cudaStream_t st);
int persistent_capacity_f32(const Params& p, int num_sms);
int run_head_f32(const Params& p, cudaStream_t st);

// Cluster-major sparse head (streams each selected centroid's rows of the token_ordering-order
// token_embd copy once per step): whether the shape and pointers allow it, and the launch.
bool head_cm_supported(const Params& p, int elem_bytes);
template <typename WT>
int run_head_cm(const Params& p, cudaStream_t st);

// token_embd rows in token_ordering order (dst[j] = src[ord[j]], rows of row_bytes, a
// multiple of 16): the rows of one centroid become one contiguous block.
int reorder_rows(const void* src, const int* ord, void* dst, int V, int row_bytes, cudaStream_t st);

// Streamed-tile cluster draft block (one sequence, one 16-CTA cluster, weights packed into
// per-CTA tile streams at init): shared-memory bytes (0: shape
// not supported), resident clusters for that size, launch; the packed stream's size and the
// packing of every projection (mats indexed like the step sequence, K entries unused).
int c2_smem_bytes(const c2::Params& p);
int c2_capacity(int smem);
int run_c2(const c2::Params& p, int smem, cudaStream_t st);
long long c2_stream_total(const c2::Params& p);
int c2_pack_all(const c2::Params& p, const void* const* mats, void* dst, cudaStream_t st);

// Grid draft block (one sequence, every co-resident cluster, split weights resident in shared
// memory): the plan (cluster size, grid, layout; returns the shared-memory bytes, 0 when the
// shape is not supported), the per-CTA weight images, the mailbox offsets (returns the words
// of both step parities) and the launch.
int gr_plan(gr::Params& p, int optin);
long long gr_image_total(const gr::Params& p);
int gr_pack(const gr::Params& p, const void* pre, const void* post, const void* cent, const void* const* q,
            const void* const* o, const void* const* gate, const void* const* up, const void* const* down,
            unsigned char* dst, cudaStream_t st);
long long gr_mailboxes(gr::Params& p);
int run_gr(const gr::Params& p, cudaStream_t st);

// Tensor maps of the tensor-core phase path (host memory; see mtp_tc.cuh): every weight
// matrix, and the staged input terms [3][bp][K] for each input width K.
struct TcPlan {
  CUtensorMap pre, post, cent, temb;
  CUtensorMap q[MTP_MAX_LAYERS], o[MTP_MAX_LAYERS], gate[MTP_MAX_LAYERS], up[MTP_MAX_LAYERS], down[MTP_MAX_LAYERS];
  CUtensorMap xs_pre, xs_h, xs_o[2], xs_f;  // K = 2 backbone, hidden, n_head * head_dim (sliding, full), ffn
  // stacked copies of projections that read the same input, one launch each: [gate ; up] of
  // every layer ([2 ffn][hidden], interleaved in 64-row blocks for the gated-GELU epilogue,
  // which writes the down projection's operand into xs_glu, mapped by xs_f2) and
  // [post_proj ; centroids] ([bb + C][hidden]); 0 in the flags when the shape does not tile
  CUtensorMap gu[MTP_MAX_LAYERS], postc, xs_f2;
  __nv_bfloat16* xs_glu;
  int gu_ok, postc_ok;
  __nv_bfloat16* xs;                         // the staging buffer
  int bp;                                    // sequences of the staged terms (multiple of 32)
};
// Split-KV attention of layer l on tensor cores (bf16, V = K, head_dim in {64, 128, 256, 512},
// at most 4 query heads per KV head): one CTA per (sequence, KV head, split), partials in the
// layout of the CUDA-core attention phase.
bool att_tc_supported(const Params& p, int l);
int att_tc_smem(int D, int hpg);  // shared-memory bytes of one CTA (0: no kernel for the shape)
int run_att_tc(const Params& p, int l, cudaStream_t st);

// One launch per phase with every GEMV as staging + tcgen05 GEMMs (bf16, B <= bp).
int run_phases_tc_bf16(const Params& p, const TcPlan& plan, cudaStream_t st);

int run_verify(const void* logits, const int* draft, int B, int n, int V, int* accept_len, int* out_tokens,
               cudaStream_t st);
// Sampled verification at temperature > 0 (one CTA per sequence).
int run_verify_sample(const void* logits, const int* draft, int B, int n, int V, float temperature,
                      const float* u_accept, const float* u_sample, int* accept_len, int* out_tokens, cudaStream_t st);

}  // namespace mtp
