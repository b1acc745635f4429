/*
 * mtp.h -- C ABI of libmtp: the Gemma-4-assistant Multi-Token-Prediction drafter step,
 * draft block and greedy verification on one NVIDIA GB300 (sm_103a).
 *
 * Conventions for every entry point
 *   - Pointers named "device" are CUDA device pointers (cudaMalloc / torch CUDA tensors)
 *     on the current device; the library borrows them and never frees them.
 *   - Matrices are row-major [out][in]; "model dtype" means bf16 (MTP_DTYPE_BF16) or fp32
 *     (MTP_DTYPE_F32) as fixed at init. Norm gains are always fp32.
 *   - Device pointers must be 16-byte aligned; row strides are multiples of 16 bytes.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Calls
 *     only enqueue work on it and return; nothing synchronises except mtp_init_weights,
 *     mtp_get_status and mtp_destroy.
 *   - Return value: MTP_OK or an MTP_ERR_* code; on error nothing was enqueued and
 *     mtp_last_error() describes the cause (per calling thread).
 *
 * Precision contract (both this library and its CPU oracle): stored tensors (weights,
 * shared K, embedding tables, the caller's hidden state, target logits) are bf16, or fp32
 * for fp32 models. Activations are fp32 and are never rounded to a narrower type: no
 * projection input, attention operand or intermediate vector is rounded to bf16, and the
 * post-projected hidden state carried to the next draft step stays fp32 (unrounded).
 * Top-k and argmax decide on fp32 values, ties going to the lower centroid index / lower
 * vocabulary id.
 */
#ifndef MTP_H_
#define MTP_H_

#include <stdint.h>

#if defined(__GNUC__)
#define MTP_API __attribute__((visibility("default")))
#else
#define MTP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MTP_MAX_LAYERS 8

enum mtp_status {
  MTP_OK = 0,
  MTP_ERR_INVALID_ARG = 1,       /* NULL / out-of-range argument (missing hidden or KV included) */
  MTP_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside what the kernels implement */
  MTP_ERR_BAD_ORDERING = 3,      /* vocab % n_centroids != 0 or ordering not a permutation */
  MTP_ERR_CUDA = 4,              /* a CUDA runtime call failed */
  MTP_ERR_TIMEOUT = 5            /* a device-side wait gave up (reported by mtp_get_status) */
};

enum mtp_dtype { MTP_DTYPE_BF16 = 0, MTP_DTYPE_F32 = 1 };

/* Value of the vocabulary entries outside the selected clusters in a materialised logits row
 * of the centroid head: -1e30f ("Gemma 4 Assistant tensor inventory", "Centroid / ordered
 * embeddings LM head", step 5: dense fill, then the sparse logits set at their ids), or the
 * smallest selected logit minus one ("Gemma 4 Assistant 使用指南", section 五, step 3 of
 * use_ordered_embeddings; named there as the MLX-style alternative). The argmax is the same
 * either way. */
enum mtp_logit_mask { MTP_MASK_NEG_1E30 = 0, MTP_MASK_MIN_MINUS_ONE = 1 };
enum mtp_layer_kind { MTP_LAYER_SLIDING = 0, MTP_LAYER_FULL = 1 };
/* Traversal of the sparse head (the candidate-row gather and GEMV, steps 3-4 of "Gemma 4
 * Assistant tensor inventory", "Centroid / ordered embeddings LM head"): per sequence (each
 * sequence reads the rows of its own top_k clusters), or cluster-major (each distinct
 * selected cluster is streamed once per step, with bulk copies, for every sequence that
 * selected it). Both give the same selected sets and the same logits up to fp32 summation
 * order. AUTO: per sequence (on GB300 the L2 already serves the rows that sequences share,
 * and the per-sequence gather was the faster of the two at every batch measured). */
enum mtp_sparse_head { MTP_HEAD_AUTO = 0, MTP_HEAD_PER_SEQUENCE = 1, MTP_HEAD_CLUSTER_MAJOR = 2 };

/* Drafter hyper-parameters.
 * Cited: "Gemma 4 Multi-Token Prediction (MTP) drafter", sections "Conversion" (metadata
 * keys backbone_hidden_size, num_centroids, centroid_intermediate_top_k,
 * use_ordered_embeddings) and "Tensor schema"; "Gemma 4 Assistant tensor inventory",
 * "HF config highlights" (layer_types, attention_k_eq_v, vocab_size, hidden_size). */
typedef struct mtp_config {
  int32_t backbone;        /* target hidden size bb (pre_projection input is 2*bb) */
  int32_t hidden;          /* assistant hidden size H */
  int32_t n_layers;        /* 1..MTP_MAX_LAYERS */
  int32_t n_head;          /* query heads */
  int32_t head_dim_swa;    /* head dim of sliding layers (and of the sliding shared K) */
  int32_t head_dim_full;   /* head dim of full layers (and of the full shared K) */
  int32_t n_kv_head;       /* shared KV heads; n_head % n_kv_head == 0 */
  int32_t ffn;             /* MLP intermediate size */
  int32_t vocab;           /* V */
  int32_t n_centroids;     /* C (ordered embeddings only) */
  int32_t top_k;           /* selected centroids (ordered embeddings only), <= 64 */
  int32_t window;          /* sliding window W (keys attended by sliding layers) */
  int32_t use_ordered_embeddings; /* 1: centroid head; 0: dense tied head */
  int32_t dtype;           /* enum mtp_dtype */
  int32_t max_batch;       /* largest B any later call will pass (sizes the workspace) */
  int32_t max_ctx;         /* largest shared-K length any later call will pass */
  uint8_t layer_type[MTP_MAX_LAYERS]; /* enum mtp_layer_kind per block */
  float rms_eps;           /* RMSNorm epsilon (1e-6) */
  float attn_scale;        /* softmax scale; 0 -> 1/sqrt(head_dim) */
  float rope_theta_swa;    /* RoPE base of sliding layers; 0 disables RoPE */
  float rope_theta_full;   /* RoPE base of full layers; 0 disables RoPE */
} mtp_config;

/* Per-block tensors ("Tensor schema": attn_q, attn_q_norm, attn_output, attn_norm,
 * post_attention_norm, ffn_norm, post_ffw_norm, ffn_gate/up/down, layer_output_scale).
 * There are no K/V projections: the drafter is Q-only and reads the target's K. */
typedef struct mtp_layer_weights {
  const void *q;      /* device [n_head*d][H], model dtype */
  const void *o;      /* device [H][n_head*d] */
  const void *gate;   /* device [ffn][H] */
  const void *up;     /* device [ffn][H] */
  const void *down;   /* device [H][ffn] */
  const float *q_norm;          /* device [d] */
  const float *attn_norm;       /* device [H] */
  const float *post_attn_norm;  /* device [H] */
  const float *ffn_norm;        /* device [H] */
  const float *post_ffn_norm;   /* device [H] */
  float layer_scalar;           /* host value: multiplies the residual after the block */
} mtp_layer_weights;

typedef struct mtp_weights {
  const void *pre_proj;     /* device [H][2*bb]  (input [target_hidden ; embed(token)]) */
  const void *post_proj;    /* device [bb][H] */
  const void *token_embd;   /* device [V][H]: tied LM head rows */
  const void *centroids;    /* device [C][H] (ordered embeddings only, else NULL) */
  const float *out_norm;    /* device [H] */
  const int32_t *token_ordering; /* device [V] viewed [C][V/C]: centroid c owns ids
                                    ordering[c*V/C .. (c+1)*V/C) (ordered only) */
  mtp_layer_weights layer[MTP_MAX_LAYERS];
} mtp_weights;

/* Shared K of one attention type: the target's last layer of that type
 * ("Gemma 4 Assistant 使用指南", section 二.4: shared_kv_states maps
 * "full_attention" / "sliding_attention" to (key, value)).
 * Element (b, t, kv_head, i) sits at k[b*stride_b + t*stride_t + kv_head*d + i].
 * v == NULL means V = K (attention_k_eq_v: "Gemma 4 Assistant tensor inventory",
 * "Notes for llama.cpp port" item 2); otherwise v has the same layout. ctx_len[b] >= 1 is the
 * number of valid keys of sequence b (right-padded storage; padding is never read); values
 * are clamped to [0, max_ctx] on the device, and a sequence with no keys attends nothing
 * (its attention output is 0). */
typedef struct mtp_kv {
  const void *k;           /* device, model dtype */
  const void *v;           /* device or NULL (V = K) */
  const int32_t *ctx_len;  /* device [B] */
  int64_t stride_b;        /* elements between sequences */
  int64_t stride_t;        /* elements between tokens (>= n_kv_head*d, multiple of 8) */
  int32_t max_ctx;         /* upper bound of ctx_len[*] (<= mtp_config.max_ctx) */
} mtp_kv;

typedef struct mtp_handle mtp_handle;

/* Validate the configuration and the weights, check token_ordering, allocate the
 * workspace for max_batch sequences, and return a handle.
 * The weight tensors must stay valid and unchanged while the handle lives: some paths read
 * them directly, others read device copies made here (token_embd in token_ordering order;
 * per-CTA weight images of the one-sequence grid path; for max_batch >= 2 in bf16, the
 * stacked [gate ; up] and [post_proj ; centroids] pairs of the tensor-core path).
 * config/weights: host structs (copied). target_embed: device [V][bb] model dtype, the
 * target's input embedding table that embed(last_token) reads ("Gemma 4 drafter
 * explained", "Target Activations": the input table is shared with the target).
 * Errors: INVALID_ARG (NULL pointer, bad field), UNSUPPORTED_SHAPE, BAD_ORDERING
 * (vocab % n_centroids != 0 -- "Gemma 4 Assistant tensor inventory", "GGUF / converter
 * layout" verification note -- or ordering not a permutation of 0..V-1), CUDA.
 * Synchronises the current device. */
MTP_API int mtp_init_weights(const mtp_config *config, const mtp_weights *weights,
                     const void *target_embed, mtp_handle **out);

/* Run a draft block: n_draft drafter steps for B independent sequences.
 * Step 1 consumes hidden[b] (the target's last hidden state) and last_token[b]; step i+1
 * consumes step i's greedy token and its post-projected hidden state, kept in fp32 without
 * rounding ("Gemma 4 Assistant 使用指南", section 二.3; "Gemma 4 drafter explained",
 * "Target Activations"). Each step: pre_projection of [hidden ; embed(token)], every block
 * (norm, Q projection, q_norm, RoPE at pos[b], attention over the shared K of the block's
 * type -- sliding blocks attend the last `window` keys, full blocks all ctx_len[b] keys --,
 * o projection, post-attention norm + residual, gated GELU-tanh MLP, post-FFN norm +
 * residual, layer_scalar), output_norm, post_projection, and the LM head (centroid head:
 * top_k centroids, gather of their token_ordering ids, sparse logits, argmax; or the
 * dense tied head + argmax).
 *   hidden      device [B][bb] model dtype
 *   last_token  device [B] int32 in [0, V)
 *   kv_sliding  host struct, required when any block is sliding (else may be NULL)
 *   kv_full     host struct, required when any block is full (else may be NULL)
 *   pos         device [B] int32: the constant position id of the block
 *   out_tokens  device [B][n_draft] int32
 *   out_hidden  device [B][n_draft][bb] fp32 post_projection output of every step, or NULL
 * Errors: INVALID_ARG (NULL hidden / token / needed KV, B outside [1, max_batch],
 * n_draft < 1, bad stride), UNSUPPORTED_SHAPE, CUDA. */
MTP_API int mtp_draft_block(mtp_handle *h, const void *hidden, const int32_t *last_token,
                    const mtp_kv *kv_sliding, const mtp_kv *kv_full, const int32_t *pos,
                    int32_t B, int32_t n_draft, int32_t *out_tokens, float *out_hidden,
                    void *stream);

/* LM head on given final-normed hidden states (testing / sampling entry point).
 * Centroid head ("Gemma 4 Assistant tensor inventory", "Centroid / ordered embeddings LM
 * head", steps 1-5): centroid logits, top_k centroids, gather of their ids, sparse logits,
 * and -- when out_logits != NULL -- the full row filled with -1e30f with the sparse logits
 * scattered at their ids (or the other mask of mtp_set_logit_mask). Dense head
 * (use_ordered_embeddings == 0): all V logits.
 *   y             device [B][H] fp32, used as given (never rounded to bf16)
 *   out_logits    device [B][V] fp32 or NULL
 *   out_token     device [B] int32 (argmax, lowest id on ties)
 *   out_centroids device [B][top_k] int32 selected centroids, best first (ties: lower
 *                 index first), or NULL; must be NULL for the dense head
 * Errors: INVALID_ARG, CUDA. */
MTP_API int mtp_centroid_head(mtp_handle *h, const float *y, int32_t B, float *out_logits,
                      int32_t *out_token, int32_t *out_centroids, void *stream);

/* Select the mask of the materialised rows of mtp_centroid_head on this handle (default
 * MTP_MASK_NEG_1E30). With MTP_MASK_MIN_MINUS_ONE, after the sparse logits are scattered,
 * every entry still holding the -1e30f fill becomes min over the sequence's candidate
 * logits minus 1 (fp32). A candidate logit equal to -1e30f exactly would be treated as
 * fill. Has no effect on the dense head or on mtp_draft_block (which materialises no row).
 * Errors: INVALID_ARG (NULL handle, unknown mode). */
MTP_API int mtp_set_logit_mask(mtp_handle *h, int32_t mode);

/* Select the sparse-head traversal (enum mtp_sparse_head) of mtp_draft_block's batched paths
 * (1 and 5; the persistent path 2 always gathers per sequence) and of mtp_centroid_head on
 * this handle; default MTP_HEAD_AUTO. Cluster-major reads the token_embd copy in
 * token_ordering order that init makes for every centroid head, and falls back to the
 * per-sequence gather where its shared-memory plan does not fit (about max_batch x hidden x 4
 * bytes of y plus a 4-stage ring of 32 KB must stay under 227 KB). It changes no output beyond
 * the fp32 summation order of a logit. No effect on the dense head or the single-sequence
 * paths. Errors: INVALID_ARG (NULL handle, unknown mode). */
MTP_API int mtp_set_sparse_head(mtp_handle *h, int32_t mode);

/* Greedy accept-prefix verification ("Gemma 4 drafter explained", "What is Speculative
 * Decoding?"): t_i = argmax of target row i (lowest id on ties); accept_len[b] = the
 * largest m with draft[b][i] == t_i for all i < m; out_tokens[b] = draft[b][0..m) followed
 * by t_m (the target's correction, or its extra token when m == n), then -1 padding.
 * Rows after the first disagreement never change the result. Rows are read in batches of up
 * to five (copied together into shared memory); batches after the one holding the first
 * disagreement are not read. accept_len[b] = -1 reports that a bounded device wait on those
 * copies gave up (not expected on a working GPU); that sequence's undecided rows stay -1.
 *   target_logits device [B][n+1][V] bf16
 *   draft         device [B][n] int32
 *   accept_len    device [B] int32
 *   out_tokens    device [B][n+1] int32
 * Errors: INVALID_ARG (NULL, B < 1, n < 0, V < 1, V % 8 != 0), CUDA. */
MTP_API int mtp_verify_greedy(const void *target_logits, const int32_t *draft, int32_t B, int32_t n,
                      int32_t V, int32_t *accept_len, int32_t *out_tokens, void *stream);

/* Sampled verification at temperature T (the pages give the accept-until-disagreement
 * structure, "Gemma 4 drafter explained", "What is Speculative Decoding?", and note that the
 * accept rate varies with temperature, "Gemma 4 Multi-Token Prediction (MTP) drafter",
 * "Status"; they give no stochastic rule). Speculative sampling with the drafter's proposal
 * a point mass on each drafted token: p_i = softmax(target row i / T); draft i is accepted
 * while u_accept[b][i] < p_i(draft[b][i]); at the first rejection the emitted token is the
 * inverse-CDF sample, over increasing ids, of p_i without the drafted token (renormalised)
 * at u_sample[b][i]; when all n drafts are accepted the extra token is the sample of p_n at
 * u_sample[b][n]. The emitted tokens are distributed as sampling from the target at T.
 * T = 0 is mtp_verify_greedy (the uniforms are not read). Decisions are taken in fp32; a
 * uniform within about 1e-6 (relative) of a decision boundary may fall either way.
 *   target_logits device [B][n+1][V] bf16
 *   draft         device [B][n] int32
 *   temperature   host float, finite, >= 0
 *   u_accept      device [B][n] fp32 uniforms in [0, 1) (may be NULL when n == 0)
 *   u_sample      device [B][n+1] fp32 uniforms in [0, 1)
 *   accept_len    device [B] int32
 *   out_tokens    device [B][n+1] int32 (-1 padded after the emitted token)
 * Rows after the first rejection are not read. Asynchronous on `stream`; caller-owned
 * buffers. Errors: INVALID_ARG (NULL, B < 1, n < 0, V < 1, V % 8 != 0, T < 0 or not
 * finite), CUDA. */
MTP_API int mtp_verify_sample(const void *target_logits, const int32_t *draft, int32_t B, int32_t n,
                              int32_t V, float temperature, const float *u_accept,
                              const float *u_sample, int32_t *accept_len, int32_t *out_tokens,
                              void *stream);

/* Size of the static device scratch of mtp_centroid_head_noalloc (1 MiB). */
#define MTP_NOALLOC_SCRATCH_BYTES (1u << 20)

/* The centroid LM head of mtp_centroid_head for callers that cannot allocate device memory:
 * code running where cudaMalloc is unavailable or forbidden, such as inside a region being
 * captured into a CUDA graph, an allocator callback, or a runtime that owns every device
 * allocation and hands out only the caller's tensors. The pages have no counterpart; this is
 * a library convenience. It needs no handle (creating one allocates a workspace): the head's
 * tensors are passed directly, and its scratch lives in a fixed device array of
 * MTP_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until the process exits.
 * Results equal mtp_centroid_head's on the same tensors. token_ordering is not validated
 * here (mtp_init_weights checks it is a permutation; this entry has no handle): a candidate
 * whose id lies outside [0, vocab) is skipped, neither read nor written.
 *   y              device [B][hidden] fp32 final-normed hidden states
 *   centroids      device [n_centroids][hidden], dtype (MTP_DTYPE_BF16 or MTP_DTYPE_F32)
 *   token_ordering device [vocab] int32, a permutation viewed [n_centroids][vocab/n_centroids]
 *   token_embd     device [vocab][hidden], dtype
 *   out_logits     device [B][vocab] fp32 (-1e30 outside the selected clusters) or NULL
 *   out_token      device [B] int32;  out_centroids device [B][top_k] int32 or NULL
 * Scratch needed: 4*B*(n_centroids + top_k + hidden) + 8*B bytes, each part rounded up to 256;
 * larger requests fail with MTP_ERR_INVALID_ARG and a message giving both sizes. The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress); make that
 * first call before any stream capture. Calls share the array and keep its last contents:
 * calls that overlap on the GPU (concurrent streams, several host threads) race. No
 * cudaMalloc, cudaFree or allocating library routine is called.
 * Errors: INVALID_ARG, BAD_ORDERING (vocab % n_centroids != 0), CUDA. */
MTP_API int mtp_centroid_head_noalloc(const float *y, const void *centroids, const int32_t *token_ordering,
                                      const void *token_embd, int32_t dtype, int32_t B, int32_t hidden,
                                      int32_t n_centroids, int32_t top_k, int32_t vocab, float *out_logits,
                                      int32_t *out_token, int32_t *out_centroids, void *stream);

/* Synchronise the device and return the handle's device-side status word: MTP_OK,
 * MTP_ERR_TIMEOUT when a bounded device wait of a previous call gave up, or
 * MTP_ERR_INVALID_ARG when a device-resident input was out of range (a last_token outside
 * [0, V): embedding row 0 was read instead). The word is cleared by this call. Also reports
 * a pending CUDA error as MTP_ERR_CUDA. */
MTP_API int mtp_get_status(mtp_handle *h);

/* Testing only: failure injection on the host side of a device wait. With
 * skip_arrival_cta >= 0, that CTA of the persistent draft-block kernel (path 2) does not
 * arrive at the first grid barrier of the next launches; every CTA's bounded wait then
 * gives up, the call's status word reads MTP_ERR_TIMEOUT (mtp_get_status), the kernel
 * returns early without a fault, and the handle stays usable. spin_limit_cycles > 0 replaces
 * the bound of the device waits of the phase and persistent paths (default about 2 s of
 * clock64 cycles). On the grid path (7), CTA skip_arrival_cta does not publish its slice of
 * the first all-reduce of the next launches; on the streamed cluster path (6), CTA
 * skip_arrival_cta of the cluster sends none of its rows in the launch's first exchange; on
 * the tensor-core path (5), CTA skip_arrival_cta of the first projection GEMM issues no copy
 * for its last k stage. Each has the same timeout outcome, and the bound applies to the
 * waits of these paths too. (-1, 0) restores the defaults. No other path is affected.
 * Errors: INVALID_ARG (NULL handle, skip_arrival_cta < -1, spin_limit_cycles < 0). */
MTP_API int mtp_set_debug(mtp_handle *h, int32_t skip_arrival_cta, int64_t spin_limit_cycles);

/* Select the implementation of mtp_draft_block: 0 = automatic, 1 = one kernel per phase,
 * 2 = persistent whole-block kernel with grid barriers, 5 = one kernel per phase with every
 * projection (and the dense tied head) as a tcgen05 tensor-core GEMM (bf16, max_batch <= 64;
 * mtp_init_weights keeps the tensor maps and a staging buffer of 3 * roundup(max_batch, 32) *
 * max input width bf16), 6 = streamed-tile cluster kernel for one sequence (one 16-CTA
 * cluster; every projection on tensor cores from weight tiles packed once into one stream
 * per CTA (see below), about the size of all projection weights; vectors exchanged
 * register-to-peer in distributed shared memory; bf16 centroid-head shapes within its
 * limits, one KV head, V = K, 16-byte aligned hidden and K rows), 7 = grid kernel for one
 * sequence (every co-resident thread-block cluster of the GPU; each projection split over
 * all CTAs by rows or by input columns, the split weights and the attended K resident in
 * shared memory -- K of long contexts is read from global memory instead --, vectors
 * exchanged by all-gathers and all-reduces over distributed shared memory and epoch-tagged
 * global mailboxes; bf16 centroid-head shapes with hidden in {64, 128, 256, 512},
 * power-of-two head dims and vocab / n_centroids, whose per-CTA share fits shared memory,
 * V = K, 16-byte aligned K rows; mtp_init_weights packs the per-CTA weight images, about the
 * size of all projection weights). Paths 3 and 4 (earlier single-sequence kernels) no longer
 * exist and are rejected. Automatic picks 7 for B = 1 when available, else 6; 5 for B >= 2
 * when available; else 2 when co-resident, else 1. Results agree within the precision
 * contract.
 * The streamed cluster path's weight streams are built (device memory about the size of the
 * projection weights, packed once; the call synchronises) when path 6 is first selected, or
 * by mtp_init_weights when the grid path cannot serve the handle and path 6 is the automatic
 * one-sequence path.
 * Errors: INVALID_ARG (NULL handle, path outside {0, 1, 2, 5, 6, 7}), CUDA (building the
 * path-6 streams); a forced path the call cannot use makes mtp_draft_block return
 * UNSUPPORTED_SHAPE. */
MTP_API int mtp_set_path(mtp_handle *h, int32_t path);

/* Free the workspace and the handle (synchronises). NULL is ignored. */
MTP_API void mtp_destroy(mtp_handle *h);

/* Text of the last error raised on the calling thread ("" when none). */
MTP_API const char *mtp_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MTP_H_ */
