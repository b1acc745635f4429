// Tensor-core (tcgen05) GEMM for the batched projections: for a weight matrix W [R][K]
// (bf16, row-major) and B <= 64 activation vectors given as their three bf16 terms
// Xs [3][B][K] (x = hi + mid + lo, so every product with a bf16 weight is exact and the sums
// are fp32), computes Y[b][r] = sum_k W[r][k] x_b[k] for all rows r.
//
// One CTA per 128-row tile of W (M = 128); N = 3B columns (the three terms of every
// sequence), accumulated in tensor memory over K in steps of 64:
//   * a producer thread (warp 4) streams W[tile][k..k+64) and Xs[*][k..k+64) into a ring of shared-
//     memory stages with TMA (128-byte swizzle, the layout the MMA descriptors describe);
//   * one thread (warp 5) issues tcgen05.mma (kind::f16, K = 16 per instruction) per stage and
//     releases the stage with tcgen05.commit when its MMAs are done;
//   * the tensor-memory accumulator adds the partial sums of its MMAs with truncation, so a
//     long chain of MMAs into one accumulator loses precision: every kGroup stages (256 of K)
//     the accumulation moves to the other of two tensor-memory regions, and warps 0..3 read
//     the finished group back (tcgen05.ld, warp w owns rows 32w..32w+31), add its three
//     term columns per sequence and sum the groups in fp32 registers (round to nearest);
//   * at the end the warps either store Y or, for the dense tied head, keep the largest
//     (logit, row) key of every sequence (atomicMax). Two projections of the same input
//     (gate and up; post_projection and the centroids) run as one launch over their stacked
//     rows, each tile storing into the output of the matrix its rows belong to; gate and up
//     interleave their rows so that one tile holds both halves of 64 MLP rows and its
//     epilogue writes gelu_tanh(gate) * up straight into the down projection's operand.
// Split K: with splits S > 1 (projections only) the S CTAs of a row tile form a thread-block
// cluster and take consecutive S-th parts of K; each writes its fp32 partial sums into its
// own (then idle) stage memory, and after a cluster barrier CTA s adds the S partials of rows
// [s 128 / S, (s + 1) 128 / S) in a fixed order through distributed shared memory, so the
// result does not depend on timing.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mtp {
namespace tc {

constexpr int kM = 128;          // rows per tile (tcgen05 M)
constexpr int kKStage = 64;      // k per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kGroup = 4;        // k stages accumulated in tensor memory before an fp32 readback
constexpr int kMaxB = 64;        // sequences per GEMM (N = 3B <= 192)
constexpr int kEpiWarps = 4;     // warps 0..3: read-back and epilogue (one tensor-memory lane quarter each)
constexpr int kThreads = 192;    // + warp 4: TMA producer, warp 5: MMA issue

struct Args {
  int R, K, B;                   // rows, inner size, sequences of the B operand (multiple of 32)
  int nvalid;                    // sequences whose outputs are written (<= B)
  float* out;                    // Y[b * ldo + r] (may be null)
  long long ldo;
  float* out2;                   // second copy Y[b * ld2 + r] (may be null)
  long long ld2;
  unsigned long long* best;      // dense head: atomicMax of argmax keys per sequence (or null)
  int splits;                    // K split over this many CTAs of one cluster (1: no split)
  int* status;
  long long spin_limit;
  int dbg_cta;  // testing: this CTA's producer issues no copy for its last k stage (-1: none)
  // two stacked matrices in one launch: rows r >= R1 (R1 > 0, a multiple of kM) are stored as
  // Y[b * ld_hi + (r - R1)] into out_hi instead of out / out2 (0: one matrix)
  int R1;
  float* out_hi;
  long long ld_hi;
  // gated-GELU epilogue (null: off): W is [gate ; up] interleaved in 64-row blocks (rows
  // 128t..128t+63 are gate rows 64t..64t+63, the next 64 the same up rows) and, instead of Y,
  // m = gelu_tanh(gate) * up of every row f < glu_K and sequence b < nvalid is stored as its
  // three bf16 terms into glu_xs [3][glu_bp][glu_K], the down projection's staged operand
  __nv_bfloat16* glu_xs;
  int glu_bp, glu_K;
};

__host__ __device__ inline int stage_bytes(int B) { return kM * kKStage * 2 + 3 * B * kKStage * 2; }
__host__ __device__ inline int smem_bytes(int B) { return 1024 + kStages * stage_bytes(B) + 256; }
// two accumulator regions of 3B columns each (alternating k groups)
__host__ __device__ inline int tmem_cols(int B) {
  int n = 32;
  while (n < 6 * B) n <<= 1;
  return n;
}

}  // namespace tc

// Host side (mtp_tc.cu): tensor maps and launches.
// A 2D bf16 tensor map over rows x cols (row pitch `pitch` elements) with a box of
// box_rows x 64 columns and 128-byte swizzle. Returns MTP_OK or an error code.
int tc_make_map(CUtensorMap* map, const void* base, long long rows, long long cols, long long pitch, int box_rows);
// Y = W Xs^T as described above. `dense` selects the argmax epilogue. a.splits <= 0 picks the
// split of K automatically (projections); the dense head never splits.
int tc_gemm(const CUtensorMap* mapW, const CUtensorMap* mapX, const tc::Args& a, bool dense, cudaStream_t st,
            bool pdl = false);
// Whether tcgen05 GEMMs can run on the current device (sm_100 family, driver entry point).
bool tc_available();

}  // namespace mtp
