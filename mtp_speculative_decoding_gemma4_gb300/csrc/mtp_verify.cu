// Greedy accept-prefix verification of a draft against the target's logits
// ("Gemma 4 drafter explained", "What is Speculative Decoding?": drafts are accepted until
// the target first disagrees; the target's own token replaces the first rejected draft, or
// is appended when every draft was accepted).
//
// One CTA per sequence scans the target rows in order: row argmax (largest bf16 value,
// lowest id on ties) with 16-byte loads and a warp-shuffle max of (value, id) keys, then
// the comparison with the draft; rows after the first disagreement are never read.
#include "mtp_common.cuh"
#include "mtp_launch.h"

namespace mtp {

constexpr int kVerifyThreads = 1024;

__global__ void __launch_bounds__(kVerifyThreads) k_verify(const __nv_bfloat16* __restrict__ logits,
                                                          const int* __restrict__ draft, int n, int V,
                                                          int* __restrict__ accept_len, int* __restrict__ out_tokens) {
  __shared__ unsigned long long wk[kVerifyThreads / 32];
  __shared__ int go;
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i <= n; i += kVerifyThreads) out_tokens[static_cast<size_t>(b) * (n + 1) + i] = -1;
  __syncthreads();
  for (int i = 0; i <= n; ++i) {
    const __nv_bfloat16* row = logits + (static_cast<size_t>(b) * (n + 1) + i) * V;
    unsigned long long best = 0ull;
    for (int k = threadIdx.x * 8; k < V; k += kVerifyThreads * 8) {
      float v[8];
      load_vec_stream(row + k, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const unsigned long long key = argmax_key(v[e], k + e);
        best = key > best ? key : best;
      }
    }
    best = warp_max_u64(best);
    if (lane == 0) wk[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kVerifyThreads / 32; ++w) m = wk[w] > m ? wk[w] : m;
      const int t = key_id(m);
      out_tokens[static_cast<size_t>(b) * (n + 1) + i] = t;
      const bool accept = i < n && draft[static_cast<size_t>(b) * n + i] == t;
      if (!accept) accept_len[b] = i;
      go = accept ? 1 : 0;
    }
    __syncthreads();
    if (!go) break;
  }
}

int run_verify(const void* logits, const int* draft, int B, int n, int V, int* accept_len, int* out_tokens,
               cudaStream_t st) {
  k_verify<<<B, kVerifyThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(logits), draft, n, V, accept_len,
                                         out_tokens);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("k_verify launch failed: %s", cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

}  // namespace mtp
