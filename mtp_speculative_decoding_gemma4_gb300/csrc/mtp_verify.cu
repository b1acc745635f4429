// Greedy accept-prefix verification of a draft against the target's logits
// ("Gemma 4 drafter explained", "What is Speculative Decoding?": drafts are accepted until
// the target first disagrees; the target's own token replaces the first rejected draft, or
// is appended when every draft was accepted).
//
// One thread-block cluster per sequence scans the target rows in order. Each CTA of the
// cluster takes a contiguous slice of the row (16-byte loads, the next row prefetched into
// registers while the current one is reduced), reduces it to one (value, id) key, and
// writes that key into every CTA's shared memory (DSMEM). After a cluster barrier each CTA
// holds all slice keys, takes the row argmax (largest bf16 value, lowest id on ties) and the
// same accept/stop decision; rows after the first disagreement are never read.
#include <cooperative_groups.h>

#include "mtp_common.cuh"
#include "mtp_launch.h"

namespace cg = cooperative_groups;

namespace mtp {

constexpr int kVerifyThreads = 512;
constexpr int kVerifyMaxCluster = 16;
constexpr int kVerifyVecPerThread = 4;  // 16-byte vectors per thread per row (covers 16384 / CTA)

__global__ void __launch_bounds__(kVerifyThreads) k_verify(const __nv_bfloat16* __restrict__ logits,
                                                          const int* __restrict__ draft, int n, int V, int slice,
                                                          int* __restrict__ accept_len, int* __restrict__ out_tokens) {
  __shared__ unsigned long long keys[2][kVerifyMaxCluster];
  __shared__ unsigned long long wk[kVerifyThreads / 32];
  cg::cluster_group cl = cg::this_cluster();
  const int cs = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / cs;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lo = rank * slice, hi = min(V, lo + slice);

  if (rank == 0)
    for (int i = threadIdx.x; i <= n; i += kVerifyThreads) out_tokens[static_cast<size_t>(b) * (n + 1) + i] = -1;

  // registers of the current and the next row: up to kVerifyVecPerThread vectors each;
  // slices wider than that are walked in further passes
  const int per_pass = kVerifyThreads * 8 * kVerifyVecPerThread;
  auto row_ptr = [&](int i) { return logits + (static_cast<size_t>(b) * (n + 1) + i) * V; };
  uint4 cur[kVerifyVecPerThread], nxt[kVerifyVecPerThread];
  auto load_pass = [&](uint4* dst, const __nv_bfloat16* row, int base) {
#pragma unroll
    for (int v = 0; v < kVerifyVecPerThread; ++v) {
      const int k = base + (v * kVerifyThreads + threadIdx.x) * 8;
      dst[v] = k < hi ? __ldcs(reinterpret_cast<const uint4*>(row + k)) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  auto reduce_pass = [&](const uint4* src, int base, unsigned long long best) {
#pragma unroll
    for (int v = 0; v < kVerifyVecPerThread; ++v) {
      const int k = base + (v * kVerifyThreads + threadIdx.x) * 8;
      if (k < hi) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&src[v]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h[e]);
          const unsigned long long k0 = argmax_key(f.x, k + 2 * e), k1 = argmax_key(f.y, k + 2 * e + 1);
          best = k0 > best ? k0 : best;
          best = k1 > best ? k1 : best;
        }
      }
    }
    return best;
  };

  load_pass(cur, row_ptr(0), lo);
  for (int i = 0; i <= n; ++i) {
    const __nv_bfloat16* row = row_ptr(i);
    unsigned long long best = 0ull;
    // further passes of this row (slices wider than one pass)
    for (int base = lo + per_pass; base < hi; base += per_pass) {
      uint4 tmp[kVerifyVecPerThread];
      load_pass(tmp, row, base);
      best = reduce_pass(tmp, base, best);
    }
    if (i < n) load_pass(nxt, row_ptr(i + 1), lo);  // prefetch the next row's first pass
    best = reduce_pass(cur, lo, best);
    best = warp_max_u64(best);
    if (lane == 0) wk[warp] = best;
    __syncthreads();
    if (threadIdx.x < cs) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kVerifyThreads / 32; ++w) m = wk[w] > m ? wk[w] : m;
      unsigned long long* dst = cl.map_shared_rank(&keys[i & 1][rank], threadIdx.x);
      *dst = m;
    }
    cl.sync();
    unsigned long long m = 0ull;
    for (int r = 0; r < cs; ++r) m = keys[i & 1][r] > m ? keys[i & 1][r] : m;
    const int t = key_id(m);
    const bool accept = i < n && draft[static_cast<size_t>(b) * n + i] == t;
    if (rank == 0 && threadIdx.x == 0) {
      out_tokens[static_cast<size_t>(b) * (n + 1) + i] = t;
      if (!accept) accept_len[b] = i;
    }
    if (!accept) break;
#pragma unroll
    for (int v = 0; v < kVerifyVecPerThread; ++v) cur[v] = nxt[v];
  }
  cl.sync();  // no CTA leaves while its shared keys may still be written by another
}

int run_verify(const void* logits, const int* draft, int B, int n, int V, int* accept_len, int* out_tokens,
               cudaStream_t st) {
  // cluster size: 16 CTAs per sequence when the grid is small, else 8 (portable)
  int cs = B <= 8 ? 16 : 8;
  int slice = ((V + cs * 8 - 1) / (cs * 8)) * 8;
  if (cs == 16) {
    cudaError_t e = cudaFuncSetAttribute(k_verify, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
      cudaGetLastError();
      cs = 8;
      slice = ((V + cs * 8 - 1) / (cs * 8)) * 8;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B * cs);
  cfg.blockDim = dim3(kVerifyThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_verify, static_cast<const __nv_bfloat16*>(logits), draft, n, V, slice,
                                     accept_len, out_tokens);
  if (e != cudaSuccess) {
    set_error("k_verify launch (%d clusters of %d) failed: %s", B, cs, cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

}  // namespace mtp
