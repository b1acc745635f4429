// Greedy accept-prefix verification of a draft against the target's logits
// ("Gemma 4 drafter explained", "What is Speculative Decoding?": drafts are accepted until
// the target first disagrees; the target's own token replaces the first rejected draft, or
// is appended when every draft was accepted).
//
// One thread-block cluster per sequence scans the target rows in batches of up to
// kVerifyRowBatch rows. Each CTA of the cluster takes a contiguous slice of every row
// (16-byte streaming loads, all rows of the batch in flight at once so that one memory round
// trip serves the batch), reduces each row's slice to one (value, id) key, and writes the keys
// into every CTA's shared memory (DSMEM). After one cluster barrier per batch each CTA holds
// all slice keys, takes each row's argmax (largest bf16 value, lowest id on ties) and walks the
// batch's accept/stop decisions in order. Rows after the first disagreement never change the
// result; the batches after the one holding it are never read.
#include <cooperative_groups.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "mtp_common.cuh"
#include "mtp_launch.h"

namespace cg = cooperative_groups;

namespace mtp {

constexpr int kVerifyThreads = 512;
constexpr int kVerifyMaxCluster = 16;
constexpr int kVerifyVecPerThread = 4;  // 16-byte vectors per thread per row and pass (16384 / CTA)
constexpr int kVerifyRowBatch = 5;      // rows whose first pass is in flight together

__global__ void __launch_bounds__(kVerifyThreads, 1) k_verify(const __nv_bfloat16* __restrict__ logits,
                                                             const int* __restrict__ draft, int n, int V, int slice,
                                                             int* __restrict__ accept_len, int* __restrict__ out_tokens) {
  __shared__ unsigned long long keys[2][kVerifyRowBatch][kVerifyMaxCluster];
  __shared__ unsigned long long wk[kVerifyRowBatch][kVerifyThreads / 32];
  __shared__ int dtok[2][kVerifyRowBatch];
  cg::cluster_group cl = cg::this_cluster();
  const int cs = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / cs;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lo = rank * slice, hi = min(V, lo + slice);

  if (rank == 0)
    for (int i = threadIdx.x; i <= n; i += kVerifyThreads) out_tokens[static_cast<size_t>(b) * (n + 1) + i] = -1;

  // the first pass of every row of a batch sits in registers; slices wider than one pass are
  // walked in further passes, one row at a time
  const int per_pass = kVerifyThreads * 8 * kVerifyVecPerThread;
  auto row_ptr = [&](int i) { return logits + (static_cast<size_t>(b) * (n + 1) + i) * V; };
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

  int buf = 0;
#pragma unroll 1
  for (int i0 = 0; i0 <= n; i0 += kVerifyRowBatch, buf ^= 1) {
    const int R = min(kVerifyRowBatch, n + 1 - i0);
    // the batch's drafted tokens, read once ahead of the decisions (made after a barrier below)
    if (threadIdx.x < R && i0 + static_cast<int>(threadIdx.x) < n)
      dtok[buf][threadIdx.x] = draft[static_cast<size_t>(b) * n + i0 + threadIdx.x];
    uint4 cur[kVerifyRowBatch][kVerifyVecPerThread];
#pragma unroll
    for (int r = 0; r < kVerifyRowBatch; ++r)
      if (r < R) load_pass(cur[r], row_ptr(i0 + r), lo);
    unsigned long long best[kVerifyRowBatch];
#pragma unroll
    for (int r = 0; r < kVerifyRowBatch; ++r) {
      best[r] = 0ull;
      if (r < R) {
        best[r] = reduce_pass(cur[r], lo, 0ull);
        // further passes of this row (slices wider than one pass)
#pragma unroll 1
        for (int base = lo + per_pass; base < hi; base += per_pass) {
          uint4 tmp[kVerifyVecPerThread];
          load_pass(tmp, row_ptr(i0 + r), base);
          best[r] = reduce_pass(tmp, base, best[r]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kVerifyRowBatch; ++r) {
      const unsigned long long m = warp_max_u64(best[r]);
      if (lane == 0) wk[r][warp] = m;
    }
    __syncthreads();
    // thread (row r, peer q) sends this CTA's key of row r to peer q
    if (threadIdx.x < R * cs) {
      const int r = threadIdx.x / cs, q = threadIdx.x - r * cs;
      unsigned long long m = 0ull;
      for (int w = 0; w < kVerifyThreads / 32; ++w) m = wk[r][w] > m ? wk[r][w] : m;
      *cl.map_shared_rank(&keys[buf][r][rank], q) = m;
    }
    cl.sync();
    bool go = true;
    for (int r = 0; r < R && go; ++r) {
      unsigned long long m = 0ull;
      for (int q = 0; q < cs; ++q) m = keys[buf][r][q] > m ? keys[buf][r][q] : m;
      const int i = i0 + r, t = key_id(m);
      const bool accept = i < n && dtok[buf][r] == t;
      if (rank == 0 && threadIdx.x == 0) {
        out_tokens[static_cast<size_t>(b) * (n + 1) + i] = t;
        if (!accept) accept_len[b] = i;
      }
      go = accept;
    }
    if (!go) break;
  }
  cl.sync();  // no CTA leaves while its shared keys may still be written by another
}

// The same with the rows' slices copied into shared memory by the bulk-copy engine (one copy
// per row and CTA, a transaction barrier per row slot): the copies of a batch are in flight
// together without holding registers. Each CTA takes its slice's largest value with packed
// bf16 maxima, then the first position holding it (packed compares), and the cluster keeps
// the largest value (fp32 comparison, so -0 equals +0), lowest position. Every wait on a copy is bounded; a CTA whose wait gives up marks the
// sequence (every CTA of the cluster learns it with the keys), which then gets
// accept_len = -1 and no further rows. Used when at least one row slice fits the
// shared-memory budget (rb rows per batch).
constexpr int kVerifySmemMax = 200 * 1024;
constexpr long long kVerifySpin = 1LL << 32;  // about 2 s of clock64 cycles

__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ bool vbar_try(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000u)
      : "memory");
  return ok != 0;
}
// false when the phase did not complete within the bound
__device__ __forceinline__ bool vbar_wait(unsigned bar, unsigned parity) {
  if (vbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (!vbar_try(bar, parity))
    if (clock64() - t0 > kVerifySpin) return false;
  return true;
}

__global__ void __launch_bounds__(kVerifyThreads, 1) k_verify_bulk(const __nv_bfloat16* __restrict__ logits,
                                                                  const int* __restrict__ draft, int n, int V,
                                                                  int slice, int rb, int* __restrict__ accept_len,
                                                                  int* __restrict__ out_tokens) {
  extern __shared__ __align__(128) unsigned char vsm[];
  __shared__ unsigned long long keys[2][kVerifyRowBatch][kVerifyMaxCluster];  // (max bits, first position)
  __shared__ float wmax[kVerifyRowBatch][kVerifyThreads / 32];
  __shared__ int wfirst[kVerifyRowBatch][kVerifyThreads / 32];
  __shared__ int dtok[2][kVerifyRowBatch];
  __shared__ int bads[2][kVerifyMaxCluster];
  __shared__ float cmx[kVerifyRowBatch];
  __shared__ int go_s;
  __shared__ __align__(8) unsigned long long bar[kVerifyRowBatch];
  cg::cluster_group cl = cg::this_cluster();
  const int cs = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / cs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lo = rank * slice, hi = min(V, lo + slice), cnt = hi > lo ? hi - lo : 0;
  const unsigned bytes = static_cast<unsigned>(cnt) * 2u;
  const unsigned sbase = static_cast<unsigned>(__cvta_generic_to_shared(vsm));
  auto bar_a = [&](int r) { return static_cast<unsigned>(__cvta_generic_to_shared(&bar[r])); };
  auto row_ptr = [&](int i) { return logits + (static_cast<size_t>(b) * (n + 1) + i) * V; };

  if (tid == 0) {
    for (int r = 0; r < rb; ++r)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_a(r)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (rank == 0)
    for (int i = tid; i <= n; i += kVerifyThreads) out_tokens[static_cast<size_t>(b) * (n + 1) + i] = -1;
  __syncthreads();

  int buf = 0, pend = 0;  // pend: slots of a batch left by a failed wait (drained before the end)
  unsigned ph = 0u;
#pragma unroll 1
  for (int i0 = 0; i0 <= n; i0 += rb, buf ^= 1, ph ^= 1u) {
    const int R = min(rb, n + 1 - i0);
    if (tid < R && i0 + tid < n) dtok[buf][tid] = draft[static_cast<size_t>(b) * n + i0 + tid];
    if (tid == 0) {
      // the slots' previous contents were read before the last cluster barrier
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      for (int r = 0; r < R; ++r) {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_a(r)), "r"(bytes) : "memory");
        if (bytes)
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                  sbase + static_cast<unsigned>(r * slice * 2)),
              "l"(row_ptr(i0 + r) + lo), "r"(bytes), "r"(bar_a(r))
              : "memory");
      }
    }
    pend = R;
    int bad = 0;
    // pass 1: the largest value of each row slice (bf16 pairs, packed max)
    float cmax[kVerifyRowBatch];
#pragma unroll
    for (int r = 0; r < kVerifyRowBatch; ++r) {
      float m = -INFINITY;
      if (r < R) {
        if (!vbar_wait(bar_a(r), ph)) bad = 1;
        const uint4* row = reinterpret_cast<const uint4*>(vsm + r * slice * 2);
        __nv_bfloat162 m2 = __float2bfloat162_rn(-INFINITY);
#pragma unroll 4
        for (int v = tid; v < cnt / 8; v += kVerifyThreads) {
          const uint4 u = row[v];
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
          m2 = __hmax2(__hmax2(m2, h[0]), __hmax2(h[1], __hmax2(h[2], h[3])));
        }
        const float2 f = __bfloat1622float2(m2);
        m = warp_max(fmaxf(f.x, f.y));
      }
      if (lane == 0) wmax[r][warp] = m;
    }
    const int cta_bad = __syncthreads_or(bad);
    if (tid < R) {  // one thread per row: the CTA's maximum
      float m = -INFINITY;
      for (int w = 0; w < kVerifyThreads / 32; ++w) m = fmaxf(m, wmax[tid][w]);
      cmx[tid] = m;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kVerifyRowBatch; ++r) cmax[r] = r < R ? cmx[r] : -INFINITY;
    // pass 2: the first position of that value in the slice (equal values: lowest id)
#pragma unroll
    for (int r = 0; r < kVerifyRowBatch; ++r) {
      int first = INT_MAX;
      if (r < R) {
        const uint4* row = reinterpret_cast<const uint4*>(vsm + r * slice * 2);
        const __nv_bfloat162 t2 = __float2bfloat162_rn(cmax[r]);
#pragma unroll 4
        for (int v = tid; v < cnt / 8 && first == INT_MAX; v += kVerifyThreads) {
          const uint4 u = row[v];
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
          for (int e = 3; e >= 0; --e) {  // last to first: the lowest match is kept
            const __nv_bfloat162 q = __heq2(h[e], t2);
            const unsigned qb = *reinterpret_cast<const unsigned*>(&q);
            if (qb) first = lo + 8 * v + 2 * e + ((qb & 0xffffu) ? 0 : 1);
          }
        }
        first = warp_min_i(first);
      }
      if (lane == 0) wfirst[r][warp] = first;
    }
    __syncthreads();
    // thread (row r, peer q) sends this CTA's (max, first position) of row r to peer q; thread
    // R * cs + q its flag
    if (tid < R * cs) {
      const int r = tid / cs, q = tid - r * cs;
      int first = INT_MAX;
      float cm = -INFINITY;
      for (int w = 0; w < kVerifyThreads / 32; ++w) {
        first = min(first, wfirst[r][w]);
        cm = fmaxf(cm, wmax[r][w]);
      }
      const unsigned long long kv =
          (static_cast<unsigned long long>(__float_as_uint(cm)) << 32) | static_cast<unsigned>(first);
      *cl.map_shared_rank(&keys[buf][r][rank], q) = kv;
    } else if (tid < R * cs + cs) {
      *cl.map_shared_rank(&bads[buf][rank], tid - R * cs) = cta_bad;
    }
    cl.sync();
    // the decisions, taken by warp 0 of every CTA (all take the same), shared with the CTA
    if (warp == 0) {
      const bool any_bad = __any_sync(0xffffffffu, lane < cs && bads[buf][lane] != 0);
      int go = any_bad ? -1 : 1;
      for (int r = 0; r < R && go == 1; ++r) {
        // the largest value over the slices (compared as fp32: -0 equals +0), lowest position
        float bv = -INFINITY;
        int bi = INT_MAX;
        if (lane < cs) {
          const unsigned long long kv = keys[buf][r][lane];
          bv = __uint_as_float(static_cast<unsigned>(kv >> 32));
          bi = static_cast<int>(static_cast<unsigned>(kv));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
          const int f2 = __shfl_xor_sync(0xffffffffu, bi, o);
          if (f2 != INT_MAX && (bi == INT_MAX || v2 > bv || (v2 == bv && f2 < bi))) {
            bv = v2;
            bi = f2;
          }
        }
        const int i = i0 + r, t = bi == INT_MAX ? 0 : bi;
        const bool accept = i < n && dtok[buf][r] == t;
        if (rank == 0 && lane == 0) {
          out_tokens[static_cast<size_t>(b) * (n + 1) + i] = t;
          if (!accept) accept_len[b] = i;
        }
        go = accept ? 1 : 0;
      }
      if (any_bad && rank == 0 && lane == 0) accept_len[b] = -1;
      if (lane == 0) go_s = go;
    }
    __syncthreads();
    const int go = go_s;
    if (go < 0) break;  // a wait gave up: leave with the batch's copies drained below
    pend = 0;
    if (go == 0) break;
  }
  // a batch left by a failed wait may still have copies in flight: drain them (bounded; the
  // loop ended by break, so ph is still that batch's parity)
  if (pend && tid == 0)
    for (int r = 0; r < pend; ++r) vbar_wait(bar_a(r), ph);
  cl.sync();  // no CTA leaves while its shared keys may still be written by another
}

namespace {
int cuda_fail_v(const char* what, cudaError_t e) {
  cudaGetLastError();
  set_error("%s: %s", what, cudaGetErrorString(e));
  return MTP_ERR_CUDA;
}
}  // namespace

int run_verify(const void* logits, const int* draft, int B, int n, int V, int* accept_len, int* out_tokens,
               cudaStream_t st) {
  // function attributes, set once per device: 16-CTA clusters (when the device takes them)
  // and the bulk-copy form's shared-memory budget
  static std::mutex mu;
  static int attrs_of[64] = {0};  // per device: 0 not set yet; 2: 16-CTA clusters available; 1: not
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    dev = 0;
  }
  int attrs;
  {
    std::lock_guard<std::mutex> lock(mu);
    attrs = attrs_of[dev] - 1;
    if (attrs < 0) {
      cudaError_t e = cudaFuncSetAttribute(k_verify, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e == cudaSuccess) e = cudaFuncSetAttribute(k_verify_bulk, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      attrs = e == cudaSuccess ? 1 : 0;
      cudaGetLastError();
      e = cudaFuncSetAttribute(k_verify_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize, kVerifySmemMax);
      if (e != cudaSuccess) return cuda_fail_v("k_verify_bulk shared memory attribute", e);
      attrs_of[dev] = attrs + 1;
    }
  }
  // cluster size: 16 CTAs per sequence when the grid is small, else 8 (portable)
  const int cs = B <= 8 && attrs == 1 ? 16 : 8;
  const int slice = ((V + cs * 8 - 1) / (cs * 8)) * 8;
  // rows of one CTA slice per batch in the shared-memory budget: the bulk-copy form when at
  // least one fits
  const int rb = std::min(kVerifyRowBatch, kVerifySmemMax / (slice * 2));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B * cs);
  cfg.blockDim = dim3(kVerifyThreads);
  cfg.dynamicSmemBytes = rb >= 1 ? static_cast<size_t>(rb) * slice * 2 : 0;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = rb >= 1 ? cudaLaunchKernelEx(&cfg, k_verify_bulk, static_cast<const __nv_bfloat16*>(logits), draft, n,
                                               V, slice, rb, accept_len, out_tokens)
                          : cudaLaunchKernelEx(&cfg, k_verify, static_cast<const __nv_bfloat16*>(logits), draft, n, V,
                                               slice, accept_len, out_tokens);
  if (e != cudaSuccess) {
    set_error("k_verify launch (%d clusters of %d) failed: %s", B, cs, cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

// ---------------------------------------------------------------------------------------
// Sampled verification at a temperature T > 0 (speculative sampling with the greedy
// drafter's proposal a point mass on the drafted token; the pages give the accept-prefix
// structure and say that accept rates vary with temperature): p_i = softmax(logits_i / T);
// draft d_i is accepted when u_accept < p_i(d_i); at the first rejection the emitted token is
// the inverse-CDF sample (increasing ids) of p_i with d_i removed and renormalised, with
// u_sample; when all drafts are accepted the bonus token is the sample of p_n.
//
// One thread-block cluster per sequence reads the rows in order until the first rejection.
// CTA c of the cluster owns the contiguous ids [c S, (c + 1) S) of a row and thread t of it
// the contiguous sub-range [t C, (t + 1) C): each thread keeps a running max and exp-sum
// over its ids in one pass (16-byte loads), the CTA scans the sums rescaled to its max, and
// the CTAs exchange (max, sum) through distributed shared memory. Every CTA then forms the
// row max, the normaliser and the CTAs' cumulative masses in the same order, so all take the
// same accept decision; the CTA, and in it the thread, whose part of the cumulative mass
// holds the sample point rescans its ids to find the sampled id.
constexpr int kVsThreads = 512;
constexpr int kVsWarps = kVsThreads / 32;
constexpr int kVsMaxCluster = 16;

// Exclusive prefix over the CTA's threads in order; returns it, and the total in *total.
__device__ __forceinline__ float block_scan_vs(float v, float* sh, float* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  __syncthreads();
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  float before = 0.f, all = 0.f;
  for (int w = 0; w < kVsWarps; ++w) {
    if (w < warp) before += sh[w];
    all += sh[w];
  }
  *total = all;
  return before + inc - v;
}

__global__ void __launch_bounds__(kVsThreads) k_verify_sample(const __nv_bfloat16* __restrict__ logits,
                                                              const int* __restrict__ draft, int n, int V, int slice,
                                                              int chunk, float k2, const float* __restrict__ u_accept,
                                                              const float* __restrict__ u_sample,
                                                              int* __restrict__ accept_len, int* __restrict__ out_tokens) {
  __shared__ float sh[kVsWarps];
  __shared__ float pres[kVsThreads];
  __shared__ float2 ex[2][kVsMaxCluster];  // (max, exp-sum) of every CTA, double-buffered by row
  __shared__ int pick;
  cg::cluster_group cl = cg::this_cluster();
  const int cs = static_cast<int>(cl.num_blocks()), rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / cs, tid = threadIdx.x;
  const int clo = min(V, rank * slice), chi = min(V, clo + slice);
  const int lo = min(chi, clo + tid * chunk), hi = min(chi, lo + chunk);
  if (rank == 0)
    for (int i = tid; i <= n; i += kVsThreads) out_tokens[static_cast<size_t>(b) * (n + 1) + i] = -1;
  // weights exp((x - m) / T) as exp2((x - m) * log2(e) / T) = exp2((x - m) * k2)
  for (int i = 0; i <= n; ++i) {
    const __nv_bfloat16* row = logits + (static_cast<size_t>(b) * (n + 1) + i) * V;
    float m = -INFINITY, s = 0.f;
    for (int v = lo; v < hi; v += 8) {
      const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(row + v));
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
      float x[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
      }
      float lm = x[0];
#pragma unroll
      for (int e = 1; e < 8; ++e) lm = fmaxf(lm, x[e]);
      if (lm > m) {
        s = m == -INFINITY ? 0.f : s * exp2f((m - lm) * k2);
        m = lm;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) s += exp2f((x[e] - m) * k2);
    }
    // this CTA: max, and the thread sums rescaled to it, scanned in id order
    float wm = warp_max(m);
    __syncthreads();
    if ((tid & 31) == 0) sh[tid >> 5] = wm;
    __syncthreads();
    float Mc = sh[0];
    for (int w = 1; w < kVsWarps; ++w) Mc = fmaxf(Mc, sh[w]);
    const float sr = s > 0.f ? s * exp2f((m - Mc) * k2) : 0.f;
    float Sc;
    const float pre = block_scan_vs(sr, sh, &Sc);
    // every CTA's (max, sum) to every CTA
    if (tid < cs) *cl.map_shared_rank(&ex[i & 1][rank], tid) = make_float2(Mc, Sc);
    cl.sync();
    float M = -INFINITY;
    for (int c = 0; c < cs; ++c) M = fmaxf(M, ex[i & 1][c].x);
    float Z = 0.f, Pc = 0.f;  // normaliser and this CTA's cumulative mass, in CTA order
    for (int c = 0; c < cs; ++c) {
      const float2 e = ex[i & 1][c];
      const float w = e.y > 0.f ? e.y * exp2f((e.x - M) * k2) : 0.f;
      if (c < rank) Pc += w;
      Z += w;
    }
    const float fc = Sc > 0.f ? exp2f((Mc - M) * k2) : 0.f;
    // the accept test of draft d, and the residual mass without it
    int d = -1;
    float wd = 0.f;
    if (i < n) {
      d = min(max(draft[static_cast<size_t>(b) * n + i], 0), V - 1);
      wd = exp2f((__bfloat162float(row[d]) - M) * k2);
      if (u_accept[static_cast<size_t>(b) * n + i] < wd / Z) {
        if (rank == 0 && tid == 0) out_tokens[static_cast<size_t>(b) * (n + 1) + i] = d;
        continue;  // every CTA and thread takes the same decision
      }
    }
    // sample point of the residual (rejection) or of p_n (bonus); CTA c owns
    // [P'_c, P'_c+1) of the cumulative mass without d, the last CTA with ids everything above
    const float target = u_sample[static_cast<size_t>(b) * (n + 1) + i] * (Z - wd);
    const int cl_last = (V - 1) / slice;
    float Pn = INFINITY;  // the next CTA's start
    if (rank < cl_last) {
      Pn = 0.f;
      for (int c = 0; c <= rank; ++c) {
        const float2 e = ex[i & 1][c];
        Pn += e.y > 0.f ? e.y * exp2f((e.x - M) * k2) : 0.f;
      }
      if (d >= 0 && d < chi) Pn -= wd;
    }
    const float Pce = Pc - (d >= 0 && d < clo ? wd : 0.f);
    const bool cta_owns = rank <= cl_last && Pce <= target && target < Pn;
    if (cta_owns) {
      const float pe = Pce + pre * fc - (d >= clo && d < lo ? wd : 0.f);
      pres[tid] = pe;
      if (tid == 0) pick = -1;
      __syncthreads();
      const int tl = (chi - clo - 1) / chunk;  // the CTA's last thread with ids
      const float upper = tid < tl ? pres[tid + 1] : Pn;
      if (tid <= tl && pe <= target && target < upper) {
        float acc = pe;
        int t = -1, last = -1;
        for (int v = lo; v < hi && t < 0; ++v) {
          const float w = v == d ? 0.f : exp2f((__bfloat162float(row[v]) - M) * k2);
          if (w > 0.f) last = v;
          if (w > 0.f && acc + w > target) t = v;
          acc += w;
        }
        pick = t >= 0 ? t : last;  // rounding left the point past the rescanned sum: the last id with mass
      }
      __syncthreads();
      if (tid == 0) {
        int tok = pick;
        if (tok < 0)  // no id of the owner carries mass (underflow): the first id of the slice at its max
          for (int v = clo; v < chi; ++v)
            if (v != d && __bfloat162float(row[v]) == Mc) {
              tok = v;
              break;
            }
        out_tokens[static_cast<size_t>(b) * (n + 1) + i] = tok < 0 ? clo : tok;
        accept_len[b] = i;
      }
    }
    break;
  }
  cl.sync();  // no CTA leaves while a peer may still write its exchange slots
}

int run_verify_sample(const void* logits, const int* draft, int B, int n, int V, float temperature,
                      const float* u_accept, const float* u_sample, int* accept_len, int* out_tokens, cudaStream_t st) {
  int cs = B <= 8 ? 16 : 8;
  if (cs == 16 && cudaFuncSetAttribute(k_verify_sample, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    cs = 8;
  }
  const int slice = ((V + cs * 8 - 1) / (cs * 8)) * 8;
  const int chunk = ((slice + kVsThreads - 1) / kVsThreads + 7) / 8 * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B * cs);
  cfg.blockDim = dim3(kVsThreads);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const float k2 = 1.4426950408889634f / temperature;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_verify_sample, static_cast<const __nv_bfloat16*>(logits), draft, n, V,
                                           slice, chunk, k2, u_accept, u_sample, accept_len, out_tokens);
  if (e != cudaSuccess) {
    set_error("k_verify_sample launch (%d clusters of %d) failed: %s", B, cs, cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

}  // namespace mtp
