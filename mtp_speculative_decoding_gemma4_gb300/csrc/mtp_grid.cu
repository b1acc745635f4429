// Grid draft block for one sequence (B = 1): see mtp_grid.cuh for the data flow.
//
// Failure handling: every wait (bulk copies, distributed-shared-memory receives, mailbox
// polls) is bounded by a clock64 budget. A wait that gives up records MTP_ERR_TIMEOUT in
// the status word and raises the abort word; a raised abort word makes every other wait of
// the launch give up at its next check. The CTA then leaves its step loop, waits (bounded)
// for its own launch-start bulk copies still in flight, and meets its cluster at the final
// barrier so that no peer writes into an exited CTA. Values taken from exchanged data that
// address memory (the token, the selected centroids) are range-checked first.
#include <cmath>
#include <cstring>

#include "mtp_grid.cuh"
#include "mtp_launch.h"

namespace mtp {
namespace gr {

// ------------------------------------------------------------------ primitives

__device__ __forceinline__ unsigned sa(const void* p) { return static_cast<unsigned>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ unsigned mapa(unsigned addr, int rank) {
  unsigned r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_async_u64(unsigned caddr, unsigned long long v, unsigned cbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(caddr), "l"(v),
               "r"(cbar)
               : "memory");
}
__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, "
      "p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(unsigned dst, const void* src, unsigned bytes, unsigned bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// A read-only global load kept in program order with the other volatile asm: issued before a
// wait, consumed after it (the compiler would otherwise sink the load to its first use).
__device__ __forceinline__ float ldg_early(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ int ldg_early_i32(const int* p) {
  int v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ double ldg_early_f64(const double* p) {
  double v;
  asm volatile("ld.global.nc.f64 %0, [%1];" : "=d"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ unsigned short ldg_early_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.b16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_rlx64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_rlx64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_rlx32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ int cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return static_cast<int>(r);
}
__device__ __forceinline__ float bf(bf16 v) { return __bfloat162float(v); }

// ------------------------------------------------------------------ bounded waits

// The abort word holds the epoch base of the launch that gave up: a word left by an earlier
// launch never matches, so no launch has to clear it first.
__device__ __forceinline__ void fail(const Params& p) {
  atomicCAS(p.status, 0, static_cast<int>(MTP_ERR_TIMEOUT));
  atomicExch(p.abort_flag, p.epoch_base);
}
__device__ __forceinline__ bool aborted(const Params& p) { return ld_rlx32(p.abort_flag) == p.epoch_base; }
// True when the caller must give up: the budget ran out (recorded) or another CTA gave up.
__device__ __forceinline__ bool expired(const Params& p, long long t0, unsigned n) {
  if ((n & 63u) != 0u) return false;
  if (aborted(p)) return true;
  if (clock64() - t0 > p.spin_limit) {
    fail(p);
    return true;
  }
  return false;
}
// A waiting thread is suspended until the phase completes or about this many ns pass.
constexpr unsigned kSuspendNs = 2000;
__device__ __forceinline__ bool mbar_try_susp(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, "
      "0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}
// Warp 0 waits on the mbarrier phase (acquire at cluster scope: the bytes peers stored with
// st.async or bulk copies wrote are visible to it); the CTA barrier then orders them before
// every other thread's reads. The other warps sleep in the barrier instead of polling the
// shared memory the incoming bytes need. Every thread calls; block-uniform result.
__device__ __forceinline__ bool mbar_wait(const Params& p, unsigned bar, unsigned parity, bool watch_abort) {
  int bad = 0;
  if (threadIdx.x < 32 && !mbar_try_susp(bar, parity)) {
    const long long t0 = clock64();
    while (!mbar_try_susp(bar, parity)) {
      if (watch_abort && aborted(p)) {
        bad = 1;
        break;
      }
      if (clock64() - t0 > p.spin_limit) {
        fail(p);
        bad = 1;
        break;
      }
    }
  }
  return !__syncthreads_or(bad);
}

__device__ __forceinline__ void put(unsigned long long* mb, long long i, float v, unsigned ep) {
  st_rlx64(mb + i, (static_cast<unsigned long long>(ep) << 32) | __float_as_uint(v));
}
__device__ __forceinline__ void put_u(unsigned long long* mb, long long i, unsigned v, unsigned ep) {
  st_rlx64(mb + i, (static_cast<unsigned long long>(ep) << 32) | v);
}

// Mailbox words -> dst[k] (payload bits), k in [0, count). Per pass a thread takes up to 16
// of its words: it issues the loads of all of them, then in rounds re-issues the loads of every
// word still missing before checking any, so a round costs one L2 round trip however many of
// its words are late. The word index of k comes from a functor; every thread calls; the result
// is block-uniform.
constexpr int kGatherBatch = 16;
template <class Idx>
__device__ __forceinline__ bool gather_t(const Params& p, const unsigned long long* mb, int count, Idx idx,
                                         unsigned* dst, unsigned ep) {
  int bad = 0;
#pragma unroll 1
  for (int base = 0; base < count; base += kGatherBatch * kT) {
    unsigned long long w[kGatherBatch];
    int ix[kGatherBatch];
    unsigned miss = 0u;
#pragma unroll
    for (int j = 0; j < kGatherBatch; ++j) {
      const int k = base + j * kT + static_cast<int>(threadIdx.x);
      ix[j] = k < count ? static_cast<int>(idx.next()) : -1;
      w[j] = ix[j] >= 0 ? ld_rlx64(mb + ix[j]) : 0ull;
      if (ix[j] >= 0) miss |= 1u << j;
    }
    const long long t0 = clock64();
#pragma unroll 1
    for (unsigned n = 1; !bad; ++n) {
#pragma unroll
      for (int j = 0; j < kGatherBatch; ++j)
        if ((miss >> j & 1u) && static_cast<unsigned>(w[j] >> 32) == ep) {
          dst[base + j * kT + threadIdx.x] = static_cast<unsigned>(w[j]);
          miss &= ~(1u << j);
        }
      if (!miss) break;
#pragma unroll
      for (int j = 0; j < kGatherBatch; ++j)
        if (miss >> j & 1u) w[j] = ld_rlx64(mb + ix[j]);
      if (expired(p, t0, n)) bad = 1;
    }
  }
  return !__syncthreads_or(bad);
}
// Index functors: next() gives the word index of the thread's next k (k = tid, tid + kT, ...).
struct IdxLin {
  long long k;
  __device__ IdxLin() : k(static_cast<long long>(threadIdx.x) - kT) {}
  __device__ long long next() { return k += kT; }
};
// All-reduce slice: k -> [k >> lg_hs][slice0 + (k & (hs - 1))] with rows of H words.
struct IdxSlice {
  int k, lg, msk, H, slice0;
  __device__ IdxSlice(int lg_hs, int H_, int s0) : k(static_cast<int>(threadIdx.x) - kT), lg(lg_hs),
                                                   msk((1 << lg_hs) - 1), H(H_), slice0(s0) {}
  __device__ long long next() {
    k += kT;
    return static_cast<long long>(k >> lg) * H + slice0 + (k & msk);
  }
};
// Attention partials of this CTA's dims [q0, q0 + nq) and the (m, l) of the heads they touch,
// from every attention CTA: k -> (a, j) with j < per; j < nq: dim q0 + j, else (m, l) of head
// hlo + (j - nq) / 2; word (a nh + h)(d + 2) + e.
struct IdxPart {
  int a, j, per, nq, q0, hlo, lg_d, d, nh, da, dj;
  __device__ IdxPart(int per_, int nq_, int q0_, int hlo_, int lg_d_, int nh_)
      : per(per_), nq(nq_), q0(q0_), hlo(hlo_), lg_d(lg_d_), d(1 << lg_d_), nh(nh_) {
    const int t = static_cast<int>(threadIdx.x);
    a = per > 0 ? t / per : 0;
    j = per > 0 ? t % per : 0;
    da = per > 0 ? kT / per : 0;
    dj = per > 0 ? kT % per : 0;
    // stepping back once lets next() advance uniformly
    a -= da;
    j -= dj;
    if (j < 0) {
      j += per;
      a -= 1;
    }
  }
  __device__ long long next() {
    a += da;
    j += dj;
    if (j >= per) {
      j -= per;
      a += 1;
    }
    int h, e;
    if (j < nq) {
      h = (q0 + j) >> lg_d;
      e = (q0 + j) & (d - 1);
    } else {
      h = hlo + ((j - nq) >> 1);
      e = d + ((j - nq) & 1);
    }
    return (static_cast<long long>(a) * nh + h) * (d + 2) + e;
  }
};
__device__ __forceinline__ bool gather_lin(const Params& p, const unsigned long long* mb, int count, unsigned* dst,
                                        unsigned ep) {
  return gather_t(p, mb, count, IdxLin(), dst, ep);
}
__device__ __forceinline__ bool gather_slice(const Params& p, const unsigned long long* mb, int count, int slice0,
                                          unsigned* dst, unsigned ep) {
  return gather_t(p, mb, count, IdxSlice(p.lg_hs, p.H, slice0), dst, ep);
}
__device__ __forceinline__ bool gather_part(const Params& p, const unsigned long long* mb, int count, int per, int nq,
                                         int q0, int hlo, int lg_d, unsigned* dst, unsigned ep) {
  return gather_t(p, mb, count, IdxPart(per, nq, q0, hlo, lg_d, p.nh), dst, ep);
}

// ------------------------------------------------------------------ per-warp vector math

// Lane l holds elements [l * EPL, (l + 1) * EPL) of an H-vector (H = 32 * EPL).
template <int EPL>
__device__ __forceinline__ void lds_vec(const float* v, float (&r)[EPL]) {
  const int l = threadIdx.x & 31;
#pragma unroll
  for (int e = 0; e < EPL; ++e) r[e] = v[l * EPL + e];
}
template <int EPL>
__device__ __forceinline__ void ldg_vec(const float* v, float (&r)[EPL]) {
  const int l = threadIdx.x & 31;
#pragma unroll
  for (int e = 0; e < EPL; ++e) r[e] = __ldg(v + l * EPL + e);
}
// 1 / sqrt(mean(v^2) + eps) over the warp's H-vector.
template <int EPL>
__device__ __forceinline__ float rms_inv(const float (&r)[EPL], float eps) {
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) s = fmaf(r[e], r[e], s);
  s = warp_sum(s);
  return rsqrtf(s / static_cast<float>(32 * EPL) + eps);
}
__device__ __forceinline__ void bf8(const uint4& u, float* f) {
  const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h2[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
// Row (bf16, H elements, 16-byte aligned) . vector held by the warp; every lane gets the sum.
template <int EPL>
__device__ __forceinline__ float dot_row(const bf16* row, const float (&a)[EPL]) {
  const int l = threadIdx.x & 31;
  float s = 0.f;
  if constexpr (EPL % 8 == 0) {
#pragma unroll
    for (int v = 0; v < EPL / 8; ++v) {
      float f[8];
      bf8(*reinterpret_cast<const uint4*>(row + l * EPL + 8 * v), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) s = fmaf(f[i], a[8 * v + i], s);
    }
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e) s = fmaf(bf(row[l * EPL + e]), a[e], s);
  }
  return warp_sum(s);
}

// Sum of w[k] v[k] over k < n: w a bf16 row of even pitch (4-byte aligned), v fp32 in shared
// memory (8-byte aligned); pairs of k in two accumulation chains.
__device__ __forceinline__ float dot_col(const bf16* w, const float* v, int n) {
  float a0 = 0.f, a1 = 0.f;
  int k = 0;
#pragma unroll 4
  for (; k + 1 < n; k += 2) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(w + k));
    const float2 u = *reinterpret_cast<const float2*>(v + k);
    a0 = fmaf(f.x, u.x, a0);
    a1 = fmaf(f.y, u.y, a1);
  }
  if (k < n) a0 = fmaf(bf(w[k]), v[k], a0);
  return a0 + a1;
}

// ------------------------------------------------------------------ all-reduce

// Sums the H-vector vs[] of every CTA of the grid; returns the shared-memory address of the
// result (valid until the all-reduce after next). Slot (arn & 1) of the receive buffers and
// barriers; parity (arn >> 1) & 1. All threads call; *ok is block-uniform.
__device__ __forceinline__ float* all_reduce(const Params& p, unsigned char* sm, const float* vs, int arn,
                                          unsigned long long* mbx, unsigned ep, int rank, int g, bool skip_publish,
                                          bool* ok) {
  const Layout& L = p.L;
  const int H = p.H, S = p.S, lg = p.lg_hs, hs = 1 << lg;
  const int slot = arn & 1;
  const unsigned par = static_cast<unsigned>(arn >> 1) & 1u;
  float* rs = reinterpret_cast<float*>(sm + L.rs) + slot * H;  // [source rank][hs]
  float* ag = reinterpret_cast<float*>(sm + L.ag) + slot * H;  // [H]
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(sm + L.bars);
  const unsigned rbar = sa(&bars[p.nl + 3 + slot]), abar = sa(&bars[p.nl + 5 + slot]);
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_expect_tx(rbar, static_cast<unsigned>(H * 4));
    mbar_expect_tx(abar, static_cast<unsigned>(H * 4));
  }
  __syncthreads();  // vs complete
  // 1) reduce-scatter in the cluster: dims [q hs, (q + 1) hs) go to rank q
#pragma unroll 1
  for (int i2 = tid; i2 < H / 2; i2 += kT) {
    const int i = 2 * i2, q = i >> lg, e = i & (hs - 1);
    const unsigned long long v =
        (static_cast<unsigned long long>(__float_as_uint(vs[i + 1])) << 32) | __float_as_uint(vs[i]);
    st_async_u64(mapa(sa(rs + rank * hs + e), q), v, mapa(rbar, q));
  }
  if (!mbar_wait(p, rbar, par, true)) {
    *ok = false;
    return ag;
  }
  // 2) this cluster's partial of my slice -> global; every cluster's partial of my slice <- global
  float* ub = reinterpret_cast<float*>(sm + L.ubuf);
  if (!skip_publish && tid < hs) {
    float s = 0.f;
#pragma unroll 1
    for (int q = 0; q < S; ++q) s += rs[q * hs + tid];
    put(mbx, static_cast<long long>(g) * H + rank * hs + tid, s, ep);
  }
  if (!gather_slice(p, mbx, p.G * hs, rank * hs, reinterpret_cast<unsigned*>(ub), ep)) {
    *ok = false;
    return ag;
  }
  // sums over the clusters in a fixed order: P consecutive lanes per dim, then a butterfly
  {
    const int lgP = kLgT - lg < 5 ? kLgT - lg : 5;  // log2 of the threads per dim
    const int P = 1 << lgP;
    const int e = tid >> lgP, part = tid & (P - 1);
    float s = 0.f;
    if (e < hs) {
#pragma unroll 1
      for (int gg = part; gg < p.G; gg += P) s += ub[gg * hs + e];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      if (o < P) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (e < hs && part == 0) rs[e] = s;  // the slot's reduce-scatter data is consumed
  }
  __syncthreads();
  // 3) all-gather of the slices in the cluster
#pragma unroll 1
  for (int t = tid; t < S * (hs / 2); t += kT) {
    const int q = t >> (lg - 1), e = 2 * (t & (hs / 2 - 1));
    const unsigned long long v =
        (static_cast<unsigned long long>(__float_as_uint(rs[e + 1])) << 32) | __float_as_uint(rs[e]);
    st_async_u64(mapa(sa(ag + rank * hs + e), q), v, mapa(abar, q));
  }
  if (!mbar_wait(p, abar, par, true)) {
    *ok = false;
    return ag;
  }
  return ag;
}

// ------------------------------------------------------------------ top-k

// Exclusive prefix sum of v over the CTA's threads in thread order (ws: 48 ints); also the
// total through *tot.
__device__ __forceinline__ int block_excl_scan(int v, int* ws, int* tot) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += u;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kW ? ws[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    if (lane < kW) ws[32 + lane] = w;
  }
  __syncthreads();
  *tot = ws[32 + kW - 1];
  const int r = (warp > 0 ? ws[32 + warp - 1] : 0) + x - v;
  __syncthreads();
  return r;
}
// (value, index) -> key whose maximum is the largest value, lowest index among equal values.
__device__ __forceinline__ unsigned long long topk_key(const float* cl, int i) {
  return (static_cast<unsigned long long>(ord_f32(cl[i])) << 32) | (0xffffffffu - static_cast<unsigned>(i));
}

// Indices of the k largest of cl[0..C) (fp32; equal values: lower index first), written to
// sel[] in increasing index order. Bound: split the C logits into k groups; the smallest of
// the k group maxima is at most the k-th largest key, so every selected key lies at or above
// it. The keys at or above the bound (few: about k to 3k) are compacted in index order and
// each is ranked against the others. All threads call.
//
// Any C and k: one warp per group, ranks by ballots (shapes the tiled form below does not
// cover, and candidate sets that overflow its buffer).
__device__ __noinline__ void topk_generic(const Params& p, unsigned char* sm, const float* cl, int* sel) {
  const Layout& L = p.L;
  const int C = p.C, k = p.topk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned long long* gmax = reinterpret_cast<unsigned long long*>(sm + L.gmax);
  int* ws = reinterpret_cast<int*>(sm + L.red);
  int* cidx = reinterpret_cast<int*>(sm + L.qs);
  unsigned long long* ckey = reinterpret_cast<unsigned long long*>(sm + L.qs + ((L.cand_cap * 4 + 15) & ~15));
  // this thread's contiguous chunk of keys, kept in registers (up to kChunk)
  constexpr int kChunk = 8;
  const int per = cdiv(C, kT), i0 = min(C, tid * per), i1 = min(C, i0 + per);
  const bool regs = per <= kChunk;
  unsigned long long key[kChunk];
#pragma unroll
  for (int j = 0; j < kChunk; ++j) key[j] = regs && i0 + j < i1 ? topk_key(cl, i0 + j) : 0ull;
  // group maxima: when the k groups are runs of 2^j whole per-thread chunks, a thread's chunk
  // maximum and a butterfly over the group's lanes; else one warp per group
  const int tpg = (C / k) / per;  // threads per group
  const bool tiled = regs && C % k == 0 && (C / k) % per == 0 && tpg >= 1 && tpg <= 32 && (tpg & (tpg - 1)) == 0 &&
                     tpg * k <= kT;
  if (tiled) {
    unsigned long long m = 0ull;
#pragma unroll
    for (int j = 0; j < kChunk; ++j) m = key[j] > m ? key[j] : m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      if (o < tpg) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, m, o);
        m = w > m ? w : m;
      }
    if ((tid & (tpg - 1)) == 0 && tid / tpg < k) gmax[tid / tpg] = m;
  }
#pragma unroll 1
  for (int r = tiled ? k : warp; r < k; r += kW) {
    const int lo = static_cast<int>(static_cast<long long>(C) * r / k), hi = static_cast<int>(static_cast<long long>(C) * (r + 1) / k);
    unsigned long long m = 0ull;
#pragma unroll 1
    for (int i = lo + lane; i < hi; i += 32) {
      const unsigned long long kk = topk_key(cl, i);
      m = kk > m ? kk : m;
    }
    m = warp_max_u64(m);
    if (lane == 0) gmax[r] = m;
  }
  __syncthreads();
  // the bound: smallest group maximum (every warp computes it)
  unsigned long long bnd = ~0ull;
#pragma unroll 1
  for (int r = lane; r < k; r += 32) bnd = gmax[r] < bnd ? gmax[r] : bnd;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, bnd, o);
    bnd = w < bnd ? w : bnd;
  }
  // candidates at or above the bound, in index order
  int n = 0;
  if (regs) {
#pragma unroll
    for (int j = 0; j < kChunk; ++j) n += key[j] >= bnd && key[j] != 0ull;
  } else {
#pragma unroll 1
    for (int i = i0; i < i1; ++i) n += topk_key(cl, i) >= bnd;
  }
  int M = 0;
  int pos = block_excl_scan(n, ws, &M);
  const bool fits = M <= L.cand_cap;
  if (fits) {
    if (regs) {
#pragma unroll
      for (int j = 0; j < kChunk; ++j)
        if (key[j] >= bnd && key[j] != 0ull) {
          cidx[pos] = i0 + j;
          ckey[pos] = key[j];
          ++pos;
        }
    } else {
#pragma unroll 1
      for (int i = i0; i < i1; ++i) {
        const unsigned long long kk = topk_key(cl, i);
        if (kk >= bnd) {
          cidx[pos] = i;
          ckey[pos] = kk;
          ++pos;
        }
      }
    }
  }
  __syncthreads();
  int nsel = 0;
  if (fits) {
    // rank of each candidate among the candidates: one warp per candidate, the lanes comparing
    // 32 candidates at a time (ballot + population count); selected when fewer than k are larger
    int* flag = reinterpret_cast<int*>(sm + L.gmax);  // the group maxima are no longer needed
#pragma unroll 1
    for (int m = warp; m < M; m += kW) {
      const unsigned long long kk = ckey[m];
      int rk = 0;
#pragma unroll 2
      for (int b = 0; b < M; b += 32) {
        const bool gt = b + lane < M && ckey[b + lane] > kk;
        rk += __popc(__ballot_sync(0xffffffffu, gt));
      }
      if (lane == 0) flag[m] = rk < k ? 1 : 0;
    }
    __syncthreads();
    // compaction in candidate (= index) order: one candidate per thread
    const int take = tid < M ? flag[tid] : 0;
    const int at = block_excl_scan(take, ws, &nsel);
    if (take && at < k) sel[at] = cidx[tid];
  } else {
    // slow exact path: every key against every key (only for pathological ties / distributions)
    int cnt = 0;
#pragma unroll 1
    for (int i = i0; i < i1; ++i) {
      const unsigned long long kk = topk_key(cl, i);
      int rk = 0;
      if (kk >= bnd) {
#pragma unroll 1
        for (int m = 0; m < C && rk < k; ++m) rk += topk_key(cl, m) > kk;
      }
      cnt += kk >= bnd && rk < k;
    }
    int at = block_excl_scan(cnt, ws, &nsel);
#pragma unroll 1
    for (int i = i0; i < i1; ++i) {
      const unsigned long long kk = topk_key(cl, i);
      if (kk < bnd) continue;
      int rk = 0;
#pragma unroll 1
      for (int m = 0; m < C && rk < k; ++m) rk += topk_key(cl, m) > kk;
      if (rk < k && at < k) sel[at++] = i;
    }
  }
  __syncthreads();
}

// The tiled form: C = 256 * per (per <= 8 keys in each thread's registers) and k groups of
// tpg = C / (k * per) consecutive threads (a power of two <= 32). The group maxima and their
// minimum (the bound) are taken on the 32-bit order of the values: a bound on the value alone
// still lies at or below the k-th largest key. The candidates (values at or above it) are
// compacted in index order with their full keys (value, then lower index first), and each is
// ranked by counting the larger candidate keys, two threads per candidate when at most 128.
// Three prefix sums by warp totals in shared memory (one barrier each).
__device__ __forceinline__ void topk_select(const Params& p, unsigned char* sm, const float* cl, int* sel) {
  const Layout& L = p.L;
  const int k = p.topk, lgper = p.tk_lg_per, lgtpg = p.tk_lg_tpg;
  if (lgtpg < 0) {
    topk_generic(p, sm, cl, sel);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per = 1 << lgper, tpg = 1 << lgtpg, i0 = tid << lgper;
  int* wsb = reinterpret_cast<int*>(sm + L.red);  // [kW] warp minima of the group maxima
  int* wsc = wsb + kW;                            // [kW] warp candidate counts
  int* wss = wsb + 2 * kW;                        // [kW] warp selection counts
  int* cidx = reinterpret_cast<int*>(sm + L.qs);
  unsigned long long* ckey = reinterpret_cast<unsigned long long*>(sm + L.qs + ((L.cand_cap * 4 + 15) & ~15));
  int* part = reinterpret_cast<int*>(sm + L.gmax);  // [2][128] partial ranks
  unsigned v[8];
  if (per == 8) {
    const float4 a = reinterpret_cast<const float4*>(cl + i0)[0], b = reinterpret_cast<const float4*>(cl + i0)[1];
    v[0] = ord_f32(a.x), v[1] = ord_f32(a.y), v[2] = ord_f32(a.z), v[3] = ord_f32(a.w);
    v[4] = ord_f32(b.x), v[5] = ord_f32(b.y), v[6] = ord_f32(b.z), v[7] = ord_f32(b.w);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = j < per ? ord_f32(cl[i0 + j]) : 0u;
  }
  // group maxima (a tree over the thread's keys, then a butterfly over the group's lanes), and
  // their minimum over the warp's groups
  unsigned gm = max(max(max(v[0], v[1]), max(v[2], v[3])), max(max(v[4], v[5]), max(v[6], v[7])));
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned w = __shfl_xor_sync(0xffffffffu, gm, o);
    gm = o < tpg ? max(gm, w) : min(gm, w);
  }
  if (lane == 0) wsb[warp] = static_cast<int>(gm);
  __syncthreads();
  unsigned bnd = 0xffffffffu;
#pragma unroll
  for (int w = 0; w < kW; ++w) bnd = min(bnd, static_cast<unsigned>(wsb[w]));
  // candidates: values at or above the bound, compacted in index order
  int n = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) n += j < per && v[j] >= bnd;
  int x = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += u;
  }
  if (lane == 31) wsc[warp] = x;
  __syncthreads();
  int M = 0, pos = x - n;
#pragma unroll
  for (int w = 0; w < kW; ++w) {
    const int c = wsc[w];
    M += c;
    pos += w < warp ? c : 0;
  }
  const int M8 = (M + 7) & ~7;
  if (M8 > L.cand_cap) {  // block-uniform; only for heavy ties at the bound
    topk_generic(p, sm, cl, sel);
    return;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < per && v[j] >= bnd) {
      cidx[pos] = i0 + j;
      ckey[pos] = (static_cast<unsigned long long>(v[j]) << 32) | (0xffffffffu - static_cast<unsigned>(i0 + j));
      ++pos;
    }
  if (tid < M8 - M) ckey[M + tid] = 0ull;  // padding: never larger than a candidate
  __syncthreads();
  // ranks: the number of larger candidate keys; candidate m, half h of the candidates
  const bool two = M8 <= 128;
  const int m = two ? (tid & 127) : tid, h = two ? (tid >> 7) : 0;
  const int span = two ? (M8 >> 1) : M8, j0 = h * span;
  if (m < M) {
    const unsigned long long mk = ckey[m];
    int rk = 0;
#pragma unroll 4
    for (int j = j0; j < j0 + span; ++j) rk += ckey[j] > mk;
    part[(h << 7) + m] = rk;
  }
  __syncthreads();
  const bool take = tid < M && (two ? part[tid] + part[128 + tid] : part[tid]) < k;
  const unsigned bal = __ballot_sync(0xffffffffu, take);
  if (lane == 0) wss[warp] = __popc(bal);
  __syncthreads();
  int at = __popc(bal & ((1u << lane) - 1u));
#pragma unroll
  for (int w = 0; w < kW; ++w) at += w < warp ? wss[w] : 0;
  if (take && at < k) sel[at] = cidx[tid];
  __syncthreads();
}

// ------------------------------------------------------------------ attention of one block

// This CTA's keys of one block: q_norm + RoPE (+ the softmax scale) of every head from the
// gathered raw q (ub), scores of every (key, head), softmax statistics (max, exp-sum) per
// head, the probability-weighted key sums (V = K); publishes [c][h][d + 2] (sums, max,
// exp-sum) to the owners of q's dims. Any head dim (the general form). g[0..7]: the q_norm
// gains (j, j + d/2) of this thread's first four RoPE pairs, loaded before the q gather waits.
// All threads call.
__device__ __forceinline__ void attend(const Params& p, unsigned char* sm, int l, int t, int c, int nk, const bf16* kb,
                                      long long kst, unsigned long long* ma, unsigned epa, const float (&g)[16]) {
  const Layout& L = p.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nh = p.nh, nkv = p.nkv, lg = p.lg_d[t], d = 1 << lg, grp = nh / nkv, half = d >> 1, ksl = L.ksl;
  float* ub = reinterpret_cast<float*>(sm + L.ubuf);
  float* qs = reinterpret_cast<float*>(sm + L.qs);
  float* sc = reinterpret_cast<float*>(sm + L.sc);
  float* red = reinterpret_cast<float*>(sm + L.red);
  const float2* cs = reinterpret_cast<const float2*>(sm + L.cs) + (t ? p.d[0] / 2 : 0);
  // per-head q_norm factor (one warp per head)
#pragma unroll 1
  for (int h = warp; h < nh; h += kW) {
    float s2 = 0.f;
#pragma unroll 1
    for (int e = lane; e < d; e += 32) s2 = fmaf(ub[h * d + e], ub[h * d + e], s2);
    s2 = warp_sum(s2);
    if (lane == 0) red[h] = rsqrtf(s2 / static_cast<float>(d) + p.eps);
  }
  __syncthreads();
  {
    const float* gqn = p.q_norm[l];
    const float scale = p.scale[t];
    int k = 0;
#pragma unroll 1
    for (int i = tid; i < nh * half; i += kT, ++k) {
      const int h = i >> (lg - 1), j = i & (half - 1);
      float g0, g1;
      if (k < 4) {  // prefetched: the gains of this thread's first four pairs
        g0 = k == 0 ? g[0] : (k == 1 ? g[2] : (k == 2 ? g[4] : g[6]));
        g1 = k == 0 ? g[1] : (k == 1 ? g[3] : (k == 2 ? g[5] : g[7]));
      } else {
        g0 = __ldg(gqn + j);
        g1 = __ldg(gqn + j + half);
      }
      const float rn = red[h];
      const float a = ub[h * d + j] * rn * g0, b = ub[h * d + j + half] * rn * g1;
      const float2 cw = cs[j];
      qs[h * d + j] = (a * cw.x - b * cw.y) * scale;
      qs[h * d + j + half] = (b * cw.x + a * cw.y) * scale;
    }
  }
  __syncthreads();
  // scores: one warp per (pair of keys, KV head, group of up to 4 of its query heads); every
  // lane a run of 16-byte vectors of the keys; the 8 partial sums (2 keys x 4 heads) are
  // reduced by a transposed butterfly that leaves each sum in 4 lanes
  const int nvec = d >> 3;
#pragma unroll 1
  for (int j0 = 2 * warp; j0 < nk; j0 += 2 * kW) {
    const bool two = j0 + 1 < nk;
#pragma unroll 1
    for (int kh = 0; kh < nkv; ++kh) {
      const bf16* kr0 = kb + static_cast<size_t>(j0) * kst + kh * d;
      const bf16* kr1 = two ? kr0 + kst : kr0;
#pragma unroll 1
      for (int q0 = 0; q0 < grp; q0 += 4) {
        const float* qh = qs + (kh * grp + q0) * d;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // [key][head]
#pragma unroll 1
        for (int v = lane; v < nvec; v += 32) {
          float k0[8], k1[8];
          bf8(*reinterpret_cast<const uint4*>(kr0 + 8 * v), k0);
          bf8(*reinterpret_cast<const uint4*>(kr1 + 8 * v), k1);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (q0 + q < grp) {
              const float4* qv = reinterpret_cast<const float4*>(qh + q * d + 8 * v);
              const float4 a = qv[0], b = qv[1];
              const float qq[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
              float u0 = acc[q], u1 = acc[4 + q];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                u0 = fmaf(qq[i], k0[i], u0);
                u1 = fmaf(qq[i], k1[i], u1);
              }
              acc[q] = u0;
              acc[4 + q] = u1;
            }
          }
        }
        // butterfly: 8 values over offsets 16, 8, 4 (each halving the values a lane keeps),
        // then the full sum over offsets 2 and 1; lane l ends with value (l >> 2) & 7
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool up = lane & 16;
          const float send = up ? acc[i] : acc[i + 4], keep = up ? acc[i + 4] : acc[i];
          acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const bool up = lane & 8;
          const float send = up ? acc[i] : acc[i + 2], keep = up ? acc[i + 2] : acc[i];
          acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        {
          const bool up = lane & 4;
          const float send = up ? acc[0] : acc[1], keep = up ? acc[1] : acc[0];
          acc[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 2);
        acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 1);
        // value index: bit 2 from lane bit 4, bit 1 from lane bit 3, bit 0 from lane bit 2
        if ((lane & 3) == 0) {
          const int vi = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
          const int key = vi >> 2, q = vi & 3;
          if (q0 + q < grp && (key == 0 || two)) sc[(kh * grp + q0 + q) * ksl + j0 + key] = acc[0];
        }
      }
    }
  }
  __syncthreads();
  // softmax statistics and probabilities (one warp per head)
#pragma unroll 1
  for (int h = warp; h < nh; h += kW) {
    float m = -INFINITY;
#pragma unroll 1
    for (int j = lane; j < nk; j += 32) m = fmaxf(m, sc[h * ksl + j]);
    m = warp_max(m);
    float lsum = 0.f;
#pragma unroll 1
    for (int j = lane; j < nk; j += 32) {
      const float e = expf(sc[h * ksl + j] - m);
      sc[h * ksl + j] = e;
      lsum += e;
    }
    lsum = warp_sum(lsum);
    if (lane == 0) {
      red[16 + h] = m;
      red[32 + h] = lsum;
    }
  }
  __syncthreads();
  // probability-weighted key sums: one thread per two dims of a KV head row and group of up
  // to 4 of its heads; published straight from registers
  const int row = nkv * d;
#pragma unroll 1
  for (int q0 = 0; q0 < grp; q0 += 4) {
#pragma unroll 1
    for (int i2 = tid; i2 < (row >> 1); i2 += kT) {
      const int i = 2 * i2, kh = i >> lg, e = i & (d - 1);
      const float* pr = sc + (kh * grp + q0) * ksl;
      float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
      const bf16* kp = kb + i;
#pragma unroll 4
      for (int j = 0; j < nk; ++j, kp += kst) {
        const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(kp));
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float pj = q0 + q < grp ? pr[q * ksl + j] : 0.f;
          a0[q] = fmaf(pj, kv.x, a0[q]);
          a1[q] = fmaf(pj, kv.y, a1[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q0 + q < grp) {
          const long long base = (static_cast<long long>(c) * nh + kh * grp + q0 + q) * (d + 2) + e;
          put(ma, base, a0[q], epa);
          put(ma, base + 1, a1[q], epa);
        }
    }
  }
  if (tid < nh) {
    put(ma, (static_cast<long long>(c) * nh + tid) * (d + 2) + d, red[16 + tid], epa);
    put(ma, (static_cast<long long>(c) * nh + tid) * (d + 2) + d + 1, red[32 + tid], epa);
  }
}

// The same for head dims d = 32 * DL (256 or 512) and four query heads (V = K):
//   A: warp h takes head h's q_norm statistic over all d dims.
//   B: lane i holds the 8-dim runs starting at 8 (i + 32 v), v < DL / 8, of q for every head
//      (q_norm gain, RoPE with the partner dims d/2 away, softmax scale); warp w takes keys w,
//      w + 8, ... in passes of KB keys: the lane's partial dot products of the pass's keys
//      with the four heads are summed over the lanes by a transposed butterfly, and the lanes
//      that end with a whole (key, head) score store it.
//   C: warp h: softmax statistics of head h over the keys; probabilities in place.
//   D: warp w owns dims [w d/8, (w+1) d/8), d/256 consecutive dims per lane: the
//      probability-weighted key sums of its dims for every head, published with the
//      statistics as [c][h][d + 2].
// The (cos, sin) table is lane-major for these dims (consecutive lanes read consecutive
// entries). g: this lane's q_norm gains of its runs, then (d = 256) of its partner runs,
// loaded before the q gather waits. All threads call.
template <int DL>
__device__ __forceinline__ void attend_g(const Params& p, unsigned char* sm, int t, int c, int nk, const bf16* kb,
                                         long long kst, unsigned long long* ma, unsigned epa, const float (&g)[16]) {
  constexpr int d = 32 * DL, half = d / 2, NV = DL / 8, LG = half / 8, NH = 4;
  constexpr int KB = DL == 8 ? 1 : 4, NVAL = KB * NH, DPL = d / 256, DW = d / kW;
  const Layout& L = p.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkv = p.nkv;
  const float* ub = reinterpret_cast<const float*>(sm + L.ubuf);
  float* sc = reinterpret_cast<float*>(sm + L.sc);    // [key][head] scores, then probabilities
  float* red = reinterpret_cast<float*>(sm + L.red);  // [h]: q_norm factor; [16 + h] max; [32 + h] exp-sum
  const float2* cs = reinterpret_cast<const float2*>(sm + L.cs) + (t ? p.d[0] / 2 : 0);
  // A
  if (warp < NH) {
    const float4* qv = reinterpret_cast<const float4*>(ub + warp * d);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < d / 128; ++i) {
      const float4 a = qv[lane + 32 * i];
      ss = fmaf(a.x, a.x, fmaf(a.y, a.y, fmaf(a.z, a.z, fmaf(a.w, a.w, ss))));
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = rsqrtf(ss / static_cast<float>(d) + p.eps);
  }
  __syncthreads();
  // B: q runs of every head
  float q[NH][DL];
  {
    const float scale = p.scale[t];
    const int pl = NV == 2 ? lane : (lane & 15);  // pair run of this lane
    float2 cw[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) cw[e] = cs[e * LG + pl];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const float rn = red[h];
      float x[DL], y[DL];
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const float4* a4 = reinterpret_cast<const float4*>(ub + h * d + 8 * (lane + 32 * v));
        const float4 a = a4[0], b = a4[1];
        x[8 * v] = a.x, x[8 * v + 1] = a.y, x[8 * v + 2] = a.z, x[8 * v + 3] = a.w;
        x[8 * v + 4] = b.x, x[8 * v + 5] = b.y, x[8 * v + 6] = b.z, x[8 * v + 7] = b.w;
      }
      if (NV == 2) {
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = x[8 + e], y[8 + e] = x[e];
#pragma unroll
        for (int i = 0; i < DL; ++i) x[i] *= rn * g[i], y[i] *= rn * g[(i + 8) & 15];
      } else {
        const float4* a4 = reinterpret_cast<const float4*>(ub + h * d + 8 * (lane ^ 16));
        const float4 a = a4[0], b = a4[1];
        y[0] = a.x, y[1] = a.y, y[2] = a.z, y[3] = a.w, y[4] = b.x, y[5] = b.y, y[6] = b.z, y[7] = b.w;
#pragma unroll
        for (int i = 0; i < DL; ++i) x[i] *= rn * g[i], y[i] *= rn * g[8 + i];
      }
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const bool lo = NV == 2 ? v == 0 : lane < 16;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xv = x[8 * v + e], yv = y[8 * v + e];
          q[h][8 * v + e] = (lo ? fmaf(xv, cw[e].x, -yv * cw[e].y) : fmaf(xv, cw[e].x, yv * cw[e].y)) * scale;
        }
      }
    }
  }
  // B: scores, KB keys per pass
#pragma unroll 1
  for (int j0 = warp; j0 < nk; j0 += KB * kW) {
    float v[NVAL];
#pragma unroll
    for (int i = 0; i < NVAL; ++i) v[i] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KB; ++kk) {
      const int j = j0 + kk * kW;
      if (j < nk) {
#pragma unroll
        for (int kh = 0; kh < NH; ++kh) {
          if (kh < nkv) {
            float kf[DL];
#pragma unroll
            for (int u = 0; u < NV; ++u)
              bf8(*reinterpret_cast<const uint4*>(kb + static_cast<long long>(j) * kst + kh * d + 8 * (lane + 32 * u)),
                  kf + 8 * u);
#pragma unroll
            for (int h = 0; h < NH; ++h)
              if ((h * nkv) / NH == kh) {
                float a = 0.f;
#pragma unroll
                for (int i = 0; i < DL; ++i) a = fmaf(q[h][i], kf[i], a);
                v[kk * NH + h] = a;
              }
          }
        }
      }
    }
    // transposed butterfly: while a lane keeps several values each offset halves them, the
    // remaining offsets finish the sums; lane i ends with value i / (32 / NVAL)
#pragma unroll
    for (int off = 16, n = NVAL; off >= 1; off >>= 1) {
      if (n > 1) {
        const bool up = lane & off;
#pragma unroll
        for (int i = 0; i < NVAL / 2; ++i)
          if (i < n / 2) {
            const float send = up ? v[i] : v[i + n / 2], keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
          }
        n >>= 1;
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
      }
    }
    const int vi = lane / (32 / NVAL), j = j0 + (vi / NH) * kW;
    if ((lane & (32 / NVAL - 1)) == 0 && j < nk) sc[j * NH + (vi & (NH - 1))] = v[0];
  }
  __syncthreads();
  // C
  if (warp < NH) {
    const int h = warp;
    float m = -INFINITY;
#pragma unroll 1
    for (int j = lane; j < nk; j += 32) m = fmaxf(m, sc[j * NH + h]);
    m = warp_max(m);
    float l = 0.f;
#pragma unroll 1
    for (int j = lane; j < nk; j += 32) {
      const float e = expf(sc[j * NH + h] - m);
      sc[j * NH + h] = e;
      l += e;
    }
    l = warp_sum(l);
    if (lane == 0) {
      red[16 + h] = m;
      red[32 + h] = l;
    }
  }
  __syncthreads();
  // D
  const int dim0 = warp * DW + lane * DPL;
  float acc[NH][DPL];
#pragma unroll
  for (int h = 0; h < NH; ++h)
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[h][k] = 0.f;
#pragma unroll 4
  for (int j = 0; j < nk; ++j) {
    const float4 pv = *reinterpret_cast<const float4*>(sc + j * NH);
    const float pj[NH] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
    for (int kh = 0; kh < NH; ++kh) {
      if (kh < nkv) {
        float kf[DPL];
        const bf16* kr = kb + static_cast<long long>(j) * kst + kh * d + dim0;
        if (DPL == 2) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(kr));
          kf[0] = f.x;
          kf[DPL - 1] = f.y;
        } else {
          kf[0] = bf(kr[0]);
        }
#pragma unroll
        for (int h = 0; h < NH; ++h)
          if ((h * nkv) / NH == kh)
#pragma unroll
            for (int k = 0; k < DPL; ++k) acc[h][k] = fmaf(pj[h], kf[k], acc[h][k]);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const long long base = (static_cast<long long>(c) * NH + h) * (d + 2);
#pragma unroll
    for (int k = 0; k < DPL; ++k) put(ma, base + dim0 + k, acc[h][k], epa);
  }
  if (tid < NH) {
    put(ma, (static_cast<long long>(c) * NH + tid) * (d + 2) + d, red[16 + tid], epa);
    put(ma, (static_cast<long long>(c) * NH + tid) * (d + 2) + d + 1, red[32 + tid], epa);
  }
}

// ------------------------------------------------------------------ the kernel

template <int EPL>
__global__ void __launch_bounds__(kT, 1) k_block_gr(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char sm[];
  const Layout& L = p.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, rank = cluster_rank(), g = c / p.S;
  const int H = p.H, nl = p.nl, nh = p.nh;
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(sm + L.bars);
  float* ub = reinterpret_cast<float*>(sm + L.ubuf);
  float* hc = reinterpret_cast<float*>(sm + L.hc);
  float* vs = reinterpret_cast<float*>(sm + L.vs);
  float* vh = reinterpret_cast<float*>(sm + L.vh);
  float* ms = reinterpret_cast<float*>(sm + L.ms);
  float2* cs = reinterpret_cast<float2*>(sm + L.cs);
  float* red = reinterpret_cast<float*>(sm + L.red);
  unsigned long long* wkeys = reinterpret_cast<unsigned long long*>(sm + L.keys);
  int* sel = reinterpret_cast<int*>(sm + L.sel);
  float* qsbuf = reinterpret_cast<float*>(sm + L.qs);  // free outside the attention: combine weights
  const int kbar = nl + 2;

  // ---- this CTA's shares (computed once): key ranges per type, q dims per type, FFN rows,
  // pre / post columns, centroid rows, candidate slots
  // (scalars per type, selected with t ? : -- no dynamically indexed local arrays, whose
  // accesses would go to local memory)
  int klo0 = 0;
  Range kr0{0, 0}, kr1{0, 0}, qr0{0, 0}, qr1{0, 0};
  if (p.has_type[0]) {
    int Lc = p.ctx_len[0][0];
    Lc = Lc < 0 ? 0 : (Lc > p.kv_max[0] ? p.kv_max[0] : Lc);
    klo0 = Lc - p.W > 0 ? Lc - p.W : 0;
    kr0 = c < p.A[0] ? split(Lc - klo0, p.A[0], c) : Range{0, 0};
    qr0 = split(nh * p.d[0], p.N, c);
  }
  if (p.has_type[1]) {
    int Lc = p.ctx_len[1][0];
    Lc = Lc < 0 ? 0 : (Lc > p.kv_max[1] ? p.kv_max[1] : Lc);
    kr1 = c < p.A[1] ? split(Lc, p.A[1], c) : Range{0, 0};
    qr1 = split(nh * p.d[1], p.N, c);
  }
  const Range fr = split(p.F, p.N, c), hr = split(p.bb, p.N, c), cr = split(p.C, p.N, c);
  const Range candr = split(p.topk * p.vsc, p.N, c);
  const int nf = fr.hi - fr.lo, nhc = hr.hi - hr.lo, ncr = cr.hi - cr.lo;
  // bulk copies of this CTA's keys of type t into the shared K region (kbuf + koff[t]); one
  // mbarrier phase per issue (both resident types together when they stay for the launch)
  int kph = 0, kwaited = 0, kcur = -1;
  auto k_bytes = [&](int t) {
    const Range kt = t ? kr1 : kr0;
    return static_cast<unsigned>((kt.hi - kt.lo) * p.nkv * p.d[t] * 2);
  };
  auto k_copy = [&](int t) {  // thread 0
    const Range kt = t ? kr1 : kr0;
    const int n = kt.hi - kt.lo, row = p.nkv * p.d[t];
    const bf16* k0 = p.k[t] + static_cast<size_t>((t ? 0 : klo0) + kt.lo) * static_cast<size_t>(p.st[t]);
    unsigned char* dst = sm + L.kbuf + L.koff[t];
    if (n <= 0) return;
    if (p.st[t] == row) {
      bulk_g2s(sa(dst), k0, static_cast<unsigned>(n * row * 2), sa(&bars[kbar]));
    } else {
#pragma unroll 1
      for (int j = 0; j < n; ++j)
        bulk_g2s(sa(dst + j * row * 2), k0 + static_cast<size_t>(j) * p.st[t], static_cast<unsigned>(row * 2),
                 sa(&bars[kbar]));
    }
  };
  auto k_resident = [&](int t) { return p.has_type[t] && p.kres[t] && c < p.A[t]; };
  auto k_issue = [&](int t) {
    if (tid == 0) {
      mbar_expect_tx(sa(&bars[kbar]), k_bytes(t));
      k_copy(t);
    }
    ++kph;
    kcur = t;
  };

  // ---- launch start. The inputs of the prologue are requested first, all at once (each one
  // is a memory round trip that would otherwise follow the previous one)
  const int h0 = p.d[0] / 2, h1 = p.d[1] / 2;
  const int pos_in = ldg_early_i32(p.pos);
  const int tok_in = ldg_early_i32(p.tok_in);
  double fq0 = 0.0, fq1 = 0.0;
  {
    const int hm = h0 > h1 ? h0 : h1;
    if (tid < h0 + h1) fq0 = ldg_early_f64(p.inv_freq + (tid < h0 ? tid : hm + tid - h0));
    if (tid + kT < h0 + h1) fq1 = ldg_early_f64(p.inv_freq + (tid + kT < h0 ? tid + kT : hm + tid + kT - h0));
  }
  const unsigned short hv = tid < nhc ? ldg_early_u16(p.hidden_in + hr.lo + tid) : static_cast<unsigned short>(0);
  // this CTA's share of the mailbox lines into L2: in a cold L2 the first poll of every word
  // of step 0's exchanges would otherwise wait on DRAM
  {
    const long long lines = (p.mb_words * 8 + 127) / 128;
    const long long l0 = lines * c / p.N, l1 = lines * (c + 1) / p.N;
    const char* mbc = reinterpret_cast<const char*>(p.mb);
#pragma unroll 1
    for (long long ln = l0 + tid; ln < l1; ln += kT) asm volatile("prefetch.global.L2 [%0];" ::"l"(mbc + ln * 128));
  }
  // barriers, bulk copies of this CTA's weight image and first keys
  if (tid == 0) {
#pragma unroll 1
    for (int i = 0; i < nl + 7; ++i) mbar_init(sa(&bars[i]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const unsigned char* src = p.img + static_cast<size_t>(c) * static_cast<size_t>(p.img_bytes);
#pragma unroll 1
    for (int gi = 0; gi < nl + 2; ++gi) {
      const unsigned b = static_cast<unsigned>(L.grp_bytes[gi]);
      mbar_expect_tx(sa(&bars[gi]), b);
      if (b) bulk_g2s(sa(sm + L.grp_off[gi]), src + L.grp_off[gi], b, sa(&bars[gi]));
    }
  }
  if (p.kboth) {
    const bool r0 = k_resident(0), r1 = k_resident(1);
    if (r0 || r1) {
      if (tid == 0) {
        mbar_expect_tx(sa(&bars[kbar]), (r0 ? k_bytes(0) : 0u) + (r1 ? k_bytes(1) : 0u));
        if (r0) k_copy(0);
        if (r1) k_copy(1);
      }
      ++kph;
    }
  } else if (k_resident(p.ltype[0])) {
    k_issue(p.ltype[0]);
  }
  __syncthreads();
  // every peer's barriers must be initialised before any st.async: arrive now, wait just
  // before the first exchange
  cluster_arrive();

  // RoPE (cos, sin) at the block's constant position: angle pos * inv_freq in fp64, reduced
  // to [-pi, pi] in fp64, then sin / cos of the reduced angle in fp32 (fast forms: absolute
  // error below 1e-6 on [-pi, pi]); pairs tid and tid + kT (the table has at most 2 kT)
  {
    const double pos = static_cast<double>(pos_in);
    const double two_pi = 6.283185307179586, inv_two_pi = 0.15915494309189535;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = tid + k * kT;
      if (i >= h0 + h1) continue;
      const int t = i < h0 ? 0 : 1, ii = t ? i - h0 : i;
      const double ang = pos * (k ? fq1 : fq0);
      const double r = fma(-rint(ang * inv_two_pi), two_pi, ang);
      const float rf = static_cast<float>(r);
      // the four-head form (head dim 256): pair j at (j % 8) * 16 + j / 8, so that lanes
      // holding consecutive 8-dim runs read consecutive entries
      const int ht = t ? h1 : h0;
      const int at = ht == 128 && p.nh == 4 ? (ii & 7) * (ht >> 3) + (ii >> 3) : ii;
      cs[(t ? h0 : 0) + at] = make_float2(__cosf(rf), __sinf(rf));
    }
  }
  if (tid < nhc) hc[tid] = bf(__ushort_as_bfloat16(hv));
  int tok = tok_in;
  if (tok < 0 || tok >= p.V) {
    if (c == 0 && tid == 0) atomicCAS(p.status, 0, static_cast<int>(MTP_ERR_INVALID_ARG));
    tok = 0;
  }
  // step 0's embedding row (this CTA's columns) into L2 while the weights arrive
  if (tid < 2 && nhc > 0)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.tgt + static_cast<size_t>(tok) * p.bb + hr.lo + tid * (nhc - 1)));
  __syncthreads();

  bool ok = true;
  unsigned loaded = 0u;  // load groups already waited for
  auto need_group = [&](int gi) {
    if (ok && !(loaded >> gi & 1u)) {
      ok = mbar_wait(p, sa(&bars[gi]), 0u, true);
      loaded |= 1u << gi;
    }
  };
  // PRE partial over the h columns: W_pre[:, my h cols] h'[my cols]
  auto pre_h = [&]() {
    const bf16* pre = reinterpret_cast<const bf16*>(sm + L.pre);
#pragma unroll 1
    for (int i = tid; i < H; i += kT) vh[i] = dot_col(pre + i * L.kcp, hc, nhc);
  };
  int arn = 0;
  need_group(0);
  if (ok) pre_h();
  cluster_wait();

#pragma unroll 1
  for (int s = 0; s < p.n_draft && ok; ++s) {
    const unsigned ep0 = p.epoch_base + static_cast<unsigned>(s) * kExPerStep;
    const long long* xo = p.ex_off[s & 1];
    // ---------------- PRE: x0 = W_pre [h ; embed(tok)] over my columns, then all-reduce
#pragma unroll 1
    for (int r = tid; r < nhc; r += kT) red[r] = bf(p.tgt[static_cast<size_t>(tok) * p.bb + hr.lo + r]);
    float gA[EPL];
    ldg_vec<EPL>(p.attn_norm[0], gA);
    __syncthreads();
    {
      const bf16* pre = reinterpret_cast<const bf16*>(sm + L.pre);
#pragma unroll 1
      for (int i = tid; i < H; i += kT) vs[i] = vh[i] + dot_col(pre + (H + i) * L.kcp, red, nhc);
    }
    const bool skip = p.dbg_skip == c + 1 && s == 0;
    float* xr = all_reduce(p, sm, vs, arn++, p.mb + xo[0], ep0, rank, g, skip, &ok);
    if (!ok) break;
    float x[EPL];
    lds_vec<EPL>(xr, x);

#pragma unroll 1
    for (int l = 0; l < nl && ok; ++l) {
      need_group(1 + l);
      if (!ok) break;
      const int t = p.ltype[l], lg = p.lg_d[t], d = 1 << lg, QD = nh * d;
      const Range q_r = t ? qr1 : qr0;
      const int nq = q_r.hi - q_r.lo;
      // ---------------- Q: a = norm(x); my rows of W_q a
      {
        const float r = rms_inv<EPL>(x, p.eps);
        float a[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) a[e] = x[e] * r * gA[e];
        const bf16* wq = reinterpret_cast<const bf16*>(sm + L.q[l]);
        unsigned long long* mq = p.mb + xo[ex_q(l)];
#pragma unroll 1
        for (int rr = warp; rr < nq; rr += 2 * kW) {  // two rows at a time: reductions overlap
          const int r2 = rr + kW;
          const float v1 = dot_row<EPL>(wq + rr * H, a);
          const float v2 = r2 < nq ? dot_row<EPL>(wq + r2 * H, a) : 0.f;
          if (lane == 0) {
            put(mq, q_r.lo + rr, v1, ep0 + ex_q(l));
            if (r2 < nq) put(mq, q_r.lo + r2, v2, ep0 + ex_q(l));
          }
        }
      }
      // ---------------- ATT (attention CTAs): the partial softmax of my keys
      unsigned long long* ma = p.mb + xo[ex_att(l)];
      if (c < p.A[t]) {
        // q_norm gains loaded before the q gather waits: for the four-head form this lane's run
        // (8 dims at 8 lane) and its RoPE partner run (16 lanes away); for the general form the
        // pairs (j, j + d/2) of this thread's first four RoPE pairs
        const bool wide = d == 256 && nh == 4;
        float gw[16];
        {
          const float* gqn = p.q_norm[l];
          const int half = d / 2, np = nh * half;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (wide) {
              gw[i] = ldg_early(gqn + 8 * (i < 8 ? lane : (lane ^ 16)) + (i & 7));
            } else {
              const int pi = tid + (i >> 1) * kT;
              gw[i] = i < 8 && pi < np ? ldg_early(gqn + (pi & (half - 1)) + (i & 1) * half) : 0.f;
            }
          }
        }
        if (!gather_lin(p, p.mb + xo[ex_q(l)], QD, reinterpret_cast<unsigned*>(ub), ep0 + ex_q(l))) {
          ok = false;
          break;
        }
        const bool res = k_resident(t);
        if (res) {
          if (!p.kboth && kcur != t) k_issue(t);  // not scheduled ahead (cannot happen with the schedule below)
          if (kwaited < kph) {
            ok = mbar_wait(p, sa(&bars[kbar]), static_cast<unsigned>(kph - 1) & 1u, true);
            kwaited = kph;
            if (!ok) break;
          }
        }
        const Range kt = t ? kr1 : kr0;
        const bf16* kb = res ? reinterpret_cast<const bf16*>(sm + L.kbuf + L.koff[t])
                             : p.k[t] + static_cast<size_t>((t ? 0 : klo0) + kt.lo) * static_cast<size_t>(p.st[t]);
        const long long kst = res ? static_cast<long long>(p.nkv) * d : p.st[t];
        if (wide)
          attend_g<8>(p, sm, t, c, kt.hi - kt.lo, kb, kst, ma, ep0 + ex_att(l), gw);
        else
          attend(p, sm, l, t, c, kt.hi - kt.lo, kb, kst, ma, ep0 + ex_att(l), gw);
        // the next block of the other type (here or in the next step) finds its keys loaded
        const bool last = l == nl - 1;
        const int tn = p.ltype[last ? 0 : l + 1];
        if (!p.kboth && tn != t && k_resident(tn) && !(last && s == p.n_draft - 1)) {
          __syncthreads();  // every read of the region is done
          k_issue(tn);
        }
      }
      // ---------------- O: combine the partials of my dims; partial o' = W_o[:, my dims] o
      {
        const int hlo = nq > 0 ? q_r.lo >> lg : 0, nht = heads_touched(q_r.lo, q_r.hi, d);
        const int per = nq + 2 * nht, At = p.A[t];
        if (!gather_part(p, ma, At * per, per, nq, q_r.lo, hlo, lg, reinterpret_cast<unsigned*>(ub),
                         ep0 + ex_att(l))) {
          ok = false;
          break;
        }
        // per head touched: the sources' weights exp(m_a - M) and the denominator (one warp per
        // head); then per dim the weighted sum of the sources' partials (one warp per dim)
        float* wgt = qsbuf;  // [nht][At] source weights
#pragma unroll 1
        for (int hl = warp; hl < nht; hl += kW) {
          float m = -INFINITY;
#pragma unroll 4
          for (int a = lane; a < At; a += 32) m = fmaxf(m, ub[a * per + nq + 2 * hl]);
          m = warp_max(m);
          float den = 0.f;
#pragma unroll 4
          for (int a = lane; a < At; a += 32) {
            const float ma_ = ub[a * per + nq + 2 * hl];
            const float w_ = ma_ == -INFINITY ? 0.f : expf(ma_ - m);
            wgt[hl * At + a] = w_;
            den = fmaf(w_, ub[a * per + nq + 2 * hl + 1], den);
          }
          den = warp_sum(den);
          if (lane == 0) red[48 + hl] = den;
        }
        __syncthreads();
#pragma unroll 1
        for (int w = warp; w < nq; w += kW) {
          const int hl = ((q_r.lo + w) >> lg) - hlo;
          float num = 0.f;
#pragma unroll 4
          for (int a = lane; a < At; a += 32) num = fmaf(wgt[hl * At + a], ub[a * per + w], num);
          num = warp_sum(num);
          const float den = red[48 + hl];
          if (lane == 0) red[w] = den > 0.f ? num / den : 0.f;
        }
        __syncthreads();
        const bf16* wo = reinterpret_cast<const bf16*>(sm + L.o[l]);
#pragma unroll 1
        for (int i = tid; i < H; i += kT) vs[i] = dot_col(wo + i * L.nqp[l], red, nq);
      }
      float gPA[EPL], gF[EPL];
      ldg_vec<EPL>(p.post_attn_norm[l], gPA);
      ldg_vec<EPL>(p.ffn_norm[l], gF);
      float* opr = all_reduce(p, sm, vs, arn++, p.mb + xo[ex_o(l)], ep0 + ex_o(l), rank, g, false, &ok);
      if (!ok) break;
      // ---------------- MLP: x += norm(o'); f = norm(x); my rows of gelu(W_g f) * W_u f
      {
        float o[EPL];
        lds_vec<EPL>(opr, o);
        const float ro = rms_inv<EPL>(o, p.eps);
#pragma unroll
        for (int e = 0; e < EPL; ++e) x[e] += o[e] * ro * gPA[e];
        const float rx = rms_inv<EPL>(x, p.eps);
        float f[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) f[e] = x[e] * rx * gF[e];
        const bf16* wg = reinterpret_cast<const bf16*>(sm + L.g[l]);
        const bf16* wu = reinterpret_cast<const bf16*>(sm + L.u[l]);
#pragma unroll 1
        for (int rr = warp; rr < nf; rr += kW) {
          const float gv = dot_row<EPL>(wg + rr * H, f);
          const float uv = dot_row<EPL>(wu + rr * H, f);
          if (lane == 0) ms[rr] = gelu_tanh(gv) * uv;
        }
        __syncthreads();
        const bf16* wd = reinterpret_cast<const bf16*>(sm + L.dn[l]);
#pragma unroll 1
        for (int i = tid; i < H; i += kT) vs[i] = dot_col(wd + i * L.nfp, ms, nf);
      }
      float gPF[EPL];
      ldg_vec<EPL>(p.post_ffn_norm[l], gPF);
      ldg_vec<EPL>(l + 1 < nl ? p.attn_norm[l + 1] : p.out_norm, gA);
      float* dnr = all_reduce(p, sm, vs, arn++, p.mb + xo[ex_dn(l)], ep0 + ex_dn(l), rank, g, false, &ok);
      if (!ok) break;
      {
        float dn[EPL];
        lds_vec<EPL>(dnr, dn);
        const float rd = rms_inv<EPL>(dn, p.eps);
        const float lam = p.lambda[l];
#pragma unroll
        for (int e = 0; e < EPL; ++e) x[e] = (x[e] + dn[e] * rd * gPF[e]) * lam;
      }
    }
    if (!ok) break;

    // ---------------- HEAD: y = output_norm(x) (gains in gA); my rows of h' and the centroid logits
    need_group(nl + 1);
    if (!ok) break;
    float y[EPL];
    {
      const float r = rms_inv<EPL>(x, p.eps);
#pragma unroll
      for (int e = 0; e < EPL; ++e) y[e] = x[e] * r * gA[e];
    }
    {
      const bf16* wp = reinterpret_cast<const bf16*>(sm + L.post);
      const bf16* wc = reinterpret_cast<const bf16*>(sm + L.cent);
      unsigned long long* mc = p.mb + xo[ex_cent(nl)];
      const unsigned epc = ep0 + ex_cent(nl);
      // rows rr (centroid rows first, then post-projection rows), two per warp at a time so
      // that their reductions overlap
      auto row_ptr = [&](int rr) { return rr < ncr ? wc + rr * H : wp + (rr - ncr) * H; };
      auto row_out = [&](int rr, float v) {
        if (lane != 0) return;
        if (rr < ncr) {
          put(mc, cr.lo + rr, v, epc);
        } else {
          const int q = rr - ncr;
          hc[q] = v;
          if (p.out_hidden) p.out_hidden[static_cast<size_t>(s) * p.bb + hr.lo + q] = v;
        }
      };
#pragma unroll 1
      for (int rr = warp; rr < ncr + nhc; rr += 2 * kW) {
        const int r2 = rr + kW;
        const float v1 = dot_row<EPL>(row_ptr(rr), y);
        const float v2 = r2 < ncr + nhc ? dot_row<EPL>(row_ptr(r2), y) : 0.f;
        row_out(rr, v1);
        if (r2 < ncr + nhc) row_out(r2, v2);
      }
    }
    __syncthreads();
    if (s + 1 < p.n_draft) pre_h();  // the next step's h part, while the other CTAs catch up
    // ---------------- TOP-K over the gathered centroid logits, then my candidate rows
    if (!gather_lin(p, p.mb + xo[ex_cent(nl)], p.C, reinterpret_cast<unsigned*>(ub), ep0 + ex_cent(nl))) {
      ok = false;
      break;
    }
    topk_select(p, sm, ub, sel);
    {
      unsigned long long best = 0ull;
      const int lgv = p.lg_vsc;
      auto row_of = [&](int sl) -> long long {
        int ce = sel[sl >> lgv];
        ce = ce < 0 ? 0 : (ce >= p.C ? p.C - 1 : ce);
        return (static_cast<long long>(ce) << lgv) + (sl & ((1 << lgv) - 1));
      };
      if constexpr (EPL % 8 == 0) {
        // four rows per warp at a time: every row's vectors and id requested before any sum
        constexpr int NV = EPL / 8, RW = 4;
#pragma unroll 1
        for (int s0 = candr.lo + warp; s0 < candr.hi; s0 += RW * kW) {
          uint4 rv[RW][NV];
          int ids[RW];
#pragma unroll
          for (int r = 0; r < RW; ++r) {
            const int sl = s0 + r * kW;
            if (sl < candr.hi) {
              const long long rowi = row_of(sl);
              ids[r] = __ldg(p.ord + rowi);
              const uint4* rp = reinterpret_cast<const uint4*>(p.temb_ord + rowi * H + lane * EPL);
#pragma unroll
              for (int v = 0; v < NV; ++v) rv[r][v] = __ldg(rp + v);
            } else {
              ids[r] = 0;
#pragma unroll
              for (int v = 0; v < NV; ++v) rv[r][v] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
#pragma unroll
          for (int r = 0; r < RW; ++r) {
            float sum = 0.f;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
              float f[8];
              bf8(rv[r][v], f);
#pragma unroll
              for (int i = 0; i < 8; ++i) sum = fmaf(f[i], y[8 * v + i], sum);
            }
            sum = warp_sum(sum);
            const unsigned long long key = argmax_key(sum, ids[r]);
            if (s0 + r * kW < candr.hi) best = key > best ? key : best;
          }
        }
      } else {
#pragma unroll 1
        for (int sl = candr.lo + warp; sl < candr.hi; sl += kW) {
          const long long rowi = row_of(sl);
          const int id = __ldg(p.ord + rowi);
          const float v = dot_row<EPL>(p.temb_ord + rowi * H, y);
          const unsigned long long key = argmax_key(v, id);
          best = key > best ? key : best;
        }
      }
      if (lane == 0) wkeys[warp] = best;
      __syncthreads();
      if (warp == 0) {
        unsigned long long b = lane < kW ? wkeys[lane] : 0ull;
        b = warp_max_u64(b);
        const int id = key_id(b);
        if (lane == 0) {
          unsigned long long* mk = p.mb + xo[ex_key(nl)];
          put_u(mk, 2 * c, static_cast<unsigned>(b >> 32), ep0 + ex_key(nl));
          put_u(mk, 2 * c + 1, static_cast<unsigned>(b), ep0 + ex_key(nl));
        }
        // warm L2 with this candidate's embedding row: the next step's PRE reads it if it wins
        if (b != 0ull && id >= 0 && id < p.V && s + 1 < p.n_draft) {
#pragma unroll 1
          for (int off = lane * 128; off < p.bb * 2; off += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(p.tgt + static_cast<size_t>(id) * p.bb) + off));
        }
      }
    }
    if (!gather_lin(p, p.mb + xo[ex_key(nl)], 2 * p.N, reinterpret_cast<unsigned*>(ub), ep0 + ex_key(nl))) {
      ok = false;
      break;
    }
    {
      const unsigned* uk = reinterpret_cast<const unsigned*>(ub);
      unsigned long long b = 0ull;
#pragma unroll 1
      for (int a = lane; a < p.N; a += 32) {
        const unsigned long long kk = (static_cast<unsigned long long>(uk[2 * a]) << 32) | uk[2 * a + 1];
        b = kk > b ? kk : b;
      }
      b = warp_max_u64(b);
      int nt = key_id(b);
      if (nt < 0 || nt >= p.V) nt = 0;
      tok = nt;
      if (c == 0 && tid == 0) p.out_tokens[s] = nt;
    }
  }
  // ---- end: copies still in flight write shared memory; peers may still write into it
#pragma unroll 1
  for (int gi = 0; gi < nl + 2; ++gi)
    if (!(loaded >> gi & 1u)) mbar_wait(p, sa(&bars[gi]), 0u, false);
  if (kwaited < kph) mbar_wait(p, sa(&bars[kbar]), static_cast<unsigned>(kph - 1) & 1u, false);
  __syncthreads();
  cluster_sync_all();
}

// ------------------------------------------------------------------ weight images

// Copies one projection's share of every CTA into the per-CTA images. Row mode: dst [rows][K]
// holds rows split(R, N, c) of W [R][K]. Column mode: dst [R][pitch] holds columns
// col0 + split(Kpart, N, c) of W [R][Ktot]. Shares shorter than the section are zero-padded.
struct PackJob {
  const bf16* W;
  int R, Ktot, col0, Kpart, mode, rows_max, pitch;  // mode 0 rows, 1 columns
  long long sec_off;
};
__global__ void k_gr_pack(PackJob j, int N, long long img_bytes, unsigned char* dst) {
  const int c = blockIdx.x;
  bf16* out = reinterpret_cast<bf16*>(dst + static_cast<size_t>(c) * img_bytes + j.sec_off);
  if (j.mode == 0) {
    const Range r = split(j.R, N, c);
    const long long n = static_cast<long long>(j.rows_max) * j.Ktot;
    #pragma unroll 1
    for (long long i = threadIdx.x + static_cast<long long>(blockIdx.y) * blockDim.x; i < n;
         i += static_cast<long long>(blockDim.x) * gridDim.y) {
      const int rr = static_cast<int>(i / j.Ktot), k = static_cast<int>(i % j.Ktot);
      out[i] = r.lo + rr < r.hi ? j.W[static_cast<size_t>(r.lo + rr) * j.Ktot + k] : __float2bfloat16(0.f);
    }
  } else {
    const Range r = split(j.Kpart, N, c);
    const long long n = static_cast<long long>(j.R) * j.pitch;
    #pragma unroll 1
    for (long long i = threadIdx.x + static_cast<long long>(blockIdx.y) * blockDim.x; i < n;
         i += static_cast<long long>(blockDim.x) * gridDim.y) {
      const int row = static_cast<int>(i / j.pitch), k = static_cast<int>(i % j.pitch);
      out[i] = r.lo + k < r.hi ? j.W[static_cast<size_t>(row) * j.Ktot + j.col0 + r.lo + k] : __float2bfloat16(0.f);
    }
  }
}

}  // namespace gr

// ------------------------------------------------------------------ host side

namespace {

template <int EPL>
bool gr_attr(int smem) {
  if (cudaFuncSetAttribute(gr::k_block_gr<EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(gr::k_block_gr<EPL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}
template <int EPL>
int gr_clusters(int S, int smem) {
  if (!gr_attr<EPL>(smem)) return 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = S;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(S);
  cfg.blockDim = dim3(gr::kT);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<void*>(gr::k_block_gr<EPL>), &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}
int clusters_for(int H, int S, int smem) {
  switch (H) {
    case 64: return gr_clusters<2>(S, smem);
    case 128: return gr_clusters<4>(S, smem);
    case 256: return gr_clusters<8>(S, smem);
    case 512: return gr_clusters<16>(S, smem);
    default: return 0;
  }
}

// Attention CTAs, resident-key rows and the layout for a grid of N CTAs; false when the
// shape cannot run on it.
bool plan_for(gr::Params& p, int N, int S, int G, bool k_full_res, bool k_swa_res, bool k_both, int optin) {
  p.N = N;
  p.S = S;
  p.G = G;
  p.kboth = k_both ? 1 : 0;
  for (int t = 0; t < 2; ++t) {
    if (!p.has_type[t]) {
      p.A[t] = 0;
      p.kres[t] = 0;
      p.kslots[t] = 0;
      continue;
    }
    const int keys = t == 0 ? (p.kv_max[t] < p.W ? p.kv_max[t] : p.W) : p.kv_max[t];
    int A = gr::cdiv(keys, gr::kKeysPerCta);
    A = A < 1 ? 1 : (A > N ? N : A);
    p.A[t] = A;
    p.kslots[t] = gr::cdiv(keys, A);
    p.kres[t] = t == 0 ? (k_swa_res ? 1 : 0) : (k_full_res ? 1 : 0);
  }
  p.L = gr::make_layout(p);
  const gr::Layout& L = p.L;
  if (L.kc > 64 || L.total > optin) return false;
  #pragma unroll 1
  for (int l = 0; l < p.nl; ++l) {
    const int t = p.ltype[l], d = p.d[t];
    if (L.nq[l] > 48) return false;  // combine: o values in red[0, 48), denominators in red[48, 64)
    int ht = 0;
    for (int c = 0; c < N; ++c) {
      const gr::Range r = gr::split(p.nh * d, N, c);
      const int h = gr::heads_touched(r.lo, r.hi, d);
      ht = h > ht ? h : ht;
    }
    if (ht > 16 || ht * p.A[t] > gr::max_qd(p)) return false;  // combine weights live in the q buffer
  }
  return true;
}

}  // namespace

// Chooses the cluster size and grid (every co-resident cluster of the largest size whose
// plan fits, preferring attended keys resident in shared memory), fills the layout; returns
// the dynamic shared-memory bytes (0: shape not supported by this path).
int gr_plan(gr::Params& p, int optin) {
  const int H = p.H;
  if (H != 64 && H != 128 && H != 256 && H != 512) return 0;
  if (p.nl < 1 || p.nl > gr::kMaxL || p.nh < 1 || p.nh > gr::kMaxHeads || p.nkv < 1 || p.nh % p.nkv ||
      p.nh / p.nkv > gr::kMaxGroup)
    return 0;
  if (p.topk < 1 || p.topk > gr::kMaxTopK || p.C < p.topk || p.vsc < 1 || static_cast<long long>(p.C) * p.vsc != p.V)
    return 0;
  #pragma unroll 1
  for (int l = 0; l < p.nl; ++l) {
    const int d = p.d[p.ltype[l]];
    if (d < 8 || d % 8 || p.nh * d > 8192) return 0;
  }
  for (int t = 0; t < 2; ++t)
    if (p.has_type[t] && ((p.st[t] * 2) % 16 || (p.nkv * p.d[t] * 2) % 16)) return 0;
  if (p.bb % 8) return 0;
  // index arithmetic by shifts: head dims, vsc and every slice width are powers of two
  auto lg2 = [](int v) {
    int l = 0;
    while ((1 << l) < v) ++l;
    return (1 << l) == v ? l : -1;
  };
  for (int t = 0; t < 2; ++t) {
    p.lg_d[t] = 0;
    if (!p.has_type[t]) continue;
    p.lg_d[t] = lg2(p.d[t]);
    if (p.lg_d[t] < 3) return 0;
  }
  p.lg_vsc = lg2(p.vsc);
  if (p.lg_vsc < 0) return 0;
  if (p.d[0] / 2 + p.d[1] / 2 > 2 * gr::kT) return 0;  // the prologue forms two RoPE pairs per thread
  // top-k tiling: C = 256 * per with per <= 8, and k groups of a power-of-two <= 32 threads
  p.tk_lg_per = p.tk_lg_tpg = -1;
  if (p.C % gr::kT == 0 && p.C % p.topk == 0) {
    const int per = p.C / gr::kT, tpg = (p.C / p.topk) / per;
    if (per <= 8 && lg2(per) >= 0 && (p.C / p.topk) % per == 0 && tpg <= 32 && lg2(tpg) >= 0) {
      p.tk_lg_per = lg2(per);
      p.tk_lg_tpg = lg2(tpg);
    }
  }
  // attended keys resident in shared memory: both types for the whole launch, else both
  // taking turns in one region, else the sliding type only, else none
  const bool res_opts[4][3] = {{true, true, true}, {true, true, false}, {false, true, false}, {false, false, false}};
  #pragma unroll 1
  for (const auto& ro : res_opts) {
    #pragma unroll 1
    for (int S : {16, 8, 4}) {
      if (H / S < 2 || (H / S) % 2) continue;
      gr::Params q = p;
      q.lg_hs = 0;
      while ((1 << q.lg_hs) < H / S) ++q.lg_hs;
      const int G = clusters_for(H, S, optin);
      if (G < 1) continue;
      if (!plan_for(q, G * S, S, G, ro[0], ro[1], ro[2], optin)) continue;
      // the grid must be co-resident at the planned size
      const int G2 = clusters_for(H, S, q.L.total);
      if (G2 < G) continue;
      p = q;
      return p.L.total;
    }
  }
  return 0;
}

long long gr_image_total(const gr::Params& p) { return static_cast<long long>(p.N) * p.L.img_bytes; }

// Packs every CTA's weight image (layout of gr::Layout) from the caller's matrices.
int gr_pack(const gr::Params& p, const void* pre, const void* post, const void* cent, const void* const* q,
            const void* const* o, const void* const* gate, const void* const* up, const void* const* down,
            unsigned char* dst, cudaStream_t st) {
  using gr::PackJob;
  typedef const __nv_bfloat16* cb;
  const gr::Layout& L = p.L;
  const int H = p.H;
  auto launch = [&](PackJob j) {
    gr::k_gr_pack<<<dim3(p.N, 8), 256, 0, st>>>(j, p.N, L.img_bytes, dst);
  };
  launch(PackJob{static_cast<cb>(pre), H, 2 * p.bb, 0, p.bb, 1, 0, L.kcp, L.pre});
  launch(PackJob{static_cast<cb>(pre), H, 2 * p.bb, p.bb, p.bb, 1, 0, L.kcp, L.pre + 2LL * H * L.kcp});
  launch(PackJob{static_cast<cb>(post), p.bb, H, 0, 0, 0, L.kc, 0, L.post});
  #pragma unroll 1
  for (int l = 0; l < p.nl; ++l) {
    const int QD = p.nh * p.d[p.ltype[l]];
    launch(PackJob{static_cast<cb>(q[l]), QD, H, 0, 0, 0, L.nq[l], 0, L.q[l]});
    launch(PackJob{static_cast<cb>(o[l]), H, QD, 0, QD, 1, 0, L.nqp[l], L.o[l]});
    launch(PackJob{static_cast<cb>(gate[l]), p.F, H, 0, 0, 0, L.nf, 0, L.g[l]});
    launch(PackJob{static_cast<cb>(up[l]), p.F, H, 0, 0, 0, L.nf, 0, L.u[l]});
    launch(PackJob{static_cast<cb>(down[l]), H, p.F, 0, p.F, 1, 0, L.nfp, L.dn[l]});
  }
  launch(PackJob{static_cast<cb>(cent), p.C, H, 0, 0, 0, L.ncent, 0, L.cent});
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("packing the grid path's weight images: %s", cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

// Mailbox offsets of every exchange (both step parities); returns the total words.
long long gr_mailboxes(gr::Params& p) {
  long long off = 0;
  const int n = gr::ex_count(p.nl);
  for (int par = 0; par < 2; ++par)
    #pragma unroll 1
    for (int x = 0; x < gr::kMaxEx; ++x) {
      p.ex_off[par][x] = off;
      if (x < n) off += (gr::ex_words(p, x) + 31) & ~31LL;
    }
  return off;
}

int run_gr(const gr::Params& p, cudaStream_t st) {
  const int smem = p.L.total;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = p.S;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(p.N);
  cfg.blockDim = dim3(gr::kT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaErrorInvalidValue;
  switch (p.H) {
    case 64: e = gr_attr<2>(smem) ? cudaLaunchKernelEx(&cfg, gr::k_block_gr<2>, p) : cudaErrorInvalidValue; break;
    case 128: e = gr_attr<4>(smem) ? cudaLaunchKernelEx(&cfg, gr::k_block_gr<4>, p) : cudaErrorInvalidValue; break;
    case 256: e = gr_attr<8>(smem) ? cudaLaunchKernelEx(&cfg, gr::k_block_gr<8>, p) : cudaErrorInvalidValue; break;
    case 512: e = gr_attr<16>(smem) ? cudaLaunchKernelEx(&cfg, gr::k_block_gr<16>, p) : cudaErrorInvalidValue; break;
    default: break;
  }
  if (e != cudaSuccess) {
    set_error("grid draft-block launch (%d CTAs in clusters of %d, %d B shared memory): %s", p.N, p.S, smem,
              cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

// ------------------------------------------------------------------ token_embd reordering

namespace {
// dst[j] = src[ord[j]] for the V rows of vec 16-byte vectors each.
__global__ void k_reorder_rows(const uint4* __restrict__ src, const int* __restrict__ ord, uint4* __restrict__ dst,
                               int V, int vec) {
  const long long total = static_cast<long long>(V) * vec;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = i / vec, c = i % vec;
    const int s = ord[row];
    dst[row * vec + c] = src[static_cast<size_t>(s) * vec + c];
  }
}
}  // namespace

int reorder_rows(const void* src, const int* ord, void* dst, int V, int row_bytes, cudaStream_t st) {
  k_reorder_rows<<<1024, 256, 0, st>>>(static_cast<const uint4*>(src), ord, static_cast<uint4*>(dst), V,
                                       row_bytes / 16);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("reordering token_embd: %s", cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

}  // namespace mtp
