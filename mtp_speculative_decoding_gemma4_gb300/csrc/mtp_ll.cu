// Latency-path draft block (B = 1): see mtp_ll.cuh for the data flow.
//
// Per-phase cost is dominated by latency (L2 round trips of mailbox polls, shared-memory
// load chains, instruction fetch), so: 512 threads per CTA, every poll issues all of a
// thread's loads before waiting on any, small gain vectors are fetched into registers
// before the poll that precedes their use, and the shared helpers are not inlined so that
// their code stays in the instruction cache across phases.
#include <cmath>
#include <cstring>

#include "mtp_launch.h"
#include "mtp_ll.cuh"

namespace mtp {
namespace ll {

// ------------------------------------------------------------------ primitives

__device__ __forceinline__ unsigned smem_addr(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mb_put(unsigned long long* mb, int i, float v, unsigned epoch) {
  const unsigned long long w = (static_cast<unsigned long long>(epoch) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(mb + i), "l"(w) : "memory");
}
__device__ __forceinline__ void mb_put_u(unsigned long long* mb, int i, unsigned v, unsigned epoch) {
  const unsigned long long w = (static_cast<unsigned long long>(epoch) << 32) | v;
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(mb + i), "l"(w) : "memory");
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

__device__ __forceinline__ float ll_block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kW; ++i) s += red[i];
  return s;
}

constexpr int kMaxW = 8;  // mailbox words in flight per thread per pass

// Records a timeout (status word + abort word) or notices a raised abort word; true when the
// caller must give up.
__device__ __forceinline__ bool poll_expired(const Params& p, long long t0, unsigned n) {
  if ((n & 63u) != 0u) return false;
  if (ld_rlx32(p.abort_flag)) return true;
  if (clock64() - t0 > p.spin_limit) {
    atomicExch(p.status, static_cast<int>(MTP_ERR_TIMEOUT));
    atomicExch(p.abort_flag, 1u);
    return true;
  }
  return false;
}

// Mailbox words [0, count) -> dst (payload bits). Each thread issues the loads of all its
// words before waiting and re-polls only the missing ones. Bounded; false when the block
// must stop. All threads call it.
__device__ __noinline__ bool gather_words(const Params& p, const unsigned long long* mb, int count, unsigned* dst,
                                          unsigned epoch) {
  int bad = 0;
  for (int base = 0; base < count && !bad; base += kMaxW * kT) {
    unsigned long long w[kMaxW];
#pragma unroll
    for (int j = 0; j < kMaxW; ++j) {
      const int k = base + j * kT + static_cast<int>(threadIdx.x);
      w[j] = k < count ? ld_rlx64(mb + k) : (static_cast<unsigned long long>(epoch) << 32);
    }
    const long long t0 = clock64();
    for (unsigned n = 1;; ++n) {
      bool all = true;
#pragma unroll
      for (int j = 0; j < kMaxW; ++j) {
        if (static_cast<unsigned>(w[j] >> 32) != epoch) {
          all = false;
          w[j] = ld_rlx64(mb + base + j * kT + static_cast<int>(threadIdx.x));
        }
      }
      if (all) break;
      if (poll_expired(p, t0, n)) {
        bad = 1;
        break;
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxW; ++j) {
      const int k = base + j * kT + static_cast<int>(threadIdx.x);
      if (k < count) dst[k] = static_cast<unsigned>(w[j]);
    }
  }
  return !__syncthreads_or(bad);
}

__device__ __forceinline__ bool gather(const Params& p, const unsigned long long* mb, int count, float* dst,
                                       unsigned epoch) {
  return gather_words(p, mb, count, reinterpret_cast<unsigned*>(dst), epoch);
}

// Attention-combine gather: for every source CTA, (m, l) of heads h0..h0+nhr-1 and the
// partial sums of flattened dims [f0, f0+nd), into buf[src][2*nhr + nd].
__device__ __noinline__ bool gather_partials(const Params& p, int d, int h0, int nhr, int f0, int nd, float* buf,
                                             unsigned epoch) {
  const int per = 2 * nhr + nd, count = p.N * per, pstride = p.nh * (d + 2);
  unsigned* dst = reinterpret_cast<unsigned*>(buf);
  int bad = 0;
  for (int base = 0; base < count && !bad; base += kMaxW * kT) {
    const unsigned long long* a[kMaxW];
    unsigned long long w[kMaxW];
#pragma unroll
    for (int j = 0; j < kMaxW; ++j) {
      const int k = base + j * kT + static_cast<int>(threadIdx.x);
      const int kk = k < count ? k : 0;
      const int src = kk / per, jj = kk % per;
      const unsigned long long* pb = p.mb_part + static_cast<size_t>(src) * pstride;
      if (jj < 2 * nhr) {
        a[j] = pb + (h0 + jj / 2) * (d + 2) + d + (jj & 1);
      } else {
        const int f = f0 + (jj - 2 * nhr);
        a[j] = pb + (f / d) * (d + 2) + f % d;
      }
      w[j] = k < count ? ld_rlx64(a[j]) : (static_cast<unsigned long long>(epoch) << 32);
    }
    const long long t0 = clock64();
    for (unsigned n = 1;; ++n) {
      bool all = true;
#pragma unroll
      for (int j = 0; j < kMaxW; ++j) {
        if (static_cast<unsigned>(w[j] >> 32) != epoch) {
          all = false;
          w[j] = ld_rlx64(a[j]);
        }
      }
      if (all) break;
      if (poll_expired(p, t0, n)) {
        bad = 1;
        break;
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxW; ++j) {
      const int k = base + j * kT + static_cast<int>(threadIdx.x);
      if (k < count) dst[k] = static_cast<unsigned>(w[j]);
    }
  }
  return !__syncthreads_or(bad);
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, unsigned long long* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ bool mbar_test(unsigned long long* bar) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar))
      : "memory");
  return ok != 0;
}
// Wait until the section's bulk copies have landed (first step only; later waits return at once).
__device__ __noinline__ bool wait_section_slow(const Params& p, unsigned long long* bar) {
  int bad = 0;
  if (!mbar_test(bar)) {
    const long long t0 = clock64();
    while (!mbar_test(bar)) {
      if (clock64() - t0 > p.spin_limit) {
        atomicExch(p.status, static_cast<int>(MTP_ERR_TIMEOUT));
        atomicExch(p.abort_flag, 1u);
        bad = 1;
        break;
      }
    }
  }
  return !__syncthreads_or(bad);
}

// out[r] = W[r] . x for nrows rows of a resident bf16 matrix with K columns; work units are
// (row, 256-column segment) pairs spread over the warps.
__device__ __noinline__ void smem_gemv(const bf16* W, int nrows, int K, const float* x, float* red, float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int segs = (K + 255) / 256;
  const int units = nrows * segs;
  for (int u = warp; u < units; u += kW) {
    const int r = u / segs, sg = u % segs;
    const int k = sg * 256 + lane * 8;
    float s = 0.f;
    if (k < K) {
      float w[8];
      load_vec(W + static_cast<size_t>(r) * K + k, w);
      const float4 a = *reinterpret_cast<const float4*>(x + k);
      const float4 b = *reinterpret_cast<const float4*>(x + k + 4);
      s = (w[0] * a.x + w[1] * a.y) + (w[2] * a.z + w[3] * a.w) + ((w[4] * b.x + w[5] * b.y) + (w[6] * b.z + w[7] * b.w));
    }
    s = warp_sum(s);
    if (lane == 0) red[u] = s;
  }
  __syncthreads();
  for (int r = threadIdx.x; r < nrows; r += kT) {
    float s = 0.f;
    for (int sg = 0; sg < segs; ++sg) s += red[r * segs + sg];
    out[r] = s;
  }
  __syncthreads();
}

// 1/sqrt(mean(v^2) + eps) of v[0, n) (all threads get it).
__device__ __noinline__ float rms_inv(const float* v, int n, float eps, float* red) {
  float s = 0.f;
  for (int i = threadIdx.x; i < n; i += kT) s += v[i] * v[i];
  return rsqrtf(ll_block_sum(s, red) / n + eps);
}

struct Smem {
  char* base;
  Layout L;
  __device__ const bf16* sec(int s) const { return reinterpret_cast<const bf16*>(base + L.sec_off[s]); }
  __device__ float* r1() const { return reinterpret_cast<float*>(base + L.r1_off); }
  __device__ float* r2() const { return reinterpret_cast<float*>(base + L.r2_off); }
  __device__ float* x() const { return reinterpret_cast<float*>(base + L.x_off); }
  __device__ float* t() const { return reinterpret_cast<float*>(base + L.t_off); }
  __device__ float* a() const { return reinterpret_cast<float*>(base + L.a_off); }
  __device__ float* sc() const { return reinterpret_cast<float*>(base + L.sc_off); }
  __device__ float* red() const { return reinterpret_cast<float*>(base + L.red_off); }
  __device__ int* hist() const { return reinterpret_cast<int*>(base + L.hist_off); }
  __device__ int* sel() const { return reinterpret_cast<int*>(base + L.sel_off); }
  __device__ int* ord() const { return reinterpret_cast<int*>(base + L.ord_off); }
  __device__ float* gq() const { return reinterpret_cast<float*>(base + L.g_off); }
  __device__ unsigned long long* bar(int s) const {
    return reinterpret_cast<unsigned long long*>(base + L.mbar_off) + s;
  }
  __device__ float2* cs() const { return reinterpret_cast<float2*>(base + L.cs_off); }
};

__device__ __forceinline__ unsigned ep(const Params& p, int step, int idx) {
  return p.epoch_base + static_cast<unsigned>(step) * kExPerStep + static_cast<unsigned>(idx);
}

// Gain element tid of a vector of length n (0 beyond), fetched early to hide its latency.
__device__ __forceinline__ float gain_reg(const float* g, int n) {
  return static_cast<int>(threadIdx.x) < n ? __ldg(g + threadIdx.x) : 0.f;
}

// Sections are waited for during the block's first step only; afterwards every section has
// landed and the wait (with its CTA barrier) is skipped.
__device__ __forceinline__ bool wait_section(const Params& p, unsigned long long* bar, bool loaded) {
  return loaded ? true : wait_section_slow(p, bar);
}

// ------------------------------------------------------------------ top-k by radix select

// Indices of the top_k largest of v[0, n) (ties: lower index), ascending index order, into
// sel[0, k). Every CTA runs this on identical data and gets identical results.
// Round 1 histograms the top 8 bits of every key (warp-aggregated shared atomics) and finds
// the bin that holds the k-th largest; keys above it are selected, keys inside it ("pending",
// typically a few hundred) are compacted and finished by one warp with three more 8-bit
// rounds, so only round 1 needs the whole block.
__device__ __noinline__ void topk_select(const float* v, int n, int k, int* hist, int* sel, float* red,
                                         unsigned* pend_key) {
  __shared__ unsigned s_bin;
  __shared__ int s_need, s_gt, s_np;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 256; i += kT) hist[i] = 0;
  __syncthreads();
  for (int base = 0; base < n; base += kT) {
    const int i = base + static_cast<int>(threadIdx.x);
    const unsigned bin = i < n ? (ord_f32(v[i]) >> 24) : 256u;
    const unsigned peers = __match_any_sync(0xffffffffu, bin);
    if (i < n && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
  }
  __syncthreads();
  if (warp == 0) {
    int cnt[8], tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      cnt[j] = hist[255 - (lane * 8 + j)];
      tot += cnt[j];
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int excl = incl - tot;
    if (excl < k && incl >= k) {
      int run = excl;
      for (int j = 0; j < 8; ++j) {
        if (run + cnt[j] >= k) {
          s_bin = 255u - static_cast<unsigned>(lane * 8 + j);
          s_gt = run;            // keys in higher bins: all selected
          s_need = k - run;      // still to take from the pending bin
          break;
        }
        run += cnt[j];
      }
    }
  }
  if (threadIdx.x == 0) s_np = 0;
  __syncthreads();
  // compact the pending bin (order does not matter; ties are resolved by index below)
  const unsigned b1 = s_bin;
  for (int base = 0; base < n; base += kT) {
    const int i = base + static_cast<int>(threadIdx.x);
    const unsigned key = i < n ? ord_f32(v[i]) : 0u;
    const bool pend = i < n && (key >> 24) == b1;
    const unsigned pm = __ballot_sync(0xffffffffu, pend);
    int slot = 0;
    if (lane == 0 && pm) slot = atomicAdd(&s_np, __popc(pm));
    slot = __shfl_sync(0xffffffffu, slot, 0);
    if (pend) pend_key[slot + __popc(pm & ((1u << lane) - 1u))] = key;  // at most n keys
  }
  __syncthreads();
  // one warp: exact threshold key T among the pending keys, and how many keys == T to take
  __shared__ unsigned s_T;
  __shared__ int s_take_eq;
  const int np = s_np;
  if (warp == 0) {
    unsigned prefix = b1 << 24, mask = 0xff000000u;
    int need = s_need;
    for (int byte = 2; byte >= 0; --byte) {
      const int shift = 8 * byte;
      for (int i = lane; i < 256; i += 32) hist[i] = 0;
      __syncwarp();
      for (int i = lane; i < np; i += 32) {
        const unsigned key = pend_key[i];
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncwarp();
      int cnt[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = hist[255 - (lane * 8 + j)];
        tot += cnt[j];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - tot;
      unsigned bin = 0;
      int newneed = 0, found = 0;
      if (excl < need && incl >= need) {
        int run = excl;
        for (int j = 0; j < 8; ++j) {
          if (run + cnt[j] >= need) {
            bin = 255u - static_cast<unsigned>(lane * 8 + j);
            newneed = need - run;
            found = 1;
            break;
          }
          run += cnt[j];
        }
      }
      const unsigned fm = __ballot_sync(0xffffffffu, found);
      const int src = __ffs(fm) - 1;
      bin = __shfl_sync(0xffffffffu, bin, src);
      need = __shfl_sync(0xffffffffu, newneed, src);
      prefix |= bin << shift;
      mask |= 255u << shift;
      __syncwarp();
    }
    if (lane == 0) {
      s_T = prefix;
      s_take_eq = need;
    }
  }
  __syncthreads();
  const unsigned T = s_T;
  const int take_eq = s_take_eq;
  // selection in ascending index order: key > T, or key == T among the take_eq lowest indices
  const int per_warp = (n + kW - 1) / kW;
  int* wcnt = reinterpret_cast<int*>(red);  // [kW] equal counts, [kW, 2kW) selected counts
  const int i0 = warp * per_warp, i1 = min(n, i0 + per_warp);
  int eq_w = 0, sel_w = 0;
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    const unsigned key = i < i1 ? ord_f32(v[i]) : 0u;
    const bool eq = i < i1 && key == T;
    eq_w += __popc(__ballot_sync(0xffffffffu, eq));
  }
  if (lane == 0) wcnt[warp] = eq_w;
  __syncthreads();
  int eq_before = 0;
  for (int w = 0; w < warp; ++w) eq_before += wcnt[w];
  int eq_seen = eq_before;
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    const unsigned key = i < i1 ? ord_f32(v[i]) : 0u;
    const bool eq = i < i1 && key == T;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const int eq_rank = eq_seen + __popc(eqm & ((1u << lane) - 1u));
    const bool take = i < i1 && (key > T || (eq && eq_rank < take_eq));
    sel_w += __popc(__ballot_sync(0xffffffffu, take));
    eq_seen += __popc(eqm);
  }
  if (lane == 0) wcnt[kW + warp] = sel_w;
  __syncthreads();
  int pos = 0;
  for (int w = 0; w < warp; ++w) pos += wcnt[kW + w];
  eq_seen = eq_before;
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    const unsigned key = i < i1 ? ord_f32(v[i]) : 0u;
    const bool eq = i < i1 && key == T;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const int eq_rank = eq_seen + __popc(eqm & ((1u << lane) - 1u));
    const bool take = i < i1 && (key > T || (eq && eq_rank < take_eq));
    const unsigned tm = __ballot_sync(0xffffffffu, take);
    if (take) sel[pos + __popc(tm & ((1u << lane) - 1u))] = i;
    pos += __popc(tm);
    eq_seen += __popc(eqm);
  }
  __syncthreads();
}

// Largest (value, id) key published by the GATHER phase of `step` (all threads get it).
__device__ __noinline__ bool best_token(const Params& p, const Smem& S, int step, int& tok) {
  unsigned* kw = reinterpret_cast<unsigned*>(S.r2());
  if (!gather_words(p, p.mb_key, 2 * p.N, kw, ep(p, step, 3 + 6 * p.nl))) return false;
  unsigned long long best = 0ull;
  for (int i = threadIdx.x; i < p.N; i += kT) {
    const unsigned long long k = (static_cast<unsigned long long>(kw[2 * i]) << 32) | (0xffffffffu - kw[2 * i + 1]);
    best = k > best ? k : best;
  }
  best = warp_max_u64(best);
  unsigned long long* kb = reinterpret_cast<unsigned long long*>(S.red());
  if ((threadIdx.x & 31) == 0) kb[threadIdx.x >> 5] = best;
  __syncthreads();
  unsigned long long m = 0ull;
  for (int w = 0; w < kW; ++w) m = kb[w] > m ? kb[w] : m;
  tok = key_id(m);
  __syncthreads();
  return true;
}

// ------------------------------------------------------------------ the kernel

__global__ void __launch_bounds__(kT, 1) k_block_ll(Params p) {
  extern __shared__ __align__(128) char smem_raw[];
  Smem S{smem_raw, make_layout(p)};
  const Layout& L = S.L;
  const int c = blockIdx.x, N = p.N;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- resident sections: bulk copies, one mbarrier per section
  const int Lf = p.has_type[1] ? min(max(p.ctx_len[1][0], 0), p.kv_max[1]) : 0;
  const int Ls = p.has_type[0] ? min(max(p.ctx_len[0][0], 0), p.kv_max[0]) : 0;
  const int ws_lo = max(0, Ls - p.W);
  const Range kr_f = split(Lf, N, c);
  const Range kr_s = split(Ls - ws_lo, N, c);
  if (tid == 0) {
    for (int s = 0; s < S_COUNT; ++s) mbar_init(S.bar(s));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid == 0) {
    auto rows = [&](int s, const bf16* W, int R, int K) {
      const Range r = split(R, N, c);
      const unsigned bytes = static_cast<unsigned>((r.hi - r.lo) * K * 2);
      mbar_expect_tx(S.bar(s), bytes);
      char* dst = S.base + L.sec_off[s];
      const char* src = reinterpret_cast<const char*>(W + static_cast<size_t>(r.lo) * K);
      for (unsigned o = 0; o < bytes; o += 32768u) {
        const unsigned n = bytes - o < 32768u ? bytes - o : 32768u;
        bulk_g2s(dst + o, src + o, n, S.bar(s));
      }
    };
    rows(S_PRE, p.pre, p.H, 2 * p.bb);
    for (int l = 0; l < p.nl; ++l) {
      const int d = p.d[p.ltype[l]];
      rows(sec_q(l), p.q[l], p.nh * d, p.H);
      rows(sec_o(l), p.o[l], p.H, p.nh * d);
      rows(sec_g(l), p.gate[l], p.F, p.H);
      rows(sec_u(l), p.up[l], p.F, p.H);
      rows(sec_d(l), p.down[l], p.H, p.F);
    }
    rows(S_POST, p.post, p.bb, p.H);
    rows(S_CENT, p.cent, p.C, p.H);
    for (int t = 1; t >= 0; --t) {  // shared K slices (one copy per key: rows may be strided)
      const int s = t ? S_KF : S_KS;
      const Range r = t ? kr_f : kr_s;
      const int first = t ? r.lo : ws_lo + r.lo;
      const unsigned row_bytes = static_cast<unsigned>(p.nkv * p.d[t] * 2);
      const int nk = p.has_type[t] ? r.hi - r.lo : 0;
      mbar_expect_tx(S.bar(s), row_bytes * nk);
      for (int j = 0; j < nk; ++j)
        bulk_g2s(S.base + L.sec_off[s] + j * row_bytes, p.k[t] + static_cast<size_t>(first + j) * p.st[t], row_bytes,
                 S.bar(s));
    }
  }
  // token_ordering columns of this CTA's offsets: ord_s[(o - lo) * C + j] = ord[j * vsc + o]
  const Range offs = split(p.vsc, N, c);
  for (int idx = tid; idx < (offs.hi - offs.lo) * p.C; idx += kT) {
    const int oo = idx / p.C, j = idx % p.C;
    S.ord()[idx] = __ldg(p.ord + static_cast<size_t>(j) * p.vsc + offs.lo + oo);
  }
  // RoPE (cos, sin) at the constant position: the angle pos * theta^(-2i/d) in fp64, reduced
  // mod 2 pi in fp64, then single-precision sin / cos of the reduced angle
  for (int t = 0; t < 2; ++t) {
    const int d = p.has_type[t] ? p.d[t] : 0;
    const double theta = p.theta[t];
    for (int i = tid; i < d / 2; i += kT) {
      float2 v = make_float2(1.f, 0.f);
      if (theta != 0.0) {
        const double two_pi = 6.283185307179586476925286766559;
        double ang = static_cast<double>(p.pos[0]) * exp2(-2.0 * i / d * log2(theta));
        ang -= two_pi * floor(ang / two_pi);
        float sv, cv;
        sincosf(static_cast<float>(ang), &sv, &cv);
        v = make_float2(cv, sv);
      }
      S.cs()[t * L.cs_half + i] = v;
    }
  }
  __syncthreads();

  float* x = S.x();
  float* t = S.t();
  float* a = S.a();
  float* red = S.red();
  const int H = p.H;

  for (int step = 0; step < p.n_draft; ++step) {
    // ================= PRE
    {
      float* u = S.r1();
      int tok;
      if (step == 0) {
        tok = p.tok_in[0];
      } else {
        if (!best_token(p, S, step - 1, tok)) return;
        if (c == 0 && tid == 0) p.out_tokens[step - 1] = tok;
      }
      if (tok < 0 || tok >= p.V) {
        if (c == 0 && tid == 0) atomicExch(p.status, static_cast<int>(MTP_ERR_INVALID_ARG));
        tok = 0;
      }
      const bf16* er = p.tgt + static_cast<size_t>(tok) * p.bb;
      for (int i = tid * 8; i < p.bb; i += kT * 8) load_vec(er + i, u + p.bb + i);
      if (step == 0) {
        for (int i = tid * 8; i < p.bb; i += kT * 8) load_vec(p.hidden_in + i, u + i);
        __syncthreads();
      } else if (!gather(p, p.mb_h, p.bb, u, ep(p, step - 1, 1 + 6 * p.nl))) {
        return;
      }
      if (!wait_section(p, S.bar(S_PRE), step > 0)) return;
      const Range r = split(H, N, c);
      smem_gemv(S.sec(S_PRE), r.hi - r.lo, 2 * p.bb, u, red, t);
      for (int i = tid; i < r.hi - r.lo; i += kT) mb_put(p.mb_x0, r.lo + i, t[i], ep(p, step, 0));
    }
    // ================= blocks
    for (int l = 0; l < p.nl; ++l) {
      const int lt = p.ltype[l];
      const int d = p.d[lt];
      const int QD = p.nh * d;
      const int e0 = 1 + 6 * l;
      // ---- Q
      {
        const float g_in = gain_reg(p.attn_norm[l], H);
        if (l == 0) {
          if (!gather(p, p.mb_x0, H, x, ep(p, step, 0))) return;
        } else {
          const float g_pf = gain_reg(p.post_ffn_norm[l - 1], H);
          if (!gather(p, p.mb_dn, H, t, ep(p, step, e0 - 1))) return;
          const float rf = rms_inv(t, H, p.eps, red);
          if (tid < H) x[tid] = p.lambda[l - 1] * (x[tid] + t[tid] * rf * g_pf);
          __syncthreads();
        }
        const float rf = rms_inv(x, H, p.eps, red);
        if (tid < H) a[tid] = x[tid] * rf * g_in;
        __syncthreads();
        if (!wait_section(p, S.bar(sec_q(l)), step > 0)) return;
        const Range r = split(QD, N, c);
        smem_gemv(S.sec(sec_q(l)), r.hi - r.lo, H, a, red, t);
        for (int i = tid; i < r.hi - r.lo; i += kT) mb_put(p.mb_q, r.lo + i, t[i], ep(p, step, e0));
      }
      // ---- ATT
      float* q = S.r2();
      {
        float* gq = S.gq();
        const float gq0 = gain_reg(p.q_norm[l], d);
        const float gq1 = tid + kT < d ? __ldg(p.q_norm[l] + tid + kT) : 0.f;
        if (!gather(p, p.mb_q, QD, q, ep(p, step, e0))) return;
        if (tid < d) gq[tid] = gq0;
        if (tid + kT < d) gq[tid + kT] = gq1;
        if (warp < p.nh) {  // q_norm factor of head `warp`
          float s = 0.f;
          for (int i = lane * 4; i < d; i += 128) {
            const float4 v = *reinterpret_cast<const float4*>(q + warp * d + i);
            s += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
          }
          s = warp_sum(s);
          if (lane == 0) red[64 + warp] = rsqrtf(s / d + p.eps);
        }
        __syncthreads();
        const float2* cs = S.cs() + lt * L.cs_half;
        const int half = d / 2;
        for (int idx = tid; idx < p.nh * half; idx += kT) {
          const int h = idx / half, i = idx % half;
          const float rf = red[64 + h];
          const float av = q[h * d + i] * rf * gq[i];
          const float bv = q[h * d + i + half] * rf * gq[i + half];
          q[h * d + i] = av * cs[i].x - bv * cs[i].y;
          q[h * d + i + half] = bv * cs[i].x + av * cs[i].y;
        }
        __syncthreads();
      }
      if (!wait_section(p, S.bar(lt ? S_KF : S_KS), step > 0)) return;
      {
        const Range kr = lt ? kr_f : kr_s;
        const int nk = p.has_type[lt] ? kr.hi - kr.lo : 0;
        const bf16* K = S.sec(lt ? S_KF : S_KS);
        const int row = p.nkv * d;
        const int hpg = p.nh / p.nkv;
        float* sc = S.sc();
        const float scale = p.scale[lt];
        // scores: one (key, head) dot per warp iteration, 8 dims per lane per pass
        for (int u = warp; u < nk * p.nh; u += kW) {
          const int j = u / p.nh, h = u % p.nh;
          const bf16* kj = K + static_cast<size_t>(j) * row + (h / hpg) * d;
          const float* qh = q + h * d;
          float s0 = 0.f, s1 = 0.f;
          for (int i = lane * 8; i < d; i += 256) {
            float kv[8];
            load_vec(kj + i, kv);
            const float4 qa = *reinterpret_cast<const float4*>(qh + i);
            const float4 qb = *reinterpret_cast<const float4*>(qh + i + 4);
            s0 += qa.x * kv[0] + qa.y * kv[1] + qa.z * kv[2] + qa.w * kv[3];
            s1 += qb.x * kv[4] + qb.y * kv[5] + qb.z * kv[6] + qb.w * kv[7];
          }
          const float s = warp_sum(s0 + s1);
          if (lane == 0) sc[j * p.nh + h] = s * scale;
        }
        __syncthreads();
        if (warp < p.nh) {  // per-head max and exp-sum
          float m = -INFINITY;
          for (int j = lane; j < nk; j += 32) m = fmaxf(m, sc[j * p.nh + warp]);
          m = warp_max(m);
          float ls = 0.f;
          for (int j = lane; j < nk; j += 32) {
            const float e = expf(sc[j * p.nh + warp] - m);
            sc[j * p.nh + warp] = e;
            ls += e;
          }
          ls = warp_sum(ls);
          if (lane == 0) {
            red[80 + warp] = m;
            red[96 + warp] = ls;
          }
        }
        __syncthreads();
        // weighted key sums: 4 consecutive dims of one head per thread
        unsigned long long* part = p.mb_part + static_cast<size_t>(c) * p.nh * (d + 2);
        const unsigned epart = ep(p, step, e0 + 1);
        for (int uu = tid; uu < p.nh * d / 4; uu += kT) {
          const int h = (uu * 4) / d, i = (uu * 4) % d;
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
          const bf16* kb = K + (h / hpg) * d + i;
          for (int j = 0; j < nk; ++j) {
            const uint2 raw = *reinterpret_cast<const uint2*>(kb + static_cast<size_t>(j) * row);
            const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
            const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
            const float w = sc[j * p.nh + h];
            a0 = fmaf(w, k01.x, a0);
            a1 = fmaf(w, k01.y, a1);
            a2 = fmaf(w, k23.x, a2);
            a3 = fmaf(w, k23.y, a3);
          }
          mb_put(part, h * (d + 2) + i, a0, epart);
          mb_put(part, h * (d + 2) + i + 1, a1, epart);
          mb_put(part, h * (d + 2) + i + 2, a2, epart);
          mb_put(part, h * (d + 2) + i + 3, a3, epart);
        }
        for (int h = tid; h < p.nh; h += kT) {
          mb_put(part, h * (d + 2) + d, red[80 + h], epart);
          mb_put(part, h * (d + 2) + d + 1, red[96 + h], epart);
        }
        __syncthreads();
      }
      // ---- CMB: this CTA's dims of o from every CTA's partial
      {
        const Range r = split(QD, N, c);
        const int nd = r.hi - r.lo;
        const int h0 = nd > 0 ? r.lo / d : 0;
        const int nhr = nd > 0 ? (r.hi - 1) / d - h0 + 1 : 0;
        const int per = 2 * nhr + nd;
        float* buf = S.r1();  // [N][per]
        if (!gather_partials(p, d, h0, nhr, r.lo, nd, buf, ep(p, step, e0 + 1))) return;
        for (int fi = warp; fi < nd; fi += kW) {
          const int f = r.lo + fi, hr = f / d - h0;
          float m = -INFINITY;
          for (int src = lane; src < N; src += 32) m = fmaxf(m, buf[src * per + 2 * hr]);
          m = warp_max(m);
          float num = 0.f, den = 0.f;
          if (m != -INFINITY) {
            for (int src = lane; src < N; src += 32) {
              const float e = expf(buf[src * per + 2 * hr] - m);
              num = fmaf(e, buf[src * per + 2 * nhr + fi], num);
              den = fmaf(e, buf[src * per + 2 * hr + 1], den);
            }
          }
          num = warp_sum(num);
          den = warp_sum(den);
          if (lane == 0) mb_put(p.mb_o, f, den > 0.f ? num / den : 0.f, ep(p, step, e0 + 2));
        }
        __syncthreads();
      }
      // ---- O
      {
        float* o = S.r2();
        if (!gather(p, p.mb_o, QD, o, ep(p, step, e0 + 2))) return;
        if (!wait_section(p, S.bar(sec_o(l)), step > 0)) return;
        const Range r = split(H, N, c);
        smem_gemv(S.sec(sec_o(l)), r.hi - r.lo, QD, o, red, t);
        for (int i = tid; i < r.hi - r.lo; i += kT) mb_put(p.mb_op, r.lo + i, t[i], ep(p, step, e0 + 3));
      }
      // ---- GU
      {
        const float g_pa = gain_reg(p.post_attn_norm[l], H);
        const float g_ff = gain_reg(p.ffn_norm[l], H);
        if (!gather(p, p.mb_op, H, t, ep(p, step, e0 + 3))) return;
        const float rf = rms_inv(t, H, p.eps, red);
        if (tid < H) x[tid] = x[tid] + t[tid] * rf * g_pa;
        __syncthreads();
        const float rf2 = rms_inv(x, H, p.eps, red);
        if (tid < H) a[tid] = x[tid] * rf2 * g_ff;
        __syncthreads();
        if (!wait_section(p, S.bar(sec_g(l)), step > 0) || !wait_section(p, S.bar(sec_u(l)), step > 0)) return;
        const Range r = split(p.F, N, c);
        const int nr = r.hi - r.lo;
        float* gt = S.r1();
        float* up = S.r1() + 64;
        smem_gemv(S.sec(sec_g(l)), nr, H, a, red, gt);
        smem_gemv(S.sec(sec_u(l)), nr, H, a, red, up);
        for (int i = tid; i < nr; i += kT) mb_put(p.mb_m, r.lo + i, gelu_tanh(gt[i]) * up[i], ep(p, step, e0 + 4));
        __syncthreads();
      }
      // ---- DN
      {
        float* m = S.r1();
        if (!gather(p, p.mb_m, p.F, m, ep(p, step, e0 + 4))) return;
        if (!wait_section(p, S.bar(sec_d(l)), step > 0)) return;
        const Range r = split(H, N, c);
        smem_gemv(S.sec(sec_d(l)), r.hi - r.lo, p.F, m, red, t);
        for (int i = tid; i < r.hi - r.lo; i += kT) mb_put(p.mb_dn, r.lo + i, t[i], ep(p, step, e0 + 5));
      }
    }
    // ================= HEAD
    {
      const int eh = 1 + 6 * p.nl;
      const float g_pf = gain_reg(p.post_ffn_norm[p.nl - 1], H);
      const float g_out = gain_reg(p.out_norm, H);
      if (!gather(p, p.mb_dn, H, t, ep(p, step, eh - 1))) return;
      const float rf = rms_inv(t, H, p.eps, red);
      if (tid < H) x[tid] = p.lambda[p.nl - 1] * (x[tid] + t[tid] * rf * g_pf);
      __syncthreads();
      const float rf2 = rms_inv(x, H, p.eps, red);
      if (tid < H) a[tid] = x[tid] * rf2 * g_out;  // a = y
      __syncthreads();
      if (!wait_section(p, S.bar(S_POST), step > 0) || !wait_section(p, S.bar(S_CENT), step > 0)) return;
      {
        const Range r = split(p.C, N, c);
        smem_gemv(S.sec(S_CENT), r.hi - r.lo, H, a, red, t);
        for (int i = tid; i < r.hi - r.lo; i += kT) mb_put(p.mb_cent, r.lo + i, t[i], ep(p, step, eh + 1));
        __syncthreads();
      }
      {
        const Range r = split(p.bb, N, c);
        smem_gemv(S.sec(S_POST), r.hi - r.lo, H, a, red, t);
        for (int i = tid; i < r.hi - r.lo; i += kT) {
          mb_put(p.mb_h, r.lo + i, t[i], ep(p, step, eh));
          if (p.out_hidden) p.out_hidden[static_cast<size_t>(step) * p.bb + r.lo + i] = t[i];
        }
        __syncthreads();
      }
      // ---- TOPK
      float* cl = S.r1();
      if (!gather(p, p.mb_cent, p.C, cl, ep(p, step, eh + 1))) return;
      // pending keys live in the q/o scratch (free in this phase; it holds C entries)
      topk_select(cl, p.C, p.topk, S.hist(), S.sel(), red, reinterpret_cast<unsigned*>(S.r2()));
      // ---- GATHER: candidates (offset o of this CTA, selected centroid j)
      unsigned long long best = 0ull;
      const int ncand = (offs.hi - offs.lo) * p.topk;
      for (int u = warp; u < ncand; u += kW) {
        const int oo = u / p.topk, j = u % p.topk;
        const int id = S.ord()[oo * p.C + S.sel()[j]];
        const bf16* rw = p.temb + static_cast<size_t>(id) * H;
        float s = 0.f;
        for (int k = lane * 8; k < H; k += 256) {
          float w[8];
          load_vec_stream(rw + k, w);
#pragma unroll
          for (int e = 0; e < 8; ++e) s = fmaf(w[e], a[k + e], s);
        }
        s = warp_sum(s);
        const unsigned long long key = argmax_key(s, id);
        best = key > best ? key : best;
      }
      unsigned long long* kb = reinterpret_cast<unsigned long long*>(red);
      if (lane == 0) kb[warp] = best;
      __syncthreads();
      unsigned long long m = 0ull;
      for (int w = 0; w < kW; ++w) m = kb[w] > m ? kb[w] : m;
      if (tid == 0) {
        mb_put_u(p.mb_key, 2 * c, static_cast<unsigned>(m >> 32), ep(p, step, eh + 2));
        mb_put_u(p.mb_key, 2 * c + 1, 0xffffffffu - static_cast<unsigned>(m), ep(p, step, eh + 2));
      }
      if (m != 0ull && warp == 1) {
        // warm L2 with this CTA's best token's embedding row (one of them is the next token)
        const char* er = reinterpret_cast<const char*>(p.tgt + static_cast<size_t>(key_id(m)) * p.bb);
        for (int off = lane * 128; off < p.bb * 2; off += 32 * 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(er + off));
      }
      __syncthreads();
    }
  }
  // tokens of the last step
  if (c == 0) {
    int tok;
    if (!best_token(p, S, p.n_draft - 1, tok)) return;
    if (tid == 0) p.out_tokens[p.n_draft - 1] = tok;
  }
}

}  // namespace ll

// Host: shared-memory bytes of the kernel for these parameters, or 0 if it cannot run
// (shape beyond the resident budget or the per-CTA work limits).
int ll_smem_bytes(const ll::Params& p) {
  const ll::Layout L = ll::make_layout(p);
  auto units = [&](int R, int K) { return ll::split_max(R, p.N) * ((K + 255) / 256); };
  int u = units(p.H, 2 * p.bb);
  int rows_max = ll::split_max(p.bb, p.N);
  rows_max = rows_max > ll::split_max(p.C, p.N) ? rows_max : ll::split_max(p.C, p.N);
  int dmax = 0;
  for (int l = 0; l < p.nl; ++l) {
    const int d = p.d[p.ltype[l]];
    dmax = d > dmax ? d : dmax;
    u = u > units(p.nh * d, p.H) ? u : units(p.nh * d, p.H);
    u = u > units(p.H, p.nh * d) ? u : units(p.H, p.nh * d);
    u = u > units(p.F, p.H) ? u : units(p.F, p.H);
    u = u > units(p.H, p.F) ? u : units(p.H, p.F);
    const int r = ll::split_max(p.nh * d, p.N);
    rows_max = rows_max > r ? rows_max : r;
  }
  u = u > units(p.bb, p.H) ? u : units(p.bb, p.H);
  u = u > units(p.C, p.H) ? u : units(p.C, p.H);
  // reduction scratch (64 floats), gate/up rows in r1 (64 each), outputs in [H], gains one
  // per thread, q_norm at most 2 per thread, heads at most one per warp
  if (u > 64 || ll::split_max(p.F, p.N) > 64 || rows_max > p.H || p.N > 256 || p.nh > 8 || p.topk > 64 ||
      p.H > ll::kT || dmax > 2 * ll::kT || p.nh > ll::kW || dmax % 4 || p.C > L.r2_floats)
    return 0;
  return L.total;
}

int run_ll(const ll::Params& p, int smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(ll::k_block_ll, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) {
    set_error("latency kernel smem attribute (%d B): %s", smem, cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  ll::Params pp = p;
  void* args[] = {&pp};
  e = cudaLaunchCooperativeKernel(reinterpret_cast<void*>(ll::k_block_ll), dim3(p.N), dim3(ll::kT), args,
                                  static_cast<size_t>(smem), st);
  if (e != cudaSuccess) {
    set_error("latency draft-block launch (%d CTAs, %d B smem): %s", p.N, smem, cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

int ll_capacity(int smem, int num_sms) {
  if (cudaFuncSetAttribute(ll::k_block_ll, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ll::k_block_ll, ll::kT, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return per_sm * num_sms;
}

}  // namespace mtp
