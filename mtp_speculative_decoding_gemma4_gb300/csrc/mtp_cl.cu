// Cluster-path draft block (B = 1): see mtp_cl.cuh for the data flow.
//
// Failure handling: every wait is bounded. A wait that gives up records MTP_ERR_TIMEOUT and
// raises the abort word; a raised abort word makes every later wait give up after a few
// polls. Control flow never depends on a wait's outcome, so every thread keeps executing the
// same sequence of named barriers, exchanges and ring releases and no barrier is left short
// of arrivals. Values derived from exchanged data (centroid ids, token ids) are clamped
// before they address memory. Before the CTA ends, its producer waits (time-bounded,
// independent of the abort word) for its own copies still in flight, and a final cluster
// barrier keeps every CTA alive while peers may still write to it.
//
// Work split inside a CTA (kCW compute warps):
//   hidden-wide GEMVs (Q, gate, up, centroids, post_projection): tensor cores on tiles packed
//     at init (mma.m16n8k16, the fp32 input split into three exact bf16 terms); warps take
//     (row tile, k quarter) pairs, the quarters added in a fixed order.
//   other GEMV slots (pre_projection, O, down): (row quad, k slice) tasks, one warp each; a
//     warp reads four rows at once and reduces the four dot products with one transposed
//     butterfly; k-split partial sums are added in a fixed order (deterministic).
//   scores: (key quad, head group, k slice) tasks; the heads sharing a KV head reuse each
//     K load.
//   weighted sum (V = K): a thread owns four dims of one KV head for a group of heads and one
//     key group; key groups are lane groups of a warp, reduced by shuffles at the end.
#include <cmath>
#include <cstring>

#include "mtp_cl.cuh"
#include "mtp_launch.h"

namespace mtp {
namespace clk {

// ------------------------------------------------------------------ primitives

__device__ __forceinline__ unsigned sa(const void* p) { return static_cast<unsigned>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ unsigned mapa(unsigned addr, int rank) {
  unsigned r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Asynchronous 4-byte store into a peer CTA's shared memory that counts its bytes on the
// peer's mbarrier (both addresses in the shared::cluster window).
__device__ __forceinline__ void st_async_f32(unsigned caddr, float v, unsigned cbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(caddr),
               "r"(__float_as_uint(v)), "r"(cbar)
               : "memory");
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from this CTA's
// shared memory into a peer CTA's, counted on the peer's mbarrier like st.async.
__device__ __forceinline__ void bulk_s2c(unsigned dst_caddr, unsigned src, unsigned bytes, unsigned cbar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_caddr),
               "r"(src), "r"(bytes), "r"(cbar)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until this thread's bulk copies have read their sources (bounded by the copies).
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Orders this thread's shared-memory writes before later bulk copies that read them.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void arrive_local(unsigned bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_g2s(unsigned dst, const void* src, unsigned bytes, unsigned bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// A waiting thread is suspended until the phase completes or this many ns pass, so waits
// do not take issue slots from the warps that still compute.
constexpr unsigned kSuspendNs = 100000;
// Phase test of a ring barrier (filled by this CTA's copies / released by its own warps).
__device__ __forceinline__ bool try_wait_cta(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}
// Phase test of a receive barrier (bytes from peer CTAs, observed at cluster scope).
__device__ __forceinline__ bool try_wait_cluster(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, "
      "p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned ld_rlx32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Loads from shared memory by 32-bit shared address (hot loops keep addresses in one register).
__device__ __forceinline__ uint4 lds128(unsigned a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 ldsf4(unsigned a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(unsigned a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ float ldsf(unsigned a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
// named barrier of the compute warps (the producer warp never takes part)
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory"); }
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void set_status(int* status, int code) { atomicCAS(status, 0, code); }

struct Fail {
  int* status;
  unsigned* abort_flag;
  long long spin_limit;
};
// Bounded wait on an mbarrier phase. A raised abort word ends it early (false); running
// past the time limit records MTP_ERR_TIMEOUT and raises the abort word (false).
__device__ __noinline__ bool wait_bar_slow(Fail f, unsigned bar, unsigned parity, bool cluster_scope) {
  const long long t0 = clock64();
  for (;;) {
    if (cluster_scope ? try_wait_cluster(bar, parity) : try_wait_cta(bar, parity)) return true;
    if (ld_rlx32(f.abort_flag)) return false;
    if (clock64() - t0 > f.spin_limit) {
      set_status(f.status, MTP_ERR_TIMEOUT);
      atomicExch(f.abort_flag, 1u);
      return false;
    }
  }
}
// The common case (phase already complete) without a call.
__device__ __forceinline__ bool wait_bar(const Fail& f, unsigned bar, unsigned parity, bool cluster_scope) {
  if (cluster_scope ? try_wait_cluster(bar, parity) : try_wait_cta(bar, parity)) return true;
  return wait_bar_slow(f, bar, parity, cluster_scope);
}
// Time-bounded wait that ignores the abort word: the drain of this CTA's own copies.
__device__ __noinline__ void drain_bar(Fail f, unsigned bar, unsigned parity) {
  const long long t0 = clock64();
  while (!try_wait_cta(bar, parity)) {
    if (clock64() - t0 > f.spin_limit) {
      set_status(f.status, MTP_ERR_TIMEOUT);
      return;
    }
  }
}

// RMSNorm factor 1/sqrt(mean(v^2) + eps) of a shared-memory vector. Every warp computes it
// on its own, in the same order, so all threads get the same value without a barrier.
__device__ __forceinline__ float rms_inv(const float* v, int n, float eps) {
  const int lane = threadIdx.x & 31;
  float s = 0.f;
  for (int i = lane; i < n; i += 32) s = fmaf(v[i], v[i], s);
  s = warp_sum(s);
  return rsqrtf(s / n + eps);
}

// acc + the dot product of 8 bf16 weights (one 16-byte word) with 8 fp32 values
__device__ __forceinline__ float dot8(uint4 w, float4 a, float4 b, float acc) {
  acc = fmaf(__uint_as_float(w.x << 16), a.x, acc);
  acc = fmaf(__uint_as_float(w.x & 0xffff0000u), a.y, acc);
  acc = fmaf(__uint_as_float(w.y << 16), a.z, acc);
  acc = fmaf(__uint_as_float(w.y & 0xffff0000u), a.w, acc);
  acc = fmaf(__uint_as_float(w.z << 16), b.x, acc);
  acc = fmaf(__uint_as_float(w.z & 0xffff0000u), b.y, acc);
  acc = fmaf(__uint_as_float(w.w << 16), b.z, acc);
  acc = fmaf(__uint_as_float(w.w & 0xffff0000u), b.w, acc);
  return acc;
}

// Sums M per-lane values over the 32 lanes of a warp with one transposed butterfly: at each
// of the first log2(M) levels a lane keeps half of its values and receives its partner's
// share of them. Afterwards every lane holds the full sum of value index lane >> (5 - log2 M).
template <int M>
__device__ __forceinline__ float xreduce(float (&a)[M], int lane) {
  int o = 16;
#pragma unroll
  for (int c = M; c > 1; c >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < c / 2; ++i) {
      const float send = up ? a[i] : a[i + c / 2];
      const float keep = up ? a[i + c / 2] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
    o >>= 1;
  }
  float v = a[0];
  for (; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
template <int M> struct Log2;
template <> struct Log2<4> { static constexpr int v = 2; };
template <> struct Log2<8> { static constexpr int v = 3; };
template <> struct Log2<16> { static constexpr int v = 4; };

// ------------------------------------------------------------------ stream schedule

__device__ __forceinline__ int n_chunks(const Sec& s) { return s.nrows > 0 ? (s.nrows + s.rpc - 1) / s.rpc : 0; }

// Sections of one step, in the order the step consumes them:
//   0 PRE | per block l: 1+6l Q, 2+6l K, 3+6l O, 4+6l gate, 5+6l up, 6+6l down | CENT | POST
__device__ __forceinline__ int sec_count(const Params& p) { return 1 + 6 * p.nl + 2; }

struct Keys {
  int f_lo, f_n, s_lo, s_n;  // this CTA's keys of the full layers and of the sliding window
};

__device__ __noinline__ Sec make_sec(const Params& p, int idx, int r, Keys kr) {
  Sec s{nullptr, 0, 0, 0, 1, 0, 0, 0};
  // a packed matrix: this CTA's block of 512-byte tiles, streamed as `rows` of one tile
  auto packed = [&](const bf16* P, int R, int K) {
    s.src = reinterpret_cast<const char*>(P) + tiles_before(R, K, r) * kTileBytes;
    s.row_bytes = kTileBytes;
    s.stride = kTileBytes;
    s.kt = K / 16;
    s.nrows = padded_rows(R, r) / 16 * s.kt;
    const Range g = split(R, kNC, r);
    s.rrows = g.hi - g.lo;
  };
  auto rows = [&](const bf16* W, int R, int K) {
    const Range rg = split(R, kNC, r);
    s.src = reinterpret_cast<const char*>(W + static_cast<size_t>(rg.lo) * K);
    s.row_bytes = K * 2;
    s.stride = s.row_bytes;
    s.nrows = rg.hi - rg.lo;
  };
  if (idx == 0) {
    rows(p.pre, p.H, 2 * p.bb);
  } else if (idx >= 1 + 6 * p.nl) {
    if (idx == 1 + 6 * p.nl) {
      if (p.mma) packed(p.pk_cent, p.C, p.H);
      else rows(p.cent, p.C, p.H);
    } else {
      if (p.mma) packed(p.pk_post, p.bb, p.H);
      else rows(p.post, p.bb, p.H);
    }
  } else {
    const int l = (idx - 1) / 6, what = (idx - 1) % 6;
    const int lt = p.ltype[l], d = p.d[lt];
    switch (what) {
      case 0:
        if (p.mma) packed(p.pk_q[l], p.nh * d, p.H);
        else rows(p.q[l], p.nh * d, p.H);
        break;
      case 1: {
        const int lo = lt ? kr.f_lo : kr.s_lo, n = lt ? kr.f_n : kr.s_n;
        s.src = reinterpret_cast<const char*>(p.k[lt] + static_cast<size_t>(lo) * p.st[lt]);
        s.row_bytes = p.nkv * d * 2;
        s.stride = p.st[lt] * 2;
        s.nrows = n;
        break;
      }
      case 2: rows(p.o[l], p.H, p.nh * d); break;
      case 3:
        if (p.mma) packed(p.pk_gate[l], p.F, p.H);
        else rows(p.gate[l], p.F, p.H);
        break;
      case 4:
        if (p.mma) packed(p.pk_up[l], p.F, p.H);
        else rows(p.up[l], p.F, p.H);
        break;
      default: rows(p.down[l], p.H, p.F); break;
    }
  }
  const bool kv = idx >= 1 && idx < 1 + 6 * p.nl && (idx - 1) % 6 == 1;
  s.pitch = s.row_bytes;
  if (kv && att_mma_ok(p)) {  // padded rows for the tensor-core attention
    s.pitch = s.row_bytes + 16;
    s.rpc = keys_per_slot_mma(s.row_bytes);
  } else {
    s.rpc = kv ? keys_per_slot(s.row_bytes) : rows_per_slot(s.row_bytes);
  }
  return s;
}

// Consumer side of the ring: shared addresses of the barriers and the generic slot base.
struct Ring {
  unsigned base, full0, empty0;  // shared addresses: slot 0, full barriers, empty barriers
  Fail f;
};
__device__ __forceinline__ unsigned ring_wait(const Ring& rg, int g) {
  const int slot = g % kSlots;
  wait_bar(rg.f, rg.full0 + 8 * slot, static_cast<unsigned>((g / kSlots) & 1), false);
  return rg.base + slot * kSlotStride;
}
__device__ __forceinline__ void ring_release(const Ring& rg, int g) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) arrive_local(rg.empty0 + 8 * (g % kSlots));
}

// ------------------------------------------------------------------ phase functions

// out[i] = W_i . x for the rows of a streamed section (chunk counter g at its first chunk);
// x is fp32 in shared memory. Returns the chunk counter after the section.
__device__ __forceinline__ int gemv_sec(Ring rg, int g, Sec s, const float* x, float* out, float* part) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nc = n_chunks(s), K = s.row_bytes / 2, V8 = K / 8;
  const int ns = gemv_ns(s.rpc), nq = (s.rpc + 3) / 4, ntask = nq * ns;
  const unsigned xs = sa(x);
  for (int ch = 0; ch < nc; ++ch, ++g) {
    const unsigned W = ring_wait(rg, g);
    const int r0 = ch * s.rpc, n = min(s.rpc, s.nrows - r0);
    for (int t = warp; t < ntask; t += kCW) {
      const int rq = 4 * (t % nq), sl = t / nq;
      if (rq >= n) continue;  // warp-uniform
      const int vlo = V8 * sl / ns, vhi = V8 * (sl + 1) / ns;
      const unsigned w0 = W + static_cast<unsigned>(min(rq, n - 1) * s.row_bytes);
      const unsigned w1 = W + static_cast<unsigned>(min(rq + 1, n - 1) * s.row_bytes);
      const unsigned w2 = W + static_cast<unsigned>(min(rq + 2, n - 1) * s.row_bytes);
      const unsigned w3 = W + static_cast<unsigned>(min(rq + 3, n - 1) * s.row_bytes);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int v = vlo + lane; v < vhi; v += 32) {
        const float4 xa = ldsf4(xs + 32 * v), xb = ldsf4(xs + 32 * v + 16);
        const uint4 q0 = lds128(w0 + 16 * v), q1 = lds128(w1 + 16 * v);
        const uint4 q2 = lds128(w2 + 16 * v), q3 = lds128(w3 + 16 * v);
        acc[0] = dot8(q0, xa, xb, acc[0]);
        acc[1] = dot8(q1, xa, xb, acc[1]);
        acc[2] = dot8(q2, xa, xb, acc[2]);
        acc[3] = dot8(q3, xa, xb, acc[3]);
      }
      const float val = xreduce<4>(acc, lane);
      const int row = rq + (lane >> 3);
      if ((lane & 7) == 0 && row < n) {
        if (ns == 1) out[r0 + row] = val;
        else part[sl * s.nrows + r0 + row] = val;
      }
    }
    ring_release(rg, g);
  }
  if (ns > 1) {
    cbar();
    for (int i = threadIdx.x; i < s.nrows; i += kCT) {
      float v = 0.f;
      for (int sl = 0; sl < ns; ++sl) v += part[sl * s.nrows + i];
      out[i] = v;
    }
  }
  cbar();
  return g;
}

// D += A (16x16 bf16, row) x B (16x8 bf16, col), fp32 accumulate. A pure register operation
// (not volatile), so the compiler may overlap it with the shared-memory loads of later steps.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t lds32(unsigned a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// Splits the n fp32 values of x into three bf16 terms hi + mid + lo (x == hi + mid + lo up to
// the rounding of lo, i.e. fp32 precision), written as rows 0..2 of xt [4][n + 8]; row 3 is
// zero. The row pitch n + 8 puts the 8 B-fragment rows a warp reads at one column in distinct
// banks. The tensor-core GEMVs multiply these terms by the bf16 weights: every product is
// exact and the sums are fp32, so the result equals an fp32 dot product up to summation order.
__device__ __forceinline__ void split_terms(const float* x, int n, bf16* xt) {
  const int pt = n + 8;
  for (int i = threadIdx.x; i < n; i += kCT) {
    const float v = x[i];
    const bf16 h = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(h);
    const bf16 m = __float2bfloat16_rn(r1);
    const bf16 l = __float2bfloat16_rn(r1 - __bfloat162float(m));
    xt[i] = h;
    xt[pt + i] = m;
    xt[2 * pt + i] = l;
    xt[3 * pt + i] = __float2bfloat16_rn(0.f);
  }
}

// Row sums of a 16-row tile's MMA result (columns 0..2 carry the three input terms, column 3
// is zero): lanes ti = 0 hold rows gi and gi + 8 after the pair reduction.
__device__ __forceinline__ void tile_rows_out(const float (&d)[4], int ti, int gi, float* part, int row0) {
  float v0 = d[0] + d[1], v1 = d[2] + d[3];
  v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
  v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
  if (ti == 0) {
    part[row0 + gi] = v0;
    part[row0 + gi + 8] = v1;
  }
}

// out[i] = W_i . x for a packed section (tiles of this CTA's rows, see Params::pk_q) with the
// input already split into xt [4][K + 8]. Per slot, warp w multiplies row tiles (w / 4),
// (w / 4) + kCW / 4, ... over the k quarter (w % 4); B column n < 3 carries term n of x, so a
// row's value is the sum of D's first three columns. The warp's B fragments are loaded once;
// for K = 256 (4 k-steps per quarter) two row tiles go at a time, their A tiles loaded first
// and their MMA chains interleaved. The four k-quarter partials are added in a fixed order.
__device__ __forceinline__ int gemv_mma_sec(Ring rg, int g, Sec s, const bf16* xt, float* out, float* part) {
  constexpr int kMaxKtn = 8;  // k-steps per quarter held as B fragments (K <= 512)
  constexpr int kStepRt = kCW / 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, ti = lane & 3;
  const int KT = s.kt, K = KT * 16, kq = warp & 3, ktn = KT / 4, kt0 = kq * ktn;
  const int nc = n_chunks(s), rts = s.rpc / KT, PR = (s.rrows + 15) / 16 * 16;
  // this lane's B column: term gi of x for gi < 3, the zero row otherwise
  const unsigned xb = sa(xt) + 2u * static_cast<unsigned>((gi < 3 ? gi : 3) * (K + 8) + 2 * ti);
  uint32_t bf[2 * kMaxKtn];
#pragma unroll
  for (int j = 0; j < kMaxKtn; ++j) {
    bf[2 * j] = bf[2 * j + 1] = 0u;
    if (j < ktn) {
      const unsigned bk = xb + 32u * static_cast<unsigned>(kt0 + j);
      bf[2 * j] = lds32(bk);
      bf[2 * j + 1] = lds32(bk + 16);
    }
  }
  for (int ch = 0; ch < nc; ++ch, ++g) {
    const unsigned W = ring_wait(rg, g);
    const int nt = min(s.rpc, s.nrows - ch * s.rpc), nrt = nt / KT;
    float* pq = part + kq * PR + ch * rts * 16;
    if (ktn == 4) {
      for (int rt = warp >> 2; rt < nrt; rt += 2 * kStepRt) {
        const int rt2 = rt + kStepRt;
        const bool two = rt2 < nrt;
        const unsigned a0 = W + static_cast<unsigned>((rt * KT + kt0) * kTileBytes + lane * 16);
        const unsigned a1 = W + static_cast<unsigned>(((two ? rt2 : rt) * KT + kt0) * kTileBytes + lane * 16);
        uint4 a[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          a[j] = lds128(a0 + j * kTileBytes);
          a[4 + j] = lds128(a1 + j * kTileBytes);
        }
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          mma_bf16(d0, a[j], bf[2 * j], bf[2 * j + 1]);
          mma_bf16(d1, a[4 + j], bf[2 * j], bf[2 * j + 1]);
        }
        tile_rows_out(d0, ti, gi, pq, rt * 16);
        if (two) tile_rows_out(d1, ti, gi, pq, rt2 * 16);
      }
    } else {
      for (int rt = warp >> 2; rt < nrt; rt += kStepRt) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        const unsigned a0 = W + static_cast<unsigned>((rt * KT + kt0) * kTileBytes + lane * 16);
#pragma unroll
        for (int j = 0; j < kMaxKtn; ++j)
          if (j < ktn) mma_bf16(d, lds128(a0 + j * kTileBytes), bf[2 * j], bf[2 * j + 1]);
        tile_rows_out(d, ti, gi, pq, rt * 16);
      }
    }
    ring_release(rg, g);
  }
  cbar();
  for (int i = threadIdx.x; i < s.rrows; i += kCT)
    out[i] = ((part[i] + part[PR + i]) + part[2 * PR + i]) + part[3 * PR + i];
  cbar();
  return g;
}

// Scores of the nh heads against the n keys of one K slot (shared address K), scaled; with
// ns > 1 k slices the partial scores go to ns slices of sstride floats each.
template <int NHT>
__device__ __noinline__ void qk_chunk(int nh, int nkv, unsigned K, int n, const float* q, float* sc, int d, float scale,
                                      int ns, int sstride) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hpg = nh / nkv, HG = hpg / NHT, nhg = nkv * HG;
  const int row = nkv * d, V8 = d / 8;
  const int nq = (n + 3) / 4, base = nq * nhg;
  const unsigned qs = sa(q);
  for (int t = warp; t < base * ns; t += kCW) {
    const int kq = 4 * (t % nq), hg = (t / nq) % nhg, sl = t / base;
    if (kq >= n) continue;  // warp-uniform
    const int gk = hg / HG, h0 = gk * hpg + (hg % HG) * NHT;
    const int vlo = V8 * sl / ns, vhi = V8 * (sl + 1) / ns;
    const unsigned k0 = K + 2u * static_cast<unsigned>(min(kq, n - 1) * row + gk * d);
    const unsigned k1 = K + 2u * static_cast<unsigned>(min(kq + 1, n - 1) * row + gk * d);
    const unsigned k2 = K + 2u * static_cast<unsigned>(min(kq + 2, n - 1) * row + gk * d);
    const unsigned k3 = K + 2u * static_cast<unsigned>(min(kq + 3, n - 1) * row + gk * d);
    const unsigned qh0 = qs + 4u * static_cast<unsigned>(h0 * d);
    float a[4 * NHT];
#pragma unroll
    for (int i = 0; i < 4 * NHT; ++i) a[i] = 0.f;
    for (int v = vlo + lane; v < vhi; v += 32) {
      const uint4 kw0 = lds128(k0 + 16 * v), kw1 = lds128(k1 + 16 * v);
      const uint4 kw2 = lds128(k2 + 16 * v), kw3 = lds128(k3 + 16 * v);
#pragma unroll
      for (int th = 0; th < NHT; ++th) {
        const unsigned qa_ = qh0 + 4u * static_cast<unsigned>(th * d) + 32 * v;
        const float4 qa = ldsf4(qa_), qb = ldsf4(qa_ + 16);
        a[0 * NHT + th] = dot8(kw0, qa, qb, a[0 * NHT + th]);
        a[1 * NHT + th] = dot8(kw1, qa, qb, a[1 * NHT + th]);
        a[2 * NHT + th] = dot8(kw2, qa, qb, a[2 * NHT + th]);
        a[3 * NHT + th] = dot8(kw3, qa, qb, a[3 * NHT + th]);
      }
    }
    const float val = xreduce<4 * NHT>(a, lane);
    const int idx = lane >> (5 - Log2<4 * NHT>::v);
    const int key = kq + idx / NHT, h = h0 + idx % NHT;
    if ((lane & ((32 >> Log2<4 * NHT>::v) - 1)) == 0 && key < n) sc[sl * sstride + key * nh + h] = val * scale;
  }
}

// Attention of the nh query heads over this CTA's keys of one block (online softmax over the
// streamed K chunks, V = K). q: [nh][d] after q_norm and RoPE. Leaves in stage the
// unnormalised sums [nh][d] followed by (m_h, l_h) of every head. Returns the chunk counter.
template <int NHT>
__device__ __noinline__ int att_sec(int nh, int nkv, Ring rg, int g, Sec s, int d, float scale, const float* q,
                                    float* sc, float* red, float* stage) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hpg = nh / nkv, HG = hpg / NHT, nhg = nkv * HG;
  const int row = nkv * d, V8 = d / 8, DQ = d / 4;
  const int nc = n_chunks(s);
  // score tasks: (key quad, head group, k slice)
  const int nq = (s.rpc + 3) / 4, base = nq * nhg;
  int ns = 1;
  while (ns * 2 <= kQkSlices && ns * 2 * base <= kCW && V8 / (ns * 2) >= 32) ns *= 2;
  const int sstride = s.rpc * nh;  // floats per score slice; two alternating buffers of ns slices
  // weighted-sum slots: (head group, dim quad) per thread, key groups in lane bits
  const int D = nhg * DQ;
  int kgw = 1;
  while (kgw * 2 <= 32 && D * kgw * 2 <= kCT) kgw *= 2;
  const int lpk = 32 / kgw, slot = warp * lpk + lane % lpk, kg = lane / lpk;
  const bool own = slot < D;
  const int dq = own ? slot % DQ : 0, hgi = own ? slot / DQ : 0;
  const int gk_pv = hgi / HG, h0_pv = gk_pv * hpg + (hgi % HG) * NHT;
  float acc[NHT][4];
#pragma unroll
  for (int t = 0; t < NHT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  for (int ch = 0; ch < nc; ++ch, ++g) {
    const unsigned K = ring_wait(rg, g);
    const int n = min(s.rpc, s.nrows - ch * s.rpc);
    float* scb = sc + (ch & 1) * (kQkSlices * sstride);
    qk_chunk<NHT>(nh, nkv, K, n, q, scb, d, scale, ns, sstride);
    cbar();
    // ---- running max / exp-sum: one warp per head; probabilities overwrite slice 0
    if (warp < nh) {
      float cm = -INFINITY;
      for (int j = lane; j < n; j += 32) {
        float v = scb[j * nh + warp];
        for (int sl = 1; sl < ns; ++sl) v += scb[sl * sstride + j * nh + warp];
        scb[j * nh + warp] = v;
        cm = fmaxf(cm, v);
      }
      cm = warp_max(cm);
      const float mold = red[48 + warp];
      const float mnew = fmaxf(mold, cm);
      float ls = 0.f;
      for (int j = lane; j < n; j += 32) {
        const float e = expf(scb[j * nh + warp] - mnew);
        scb[j * nh + warp] = e;
        ls += e;
      }
      ls = warp_sum(ls);
      if (lane == 0) {
        const float corr = expf(mold - mnew);
        red[80 + warp] = corr;
        red[64 + warp] = red[64 + warp] * corr + ls;
        red[48 + warp] = mnew;
      }
    }
    cbar();
    // ---- weighted sum of the keys
    if (own) {
#pragma unroll
      for (int t = 0; t < NHT; ++t) {
        const float c = red[80 + h0_pv + t];
        acc[t][0] *= c;
        acc[t][1] *= c;
        acc[t][2] *= c;
        acc[t][3] *= c;
      }
      const unsigned kb = K + 2u * static_cast<unsigned>(gk_pv * d + 4 * dq);
      for (int j = kg; j < n; j += kgw) {
        const uint2 raw = lds64(kb + 2u * static_cast<unsigned>(j * row));
        const float k0 = __uint_as_float(raw.x << 16), k1 = __uint_as_float(raw.x & 0xffff0000u);
        const float k2 = __uint_as_float(raw.y << 16), k3 = __uint_as_float(raw.y & 0xffff0000u);
        const unsigned pj = sa(scb) + 4u * static_cast<unsigned>(j * nh + h0_pv);
#pragma unroll
        for (int t = 0; t < NHT; ++t) {
          const float w = ldsf(pj + 4 * t);
          acc[t][0] = fmaf(w, k0, acc[t][0]);
          acc[t][1] = fmaf(w, k1, acc[t][1]);
          acc[t][2] = fmaf(w, k2, acc[t][2]);
          acc[t][3] = fmaf(w, k3, acc[t][3]);
        }
      }
    }
    // no barrier here: the next chunk's scores go to the other buffer, and the barrier after
    // them orders this chunk's reads of its buffer before that buffer is written again
    ring_release(rg, g);
  }
  // key groups -> one sum per (head, dim)
#pragma unroll
  for (int t = 0; t < NHT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      for (int o = lpk; o < 32; o <<= 1) acc[t][i] += __shfl_xor_sync(0xffffffffu, acc[t][i], o);
  if (own && kg == 0) {
#pragma unroll
    for (int t = 0; t < NHT; ++t)
      *reinterpret_cast<float4*>(stage + (h0_pv + t) * d + 4 * dq) = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
  }
  if (tid < nh) {
    stage[nh * d + 2 * tid] = red[48 + tid];
    stage[nh * d + 2 * tid + 1] = red[64 + tid];
  }
  cbar();
  return g;
}

// Four 8x8 bf16 matrices from shared memory (lane i gives a row address of matrix i / 8).
__device__ __forceinline__ uint4 ldsm_x4(unsigned addr) {
  uint4 r;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}
// The same, each matrix transposed.
__device__ __forceinline__ uint4 ldsm_x4_t(unsigned addr) {
  uint4 r;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}
// The bf16 pair of keys (key, key + 1) in v with the keys at or past n set to zero.
__device__ __forceinline__ uint32_t keep_keys(uint32_t v, int key, int n) {
  return key + 1 < n ? v : (key < n ? (v & 0xffffu) : 0u);
}
// Three bf16 terms of v (hi + mid + lo == v to fp32 precision) at rows 0, rs, 2 rs of dst.
__device__ __forceinline__ void put_terms(bf16* dst, int rs, float v) {
  const bf16 h = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(h);
  const bf16 m = __float2bfloat16_rn(r1);
  dst[0] = h;
  dst[rs] = m;
  dst[2 * rs] = __float2bfloat16_rn(r1 - __bfloat162float(m));
}

constexpr int kAttMaxNT = 2;  // n tiles of the attention MMAs: 4 columns per head, nh <= 4
constexpr int kAttMaxMT = 4;  // dim tiles of the weighted sum per warp: d <= 16 * 4 * kCW
constexpr int kAttMaxKU = 4;  // keys per lane in the softmax: a slot holds at most 128 keys

// Attention of the nh query heads (one KV head, V = K) over this CTA's keys of one block on
// tensor cores (mma.m16n8k16, bf16 operands, fp32 accumulation). K rows sit in the slots at
// pitch s.pitch (= 2d + 16 bytes). q is given as three bf16 terms per head, row 3h + t of qt
// (pitch d + 8 elements); column 4h + t of the MMAs carries term t of head h (t < 3, the
// fourth column is zero), so every product is exact and a head's value is the sum of its
// three columns. Per slot of n keys:
//   scores  S[key][col] = K q: tasks (16-key tile, quarter of the dims) over the warps, the
//           dims chained in the MMA in groups of 4 steps (64 dims), then added in fp32;
//   softmax one warp per head sums the four quarter partials in a fixed order, updates the
//           running max / exp-sum and writes p as three bf16 terms (row 3h + t of pt);
//   sums    O^T[dim][col] += K^T P^T: every warp owns dim tiles, keys chained per slot.
// Leaves the unnormalised sums [nh][d] and (m_h, l_h) in stage, like att_sec.
__device__ __forceinline__ int att_sec_mma(int nh, Ring rg, int g, Sec s, int d, float scale, const bf16* qt,
                                        float* sc, bf16* pt, float* red, float* stage) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gi = lane >> 2, ti = lane & 3;
  const int nc = n_chunks(s), kps = s.rpc, P = s.pitch, qp = d + 8, pp = kps + 8;
  const int KS = d / 16, KQ = (KS + 3) / 4, NT = (nh + 1) / 2, MT = d / 16;
  const unsigned qts = sa(qt), pts = sa(pt);
  // this lane's B column of n tile nt: head and term (term 3: the zero column)
  auto bcol_row = [&](int nt) -> int {
    const int c = nt * 8 + gi, h = c >> 2, t = c & 3;
    return (t == 3 || h >= nh) ? -1 : 3 * h + t;
  };
  float acc[kAttMaxMT][kAttMaxNT][4];
#pragma unroll
  for (int m = 0; m < kAttMaxMT; ++m)
#pragma unroll
    for (int nt = 0; nt < kAttMaxNT; ++nt) acc[m][nt][0] = acc[m][nt][1] = acc[m][nt][2] = acc[m][nt][3] = 0.f;

  for (int ch = 0; ch < nc; ++ch, ++g) {
    const unsigned K = ring_wait(rg, g);
    const int n = min(kps, s.nrows - ch * kps), nmt = (n + 15) / 16;
    // ---- scores: task (key tile, dim quarter)
    for (int task = warp; task < nmt * 4; task += kCW) {
      const int j0 = (task >> 2) * 16, kq = task & 3;
      const int ks0 = kq * KQ, ks1 = min(KS, ks0 + KQ);
      float sv[kAttMaxNT][4];
#pragma unroll
      for (int nt = 0; nt < kAttMaxNT; ++nt) sv[nt][0] = sv[nt][1] = sv[nt][2] = sv[nt][3] = 0.f;
      // lane's ldmatrix row: key j0 + (lane & 7) + 8 * ((lane >> 3) & 1), dims + 8 * (lane >> 4)
      const unsigned arow = K + static_cast<unsigned>((j0 + (lane & 7) + ((lane >> 3) & 1) * 8) * P + (lane >> 4) * 16);
      for (int kb = ks0; kb < ks1; kb += 4) {
        float dg[kAttMaxNT][4];
#pragma unroll
        for (int nt = 0; nt < kAttMaxNT; ++nt) dg[nt][0] = dg[nt][1] = dg[nt][2] = dg[nt][3] = 0.f;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int ks = kb + k4;
          if (ks >= ks1) break;
          const uint4 a = ldsm_x4(arow + ks * 32);
#pragma unroll
          for (int nt = 0; nt < kAttMaxNT; ++nt) {
            if (nt < NT) {
              const int row = bcol_row(nt);
              uint32_t b0 = 0u, b1 = 0u;
              if (row >= 0) {
                const unsigned bq = qts + 2u * static_cast<unsigned>(row * qp + ks * 16 + 2 * ti);
                b0 = lds32(bq);
                b1 = lds32(bq + 16);
              }
              mma_bf16(dg[nt], a, b0, b1);
            }
          }
        }
#pragma unroll
        for (int nt = 0; nt < kAttMaxNT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) sv[nt][i] += dg[nt][i];
      }
      // head values: columns 2ti, 2ti + 1 of lanes ti and ti ^ 1 hold the three terms
#pragma unroll
      for (int nt = 0; nt < kAttMaxNT; ++nt) {
        if (nt < NT) {
          float v0 = sv[nt][0] + sv[nt][1], v1 = sv[nt][2] + sv[nt][3];
          v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
          v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
          const int h = (nt * 8 + 2 * ti) >> 2;
          if ((ti & 1) == 0 && h < nh) {
            sc[(kq * kps + j0 + gi) * nh + h] = v0;
            sc[(kq * kps + j0 + gi + 8) * nh + h] = v1;
          }
        }
      }
    }
    cbar();
    // ---- running max / exp-sum per head; p of the slot's keys as three bf16 terms
    if (warp < nh) {
      const int h = warp;
      float sv[kAttMaxKU];
      float cm = -INFINITY;
#pragma unroll
      for (int u = 0; u < kAttMaxKU; ++u) {
        const int j = lane + 32 * u;
        float v = -INFINITY;
        if (j < n) {
          v = ((sc[(0 * kps + j) * nh + h] + sc[(1 * kps + j) * nh + h]) + sc[(2 * kps + j) * nh + h]) +
              sc[(3 * kps + j) * nh + h];
          v *= scale;
        }
        sv[u] = v;
        cm = fmaxf(cm, v);
      }
      cm = warp_max(cm);
      const float mold = red[48 + h];
      const float mnew = fmaxf(mold, cm);
      float ls = 0.f;
#pragma unroll
      for (int u = 0; u < kAttMaxKU; ++u) {
        const int j = lane + 32 * u;
        if (j < nmt * 16) {
          const float e = j < n ? expf(sv[u] - mnew) : 0.f;
          ls += e;
          put_terms(pt + 3 * h * pp + j, pp, e);
        }
      }
      ls = warp_sum(ls);
      if (lane == 0) {
        const float corr = expf(mold - mnew);
        red[80 + h] = corr;
        red[64 + h] = red[64 + h] * corr + ls;
        red[48 + h] = mnew;
      }
    }
    cbar();
    // ---- weighted sums: this warp's dim tiles
    {
      float cr[kAttMaxNT];
#pragma unroll
      for (int nt = 0; nt < kAttMaxNT; ++nt) {
        const int h = (nt * 8 + 2 * ti) >> 2;
        cr[nt] = (nt < NT && h < nh) ? red[80 + h] : 0.f;
      }
      float dg[kAttMaxMT][kAttMaxNT][4];
#pragma unroll
      for (int m = 0; m < kAttMaxMT; ++m)
#pragma unroll
        for (int nt = 0; nt < kAttMaxNT; ++nt) dg[m][nt][0] = dg[m][nt][1] = dg[m][nt][2] = dg[m][nt][3] = 0.f;
      for (int ks = 0; ks < nmt; ++ks) {
        const int j0 = ks * 16;
        uint32_t b0[kAttMaxNT], b1[kAttMaxNT];
#pragma unroll
        for (int nt = 0; nt < kAttMaxNT; ++nt) {
          const int row = nt < NT ? bcol_row(nt) : -1;
          b0[nt] = b1[nt] = 0u;
          if (row >= 0) {
            const unsigned bp = pts + 2u * static_cast<unsigned>(row * pp + j0 + 2 * ti);
            b0[nt] = lds32(bp);
            b1[nt] = lds32(bp + 16);
          }
        }
        // lane's transposed-ldmatrix row: key j0 + (lane & 7) + 8 * (lane >> 4), dims + 8 * ((lane >> 3) & 1)
        const unsigned arow = K + static_cast<unsigned>((j0 + (lane & 7) + (lane >> 4) * 8) * P + ((lane >> 3) & 1) * 16);
        const bool tail = j0 + 16 > n;
#pragma unroll
        for (int m = 0; m < kAttMaxMT; ++m) {
          const int mt = warp + m * kCW;
          if (mt < MT) {
            uint4 a = ldsm_x4_t(arow + mt * 32);
            if (tail) {  // keys past the slot's rows: zero (their rows hold no K)
              a.x = keep_keys(a.x, j0 + 2 * ti, n);
              a.y = keep_keys(a.y, j0 + 2 * ti, n);
              a.z = keep_keys(a.z, j0 + 8 + 2 * ti, n);
              a.w = keep_keys(a.w, j0 + 8 + 2 * ti, n);
            }
#pragma unroll
            for (int nt = 0; nt < kAttMaxNT; ++nt)
              if (nt < NT) mma_bf16(dg[m][nt], a, b0[nt], b1[nt]);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kAttMaxMT; ++m)
#pragma unroll
        for (int nt = 0; nt < kAttMaxNT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[m][nt][i] = fmaf(acc[m][nt][i], cr[nt], dg[m][nt][i]);
    }
    // the next slot's scores and probabilities are written only after the barrier that
    // follows its score pass, which every warp reaches after these reads
    ring_release(rg, g);
  }
  // head sums of the term columns -> stage [h][dim]
#pragma unroll
  for (int m = 0; m < kAttMaxMT; ++m) {
    const int mt = warp + m * kCW;
#pragma unroll
    for (int nt = 0; nt < kAttMaxNT; ++nt) {
      float v0 = acc[m][nt][0] + acc[m][nt][1], v1 = acc[m][nt][2] + acc[m][nt][3];
      v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
      v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
      const int h = (nt * 8 + 2 * ti) >> 2;
      if (mt < MT && nt < NT && (ti & 1) == 0 && h < nh) {
        stage[h * d + mt * 16 + gi] = v0;
        stage[h * d + mt * 16 + gi + 8] = v1;
      }
    }
  }
  if (tid < nh) {
    stage[nh * d + 2 * tid] = red[48 + tid];
    stage[nh * d + 2 * tid + 1] = red[64 + tid];
  }
  cbar();
  return g;
}

// Logits of the rows of this CTA's selected centroids [slo, shi) (contiguous blocks of the
// cluster-ordered embedding copy) against y; each warp's best (value, id) key goes to lk.
__device__ __forceinline__ void gather_best(const bf16* temb_ord, const int* ord, int H, int vsc, int nclust, const int* selc,
                                         int slo, int shi, const float* y, unsigned long long* lk) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // request every candidate block (vsc rows of H bf16, and its vsc ids) from memory at once
  if (threadIdx.x < shi - slo) {
    const size_t base = static_cast<size_t>(min(max(selc[slo + threadIdx.x], 0), nclust - 1)) * vsc;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(temb_ord + base * H),
                 "r"(static_cast<unsigned>(vsc * H * 2))
                 : "memory");
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ord + base), "r"(static_cast<unsigned>(vsc * 4))
                 : "memory");
  }
  unsigned long long best = 0ull;
  for (int c = slo; c < shi; ++c) {
    // selc entries are clamped where written, but a rank slot left unwritten (only possible
    // after an aborted exchange) must not address memory either
    const size_t base = static_cast<size_t>(min(max(selc[c], 0), nclust - 1)) * vsc;
    for (int jb = warp * 8; jb < vsc; jb += kCW * 8) {
      const int myrow = jb + (lane >> 2);  // the row this lane holds after the reduction
      const int id = myrow < vsc ? __ldg(ord + base + myrow) : 0;
      float a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = 0.f;
      for (int k = lane * 8; k < H; k += 256) {
        uint4 raw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          raw[i] = __ldcs(reinterpret_cast<const uint4*>(temb_ord + (base + min(jb + i, vsc - 1)) * H + k));
        const float4 ya = *reinterpret_cast<const float4*>(y + k);
        const float4 yb = *reinterpret_cast<const float4*>(y + k + 4);
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = dot8(raw[i], ya, yb, a[i]);
      }
      const float v = xreduce<8>(a, lane);
      if ((lane & 3) == 0 && myrow < vsc) {
        const unsigned long long key = argmax_key(v, id);
        best = key > best ? key : best;
      }
    }
  }
  best = warp_max_u64(best);
  if (lane == 0) lk[warp] = best;
}

// Global top-k of kNC sorted (descending) lists of k <= 64 distinct keys, by a tree of pairwise
// merges (16 -> 8 -> 4 -> 2 -> 1 lists, one warp per merge, a named barrier between levels).
// In a merge of lists A and B, A[i] lands at i + #{B > A[i]} and B[j] at j + #{A > B[j]}
// (binary searches); only positions < k are kept. Level inputs and outputs alternate between
// two scratch areas; the last level writes the selected centroid ids to selc.
__device__ __forceinline__ int count_greater(const unsigned long long* L, int k, unsigned long long e) {
  int pos = 0;
  for (int step = 64; step > 0; step >>= 1)  // k <= 64
    if (pos + step <= k && L[pos + step - 1] > e) pos += step;
  return pos;
}
__device__ __forceinline__ void merge_tree(const unsigned* lists, int k, int C, unsigned long long* buf_a,
                                        unsigned long long* buf_b, int* selc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // level 0: word-pair lists -> buf_a as 64-bit keys
  for (int i = threadIdx.x; i < kNC * k; i += kCT)
    buf_a[i] = (static_cast<unsigned long long>(lists[2 * i]) << 32) | lists[2 * i + 1];
  cbar();
  unsigned long long* in = buf_a;
  unsigned long long* out = buf_b;
  for (int n = kNC; n > 1; n >>= 1) {
    for (int m = warp; m < n / 2; m += kCW) {
      const unsigned long long* A = in + (2 * m) * k;
      const unsigned long long* B = in + (2 * m + 1) * k;
      for (int i = lane; i < k; i += 32) {
        const unsigned long long ea = A[i], eb = B[i];
        const int pa = i + count_greater(B, k, ea), pb = i + count_greater(A, k, eb);
        if (n > 2) {
          if (pa < k) out[m * k + pa] = ea;
          if (pb < k) out[m * k + pb] = eb;
        } else {
          if (pa < k) selc[pa] = min(max(key_id(ea), 0), C - 1);
          if (pb < k) selc[pb] = min(max(key_id(eb), 0), C - 1);
        }
      }
    }
    cbar();
    unsigned long long* t = in;
    in = out;
    out = t;
  }
}

// ------------------------------------------------------------------ the kernel

__global__ void __launch_bounds__(kT, 1) k_block_cl(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) char sm[];
  const Layout L = make_layout(p);
  unsigned rank_u;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank_u));
  const int r = static_cast<int>(rank_u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(sm + L.bars);
  const unsigned full0 = sa(bars), empty0 = sa(bars + kSlots), xbar0 = sa(bars + 2 * kSlots);
  const unsigned ring0 = sa(sm + L.ring);
  // receive buffers: set 1 directly follows set 0
  float* const xb0 = reinterpret_cast<float*>(sm + L.xch0);
  const unsigned xba0 = sa(sm + L.xch0);
  float* u = reinterpret_cast<float*>(sm + L.u);
  float* x = reinterpret_cast<float*>(sm + L.x);
  float* a = reinterpret_cast<float*>(sm + L.a);
  float* rowsb = reinterpret_cast<float*>(sm + L.rows);
  float* gtb = reinterpret_cast<float*>(sm + L.gt);
  float* utb = reinterpret_cast<float*>(sm + L.ut);
  float* part = reinterpret_cast<float*>(sm + L.part);
  bf16* xt = reinterpret_cast<bf16*>(sm + L.xt);
  float* sc = reinterpret_cast<float*>(sm + L.sc);
  float* red = reinterpret_cast<float*>(sm + L.red);
  float2* cs = reinterpret_cast<float2*>(sm + L.cs);
  unsigned long long* lk = reinterpret_cast<unsigned long long*>(sm + L.lk);
  int* selc = reinterpret_cast<int*>(sm + L.ids);
  Sec* tab = reinterpret_cast<Sec*>(sm + L.tab);
  float* nrm = reinterpret_cast<float*>(sm + L.nrm);
  const Fail fl{p.status, p.abort_flag, p.spin_limit};

  // this CTA's keys: a contiguous share of the full layers' [0, L) and of the window
  Keys kr{0, 0, 0, 0};
  {
    const int Lf = p.has_type[1] ? min(max(p.ctx_len[1][0], 0), p.kv_max[1]) : 0;
    const int Ls = p.has_type[0] ? min(max(p.ctx_len[0][0], 0), p.kv_max[0]) : 0;
    const int ws_lo = max(0, Ls - p.W);
    const Range f = split(Lf, kNC, r), s = split(Ls - ws_lo, kNC, r);
    kr = Keys{f.lo, f.hi - f.lo, ws_lo + s.lo, s.hi - s.lo};
  }

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kCW);
    }
    mbar_init(xbar0, 1);  // receive barriers: the local expect_tx arrival + the bytes of the peers
    mbar_init(xbar0 + 8, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // RoPE (cos, sin) at the block's position: the angle pos * theta^(-2i/d) in fp64, reduced
  // mod 2 pi, then fp32 sin / cos
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
      cs[(t ? L.cs_off1 : 0) + i] = v;
    }
  }
  for (int i = tid; i < 64; i += kT) selc[i] = 0;
  // this CTA's stream sections, and every norm gain, once per launch
  const int nsec = sec_count(p);
  for (int i = tid; i < nsec; i += kT) tab[i] = make_sec(p, i, r, kr);
  for (int l = 0; l < p.nl; ++l) {
    float* nl_ = nrm + l * L.nrm_stride;
    const int d = p.d[p.ltype[l]];
    for (int i = tid; i < p.H; i += kT) {
      nl_[i] = __ldg(p.attn_norm[l] + i);
      nl_[p.H + i] = __ldg(p.post_attn_norm[l] + i);
      nl_[2 * p.H + i] = __ldg(p.ffn_norm[l] + i);
      nl_[3 * p.H + i] = __ldg(p.post_ffn_norm[l] + i);
    }
    for (int i = tid; i < d; i += kT) nl_[4 * p.H + i] = __ldg(p.q_norm[l] + i);
  }
  for (int i = tid; i < p.H; i += kT) nrm[p.nl * L.nrm_stride + i] = __ldg(p.out_norm + i);
  // every barrier of the cluster is initialised before any CTA arrives on a peer's (this
  // also orders the tables above before their first use)
  cluster_sync_all();

  if (warp == kCW) {
    // ====================== producer warp: stream every section of every step in order
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int step = 0; step < p.n_draft && ok; ++step) {
        for (int si = 0; si < nsec && ok; ++si) {
          const Sec s = tab[si];
          const int nc = n_chunks(s);
          for (int ch = 0; ch < nc; ++ch) {
            const int slot = g % kSlots;
            if (g >= kSlots && !wait_bar(fl, empty0 + 8 * slot, static_cast<unsigned>((g / kSlots - 1) & 1), false)) {
              ok = false;
              break;
            }
            const int r0 = ch * s.rpc, n = min(s.rpc, s.nrows - r0);
            const unsigned bytes = static_cast<unsigned>(n * s.row_bytes);
            const unsigned fb = full0 + 8 * slot, dst = ring0 + slot * kSlotStride;
            mbar_expect_tx(fb, bytes);
            if (s.stride == s.row_bytes && s.pitch == s.row_bytes) {
              bulk_g2s(dst, s.src + static_cast<size_t>(r0) * s.row_bytes, bytes, fb);
            } else {
              for (int j = 0; j < n; ++j)
                bulk_g2s(dst + j * s.pitch, s.src + static_cast<size_t>(r0 + j) * s.stride,
                         static_cast<unsigned>(s.row_bytes), fb);
            }
            ++g;
          }
        }
      }
      // no copy of this CTA may still be in flight when it ends
      for (int h = (g > kSlots ? g - kSlots : 0); h < g; ++h)
        drain_bar(fl, full0 + 8 * (h % kSlots), static_cast<unsigned>((h / kSlots) & 1));
    }
    __syncwarp();
  } else {
    // ====================== compute warps
    const Ring rg{ring0, full0, empty0, fl};
    const bool amma = att_mma_ok(p);  // tensor-core attention (K rows at a padded pitch)
    int gc = 0;  // chunks consumed
    int xe = 0;  // exchanges done: buffer xe & 1, phase parity (xe >> 1) & 1
    const int H = p.H;

    // Exchange protocol. Each exchange uses receive buffer xe & 1 and its mbarrier (phase
    // parity (xe >> 1) & 1). The receiver arms the barrier with the number of bytes it will get
    // (one local arrival); warp w % kCW of every CTA writes that CTA's payload for CTA w with
    // st.async, whose bytes complete on CTA w's barrier. A buffer is rewritten only two
    // exchanges later, which no CTA can start before every CTA has sent the exchange in
    // between, i.e. has finished reading this one (a named barrier separates every last read
    // from the next send).
    // After a failed exchange wait a thread neither arms nor sends any more: a barrier must not
    // get a second arrival in an unfinished phase, nor unbounded bytes without an arm.
    bool live = true;
    auto xch_arm = [&](int nfloats) {
      if (tid == 0 && live) mbar_expect_tx(xbar0 + 8 * (xe & 1), 4u * static_cast<unsigned>(nfloats));
    };
    auto xch_dst = [&](int w) { return mapa(xba0 + (xe & 1) * (kXchFloats * 4), w); };
    auto xch_bar = [&](int w) { return mapa(xbar0 + 8 * (xe & 1), w); };
    // The named barrier first: a warp past its receive wait must not overwrite the staged
    // slice a sibling warp is still sending (the wait only covers this CTA's incoming data).
    bool bulk_sent = false;  // this thread issued bulk copies not yet known to have read their source
    auto xch_wait = [&]() -> float* {
      const int cur = xe & 1;
      if (bulk_sent) {  // the sources may be rewritten after the barrier
        bulk_wait_read();
        bulk_sent = false;
      }
      cbar();
      if (live && !wait_bar(fl, xbar0 + 8 * cur, static_cast<unsigned>((xe >> 1) & 1), true)) live = false;
      ++xe;
      return xb0 + cur * kXchFloats;
    };
    // Start of a send: every thread's writes of the payloads become visible to the bulk
    // copies (proxy fence, then the barrier), and every earlier read of the receive buffer
    // that the coming exchanges may rewrite is ordered before them.
    auto send_begin = [&]() {
      fence_async_smem();
      cbar();
    };
    // This warp's part of sending n floats of src (this CTA's shared memory) to float offset
    // off of peer w2's receive buffer: one bulk copy when both ends are 16-byte aligned and the
    // size is a multiple of 16 bytes, else 4-byte st.async stores by the lanes.
    auto send = [&](int w2, int off, const float* src, int n) {
      if (n <= 0) return;
      const unsigned dst = xch_dst(w2) + 4u * static_cast<unsigned>(off), rb = xch_bar(w2), sp = sa(src);
      if (((dst | sp) & 15u) == 0 && (n & 3) == 0) {
        if (lane == 0) {
          bulk_s2c(dst, sp, 4u * static_cast<unsigned>(n), rb);
          bulk_sent = true;
        }
      } else {
        for (int i = lane; i < n; i += 32) st_async_f32(dst + 4u * i, src[i], rb);
      }
    };
    // all-gather of a vector of `total` floats: every CTA receives this CTA's slice [lo, hi)
    // (held in src from index 0)
    auto all_gather = [&](int lo, int hi, const float* src, int total) -> float* {
      xch_arm(total);
      send_begin();
      for (int w2 = warp; w2 < kNC && live; w2 += kCW) send(w2, lo, src, hi - lo);
      return xch_wait();
    };
    auto sec = [&](int idx) { return tab[idx]; };

    int tok = 0;
    for (int step = 0; step < p.n_draft; ++step) {
      // ================= PRE: x0 = W_pre [h ; embed(token)]
      {
        if (step == 0) {
          tok = p.tok_in[0];
          for (int i = tid * 8; i < p.bb; i += kCT * 8) load_vec(p.hidden_in + i, u + i);
        }
        if (tok < 0 || tok >= p.V) {
          if (r == 0 && tid == 0) set_status(p.status, MTP_ERR_INVALID_ARG);
          tok = 0;
        }
        const bf16* er = p.tgt + static_cast<size_t>(tok) * p.bb;
        for (int i = tid * 8; i < p.bb; i += kCT * 8) load_vec(er + i, u + p.bb + i);
        cbar();
        gc = gemv_sec(rg, gc, sec(0), u, rowsb, part);
        const Range rg0 = split(H, kNC, r);
        const float* xg = all_gather(rg0.lo, rg0.hi, rowsb, H);
        for (int i = tid; i < H; i += kCT) x[i] = xg[i];
        cbar();
      }
      // ================= decoder blocks
      for (int l = 0; l < p.nl; ++l) {
        const int lt = p.ltype[l], d = p.d[lt], QD = p.nh * d;
        const Range hr = split(H, kNC, r);
        // ---- Q rows of attn_norm(x)
        {
          const float rf = rms_inv(x, H, p.eps);
          for (int i = tid; i < H; i += kCT) a[i] = x[i] * rf * nrm[l * L.nrm_stride + i];
          cbar();
          if (p.mma) {
            split_terms(a, H, xt);
            cbar();
            gc = gemv_mma_sec(rg, gc, sec(1 + 6 * l), xt, rowsb, part);
          } else {
            gc = gemv_sec(rg, gc, sec(1 + 6 * l), a, rowsb, part);
          }
        }
        const Range qr = split(QD, kNC, r);
        float* q = all_gather(qr.lo, qr.hi, rowsb, QD);
        // ---- q_norm + RoPE in place (the receive buffer stays ours until the next-but-one exchange)
        {
          if (warp < p.nh) {
            float s = 0.f;
            for (int i = lane * 4; i < d; i += 128) {
              const float4 v = *reinterpret_cast<const float4*>(q + warp * d + i);
              s += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            }
            s = warp_sum(s);
            if (lane == 0) red[32 + warp] = rsqrtf(s / d + p.eps);
          }
          if (tid < p.nh) {  // running max and exp-sum of every head
            red[48 + tid] = -INFINITY;
            red[64 + tid] = 0.f;
          }
          cbar();
          const float2* c2 = cs + (lt ? L.cs_off1 : 0);
          const float* gq = nrm + l * L.nrm_stride + 4 * H;
          const int half = d / 2;
          if (amma) {
            // rotated pairs (h, i), at most 4 per thread, then three bf16 terms per value into
            // rows 3h + t of the same buffer (pitch d + 8) once every thread has read its pairs
            float va[4], vb[4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
              const int idx = tid + k2 * kCT;
              va[k2] = vb[k2] = 0.f;
              if (idx < p.nh * half) {
                const int h = idx / half, i = idx % half;
                const float rfq = red[32 + h];
                const float av = q[h * d + i] * rfq * gq[i];
                const float bv = q[h * d + i + half] * rfq * gq[i + half];
                va[k2] = av * c2[i].x - bv * c2[i].y;
                vb[k2] = bv * c2[i].x + av * c2[i].y;
              }
            }
            cbar();
            bf16* qt = reinterpret_cast<bf16*>(q);
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
              const int idx = tid + k2 * kCT;
              if (idx < p.nh * half) {
                const int h = idx / half, i = idx % half;
                put_terms(qt + 3 * h * (d + 8) + i, d + 8, va[k2]);
                put_terms(qt + 3 * h * (d + 8) + i + half, d + 8, vb[k2]);
              }
            }
          } else {
            for (int idx = tid; idx < p.nh * half; idx += kCT) {
              const int h = idx / half, i = idx % half;
              const float rfq = red[32 + h];
              const float av = q[h * d + i] * rfq * gq[i];
              const float bv = q[h * d + i + half] * rfq * gq[i + half];
              q[h * d + i] = av * c2[i].x - bv * c2[i].y;
              q[h * d + i + half] = bv * c2[i].x + av * c2[i].y;
            }
          }
          cbar();
        }
        // ---- attention over this CTA's keys
        {
          const Sec s = sec(2 + 6 * l);
          const int hpg = p.nh / p.nkv;
          if (amma)
            gc = att_sec_mma(p.nh, rg, gc, s, d, p.scale[lt], reinterpret_cast<const bf16*>(q), sc,
                             reinterpret_cast<bf16*>(part), red, rowsb);
          else if (hpg % 4 == 0) gc = att_sec<4>(p.nh, p.nkv, rg, gc, s, d, p.scale[lt], q, sc, red, rowsb);
          else if (hpg == 2) gc = att_sec<2>(p.nh, p.nkv, rg, gc, s, d, p.scale[lt], q, sc, red, rowsb);
          else gc = att_sec<1>(p.nh, p.nkv, rg, gc, s, d, p.scale[lt], q, sc, red, rowsb);
        }
        // ---- partials to the owner of each output dim: CTA w receives, from every CTA r,
        // [m_0 l_0 .. m_nh-1 l_nh-1 | r's sums of w's dims] at offset r * per
        const int per = 2 * p.nh + split_max(QD, kNC);
        const Range dr = split(QD, kNC, r);
        xch_arm(kNC * (2 * p.nh + (dr.hi - dr.lo)));
        send_begin();
        for (int w2 = warp; w2 < kNC && live; w2 += kCW) {
          const Range dw = split(QD, kNC, w2);
          send(w2, r * per, rowsb + QD, 2 * p.nh);
          send(w2, r * per + 2 * p.nh, rowsb + dw.lo, dw.hi - dw.lo);
        }
        const float* pb = xch_wait();
        // ---- combine this CTA's dims: per head, the weight of every source's partial sums
        // exp(m_s - M) / sum_s' exp(m_s' - M) l_s'; then one thread per dim
        // (one thread per (head, source): kNC consecutive lanes share a head)
        float* wgt = sc;  // [nh][kNC]
        static_assert(32 % kNC == 0, "a head's sources lie inside one warp");
        if (tid < (p.nh * kNC + 31) / 32 * 32) {  // whole warps (the shuffles need every lane)
          const int h = tid / kNC, s2 = tid % kNC;
          const bool on = h < p.nh;
          const float m_s = on ? pb[s2 * per + 2 * h] : -INFINITY;
          float M = m_s;
#pragma unroll
          for (int o = 1; o < kNC; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
          const float e = M == -INFINITY ? 0.f : expf(m_s - M);
          float den = on ? e * pb[s2 * per + 2 * h + 1] : 0.f;
#pragma unroll
          for (int o = 1; o < kNC; o <<= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
          if (on) wgt[h * kNC + s2] = den > 0.f ? e * (1.f / den) : 0.f;
        }
        cbar();
        for (int fi = tid; fi < dr.hi - dr.lo; fi += kCT) {
          const float* wh = wgt + ((dr.lo + fi) / d) * kNC;
          float v = 0.f;
          for (int s2 = 0; s2 < kNC; ++s2) v = fmaf(wh[s2], pb[s2 * per + 2 * p.nh + fi], v);
          rowsb[fi] = v;
        }
        cbar();
        const float* o = all_gather(dr.lo, dr.hi, rowsb, QD);
        // ---- O rows, residual with post_attn_norm, ffn_norm
        gc = gemv_sec(rg, gc, sec(3 + 6 * l), o, rowsb, part);
        const float* op = all_gather(hr.lo, hr.hi, rowsb, H);
        {
          const float rf = rms_inv(op, H, p.eps);
          for (int i = tid; i < H; i += kCT) x[i] = x[i] + op[i] * rf * nrm[l * L.nrm_stride + H + i];
          cbar();
          const float rf2 = rms_inv(x, H, p.eps);
          for (int i = tid; i < H; i += kCT) a[i] = x[i] * rf2 * nrm[l * L.nrm_stride + 2 * H + i];
          cbar();
        }
        // ---- MLP: gate / up rows, m = gelu_tanh(gate) * up, down rows
        if (p.mma) {
          split_terms(a, H, xt);
          cbar();
          gc = gemv_mma_sec(rg, gc, sec(4 + 6 * l), xt, gtb, part);
          gc = gemv_mma_sec(rg, gc, sec(5 + 6 * l), xt, utb, part);
        } else {
          gc = gemv_sec(rg, gc, sec(4 + 6 * l), a, gtb, part);
          gc = gemv_sec(rg, gc, sec(5 + 6 * l), a, utb, part);
        }
        const Range fr = split(p.F, kNC, r);
        for (int i = tid; i < fr.hi - fr.lo; i += kCT) rowsb[i] = gelu_tanh(gtb[i]) * utb[i];
        cbar();
        const float* mv = all_gather(fr.lo, fr.hi, rowsb, p.F);
        gc = gemv_sec(rg, gc, sec(6 + 6 * l), mv, rowsb, part);
        const float* dn = all_gather(hr.lo, hr.hi, rowsb, H);
        {
          const float rf = rms_inv(dn, H, p.eps);
          for (int i = tid; i < H; i += kCT)
            x[i] = p.lambda[l] * (x[i] + dn[i] * rf * nrm[l * L.nrm_stride + 3 * H + i]);
          cbar();
        }
      }
      // ================= HEAD
      const int k = p.topk;
      {
        const float rf = rms_inv(x, H, p.eps);
        for (int i = tid; i < H; i += kCT) a[i] = x[i] * rf * nrm[p.nl * L.nrm_stride + i];  // a = y
        cbar();
      }
      // centroid logits of this CTA's centroids -> local top-k (warp 0)
      if (p.mma) {
        split_terms(a, H, xt);
        cbar();
        gc = gemv_mma_sec(rg, gc, sec(1 + 6 * p.nl), xt, gtb, part);
      } else {
        gc = gemv_sec(rg, gc, sec(1 + 6 * p.nl), a, gtb, part);
      }
      {
        // local top-k by rank: key i goes to position #{j : key_j > key_i} when that is < k
        const Range cr = split(p.C, kNC, r);
        const int nce = cr.hi - cr.lo;
        unsigned long long* ck = reinterpret_cast<unsigned long long*>(sc);
        for (int i = tid; i < nce; i += kCT) ck[i] = argmax_key(gtb[i], cr.lo + i);
        cbar();
        // two threads per key, each counting over half of the keys
        for (int base = 0; base < nce; base += kCT / 2) {  // warp-uniform trip count
          const int i = base + (tid >> 1), ic = min(i, nce - 1);
          const unsigned long long key = ck[ic];
          const int half = tid & 1, jlo = half * (nce / 2), jhi = half ? nce : nce / 2;
          int rank = 0;
          for (int j = jlo; j < jhi; ++j) rank += ck[j] > key ? 1 : 0;
          rank += __shfl_xor_sync(0xffffffffu, rank, 1);
          if (half == 0 && i < nce && rank < k) lk[rank] = key;
        }
      }
      // post rows -> this CTA's slice of h' (output, and the next step's input)
      if (p.mma) gc = gemv_mma_sec(rg, gc, sec(2 + 6 * p.nl), xt, rowsb, part);
      else gc = gemv_sec(rg, gc, sec(2 + 6 * p.nl), a, rowsb, part);
      const Range br = split(p.bb, kNC, r);
      if (p.out_hidden)
        for (int i = tid; i < br.hi - br.lo; i += kCT) p.out_hidden[static_cast<size_t>(step) * p.bb + br.lo + i] = rowsb[i];
      for (int i = tid; i < k; i += kCT) {
        gtb[2 * i] = __uint_as_float(static_cast<unsigned>(lk[i] >> 32));
        gtb[2 * i + 1] = __uint_as_float(static_cast<unsigned>(lk[i]));
      }
      cbar();
      // exchange: every CTA receives [h' (bb floats) | kNC local top-k lists of 2k words]
      xch_arm(p.bb + kNC * 2 * k);
      send_begin();
      for (int w2 = warp; w2 < kNC && live; w2 += kCW) {
        send(w2, br.lo, rowsb, br.hi - br.lo);
        send(w2, p.bb + r * 2 * k, gtb, 2 * k);
      }
      const float* hx = xch_wait();
      for (int i = tid; i < p.bb; i += kCT) u[i] = hx[i];
      // global top-k: tree merge of the kNC sorted lists (scratch: the score buffer, and the
      // received lists' own area once level 1 has read them)
      merge_tree(reinterpret_cast<const unsigned*>(hx + p.bb), k, p.C, reinterpret_cast<unsigned long long*>(sc),
                 reinterpret_cast<unsigned long long*>(const_cast<float*>(hx) + p.bb), selc);
      // ---- logits of this CTA's share of the candidate rows -> best key per warp
      {
        const Range sr = split(k, kNC, r);
        gather_best(p.temb_ord, p.ord, p.H, p.vsc, p.C, selc, sr.lo, sr.hi, a, lk);
      }
      cbar();
      if (warp == 0) {
        unsigned long long m = lane < kCW ? lk[lane] : 0ull;
        m = warp_max_u64(m);
        if (lane == 0) {
          gtb[0] = __uint_as_float(static_cast<unsigned>(m >> 32));
          gtb[1] = __uint_as_float(static_cast<unsigned>(m));
        }
        if (m != 0ull) {  // warm L2 with the embedding row of this CTA's best token
          const int id = min(max(key_id(m), 0), p.V - 1);
          const char* er = reinterpret_cast<const char*>(p.tgt + static_cast<size_t>(id) * p.bb);
          for (int off = lane * 128; off < p.bb * 2; off += 32 * 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(er + off));
        }
      }
      cbar();
      const float* kx = all_gather(2 * r, 2 * r + 2, gtb, 2 * kNC);
      unsigned long long m = 0ull;
      for (int i = 0; i < kNC; ++i) {
        const unsigned long long kv = (static_cast<unsigned long long>(__float_as_uint(kx[2 * i])) << 32) |
                                      __float_as_uint(kx[2 * i + 1]);
        m = kv > m ? kv : m;
      }
      tok = min(max(key_id(m), 0), p.V - 1);
      if (r == 0 && tid == 0) p.out_tokens[step] = tok;
      cbar();
    }
  }
  // no CTA leaves while a peer may still write into its shared memory
  cluster_sync_all();
}

}  // namespace clk

// Host: shared-memory bytes of the cluster kernel for these parameters, or 0 when the shape
// is outside the kernel's limits.
int cl_smem_bytes(const clk::Params& p) {
  using namespace clk;
  if (p.nl < 1 || p.nl > kMaxL) return 0;
  int dmax = 0;
  for (int l = 0; l < p.nl; ++l) {
    const int d = p.d[p.ltype[l]];
    if (d < 8 || d % 8) return 0;
    dmax = d > dmax ? d : dmax;
  }
  const int per = 2 * p.nh + split_max(p.nh * dmax, kNC);
  // weighted-sum slots (head groups x dim quads) must fit the compute threads
  const int hpg = p.nkv > 0 ? p.nh / p.nkv : 0;
  const int nht = hpg % 4 == 0 ? 4 : (hpg == 2 ? 2 : 1);
  if (hpg < 1 || p.nkv * (hpg / nht) * (dmax / 4) > kCT) return 0;
  const bool fits =
      p.H % 8 == 0 && p.bb % 8 == 0 && p.F % 8 == 0 && p.H >= 8 &&  // 16-byte rows and vector loads
      p.nh >= 1 && p.nh <= 16 && p.nkv >= 1 && p.nh % p.nkv == 0 &&
      p.nh * dmax <= kXchFloats && kNC * per <= kXchFloats && p.F <= kXchFloats && p.H <= kXchFloats &&
      p.bb + kNC * 2 * p.topk <= kXchFloats && 2 * kNC <= kXchFloats &&
      2 * p.bb * 2 <= kSlotBytes && p.H * 2 <= kSlotBytes && p.F * 2 <= kSlotBytes &&
      p.nh * dmax * 2 <= kSlotBytes && p.nkv * dmax * 2 <= kSlotBytes &&
      p.topk >= 1 && p.topk <= 64 && p.C >= kNC && split_max(p.C, kNC) <= 128 && p.topk <= p.C / kNC &&
      p.vsc > 0 && static_cast<long long>(p.C) * p.vsc == p.V;
  if (!fits) return 0;
  return make_layout(p).total;
}

int run_cl(const clk::Params& p, int smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(clk::k_block_cl, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(clk::k_block_cl, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) {
    set_error("cluster kernel attributes: %s", cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clk::kNC);
  cfg.blockDim = dim3(clk::kT);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = clk::kNC;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, clk::k_block_cl, p);
  if (e != cudaSuccess) {
    set_error("cluster draft-block launch (%d CTAs, %d B shared memory): %s", clk::kNC, smem, cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

// Number of kNC-CTA clusters of this kernel that can be resident at once (0: none).
int cl_capacity(int smem) {
  if (cudaFuncSetAttribute(clk::k_block_cl, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(clk::k_block_cl, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clk::kNC);
  cfg.blockDim = dim3(clk::kT);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = clk::kNC;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<void*>(clk::k_block_cl), &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// dst[j] = src[ord[j]] for the V rows of row_bytes bytes (a multiple of 16): token_embd in
// token_ordering order, so that the rows of one centroid are one contiguous block.
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

// Packs W [R][K] (bf16, row-major) for the cluster kernel's tensor-core GEMVs: per CTA r of
// the cluster its rows split(R, kNC, r), padded with zero rows to a multiple of 16, as 16x16
// tiles (row tile major) of 32 lanes x 16 bytes in mma.m16n8k16 A-fragment order: lane
// (g = lane / 4, t = lane % 4) holds rows g and g + 8 at columns 2t, 2t + 1 and 2t + 8, 2t + 9.
__global__ void k_pack_tiles(const __nv_bfloat16* __restrict__ W, int R, int K, uint4* __restrict__ dst) {
  const int KT = K / 16;
  long long total = 0;
  for (int r = 0; r < clk::kNC; ++r) total += static_cast<long long>(clk::padded_rows(R, r) / 16) * KT * 32;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    // locate the CTA block, tile and lane of entry i
    long long rem = i;
    int r = 0;
    for (; r < clk::kNC; ++r) {
      const long long n = static_cast<long long>(clk::padded_rows(R, r) / 16) * KT * 32;
      if (rem < n) break;
      rem -= n;
    }
    const int lane = static_cast<int>(rem % 32), tile = static_cast<int>(rem / 32);
    const int rt = tile / KT, kt = tile % KT, g = lane >> 2, t = lane & 3;
    const clk::Range rg = clk::split(R, clk::kNC, r);
    auto word = [&](int row, int col) -> uint32_t {
      const int gr = rg.lo + rt * 16 + row;
      if (gr >= rg.hi) return 0u;
      const uint16_t* p = reinterpret_cast<const uint16_t*>(W + static_cast<size_t>(gr) * K + kt * 16 + col);
      return static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 16);
    };
    dst[i] = make_uint4(word(g, 2 * t), word(g + 8, 2 * t), word(g, 2 * t + 8), word(g + 8, 2 * t + 8));
  }
}

long long packed_tile_bytes(int R, int K) { return clk::tiles_before(R, K, clk::kNC) * clk::kTileBytes; }

int pack_tiles(const void* W, int R, int K, void* dst, cudaStream_t st) {
  k_pack_tiles<<<512, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(W), R, K, static_cast<uint4*>(dst));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("packing weight tiles: %s", cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

}  // namespace mtp
