// Streamed-tile cluster draft block (B = 1): see mtp_c2.cuh for the data flow.
//
// Failure handling: every wait is bounded. A wait that gives up records MTP_ERR_TIMEOUT and
// raises the abort word; a raised abort word makes every later wait give up after a few
// polls. Control flow never depends on a wait's outcome, so every thread executes the same
// sequence of named barriers and ring releases; a thread whose wait failed stops arming and
// sending. Values derived from exchanged data (centroid ids, token ids) are clamped before
// they address memory. Before the CTA ends, its producer waits (time-bounded) for its own
// copies still in flight, and a final cluster barrier keeps every CTA alive while a peer may
// still write into it.
#include <cmath>
#include <cstring>

#include "mtp_c2.cuh"
#include "mtp_launch.h"

namespace mtp {
namespace c2 {

// ------------------------------------------------------------------ primitives

__device__ __forceinline__ unsigned sa(const void* p) { return static_cast<unsigned>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ unsigned mapa(unsigned addr, int rank) {
  unsigned r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Asynchronous stores into a peer CTA's shared memory whose bytes complete on the peer's
// mbarrier (both addresses in the shared::cluster window).
__device__ __forceinline__ void st_async_u32(unsigned caddr, unsigned v, unsigned cbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(caddr), "r"(v),
               "r"(cbar)
               : "memory");
}
__device__ __forceinline__ void st_async_u64(unsigned caddr, unsigned long long v, unsigned cbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(caddr), "l"(v),
               "r"(cbar)
               : "memory");
}
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
// A waiting thread is suspended until the phase completes or this many ns pass.
constexpr unsigned kSuspendNs = 100000;
__device__ __forceinline__ bool try_wait_cta(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}
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
__device__ __forceinline__ uint4 lds128(unsigned a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(unsigned a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 ldsm_x4(unsigned addr) {
  uint4 r;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}
__device__ __forceinline__ uint4 ldsm_x4_t(unsigned addr) {
  uint4 r;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}
// D += A (16x16 bf16, row) x B (16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
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
// Bounded wait on an mbarrier phase: false when the abort word is raised or the time limit
// passes (which records MTP_ERR_TIMEOUT and raises the abort word).
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

// RMSNorm factor 1/sqrt(mean(v^2) + eps) of a shared-memory vector, computed by every warp
// in the same order (all threads get the same value without a barrier).
__device__ __forceinline__ float rms_inv(const float* v, int n, float eps) {
  const int lane = threadIdx.x & 31;
  float s = 0.f;
  for (int i = lane; i < n; i += 32) s = fmaf(v[i], v[i], s);
  s = warp_sum(s);
  return rsqrtf(s / n + eps);
}

// Three bf16 terms of v: hi = bf16(v), mid = bf16(v - hi), lo = bf16(v - hi - mid); their sum
// is v to fp32 precision and each product with a bf16 weight is exact in fp32.
__device__ __forceinline__ void split3(float v, uint32_t& h, uint32_t& m, uint32_t& l) {
  const bf16 bh = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(bh);
  const bf16 bm = __float2bfloat16_rn(r1);
  const bf16 bl = __float2bfloat16_rn(r1 - __bfloat162float(bm));
  h = __bfloat16_as_ushort(bh);
  m = __bfloat16_as_ushort(bm);
  l = __bfloat16_as_ushort(bl);
}
// The terms of v at rows 0, 1, 2 (pitch rs elements) of dst.
__device__ __forceinline__ void put3(bf16* dst, int rs, float v) {
  uint32_t h, m, l;
  split3(v, h, m, l);
  dst[0] = __ushort_as_bfloat16(static_cast<unsigned short>(h));
  dst[rs] = __ushort_as_bfloat16(static_cast<unsigned short>(m));
  dst[2 * rs] = __ushort_as_bfloat16(static_cast<unsigned short>(l));
}
// The terms of the pair (a, b) as three 32-bit words (a in the low half).
__device__ __forceinline__ uint3 terms2(float a, float b) {
  uint32_t ha, ma, la, hb, mb, lb;
  split3(a, ha, ma, la);
  split3(b, hb, mb, lb);
  return make_uint3(ha | (hb << 16), ma | (mb << 16), la | (lb << 16));
}

// Sends to every CTA of the cluster (this one included) at local shared address `addr`,
// counted on the barrier at local address `bar`.
__device__ __forceinline__ void bcast_u32(unsigned addr, unsigned bar, unsigned v) {
#pragma unroll 4
  for (int w = 0; w < kNC; ++w) st_async_u32(mapa(addr, w), v, mapa(bar, w));
}
__device__ __forceinline__ void bcast_f32(unsigned addr, unsigned bar, float v) { bcast_u32(addr, bar, __float_as_uint(v)); }
__device__ __forceinline__ void bcast_u64(unsigned addr, unsigned bar, unsigned long long v) {
#pragma unroll 4
  for (int w = 0; w < kNC; ++w) st_async_u64(mapa(addr, w), v, mapa(bar, w));
}
// The three term words of a pair, rows `pitch` bytes apart.
__device__ __forceinline__ void bcast3(unsigned addr, unsigned pitch, unsigned bar, uint3 t) {
#pragma unroll 2
  for (int w = 0; w < kNC; ++w) {
    const unsigned a = mapa(addr, w), b = mapa(bar, w);
    st_async_u32(a, t.x, b);
    st_async_u32(a + pitch, t.y, b);
    st_async_u32(a + 2 * pitch, t.z, b);
  }
}

// ------------------------------------------------------------------ ring (consumer side)

struct Ring {
  unsigned base, full0, empty0;
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

// ------------------------------------------------------------------ projections

// Partial row sums of a weight section: warp w < RT * P multiplies its 4 k tiles of every slot
// (A tiles straight from the slot, B = column c < 3 of term c of the input, read from xt with
// rows `xp` bytes apart; columns 3..7 are zero) into one accumulator, then writes its row
// tile's sums (the three term columns added) to part[(w / RT) * RT * 16 + row]. The caller
// adds the P parts after a barrier (sum_parts). Returns the slot counter after the section.
__device__ __forceinline__ int gemv2(Ring rg, int g, const SecE* se, unsigned xt, int xp, float* part) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, ti = lane & 3;
  const int RT = se->w.RT, P = se->w.P, KT = se->w.KT, nsl = se->w.nsl;
  const bool act = warp < RT * P;
  const int rt = act ? warp % RT : 0, pp = act ? warp / RT : 0;
  const int kt0 = pp * (KT / P);
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  const unsigned xb = xt + static_cast<unsigned>(gi * xp + 4 * ti);
  const bool bl = gi < 3;
  for (int s = 0; s < nsl; ++s, ++g) {
    const unsigned W = ring_wait(rg, g);
    if (act) {
      const unsigned a0 = W + static_cast<unsigned>(4 * warp * kTile + lane * 16);
      const unsigned b0a = xb + static_cast<unsigned>((kt0 + 4 * s) * 32);
      uint4 a[4];
      uint32_t b[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        a[j] = lds128(a0 + j * kTile);
        b[2 * j] = bl ? lds32(b0a + j * 32) : 0u;
        b[2 * j + 1] = bl ? lds32(b0a + j * 32 + 16) : 0u;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_bf16(d, a[j], b[2 * j], b[2 * j + 1]);
    }
    ring_release(rg, g);
  }
  if (act) {
    float v0 = d[0] + d[1], v1 = d[2] + d[3];
    v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
    v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
    if (ti == 0) {
      part[pp * RT * 16 + rt * 16 + gi] = v0;
      part[pp * RT * 16 + rt * 16 + gi + 8] = v1;
    }
  }
  return g;
}
// Row i of a section after gemv2 and a barrier: its P parts added in a fixed order.
__device__ __forceinline__ float sum_parts(const float* part, const SecE* se, int i) {
  const int RT = se->w.RT, P = se->w.P;
  float v = 0.f;
  for (int pp = 0; pp < P; ++pp) v += part[pp * RT * 16 + i];
  return v;
}

// ------------------------------------------------------------------ attention

// The bf16 pair of keys (key, key + 1) in v with keys at or past n set to zero.
__device__ __forceinline__ uint32_t keep_keys(uint32_t v, int key, int n) {
  return key + 1 < n ? v : (key < n ? (v & 0xffffu) : 0u);
}

// Attention of the nh query heads over this CTA's keys of one block, on tensor cores: K rows
// sit in the slots at pitch nkv * d bf16 + 16 bytes (kKps rows per slot); q is given as three
// bf16 terms per head (row 3h + t of qt, pitch (d + 8) elements). Column 4c + t of an MMA
// carries term t of head c of the KV group (t < 3; the fourth column is zero). The keys go in
// chunks of up to kSlots slots (16-key tile kt of a chunk is rows (kt % 2) * 16.. of its slot
// kt / 2); per chunk of n keys:
//   scores   S[key][col] = K q: tasks (group, key tile, dim part) over the warps, partial sums
//            per dim part to sp[part][key][head];
//   softmax  warp h adds the parts, updates the running max / exp-sum of head h over the
//            chunk and writes p as three bf16 terms (row 3h + t of pt, pitch kSlots kKps + 8);
//   sums     O^T[dim][col] += K^T P^T: warp tasks (group, 16-dim tile) over every key tile of
//            the chunk, rescaled once by the running-max correction; a slot is released as
//            soon as the warp has passed its key tiles.
// At the end, every unnormalised sum o[h][dim] goes to its owner (CTA (h d + dim) / dpo) at
// float offset r (2 + dpo) + 2 + (h d + dim) % dpo of the receive buffer xdst, and (m_h, l_h)
// to float offset r (2 + dpo) of every owner of head h's dims. Returns the slot counter.
// D_, NH_, NKV_ > 0 fix head_dim, heads and KV heads at compile time (0: the runtime values).
template <int D_, int NH_, int NKV_>
__device__ __forceinline__ int att3(Ring rg, int g, const SecE* se, int nh_rt, int nkv_rt, int d_rt, float scale,
                                 unsigned qt, float* sp, bf16* pt, float* red, unsigned xdst, unsigned xbar, int dpo,
                                 int r, bool live) {
  constexpr int CH = kSlots * kKps;  // keys per chunk
  const int d = D_ > 0 ? D_ : d_rt, nh = NH_ > 0 ? NH_ : nh_rt, nkv = NKV_ > 0 ? NKV_ : nkv_rt;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gi = lane >> 2, ti = lane & 3;
  const int hpg = nh / nkv, NT = (hpg + 1) / 2, KS = d / 16, MT = d / 16, QP = d + 8;
  constexpr int PP = CH + 8;
  const int P = nkv * d * 2 + 16, nkeys = se->nkeys;
  const unsigned pts = sa(pt);
  // per-lane constants: ldmatrix row offsets (scores: rows + k halves; sums: transposed), the
  // B rows of the two n tiles of every group
  const unsigned arow_s = static_cast<unsigned>(((lane & 7) + ((lane >> 3) & 1) * 8) * P + (lane >> 4) * 16);
  const unsigned arow_w = static_cast<unsigned>(((lane & 7) + (lane >> 4) * 8) * P + ((lane >> 3) & 1) * 16);
  auto brow = [&](int grp, int nt) -> int {
    const int c = nt * 8 + gi, hh = c >> 2, t = c & 3;
    return (t == 3 || hh >= hpg) ? -1 : 3 * (grp * hpg + hh) + t;
  };
  // weighted-sum tasks of this warp: A offset (group, dim tile) and B offsets per n tile
  unsigned woff[kAttMT];
  int wb[kAttMT][2];
  bool wact[kAttMT];
  float acc[kAttMT][2][4];
#pragma unroll
  for (int m = 0; m < kAttMT; ++m) {
    const int task = warp + m * kCW;
    wact[m] = task < nkv * MT;
    const int grp = wact[m] ? task / MT : 0, mt = wact[m] ? task % MT : 0;
    woff[m] = arow_w + static_cast<unsigned>(grp * d * 2 + mt * 32);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int rw = nt < NT ? brow(grp, nt) : -1;
      wb[m][nt] = rw >= 0 ? 2 * (rw * PP + 2 * ti) : -1;
      acc[m][nt][0] = acc[m][nt][1] = acc[m][nt][2] = acc[m][nt][3] = 0.f;
    }
  }
  if (tid < nh) {
    red[tid] = -INFINITY;
    red[16 + tid] = 0.f;
  }
  const int nslot = (nkeys + kKps - 1) / kKps;
  for (int c0 = 0; c0 < nslot; c0 += kSlots) {
    const int ns = min(kSlots, nslot - c0);
    const int n = min(CH, nkeys - c0 * kKps), nkt = (n + 15) / 16, KT16 = nkt * 16;
    for (int j = 0; j < ns; ++j) ring_wait(rg, g + j);
    // slot addresses of the chunk (slot gg of the ring at rg.base + (gg % kSlots) * stride)
    unsigned sbase[kSlots];
#pragma unroll
    for (int j = 0; j < kSlots; ++j) sbase[j] = rg.base + static_cast<unsigned>(((g + j) % kSlots) * kSlotStride);
    // ---- scores: dim parts DP (log2 ldp), the largest power of two with nkv nkt DP <= kCW
    // dividing d / 16
    int ldp = 0;
    while (nkv * nkt * (2 << ldp) <= kCW && KS % (2 << ldp) == 0) ++ldp;
    const int DP = 1 << ldp;
    if (warp < nkv * nkt * DP) {
      const int dpart = warp & (DP - 1), kq = warp >> ldp, kt = kq % nkt, grp = kq / nkt;
      const int nks = KS >> ldp, ks0 = dpart * nks;
      float sv[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) sv[nt][0] = sv[nt][1] = sv[nt][2] = sv[nt][3] = 0.f;
      unsigned sb = sbase[0];
#pragma unroll
      for (int j = 1; j < kSlots; ++j)
        if ((kt >> 1) == j) sb = sbase[j];
      unsigned a_addr = sb + static_cast<unsigned>((kt & 1) * 16 * P + grp * d * 2 + ks0 * 32) + arow_s;
      unsigned b_addr[2];
      bool bon[2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int rw = nt < NT ? brow(grp, nt) : -1;
        bon[nt] = rw >= 0;
        b_addr[nt] = qt + 2u * static_cast<unsigned>((bon[nt] ? rw : 0) * QP + ks0 * 16 + 2 * ti);
      }
      for (int ks = 0; ks < nks; ++ks) {
        const uint4 a = ldsm_x4(a_addr);
        a_addr += 32;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          if (nt < NT) {
            const uint32_t b0 = bon[nt] ? lds32(b_addr[nt]) : 0u;
            const uint32_t b1 = bon[nt] ? lds32(b_addr[nt] + 16) : 0u;
            b_addr[nt] += 32;
            mma_bf16(sv[nt], a, b0, b1);
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        if (nt < NT) {
          float v0 = sv[nt][0] + sv[nt][1], v1 = sv[nt][2] + sv[nt][3];
          v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
          v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
          const int hh = (nt * 8 + 2 * ti) >> 2;
          if ((ti & 1) == 0 && hh < hpg) {
            const int h = grp * hpg + hh;
            float* spp = sp + (dpart * KT16 + kt * 16 + gi) * nh + h;
            spp[0] = v0;
            spp[8 * nh] = v1;
          }
        }
      }
    }
    cbar();
    // ---- running max / exp-sum of head `warp` over the chunk; p as three bf16 terms
    if (warp < nh) {
      const int h = warp;
      float v[CH / 32];
      float cm = -INFINITY;
#pragma unroll
      for (int u = 0; u < CH / 32; ++u) {
        const int j = lane + 32 * u;
        v[u] = -INFINITY;
        if (j < n) {
          const float* spp = sp + j * nh + h;
          float s2 = 0.f;
          for (int dp = 0; dp < DP; ++dp) s2 += spp[dp * KT16 * nh];
          v[u] = s2 * scale;
        }
        cm = fmaxf(cm, v[u]);
      }
      const float mold = red[h];
      const float mnew = fmaxf(mold, warp_max(cm));
      float ls = 0.f;
#pragma unroll
      for (int u = 0; u < CH / 32; ++u) {
        const int j = lane + 32 * u;
        const float e = j < n ? expf(v[u] - mnew) : 0.f;
        ls += e;
        if (j < KT16) put3(pt + 3 * h * PP + j, PP, e);
      }
      ls = warp_sum(ls);
      if (lane == 0) {
        const float corr = expf(mold - mnew);
        red[32 + h] = corr;
        red[16 + h] = red[16 + h] * corr + ls;
        red[h] = mnew;
      }
    }
    cbar();
    // ---- weighted sums of this warp's dim tiles over the chunk's key tiles
    {
      float dg[kAttMT][2][4];
#pragma unroll
      for (int m = 0; m < kAttMT; ++m)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) dg[m][nt][0] = dg[m][nt][1] = dg[m][nt][2] = dg[m][nt][3] = 0.f;
      for (int kk = 0; kk < nkt; ++kk) {
        const int j0 = kk * 16;
        unsigned kb = sbase[0];
#pragma unroll
        for (int j = 1; j < kSlots; ++j)
          if ((kk >> 1) == j) kb = sbase[j];
        kb += static_cast<unsigned>((kk & 1) * 16 * P);
        const bool tail = j0 + 16 > n;
        uint32_t b0[2], b1[2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          b0[nt] = b1[nt] = 0u;
          if (nt < NT && wb[0][nt] >= 0) {
            const unsigned bp = pts + static_cast<unsigned>(wb[0][nt] + 2 * j0);
            b0[nt] = lds32(bp);
            b1[nt] = lds32(bp + 16);
          }
        }
#pragma unroll
        for (int m = 0; m < kAttMT; ++m) {
          if (wact[m]) {
            uint4 a = ldsm_x4_t(kb + woff[m]);
            if (tail) {  // keys past the chunk's rows: zero (their rows hold no K)
              a.x = keep_keys(a.x, j0 + 2 * ti, n);
              a.y = keep_keys(a.y, j0 + 2 * ti, n);
              a.z = keep_keys(a.z, j0 + 8 + 2 * ti, n);
              a.w = keep_keys(a.w, j0 + 8 + 2 * ti, n);
            }
            uint32_t c0 = b0[0], c1 = b1[0], e0 = b0[1], e1 = b1[1];
            if (m > 0 && (wb[m][0] != wb[0][0] || wb[m][1] != wb[0][1])) {  // another group's heads
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
                uint32_t x0 = 0u, x1 = 0u;
                if (nt < NT && wb[m][nt] >= 0) {
                  const unsigned bp = pts + static_cast<unsigned>(wb[m][nt] + 2 * j0);
                  x0 = lds32(bp);
                  x1 = lds32(bp + 16);
                }
                if (nt == 0) { c0 = x0; c1 = x1; } else { e0 = x0; e1 = x1; }
              }
            }
            mma_bf16(dg[m][0], a, c0, c1);
            if (NT > 1) mma_bf16(dg[m][1], a, e0, e1);
          }
        }
        // this warp is done with slot kk / 2 once it has passed both of its key tiles
        if ((kk & 1) == 1 || kk == nkt - 1) ring_release(rg, g + (kk >> 1));
      }
#pragma unroll
      for (int m = 0; m < kAttMT; ++m) {
        const int task = warp + m * kCW;
        const int grp = wact[m] ? task / MT : 0;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int hh = (nt * 8 + 2 * ti) >> 2;
          const float cr = (nt < NT && hh < hpg) ? red[32 + grp * hpg + hh] : 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[m][nt][i] = fmaf(acc[m][nt][i], cr, dg[m][nt][i]);
        }
      }
    }
    g += ns;
  }
  // ---- partial sums and (m, l) to the owners of the dims
  if (live) {
    const int per = 2 + dpo;
#pragma unroll
    for (int m = 0; m < kAttMT; ++m) {
      const int task = warp + m * kCW;
      if (wact[m]) {
        const int grp = task / MT, mt = task % MT;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          if (nt < NT) {
            float v0 = acc[m][nt][0] + acc[m][nt][1], v1 = acc[m][nt][2] + acc[m][nt][3];
            v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
            v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
            const int hh = (nt * 8 + 2 * ti) >> 2;
            if ((ti & 1) == 0 && hh < hpg) {
              const int h = grp * hpg + hh;
              const int i0 = h * d + mt * 16 + gi, i1 = i0 + 8;
              const int w0 = i0 / dpo, w1 = i1 / dpo;
              st_async_u32(mapa(xdst + 4u * (r * per + 2 + i0 - w0 * dpo), w0), __float_as_uint(v0), mapa(xbar, w0));
              st_async_u32(mapa(xdst + 4u * (r * per + 2 + i1 - w1 * dpo), w1), __float_as_uint(v1), mapa(xbar, w1));
            }
          }
        }
      }
    }
    if (tid < nh) {
      const int h = tid;
      const float mh = red[h], lh = red[16 + h];
      for (int w = (h * d) / dpo; w <= (h * d + d - 1) / dpo; ++w) {
        const unsigned a = mapa(xdst + 4u * (r * per), w), b = mapa(xbar, w);
        st_async_u32(a, __float_as_uint(mh), b);
        st_async_u32(a + 4, __float_as_uint(lh), b);
      }
    }
  }
  return g;
}

// ------------------------------------------------------------------ head helpers

// Logits of the rows of this CTA's selected centroids [slo, shi) (contiguous blocks of the
// cluster-ordered embedding copy) against y; each warp's best (value, id) key goes to lk.
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
// Sums 8 per-lane values over the warp with a transposed butterfly; afterwards lane l holds
// the full sum of value l >> 2.
__device__ __forceinline__ float xreduce8(float (&a)[8], int lane) {
  int o = 16;
#pragma unroll
  for (int c = 8; c > 1; c >>= 1) {
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
__device__ __noinline__ void gather_best(const bf16* temb_ord, const int* ord, int H, int vsc, int nclust,
                                         const int* selc, int slo, int shi, const float* y, unsigned long long* lk) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long best = 0ull;
  for (int c = slo; c < shi; ++c) {
    const size_t base = static_cast<size_t>(min(max(selc[c], 0), nclust - 1)) * vsc;
    for (int jb = warp * 8; jb < vsc; jb += kCW * 8) {
      const int myrow = jb + (lane >> 2);
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
      const float v = xreduce8(a, lane);
      if ((lane & 3) == 0 && myrow < vsc) {
        const unsigned long long key = argmax_key(v, id);
        best = key > best ? key : best;
      }
    }
  }
  best = warp_max_u64(best);
  if (lane == 0) lk[warp] = best;
}

// Global top-k of kNC sorted (descending) lists of k distinct keys by a tree of pairwise
// merges (kNC -> kNC/2 -> ... -> 1, one warp per merge, a barrier between levels). In a merge
// of A and B, A[i] lands at i + #{B > A[i]} and B[j] at j + #{A > B[j]} (binary searches);
// positions >= k are dropped. The last level writes the selected centroid ids to selc.
__device__ __forceinline__ int count_greater(const unsigned long long* L, int k, unsigned long long e) {
  int pos = 0;
  for (int step = 64; step > 0; step >>= 1)  // k <= 64
    if (pos + step <= k && L[pos + step - 1] > e) pos += step;
  return pos;
}
__device__ __noinline__ void merge_tree(const unsigned long long* lists, int k, int C, unsigned long long* buf_a,
                                        unsigned long long* buf_b, int* selc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long* in = lists;
  unsigned long long* out = buf_a;
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
    in = out;
    out = (out == buf_a) ? buf_b : buf_a;
  }
}

// ------------------------------------------------------------------ the kernel

__global__ void __launch_bounds__(kT, 1) k_block_c2(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) char sm[];
  const Layout L = make_layout(p);
  unsigned rank_u;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank_u));
  const int r = static_cast<int>(rank_u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(sm + L.bars);
  const unsigned full0 = sa(bars), empty0 = sa(bars + kSlots), xbar0 = sa(bars + 2 * kSlots),
                 ubar = sa(bars + 2 * kSlots + 2);
  const unsigned ring0 = sa(sm + L.ring);
  const unsigned xs0 = sa(sm + L.xs);
  bf16* U = reinterpret_cast<bf16*>(sm + L.u);
  bf16* T = reinterpret_cast<bf16*>(sm + L.t);
  float* x = reinterpret_cast<float*>(sm + L.x);
  float* yv = reinterpret_cast<float*>(sm + L.y);
  float* part0 = reinterpret_cast<float*>(sm + L.part);
  float* part1 = part0 + kCW * 16;
  float* sp = reinterpret_cast<float*>(sm + L.sp);
  bf16* pt = reinterpret_cast<bf16*>(sm + L.pt);
  float* red = reinterpret_cast<float*>(sm + L.red);
  float2* cs = reinterpret_cast<float2*>(sm + L.cs);
  float* nrm = reinterpret_cast<float*>(sm + L.nrm);
  unsigned long long* ck = reinterpret_cast<unsigned long long*>(sm + L.keys);
  unsigned long long* lk = reinterpret_cast<unsigned long long*>(sm + L.lk);
  int* selc = reinterpret_cast<int*>(sm + L.selc);
  SecE* tab = reinterpret_cast<SecE*>(sm + L.tab);
  const Fail fl{p.status, p.abort_flag, p.spin_limit};
  const int H = p.H, UPe = 2 * p.bb + 8, TPe = H + 8;
  const int nseq = seq_count(p);

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kCW);
    }
    mbar_init(xbar0, 1);
    mbar_init(xbar0 + 8, 1);
    mbar_init(ubar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // phase 0 of the hidden-state buffer receives step 0's post-projected rows
    if (p.n_draft > 1) mbar_expect_tx(ubar, 3u * static_cast<unsigned>(p.bb) * 2u);
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
  // every norm gain, once per launch
  for (int l = 0; l < p.nl; ++l) {
    float* nl_ = nrm + l * L.nrm_stride;
    const int d = p.d[p.ltype[l]];
    for (int i = tid; i < H; i += kT) {
      nl_[i] = __ldg(p.attn_norm[l] + i);
      nl_[H + i] = __ldg(p.post_attn_norm[l] + i);
      nl_[2 * H + i] = __ldg(p.ffn_norm[l] + i);
      nl_[3 * H + i] = __ldg(p.post_ffn_norm[l] + i);
    }
    for (int i = tid; i < d; i += kT) nl_[4 * H + i] = __ldg(p.q_norm[l] + i);
  }
  for (int i = tid; i < H; i += kT) nrm[p.nl * L.nrm_stride + i] = __ldg(p.out_norm + i);
  // this CTA's step sequence: weight sections of its stream, and its keys of each type (a
  // contiguous share of the full layers' [0, L) and of the sliding window)
  if (tid == 0) {
    long long soff = 0;
    for (int rr = 0; rr < r; ++rr) soff += stream_bytes(p, rr);
    const char* base = reinterpret_cast<const char*>(p.wstream) + soff;
    const int Lf = p.has_type[1] ? min(max(p.ctx_len[1][0], 0), p.kv_max[1]) : 0;
    const int Ls = p.has_type[0] ? min(max(p.ctx_len[0][0], 0), p.kv_max[0]) : 0;
    const int ws_lo = max(0, Ls - p.W);
    const Range fk = split(Lf, kNC, r), sk = split(Ls - ws_lo, kNC, r);
    for (int i = 0; i < nseq; ++i) {
      SecE e;
      memset(&e, 0, sizeof(e));
      if (seq_is_k(p, i)) {
        const int lt = p.ltype[(i - 1) / 6];
        const int lo = lt ? fk.lo : ws_lo + sk.lo;
        e.kind = 1;
        e.nkeys = lt ? fk.hi - fk.lo : sk.hi - sk.lo;
        e.row_bytes = p.nkv * p.d[lt] * 2;
        e.pitch = e.row_bytes + 16;
        e.stride = p.st[lt] * 2;
        e.src = reinterpret_cast<const char*>(p.k[lt]) + static_cast<long long>(lo) * e.stride;
      } else {
        int R, K;
        seq_shape(p, i, R, K);
        e.kind = 0;
        e.w = wsec(R, K, r);
        e.src = base;
        base += wsec_bytes(e.w);
      }
      tab[i] = e;
    }
  }
  // every barrier of the cluster is initialised before any CTA sends to a peer's (this also
  // orders the tables above before their first use)
  cluster_sync_all();

  if (warp == kCW) {
    // ====================== producer warp: every section of every step, in order
    int g = 0;
    bool ok = true;
    for (int step = 0; step < p.n_draft && ok; ++step) {
      for (int si = 0; si < nseq && ok; ++si) {
        const SecE* e = tab + si;
        const int n_sl = e->kind ? (e->nkeys + kKps - 1) / kKps : e->w.nsl;
        for (int c = 0; c < n_sl; ++c, ++g) {
          const int slot = g % kSlots;
          const unsigned fb = full0 + 8 * slot, dst = ring0 + slot * kSlotStride;
          if (lane == 0 && g >= kSlots &&
              !wait_bar(fl, empty0 + 8 * slot, static_cast<unsigned>((g / kSlots - 1) & 1), false))
            ok = false;
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (e->kind == 0) {
            if (lane == 0) {
              const unsigned bytes = static_cast<unsigned>(e->w.slot_bytes);
              mbar_expect_tx(fb, bytes);
              bulk_g2s(dst, e->src + static_cast<long long>(c) * bytes, bytes, fb);
            }
          } else {
            const int n = min(kKps, e->nkeys - c * kKps);
            if (lane == 0) mbar_expect_tx(fb, static_cast<unsigned>(n * e->row_bytes));
            if (lane < n)
              bulk_g2s(dst + lane * e->pitch, e->src + static_cast<long long>(c * kKps + lane) * e->stride,
                       static_cast<unsigned>(e->row_bytes), fb);
          }
        }
      }
    }
    // no copy of this CTA may still be in flight when it ends
    if (lane == 0)
      for (int h = (g > kSlots ? g - kSlots : 0); h < g; ++h)
        drain_bar(fl, full0 + 8 * (h % kSlots), static_cast<unsigned>((h / kSlots) & 1));
    __syncwarp();
  } else {
    // ====================== compute warps
    const Ring rg{ring0, full0, empty0, fl};
    int g = 0;   // ring slots consumed
    int xe = 0;  // exchanges done: set xe & 1, phase parity (xe >> 1) & 1
    bool live = true;
    auto xset = [&](int e) -> unsigned { return xs0 + static_cast<unsigned>((e & 1) * L.xs_bytes); };
    auto xsf = [&](int e) -> const float* { return reinterpret_cast<const float*>(sm + L.xs + (e & 1) * L.xs_bytes); };
    auto xbar = [&](int e) -> unsigned { return xbar0 + 8u * static_cast<unsigned>(e & 1); };
    auto arm = [&](int e, int bytes) {
      if (tid == 0 && live) mbar_expect_tx(xbar(e), static_cast<unsigned>(bytes));
    };
    auto xwait = [&](int e) {
      if (live && !wait_bar(fl, xbar(e), static_cast<unsigned>((e >> 1) & 1), true)) live = false;
    };
    // all-gather of the rows of a section (fp32, at the rows' offsets)
    auto gather_rows = [&](const SecE* se, const float* part, int total) -> const float* {
      arm(xe, 4 * total);
      if (live && !(xe == 0 && p.dbg_skip == r + 1))
        for (int i = tid; i < se->w.rows; i += kCT)
          bcast_f32(xset(xe) + 4u * static_cast<unsigned>(se->w.lo + i), xbar(xe), sum_parts(part, se, i));
      xwait(xe);
      return xsf(xe++);
    };
    const unsigned Us = sa(U), Ts = sa(T);

    int tok = 0;
    for (int step = 0; step < p.n_draft; ++step) {
      // ================= PRE: x0 = W_pre [h ; embed(token)]
      if (step == 0) {
        tok = p.tok_in[0];
        for (int v = tid; v < p.bb / 8; v += kCT) {  // h as exact terms (hi = h)
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(p.hidden_in) + v);
          *reinterpret_cast<uint4*>(U + 8 * v) = w;
          *reinterpret_cast<uint4*>(U + UPe + 8 * v) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(U + 2 * UPe + 8 * v) = make_uint4(0u, 0u, 0u, 0u);
        }
      } else {
        if (live && !wait_bar(fl, ubar, static_cast<unsigned>((step - 1) & 1), true)) live = false;
        if (tid == 0 && live && step + 1 < p.n_draft) mbar_expect_tx(ubar, 3u * static_cast<unsigned>(p.bb) * 2u);
      }
      if (tok < 0 || tok >= p.V) {
        if (r == 0 && tid == 0) set_status(p.status, MTP_ERR_INVALID_ARG);
        tok = 0;
      }
      {
        const uint4* er = reinterpret_cast<const uint4*>(p.tgt + static_cast<size_t>(tok) * p.bb);
        for (int v = tid; v < p.bb / 8; v += kCT) {
          const uint4 w = __ldg(er + v);
          *reinterpret_cast<uint4*>(U + p.bb + 8 * v) = w;
          *reinterpret_cast<uint4*>(U + UPe + p.bb + 8 * v) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(U + 2 * UPe + p.bb + 8 * v) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      cbar();
      g = gemv2(rg, g, tab + 0, Us, UPe * 2, part0);
      cbar();
      {
        const float* xg = gather_rows(tab + 0, part0, H);
        for (int i = tid; i < H; i += kCT) x[i] = xg[i];
        cbar();
      }
      // ================= decoder blocks
      for (int l = 0; l < p.nl; ++l) {
        const int lt = p.ltype[l], d = p.d[lt], QD = p.nh * d, half = d / 2, dpo = QD / kNC;
        const float* gn = nrm + l * L.nrm_stride;
        const SecE* sq = tab + 1 + 6 * l;
        // ---- Q rows of attn_norm(x)
        {
          const float rf = rms_inv(x, H, p.eps);
          for (int i = tid; i < H; i += kCT) put3(T + i, TPe, x[i] * rf * gn[i]);
          cbar();
        }
        g = gemv2(rg, g, sq, Ts, TPe * 2, part0);
        cbar();
        const float* q = gather_rows(sq, part0, QD);
        // ---- q_norm + RoPE -> three bf16 terms per head (rows 3h + t, pitch d + 8) in U
        {
          const int QPe = d + 8;
          const int wph = kCW / p.nh >= 1 ? kCW / p.nh : 1;
          const float2* c2 = cs + (lt ? L.cs_off1 : 0);
          const float* gq = gn + 4 * H;
          for (int h = warp / wph; h < p.nh; h += kCW / wph) {
            const float* qh = q + h * d;
            float s = 0.f;
            for (int i = lane; i < d; i += 32) s = fmaf(qh[i], qh[i], s);
            const float rf = rsqrtf(warp_sum(s) / d + p.eps);
            for (int i = (warp % wph) * 32 + lane; i < half; i += 32 * wph) {
              const float av = qh[i] * rf * gq[i], bv = qh[i + half] * rf * gq[i + half];
              const float2 cv = c2[i];
              put3(U + 3 * h * QPe + i, QPe, av * cv.x - bv * cv.y);
              put3(U + 3 * h * QPe + i + half, QPe, bv * cv.x + av * cv.y);
            }
          }
          cbar();
        }
        // ---- attention over this CTA's keys; partial sums to the owners of the dims
        arm(xe, kNC * (2 + dpo) * 4);
        {
          const SecE* sk = tab + 2 + 6 * l;
          if (p.nh == 4 && p.nkv == 1 && d == 512)
            g = att3<512, 4, 1>(rg, g, sk, 4, 1, 512, p.scale[lt], Us, sp, pt, red, xset(xe), xbar(xe), dpo, r, live);
          else if (p.nh == 4 && p.nkv == 1 && d == 256)
            g = att3<256, 4, 1>(rg, g, sk, 4, 1, 256, p.scale[lt], Us, sp, pt, red, xset(xe), xbar(xe), dpo, r, live);
          else
            g = att3<0, 0, 0>(rg, g, sk, p.nh, p.nkv, d, p.scale[lt], Us, sp, pt, red, xset(xe), xbar(xe), dpo, r, live);
        }
        xwait(xe);
        const float* pb = xsf(xe++);
        // ---- combine this CTA's dims (one head): weight of source s is
        // exp(m_s - M) / sum_s' exp(m_s' - M) l_s'; then the terms of o to every CTA
        {
          float* wt = red + 64;
          const int per = 2 + dpo;
          if (warp == 0) {
            const bool on = lane < kNC;
            const float m_s = on ? pb[lane * per] : -INFINITY;
            float M = m_s;
#pragma unroll
            for (int o = 1; o < kNC; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float e = (M == -INFINITY || m_s == -INFINITY) ? 0.f : expf(m_s - M);
            float den = on ? e * pb[lane * per + 1] : 0.f;
#pragma unroll
            for (int o = 1; o < kNC; o <<= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
            if (on) wt[lane] = den > 0.f ? e / den : 0.f;
          }
          cbar();
          arm(xe, 3 * QD * 2);
          if (live)
            for (int i = tid; i < dpo / 2; i += kCT) {
              float a0 = 0.f, a1 = 0.f;
              for (int s2 = 0; s2 < kNC; ++s2) {
                const float w2 = wt[s2];
                a0 = fmaf(w2, pb[s2 * per + 2 + 2 * i], a0);
                a1 = fmaf(w2, pb[s2 * per + 3 + 2 * i], a1);
              }
              bcast3(xset(xe) + 2u * static_cast<unsigned>(r * dpo + 2 * i), 2u * static_cast<unsigned>(QD + 8),
                     xbar(xe), terms2(a0, a1));
            }
          xwait(xe);
        }
        const unsigned ot = xset(xe++);
        // ---- O rows, residual with post_attn_norm, ffn_norm
        const SecE* so = tab + 3 + 6 * l;
        g = gemv2(rg, g, so, ot, (QD + 8) * 2, part0);
        cbar();
        {
          const float* op = gather_rows(so, part0, H);
          const float rf = rms_inv(op, H, p.eps);
          for (int i = tid; i < H; i += kCT) x[i] = x[i] + op[i] * rf * gn[H + i];
          cbar();
          const float rf2 = rms_inv(x, H, p.eps);
          for (int i = tid; i < H; i += kCT) put3(T + i, TPe, x[i] * rf2 * gn[2 * H + i]);
          cbar();
        }
        // ---- MLP: gate / up rows, m = gelu_tanh(gate) * up -> terms to every CTA
        const SecE* sg = tab + 4 + 6 * l;
        const SecE* su = tab + 5 + 6 * l;
        g = gemv2(rg, g, sg, Ts, TPe * 2, part0);
        g = gemv2(rg, g, su, Ts, TPe * 2, part1);
        cbar();
        arm(xe, 3 * p.F * 2);
        if (live)
          for (int i = tid; i < sg->w.rows / 2; i += kCT) {
            const float g0 = sum_parts(part0, sg, 2 * i), g1 = sum_parts(part0, sg, 2 * i + 1);
            const float u0 = sum_parts(part1, su, 2 * i), u1 = sum_parts(part1, su, 2 * i + 1);
            bcast3(xset(xe) + 2u * static_cast<unsigned>(sg->w.lo + 2 * i), 2u * static_cast<unsigned>(p.F + 8),
                   xbar(xe), terms2(gelu_tanh(g0) * u0, gelu_tanh(g1) * u1));
          }
        xwait(xe);
        const unsigned mt = xset(xe++);
        const SecE* sd = tab + 6 + 6 * l;
        g = gemv2(rg, g, sd, mt, (p.F + 8) * 2, part0);
        cbar();
        {
          const float* dn = gather_rows(sd, part0, H);
          const float rf = rms_inv(dn, H, p.eps);
          for (int i = tid; i < H; i += kCT) x[i] = p.lambda[l] * (x[i] + dn[i] * rf * gn[3 * H + i]);
          cbar();
        }
      }
      // ================= HEAD
      const int k = p.topk;
      {
        const float rf = rms_inv(x, H, p.eps);
        const float* go = nrm + p.nl * L.nrm_stride;
        for (int i = tid; i < H; i += kCT) {
          const float yy = x[i] * rf * go[i];
          yv[i] = yy;
          put3(T + i, TPe, yy);
        }
        cbar();
      }
      // centroid logits of this CTA's centroids -> local top-k by rank -> every CTA
      const SecE* sc = tab + 1 + 6 * p.nl;
      g = gemv2(rg, g, sc, Ts, TPe * 2, part0);
      cbar();
      for (int i = tid; i < sc->w.rows; i += kCT) ck[i] = argmax_key(sum_parts(part0, sc, i), sc->w.lo + i);
      cbar();
      for (int i = tid; i < sc->w.rows; i += kCT) {
        const unsigned long long key = ck[i];
        int rank = 0;
        for (int j = 0; j < sc->w.rows; ++j) rank += ck[j] > key ? 1 : 0;
        if (rank < k) lk[rank] = key;
      }
      cbar();
      const int xl = xe++;
      arm(xl, kNC * k * 8);
      if (live)
        for (int j = tid; j < k; j += kCT) bcast_u64(xset(xl) + 8u * static_cast<unsigned>(r * k + j), xbar(xl), lk[j]);
      // post rows -> h' (output, and the terms of the next step's input to every CTA)
      const SecE* spo = tab + 2 + 6 * p.nl;
      g = gemv2(rg, g, spo, Ts, TPe * 2, part1);
      cbar();
      for (int i = tid; i < spo->w.rows / 2; i += kCT) {
        const float h0 = sum_parts(part1, spo, 2 * i), h1 = sum_parts(part1, spo, 2 * i + 1);
        const int row = spo->w.lo + 2 * i;
        if (p.out_hidden) {
          p.out_hidden[static_cast<size_t>(step) * p.bb + row] = h0;
          p.out_hidden[static_cast<size_t>(step) * p.bb + row + 1] = h1;
        }
        if (live && step + 1 < p.n_draft) bcast3(Us + 2u * static_cast<unsigned>(row), 2u * UPe, ubar, terms2(h0, h1));
      }
      // merge of the lists -> selected centroids
      xwait(xl);
      merge_tree(reinterpret_cast<const unsigned long long*>(sm + L.xs + (xl & 1) * L.xs_bytes), k, p.C,
                 reinterpret_cast<unsigned long long*>(sp),
                 reinterpret_cast<unsigned long long*>(sp) + (kNC / 2) * k, selc);
      // ---- logits of this CTA's share of the candidate rows -> best key
      {
        const Range sr = split(k, kNC, r);
        if (tid < sr.hi - sr.lo) {  // request every candidate block from memory at once
          const size_t base = static_cast<size_t>(min(max(selc[sr.lo + tid], 0), p.C - 1)) * p.vsc;
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.temb_ord + base * H),
                       "r"(static_cast<unsigned>(p.vsc * H * 2))
                       : "memory");
        }
        gather_best(p.temb_ord, p.ord, H, p.vsc, p.C, selc, sr.lo, sr.hi, yv, lk);
      }
      cbar();
      const int xk = xe++;
      arm(xk, kNC * 8);
      if (warp == 0) {
        unsigned long long m = lane < kCW ? lk[lane] : 0ull;
        m = warp_max_u64(m);
        if (lane == 0 && live) bcast_u64(xset(xk) + 8u * static_cast<unsigned>(r), xbar(xk), m);
        if (m != 0ull) {  // warm L2 with the embedding row of this CTA's best token
          const int id = min(max(key_id(m), 0), p.V - 1);
          const char* er = reinterpret_cast<const char*>(p.tgt + static_cast<size_t>(id) * p.bb);
          for (int off = lane * 128; off < p.bb * 2; off += 32 * 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(er + off));
        }
      }
      xwait(xk);
      {
        const unsigned long long* kk = reinterpret_cast<const unsigned long long*>(sm + L.xs + (xk & 1) * L.xs_bytes);
        unsigned long long m = 0ull;
        for (int i = 0; i < kNC; ++i) m = kk[i] > m ? kk[i] : m;
        tok = min(max(key_id(m), 0), p.V - 1);
        if (r == 0 && tid == 0) p.out_tokens[step] = tok;
      }
      cbar();
    }
  }
  // no CTA leaves while a peer may still write into its shared memory
  cluster_sync_all();
}

// ------------------------------------------------------------------ packing

// Packs every CTA's section of W [R][K] (bf16, row-major) into its stream (CTA r =
// blockIdx.y, at byte offset off.b[r] of dst): tile (slot s, warp w, j < 4) in the order of
// WSec, each tile as 32 lanes x 16 bytes in mma.m16n8k16 A-fragment order (lane g = lane / 4,
// t = lane % 4 holds rows g and g + 8 at columns 2t, 2t + 1 and 2t + 8, 2t + 9); rows past the
// CTA's share are zero.
struct PackOffsets {
  long long b[kNC];
};
__global__ void k_c2_pack(const bf16* __restrict__ W, int R, int K, const __grid_constant__ PackOffsets off,
                          char* __restrict__ dst_base) {
  const int r = blockIdx.y;
  const WSec s = wsec(R, K, r);
  uint4* dst = reinterpret_cast<uint4*>(dst_base + off.b[r]);
  const int A = s.RT * s.P;
  const long long total = static_cast<long long>(s.RT) * s.KT * 32;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int lane = static_cast<int>(i % 32), tile = static_cast<int>(i / 32);
    const int sl = tile / (4 * A), rem = tile % (4 * A), w = rem / 4, j = rem % 4;
    const int rt = w % s.RT, pp = w / s.RT;
    const int kt = pp * (s.KT / s.P) + 4 * sl + j;
    const int g = lane >> 2, t = lane & 3;
    auto word = [&](int row, int col) -> uint32_t {
      const int lr = rt * 16 + row;
      if (lr >= s.rows) return 0u;
      const uint16_t* q = reinterpret_cast<const uint16_t*>(W + static_cast<size_t>(s.lo + lr) * K + kt * 16 + col);
      return static_cast<uint32_t>(q[0]) | (static_cast<uint32_t>(q[1]) << 16);
    };
    dst[i] = make_uint4(word(g, 2 * t), word(g + 8, 2 * t), word(g, 2 * t + 8), word(g + 8, 2 * t + 8));
  }
}

}  // namespace c2

// ------------------------------------------------------------------ host

namespace {
bool c2_attr(int smem) {
  if (cudaFuncSetAttribute(c2::k_block_c2, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(c2::k_block_c2, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}
cudaLaunchConfig_t c2_cfg(int smem, cudaStream_t st, cudaLaunchAttribute* at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c2::kNC);
  cfg.blockDim = dim3(c2::kT);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = c2::kNC;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cfg;
}
}  // namespace

int c2_smem_bytes(const c2::Params& p) {
  using namespace c2;
  if (p.nl < 1 || p.nl > kMaxL) return 0;
  if (p.H % 64 || p.bb % 32 || p.F % 64 || p.H < 64) return 0;  // k tiles in groups of 4; term pairs
  if (p.nkv < 1 || p.nh % p.nkv || p.nh / p.nkv > 4 || p.nh > 16) return 0;
  int dmax = 0;
  for (int l = 0; l < p.nl; ++l) {
    const int d = p.d[p.ltype[l]];
    const int QD = p.nh * d;
    if (d < 16 || d % 16 || QD % 64 || (2 * p.bb) % 64) return 0;
    const int dpo = QD / kNC;
    if (dpo > d || d % dpo) return 0;  // an owner's dims lie in one head
    if (p.nkv * (d / 16) > kAttMT * kCW) return 0;
    dmax = d > dmax ? d : dmax;
  }
  for (int t = 0; t < 2; ++t)
    if (p.has_type[t] && ((p.st[t] * 2) % 16 || p.nkv * p.d[t] * 2 + 16 > kSlotStride / kKps)) return 0;
  // every section's rows fit the compute warps (row tiles <= kCW) and a slot
  for (int i = 0; i < seq_count(p); ++i) {
    if (seq_is_k(p, i)) continue;
    int R, K;
    seq_shape(p, i, R, K);
    if (R < kNC || K % 64) return 0;
    for (int r = 0; r < kNC; ++r) {
      const WSec s = wsec(R, K, r);
      if (s.RT > kCW || s.slot_bytes > kSlotBytes || s.KT % (4 * s.P)) return 0;
    }
  }
  if (p.F % 32 || p.bb % 32) return 0;  // even row boundaries for the term pairs of m and h'
  if (p.topk < 1 || p.topk > 64 || p.C < kNC || p.topk > p.C / kNC || split_max(p.C, kNC) > kCT) return 0;
  if (p.vsc <= 0 || static_cast<long long>(p.C) * p.vsc != p.V) return 0;
  return make_layout(p).total;
}

int c2_capacity(int smem) {
  if (!c2_attr(smem)) return 0;
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = c2_cfg(smem, 0, at);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<void*>(c2::k_block_c2), &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int run_c2(const c2::Params& p, int smem, cudaStream_t st) {
  if (!c2_attr(smem)) {
    set_error("streamed cluster kernel attributes");
    return MTP_ERR_CUDA;
  }
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = c2_cfg(smem, st, at);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, c2::k_block_c2, p);
  if (e != cudaSuccess) {
    set_error("streamed cluster draft-block launch (%d CTAs, %d B shared memory): %s", c2::kNC, smem,
              cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

long long c2_stream_total(const c2::Params& p) {
  long long b = 0;
  for (int r = 0; r < c2::kNC; ++r) b += c2::stream_bytes(p, r);
  return b;
}

// Packs every weight section of every CTA into the stream buffer (layout of stream_bytes):
// one launch per section, all CTAs at once.
int c2_pack_all(const c2::Params& p, const void* const* mats, void* dst, cudaStream_t st) {
  using namespace c2;
  long long base[kNC];
  base[0] = 0;
  for (int r = 1; r < kNC; ++r) base[r] = base[r - 1] + stream_bytes(p, r - 1);
  PackOffsets off;
  for (int i = 0; i < seq_count(p); ++i) {
    if (seq_is_k(p, i)) continue;
    int R, K;
    seq_shape(p, i, R, K);
    for (int r = 0; r < kNC; ++r) off.b[r] = base[r];
    k_c2_pack<<<dim3(32, kNC), 256, 0, st>>>(static_cast<const bf16*>(mats[i]), R, K, off, static_cast<char*>(dst));
    for (int r = 0; r < kNC; ++r) base[r] += wsec_bytes(wsec(R, K, r));
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("packing the streamed weight tiles: %s", cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

}  // namespace mtp
