// Split-KV attention of the batched drafter on tensor cores (bf16, V = K): the query heads of
// one KV head attend the target's shared K (Gemma 4 MTP drafter, "What it is": Q-only
// attention over the target's last K/V of each type, values equal to the keys), each split of
// the attended keys giving unnormalised partial sums and its (max, exp-sum) per head for the
// combine phase.
//
// One CTA of 8 warps per (sequence, KV head, key split). The split's keys go in chunks of 64,
// copied with cp.async into a double buffer at a padded pitch (row + 16 bytes, so ldmatrix
// reads 8 rows without bank conflicts). q_norm and RoPE are applied to the group's query heads
// and every value is split into three bf16 terms (hi + mid + lo == the fp32 value to fp32
// precision), so each product with a bf16 key element is exact. Per chunk:
//   scores   S[key][col] = K q (mma.m16n8k16): tasks (16-key tile, dim part) over the warps,
//            the parts' partial sums added in a fixed order by the softmax warps;
//   softmax  warp h updates the running max / exp-sum of head h over the chunk and writes p
//            as three bf16 terms;
//   sums     O^T[dim][col] += K^T P^T: each warp owns 16-dim tiles, rescaled once per chunk.
// Column 4c + t of an MMA carries term t of head c of the pair of heads of its n tile (the
// fourth column is zero), so a head's value is the sum of its three columns.
#include "mtp_launch.h"
#include "mtp_phases.cuh"

namespace mtp {
namespace atc {

constexpr int kW = 8;         // warps per CTA
constexpr int kT = kW * 32;
constexpr int kCK = 64;       // keys per chunk (4 tiles of 16)
constexpr int kMaxMT = 4;     // 16-dim tiles per warp in the weighted sum (head_dim <= 16 * 4 * kW)

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ unsigned sa(const void* p) { return static_cast<unsigned>(__cvta_generic_to_shared(p)); }
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
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}
// The terms of v at rows 0, 1, 2 (pitch rs elements) of dst.
__device__ __forceinline__ void put3(bf16* dst, int rs, float v) {
  const bf16 h = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(h);
  const bf16 m = __float2bfloat16_rn(r1);
  dst[0] = h;
  dst[rs] = m;
  dst[2 * rs] = __float2bfloat16_rn(r1 - __bfloat162float(m));
}
// The bf16 pair of keys (key, key + 1) in v with keys at or past n set to zero.
__device__ __forceinline__ uint32_t keep_keys(uint32_t v, int key, int n) {
  return key + 1 < n ? v : (key < n ? (v & 0xffffu) : 0u);
}

template <int D, int HPG>
struct Lay {
  static constexpr int P = 2 * D + 16;   // bytes between K rows
  static constexpr int QP = D + 8;       // elements between q-term rows
  static constexpr int PP = kCK + 8;     // elements between p-term rows
  static constexpr int kbuf = 0;
  static constexpr int qt = kbuf + 2 * kCK * P;
  static constexpr int pt = qt + 3 * HPG * QP * 2;
  static constexpr int sp = (pt + 3 * HPG * PP * 2 + 15) / 16 * 16;  // [parts <= kW][kCK][HPG] floats
  static constexpr int red = sp + kW * kCK * HPG * 4;                 // m [16], l [16], corr [16], rf [16]
  static constexpr int total = red + 64 * 4;
};

template <int D, int HPG>
__global__ void __launch_bounds__(kT) k_att_tc(const __grid_constant__ Params p, int l) {
  // programmatic dependent launch: the first K chunk (the target's cache, which the draft
  // block never writes) is requested before the wait for the kernels that write q
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using LY = Lay<D, HPG>;
  constexpr int P = LY::P, QP = LY::QP, PP = LY::PP;
  constexpr int NT = (HPG + 1) / 2, KS = D / 16, MT = D / 16, half = D / 2;
  extern __shared__ __align__(128) char sm[];
  bf16* qt = reinterpret_cast<bf16*>(sm + LY::qt);
  bf16* pt = reinterpret_cast<bf16*>(sm + LY::pt);
  float* sp = reinterpret_cast<float*>(sm + LY::sp);
  float* red = reinterpret_cast<float*>(sm + LY::red);
  const unsigned kb0 = sa(sm + LY::kbuf), qts = sa(qt), pts = sa(pt);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gi = lane >> 2, ti = lane & 3;

  const int t = p.L[l].type;
  const KvP& kv = p.kv[t];
  const int nsp = p.s.nsplit[t], nkv = p.s.nkv;
  const int c = blockIdx.x % nsp, g = (blockIdx.x / nsp) % nkv, b = blockIdx.x / (nsp * nkv);
  const int Lb = min(max(kv.ctx_len[b], 0), kv.max_ctx);  // never read past the buffer
  const int lo = t == 0 ? max(0, Lb - p.s.W) : 0, hi = Lb;
  const int chunk = (max(hi - lo, 0) + nsp - 1) / nsp;
  const int j0 = lo + c * chunk, nkeys = max(0, min(hi, j0 + chunk) - j0);
  const bf16* kbase = static_cast<const bf16*>(kv.k) + static_cast<size_t>(b) * kv.sb + static_cast<size_t>(g) * D;
  const int nchunks = (nkeys + kCK - 1) / kCK;

  // chunk q of the split -> buffer q & 1 (one commit group per chunk index, empty or not)
  auto load = [&](int q) {
    if (q < nchunks) {
      const int n = min(kCK, nkeys - q * kCK);
      const unsigned dst = kb0 + static_cast<unsigned>((q & 1) * kCK * P);
      for (int v = tid; v < n * (D / 8); v += kT) {
        const int r = v / (D / 8), cc = v % (D / 8);
        cp_async16(dst + r * P + cc * 16, kbase + static_cast<size_t>(j0 + q * kCK + r) * kv.st + cc * 8, 16);
      }
    }
    cp_async_commit();
  };
  load(0);
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // q_norm + RoPE at the constant position of the group's heads -> three bf16 terms per head
  {
    const float* qr0 = p.w.qraw + static_cast<size_t>(b) * p.s.nh * p.w.dmax + static_cast<size_t>(g * HPG) * D;
    if (warp < HPG) {
      const float* qh = qr0 + warp * D;
      float s = 0.f;
      for (int i = lane; i < D; i += 32) s = fmaf(qh[i], qh[i], s);
      s = warp_sum(s);
      if (lane == 0) red[48 + warp] = rsqrtf(s / D + p.s.eps);
    }
    if (tid < HPG) {
      red[tid] = -INFINITY;   // running max of head tid
      red[16 + tid] = 0.f;    // running exp-sum
    }
    __syncthreads();
    const float2* cs = p.w.cs + (static_cast<size_t>(b) * 2 + t) * (p.w.dmax / 2);
    const float* gq = p.L[l].q_norm;
    for (int it = tid; it < HPG * half; it += kT) {
      const int hh = it / half, i = it % half;
      const float* qh = qr0 + hh * D;
      const float rf = red[48 + hh];
      const float av = qh[i] * rf * gq[i], bv = qh[i + half] * rf * gq[i + half];
      const float2 r = cs[i];
      put3(qt + 3 * hh * QP + i, QP, av * r.x - bv * r.y);
      put3(qt + 3 * hh * QP + i + half, QP, bv * r.x + av * r.y);
    }
  }
  // this lane's B row of n tile nt in the head-term layout (-1: a zero column)
  auto brow = [&](int nt) -> int {
    const int col = nt * 8 + gi, hh = col >> 2, tt = col & 3;
    return (tt == 3 || hh >= HPG) ? -1 : 3 * hh + tt;
  };
  float acc[kMaxMT][2][4];
#pragma unroll
  for (int m = 0; m < kMaxMT; ++m)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) acc[m][nt][0] = acc[m][nt][1] = acc[m][nt][2] = acc[m][nt][3] = 0.f;

  for (int q = 0; q < nchunks; ++q) {
    load(q + 1);
    cp_async_wait<1>();
    __syncthreads();  // chunk q is in place for every thread (and the q terms, on the first chunk)
    const int n = min(kCK, nkeys - q * kCK), nkt = (n + 15) / 16, KT16 = nkt * 16;
    const unsigned K = kb0 + static_cast<unsigned>((q & 1) * kCK * P);
    // ---- scores: dim parts DP, the largest power of two with nkt DP <= kW dividing d / 16
    int ldp = 0;
    while (nkt * (2 << ldp) <= kW && KS % (2 << ldp) == 0) ++ldp;
    const int DP = 1 << ldp;
    if (warp < nkt * DP) {
      const int dpart = warp & (DP - 1), kt = warp >> ldp, nks = KS >> ldp, ks0 = dpart * nks;
      float sv[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) sv[nt][0] = sv[nt][1] = sv[nt][2] = sv[nt][3] = 0.f;
      unsigned a_addr = K + static_cast<unsigned>((kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * P +
                                                  (lane >> 4) * 16 + ks0 * 32);
      unsigned b_addr[2];
      bool bon[2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int rw = nt < NT ? brow(nt) : -1;
        bon[nt] = rw >= 0;
        b_addr[nt] = qts + 2u * static_cast<unsigned>((bon[nt] ? rw : 0) * QP + ks0 * 16 + 2 * ti);
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
          if ((ti & 1) == 0 && hh < HPG) {
            float* spp = sp + (dpart * KT16 + kt * 16 + gi) * HPG + hh;
            spp[0] = v0;
            spp[8 * HPG] = v1;
          }
        }
      }
    }
    __syncthreads();
    // ---- running max / exp-sum of head `warp` over the chunk; p as three bf16 terms
    if (warp < HPG) {
      const int h = warp;
      const float scale = p.s.scale[t];
      float v[kCK / 32];
      float cm = -INFINITY;
#pragma unroll
      for (int u = 0; u < kCK / 32; ++u) {
        const int j = lane + 32 * u;
        v[u] = -INFINITY;
        if (j < n) {
          float s2 = 0.f;
          for (int dp = 0; dp < DP; ++dp) s2 += sp[(dp * KT16 + j) * HPG + h];
          v[u] = s2 * scale;
        }
        cm = fmaxf(cm, v[u]);
      }
      const float mold = red[h];
      const float mnew = fmaxf(mold, warp_max(cm));
      float ls = 0.f;
#pragma unroll
      for (int u = 0; u < kCK / 32; ++u) {
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
    __syncthreads();
    // ---- weighted sums of this warp's dim tiles over the chunk's key tiles
    {
      float dg[kMaxMT][2][4];
#pragma unroll
      for (int m = 0; m < kMaxMT; ++m)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) dg[m][nt][0] = dg[m][nt][1] = dg[m][nt][2] = dg[m][nt][3] = 0.f;
      const unsigned arow = K + static_cast<unsigned>(((lane & 7) + (lane >> 4) * 8) * P + ((lane >> 3) & 1) * 16);
      for (int kk = 0; kk < nkt; ++kk) {
        const int j0k = kk * 16;
        uint32_t b0[2], b1[2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int rw = nt < NT ? brow(nt) : -1;
          b0[nt] = b1[nt] = 0u;
          if (rw >= 0) {
            const unsigned bp = pts + 2u * static_cast<unsigned>(rw * PP + j0k + 2 * ti);
            b0[nt] = lds32(bp);
            b1[nt] = lds32(bp + 16);
          }
        }
        const bool tail = j0k + 16 > n;
#pragma unroll
        for (int m = 0; m < kMaxMT; ++m) {
          const int mt = warp + m * kW;
          if (mt < MT) {
            uint4 a = ldsm_x4_t(arow + static_cast<unsigned>(j0k * P + mt * 32));
            if (tail) {  // keys past the chunk's rows: zero (their rows hold no K of this split)
              a.x = keep_keys(a.x, j0k + 2 * ti, n);
              a.y = keep_keys(a.y, j0k + 2 * ti, n);
              a.z = keep_keys(a.z, j0k + 8 + 2 * ti, n);
              a.w = keep_keys(a.w, j0k + 8 + 2 * ti, n);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
              if (nt < NT) mma_bf16(dg[m][nt], a, b0[nt], b1[nt]);
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int hh = (nt * 8 + 2 * ti) >> 2;
        const float cr = (nt < NT && hh < HPG) ? red[32 + hh] : 0.f;
#pragma unroll
        for (int m = 0; m < kMaxMT; ++m)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[m][nt][i] = fmaf(acc[m][nt][i], cr, dg[m][nt][i]);
      }
    }
    __syncthreads();  // the buffer of chunk q is reloaded by the next iteration's prefetch
  }
  cp_async_wait<0>();
  // ---- partial sums and (max, exp-sum) of every head of the group for the combine phase
#pragma unroll
  for (int m = 0; m < kMaxMT; ++m) {
    const int mt = warp + m * kW;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (nt < NT) {
        float v0 = acc[m][nt][0] + acc[m][nt][1], v1 = acc[m][nt][2] + acc[m][nt][3];
        v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        const int hh = (nt * 8 + 2 * ti) >> 2;
        if (mt < MT && (ti & 1) == 0 && hh < HPG) {
          const size_t slot = (static_cast<size_t>(b) * p.s.nh + g * HPG + hh) * p.w.nsplit_max + c;
          float* dst = p.w.part_acc + slot * p.w.dmax + mt * 16 + gi;
          dst[0] = v0;
          dst[8] = v1;
        }
      }
    }
  }
  if (tid < HPG) {
    const size_t slot = (static_cast<size_t>(b) * p.s.nh + g * HPG + tid) * p.w.nsplit_max + c;
    p.w.part_ml[slot * 2] = red[tid];
    p.w.part_ml[slot * 2 + 1] = red[16 + tid];
  }
}

template <int D, int HPG>
int launch(const Params& p, int l, cudaStream_t st) {
  const int smem = Lay<D, HPG>::total;
  cudaError_t e = cudaFuncSetAttribute(k_att_tc<D, HPG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) {
    const int t = p.L[l].type;
    // a programmatic dependent launch in the tensor-core path's chain (pdl_enter waits)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.s.B * p.s.nkv * p.s.nsplit[t]);
    cfg.blockDim = dim3(kT);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_att_tc<D, HPG>, p, l);
  }
  if (e != cudaSuccess) {
    set_error("tensor-core attention launch: %s", cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

}  // namespace atc

bool att_tc_supported(const Params& p, int l) {
  const int t = p.L[l].type, D = p.s.d[t], hpg = p.s.nkv > 0 ? p.s.nh / p.s.nkv : 0;
  const KvP& kv = p.kv[t];
  const bool v_is_k = kv.v == nullptr || kv.v == kv.k;
  const bool aligned = (reinterpret_cast<uintptr_t>(kv.k) & 15) == 0 && (kv.st * 2) % 16 == 0 && (kv.sb * 2) % 16 == 0;
  return v_is_k && aligned && (D == 64 || D == 128 || D == 256 || D == 512) && hpg >= 1 && hpg <= 4;
}

int att_tc_smem(int D, int hpg) {
#define MTP_ATC_SMEM(DD, HH) \
  if (D == DD && hpg == HH) return atc::Lay<DD, HH>::total;
  MTP_ATC_SMEM(64, 1) MTP_ATC_SMEM(64, 2) MTP_ATC_SMEM(64, 4)
  MTP_ATC_SMEM(128, 1) MTP_ATC_SMEM(128, 2) MTP_ATC_SMEM(128, 4)
  MTP_ATC_SMEM(256, 1) MTP_ATC_SMEM(256, 2) MTP_ATC_SMEM(256, 4)
  MTP_ATC_SMEM(512, 1) MTP_ATC_SMEM(512, 2) MTP_ATC_SMEM(512, 4)
#undef MTP_ATC_SMEM
  return 0;
}

int run_att_tc(const Params& p, int l, cudaStream_t st) {
  const int t = p.L[l].type, D = p.s.d[t], hpg = p.s.nh / p.s.nkv;
#define MTP_ATC_CASE(DD, HH) \
  if (D == DD && hpg == HH) return atc::launch<DD, HH>(p, l, st);
  MTP_ATC_CASE(64, 1) MTP_ATC_CASE(64, 2) MTP_ATC_CASE(64, 4)
  MTP_ATC_CASE(128, 1) MTP_ATC_CASE(128, 2) MTP_ATC_CASE(128, 4)
  MTP_ATC_CASE(256, 1) MTP_ATC_CASE(256, 2) MTP_ATC_CASE(256, 4)
  MTP_ATC_CASE(512, 1) MTP_ATC_CASE(512, 2) MTP_ATC_CASE(512, 4)
#undef MTP_ATC_CASE
  set_error("no tensor-core attention for head_dim %d with %d query heads per KV head", D, hpg);
  return MTP_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace mtp
