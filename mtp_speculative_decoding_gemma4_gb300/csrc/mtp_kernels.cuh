// Kernels of the drafter step (one launch per phase, or one persistent launch for the
// whole draft block) and their host-side launchers, templated on the model dtype.
#pragma once

#include <cstdio>

#include "mtp_launch.h"
#include "mtp_phases.cuh"
#include "mtp_tc.cuh"

namespace mtp {

// ---------------------------------------------------------------- grid barrier

__device__ inline unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of the persistent kernel: a monotone arrival counter (bar[0]) that
// every CTA bumps once per barrier, and an abort word (bar[1]). Waits are bounded: after
// spin_limit cycles the waiting CTA records MTP_ERR_TIMEOUT and raises the abort word, and
// every CTA that sees the abort word returns. Returns false when the kernel must stop.
__device__ inline bool grid_sync(const Params& p, unsigned int& epoch) {
  __shared__ int ok;
  __syncthreads();
  ++epoch;
  if (threadIdx.x == 0) {
    const unsigned int target = epoch * gridDim.x;
    __threadfence();
    if (p.dbg_skip == 0 || epoch != 1u || static_cast<int>(blockIdx.x) != p.dbg_skip - 1) atomicAdd(p.w.bar, 1u);
    const long long t0 = clock64();
    int good = 1;
    while (ld_acquire_u32(p.w.bar) < target) {
      if (ld_acquire_u32(p.w.bar + 1) != 0u) { good = 0; break; }
      if (clock64() - t0 > p.spin_limit) {
        atomicExch(p.w.status, static_cast<int>(MTP_ERR_TIMEOUT));
        atomicExch(p.w.bar + 1, 1u);
        good = 0;
        break;
      }
    }
    __threadfence();
    ok = good;
  }
  __syncthreads();
  return ok != 0;
}

// ---------------------------------------------------------------- per-phase kernels

#define MTP_KERNEL_PROLOGUE \
  extern __shared__ __align__(16) char smem[]; \
  pdl_enter();

template <typename WT> __global__ void __launch_bounds__(kThreads) k_rope(Params p) {
  pdl_enter();
  phase_rope(p, blockIdx.x, gridDim.x);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_pre(Params p, int step, int par) {
  MTP_KERNEL_PROLOGUE phase_pre<WT>(p, step, par, blockIdx.x, gridDim.x, smem);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_q(Params p, int l, int par) {
  MTP_KERNEL_PROLOGUE phase_q<WT>(p, l, par, blockIdx.x, gridDim.x, smem);
}
// One attention kernel per (head dim, heads per KV head): each gets its own register budget.
template <typename WT, int D, int HPG> __global__ void __launch_bounds__(kThreads) k_att(Params p, int l) {
  MTP_KERNEL_PROLOGUE att_phase_t<WT, D, HPG>(p, l, blockIdx.x, gridDim.x, smem);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_cmb(Params p, int l) {
  MTP_KERNEL_PROLOGUE phase_cmb<WT>(p, l, blockIdx.x, gridDim.x, smem);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_o(Params p, int l) {
  MTP_KERNEL_PROLOGUE phase_o<WT>(p, l, blockIdx.x, gridDim.x, smem);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_gu(Params p, int l, int par) {
  MTP_KERNEL_PROLOGUE phase_gu<WT>(p, l, par, blockIdx.x, gridDim.x, smem);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_dn(Params p, int l) {
  MTP_KERNEL_PROLOGUE phase_dn<WT>(p, l, blockIdx.x, gridDim.x, smem);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_head1(Params p, int step, int par) {
  MTP_KERNEL_PROLOGUE phase_head1<WT>(p, step, par, blockIdx.x, gridDim.x, smem);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_head_entry(Params p) {
  MTP_KERNEL_PROLOGUE phase_head_entry<WT>(p, blockIdx.x, gridDim.x, smem);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_topk(Params p) {
  MTP_KERNEL_PROLOGUE phase_topk<WT>(p, blockIdx.x, gridDim.x, smem);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_gather(Params p) {
  MTP_KERNEL_PROLOGUE phase_gather<WT>(p, blockIdx.x, gridDim.x, smem);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_dense(Params p) {
  MTP_KERNEL_PROLOGUE phase_dense<WT>(p, blockIdx.x, gridDim.x, smem);
}
template <typename WT> __global__ void __launch_bounds__(kThreads) k_fin(Params p, int stride, int col) {
  pdl_enter();
  phase_fin(p, stride, col, blockIdx.x, gridDim.x);
}

template <typename WT> __global__ void __launch_bounds__(kThreads) k_cand_min(Params p) {
  MTP_KERNEL_PROLOGUE phase_cand_min<WT>(p, blockIdx.x, gridDim.x, smem);
}
// Entries of the materialised rows still holding the -1e30 fill (those outside the selected
// clusters) -> the sequence's smallest candidate logit minus one.
template <typename WT>
__global__ void __launch_bounds__(kThreads) k_remask(float* out, long long V, long long n, const float* lmin) {
  const unsigned fill = __float_as_uint(-1e30f);
  for (long long i = blockIdx.x * static_cast<long long>(kThreads) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * kThreads)
    if (__float_as_uint(out[i]) == fill) out[i] = lmin[i / V] - 1.f;
}

// Fill of the materialised logits row (-1e30 everywhere before the sparse scatter).
template <typename WT>
__global__ void __launch_bounds__(kThreads) k_fill(float* out, long long n, float v) {
  for (long long i = blockIdx.x * static_cast<long long>(kThreads) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * kThreads)
    out[i] = v;
}

// ---------------------------------------------------------------- persistent draft block

template <typename WT>
__global__ void __launch_bounds__(kThreads, 1) k_block(Params p) {
  MTP_KERNEL_PROLOGUE
  const int cta = blockIdx.x, ncta = gridDim.x;
  unsigned int epoch = 0;
  phase_rope(p, cta, ncta);
  int par = 0;
  for (int s = 0; s < p.n_draft; ++s) {
    phase_pre<WT>(p, s, par, cta, ncta, smem);
    if (!grid_sync(p, epoch)) return;
    for (int l = 0; l < p.s.nl; ++l) {
      phase_q<WT>(p, l, par, cta, ncta, smem);
      if (l > 0) par ^= 1;
      if (!grid_sync(p, epoch)) return;
      phase_att<WT>(p, l, cta, ncta, smem);
      if (!grid_sync(p, epoch)) return;
      phase_cmb<WT>(p, l, cta, ncta, smem);
      if (!grid_sync(p, epoch)) return;
      phase_o<WT>(p, l, cta, ncta, smem);
      if (!grid_sync(p, epoch)) return;
      phase_gu<WT>(p, l, par, cta, ncta, smem);
      par ^= 1;
      if (!grid_sync(p, epoch)) return;
      phase_dn<WT>(p, l, cta, ncta, smem);
      if (!grid_sync(p, epoch)) return;
    }
    phase_head1<WT>(p, s, par, cta, ncta, smem);
    if (!grid_sync(p, epoch)) return;
    if (p.s.ordered) {
      phase_topk<WT>(p, cta, ncta, smem);
      if (!grid_sync(p, epoch)) return;
      phase_gather<WT>(p, cta, ncta, smem);
    } else {
      phase_dense<WT>(p, cta, ncta, smem);
    }
    if (!grid_sync(p, epoch)) return;
  }
  phase_fin(p, p.n_draft, p.n_draft - 1, cta, ncta);
}

// ---------------------------------------------------------------- host: sizes

struct PhaseSizes {
  int pre, q[kMaxLayers], att[kMaxLayers], cmb[kMaxLayers], o, gu, dn, head1, head_entry, topk, gather, dense;
  int smem_pre, smem_q, smem_att, smem_o[2], smem_gu, smem_dn, smem_head1, smem_topk, smem_gather, smem_dense;
  int smem_max;
};

template <typename WT>
inline int att_smem_for(const ShapeP& s, int t) { return att_smem_bytes<WT>(s.d[t], s.nh / s.nkv); }

template <typename WT>
PhaseSizes phase_sizes(const Params& p) {
  const ShapeP& s = p.s;
  PhaseSizes z{};
  const int nh = s.ncta_hint;
  z.pre = gemv_items(s.H, s.B, 2 * s.bb, nh);
  z.dn = gemv_items(s.H, s.B, s.F, nh);
  {
    const int ng = ceil_div(s.B, gemv_group(s.B, s.H));
    const int ks = choose_ks(2 * s.F, ng, nh);
    z.gu = ng * 2 * ceil_div(s.F, kWarps / ks);
    const int rows = s.bb + (s.ordered ? s.C : 0);
    const int ks2 = choose_ks(rows, ng, nh);
    z.head1 = ng * (ceil_div(s.bb, kWarps / ks2) + (s.ordered ? ceil_div(s.C, kWarps / ks2) : 0));
    z.head_entry = s.ordered ? gemv_items(s.C, s.B, s.H, nh) : ng;
  }
  for (int l = 0; l < s.nl; ++l) {
    const int t = p.L[l].type, d = s.d[t];
    z.q[l] = gemv_items(s.nh * d, s.B, s.H, nh);
    z.att[l] = ceil_div(s.B * s.nkv * s.nsplit[t], kWarps);  // one warp per item
    z.cmb[l] = s.B * s.nh * ceil_div(d, kCmbDims);
  }
  z.o = 0;
  z.topk = s.B;
  z.gather = s.ordered ? s.B * ceil_div(s.topk * s.vsc, kGatherPerItem) : 0;
  z.dense = s.ordered ? 0 : ceil_div(s.B, kDenseBG) * ceil_div(s.V, kDenseRowsPerItem);
  auto gs = [&](int K) { return gemv_smem(K, gemv_group(s.B, K), s.H).total; };
  z.smem_pre = gs(2 * s.bb);
  z.smem_q = gs(s.H);
  z.smem_o[0] = gs(s.nh * s.d[0]);
  z.smem_o[1] = gs(s.nh * s.d[1]);
  z.smem_gu = gs(s.H);
  z.smem_dn = gs(s.F);
  z.smem_head1 = gs(s.H);
  int att = 0;
  for (int l = 0; l < s.nl; ++l) {
    const int a = att_smem_for<WT>(s, p.L[l].type);
    att = a > att ? a : att;
  }
  z.smem_att = att;
  z.smem_topk = s.ordered ? topk_smem_bytes(s.C, s.topk) : 0;
  z.smem_gather = (s.H + 2) * 4 + kWarps * 8 + 16;
  z.smem_dense = s.ordered ? 0 : kDenseBG * s.H * 4 + kWarps * 32 * 8;
  const int cmb = 2 * (kThreads / kCmbDims) * kCmbDims * 4;
  int m = cmb;
  const int all[] = {z.smem_pre, z.smem_q, z.smem_o[0], z.smem_o[1], z.smem_gu, z.smem_dn, z.smem_head1,
                     z.smem_att, z.smem_topk, z.smem_gather, z.smem_dense};
  for (int v : all) m = v > m ? v : m;
  z.smem_max = m;
  return z;
}

// Items of the O phase of layer l (input width depends on the layer's head dim).
inline int o_items(const Params& p, int l) {
  const ShapeP& s = p.s;
  return gemv_items(s.H, s.B, s.nh * s.d[p.L[l].type], s.ncta_hint);
}

#define MTP_CHECK_LAUNCH(what)                                                          \
  do {                                                                                  \
    cudaError_t e_ = cudaGetLastError();                                                \
    if (e_ != cudaSuccess) {                                                            \
      set_error("%s launch failed: %s", what, cudaGetErrorString(e_));                  \
      return MTP_ERR_CUDA;                                                              \
    }                                                                                   \
  } while (0)

template <typename K>
inline int allow_smem(K kernel, int bytes) {
  if (bytes + 1024 > 48 * 1024) {  // the default limit also covers the kernel's static shared memory
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) {
      set_error("cudaFuncSetAttribute(%d bytes): %s", bytes, cudaGetErrorString(e));
      return MTP_ERR_CUDA;
    }
  }
  return MTP_OK;
}

#define MTP_LAUNCH(kernel, grid, smem_bytes, ...)                                       \
  do {                                                                                  \
    if ((grid) > 0) {                                                                   \
      int rc_ = allow_smem(kernel, smem_bytes);                                         \
      if (rc_) return rc_;                                                              \
      kernel<<<(grid), kThreads, (smem_bytes), st>>>(__VA_ARGS__);                      \
      MTP_CHECK_LAUNCH(#kernel);                                                        \
    }                                                                                   \
  } while (0)

// The same as a programmatic dependent launch (the tensor-core path's chain): the kernel may
// start launching while its predecessor runs and waits for it in pdl_enter().
#define MTP_LAUNCH_PDL(kernel, grid, smem_bytes, ...)                                   \
  do {                                                                                  \
    if ((grid) > 0) {                                                                   \
      int rc_ = allow_smem(kernel, smem_bytes);                                         \
      if (rc_) return rc_;                                                              \
      cudaLaunchConfig_t cfg_ = {};                                                     \
      cfg_.gridDim = dim3(grid);                                                        \
      cfg_.blockDim = dim3(kThreads);                                                   \
      cfg_.dynamicSmemBytes = static_cast<size_t>(smem_bytes);                          \
      cfg_.stream = st;                                                                 \
      cudaLaunchAttribute at_[1];                                                       \
      at_[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;                   \
      at_[0].val.programmaticStreamSerializationAllowed = 1;                            \
      cfg_.attrs = at_;                                                                 \
      cfg_.numAttrs = 1;                                                                \
      cudaError_t e_ = cudaLaunchKernelEx(&cfg_, kernel, __VA_ARGS__);                  \
      if (e_ != cudaSuccess) {                                                          \
        cudaGetLastError();                                                             \
        set_error("launch of %s failed: %s", #kernel, cudaGetErrorString(e_));          \
        return MTP_ERR_CUDA;                                                            \
      }                                                                                 \
    }                                                                                   \
  } while (0)

// The sparse head over the selected centroids: per sequence, or cluster-major (its own
// streamed kernel, mtp_head_cm.cu).
#define MTP_LAUNCH_GATHER()                                                            \
  do {                                                                                  \
    if (p.s.head_dd) {                                                                  \
      const int rc_ = run_head_cm<WT>(p, st);                                           \
      if (rc_) return rc_;                                                              \
    } else {                                                                            \
      MTP_LAUNCH(k_gather<WT>, z.gather, z.smem_gather, p);                             \
    }                                                                                   \
  } while (0)

// Launches the attention kernel of layer l's head dim and group size on `grid` CTAs.
template <typename WT>
int launch_att(const Params& p, int l, int grid, cudaStream_t st) {
  const int D = p.s.d[p.L[l].type], hpg = p.s.nh / p.s.nkv;
  const int smem = att_smem_bytes<WT>(D, hpg);
#define MTP_ATT_CASE(DD, HH) \
  if (D == DD && hpg == HH) {                    \
    MTP_LAUNCH((k_att<WT, DD, HH>), grid, smem, p, l); \
    return MTP_OK;                               \
  }
  MTP_ATT_CASES
#undef MTP_ATT_CASE
  set_error("no attention kernel for head_dim %d with %d query heads per KV head", D, hpg);
  return MTP_ERR_UNSUPPORTED_SHAPE;
}

#define MTP_LAUNCH_ATT(l)                                 \
  do {                                                    \
    int rc_a_ = launch_att<WT>(p, (l), z.att[(l)], st);   \
    if (rc_a_) return rc_a_;                              \
  } while (0)

// One launch per phase.
template <typename WT>
int run_phases(const Params& p, cudaStream_t st) {
  const PhaseSizes z = phase_sizes<WT>(p);
  const ShapeP& s = p.s;
  MTP_LAUNCH(k_rope<WT>, s.B, 0, p);
  int par = 0;
  for (int step = 0; step < p.n_draft; ++step) {
    MTP_LAUNCH(k_pre<WT>, z.pre, z.smem_pre, p, step, par);
    for (int l = 0; l < s.nl; ++l) {
      const int t = p.L[l].type;
      MTP_LAUNCH(k_q<WT>, z.q[l], z.smem_q, p, l, par);
      if (l > 0) par ^= 1;
      MTP_LAUNCH_ATT(l);
      MTP_LAUNCH(k_cmb<WT>, z.cmb[l], 2 * (kThreads / kCmbDims) * kCmbDims * 4, p, l);
      MTP_LAUNCH(k_o<WT>, o_items(p, l), z.smem_o[t], p, l);
      MTP_LAUNCH(k_gu<WT>, z.gu, z.smem_gu, p, l, par);
      par ^= 1;
      MTP_LAUNCH(k_dn<WT>, z.dn, z.smem_dn, p, l);
    }
    MTP_LAUNCH(k_head1<WT>, z.head1, z.smem_head1, p, step, par);
    if (s.ordered) {
      MTP_LAUNCH(k_topk<WT>, z.topk, z.smem_topk, p);
      MTP_LAUNCH_GATHER();
    } else {
      MTP_LAUNCH(k_dense<WT>, z.dense, z.smem_dense, p);
    }
  }
  MTP_LAUNCH(k_fin<WT>, 1, 0, p, p.n_draft, p.n_draft - 1);
  return MTP_OK;
}

// One launch per phase, every GEMV split into staging (the phase kernel with p.tc_xs set, one
// CTA per batch group) and tcgen05 GEMMs over the staged terms.
template <typename WT>
int run_phases_tc(const Params& p, const TcPlan& plan, cudaStream_t st) {
  const PhaseSizes z = phase_sizes<WT>(p);
  const ShapeP& s = p.s;
  Params ps = p;
  ps.tc_xs = plan.xs;
  ps.tc_bp = plan.bp;
  auto groups = [&](int) { return s.B; };  // staging runs one sequence per CTA
  auto gemm = [&](const CUtensorMap& w, const CUtensorMap& x, int R, int K, float* out, long long ldo, float* out2,
                  long long ld2, unsigned long long* best, int dbg_cta = -1, int R1 = 0, float* out_hi = nullptr,
                  long long ld_hi = 0, __nv_bfloat16* glu_xs = nullptr) -> int {
    tc::Args a{R,     K,           plan.bp, s.B,     out,   ldo,    out2,    ld2,     best,
               0,     p.w.status,  p.spin_limit,     dbg_cta, R1, out_hi, ld_hi, glu_xs, plan.bp, R / 2};
    return tc_gemm(&w, &x, a, best != nullptr, st, true);
  };
  int rc;
  MTP_LAUNCH(k_rope<WT>, s.B, 0, p);
  int par = 0;
  for (int step = 0; step < p.n_draft; ++step) {
    MTP_LAUNCH_PDL(k_pre<WT>, groups(2 * s.bb), z.smem_pre, ps, step, par);
    if ((rc = gemm(plan.pre, plan.xs_pre, s.H, 2 * s.bb, p.w.x[par], s.H, nullptr, 0, nullptr,
                   step == 0 ? p.dbg_skip - 1 : -1)))
      return rc;
    for (int l = 0; l < s.nl; ++l) {
      const int t = p.L[l].type, QD = s.nh * s.d[t];
      MTP_LAUNCH_PDL(k_q<WT>, groups(s.H), z.smem_q, ps, l, par);
      if ((rc = gemm(plan.q[l], plan.xs_h, QD, s.H, p.w.qraw, static_cast<long long>(s.nh) * p.w.dmax, nullptr, 0,
                     nullptr)))
        return rc;
      if (l > 0) par ^= 1;
      if (att_tc_supported(p, l)) {  // split-KV attention on tensor cores (bf16, V = K)
        if ((rc = run_att_tc(p, l, st))) return rc;
      } else {
        MTP_LAUNCH_ATT(l);
      }
      // the combine of the attention splits writes the O projection's staged operand
      MTP_LAUNCH_PDL(k_cmb<WT>, z.cmb[l], 2 * (kThreads / kCmbDims) * kCmbDims * 4, ps, l);
      if ((rc = gemm(plan.o[l], plan.xs_o[t], s.H, QD, p.w.ao, s.H, nullptr, 0, nullptr))) return rc;
      MTP_LAUNCH_PDL(k_gu<WT>, groups(s.H), z.smem_gu, ps, l, par);
      if (plan.gu_ok) {
        // gate and up as one launch whose epilogue stages gelu_tanh(gate) * up for the down
        // projection
        if ((rc = gemm(plan.gu[l], plan.xs_h, 2 * s.F, s.H, nullptr, 0, nullptr, 0, nullptr, -1, 0, nullptr, 0,
                       plan.xs_glu)))
          return rc;
        par ^= 1;
        if ((rc = gemm(plan.down[l], plan.xs_f2, s.H, s.F, p.w.dn, s.H, nullptr, 0, nullptr))) return rc;
      } else {
        if ((rc = gemm(plan.gate[l], plan.xs_h, s.F, s.H, p.w.gate, s.F, nullptr, 0, nullptr))) return rc;
        if ((rc = gemm(plan.up[l], plan.xs_h, s.F, s.H, p.w.up, s.F, nullptr, 0, nullptr))) return rc;
        par ^= 1;
        MTP_LAUNCH_PDL(k_dn<WT>, groups(s.F), z.smem_dn, ps, l);
        if ((rc = gemm(plan.down[l], plan.xs_f, s.H, s.F, p.w.dn, s.H, nullptr, 0, nullptr))) return rc;
      }
    }
    MTP_LAUNCH_PDL(k_head1<WT>, groups(s.H), z.smem_head1, ps, step, par);
    float* hout = p.out_hidden ? p.out_hidden + static_cast<size_t>(step) * s.bb : nullptr;
    const long long ldh = static_cast<long long>(p.n_draft) * s.bb;
    const bool postc = s.ordered && plan.postc_ok;  // post_projection and centroids as one launch
    if ((rc = postc ? gemm(plan.postc, plan.xs_h, s.bb + s.C, s.H, hout, ldh, p.w.h_cur, s.bb, nullptr, -1, s.bb,
                           p.w.cl, s.C)
                    : gemm(plan.post, plan.xs_h, s.bb, s.H, hout, ldh, p.w.h_cur, s.bb, nullptr)))
      return rc;
    if (s.ordered) {
      if (!postc && (rc = gemm(plan.cent, plan.xs_h, s.C, s.H, p.w.cl, s.C, nullptr, 0, nullptr))) return rc;
      MTP_LAUNCH_PDL(k_topk<WT>, z.topk, z.smem_topk, p);
      MTP_LAUNCH_GATHER();
    } else {
      if ((rc = gemm(plan.temb, plan.xs_h, s.V, s.H, nullptr, 0, nullptr, 0, p.w.best))) return rc;
    }
  }
  MTP_LAUNCH_PDL(k_fin<WT>, 1, 0, p, p.n_draft, p.n_draft - 1);
  return MTP_OK;
}

// One cooperative persistent launch for the whole block.
template <typename WT>
int run_persistent(const Params& p, cudaStream_t st) {
  const PhaseSizes z = phase_sizes<WT>(p);
  int rc = allow_smem(k_block<WT>, z.smem_max);
  if (rc) return rc;
  cudaError_t e = cudaMemsetAsync(p.w.bar, 0, 2 * sizeof(unsigned int), st);
  if (e != cudaSuccess) {
    set_error("cudaMemsetAsync: %s", cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  Params pp = p;
  void* args[] = {&pp};
  e = cudaLaunchCooperativeKernel(reinterpret_cast<void*>(k_block<WT>), dim3(p.s.ncta_hint), dim3(kThreads), args,
                                  static_cast<size_t>(z.smem_max), st);
  if (e != cudaSuccess) {
    set_error("persistent draft-block launch (%d CTAs, %d B smem): %s", p.s.ncta_hint, z.smem_max,
              cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

// Largest co-resident grid of the persistent kernel (0 when it cannot be resident).
template <typename WT>
int persistent_capacity(const Params& p, int num_sms) {
  const PhaseSizes z = phase_sizes<WT>(p);
  if (allow_smem(k_block<WT>, z.smem_max)) return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_block<WT>, kThreads, z.smem_max) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return per_sm * num_sms;
}

template <typename WT>
int run_head(const Params& p, cudaStream_t st) {
  const PhaseSizes z = phase_sizes<WT>(p);
  const ShapeP& s = p.s;
  if (p.out_logits && s.ordered) {
    const long long n = static_cast<long long>(s.B) * s.V;
    k_fill<WT><<<1024, kThreads, 0, st>>>(p.out_logits, n, -1e30f);
    MTP_CHECK_LAUNCH("k_fill");
  }
  MTP_LAUNCH(k_head_entry<WT>, z.head_entry, z.smem_head1, p);
  if (s.ordered) {
    MTP_LAUNCH(k_topk<WT>, z.topk, z.smem_topk, p);
    MTP_LAUNCH_GATHER();
    if (p.out_logits && p.mask_mode == MTP_MASK_MIN_MINUS_ONE) {
      MTP_LAUNCH(k_cand_min<WT>, s.B, kWarps * 4, p);
      const long long n = static_cast<long long>(s.B) * s.V;
      k_remask<WT><<<1024, kThreads, 0, st>>>(p.out_logits, s.V, n, p.w.lmin);
      MTP_CHECK_LAUNCH("k_remask");
    }
  } else {
    MTP_LAUNCH(k_dense<WT>, z.dense, z.smem_dense, p);
  }
  MTP_LAUNCH(k_fin<WT>, 1, 0, p, 1, 0);
  return MTP_OK;
}

}  // namespace mtp
