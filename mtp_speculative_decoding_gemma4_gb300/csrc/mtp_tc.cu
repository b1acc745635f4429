// Tensor-core GEMM of the batched projections: see mtp_tc.cuh.
#include <cudaTypedefs.h>

#include <mutex>

#include "mtp.h"
#include "mtp_common.cuh"
#include "mtp_launch.h"
#include "mtp_stage.cuh"
#include "mtp_tc.cuh"

namespace mtp {
namespace tc {

__device__ __forceinline__ unsigned sa(const void* p) { return static_cast<unsigned>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool try_wait(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(100000u)
      : "memory");
  return ok != 0;
}
// Bounded wait: false (and MTP_ERR_TIMEOUT recorded) when the phase does not complete in time.
__device__ __noinline__ bool wait_bar(unsigned bar, unsigned parity, int* status, long long limit) {
  if (try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!try_wait(bar, parity)) {
    if (clock64() - t0 > limit) {
      atomicCAS(status, 0, static_cast<int>(MTP_ERR_TIMEOUT));
      return false;
    }
  }
  return true;
}

// TMA: a box of the tensor map at (x = column, y = row) into shared memory, completing on bar.
__device__ __forceinline__ void tma_load_2d(unsigned dst, const CUtensorMap* map, int x, int y, unsigned bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzle layout: rows of
// 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), version 1, layout SWIZZLE_128B.
// The leading byte offset is unused for this layout.
__device__ __forceinline__ unsigned long long smem_desc(unsigned addr) {
  return static_cast<unsigned long long>((addr & 0x3FFFFu) >> 4) | (1ull << 16) | (static_cast<unsigned long long>(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both K-major, N, M = 128.
__device__ __forceinline__ unsigned instr_desc(int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<unsigned>(N >> 3) << 17) | (static_cast<unsigned>(kM >> 4) << 24);
}
__device__ __forceinline__ void mma(unsigned tmem_d, unsigned long long adesc, unsigned long long bdesc, unsigned idesc,
                                    bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
__device__ __forceinline__ void commit(unsigned bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 accumulator columns of this thread's row (lane) into v.
__device__ __forceinline__ void tmem_ld32(unsigned taddr, float (&v)[32]) {
  unsigned r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Adds the three term columns of sequences [b0, b0 + 32) of accumulator region `region`
// (tensor-memory address of this warp's rows) into acc.
__device__ __forceinline__ void read_group(unsigned tw, int B, int b0, float (&acc)[32]) {
  float t[32];
#pragma unroll
  for (int term = 0; term < 3; ++term) {
    tmem_ld32(tw + static_cast<unsigned>(term * B + b0), t);
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] += t[j];
  }
}

template <bool DENSE, int NB>  // NB: sequences / 32 (1 or 2)
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX, const Args a) {
  extern __shared__ __align__(1024) char sm_raw[];
  // programmatic dependent launch: the next kernel may start launching; the producer waits
  // for this kernel's predecessors only before its first read of the staged operand (the
  // weights do not depend on them), and every other read or write follows from that
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const unsigned raw = sa(sm_raw);
  const unsigned base = (raw + 1023u) & ~1023u;  // the swizzle layout needs 1024-byte alignment
  const int B = NB * 32, N = 3 * B, SB = stage_bytes(B), ncols = tmem_cols(B);
  // this CTA's share of K (split over the S CTAs of a cluster): stages [kt_lo, kt_lo + KT)
  const int S = DENSE ? 1 : (a.splits > 1 ? a.splits : 1);
  const int sp = static_cast<int>(blockIdx.x) % S, KTall = a.K / kKStage;
  const int kt_lo = KTall * sp / S, KT = KTall * (sp + 1) / S - kt_lo;
  const int NG = (KT + kGroup - 1) / kGroup;  // k groups
  const unsigned full0 = base + kStages * SB, empty0 = full0 + 8 * kStages;
  const unsigned gdone0 = empty0 + 8 * kStages, gfree0 = gdone0 + 16;  // per accumulator region
  const unsigned tslot = gfree0 + 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, tile = static_cast<int>(blockIdx.x) / S;
  const bool hi = a.R1 > 0 && tile * kM >= a.R1;  // this tile's rows belong to the second matrix

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(gdone0 + 8 * r, 1);             // tcgen05.commit of the group's last MMAs
      mbar_init(gfree0 + 8 * r, kEpiWarps);      // every epilogue warp has read the region back
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tslot), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  unsigned taddr;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(taddr) : "r"(tslot));

  if (warp == kEpiWarps) {
    if (lane == 0) {
      // ---- producer: W tile rows and all of Xs, 64 columns per stage. The first stages' W
      // tiles are requested before the wait for the kernels that write Xs.
      // testing: with dbg_cta this CTA issues no copy for its last stage (the MMA warp's wait
      // on it runs out)
      const int last = static_cast<int>(blockIdx.x) == a.dbg_cta ? KT - 1 : KT;
      const int pre = min(last, kStages);
      for (int kt = 0; kt < pre; ++kt) {
        mbar_expect_tx(full0 + 8 * kt, static_cast<unsigned>(SB));
        tma_load_2d(base + kt * SB, &mapW, (kt_lo + kt) * kKStage, tile * kM, full0 + 8 * kt);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int kt = 0; kt < pre; ++kt)
        tma_load_2d(base + kt * SB + kM * kKStage * 2, &mapX, (kt_lo + kt) * kKStage, 0, full0 + 8 * kt);
      int issued = pre;
      for (int kt = pre; kt < last; ++kt) {
        const int s = kt % kStages;
        if (!wait_bar(empty0 + 8 * s, static_cast<unsigned>((kt / kStages - 1) & 1), a.status, a.spin_limit))
          break;
        const unsigned st = base + s * SB;
        mbar_expect_tx(full0 + 8 * s, static_cast<unsigned>(SB));
        tma_load_2d(st, &mapW, (kt_lo + kt) * kKStage, tile * kM, full0 + 8 * s);
        tma_load_2d(st + kM * kKStage * 2, &mapX, (kt_lo + kt) * kKStage, 0, full0 + 8 * s);
        ++issued;
      }
      // no copy may still be in flight when the CTA ends
      for (int kt = issued > kStages ? issued - kStages : 0; kt < issued; ++kt)
        wait_bar(full0 + 8 * (kt % kStages), static_cast<unsigned>((kt / kStages) & 1), a.status, a.spin_limit);
    }
    __syncwarp();
  } else if (warp == kEpiWarps + 1) {
    if (lane == 0) {
      // ---- MMA issue: 4 x (K = 16) per stage; group g accumulates in region g % 2
      const unsigned idesc = instr_desc(N);
      bool ok = true;
      for (int g = 0; g < NG && ok; ++g) {
        const int region = g & 1;
        // the region's previous group (g - 2) must have been read back
        if (g >= 2 && !wait_bar(gfree0 + 8 * region, static_cast<unsigned>((g / 2 - 1) & 1), a.status, a.spin_limit)) {
          ok = false;
          break;
        }
        fence_after();
        const unsigned td = taddr + static_cast<unsigned>(region * N);
        for (int kt = g * kGroup; kt < min(KT, (g + 1) * kGroup); ++kt) {
          const int s = kt % kStages;
          if (!wait_bar(full0 + 8 * s, static_cast<unsigned>((kt / kStages) & 1), a.status, a.spin_limit)) {
            ok = false;
            break;
          }
          fence_after();
          const unsigned st = base + s * SB;
#pragma unroll
          for (int kk = 0; kk < kKStage / 16; ++kk)
            mma(td, smem_desc(st + kk * 32), smem_desc(st + kM * kKStage * 2 + kk * 32), idesc,
                kt > g * kGroup || kk > 0);
          commit(empty0 + 8 * s);  // the stage is free once these MMAs are done
        }
        commit(gdone0 + 8 * region);  // the group's sums are complete once its MMAs are done
      }
    }
    __syncwarp();
  } else {
  // ---- epilogue: warp w reads rows 32w..32w+31 of each finished group and sums the groups
  const int r = tile * kM + 32 * warp + lane;
  float acc[NB][32];
#pragma unroll
  for (int q = 0; q < NB; ++q)
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[q][j] = 0.f;
  for (int g = 0; g < NG; ++g) {
    const int region = g & 1;
    wait_bar(gdone0 + 8 * region, static_cast<unsigned>((g / 2) & 1), a.status, a.spin_limit);
    fence_after();
    const unsigned tw = taddr + (static_cast<unsigned>(32 * warp) << 16) + static_cast<unsigned>(region * N);
#pragma unroll
    for (int q = 0; q < NB; ++q) read_group(tw, B, 32 * q, acc[q]);
    fence_before();
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(gfree0 + 8 * region) : "memory");
  }
  if (!DENSE && S > 1) {
    // this row's partial sums into this CTA's stage memory (pitch B + 1 floats: conflict-free)
    float* pbuf = reinterpret_cast<float*>(sm_raw + (base - raw));
    const int row = 32 * warp + lane;
#pragma unroll
    for (int q = 0; q < NB; ++q)
#pragma unroll
      for (int j = 0; j < 32; ++j) pbuf[row * (B + 1) + 32 * q + j] = acc[q][j];
  }
  if (!DENSE && S == 1 && a.glu_xs) {
    // gated GELU: warps 2..3 hold the up rows of the gate rows of warps 0..1; they pass them
    // through the idle stage memory (every MMA has completed, every copy has landed)
    float* pbuf = reinterpret_cast<float*>(sm_raw + (base - raw));
    const int row = 32 * warp + lane;
    if (warp >= 2) {
#pragma unroll
      for (int q = 0; q < NB; ++q)
#pragma unroll
        for (int j = 0; j < 32; ++j) pbuf[(row - 64) * (B + 1) + 32 * q + j] = acc[q][j];
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
    const int f = 64 * tile + row;
    if (warp < 2 && f < a.glu_K) {
#pragma unroll
      for (int q = 0; q < NB; ++q)
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (32 * q + j < a.nvalid)
            stage_terms(a.glu_xs, a.glu_bp, a.glu_K, 32 * q + j, f,
                        gelu_tanh(acc[q][j]) * pbuf[row * (B + 1) + 32 * q + j]);
    }
  } else if (DENSE || S == 1) {
#pragma unroll
  for (int q = 0; q < NB; ++q) {
    const int b0 = 32 * q;
    if (!DENSE) {
      if (r < a.R) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (b0 + j < a.nvalid) {
            if (hi) {
              a.out_hi[static_cast<size_t>(b0 + j) * a.ld_hi + (r - a.R1)] = acc[q][j];
            } else {
              if (a.out) a.out[static_cast<size_t>(b0 + j) * a.ldo + r] = acc[q][j];
              if (a.out2) a.out2[static_cast<size_t>(b0 + j) * a.ld2 + r] = acc[q][j];
            }
          }
        }
      }
    } else {
      // argmax keys: a transposing max leaves in lane l the best key of sequence b0 + l
      unsigned long long k[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) k[j] = r < a.R ? argmax_key(acc[q][j], r) : 0ull;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
          const unsigned long long send = up ? k[i] : k[i + off];
          const unsigned long long keep = up ? k[i + off] : k[i];
          const unsigned long long got = __shfl_xor_sync(0xffffffffu, send, off);
          k[i] = got > keep ? got : keep;
        }
      }
      if (b0 + lane < a.nvalid) atomicMax(a.best + b0 + lane, k[0]);
    }
  }
  }
  }  // epilogue warps
  if (!DENSE && S > 1) {
    // every CTA of the cluster has its partials in place (the stage memory is idle: every MMA
    // has completed and every copy has landed); CTA sp adds the S partials of its rows in
    // order 0..S-1 and stores them; a second barrier keeps the partials alive until then
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (tid < kEpiWarps * 32 && a.glu_xs) {
      // gated GELU: CTA sp sums the S partials of its gate rows i and of the up rows i + 64
      const unsigned pb = base;
      const int i_lo = 64 * sp / S, i_hi = 64 * (sp + 1) / S, ni = i_hi - i_lo;
      for (int e = tid; e < ni * a.nvalid; e += kEpiWarps * 32) {
        const int i = i_lo + e / a.nvalid, b = e % a.nvalid;
        const unsigned og = pb + 4u * static_cast<unsigned>(i * (B + 1) + b);
        const unsigned ou = pb + 4u * static_cast<unsigned>((i + 64) * (B + 1) + b);
        float g = 0.f, u = 0.f;
        for (int s2 = 0; s2 < S; ++s2) {
          unsigned rg, ru;
          asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rg) : "r"(og), "r"(s2));
          asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ru) : "r"(ou), "r"(s2));
          float x, y;
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(x) : "r"(rg) : "memory");
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(y) : "r"(ru) : "memory");
          g += x;
          u += y;
        }
        const int f = 64 * tile + i;
        if (f < a.glu_K) stage_terms(a.glu_xs, a.glu_bp, a.glu_K, b, f, gelu_tanh(g) * u);
      }
    } else if (tid < kEpiWarps * 32) {
      const unsigned pb = base;
      const int r_lo = kM * sp / S, r_hi = kM * (sp + 1) / S, nrow = r_hi - r_lo;
      for (int e = tid; e < nrow * a.nvalid; e += kEpiWarps * 32) {
        const int rr = r_lo + e / a.nvalid, b = e % a.nvalid;
        const unsigned off = pb + 4u * static_cast<unsigned>(rr * (B + 1) + b);
        float v = 0.f;
        for (int s2 = 0; s2 < S; ++s2) {
          unsigned ra;
          asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(off), "r"(s2));
          float x;
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(x) : "r"(ra) : "memory");
          v += x;
        }
        const int r = tile * kM + rr;
        if (r < a.R) {
          if (hi) {
            a.out_hi[static_cast<size_t>(b) * a.ld_hi + (r - a.R1)] = v;
          } else {
            if (a.out) a.out[static_cast<size_t>(b) * a.ldo + r] = v;
            if (a.out2) a.out2[static_cast<size_t>(b) * a.ld2 + r] = v;
          }
        }
      }
    }
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  }
}

}  // namespace tc

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cudaGetLastError();
  });
  return g_encode;
}

}  // namespace

bool tc_available() {
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return major == 10 && encoder() != nullptr;
}

int tc_make_map(CUtensorMap* map, const void* base, long long rows, long long cols, long long pitch, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return MTP_ERR_CUDA;
  }
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(pitch * 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(tc::kKStage), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for a %lld x %lld bf16 matrix", static_cast<int>(r), rows, cols);
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

int tc_gemm(const CUtensorMap* mapW, const CUtensorMap* mapX, const tc::Args& a, bool dense, cudaStream_t st,
            bool pdl) {
  if (a.B < 32 || a.B > tc::kMaxB || a.B % 32 || a.nvalid < 1 || a.nvalid > a.B || a.K < tc::kKStage ||
      a.K % tc::kKStage || a.R < 1) {
    set_error("tensor-core GEMM: unsupported R=%d K=%d B=%d", a.R, a.K, a.B);
    return MTP_ERR_UNSUPPORTED_SHAPE;
  }
  if (a.glu_xs && (dense || a.R1 != 0 || a.R % tc::kM || a.glu_K * 2 != a.R || a.glu_bp < a.nvalid)) {
    set_error("tensor-core GEMM: unsupported gated-GELU epilogue R=%d glu_K=%d", a.R, a.glu_K);
    return MTP_ERR_UNSUPPORTED_SHAPE;
  }
  if (a.R1 != 0 && (dense || a.R1 < 0 || a.R1 % tc::kM || a.R1 >= a.R || !a.out_hi)) {
    set_error("tensor-core GEMM: unsupported stacked split R1=%d of R=%d", a.R1, a.R);
    return MTP_ERR_UNSUPPORTED_SHAPE;
  }
  const int smem = tc::smem_bytes(a.B);
  auto kern = a.B == 32 ? (dense ? tc::k_tc_gemm<true, 1> : tc::k_tc_gemm<false, 1>)
                        : (dense ? tc::k_tc_gemm<true, 2> : tc::k_tc_gemm<false, 2>);
  const int tiles = (a.R + tc::kM - 1) / tc::kM, KT = a.K / tc::kKStage;
  tc::Args aa = a;
  if (dense) {
    aa.splits = 1;
  } else if (aa.splits <= 0) {  // about one wave of CTAs, at least one k stage each, clusters of <= 8
    int S = 1;
    while (2 * S <= 8 && 2 * S <= KT && tiles * 2 * S <= 128) S *= 2;
    aa.splits = S;
  }
  if (aa.splits > 8 || aa.splits > KT || (aa.splits > 1 && (a.B + 1) * tc::kM * 4 > tc::kStages * tc::stage_bytes(a.B))) {
    set_error("tensor-core GEMM: unsupported split %d of K=%d", aa.splits, a.K);
    return MTP_ERR_UNSUPPORTED_SHAPE;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles * aa.splits);
    cfg.blockDim = dim3(tc::kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = aa.splits;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // pdl_enter waits
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, *mapW, *mapX, aa);
  }
  if (e != cudaSuccess) {
    set_error("tensor-core GEMM launch: %s", cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

}  // namespace mtp
