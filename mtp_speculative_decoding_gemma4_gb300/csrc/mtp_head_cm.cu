// Cluster-major sparse head, streamed ("Gemma 4 Assistant tensor inventory", "Centroid /
// ordered embeddings LM head", steps 3-4: the candidate token ids of the selected centroids
// and the logits of their token_embd rows; the argmax follows the draft-step rule, lowest
// vocab id on ties).
//
// Every centroid that at least one sequence of the batch selected this step is visited once:
// its vsc rows are one contiguous block of the token_embd copy in token_ordering order, so a
// CTA fetches them in chunks with single bulk copies (rows and their vocab ids in one ring
// stage, completing on one mbarrier) and scores each chunk for all sequences that selected the
// centroid. A row that several sequences selected crosses HBM once per step.
//
// Work split: each CTA counts the step's selections (B x top_k ids, L2-resident) into a
// shared histogram, numbers the selected centroids in increasing order, and takes numbers
// cta, cta + grid, ...: every CTA gets the same number of centroids to within one. It then
// lists, for each of its centroids, the sequences that chose it. One CTA per SM; y of the whole
// batch arrives by one more bulk copy. 8 warps score 8-row batches of a chunk (a lane holds
// one 16-byte slice of every row; a reduce-scatter over the lanes leaves row (lane >> 2) & 7's
// logit in lanes 4r..4r+3). The best (logit, id) key of every listed sequence is reduced per
// centroid (a warp maximum, then one shared atomicMax per warp) before one atomicMax into the
// step's per-sequence key.
//
// Failure handling: a wait on a bulk copy gives up after spin_limit cycles, records
// MTP_ERR_TIMEOUT in the status word, waits (bounded) for the copies still in flight and
// returns.

#include "mtp_launch.h"
#include "mtp_phases.cuh"

namespace mtp {
namespace hcm {

constexpr int kRowsPerWarp = 8;                 // rows of one warp batch
constexpr int kRowsPerPass = kWarps * kRowsPerWarp;  // rows the CTA scores side by side
constexpr int kStageRowBytes = 32768;          // row bytes per ring stage (at most)
constexpr int kMaxStages = 4;

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
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
__device__ __forceinline__ bool try_wait(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}
// Bounded wait for a stage; false after `limit` cycles.
__device__ __forceinline__ bool wait_stage(unsigned bar, unsigned parity, long long limit) {
  const long long t0 = clock64();
  while (!try_wait(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}

// Geometry of the ring and of the shared-memory carve-up, shared by host and device.
struct Geo {
  int rows;         // rows per chunk (a multiple of 8 that divides vsc)
  int nchk;         // chunks per centroid
  int row_bytes;    // H * element size
  int stage_bytes;  // rows + their ids
  int stages;
  int mine;         // centroids per CTA (upper bound)
  int grid;
  int smem;         // dynamic shared memory bytes (0: unsupported)
};

__host__ __device__ inline int align16(int v) { return (v + 15) & ~15; }

// Bytes after the ring: y [B][H] fp32 | kb [2][B] u64 | map [C] | list, lcnt, fill [mine] |
// seqs [mine][B] | mbarriers [kMaxStages + 1] | scan scratch and flags.
__host__ __device__ inline int tail_bytes(const ShapeP& s, int mine) {
  return s.B * s.H * 4 + 2 * s.B * 8 + align16(s.C * 4) + align16(3 * mine * 4) + align16(mine * s.B * 4) +
         (kMaxStages + 1) * 8 + (kWarps + 4) * 4;
}

__host__ __device__ inline Geo geometry(const ShapeP& s, int eb) {
  Geo g{};
  g.row_bytes = s.H * eb;
  g.grid = s.nsm < s.C ? s.nsm : s.C;
  if (g.grid < 1 || s.vsc < 8 || g.row_bytes % 16 != 0 || s.vsc % 8 != 0 || s.B < 1 || s.topk < 1) return g;
  int rows = kStageRowBytes / g.row_bytes;
  rows -= rows % 8;
  if (rows > s.vsc) rows = s.vsc;
  while (rows > 8 && s.vsc % rows != 0) rows -= 8;
  if (rows < 8) return g;
  g.rows = rows;
  g.nchk = s.vsc / rows;
  g.stage_bytes = rows * g.row_bytes + rows * 4;
  const int selected = s.B * s.topk < s.C ? s.B * s.topk : s.C;
  g.mine = (selected + g.grid - 1) / g.grid;
  const int tail = tail_bytes(s, g.mine);
  for (int st = kMaxStages; st >= 2; --st) {
    const int total = st * g.stage_bytes + tail + 128;
    if (total <= 227 * 1024) {
      g.stages = st;
      g.smem = total;
      return g;
    }
  }
  return g;
}

template <typename WT>
__global__ void __launch_bounds__(kThreads, 1) k_head_cm(Params p, Geo g) {
  pdl_enter();
  extern __shared__ __align__(128) char smem_raw[];
  constexpr int V = Elem<WT>::kVec;  // elements per 16-byte slice
  const int H = p.s.H, vsc = p.s.vsc, C = p.s.C, B = p.s.B, K = p.s.topk, nsel = B * K;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, grid = gridDim.x;
  char* stage0 = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  float* ys = reinterpret_cast<float*>(stage0 + g.stages * g.stage_bytes);
  unsigned long long* kb = reinterpret_cast<unsigned long long*>(ys + B * H);
  int* map = reinterpret_cast<int*>(kb + 2 * B);
  int* list = map + (align16(C * 4) >> 2);
  int* lcnt = list + g.mine;
  int* fill = lcnt + g.mine;
  int* seqs = list + (align16(3 * g.mine * 4) >> 2);
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(seqs + (align16(g.mine * B * 4) >> 2));
  int* scan = reinterpret_cast<int*>(bars + kMaxStages + 1);  // [kWarps] warp totals
  int* flags = scan + kWarps;                                 // [0] selected centroids, [1] abort
  const unsigned bar0 = smem_u32(bars), ybar = bar0 + 8 * kMaxStages;

  if (tid == 0) {
    for (int s = 0; s <= kMaxStages; ++s) mbar_init(bar0 + 8 * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    flags[1] = 0;
    // y of every sequence: one bulk copy, overlapping the bookkeeping below
    mbar_expect_tx(ybar, static_cast<unsigned>(B * H * 4));
    bulk_g2s(smem_u32(ys), p.w.y, static_cast<unsigned>(B * H * 4), ybar);
  }
  // 1. histogram of the step's selected centroids
  for (int i = tid; i < C; i += kThreads) map[i] = 0;
  for (int i = tid; i < 2 * B; i += kThreads) kb[i] = 0ull;
  __syncthreads();
  for (int i0 = tid; i0 < nsel; i0 += 8 * kThreads) {
    int cs[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int i = i0 + t * kThreads;
      cs[t] = i < nsel ? __ldg(p.w.sel + i) : -1;
    }
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (cs[t] >= 0 && cs[t] < C) atomicAdd(map + cs[t], 1);
  }
  __syncthreads();
  // 2. number the selected centroids in increasing order; this CTA takes numbers cta + i * grid
  const int per = (C + kThreads - 1) / kThreads, c0 = tid * per, c1 = min(c0 + per, C);
  int n = 0;
  for (int c = c0; c < c1; ++c) n += map[c] > 0;
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scan[warp] = incl;
  __syncthreads();
  int u = incl - n, all = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) u += scan[w];
    all += scan[w];
  }
  for (int c = c0; c < c1; ++c) {
    const int m = map[c];
    int slot = -1;
    if (m > 0) {
      if (u % grid == cta) {
        slot = u / grid;
        list[slot] = c;
        lcnt[slot] = min(m, B);
        fill[slot] = 0;
      }
      ++u;
    }
    map[c] = slot;
  }
  const int nw = all > cta ? (all - cta + grid - 1) / grid : 0;
  const int total = nw * g.nchk;
  __syncthreads();
  const WT* temb = static_cast<const WT*>(p.temb_ord);
  const int rows_bytes = g.rows * g.row_bytes;
  auto issue = [&](int j) {  // chunk j of the CTA's work into its ring stage (thread 0)
    const int r0 = list[j / g.nchk] * vsc + (j % g.nchk) * g.rows;
    const unsigned st = smem_u32(stage0 + (j % g.stages) * g.stage_bytes);
    const unsigned bar = bar0 + 8 * (j % g.stages);
    mbar_expect_tx(bar, static_cast<unsigned>(rows_bytes + g.rows * 4));
    bulk_g2s(st, temb + static_cast<size_t>(r0) * H, rows_bytes, bar);
    bulk_g2s(st + rows_bytes, p.ord + r0, g.rows * 4u, bar);
  };
  if (tid == 0)
    for (int j = 0; j < g.stages && j < total; ++j) issue(j);
  // 3. the sequences of each of this CTA's centroids (the order within a list is free)
  for (int i = tid; i < nsel; i += kThreads) {
    const int c = __ldg(p.w.sel + i);
    const int slot = (c >= 0 && c < C) ? map[c] : -1;
    if (slot >= 0) {
      const int pos = atomicAdd(fill + slot, 1);
      if (pos < B) seqs[slot * B + pos] = i / K;
    }
  }
  bool ok = wait_stage(ybar, 0u, p.spin_limit);
  if (!ok) flags[1] = 1;
  __syncthreads();

  int j = 0;
  if (!flags[1]) {
    for (; j < total; ++j) {
      const int uu = j / g.nchk, q = j % g.nchk;
      const int m = lcnt[uu];
      const int* sq = seqs + uu * B;
      const char* st = stage0 + (j % g.stages) * g.stage_bytes;
      const int* ids = reinterpret_cast<const int*>(st + rows_bytes);
      unsigned long long* kbuf = kb + (uu & 1) * B;
      if (!wait_stage(bar0 + 8 * (j % g.stages), static_cast<unsigned>((j / g.stages) & 1), p.spin_limit))
        flags[1] = 1;
      __syncthreads();
      if (flags[1]) break;
      for (int rb = warp * kRowsPerWarp; rb < g.rows; rb += kRowsPerPass) {
        const WT* rows = reinterpret_cast<const WT*>(st) + static_cast<size_t>(rb) * H;
        const int rid = ids[rb + ((lane >> 2) & (kRowsPerWarp - 1))];
        for (int s0 = 0; s0 < m; s0 += 2) {
          const int ns = m - s0 >= 2 ? 2 : 1;
          const float* y0 = ys + sq[s0] * H;
          const float* y1 = ys + sq[s0 + ns - 1] * H;
          float a0[kRowsPerWarp], a1[kRowsPerWarp];
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r) a0[r] = a1[r] = 0.f;
          for (int k = lane * V; k < H; k += 32 * V) {
            float yv0[V], yv1[V];
#pragma unroll
            for (int v = 0; v < V; v += 4) {
              const float4 f0 = *reinterpret_cast<const float4*>(y0 + k + v);
              const float4 f1 = *reinterpret_cast<const float4*>(y1 + k + v);
              yv0[v] = f0.x; yv0[v + 1] = f0.y; yv0[v + 2] = f0.z; yv0[v + 3] = f0.w;
              yv1[v] = f1.x; yv1[v + 1] = f1.y; yv1[v + 2] = f1.z; yv1[v + 3] = f1.w;
            }
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
              const uint4 raw = *reinterpret_cast<const uint4*>(rows + static_cast<size_t>(r) * H + k);
              float w[V];
              if constexpr (V == 8) {
                vec_to_f32(raw, w);
              } else {
                w[0] = __uint_as_float(raw.x); w[1] = __uint_as_float(raw.y);
                w[2] = __uint_as_float(raw.z); w[3] = __uint_as_float(raw.w);
              }
#pragma unroll
              for (int v = 0; v < V; ++v) {
                a0[r] = fmaf(w[v], yv0[v], a0[r]);
                a1[r] = fmaf(w[v], yv1[v], a1[r]);
              }
            }
          }
          reduce_scatter<kRowsPerWarp, 16>(a0, lane);
          reduce_scatter<kRowsPerWarp, 16>(a1, lane);
          if (p.out_logits && (lane & 3) == 0) {  // one lane per row
            p.out_logits[static_cast<size_t>(sq[s0]) * p.s.V + rid] = a0[0];
            if (ns == 2) p.out_logits[static_cast<size_t>(sq[s0 + 1]) * p.s.V + rid] = a1[0];
          }
          // the warp's best key per sequence (over the row bits 2..4 of the lane), one atomic
          unsigned long long k0 = argmax_key(a0[0], rid), k1 = argmax_key(a1[0], rid);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            const unsigned long long t0 = __shfl_xor_sync(0xffffffffu, k0, o);
            const unsigned long long t1 = __shfl_xor_sync(0xffffffffu, k1, o);
            k0 = t0 > k0 ? t0 : k0;
            k1 = t1 > k1 ? t1 : k1;
          }
          if (lane == 0) {
            atomicMax(kbuf + s0, k0);
            if (ns == 2) atomicMax(kbuf + s0 + 1, k1);
          }
        }
      }
      __syncthreads();  // the stage is free; this chunk's keys are in kbuf
      if (tid == 0 && j + g.stages < total) issue(j + g.stages);
      if (q == g.nchk - 1)  // the centroid is done: its keys to the step's keys
        for (int i = tid; i < m; i += kThreads) {
          atomicMax(p.w.best + sq[i], kbuf[i]);
          kbuf[i] = 0ull;
        }
    }
  }
  if (flags[1]) {
    // gave up: record it, then wait (bounded) for the copies still in flight
    if (tid == 0) {
      atomicExch(p.w.status, static_cast<int>(MTP_ERR_TIMEOUT));
      wait_stage(ybar, 0u, p.spin_limit);
      for (int jj = j; jj < total && jj < j + g.stages; ++jj)
        wait_stage(bar0 + 8 * (jj % g.stages), static_cast<unsigned>((jj / g.stages) & 1), p.spin_limit);
    }
    __syncthreads();
  }
}

}  // namespace hcm

template <typename WT>
int run_head_cm(const Params& p, cudaStream_t st) {
  const hcm::Geo g = hcm::geometry(p.s, static_cast<int>(sizeof(WT)));
  if (!head_cm_supported(p, static_cast<int>(sizeof(WT)))) {
    set_error("cluster-major sparse head: shape not supported (vsc %d, H %d, B %d)", p.s.vsc, p.s.H, p.s.B);
    return MTP_ERR_UNSUPPORTED_SHAPE;
  }
  cudaError_t e = cudaFuncSetAttribute(hcm::k_head_cm<WT>, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem);
  if (e == cudaSuccess) {
    hcm::k_head_cm<WT><<<g.grid, kThreads, g.smem, st>>>(p, g);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("cluster-major sparse head (%d CTAs, %d B smem): %s", g.grid, g.smem, cudaGetErrorString(e));
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

bool head_cm_supported(const Params& p, int elem_bytes) {
  return hcm::geometry(p.s, elem_bytes).smem > 0 && p.temb_ord && p.ord &&
         reinterpret_cast<uintptr_t>(p.ord) % 16 == 0 && reinterpret_cast<uintptr_t>(p.temb_ord) % 16 == 0;
}

template int run_head_cm<__nv_bfloat16>(const Params&, cudaStream_t);
template int run_head_cm<float>(const Params&, cudaStream_t);

}  // namespace mtp
