// Internal interface between the C ABI (mtp_api.cu) and the dtype-specific kernel
// translation units (mtp_bf16.cu, mtp_f32.cu, mtp_verify.cu).
#pragma once

#include <cuda_runtime.h>

#include "mtp.h"

namespace mtp {

struct Params;
namespace ll {
struct Params;
}

// Records the calling thread's last error text (printf-style).
void set_error(const char* fmt, ...);

int run_phases_bf16(const Params& p, cudaStream_t st);
int run_persistent_bf16(const Params& p, cudaStream_t st);
int persistent_capacity_bf16(const Params& p, int num_sms);
int run_head_bf16(const Params& p, cudaStream_t st);

int run_phases_f32(const Params& p, cudaStream_t st);
int run_persistent_f32(const Params& p, cudaStream_t st);
int persistent_capacity_f32(const Params& p, int num_sms);
int run_head_f32(const Params& p, cudaStream_t st);

// Latency-path draft block (one sequence): shared-memory bytes it needs for these
// parameters (0: shape not supported), co-resident capacity for that size, launch.
int ll_smem_bytes(const ll::Params& p);
int ll_capacity(int smem, int num_sms);
int run_ll(const ll::Params& p, int smem, cudaStream_t st);

int run_verify(const void* logits, const int* draft, int B, int n, int V, int* accept_len, int* out_tokens,
               cudaStream_t st);

}  // namespace mtp
