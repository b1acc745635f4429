// Drafter-step kernels instantiated for model dtype __nv_bfloat16.
#include "mtp_kernels.cuh"

namespace mtp {
int run_phases_bf16(const Params& p, cudaStream_t st) { return run_phases<__nv_bfloat16>(p, st); }
int run_phases_tc_bf16(const Params& p, const TcPlan& plan, cudaStream_t st) {
  return run_phases_tc<__nv_bfloat16>(p, plan, st);
}
int run_persistent_bf16(const Params& p, cudaStream_t st) { return run_persistent<__nv_bfloat16>(p, st); }
int persistent_capacity_bf16(const Params& p, int num_sms) { return persistent_capacity<__nv_bfloat16>(p, num_sms); }
int run_head_bf16(const Params& p, cudaStream_t st) { return run_head<__nv_bfloat16>(p, st); }
}  // namespace mtp
