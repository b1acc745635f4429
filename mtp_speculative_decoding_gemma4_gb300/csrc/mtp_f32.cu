// Drafter-step kernels instantiated for model dtype float.
#include "mtp_kernels.cuh"

namespace mtp {
int run_phases_f32(const Params& p, cudaStream_t st) { return run_phases<float>(p, st); }
int run_persistent_f32(const Params& p, cudaStream_t st) { return run_persistent<float>(p, st); }
int persistent_capacity_f32(const Params& p, int num_sms) { return persistent_capacity<float>(p, num_sms); }
int run_head_f32(const Params& p, cudaStream_t st) { return run_head<float>(p, st); }
}  // namespace mtp
