// gdn_launch.h -- internal launchers behind the C ABI of libgdn_spec.so.
#pragma once

#include <cuda_runtime.h>

namespace gdn {

struct VerifyParams;
struct CommitParams;
struct ConvParams;

// kda: per-channel decay (gates a [T][HV][K], dt_bias [HV][K], record
// gates [B][HV][W][K]) instead of the scalar decay.
int launch_verify(const VerifyParams& p, int head_k, int qkv_dtype, int state_dtype,
                  bool native, bool kda, cudaStream_t stream);
int launch_commit(const CommitParams& p, int head_k, int state_dtype, bool kda,
                  cudaStream_t stream);
int launch_conv_commit(const ConvParams& p, int dtype, cudaStream_t stream);

}  // namespace gdn
