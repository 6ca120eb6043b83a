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
// One head width and gate kind each (gdn_verify_k*.cu).
#define GDN_VERIFY_UNIT(name)                                                          \
  int name(const VerifyParams& p, int qkv_dtype, int state_dtype, bool native,      \
           cudaStream_t stream);
GDN_VERIFY_UNIT(launch_verify_k16)
GDN_VERIFY_UNIT(launch_verify_k16_kda)
GDN_VERIFY_UNIT(launch_verify_k32)
GDN_VERIFY_UNIT(launch_verify_k32_kda)
GDN_VERIFY_UNIT(launch_verify_k64)
GDN_VERIFY_UNIT(launch_verify_k64_kda)
GDN_VERIFY_UNIT(launch_verify_k128)
GDN_VERIFY_UNIT(launch_verify_k128_kda)
#undef GDN_VERIFY_UNIT
int launch_commit(const CommitParams& p, int head_k, int state_dtype, bool kda,
                  cudaStream_t stream);
int launch_conv_commit(const ConvParams& p, int dtype, cudaStream_t stream);

}  // namespace gdn
