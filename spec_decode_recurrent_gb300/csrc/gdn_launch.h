// gdn_launch.h -- internal launchers behind the C ABI of libgdn_spec.so.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace gdn {

struct VerifyParams;
struct CommitParams;
struct ConvParams;

int launch_verify(const VerifyParams& p, int head_k, int qkv_dtype, int state_dtype,
                  bool native, cudaStream_t stream);
int launch_commit(const CommitParams& p, int head_k, int state_dtype, cudaStream_t stream);
int launch_conv_commit(const ConvParams& p, int dtype, cudaStream_t stream);

size_t verify_smem_bytes(int head_k, int W);
int verify_rows_per_cta(int head_k);
size_t commit_smem_bytes(int head_k, int head_v, int W);

}  // namespace gdn
