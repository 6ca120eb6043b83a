// gdn_verify_k16_k32.cu -- verify and native-snapshot kernels for head widths 16 and 32, both gate kinds.
#include "gdn_verify_impl.cuh"

namespace gdn {

int launch_verify_k16(const VerifyParams& p, int qkv_dtype, int state_dtype, bool native,
                     cudaStream_t stream) {
  return dispatch_native<16, false>(p, qkv_dtype, state_dtype, native, stream);
}

int launch_verify_k16_kda(const VerifyParams& p, int qkv_dtype, int state_dtype, bool native,
                         cudaStream_t stream) {
  return dispatch_native<16, true>(p, qkv_dtype, state_dtype, native, stream);
}

int launch_verify_k32(const VerifyParams& p, int qkv_dtype, int state_dtype, bool native,
                     cudaStream_t stream) {
  return dispatch_native<32, false>(p, qkv_dtype, state_dtype, native, stream);
}

int launch_verify_k32_kda(const VerifyParams& p, int qkv_dtype, int state_dtype, bool native,
                         cudaStream_t stream) {
  return dispatch_native<32, true>(p, qkv_dtype, state_dtype, native, stream);
}

}  // namespace gdn
