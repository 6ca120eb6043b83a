// gdn_verify.cu -- dispatch of a verify or native-snapshot call to the
// translation unit that holds its head width and gate kind (the kernels are
// in gdn_verify_impl.cuh).
#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {

int launch_verify(const VerifyParams& p, int head_k, int qkv_dtype, int state_dtype,
                  bool native, bool kda, cudaStream_t stream) {
  switch (head_k) {
    case 16:
      return kda ? launch_verify_k16_kda(p, qkv_dtype, state_dtype, native, stream)
                 : launch_verify_k16(p, qkv_dtype, state_dtype, native, stream);
    case 32:
      return kda ? launch_verify_k32_kda(p, qkv_dtype, state_dtype, native, stream)
                 : launch_verify_k32(p, qkv_dtype, state_dtype, native, stream);
    case 64:
      return kda ? launch_verify_k64_kda(p, qkv_dtype, state_dtype, native, stream)
                 : launch_verify_k64(p, qkv_dtype, state_dtype, native, stream);
    case 128:
      return kda ? launch_verify_k128_kda(p, qkv_dtype, state_dtype, native, stream)
                 : launch_verify_k128(p, qkv_dtype, state_dtype, native, stream);
    default:
      return GDN_ERR_UNSUPPORTED;
  }
}

}  // namespace gdn
