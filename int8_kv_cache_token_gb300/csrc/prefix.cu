// prefix.cu -- placeholder launchers (filled in by the prefix and BF16 kernels).
#include "common.cuh"
#include "kernels.h"
namespace i8kv {
I8KV_DEFINE_ERROR_ACCESSOR(read_error_prefix)
cudaError_t launch_int8_prefix(const PrefixParams&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_bf16_decode(const DecodeParams&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace i8kv
