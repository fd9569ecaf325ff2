// bf16 queries over a bf16 KV cache.
#include "decode_launch.cuh"
namespace pa {
pa_status launch_decode_bf16(const DecodeParams& p, int head_size, int group, cudaStream_t s) {
    return launch_decode_dtype<PA_BF16, PA_BF16>(p, head_size, group, s);
}
}  // namespace pa
