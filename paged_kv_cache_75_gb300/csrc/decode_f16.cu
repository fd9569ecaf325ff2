// fp16 queries over an fp16 KV cache.
#include "decode_launch.cuh"
namespace pa {
pa_status launch_decode_f16(const DecodeParams& p, int head_size, int group, cudaStream_t s) {
    return launch_decode_dtype<PA_F16, PA_F16>(p, head_size, group, s);
}
}  // namespace pa
