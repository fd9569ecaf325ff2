// fp16 queries over an fp16 KV cache, block size 64.
#include "decode_launch.cuh"
namespace pa {
pa_status launch_decode_f16_bs64(const DecodeParams& p, int, int head_size, int group, cudaStream_t s) {
    return launch_decode_bs<PA_F16, PA_F16, 64>(p, head_size, group, s);
}
}  // namespace pa
