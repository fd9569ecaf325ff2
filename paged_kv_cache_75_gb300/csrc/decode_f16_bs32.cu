// fp16 queries over an fp16 KV cache, block size 32.
#include "decode_launch.cuh"
namespace pa {
pa_status launch_decode_f16_bs32(const DecodeParams& p, int, int head_size, int group, cudaStream_t s) {
    return launch_decode_bs<PA_F16, PA_F16, 32>(p, head_size, group, s);
}
}  // namespace pa
