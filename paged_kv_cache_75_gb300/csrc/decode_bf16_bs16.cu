// bf16 queries over a bf16 KV cache, block size 16.
#include "decode_launch.cuh"
namespace pa {
pa_status launch_decode_bf16_bs16(const DecodeParams& p, int, int head_size, int group, cudaStream_t s) {
    return launch_decode_bs<PA_BF16, PA_BF16, 16>(p, head_size, group, s);
}
}  // namespace pa
