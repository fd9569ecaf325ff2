// bf16 queries over a bf16 KV cache, block size 64.
#include "decode_launch.cuh"
namespace pa {
pa_status launch_decode_bf16_bs64(const DecodeParams& p, int, int head_size, int group, cudaStream_t s) {
    return launch_decode_bs<PA_BF16, PA_BF16, 64>(p, head_size, group, s);
}
}  // namespace pa
