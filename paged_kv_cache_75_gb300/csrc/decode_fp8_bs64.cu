// fp16 or bf16 queries over an FP8 E4M3 KV cache, block size 64.
#include "decode_launch.cuh"
namespace pa {
pa_status launch_decode_fp8_bs64(const DecodeParams& p, int q_dtype, int head_size, int group, cudaStream_t s) {
    return q_dtype == PA_F16 ? launch_decode_bs<PA_F16, PA_FP8_E4M3, 64>(p, head_size, group, s)
                             : launch_decode_bs<PA_BF16, PA_FP8_E4M3, 64>(p, head_size, group, s);
}
}  // namespace pa
