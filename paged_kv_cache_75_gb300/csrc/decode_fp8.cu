// fp16 or bf16 queries over an FP8 E4M3 KV cache.
#include "decode_launch.cuh"
namespace pa {
pa_status launch_decode_fp8_qf16(const DecodeParams& p, int head_size, int group, cudaStream_t s) {
    return launch_decode_dtype<PA_F16, PA_FP8_E4M3>(p, head_size, group, s);
}
pa_status launch_decode_fp8_qbf16(const DecodeParams& p, int head_size, int group, cudaStream_t s) {
    return launch_decode_dtype<PA_BF16, PA_FP8_E4M3>(p, head_size, group, s);
}
}  // namespace pa
