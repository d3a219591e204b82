// Decode kernel instantiations for float32 (FMA variant only: fp32 inputs
// never go through reduced-precision tensor-core math).
#define WLLM_ELT float
#define WLLM_HAS_MMA 0
#define WLLM_LAUNCH_FN launch_decode_f32
#define WLLM_SMEM_FN smem_decode_f32
#define WLLM_THREADS_FN threads_decode_f32
#include "decode_dispatch.inc"
