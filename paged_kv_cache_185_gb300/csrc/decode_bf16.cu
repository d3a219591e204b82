// Decode kernel instantiations for bfloat16 (tensor-core and FMA variants).
#define WLLM_ELT __nv_bfloat16
#define WLLM_HAS_MMA 1
#define WLLM_LAUNCH_FN launch_decode_bf16
#define WLLM_SMEM_FN smem_decode_bf16
#define WLLM_THREADS_FN threads_decode_bf16
#define WLLM_PERSIST_FN launch_persistent_bf16
#define WLLM_POCC_FN occupancy_persistent_bf16
#include "decode_dispatch.inc"
