// Persistent decode over an fp8 (E4M3) KV cache with bfloat16 queries.
#define WLLM_ELT __nv_bfloat16
#define WLLM_PERSIST_F8_FN launch_persistent_f8_bf16
#define WLLM_POCC_F8_FN occupancy_persistent_f8_bf16
#include "decode_f8_dispatch.inc"
