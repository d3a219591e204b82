// Persistent decode over an fp8 (E4M3) KV cache with float16 queries.
#define WLLM_ELT __half
#define WLLM_PERSIST_F8_FN launch_persistent_f8_f16
#define WLLM_POCC_F8_FN occupancy_persistent_f8_f16
#include "decode_f8_dispatch.inc"
