// launch.h -- internal interface between the C ABI (api.cu) and the kernel
// translation units.  Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace wllm {

// The 256-byte per-device control block, offsets in ints: the error word;
// two spare words used only by the bounded-wait self-test (a counter that
// stays zero, and its result); the persistent scheduler's claim and finish
// counters; the fused step's 64-bit count of CTAs whose KV append is written.
constexpr int kCtrlBytes = 256;
constexpr int kSelftestNeverOffset = 8;
constexpr int kSelftestResultOffset = 9;
constexpr int kSchedNextOffset = 16;
constexpr int kSchedDoneOffset = 32;
constexpr int kGridCountOffset = 48;  // 8-byte aligned: two ints

// Kernel launches the library has issued (successful launch calls), for
// wllm_launch_count().  Every launch site calls note_launch() once per kernel.
void note_launch();

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device: `configured` is the kernel's own per-device record
// (64 entries).  Thread-safe; two threads racing only repeat the attribute call.
inline int raise_smem_limit(std::atomic<int>* configured, const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < 64;
  if (tracked && configured[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (tracked) configured[dev].store(bytes, std::memory_order_release);
  return cudaSuccess;
}

// Everything one paged-decode launch needs besides the two tensor maps.
struct DecodeParams {
  void* out;                 // [B][Hq][D]
  const void* q;             // [B][Hq][D]
  int64_t q_sb, q_sh;        // q strides (elements) of the seq and head dims
  int64_t o_sb, o_sh;        // out strides
  const int32_t* block_tables;
  int64_t bt_stride;         // elements between two sequences' tables
  const int32_t* context_lens;
  int num_seqs, num_q_heads, num_kv_heads, group;
  int head_tile, num_head_tiles;  // query heads per CTA, tiles per kv head
  int max_blocks, block_size, log2_bs, num_blocks;
  int part_tokens, max_parts;     // split-KV partition size / count
  float scale_log2;               // scale * log2(e) (times k_scale for an fp8 cache)
  float v_scale;                  // fp8 cache: factor of every output (1 otherwise)
  float* ws_o;                    // [B*Hq][max_parts][D] unnormalised partial sums
  float* ws_ml;                   // [B*Hq][max_parts][2] running max (log2 units), sum
  int* ws_count;                  // counters, zero between calls: grid kernel [B*Hkv*tiles] arrivals;
                                  // persistent kernel [2][B*Hkv*tiles] units finished, rows merged
  int* err;                       // device error word
  unsigned long long wait_limit_ns;
  int prefix_groups;              // process shared-prefix partitions once per group of sequences
};

struct AppendParams {
  const uint8_t* key;
  const uint8_t* value;
  uint8_t* k_cache;
  uint8_t* v_cache;
  const void* slots;
  int slots_are_i64;
  int num_tokens, num_kv_heads;
  int row_bytes;                  // bytes of one cache row: head_dim * cache element size
  int64_t key_st, key_sh;         // strides in bytes
  int64_t val_st, val_sh;
  int log2_bs;
  int64_t num_slots;              // num_blocks * block_size
  int vec16;                      // rows and strides allow 16-byte copies
  int kv_fp8;                     // caches hold E4M3 codes of key * k_inv and value * v_inv
  int src_dtype;                  // fp8: key/value element type, a wllm_dtype code (0 f32, 1 f16, 2 bf16)
  float k_inv, v_inv;             // fp8: binary32 reciprocals of the scales
  int* err;
};

// Kernel variants of the decode: tensor-core (16-bit only) or fp32 FMA.
enum class DecodeVariant { kMma, kFma };

// Head tile (query heads of one KV head handled by one CTA) for a variant.
int decode_head_tile(int dtype, int head_dim, int group, DecodeVariant v, bool kv_fp8);

// Launch the decode kernel; returns a cudaError_t value.
int launch_decode(int dtype, int head_dim, DecodeVariant v, const CUtensorMap& kmap,
                  const CUtensorMap& vmap, const DecodeParams& p, cudaStream_t stream);

// Persistent warp-specialised decode (f16/bf16 only).  `separate_combine`
// appends the split-KV combine kernel (needed when a sequence can span
// several partitions and `fuse_combine` is not set).  `ap` (may be null)
// fuses the KV append in front; `fuse_combine` merges the partitions inside
// the launch, as they complete (p.ws_count must then hold the zeroed
// counters).  Either makes it a cooperative launch.
// `kv_fp8`: the caches hold E4M3 codes (head_dim 128 or 256, head tile 8);
// dtype is then the query / output type.
int launch_decode_persistent(int dtype, int head_dim, int head_tile, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, const DecodeParams& p, int grid, bool separate_combine,
                             const AppendParams* ap, bool fuse_combine, bool kv_fp8, cudaStream_t stream);
int decode_persistent_occupancy(int dtype, int head_dim, int head_tile, int num_seqs, bool kv_fp8);
constexpr int kPersistentConsumers = 4;
constexpr int kPersistentMaxSeqs = 1024;      // sequences per launch (the host splits larger batches)
constexpr int kPersistentMaxParts = 256;      // partitions per sequence (the host widens partitions to fit)

int launch_append(const AppendParams& p, cudaStream_t stream);

// One-thread kernel whose two bounded waits (an mbarrier and the counter at
// ctrl[never_offset], which must stay below 1) time out after limit_ns: sets
// kErrWaitTimeout in ctrl[0], adds 1 to ctrl[sched_offset] and writes which
// waits gave up (bit 0 mbarrier, bit 1 counter) to *result (device memory).
int launch_wait_selftest(int* ctrl, int never_offset, int sched_offset, unsigned long long limit_ns, int* result,
                         cudaStream_t stream);

// Chunked-prefill (multi-query) paged attention: q/out [T][Hq][D] packed by
// sequence (query_start_loc [B+1]); each chunk is the last n_b of the
// sequence's context_lens[b] tokens and attends causally.
struct PrefillParams {
  void* out;
  const void* q;
  int64_t q_st, q_sh;             // q strides (elements) of the token and head dims
  int64_t o_st, o_sh;             // out strides
  const int32_t* block_tables;
  int64_t bt_stride;
  const int32_t* context_lens;
  const int32_t* query_start_loc;
  int num_seqs, num_tokens, num_q_heads, num_kv_heads, group;
  int max_blocks, block_size, log2_bs, num_blocks;
  float scale_log2;               // scale * log2(e) (times k_scale for an fp8 cache)
  float v_scale;                  // fp8 cache: factor of every output (1 otherwise)
  int* err;
  unsigned long long wait_limit_ns;
};
// CTAs along x for T packed tokens of B sequences (grid y = kv heads).
int prefill_grid_x(int64_t num_tokens, int64_t num_seqs, int group);
// f16/bf16 queries (dtype code 1/2), head_dim 64 or 128; `kv_fp8`: E4M3 caches
// (head_dim 64 needs blocks of >= 16 tokens).  Returns a cudaError_t value.
int launch_prefill(int dtype, int head_dim, bool kv_fp8, const CUtensorMap& kmap, const CUtensorMap& vmap,
                   const PrefillParams& p, int grid_x, cudaStream_t stream);

// The same operation on the fifth-generation tensor cores (tcgen05 MMAs with
// TMEM accumulators): 16-bit caches, head_dim 64 or 128, q/out rows 16-byte
// aligned (base and strides), a positive scale.  256 query rows per CTA.
int prefill_tc_grid_x(int64_t num_tokens, int64_t num_seqs, int group);
int launch_prefill_tc(int dtype, int head_dim, const CUtensorMap& kmap, const CUtensorMap& vmap,
                      const PrefillParams& p, int grid_x, cudaStream_t stream);

// Check-mode kernels: record index errors in the device error word.
int launch_check_decode(const int32_t* block_tables, int64_t bt_stride,
                        const int32_t* context_lens, int num_seqs, int max_blocks,
                        int block_size, int num_blocks, int* err, cudaStream_t stream);
int launch_check_append(const void* slots, int slots_are_i64, int num_tokens,
                        int64_t num_slots, int* err, cudaStream_t stream);

// Bytes of shared memory one decode CTA uses, and its thread count.
int decode_smem_bytes(int dtype, int head_dim, DecodeVariant v, int head_tile);
int decode_threads(int dtype, int head_dim);

}  // namespace wllm
