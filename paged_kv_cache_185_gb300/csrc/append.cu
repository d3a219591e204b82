// append.cu -- the KV-cache append ("reshape and cache"), the check-mode
// index validation kernels and the self-test of the bounded waits.
//
// Method: "mini-vLLM" README, results paragraph on what changed -- the K/V
// write is one indexed assignment per layer rather than a loop over
// sequences.  Here that assignment is one kernel: a warp per (token, kv head)
// copies the token's K row and V row (head_dim elements each) into slot
// slot_mapping[t] = physical block * block_size + offset of the cache laid out
// [num_blocks][num_kv_heads][block_size][head_dim].  The copy moves raw bits
// (16-byte vectors when rows and strides allow), so it is bit-exact for every
// element type.
#include "append_row.cuh"
#include "common.cuh"
#include "launch.h"

namespace wllm {

namespace {

constexpr int kAppendWarps = 8;

__global__ void __launch_bounds__(kAppendWarps * 32) append_kernel(const AppendParams p) {
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
  if (gw >= static_cast<int64_t>(p.num_tokens) * p.num_kv_heads) return;
  append_row(p, gw, threadIdx.x & 31);
}

__global__ void check_decode_kernel(const int32_t* block_tables, int64_t bt_stride,
                                    const int32_t* context_lens, int num_seqs, int max_blocks,
                                    int block_size, int num_blocks, int* err) {
  const int b = blockIdx.x;
  if (b >= num_seqs) return;
  const int L = context_lens[b];
  if (L < 0 || static_cast<int64_t>(L) > static_cast<int64_t>(max_blocks) * block_size) {
    if (threadIdx.x == 0) atomicOr(err, kErrLen);
    return;
  }
  const int used = (L + block_size - 1) / block_size;
  for (int j = threadIdx.x; j < used; j += blockDim.x) {
    const int e = block_tables[b * bt_stride + j];
    if (e < 0 || e >= num_blocks) atomicOr(err, kErrBlock);
  }
}

__global__ void check_append_kernel(const void* slots, int slots_are_i64, int num_tokens,
                                    int64_t num_slots, int* err) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= num_tokens) return;
  auto slot_at = [&](int i) -> int64_t {
    return slots_are_i64 ? static_cast<const int64_t*>(slots)[i]
                         : static_cast<int64_t>(static_cast<const int32_t*>(slots)[i]);
  };
  const int64_t s = slot_at(t);
  if (s >= num_slots) atomicOr(err, kErrSlot);
  if (s < 0) return;
  for (int u = 0; u < t; ++u)  // quadratic, check mode only
    if (slot_at(u) == s) {
      atomicOr(err, kErrDupSlot);
      break;
    }
}

// Self-test of the bounded waits: one thread waits on an mbarrier that never
// receives its arrival (no copy is in flight on it) and then polls a counter
// that nothing increments, each with the library's bounded waits.  Both give
// up after limit_ns; each timeout sets kErrWaitTimeout, as in the decode
// kernels.  The scheduler counter is then left non-zero, as a launch that
// gave up half-way would leave it, so that the caller can check that reading
// the error word also restores the counters.
__global__ void wait_selftest_kernel(int* err, const int* never, int* sched_next, unsigned long long limit_ns,
                                     int* result) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  int r = 0;
  if (!mbar_wait_bounded(smem_u32(&bar), 0, limit_ns)) r |= 1;
  if (!counter_wait_bounded(never, 1, limit_ns)) r |= 2;
  if (r != 0) {
    atomicOr(err, kErrWaitTimeout);
    atomicAdd(sched_next, 1);
  }
  *result = r;
}

}  // namespace

int launch_wait_selftest(int* ctrl, int never_offset, int sched_offset, unsigned long long limit_ns, int* result,
                         cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(ctrl, ctrl + never_offset, ctrl + sched_offset, limit_ns, result);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

int launch_append(const AppendParams& p, cudaStream_t stream) {
  const int64_t warps = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads;
  const int64_t blocks = (warps + kAppendWarps - 1) / kAppendWarps;
  if (blocks == 0) return cudaSuccess;
  append_kernel<<<static_cast<unsigned>(blocks), kAppendWarps * 32, 0, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

int launch_check_decode(const int32_t* block_tables, int64_t bt_stride, const int32_t* context_lens,
                        int num_seqs, int max_blocks, int block_size, int num_blocks, int* err,
                        cudaStream_t stream) {
  if (num_seqs == 0) return cudaSuccess;
  check_decode_kernel<<<num_seqs, 128, 0, stream>>>(block_tables, bt_stride, context_lens, num_seqs,
                                                    max_blocks, block_size, num_blocks, err);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

int launch_check_append(const void* slots, int slots_are_i64, int num_tokens, int64_t num_slots,
                        int* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  check_append_kernel<<<(num_tokens + 127) / 128, 128, 0, stream>>>(slots, slots_are_i64, num_tokens,
                                                                    num_slots, err);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace wllm
