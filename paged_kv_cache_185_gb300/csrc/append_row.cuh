// append_row.cuh -- one (token, kv head) row of the KV append, done by one
// warp: the token's K row and V row (head_dim elements each) are copied bit
// for bit into slot slot_mapping[t] of the caches, or, for an fp8 cache,
// stored as scaled E4M3 codes.  Shared by the append kernel and the fused
// decode step.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace wllm {

// Row `row` = t * num_kv_heads + h.  All 32 lanes of the warp call this.
__device__ __forceinline__ void append_row(const AppendParams& p, int64_t row, int lane) {
  const int t = static_cast<int>(row / p.num_kv_heads);
  const int h = static_cast<int>(row - static_cast<int64_t>(t) * p.num_kv_heads);
  const int64_t slot = p.slots_are_i64 ? static_cast<const int64_t*>(p.slots)[t]
                                       : static_cast<int64_t>(static_cast<const int32_t*>(p.slots)[t]);
  // 16-bit rows of up to 256 bytes (the common case): this lane's unit of the
  // K or V row is loaded together with the slot, one memory round trip
  if (p.vec16 && !p.kv_fp8 && (p.row_bytes >> 4) <= 16) {  // one 16-byte unit of K or V per lane
    const int n = p.row_bytes >> 4;
    const bool mine = lane < 2 * n;
    const int u = lane < n ? lane : lane - n;
    const uint8_t* src = (lane < n ? p.key + t * p.key_st : p.value + t * p.val_st) +
                         static_cast<int64_t>(h) * (lane < n ? p.key_sh : p.val_sh);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (mine) v = reinterpret_cast<const uint4*>(src)[u];
    if (slot < 0) return;  // padding token
    if (slot >= p.num_slots) {
      if (lane == 0) atomicOr(p.err, kErrSlot);
      return;
    }
    const int64_t blk = slot >> p.log2_bs;
    const int64_t off = slot & ((int64_t(1) << p.log2_bs) - 1);
    const int64_t dst = (((blk * p.num_kv_heads + h) << p.log2_bs) + off) * p.row_bytes;
    if (mine) reinterpret_cast<uint4*>((lane < n ? p.k_cache : p.v_cache) + dst)[u] = v;
    return;
  }
  if (slot < 0) return;  // padding token
  if (slot >= p.num_slots) {
    if (lane == 0) atomicOr(p.err, kErrSlot);
    return;
  }
  const int64_t blk = slot >> p.log2_bs;
  const int64_t off = slot & ((int64_t(1) << p.log2_bs) - 1);
  const int64_t dst = (((blk * p.num_kv_heads + h) << p.log2_bs) + off) * p.row_bytes;
  const uint8_t* ks = p.key + t * p.key_st + h * p.key_sh;
  const uint8_t* vs = p.value + t * p.val_st + h * p.val_sh;
  uint8_t* kd = p.k_cache + dst;
  uint8_t* vd = p.v_cache + dst;
  if (p.kv_fp8) {
    // E4M3 codes of x * (1/scale): the product rounded to binary32, then to
    // the nearest code (ties to even), saturating at +-448.  Lane u of the row
    // handles four consecutive elements (head_dim is a multiple of 4).
    const int n4 = p.row_bytes >> 2;
    for (int u = lane; u < 2 * n4; u += 32) {
      const bool is_k = u < n4;
      const int j = is_k ? u : u - n4;
      const uint8_t* src = is_k ? ks : vs;
      const float inv = is_k ? p.k_inv : p.v_inv;
      float x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = 4 * j + i;
        x[i] = p.src_dtype == 0   ? reinterpret_cast<const float*>(src)[e]
               : p.src_dtype == 1 ? __half2float(reinterpret_cast<const __half*>(src)[e])
                                  : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(src)[e]);
        x[i] = __fmul_rn(x[i], inv);
      }
      const uint32_t lo = f32x2_to_e4m3x2(x[1], x[0]), hi = f32x2_to_e4m3x2(x[3], x[2]);
      reinterpret_cast<uint32_t*>(is_k ? kd : vd)[j] = lo | (hi << 16);
    }
    return;
  }
  if (p.vec16) {
    const int n = p.row_bytes >> 4;  // 16-byte units per row
    for (int u = lane; u < 2 * n; u += 32) {
      if (u < n)
        reinterpret_cast<uint4*>(kd)[u] = reinterpret_cast<const uint4*>(ks)[u];
      else
        reinterpret_cast<uint4*>(vd)[u - n] = reinterpret_cast<const uint4*>(vs)[u - n];
    }
  } else {
    const int n = p.row_bytes >> 1;  // 2-byte units (every supported element is 2 or 4 bytes)
    for (int u = lane; u < 2 * n; u += 32) {
      if (u < n)
        reinterpret_cast<uint16_t*>(kd)[u] = reinterpret_cast<const uint16_t*>(ks)[u];
      else
        reinterpret_cast<uint16_t*>(vd)[u - n] = reinterpret_cast<const uint16_t*>(vs)[u - n];
    }
  }
}

}  // namespace wllm
