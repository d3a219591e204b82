// decode_kernel.cuh -- paged decode attention for sm_103a.
//
// One CTA owns (sequence b, split-KV partition, kv head, head tile).  Its
// warps stream disjoint 16-token chunks of the partition: chunk i goes to warp
// i % W.  Each warp runs its own TMA pipeline: lane 0 looks the chunk's
// physical block up in the block table (entries prefetched into registers,
// 32 chunks at a time), issues 3-D tiled bulk tensor copies of the 16 K rows
// and 16 V rows of that kv head into a 128-byte-swizzled shared-memory stage,
// and the warp waits on the stage's mbarrier.  Per chunk the warp computes
// QK^T, an online-softmax update and PV, keeping a running max m, sum l and
// unnormalised output O per query head.  At the end the CTA merges its warps'
// (m, l, O) through shared memory; a sequence whose context spans several
// partitions writes (m, l, O) to the workspace and the last CTA to arrive for
// that (sequence, kv head, head tile) -- found with an atomic counter, never
// waited for -- combines the partitions and writes the output.
//
// Method: "mini-vLLM" README, "How it works / Paged KV-cache" (block-table
// indirection into a pool of physical blocks) and "Results / Correctness"
// (result equals dense attention; grouped-query heads read their KV head).
// The split-KV partition-and-reduce and the online softmax are this
// library's design: the pages do not describe kernel internals.
//
// Two compute variants share the pipeline:
//   kMma (f16/bf16): S^T[16 tok x 8 heads] = K[16 x D] * Q^T with
//     mma.sync.m16n8k16 (A = K rows via ldmatrix, B = Q held in registers),
//     P^T moved into B-operand layout with movmatrix.trans, and
//     O^T[D x 8 heads] += V^T * P^T (A = V via ldmatrix.trans).  The query
//     heads of a GQA group (up to 8 per n-tile, 16 with two n-tiles) share
//     every K/V byte read.
//   kFma (f32, or any type on request): fp32 FMA on CUDA cores; a lane owns
//     (token, half of head_dim) for QK^T and head_dim/32 output columns for PV.
#pragma once

#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace wllm {

constexpr int kChunk = 16;  // tokens per pipeline stage of one warp

template <typename T, int D>
struct Geom {
  static constexpr int kElt = static_cast<int>(sizeof(T));
  static constexpr int kBoxCols = 128 / kElt;          // elements in one 128-byte box row
  static constexpr int kColBoxes = D / kBoxCols;       // boxes across a row of D elements
  static constexpr int kTileBytes = kColBoxes * 2048;  // 16 rows of one head's K (or V)
  static constexpr int kStageBytes = 2 * kTileBytes;   // K tile then V tile
  static constexpr bool kPairRows = false;
  static_assert(D % kBoxCols == 0, "head_dim must fill whole 128-byte rows");
};

// E4M3 codes with head_dim 64: a token row is 64 bytes, so the pool is viewed
// as rows of two tokens (128 bytes, still one swizzled box row); 16 tokens are
// one box of 8 such rows.  Token r of a tile sits in box row r / 2, bytes
// 64 (r % 2) .. 64 (r % 2) + 63.
template <>
struct Geom<uint8_t, 64> {
  static constexpr int kElt = 1;
  static constexpr int kBoxCols = 128;
  static constexpr int kColBoxes = 1;
  static constexpr int kTileBytes = 1024;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr bool kPairRows = true;
};

template <typename T, int D>
struct Tuning {
  static constexpr int kStageBytes = Geom<T, D>::kStageBytes;
  static constexpr int kWarps = kStageBytes >= 32768 ? 2 : 4;
  static constexpr int kRingBudget = 96 * 1024;
  static constexpr int kStagesRaw = kRingBudget / (kWarps * kStageBytes);
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
  static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
};

// ---------------------------------------------------------------------------
// tensor-core variant state and chunk update
// ---------------------------------------------------------------------------
template <typename T, int D, int NT>
struct MmaState {
  float o[D / 16][NT][4];    // O^T fragments: rows d, columns heads
  float m[NT][2];            // running max (log2 units) of this lane's two heads per n-tile
  float l[NT][2];            // running sum, partial over this lane's tokens
  uint32_t qb[NT][D / 16][2];  // Q^T B-operand fragments
};

template <typename T, int D, int NT>
__device__ __forceinline__ void mma_init(MmaState<T, D, NT>& st, const T* q, int64_t q_sh, int nh,
                                         int lane) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 8 + (lane >> 2);
    const bool valid = hh < nh;
    const T* row = q + static_cast<int64_t>(valid ? hh : 0) * q_sh;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int d = ks * 16 + 2 * (lane & 3);
      st.qb[nt][ks][0] = valid ? *reinterpret_cast<const uint32_t*>(row + d) : 0u;
      st.qb[nt][ks][1] = valid ? *reinterpret_cast<const uint32_t*>(row + d + 8) : 0u;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      st.m[nt][j] = -INFINITY;
      st.l[nt][j] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) st.o[mt][nt][i] = 0.f;
  }
}

template <typename T, int D, int NT>
__device__ __forceinline__ void mma_chunk(MmaState<T, D, NT>& st, uint32_t k_tile, uint32_t v_tile,
                                          int t0, int tok_end, float scale_log2, int lane) {
  // S^T = K Q^T : rows = 16 tokens, columns = 8 heads per n-tile
  float s[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) s[nt][i] = 0.f;
  const int a_row = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int a_chunk = lane >> 4;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t a[4];
    ldsm_x4(k_tile + tile_offset(a_row, 2 * ks + a_chunk), a);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) Mma<T>::run(s[nt], a, st.qb[nt][ks]);
  }

  // online softmax over this chunk (tokens lane/4 and lane/4 + 8)
  const int tok_a = t0 + (lane >> 2);
  const bool va = tok_a < tok_end;
  const bool vb = tok_a + 8 < tok_end;
  float alpha[NT][2];
  uint32_t pb[NT][2];
  bool rescale = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float x0 = va ? s[nt][0] * scale_log2 : -INFINITY;
    const float x1 = va ? s[nt][1] * scale_log2 : -INFINITY;
    const float x2 = vb ? s[nt][2] * scale_log2 : -INFINITY;
    const float x3 = vb ? s[nt][3] * scale_log2 : -INFINITY;
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, off));
    }
    const float mn0 = fmaxf(st.m[nt][0], mx0), mn1 = fmaxf(st.m[nt][1], mx1);
    alpha[nt][0] = exp2f(st.m[nt][0] - mn0);
    alpha[nt][1] = exp2f(st.m[nt][1] - mn1);
    st.m[nt][0] = mn0;
    st.m[nt][1] = mn1;
    const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
    const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
    st.l[nt][0] = st.l[nt][0] * alpha[nt][0] + (p0 + p2);
    st.l[nt][1] = st.l[nt][1] * alpha[nt][1] + (p1 + p3);
    rescale |= (alpha[nt][0] != 1.f) || (alpha[nt][1] != 1.f);
    pb[nt][0] = movmatrix_trans(Mma<T>::pack(p0, p1));
    pb[nt][1] = movmatrix_trans(Mma<T>::pack(p2, p3));
  }
  if (__any_sync(kFullMask, rescale)) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        st.o[mt][nt][0] *= alpha[nt][0];
        st.o[mt][nt][1] *= alpha[nt][1];
        st.o[mt][nt][2] *= alpha[nt][0];
        st.o[mt][nt][3] *= alpha[nt][1];
      }
  }

  // O^T += V^T P^T ; V rows past the context are zeroed (they may hold anything)
  const int v_row = (lane & 7) + ((lane >> 4) << 3);
  const int v_chunk = (lane >> 3) & 1;
  const bool tail = t0 + kChunk > tok_end;
  const int tk = t0 + 2 * (lane & 3);
  const uint32_t keep_lo = (tk < tok_end ? 0x0000ffffu : 0u) | (tk + 1 < tok_end ? 0xffff0000u : 0u);
  const uint32_t keep_hi = (tk + 8 < tok_end ? 0x0000ffffu : 0u) | (tk + 9 < tok_end ? 0xffff0000u : 0u);
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    uint32_t a[4];
    ldsm_x4_trans(v_tile + tile_offset(v_row, 2 * mt + v_chunk), a);
    if (tail) {
      a[0] &= keep_lo;
      a[1] &= keep_lo;
      a[2] &= keep_hi;
      a[3] &= keep_hi;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) Mma<T>::run(st.o[mt][nt], a, pb[nt]);
  }
}

// Write this warp's (m, l, O) for its heads into the CTA reduction area.
template <typename T, int D, int NT>
__device__ __forceinline__ void mma_store(MmaState<T, D, NT>& st, float* red_o, float* red_m,
                                          float* red_l, int lane) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = st.l[nt][j];
      l += __shfl_xor_sync(kFullMask, l, 4);
      l += __shfl_xor_sync(kFullMask, l, 8);
      l += __shfl_xor_sync(kFullMask, l, 16);
      if (lane < 4) {
        const int hh = nt * 8 + 2 * lane + j;
        red_m[hh] = st.m[nt][j];
        red_l[hh] = l;
      }
    }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hh = nt * 8 + 2 * (lane & 3);
      const int d = mt * 16 + (lane >> 2);
      red_o[hh * D + d] = st.o[mt][nt][0];
      red_o[(hh + 1) * D + d] = st.o[mt][nt][1];
      red_o[hh * D + d + 8] = st.o[mt][nt][2];
      red_o[(hh + 1) * D + d + 8] = st.o[mt][nt][3];
    }
}

// ---------------------------------------------------------------------------
// fp32 FMA variant (8 query heads per CTA)
// ---------------------------------------------------------------------------
template <typename T, int N>
__device__ __forceinline__ void unpack16(const uint4& raw, float (&out)[N]) {
  const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
  for (int i = 0; i < N; ++i) out[i] = to_f32(e[i]);
}

// Load N consecutive elements of row `row` starting at element `e0` from a
// swizzled tile.  N * sizeof(T) is 4, 8 or a multiple of 16, and e0 is a
// multiple of N.
template <typename T, int N>
__device__ __forceinline__ void tile_load(const uint8_t* tile, int row, int e0, float (&out)[N]) {
  constexpr int kBytes = N * static_cast<int>(sizeof(T));
  const int byte0 = e0 * static_cast<int>(sizeof(T));
  if constexpr (kBytes >= 16) {
    constexpr int kPer = 16 / static_cast<int>(sizeof(T));
#pragma unroll
    for (int piece = 0; piece < kBytes / 16; ++piece) {
      const uint4 raw = *reinterpret_cast<const uint4*>(tile + tile_offset(row, byte0 / 16 + piece));
      float tmp[kPer];
      unpack16<T, kPer>(raw, tmp);
#pragma unroll
      for (int i = 0; i < kPer; ++i) out[piece * kPer + i] = tmp[i];
    }
  } else {
    const uint8_t* ptr = tile + tile_offset(row, byte0 / 16) + (byte0 & 15);
    if constexpr (kBytes == 8) {
      const uint2 raw = *reinterpret_cast<const uint2*>(ptr);
      const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
      for (int i = 0; i < N; ++i) out[i] = to_f32(e[i]);
    } else {
      static_assert(kBytes == 4, "unsupported load width");
      const uint32_t raw = *reinterpret_cast<const uint32_t*>(ptr);
      const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
      for (int i = 0; i < N; ++i) out[i] = to_f32(e[i]);
    }
  }
}

template <int D>
struct FmaState {
  static constexpr int kDL = D / 32;  // output columns per lane
  float o[8][kDL];
  float m[8];  // warp-uniform running max (log2 units)
  float l[8];  // per-lane partial sum over this lane's token
};

template <int D>
__device__ __forceinline__ void fma_init(FmaState<D>& st) {
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    st.m[h] = -INFINITY;
    st.l[h] = 0.f;
#pragma unroll
    for (int i = 0; i < FmaState<D>::kDL; ++i) st.o[h][i] = 0.f;
  }
}

template <typename T, int D>
__device__ __forceinline__ void fma_chunk(FmaState<D>& st, const uint8_t* k_tile, const uint8_t* v_tile,
                                          const float* qs, int nh, int t0, int tok_end,
                                          float scale_log2, int lane) {
  constexpr int kPer = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte chunk
  constexpr int kHalfChunks = D / 2 / kPer;
  const int tok = lane & 15, half = lane >> 4;
  float s[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) s[h] = 0.f;
#pragma unroll
  for (int c = 0; c < kHalfChunks; ++c) {
    const int chunk = half * kHalfChunks + c;
    const uint4 raw = *reinterpret_cast<const uint4*>(k_tile + tile_offset(tok, chunk));
    float kv[kPer];
    unpack16<T, kPer>(raw, kv);
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      if (h < nh) {
        const float* qh = qs + h * D + chunk * kPer;
#pragma unroll
        for (int e = 0; e < kPer; e += 4) {
          const float4 qv = *reinterpret_cast<const float4*>(qh + e);
          s[h] = fmaf(qv.x, kv[e], s[h]);
          s[h] = fmaf(qv.y, kv[e + 1], s[h]);
          s[h] = fmaf(qv.z, kv[e + 2], s[h]);
          s[h] = fmaf(qv.w, kv[e + 3], s[h]);
        }
      }
    }
  }
  const bool valid = t0 + tok < tok_end;
  float pv[8], alpha[8];
  bool rescale = false;
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h < nh) {
      s[h] += __shfl_xor_sync(kFullMask, s[h], 16);
      const float x = valid ? s[h] * scale_log2 : -INFINITY;
      float mx = x;
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, off));
      const float mn = fmaxf(st.m[h], mx);
      alpha[h] = exp2f(st.m[h] - mn);
      st.m[h] = mn;
      pv[h] = exp2f(x - mn);
      st.l[h] = st.l[h] * alpha[h] + pv[h];
      rescale |= alpha[h] != 1.f;
    } else {
      pv[h] = 0.f;
      alpha[h] = 1.f;
    }
  }
  if (rescale) {  // warp-uniform: m is the same in every lane
#pragma unroll
    for (int h = 0; h < 8; ++h)
#pragma unroll
      for (int i = 0; i < FmaState<D>::kDL; ++i) st.o[h][i] *= alpha[h];
  }
  const int n_valid = min(kChunk, tok_end - t0);
  for (int j = 0; j < n_valid; ++j) {
    float v[FmaState<D>::kDL];
    tile_load<T, FmaState<D>::kDL>(v_tile, j, lane * FmaState<D>::kDL, v);
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      if (h < nh) {
        const float ph = __shfl_sync(kFullMask, pv[h], j);
#pragma unroll
        for (int i = 0; i < FmaState<D>::kDL; ++i) st.o[h][i] = fmaf(ph, v[i], st.o[h][i]);
      }
    }
  }
}

template <int D>
__device__ __forceinline__ void fma_store(FmaState<D>& st, float* red_o, float* red_m, float* red_l,
                                          int nh, int lane) {
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h < nh) {
      float l = (lane < 16) ? st.l[h] : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) l += __shfl_xor_sync(kFullMask, l, off);
      if (lane == 0) {
        red_m[h] = st.m[h];
        red_l[h] = l;
      }
#pragma unroll
      for (int i = 0; i < FmaState<D>::kDL; ++i) red_o[h * D + lane * FmaState<D>::kDL + i] = st.o[h][i];
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <typename T, int D, int NT, bool kMma>
struct KernelShape {
  using TU = Tuning<T, D>;
  static constexpr int kWarps = TU::kWarps;
  static constexpr int kStages = TU::kStages;
  static constexpr int kHeadTile = kMma ? 8 * NT : 8;
  static constexpr int kBarBytes = kWarps * kStages * 8;
  static constexpr int kQsBytes = kMma ? 0 : kHeadTile * D * 4;
  static constexpr int kMiscBytes = 64;
  static constexpr int kSmemBytes = 1024 + TU::kRingBytes + kBarBytes + kQsBytes + kMiscBytes;
  static constexpr int kRedBytes = kWarps * kHeadTile * (D + 2) * 4;
  static_assert(kRedBytes <= TU::kRingBytes, "reduction area must fit in the stage ring");
};

template <typename T, int D, int NT, bool kMma>
__global__ void __launch_bounds__(Tuning<T, D>::kWarps * 32)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  using G = Geom<T, D>;
  using KS = KernelShape<T, D, NT, kMma>;
  constexpr int W = KS::kWarps;
  constexpr int S = KS::kStages;
  constexpr int HT = KS::kHeadTile;
  constexpr int kThreads = W * 32;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tuning<T, D>::kRingBytes);
  float* qs = reinterpret_cast<float*>(smem + Tuning<T, D>::kRingBytes + KS::kBarBytes);
  int* misc = reinterpret_cast<int*>(smem + Tuning<T, D>::kRingBytes + KS::kBarBytes + KS::kQsBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x, part = blockIdx.y;
  const int kvh = blockIdx.z / p.num_head_tiles;
  const int ht = blockIdx.z - kvh * p.num_head_tiles;
  const int h0 = kvh * p.group + ht * p.head_tile;
  const int nh = min(p.head_tile, p.group - ht * p.head_tile);

  // a wait on a copy already timed out in this launch: stop early
  if (*reinterpret_cast<volatile int*>(p.err) & kErrWaitTimeout) return;

  int L = p.context_lens[b];
  const int l_max = p.max_blocks * p.block_size;
  if (L < 0 || L > l_max) {
    if (threadIdx.x == 0 && part == 0 && blockIdx.z == 0) atomicOr(p.err, kErrLen);
    L = L < 0 ? 0 : l_max;
  }
  const int n_parts = L == 0 ? 1 : (L + p.part_tokens - 1) / p.part_tokens;
  if (part >= n_parts) return;

  T* out = reinterpret_cast<T*>(p.out);
  if (L == 0) {
    for (int idx = threadIdx.x; idx < nh * D; idx += kThreads) {
      const int hh = idx / D, d = idx - (idx / D) * D;
      out[b * p.o_sb + static_cast<int64_t>(h0 + hh) * p.o_sh + d] = from_f32<T>(0.f);
    }
    return;
  }

  const int tok_begin = part * p.part_tokens;
  const int tok_end = min(L, tok_begin + p.part_tokens);
  const int n_chunks = (tok_end - tok_begin + kChunk - 1) / kChunk;
  const int my_chunks = n_chunks > warp ? (n_chunks - warp + W - 1) / W : 0;
  const int32_t* bt_row = p.block_tables + static_cast<int64_t>(b) * p.bt_stride;
  const int bs = p.block_size;

  const uint32_t ring_base = smem_u32(ring) + warp * S * G::kStageBytes;
  const uint32_t bar_base = smem_u32(bars) + warp * S * 8;
  if (lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(bar_base + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  // block-table entries of this warp's chunks, 32 chunks per refill
  int e0 = 0, e1 = 0;
  auto refill = [&](int kbase) {
    const int k = kbase + lane;
    e0 = 0;
    e1 = 0;
    if (k < my_chunks) {
      const int t0 = tok_begin + kChunk * (warp + k * W);
      int x0, x1 = 0;
      if (p.log2_bs >= 4) {
        x0 = bt_row[t0 >> p.log2_bs];
      } else {
        x0 = bt_row[t0 >> p.log2_bs];
        if (t0 + 8 < tok_end) x1 = bt_row[(t0 >> p.log2_bs) + 1];
      }
      if (x0 < 0 || x0 >= p.num_blocks || x1 < 0 || x1 >= p.num_blocks) {
        atomicOr(p.err, kErrBlock);
        x0 = (x0 < 0 || x0 >= p.num_blocks) ? 0 : x0;
        x1 = (x1 < 0 || x1 >= p.num_blocks) ? 0 : x1;
      }
      e0 = x0;
      e1 = x1;
    }
  };
  auto issue = [&](int k) {  // warp-collective
    if ((k & 31) == 0) refill(k);
    const int pb0 = __shfl_sync(kFullMask, e0, k & 31);
    const int pb1 = __shfl_sync(kFullMask, e1, k & 31);
    if (lane == 0) {
      const int t0 = tok_begin + kChunk * (warp + k * W);
      const int s = k % S;
      const uint32_t stage = ring_base + s * G::kStageBytes;
      const uint32_t bar = bar_base + 8 * s;
      if (p.log2_bs >= 4) {
        const int y = kvh * bs + (t0 & (bs - 1));
        mbar_arrive_expect_tx(bar, G::kStageBytes);
#pragma unroll
        for (int cb = 0; cb < G::kColBoxes; ++cb)
          tma_load_3d(stage + cb * 2048, &kmap, bar, cb * G::kBoxCols, y, pb0);
#pragma unroll
        for (int cb = 0; cb < G::kColBoxes; ++cb)
          tma_load_3d(stage + G::kTileBytes + cb * 2048, &vmap, bar, cb * G::kBoxCols, y, pb0);
      } else {  // block_size 8: two 8-row boxes per chunk
        const bool has1 = t0 + 8 < tok_end;
        const int y = kvh * bs;
        mbar_arrive_expect_tx(bar, has1 ? G::kStageBytes : G::kStageBytes / 2);
#pragma unroll
        for (int cb = 0; cb < G::kColBoxes; ++cb) {
          tma_load_3d(stage + cb * 2048, &kmap, bar, cb * G::kBoxCols, y, pb0);
          tma_load_3d(stage + G::kTileBytes + cb * 2048, &vmap, bar, cb * G::kBoxCols, y, pb0);
          if (has1) {
            tma_load_3d(stage + cb * 2048 + 1024, &kmap, bar, cb * G::kBoxCols, y, pb1);
            tma_load_3d(stage + G::kTileBytes + cb * 2048 + 1024, &vmap, bar, cb * G::kBoxCols, y, pb1);
          }
        }
      }
    }
  };

  const int n_pro = my_chunks < S ? my_chunks : S;
  for (int k = 0; k < n_pro; ++k) issue(k);

  // per-variant state; the query tile
  MmaState<T, D, (kMma ? NT : 1)> mst;
  FmaState<D> fst;
  const T* qrow0 = reinterpret_cast<const T*>(p.q) + b * p.q_sb + static_cast<int64_t>(h0) * p.q_sh;
  if constexpr (kMma) {
    mma_init<T, D, NT>(mst, qrow0, p.q_sh, nh, lane);
  } else {
    fma_init<D>(fst);
    for (int idx = threadIdx.x; idx < HT * D; idx += kThreads) {
      const int hh = idx / D, d = idx - (idx / D) * D;
      qs[idx] = hh < nh ? to_f32(qrow0[static_cast<int64_t>(hh) * p.q_sh + d]) : 0.f;
    }
    __syncthreads();
  }

  bool ok = true;
  int k_fail = my_chunks;
  for (int k = 0; k < my_chunks; ++k) {
    const int s = k % S;
    const bool got = mbar_wait_bounded(bar_base + 8 * s, (k / S) & 1, p.wait_limit_ns);
    if (!__all_sync(kFullMask, got)) {
      ok = false;
      k_fail = k;
      break;
    }
    const int t0 = tok_begin + kChunk * (warp + k * W);
    const uint32_t stage = ring_base + s * G::kStageBytes;
    if constexpr (kMma) {
      mma_chunk<T, D, NT>(mst, stage, stage + G::kTileBytes, t0, tok_end, p.scale_log2, lane);
    } else {
      const uint8_t* st_ptr = ring + (warp * S + s) * G::kStageBytes;
      fma_chunk<T, D>(fst, st_ptr, st_ptr + G::kTileBytes, qs, nh, t0, tok_end, p.scale_log2, lane);
    }
    __syncwarp();
    if (k + S < my_chunks) issue(k + S);
  }
  if (!ok) {
    // drain this warp's copies still in flight (bounded), then give up on the CTA
    if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
    const int issued = (k_fail + S < my_chunks) ? k_fail + S : my_chunks;
    for (int k = k_fail; k < issued; ++k)
      mbar_wait_bounded(bar_base + 8 * (k % S), (k / S) & 1, p.wait_limit_ns);
  }
  if (!__syncthreads_and(ok)) return;

  // merge the warps' (m, l, O) through shared memory (the ring is free now)
  float* red_o = reinterpret_cast<float*>(ring);
  float* red_m = red_o + W * HT * D;
  float* red_l = red_m + W * HT;
  if constexpr (kMma) {
    mma_store<T, D, NT>(mst, red_o + warp * HT * D, red_m + warp * HT, red_l + warp * HT, lane);
  } else {
    fma_store<D>(fst, red_o + warp * HT * D, red_m + warp * HT, red_l + warp * HT, nh, lane);
  }
  __syncthreads();

  const int row0 = b * p.num_q_heads + h0;  // flat index of this tile's first query head
  for (int hh = warp; hh < nh; hh += W) {
    float mw[W], M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      mw[w] = red_m[w * HT + hh];
      M = fmaxf(M, mw[w]);
    }
    float fw[W], den = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      fw[w] = mw[w] == -INFINITY ? 0.f : exp2f(mw[w] - M);
      den += fw[w] * red_l[w * HT + hh];
    }
    if (n_parts == 1) {
      const float inv = 1.f / den;
      T* orow = out + b * p.o_sb + static_cast<int64_t>(h0 + hh) * p.o_sh;
      for (int d = lane; d < D; d += 32) {
        float num = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) num += fw[w] * red_o[(w * HT + hh) * D + d];
        orow[d] = from_f32<T>(num * inv);
      }
    } else {
      const int64_t slot = static_cast<int64_t>(row0 + hh) * p.max_parts + part;
      float* wo = p.ws_o + slot * D;
      for (int d = lane; d < D; d += 32) {
        float num = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) num += fw[w] * red_o[(w * HT + hh) * D + d];
        wo[d] = num;
      }
      if (lane == 0) {
        p.ws_ml[slot * 2] = M;
        p.ws_ml[slot * 2 + 1] = den;
      }
    }
  }
  if (n_parts == 1) return;

  // split-KV: the last partition CTA to arrive combines all partitions
  __threadfence();
  __syncthreads();
  int* counter = p.ws_count + (static_cast<int64_t>(b) * p.num_kv_heads + kvh) * p.num_head_tiles + ht;
  if (threadIdx.x == 0) misc[0] = (atomicAdd(counter, 1) == n_parts - 1);
  __syncthreads();
  if (!misc[0]) return;
  __threadfence();
  for (int hh = warp; hh < nh; hh += W) {
    const int64_t base = static_cast<int64_t>(row0 + hh) * p.max_parts;
    float M = -INFINITY;
    for (int pp = lane; pp < n_parts; pp += 32) M = fmaxf(M, __ldcg(p.ws_ml + (base + pp) * 2));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
    float den = 0.f;
    for (int pp = lane; pp < n_parts; pp += 32)
      den += exp2f(__ldcg(p.ws_ml + (base + pp) * 2) - M) * __ldcg(p.ws_ml + (base + pp) * 2 + 1);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(kFullMask, den, off);
    constexpr int kDL = D / 32;
    float num[kDL];
#pragma unroll
    for (int i = 0; i < kDL; ++i) num[i] = 0.f;
    for (int pp = 0; pp < n_parts; ++pp) {
      const float f = exp2f(__ldcg(p.ws_ml + (base + pp) * 2) - M);
      const float* wo = p.ws_o + (base + pp) * D;
#pragma unroll
      for (int i = 0; i < kDL; ++i) num[i] = fmaf(f, __ldcg(wo + lane + 32 * i), num[i]);
    }
    const float inv = 1.f / den;
    T* orow = out + b * p.o_sb + static_cast<int64_t>(h0 + hh) * p.o_sh;
#pragma unroll
    for (int i = 0; i < kDL; ++i) orow[lane + 32 * i] = from_f32<T>(num[i] * inv);
  }
  if (threadIdx.x == 0) *counter = 0;
}

// ---------------------------------------------------------------------------
// host-side launch of one instantiation
// ---------------------------------------------------------------------------
template <typename T, int D, int NT, bool kMma>
int launch_decode_inst(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                       cudaStream_t stream) {
  using KS = KernelShape<T, D, NT, kMma>;
  auto kernel = paged_decode_kernel<T, D, NT, kMma>;
  static std::atomic<int> configured_for[64];  // per device: shared-memory attribute set
  cudaError_t e = static_cast<cudaError_t>(
      raise_smem_limit(configured_for, reinterpret_cast<const void*>(kernel), KS::kSmemBytes));
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_seqs, p.max_parts, p.num_kv_heads * p.num_head_tiles);
  kernel<<<grid, KS::kWarps * 32, KS::kSmemBytes, stream>>>(kmap, vmap, p);
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

template <typename T, int D, int NT, bool kMma>
constexpr int smem_of() {
  return KernelShape<T, D, NT, kMma>::kSmemBytes;
}

}  // namespace wllm
