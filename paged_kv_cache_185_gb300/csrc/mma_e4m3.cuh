// mma_e4m3.cuh -- tensor-core decode over an fp8 (E4M3) KV cache.
//
// The cache holds E4M3 codes of K/scale_k and V/scale_v.  Every E4M3 value is
// exactly representable in f16, so a staged 16-token sub-chunk is widened in
// registers (cvt.rn.f16x2.e4m3x2, exact) and the two products run as f16
// mma.sync m16n8k16 with fp32 accumulation; the query is converted to f16
// once per unit.  scale_k is folded into the softmax scale and scale_v into
// the output by the caller of these helpers.
//
// Fragment layouts.  Staged rows are 128-byte swizzled exactly like the
// 16-bit tiles (tile_offset), but one 16-byte chunk now holds 16 head_dim
// elements.
//   S^T = K Q^T: ldmatrix (b16 view) of chunk j gives lane (g = lane/4,
//     c = lane%4) bytes 4c..4c+3 of token row g: head_dim elements
//     16j+4c .. 16j+4c+3.  They serve as the k indices 2c, 2c+1 (low pair)
//     and 2c+8, 2c+9 (high pair) of the A fragment; the sum over head_dim
//     does not depend on the order, so the query's B fragment takes the same
//     permutation (q[16j+4c], q[16j+4c+1]) and (q[16j+4c+2], q[16j+4c+3]).
//   O^T += V^T P^T: ldmatrix.trans (b16 view) of 8 tokens x chunk j gives
//     lane (g, c) the byte pairs (V[2c][16j+2g], V[2c][16j+2g+1]) and
//     (V[2c+1][16j+2g], V[2c+1][16j+2g+1]); one byte permute regroups them
//     by head_dim element, so the A fragment's row g holds element 16j+2g and
//     row g+8 element 16j+2g+1, tokens along k as the P^T fragment expects.
//     The output rows of m-tile j are therefore d = 16j + 2g (accumulator
//     entries 0, 1) and d = 16j + 2g + 1 (entries 2, 3).
#pragma once

#include <type_traits>

#include "decode_kernel.cuh"

namespace wllm {

// f16x2 of a pair of query elements (exact for f16; bf16 rounded to f16).
template <typename T>
__device__ __forceinline__ uint32_t to_f16x2(uint32_t pair) {
  if constexpr (std::is_same<T, __half>::value) {
    return pair;
  } else {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pair));
    return Mma<__half>::pack(f.x, f.y);
  }
}

// Byte offset of 16-byte chunk `chunk` of token row `row` in a staged tile of
// codes (two tokens per 128-byte row when head_dim is 64).
template <int D>
__device__ __forceinline__ uint32_t code_offset(int row, int chunk) {
  if constexpr (Geom<uint8_t, D>::kPairRows)
    return tile_offset(row >> 1, ((row & 1) << 2) | chunk);
  else
    return tile_offset(row, chunk);
}

// Query B fragments in the permuted head_dim order above, converted to f16
// (exact for f16 queries; bf16 queries are rounded to f16).  Row stride D.
template <typename T, int D, int NT>
__device__ __forceinline__ void load_q_smem_e4m3(MmaState<__half, D, NT>& st, const uint8_t* qtile, int nh,
                                                 int lane) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 8 + (lane >> 2);
    const bool valid = hh < nh;
    const T* row = reinterpret_cast<const T*>(qtile) + (valid ? hh : 0) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int d = ks * 16 + 4 * (lane & 3);
      uint32_t b0 = 0u, b1 = 0u;
      if (valid) {
        const uint2 raw = *reinterpret_cast<const uint2*>(row + d);  // 4 elements, 8 bytes
        if constexpr (std::is_same<T, __half>::value) {
          b0 = raw.x;
          b1 = raw.y;
        } else {
          const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
          const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
          b0 = Mma<__half>::pack(f0.x, f0.y);
          b1 = Mma<__half>::pack(f1.x, f1.y);
        }
      }
      st.qb[nt][ks][0] = b0;
      st.qb[nt][ks][1] = b1;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      st.m[nt][j] = -INFINITY;
      st.l[nt][j] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.o[mt][nt][e] = 0.f;
  }
}

// NS consecutive 16-token sub-chunks as one softmax step: sub-chunk j's K tile
// (16 rows x D codes) at k_base + j * kTile, its V tile at v_base + j * kTile.
// The NS score chains are independent, which keeps more tensor-core work in
// flight per warp; tokens at or past tok_end are masked (their bytes may be
// stale or never written).
template <int D, int NT, int NS>
__device__ __forceinline__ void mma_chunks_e4m3(MmaState<__half, D, NT>& st, uint32_t k_base, uint32_t v_base,
                                                int t0, int tok_end, float scale_log2, int lane) {
  static_assert(D % 32 == 0, "two 16-element k steps per ldmatrix");
  constexpr int kTile = Geom<uint8_t, D>::kTileBytes;
  float s[NS][NT][4];
#pragma unroll
  for (int j = 0; j < NS; ++j)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[j][nt][i] = 0.f;
  // lanes 0-7 / 8-15 / 16-23 / 24-31 address rows 0-7 / 8-15 of chunk 2kp, then of chunk 2kp+1
  const int a_row = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int a_chunk = lane >> 4;
#pragma unroll
  for (int kp = 0; kp < D / 32; ++kp) {
#pragma unroll
    for (int j = 0; j < NS; ++j) {
      uint32_t r[4];
      ldsm_x4(k_base + j * kTile + code_offset<D>(a_row, 2 * kp + a_chunk), r);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // token rows g (r[2 half]) and g + 8 (r[2 half + 1]): low pairs -> k 2c, 2c+1, high -> 2c+8, 2c+9
        uint32_t a[4];
        e4m3x4_to_f16x2x2(r[2 * half], a[0], a[2]);
        e4m3x4_to_f16x2x2(r[2 * half + 1], a[1], a[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) Mma<__half>::run(s[j][nt], a, st.qb[nt][2 * kp + half]);
      }
    }
  }

  // online softmax over the NS sub-chunks (this lane: tokens lane/4 and lane/4 + 8 of each);
  // a step wholly inside the context needs no mask
  const bool full = t0 + NS * kChunk <= tok_end;
  float alpha[NT][2];
  uint32_t pb[NS][NT][2];
  bool rescale = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < NS; ++j) {
      const int tok_a = t0 + j * kChunk + (lane >> 2);
      const bool va = full || tok_a < tok_end, vb = full || tok_a + 8 < tok_end;
      s[j][nt][0] = va ? s[j][nt][0] * scale_log2 : -INFINITY;
      s[j][nt][1] = va ? s[j][nt][1] * scale_log2 : -INFINITY;
      s[j][nt][2] = vb ? s[j][nt][2] * scale_log2 : -INFINITY;
      s[j][nt][3] = vb ? s[j][nt][3] * scale_log2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[j][nt][0], s[j][nt][2]));
      mx1 = fmaxf(mx1, fmaxf(s[j][nt][1], s[j][nt][3]));
    }
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
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int j = 0; j < NS; ++j) {  // one SFU exponential each: the weights are rounded to f16 next
      const float p0 = ex2_approx(s[j][nt][0] - mn0), p1 = ex2_approx(s[j][nt][1] - mn1);
      const float p2 = ex2_approx(s[j][nt][2] - mn0), p3 = ex2_approx(s[j][nt][3] - mn1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      pb[j][nt][0] = movmatrix_trans(Mma<__half>::pack(p0, p1));
      pb[j][nt][1] = movmatrix_trans(Mma<__half>::pack(p2, p3));
    }
    st.l[nt][0] = st.l[nt][0] * alpha[nt][0] + l0;
    st.l[nt][1] = st.l[nt][1] * alpha[nt][1] + l1;
    rescale |= (alpha[nt][0] != 1.f) || (alpha[nt][1] != 1.f);
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
#pragma unroll
  for (int j = 0; j < NS; ++j) {
    const int tj = t0 + j * kChunk;
    const bool tail = tj + kChunk > tok_end;
#pragma unroll
    for (int mp = 0; mp < D / 32; ++mp) {
      uint32_t r[4];  // tokens 0-7 / 8-15 of chunk 2mp, then of chunk 2mp + 1
      ldsm_x4_trans(v_base + j * kTile + code_offset<D>(a_row, 2 * mp + a_chunk), r);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // bytes (t, e), (t, e+1), (t+1, e), (t+1, e+1) -> (t, e), (t+1, e), (t, e+1), (t+1, e+1)
        uint32_t a[4];
        e4m3x4_to_f16x2x2(__byte_perm(r[2 * half], 0u, 0x3120), a[0], a[1]);
        e4m3x4_to_f16x2x2(__byte_perm(r[2 * half + 1], 0u, 0x3120), a[2], a[3]);
        if (tail) {
          const int tk = tj + 2 * (lane & 3);
          const uint32_t keep_lo = (tk < tok_end ? 0x0000ffffu : 0u) | (tk + 1 < tok_end ? 0xffff0000u : 0u);
          const uint32_t keep_hi = (tk + 8 < tok_end ? 0x0000ffffu : 0u) | (tk + 9 < tok_end ? 0xffff0000u : 0u);
          a[0] &= keep_lo;
          a[1] &= keep_lo;
          a[2] &= keep_hi;
          a[3] &= keep_hi;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) Mma<__half>::run(st.o[2 * mp + half][nt], a, pb[j][nt]);
      }
    }
  }
}

// Query fragments of a prefix-group unit: column tile nt holds heads
// h0 .. h0+nh-1 of member sequence b0 + nt (zeros past the group's last
// member), read from global memory in the permuted head_dim order and
// converted to f16; the running state starts empty.  Query rows are 16-byte
// aligned (the host requires it for an fp8 cache).
template <typename T, int D, int NT>
__device__ __forceinline__ void load_q_members_e4m3(MmaState<__half, D, NT>& st, const DecodeParams& p, int b0,
                                                    int n_members, int h0, int nh, int lane) {
  const int hh = lane >> 2;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const bool valid = hh < nh && nt < n_members;
    const T* row = reinterpret_cast<const T*>(p.q) + (valid ? b0 + nt : 0) * p.q_sb +
                   static_cast<int64_t>(h0 + (valid ? hh : 0)) * p.q_sh;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int d = ks * 16 + 4 * (lane & 3);
      uint32_t b0r = 0u, b1r = 0u;
      if (valid) {
        const uint2 raw = *reinterpret_cast<const uint2*>(row + d);
        if constexpr (std::is_same<T, __half>::value) {
          b0r = raw.x;
          b1r = raw.y;
        } else {
          const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
          const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
          b0r = Mma<__half>::pack(f0.x, f0.y);
          b1r = Mma<__half>::pack(f1.x, f1.y);
        }
      }
      st.qb[nt][ks][0] = b0r;
      st.qb[nt][ks][1] = b1r;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      st.m[nt][j] = -INFINITY;
      st.l[nt][j] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.o[mt][nt][e] = 0.f;
  }
}

// Finish the member sequences b0 .. b0+n_members-1 (column tiles of one warp)
// of a prefix-group unit over partition `part`: each member's output (times
// v_scale) when it has one partition, otherwise its partial (O times v_scale).
// Output rows follow the V fragment order: m-tile mt holds d = 16 mt + 2g
// (entries 0, 1) and 16 mt + 2g + 1 (entries 2, 3).
template <typename T, int D, int NT>
__device__ __forceinline__ void finish_members_e4m3(MmaState<__half, D, NT>& st, const DecodeParams& p, int b0,
                                                    int n_members, int part, int h0, int nh, int lane) {
  const int l_max = p.max_blocks * p.block_size;
  const int hh = 2 * (lane & 3);
  T* out = reinterpret_cast<T*>(p.out);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if (nt >= n_members) break;
    const int b = b0 + nt;
    int L = p.context_lens[b];
    L = L < 0 ? 0 : (L > l_max ? l_max : L);
    const int n_parts = L == 0 ? 1 : (L + p.part_tokens - 1) / p.part_tokens;
    float l[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float v = st.l[nt][j];
      v += __shfl_xor_sync(kFullMask, v, 4);
      v += __shfl_xor_sync(kFullMask, v, 8);
      v += __shfl_xor_sync(kFullMask, v, 16);
      l[j] = v;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (hh + j >= nh) continue;
      if (n_parts == 1) {
        const float inv = p.v_scale / l[j];
        T* r = out + b * p.o_sb + static_cast<int64_t>(h0 + hh + j) * p.o_sh;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const int d = mt * 16 + 2 * (lane >> 2);
          r[d] = from_f32<T>(st.o[mt][nt][j] * inv);
          r[d + 1] = from_f32<T>(st.o[mt][nt][2 + j] * inv);
        }
      } else {
        const int64_t slot = static_cast<int64_t>(b * p.num_q_heads + h0 + hh + j) * p.max_parts + part;
        float* wo = p.ws_o + slot * D;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const int d = mt * 16 + 2 * (lane >> 2);
          *reinterpret_cast<float2*>(wo + d) = make_float2(st.o[mt][nt][j] * p.v_scale, st.o[mt][nt][2 + j] * p.v_scale);
        }
        if ((lane >> 2) == 0) reinterpret_cast<float2*>(p.ws_ml)[slot] = make_float2(st.m[nt][j], l[j]);
      }
    }
  }
}

// This warp's (m, l, O) into the CTA reduction area, undoing the row order of
// the V fragments (m-tile mt holds d = 16 mt + 2g and 16 mt + 2g + 1).
template <int D, int NT>
__device__ __forceinline__ void mma_store_e4m3(MmaState<__half, D, NT>& st, float* red_o, float* red_m,
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
      const int d = mt * 16 + 2 * (lane >> 2);
      *reinterpret_cast<float2*>(red_o + hh * D + d) = make_float2(st.o[mt][nt][0], st.o[mt][nt][2]);
      *reinterpret_cast<float2*>(red_o + (hh + 1) * D + d) = make_float2(st.o[mt][nt][1], st.o[mt][nt][3]);
    }
}

}  // namespace wllm
