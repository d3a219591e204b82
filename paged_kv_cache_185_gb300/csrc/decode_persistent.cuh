// decode_persistent.cuh -- persistent, warp-specialised paged decode for
// f16/bf16 (tensor-core QK^T and PV), sm_103a.
//
// Work is cut into units (sequence b, kv-head tile z, partition p of P tokens).
// The grid is a few CTAs per SM; each CTA loops until the units run out.
//
//   producer warp: takes the next unit from a device-wide atomic counter,
//     loads that unit's block-table entries (32 chunks per coalesced load),
//     and for every 16-token chunk waits for a free stage of the CTA's ring,
//     writes the chunk's metadata, and issues 3-D TMA tiled copies of the 16
//     K rows and 16 V rows of the kv head (128-byte swizzled); the first chunk
//     of a unit also carries the unit's query rows (bulk copy).  It runs
//     ahead across unit boundaries, so the copies of the next unit are in
//     flight while the consumers finish the current one.
//   consumer warps (4): every consumer sees every chunk.  Each computes the
//     full S^T = K Q^T tile with mma.sync (cheap, so done redundantly), the
//     online-softmax update, and PV for its own quarter of head_dim; after
//     the chunk it releases the stage.  No cross-warp merge is needed: the
//     running max and sum are the same in every consumer warp.
//
// A unit's result is written to `out` when the sequence has one partition.
// Otherwise each consumer warp writes its partial (m, l, O slice) to the
// workspace; with few partitions the last warp to arrive for (b, z, quarter)
// -- an atomic counter, never waited for -- combines them, with many a
// separate combine kernel does it after the launch.
//
// Every wait is bounded: on timeout the warp records an error bit and leaves.
// The scheduler counter is reset by the last CTA to finish, so it is zero
// between launches.
#pragma once

#include "decode_kernel.cuh"

namespace wllm {

// the scheduler words live next to the error word (offsets in ints)
constexpr int kSchedNextOffset = 16;
constexpr int kSchedDoneOffset = 32;

struct ChunkMeta {
  int b, p, t0, tok_end;
  int n_parts, h0, nh, flags;
  int z, pad0, pad1, pad2;
};
enum : int { kFirst = 1, kLast = 2, kEmptySeq = 4, kStop = 8 };

template <typename T, int D, int NT>
struct PShape {
  static constexpr int kConsumers = 4;
  static constexpr int kThreads = (kConsumers + 1) * 32;
  static constexpr int kHeadTile = 8 * NT;
  static constexpr int kKV = Geom<T, D>::kTileBytes;
  static constexpr int kQBytes = kHeadTile * D * static_cast<int>(sizeof(T));
  static constexpr int kStageBytes = ((2 * kKV + kQBytes) + 1023) / 1024 * 1024;
  static constexpr int kStages = D == 64 ? 12 : (D == 128 ? 8 : 5);
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kBarBytes = 2 * kStages * 8;
  static constexpr int kMetaBytes = kStages * static_cast<int>(sizeof(ChunkMeta));
  static constexpr int kFixedSmem = 1024 + kRingBytes + kBarBytes + kMetaBytes;
  static constexpr int kMT = D / 16 / kConsumers;  // PV m-tiles (16 columns of d) per consumer
  static constexpr int kDW = D / kConsumers;       // output columns per consumer
  static_assert(kMT >= 1, "head_dim too small for the consumer split");
};

// Consumer state: full-width Q^T fragments, this warp's quarter of O^T.
template <typename T, int D, int NT>
struct PState {
  float o[PShape<T, D, NT>::kMT][NT][4];
  float m[NT][2];
  float l[NT][2];
  uint32_t qb[NT][D / 16][2];
};

template <typename T, int D, int NT>
__device__ __forceinline__ void pstate_begin(PState<T, D, NT>& st, const uint8_t* qtile, int nh, int lane) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 8 + (lane >> 2);
    const bool valid = hh < nh;
    const T* row = reinterpret_cast<const T*>(qtile) + (valid ? hh : 0) * D;
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
    for (int i = 0; i < PShape<T, D, NT>::kMT; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.o[i][nt][e] = 0.f;
  }
}

template <typename T, int D, int NT>
__device__ __forceinline__ void pstate_chunk(PState<T, D, NT>& st, uint32_t k_tile, uint32_t v_tile, int t0,
                                             int tok_end, float scale_log2, int cw, int lane) {
  constexpr int kMT = PShape<T, D, NT>::kMT;
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
    for (int i = 0; i < kMT; ++i)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        st.o[i][nt][0] *= alpha[nt][0];
        st.o[i][nt][1] *= alpha[nt][1];
        st.o[i][nt][2] *= alpha[nt][0];
        st.o[i][nt][3] *= alpha[nt][1];
      }
  }

  const int v_row = (lane & 7) + ((lane >> 4) << 3);
  const int v_chunk = (lane >> 3) & 1;
  const bool tail = t0 + kChunk > tok_end;
  const int tk = t0 + 2 * (lane & 3);
  const uint32_t keep_lo = (tk < tok_end ? 0x0000ffffu : 0u) | (tk + 1 < tok_end ? 0xffff0000u : 0u);
  const uint32_t keep_hi = (tk + 8 < tok_end ? 0x0000ffffu : 0u) | (tk + 9 < tok_end ? 0xffff0000u : 0u);
#pragma unroll
  for (int i = 0; i < kMT; ++i) {
    const int mt = cw * kMT + i;
    uint32_t a[4];
    ldsm_x4_trans(v_tile + tile_offset(v_row, 2 * mt + v_chunk), a);
    if (tail) {
      a[0] &= keep_lo;
      a[1] &= keep_lo;
      a[2] &= keep_hi;
      a[3] &= keep_hi;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) Mma<T>::run(st.o[i][nt], a, pb[nt]);
  }
}

// The split-KV partials of one (row, partition): ws_o[row][part][D] holds the
// unnormalised O, ws_ml[row][part][consumer] the (max in log2 units, sum) pair
// written by each consumer warp (identical values, one copy per writer so that
// a combining warp reads only its own writers' data).
template <typename T, int D, int NT>
__device__ __forceinline__ void pstate_finish(PState<T, D, NT>& st, const ChunkMeta& mt_, const DecodeParams& p,
                                              int cw, int lane) {
  constexpr int kMT = PShape<T, D, NT>::kMT;
  constexpr int kW = PShape<T, D, NT>::kConsumers;
  constexpr int kDW = PShape<T, D, NT>::kDW;
  T* out = reinterpret_cast<T*>(p.out);
  const int b = mt_.b, h0 = mt_.h0, nh = mt_.nh;
  if (mt_.flags & kEmptySeq) {
    for (int idx = lane; idx < nh * kDW; idx += 32) {
      const int hh = idx / kDW, d = cw * kDW + idx % kDW;
      out[b * p.o_sb + static_cast<int64_t>(h0 + hh) * p.o_sh + d] = from_f32<T>(0.f);
    }
    return;
  }
  float l[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float v = st.l[nt][j];
      v += __shfl_xor_sync(kFullMask, v, 4);
      v += __shfl_xor_sync(kFullMask, v, 8);
      v += __shfl_xor_sync(kFullMask, v, 16);
      l[nt][j] = v;
    }
  if (mt_.n_parts == 1) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hh = nt * 8 + 2 * (lane & 3);
      const float inv0 = 1.f / l[nt][0], inv1 = 1.f / l[nt][1];
#pragma unroll
      for (int i = 0; i < kMT; ++i) {
        const int d = (cw * kMT + i) * 16 + (lane >> 2);
        if (hh < nh) {
          T* r = out + b * p.o_sb + static_cast<int64_t>(h0 + hh) * p.o_sh;
          r[d] = from_f32<T>(st.o[i][nt][0] * inv0);
          r[d + 8] = from_f32<T>(st.o[i][nt][2] * inv0);
        }
        if (hh + 1 < nh) {
          T* r = out + b * p.o_sb + static_cast<int64_t>(h0 + hh + 1) * p.o_sh;
          r[d] = from_f32<T>(st.o[i][nt][1] * inv1);
          r[d + 8] = from_f32<T>(st.o[i][nt][3] * inv1);
        }
      }
    }
    return;
  }

  // several partitions: write this warp's partial
  const int row0 = b * p.num_q_heads + h0;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 8 + 2 * (lane & 3);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (hh + j < nh) {
        const int64_t slot = static_cast<int64_t>(row0 + hh + j) * p.max_parts + mt_.p;
        float* wo = p.ws_o + slot * D;
#pragma unroll
        for (int i = 0; i < kMT; ++i) {
          const int d = (cw * kMT + i) * 16 + (lane >> 2);
          wo[d] = st.o[i][nt][j];
          wo[d + 8] = st.o[i][nt][2 + j];
        }
        if ((lane >> 2) == 0)
          reinterpret_cast<float2*>(p.ws_ml)[slot * kW + cw] = make_float2(st.m[nt][j], l[nt][j]);
      }
    }
  }
  if (p.ws_count == nullptr) return;  // a separate combine kernel finishes the job

  __threadfence();
  __syncwarp();
  const int z = mt_.z;
  int* counter = p.ws_count + (static_cast<int64_t>(b) * p.num_kv_heads * p.num_head_tiles + z) * kW + cw;
  int last = 0;
  if (lane == 0) last = atomicAdd(counter, 1) == mt_.n_parts - 1;
  last = __shfl_sync(kFullMask, last, 0);
  if (!last) return;
  __threadfence();
  const int n_parts = mt_.n_parts;
  for (int hh = 0; hh < nh; ++hh) {
    const int64_t base = static_cast<int64_t>(row0 + hh) * p.max_parts;
    float M = -INFINITY;
    for (int pp = lane; pp < n_parts; pp += 32)
      M = fmaxf(M, __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + (base + pp) * kW + cw).x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
    float den = 0.f;
    for (int pp = lane; pp < n_parts; pp += 32) {
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + (base + pp) * kW + cw);
      den += exp2f(ml.x - M) * ml.y;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(kFullMask, den, off);
    const float inv = 1.f / den;
    T* orow = out + b * p.o_sb + static_cast<int64_t>(h0 + hh) * p.o_sh;
    // lanes cover the warp's kDW columns; extra lanes take every other partition
    constexpr int kLanesPerCol = kDW >= 32 ? 1 : 32 / kDW;
    constexpr int kCols = kDW >= 32 ? kDW / 32 : 1;
    const int sub = kDW >= 32 ? 0 : lane / kDW;
#pragma unroll
    for (int c = 0; c < kCols; ++c) {
      const int d = cw * kDW + (kDW >= 32 ? lane + 32 * c : lane % kDW);
      float num = 0.f;
      for (int pp = sub; pp < n_parts; pp += kLanesPerCol) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + (base + pp) * kW + cw);
        num = fmaf(exp2f(ml.x - M), __ldcg(p.ws_o + (base + pp) * D + d), num);
      }
      // fold the kLanesPerCol partial sums of column d (lanes d, d + kDW, ...)
      if constexpr (kDW < 32) {
#pragma unroll
        for (int off = kDW; off < 32; off <<= 1) num += __shfl_xor_sync(kFullMask, num, off);
      }
      if (sub == 0) orow[d] = from_f32<T>(num * inv);
    }
  }
  if (lane == 0) *counter = 0;
}

template <typename T, int D, int NT>
__global__ void __launch_bounds__(PShape<T, D, NT>::kThreads)
    paged_decode_persistent(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                            const DecodeParams p) {
  using G = Geom<T, D>;
  using PS = PShape<T, D, NT>;
  constexpr int S = PS::kStages;
  constexpr int W = PS::kConsumers;
  constexpr int HT = PS::kHeadTile;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + PS::kRingBytes);
  uint64_t* empty = full + S;
  ChunkMeta* meta = reinterpret_cast<ChunkMeta*>(empty + S);
  int* prefix = reinterpret_cast<int*>(meta + S);  // [B + 1] units before sequence b

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = p.num_seqs;
  const int Z = p.num_kv_heads * p.num_head_tiles;
  const int l_max = p.max_blocks * p.block_size;

  // units per sequence and their prefix sums (every CTA computes them)
  {
    const int nthr = PS::kThreads;
    const int per = (B + nthr - 1) / nthr;
    const int lo = threadIdx.x * per, hi = min(B, lo + per);
    int local = 0;
    for (int b = lo; b < hi; ++b) {
      int L = p.context_lens[b];
      L = L < 0 ? 0 : (L > l_max ? l_max : L);
      local += (L == 0 ? 1 : (L + p.part_tokens - 1) / p.part_tokens) * Z;
    }
    // exclusive scan of the per-thread sums (one warp, serially over warps' totals)
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(kFullMask, incl, off);
      if (lane >= off) incl += v;
    }
    int* wsum = reinterpret_cast<int*>(meta);  // scratch before meta is used
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int woff = 0;
    for (int w = 0; w < warp; ++w) woff += wsum[w];
    int run = woff + incl - local;
    for (int b = lo; b < hi; ++b) {
      prefix[b] = run;
      int L = p.context_lens[b];
      L = L < 0 ? 0 : (L > l_max ? l_max : L);
      run += (L == 0 ? 1 : (L + p.part_tokens - 1) / p.part_tokens) * Z;
    }
    if (threadIdx.x == PS::kThreads - 1) {
      int tot = 0;
      for (int w = 0; w < PS::kThreads / 32; ++w) tot += wsum[w];
      prefix[B] = tot;
    }
    if (threadIdx.x == 0) {
      for (int s = 0; s < S; ++s) {
        mbar_init(smem_u32(full + s), 1);
        mbar_init(smem_u32(empty + s), W);
      }
      fence_mbar_init();
    }
    __syncthreads();
  }
  const int total_units = prefix[B];

  if (warp == W) {
    // ------------------------------- producer -------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    int* sched_next = p.err + kSchedNextOffset;
    int* sched_done = p.err + kSchedDoneOffset;
    int k = 0;
    bool ok = true;
    auto acquire_stage = [&](int kk) -> bool {
      const int s = kk % S;
      bool got = true;
      if (lane == 0) got = mbar_wait_bounded(smem_u32(empty + s), ((kk / S) & 1) ^ 1, p.wait_limit_ns);
      return __shfl_sync(kFullMask, got ? 1 : 0, 0) != 0;
    };
    while (ok) {
      int u = 0;
      if (lane == 0) u = atomicAdd(sched_next, 1);
      u = __shfl_sync(kFullMask, u, 0);
      if (u >= total_units) break;
      // sequence of unit u: prefix[b] <= u < prefix[b+1]
      int lo = 0, hi = B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= u) lo = mid;
        else hi = mid - 1;
      }
      const int b = lo;
      const int r = u - prefix[b];
      const int part = r / Z, z = r - (r / Z) * Z;
      int L = p.context_lens[b];
      if (L < 0 || L > l_max) {
        if (lane == 0 && part == 0 && z == 0) atomicOr(p.err, kErrLen);
        L = L < 0 ? 0 : l_max;
      }
      const int n_parts = L == 0 ? 1 : (L + p.part_tokens - 1) / p.part_tokens;
      const int kvh = z / p.num_head_tiles, ht = z - kvh * p.num_head_tiles;
      const int h0 = kvh * p.group + ht * HT;
      const int nh = min(HT, p.group - ht * HT);
      const int tb = part * p.part_tokens;
      const int te = min(L, tb + p.part_tokens);
      const int n_chunks = L == 0 ? 0 : (te - tb + kChunk - 1) / kChunk;
      if (n_chunks == 0) {
        if (!acquire_stage(k)) { ok = false; break; }
        if (lane == 0) {
          meta[k % S] = ChunkMeta{b, part, 0, 0, n_parts, h0, nh, kFirst | kLast | kEmptySeq, z, 0, 0, 0};
          mbar_arrive_expect_tx(smem_u32(full + k % S), 0);
        }
        ++k;
        continue;
      }
      const int32_t* bt_row = p.block_tables + static_cast<int64_t>(b) * p.bt_stride;
      const T* qsrc = reinterpret_cast<const T*>(p.q) + b * p.q_sb + static_cast<int64_t>(h0) * p.q_sh;
      int e0 = 0, e1 = 0;
      for (int c = 0; c < n_chunks; ++c) {
        if ((c & 31) == 0) {  // this unit's next 32 table entries, one per lane
          const int cc = c + lane;
          e0 = 0;
          e1 = 0;
          if (cc < n_chunks) {
            const int t0 = tb + kChunk * cc;
            int x0 = bt_row[t0 >> p.log2_bs], x1 = 0;
            if (p.log2_bs < 4 && t0 + 8 < te) x1 = bt_row[(t0 >> p.log2_bs) + 1];
            if (x0 < 0 || x0 >= p.num_blocks || x1 < 0 || x1 >= p.num_blocks) {
              atomicOr(p.err, kErrBlock);
              x0 = (x0 < 0 || x0 >= p.num_blocks) ? 0 : x0;
              x1 = (x1 < 0 || x1 >= p.num_blocks) ? 0 : x1;
            }
            e0 = x0;
            e1 = x1;
          }
        }
        const int pb0 = __shfl_sync(kFullMask, e0, c & 31);
        const int pb1 = __shfl_sync(kFullMask, e1, c & 31);
        if (!acquire_stage(k)) { ok = false; break; }
        if (lane == 0) {
          const int s = k % S;
          const int t0 = tb + kChunk * c;
          const uint32_t stage = smem_u32(ring + s * PS::kStageBytes);
          const uint32_t bar = smem_u32(full + s);
          const int flags = (c == 0 ? kFirst : 0) | (c == n_chunks - 1 ? kLast : 0);
          meta[s] = ChunkMeta{b, part, t0, te, n_parts, h0, nh, flags, z, 0, 0, 0};
          const bool two = p.log2_bs < 4;
          const bool has1 = two && (t0 + 8 < te);
          uint32_t bytes = (two && !has1) ? G::kStageBytes / 2 : G::kStageBytes;
          if (c == 0) bytes += nh * D * static_cast<int>(sizeof(T));
          mbar_arrive_expect_tx(bar, bytes);
          if (!two) {
            const int y = kvh * p.block_size + (t0 & (p.block_size - 1));
#pragma unroll
            for (int cb = 0; cb < G::kColBoxes; ++cb) {
              tma_load_3d(stage + cb * 2048, &kmap, bar, cb * G::kBoxCols, y, pb0);
              tma_load_3d(stage + PS::kKV + cb * 2048, &vmap, bar, cb * G::kBoxCols, y, pb0);
            }
          } else {
            const int y = kvh * p.block_size;
#pragma unroll
            for (int cb = 0; cb < G::kColBoxes; ++cb) {
              tma_load_3d(stage + cb * 2048, &kmap, bar, cb * G::kBoxCols, y, pb0);
              tma_load_3d(stage + PS::kKV + cb * 2048, &vmap, bar, cb * G::kBoxCols, y, pb0);
              if (has1) {
                tma_load_3d(stage + cb * 2048 + 1024, &kmap, bar, cb * G::kBoxCols, y, pb1);
                tma_load_3d(stage + PS::kKV + cb * 2048 + 1024, &vmap, bar, cb * G::kBoxCols, y, pb1);
              }
            }
          }
          if (c == 0) {
            for (int hh = 0; hh < nh; ++hh)
              bulk_load(stage + 2 * PS::kKV + hh * D * static_cast<int>(sizeof(T)), qsrc + hh * p.q_sh,
                        D * static_cast<int>(sizeof(T)), bar);
          }
        }
        ++k;
      }
    }
    // tell the consumers to stop, then leave the scheduler clean
    if (ok && acquire_stage(k)) {
      if (lane == 0) {
        meta[k % S].flags = kStop;
        mbar_arrive_expect_tx(smem_u32(full + k % S), 0);
      }
    } else if (lane == 0) {
      atomicOr(p.err, kErrWaitTimeout);
    }
    if (lane == 0) {
      __threadfence();
      if (atomicAdd(sched_done, 1) == static_cast<int>(gridDim.x) - 1) {
        atomicExch(sched_next, 0);
        atomicExch(sched_done, 0);
      }
    }
    return;
  }

  // ------------------------------- consumers --------------------------------
  PState<T, D, NT> st;
  const int cw = warp;
  for (int k = 0;; ++k) {
    const int s = k % S;
    if (!mbar_wait_bounded(smem_u32(full + s), (k / S) & 1, p.wait_limit_ns)) {
      if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
      return;
    }
    const ChunkMeta mt_ = meta[s];
    if (mt_.flags & kStop) return;
    const uint32_t stage = smem_u32(ring + s * PS::kStageBytes);
    if (!(mt_.flags & kEmptySeq)) {
      if (mt_.flags & kFirst) pstate_begin<T, D, NT>(st, ring + s * PS::kStageBytes + 2 * PS::kKV, mt_.nh, lane);
      pstate_chunk<T, D, NT>(st, stage, stage + PS::kKV, mt_.t0, mt_.tok_end, p.scale_log2, cw, lane);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + s));
    if (mt_.flags & kLast) pstate_finish<T, D, NT>(st, mt_, p, cw, lane);
  }
}

// Combine kernel for launches with many partitions per sequence: one CTA per
// query row (b, h); warps split the partitions, lanes the columns.
template <typename T, int D>
__global__ void __launch_bounds__(256) splitkv_combine(const DecodeParams p, int ml_stride) {
  const int row = blockIdx.x;
  const int b = row / p.num_q_heads;
  int L = p.context_lens[b];
  const int l_max = p.max_blocks * p.block_size;
  L = L < 0 ? 0 : (L > l_max ? l_max : L);
  const int n_parts = L == 0 ? 1 : (L + p.part_tokens - 1) / p.part_tokens;
  if (n_parts == 1) return;  // written by the decode kernel
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = 8;
  constexpr int kPer = D / 32;  // columns per lane
  __shared__ float red_m[kWarps];
  __shared__ float red_l[kWarps];
  __shared__ float red_o[kWarps][D];
  const int64_t base = static_cast<int64_t>(row) * p.max_parts;
  const float2* ml = reinterpret_cast<const float2*>(p.ws_ml);
  float M = -INFINITY;
  for (int pp = threadIdx.x; pp < n_parts; pp += blockDim.x) M = fmaxf(M, ml[(base + pp) * ml_stride].x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
  if (lane == 0) red_m[warp] = M;
  __syncthreads();
  M = red_m[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, red_m[w]);
  float den = 0.f, num[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) num[i] = 0.f;
  for (int pp = warp; pp < n_parts; pp += kWarps) {
    const float2 v = ml[(base + pp) * ml_stride];
    const float f = exp2f(v.x - M);
    den += f * v.y;
    const float* o = p.ws_o + (base + pp) * D;
#pragma unroll
    for (int i = 0; i < kPer; ++i) num[i] = fmaf(f, o[lane + 32 * i], num[i]);
  }
  if (lane == 0) red_l[warp] = den;
#pragma unroll
  for (int i = 0; i < kPer; ++i) red_o[warp][lane + 32 * i] = num[i];
  __syncthreads();
  if (warp == 0) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += red_l[w];
    const float inv = 1.f / tot;
    const int h = row - b * p.num_q_heads;
    T* orow = reinterpret_cast<T*>(p.out) + b * p.o_sb + static_cast<int64_t>(h) * p.o_sh;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) acc += red_o[w][lane + 32 * i];
      orow[lane + 32 * i] = from_f32<T>(acc * inv);
    }
  }
}

template <typename T, int D, int NT>
int persistent_smem(int num_seqs) {
  return PShape<T, D, NT>::kFixedSmem + ((num_seqs + 1) * 4 + 15) / 16 * 16;
}

template <typename T, int D, int NT>
int launch_persistent_inst(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p, int grid,
                           bool separate_combine, cudaStream_t stream) {
  using PS = PShape<T, D, NT>;
  auto kernel = paged_decode_persistent<T, D, NT>;
  const int smem = persistent_smem<T, D, NT>(p.num_seqs);
  static int configured_for[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && configured_for[dev] < smem) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured_for[dev] = 227 * 1024;
  }
  kernel<<<grid, PS::kThreads, smem, stream>>>(kmap, vmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || !separate_combine) return e;
  splitkv_combine<T, D><<<p.num_seqs * p.num_q_heads, 256, 0, stream>>>(p, PS::kConsumers);
  return cudaGetLastError();
}

template <typename T, int D, int NT>
int persistent_occupancy(int num_seqs) {
  int blocks = 0;
  const int smem = persistent_smem<T, D, NT>(num_seqs);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, paged_decode_persistent<T, D, NT>,
                                                    PShape<T, D, NT>::kThreads, smem) != cudaSuccess)
    return 1;
  return blocks < 1 ? 1 : blocks;
}

}  // namespace wllm
