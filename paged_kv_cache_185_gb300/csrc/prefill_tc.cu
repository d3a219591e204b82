// prefill_tc.cu -- chunked-prefill (multi-query) paged attention on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory), for
// f16/bf16 caches with head_dim 64 or 128.
//
// The operation is that of prefill.cu ("wLLM" project page, "Features / Core
// engine": chunked prefill into the paged KV cache; "mini-vLLM" README, "How it
// works / Paged KV-cache": block tables over a pool of physical blocks): chunk
// token i of sequence b sits at position P = L_b - n_b + i and attends to the
// cached tokens 0 .. P.  The tiling is this library's design.
//
// One CTA owns 128 query rows of one sequence and one kv head -- row r of the
// sequence's chunk is (token r / G, query head r % G of the kv head's group), so
// the G heads of a group share every staged K/V byte -- and walks the rows'
// context in 64-token tiles.  Six warps:
//
//   warp 0 (producer): reads the block table and stages each tile's K and then
//     its V (16-row TMA boxes, 128-byte swizzle) into a ring of slots laid out
//     [head_dim / 64][64 tokens][128 bytes], so that the 8-row groups of a slot
//     sit 1024 bytes apart, as the MMA descriptors require;
//   warp 1 (MMA): one thread issues S_j = Q K_j^T (M = 128, N = 64, K = 16 per
//     instruction; Q and K both K-major) into one of two TMEM buffers, then,
//     once the softmax has written P_{j-1} to shared memory, O += P_{j-1} V_{j-1}
//     (M = 128, N = head_dim; V read MN-major straight from its slot); each
//     group of MMAs completes onto an mbarrier (tcgen05.commit), which also
//     hands the slot back to the producer.  S_{j+1} is computed while the
//     softmax works on S_j;
//   warps 2-5 (softmax): thread r owns row r (TMEM lane r): it loads its row of
//     Q into shared memory once, then per tile reads its 64 scores from TMEM,
//     applies the scale and the causal mask, and updates a running maximum that
//     is only moved when a score exceeds it by more than 8 in the log2 domain
//     (so weights stay below 2^8; O in TMEM is rescaled only on such a move),
//     rounds the weights P to the input type, writes them into the
//     shared-memory A operand of the PV product and adds the ROUNDED weights to
//     the running sum: numerator and denominator then use the same weights, so
//     a dominant token whose weight is not exactly 1 (the maximum being stale)
//     adds no rounding error of its own.  At the end it divides O by the
//     running sum and stores the row.
//
// Two CTAs fit on an SM (shared memory ~99 KB each, 256 TMEM columns each: S0,
// S1 and O), so one CTA's softmax overlaps the other's tensor-core work.  Every
// mbarrier wait is bounded; on a timeout the CTA records the error, waits
// (bounded) for its copies and MMAs in flight, frees its TMEM and returns.
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace wllm {

namespace {

constexpr int kTcRows = 128;        // query rows per CTA (one M = 128 tile)
constexpr int kTcKv = 64;           // kv tokens per tile
constexpr int kTcThreads = 6 * 32;  // producer, MMA, four softmax warps
constexpr float kTcRescale = 8.f;   // the running maximum moves by more than 2^8 only

template <int D>
struct TcShape {
  static constexpr int kChunks = D / 64;               // 128-byte chunks of a 16-bit row
  static constexpr int kQBytes = kTcRows * D * 2;      // [chunk][128 rows][128 B]
  static constexpr int kPBytes = kTcRows * kTcKv * 2;  // [128 rows][128 B]
  static constexpr int kSlotBytes = kTcKv * D * 2;     // [chunk][64 tokens][128 B]
  static constexpr int kSlots = D == 64 ? 8 : 3;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmem = 1024 + kQBytes + kPBytes + kSlots * kSlotBytes + kBarBytes;
  static constexpr uint32_t kTmemCols = 256;
  static constexpr int kS0 = 0, kS1 = 64, kO = 128;  // TMEM columns: scores (two buffers), output
};
// At most two CTAs fit on an SM, so their 2 x 256 TMEM columns always fit and
// an allocation never waits.
static_assert(3 * (TcShape<64>::kSmem + 1024) > 233472 && 3 * (TcShape<128>::kSmem + 1024) > 233472,
              "a third resident CTA would contend for TMEM");
static_assert(2 * (TcShape<128>::kSmem + 1024) <= 233472, "two CTAs per SM");

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Sum of the two 16-bit values of a pair (exact in fp32).
template <typename T>
__device__ __forceinline__ float pair_sum(uint32_t w);
template <>
__device__ __forceinline__ float pair_sum<__nv_bfloat16>(uint32_t w) {
  return __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
}
template <>
__device__ __forceinline__ float pair_sum<__half>(uint32_t w) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
  return f.x + f.y;
}

template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 2)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                            const PrefillParams p) {
  using TS = TcShape<D>;
  constexpr int R = TS::kSlots;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* p_s = q_s + TS::kQBytes;
  uint8_t* ring = p_s + TS::kPBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + R * TS::kSlotBytes);
  uint64_t* empty = full + R;
  uint64_t* sfull = empty + R;   // [2] S buffer written (MMA -> softmax)
  uint64_t* sfree = sfull + 2;   // [2] S buffer read (softmax -> MMA)
  uint64_t* pfull = sfree + 2;   // P written, O rescaled (softmax -> MMA)
  uint64_t* odone = pfull + 1;   // a PV product done (MMA -> softmax)
  uint64_t* qfull = odone + 1;   // Q written (softmax -> MMA)
  uint64_t* fin = qfull + 1;     // every MMA of the CTA done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(fin + 1);
  int* info = reinterpret_cast<int*>(tslot + 1);  // [0] sequence (-1: none), [1] its row tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int kvh = blockIdx.y;

  // ---- which (sequence, row tile) this CTA owns: sequence b owns
  // ceil(n_b * G / 128) consecutive slots of blockIdx.x
  if (warp == 0) {
    int seq = -1, tile = 0, base = 0;
    for (int b0 = 0; b0 < p.num_seqs && seq < 0; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < p.num_seqs) n = p.query_start_loc[b + 1] - p.query_start_loc[b];
      n = n < 0 ? 0 : n;
      const int tiles = static_cast<int>((static_cast<int64_t>(n) * G + kTcRows - 1) / kTcRows);
      int incl = tiles;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(kFullMask, incl, off);
        if (lane >= off) incl += v;
      }
      const int excl = incl - tiles;
      const int tgt = static_cast<int>(blockIdx.x) - base;
      const unsigned hit = __ballot_sync(kFullMask, b < p.num_seqs && tgt >= excl && tgt < incl);
      if (hit != 0u) {
        const int src = __ffs(hit) - 1;
        seq = b0 + src;
        const int t_in = tgt - __shfl_sync(kFullMask, excl, src);
        const int t_all = __shfl_sync(kFullMask, tiles, src);
        tile = t_all - 1 - t_in;  // the sequence's last rows (longest context) first
      }
      base += __shfl_sync(kFullMask, incl, 31);
    }
    if (lane == 0) {
      info[0] = seq;
      info[1] = tile;
      for (int s = 0; s < R; ++s) {
        mbar_init(smem_u32(full + s), 1);
        mbar_init(smem_u32(empty + s), 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(smem_u32(sfull + i), 1);
        mbar_init(smem_u32(sfree + i), 4);
      }
      mbar_init(smem_u32(pfull), 4);
      mbar_init(smem_u32(odone), 1);
      mbar_init(smem_u32(qfull), 4);
      mbar_init(smem_u32(fin), 1);
      fence_mbar_init();
    }
  } else if (warp == 1) {
    tc::alloc(smem_u32(tslot), TS::kTmemCols);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;

  // ---- the tile's rows and the context they see (uniform over the CTA)
  const int b = info[0];
  int n_tiles = 0, row0 = 0, n_rows = 0, pos0 = 0, kv_end = 0, s0 = 0;
  if (b >= 0) {
    const int l_max = p.max_blocks * p.block_size;
    s0 = p.query_start_loc[b];
    int n = p.query_start_loc[b + 1] - s0;
    if (s0 < 0 || n < 0 || static_cast<int64_t>(s0) + n > p.num_tokens) {  // inconsistent query starts
      if (threadIdx.x == 0) atomicOr(p.err, kErrLen);
    } else {
      int L = p.context_lens[b];
      if (L < 0 || L > l_max || n > L) {
        if (threadIdx.x == 0) atomicOr(p.err, kErrLen);
        L = L < 0 ? 0 : (L > l_max ? l_max : L);
        n = n > L ? L : n;
      }
      n_rows = n * G;
      row0 = info[1] * kTcRows;
      if (row0 < n_rows) {  // (not so only when n was clamped, error already flagged)
        const int row_last = min(n_rows, row0 + kTcRows) - 1;
        pos0 = L - n;
        kv_end = pos0 + row_last / G + 1;
        n_tiles = (kv_end + kTcKv - 1) / kTcKv;
      }
    }
  }

  // one lane waits, the warp learns the outcome
  auto wait_warp = [&](uint64_t* bar, int parity) -> bool {
    bool got = true;
    if (lane == 0) got = mbar_wait_bounded(smem_u32(bar), static_cast<uint32_t>(parity), p.wait_limit_ns);
    return __shfl_sync(kFullMask, got ? 1 : 0, 0) != 0;
  };
  bool ok = true;

  if (warp == 0 && n_tiles > 0) {
    // ------------------------------- producer -------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    const int32_t* bt_row = p.block_tables + static_cast<int64_t>(b) * p.bt_stride;
    const bool two = p.log2_bs < 4;  // 8-token blocks: two 8-row boxes per 16 tokens
    int issued = 0;                  // slot uses whose copies were issued
    for (int j = 0; ok && j < n_tiles; ++j) {
      // lanes 0..3: the table entries of the tile's four 16-token sub-tiles
      int e0 = 0, e1 = 0;
      const int tj = j * kTcKv + 16 * lane;
      if (lane < 4 && tj < kv_end) {
        e0 = bt_row[tj >> p.log2_bs];
        if (two && tj + 8 < kv_end) e1 = bt_row[(tj >> p.log2_bs) + 1];
        if (e0 < 0 || e0 >= p.num_blocks || e1 < 0 || e1 >= p.num_blocks) {
          atomicOr(p.err, kErrBlock);
          e0 = (e0 < 0 || e0 >= p.num_blocks) ? 0 : e0;
          e1 = (e1 < 0 || e1 >= p.num_blocks) ? 0 : e1;
        }
      }
      int ent0[4], ent1[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        ent0[jj] = __shfl_sync(kFullMask, e0, jj);
        ent1[jj] = __shfl_sync(kFullMask, e1, jj);
      }
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {  // K, then V
        const int c = 2 * j + half, s = c % R;
        if (!wait_warp(empty + s, ((c / R) & 1) ^ 1)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const CUtensorMap* map = half ? &vmap : &kmap;
          const uint32_t slot = smem_u32(ring + s * TS::kSlotBytes);
          const uint32_t bar = smem_u32(full + s);
          uint32_t bytes = 0;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int t = j * kTcKv + 16 * jj;
            if (t < kv_end) bytes += ((two && !(t + 8 < kv_end)) ? 8u : 16u) * 128u * TS::kChunks;
          }
          mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int t = j * kTcKv + 16 * jj;
            if (t >= kv_end) continue;
#pragma unroll
            for (int cb = 0; cb < TS::kChunks; ++cb) {
              const uint32_t dst = slot + cb * (kTcKv * 128) + jj * 2048;
              if (!two) {
                tma_load_3d(dst, map, bar, cb * 64, kvh * p.block_size + (t & (p.block_size - 1)), ent0[jj]);
              } else {
                tma_load_3d(dst, map, bar, cb * 64, kvh * p.block_size, ent0[jj]);
                if (t + 8 < kv_end) tma_load_3d(dst + 1024, map, bar, cb * 64, kvh * p.block_size, ent1[jj]);
              }
            }
          }
        }
        ++issued;
      }
    }
    // every copy still in flight lands before the CTA may leave
    for (int c = issued - R > 0 ? issued - R : 0; c < issued; ++c)
      if (!wait_warp(full + c % R, (c / R) & 1)) ok = false;
  } else if (warp == 1 && n_tiles > 0) {
    // --------------------------------- MMA ----------------------------------
    constexpr uint32_t kIdS = tc::f16_idesc(kBf16, false, false, kTcRows, kTcKv);
    constexpr uint32_t kIdO = tc::f16_idesc(kBf16, false, true, kTcRows, D);
    const uint32_t q_a = smem_u32(q_s), p_a = smem_u32(p_s), ring_a = smem_u32(ring);
    auto issue_pv = [&](int i) -> bool {
      if (!wait_warp(pfull, i & 1)) return false;
      const int c = 2 * i + 1, s = c % R;
      if (!wait_warp(full + s, (c / R) & 1)) return false;
      const int t0 = i * kTcKv;
      if (t0 + kTcKv > kv_end) {
        // V rows at or past kv_end were never staged (or hold slots past the
        // sequence's end): zero them, since P = 0 there does not cancel NaN
        const int r0 = kv_end - t0;
        uint8_t* slot = ring + s * TS::kSlotBytes;
        for (int idx = lane; idx < (kTcKv - r0) * TS::kChunks * 8; idx += 32) {
          const int row = r0 + idx / (TS::kChunks * 8);
          const int rem = idx - (idx / (TS::kChunks * 8)) * (TS::kChunks * 8);
          *reinterpret_cast<uint4*>(slot + (rem >> 3) * (kTcKv * 128) + row * 128 + (rem & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        tc::fence_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc::fence_after_sync();
        const uint32_t v0 = ring_a + s * TS::kSlotBytes;
#pragma unroll
        for (int kk = 0; kk < kTcKv / 16; ++kk)
          tc::mma_f16(tmem + TS::kO, tc::sw128_desc(p_a + kk * 32, 16, 1024),
                      tc::sw128_desc(v0 + kk * 2048, kTcKv * 128, 1024), kIdO, (i > 0 || kk > 0) ? 1u : 0u);
        tc::commit(smem_u32(odone));
        tc::commit(smem_u32(empty + s));
      }
      __syncwarp();
      return true;
    };
    ok = wait_warp(qfull, 0);
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int c = 2 * j, s = c % R;
      ok = wait_warp(full + s, (c / R) & 1) && wait_warp(sfree + (j & 1), ((j >> 1) & 1) ^ 1);
      if (!ok) break;
      if (lane == 0) {
        tc::fence_after_sync();
        const uint32_t k0 = ring_a + s * TS::kSlotBytes;
        const uint32_t d = tmem + ((j & 1) ? TS::kS1 : TS::kS0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int kc = ks >> 2, kin = ks & 3;
          tc::mma_f16(d, tc::sw128_desc(q_a + kc * (kTcRows * 128) + kin * 32, 16, 1024),
                      tc::sw128_desc(k0 + kc * (kTcKv * 128) + kin * 32, 16, 1024), kIdS, ks > 0 ? 1u : 0u);
        }
        tc::commit(smem_u32(sfull + (j & 1)));
        tc::commit(smem_u32(empty + s));
      }
      __syncwarp();
      if (j > 0) ok = issue_pv(j - 1);
    }
    if (ok) ok = issue_pv(n_tiles - 1);
    if (lane == 0) tc::commit(smem_u32(fin));  // every MMA issued above, on every path
    __syncwarp();
  } else if (warp >= 2 && n_tiles > 0) {
    // ------------------------------- softmax --------------------------------
    const int quarter = warp & 3;           // the TMEM lanes this warp reaches
    const int r = quarter * 32 + lane;      // this thread's row of the tile
    const int rowg = row0 + r;
    const bool valid = rowg < n_rows;
    const int tok = valid ? rowg / G : 0;
    const int gh = valid ? rowg - tok * G : 0;
    const int pos = valid ? pos0 + tok : 0;  // padding rows see token 0 only (output dropped)
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    {
      const T* qrow = reinterpret_cast<const T*>(p.q) + static_cast<int64_t>(s0 + tok) * p.q_st +
                      static_cast<int64_t>(kvh * G + gh) * p.q_sh;
#pragma unroll
      for (int c16 = 0; c16 < D / 8; ++c16) {
        const uint4 v = valid ? *reinterpret_cast<const uint4*>(qrow + c16 * 8) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(q_s + (c16 >> 3) * (kTcRows * 128) + r * 128 + (((c16 & 7) ^ (r & 7)) << 4)) = v;
      }
      tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(qfull));
    }
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < n_tiles; ++j) {
      if (!wait_warp(sfull + (j & 1), (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      float x[2][32];
      const uint32_t sc = trow + ((j & 1) ? TS::kS1 : TS::kS0);
      tc::ld32(sc, x[0]);
      tc::ld32(sc + 32, x[1]);
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(sfree + (j & 1)));
      const int t0 = j * kTcKv;
      float mx = -INFINITY;
      if (t0 + kTcKv - 1 <= pos) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            x[h][i] *= p.scale_log2;
            mx = fmaxf(mx, x[h][i]);
          }
      } else {  // the causal edge (and tokens past kv_end, whose K was never staged)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            x[h][i] = t0 + 32 * h + i <= pos ? x[h][i] * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, x[h][i]);
          }
      }
      float alpha = 1.f;
      if (mx > m + kTcRescale) {  // also the first tile (m = -inf): token 0 is always seen
        alpha = exp2f(m - mx);
        m = mx;
      }
      float sum = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t w = pack2<T>(exp2f(x[h][2 * i] - m), exp2f(x[h][2 * i + 1] - m));
          sum += pair_sum<T>(w);  // the rounded weights the PV product uses
          pk[16 * h + i] = w;
        }
      l = l * alpha + sum;
      if (j > 0) {  // PV_{j-1} has read P and written O
        if (!wait_warp(odone, (j - 1) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (__any_sync(kFullMask, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tc::ld32(trow + TS::kO + 32 * c, o);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tc::st32(trow + TS::kO + 32 * c, o);
          }
          tc::wait_st();
        }
      }
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<uint4*>(p_s + r * 128 + ((cc ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      tc::fence_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(pfull));
    }
    if (ok) ok = wait_warp(fin, 0);
    if (ok) {
      tc::fence_after_sync();
      const float inv = 1.f / l;
      T* orow = reinterpret_cast<T*>(p.out) + static_cast<int64_t>(s0 + tok) * p.o_st +
                static_cast<int64_t>(kvh * G + gh) * p.o_sh;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tc::ld32(trow + TS::kO + 32 * c, o);
        tc::wait_ld();
        if (valid) {
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8)
            *reinterpret_cast<uint4*>(orow + 32 * c + 8 * q8) =
                make_uint4(pack2<T>(o[8 * q8] * inv, o[8 * q8 + 1] * inv),
                           pack2<T>(o[8 * q8 + 2] * inv, o[8 * q8 + 3] * inv),
                           pack2<T>(o[8 * q8 + 4] * inv, o[8 * q8 + 5] * inv),
                           pack2<T>(o[8 * q8 + 6] * inv, o[8 * q8 + 7] * inv));
        }
      }
    }
  }
  if (!ok && lane == 0) atomicOr(p.err, kErrWaitTimeout);

  // ---- teardown: every MMA has completed before the columns are freed
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    if (n_tiles > 0) wait_warp(fin, 0);
    tc::fence_after_sync();
    tc::dealloc(tmem, TS::kTmemCols);
  }
}

template <typename T, int D>
int launch_tc_inst(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p, int grid_x,
                   cudaStream_t stream) {
  using TS = TcShape<D>;
  auto kernel = paged_prefill_tc_kernel<T, D>;
  static std::atomic<int> configured_for[64];
  cudaError_t e =
      static_cast<cudaError_t>(raise_smem_limit(configured_for, reinterpret_cast<const void*>(kernel), TS::kSmem));
  if (e != cudaSuccess) return e;
  kernel<<<dim3(grid_x, p.num_kv_heads), kTcThreads, TS::kSmem, stream>>>(kmap, vmap, p);
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace

int prefill_tc_grid_x(int64_t num_tokens, int64_t num_seqs, int group) {
  // an upper bound on the row tiles: sum_b ceil(n_b G / 128) <= ceil(T G / 128) + B
  return static_cast<int>((num_tokens * group + kTcRows - 1) / kTcRows + num_seqs);
}

int launch_prefill_tc(int dtype, int head_dim, const CUtensorMap& kmap, const CUtensorMap& vmap,
                      const PrefillParams& p, int grid_x, cudaStream_t stream) {
  if (grid_x <= 0) return cudaSuccess;
  const bool bf16 = dtype == 2;  // wllm_dtype codes: 1 f16, 2 bf16
  switch (head_dim) {
    case 64:
      return bf16 ? launch_tc_inst<__nv_bfloat16, 64>(kmap, vmap, p, grid_x, stream)
                  : launch_tc_inst<__half, 64>(kmap, vmap, p, grid_x, stream);
    case 128:
      return bf16 ? launch_tc_inst<__nv_bfloat16, 128>(kmap, vmap, p, grid_x, stream)
                  : launch_tc_inst<__half, 128>(kmap, vmap, p, grid_x, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace wllm
