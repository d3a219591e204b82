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
// One CTA (one per SM) owns 256 query rows of one sequence and one kv head,
// as two 128-row tiles -- row r of the sequence's chunk is (token r / G, query
// head r % G of the kv head's group), so the G heads of a group and both tiles
// share every staged K/V byte.  CTAs are launched longest context first (the
// kv heads of a row block together), so that the short ones fill the end of
// the launch.  A CTA walks the rows' context in 128-token kv
// tiles.  Tensor memory holds, per Q tile, the scores S (128 columns, fp32),
// over which the softmax writes the weights P (16-bit, two per column), and the
// output O (head_dim columns).  Ten warps:
//
//   warp 0 (producer): reads the block table and stages each kv tile's K and
//     then its V (16-row TMA boxes, 128-byte swizzle) into a ring of slots laid
//     out [head_dim / 64][128 tokens][128 bytes], so that the 8-row groups of a
//     slot sit 1024 bytes apart, as the MMA descriptors require; rows of the
//     last kv tile past the context are zeroed once their copy has landed;
//   warp 1 (MMA): one thread issues, for each Q tile x, S_x = Q_x K^T (M = 128,
//     N = 128, K = 16 per instruction; Q and K K-major, from shared memory) and
//     O_x += P_x V (M = 128, N = head_dim; P read from tensor memory, V
//     MN-major straight from its slot).  S_x of the next kv tile is issued once
//     O_x += P_x V has completed (it overwrites P_x), so while one Q tile's
//     softmax runs the tensor core works on the other tile.  It takes the
//     products of each kind in order but issues whichever is ready first.
//     Each group of MMAs completes onto an mbarrier (tcgen05.commit), which
//     also hands a slot back to the producer once both tiles are done with it;
//   warps 2-5 and 6-9 (softmax of Q tile 0 and 1): thread r owns row r of its
//     tile (TMEM lane r): it loads its row of Q into shared memory once, then
//     per kv tile reads its 128 scores from TMEM, applies the causal mask and
//     updates a running maximum that is only moved when a scaled score exceeds
//     it by more than 8 in the log2 domain (so weights stay below 2^8; O is
//     rescaled in TMEM only on such a move -- O is at rest then, its last
//     product having completed before these scores were computed), rounds the
//     weights exp2(scale * s - m) (one FFMA and one SFU exp2 each) to the input
//     type, stores them over the scores, and adds the ROUNDED weights to the
//     running sum: numerator and denominator then use the same weights, so a
//     dominant token whose weight is not exactly 1 (the maximum being stale)
//     adds no rounding error of its own.  At the end it divides O by the
//     running sum and stores the row.
//
// Every wait is bounded; on a timeout the CTA records the error, waits
// (bounded) for its copies and MMAs in flight, frees its TMEM and returns.
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace wllm {

namespace {

constexpr int kTcTileRows = 128;                      // rows of one Q tile (M = 128)
constexpr int kTcTiles = 2;                           // Q tiles per CTA
constexpr int kTcRows = kTcTileRows * kTcTiles;       // query rows per CTA
constexpr int kTcKv = 128;                            // kv tokens per kv tile
constexpr int kTcThreads = (2 + 4 * kTcTiles) * 32;   // producer, MMA, four softmax warps per Q tile
constexpr float kTcRescale = 8.f;                     // the running maximum moves by more than 8 (log2) only
constexpr int kTcSortSeqs = 64;                       // batches of up to this many sequences: longest first

template <int D>
struct TcShape {
  static constexpr int kChunks = D / 64;                     // 128-byte chunks of a 16-bit row
  static constexpr int kQTileBytes = kTcTileRows * D * 2;    // [chunk][128 rows][128 B]
  static constexpr int kSlotBytes = kTcKv * D * 2;           // [chunk][128 tokens][128 B]
  static constexpr int kChunkStride = kTcKv * 128;           // bytes between the chunks of a slot
  static constexpr int kBarBytes = 512;
  static constexpr int kFixed = 1024 + kTcTiles * kQTileBytes + kBarBytes;
  static constexpr int kSlotsRaw = (232448 - kFixed) / kSlotBytes;  // 227 KB of dynamic shared memory
  static constexpr int kSlots = kSlotsRaw > 16 ? 16 : kSlotsRaw;
  static constexpr int kSmem = kFixed + kSlots * kSlotBytes;
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns of Q tile x start at x * kTileCols: scores S (P over its
  // first 64 columns), output O
  static constexpr int kTileCols = 256;
  static constexpr int kS = 0, kO = 128;
};
// One CTA per SM, so the 512 TMEM columns are always free to allocate.
static_assert(2 * (TcShape<64>::kSmem + 1024) > 233472 && 2 * (TcShape<128>::kSmem + 1024) > 233472,
              "a second resident CTA would contend for TMEM");
static_assert(TcShape<128>::kSlots >= 5 && TcShape<64>::kSlots >= 5, "at least two kv tiles in flight");

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

// acc + lo + hi for the two 16-bit values of a pair, each added by one
// mixed-precision add (the 16-bit operand widened exactly, fp32 result).
template <typename T>
__device__ __forceinline__ float add_pair(float acc, uint32_t w);
template <>
__device__ __forceinline__ float add_pair<__nv_bfloat16>(float acc, uint32_t w) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %0, hi, %0;\n\t}"
      : "+f"(acc)
      : "r"(w));
  return acc;
}
template <>
__device__ __forceinline__ float add_pair<__half>(float acc, uint32_t w) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %0, hi, %0;\n\t}"
      : "+f"(acc)
      : "r"(w));
  return acc;
}

// max(a, b, c) in one three-input max.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                            const PrefillParams p) {
  using TS = TcShape<D>;
  constexpr int R = TS::kSlots;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;                              // [2][Q tile]
  uint8_t* ring = q_s + kTcTiles * TS::kQTileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + R * TS::kSlotBytes);
  uint64_t* empty = full + R;
  uint64_t* sfull = empty + R;     // [tile] S written (MMA -> softmax)
  uint64_t* pfull = sfull + 2;     // [tile] P written, O rescaled (softmax -> MMA)
  uint64_t* pvdone = pfull + 2;    // [tile] the PV product done (MMA -> MMA, softmax)
  uint64_t* vzero = pvdone + 2;    // the last kv tile's V rows past the context zeroed (producer -> MMA)
  uint64_t* qfull = vzero + 1;     // Q written (softmax -> MMA)
  uint64_t* fin = qfull + 1;       // every MMA of the CTA done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(fin + 1);
  int* info = reinterpret_cast<int*>(tslot + 1);  // [0] sequence (-1: none), [1] its row block

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  // CTA i works on kv head i % Hkv of row block i / Hkv: the kv heads of a
  // row block are launched together
  const int kvh = static_cast<int>(blockIdx.x % p.num_kv_heads);
  const int tgt_block = static_cast<int>(blockIdx.x / p.num_kv_heads);

  // ---- which (sequence, row block) this CTA owns: sequence b owns
  // ceil(n_b * G / 256) consecutive row blocks.  With up to kTcSortSeqs
  // sequences they are taken longest context first (the block scheduler
  // starts CTAs in launch order, so the longest CTAs start first and the
  // short ones fill the end); within a sequence its last rows (the longest
  // context) come first.
  if (warp == 0) {
    int seq = -1, tile = 0, base = 0;
    if (p.num_seqs <= kTcSortSeqs) {
      // lane l holds sequences l and l + 32: length (the sort key) and row blocks
      int key[2], nb[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = lane + 32 * h;
        key[h] = -1;
        nb[h] = 0;
        if (b < p.num_seqs) {
          int n = p.query_start_loc[b + 1] - p.query_start_loc[b];
          n = n < 0 ? 0 : n;
          nb[h] = static_cast<int>((static_cast<int64_t>(n) * G + kTcRows - 1) / kTcRows);
          key[h] = p.context_lens[b];
        }
      }
      // start of each of this lane's sequences in the sorted order (ties in sequence order)
      int start[2] = {0, 0};
      for (int bb = 0; bb < p.num_seqs; ++bb) {
        const int kb = __shfl_sync(kFullMask, bb < 32 ? key[0] : key[1], bb & 31);
        const int nbb = __shfl_sync(kFullMask, bb < 32 ? nb[0] : nb[1], bb & 31);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int b = lane + 32 * h;
          if (kb > key[h] || (kb == key[h] && bb < b)) start[h] += nbb;
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = lane + 32 * h;
        const bool hit = b < p.num_seqs && tgt_block >= start[h] && tgt_block < start[h] + nb[h];
        const unsigned m = __ballot_sync(kFullMask, hit);
        if (m != 0u) {
          const int src = __ffs(m) - 1;
          seq = src + 32 * h;
          tile = __shfl_sync(kFullMask, nb[h] - 1 - (tgt_block - start[h]), src);
        }
      }
    }
    for (int b0 = 0; b0 < p.num_seqs && seq < 0 && p.num_seqs > kTcSortSeqs; b0 += 32) {
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
      const int tgt = tgt_block - base;
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
      for (int x = 0; x < kTcTiles; ++x) {
        mbar_init(smem_u32(sfull + x), 1);
        mbar_init(smem_u32(pfull + x), 4);
        mbar_init(smem_u32(pvdone + x), 1);
      }
      mbar_init(smem_u32(vzero), 1);
      mbar_init(smem_u32(qfull), 4 * kTcTiles);
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

  // ---- the block's rows and the context they see (uniform over the CTA)
  const int b = info[0];
  int n_rows = 0, row0 = 0, pos0 = 0, s0 = 0;
  int nt[kTcTiles] = {0, 0};  // kv tiles each Q tile needs
  int kv_end = 0;             // tokens any row of the block sees
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
      pos0 = L - n;
#pragma unroll
      for (int x = 0; x < kTcTiles; ++x) {  // (no rows only when n was clamped, error already flagged)
        const int rx = row0 + x * kTcTileRows;
        if (rx < n_rows) {
          const int end_x = pos0 + (min(n_rows, rx + kTcTileRows) - 1) / G + 1;
          nt[x] = (end_x + kTcKv - 1) / kTcKv;
          kv_end = max(kv_end, end_x);
        }
      }
    }
  }
  const int n_tiles = max(nt[0], nt[1]);
  const bool v_tail = n_tiles * kTcKv > kv_end;  // the last kv tile reaches past the context

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
    constexpr int kSub = kTcKv / 16;  // 16-token sub-tiles of a kv tile
    const int32_t* bt_row = p.block_tables + static_cast<int64_t>(b) * p.bt_stride;
    const bool two = p.log2_bs < 4;  // 8-token blocks: two 8-row boxes per 16 tokens
    int issued = 0;                  // slot uses whose copies were issued
    for (int j = 0; ok && j < n_tiles; ++j) {
      // lanes 0..7: the table entries of the tile's 16-token sub-tiles
      int e0 = 0, e1 = 0;
      const int tj = j * kTcKv + 16 * lane;
      if (lane < kSub && tj < kv_end) {
        e0 = bt_row[tj >> p.log2_bs];
        if (two && tj + 8 < kv_end) e1 = bt_row[(tj >> p.log2_bs) + 1];
        if (e0 < 0 || e0 >= p.num_blocks || e1 < 0 || e1 >= p.num_blocks) {
          atomicOr(p.err, kErrBlock);
          e0 = (e0 < 0 || e0 >= p.num_blocks) ? 0 : e0;
          e1 = (e1 < 0 || e1 >= p.num_blocks) ? 0 : e1;
        }
      }
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {  // K, then V
        const int c = 2 * j + half, s = c % R;
        if (!wait_warp(empty + s, ((c / R) & 1) ^ 1)) {
          ok = false;
          break;
        }
        const CUtensorMap* map = half ? &vmap : &kmap;
        const uint32_t slot = smem_u32(ring + s * TS::kSlotBytes);
        const uint32_t bar = smem_u32(full + s);
        // lane jj < kSub issues sub-tile jj's boxes after lane 0 set the byte count
        const int t = j * kTcKv + 16 * lane;
        const bool live = lane < kSub && t < kv_end;
        const uint32_t my_bytes = live ? ((two && !(t + 8 < kv_end)) ? 8u : 16u) * 128u * TS::kChunks : 0u;
        uint32_t bytes = my_bytes;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) bytes += __shfl_xor_sync(kFullMask, bytes, off);
        if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
        __syncwarp();
        if (live) {
#pragma unroll
          for (int cb = 0; cb < TS::kChunks; ++cb) {
            const uint32_t dst = slot + cb * TS::kChunkStride + lane * 2048;
            if (!two) {
              tma_load_3d(dst, map, bar, cb * 64, kvh * p.block_size + (t & (p.block_size - 1)), e0);
            } else {
              tma_load_3d(dst, map, bar, cb * 64, kvh * p.block_size, e0);
              if (t + 8 < kv_end) tma_load_3d(dst + 1024, map, bar, cb * 64, kvh * p.block_size, e1);
            }
          }
        }
        ++issued;
        if (half == 1 && j == n_tiles - 1 && v_tail) {
          // V rows at or past kv_end were never staged (or hold slots past the
          // sequence's end): once the copy has landed, zero them, since a zero
          // weight does not cancel a NaN
          if (!wait_warp(full + s, (c / R) & 1)) {
            ok = false;
            break;
          }
          const int r0 = kv_end - j * kTcKv;
          uint8_t* vs = ring + s * TS::kSlotBytes;
          for (int idx = lane; idx < (kTcKv - r0) * TS::kChunks * 8; idx += 32) {
            const int row = r0 + idx / (TS::kChunks * 8);
            const int rem = idx - (idx / (TS::kChunks * 8)) * (TS::kChunks * 8);
            *reinterpret_cast<uint4*>(vs + (rem >> 3) * TS::kChunkStride + row * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          tc::fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(vzero));
        }
      }
    }
    // every copy still in flight lands before the CTA may leave
    for (int c = issued - R > 0 ? issued - R : 0; c < issued; ++c)
      if (!wait_warp(full + c % R, (c / R) & 1)) ok = false;
  } else if (warp == 1 && n_tiles > 0) {
    // --------------------------------- MMA ----------------------------------
    if (lane == 0) {
      constexpr uint32_t kIdS = tc::f16_idesc(kBf16, false, false, kTcTileRows, kTcKv);
      constexpr uint32_t kIdO = tc::f16_idesc(kBf16, false, true, kTcTileRows, D);
      const uint32_t q_a = smem_u32(q_s), ring_a = smem_u32(ring);
      // the operations of one kind in order: kv tile by kv tile, Q tile 0 then
      // 1, skipping Q tiles that need fewer kv tiles
      const int m2 = min(nt[0], nt[1]);
      const int total = nt[0] + nt[1];
      auto op_at = [&](int k, int& j, int& x) {
        if (k < 2 * m2) {
          j = k >> 1;
          x = k & 1;
        } else {
          j = m2 + (k - 2 * m2);
          x = nt[0] > nt[1] ? 0 : 1;
        }
      };
      // the last operation of its kind on kv tile j (then the slot can go back)
      auto last_on_tile = [&](int j, int x) { return x == 1 || j >= nt[1]; };
      ok = mbar_wait_bounded(smem_u32(qfull), 0, p.wait_limit_ns);
      int ks = 0, kp = 0;  // next S product, next PV product
      uint64_t t_idle = 0;
      int idle = 0;        // polls since the last issue (the timer is read every 64)
      while (ok && kp < total) {
        bool did = false;
        if (ks < total) {
          int j, x;
          op_at(ks, j, x);
          const int c = 2 * j, s = c % R;
          // S_x(j) overwrites P_x(j-1): O_x += P_x(j-1) V must be done
          if (mbar_test_wait(smem_u32(full + s), (c / R) & 1) &&
              (j == 0 || mbar_test_wait(smem_u32(pvdone + x), (j - 1) & 1))) {
            tc::fence_after_sync();
            const uint64_t qd = tc::sw128_desc(q_a + x * TS::kQTileBytes, 16, 1024);
            const uint64_t kd = tc::sw128_desc(ring_a + s * TS::kSlotBytes, 16, 1024);
            const uint32_t d = tmem + x * TS::kTileCols + TS::kS;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              // descriptor start addresses advance in 16-byte units
              const uint32_t qo = ((kk >> 2) * kTcTileRows * 128 + (kk & 3) * 32) >> 4;
              const uint32_t ko = ((kk >> 2) * TS::kChunkStride + (kk & 3) * 32) >> 4;
              tc::mma_f16(d, qd + qo, kd + ko, kIdS, kk > 0 ? 1u : 0u);
            }
            tc::commit(smem_u32(sfull + x));
            if (last_on_tile(j, x)) tc::commit(smem_u32(empty + s));
            ++ks;
            did = true;
          }
        }
        if (kp < ks) {
          int j, x;
          op_at(kp, j, x);
          const int c = 2 * j + 1, s = c % R;
          if (mbar_test_wait(smem_u32(pfull + x), j & 1) && mbar_test_wait(smem_u32(full + s), (c / R) & 1) &&
              (!(v_tail && j == n_tiles - 1) || mbar_test_wait(smem_u32(vzero), 0))) {
            tc::fence_after_sync();
            const uint64_t vd = tc::sw128_desc(ring_a + s * TS::kSlotBytes, TS::kChunkStride, 1024);
            const uint32_t d = tmem + x * TS::kTileCols + TS::kO;
            const uint32_t pa = tmem + x * TS::kTileCols + TS::kS;  // P: 8 columns per 16 tokens
#pragma unroll
            for (int kk = 0; kk < kTcKv / 16; ++kk)
              tc::mma_f16_ts(d, pa + kk * 8, vd + ((kk * 2048) >> 4), kIdO, (j > 0 || kk > 0) ? 1u : 0u);
            tc::commit(smem_u32(pvdone + x));
            if (last_on_tile(j, x)) tc::commit(smem_u32(empty + s));
            ++kp;
            did = true;
          }
        }
        if (did) {
          idle = 0;
        } else if ((++idle & 63) == 0) {  // a bounded wait: no issue for wait_limit_ns gives up
          const uint64_t now = global_timer_ns();
          if (idle == 64) t_idle = now;
          else if (now - t_idle > p.wait_limit_ns) ok = false;
        }
      }
      tc::commit(smem_u32(fin));  // every MMA issued above, on every path
    }
    __syncwarp();
    ok = __shfl_sync(kFullMask, ok ? 1 : 0, 0) != 0;
  } else if (warp >= 2 && n_tiles > 0) {
    // ------------------------------- softmax --------------------------------
    const int x = (warp - 2) >> 2;           // this warp's Q tile
    const int quarter = warp & 3;            // the TMEM lanes this warp reaches
    const int r = quarter * 32 + lane;       // this thread's row of the tile
    const int rowg = row0 + x * kTcTileRows + r;
    const bool valid = rowg < n_rows;
    const int tok = valid ? rowg / G : 0;
    const int gh = valid ? rowg - tok * G : 0;
    const int pos = valid ? pos0 + tok : 0;  // padding rows see token 0 only (output dropped)
    const uint32_t trow = tmem + x * TS::kTileCols + (static_cast<uint32_t>(quarter * 32) << 16);
    {
      uint8_t* qx = q_s + x * TS::kQTileBytes;
      const T* qrow = reinterpret_cast<const T*>(p.q) + static_cast<int64_t>(s0 + tok) * p.q_st +
                      static_cast<int64_t>(kvh * G + gh) * p.q_sh;
#pragma unroll
      for (int c16 = 0; c16 < D / 8; ++c16) {
        const uint4 v = valid ? *reinterpret_cast<const uint4*>(qrow + c16 * 8) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(qx + (c16 >> 3) * (kTcTileRows * 128) + r * 128 + (((c16 & 7) ^ (r & 7)) << 4)) = v;
      }
      tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(qfull));
    }
    const float sl2 = p.scale_log2;  // positive (host-checked): the largest score scales to the largest
    float m = -INFINITY, l = 0.f;
    const int ntx = x ? nt[1] : nt[0];
    for (int j = 0; j < ntx; ++j) {
      if (!wait_warp(sfull + x, j & 1)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      float v[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tc::ld32(trow + TS::kS + 32 * q, v[q]);
      tc::wait_ld();
      const int t0 = j * kTcKv;
      if (t0 + kTcKv - 1 > pos) {  // the causal edge (and tokens past kv_end, whose K was never staged)
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i) v[q][i] = t0 + 32 * q + i <= pos ? v[q][i] : -INFINITY;
      }
      float mxs[8];  // eight independent maxima of the raw scores: a short dependency chain
#pragma unroll
      for (int k = 0; k < 8; ++k) mxs[k] = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int i = 0; i < 32; i += 2) mxs[(i >> 1) & 7] = max3f(mxs[(i >> 1) & 7], v[q][i], v[q][i + 1]);
      const float mx = sl2 * fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                                   fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
      float alpha = 1.f;
      if (mx > m + kTcRescale) {  // also the first kv tile (m = -inf): token 0 is always seen
        alpha = ex2_approx(m - mx);
        m = mx;
      }
      const float nm = -m;
      float sums[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {  // 64 scores -> 32 packed weights -> one TMEM store
        float w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int q = 2 * hq + (i >> 4), e = 2 * (i & 15);
          const uint32_t pw = pack2<T>(ex2_approx(fmaf(v[q][e], sl2, nm)), ex2_approx(fmaf(v[q][e + 1], sl2, nm)));
          sums[i & 3] = add_pair<T>(sums[i & 3], pw);  // the rounded weights the PV product uses
          w[i] = __uint_as_float(pw);
        }
        tc::st32(trow + TS::kS + 32 * hq, w);
      }
      l = l * alpha + ((sums[0] + sums[1]) + (sums[2] + sums[3]));
      if (j > 0 && __any_sync(kFullMask, alpha != 1.f)) {
        // O is at rest: its last product completed before S_j was issued
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tc::ld32(trow + TS::kO + 32 * c, o);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tc::st32(trow + TS::kO + 32 * c, o);
        }
      }
      tc::wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(pfull + x));
    }
    if (ok && ntx > 0) ok = wait_warp(pvdone + x, (ntx - 1) & 1);  // this tile's last PV product
    if (ok && ntx > 0) {
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
  kernel<<<static_cast<unsigned>(grid_x) * static_cast<unsigned>(p.num_kv_heads), kTcThreads, TS::kSmem, stream>>>(
      kmap, vmap, p);
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace

int prefill_tc_grid_x(int64_t num_tokens, int64_t num_seqs, int group) {
  // an upper bound on the row blocks: sum_b ceil(n_b G / 256) <= ceil(T G / 256) + B
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
