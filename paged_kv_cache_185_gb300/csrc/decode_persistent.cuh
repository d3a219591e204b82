// decode_persistent.cuh -- persistent, warp-specialised paged decode for
// f16/bf16 queries (tensor-core QK^T and PV), sm_103a, over a 16-bit cache or
// (F8 instantiations) an E4M3 cache with per-tensor K/V scales: the same
// schedule and pipeline, 128-token stages of codes widened in registers
// (mma_e4m3.cuh), each consumer warp taking two 16-token sub-chunks.
//
// Work is cut into units (sequence b, kv-head tile z, partition p of P tokens).
// The grid is two CTAs per SM (one for head_dim 256); each CTA loops until the
// units run out.  Six warps per CTA:
//
//   scheduler warp: claims units (CTA i starts with unit i, the rest come
//     from a device-wide atomic counter), decodes them, loads their
//     block-table entries (32 chunks per coalesced load), detects prefix
//     groups, and hands the producer pieces of up to 32 chunks through a
//     small shared-memory queue.  It also counts finished units of split
//     sequences (below).
//   producer warp: for every 64-token stage of a piece waits for a free slot
//     of the CTA's ring, writes the stage record, and issues 3-D TMA tiled
//     copies of the 4 x 16 K rows and 4 x 16 V rows of the kv head (128-byte
//     swizzled); a unit's first stage also carries its query rows (bulk copy).
//   consumer warps (4): consumer j takes 16-token sub-chunk j of each stage:
//     S^T = K Q^T (mma.sync m16n8k16, the GQA heads of the tile on the N
//     side), the online-softmax update and O^T += V^T P^T over the full
//     head_dim, keeping its own running (m, l, O).  A prefix-group unit is
//     instead consumed two member sequences per warp over whole stages.
//
// At the end of a unit the consumers merge their four (m, l, O) in the ring
// slot of the unit's last stage.  A sequence with one partition gets its
// output written there; otherwise the partial goes to the workspace, the
// scheduler warp counts it, and after its own work every warp of the launch
// merges the rows whose sequences are complete (counters, bounded polling).
//
// Unit order: partitions 0 and 1 of every sequence, partition-major (no
// schedule needed, shared prefixes first); then the remaining partitions but
// each sequence's last, sequence-major (prefix sums built by the consumer
// warps at launch start); then the last partitions, longest first.
//
// Every wait is bounded: on timeout the warp records an error bit and leaves.
// The scheduler counters and the merge counters are left at zero by every
// launch.
#pragma once

#include "append_row.cuh"
#include "decode_kernel.cuh"
#include "mma_e4m3.cuh"

namespace wllm {

// fused-step flags of one launch
enum : int { kFuseAppend = 1, kOverlapCombine = 2 };

// Grid-wide "every CTA's KV append is written", in two halves so that only
// the warp that reads the cache waits.  The count of arrivals only grows (64
// bits: it does not wrap) and is never reset: every launch adds exactly
// kGridWeight in total, CTA i of g adding
// floor(kGridWeight (i+1) / g) - floor(kGridWeight i / g) (at least 1), so the
// count is a multiple of kGridWeight between launches whatever their grid
// sizes, and a launch's barrier opens at the next multiple.  A CTA reads its
// target (a relaxed load: only the value matters) before it arrives, so the
// count cannot reach the target without it.  Arrival is one release
// reduction by one thread, after the CTA's rows are written and ordered
// before it; the wait polls with acquire loads.  The launch is cooperative,
// so every CTA is resident and the wait ends; it still gives up after
// limit_ns.
constexpr unsigned long long kGridWeight = 1ull << 20;  // > any grid size

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long grid_target(const int* ctrl) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctrl + kGridCountOffset));
  return (v / kGridWeight + 1) * kGridWeight;
}

// one thread per CTA
__device__ __forceinline__ void grid_arrive(int* ctrl) {
  const unsigned long long g = gridDim.x, i = blockIdx.x;
  const unsigned long long w = kGridWeight * (i + 1) / g - kGridWeight * i / g;
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(ctrl + kGridCountOffset), "l"(w) : "memory");
}

__device__ __forceinline__ bool grid_wait(int* ctrl, unsigned long long target, uint64_t limit_ns) {
  const unsigned long long* c = reinterpret_cast<const unsigned long long*>(ctrl + kGridCountOffset);
  if (ld_acquire_u64(c) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_u64(c) < target)
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

struct StageMeta {
  int b, p, t0, tok_end;
  int n_parts, h0, nh, flags;
  int z, nsub, group, pad1;
};
enum : int { kFirst = 1, kLast = 2, kEmptySeq = 4, kStop = 8, kGroup = 16 };

// Consecutive sequences whose tables name the same physical blocks for a whole
// partition (a shared prompt prefix) are processed as one unit of up to
// kMaxGroup sequences: the K/V bytes are read once for all of them.
constexpr int kMaxGroup = 8;

// Unit order.  Phase A: partitions below kPhaseAParts, decoded without a
// schedule: partition 0 of the sequences at multiples of kMaxGroup (the
// possible leaders of prefix groups, so a shared prompt prefix is handed out
// first), then partition 1 of every sequence, then partition 0 of the rest
// (units a group leader may cover: claimed while earlier work runs, so no CTA
// starts the launch skipping covered units).  Phase B: the later
// partitions except each sequence's last, sequence-major (prefix sums).
// Phase C: each sequence's last partition when it lies beyond phase A,
// longest first (32 length buckets, ties in sequence order), so the units
// handed out last are the shortest.
constexpr int kPhaseAParts = 2;
constexpr int kOrderKeys = 36;  // phase-C length buckets 1..32 (0: no phase-C unit), padded

// 16-token sub-chunks per 16-bit stage (64 tokens); the scheduler's work
// estimates count in these stages.  An fp8 stage holds twice as many
// sub-chunks in the same bytes (PShape::kSub).
constexpr int kSub = 4;

// One unit of work: query heads h0 .. h0+nh-1 (kv head kvh, head tile z) of
// sequence b over tokens [tb, te) of partition `part`.
struct UnitInfo {
  int b, part, z, n_parts, tb, te, n_chunks, kvh, h0, nh;
  int group;  // sequences b .. b+group-1 share this partition (1: no sharing); 0: covered by a leader
};

// A piece of a unit handed from the scheduler warp to the producer warp: the
// block-table entries of up to kPieceChunks 16-token chunks starting at chunk
// c0 of the unit (two entries per chunk when blocks hold 8 tokens).
constexpr int kPieceChunks = 32;
constexpr int kQueue = 4;  // pieces in flight between scheduler and producer
// The scheduler claims another unit only when at most this much work (in
// stage equivalents) waits in its queue: little when the launch has few units
// per CTA (the finish balances better), more when it has many (a claim and
// its decode take a few microseconds of dependent round trips, which a short
// unit does not cover).  Measured on GB300 against one bound of 8 for all:
// TinyLlama-shaped step 33.7 -> 32.1 us, Qwen2.5 prefix 176.8 -> 174.4 us,
// its fp8 step 128.7 -> 126.1 us, long-context step unchanged.
constexpr int kLookaheadFew = 4, kLookaheadMany = 12;
enum : int { kPieceFirst = 1, kPieceLast = 2, kPieceStop = 4 };
struct Piece {
  UnitInfo u;
  int c0, flags, pad0, pad1, pad2;
  int e[2 * kPieceChunks];
};
static_assert(sizeof(Piece) % 16 == 0, "pieces stay 16-byte aligned");

// A finished unit of split sequences, handed from the consumers to the
// scheduler warp, which counts it: sequences b .. b+members-1 (a prefix group
// when members > 1; then only the split ones among them are counted), head
// tile z.  b < 0: the consumers have stopped.
struct DoneInfo {
  int b, z, members, pad;
};
constexpr int kDoneSlots = 4;

// F8: the KV cache holds E4M3 codes (one byte per element); T is the query
// and output type.
template <typename T, int D, int NT, bool F8 = false>
struct PShape {
  static constexpr int kConsumers = 4;
  static constexpr int kThreads = (kConsumers + 2) * 32;  // consumers, producer, scheduler
  static constexpr int kHeadTile = 8 * NT;
  using KT = typename std::conditional<F8, uint8_t, T>::type;  // cache element
  static constexpr int kKV = Geom<KT, D>::kTileBytes;  // one 16-row K (or V) sub-tile
  // sub-chunks per stage: 64 tokens, or 128 over an fp8 cache, where every
  // consumer warp takes two sub-chunks of a stage as one softmax step (tried
  // for 16-bit head_dim 64 too: no faster, the TinyLlama-shaped batch is bound
  // by start-up and tail, not by the consumers' issue rate)
  static constexpr int kSub = F8 ? 8 : 4;
  static constexpr int kQBytes = kHeadTile * D * static_cast<int>(sizeof(T));
  static constexpr int kStageBytes = ((2 * kSub * kKV + kQBytes) + 1023) / 1024 * 1024;
  // the unit merge writes each consumer's (m, l, O) into the ring slot of
  // the unit's last stage once every consumer is done reading it
  static constexpr int kRedBytes = (kConsumers * kHeadTile * (D + 2) * 4 + 127) / 128 * 128;
  static_assert(kRedBytes <= kStageBytes, "unit merge must fit in one ring slot");
  // Consumer warps bound the rate of one CTA (each 16-token sub-chunk is a
  // ~1k-cycle dependency chain), so the target is two CTAs per SM (eight
  // consumer warps); a third would need under 100 registers a thread (each
  // SM sub-partition holds 16K registers and would host five of the 18
  // warps).  The ring gets what is left of the
  // per-CTA share of shared memory (228 KB per SM, 1 KB of it reserved per
  // CTA) after the alignment pad, the barriers and stage records (64 B per
  // stage), the piece queue and the prefix-sum array (up to
  // kPersistentMaxSeqs + 1 ints).
  static constexpr int kCtasPerSm = D <= 128 ? 2 : 1;
  // registers per thread that keep kCtasPerSm CTAs resident (64K per SM, a
  // multiple of 8 per thread)
  static constexpr int kMaxRegsRaw = 65536 / (kCtasPerSm * kThreads) / 8 * 8;
  static constexpr int kMaxRegs = kMaxRegsRaw > 255 ? 255 : kMaxRegsRaw;
  // prefix sums; phase-C bucket starts, order and keys
  static constexpr int kSeqBytes = ((kPersistentMaxSeqs + 1) * 4 + 15) / 16 * 16 + kOrderKeys * 4 +
                                   (kPersistentMaxSeqs * 3 + 15) / 16 * 16;
  static constexpr int kSmemPerCta = 233472 / kCtasPerSm - 1024;
  static constexpr int kQueueBytes =
      kQueue * (static_cast<int>(sizeof(Piece)) + 16) + kDoneSlots * (static_cast<int>(sizeof(DoneInfo)) + 16) + 16;
  static constexpr int kStagesRaw = (kSmemPerCta - 1024 - 64 - 16 - kSeqBytes - kQueueBytes) / (kStageBytes + 64);
  static constexpr int kStages = kStagesRaw > 16 ? 16 : (kStagesRaw < 2 ? 2 : kStagesRaw);
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kBarBytes = (2 * kStages + 2 + 2 * kQueue + 2 * kDoneSlots) * 8;
  static constexpr int kMetaBytes = kStages * static_cast<int>(sizeof(StageMeta));
  static constexpr int kDoneBytes = kDoneSlots * static_cast<int>(sizeof(DoneInfo));
  static constexpr int kFixedSmem =
      1024 + kRingBytes + kBarBytes + kMetaBytes + kQueue * static_cast<int>(sizeof(Piece)) + kDoneBytes + 64;
};

// Query fragments of a unit from the stage's query rows (row stride D).
template <typename T, int D, int NT>
__device__ __forceinline__ void load_q_smem(MmaState<T, D, NT>& st, const uint8_t* qtile, int nh, int lane) {
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
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.o[mt][nt][e] = 0.f;
  }
}

// Rendezvous of the four consumer warps on an mbarrier (count 4, one arrival
// per warp), bounded like every other wait.  `phase` counts the uses.
__device__ __forceinline__ bool consumer_sync(uint32_t bar, int& phase, uint64_t limit_ns, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = mbar_wait_bounded(bar, phase & 1, limit_ns);
  ++phase;
  return __all_sync(kFullMask, ok);
}

// Merge the partitions of R query rows at once (one warp): for each row
// (b, h), weights exp2(m_p - M) with M the largest m_p, fp32 sums,
// round-to-nearest into `out`.  Lane l owns dims [l*D/32, (l+1)*D/32), so a
// partial is one or two vector loads per lane.  Two memory round trips cover
// all R rows when each has at most kBatch partitions: the context lengths,
// then every (m, l) pair and partial at once.  rows[r] < 0 skips slot r; rows
// with one partition were written by the decode itself.
// The same with the rows' partition counts given (n[r] < 2 skips row r).
template <typename T, int D, int R>
__device__ __forceinline__ void combine_rows_np(const DecodeParams& p, const int (&rows)[R], const int (&n)[R],
                                                int lane) {
  constexpr int V = D / 32;
  constexpr int kBatch = 32 / V;
  auto load_part = [&](const float* src, float* dst) {
    if constexpr (V >= 4) {
#pragma unroll
      for (int i = 0; i < V; i += 4) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(src + i));
        dst[i] = x.x;
        dst[i + 1] = x.y;
        dst[i + 2] = x.z;
        dst[i + 3] = x.w;
      }
    } else {
      const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
      dst[0] = x.x;
      dst[1] = x.y;
    }
  };
  float2 v[R];
  float o[R][kBatch][V];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (n[r] < 2) continue;
    const int64_t base = static_cast<int64_t>(rows[r]) * p.max_parts;
    v[r] = lane < min(32, n[r]) ? __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + base + lane)
                                : make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (j < n[r]) load_part(p.ws_o + (base + j) * D + lane * V, o[r][j]);
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (n[r] < 2) continue;
    const int64_t base = static_cast<int64_t>(rows[r]) * p.max_parts;
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    float M = -INFINITY, den = 0.f;
    for (int p0 = 0; p0 < n[r]; p0 += 32) {  // groups of 32 partitions, one (m, l) per lane
      const int cnt = min(32, n[r] - p0);
      float2 w = v[r];
      if (p0 > 0) w = lane < cnt ? __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + base + p0 + lane)
                                 : make_float2(-INFINITY, 0.f);
      float mg = w.x;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mg = fmaxf(mg, __shfl_xor_sync(kFullMask, mg, off));
      const float Mn = fmaxf(M, mg);
      const float rescale = exp2f(M - Mn);  // 0 for the first group
      M = Mn;
      den *= rescale;
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] *= rescale;
      const float f = lane < cnt ? exp2f(w.x - M) : 0.f;
      float dsum = f * w.y;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dsum += __shfl_xor_sync(kFullMask, dsum, off);
      den += dsum;
      for (int j0 = 0; j0 < cnt; j0 += kBatch) {
        if (p0 + j0 > 0) {
#pragma unroll
          for (int j = 0; j < kBatch; ++j)
            if (j0 + j < cnt) load_part(p.ws_o + (base + p0 + j0 + j) * D + lane * V, o[r][j]);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const float fp = __shfl_sync(kFullMask, f, (j0 + j) & 31);
          if (j0 + j < cnt) {
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = fmaf(fp, o[r][j][i], acc[i]);
          }
        }
      }
    }
    const float inv = 1.f / den;
    const int b = rows[r] / p.num_q_heads;
    const int h = rows[r] - b * p.num_q_heads;
    T* orow = reinterpret_cast<T*>(p.out) + b * p.o_sb + static_cast<int64_t>(h) * p.o_sh + lane * V;
#pragma unroll
    for (int i = 0; i < V; ++i) orow[i] = from_f32<T>(acc[i] * inv);
  }
}

// One warp's share of a split row's merge: partitions [p0, p1) of query row
// `row` folded into a running maximum M (log2 domain), a sum `den` of the
// partitions' sums scaled to M, and the correspondingly scaled sum of their
// unnormalised outputs (lane: head_dim elements lane*V .. lane*V+V-1).
// Partials are read through L2 (other CTAs wrote them).
template <int D>
__device__ __forceinline__ void merge_part_range(const DecodeParams& p, int row, int p0, int p1, int lane, float& M,
                                                 float& den, float (&acc)[D / 32]) {
  constexpr int V = D / 32;
  constexpr int kBatch = 32 / V;  // partitions whose outputs are loaded together
  M = -INFINITY;
  den = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  const int64_t base = static_cast<int64_t>(row) * p.max_parts;
  for (int c0 = p0; c0 < p1; c0 += 32) {  // one (m, l) per lane
    const int cnt = min(32, p1 - c0);
    const float2 w = lane < cnt ? __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + base + c0 + lane)
                                : make_float2(-INFINITY, 0.f);
    float mg = w.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mg = fmaxf(mg, __shfl_xor_sync(kFullMask, mg, off));
    const float Mn = fmaxf(M, mg);
    const float rescale = M == -INFINITY ? 0.f : exp2f(M - Mn);
    M = Mn;
    den *= rescale;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] *= rescale;
    const float f = lane < cnt ? exp2f(w.x - M) : 0.f;
    float dsum = f * w.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dsum += __shfl_xor_sync(kFullMask, dsum, off);
    den += dsum;
    for (int j0 = 0; j0 < cnt; j0 += kBatch) {
      float o[kBatch][V];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (j0 + j < cnt) {
          const float* src = p.ws_o + (base + c0 + j0 + j) * D + lane * V;
          if constexpr (V >= 4) {
#pragma unroll
            for (int i = 0; i < V; i += 4) {
              const float4 x = __ldcg(reinterpret_cast<const float4*>(src + i));
              o[j][i] = x.x;
              o[j][i + 1] = x.y;
              o[j][i + 2] = x.z;
              o[j][i + 3] = x.w;
            }
          } else {
            const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
            o[j][0] = x.x;
            o[j][1] = x.y;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const float fp = __shfl_sync(kFullMask, f, (j0 + j) & 31);
        if (j0 + j < cnt) {
#pragma unroll
          for (int i = 0; i < V; ++i) acc[i] = fmaf(fp, o[j][i], acc[i]);
        }
      }
    }
  }
}

template <typename T, int D, int R>
__device__ __forceinline__ void combine_rows(const DecodeParams& p, const int (&rows)[R], int lane) {
  const int l_max = p.max_blocks * p.block_size;
  int n[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    int L = rows[r] >= 0 ? p.context_lens[rows[r] / p.num_q_heads] : 0;
    L = L < 0 ? 0 : (L > l_max ? l_max : L);
    n[r] = (rows[r] < 0 || L == 0) ? 1 : (L + p.part_tokens - 1) / p.part_tokens;
  }
  combine_rows_np<T, D, R>(p, rows, n, lane);
}

// NS consecutive 16-token sub-chunks (sub-chunk j's K at k_base + j * kKV,
// its V at v_base + j * kKV; the first nsub hold tokens) for the NT column
// tiles of `st`: NS x NT independent S^T tiles in flight, one online-softmax
// update per column tile over all NS sub-chunks, then PV over the full
// head_dim.  Used by prefix-group units, where each column tile is one
// member sequence.  The first sub-chunk must hold at least one token.
template <typename T, int D, int NT, int NS>
__device__ __forceinline__ void mma_multi(MmaState<T, D, NT>& st, uint32_t k_base, uint32_t v_base, int t0,
                                          int tok_end, int nsub, float scale_log2, int lane) {
  constexpr int kKV = Geom<T, D>::kTileBytes;
  float s[NS][NT][4];
#pragma unroll
  for (int j = 0; j < NS; ++j)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[j][nt][i] = 0.f;
  const int a_row = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int a_chunk = lane >> 4;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
    for (int j = 0; j < NS; ++j) {
      if (j < nsub) {
        uint32_t a[4];
        ldsm_x4(k_base + j * kKV + tile_offset(a_row, 2 * ks + a_chunk), a);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) Mma<T>::run(s[j][nt], a, st.qb[nt][ks]);
      }
    }
  }
  uint32_t pb[NS][NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < NS; ++j) {
      const int tok_a = t0 + j * kChunk + (lane >> 2);
      const bool va = j < nsub && tok_a < tok_end, vb = j < nsub && tok_a + 8 < tok_end;
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
    const float alpha0 = exp2f(st.m[nt][0] - mn0), alpha1 = exp2f(st.m[nt][1] - mn1);
    st.m[nt][0] = mn0;
    st.m[nt][1] = mn1;
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int j = 0; j < NS; ++j) {
      const float p0 = exp2f(s[j][nt][0] - mn0), p1 = exp2f(s[j][nt][1] - mn1);
      const float p2 = exp2f(s[j][nt][2] - mn0), p3 = exp2f(s[j][nt][3] - mn1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      pb[j][nt][0] = movmatrix_trans(Mma<T>::pack(p0, p1));
      pb[j][nt][1] = movmatrix_trans(Mma<T>::pack(p2, p3));
    }
    st.l[nt][0] = st.l[nt][0] * alpha0 + l0;
    st.l[nt][1] = st.l[nt][1] * alpha1 + l1;
    if (__any_sync(kFullMask, (alpha0 != 1.f) || (alpha1 != 1.f))) {
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        st.o[mt][nt][0] *= alpha0;
        st.o[mt][nt][1] *= alpha1;
        st.o[mt][nt][2] *= alpha0;
        st.o[mt][nt][3] *= alpha1;
      }
    }
  }
  const int v_row = (lane & 7) + ((lane >> 4) << 3);
  const int v_chunk = (lane >> 3) & 1;
#pragma unroll
  for (int j = 0; j < NS; ++j) {
    if (j < nsub) {
      const int tj = t0 + j * kChunk;
      const bool tail = tj + kChunk > tok_end;
      const int tk = tj + 2 * (lane & 3);
      const uint32_t keep_lo = (tk < tok_end ? 0x0000ffffu : 0u) | (tk + 1 < tok_end ? 0xffff0000u : 0u);
      const uint32_t keep_hi = (tk + 8 < tok_end ? 0x0000ffffu : 0u) | (tk + 9 < tok_end ? 0xffff0000u : 0u);
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        uint32_t a[4];
        ldsm_x4_trans(v_base + j * kKV + tile_offset(v_row, 2 * mt + v_chunk), a);
        if (tail) {
          a[0] &= keep_lo;
          a[1] &= keep_lo;
          a[2] &= keep_hi;
          a[3] &= keep_hi;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) Mma<T>::run(st.o[mt][nt], a, pb[j][nt]);
      }
    }
  }
}

// Query fragments for a prefix-group unit: column tile nt holds heads
// h0 .. h0+nh-1 of member sequence b0 + nt (zeros past the group's last
// member), read from global memory; the running state starts empty.
template <typename T, int D, int NT>
__device__ __forceinline__ void load_q_members(MmaState<T, D, NT>& st, const DecodeParams& p, int b0,
                                               int n_members, int h0, int nh, int lane) {
  const int hh = lane >> 2;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const bool valid = hh < nh && nt < n_members;
    const T* row = reinterpret_cast<const T*>(p.q) + (valid ? b0 + nt : 0) * p.q_sb +
                   static_cast<int64_t>(h0 + (valid ? hh : 0)) * p.q_sh;
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
      for (int e = 0; e < 4; ++e) st.o[mt][nt][e] = 0.f;
  }
}

// Finish the member sequences b0 .. b0+n_members-1 (column tiles of one warp)
// of a prefix-group unit over partition `part`: each member's output when it
// has one partition, otherwise its partial.
template <typename T, int D, int NT>
__device__ __forceinline__ void finish_members(MmaState<T, D, NT>& st, const DecodeParams& p, int b0, int n_members,
                                               int part, int h0, int nh, int lane) {
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
        const float inv = 1.f / l[j];
        T* r = out + b * p.o_sb + static_cast<int64_t>(h0 + hh + j) * p.o_sh;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const int d = mt * 16 + (lane >> 2);
          r[d] = from_f32<T>(st.o[mt][nt][j] * inv);
          r[d + 8] = from_f32<T>(st.o[mt][nt][2 + j] * inv);
        }
      } else {
        const int64_t slot = static_cast<int64_t>(b * p.num_q_heads + h0 + hh + j) * p.max_parts + part;
        float* wo = p.ws_o + slot * D;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const int d = mt * 16 + (lane >> 2);
          wo[d] = st.o[mt][nt][j];
          wo[d + 8] = st.o[mt][nt][2 + j];
        }
        if ((lane >> 2) == 0) reinterpret_cast<float2*>(p.ws_ml)[slot] = make_float2(st.m[nt][j], l[j]);
      }
    }
  }
}

template <typename T, int D, int NT, bool F8>
__global__ void __launch_bounds__(PShape<T, D, NT, F8>::kThreads) __maxnreg__((PShape<T, D, NT, F8>::kMaxRegs))
    paged_decode_persistent(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                            const DecodeParams p, const AppendParams ap, const int flags) {
  using PS = PShape<T, D, NT, F8>;
  using G = Geom<typename PS::KT, D>;
  using MT = typename std::conditional<F8, __half, T>::type;  // tensor-core operand type
  constexpr int S = PS::kStages;
  constexpr int W = PS::kConsumers;
  constexpr int HT = PS::kHeadTile;
  constexpr int Q = kQueue;
  constexpr bool kGroupOK = NT == 1 && D <= 128;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + PS::kRingBytes);
  uint64_t* empty = full + S;
  uint64_t* cbar = empty + S;                 // consumer rendezvous
  uint64_t* pbar = cbar + 1;                  // prefix sums ready (consumers -> scheduler)
  uint64_t* qfull = pbar + 1;                 // piece queue: scheduler -> producer
  uint64_t* qempty = qfull + kQueue;
  uint64_t* done_full = qempty + kQueue;      // finished split units: consumers -> scheduler
  uint64_t* done_empty = done_full + kDoneSlots;
  StageMeta* meta = reinterpret_cast<StageMeta*>(done_empty + kDoneSlots);
  Piece* pieces = reinterpret_cast<Piece*>(meta + S);
  DoneInfo* done_info = reinterpret_cast<DoneInfo*>(pieces + kQueue);
  int* wsum = reinterpret_cast<int*>(done_info + kDoneSlots);  // 16 ints of scratch
  int* prefix = wsum + 16;                       // [B + 1] units before sequence b
  int* order_cnt = prefix + ((p.num_seqs + 1 + 3) & ~3);                  // [kOrderKeys] bucket starts
  uint16_t* order = reinterpret_cast<uint16_t*>(order_cnt + kOrderKeys);  // [B] phase-C sequences
  uint8_t* okey = reinterpret_cast<uint8_t*>(order + p.num_seqs);         // [B] their buckets

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = p.num_seqs;
  const int Z = p.num_kv_heads * p.num_head_tiles;
  const int l_max = p.max_blocks * p.block_size;
  // a separate merge kernel launched behind this one may be scheduled now: its
  // CTAs take the SMs as this grid's CTAs leave, and wait for the whole grid
  asm volatile("griddepcontrol.launch_dependents;");

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), W);
    }
    mbar_init(smem_u32(cbar), W);
    mbar_init(smem_u32(pbar), 1);
    for (int i = 0; i < Q; ++i) {
      mbar_init(smem_u32(qfull + i), 1);
      mbar_init(smem_u32(qempty + i), 1);
    }
    for (int i = 0; i < kDoneSlots; ++i) {
      mbar_init(smem_u32(done_full + i), W);
      mbar_init(smem_u32(done_empty + i), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int BZ = B * Z;  // partition-0 units

  // fused step: the count the arrivals of this launch end at, read before this
  // CTA arrives (only the producer's first lane uses it)
  unsigned long long grid_target_ = 0;
  if ((flags & kFuseAppend) && warp == W && lane == 0) grid_target_ = grid_target(p.err);
  // fused step: this CTA's share of the KV append (consumer and producer
  // warps), made visible to the other CTAs' tensor copies before any of them
  // reads the cache (the producer announces this CTA's rows and waits for
  // every other CTA's, below).  The scheduler warp does not take part: it
  // decodes its first units meanwhile (only tensor copies read the cache).
  if ((flags & kFuseAppend) && warp <= W) {
    const int64_t rows = static_cast<int64_t>(ap.num_tokens) * ap.num_kv_heads;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * (W + 1) + warp; r < rows;
         r += static_cast<int64_t>(gridDim.x) * (W + 1))
      append_row(ap, r, lane);
    asm volatile("fence.proxy.async.global;" ::: "memory");
    // this CTA's rows are written; the producer announces them (grid_arrive)
    asm volatile("bar.sync 2, %0;" ::"r"((W + 1) * 32) : "memory");
  }
  bool failed = false;  // a bounded wait gave up: skip to the end, still meet every barrier

  if (warp == W + 1) {
    // ------------------------------- scheduler -------------------------------
    // Claims units (CTA i starts with unit i; later ones come from the global
    // counter, offset by the grid size), decodes them, loads their block-table
    // entries and hands them to the producer as pieces of at most kPieceChunks
    // chunks through a kQueue-deep queue in shared memory.  Every
    // global-memory round trip of the schedule happens here, off the path
    // between two tensor-copy issues.
    int* sched_next = p.err + kSchedNextOffset;
    int* sched_done = p.err + kSchedDoneOffset;

    // block-table entries of 16-token chunks cbase + lane (two when blocks hold 8 tokens)
    auto load_entries = [&](const UnitInfo& x, int cbase, int& e0, int& e1) {
      e0 = 0;
      e1 = 0;
      const int cc = cbase + lane;
      if (cc < x.n_chunks) {
        const int32_t* bt_row = p.block_tables + static_cast<int64_t>(x.b) * p.bt_stride;
        const int t0 = x.tb + kChunk * cc;
        int x0 = bt_row[t0 >> p.log2_bs], x1 = 0;
        if (p.log2_bs < 4 && t0 + 8 < x.te) x1 = bt_row[(t0 >> p.log2_bs) + 1];
        if (x0 < 0 || x0 >= p.num_blocks || x1 < 0 || x1 >= p.num_blocks) {
          atomicOr(p.err, kErrBlock);
          x0 = (x0 < 0 || x0 >= p.num_blocks) ? 0 : x0;
          x1 = (x1 < 0 || x1 >= p.num_blocks) ? 0 : x1;
        }
        e0 = x0;
        e1 = x1;
      }
    };
    // Sharing of the full partition starting at token tb of sequence b with its
    // neighbours.  Groups are the runs of consecutive sequences whose tables
    // name the same physical blocks for the whole partition, cut at every
    // multiple of kMaxGroup: sequence b leads a group unless b - 1 shares with
    // it and b is not a multiple of kMaxGroup.  Returns 0 for a covered
    // sequence, else the group's size (1: no sharing).  Block lists are
    // compared a warp at a time (up to 64 blocks: two per lane); the rows
    // needed (b - 1 .. the group's end) are loaded in one batch.
    auto prefix_group = [&](int b, int tb) -> int {
      const int nblk = p.part_tokens >> p.log2_bs;
      const int j0 = tb >> p.log2_bs;
      const int span = kMaxGroup - (b % kMaxGroup);  // b .. b+span-1 may form b's group
      auto load_row = [&](int bb, int& v0, int& v1) {  // entries within the table's width only
        v0 = -1;
        v1 = -1;
        if (bb >= 0 && bb < B) {
          const int32_t* r = p.block_tables + static_cast<int64_t>(bb) * p.bt_stride + j0;
          if (lane < nblk && j0 + lane < p.max_blocks) v0 = r[lane];
          if (lane + 32 < nblk && j0 + lane + 32 < p.max_blocks) v1 = r[lane + 32];
        }
      };
      // lane i <= kMaxGroup: whether row b-1+i fills the partition, and the
      // partition's first block in that row (one round trip for both)
      const int bb_l = b - 1 + lane;
      bool cov = false;
      int first = -1;
      if (lane <= kMaxGroup && bb_l >= 0 && bb_l < B) {
        int Lb = p.context_lens[bb_l];
        if (j0 < p.max_blocks) first = p.block_tables[static_cast<int64_t>(bb_l) * p.bt_stride + j0];
        Lb = Lb < 0 ? 0 : (Lb > l_max ? l_max : Lb);
        cov = Lb >= tb + p.part_tokens;
      }
      const unsigned covm = __ballot_sync(kFullMask, cov);
      // rows whose first block differs cannot share the partition: when no
      // neighbour that could join (b-1 as b's leader, b+1 as its first
      // follower) starts with b's block, there is no group and no table is
      // compared
      const int b_first = __shfl_sync(kFullMask, first, 1);
      const unsigned cand = __ballot_sync(kFullMask, cov && first == b_first) & covm;
      const bool lead_cand = b % kMaxGroup != 0 && b > 0 && (cand & 1u);
      const bool next_cand = span >= 2 && ((cand >> 2) & 1u);
      if (!lead_cand && !next_cand) return 1;
      int r0[kMaxGroup + 1], r1[kMaxGroup + 1];  // rows b-1 .. b+kMaxGroup-1
#pragma unroll
      for (int i = 0; i <= kMaxGroup; ++i) {
        if (i == 0 || i <= span) load_row(b - 1 + i, r0[i], r1[i]);
        else r0[i] = r1[i] = -1;
      }
      const int c0 = r0[1], c1 = r1[1];  // sequence b's own blocks
      auto same = [&](int i) {  // row b-1+i names b's blocks and fills the partition
        return ((covm >> i) & 1) && __all_sync(kFullMask, r0[i] == c0 && r1[i] == c1);
      };
      if (b % kMaxGroup != 0 && b > 0 && same(0)) return 0;
      int g = 1;
#pragma unroll
      for (int i = 2; i <= kMaxGroup; ++i) {
        if (g == i - 1 && i <= span && same(i)) g = i;
      }
      return g;
    };
    bool have_prefix = false;
    bool wait_ok = true;
    // Phase-C order, built once by this warp right after the consumers'
    // prefix pass (which also wrote each sequence's bucket): the sequences
    // whose last partition lies past phase A, bucketed by that partition's
    // length (32 buckets over P tokens), most first, ties in sequence order --
    // a stable counting sort, 32 sequences at a time.  order_cnt[0] = their
    // number.
    auto build_order = [&]() {
      for (int i = lane; i < kOrderKeys; i += 32) order_cnt[i] = 0;
      __syncwarp();
      for (int b0 = 0; b0 < B; b0 += 32) {
        const int k = b0 + lane < B ? okey[b0 + lane] : -1;
        const unsigned same = __match_any_sync(kFullMask, k);
        if (k > 0 && lane == __ffs(same) - 1) order_cnt[k] += __popc(same);
        __syncwarp();
      }
      if (lane == 0) {  // bucket k starts after every bucket above it; [0] = total
        int run = 0;
        for (int k = 32; k >= 1; --k) {
          const int c = order_cnt[k];
          order_cnt[k] = run;
          run += c;
        }
        order_cnt[0] = run;
      }
      __syncwarp();
      for (int b0 = 0; b0 < B; b0 += 32) {
        const int k = b0 + lane < B ? okey[b0 + lane] : -1;
        const unsigned same = __match_any_sync(kFullMask, k);
        const int leader = __ffs(same) - 1;
        int base = (lane == leader && k > 0) ? order_cnt[k] : 0;
        base = __shfl_sync(kFullMask, base, leader);
        if (k > 0) order[base + __popc(same & ((1u << lane) - 1u))] = static_cast<uint16_t>(b0 + lane);
        __syncwarp();
        if (lane == leader && k > 0) order_cnt[k] = base + __popc(same);
        __syncwarp();
      }
    };
    // unit u -> (sequence, partition, kv-head tile) and the table entries of
    // its first 32 chunks (two per chunk when blocks hold 8 tokens).  Returns
    // false past the last unit.
    // prefix groups apply to whole partitions of whole blocks, at most 64 of them
    const bool groups_on = kGroupOK && p.prefix_groups && (p.part_tokens & (p.block_size - 1)) == 0 &&
                           (p.part_tokens >> p.log2_bs) <= 64;
    auto decode_unit = [&](int u, UnitInfo& x, int& e0, int& e1) -> bool {
      int L;
      int grp = -1;  // prefix group, when already found
      if (u < kPhaseAParts * BZ) {
        static_assert(kPhaseAParts == 2, "phase A is partitions 0 and 1");
        // sequences in the order 0, 8, 16, ..., 1, 9, 17, ... (prefix groups are
        // cut at multiples of kMaxGroup): units [0, n0 Z) are partition 0 of
        // the first n0 of that order, [n0 Z, n0 Z + BZ) partition 1 of all,
        // the rest partition 0 of the others
        const int n0Z = (B + kMaxGroup - 1) / kMaxGroup * Z;
        int r = u;
        x.part = 0;
        if (u >= n0Z + BZ) {
          r = u - BZ;
        } else if (u >= n0Z) {
          x.part = 1;
          r = u - n0Z;
        }
        const int bi = r / Z;
        int k = 0, base = 0, cnt = (B + kMaxGroup - 1) / kMaxGroup;
        while (k < kMaxGroup - 1 && bi >= base + cnt) {
          base += cnt;
          ++k;
          cnt = (B - k + kMaxGroup - 1) / kMaxGroup;
        }
        x.b = k + kMaxGroup * (bi - base);
        x.z = r - bi * Z;
        int Lraw = p.context_lens[x.b];  // issued together with the table loads below
        const int32_t* bt_row = p.block_tables + static_cast<int64_t>(x.b) * p.bt_stride;
        x.tb = x.part * p.part_tokens;
        const int j0 = (x.tb + kChunk * lane) >> p.log2_bs;
        int r0 = j0 < p.max_blocks ? bt_row[j0] : 0;
        int r1 = (p.log2_bs < 4 && j0 + 1 < p.max_blocks) ? bt_row[j0 + 1] : 0;
        // the launch's first units: the neighbours' lengths and tables load
        // alongside this unit's own (one round trip, not two); the result is
        // used only if the sequence fills the partition
        if (groups_on) grp = prefix_group(x.b, x.tb);
        if (Lraw < 0 || Lraw > l_max) {
          if (lane == 0 && x.part == 0) atomicOr(p.err, kErrLen);
          Lraw = Lraw < 0 ? 0 : l_max;
        }
        L = Lraw;
        if (x.part > 0 && L <= x.tb) {  // the sequence has no such partition: nothing to do
          x.group = 0;
          x.n_chunks = 0;
          return true;
        }
        x.te = min(L, x.tb + p.part_tokens);
        x.n_chunks = L == 0 ? 0 : (x.te - x.tb + kChunk - 1) / kChunk;
        const int t0 = x.tb + kChunk * lane;
        const bool need0 = lane < x.n_chunks, need1 = need0 && p.log2_bs < 4 && t0 + 8 < x.te;
        if ((need0 && (r0 < 0 || r0 >= p.num_blocks)) || (need1 && (r1 < 0 || r1 >= p.num_blocks))) {
          atomicOr(p.err, kErrBlock);
        }
        e0 = (need0 && r0 >= 0 && r0 < p.num_blocks) ? r0 : 0;
        e1 = (need1 && r1 >= 0 && r1 < p.num_blocks) ? r1 : 0;
      } else {
        if (!have_prefix) {
          bool got = true;
          if (lane == 0) got = mbar_wait_bounded(smem_u32(pbar), 0, p.wait_limit_ns);
          wait_ok = __shfl_sync(kFullMask, got ? 1 : 0, 0) != 0;
          have_prefix = true;
          if (!wait_ok) return false;
          build_order();
        }
        const int u2 = u - kPhaseAParts * BZ;
        if (u2 >= prefix[B]) {  // phase C
          const int u3 = u2 - prefix[B];
          if (u3 >= order_cnt[0] * Z) return false;
          const int idx = u3 / Z;
          x.b = order[idx];
          x.z = u3 - idx * Z;
          L = p.context_lens[x.b];
          L = L < 0 ? 0 : (L > l_max ? l_max : L);
          const int np = (L + p.part_tokens - 1) / p.part_tokens;
          x.part = np - 1;
          x.tb = x.part * p.part_tokens;
          x.te = L;
          x.n_chunks = (x.te - x.tb + kChunk - 1) / kChunk;
          load_entries(x, 0, e0, e1);
        } else {
          int lo = 0, hi = B - 1;
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= u2) lo = mid;
            else hi = mid - 1;
          }
          x.b = lo;
          const int r = u2 - prefix[lo];
          x.part = kPhaseAParts + r / Z;
          x.z = r - (r / Z) * Z;
          // (a phase-B partition is never a sequence's last, so it is full)
          if (groups_on) grp = prefix_group(x.b, x.part * p.part_tokens);
          L = p.context_lens[lo];  // checked and clamped by the consumers' prefix pass
          L = L < 0 ? 0 : (L > l_max ? l_max : L);
          x.tb = x.part * p.part_tokens;
          x.te = min(L, x.tb + p.part_tokens);
          x.n_chunks = (x.te - x.tb + kChunk - 1) / kChunk;
          load_entries(x, 0, e0, e1);
        }
      }
      x.n_parts = L == 0 ? 1 : (L + p.part_tokens - 1) / p.part_tokens;
      x.kvh = x.z / p.num_head_tiles;
      x.h0 = x.kvh * p.group + (x.z - x.kvh * p.num_head_tiles) * HT;
      x.nh = min(HT, p.group - (x.z - x.kvh * p.num_head_tiles) * HT);
      x.group = 1;
      if (groups_on && L >= x.tb + p.part_tokens) x.group = grp >= 0 ? grp : prefix_group(x.b, x.tb);
      return true;
    };
    // Finished units of split sequences (the consumers' done ring): each is
    // counted on its (sequence, head tile) counter, which the merge at the
    // end of the launch waits on.  The fence publishes the partials the
    // consumers wrote before arriving on the ring.  Never blocks.
    int dd = 0;  // ring records taken
    bool consumers_done = (flags & kOverlapCombine) == 0;
    auto service = [&]() {
      while (!consumers_done) {
        // take every record that is ready, then one fence for all of them
        DoneInfo rec[kDoneSlots];
        int nrec = 0;
#pragma unroll
        for (int i = 0; i < kDoneSlots; ++i) {
          if (nrec != i || consumers_done) break;
          const int slot = dd % kDoneSlots;
          bool ready = false;
          if (lane == 0) ready = mbar_test_wait(smem_u32(done_full + slot), (dd / kDoneSlots) & 1);
          if (__shfl_sync(kFullMask, ready ? 1 : 0, 0) == 0) break;
          rec[i] = done_info[slot];
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(done_empty + slot));
          ++dd;
          ++nrec;
          if (rec[i].b < 0) consumers_done = true;
        }
        if (nrec == 0) return;
        __threadfence();
#pragma unroll
        for (int i = 0; i < kDoneSlots; ++i) {
          if (i < nrec && rec[i].b >= 0 && lane < rec[i].members) {
            const int bm = rec[i].b + lane;
            bool split = true;
            if (rec[i].members > 1) {  // group members: only split sequences are merged
              int L = p.context_lens[bm];
              L = L < 0 ? 0 : (L > l_max ? l_max : L);
              split = L > p.part_tokens;
            }
            if (split) atomicAdd(p.ws_count + static_cast<int64_t>(bm) * Z + rec[i].z, 1);
          }
        }
      }
    };
    // poll `bar` for phase `parity`, serving the done ring meanwhile (bounded)
    auto wait_serving = [&](uint64_t* bar, int parity) -> bool {
      uint64_t t0 = 0;
      if (lane == 0) t0 = global_timer_ns();
      while (true) {
        bool got = false;
        if (lane == 0) got = mbar_test_wait(smem_u32(bar), parity);
        if (__shfl_sync(kFullMask, got ? 1 : 0, 0) != 0) return true;
        service();
        bool late = false;
        if (lane == 0) late = global_timer_ns() - t0 > p.wait_limit_ns;
        if (__shfl_sync(kFullMask, late ? 1 : 0, 0) != 0) return false;
      }
    };
    bool ok = true;
    // phase A alone has 2 B Z units: fewer than 4 per CTA is a launch of few units
    const int lookahead = 2 * BZ < 4 * static_cast<int>(gridDim.x) ? kLookaheadFew : kLookaheadMany;
    int pk = 0;        // pieces handed over
    int taken = 0;     // pieces the producer is known to have taken
    int queued = 0;    // work handed over but not yet taken, in stage equivalents
    int work_reg = 0;  // lane j < Q: work of the last piece put in queue slot j
    // wait until the producer has taken piece `taken`
    auto retire = [&]() -> bool {
      if (!wait_serving(qempty + taken % Q, (taken / Q) & 1)) return false;
      queued -= __shfl_sync(kFullMask, work_reg, taken % Q);
      ++taken;
      return true;
    };
    auto put_piece = [&](const UnitInfo& x, int c0, int pflags, int e0, int e1, int work) -> bool {
      while (taken <= pk - Q)  // the slot's previous piece must be taken
        if (!retire()) return false;
      Piece& pc = pieces[pk % Q];
      if (lane == 0) {
        pc.u = x;
        pc.c0 = c0;
        pc.flags = pflags;
      }
      pc.e[2 * lane] = e0;
      pc.e[2 * lane + 1] = e1;
      if (lane == pk % Q) work_reg = work;
      queued += work;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(qfull + pk % Q));
      ++pk;
      return true;
    };
    UnitInfo cur{};
    int e0 = 0, e1 = 0;
    bool have_cur = decode_unit(static_cast<int>(blockIdx.x), cur, e0, e1);
    while (ok && have_cur) {
      // work estimates: a stage, plus one for the unit merge; stages of a
      // prefix group carry several sequences
      const int per_stage = cur.group > 1 ? 4 : 1;
      if (cur.group == 0) {
        // covered by its group's leader: nothing to hand over
      } else if (cur.n_chunks == 0) {
        ok = put_piece(cur, 0, kPieceFirst | kPieceLast, 0, 0, 1);
      } else {
        for (int c0 = 0; ok && c0 < cur.n_chunks; c0 += kPieceChunks) {
          if (c0 > 0) load_entries(cur, c0, e0, e1);
          const bool last = c0 + kPieceChunks >= cur.n_chunks;
          const int stages = (min(kPieceChunks, cur.n_chunks - c0) + kSub - 1) / kSub;
          ok = put_piece(cur, c0, (c0 == 0 ? kPieceFirst : 0) | (last ? kPieceLast : 0), e0, e1,
                         stages * per_stage + (last ? 1 : 0));
        }
      }
      if (!ok) break;
      service();
      // claim the next unit only when little work is left queued, so that at
      // the end no CTA sits on claimed units while others run dry
      while (ok && taken < pk && queued > lookahead) ok = retire();
      if (!ok) break;
      int u_nxt = 0;
      if (lane == 0) u_nxt = static_cast<int>(gridDim.x) + atomicAdd(sched_next, 1);
      u_nxt = __shfl_sync(kFullMask, u_nxt, 0);
      have_cur = decode_unit(u_nxt, cur, e0, e1);
      if (!wait_ok) {
        ok = false;
        break;
      }
    }
    if (!put_piece(UnitInfo{}, 0, kPieceStop, 0, 0, 0)) ok = false;
    if (ok && !consumers_done) {  // serve the consumers until their last unit is counted
      uint64_t t0 = 0;
      if (lane == 0) t0 = global_timer_ns();
      while (!consumers_done) {
        service();
        bool late = false;
        if (lane == 0) late = global_timer_ns() - t0 > p.wait_limit_ns;
        if (__shfl_sync(kFullMask, late ? 1 : 0, 0) != 0) {
          ok = false;
          break;
        }
      }
    }
    if (!ok && lane == 0) atomicOr(p.err, kErrWaitTimeout);
    if (lane == 0) {  // the last CTA to finish leaves the counters at zero for the next launch
      __threadfence();
      if (atomicAdd(sched_done, 1) == static_cast<int>(gridDim.x) - 1) {
        atomicExch(sched_next, 0);
        atomicExch(sched_done, 0);
      }
    }
    failed = !ok;
  } else if (warp == W) {
    // ------------------------------- producer -------------------------------
    // Turns queued pieces into 64-token stages: waits for a free ring slot,
    // records the stage, and issues its tensor copies (plus the unit's query
    // rows with its first stage).
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    if (flags & kFuseAppend) {  // no cache read before every CTA's append is done
      if (lane == 0) grid_arrive(p.err);  // this CTA's rows (ordered by the bar.sync after the append)
      bool got = true;
      if (lane == 0) got = grid_wait(p.err, grid_target_, p.wait_limit_ns);
      if (__shfl_sync(kFullMask, got ? 1 : 0, 0) == 0) {
        failed = true;
        if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");  // the other CTAs' rows, for the tensor copies
    }
    int k = 0;   // stage sequence number
    int pk = 0;  // pieces taken
    bool ok = !failed;
    auto acquire_stage = [&](int kk) -> bool {
      bool got = true;
      if (lane == 0) got = mbar_wait_bounded(smem_u32(empty + kk % S), ((kk / S) & 1) ^ 1, p.wait_limit_ns);
      return __shfl_sync(kFullMask, got ? 1 : 0, 0) != 0;
    };
    while (ok) {
      bool got = true;
      if (lane == 0) got = mbar_wait_bounded(smem_u32(qfull + pk % Q), (pk / Q) & 1, p.wait_limit_ns);
      if (__shfl_sync(kFullMask, got ? 1 : 0, 0) == 0) {
        ok = false;
        break;
      }
      const Piece& pc = pieces[pk % Q];
      const UnitInfo cur = pc.u;
      const int pc0 = pc.c0, pflags = pc.flags;
      const int e0 = pc.e[2 * lane], e1 = pc.e[2 * lane + 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(qempty + pk % Q));  // the piece is copied out: slot free
      ++pk;
      if (pflags & kPieceStop) break;
      if (cur.n_chunks == 0) {
        if (!acquire_stage(k)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          meta[k % S] = StageMeta{cur.b, cur.part, 0, 0, cur.n_parts, cur.h0, cur.nh,
                                  kFirst | kLast | kEmptySeq, cur.z, 0, 0, 0};
          mbar_arrive_expect_tx(smem_u32(full + k % S), 0);
        }
        ++k;
      } else {
        const T* qsrc = reinterpret_cast<const T*>(p.q) + cur.b * p.q_sb + static_cast<int64_t>(cur.h0) * p.q_sh;
        const int piece_chunks = min(kPieceChunks, cur.n_chunks - pc0);
        constexpr int SUB = PS::kSub;
        static_assert(kPieceChunks % SUB == 0, "a piece is whole stages");
        const int n_stages = (piece_chunks + SUB - 1) / SUB;
        for (int sg = 0; sg < n_stages; ++sg) {
          const int c0 = pc0 + sg * SUB;
          if (!acquire_stage(k)) { ok = false; break; }
          const int s = k % S;
          const int t0 = cur.tb + kChunk * c0;
          const int nsub = min(SUB, cur.n_chunks - c0);
          const uint32_t stage = smem_u32(ring + s * PS::kStageBytes);
          const uint32_t bar = smem_u32(full + s);
          const bool first = (pflags & kPieceFirst) && sg == 0;
          const bool two = p.log2_bs < 4;  // 8-token blocks: two 8-row boxes per 16-token sub-chunk
          const bool q_rows = first && cur.group == 1;  // group units read q from global memory
          if (lane == 0) {
            const int flags = (first ? kFirst : 0) | ((pflags & kPieceLast) && sg == n_stages - 1 ? kLast : 0) |
                              (cur.group > 1 ? kGroup : 0);
            meta[s] = StageMeta{cur.b, cur.part, t0, cur.te, cur.n_parts, cur.h0, cur.nh, flags, cur.z, nsub,
                                cur.group, 0};
            uint32_t bytes = 0;
#pragma unroll
            for (int j = 0; j < SUB; ++j) {
              if (j < nsub) {
                const int tj = t0 + kChunk * j;
                bytes += (two && !(tj + 8 < cur.te)) ? G::kStageBytes / 2 : G::kStageBytes;
              }
            }
            if (q_rows) bytes += cur.nh * D * static_cast<int>(sizeof(T));
            mbar_arrive_expect_tx(bar, bytes);
          }
          __syncwarp();
          // the stage's tensor copies, one per lane (issued from one lane they
          // take about a microsecond per stage, which bounds a CTA's stream):
          // copy i is box cb (and, with 8-token blocks, 8-row half `half`) of
          // the K (kv = 0) or V tile of sub-chunk j,
          // i = ((j * 2 + kv) * kColBoxes + cb) * H + half
          const int H = (!G::kPairRows && two) ? 2 : 1;
          const int n_copies = nsub * 2 * G::kColBoxes * H;
          for (int base = 0; base < n_copies; base += 32) {
            const int i = base + lane;
            int r = i < n_copies ? i : 0;
            const int half = r % H;
            r /= H;
            const int cb = r % G::kColBoxes;
            r /= G::kColBoxes;
            const int kv = r & 1, j = r >> 1;
            const int src = (sg * SUB + j) & 31;
            const int blk0 = __shfl_sync(kFullMask, e0, src), blk1 = __shfl_sync(kFullMask, e1, src);
            const int tj = t0 + kChunk * j;
            if (i < n_copies && !(half == 1 && !(tj + 8 < cur.te))) {
              const uint32_t dst = stage + (kv * SUB + j) * PS::kKV + cb * 2048 + half * 1024;
              const CUtensorMap* map = kv ? &vmap : &kmap;
              if constexpr (G::kPairRows) {  // rows of two tokens; blocks of >= 16 tokens (host-checked)
                tma_load_3d(dst, map, bar, 0, (cur.kvh * p.block_size + (tj & (p.block_size - 1))) >> 1, blk0);
              } else if (!two) {
                tma_load_3d(dst, map, bar, cb * G::kBoxCols, cur.kvh * p.block_size + (tj & (p.block_size - 1)),
                            blk0);
              } else {
                tma_load_3d(dst, map, bar, cb * G::kBoxCols, cur.kvh * p.block_size, half ? blk1 : blk0);
              }
            }
          }
          if (q_rows) {
            for (int hh = lane; hh < cur.nh; hh += 32)
              bulk_load(stage + 2 * SUB * PS::kKV + hh * D * static_cast<int>(sizeof(T)), qsrc + hh * p.q_sh,
                        D * static_cast<int>(sizeof(T)), bar);
          }
          ++k;
        }
      }
    }
    // tell the consumers to stop
    if (ok && acquire_stage(k)) {
      if (lane == 0) {
        meta[k % S].flags = kStop;
        mbar_arrive_expect_tx(smem_u32(full + k % S), 0);
      }
    } else {
      ok = false;
      if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
    }
    failed = !ok;

  } else {

  // ------------------------------- consumers --------------------------------
  // prefix sums of the phase-B units (partitions >= kPhaseAParts but the
  // last), sequence-major, and the phase-C buckets; then tell the scheduler
  {
    constexpr int kCT = W * 32;
    const int per = (B + kCT - 1) / kCT;
    const int lo = threadIdx.x * per, hi = min(B, lo + per);
    int local = 0;
    for (int b = lo; b < hi; ++b) {
      int L = p.context_lens[b];
      L = L < 0 ? 0 : (L > l_max ? l_max : L);
      local += max(0, (L + p.part_tokens - 1) / p.part_tokens - kPhaseAParts - 1) * Z;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(kFullMask, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    asm volatile("bar.sync 1, %0;" ::"r"(kCT) : "memory");
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += wsum[w];
    for (int b = lo; b < hi; ++b) {  // second read of the same lengths: L1/L2 hits
      prefix[b] = run;
      int L = p.context_lens[b];
      L = L < 0 ? 0 : (L > l_max ? l_max : L);
      const int np = (L + p.part_tokens - 1) / p.part_tokens;
      run += max(0, np - kPhaseAParts - 1) * Z;
      // phase-C bucket: length of the last partition in 32nds of P (0: none)
      const int last = L - (np - 1) * p.part_tokens;
      okey[b] = static_cast<uint8_t>(np <= kPhaseAParts ? 0 : min(32, (last * 32 + p.part_tokens - 1) / p.part_tokens));
    }
    if (threadIdx.x == kCT - 1) prefix[B] = wsum[0] + wsum[1] + wsum[2] + wsum[3];
    asm volatile("bar.sync 1, %0;" ::"r"(kCT) : "memory");
    if (threadIdx.x == 0) mbar_arrive(smem_u32(pbar));
  }
  MmaState<MT, D, NT> st;
  const int cw = warp;
  const uint32_t sync_bar = smem_u32(cbar);
  int sync_phase = 0;
  int dk = 0;  // records handed to the scheduler
  // Every consumer warp arrives on the record's barrier after writing its
  // partials; warp 0 first takes the slot (freed by the scheduler) and fills it.
  auto post_done = [&](const DoneInfo& di) -> bool {
    const int slot = dk % kDoneSlots;
    bool ok = true;
    if (cw == 0) {
      if (lane == 0) ok = mbar_wait_bounded(smem_u32(done_empty + slot), ((dk / kDoneSlots) & 1) ^ 1, p.wait_limit_ns);
      ok = __shfl_sync(kFullMask, ok ? 1 : 0, 0) != 0;
      if (ok && lane == 0) done_info[slot] = di;
    }
    __syncwarp();
    if (ok && lane == 0) mbar_arrive(smem_u32(done_full + slot));
    ++dk;
    if (!ok && lane == 0) atomicOr(p.err, kErrWaitTimeout);
    return ok;
  };
  const bool count_units = (flags & kOverlapCombine) != 0;
  T* out = reinterpret_cast<T*>(p.out);
  for (int k = 0; !failed; ++k) {
    const int s = k % S;
    if (!mbar_wait_bounded(smem_u32(full + s), (k / S) & 1, p.wait_limit_ns)) {
      if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
      failed = true;
      break;
    }
    const StageMeta mt_ = meta[s];
    if (mt_.flags & kStop) break;
    const uint32_t stage = smem_u32(ring + s * PS::kStageBytes);
    if constexpr (kGroupOK) {
      if (mt_.flags & kGroup) {
        // A prefix-group unit, consumed here stage by stage up to its last:
        // warp cw runs members 2cw and 2cw+1 as the two column tiles of one
        // state, each stage as two 32-token halves.
        constexpr int kPerWarp = kMaxGroup / W;
        static_assert(kPerWarp * W == kMaxGroup, "group members split evenly over the consumers");
        MmaState<MT, D, kPerWarp> gs;
        const int gb = mt_.b, gpart = mt_.p, gh0 = mt_.h0, gnh = mt_.nh, gz = mt_.z;
        const int m0 = kPerWarp * cw;
        const int n_mine = max(0, min(kPerWarp, mt_.group - m0));
        if constexpr (F8)
          load_q_members_e4m3<T, D, kPerWarp>(gs, p, gb + m0, n_mine, gh0, gnh, lane);
        else
          load_q_members<T, D, kPerWarp>(gs, p, gb + m0, n_mine, gh0, gnh, lane);
        int t0 = mt_.t0, tok_end = mt_.tok_end, nsub = mt_.nsub, gflags = mt_.flags;
        for (;;) {
          const uint32_t stg = smem_u32(ring + (k % S) * PS::kStageBytes);
          if (n_mine > 0) {
            if constexpr (F8) {  // sub-chunk by sub-chunk (the two members give the parallel work)
#pragma unroll 1
              for (int qq = 0; qq < nsub; ++qq)
                mma_chunks_e4m3<D, kPerWarp, 1>(gs, stg + qq * PS::kKV, stg + (PS::kSub + qq) * PS::kKV,
                                                t0 + qq * kChunk, tok_end, p.scale_log2, lane);
            } else {  // the stage as 32-token pieces
#pragma unroll 1
              for (int qq = 0; qq < nsub; qq += 2)
                mma_multi<T, D, kPerWarp, 2>(gs, stg + qq * PS::kKV, stg + (PS::kSub + qq) * PS::kKV,
                                             t0 + qq * kChunk, tok_end, nsub - qq, p.scale_log2, lane);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(empty + k % S));
          if (gflags & kLast) break;
          ++k;
          if (!mbar_wait_bounded(smem_u32(full + k % S), (k / S) & 1, p.wait_limit_ns)) {
            if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
            failed = true;
            break;
          }
          const StageMeta& gm = meta[k % S];
          t0 = gm.t0;
          tok_end = gm.tok_end;
          nsub = gm.nsub;
          gflags = gm.flags;
        }
        if (failed) break;
        if constexpr (F8)
          finish_members_e4m3<T, D, kPerWarp>(gs, p, gb + m0, n_mine, gpart, gh0, gnh, lane);
        else
          finish_members<T, D, kPerWarp>(gs, p, gb + m0, n_mine, gpart, gh0, gnh, lane);
        if (count_units && !post_done(DoneInfo{gb, gz, mt_.group, 0})) {
          failed = true;
          break;
        }
        // the unit state is not carried past a group unit
        if constexpr (F8)
          load_q_members_e4m3<T, D, NT>(st, p, 0, 0, 0, 0, lane);
        else
          load_q_members<T, D, NT>(st, p, 0, 0, 0, 0, lane);
        continue;
      }
    }
    if (!(mt_.flags & kEmptySeq)) {
      const uint8_t* qtile = ring + s * PS::kStageBytes + 2 * PS::kSub * PS::kKV;
      if constexpr (F8) {
        // consumer cw: sub-chunks 2cw and 2cw + 1 of the 8
        static_assert(PS::kSub == 2 * W, "two sub-chunks per consumer warp");
        if (mt_.flags & kFirst) load_q_smem_e4m3<T, D, NT>(st, qtile, mt_.nh, lane);
        if (2 * cw < mt_.nsub)
          mma_chunks_e4m3<D, NT, 2>(st, stage + 2 * cw * PS::kKV, stage + (PS::kSub + 2 * cw) * PS::kKV,
                                    mt_.t0 + 2 * cw * kChunk, mt_.tok_end, p.scale_log2, lane);
      } else {
        if (mt_.flags & kFirst) load_q_smem<T, D, NT>(st, qtile, mt_.nh, lane);
        if constexpr (PS::kSub == 2 * W) {  // consumer cw: sub-chunks 2cw and 2cw + 1
          if (2 * cw < mt_.nsub)
            mma_multi<T, D, NT, 2>(st, stage + 2 * cw * PS::kKV, stage + (PS::kSub + 2 * cw) * PS::kKV,
                                   mt_.t0 + 2 * cw * kChunk, mt_.tok_end, mt_.nsub - 2 * cw, p.scale_log2, lane);
        } else {
          if (cw < mt_.nsub)
            mma_chunk<T, D, NT>(st, stage + cw * PS::kKV, stage + (PS::kSub + cw) * PS::kKV,
                                mt_.t0 + cw * kChunk, mt_.tok_end, p.scale_log2, lane);
        }
      }
    }
    __syncwarp();
    // the slot of a unit's last stage is kept for the merge and released after it
    if (!(mt_.flags & kLast) || (mt_.flags & kEmptySeq)) {
      if (lane == 0) mbar_arrive(smem_u32(empty + s));
    }
    if (!(mt_.flags & kLast)) continue;

    // ---- the unit is complete: merge the four warps, write out or a partial
    const int b = mt_.b, h0 = mt_.h0, nh = mt_.nh;
    if (mt_.flags & kEmptySeq) {
      for (int idx = cw * 32 + lane; idx < nh * D; idx += W * 32) {
        const int hh = idx / D, d = idx - (idx / D) * D;
        out[b * p.o_sb + static_cast<int64_t>(h0 + hh) * p.o_sh + d] = from_f32<T>(0.f);
      }
      continue;
    }
    // every consumer is done reading the slot's K/V before any overwrites it
    if (!consumer_sync(sync_bar, sync_phase, p.wait_limit_ns, lane)) {
      if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
      failed = true;
      break;
    }
    float* red_o = reinterpret_cast<float*>(ring + s * PS::kStageBytes);  // [W][HT][D]
    float* red_m = red_o + W * HT * D;                                      // [W][HT]
    float* red_l = red_m + W * HT;                                          // [W][HT]
    if constexpr (F8)
      mma_store_e4m3<D, NT>(st, red_o + cw * HT * D, red_m + cw * HT, red_l + cw * HT, lane);
    else
      mma_store<T, D, NT>(st, red_o + cw * HT * D, red_m + cw * HT, red_l + cw * HT, lane);
    if (!consumer_sync(sync_bar, sync_phase, p.wait_limit_ns, lane)) {
      if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
      failed = true;
      break;
    }
    const bool split = mt_.n_parts > 1;
    const int row0 = b * p.num_q_heads + h0;
    for (int hh = cw; hh < nh; hh += W) {
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
      // an fp8 cache holds V / v_scale: the scale comes back here (the
      // partials carry it into the split merge)
      const float vsc = F8 ? p.v_scale : 1.f;
      if (!split) {
        const float inv = vsc / den;
        T* orow = out + b * p.o_sb + static_cast<int64_t>(h0 + hh) * p.o_sh;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          const int d = lane + 32 * i;
          float num = 0.f;
#pragma unroll
          for (int w = 0; w < W; ++w) num += fw[w] * red_o[(w * HT + hh) * D + d];
          orow[d] = from_f32<T>(num * inv);
        }
      } else {
        const int64_t slot = static_cast<int64_t>(row0 + hh) * p.max_parts + mt_.p;
        float* wo = p.ws_o + slot * D;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          const int d = lane + 32 * i;
          float num = 0.f;
#pragma unroll
          for (int w = 0; w < W; ++w) num += fw[w] * red_o[(w * HT + hh) * D + d];
          wo[d] = F8 ? num * vsc : num;
        }
        if (lane == 0) reinterpret_cast<float2*>(p.ws_ml)[slot] = make_float2(M, den);
      }
    }
    // this warp's merge-area accesses are done: order them before the tensor
    // copies that will refill the slot, then release it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + s));
    if (split && count_units && !post_done(DoneInfo{b, mt_.z, 1, 0})) {
      failed = true;
      break;
    }
  }
  if (count_units && !failed && !post_done(DoneInfo{-1, 0, 0, 0})) failed = true;  // no more units
  }  // consumers

  // fused step: once every CTA's partials are written, all warps of all CTAs
  // merge the split rows (one warp per query row)
  // Merge of split sequences, overlapped with other CTAs' decode: warp g of
  // the launch takes rows g, g + (warps in the launch), ...; a row is merged
  // once every unit of its (sequence, head tile) has been counted, rows of a
  // warp in the order they become ready (bounded waits).  The last row of a
  // (sequence, head tile) puts its two counters back to zero.  Every CTA is
  // resident (cooperative launch), so the waits end.
  // Few rows with many partitions each (every row fits one CTA): CTA c merges
  // rows c, c + grid, ... with all its warps, each folding a share of the
  // row's partitions, then combining the shares through shared memory (the
  // ring, idle now).  A row with 128 partitions is then three batched loads
  // per warp instead of sixteen for one warp.  Every decision that guards a
  // barrier is the same for the whole CTA.
  if ((flags & kOverlapCombine) && B * p.num_q_heads <= static_cast<int>(gridDim.x) && p.max_parts >= 8) {
    constexpr int NWARP = W + 2;
    constexpr int V = D / 32;
    const bool cta_failed = __syncthreads_or(failed ? 1 : 0) != 0;
    float* red = reinterpret_cast<float*>(ring);  // [NWARP][D + 2]: each warp's (O, M, den)
    int* flag = reinterpret_cast<int*>(red + NWARP * (D + 2));
    int* count = p.ws_count;
    int* rows_done = p.ws_count + B * Z;
    const int n_rows = B * p.num_q_heads;
    for (int row = static_cast<int>(blockIdx.x); !cta_failed && row < n_rows; row += static_cast<int>(gridDim.x)) {
      const int b = row / p.num_q_heads;
      const int h = row - b * p.num_q_heads;
      int L = p.context_lens[b];
      L = L < 0 ? 0 : (L > l_max ? l_max : L);
      const int np = L == 0 ? 1 : (L + p.part_tokens - 1) / p.part_tokens;
      if (np < 2) continue;  // written by its unit
      const int kvh = h / p.group;
      const int tile = (h - kvh * p.group) / HT;
      const int bz = b * Z + kvh * p.num_head_tiles + tile;
      const int nh = min(HT, p.group - tile * HT);
      if (threadIdx.x == 0) {
        const bool got = counter_wait_bounded(count + bz, np, p.wait_limit_ns);
        if (!got) atomicOr(p.err, kErrWaitTimeout);
        *flag = got ? 1 : 0;
      }
      __syncthreads();  // the acquire above orders every thread's partial loads below
      if (*flag == 0) break;
      const int per = (np + NWARP - 1) / NWARP;
      const int p0 = min(np, warp * per), p1 = min(np, p0 + per);
      float M, den, acc[V];
      merge_part_range<D>(p, row, p0, p1, lane, M, den, acc);
      float* mine = red + warp * (D + 2);
#pragma unroll
      for (int i = 0; i < V; ++i) mine[lane * V + i] = acc[i];
      if (lane == 0) {
        mine[D] = M;
        mine[D + 1] = den;
      }
      __syncthreads();
      if (warp == 0) {
        float Mt = -INFINITY;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) Mt = fmaxf(Mt, red[w * (D + 2) + D]);
        float o[V], dt = 0.f;
#pragma unroll
        for (int i = 0; i < V; ++i) o[i] = 0.f;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) {
          const float mw = red[w * (D + 2) + D];
          const float fw = mw == -INFINITY ? 0.f : exp2f(mw - Mt);
          dt += fw * red[w * (D + 2) + D + 1];
#pragma unroll
          for (int i = 0; i < V; ++i) o[i] = fmaf(fw, red[w * (D + 2) + lane * V + i], o[i]);
        }
        const float inv = 1.f / dt;
        T* orow = reinterpret_cast<T*>(p.out) + b * p.o_sb + static_cast<int64_t>(h) * p.o_sh + lane * V;
#pragma unroll
        for (int i = 0; i < V; ++i) orow[i] = from_f32<T>(o[i] * inv);
        if (lane == 0 && atomicAdd(rows_done + bz, 1) == nh - 1) {  // the tile's last row: counters back to zero
          count[bz] = 0;
          rows_done[bz] = 0;
        }
      }
      __syncthreads();  // the shares are read before the next row overwrites them
    }
  } else if ((flags & kOverlapCombine) && !failed) {
    const int nw = static_cast<int>(gridDim.x) * (W + 2);
    const int gwarp = static_cast<int>(blockIdx.x) * (W + 2) + warp;
    const int n_rows = B * p.num_q_heads;
    int* count = p.ws_count;
    int* rows_done = p.ws_count + B * Z;
    int pend_old = 0, pend_bz = -1, pend_nh = 0;  // row-count arrival whose result is read one row later
    auto settle = [&]() {
      if (pend_bz < 0) return;
      const int old = __shfl_sync(kFullMask, pend_old, 0);
      if (old == pend_nh - 1 && lane == 0) {
        count[pend_bz] = 0;
        rows_done[pend_bz] = 0;
      }
      pend_bz = -1;
    };
    // rows are taken kRowsAtOnce at a time (lane r holds row r) and merged in
    // the order their sequences complete
    constexpr int kRowsAtOnce = 8;
    constexpr int kMergeBatch = 2;
    for (int row0 = gwarp; row0 < n_rows; row0 += kRowsAtOnce * nw) {
      const int my_row = row0 + lane * nw;
      const bool mine = lane < kRowsAtOnce && my_row < n_rows;
      int my_np = 1, my_bz = 0, my_nh = 0;
      if (mine) {
        const int b = my_row / p.num_q_heads;
        const int h = my_row - b * p.num_q_heads;
        int L = p.context_lens[b];
        L = L < 0 ? 0 : (L > l_max ? l_max : L);
        my_np = L == 0 ? 1 : (L + p.part_tokens - 1) / p.part_tokens;
        const int kvh = h / p.group;
        const int tile = (h - kvh * p.group) / HT;
        my_bz = b * Z + kvh * p.num_head_tiles + tile;
        my_nh = min(HT, p.group - tile * HT);
      }
      unsigned pending = __ballot_sync(kFullMask, mine && my_np >= 2);
      uint64_t t0 = 0;
      if (lane == 0) t0 = global_timer_ns();
      bool timed_out = false;
      while (pending != 0) {
        bool rdy = false;
        if ((pending >> lane) & 1) {
          int c;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(c) : "l"(count + my_bz) : "memory");
          rdy = c >= my_np;
        }
        unsigned ready = __ballot_sync(kFullMask, rdy) & pending;
        if (ready == 0) {
          bool late = false;
          if (lane == 0) late = global_timer_ns() - t0 > p.wait_limit_ns;
          if (__shfl_sync(kFullMask, late ? 1 : 0, 0) != 0) {
            timed_out = true;
            break;
          }
          __nanosleep(128);
          continue;
        }
        __syncwarp();  // the ready lanes' acquires order every lane's partial loads below
        pending &= ~ready;
        while (ready != 0) {  // up to kMergeBatch ready rows per batched load
          int rows_b[kMergeBatch], np_b[kMergeBatch], bz_b[kMergeBatch], nh_b[kMergeBatch];
#pragma unroll
          for (int i = 0; i < kMergeBatch; ++i) {
            const int r = ready != 0 ? __ffs(ready) - 1 : -1;
            if (r >= 0) ready &= ready - 1;
            const int rs = r >= 0 ? r : 0;
            rows_b[i] = r >= 0 ? __shfl_sync(kFullMask, my_row, rs) : -1;
            np_b[i] = r >= 0 ? __shfl_sync(kFullMask, my_np, rs) : 1;
            bz_b[i] = __shfl_sync(kFullMask, my_bz, rs);
            nh_b[i] = __shfl_sync(kFullMask, my_nh, rs);
          }
          combine_rows_np<T, D, kMergeBatch>(p, rows_b, np_b, lane);
#pragma unroll
          for (int i = 0; i < kMergeBatch; ++i) {
            if (rows_b[i] < 0) break;
            settle();
            if (lane == 0) pend_old = atomicAdd(rows_done + bz_b[i], 1);
            pend_bz = bz_b[i];
            pend_nh = nh_b[i];
          }
        }
      }
      if (timed_out) {
        if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
        break;
      }
    }
    settle();
  }
}

// Combine kernel for launches that split sequences into partitions: one warp
// per query row.
// Launched as a programmatic dependent of the decode: its CTAs may start
// while the decode's last CTAs still run, and wait here until the decode grid
// has completed and its partials are visible.
template <typename T, int D>
__global__ void __launch_bounds__(256) splitkv_combine(const DecodeParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= p.num_seqs * p.num_q_heads) return;
  const int rows[1] = {row};
  combine_rows<T, D, 1>(p, rows, threadIdx.x & 31);
}

template <typename T, int D, int NT, bool F8>
int persistent_smem(int num_seqs) {
  return PShape<T, D, NT, F8>::kFixedSmem + ((num_seqs + 1 + 3) & ~3) * 4 + kOrderKeys * 4 + (num_seqs * 3 + 15) / 16 * 16;
}

// Launch the persistent decode.  `ap` non-null fuses the KV append in front of
// the decode (behind a grid barrier); `fuse_combine` merges split partitions
// inside the launch (p.ws_count: two zeroed counters per sequence and head
// tile).  Either makes the launch cooperative (the barrier and the merge's
// waits need every CTA resident; the grid never exceeds SMs x occupancy).
// Otherwise split partitions are merged by the separate combine kernel when
// `separate_combine` is set.
template <typename T, int D, int NT, bool F8 = false>
int launch_persistent_inst(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p, int grid,
                           bool separate_combine, const AppendParams* ap, bool fuse_combine,
                           cudaStream_t stream) {
  using PS = PShape<T, D, NT, F8>;
  auto kernel = paged_decode_persistent<T, D, NT, F8>;
  const int smem = persistent_smem<T, D, NT, F8>(p.num_seqs);
  static std::atomic<int> configured_for[64];
  cudaError_t e = static_cast<cudaError_t>(
      raise_smem_limit(configured_for, reinterpret_cast<const void*>(kernel), 227 * 1024));
  if (e != cudaSuccess) return e;
  AppendParams none{};
  const AppendParams& app = ap != nullptr ? *ap : none;
  const int flags = (ap != nullptr ? kFuseAppend : 0) | (fuse_combine ? kOverlapCombine : 0);
  if (flags == 0) {
    kernel<<<grid, PS::kThreads, smem, stream>>>(kmap, vmap, p, app, flags);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    note_launch();
  } else {
    // cooperative (every CTA resident), through the extensible launch so that
    // stream capture records it as a cooperative kernel node
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(PS::kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, kmap, vmap, p, app, flags);
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    note_launch();
  }
  if (!separate_combine || fuse_combine) return cudaSuccess;
  // programmatic dependent launch: no launch gap between the decode's last
  // CTAs and the merge (the merge's griddepcontrol.wait orders its reads)
  cudaLaunchConfig_t ccfg{};
  ccfg.gridDim = dim3((p.num_seqs * p.num_q_heads + 7) / 8);
  ccfg.blockDim = dim3(256);
  ccfg.dynamicSmemBytes = 0;
  ccfg.stream = stream;
  cudaLaunchAttribute cattr[1];
  cattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  cattr[0].val.programmaticStreamSerializationAllowed = 1;
  ccfg.attrs = cattr;
  ccfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&ccfg, splitkv_combine<T, D>, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

template <typename T, int D, int NT, bool F8 = false>
int persistent_occupancy(int num_seqs) {
  // the answer depends only on the shared-memory size: the last one asked per
  // device is remembered as (smem << 8 | blocks)
  static std::atomic<long long> last[64];
  const int smem = persistent_smem<T, D, NT, F8>(num_seqs);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  const bool tracked = dev >= 0 && dev < 64;
  if (tracked) {
    const long long v = last[dev].load(std::memory_order_relaxed);
    if (v != 0 && (v >> 8) == smem) return static_cast<int>(v & 255);
  }
  static std::atomic<int> configured_for[64];
  if (raise_smem_limit(configured_for, reinterpret_cast<const void*>(paged_decode_persistent<T, D, NT, F8>),
                       227 * 1024) != cudaSuccess)
    return 1;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, paged_decode_persistent<T, D, NT, F8>,
                                                    PShape<T, D, NT, F8>::kThreads, smem) != cudaSuccess)
    return 1;
  blocks = blocks < 1 ? 1 : (blocks > 255 ? 255 : blocks);
  if (tracked) last[dev].store((static_cast<long long>(smem) << 8) | blocks, std::memory_order_relaxed);
  return blocks;
}

}  // namespace wllm
