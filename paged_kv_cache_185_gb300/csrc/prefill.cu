// prefill.cu -- chunked-prefill (multi-query) paged attention for sm_103a.
//
// Every sequence b brings a chunk of n_b query tokens, the last n_b of its
// L_b cached tokens (their K/V already appended); the chunk token at position
// P attends causally to the cached tokens 0 .. P through the block table.
// Method: "wLLM" project page, "Features / Core engine" (chunked prefill into
// the paged KV cache) and "mini-vLLM" README, "How it works / Paged
// KV-cache" (block tables over a pool of physical blocks); the tiling below
// is this library's design.
//
// One CTA owns 64 query rows of one sequence and one kv head: row r of the
// sequence's chunk is (token r / G, query head r % G of the kv head's group),
// so the G heads of a group share every staged K/V byte.  A producer warp
// walks the block table and stages 64-token K and V tiles (four 16-row TMA
// boxes each, 128-byte swizzled) into a ring of mbarrier-guarded stages; four
// consumer warps own 16 rows each and run, per tile, S = Q K^T
// (mma.sync m16n8k16, Q fragments held in registers for the whole CTA), the
// causal mask (only on tiles that reach past a row's position), an online
// softmax in the log2 domain, and O += P V with P taken straight from the S
// accumulators.  CTAs are ordered so that the rows with the longest context
// start first.  Every wait is bounded.
//
// Over an fp8 (E4M3) cache (F8) the stages hold codes (half the bytes) and the
// products run in f16: K codes are widened in registers straight into B
// fragments whose k order is a permutation of head_dim (the query's A
// fragments take the same permutation), and V codes go through ldmatrix.trans
// and a byte permute into B fragments of two interleaved head_dim tiles (even
// and odd elements), re-interleaved at the output store; k_scale is folded into
// the softmax scale and v_scale into the output.
#include "common.cuh"
#include "decode_kernel.cuh"
#include "launch.h"
#include "mma_e4m3.cuh"

namespace wllm {

namespace {

constexpr int kPfRows = 64;      // query rows per CTA
constexpr int kPfWarps = 4;      // consumer warps (16 rows each)
constexpr int kPfKv = 64;        // kv tokens per stage
constexpr int kPfStep = 32;      // kv tokens per softmax step (a divisor of kPfKv; 64 measured slower)
constexpr int kPfThreads = (kPfWarps + 1) * 32;

template <typename T, int D, bool F8>
struct PfShape {
  using KT = typename std::conditional<F8, uint8_t, T>::type;  // cache element
  static constexpr int kSub = Geom<KT, D>::kTileBytes;  // 16 rows of one head's K (or V)
  static constexpr int kStageBytes = 2 * (kPfKv / 16) * kSub;
  static constexpr int kStages = (96 * 1024) / kStageBytes;  // two CTAs per SM
  static constexpr int kSmem = 1024 + kStages * kStageBytes + 2 * kStages * 8 + 64;
};

template <typename T, int D, bool F8>
__global__ void __launch_bounds__(kPfThreads, 2)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                         const PrefillParams p) {
  using PS = PfShape<T, D, F8>;
  using MT = typename std::conditional<F8, __half, T>::type;  // tensor-core operand type
  constexpr int S = PS::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * PS::kStageBytes);
  uint64_t* empty = full + S;
  int* info = reinterpret_cast<int*>(empty + S);  // [0] sequence (-1: no tile), [1] tile of it

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int kvh = blockIdx.y;

  // ---- which (sequence, row tile) this CTA owns: sequence b owns
  // ceil(n_b * G / 64) consecutive slots of blockIdx.x
  if (warp == 0) {
    int seq = -1, tile = 0, base = 0;
    for (int b0 = 0; b0 < p.num_seqs && seq < 0; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < p.num_seqs) n = p.query_start_loc[b + 1] - p.query_start_loc[b];
      n = n < 0 ? 0 : n;
      const int tiles = static_cast<int>((static_cast<int64_t>(n) * G + kPfRows - 1) / kPfRows);
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
      for (int s = 0; s < S; ++s) {
        mbar_init(smem_u32(full + s), 1);
        mbar_init(smem_u32(empty + s), kPfWarps);
      }
      fence_mbar_init();
    }
  }
  __syncthreads();
  const int b = info[0];
  if (b < 0) return;
  const int tile = info[1];

  const int l_max = p.max_blocks * p.block_size;
  const int s0 = p.query_start_loc[b];
  int n = p.query_start_loc[b + 1] - s0;
  if (s0 < 0 || n < 0 || static_cast<int64_t>(s0) + n > p.num_tokens) {  // inconsistent query starts
    if (threadIdx.x == 0) atomicOr(p.err, kErrLen);
    return;
  }
  int L = p.context_lens[b];
  if (L < 0 || L > l_max || n > L) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrLen);
    L = L < 0 ? 0 : (L > l_max ? l_max : L);
    n = n > L ? L : n;
  }
  const int n_rows = n * G;
  const int row0 = tile * kPfRows;
  if (row0 >= n_rows) return;  // only when n was clamped (error already flagged)
  const int row_last = min(n_rows, row0 + kPfRows) - 1;
  const int pos0 = L - n;                          // position of the chunk's first token
  const int kv_end = pos0 + row_last / G + 1;      // tokens any row of this CTA sees
  const int n_tiles = (kv_end + kPfKv - 1) / kPfKv;

  if (warp == kPfWarps) {
    // ------------------------------- producer -------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    const int32_t* bt_row = p.block_tables + static_cast<int64_t>(b) * p.bt_stride;
    const bool two = p.log2_bs < 4;  // 8-token blocks: two boxes per 16-row sub-tile
    for (int k = 0; k < n_tiles; ++k) {
      const int s = k % S;
      // lanes 0..3: the table entries of the tile's four 16-token sub-tiles
      int e0 = 0, e1 = 0;
      const int tj = k * kPfKv + 16 * lane;
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
      for (int j = 0; j < 4; ++j) {
        ent0[j] = __shfl_sync(kFullMask, e0, j);
        ent1[j] = __shfl_sync(kFullMask, e1, j);
      }
      bool got = true;
      if (lane == 0) got = mbar_wait_bounded(smem_u32(empty + s), ((k / S) & 1) ^ 1, p.wait_limit_ns);
      if (__shfl_sync(kFullMask, got ? 1 : 0, 0) == 0) {
        if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
        break;
      }
      if (lane == 0) {
        using G16 = Geom<typename PS::KT, D>;
        const uint32_t stage = smem_u32(ring + s * PS::kStageBytes);
        const uint32_t bar = smem_u32(full + s);
        uint32_t bytes = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = k * kPfKv + 16 * j;
          if (t < kv_end) bytes += (two && !(t + 8 < kv_end)) ? G16::kStageBytes / 2 : G16::kStageBytes;
        }
        mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = k * kPfKv + 16 * j;
          if (t >= kv_end) continue;
          const uint32_t kdst = stage + j * PS::kSub;
          const uint32_t vdst = stage + (4 + j) * PS::kSub;
          if constexpr (G16::kPairRows) {  // rows of two tokens; blocks of >= 16 tokens (host-checked)
            const int y = (kvh * p.block_size + (t & (p.block_size - 1))) >> 1;
            tma_load_3d(kdst, &kmap, bar, 0, y, ent0[j]);
            tma_load_3d(vdst, &vmap, bar, 0, y, ent0[j]);
          } else if (!two) {
            const int y = kvh * p.block_size + (t & (p.block_size - 1));
#pragma unroll
            for (int cb = 0; cb < G16::kColBoxes; ++cb) {
              tma_load_3d(kdst + cb * 2048, &kmap, bar, cb * G16::kBoxCols, y, ent0[j]);
              tma_load_3d(vdst + cb * 2048, &vmap, bar, cb * G16::kBoxCols, y, ent0[j]);
            }
          } else {
            const int y = kvh * p.block_size;
#pragma unroll
            for (int cb = 0; cb < G16::kColBoxes; ++cb) {
              tma_load_3d(kdst + cb * 2048, &kmap, bar, cb * G16::kBoxCols, y, ent0[j]);
              tma_load_3d(vdst + cb * 2048, &vmap, bar, cb * G16::kBoxCols, y, ent0[j]);
              if (t + 8 < kv_end) {
                tma_load_3d(kdst + cb * 2048 + 1024, &kmap, bar, cb * G16::kBoxCols, y, ent1[j]);
                tma_load_3d(vdst + cb * 2048 + 1024, &vmap, bar, cb * G16::kBoxCols, y, ent1[j]);
              }
            }
          }
        }
      }
    }
    return;
  }

  // ------------------------------- consumers --------------------------------
  // this warp's rows: wr0 .. wr0+15 of the sequence's chunk rows; this lane
  // holds rows g = lane/4 and g + 8 of them
  const int wr0 = row0 + warp * 16;
  const int g = lane >> 2, c = lane & 3;
  const int ra = wr0 + g, rb = wr0 + g + 8;
  const bool va = ra < n_rows, vb = rb < n_rows;
  // position of each row's token; padding rows see token 0 only (output dropped)
  const int pa = va ? pos0 + ra / G : 0;
  const int pb = vb ? pos0 + rb / G : 0;
  const int warp_last = min(n_rows - 1, wr0 + 15);
  const bool warp_live = wr0 < n_rows;
  const int warp_pmin = warp_live ? pos0 + wr0 / G : 0;
  const int warp_pmax = warp_live ? pos0 + warp_last / G : -1;

  // Q A-fragments for all of head_dim: (row, d) with rows g / g+8, d pairs 2c, 2c+8
  uint32_t qa[D / 16][4];
  {
    const T* qrow_a = reinterpret_cast<const T*>(p.q) +
                      static_cast<int64_t>(s0 + (va ? ra / G : 0)) * p.q_st +
                      static_cast<int64_t>(kvh * G + (va ? ra % G : 0)) * p.q_sh;
    const T* qrow_b = reinterpret_cast<const T*>(p.q) +
                      static_cast<int64_t>(s0 + (vb ? rb / G : 0)) * p.q_st +
                      static_cast<int64_t>(kvh * G + (vb ? rb % G : 0)) * p.q_sh;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      if constexpr (F8) {
        // k 2c, 2c+1 <-> d 16ks+4c, +1 and k 2c+8, 2c+9 <-> d 16ks+4c+2, +3 (the K codes' order)
        const int d = ks * 16 + 4 * c;
        const uint2 za = va ? *reinterpret_cast<const uint2*>(qrow_a + d) : make_uint2(0u, 0u);
        const uint2 zb = vb ? *reinterpret_cast<const uint2*>(qrow_b + d) : make_uint2(0u, 0u);
        qa[ks][0] = to_f16x2<T>(za.x);
        qa[ks][1] = to_f16x2<T>(zb.x);
        qa[ks][2] = to_f16x2<T>(za.y);
        qa[ks][3] = to_f16x2<T>(zb.y);
      } else {
        const int d = ks * 16 + 2 * c;
        qa[ks][0] = va ? *reinterpret_cast<const uint32_t*>(qrow_a + d) : 0u;
        qa[ks][1] = vb ? *reinterpret_cast<const uint32_t*>(qrow_b + d) : 0u;
        qa[ks][2] = va ? *reinterpret_cast<const uint32_t*>(qrow_a + d + 8) : 0u;
        qa[ks][3] = vb ? *reinterpret_cast<const uint32_t*>(qrow_b + d + 8) : 0u;
      }
    }
  }
  float o[D / 8][4];
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[dt][e] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

  // ldmatrix lane addressing: K (non-trans) -> B fragments of two 8-token n-tiles;
  // V (trans) -> B fragments of two 8-wide d-tiles
  const int kb_row = (lane & 7) + ((lane >> 4) << 3), kb_chunk = (lane >> 3) & 1;
  const int vb_row = (lane & 7) + (((lane >> 3) & 1) << 3), vb_chunk = lane >> 4;

  for (int k = 0; k < n_tiles; ++k) {
    const int s = k % S;
    if (!mbar_wait_bounded(smem_u32(full + s), (k / S) & 1, p.wait_limit_ns)) {
      if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
      break;
    }
    const int t0 = k * kPfKv;
    if (warp_live && t0 <= warp_pmax) {
      const uint32_t kt = smem_u32(ring + s * PS::kStageBytes);
      const uint32_t vt = kt + 4 * PS::kSub;
      // the stage as kPfKv / kPfStep softmax steps
      constexpr int NJ = kPfStep / 16;  // 16-token sub-tiles per step
      constexpr int NN = kPfStep / 8;   // 8-token n-tiles per step
#pragma unroll 1
      for (int h = 0; h < kPfKv / kPfStep; ++h) {
        const int th = t0 + kPfStep * h;
        if (th > warp_pmax) break;
        // S = Q K^T over the step: n-tile nt covers tokens th + 8nt .. th + 8nt + 7
        float sc[NN][4];
#pragma unroll
        for (int nt = 0; nt < NN; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
        if constexpr (F8) {
          // one ldmatrix: tokens 0-7 / 8-15 of the sub-tile x code chunks 2kp, 2kp+1 (k steps 2kp, 2kp+1)
#pragma unroll
          for (int kp = 0; kp < D / 32; ++kp) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
              uint32_t r[4];
              ldsm_x4(kt + (NJ * h + j) * PS::kSub + code_offset<D>(kb_row, 2 * kp + kb_chunk), r);
              uint32_t b[4][2];
#pragma unroll
              for (int i = 0; i < 4; ++i) e4m3x4_to_f16x2x2(r[i], b[i][0], b[i][1]);
              Mma<__half>::run(sc[2 * j], qa[2 * kp], b[0]);
              Mma<__half>::run(sc[2 * j], qa[2 * kp + 1], b[1]);
              Mma<__half>::run(sc[2 * j + 1], qa[2 * kp], b[2]);
              Mma<__half>::run(sc[2 * j + 1], qa[2 * kp + 1], b[3]);
            }
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
              uint32_t r[4];
              ldsm_x4(kt + (NJ * h + j) * PS::kSub + tile_offset(kb_row, 2 * ks + kb_chunk), r);
              const uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
              Mma<T>::run(sc[2 * j], qa[ks], b0);
              Mma<T>::run(sc[2 * j + 1], qa[ks], b1);
            }
          }
        }
        // causal mask where the step reaches past a row's position (and past kv_end)
        const bool masked = th + kPfStep - 1 > warp_pmin;
        float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NN; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tok = th + nt * 8 + 2 * c + e;
            float xa = sc[nt][e] * p.scale_log2, xb = sc[nt][2 + e] * p.scale_log2;
            if (masked) {
              xa = tok <= pa ? xa : -INFINITY;
              xb = tok <= pb ? xb : -INFINITY;
            }
            sc[nt][e] = xa;
            sc[nt][2 + e] = xb;
            mx_a = fmaxf(mx_a, xa);
            mx_b = fmaxf(mx_b, xb);
          }
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(kFullMask, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(kFullMask, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(kFullMask, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(kFullMask, mx_b, 2));
        // the first step holds token 0, which every row sees: the running max is finite from there on
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float al_a = exp2f(m_a - mn_a), al_b = exp2f(m_b - mn_b);
        m_a = mn_a;
        m_b = mn_b;
        uint32_t pa_frag[NJ][4];  // P as A fragments of the step's 16-token k steps
        float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
        for (int nt = 0; nt < NN; ++nt) {
          const float p0 = exp2f(sc[nt][0] - mn_a), p1 = exp2f(sc[nt][1] - mn_a);
          const float p2 = exp2f(sc[nt][2] - mn_b), p3 = exp2f(sc[nt][3] - mn_b);
          sum_a += p0 + p1;
          sum_b += p2 + p3;
          pa_frag[nt >> 1][(nt & 1) * 2 + 0] = Mma<MT>::pack(p0, p1);
          pa_frag[nt >> 1][(nt & 1) * 2 + 1] = Mma<MT>::pack(p2, p3);
        }
        l_a = l_a * al_a + sum_a;
        l_b = l_b * al_b + sum_b;
        if (__any_sync(kFullMask, al_a != 1.f || al_b != 1.f)) {
#pragma unroll
          for (int dt = 0; dt < D / 8; ++dt) {
            o[dt][0] *= al_a;
            o[dt][1] *= al_a;
            o[dt][2] *= al_b;
            o[dt][3] *= al_b;
          }
        }
        // O += P V; V rows at or past kv_end were not staged this time: zero them
        const bool tail = th + kPfStep > kv_end;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          uint32_t keep0 = 0xffffffffu, keep1 = 0xffffffffu;
          if (tail) {
            const int tk = th + 16 * j + 2 * c;
            keep0 = (tk < kv_end ? 0x0000ffffu : 0u) | (tk + 1 < kv_end ? 0xffff0000u : 0u);
            keep1 = (tk + 8 < kv_end ? 0x0000ffffu : 0u) | (tk + 9 < kv_end ? 0xffff0000u : 0u);
          }
          if constexpr (F8) {
            // tokens 0-7 / 8-15 x code chunks 2dq, 2dq+1; per chunk m two output tiles:
            // o[2m] holds d = 16m + 2g (even elements), o[2m+1] d = 16m + 2g + 1
#pragma unroll
            for (int dq = 0; dq < D / 32; ++dq) {
              uint32_t r[4];
              ldsm_x4_trans(vt + (NJ * h + j) * PS::kSub + code_offset<D>(vb_row, 2 * dq + vb_chunk), r);
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                uint32_t ev[2], od[2];  // [tokens 0-7, tokens 8-15]
                e4m3x4_to_f16x2x2(__byte_perm(r[2 * half], 0u, 0x3120), ev[0], od[0]);
                e4m3x4_to_f16x2x2(__byte_perm(r[2 * half + 1], 0u, 0x3120), ev[1], od[1]);
                ev[0] &= keep0;
                od[0] &= keep0;
                ev[1] &= keep1;
                od[1] &= keep1;
                const int m = 2 * dq + half;
                Mma<__half>::run(o[2 * m], pa_frag[j], ev);
                Mma<__half>::run(o[2 * m + 1], pa_frag[j], od);
              }
            }
          } else {
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
              uint32_t r[4];
              ldsm_x4_trans(vt + (NJ * h + j) * PS::kSub + tile_offset(vb_row, 2 * dp + vb_chunk), r);
              const uint32_t b0[2] = {r[0] & keep0, r[1] & keep1}, b1[2] = {r[2] & keep0, r[3] & keep1};
              Mma<T>::run(o[2 * dp], pa_frag[j], b0);
              Mma<T>::run(o[2 * dp + 1], pa_frag[j], b1);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + s));
  }

  // ---- epilogue: O / l into the rows' output
  l_a += __shfl_xor_sync(kFullMask, l_a, 1);
  l_a += __shfl_xor_sync(kFullMask, l_a, 2);
  l_b += __shfl_xor_sync(kFullMask, l_b, 1);
  l_b += __shfl_xor_sync(kFullMask, l_b, 2);
  T* out = reinterpret_cast<T*>(p.out);
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {  // row a (accumulator entries 0, 1), then row b (2, 3)
    const bool valid = rr == 0 ? va : vb;
    if (!valid) continue;
    const int row = rr == 0 ? ra : rb;
    const float inv = (F8 ? p.v_scale : 1.f) / (rr == 0 ? l_a : l_b);
    T* orow = out + static_cast<int64_t>(s0 + row / G) * p.o_st + static_cast<int64_t>(kvh * G + row % G) * p.o_sh;
    if constexpr (F8) {
      // chunk m: d = 16m + 4c + {0, 1, 2, 3} = even tile entry 0, odd 0, even 1, odd 1
#pragma unroll
      for (int m = 0; m < D / 16; ++m) {
        const float* ev = o[2 * m];
        const float* od = o[2 * m + 1];
        *reinterpret_cast<uint2*>(orow + 16 * m + 4 * c) =
            make_uint2(Mma<T>::pack(ev[2 * rr] * inv, od[2 * rr] * inv),
                       Mma<T>::pack(ev[2 * rr + 1] * inv, od[2 * rr + 1] * inv));
      }
    } else {
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt)
        *reinterpret_cast<uint32_t*>(orow + dt * 8 + 2 * c) =
            Mma<T>::pack(o[dt][2 * rr] * inv, o[dt][2 * rr + 1] * inv);
    }
  }
}

template <typename T, int D, bool F8>
int launch_prefill_inst(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p, int grid_x,
                        cudaStream_t stream) {
  using PS = PfShape<T, D, F8>;
  auto kernel = paged_prefill_kernel<T, D, F8>;
  static std::atomic<int> configured_for[64];
  cudaError_t e = static_cast<cudaError_t>(
      raise_smem_limit(configured_for, reinterpret_cast<const void*>(kernel), PS::kSmem));
  if (e != cudaSuccess) return e;
  kernel<<<dim3(grid_x, p.num_kv_heads), kPfThreads, PS::kSmem, stream>>>(kmap, vmap, p);
  e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

template <bool F8>
int launch_prefill_f(int dtype, int head_dim, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     const PrefillParams& p, int grid_x, cudaStream_t stream) {
  const bool bf16 = dtype == 2;  // wllm_dtype codes: 1 f16, 2 bf16
  switch (head_dim) {
    case 64:
      return bf16 ? launch_prefill_inst<__nv_bfloat16, 64, F8>(kmap, vmap, p, grid_x, stream)
                  : launch_prefill_inst<__half, 64, F8>(kmap, vmap, p, grid_x, stream);
    case 128:
      return bf16 ? launch_prefill_inst<__nv_bfloat16, 128, F8>(kmap, vmap, p, grid_x, stream)
                  : launch_prefill_inst<__half, 128, F8>(kmap, vmap, p, grid_x, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

int prefill_grid_x(int64_t num_tokens, int64_t num_seqs, int group) {
  // an upper bound on the row tiles: sum_b ceil(n_b G / 64) <= ceil(T G / 64) + B
  return static_cast<int>((num_tokens * group + kPfRows - 1) / kPfRows + num_seqs);
}

int launch_prefill(int dtype, int head_dim, bool kv_fp8, const CUtensorMap& kmap, const CUtensorMap& vmap,
                   const PrefillParams& p, int grid_x, cudaStream_t stream) {
  if (grid_x <= 0) return cudaSuccess;
  return kv_fp8 ? launch_prefill_f<true>(dtype, head_dim, kmap, vmap, p, grid_x, stream)
                : launch_prefill_f<false>(dtype, head_dim, kmap, vmap, p, grid_x, stream);
}

}  // namespace wllm
