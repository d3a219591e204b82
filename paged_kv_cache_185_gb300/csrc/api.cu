// api.cu -- the C ABI of libwllm (declared in include/wllm.h): argument
// validation, per-device state (error word, split-KV workspace), TMA tensor
// maps over the KV pools, variant and partition choice, and the launches.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>

#include "launch.h"
#include "wllm.h"

namespace wllm {
int launch_decode_bf16(int, DecodeVariant, int, const CUtensorMap&, const CUtensorMap&,
                       const DecodeParams&, cudaStream_t);
int launch_decode_f16(int, DecodeVariant, int, const CUtensorMap&, const CUtensorMap&,
                      const DecodeParams&, cudaStream_t);
int launch_decode_f32(int, DecodeVariant, int, const CUtensorMap&, const CUtensorMap&,
                      const DecodeParams&, cudaStream_t);
int smem_decode_bf16(int, DecodeVariant, int);
int smem_decode_f16(int, DecodeVariant, int);
int smem_decode_f32(int, DecodeVariant, int);
int threads_decode_bf16(int);
int threads_decode_f16(int);
int threads_decode_f32(int);
int launch_persistent_bf16(int, int, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int, bool,
                           const AppendParams*, bool, cudaStream_t);
int launch_persistent_f16(int, int, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int, bool,
                          const AppendParams*, bool, cudaStream_t);
int occupancy_persistent_bf16(int, int, int);
int occupancy_persistent_f16(int, int, int);
int launch_persistent_f8_bf16(int, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int, bool,
                              const AppendParams*, bool, cudaStream_t);
int launch_persistent_f8_f16(int, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int, bool,
                             const AppendParams*, bool, cudaStream_t);
int occupancy_persistent_f8_bf16(int, int);
int occupancy_persistent_f8_f16(int, int);

int launch_decode_persistent(int dtype, int head_dim, int head_tile, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, const DecodeParams& p, int grid, bool separate_combine,
                             const AppendParams* ap, bool fuse_combine, bool kv_fp8, cudaStream_t stream) {
  if (kv_fp8) {
    if (head_tile != 8) return cudaErrorInvalidValue;
    switch (dtype) {
      case WLLM_BF16:
        return launch_persistent_f8_bf16(head_dim, kmap, vmap, p, grid, separate_combine, ap, fuse_combine, stream);
      case WLLM_F16:
        return launch_persistent_f8_f16(head_dim, kmap, vmap, p, grid, separate_combine, ap, fuse_combine, stream);
      default:
        return cudaErrorInvalidValue;
    }
  }
  switch (dtype) {
    case WLLM_BF16:
      return launch_persistent_bf16(head_dim, head_tile, kmap, vmap, p, grid, separate_combine, ap, fuse_combine,
                                    stream);
    case WLLM_F16:
      return launch_persistent_f16(head_dim, head_tile, kmap, vmap, p, grid, separate_combine, ap, fuse_combine,
                                   stream);
    default:
      return cudaErrorInvalidValue;
  }
}

int decode_persistent_occupancy(int dtype, int head_dim, int head_tile, int num_seqs, bool kv_fp8) {
  if (kv_fp8)
    return dtype == WLLM_BF16 ? occupancy_persistent_f8_bf16(head_dim, num_seqs)
                              : occupancy_persistent_f8_f16(head_dim, num_seqs);
  return dtype == WLLM_BF16 ? occupancy_persistent_bf16(head_dim, head_tile, num_seqs)
                            : occupancy_persistent_f16(head_dim, head_tile, num_seqs);
}

int decode_head_tile(int dtype, int head_dim, int group, DecodeVariant v, bool kv_fp8) {
  // the fp8 kernel's unit merge fits one ring slot with 8 heads only
  if (kv_fp8 || v == DecodeVariant::kFma || dtype == WLLM_F32) return 8;
  // two 8-head n-tiles when a group needs them and registers allow (D <= 128)
  return (group > 8 && head_dim <= 128) ? 16 : 8;
}

int launch_decode(int dtype, int head_dim, DecodeVariant v, const CUtensorMap& kmap,
                  const CUtensorMap& vmap, const DecodeParams& p, cudaStream_t stream) {
  switch (dtype) {
    case WLLM_BF16: return launch_decode_bf16(head_dim, v, p.head_tile, kmap, vmap, p, stream);
    case WLLM_F16: return launch_decode_f16(head_dim, v, p.head_tile, kmap, vmap, p, stream);
    case WLLM_F32: return launch_decode_f32(head_dim, DecodeVariant::kFma, p.head_tile, kmap, vmap, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

int decode_smem_bytes(int dtype, int head_dim, DecodeVariant v, int head_tile) {
  switch (dtype) {
    case WLLM_BF16: return smem_decode_bf16(head_dim, v, head_tile);
    case WLLM_F16: return smem_decode_f16(head_dim, v, head_tile);
    case WLLM_F32: return smem_decode_f32(head_dim, DecodeVariant::kFma, head_tile);
    default: return -1;
  }
}

namespace {
std::atomic<unsigned long long> g_launches{0};
}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int decode_threads(int dtype, int head_dim) {
  switch (dtype) {
    case WLLM_BF16: return threads_decode_bf16(head_dim);
    case WLLM_F16: return threads_decode_f16(head_dim);
    case WLLM_F32: return threads_decode_f32(head_dim);
    default: return -1;
  }
}
}  // namespace wllm

using namespace wllm;

namespace {

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(WLLM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int* err = nullptr;               // device error word
  uint8_t* ws = nullptr;            // split-KV workspace
  size_t ws_bytes = 0;
  bool ws_owned = true;
  size_t counter_bytes = 0;         // leading bytes reserved for arrival counters (kept zero)
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

bool env_flag(const char* name) {
  const char* v = std::getenv(name);
  return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
}

long long env_int(const char* name, long long dflt) {
  const char* v = std::getenv(name);
  if (v == nullptr || v[0] == '\0') return dflt;
  return std::strtoll(v, nullptr, 10);
}

// Current device's state, created on first use (error word allocated and zeroed).
int device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(WLLM_ERR_UNSUPPORTED, "device index %d too large", dev);
  DeviceState& s = g_devices[dev];
  if (!s.ready) {
    e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = cudaMalloc(reinterpret_cast<void**>(&s.err), kCtrlBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
    e = cudaMemset(s.err, 0, kCtrlBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
    s.ready = true;
  }
  *out = &s;
  return WLLM_OK;
}

// Read and clear the error word after synchronising `stream`.
int collect_device_errors(DeviceState* s, cudaStream_t stream, const char* op) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpy(&word, s->err, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(error word)");
  if (word != 0) {
    cudaMemset(s->err, 0, kCtrlBytes);
    return fail(WLLM_ERR_OUT_OF_RANGE, "%s: device index check failed (error bits 0x%x)", op, word);
  }
  return WLLM_OK;
}

int elt_size(int dtype) {
  switch (dtype) {
    case WLLM_F32: return 4;
    case WLLM_F16: return 2;
    case WLLM_BF16: return 2;
    case WLLM_I32: return 4;
    case WLLM_I64: return 8;
    case WLLM_FP8_E4M3: return 1;
    default: return 0;
  }
}

bool is_float(int dtype) { return dtype == WLLM_F32 || dtype == WLLM_F16 || dtype == WLLM_BF16; }

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

int ilog2(int64_t x) {
  int r = 0;
  while ((int64_t(1) << r) < x) ++r;
  return r;
}

int64_t numel(const wllm_tensor* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

int check_desc(const wllm_tensor* t, const char* name, int ndim) {
  if (t == nullptr) return fail(WLLM_ERR_INVALID_ARG, "%s: null descriptor", name);
  if (t->ndim != ndim) return fail(WLLM_ERR_INVALID_ARG, "%s: expected %d dims, got %d", name, ndim, t->ndim);
  if (elt_size(t->dtype) == 0) return fail(WLLM_ERR_INVALID_ARG, "%s: unknown dtype %d", name, t->dtype);
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0) return fail(WLLM_ERR_INVALID_ARG, "%s: negative size in dim %d", name, i);
  if (t->data == nullptr && numel(t) > 0) return fail(WLLM_ERR_INVALID_ARG, "%s: null data pointer", name);
  return WLLM_OK;
}

bool contiguous(const wllm_tensor* t) {
  int64_t expect = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] != 1 && t->stride[i] != expect) return false;
    expect *= t->shape[i];
  }
  return true;
}

bool same_shape(const wllm_tensor* a, const wllm_tensor* b) {
  if (a->ndim != b->ndim) return false;
  for (int i = 0; i < a->ndim; ++i)
    if (a->shape[i] != b->shape[i]) return false;
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// --- TMA descriptors ---------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 3-D view {D, Hkv*bs, N_b} of a [N_b][Hkv][bs][D] pool; one box is 128 bytes
// of a row by min(bs, 16) rows, 128-byte swizzled.
int make_pool_map(CUtensorMap* map, const void* base, int dtype, int64_t num_blocks, int64_t hkv,
                  int64_t bs, int64_t d, const char* name) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(WLLM_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  const int elt = elt_size(dtype);
  CUtensorMapDataType dt = dtype == WLLM_F32        ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                           : dtype == WLLM_F16      ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                           : dtype == WLLM_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv * bs),
                        static_cast<cuuint64_t>(num_blocks)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * elt), static_cast<cuuint64_t>(hkv * bs * d * elt)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elt), static_cast<cuuint32_t>(bs < 16 ? bs : 16), 1};
  if (dtype == WLLM_FP8_E4M3 && d == 64) {
    // 64-byte rows of codes: view the pool as rows of two tokens (128 bytes),
    // 16 tokens being one box of 8 such rows (block_size >= 16, checked)
    dims[0] = 128;
    dims[1] = static_cast<cuuint64_t>(hkv * bs / 2);
    strides[0] = 128;
    box[1] = 8;
  }
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(WLLM_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", name, (int)r);
  return WLLM_OK;
}

// --- split-KV sizing -----------------------------------------------------------
// Grid kernel: one CTA per (sequence, partition, kv-head tile); the largest
// power of two in [128, 16384] that still gives >= 64 CTAs per SM when every
// sequence is as long as the table allows.
int choose_partition_grid(int64_t num_seqs, int64_t units_per_part, int64_t tokens_max, int num_sms) {
  long long forced = env_int("WLLM_PARTITION_TOKENS", 0);
  int64_t P;
  if (forced > 0) {
    P = (forced + 63) / 64 * 64;
  } else {
    const int64_t target = 64LL * (num_sms > 0 ? num_sms : 148);
    P = 128;
    for (int64_t cand = 16384; cand >= 128; cand >>= 1) {
      if (num_seqs * units_per_part * ((tokens_max + cand - 1) / cand) >= target) {
        P = cand;
        break;
      }
    }
  }
  while ((tokens_max + P - 1) / P > 65535) P *= 2;  // grid.y limit
  return static_cast<int>(P);
}

// Persistent kernel: units are taken dynamically, so what matters is that a
// unit is small against one CTA's share of the work, and that a sequence is
// not cut into so many partitions that merging them costs more than the
// balance gains.  The largest power of two in [512, 4096] that gives >= 8
// units per CTA when sequences are half as long as the table allows (lengths
// are on the device; the table width is all the host knows), but at most 128
// partitions per sequence.  Measured on GB300 over P = 128..4096 on the
// TinyLlama / Llama-2-7B / Qwen2.5-7B / long-context workloads: this picks
// 512 / 4096 / 1024 / 1024 tokens; on the small TinyLlama-shaped batch 512
// beats 256 by ~8% (fewer partials to merge at the end of the launch).
int choose_partition_persistent(int64_t num_seqs, int64_t units_per_part, int64_t tokens_max, int64_t n_ctas) {
  long long forced = env_int("WLLM_PARTITION_TOKENS", 0);
  if (forced > 0) return static_cast<int>((forced + 15) / 16 * 16);
  const int64_t est = tokens_max / 2 > 0 ? tokens_max / 2 : 1;
  int64_t P = 512;
  for (int64_t cand = 4096; cand >= 512; cand >>= 1)
    if (num_seqs * units_per_part * ((est + cand - 1) / cand) >= 8 * n_ctas) {
      P = cand;
      break;
    }
  while (P < 4096 && (tokens_max + P - 1) / P > 128) P *= 2;
  return static_cast<int>(P);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct DecodePlan {
  DecodeVariant variant = DecodeVariant::kMma;
  bool persistent = false;
  int head_tile = 8, tiles = 1, part_tokens = 0, max_parts = 1, grid = 0;
  bool separate_combine = false;
  size_t counter_bytes = 0, ml_bytes = 0, o_bytes = 0;  // all 0 when no sequence is split
};

bool env_is(const char* name, const char* value) {
  const char* v = std::getenv(name);
  return v != nullptr && std::strcmp(v, value) == 0;
}

// Variant, kernel, partition size and workspace layout of one launch over B
// sequences.  `q_bulk_ok`: query rows are 16-byte aligned (bulk-copyable).
// `kv_fp8`: E4M3 caches, which only the persistent kernel reads.
DecodePlan make_plan(int dt, int64_t B, int64_t hq, int64_t hkv, int64_t d, int64_t mb, int64_t bs,
                     bool q_bulk_ok, int num_sms, bool kv_fp8 = false) {
  DecodePlan pl;
  if (kv_fp8) {
    pl.variant = DecodeVariant::kMma;
    pl.persistent = true;
  } else {
    pl.variant = (dt == WLLM_F32 || env_flag("WLLM_FORCE_FMA")) ? DecodeVariant::kFma : DecodeVariant::kMma;
    pl.persistent = pl.variant == DecodeVariant::kMma && q_bulk_ok && !env_is("WLLM_DECODE_KERNEL", "grid");
  }
  const int64_t group = hq / hkv;
  pl.head_tile = decode_head_tile(dt, static_cast<int>(d), static_cast<int>(group), pl.variant, kv_fp8);
  pl.tiles = static_cast<int>((group + pl.head_tile - 1) / pl.head_tile);
  const int64_t tokens_max = std::max<int64_t>(1, mb * bs);
  const int64_t z = hkv * pl.tiles;
  if (pl.persistent) {
    const int occ =
        decode_persistent_occupancy(dt, static_cast<int>(d), pl.head_tile, static_cast<int>(B), kv_fp8);
    const int64_t n_ctas = int64_t(num_sms > 0 ? num_sms : 148) * occ;
    pl.part_tokens = choose_partition_persistent(B, z, tokens_max, n_ctas);
    // An fp8 unit carries half the bytes of a 16-bit one: over long tables the
    // partitions double, halving the partials to merge (GB300, 8 sequences of
    // 32K-128K tokens: 198 -> 187 us).  Shorter tables keep the 16-bit size,
    // which is also the granularity at which prefix groups share a partition.
    if (kv_fp8 && tokens_max >= 65536 && env_int("WLLM_PARTITION_TOKENS", 0) <= 0)
      pl.part_tokens = std::min(4096, 2 * pl.part_tokens);
    while ((tokens_max + pl.part_tokens - 1) / pl.part_tokens > kPersistentMaxParts) pl.part_tokens *= 2;
    pl.max_parts = static_cast<int>((tokens_max + pl.part_tokens - 1) / pl.part_tokens);
    pl.grid = static_cast<int>(std::min<int64_t>(n_ctas, std::max<int64_t>(1, B * z * pl.max_parts)));
    pl.separate_combine = pl.max_parts > 1;
    if (pl.max_parts > 1) {
      // two counters per (sequence, head tile) for the merge inside the launch
      pl.counter_bytes = align256(size_t(B) * z * 2 * sizeof(int));
      pl.ml_bytes = align256(size_t(B) * hq * pl.max_parts * 2 * sizeof(float));
      pl.o_bytes = align256(size_t(B) * hq * pl.max_parts * d * sizeof(float));
    }
  } else {
    pl.part_tokens = choose_partition_grid(B, z, tokens_max, num_sms);
    pl.max_parts = static_cast<int>((tokens_max + pl.part_tokens - 1) / pl.part_tokens);
    if (pl.max_parts > 1) {
      pl.counter_bytes = align256(size_t(B) * z * sizeof(int));
      pl.ml_bytes = align256(size_t(B) * hq * pl.max_parts * 2 * sizeof(float));
      pl.o_bytes = align256(size_t(B) * hq * pl.max_parts * d * sizeof(float));
    }
  }
  return pl;
}


}  // namespace

extern "C" {

const char* wllm_last_error(void) { return g_last_error.c_str(); }

const char* wllm_version(void) { return "wllm-gb300 0.2.0 (sm_103a)"; }

unsigned long long wllm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"

namespace {

bool positive_finite(float x) { return x > 0.f && x < INFINITY; }

// Check the append arguments and fill `ap` (all but the error word).  Leaves
// ap.num_tokens == 0 when there is nothing to write.  `kv_fp8`: the caches
// hold E4M3 codes of key / k_scale and value / v_scale.
int prepare_append(const wllm_tensor* key, const wllm_tensor* value, const wllm_tensor* k_cache,
                   const wllm_tensor* v_cache, const wllm_tensor* slot_mapping, AppendParams& ap,
                   bool kv_fp8 = false, float k_scale = 1.f, float v_scale = 1.f) {
  int rc;
  if ((rc = check_desc(key, "key", 3)) || (rc = check_desc(value, "value", 3)) ||
      (rc = check_desc(k_cache, "k_cache", 4)) || (rc = check_desc(v_cache, "v_cache", 4)) ||
      (rc = check_desc(slot_mapping, "slot_mapping", 1)))
    return rc;
  const int dt = key->dtype;
  if (!is_float(dt)) return fail(WLLM_ERR_INVALID_ARG, "key: dtype must be F32, F16 or BF16");
  if (kv_fp8) {
    if (value->dtype != dt) return fail(WLLM_ERR_INVALID_ARG, "key and value must share one dtype");
    if (k_cache->dtype != WLLM_FP8_E4M3 || v_cache->dtype != WLLM_FP8_E4M3)
      return fail(WLLM_ERR_INVALID_ARG, "caches must be FP8_E4M3");
    if (!positive_finite(k_scale) || !positive_finite(v_scale))
      return fail(WLLM_ERR_INVALID_ARG, "k_scale and v_scale must be positive and finite");
  } else if (value->dtype != dt || k_cache->dtype != dt || v_cache->dtype != dt) {
    return fail(WLLM_ERR_INVALID_ARG, "key, value and caches must share one dtype");
  }
  if (slot_mapping->dtype != WLLM_I64 && slot_mapping->dtype != WLLM_I32)
    return fail(WLLM_ERR_INVALID_ARG, "slot_mapping: dtype must be I64 or I32");
  if (!same_shape(key, value)) return fail(WLLM_ERR_INVALID_ARG, "key and value shapes differ");
  if (!same_shape(k_cache, v_cache)) return fail(WLLM_ERR_INVALID_ARG, "k_cache and v_cache shapes differ");
  const int64_t T = key->shape[0], hkv = key->shape[1], d = key->shape[2];
  const int64_t nb = k_cache->shape[0], bs = k_cache->shape[2];
  if (k_cache->shape[1] != hkv || k_cache->shape[3] != d)
    return fail(WLLM_ERR_INVALID_ARG, "cache shape [%lld,%lld,%lld,%lld] does not match key [T,%lld,%lld]",
                (long long)nb, (long long)k_cache->shape[1], (long long)bs, (long long)k_cache->shape[3],
                (long long)hkv, (long long)d);
  if (!contiguous(k_cache) || !contiguous(v_cache)) return fail(WLLM_ERR_INVALID_ARG, "caches must be dense");
  if (slot_mapping->shape[0] != T) return fail(WLLM_ERR_INVALID_ARG, "slot_mapping must have T entries");
  if (T > 1 && slot_mapping->stride[0] != 1) return fail(WLLM_ERR_INVALID_ARG, "slot_mapping must be contiguous");
  if (d > 1 && (key->stride[2] != 1 || value->stride[2] != 1))
    return fail(WLLM_ERR_INVALID_ARG, "key/value last dimension must be contiguous");
  if (!is_pow2(bs)) return fail(WLLM_ERR_UNSUPPORTED, "block_size %lld is not a power of two", (long long)bs);
  if (kv_fp8 && d % 4 != 0)
    return fail(WLLM_ERR_UNSUPPORTED, "an fp8 cache needs head_dim a multiple of 4, got %lld", (long long)d);
  if (T > INT32_MAX || hkv > INT32_MAX || d * elt_size(dt) > INT32_MAX)
    return fail(WLLM_ERR_UNSUPPORTED, "sizes too large");
  ap = AppendParams{};
  if (T == 0 || hkv == 0 || d == 0) return WLLM_OK;
  const int elt = elt_size(dt);
  ap.key = static_cast<const uint8_t*>(key->data);
  ap.value = static_cast<const uint8_t*>(value->data);
  ap.k_cache = static_cast<uint8_t*>(k_cache->data);
  ap.v_cache = static_cast<uint8_t*>(v_cache->data);
  ap.slots = slot_mapping->data;
  ap.slots_are_i64 = slot_mapping->dtype == WLLM_I64;
  ap.num_tokens = static_cast<int>(T);
  ap.num_kv_heads = static_cast<int>(hkv);
  ap.row_bytes = static_cast<int>(kv_fp8 ? d : d * elt);
  ap.key_st = key->stride[0] * elt;
  ap.key_sh = key->stride[1] * elt;
  ap.val_st = value->stride[0] * elt;
  ap.val_sh = value->stride[1] * elt;
  ap.log2_bs = ilog2(bs);
  ap.num_slots = nb * bs;
  ap.vec16 = !kv_fp8 && (ap.row_bytes % 16 == 0) && aligned(ap.key, 16) && aligned(ap.value, 16) && aligned(ap.k_cache, 16) &&
             aligned(ap.v_cache, 16) && ap.key_st % 16 == 0 && ap.key_sh % 16 == 0 && ap.val_st % 16 == 0 &&
             ap.val_sh % 16 == 0;
  if (kv_fp8) {
    if (!(aligned(ap.key, elt) && aligned(ap.value, elt)))
      return fail(WLLM_ERR_INVALID_ARG, "key/value must be aligned to their element size");
    if (!(aligned(ap.k_cache, 4) && aligned(ap.v_cache, 4)))
      return fail(WLLM_ERR_INVALID_ARG, "fp8 caches must be 4-byte aligned");
    ap.kv_fp8 = 1;
    ap.src_dtype = dt;
    ap.k_inv = 1.f / k_scale;
    ap.v_inv = 1.f / v_scale;
  } else if (!ap.vec16 && !(aligned(ap.key, 2) && aligned(ap.value, 2))) {
    return fail(WLLM_ERR_INVALID_ARG, "key/value must be at least 2-byte aligned");
  }
  return WLLM_OK;
}

// Check-mode pass over the slots (bounds, duplicates): synchronising.
int check_append_slots(DeviceState* s, const AppendParams& ap, cudaStream_t st) {
  cudaError_t e = static_cast<cudaError_t>(
      launch_check_append(ap.slots, ap.slots_are_i64, ap.num_tokens, ap.num_slots, s->err, st));
  if (e != cudaSuccess) return cuda_fail(e, "check_append launch");
  return collect_device_errors(s, st, "reshape_and_cache");
}

}  // namespace

extern "C" {

}  // extern "C"

namespace {

// The allocation-free decode's error word on the current device (defined
// with that call, below).
int noalloc_take_errors();

// The append after its argument checks.
int run_append(AppendParams& ap, wllm_stream stream) {
  int rc;
  DeviceState* s = nullptr;
  if ((rc = device_state(&s))) return rc;
  ap.err = s->err;
  const bool check = env_flag("WLLM_CHECK");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (check && (rc = check_append_slots(s, ap, st))) return rc;
  cudaError_t e = static_cast<cudaError_t>(launch_append(ap, st));
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  if (check) return collect_device_errors(s, st, "reshape_and_cache");
  return WLLM_OK;
}

}  // namespace

extern "C" {

int wllm_reshape_and_cache(const wllm_tensor* key, const wllm_tensor* value, const wllm_tensor* k_cache,
                           const wllm_tensor* v_cache, const wllm_tensor* slot_mapping, wllm_stream stream) {
  AppendParams ap{};
  int rc = prepare_append(key, value, k_cache, v_cache, slot_mapping, ap);
  if (rc || ap.num_tokens == 0) return rc;
  return run_append(ap, stream);
}

int wllm_reshape_and_cache_fp8(const wllm_tensor* key, const wllm_tensor* value, const wllm_tensor* k_cache,
                               const wllm_tensor* v_cache, const wllm_tensor* slot_mapping, float k_scale,
                               float v_scale, wllm_stream stream) {
  AppendParams ap{};
  int rc = prepare_append(key, value, k_cache, v_cache, slot_mapping, ap, true, k_scale, v_scale);
  if (rc || ap.num_tokens == 0) return rc;
  return run_append(ap, stream);
}

size_t wllm_paged_attention_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                            int max_blocks_per_seq, int block_size) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks_per_seq < 0 || num_q_heads % num_kv_heads != 0)
    return 0;
  DeviceState* s = nullptr;
  const int sms = device_state(&s) == WLLM_OK ? s->num_sms : 148;
  // the largest need over the element types and kernels a call may use
  size_t need = 0;
  for (int dt : {WLLM_BF16, WLLM_F32}) {
    for (bool bulk : {true, false}) {
      const int64_t B = std::min<int64_t>(num_seqs, kPersistentMaxSeqs);
      const DecodePlan pl = make_plan(dt, bulk ? B : num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      max_blocks_per_seq, block_size, bulk, sms);
      need = std::max(need, pl.counter_bytes + pl.ml_bytes + pl.o_bytes);
    }
  }
  {  // decode over an fp8 cache
    const int64_t B = std::min<int64_t>(num_seqs, kPersistentMaxSeqs);
    const DecodePlan pl = make_plan(WLLM_BF16, B, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                    block_size, true, sms, true);
    need = std::max(need, pl.counter_bytes + pl.ml_bytes + pl.o_bytes);
  }
  return need;
}

int wllm_partition_tokens(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                          int block_size, int dtype) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
      block_size <= 0 || max_blocks_per_seq < 0 || !is_float(dtype))
    return -1;
  DeviceState* s = nullptr;
  const int sms = device_state(&s) == WLLM_OK ? s->num_sms : 148;
  const int64_t B = std::min<int64_t>(std::max(num_seqs, 1), kPersistentMaxSeqs);
  return make_plan(dtype, B, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size, true, sms)
      .part_tokens;
}

int wllm_set_workspace(void* ptr, size_t bytes) {
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* s = nullptr;
  int rc = device_state(&s);
  if (rc) return rc;
  if ((ptr == nullptr) != (bytes == 0)) return fail(WLLM_ERR_INVALID_ARG, "ptr and bytes must be both set or both 0");
  if (ptr != nullptr && !aligned(ptr, 256)) return fail(WLLM_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  if (s->ws_owned && s->ws != nullptr) cudaFree(s->ws);
  s->ws = static_cast<uint8_t*>(ptr);
  s->ws_bytes = bytes;
  s->ws_owned = ptr == nullptr;
  s->counter_bytes = 0;
  if (ptr != nullptr) {
    e = cudaMemset(ptr, 0, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(workspace)");
  }
  return WLLM_OK;
}

int wllm_device_errors(void) {
  DeviceState* s = nullptr;
  if (device_state(&s) != WLLM_OK) return -1;
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  int word = 0;
  if (cudaMemcpy(&word, s->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  // clearing also resets the persistent kernel's scheduler words, which an
  // aborted launch may have left non-zero, and after a timed-out wait (bit 4)
  // the merge counters
  if (word != 0 && cudaMemset(s->err, 0, kCtrlBytes) != cudaSuccess) return -1;
  if ((word & 16) && s->counter_bytes > 0 && cudaMemset(s->ws, 0, s->counter_bytes) != cudaSuccess) return -1;
  const int noalloc = noalloc_take_errors();
  if (noalloc < 0) return -1;
  return word | noalloc;
}

int wllm_selftest_wait_timeout(unsigned long long limit_ns, wllm_stream stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ULL)
    return fail(WLLM_ERR_INVALID_ARG, "limit_ns must be in (0, 1e9]");
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* s = nullptr;
  int rc = device_state(&s);
  if (rc) return rc;
  int* result = nullptr;  // which waits gave up, kept in the control block's spare words
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  result = s->err + kSelftestResultOffset;
  cudaError_t e = static_cast<cudaError_t>(
      launch_wait_selftest(s->err, kSelftestNeverOffset, kSchedNextOffset, limit_ns, result, st));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  int r = 0;
  e = cudaMemcpyAsync(&r, result, sizeof r, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "self-test result");
  if (r != 3) return fail(WLLM_ERR_CUDA, "self-test: waits that gave up 0x%x, expected both (0x3)", r);
  return WLLM_OK;
}

namespace {

// Point the plan's workspace regions into the device workspace, growing a
// library-owned one when needed.  Arrival counters sit in a leading region
// that is kept zero between calls (extended with a stream-ordered memset).
int bind_workspace(DeviceState* s, const DecodePlan& pl, cudaStream_t st, DecodeParams& p) {
  p.ws_count = nullptr;
  p.ws_ml = nullptr;
  p.ws_o = nullptr;
  if (pl.ml_bytes == 0) return WLLM_OK;
  const size_t partials = pl.ml_bytes + pl.o_bytes;
  size_t reserved = std::max(s->counter_bytes, pl.counter_bytes);
  if (reserved + partials > s->ws_bytes) {
    if (!s->ws_owned)
      return fail(WLLM_ERR_INVALID_ARG, "workspace too small: %zu bytes set, %zu needed", s->ws_bytes,
                  reserved + partials);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    if (s->ws != nullptr) cudaFree(s->ws);
    s->ws = nullptr;
    s->ws_bytes = 0;
    s->counter_bytes = 0;
    reserved = pl.counter_bytes;
    const size_t want = (reserved + partials) + (reserved + partials) / 4;
    e = cudaMalloc(reinterpret_cast<void**>(&s->ws), want);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
    s->ws_bytes = want;
  }
  if (pl.counter_bytes > s->counter_bytes) {
    cudaError_t e = cudaMemsetAsync(s->ws + s->counter_bytes, 0, pl.counter_bytes - s->counter_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(counters)");
    s->counter_bytes = pl.counter_bytes;
  }
  if (pl.counter_bytes > 0) p.ws_count = reinterpret_cast<int*>(s->ws);
  p.ws_ml = reinterpret_cast<float*>(s->ws + s->counter_bytes);
  p.ws_o = reinterpret_cast<float*>(s->ws + s->counter_bytes + pl.ml_bytes);
  return WLLM_OK;
}

}  // namespace

}  // extern "C"

namespace {

struct DecodeArgs {
  int dt = 0, elt = 0;  // query / output type and its size
  int kv_dt = 0;        // cache element type (dt, or WLLM_FP8_E4M3)
  int64_t B = 0, hq = 0, d = 0, nb = 0, hkv = 0, bs = 0, mb = 0;
  bool q_bulk_ok = false;
  bool kv_fp8 = false;
  float k_scale = 1.f, v_scale = 1.f;
};

// Check the decode arguments; a.B == 0 (or no heads) means nothing to do.
// `kv_fp8`: E4M3 caches holding K / k_scale and V / v_scale.
int prepare_decode(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* k_cache,
                   const wllm_tensor* v_cache, const wllm_tensor* block_tables, const wllm_tensor* context_lens,
                   int num_kv_heads, float scale, int block_size, DecodeArgs& a, bool kv_fp8 = false,
                   float k_scale = 1.f, float v_scale = 1.f) {
  int rc;
  if ((rc = check_desc(out, "out", 3)) || (rc = check_desc(q, "q", 3)) ||
      (rc = check_desc(k_cache, "k_cache", 4)) || (rc = check_desc(v_cache, "v_cache", 4)) ||
      (rc = check_desc(block_tables, "block_tables", 2)) || (rc = check_desc(context_lens, "context_lens", 1)))
    return rc;
  const int dt = q->dtype;
  if (kv_fp8) {
    if (dt != WLLM_F16 && dt != WLLM_BF16)
      return fail(WLLM_ERR_INVALID_ARG, "q: dtype must be F16 or BF16 with an fp8 cache");
    if (out->dtype != dt) return fail(WLLM_ERR_INVALID_ARG, "out must have the dtype of q");
    if (k_cache->dtype != WLLM_FP8_E4M3 || v_cache->dtype != WLLM_FP8_E4M3)
      return fail(WLLM_ERR_INVALID_ARG, "caches must be FP8_E4M3");
    if (!positive_finite(k_scale) || !positive_finite(v_scale))
      return fail(WLLM_ERR_INVALID_ARG, "k_scale and v_scale must be positive and finite");
  } else {
    if (!is_float(dt)) return fail(WLLM_ERR_INVALID_ARG, "q: dtype must be F32, F16 or BF16");
    if (out->dtype != dt || k_cache->dtype != dt || v_cache->dtype != dt)
      return fail(WLLM_ERR_INVALID_ARG, "q, out and caches must share one dtype");
  }
  if (block_tables->dtype != WLLM_I32) return fail(WLLM_ERR_INVALID_ARG, "block_tables: dtype must be I32");
  if (context_lens->dtype != WLLM_I32) return fail(WLLM_ERR_INVALID_ARG, "context_lens: dtype must be I32");
  if (!same_shape(out, q)) return fail(WLLM_ERR_INVALID_ARG, "out and q shapes differ");
  if (!same_shape(k_cache, v_cache)) return fail(WLLM_ERR_INVALID_ARG, "k_cache and v_cache shapes differ");
  const int64_t B = q->shape[0], hq = q->shape[1], d = q->shape[2];
  const int64_t nb = k_cache->shape[0], hkv = k_cache->shape[1], bs = k_cache->shape[2];
  if (k_cache->shape[3] != d) return fail(WLLM_ERR_INVALID_ARG, "cache head_dim differs from q");
  if (hkv != num_kv_heads)
    return fail(WLLM_ERR_INVALID_ARG, "num_kv_heads %d differs from cache dim %lld", num_kv_heads, (long long)hkv);
  if (bs != block_size)
    return fail(WLLM_ERR_INVALID_ARG, "block_size %d differs from cache dim %lld", block_size, (long long)bs);
  if (hkv <= 0 || hq % hkv != 0) return fail(WLLM_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
  if (block_tables->shape[0] != B) return fail(WLLM_ERR_INVALID_ARG, "block_tables must have B rows");
  if (context_lens->shape[0] != B) return fail(WLLM_ERR_INVALID_ARG, "context_lens must have B entries");
  if (B > 1 && context_lens->stride[0] != 1) return fail(WLLM_ERR_INVALID_ARG, "context_lens must be contiguous");
  const int64_t mb = block_tables->shape[1];
  if (mb > 1 && block_tables->stride[1] != 1)
    return fail(WLLM_ERR_INVALID_ARG, "block_tables rows must be contiguous");
  if (!contiguous(k_cache) || !contiguous(v_cache)) return fail(WLLM_ERR_INVALID_ARG, "caches must be dense");
  if (d > 1 && (q->stride[2] != 1 || out->stride[2] != 1))
    return fail(WLLM_ERR_INVALID_ARG, "q/out last dimension must be contiguous");
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return fail(WLLM_ERR_INVALID_ARG, "scale must be finite");
  if (d != 64 && d != 128 && d != 256)
    return fail(WLLM_ERR_UNSUPPORTED, "head_dim %lld not supported (64, 128, 256)", (long long)d);
  if (!is_pow2(bs) || bs < 8 || bs > 256)
    return fail(WLLM_ERR_UNSUPPORTED, "block_size %lld not supported (power of two in [8, 256])", (long long)bs);
  if (B > INT32_MAX || hq > 65535 || mb * bs > INT32_MAX || nb > INT32_MAX)
    return fail(WLLM_ERR_UNSUPPORTED, "sizes too large");
  if (kv_fp8 && d == 64 && bs < 16)
    return fail(WLLM_ERR_UNSUPPORTED, "an fp8 cache with head_dim 64 needs block_size >= 16");
  a = DecodeArgs{};
  a.kv_dt = kv_fp8 ? WLLM_FP8_E4M3 : dt;
  a.kv_fp8 = kv_fp8;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.dt = dt;
  a.B = B;
  a.hq = hq;
  if (B == 0 || hq == 0) return WLLM_OK;
  if (nb < 1) return fail(WLLM_ERR_INVALID_ARG, "the pool has no blocks");
  if (!aligned(k_cache->data, 16) || !aligned(v_cache->data, 16))
    return fail(WLLM_ERR_INVALID_ARG, "cache base pointers must be 16-byte aligned");
  const int elt = elt_size(dt);
  if (dt != WLLM_F32 && !(aligned(q->data, 4) && q->stride[0] % 2 == 0 && q->stride[1] % 2 == 0))
    return fail(WLLM_ERR_INVALID_ARG, "q rows must be 4-byte aligned");
  a.elt = elt;
  a.d = d;
  a.nb = nb;
  a.hkv = hkv;
  a.bs = bs;
  a.mb = mb;
  a.q_bulk_ok = aligned(q->data, 16) && (q->stride[0] * elt) % 16 == 0 && (q->stride[1] * elt) % 16 == 0;
  if (kv_fp8 && !a.q_bulk_ok)
    return fail(WLLM_ERR_UNSUPPORTED, "decode over an fp8 cache needs 16-byte aligned query rows");
  return WLLM_OK;
}

// Launch the decode (slices of at most kPersistentMaxSeqs sequences for the
// persistent kernel).  `fuse_ap` non-null runs the KV append inside the first
// persistent launch.  Caller holds g_mutex.
int run_decode(const DecodeArgs& a, const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* k_cache,
               const wllm_tensor* v_cache, const wllm_tensor* block_tables, const wllm_tensor* context_lens,
               float scale, DeviceState* s, cudaStream_t st, const AppendParams* fuse_ap) {
  int rc;
  CUtensorMap kmap, vmap;
  if ((rc = make_pool_map(&kmap, k_cache->data, a.kv_dt, a.nb, a.hkv, a.bs, a.d, "k_cache"))) return rc;
  if ((rc = make_pool_map(&vmap, v_cache->data, a.kv_dt, a.nb, a.hkv, a.bs, a.d, "v_cache"))) return rc;
  const bool check = env_flag("WLLM_CHECK");
  if (check) {
    cudaError_t e = static_cast<cudaError_t>(launch_check_decode(
        static_cast<const int32_t*>(block_tables->data), block_tables->stride[0],
        static_cast<const int32_t*>(context_lens->data), static_cast<int>(a.B), static_cast<int>(a.mb),
        static_cast<int>(a.bs), static_cast<int>(a.nb), s->err, st));
    if (e != cudaSuccess) return cuda_fail(e, "check_decode launch");
    if ((rc = collect_device_errors(s, st, "paged_attention_decode"))) return rc;
  }
  // Split partitions are merged inside the (cooperative) launch, overlapped
  // with the decode, for batches of up to 512 query rows, and by a second
  // kernel (a programmatic dependent of the decode) for larger ones: measured
  // on GB300, merging in the launch is ahead for few rows with many
  // partitions (long contexts: 256 rows, up to 128 partitions each, 328.0 vs
  // 336.3 us) and behind from 1024 rows on (8-head MQA, 1024 rows: 91.3 vs
  // 87.0 us; TinyLlama-shaped, 2048 rows: 34.6 vs 31.9 us; a shared-prefix
  // batch, 7168 rows: 180.8 vs 174.8 us), where the launch's bookkeeping of
  // finished units costs more than a second kernel.
  // WLLM_SEPARATE_COMBINE=1 / 0 forces one or the other.
  const char* sc = std::getenv("WLLM_SEPARATE_COMBINE");
  const bool separate_kernel = (sc != nullptr && sc[0] != '\0') ? std::strcmp(sc, "0") != 0 : a.B * a.hq > 512;
  const DecodePlan first = make_plan(a.dt, std::min<int64_t>(a.B, kPersistentMaxSeqs), a.hq, a.hkv, a.d, a.mb,
                                     a.bs, a.q_bulk_ok, s->num_sms, a.kv_fp8);
  const int64_t slice = first.persistent ? kPersistentMaxSeqs : a.B;
  for (int64_t b0 = 0; b0 < a.B; b0 += slice) {
    const int64_t nbat = std::min<int64_t>(slice, a.B - b0);
    const DecodePlan pl = make_plan(a.dt, nbat, a.hq, a.hkv, a.d, a.mb, a.bs, a.q_bulk_ok, s->num_sms, a.kv_fp8);
    DecodeParams p{};
    p.out = static_cast<uint8_t*>(out->data) + b0 * out->stride[0] * a.elt;
    p.q = static_cast<const uint8_t*>(q->data) + b0 * q->stride[0] * a.elt;
    p.q_sb = q->stride[0];
    p.q_sh = q->stride[1];
    p.o_sb = out->stride[0];
    p.o_sh = out->stride[1];
    p.block_tables = static_cast<const int32_t*>(block_tables->data) + b0 * block_tables->stride[0];
    p.bt_stride = block_tables->stride[0];
    p.context_lens = static_cast<const int32_t*>(context_lens->data) + b0;
    p.num_seqs = static_cast<int>(nbat);
    p.num_q_heads = static_cast<int>(a.hq);
    p.num_kv_heads = static_cast<int>(a.hkv);
    p.group = static_cast<int>(a.hq / a.hkv);
    p.head_tile = pl.head_tile;
    p.num_head_tiles = pl.tiles;
    p.max_blocks = static_cast<int>(a.mb);
    p.block_size = static_cast<int>(a.bs);
    p.log2_bs = ilog2(a.bs);
    p.num_blocks = static_cast<int>(a.nb);
    p.part_tokens = pl.part_tokens;
    p.max_parts = pl.max_parts;
    // an fp8 cache holds K / k_scale: the scale returns in the softmax scale
    p.scale_log2 = (a.kv_fp8 ? scale * a.k_scale : scale) * 1.4426950408889634f;
    p.v_scale = a.v_scale;
    p.err = s->err;
    p.wait_limit_ns = static_cast<unsigned long long>(env_int("WLLM_WAIT_LIMIT_NS", 200000000LL));
    p.prefix_groups = env_int("WLLM_PREFIX_GROUPS", 1) != 0;
    if (!pl.persistent && a.hkv * pl.tiles > 65535) return fail(WLLM_ERR_UNSUPPORTED, "too many kv heads");
    if ((rc = bind_workspace(s, pl, st, p))) return rc;
    cudaError_t e;
    if (pl.persistent) {
      const AppendParams* ap = b0 == 0 ? fuse_ap : nullptr;
      const bool fuse_combine = pl.max_parts > 1 && !separate_kernel;
      e = static_cast<cudaError_t>(launch_decode_persistent(a.dt, static_cast<int>(a.d), pl.head_tile, kmap, vmap,
                                                            p, pl.grid, pl.separate_combine, ap, fuse_combine,
                                                            a.kv_fp8, st));
    } else {
      if (b0 == 0 && fuse_ap != nullptr) {  // no fused form for this kernel: append first
        e = static_cast<cudaError_t>(launch_append(*fuse_ap, st));
        if (e != cudaSuccess) return cuda_fail(e, "append launch");
      }
      e = static_cast<cudaError_t>(launch_decode(a.dt, static_cast<int>(a.d), pl.variant, kmap, vmap, p, st));
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  }
  if (check) return collect_device_errors(s, st, "paged_attention_decode");
  return WLLM_OK;
}

}  // namespace

extern "C" {

}  // extern "C"

namespace {

int decode_call(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* k_cache,
                const wllm_tensor* v_cache, const wllm_tensor* block_tables, const wllm_tensor* context_lens,
                int num_kv_heads, float scale, int block_size, wllm_stream stream, bool kv_fp8, float k_scale,
                float v_scale) {
  DecodeArgs a;
  int rc = prepare_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_kv_heads, scale, block_size, a,
                          kv_fp8, k_scale, v_scale);
  if (rc || a.B == 0 || a.hq == 0) return rc;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* s = nullptr;
  if ((rc = device_state(&s))) return rc;
  return run_decode(a, out, q, k_cache, v_cache, block_tables, context_lens, scale, s,
                    reinterpret_cast<cudaStream_t>(stream), nullptr);
}

int step_call(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* key, const wllm_tensor* value,
              const wllm_tensor* k_cache, const wllm_tensor* v_cache, const wllm_tensor* slot_mapping,
              const wllm_tensor* block_tables, const wllm_tensor* context_lens, int num_kv_heads, float scale,
              int block_size, wllm_stream stream, bool kv_fp8, float k_scale, float v_scale) {
  AppendParams ap{};
  int rc = prepare_append(key, value, k_cache, v_cache, slot_mapping, ap, kv_fp8, k_scale, v_scale);
  if (rc) return rc;
  DecodeArgs a;
  if ((rc = prepare_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_kv_heads, scale, block_size, a,
                           kv_fp8, k_scale, v_scale)))
    return rc;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* s = nullptr;
  if ((rc = device_state(&s))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ap.err = s->err;
  const bool have_append = ap.num_tokens > 0;
  if (have_append && env_flag("WLLM_CHECK") && (rc = check_append_slots(s, ap, st))) return rc;
  if (a.B == 0 || a.hq == 0) {  // nothing to attend: the append alone
    if (!have_append) return WLLM_OK;
    cudaError_t e = static_cast<cudaError_t>(launch_append(ap, st));
    return e == cudaSuccess ? WLLM_OK : cuda_fail(e, "append launch");
  }
  return run_decode(a, out, q, k_cache, v_cache, block_tables, context_lens, scale, s, st,
                    have_append ? &ap : nullptr);
}

}  // namespace

extern "C" {

int wllm_paged_attention_decode(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* k_cache,
                                const wllm_tensor* v_cache, const wllm_tensor* block_tables,
                                const wllm_tensor* context_lens, int num_kv_heads, float scale, int block_size,
                                wllm_stream stream) {
  return decode_call(out, q, k_cache, v_cache, block_tables, context_lens, num_kv_heads, scale, block_size, stream,
                     false, 1.f, 1.f);
}

int wllm_paged_attention_decode_fp8(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* k_cache,
                                    const wllm_tensor* v_cache, const wllm_tensor* block_tables,
                                    const wllm_tensor* context_lens, int num_kv_heads, float scale, float k_scale,
                                    float v_scale, int block_size, wllm_stream stream) {
  return decode_call(out, q, k_cache, v_cache, block_tables, context_lens, num_kv_heads, scale, block_size, stream,
                     true, k_scale, v_scale);
}

int wllm_decode_step(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* key, const wllm_tensor* value,
                     const wllm_tensor* k_cache, const wllm_tensor* v_cache, const wllm_tensor* slot_mapping,
                     const wllm_tensor* block_tables, const wllm_tensor* context_lens, int num_kv_heads, float scale,
                     int block_size, wllm_stream stream) {
  return step_call(out, q, key, value, k_cache, v_cache, slot_mapping, block_tables, context_lens, num_kv_heads,
                   scale, block_size, stream, false, 1.f, 1.f);
}

int wllm_decode_step_fp8(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* key,
                         const wllm_tensor* value, const wllm_tensor* k_cache, const wllm_tensor* v_cache,
                         const wllm_tensor* slot_mapping, const wllm_tensor* block_tables,
                         const wllm_tensor* context_lens, int num_kv_heads, float scale, float k_scale,
                         float v_scale, int block_size, wllm_stream stream) {
  return step_call(out, q, key, value, k_cache, v_cache, slot_mapping, block_tables, context_lens, num_kv_heads,
                   scale, block_size, stream, true, k_scale, v_scale);
}

// ---------------------------------------------------------------------------
// Chunked-prefill (multi-query) paged attention.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

int prefill_call(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* k_cache,
                 const wllm_tensor* v_cache, const wllm_tensor* block_tables, const wllm_tensor* context_lens,
                 const wllm_tensor* query_start_loc, int num_kv_heads, float scale, int block_size,
                 wllm_stream stream, bool kv_fp8, float k_scale, float v_scale) {
  int rc;
  if ((rc = check_desc(out, "out", 3)) || (rc = check_desc(q, "q", 3)) ||
      (rc = check_desc(k_cache, "k_cache", 4)) || (rc = check_desc(v_cache, "v_cache", 4)) ||
      (rc = check_desc(block_tables, "block_tables", 2)) || (rc = check_desc(context_lens, "context_lens", 1)) ||
      (rc = check_desc(query_start_loc, "query_start_loc", 1)))
    return rc;
  const int dt = q->dtype;
  if (dt != WLLM_F16 && dt != WLLM_BF16) return fail(WLLM_ERR_UNSUPPORTED, "prefill takes F16 or BF16 inputs");
  const int kv_dt = kv_fp8 ? WLLM_FP8_E4M3 : dt;
  if (out->dtype != dt) return fail(WLLM_ERR_INVALID_ARG, "out must have the dtype of q");
  if (k_cache->dtype != kv_dt || v_cache->dtype != kv_dt)
    return fail(WLLM_ERR_INVALID_ARG, kv_fp8 ? "caches must be FP8_E4M3" : "q, out and caches must share one dtype");
  if (kv_fp8 && (!positive_finite(k_scale) || !positive_finite(v_scale)))
    return fail(WLLM_ERR_INVALID_ARG, "k_scale and v_scale must be positive and finite");
  if (block_tables->dtype != WLLM_I32 || context_lens->dtype != WLLM_I32 || query_start_loc->dtype != WLLM_I32)
    return fail(WLLM_ERR_INVALID_ARG, "block_tables, context_lens and query_start_loc must be I32");
  if (!same_shape(out, q)) return fail(WLLM_ERR_INVALID_ARG, "out and q shapes differ");
  if (!same_shape(k_cache, v_cache)) return fail(WLLM_ERR_INVALID_ARG, "k_cache and v_cache shapes differ");
  const int64_t T = q->shape[0], hq = q->shape[1], d = q->shape[2];
  const int64_t nb = k_cache->shape[0], hkv = k_cache->shape[1], bs = k_cache->shape[2];
  const int64_t B = context_lens->shape[0], mb = block_tables->shape[1];
  if (k_cache->shape[3] != d) return fail(WLLM_ERR_INVALID_ARG, "cache head_dim differs from q");
  if (hkv != num_kv_heads)
    return fail(WLLM_ERR_INVALID_ARG, "num_kv_heads %d differs from cache dim %lld", num_kv_heads, (long long)hkv);
  if (bs != block_size)
    return fail(WLLM_ERR_INVALID_ARG, "block_size %d differs from cache dim %lld", block_size, (long long)bs);
  if (hkv <= 0 || hq % hkv != 0) return fail(WLLM_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
  if (block_tables->shape[0] != B) return fail(WLLM_ERR_INVALID_ARG, "block_tables must have B rows");
  if (query_start_loc->shape[0] != B + 1) return fail(WLLM_ERR_INVALID_ARG, "query_start_loc must have B+1 entries");
  if (B > 1 && context_lens->stride[0] != 1) return fail(WLLM_ERR_INVALID_ARG, "context_lens must be contiguous");
  if (query_start_loc->stride[0] != 1) return fail(WLLM_ERR_INVALID_ARG, "query_start_loc must be contiguous");
  if (mb > 1 && block_tables->stride[1] != 1)
    return fail(WLLM_ERR_INVALID_ARG, "block_tables rows must be contiguous");
  if (!contiguous(k_cache) || !contiguous(v_cache)) return fail(WLLM_ERR_INVALID_ARG, "caches must be dense");
  if (d > 1 && (q->stride[2] != 1 || out->stride[2] != 1))
    return fail(WLLM_ERR_INVALID_ARG, "q/out last dimension must be contiguous");
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return fail(WLLM_ERR_INVALID_ARG, "scale must be finite");
  if (d != 64 && d != 128) return fail(WLLM_ERR_UNSUPPORTED, "prefill head_dim %lld not supported (64, 128)", (long long)d);
  if (!is_pow2(bs) || bs < 8 || bs > 256)
    return fail(WLLM_ERR_UNSUPPORTED, "block_size %lld not supported (power of two in [8, 256])", (long long)bs);
  if (kv_fp8 && d == 64 && bs < 16)
    return fail(WLLM_ERR_UNSUPPORTED, "an fp8 cache with head_dim 64 needs block_size >= 16");
  if (T > INT32_MAX / 64 || B > INT32_MAX / 2 || hq > 65535 || hkv > 65535 || mb * bs > INT32_MAX || nb > INT32_MAX)
    return fail(WLLM_ERR_UNSUPPORTED, "sizes too large");
  if (T == 0 || B == 0 || hq == 0) return WLLM_OK;
  if (nb < 1) return fail(WLLM_ERR_INVALID_ARG, "the pool has no blocks");
  if (!aligned(k_cache->data, 16) || !aligned(v_cache->data, 16))
    return fail(WLLM_ERR_INVALID_ARG, "cache base pointers must be 16-byte aligned");
  if (!(aligned(q->data, 4) && aligned(out->data, 4) && q->stride[0] % 2 == 0 && q->stride[1] % 2 == 0 &&
        out->stride[0] % 2 == 0 && out->stride[1] % 2 == 0))
    return fail(WLLM_ERR_INVALID_ARG, "q/out rows must be 4-byte aligned");
  if (kv_fp8 && !(aligned(q->data, 8) && aligned(out->data, 8) && q->stride[0] % 4 == 0 && q->stride[1] % 4 == 0 &&
                  out->stride[0] % 4 == 0 && out->stride[1] % 4 == 0))
    return fail(WLLM_ERR_INVALID_ARG, "prefill over an fp8 cache needs 8-byte aligned q/out rows");

  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* s = nullptr;
  if ((rc = device_state(&s))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap kmap, vmap;
  if ((rc = make_pool_map(&kmap, k_cache->data, kv_dt, nb, hkv, bs, d, "k_cache"))) return rc;
  if ((rc = make_pool_map(&vmap, v_cache->data, kv_dt, nb, hkv, bs, d, "v_cache"))) return rc;
  const bool check = env_flag("WLLM_CHECK");
  if (check) {
    cudaError_t e = static_cast<cudaError_t>(launch_check_decode(
        static_cast<const int32_t*>(block_tables->data), block_tables->stride[0],
        static_cast<const int32_t*>(context_lens->data), static_cast<int>(B), static_cast<int>(mb),
        static_cast<int>(bs), static_cast<int>(nb), s->err, st));
    if (e != cudaSuccess) return cuda_fail(e, "check_decode launch");
    if ((rc = collect_device_errors(s, st, "paged_attention_prefill"))) return rc;
  }
  PrefillParams p{};
  p.out = out->data;
  p.q = q->data;
  p.q_st = q->stride[0];
  p.q_sh = q->stride[1];
  p.o_st = out->stride[0];
  p.o_sh = out->stride[1];
  p.block_tables = static_cast<const int32_t*>(block_tables->data);
  p.bt_stride = block_tables->stride[0];
  p.context_lens = static_cast<const int32_t*>(context_lens->data);
  p.query_start_loc = static_cast<const int32_t*>(query_start_loc->data);
  p.num_seqs = static_cast<int>(B);
  p.num_tokens = static_cast<int>(T);
  p.num_q_heads = static_cast<int>(hq);
  p.num_kv_heads = static_cast<int>(hkv);
  p.group = static_cast<int>(hq / hkv);
  p.max_blocks = static_cast<int>(mb);
  p.block_size = static_cast<int>(bs);
  p.log2_bs = ilog2(bs);
  p.num_blocks = static_cast<int>(nb);
  // an fp8 cache holds K / k_scale and V / v_scale: the scales return here
  p.scale_log2 = (kv_fp8 ? scale * k_scale : scale) * 1.4426950408889634f;
  p.v_scale = kv_fp8 ? v_scale : 1.f;
  p.err = s->err;
  p.wait_limit_ns = static_cast<unsigned long long>(env_int("WLLM_WAIT_LIMIT_NS", 200000000LL));
  // the tcgen05 kernel for 16-bit caches with 16-byte aligned q/out rows;
  // WLLM_PREFILL_KERNEL=mma selects the mma.sync kernel
  const bool rows16 = aligned(q->data, 16) && aligned(out->data, 16) && q->stride[0] % 8 == 0 &&
                      q->stride[1] % 8 == 0 && out->stride[0] % 8 == 0 && out->stride[1] % 8 == 0;
  const bool use_tc = !kv_fp8 && rows16 && scale > 0.f && !env_is("WLLM_PREFILL_KERNEL", "mma");
  cudaError_t e;
  if (use_tc) {
    const int grid_x = prefill_tc_grid_x(T, B, p.group);
    e = static_cast<cudaError_t>(launch_prefill_tc(dt, static_cast<int>(d), kmap, vmap, p, grid_x, st));
  } else {
    const int grid_x = prefill_grid_x(T, B, p.group);
    e = static_cast<cudaError_t>(launch_prefill(dt, static_cast<int>(d), kv_fp8, kmap, vmap, p, grid_x, st));
  }
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  if (check) return collect_device_errors(s, st, "paged_attention_prefill");
  return WLLM_OK;
}

}  // namespace

extern "C" {

int wllm_paged_attention_prefill(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* k_cache,
                                 const wllm_tensor* v_cache, const wllm_tensor* block_tables,
                                 const wllm_tensor* context_lens, const wllm_tensor* query_start_loc,
                                 int num_kv_heads, float scale, int block_size, wllm_stream stream) {
  return prefill_call(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc, num_kv_heads, scale,
                      block_size, stream, false, 1.f, 1.f);
}

int wllm_paged_attention_prefill_fp8(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* k_cache,
                                     const wllm_tensor* v_cache, const wllm_tensor* block_tables,
                                     const wllm_tensor* context_lens, const wllm_tensor* query_start_loc,
                                     int num_kv_heads, float scale, float k_scale, float v_scale, int block_size,
                                     wllm_stream stream) {
  return prefill_call(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc, num_kv_heads, scale,
                      block_size, stream, true, k_scale, v_scale);
}

// ---------------------------------------------------------------------------
// Allocation-free decode.
//
// Some callers cannot let a library allocate device memory: an engine whose
// memory manager has reserved all device memory for its own KV pool and
// activations, or a latency-critical caller that cannot accept the implicit
// device synchronisation of cudaMalloc/cudaFree.  For them this
// entry point takes its split-KV scratch (the per-partition partial results)
// and its scheduler/error words from a fixed array in the library's device
// image, sized kNoAllocScratchBytes.  Every GPU that loads the library holds
// that array until the process exits.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per device
constexpr size_t kNoAllocControlBytes = kCtrlBytes;         // error + scheduler words

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
uint8_t* g_noalloc_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.  The host-side
// symbol is only a stand-in; the real address comes from the runtime, once per
// device, with that device current.  That lookup is refused while `stream` is
// being captured into a graph.
int noalloc_scratch(uint8_t** out, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(WLLM_ERR_UNSUPPORTED, "device index %d too large", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_addr[dev] == nullptr) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
      return fail(WLLM_ERR_INVALID_ARG,
                  "the first allocation-free decode on a device looks up its scratch array and must not be made "
                  "while the stream is being captured");
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_noalloc_addr[dev] = static_cast<uint8_t*>(ptr);
  }
  *out = g_noalloc_addr[dev];
  return WLLM_OK;
}

// Read and clear the allocation-free decode's error word on the current device
// (0 when that call has not been used there); the caller has synchronised the
// device.  Clearing also resets its scheduler words.  -1 on a CUDA error.
int noalloc_take_errors() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  uint8_t* ctrl = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    ctrl = g_noalloc_addr[dev];
  }
  if (ctrl == nullptr) return 0;
  int word = 0;
  if (cudaMemcpy(&word, ctrl, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  if (word != 0 && cudaMemset(ctrl, 0, kNoAllocControlBytes) != cudaSuccess) return -1;
  return word;
}

}  // namespace

extern "C" {

int wllm_paged_attention_decode_noalloc(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* k_cache,
                                        const wllm_tensor* v_cache, const wllm_tensor* block_tables,
                                        const wllm_tensor* context_lens, int num_kv_heads, float scale,
                                        int block_size, wllm_stream stream) {
  int rc;
  if ((rc = check_desc(out, "out", 3)) || (rc = check_desc(q, "q", 3)) ||
      (rc = check_desc(k_cache, "k_cache", 4)) || (rc = check_desc(v_cache, "v_cache", 4)) ||
      (rc = check_desc(block_tables, "block_tables", 2)) || (rc = check_desc(context_lens, "context_lens", 1)))
    return rc;
  const int dt = q->dtype;
  if (dt != WLLM_F16 && dt != WLLM_BF16)
    return fail(WLLM_ERR_UNSUPPORTED, "the allocation-free decode takes F16 or BF16 inputs");
  if (out->dtype != dt || k_cache->dtype != dt || v_cache->dtype != dt)
    return fail(WLLM_ERR_INVALID_ARG, "q, out and caches must share one dtype");
  if (block_tables->dtype != WLLM_I32) return fail(WLLM_ERR_INVALID_ARG, "block_tables: dtype must be I32");
  if (context_lens->dtype != WLLM_I32) return fail(WLLM_ERR_INVALID_ARG, "context_lens: dtype must be I32");
  if (!same_shape(out, q)) return fail(WLLM_ERR_INVALID_ARG, "out and q shapes differ");
  if (!same_shape(k_cache, v_cache)) return fail(WLLM_ERR_INVALID_ARG, "k_cache and v_cache shapes differ");
  const int64_t B = q->shape[0], hq = q->shape[1], d = q->shape[2];
  const int64_t nb = k_cache->shape[0], hkv = k_cache->shape[1], bs = k_cache->shape[2];
  if (k_cache->shape[3] != d) return fail(WLLM_ERR_INVALID_ARG, "cache head_dim differs from q");
  if (hkv != num_kv_heads)
    return fail(WLLM_ERR_INVALID_ARG, "num_kv_heads %d differs from cache dim %lld", num_kv_heads, (long long)hkv);
  if (bs != block_size)
    return fail(WLLM_ERR_INVALID_ARG, "block_size %d differs from cache dim %lld", block_size, (long long)bs);
  if (hkv <= 0 || hq % hkv != 0) return fail(WLLM_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
  if (block_tables->shape[0] != B) return fail(WLLM_ERR_INVALID_ARG, "block_tables must have B rows");
  if (context_lens->shape[0] != B) return fail(WLLM_ERR_INVALID_ARG, "context_lens must have B entries");
  if (B > 1 && context_lens->stride[0] != 1) return fail(WLLM_ERR_INVALID_ARG, "context_lens must be contiguous");
  const int64_t mb = block_tables->shape[1];
  if (mb > 1 && block_tables->stride[1] != 1)
    return fail(WLLM_ERR_INVALID_ARG, "block_tables rows must be contiguous");
  if (!contiguous(k_cache) || !contiguous(v_cache)) return fail(WLLM_ERR_INVALID_ARG, "caches must be dense");
  if (d > 1 && (q->stride[2] != 1 || out->stride[2] != 1))
    return fail(WLLM_ERR_INVALID_ARG, "q/out last dimension must be contiguous");
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return fail(WLLM_ERR_INVALID_ARG, "scale must be finite");
  if (d != 64 && d != 128 && d != 256)
    return fail(WLLM_ERR_UNSUPPORTED, "head_dim %lld not supported (64, 128, 256)", (long long)d);
  if (!is_pow2(bs) || bs < 8 || bs > 256)
    return fail(WLLM_ERR_UNSUPPORTED, "block_size %lld not supported (power of two in [8, 256])", (long long)bs);
  if (B > INT32_MAX || hq > 65535 || mb * bs > INT32_MAX || nb > INT32_MAX)
    return fail(WLLM_ERR_UNSUPPORTED, "sizes too large");
  if (B == 0 || hq == 0) return WLLM_OK;
  if (nb < 1) return fail(WLLM_ERR_INVALID_ARG, "the pool has no blocks");
  if (!aligned(k_cache->data, 16) || !aligned(v_cache->data, 16))
    return fail(WLLM_ERR_INVALID_ARG, "cache base pointers must be 16-byte aligned");
  const int elt = elt_size(dt);
  if (!(aligned(q->data, 16) && (q->stride[0] * elt) % 16 == 0 && (q->stride[1] * elt) % 16 == 0))
    return fail(WLLM_ERR_UNSUPPORTED, "the allocation-free decode needs 16-byte aligned query rows");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int num_sms = 0;
  e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch, st))) return rc;

  // plan every slice first: reject before launching anything
  for (int64_t b0 = 0; b0 < B; b0 += kPersistentMaxSeqs) {
    const int64_t nbat = std::min<int64_t>(kPersistentMaxSeqs, B - b0);
    const DecodePlan pl = make_plan(dt, nbat, hq, hkv, d, mb, bs, true, num_sms);
    if (!pl.persistent)
      return fail(WLLM_ERR_UNSUPPORTED, "the allocation-free decode runs only the persistent tensor-core kernel");
    const size_t need = pl.ml_bytes + pl.o_bytes;
    if (need > kNoAllocScratchBytes - kNoAllocControlBytes)
      return fail(WLLM_ERR_UNSUPPORTED,
                  "allocation-free decode: these sizes need %zu bytes of split-KV scratch, the fixed array holds %zu",
                  need, kNoAllocScratchBytes - kNoAllocControlBytes);
  }

  CUtensorMap kmap, vmap;
  if ((rc = make_pool_map(&kmap, k_cache->data, dt, nb, hkv, bs, d, "k_cache"))) return rc;
  if ((rc = make_pool_map(&vmap, v_cache->data, dt, nb, hkv, bs, d, "v_cache"))) return rc;

  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  for (int64_t b0 = 0; b0 < B; b0 += kPersistentMaxSeqs) {
    const int64_t nbat = std::min<int64_t>(kPersistentMaxSeqs, B - b0);
    const DecodePlan pl = make_plan(dt, nbat, hq, hkv, d, mb, bs, true, num_sms);
    // the scheduler words must start at zero; the error word (the first
    // 64 bytes) keeps its bits until wllm_device_errors() reads it; partials
    // need no clearing
    e = cudaMemsetAsync(scratch + kSchedNextOffset * sizeof(int), 0,
                        kNoAllocControlBytes - kSchedNextOffset * sizeof(int), st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(scheduler words)");
    DecodeParams p{};
    p.out = static_cast<uint8_t*>(out->data) + b0 * out->stride[0] * elt;
    p.q = static_cast<const uint8_t*>(q->data) + b0 * q->stride[0] * elt;
    p.q_sb = q->stride[0];
    p.q_sh = q->stride[1];
    p.o_sb = out->stride[0];
    p.o_sh = out->stride[1];
    p.block_tables = static_cast<const int32_t*>(block_tables->data) + b0 * block_tables->stride[0];
    p.bt_stride = block_tables->stride[0];
    p.context_lens = static_cast<const int32_t*>(context_lens->data) + b0;
    p.num_seqs = static_cast<int>(nbat);
    p.num_q_heads = static_cast<int>(hq);
    p.num_kv_heads = static_cast<int>(hkv);
    p.group = static_cast<int>(hq / hkv);
    p.head_tile = pl.head_tile;
    p.num_head_tiles = pl.tiles;
    p.max_blocks = static_cast<int>(mb);
    p.block_size = static_cast<int>(bs);
    p.log2_bs = ilog2(bs);
    p.num_blocks = static_cast<int>(nb);
    p.part_tokens = pl.part_tokens;
    p.max_parts = pl.max_parts;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.v_scale = 1.f;
    p.err = reinterpret_cast<int*>(scratch);
    p.wait_limit_ns = static_cast<unsigned long long>(env_int("WLLM_WAIT_LIMIT_NS", 200000000LL));
    p.prefix_groups = env_int("WLLM_PREFIX_GROUPS", 1) != 0;
    p.ws_count = nullptr;
    p.ws_ml = pl.ml_bytes ? reinterpret_cast<float*>(scratch + kNoAllocControlBytes) : nullptr;
    p.ws_o = pl.ml_bytes ? reinterpret_cast<float*>(scratch + kNoAllocControlBytes + pl.ml_bytes) : nullptr;
    e = static_cast<cudaError_t>(launch_decode_persistent(dt, static_cast<int>(d), pl.head_tile, kmap, vmap, p,
                                                          pl.grid, pl.separate_combine, nullptr, false, false, st));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  }
  return WLLM_OK;
}

}  // extern "C"
