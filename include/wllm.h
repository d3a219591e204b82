/*
 * wllm.h -- C ABI of the GB300 paged KV-cache library (libwllm.so).
 *
 * Two operations make one decode step of a continuously batched engine over a
 * paged KV cache:
 *
 *   wllm_reshape_and_cache       -- the KV append: scatter this step's new key
 *                                   and value rows into the cache slots named
 *                                   by a slot mapping;
 *   wllm_paged_attention_decode  -- single-query attention for every running
 *                                   sequence, reading K/V through its block
 *                                   table from the fixed pool of physical
 *                                   blocks.
 *
 * Sources (page title, then section):
 *   "mini-vLLM" README, "How it works / Paged KV-cache": a fixed pool of
 *     physical blocks of block_size token slots and a per-sequence block table
 *     from logical positions to physical storage;
 *   "mini-vLLM" README, "Results / End-to-end throughput vs baselines" (what
 *     changed): each query head reads its KV head (grouped-query), K/V writes
 *     are one indexed assignment per layer;
 *   "mini-vLLM" README, "Results / Correctness": paged attention equals dense
 *     attention over the same tokens scattered into blocks;
 *   "wLLM" project page, "Features / Core engine": block-based KV cache with
 *     no over-allocation, decode-time paged attention kernel.
 *
 * Conventions shared by every call:
 *   - Every tensor is described by a wllm_tensor: a device pointer, an element
 *     type, a rank and per-dimension sizes and strides counted in ELEMENTS.
 *     The caller owns every buffer; the library never frees or keeps them.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and performs no host synchronisation, except in
 *     check mode (environment variable WLLM_CHECK=1), where it synchronises
 *     the stream after the launch and reports device-detected index errors.
 *   - All argument checks run on the host before anything is launched; a
 *     failed check returns a non-zero wllm_status, launches nothing and
 *     records a message for wllm_last_error().
 *   - Cache layout (both K and V): [num_blocks][num_kv_heads][block_size]
 *     [head_dim], dense (strides D*bs*Hkv, D*bs, D, 1).  Token j of a sequence
 *     sits in physical block table[j / block_size] at slot j % block_size; slot
 *     number s names block s / block_size, offset s % block_size.
 *   - Element types: q, out, key, value and both caches share one type:
 *     WLLM_F32, WLLM_F16 or WLLM_BF16.  Accumulation is fp32 throughout; fp32
 *     inputs never go through reduced-precision tensor-core math.  The *_fp8
 *     calls below take caches of WLLM_FP8_E4M3 codes instead.
 */
#ifndef WLLM_H_
#define WLLM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WLLM_OK = 0,
  WLLM_ERR_INVALID_ARG = 1,  /* shape, type, stride, alignment or pointer    */
  WLLM_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head_dim 96)  */
  WLLM_ERR_OUT_OF_RANGE = 3, /* check mode: an index read on the device was   */
                             /* outside its range (slot, block id, length)    */
  WLLM_ERR_CUDA = 4          /* a CUDA runtime call or launch failed          */
} wllm_status;

typedef enum {
  WLLM_F32 = 0,
  WLLM_F16 = 1,
  WLLM_BF16 = 2,
  WLLM_I32 = 3,
  WLLM_I64 = 4,
  WLLM_FP8_E4M3 = 5  /* one byte: OCP E4M3 "fn" (bias 7, no infinities,      */
                     /* 0x7f/0xff NaN, largest finite +-448)                */
} wllm_dtype;

#define WLLM_MAX_DIMS 4

typedef struct {
  void* data;                      /* device pointer                         */
  int32_t dtype;                   /* a wllm_dtype                           */
  int32_t ndim;                    /* 1..WLLM_MAX_DIMS                       */
  int64_t shape[WLLM_MAX_DIMS];    /* sizes; entries past ndim ignored       */
  int64_t stride[WLLM_MAX_DIMS];   /* strides in elements                    */
} wllm_tensor;

typedef struct CUstream_st* wllm_stream; /* == cudaStream_t */

/*
 * KV append ("reshape and cache").
 *
 * Passage: "mini-vLLM" README, results paragraph on what changed -- the K/V
 * write is one indexed assignment per layer, not a loop over sequences.
 *
 *   key, value    [T][Hkv][D]  F32/F16/BF16, last dimension contiguous, other
 *                 strides free (e.g. a slice of a fused QKV projection output).
 *   k_cache,
 *   v_cache       [N_b][Hkv][bs][D] dense, same type as key.
 *   slot_mapping  [T] WLLM_I64 (or WLLM_I32), contiguous.
 *
 * For every t with s = slot_mapping[t] >= 0 and every kv head h, the D stored
 * elements of key[t][h] are copied bit for bit to k_cache[s/bs][h][s%bs], and
 * value[t][h] to v_cache likewise.  A negative slot is padding: nothing is
 * written.  Slots must be distinct (otherwise which copy lands is undefined).
 * A slot >= N_b*bs is never written; in check mode the call then returns
 * WLLM_ERR_OUT_OF_RANGE (check mode also rejects duplicate slots).
 * T == 0 is valid and launches nothing.
 */
int wllm_reshape_and_cache(const wllm_tensor* key, const wllm_tensor* value,
                           const wllm_tensor* k_cache, const wllm_tensor* v_cache,
                           const wllm_tensor* slot_mapping, wllm_stream stream);

/*
 * Paged decode attention (one query token per sequence).
 *
 * Passages: "mini-vLLM" README, "How it works / Paged KV-cache" (block tables
 * over a fixed pool) and "Results / Correctness" (equal to dense attention,
 * grouped-query heads included); "wLLM" project page, "Features / Core engine"
 * (custom PagedAttention kernel over a block-based KV cache).
 *
 *   out           [B][Hq][D]  written; same type as q; last dim contiguous.
 *   q             [B][Hq][D]  last dimension contiguous.
 *   k_cache,
 *   v_cache       [N_b][Hkv][bs][D] dense, same type as q.
 *   block_tables  [B][M_b] WLLM_I32, last dimension contiguous.  Entries past
 *                 ceil(context_lens[b]/bs) are never read.
 *   context_lens  [B] WLLM_I32, contiguous: tokens sequence b attends to
 *                 (this step's appended token included), 0 <= L <= M_b*bs.
 *   num_kv_heads  must equal the caches' Hkv; Hq % Hkv == 0.  Query head h
 *                 reads KV head h / (Hq/Hkv).
 *   scale         softmax scale applied to q.k (binary32), e.g. 1/sqrt(D).
 *   block_size    must equal the caches' bs; a power of two in [8, 256].
 *
 * out[b][h] = sum_j softmax_j(scale * q[b][h].k_j) * v_j over j < L; a sequence
 * with L == 0 gets zeros.  No masking, ALiBi, soft-capping or sliding window.
 * Supported: D in {64, 128, 256}.  F16/BF16 use tensor-core QK^T and PV with
 * fp32 accumulation; F32 uses fp32 FMA.  The cache base pointers must be
 * 16-byte aligned.  Long contexts are split over several CTAs and combined on
 * the device (split-KV); this uses the device workspace (see below).  With
 * F16/BF16 the partitions of a sequence are merged inside the same
 * (cooperative) launch as soon as all of them are done -- per-sequence
 * counters in the workspace, waits bounded in time -- for batches of up to
 * 512 query rows (B * Hq), and by a second kernel for larger batches; the
 * environment variable WLLM_SEPARATE_COMBINE=1 (or 0) forces the second
 * kernel (or the merge inside the launch).  With a
 * caller workspace set (wllm_set_workspace) the call allocates nothing and can
 * be captured in a CUDA graph.
 * A block-table entry outside [0, N_b) or a length above M_b*bs is clamped on
 * the device (the output of that sequence is then meaningless) and, in check
 * mode, reported as WLLM_ERR_OUT_OF_RANGE.
 */
int wllm_paged_attention_decode(const wllm_tensor* out, const wllm_tensor* q,
                                const wllm_tensor* k_cache, const wllm_tensor* v_cache,
                                const wllm_tensor* block_tables,
                                const wllm_tensor* context_lens, int num_kv_heads,
                                float scale, int block_size, wllm_stream stream);

/*
 * One whole decode step: the KV append followed by paged decode attention,
 * in one launch where the kernel allows it.
 *
 * Passages: those of wllm_reshape_and_cache and wllm_paged_attention_decode;
 * "wLLM" project page, "Features / Core engine" (decode is launch-bound for
 * small models; its launches are worth removing).
 *
 * Arguments are the union of the two calls' arguments, with the same meaning,
 * layout and checks: key/value/slot_mapping as in wllm_reshape_and_cache,
 * out/q/block_tables/context_lens/num_kv_heads/scale/block_size as in
 * wllm_paged_attention_decode, both on the same k_cache/v_cache.  The result is
 * the same as calling the two in order: every appended row is visible to the
 * attention.  For F16/BF16 with 16-byte aligned query rows it is one
 * cooperative launch of the persistent kernel: its CTAs append their share of
 * the rows, meet at a bounded grid barrier, then attend, split sequences being
 * merged as in wllm_paged_attention_decode.  Other inputs run the two calls'
 * kernels back to back.  T == 0 skips the append; B == 0 skips the attention.
 * With a caller workspace set the step allocates nothing, so a model's layers
 * can be captured once in a CUDA graph and replayed.
 */
int wllm_decode_step(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* key,
                     const wllm_tensor* value, const wllm_tensor* k_cache, const wllm_tensor* v_cache,
                     const wllm_tensor* slot_mapping, const wllm_tensor* block_tables,
                     const wllm_tensor* context_lens, int num_kv_heads, float scale, int block_size,
                     wllm_stream stream);

/*
 * Chunked-prefill (multi-query) paged attention.
 *
 * Passages: "wLLM" project page, "Features / Core engine" (chunked prefill: a
 * long prompt enters the paged KV cache a chunk at a time between decode
 * steps); "mini-vLLM" README, "How it works / Paged KV-cache" (block tables).
 * Reading (the pages give no formula): causal attention, each chunk token
 * seeing the sequence's cached tokens before it and itself.
 *
 *   out              [T][Hq][D]  written; same type as q; last dim contiguous.
 *   q                [T][Hq][D]  F16 or BF16; the query chunks of all
 *                    sequences packed one after another; rows 4-byte aligned.
 *   k_cache, v_cache [N_b][Hkv][bs][D] dense, same type as q.
 *   block_tables     [B][M_b] WLLM_I32, last dimension contiguous.
 *   context_lens     [B] WLLM_I32: L_b, the sequence's tokens in the cache,
 *                    its chunk included (append the chunk's K/V first).
 *   query_start_loc  [B+1] WLLM_I32, contiguous: sequence b owns q rows
 *                    query_start_loc[b] .. query_start_loc[b+1]-1 (n_b of them,
 *                    0 allowed); query_start_loc[0] = 0, [B] = T, n_b <= L_b.
 *
 * Chunk token i of sequence b sits at position P = L_b - n_b + i and
 *   out[t][h] = sum_{j <= P} softmax_j(scale * q[t][h].k_j) v_j
 * with query head h reading kv head h / (Hq/Hkv).  A chunk of one token is
 * the decode.  D 64 or 128; tensor-core products with fp32 accumulation, one
 * launch, no workspace, no allocation, no host synchronisation (graph
 * capturable).  Inconsistent query starts or lengths found on the device set
 * the error word (bit 2) and leave those rows unwritten; in check mode the
 * call then returns WLLM_ERR_OUT_OF_RANGE.
 */
int wllm_paged_attention_prefill(const wllm_tensor* out, const wllm_tensor* q,
                                 const wllm_tensor* k_cache, const wllm_tensor* v_cache,
                                 const wllm_tensor* block_tables, const wllm_tensor* context_lens,
                                 const wllm_tensor* query_start_loc, int num_kv_heads,
                                 float scale, int block_size, wllm_stream stream);

/*
 * Chunked prefill over E4M3 caches (the format of wllm_reshape_and_cache_fp8):
 * the same call with K = code * k_scale and V = code * v_scale.  q/out rows
 * 8-byte aligned; D 64 (block_size >= 16) or 128.  The codes are widened to
 * f16 exactly on the device; bf16 queries are rounded to f16 for the
 * products; accumulation is fp32.
 */
int wllm_paged_attention_prefill_fp8(const wllm_tensor* out, const wllm_tensor* q,
                                     const wllm_tensor* k_cache, const wllm_tensor* v_cache,
                                     const wllm_tensor* block_tables,
                                     const wllm_tensor* context_lens,
                                     const wllm_tensor* query_start_loc, int num_kv_heads,
                                     float scale, float k_scale, float v_scale, int block_size,
                                     wllm_stream stream);

/* ---------------------------------------------------------------------------
 * FP8 (E4M3) KV cache.
 *
 * Passage: "vLLM on Windows" build README, release table ("KV compression"
 * column: fp8 listed as a KV-cache dtype of every release).  The page names
 * no format; the storage format is this library's
 * reading: each cache element is the E4M3 code of the element divided by a
 * per-tensor scale (one k_scale for every K element, one v_scale for every V
 * element, binary32, positive and finite):
 *
 *   code = E4M3( fp32(x) * fp32(1 / scale) )
 *
 * the product rounded to binary32, then to the nearest E4M3 value (ties to
 * even), magnitudes above 448 saturating to +-448 (NaN stays NaN).  Reading
 * dequantises value(code) * scale.  Layout, slots, block tables, lengths and
 * every other argument and check are those of the calls above.
 * ------------------------------------------------------------------------- */

/*
 * KV append into E4M3 caches.  key, value: [T][Hkv][D] F32/F16/BF16 (one
 * type), last dimension contiguous, aligned to their element size; caches
 * [N_b][Hkv][bs][D] WLLM_FP8_E4M3, dense, 4-byte aligned; D a multiple of 4.
 * Stores the codes defined above; padding (negative) slots write nothing.
 */
int wllm_reshape_and_cache_fp8(const wllm_tensor* key, const wllm_tensor* value,
                               const wllm_tensor* k_cache, const wllm_tensor* v_cache,
                               const wllm_tensor* slot_mapping, float k_scale, float v_scale,
                               wllm_stream stream);

/*
 * Paged decode attention over E4M3 caches:
 *   out[b][h] = sum_j softmax_j(scale * q.(k_scale * K_j)) * (v_scale * V_j)
 * with K_j, V_j the dequantised codes.  q and out F16 or BF16 (one type),
 * query rows 16-byte aligned; D 64 (block_size >= 16), 128 or 256.  The codes
 * are widened to f16 exactly on the device; bf16 queries are rounded to f16 for
 * the tensor-core products (|q| must stay within the f16 range); accumulation
 * is fp32.  Runs the persistent kernel with split-KV merged inside the launch,
 * like wllm_paged_attention_decode (same workspace rules, graph-capturable with
 * a caller workspace, shared prompt prefixes read once per group for D <= 128).
 */
int wllm_paged_attention_decode_fp8(const wllm_tensor* out, const wllm_tensor* q,
                                    const wllm_tensor* k_cache, const wllm_tensor* v_cache,
                                    const wllm_tensor* block_tables,
                                    const wllm_tensor* context_lens, int num_kv_heads,
                                    float scale, float k_scale, float v_scale, int block_size,
                                    wllm_stream stream);

/*
 * One decode step over E4M3 caches: wllm_reshape_and_cache_fp8 then
 * wllm_paged_attention_decode_fp8 with the same scales, fused into one
 * cooperative launch as in wllm_decode_step.
 */
int wllm_decode_step_fp8(const wllm_tensor* out, const wllm_tensor* q, const wllm_tensor* key,
                         const wllm_tensor* value, const wllm_tensor* k_cache,
                         const wllm_tensor* v_cache, const wllm_tensor* slot_mapping,
                         const wllm_tensor* block_tables, const wllm_tensor* context_lens,
                         int num_kv_heads, float scale, float k_scale, float v_scale,
                         int block_size, wllm_stream stream);

/*
 * Paged decode attention that allocates no device memory.
 *
 * There is no counterpart to this call in the pages.  It is for callers that
 * cannot let a library allocate device memory: an engine whose memory manager
 * has already reserved all device memory for its own KV pool and activations
 * (a cudaMalloc there fails, or takes memory the manager counts on), or a
 * latency-critical caller that cannot accept the implicit device
 * synchronisation of cudaMalloc/cudaFree.  It computes the same result with
 * the same kernel as wllm_paged_attention_decode and takes the same
 * arguments; the caller still owns and passes every input and output.
 *
 * Scratch: the split-KV partial results and the kernel's error and scheduler
 * words live in one fixed 32 MiB array inside the library's device image,
 * which every GPU that loads the library holds until the process exits.
 *   - The first call on a device looks that array's device address up (once,
 *     with the device current).  Make that first call before any stream
 *     capture: made while its stream is capturing, it returns
 *     WLLM_ERR_INVALID_ARG and launches nothing.
 *   - Each call clears the scheduler words, which must start at zero (a
 *     stream-ordered memset of 192 bytes); the partials keep the last call's
 *     contents, and the error word keeps its bits until wllm_device_errors()
 *     reads and clears it (it reports this call's errors together with the
 *     other calls').
 *   - All calls on a device share the array: calls that overlap on the GPU
 *     (different streams, not ordered) race and give wrong results.
 * Supported: F16/BF16 inputs, query rows 16-byte aligned (the persistent
 * tensor-core kernel); anything else returns WLLM_ERR_UNSUPPORTED.  Sizes
 * whose partial results would not fit in the array (many long sequences cut
 * into many partitions) return WLLM_ERR_UNSUPPORTED with the byte counts in
 * wllm_last_error(); nothing is launched then.  Check mode is not available
 * here: a block-table entry outside [0, N_b) or a length above M_b*bs is
 * clamped on the device, as in wllm_paged_attention_decode, and recorded in
 * the error word for wllm_device_errors().
 */
int wllm_paged_attention_decode_noalloc(const wllm_tensor* out, const wllm_tensor* q,
                                        const wllm_tensor* k_cache, const wllm_tensor* v_cache,
                                        const wllm_tensor* block_tables,
                                        const wllm_tensor* context_lens, int num_kv_heads,
                                        float scale, int block_size, wllm_stream stream);

/*
 * Bytes of device workspace that wllm_paged_attention_decode needs for these
 * sizes (0 when no sequence is split).  num_kv_heads is an argument because
 * the merge counters are kept per (sequence, kv head, head tile).  The workspace holds the split-KV
 * partial results and two counters per (sequence, kv head, head tile) for the
 * merge inside the launch.  Every launch leaves the counters at zero; after a
 * launch reports a timed-out wait (error bit 4), wllm_device_errors() zeroes
 * them again.
 */
size_t wllm_paged_attention_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                            int head_dim, int max_blocks_per_seq,
                                            int block_size);

/*
 * Give the library a caller-owned device workspace for the current device
 * (ptr == NULL, bytes == 0 returns to the library-owned one).  The region must
 * stay valid until replaced; it is zeroed here (synchronously).  With a large
 * enough workspace set, decode calls allocate nothing.  Without one, the
 * library allocates its own on first need (cudaMalloc, synchronous) and grows
 * it when a call needs more.  Calls that share a workspace must be ordered on
 * the GPU (same stream, or synchronised): concurrent decode calls on different
 * streams race on it.
 */
int wllm_set_workspace(void* ptr, size_t bytes);

/*
 * Split-KV partition size (tokens per CTA) the library would pick for these
 * sizes on the current device; a multiple of 64.  The environment variable
 * WLLM_PARTITION_TOKENS overrides the choice.  Returns -1 on invalid sizes.
 */
int wllm_partition_tokens(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                          int max_blocks_per_seq, int block_size, int dtype);

/*
 * Read and clear the device error words of the current device (the one of
 * the regular calls and the one of wllm_paged_attention_decode_noalloc, OR-ed
 * together): bit 0 slot out of range, bit 1 block id out of range, bit 2
 * context length out of range, bit 3 duplicate slot (check mode), bit 4 a
 * bounded wait timed out.  Clearing also puts the scheduler and merge counters
 * back to zero, which a launch that gave up on a wait may have left set.
 * Synchronises the device.  Returns -1 if it could not be read.
 */
int wllm_device_errors(void);

/*
 * Self-test of the bounded waits (no counterpart in the pages; it tests this
 * library's failure reporting).  Launches a one-thread kernel that waits on an
 * mbarrier that never receives its arrival and then polls a device counter
 * that never reaches its target, each with the same bounded waits the decode
 * kernels use, limited to limit_ns (in (0, 1e9], else WLLM_ERR_INVALID_ARG).
 * Both waits give up: the kernel sets bit 4 of the device error word and
 * leaves the persistent scheduler's claim counter non-zero, as a decode that
 * gave up half-way would.  The call synchronises `stream` and returns WLLM_OK
 * when both waits reported their timeout.  Call wllm_device_errors() next: it
 * returns bit 4 and puts the counters back to zero; decode calls made before
 * that are wrong.
 */
int wllm_selftest_wait_timeout(unsigned long long limit_ns, wllm_stream stream);

/* Kernel launches the library has issued in this process (a running count;
 * the difference over a region counts that region's launches). */
unsigned long long wllm_launch_count(void);

/* Thread-local message for the last call that did not return WLLM_OK. */
const char* wllm_last_error(void);

/* Library version string. */
const char* wllm_version(void);

/* ---------------------------------------------------------------------------
 * Prefix-caching block manager (host side).
 *
 * Passages: "wLLM" project page, "Features / Core engine" (block-based KV
 * cache; prefix sharing is a block-table operation); "mini-vLLM" README,
 * "How it works / Paged KV-cache" and "What changed" (block tables, a
 * reference count reserved per block for sharing).
 *
 * Decides which physical block of a pool of num_blocks blocks of block_size
 * token slots holds which tokens of which sequence, and produces the block
 * tables, context lengths and slot mappings the calls above consume.  A full
 * block is identified by the chain hash of all tokens up to its last one and
 * keeps its tokens (a hit is checked token for token); sequences whose prompts
 * share full leading blocks share those physical blocks.  Each block counts
 * the sequences that name it; writing into a block that others also name
 * first moves the writer to a private copy (copy-on-write, reported to the
 * caller, who copies the slots on the device).  Unreferenced full blocks stay
 * cached, evictable least recently freed first; other free blocks are used
 * first.  A manager is not thread-safe.  Calls that fail leave it unchanged:
 * WLLM_ERR_INVALID_ARG for unknown or duplicate sequence ids and bad
 * arguments, WLLM_ERR_OUT_OF_RANGE when the pool has too few free blocks (or a
 * table row is too short).  All pointers are host pointers owned by the
 * caller.
 * ------------------------------------------------------------------------- */
typedef struct wllm_block_manager wllm_block_manager;

/* New manager over blocks 0 .. num_blocks-1 (block 0 is handed out first). */
int wllm_bm_create(int num_blocks, int block_size, wllm_block_manager** out);
void wllm_bm_destroy(wllm_block_manager* bm);

/*
 * Register sequence seq_id with its n prompt tokens.  Leading full blocks
 * already cached with the same tokens are shared; the rest are fresh blocks.
 * slots (may be NULL) receives [n] the slot (block * block_size + offset) of
 * every token; *cached_tokens (may be NULL) the number of leading tokens whose
 * K/V is already in the cache (a multiple of block_size): only slots from
 * there on need writing.
 */
int wllm_bm_add_sequence(wllm_block_manager* bm, int64_t seq_id, const int32_t* tokens, int64_t n,
                         int64_t* slots, int64_t* cached_tokens);

/*
 * Append one token to seq_id (a decode step): *slot receives the slot the
 * token's K/V goes to.  If the sequence's last block was shared and partly
 * filled, the sequence first moves to a private copy: *copy_src / *copy_dst
 * receive the two blocks and the caller must copy the first
 * (context_len % block_size) slots of each kv head from src to dst before
 * writing; otherwise both receive -1.  A block that becomes full is cached.
 */
int wllm_bm_append_token(wllm_block_manager* bm, int64_t seq_id, int32_t token, int64_t* slot,
                         int32_t* copy_src, int32_t* copy_dst);

/* child shares all of parent's blocks (e.g. several samples of one prompt). */
int wllm_bm_fork(wllm_block_manager* bm, int64_t parent, int64_t child);

/* Drop seq_id; blocks no longer named by any sequence become free. */
int wllm_bm_free_sequence(wllm_block_manager* bm, int64_t seq_id);

/*
 * seq_id's block-table row: row[0 .. max_blocks) gets its blocks, -1 past the
 * last; *context_len (may be NULL) its token count.  WLLM_ERR_OUT_OF_RANGE if
 * the sequence holds more than max_blocks blocks.
 */
int wllm_bm_block_table(const wllm_block_manager* bm, int64_t seq_id, int32_t* row, int max_blocks,
                        int64_t* context_len);

/* Free blocks (unreferenced, cached ones included); -1 for a NULL manager. */
int64_t wllm_bm_num_free_blocks(const wllm_block_manager* bm);
/* Full blocks currently findable by prompt tokens; -1 for a NULL manager. */
int64_t wllm_bm_num_cached_blocks(const wllm_block_manager* bm);
/* Sequences naming block (its reference count); -1 if out of range. */
int wllm_bm_block_ref(const wllm_block_manager* bm, int32_t block);

#ifdef __cplusplus
}
#endif

#endif /* WLLM_H_ */
