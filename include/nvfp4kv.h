/*
 * nvfp4kv: NVFP4 (and FP8 E4M3) paged KV cache for LLM decode on one GB300
 * (sm_103a).  C ABI: plain pointers and sizes; no framework types.
 *
 * Sources (page title, section):
 *   [P1] "SOAR Weekly Champion Notes 05 | Zhisuan Team One: NVFP4 KV Cache and
 *        Mixed-Precision Practice": 02 NVFP4 KV Cache (E2M1 = 1 sign + 2
 *        exponent + 1 mantissa bit, two values per byte, quantized write and
 *        dequantized read paths, FP4 memory pool); 03 Mixed-precision KV
 *        Cache (FP8 for the sensitive first/last layers, NVFP4 elsewhere).
 *   [P2] "SGLang x Qwen x NVIDIA Collaboration: NVFP4 KV Cache Breaks
 *        Long-Context and Agentic Inference Bottlenecks": The Core of the
 *        Ledger (one E4M3 block scale per 16 values, one FP32 global scale per
 *        tensor, 9 bytes per 16 values); Three Paths (the initial prefill
 *        requantizes its FP8 KV into the cache; decode reads NVFP4 from the
 *        paged cache and dequantizes inside the kernel; chunked extend
 *        dequantizes the cached prefix into a shared FP8 workspace, runs FP8
 *        attention over it and the new chunk, and quantizes the new chunk
 *        into the cache); the equal-capacity comparison (page ledger).
 *
 * Number formats.  E2M1 codes: magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6, bit 3 =
 * sign; byte j of a row holds element 2j in its low nibble and 2j+1 in its
 * high nibble.  E4M3: the OCP "fn" byte (bias 7, largest finite 448).
 *
 * Quantizer (FP32, IEEE round-to-nearest-even, no fused multiply-add):
 *   g     = amax(|x|) / 2688                    per tensor (K and V separately)
 *   sbyte = E4M3_rne_satfinite(amax16 / (6*g))  per 16 consecutive head_dim values
 *   code  = E2M1_rne_satfinite(x / (E4M3(sbyte) * g))
 *   g == 0 -> scale byte 0 and codes 0; a block whose E4M3(sbyte)*g is 0 has
 *   codes 0.  FP8 layers: s8 = amax / 448, byte = E4M3_rne_satfinite(x / s8),
 *   s8 == 0 -> byte 0.
 *
 * Cache layout (one layer, device memory owned by the caller): one contiguous
 * block per (page, KV head), pages outermost: data[num_pages][num_kv_heads][block],
 * block = P * 144 bytes (NVFP4) or P * 256 bytes (FP8) at head_dim 128,
 * P = page_size.  A token at slot s lives at page s / P, offset off = s % P,
 * in group off / 8 (eight consecutive offsets), row r = off % 8.  Groups:
 *   NVFP4 (1152 bytes): [K codes 8 x 64 | K scales 8 x 8 | V codes 8 x 64 |
 *                        V scales 8 x 8]
 *   FP8 (2048 bytes):   [K 8 x 128 | V 8 x 128]
 * K bytes are stored in 16-byte chunks, chunk-major: byte j of row r at
 * (j / 16) * 128 + r * 16 + j % 16 (the K-major core-matrix order of a
 * tensor-core operand, so a staged tile of K codes is an MMA operand as it
 * stands); K scales row-major (block b of row r at r * 8 + b).  V is stored by
 * row pairs (2c, 2c+1), the register layout of a P.V operand (two tokens of
 * one value): NVFP4 code of value d = 16 b + j of row r at byte b * 64 +
 * (r / 2) * 16 + j of the V codes, in the low nibble for even r and the high
 * nibble for odd r; V scales block-major (b * 8 + r); FP8 byte of value
 * 16 b + j at (j / 8) * 512 + b * 64 + (r / 2) * 16 + (j % 8) * 2 + r % 2 of
 * V.  A page of one KV head is one contiguous run of bytes, which decode
 * fetches with a single bulk copy.  The contents are the quantizer's output
 * above; only their positions are fixed here (an NVFP4 V write changes only
 * its own row's nibbles: with atomic byte-lane updates, or with plain stores
 * of both rows of a pair when the call writes both).
 *   Supported: head_dim 128; page_size 16, 32 or 64; every pointer 16-byte
 *   aligned.  Anything else -> NVKV_ERR_UNSUPPORTED.
 *
 * Conventions.  Every call is asynchronous on `stream` (a cudaStream_t, NULL
 * = the legacy default stream) and returns after launching.  Argument errors
 * are found on the host before any launch (nothing is written).  Launch
 * failures return NVKV_ERR_CUDA.  Out-of-range device-side indices (a slot,
 * a block-table entry, a sequence longer than its block-table row) never fault:
 * the element is skipped or clamped and a nonzero code is stored into
 * cache->err_flag when that pointer is non-NULL.  The library allocates no
 * memory; scratch comes from the caller's workspace.  Calls on the same
 * stream are ordered; calls that share a workspace must not overlap.
 */
#ifndef NVFP4KV_H
#define NVFP4KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NVKV_OK = 0,
  NVKV_ERR_INVALID_ARG = 1,
  NVKV_ERR_UNSUPPORTED = 2,
  NVKV_ERR_CUDA = 3,
  NVKV_ERR_WORKSPACE_TOO_SMALL = 4
} nvkv_status;

typedef enum { NVKV_PREC_NVFP4 = 0, NVKV_PREC_FP8_E4M3 = 1 } nvkv_precision;

typedef enum { NVKV_DTYPE_F32 = 0, NVKV_DTYPE_BF16 = 1 } nvkv_dtype;

/* Device error codes written to cache->err_flag (first one wins). */
#define NVKV_DEVERR_SLOT 1       /* slot >= num_pages * page_size            */
#define NVKV_DEVERR_PAGE 2       /* block-table entry outside [0, num_pages) */
#define NVKV_DEVERR_SEQLEN 3     /* seq_len > max_pages * page_size or < 0   */
#define NVKV_DEVERR_TIMEOUT 4    /* a bounded wait inside a kernel ran out   */
#define NVKV_DEVERR_WS_ROWS 5    /* workspace rows smaller than the prefixes */
#define NVKV_DEVERR_ALIGN 6      /* extend: a sequence's first workspace row not a multiple of 8 */

/* One layer's cache.  The struct itself is host memory read during the call. */
typedef struct {
  int32_t prec;                /* nvkv_precision                               */
  int32_t num_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t reserved;
  uint8_t *data;               /* [num_pages][num_kv_heads][block], see above  */
  const float *kv_scale;       /* device float[2] {K, V}: NVFP4 global g, FP8 s8 */
  int32_t *err_flag;           /* optional device int32, 0 = no error          */
} nvkv_cache;

/* Readable name of a status. */
const char *nvkv_status_string(nvkv_status s);

/* Global scale of one tensor ([P2] The Core of the Ledger: "the whole tensor
 * gets one FP32 global scale"): out[0] = max|x[i]| / divisor, FP32 divide.
 * divisor 2688 (= 6 * 448) gives the NVFP4 g, 448 the FP8 s8.  x: n values of
 * `dtype`, device.  out: device float.  n == 0 gives 0.  Three stream operations
 * (a memset and two kernels). */
nvkv_status nvkv_global_scale(const void *x, nvkv_dtype dtype, int64_t n, float divisor, float *out,
                              void *stream);

/* Running maximum for a global scale computed over a tensor stored in pieces:
 * amax[0] = max(amax[0], max|x[i]|).  amax: device float, >= 0, set to 0 by
 * the caller before the first piece; the global scale is then
 * nvkv_global_scale(amax, F32, 1, divisor, out) (division is monotonic, so
 * this equals the scale of the whole tensor). */
nvkv_status nvkv_amax_update(const void *x, nvkv_dtype dtype, int64_t n, float *amax, void *stream);

/* NVFP4 quantized write into paged slots ([P1] 02, the quantized write; [P2]
 * Three Paths: new KV goes into the NVFP4 cache quantized).
 *   k, v          [num_tokens][num_kv_heads][head_dim] of `dtype` (BF16 widens exactly)
 *   slot_mapping  [num_tokens] int64 device; a negative slot skips the token
 *   global_scale  device float[2] {g_K, g_V}; NULL -> cache->kv_scale
 *   cache         prec must be NVKV_PREC_NVFP4
 * Bytes are identical to the quantizer stated at the top of this file. */
nvkv_status nvfp4_kv_quantize_write(const void *k, const void *v, nvkv_dtype dtype, int64_t num_tokens,
                                    const int64_t *slot_mapping, const float *global_scale,
                                    const nvkv_cache *cache, void *stream);

/* Initial-prefill write from FP8 K/V into the NVFP4 cache ([P2] Three Paths:
 * the initial prefill computes on FP8 K/V and requantizes that KV into the
 * NVFP4 cache; it reads no cache, so no dequant round trip).  Each value is
 * decoded with its tensor's FP8 scale, x = E4M3(byte) * in_scale[kind] (one
 * FP32 multiply), then quantized exactly as nvfp4_kv_quantize_write does.
 *   k8, v8        [num_tokens][num_kv_heads][head_dim] E4M3 bytes, device,
 *                 16-byte aligned
 *   in_scale      device float[2] {K, V}: the FP8 per-tensor scales
 *   slot_mapping, global_scale, cache: as nvfp4_kv_quantize_write (the global
 *                 scales are those of the decoded values)
 * One kernel on `stream`. */
nvkv_status nvfp4_kv_requantize_write_fp8(const uint8_t *k8, const uint8_t *v8, const float *in_scale,
                                          int64_t num_tokens, const int64_t *slot_mapping, const float *global_scale,
                                          const nvkv_cache *cache, void *stream);

/* FP8 E4M3 write for the FP8 layers ([P1] 03: sensitive layers keep an FP8 KV
 * cache).  Same arguments; global_scale = per-tensor {s8_K, s8_V}; cache->prec
 * must be NVKV_PREC_FP8_E4M3. */
nvkv_status fp8_kv_quantize_write(const void *k, const void *v, nvkv_dtype dtype, int64_t num_tokens,
                                  const int64_t *slot_mapping, const float *global_scale,
                                  const nvkv_cache *cache, void *stream);

/* Bytes of decode workspace for this problem size: num_splits > 0 as passed to
 * the decode call, 0 for the library's choice on the current device.  The
 * workspace holds a 4-byte arrival counter per (sequence, KV head) (the
 * first batch * num_kv_heads * 4 bytes, rounded up to 256) and then two
 * split-KV partial slots of 4160 bytes per CTA.  The counters must be zero
 * before the first decode call that uses the workspace (zero it once with
 * nvkv_decode_workspace_init or any memset); every call leaves them zero
 * again.  A call that ends with a device error (NVKV_DEVERR_* in the cache's
 * error word, or a CUDA error) can leave them nonzero: zero the workspace
 * again before reusing it.  Returns 0 for unsupported sizes. */
size_t nvkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t num_splits);

/* Zero `bytes` of workspace on `stream` (a cudaMemsetAsync): once before the
 * workspace's first decode call, and after a call that failed on the device. */
nvkv_status nvkv_decode_workspace_init(void *workspace, size_t bytes, void *stream);

/* Paged GQA decode attention over the NVFP4 or FP8 cache ([P2] Three Paths:
 * the decode kernel reads the NVFP4 cache itself and dequantizes inside the
 * kernel; [P1] 03 per-layer precision).
 *   q               [batch][num_q_heads][head_dim] BF16, device
 *   block_table     [batch][max_pages] int32 page ids, device
 *   seq_lens        [batch] int32 visible tokens per sequence (the token written
 *                   in this step included), device; 0 gives a zero output row
 *   layer_precision must equal cache->prec (else NVKV_ERR_INVALID_ARG)
 *   sm_scale        softmax scale; 0 -> 1/sqrt(head_dim)
 *   num_splits      0: balance the work over the GPU (split-KV wherever it
 *                   helps); > 0: cut every sequence into at most that many
 *                   partitions (exactly so when all sequences have equal
 *                   length and batch * num_kv_heads * num_splits CTAs fit on
 *                   the device at once; a larger request is capped there)
 *   workspace       scratch of nvkv_decode_workspace_size(...) bytes, device
 *   out             [batch][num_q_heads][head_dim] BF16, device
 * Query head h reads KV head h / (num_q_heads / num_kv_heads); every token in
 * [0, seq_len) is visible.  out = softmax(q k^T * sm_scale) v with the FP32
 * result rounded to BF16.  Split partitions are merged with the log-sum-exp
 * rule inside the same launch: each contributor of a split (sequence, KV
 * head) counts itself on the pair's counter and the CTA that arrives last
 * merges the parts in contributor order (one kernel launch on `stream`,
 * programmatic dependent launch so its set-up overlaps the previous kernel;
 * the result does not depend on arrival order).  Requires num_q_heads /
 * num_kv_heads <= 8, num_kv_heads >= 1 and batch <= 1024; the CTA count is at
 * most one resident wave and at most 184.  Each CTA streams one contiguous
 * run of 128-token tiles; when batch * num_kv_heads is at least four per CTA
 * the runs are balanced on tiles plus a charge of three tiles per (sequence,
 * KV head) they hold, else on tiles alone.  Calls that share a workspace must
 * be ordered (one stream). */
nvkv_status nvfp4_paged_decode_attention(const void *q, const nvkv_cache *cache, const int32_t *block_table,
                                         int32_t max_pages, const int32_t *seq_lens, int32_t batch,
                                         int32_t num_q_heads, int32_t layer_precision, float sm_scale,
                                         int32_t num_splits, void *workspace, size_t workspace_bytes, void *out,
                                         void *stream);

/* The FP8 E4M3 variant: the same call for a cache with prec == NVKV_PREC_FP8_E4M3. */
nvkv_status fp8_paged_decode_attention(const void *q, const nvkv_cache *cache, const int32_t *block_table,
                                       int32_t max_pages, const int32_t *seq_lens, int32_t batch,
                                       int32_t num_q_heads, float sm_scale, int32_t num_splits, void *workspace,
                                       size_t workspace_bytes, void *out, void *stream);

/* One decode step of a layer in one launch: the quantized write of each
 * sequence's newest token followed by the paged decode attention over the
 * cache that now holds it ([P2] Three Paths: in decode each new token's K/V
 * is quantized into the NVFP4 cache and the decode kernel reads the cache;
 * [P1] 03 per-layer precision).  The result, cache bytes and output, is that
 * of nvfp4_kv_quantize_write (or fp8_kv_quantize_write) of k_new / v_new to
 * the slot of position seq_lens[b] - 1 of each sequence b, i.e. slot
 * block_table[b][(L - 1) / P] * P + (L - 1) % P, with global_scale =
 * cache->kv_scale, then nvfp4_paged_decode_attention with the same arguments;
 * one launch instead of two.  The token is written by the CTA that streams
 * the sequence's last tile, just before it copies the tile.
 *   k_new, v_new  [batch][num_kv_heads][head_dim] of `dtype` (FP32 or BF16),
 *                 device, 16-byte aligned: row b is the newest token of
 *                 sequence b (rows of sequences with seq_lens[b] == 0 are
 *                 not read)
 *   other arguments, workspace contract and errors as for
 *   nvfp4_paged_decode_attention; a page id out of range sets
 *   NVKV_DEVERR_PAGE and that token is not written. */
nvkv_status nvfp4_paged_decode_step(const void *q, const void *k_new, const void *v_new, nvkv_dtype dtype,
                                    const nvkv_cache *cache, const int32_t *block_table, int32_t max_pages,
                                    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                    int32_t layer_precision, float sm_scale, int32_t num_splits, void *workspace,
                                    size_t workspace_bytes, void *out, void *stream);

/* Decode attention that allocates nothing and takes no workspace (no
 * counterpart in the pages: this is a convenience of this library).  For
 * callers that cannot hand out device memory per call: serving engines that
 * give all free HBM to their KV page pool at start-up and keep no allocator
 * for scratch, and plugin hosts that pass a kernel only its input and output
 * pointers.  Same arguments and result as nvfp4_paged_decode_attention without
 * workspace/workspace_bytes; the split-KV scratch lives in a fixed array of
 * NVKV_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the
 * library keeps until the process exits.  The scratch a call needs is a
 * 4-byte arrival counter per (sequence, KV head) (batch * num_kv_heads * 4
 * bytes, rounded up to 256) plus two 4160-byte partial slots per CTA, and the
 * CTA count never exceeds one resident wave (152 on a GB300, 1.27 MB of
 * slots), so on a GB300 every problem with batch * num_kv_heads <= 1,700,000
 * fits (batch <= 1024 as for every decode call; num_kv_heads has no other
 * bound).  A problem whose counters alone exceed the array is refused with
 * NVKV_ERR_WORKSPACE_TOO_SMALL before any CUDA call, and one whose counters
 * and slots together exceed it with the same code before any launch.  Each call first clears its counters with one
 * cudaMemsetAsync on `stream` (so a call after a failed one starts clean), then
 * launches the decode kernel.  The first call on a device looks up the
 * array's device address (set-up, once per device, with that device current);
 * make that first call before any stream capture.  The cached address belongs
 * to the CUDA context it was looked up in: after cudaDeviceReset (or any
 * teardown of the primary context) it is stale, so do not call this entry
 * point again in that process.  All calls share the one array and it keeps
 * the last call's contents, so calls that can overlap on the GPU (different
 * streams, different host threads without ordering) race and give wrong
 * results: order them on one stream.  No cudaMalloc, cudaFree or allocating
 * library routine is called. */
#define NVKV_NOALLOC_SCRATCH_BYTES (8u << 20)
nvkv_status nvfp4_paged_decode_attention_noalloc(const void *q, const nvkv_cache *cache,
                                                 const int32_t *block_table, int32_t max_pages,
                                                 const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                                 int32_t layer_precision, float sm_scale, int32_t num_splits,
                                                 void *out, void *stream);

/* Chunked-extend prefix dequant into the shared FP8 workspace ([P2] Three
 * Paths: for chunked extend the cached prefix is gathered and dequantized into
 * an FP8 workspace shared by all layers).  For i < n, tokens [0, prefix_lens[i]) of sequence
 * seq_ids[i] land in rows cu_prefix[i] + t of ws_k / ws_v, layout
 * [rows][num_kv_heads][head_dim] E4M3:
 *   byte = E4M3_rne_satfinite((e2m1 * S) * (g / ws_scale))   (FP32, per K and V)
 *   seq_ids, prefix_lens  [n] int32 device; each seq_ids[i] must index a row
 *                         of block_table; a prefix longer than its row
 *                         (max_pages * page_size) is skipped and
 *                         NVKV_DEVERR_SEQLEN raised
 *   cu_prefix             [n+1] int64 device: cu_prefix[i] (i < n) is the
 *                         first workspace row of sequence i's prefix; the
 *                         starts are non-decreasing with room for each prefix,
 *                         cu_prefix[i] + prefix_lens[i] <= cu_prefix[i+1], and
 *                         cu_prefix[n] (<= ws_rows) ends the rows the call
 *                         visits.  Rows between one prefix's end and the next
 *                         start are not touched, so a caller can reserve the
 *                         chunk's rows right behind each prefix and start each
 *                         sequence on a multiple of 8 rows, the layout
 *                         fp8_chunked_extend_attention reads ([prefix || chunk]
 *                         per sequence, cu_kv[i] = cu_prefix[i]); the exclusive
 *                         prefix sums of prefix_lens pack the prefixes back to
 *                         back
 *   ws_scale              device float[2] {K, V}, > 0 (e.g. 6 * g)
 *   ws_rows               rows allocated in ws_k and ws_v (host value); rows
 *                         past it are skipped and NVKV_DEVERR_WS_ROWS raised
 * cache->prec must be NVKV_PREC_NVFP4. */
nvkv_status nvfp4_kv_dequant_to_fp8_workspace(const int32_t *block_table, int32_t max_pages,
                                              const int32_t *seq_ids, const int32_t *prefix_lens,
                                              const int64_t *cu_prefix, int32_t n, const nvkv_cache *cache,
                                              const float *ws_scale, uint8_t *ws_k, uint8_t *ws_v,
                                              int64_t ws_rows, void *stream);

/* The current chunk's K/V into the shared FP8 workspace ([P2] Three Paths:
 * the chunk's KV is appended to the dequantized prefix and FP8 attention runs
 * over both).  The pages give no rule for the chunk's bytes; this library
 * uses the FP8 layers' per-tensor quantizer with the workspace scale:
 *   byte = E4M3_rne_satfinite(x / ws_scale)          (FP32 divide, per K and V)
 *   k, v        [num_tokens][num_kv_heads][head_dim] of `dtype`, device,
 *               16-byte aligned; head_dim a multiple of 16
 *   rows        [num_tokens] int64 device: the workspace row of each token
 *               (negative: skipped; >= ws_rows: skipped and
 *               NVKV_DEVERR_WS_ROWS raised in *err_flag, if given)
 *   ws_scale    device float[2] {K, V}, > 0 (the scale the prefix dequant used)
 *   ws_k, ws_v  [ws_rows][num_kv_heads][head_dim] E4M3, device, 16-byte aligned
 * One kernel on `stream`.  Bytes are identical to the oracle's rule above. */
nvkv_status fp8_workspace_append_chunk(const void *k, const void *v, nvkv_dtype dtype, int64_t num_tokens,
                                       const int64_t *rows, int32_t num_kv_heads, int32_t head_dim,
                                       const float *ws_scale, uint8_t *ws_k, uint8_t *ws_v, int64_t ws_rows,
                                       int32_t *err_flag, void *stream);

/* Chunked-extend attention over the shared FP8 workspace ([P2] Three Paths:
 * chunked prefill / extend runs FP8 attention over the dequantized prefix
 * concatenated with the current chunk).  Sequence i (i < n) owns workspace
 * rows [cu_kv[i], cu_kv[i] + kv_lens[i]): positions 0 .. kv_lens[i]-1, prefix
 * first, then the chunk.  Its nq_i = cu_q[i+1] - cu_q[i] queries are the last
 * nq_i positions: query j sits at position kv_lens[i] - nq_i + j and attends
 * to positions [0, that position] (causal inside the chunk).  Query head qh
 * reads KV head qh / (num_q_heads / num_kv_heads).
 *   out = softmax(sm_scale * q . K) V,  K = E4M3(ws_k) * ws_scale[0],
 *                                        V = E4M3(ws_v) * ws_scale[1]
 *   q        [cu_q[n]][num_q_heads][128] BF16, device, 16-byte aligned; used
 *            at FP16 precision (exact for |q| in [2^-14, 65504])
 *   cu_q     [n+1] int64 device, non-decreasing; max_q_len (host) >= every
 *            nq_i (queries beyond it are not computed: NVKV_DEVERR_SEQLEN)
 *   cu_kv    [n] int64 device, each a multiple of 8; kv_lens [n] int32
 *            device, nq_i <= kv_lens[i] and cu_kv[i] + kv_lens[i] <= ws_rows,
 *            else the sequence is skipped and NVKV_DEVERR_ALIGN /
 *            NVKV_DEVERR_SEQLEN / NVKV_DEVERR_WS_ROWS raised
 *   ws_k, ws_v  [ws_rows][num_kv_heads][128] E4M3 (finite bytes), device,
 *            16-byte aligned; ws_scale device float[2] {K, V}
 *   sm_scale <= 0 -> 1/sqrt(128)
 *   scratch  device, 16-byte aligned, >= fp8_extend_scratch_size(ws_rows,
 *            num_kv_heads, 128) bytes (else NVKV_ERR_WORKSPACE_TOO_SMALL):
 *            the workspace expanded once into FP16 operand tiles
 *   out      [cu_q[n]][num_q_heads][128] BF16, device, 16-byte aligned
 *   err_flag optional device int32 (first error code wins)
 * head_dim must be 128 and num_q_heads / num_kv_heads a power of two <= 128
 * (else NVKV_ERR_UNSUPPORTED).  QK^T and P.V run on the tensor cores with
 * FP16 operands (E4M3 converts exactly) and FP32 accumulation; P is rounded
 * to FP16.  Two kernels on `stream` (the tile expansion, the attention); it
 * allocates nothing. */
size_t fp8_extend_scratch_size(int64_t ws_rows, int32_t num_kv_heads, int32_t head_dim);
nvkv_status fp8_chunked_extend_attention(const void *q, const int64_t *cu_q, int32_t n, int32_t max_q_len,
                                         int32_t num_q_heads, const uint8_t *ws_k, const uint8_t *ws_v,
                                         const int64_t *cu_kv, const int32_t *kv_lens, int32_t num_kv_heads,
                                         int32_t head_dim, int64_t ws_rows, const float *ws_scale, float sm_scale,
                                         void *scratch, size_t scratch_bytes, void *out, int32_t *err_flag,
                                         void *stream);

/* Page ledger and page pool (host functions, no GPU work).  [P2] The Core of
 * the Ledger: 16 values take 9 bytes in NVFP4 and 16 in FP8, so the same KV
 * memory holds more sequences.  Every layer's cache is indexed by the same
 * page ids, so a KV budget buys
 *   pages = floor(budget / sum_l nvkv_cache_page_bytes(prec_l, ...))
 * and a sequence of L tokens holds ceil(L / page_size) pages.
 *   nvkv_cache_page_bytes       one page of one layer's cache (all KV heads):
 *                               page_size * Hkv * (NVFP4: head_dim * 9/8 * 2;
 *                               FP8: head_dim * 2); 0 for bad arguments
 *   nvkv_pool_pages_for_budget  pages for `budget_bytes` under the per-layer
 *                               precision map layer_prec[num_layers]; -1 for
 *                               bad arguments
 * The pool hands out page ids 0 .. num_pages-1 (lowest first when fresh; a
 * released page is the next one handed out) and is not thread-safe.
 *   nvkv_pool_create   NULL if num_pages < 0 or out of host memory
 *   nvkv_pool_alloc    n pages into out[n], all or nothing: returns n, or -1
 *                      (nothing taken) when fewer than n are free
 *   nvkv_pool_release  returns pages to the pool; a page not held, out of
 *                      range or listed twice -> NVKV_ERR_INVALID_ARG and
 *                      nothing released */
typedef struct nvkv_page_pool nvkv_page_pool;
size_t nvkv_cache_page_bytes(int32_t prec, int32_t page_size, int32_t num_kv_heads, int32_t head_dim);
int32_t nvkv_pool_pages_for_budget(size_t budget_bytes, const int32_t *layer_prec, int32_t num_layers,
                                   int32_t page_size, int32_t num_kv_heads, int32_t head_dim);
nvkv_page_pool *nvkv_pool_create(int32_t num_pages);
void nvkv_pool_destroy(nvkv_page_pool *pool);
int32_t nvkv_pool_num_free(const nvkv_page_pool *pool);
int32_t nvkv_pool_alloc(nvkv_page_pool *pool, int32_t n, int32_t *out);
nvkv_status nvkv_pool_release(nvkv_page_pool *pool, const int32_t *pages, int32_t n);

/* Element encoders of the quantizer, one output byte per FP32 input: E2M1
 * code (low nibble, round-to-nearest-even, saturating at 6) and E4M3 byte
 * (round-to-nearest-even, saturating at 448).  x, out: device. */
nvkv_status nvkv_encode_e2m1(const float *x, int64_t n, uint8_t *out, void *stream);
nvkv_status nvkv_encode_e4m3(const float *x, int64_t n, uint8_t *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4KV_H */
