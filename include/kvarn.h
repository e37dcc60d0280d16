/*
 * kvarn.h -- C ABI of the KVarN K4V2 g128 KV-cache path (and the other k/v bit presets) for
 * GB300 (sm_103a).
 *
 * What is computed (sources cited by page title and section):
 *  - [hotdry]  blog.hotdry.top "KVarN Hadamard 旋转与方差归一化：KV-cache 量化的校准算法实现"
 *  - [aifeeds] ai-feeds.com "KVarN: 方差归一化的KV-Cache量化缓解推理任务中的误差累积"
 *  - [vatt]    vatt-ghern.pages.dev "KV cache 為什麼能壓到 4-bit／2-bit 還不掉準確度——從
 *              variance normalization 講起"
 *
 * Every 128-token tile of every KV head is (1) zero-padded along head_dim to the next power of
 * two d [aifeeds §局限], (2) rotated along head_dim by the orthonormal Sylvester Hadamard
 * H_d / sqrt(d) [hotdry §Hadamard 旋转], (3) variance-normalised by alternating channel-std and
 * token-std steps whose factors live in log space, for a fixed iteration count (or fewer,
 * with kvarn_quantize_tiles_adaptive) [hotdry §迭代方差归一化; vatt §四個步驟], (4) quantised
 * by asymmetric round-to-nearest, keys to 4 bits per channel and values to 2 bits per token
 * (other presets: other widths, same steps [vatt §四個步驟, bit-width assignment]), with the
 * normalisation factors folded into the stored fp16 scales [hotdry §非对称量化与尺度折叠].  Decode attention reads the packed cache
 * directly [vatt §怎麼用: one paged-attention block == one tile; attention computed in fp16
 * over the quantised cache].
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library allocates
 *    nothing, keeps no per-call state, never synchronises and launches on `stream`
 *    (a cudaStream_t passed as void*; NULL = legacy default stream).
 *  - fp16 means IEEE binary16; all tensors are little-endian and row-major.
 *  - Return value: KVARN_OK (0) or a negative KVARN_ERR_* code.  Argument errors are found
 *    on the host before any launch.  Errors that depend on device data (a page id outside
 *    the pool, a seq_len above the block-table capacity, a copy that did not arrive) are
 *    OR-ed as KVARN_DEV_* bits into *dev_status when dev_status is non-NULL (a device
 *    int32 the caller zeroes and reads); the kernels then clamp to in-bounds data and
 *    never trap.
 *  - head_dim d0: 40..256 and a multiple of 8; it is padded to the next power of two,
 *    d = 64, 128 or 256 [aifeeds §局限].  d0 <= 32 would pad to 8, 16 or 32, widths that have
 *    no page record layout, and is refused (KVARN_ERR_UNSUPPORTED).
 *  - GQA: query head hq reads KV head hq / G, G = num_q_heads / num_kv_heads in {1,2,4,8}.
 *
 * Page record: the packed K/V of one (page, kv head), record_bytes bytes, 16-byte aligned
 * sections.  The page pool is [num_pool_pages][num_kv_heads][record_bytes]; record (p, h)
 * starts at byte ((p * num_kv_heads) + h) * record_bytes.  With T = 128 and kb / vb the K / V
 * code bits (4 / 2 for kvarn_k4v2_g128):
 *    K codes  T*d*kb/8 B   uint32 words
 *    K scale s'[d], K zero z'[d], K token factor r[T]            (fp16)
 *    V codes  T*d*vb/8 B   uint32 words
 *    V scale s'[T], V zero z'[T], V channel factor c[d]          (fp16)
 * (the K half precedes the V half, so each can be fetched alone).
 * Dequantised rotated-domain values: K~[t][j] = r[t] (code*s'[j] + z'[j]),
 * V~[t][j] = c[j] (code*s'[t] + z'[t]); original basis = rows of (.) H_d / sqrt(d), first d0.
 * Code words carry m16n8k16 A-operand fragments of 16 x 16 blocks: K as [token x channel],
 * V transposed as [channel x token]; lane = 4g + tq, element (rho, h, p) of a fragment is at
 * row g + 8rho, column 8h + 2tq + p of its block.  Blocks (o, i): o = token block (< 8),
 * i = channel block (< d/16).
 *  4-bit: word ((o*(d/64) + i/4)*32 + lane)*4 + i%4 is fragment (o, i), element (rho, h, p)
 *         at nibble h + 2rho + 4p.
 *  2-bit: word ((o/2*(d/64) + i/4)*32 + lane)*4 + i%4 holds fragments (o, i) of both token
 *         blocks o of a pair, element (rho, h, p) at 2-bit slot 2(o%2) + h + 4rho + 8p.
 *  8-bit: words ((o*(d/32) + i/2)*32 + lane)*4 + 2(i%2) + h, h = 0, 1, hold fragment (o, i),
 *         element (rho, h, p) at byte rho + 2p of word h.
 * For kvarn_k4v2_g128 K word (mi, kk, lane) holds token 16mi + g + 8rho, channel
 * 16kk + 8h + 2tq + p at nibble h + 2rho + 4p; V word (ks2, mc, lane) holds channel
 * 16mc + g + 8rho, token 16(2ks2 + f) + 8h + 2tq + p at slot 2f + h + 4rho + 8p.
 * record_bytes (d = 128 / 256): kvarn_k4v2_g128 13824 / 26880, kvarn_k4v4_g128 17920 / 35072,
 * kvarn_k2v2_g128 9728 / 18688, kvarn_k8v4_g128 26112 / 51456.
 */
#ifndef KVARN_H
#define KVARN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVARN_OK 0
#define KVARN_ERR_INVALID_ARG (-1)          /* NULL pointer, bad size/stride/alignment      */
#define KVARN_ERR_UNSUPPORTED (-2)          /* preset, head_dim, bits, tile or GQA group    */
#define KVARN_ERR_WORKSPACE_TOO_SMALL (-3)  /* decode workspace below the required size     */
#define KVARN_ERR_CUDA (-4)                 /* a CUDA launch or attribute call failed       */

#define KVARN_DEV_BAD_PAGE_ID 1      /* a page id outside [0, num_pool_pages): page 0 used   */
#define KVARN_DEV_SEQ_TOO_LONG 2     /* seq_len < 0, or its pages exceed the block table row  */
#define KVARN_DEV_WAIT_TIMEOUT 4     /* an asynchronous page copy did not arrive in ~2 s     */
#define KVARN_DEV_NO_PARTIAL 8       /* a length has a remainder but partial_k/v were NULL   */

/* Method constants of one cache.  Fill it with kvarn_desc_from_preset. */
typedef struct kvarn_desc {
  int32_t head_dim;          /* d0, true head_dim                                   */
  int32_t head_dim_padded;   /* d = 64, 128 or 256                                  */
  int32_t num_kv_heads;      /* Hkv                                                 */
  int32_t tile_tokens;       /* 128 (one tile == one page) [vatt §怎麼用 knob table]  */
  int32_t k_bits;            /* 4 (kvarn_k4v2_g128, kvarn_k4v4_g128), 2 or 8        */
  int32_t v_bits;            /* 2 (kvarn_k4v2_g128, kvarn_k2v2_g128) or 4           */
  int32_t sinkhorn_iters;    /* 4 (0..8 accepted)                                   */
  float sinkhorn_eps;        /* 1e-6, floor of a std before its log                 */
  int64_t page_record_bytes; /* bytes of one (page, kv head) record                 */
} kvarn_desc;

/* Fill *out for a preset: "kvarn_k4v2_g128" [hotdry §核心配置参数: kv_cache_dtype
 * kvarn_k4v2_g128, block_size 128], or "kvarn_k4v4_g128" / "kvarn_k2v2_g128" /
 * "kvarn_k8v4_g128" (other k/v bit presets through the same pipeline [vatt §四個步驟,
 * bit-width assignment]).  Host only.
 * UNSUPPORTED for another name or a head_dim outside 40..256 / not a multiple of 8;
 * INVALID_ARG for NULL or Hkv < 1. */
int kvarn_desc_from_preset(const char* preset, int head_dim, int num_kv_heads, kvarn_desc* out);

/* Bytes of one page record for this descriptor (host only). */
int64_t kvarn_page_record_bytes(const kvarn_desc* desc);

/* Quantise whole 128-token tiles into page records [hotdry §Hadamard 旋转 to
 * §非对称量化与尺度折叠].
 *  k, v        fp16; element (token t, kv head h, channel c < d0) at [t*tok_stride +
 *              h*head_stride + c]; tile i covers tokens 128i .. 128i+127.  Base 16-byte
 *              aligned, tok_stride and head_stride multiples of 8 (elements).
 *  page_ids    device int32 [num_tiles]: tile i is written to record (page_ids[i], h).
 *  page_pool   device, num_pool_pages pages (see the layout above); written.
 * num_tiles == 0 is a no-op. */
int kvarn_quantize_tiles(const kvarn_desc* desc, const void* k, const void* v, int64_t tok_stride,
                         int64_t head_stride, int num_tiles, const int32_t* page_ids,
                         void* page_pool, int64_t num_pool_pages, int32_t* dev_status,
                         void* stream);

/* kvarn_quantize_tiles with an early stop of the normalisation and per-unit telemetry
 * [hotdry §迭代方差归一化: three to five iterations typical; vatt §四個步驟, Sinkhorn paragraph:
 * alternate until both directions balance].
 *  sinkhorn_tol  >= 0 (and <= 10).  0: always desc->sinkhorn_iters iterations, identical to
 *                kvarn_quantize_tiles.  > 0: a unit (tile, head, K or V) stops after the
 *                first iteration in which no std step moved a log factor by more than
 *                sinkhorn_tol (every sigma within [e^-tol, e^tol]), at most sinkhorn_iters.
 *  iters_used    device int32 [num_tiles][Hkv][2] (K, V) or NULL: iterations each unit used.
 * Other arguments, layout and errors as kvarn_quantize_tiles; INVALID_ARG for a negative,
 * NaN or too large sinkhorn_tol. */
int kvarn_quantize_tiles_adaptive(const kvarn_desc* desc, const void* k, const void* v,
                                  int64_t tok_stride, int64_t head_stride, int num_tiles,
                                  const int32_t* page_ids, void* page_pool, int64_t num_pool_pages,
                                  float sinkhorn_tol, int32_t* iters_used, int32_t* dev_status,
                                  void* stream);

/* Append one decode token per sequence and seal full tiles (tile filling implied by paging:
 * vatt §怎麼用, one block == one tile).
 *  k_new, v_new          fp16 [batch][Hkv][d0].
 *  partial_k, partial_v  fp16 [batch][Hkv][128][d0]: the unsealed tile of each sequence.
 *  seq_lens              device int32 [batch], length BEFORE this token, < max_pages*128
 *                        (else the sequence is skipped and flagged).  The token goes to
 *                        row seq_lens[b] % 128 of the partial tile; when that row is 127 the
 *                        tile is quantised into record (block_table[b][seq_lens[b]/128], h),
 *                        bit-identical to kvarn_quantize_tiles on the same 128 tokens.
 *  seq_lens_out          device int32 [batch] or NULL: receives seq_lens[b] + 1.  Must not
 *                        alias seq_lens.
 *  block_table           device int32 [batch][max_pages]. */
int kvarn_append_token(const kvarn_desc* desc, int batch, const void* k_new, const void* v_new,
                       void* partial_k, void* partial_v, const int32_t* seq_lens,
                       int32_t* seq_lens_out, const int32_t* block_table, int max_pages,
                       void* page_pool, int64_t num_pool_pages, int32_t* dev_status,
                       void* stream);

/* Workspace bytes kvarn_decode_attention needs for this batch shape (host only): fp32 split
 * partials, ceil(max_pages / 32) + 2 per query row.  The mma.sync kernels fill one per split
 * of 32 or more pages (a block table wider than 256 pages may take larger splits, chosen from
 * the GPU's SM count) plus the raw partial tile's; the persistent kernels (the default, and the
 * tcgen05 kernel of GQA groups of 8 at head_dim 128, K4V2) lay the sealed pages of the batch on a
 * line where each row with pages first takes 8 units for a segment's fixed work, then one unit per
 * page, and cut it into ranges of equal length, each at least 32 units, so that a row's pages fall
 * in at most ceil(n / 32) + 1 ranges.  Needs no GPU.  Two environment variables (read on every
 * call) pick the decode kernels for comparing them: KVARN_DECODE_KERNEL "split" (one CTA per split
 * of 32 or more pages) or "tc" (GQA 8, head_dim 128, K4V2: the tcgen05 kernel); by default
 * persistent CTAs take those ranges.  KVARN_DECODE_OPEN_TILES "split" attends to the raw partial
 * tiles in the decode kernels as splits of their own; by default the merge kernel does. */
size_t kvarn_decode_workspace_bytes(const kvarn_desc* desc, int batch, int num_q_heads,
                                    int max_pages);

/* One decode step of attention over the packed cache [vatt §一次 16K context…: decode reads
 * the whole cache each step; §四個步驟: the rotation keeps q.k unchanged].
 *  q            fp16 [batch][Hq][d0] (one query per sequence and head).
 *  block_table  device int32 [batch][max_pages], seq_lens device int32 [batch]: TOTAL length,
 *               i.e. seq_lens[b]/128 sealed pages plus seq_lens[b]%128 raw tokens in the
 *               partial tile; seq_lens[b]/128 <= max_pages (else clamped and flagged).
 *  partial_k/v  fp16 [batch][Hkv][128][d0] as for kvarn_append_token (16-byte aligned, else
 *               INVALID_ARG); may be NULL only if no length has a remainder.
 *  softmax_scale  tau in softmax(tau q.k).
 *  out          fp16 [batch][Hq][d0]; a sequence of length 0 gives zeros.
 *  workspace    device scratch of at least kvarn_decode_workspace_bytes (16-byte aligned). */
int kvarn_decode_attention(const kvarn_desc* desc, int batch, int num_q_heads, const void* q,
                           const void* page_pool, int64_t num_pool_pages,
                           const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                           const void* partial_k, const void* partial_v, float softmax_scale,
                           void* out, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream);

/* kvarn_decode_attention in two launches, for callers that schedule the merge themselves (or
 * time the two kernels apart): kvarn_decode_partials runs the page splits and leaves their
 * partials (m, l, unnormalised output, rotated basis) in the workspace; kvarn_decode_combine,
 * called with the same arguments after it on the same stream (the workspace untouched in
 * between), merges them and writes `out`.  The pair gives the same bytes as
 * kvarn_decode_attention; arguments, checks and errors are those of kvarn_decode_attention
 * (each call checks them all; only decode_combine writes `out`, only decode_partials reads
 * the page pool and the partial tiles). */
int kvarn_decode_partials(const kvarn_desc* desc, int batch, int num_q_heads, const void* q,
                          const void* page_pool, int64_t num_pool_pages,
                          const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                          const void* partial_k, const void* partial_v, float softmax_scale,
                          void* out, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream);
int kvarn_decode_combine(const kvarn_desc* desc, int batch, int num_q_heads, const void* q,
                         const void* page_pool, int64_t num_pool_pages,
                         const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                         const void* partial_k, const void* partial_v, float softmax_scale,
                         void* out, void* workspace, size_t workspace_bytes,
                         int32_t* dev_status, void* stream);

/* Size of the fixed device buffer used by kvarn_decode_attention_noalloc (16 MiB). */
#define KVARN_DECODE_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* Workspace bytes kvarn_prefill_attention needs for this shape (host only; 0 if invalid). */
size_t kvarn_prefill_workspace_bytes(const kvarn_desc* desc, int batch, int num_q_heads,
                                     int chunk_len, int max_pages);

/* Chunked-prefill attention: a chunk of chunk_len new tokens per sequence attends to the
 * packed cache and, causally, to itself (the step before decode; the cache side reads the
 * same packed pages as decode [vatt §怎麼用: one block == one tile]).  Query token c of
 * sequence b attends to the cache_lens[b] cached tokens (sealed pages + raw partial tile)
 * and to chunk tokens 0..c.
 *  q            fp16 [batch][chunk_len][Hq][d0];  out fp16 [batch][chunk_len][Hq][d0].
 *  chunk_k/v    fp16 [batch][chunk_len][Hkv][d0], 16-byte aligned: the chunk's own keys and
 *               values (raw; quantise them into the cache afterwards with kvarn_quantize_tiles /
 *               kvarn_append_token).
 *  cache_lens   device int32 [batch]: cached tokens before the chunk (as seq_lens of decode).
 *  Other arguments as kvarn_decode_attention; workspace >= kvarn_prefill_workspace_bytes.
 *  UNSUPPORTED if chunk_len * G / 8 (/ 4 at head_dim 256) * Hkv exceeds 65535. */
int kvarn_prefill_attention(const kvarn_desc* desc, int batch, int num_q_heads, int chunk_len,
                            const void* q, const void* chunk_k, const void* chunk_v,
                            const void* page_pool, int64_t num_pool_pages,
                            const int32_t* block_table, int max_pages, const int32_t* cache_lens,
                            const void* partial_k, const void* partial_v, float softmax_scale,
                            void* out, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, void* stream);

/* kvarn_decode_attention without a workspace argument, for callers that cannot allocate
 * device memory: plugins in engines that plan and own all device memory in advance, code
 * that must not call cudaMalloc on the decode path (it may synchronise the device), and
 * embedders without an allocator.  The pages have no counterpart; this is an interface
 * variant of the decode call above, with identical arguments, results and errors otherwise.
 *  - The split partials live in a library-owned buffer of
 *    KVARN_DECODE_NOALLOC_SCRATCH_BYTES per GPU, held from the library's load until exit.
 *    A shape whose kvarn_decode_workspace_bytes exceeds it returns
 *    KVARN_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 *  - Arguments are checked first, with the same results as kvarn_decode_attention (an
 *    empty batch returns KVARN_OK without touching the GPU).  Then the first call on each
 *    device looks up the buffer's device address (cudaGetSymbolAddress) with that device
 *    current; make that first call before any stream capture.  The address is kept until
 *    the process exits: do not use this entry point on a device after cudaDeviceReset on it.
 *    The current device must own stream and pointers.
 *  - All calls on a device share the buffer and it keeps the last call's contents; nothing
 *    in it needs to start at zero.  Calls that overlap on the GPU (other streams, other
 *    threads) race on it: order them on one stream or serialise them. */
int kvarn_decode_attention_noalloc(const kvarn_desc* desc, int batch, int num_q_heads,
                                   const void* q, const void* page_pool, int64_t num_pool_pages,
                                   const int32_t* block_table, int max_pages,
                                   const int32_t* seq_lens, const void* partial_k,
                                   const void* partial_v, float softmax_scale, void* out,
                                   int32_t* dev_status, void* stream);

/* Dequantise page records back to fp16 K/V in the original basis [hotdry
 * §非对称量化与尺度折叠: scales multiplied back at read].
 *  page_ids  device int32 [num_pages]; k_out, v_out fp16 [num_pages][Hkv][128][d0]. */
int kvarn_dequantize_tiles(const kvarn_desc* desc, const void* page_pool, int64_t num_pool_pages,
                           const int32_t* page_ids, int num_pages, void* k_out, void* v_out,
                           int32_t* dev_status, void* stream);

/* Quantisation-error telemetry: page records checked against the fp16 tiles they were
 * quantised from [hotdry §监控要点: sample the dequantised values periodically and watch the
 * quantisation error].  Tiles and pages are given as to kvarn_quantize_tiles (the same k, v,
 * strides, num_tiles and page_ids; pass a subset of the tiles to sample).  For each tile i,
 * kv head h and half (0 = K, 1 = V) it writes four floats at err_stats[((i*Hkv + h)*2 + half)*4]:
 *    sum over the 128 x d0 values of (x - x^)^2,   sum of x^2,   max |x - x^|,   max |x|
 * with x the fp16 source value and x^ the record's dequantised value in the original basis
 * (float32, before the fp16 rounding of kvarn_dequantize_tiles).  The relative Frobenius error
 * of the unit is sqrt(first / second).
 *  err_stats  device float [num_tiles][Hkv][2][4], 16-byte aligned.
 * Reads the records and the source tiles once; launches one kernel. */
int kvarn_quantization_error(const kvarn_desc* desc, const void* k, const void* v,
                             int64_t tok_stride, int64_t head_stride, int num_tiles,
                             const int32_t* page_ids, const void* page_pool, int64_t num_pool_pages,
                             float* err_stats, int32_t* dev_status, void* stream);

/* ---- Uncompressed fp16 paged decode: the baseline the packed cache is measured against ----
 * [hotdry §监控要点: throughput is judged against fp16 KV caches; vatt §一次 16K context…:
 *  every decode step reads every cached byte].  Same paging (128-token pages, block table,
 *  seq_lens), split-K and merge as kvarn_decode_attention, no quantisation, no rotation.
 *  Page record per (page, kv head): fp16 K rows then V rows, [2][128][head_dim], records laid
 *  out [num_pool_pages][Hkv]; a length L uses ceil(L/128) pages, rows past L of the last page
 *  are never read.  head_dim 64 or 128 (else UNSUPPORTED); G = Hq/Hkv in {1, 2, 4, 8}. */

/* Bytes of one fp16 (page, kv head) record: 2 * 128 * head_dim * 2 (0 if unsupported). */
size_t kvarn_fp16_page_bytes(int head_dim);

/* Workspace bytes kvarn_fp16_decode_attention needs (host only; 0 if invalid). */
size_t kvarn_fp16_decode_workspace_bytes(int head_dim, int batch, int num_q_heads, int max_pages);

/*  q            fp16 [batch][Hq][head_dim] (4-byte aligned); out fp16 [batch][Hq][head_dim].
 *  page_pool    16-byte aligned; block_table device int32 [batch][max_pages]; seq_lens device
 *               int32 [batch] with ceil(L/128) <= max_pages (else clamped, KVARN_DEV_SEQ_TOO_LONG).
 *  softmax_scale  tau in softmax(tau q.k); a sequence of length 0 gives zeros.
 *  Device-side problems are OR-ed into *dev_status as for kvarn_decode_attention. */
int kvarn_fp16_decode_attention(int head_dim, int num_kv_heads, int batch, int num_q_heads,
                                const void* q, const void* page_pool, int64_t num_pool_pages,
                                const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                                float softmax_scale, void* out, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream);

/* Self-test of the kernels' bounded waits: one thread waits on an mbarrier that nothing
 * completes; after ~2 s the wait gives up and KVARN_DEV_WAIT_TIMEOUT is OR-ed into
 * *dev_status (device int32, required).  Launches on `stream` and returns; the GPU context
 * stays usable.  INVALID_ARG if dev_status is NULL. */
int kvarn_selftest_wait_timeout(int32_t* dev_status, void* stream);

/* Static description of a KVARN_OK / KVARN_ERR_* code. */
const char* kvarn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* KVARN_H */
