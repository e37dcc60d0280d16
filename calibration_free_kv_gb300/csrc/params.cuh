// Launch parameters of the KVarN kernels, shared by the kernels and the C-ABI layer.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "kvarn.h"

namespace kvarn {

struct QuantizeParams {
  // tile mode
  const __half* k;
  const __half* v;
  int64_t tok_stride;
  int64_t head_stride;
  const int32_t* page_ids;
  // append mode
  const __half* k_new;
  const __half* v_new;
  __half* partial_k;
  __half* partial_v;
  const int32_t* seq_lens;
  int32_t* seq_lens_out;
  const int32_t* block_table;
  int max_pages;
  // common
  uint8_t* pool;
  int64_t num_pool_pages;
  int64_t rec_bytes;
  int num_kv_heads;
  int d0;
  int iters;
  float eps;
  // early stop: after an iteration in which every std step's sigma stayed within
  // [tol_lo, tol_hi] = [e^-tol, e^tol]; tol_hi == 0 disables it
  float tol_lo, tol_hi;
  int32_t* iters_out;  // iterations used per unit [tile][head][K, V], or null
  int32_t* status;
  int append;  // 0: quantise whole tiles, 1: append one token and seal full tiles
};

struct DecodeParams {
  const __half* q;
  const uint8_t* pool;
  int64_t num_pool_pages;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  const __half* partial_k;
  const __half* partial_v;
  float qscale;  // softmax_scale * log2(e)
  __half* out;
  float* part;   // [batch][chunk][Hq][max_splits][D + 4]: m, l, -, -, o~[D]
  int batch, num_kv_heads, num_q_heads, group, d0;
  int pages_per_split, max_splits;
  // Prefill: `chunk` query tokens per sequence (1 for decode), q / out [batch][chunk][Hq][d0].
  // The chunk * group query vectors of a kv head are split into `vgroups` CTAs of up to
  // 4 * NT each; chunk_k / chunk_v [batch][chunk][Hkv][d0] (NULL for decode) are attended
  // causally by the chunk kernel, whose partial is the split after the cache's.
  int chunk, vgroups;
  const __half* chunk_k;
  const __half* chunk_v;
  int32_t* status;
  // Persistent decode (decode_kernel with part_mode 1, or decode_tc.cu): 0, or the CTAs the
  // balanced page partition of the sealed pages is cut for (decode_util.cuh).  When set, the
  // sealed pages' partials of row (b, kv head) fill splits [0, row_segments) and decode_kernel
  // with part_mode 2, launched over (1, Hkv, batch), writes the partial tile's split after them.
  int part_ctas;
  // 1: the merge kernel attends to the raw partial tiles itself (decode); decode_kernel and the
  // tcgen05 kernel then leave them alone and no split holds them
  int partial_in_merge;
  int part_mode;  // 0: one CTA per split (grid splits x Hkv*vgroups x batch); 1: persistent
                  // CTAs over the partition's sealed pages; 2: partial tiles only; 3: the
                  // tcgen05 kernel over the sealed pages
};

struct DequantParams {
  const uint8_t* pool;
  int64_t num_pool_pages;
  const int32_t* page_ids;
  __half* k_out;
  __half* v_out;
  int num_kv_heads;
  int d0;
  int32_t* status;
  // error telemetry (err_out non-null): the fp16 tiles the records were quantised from, laid
  // out as kvarn_quantize_tiles' inputs, and four floats per (tile, kv head, K or V)
  const __half* k_src;
  const __half* v_src;
  int64_t tok_stride, head_stride;
  float* err_out;
};

// decode_args_check: a valid decode call with nothing to launch (batch 0).
constexpr int kDecodeNothingToDo = 1;
// Host-side checks of a decode call's arguments other than its workspace (kvarn_api.cu):
// KVARN_OK, kDecodeNothingToDo or a KVARN_ERR_* code.
int decode_args_check(const kvarn_desc* desc, int batch, int num_q_heads, const void* q,
                      const void* page_pool, int64_t num_pool_pages, const int32_t* block_table,
                      int max_pages, const int32_t* seq_lens, const void* partial_k,
                      const void* partial_v, float softmax_scale, const void* out);

int launch_quantize_any(int d, int kb, int vb, const QuantizeParams& p, int units, cudaStream_t stream);
// Kernels of a decode launch: the split partials (decode_kernel), the merge (combine_kernel).
constexpr int kDecodeSplits = 1, kDecodeMerge = 2;
int launch_decode_any(int d, int nt, int kb, int vb, const DecodeParams& p, cudaStream_t stream,
                      int phases = kDecodeSplits | kDecodeMerge);
// Sealed pages per decode CTA for `units` (sequence, kv head, vector group) rows of a block
// table `max_pages` wide: 32, or for tables over 256 pages the size in [32, 128] that fills
// the GPU's CTA slots best.  Never below 32, the size the workspace is laid out for.
int decode_split_pages(int d, int nt, int kb, int vb, int64_t units, int max_pages);
int launch_chunk_any(int d, const DecodeParams& p, cudaStream_t stream);
// The tcgen05 decode of GQA groups of 8 at head_dim 128, K4V2 (decode_tc.cu): whether it
// serves this launch, its CTA count, and the launch of the phases requested.
bool decode_tc_serves(int d, int nt, int kb, int vb, const DecodeParams& p);
int decode_tc_ctas();
int launch_decode_tc(const DecodeParams& p, int phases, cudaStream_t stream);
// decode_kernel<128, 2, 4, 2> over (1, Hkv, batch) for the partial tiles of a tcgen05 launch
int launch_decode_partial_tiles(const DecodeParams& p, cudaStream_t stream);
// CTAs of the persistent mma.sync decode for this shape (SMs x CTAs per SM), 0 on error.
int decode_persistent_ctas(int d, int nt, int kb, int vb);
int launch_decode_combine(int d, const DecodeParams& p, cudaStream_t stream);
int launch_dequant_any(int d, int kb, int vb, const DequantParams& p, int num_pages, cudaStream_t stream);

}  // namespace kvarn
