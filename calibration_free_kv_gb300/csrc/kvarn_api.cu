// C ABI of the KVarN kernels: argument validation, launch configuration, status codes.
// Nothing here allocates, synchronises or keeps state between calls.
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "params.cuh"

using namespace kvarn;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The presets: name -> K and V code bits, 128-token tiles.  kvarn_k4v2_g128 is the one the
// pages ship; other k/v bit presets run the same pipeline [vatt §四個步驟, bit-width
// assignment].
struct Preset {
  const char* name;
  int k_bits, v_bits;
};
constexpr Preset kPresets[] = {
    {"kvarn_k4v2_g128", 4, 2}, {"kvarn_k4v4_g128", 4, 4}, {"kvarn_k2v2_g128", 2, 2},
    {"kvarn_k8v4_g128", 8, 4}};

bool supported_bits(int kb, int vb) {
  for (const Preset& pr : kPresets)
    if (pr.k_bits == kb && pr.v_bits == vb) return true;
  return false;
}

// Next power of two >= d0 [aifeeds §局限: a head_dim that is not a power of two is padded up to
// the nearest one].
int padded_dim(int d0) {
  int d = 1;
  while (d < d0) d *= 2;
  return d;
}

// head_dim 40..256 in steps of 8: padded to 64, 128 or 256, the widths a page record exists for
// (its code words tile 64-channel groups).  head_dim <= 32 would pad to itself (8, 16, 32) and
// is refused.
bool supported_head_dim(int d0) { return d0 > 32 && d0 <= 256 && d0 % 8 == 0; }

int check_desc(const kvarn_desc* d) {
  if (d == nullptr) return KVARN_ERR_INVALID_ARG;
  if (d->tile_tokens != kTile || !supported_bits(d->k_bits, d->v_bits)) return KVARN_ERR_UNSUPPORTED;
  if (!supported_head_dim(d->head_dim)) return KVARN_ERR_UNSUPPORTED;
  if (d->head_dim_padded != padded_dim(d->head_dim)) return KVARN_ERR_UNSUPPORTED;
  if (d->num_kv_heads < 1) return KVARN_ERR_INVALID_ARG;
  if (d->sinkhorn_iters < 0 || d->sinkhorn_iters > 8) return KVARN_ERR_UNSUPPORTED;
  if (!(d->sinkhorn_eps > 0.0f)) return KVARN_ERR_INVALID_ARG;
  if (d->page_record_bytes != record_layout(d->head_dim_padded, d->k_bits, d->v_bits).bytes)
    return KVARN_ERR_INVALID_ARG;
  return KVARN_OK;
}

}  // namespace

extern "C" {

int kvarn_desc_from_preset(const char* preset, int head_dim, int num_kv_heads, kvarn_desc* out) {
  if (preset == nullptr || out == nullptr) return KVARN_ERR_INVALID_ARG;
  const Preset* pr = nullptr;
  for (const Preset& c : kPresets)
    if (std::strcmp(preset, c.name) == 0) pr = &c;
  if (pr == nullptr) return KVARN_ERR_UNSUPPORTED;
  if (!supported_head_dim(head_dim)) return KVARN_ERR_UNSUPPORTED;
  if (num_kv_heads < 1) return KVARN_ERR_INVALID_ARG;
  kvarn_desc d;
  d.head_dim = head_dim;
  d.head_dim_padded = padded_dim(head_dim);
  d.num_kv_heads = num_kv_heads;
  d.tile_tokens = kTile;
  d.k_bits = pr->k_bits;
  d.v_bits = pr->v_bits;
  d.sinkhorn_iters = 4;
  d.sinkhorn_eps = 1e-6f;
  d.page_record_bytes = record_layout(d.head_dim_padded, d.k_bits, d.v_bits).bytes;
  *out = d;
  return KVARN_OK;
}

int64_t kvarn_page_record_bytes(const kvarn_desc* desc) {
  if (check_desc(desc) != KVARN_OK) return -1;
  return desc->page_record_bytes;
}

int kvarn_quantize_tiles(const kvarn_desc* desc, const void* k, const void* v, int64_t tok_stride,
                         int64_t head_stride, int num_tiles, const int32_t* page_ids,
                         void* page_pool, int64_t num_pool_pages, int32_t* dev_status,
                         void* stream) {
  return kvarn_quantize_tiles_adaptive(desc, k, v, tok_stride, head_stride, num_tiles, page_ids,
                                       page_pool, num_pool_pages, 0.0f, nullptr, dev_status, stream);
}

int kvarn_quantize_tiles_adaptive(const kvarn_desc* desc, const void* k, const void* v,
                                  int64_t tok_stride, int64_t head_stride, int num_tiles,
                                  const int32_t* page_ids, void* page_pool, int64_t num_pool_pages,
                                  float sinkhorn_tol, int32_t* iters_used, int32_t* dev_status,
                                  void* stream) {
  if (!(sinkhorn_tol >= 0.0f) || sinkhorn_tol > 10.0f) return KVARN_ERR_INVALID_ARG;
  int st = check_desc(desc);
  if (st != KVARN_OK) return st;
  if (num_tiles < 0) return KVARN_ERR_INVALID_ARG;
  if (num_tiles == 0) return KVARN_OK;
  if (k == nullptr || v == nullptr || page_ids == nullptr || page_pool == nullptr)
    return KVARN_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(page_pool)) return KVARN_ERR_INVALID_ARG;
  if (tok_stride <= 0 || head_stride < 0 || tok_stride % 8 != 0 || head_stride % 8 != 0)
    return KVARN_ERR_INVALID_ARG;
  if (num_pool_pages < 1) return KVARN_ERR_INVALID_ARG;
  if ((int64_t)num_tiles * desc->num_kv_heads * 2 > 0x7fffffffLL) return KVARN_ERR_INVALID_ARG;
  QuantizeParams p{};
  p.k = static_cast<const __half*>(k);
  p.v = static_cast<const __half*>(v);
  p.tok_stride = tok_stride;
  p.head_stride = head_stride;
  p.page_ids = page_ids;
  p.pool = static_cast<uint8_t*>(page_pool);
  p.num_pool_pages = num_pool_pages;
  p.rec_bytes = desc->page_record_bytes;
  p.num_kv_heads = desc->num_kv_heads;
  p.d0 = desc->head_dim;
  p.iters = desc->sinkhorn_iters;
  p.eps = desc->sinkhorn_eps;
  if (sinkhorn_tol > 0.0f) {
    p.tol_hi = std::exp(sinkhorn_tol);
    p.tol_lo = std::exp(-sinkhorn_tol);
  }
  p.iters_out = iters_used;
  p.status = dev_status;
  p.append = 0;
  return launch_quantize_any(desc->head_dim_padded, desc->k_bits, desc->v_bits, p,
                             num_tiles * desc->num_kv_heads,
                             static_cast<cudaStream_t>(stream));
}

int kvarn_append_token(const kvarn_desc* desc, int batch, const void* k_new, const void* v_new,
                       void* partial_k, void* partial_v, const int32_t* seq_lens,
                       int32_t* seq_lens_out, const int32_t* block_table, int max_pages,
                       void* page_pool, int64_t num_pool_pages, int32_t* dev_status,
                       void* stream) {
  int st = check_desc(desc);
  if (st != KVARN_OK) return st;
  if (batch < 0 || max_pages < 1) return KVARN_ERR_INVALID_ARG;
  if (batch == 0) return KVARN_OK;
  if (k_new == nullptr || v_new == nullptr || partial_k == nullptr || partial_v == nullptr ||
      seq_lens == nullptr || block_table == nullptr || page_pool == nullptr)
    return KVARN_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(partial_k) || !aligned16(partial_v) ||
      !aligned16(page_pool))
    return KVARN_ERR_INVALID_ARG;
  if (seq_lens_out != nullptr && static_cast<const void*>(seq_lens_out) == seq_lens)
    return KVARN_ERR_INVALID_ARG;
  if (num_pool_pages < 1) return KVARN_ERR_INVALID_ARG;
  QuantizeParams p{};
  p.k_new = static_cast<const __half*>(k_new);
  p.v_new = static_cast<const __half*>(v_new);
  p.partial_k = static_cast<__half*>(partial_k);
  p.partial_v = static_cast<__half*>(partial_v);
  p.seq_lens = seq_lens;
  p.seq_lens_out = seq_lens_out;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.pool = static_cast<uint8_t*>(page_pool);
  p.num_pool_pages = num_pool_pages;
  p.rec_bytes = desc->page_record_bytes;
  p.num_kv_heads = desc->num_kv_heads;
  p.d0 = desc->head_dim;
  p.iters = desc->sinkhorn_iters;
  p.eps = desc->sinkhorn_eps;
  p.status = dev_status;
  p.append = 1;
  return launch_quantize_any(desc->head_dim_padded, desc->k_bits, desc->v_bits, p,
                             batch * desc->num_kv_heads,
                             static_cast<cudaStream_t>(stream));
}

// Smallest split size (sealed pages per decode CTA, its warps taking them round-robin): the
// workspace holds the partials of this many splits per row.  A launch may take a larger size
// (decode_split_pages), which needs fewer.
static int decode_pages_per_split(const kvarn_desc*, int) { return 32; }

size_t kvarn_decode_workspace_bytes(const kvarn_desc* desc, int batch, int num_q_heads,
                                    int max_pages) {
  if (check_desc(desc) != KVARN_OK || batch < 0 || num_q_heads < 1 || max_pages < 1) return 0;
  const int pps = decode_pages_per_split(desc, max_pages);
  const int64_t max_splits = (max_pages + pps - 1) / pps + 2;  // + the partial tile + one
  return (size_t)batch * num_q_heads * max_splits * (desc->head_dim_padded + 4) * sizeof(float);
}

}  // extern "C"

namespace kvarn {

// Host-side checks of a decode call's arguments other than its workspace: a KVARN_ERR_* code,
// KVARN_OK, or kDecodeNothingToDo for an empty batch (a valid call that launches nothing).
int decode_args_check(const kvarn_desc* desc, int batch, int num_q_heads, const void* q,
                      const void* page_pool, int64_t num_pool_pages, const int32_t* block_table,
                      int max_pages, const int32_t* seq_lens, const void* partial_k,
                      const void* partial_v, float softmax_scale, const void* out) {
  const int st = check_desc(desc);
  if (st != KVARN_OK) return st;
  if (batch < 0 || num_q_heads < 1 || max_pages < 1) return KVARN_ERR_INVALID_ARG;
  if (num_q_heads % desc->num_kv_heads != 0) return KVARN_ERR_UNSUPPORTED;
  const int group = num_q_heads / desc->num_kv_heads;
  if (!(group == 1 || group == 2 || group == 4 || group == 8)) return KVARN_ERR_UNSUPPORTED;
  if (group == 8 && desc->head_dim_padded == 256) return KVARN_ERR_UNSUPPORTED;
  if (batch == 0) return kDecodeNothingToDo;
  if (q == nullptr || page_pool == nullptr || block_table == nullptr || seq_lens == nullptr ||
      out == nullptr)
    return KVARN_ERR_INVALID_ARG;
  if ((partial_k == nullptr) != (partial_v == nullptr)) return KVARN_ERR_INVALID_ARG;
  if (!aligned16(page_pool) || !aligned16(partial_k) || !aligned16(partial_v))
    return KVARN_ERR_INVALID_ARG;
  if (num_pool_pages < 1 || !(softmax_scale > 0.0f)) return KVARN_ERR_INVALID_ARG;
  return KVARN_OK;
}

}  // namespace kvarn

extern "C" {

// The decode kernels, chosen for comparing them through the environment (read on every call):
// KVARN_DECODE_KERNEL "split" runs the mma.sync kernel with one CTA per split of 32 or more
// pages, "tc" GQA-8 decode (head_dim 128, K4V2) on the tcgen05 kernel; by default the mma.sync
// kernel runs as persistent CTAs over a balanced partition of the sealed pages (no tail of short
// splits, one pipeline per CTA).  KVARN_DECODE_OPEN_TILES "split" attends to the raw partial
// tiles in the decode kernels, as splits of their own; by default the merge kernel attends to
// them (from shared memory, one CTA per sequence and kv head).
static bool decode_env(const char* var, const char* value) {
  const char* v = std::getenv(var);
  return v != nullptr && std::strcmp(v, value) == 0;
}
static bool decode_kernel_env(const char* name) { return decode_env("KVARN_DECODE_KERNEL", name); }
static bool decode_tc_requested() { return decode_kernel_env("tc"); }

static int decode_phases(const kvarn_desc* desc, int batch, int num_q_heads, const void* q,
                         const void* page_pool, int64_t num_pool_pages, const int32_t* block_table,
                         int max_pages, const int32_t* seq_lens, const void* partial_k,
                         const void* partial_v, float softmax_scale, void* out, void* workspace,
                         size_t workspace_bytes, int32_t* dev_status, void* stream, int phases) {
  const int st = decode_args_check(desc, batch, num_q_heads, q, page_pool, num_pool_pages,
                                   block_table, max_pages, seq_lens, partial_k, partial_v,
                                   softmax_scale, out);
  if (st == kDecodeNothingToDo) return KVARN_OK;
  if (st != KVARN_OK) return st;
  if (workspace == nullptr || !aligned16(workspace)) return KVARN_ERR_INVALID_ARG;
  const size_t need = kvarn_decode_workspace_bytes(desc, batch, num_q_heads, max_pages);
  if (workspace_bytes < need) return KVARN_ERR_WORKSPACE_TOO_SMALL;
  const int group = num_q_heads / desc->num_kv_heads;
  const int nt = group <= 4 ? 1 : 2;
  const int pps = decode_pages_per_split(desc, max_pages);
  DecodeParams p{};
  p.q = static_cast<const __half*>(q);
  p.pool = static_cast<const uint8_t*>(page_pool);
  p.num_pool_pages = num_pool_pages;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.seq_lens = seq_lens;
  p.partial_k = static_cast<const __half*>(partial_k);
  p.partial_v = static_cast<const __half*>(partial_v);
  p.qscale = softmax_scale * kLog2e;
  p.out = static_cast<__half*>(out);
  p.part = static_cast<float*>(workspace);
  p.batch = batch;
  p.num_kv_heads = desc->num_kv_heads;
  p.num_q_heads = num_q_heads;
  p.group = group;
  p.d0 = desc->head_dim;
  p.max_splits = (max_pages + pps - 1) / pps + 2;  // workspace stride at the smallest size
  p.pages_per_split = decode_split_pages(desc->head_dim_padded, nt, desc->k_bits, desc->v_bits,
                                         (int64_t)batch * desc->num_kv_heads, max_pages);
  p.chunk = 1;
  p.vgroups = 1;
  p.status = dev_status;
  p.partial_in_merge = decode_env("KVARN_DECODE_OPEN_TILES", "split") ? 0 : 1;
  if (decode_tc_requested() && decode_tc_serves(desc->head_dim_padded, nt, desc->k_bits, desc->v_bits, p)) {
    p.part_mode = 3;
    p.part_ctas = decode_tc_ctas();
  } else if (!decode_kernel_env("split")) {
    p.part_mode = 1;
    p.part_ctas = decode_persistent_ctas(desc->head_dim_padded, nt, desc->k_bits, desc->v_bits);
  }
  if (p.part_mode != 0 && p.part_ctas < 1) return KVARN_ERR_CUDA;
  return launch_decode_any(desc->head_dim_padded, nt, desc->k_bits, desc->v_bits, p,
                           static_cast<cudaStream_t>(stream), phases);
}

int kvarn_decode_attention(const kvarn_desc* desc, int batch, int num_q_heads, const void* q,
                           const void* page_pool, int64_t num_pool_pages,
                           const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                           const void* partial_k, const void* partial_v, float softmax_scale,
                           void* out, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream) {
  return decode_phases(desc, batch, num_q_heads, q, page_pool, num_pool_pages, block_table,
                       max_pages, seq_lens, partial_k, partial_v, softmax_scale, out, workspace,
                       workspace_bytes, dev_status, stream, kDecodeSplits | kDecodeMerge);
}

int kvarn_decode_partials(const kvarn_desc* desc, int batch, int num_q_heads, const void* q,
                          const void* page_pool, int64_t num_pool_pages,
                          const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                          const void* partial_k, const void* partial_v, float softmax_scale,
                          void* out, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream) {
  return decode_phases(desc, batch, num_q_heads, q, page_pool, num_pool_pages, block_table,
                       max_pages, seq_lens, partial_k, partial_v, softmax_scale, out, workspace,
                       workspace_bytes, dev_status, stream, kDecodeSplits);
}

int kvarn_decode_combine(const kvarn_desc* desc, int batch, int num_q_heads, const void* q,
                         const void* page_pool, int64_t num_pool_pages,
                         const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                         const void* partial_k, const void* partial_v, float softmax_scale,
                         void* out, void* workspace, size_t workspace_bytes,
                         int32_t* dev_status, void* stream) {
  return decode_phases(desc, batch, num_q_heads, q, page_pool, num_pool_pages, block_table,
                       max_pages, seq_lens, partial_k, partial_v, softmax_scale, out, workspace,
                       workspace_bytes, dev_status, stream, kDecodeMerge);
}

size_t kvarn_prefill_workspace_bytes(const kvarn_desc* desc, int batch, int num_q_heads,
                                     int chunk_len, int max_pages) {
  if (check_desc(desc) != KVARN_OK || batch < 0 || num_q_heads < 1 || chunk_len < 1 || max_pages < 1)
    return 0;
  const int pps = decode_pages_per_split(desc, max_pages);
  const int64_t max_splits = (max_pages + pps - 1) / pps + 2;  // + partial tile + chunk
  return (size_t)batch * chunk_len * num_q_heads * max_splits * (desc->head_dim_padded + 4) *
         sizeof(float);
}

int kvarn_prefill_attention(const kvarn_desc* desc, int batch, int num_q_heads, int chunk_len,
                            const void* q, const void* chunk_k, const void* chunk_v,
                            const void* page_pool, int64_t num_pool_pages,
                            const int32_t* block_table, int max_pages, const int32_t* cache_lens,
                            const void* partial_k, const void* partial_v, float softmax_scale,
                            void* out, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, void* stream) {
  int st = check_desc(desc);
  if (st != KVARN_OK) return st;
  if (batch < 0 || num_q_heads < 1 || max_pages < 1 || chunk_len < 1) return KVARN_ERR_INVALID_ARG;
  if (num_q_heads % desc->num_kv_heads != 0) return KVARN_ERR_UNSUPPORTED;
  const int group = num_q_heads / desc->num_kv_heads;
  if (!(group == 1 || group == 2 || group == 4 || group == 8)) return KVARN_ERR_UNSUPPORTED;
  // query vectors of a kv head per CTA: 8 (4 at head_dim 256)
  const int nt = desc->head_dim_padded <= 128 ? 2 : 1;
  const int64_t vgroups = ((int64_t)chunk_len * group + 4 * nt - 1) / (4 * nt);
  if (vgroups * desc->num_kv_heads > 65535 || (int64_t)batch > 65535) return KVARN_ERR_UNSUPPORTED;
  if (batch == 0) return KVARN_OK;
  if (q == nullptr || chunk_k == nullptr || chunk_v == nullptr || page_pool == nullptr ||
      block_table == nullptr || cache_lens == nullptr || out == nullptr || workspace == nullptr)
    return KVARN_ERR_INVALID_ARG;
  if (!aligned16(chunk_k) || !aligned16(chunk_v)) return KVARN_ERR_INVALID_ARG;
  if ((partial_k == nullptr) != (partial_v == nullptr)) return KVARN_ERR_INVALID_ARG;
  if (!aligned16(page_pool) || !aligned16(workspace) || !aligned16(partial_k) || !aligned16(partial_v))
    return KVARN_ERR_INVALID_ARG;
  if (num_pool_pages < 1 || !(softmax_scale > 0.0f)) return KVARN_ERR_INVALID_ARG;
  const size_t need = kvarn_prefill_workspace_bytes(desc, batch, num_q_heads, chunk_len, max_pages);
  if (workspace_bytes < need) return KVARN_ERR_WORKSPACE_TOO_SMALL;
  const int pps = decode_pages_per_split(desc, max_pages);
  DecodeParams p{};
  p.q = static_cast<const __half*>(q);
  p.pool = static_cast<const uint8_t*>(page_pool);
  p.num_pool_pages = num_pool_pages;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.seq_lens = cache_lens;
  p.partial_k = static_cast<const __half*>(partial_k);
  p.partial_v = static_cast<const __half*>(partial_v);
  p.qscale = softmax_scale * kLog2e;
  p.out = static_cast<__half*>(out);
  p.part = static_cast<float*>(workspace);
  p.batch = batch;
  p.num_kv_heads = desc->num_kv_heads;
  p.num_q_heads = num_q_heads;
  p.group = group;
  p.d0 = desc->head_dim;
  p.max_splits = (max_pages + pps - 1) / pps + 2;  // workspace stride at the smallest size
  p.pages_per_split = decode_split_pages(desc->head_dim_padded, nt, desc->k_bits, desc->v_bits,
                                         (int64_t)batch * desc->num_kv_heads * vgroups, max_pages);
  p.chunk = chunk_len;
  p.vgroups = (int)vgroups;
  p.chunk_k = static_cast<const __half*>(chunk_k);
  p.chunk_v = static_cast<const __half*>(chunk_v);
  p.status = dev_status;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the chunk's causal part first (its own split slot), then the cache splits and the merge
  st = launch_chunk_any(desc->head_dim_padded, p, s);
  if (st != KVARN_OK) return st;
  return launch_decode_any(desc->head_dim_padded, nt, desc->k_bits, desc->v_bits, p, s);
}

int kvarn_dequantize_tiles(const kvarn_desc* desc, const void* page_pool, int64_t num_pool_pages,
                           const int32_t* page_ids, int num_pages, void* k_out, void* v_out,
                           int32_t* dev_status, void* stream) {
  int st = check_desc(desc);
  if (st != KVARN_OK) return st;
  if (num_pages < 0) return KVARN_ERR_INVALID_ARG;
  if (num_pages == 0) return KVARN_OK;
  if (page_pool == nullptr || page_ids == nullptr || k_out == nullptr || v_out == nullptr)
    return KVARN_ERR_INVALID_ARG;
  if (num_pool_pages < 1) return KVARN_ERR_INVALID_ARG;
  DequantParams p{};
  p.pool = static_cast<const uint8_t*>(page_pool);
  p.num_pool_pages = num_pool_pages;
  p.page_ids = page_ids;
  p.k_out = static_cast<__half*>(k_out);
  p.v_out = static_cast<__half*>(v_out);
  p.num_kv_heads = desc->num_kv_heads;
  p.d0 = desc->head_dim;
  p.status = dev_status;
  return launch_dequant_any(desc->head_dim_padded, desc->k_bits, desc->v_bits, p, num_pages,
                            static_cast<cudaStream_t>(stream));
}

int kvarn_quantization_error(const kvarn_desc* desc, const void* k, const void* v,
                             int64_t tok_stride, int64_t head_stride, int num_tiles,
                             const int32_t* page_ids, const void* page_pool, int64_t num_pool_pages,
                             float* err_stats, int32_t* dev_status, void* stream) {
  int st = check_desc(desc);
  if (st != KVARN_OK) return st;
  if (num_tiles < 0) return KVARN_ERR_INVALID_ARG;
  if (num_tiles == 0) return KVARN_OK;
  if (k == nullptr || v == nullptr || page_ids == nullptr || page_pool == nullptr ||
      err_stats == nullptr)
    return KVARN_ERR_INVALID_ARG;
  if (!aligned16(err_stats)) return KVARN_ERR_INVALID_ARG;
  if (tok_stride <= 0 || head_stride < 0) return KVARN_ERR_INVALID_ARG;
  if (num_pool_pages < 1) return KVARN_ERR_INVALID_ARG;
  if ((int64_t)num_tiles * desc->num_kv_heads * 2 > 0x7fffffffLL) return KVARN_ERR_INVALID_ARG;
  DequantParams p{};
  p.pool = static_cast<const uint8_t*>(page_pool);
  p.num_pool_pages = num_pool_pages;
  p.page_ids = page_ids;
  p.num_kv_heads = desc->num_kv_heads;
  p.d0 = desc->head_dim;
  p.status = dev_status;
  p.k_src = static_cast<const __half*>(k);
  p.v_src = static_cast<const __half*>(v);
  p.tok_stride = tok_stride;
  p.head_stride = head_stride;
  p.err_out = err_stats;
  return launch_dequant_any(desc->head_dim_padded, desc->k_bits, desc->v_bits, p, num_tiles,
                            static_cast<cudaStream_t>(stream));
}

const char* kvarn_status_string(int status) {
  switch (status) {
    case KVARN_OK: return "ok";
    case KVARN_ERR_INVALID_ARG: return "invalid argument (null pointer, size, stride or alignment)";
    case KVARN_ERR_UNSUPPORTED: return "unsupported configuration (preset, head_dim, bits or GQA group)";
    case KVARN_ERR_WORKSPACE_TOO_SMALL: return "decode workspace smaller than kvarn_decode_workspace_bytes";
    case KVARN_ERR_CUDA: return "CUDA launch or attribute call failed";
    default: return "unknown status";
  }
}

}  // extern "C"
