// Uncompressed fp16 paged decode attention: the baseline the packed cache is measured
// against.
//
// The pages compare serving throughput with KVarN against fp16 KV caches (a normal ratio of
// 1.0-1.3x) and state that decode is bound by reading the cache [hotdry §监控要点;
// vatt §一次 16K context…: every decode step reads every cached K/V byte].  This kernel
// decodes from a plain fp16 paged cache with the same split-K / combine structure, page
// size and launch shapes as the packed-cache decode, so the two can be timed in the same
// harness on the same workload.
//
// Cache: per (page, kv head) one record of 128 K rows then 128 V rows, fp16 [2][128][d]
// (d = 64 or 128, no rotation, no padding); a sequence of length L uses ceil(L / 128) pages
// and only the first L % 128 rows of a partly filled last page are read.
//
// decode (grid (split, kv head, sequence), 8 warps): the CTA walks its split's pages in
// order, three in shared memory (two in flight): every thread moves 16-byte chunks with
// cp.async, chunk c of row r landing at chunk c ^ (r % 8) so that the 8 rows an ldmatrix
// reads fall in distinct banks; rows past the sequence's end are zero-filled.  Warp w takes
// tokens 16w..16w+15 of every page: QK with mma.sync m16n8k16 (A = K rows by ldmatrix,
// B = the fp16 queries, fp32 accumulation), online softmax in the log2 domain, PV with
// A = V^T by ldmatrix.trans and B = the probabilities split into fp16 hi + lo.  The CTA then
// merges its warps into one (m, l, o) partial per query head; combine merges the splits.
#include "common.cuh"
#include "params.cuh"

namespace kvarn {
namespace f16dec {

constexpr int kWarps = 8;
constexpr int kBuf = 3;          // pages in shared memory: one being read, two in flight
constexpr int kPagesPerSplit = 32;

template <int D>
struct Shape {
  static constexpr int kRowBytes = 2 * D;            // one K or V row (swizzled 16-byte chunks)
  static constexpr int kPageBytes = 256 * kRowBytes; // K rows 0..127, V rows 128..255
  static constexpr int kQBytes = 8 * D * 2;          // fp16 queries, 8 head slots
  static constexpr int kSmem = kBuf * kPageBytes + kQBytes;
  static_assert(kSmem <= 232448, "three pages fit in shared memory");
  static_assert(kBuf * kPageBytes >= kWarps * 8 * (D + 2) * 4, "merge scratch fits the pages");
};

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// byte offset of 16-byte chunk c of row r in a page buffer
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 2 * D + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

template <int D, int NT>
__global__ void __launch_bounds__(kWarps * 32, 1) decode_f16_kernel(DecodeParams p) {
  using S = Shape<D>;
  constexpr int NH = 4 * NT;
  extern __shared__ __align__(128) uint8_t smem_f[];
  uint8_t* pages = smem_f;
  __half* qs = reinterpret_cast<__half*>(smem_f + kBuf * S::kPageBytes);  // [8][D]

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tq = lane & 3;
  grid_dependency_wait();
  const int cap = p.max_pages * kTile;
  int len = p.seq_lens[b];
  if (len < 0 || len > cap) {
    if (threadIdx.x == 0 && split == 0 && h == 0) flag_error(p.status, KVARN_DEV_SEQ_TOO_LONG);
    len = len < 0 ? 0 : cap;
  }
  const int n_pages = (len + kTile - 1) / kTile;
  const int first = split * p.pages_per_split;
  if (first >= n_pages) return;
  const int n = min(n_pages, first + p.pages_per_split) - first;
  const int32_t* bt = p.block_table + (int64_t)b * p.max_pages;
  const int64_t rec = 2 * kTile * D * 2;  // bytes of one (page, kv head) record
  const uint32_t sbase = smem_u32(pages);

  // rows of the CTA's j-th page that hold tokens
  auto rows_of = [&](int j) { return min(kTile, len - (first + j) * kTile); };
  // all threads: page j into buffer j % kBuf, one cp.async group (rows past the end zero-filled)
  auto issue = [&](int j) {
    if (j < n) {
      const int rows = rows_of(j);
      int64_t id = bt[first + j];
      if (id < 0 || id >= p.num_pool_pages) {
        if (threadIdx.x == 0) flag_error(p.status, KVARN_DEV_BAD_PAGE_ID);
        id = 0;
      }
      const uint8_t* src = p.pool + (id * p.num_kv_heads + h) * rec;
      const uint32_t dst = sbase + (j % kBuf) * S::kPageBytes;
      constexpr int kChunks = D / 8;  // 16-byte chunks per row
#pragma unroll 4
      for (int qi = threadIdx.x; qi < 256 * kChunks; qi += kWarps * 32) {
        const int r = qi / kChunks, c = qi - r * kChunks;
        const bool in = (r & (kTile - 1)) < rows;
        cp_async16(dst + swz<D>(r, c), in ? src + (int64_t)qi * 16 : src, in ? 16u : 0u);
      }
    }
    cp_async_commit();  // an empty group past the end keeps the group count uniform
  };
  for (int j = 0; j < kBuf - 1; ++j) issue(j);
  // the fp16 queries of this kv head's group: head slot hl -> row hl (zero beyond the group)
  for (int i = threadIdx.x; i < NH * D; i += blockDim.x) {
    const int hl = i / D, c = i - hl * D;
    qs[i] = hl < p.group ? p.q[((int64_t)b * p.num_q_heads + h * p.group + hl) * D + c]
                         : __float2half(0.0f);
  }
  __syncthreads();
  // QK B operand, fixed for the whole split: column 2j = head 4nt + j, column 2j + 1 = 0, so
  // the lane's accumulator pairs hold (logit, 0) of head 4nt + tq
  uint32_t bq[D / 16][NT][2];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const __half* qr = qs + (4 * nt + (g >> 1)) * D + 16 * kk + 2 * tq;
      const bool zero = (g & 1) != 0;
      bq[kk][nt][0] = zero ? 0u : *reinterpret_cast<const uint32_t*>(qr);
      bq[kk][nt][1] = zero ? 0u : *reinterpret_cast<const uint32_t*>(qr + 8);
    }

  float m[NT], l[NT], o[D / 16][NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt] = -INFINITY;
    l[nt] = 0.0f;
#pragma unroll
    for (int mc = 0; mc < D / 16; ++mc) o[mc][nt][0] = o[mc][nt][1] = 0.0f;
  }
  const int t0 = 16 * warp;  // this warp's tokens in every page
  for (int j = 0; j < n; ++j) {
    __syncthreads();  // every warp is done with page j - 1: its buffer takes page j + kBuf - 1
    issue(j + kBuf - 1);
    cp_async_wait<kBuf - 1>();  // this thread's chunks of page j have landed
    __syncthreads();            // and everyone's
    const int rows = rows_of(j);
    if (t0 >= rows) continue;  // a partly filled last page: nothing for this warp
    const uint32_t kbase = sbase + (j % kBuf) * S::kPageBytes;
    // ---- QK: logits of tokens t0 + g, t0 + g + 8 for head 4nt + tq ----
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
    {
      const int row = t0 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4(kbase + swz<D>(row, 2 * kk + (lane >> 4)), a);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt], a[0], a[1], a[2], a[3], bq[kk][nt][0], bq[kk][nt][1]);
      }
    }
    const bool v0 = t0 + g < rows, v1 = t0 + g + 8 < rows;
    float pr[NT][2], alpha[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float s0 = v0 ? (acc[nt][0] + acc[nt][1]) * p.qscale : -INFINITY;
      const float s1 = v1 ? (acc[nt][2] + acc[nt][3]) * p.qscale : -INFINITY;
      float mx = fmaxf(s0, s1);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float mnew = fmaxf(m[nt], mx);  // finite: token t0 (g = 0) is valid
      alpha[nt] = exp2f(m[nt] - mnew);
      m[nt] = mnew;
      pr[nt][0] = exp2f(s0 - mnew);
      pr[nt][1] = exp2f(s1 - mnew);
      l[nt] = fmaf(l[nt], alpha[nt], pr[nt][0] + pr[nt][1]);
    }
    // ---- PV: B = probabilities as (hi, lo) column pairs, moved into the B layout ----
    uint32_t bw[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const __half2 hi = __floats2half2_rn(pr[nt][0], pr[nt][1]);
      const float2 hf = __half22float2(hi);
      const __half2 lo = __floats2half2_rn(pr[nt][0] - hf.x, pr[nt][1] - hf.y);
      bw[nt][0] = movmatrix_trans(h2u(__lows2half2(hi, lo)));   // (hi, lo) of token row g
      bw[nt][1] = movmatrix_trans(h2u(__highs2half2(hi, lo)));  // (hi, lo) of token row g + 8
    }
    {
      const int row = kTile + t0 + (lane & 7) + 8 * (lane >> 4);
#pragma unroll
      for (int mc = 0; mc < D / 16; ++mc) {
        uint32_t a[4];
        ldsm_x4_trans(kbase + swz<D>(row, 2 * mc + ((lane >> 3) & 1)), a);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float pacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          mma16816(pacc, a[0], a[1], a[2], a[3], bw[nt][0], bw[nt][1]);
          o[mc][nt][0] = fmaf(o[mc][nt][0], alpha[nt], pacc[0] + pacc[1]);
          o[mc][nt][1] = fmaf(o[mc][nt][1], alpha[nt], pacc[2] + pacc[3]);
        }
      }
    }
  }
  // ---- merge the warps: (m, l, o) per head slot ----
  __syncthreads();
  grid_launch_dependents();
  float* mS = reinterpret_cast<float*>(pages);
  float* lS = mS + kWarps * NH;
  float* oS = lS + kWarps * NH;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float lt = l[nt];
    lt += __shfl_xor_sync(0xffffffffu, lt, 4);
    lt += __shfl_xor_sync(0xffffffffu, lt, 8);
    lt += __shfl_xor_sync(0xffffffffu, lt, 16);
    const int hl = 4 * nt + tq;
    if (g == 0) {
      mS[warp * NH + hl] = m[nt];
      lS[warp * NH + hl] = lt;
    }
#pragma unroll
    for (int mc = 0; mc < D / 16; ++mc) {
      oS[(warp * NH + hl) * D + 16 * mc + g] = o[mc][nt][0];
      oS[(warp * NH + hl) * D + 16 * mc + g + 8] = o[mc][nt][1];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < NH * D; idx += blockDim.x) {
    const int hl = idx / D, c = idx - hl * D;
    if (hl >= p.group) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mS[w * NH + hl]);
    float ov = 0.0f, lv = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = mS[w * NH + hl];
      const float sc = mw == -INFINITY ? 0.0f : exp2f(mw - M);  // warps that saw no token
      ov = fmaf(sc, oS[(w * NH + hl) * D + c], ov);
      lv = fmaf(sc, lS[w * NH + hl], lv);
    }
    float* dst = p.part + (((int64_t)b * p.num_q_heads + h * p.group + hl) * p.max_splits + split) * (D + 4);
    dst[4 + c] = ov;
    if (c == 0) {
      dst[0] = M;
      dst[1] = lv;
    }
  }
}

// One warp per (sequence, query head): merge the splits and normalise.
template <int D>
__global__ void __launch_bounds__(128) combine_f16_kernel(DecodeParams p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
  grid_dependency_wait();
  grid_launch_dependents();
  if (gw >= p.batch * p.num_q_heads) return;
  const int b = gw / p.num_q_heads;
  const int cap = p.max_pages * kTile;
  int len = p.seq_lens[b];
  len = len < 0 ? 0 : (len > cap ? cap : len);
  const int n_pages = (len + kTile - 1) / kTile;
  const int n_splits = (n_pages + p.pages_per_split - 1) / p.pages_per_split;
  const float* src = p.part + (int64_t)gw * p.max_splits * (D + 4);
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, src[s * (D + 4)]);
  float acc[E], lsum = 0.0f;
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.0f;
  for (int s = 0; s < n_splits; ++s) {
    const float* r = src + s * (D + 4);
    const float sc = exp2f(r[0] - M);
    lsum = fmaf(sc, r[1], lsum);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(sc, r[4 + lane + 32 * e], acc[e]);
  }
  const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
  __half* out = p.out + (int64_t)gw * D;
#pragma unroll
  for (int e = 0; e < E; ++e) out[lane + 32 * e] = __float2half_rn(acc[e] * inv);
}

template <int D, int NT>
static int launch(const DecodeParams& p, cudaStream_t stream) {
  static PerDeviceOnce smem_once;  // the attribute is set once per device
  const void* fn = reinterpret_cast<const void*>(decode_f16_kernel<D, NT>);
  if (const int st = set_smem_limit(smem_once, fn, Shape<D>::kSmem); st != KVARN_OK) return st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.max_splits, p.num_kv_heads, p.batch);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = Shape<D>::kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_f16_kernel<D, NT>, p) != cudaSuccess) return KVARN_ERR_CUDA;
  cfg.gridDim = dim3((p.batch * p.num_q_heads + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  if (cudaLaunchKernelEx(&cfg, combine_f16_kernel<D>, p) != cudaSuccess) return KVARN_ERR_CUDA;
  return KVARN_OK;
}

}  // namespace f16dec
}  // namespace kvarn

using namespace kvarn;

extern "C" {

size_t kvarn_fp16_page_bytes(int head_dim) {
  if (head_dim != 64 && head_dim != 128) return 0;
  return (size_t)2 * kTile * head_dim * 2;
}

size_t kvarn_fp16_decode_workspace_bytes(int head_dim, int batch, int num_q_heads, int max_pages) {
  if ((head_dim != 64 && head_dim != 128) || batch < 0 || num_q_heads < 1 || max_pages < 1) return 0;
  const int64_t splits = (max_pages + f16dec::kPagesPerSplit - 1) / f16dec::kPagesPerSplit;
  return (size_t)batch * num_q_heads * splits * (head_dim + 4) * sizeof(float);
}

int kvarn_fp16_decode_attention(int head_dim, int num_kv_heads, int batch, int num_q_heads,
                                const void* q, const void* page_pool, int64_t num_pool_pages,
                                const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                                float softmax_scale, void* out, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (head_dim != 64 && head_dim != 128) return KVARN_ERR_UNSUPPORTED;
  if (num_kv_heads < 1 || batch < 0 || num_q_heads < 1 || max_pages < 1) return KVARN_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return KVARN_ERR_UNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  if (!(group == 1 || group == 2 || group == 4 || group == 8)) return KVARN_ERR_UNSUPPORTED;
  if (batch == 0) return KVARN_OK;
  if (q == nullptr || page_pool == nullptr || block_table == nullptr || seq_lens == nullptr ||
      out == nullptr || workspace == nullptr)
    return KVARN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(page_pool) & 15u) != 0 || (reinterpret_cast<uintptr_t>(q) & 3u) != 0)
    return KVARN_ERR_INVALID_ARG;
  if (num_pool_pages < 1 || !(softmax_scale > 0.0f) || batch > 65535 || num_kv_heads > 65535)
    return KVARN_ERR_INVALID_ARG;
  if (workspace_bytes < kvarn_fp16_decode_workspace_bytes(head_dim, batch, num_q_heads, max_pages))
    return KVARN_ERR_WORKSPACE_TOO_SMALL;
  DecodeParams p{};
  p.q = static_cast<const __half*>(q);
  p.pool = static_cast<const uint8_t*>(page_pool);
  p.num_pool_pages = num_pool_pages;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.seq_lens = seq_lens;
  p.qscale = softmax_scale * 1.4426950408889634f;
  p.out = static_cast<__half*>(out);
  p.part = static_cast<float*>(workspace);
  p.batch = batch;
  p.num_kv_heads = num_kv_heads;
  p.num_q_heads = num_q_heads;
  p.group = group;
  p.d0 = head_dim;
  p.pages_per_split = f16dec::kPagesPerSplit;
  p.max_splits = (max_pages + f16dec::kPagesPerSplit - 1) / f16dec::kPagesPerSplit;
  p.chunk = 1;
  p.vgroups = 1;
  p.status = dev_status;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nt = group <= 4 ? 1 : 2;
  if (head_dim == 64) return nt == 1 ? f16dec::launch<64, 1>(p, s) : f16dec::launch<64, 2>(p, s);
  return nt == 1 ? f16dec::launch<128, 1>(p, s) : f16dec::launch<128, 2>(p, s);
}

}  // extern "C"
