// Device helpers shared by the packed-cache decode kernels (mma.sync and tcgen05 forms).
#pragma once

#include "common.cuh"
#include "params.cuh"

namespace kvarn {

constexpr float kTwo24 = 16777216.0f;  // undoes the 2^-24 of a code held as an fp16 subnormal

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// K word -> A fragment as fp16 subnormals: a0/a1 (channels 2tq..) = code * 2^-24,
// a2/a3 (channels 2tq+8..) = code * 2^-20.
__device__ __forceinline__ void unpack_k(uint32_t x, uint32_t (&a)[4]) {
  const uint32_t y = x >> 8;
  a[0] = x & 0x000F000Fu;
  a[2] = x & 0x00F000F0u;
  a[1] = y & 0x000F000Fu;
  a[3] = y & 0x00F000F0u;
}

// 8-bit fragment words w0, w1 -> A fragment as fp16 subnormals code * 2^-24: register rho + 2h
// takes bytes rho and rho + 2 of word h (every code below 2^10, so each is exact).
__device__ __forceinline__ void unpack_k8(uint32_t w0, uint32_t w1, uint32_t (&a)[4]) {
  a[0] = __byte_perm(w0, 0u, 0x4240);
  a[1] = __byte_perm(w0, 0u, 0x4341);
  a[2] = __byte_perm(w1, 0u, 0x4240);
  a[3] = __byte_perm(w1, 0u, 0x4341);
}

// V word -> the A fragments of token blocks 2ks2 (a0) and 2ks2+1 (a1) as fp16 subnormals:
// block f, token half h -> code * 2^(-24 + 4f + 2h).
__device__ __forceinline__ void unpack_v(uint32_t x, uint32_t (&a0)[4], uint32_t (&a1)[4]) {
  const uint32_t y = x >> 8;
  a0[0] = x & 0x00030003u;
  a0[2] = x & 0x000C000Cu;
  a0[1] = y & 0x00030003u;
  a0[3] = y & 0x000C000Cu;
  a1[0] = x & 0x00300030u;
  a1[2] = x & 0x00C000C0u;
  a1[1] = y & 0x00300030u;
  a1[3] = y & 0x00C000C0u;
}

// ---- fp16 rows in shared memory for ldmatrix -----------------------------------------------
// Byte offset of 16-byte chunk c of row r in a buffer of D-channel fp16 rows, chunk c of row r
// stored at chunk c ^ (r % 8), so that the 8 rows an ldmatrix reads fall in distinct banks.
template <int D>
__device__ __forceinline__ uint32_t swz_row(int r, int c) {
  return (uint32_t)(r * 2 * D + ((c ^ (r & 7)) << 4));
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
// 16-byte global -> shared copy, zero-filled beyond `bytes` (0 or 16)
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit_all() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// all but the most recent committed group complete
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Walsh-Hadamard transform of D values spread over a warp, lane holding D/32 consecutive.
template <int D>
__device__ __forceinline__ void warp_fwht(float (&v)[D / 32], int lane) {
  constexpr int E = D / 32;
#pragma unroll
  for (int h = 1; h < E; h <<= 1)
#pragma unroll
    for (int i = 0; i < E; ++i)
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
      v[i] = upper ? (o - v[i]) : (v[i] + o);
    }
  }
}

// E consecutive fp16 / fp32 values from shared memory (8, 16 or 32 bytes, aligned) as floats.
template <int E>
__device__ __forceinline__ void load_f16(const __half* src, float (&f)[E]) {
  static_assert(E == 2 || E == 4 || E == 8, "2, 4 or 8 halves");
  if constexpr (E == 2) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(src));
    f[0] = a.x;
    f[1] = a.y;
  } else {
#pragma unroll
    for (int i = 0; i < E / 4; ++i) {
      const uint2 u = reinterpret_cast<const uint2*>(src)[i];
      const float2 a = __half22float2(u2h2(u.x)), c = __half22float2(u2h2(u.y));
      f[4 * i] = a.x;
      f[4 * i + 1] = a.y;
      f[4 * i + 2] = c.x;
      f[4 * i + 3] = c.y;
    }
  }
}
template <int E>
__device__ __forceinline__ void load_f32(const float* src, float (&f)[E]) {
  if constexpr (E % 4 == 0) {
#pragma unroll
    for (int i = 0; i < E / 4; ++i) {
      const float4 a = reinterpret_cast<const float4*>(src)[i];
      f[4 * i] = a.x;
      f[4 * i + 1] = a.y;
      f[4 * i + 2] = a.z;
      f[4 * i + 3] = a.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) f[e] = src[e];
  }
}

template <int D>
__device__ __forceinline__ float inv_sqrt_d() {
  return D == 64 ? 0.125f : (D == 128 ? 0.08838834764831845f : 0.0625f);
}

// ---- balanced page partition of the persistent decode kernels -----------------------------
// The sealed pages of all (sequence b, kv head h) rows, in (b, h, page) order, are laid on a
// line of virtual pages where every row with sealed pages first takes kSegPages units for the
// fixed work of a segment (its queries, its first page's latency, the CTA merge), then one unit
// per page.  The line is cut into `ctas` contiguous ranges of floor or ceil(total / ctas) units,
// one per CTA, with ctas no larger than total / 32: every range holds at least 32 units, so a
// row's pages (n consecutive units) fall in row_segments <= ceil(n / 32) + 1 ranges, and the
// segment whose first page sits at unit x writes split owner_cta(x) - owner_cta(the row's first
// page).  A range may hold only the fixed units of a row (no page): that CTA has no work.  Every
// kernel of the launch derives the same partition from seq_lens.
constexpr int kMinRangePages = 32;
constexpr int kSegPages = 8;  // virtual pages of a segment's fixed work

__device__ __forceinline__ int sealed_pages(const DecodeParams& p, int b) {
  const int cap = p.max_pages * kTile + (kTile - 1);
  int len = p.seq_lens[b];
  len = len < 0 ? 0 : (len > cap ? cap : len);
  return len / kTile;
}

// Virtual length of one row of n sealed pages.
__device__ __forceinline__ int row_units(int n) { return n > 0 ? n + kSegPages : 0; }

// Warp-collective: virtual length of one kv head's rows of sequences 0..lim-1 (every lane gets
// the sum).
__device__ __forceinline__ int64_t units_prefix(const DecodeParams& p, int lim, int lane) {
  long long s = 0;
  for (int b = lane; b < lim; b += 32) s += row_units(sealed_pages(p, b));
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
  return s;
}

struct PagePartition {
  int64_t total;  // virtual pages of all rows
  int64_t ctas;   // ranges; 0 when there are no sealed pages
};

__device__ __forceinline__ PagePartition page_partition(const DecodeParams& p, int lane) {
  PagePartition pp;
  pp.total = units_prefix(p, p.batch, lane) * p.num_kv_heads;
  int64_t c = pp.total / kMinRangePages;
  c = c < 1 ? 1 : (c > p.part_ctas ? p.part_ctas : c);
  pp.ctas = pp.total > 0 ? c : 0;
  return pp;
}

// First unit of range c, and the range that holds unit x.
__device__ __forceinline__ int64_t range_start(const PagePartition& pp, int64_t c) {
  return c * pp.total / pp.ctas;
}
__device__ __forceinline__ int64_t owner_cta(const PagePartition& pp, int64_t x) {
  return ((x + 1) * pp.ctas + pp.total - 1) / pp.total - 1;
}

// Warp-collective: the number of splits the sealed pages of row (b, h) fill.
__device__ __forceinline__ int row_segments(const DecodeParams& p, const PagePartition& pp, int b, int h,
                                            int lane) {
  const int n = sealed_pages(p, b);
  if (n == 0) return 0;
  // the unit of the row's first page
  const int64_t a = units_prefix(p, b, lane) * p.num_kv_heads + (int64_t)h * row_units(n) + kSegPages;
  return (int)(owner_cta(pp, a + n - 1) - owner_cta(pp, a) + 1);
}

// Segment walk over a CTA's range: a maximal run of pages of one row.
struct Walk {
  int b, h, j, n;    // row (sequence b, kv head h), first page j of the segment, sealed pages n
  int slot;          // split the segment's partial goes to
  int64_t left;      // units of the range from page j of this row on (0: no more pages)
  __device__ int count() const { return (int)min((int64_t)(n - j), left); }
  // next segment: the next row with sealed pages (slot 0, page 0), past its fixed units
  __device__ void next(const DecodeParams& p) {
    left -= count();
    if (left <= 0) return;
    j = 0;
    slot = 0;
    for (;;) {
      if (++h == p.num_kv_heads) {
        h = 0;
        ++b;
      }
      if (b >= p.batch) {  // unreachable while the lengths match the partition
        left = 0;
        return;
      }
      n = sealed_pages(p, b);
      if (n > 0) {
        left -= kSegPages;  // the range may end inside the row's fixed units
        if (left < 0) left = 0;
        return;
      }
      h = p.num_kv_heads - 1;  // skip the whole sequence
    }
  }
};

// Warp-collective: the walk of CTA c's range (left = 0 when the CTA has no pages).
__device__ __forceinline__ Walk range_walk(const DecodeParams& p, int64_t c, int lane) {
  const PagePartition pp = page_partition(p, lane);
  Walk w;
  w.b = w.h = w.j = w.n = w.slot = 0;
  w.left = 0;
  if (c >= pp.ctas) return w;
  const int64_t x0 = range_start(pp, c), x1 = range_start(pp, c + 1);
  // the row holding unit x0: scan the sequences 32 at a time
  long long cum = 0;
  for (int b0 = 0; b0 < p.batch; b0 += 32) {
    const int bb = b0 + lane;
    const int n = bb < p.batch ? sealed_pages(p, bb) : 0;
    long long incl = (long long)row_units(n) * p.num_kv_heads;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const long long o = __shfl_up_sync(0xffffffffu, incl, m);
      if (lane >= m) incl += o;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, cum + incl > x0);
    if (hit != 0u) {
      const int l = __ffs(hit) - 1;  // a sequence with sealed pages: its units hold x0
      const int nb = __shfl_sync(0xffffffffu, n, l);
      const int ru = row_units(nb);
      const long long excl = cum + __shfl_sync(0xffffffffu, incl, l) - (long long)ru * p.num_kv_heads;
      w.b = b0 + l;
      w.n = nb;
      w.h = (int)((x0 - excl) / ru);
      const int off = (int)((x0 - excl) - (long long)w.h * ru);  // unit of the row, fixed ones first
      const long long first = excl + (long long)w.h * ru + kSegPages;  // unit of the row's page 0
      w.j = off < kSegPages ? 0 : off - kSegPages;
      w.slot = (int)(c - owner_cta(pp, first));
      w.left = x1 - (first + w.j);
      if (w.left < 0) w.left = 0;  // the range ends inside the row's fixed units
      return w;
    }
    cum += __shfl_sync(0xffffffffu, incl, 31);
  }
  return w;
}

}  // namespace kvarn
