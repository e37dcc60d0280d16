// KVarN paged decode attention over the packed K4/V2 cache (sm_103a).
//
// Math (rotated basis, R = H_d / sqrt(d) orthonormal and symmetric):
//   logit_t = tau q . K_t = tau (qR) . (K_t R) = tau r_t ( sum_j q~_j s'_j code_tj + sum_j q~_j z'_j )
//   o = sum_t p_t V_t = ( sum_t p_t V~_t ) R,  V~_tj = c_j ( code_tj s'_t + z'_t )
// [vatt §四個步驟: the rotation is orthonormal so attention scores are unchanged;
//  hotdry §非对称量化与尺度折叠: the folded scales are multiplied back at read time]
//
// decode_kernel: grid (split, kv head, sequence).  Each CTA owns up to `pages_per_split`
// sealed pages of one (sequence, kv head), or the raw fp16 partial tile.  Its warps take
// pages round-robin; each warp streams whole page records into shared memory with 1-D bulk
// copies (double-buffered on mbarriers), then per page:
//   QK:  m16n8k16 MMAs, A = 4-bit codes [token x channel] unpacked exactly to fp16,
//        B = q~ . s'_K split into fp16 hi + lo (columns: 4 heads x {hi, lo}).
//   softmax: online, in the log2 domain (tau log2(e) folded into q~).
//   PV:  m16n8k16 MMAs, A = 2-bit codes^T [channel x token], B = p . s'_V split hi + lo,
//        moved from the QK accumulator layout with movmatrix.trans.
// The CTA merges its warps and writes (m, l, unnormalised o~) for its split; combine_kernel
// merges the splits, divides by l, undoes the rotation and stores fp16.
#include "common.cuh"
#include "params.cuh"

namespace kvarn {

constexpr int kDecWarps = 4;
constexpr int kDecStages = 2;


template <int D, int NT>
struct DecodeShape {
  static constexpr int kNH = 4 * NT;                 // head slots per kv head (G padded)
  static constexpr int kRec = record_layout(D).bytes;
  static constexpr int kQld = D + 8;                 // fp32 row stride of q in shared memory
  static constexpr int kRecBytes = kDecWarps * kDecStages * kRec;
  static constexpr int kQBytes = kNH * kQld * 4;
  static constexpr int kSmemBytes = kRecBytes + kQBytes + kDecWarps * kDecStages * 8;
};

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// 0x6400 | (code << b) is the fp16 value 1024 + code * 2^b; c = v * 2^-b - 1024 * 2^-b exactly.
__device__ __forceinline__ uint32_t code_to_f16(uint32_t biased, float inv_pow2) {
  const __half2 sc = __float2half2_rn(inv_pow2);
  const __half2 off = __float2half2_rn(-1024.0f * inv_pow2);
  return h2u(__hfma2(u2h(biased), sc, off));
}

// K word -> A fragment (a0: row g, a1: row g+8, a2: row g cols+8, a3: row g+8 cols+8).
__device__ __forceinline__ void unpack_k(uint32_t x, uint32_t (&a)[4]) {
  const uint32_t y = x >> 8;
  a[0] = code_to_f16(and_or(x, 0x000F000Fu, 0x64006400u), 1.0f);
  a[2] = code_to_f16(and_or(x, 0x00F000F0u, 0x64006400u), 1.0f / 16.0f);
  a[1] = code_to_f16(and_or(y, 0x000F000Fu, 0x64006400u), 1.0f);
  a[3] = code_to_f16(and_or(y, 0x00F000F0u, 0x64006400u), 1.0f / 16.0f);
}

// V word -> the two A fragments (token blocks 2ks2 and 2ks2+1) it carries.
__device__ __forceinline__ void unpack_v(uint32_t x, uint32_t (&a0)[4], uint32_t (&a1)[4]) {
  const uint32_t y = x >> 8;
  a0[0] = code_to_f16(and_or(x, 0x00030003u, 0x64006400u), 1.0f);
  a0[2] = code_to_f16(and_or(x, 0x000C000Cu, 0x64006400u), 0.25f);
  a0[1] = code_to_f16(and_or(y, 0x00030003u, 0x64006400u), 1.0f);
  a0[3] = code_to_f16(and_or(y, 0x000C000Cu, 0x64006400u), 0.25f);
  a1[0] = code_to_f16(and_or(x, 0x00300030u, 0x64006400u), 1.0f / 16.0f);
  a1[2] = code_to_f16(and_or(x, 0x00C000C0u, 0x64006400u), 1.0f / 64.0f);
  a1[1] = code_to_f16(and_or(y, 0x00300030u, 0x64006400u), 1.0f / 16.0f);
  a1[3] = code_to_f16(and_or(y, 0x00C000C0u, 0x64006400u), 1.0f / 64.0f);
}

// fp32 x -> (hi, lo) fp16 with hi + lo ~ x to ~22 bits; returns hi (sel == 0) or lo.
__device__ __forceinline__ __half2 split_pick(float x0, float x1, bool lo) {
  const __half2 hi = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(hi);
  const __half2 lw = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  return lo ? lw : hi;
}

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

template <int D>
__device__ __forceinline__ float inv_sqrt_d() {
  return D == 64 ? 0.125f : (D == 128 ? 0.08838834764831845f : 0.0625f);
}

template <int D, int NT>
struct WarpAcc {
  float m[NT], l[NT];
  float o[D / 16][NT][2];  // head 4nt + tq, channels 16mc + g + 8r (rotated basis)
};

template <int D, int NT>
__device__ __forceinline__ void process_page(const uint8_t* __restrict__ R,
                                             const float* __restrict__ qrot, int lane,
                                             WarpAcc<D, NT>& st) {
  constexpr RecordLayout RL = record_layout(D);
  constexpr int QLD = DecodeShape<D, NT>::kQld;
  const int g = lane >> 2, tq = lane & 3;
  const __half* Ks = reinterpret_cast<const __half*>(R + RL.kscale);
  const __half* Kz = reinterpret_cast<const __half*>(R + RL.kzero);
  const __half* Kr = reinterpret_cast<const __half*>(R + RL.kfactor);
  const __half* Vs = reinterpret_cast<const __half*>(R + RL.vscale);
  const __half* Vz = reinterpret_cast<const __half*>(R + RL.vzero);
  const __half* Vc = reinterpret_cast<const __half*>(R + RL.vfactor);

  // ---- B operand of QK: q~_j s'_j (hi or lo by column parity), and q~ . z' per head ---------
  uint32_t bq[D / 16][NT][2];
  float qz[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) qz[nt] = 0.0f;
  const bool lo_col = (g & 1) != 0;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int j0 = 16 * kk + 2 * tq;
    const float2 s0 = __half22float2(*reinterpret_cast<const __half2*>(Ks + j0));
    const float2 s1 = __half22float2(*reinterpret_cast<const __half2*>(Ks + j0 + 8));
    const float2 z0 = __half22float2(*reinterpret_cast<const __half2*>(Kz + j0));
    const float2 z1 = __half22float2(*reinterpret_cast<const __half2*>(Kz + j0 + 8));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float* qr = qrot + (4 * nt + (g >> 1)) * QLD;
      const float2 qa = *reinterpret_cast<const float2*>(qr + j0);
      const float2 qb = *reinterpret_cast<const float2*>(qr + j0 + 8);
      qz[nt] = fmaf(qa.x, z0.x, fmaf(qa.y, z0.y, fmaf(qb.x, z1.x, fmaf(qb.y, z1.y, qz[nt]))));
      bq[kk][nt][0] = h2u(split_pick(qa.x * s0.x, qa.y * s0.y, lo_col));
      bq[kk][nt][1] = h2u(split_pick(qb.x * s1.x, qb.y * s1.y, lo_col));
    }
  }
  float qzm[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float v = qz[nt];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    qzm[nt] = __shfl_sync(0xffffffffu, v, 8 * tq);  // head 4nt + tq lives in lanes g = 2tq
  }

  // ---- QK ---------------------------------------------------------------------------------
  float lg[8][NT][2];
#pragma unroll
  for (int mi = 0; mi < 8; ++mi) {
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
#pragma unroll
    for (int kq = 0; kq < D / 64; ++kq) {
      const uint4 w4 =
          *reinterpret_cast<const uint4*>(R + RL.kcodes + ((mi * (D / 64) + kq) * 32 + lane) * 16);
      const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t a[4];
        unpack_k(ws[e], a);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt], a, bq[4 * kq + e][nt][0], bq[4 * kq + e][nt][1]);
      }
    }
    const float r0 = __half2float(Kr[16 * mi + g]);
    const float r1 = __half2float(Kr[16 * mi + g + 8]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      lg[mi][nt][0] = r0 * ((acc[nt][0] + acc[nt][1]) + qzm[nt]);
      lg[mi][nt][1] = r1 * ((acc[nt][2] + acc[nt][3]) + qzm[nt]);
    }
  }

  // ---- online softmax ------------------------------------------------------------------------
  float alpha[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float mx = lg[0][nt][0];
#pragma unroll
    for (int mi = 0; mi < 8; ++mi) mx = fmaxf(mx, fmaxf(lg[mi][nt][0], lg[mi][nt][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mnew = fmaxf(st.m[nt], mx);
    alpha[nt] = exp2f(st.m[nt] - mnew);
    st.m[nt] = mnew;
    float ps = 0.0f;
#pragma unroll
    for (int mi = 0; mi < 8; ++mi)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float pv = exp2f(lg[mi][nt][r] - mnew);
        lg[mi][nt][r] = pv;
        ps += pv;
      }
    st.l[nt] = fmaf(st.l[nt], alpha[nt], ps);
  }

  // ---- PV --------------------------------------------------------------------------------------
  float pacc[D / 16][NT][4];
#pragma unroll
  for (int mc = 0; mc < D / 16; ++mc)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) pacc[mc][nt][0] = pacc[mc][nt][1] = pacc[mc][nt][2] = pacc[mc][nt][3] = 0.0f;
  float zs[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) zs[nt] = 0.0f;
#pragma unroll
  for (int ks2 = 0; ks2 < 4; ++ks2) {
    uint32_t bw[2][NT][2];
#pragma unroll
    for (int f = 0; f < 2; ++f) {
      const int ks = 2 * ks2 + f;
      const float sv0 = __half2float(Vs[16 * ks + g]), sv1 = __half2float(Vs[16 * ks + g + 8]);
      const float zv0 = __half2float(Vz[16 * ks + g]), zv1 = __half2float(Vz[16 * ks + g + 8]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float p0 = lg[ks][nt][0], p1 = lg[ks][nt][1];
        zs[nt] = fmaf(p0, zv0, fmaf(p1, zv1, zs[nt]));
        const float w0 = p0 * sv0, w1 = p1 * sv1;
        const __half hi0 = __float2half_rn(w0), hi1 = __float2half_rn(w1);
        const __half lo0 = __float2half_rn(w0 - __half2float(hi0));
        const __half lo1 = __float2half_rn(w1 - __half2float(hi1));
        bw[f][nt][0] = movmatrix_trans(h2u(__halves2half2(hi0, lo0)));
        bw[f][nt][1] = movmatrix_trans(h2u(__halves2half2(hi1, lo1)));
      }
    }
#pragma unroll
    for (int mq = 0; mq < D / 64; ++mq) {
      const uint4 w4 =
          *reinterpret_cast<const uint4*>(R + RL.vcodes + ((ks2 * (D / 64) + mq) * 32 + lane) * 16);
      const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int mc = 4 * mq + e;
        uint32_t a0[4], a1[4];
        unpack_v(ws[e], a0, a1);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma16816(pacc[mc][nt], a0, bw[0][nt][0], bw[0][nt][1]);
          mma16816(pacc[mc][nt], a1, bw[1][nt][0], bw[1][nt][1]);
        }
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    zs[nt] += __shfl_xor_sync(0xffffffffu, zs[nt], 4);
    zs[nt] += __shfl_xor_sync(0xffffffffu, zs[nt], 8);
    zs[nt] += __shfl_xor_sync(0xffffffffu, zs[nt], 16);
  }
#pragma unroll
  for (int mc = 0; mc < D / 16; ++mc) {
    const float c0 = __half2float(Vc[16 * mc + g]), c1 = __half2float(Vc[16 * mc + g + 8]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      st.o[mc][nt][0] = fmaf(st.o[mc][nt][0], alpha[nt], c0 * ((pacc[mc][nt][0] + pacc[mc][nt][1]) + zs[nt]));
      st.o[mc][nt][1] = fmaf(st.o[mc][nt][1], alpha[nt], c1 * ((pacc[mc][nt][2] + pacc[mc][nt][3]) + zs[nt]));
    }
  }
}

template <int D, int NT>
__global__ void __launch_bounds__(kDecWarps * 32) decode_kernel(DecodeParams p) {
  using S = DecodeShape<D, NT>;
  constexpr int NH = S::kNH;
  constexpr int REC = S::kRec;
  constexpr int QLD = S::kQld;
  extern __shared__ __align__(128) uint8_t smem_d[];
  uint8_t* recs = smem_d;
  float* qsm = reinterpret_cast<float*>(smem_d + S::kRecBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_d + S::kRecBytes + S::kQBytes);

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cap = p.max_pages * kTile + (kTile - 1);  // sealed pages must fit the block table
  int len = p.seq_lens[b];
  if (len < 0 || len > cap) {
    if (threadIdx.x == 0 && split == 0 && h == 0) flag_error(p.status, KVARN_DEV_SEQ_TOO_LONG);
    len = len < 0 ? 0 : cap;
  }
  const int n_sealed = len / kTile, n_part = len % kTile;
  const int n_ss = (n_sealed + p.pages_per_split - 1) / p.pages_per_split;
  const bool partial_split = (split == n_ss) && n_part > 0;
  if (split >= n_ss && !partial_split) return;
  if (partial_split && (p.partial_k == nullptr || p.partial_v == nullptr)) {
    if (threadIdx.x == 0) flag_error(p.status, KVARN_DEV_NO_PARTIAL);
    return;
  }

  // ---- queries of this kv head's group: rotated (sealed pages) or original (partial tile) ----
  for (int hl = warp; hl < NH; hl += kDecWarps) {
    float v[D / 32];
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      const int j = lane * (D / 32) + e;
      v[e] = (hl < p.group && j < p.d0)
                 ? __half2float(p.q[((int64_t)b * p.num_q_heads + h * p.group + hl) * p.d0 + j])
                 : 0.0f;
    }
    float sc = p.qscale;
    if (!partial_split) {
      warp_fwht<D>(v, lane);
      sc *= inv_sqrt_d<D>();
    }
#pragma unroll
    for (int e = 0; e < D / 32; ++e) qsm[hl * QLD + lane * (D / 32) + e] = v[e] * sc;
  }
  __syncthreads();

  float* part_base = p.part + ((int64_t)(b * p.num_q_heads + h * p.group) * p.max_splits + split) * (D + 4);
  const int64_t head_stride = (int64_t)p.max_splits * (D + 4);

  if (!partial_split) {
    WarpAcc<D, NT> st;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      st.m[nt] = -INFINITY;
      st.l[nt] = 0.0f;
#pragma unroll
      for (int mc = 0; mc < D / 16; ++mc) st.o[mc][nt][0] = st.o[mc][nt][1] = 0.0f;
    }
    const int first = split * p.pages_per_split;
    const int last = min(n_sealed, first + p.pages_per_split);
    const int cnt = (last - first - warp + kDecWarps - 1) / kDecWarps;
    uint64_t* bar = bars + warp * kDecStages;
    uint8_t* rb = recs + warp * kDecStages * REC;
    const int32_t* bt = p.block_table + (int64_t)b * p.max_pages;
    auto page_src = [&](int k) -> const uint8_t* {
      int64_t id = bt[first + warp + kDecWarps * k];
      if (id < 0 || id >= p.num_pool_pages) {
        flag_error(p.status, KVARN_DEV_BAD_PAGE_ID);
        id = 0;
      }
      return p.pool + (id * p.num_kv_heads + h) * REC;
    };
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < kDecStages; ++s) mbar_init(&bar[s], 1);
      fence_mbar_init();
      for (int k = 0; k < kDecStages && k < cnt; ++k) {
        mbar_expect_tx(&bar[k], REC);
        bulk_copy_g2s(rb + k * REC, page_src(k), REC, &bar[k]);
      }
    }
    __syncwarp();
    for (int k = 0; k < cnt; ++k) {
      const int s = k % kDecStages;
      if (!mbar_wait(&bar[s], (k / kDecStages) & 1)) {
        // a copy never arrived: report, drain the copies this warp still has in flight, stop
        if (lane == 0) flag_error(p.status, KVARN_DEV_WAIT_TIMEOUT);
        for (int k2 = k + 1; k2 < cnt && k2 < k + kDecStages; ++k2)
          mbar_wait(&bar[k2 % kDecStages], (k2 / kDecStages) & 1);
        break;
      }
      process_page<D, NT>(rb + s * REC, qsm, lane, st);
      __syncwarp();
      if (lane == 0 && k + kDecStages < cnt) {
        fence_proxy_async_smem();
        mbar_expect_tx(&bar[s], REC);
        bulk_copy_g2s(rb + s * REC, page_src(k + kDecStages), REC, &bar[s]);
      }
    }
    // ---- merge the warps of this CTA ----
    __syncthreads();  // every warp is done with its record buffers
    float* mS = reinterpret_cast<float*>(recs);
    float* lS = mS + kDecWarps * NH;
    float* oS = lS + kDecWarps * NH;
    const int g = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float l = st.l[nt];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      const int hl = 4 * nt + tq;
      if (g == 0) {
        mS[warp * NH + hl] = st.m[nt];
        lS[warp * NH + hl] = l;
      }
#pragma unroll
      for (int mc = 0; mc < D / 16; ++mc) {
        oS[(warp * NH + hl) * D + 16 * mc + g] = st.o[mc][nt][0];
        oS[(warp * NH + hl) * D + 16 * mc + g + 8] = st.o[mc][nt][1];
      }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < p.group * D; idx += blockDim.x) {
      const int hl = idx / D, j = idx - hl * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, mS[w * NH + hl]);
      float o = 0.0f, l = 0.0f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float sc = exp2f(mS[w * NH + hl] - M);
        o = fmaf(sc, oS[(w * NH + hl) * D + j], o);
        l = fmaf(sc, lS[w * NH + hl], l);
      }
      float* dst = part_base + hl * head_stride;
      dst[4 + j] = o;
      if (j == 0) {
        dst[0] = M;
        dst[1] = l;
      }
    }
    return;
  }

  // ---- partial tile: raw fp16 tokens in the original basis ---------------------------------
  {
    constexpr int E = D / 32;
    float m[NH], l[NH], acc[NH][E];
#pragma unroll
    for (int hl = 0; hl < NH; ++hl) {
      m[hl] = -INFINITY;
      l[hl] = 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[hl][e] = 0.0f;
    }
    const int64_t base = ((int64_t)b * p.num_kv_heads + h) * kTile * p.d0;
    for (int t = warp; t < n_part; t += kDecWarps) {
      float kv[E], vv[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int j = lane + 32 * e;
        kv[e] = j < p.d0 ? __half2float(p.partial_k[base + (int64_t)t * p.d0 + j]) : 0.0f;
        vv[e] = j < p.d0 ? __half2float(p.partial_v[base + (int64_t)t * p.d0 + j]) : 0.0f;
      }
#pragma unroll
      for (int hl = 0; hl < NH; ++hl) {
        if (hl >= p.group) break;
        float dot = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot = fmaf(qsm[hl * QLD + lane + 32 * e], kv[e], dot);
#pragma unroll
        for (int msk = 16; msk > 0; msk >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, msk);
        const float mnew = fmaxf(m[hl], dot);
        const float a = exp2f(m[hl] - mnew), pv = exp2f(dot - mnew);
        m[hl] = mnew;
        l[hl] = fmaf(l[hl], a, pv);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[hl][e] = fmaf(acc[hl][e], a, pv * vv[e]);
      }
    }
    float* mS = reinterpret_cast<float*>(recs);
    float* lS = mS + kDecWarps * NH;
    float* oS = lS + kDecWarps * NH;
#pragma unroll
    for (int hl = 0; hl < NH; ++hl) {
      if (lane == 0) {
        mS[warp * NH + hl] = m[hl];
        lS[warp * NH + hl] = l[hl];
      }
#pragma unroll
      for (int e = 0; e < E; ++e) oS[(warp * NH + hl) * D + lane + 32 * e] = acc[hl][e];
    }
    __syncthreads();
    // merge warps, rotate o into the basis of the sealed splits, store
    for (int hl = warp; hl < p.group; hl += kDecWarps) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, mS[w * NH + hl]);
      float v[E], lsum = 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = 0.0f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float sc = exp2f(mS[w * NH + hl] - M);
        lsum = fmaf(sc, lS[w * NH + hl], lsum);
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = fmaf(sc, oS[(w * NH + hl) * D + lane * E + e], v[e]);
      }
      warp_fwht<D>(v, lane);
      float* dst = part_base + hl * head_stride;
#pragma unroll
      for (int e = 0; e < E; ++e) dst[4 + lane * E + e] = v[e] * inv_sqrt_d<D>();
      if (lane == 0) {
        dst[0] = M;
        dst[1] = lsum;
      }
    }
  }
}

// One warp per (sequence, query head): merge the splits, normalise, undo the rotation.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(DecodeParams p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (gw >= p.batch * p.num_q_heads) return;
  const int b = gw / p.num_q_heads;
  const int cap = p.max_pages * kTile + (kTile - 1);
  int len = p.seq_lens[b];
  len = len < 0 ? 0 : (len > cap ? cap : len);
  const int n_sealed = len / kTile;
  const int n_splits = (n_sealed + p.pages_per_split - 1) / p.pages_per_split + (len % kTile > 0 ? 1 : 0);
  float v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = 0.0f;
  if (n_splits > 0) {
    const float* base = p.part + (int64_t)gw * p.max_splits * (D + 4);
    float M = -INFINITY;
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, base[s * (D + 4)]);
    float lsum = 0.0f;
    for (int s = 0; s < n_splits; ++s) {
      const float* src = base + s * (D + 4);
      const float sc = exp2f(src[0] - M);
      lsum = fmaf(sc, src[1], lsum);
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = fmaf(sc, src[4 + lane * E + e], v[e]);
    }
    const float inv = inv_sqrt_d<D>() / lsum;
    warp_fwht<D>(v, lane);
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] *= inv;
  }
  __half* dst = p.out + (int64_t)gw * p.d0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane * E + e;
    if (j < p.d0) dst[j] = __float2half_rn(v[e]);
  }
}

template <int D, int NT>
static int launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  using S = DecodeShape<D, NT>;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(decode_kernel<D, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::kSmemBytes) != cudaSuccess)
      return KVARN_ERR_CUDA;
    attr_set = true;
  }
  dim3 grid(p.max_splits, p.num_kv_heads, p.batch);
  decode_kernel<D, NT><<<grid, kDecWarps * 32, S::kSmemBytes, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return KVARN_ERR_CUDA;
  const int warps = p.batch * p.num_q_heads;
  combine_kernel<D><<<(warps + 3) / 4, 128, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA;
}

int launch_decode_any(int d, int nt, const DecodeParams& p, cudaStream_t stream) {
  if (nt == 1) {
    if (d == 64) return launch_decode_t<64, 1>(p, stream);
    if (d == 128) return launch_decode_t<128, 1>(p, stream);
    if (d == 256) return launch_decode_t<256, 1>(p, stream);
  } else if (nt == 2) {
    if (d == 64) return launch_decode_t<64, 2>(p, stream);
    if (d == 128) return launch_decode_t<128, 2>(p, stream);
  }
  return KVARN_ERR_UNSUPPORTED;
}

int decode_smem_bytes(int d, int nt) {
  if (nt == 1) {
    if (d == 64) return DecodeShape<64, 1>::kSmemBytes;
    if (d == 128) return DecodeShape<128, 1>::kSmemBytes;
    if (d == 256) return DecodeShape<256, 1>::kSmemBytes;
  } else if (nt == 2) {
    if (d == 64) return DecodeShape<64, 2>::kSmemBytes;
    if (d == 128) return DecodeShape<128, 2>::kSmemBytes;
  }
  return -1;
}

}  // namespace kvarn
