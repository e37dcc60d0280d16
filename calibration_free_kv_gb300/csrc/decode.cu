// KVarN paged decode (and chunked-prefill) attention over the packed cache (sm_103a).
//
// Math (rotated basis, R = H_d / sqrt(d) orthonormal and symmetric):
//   logit_t = tau q . K_t = tau (qR) . (K_t R) = tau r_t ( sum_j q~_j s'_j code_tj + sum_j q~_j z'_j )
//   o = sum_t p_t V_t = ( sum_t p_t V~_t ) R,  V~_tj = c_j ( code_tj s'_t + z'_t )
// [vatt §四個步驟: the rotation is orthonormal so attention scores are unchanged;
//  hotdry §非对称量化与尺度折叠: the folded scales are multiplied back at read time]
//
// decode_kernel: by default (decode) persistent CTAs, two per SM, each walking one range of
// the segment-weighted page partition (decode_util.cuh) as segments of one (sequence, kv head)
// row; otherwise (prefill, and the split form kept for comparison) grid (split, kv head x
// query block, sequence), a CTA owning up to `pages_per_split` sealed pages of one (sequence,
// kv head), or the raw fp16 partial tile.  Either way a CTA serves up to 4 * NT query vectors
// of that kv head (decode: its G query heads; prefill: blocks of the chunk's C * G query
// vectors).  Its warps (8, or 4 where 8 page slots do not fit) take whole pages round-robin.  Every warp owns two shared-memory slots, one for the K half of a page
// record and one for the V half, each filled by a 1-D bulk copy completed on its own
// mbarrier: the K half of the next page streams in while the warp works on the current
// page's V half, and the V half of the next page while it works on the next K half.
//   QK:  m16n8k16 MMAs, A = codes [token x channel] (4- or 2-bit), B = q~ . s'_K split into fp16
//        hi + lo (columns: 4 heads x {hi, lo}); hi = fp16(qh s'), lo = fp16(ql s' + (qh s' -
//        hi)) with q~ = qh + ql pre-split once per CTA and the product error taken exactly
//        by an fp16 fma.
//   softmax: online, log2 domain (tau log2(e) folded into q~).
//   PV:  m16n8k16 MMAs, A = codes^T [channel x token] (2- or 4-bit), B = p . s'_V split hi + lo,
//        moved from the QK accumulator layout with movmatrix.trans.
// Codes enter the MMAs as exact fp16 subnormals: masking a code into the low mantissa bits
// of a zero exponent gives code * 2^-24 (code * 2^-22 .. 2^-18 for higher bit positions), so
// unpacking costs one AND per two codes; the powers of two are folded into B and into the
// fp32 results.  The CTA merges its warps and writes (m, l, unnormalised o~) for its split (G = 8
// and prefill use NT = 2 with the heads on the MMA's M axis instead, qk_page_t / pv_page_t).
// combine_kernel attends to the raw open tiles (decode), merges the splits, divides by l,
// undoes the rotation and stores fp16.  chunk_tc_kernel (chunk_kernel at head_dim 256) adds
// the causal part of a prefill chunk as one more split.
#include "common.cuh"
#include "decode_util.cuh"
#include "params.cuh"

namespace kvarn {

constexpr int kMaxSmem = 232448;  // dynamic shared memory a CTA may opt in to

template <int D, int NT, int KB, int VB>
struct DecodeShape {
  static constexpr RecordLayout kRL = record_layout(D, KB, VB);
  static constexpr int kNH = 4 * NT;                 // head slots per kv head (G padded)
  static constexpr int kRec = kRL.bytes;
  static constexpr int kKHalf = kRL.vcodes;          // K codes + K metadata
  static constexpr int kVHalf = kRec - kKHalf;       // V codes + V metadata
  static constexpr int kQld = D + 8;                 // fp32 row stride of q in shared memory
  // q~ (fp32) for q~ . z'; 8 heads per warp take q~ . z' from the fp16 hi + lo parts instead
  static constexpr int kQBytes = NT == 2 ? 0 : kNH * kQld * 4;
  static constexpr int kQhBytes = 2 * kNH * (D / 2 + 4) * 4;  // q~ as fp16 hi and lo, padded rows
  // warps per CTA: 8, or 4 where 8 page slots would not fit in shared memory
  static constexpr int kWarps = 8 * kRec + kQBytes + kQhBytes + 8 * 16 <= kMaxSmem ? 8 : 4;
  static constexpr int kRecBytes = kWarps * kRec;    // one K slot + one V slot per warp
  // page slots, q, and the barriers: two per warp plus one for the raw partial tile
  static constexpr int kSmemBytes = kRecBytes + kQBytes + kQhBytes + (kWarps * 2 + 1) * 8;
  static_assert(kSmemBytes <= kMaxSmem, "page slots fit in shared memory");
  static_assert(kRecBytes >= (kWarps * kNH * (D + 3) + 2 * kNH) * 4, "the merge scratch fits the page slots");
  // two CTAs per SM where their shared memory fits (registers then capped at 128 a thread)
  static constexpr int kMinBlocks = 2 * (kSmemBytes + 1024) <= 233472 ? 2 : 1;
};

// Power-of-two factors on the fp16 hi + lo query of the QK operand for channels 0..7 (kH0) and
// 8..15 (kH1) of every 16, and on the MMA sum (kAcc).  4- and 2-bit codes of channels 8..15 sit
// 4 / 2 bits higher in their fp16 subnormals, so those channels take 1/16 / 1/4 of the others'
// factor.  q is lifted so that the lo parts of q and of q s' stay out of the fp16 subnormal
// range (the code sum cancels against q~ . z', so their precision shows in the logits): by
// 2^4 / 2^2 at 4 / 2 bits (channels 8..15 at 1), by 2^8 at 8 bits, whose scale s' is smallest.
template <int KB>
struct QkScale {
  static constexpr float kH0 = KB == 8 ? 256.0f : (KB == 4 ? 16.0f : 4.0f);
  static constexpr float kH1 = KB == 8 ? 256.0f : 1.0f;
  static constexpr float kAcc = kTwo24 / kH0;
};

// Power-of-two factors on the PV weights p s' of tokens 0..7 (h = 0) and 8..15 (h = 1) of
// 16-token block f of a pair, and on the MMA sum (kAcc).  2-bit codes of token half h of block
// f sit 4f + 2h bits higher in their fp16 subnormals, 4-bit codes of half 1 four bits higher:
// those weights take the inverse.  No lift (kLift = 1): unlike the QK operand, lifting the
// weights by 2^4 left every decode error unchanged, and the weights keep the full fp16 range.
template <int VB>
struct PvScale {
  static_assert(VB == 2 || VB == 4, "2- or 4-bit V codes");
  static constexpr float kLift = 1.0f;
  static constexpr float kAcc = kTwo24 / kLift;
  __device__ static constexpr float c(int f, int h) {
    return kLift * (VB == 2 ? 1.0f / float(1 << (4 * f + 2 * h)) : (h ? 1.0f / 16.0f : 1.0f));
  }
};

template <int D, int NT>
struct WarpAcc {
  float m[NT], l[NT];
  float o[D / 16][NT][2];  // head 4nt + tq, channels 16mc + g + 8r (rotated basis)
};

// One column pair of the QK B operand for the lane's head: fp16 hi = qh s' (lanes with even g)
// or lo = ql s' + (qh s' - hi) (odd g); the fma takes the rounding error of qh s' exactly.
__device__ __forceinline__ uint32_t b_split(__half2 qh, __half2 ql, __half2 s, bool lo) {
  const __half2 hi = __hmul2(qh, s);
  const __half2 err = __hfma2(qh, s, __hneg2(hi));
  return h2u(lo ? __hfma2(ql, s, err) : hi);
}

// QK of one whole page from its K half Rk: logits -> probabilities lg (tokens 16mi + g + 8r
// of head 4nt + tq), online-softmax state updated, alpha = rescale of the previous state.
template <int D, int NT, int KB, int VB>
__device__ __forceinline__ void qk_page(const uint8_t* __restrict__ Rk, const float* __restrict__ qsm,
                                        const uint2* __restrict__ qhl, int lane, WarpAcc<D, NT>& st,
                                        float (&lg)[8][NT][2], float (&alpha)[NT]) {
  constexpr RecordLayout RL = record_layout(D, KB, VB);
  constexpr int QLD = DecodeShape<D, NT, KB, VB>::kQld;
  constexpr int QH = D / 2 + 4;  // row stride of qhl (one entry per channel pair)
  const int g = lane >> 2, tq = lane & 3;
  const __half2* Ks2 = reinterpret_cast<const __half2*>(Rk + RL.kscale);
  const __half2* Kz2 = reinterpret_cast<const __half2*>(Rk + RL.kzero);
  const __half* Kr = reinterpret_cast<const __half*>(Rk + RL.kfactor);

  uint32_t bq[D / 16][NT][2];
  float2 qz2[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) qz2[nt] = make_float2(0.0f, 0.0f);
  const bool lo_col = (g & 1) != 0;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int jp = 8 * kk + tq;  // channel pair (16kk + 2tq, +1); jp + 4: (16kk + 2tq + 8, +9)
    const __half2 s0 = Ks2[jp], s1 = Ks2[jp + 4];
    const float2 z0 = __half22float2(Kz2[jp]), z1 = __half22float2(Kz2[jp + 4]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int head = 4 * nt + (g >> 1);
      const float4 q4 = *reinterpret_cast<const float4*>(qsm + head * QLD + 16 * kk + 4 * tq);
      qz2[nt] = fma2(make_float2(q4.x, q4.y), z0, qz2[nt]);
      qz2[nt] = fma2(make_float2(q4.z, q4.w), z1, qz2[nt]);
      const uint2 u0 = qhl[head * QH + jp], u1 = qhl[head * QH + jp + 4];
      bq[kk][nt][0] = b_split(u2h2(u0.x), u2h2(u0.y), s0, lo_col);
      bq[kk][nt][1] = b_split(u2h2(u1.x), u2h2(u1.y), s1, lo_col);
    }
  }
  float qzm[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float v = qz2[nt].x + qz2[nt].y;
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    qzm[nt] = __shfl_sync(0xffffffffu, v, 8 * tq);  // head 4nt + tq lives in lanes g = 2tq
  }
  auto logits = [&](int mi, const float (&acc)[NT][4], float cf) {
    const float2 r = make_float2(__half2float(Kr[16 * mi + g]), __half2float(Kr[16 * mi + g + 8]));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 t = add2(make_float2(acc[nt][0], acc[nt][2]), make_float2(acc[nt][1], acc[nt][3]));
      const float2 u = mul2(fma2(t, make_float2(cf, cf), make_float2(qzm[nt], qzm[nt])), r);
      lg[mi][nt][0] = u.x;
      lg[mi][nt][1] = u.y;
    }
  };
  if constexpr (KB == 4) {  // one word per fragment (token block mi, channel block kk)
#pragma unroll
    for (int mi = 0; mi < 8; ++mi) {
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
#pragma unroll
      for (int kq = 0; kq < D / 64; ++kq) {
        const uint4 w4 =
            *reinterpret_cast<const uint4*>(Rk + RL.kcodes + ((mi * (D / 64) + kq) * 32 + lane) * 16);
        const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t a[4];
          unpack_k(ws[e], a);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt], a, bq[4 * kq + e][nt][0], bq[4 * kq + e][nt][1]);
        }
      }
      logits(mi, acc, QkScale<KB>::kAcc);
    }
  } else if constexpr (KB == 8) {  // two words per fragment; a 16-byte load holds two
#pragma unroll
    for (int mi = 0; mi < 8; ++mi) {
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
#pragma unroll
      for (int kp = 0; kp < D / 32; ++kp) {
        const uint4 w4 =
            *reinterpret_cast<const uint4*>(Rk + RL.kcodes + ((mi * (D / 32) + kp) * 32 + lane) * 16);
        uint32_t a0[4], a1[4];
        unpack_k8(w4.x, w4.y, a0);
        unpack_k8(w4.z, w4.w, a1);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma16816(acc[nt], a0, bq[2 * kp][nt][0], bq[2 * kp][nt][1]);
          mma16816(acc[nt], a1, bq[2 * kp + 1][nt][0], bq[2 * kp + 1][nt][1]);
        }
      }
      logits(mi, acc, QkScale<KB>::kAcc);
    }
  } else {  // 2-bit: one word per channel block kk holds token blocks 2mi2 and 2mi2 + 1
    static_assert(KB == 2, "2-, 4- or 8-bit K codes");
#pragma unroll
    for (int mi2 = 0; mi2 < 4; ++mi2) {
      float acc0[NT][4], acc1[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc0[nt][e] = acc1[nt][e] = 0.0f;
#pragma unroll
      for (int kq = 0; kq < D / 64; ++kq) {
        const uint4 w4 =
            *reinterpret_cast<const uint4*>(Rk + RL.kcodes + ((mi2 * (D / 64) + kq) * 32 + lane) * 16);
        const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t a0[4], a1[4];
          unpack_v(ws[e], a0, a1);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(acc0[nt], a0, bq[4 * kq + e][nt][0], bq[4 * kq + e][nt][1]);
            mma16816(acc1[nt], a1, bq[4 * kq + e][nt][0], bq[4 * kq + e][nt][1]);
          }
        }
      }
      logits(2 * mi2, acc0, QkScale<KB>::kAcc);
      logits(2 * mi2 + 1, acc1, QkScale<KB>::kAcc * 0.0625f);  // the odd block's codes sit 4 bits higher
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float mx = fmaxf(lg[0][nt][0], lg[0][nt][1]);
#pragma unroll
    for (int mi = 1; mi < 8; ++mi) mx = fmax3(mx, lg[mi][nt][0], lg[mi][nt][1]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mnew = fmaxf(st.m[nt], mx);
    alpha[nt] = ex2_approx(st.m[nt] - mnew);
    st.m[nt] = mnew;
    float2 ps = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int mi = 0; mi < 8; ++mi) {
      const float2 d = sub2(make_float2(lg[mi][nt][0], lg[mi][nt][1]), make_float2(mnew, mnew));
      const float2 pv = make_float2(ex2_approx(d.x), ex2_approx(d.y));
      lg[mi][nt][0] = pv.x;
      lg[mi][nt][1] = pv.y;
      ps = add2(ps, pv);
    }
    st.l[nt] = fmaf(st.l[nt], alpha[nt], ps.x + ps.y);
  }
}

// PV of one whole page from its V half Rv with the probabilities of qk_page.
template <int D, int NT, int KB, int VB>
__device__ __forceinline__ void pv_page(const uint8_t* __restrict__ Rv, const float (&lg)[8][NT][2],
                                        const float (&alpha)[NT], int lane, WarpAcc<D, NT>& st) {
  constexpr RecordLayout RL = record_layout(D, KB, VB);
  const int g = lane >> 2;
  const __half* Vs = reinterpret_cast<const __half*>(Rv + (RL.vscale - RL.vcodes));
  const __half* Vz = reinterpret_cast<const __half*>(Rv + (RL.vzero - RL.vcodes));
  const __half* Vc = reinterpret_cast<const __half*>(Rv + (RL.vfactor - RL.vcodes));
  float pacc[D / 16][NT][4];
#pragma unroll
  for (int mc = 0; mc < D / 16; ++mc)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) pacc[mc][nt][0] = pacc[mc][nt][1] = pacc[mc][nt][2] = pacc[mc][nt][3] = 0.0f;
  float2 zs2[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) zs2[nt] = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int ks2 = 0; ks2 < 4; ++ks2) {
    uint32_t bw[2][NT][2];
#pragma unroll
    for (int f = 0; f < 2; ++f) {
      const int ks = 2 * ks2 + f;
      // token scales times the PvScale factors of this block (h = 0: rows g); powers of two
      // keep the products exact
      const float c0 = PvScale<VB>::c(f, 0), c1 = PvScale<VB>::c(f, 1);
      const float2 svc = make_float2(__half2float(Vs[16 * ks + g]) * c0, __half2float(Vs[16 * ks + g + 8]) * c1);
      const float2 zv = make_float2(__half2float(Vz[16 * ks + g]), __half2float(Vz[16 * ks + g + 8]));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float2 pp = make_float2(lg[ks][nt][0], lg[ks][nt][1]);
        zs2[nt] = fma2(pp, zv, zs2[nt]);
        const float2 w = mul2(pp, svc);
        const __half2 hi = __floats2half2_rn(w.x, w.y);
        const float2 r = sub2(w, __half22float2(hi));
        const __half2 lo = __floats2half2_rn(r.x, r.y);
        bw[f][nt][0] = movmatrix_trans(h2u(__lows2half2(hi, lo)));   // (hi, lo) of row g
        bw[f][nt][1] = movmatrix_trans(h2u(__highs2half2(hi, lo)));  // (hi, lo) of row g + 8
      }
    }
#pragma unroll
    for (int mq = 0; mq < D / 64; ++mq) {
      uint32_t ws0[4], ws1[4];  // 2-bit: token blocks 2ks2 and 2ks2 + 1 share words; 4-bit: one each
      if constexpr (VB == 2) {
        const uint4 w4 = *reinterpret_cast<const uint4*>(Rv + ((ks2 * (D / 64) + mq) * 32 + lane) * 16);
        ws0[0] = w4.x; ws0[1] = w4.y; ws0[2] = w4.z; ws0[3] = w4.w;
      } else {
        static_assert(VB == 4, "2- or 4-bit V codes");
        const uint4 w0 = *reinterpret_cast<const uint4*>(Rv + (((2 * ks2) * (D / 64) + mq) * 32 + lane) * 16);
        const uint4 w1 = *reinterpret_cast<const uint4*>(Rv + (((2 * ks2 + 1) * (D / 64) + mq) * 32 + lane) * 16);
        ws0[0] = w0.x; ws0[1] = w0.y; ws0[2] = w0.z; ws0[3] = w0.w;
        ws1[0] = w1.x; ws1[1] = w1.y; ws1[2] = w1.z; ws1[3] = w1.w;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int mc = 4 * mq + e;
        uint32_t a0[4], a1[4];
        if constexpr (VB == 2) {
          unpack_v(ws0[e], a0, a1);
        } else {
          unpack_k(ws0[e], a0);
          unpack_k(ws1[e], a1);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma16816(pacc[mc][nt], a0, bw[0][nt][0], bw[0][nt][1]);
          mma16816(pacc[mc][nt], a1, bw[1][nt][0], bw[1][nt][1]);
        }
      }
    }
  }
  float zs[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    zs[nt] = zs2[nt].x + zs2[nt].y;
    zs[nt] += __shfl_xor_sync(0xffffffffu, zs[nt], 4);
    zs[nt] += __shfl_xor_sync(0xffffffffu, zs[nt], 8);
    zs[nt] += __shfl_xor_sync(0xffffffffu, zs[nt], 16);
  }
#pragma unroll
  for (int mc = 0; mc < D / 16; ++mc) {
    const float2 cj = make_float2(__half2float(Vc[16 * mc + g]), __half2float(Vc[16 * mc + g + 8]));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float2 t = add2(make_float2(pacc[mc][nt][0], pacc[mc][nt][2]), make_float2(pacc[mc][nt][1], pacc[mc][nt][3]));
      t = mul2(fma2(t, make_float2(PvScale<VB>::kAcc, PvScale<VB>::kAcc), make_float2(zs[nt], zs[nt])), cj);
      const float2 o = fma2(make_float2(st.o[mc][nt][0], st.o[mc][nt][1]), make_float2(alpha[nt], alpha[nt]), t);
      st.o[mc][nt][0] = o.x;
      st.o[mc][nt][1] = o.y;
    }
  }
}

// ---- eight query vectors per warp (NT = 2): the heads on the MMA's M axis --------------------
// Rows g and g + 8 of a 16-row A operand hold head g's fp16 hi and lo parts and the page's codes
// are the B operand: an A-fragment word of 16 tokens (or 16 channels, for V) holds exactly the
// B fragments of two 8-wide blocks.  QK then leaves head g's logits of tokens 2tq, 2tq + 1 of
// each 8-token block in lane (g, tq), which is the layout of PV's A operand: no transposes, and
// each lane splits one head's operands instead of building a B column pair per head slot.

template <int D>
struct WarpAccT {
  float m[1], l[1];   // head g; l is this lane's share until the CTA merge sums the tq lanes
  float o[D / 8][2];  // head g, channels 8cb + 2tq, +1 (rotated basis)
};

// qh s (rounded) and the rest of (qh + ql) s, with the rounding error of qh s taken exactly.
__device__ __forceinline__ void split_hi_lo(__half2 qh, __half2 ql, __half2 s, uint32_t& hi,
                                            uint32_t& lo) {
  const __half2 h = __hmul2(qh, s);
  hi = h2u(h);
  lo = h2u(__hfma2(ql, s, __hfma2(qh, s, __hneg2(h))));
}

// QK of one page for head g: probabilities of tokens 8b + 2tq, +1 in lg[b][0], online state
// updated, alpha = rescale of the previous state.
template <int D, int KB, int VB>
__device__ __forceinline__ void qk_page_t(const uint8_t* __restrict__ Rk, const float* __restrict__ /* no fp32 q~ */,
                                          const uint2* __restrict__ qhl, int lane, WarpAccT<D>& st,
                                          float (&lg)[16][1][2], float (&alpha)[1]) {
  constexpr RecordLayout RL = record_layout(D, KB, VB);
  constexpr int QH = D / 2 + 4;
  const int g = lane >> 2, tq = lane & 3;
  const __half2* Ks2 = reinterpret_cast<const __half2*>(Rk + RL.kscale);
  const __half2* Kz2 = reinterpret_cast<const __half2*>(Rk + RL.kzero);
  const __half2* Kr2 = reinterpret_cast<const __half2*>(Rk + RL.kfactor);
  uint32_t aq[D / 16][4];  // head g: rows g = hi, g + 8 = lo; channels 2tq.. and 2tq + 8..
  // q~ . z' from q~ = hi + lo, with the operand factors of QkScale undone
  constexpr float kUndo0 = 1.0f / QkScale<KB>::kH0, kUndo1 = 1.0f / QkScale<KB>::kH1;
  float2 qz2 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int jp = 8 * kk + tq;
    const __half2 s0 = Ks2[jp], s1 = Ks2[jp + 4];
    const float2 z0 = __half22float2(Kz2[jp]), z1 = __half22float2(Kz2[jp + 4]);
    const uint2 u0 = qhl[g * QH + jp], u1 = qhl[g * QH + jp + 4];
    float2 q0 = add2(__half22float2(u2h2(u0.x)), __half22float2(u2h2(u0.y)));
    float2 q1 = add2(__half22float2(u2h2(u1.x)), __half22float2(u2h2(u1.y)));
    if constexpr (QkScale<KB>::kH0 != 1.0f) q0 = mul2(q0, make_float2(kUndo0, kUndo0));
    if constexpr (QkScale<KB>::kH1 != 1.0f) q1 = mul2(q1, make_float2(kUndo1, kUndo1));
    qz2 = fma2(q0, z0, qz2);
    qz2 = fma2(q1, z1, qz2);
    split_hi_lo(u2h2(u0.x), u2h2(u0.y), s0, aq[kk][0], aq[kk][1]);
    split_hi_lo(u2h2(u1.x), u2h2(u1.y), s1, aq[kk][2], aq[kk][3]);
  }
  float qz = qz2.x + qz2.y;
  qz += __shfl_xor_sync(0xffffffffu, qz, 1);
  qz += __shfl_xor_sync(0xffffffffu, qz, 2);
  // 8-token block b: rows g (hi) + g + 8 (lo) of columns 2tq, 2tq + 1
  auto logits = [&](int b, const float (&acc)[4], float cf) {
    const float2 r = __half22float2(Kr2[4 * b + tq]);
    const float2 t = add2(make_float2(acc[0], acc[1]), make_float2(acc[2], acc[3]));
    const float2 u = mul2(fma2(t, make_float2(cf, cf), make_float2(qz, qz)), r);
    lg[b][0][0] = u.x;
    lg[b][0][1] = u.y;
  };
  if constexpr (KB == 4) {  // word (16 tokens x 16 channels): tokens g -> a0, a2; g + 8 -> a1, a3
#pragma unroll
    for (int mi = 0; mi < 8; ++mi) {
      float acc0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int kq = 0; kq < D / 64; ++kq) {
        const uint4 w4 =
            *reinterpret_cast<const uint4*>(Rk + RL.kcodes + ((mi * (D / 64) + kq) * 32 + lane) * 16);
        const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t a[4];
          unpack_k(ws[e], a);
          mma16816(acc0, aq[4 * kq + e], a[0], a[2]);
          mma16816(acc1, aq[4 * kq + e], a[1], a[3]);
        }
      }
      logits(2 * mi, acc0, QkScale<KB>::kAcc);
      logits(2 * mi + 1, acc1, QkScale<KB>::kAcc);
    }
  } else if constexpr (KB == 8) {  // two words per 16 x 16 block; a 16-byte load holds two blocks
#pragma unroll
    for (int mi = 0; mi < 8; ++mi) {
      float acc0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int kp = 0; kp < D / 32; ++kp) {
        const uint4 w4 =
            *reinterpret_cast<const uint4*>(Rk + RL.kcodes + ((mi * (D / 32) + kp) * 32 + lane) * 16);
        uint32_t a[4];
        unpack_k8(w4.x, w4.y, a);
        mma16816(acc0, aq[2 * kp], a[0], a[2]);
        mma16816(acc1, aq[2 * kp], a[1], a[3]);
        unpack_k8(w4.z, w4.w, a);
        mma16816(acc0, aq[2 * kp + 1], a[0], a[2]);
        mma16816(acc1, aq[2 * kp + 1], a[1], a[3]);
      }
      logits(2 * mi, acc0, QkScale<KB>::kAcc);
      logits(2 * mi + 1, acc1, QkScale<KB>::kAcc);
    }
  } else {  // 2-bit: one word holds 16-token blocks 2mi2 and 2mi2 + 1 of a channel block
    static_assert(KB == 2, "2-, 4- or 8-bit K codes");
#pragma unroll
    for (int mi2 = 0; mi2 < 4; ++mi2) {
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
#pragma unroll
      for (int kq = 0; kq < D / 64; ++kq) {
        const uint4 w4 =
            *reinterpret_cast<const uint4*>(Rk + RL.kcodes + ((mi2 * (D / 64) + kq) * 32 + lane) * 16);
        const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t a0[4], a1[4];
          unpack_v(ws[e], a0, a1);
          mma16816(acc[0], aq[4 * kq + e], a0[0], a0[2]);
          mma16816(acc[1], aq[4 * kq + e], a0[1], a0[3]);
          mma16816(acc[2], aq[4 * kq + e], a1[0], a1[2]);
          mma16816(acc[3], aq[4 * kq + e], a1[1], a1[3]);
        }
      }
      logits(4 * mi2, acc[0], QkScale<KB>::kAcc);
      logits(4 * mi2 + 1, acc[1], QkScale<KB>::kAcc);
      logits(4 * mi2 + 2, acc[2], QkScale<KB>::kAcc * 0.0625f);  // the odd 16-token block sits 4 bits higher
      logits(4 * mi2 + 3, acc[3], QkScale<KB>::kAcc * 0.0625f);
    }
  }
  float mx = fmaxf(lg[0][0][0], lg[0][0][1]);
#pragma unroll
  for (int b = 1; b < 16; ++b) mx = fmax3(mx, lg[b][0][0], lg[b][0][1]);
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const float mnew = fmaxf(st.m[0], mx);
  alpha[0] = ex2_approx(st.m[0] - mnew);
  st.m[0] = mnew;
  float2 ps = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int b = 0; b < 16; ++b) {
    const float2 d = sub2(make_float2(lg[b][0][0], lg[b][0][1]), make_float2(mnew, mnew));
    const float2 pv = make_float2(ex2_approx(d.x), ex2_approx(d.y));
    lg[b][0][0] = pv.x;
    lg[b][0][1] = pv.y;
    ps = add2(ps, pv);
  }
  st.l[0] = fmaf(st.l[0], alpha[0], ps.x + ps.y);
}

// PV of one page for head g with the probabilities of qk_page_t.  The A operands of all
// eight 16-token blocks are built first; the channels are then taken 64 at a time, so only
// one slice of accumulators is live (two CTAs of 8 warps fit an SM).
template <int D, int KB, int VB>
__device__ __forceinline__ void pv_page_t(const uint8_t* __restrict__ Rv, const float (&lg)[16][1][2],
                                          const float (&alpha)[1], int lane, WarpAccT<D>& st) {
  constexpr RecordLayout RL = record_layout(D, KB, VB);
  const int tq = lane & 3;
  const __half2* Vs2 = reinterpret_cast<const __half2*>(Rv + (RL.vscale - RL.vcodes));
  const __half2* Vz2 = reinterpret_cast<const __half2*>(Rv + (RL.vzero - RL.vcodes));
  const __half2* Vc2 = reinterpret_cast<const __half2*>(Rv + (RL.vfactor - RL.vcodes));
  uint32_t ap[8][4];  // 16-token block k: rows g = hi, g + 8 = lo of p s'_V
  float2 zs2 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int f = k & 1;
    // the PvScale factors of this block, h = token half
    const float c0 = PvScale<VB>::c(f, 0), c1 = PvScale<VB>::c(f, 1);
    const float2 pa = make_float2(lg[2 * k][0][0], lg[2 * k][0][1]);          // tokens 16k + 2tq, +1
    const float2 pb = make_float2(lg[2 * k + 1][0][0], lg[2 * k + 1][0][1]);  // tokens 16k + 8 + 2tq, +1
    zs2 = fma2(pa, __half22float2(Vz2[8 * k + tq]), zs2);
    zs2 = fma2(pb, __half22float2(Vz2[8 * k + 4 + tq]), zs2);
    const float2 wa = mul2(pa, mul2(__half22float2(Vs2[8 * k + tq]), make_float2(c0, c0)));
    const float2 wb = mul2(pb, mul2(__half22float2(Vs2[8 * k + 4 + tq]), make_float2(c1, c1)));
    const __half2 ha = __floats2half2_rn(wa.x, wa.y), hb = __floats2half2_rn(wb.x, wb.y);
    const float2 ra = sub2(wa, __half22float2(ha)), rb = sub2(wb, __half22float2(hb));
    ap[k][0] = h2u(ha);
    ap[k][1] = h2u(__floats2half2_rn(ra.x, ra.y));
    ap[k][2] = h2u(hb);
    ap[k][3] = h2u(__floats2half2_rn(rb.x, rb.y));
  }
  float zs = zs2.x + zs2.y;
  zs += __shfl_xor_sync(0xffffffffu, zs, 1);
  zs += __shfl_xor_sync(0xffffffffu, zs, 2);
#pragma unroll
  for (int mq = 0; mq < D / 64; ++mq) {  // channels 64mq..64mq + 63: 8-channel blocks 8mq + cl
    float pacc[8][4];
#pragma unroll
    for (int cl = 0; cl < 8; ++cl) pacc[cl][0] = pacc[cl][1] = pacc[cl][2] = pacc[cl][3] = 0.0f;
#pragma unroll
    for (int ks2 = 0; ks2 < 4; ++ks2) {
      uint32_t ws0[4], ws1[4];
      if constexpr (VB == 2) {
        const uint4 w4 = *reinterpret_cast<const uint4*>(Rv + ((ks2 * (D / 64) + mq) * 32 + lane) * 16);
        ws0[0] = w4.x; ws0[1] = w4.y; ws0[2] = w4.z; ws0[3] = w4.w;
      } else {
        static_assert(VB == 4, "2- or 4-bit V codes");
        const uint4 w0 = *reinterpret_cast<const uint4*>(Rv + (((2 * ks2) * (D / 64) + mq) * 32 + lane) * 16);
        const uint4 w1 = *reinterpret_cast<const uint4*>(Rv + (((2 * ks2 + 1) * (D / 64) + mq) * 32 + lane) * 16);
        ws0[0] = w0.x; ws0[1] = w0.y; ws0[2] = w0.z; ws0[3] = w0.w;
        ws1[0] = w1.x; ws1[1] = w1.y; ws1[2] = w1.z; ws1[3] = w1.w;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {  // channels 16(4mq + e)..: 8-channel blocks 2e (a0, a2), 2e + 1 (a1, a3)
        uint32_t a0[4], a1[4];
        if constexpr (VB == 2) {
          unpack_v(ws0[e], a0, a1);
        } else {
          unpack_k(ws0[e], a0);
          unpack_k(ws1[e], a1);
        }
        mma16816(pacc[2 * e], ap[2 * ks2], a0[0], a0[2]);
        mma16816(pacc[2 * e + 1], ap[2 * ks2], a0[1], a0[3]);
        mma16816(pacc[2 * e], ap[2 * ks2 + 1], a1[0], a1[2]);
        mma16816(pacc[2 * e + 1], ap[2 * ks2 + 1], a1[1], a1[3]);
      }
    }
#pragma unroll
    for (int cl = 0; cl < 8; ++cl) {
      const int cb = 8 * mq + cl;
      const float2 cj = __half22float2(Vc2[4 * cb + tq]);
      float2 t = add2(make_float2(pacc[cl][0], pacc[cl][1]), make_float2(pacc[cl][2], pacc[cl][3]));
      t = mul2(fma2(t, make_float2(PvScale<VB>::kAcc, PvScale<VB>::kAcc), make_float2(zs, zs)), cj);
      const float2 o = fma2(make_float2(st.o[cb][0], st.o[cb][1]), make_float2(alpha[0], alpha[0]), t);
      st.o[cb][0] = o.x;
      st.o[cb][1] = o.y;
    }
  }
}

// The per-warp decode path of NT head slots: NT = 2 takes the heads-on-M form above.
template <int D, int NT, int KB, int VB>
struct PagePath {
  using State = WarpAcc<D, NT>;
  static constexpr int kLgBlocks = 8, kLgNt = NT;
  __device__ static void init(State& st) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      st.m[nt] = -INFINITY;
      st.l[nt] = 0.0f;
#pragma unroll
      for (int mc = 0; mc < D / 16; ++mc) st.o[mc][nt][0] = st.o[mc][nt][1] = 0.0f;
    }
  }
  __device__ static void qk(const uint8_t* Rk, const float* qsm, const uint2* qhl, int lane, State& st,
                            float (&lg)[kLgBlocks][kLgNt][2], float (&alpha)[kLgNt]) {
    qk_page<D, NT, KB, VB>(Rk, qsm, qhl, lane, st, lg, alpha);
  }
  __device__ static void pv(const uint8_t* Rv, const float (&lg)[kLgBlocks][kLgNt][2],
                            const float (&alpha)[kLgNt], int lane, State& st) {
    pv_page<D, NT, KB, VB>(Rv, lg, alpha, lane, st);
  }
  // (m, l, o) of every head slot of this warp into the CTA's merge scratch
  __device__ static void store(const State& st, int warp, int lane, float* mS, float* lS, float* oS) {
    constexpr int NH = 4 * NT;
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
  }
};

template <int D, int KB, int VB>
struct PagePath<D, 2, KB, VB> {
  using State = WarpAccT<D>;
  static constexpr int kLgBlocks = 16, kLgNt = 1;
  __device__ static void init(State& st) {
    st.m[0] = -INFINITY;
    st.l[0] = 0.0f;
#pragma unroll
    for (int cb = 0; cb < D / 8; ++cb) st.o[cb][0] = st.o[cb][1] = 0.0f;
  }
  __device__ static void qk(const uint8_t* Rk, const float* qsm, const uint2* qhl, int lane, State& st,
                            float (&lg)[kLgBlocks][kLgNt][2], float (&alpha)[kLgNt]) {
    qk_page_t<D, KB, VB>(Rk, qsm, qhl, lane, st, lg, alpha);
  }
  __device__ static void pv(const uint8_t* Rv, const float (&lg)[kLgBlocks][kLgNt][2],
                            const float (&alpha)[kLgNt], int lane, State& st) {
    pv_page_t<D, KB, VB>(Rv, lg, alpha, lane, st);
  }
  __device__ static void store(const State& st, int warp, int lane, float* mS, float* lS, float* oS) {
    constexpr int NH = 8;
    const int g = lane >> 2, tq = lane & 3;
    float l = st.l[0];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (tq == 0) {
      mS[warp * NH + g] = st.m[0];
      lS[warp * NH + g] = l;
    }
#pragma unroll
    for (int cb = 0; cb < D / 8; ++cb)
      *reinterpret_cast<float2*>(&oS[(warp * NH + g) * D + 8 * cb + 2 * tq]) = make_float2(st.o[cb][0], st.o[cb][1]);
  }
};

// Warp-collective: the splits the tcgen05 kernel's partition gives row (b, h) (a cold path of
// the partial-tile launch, kept out of line).
__device__ __noinline__ int tc_row_segments(const DecodeParams& p, int b, int h, int lane) {
  return row_segments(p, page_partition(p, lane), b, h, lane);
}

template <int D, int NT, int KB, int VB>
__global__ void __launch_bounds__(DecodeShape<D, NT, KB, VB>::kWarps * 32, DecodeShape<D, NT, KB, VB>::kMinBlocks)
    decode_kernel(DecodeParams p) {
  using S = DecodeShape<D, NT, KB, VB>;
  constexpr int kDecWarps = S::kWarps;
  constexpr int NH = S::kNH;
  constexpr int REC = S::kRec;
  constexpr int KH = S::kKHalf;
  constexpr int VH = S::kVHalf;
  constexpr int QLD = S::kQld;
  constexpr int QH = D / 2 + 4;
  extern __shared__ __align__(128) uint8_t smem_d[];
  uint8_t* recs = smem_d;
  float* qsm = reinterpret_cast<float*>(smem_d + S::kRecBytes);
  uint2* qhl = reinterpret_cast<uint2*>(smem_d + S::kRecBytes + S::kQBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_d + S::kRecBytes + S::kQBytes + S::kQhBytes);
  uint64_t* pbar = bars + 2 * kDecWarps;  // the raw partial tile's copies
  uint32_t pph = 0;                        // its phase
  if (threadIdx.x == 0) {
    mbar_init(pbar, 1);
    fence_mbar_init();
  }

  int split = blockIdx.x;
  int b = blockIdx.z;  // the row (b, h) changes per segment in the persistent mode
  int h = blockIdx.y / p.vgroups;
  const int vg = blockIdx.y - h * p.vgroups;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // head slot hl of this CTA is query vector vh = vg * NH + hl of kv head h: chunk token
  // vh / group, query head h * group + vh % group (decode: chunk 1, vh = group member)
  const int n_vh = p.chunk * p.group;
  auto valid = [&](int hl) { return vg * NH + hl < n_vh; };
  auto vrow = [&](int hl) -> int64_t {
    const int vh = vg * NH + hl;
    return ((int64_t)b * p.chunk + vh / p.group) * p.num_q_heads + h * p.group + vh % p.group;
  };
  grid_dependency_wait();  // lengths, partial tiles and pages come from the previous kernel
  const int cap = p.max_pages * kTile + (kTile - 1);  // sealed pages must fit the block table
  auto part_row = [&](int hl, int slot) { return p.part + (vrow(hl) * p.max_splits + slot) * (D + 4); };
  // This warp's fp16 query values of row (bb, hh) for the staging of the rotated queries: head
  // slot warp + i * kDecWarps, channels lane * D / 32 .., zero outside the group and past d0.
  // Loaded ahead of the run that stages them (the persistent walk fetches the next segment's).
  constexpr int kQPer = (NH + kDecWarps - 1) / kDecWarps;
  __half2 qv[kQPer][D / 64];
  auto q_load = [&](int bb, int hh) {
#pragma unroll
    for (int i = 0; i < kQPer; ++i) {
      const int hl = warp + i * kDecWarps;
      const int vh = vg * NH + hl;
      const bool ok = hl < NH && vh < n_vh;
      const int64_t row = ((int64_t)bb * p.chunk + vh / p.group) * p.num_q_heads + hh * p.group + vh % p.group;
      const __half* src = p.q + (ok ? row : 0) * p.d0;
#pragma unroll
      for (int e2 = 0; e2 < D / 64; ++e2) {
        const int j = lane * (D / 32) + 2 * e2;
        const __half lo = (ok && j < p.d0) ? src[j] : __float2half(0.0f);
        const __half hi = (ok && j + 1 < p.d0) ? src[j + 1] : __float2half(0.0f);
        qv[i][e2] = __halves2half2(lo, hi);
      }
    }
  };
  // Sealed pages first..first+n-1 of row (b, h) -> partial row `slot`.  pc counts the pages this
  // warp has taken in earlier calls (the phases of its two barriers); `init` sets them up.  The
  // row's queries are in qv; after they are staged, ahead() runs (it may load the next run's).
  auto sealed_run = [&](int first, int n, int slot, int& pc, bool init, auto&& ahead) {
    const int cnt = n > warp ? (n - warp + kDecWarps - 1) / kDecWarps : 0;  // pages of this warp
    uint8_t* kslot = recs + warp * REC;
    uint8_t* vslot = kslot + KH;
    uint64_t* kbar = bars + 2 * warp;
    uint64_t* vbar = kbar + 1;
    const int32_t* bt = p.block_table + (int64_t)b * p.max_pages;
    auto page_src = [&](int j) -> const uint8_t* {  // record of this warp's j-th page
      int64_t id = bt[first + warp + kDecWarps * j];
      if (id < 0 || id >= p.num_pool_pages) {
        flag_error(p.status, KVARN_DEV_BAD_PAGE_ID);
        id = 0;
      }
      return p.pool + (id * p.num_kv_heads + h) * REC;
    };
    // start this warp's page stream before anything else
    if (lane == 0) {
      if (init) {
        mbar_init(kbar, 1);
        mbar_init(vbar, 1);
        fence_mbar_init();
      }
      if (cnt > 0) {
        const uint8_t* src = page_src(0);
        fence_proxy_async_smem();  // the slots held the previous merge's scratch
        mbar_expect_tx(kbar, KH);
        bulk_copy_g2s(kslot, src, KH, kbar);
        mbar_expect_tx(vbar, VH);
        bulk_copy_g2s(vslot, src + KH, VH, vbar);
      }
    }
    // rotated queries of this kv head's group, scaled by tau log2(e) / sqrt(d): fp32 for q~.z'
    // (channels 16k + {2t, 2t+1, 2t+8, 2t+9} adjacent), fp16 hi + lo for the B operand
    // (times the QkScale factors of the code width; one {hi pair, lo pair} entry per channel
    // pair)
#pragma unroll
    for (int i = 0; i < kQPer; ++i) {
      const int hl = warp + i * kDecWarps;
      if (hl >= NH) break;
      float v[D / 32];
#pragma unroll
      for (int e2 = 0; e2 < D / 64; ++e2) {
        const float2 f = __half22float2(qv[i][e2]);
        v[2 * e2] = f.x;
        v[2 * e2 + 1] = f.y;
      }
      warp_fwht<D>(v, lane);
      const float sc = p.qscale * inv_sqrt_d<D>();
      __half* qe = reinterpret_cast<__half*>(qhl + hl * QH);
#pragma unroll
      for (int e = 0; e < D / 32; ++e) {
        const int j = lane * (D / 32) + e;
        const float x = v[e] * sc;
        if constexpr (S::kQBytes > 0) qsm[hl * QLD + (j & ~15) + 4 * ((j & 7) >> 1) + 2 * ((j >> 3) & 1) + (j & 1)] = x;
        const float xb = x * ((j & 15) >= 8 ? QkScale<KB>::kH1 : QkScale<KB>::kH0);
        const __half hi = __float2half_rn(xb);
        qe[4 * (j >> 1) + (j & 1)] = hi;
        qe[4 * (j >> 1) + 2 + (j & 1)] = __float2half_rn(xb - __half2float(hi));
      }
    }
    __syncthreads();  // q in shared memory for every warp
    ahead();

    using Path = PagePath<D, NT, KB, VB>;
    typename Path::State st;
    Path::init(st);
    // record of the warp's next page, looked up one page ahead so that issuing its copies
    // never waits on the block-table load
    const uint8_t* nxt = cnt > 1 ? page_src(1) : nullptr;
    for (int j = 0; j < cnt; ++j) {
      const uint32_t par = (uint32_t)((pc + j) & 1);
      if (!__all_sync(0xffffffffu, mbar_wait(kbar, par))) {
        // a copy never arrived: report, drain this warp's copies still in flight, stop
        if (lane == 0) {
          flag_error(p.status, KVARN_DEV_WAIT_TIMEOUT);
          mbar_wait(kbar, par);
          mbar_wait(vbar, par);
        }
        break;
      }
      float lg[Path::kLgBlocks][Path::kLgNt][2], alpha[Path::kLgNt];
      Path::qk(kslot, qsm, qhl, lane, st, lg, alpha);
      __syncwarp();
      const bool more = j + 1 < cnt;
      if (lane == 0 && more) {  // the K slot is free: fetch the next page's K half
        fence_proxy_async_smem();
        mbar_expect_tx(kbar, KH);
        bulk_copy_g2s(kslot, nxt, KH, kbar);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(vbar, par))) {
        if (lane == 0) {
          flag_error(p.status, KVARN_DEV_WAIT_TIMEOUT);
          mbar_wait(vbar, par);
          if (more) mbar_wait(kbar, par ^ 1u);
        }
        break;
      }
      Path::pv(vslot, lg, alpha, lane, st);
      __syncwarp();
      if (lane == 0 && more) {  // the V slot is free: fetch the next page's V half
        fence_proxy_async_smem();
        mbar_expect_tx(vbar, VH);
        bulk_copy_g2s(vslot, nxt + KH, VH, vbar);
      }
      nxt = j + 2 < cnt ? page_src(j + 2) : nullptr;
    }
    // ---- merge the warps of this CTA ----
    __syncthreads();  // every warp is done with its slots
    if (p.part_mode != 1) grid_launch_dependents();  // (the persistent walk signals once, up front)
    float* mS = reinterpret_cast<float*>(recs);
    float* lS = mS + kDecWarps * NH;
    float* oS = lS + kDecWarps * NH;
    float* scS = oS + kDecWarps * NH * D;  // per (warp, head slot): exp2(m_w - M)
    float* MS = scS + kDecWarps * NH;       // per head slot: max over the warps, merged l
    float* LS = MS + NH;
    Path::store(st, warp, lane, mS, lS, oS);
    __syncthreads();
    // the warps' rescale factors of each head slot, once
    if (threadIdx.x < NH) {
      const int hl = threadIdx.x;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, mS[w * NH + hl]);
      float l = 0.0f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float sc = exp2f(mS[w * NH + hl] - M);
        scS[w * NH + hl] = sc;
        l = fmaf(sc, lS[w * NH + hl], l);
      }
      MS[hl] = M;
      LS[hl] = l;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < NH * D; idx += blockDim.x) {
      const int hl = idx / D, j = idx - hl * D;
      if (!valid(hl)) continue;
      float o = 0.0f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) o = fmaf(scS[w * NH + hl], oS[(w * NH + hl) * D + j], o);
      float* dst = part_row(hl, slot);
      dst[4 + j] = o;
      if (j == 0) {
        dst[0] = MS[hl];
        dst[1] = LS[hl];
      }
    }
    pc += cnt;
    __syncthreads();  // the merge scratch overlays the page slots the next run fills
  };

  // ---- partial tile: raw fp16 tokens in the original basis ---------------------------------
  // Row (b, h)'s n_part raw tokens -> partial row `split`; false if its copies never arrived.
  auto partial_run = [&](int n_part, int split) -> bool {
    // The n_part rows of K and of V are contiguous for one (sequence, kv head): two bulk copies
    // bring them into the page-slot area, then logits, softmax and PV run from shared memory.
    // Layout there: K rows [0, 256 D), V rows [256 D, 512 D) (row stride d0), probabilities
    // [t][NH] after them, then the head maxima and sums; the PV warp sums later overlay K.
    constexpr int E = D / 32;   // channels per lane, lane-contiguous
    constexpr int R = 32 / NH;  // tokens per logit round: 32 (token, head slot) pairs
    static_assert(S::kRecBytes >= 512 * D + 4 * NH * (kTile + 2), "partial tile fits the page slots");
    static_assert(kDecWarps * NH * D * 4 <= 256 * D, "PV warp sums fit over the K rows");
    const __half* Ks = reinterpret_cast<const __half*>(recs);
    const __half* Vs = reinterpret_cast<const __half*>(recs + 256 * D);
    float* pS = reinterpret_cast<float*>(recs + 512 * D);
    float* mS = pS + kTile * NH;
    float* lS = mS + NH;
    // q in the original basis: the fp32 q~ area, or after the softmax scratch where there is none
    constexpr int kPartQ = (512 * D + 4 * NH * (kTile + 2) + 15) & ~15;
    static_assert(S::kQBytes > 0 || S::kRecBytes >= kPartQ + NH * QLD * 4, "partial q fits");
    float* qp = S::kQBytes > 0 ? qsm : reinterpret_cast<float*>(recs + kPartQ);
    const int c0 = lane * E;
    const bool in = c0 < p.d0;  // d0 % 8 == 0: a lane's channels are all inside or all outside
    if (threadIdx.x == 0) {
      const int64_t base = ((int64_t)b * p.num_kv_heads + h) * kTile * p.d0;
      const uint32_t bytes = (uint32_t)(n_part * p.d0 * 2);  // a multiple of 16
      mbar_expect_tx(pbar, 2 * bytes);
      bulk_copy_g2s(recs, p.partial_k + base, bytes, pbar);
      bulk_copy_g2s(recs + 256 * D, p.partial_v + base, bytes, pbar);
    }
    for (int hl = warp; hl < NH; hl += kDecWarps) {
  #pragma unroll
      for (int e = 0; e < E; ++e) {
        const int j = c0 + e;
        qp[hl * QLD + j] =
            (valid(hl) && j < p.d0) ? __half2float(p.q[vrow(hl) * p.d0 + j]) * p.qscale : 0.0f;
      }
    }
    __syncthreads();  // q staged
    if (!__syncthreads_and(mbar_wait(pbar, pph) ? 1 : 0)) {
      if (threadIdx.x == 0) {
        flag_error(p.status, KVARN_DEV_WAIT_TIMEOUT);
        mbar_wait(pbar, pph);  // the copies may still land: wait (bounded) before leaving
      }
      return false;
    }
    // logits: each lane sums its E channels for the 32 pairs of a round, then a halving
    // butterfly leaves pair i = r * NH + hl complete in lane i
    for (int tb = warp; tb * R < n_part; tb += kDecWarps) {
      float v[32];
      float qv[NH][E];
  #pragma unroll
      for (int hl = 0; hl < NH; ++hl) load_f32<E>(qp + hl * QLD + c0, qv[hl]);
  #pragma unroll
      for (int r = 0; r < R; ++r) {
        const int t = tb * R + r;
        float kf[E];
        if (t < n_part && in) {
          load_f16<E>(Ks + t * p.d0 + c0, kf);
        } else {
  #pragma unroll
          for (int e = 0; e < E; ++e) kf[e] = 0.0f;
        }
  #pragma unroll
        for (int hl = 0; hl < NH; ++hl) {
          float acc = 0.0f;
  #pragma unroll
          for (int e = 0; e < E; ++e) acc = fmaf(qv[hl][e], kf[e], acc);
          v[r * NH + hl] = acc;
        }
      }
  #pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
  #pragma unroll
        for (int i = 0; i < o; ++i) {
          const float send = up ? v[i] : v[i + o];
          const float keep = up ? v[i + o] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      const int t = tb * R + lane / NH;
      if (t < n_part) pS[t * NH + lane % NH] = v[0];
    }
    __syncthreads();
    // softmax over the partial tokens, one warp per head slot
    for (int hl = warp; hl < NH; hl += kDecWarps) {
      if (!valid(hl)) break;
      float mx = -INFINITY;
      for (int t = lane; t < n_part; t += 32) mx = fmaxf(mx, pS[t * NH + hl]);
  #pragma unroll
      for (int msk = 16; msk > 0; msk >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
      float sum = 0.0f;
      for (int t = lane; t < n_part; t += 32) {
        const float pv = exp2f(pS[t * NH + hl] - mx);
        pS[t * NH + hl] = pv;
        sum += pv;
      }
  #pragma unroll
      for (int msk = 16; msk > 0; msk >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, msk);
      if (lane == 0) {
        mS[hl] = mx;
        lS[hl] = sum;
      }
    }
    __syncthreads();
    // PV: warp w takes tokens w, w + kDecWarps, ...; the warp sums meet in shared memory
    {
      float acc[NH][E];
  #pragma unroll
      for (int hl = 0; hl < NH; ++hl)
  #pragma unroll
        for (int e = 0; e < E; ++e) acc[hl][e] = 0.0f;
      if (in) {
        for (int t = warp; t < n_part; t += kDecWarps) {
          float vf[E];
          load_f16<E>(Vs + t * p.d0 + c0, vf);
  #pragma unroll
          for (int hl = 0; hl < NH; ++hl) {
            const float pw = pS[t * NH + hl];
  #pragma unroll
            for (int e = 0; e < E; ++e) acc[hl][e] = fmaf(pw, vf[e], acc[hl][e]);
          }
        }
      }
      float* oS = reinterpret_cast<float*>(recs);  // K rows are no longer read
  #pragma unroll
      for (int hl = 0; hl < NH; ++hl)
  #pragma unroll
        for (int e = 0; e < E; ++e) oS[(warp * NH + hl) * D + c0 + e] = acc[hl][e];
    }
    __syncthreads();
    // sum the warps, rotate o into the basis of the sealed splits, store
    for (int hl = warp; hl < NH; hl += kDecWarps) {
      if (!valid(hl)) break;
      const float* oS = reinterpret_cast<const float*>(recs);
      float v[E];
  #pragma unroll
      for (int e = 0; e < E; ++e) v[e] = 0.0f;
  #pragma unroll
      for (int w = 0; w < kDecWarps; ++w)
  #pragma unroll
        for (int e = 0; e < E; ++e) v[e] += oS[(w * NH + hl) * D + c0 + e];
      warp_fwht<D>(v, lane);
      float* dst = part_row(hl, split);
  #pragma unroll
      for (int e = 0; e < E; ++e) dst[4 + c0 + e] = v[e] * inv_sqrt_d<D>();
      if (lane == 0) {
        dst[0] = mS[hl];
        dst[1] = lS[hl];
      }
    }
    pph ^= 1u;
    __syncthreads();  // the page slots are reused next
    return true;
  };
  if (p.part_mode == 1) {
    // persistent: this CTA's range of the balanced partition, segment by segment
    __shared__ Walk walk0;
    if (warp == 0) {
      const Walk w = range_walk(p, blockIdx.x, lane);
      if (lane == 0) walk0 = w;
    }
    if (blockIdx.x == 0) {  // the length checks of the one-CTA-per-split form, once
      for (int bb = threadIdx.x; bb < p.batch; bb += blockDim.x) {
        const int lb = p.seq_lens[bb];
        if (lb < 0 || lb > cap) flag_error(p.status, KVARN_DEV_SEQ_TOO_LONG);
        else if (lb % kTile != 0 && p.partial_k == nullptr && p.partial_in_merge == 0)
          flag_error(p.status, KVARN_DEV_NO_PARTIAL);
      }
    }
    __syncthreads();
    // the dependent merge kernel may be scheduled now: its CTAs take an SM's resources only as
    // this grid's CTAs leave, and it waits for this grid's completion before reading the splits
    grid_launch_dependents();
    int pc = 0;
    bool init = true;
    Walk w = walk0;
    q_load(w.b, w.h);
    while (w.left > 0) {
      b = w.b;
      h = w.h;
      Walk wn = w;  // the next segment, and its queries while this one runs
      sealed_run(w.j, w.count(), w.slot, pc, init, [&]() {
        wn.next(p);
        if (wn.left > 0) q_load(wn.b, wn.h);
      });
      init = false;
      w = wn;
    }
    // raw partial tiles (unless the merge takes them): row k = b * Hkv + h goes to CTA k mod
    // gridDim.x, its split after the row's sealed segments
    for (int k = blockIdx.x; p.partial_in_merge == 0 && k < p.batch * p.num_kv_heads; k += gridDim.x) {
      b = k / p.num_kv_heads;
      h = k - b * p.num_kv_heads;
      int lb = p.seq_lens[b];
      lb = lb < 0 ? 0 : (lb > cap ? cap : lb);
      const int np = lb % kTile;
      if (np == 0 || p.partial_k == nullptr || p.partial_v == nullptr) continue;
      if (!partial_run(np, tc_row_segments(p, b, h, lane))) break;
    }
    grid_launch_dependents();
    return;
  }
  int len = p.seq_lens[b];
  if (len < 0 || len > cap) {
    if (threadIdx.x == 0 && split == 0 && h == 0) flag_error(p.status, KVARN_DEV_SEQ_TOO_LONG);
    len = len < 0 ? 0 : cap;
  }
  const int n_sealed = len / kTile, n_part = len % kTile;
  int n_ss = (n_sealed + p.pages_per_split - 1) / p.pages_per_split;
  if (p.part_mode == 2) {  // the persistent kernel took the sealed pages: the partial tile's split
    n_ss = tc_row_segments(p, b, h, lane);
    split = n_ss;
  }
  const bool partial_split = (split == n_ss) && n_part > 0 && p.partial_in_merge == 0;
  if (split >= n_ss && !partial_split) return;
  if (partial_split && (p.partial_k == nullptr || p.partial_v == nullptr)) {
    if (threadIdx.x == 0) flag_error(p.status, KVARN_DEV_NO_PARTIAL);
    return;
  }
  if (!partial_split) {
    int pc = 0;
    const int first = split * p.pages_per_split;
    q_load(b, h);
    sealed_run(first, min(n_sealed, first + p.pages_per_split) - first, split, pc, true, []() {});
    return;
  }
  partial_run(n_part, split);
}


// Attention of one query (E = D/32 channels per lane, original basis, times tau log2(e)) to
// n_tok raw fp16 tokens whose rows start at k_row / v_row (this lane's channels; row stride
// rstride): online softmax in the log2 domain, unnormalised output o in the original basis.
// 32 tokens at a time: each lane sums its channels for 32 tokens, a halving shuffle butterfly
// leaves token t0 + i's logit complete in lane i.
template <int D>
__device__ __forceinline__ void raw_attend(const float (&q)[D / 32], const __half* k_row, const __half* v_row,
                                           int64_t rstride, int n_tok, bool in, int lane, float& m, float& l,
                                           float (&o)[D / 32]) {
  constexpr int E = D / 32;
  for (int t0 = 0; t0 < n_tok; t0 += 32) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float kf[E];
      if (t0 + i < n_tok && in) {
        load_f16<E>(k_row + (t0 + i) * rstride, kf);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) kf[e] = 0.0f;
      }
      float acc = 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc = fmaf(q[e], kf[e], acc);
      v[i] = acc;
    }
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
      const bool up = (lane & w) != 0;
#pragma unroll
      for (int i = 0; i < w; ++i) {
        const float send = up ? v[i] : v[i + w];
        const float keep = up ? v[i + w] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
      }
    }
    const bool live = t0 + lane < n_tok;
    float mx = live ? v[0] : -INFINITY;
#pragma unroll
    for (int msk = 16; msk > 0; msk >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
    const float mnew = fmaxf(m, mx);
    const float a = exp2f(m - mnew);
    const float pv = live ? exp2f(v[0] - mnew) : 0.0f;
    float ps = pv;
#pragma unroll
    for (int msk = 16; msk > 0; msk >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, msk);
    m = mnew;
    l = fmaf(l, a, ps);
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] *= a;
    // PV eight tokens at a time, their eight row loads issued before the first use
    const int cnt = min(32, n_tok - t0);
    for (int i0 = 0; i0 < cnt; i0 += 8) {
      float vf[8][E];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (in && i0 + i < cnt) {
          load_f16<E>(v_row + (t0 + i0 + i) * rstride, vf[i]);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) vf[i][e] = 0.0f;
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float pw = __shfl_sync(0xffffffffu, pv, (i0 + i) & 31);  // 0 past the last token
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = fmaf(pw, vf[i][e], o[e]);
      }
    }
  }
}

// One warp per (sequence, chunk token, query head): merge the splits, normalise, undo the
// rotation.  When p.partial_in_merge is set (decode), the warp also attends to the sequence's raw
// partial tile itself, before waiting for the splits (the tile does not depend on them): its
// output is in the original basis and joins after the inverse rotation [vatt §四個步驟: R is
// orthonormal and symmetric, so R (sum_s w_s o~_s) + w_p o_p is the merged output].
// RAW (decode with p.partial_in_merge): one CTA of 8 warps per (sequence, kv head); the row's raw
// partial tile is staged in shared memory as fp16 rows (16-byte chunks XOR-swizzled by row, rows
// past the tile zero-filled): K tokens 0..127 in rows 0..127 and V tokens 0..63 in rows 128..191,
// then, once every warp's QK has read them, V tokens 64..127 over rows 0..63 (48 KB, so that four
// CTAs share an SM and a batch of 64 x 8 rows is one wave).  It is attended on the tensor cores:
// warp w takes tokens 16w..16w+15, QK as mma.sync m16n8k16 with A = K rows by ldmatrix and B = the
// fp16 queries (heads 4nt + j in column pairs (j, 0)), PV with A = V^T by ldmatrix.trans and B =
// the probabilities in fp16 hi + lo; the warps meet in shared memory, and warp w < G then merges
// query head w's splits.  Otherwise four warps per CTA over (sequence, chunk token, query head),
// and any partial tile is a split of its own.
template <int D, bool RAW, int NT = 1>
__global__ void __launch_bounds__(RAW ? 256 : 128) combine_kernel(DecodeParams p) {
  constexpr int E = D / 32;
  constexpr int NH = 4 * NT;  // RAW: head slots (the group padded to 4 or 8)
  const int lane = threadIdx.x & 31;
  const int wi = threadIdx.x >> 5;
  const int gw = RAW ? (blockIdx.x / p.num_kv_heads) * p.num_q_heads + (blockIdx.x % p.num_kv_heads) * p.group + wi
                     : blockIdx.x * (blockDim.x / 32) + wi;
  const bool live = RAW ? wi < p.group : gw < p.batch * p.chunk * p.num_q_heads;
  const int b = RAW ? blockIdx.x / p.num_kv_heads : gw / (p.chunk * p.num_q_heads);
  const int h = RAW ? blockIdx.x % p.num_kv_heads : (gw % p.num_q_heads) / p.group;
  const int cap = p.max_pages * kTile + (kTile - 1);
  // The lengths and the raw partial tiles come from before decode_kernel, which waited for their
  // writer before it let this kernel start: they can be read ahead of the wait for the splits.
  int len = (RAW || live) ? p.seq_lens[b] : 0;
  len = len < 0 ? 0 : (len > cap ? cap : len);
  const int n_part = len % kTile;
  // the splits of the row's sealed pages (a warp-collective; lengths and block tables are inputs)
  auto cache_splits = [&]() -> int {
    return p.part_ctas > 0 ? tc_row_segments(p, b, h, lane)
                           : (len / kTile + p.pages_per_split - 1) / p.pages_per_split;
  };
  int n_cache = -1;
  float mp = -INFINITY, lp = 0.0f, op[E];
#pragma unroll
  for (int e = 0; e < E; ++e) op[e] = 0.0f;
  bool has_part = false;
  if constexpr (RAW) {
    extern __shared__ __align__(128) uint8_t raw_s[];  // rows [192][2 D], then q [NH][D]
    constexpr int kRows = kTile + kTile / 2;
    has_part = n_part > 0 && p.partial_k != nullptr && p.partial_v != nullptr;
    if (n_part > 0 && !has_part && threadIdx.x == 0) flag_error(p.status, KVARN_DEV_NO_PARTIAL);
    if (has_part) {
      const int g = lane >> 2, tq = lane & 3;
      const uint32_t sbase = smem_u32(raw_s);
      __half* qs = reinterpret_cast<__half*>(raw_s + kRows * 2 * D);
      const int64_t base = ((int64_t)b * p.num_kv_heads + h) * kTile * p.d0;
      const int dch = p.d0 / 8;  // 16-byte chunks of a raw row (d0 % 8 == 0)
      // row r of the staging area <- token t of K or V (zero past the tile)
      auto stage = [&](int r, int c, const __half* src_base, int t) {
        const bool in = t < n_part && c < dch;
        cp_async_16(sbase + swz_row<D>(r, c), in ? src_base + base + (int64_t)t * p.d0 + 8 * c : p.partial_k,
                    in ? 16u : 0u);
      };
      for (int qi = threadIdx.x; qi < kRows * (D / 8); qi += blockDim.x) {
        const int r = qi / (D / 8), c = qi - r * (D / 8);
        if (r < kTile) stage(r, c, p.partial_k, r);
        else stage(r, c, p.partial_v, r - kTile);
      }
      cp_async_commit_all();
      for (int i = threadIdx.x; i < NH * D; i += blockDim.x) {
        const int hl = i / D, c = i - hl * D;
        qs[i] = (hl < p.group && c < p.d0) ? p.q[((int64_t)b * p.num_q_heads + h * p.group + hl) * p.d0 + c]
                                           : __float2half(0.0f);
      }
      if (live) n_cache = cache_splits();  // while the tile is in flight
      cp_async_wait_all();
      __syncthreads();
      const int t0 = 16 * wi;  // this warp's tokens
      float m[NT], l[NT], o[D / 16][NT][2];
      uint32_t bw[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        m[nt] = -INFINITY;
        l[nt] = 0.0f;
        bw[nt][0] = bw[nt][1] = 0u;
#pragma unroll
        for (int mc = 0; mc < D / 16; ++mc) o[mc][nt][0] = o[mc][nt][1] = 0.0f;
      }
      if (t0 < n_part) {
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
        {
          const int row = t0 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[4];
            ldsm_x4(sbase + swz_row<D>(row, 2 * kk + (lane >> 4)), a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              // B: column 2j = head 4nt + j, column 2j + 1 = 0
              const __half* qr = qs + (4 * nt + (g >> 1)) * D + 16 * kk + 2 * tq;
              const bool zero = (g & 1) != 0;
              const uint32_t b0 = zero ? 0u : *reinterpret_cast<const uint32_t*>(qr);
              const uint32_t b1 = zero ? 0u : *reinterpret_cast<const uint32_t*>(qr + 8);
              mma16816(acc[nt], a, b0, b1);
            }
          }
        }
        const bool v0 = t0 + g < n_part, v1 = t0 + g + 8 < n_part;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float s0 = v0 ? (acc[nt][0] + acc[nt][1]) * p.qscale : -INFINITY;
          const float s1 = v1 ? (acc[nt][2] + acc[nt][3]) * p.qscale : -INFINITY;
          float mx = fmaxf(s0, s1);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          m[nt] = mx;  // finite: token t0 (g = 0) is in the tile
          const float p0 = exp2f(s0 - mx), p1 = exp2f(s1 - mx);
          l[nt] = p0 + p1;
          const __half2 hi = __floats2half2_rn(p0, p1);
          const float2 hf = __half22float2(hi);
          const __half2 lo = __floats2half2_rn(p0 - hf.x, p1 - hf.y);
          bw[nt][0] = movmatrix_trans(h2u(__lows2half2(hi, lo)));   // (hi, lo) of token row g
          bw[nt][1] = movmatrix_trans(h2u(__highs2half2(hi, lo)));  // (hi, lo) of token row g + 8
        }
      }
      // every warp's QK is done: V tokens 64..127 replace K tokens 0..63
      __syncthreads();
      const bool second = n_part > kTile / 2;  // the same for the whole CTA
      if (second) {
        for (int qi = threadIdx.x; qi < (kTile / 2) * (D / 8); qi += blockDim.x) {
          const int r = qi / (D / 8), c = qi - r * (D / 8);
          stage(r, c, p.partial_v, r + kTile / 2);
        }
        cp_async_commit_all();
      }
      auto pv = [&](int vrow) {  // V rows of this warp's tokens start at vrow
        const int row = vrow + (lane & 7) + 8 * (lane >> 4);
#pragma unroll
        for (int mc = 0; mc < D / 16; ++mc) {
          uint32_t a[4];
          ldsm_x4_trans(sbase + swz_row<D>(row, 2 * mc + ((lane >> 3) & 1)), a);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float pacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            mma16816(pacc, a, bw[nt][0], bw[nt][1]);
            o[mc][nt][0] = pacc[0] + pacc[1];
            o[mc][nt][1] = pacc[2] + pacc[3];
          }
        }
      };
      if (t0 < kTile / 2 && t0 < n_part) pv(kTile + t0);
      if (second) cp_async_wait_all();
      __syncthreads();
      if (t0 >= kTile / 2 && t0 < n_part) pv(t0 - kTile / 2);
      // the warps meet: (m, l, o) per (warp, head slot) over the staging rows
      __syncthreads();
      float* mS = reinterpret_cast<float*>(raw_s);
      float* lS = mS + 8 * NH;
      float* oS = lS + 8 * NH;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float lt = l[nt];
        lt += __shfl_xor_sync(0xffffffffu, lt, 4);
        lt += __shfl_xor_sync(0xffffffffu, lt, 8);
        lt += __shfl_xor_sync(0xffffffffu, lt, 16);
        const int hl = 4 * nt + tq;
        if (g == 0) {
          mS[wi * NH + hl] = m[nt];
          lS[wi * NH + hl] = lt;
        }
#pragma unroll
        for (int mc = 0; mc < D / 16; ++mc) {
          oS[(wi * NH + hl) * D + 16 * mc + g] = o[mc][nt][0];
          oS[(wi * NH + hl) * D + 16 * mc + g + 8] = o[mc][nt][1];
        }
      }
      __syncthreads();
      if (live) {  // warp wi merges head slot wi's eight parts; its lanes hold channels lane*E..
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 8; ++w) M = fmaxf(M, mS[w * NH + wi]);
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const float mw = mS[w * NH + wi];
          const float sc = mw == -INFINITY ? 0.0f : exp2f(mw - M);  // warps that saw no token
          lp = fmaf(sc, lS[w * NH + wi], lp);
#pragma unroll
          for (int e = 0; e < E; ++e) op[e] = fmaf(sc, oS[(w * NH + wi) * D + lane * E + e], op[e]);
        }
        mp = M;
      }
    }
  }
  if (live && n_cache < 0) n_cache = cache_splits();
  grid_dependency_wait();  // the split partials of decode_kernel (and of the chunk kernel)
  grid_launch_dependents();  // the next kernel (say, the next step's append) may start arriving
  if (!live) return;
  const int n_splits = n_cache + (n_part > 0 && p.partial_in_merge == 0 ? 1 : 0) + (p.chunk_k != nullptr ? 1 : 0);
  const float* base = p.part + (int64_t)gw * p.max_splits * (D + 4);
  float v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = 0.0f;
  float M = mp, lsum = 0.0f;  // over the splits and the raw tile
  if (n_splits > 0 && n_splits <= 4) {
    // up to four splits (the common case): every load issued before the first use
    float2 ml[4];
    float o[4][E];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      if (s < n_splits) {
        ml[s] = *reinterpret_cast<const float2*>(base + s * (D + 4));
        load_f32<E>(base + s * (D + 4) + 4 + lane * E, o[s]);
      } else {
        ml[s] = make_float2(-INFINITY, 0.0f);
#pragma unroll
        for (int e = 0; e < E; ++e) o[s][e] = 0.0f;
      }
    }
    M = fmaxf(M, fmaxf(fmaxf(ml[0].x, ml[1].x), fmaxf(ml[2].x, ml[3].x)));
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const float w = s < n_splits ? exp2f(ml[s].x - M) : 0.0f;
      lsum = fmaf(w, ml[s].y, lsum);
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = fmaf(w, o[s][e], v[e]);
    }
  } else if (n_splits > 0 && n_splits <= 32) {
    // up to 32 splits: (m, l) one split per lane in one load, then the partial outputs eight
    // splits at a time with all eight loads issued before their use
    const bool mine = lane < n_splits;
    const float2 ml = mine ? *reinterpret_cast<const float2*>(base + lane * (D + 4)) : make_float2(-INFINITY, 0.0f);
    float Ms = ml.x;
#pragma unroll
    for (int msk = 16; msk > 0; msk >>= 1) Ms = fmaxf(Ms, __shfl_xor_sync(0xffffffffu, Ms, msk));
    M = fmaxf(M, Ms);
    const float w = mine ? exp2f(ml.x - M) : 0.0f;
    lsum = w * ml.y;
#pragma unroll
    for (int msk = 16; msk > 0; msk >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, msk);
    for (int s0 = 0; s0 < n_splits; s0 += 8) {
      float o[8][E];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (s0 + j < n_splits) {
          load_f32<E>(base + (s0 + j) * (D + 4) + 4 + lane * E, o[j]);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) o[j][e] = 0.0f;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, (s0 + j) & 31);  // 0 past the last split
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = fmaf(wj, o[j][e], v[e]);
      }
    }
  } else if (n_splits > 0) {
    // split statistics, one split per lane, 32 per pass
    for (int s0 = 0; s0 < n_splits; s0 += 32) {
      const int s = s0 + lane;
      float m = s < n_splits ? base[s * (D + 4)] : -INFINITY;
#pragma unroll
      for (int msk = 16; msk > 0; msk >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, msk));
      M = fmaxf(M, m);
    }
    for (int s0 = 0; s0 < n_splits; s0 += 32) {
      const int s = s0 + lane;
      const float w = s < n_splits ? exp2f(base[s * (D + 4)] - M) : 0.0f;
      float lw = s < n_splits ? w * base[s * (D + 4) + 1] : 0.0f;
#pragma unroll
      for (int msk = 16; msk > 0; msk >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, msk);
      lsum += lw;
      const int cnt = min(32, n_splits - s0);
#pragma unroll 4
      for (int i = 0; i < cnt; ++i) {
        const float wi = __shfl_sync(0xffffffffu, w, i);
        const float* src = base + (s0 + i) * (D + 4) + 4 + lane * E;
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 o = *reinterpret_cast<const float2*>(src + e);
          v[e] = fmaf(wi, o.x, v[e]);
          v[e + 1] = fmaf(wi, o.y, v[e + 1]);
        }
      }
    }
  }
  // the raw tile joins after the inverse rotation of the splits' sum
  const float wp = has_part ? exp2f(mp - M) : 0.0f;
  lsum = fmaf(wp, lp, lsum);
  if (n_splits > 0) warp_fwht<D>(v, lane);
  const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = fmaf(v[e], inv_sqrt_d<D>(), wp * op[e]) * inv;
  __half* dst = p.out + (int64_t)gw * p.d0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane * E + e;
    if (j < p.d0) dst[j] = __float2half_rn(v[e]);
  }
}

template <int D, int NT, int KB, int VB>
static int launch_decode_t(const DecodeParams& p, int phases, cudaStream_t stream) {
  using S = DecodeShape<D, NT, KB, VB>;
  static PerDeviceOnce smem_once;  // the attribute is set once per device
  const void* fn = reinterpret_cast<const void*>(decode_kernel<D, NT, KB, VB>);
  if (const int st = set_smem_limit(smem_once, fn, S::kSmemBytes); st != KVARN_OK) return st;
  // both kernels may start while their predecessor in the stream drains; each waits for it
  // (griddepcontrol.wait) before touching its results
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(S::kWarps * 32);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((phases & kDecodeSplits) != 0) {
    if (p.part_mode == 1) {
      // persistent CTAs over the sealed pages and the raw partial tiles
      cfg.gridDim = dim3(p.part_ctas);
      if (cudaLaunchKernelEx(&cfg, decode_kernel<D, NT, KB, VB>, p) != cudaSuccess) return KVARN_ERR_CUDA;
    } else {
      // the sealed splits at this split size plus the partial tile's (the workspace stride
      // max_splits is laid out for the smallest size and may be larger)
      const int splits = min(p.max_splits, (p.max_pages + p.pages_per_split - 1) / p.pages_per_split +
                                               (p.partial_in_merge != 0 ? 0 : 1));
      cfg.gridDim = dim3(splits, p.num_kv_heads * p.vgroups, p.batch);
      if (cudaLaunchKernelEx(&cfg, decode_kernel<D, NT, KB, VB>, p) != cudaSuccess) return KVARN_ERR_CUDA;
    }
  }
  if ((phases & kDecodeMerge) == 0) return KVARN_OK;
  return launch_decode_combine(D, p, stream);
}

template <int D>
static int launch_combine_t(const DecodeParams& p, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.partial_in_merge != 0 && p.chunk == 1) {
    // one CTA of 8 warps per (sequence, kv head): 192 fp16 rows of the raw partial tile in shared
    // memory, then the fp16 queries of 4 or 8 head slots
    cfg.gridDim = dim3(p.batch * p.num_kv_heads);
    cfg.blockDim = dim3(256);
    if (p.group <= 4) {
      constexpr int kSmem = (kTile + kTile / 2) * 2 * D + 4 * D * 2;
      static PerDeviceOnce smem_once;
      const void* fn = reinterpret_cast<const void*>(combine_kernel<D, true, 1>);
      if (const int st = set_smem_limit(smem_once, fn, kSmem); st != KVARN_OK) return st;
      cfg.dynamicSmemBytes = kSmem;
      return cudaLaunchKernelEx(&cfg, combine_kernel<D, true, 1>, p) == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA;
    }
    if constexpr (D <= 128) {
      constexpr int kSmem = (kTile + kTile / 2) * 2 * D + 8 * D * 2;
      static PerDeviceOnce smem_once;
      const void* fn = reinterpret_cast<const void*>(combine_kernel<D, true, 2>);
      if (const int st = set_smem_limit(smem_once, fn, kSmem); st != KVARN_OK) return st;
      cfg.dynamicSmemBytes = kSmem;
      return cudaLaunchKernelEx(&cfg, combine_kernel<D, true, 2>, p) == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA;
    }
    return KVARN_ERR_UNSUPPORTED;
  }
  const int warps = p.batch * p.chunk * p.num_q_heads;
  cfg.gridDim = dim3((warps + 3) / 4);
  cfg.blockDim = dim3(128);
  return cudaLaunchKernelEx(&cfg, combine_kernel<D, false, 1>, p) == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA;
}

int launch_decode_combine(int d, const DecodeParams& p, cudaStream_t stream) {
  if (d == 64) return launch_combine_t<64>(p, stream);
  if (d == 128) return launch_combine_t<128>(p, stream);
  if (d == 256) return launch_combine_t<256>(p, stream);
  return KVARN_ERR_UNSUPPORTED;
}

int launch_decode_partial_tiles(const DecodeParams& p, cudaStream_t stream) {
  using S = DecodeShape<128, 2, 4, 2>;
  static PerDeviceOnce smem_once;
  const void* fn = reinterpret_cast<const void*>(decode_kernel<128, 2, 4, 2>);
  if (const int st = set_smem_limit(smem_once, fn, S::kSmemBytes); st != KVARN_OK) return st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, p.num_kv_heads * p.vgroups, p.batch);
  cfg.blockDim = dim3(S::kWarps * 32);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  DecodeParams pt = p;
  pt.part_mode = 2;
  return cudaLaunchKernelEx(&cfg, decode_kernel<128, 2, 4, 2>, pt) == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA;
}

template <int D, int NT, int KB, int VB>
static int persistent_ctas_t() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return 0;
  return sms * DecodeShape<D, NT, KB, VB>::kMinBlocks;
}

template <int KB, int VB>
static int persistent_ctas_bits(int d, int nt) {
  if (nt == 1) {
    if (d == 64) return persistent_ctas_t<64, 1, KB, VB>();
    if (d == 128) return persistent_ctas_t<128, 1, KB, VB>();
    if (d == 256) return persistent_ctas_t<256, 1, KB, VB>();
  } else if (nt == 2) {
    if (d == 64) return persistent_ctas_t<64, 2, KB, VB>();
    if (d == 128) return persistent_ctas_t<128, 2, KB, VB>();
  }
  return 0;
}

int decode_persistent_ctas(int d, int nt, int kb, int vb) {
  if (kb == 4 && vb == 2) return persistent_ctas_bits<4, 2>(d, nt);
  if (kb == 4 && vb == 4) return persistent_ctas_bits<4, 4>(d, nt);
  if (kb == 2 && vb == 2) return persistent_ctas_bits<2, 2>(d, nt);
  if (kb == 8 && vb == 4) return persistent_ctas_bits<8, 4>(d, nt);
  return 0;
}

// Causal attention of each chunk query to the chunk's own raw fp16 tokens (prefill): one
// warp per (sequence, chunk token c, query head), tokens 0..c, original basis, online
// softmax in the log2 domain; the unnormalised output is rotated and written as the split
// after the cache's splits [vatt §四個步驟: the rotation keeps q.k unchanged, so partials in
// the rotated basis merge with the cache's].
template <int D>
__global__ void __launch_bounds__(128) chunk_kernel(DecodeParams p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  grid_dependency_wait();
  if (gw >= p.batch * p.chunk * p.num_q_heads) return;
  const int hq = gw % p.num_q_heads, bc = gw / p.num_q_heads;
  const int b = bc / p.chunk, c = bc - b * p.chunk;
  const int h = hq / p.group;
  const int c0 = lane * E;
  const bool in = c0 < p.d0;  // d0 % 8 == 0: a lane's channels are all inside or all outside
  float q[E], o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    q[e] = in ? __half2float(p.q[(int64_t)gw * p.d0 + c0 + e]) * p.qscale : 0.0f;
    o[e] = 0.0f;
  }
  float m = -INFINITY, l = 0.0f;
  const int n_tok = c + 1;  // chunk tokens 0..c
  const int64_t rstride = (int64_t)p.num_kv_heads * p.d0;
  const __half* kbase = p.chunk_k + ((int64_t)b * p.chunk * p.num_kv_heads + h) * p.d0 + c0;
  const __half* vbase = p.chunk_v + ((int64_t)b * p.chunk * p.num_kv_heads + h) * p.d0 + c0;
  raw_attend<D>(q, kbase, vbase, rstride, n_tok, in, lane, m, l, o);
  warp_fwht<D>(o, lane);
  const int cap = p.max_pages * kTile + (kTile - 1);
  int len = p.seq_lens[b];
  len = len < 0 ? 0 : (len > cap ? cap : len);
  const int split = (len / kTile + p.pages_per_split - 1) / p.pages_per_split + (len % kTile > 0 ? 1 : 0);
  float* dst = p.part + ((int64_t)gw * p.max_splits + split) * (D + 4);
#pragma unroll
  for (int e = 0; e < E; ++e) dst[4 + lane * E + e] = o[e] * inv_sqrt_d<D>();
  if (lane == 0) {
    dst[0] = m;
    dst[1] = l;
  }
}

// The same causal attention on the tensor cores (head_dim 64 and 128): one CTA of 8 warps per
// (128 query rows, kv head, sequence), query row r = c * G + j for chunk token c and group head
// j, warp w taking rows 16w..16w+15.  The chunk's K and V rows stream through shared memory 64
// tokens at a time (cp.async into swizzled fp16 rows, two stages).  QK is mma.sync m16n8k16
// with A = the fp16 queries (exact products, the scale applied to the fp32 sums) and B = K rows
// by ldmatrix; the softmax is online in the log2 domain with the tokens past a row's own masked;
// PV takes A = the probabilities as fp16 hi + lo, read from the QK accumulators' layout, and B =
// V rows by ldmatrix.trans.  The unnormalised output is rotated in registers (its channels are
// 8n + 2tq + e for n-tile n, quad lane tq and pair element e: butterflies within the lane, across
// the quad and across n-tiles) and written as the split after the cache's [vatt §四個步驟].
template <int D>
__global__ void __launch_bounds__(256, 1) chunk_tc_kernel(DecodeParams p) {
  constexpr int NB = 64;      // tokens per stage
  constexpr int NN = D / 8;   // channel n-tiles
  constexpr int KK = D / 16;  // channel k-steps
  constexpr uint32_t kStage = 2 * NB * 2 * D;  // K rows then V rows, fp16
  extern __shared__ __align__(128) uint8_t cs[];
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const int b = blockIdx.z, h = blockIdx.y;
  const int G = p.group, C = p.chunk;
  const int rows = C * G;
  const int rbase = blockIdx.x * 128;
  const int r0 = rbase + 16 * wi;  // this warp's first query row
  const bool warp_live = r0 < rows;
  const int c_last_w = (min(r0 + 15, rows - 1)) / G;      // the warp's last chunk token
  const int c_last = (min(rbase + 127, rows - 1)) / G;    // the CTA's
  const int ra = r0 + g, rb = r0 + g + 8;                 // the lane's two rows
  const int ca = ra < rows ? ra / G : -1, cb = rb < rows ? rb / G : -1;  // -1: padding row
  grid_dependency_wait();
  const uint32_t sbase = smem_u32(cs);
  const int64_t rstride = (int64_t)p.num_kv_heads * p.d0;
  const __half* kg = p.chunk_k + ((int64_t)b * C * p.num_kv_heads + h) * p.d0;
  const __half* vg = p.chunk_v + ((int64_t)b * C * p.num_kv_heads + h) * p.d0;
  const int dch = p.d0 / 8;  // 16-byte chunks of a row (d0 % 8 == 0)
  const int nblk = c_last / NB + 1;
  auto stage = [&](int blk) {
    const uint32_t base = sbase + (uint32_t)(blk & 1) * kStage;
    for (int qi = threadIdx.x; qi < 2 * NB * (D / 8); qi += blockDim.x) {
      const int r = qi / (D / 8), c = qi - r * (D / 8);
      const int t = blk * NB + (r < NB ? r : r - NB);
      const bool in = t < C && c < dch;
      const __half* src = (r < NB ? kg : vg) + (int64_t)t * rstride + 8 * c;
      cp_async_16(base + swz_row<D>(r, c), in ? src : kg, in ? 16u : 0u);
    }
    cp_async_commit_all();
  };
  stage(0);
  // the warp's queries as A fragments: rows g (ra) and g + 8 (rb), channels 16kk + 2tq.. and +8
  uint32_t aq[KK][4];
  {
    auto qrow = [&](int r) {
      const int c = r / G, j = r - c * G;
      return p.q + (((int64_t)b * C + c) * p.num_q_heads + h * G + j) * p.d0;
    };
    const __half* qa = qrow(ca >= 0 ? ra : 0);
    const __half* qb = qrow(cb >= 0 ? rb : 0);
    // rows start at even element offsets (d0 is a multiple of 8), so with q 4-byte aligned a
    // channel pair is one 32-bit load
    const bool q4 = (reinterpret_cast<uintptr_t>(p.q) & 3u) == 0u;
    auto pair = [&](const __half* row, bool ok, int ch) -> uint32_t {
      if (!(ok && ch < p.d0)) return 0u;
      return q4 ? *reinterpret_cast<const uint32_t*>(row + ch) : h2u(__halves2half2(row[ch], row[ch + 1]));
    };
#pragma unroll
    for (int kk = 0; kk < KK; ++kk) {
      const int ch = 16 * kk + 2 * tq;
      aq[kk][0] = pair(qa, ca >= 0, ch);
      aq[kk][1] = pair(qb, cb >= 0, ch);
      aq[kk][2] = pair(qa, ca >= 0, ch + 8);
      aq[kk][3] = pair(qb, cb >= 0, ch + 8);
    }
  }
  float ma = -INFINITY, mb = -INFINITY, la = 0.0f, lb = 0.0f;  // l: this lane's share
  float o[NN][4];
#pragma unroll
  for (int n = 0; n < NN; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
  for (int blk = 0; blk < nblk; ++blk) {
    if (blk + 1 < nblk) {
      stage(blk + 1);  // its buffer was released by the barrier closing blk - 1
      cp_async_wait_prev();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
    const int t0 = blk * NB;
    if (warp_live && t0 <= c_last_w) {
      const uint32_t base = sbase + (uint32_t)(blk & 1) * kStage;
      float s[NB / 8][4];
#pragma unroll
      for (int nt = 0; nt < NB / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.0f;
#pragma unroll
      for (int kk = 0; kk < KK; ++kk) {
#pragma unroll
        for (int np = 0; np < NB / 16; ++np) {  // token n-tiles 2np, 2np + 1
          uint32_t bk[4];
          ldsm_x4(base + swz_row<D>(16 * np + (lane & 7) + 8 * (lane >> 4), 2 * kk + ((lane >> 3) & 1)), bk);
          mma16816(s[2 * np], aq[kk], bk[0], bk[1]);
          mma16816(s[2 * np + 1], aq[kk], bk[2], bk[3]);
        }
      }
      // logits of rows ra (s[.][0..1]) and rb (s[.][2..3]), tokens t0 + 8nt + 2tq + e
      float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < NB / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = t0 + 8 * nt + 2 * tq + e;
          s[nt][e] = t <= ca ? s[nt][e] * p.qscale : -INFINITY;
          s[nt][2 + e] = t <= cb ? s[nt][2 + e] * p.qscale : -INFINITY;
          mxa = fmaxf(mxa, s[nt][e]);
          mxb = fmaxf(mxb, s[nt][2 + e]);
        }
      }
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
      const float na = fmaxf(ma, mxa), nb = fmaxf(mb, mxb);
      // a row with no token yet keeps m = -inf, l = 0 and o = 0
      const float sa = na == -INFINITY ? 0.0f : na, sb = nb == -INFINITY ? 0.0f : nb;
      const float aa = ma == -INFINITY ? 0.0f : exp2f(ma - na);
      const float ab = mb == -INFINITY ? 0.0f : exp2f(mb - nb);
      ma = na;
      mb = nb;
      float pa = 0.0f, pb = 0.0f;
#pragma unroll
      for (int nt = 0; nt < NB / 8; ++nt) {
        s[nt][0] = exp2f(s[nt][0] - sa);
        s[nt][1] = exp2f(s[nt][1] - sa);
        s[nt][2] = exp2f(s[nt][2] - sb);
        s[nt][3] = exp2f(s[nt][3] - sb);
        pa += s[nt][0] + s[nt][1];
        pb += s[nt][2] + s[nt][3];
      }
      la = fmaf(la, aa, pa);
      lb = fmaf(lb, ab, pb);
#pragma unroll
      for (int n = 0; n < NN; ++n) {
        o[n][0] *= aa;
        o[n][1] *= aa;
        o[n][2] *= ab;
        o[n][3] *= ab;
      }
#pragma unroll
      for (int ks = 0; ks < NB / 16; ++ks) {
        if (t0 + 16 * ks > c_last_w) break;  // every row masked from here on (warp-uniform)
        // A = p of tokens t0 + 16ks..: n-tiles 2ks (k 0..7) and 2ks + 1 (k 8..15), hi + lo
        uint32_t ah[4], al[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x = s[2 * ks + (i >> 1)][2 * (i & 1)], y = s[2 * ks + (i >> 1)][2 * (i & 1) + 1];
          const __half2 hi = __floats2half2_rn(x, y);
          const float2 hf = __half22float2(hi);
          ah[i] = h2u(hi);
          al[i] = h2u(__floats2half2_rn(x - hf.x, y - hf.y));
        }
#pragma unroll
        for (int np = 0; np < NN / 2; ++np) {  // channel n-tiles 2np, 2np + 1
          uint32_t bv[4];
          ldsm_x4_trans(base + swz_row<D>(NB + 16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * np + (lane >> 4)), bv);
          mma16816(o[2 * np], ah, bv[0], bv[1]);
          mma16816(o[2 * np], al, bv[0], bv[1]);
          mma16816(o[2 * np + 1], ah, bv[2], bv[3]);
          mma16816(o[2 * np + 1], al, bv[2], bv[3]);
        }
      }
    }
    __syncthreads();  // the stage buffer is refilled two blocks on
  }
  if (!warp_live) return;
  la += __shfl_xor_sync(0xffffffffu, la, 1);
  la += __shfl_xor_sync(0xffffffffu, la, 2);
  lb += __shfl_xor_sync(0xffffffffu, lb, 1);
  lb += __shfl_xor_sync(0xffffffffu, lb, 2);
  // rotation: channel bit 0 within the lane, bits 1-2 across the quad, bits 3.. across n-tiles
#pragma unroll
  for (int n = 0; n < NN; ++n) {
#pragma unroll
    for (int r = 0; r < 4; r += 2) {
      const float x = o[n][r], y = o[n][r + 1];
      o[n][r] = x + y;
      o[n][r + 1] = x - y;
    }
  }
#pragma unroll
  for (int msk = 1; msk <= 2; msk <<= 1) {
    const bool upper = (tq & msk) != 0;
#pragma unroll
    for (int n = 0; n < NN; ++n)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float v = o[n][r], w = __shfl_xor_sync(0xffffffffu, v, msk);
        o[n][r] = upper ? w - v : v + w;
      }
  }
#pragma unroll
  for (int st = 1; st < NN; st <<= 1)
#pragma unroll
    for (int n = 0; n < NN; ++n)
      if ((n & st) == 0)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float x = o[n][r], y = o[n + st][r];
          o[n][r] = x + y;
          o[n + st][r] = x - y;
        }
  const int cap = p.max_pages * kTile + (kTile - 1);
  int len = p.seq_lens[b];
  len = len < 0 ? 0 : (len > cap ? cap : len);
  const int split = (len / kTile + p.pages_per_split - 1) / p.pages_per_split + (len % kTile > 0 ? 1 : 0);
  auto store = [&](int r, int c, int hf, float m, float l) {  // hf: o[.][2 hf..2 hf + 1]
    const int j = r - c * G;
    const int64_t gw = ((int64_t)b * C + c) * p.num_q_heads + h * G + j;
    float* dst = p.part + (gw * p.max_splits + split) * (D + 4);
#pragma unroll
    for (int n = 0; n < NN; ++n)
      *reinterpret_cast<float2*>(dst + 4 + 8 * n + 2 * tq) =
          make_float2(o[n][2 * hf] * inv_sqrt_d<D>(), o[n][2 * hf + 1] * inv_sqrt_d<D>());
    if (tq == 0) {
      dst[0] = m;
      dst[1] = l;
    }
  };
  if (ca >= 0) store(ra, ca, 0, ma, la);
  if (cb >= 0) store(rb, cb, 1, mb, lb);
}

template <int D>
static int launch_chunk_tc_t(const DecodeParams& p, cudaStream_t stream) {
  constexpr int kSmem = 2 * 2 * 64 * 2 * D;
  static PerDeviceOnce smem_once;
  const void* fn = reinterpret_cast<const void*>(chunk_tc_kernel<D>);
  if (const int st = set_smem_limit(smem_once, fn, kSmem); st != KVARN_OK) return st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  const int64_t rows = (int64_t)p.chunk * p.group;
  cfg.gridDim = dim3((unsigned)((rows + 127) / 128), p.num_kv_heads, p.batch);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chunk_tc_kernel<D>, p) == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA;
}

template <int D>
static int launch_chunk_t(const DecodeParams& p, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  const int warps = p.batch * p.chunk * p.num_q_heads;
  cfg.gridDim = dim3((warps + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chunk_kernel<D>, p) == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA;
}

int launch_chunk_any(int d, const DecodeParams& p, cudaStream_t stream) {
  if (d == 64) return launch_chunk_tc_t<64>(p, stream);
  if (d == 128) return launch_chunk_tc_t<128>(p, stream);
  if (d == 256) return launch_chunk_t<256>(p, stream);
  return KVARN_ERR_UNSUPPORTED;
}

// Split size for long block tables.  Their sequences are long and, in a batch, of similar
// length, so the CTAs of sequences at the full table length are taken as the work: the cost
// of a size is its waves of CTAs over the GPU's CTA slots times the page rounds of one warp
// (ceil(pages / warps)); the cheapest size wins, ties going to the larger (fewer CTAs and
// partials to merge).  Tables up to 256 pages, whose lengths vary, keep 32.
template <int D, int NT, int KB, int VB>
static int split_pages_t(int64_t units, int max_pages) {
  using S = DecodeShape<D, NT, KB, VB>;
  constexpr int kBase = 32, kMax = 128;
  if (max_pages <= 256 || units < 1) return kBase;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return kBase;
  const int64_t slots = (int64_t)sms * S::kMinBlocks;
  int best = kBase;
  int64_t best_cost = INT64_MAX;
  for (int pps = kBase; pps <= kMax; ++pps) {
    const int64_t ctas = units * ((max_pages + pps - 1) / pps);
    const int64_t cost = ((ctas + slots - 1) / slots) * ((pps + S::kWarps - 1) / S::kWarps);
    if (cost <= best_cost) {
      best_cost = cost;
      best = pps;
    }
  }
  return best;
}

template <int KB, int VB>
static int split_pages_bits(int d, int nt, int64_t units, int max_pages) {
  if (nt == 1) {
    if (d == 64) return split_pages_t<64, 1, KB, VB>(units, max_pages);
    if (d == 128) return split_pages_t<128, 1, KB, VB>(units, max_pages);
    if (d == 256) return split_pages_t<256, 1, KB, VB>(units, max_pages);
  } else if (nt == 2) {
    if (d == 64) return split_pages_t<64, 2, KB, VB>(units, max_pages);
    if (d == 128) return split_pages_t<128, 2, KB, VB>(units, max_pages);
  }
  return 32;
}

int decode_split_pages(int d, int nt, int kb, int vb, int64_t units, int max_pages) {
  if (kb == 4 && vb == 2) return split_pages_bits<4, 2>(d, nt, units, max_pages);
  if (kb == 4 && vb == 4) return split_pages_bits<4, 4>(d, nt, units, max_pages);
  if (kb == 2 && vb == 2) return split_pages_bits<2, 2>(d, nt, units, max_pages);
  if (kb == 8 && vb == 4) return split_pages_bits<8, 4>(d, nt, units, max_pages);
  return 32;
}

template <int KB, int VB>
static int launch_decode_bits(int d, int nt, const DecodeParams& p, int phases, cudaStream_t stream) {
  if (nt == 1) {
    if (d == 64) return launch_decode_t<64, 1, KB, VB>(p, phases, stream);
    if (d == 128) return launch_decode_t<128, 1, KB, VB>(p, phases, stream);
    if (d == 256) return launch_decode_t<256, 1, KB, VB>(p, phases, stream);
  } else if (nt == 2) {
    if (d == 64) return launch_decode_t<64, 2, KB, VB>(p, phases, stream);
    if (d == 128) return launch_decode_t<128, 2, KB, VB>(p, phases, stream);
  }
  return KVARN_ERR_UNSUPPORTED;
}

int launch_decode_any(int d, int nt, int kb, int vb, const DecodeParams& p, cudaStream_t stream, int phases) {
  if (p.part_mode == 3) {
    if (!decode_tc_serves(d, nt, kb, vb, p) || p.part_ctas < 1) return KVARN_ERR_INVALID_ARG;
    return launch_decode_tc(p, phases, stream);
  }
  if (kb == 4 && vb == 2) return launch_decode_bits<4, 2>(d, nt, p, phases, stream);
  if (kb == 4 && vb == 4) return launch_decode_bits<4, 4>(d, nt, p, phases, stream);
  if (kb == 2 && vb == 2) return launch_decode_bits<2, 2>(d, nt, p, phases, stream);
  if (kb == 8 && vb == 4) return launch_decode_bits<8, 4>(d, nt, p, phases, stream);
  return KVARN_ERR_UNSUPPORTED;
}

}  // namespace kvarn
