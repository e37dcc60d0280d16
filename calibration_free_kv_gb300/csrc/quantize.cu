// KVarN tile quantisation: rotate, variance-normalise, round, fold, pack (sm_103a).
//
// Each (tile, kv head, K-or-V) unit of 128 tokens x d channels is quantised by one CTA
// (quantize_tc_kernel, d = 128: persistent CTAs walking a list of units; quantize_kernel,
// d = 64 / 256: one CTA per unit).
//  1. rotate: every token row is zero-padded to d and multiplied by H_d / sqrt(d)
//     [hotdry §Hadamard 旋转]: tcgen05.mma against H_128 (d = 128) or an FWHT in shared
//     memory (d = 64, 256)
//  2. normalise: channel-std step then token-std step, `iters` times (or fewer with an
//     early-stop tolerance); the log-space factor updates of the pages telescope, so the
//     kernel keeps the factors themselves (f_new = 1 / std of the un-normalised axis;
//     unchanged when the std is below eps) [hotdry §迭代方差归一化; vatt §四個步驟, Sinkhorn
//     paragraph]
//  3. asymmetric RTN: K per channel over tokens, V per token over channels (4 / 2 bits for
//     kvarn_k4v2_g128, other widths for the other presets); normalisation factors folded into
//     the fp16 scale/zero [hotdry §非对称量化与尺度折叠]
//  4. codes packed as m16n8k16 A-operand fragments (layout in kvarn.h).
//
// Thread layout.  The unit is viewed as L x C: K has L = tokens, C = channels; V is held
// transposed, L = channels, C = tokens.  Warp w owns L rows [32(w % NLQ), +32) and C columns
// [64(w / NLQ), +64); lane (g = lane/4, tq = lane%4) owns L rows {g + 8l : l < 4} and C columns
// {8u + 2tq + p : u < 8, p < 2} of that block (64 values).  In both K and V the quantisation
// group runs along L, and each lane's values are exactly the code fragments it packs.
#include "common.cuh"
#include "params.cuh"

namespace kvarn {

// Launch as a programmatic dependent of the previous kernel in the stream: the CTAs may be
// scheduled while it drains and wait for it (griddepcontrol.wait) before reading anything.
template <typename... KArgs, typename... Args>
static int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, int smem, cudaStream_t stream,
                      Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA;
}

template <int D>
struct QuantShape {
  static constexpr int kThreads = 2 * D;       // D/16 warps, 64 values per thread
  static constexpr int kLd = D + 8;            // fp32 row stride of the staged tile
  static constexpr int kSmemBytes = kTile * kLd * 4;
};

template <int N>
__device__ __forceinline__ void fwht_regs(float (&v)[N]) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
}

// One reduce-scatter step across lanes `mask` apart, merging (sum, centred sum of squares)
// pairs of equal count n with Chan's formula.  Keeps K/2 of the K pairs.
template <int K>
__device__ __forceinline__ void rs_chan(float (&s)[K], float (&m2)[K], int mask, bool up, float n) {
#pragma unroll
  for (int i = 0; i < K / 2; ++i) {
    const float s_send = up ? s[i] : s[i + K / 2];
    const float m_send = up ? m2[i] : m2[i + K / 2];
    const float s_keep = up ? s[i + K / 2] : s[i];
    const float m_keep = up ? m2[i + K / 2] : m2[i];
    const float s_oth = __shfl_xor_sync(0xffffffffu, s_send, mask);
    const float m_oth = __shfl_xor_sync(0xffffffffu, m_send, mask);
    const float delta = (s_oth - s_keep) * (1.0f / n);
    s[i] = s_keep + s_oth;
    m2[i] = fmaf(delta * delta, 0.5f * n, m_keep + m_oth);
  }
}

template <int K>
__device__ __forceinline__ void rs_minmax(float (&mn)[K], float (&mx)[K], int mask, bool up) {
#pragma unroll
  for (int i = 0; i < K / 2; ++i) {
    const float a_send = up ? mn[i] : mn[i + K / 2];
    const float b_send = up ? mx[i] : mx[i + K / 2];
    const float a_keep = up ? mn[i + K / 2] : mn[i];
    const float b_keep = up ? mx[i + K / 2] : mx[i];
    mn[i] = fminf(a_keep, __shfl_xor_sync(0xffffffffu, a_send, mask));
    mx[i] = fmaxf(b_keep, __shfl_xor_sync(0xffffffffu, b_send, mask));
  }
}

__device__ __forceinline__ void chan_merge(float& s, float& m2, float s2, float m22, float n) {
  const float delta = (s2 - s) * (1.0f / n);
  s = s + s2;
  m2 = fmaf(delta * delta, 0.5f * n, m2 + m22);
}

// chan_merge for two columns at once.
__device__ __forceinline__ void chan_merge2(float2& s, float2& m2, float2 s2, float2 m22, float n) {
  const float2 delta = mul2(sub2(s2, s), make_float2(1.0f / n, 1.0f / n));
  s = add2(s, s2);
  m2 = fma2(mul2(delta, delta), make_float2(0.5f * n, 0.5f * n), add2(m2, m22));
}

// rs_chan over pairs of columns: keeps K/2 of the first K pairs.
template <int K, int N>
__device__ __forceinline__ void rs_chan2(float2 (&s)[N], float2 (&m2)[N], int mask, bool up, float n) {
  static_assert(K <= N, "pairs in the array");
#pragma unroll
  for (int i = 0; i < K / 2; ++i) {
    const float2 s_send = up ? s[i] : s[i + K / 2];
    const float2 m_send = up ? m2[i] : m2[i + K / 2];
    float2 s_keep = up ? s[i + K / 2] : s[i];
    float2 m_keep = up ? m2[i + K / 2] : m2[i];
    const float2 s_oth = make_float2(__shfl_xor_sync(0xffffffffu, s_send.x, mask),
                                     __shfl_xor_sync(0xffffffffu, s_send.y, mask));
    const float2 m_oth = make_float2(__shfl_xor_sync(0xffffffffu, m_send.x, mask),
                                     __shfl_xor_sync(0xffffffffu, m_send.y, mask));
    chan_merge2(s_keep, m_keep, s_oth, m_oth, n);
    s[i] = s_keep;
    m2[i] = m_keep;
  }
}


// Barrier among the `count` threads (a multiple of 32) that use barrier `id` (1..15).
__device__ __forceinline__ void group_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// New factor after one std step.  The log-space update ln f -= ln sigma (sigma = f_old * sd,
// the std of the current normalised values) telescopes to f = 1 / sd; a std below eps has
// nothing to normalise and the factor is kept.
__device__ __forceinline__ float std_step_factor(float f_old, float m2, float inv_count,
                                                 float eps, float tol_lo, float tol_hi, bool& moved) {
  const float sd = sqrtf(fmaxf(m2 * inv_count, 0.0f));
  const float sigma = f_old * sd;
  if (sigma < eps) return f_old;
  moved |= sigma > tol_hi || sigma < tol_lo;  // |ln sigma| beyond the early-stop tolerance
  return __frcp_rn(sd);
}

template <int D, bool TRANS>
__device__ __forceinline__ void stage_and_rotate(const __half* __restrict__ src, int64_t tok_stride,
                                                 int d0, float* smem, float (&x)[4][16]) {
  constexpr int NTH = QuantShape<D>::kThreads;
  constexpr int LD = QuantShape<D>::kLd;
  constexpr int LSIZE = TRANS ? D : kTile;
  constexpr int CSIZE = TRANS ? kTile : D;
  constexpr int NLQ = LSIZE / 32;
  constexpr float kInvSqrtD = D == 64 ? 0.125f : (D == 128 ? 0.08838834764831845f : 0.0625f);
  static_assert(CSIZE % 64 == 0, "C blocks of 64");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const int lq = warp % NLQ, ch = warp / NLQ;

  // ---- 1. stage the tile as fp32 and rotate every token row ---------------------------------
  float* X = smem;
  {
    constexpr int CH8 = D / 8;
    for (int idx = tid; idx < kTile * CH8; idx += NTH) {
      const int t = idx / CH8, c8 = idx - t * CH8;
      float v[8];
      if (c8 * 8 < d0) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src + t * tok_stride + c8 * 8));
        const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(h2[e]);
          v[2 * e] = f.x;
          v[2 * e + 1] = f.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.0f;
      }
      fwht_regs(v);
      float4* dst = reinterpret_cast<float4*>(X + t * LD + c8 * 8);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    __syncthreads();
    constexpr int NV = D / 8;
    for (int idx = tid; idx < kTile * 8; idx += NTH) {
      const int t = idx >> 3, c0 = idx & 7;
      float v[NV];
#pragma unroll
      for (int k = 0; k < NV; ++k) v[k] = X[t * LD + c0 + 8 * k];
      fwht_regs(v);
#pragma unroll
      for (int k = 0; k < NV; ++k) X[t * LD + c0 + 8 * k] = v[k];
    }
    __syncthreads();
  }

#pragma unroll
  for (int l = 0; l < 4; ++l) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (!TRANS) {
        const int tok = 32 * lq + g + 8 * l, c = 64 * ch + 8 * u + 2 * tq;
        const float2 f = *reinterpret_cast<const float2*>(X + tok * LD + c);
        x[l][2 * u] = f.x * kInvSqrtD;
        x[l][2 * u + 1] = f.y * kInvSqrtD;
      } else {
        const int chn = 32 * lq + g + 8 * l, tok = 64 * ch + 8 * u + 2 * tq;
        x[l][2 * u] = X[tok * LD + chn] * kInvSqrtD;
        x[l][2 * u + 1] = X[(tok + 1) * LD + chn] * kInvSqrtD;
      }
    }
  }
  __syncthreads();  // the staged tile is dead; its shared memory becomes reduction scratch

}

// Scratch floats quantize_rotated needs: two [NLQ][CSIZE] and two [NCH][LSIZE] buffers of
// (sum, centred sum of squares) pairs, plus every warp's copy of its 64 column and 32 row factors.
template <int D>
struct RotScratch {
  static constexpr int kL = D > kTile ? D : kTile;  // LSIZE or CSIZE, whichever is larger
  static constexpr int kWarps = QuantShape<D>::kThreads / 32;
  static constexpr int kFloats = 2 * (2 * (kL / 32) * kL) + 2 * (2 * (kL / 64) * kL) + kWarps * 96;
  static_assert(kFloats * 4 <= QuantShape<D>::kSmemBytes, "scratch fits the staged tile");
};

// Normalise, quantise, fold and pack one rotated unit held as x (layout above) into its half of
// the page record.  smem: at least RotScratch<D>::kFloats floats of scratch.
//
// Reductions along C stay within the two (D = 64: one; D = 256: four) warps that share an L
// block, reductions along L within the warps that share a C block, so each std step needs one
// barrier among those warps only.  Every warp of such a group merges the group's partials
// itself and keeps its own copy of the factors it needs, which removes the second barrier a
// single merging warp would need to hand its result out.  The partial buffers alternate between
// two copies from one step to the next: a warp can only refill a copy after every warp of its
// group has passed the barrier of the step in between, i.e. finished reading it.
// Returns the iterations used: `iters`, or fewer when tol_hi > 0 and an iteration's std
// steps all had sigma within [tol_lo, tol_hi] (decided for the whole CTA).
template <int D, bool TRANS, int KB, int VB>
__device__ __forceinline__ int quantize_rotated(float (&x)[4][16], uint8_t* __restrict__ rec,
                                                int iters, float eps, float tol_lo, float tol_hi,
                                                float* smem) {
  constexpr int LSIZE = TRANS ? D : kTile;
  constexpr int CSIZE = TRANS ? kTile : D;
  constexpr int NLQ = LSIZE / 32;
  constexpr int NCH = CSIZE / 64;
  constexpr int BITS = TRANS ? VB : KB;
  constexpr int QMAX = (1 << BITS) - 1;
  constexpr RecordLayout RL = record_layout(D, KB, VB);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const int lq = warp % NLQ, ch = warp / NLQ;

  constexpr int kMaxL = RotScratch<D>::kL;
  float2* redA = reinterpret_cast<float2*>(smem);         // [2][NLQ][CSIZE]  reductions along L
  float2* redB = redA + 2 * (kMaxL / 32) * kMaxL;          // [2][NCH][LSIZE]  reductions along C
  float* fCw = reinterpret_cast<float*>(redB + 2 * (kMaxL / 64) * kMaxL) + warp * 96;  // [64]
  float* fLw = fCw + 64;                                   // [32]

  // After the reduce-scatters a lane holds the statistics of C columns 64ch + ci, ci + 1 and
  // of L row 32lq + ri: these are the entries of fCw / fLw it owns.
  const int ci = 8 * g + 2 * tq;
  const int l_fin = 2 * (tq & 1) + (tq >> 1);
  const int ri = g + 8 * l_fin;
  const int c_col = 64 * ch + ci;
  const int l_row = 32 * lq + ri;

  float fL[4], fC[16];
#pragma unroll
  for (int l = 0; l < 4; ++l) fL[l] = 1.0f;
#pragma unroll
  for (int c = 0; c < 16; ++c) fC[c] = 1.0f;
  *reinterpret_cast<float2*>(&fCw[ci]) = make_float2(1.0f, 1.0f);
  fLw[ri] = 1.0f;

  auto X = [&](int l, int u) { return make_float2(x[l][2 * u], x[l][2 * u + 1]); };
  auto FC = [&](int u) { return make_float2(fC[2 * u], fC[2 * u + 1]); };
  auto FL = [&](int l) { return make_float2(fL[l], fL[l]); };

  // std over L of each C column -> new C factors (the k-th such step uses buffer k % 2)
  bool moved = false;  // a factor this thread computed moved beyond the early-stop tolerance
  auto update_c = [&](int k) {
    // Column pairs (2u, 2u + 1): sum and centred sum of squares of 4 rows.  The products are
    // rounded before a pairwise sum, so identical values give an exact mean and a zero sum of
    // squares (a constant column has std 0, not rounding noise that could exceed eps).
    float2 S[8], M[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float2 y0 = mul2(X(0, u), FL(0)), y1 = mul2(X(1, u), FL(1));
      const float2 y2 = mul2(X(2, u), FL(2)), y3 = mul2(X(3, u), FL(3));
      const float2 s = add2(add2(y0, y1), add2(y2, y3));
      const float2 mu = mul2(s, make_float2(0.25f, 0.25f));
      const float2 d0_ = sub2(y0, mu), d1 = sub2(y1, mu), d2 = sub2(y2, mu), d3 = sub2(y3, mu);
      S[u] = s;
      M[u] = add2(fma2(d0_, d0_, mul2(d1, d1)), fma2(d2, d2, mul2(d3, d3)));
    }
    rs_chan2<8>(S, M, 16, (lane & 16) != 0, 4.0f);
    rs_chan2<4>(S, M, 8, (lane & 8) != 0, 8.0f);
    rs_chan2<2>(S, M, 4, (lane & 4) != 0, 16.0f);  // S[0], M[0]: columns c_col, c_col + 1
    float2 s = S[0], m = M[0];
    if (NLQ > 1) {
      float4* buf = reinterpret_cast<float4*>(redA + (k & 1) * NLQ * CSIZE);
      buf[(lq * CSIZE + c_col) >> 1] = make_float4(s.x, s.y, m.x, m.y);
      group_sync(1 + ch, NLQ * 32);
      float2 ps[NLQ], pm[NLQ];
#pragma unroll
      for (int q = 0; q < NLQ; ++q) {
        const float4 v = buf[(q * CSIZE + c_col) >> 1];
        ps[q] = make_float2(v.x, v.y);
        pm[q] = make_float2(v.z, v.w);
      }
      float n = 32.0f;
#pragma unroll
      for (int w = 1; w < NLQ; w <<= 1) {
#pragma unroll
        for (int q = 0; q + w < NLQ; q += 2 * w) chan_merge2(ps[q], pm[q], ps[q + w], pm[q + w], n);
        n *= 2.0f;
      }
      m = pm[0];
    }
    float2 f = *reinterpret_cast<const float2*>(&fCw[ci]);
    f.x = std_step_factor(f.x, m.x, 1.0f / LSIZE, eps, tol_lo, tol_hi, moved);
    f.y = std_step_factor(f.y, m.y, 1.0f / LSIZE, eps, tol_lo, tol_hi, moved);
    *reinterpret_cast<float2*>(&fCw[ci]) = f;
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float2 v = *reinterpret_cast<const float2*>(&fCw[8 * u + 2 * tq]);
      fC[2 * u] = v.x;
      fC[2 * u + 1] = v.y;
    }
  };

  // std over C of each L row -> new L factors (the k-th such step uses buffer k % 2)
  auto update_l = [&](int k) {
    float2 S2[2], M2[2];  // rows (0, 1) and (2, 3): sum and centred sum of squares of 16 columns
#pragma unroll
    for (int l = 0; l < 4; ++l) {  // rounded products, pairwise sum (exact for a constant row)
      float2 y[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) y[u] = mul2(X(l, u), FC(u));
      const float2 t = add2(add2(add2(y[0], y[1]), add2(y[2], y[3])), add2(add2(y[4], y[5]), add2(y[6], y[7])));
      const float s = t.x + t.y;
      const float mu = s * (1.0f / 16.0f);
      float2 q = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float2 d = sub2(y[u], make_float2(mu, mu));
        q = fma2(d, d, q);
      }
      if (l & 1) {
        S2[l >> 1].y = s;
        M2[l >> 1].y = q.x + q.y;
      } else {
        S2[l >> 1].x = s;
        M2[l >> 1].x = q.x + q.y;
      }
    }
    rs_chan2<2>(S2, M2, 1, (lane & 1) != 0, 16.0f);  // rows (0, 1) or (2, 3)
    float s1[2] = {S2[0].x, S2[0].y}, m1[2] = {M2[0].x, M2[0].y};
    rs_chan<2>(s1, m1, 2, (lane & 2) != 0, 32.0f);  // row l_fin
    float s = s1[0], m = m1[0];
    if (NCH > 1) {
      float2* buf = redB + (k & 1) * NCH * LSIZE;
      buf[ch * LSIZE + l_row] = make_float2(s, m);
      group_sync(1 + NCH + lq, NCH * 32);
      float ps[NCH], pm[NCH];
#pragma unroll
      for (int q = 0; q < NCH; ++q) {
        const float2 v = buf[q * LSIZE + l_row];
        ps[q] = v.x;
        pm[q] = v.y;
      }
      float n = 64.0f;
#pragma unroll
      for (int w = 1; w < NCH; w <<= 1) {
#pragma unroll
        for (int q = 0; q + w < NCH; q += 2 * w) chan_merge(ps[q], pm[q], ps[q + w], pm[q + w], n);
        n *= 2.0f;
      }
      m = pm[0];
    }
    fLw[ri] = std_step_factor(fLw[ri], m, 1.0f / CSIZE, eps, tol_lo, tol_hi, moved);
    __syncwarp();
#pragma unroll
    for (int l = 0; l < 4; ++l) fL[l] = fLw[g + 8 * l];
  };

  // ---- 2. variance normalisation: channel-std step, then token-std step -------------------
  int used = 0;
  for (int it = 0; it < iters; ++it) {
    if (!TRANS) {  // K: channels are C, tokens are L
      update_c(it);
      update_l(it);
    } else {       // V: channels are L, tokens are C
      update_l(it);
      update_c(it);
    }
    ++used;
    if (tol_hi > 0.0f) {  // one decision for the CTA: stop unless some factor still moved
      if (!__syncthreads_or(moved ? 1 : 0)) break;
      moved = false;
    }
  }

  // ---- 3. per-column (along L) min / max, scale, zero-point ---------------------------------
  // N = (x fL) fC with fC > 0 fixed per column, and rounding is monotonic, so the extremes of N
  // are the extremes of z = x fL times fC, rounded once.
  float4* qbuf = reinterpret_cast<float4*>(redA + ((used + 1) & 1) * NLQ * CSIZE + lq * CSIZE + 64 * ch);
  {
    float mn[16], mx[16];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float2 z0 = mul2(X(0, u), FL(0)), z1 = mul2(X(1, u), FL(1));
      const float2 z2 = mul2(X(2, u), FL(2)), z3 = mul2(X(3, u), FL(3));
      mn[2 * u] = fminf(fmin3(z0.x, z1.x, z2.x), z3.x);
      mn[2 * u + 1] = fminf(fmin3(z0.y, z1.y, z2.y), z3.y);
      mx[2 * u] = fmaxf(fmax3(z0.x, z1.x, z2.x), z3.x);
      mx[2 * u + 1] = fmaxf(fmax3(z0.y, z1.y, z2.y), z3.y);
    }
    float mn8[8], mx8[8], mn4[4], mx4[4];
    rs_minmax<16>(mn, mx, 16, (lane & 16) != 0);
#pragma unroll
    for (int i = 0; i < 8; ++i) { mn8[i] = mn[i]; mx8[i] = mx[i]; }
    rs_minmax<8>(mn8, mx8, 8, (lane & 8) != 0);
#pragma unroll
    for (int i = 0; i < 4; ++i) { mn4[i] = mn8[i]; mx4[i] = mx8[i]; }
    rs_minmax<4>(mn4, mx4, 4, (lane & 4) != 0);
    float2 zmin = make_float2(mn4[0], mn4[1]), zmax = make_float2(mx4[0], mx4[1]);
    if (NLQ > 1) {
      float4* buf = reinterpret_cast<float4*>(redA + (used & 1) * NLQ * CSIZE);
      buf[(lq * CSIZE + c_col) >> 1] = make_float4(zmin.x, zmin.y, zmax.x, zmax.y);
      group_sync(1 + ch, NLQ * 32);
#pragma unroll
      for (int q = 0; q < NLQ; ++q) {
        if (q == lq) continue;
        const float4 v = buf[(q * CSIZE + c_col) >> 1];
        zmin = make_float2(fminf(zmin.x, v.x), fminf(zmin.y, v.y));
        zmax = make_float2(fmaxf(zmax.x, v.z), fmaxf(zmax.y, v.w));
      }
    }
    const float2 fc = *reinterpret_cast<const float2*>(&fCw[ci]);
    const float2 m = mul2(zmin, fc), M = mul2(zmax, fc);
    const float s0 = fmaxf(__fdiv_rn(__fsub_rn(M.x, m.x), (float)QMAX), 1e-8f);
    const float s1 = fmaxf(__fdiv_rn(__fsub_rn(M.y, m.y), (float)QMAX), 1e-8f);
    qbuf[ci >> 1] = make_float4(m.x, m.y, __frcp_rn(s0), __frcp_rn(s1));
    if (lq == 0) {  // folded: s' = s / fC, z' = m / fC
      __half* scale_out = reinterpret_cast<__half*>(rec + (TRANS ? RL.vscale : RL.kscale));
      __half* zero_out = reinterpret_cast<__half*>(rec + (TRANS ? RL.vzero : RL.kzero));
      *reinterpret_cast<__half2*>(&scale_out[c_col]) =
          __floats2half2_rn(__fdiv_rn(s0, fc.x), __fdiv_rn(s1, fc.y));
      *reinterpret_cast<__half2*>(&zero_out[c_col]) =
          __floats2half2_rn(__fdiv_rn(m.x, fc.x), __fdiv_rn(m.y, fc.y));
    }
  }

  // token / channel factor of the L axis: r = 1/fL (K) or c = 1/fL (V)
  if (ch == 0) {
    __half* fac_out = reinterpret_cast<__half*>(rec + (TRANS ? RL.vfactor : RL.kfactor));
    fac_out[l_row] = __float2half_rn(__frcp_rn(fLw[ri]));
  }
  __syncwarp();

  // ---- 4. codes, packed as mma fragments -----------------------------------------------------
  // (N - m) / s lies in [0, QMAX] for finite input, so adding 1.5 * 2^23 (round half to even)
  // leaves the code alone in the low byte of the float's bits.
  uint32_t code[4][16];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float4 q = qbuf[4 * u + tq];
    const float2 m = make_float2(q.x, q.y), inv = make_float2(q.z, q.w);
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const float2 nv = mul2(mul2(X(l, u), FL(l)), FC(u));
      const float2 v = add2(mul2(sub2(nv, m), inv), make_float2(12582912.0f, 12582912.0f));
      code[l][2 * u] = __float_as_uint(v.x);
      code[l][2 * u + 1] = __float_as_uint(v.y);
    }
  }
  // low bytes of four code registers -> one word, byte i from register i
  auto gather4 = [](uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x4000), 0x7610);
  };
  // Words of BITS-bit codes (layout in kvarn.h).  A lane's codes form the fragments of row
  // blocks 2lq + lh (from L) and column blocks 4ch + j (from C), element (rho, h, p) at row
  // 2lh + rho, column 2(2j + h) + p of x.  K: token block = row block; V: token block =
  // column block.
  constexpr int NI4 = D / 64;
  if constexpr (BITS == 4) {
    // nibble h + 2rho + 4p: byte rho + 2p holds h = 0 in its low and h = 1 in its high nibble
    uint32_t w[2][4];
#pragma unroll
    for (int lh = 0; lh < 2; ++lh)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c0 = 4 * j, c1 = 4 * j + 2, r0 = 2 * lh, r1 = 2 * lh + 1;
        const uint32_t lo = gather4(code[r0][c0], code[r1][c0], code[r0][c0 + 1], code[r1][c0 + 1]);
        const uint32_t hi = gather4(code[r0][c1], code[r1][c1], code[r0][c1 + 1], code[r1][c1 + 1]);
        w[lh][j] = (lo & 0x0F0F0F0Fu) | ((hi << 4) & 0xF0F0F0F0u);
      }
    if constexpr (!TRANS) {  // word (token block 2lq + lh, channel block 4ch + j)
      uint8_t* kc = rec + RL.kcodes;
#pragma unroll
      for (int lh = 0; lh < 2; ++lh)
        *reinterpret_cast<uint4*>(kc + (((2 * lq + lh) * NI4 + ch) * 32 + lane) * 16) =
            make_uint4(w[lh][0], w[lh][1], w[lh][2], w[lh][3]);
    } else {                 // word (token block 4ch + j, channel block 2lq + lh)
      uint8_t* vc = rec + RL.vcodes;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint2*>(vc + ((((4 * ch + j) * NI4 + lq / 2) * 32 + lane) * 4 + 2 * (lq & 1)) * 4) =
            make_uint2(w[0][j], w[1][j]);
    }
  } else if constexpr (BITS == 8) {
    // fragment (row block 2lq + lh, column block 4ch + j) in two words h = 0, 1: element
    // (rho, h, p) at byte rho + 2p of word h, which is gather4's order
    auto w8 = [&](int lh, int j, int hh) {
      const int c = 2 * (2 * j + hh), r0 = 2 * lh, r1 = 2 * lh + 1;
      return gather4(code[r0][c], code[r1][c], code[r0][c + 1], code[r1][c + 1]);
    };
    constexpr int NI2 = D / 32;
    if constexpr (!TRANS) {  // words of (token block 2lq + lh, channel blocks 4ch + 2jj, + 1)
      uint8_t* kc = rec + RL.kcodes;
#pragma unroll
      for (int lh = 0; lh < 2; ++lh)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
          *reinterpret_cast<uint4*>(kc + (((2 * lq + lh) * NI2 + 2 * ch + jj) * 32 + lane) * 16) =
              make_uint4(w8(lh, 2 * jj, 0), w8(lh, 2 * jj, 1), w8(lh, 2 * jj + 1, 0), w8(lh, 2 * jj + 1, 1));
    } else {                 // words of (token block 4ch + j, channel blocks 2lq, 2lq + 1)
      uint8_t* vc = rec + RL.vcodes;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(vc + (((4 * ch + j) * NI2 + lq) * 32 + lane) * 16) =
            make_uint4(w8(0, j, 0), w8(0, j, 1), w8(1, j, 0), w8(1, j, 1));
    }
  } else {
    static_assert(BITS == 2, "2-, 4- or 8-bit codes");
    if constexpr (!TRANS) {
      // word (token blocks 2lq and 2lq + 1, channel block 4ch + j): slot 2lh + h + 4rho + 8p,
      // i.e. byte rho + 2p, bit pair 2lh + h
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t acc = 0u;
#pragma unroll
        for (int s2 = 3; s2 >= 0; --s2) {
          const int lh = s2 >> 1, c = 2 * (2 * j + (s2 & 1)), r0 = 2 * lh, r1 = 2 * lh + 1;
          const uint32_t b = gather4(code[r0][c], code[r1][c], code[r0][c + 1], code[r1][c + 1]);
          acc = (acc << 2) | (b & 0x03030303u);
        }
        w[j] = acc;
      }
      *reinterpret_cast<uint4*>(rec + RL.kcodes + ((lq * NI4 + ch) * 32 + lane) * 16) =
          make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      // word (token blocks 4ch + 2uh and + 1, channel block 2lq + lh): slot uu + 4rho + 8p for
      // column 2(4uh + uu) + p, i.e. byte rho + 2p, bit pair uu
      uint8_t* vc = rec + RL.vcodes;
#pragma unroll
      for (int uh = 0; uh < 2; ++uh) {
        uint32_t w[2];
#pragma unroll
        for (int lh = 0; lh < 2; ++lh) {
          uint32_t acc = 0u;
#pragma unroll
          for (int uu = 3; uu >= 0; --uu) {
            const int c = 2 * (4 * uh + uu), r0 = 2 * lh, r1 = 2 * lh + 1;
            const uint32_t b = gather4(code[r0][c], code[r1][c], code[r0][c + 1], code[r1][c + 1]);
            acc = (acc << 2) | (b & 0x03030303u);
          }
          w[lh] = acc;
        }
        const int ks2 = 2 * ch + uh;
        *reinterpret_cast<uint2*>(vc + (((ks2 * NI4 + lq / 2) * 32 + lane) * 4 + 2 * (lq & 1)) * 4) =
            make_uint2(w[0], w[1]);
      }
    }
  }
  return used;
}

template <int D, bool TRANS, int KB, int VB>
__device__ __forceinline__ int quantize_unit(const __half* __restrict__ src, int64_t tok_stride,
                                             int d0, uint8_t* __restrict__ rec, const QuantizeParams& p,
                                             float* smem) {
  float x[4][16];
  stage_and_rotate<D, TRANS>(src, tok_stride, d0, smem, x);
  return quantize_rotated<D, TRANS, KB, VB>(x, rec, p.iters, p.eps, p.tol_lo, p.tol_hi, smem);
}

// ---- kernels --------------------------------------------------------------------------------


// grid.x = units * 2 (K and V of one (tile or sequence, kv head)), block = 2*D threads.
template <int D, int KB, int VB>
__global__ void __launch_bounds__(QuantShape<D>::kThreads)
    quantize_kernel(QuantizeParams p) {
  extern __shared__ __align__(16) float smem_q[];
  grid_dependency_wait();  // inputs, lengths and partial tiles may come from the previous kernel
  grid_launch_dependents();
  const int unit = blockIdx.x >> 1;
  const bool is_v = (blockIdx.x & 1) != 0;
  const int h = unit % p.num_kv_heads;
  const int tile = unit / p.num_kv_heads;

  const __half* src;
  int64_t tok_stride;
  int64_t page;
  if (!p.append) {
    src = (is_v ? p.v : p.k) + (int64_t)tile * kTile * p.tok_stride + (int64_t)h * p.head_stride;
    tok_stride = p.tok_stride;
    page = p.page_ids[tile];
  } else {
    // append: tile == sequence index b
    const int b = tile;
    const int len = p.seq_lens[b];
    const int cap = p.max_pages * kTile;
    if (len < 0 || len >= cap) {
      if (threadIdx.x == 0 && !is_v && h == 0) flag_error(p.status, KVARN_DEV_SEQ_TOO_LONG);
      return;
    }
    const int row = len % kTile;
    __half* part = (is_v ? p.partial_v : p.partial_k) + ((int64_t)b * p.num_kv_heads + h) * kTile * p.d0;
    const __half* nw = (is_v ? p.v_new : p.k_new) + ((int64_t)b * p.num_kv_heads + h) * p.d0;
    for (int c = threadIdx.x * 8; c < p.d0; c += blockDim.x * 8)
      *reinterpret_cast<uint4*>(part + row * p.d0 + c) = *reinterpret_cast<const uint4*>(nw + c);
    if (threadIdx.x == 0 && !is_v && h == 0 && p.seq_lens_out != nullptr) p.seq_lens_out[b] = len + 1;
    if (row != kTile - 1) return;
    __syncthreads();  // the new row is visible to the whole block
    src = part;
    tok_stride = p.d0;
    page = p.block_table[(int64_t)b * p.max_pages + len / kTile];
  }
  if (page < 0 || page >= p.num_pool_pages) {
    if (threadIdx.x == 0) flag_error(p.status, KVARN_DEV_BAD_PAGE_ID);
    return;
  }
  uint8_t* rec = p.pool + (page * p.num_kv_heads + h) * p.rec_bytes;
  const int used = is_v ? quantize_unit<D, true, KB, VB>(src, tok_stride, p.d0, rec, p, smem_q)
                        : quantize_unit<D, false, KB, VB>(src, tok_stride, p.d0, rec, p, smem_q);
  if (p.iters_out != nullptr && !p.append && threadIdx.x == 0) p.iters_out[blockIdx.x] = used;
}

template <int D, int KB, int VB>
static int launch_quantize(const QuantizeParams& p, int units, cudaStream_t stream) {
  constexpr int kSmem = QuantShape<D>::kSmemBytes;
  static PerDeviceOnce smem_once;  // the attribute is set once per device
  const void* fn = reinterpret_cast<const void*>(quantize_kernel<D, KB, VB>);
  if (const int st = set_smem_limit(smem_once, fn, kSmem); st != KVARN_OK) return st;
  return launch_pdl(quantize_kernel<D, KB, VB>, dim3(units * 2), dim3(QuantShape<D>::kThreads), kSmem,
                    stream, p);
}

// ---- head_dim 128: the rotation on the tensor cores, the statistics one line per thread -------
//
// Persistent CTAs of 256 threads (two per SM) walk a list of units.  Each CTA builds H_128 once
// in shared memory.  Per unit, two tcgen05.mma rotations (fp16 operands, exact +-1 entries, fp32
// accumulation) put the tile into tensor memory twice: A = Z.H (TMEM lanes = tokens, columns =
// channels) and B = H.Z^T (lanes = channels, columns = tokens).  The rotation's 1/sqrt(d) is
// folded into the initial token factors instead of being applied to the values.
//
// A std step normalises the lines of one orientation: the channel step the lines of B, the
// token step the lines of A.  Thread (warp w, lane t) owns line 32(w % 4) + t and its columns
// [64(w / 4), +64): it streams its 64 values out of tensor memory and scales them by the other
// axis' factors (broadcast from shared memory); the half line gets an exact two-pass mean and
// centred sum of squares, and one shared-memory exchange with the partner thread that holds
// the other 64 columns merges the halves (Chan's formula).
//
// Quantisation: the min / max of each group is taken one group per line (K: lines of B, V:
// lines of A) and the codes are formed in the 16x256b layout of the other orientation (K: A,
// V: B), where every thread holds exactly the fragments it packs.
namespace tc {
constexpr int kThreads = 256;
constexpr int kOpBytes = 128 * 128 * 2;              // one 128 x 128 fp16 operand
constexpr uint32_t kLbo = 128;                       // K-adjacent 8x8 core matrices
constexpr uint32_t kSbo = 2048;                      // row-band-adjacent core matrices
constexpr int kHOff = 0;
constexpr int kZOff = kOpBytes;                      // two tile buffers
constexpr int kFOff = 3 * kOpBytes;                  // token factors fT[128], channel factors fC[128]
constexpr int kXOff = kFOff + 2 * 128 * 4;           // partner exchange, float4 [256]
constexpr int kQOff = kXOff + kThreads * 16;         // group (m, 1/s), float2 [128]
constexpr int kListCap = 256;                        // units per CTA
constexpr int kIoOff = kQOff + 64 * 16;                // per listed unit: tile source, record
constexpr int kListOff = kIoOff + kListCap * 16;
constexpr int kBarOff = kListOff + kListCap * 4;
constexpr int kSmemBytes = kBarOff + 64;
constexpr int kTmemCols = 256;                       // A (columns 0..127) and B (128..255)
// kind::f16 instruction descriptor: f32 accumulate, f16 A and B, both K-major, N = 128, M = 128
constexpr uint32_t kIdesc = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr float kInvSqrt128 = 0.08838834764831845f;

__device__ __forceinline__ uint32_t canon(int r, int k) {  // byte offset of element (r, k)
  return (uint32_t)((r >> 3) * kSbo + (k >> 3) * kLbo + (r & 7) * 16 + (k & 7) * 2);
}

// Shared-memory matrix descriptor: no swizzle, canonical K-major layout.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(kLbo >> 4) << 16) |
         ((uint64_t)(kSbo >> 4) << 32) | ((uint64_t)1 << 46);
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
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 consecutive accumulator columns of 16 TMEM lanes (16x256b, 8 repetitions).
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 32 consecutive columns of the warp's 32 TMEM lanes (32x32b, 32 repetitions): lane t of the
// warp receives its own lane's values.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// The thread's 64 values of its line: columns [64 hf, +64) of TMEM lane `line`.
__device__ __forceinline__ void load_line(uint32_t taddr, uint32_t (&r)[64]) {
  uint32_t (&lo)[32] = *reinterpret_cast<uint32_t (*)[32]>(&r[0]);
  uint32_t (&hi)[32] = *reinterpret_cast<uint32_t (*)[32]>(&r[32]);
  tmem_ld_32x32b_x32(taddr, lo);
  tmem_ld_32x32b_x32(taddr + 32, hi);
  tmem_wait_ld();
}

// Source tile and destination record of a unit; false if the unit has nothing to do.
__device__ __forceinline__ bool unit_io(const QuantizeParams& p, int u, const __half*& src,
                                        int64_t& tok_stride, uint8_t*& rec) {
  const int h = (u >> 1) % p.num_kv_heads;
  const int t = (u >> 1) / p.num_kv_heads;  // tile, or sequence in append mode
  const bool is_v = (u & 1) != 0;
  int64_t page;
  if (!p.append) {
    src = (is_v ? p.v : p.k) + (int64_t)t * kTile * p.tok_stride + (int64_t)h * p.head_stride;
    tok_stride = p.tok_stride;
    page = p.page_ids[t];
  } else {
    const int len = p.seq_lens[t];
    if (len < 0 || len >= p.max_pages * kTile || len % kTile != kTile - 1) return false;
    src = (is_v ? p.partial_v : p.partial_k) + ((int64_t)t * p.num_kv_heads + h) * kTile * p.d0;
    tok_stride = p.d0;
    page = p.block_table[(int64_t)t * p.max_pages + len / kTile];
  }
  if (page < 0 || page >= p.num_pool_pages) return false;
  rec = p.pool + (page * p.num_kv_heads + h) * p.rec_bytes;
  return true;
}

// Stage one fp16 tile (128 tokens x d0, zero-padded to 128) into a canonical K-major buffer:
// thread t copies the 16-byte chunk c8 = (t / 8) % 16 of tokens t0 + 16j, t0 = t % 8 + 8 (t / 128),
// j < 8 (16-byte chunks past d0 are zero-filled).
__device__ __forceinline__ void load_tile(uint32_t zbuf, const __half* src, int64_t tok_stride,
                                          int d0) {
  const int tid = threadIdx.x;
  const int c8 = (tid >> 3) & 15, t0 = (tid & 7) | ((tid >> 7) << 3);
  const bool in = c8 * 8 < d0;
  const __half* g = src + t0 * tok_stride + c8 * 8;
  const int64_t step = 16 * tok_stride;
  const uint32_t s = zbuf + canon(t0, c8 * 8);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    cp_async16(s + j * 2 * kSbo, in ? (const void*)(g + j * step) : (const void*)src, in ? 16u : 0u);
}

// reciprocal square root (MUFU, relative error below 2^-22; +inf at 0)
__device__ __forceinline__ float rsqrt_approx(float x) {
  float r;
  asm("rsqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// New factor of a line from its variance: 1 / sd, or the old factor where the line's std under
// the old factor (sigma = f_old sd) is below eps.  `moved`: |ln sigma| beyond the early-stop
// tolerance.
__device__ __forceinline__ float line_factor(float f_old, float var, float eps, float tol_lo, float tol_hi,
                                             bool& moved) {
  const float v = fmaxf(var, 0.0f);
  const float rs = rsqrt_approx(v);
  const float sigma = v > 0.0f ? f_old * (v * rs) : 0.0f;
  if (!(sigma >= eps)) return f_old;
  moved = sigma > tol_hi || sigma < tol_lo;
  return rs;
}

// y = x f for the thread's 64 values, in place, each product rounded toward zero.  A product
// in another rounding mode than the adds that follow is never fused into them, so a later
// y - mean sees exactly the stored product: a line of identical y has centred values of
// exactly 0.  (Round-toward-zero is one unit in the last place at most, well inside the
// precision the normalisation needs.)
__device__ __forceinline__ float2 mul2_rz(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack_f2(a)), "l"(pack_f2(b)));
  return unpack_f2(d);
}
__device__ __forceinline__ void scale_line(uint32_t (&r)[64], const float4* f4) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float4 f = f4[k];
    const float2 y0 = mul2_rz(make_float2(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1])),
                              make_float2(f.x, f.y));
    const float2 y1 = mul2_rz(make_float2(__uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3])),
                              make_float2(f.z, f.w));
    r[4 * k] = __float_as_uint(y0.x);
    r[4 * k + 1] = __float_as_uint(y0.y);
    r[4 * k + 2] = __float_as_uint(y1.x);
    r[4 * k + 3] = __float_as_uint(y1.y);
  }
}

// One std step over the lines of one orientation (TMEM columns at taddr): every line's values
// scaled by the column factors `fcol`, its own factor in `fline[line]` replaced by the new one.
// Returns whether the factor moved beyond the early-stop tolerance.  Every thread of the CTA
// calls it; it ends with a CTA barrier, after which the new factors are visible.
//
// Each thread takes its half line (64 values) in an exact two-pass form: y = x f rounded, a
// pairwise sum (so a half line of identical values has a mean equal to its values), then the
// centred squares.  The two halves are merged with Chan's formula after one exchange with the
// partner thread: a line of identical values gets a std of exactly 0, and a large mean costs no
// precision.
__device__ __forceinline__ bool std_step(uint32_t taddr, const float* fcol, float* fline, float4* xbuf,
                                         int line, int hf, float eps, float tol_lo, float tol_hi) {
  const int tid = threadIdx.x;
  const float4* f4 = reinterpret_cast<const float4*>(fcol + 64 * hf);
  const float f_old = fline[line];
  uint32_t r[64];
  load_line(taddr, r);
  scale_line(r, f4);
  // pairwise sum of the 64 rounded y (as 32 pairs)
  float2 ps[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    ps[i] = add2(make_float2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])),
                 make_float2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) ps[i] = add2(ps[2 * i], ps[2 * i + 1]);
  const float mean_h = (ps[0].x + ps[0].y) * (1.0f / 64.0f);
  float2 q[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) q[a] = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const float2 d = sub2(make_float2(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1])),
                          make_float2(mean_h, mean_h));
    q[k & 3] = fma2(d, d, q[k & 3]);
  }
  const float2 tq = add2(add2(q[0], q[1]), add2(q[2], q[3]));
  const float m2_h = tq.x + tq.y;
  float2* x2 = reinterpret_cast<float2*>(xbuf);
  x2[2 * tid] = make_float2(mean_h, m2_h);
  __syncthreads();
  const float2 o = x2[2 * (tid ^ 128)];
  // Chan's merge of two halves of 64, the lower column half first (both partners agree)
  const float mean_lo = hf ? o.x : mean_h, m2_lo = hf ? o.y : m2_h;
  const float mean_hi = hf ? mean_h : o.x, m2_hi = hf ? m2_h : o.y;
  const float delta = mean_hi - mean_lo;
  const float var = fmaf(delta * delta, 32.0f, m2_lo + m2_hi) * (1.0f / 128.0f);
  bool moved = false;
  const float f_new = line_factor(f_old, var, eps, tol_lo, tol_hi, moved);
  if (hf == 0) fline[line] = f_new;
  __syncthreads();
  return moved;
}

// Codes of a 4 x 16 block in the 16x256b layout (rows g + 8l of the warp's 32-lane quarter,
// columns 8u + 2tq + p of its 64-column half): v = (x fL_l fC_c - m_c) / s_c, rounded half to
// even by the 1.5 * 2^23 addition (the code is the low byte of the float's bits), then packed
// as mma fragments into the record (layout in kvarn.h).
template <bool TRANS, int KB, int VB>
__device__ __forceinline__ void codes_and_pack(const float (&x)[4][16], const float (&fl)[4], const float* fcol,
                                               const float4* qpair, uint8_t* __restrict__ rec) {
  constexpr int D = 128;
  constexpr int BITS = TRANS ? VB : KB;
  constexpr RecordLayout RL = record_layout(D, KB, VB);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tq = lane & 3;
  const int lq = warp & 3, ch = warp >> 2;
  uint32_t code[4][16];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int c = 64 * ch + 8 * u + 2 * tq;
    const float4 q = qpair[c >> 1];                 // (m_c, 1/s_c, m_c+1, 1/s_c+1)
    const float2 fc = *reinterpret_cast<const float2*>(fcol + c);
    const float2 nm = make_float2(-q.x, -q.z), inv = make_float2(q.y, q.w);
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const float2 z = mul2(make_float2(x[l][2 * u], x[l][2 * u + 1]), make_float2(fl[l], fl[l]));
      const float2 dlt = fma2(z, fc, nm);
      const float2 v = fma2(dlt, inv, make_float2(12582912.0f, 12582912.0f));
      code[l][2 * u] = __float_as_uint(v.x);
      code[l][2 * u + 1] = __float_as_uint(v.y);
    }
  }
  // low bytes of four code registers -> one word, byte i from register i
  auto gather4 = [](uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x4000), 0x7610);
  };
  // A lane's codes form the fragments of row blocks 2lq + lh and column blocks 4ch + j, element
  // (rho, h, p) at row 2lh + rho, column 2(2j + h) + p of code[][].  K: token block = row
  // block; V: token block = column block.
  constexpr int NI4 = D / 64;
  if constexpr (BITS == 4) {
    uint32_t w[2][4];
#pragma unroll
    for (int lh = 0; lh < 2; ++lh)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c0 = 4 * j, c1 = 4 * j + 2, r0 = 2 * lh, r1 = 2 * lh + 1;
        const uint32_t lo = gather4(code[r0][c0], code[r1][c0], code[r0][c0 + 1], code[r1][c0 + 1]);
        const uint32_t hi = gather4(code[r0][c1], code[r1][c1], code[r0][c1 + 1], code[r1][c1 + 1]);
        w[lh][j] = (lo & 0x0F0F0F0Fu) | ((hi << 4) & 0xF0F0F0F0u);
      }
    if constexpr (!TRANS) {
      uint8_t* kc = rec + RL.kcodes;
#pragma unroll
      for (int lh = 0; lh < 2; ++lh)
        *reinterpret_cast<uint4*>(kc + (((2 * lq + lh) * NI4 + ch) * 32 + lane) * 16) =
            make_uint4(w[lh][0], w[lh][1], w[lh][2], w[lh][3]);
    } else {
      uint8_t* vc = rec + RL.vcodes;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint2*>(vc + ((((4 * ch + j) * NI4 + lq / 2) * 32 + lane) * 4 + 2 * (lq & 1)) * 4) =
            make_uint2(w[0][j], w[1][j]);
    }
  } else if constexpr (BITS == 8) {
    auto w8 = [&](int lh, int j, int hh) {
      const int c = 2 * (2 * j + hh), r0 = 2 * lh, r1 = 2 * lh + 1;
      return gather4(code[r0][c], code[r1][c], code[r0][c + 1], code[r1][c + 1]);
    };
    constexpr int NI2 = D / 32;
    if constexpr (!TRANS) {
      uint8_t* kc = rec + RL.kcodes;
#pragma unroll
      for (int lh = 0; lh < 2; ++lh)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
          *reinterpret_cast<uint4*>(kc + (((2 * lq + lh) * NI2 + 2 * ch + jj) * 32 + lane) * 16) =
              make_uint4(w8(lh, 2 * jj, 0), w8(lh, 2 * jj, 1), w8(lh, 2 * jj + 1, 0), w8(lh, 2 * jj + 1, 1));
    } else {
      uint8_t* vc = rec + RL.vcodes;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(vc + (((4 * ch + j) * NI2 + lq) * 32 + lane) * 16) =
            make_uint4(w8(0, j, 0), w8(0, j, 1), w8(1, j, 0), w8(1, j, 1));
    }
  } else {
    static_assert(BITS == 2, "2-, 4- or 8-bit codes");
    if constexpr (!TRANS) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t acc = 0u;
#pragma unroll
        for (int s2 = 3; s2 >= 0; --s2) {
          const int lh = s2 >> 1, c = 2 * (2 * j + (s2 & 1)), r0 = 2 * lh, r1 = 2 * lh + 1;
          const uint32_t b = gather4(code[r0][c], code[r1][c], code[r0][c + 1], code[r1][c + 1]);
          acc = (acc << 2) | (b & 0x03030303u);
        }
        w[j] = acc;
      }
      *reinterpret_cast<uint4*>(rec + RL.kcodes + ((lq * NI4 + ch) * 32 + lane) * 16) =
          make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      uint8_t* vc = rec + RL.vcodes;
#pragma unroll
      for (int uh = 0; uh < 2; ++uh) {
        uint32_t w[2];
#pragma unroll
        for (int lh = 0; lh < 2; ++lh) {
          uint32_t acc = 0u;
#pragma unroll
          for (int uu = 3; uu >= 0; --uu) {
            const int c = 2 * (4 * uh + uu), r0 = 2 * lh, r1 = 2 * lh + 1;
            const uint32_t b = gather4(code[r0][c], code[r1][c], code[r0][c + 1], code[r1][c + 1]);
            acc = (acc << 2) | (b & 0x03030303u);
          }
          w[lh] = acc;
        }
        const int ks2 = 2 * ch + uh;
        *reinterpret_cast<uint2*>(vc + (((ks2 * NI4 + lq / 2) * 32 + lane) * 4 + 2 * (lq & 1)) * 4) =
            make_uint2(w[0], w[1]);
      }
    }
  }
}

// Normalise, quantise, fold and pack one unit.  Its rotation B is in TMEM columns bufB when
// this is called; A (columns bufA) may still be in flight: wait_a() (CTA-uniform, idempotent,
// false on a timeout) is called before A's first use.  Between the group pass and the codes
// pass, once every thread has finished reading the buffer the group pass used, group_done(
// freed columns) runs (the caller may rotate the next unit into it).  Returns the iterations
// used, or -1 after a timeout.  fT / fC: the CTA's token and channel factor arrays.
template <int KB, int VB, class WaitA, class GroupDone>
__device__ __forceinline__ int quantize_unit_tc(bool is_v, uint32_t tmem_base, uint32_t bufB, uint32_t bufA,
                                                uint8_t* __restrict__ rec, const QuantizeParams& p, float* fT,
                                                float* fC, float4* xbuf, float4* qpair, WaitA wait_a,
                                                GroupDone group_done) {
  constexpr RecordLayout RL = record_layout(128, KB, VB);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lg = warp & 3, hf = warp >> 2;
  const int line = 32 * lg + lane;
  // token factors start at 1/sqrt(d): the values in TMEM are Z.H without the rotation's scale
  if (tid < 128) fT[tid] = kInvSqrt128; else fC[tid - 128] = 1.0f;
  __syncthreads();
  const uint32_t lanes = ((uint32_t)(32 * lg) << 16) + 64 * hf;
  const uint32_t tA = tmem_base + bufA + lanes;  // lines = tokens
  const uint32_t tB = tmem_base + bufB + lanes;  // lines = channels

  // ---- variance normalisation: channel-std step (lines of B), then token-std step (lines of A)
  int used = 0;
  for (int it = 0; it < p.iters; ++it) {
    bool moved = std_step(tB, fT, fC, xbuf, line, hf, p.eps, p.tol_lo, p.tol_hi);
    if (!wait_a()) return -1;
    moved |= std_step(tA, fC, fT, xbuf, line, hf, p.eps, p.tol_lo, p.tol_hi);
    ++used;
    if (p.tol_hi > 0.0f && !__syncthreads_or(moved ? 1 : 0)) break;
  }
  if (!wait_a()) return -1;

  // ---- group extremes, one group per line: K groups are channels (lines of B, over tokens),
  // V groups are tokens (lines of A, over channels).  N = x fL fC with positive factors and
  // monotonic rounding, so the extremes of N are those of x f_other times the group's factor.
  constexpr int QMAXK = (1 << KB) - 1, QMAXV = (1 << VB) - 1;
  {
    const float* fo = is_v ? fC : fT;  // factors of the columns of the group's line
    const float4* f4 = reinterpret_cast<const float4*>(fo + 64 * hf);
    uint32_t r[64];
    load_line(is_v ? tA : tB, r);
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float4 f = f4[k];
      const float2 y0 = mul2(make_float2(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1])),
                             make_float2(f.x, f.y));
      const float2 y1 = mul2(make_float2(__uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3])),
                             make_float2(f.z, f.w));
      mn = fmin3(fmin3(mn, y0.x, y0.y), y1.x, y1.y);
      mx = fmax3(fmax3(mx, y0.x, y0.y), y1.x, y1.y);
    }
    xbuf[tid] = make_float4(mn, mx, 0.0f, 0.0f);
    __syncthreads();
    const float4 o = xbuf[tid ^ 128];
    mn = fminf(mn, o.x);
    mx = fmaxf(mx, o.y);
    const float fg = (is_v ? fT : fC)[line];  // the group's own factor
    const float m = mn * fg, M = mx * fg;
    const float s = fmaxf(__fdiv_rn(__fsub_rn(M, m), (float)(is_v ? QMAXV : QMAXK)), 1e-8f);
    if (hf == 0) reinterpret_cast<float2*>(qpair)[line] = make_float2(m, __frcp_rn(s));
    if (rec == nullptr) {
      // page id outside the pool (flagged): computed, not stored
    } else if (hf == 0) {
      // folded metadata: K s' = s c, z' = m c with c = 1 / fC (fp16); V s' = s r, z' = m r with
      // r = 1 / (sqrt(d) fT) (the token factors carry the rotation's 1/sqrt(d))
      const float fold = is_v ? fg * 11.313708498984761f : fg;
      __half* scale_out = reinterpret_cast<__half*>(rec + (is_v ? RL.vscale : RL.kscale));
      __half* zero_out = reinterpret_cast<__half*>(rec + (is_v ? RL.vzero : RL.kzero));
      scale_out[line] = __float2half_rn(__fdiv_rn(s, fold));
      zero_out[line] = __float2half_rn(__fdiv_rn(m, fold));
    } else {
      // the other axis' factor record: K token factor r = 1 / (sqrt(d) fT), V channel factor
      // c = 1 / fC
      __half* fac_out = reinterpret_cast<__half*>(rec + (is_v ? RL.vfactor : RL.kfactor));
      fac_out[line] = __float2half_rn(is_v ? __frcp_rn(fC[line]) : __fdiv_rn(kInvSqrt128, fT[line]));
    }
  }
  // group parameters visible ((m, 1/s) stored as float2 per group); every thread is done with
  // the group pass' TMEM buffer
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  group_done(is_v ? bufA : bufB);

  // ---- codes in the 16x256b layout: K from A (rows tokens, columns = channel groups), V from B
  // (rows channels, columns = token groups)
  {
    const int g = lane >> 2;
    float x[4][16];
    const uint32_t col = tmem_base + (is_v ? bufB : bufA) + 64 * hf;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t r[32];
      tmem_ld_16x256b_x8(col + ((uint32_t)(32 * lg + 16 * half) << 16), r);
      tmem_wait_ld();
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        x[2 * half][2 * u] = __uint_as_float(r[4 * u]);
        x[2 * half][2 * u + 1] = __uint_as_float(r[4 * u + 1]);
        x[2 * half + 1][2 * u] = __uint_as_float(r[4 * u + 2]);
        x[2 * half + 1][2 * u + 1] = __uint_as_float(r[4 * u + 3]);
      }
    }
    const float* frow = is_v ? fC : fT;  // factors of the rows (L axis)
    const float* fcol = is_v ? fT : fC;  // factors of the columns (the groups)
    float fl[4];
#pragma unroll
    for (int l = 0; l < 4; ++l) fl[l] = frow[32 * lg + g + 8 * l];
    // (m, 1/s) of groups c and c + 1 as one float4
    const float4* q4 = reinterpret_cast<const float4*>(qpair);
    if (rec == nullptr) {
    } else if (is_v) {
      codes_and_pack<true, KB, VB>(x, fl, fcol, q4, rec);
    } else {
      codes_and_pack<false, KB, VB>(x, fl, fcol, q4, rec);
    }
  }
  return used;
}

}  // namespace tc

template <int KB, int VB>
__global__ void __launch_bounds__(tc::kThreads, 2) quantize_tc_kernel(QuantizeParams p, int units) {
  extern __shared__ __align__(1024) uint8_t smem_tc[];
  using namespace tc;
  const uint32_t sbase = smem_u32(smem_tc);
  int* list = reinterpret_cast<int*>(smem_tc + kListOff);
  const __half** srcs = reinterpret_cast<const __half**>(smem_tc + kIoOff);
  uint8_t** recs = reinterpret_cast<uint8_t**>(smem_tc + kIoOff + kListCap * 8);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem_tc + kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_tc + kBarOff + 16);
  int* count = reinterpret_cast<int*>(smem_tc + kBarOff + 24);
  float* fT = reinterpret_cast<float*>(smem_tc + kFOff);
  float* fC = fT + 128;
  float4* xbuf = reinterpret_cast<float4*>(smem_tc + kXOff);
  float4* qpair = reinterpret_cast<float4*>(smem_tc + kQOff);
  const int tid = threadIdx.x, warp = tid >> 5;

  // ---- this CTA's units ----
  // Tile mode: units blockIdx.x + k gridDim.x, in that order, so that the first tile can be
  // requested before anything else; a unit whose page id is outside the pool is flagged and
  // computed without writing its record (rec = null).  Append mode: every token is written
  // first, and only the tiles that seal are listed; each warp takes every 8th of the CTA's units
  // so that the dependent loads of different units (length, then token) overlap.
  grid_dependency_wait();    // inputs, lengths and partial tiles may come from the previous kernel
  grid_launch_dependents();  // a dependent kernel still waits for this grid to complete
  const int64_t tstride = p.append ? (int64_t)p.d0 : p.tok_stride;  // token stride of every tile
  const int lane = tid & 31;
  constexpr int kWarps = kThreads / 32;
  int n_my;
  if (!p.append) {
    n_my = blockIdx.x < units ? min((units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1, kListCap) : 0;
    if (n_my == 0) return;
    {
      const int u = blockIdx.x;
      const int h = (u >> 1) % p.num_kv_heads, t = (u >> 1) / p.num_kv_heads;
      load_tile(sbase + kZOff,
                ((u & 1) ? p.v : p.k) + (int64_t)t * kTile * p.tok_stride + (int64_t)h * p.head_stride,
                tstride, p.d0);
      cp_async_commit();
    }
    for (int k = tid; k < n_my; k += kThreads) {
      const int u = blockIdx.x + k * gridDim.x;
      const __half* src;
      int64_t ts;
      uint8_t* rec;
      if (!tc::unit_io(p, u, src, ts, rec)) {
        flag_error(p.status, KVARN_DEV_BAD_PAGE_ID);
        rec = nullptr;
      }
      list[k] = u;
      srcs[k] = src;
      recs[k] = rec;
    }
    __syncthreads();
  } else {
    if (tid == 0) *count = 0;
    __syncthreads();
    for (int u = blockIdx.x + gridDim.x * warp; u < units; u += gridDim.x * kWarps) {
      const int h = (u >> 1) % p.num_kv_heads, b = (u >> 1) / p.num_kv_heads;
      const bool is_v = (u & 1) != 0;
      // the new token's 16-byte chunk of this lane (d0 <= 128 here) is read before the length,
      // so that the two loads are in flight together
      const __half* nw = (is_v ? p.v_new : p.k_new) + ((int64_t)b * p.num_kv_heads + h) * p.d0;
      const int c = lane * 8;
      const uint4 tok = c < p.d0 ? *reinterpret_cast<const uint4*>(nw + c) : make_uint4(0u, 0u, 0u, 0u);
      const int len = p.seq_lens[b];
      if (len < 0 || len >= p.max_pages * kTile) {
        if (lane == 0 && !is_v && h == 0) flag_error(p.status, KVARN_DEV_SEQ_TOO_LONG);
        continue;
      }
      __half* part = (is_v ? p.partial_v : p.partial_k) + ((int64_t)b * p.num_kv_heads + h) * kTile * p.d0;
      if (c < p.d0) *reinterpret_cast<uint4*>(part + (len % kTile) * p.d0 + c) = tok;
      if (lane == 0 && !is_v && h == 0 && p.seq_lens_out != nullptr) p.seq_lens_out[b] = len + 1;
      if (len % kTile != kTile - 1) continue;
      const __half* src;
      int64_t ts;
      uint8_t* rec;
      if (!tc::unit_io(p, u, src, ts, rec)) {  // page id outside the pool: skip the unit
        if (lane == 0) flag_error(p.status, KVARN_DEV_BAD_PAGE_ID);
        continue;
      }
      if (lane == 0) {
        const int n = atomicAdd(count, 1);
        if (n < kListCap) {  // the grid is sized so that n stays below kListCap
          list[n] = u;
          srcs[n] = src;
          recs[n] = rec;
        }
      }
    }
    __threadfence_block();
    __syncthreads();
    n_my = min(*count, kListCap);
    if (n_my == 0) return;
  }

  // ---- set-up: H_128 in shared memory, the TMEM accumulators, one mbarrier ----
  for (int q = tid; q < 128 * 16; q += kThreads) {
    const int n = q >> 4, c8 = q & 15;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k0 = c8 * 8 + 2 * e;
      const uint32_t lo = (__popc(n & k0) & 1) ? 0xBC00u : 0x3C00u;
      const uint32_t hi = (__popc(n & (k0 + 1)) & 1) ? 0xBC00u : 0x3C00u;
      w[e] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(smem_tc + kHOff + canon(n, c8 * 8)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "n"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    mbar_init(&mbar[0], 1);  // rotation B of a unit done
    mbar_init(&mbar[1], 1);  // rotation A of a unit done
    fence_mbar_init();
  }
  if (p.append) {  // tile mode requested the first tile at the start
    load_tile(sbase + kZOff, srcs[0], tstride, p.d0);
    cp_async_commit();
  }
  if (n_my > 1) load_tile(sbase + kZOff + kOpBytes, srcs[1], tstride, p.d0);
  cp_async_commit();
  cp_async_wait<1>();
  fence_proxy_async_smem();  // H and tile 0 written by the generic proxy, read by the MMA
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // One rotation of the tile in Z buffer zb into TMEM columns `cols`: B = H.Z^T (lanes =
  // channels) or A = Z.H (lanes = tokens); completes on mbar[0] (B) or mbar[1] (A).
  auto issue_rotation = [&](int zb, uint32_t cols, bool orient_b) {
    if (tid == 0) {
      const uint32_t z = sbase + kZOff + zb * kOpBytes, hm = sbase + kHOff;
      const uint32_t a = orient_b ? hm : z, bb = orient_b ? z : hm;
      const uint32_t d = tmem_base + cols;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t da = smem_desc(a + kk * 2 * kLbo), db = smem_desc(bb + kk * 2 * kLbo);
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(da), "l"(db), "r"(kIdesc), "r"((uint32_t)kk));
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                       smem_u32(&mbar[orient_b ? 0 : 1]))
                   : "memory");
    }
  };
  // Unit i's rotations sit in TMEM columns (bufB, bufA).  The next unit's B is issued into the
  // buffer unit i's group pass has finished with, its A into the buffer of unit i's codes pass
  // once that pass is done: the next unit's rotations overlap this unit's codes and its own
  // first channel step.
  uint32_t bufB = 128, bufA = 0;
  issue_rotation(0, bufB, true);
  issue_rotation(0, bufA, false);
  int issued = 1;  // rotation pairs issued (for draining after a timeout)
  bool ok = true;
  for (int i = 0; i < n_my; ++i) {
    // one decision for the whole CTA, so that no thread leaves while others wait at a barrier
    ok = __syncthreads_and(mbar_wait(&mbar[0], i & 1) ? 1 : 0) != 0;
    if (!ok) break;
    tc_fence_after();
    bool a_ready = false;
    auto wait_a = [&]() -> bool {
      if (a_ready) return true;
      a_ready = true;
      const bool ok_a = __syncthreads_and(mbar_wait(&mbar[1], i & 1) ? 1 : 0) != 0;
      tc_fence_after();
      if (!ok_a) return false;
      // both rotations of unit i are done, its Z buffer is free: fetch list[i + 2] into it
      if (i + 2 < n_my) load_tile(sbase + kZOff + (i & 1) * kOpBytes, srcs[i + 2], tstride, p.d0);
      cp_async_commit();
      return true;
    };
    uint32_t next_b = bufB;
    auto group_done = [&](uint32_t freed) {
      next_b = freed;
      if (i + 1 < n_my) issue_rotation((i + 1) & 1, freed, true);
    };
    uint8_t* rec = recs[i];
    const bool is_v = (list[i] & 1) != 0;
    const int used = tc::quantize_unit_tc<KB, VB>(
        is_v, tmem_base, bufB, bufA, rec, p, fT, fC, xbuf, qpair,
        [&]() -> bool {
          if (!wait_a()) return false;
          cp_async_wait<1>();          // the tile of list[i + 1] has landed (list[i + 2] may not)
          fence_proxy_async_smem();    // visible to the tensor core after the pass' barrier
          return true;
        },
        group_done);
    if (used < 0) {
      ok = false;
      break;
    }
    if (p.iters_out != nullptr && !p.append && tid == 0) p.iters_out[list[i]] = used;
    const uint32_t codes_buf = is_v ? bufB : bufA;  // free once every thread is past the codes
    if (i + 1 < n_my) {
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      issue_rotation((i + 1) & 1, codes_buf, false);
      ++issued;
    }
    bufB = next_b;
    bufA = codes_buf;
  }
  if (!ok && tid == 0) flag_error(p.status, KVARN_DEV_WAIT_TIMEOUT);
  // ---- tear-down: no MMA may still write TMEM when it is released ----
  cp_async_wait<0>();
  if (!ok && tid == 0) {  // the last rotations issued (bounded waits)
    mbar_wait(&mbar[0], (issued - 1) & 1);
    mbar_wait(&mbar[1], (issued - 1) & 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "n"(kTmemCols));
  }
}

template <int KB, int VB>
static int launch_quantize_tc(const QuantizeParams& p, int units2, cudaStream_t stream) {
  static PerDeviceOnce smem_once;  // the attribute is set once per device
  const void* fn = reinterpret_cast<const void*>(quantize_tc_kernel<KB, VB>);
  if (const int st = set_smem_limit(smem_once, fn, tc::kSmemBytes); st != KVARN_OK) return st;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int grid = 2 * sms;
  grid = max(grid, (units2 + tc::kListCap - 1) / tc::kListCap);
  grid = min(grid, units2);
  return launch_pdl(quantize_tc_kernel<KB, VB>, dim3(grid), dim3(tc::kThreads), tc::kSmemBytes, stream,
                    p, units2);
}

template <int KB, int VB>
static int launch_quantize_bits(int d, const QuantizeParams& p, int units, cudaStream_t stream) {
  switch (d) {
    case 64: return launch_quantize<64, KB, VB>(p, units, stream);
    case 128: return launch_quantize_tc<KB, VB>(p, units * 2, stream);
    case 256: return launch_quantize<256, KB, VB>(p, units, stream);
    default: return KVARN_ERR_UNSUPPORTED;
  }
}

int launch_quantize_any(int d, int kb, int vb, const QuantizeParams& p, int units, cudaStream_t stream) {
  if (units <= 0) return KVARN_OK;
  if (kb == 4 && vb == 2) return launch_quantize_bits<4, 2>(d, p, units, stream);
  if (kb == 4 && vb == 4) return launch_quantize_bits<4, 4>(d, p, units, stream);
  if (kb == 2 && vb == 2) return launch_quantize_bits<2, 2>(d, p, units, stream);
  if (kb == 8 && vb == 4) return launch_quantize_bits<8, 4>(d, p, units, stream);
  return KVARN_ERR_UNSUPPORTED;
}

}  // namespace kvarn
