// KVarN page record -> fp16 K/V in the original basis (sm_103a).
//
// K~[t][j] = r[t] (code s'[j] + z'[j]),  V~[t][j] = c[j] (code s'[t] + z'[t])  (rotated basis),
// then each token row is multiplied by H_d / sqrt(d) (the rotation is its own inverse) and the
// padded channels are dropped [hotdry §非对称量化与尺度折叠: scales multiplied back at read;
// vatt §四個步驟: orthonormal rotation, invertible].  Not on the decode path: used for
// checking and for consumers that want plain fp16 K/V back.
#include "common.cuh"
#include "params.cuh"

namespace kvarn {


template <int D>
struct DequantShape {
  static constexpr int kLd = D + 4;
  static constexpr int kSmemBytes = kTile * kLd * 4;
};

// Code of element (rho, h, p) of fragment (o, i) for lane `lane` (layout in kvarn.h): a 4-bit
// word holds one fragment, a 2-bit word the fragments of token blocks o and o ^ 1, an 8-bit
// fragment two words.
template <int D, int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t* w, int o, int i, int lane, int rho, int h,
                                            int pp) {
  int word, sh;
  if constexpr (BITS == 4) {
    word = ((o * (D / 64) + i / 4) * 32 + lane) * 4 + (i & 3);
    sh = 4 * (h + 2 * rho + 4 * pp);
  } else if constexpr (BITS == 8) {
    word = ((o * (D / 32) + i / 2) * 32 + lane) * 4 + 2 * (i & 1) + h;
    sh = 8 * (rho + 2 * pp);
  } else {
    static_assert(BITS == 2, "2-, 4- or 8-bit codes");
    word = (((o >> 1) * (D / 64) + i / 4) * 32 + lane) * 4 + (i & 3);
    sh = 2 * (2 * (o & 1) + h + 4 * rho + 8 * pp);
  }
  return (w[word] >> sh) & ((1u << BITS) - 1u);
}

// grid.x = pages * Hkv * 2, block = 128 threads (one token row each while decoding codes).
// ERR: instead of storing fp16, compare the dequantised tile (fp32) with the fp16 tile it was
// quantised from and write the unit's four error statistics (kvarn_quantization_error).
template <int D, int KB, int VB, bool ERR>
__global__ void __launch_bounds__(128) dequantize_kernel(DequantParams p) {
  constexpr RecordLayout RL = record_layout(D, KB, VB);
  constexpr int LD = DequantShape<D>::kLd;
  extern __shared__ __align__(16) float smem_x[];
  const int unit = blockIdx.x >> 1;
  const bool is_v = (blockIdx.x & 1) != 0;
  const int h = unit % p.num_kv_heads;
  const int pi = unit / p.num_kv_heads;
  int64_t page = p.page_ids[pi];
  if (page < 0 || page >= p.num_pool_pages) {
    if (threadIdx.x == 0) flag_error(p.status, KVARN_DEV_BAD_PAGE_ID);
    page = 0;
  }
  const uint8_t* rec = p.pool + (page * p.num_kv_heads + h) * (int64_t)RL.bytes;
  const int t = threadIdx.x;
  const int g_t = t & 7, rho_or_h = (t & 15) >> 3;

  if (!is_v) {
    const uint32_t* kw = reinterpret_cast<const uint32_t*>(rec + RL.kcodes);
    const __half* ks = reinterpret_cast<const __half*>(rec + RL.kscale);
    const __half* kz = reinterpret_cast<const __half*>(rec + RL.kzero);
    const float r = __half2float(reinterpret_cast<const __half*>(rec + RL.kfactor)[t]);
    const int mi = t >> 4, rho = rho_or_h;
    for (int kk = 0; kk < D / 16; ++kk) {
      for (int tq = 0; tq < 4; ++tq) {
        const int lane = 4 * g_t + tq;
        for (int hh = 0; hh < 2; ++hh)
          for (int pp = 0; pp < 2; ++pp) {
            const int j = 16 * kk + 8 * hh + 2 * tq + pp;
            const uint32_t code = code_at<D, KB>(kw, mi, kk, lane, rho, hh, pp);
            smem_x[t * LD + j] =
                r * fmaf((float)code, __half2float(ks[j]), __half2float(kz[j]));
          }
      }
    }
  } else {
    const uint32_t* vw = reinterpret_cast<const uint32_t*>(rec + RL.vcodes);
    const float s = __half2float(reinterpret_cast<const __half*>(rec + RL.vscale)[t]);
    const float z = __half2float(reinterpret_cast<const __half*>(rec + RL.vzero)[t]);
    const __half* vc = reinterpret_cast<const __half*>(rec + RL.vfactor);
    const int ks = t >> 4, hh = rho_or_h;
    const int tq = (t & 7) >> 1, pp = t & 1;
    for (int mc = 0; mc < D / 16; ++mc)
      for (int g = 0; g < 8; ++g) {
        const int lane = 4 * g + tq;
        for (int rho = 0; rho < 2; ++rho) {
          const int j = 16 * mc + g + 8 * rho;
          const uint32_t code = code_at<D, VB>(vw, ks, mc, lane, rho, hh, pp);
          smem_x[t * LD + j] = __half2float(vc[j]) * fmaf((float)code, s, z);
        }
      }
  }
  __syncthreads();
  // inverse rotation along channels: log2(D) butterfly stages over the whole tile
  for (int hstep = 1; hstep < D; hstep <<= 1) {
    for (int idx = threadIdx.x; idx < kTile * D / 2; idx += blockDim.x) {
      const int row = idx / (D / 2), k = idx - row * (D / 2);
      const int i0 = (k / hstep) * 2 * hstep + (k % hstep);
      const float a = smem_x[row * LD + i0], b = smem_x[row * LD + i0 + hstep];
      smem_x[row * LD + i0] = a + b;
      smem_x[row * LD + i0 + hstep] = a - b;
    }
    __syncthreads();
  }
  const float isd = D == 64 ? 0.125f : (D == 128 ? 0.08838834764831845f : 0.0625f);
  if constexpr (!ERR) {
    __half* dst = (is_v ? p.v_out : p.k_out) + ((int64_t)pi * p.num_kv_heads + h) * kTile * p.d0;
    for (int idx = threadIdx.x; idx < kTile * p.d0; idx += blockDim.x) {
      const int row = idx / p.d0, j = idx - row * p.d0;
      dst[idx] = __float2half_rn(smem_x[row * LD + j] * isd);
    }
  } else {
    // sum (x - x^)^2, sum x^2, max |x - x^|, max |x| over the 128 x d0 values of the unit
    const __half* src = (is_v ? p.v_src : p.k_src) + (int64_t)pi * kTile * p.tok_stride +
                        (int64_t)h * p.head_stride;
    float se = 0.0f, sx = 0.0f, me = 0.0f, mx = 0.0f;
    for (int idx = threadIdx.x; idx < kTile * p.d0; idx += blockDim.x) {
      const int row = idx / p.d0, j = idx - row * p.d0;
      const float x = __half2float(src[row * p.tok_stride + j]);
      const float e = x - smem_x[row * LD + j] * isd;
      se = fmaf(e, e, se);
      sx = fmaf(x, x, sx);
      me = fmaxf(me, fabsf(e));
      mx = fmaxf(mx, fabsf(x));
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
      se += __shfl_xor_sync(0xffffffffu, se, m);
      sx += __shfl_xor_sync(0xffffffffu, sx, m);
      me = fmaxf(me, __shfl_xor_sync(0xffffffffu, me, m));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    }
    __syncthreads();  // smem_x is read by every thread above; reuse its head for the warps' sums
    float4* part = reinterpret_cast<float4*>(smem_x);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = make_float4(se, sx, me, mx);
    __syncthreads();
    if (threadIdx.x == 0) {
      float4 a = part[0];
#pragma unroll
      for (int w = 1; w < 4; ++w) {
        const float4 b = part[w];
        a = make_float4(a.x + b.x, a.y + b.y, fmaxf(a.z, b.z), fmaxf(a.w, b.w));
      }
      reinterpret_cast<float4*>(p.err_out)[((int64_t)pi * p.num_kv_heads + h) * 2 + (is_v ? 1 : 0)] = a;
    }
  }
}

template <int D, int KB, int VB>
static int launch_dequant_t(const DequantParams& p, int num_pages, cudaStream_t stream) {
  constexpr int kSmem = DequantShape<D>::kSmemBytes;
  if (p.err_out == nullptr) {
    static PerDeviceOnce smem_once;  // the attribute is set once per device
    const void* fn = reinterpret_cast<const void*>(dequantize_kernel<D, KB, VB, false>);
    if (const int st = set_smem_limit(smem_once, fn, kSmem); st != KVARN_OK) return st;
    dequantize_kernel<D, KB, VB, false><<<num_pages * p.num_kv_heads * 2, 128, kSmem, stream>>>(p);
  } else {
    static PerDeviceOnce smem_once;
    const void* fn = reinterpret_cast<const void*>(dequantize_kernel<D, KB, VB, true>);
    if (const int st = set_smem_limit(smem_once, fn, kSmem); st != KVARN_OK) return st;
    dequantize_kernel<D, KB, VB, true><<<num_pages * p.num_kv_heads * 2, 128, kSmem, stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA;
}

template <int KB, int VB>
static int launch_dequant_bits(int d, const DequantParams& p, int num_pages, cudaStream_t stream) {
  switch (d) {
    case 64: return launch_dequant_t<64, KB, VB>(p, num_pages, stream);
    case 128: return launch_dequant_t<128, KB, VB>(p, num_pages, stream);
    case 256: return launch_dequant_t<256, KB, VB>(p, num_pages, stream);
    default: return KVARN_ERR_UNSUPPORTED;
  }
}

int launch_dequant_any(int d, int kb, int vb, const DequantParams& p, int num_pages, cudaStream_t stream) {
  if (num_pages <= 0) return KVARN_OK;
  if (kb == 4 && vb == 2) return launch_dequant_bits<4, 2>(d, p, num_pages, stream);
  if (kb == 4 && vb == 4) return launch_dequant_bits<4, 4>(d, p, num_pages, stream);
  if (kb == 2 && vb == 2) return launch_dequant_bits<2, 2>(d, p, num_pages, stream);
  if (kb == 8 && vb == 4) return launch_dequant_bits<8, 4>(d, p, num_pages, stream);
  return KVARN_ERR_UNSUPPORTED;
}

}  // namespace kvarn
