// KVarN paged decode for GQA groups of 8 on the fifth-generation tensor cores (sm_103a):
// head_dim 128, K 4-bit per channel, V 2-bit per token.
//
// Same arithmetic as decode_kernel (rotated basis, codes as fp16 subnormals, fp16 hi + lo
// operands, log2-domain online softmax; [vatt §四個步驟: the rotation keeps q.k unchanged;
// hotdry §非对称量化与尺度折叠: the folded scales are multiplied back at read time]), with the
// contractions on tcgen05.mma instead of mma.sync.  Per page (one 128-token tile of one kv head)
// and the 8 query heads of that kv head:
//   QK:  D_QK[t][n] = sum_j A_K[t][j] B_QK[j][n]   M = 128 tokens, N = 16, K = 128 channels
//        A_K = codes (fp16 subnormals) in tensor memory, B_QK = q~ . s'_K as fp16 hi (n = head)
//        and lo (n = 8 + head) in shared memory;
//        logit = r_t (2^20 (D_QK[t][h] + D_QK[t][8 + h]) + q~ . z'_K)
//   PV:  D_PV[c][n] = sum_t A_V[c][t] B_PV[t][n] + sum_t 2^-24 B_PVZ[t][n]   M = 128 channels
//        A_V = codes^T in tensor memory, B_PV = p . s'_V hi / lo, B_PVZ = p . z'_V hi / lo
//        against a constant A of 2^-24 (the zero-point term of every channel);
//        o~[h][c] += c_c 2^24 (D_PV[c][h] + D_PV[c][8 + h])
// A persistent CTA per SM walks a balanced range of pages (decode_util.cuh) with six roles:
//   warps 0-3    K codes -> tensor memory (tcgen05.st, one AND per two codes), B_QK and
//                q~ . z'_K of every page; the row's rotated queries at each new row;
//   warp 12      QK MMAs, lanes 0-1 each issuing four of the eight channel steps into an
//                accumulator of its own (one lane issues an MMA about every 120 cycles; two
//                lanes of a warp issue two in about 160);
//   warps 4-7    softmax (thread = token), B_PV, the page's rescale factors and the warp sums of
//                p . z'_V; the row's (m, l) at its end;
//   warp 13      PV MMAs, lanes 0-1 each taking four token blocks into an accumulator;
//   warps 8-11   V codes -> tensor memory once QK has read the K codes there, and the output
//                update (thread = channel); the row's o~ at its end;
//   warp 14      page records into a ring of shared-memory slots (1-D bulk copies).
// Tensor memory holds four stages of 128 columns: the codes (K, then V: 64 columns) and two
// accumulators of 16 (QK, then PV).  Every hand-off is an mbarrier, every wait is bounded.
#include "common.cuh"
#include "decode_util.cuh"
#include "params.cuh"

namespace kvarn {
namespace dtc {

constexpr int D = 128;
constexpr RecordLayout kRL = record_layout(D, 4, 2);
constexpr int kRec = kRL.bytes;
constexpr int kSlots = 12;   // page records in flight per CTA
constexpr int kStages = 4;   // operand stages in tensor memory and shared memory
constexpr int kThreads = 480;
constexpr int kQkWarp = 12, kPvWarp = 13, kLoadWarp = 14;
constexpr int kCvBar = 1, kSmBar = 2;  // named barriers of the K-convert and the softmax warps

// shared memory
constexpr int kBOff = kSlots * kRec;                 // per stage: B_QK, B_PV (4096 bytes each)
constexpr int kBTile = 4096;
constexpr int kQOff = kBOff + kStages * 2 * kBTile;  // q~ of the row: fp16 hi [8][128], lo, fp32
constexpr int kQzOff = kQOff + 2 * 2048 + 4096;      // q~ . z'_K per stage and warp [4][4][8]
constexpr int kMxOff = kQzOff + kStages * 4 * 32;    // page maxima per warp [2][4][8]
constexpr int kAzOff = kMxOff + 2 * 4 * 32;          // per stage: rescale [8], p . z'_V per warp [4][8]
constexpr int kLrOff = kAzOff + kStages * 40 * 4;    // row sums per warp [4][8]
constexpr int kBarOff = kLrOff + 4 * 32;
constexpr int kNumBars = 2 * kSlots + 6 * kStages;
constexpr int kTslotOff = kBarOff + kNumBars * 8;
constexpr int kSmemBytes = kTslotOff + 16;
static_assert(kSmemBytes <= 232448 - 1024, "fits one CTA per SM");
static_assert(kRec % 16 == 0 && kBOff % 1024 == 0, "bulk copies and descriptors stay aligned");

// tensor memory: stage s at 128 s: codes [0, 64), accumulators [64, 96) (16 columns each)
constexpr uint32_t kColStage = 128, kColD = 64;
constexpr int kTmemCols = 512;

// kind::f16 instruction descriptors: f32 accumulate, f16 A and B, M = 128, N = 16; B K-major
// (QK) or MN-major (PV).  Shared-memory B tiles (16 x 16, no swizzle): K-major core matrices at
// LBO 128 along K, SBO 256 along N; MN-major at LBO 256 along K, SBO 128 along N.
constexpr uint32_t kIdescQK = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = kIdescQK | (1u << 16);

constexpr float kAccQK = kTwo24 / 16.0f;  // QK sum: codes 2^-24 (x16 for channels 8..15), q lifted x16
constexpr float kAccPV = kTwo24;          // PV sum: codes 2^-24 times the powers of 4 in B_PV

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         ((uint64_t)1 << 46);
}

__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void st_16x256b_x8(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void ld_32x32b_x16(uint32_t taddr, float (&f)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(r[i]);
}

// Barrier of the 128 threads of one role group; returns whether any of them passed `flag`.
__device__ __forceinline__ bool group_any(int id, bool flag) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, 128, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)flag), "r"(id)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait_sleep(bar, parity));
}

// The two accumulators of a stage summed per column: s[n] = D[n] + D[16 + n], n < 16.
__device__ __forceinline__ void ld_sum2(uint32_t taddr, float (&sum)[16]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int n = 0; n < 16; ++n) sum[n] = __uint_as_float(r[n]) + __uint_as_float(r[16 + n]);
}

}  // namespace dtc

using namespace dtc;

__global__ void __launch_bounds__(dtc::kThreads, 1) decode_tc_kernel(DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ Walk ws;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* rec_full = reinterpret_cast<uint64_t*>(sm + kBarOff);
  uint64_t* rec_empty = rec_full + kSlots;
  uint64_t* ops_k = rec_empty + kSlots;  // K codes, B_QK and q~ . z'_K of a stage written
  uint64_t* qk_full = ops_k + kStages;   // QK of a stage done (four lanes commit)
  uint64_t* ops_v = qk_full + kStages;   // V codes of a stage written
  uint64_t* p_full = ops_v + kStages;    // B_PV, rescale and p . z'_V of a stage written
  uint64_t* pv_done = p_full + kStages;  // PV of a stage done: the codes columns are free
  uint64_t* pv_read = pv_done + kStages; // the stage's PV sums read: its accumulators are free
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kTslotOff);

  grid_dependency_wait();  // lengths and pages may come from the previous kernel
  if (warp == kLoadWarp) {
    const Walk w = range_walk(p, blockIdx.x, lane);
    if (lane == 0) ws = w;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&rec_full[i], 1);
      mbar_init(&rec_empty[i], 4);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ops_k[s], 4);
      mbar_init(&qk_full[s], 2);
      mbar_init(&ops_v[s], 4);
      mbar_init(&p_full[s], 4);
      mbar_init(&pv_done[s], 2);
      mbar_init(&pv_read[s], 4);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  int64_t total = 0;  // pages of this CTA's range
  for (Walk w = ws; w.left > 0; w.next(p)) total += w.count();
  if (total <= 0) {
    grid_launch_dependents();
    return;
  }
  if (warp == kPvWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "n"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  volatile int* abort_v = &abort_flag;
  auto fail = [&]() {
    *abort_v = 1;
    flag_error(p.status, KVARN_DEV_WAIT_TIMEOUT);
  };
  const Walk w0 = ws;
  uint8_t* recs = sm;
  auto stage_tmem = [&](int s) { return tmem + kColStage * (uint32_t)s; };
  auto b_qk = [&](int s) { return sm + kBOff + 2 * s * kBTile; };
  auto b_pv = [&](int s) { return sm + kBOff + (2 * s + 1) * kBTile; };
  float* qz_s = reinterpret_cast<float*>(sm + kQzOff);
  float* az_s = reinterpret_cast<float*>(sm + kAzOff);  // per stage: rescale [8], z sums [4][8]
  // partial row of head slot hh of the segment's (b, h, slot)
  auto part_row = [&](const Walk& w, int hh) {
    return p.part + (((int64_t)w.b * p.num_q_heads + w.h * 8 + hh) * p.max_splits + w.slot) * (D + 4);
  };

  if (warp == kLoadWarp) {
    // ---- page records -> shared-memory slots ----
    if (lane == 0) {
      int64_t g = 0;
      int r = 0;
      uint32_t rph = 0;
      for (Walk w = w0; w.left > 0 && *abort_v == 0; w.next(p)) {
        const int cnt = w.count();
        const int32_t* bt = p.block_table + (int64_t)w.b * p.max_pages + w.j;
        for (int i = 0; i < cnt; ++i, ++g) {
          if (!mbar_wait_sleep(&rec_empty[r], rph ^ 1u) || *abort_v != 0) {
            fail();
            break;
          }
          int64_t id = bt[i];
          if (id < 0 || id >= p.num_pool_pages) {
            flag_error(p.status, KVARN_DEV_BAD_PAGE_ID);
            id = 0;
          }
          fence_proxy_async_smem();
          mbar_expect_tx(&rec_full[r], kRec);
          bulk_copy_g2s(recs + r * kRec, p.pool + (id * p.num_kv_heads + w.h) * (int64_t)kRec, kRec, &rec_full[r]);
          if (++r == kSlots) {
            r = 0;
            rph ^= 1u;
          }
        }
      }
      // copies still in flight land before the CTA may leave
      for (int64_t k = g > kSlots ? g - kSlots : 0; k < g; ++k)
        mbar_wait_sleep(&rec_full[k % kSlots], (uint32_t)((k / kSlots) & 1));
    }
    __syncwarp();
  } else if (warp == kQkWarp || warp == kPvWarp) {
    // ---- MMA issue: lane i < 2 takes four of the eight K steps into accumulator i ----
    if (lane < 2) {
      const bool is_qk = warp == kQkWarp;
      uint64_t* last = nullptr;
      uint32_t last_par = 0;
      for (int64_t g = 0; g < total; ++g) {
        const int s = (int)(g & 3);
        const uint32_t par = (uint32_t)((g >> 2) & 1);
        // QK: the K codes written and the accumulators read (PV of page g - 4); PV: the V codes
        // and B_PV written
        const bool ok = is_qk ? (mbar_wait_sleep(&ops_k[s], par) && mbar_wait_sleep(&pv_read[s], par ^ 1u))
                              : (mbar_wait_sleep(&ops_v[s], par) && mbar_wait_sleep(&p_full[s], par));
        if (!__all_sync(0x3u, ok) || *abort_v != 0) {
          if (lane == 0) fail();
          break;
        }
        fence_after();
        const uint32_t st = stage_tmem(s);
        const uint32_t acc = st + kColD + 16 * lane;
        if (is_qk) {
          const uint32_t bq = smem_u32(b_qk(s));
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kk = 4 * lane + e;
            mma_ts(acc, st + 8 * kk, smem_desc(bq + 512 * kk, 128, 256), kIdescQK, e);
          }
          mma_commit(&qk_full[s]);
          last = &qk_full[s];
        } else {
          const uint32_t bp = smem_u32(b_pv(s));
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int o = 4 * lane + e;
            mma_ts(acc, st + 8 * o, smem_desc(bp + 512 * o, 256, 128), kIdescPV, e);
          }
          mma_commit(&pv_done[s]);
          last = &pv_done[s];
        }
        last_par = par;
      }
      if (last != nullptr) mbar_wait_sleep(last, last_par);  // this lane's MMAs have completed
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---- K convert: codes -> tensor memory, B_QK, q~ . z'_K ----
    const int t = threadIdx.x;          // 0..127
    const int q = warp;                 // tensor-memory lane quarter
    const int hd = t & 7, oc = t >> 3;  // B_QK: head hd, channel octet oc (8 heads side by side)
    const int kk = oc >> 1, kb = oc & 1;
    const int cbase = 16 * kk + 4 * kb;  // channels cbase + {0, 1, 8, 9, 2, 3, 10, 11}: K index 8kb..8kb+7
    __half* qh_s = reinterpret_cast<__half*>(sm + kQOff);
    __half* ql_s = qh_s + 8 * D;
    float* qf_s = reinterpret_cast<float*>(sm + kQOff + 4096);
    const float qsc = p.qscale * inv_sqrt_d<D>();
    int64_t g = 0;
    int r = 0;
    uint32_t rph = 0;
    bool bad = false;
    for (Walk w = w0; w.left > 0; w.next(p)) {
      // rotated queries of the row's 8 heads: two per warp, fp32 and fp16 hi + lo (x16 on
      // channels 0..7 of every 16, the factor their codes lack)
      if (group_any(kCvBar, bad || *abort_v != 0)) break;
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int hh = 2 * q + e2;
        const __half* src = p.q + ((int64_t)w.b * p.num_q_heads + w.h * 8 + hh) * p.d0;
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 4 * lane + e;
          v[e] = j < p.d0 ? __half2float(src[j]) : 0.0f;
        }
        warp_fwht<D>(v, lane);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 4 * lane + e;
          const float x = v[e] * qsc;
          const float xb = x * ((j & 15) < 8 ? 16.0f : 1.0f);
          const __half hi = __float2half_rn(xb);
          qf_s[hh * D + j] = x;
          qh_s[hh * D + j] = hi;
          ql_s[hh * D + j] = __float2half_rn(xb - __half2float(hi));
        }
      }
      group_any(kCvBar, false);
      __half2 qh[4], ql[4];
      float qf[8];
      {
        const int pj[4] = {cbase, cbase + 8, cbase + 2, cbase + 10};  // pair starts in K order
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          qh[i] = *reinterpret_cast<const __half2*>(qh_s + hd * D + pj[i]);
          ql[i] = *reinterpret_cast<const __half2*>(ql_s + hd * D + pj[i]);
          qf[2 * i] = qf_s[hd * D + pj[i]];
          qf[2 * i + 1] = qf_s[hd * D + pj[i] + 1];
        }
      }
      const int cnt = w.count();
      for (int i = 0; i < cnt; ++i, ++g) {
        const int s = (int)(g & 3);
        if (!wait_all(&rec_full[r], rph) || !wait_all(&pv_done[s], (uint32_t)((g >> 2) & 1) ^ 1u)) {
          bad = true;
          fail();
          break;
        }
        fence_after();
        const uint8_t* R = recs + r * kRec;
        const uint32_t st = stage_tmem(s);
        if (++r == kSlots) {
          r = 0;
          rph ^= 1u;
        }
        // K codes: token blocks 2q, 2q + 1 of this quarter; a word of fragment (o, i) is the
        // 16x256b block of lanes 16o.., columns 8i..8i+7, column 2tq + h holding channels
        // 16i + 8h + 2tq, +1 (x16 at h = 1)
        {
          const uint4* kc = reinterpret_cast<const uint4*>(R + kRL.kcodes);
#pragma unroll
          for (int oo = 0; oo < 2; ++oo)
#pragma unroll
            for (int kq = 0; kq < 2; ++kq) {
              const uint4 w4 = kc[((2 * q + oo) * 2 + kq) * 32 + lane];
              const uint32_t wsx[4] = {w4.x, w4.y, w4.z, w4.w};
              uint32_t rr[16];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const uint32_t x = wsx[e], y = x >> 8;
                rr[4 * e] = x & 0x000F000Fu;
                rr[4 * e + 1] = x & 0x00F000F0u;
                rr[4 * e + 2] = y & 0x000F000Fu;
                rr[4 * e + 3] = y & 0x00F000F0u;
              }
              st_16x256b_x4(st + ((uint32_t)(32 * q + 16 * oo) << 16) + 32 * kq, rr);
            }
        }
        // B_QK row pair (hi: n = hd, lo: n = 8 + hd) over K index 8kb..8kb+7 of tile kk, and
        // this warp's four octets of q~ . z'_K for head hd (lanes hd, hd + 8, hd + 16, hd + 24)
        {
          const uint2 sa = *reinterpret_cast<const uint2*>(R + kRL.kscale + 2 * cbase);
          const uint2 sb = *reinterpret_cast<const uint2*>(R + kRL.kscale + 2 * (cbase + 8));
          const uint2 za = *reinterpret_cast<const uint2*>(R + kRL.kzero + 2 * cbase);
          const uint2 zb = *reinterpret_cast<const uint2*>(R + kRL.kzero + 2 * (cbase + 8));
          const __half2 sv[4] = {u2h2(sa.x), u2h2(sb.x), u2h2(sa.y), u2h2(sb.y)};
          const __half2 zv[4] = {u2h2(za.x), u2h2(zb.x), u2h2(za.y), u2h2(zb.y)};
          uint32_t hi[4], lo[4];
          float2 qz2 = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int i2 = 0; i2 < 4; ++i2) {
            const __half2 hv = __hmul2(qh[i2], sv[i2]);
            hi[i2] = h2u(hv);
            lo[i2] = h2u(__hfma2(ql[i2], sv[i2], __hfma2(qh[i2], sv[i2], __hneg2(hv))));
            qz2 = fma2(make_float2(qf[2 * i2], qf[2 * i2 + 1]), __half22float2(zv[i2]), qz2);
          }
          uint8_t* bq = b_qk(s) + 512 * kk + 128 * kb + 16 * hd;
          *reinterpret_cast<uint4*>(bq) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(bq + 256) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          float qz = qz2.x + qz2.y;
          qz += __shfl_xor_sync(0xffffffffu, qz, 8);
          qz += __shfl_xor_sync(0xffffffffu, qz, 16);
          if (lane < 8) qz_s[(s * 4 + q) * 8 + hd] = qz;
        }
        wait_st();
        fence_proxy_async_smem();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ops_k[s]);
      }
    }
  } else if (warp < 8) {
    // ---- softmax (thread = token) ----
    const int u = threadIdx.x - 128;  // token 0..127
    const int q = warp - 4;           // tensor-memory lane quarter
    const int ob = u >> 4, hb = (u >> 3) & 1;
    const float cfac = 1.0f / (float)(1 << (2 * (2 * (ob & 1) + hb)));  // the code's power of 4
    const int kpos = 4 * ((u >> 1) & 3) + 2 * hb + (u & 1);              // K index in tile ob
    const int boff = 512 * ob + 256 * (kpos >> 3) + 16 * (kpos & 7);
    // after the butterfly below, lane l (l % 4 == 0) holds the warp's sum of head zhead
    const int zhead = 4 * ((lane >> 4) & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
    float* mx_s = reinterpret_cast<float*>(sm + kMxOff);
    float* lr_s = reinterpret_cast<float*>(sm + kLrOff);
    int64_t g = 0;
    int r = 0;
    uint32_t rph = 0;
    bool bad = false, stop = false;  // this thread's failed wait; the group's decision to stop
    float M[8], L[8];
    for (Walk w = w0; w.left > 0; w.next(p)) {
#pragma unroll
      for (int hh = 0; hh < 8; ++hh) {
        M[hh] = -INFINITY;
        L[hh] = 0.0f;
      }
      const int cnt = w.count();
      for (int i = 0; i < cnt; ++i, ++g) {
        const int s = (int)(g & 3);
        const uint32_t par = (uint32_t)((g >> 2) & 1);
        const bool ok = !bad && wait_all(&qk_full[s], par) && wait_all(&ops_k[s], par) && wait_all(&rec_full[r], rph);
        const uint8_t* R = recs + r * kRec;
        if (++r == kSlots) {
          r = 0;
          rph ^= 1u;
        }
        float lg[8];
        if (ok) {
          fence_after();
          float d[16];
          ld_sum2(stage_tmem(s) + kColD + ((uint32_t)(32 * q) << 16), d);
          const float rt = __half2float(reinterpret_cast<const __half*>(R + kRL.kfactor)[u]);
          float qz[8];
#pragma unroll
          for (int hh = 0; hh < 8; ++hh) {
            const float* z = qz_s + s * 32 + hh;
            qz[hh] = (z[0] + z[8]) + (z[16] + z[24]);
          }
#pragma unroll
          for (int hh = 0; hh < 8; ++hh) lg[hh] = rt * fmaf(d[hh] + d[8 + hh], kAccQK, qz[hh]);
#pragma unroll
          for (int hh = 0; hh < 8; ++hh) {
            const float m = warp_max(lg[hh]);
            if (lane == 0) mx_s[((g & 1) * 4 + q) * 8 + hh] = m;
          }
        } else if (!bad) {
          bad = true;
          fail();
        }
        stop = group_any(kSmBar, bad);
        if (stop) break;
        const float* mx = mx_s + (g & 1) * 32;
        const float svc = __half2float(reinterpret_cast<const __half*>(R + kRL.vscale)[u]) * cfac;
        const float zv = __half2float(reinterpret_cast<const __half*>(R + kRL.vzero)[u]);
        float al[8], zz[8];
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int hp = 0; hp < 4; ++hp) {
          float pr[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int hh = 2 * hp + e;
            const float pm = fmaxf(fmaxf(mx[hh], mx[8 + hh]), fmaxf(mx[16 + hh], mx[24 + hh]));
            const float mn = fmaxf(M[hh], pm);
            al[hh] = ex2_approx(M[hh] - mn);
            M[hh] = mn;
            pr[e] = ex2_approx(lg[hh] - mn);
            L[hh] = fmaf(L[hh], al[hh], pr[e]);
            zz[hh] = pr[e] * zv;
          }
          const float2 wv = make_float2(pr[0] * svc, pr[1] * svc);
          const __half2 wh = __floats2half2_rn(wv.x, wv.y);
          ph[hp] = h2u(wh);
          pl[hp] = h2u(__floats2half2_rn(wv.x - __low2float(wh), wv.y - __high2float(wh)));
        }
        uint8_t* bp = b_pv(s) + boff;
        *reinterpret_cast<uint4*>(bp) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
        *reinterpret_cast<uint4*>(bp + 128) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
        // the warp's sums of p . z'_V: a halving butterfly leaves head zhead in lanes 4k
#pragma unroll
        for (int o = 16, nv = 4; o >= 4; o >>= 1, nv >>= 1) {
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int i2 = 0; i2 < nv; ++i2) {
            const float send = up ? zz[i2] : zz[i2 + nv];
            const float keep = up ? zz[i2 + nv] : zz[i2];
            zz[i2] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        float zsum = zz[0];
        zsum += __shfl_xor_sync(0xffffffffu, zsum, 2);
        zsum += __shfl_xor_sync(0xffffffffu, zsum, 1);
        float* az = az_s + s * 40;
        if ((lane & 3) == 0) az[8 + q * 8 + zhead] = zsum;
        if (u == 0) {
          *reinterpret_cast<float4*>(az) = make_float4(al[0], al[1], al[2], al[3]);
          *reinterpret_cast<float4*>(az + 4) = make_float4(al[4], al[5], al[6], al[7]);
        }
        fence_proxy_async_smem();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[s]);
      }
      // the row's (m, l): l summed over the 128 tokens
#pragma unroll
      for (int hh = 0; hh < 8; ++hh) {
        float v = L[hh];
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
        if (lane == 0) lr_s[q * 8 + hh] = v;
      }
      if (group_any(kSmBar, bad || stop)) break;
      if (u < 8) {
        float* dst = part_row(w, u);
        float mu = M[0], lu = 0.0f;
#pragma unroll
        for (int hh = 0; hh < 8; ++hh)
          if (hh == u) mu = M[hh];
        lu = (lr_s[u] + lr_s[8 + u]) + (lr_s[16 + u] + lr_s[24 + u]);
        dst[0] = mu;
        dst[1] = lu;
      }
      group_any(kSmBar, false);  // lr_s is read before the next row writes it
    }
  } else {
    // ---- V convert and output update (thread = channel) ----
    const int c = threadIdx.x - 256;  // channel 0..127
    const int q = warp - 8;           // tensor-memory lane quarter
    int64_t g = 0;
    int r = 0;
    uint32_t rph = 0;
    int re = 0;  // record slot of the page the output update takes next
    bool bad = false;
    float O[8];
    // output update of page gp (its record slot re)
    auto epilogue = [&](int64_t gp) {
      const int s = (int)(gp & 3);
      const uint32_t par = (uint32_t)((gp >> 2) & 1);
      if (!wait_all(&pv_done[s], par) || !wait_all(&p_full[s], par)) {
        bad = true;
        fail();
        return;
      }
      fence_after();
      float d[16];
      ld_sum2(stage_tmem(s) + kColD + ((uint32_t)(32 * q) << 16), d);
      // the page's rescale and z sums, and the channel factor, are read before the stage and
      // the record slot are handed back
      const float* az = az_s + s * 40;
      float al[8], z[8];
#pragma unroll
      for (int hh = 0; hh < 8; ++hh) {
        al[hh] = az[hh];
        z[hh] = (az[8 + hh] + az[16 + hh]) + (az[24 + hh] + az[32 + hh]);
      }
      const float cv = __half2float(reinterpret_cast<const __half*>(recs + re * kRec + kRL.vfactor)[c]);
      fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&pv_read[s]);
        mbar_arrive(&rec_empty[re]);
      }
      if (++re == kSlots) re = 0;
#pragma unroll
      for (int hh = 0; hh < 8; ++hh) O[hh] = fmaf(O[hh], al[hh], cv * fmaf(d[hh] + d[8 + hh], kAccPV, z[hh]));
    };
    for (Walk w = w0; w.left > 0 && !bad; w.next(p)) {
#pragma unroll
      for (int hh = 0; hh < 8; ++hh) O[hh] = 0.0f;
      const int cnt = w.count();
      for (int i = 0; i < cnt; ++i, ++g) {
        const int s = (int)(g & 3);
        const uint32_t par = (uint32_t)((g >> 2) & 1);
        // V codes into the stage once QK has read its K codes: channel blocks 2q, 2q + 1;
        // token block o = 2op + a at columns 8o..8o+7, column 8o + 2tq + hh holding tokens
        // 16o + 8hh + 2tq, +1 (x4^(2a + hh))
        if (!wait_all(&qk_full[s], par) || !wait_all(&rec_full[r], rph)) {
          bad = true;
          fail();
          break;
        }
        fence_after();
        {
          const uint2* vc = reinterpret_cast<const uint2*>(recs + r * kRec + kRL.vcodes);
#pragma unroll
          for (int ii = 0; ii < 2; ++ii) {
            uint32_t rr[32];
#pragma unroll
            for (int op = 0; op < 4; ++op) {
              const uint2 w2 = vc[(((op * 2 + (q >> 1)) * 32 + lane) * 4 + 2 * (q & 1)) >> 1];
              const uint32_t x = ii ? w2.y : w2.x, y = x >> 8;
              rr[8 * op] = x & 0x00030003u;
              rr[8 * op + 1] = x & 0x000C000Cu;
              rr[8 * op + 2] = y & 0x00030003u;
              rr[8 * op + 3] = y & 0x000C000Cu;
              rr[8 * op + 4] = x & 0x00300030u;
              rr[8 * op + 5] = x & 0x00C000C0u;
              rr[8 * op + 6] = y & 0x00300030u;
              rr[8 * op + 7] = y & 0x00C000C0u;
            }
            st_16x256b_x8(stage_tmem(s) + ((uint32_t)(32 * q + 16 * ii) << 16), rr);
          }
        }
        if (++r == kSlots) {
          r = 0;
          rph ^= 1u;
        }
        wait_st();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ops_v[s]);
        if (i > 0) {
          epilogue(g - 1);
          if (bad) break;
        }
      }
      if (bad) break;
      if (cnt > 0) epilogue(g - 1);
      if (bad) break;
#pragma unroll
      for (int hh = 0; hh < 8; ++hh) part_row(w, hh)[4 + c] = O[hh];
    }
  }

  // ---- tear-down: every role is past its last wait ----
  fence_before();
  __syncthreads();
  grid_launch_dependents();
  if (warp == kPvWarp) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols));
  }
}

bool decode_tc_serves(int d, int nt, int kb, int vb, const DecodeParams& p) {
  return d == 128 && nt == 2 && kb == 4 && vb == 2 && p.group == 8 && p.chunk == 1 && p.chunk_k == nullptr;
}

int decode_tc_ctas() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

int launch_decode_tc(const DecodeParams& p, int phases, cudaStream_t stream) {
  if (p.part_ctas < 1) return KVARN_ERR_INVALID_ARG;
  if ((phases & kDecodeSplits) != 0) {
    static PerDeviceOnce smem_once;
    const void* fn = reinterpret_cast<const void*>(decode_tc_kernel);
    if (const int st = set_smem_limit(smem_once, fn, kSmemBytes); st != KVARN_OK) return st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.part_ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_tc_kernel, p) != cudaSuccess) return KVARN_ERR_CUDA;
    if (p.partial_k != nullptr && p.partial_in_merge == 0) {
      if (const int st = launch_decode_partial_tiles(p, stream); st != KVARN_OK) return st;
    }
  }
  if ((phases & kDecodeMerge) != 0) return launch_decode_combine(D, p, stream);
  return KVARN_OK;
}

}  // namespace kvarn
