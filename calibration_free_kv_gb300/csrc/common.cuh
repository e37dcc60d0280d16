// Shared device helpers and the page-record geometry of the KVarN kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>

#include "kvarn.h"

namespace kvarn {

constexpr int kTile = 128;                 // tokens per tile == tokens per page
constexpr float kLog2e = 1.4426950408889634f;

// Byte offsets of the sections of one (page, kv head) record for padded head_dim d: the K half
// (codes, scale, zero, token factor) then the V half (codes, scale, zero, channel factor).
struct RecordLayout {
  int kcodes, kscale, kzero, kfactor, vcodes, vscale, vzero, vfactor, bytes;
};

// Page record of one (page, kv head) with kb-bit K codes and vb-bit V codes: the K half
// (codes, scale[d], zero[d], token factor[128]) then the V half (codes, scale[128],
// zero[128], channel factor[d]); metadata fp16, every section 16-byte aligned.
__host__ __device__ constexpr RecordLayout record_layout(int d, int kb = 4, int vb = 2) {
  return RecordLayout{0,
                      kTile * d * kb / 8,
                      kTile * d * kb / 8 + 2 * d,
                      kTile * d * kb / 8 + 4 * d,
                      kTile * d * kb / 8 + 4 * d + 2 * kTile,
                      kTile * d * kb / 8 + 4 * d + 2 * kTile + kTile * d * vb / 8,
                      kTile * d * kb / 8 + 4 * d + 4 * kTile + kTile * d * vb / 8,
                      kTile * d * kb / 8 + 4 * d + 6 * kTile + kTile * d * vb / 8,
                      kTile * d * kb / 8 + 6 * d + 6 * kTile + kTile * d * vb / 8};
}

// Raises a kernel's dynamic shared-memory limit to `bytes` once per device.  The attribute
// belongs to the device's context, so a process that launches on several GPUs sets it on each:
// `once` (one static object per kernel) remembers the devices done, 0..63; devices beyond that
// set it on every launch.  Concurrent first calls both set it, which is harmless.
struct PerDeviceOnce {
  std::atomic<uint64_t> done{0};
};
inline int set_smem_limit(PerDeviceOnce& once, const void* kernel, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return KVARN_ERR_CUDA;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit != 0ull && (once.done.load(std::memory_order_acquire) & bit) != 0ull) return KVARN_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return KVARN_ERR_CUDA;
  if (bit != 0ull) once.done.fetch_or(bit, std::memory_order_release);
  return KVARN_OK;
}

__device__ __forceinline__ void flag_error(int32_t* status, int bits) {
  if (status != nullptr) atomicOr(status, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- packed fp32 pairs (sm_100+: one instruction issues two IEEE round-to-nearest ops) -------
__device__ __forceinline__ unsigned long long pack_f2(float2 v) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
  return r;
}
__device__ __forceinline__ float2 unpack_f2(unsigned long long r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack_f2(a)), "l"(pack_f2(b)));
  return unpack_f2(d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack_f2(a)), "l"(pack_f2(b)));
  return unpack_f2(d);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack_f2(a)), "l"(pack_f2(b)));
  return unpack_f2(d);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pack_f2(a)), "l"(pack_f2(b)), "l"(pack_f2(c)));
  return unpack_f2(d);
}

// three-input min / max (sm_100+)
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ---- programmatic dependent launch ----------------------------------------------------------
// A kernel launched with programmatic stream serialization may start before the previous
// kernel of the stream has finished; grid_dependency_wait() blocks until that kernel has
// completed and its memory is visible (a no-op when there is no such dependency).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel of the stream (if launched as a dependent) start its CTAs.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier + 1-D bulk copy (TMA engine, no tensor map) ---------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Global -> shared bulk copy completing on `bar`.  dst/src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after ~2 s of wall time (or 2^26 polls) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1; it < (1u << 26); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > 2000000000ull) return false;
  }
  return false;
}

// Bounded wait for warps that share their scheduler with busy ones: between polls the thread
// sleeps (32 ns doubling to 256 ns), so a waiting warp takes few issue slots.  Gives up after
// ~2 s of wall time and returns false.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t ns = 32;
  for (uint32_t it = 1; it < (1u << 26); ++it) {
    __nanosleep(ns);
    if (mbar_try_wait(bar, parity)) return true;
    if (ns < 256) ns <<= 1;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > 2000000000ull) return false;
  }
  return false;
}

}  // namespace kvarn
