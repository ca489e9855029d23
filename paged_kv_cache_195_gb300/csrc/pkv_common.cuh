// pkv_common.cuh -- shared constants and sm_103a PTX helpers for the
// paged-KV kernels: mbarriers, bulk (non-tensor) async copies, bounded waits,
// packed fp32 arithmetic and bf16 unpacking.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

namespace pkv {

constexpr int kHeadDim = 128;
constexpr int kBlockSize = 16;
// One (block, KV head) tile of the pool: 16 tokens x 128 dims x 2 bytes.
constexpr int kTileBytes = kBlockSize * kHeadDim * 2;
// Largest num_reqs pkv_attention accepts.
constexpr int kMaxReqs = 65536;

// Device error word bits (see pkv_get_device_error).
constexpr int kErrBounds = 1;   // block id / slot / lengths out of range
constexpr int kErrTimeout = 2;  // a bounded wait ran out
constexpr int kErrCapacity = 4; // plan exceeded the workspace bound

// Default of the bounded waits' limit (nanoseconds of %globaltimer); the
// host passes the limit to every kernel (pkv_options.wait_limit_us).
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // 2 s

// Per-CTA state of the bounded waits, in shared memory: the abort flag every
// wait checks, and the limit after which a wait gives up.
struct WaitCtl {
  volatile int abort;
  int pad;
  unsigned long long limit_ns;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_error(int* err, int bits) {
  if (err != nullptr) atomicOr(err, bits);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One probe of an mbarrier phase (returns at once).
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

// Waits for the phase with the given parity to complete.  Gives up and
// returns false if the CTA's abort flag is set, or after ctl->limit_ns (then
// it records kErrTimeout and sets the abort flag so that every other wait of
// the CTA returns at once).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err,
                                          WaitCtl* ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    if (ctl->abort) return false;
    #pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > ctl->limit_ns) {
      record_error(err, kErrTimeout);
      ctl->abort = 1;
      return false;
    }
  }
}

// The same wait without the abort flag, for draining an aborted CTA: it
// still gives up after ctl->limit_ns (recording kErrTimeout).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, int* err,
                                                WaitCtl* ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    #pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > ctl->limit_ns) {
      record_error(err, kErrTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------- bulk async copy
// Global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) that completes `bytes` transactions on `bar`.  Streaming data is
// marked evict-first in L2: every KV tile is read once per step.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its writes are visible (a no-op when the launch
// had no programmatic dependency), and allow the next kernel to be scheduled.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// *p += v at GPU scope with acquire-release semantics (returns the old
// value): one instruction instead of a fence, a relaxed atomic and a fence.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Named barrier over `threads` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------------- arithmetic
// OR of `v` over the `threads` threads (a multiple of 32) that meet at named
// barrier `id`; also a barrier for them.
__device__ __forceinline__ bool barrier_or(int id, int threads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

// s0 += low bf16 of w, s1 += high bf16 of w, each by one mixed-precision FMA
// (bf16 times bf16 one, plus fp32): the same fp32 sums as widening first.
__device__ __forceinline__ void add_bf16x2(float& s0, float& s1, uint32_t w) {
  const unsigned short one = 0x3F80;  // bf16 1.0
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "fma.rn.f32.bf16 %0, lo, %3, %0;\n\t"
      "fma.rn.f32.bf16 %1, hi, %3, %1;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "r"(w), "h"(one));
}

// max(a, b, c) in one instruction (the three-input form of max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32: d = a * b + c on both lanes of a float2 (one instruction).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(reinterpret_cast<unsigned long long&>(d))
      : "l"(reinterpret_cast<unsigned long long&>(a)),
        "l"(reinterpret_cast<unsigned long long&>(b)),
        "l"(reinterpret_cast<unsigned long long&>(c)));
  return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(reinterpret_cast<unsigned long long&>(d))
      : "l"(reinterpret_cast<unsigned long long&>(a)),
        "l"(reinterpret_cast<unsigned long long&>(b)));
  return d;
}

// Two packed bf16 -> two fp32 (exact: a bf16 is the top half of an fp32).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  float2 r;
  r.x = __uint_as_float(w << 16);
  r.y = __uint_as_float(w & 0xffff0000u);
  return r;
}

// Two e4m3 codes (low byte first) to fp32, exactly: the hardware
// e4m3x2 -> f16x2 conversion (every e4m3 value is an f16 value), then f16 -> f32.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
  const __half2_raw h =
      __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two_codes, __NV_E4M3);
  return __half22float2(__half2(h));
}

// 16-byte shared-memory load (a plain access, so the compiler orders it
// after the mbarrier waits, which clobber memory).
__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

}  // namespace pkv
