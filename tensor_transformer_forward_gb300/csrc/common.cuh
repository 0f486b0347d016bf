// Shared device helpers: status flags, bounded waits, bf16 / fp16 conversion.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

// Bits OR-ed into the caller's device status word (read back by tp_read_status).
#define TP_DEVFLAG_BAD_TOKEN 1
#define TP_DEVFLAG_TIMEOUT 2
#define TP_DEVFLAG_SATURATED 4  // an fp16 operand was clamped to +-65504

// Every spin-wait in these kernels gives up after this long, sets
// TP_DEVFLAG_TIMEOUT and lets the kernel return.
#define TP_WAIT_LIMIT_NS 2000000000ull

namespace tpk {

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void raise_flag(int* status, int flag) {
  if (status) atomicOr(status, flag);
}

// True on every lane when v is true on every lane of the (converged) warp.  A
// bounded wait can give up on one lane and succeed on another; warp-collective
// instructions after it (tcgen05.ld/st, __syncwarp) need one decision per warp.
__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// Programmatic dependent launch: every kernel of the path is launched so that it
// may start while the previous kernel in the stream finishes.  A kernel calls
// griddep_wait() before it reads anything an earlier kernel wrote and before
// its first global write; griddep_launch() lets the next kernel be scheduled.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Drops the 128-byte L2 line at p (128-byte aligned) without writing it back: only
// for data that is dead (no reader before its next write).
__device__ __forceinline__ void l2_discard(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ __nv_bfloat16 f2bf(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

#define TP_F16_MAX 65504.0f

// fp16 operands (GEMM / attention inputs): saturate to the finite fp16 range.  Each
// conversion ORs into `sat` (a per-thread accumulator) whether it clamped; the
// thread reports it with report_sat, which sets TP_DEVFLAG_SATURATED in the
// status word, so a clamp is never silent.  NaN passes through unflagged.
__device__ __forceinline__ float sat_f16(float x, uint32_t& sat) {
  const bool over = fabsf(x) > TP_F16_MAX;
  sat |= over ? 1u : 0u;
  return over ? copysignf(TP_F16_MAX, x) : x;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi, uint32_t& sat) {
  lo = sat_f16(lo, sat);
  hi = sat_f16(hi, sat);
  __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ __half to_f16(float x, uint32_t& sat) { return __float2half_rn(sat_f16(x, sat)); }
// Per thread, no warp collective (callers may have diverged); the branch is rarely taken.
__device__ __forceinline__ void report_sat(int* status, uint32_t sat) {
  if (sat) raise_flag(status, TP_DEVFLAG_SATURATED);
}
__device__ __forceinline__ float f16lo(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu))); }
__device__ __forceinline__ float f16hi(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace tpk
