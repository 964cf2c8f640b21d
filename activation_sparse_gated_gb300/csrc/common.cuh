// common.cuh -- sm_103a device helpers: mbarriers, bulk async copies (TMA
// engine, non-tensor form), programmatic dependent launch, bounded waits, and
// bf16/fp32 unpacking for the fp32-accumulating dot products.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sffn {

// device error word bits (the handle's ctrl[CTRL_ERR])
constexpr int DEV_ERR_TIMEOUT = 1;
constexpr int DEV_ERR_CHECK = 2;  // a device-side bounds or alignment check failed (the access was skipped)

// ctrl[] layout: one small int array per handle
constexpr int CTRL_TICKET = 0;   // blocks finished in the current forward
constexpr int CTRL_ERR = 1;      // device error word (sticky until read)
constexpr int CTRL_PROBE = 2;    // flag the timeout probe waits on (never set)
constexpr int CTRL_COUNT = 4;    // [B_max] live-count accumulators
constexpr int CTRL_INTS = 4 + 128;
// the streaming kernel spreads its cross-block sum over this many fp32 copies
// of the accumulator (a handle's accumulator holds at least this many rows)
constexpr int YACC_COPIES = 4;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
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

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase.  Gives up when `abort` (a shared flag
// another role raised) becomes non-zero or after `limit_ns`, in which case it
// raises `abort`, records DEV_ERR_TIMEOUT in `err` and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* err, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        atomicOr(err, DEV_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// One contiguous global -> shared copy on the bulk-copy (TMA) engine,
// completing `bytes` of transaction count on `bar`.  Both addresses 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// The same by shared-window addresses (destination and mbarrier as 32-bit shared addresses).
__device__ __forceinline__ void bulk_g2s_a(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst), "l"(src),
      "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_a(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
  uint32_t v;
  asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
  return v;
}

// Same, with an L2 eviction-priority policy (createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Request `bytes` (a multiple of 16) starting at a 16-byte aligned address into
// L2, one bulk-copy-engine operation.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Programmatic dependent launch: wait for the preceding kernel in the stream
// (and its memory) / allow the next kernel to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Element traits: a 16-byte chunk holds VPC values; `unpack` widens it to fp32.
template <typename T>
struct Elt;

struct bf16_tag {};

template <>
struct Elt<float> {
  static constexpr int VPC = 4;
  static constexpr int BYTES = 4;
  __device__ __forceinline__ static void unpack(const uint4& c, float (&v)[4]) {
    v[0] = __uint_as_float(c.x);
    v[1] = __uint_as_float(c.y);
    v[2] = __uint_as_float(c.z);
    v[3] = __uint_as_float(c.w);
  }
};

template <>
struct Elt<bf16_tag> {
  static constexpr int VPC = 8;
  static constexpr int BYTES = 2;
  // a bf16 value is the upper half of a binary32: widening is a shift
  __device__ __forceinline__ static void unpack(const uint4& c, float (&v)[8]) {
    v[0] = __uint_as_float(c.x << 16);
    v[1] = __uint_as_float(c.x & 0xffff0000u);
    v[2] = __uint_as_float(c.y << 16);
    v[3] = __uint_as_float(c.y & 0xffff0000u);
    v[4] = __uint_as_float(c.z << 16);
    v[5] = __uint_as_float(c.z & 0xffff0000u);
    v[6] = __uint_as_float(c.w << 16);
    v[7] = __uint_as_float(c.w & 0xffff0000u);
  }
};

// Packed fp32x2 arithmetic (sm_100 and later): two lanes of fp32 per
// instruction, each lane rounded exactly as the scalar operation.
__device__ __forceinline__ void ffma2(float2& acc, float2 a, float2 b) {
  asm("{\n\t.reg .b64 A, B, C;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\tmov.b64 C, {%0, %1};\n\t"
      "fma.rn.f32x2 C, A, B, C;\n\tmov.b64 {%0, %1}, C;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 A, B, D;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\t"
      "add.rn.f32x2 D, A, B;\n\tmov.b64 {%0, %1}, D;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// 16-byte shared-memory loads through the shared window explicitly: a pointer
// that reaches a kernel's loop through a lambda capture may otherwise compile
// to a generic load (measured: 0.1 us per call on the bf16 streaming kernel,
// 0.6 us on the int8 one).
__device__ __forceinline__ float4 lds_f4(const float4* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(smem_u32(p)));
  return v;
}
__device__ __forceinline__ uint4 lds16(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)));
  return v;
}

// fp32 -> storage type, round to nearest even (bf16 via the CUDA intrinsic)
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Options of the full low-rank gate ("LoPA Gating: moving the ceiling"),
// the values of SFFN_GATE_TILED_G, SFFN_GATE_RMSNORM, SFFN_DOUBLE_ACT:
//   tiled identity G:  z_i += x_{i mod D}
//   RMSNorm:           t = V x  ->  t / sqrt(mean(t^2) + eps), no gain
//   double activation: the up value of a unit is A(W3 x) instead of W3 x
constexpr int FLAG_TILED_G = 1;
constexpr int FLAG_RMSNORM = 2;
constexpr int FLAG_DOUBLE_ACT = 4;
constexpr int FLAG_DETERMINISTIC = 8;  // blocks write partial y rows, summed in block order
constexpr float RMSNORM_EPS = 1e-6f;

// Element e of a vector staged as 16-byte chunks of its storage type.
template <typename T>
__device__ __forceinline__ float staged_elem(const uint4* v, int e);
template <>
__device__ __forceinline__ float staged_elem<float>(const uint4* v, int e) {
  return reinterpret_cast<const float*>(v)[e];
}
template <>
__device__ __forceinline__ float staged_elem<bf16_tag>(const uint4* v, int e) {
  return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(v)[e] << 16);
}

// In place t_b <- t_b / sqrt(mean(t_b^2) + eps) for nb <= warps-per-block
// vectors of k fp32 values in shared memory (warp b sums vector b).  Every
// thread of the block calls it; scale[] holds nb floats of shared scratch.
__device__ __forceinline__ void rmsnorm_shared(float* t, int nb, int k, float* scale, int nthreads) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp < nb) {
    float ss = 0.f;
    for (int i = lane; i < k; i += 32) ss = fmaf(t[(size_t)warp * k + i], t[(size_t)warp * k + i], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) scale[warp] = 1.f / sqrtf(ss / (float)k + RMSNORM_EPS);
  }
  __syncthreads();
  for (int i = tid; i < nb * k; i += nthreads) t[i] *= scale[i / k];
  __syncthreads();
}

// The activation A on the gate: ReLU (0), R-S+ (1: z * sigmoid(z) = z / (1 + e^-z)
// for z > 0, else 0) and the smooth SiLU (2: z * sigmoid(z) everywhere).
constexpr int ACT_SILU = 2;
__device__ __forceinline__ float activation(int act, float z) {
  if (act == ACT_SILU) return z / (1.f + expf(-z));
  if (!(z > 0.f)) return 0.f;
  if (act == 0) return z;
  return z / (1.f + expf(-z));
}

// A unit is live when |A(z)| exceeds the handle's threshold (0 by default,
// which for ReLU and R-S+ is z > 0).
__device__ __forceinline__ bool is_live(float a, float thr) { return fabsf(a) > thr; }

}  // namespace sffn
