// lopa_t.cu -- first stage of the low-rank gate: t = V x (fp32, not rounded).
//
// "LoPA Gating: moving the ceiling" (ai.thesatyajit.com): W1 = G + UV with
// U in R^{H x r}, V in R^{r x D}; the gate costs r(D + H) instead of HD.  This
// library evaluates the UV part as U (V x); this kernel produces t = V x for
// every token of the batch, and the fused kernel (ffn_b1.cu) or the batched
// gate applies U.
//
// One warp per row k of V.  The row (a contiguous D-element run) is loaded into
// registers before the programmatic-dependent-launch wait: weights never depend
// on earlier kernels, so the load overlaps the previous call's tail; x (which
// may be the previous call's output) is read only after the wait.
//
// Batches (lopa_t_batch_kernel): the block stages the x rows of up to TBB
// tokens at a time in shared memory (one coalesced round trip per group, read
// by all of the block's rows), and each warp dots its register-held V row with
// them.  For bf16 tensor-core batches (ffn_tc.cu) t is written as a bf16 pair,
// t = t_hi + t_lo to about 16 bits: t_hi of token b in row b and t_lo in row
// NB + b of a [2 NB, r] buffer, zero rows for b >= B.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace sffn {

namespace {

constexpr int T_WARPS = 8;
constexpr int T_PF = 10;  // 16-byte chunks of the V row prefetched per lane (a whole bf16 row at D=2560)

template <typename T>
__global__ void __launch_bounds__(T_WARPS * 32) lopa_t_kernel(const void* __restrict__ V,
                                                              const void* __restrict__ x,
                                                              float* __restrict__ t, int r, int D,
                                                              int B) {
  using E = Elt<T>;
  constexpr int VPC = E::VPC;
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int k = blockIdx.x * T_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int nch = D * E::BYTES / 16;
  const uint4* vrow = reinterpret_cast<const uint4*>(V) + (size_t)(k < r ? k : 0) * nch;
  uint4 wv[T_PF];
#pragma unroll
  for (int j = 0; j < T_PF; ++j) {
    const int c = lane + 32 * j;
    wv[j] = (k < r && c < nch) ? __ldg(vrow + c) : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();
  if (k >= r) return;
  for (int b = 0; b < B; ++b) {
    const uint4* xv = reinterpret_cast<const uint4*>(x) + (size_t)b * nch;
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int j = 0; j < T_PF; ++j) {
      const int c = lane + 32 * j;
      if (c < nch) {
        float wf[VPC], xf[VPC];
        E::unpack(wv[j], wf);
        E::unpack(xv[c], xf);
#pragma unroll
        for (int v = 0; v < VPC; v += 2) {
          a0 = fmaf(wf[v], xf[v], a0);
          a1 = fmaf(wf[v + 1], xf[v + 1], a1);
        }
      }
    }
    for (int c = lane + 32 * T_PF; c < nch; c += 32) {
      float wf[VPC], xf[VPC];
      E::unpack(__ldg(vrow + c), wf);
      E::unpack(xv[c], xf);
#pragma unroll
      for (int v = 0; v < VPC; v += 2) {
        a0 = fmaf(wf[v], xf[v], a0);
        a1 = fmaf(wf[v + 1], xf[v + 1], a1);
      }
    }
    const float s = warp_sum(a0 + a1);
    if (lane == 0) t[(size_t)b * r + k] = s;
  }
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}

constexpr int T_PFB = 16;          // chunks of the V row held per lane by the batch kernel (bf16 D <= 4096)
constexpr size_t T_XS_BYTES = 96 * 1024;  // shared x rows of one token group

template <typename T, bool PAIR>
__global__ void __launch_bounds__(T_WARPS * 32) lopa_t_batch_kernel(const void* __restrict__ V,
                                                                    const void* __restrict__ x,
                                                                    void* __restrict__ out, int r, int D,
                                                                    int B, int NB, int TBB) {
  using E = Elt<T>;
  constexpr int VPC = E::VPC;
  extern __shared__ __align__(16) uint4 xs[];  // [TBB][nch]
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int k = blockIdx.x * T_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int nch = D * E::BYTES / 16;
  const uint4* vrow = reinterpret_cast<const uint4*>(V) + (size_t)(k < r ? k : 0) * nch;
  uint4 wv[T_PFB];
#pragma unroll
  for (int j = 0; j < T_PFB; ++j) {
    const int c = lane + 32 * j;
    wv[j] = (k < r && c < nch) ? __ldg(vrow + c) : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();
  const uint4* xg = reinterpret_cast<const uint4*>(x);
  for (int b0 = 0; b0 < B; b0 += TBB) {
    const int nb = min(TBB, B - b0);
    __syncthreads();  // the previous group's rows are no longer read
    // every copy in flight at once (a load-then-store loop would wait on each load in turn)
    for (int i = threadIdx.x; i < nb * nch; i += blockDim.x) cp_async16(xs + i, xg + (size_t)b0 * nch + i);
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    if (k < r) {
      for (int t = 0; t < nb; ++t) {
        const uint4* xr = xs + (size_t)t * nch;
        float a0 = 0.f, a1 = 0.f;
        auto chunk = [&](const uint4& w, int c) {
          float wf[VPC], xf[VPC];
          E::unpack(w, wf);
          E::unpack(lds16(xr + c), xf);
#pragma unroll
          for (int v = 0; v < VPC; v += 2) {
            a0 = fmaf(wf[v], xf[v], a0);
            a1 = fmaf(wf[v + 1], xf[v + 1], a1);
          }
        };
#pragma unroll
        for (int j = 0; j < T_PFB; ++j) {
          const int c = lane + 32 * j;
          if (c < nch) chunk(wv[j], c);
        }
        for (int c = lane + 32 * T_PFB; c < nch; c += 32) chunk(__ldg(vrow + c), c);
        const float sum = warp_sum(a0 + a1);
        if (lane == 0) {
          const int b = b0 + t;
          if constexpr (PAIR) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(sum);
            const __nv_bfloat16 lo = __float2bfloat16_rn(sum - __bfloat162float(hi));
            uint16_t* tp = static_cast<uint16_t*>(out);
            tp[(size_t)b * r + k] = __bfloat16_as_ushort(hi);
            tp[(size_t)(NB + b) * r + k] = __bfloat16_as_ushort(lo);
          } else {
            static_cast<float*>(out)[(size_t)b * r + k] = sum;
          }
        }
      }
    }
  }
  if (PAIR && k < r) {  // padding tokens: zero rows, so the MMA columns past B stay finite
    uint16_t* tp = static_cast<uint16_t*>(out);
    for (int b = B + lane; b < NB; b += 32) {
      tp[(size_t)b * r + k] = 0;
      tp[(size_t)(NB + b) * r + k] = 0;
    }
  }
}

// W2[rows=D, cols=H] -> W2t[H, D] through 32x32 shared tiles.
template <typename U>
__global__ void transpose_kernel(const U* __restrict__ src, U* __restrict__ dst, int rows, int cols) {
  __shared__ U tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int rr = r0 + i, cc = c0 + threadIdx.x;
    if (rr < rows && cc < cols) tile[i][threadIdx.x] = src[(size_t)rr * cols + cc];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int cc = c0 + i, rr = r0 + threadIdx.x;
    if (cc < cols && rr < rows) dst[(size_t)cc * rows + rr] = tile[threadIdx.x][i];
  }
}

// Failure-detection probe: wait on a flag nothing sets, bounded by limit_ns.
__global__ void timeout_probe_kernel(int* ctrl, unsigned long long limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  volatile int* flag = ctrl + CTRL_PROBE;
  while (*flag == 0) {
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(ctrl + CTRL_ERR, DEV_ERR_TIMEOUT);
      return;
    }
    __nanosleep(1000);
  }
}

}  // namespace

cudaError_t lopa_t_prepare() {
  cudaError_t e = cudaFuncSetAttribute(lopa_t_batch_kernel<float, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)T_XS_BYTES);
  if (!e)
    e = cudaFuncSetAttribute(lopa_t_batch_kernel<bf16_tag, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)T_XS_BYTES);
  if (!e)
    e = cudaFuncSetAttribute(lopa_t_batch_kernel<bf16_tag, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)T_XS_BYTES);
  return e;
}

namespace {
int tokens_per_group(int D, int elt) { return (int)std::max<size_t>(1, std::min<size_t>(8, T_XS_BYTES / ((size_t)D * elt))); }
}  // namespace

cudaError_t launch_lopa_t(const void* V, const void* x, float* t, int r, int D, int B, int dtype,
                          cudaStream_t s) {
  const dim3 g((r + T_WARPS - 1) / T_WARPS), b(T_WARPS * 32);
  if (B > 1) {
    const int elt = dtype == 0 ? 4 : 2, tbb = tokens_per_group(D, elt);
    const size_t smem = (size_t)tbb * D * elt;
    void* out = t;
    if (dtype == 0) return launch_pdl(lopa_t_batch_kernel<float, false>, g, b, smem, s, V, x, out, r, D, B, B, tbb);
    return launch_pdl(lopa_t_batch_kernel<bf16_tag, false>, g, b, smem, s, V, x, out, r, D, B, B, tbb);
  }
  if (dtype == 0) return launch_pdl(lopa_t_kernel<float>, g, b, 0, s, V, x, t, r, D, B);
  return launch_pdl(lopa_t_kernel<bf16_tag>, g, b, 0, s, V, x, t, r, D, B);
}

cudaError_t launch_lopa_t_pair(const void* V, const void* x, uint16_t* tpair, int r, int D, int B, int NB,
                               cudaStream_t s) {
  const dim3 g((r + T_WARPS - 1) / T_WARPS), b(T_WARPS * 32);
  const int tbb = tokens_per_group(D, 2);
  void* out = tpair;
  return launch_pdl(lopa_t_batch_kernel<bf16_tag, true>, g, b, (size_t)tbb * D * 2, s, V, x, out, r, D, B, NB, tbb);
}

cudaError_t launch_transpose(const void* src, void* dst, int rows, int cols, int elt_bytes,
                             cudaStream_t s) {
  const dim3 g((cols + 31) / 32, (rows + 31) / 32), b(32, 8);
  if (elt_bytes == 4)
    transpose_kernel<uint32_t><<<g, b, 0, s>>>(static_cast<const uint32_t*>(src),
                                               static_cast<uint32_t*>(dst), rows, cols);
  else if (elt_bytes == 1)
    transpose_kernel<uint8_t><<<g, b, 0, s>>>(static_cast<const uint8_t*>(src),
                                              static_cast<uint8_t*>(dst), rows, cols);
  else
    transpose_kernel<uint16_t><<<g, b, 0, s>>>(static_cast<const uint16_t*>(src),
                                               static_cast<uint16_t*>(dst), rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_timeout_probe(int* ctrl, unsigned long long limit_ns, cudaStream_t s) {
  timeout_probe_kernel<<<1, 1, 0, s>>>(ctrl, limit_ns);
  return cudaGetLastError();
}

}  // namespace sffn
