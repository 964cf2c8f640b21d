// finalize.cu -- last step of a forward: y = sum of the fp32 accumulator copies.
//
// The forward kernels add each block's partial y into one of YACC_COPIES fp32
// copies of the accumulator (fewer blocks per address) and end.  This kernel,
// launched right behind them with programmatic dependent launch, waits for
// their completion (which orders all of their atomics), then per 16-byte
// group of y: loads the copies, clears them for the next call, rounds the sum
// once to the output dtype (round to nearest even for bf16) and stores it.
// Block 0 also publishes the per-token live counts and clears their
// accumulators.  One thread per float4 of y per token.
#include "common.cuh"
#include "internal.h"

namespace sffn {

namespace {

constexpr int FT = 128;

template <typename T>
__global__ void __launch_bounds__(FT) finalize_kernel(float* __restrict__ yacc, void* __restrict__ y,
                                                      int* __restrict__ ctrl, int* __restrict__ counts,
                                                      int count_slot, int D, int nb) {
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();
  const int n4 = D / 4;
  const int idx = blockIdx.x * FT + threadIdx.x;
  float4* ya = reinterpret_cast<float4*>(yacc);
  if (idx < nb * n4) {
    const int b = idx / n4, i = idx - b * n4;
    float4 c[YACC_COPIES];
#pragma unroll
    for (int r = 0; r < YACC_COPIES; ++r) c[r] = __ldcg(ya + ((size_t)b * YACC_COPIES + r) * n4 + i);
    float4 v = c[0];
#pragma unroll
    for (int r = 1; r < YACC_COPIES; ++r) {
      v.x += c[r].x;
      v.y += c[r].y;
      v.z += c[r].z;
      v.w += c[r].w;
    }
#pragma unroll
    for (int r = 0; r < YACC_COPIES; ++r)
      __stcg(ya + ((size_t)b * YACC_COPIES + r) * n4 + i, make_float4(0.f, 0.f, 0.f, 0.f));
    if constexpr (Elt<T>::VPC == 4) {
      reinterpret_cast<float4*>(y)[(size_t)b * n4 + i] = v;
    } else {
      reinterpret_cast<uint2*>(y)[(size_t)b * n4 + i] =
          make_uint2(pack_bf16x2_rn(v.x, v.y), pack_bf16x2_rn(v.z, v.w));
    }
  }
  if (blockIdx.x == 0 && threadIdx.x < nb) {
    counts[threadIdx.x] = __ldcg(ctrl + CTRL_COUNT + count_slot + threadIdx.x);
    __stcg(ctrl + CTRL_COUNT + count_slot + threadIdx.x, 0);
  }
}

// One thread per float4 of y: the blocks' partial rows summed in block order
// (one fixed order, hence bitwise reproducible), rounded once.
__global__ void __launch_bounds__(FT) finalize_ordered_kernel(const float* __restrict__ ypart, int nblocks,
                                                              uint2* __restrict__ y, int* __restrict__ ctrl,
                                                              int* __restrict__ counts, int count_slot, int D) {
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();
  const int n4 = D / 4;
  const int i = blockIdx.x * FT + threadIdx.x;
  if (i < n4) {
    const float4* yp = reinterpret_cast<const float4*>(ypart) + i;
    float4 v = __ldcg(yp);
    for (int b = 1; b < nblocks; ++b) {
      const float4 w = __ldcg(yp + (size_t)b * n4);
      v.x += w.x;
      v.y += w.y;
      v.z += w.z;
      v.w += w.w;
    }
    y[i] = make_uint2(pack_bf16x2_rn(v.x, v.y), pack_bf16x2_rn(v.z, v.w));
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    counts[0] = __ldcg(ctrl + CTRL_COUNT + count_slot);
    __stcg(ctrl + CTRL_COUNT + count_slot, 0);
  }
}

}  // namespace

cudaError_t launch_finalize_ordered(const float* ypart, int nblocks, void* y, int* ctrl, int* counts, int count_slot,
                                    int D, cudaStream_t s) {
  const dim3 g((D / 4 + FT - 1) / FT), b(FT);
  return launch_pdl(finalize_ordered_kernel, g, b, 0, s, ypart, nblocks, static_cast<uint2*>(y), ctrl, counts,
                    count_slot, D);
}

cudaError_t launch_finalize(float* yacc, void* y, int* ctrl, int* counts, int count_slot, int D, int nb,
                            int dtype, cudaStream_t s) {
  const int n = nb * (D / 4);
  const dim3 g((n + FT - 1) / FT), b(FT);
  if (dtype == 0) return launch_pdl(finalize_kernel<float>, g, b, 0, s, yacc, y, ctrl, counts, count_slot, D, nb);
  return launch_pdl(finalize_kernel<bf16_tag>, g, b, 0, s, yacc, y, ctrl, counts, count_slot, D, nb);
}

}  // namespace sffn
