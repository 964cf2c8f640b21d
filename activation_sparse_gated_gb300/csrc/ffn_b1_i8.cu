// ffn_b1_i8.cu -- single-token gate-first sparse FFN with weight-only int8
// weights (standard gate), streaming form; and the per-row quantiser.
//
// "Model Casting and Low-Parameter Gating", appendix Table 17, quantises the
// cast models weight-only to int8.  Convention of this library (the pages give
// none): symmetric, one fp32 scale per output channel -- per row of W1 and W3
// (unit i), per row of W2 (output element m) -- s = max|w| / 127, code =
// round-half-to-even(w / s) clamped to [-127, 127], decided in binary32.  The
// forward is the formula of "Model casting: compute the gate, then skip most of
// the FFN" with every weight replaced by q * s:
//     z_i = s1_i (q1[i, :] . x),   u_i = s3_i (q3[i, :] . x),   h_i = A(z_i) u_i
//     y_m = s2_m sum_{i live} q2t[i, m] h_i      (q2t = the codes of W2, transposed)
// Each block multiplies its partial y by s2 (staged in shared memory before the
// dependency wait) before adding it to the accumulator.  x and y are bf16.
//
// GB300 mapping: the pipeline of the bf16 streaming kernel (ffn_b1_stream.cu)
// with rows of D bytes instead of 2D -- the gate, which is always read in
// full, moves half the bytes.  A 16-byte chunk holds 16 codes, which pair with
// 16 values of x, widened to fp32 once per block in shared memory.  Codes are
// widened to fp32 exactly with a byte permute and a packed add (no int->float
// conversion instruction): the biased byte q + 128 becomes the low mantissa
// byte of 2^23.  q * x is exact in fp32 (7 x 8 significant bits); the sums
// are fp32, two lanes per packed fp32x2 FMA.  There are no spin-waits in this file.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace sffn {

namespace {

constexpr int QW = 12;        // warps per block (two blocks fit an SM)
constexpr int QT = QW * 32;
constexpr int QPIECE = 5;     // 16-byte chunks per lane per piece of a streamed gate row

__host__ __device__ constexpr size_t a16(size_t v) { return (v + 15) & ~size_t(15); }

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void cpa16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cpa_wait() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void pf_l2(const void* row, uint32_t bytes, int j, int nl) {
  const char* b = static_cast<const char*>(row);
  for (uint32_t off = (uint32_t)j * 128u; off < bytes; off += (uint32_t)nl * 128u)
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(b + off));
}

// 4 int8 codes (one 32-bit word) -> 4 exact fp32 values, as 2 pairs.
__device__ __forceinline__ void widen_i8x4(uint32_t word, float2& v01, float2& v23) {
  const uint32_t w = word ^ 0x80808080u;
  const float2 bias = make_float2(-8388736.f, -8388736.f);
  v01 = fadd2(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u)),
                          __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541u))), bias);
  v23 = fadd2(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7542u)),
                          __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7543u))), bias);
}

// acc += code chunk c . x[16c, 16c + 16), two lanes of fp32 per FMA.  x is
// staged as fp32 in the interleaved layout xq[k * ncw + c] = x[16c + 4k .. +4),
// so lanes reading consecutive chunks read consecutive 16-byte words.
__device__ __forceinline__ void dot_chunk(const uint4& w, const float4* xq, int ncw, int c, float2& acc) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 v01, v23;
    widen_i8x4(words[k], v01, v23);
    const float4 xv = lds_f4(xq + k * ncw + c);
    ffma2(acc, v01, make_float2(xv.x, xv.y));
    ffma2(acc, v23, make_float2(xv.z, xv.w));
  }
}

__device__ __forceinline__ void load_piece_i8(uint4 (&w)[QPIECE], const uint4* row, int pc, int lane, int ncw) {
#pragma unroll
  for (int k = 0; k < QPIECE; ++k) {
    const int c = pc * 32 * QPIECE + lane + 32 * k;
    w[k] = (c < ncw) ? ldg_stream(row + c) : make_uint4(0, 0, 0, 0);
  }
}

__global__ void __launch_bounds__(QT, 2) ffn_b1_i8_kernel(const B1Params p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int D = p.D;
  const int nch = D / 8;    // 16-byte bf16 chunks of x
  const int ncw = D / 16;   // 16-byte code chunks of a weight row
  const int npg = (ncw + 32 * QPIECE - 1) / (32 * QPIECE);
  const int row0 = (int)(((long long)blockIdx.x * p.H) / gridDim.x);
  const int row1 = (int)(((long long)(blockIdx.x + 1) * p.H) / gridDim.x);
  const int cap = p.rows_cap;
  // shared: x | W2 scales | the block's W1, W3 scales | live list (unit, A(z), h) | counters |
  // live flags | prefetch / gather area
  uint8_t* sp = smem;
  float4* xq = reinterpret_cast<float4*>(sp);  // x widened to fp32 once per block (interleaved)
  sp += a16((size_t)D * 4);
  float* s2s = reinterpret_cast<float*>(sp);
  sp += a16((size_t)D * 4);
  float* s1s = reinterpret_cast<float*>(sp);
  float* s3s = s1s + cap;
  sp += a16((size_t)cap * 8);
  int* l_unit = reinterpret_cast<int*>(sp);
  float* l_a = reinterpret_cast<float*>(l_unit + cap);
  float* l_h = l_a + cap;
  int* misc = reinterpret_cast<int*>(l_h + cap);  // 0: live count
  uint8_t* l_mask = reinterpret_cast<uint8_t*>(misc + 4);
  sp += a16((size_t)cap * 13 + 16);
  uint4* srows = reinterpret_cast<uint4*>(sp);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint4* G = static_cast<const uint4*>(p.gate_w);
  const uint4* W3 = static_cast<const uint4*>(p.W3);
  const uint4* W2t = static_cast<const uint4*>(p.W2t);

  if (tid == 0) {
    pdl_launch_dependents();
    misc[0] = 0;
  }

  // Gate rows of the block: [0, R) copied into shared memory before the
  // dependency wait, [R, R + nreg) one per warp through registers (first two
  // pieces requested before the wait), the rest in shared-memory batches.
  const int nrows = row1 - row0;
  const int R = min(p.pref_rows, nrows);
  const int nreg = max(0, min(QW, nrows - R));
  auto copy_rows = [&](int first, int n) {
    const uint4* src = G + (size_t)(row0 + first) * ncw;
    for (int i = tid; i < n * ncw; i += QT) cpa16(srows + i, src + i);
    cpa_commit();
  };
  for (int i = tid; i < D / 4; i += QT) cpa16(s2s + 4 * i, p.s2 + 4 * i);  // committed with the rows
  for (int i = tid; i < row1 - row0; i += QT) {  // scales of the block's units (weights: before the wait)
    s1s[i] = __ldg(p.s1 + row0 + i);
    s3s[i] = __ldg(p.s3 + row0 + i);
  }
  copy_rows(0, R);
  const int n_seq = warp < nreg ? npg : 0;
  const uint4* my_row = G + (size_t)(row0 + R + warp) * ncw;
  uint4 wa[QPIECE], wb[QPIECE];
  if (n_seq > 0) load_piece_i8(wa, my_row, 0, lane, ncw);
  if (n_seq > 1) load_piece_i8(wb, my_row, 1, lane, ncw);
  if (tid == 0) asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.x), "r"((uint32_t)nch * 16u)
                             : "memory");

  pdl_wait();  // x, the accumulators and the counters follow stream order
  for (int i = tid; i < nch; i += QT) {  // bf16 chunk i = float4 words 2i, 2i + 1 of x
    float v[8];
    Elt<bf16_tag>::unpack(__ldcg(static_cast<const uint4*>(p.x) + i), v);
    const int f0 = 2 * i, f1 = 2 * i + 1;  // word f: chunk f / 4, quarter f % 4
    xq[(f0 & 3) * ncw + (f0 >> 2)] = make_float4(v[0], v[1], v[2], v[3]);
    xq[(f1 & 3) * ncw + (f1 >> 2)] = make_float4(v[4], v[5], v[6], v[7]);
  }
  cpa_wait();
  __syncthreads();

  auto decide = [&](int q, float dotv) {  // dotv identical in every lane of the warp
    const float z = s1s[q - row0] * dotv;
    const float a = activation(p.act, z);
    const bool live = is_live(a, p.thr);
    if (lane == 0) {
      l_mask[q - row0] = live ? 1 : 0;
      if (live) {
        const int j = atomicAdd(misc, 1);
        l_unit[j] = q;
        l_a[j] = a;
      }
    }
    if (live) {
      pf_l2(W3 + (size_t)q * ncw, (uint32_t)D, lane, 32);
      pf_l2(W2t + (size_t)q * ncw, (uint32_t)D, lane, 32);
    }
  };
  auto shared_rows = [&](int first, int n) {
    for (int i = warp; i < n; i += QW) {
      const uint4* r = srows + (size_t)i * ncw;
      float2 acc = make_float2(0.f, 0.f);
      for (int c = lane; c < ncw; c += 32) dot_chunk(lds16(r + c), xq, ncw, c, acc);
      decide(row0 + first + i, warp_sum(acc.x + acc.y));
    }
  };
  shared_rows(0, R);
  __syncthreads();
  int next = R + nreg;
  int nb1 = min(R, nrows - next);
  if (nb1 > 0) copy_rows(next, nb1);

  float2 acc = make_float2(0.f, 0.f);
  auto consume = [&](const uint4(&w)[QPIECE], int pc) {
#pragma unroll
    for (int k = 0; k < QPIECE; ++k) {
      const int c = pc * 32 * QPIECE + lane + 32 * k;
      if (c < ncw) dot_chunk(w[k], xq, ncw, c, acc);
    }
    if (pc == npg - 1) {
      const float d = warp_sum(acc.x + acc.y);
      acc = make_float2(0.f, 0.f);
      decide(row0 + R + warp, d);
    }
  };
  for (int pc = 0; pc < n_seq; pc += 2) {
    consume(wa, pc);
    if (pc + 2 < n_seq) load_piece_i8(wa, my_row, pc + 2, lane, ncw);
    if (pc + 1 < n_seq) {
      consume(wb, pc + 1);
      if (pc + 3 < n_seq) load_piece_i8(wb, my_row, pc + 3, lane, ncw);
    }
  }
  while (nb1 > 0) {
    cpa_wait();
    __syncthreads();
    shared_rows(next, nb1);
    __syncthreads();
    next += nb1;
    nb1 = min(R, nrows - next);
    if (nb1 > 0) copy_rows(next, nb1);
  }
  __syncthreads();
  const int n_live = misc[0];

  // ---- gathers.  Warp w owns code chunks [cs0, cs0 + cs_n) of a W2^T row,
  // i.e. outputs [16 cs0, 16 (cs0 + cs_n)); lane l holds the 16 outputs of
  // chunk cs0 + l (and of cs0 + 32 + l in a second pass for wide rows).
  const int per = (ncw + QW - 1) / QW;
  const int cs0 = warp * per;
  const int cs_n = min(per, ncw - cs0);
  const bool owns = lane < cs_n;
  const uint4* col = W2t + cs0 + lane;
  const int RB = p.gather_rows;
  const bool dbl = (p.flags & FLAG_DOUBLE_ACT) != 0;
  float yr[16];
#pragma unroll
  for (int v = 0; v < 16; ++v) yr[v] = 0.f;
  auto fold = [&](const uint4& wv, float h) {
    const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
    const float2 hh = make_float2(h, h);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 v01, v23;
      widen_i8x4(words[k], v01, v23);
      float2 a = make_float2(yr[4 * k], yr[4 * k + 1]), b = make_float2(yr[4 * k + 2], yr[4 * k + 3]);
      ffma2(a, v01, hh);
      ffma2(b, v23, hh);
      yr[4 * k] = a.x;
      yr[4 * k + 1] = a.y;
      yr[4 * k + 2] = b.x;
      yr[4 * k + 3] = b.y;
    }
  };
  uint4 r8[8];
  for (int b0 = 0; b0 < n_live; b0 += RB) {
    const int nb = min(RB, n_live - b0);
    for (int i = tid; i < nb * ncw; i += QT) {
      const int u = i / ncw, c = i - u * ncw;
      cpa16(srows + i, W3 + (size_t)l_unit[b0 + u] * ncw + c);
    }
    cpa_commit();
#pragma unroll
    for (int m = 0; m < 8; ++m)
      r8[m] = (owns && m < nb) ? ldg_stream(col + (size_t)l_unit[b0 + m] * ncw) : make_uint4(0, 0, 0, 0);
    cpa_wait();
    __syncthreads();
    for (int u = warp; u < nb; u += QW) {
      const uint4* r = srows + (size_t)u * ncw;
      float2 acc2 = make_float2(0.f, 0.f);
      for (int c = lane; c < ncw; c += 32) dot_chunk(lds16(r + c), xq, ncw, c, acc2);
      const float uval = s3s[l_unit[b0 + u] - row0] * warp_sum(acc2.x + acc2.y);
      if (lane == 0) l_h[b0 + u] = l_a[b0 + u] * (dbl ? activation(p.act, uval) : uval);
    }
    __syncthreads();
    if (owns) {
#pragma unroll
      for (int m = 0; m < 8; ++m)
        if (m < nb) fold(r8[m], l_h[b0 + m]);
      for (int j = 8; j < nb; j += 4) {
#pragma unroll
        for (int m = 0; m < 4; ++m)
          r8[m] = j + m < nb ? ldg_stream(col + (size_t)l_unit[b0 + j + m] * ncw) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          if (j + m < nb) fold(r8[m], l_h[b0 + j + m]);
      }
    }
    __syncthreads();
  }
  float* yc = p.yacc + (size_t)(blockIdx.x % YACC_COPIES) * D;
  auto add_scaled = [&](int chunk) {  // y[16 chunk + v] += s2[16 chunk + v] * yr[v]
    const float4* sc = reinterpret_cast<const float4*>(s2s + (size_t)chunk * 16);
#pragma unroll
    for (int v = 0; v < 16; v += 4) {
      const float4 f = sc[v / 4];
      atomicAdd(reinterpret_cast<float4*>(yc + (size_t)chunk * 16 + v),
                make_float4(f.x * yr[v], f.y * yr[v + 1], f.z * yr[v + 2], f.w * yr[v + 3]));
    }
  };
  if (n_live > 0 && owns) add_scaled(cs0 + lane);
  if (n_live > 0 && lane + 32 < cs_n) {  // rows wider than 32 chunks per warp
#pragma unroll
    for (int v = 0; v < 16; ++v) yr[v] = 0.f;
    for (int j = 0; j < n_live; j += 4) {
#pragma unroll
      for (int m = 0; m < 4; ++m)
        r8[m] = j + m < n_live ? ldg_stream(col + 32 + (size_t)l_unit[j + m] * ncw) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        if (j + m < n_live) fold(r8[m], l_h[j + m]);
    }
    add_scaled(cs0 + 32 + lane);
  }
  if (tid == 0 && n_live > 0) atomicAdd(p.ctrl + CTRL_COUNT + p.count_slot, n_live);
  if (p.mask)
    for (int i = tid; i < nrows; i += QT) p.mask[row0 + i] = l_mask[i];
}

// One block per row of a bf16 matrix: s = max|w| / 127, codes = round-half-even(w / s)
// clamped to [-127, 127] (binary32 division, correctly rounded); s = 0 and codes 0 for
// an all-zero row.
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint16_t* __restrict__ src,
                                                            int8_t* __restrict__ dst, float* __restrict__ scale,
                                                            int cols) {
  __shared__ float red[8];
  const uint16_t* w = src + (size_t)blockIdx.x * cols;
  int8_t* q = dst + (size_t)blockIdx.x * cols;
  float amax = 0.f;
  for (int j = threadIdx.x; j < cols; j += 256) amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)w[j] << 16)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) amax = fmaxf(amax, red[k]);
  const float s = __fdiv_rn(amax, 127.f);
  if (threadIdx.x == 0) scale[blockIdx.x] = s;
  for (int j = threadIdx.x; j < cols; j += 256) {
    int v = 0;
    if (s > 0.f) {
      v = __float2int_rn(__fdiv_rn(__uint_as_float((uint32_t)w[j] << 16), s));
      v = max(-127, min(127, v));
    }
    q[j] = (int8_t)v;
  }
}

}  // namespace

StreamPlan plan_ffn_b1_i8(int D, int rows_cap) {
  StreamPlan pl;
  const size_t row = (size_t)D;  // bytes of a code row
  // two blocks per SM (the next call's blocks prefetch while this call runs):
  // at most 110 KB per block, of which the gate-row area takes what is left
  const size_t fixed = 2 * a16((size_t)D * 4) + a16((size_t)rows_cap * 8) + a16((size_t)rows_cap * 13 + 16);
  const size_t budget = 110u * 1024u;
  const size_t free_area = budget > fixed ? budget - fixed : 0;
  pl.pref_rows = (int)std::min<size_t>((size_t)rows_cap, std::max<size_t>(1, free_area / row));
  const size_t area = std::max((size_t)pl.pref_rows * row, (size_t)std::min(rows_cap, 16) * row);
  pl.gather_rows = (int)std::max<size_t>(1, area / row);
  pl.smem = fixed + area;
  return pl;
}

cudaError_t ffn_b1_i8_prepare(size_t max_smem) {
  cudaError_t e = cudaFuncSetAttribute(ffn_b1_i8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(ffn_b1_i8_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return e;
}

cudaError_t launch_ffn_b1_i8(const B1Params& p, int grid, size_t smem, cudaStream_t s) {
  return launch_pdl(ffn_b1_i8_kernel, dim3(grid), dim3(QT), smem, s, p);
}

cudaError_t launch_quantize_rows(const void* src_bf16, int8_t* dst, float* scale, int rows, int cols,
                                 cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  quantize_rows_kernel<<<rows, 256, 0, s>>>(static_cast<const uint16_t*>(src_bf16), dst, scale, cols);
  return cudaGetLastError();
}

}  // namespace sffn
