// ffn_b1_stream.cu -- fused single-token gate-first sparse FFN, standard gate,
// streaming form.
//
// The method ("Model casting: compute the gate, then skip most of the FFN",
// sections "What an FFN actually computes" and "The 3x ceiling, and why W1 is
// always on"): compute the whole gate z = W1 x, keep S = {i : z_i > 0}, and for
// those units only read row i of W3 and column i of W2 (row i of W2^T):
//     y = sum_{i in S} W2^T[i, :] * A(z_i) * (W3[i, :] . x).
//
// GB300 mapping.  A call moves ~44 MB (D=2560, H=7168, 90 % sparsity) in a few
// microseconds, so fixed costs (launch gap, ramp-up, reduction tail) matter as
// much as streaming speed.  The kernel is therefore kept light -- 512 threads,
// at most 64 registers, ~15 KB of shared memory -- so that the next call's
// blocks (launched early by programmatic dependent launch) sit on the same SMs
// and start pulling their weights while this call finishes.
//   * 16 warps per block, each block owning a contiguous slice of units.  A warp
//     streams its gate rows as half-row pieces through two register buffers
//     (one piece multiplied with x from shared memory while the next is in
//     flight), so loads stay outstanding continuously instead of in waves.
//     The first pieces are requested before the dependency wait: weights
//     never depend on earlier kernels.
//   * A live unit never stalls the gate stream: lane 0 appends (unit, A(z)) to
//     the block's shared list (a shared atomic counter: the compaction) and
//     asks the copy engine to prefetch the unit's W3 row and W2^T row into L2.
//   * After the gate stream, warps take list entries and compute
//     h_i = A(z_i) (W3[i,:] . x) from L2; then every thread owns whole 16-byte
//     chunks of y and accumulates sum_i h_i W2^T[i, chunk] in registers.
//   * Blocks add their partial y into a per-handle fp32 accumulator with
//     128-bit atomics (each block starting at a different offset to spread
//     same-address traffic); the last block (ticket counter) rounds y, clears
//     the accumulator and publishes the live count.
// There are no spin-waits in this kernel.
#include "common.cuh"
#include "internal.h"

namespace sffn {

namespace {

constexpr int SW = 16;          // warps per block
constexpr int ST = SW * 32;     // threads per block
constexpr int PIECE = 5;        // 16-byte chunks per lane per piece (2.5 KB per warp for bf16)

__host__ __device__ constexpr size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// L2 prefetch of a row by a whole warp, one 128-byte line per lane per step
// (plain prefetch instructions, no copy-engine operation per row).
__device__ __forceinline__ void prefetch_row_l2(const void* row, uint32_t bytes, int lane) {
  const char* b = static_cast<const char*>(row);
  for (uint32_t off = (uint32_t)lane * 128u; off < bytes; off += 32u * 128u)
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(b + off));
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Load piece `pc` of a D-row (chunks pc*32*PIECE + lane + 32k) into registers.
__device__ __forceinline__ void load_piece(uint4 (&w)[PIECE], const uint4* row, int pc, int lane, int nch) {
#pragma unroll
  for (int k = 0; k < PIECE; ++k) {
    const int c = pc * 32 * PIECE + lane + 32 * k;
    w[k] = (c < nch) ? ld_stream(row + c) : make_uint4(0, 0, 0, 0);
  }
}

template <typename E>
__device__ __forceinline__ float dot_piece(const uint4 (&w)[PIECE], const uint4* xs, int pc, int lane,
                                           int nch) {
  constexpr int VPC = E::VPC;
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int k = 0; k < PIECE; ++k) {
    const int c = pc * 32 * PIECE + lane + 32 * k;
    if (c < nch) {
      float wf[VPC], xf[VPC];
      E::unpack(w[k], wf);
      E::unpack(xs[c], xf);
#pragma unroll
      for (int v = 0; v < VPC; v += 2) {
        a0 = fmaf(wf[v], xf[v], a0);
        a1 = fmaf(wf[v + 1], xf[v + 1], a1);
      }
    }
  }
  return a0 + a1;
}

// u = row . x over all pieces (the first piece already in `w` if `have0`)
template <typename E>
__device__ __forceinline__ float row_dot(uint4 (&w)[PIECE], const uint4* row, const uint4* xs, int lane,
                                         int nch, int npieces, bool have0) {
  float acc = 0.f;
  for (int pc = 0; pc < npieces; ++pc) {
    if (pc > 0 || !have0) load_piece(w, row, pc, lane, nch);
    acc += dot_piece<E>(w, xs, pc, lane, nch);
  }
  return warp_sum(acc);
}

template <typename T>
__global__ void __launch_bounds__(ST, 2) ffn_b1_stream_kernel(const B1Params p) {
  using E = Elt<T>;
  constexpr int VPC = E::VPC;
  extern __shared__ __align__(16) uint8_t smem[];
  const int D = p.D;
  const int nch = D * E::BYTES / 16;  // 16-byte chunks of a row
  const int npieces = (nch + 32 * PIECE - 1) / (32 * PIECE);
  const int row0 = (int)(((long long)blockIdx.x * p.H) / gridDim.x);
  const int row1 = (int)(((long long)(blockIdx.x + 1) * p.H) / gridDim.x);
  const int cap = p.rows_cap;  // >= units of this block
  // shared: x | live list (unit, A(z), h) | counters | prefetched gate rows
  uint4* xs = reinterpret_cast<uint4*>(smem);
  int* l_unit = reinterpret_cast<int*>(smem + align16((size_t)nch * 16));  // [cap]
  float* l_a = reinterpret_cast<float*>(l_unit + cap);                      // [cap]
  float* l_h = l_a + cap;                                                   // [cap]
  int* misc = reinterpret_cast<int*>(l_h + cap);  // 0: live count, 1: last-block flag
  uint4* srows = reinterpret_cast<uint4*>(smem + align16((size_t)nch * 16) + align16((size_t)cap * 12 + 16));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint4* W1 = static_cast<const uint4*>(p.gate_w);
  const uint4* W3 = static_cast<const uint4*>(p.W3);
  const uint4* W2t = static_cast<const uint4*>(p.W2t);
  float4* ya = reinterpret_cast<float4*>(p.yacc);

  if (tid == 0) {
    pdl_launch_dependents();
    misc[0] = 0;
  }

  // ---- prefetch before the dependency wait (weights never depend on earlier
  // kernels).  The block's first R rows are copied into shared memory with
  // 16-byte asynchronous copies; the rest are streamed by the warps (rows
  // row0 + R + warp + SW*k) as pieces, npieces per row, alternating between two
  // register buffers -- one piece multiplied with x while the next is in flight
  // -- and the first two pieces are requested now.  x is prefetched into L2,
  // which is harmless whatever the previous kernel does to it.
  const int nrows = row1 - row0;
  const int R = min(p.pref_rows, nrows);
  {
    const uint4* src = W1 + (size_t)row0 * nch;
    for (int i = tid; i < R * nch; i += ST) cp_async16(srows + i, src + i);
    cp_async_commit();
  }
  const int my_rows = (nrows - R - warp + SW - 1) / SW;
  const int n_seq = my_rows > 0 ? my_rows * npieces : 0;
  auto seq_row = [&](int sidx) { return W1 + (size_t)(row0 + R + warp + (sidx / npieces) * SW) * nch; };
  uint4 wa[PIECE], wb[PIECE];
  if (n_seq > 0) load_piece(wa, seq_row(0), 0, lane, nch);
  if (n_seq > 1) load_piece(wb, seq_row(1), 1 % npieces, lane, nch);
  if (tid == 0) prefetch_l2(p.x, (uint32_t)nch * 16u);

  pdl_wait();  // x, the outputs and the accumulators follow stream order
  for (int i = tid; i < nch; i += ST) xs[i] = __ldcg(static_cast<const uint4*>(p.x) + i);
  cp_async_wait_all();
  __syncthreads();

  auto decide = [&](int q, float z) {  // z identical in every lane (butterfly sum)
    const bool live = z > 0.f;
    if (lane == 0) {
      if (p.mask) p.mask[q] = live ? 1 : 0;
      if (live) {  // compaction: append to the block's live list
        const int j = atomicAdd(misc, 1);
        l_unit[j] = q;
        l_a[j] = activation(p.act, z);
      }
    }
    if (live) {  // both gathered rows of the unit start moving into L2 now
      prefetch_row_l2(W3 + (size_t)q * nch, (uint32_t)nch * 16u, lane);
      prefetch_row_l2(W2t + (size_t)q * nch, (uint32_t)nch * 16u, lane);
    }
  };
  // gate rows already in shared memory
  for (int i = warp; i < R; i += SW) {
    const uint4* r = srows + (size_t)i * nch;
    float a0 = 0.f, a1 = 0.f;
    for (int c = lane; c < nch; c += 32) {
      float wf[VPC], xf[VPC];
      E::unpack(r[c], wf);
      E::unpack(xs[c], xf);
#pragma unroll
      for (int v = 0; v < VPC; v += 2) {
        a0 = fmaf(wf[v], xf[v], a0);
        a1 = fmaf(wf[v + 1], xf[v + 1], a1);
      }
    }
    decide(row0 + i, warp_sum(a0 + a1));
  }
  // streamed gate rows
  float acc = 0.f;
  auto finish_piece = [&](int sidx) {
    if (sidx % npieces != npieces - 1) return;
    const float z = warp_sum(acc);
    acc = 0.f;
    decide(row0 + R + warp + (sidx / npieces) * SW, z);
  };
  for (int sidx = 0; sidx < n_seq; sidx += 2) {
    acc += dot_piece<E>(wa, xs, sidx % npieces, lane, nch);
    finish_piece(sidx);
    if (sidx + 2 < n_seq) load_piece(wa, seq_row(sidx + 2), (sidx + 2) % npieces, lane, nch);
    if (sidx + 1 < n_seq) {
      acc += dot_piece<E>(wb, xs, (sidx + 1) % npieces, lane, nch);
      finish_piece(sidx + 1);
      if (sidx + 3 < n_seq) load_piece(wb, seq_row(sidx + 3), (sidx + 3) % npieces, lane, nch);
    }
  }
  __syncthreads();
  const int n_live = misc[0];

  // ---- gathers (both rows of every live unit were prefetched into L2), in as
  // few round trips as possible.  Warp w owns chunks [cs0, cs0 + cs_n) of y,
  // lane l chunk cs0 + l (a slice has at most 32 chunks because a row has at
  // most 512).  Per batch of up to RB live units: their W3 rows are copied into
  // the (now free) shared prefetch area while every warp requests its W2^T
  // slices of the first eight units of the batch; then h = A(z) (W3 . x) from
  // shared memory, and y_slice += h W2^T[unit, slice] in registers.
  const int per = (nch + SW - 1) / SW;
  const int cs0 = warp * per;
  const int cs_n = min(per, nch - cs0);  // may be <= 0 for tiny D
  const bool owns = lane < cs_n;
  const uint4* col = W2t + cs0 + lane;
  const int RB = max(1, p.pref_rows);
  float yr[VPC];
#pragma unroll
  for (int v = 0; v < VPC; ++v) yr[v] = 0.f;
  auto fma_slice = [&](const uint4& wv, float h) {
    float wf[VPC];
    E::unpack(wv, wf);
#pragma unroll
    for (int v = 0; v < VPC; ++v) yr[v] = fmaf(h, wf[v], yr[v]);
  };
  for (int b0 = 0; b0 < n_live; b0 += RB) {
    const int nb = min(RB, n_live - b0);
    for (int i = tid; i < nb * nch; i += ST) {
      const int u = i / nch, c = i - u * nch;
      cp_async16(srows + i, W3 + (size_t)l_unit[b0 + u] * nch + c);
    }
    cp_async_commit();
    uint4 r8[8];
#pragma unroll
    for (int m = 0; m < 8; ++m)
      r8[m] = (owns && m < nb) ? ld_stream(col + (size_t)l_unit[b0 + m] * nch) : make_uint4(0, 0, 0, 0);
    cp_async_wait_all();
    __syncthreads();
    for (int u = warp; u < nb; u += SW) {
      const uint4* r = srows + (size_t)u * nch;
      float a0 = 0.f, a1 = 0.f;
      for (int c = lane; c < nch; c += 32) {
        float wf[VPC], xf[VPC];
        E::unpack(r[c], wf);
        E::unpack(xs[c], xf);
#pragma unroll
        for (int v = 0; v < VPC; v += 2) {
          a0 = fmaf(wf[v], xf[v], a0);
          a1 = fmaf(wf[v + 1], xf[v + 1], a1);
        }
      }
      const float uval = warp_sum(a0 + a1);
      if (lane == 0) l_h[b0 + u] = l_a[b0 + u] * uval;
    }
    __syncthreads();
    if (owns) {
#pragma unroll
      for (int m = 0; m < 8; ++m)
        if (m < nb) fma_slice(r8[m], l_h[b0 + m]);
      int j = 8;
      for (; j + 4 <= nb; j += 4) {
        uint4 r[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) r[m] = ld_stream(col + (size_t)l_unit[b0 + j + m] * nch);
#pragma unroll
        for (int m = 0; m < 4; ++m) fma_slice(r[m], l_h[b0 + j + m]);
      }
      for (; j < nb; ++j) fma_slice(ld_stream(col + (size_t)l_unit[b0 + j] * nch), l_h[b0 + j]);
    }
    __syncthreads();  // the shared area is reused by the next batch
  }
  if (n_live > 0 && owns) {
    // into accumulator copy (block mod YACC_COPIES): fewer blocks per address
    float* yc = p.yacc + (size_t)(blockIdx.x % YACC_COPIES) * D + (size_t)(cs0 + lane) * VPC;
#pragma unroll
    for (int v = 0; v < VPC; v += 4)
      atomicAdd(reinterpret_cast<float4*>(yc + v), make_float4(yr[v], yr[v + 1], yr[v + 2], yr[v + 3]));
  }
  __threadfence();
  __syncthreads();
  const int n4 = D / 4;
  if (tid == 0) {
    if (n_live > 0) atomicAdd(p.ctrl + CTRL_COUNT + p.count_slot, n_live);
    __threadfence();
    const int ticket = atomicAdd(p.ctrl + CTRL_TICKET, 1);
    misc[1] = (ticket == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (misc[1]) {
    // every other block has added its partial and taken its ticket
    __threadfence();
    // every load before any store: one L2 round trip (n4 <= 2 * ST)
    float4 c[2][YACC_COPIES];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = tid + k * ST;
#pragma unroll
      for (int r = 0; r < YACC_COPIES; ++r)
        c[k][r] = i < n4 ? __ldcg(ya + (size_t)r * n4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = tid + k * ST;
      if (i >= n4) continue;
      float4 v = c[k][0];
#pragma unroll
      for (int r = 1; r < YACC_COPIES; ++r) {
        v.x += c[k][r].x; v.y += c[k][r].y; v.z += c[k][r].z; v.w += c[k][r].w;
      }
#pragma unroll
      for (int r = 0; r < YACC_COPIES; ++r) __stcg(ya + (size_t)r * n4 + i, make_float4(0.f, 0.f, 0.f, 0.f));
      if constexpr (VPC == 4) {
        reinterpret_cast<float4*>(p.y)[i] = v;
      } else {
        reinterpret_cast<uint2*>(p.y)[i] = make_uint2(pack_bf16x2_rn(v.x, v.y), pack_bf16x2_rn(v.z, v.w));
      }
    }
    if (tid == 0) {
      // no other block touches these any more: plain loads and stores
      p.counts[0] = __ldcg(p.ctrl + CTRL_COUNT + p.count_slot);
      __stcg(p.ctrl + CTRL_COUNT + p.count_slot, 0);
      __stcg(p.ctrl + CTRL_TICKET, 0);
    }
  }
}

}  // namespace

size_t ffn_b1_stream_smem_bytes(int D, int elt_bytes, int rows_cap, int pref_rows) {
  return align16((size_t)D * elt_bytes) + align16((size_t)rows_cap * 12 + 16) +
         (size_t)pref_rows * D * elt_bytes;
}

cudaError_t ffn_b1_stream_prepare(size_t max_smem) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(ffn_b1_stream_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)max_smem)))
    return e;
  if ((e = cudaFuncSetAttribute(ffn_b1_stream_kernel<bf16_tag>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)max_smem)))
    return e;
  if ((e = cudaFuncSetAttribute(ffn_b1_stream_kernel<float>, cudaFuncAttributePreferredSharedMemoryCarveout, 100)))
    return e;
  return cudaFuncSetAttribute(ffn_b1_stream_kernel<bf16_tag>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

int ffn_b1_stream_threads() { return ST; }

cudaError_t launch_ffn_b1_stream(const B1Params& p, int dtype, int grid, cudaStream_t s) {
  const size_t smem = ffn_b1_stream_smem_bytes(p.D, dtype == 0 ? 4 : 2, p.rows_cap, p.pref_rows);
  if (dtype == 0) return launch_pdl(ffn_b1_stream_kernel<float>, dim3(grid), dim3(ST), smem, s, p);
  return launch_pdl(ffn_b1_stream_kernel<bf16_tag>, dim3(grid), dim3(ST), smem, s, p);
}

}  // namespace sffn
