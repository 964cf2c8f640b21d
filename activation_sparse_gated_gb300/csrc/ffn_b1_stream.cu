// ffn_b1_stream.cu -- fused single-token gate-first sparse FFN (standard or
// low-rank gate), streaming form.
//
// The method ("Model casting: compute the gate, then skip most of the FFN",
// sections "What an FFN actually computes" and "The 3x ceiling, and why W1 is
// always on"): compute the whole gate z, keep S = {i : z_i > 0}, and for those
// units only read row i of W3 and column i of W2 (row i of W2^T):
//     y = sum_{i in S} W2^T[i, :] * A(z_i) * (W3[i, :] . x).
// Standard gate: z = W1 x.  Low-rank gate ("LoPA Gating: moving the ceiling"):
// z = U t with t = V x computed in fp32 by the preceding kernel (lopa_t.cu).
//
// GB300 mapping.  A call moves tens of MB in a few microseconds and consecutive
// calls are stream-ordered, so what counts is how much of a call's weight
// traffic happens before it may start (the dependency wait) and how short the
// chain of dependent memory round trips after its gate is.
//   * The kernel is light (384 threads, <= 64 registers, ~100 KB of shared
//     memory) so the next call's blocks, launched early by programmatic
//     dependent launch, co-reside with this call's and prefetch their gate
//     rows while this call finishes.
//   * Before the wait, a block copies the first rows of its gate slice into
//     shared memory (16-byte cp.async, ~96 KB, the whole slice for the
//     low-rank gate) and every warp requests the first pieces of one more row
//     into registers.  After the wait, once the shared rows are consumed, the
//     rest of the slice is copied into the freed area in as few batches as
//     possible (one round trip each) while warps finish their register rows.
//   * A live unit goes on the block's list (shared atomic counter: the
//     compaction) and its W3 and W2^T rows are prefetched into L2 at once.
//   * After the gate: the live units' W3 rows are copied into the now free
//     shared area while every warp requests its W2^T slices of them -- one
//     round trip; h_i = A(z_i) (W3[i,:] . x) from shared memory; warp w then
//     folds its own slice of y over the list in registers (no atomics).
//   * Blocks add their partial y into one of four fp32 accumulator copies
//     (fewer blocks per address) with 128-bit atomics and end; a small
//     finalize kernel chained behind (finalize.cu) sums the copies, rounds y,
//     clears the copies and publishes the count.  That is one kernel boundary
//     instead of a fence, a ticket and a serial last block.
// There are no spin-waits in this kernel.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace sffn {

namespace {

constexpr int SW = 12;          // warps per block (two blocks and a finalize block fit an SM)
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

// L2 prefetch of a row by nl lanes (lane j of them), one 128-byte line per
// lane per step (plain prefetch instructions, no copy-engine operation per row).
__device__ __forceinline__ void prefetch_row_l2(const void* row, uint32_t bytes, int j, int nl) {
  const char* b = static_cast<const char*>(row);
  for (uint32_t off = (uint32_t)j * 128u; off < bytes; off += (uint32_t)nl * 128u)
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
      E::unpack(lds16(xs + c), xf);
#pragma unroll
      for (int v = 0; v < VPC; v += 2) {
        a0 = fmaf(wf[v], xf[v], a0);
        a1 = fmaf(wf[v + 1], xf[v + 1], a1);
      }
    }
  }
  return a0 + a1;
}

// One 16-byte gate chunk c dotted with the fp32 low-rank vector t.
template <typename E>
__device__ __forceinline__ void dot_chunk_t(const uint4& w, const float* ts, int c, float& a0, float& a1) {
  constexpr int VPC = E::VPC;
  float wf[VPC];
  E::unpack(w, wf);
  const float4* t4 = reinterpret_cast<const float4*>(ts + c * VPC);
#pragma unroll
  for (int v = 0; v < VPC; v += 4) {
    const float4 tv = t4[v / 4];
    a0 = fmaf(wf[v], tv.x, a0);
    a1 = fmaf(wf[v + 1], tv.y, a1);
    a0 = fmaf(wf[v + 2], tv.z, a0);
    a1 = fmaf(wf[v + 3], tv.w, a1);
  }
}

template <typename E>
__device__ __forceinline__ float dot_piece_t(const uint4 (&w)[PIECE], const float* ts, int pc, int lane,
                                             int nch) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int k = 0; k < PIECE; ++k) {
    const int c = pc * 32 * PIECE + lane + 32 * k;
    if (c < nch) dot_chunk_t<E>(w[k], ts, c, a0, a1);
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

// EXT: the options of the full low-rank gate, the smooth gate or a live
// threshold are in use.  The plain instantiation keeps the hot loops free of
// their registers (the kernel runs at its register cap).
template <typename T, bool LOPA, bool EXT>
__global__ void __launch_bounds__(ST, 2) ffn_b1_stream_kernel(const B1Params p) {
  using E = Elt<T>;
  constexpr int VPC = E::VPC;
  extern __shared__ __align__(16) uint8_t smem[];
  const int D = p.D;
  const int nch = D * E::BYTES / 16;          // 16-byte chunks of a D-row (x, W3, W2^T)
  const int nchg = p.gate_k * E::BYTES / 16;  // ... of a gate row (W1 or U)
  const int npg = (nchg + 32 * PIECE - 1) / (32 * PIECE);
  const int row0 = (int)(((long long)blockIdx.x * p.H) / gridDim.x);
  const int row1 = (int)(((long long)(blockIdx.x + 1) * p.H) / gridDim.x);
  const int cap = p.rows_cap;  // >= units of this block
  // shared: x | t (low-rank gate) | live list (unit, A(z), h) | counters | prefetch / gather area
  uint8_t* sp = smem;
  uint4* xs = reinterpret_cast<uint4*>(sp);
  sp += align16((size_t)nch * 16);
  float* ts = reinterpret_cast<float*>(sp);
  sp += LOPA ? align16((size_t)p.gate_k * 4) : 0;
  int* l_unit = reinterpret_cast<int*>(sp);
  float* l_a = reinterpret_cast<float*>(l_unit + cap);
  float* l_h = l_a + cap;
  int* misc = reinterpret_cast<int*>(l_h + cap);  // 0: live count, 2..3: RMSNorm scratch
  uint8_t* l_mask = reinterpret_cast<uint8_t*>(misc + 4);  // live flag of every unit of the block
  sp += align16((size_t)cap * 13 + 16);
  uint4* srows = reinterpret_cast<uint4*>(sp);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint4* G = static_cast<const uint4*>(p.gate_w);
  const uint4* W3 = static_cast<const uint4*>(p.W3);
  const uint4* W2t = static_cast<const uint4*>(p.W2t);

  if (tid == 0) {
    pdl_launch_dependents();
    misc[0] = 0;
  }

  // ---- Gate rows of the block, in three parts:
  //   [0, R)             copied into the shared area before the dependency wait;
  //   [R, R + nreg)      one row per warp, streamed as pieces through two
  //                      register buffers, the first two requested before the wait;
  //   [R + nreg, nrows)  copied into the shared area in batches of up to R rows
  //                      once the first part has been consumed (one round trip
  //                      per batch instead of one per piece).
  // Weights never depend on earlier kernels; x is prefetched into L2, which is
  // harmless whatever the previous kernel does to it.
  const int nrows = row1 - row0;
  const int R = min(p.pref_rows, nrows);
  const int nreg = max(0, min(SW, nrows - R));
  auto copy_rows = [&](int first, int n) {  // rows [first, first + n) of the slice -> shared area
    const uint4* src = G + (size_t)(row0 + first) * nchg;
    for (int i = tid; i < n * nchg; i += ST) cp_async16(srows + i, src + i);
    cp_async_commit();
  };
  copy_rows(0, R);
  const int n_seq = warp < nreg ? npg : 0;
  const uint4* my_row = G + (size_t)(row0 + R + warp) * nchg;
  uint4 wa[PIECE], wb[PIECE];
  if (n_seq > 0) load_piece(wa, my_row, 0, lane, nchg);
  if (n_seq > 1) load_piece(wb, my_row, 1, lane, nchg);
  if (tid == 0) prefetch_l2(p.x, (uint32_t)nch * 16u);

  pdl_wait();  // x, t, the outputs and the accumulators follow stream order
  for (int i = tid; i < nch; i += ST) xs[i] = __ldcg(static_cast<const uint4*>(p.x) + i);
  if constexpr (LOPA) {
    for (int i = tid; i < p.gate_k / 4; i += ST)
      reinterpret_cast<float4*>(ts)[i] = __ldcg(reinterpret_cast<const float4*>(p.t) + i);
  }
  cp_async_wait_all();
  __syncthreads();
  if constexpr (LOPA && EXT) {
    if (p.flags & FLAG_RMSNORM) rmsnorm_shared(ts, 1, p.gate_k, reinterpret_cast<float*>(misc + 2), ST);
  }

  // z of unit q is known to lanes [j0, j0 + nl) of the warp (identical in each);
  // this lane is lane j of them
  auto decide = [&](int q, float z, int j, int nl) {
    if constexpr (LOPA && EXT) {
      if (p.flags & FLAG_TILED_G) z += staged_elem<T>(xs, q % D);  // (G x)_q = x_{q mod D}
    }
    bool live;
    float a;
    if constexpr (EXT) {
      a = activation(p.act, z);
      live = is_live(a, p.thr);
    } else {  // ReLU or R-S+, threshold 0: live iff z > 0
      live = z > 0.f;
      a = live ? activation(p.act, z) : 0.f;
    }
    if (j == 0) {
      l_mask[q - row0] = live ? 1 : 0;  // written out once at the end
      if (live) {  // compaction: append to the block's live list
        const int j = atomicAdd(misc, 1);
#ifdef SFFN_DEBUG
        if (j >= cap) {  // debug builds: the list capacity is checked
          atomicOr(p.ctrl + CTRL_ERR, DEV_ERR_CHECK);
          return;
        }
#endif
        l_unit[j] = q;
        l_a[j] = a;
      }
    }
    if (live) {  // both gathered rows of the unit start moving into L2 now
      prefetch_row_l2(W3 + (size_t)q * nch, (uint32_t)nch * 16u, j, nl);
      prefetch_row_l2(W2t + (size_t)q * nch, (uint32_t)nch * 16u, j, nl);
    }
  };
  // z for n rows of the shared area, the first being slice row `first`
  auto shared_rows = [&](int first, int n) {
    if constexpr (LOPA) {
      // Low-rank gate rows are short (r values): a warp per row would spend
      // most of its time in the five-step sum and the per-row decision.  Here
      // 8 lanes share a row and a warp takes four rows at a time: the groups
      // read the same chunks of t (one broadcast), the sum takes three steps
      // and the four decisions run side by side.
      const int g = lane >> 3, j = lane & 7;
      for (int i0 = warp * 4; i0 < n; i0 += SW * 4) {
        const int i = i0 + g;
        float a0 = 0.f, a1 = 0.f;
        if (i < n) {
          const uint4* r = srows + (size_t)i * nchg;
          for (int c = j; c < nchg; c += 8) dot_chunk_t<E>(lds16(r + c), ts, c, a0, a1);
        }
        float z = a0 + a1;
        z += __shfl_xor_sync(0xffffffffu, z, 4);
        z += __shfl_xor_sync(0xffffffffu, z, 2);
        z += __shfl_xor_sync(0xffffffffu, z, 1);
        if (i < n) decide(row0 + first + i, z, j, 8);
      }
    } else {
      for (int i = warp; i < n; i += SW) {
        const uint4* r = srows + (size_t)i * nchg;
        float a0 = 0.f, a1 = 0.f;
        for (int c = lane; c < nchg; c += 32) {
          float wf[VPC], xf[VPC];
          E::unpack(lds16(r + c), wf);
          E::unpack(lds16(xs + c), xf);
#pragma unroll
          for (int v = 0; v < VPC; v += 2) {
            a0 = fmaf(wf[v], xf[v], a0);
            a1 = fmaf(wf[v + 1], xf[v + 1], a1);
          }
        }
        decide(row0 + first + i, warp_sum(a0 + a1), lane, 32);
      }
    }
  };
  shared_rows(0, R);
  __syncthreads();  // the shared area is free again
  int next = R + nreg;
  int nb1 = min(R, nrows - next);
  if (nb1 > 0) copy_rows(next, nb1);

  // the register-streamed row of this warp (its first pieces landed before the wait)
  float acc = 0.f;
  auto consume = [&](const uint4(&w)[PIECE], int pc) {
    if constexpr (LOPA)
      acc += dot_piece_t<E>(w, ts, pc, lane, nchg);
    else
      acc += dot_piece<E>(w, xs, pc, lane, nchg);
    if (pc == npg - 1) {
      const float z = warp_sum(acc);
      acc = 0.f;
      decide(row0 + R + warp, z, lane, 32);
    }
  };
  for (int pc = 0; pc < n_seq; pc += 2) {
    consume(wa, pc);
    if (pc + 2 < n_seq) load_piece(wa, my_row, pc + 2, lane, nchg);
    if (pc + 1 < n_seq) {
      consume(wb, pc + 1);
      if (pc + 3 < n_seq) load_piece(wb, my_row, pc + 3, lane, nchg);
    }
  }
  // the remaining rows, a shared-area batch at a time
  while (nb1 > 0) {
    cp_async_wait_all();
    __syncthreads();
    shared_rows(next, nb1);
    __syncthreads();
    next += nb1;
    nb1 = min(R, nrows - next);
    if (nb1 > 0) copy_rows(next, nb1);
  }
  __syncthreads();
  const int n_live = min(misc[0], cap);
#ifdef SFFN_DEBUG
  // debug builds: every listed unit must belong to this block's slice; one that
  // does not is recorded and replaced by a unit of the slice with A(z) = 0, so
  // it contributes nothing
  for (int i = tid; i < n_live; i += ST)
    if (l_unit[i] < row0 || l_unit[i] >= row1) {
      atomicOr(p.ctrl + CTRL_ERR, DEV_ERR_CHECK);
      l_unit[i] = row0;
      l_a[i] = 0.f;
    }
  __syncthreads();
#endif

  // ---- gathers (both rows of every live unit were prefetched into L2), in as
  // few round trips as possible.  Warp w owns chunks [cs0, cs0 + cs_n) of y,
  // lane l chunk cs0 + l and, when a slice is wider than 32 chunks (a row has
  // at most 512 chunks, so a slice at most 43), chunk cs0 + 32 + l in a second
  // pass.  Per batch of up to RB live units: their W3 rows are copied into
  // the (now free) shared area while every warp requests its W2^T slices of the
  // first eight units of the batch; then h = A(z) (W3 . x) from shared memory,
  // and y_slice += h W2^T[unit, slice] in registers.
  const int per = (nch + SW - 1) / SW;
  const int cs0 = warp * per;
  const int cs_n = min(per, nch - cs0);  // may be <= 0 for tiny D
  const bool owns = lane < cs_n;
  const uint4* col = W2t + cs0 + lane;
  const int RB = p.gather_rows;
  float yr[VPC];
#pragma unroll
  for (int v = 0; v < VPC; ++v) yr[v] = 0.f;
  auto fma_slice = [&](const uint4& wv, float h) {
    float wf[VPC];
    E::unpack(wv, wf);
#pragma unroll
    for (int v = 0; v < VPC; ++v) yr[v] = fmaf(h, wf[v], yr[v]);
  };
  uint4 r8[8];  // W2^T slices in flight
  for (int b0 = 0; b0 < n_live; b0 += RB) {
    const int nb = min(RB, n_live - b0);
    for (int i = tid; i < nb * nch; i += ST) {
      const int u = i / nch, c = i - u * nch;
      cp_async16(srows + i, W3 + (size_t)l_unit[b0 + u] * nch + c);
    }
    cp_async_commit();
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
        E::unpack(lds16(r + c), wf);
        E::unpack(lds16(xs + c), xf);
#pragma unroll
        for (int v = 0; v < VPC; v += 2) {
          a0 = fmaf(wf[v], xf[v], a0);
          a1 = fmaf(wf[v + 1], xf[v + 1], a1);
        }
      }
      const float uval = warp_sum(a0 + a1);
      if (lane == 0)
        l_h[b0 + u] = l_a[b0 + u] * ((EXT && (p.flags & FLAG_DOUBLE_ACT)) ? activation(p.act, uval) : uval);
    }
    __syncthreads();
    if (owns) {
#pragma unroll
      for (int m = 0; m < 8; ++m)
        if (m < nb) fma_slice(r8[m], l_h[b0 + m]);
      // the rest of the batch in predicated rounds of four loads in flight (a
      // block with many live units sets the pace of the whole call)
      for (int j = 8; j < nb; j += 4) {
#pragma unroll
        for (int m = 0; m < 4; ++m)
          r8[m] = j + m < nb ? ld_stream(col + (size_t)l_unit[b0 + j + m] * nch) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          if (j + m < nb) fma_slice(r8[m], l_h[b0 + j + m]);
      }
    }
    __syncthreads();  // the shared area is reused by the next batch
  }
  // into accumulator copy (block mod YACC_COPIES): fewer blocks per address
  float* yc = p.yacc + (size_t)(blockIdx.x % YACC_COPIES) * D;
  if (n_live > 0 && owns) {
#pragma unroll
    for (int v = 0; v < VPC; v += 4)
      atomicAdd(reinterpret_cast<float4*>(yc + (size_t)(cs0 + lane) * VPC + v),
                make_float4(yr[v], yr[v + 1], yr[v + 2], yr[v + 3]));
  }
  // second chunk of the lane when the slice is wider than 32 chunks (every h is known now)
  if (n_live > 0 && lane + 32 < cs_n) {
#pragma unroll
    for (int v = 0; v < VPC; ++v) yr[v] = 0.f;
    const uint4* col2 = col + 32;
    for (int j = 0; j < n_live; j += 8) {
#pragma unroll
      for (int m = 0; m < 8; ++m)
        r8[m] = j + m < n_live ? ld_stream(col2 + (size_t)l_unit[j + m] * nch) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int m = 0; m < 8; ++m)
        if (j + m < n_live) fma_slice(r8[m], l_h[j + m]);
    }
#pragma unroll
    for (int v = 0; v < VPC; v += 4)
      atomicAdd(reinterpret_cast<float4*>(yc + (size_t)(cs0 + 32 + lane) * VPC + v),
                make_float4(yr[v], yr[v + 1], yr[v + 2], yr[v + 3]));
  }
  // the block's live count; the finalize kernel that follows in the stream
  // sums the accumulator copies once every block has finished (kernel
  // completion orders all of these atomics before it)
  if (tid == 0 && n_live > 0) atomicAdd(p.ctrl + CTRL_COUNT + p.count_slot, n_live);
  if (p.mask)  // the block's live flags, one coalesced store (a byte store per gate row stalls the gate)
    for (int i = tid; i < nrows; i += ST) p.mask[row0 + i] = l_mask[i];
}

}  // namespace

StreamPlan plan_ffn_b1_stream(int D, int gate_k, int elt_bytes, bool lopa, int rows_cap) {
  StreamPlan pl;
  const size_t grow = (size_t)gate_k * elt_bytes, row = (size_t)D * elt_bytes;
  // Two blocks per SM (the next call's blocks prefetch while this call runs):
  // at most 110 KB per block.  The shared area holds up to 96 KB of gate rows
  // before the wait and then a gather batch of up to 16 W3 rows (a block with
  // more live units than fit pays another round trip per further batch).
  const size_t fixed = align16((size_t)D * elt_bytes) + (lopa ? align16((size_t)gate_k * 4) : 0) +
                       align16((size_t)rows_cap * 13 + 16);
  const size_t budget = 110u * 1024u;
  const size_t free_area = budget > fixed ? budget - fixed : 0;
  pl.pref_rows = (int)std::max<size_t>(1, std::min<size_t>((size_t)rows_cap,
                                                           std::min<size_t>(96u * 1024u, free_area) / grow));
  const size_t g = std::max<size_t>(1, std::min<size_t>(std::min(rows_cap, 16), free_area / row));
  const size_t area = std::max((size_t)pl.pref_rows * grow, g * row);
  pl.gather_rows = (int)std::max<size_t>(1, area / row);
  pl.smem = fixed + area;
  return pl;
}

cudaError_t ffn_b1_stream_prepare(size_t max_smem) {
  void (*ks[8])(const B1Params) = {
      ffn_b1_stream_kernel<float, false, false>,    ffn_b1_stream_kernel<float, true, false>,
      ffn_b1_stream_kernel<bf16_tag, false, false>, ffn_b1_stream_kernel<bf16_tag, true, false>,
      ffn_b1_stream_kernel<float, false, true>,     ffn_b1_stream_kernel<float, true, true>,
      ffn_b1_stream_kernel<bf16_tag, false, true>,  ffn_b1_stream_kernel<bf16_tag, true, true>};
  for (auto k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int ffn_b1_stream_threads() { return ST; }

cudaError_t launch_ffn_b1_stream(const B1Params& p, int dtype, bool lopa, int grid, size_t smem,
                                 cudaStream_t s) {
  const dim3 g(grid), b(ST);
  const bool ext = p.flags != 0 || p.act == ACT_SILU || p.thr != 0.f;
  if (dtype == 0) {
    if (ext)
      return lopa ? launch_pdl(ffn_b1_stream_kernel<float, true, true>, g, b, smem, s, p)
                  : launch_pdl(ffn_b1_stream_kernel<float, false, true>, g, b, smem, s, p);
    return lopa ? launch_pdl(ffn_b1_stream_kernel<float, true, false>, g, b, smem, s, p)
                : launch_pdl(ffn_b1_stream_kernel<float, false, false>, g, b, smem, s, p);
  }
  if (ext)
    return lopa ? launch_pdl(ffn_b1_stream_kernel<bf16_tag, true, true>, g, b, smem, s, p)
                : launch_pdl(ffn_b1_stream_kernel<bf16_tag, false, true>, g, b, smem, s, p);
  return lopa ? launch_pdl(ffn_b1_stream_kernel<bf16_tag, true, false>, g, b, smem, s, p)
              : launch_pdl(ffn_b1_stream_kernel<bf16_tag, false, false>, g, b, smem, s, p);
}

}  // namespace sffn
