// ffn_batch.cu -- gate-first sparse FFN for a small batch of tokens (2..8 per
// pass), standard or low-rank gate.
//
// Per token b the method is unchanged ("Model casting: compute the gate, then
// skip most of the FFN", section "What an FFN actually computes"):
//     y_b = sum_{i : z_bi > 0} W2^T[i, :] * A(z_bi) * (W3[i, :] . x_b).
// A batch shares the weights, so a block reads each gate row once and dots it
// with all tokens, and reads the W3 / W2^T rows of a unit once for every token
// that needs it: the union of the tokens' live sets (the pages note that
// batching erodes the win -- the union grows like 1 - s^B).
//
// Layout and flow follow the single-token streaming kernel (ffn_b1_stream.cu):
// one block per SM owning a slice of units, the head of the gate slice copied
// into shared memory before the dependency wait, the rest streamed as pieces
// through two register buffers, union units compacted into a block list with
// per-token A(z) (zero where the token's gate is dead), their W3 rows gathered
// through shared memory and their W2^T slices folded by the warp that owns the
// slice, per token, in registers.  Per-token partial sums go to four fp32
// accumulator copies; the finalize kernel chained behind sums them, rounds y
// and publishes the per-token live counts.  CUDA cores only: up to 8 tokens the gate is cheap
// next to its weight stream.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace sffn {

namespace {

constexpr int BW = 16;       // warps per block
constexpr int BT = BW * 32;  // threads per block
constexpr int BPC = 4;       // 16-byte chunks per lane per piece

__host__ __device__ constexpr size_t al16(size_t v) { return (v + 15) & ~size_t(15); }

__device__ __forceinline__ uint4 ldnc(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void cpa16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cpa_wait() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void pf_row(const void* row, uint32_t bytes, int lane) {
  const char* b = static_cast<const char*>(row);
  for (uint32_t off = (uint32_t)lane * 128u; off < bytes; off += 32u * 128u)
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(b + off));
}

__device__ __forceinline__ void load_pc(uint4 (&w)[BPC], const uint4* row, int pc, int lane, int nch) {
#pragma unroll
  for (int k = 0; k < BPC; ++k) {
    const int c = pc * 32 * BPC + lane + 32 * k;
    w[k] = (c < nch) ? ldnc(row + c) : make_uint4(0, 0, 0, 0);
  }
}

// acc[b] += chunk c of a gate/W3 row . token b's vector, for b < nb.
// Standard gate and W3 rows: the vector is x_b (stored dtype, chunk-aligned).
// Low-rank gate: the vector is t_b (fp32, r values per token).
template <typename E, int NB, bool FP32VEC>
__device__ __forceinline__ void chunk_dot_all(const uint4& w, const uint4* xs, const float* ts, int nchv,
                                              int kv, int c, int nb, float (&acc)[NB]) {
  constexpr int VPC = E::VPC;
  float wf[VPC];
  E::unpack(w, wf);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (b < nb) {
      if constexpr (FP32VEC) {
        const float4* t4 = reinterpret_cast<const float4*>(ts + (size_t)b * kv + c * VPC);
#pragma unroll
        for (int v = 0; v < VPC; v += 4) {
          const float4 tv = t4[v / 4];
          acc[b] = fmaf(wf[v], tv.x, acc[b]);
          acc[b] = fmaf(wf[v + 1], tv.y, acc[b]);
          acc[b] = fmaf(wf[v + 2], tv.z, acc[b]);
          acc[b] = fmaf(wf[v + 3], tv.w, acc[b]);
        }
      } else {
        float xf[VPC];
        E::unpack(xs[(size_t)b * nchv + c], xf);
#pragma unroll
        for (int v = 0; v < VPC; ++v) acc[b] = fmaf(wf[v], xf[v], acc[b]);
      }
    }
  }
}

template <typename T, bool LOPA, int NB>
__global__ void __launch_bounds__(BT, 1) ffn_batch_kernel(const B1Params p, int nb) {
  using E = Elt<T>;
  constexpr int VPC = E::VPC;
  extern __shared__ __align__(16) uint8_t smem[];
  const int D = p.D;
  const int nch = D * E::BYTES / 16;
  const int nchg = p.gate_k * E::BYTES / 16;
  const int npg = (nchg + 32 * BPC - 1) / (32 * BPC);
  const int row0 = (int)(((long long)blockIdx.x * p.H) / gridDim.x);
  const int row1 = (int)(((long long)(blockIdx.x + 1) * p.H) / gridDim.x);
  const int cap = p.rows_cap;
  // shared: x[nb] | t[nb] (low-rank) | list: unit, A(z)[NB], h[NB] | counters | prefetch/gather area
  uint8_t* sp = smem;
  uint4* xs = reinterpret_cast<uint4*>(sp);
  sp += al16((size_t)NB * nch * 16);
  float* ts = reinterpret_cast<float*>(sp);
  sp += LOPA ? al16((size_t)NB * p.gate_k * 4) : 0;
  int* l_unit = reinterpret_cast<int*>(sp);
  float* l_a = reinterpret_cast<float*>(l_unit + cap);  // [cap][NB]
  float* l_h = l_a + (size_t)cap * NB;                  // [cap][NB]
  int* misc = reinterpret_cast<int*>(l_h + (size_t)cap * NB);  // 0: list, 1: last, 2..: per-token counts
  float* rms_scale = reinterpret_cast<float*>(misc + 2 + NB);  // [NB] RMSNorm scratch
  uint8_t* l_mask = reinterpret_cast<uint8_t*>(rms_scale + NB);  // [rows][NB] live flags
  sp += al16((size_t)cap * (4 + 8 * NB) + 4 * (2 + 2 * NB) + (size_t)cap * NB);
  uint4* srows = reinterpret_cast<uint4*>(sp);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint4* G = static_cast<const uint4*>(p.gate_w);
  const uint4* W3 = static_cast<const uint4*>(p.W3);
  const uint4* W2t = static_cast<const uint4*>(p.W2t);

  if (tid == 0) pdl_launch_dependents();
  if (tid < 2 + NB) misc[tid] = 0;

  // ---- before the dependency wait: head of the gate slice into shared memory,
  // first two pieces of every warp's streamed rows into registers
  const int nrows = row1 - row0;
  const int R = min(p.pref_rows, nrows);
  {
    const uint4* src = G + (size_t)row0 * nchg;
    for (int i = tid; i < R * nchg; i += BT) cpa16(srows + i, src + i);
    cpa_commit();
  }
  const int my_rows = (nrows - R - warp + BW - 1) / BW;
  const int n_seq = my_rows > 0 ? my_rows * npg : 0;
  auto seq_row = [&](int s) { return G + (size_t)(row0 + R + warp + (s / npg) * BW) * nchg; };
  uint4 wa[BPC], wb[BPC];
  if (n_seq > 0) load_pc(wa, seq_row(0), 0, lane, nchg);
  if (n_seq > 1) load_pc(wb, seq_row(1), 1 % npg, lane, nchg);

  pdl_wait();
  for (int i = tid; i < nb * nch; i += BT) xs[i] = __ldcg(static_cast<const uint4*>(p.x) + i);
  if constexpr (LOPA) {
    for (int i = tid; i < nb * p.gate_k / 4; i += BT)
      reinterpret_cast<float4*>(ts)[i] = __ldcg(reinterpret_cast<const float4*>(p.t) + i);
  }
  cpa_wait();
  __syncthreads();
  if constexpr (LOPA) {
    if (p.flags & FLAG_RMSNORM) rmsnorm_shared(ts, nb, p.gate_k, rms_scale, BT);
  }

  // a unit is kept if any token's gate is live; dead tokens get A(z) = 0
  auto decide = [&](int q, const float (&z0)[NB]) {
    float z[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      z[b] = z0[b];
      if constexpr (LOPA) {
        if ((p.flags & FLAG_TILED_G) && b < nb) z[b] += staged_elem<T>(xs + (size_t)b * nch, q % D);
      }
    }
    float av[NB];  // A(z), zero where the token's unit is dead
    bool lv[NB];
    bool any = false;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      av[b] = b < nb ? activation(p.act, z[b]) : 0.f;
      lv[b] = b < nb && is_live(av[b], p.thr);
      if (!lv[b]) av[b] = 0.f;
      any |= lv[b];
    }
    if (lane == 0) {
#pragma unroll
      for (int b = 0; b < NB; ++b) l_mask[(size_t)(q - row0) * NB + b] = lv[b] ? 1 : 0;  // written out at the end
      if (any) {
        const int j = atomicAdd(misc, 1);
        l_unit[j] = q;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          l_a[(size_t)j * NB + b] = av[b];
          if (lv[b]) atomicAdd(misc + 2 + b, 1);
        }
      }
    }
    if (any) {
      pf_row(W3 + (size_t)q * nch, (uint32_t)nch * 16u, lane);
      pf_row(W2t + (size_t)q * nch, (uint32_t)nch * 16u, lane);
    }
  };
  // gate rows in shared memory
  for (int i = warp; i < R; i += BW) {
    const uint4* r = srows + (size_t)i * nchg;
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
    for (int c = lane; c < nchg; c += 32) chunk_dot_all<E, NB, LOPA>(r[c], xs, ts, nch, p.gate_k, c, nb, acc);
    float z[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) z[b] = warp_sum(acc[b]);
    decide(row0 + i, z);
  }
  // streamed gate rows
  float acc[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) acc[b] = 0.f;
  auto consume = [&](const uint4(&w)[BPC], int s) {
    const int pc = s % npg;
#pragma unroll
    for (int k = 0; k < BPC; ++k) {
      const int c = pc * 32 * BPC + lane + 32 * k;
      if (c < nchg) chunk_dot_all<E, NB, LOPA>(w[k], xs, ts, nch, p.gate_k, c, nb, acc);
    }
    if (pc == npg - 1) {
      float z[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        z[b] = warp_sum(acc[b]);
        acc[b] = 0.f;
      }
      decide(row0 + R + warp + (s / npg) * BW, z);
    }
  };
  for (int s = 0; s < n_seq; s += 2) {
    consume(wa, s);
    if (s + 2 < n_seq) load_pc(wa, seq_row(s + 2), (s + 2) % npg, lane, nchg);
    if (s + 1 < n_seq) {
      consume(wb, s + 1);
      if (s + 3 < n_seq) load_pc(wb, seq_row(s + 3), (s + 3) % npg, lane, nchg);
    }
  }
  __syncthreads();
  const int n_list = misc[0];

  // ---- gathers: W3 rows of a batch of units through shared memory
  // (h_bj = A(z_bj) (W3[unit_j, :] . x_b)), then per-token W2^T slices folded
  // by the warp that owns the slice (warp w: chunks [cs0, cs0 + cs_n), lane l
  // chunk cs0 + l), tokens in groups of four to bound registers.
  const int per = (nch + BW - 1) / BW;
  const int cs0 = warp * per;
  const int cs_n = min(per, nch - cs0);
  const bool owns = lane < cs_n;
  const uint4* col = W2t + cs0 + lane;
  const int RB = p.gather_rows;
  constexpr int TG = NB < 4 ? NB : 4;
  float yr[NB][VPC];
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int v = 0; v < VPC; ++v) yr[b][v] = 0.f;
  for (int b0 = 0; b0 < n_list; b0 += RB) {
    const int nbat = min(RB, n_list - b0);
    for (int i = tid; i < nbat * nch; i += BT) {
      const int u = i / nch, c = i - u * nch;
      cpa16(srows + i, W3 + (size_t)l_unit[b0 + u] * nch + c);
    }
    cpa_commit();
    cpa_wait();
    __syncthreads();
    for (int u = warp; u < nbat; u += BW) {
      const uint4* r = srows + (size_t)u * nch;
      float a2[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) a2[b] = 0.f;
      for (int c = lane; c < nch; c += 32) chunk_dot_all<E, NB, false>(r[c], xs, nullptr, nch, 0, c, nb, a2);
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float uval = warp_sum(a2[b]);
        if (lane == 0)
          l_h[(size_t)(b0 + u) * NB + b] =
              l_a[(size_t)(b0 + u) * NB + b] * ((p.flags & FLAG_DOUBLE_ACT) ? activation(p.act, uval) : uval);
      }
    }
    __syncthreads();
    if (owns) {
      // eight slice loads in flight, then their FMAs
      for (int j0 = 0; j0 < nbat; j0 += 8) {
        uint4 r[8];
#pragma unroll
        for (int m = 0; m < 8; ++m)
          r[m] = (j0 + m < nbat) ? ldnc(col + (size_t)l_unit[b0 + j0 + m] * nch) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          if (j0 + m < nbat) {
            float wf[VPC];
            E::unpack(r[m], wf);
            const float* hj = l_h + (size_t)(b0 + j0 + m) * NB;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              const float h = hj[b];
#pragma unroll
              for (int v = 0; v < VPC; ++v) yr[b][v] = fmaf(h, wf[v], yr[b][v]);
            }
          }
        }
      }
    }
    __syncthreads();  // shared area reused by the next batch
  }
  (void)TG;
  if (n_list > 0 && owns) {
    const int cp = blockIdx.x % YACC_COPIES;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b < nb) {
        float* yc = p.yacc + ((size_t)b * YACC_COPIES + cp) * D + (size_t)(cs0 + lane) * VPC;
#pragma unroll
        for (int v = 0; v < VPC; v += 4)
          atomicAdd(reinterpret_cast<float4*>(yc + v),
                    make_float4(yr[b][v], yr[b][v + 1], yr[b][v + 2], yr[b][v + 3]));
      }
    }
  }
  // per-token live counts; the finalize kernel chained behind sums the copies
  if (tid < nb && misc[2 + tid] > 0) atomicAdd(p.ctrl + CTRL_COUNT + p.count_slot + tid, misc[2 + tid]);
  if (p.mask)  // the block's live flags, coalesced per token
    for (int i = tid; i < nb * (row1 - row0); i += BT) {
      const int b = i / (row1 - row0), u = i - b * (row1 - row0);
      p.mask[(size_t)b * p.H + row0 + u] = l_mask[(size_t)u * NB + b];
    }
}

template <typename T, bool LOPA, int NB>
cudaError_t set_attr(size_t max_smem) {
  cudaError_t e = cudaFuncSetAttribute(ffn_batch_kernel<T, LOPA, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ffn_batch_kernel<T, LOPA, NB>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return e;
}

template <typename T, bool LOPA>
cudaError_t launch_nb(const B1Params& p, int nb, int grid, size_t smem, cudaStream_t s) {
  const dim3 g(grid), b(BT);
  if (nb <= 2) return launch_pdl(ffn_batch_kernel<T, LOPA, 2>, g, b, smem, s, p, nb);
  if (nb <= 4) return launch_pdl(ffn_batch_kernel<T, LOPA, 4>, g, b, smem, s, p, nb);
  return launch_pdl(ffn_batch_kernel<T, LOPA, 8>, g, b, smem, s, p, nb);
}

}  // namespace

BatchPlan plan_ffn_batch(int D, int gate_k, int elt_bytes, bool lopa, int rows_cap, int nb_max) {
  BatchPlan pl;
  const size_t grow = (size_t)gate_k * elt_bytes, row = (size_t)D * elt_bytes;
  pl.pref_rows = (int)std::min<size_t>((size_t)rows_cap, (64u * 1024u) / grow);
  const size_t area = std::max((size_t)pl.pref_rows * grow, (size_t)std::min(rows_cap, 8) * row);
  pl.gather_rows = (int)std::max<size_t>(1, area / row);
  pl.smem = al16((size_t)nb_max * D * elt_bytes) + (lopa ? al16((size_t)nb_max * gate_k * 4) : 0) +
            al16((size_t)rows_cap * (4 + 8 * nb_max) + 4 * (2 + 2 * nb_max) + (size_t)rows_cap * nb_max) + area;
  return pl;
}

cudaError_t ffn_batch_prepare(size_t max_smem) {
  cudaError_t e;
  if ((e = set_attr<float, false, 2>(max_smem)) || (e = set_attr<float, false, 4>(max_smem)) ||
      (e = set_attr<float, false, 8>(max_smem)) || (e = set_attr<float, true, 2>(max_smem)) ||
      (e = set_attr<float, true, 4>(max_smem)) || (e = set_attr<float, true, 8>(max_smem)) ||
      (e = set_attr<bf16_tag, false, 2>(max_smem)) || (e = set_attr<bf16_tag, false, 4>(max_smem)) ||
      (e = set_attr<bf16_tag, false, 8>(max_smem)) || (e = set_attr<bf16_tag, true, 2>(max_smem)) ||
      (e = set_attr<bf16_tag, true, 4>(max_smem)) || (e = set_attr<bf16_tag, true, 8>(max_smem)))
    return e;
  return cudaSuccess;
}

cudaError_t launch_ffn_batch(const B1Params& p, int nb, int dtype, bool lopa, int grid, size_t smem,
                             cudaStream_t s) {
  if (nb < 2 || nb > 8) return cudaErrorInvalidValue;
  if (dtype == 0) return lopa ? launch_nb<float, true>(p, nb, grid, smem, s) : launch_nb<float, false>(p, nb, grid, smem, s);
  return lopa ? launch_nb<bf16_tag, true>(p, nb, grid, smem, s) : launch_nb<bf16_tag, false>(p, nb, grid, smem, s);
}

}  // namespace sffn
