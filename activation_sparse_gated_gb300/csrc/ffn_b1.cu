// ffn_b1.cu -- fused single-token gate-first sparse FFN (standard or low-rank gate).
//
// The method ("Model casting: compute the gate, then skip most of the FFN",
// sections "What an FFN actually computes" and "The 3x ceiling, and why W1 is
// always on"): compute the whole gate z, keep the live units S = {i : z_i > 0},
// and for those only read row i of W3 and column i of W2:
//     y = sum_{i in S} W2[:, i] * A(z_i) * (W3[i, :] . x).
// With the low-rank gate ("LoPA Gating: moving the ceiling") z = U t with
// t = V x computed by the preceding kernel (lopa_t.cu).
//
// GB300 mapping.  One block per SM owns a contiguous slice of hidden units.
//   warp 0 (producer)   streams the slice's gate rows (W1 or U) into a shared
//                       ring with bulk async copies; the weights do not depend
//                       on earlier kernels, so this starts before the
//                       programmatic-dependent-launch wait and overlaps the
//                       previous call's tail.
//   warps 1..8 (gate)   one gate row per warp: fp32 dot with x (or t), the
//                       activation, the live decision; a live unit takes the
//                       next gather slot and its W3 row and W2^T row (both
//                       contiguous D-element rows) are copied in at once, so
//                       gathers overlap the rest of the gate stream.  Slots are
//                       taken with a shared atomic counter: this is the
//                       compaction of the live set.
//   warps 9..12 (gather) consume slots in order: u_i = W3[i,:] . x across the
//                       group, h_i = A(z_i) u_i, and y += h_i W2^T[i, :] held in
//                       registers (each thread owns fixed 16-byte chunks of y).
// Blocks add their fp32 partial y into a per-handle accumulator with 128-bit
// vector atomics; the last block to finish (ticket counter) rounds y to the
// output dtype, clears the accumulator and publishes the live count.
#include "common.cuh"
#include "internal.h"

namespace sffn {

namespace {

struct B1Smem {
  uint64_t full1[B1_NS1_MAX];
  uint64_t empty1[B1_NS1_MAX];
  uint64_t full2[B1_NS2_MAX];
  uint64_t empty2[B1_NS2_MAX];
  uint64_t xbar;
  uint64_t gate_done;
  int issued1[B1_NS1_MAX];          // fills issued per gate-ring slot (drain on abort)
  int issued2[B1_NS2_MAX];          // fills issued per gather slot
  int2 meta[B1_NS2_MAX];            // (hidden unit, bits of A(z)) per gather slot
  float red[B1_NS2_MAX][B1_NGA];    // per-warp partial W3 dots
  int n_live;                       // gather slots taken == live units of this block
  int abort;
  int decision;
  int last;
};

__host__ __device__ constexpr size_t align128(size_t v) { return (v + 127) & ~size_t(127); }

struct Layout {
  size_t x, t, ring1, ring2, total;
};

__host__ __device__ inline Layout b1_layout(int D, int gate_k, int elt, bool lopa, int ns1, int ns2) {
  Layout L;
  L.x = align128(sizeof(B1Smem));
  L.t = L.x + align128((size_t)D * elt);
  L.ring1 = L.t + (lopa ? align128((size_t)gate_k * 4) : 0);
  L.ring2 = L.ring1 + align128((size_t)ns1 * gate_k * elt);
  L.total = L.ring2 + (size_t)ns2 * 2 * D * elt;
  return L;
}

// Drain wait used only after an abort: wait for in-flight copies to land so the
// block never exits with a bulk copy still writing its shared memory.
__device__ void drain(uint64_t* bar, int fills) {
  if (fills <= 0) return;
  const uint32_t parity = (uint32_t)(fills - 1) & 1u;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 20000000ull) break;  // 20 ms: copies of valid memory end long before
  }
}

template <typename T, bool LOPA>
__global__ void __launch_bounds__(B1_THREADS, 1) ffn_b1_kernel(const B1Params p) {
  using E = Elt<T>;
  constexpr int VPC = E::VPC;
  extern __shared__ __align__(128) uint8_t smem[];
  B1Smem& S = *reinterpret_cast<B1Smem*>(smem);

  const int D = p.D;
  const uint32_t row_bytes = (uint32_t)D * E::BYTES;        // W3 / W2^T / x rows
  const uint32_t grow_bytes = (uint32_t)p.gate_k * E::BYTES; // W1 / U rows
  const int nch = (int)(row_bytes / 16);
  const int nchg = (int)(grow_bytes / 16);
  const Layout L = b1_layout(D, p.gate_k, E::BYTES, LOPA, p.ns1, p.ns2);
  uint8_t* xs = smem + L.x;
  const float* ts = reinterpret_cast<const float*>(smem + L.t);
  uint8_t* ring1 = smem + L.ring1;
  uint8_t* ring2 = smem + L.ring2;
  const uint32_t slot2_bytes = 2 * row_bytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = (int)(((long long)blockIdx.x * p.H) / gridDim.x);
  const int row1 = (int)(((long long)(blockIdx.x + 1) * p.H) / gridDim.x);
  const int nrows = row1 - row0;
  int* err = p.ctrl + CTRL_ERR;
  volatile int* abort = &S.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.ns1; ++i) {
      mbar_init(&S.full1[i], 1);
      mbar_init(&S.empty1[i], 1);
      S.issued1[i] = 0;
    }
    for (int i = 0; i < p.ns2; ++i) {
      mbar_init(&S.full2[i], 1);
      mbar_init(&S.empty2[i], B1_NGA);
      S.issued2[i] = 0;
    }
    mbar_init(&S.xbar, 1);
    mbar_init(&S.gate_done, B1_NWG);
    S.n_live = 0;
    S.abort = 0;
    S.last = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint8_t* src = static_cast<const uint8_t*>(p.gate_w) + (size_t)row0 * grow_bytes;
      const uint64_t pol = policy_evict_first();
      for (int q = 0; q < nrows; ++q) {
        const int s = q % p.ns1;
        const int k = q / p.ns1;
        if (k > 0 && !mbar_wait(&S.empty1[s], (uint32_t)(k - 1) & 1u, abort, err, p.timeout_ns))
          break;
        mbar_arrive_expect_tx(&S.full1[s], grow_bytes);
        bulk_g2s_hint(ring1 + (size_t)s * grow_bytes, src + (size_t)q * grow_bytes, grow_bytes,
                      &S.full1[s], pol);
        S.issued1[s] = k + 1;
      }
    }
    __syncwarp();
  } else if (warp <= B1_NWG) {
    // ---------------------------------------------------------------- gate warps
    const int gw = warp - 1;
    pdl_wait();  // x, t, outputs and accumulators belong to the stream order
    if (gw == 0 && lane == 0) {
      mbar_arrive_expect_tx(&S.xbar, row_bytes + (LOPA ? (uint32_t)p.gate_k * 4u : 0u));
      bulk_g2s(xs, p.x, row_bytes, &S.xbar);
      if (LOPA) bulk_g2s(smem + L.t, p.t, (uint32_t)p.gate_k * 4u, &S.xbar);
    }
    // every wait is voted on so that the lanes of a warp leave a loop together
    bool ok = __all_sync(0xffffffffu, mbar_wait(&S.xbar, 0, abort, err, p.timeout_ns));
    for (int q = gw; ok && q < nrows; q += B1_NWG) {
      const int s = q % p.ns1;
      const bool got = mbar_wait(&S.full1[s], (uint32_t)(q / p.ns1) & 1u, abort, err, p.timeout_ns);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      const uint4* w = reinterpret_cast<const uint4*>(ring1 + (size_t)s * grow_bytes);
      float acc0 = 0.f, acc1 = 0.f;
      if constexpr (!LOPA) {
        const uint4* xv = reinterpret_cast<const uint4*>(xs);
        for (int c = lane; c < nchg; c += 32) {
          float wv[VPC], xf[VPC];
          E::unpack(w[c], wv);
          E::unpack(xv[c], xf);
#pragma unroll
          for (int v = 0; v < VPC; v += 2) {
            acc0 = fmaf(wv[v], xf[v], acc0);
            acc1 = fmaf(wv[v + 1], xf[v + 1], acc1);
          }
        }
      } else {
        const float4* tv = reinterpret_cast<const float4*>(ts);
        for (int c = lane; c < nchg; c += 32) {
          float wv[VPC];
          E::unpack(w[c], wv);
#pragma unroll
          for (int v = 0; v < VPC; v += 4) {
            const float4 t4 = tv[(c * VPC + v) >> 2];
            acc0 = fmaf(wv[v], t4.x, acc0);
            acc1 = fmaf(wv[v + 1], t4.y, acc1);
            acc0 = fmaf(wv[v + 2], t4.z, acc0);
            acc1 = fmaf(wv[v + 3], t4.w, acc1);
          }
        }
      }
      const float z = warp_sum(acc0 + acc1);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.empty1[s]);
        const int row = row0 + q;
        const bool live = z > 0.f;
        if (p.mask) p.mask[row] = live ? 1 : 0;
        if (live) {
          const int g = atomicAdd(&S.n_live, 1);
          const int s2 = g % p.ns2;
          if (mbar_wait(&S.empty2[s2], ((uint32_t)(g / p.ns2) & 1u) ^ 1u, abort, err,
                        p.timeout_ns)) {
            S.meta[s2] = make_int2(row, __float_as_int(activation(p.act, z)));
            mbar_arrive_expect_tx(&S.full2[s2], 2 * row_bytes);
            uint8_t* dst = ring2 + (size_t)s2 * slot2_bytes;
            bulk_g2s(dst, static_cast<const uint8_t*>(p.W3) + (size_t)row * row_bytes, row_bytes,
                     &S.full2[s2]);
            bulk_g2s(dst + row_bytes, static_cast<const uint8_t*>(p.W2t) + (size_t)row * row_bytes,
                     row_bytes, &S.full2[s2]);
            S.issued2[s2] = g / p.ns2 + 1;
          } else {
            ok = false;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.gate_done);
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- gather warps
    const int gt = threadIdx.x - (1 + B1_NWG) * 32;  // 0 .. 32*B1_NGA-1
    const int gwarp = gt >> 5;
    constexpr int NGT = B1_NGA * 32;
    pdl_wait();
    float acc[B1_MAXC][VPC];
#pragma unroll
    for (int k = 0; k < B1_MAXC; ++k)
#pragma unroll
      for (int v = 0; v < VPC; ++v) acc[k][v] = 0.f;
    bool ok = __all_sync(0xffffffffu, mbar_wait(&S.xbar, 0, abort, err, p.timeout_ns));
    uint4 xr[B1_MAXC];
    {
      const uint4* xv = reinterpret_cast<const uint4*>(xs);
#pragma unroll
      for (int k = 0; k < B1_MAXC; ++k) {
        const int c = gt + NGT * k;
        xr[k] = (c < nch) ? xv[c] : make_uint4(0, 0, 0, 0);
      }
    }
    int g = 0;
    for (;;) {
      const int s2 = g % p.ns2;
      const uint32_t par = (uint32_t)(g / p.ns2) & 1u;
      // One thread decides for the group whether slot g holds a live unit
      // (1), or the gate has finished with fewer than g+1 live units (0), or
      // the block aborted (-1); the others take its decision.
      if (gt == 0) {
        int d = ok ? -2 : -1;
        uint64_t t0 = 0;
        for (uint32_t i = 0; d == -2; ++i) {
          if (mbar_try_wait(&S.full2[s2], par)) {
            d = 1;
          } else if (mbar_try_wait(&S.gate_done, 0) && g >= *(volatile int*)&S.n_live) {
            d = 0;
          } else if ((i & 63u) == 63u) {
            if (*abort) {
              d = -1;
            } else {
              const uint64_t now = globaltimer_ns();
              if (t0 == 0) {
                t0 = now;
              } else if (now - t0 > p.timeout_ns) {
                *abort = 1;
                atomicOr(err, DEV_ERR_TIMEOUT);
                d = -1;
              }
            }
          }
        }
        S.decision = d;
      }
      __syncwarp();
      named_barrier(1, NGT);
      const int d = *(volatile int*)&S.decision;
      if (d != 1) {
        ok = ok && (d == 0);
        break;
      }
      const uint4* w3 = reinterpret_cast<const uint4*>(ring2 + (size_t)s2 * slot2_bytes);
      const uint4* w2 = reinterpret_cast<const uint4*>(ring2 + (size_t)s2 * slot2_bytes + row_bytes);
      float d0 = 0.f, d1 = 0.f;
#pragma unroll
      for (int k = 0; k < B1_MAXC; ++k) {
        const int c = gt + NGT * k;
        if (c < nch) {
          float wv[VPC], xf[VPC];
          E::unpack(w3[c], wv);
          E::unpack(xr[k], xf);
#pragma unroll
          for (int v = 0; v < VPC; v += 2) {
            d0 = fmaf(wv[v], xf[v], d0);
            d1 = fmaf(wv[v + 1], xf[v + 1], d1);
          }
        }
      }
      const float part = warp_sum(d0 + d1);
      if (lane == 0) S.red[s2][gwarp] = part;
      __syncwarp();
      named_barrier(1, NGT);
      float u = 0.f;
#pragma unroll
      for (int w = 0; w < B1_NGA; ++w) u += S.red[s2][w];
      const float h = __int_as_float(S.meta[s2].y) * u;
#pragma unroll
      for (int k = 0; k < B1_MAXC; ++k) {
        const int c = gt + NGT * k;
        if (c < nch) {
          float wv[VPC];
          E::unpack(w2[c], wv);
#pragma unroll
          for (int v = 0; v < VPC; ++v) acc[k][v] = fmaf(h, wv[v], acc[k][v]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty2[s2]);
      ++g;
    }
    // add this block's partial y into the accumulator
    if (ok && g > 0) {
#pragma unroll
      for (int k = 0; k < B1_MAXC; ++k) {
        const int c = gt + NGT * k;
        if (c < nch) {
          float4* dst = reinterpret_cast<float4*>(p.yacc + (size_t)c * VPC);
#pragma unroll
          for (int v = 0; v < VPC; v += 4)
            atomicAdd(dst + v / 4, make_float4(acc[k][v], acc[k][v + 1], acc[k][v + 2], acc[k][v + 3]));
        }
      }
    }
    __threadfence();
  }

  // ------------------------------------------------------------------ block epilogue
  constexpr int NCONS = (B1_NWG + B1_NGA) * 32;
  if (warp > 0) {
    __syncwarp();
    named_barrier(2, NCONS);
    if (threadIdx.x == 32) {
      if (!*abort) atomicAdd(p.ctrl + CTRL_COUNT + p.count_slot, S.n_live);
      __threadfence();
      const int ticket = atomicAdd(p.ctrl + CTRL_TICKET, 1);
      S.last = (ticket == (int)gridDim.x - 1);
    }
    __syncwarp();
    named_barrier(2, NCONS);
    if (S.last) {
      // every other block has added its partial and taken its ticket
      __threadfence();
      const int ct = threadIdx.x - 32;
      const int n4 = D / 4;
      float4* ya = reinterpret_cast<float4*>(p.yacc);
      for (int i = ct; i < n4; i += NCONS) {
        const float4 v = __ldcg(ya + i);
        if constexpr (VPC == 4) {
          reinterpret_cast<float4*>(p.y)[i] = v;
        } else {
          reinterpret_cast<uint2*>(p.y)[i] = make_uint2(pack_bf16x2_rn(v.x, v.y), pack_bf16x2_rn(v.z, v.w));
        }
        __stcg(ya + i, make_float4(0.f, 0.f, 0.f, 0.f));
      }
      if (ct == 0) {
        p.counts[0] = atomicExch(p.ctrl + CTRL_COUNT + p.count_slot, 0);
        atomicExch(p.ctrl + CTRL_TICKET, 0);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort) {
    for (int s = 0; s < p.ns1; ++s) drain(&S.full1[s], S.issued1[s]);
    for (int s = 0; s < p.ns2; ++s) drain(&S.full2[s], S.issued2[s]);
  }
}

}  // namespace

size_t ffn_b1_smem_bytes(int D, int gate_k, int elt_bytes, bool lopa, int ns1, int ns2) {
  return b1_layout(D, gate_k, elt_bytes, lopa, ns1, ns2).total;
}

cudaError_t ffn_b1_prepare(size_t max_smem) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(ffn_b1_kernel<float, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem)))
    return e;
  if ((e = cudaFuncSetAttribute(ffn_b1_kernel<float, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem)))
    return e;
  if ((e = cudaFuncSetAttribute(ffn_b1_kernel<bf16_tag, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem)))
    return e;
  return cudaFuncSetAttribute(ffn_b1_kernel<bf16_tag, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
}

cudaError_t launch_ffn_b1(const B1Params& p, int dtype, bool lopa, int grid, size_t smem,
                          cudaStream_t s) {
  const dim3 g(grid), b(B1_THREADS);
  if (dtype == 0)
    return lopa ? launch_pdl(ffn_b1_kernel<float, true>, g, b, smem, s, p)
                : launch_pdl(ffn_b1_kernel<float, false>, g, b, smem, s, p);
  return lopa ? launch_pdl(ffn_b1_kernel<bf16_tag, true>, g, b, smem, s, p)
              : launch_pdl(ffn_b1_kernel<bf16_tag, false>, g, b, smem, s, p);
}

}  // namespace sffn
