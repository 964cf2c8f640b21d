// ffn_b1_bf16.cu -- fused single-token gate-first sparse FFN for bf16 weights
// (standard or low-rank gate).
//
// The method ("Model casting: compute the gate, then skip most of the FFN",
// sections "What an FFN actually computes" and "The 3x ceiling, and why W1 is
// always on"): compute the whole gate z, keep S = {i : z_i > 0}, and for those
// units only read row i of W3 and column i of W2 (row i of W2^T):
//     y = sum_{i in S} W2^T[i, :] * A(z_i) * (W3[i, :] . x).
// Standard gate: z = W1 x.  Low-rank gate ("LoPA Gating: moving the ceiling"):
// z = U t with t = V x computed in fp32 by the preceding kernel (lopa_t.cu).
//
// GB300 mapping.  One call moves tens of MB in a few microseconds, and
// consecutive calls are stream-ordered: what sets the pace is how much of a
// call's weight traffic is on chip before its dependency wait, how soon the
// rest is requested after it, and how many instructions each byte costs once
// it is on chip (at 45 GB/s of HBM per SM, a bf16 dot product that needs more
// than ~25 instructions per 16 bytes falls behind the memory).
//   * Gate rows.  The block's slice of W1 (or U) is contiguous.  Two halves of
//     a shared area are filled by one bulk copy each (the TMA engine's
//     non-tensor form, completion on an mbarrier) before the wait.  After the
//     wait the halves are consumed in turn, and each is refilled with the next
//     rows of the slice as soon as it has been read, so the rest of the slice
//     is requested within a few hundred nanoseconds of the wait.  Nothing else
//     is held across the wait: at 384 threads x 80 registers (two blocks per
//     SM) every register given to prefetched rows is taken from the dot
//     products (measured 1 us per call slower with 12 rows held that way).
//   * Dot products.  Two rows per warp share every load of x; each lane widens
//     bf16 pairs with one shift or mask per value and accumulates with packed
//     fp32x2 FMAs; shared memory is read through explicit shared-window loads.
//   * Compaction: a live unit is appended to the block's list through a
//     shared counter; one lane requests its W3 row and W2^T row into L2 with
//     two bulk prefetches.
//   * Gathers.  Thread t owns the 16-byte chunks t and t + 384 of x, of every
//     gathered row and of y.  A round of up to MG units loads their W3 and
//     W2^T chunks straight into registers (one L2 round trip), forms the
//     partial dots W3[i] . x per warp, sums the twelve warp partials in shared
//     memory, and folds h_i W2^T[i] into the thread's y chunks.
//   * The block adds its partial y into one of four fp32 accumulator copies
//     with 128-bit atomics; the finalize kernel chained behind sums the copies.
// Every wait on a bulk copy is bounded; on timeout the kernel records the
// error word and carries on with whatever the buffer holds (no fault).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace sffn {

namespace {

constexpr int NW = 12;          // warps per block (two blocks and a finalize block fit an SM)
constexpr int NT = NW * 32;     // threads per block
constexpr int MG = 5;           // units per gather round (registers: 2 chunks per unit and thread-chunk)
constexpr unsigned long long kCopyLimitNs = 250000000ull;

__host__ __device__ constexpr size_t al16(size_t v) { return (v + 15) & ~size_t(15); }

__device__ __forceinline__ uint4 ld_l2(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// shared-window loads by 32-bit shared address
__device__ __forceinline__ uint4 lda16(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 ldaf4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}

// bf16 pair (low half first) -> fp32 pair: the bf16 bits are the top half of a binary32
__device__ __forceinline__ float2 bfp(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ void unpack4(const uint4& c, float2 (&f)[4]) {
  f[0] = bfp(c.x);
  f[1] = bfp(c.y);
  f[2] = bfp(c.z);
  f[3] = bfp(c.w);
}
// acc += w (8 bf16) . x (8 fp32 as pairs)
__device__ __forceinline__ void fma8(float2& acc, const uint4& w, const float2 (&x)[4]) {
  ffma2(acc, bfp(w.x), x[0]);
  ffma2(acc, bfp(w.y), x[1]);
  ffma2(acc, bfp(w.z), x[2]);
  ffma2(acc, bfp(w.w), x[3]);
}
__device__ __forceinline__ float hsum(float2 a) { return a.x + a.y; }

// ---- dot products of staged gate rows (shared addresses) with x or t, lanes
// striding 32 chunks.  Standard gate: x bf16 (16 bytes per chunk).
__device__ __forceinline__ float dot1_x(uint32_t r, uint32_t xs, int lane, int nch) {
  float2 a0 = make_float2(0.f, 0.f), a1 = a0;
  int c = lane;
  for (; c + 32 < nch; c += 64) {
    const uint32_t o0 = (uint32_t)c * 16u, o1 = o0 + 512u;
    const uint4 w0 = lda16(r + o0), w1 = lda16(r + o1);
    const uint4 x0 = lda16(xs + o0), x1 = lda16(xs + o1);
    float2 f0[4], f1[4];
    unpack4(x0, f0);
    unpack4(x1, f1);
    fma8(a0, w0, f0);
    fma8(a1, w1, f1);
  }
  if (c < nch) {
    const uint32_t o0 = (uint32_t)c * 16u;
    float2 f0[4];
    unpack4(lda16(xs + o0), f0);
    fma8(a0, lda16(r + o0), f0);
  }
  return warp_sum(hsum(a0) + hsum(a1));
}
__device__ __forceinline__ void dot2_x(uint32_t ra, uint32_t rb, uint32_t xs, int lane, int nch, float& za,
                                       float& zb) {
  float2 a = make_float2(0.f, 0.f), b = a;
  for (int c = lane; c < nch; c += 32) {
    const uint32_t o = (uint32_t)c * 16u;
    const uint4 wa = lda16(ra + o), wb = lda16(rb + o), xv = lda16(xs + o);
    float2 f[4];
    unpack4(xv, f);
    fma8(a, wa, f);
    fma8(b, wb, f);
  }
  za = warp_sum(hsum(a));
  zb = warp_sum(hsum(b));
}
// Low-rank gate: t fp32 (32 bytes per chunk of 8 values)
__device__ __forceinline__ void tpairs(uint32_t ts, int c, float2 (&f)[4]) {
  const float4 t0 = ldaf4(ts + (uint32_t)c * 32u), t1 = ldaf4(ts + (uint32_t)c * 32u + 16u);
  f[0] = make_float2(t0.x, t0.y);
  f[1] = make_float2(t0.z, t0.w);
  f[2] = make_float2(t1.x, t1.y);
  f[3] = make_float2(t1.z, t1.w);
}
__device__ __forceinline__ float dot1_t(uint32_t r, uint32_t ts, int lane, int nch) {
  float2 a0 = make_float2(0.f, 0.f), a1 = a0;
  int c = lane;
  for (; c + 32 < nch; c += 64) {
    const uint4 w0 = lda16(r + (uint32_t)c * 16u), w1 = lda16(r + (uint32_t)(c + 32) * 16u);
    float2 f0[4], f1[4];
    tpairs(ts, c, f0);
    tpairs(ts, c + 32, f1);
    fma8(a0, w0, f0);
    fma8(a1, w1, f1);
  }
  if (c < nch) {
    float2 f0[4];
    tpairs(ts, c, f0);
    fma8(a0, lda16(r + (uint32_t)c * 16u), f0);
  }
  return warp_sum(hsum(a0) + hsum(a1));
}
__device__ __forceinline__ void dot2_t(uint32_t ra, uint32_t rb, uint32_t ts, int lane, int nch, float& za,
                                       float& zb) {
  float2 a = make_float2(0.f, 0.f), b = a;
  for (int c = lane; c < nch; c += 32) {
    const uint32_t o = (uint32_t)c * 16u;
    const uint4 wa = lda16(ra + o), wb = lda16(rb + o);
    float2 f[4];
    tpairs(ts, c, f);
    fma8(a, wa, f);
    fma8(b, wb, f);
  }
  za = warp_sum(hsum(a));
  zb = warp_sum(hsum(b));
}

// SFFN_DEBUG builds check every live-list append and every gathered unit
// index (against the list capacity and the block's own slice of units) and
// record a violation as DEV_ERR_CHECK instead of making the access.
#ifdef SFFN_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// One bulk copy of `bytes` of consecutive gate rows into shared memory at
// `dst`, completing on the mbarrier at `bar` (both shared-window addresses).
// The copy is checked first -- 16-byte alignment of both ends and of the size,
// destination inside this block's dynamic shared memory [s_lo, s_hi), 8-byte
// mbarrier: a failing check records DEV_ERR_CHECK, raises the block's abort
// flag (every later wait returns at once) and issues nothing.
__device__ __forceinline__ void fill_rows(uint32_t dst, uint32_t bar, const void* src, uint32_t bytes, uint32_t s_lo,
                                          uint32_t s_hi, int* abortf, int* err) {
  const bool ok = ((dst | bytes | (uint32_t)reinterpret_cast<uintptr_t>(src)) & 15u) == 0 && (bar & 7u) == 0 &&
                  dst >= s_lo && dst + bytes <= s_hi && bytes > 0;
  if (!ok) {
    atomicOr(err, DEV_ERR_CHECK);
    *reinterpret_cast<volatile int*>(abortf) = 1;
    return;
  }
  mbar_arrive_expect_tx_a(bar, bytes);
  bulk_g2s_a(dst, src, bytes, bar);
}

// Bounded wait on phase `parity` of the mbarrier at shared address `bar`
// (gives up when the block's abort flag is raised or after kCopyLimitNs).
__device__ __forceinline__ bool bar_wait_a(uint32_t bar, uint32_t parity, int* abortf, int* err) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  if (ok) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((i & 63u) == 0) {
      if (*reinterpret_cast<volatile int*>(abortf)) return false;
      if (globaltimer_ns() - t0 > kCopyLimitNs) {
        *reinterpret_cast<volatile int*>(abortf) = 1;
        atomicOr(err, DEV_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// CPT: 16-byte chunks of a D-row per thread (1: D <= 3072, 2: D <= 6144)
template <bool LOPA, bool EXT, int CPT>
__global__ void __launch_bounds__(NT, 2) ffn_b1_bf16_kernel(const B1Params p) {
  constexpr int M = CPT == 1 ? MG : 2;  // units per gather round (registers)
  extern __shared__ __align__(16) uint8_t smem[];
  const int D = p.D;
  const int nch = D / 8;          // 16-byte chunks of x, W3 and W2^T rows
  const int nchg = p.gate_k / 8;  // ... of a gate row (W1 or U)
  const int row0 = (int)(((long long)blockIdx.x * p.H) / gridDim.x);
  const int row1 = (int)(((long long)(blockIdx.x + 1) * p.H) / gridDim.x);
  const int cap = p.rows_cap;  // >= units of this block
  uint8_t* sp = smem;
  uint4* xs = reinterpret_cast<uint4*>(sp);
  sp += al16((size_t)nch * 16);
  float* ts = reinterpret_cast<float*>(sp);
  sp += LOPA ? al16((size_t)p.gate_k * 4) : 0;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sp);  // [0] half A, [1] half B
  sp += 16;
  int* l_unit = reinterpret_cast<int*>(sp);
  float* l_a = reinterpret_cast<float*>(l_unit + cap);
  int* misc = reinterpret_cast<int*>(l_a + cap);  // 0: live count, 1: abort flag, 2..3: RMSNorm scratch
  float* part = reinterpret_cast<float*>(misc + 4);  // [NW][MG] warp partials of a gather round
  float* hval = part + NW * MG;                      // [MG] h of the round's units
  uint8_t* l_mask = reinterpret_cast<uint8_t*>(hval + MG);  // live flag of every unit of the block
  sp += al16((size_t)cap * 9 + 16 + 4 * (NW * MG + MG));
  uint4* srows = reinterpret_cast<uint4*>(sp);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint4* G = static_cast<const uint4*>(p.gate_w);
  const uint4* W3 = static_cast<const uint4*>(p.W3);
  const uint4* W2t = static_cast<const uint4*>(p.W2t);
  int* err = p.ctrl + CTRL_ERR;

  // ---- gate rows: [0, RA) half A, [RA, R) half B (bulk copies before the wait),
  // the rest refilled into A and B after it.  Shared addresses below are 32-bit
  // offsets in the shared window.
  const int nrows = row1 - row0;
  const int R = min(p.pref_rows, nrows);
  const int RA = (R + 1) / 2, RB = R - RA;
  const uint32_t rowb = (uint32_t)nchg * 16u;  // bytes of a gate row
  const uint32_t s_lo = smem_u32(smem), s_hi = s_lo + dynamic_smem_bytes();
  const uint32_t hA_a = smem_u32(srows), hB_a = hA_a + (uint32_t)RA * rowb;
  const uint32_t barA = smem_u32(&bars[0]), barB = smem_u32(&bars[1]);
  if (tid == 0) {
    pdl_launch_dependents();
    misc[0] = 0;
    misc[1] = 0;
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    if (RA > 0) fill_rows(hA_a, barA, G + (size_t)row0 * nchg, (uint32_t)RA * rowb, s_lo, s_hi, misc + 1, err);
    if (RB > 0) fill_rows(hB_a, barB, G + (size_t)(row0 + RA) * nchg, (uint32_t)RB * rowb, s_lo, s_hi, misc + 1, err);
    prefetch_l2_bulk(p.x, (uint32_t)nch * 16u);
  }

  pdl_wait();  // x, t, the outputs and the accumulators follow stream order
  for (int i = tid; i < nch; i += NT) xs[i] = __ldcg(static_cast<const uint4*>(p.x) + i);
  if constexpr (LOPA) {
    for (int i = tid; i < p.gate_k / 4; i += NT)
      reinterpret_cast<float4*>(ts)[i] = __ldcg(reinterpret_cast<const float4*>(p.t) + i);
  }
  __syncthreads();
  if constexpr (LOPA && EXT) {
    if (p.flags & FLAG_RMSNORM) rmsnorm_shared(ts, 1, p.gate_k, reinterpret_cast<float*>(misc + 2), NT);
  }
  const uint32_t xs_a = smem_u32(xs), vs_a = LOPA ? smem_u32(ts) : smem_u32(xs);

  // z of unit q (identical in every lane of the warp)
  auto decide = [&](int q, float z) {
    if constexpr (LOPA && EXT) {
      if (p.flags & FLAG_TILED_G) z += staged_elem<bf16_tag>(xs, q % D);  // (G x)_q = x_{q mod D}
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
    if (lane == 0) {
      l_mask[q - row0] = live ? 1 : 0;  // written out once at the end
      if (live) {  // compaction: append to the block's list; both gathered rows start moving into L2
        const int j = atomicAdd(misc, 1);
        if (kDebugChecks && (j >= cap || q < row0 || q >= row1)) {
          atomicOr(err, DEV_ERR_CHECK);
          return;
        }
        l_unit[j] = q;
        l_a[j] = a;
        prefetch_l2_bulk(W3 + (size_t)q * nch, (uint32_t)nch * 16u);
        prefetch_l2_bulk(W2t + (size_t)q * nch, (uint32_t)nch * 16u);
      }
    }
  };
  // rows [0, n) of a half at shared address ha whose first row is slice row `first`
  auto half_rows = [&](uint32_t ha, int first, int n) {
    if (n > NW) {  // two rows per warp share the loads of x (or t)
      for (int i = 2 * warp; i < n; i += 2 * NW) {
        const bool two = i + 1 < n;
        float za, zb;
        if constexpr (LOPA)
          dot2_t(ha + (uint32_t)i * rowb, ha + (uint32_t)(two ? i + 1 : i) * rowb, vs_a, lane, nchg, za, zb);
        else
          dot2_x(ha + (uint32_t)i * rowb, ha + (uint32_t)(two ? i + 1 : i) * rowb, vs_a, lane, nchg, za, zb);
        decide(row0 + first + i, za);
        if (two) decide(row0 + first + i + 1, zb);
      }
    } else if (warp < n) {
      const float z = LOPA ? dot1_t(ha + (uint32_t)warp * rowb, vs_a, lane, nchg)
                           : dot1_x(ha + (uint32_t)warp * rowb, vs_a, lane, nchg);
      decide(row0 + first + warp, z);
    }
  };

  // Each half holds one batch of consecutive slice rows at a time: it is
  // waited on, read, and (after a barrier) refilled with the next rows of the
  // slice still to copy, which start at `next`.  The halves alternate, A
  // first.  All of this state is uniform over the block.
  int next = R;
  uint32_t phA = 0, phB = 0;
  int firstA = 0, nA = RA, firstB = RA, nB = RB;
  for (int step = 0;; ++step) {
    const bool b = step & 1;  // this step's half: A (false) or B
    const int n = b ? nB : nA;
    if (n > 0) {
      if (!bar_wait_a(b ? barB : barA, b ? phB : phA, misc + 1, err)) misc[1] = 1;  // timed out: rows as they are
      if (b)
        phB ^= 1u;
      else
        phA ^= 1u;
      half_rows(b ? hB_a : hA_a, b ? firstB : firstA, n);
      __syncthreads();  // every read of the half is done (and misc[1] is settled)
      // refill with the next rows of the slice (nothing more after a failed copy)
      const int m = misc[1] ? 0 : min(b ? RB : RA, nrows - next);
      if (b) {
        firstB = next;
        nB = max(m, 0);
      } else {
        firstA = next;
        nA = max(m, 0);
      }
      if (m > 0) {
        if (tid == 0)
          fill_rows(b ? hB_a : hA_a, b ? barB : barA, G + (size_t)(row0 + next) * nchg, (uint32_t)m * rowb, s_lo,
                    s_hi, misc + 1, err);
        next += m;
      }
    }
    if (step >= 1 && nA == 0 && nB == 0) break;
  }
  __syncthreads();
  const int n_live = min(misc[0], cap);
  if (p.ypart) {
    // deterministic option: the list in ascending unit order, so that the fold
    // order does not depend on which warp decided first (cap <= NT is checked
    // when the handle is created)
    int u = 0, rank = 0;
    float a = 0.f;
    if (tid < n_live) {
      u = l_unit[tid];
      a = l_a[tid];
      for (int k = 0; k < n_live; ++k) rank += l_unit[k] < u;
    }
    __syncthreads();
    if (tid < n_live) {
      l_unit[rank] = u;
      l_a[rank] = a;
    }
    __syncthreads();
  }

  // ---- gathers: thread t owns chunks t and t + NT of x, of the gathered rows and of y
  const int c0 = tid, c1 = tid + NT;
  const bool h0 = c0 < nch, h1 = CPT > 1 && c1 < nch;
  float2 xf0[4], xf1[4], y0[4], y1[4];
  {
    const uint4 z4 = make_uint4(0, 0, 0, 0);
    unpack4(h0 ? lda16(xs_a + (uint32_t)c0 * 16u) : z4, xf0);
    if constexpr (CPT > 1) unpack4(h1 ? lda16(xs_a + (uint32_t)c1 * 16u) : z4, xf1);
#pragma unroll
    for (int k = 0; k < 4; ++k) y0[k] = y1[k] = make_float2(0.f, 0.f);
  }
  const bool dbl = EXT && (p.flags & FLAG_DOUBLE_ACT);
  for (int b0 = 0; b0 < n_live; b0 += M) {
    const int m = min(M, n_live - b0);
    uint4 w3[M], w2[M], w3b[CPT > 1 ? M : 1], w2b[CPT > 1 ? M : 1];
#pragma unroll
    for (int u = 0; u < M; ++u) {
      const int q = l_unit[b0 + (u < m ? u : 0)];
      const size_t rowo = (size_t)q * nch;
      bool ok = u < m;
      if (kDebugChecks && ok && (q < row0 || q >= row1)) {
        if (lane == 0) atomicOr(err, DEV_ERR_CHECK);
        ok = false;  // the unit contributes nothing
      }
      w3[u] = (ok && h0) ? ld_l2(W3 + rowo + c0) : make_uint4(0, 0, 0, 0);
      w2[u] = (ok && h0) ? ld_l2(W2t + rowo + c0) : make_uint4(0, 0, 0, 0);
      if constexpr (CPT > 1) {
        w3b[u] = (ok && h1) ? ld_l2(W3 + rowo + c1) : make_uint4(0, 0, 0, 0);
        w2b[u] = (ok && h1) ? ld_l2(W2t + rowo + c1) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < M; ++u) {
      float2 acc = make_float2(0.f, 0.f);
      fma8(acc, w3[u], xf0);
      if constexpr (CPT > 1) fma8(acc, w3b[u], xf1);
      const float s = warp_sum(hsum(acc));
      if (lane == 0) part[warp * MG + u] = s;
    }
    __syncthreads();
    if (tid < m) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) s += part[w * MG + tid];
      hval[tid] = l_a[b0 + tid] * (dbl ? activation(p.act, s) : s);
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < M; ++u) {
      if (u < m) {
        const float h = hval[u];
        const float2 hh = make_float2(h, h);
        ffma2(y0[0], hh, bfp(w2[u].x));
        ffma2(y0[1], hh, bfp(w2[u].y));
        ffma2(y0[2], hh, bfp(w2[u].z));
        ffma2(y0[3], hh, bfp(w2[u].w));
        if constexpr (CPT > 1) {
          ffma2(y1[0], hh, bfp(w2b[u].x));
          ffma2(y1[1], hh, bfp(w2b[u].y));
          ffma2(y1[2], hh, bfp(w2b[u].z));
          ffma2(y1[3], hh, bfp(w2b[u].w));
        }
      }
    }
    // part[] and hval[] are rewritten by the next round only after its first barrier
  }
  if (p.ypart) {  // deterministic option: the block's partial y, every element, into its own row
    float* yr = p.ypart + (size_t)blockIdx.x * D;
    if (h0) {
      __stcg(reinterpret_cast<float4*>(yr + (size_t)c0 * 8), make_float4(y0[0].x, y0[0].y, y0[1].x, y0[1].y));
      __stcg(reinterpret_cast<float4*>(yr + (size_t)c0 * 8 + 4), make_float4(y0[2].x, y0[2].y, y0[3].x, y0[3].y));
    }
    if (CPT > 1 && h1) {
      __stcg(reinterpret_cast<float4*>(yr + (size_t)c1 * 8), make_float4(y1[0].x, y1[0].y, y1[1].x, y1[1].y));
      __stcg(reinterpret_cast<float4*>(yr + (size_t)c1 * 8 + 4), make_float4(y1[2].x, y1[2].y, y1[3].x, y1[3].y));
    }
  }
  // into accumulator copy (block mod YACC_COPIES): fewer blocks per address
  float* yc = p.yacc + (size_t)(blockIdx.x % YACC_COPIES) * D;
  if (n_live > 0 && !p.ypart) {
    if (h0) {
      atomicAdd(reinterpret_cast<float4*>(yc + (size_t)c0 * 8), make_float4(y0[0].x, y0[0].y, y0[1].x, y0[1].y));
      atomicAdd(reinterpret_cast<float4*>(yc + (size_t)c0 * 8 + 4), make_float4(y0[2].x, y0[2].y, y0[3].x, y0[3].y));
    }
    if (CPT > 1 && h1) {
      atomicAdd(reinterpret_cast<float4*>(yc + (size_t)c1 * 8), make_float4(y1[0].x, y1[0].y, y1[1].x, y1[1].y));
      atomicAdd(reinterpret_cast<float4*>(yc + (size_t)c1 * 8 + 4), make_float4(y1[2].x, y1[2].y, y1[3].x, y1[3].y));
    }
  }
  // the block's live count; the finalize kernel that follows in the stream
  // sums the accumulator copies once every block has finished
  if (tid == 0 && n_live > 0) atomicAdd(p.ctrl + CTRL_COUNT + p.count_slot, n_live);
  if (p.mask)  // the block's live flags, one coalesced store
    for (int i = tid; i < nrows; i += NT) p.mask[row0 + i] = l_mask[i];
}

}  // namespace

StreamPlan plan_ffn_b1_bf16(int D, int gate_k, bool lopa, int rows_cap) {
  StreamPlan pl;
  const size_t grow = (size_t)gate_k * 2, fixed = al16((size_t)D * 2) + (lopa ? al16((size_t)gate_k * 4) : 0) + 16 +
                                               al16((size_t)rows_cap * 9 + 16 + 4 * (NW * MG + MG));
  // two blocks per SM (the next call's blocks prefetch while this call runs): at most 110 KB per block
  const size_t budget = 110u * 1024u;
  const size_t area = budget > fixed ? budget - fixed : 0;
  pl.pref_rows = (int)std::max<size_t>(1, std::min<size_t>((size_t)rows_cap, area / grow));
  pl.gather_rows = 0;
  pl.smem = fixed + (size_t)pl.pref_rows * grow;
  return pl;
}

cudaError_t ffn_b1_bf16_prepare(size_t max_smem) {
  void (*ks[8])(const B1Params) = {
      ffn_b1_bf16_kernel<false, false, 1>, ffn_b1_bf16_kernel<true, false, 1>, ffn_b1_bf16_kernel<false, true, 1>,
      ffn_b1_bf16_kernel<true, true, 1>,   ffn_b1_bf16_kernel<false, false, 2>, ffn_b1_bf16_kernel<true, false, 2>,
      ffn_b1_bf16_kernel<false, true, 2>,  ffn_b1_bf16_kernel<true, true, 2>};
  for (auto k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int ffn_b1_bf16_threads() { return NT; }

cudaError_t launch_ffn_b1_bf16(const B1Params& p, bool lopa, int grid, size_t smem, cudaStream_t s) {
  const dim3 g(grid), b(NT);
  const bool ext = p.flags != 0 || p.act == ACT_SILU || p.thr != 0.f;
  void (*k)(const B1Params);
  if (p.D / 8 <= NT)
    k = ext ? (lopa ? ffn_b1_bf16_kernel<true, true, 1> : ffn_b1_bf16_kernel<false, true, 1>)
            : (lopa ? ffn_b1_bf16_kernel<true, false, 1> : ffn_b1_bf16_kernel<false, false, 1>);
  else
    k = ext ? (lopa ? ffn_b1_bf16_kernel<true, true, 2> : ffn_b1_bf16_kernel<false, true, 2>)
            : (lopa ? ffn_b1_bf16_kernel<true, false, 2> : ffn_b1_bf16_kernel<false, false, 2>);
  return launch_pdl(k, g, b, smem, s, p);
}

}  // namespace sffn
