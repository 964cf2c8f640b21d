// ffn_tcg.cu -- small batches on the tensor cores with the union skip: only
// the W3 rows and W2 columns of units live for at least one token are read
// (bf16 weights and tokens, standard gate, B <= TCG_MAX_BATCH).
//
// The method per token b ("Model casting: compute the gate, then skip most of
// the FFN", section "What an FFN actually computes"):
//     y_b = sum_{i : z_bi live} W2[:, i] * A(z_bi) * (W3[i, :] . x_b),  z_b = W1 x_b.
// With B tokens a unit's W3 row and W2 column are needed when ANY token keeps
// it: the union of the live sets, which the pages warn grows with the batch.
// While the union is well below H this path reads W1 in full and then only
// the union's rows of W3 and W2^T:
//
//   gate kernel, one block per slice of NU units:
//     phase 1: Z[slice, :] = W1[slice, :] X^T on tcgen05 (2D TMA tiles of W1
//              and x, 128-byte swizzle, TMEM accumulators);
//     epilogue 1: live flags, per-token counts and A(z) per (unit, token);
//              the slice's union compacted in ascending order by warp ballots;
//     phase 2: P[union, :] = W3[union, :] X^T on tcgen05.  The union's W3
//              rows are gathered by five warps with 16-byte cp.async straight
//              into the swizzled K-major operand layout, one 64-wide K chunk
//              per slot of a ring laid over the phase-1 stages (nu rows per
//              slot instead of NU, so most of the gather is in flight at
//              once); each thread's copies arrive on the slot's barrier when
//              they land (cp.async.mbarrier.arrive), x comes by TMA, and the
//              MMA thread fences the slot to the async proxy before reading;
//     epilogue 2: one atomic on a global counter reserves the slice's
//              positions in the batch's union list; h = A(z) * p (exactly 0
//              for a dead pair), rounded to bf16, at those positions of hbuf
//              row b.
//   down kernel, one block per (128-wide slice of y, range of the union):
//     y^T[d-slice, :] += W2^T[union, d-slice]^T h: the union's
//     W2^T row segments gathered the same way into the MN-major operand
//     layout, a 64-position chunk per ring slot; h by TMA (the chunk that
//     holds the end of the union by cp.async, zero past it); fp32 atomics
//     into the accumulator, the last block of a y slice rounds it into y; the
//     last block of the grid resets the union counter for the next call.
// Every wait is bounded (error word + early exit); a block drains its copies
// and MMAs before it releases TMEM.
#include <cudaTypedefs.h>

#include <algorithm>

#include "internal.h"
#include "tc.cuh"

namespace sffn {

namespace {

constexpr int G_THREADS = 288;  // gate kernel: warps 0-3 TMEM epilogue, 4 producer, 5-8 MMA issuers
constexpr int G_PRODUCER = 4;
constexpr int G_MMA0 = 5;
constexpr int GATHER_THREADS = 160;  // warps 0-4 gather in phase 2 and in the down kernel
constexpr int D_THREADS = 192;  // down kernel: warps 0-4 gatherers (0-3 then the epilogue), 5 MMA issuer
constexpr int D_MMA = 5;
constexpr int DT = 128;         // y values per down-kernel block (MMA M)
constexpr int UCH = 64;         // union positions per down-kernel K chunk
constexpr int NS_MAX = 8;
constexpr int DRING_MAX = 16;   // down kernel: ring slots
constexpr int Y_LD = 132;       // down kernel, cluster form: the partial tile [token][Y_LD] fp32
constexpr size_t SMEM_BUDGET = 200 * 1024;

struct GateArgs {
  int D, H, B, NB, NU, KC, C, NCG, NS, act, flags, Hs, nacc, apw;  // nacc MMA warps, apw accumulators each
  int XR;  // rows of phase 1's B tiles: NB (x), or 2 NB (the low-rank gate's t pair, t_hi then t_lo)
  int NX;  // phase 2: tokens padded to 8
  float thr;
  uint32_t tmem_cols;
  const uint16_t* W3;  // [H, D] bf16 (gathered rows)
  const uint16_t* W2t; // [H, D] bf16 (the union's rows are requested into L2 for the down kernel)
  const uint16_t* x;   // [B, D] bf16
  int* ctrl;
  uint8_t* mask;       // [B_max, H]
  uint16_t* hbuf;      // [256][Hs]: h of token b in row b, columns = union positions
  int* ulist;          // [H] the batch's union
  int* ucount;         // [1] units in the union (zero between calls)
  unsigned long long timeout_ns;
};

struct DownArgs {
  int D, H, B, NB, ndt, nsplit, RD, nacc, Hs, maxpos;
  int cluster;           // 1: the nsplit blocks of a y slice are a cluster (block = dt * nsplit + sp) and
                         // sum in distributed shared memory; 0: block = sp * ndt + dt, atomics, last block
  uint32_t tmem_cols;
  const uint16_t* W2t;   // [H, D] bf16 (gathered row segments)
  const uint16_t* hbuf;  // the gate kernel's h (the union's last chunk is read directly)
  const int* ulist;
  int* ucount;           // reset by the last block
  int* dticket;          // [1] blocks done (for that reset), zero between calls
  float* yacc;           // [B_max * YACC_COPIES, D]; copy 0 used, zero between calls
  void* y;
  int* ctrl;
  int* counts;
  int* tickets;          // [ndt] blocks of a y slice done, zero between calls
  unsigned long long timeout_ns;
};

__host__ __device__ constexpr uint32_t g_stage_bytes(int C, int NU, int NB) {
  return (uint32_t)C * 128u * (uint32_t)(NU + NB);
}
// An MMA reads 128 rows from an A region's start; the last A region of a stage
// is followed by the stage's x regions, and past the last stage lies slack.
__host__ __device__ inline uint32_t g_slack_bytes(int C, int NU, int NB) {
  const int over = (128 - NU) * 128 - C * NB * 128;
  return over > 0 ? (uint32_t)(over + 1023) / 1024 * 1024 : 0u;
}
// Phase 2 holds NBUF segment buffers over the stages: rows of 2 SEG + 16 bytes
// (the 16-byte pad keeps the rows of an 8x8 ldmatrix on distinct banks), the
// slice's union rows padded to 16, then the tokens padded to 8.
constexpr int NBUF = 4;
constexpr int SEG_MAX = 1280;
__host__ __device__ constexpr uint32_t g_seg_buffer_bytes(int nu16, int NX, int SEG) {
  return (uint32_t)(nu16 + NX) * (uint32_t)(2 * SEG + 16);
}
// the longest segment (a multiple of 64 values, at most SEG_MAX) whose NBUF buffers fit in `area` bytes
// (0: none fits)
__host__ __device__ inline int g_segment(uint32_t area, int nu16, int NX) {
  int seg = SEG_MAX;
  while (seg >= 64 && (uint32_t)NBUF * g_seg_buffer_bytes(nu16, NX, seg) > area) seg -= 64;
  return seg >= 64 ? seg : 0;
}
// after the stages and slack: 2 NS + 2 NBUF + 1 mbarriers, then tslot,
// abort flag, union count and base, per-token counts [NB], union flags [NU],
// union list [NU], A(z) [NU][NB + 1]
size_t g_smem_bytes(int C, int NU, int NB, int XR, int NS) {
  return 1024 + (size_t)NS * g_stage_bytes(C, NU, XR) + g_slack_bytes(C, NU, XR) + 8 * (2 * NS + 2 * NBUF + 1) +
         16 + 4 * (size_t)NB + 8 * (size_t)NU + 4 * (size_t)NU * (NB + 1) + 64;
}
__host__ __device__ constexpr uint32_t d_slot_bytes(int NB) { return 2u * UCH * 128u + (uint32_t)NB * 128u; }
// ring, 2 DRING_MAX + 2 mbarriers, tslot, abort flag, last-block flag, the block's union units [maxpos]
size_t d_smem_bytes(int NB, int RD, int maxpos) {
  return 1024 + (size_t)RD * d_slot_bytes(NB) + 8 * (2 * DRING_MAX + 2) + 16 + 4 * (size_t)maxpos + 64;
}

// Round a dynamic shared-memory pointer up to 1024 bytes by pointer arithmetic
// (keeps the shared address space visible to the compiler).
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}
// 16-byte cp.async of the first src_bytes (0..16) of src, zero-filling the rest
// (src_bytes = 0 reads nothing).
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival counts toward the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void st_shared16(uint32_t dst, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
// 8x8 b16 matrices from shared memory (lane l gives the row address of matrix l / 8)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
// d (16x8 fp32) += a (16x16 bf16, rows) * b (16x8 bf16, columns), one warp
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
               "{%0, %1, %2, %3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// Generic-proxy writes to shared memory made visible to this thread (here:
// gathered by cp.async, observed through an mbarrier) become visible to the
// async proxy, which the MMA reads through.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// --------------------------------------------------------------------------- gate kernel
// Phase-1 stage layout: A regions [C][NU rows x 128 B] of W1, then x regions
// [C][NB rows x 128 B].  K chunk group q covers chunks q*C .. q*C+C-1.  Phase
// 2 lays a ring of slots [nu8 rows of W3 | NB rows of x] over the same bytes.
// TMEM: nacc * apw accumulators of NB columns (lanes = slice rows in phase 1, union
// entries in phase 2).
// LOPA: phase 1 is the low-rank gate z = U t: mW1 maps U [H, r] (K chunks over
// r) and mX the t pair [2 NB, r]; two MMAs per K step, U t_hi and U t_lo, into
// one accumulator.  Phases 2 and the down kernel are the standard gate's.
template <bool LOPA>
__global__ void __launch_bounds__(G_THREADS, 1)
    ffn_tcg_gate_kernel(const __grid_constant__ CUtensorMap mW1, const __grid_constant__ CUtensorMap mX,
                        const GateArgs p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  const int NS = p.NS, NB = p.NB, C = p.C, NU = p.NU;
  const uint32_t wreg = (uint32_t)NU * 128u, xreg = (uint32_t)p.XR * 128u;
  const uint32_t st_bytes = g_stage_bytes(C, NU, p.XR);
  const uint32_t ring_bytes = (uint32_t)NS * st_bytes + g_slack_bytes(C, NU, p.XR);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + ring_bytes);
  uint64_t* empty = full + NS;
  uint64_t* f2 = empty + NS;  // phase 2: segment buffer filled (bulk copies)
  uint64_t* e2 = f2 + NBUF;   // phase 2: segment buffer read by the 8 computing warps
  uint64_t* done = e2 + NBUF; // phase-1 MMAs complete (one commit per MMA warp)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  int* s_nu = reinterpret_cast<int*>(tslot + 2);  // units of the slice in the union
  int* s_base = s_nu + 1;                         // their first position in the batch's list
  int* s_cnt = s_base + 1;                        // [NB] live counts of this slice
  int* s_uf = s_cnt + NB;                         // [NU] unit live for some token
  int* s_list = s_uf + NU;                        // [NU] the slice's union, ascending (slice rows)
  float* s_a = reinterpret_cast<float*>(s_list + NU);  // [NU][NB + 1] A(z), 0 for a dead pair
  const int lda = NB + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u0 = blockIdx.x * NU;
  const int KC = p.KC, NCG = p.NCG, D = p.D;
  int* err = p.ctrl + CTRL_ERR;
  auto nchunks = [&](int q) { return min(C, KC - q * C); };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], p.nacc);
    }
    for (int s = 0; s < NBUF; ++s) {
      mbar_init(&f2[s], 1);
      mbar_init(&e2[s], 8);
    }
    mbar_init(done, p.nacc);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < NB) s_cnt[tid] = 0;
  for (int i = tid; i < NU; i += G_THREADS) s_uf[i] = 0;
  if (warp == G_MMA0) tmem_alloc(tslot, p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) pdl_launch_dependents();  // after the TMEM allocation: a later kernel never takes these columns
  const int ldc = NB + 1;
  const int nacc_used = p.nacc * min(p.apw, KC);  // accumulators 0 .. nacc_used-1 hold partial sums
  float* s_acc = reinterpret_cast<float*>(sm);  // epilogue copy of Z [128][NB + 1], over the stages
  int ok1 = 1;

  // ---- phase 1: Z = W1 X^T
  if (warp == G_PRODUCER) {
    if (lane == 0) {
      tma_prefetch_map(&mW1);
      tma_prefetch_map(&mX);
    }
    const int npre = min(NS, NCG);
    for (int q = 0; q < npre; ++q) {  // W1 does not depend on the previous kernel: requested first
      const int nc = nchunks(q);
      if (lane == 0) mbar_arrive_expect_tx(&full[q], (uint32_t)nc * (wreg + xreg));
      __syncwarp();
      if (lane < nc) tma_tile_2d(sm + (size_t)q * st_bytes + lane * wreg, &mW1, (q * C + lane) * 64, u0, &full[q]);
    }
    pdl_wait();
    for (int q = 0; q < npre; ++q)
      if (lane < nchunks(q))
        tma_tile_2d(sm + (size_t)q * st_bytes + C * wreg + lane * xreg, &mX, (q * C + lane) * 64, 0, &full[q]);
    int issued = npre;
    for (int q = npre; q < NCG; ++q) {
      const int s = q % NS;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&empty[s], ((q / NS) - 1) & 1, abort_flag, err, p.timeout_ns);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint8_t* st = sm + (size_t)s * st_bytes;
      const int nc = nchunks(q);
      if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)nc * (wreg + xreg));
      __syncwarp();
      if (lane < 2 * nc) {
        const int c = lane >> 1;
        if ((lane & 1) == 0)
          tma_tile_2d(st + c * wreg, &mW1, (q * C + c) * 64, u0, &full[s]);
        else
          tma_tile_2d(st + C * wreg + c * xreg, &mX, (q * C + c) * 64, 0, &full[s]);
      }
      issued = q + 1;
    }
    if (lane == 0)
      for (int q = max(0, issued - NS); q < issued; ++q) mbar_wait_drain(&full[q % NS], (q / NS) & 1, p.timeout_ns);
    __syncwarp();
  } else if (warp >= G_MMA0) {
    // K step kk = mw of chunk kc into accumulator mw + nacc * (kc mod apw): MMAs into one
    // accumulator form a dependent chain whose latency, not the tensor pipe, sets the pace
    const int mw = warp - G_MMA0;
    if (mw < p.nacc && lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, NB, false, false);
      for (int q = 0; q < NCG; ++q) {
        const int s = q % NS;
        if (!mbar_wait(&full[s], (q / NS) & 1, abort_flag, err, p.timeout_ns)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(sm + (size_t)s * st_bytes);
        const uint64_t a0 = smem_desc(sa, 16, 1024, SMEM_LAYOUT_SW128);
        const uint64_t b0 = smem_desc(sa + C * wreg, 16, 1024, SMEM_LAYOUT_SW128);
        const int nc = nchunks(q);
        for (int c = 0; c < nc; ++c) {
          const uint64_t ac = a0 + ((c * wreg) >> 4), bc = b0 + ((c * xreg) >> 4);
          const int kc = q * C + c;
          const uint32_t da = tmem + (uint32_t)(mw + p.nacc * (kc % p.apw)) * NB;
          for (int kk = mw; kk < 4; kk += p.nacc) {
            tc_mma(da, ac + 2 * kk, bc + 2 * kk, idesc, kc >= p.apw);
            if constexpr (LOPA) tc_mma(da, ac + 2 * kk, bc + (uint32_t)NB * 8u + 2 * kk, idesc, true);  // U t_lo
          }
        }
        tc_commit(&empty[s]);
      }
      tc_commit(done);
      mbar_wait_drain(done, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // warps 0..3: TMEM lanes 32w..32w+31 (summing the accumulators) into s_acc
    pdl_wait();  // hbuf, the masks, the counts and the union list may still be read by the previous forward
    ok1 = __all_sync(0xffffffffu, mbar_wait(done, 0, abort_flag, err, p.timeout_ns));
    if (ok1) {
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
      float* row = s_acc + (size_t)(32 * warp + lane) * ldc;
      for (int c0 = 0; c0 < NB; c0 += 16) {
        float v[16];
        tmem_ld_sum(tl + c0, NB, nacc_used, v);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) row[c0 + jj] = v[jj];
      }
    }
  }
  tc_fence_before();
  const bool ok = __syncthreads_and(ok1) != 0;

  // ---- epilogue 1 on warps 0..7: thread (unit r, token group g = tid / 64)
  // takes tokens g, g + 4, ...; a warp shares each token, so counts are ballots
  if (ok && warp < 8) {
    for (int r0 = 0; r0 < NU; r0 += 64) {
      const int r = r0 + (tid & 63), g = tid >> 6;
      const bool valid = r < NU && u0 + r < p.H;
      const int u = u0 + r;
      bool any = false;
      for (int b = g; b < p.B; b += 4) {
        float z = valid ? s_acc[(size_t)r * ldc + b] : 0.f;
        if (LOPA && valid && (p.flags & FLAG_TILED_G))  // (G x)_u = x_{u mod D}
          z += __bfloat162float(__ushort_as_bfloat16(p.x[(size_t)b * D + u % D]));
        const float az = activation(p.act, z);
        const bool lv = valid && is_live(az, p.thr);
        const unsigned bal = __ballot_sync(0xffffffffu, lv);
        if (lane == 0 && bal) atomicAdd(&s_cnt[b], __popc(bal));
        if (valid) {
          if (p.mask) p.mask[(size_t)b * p.H + u] = lv ? 1 : 0;
          s_a[r * lda + b] = lv ? az : 0.f;
        }
        any |= lv;
      }
      if (any) s_uf[r] = 1;
    }
    named_barrier(1, 256);
    if (tid < p.B && s_cnt[tid]) atomicAdd(p.ctrl + CTRL_COUNT + tid, s_cnt[tid]);
    if (warp == 0) {  // the slice's union in ascending order
      int n = 0;
      for (int r0 = 0; r0 < NU; r0 += 32) {
        const bool f = r0 + lane < NU && s_uf[r0 + lane];
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (f) s_list[n + __popc(bal & ((1u << lane) - 1u))] = r0 + lane;
        n += __popc(bal);
      }
      if (lane == 0) *s_nu = n;
    }
  }
  if (!ok && tid == 0) *s_nu = 0;
  // the stage bytes (read above as s_acc) are written next by bulk copies (async proxy)
  fence_proxy_async();
  __syncthreads();
  const int nu = *s_nu;

  // ---- phase 2: P = W3[union] X^T on the CUDA cores' tensor path (mma.sync m16n8k16) straight from
  // whole-row segments that bulk copies place in shared memory (nothing to do for an empty union)
  if (nu > 0) {
    const int NU16 = (nu + 15) & ~15, nrg = NU16 / 16, NX = p.NX, ntg = NX / 8, B = p.B;
    const int SEG = g_segment(ring_bytes, NU16, NX), NSEG = (D + SEG - 1) / SEG;  // SEG >= 64 (host-checked)
    const uint32_t STR = (uint32_t)SEG * 2u + 16u, bufb = g_seg_buffer_bytes(NU16, NX, SEG);
    const uint32_t sbase = smem_u32(sm);
    if (warp == 8) {
      // producer: each segment's union rows and token rows by bulk copies (one per row, spread over the
      // lanes); after the first segments, the union's W2^T rows into L2 for the down kernel
      int s = 0;
      for (; s < NSEG; ++s) {
        const int b = s % NBUF;
        if (s >= NBUF) {
          int w = 1;
          if (lane == 0) w = mbar_wait(&e2[b], ((s / NBUF) - 1) & 1, abort_flag, err, p.timeout_ns);
          if (!__shfl_sync(0xffffffffu, w, 0)) break;
        }
        const int e0 = s * SEG;
        const uint32_t bytes = (uint32_t)min(SEG, D - e0) * 2u;
        if (lane == 0) mbar_arrive_expect_tx(&f2[b], (uint32_t)(nu + B) * bytes);
        __syncwarp();
        uint8_t* bb = sm + (size_t)b * bufb;
        for (int i = lane; i < nu + B; i += 32) {
          const uint16_t* src = i < nu ? p.W3 + (size_t)(u0 + s_list[i]) * D + e0 : p.x + (size_t)(i - nu) * D + e0;
          bulk_g2s(bb + (size_t)(i < nu ? i : NU16 + i - nu) * STR, src, bytes, &f2[b]);
        }
        if (s == min(1, NSEG - 1))
          for (int i = lane; i < nu; i += 32) prefetch_l2_bulk(p.W2t + (size_t)(u0 + s_list[i]) * D, (uint32_t)D * 2u);
      }
      if (lane == 0)  // the copies of the last segments have landed before the block exits
        for (int q = max(0, s - NBUF); q < s; ++q) mbar_wait_drain(&f2[q % NBUF], (q / NBUF) & 1, p.timeout_ns);
      __syncwarp();
    } else {
      // warps 0-7: warp (rg, kp) = (warp / KW, warp % KW) takes row group rg (16 union rows) and every
      // KW-th 16-wide K step of each segment, for all token groups
      if (tid == 0) *s_base = atomicAdd(p.ucount, nu);
      {  // padding token rows of both buffers: zeros (never copied)
        const int per_row = SEG / 8, rows = NX - B;
        for (int i = tid; i < NBUF * rows * per_row; i += 256) {
          const int rr = i / per_row, c = i - rr * per_row;
          st_shared16(sbase + (uint32_t)(rr / rows) * bufb + (uint32_t)(NU16 + B + rr % rows) * STR + (uint32_t)c * 16u,
                      make_uint4(0u, 0u, 0u, 0u));
        }
      }
      named_barrier(3, 256);
      const int base = *s_base;
      for (int j = tid; j < nu; j += 256) p.ulist[base + j] = u0 + s_list[j];
      const int KW = max(1, 8 / nrg), rg = warp / KW, kp = warp % KW;
      const bool active = warp < nrg * KW;
      float acc[4][4];
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;
      bool good = true;
      for (int s = 0; s < NSEG; ++s) {
        const int b = s % NBUF;
        if (!__all_sync(0xffffffffu, mbar_wait(&f2[b], (s / NBUF) & 1, abort_flag, err, p.timeout_ns))) {
          good = false;
          break;
        }
        const int len = min(SEG, D - s * SEG), nks = (len + 15) / 16;
        const uint32_t bb = sbase + (uint32_t)b * bufb;
        if (active) {
          if (len & 15) {  // a ragged last segment: zeros in the 8 values past its end in the rows this warp reads
            for (int r = lane; r < 16 + NX; r += 32)
              st_shared16(bb + (uint32_t)(r < 16 ? rg * 16 + r : NU16 + r - 16) * STR + (uint32_t)len * 2u,
                          make_uint4(0u, 0u, 0u, 0u));
            __syncwarp();
          }
          const uint32_t arow = bb + (uint32_t)(rg * 16 + (lane & 15)) * STR + (uint32_t)(lane >> 4) * 16u;
          const uint32_t brow = bb + (uint32_t)(NU16 + (lane & 7)) * STR + (uint32_t)((lane >> 3) & 1) * 16u;
          for (int ks = kp; ks < nks; ks += KW) {
            uint32_t a[4];
            ldsm_x4(arow + (uint32_t)ks * 32u, a);
#pragma unroll
            for (int tg = 0; tg < 4; ++tg)
              if (tg < ntg) {
                uint32_t bf[2];
                ldsm_x2(brow + (uint32_t)(tg * 8) * STR + (uint32_t)ks * 32u, bf);
                mma_bf16_16816(acc[tg], a, bf);
              }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&e2[b]);
      }
      // the partial tiles of every warp, then h = A(z) * p for each (union entry, token)
      named_barrier(3, 256);  // every warp is done with the segment buffers (red lies over them)
      float* red = reinterpret_cast<float*>(sm);  // [8 warps][16 rows][NX + 1]
      const int ldr = NX + 1;
      if (good && active) {
#pragma unroll
        for (int tg = 0; tg < 4; ++tg)
          if (tg < ntg) {
            const int r = lane >> 2, n = tg * 8 + (lane & 3) * 2;
            float* w = red + (size_t)warp * 16 * ldr;
            w[r * ldr + n] = acc[tg][0];
            w[r * ldr + n + 1] = acc[tg][1];
            w[(r + 8) * ldr + n] = acc[tg][2];
            w[(r + 8) * ldr + n + 1] = acc[tg][3];
          }
      }
      named_barrier(3, 256);
      if (good) {
        const bool dbl = (p.flags & FLAG_DOUBLE_ACT) != 0;
        for (int it = tid; it < nu * B; it += 256) {
          const int b = it / nu, j = it - b * nu, g = j >> 4, r = j & 15;
          float pv = 0.f;
          for (int k = 0; k < KW; ++k) pv += red[(size_t)(g * KW + k) * 16 * ldr + r * ldr + b];
          if (dbl) pv = activation(p.act, pv);
          const float hv = s_a[s_list[j] * lda + b] * pv;  // exactly 0 for a dead pair
          p.hbuf[(size_t)b * p.Hs + base + j] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == G_MMA0) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// --------------------------------------------------------------------------- down kernel
// Ring slot, one chunk of UCH union positions: the gathered W2^T row segments
// for y values d0..d0+63 and d0+64..d0+127 (two 8 KB MN-major atom columns:
// row = position, 128 B = 64 y values, swizzled), then the h rows
// [NB rows x 128 B] (K-major: row = token, 64 positions).
__global__ void __launch_bounds__(D_THREADS, 1)
    ffn_tcg_down_kernel(const __grid_constant__ CUtensorMap mH, const DownArgs p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  const int NB = p.NB;
  const uint32_t half = UCH * 128u, slot_b = d_slot_bytes(NB), hbytes = (uint32_t)NB * 128u;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)p.RD * slot_b);
  uint64_t* empty = full + DRING_MAX;
  uint64_t* done = empty + DRING_MAX;
  uint64_t* mdone = done + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mdone + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  int* s_last = reinterpret_cast<int*>(tslot + 2);
  int* s_units = s_last + 2;  // [maxpos] the units of this block's union positions
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool clus = p.cluster != 0;
  const int dt = clus ? blockIdx.x / p.nsplit : blockIdx.x % p.ndt;
  const int sp = clus ? blockIdx.x % p.nsplit : blockIdx.x / p.ndt, d0 = dt * DT;  // sp = rank in the cluster
  const int D = p.D;
  int* err = p.ctrl + CTRL_ERR;

  if (tid == 0) {
    for (int s = 0; s < DRING_MAX; ++s) {
      mbar_init(&full[s], GATHER_THREADS + 1);  // every gathering thread's copies + the h copy
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    mbar_init(mdone, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == D_MMA) tmem_alloc(tslot, p.tmem_cols);
  if (tid == 0) tma_prefetch_map(&mH);
  // the union (its size, units and h) comes from the gate kernel
  pdl_wait();
  int U = __ldcg(p.ucount);
#ifdef SFFN_DEBUG
  if ((unsigned)U > (unsigned)p.H) {
    atomicOr(err, DEV_ERR_CHECK);
    U = 0;
  }
#endif
  const int nchu = (U + UCH - 1) / UCH;
  const int c0 = (int)((long long)sp * nchu / p.nsplit), c1 = (int)((long long)(sp + 1) * nchu / p.nsplit);
  const int nch = c1 - c0;
  const int pos0 = c0 * UCH, npos = min(U, c1 * UCH) - pos0;
  const int nload = min(npos, p.maxpos);
  for (int i0 = tid; i0 < nload; i0 += 4 * D_THREADS) {  // four loads in flight per thread, then the stores
    int u[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) u[e] = i0 + e * D_THREADS < nload ? __ldcg(p.ulist + pos0 + i0 + e * D_THREADS) : 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (i0 + e * D_THREADS >= nload) continue;
#ifdef SFFN_DEBUG
      if ((unsigned)u[e] >= (unsigned)p.H) {
        atomicOr(err, DEV_ERR_CHECK);
        u[e] = 0;
      }
#endif
      s_units[i0 + e * D_THREADS] = u[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) pdl_launch_dependents();
  const int RD = p.RD;
  const uint32_t ring = smem_u32(sm);

  // GCD chunks share a barrier (an arrival per thread and group): about three groups, at least two
  // groups in the ring when it cannot hold every chunk
  const int GCD = max(1, min(RD >= nch ? RD : RD / 2, (nch + 2) / 3));
  const int RSD = max(1, RD / GCD), NGD = (nch + GCD - 1) / GCD;
  auto slot_addr = [&](int c) { return (uint32_t)(((c / GCD) % RSD) * GCD + c % GCD) * slot_b; };

  if (warp < 5) {
    // gatherers: warps 0-3 the W2^T segments (thread: piece k = tid % 8 of y half mh = (tid / 8) % 2,
    // positions tid / 16 + 8 i), warp 4 the h rows
    const int k = tid & 7, mh = (tid >> 3) & 1, i0 = tid >> 4;
    const int d = d0 + 64 * mh + 8 * k;
    int g = 0;
    for (; g < NGD; ++g) {
      const int slot = g % RSD, cb = g * GCD, ncg = min(GCD, nch - cb);
      if (g >= RSD) {
        int w = 1;
        if (lane == 0) w = mbar_wait(&empty[slot], ((g / RSD) - 1) & 1, abort_flag, err, p.timeout_ns);
        if (!__shfl_sync(0xffffffffu, w, 0)) break;
      }
      if (warp < 4) {
        for (int c = cb; c < cb + ncg; ++c) {
          const int pb = (c0 + c) * UCH;  // first union position of the chunk
          const uint32_t sb = ring + slot_addr(c);
          int u[8];
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int pos = pb + i0 + 8 * it;
            u[it] = pos < U ? s_units[pos - pos0] : -1;
          }
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int i = i0 + 8 * it;
            const bool in = u[it] >= 0 && d < D;  // past the union or past D: zeros, contributes nothing
            cp_async16_zfill(sb + (uint32_t)mh * half + (uint32_t)i * 128u + ((uint32_t)(k ^ (i & 7)) << 4),
                             in ? p.W2t + (size_t)u[it] * D + d : p.W2t, in ? 16u : 0u);
          }
        }
      } else {
        // h rows: one TMA per whole chunk (spread over the lanes); the chunk that holds the end of the
        // union by cp.async, zero past the end (the buffer holds stale values there, which
        // 0 * stale must not turn into a NaN)
        const bool ragged = (c0 + cb + ncg) * UCH > U;  // only the union's last chunk can be
        const int nfull = ncg - (ragged ? 1 : 0);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)nfull * hbytes);
        __syncwarp();
        if (lane < nfull)
          tma_tile_2d(sm + slot_addr(cb + lane) + 2 * half, &mH, (c0 + cb + lane) * UCH, 0, &full[slot]);
        if (ragged) {
          const int c = cb + ncg - 1, pb = (c0 + c) * UCH;
          const uint32_t hb = ring + slot_addr(c) + 2 * half;
          for (int t = lane; t < NB * 8; t += 32) {
            const int n = t >> 3, kk = t & 7, pp = pb + 8 * kk;
            const int keep = min(8, max(0, U - pp));  // values of the piece inside the union
            cp_async16_zfill(hb + (uint32_t)n * 128u + ((uint32_t)(kk ^ (n & 7)) << 4),
                             keep > 0 ? p.hbuf + (size_t)n * p.Hs + pp : p.hbuf, 2u * (uint32_t)keep);
          }
        }
      }
      cp_async_arrive_noinc(&full[slot]);
    }
    cp_async_wait_all();
    if (tid == GATHER_THREADS - 32)  // the h copies of the last groups have landed before the block exits
      for (int q = max(0, g - RSD); q < g; ++q) mbar_wait_drain(&full[q % RSD], (q / RSD) & 1, p.timeout_ns);
  } else if (lane == 0) {
    // warp 5: the MMA issuer
    const uint32_t idesc = idesc_bf16_f32(DT, NB, true, false);  // N = the tokens of h
    int gk = 0;
    for (int g = 0; g < NGD; ++g) {
      const int slot = g % RSD, cb = g * GCD, ncg = min(GCD, nch - cb);
      if (!mbar_wait(&full[slot], (g / RSD) & 1, abort_flag, err, p.timeout_ns)) break;
      fence_proxy_async();
      tc_fence_after();
      for (int c = cb; c < cb + ncg; ++c) {
        const uint32_t sb = ring + slot_addr(c);
        // 16 positions per K step: two 8-position K groups of 1 KB; the y halves are `half` bytes apart
        const uint64_t ad0 = smem_desc(sb, half, 1024, SMEM_LAYOUT_SW128);
        const uint64_t bd0 = smem_desc(sb + 2 * half, 16, 1024, SMEM_LAYOUT_SW128);
#pragma unroll
        for (int kk = 0; kk < UCH / 16; ++kk, ++gk)
          tc_mma(tmem + (uint32_t)(gk & (p.nacc - 1)) * (uint32_t)NB, ad0 + (kk * 2048 >> 4), bd0 + 2 * kk, idesc,
                 gk >= p.nacc);
      }
      tc_commit(&empty[slot]);
    }
    tc_commit(done);
    tc_commit(mdone);
    mbar_wait_drain(mdone, 0, p.timeout_ns);
  }
  __syncwarp();
  if (warp < 4) {
    // ---- epilogue warps 0..3: lane = one y value of the slice
    if (blockIdx.x == 0 && tid < p.B) {  // the gate kernel is complete: publish the live counts
      p.counts[tid] = __ldcg(p.ctrl + CTRL_COUNT + tid);
      __stcg(p.ctrl + CTRL_COUNT + tid, 0);
    }
    const int d = d0 + 32 * warp + lane;
    const int used = min(p.nacc, nch * (UCH / 16));  // accumulators that received a K step
    const bool okd = nch > 0 && __all_sync(0xffffffffu, mbar_wait(done, 0, abort_flag, err, p.timeout_ns));
    // cluster form: the partial tile goes to the drained ring token-major (zero for a block with no
    // union chunk), for the reduction after the warp roles end
    float* s_y = reinterpret_cast<float*>(sm) + 32 * warp + lane;
    if (okd) {
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
      float* ya = p.yacc + d;
      for (int cc = 0; cc < NB; cc += 16) {
        float v[16];
        tmem_ld_sum(tl + cc, NB, used, v);
        if (clus) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) s_y[(size_t)(cc + jj) * Y_LD] = v[jj];
        } else if (d < D) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (cc + jj < p.B) atomicAdd(ya + (size_t)(cc + jj) * YACC_COPIES * D, v[jj]);
        }
      }
    } else if (clus && nch == 0) {
      for (int c = 0; c < NB; ++c) s_y[(size_t)c * Y_LD] = 0.f;
    }
    // the last block of this y slice rounds the sum into y and clears the accumulator
    if (!clus) {
      __threadfence();
      named_barrier(1, 128);
      if (tid == 0) *s_last = atomicAdd(p.tickets + dt, 1) == p.nsplit - 1;
      named_barrier(1, 128);
      if (*s_last) {
        __threadfence();
        if (d < D) {
          float* ya = p.yacc + d;
          __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y) + d;
          for (int b0 = 0; b0 < p.B; b0 += 16) {  // 16 loads in flight, then the stores
            float v[16];
  #pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = b0 + j < p.B ? __ldcg(ya + (size_t)(b0 + j) * YACC_COPIES * D) : 0.f;
  #pragma unroll
            for (int j = 0; j < 16; ++j)
              if (b0 + j < p.B) {
                __stcg(ya + (size_t)(b0 + j) * YACC_COPIES * D, 0.f);
                y[(size_t)(b0 + j) * D] = __float2bfloat16_rn(v[j]);
              }
          }
        }
        if (tid == 0) p.tickets[dt] = 0;
      }
    }
  }
  if (clus) {
    // after the cluster barrier block sp sums the slice's nsplit tiles for its share of the tokens
    // (16-byte items read through distributed shared memory) and rounds them into y; the second
    // barrier keeps every tile in place until all blocks have read it
    __syncwarp();
    cluster_sync_all();
    const int B = p.B, ns = p.nsplit;
    const int b0 = (int)((long long)sp * B / ns), b1 = (int)((long long)(sp + 1) * B / ns);
    const int items = (b1 - b0) * (DT / 4);
    const uint32_t base = smem_u32(sm);
    uint16_t* const yo = static_cast<uint16_t*>(p.y);
    for (int i = tid; i < items; i += D_THREADS) {
      const int b = b0 + i / (DT / 4), j = 4 * (i % (DT / 4));
      const uint32_t off = base + (uint32_t)((b * Y_LD + j) * 4);
      float4 v[8];
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r0 = 0; r0 < ns; r0 += 8) {  // up to eight loads in flight
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r0 + r < ns) v[r] = ld_cluster_f4(cluster_map(off, (uint32_t)(r0 + r)));
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r0 + r < ns) {
            acc.x += v[r].x;
            acc.y += v[r].y;
            acc.z += v[r].z;
            acc.w += v[r].w;
          }
      }
      if (d0 + j < D) {  // D is a multiple of 8: the whole quad is in range
        const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc.x)) |
                            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.y)) << 16);
        const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc.z)) |
                            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.w)) << 16);
        *reinterpret_cast<uint2*>(yo + (size_t)b * D + d0 + j) = make_uint2(lo, hi);
      }
    }
    cluster_sync_all();
  }
  tc_fence_before();
  __syncthreads();
  // every block has read the union count: the last one resets it for the next call
  if (tid == 0 && atomicAdd(p.dticket, 1) == (int)gridDim.x - 1) {
    __stcg(p.ucount, 0);
    __stcg(p.dticket, 0);
  }
  if (warp == D_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

uint32_t tmem_cols_pow2(int n) {
  uint32_t c = 32;
  while (c < (uint32_t)n) c <<= 1;
  return c;
}

}  // namespace

cudaError_t ffn_tcg_plan_cluster(TcPlan& plan, size_t max_smem) {
  plan.tcg_down_cluster = 0;
  if (!plan.ok || plan.ndt < 1) return cudaSuccess;
  for (int cs = std::min(std::min(8, plan.nch), plan.num_sms / plan.ndt); cs >= 2; --cs) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.ndt * cs);
    cfg.blockDim = dim3(D_THREADS);
    cfg.dynamicSmemBytes = max_smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = (unsigned)cs;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, ffn_tcg_down_kernel, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      continue;
    }
    if (n >= plan.ndt) {
      plan.tcg_down_cluster = cs;
      break;
    }
  }
  return cudaSuccess;
}

cudaError_t ffn_tcg_prepare(size_t max_smem) {
  cudaError_t e =
      cudaFuncSetAttribute(ffn_tcg_gate_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
  if (!e) e = cudaFuncSetAttribute(ffn_tcg_gate_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
  if (!e) e = cudaFuncSetAttribute(ffn_tcg_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
  return e;
}

int launch_ffn_tcg(const TcPlan& plan, const TcMaps& maps, const TcBuffers& buf, const TcgBuffers& ub, const void* W3,
                   const void* W2t, const void* x, void* y, int D, int H, int B, int act, int flags, float thr,
                   unsigned long long timeout_ns, size_t max_smem, cudaStream_t s, cudaError_t* cuda_err) {
  *cuda_err = cudaSuccess;
  const bool lopa = plan.r > 0;
  if (!plan.ok || B < 1 || B > TCG_MAX_BATCH || plan.NU > 128 || !ub.ulist || !ub.ucount || !ub.dticket ||
      (lopa && !buf.tpair))
    return -1;
  const int NB = (B + 15) / 16 * 16;
  // phase 1's B operand: x [B, D], or the low-rank gate's t pair [2 NB, r] (written before this launch)
  CUtensorMap mx;
  if (int rc = lopa ? encode_2d(&mx, buf.tpair, (uint64_t)(2 * NB), (uint64_t)plan.r, (uint64_t)plan.r * 2,
                                (uint32_t)(2 * NB))
                    : encode_2d(&mx, x, (uint64_t)B, (uint64_t)D, (uint64_t)D * 2, (uint32_t)NB))
    return rc;
  const size_t budget = std::min(max_smem, SMEM_BUDGET);
  GateArgs g;
  g.D = D;
  g.H = H;
  g.B = B;
  g.NB = NB;
  g.NU = plan.NU;
  g.KC = lopa ? plan.KCZ : plan.KC;  // phase 1's 64-wide K chunks (over r or D)
  g.XR = lopa ? 2 * NB : NB;
  g.C = 4;
  while (g.C > 1 && g_smem_bytes(g.C, g.NU, NB, g.XR, 2) > budget) g.C >>= 1;
  g.NCG = (g.KC + g.C - 1) / g.C;
  g.NS = 2;
  // phase 1 keeps up to NS_MAX stages; phase 2's ring spans all of them
  while (g.NS < NS_MAX && g_smem_bytes(g.C, g.NU, NB, g.XR, g.NS + 1) <= budget) ++g.NS;
  g.act = act;
  g.flags = flags;
  g.thr = thr;
  g.Hs = plan.Hs;
  g.nacc = 4;
  g.apw = std::max(1, std::min(plan.tcg_acc, 64 / NB));  // at most 256 TMEM columns
  g.tmem_cols = tmem_cols_pow2(g.nacc * g.apw * NB);
  g.W3 = static_cast<const uint16_t*>(W3);
  g.W2t = static_cast<const uint16_t*>(W2t);
  g.x = static_cast<const uint16_t*>(x);
  g.NX = (B + 7) / 8 * 8;
  {  // phase 2: NBUF segment buffers of the largest possible union (every unit of a slice) fit over the stages
    const uint32_t area = (uint32_t)g.NS * g_stage_bytes(g.C, g.NU, g.XR) + g_slack_bytes(g.C, g.NU, g.XR);
    if (g_segment(area, (g.NU + 15) / 16 * 16, g.NX) == 0 || 8u * 16u * (uint32_t)(g.NX + 1) * 4u > area) {
      *cuda_err = cudaErrorInvalidConfiguration;
      return 0;
    }
  }
  g.ctrl = buf.ctrl;
  g.mask = buf.mask;
  g.hbuf = buf.hbuf;
  g.ulist = ub.ulist;
  g.ucount = ub.ucount;
  g.timeout_ns = timeout_ns;
  const size_t smem1 = g_smem_bytes(g.C, g.NU, NB, g.XR, g.NS);
  // the epilogue's copy of Z ([128][NB + 1] fp32) lies over the stages
  if (smem1 > max_smem || (size_t)g.NS * g_stage_bytes(g.C, g.NU, g.XR) < (size_t)128 * (NB + 1) * 4) {
    *cuda_err = cudaErrorInvalidConfiguration;
    return 0;
  }
  cudaError_t e = lopa ? launch_pdl(ffn_tcg_gate_kernel<true>, dim3(plan.ntiles), dim3(G_THREADS), smem1, s, maps.w1,
                                    mx, g)
                       : launch_pdl(ffn_tcg_gate_kernel<false>, dim3(plan.ntiles), dim3(G_THREADS), smem1, s, maps.w1,
                                    mx, g);
  if (e) {
    *cuda_err = e;
    return 0;
  }
  DownArgs d;
  d.D = D;
  d.H = H;
  d.B = B;
  d.NB = NB;
  d.ndt = plan.ndt;
  d.cluster = plan.tcg_down_cluster > 0 ? 1 : 0;
  d.nsplit = d.cluster ? plan.tcg_down_cluster : plan.nsplit;
  d.Hs = plan.Hs;
  d.maxpos = (plan.nch + d.nsplit - 1) / d.nsplit * UCH;  // the union has at most nch chunks
  d.RD = 2;
  while (d.RD < DRING_MAX && d.RD * UCH < d.maxpos && d_smem_bytes(NB, d.RD + 1, d.maxpos) <= budget) ++d.RD;
  d.nacc = 8;  // a power of two, nacc * NB <= 256 TMEM columns (NB <= 32)
  d.tmem_cols = tmem_cols_pow2(d.nacc * NB);
  d.W2t = static_cast<const uint16_t*>(W2t);
  d.hbuf = buf.hbuf;
  d.ulist = ub.ulist;
  d.ucount = ub.ucount;
  d.dticket = ub.dticket;
  d.yacc = buf.yacc;
  d.y = y;
  d.ctrl = buf.ctrl;
  d.counts = buf.counts;
  d.tickets = buf.tickets;
  d.timeout_ns = timeout_ns;
  const size_t smem2 = d_smem_bytes(NB, d.RD, d.maxpos);
  if (smem2 > max_smem) {
    *cuda_err = cudaErrorInvalidConfiguration;
    return 0;
  }
  if (d.cluster)
    *cuda_err = launch_pdl_cluster(ffn_tcg_down_kernel, dim3(plan.ndt * d.nsplit), dim3(D_THREADS), smem2, s,
                                   (unsigned)d.nsplit, maps.h[NB / 16 - 1], d);
  else
    *cuda_err = launch_pdl(ffn_tcg_down_kernel, dim3(plan.ndt * d.nsplit), dim3(D_THREADS), smem2, s,
                           maps.h[NB / 16 - 1], d);
  return 0;
}

}  // namespace sffn
