// ffn_tc.cu -- gate-first FFN for a batch of tokens on the tensor cores (bf16
// weights and tokens, fp32 accumulation, standard or low-rank gate).
//
// Per token b the method is unchanged ("Model casting: compute the gate, then
// skip most of the FFN", section "What an FFN actually computes"):
//     y_b = sum_{i : z_bi > 0} W2[:, i] * A(z_bi) * (W3[i, :] . x_b),  z_b = W1 x_b.
// With B tokens a unit's W3 row and W2 column are needed when ANY token keeps
// it -- the union of the live sets, which the pages warn grows with the batch
// (at 90 % sparsity it holds 57 % of the units at B = 8 and 82 % at B = 16).
// From a handful of tokens up, this path therefore streams every unit slice
// and lets the gate decide, per token and unit, what reaches y (the union-skip
// kernels of ffn_tcg.cu take small batches whose union is small):
//
//   gate-up kernel, one block per slice of NU units:
//     [Z ; P][slice, :] = [W1 ; W3][slice, :] X^T   one pass; the W1 and W3 rows
//                                                   of a K chunk sit back to back,
//                                                   so one M = 128 MMA per K step
//                                                   serves both products (NU <= 64;
//                                                   two MMAs otherwise)
//     epilogue: live = z > 0, per-token counts and flags, and
//               h = A(z) * p where live, else exactly 0, rounded to bf16 (the
//               precision of a dense bf16 FFN's intermediate): hbuf row b
//   down kernel, one block per (128-wide slice of y, range of units):
//     y^T[d-slice, :] += W2^T[units, d-slice]^T h   MN-major A (W2^T rows as
//               stored), h the N = NB operand (one TMA box of NB rows);
//               the blocks of a y slice form a thread-block cluster and sum
//               their partial tiles through distributed shared memory, each
//               rounding its share of the tokens into y (where the clusters do
//               not fit: fp32 atomics into an accumulator and a last block per
//               slice, found by a ticket); block 0 publishes the live counts.
//
// Low-rank gate ("LoPA Gating: moving the ceiling", W1 = UV), three kernels:
//   t kernel: the gate-up kernel's low-rank form with no U chunks and V in
//             place of W3, so it computes T = V X^T; its blocks split K: one
//             block per (128 rows of V, range of D), the splits of a row tile
//             one cluster summing through distributed shared memory (else
//             fp32 atomics and a last block), which store t_b as a bf16 pair,
//             t_hi in rows [0, NB) and t_lo in rows [NB, 2 NB) of one buffer;
//   gate-up:  the first K chunk groups run over the r columns of U, two MMAs
//             per K step into the Z accumulator (U t_hi, then U t_lo), the
//             remaining groups over the D columns of W3 into the P accumulator;
//             the accumulator layout is the unfused one, so the epilogue and
//   down:     the down kernel are the standard gate's.
//
// All operands move by 2D TMA tiles with 128-byte swizzle, several tiles per
// pipeline stage (one lane of a producer warp issues them, one lane of an MMA
// warp issues tcgen05.mma; the stage is released by tcgen05.commit).  The
// weights of the first stages are requested before the dependency wait.  The
// K steps of a product go round-robin over `nacc` TMEM accumulators (summed
// by the epilogue): small MMAs into one accumulator form a serial chain whose
// latency, not the tensor pipe, would set the pace.
// Ragged edges (units past H, y past D, K past D) are zero-filled by the TMA
// unit; MMA rows past NU read neighbouring shared memory and land in TMEM
// lanes the epilogue never reads.  Every wait is bounded (error word + early
// exit), and a block drains its copies and MMAs before it releases TMEM.
#include <cudaTypedefs.h>

#include <algorithm>

#include "internal.h"
#include "tc.cuh"

namespace sffn {

namespace {

constexpr int TC_THREADS = 192;  // down kernel: warps 0-3 epilogue, 4 TMA producer, 5 MMA issuer
// gate-up kernel: warps 0-3 epilogue, 4 TMA producer, 5-8 MMA issuers.  An MMA
// costs its issuing thread on the order of 150 cycles however small it is, so
// the K steps of a chunk are split over up to four issuing warps, each into its
// own TMEM accumulator.
constexpr int TC_GATE_THREADS = 288;
constexpr int TC_GATE_MMA_WARP0 = 5;
constexpr int TC_PRODUCER_WARP = 4;
constexpr int TC_MMA_WARP = 5;
constexpr int TC_DTILE = 128;    // y values per down-kernel block (MMA M)
constexpr int TC_UCH = 64;       // units per down-kernel K chunk (one TMA box)
constexpr int TC_DC = 2;         // unit chunks per down-kernel stage
constexpr size_t TC_SMEM_BUDGET = 200 * 1024;
constexpr int TC_NS_MAX = 8;

struct TcGateArgs {
  int D, H, B, NB, NU, KC, C, NCG, NS, act, Hs, nacc, flags;
  int KCZ, NCZ;          // low-rank gate: K chunks of r and the chunk groups they fill (the first NCZ)
  const uint16_t* x;     // [B, D] bf16 bits (the tiled identity G of the low-rank gate)
  uint16_t* tout;        // t kernel: the t pair [2 NB, H] (H = r) instead of h, masks and counts
  int ksplit;            // blocks per slice, each over a range of the K chunks (the t kernel; else 1)
  int tcluster;          // t kernel: the ksplit blocks of a slice are a cluster and sum in distributed
                         // shared memory (1), or add into tacc with a ticket and a last block (0)
  float* tacc;           // t kernel: [B, H] fp32 partial sums, zero between calls
  int* tickets;          // t kernel: [slices] blocks done, zero between calls
  float thr;  // live iff |A(z)| > thr
  uint32_t tmem_cols;
  int* ctrl;
  uint8_t* mask;
  uint16_t* hbuf;  // [256][Hs] bf16 bits: h of token b in row b
  unsigned long long timeout_ns;
};

struct TcDownArgs {
  int D, B, NB, nch, ndt, nsplit, NS, nacc;
  int cluster;  // 1: the nsplit blocks of a slice are a cluster (block = dt * nsplit + sp) and sum in
                // distributed shared memory; 0: block = sp * ndt + dt, fp32 atomics and a last block
  uint32_t tmem_cols;
  float* yacc;  // [B_max * YACC_COPIES, D]; the atomic form uses copy 0, zero between calls
  void* y;      // [B, D] bf16
  int* ctrl;
  int* counts;  // [B] published live counts
  int* tickets; // [ndt] blocks of a y slice done, zero between calls
  unsigned long long timeout_ns;
};

__host__ __device__ constexpr uint32_t gate_stage_bytes(int C, int NU, int NB) {
  return (uint32_t)C * 128u * (uint32_t)(2 * NU + NB);
}
// The epilogue's copy of the accumulator, transposed: [2 NB columns][TC_ACC_LD]
// fp32 (128 TMEM lanes, padded so that every column starts 16-byte aligned and
// a warp's 16-byte reads of neighbouring columns fall in different banks).
constexpr int TC_ACC_LD = 132;
__host__ __device__ constexpr size_t tc_acc_copy_bytes(int NB) { return (size_t)2 * NB * TC_ACC_LD * 4; }
__host__ __device__ constexpr uint32_t down_chunk_bytes(int NB) { return 2u * TC_UCH * 128u + (uint32_t)NB * 128u; }

// Bytes an MMA may read past the last A region of the last stage: it reads
// 128 rows (2 NU <= 128, W1 and W3 stacked) or MT rows from a chunk's start,
// and what follows the last A region is the stage's x regions.
__host__ __device__ inline uint32_t gate_slack_bytes(int C, int MT, int NU, int NB) {
  const int rows = 2 * NU <= 128 ? 128 - 2 * NU : MT - NU;
  const int over = rows * 128 - C * NB * 128;
  return over > 0 ? (uint32_t)(over + 1023) / 1024 * 1024 : 0u;
}
size_t gate_smem_bytes(int C, int MT, int NU, int NB, int NS) {
  return 1024 + (size_t)NS * gate_stage_bytes(C, NU, NB) + gate_slack_bytes(C, MT, NU, NB) + 8 * (2 * NS + 2) + 8 +
         4 * NB + 64;
}
// Low-rank stages: A regions [C][NU x 128 B] (U or W3 rows), then max(C, 2) B
// regions of [NB x 128 B].  A group of W3 chunks fills C A regions and C B
// regions (x); a group of U chunks fills lopa_zchunks(C) A regions and two B
// regions per chunk (t_hi, t_lo): the t pair's rows do not take stage space
// from the 40-odd W3 groups that follow.  An MMA reads MT rows from an A
// region's start; past the last one lie the B regions.
__host__ __device__ constexpr int lopa_zchunks(int C) { return C >= 2 ? C / 2 : 1; }
__host__ __device__ constexpr uint32_t lopa_stage_bytes(int C, int NU, int NB) {
  return 128u * (uint32_t)(C * NU + (C >= 2 ? C : 2) * NB);
}
__host__ __device__ inline uint32_t lopa_slack_bytes(int C, int MT, int NU, int NB) {
  const int over = (MT - NU) * 128 - (C >= 2 ? C : 2) * NB * 128;
  return over > 0 ? (uint32_t)(over + 1023) / 1024 * 1024 : 0u;
}
size_t lopa_smem_bytes(int C, int MT, int NU, int NB, int NS) {
  return 1024 + (size_t)NS * lopa_stage_bytes(C, NU, NB) + lopa_slack_bytes(C, MT, NU, NB) + 8 * (2 * NS + 2) + 8 +
         4 * NB + 64;
}
size_t down_smem_bytes(int NB, int NS) {
  return 1024 + (size_t)NS * TC_DC * down_chunk_bytes(NB) + 8 * (2 * NS + 2) + 8 + 64;
}

uint32_t tmem_cols_for(int n) {
  uint32_t c = 32;
  while (c < (uint32_t)n) c <<= 1;
  return c;
}

// Round a dynamic shared-memory pointer up to 1024 bytes by pointer arithmetic
// (an integer round trip would hide the shared address space from the
// compiler and turn every access through the result into a generic one).
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// --------------------------------------------------------------------------- gate-up kernel
// Stage layout: per 64-wide K chunk c, W1 rows [NU x 128 B] then W3 rows
// [NU x 128 B]; then X regions [C][NB x 128 B].  K chunk group q covers chunks
// q*C .. q*C+C-1.  TMEM: fused (2 NU <= 128): lanes [0, NU) = Z, [NU, 2 NU) =
// P, NB columns; otherwise lanes [0, NU), Z in columns [0, NB), P in [NB, 2 NB).
// LOPA: mW1 maps U [H, r] and mT the t pair [2 NB, r]; the stages hold the
// low-rank layout (lopa_stage_bytes) and TMEM the unfused one.
template <int MT, bool LOPA>
__global__ void __launch_bounds__(TC_GATE_THREADS, 1)
    ffn_tc_gateup_kernel(const __grid_constant__ CUtensorMap mW1, const __grid_constant__ CUtensorMap mW3,
                         const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mT,
                         const TcGateArgs p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  const int NS = p.NS, NB = p.NB, C = p.C;
  const uint32_t wreg = (uint32_t)p.NU * 128u, xreg = (uint32_t)NB * 128u;
  const uint32_t st_bytes = LOPA ? lopa_stage_bytes(C, p.NU, NB) : gate_stage_bytes(C, p.NU, NB);
  const uint32_t slack = LOPA ? lopa_slack_bytes(C, MT, p.NU, NB) : gate_slack_bytes(C, MT, p.NU, NB);
  // stages, then slack for the rows an MMA reads past the last A region
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)NS * st_bytes + slack);
  uint64_t* empty = full + NS;
  uint64_t* done = empty + NS;  // every MMA complete (one commit per MMA warp)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  int* s_cnt = reinterpret_cast<int*>(tslot + 2);  // [NB] live counts of this slice
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x / p.ksplit, split = blockIdx.x - tile * p.ksplit;
  const int u0 = tile * p.NU;
  // this block's K chunks of the D-wide product: a range when the t kernel splits K, else all of them
  const int kc0 = (int)((long long)split * p.KC / p.ksplit), kc1 = (int)((long long)(split + 1) * p.KC / p.ksplit);
  const int NCG = p.NCZ + (kc1 - kc0 + C - 1) / C;
  int* err = p.ctrl + CTRL_ERR;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], p.nacc);  // one commit per MMA warp
    }
    mbar_init(done, p.nacc);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < NB) s_cnt[tid] = 0;
  if (warp == TC_GATE_MMA_WARP0) tmem_alloc(tslot, p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // Let the next kernel launch only once this block holds its TMEM: a later
  // kernel's blocks then never take the columns an earlier one still needs.
  if (tid == 0) pdl_launch_dependents();
  const bool fused = !LOPA && 2 * p.NU <= 128;
  const int ncol = fused ? NB : 2 * NB;  // accumulator columns the epilogue copies
  float* s_acc = reinterpret_cast<float*>(sm);
  int stage_ok = 1;

  if (warp == TC_PRODUCER_WARP) {
    // One TMA copy costs the issuing thread on the order of 100 ns, so the
    // copies of a stage are spread over the warp's lanes: lane l issues copy l.
    if (lane == 0) {
      tma_prefetch_map(&mW1);
      tma_prefetch_map(&mW3);
      tma_prefetch_map(&mX);
      if (LOPA) tma_prefetch_map(&mT);
    }
    if constexpr (LOPA) {
      // groups [0, NCZ): U and t chunks (K over r, CZ per group); then W3 and x chunks (K over D)
      const int CZ = lopa_zchunks(C);
      auto zgroup = [&](int q) { return q < p.NCZ; };
      auto kbase = [&](int q) { return zgroup(q) ? q * CZ : kc0 + (q - p.NCZ) * C; };
      auto nchunks = [&](int q) { return zgroup(q) ? min(CZ, p.KCZ - q * CZ) : min(C, kc1 - kbase(q)); };
      auto breg = [&](int q, int c) { return C * wreg + (uint32_t)c * (zgroup(q) ? 2u : 1u) * xreg; };
      auto tx = [&](int q) { return (uint32_t)nchunks(q) * (wreg + (zgroup(q) ? 2u : 1u) * xreg); };
      const int npre = min(NS, NCG);
      for (int q = 0; q < npre; ++q) {  // weights first, before the dependency wait
        uint8_t* st = sm + (size_t)q * st_bytes;
        if (lane == 0) mbar_arrive_expect_tx(&full[q], tx(q));
        __syncwarp();
        if (lane < nchunks(q))
          tma_tile_2d(st + lane * wreg, zgroup(q) ? &mW1 : &mW3, (kbase(q) + lane) * 64, u0, &full[q]);
      }
      pdl_wait();  // t and x come from earlier kernels
      for (int q = 0; q < npre; ++q)
        if (lane < nchunks(q))
          tma_tile_2d(sm + (size_t)q * st_bytes + breg(q, lane), zgroup(q) ? &mT : &mX, (kbase(q) + lane) * 64, 0,
                      &full[q]);
      int issued = npre;
      for (int q = npre; q < NCG; ++q) {
        const int s = q % NS;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&empty[s], ((q / NS) - 1) & 1, abort_flag, err, p.timeout_ns);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        uint8_t* st = sm + (size_t)s * st_bytes;
        const int nc = nchunks(q);
        if (lane == 0) mbar_arrive_expect_tx(&full[s], tx(q));
        __syncwarp();
        if (lane < 2 * nc) {
          const int c = lane >> 1, kb = (kbase(q) + c) * 64;
          if ((lane & 1) == 0)
            tma_tile_2d(st + c * wreg, zgroup(q) ? &mW1 : &mW3, kb, u0, &full[s]);
          else
            tma_tile_2d(st + breg(q, c), zgroup(q) ? &mT : &mX, kb, 0, &full[s]);
        }
        issued = q + 1;
      }
      if (lane == 0)
        for (int q = max(0, issued - NS); q < issued; ++q) mbar_wait_drain(&full[q % NS], (q / NS) & 1, p.timeout_ns);
      __syncwarp();
    } else {
    auto nchunks = [&](int q) { return min(C, p.KC - q * C); };
    const int npre = min(NS, p.NCG);
    // the weights do not depend on the previous kernel: request them first
    for (int q = 0; q < npre; ++q) {
      uint8_t* st = sm + (size_t)q * st_bytes;
      const int nc = nchunks(q);
      if (lane == 0) mbar_arrive_expect_tx(&full[q], (uint32_t)nc * (2 * wreg + xreg));
      __syncwarp();
      if (lane < 2 * nc)
        tma_tile_2d(st + lane * wreg, (lane & 1) ? &mW3 : &mW1, (q * C + (lane >> 1)) * 64, u0, &full[q]);
    }
    pdl_wait();
    for (int q = 0; q < npre; ++q)
      if (lane < nchunks(q))
        tma_tile_2d(sm + (size_t)q * st_bytes + 2 * C * wreg + lane * xreg, &mX, (q * C + lane) * 64, 0, &full[q]);
    int issued = npre;
    for (int q = npre; q < p.NCG; ++q) {
      const int s = q % NS;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&empty[s], ((q / NS) - 1) & 1, abort_flag, err, p.timeout_ns);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint8_t* st = sm + (size_t)s * st_bytes;
      const int nc = nchunks(q);
      if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)nc * (2 * wreg + xreg));
      __syncwarp();
      if (lane < 3 * nc) {
        const int c = lane / 3, k = lane - 3 * c;  // k: 0 W1, 1 W3, 2 x
        if (k < 2)
          tma_tile_2d(st + (2 * c + k) * wreg, k ? &mW3 : &mW1, (q * C + c) * 64, u0, &full[s]);
        else
          tma_tile_2d(st + 2 * C * wreg + c * xreg, &mX, (q * C + c) * 64, 0, &full[s]);
      }
      issued = q + 1;
    }
    if (lane == 0)
      for (int q = max(0, issued - NS); q < issued; ++q) mbar_wait_drain(&full[q % NS], (q / NS) & 1, p.timeout_ns);
    __syncwarp();
    }
  } else if (warp >= TC_GATE_MMA_WARP0) {
    const int mw = warp - TC_GATE_MMA_WARP0;  // this warp issues K steps kk = mw (mod nacc) into accumulator mw
    if (mw < p.nacc && lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(fused ? 128 : MT, NB, false, false);
      const uint32_t acc_cols = fused ? (uint32_t)NB : 2u * NB;  // columns of one accumulator
      const uint32_t da = tmem + (uint32_t)mw * acc_cols;
      bool started = false;
      if constexpr (LOPA) {
        bool started_p = false;
        for (int q = 0; q < NCG; ++q) {
          const int s = q % NS;
          if (!mbar_wait(&full[s], (q / NS) & 1, abort_flag, err, p.timeout_ns)) break;
          tc_fence_after();
          const uint32_t sa = smem_u32(sm + (size_t)s * st_bytes);
          const uint64_t a0 = smem_desc(sa, 16, 1024, SMEM_LAYOUT_SW128);
          const uint64_t b0 = smem_desc(sa + C * wreg, 16, 1024, SMEM_LAYOUT_SW128);
          const bool zq = q < p.NCZ;
          const int CZ = lopa_zchunks(C);
          const int nc = zq ? min(CZ, p.KCZ - q * CZ) : min(C, kc1 - (kc0 + (q - p.NCZ) * C));
          for (int c = 0; c < nc; ++c) {
            const uint64_t ac = a0 + ((c * wreg) >> 4), bc = b0 + ((c * (zq ? 2 : 1) * xreg) >> 4);
            for (int kk = mw; kk < 4; kk += p.nacc) {
              if (zq) {  // z += U t_hi + U t_lo
                tc_mma(da, ac + 2 * kk, bc + 2 * kk, idesc, started);
                tc_mma(da, ac + 2 * kk, bc + (xreg >> 4) + 2 * kk, idesc, true);
                started = true;
              } else {   // p += W3 x
                tc_mma(da + (uint32_t)NB, ac + 2 * kk, bc + 2 * kk, idesc, started_p);
                started_p = true;
              }
            }
          }
          tc_commit(&empty[s]);
        }
      } else {
      for (int q = 0; q < p.NCG; ++q) {
        const int s = q % NS;
        if (!mbar_wait(&full[s], (q / NS) & 1, abort_flag, err, p.timeout_ns)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(sm + (size_t)s * st_bytes);
        const uint64_t a0 = smem_desc(sa, 16, 1024, SMEM_LAYOUT_SW128);
        const uint64_t b0 = smem_desc(sa + 2 * C * wreg, 16, 1024, SMEM_LAYOUT_SW128);
        const int nc = min(C, p.KC - q * C);
        for (int c = 0; c < nc; ++c) {
          // descriptors advance by adds (16-byte units): no divisions on the issue path
          const uint64_t ac = a0 + ((2 * c * wreg) >> 4), bc = b0 + ((c * xreg) >> 4);
          for (int kk = mw; kk < 4; kk += p.nacc) {
            tc_mma(da, ac + 2 * kk, bc + 2 * kk, idesc, started);
            if (!fused) tc_mma(da + (uint32_t)NB, ac + (wreg >> 4) + 2 * kk, bc + 2 * kk, idesc, started);
            started = true;
          }
        }
        tc_commit(&empty[s]);
      }
      }
      tc_commit(done);
      mbar_wait_drain(done, 0, p.timeout_ns);  // every MMA warp's work complete before TMEM is released
    }
    __syncwarp();
  } else {
    // ---- warps 0..3: warp q copies TMEM lanes 32q..32q+31 (summing the
    // accumulators) into a shared [128 lanes][ncol] array; the stages are free
    // once every MMA is done
    pdl_wait();  // the outputs below may still be read by the previous forward
    stage_ok = __all_sync(0xffffffffu, mbar_wait(done, 0, abort_flag, err, p.timeout_ns));
    if (stage_ok) {
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
      float* col = s_acc + 32 * warp + lane;  // transposed: column c at s_acc[c * TC_ACC_LD]
      for (int c0 = 0; c0 < ncol; c0 += 16) {
        float v[16];
        tmem_ld_sum(tl + c0, ncol, p.nacc, v);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) col[(size_t)(c0 + jj) * TC_ACC_LD] = v[jj];
      }
    }
  }
  // ---- epilogue on warps 0..7: thread (unit r, token group g = tid / 64) takes
  // tokens g, g + 4, ... (units in rounds of 64); a warp shares each token, so
  // the counts are ballots
  if (LOPA && p.tout && p.tcluster) {
    // t kernel, cluster form: the slice's ksplit blocks (cluster ranks = splits) hold their partials
    // of T = V X^T in the transposed copy (columns NB + b); after the cluster barrier, block k sums
    // the partials of its share of the (token, four rows) items through distributed shared memory
    // and stores them as bf16 pairs (zero for the padding tokens, so the gate's MMA columns stay
    // finite); the second barrier keeps every copy in place until all blocks have read it.
    __syncwarp();
    cluster_sync_all();
    const int ks = p.ksplit, nq = p.NU / 4, total = NB * nq;
    const int i0 = (int)((long long)split * total / ks), i1 = (int)((long long)(split + 1) * total / ks);
    const uint32_t base = smem_u32(s_acc);
    for (int i = i0 + tid; i < i1; i += TC_GATE_THREADS) {
      const int b = i / nq, r = 4 * (i - b * nq), u = u0 + r;
      if (u >= p.H) continue;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (b < p.B) {
        const uint32_t off = base + (uint32_t)(((NB + b) * TC_ACC_LD + r) * 4);
        float4 v[8];
        for (int q0 = 0; q0 < ks; q0 += 8) {  // up to eight loads in flight
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q0 + q < ks) v[q] = ld_cluster_f4(cluster_map(off, (uint32_t)(q0 + q)));
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q0 + q < ks) {
              acc.x += v[q].x;
              acc.y += v[q].y;
              acc.z += v[q].z;
              acc.w += v[q].w;
            }
        }
      }
      const float tv[4] = {acc.x, acc.y, acc.z, acc.w};
      uint16_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat16 h = __float2bfloat16_rn(tv[k]);
        hi[k] = __bfloat16_as_ushort(h);
        lo[k] = __bfloat16_as_ushort(__float2bfloat16_rn(tv[k] - __bfloat162float(h)));
      }
      *reinterpret_cast<uint2*>(p.tout + (size_t)b * p.H + u) =
          make_uint2(hi[0] | ((uint32_t)hi[1] << 16), hi[2] | ((uint32_t)hi[3] << 16));
      *reinterpret_cast<uint2*>(p.tout + (size_t)(NB + b) * p.H + u) =
          make_uint2(lo[0] | ((uint32_t)lo[1] << 16), lo[2] | ((uint32_t)lo[3] << 16));
    }
    cluster_sync_all();
  } else if (LOPA && p.tout) {
    // t kernel: this block's partial of T = V X^T (its rows of V, its range of
    // D) into the fp32 sums; the last block of the row tile stores the sums as
    // bf16 pairs (zero rows for the padding tokens, so the gate's MMA columns
    // stay finite) and clears them
    if (__syncthreads_and(stage_ok) && warp < 8) {
      // four consecutive rows of one token per 128-bit atomic (r and the slice starts are multiples of 8)
      const int nq = p.NU / 4;
      for (int i = tid; i < p.B * nq; i += 256) {
        const int b = i / nq, r = 4 * (i - b * nq), u = u0 + r;
        if (u < p.H) {
          atomicAdd(reinterpret_cast<float4*>(p.tacc + (size_t)b * p.H + u),
                    *reinterpret_cast<const float4*>(s_acc + (size_t)(NB + b) * TC_ACC_LD + r));
        }
      }
    }
    __threadfence();
    __syncthreads();
    volatile int* s_last = s_cnt;
    if (tid == 0) *s_last = atomicAdd(p.tickets + tile, 1) == p.ksplit - 1;
    __syncthreads();
    if (*s_last) {
      __threadfence();
      // four consecutive rows per item, four items' loads in flight per thread (a loop that
      // waited on each load in turn took one L2 round trip per item)
      const int nq = p.NU / 4, items = NB * nq;
      for (int i0 = tid; i0 < items; i0 += 4 * TC_GATE_THREADS) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = i0 + j * TC_GATE_THREADS, b = i / nq, u = u0 + 4 * (i - b * nq);
          v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (i < items && b < p.B && u < p.H) v[j] = __ldcg(reinterpret_cast<const float4*>(p.tacc + (size_t)b * p.H + u));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = i0 + j * TC_GATE_THREADS, b = i / nq, u = u0 + 4 * (i - b * nq);
          if (i < items && u < p.H) {
            if (b < p.B) __stcg(reinterpret_cast<float4*>(p.tacc + (size_t)b * p.H + u), make_float4(0.f, 0.f, 0.f, 0.f));
            const float tv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            uint16_t hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __nv_bfloat16 h = __float2bfloat16_rn(tv[k]);
              hi[k] = __bfloat16_as_ushort(h);
              lo[k] = __bfloat16_as_ushort(__float2bfloat16_rn(tv[k] - __bfloat162float(h)));
            }
            *reinterpret_cast<uint2*>(p.tout + (size_t)b * p.H + u) =
                make_uint2(hi[0] | ((uint32_t)hi[1] << 16), hi[2] | ((uint32_t)hi[3] << 16));
            *reinterpret_cast<uint2*>(p.tout + (size_t)(NB + b) * p.H + u) =
                make_uint2(lo[0] | ((uint32_t)lo[1] << 16), lo[2] | ((uint32_t)lo[3] << 16));
          }
        }
      }
      if (tid == 0) p.tickets[tile] = 0;
    }
  } else if (__syncthreads_and(stage_ok) && warp < 8) {
    // item = (token b, units 4q..4q+3): one 16-byte load of each operand from the
    // transposed copy, one 8-byte store of h, the four mask bytes as one word where
    // aligned, one count update.  (A loop over single units, with a ballot and a
    // shared atomic per unit and token, was latency-bound: 16 rounds at 64 tokens.)
    const int NU = p.NU, B = p.B, H = p.H, Hs = p.Hs, D = p.D, act = p.act, flags = p.flags;
    const float thr = p.thr;
    uint8_t* const mask = p.mask;
    uint16_t* const hbuf = p.hbuf;
    const uint16_t* const xin = p.x;
    const int nq = NU / 4, items = B * nq;
    for (int i = tid; i < items; i += 256) {
      const int b = i / nq, r = 4 * (i - b * nq), u = u0 + r;
      const float4 z4 = *reinterpret_cast<const float4*>(s_acc + (size_t)b * TC_ACC_LD + r);
      const float4 p4 = *reinterpret_cast<const float4*>(
          fused ? s_acc + (size_t)b * TC_ACC_LD + NU + r : s_acc + (size_t)(NB + b) * TC_ACC_LD + r);
      const float zv[4] = {z4.x, z4.y, z4.z, z4.w}, pv[4] = {p4.x, p4.y, p4.z, p4.w};
      uint32_t hw[2] = {0u, 0u}, mw = 0u;
      int n = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool valid = u + j < H;
        float z = zv[j];
        if (LOPA && valid && (flags & FLAG_TILED_G))  // (G x)_u = x_{u mod D}
          z += __bfloat162float(__ushort_as_bfloat16(xin[(size_t)b * D + (u + j) % D]));
        const float az = activation(act, z);
        const bool lv = valid && is_live(az, thr);
        const float up = (flags & FLAG_DOUBLE_ACT) ? activation(act, pv[j]) : pv[j];
        const float hv = lv ? az * up : 0.f;
        hw[j >> 1] |= (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hv)) << (16 * (j & 1));
        mw |= (uint32_t)lv << (8 * j);
        n += lv;
      }
      if (n) atomicAdd(&s_cnt[b], n);
      uint16_t* hp = hbuf + (size_t)b * Hs + u;  // 8-byte aligned: Hs and u are multiples of 4
      uint8_t* mp = mask ? mask + (size_t)b * H + u : nullptr;
      if (u + 3 < H) {
        *reinterpret_cast<uint2*>(hp) = make_uint2(hw[0], hw[1]);
        if (mp && (reinterpret_cast<uintptr_t>(mp) & 3u) == 0) {
          *reinterpret_cast<uint32_t*>(mp) = mw;
        } else if (mp) {
#pragma unroll
          for (int j = 0; j < 4; ++j) mp[j] = (uint8_t)(mw >> (8 * j));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (u + j < H) {
            hp[j] = (uint16_t)(hw[j >> 1] >> (16 * (j & 1)));
            if (mp) mp[j] = (uint8_t)(mw >> (8 * j));
          }
      }
    }
    named_barrier(1, 256);
    if (tid < B && s_cnt[tid]) atomicAdd(p.ctrl + CTRL_COUNT + tid, s_cnt[tid]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == TC_GATE_MMA_WARP0) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// --------------------------------------------------------------------------- down kernel
// Stage layout, per unit chunk (64 units): W2^T rows for y values d0..d0+63
// and d0+64..d0+127 (two 8 KB MN-major atom columns), then h ([NB rows x 128 B]).
__global__ void __launch_bounds__(TC_THREADS, 1)
    ffn_tc_down_kernel(const __grid_constant__ CUtensorMap mW2, const __grid_constant__ CUtensorMap mH,
                       const TcDownArgs p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  const int NS = p.NS, NB = p.NB;
  const uint32_t half = TC_UCH * 128u, chb = down_chunk_bytes(NB);
  const uint32_t st_bytes = TC_DC * chb;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)NS * st_bytes);
  uint64_t* empty = full + NS;
  uint64_t* done = empty + NS;
  uint64_t* mdone = done + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool clus = p.cluster != 0;
  const int dt = clus ? blockIdx.x / p.nsplit : blockIdx.x % p.ndt;
  const int sp = clus ? blockIdx.x % p.nsplit : blockIdx.x / p.ndt, d0 = dt * TC_DTILE;  // sp = rank in the cluster
  const int c0 = (int)((long long)sp * p.nch / p.nsplit), c1 = (int)((long long)(sp + 1) * p.nch / p.nsplit);
  const int nst = (c1 - c0 + TC_DC - 1) / TC_DC;
  int* err = p.ctrl + CTRL_ERR;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    mbar_init(mdone, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == TC_MMA_WARP) tmem_alloc(tslot, p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) pdl_launch_dependents();  // after the TMEM allocation (see the gate-up kernel)

  if (warp == TC_PRODUCER_WARP) {
    // copies of a stage spread over the lanes (see the gate-up kernel)
    if (lane == 0) {
      tma_prefetch_map(&mW2);
      tma_prefetch_map(&mH);
    }
    auto nchunks = [&](int q) { return min(TC_DC, c1 - c0 - q * TC_DC); };
    const int npre = min(NS, nst);
    for (int q = 0; q < npre; ++q) {  // W2^T is constant: request it before the dependency wait
      uint8_t* st = sm + (size_t)q * st_bytes;
      const int nc = nchunks(q);
      if (lane == 0) mbar_arrive_expect_tx(&full[q], (uint32_t)nc * chb);
      __syncwarp();
      if (lane < 2 * nc) {
        const int c = lane >> 1, mh = lane & 1;
        tma_tile_2d(st + c * chb + mh * half, &mW2, d0 + 64 * mh, (c0 + q * TC_DC + c) * TC_UCH, &full[q]);
      }
    }
    pdl_wait();  // h comes from the gate-up kernel
    for (int q = 0; q < npre; ++q)
      if (lane < nchunks(q))
        tma_tile_2d(sm + (size_t)q * st_bytes + lane * chb + 2 * half, &mH, (c0 + q * TC_DC + lane) * TC_UCH, 0,
                    &full[q]);
    int issued = npre;
    for (int q = npre; q < nst; ++q) {
      const int s = q % NS;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&empty[s], ((q / NS) - 1) & 1, abort_flag, err, p.timeout_ns);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const int nc = nchunks(q);
      if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)nc * chb);
      __syncwarp();
      if (lane < 3 * nc) {
        const int c = lane / 3, k = lane - 3 * c;  // k: 0, 1 the two y halves of W2^T, 2 the h rows
        uint8_t* cb = sm + (size_t)s * st_bytes + c * chb;
        const int u = (c0 + q * TC_DC + c) * TC_UCH;
        if (k < 2)
          tma_tile_2d(cb + k * half, &mW2, d0 + 64 * k, u, &full[s]);
        else
          tma_tile_2d(cb + 2 * half, &mH, u, 0, &full[s]);
      }
      issued = q + 1;
    }
    if (lane == 0)
      for (int q = max(0, issued - NS); q < issued; ++q) mbar_wait_drain(&full[q % NS], (q / NS) & 1, p.timeout_ns);
    __syncwarp();
  } else if (warp == TC_MMA_WARP) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(TC_DTILE, NB, true, false);  // N = the tokens of h
      int gk = 0;  // K step over the block's units
      for (int q = 0; q < nst; ++q) {
        const int s = q % NS;
        if (!mbar_wait(&full[s], (q / NS) & 1, abort_flag, err, p.timeout_ns)) break;
        tc_fence_after();
        const int nc = min(TC_DC, c1 - c0 - q * TC_DC);
        for (int c = 0; c < nc; ++c) {
          const uint32_t cb = smem_u32(sm + (size_t)s * st_bytes + c * chb);
          // 16 units per K step: two 8-unit K groups of 1 KB; the y halves are `half` bytes apart
          const uint64_t ad0 = smem_desc(cb, half, 1024, SMEM_LAYOUT_SW128);
          const uint64_t bd0 = smem_desc(cb + 2 * half, 16, 1024, SMEM_LAYOUT_SW128);
#pragma unroll
          for (int k = 0; k < TC_UCH / 16; ++k, ++gk)
            tc_mma(tmem + (uint32_t)(gk & (p.nacc - 1)) * (uint32_t)NB, ad0 + (k * 2048 >> 4), bd0 + 2 * k, idesc,
                   gk >= p.nacc);
        }
        tc_commit(&empty[s]);
      }
      tc_commit(done);
      tc_commit(mdone);
      mbar_wait_drain(mdone, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ---- epilogue warps 0..3: lane = one y value of the slice
    pdl_wait();
    int* s_last = reinterpret_cast<int*>(tslot + 2);
    if (blockIdx.x == 0 && tid < p.B) {  // the gate-up kernel is complete: publish the live counts
      p.counts[tid] = __ldcg(p.ctrl + CTRL_COUNT + tid);
      __stcg(p.ctrl + CTRL_COUNT + tid, 0);
    }
    const int used = min(p.nacc, (c1 - c0) * (TC_UCH / 16));  // accumulators that received a K step
    const bool mma_ok = nst > 0 && __all_sync(0xffffffffu, mbar_wait(done, 0, abort_flag, err, p.timeout_ns));
    // the slice's sums, transposed through the (drained) stages: s_y[token][TC_ACC_LD], then one
    // 16-byte atomic per (token, four y values) instead of one 4-byte atomic per value
    float* s_y = reinterpret_cast<float*>(sm);
    if (mma_ok) {
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
      for (int cc = 0; cc < NB; cc += 16) {
        float v[16];
        tmem_ld_sum(tl + cc, NB, used, v);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) s_y[(size_t)(cc + jj) * TC_ACC_LD + 32 * warp + lane] = v[jj];
      }
    }
    if (named_barrier_and(1, 128, mma_ok) && !clus) {  // all four warps copied their rows
      const int B = p.B, D = p.D;
      for (int i = tid; i < B * (TC_DTILE / 4); i += 128) {
        const int b = i / (TC_DTILE / 4), j = 4 * (i - b * (TC_DTILE / 4));
        if (d0 + j < D)  // D is a multiple of 8: the whole quad is in range
          atomicAdd(reinterpret_cast<float4*>(p.yacc + (size_t)b * YACC_COPIES * D + d0 + j),
                    *reinterpret_cast<const float4*>(s_y + (size_t)b * TC_ACC_LD + j));
      }
    }
    // the last block of this y slice rounds the sum into y and clears the accumulator
    if (!clus) {
      __threadfence();
      named_barrier(1, 128);
      if (tid == 0) *s_last = atomicAdd(p.tickets + dt, 1) == p.nsplit - 1;
      named_barrier(1, 128);
      if (*s_last) {
        // 16-byte items (token b, four y values), sixteen loads in flight per thread before any
        // store: the whole slice of up to 64 tokens in one round trip.  This pass ends the
        // kernel, and the next kernel's dependency wait, for the slowest slice.
        __threadfence();
        const int B = p.B, D = p.D, items = B * (TC_DTILE / 4);
        uint16_t* const y = static_cast<uint16_t*>(p.y);
        for (int i0 = 0; i0 < items; i0 += 16 * 128) {
          float4 v[16];
  #pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = i0 + e * 128 + tid, b = i / (TC_DTILE / 4), j = 4 * (i % (TC_DTILE / 4));
            v[e] = i < items && d0 + j < D
                       ? __ldcg(reinterpret_cast<const float4*>(p.yacc + (size_t)b * YACC_COPIES * D + d0 + j))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
          }
  #pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = i0 + e * 128 + tid, b = i / (TC_DTILE / 4), j = 4 * (i % (TC_DTILE / 4));
            if (i < items && d0 + j < D) {
              __stcg(reinterpret_cast<float4*>(p.yacc + (size_t)b * YACC_COPIES * D + d0 + j),
                     make_float4(0.f, 0.f, 0.f, 0.f));
              const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[e].x)) |
                                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[e].y)) << 16);
              const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[e].z)) |
                                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[e].w)) << 16);
              *reinterpret_cast<uint2*>(y + (size_t)b * D + d0 + j) = make_uint2(lo, hi);
            }
          }
        }
        if (tid == 0) p.tickets[dt] = 0;
      }
    }
  }
  if (clus) {
    // every block's partial tile s_y[token][TC_ACC_LD] is complete once the cluster barrier
    // passes; block sp then sums the nsplit tiles for its share of the tokens, 16-byte items
    // (token b, four y values) read from each block's shared memory, and rounds them into y.
    // The second barrier keeps every tile in place until all blocks have read it.
    __syncwarp();
    cluster_sync_all();
    const int B = p.B, D = p.D, ns = p.nsplit;
    const int b0 = (int)((long long)sp * B / ns), b1 = (int)((long long)(sp + 1) * B / ns);
    const int items = (b1 - b0) * (TC_DTILE / 4);
    const uint32_t s_y = smem_u32(sm);
    uint16_t* const y = static_cast<uint16_t*>(p.y);
    for (int i = tid; i < items; i += TC_THREADS) {
      const int b = b0 + i / (TC_DTILE / 4), j = 4 * (i % (TC_DTILE / 4));
      const uint32_t off = s_y + (uint32_t)((b * TC_ACC_LD + j) * 4);
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
        *reinterpret_cast<uint2*>(y + (size_t)b * D + d0 + j) = make_uint2(lo, hi);
      }
    }
    cluster_sync_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == TC_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// --------------------------------------------------------------------------- host side
}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// bf16 matrix [rows, cols] (row stride in bytes), boxes of 64 columns x box_rows, 128-byte swizzle
int encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t stride_bytes, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return -1;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {stride_bytes};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)r;
}

TcPlan plan_ffn_tc(int D, int H, int r, int num_sms) {
  TcPlan p;
  if (D % 8 != 0 || r % 8 != 0 || num_sms < 1) return p;
  const int per = (H + num_sms - 1) / num_sms;
  // one slice per SM; an MMA covers at most 128 units, so past 128 units per
  // SM the slices fill more than one wave
  p.NU = std::min(128, std::max(8, (per + 7) / 8 * 8));
  // An M = 64 MMA does not map accumulator rows to TMEM lanes one to one (16
  // rows per 32-lane quarter), so every product that the epilogue reads by
  // lane runs with M = 128; the rows past NU are never read.  Only the
  // standard gate's stacked form (2 NU <= 128) has NU <= 64, and it issues M = 128.
  p.MT = 128;
  p.ntiles = (H + p.NU - 1) / p.NU;
  p.KC = (D + 63) / 64;
  p.r = r;
  p.KCZ = (r + 63) / 64;
  p.num_sms = num_sms;
  if (r > 0) {  // the t kernel: slices of up to 128 rows of V, each over ksplit_t ranges of D
    p.NUt = std::min(128, (r + 7) / 8 * 8);
    p.ntiles_t = (r + p.NUt - 1) / p.NUt;
    p.ksplit_t = std::max(1, std::min(p.KC, num_sms / p.ntiles_t));
    if (p.ntiles_t > TC_TICKETS) return p;
  }
  p.ndt = (D + TC_DTILE - 1) / TC_DTILE;
  p.nch = (H + TC_UCH - 1) / TC_UCH;
  p.nsplit = std::max(1, std::min(p.nch, num_sms / p.ndt));
  p.Hs = (H + 7) / 8 * 8;
  // the low-rank gate's stages are large (its t-pair groups and x regions): 220 KB keeps a third stage
  // at 64 tokens (measured: 41.2 -> 39.0 us per call; the standard gate is the same at 200 or 220)
  p.gate_smem_budget = r > 0 ? 220 * 1024 : TC_SMEM_BUDGET;
  p.gate_chunks = 0;
  p.down_smem_budget = TC_SMEM_BUDGET;
  p.ok = true;
  return p;
}

size_t ffn_tc_hbuf_elems(const TcPlan& p) { return (size_t)2 * 128 * p.Hs; }

int encode_tc_maps(TcMaps* m, const TcPlan& p, const void* W1, const void* V, const void* W3, const void* W2t,
                   uint16_t* hbuf, int D, int H) {
  const int gk = p.r > 0 ? p.r : D;  // W1 [H, D] or U [H, r]
  int rc = encode_2d(&m->w1, W1, (uint64_t)H, (uint64_t)gk, (uint64_t)gk * 2, (uint32_t)p.NU);
  if (!rc && p.r > 0) rc = encode_2d(&m->v, V, (uint64_t)p.r, (uint64_t)D, (uint64_t)D * 2, (uint32_t)p.NUt);
  if (!rc) rc = encode_2d(&m->w3, W3, (uint64_t)H, (uint64_t)D, (uint64_t)D * 2, (uint32_t)p.NU);
  if (!rc) rc = encode_2d(&m->w2, W2t, (uint64_t)H, (uint64_t)D, (uint64_t)D * 2, TC_UCH);
  for (int i = 0; i < 8 && !rc; ++i)  // h boxes of 2 NB rows, NB = 16 (i + 1)
    rc = encode_2d(&m->h[i], hbuf, 256, (uint64_t)H, (uint64_t)p.Hs * 2, (uint32_t)(16 * (i + 1)));
  return rc;
}

cudaError_t ffn_tc_prepare(size_t max_smem) {
  void (*ks[2])(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const TcGateArgs) = {
      ffn_tc_gateup_kernel<128, false>, ffn_tc_gateup_kernel<128, true>};
  cudaError_t e = cudaSuccess;
  for (auto k : ks)
    if (!e) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
  if (!e) e = cudaFuncSetAttribute(ffn_tc_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
  return e;
}

namespace {
// pipeline stages of the down kernel for NB padded tokens
int down_stages(const TcPlan& plan, int NB, size_t max_smem) {
  int ns = (int)std::max<size_t>(2, std::min<size_t>(TC_NS_MAX, plan.down_smem_budget / (TC_DC * down_chunk_bytes(NB))));
  while (ns > 2 && down_smem_bytes(NB, ns) > max_smem) --ns;
  return ns;
}
}  // namespace

cudaError_t ffn_tc_plan_cluster(TcPlan& plan, size_t max_smem) {
  plan.down_cluster = 0;
  if (!plan.ok || plan.ndt < 1) return cudaSuccess;
  size_t smem = 0;  // the largest down-kernel footprint of any batch size
  for (int NB = 16; NB <= 128; NB += 16) smem = std::max(smem, down_smem_bytes(NB, down_stages(plan, NB, max_smem)));
  for (int cs = std::min(std::min(8, plan.nch), plan.num_sms / plan.ndt); cs >= 2; --cs) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.ndt * cs);
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = (unsigned)cs;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, ffn_tc_down_kernel, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();  // this size is not possible here: try a smaller one
      continue;
    }
    if (n >= plan.ndt) {  // every slice's cluster resident at once: one wave
      plan.down_cluster = cs;
      break;
    }
  }
  plan.t_cluster = 0;
  for (int cs = std::min(8, plan.KC); plan.r > 0 && cs >= 2; --cs) {  // the low-rank t kernel's K splits
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.ntiles_t * cs);
    cfg.blockDim = dim3(TC_GATE_THREADS);
    cfg.dynamicSmemBytes = max_smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = (unsigned)cs;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, ffn_tc_gateup_kernel<128, true>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      continue;
    }
    if (n >= plan.ntiles_t) {
      plan.t_cluster = cs;
      break;
    }
  }
  return cudaSuccess;
}

int launch_ffn_tc(const TcPlan& plan, const TcMaps& maps, const TcBuffers& buf, const void* x, void* y, int D, int H,
                  int B, int act, int flags, float thr, unsigned long long timeout_ns, size_t max_smem, cudaStream_t s,
                  cudaError_t* cuda_err, bool tpair_ready, bool t_only) {
  *cuda_err = cudaSuccess;
  const bool lopa = plan.r > 0;
  if (!plan.ok || B < 1 || B > 128 || (lopa && !buf.tpair)) return -1;
  const int NB = (B + 15) / 16 * 16;
  CUtensorMap mx, mt;
  if (int rc = encode_2d(&mx, x, (uint64_t)B, (uint64_t)D, (uint64_t)D * 2, (uint32_t)NB)) return rc;
  if (lopa) {  // the t pair of every token: rows [0, NB) t_hi, [NB, 2 NB) t_lo
    if (int rc = encode_2d(&mt, buf.tpair, (uint64_t)(2 * NB), (uint64_t)plan.r, (uint64_t)plan.r * 2,
                           (uint32_t)(2 * NB)))
      return rc;
  } else {
    mt = mx;  // not read
  }
  // gate-up arguments for slices of NU rows of a [Hg, .] matrix (the t kernel: V's r rows, no U chunks).
  // More slices than SMs: two blocks per SM (half the shared memory and TMEM each), so that the
  // slices run in one wave; not with NB = 128, whose accumulator copy needs 132 KB.
  auto gate_args = [&](int NU, int Hg, bool with_u, uint16_t* tout, int ksplit, TcGateArgs& g, size_t& smem) {
    const bool two = (Hg + NU - 1) / NU > plan.num_sms && NB <= 64;
    const size_t cap = two ? std::min(max_smem, (size_t)110 * 1024) : max_smem;
    const size_t budget = two ? std::min(plan.gate_smem_budget, (size_t)100 * 1024) : plan.gate_smem_budget;
    auto stage_bytes = [&](int C) { return lopa ? lopa_stage_bytes(C, NU, NB) : gate_stage_bytes(C, NU, NB); };
    auto smem_bytes = [&](int C, int NS) {
      return lopa ? lopa_smem_bytes(C, plan.MT, NU, NB, NS) : gate_smem_bytes(C, plan.MT, NU, NB, NS);
    };
    g.D = D;
    g.H = Hg;
    g.B = B;
    g.NB = NB;
    g.NU = NU;
    g.KC = plan.KC;
    // four K chunks per stage; for the standard gate two once x makes up a large part of a
    // stage (measured: at 64 tokens 32.0 us per call with two, the low-rank gate 43.3 with four
    // against 49.6 with two)
    g.C = plan.gate_chunks > 0 ? plan.gate_chunks : (!lopa && NB >= 48 ? 2 : 4);
    while (g.C > 1 && smem_bytes(g.C, 2) > std::min(cap, (size_t)TC_SMEM_BUDGET)) g.C >>= 1;
    g.KCZ = with_u ? plan.KCZ : 0;
    g.NCZ = (g.KCZ + lopa_zchunks(g.C) - 1) / lopa_zchunks(g.C);  // KCZ = 0 for the standard gate
    g.NCG = g.NCZ + (plan.KC + g.C - 1) / g.C;
    g.NS = (int)std::max<size_t>(2, std::min<size_t>(TC_NS_MAX, budget / stage_bytes(g.C)));
    {  // a K-split block has few chunk groups: no more stages than it fills or the epilogue's copy needs
      const int kc_blk = (plan.KC + ksplit - 1) / ksplit;
      const int groups = g.NCZ + (kc_blk + g.C - 1) / g.C;
      const size_t acc_copy = tc_acc_copy_bytes(NB);
      const int need = (int)((acc_copy + stage_bytes(g.C) - 1) / stage_bytes(g.C));
      g.NS = std::max(std::min(g.NS, std::max(2, groups)), need);
    }
    while (g.NS > 2 && smem_bytes(g.C, g.NS) > cap) --g.NS;
    g.act = act;
    g.flags = flags;
    g.thr = thr;
    g.Hs = plan.Hs;
    g.x = static_cast<const uint16_t*>(x);
    g.tout = tout;
    g.ksplit = ksplit;
    g.tcluster = 0;
    g.tacc = buf.tacc;
    g.tickets = buf.tickets_t;
    const int cols = !lopa && 2 * NU <= 128 ? NB : 2 * NB;  // one accumulator
    g.nacc = cols <= 128 ? 4 : 2;  // MMA warps = accumulators, nacc * cols <= 512
    if (two) g.nacc = std::min(g.nacc, 256 / cols);  // <= 256 columns per block
    g.tmem_cols = tmem_cols_for(g.nacc * cols);
    g.ctrl = buf.ctrl;
    g.mask = buf.mask;
    g.hbuf = buf.hbuf;
    g.timeout_ns = timeout_ns;
    smem = smem_bytes(g.C, g.NS);
    // the epilogue stages the transposed accumulator (tc_acc_copy_bytes) over the pipeline stages
    return (size_t)g.NS * stage_bytes(g.C) >= tc_acc_copy_bytes(NB) && smem <= cap;
  };
  const dim3 gb(TC_GATE_THREADS);
  cudaError_t e = cudaSuccess;
  if (lopa && !tpair_ready) {
    TcGateArgs gt;
    size_t smt = 0;
    const bool tclus = plan.t_cluster > 0;
    const int ksplit = tclus ? plan.t_cluster : std::max(1, std::min(plan.ksplit_t, plan.t_split_tokens / NB));
    if (!gate_args(plan.NUt, plan.r, false, buf.tpair, ksplit, gt, smt)) {
      *cuda_err = cudaErrorInvalidConfiguration;
      return 0;
    }
    gt.tcluster = tclus ? 1 : 0;
    if (tclus)
      e = launch_pdl_cluster(ffn_tc_gateup_kernel<128, true>, dim3(plan.ntiles_t * gt.ksplit), gb, smt, s,
                             (unsigned)gt.ksplit, maps.v, maps.v, mx, mx, gt);
    else
      e = launch_pdl(ffn_tc_gateup_kernel<128, true>, dim3(plan.ntiles_t * gt.ksplit), gb, smt, s, maps.v, maps.v,
                     mx, mx, gt);
    if (e || t_only) {
      *cuda_err = e;
      return 0;
    }
  }
  TcGateArgs g;
  size_t smem1 = 0;
  if (!gate_args(plan.NU, H, lopa, nullptr, 1, g, smem1)) {
    *cuda_err = cudaErrorInvalidConfiguration;
    return 0;
  }
  const dim3 gg(plan.ntiles);
  e = lopa ? launch_pdl(ffn_tc_gateup_kernel<128, true>, gg, gb, smem1, s, maps.w1, maps.w3, mx, mt, g)
           : launch_pdl(ffn_tc_gateup_kernel<128, false>, gg, gb, smem1, s, maps.w1, maps.w3, mx, mt, g);
  if (e) {
    *cuda_err = e;
    return 0;
  }

  TcDownArgs d;
  d.D = D;
  d.B = B;
  d.NB = NB;
  d.nch = plan.nch;
  d.ndt = plan.ndt;
  d.cluster = plan.down_cluster > 0 ? 1 : 0;
  d.nsplit = d.cluster ? plan.down_cluster : plan.nsplit;
  d.NS = down_stages(plan, NB, max_smem);
  d.nacc = NB <= 64 ? 4 : 2;  // a power of two, nacc * NB <= 256
  d.tmem_cols = tmem_cols_for(d.nacc * NB);
  d.y = y;
  d.counts = buf.counts;
  d.tickets = buf.tickets;
  d.yacc = buf.yacc;
  d.ctrl = buf.ctrl;
  d.timeout_ns = timeout_ns;
  const size_t smem2 = down_smem_bytes(NB, d.NS);
  if (smem2 > max_smem) {
    *cuda_err = cudaErrorInvalidConfiguration;
    return 0;
  }
  if (d.cluster)
    *cuda_err = launch_pdl_cluster(ffn_tc_down_kernel, dim3(plan.ndt * d.nsplit), dim3(TC_THREADS), smem2, s,
                                   (unsigned)d.nsplit, maps.w2, maps.h[NB / 16 - 1], d);
  else
    *cuda_err = launch_pdl(ffn_tc_down_kernel, dim3(plan.ndt * d.nsplit), dim3(TC_THREADS), smem2, s, maps.w2,
                           maps.h[NB / 16 - 1], d);
  return 0;
}

}  // namespace sffn
