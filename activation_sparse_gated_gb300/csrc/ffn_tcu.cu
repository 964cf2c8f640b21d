// ffn_tcu.cu -- gate-first FFN for a small batch of tokens (2..8, bf16
// weights and tokens, standard gate): the gate on the tensor cores, the union
// of the tokens' live sets gathered on the CUDA cores.
//
// "Model casting: compute the gate, then skip most of the FFN" (sections "What
// an FFN actually computes" and on batching): per token b
//     y_b = sum_{i : z_bi live} W2[:, i] A(z_bi) (W3[i, :] . x_b),  z_b = W1 x_b,
// and a batch needs the W3 row and W2 column of every unit that ANY of its
// tokens keeps -- the union of the live sets, 1 - s^B of the units (34 % at
// B = 4, 57 % at B = 8 for s = 0.9).  For small batches this kernel reads
// exactly that, one block per slice of NU units:
//   * gate: Z[slice, tokens] = W1[slice, :] X^T with tcgen05 -- TMA-fed stages
//     of the slice's W1 rows and of x (128-byte swizzle), the weights of the
//     first stages requested before the dependency wait, K steps round-robin
//     over `nacc` TMEM accumulators issued by as many warps; the MMA is
//     M = 128, of which the first NU rows are the slice (the others read
//     neighbouring shared memory and land in TMEM lanes nobody reads);
//   * decisions: live_bi = |A(z_bi)| > thr, per-token flags and counts; the
//     block's union (units live for some token) is compacted in ascending
//     order with warp ballots and its W3 and W2^T rows are prefetched into L2;
//   * gathers, a batch of union units at a time in the (then idle) stage
//     buffers: their W3 rows are copied into shared memory in one go (one
//     round trip), h_bk = A(z_bk) (W3[unit_k, :] . x_b) -- exactly 0 for a
//     token whose gate is dead -- with one warp per unit against x of every
//     token (staged once as fp32); then their W2^T rows replace them and
//     thread t folds y_b[8t, 8t + 8) += h_bk W2^T[unit_k, 8t..] for every
//     token; fp32 atomics into one of the accumulator copies; the finalize
//     kernel chained behind sums the copies, rounds y and publishes the
//     counts.  h stays fp32.
// Every wait is bounded (error word + early exit); a block drains its copies
// and MMAs before it releases TMEM.
#include <algorithm>

#include "internal.h"
#include "tc.cuh"

namespace sffn {

namespace {

constexpr int TU_THREADS = 320;       // warps 0-3 TMEM copy, 4 TMA producer, 5-8 MMA issuers; all 10 gather
constexpr int TU_WARPS = TU_THREADS / 32;
constexpr int TU_PRODUCER_WARP = 4;
constexpr int TU_MMA_WARP0 = 5;
constexpr int TU_BMAX = 8;            // tokens per launch
constexpr int TU_ROWS = 128;          // MMA M: the slice's NU <= 128 rows
constexpr size_t TU_SMEM_BUDGET = 200 * 1024;
constexpr int TU_NS_MAX = 8;

struct TcuArgs {
  int D, H, B, NB, NU, KC, C, NCG, NS, act, nacc, flags;
  float thr;
  uint32_t tmem_cols;
  const uint4* W3;   // [H, D] bf16
  const uint4* W2t;  // [H, D] bf16 (W2 transposed)
  const uint4* x;    // [B, D] bf16
  float* yacc;       // [B_max * YACC_COPIES, D], zero between calls
  int* ctrl;
  uint8_t* mask;     // [B_max, H]
  unsigned long long timeout_ns;
};

__host__ __device__ constexpr uint32_t tcu_stage_bytes(int C, int NU, int NB) {
  return (uint32_t)C * 128u * (uint32_t)(NU + NB);
}
// An M = 128 MMA reads 128 rows from the start of the last W1 region of the
// last stage: 128 - NU rows past it, of which the stage's x regions cover C NB.
__host__ __device__ inline uint32_t tcu_slack_bytes(int C, int NU, int NB) {
  const int over = (TU_ROWS - NU) * 128 - C * NB * 128;
  return over > 0 ? (uint32_t)(over + 1023) / 1024 * 1024 : 0u;
}
__host__ __device__ constexpr size_t tcu_a16(size_t v) { return (v + 15) & ~size_t(15); }
// barriers, TMEM slot, abort flag, counts, union list and decisions after the stages
__host__ __device__ constexpr size_t tcu_tail_bytes(int NS) {
  return (size_t)8 * (2 * NS + 1) + 8 + 4 * TU_BMAX + 16 + 4 * TU_ROWS + 2 * 4 * TU_ROWS * TU_BMAX +
         TU_BMAX * TU_ROWS + 64;
}
size_t tcu_smem_bytes(int C, int NU, int NB, int NS) {
  return 1024 + (size_t)NS * tcu_stage_bytes(C, NU, NB) + tcu_slack_bytes(C, NU, NB) + tcu_tail_bytes(NS);
}
// the epilogue reuses the stages: z copy [128][NB + 1] fp32, x [B][D] fp32, then
// the gather area (at least one D-row)
size_t tcu_epilogue_bytes(int NB, int B, int D) {
  return tcu_a16((size_t)TU_ROWS * (NB + 1) * 4) + (size_t)B * D * 4 + (size_t)D * 2;
}

__device__ __forceinline__ void pf_row(const void* row, uint32_t bytes, int lane) {
  const char* b = static_cast<const char*>(row);
  for (uint32_t off = (uint32_t)lane * 128u; off < bytes; off += 32u * 128u)
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(b + off));
}

__device__ __forceinline__ void cpa16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cpa_commit_wait() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__global__ void __launch_bounds__(TU_THREADS, 1)
    ffn_tcu_kernel(const __grid_constant__ CUtensorMap mW1, const __grid_constant__ CUtensorMap mX, const TcuArgs p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
  const int NS = p.NS, NB = p.NB, C = p.C, NU = p.NU, B = p.B, D = p.D;
  const int nch = D / 8;  // 16-byte chunks of a D-row
  const uint32_t wreg = (uint32_t)NU * 128u, xreg = (uint32_t)NB * 128u;
  const uint32_t st_bytes = tcu_stage_bytes(C, NU, NB);
  uint8_t* tail = sm + (size_t)NS * st_bytes + tcu_slack_bytes(C, NU, NB);
  uint64_t* full = reinterpret_cast<uint64_t*>(tail);
  uint64_t* empty = full + NS;
  uint64_t* done = empty + NS;  // every MMA complete (one commit per MMA warp)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  int* s_cnt = reinterpret_cast<int*>(tslot + 2);  // [TU_BMAX] live counts of the slice per token
  int* s_wc = s_cnt + TU_BMAX;                     // [4] union units per 32 rows
  int* l_row = s_wc + 4;                           // [128] union list: rows of the slice, ascending
  float* l_a = reinterpret_cast<float*>(l_row + TU_ROWS);  // [128 rows][TU_BMAX] A(z), 0 where dead
  float* l_h = l_a + TU_ROWS * TU_BMAX;                    // [128 list][TU_BMAX] h
  uint8_t* s_live = reinterpret_cast<uint8_t*>(l_h + TU_ROWS * TU_BMAX);  // [TU_BMAX][128] flags
  const int ldz = NB + 1;
  // over the stages, once every MMA is done: z copy [128][ldz]; x of every token
  // as fp32 in the interleaved layout xq[(b * 2 + k) * nch + c] = x_b[8c + 4k .. + 4)
  // (lanes reading consecutive chunks read consecutive 16-byte words); the gather area
  float* s_z = reinterpret_cast<float*>(sm);
  float4* xq = reinterpret_cast<float4*>(sm + tcu_a16((size_t)TU_ROWS * ldz * 4));
  uint4* area = reinterpret_cast<uint4*>(xq + (size_t)B * 2 * nch);
  const int RB = max(1, (int)(((size_t)NS * st_bytes - (reinterpret_cast<uint8_t*>(area) - sm)) / ((size_t)nch * 16)));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u0 = blockIdx.x * NU;
  const int nrows = min(NU, p.H - u0);
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
  if (tid < TU_BMAX) s_cnt[tid] = 0;
  if (warp == TU_MMA_WARP0) tmem_alloc(tslot, p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // the next kernel launches only once this block holds its TMEM
  if (tid == 0) pdl_launch_dependents();
  int stage_ok = 1;

  if (warp == TU_PRODUCER_WARP) {
    if (lane == 0) {
      tma_prefetch_map(&mW1);
      tma_prefetch_map(&mX);
    }
    auto nchunks = [&](int q) { return min(C, p.KC - q * C); };
    const int npre = min(NS, p.NCG);
    for (int q = 0; q < npre; ++q) {  // W1 does not depend on the previous kernel
      uint8_t* st = sm + (size_t)q * st_bytes;
      const int nc = nchunks(q);
      if (lane == 0) mbar_arrive_expect_tx(&full[q], (uint32_t)nc * (wreg + xreg));
      __syncwarp();
      if (lane < nc) tma_tile_2d(st + lane * wreg, &mW1, (q * C + lane) * 64, u0, &full[q]);
    }
    pdl_wait();
    for (int q = 0; q < npre; ++q)
      if (lane < nchunks(q))
        tma_tile_2d(sm + (size_t)q * st_bytes + C * wreg + lane * xreg, &mX, (q * C + lane) * 64, 0, &full[q]);
    int issued = npre;
    for (int q = npre; q < p.NCG; ++q) {
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
  } else if (warp >= TU_MMA_WARP0 && warp < TU_MMA_WARP0 + 4) {
    const int mw = warp - TU_MMA_WARP0;  // K steps kk = mw (mod nacc) into accumulator mw
    if (mw < p.nacc && lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(TU_ROWS, NB, false, false);
      const uint32_t da = tmem + (uint32_t)mw * NB;
      bool started = false;
      for (int q = 0; q < p.NCG; ++q) {
        const int s = q % NS;
        if (!mbar_wait(&full[s], (q / NS) & 1, abort_flag, err, p.timeout_ns)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(sm + (size_t)s * st_bytes);
        const uint64_t a0 = smem_desc(sa, 16, 1024, SMEM_LAYOUT_SW128);
        const uint64_t b0 = smem_desc(sa + C * wreg, 16, 1024, SMEM_LAYOUT_SW128);
        const int nc = min(C, p.KC - q * C);
        for (int c = 0; c < nc; ++c) {
          const uint64_t ac = a0 + ((c * wreg) >> 4), bc = b0 + ((c * xreg) >> 4);
          for (int kk = mw; kk < 4; kk += p.nacc) {
            tc_mma(da, ac + 2 * kk, bc + 2 * kk, idesc, started);
            started = true;
          }
        }
        tc_commit(&empty[s]);
      }
      tc_commit(done);
      mbar_wait_drain(done, 0, p.timeout_ns);  // every MMA warp's work complete before TMEM is released
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---- warps 0..3: TMEM lanes 32q..32q+31 (summing the accumulators) into s_z
    pdl_wait();  // x, the accumulators, the flags and the counts follow stream order
    stage_ok = __all_sync(0xffffffffu, mbar_wait(done, 0, abort_flag, err, p.timeout_ns));
    if (stage_ok) {
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
      float* row = s_z + (size_t)(32 * warp + lane) * ldz;
      for (int c0 = 0; c0 < NB; c0 += 16) {
        float v[16];
        tmem_ld_sum(tl + c0, NB, p.nacc, v);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) row[c0 + jj] = v[jj];
      }
    }
  }
  if (__syncthreads_and(stage_ok)) {
    // ---- decisions per (row, token); the row's A(z) where live, else 0
    for (int i = tid; i < TU_ROWS * TU_BMAX; i += TU_THREADS) {
      const int r = i / TU_BMAX, b = i - r * TU_BMAX;
      const bool valid = r < nrows && b < B;
      const float z = valid ? s_z[(size_t)r * ldz + b] : 0.f;
      const float a = activation(p.act, z);
      const bool lv = valid && is_live(a, p.thr);
      s_live[b * TU_ROWS + r] = lv ? 1 : 0;
      l_a[r * TU_BMAX + b] = lv ? a : 0.f;
      if (lv) atomicAdd(&s_cnt[b], 1);
    }
    __syncthreads();
    // ---- the union, ascending: a ballot per 32 rows, then an exclusive prefix
    const int r = 32 * warp + lane;
    bool any = false;
    if (warp < 4) {
#pragma unroll
      for (int b = 0; b < TU_BMAX; ++b) any |= s_live[b * TU_ROWS + r] != 0;
      const unsigned m = __ballot_sync(0xffffffffu, any);
      if (lane == 0) s_wc[warp] = __popc(m);
    }
    __syncthreads();
    const int n_u = s_wc[0] + s_wc[1] + s_wc[2] + s_wc[3];
    if (warp < 4) {
      int base = 0;
      for (int k = 0; k < warp; ++k) base += s_wc[k];
      const unsigned m = __ballot_sync(0xffffffffu, any);
      if (any) l_row[base + __popc(m & ((1u << lane) - 1u))] = r;
    }
    __syncthreads();
    // both gathered rows of every union unit start moving into L2 now
    for (int k = warp; k < n_u; k += TU_WARPS) {
      const size_t unit = (size_t)(u0 + l_row[k]);
      pf_row(p.W3 + unit * nch, (uint32_t)nch * 16u, lane);
      pf_row(p.W2t + unit * nch, (uint32_t)nch * 16u, lane);
    }
    // flags and counts of the slice; x of every token into shared memory
    for (int i = tid; i < B * nrows; i += TU_THREADS) {
      const int b = i / nrows, rr = i - b * nrows;
      p.mask[(size_t)b * p.H + u0 + rr] = s_live[b * TU_ROWS + rr];
    }
    if (tid < B && s_cnt[tid] > 0) atomicAdd(p.ctrl + CTRL_COUNT + tid, s_cnt[tid]);
    for (int i = tid; i < B * nch; i += TU_THREADS) {  // token b = i / nch, chunk c
      const int b = i / nch, c = i - b * nch;
      float v[8];
      Elt<bf16_tag>::unpack(__ldcg(p.x + i), v);
      xq[(size_t)(2 * b) * nch + c] = make_float4(v[0], v[1], v[2], v[3]);
      xq[(size_t)(2 * b + 1) * nch + c] = make_float4(v[4], v[5], v[6], v[7]);
    }
    __syncthreads();

    const bool dbl = (p.flags & FLAG_DOUBLE_ACT) != 0;
    const int cp = blockIdx.x % YACC_COPIES;
    for (int k0 = 0; k0 < n_u; k0 += RB) {
      const int nb = min(RB, n_u - k0);
      // W3 rows of the batch, all in flight at once
      for (int i = tid; i < nb * nch; i += TU_THREADS) {
        const int u = i / nch, c = i - u * nch;
        cpa16(area + i, p.W3 + (size_t)(u0 + l_row[k0 + u]) * nch + c);
      }
      cpa_commit_wait();
      __syncthreads();
      // h_bk = A(z_bk) (W3[unit_k, :] . x_b): one warp per unit
      for (int u = warp; u < nb; u += TU_WARPS) {
        const uint4* w3 = area + (size_t)u * nch;
        float acc[TU_BMAX];
#pragma unroll
        for (int b = 0; b < TU_BMAX; ++b) acc[b] = 0.f;
        for (int c = lane; c < nch; c += 32) {
          float wf[8];
          Elt<bf16_tag>::unpack(lds16(w3 + c), wf);
#pragma unroll
          for (int b = 0; b < TU_BMAX; ++b) {
            if (b < B) {
              const float4 x0 = xq[(size_t)(2 * b) * nch + c], x1 = xq[(size_t)(2 * b + 1) * nch + c];
              float a = acc[b];
              a = fmaf(wf[0], x0.x, a);
              a = fmaf(wf[1], x0.y, a);
              a = fmaf(wf[2], x0.z, a);
              a = fmaf(wf[3], x0.w, a);
              a = fmaf(wf[4], x1.x, a);
              a = fmaf(wf[5], x1.y, a);
              a = fmaf(wf[6], x1.z, a);
              acc[b] = fmaf(wf[7], x1.w, a);
            }
          }
        }
        const int row = l_row[k0 + u];
#pragma unroll
        for (int b = 0; b < TU_BMAX; ++b) {
          if (b < B) {
            const float uv = warp_sum(acc[b]);
            if (lane == 0) l_h[(k0 + u) * TU_BMAX + b] = l_a[row * TU_BMAX + b] * (dbl ? activation(p.act, uv) : uv);
          }
        }
      }
      __syncthreads();
      // W2^T rows of the batch replace them; thread t folds chunk c = t (+ 320 j) for every token
      for (int i = tid; i < nb * nch; i += TU_THREADS) {
        const int u = i / nch, c = i - u * nch;
        cpa16(area + i, p.W2t + (size_t)(u0 + l_row[k0 + u]) * nch + c);
      }
      cpa_commit_wait();
      __syncthreads();
      for (int c = tid; c < nch; c += TU_THREADS) {
        float yr[TU_BMAX][8];
#pragma unroll
        for (int b = 0; b < TU_BMAX; ++b)
#pragma unroll
          for (int v = 0; v < 8; ++v) yr[b][v] = 0.f;
        for (int u = 0; u < nb; ++u) {
          float wf[8];
          Elt<bf16_tag>::unpack(lds16(area + (size_t)u * nch + c), wf);
#pragma unroll
          for (int b = 0; b < TU_BMAX; ++b) {
            if (b < B) {
              const float h = l_h[(k0 + u) * TU_BMAX + b];
#pragma unroll
              for (int v = 0; v < 8; ++v) yr[b][v] = fmaf(h, wf[v], yr[b][v]);
            }
          }
        }
#pragma unroll
        for (int b = 0; b < TU_BMAX; ++b) {
          if (b < B) {
            float* yc = p.yacc + ((size_t)b * YACC_COPIES + cp) * D + (size_t)c * 8;
            atomicAdd(reinterpret_cast<float4*>(yc), make_float4(yr[b][0], yr[b][1], yr[b][2], yr[b][3]));
            atomicAdd(reinterpret_cast<float4*>(yc + 4), make_float4(yr[b][4], yr[b][5], yr[b][6], yr[b][7]));
          }
        }
      }
      __syncthreads();  // the area is reused by the next batch
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == TU_MMA_WARP0) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

}  // namespace

cudaError_t ffn_tcu_prepare(size_t max_smem) {
  return cudaFuncSetAttribute(ffn_tcu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
}

int launch_ffn_tcu(const TcPlan& plan, const TcMaps& maps, const void* W3, const void* W2t, float* yacc, int* ctrl,
                   uint8_t* mask, const void* x, int D, int H, int B, int act, int flags, float thr,
                   unsigned long long timeout_ns, size_t max_smem, cudaStream_t s, cudaError_t* cuda_err) {
  *cuda_err = cudaSuccess;
  if (!plan.ok || B < 1 || B > TU_BMAX || plan.NU > TU_ROWS) return -1;
  const int NB = 16;  // x box rows (B <= 8 tokens, zero-filled past B)
  CUtensorMap mx;
  if (int rc = encode_2d(&mx, x, (uint64_t)B, (uint64_t)D, (uint64_t)D * 2, (uint32_t)NB)) return rc;
  TcuArgs a;
  a.D = D;
  a.H = H;
  a.B = B;
  a.NB = NB;
  a.NU = plan.NU;
  a.KC = plan.KC;
  a.C = 4;
  a.NCG = (plan.KC + a.C - 1) / a.C;
  a.NS = (int)std::max<size_t>(2, std::min<size_t>(TU_NS_MAX, TU_SMEM_BUDGET / tcu_stage_bytes(a.C, plan.NU, NB)));
  while (a.NS > 2 && tcu_smem_bytes(a.C, plan.NU, NB, a.NS) > max_smem) --a.NS;
  a.act = act;
  a.flags = flags;
  a.thr = thr;
  a.nacc = 4;
  a.tmem_cols = 64;  // 4 accumulators x NB = 16 fp32 columns
  a.W3 = static_cast<const uint4*>(W3);
  a.W2t = static_cast<const uint4*>(W2t);
  a.x = static_cast<const uint4*>(x);
  a.yacc = yacc;
  a.ctrl = ctrl;
  a.mask = mask;
  a.timeout_ns = timeout_ns;
  const size_t smem = tcu_smem_bytes(a.C, plan.NU, NB, a.NS);
  if (smem > max_smem ||
      (size_t)a.NS * tcu_stage_bytes(a.C, plan.NU, NB) < tcu_epilogue_bytes(NB, B, D)) {
    *cuda_err = cudaErrorInvalidConfiguration;
    return 0;
  }
  *cuda_err = launch_pdl(ffn_tcu_kernel, dim3(plan.ntiles), dim3(TU_THREADS), smem, s, maps.w1, mx, a);
  return 0;
}

}  // namespace sffn
