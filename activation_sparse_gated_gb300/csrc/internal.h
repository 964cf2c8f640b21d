// internal.h -- kernel launchers shared by the C-ABI host code (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sffn {

// Fused single-token forward: gate -> compaction -> gathered W3 rows ->
// gathered W2^T rows -> cross-block reduction.
struct B1Params {
  const void* gate_w;     // W1[H, D] (standard gate) or U[H, r] (low-rank gate)
  const void* W3;         // [H, D]
  const void* W2t;        // [H, D]  (W2 transposed: the column of unit i is row i)
  const void* x;          // [D]
  const float* t = nullptr;  // [r] fp32 t = V x for the low-rank gate, else nullptr
  void* y;                // [D]
  float* yacc;            // [D] fp32 accumulator, all zero between calls
  int* ctrl;              // ticket / error word / live-count accumulator
  int* counts;            // [1] live count of this call
  uint8_t* mask;          // [H] live flags of this call (nullptr: not recorded)
  int D, H, gate_k;       // gate_k = D (standard) or r (low-rank)
  int act;
  int count_slot;         // index of this token's live-count accumulator
  int rows_cap;           // streaming kernel: max units per block (live-list capacity)
  int pref_rows;          // streaming kernel: gate rows per block prefetched into shared memory
  int gather_rows;        // streaming kernel: W3 rows per gather batch (shared area / row)
  int flags = 0;          // FLAG_TILED_G | FLAG_RMSNORM (low-rank gate) | FLAG_DOUBLE_ACT
  float thr = 0.f;        // live iff |A(z)| > thr
  const float* s1 = nullptr;  // int8 weights: per-unit scales of the W1 and W3 codes,
  const float* s3 = nullptr;  // per-output scales of the W2 codes
  const float* s2 = nullptr;
  float* ypart = nullptr;  // deterministic option: [grid, D] partial y of every block (plain stores)
};

// Streaming form of the fused forward (16 warps, no spin-waits); grid =
// blocks, each owning a slice of units.  The plan fixes the shared-memory
// prefetch depth, the gather batch and the dynamic shared-memory size.
struct StreamPlan {
  int pref_rows = 0, gather_rows = 1;
  size_t smem = 0;
};
StreamPlan plan_ffn_b1_stream(int D, int gate_k, int elt_bytes, bool lopa, int rows_cap);
cudaError_t ffn_b1_stream_prepare(size_t max_smem);
int ffn_b1_stream_threads();
cudaError_t launch_ffn_b1_stream(const B1Params& p, int dtype, bool lopa, int grid, size_t smem,
                                 cudaStream_t s);

// bf16 form of the single-token forward (ffn_b1_bf16.cu): gate rows through
// two refilled shared halves, packed fp32x2 dot products, register gathers.
StreamPlan plan_ffn_b1_bf16(int D, int gate_k, bool lopa, int rows_cap);
cudaError_t ffn_b1_bf16_prepare(size_t max_smem);
cudaError_t launch_ffn_b1_bf16(const B1Params& p, bool lopa, int grid, size_t smem, cudaStream_t s);
int ffn_b1_bf16_threads();

// Small-batch form (2..8 tokens per launch, CUDA cores): one pass over the
// gate slice serves every token; gathers follow the union of live sets.
struct BatchPlan {
  int pref_rows = 0, gather_rows = 1;
  size_t smem = 0;
};
BatchPlan plan_ffn_batch(int D, int gate_k, int elt_bytes, bool lopa, int rows_cap, int nb_max);
cudaError_t ffn_batch_prepare(size_t max_smem);
cudaError_t launch_ffn_batch(const B1Params& p, int nb, int dtype, bool lopa, int grid, size_t smem,
                             cudaStream_t s);

// Batched forward on the tensor cores (bf16, standard gate): a gate-up kernel
// ([Z | P] = [W1 | W3] X^T, live flags and counts, h = A(z) * p where z > 0)
// and a down kernel (y^T += W2^T[units]^T h into the accumulator copies); the
// finalize kernel follows.  Gate-up: one block per slice of NU units, MT = MMA
// rows (64 or 128).  Down: ndt slices of 128 y values x nsplit ranges of the
// nch 64-unit chunks.
struct TcPlan {
  bool ok = false;
  int NU = 0, MT = 0, ntiles = 0, KC = 0;
  int r = 0, KCZ = 0;  // low-rank gate: rank and its 64-wide K chunks (0: standard gate)
  int NUt = 0, ntiles_t = 0, ksplit_t = 0;  // low-rank gate, t kernel: rows of V per slice, slices, K ranges
  int t_split_tokens = 1024;  // t kernel: K ranges x padded tokens <= this (its partial sums grow with both)
  int num_sms = 0;
  int ndt = 0, nch = 0, nsplit = 0;
  int Hs = 0;  // row stride (elements) of the h buffer
  size_t gate_smem_budget = 0, down_smem_budget = 0;  // pipeline-stage bytes per block
  int gate_chunks = 0;                                // 64-wide K chunks per gate-up stage (0: 4)
  int tcg_acc = 1;  // union-skip gate kernel: TMEM accumulators per MMA warp
  // streaming down kernel: blocks of an output slice that form a cluster and sum their partial
  // tiles through distributed shared memory (0: nsplit blocks adding into fp32 accumulators)
  int down_cluster = 0;
  // low-rank t kernel: K splits per slice that form a cluster and sum in distributed shared memory
  // (0: ksplit_t splits adding into fp32 sums with a ticket and a last block)
  int t_cluster = 0;
  int tcg_down_cluster = 0;  // union-skip down kernel: blocks per output slice in a cluster (0: atomics)
};
struct TcMaps {
  CUtensorMap w1, w3;  // W1 [H, D] (or U [H, r]), W3 [H, D]: boxes of 64 columns x NU rows
  CUtensorMap w2;      // W2^T [H, D]: boxes of 64 columns x 64 rows
  CUtensorMap v;       // V [r, D] (low-rank gate): boxes of 64 columns x NUt rows
  CUtensorMap h[8];    // h buffer [256, H]: boxes of 64 columns x NB rows, NB = 16 (i + 1)
};
struct TcBuffers {
  uint16_t* hbuf;  // ffn_tc_hbuf_elems(plan) bf16 values: h of token b in row b
  float* yacc;     // [B_max * YACC_COPIES, D]
  int* ctrl;
  uint8_t* mask;   // [B_max, H]
  int* counts;     // [B_max] published live counts
  int* tickets;    // [TC_TICKETS] zero between calls
  uint16_t* tpair; // low-rank gate: [2 NB, r] bf16, t_hi rows then t_lo rows (the t kernel); else null
  float* tacc;     // low-rank gate: [128, r] fp32 partial sums of t, zero between calls
  int* tickets_t;  // low-rank gate: [TC_TICKETS] slices of the t kernel, zero between calls
};
constexpr int TC_TICKETS = 64;  // >= slices of 128 y values (D <= 8192)
TcPlan plan_ffn_tc(int D, int H, int r, int num_sms);
// Tensor map of a bf16 matrix [rows, cols] (row stride in bytes): boxes of 64
// columns x box_rows rows, 128-byte swizzle.  0 on success, else a driver
// status (-1: the encoder entry point is unavailable).
int encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t stride_bytes,
              uint32_t box_rows);
size_t ffn_tc_hbuf_elems(const TcPlan& p);
// 0 on success, else a driver status (or -1: tensor-map encoder unavailable)
int encode_tc_maps(TcMaps* m, const TcPlan& p, const void* W1, const void* V, const void* W3, const void* W2t,
                   uint16_t* hbuf, int D, int H);
cudaError_t ffn_tc_prepare(size_t max_smem);
// Chooses TcPlan::down_cluster (and, for a low-rank gate, TcPlan::t_cluster): the largest cluster
// of 2..8 blocks per slice whose clusters are all resident at once (cudaOccupancyMaxActiveClusters);
// 0 when none is.
cudaError_t ffn_tc_plan_cluster(TcPlan& plan, size_t max_smem);
// Whole forward (y and counts written; no finalize kernel).  Low-rank gate:
// tpair_ready says the caller already wrote the t pair (launch_lopa_t_pair);
// otherwise the t kernel runs on the tensor cores first (t_only: and nothing
// else -- the t pair for the union-skip kernels).  Returns 0 and sets
// *cuda_err to the launch status, or a non-zero encode status.
int launch_ffn_tc(const TcPlan& plan, const TcMaps& maps, const TcBuffers& buf, const void* x, void* y, int D, int H,
                  int B, int act, int flags, float thr, unsigned long long timeout_ns, size_t max_smem, cudaStream_t s,
                  cudaError_t* cuda_err, bool tpair_ready = false, bool t_only = false);
// Low-rank batches of up to this many tokens take the CUDA-core t kernel
// (measured per call on the low-rank workload: 31.5 against 31.6 us at B = 2;
// at B = 4 the split tensor-core t kernel is faster, 31.9 against 33.9 us).
constexpr int TC_T_CUDA_CORE_MAX_B = 2;

// Small batches (2..8 tokens, bf16, standard gate; ffn_tcu.cu): the gate on the
// tensor cores, the union of the live sets gathered on the CUDA cores, fp32
// atomics into the accumulator copies (the finalize kernel follows).  Returns 0
// and sets *cuda_err to the launch status, or a non-zero encode status.
cudaError_t ffn_tcu_prepare(size_t max_smem);
int launch_ffn_tcu(const TcPlan& plan, const TcMaps& maps, const void* W3, const void* W2t, float* yacc, int* ctrl,
                   uint8_t* mask, const void* x, int D, int H, int B, int act, int flags, float thr,
                   unsigned long long timeout_ns, size_t max_smem, cudaStream_t s, cudaError_t* cuda_err);

// Small batches with the union skip (bf16, standard gate; ffn_tcg.cu): a gate
// kernel (Z = W1 X^T on the tensor cores, live flags, the union of the live
// sets compacted into a list, then P = W3[union] X^T from gathered rows and
// h = A(z) * p at the union positions) and a down kernel (y^T += the union's
// gathered W2^T rows^T h; the last block of a y slice rounds y).  Returns 0
// and sets *cuda_err to the launch status, or a non-zero encode status.
constexpr int TCG_MAX_BATCH = 32;
struct TcgBuffers {
  int* ulist;    // [H] the union's units, in the order the gate blocks reserved them
  int* ucount;   // [1] units in the union, zero between calls
  int* dticket;  // [1] down blocks done, zero between calls
};
cudaError_t ffn_tcg_prepare(size_t max_smem);
// Chooses TcPlan::tcg_down_cluster as ffn_tc_plan_cluster does for the streaming down kernel.
cudaError_t ffn_tcg_plan_cluster(TcPlan& plan, size_t max_smem);
int launch_ffn_tcg(const TcPlan& plan, const TcMaps& maps, const TcBuffers& buf, const TcgBuffers& ub, const void* W3,
                   const void* W2t, const void* x, void* y, int D, int H, int B, int act, int flags, float thr,
                   unsigned long long timeout_ns, size_t max_smem, cudaStream_t s, cudaError_t* cuda_err);

// Deterministic option: y = round(sum over blocks b = 0 .. nblocks-1, in that
// order, of ypart[b, :]) for one token, and its live count published.
cudaError_t launch_finalize_ordered(const float* ypart, int nblocks, void* y, int* ctrl, int* counts, int count_slot,
                                    int D, cudaStream_t s);

// y[b] = round(sum of the accumulator copies of token b) for b < nb; clears the
// copies and publishes the nb live counts (chained behind a forward kernel).
cudaError_t launch_finalize(float* yacc, void* y, int* ctrl, int* counts, int count_slot, int D, int nb,
                            int dtype, cudaStream_t s);

// Weight-only int8 or int4 (bits), standard gate, one token per launch (ffn_b1_i8.cu):
// codes W1q, W3q, W2tq [H, D] in gate_w, W3, W2t (int4: two per byte, D / 2 bytes a
// row, code 2b in the low nibble of byte b); scales s1, s3 [H] (int4: [H, D / 64], one
// per group of 64 columns), s2 [D] in the params (each block scales its partial y by
// s2 before adding it up).
StreamPlan plan_ffn_b1_i8(int D, int gate_k, int rows_cap, int bits, bool lowrank);
// Low-rank gate, int8 weights: t [r] fp32 = sV * (qV [r, D] . x) for one bf16 token x (D % 16 == 0,
// D <= 4096); the int8 kernel then takes gate_k = r, gate_w = qU [H, r], t.
cudaError_t launch_lopa_t_i8(const void* qV, const float* sV, const void* x, float* t, int r, int D, cudaStream_t s);
cudaError_t ffn_b1_i8_prepare(size_t max_smem);
cudaError_t launch_ffn_b1_i8(const B1Params& p, int grid, size_t smem, cudaStream_t s, int bits);
// Per-row symmetric quantisation of a bf16 matrix [rows, cols] to one code per byte in
// [-qmax, qmax] (127: int8, 7: int4 before packing).
cudaError_t launch_quantize_rows(const void* src_bf16, int8_t* dst, float* scale, int rows, int cols, cudaStream_t s,
                                 int qmax);
// int4 W1, W3: one scale per group of 64 columns, scale[row * (cols / 64) + g], codes one per byte.
cudaError_t launch_quantize_groups4(const void* src_bf16, int8_t* dst, float* scale, int rows, int cols,
                                    cudaStream_t s);
constexpr int INT4_GROUP = 64;
// int4 codes one per byte -> two per byte (n_codes even); a code outside [-7, 7] sets
// DEV_ERR_CHECK in *err.  And back, sign-extended.
cudaError_t launch_pack_int4(const int8_t* codes, void* packed, size_t n_codes, int* err, cudaStream_t s);
cudaError_t launch_unpack_int4(const void* packed, int8_t* codes, size_t n_codes, cudaStream_t s);

// t[b, :] = V x[b, :] in fp32 for the low-rank gate (one warp per row of V).
cudaError_t launch_lopa_t(const void* V, const void* x, float* t, int r, int D, int B, int dtype,
                          cudaStream_t s);
// The same for bf16 tensor-core batches, written as a bf16 pair into tpair
// [2 NB, r]: t_hi of token b in row b, t_lo in row NB + b, zero rows for b >= B.
// lopa_t_prepare raises the batch kernel's shared-memory limit (once per process).
cudaError_t lopa_t_prepare();
cudaError_t launch_lopa_t_pair(const void* V, const void* x, uint16_t* tpair, int r, int D, int B, int NB,
                               cudaStream_t s);

// W2[D, H] -> W2t[H, D] (element size 1, 2 or 4 bytes).
cudaError_t launch_transpose(const void* src, void* dst, int rows, int cols, int elt_bytes,
                             cudaStream_t s);

// Wait on a flag nothing sets for at most limit_ns, then record a timeout.
cudaError_t launch_timeout_probe(int* ctrl, unsigned long long limit_ns, cudaStream_t s);

// Store a message for sffn_last_error() on the calling thread.
void set_last_error(const char* msg);

// Launch helper: programmatic stream serialization on (the kernel may start
// before its predecessor finishes and must call griddepcontrol.wait first).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// The same with thread-block clusters of cluster_x blocks along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace sffn
