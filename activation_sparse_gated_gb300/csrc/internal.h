// internal.h -- kernel launchers shared by the C-ABI host code (not installed).
#pragma once

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
  const float* t;         // [r] fp32 t = V x for the low-rank gate, else nullptr
  void* y;                // [D]
  float* yacc;            // [D] fp32 accumulator, all zero between calls
  int* ctrl;              // ticket / error word / live-count accumulator
  int* counts;            // [1] live count of this call
  uint8_t* mask;          // [H] live flags of this call (nullptr: not recorded)
  int D, H, gate_k;       // gate_k = D (standard) or r (low-rank)
  int ns1, ns2;           // gate-row ring slots, gather ring slots
  int act;
  int count_slot;         // index of this token's live-count accumulator
  int rows_cap;           // streaming kernel: max units per block (live-list capacity)
  int pref_rows;          // streaming kernel: gate rows per block prefetched into shared memory
  int gather_rows;        // streaming kernel: W3 rows per gather batch (shared area / row)
  unsigned long long timeout_ns;
};

constexpr int B1_NWG = 8;                               // gate warps
constexpr int B1_NGA = 4;                               // gather warps
constexpr int B1_THREADS = (1 + B1_NWG + B1_NGA) * 32;  // + one producer warp
constexpr int B1_NS1_MAX = 128;
constexpr int B1_NS2_MAX = 16;
constexpr int B1_MAXC = 4;  // 16-byte chunks of a D-row per gather thread (D*elt <= 8 KB)

// Shared-memory bytes of the fused kernel for a given ring configuration.
size_t ffn_b1_smem_bytes(int D, int gate_k, int elt_bytes, bool lopa, int ns1, int ns2);
// Raise the kernels' dynamic shared-memory limit (once per device).
cudaError_t ffn_b1_prepare(size_t max_smem);
cudaError_t launch_ffn_b1(const B1Params& p, int dtype, bool lopa, int grid, size_t smem,
                          cudaStream_t s);

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

// y[b] = round(sum of the accumulator copies of token b) for b < nb; clears the
// copies and publishes the nb live counts (chained behind a forward kernel).
cudaError_t launch_finalize(float* yacc, void* y, int* ctrl, int* counts, int count_slot, int D, int nb,
                            int dtype, cudaStream_t s);

// t[b, :] = V x[b, :] in fp32 for the low-rank gate (one warp per row of V).
cudaError_t launch_lopa_t(const void* V, const void* x, float* t, int r, int D, int B, int dtype,
                          cudaStream_t s);

// W2[D, H] -> W2t[H, D] (element size 2 or 4 bytes).
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

}  // namespace sffn
