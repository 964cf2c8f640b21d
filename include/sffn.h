/*
 * sffn.h -- gate-first sparse gated-FFN forward (C ABI).
 *
 * One handle holds one FFN layer.  For each token x in R^D the forward pass
 * computes the gate first, keeps only the live hidden units and reads only
 * their rows of W3 and their columns of W2:
 *
 *     z = W1 x                (standard gate, W1 in R^{H x D}), or
 *     z = U (V x)             (low-rank gate, U in R^{H x r}, V in R^{r x D})
 *     S = { i : z_i > 0 }     (the live units; ReLU and R-S+ vanish for z <= 0)
 *     y = sum_{i in S} W2[:, i] * A(z_i) * (W3[i, :] . x)
 *
 * which equals the dense gated FFN y = W2 (A(W1 x) .* (W3 x)) exactly in real
 * arithmetic.  Sources: "Model casting: compute the gate, then skip most of
 * the FFN" (ai.thesatyajit.com), sections "What an FFN actually computes"
 * (the formula and the skip argument), "The 3x ceiling, and why W1 is always
 * on" (the gate must run in full), "Model casting: make sparsity a target"
 * (R-S+), "LoPA Gating: moving the ceiling" (W1 = G + UV; this library
 * implements the UV part, with no G, no RMSNorm between V and U and the
 * activation on the gate only).
 *
 * Conventions
 *   - Every call returns SFFN_OK (0) or a negative SFFN_ERR_* code; the
 *     thread-local sffn_last_error() then holds a one-line message.  No C++
 *     exception crosses this boundary.
 *   - Matrices are dense row-major.  x and y are [B, D] row-major.
 *   - Arithmetic: products and sums in fp32 (FFMA, never TF32); the low-rank
 *     vector t = V x and the products h_i stay fp32; y is rounded once to the
 *     handle's dtype (round-to-nearest-even for bf16).
 *   - The handle owns all library memory (packed weights, accumulators,
 *     counters).  It is not thread-safe and must not be used by two streams
 *     at once; concurrent layers need separate handles.
 *   - Numerical sums over live units are accumulated across thread blocks.
 *     The single-token and union-gather kernels add partial y with fp32
 *     atomics, so there y can differ from run to run in its last bits (unless
 *     the handle is created with SFFN_DETERMINISTIC); the tensor-core batched
 *     down kernels sum their partial tiles inside a thread-block cluster in a
 *     fixed order when the cluster fits (the default).  The live set and the
 *     counts are deterministic.
 */
#ifndef SFFN_H
#define SFFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sffn_s* sffn_t;

/* element type of W1/U, V, W3, W2, x and y.  SFFN_I8W: weight-only int8 --
   W1 (or U and V), W3 and W2 are held as int8 codes with one fp32 scale per
   output channel, x and y are bf16 (see sffn_set_weights_int8).  SFFN_I4W:
   the same with int4 codes in [-7, 7], held two per byte, and one scale per
   group of 64 columns for W1 and W3 */
enum { SFFN_F32 = 0, SFFN_BF16 = 1, SFFN_I8W = 2, SFFN_I4W = 3 };

/* activation A: ReLU, or R-S+ (z * sigmoid(z) for z >= 0, 0 for z < 0;
   "Model casting: make sparsity a target") */
enum { SFFN_ACT_RELU = 0, SFFN_ACT_RSP = 1, SFFN_ACT_SILU = 2 };

enum {
  SFFN_OK = 0,
  SFFN_ERR_ARG = -1,      /* bad size, null pointer, unknown enum value      */
  SFFN_ERR_ALIGN = -2,    /* a pointer is not 16-byte aligned                */
  SFFN_ERR_DTYPE = -3,    /* dtype/shape combination not supported           */
  SFFN_ERR_CUDA = -4,     /* a CUDA runtime call failed (message has details) */
  SFFN_ERR_TIMEOUT = -5,  /* a device-side wait ran out of time; the kernel
                             returned early and its outputs are invalid      */
  SFFN_ERR_STATE = -6,    /* call out of order (e.g. forward before weights) */
  SFFN_ERR_NOMEM = -7,    /* device allocation failed                        */
  SFFN_ERR_DEVICE = -8    /* a device-side bounds or alignment check failed:
                             the checked access was skipped, outputs of the
                             affected forward are invalid                     */
};

/* limits of this build */
#define SFFN_MAX_BATCH 128
#define SFFN_MAX_D_BF16 4096
#define SFFN_MAX_D_F32 2048

/*
 * Create a layer on the current CUDA device.
 *   D      model width, D % 8 == 0, 8 <= D <= SFFN_MAX_D_BF16 (bf16) or
 *          SFFN_MAX_D_F32 (f32)
 *   H      hidden width (H' for the low-rank gate), any H >= 1
 *   r      0 for the standard gate W1; r > 0 selects the low-rank gate U(Vx)
 *          with rank r, r % 8 == 0, r <= D
 *   act    SFFN_ACT_RELU, SFFN_ACT_RSP, or SFFN_ACT_SILU (z sigmoid(z) for every
 *          z: the smooth gate, never exactly zero; see sffn_set_live_threshold)
 *   dtype  SFFN_F32, SFFN_BF16, SFFN_I8W (int8 weights, bf16 x and y; needs
 *          D % 16 == 0 and r % 16 == 0; flags may only hold SFFN_DOUBLE_ACT), or
 *          SFFN_I4W (int4 weights, standard gate, D % 64 == 0)
 * Returns NULL on error (see sffn_last_error()).  Allocates device memory:
 * 3*H*D (+ r*D + H*r) elements of weights plus O(B_max * (D + r + H)) bytes of
 * accumulators.
 * Kernel selection reads these environment variables once, here (tuning and
 * measurement only; the defaults are the measured best, the results are the
 * same up to fp32 summation order): SFFN_STREAM_BLOCKS_PER_SM (1..4, default
 * 1), SFFN_TC_MIN_BATCH (smallest bf16 batch on the tensor cores, default 2),
 * SFFN_TCU_MAX_BATCH (largest standard-gate batch taking the union-gather
 * kernel, 0..8, default 2), SFFN_TC_T_CUDA_MAX_B (largest low-rank batch whose
 * t runs on the CUDA cores, default 2), SFFN_TC_T_SPLIT_TOKENS (K ranges of
 * the tensor-core t kernel times padded tokens, default 1024),
 * SFFN_TC_GATE_KB / SFFN_TC_DOWN_KB (pipeline-stage bytes per block of the
 * tensor-core kernels, default 200; 220 for the low-rank gate-up kernel),
 * SFFN_TC_GATE_CHUNKS (64-wide K chunks per gate-up stage, 1..4, default by
 * batch), SFFN_TC_DOWN_CLUSTER / SFFN_TC_T_CLUSTER (0: the down kernels and
 * the low-rank t kernel sum their K splits with fp32 atomics and a last block
 * instead of inside a thread-block cluster), SFFN_TCG_MAX_BATCH (batches of
 * 3..N tokens always take the union-skip kernels, 0: never; unset: the
 * live-fraction rule), SFFN_TCG_ACC (TMEM accumulators per MMA warp of the
 * union-skip gate kernel, 1..4, default 1).
 */
sffn_t sffn_create(int D, int H, int r, int act, int dtype);

/*
 * Options of the pages' full low-rank gate ("LoPA Gating: moving the ceiling",
 * W1(x) = Gx + U RMSNorm(Vx), with the activation applied to both W1 x and
 * W3 x), combined with | in sffn_create_ex's flags:
 *   SFFN_GATE_TILED_G  z_i += x_{i mod D}: G is the fixed tiled identity
 *                      ("Model Casting and Low-Parameter Gating", appendix
 *                      Figure 6 (c)); low-rank gate only
 *   SFFN_GATE_RMSNORM  t = V x is replaced by t / sqrt(mean(t^2) + 1e-6), no
 *                      gain (the pages give neither eps nor a gain); low-rank
 *                      gate only
 *   SFFN_DOUBLE_ACT    a unit's up value is A(W3 x) instead of W3 x; either gate
 * The live test stays z_i > 0 on the (full) gate.
 */
enum { SFFN_GATE_TILED_G = 1, SFFN_GATE_RMSNORM = 2, SFFN_DOUBLE_ACT = 4 };

/*
 * SFFN_DETERMINISTIC (bf16 handles): y is bitwise reproducible run to run.
 * The pages are silent on summation order; by default the single-token and
 * union-gather kernels add each thread block's partial y into an fp32
 * accumulator with atomics, so the last bits of y follow the order in which
 * blocks finish.  With this option every token runs
 * the single-token kernel, a block folds its live units in ascending unit
 * order and writes its partial y to a row of its own, and a finalize kernel
 * sums the rows in block order.  Costs a [blocks, D] fp32 buffer in the handle
 * and one single-token pass per token (batches do not use the batched paths).
 * SFFN_ERR_DTYPE for fp32 and int8 handles.
 */
enum { SFFN_DETERMINISTIC = 8 };

/*
 * sffn_create with options: flags is 0 or a combination of the values above.
 * SFFN_ERR_ARG (NULL return) for unknown bits or a low-rank option with r == 0;
 * SFFN_ERR_DTYPE for SFFN_DETERMINISTIC on a handle that is not bf16.
 * sffn_create(D, H, r, act, dtype) is sffn_create_ex(D, H, r, act, dtype, 0).
 */
sffn_t sffn_create_ex(int D, int H, int r, int act, int dtype, int flags);

/*
 * Live threshold (default 0): unit i is live -- its W3 row and W2 column are
 * read -- iff |A(z_i)| > thr; a dead unit contributes exactly nothing.  With
 * thr = 0, ReLU and R-S+ keep {i : z_i > 0} (the exact skip); SiLU needs a
 * thr > 0 to skip anything, which makes the result an approximation whose
 * error per output is at most thr * sum_i |W2[m, i]| |(W3 x)_i| ("Model
 * casting: compute the gate, then skip most of the FFN": thresholding the
 * small values of a smooth gate).  thr must be finite and >= 0 (SFFN_ERR_ARG);
 * it applies to the forwards issued after the call.
 */
int sffn_set_live_threshold(sffn_t h, float thr);

/*
 * Expected live fraction rho per token, which picks the kernels of a batch of
 * 3 <= B <= 16 tokens (bf16 handles; the low-rank gate without RMSNorm).  A
 * batch needs the W3 rows and W2 columns of the union of its tokens' live
 * sets, about 1 - (1 - rho)^B of the units ("Model casting: compute the gate, then skip most of the FFN", on
 * batching).  The union-skip kernels read the gate (W1, or U after t = V x) in
 * full and then only the union's rows of W3 and W2^T; the streaming kernels
 * read every slice of W3 and W2 and let the gate zero the dead terms.  The
 * forward takes the union-skip kernels when the expected union is at most 30 %
 * of the units and the W3 and W2 bytes of the other units come to at
 * least 128 MB (64 MB for the low-rank gate), else the streaming kernels:
 * on this GPU a gathered row arrives at a fraction of the streaming bandwidth,
 * and the rows can only be requested once the gate is known.  Both compute the
 * same y within rounding.  rho in [0, 1] (SFFN_ERR_ARG otherwise); a negative
 * value forgets it (then batches stream, the default).  sffn_active_counts sets
 * rho to the mean count / H it returns.  Setting the environment variable
 * SFFN_TCG_MAX_BATCH=N before sffn_create forces the union-skip kernels for
 * 3 <= B <= N (N <= 32; 0 never).
 */
int sffn_set_live_fraction_hint(sffn_t h, float rho);

/*
 * Copy the layer's weights into the handle (host or device pointers, any
 * alignment, dtype of the handle):
 *   W1_or_U  W1[H, D] when r == 0, else U[H, r]
 *   V        V[r, D] when r > 0, else ignored (may be NULL)
 *   W3       W3[H, D]
 *   W2       W2[D, H]  -- stored transposed (H-major) inside the handle so that
 *            the column of a live unit is one contiguous row
 * Work is issued on `stream` (a cudaStream_t, NULL = legacy default) and the
 * call returns after it has completed.  The caller keeps ownership of its
 * buffers.  May be called again to replace the weights.
 */
int sffn_set_weights(sffn_t h, const void* W1_or_U, const void* V, const void* W3,
                     const void* W2, void* stream);

/*
 * Weight-only int8 and int4 handles (dtypes SFFN_I8W, SFFN_I4W).  "Model
 * Casting and Low-Parameter Gating", appendix Table 17, quantises cast models
 * weight-only to int8 and to int4 and gives no scale convention; this library
 * uses symmetric per-output-channel scales: one fp32 scale per row of W1 and of
 * W3 (per unit) and per row of W2 (per output element), s = max|w| / Q, code =
 * round-half-to-even(w / s) clamped to [-Q, Q], both computed in binary32 (s = 0
 * and codes 0 for an all-zero row); Q = 127 for int8, 7 for int4.  int4 W1 and
 * W3 take one scale per group of 64 consecutive columns of a row instead (the
 * max over the group): with one int4 scale per row a single large entry, such
 * as a gate bias carried as a weight column, rounds the rest of the row to 0.
 * The forward uses the dequantised weights q * s:
 *     z_i = s1_i (q1[i, :] . x),   u_i = s3_i (q3[i, :] . x),
 *     y_m = s2_m sum_{i live} q2[m, i] A(z_i) u_i
 * (int4: z_i = sum_g s1_{i,g} (q1[i, 64g .. 64g + 63] . x[64g .. 64g + 63]),
 * likewise u_i) with fp32 sums and y rounded once to bf16.
 *
 * On such a handle sffn_set_weights takes bf16 W1[H, D], W3[H, D], W2[D, H]
 * (V ignored) and quantises them on the device.  With the low-rank gate (int8
 * only, the plain form z = U (V x)) it takes bf16 U[H, r], V[r, D], W3, W2 and
 * gives U and V one scale per row as well: t = sV (qV x), z = sU (qU t).  sffn_set_weights_int8 loads
 * codes and scales quantised elsewhere (a quantisation-aware-trained layer):
 *   W1q, W3q [H, D] int8 with s1, s3 [H] fp32;  W2q [D, H] int8 with s2 [D] fp32
 * (host or device pointers, any alignment).  On an SFFN_I4W handle the code
 * arrays hold one int4 code per byte, each in [-7, 7] (the library packs them
 * two per byte; a code outside that range gives SFFN_ERR_ARG and leaves the
 * handle without weights), and s1, s3 are [H, D / 64] (scale of row i, columns
 * 64 g .. 64 g + 63 at i * D / 64 + g).  sffn_get_weights_int8 copies the handle's codes (one per
 * byte) and scales out in the same layout (any pointer may be NULL to skip that
 * array); on a low-rank int8 handle W1q and s1 receive U's codes [H, r] and
 * scales [H], and sffn_set_weights_int8 returns SFFN_ERR_STATE (such a handle
 * takes bf16 weights).  Both return after `stream` has finished the copies, and
 * return SFFN_ERR_STATE on a handle of another dtype.
 */
int sffn_set_weights_int8(sffn_t h, const int8_t* W1q, const float* s1, const int8_t* W3q, const float* s3,
                          const int8_t* W2q, const float* s2, void* stream);
int sffn_get_weights_int8(sffn_t h, int8_t* W1q, float* s1, int8_t* W3q, float* s3, int8_t* W2q, float* s2,
                          void* stream);

/*
 * y[B, D] = FFN(x[B, D]) for 1 <= B <= SFFN_MAX_BATCH.  x and y are device
 * pointers of the handle's dtype, 16-byte aligned, and must not overlap.  The
 * call is asynchronous and stream-ordered on `stream`; y is fully overwritten.
 * Successive forwards on one stream overlap the weight prefetch of the next
 * call with the tail of the previous one (programmatic dependent launch); a
 * forward still observes every write an earlier operation in the stream made
 * to x.  Device-side failures (SFFN_ERR_TIMEOUT) surface at the next
 * sffn_synchronize / sffn_active_counts / sffn_active_mask call.
 */
int sffn_forward(sffn_t h, const void* x, void* y, int B, void* stream);

/*
 * Number of live units |S_b| per token of the most recent forward, B values
 * (B must equal that forward's batch).  Waits for that forward to finish.
 */
int sffn_active_counts(sffn_t h, int* counts_host, int B);

/*
 * Live flags of the most recent forward: mask_host[b*H + i] = 1 iff z_i > 0
 * for token b, else 0 (B*H bytes).  Waits for that forward to finish.
 */
int sffn_active_mask(sffn_t h, uint8_t* mask_host, int B);

/*
 * Wait for all work this handle issued and report any device-side error
 * recorded since the last check (the error word is cleared).
 */
int sffn_synchronize(sffn_t h);

/* Release the handle and its device memory (waits for its pending work). */
void sffn_destroy(sffn_t h);

/* Static description of a status code. */
const char* sffn_strerror(int code);

/* The calling thread's message for its most recent failed call ("" if none). */
const char* sffn_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int sffn_version(void);

/*
 * Test hook for failure detection: launch one block on `stream` that waits on
 * a device flag nothing ever sets, with a limit of `limit_us` microseconds
 * (1..1000000), after which it records SFFN_ERR_TIMEOUT in the handle's error
 * word and returns.  The next sffn_synchronize reports it.  Faults nothing.
 */
int sffn_debug_timeout_probe(sffn_t h, int limit_us, void* stream);

/*
 * Forward without any device allocation, for callers that cannot call
 * cudaMalloc (a runtime that owns all device memory through its own arena, code
 * on a latency path where an allocation would stall the device, a host that
 * only lends out buffers it owns).  The pages have no counterpart: this is a
 * packaging of the same standard-gate forward as sffn_forward.
 *   W1, W3   [H, D] row-major device pointers
 *   W2t      W2 transposed, [H, D] row-major (row i = column i of W2), device
 *   x, y     [B, D] device pointers, must not overlap; y fully overwritten
 *   counts   optional device int[B] receiving |S_b| per token, or NULL
 *   D, H, B, act, dtype as for sffn_create / sffn_forward (standard gate,
 *            ReLU or R-S+ only)
 * W1, W3, W2t, x and y must be 16-byte aligned, counts 4-byte aligned
 * (SFFN_ERR_ALIGN otherwise).  The scratch (four fp32 accumulator copies of D
 * floats, control words, count accumulators) is one static device array of
 * 66,816 bytes inside the library, so D is limited to 4096 (bf16) / 2048
 * (f32); larger D is rejected with SFFN_ERR_ARG and a message.
 * Each token is one pass of the single-token streaming kernel plus the
 * finalize kernel, so the cost grows linearly with B (a full read of W1 per
 * token): the entry point is meant for B = 1, batches belong on a handle.
 * The kernels wait on nothing on the device, so there is no device-side
 * timeout to report.
 * The first call on a device looks up that array's address and sets kernel
 * attributes for the device, so make it before any stream capture.  Every
 * call clears the scratch it needs on `stream` and then launches; calls that
 * overlap on the GPU (different streams, or several threads) share the one
 * array and race, so serialise them.  Returns SFFN_OK once the work is
 * enqueued.
 */
int sffn_forward_noalloc(const void* W1, const void* W3, const void* W2t, const void* x, void* y,
                         int* counts, int D, int H, int B, int act, int dtype, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SFFN_H */
