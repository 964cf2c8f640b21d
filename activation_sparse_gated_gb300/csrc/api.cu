// api.cu -- the C ABI of include/sffn.h: handles, argument checks, weight
// repacking (W2 -> W2^T), launch planning and dispatch, error reporting.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <new>

#include "common.cuh"
#include "internal.h"
#include "sffn.h"

using namespace sffn;

namespace {

thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return code;
}

#define SFFN_CUDA(call)                                                                        \
  do {                                                                                         \
    cudaError_t e_ = (call);                                                                   \
    if (e_ != cudaSuccess)                                                                     \
      return fail(e_ == cudaErrorMemoryAllocation ? SFFN_ERR_NOMEM : SFFN_ERR_CUDA,            \
                  "%s failed: %s", #call, cudaGetErrorString(e_));                             \
  } while (0)

constexpr unsigned long long kTimeoutNs = 250000000ull;  // 250 ms per device-side wait
constexpr int kTicketInts = 2 * TC_TICKETS + 2;  // down-kernel slices, t-kernel slices, union count and ticket

}  // namespace

void sffn::set_last_error(const char* msg) { snprintf(g_msg, sizeof g_msg, "%s", msg); }

struct sffn_s {
  int D = 0, H = 0, r = 0, act = 0, dtype = 0, elt = 0;
  int welt = 0;  // bytes of a stored weight element (1: the int8 / int4 code arrays of SFFN_I8W / SFFN_I4W)
  int qbits = 0; // weight-only codes: 8 (SFFN_I8W), 4 (SFFN_I4W, two per byte), else 0
  int flags = 0;  // SFFN_GATE_TILED_G | SFFN_GATE_RMSNORM | SFFN_DOUBLE_ACT
  float thr = 0.f;  // live iff |A(z)| > thr (sffn_set_live_threshold)
  int device = 0, num_sms = 0;
  size_t max_smem = 0;
  void* gate_w = nullptr;  // W1[H, D] or U[H, r]
  void* V = nullptr;       // V[r, D]
  void* W3 = nullptr;      // W3[H, D]
  void* W2t = nullptr;     // W2^T[H, D]
  float* yacc = nullptr;   // [SFFN_MAX_BATCH * YACC_COPIES, D]
  float* tbuf = nullptr;   // [SFFN_MAX_BATCH, r]
  int* ctrl = nullptr;     // CTRL_INTS
  int* counts = nullptr;   // [SFFN_MAX_BATCH]
  uint8_t* mask = nullptr; // [SFFN_MAX_BATCH, H]
  bool weights_set = false;
  int last_B = 0;
  cudaEvent_t ev = nullptr;
  bool ev_valid = false;
  int stream_grid = 0;  // blocks of the streaming standard-gate kernel
  int stream_rows_cap = 0;
  StreamPlan stream_plan;
  BatchPlan batch_plan;  // groups of up to 8 tokens
  // tensor-core batched path (bf16; standard gate, or the low-rank gate without RMSNorm)
  TcPlan tc;
  TcMaps tcm;
  bool tc_ready = false;
  int tc_min_batch = 2;    // batches of at least this many tokens take the tensor-core path
  int tc_t_cuda_max = TC_T_CUDA_CORE_MAX_B;  // low-rank batches up to this many tokens: t on the CUDA cores
  int tcu_max_batch = 2;   // ... and up to this many gather the union of their live sets (ffn_tcu.cu;
                           // from B = 3 its per-block partial sums of all B x D outputs cost more)
  int tcg_force = -1;      // >= 0: batches of 3 .. tcg_force tokens take the union-skip kernels (ffn_tcg.cu)
  float live_frac = -1.f;  // expected live fraction per token (< 0: unknown), for the batch-path choice
  uint16_t* hbuf = nullptr;
  int* tickets = nullptr;  // [2 TC_TICKETS + 2]: down-kernel slices, t-kernel slices, union count, union ticket
  int* ulist = nullptr;    // [H] the union of a small batch's live sets
  float* ypart = nullptr;     // deterministic option: [blocks, D] partial y rows of the single-token kernel
  uint16_t* tpair = nullptr;  // low-rank gate: [256, r] bf16 t pairs of a tensor-core batch
  float* tacc = nullptr;      // low-rank gate: [128, r] fp32 partial sums of the t kernel
  // weight-only int8 / int4: per-output-channel scales of W1 (or U), W3 [H] and W2 [D]; of V [r]
  // for the low-rank gate with int8 weights
  float* qs1 = nullptr;
  float* qs3 = nullptr;
  float* qs2 = nullptr;
  float* qsv = nullptr;
  StreamPlan i8_plan;
  bool b1_bf16 = true;    // bf16 single tokens: ffn_b1_bf16.cu (false: the fp32 streaming kernel's bf16 form)
  StreamPlan bf16_plan;
};

namespace {

int gate_k(const sffn_s* h) { return h->r > 0 ? h->r : h->D; }

void release(sffn_s* h) {
  cudaFree(h->gate_w);
  cudaFree(h->V);
  cudaFree(h->W3);
  cudaFree(h->W2t);
  cudaFree(h->yacc);
  cudaFree(h->tbuf);
  cudaFree(h->ctrl);
  cudaFree(h->counts);
  cudaFree(h->mask);
  cudaFree(h->hbuf);
  cudaFree(h->tickets);
  cudaFree(h->ulist);
  cudaFree(h->tpair);
  cudaFree(h->tacc);
  cudaFree(h->ypart);
  cudaFree(h->qs1);
  cudaFree(h->qs3);
  cudaFree(h->qs2);
  cudaFree(h->qsv);
  if (h->ev) cudaEventDestroy(h->ev);
}

int check_device(const sffn_s* h) {
  int dev = -1;
  SFFN_CUDA(cudaGetDevice(&dev));
  if (dev != h->device)
    return fail(SFFN_ERR_STATE, "handle belongs to device %d but device %d is current", h->device, dev);
  return SFFN_OK;
}

// Wait for the handle's last forward; report and clear a device-side error.
int sync_and_check(sffn_s* h) {
  if (h->ev_valid) {
    SFFN_CUDA(cudaEventSynchronize(h->ev));
  } else {
    SFFN_CUDA(cudaDeviceSynchronize());
  }
  int err = 0;
  SFFN_CUDA(cudaMemcpy(&err, h->ctrl + CTRL_ERR, sizeof(int), cudaMemcpyDeviceToHost));
  if (err != 0) {
    // the aborted kernel may have left partial sums and counters behind
    SFFN_CUDA(cudaMemset(h->ctrl, 0, sizeof(int) * CTRL_INTS));
    SFFN_CUDA(cudaMemset(h->yacc, 0, sizeof(float) * SFFN_MAX_BATCH * YACC_COPIES * h->D));
    if (h->tickets) SFFN_CUDA(cudaMemset(h->tickets, 0, sizeof(int) * kTicketInts));
    if (h->tacc) SFFN_CUDA(cudaMemset(h->tacc, 0, sizeof(float) * 128 * h->r));  // the t kernel's partial sums
    if (err & DEV_ERR_CHECK)
      return fail(SFFN_ERR_DEVICE, "a device-side bounds or alignment check failed (error word 0x%x); outputs "
                  "of the affected forward are invalid", err);
    return fail(SFFN_ERR_TIMEOUT, "a device-side wait ran out of time (error word 0x%x); outputs of "
                "the affected forward are invalid", err);
  }
  return SFFN_OK;
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
  return pa < pb + nb && pb < pa + na;
}

}  // namespace

extern "C" {

int sffn_version(void) { return 100; }

const char* sffn_last_error(void) { return g_msg; }

const char* sffn_strerror(int code) {
  switch (code) {
    case SFFN_OK: return "success";
    case SFFN_ERR_ARG: return "invalid argument";
    case SFFN_ERR_ALIGN: return "pointer not 16-byte aligned";
    case SFFN_ERR_DTYPE: return "unsupported dtype or shape";
    case SFFN_ERR_CUDA: return "CUDA runtime error";
    case SFFN_ERR_TIMEOUT: return "device-side wait timed out";
    case SFFN_ERR_STATE: return "call out of order";
    case SFFN_ERR_NOMEM: return "device memory allocation failed";
    case SFFN_ERR_DEVICE: return "device-side bounds or alignment check failed";
    default: return "unknown status";
  }
}

namespace {
// scales per row of W1 and of W3 on a quantised handle: one (int8), one per 64 columns (int4)
size_t qscale_per_row(const sffn_s* h) { return h->qbits == 4 ? (size_t)h->D / INT4_GROUP : 1; }
}  // namespace

sffn_t sffn_create(int D, int H, int r, int act, int dtype) { return sffn_create_ex(D, H, r, act, dtype, 0); }

sffn_t sffn_create_ex(int D, int H, int r, int act, int dtype, int flags) {
  g_msg[0] = 0;
  static_assert(SFFN_GATE_TILED_G == FLAG_TILED_G && SFFN_GATE_RMSNORM == FLAG_RMSNORM &&
                    SFFN_DOUBLE_ACT == FLAG_DOUBLE_ACT,
                "option bits of the ABI and of the kernels agree");
  static_assert(SFFN_DETERMINISTIC == FLAG_DETERMINISTIC, "option bits of the ABI and of the kernels agree");
  if (flags & ~(SFFN_GATE_TILED_G | SFFN_GATE_RMSNORM | SFFN_DOUBLE_ACT | SFFN_DETERMINISTIC)) {
    fail(SFFN_ERR_ARG, "flags 0x%x has unknown bits", flags);
    return nullptr;
  }
  if ((flags & (SFFN_GATE_TILED_G | SFFN_GATE_RMSNORM)) && r == 0) {
    fail(SFFN_ERR_ARG, "the tiled identity and RMSNorm options belong to the low-rank gate (r > 0)");
    return nullptr;
  }
  if (dtype != SFFN_F32 && dtype != SFFN_BF16 && dtype != SFFN_I8W && dtype != SFFN_I4W) {
    fail(SFFN_ERR_ARG, "dtype %d unknown", dtype);
    return nullptr;
  }
  if (dtype == SFFN_I8W && (r % 16 != 0 || D % 16 != 0 || (flags & ~SFFN_DOUBLE_ACT))) {
    fail(SFFN_ERR_DTYPE, "int8 weights need D %% 16 == 0, r %% 16 == 0 and no option but the double activation");
    return nullptr;
  }
  if (dtype == SFFN_I4W && (r != 0 || D % INT4_GROUP != 0 || (flags & ~SFFN_DOUBLE_ACT))) {
    fail(SFFN_ERR_DTYPE, "int4 weights need the standard gate (r = 0), D %% 64 == 0 and no low-rank option");
    return nullptr;
  }
  if ((flags & SFFN_DETERMINISTIC) && dtype != SFFN_BF16) {
    fail(SFFN_ERR_DTYPE, "the deterministic option is available for bf16 handles");
    return nullptr;
  }
  if (act != SFFN_ACT_RELU && act != SFFN_ACT_RSP && act != SFFN_ACT_SILU) {
    fail(SFFN_ERR_ARG, "act %d unknown", act);
    return nullptr;
  }
  const int dmax = dtype == SFFN_F32 ? SFFN_MAX_D_F32 : SFFN_MAX_D_BF16;
  if (D < 8 || D % 8 != 0 || D > dmax) { fail(SFFN_ERR_ARG, "D=%d must be a multiple of 8 in [8, %d]", D, dmax); return nullptr; }
  if (H < 1) { fail(SFFN_ERR_ARG, "H=%d must be >= 1", H); return nullptr; }
  if (r < 0 || r % 8 != 0 || r > D) { fail(SFFN_ERR_ARG, "r=%d must be 0 or a multiple of 8 <= D", r); return nullptr; }

  sffn_s* h = new (std::nothrow) sffn_s;
  if (!h) { fail(SFFN_ERR_NOMEM, "host allocation failed"); return nullptr; }
  h->D = D; h->H = H; h->r = r; h->act = act; h->dtype = dtype; h->flags = flags;
  h->elt = dtype == SFFN_F32 ? 4 : 2;
  h->qbits = dtype == SFFN_I8W ? 8 : dtype == SFFN_I4W ? 4 : 0;
  h->welt = h->qbits ? 1 : h->elt;

  auto bail = [&](int code, const char* what, cudaError_t e) -> sffn_t {
    fail(code, "%s: %s", what, cudaGetErrorString(e));
    release(h);
    delete h;
    return nullptr;
  };
  cudaError_t e;
  if ((e = cudaGetDevice(&h->device))) return bail(SFFN_ERR_CUDA, "cudaGetDevice", e);
  if ((e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device)))
    return bail(SFFN_ERR_CUDA, "cudaDeviceGetAttribute", e);
  int optin = 0;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device)))
    return bail(SFFN_ERR_CUDA, "cudaDeviceGetAttribute", e);
  h->max_smem = (size_t)optin;

  const size_t welt = h->welt;
  const size_t gk = (size_t)gate_k(h);
  const bool i8 = h->qbits != 0;  // int8 or int4 codes with per-channel scales
  struct { void** p; size_t bytes; } allocs[] = {
      {&h->gate_w, (size_t)H * gk * welt},
      {&h->V, (size_t)std::max(r, 1) * D * welt},
      {&h->W3, (size_t)H * D * welt},
      {&h->W2t, (size_t)H * D * welt},
      {(void**)&h->qs1, i8 ? sizeof(float) * H * qscale_per_row(h) : 16},
      {(void**)&h->qs3, i8 ? sizeof(float) * H * qscale_per_row(h) : 16},
      {(void**)&h->qs2, i8 ? sizeof(float) * D : 16},
      {(void**)&h->qsv, i8 && r > 0 ? sizeof(float) * r : 16},
      {(void**)&h->yacc, sizeof(float) * SFFN_MAX_BATCH * YACC_COPIES * D},
      {(void**)&h->tbuf, sizeof(float) * SFFN_MAX_BATCH * std::max(r, 8)},
      {(void**)&h->ctrl, sizeof(int) * CTRL_INTS},
      {(void**)&h->counts, sizeof(int) * SFFN_MAX_BATCH},
      {(void**)&h->mask, (size_t)SFFN_MAX_BATCH * H},
  };
  for (auto& a : allocs) {
    if ((e = cudaMalloc(a.p, a.bytes))) return bail(SFFN_ERR_NOMEM, "cudaMalloc", e);
  }
  if ((e = cudaMemset(h->yacc, 0, sizeof(float) * SFFN_MAX_BATCH * YACC_COPIES * D)) ||
      (e = cudaMemset(h->ctrl, 0, sizeof(int) * CTRL_INTS)) ||
      (e = cudaMemset(h->counts, 0, sizeof(int) * SFFN_MAX_BATCH)) ||
      (e = cudaMemset(h->mask, 0, (size_t)SFFN_MAX_BATCH * H)))
    return bail(SFFN_ERR_CUDA, "cudaMemset", e);
  if ((e = cudaEventCreateWithFlags(&h->ev, cudaEventDisableTiming)))
    return bail(SFFN_ERR_CUDA, "cudaEventCreate", e);
  {
    // blocks per SM of the streaming kernel (1 leaves room for the next call's blocks)
    int mult = 1;
    if (const char* env = std::getenv("SFFN_STREAM_BLOCKS_PER_SM")) mult = std::max(1, std::min(4, std::atoi(env)));
    h->stream_grid = std::min(h->num_sms * mult, H);
    h->stream_rows_cap = (H + h->stream_grid - 1) / h->stream_grid;
    if (const char* env = std::getenv("SFFN_B1_KERNEL")) h->b1_bf16 = std::strcmp(env, "stream") != 0;
    if (dtype == SFFN_BF16) {
      const int g = std::min(h->num_sms, H), cap = (H + g - 1) / g;
      h->bf16_plan = plan_ffn_b1_bf16(D, gate_k(h), r > 0, cap);
      if ((e = ffn_b1_bf16_prepare(h->max_smem))) return bail(SFFN_ERR_CUDA, "cudaFuncSetAttribute", e);
      if (flags & SFFN_DETERMINISTIC) {
        if (cap > ffn_b1_bf16_threads()) {
          fail(SFFN_ERR_DTYPE, "the deterministic option needs at most %d units per block (H <= %d)",
               ffn_b1_bf16_threads(), ffn_b1_bf16_threads() * g);
          release(h);
          delete h;
          return nullptr;
        }
        if ((e = cudaMalloc(&h->ypart, sizeof(float) * (size_t)g * D))) return bail(SFFN_ERR_NOMEM, "cudaMalloc", e);
      }
    }
    h->stream_plan = plan_ffn_b1_stream(D, gate_k(h), h->elt, r > 0, h->stream_rows_cap);
    if (h->stream_plan.smem > h->max_smem) {
      fail(SFFN_ERR_DTYPE, "shared-memory plan of the streaming kernel exceeds the device limit");
      char keep[sizeof g_msg];
      std::memcpy(keep, g_msg, sizeof keep);
      release(h);
      delete h;
      std::memcpy(g_msg, keep, sizeof keep);
      return nullptr;
    }
    h->batch_plan = plan_ffn_batch(D, gate_k(h), h->elt, r > 0, h->stream_rows_cap, 8);
    if (h->batch_plan.smem > h->max_smem) {
      fail(SFFN_ERR_DTYPE, "shared-memory plan of the batched kernel exceeds the device limit");
      char keep[sizeof g_msg];
      std::memcpy(keep, g_msg, sizeof keep);
      release(h);
      delete h;
      std::memcpy(g_msg, keep, sizeof keep);
      return nullptr;
    }
    if ((e = ffn_batch_prepare(h->max_smem))) return bail(SFFN_ERR_CUDA, "cudaFuncSetAttribute", e);
    if (i8) {
      h->i8_plan = plan_ffn_b1_i8(D, (int)gate_k(h), h->stream_rows_cap, h->qbits, r > 0);
      if (h->i8_plan.smem > h->max_smem) {
        fail(SFFN_ERR_DTYPE, "shared-memory plan of the int8 / int4 kernel exceeds the device limit");
        char keep[sizeof g_msg];
        std::memcpy(keep, g_msg, sizeof keep);
        release(h);
        delete h;
        std::memcpy(g_msg, keep, sizeof keep);
        return nullptr;
      }
      if ((e = ffn_b1_i8_prepare(h->max_smem))) return bail(SFFN_ERR_CUDA, "cudaFuncSetAttribute", e);
    }
    if (r > 0 && (e = lopa_t_prepare())) return bail(SFFN_ERR_CUDA, "cudaFuncSetAttribute", e);
    if ((e = ffn_b1_stream_prepare(h->max_smem)))
      return bail(SFFN_ERR_CUDA, "cudaFuncSetAttribute", e);
  }
  if (dtype == SFFN_BF16) {
    h->tc = plan_ffn_tc(D, H, r, h->num_sms);
    if (h->tc.ok && r > 0) {
      h->tcu_max_batch = 0;  // the union-gather kernel computes a standard gate only
      if ((e = cudaMalloc(&h->tpair, sizeof(uint16_t) * 256 * r)) || (e = cudaMalloc(&h->tacc, sizeof(float) * 128 * r)))
        return bail(SFFN_ERR_NOMEM, "cudaMalloc", e);
      if ((e = cudaMemset(h->tpair, 0, sizeof(uint16_t) * 256 * r)) || (e = cudaMemset(h->tacc, 0, sizeof(float) * 128 * r)))
        return bail(SFFN_ERR_CUDA, "cudaMemset", e);
    }
    if (h->tc.ok) {
      if ((e = cudaMalloc(&h->hbuf, sizeof(uint16_t) * ffn_tc_hbuf_elems(h->tc))) ||
          (e = cudaMalloc(&h->tickets, sizeof(int) * kTicketInts)) ||
          (e = cudaMalloc(&h->ulist, sizeof(int) * (size_t)H)))
        return bail(SFFN_ERR_NOMEM, "cudaMalloc", e);
      if ((e = cudaMemset(h->tickets, 0, sizeof(int) * kTicketInts))) return bail(SFFN_ERR_CUDA, "cudaMemset", e);
      if (const char* env = std::getenv("SFFN_TC_GATE_KB")) h->tc.gate_smem_budget = (size_t)std::atoi(env) * 1024;
      if (const char* env = std::getenv("SFFN_TC_DOWN_KB")) h->tc.down_smem_budget = (size_t)std::atoi(env) * 1024;
      if (const char* env = std::getenv("SFFN_TC_GATE_CHUNKS")) h->tc.gate_chunks = std::max(1, std::min(4, std::atoi(env)));
      if ((e = cudaMemset(h->hbuf, 0, sizeof(uint16_t) * ffn_tc_hbuf_elems(h->tc))))
        return bail(SFFN_ERR_CUDA, "cudaMemset", e);
      if ((e = ffn_tc_prepare(h->max_smem))) return bail(SFFN_ERR_CUDA, "cudaFuncSetAttribute", e);
      if ((e = ffn_tc_plan_cluster(h->tc, h->max_smem))) return bail(SFFN_ERR_CUDA, "cudaOccupancyMaxActiveClusters", e);
      if ((e = ffn_tcu_prepare(h->max_smem))) return bail(SFFN_ERR_CUDA, "cudaFuncSetAttribute", e);
      if ((e = ffn_tcg_prepare(h->max_smem))) return bail(SFFN_ERR_CUDA, "cudaFuncSetAttribute", e);
      if ((e = ffn_tcg_plan_cluster(h->tc, h->max_smem)))
        return bail(SFFN_ERR_CUDA, "cudaOccupancyMaxActiveClusters", e);
      if (const char* env = std::getenv("SFFN_TC_DOWN_CLUSTER"))
        if (std::atoi(env) == 0) h->tc.down_cluster = h->tc.tcg_down_cluster = 0;
      if (const char* env = std::getenv("SFFN_TC_T_CLUSTER"))
        if (std::atoi(env) == 0) h->tc.t_cluster = 0;
      if (const char* env = std::getenv("SFFN_TCG_ACC")) h->tc.tcg_acc = std::max(1, std::min(4, std::atoi(env)));
      if (const char* env = std::getenv("SFFN_TCG_MAX_BATCH"))
        h->tcg_force = std::max(0, std::min(TCG_MAX_BATCH, std::atoi(env)));
      if (const char* env = std::getenv("SFFN_TCU_MAX_BATCH"))
        if (r == 0) h->tcu_max_batch = std::max(0, std::min(8, std::atoi(env)));
      if (const char* env = std::getenv("SFFN_TC_MIN_BATCH")) h->tc_min_batch = std::max(1, std::atoi(env));
      if (const char* env = std::getenv("SFFN_TC_T_CUDA_MAX_B")) h->tc_t_cuda_max = std::max(0, std::atoi(env));
      if (const char* env = std::getenv("SFFN_TC_T_SPLIT_TOKENS")) h->tc.t_split_tokens = std::max(16, std::atoi(env));
    }
  }
  if ((e = cudaDeviceSynchronize())) return bail(SFFN_ERR_CUDA, "cudaDeviceSynchronize", e);
  return h;
}

int sffn_set_weights(sffn_t h, const void* W1_or_U, const void* V, const void* W3, const void* W2,
                     void* stream) {
  if (!h) return fail(SFFN_ERR_ARG, "null handle");
  if (!W1_or_U || !W3 || !W2 || (h->r > 0 && !V)) return fail(SFFN_ERR_ARG, "null weight pointer");
  if (int rc = check_device(h)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (h->qbits) {
    // bf16 weights in, per-output-channel codes and scales out (W2's codes transposed); int4
    // codes are decided one per byte, then packed two per byte
    const size_t D = h->D, H = h->H;
    const bool i4 = h->qbits == 4;
    const int qmax = i4 ? 7 : 127;
    void* stage = nullptr;
    int8_t *q2 = nullptr, *codes = nullptr;
    int* perr = nullptr;
    SFFN_CUDA(cudaMalloc(&stage, D * H * 2));
    cudaError_t e = cudaMalloc(&q2, D * H);
    if (!e && i4) e = cudaMalloc(&codes, D * H);
    if (!e && i4) e = cudaMalloc(&perr, sizeof(int));
    if (!e && i4) e = cudaMemsetAsync(perr, 0, sizeof(int), s);
    auto store = [&](void* dst, const int8_t* src) {  // int4: pack the one-per-byte codes
      return i4 ? launch_pack_int4(src, dst, H * D, perr, s) : cudaSuccess;
    };
    // W1 (or U [H, r]) and W3: int8 one scale per row, int4 one per group of 64 columns
    const size_t gk = gate_k(h);
    auto quant_rows = [&](int8_t* dst, float* sc, size_t cols) {
      return i4 ? launch_quantize_groups4(stage, dst, sc, (int)H, (int)cols, s)
                : launch_quantize_rows(stage, dst, sc, (int)H, (int)cols, s, qmax);
    };
    int8_t* c1 = i4 ? codes : static_cast<int8_t*>(h->gate_w);
    if (!e) e = cudaMemcpyAsync(stage, W1_or_U, H * gk * 2, cudaMemcpyDefault, s);
    if (!e) e = quant_rows(c1, h->qs1, gk);
    if (!e) e = store(h->gate_w, c1);
    if (!e && h->r > 0) {  // the low-rank gate's V [r, D] (int8 only): one scale per row
      e = cudaMemcpyAsync(stage, V, (size_t)h->r * D * 2, cudaMemcpyDefault, s);
      if (!e) e = launch_quantize_rows(stage, static_cast<int8_t*>(h->V), h->qsv, h->r, (int)D, s, 127);
    }
    int8_t* c3 = i4 ? codes : static_cast<int8_t*>(h->W3);
    if (!e) e = cudaMemcpyAsync(stage, W3, H * D * 2, cudaMemcpyDefault, s);
    if (!e) e = quant_rows(c3, h->qs3, D);
    if (!e) e = store(h->W3, c3);
    if (!e) e = cudaMemcpyAsync(stage, W2, D * H * 2, cudaMemcpyDefault, s);
    if (!e) e = launch_quantize_rows(stage, q2, h->qs2, (int)D, (int)H, s, qmax);
    if (!e) e = launch_transpose(q2, i4 ? static_cast<void*>(codes) : h->W2t, (int)D, (int)H, 1, s);
    if (!e) e = store(h->W2t, codes);
    if (!e) e = cudaStreamSynchronize(s);
    cudaFree(stage);
    cudaFree(q2);
    cudaFree(codes);
    cudaFree(perr);
    if (e) return fail(SFFN_ERR_CUDA, "weight quantisation failed: %s", cudaGetErrorString(e));
    h->weights_set = true;
    return SFFN_OK;
  }
  const size_t elt = h->elt, D = h->D, H = h->H, gk = gate_k(h);
  SFFN_CUDA(cudaMemcpyAsync(h->gate_w, W1_or_U, H * gk * elt, cudaMemcpyDefault, s));
  if (h->r > 0) SFFN_CUDA(cudaMemcpyAsync(h->V, V, (size_t)h->r * D * elt, cudaMemcpyDefault, s));
  SFFN_CUDA(cudaMemcpyAsync(h->W3, W3, H * D * elt, cudaMemcpyDefault, s));
  void* stage = nullptr;
  SFFN_CUDA(cudaMalloc(&stage, D * H * elt));
  cudaError_t e = cudaMemcpyAsync(stage, W2, D * H * elt, cudaMemcpyDefault, s);
  if (!e) e = launch_transpose(stage, h->W2t, (int)D, (int)H, (int)elt, s);
  if (!e) e = cudaStreamSynchronize(s);
  cudaFree(stage);
  if (e) return fail(SFFN_ERR_CUDA, "weight upload failed: %s", cudaGetErrorString(e));
  if (h->tc.ok) {
    if (int rc = encode_tc_maps(&h->tcm, h->tc, h->gate_w, h->V, h->W3, h->W2t, h->hbuf, h->D, h->H))
      return fail(SFFN_ERR_CUDA, "tensor-map encoding of the weights failed (status %d)", rc);
    h->tc_ready = true;
  }
  h->weights_set = true;
  return SFFN_OK;
}

int sffn_set_weights_int8(sffn_t h, const int8_t* W1q, const float* s1, const int8_t* W3q, const float* s3,
                          const int8_t* W2q, const float* s2, void* stream) {
  if (!h) return fail(SFFN_ERR_ARG, "null handle");
  if (!h->qbits) return fail(SFFN_ERR_STATE, "the handle does not hold int8 or int4 weights");
  if (h->r > 0)
    return fail(SFFN_ERR_STATE, "a low-rank int8 handle takes bf16 weights through sffn_set_weights");
  if (!W1q || !s1 || !W3q || !s3 || !W2q || !s2) return fail(SFFN_ERR_ARG, "null weight pointer");
  if (int rc = check_device(h)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t D = h->D, H = h->H;
  const bool i4 = h->qbits == 4;
  int8_t *q2 = nullptr, *codes = nullptr;
  int* perr = nullptr;
  SFFN_CUDA(cudaMalloc(&q2, D * H));
  cudaError_t e = i4 ? cudaMalloc(&codes, D * H) : cudaSuccess;
  if (!e && i4) e = cudaMalloc(&perr, sizeof(int));
  if (!e && i4) e = cudaMemsetAsync(perr, 0, sizeof(int), s);
  // int4: each array goes through `codes` and is packed two per byte, codes outside [-7, 7] flagged
  auto put = [&](void* dst, const int8_t* src) {
    if (!i4) return cudaMemcpyAsync(dst, src, H * D, cudaMemcpyDefault, s);
    cudaError_t r = cudaMemcpyAsync(codes, src, H * D, cudaMemcpyDefault, s);
    return r ? r : launch_pack_int4(codes, dst, H * D, perr, s);
  };
  const size_t nsc = H * qscale_per_row(h);
  if (!e) e = put(h->gate_w, W1q);
  if (!e) e = put(h->W3, W3q);
  if (!e) e = cudaMemcpyAsync(h->qs1, s1, sizeof(float) * nsc, cudaMemcpyDefault, s);
  if (!e) e = cudaMemcpyAsync(h->qs3, s3, sizeof(float) * nsc, cudaMemcpyDefault, s);
  if (!e) e = cudaMemcpyAsync(h->qs2, s2, sizeof(float) * D, cudaMemcpyDefault, s);
  if (!e) e = cudaMemcpyAsync(q2, W2q, D * H, cudaMemcpyDefault, s);
  if (!e) e = launch_transpose(q2, i4 ? static_cast<void*>(codes) : h->W2t, (int)D, (int)H, 1, s);
  if (!e && i4) e = launch_pack_int4(codes, h->W2t, H * D, perr, s);
  int bad = 0;
  if (!e && i4) e = cudaMemcpyAsync(&bad, perr, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (!e) e = cudaStreamSynchronize(s);
  cudaFree(q2);
  cudaFree(codes);
  cudaFree(perr);
  if (e) return fail(SFFN_ERR_CUDA, "int8 / int4 weight upload failed: %s", cudaGetErrorString(e));
  if (bad) {
    h->weights_set = false;
    return fail(SFFN_ERR_ARG, "int4 codes must lie in [-7, 7]");
  }
  h->weights_set = true;
  return SFFN_OK;
}

int sffn_get_weights_int8(sffn_t h, int8_t* W1q, float* s1, int8_t* W3q, float* s3, int8_t* W2q, float* s2,
                          void* stream) {
  if (!h) return fail(SFFN_ERR_ARG, "null handle");
  if (!h->qbits) return fail(SFFN_ERR_STATE, "the handle does not hold int8 or int4 weights");
  if (!h->weights_set) return fail(SFFN_ERR_STATE, "no weights have been set");
  if (int rc = check_device(h)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t D = h->D, H = h->H;
  const bool i4 = h->qbits == 4;
  cudaError_t e = cudaSuccess;
  int8_t *q2 = nullptr, *codes = nullptr;
  if (i4) e = cudaMalloc(&codes, D * H);
  // int4: unpacked to one code per byte on the way out
  auto get = [&](int8_t* dst, const void* src, size_t cols) {
    if (!i4) return cudaMemcpyAsync(dst, src, H * cols, cudaMemcpyDefault, s);
    cudaError_t r = launch_unpack_int4(src, codes, H * cols, s);
    return r ? r : cudaMemcpyAsync(dst, codes, H * cols, cudaMemcpyDefault, s);
  };
  if (!e && W1q) e = get(W1q, h->gate_w, (size_t)gate_k(h));  // the low-rank gate: U's codes [H, r]
  if (!e && W3q) e = get(W3q, h->W3, D);
  if (!e && s1) e = cudaMemcpyAsync(s1, h->qs1, sizeof(float) * H * qscale_per_row(h), cudaMemcpyDefault, s);
  if (!e && s3) e = cudaMemcpyAsync(s3, h->qs3, sizeof(float) * H * qscale_per_row(h), cudaMemcpyDefault, s);
  if (!e && s2) e = cudaMemcpyAsync(s2, h->qs2, sizeof(float) * D, cudaMemcpyDefault, s);
  if (!e && W2q) {
    e = cudaMalloc(&q2, D * H);
    if (!e && i4) e = launch_unpack_int4(h->W2t, codes, H * D, s);
    if (!e) e = launch_transpose(i4 ? static_cast<const void*>(codes) : h->W2t, q2, (int)H, (int)D, 1, s);
    if (!e) e = cudaMemcpyAsync(W2q, q2, D * H, cudaMemcpyDefault, s);
  }
  if (!e) e = cudaStreamSynchronize(s);
  cudaFree(q2);
  cudaFree(codes);
  if (e) return fail(SFFN_ERR_CUDA, "int8 weight download failed: %s", cudaGetErrorString(e));
  return SFFN_OK;
}

namespace {
// Batches of 3..16 tokens (bf16) read only the union of the live sets when that pays: the expected
// union u = 1 - (1 - rho)^B is at most 30 % of the units and the W3 and W2 bytes of the other units
// come to at least 128 MB (standard gate) or 64 MB (low-rank gate, whose streaming form pays a t kernel
// and whose union form streams only U before the union is known).  Below that the streaming kernels win
// on this GPU: they stream every slice at close to the copy bandwidth, while the union's scattered rows
// arrive at a fraction of it and the gate must finish before they can be requested.
bool use_union_skip(const sffn_s* h, int B) {
  if (B > TCG_MAX_BATCH) return false;
  if (h->tcg_force >= 0) return B <= h->tcg_force;
  if (h->live_frac < 0.f || B > 16) return false;
  const double u = 1.0 - std::pow(1.0 - (double)h->live_frac, B);
  const double saved = (1.0 - u) * 2.0 * 2.0 * (double)h->H * (double)h->D;
  return u <= 0.30 && saved >= (h->r > 0 ? 64e6 : 128e6);
}
}  // namespace

int sffn_forward(sffn_t h, const void* x, void* y, int B, void* stream) {
  if (!h) return fail(SFFN_ERR_ARG, "null handle");
  if (!x || !y) return fail(SFFN_ERR_ARG, "null x or y");
  if (B < 1 || B > SFFN_MAX_BATCH) return fail(SFFN_ERR_ARG, "B=%d outside [1, %d]", B, SFFN_MAX_BATCH);
  if (((uintptr_t)x & 15) || ((uintptr_t)y & 15)) return fail(SFFN_ERR_ALIGN, "x and y must be 16-byte aligned");
  const size_t xbytes = (size_t)B * h->D * h->elt;
  if (ranges_overlap(x, xbytes, y, xbytes)) return fail(SFFN_ERR_ARG, "x and y overlap");
  if (!h->weights_set) return fail(SFFN_ERR_STATE, "sffn_set_weights has not been called");
  if (int rc = check_device(h)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool lopa = h->r > 0;
  const size_t row = (size_t)h->D * h->elt;

  const bool det = (h->flags & FLAG_DETERMINISTIC) != 0;  // one single-token pass per token, ordered sums
  // batches on the tensor cores (the low-rank gate's RMSNorm needs all of t first: CUDA-core path)
  const bool tc_batch = !det && h->tc_ready && B >= h->tc_min_batch && !(lopa && (h->flags & FLAG_RMSNORM));
  const bool tcu = tc_batch && !lopa && B <= h->tcu_max_batch;
  const bool tcg = tc_batch && !tcu && B >= 3 && use_union_skip(h, B);
  if (tcg) {
    // small batch, union skip: gate kernel (W1 or U t, then the union's W3 rows), down kernel (the union's W2
    // columns); the low-rank gate's t pair first
    TcBuffers buf{h->hbuf, h->yacc, h->ctrl, h->mask, h->counts, h->tickets, h->tpair, h->tacc,
                  h->tickets + TC_TICKETS};
    TcgBuffers ub{h->ulist, h->tickets + 2 * TC_TICKETS, h->tickets + 2 * TC_TICKETS + 1};
    cudaError_t ce = cudaSuccess;
    if (lopa) {
      if (B <= h->tc_t_cuda_max) {
        SFFN_CUDA(launch_lopa_t_pair(h->V, x, h->tpair, h->r, h->D, B, (B + 15) / 16 * 16, s));
      } else {
        if (int rc = launch_ffn_tc(h->tc, h->tcm, buf, x, y, h->D, h->H, B, h->act, h->flags, h->thr, kTimeoutNs,
                                   h->max_smem, s, &ce, false, true))
          return fail(SFFN_ERR_CUDA, "tensor-map encoding of x failed (status %d)", rc);
        SFFN_CUDA(ce);
      }
    }
    if (int rc = launch_ffn_tcg(h->tc, h->tcm, buf, ub, h->W3, h->W2t, x, y, h->D, h->H, B, h->act, h->flags, h->thr,
                                kTimeoutNs, h->max_smem, s, &ce))
      return fail(SFFN_ERR_CUDA, "tensor-map encoding of x failed (status %d)", rc);
    SFFN_CUDA(ce);
  } else if (tcu) {
    // small batch: the gate on the tensor cores, the union of the live sets gathered, then finalize
    cudaError_t ce = cudaSuccess;
    if (int rc = launch_ffn_tcu(h->tc, h->tcm, h->W3, h->W2t, h->yacc, h->ctrl, h->mask, x, h->D, h->H, B, h->act,
                                h->flags, h->thr, kTimeoutNs, h->max_smem, s, &ce))
      return fail(SFFN_ERR_CUDA, "tensor-map encoding of x failed (status %d)", rc);
    SFFN_CUDA(ce);
    SFFN_CUDA(launch_finalize(h->yacc, y, h->ctrl, h->counts, 0, h->D, B, h->dtype, s));
  } else if (tc_batch) {
    // whole batch on the tensor cores: (t kernel,) gate-up kernel, down kernel
    const bool t_cuda_cores = lopa && B <= h->tc_t_cuda_max;
    if (t_cuda_cores) SFFN_CUDA(launch_lopa_t_pair(h->V, x, h->tpair, h->r, h->D, B, (B + 15) / 16 * 16, s));
    TcBuffers buf{h->hbuf, h->yacc, h->ctrl, h->mask, h->counts, h->tickets, h->tpair, h->tacc,
                  h->tickets + TC_TICKETS};
    cudaError_t ce = cudaSuccess;
    if (int rc = launch_ffn_tc(h->tc, h->tcm, buf, x, y, h->D, h->H, B, h->act, h->flags, h->thr, kTimeoutNs,
                               h->max_smem, s, &ce, t_cuda_cores))
      return fail(SFFN_ERR_CUDA, "tensor-map encoding of x failed (status %d)", rc);
    SFFN_CUDA(ce);
  }
  if (h->qbits) {
    // weight-only int8 / int4: one streaming pass per token (the low-rank gate's t kernel first)
    for (int b = 0; b < B; ++b) {
      B1Params p;
      if (lopa) {
        float* tb = h->tbuf + (size_t)b * h->r;
        SFFN_CUDA(launch_lopa_t_i8(h->V, h->qsv, static_cast<const uint8_t*>(x) + b * row, tb, h->r, h->D, s));
        p.t = tb;
      }
      p.gate_w = h->gate_w;
      p.W3 = h->W3;
      p.W2t = h->W2t;
      p.x = static_cast<const uint8_t*>(x) + b * row;
      p.y = static_cast<uint8_t*>(y) + b * row;
      p.yacc = h->yacc;
      p.ctrl = h->ctrl;
      p.counts = h->counts + b;
      p.mask = h->mask + (size_t)b * h->H;
      p.D = h->D;
      p.H = h->H;
      p.gate_k = gate_k(h);
      p.act = h->act;
      p.count_slot = b;
      p.rows_cap = h->stream_rows_cap;
      p.pref_rows = h->i8_plan.pref_rows;
      p.gather_rows = h->i8_plan.gather_rows;
      p.flags = h->flags;
      p.thr = h->thr;
      p.s1 = h->qs1;
      p.s3 = h->qs3;
      p.s2 = h->qs2;
      SFFN_CUDA(launch_ffn_b1_i8(p, h->stream_grid, h->i8_plan.smem, s, h->qbits));
      SFFN_CUDA(launch_finalize(h->yacc, p.y, h->ctrl, p.counts, b, h->D, 1, SFFN_BF16, s));
    }
  }
  if (lopa && !tc_batch && !h->qbits) SFFN_CUDA(launch_lopa_t(h->V, x, h->tbuf, h->r, h->D, B, h->dtype, s));
  // tokens in groups of up to 8: one pass over the weights per group
  for (int b = 0; b < B && !h->qbits && !tc_batch;) {
    const int nb = det ? 1 : std::min(8, B - b);
    B1Params p;
    p.gate_w = h->gate_w;
    p.W3 = h->W3;
    p.W2t = h->W2t;
    p.x = static_cast<const uint8_t*>(x) + b * row;
    p.t = lopa ? h->tbuf + (size_t)b * h->r : nullptr;
    p.y = static_cast<uint8_t*>(y) + b * row;
    p.yacc = h->yacc;
    p.ctrl = h->ctrl;
    p.counts = h->counts + b;
    p.mask = h->mask + (size_t)b * h->H;
    p.D = h->D;
    p.H = h->H;
    p.gate_k = gate_k(h);
    p.act = h->act;
    p.count_slot = b;
    p.rows_cap = h->stream_rows_cap;
    p.flags = h->flags & ~FLAG_DETERMINISTIC;
    p.thr = h->thr;
    if (nb == 1) {
      if (h->dtype == SFFN_BF16 && (h->b1_bf16 || det)) {  // (the partial-row output is this kernel's)
        const int grid = std::min(h->num_sms, h->H);
        p.rows_cap = (h->H + grid - 1) / grid;
        p.pref_rows = h->bf16_plan.pref_rows;
        p.ypart = h->ypart;  // null unless deterministic
        SFFN_CUDA(launch_ffn_b1_bf16(p, lopa, grid, h->bf16_plan.smem, s));
      } else {
        p.pref_rows = h->stream_plan.pref_rows;
        p.gather_rows = h->stream_plan.gather_rows;
        SFFN_CUDA(launch_ffn_b1_stream(p, h->dtype, lopa, h->stream_grid, h->stream_plan.smem, s));
      }
    } else {
      p.pref_rows = h->batch_plan.pref_rows;
      p.gather_rows = h->batch_plan.gather_rows;
      SFFN_CUDA(launch_ffn_batch(p, nb, h->dtype, lopa, h->stream_grid, h->batch_plan.smem, s));
    }
    if (det)
      SFFN_CUDA(launch_finalize_ordered(h->ypart, std::min(h->num_sms, h->H), p.y, h->ctrl, p.counts, b, h->D, s));
    else
      SFFN_CUDA(launch_finalize(h->yacc, p.y, h->ctrl, p.counts, b, h->D, nb, h->dtype, s));
    b += nb;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  SFFN_CUDA(cudaStreamIsCapturing(s, &cs));
  if (cs == cudaStreamCaptureStatusNone) {
    SFFN_CUDA(cudaEventRecord(h->ev, s));
    h->ev_valid = true;
  } else {
    h->ev_valid = false;  // inside a capture: readers fall back to a device-wide sync
  }
  h->last_B = B;
  return SFFN_OK;
}

int sffn_active_counts(sffn_t h, int* counts_host, int B) {
  if (!h || !counts_host) return fail(SFFN_ERR_ARG, "null argument");
  if (h->last_B == 0) return fail(SFFN_ERR_STATE, "no forward has run on this handle");
  if (B != h->last_B) return fail(SFFN_ERR_ARG, "B=%d but the last forward had B=%d", B, h->last_B);
  if (int rc = sync_and_check(h)) return rc;
  SFFN_CUDA(cudaMemcpy(counts_host, h->counts, sizeof(int) * B, cudaMemcpyDeviceToHost));
  double sum = 0;
  for (int b = 0; b < B; ++b) sum += counts_host[b];
  h->live_frac = (float)(sum / ((double)B * h->H));  // the batch-path choice follows the observed sparsity
  return SFFN_OK;
}

int sffn_set_live_fraction_hint(sffn_t h, float rho) {
  if (!h) return fail(SFFN_ERR_ARG, "null handle");
  if (!(rho <= 1.f) || rho != rho) return fail(SFFN_ERR_ARG, "live fraction %g must be <= 1", (double)rho);
  h->live_frac = rho < 0.f ? -1.f : rho;
  return SFFN_OK;
}

int sffn_active_mask(sffn_t h, uint8_t* mask_host, int B) {
  if (!h || !mask_host) return fail(SFFN_ERR_ARG, "null argument");
  if (h->last_B == 0) return fail(SFFN_ERR_STATE, "no forward has run on this handle");
  if (B != h->last_B) return fail(SFFN_ERR_ARG, "B=%d but the last forward had B=%d", B, h->last_B);
  if (int rc = sync_and_check(h)) return rc;
  SFFN_CUDA(cudaMemcpy(mask_host, h->mask, (size_t)B * h->H, cudaMemcpyDeviceToHost));
  return SFFN_OK;
}

int sffn_set_live_threshold(sffn_t h, float thr) {
  if (!h) return fail(SFFN_ERR_ARG, "null handle");
  if (!(thr >= 0.f) || thr > 3.0e38f) return fail(SFFN_ERR_ARG, "threshold %g must be finite and >= 0", (double)thr);
  h->thr = thr;
  return SFFN_OK;
}

int sffn_synchronize(sffn_t h) {
  if (!h) return fail(SFFN_ERR_ARG, "null handle");
  return sync_and_check(h);
}

int sffn_debug_timeout_probe(sffn_t h, int limit_us, void* stream) {
  if (!h) return fail(SFFN_ERR_ARG, "null handle");
  if (limit_us < 1 || limit_us > 1000000) return fail(SFFN_ERR_ARG, "limit_us=%d outside [1, 1e6]", limit_us);
  if (int rc = check_device(h)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SFFN_CUDA(launch_timeout_probe(h->ctrl, (unsigned long long)limit_us * 1000ull, s));
  SFFN_CUDA(cudaEventRecord(h->ev, s));
  h->ev_valid = true;
  return SFFN_OK;
}

void sffn_destroy(sffn_t h) {
  if (!h) return;
  if (h->ev_valid) cudaEventSynchronize(h->ev);
  release(h);
  delete h;
}

}  // extern "C"
