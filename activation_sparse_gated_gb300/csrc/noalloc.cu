// noalloc.cu -- a forward entry point that allocates no device memory.
//
// Some callers cannot call cudaMalloc at all: an inference runtime that hands
// every byte of device memory to its own arena at start-up, code running where
// allocation would synchronise the device or break a latency budget, or an
// embedding host that only lends out buffers it owns.  sffn_forward_noalloc
// serves them.  The caller passes the weights, x and y (and optionally a
// counts buffer); the only scratch the forward needs -- the fp32 accumulator
// copies of y, the control words and the live-count accumulators -- lives in
// the fixed static device array below, which the library image brings with it
// (every GPU that loads the library holds it until exit).
//
// Each token runs the handle path's single-token streaming kernel followed by
// the finalize kernel (the same two launches sffn_forward makes for B = 1).
// Neither kernel waits on anything on the device, so no device-side timeout
// can leave y half-written.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sffn.h"

using namespace sffn;

namespace {

// Scratch layout (bytes): YACC_COPIES fp32 accumulator copies of D <= 4096
// values; the control words (256-byte aligned); SFFN_MAX_BATCH ints of live
// counts used when the caller passes no counts buffer.
constexpr int kMaxD = SFFN_MAX_D_BF16;
constexpr size_t kYaccOff = 0;
constexpr size_t kCtrlOff = sizeof(float) * YACC_COPIES * kMaxD;
constexpr size_t kCountsOff = kCtrlOff + ((sizeof(int) * CTRL_INTS + 255) / 256) * 256;
constexpr size_t kScratchBytes = kCountsOff + sizeof(int) * SFFN_MAX_BATCH;  // 66,816 bytes
static_assert(kScratchBytes == 66816, "the header states this size");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on that device
  int num_sms = 0;
  size_t max_smem = 0;
};

std::mutex g_mu;
DeviceSetup g_dev[kMaxDevices];

int fail(int code, const char* msg, cudaError_t e = cudaSuccess) {
  char buf[256];
  if (e != cudaSuccess)
    snprintf(buf, sizeof buf, "sffn_forward_noalloc: %s: %s", msg, cudaGetErrorString(e));
  else
    snprintf(buf, sizeof buf, "sffn_forward_noalloc: %s", msg);
  set_last_error(buf);
  return code;
}

// Once per device, with that device current: look up the scratch array's
// device address (in host code the array's name is only a host-side stand-in)
// and raise the streaming kernel's shared-memory limit.
int setup(int dev, DeviceSetup** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceSetup& d = g_dev[dev];
  if (!d.ready) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return fail(SFFN_ERR_CUDA, "cudaGetSymbolAddress", e);
    int sms = 0, optin = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return fail(SFFN_ERR_CUDA, "cudaDeviceGetAttribute", e);
    if ((e = ffn_b1_stream_prepare((size_t)optin)) != cudaSuccess)
      return fail(SFFN_ERR_CUDA, "cudaFuncSetAttribute", e);
    d.scratch = static_cast<unsigned char*>(ptr);
    d.num_sms = sms;
    d.max_smem = (size_t)optin;
    d.ready = true;
  }
  *out = &d;
  return SFFN_OK;
}

}  // namespace

extern "C" int sffn_forward_noalloc(const void* W1, const void* W3, const void* W2t, const void* x,
                                    void* y, int* counts, int D, int H, int B, int act, int dtype,
                                    void* stream) {
  if (dtype != SFFN_F32 && dtype != SFFN_BF16) return fail(SFFN_ERR_ARG, "unknown dtype");
  if (act != SFFN_ACT_RELU && act != SFFN_ACT_RSP) return fail(SFFN_ERR_ARG, "unknown activation");
  const int dmax = dtype == SFFN_BF16 ? SFFN_MAX_D_BF16 : SFFN_MAX_D_F32;
  if (D < 8 || D % 8 != 0 || D > dmax)
    return fail(SFFN_ERR_ARG, "D must be a multiple of 8 no larger than the static scratch allows "
                              "(4096 for bf16, 2048 for f32)");
  if (H < 1) return fail(SFFN_ERR_ARG, "H must be >= 1");
  if (B < 1 || B > SFFN_MAX_BATCH) return fail(SFFN_ERR_ARG, "B must be in [1, 128]");
  if (!W1 || !W3 || !W2t || !x || !y) return fail(SFFN_ERR_ARG, "null pointer");
  // weights, x and y are read and written with 16-byte vector accesses; the
  // kernels store one int per token into counts
  const uintptr_t a = (uintptr_t)W1 | (uintptr_t)W3 | (uintptr_t)W2t | (uintptr_t)x | (uintptr_t)y;
  if (a & 15) return fail(SFFN_ERR_ALIGN, "W1, W3, W2t, x and y must be 16-byte aligned");
  if ((uintptr_t)counts & 3) return fail(SFFN_ERR_ALIGN, "counts must be 4-byte aligned");
  const int elt = dtype == SFFN_BF16 ? 2 : 4;
  const size_t xbytes = (size_t)B * D * elt;
  const uintptr_t px = (uintptr_t)x, py = (uintptr_t)y;
  if (px < py + xbytes && py < px + xbytes) return fail(SFFN_ERR_ARG, "x and y overlap");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SFFN_ERR_CUDA, "cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return fail(SFFN_ERR_ARG, "device ordinal out of range");
  DeviceSetup* d = nullptr;
  if (int rc = setup(dev, &d)) return rc;

  // the streaming kernel's launch plan (the rules of a handle's plan)
  const int grid = d->num_sms < H ? d->num_sms : H;
  const int rows_cap = (H + grid - 1) / grid;
  const StreamPlan plan = plan_ffn_b1_stream(D, D, elt, false, rows_cap);
  if (plan.smem > d->max_smem) return fail(SFFN_ERR_DTYPE, "D does not fit the streaming kernel's shared memory");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* yacc = reinterpret_cast<float*>(d->scratch + kYaccOff);
  int* ctrl = reinterpret_cast<int*>(d->scratch + kCtrlOff);
  int* own_counts = reinterpret_cast<int*>(d->scratch + kCountsOff);
  // The scratch keeps whatever the previous call left (the finalize kernel
  // clears the accumulators and count words it used); clear what must start
  // at zero anyway, so that a call never depends on an earlier one.
  if ((e = cudaMemsetAsync(yacc, 0, sizeof(float) * YACC_COPIES * D, s)) != cudaSuccess ||
      (e = cudaMemsetAsync(ctrl, 0, sizeof(int) * CTRL_INTS, s)) != cudaSuccess)
    return fail(SFFN_ERR_CUDA, "cudaMemsetAsync", e);
  const size_t row = (size_t)D * elt;
  for (int b = 0; b < B; ++b) {
    B1Params p;
    p.gate_w = W1;
    p.W3 = W3;
    p.W2t = W2t;
    p.x = static_cast<const unsigned char*>(x) + b * row;
    p.t = nullptr;
    p.y = static_cast<unsigned char*>(y) + b * row;
    p.yacc = yacc;
    p.ctrl = ctrl;
    p.counts = counts ? counts + b : own_counts + b;
    p.mask = nullptr;
    p.D = D;
    p.H = H;
    p.gate_k = D;
    p.act = act;
    p.count_slot = b;
    p.rows_cap = rows_cap;
    p.pref_rows = plan.pref_rows;
    p.gather_rows = plan.gather_rows;
    if ((e = launch_ffn_b1_stream(p, dtype, false, grid, plan.smem, s)) != cudaSuccess)
      return fail(SFFN_ERR_CUDA, "kernel launch", e);
    if ((e = launch_finalize(yacc, p.y, ctrl, p.counts, b, D, 1, dtype, s)) != cudaSuccess)
      return fail(SFFN_ERR_CUDA, "kernel launch", e);
  }
  return SFFN_OK;
}
