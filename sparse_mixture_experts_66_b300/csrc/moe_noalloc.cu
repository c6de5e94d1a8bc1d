// moe_forward_noalloc: the layer forward for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc or any allocating routine: plugin and
// custom-op hosts that hand a kernel only its inputs and outputs, and code
// whose device memory is owned by another allocator that forbids direct
// allocation (cudaMalloc may also synchronise the device, which
// latency-critical paths must avoid). For them this entry point keeps the
// forward's scratch in a file-scope device array of fixed size instead of a
// caller-provided workspace.
//
// Properties, all deliberate:
//   - the array is kNoallocBytes (32 MiB). Every GPU that loads this library
//     reserves it until the process exits;
//   - a config whose workspace (moe_workspace_bytes) is larger is rejected with
//     MOE_ERR_WORKSPACE before anything is enqueued;
//   - the first call on a device looks up the array's device address with
//     cudaGetSymbolAddress (once per device, with that device current); make
//     that first call before any stream capture;
//   - every call shares the one array, which keeps the previous call's
//     contents. Each call clears the status word at the start (the only part
//     that must start at zero); calls whose GPU work overlaps (two streams, or
//     two host threads) race on the array;
//   - device-side error words (bounded-wait timeouts, bounds checks) land in
//     the array's status word, which moe_get_device_status cannot reach: this
//     entry point reports host-side errors only.
// It calls no cudaMalloc, cudaFree or other allocating routine.
#include <stdio.h>

#include <mutex>

#include "moe_internal.cuh"

namespace {

constexpr size_t kNoallocBytes = (size_t)32 << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device). Returns a cudaError_t.
cudaError_t scratch_on_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

thread_local char g_noalloc_err[512] = "";

}  // namespace

extern "C" {

moe_status moe_forward_noalloc(const moe_config *cfg, const void *x, const void *w_g, const float *router_bias,
                               const void *w1, const void *b1, const void *w2, const void *b2, void *y,
                               moe_stream_t stream) {
  const size_t need = moe_workspace_bytes(cfg);
  if (need == 0) return moe_get_workspace_layout(cfg, nullptr);  // invalid config: report why
  if (need > kNoallocBytes) {
    snprintf(g_noalloc_err, sizeof(g_noalloc_err),
             "moe_forward_noalloc: this config needs %zu bytes of scratch, more than the fixed %zu bytes; use "
             "moe_forward with a caller-provided workspace",
             need, kNoallocBytes);
    moe::set_last_error(g_noalloc_err);
    return MOE_ERR_WORKSPACE;
  }
  void *ws = nullptr;
  cudaError_t e = scratch_on_current_device(&ws);
  if (e != cudaSuccess) {
    snprintf(g_noalloc_err, sizeof(g_noalloc_err), "moe_forward_noalloc: scratch set-up failed: %s (%s)",
             cudaGetErrorName(e), cudaGetErrorString(e));
    moe::set_last_error(g_noalloc_err);
    return MOE_ERR_CUDA;
  }
  moe_workspace_layout L;
  moe_status st = moe_get_workspace_layout(cfg, &L);
  if (st != MOE_OK) return st;
  e = cudaMemsetAsync(static_cast<char *>(ws) + L.status, 0, 64, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    snprintf(g_noalloc_err, sizeof(g_noalloc_err), "moe_forward_noalloc: clearing the status word failed: %s",
             cudaGetErrorName(e));
    moe::set_last_error(g_noalloc_err);
    return MOE_ERR_CUDA;
  }
  return moe_forward(cfg, x, w_g, router_bias, w1, b1, w2, b2, y, ws, stream);
}

}  // extern "C"
