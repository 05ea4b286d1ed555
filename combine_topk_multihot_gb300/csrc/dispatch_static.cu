// moe_dispatch_static_scratch: moe_dispatch for callers that cannot allocate
// device memory.
//
// moe_dispatch needs a small scratch buffer for its per-chunk expert masks and
// start rows (moe_layout.workspace, 2 * E * ceil(T/32) int32, plus a
// grid-barrier counter).  Some callers have no way to
// get one: a plugin inside an inference engine that owns every byte of the
// device pool and hands a layer only its declared inputs and outputs, or a
// serving loop that must never call cudaMalloc because it can synchronise the
// device and stall every stream.  This entry point takes its scratch from a
// fixed array that lives in the library's own device memory instead.
//
// The array below is a file-scope __device__ variable: every GPU on which
// the library is loaded holds its 2 MiB (+ 33 KiB) from load until the
// process exits.
// Host code only knows the symbol, not its device address, so the address is
// looked up with cudaGetSymbolAddress on the first call for each device (and
// again after a device reset, which loads the module into a new context) and
// handed to the kernels through the layout's workspace pointer.

#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr long long STATIC_SCRATCH_INTS = MOE_STATIC_SCRATCH_INTS;  // (expert, chunk) pairs

// Per (expert, chunk) pair a token mask and a start row (2 MiB), then the
// dispatch kernel's grid-barrier words and 8 copies of up to 1024 expert
// counts (33 KiB).
static __device__ __align__(256) int g_dispatch_scratch[2 * STATIC_SCRATCH_INTS + (1280 + 8 * 1024 * 4) / 4];

constexpr int MAX_DEVICES = 64;
std::mutex g_scratch_mu;
// Device address of g_dispatch_scratch per device, and the unique id of the
// context it was looked up in: after a device reset the module is loaded
// again into a new context and the old address is stale.
int* g_scratch_ptr[MAX_DEVICES];
unsigned long long g_scratch_ctx[MAX_DEVICES];

// Device address of the static scratch on the current device.  It is looked
// up on the first call for the device, and again after the device's context
// has changed (a device reset).  The lookup can load the library's module, so
// it is refused while `stream` is being captured.
moe_status static_scratch(cudaStream_t stream, int** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) {
    char msg[160];
    snprintf(msg, sizeof(msg), "moe_dispatch_static_scratch: cudaGetDevice: %s", cudaGetErrorString(err));
    return set_last_error(MOE_ERR_CUDA, msg);
  }
  if (dev < 0 || dev >= MAX_DEVICES)
    return set_last_error(MOE_ERR_DEVICE, "moe_dispatch_static_scratch: device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long ctx = 0;
  const bool known_ctx = current_context_id(&ctx);
  if (g_scratch_ptr[dev] && known_ctx && ctx == g_scratch_ctx[dev]) {
    *out = g_scratch_ptr[dev];
    return MOE_OK;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  err = cudaStreamIsCapturing(stream, &cap);
  if (err != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return set_last_error(MOE_ERR_INVALID_ARG,
                          "moe_dispatch_static_scratch: the first call on a device (and the first "
                          "after a device reset) looks up the static scratch's address and must not "
                          "be made while its stream is being captured");
  void* p = nullptr;
  err = cudaGetSymbolAddress(&p, g_dispatch_scratch);
  if (err != cudaSuccess || p == nullptr) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "moe_dispatch_static_scratch: cudaGetSymbolAddress of the static scratch failed: %s",
             cudaGetErrorString(err));
    return set_last_error(MOE_ERR_CUDA, msg);
  }
  // Cache the address only when the context is known, so a reset is seen.
  unsigned long long now = 0;
  g_scratch_ptr[dev] = current_context_id(&now) ? static_cast<int*>(p) : nullptr;
  g_scratch_ctx[dev] = now;
  *out = static_cast<int*>(p);
  return MOE_OK;
}

}  // namespace

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (driver entry points
// reached through the runtime, so the library does not link libcuda);
// false when there is none yet or the driver does not say.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  return get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
         get_id(ctx, id) == CUDA_SUCCESS;
}


}  // namespace moe

using namespace moe;

extern "C" moe_status moe_dispatch_static_scratch(const moe_bf16* x, const uint8_t* routing_map,
                                                  const float* probs, int32_t H,
                                                  const moe_layout* L, moe_bf16* x_disp,
                                                  int64_t* rows_host, moe_stream_t stream) {
  if (L == nullptr) return set_last_error(MOE_ERR_INVALID_ARG, "moe_dispatch_static_scratch: layout is NULL");
  if (L->T < 0 || L->E < 1)
    return set_last_error(MOE_ERR_INVALID_ARG, "moe_dispatch_static_scratch: bad T or E");
  const long long needed = layout_chunks(L->T) * static_cast<long long>(L->E);
  size_t ws_bytes = 0;
  if (moe_layout_workspace_bytes(L->T, L->E, &ws_bytes) != MOE_OK || needed > STATIC_SCRATCH_INTS ||
      ws_bytes > sizeof(g_dispatch_scratch)) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "moe_dispatch_static_scratch: E * ceil(T/32) = %lld (expert, chunk) pairs exceeds the "
             "static scratch's %lld (T=%d, E=%d); use moe_dispatch with a caller-provided workspace",
             needed, STATIC_SCRATCH_INTS, L->T, L->E);
    return set_last_error(MOE_ERR_UNSUPPORTED_SHAPE, msg);
  }
  int* scratch = nullptr;
  moe_status st = static_scratch(stream, &scratch);
  if (st != MOE_OK) return st;
  // Same call as moe_dispatch; only the scratch differs.  Every counter the
  // kernels read is written earlier in the same call (the barrier counter is
  // zeroed by the launch itself), so nothing in the array has to start at zero.
  moe_layout with_scratch = *L;
  with_scratch.workspace = scratch;
  return moe_dispatch(x, routing_map, probs, H, &with_scratch, x_disp, rows_host, stream);
}
