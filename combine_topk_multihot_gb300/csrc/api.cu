// The C ABI declared in include/moe.h: argument validation on the host, then
// the launches.  No allocation, no global state besides per-device caches of
// immutable device properties and the thread-local error text.

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <chrono>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

thread_local char g_last_error[512] = "";

moe_status fail(moe_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

moe_status cuda_fail(cudaError_t err, const char* where) {
  return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(err));
}

constexpr int MAX_DEVICES = 64;
int g_cc_ok[MAX_DEVICES];    // 0 unknown, 1 compute capability 10.3, -1 other
int g_sms[MAX_DEVICES];

// The host-synced dispatch reads R, N and the status word from 16 bytes of
// mapped pinned host memory that the layout kernel writes directly, so the
// readback needs no copy engine and cannot queue behind bulk copies on other
// streams.  One buffer per device, made on first use; the mutex is held from
// the launch until the kernel can no longer write to it, so concurrent
// host-synced calls take turns.
std::mutex g_rb_mu;
// The host polls the mapped buffer for this long before it falls back to a
// stream synchronisation (the layout kernel's own waits give up after 2 s).
constexpr int READBACK_POLL_LIMIT_S = 10;
int* g_rb_host[MAX_DEVICES];
int* g_rb_dev[MAX_DEVICES];

bool readback_buffer(int dev, int** host, int** dev_ptr) {
  if (dev < 0 || dev >= MAX_DEVICES) return false;
  if (!g_rb_host[dev]) {
    void* h = nullptr;
    void* d = nullptr;
    if (cudaHostAlloc(&h, 16, cudaHostAllocMapped) != cudaSuccess) return false;
    if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess) {
      cudaFreeHost(h);
      return false;
    }
    g_rb_host[dev] = static_cast<int*>(h);
    g_rb_dev[dev] = static_cast<int*>(d);
  }
  *host = g_rb_host[dev];
  *dev_ptr = g_rb_dev[dev];
  return true;
}

moe_status check_device() {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (dev < 0 || dev >= MAX_DEVICES) return fail(MOE_ERR_DEVICE, "device ordinal %d unsupported", dev);
  if (g_cc_ok[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    if ((err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(err, "cudaDeviceGetAttribute");
    g_sms[dev] = sms;
    g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    if (g_cc_ok[dev] < 0) {
      return fail(MOE_ERR_DEVICE, "device %d has compute capability %d.%d; this library is built for 10.3 (sm_103a)",
                  dev, major, minor);
    }
  }
  if (g_cc_ok[dev] < 0) return fail(MOE_ERR_DEVICE, "device %d is not compute capability 10.3", dev);
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define MOE_REQUIRE(cond, st, ...) \
  do {                             \
    if (!(cond)) return fail(st, __VA_ARGS__); \
  } while (0)

moe_status check_routing_shape(int32_t T, int32_t K, int32_t E) {
  MOE_REQUIRE(T >= 0, MOE_ERR_INVALID_ARG, "T must be >= 0 (got %d)", T);
  MOE_REQUIRE(E >= 1 && E <= 1024, MOE_ERR_UNSUPPORTED_SHAPE, "E must be in [1, 1024] (got %d)", E);
  MOE_REQUIRE(E % 4 == 0, MOE_ERR_UNSUPPORTED_SHAPE, "E must be a multiple of 4 (got %d)", E);
  MOE_REQUIRE(K >= 1 && K <= E && K <= 127, MOE_ERR_UNSUPPORTED_SHAPE,
              "K must be in [1, min(E, 127)] (got K=%d, E=%d)", K, E);
  return MOE_OK;
}

moe_status check_hidden(int32_t H) {
  MOE_REQUIRE(H > 0 && H % 256 == 0, MOE_ERR_UNSUPPORTED_SHAPE,
              "the hidden size must be a positive multiple of 256 (got %d)", H);
  return MOE_OK;
}

moe_status check_layout(const moe_layout* L) {
  MOE_REQUIRE(L != nullptr, MOE_ERR_INVALID_ARG, "layout is NULL");
  moe_status st = check_routing_shape(L->T, L->K, L->E);
  if (st != MOE_OK) return st;
  MOE_REQUIRE(L->pad_multiple >= 1, MOE_ERR_INVALID_ARG, "pad_multiple must be >= 1 (got %d)",
              L->pad_multiple);
  MOE_REQUIRE(L->capacity >= 0, MOE_ERR_INVALID_ARG, "capacity must be >= 0");
  const int64_t worst = static_cast<int64_t>(L->T) * L->K +
                        static_cast<int64_t>(L->E) * (L->pad_multiple - 1);
  MOE_REQUIRE(worst < (int64_t(1) << 31) && L->capacity < (int64_t(1) << 31),
              MOE_ERR_UNSUPPORTED_SHAPE, "row counts must fit in int32");
  MOE_REQUIRE(L->tokens_per_expert && L->offsets && L->totals && L->status && L->workspace,
              MOE_ERR_INVALID_ARG, "layout has a NULL count/offset/total/status/workspace pointer");
  MOE_REQUIRE(L->capacity == 0 || (L->row_token && L->row_expert && L->row_weight),
              MOE_ERR_INVALID_ARG, "layout has a NULL row buffer");
  MOE_REQUIRE(L->T == 0 || L->token_row, MOE_ERR_INVALID_ARG, "layout has a NULL token_row");
  MOE_REQUIRE(aligned16(L->workspace), MOE_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  return MOE_OK;
}

}  // namespace

moe_status set_last_error(moe_status st, const char* text) { return fail(st, "%s", text); }

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return 148;
  if (g_sms[dev] == 0) {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = sms > 0 ? sms : 148;
  }
  return g_sms[dev];
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY";
    case MOE_ERR_BAD_INDEX: return "MOE_ERR_BAD_INDEX";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_last_error(void) { return g_last_error; }

moe_status moe_device_check(void) { return check_device(); }

uint32_t moe_build_flags(void) {
#ifdef MOE_DEBUG_BOUNDS
  return MOE_BUILD_BOUNDS_CHECKS;
#else
  return 0u;
#endif
}

int64_t moe_worst_case_rows(int32_t T, int32_t E, int32_t K, int32_t pad_multiple) {
  if (T < 0 || E < 1 || K < 1 || pad_multiple < 1) return -1;
  return static_cast<int64_t>(T) * K + static_cast<int64_t>(E) * (pad_multiple - 1);
}

moe_status moe_layout_workspace_bytes(int32_t T, int32_t E, size_t* bytes) {
  MOE_REQUIRE(bytes != nullptr, MOE_ERR_INVALID_ARG, "bytes is NULL");
  MOE_REQUIRE(T >= 0 && E >= 1, MOE_ERR_INVALID_ARG, "bad T/E");
  *bytes = dispatch_workspace_bytes(T, E);
  return MOE_OK;
}

moe_status moe_route_to_multihot(const int64_t* topk_idx, const float* topk_probs, int32_t T,
                                 int32_t K, int32_t E, uint8_t* routing_map, float* probs,
                                 int8_t* winner_slot, int32_t* status, moe_stream_t stream) {
  moe_status st = check_routing_shape(T, K, E);
  if (st != MOE_OK) return st;
  MOE_REQUIRE(T == 0 || (topk_idx && topk_probs && routing_map && probs && winner_slot && status),
              MOE_ERR_INVALID_ARG, "moe_route_to_multihot: NULL pointer");
  MOE_REQUIRE(aligned16(routing_map) && aligned16(probs) && aligned16(winner_slot),
              MOE_ERR_INVALID_ARG, "moe_route_to_multihot: outputs must be 16-byte aligned");
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t err = launch_multihot(topk_idx, topk_probs, T, K, E, routing_map, probs, winner_slot,
                                    status, stream);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_route_to_multihot launch");
}

}  // extern "C"

namespace {

// moe_dispatch and moe_dispatch_fp8: the layout (host-synced or sync-free),
// then the rows, in bf16 (x_disp) or as e4m3 codes with per-row scales.
// With topk_idx non-NULL the input is the top-k choices, and routing_map /
// probs / winner are outputs (the multihot step fused into the dispatch).
moe_status dispatch_impl(const char* who, const moe_bf16* x, const uint8_t* routing_map,
                         const float* probs, int32_t H, const moe_layout* L, moe_bf16* x_disp,
                         uint8_t* x_q, float* x_scale, int64_t* rows_host, moe_stream_t stream,
                         bool layout_only = false, const int64_t* topk_idx = nullptr,
                         const float* topk_probs = nullptr, int8_t* winner = nullptr) {
  moe_status st = check_layout(L);
  if (st != MOE_OK) return st;
  if (layout_only) H = 256;  // no rows are copied; any valid hidden size will do
  if ((st = check_hidden(H)) != MOE_OK) return st;
  MOE_REQUIRE(L->T == 0 || ((x || layout_only) && routing_map && probs), MOE_ERR_INVALID_ARG,
              "%s: NULL input", who);
  MOE_REQUIRE(!topk_idx || L->T == 0 || (topk_probs && winner), MOE_ERR_INVALID_ARG,
              "%s: NULL top-k input or multihot output", who);
  MOE_REQUIRE(aligned16(probs) && aligned16(winner), MOE_ERR_INVALID_ARG,
              "%s: probs and winner_slot must be 16-byte aligned", who);
  MOE_REQUIRE(L->capacity == 0 || layout_only || x_disp || (x_q && x_scale), MOE_ERR_INVALID_ARG,
              "%s: NULL output rows", who);
  MOE_REQUIRE(aligned16(x) && aligned16(x_disp) && aligned16(x_q) && aligned16(routing_map),
              MOE_ERR_INVALID_ARG, "%s: x, the output rows and routing_map must be 16-byte aligned",
              who);
  const int64_t worst = moe_worst_case_rows(L->T, L->E, L->K, L->pad_multiple);
  if (!rows_host && L->capacity < worst)
    return fail(MOE_ERR_CAPACITY,
                "sync-free dispatch needs capacity >= T*K + E*(pad_multiple-1) = %lld rows (got %lld)",
                static_cast<long long>(worst), static_cast<long long>(L->capacity));
  if ((st = check_device()) != MOE_OK) return st;

  // Host-synced callers get R, N and the status word through mapped pinned
  // memory that the layout kernel writes as soon as the offsets are known.
  int *rb_host = nullptr, *rb_dev = nullptr;
  std::unique_lock<std::mutex> rb_lock(g_rb_mu, std::defer_lock);
  bool mapped = false;
  if (rows_host) {
    int dev = 0;
    rb_lock.lock();
    mapped = cudaGetDevice(&dev) == cudaSuccess && readback_buffer(dev, &rb_host, &rb_dev);
    if (mapped) {
      volatile int* rb = rb_host;
      rb[0] = rb[1] = rb[2] = -1;  // overwritten by the layout kernel
    } else {
      rb_lock.unlock();
    }
  }
  // The layout, then the rows (or, for the layout alone, just the pad and
  // spare rows' metadata), queued at once in both modes.  When the rows do
  // not fit (host-synced, R > capacity) both kernels write nothing.
  cudaError_t err;
  bool rows_done = false;  // the layout kernel did the row pass itself
  const bool bf16_rows = x_disp || layout_only;
  const bool fp8_rows = !bf16_rows && x_q != nullptr;
  const bool fused = (bf16_rows || fp8_rows) && dispatch_fused_fits(*L);
  const uint16_t* x16 = reinterpret_cast<const uint16_t*>(x);
  uint16_t* xd16 = reinterpret_cast<uint16_t*>(x_disp);
  int* rb_kernel = mapped ? rb_dev : nullptr;
  if (topk_idx && !fused) {
    // small layers: the multihot step first, then the layout from its map
    if ((err = launch_multihot(topk_idx, topk_probs, L->T, L->K, L->E, const_cast<uint8_t*>(routing_map),
                               const_cast<float*>(probs), winner, L->status, stream)) != cudaSuccess) {
      if (mapped) rb_lock.unlock();
      return cuda_fail(err, "dispatch: multihot");
    }
  }
  if (fused) {
    if (topk_idx)
      err = fp8_rows ? launch_dispatch_fused_topk_fp8(topk_idx, topk_probs, const_cast<uint8_t*>(routing_map),
                                                      const_cast<float*>(probs), winner, *L, H, x16, x_q, x_scale,
                                                      rb_kernel, stream)
                     : launch_dispatch_fused_topk(topk_idx, topk_probs, const_cast<uint8_t*>(routing_map),
                                                  const_cast<float*>(probs), winner, *L, H, x16, xd16, rb_kernel,
                                                  stream);
    else
      err = fp8_rows ? launch_dispatch_fused_map_fp8(routing_map, probs, *L, H, x16, x_q, x_scale, rb_kernel, stream)
                     : launch_dispatch_fused_map(routing_map, probs, *L, H, x16, xd16, rb_kernel, stream);
    if (err != cudaSuccess) {
      if (mapped) cudaStreamSynchronize(stream);  // the kernel may still write the readback buffer
      return cuda_fail(err, "dispatch: fused layout and rows");
    }
    rows_done = true;
  } else if ((err = launch_layout(routing_map, probs, *L, L->workspace, stream, rb_kernel, x16, xd16, H,
                                  bf16_rows ? &rows_done : nullptr)) != cudaSuccess) {
    return cuda_fail(err, "dispatch: layout");
  }
  if (!rows_done) {
    err = bf16_rows ? launch_row_gather(x, *L, H, x_disp, true, nullptr, nullptr, stream)
                    : launch_row_gather_fp8(x, *L, H, x_q, x_scale, stream);
    if (err != cudaSuccess) {
      // the layout kernel may still write the readback buffer: let it finish
      // before the buffer goes to the next caller
      if (mapped) cudaStreamSynchronize(stream);
      return cuda_fail(err, "dispatch: rows");
    }
  }
  if (!rows_host) return MOE_OK;

  // Host-synced: wait for the counts.  With the mapped buffer, until the
  // layout kernel publishes R (the kernels behind it keep running), or until
  // the stream is idle without it (the kernel gave up: read the device
  // copies).
  int32_t tot[2] = {0, 0}, dev_status = 0;
  volatile int* rb = rb_host;
  bool published = false;
  if (mapped) {
    const auto t0 = std::chrono::steady_clock::now();
    for (unsigned spin = 0;; ++spin) {
      if (rb[0] >= 0) {
        published = true;
        break;
      }
      if ((spin & 255u) != 255u) continue;
      const cudaError_t q = cudaStreamQuery(stream);
      if (q == cudaSuccess) {
        published = rb[0] >= 0;
        break;
      }
      if (q != cudaErrorNotReady) {
        cudaStreamSynchronize(stream);  // as above: nothing may write the buffer afterwards
        return cuda_fail(q, "dispatch: waiting for the row counts");
      }
      if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(READBACK_POLL_LIMIT_S)) break;
    }
  }
  if (published) {
    std::atomic_thread_fence(std::memory_order_acquire);
    tot[0] = rb[0];
    tot[1] = rb[1];
    dev_status = rb[2];
  } else if ((err = cudaStreamSynchronize(stream)) != cudaSuccess ||
             (err = cudaMemcpy(tot, L->totals, sizeof(tot), cudaMemcpyDeviceToHost)) != cudaSuccess ||
             (err = cudaMemcpy(&dev_status, L->status, sizeof(int32_t), cudaMemcpyDeviceToHost)) != cudaSuccess) {
    return cuda_fail(err, "dispatch: reading the row counts");
  }
  if (rb_lock.owns_lock()) rb_lock.unlock();
  rows_host[0] = tot[0];
  rows_host[1] = tot[1];
  if (dev_status & MOE_DEVERR_TIMEOUT)
    return fail(MOE_ERR_TIMEOUT, "the layout kernel's grid barrier timed out");
  if (dev_status & MOE_DEVERR_BAD_INDEX)
    return fail(MOE_ERR_BAD_INDEX, "an expert index outside [-1, E) was seen");
  if (tot[0] > L->capacity)
    return fail(MOE_ERR_CAPACITY, "the layout needs %d rows, capacity is %lld", tot[0],
                static_cast<long long>(L->capacity));
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_dispatch(const moe_bf16* x, const uint8_t* routing_map, const float* probs,
                        int32_t H, const moe_layout* L, moe_bf16* x_disp, int64_t* rows_host,
                        moe_stream_t stream) {
  MOE_REQUIRE(L == nullptr || L->capacity == 0 || x_disp, MOE_ERR_INVALID_ARG,
              "moe_dispatch: NULL x_disp");
  return dispatch_impl("moe_dispatch", x, routing_map, probs, H, L, x_disp, nullptr, nullptr,
                       rows_host, stream);
}

moe_status moe_dispatch_topk(const moe_bf16* x, const int64_t* topk_idx, const float* topk_probs,
                             int32_t H, const moe_layout* L, uint8_t* routing_map, float* probs,
                             int8_t* winner_slot, moe_bf16* x_disp, int64_t* rows_host,
                             moe_stream_t stream) {
  MOE_REQUIRE(L == nullptr || L->capacity == 0 || x_disp, MOE_ERR_INVALID_ARG,
              "moe_dispatch_topk: NULL x_disp");
  MOE_REQUIRE(L == nullptr || L->T == 0 || (topk_idx && topk_probs), MOE_ERR_INVALID_ARG,
              "moe_dispatch_topk: NULL top-k input");
  static const int64_t no_slots = 0;  // T == 0: marks the top-k input without reading it
  return dispatch_impl("moe_dispatch_topk", x, routing_map, probs, H, L, x_disp, nullptr, nullptr,
                       rows_host, stream, false, topk_idx ? topk_idx : &no_slots, topk_probs,
                       winner_slot);
}

moe_status moe_dispatch_topk_fp8(const moe_bf16* x, const int64_t* topk_idx, const float* topk_probs,
                                 int32_t H, const moe_layout* L, uint8_t* routing_map, float* probs,
                                 int8_t* winner_slot, uint8_t* x_disp_q, float* x_disp_scale, int64_t* rows_host,
                                 moe_stream_t stream) {
  MOE_REQUIRE(L == nullptr || L->capacity == 0 || (x_disp_q && x_disp_scale), MOE_ERR_INVALID_ARG,
              "moe_dispatch_topk_fp8: NULL x_disp_q or x_disp_scale");
  MOE_REQUIRE(L == nullptr || L->T == 0 || (topk_idx && topk_probs), MOE_ERR_INVALID_ARG,
              "moe_dispatch_topk_fp8: NULL top-k input");
  static const int64_t no_slots = 0;  // T == 0: marks the top-k input without reading it
  return dispatch_impl("moe_dispatch_topk_fp8", x, routing_map, probs, H, L, nullptr, x_disp_q, x_disp_scale,
                       rows_host, stream, false, topk_idx ? topk_idx : &no_slots, topk_probs, winner_slot);
}

moe_status moe_dispatch_fp8(const moe_bf16* x, const uint8_t* routing_map, const float* probs,
                            int32_t H, const moe_layout* L, uint8_t* x_disp_q, float* x_disp_scale,
                            int64_t* rows_host, moe_stream_t stream) {
  MOE_REQUIRE(L == nullptr || L->capacity == 0 || (x_disp_q && x_disp_scale), MOE_ERR_INVALID_ARG,
              "moe_dispatch_fp8: NULL x_disp_q or x_disp_scale");
  return dispatch_impl("moe_dispatch_fp8", x, routing_map, probs, H, L, nullptr, x_disp_q,
                       x_disp_scale, rows_host, stream);
}

moe_status moe_dispatch_layout(const uint8_t* routing_map, const float* probs, const moe_layout* L,
                               int64_t* rows_host, moe_stream_t stream) {
  return dispatch_impl("moe_dispatch_layout", nullptr, routing_map, probs, 256, L, nullptr, nullptr,
                       nullptr, rows_host, stream, /*layout_only=*/true);
}

moe_status moe_grouped_experts_gather(const moe_bf16* x, const moe_layout* L, int32_t H, int32_t I,
                                      const moe_bf16* W1, const moe_bf16* W2, moe_bf16* h,
                                      moe_bf16* y_disp, moe_bf16* o_save, moe_bf16* gu_save,
                                      moe_stream_t stream) {
  moe_status st = check_layout(L);
  if (st != MOE_OK) return st;
  if ((st = check_hidden(H)) != MOE_OK) return st;
  MOE_REQUIRE(I > 0 && I % 128 == 0, MOE_ERR_UNSUPPORTED_SHAPE,
              "the intermediate size must be a positive multiple of 128 (got %d)", I);
  MOE_REQUIRE(L->capacity == 0 || ((x || L->T == 0) && W1 && W2 && h && y_disp), MOE_ERR_INVALID_ARG,
              "moe_grouped_experts_gather: NULL pointer");
  MOE_REQUIRE(aligned16(x) && aligned16(W1) && aligned16(W2) && aligned16(h) && aligned16(y_disp) &&
                  aligned16(o_save) && aligned16(gu_save),
              MOE_ERR_INVALID_ARG, "moe_grouped_experts_gather: pointers must be 16-byte aligned");
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t err = launch_experts_forward_gather(x, *L, H, I, W1, W2, h, y_disp, o_save, gu_save, stream);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_grouped_experts_gather launch");
}

moe_status moe_quantize_fp8(const moe_bf16* src, int64_t rows, int32_t cols, uint8_t* codes,
                            float* scales, moe_stream_t stream) {
  MOE_REQUIRE(rows >= 0, MOE_ERR_INVALID_ARG, "moe_quantize_fp8: rows must be >= 0");
  MOE_REQUIRE(cols > 0 && cols % 256 == 0, MOE_ERR_UNSUPPORTED_SHAPE,
              "moe_quantize_fp8: cols must be a positive multiple of 256 (got %d)", cols);
  MOE_REQUIRE(rows == 0 || (src && codes && scales), MOE_ERR_INVALID_ARG,
              "moe_quantize_fp8: NULL pointer");
  MOE_REQUIRE(aligned16(src) && aligned16(codes), MOE_ERR_INVALID_ARG,
              "moe_quantize_fp8: src and codes must be 16-byte aligned");
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  cudaError_t err = launch_quantize_rows_fp8(src, rows, cols, codes, scales, stream);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_quantize_fp8 launch");
}

moe_status moe_grouped_experts_fp8(const uint8_t* x_disp_q, const float* x_disp_scale,
                                   const moe_layout* L, int32_t H, int32_t I, const uint8_t* W1_q,
                                   const float* W1_scale, const moe_bf16* W2, moe_bf16* h,
                                   moe_bf16* y_disp, moe_stream_t stream) {
  moe_status st = check_layout(L);
  if (st != MOE_OK) return st;
  if ((st = check_hidden(H)) != MOE_OK) return st;
  MOE_REQUIRE(I > 0 && I % 128 == 0, MOE_ERR_UNSUPPORTED_SHAPE,
              "the intermediate size must be a positive multiple of 128 (got %d)", I);
  MOE_REQUIRE(L->capacity == 0 || (x_disp_q && x_disp_scale && W1_q && W1_scale && W2 && h && y_disp),
              MOE_ERR_INVALID_ARG, "moe_grouped_experts_fp8: NULL pointer");
  MOE_REQUIRE(aligned16(x_disp_q) && aligned16(W1_q) && aligned16(W2) && aligned16(h) &&
                  aligned16(y_disp),
              MOE_ERR_INVALID_ARG, "moe_grouped_experts_fp8: pointers must be 16-byte aligned");
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t err = launch_experts_forward_fp8(x_disp_q, x_disp_scale, *L, H, I, W1_q, W1_scale, W2,
                                               h, y_disp, stream);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_grouped_experts_fp8 launch");
}

moe_status moe_grouped_experts(const moe_bf16* x_disp, const moe_layout* L, int32_t H, int32_t I,
                               const moe_bf16* W1, const moe_bf16* W2, moe_bf16* h,
                               moe_bf16* y_disp, moe_bf16* o_save, moe_bf16* gu_save,
                               moe_stream_t stream) {
  moe_status st = check_layout(L);
  if (st != MOE_OK) return st;
  if ((st = check_hidden(H)) != MOE_OK) return st;
  MOE_REQUIRE(I > 0 && I % 128 == 0, MOE_ERR_UNSUPPORTED_SHAPE,
              "the intermediate size must be a positive multiple of 128 (got %d)", I);
  MOE_REQUIRE(L->capacity == 0 || (x_disp && W1 && W2 && h && y_disp), MOE_ERR_INVALID_ARG,
              "moe_grouped_experts: NULL pointer");
  MOE_REQUIRE(aligned16(x_disp) && aligned16(W1) && aligned16(W2) && aligned16(h) &&
                  aligned16(y_disp) && aligned16(o_save) && aligned16(gu_save),
              MOE_ERR_INVALID_ARG, "moe_grouped_experts: pointers must be 16-byte aligned");
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t err = launch_experts_forward(x_disp, *L, H, I, W1, W2, h, y_disp, o_save, gu_save, stream);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_grouped_experts launch");
}

moe_status moe_combine(const moe_bf16* y_disp, const moe_layout* L, int32_t H, moe_bf16* out,
                       moe_stream_t stream) {
  moe_status st = check_layout(L);
  if (st != MOE_OK) return st;
  if ((st = check_hidden(H)) != MOE_OK) return st;
  MOE_REQUIRE(L->T == 0 || (y_disp && out), MOE_ERR_INVALID_ARG, "moe_combine: NULL pointer");
  MOE_REQUIRE(aligned16(y_disp) && aligned16(out), MOE_ERR_INVALID_ARG,
              "moe_combine: pointers must be 16-byte aligned");
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t err = launch_combine(y_disp, *L, H, out, nullptr, nullptr, stream);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_combine launch");
}

}  // extern "C"

namespace {

moe_status combine_backward_impl(const char* who, const moe_bf16* grad_out, const moe_bf16* o_save,
                                 const moe_layout* L, int32_t H, moe_bf16* grad_y, float* grad_w,
                                 moe_stream_t stream, bool scale) {
  moe_status st = check_layout(L);
  if (st != MOE_OK) return st;
  if ((st = check_hidden(H)) != MOE_OK) return st;
  MOE_REQUIRE(L->capacity == 0 || (grad_out && grad_y), MOE_ERR_INVALID_ARG, "%s: NULL pointer", who);
  MOE_REQUIRE(!grad_w || o_save, MOE_ERR_INVALID_ARG, "%s: grad_w needs o_save", who);
  MOE_REQUIRE(aligned16(grad_out) && aligned16(grad_y) && aligned16(o_save), MOE_ERR_INVALID_ARG,
              "%s: pointers must be 16-byte aligned", who);
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t err = launch_row_gather(grad_out, *L, H, grad_y, false, o_save, grad_w, stream, scale);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, who);
}

moe_status experts_backward_impl(const char* who, const moe_bf16* grad_y, const moe_bf16* x_disp,
                                 const moe_bf16* h, const moe_bf16* gu_save, const moe_layout* L,
                                 int32_t H, int32_t I, const moe_bf16* W1, const moe_bf16* W2,
                                 moe_bf16* grad_x_disp, float* dW1, float* dW2, void* workspace,
                                 moe_stream_t stream, bool g_o_given) {
  moe_status st = check_layout(L);
  if (st != MOE_OK) return st;
  if ((st = check_hidden(H)) != MOE_OK) return st;
  MOE_REQUIRE(I > 0 && I % 128 == 0, MOE_ERR_UNSUPPORTED_SHAPE,
              "the intermediate size must be a positive multiple of 128 (got %d)", I);
  MOE_REQUIRE(W1 && W2 && dW1 && dW2 && workspace, MOE_ERR_INVALID_ARG,
              "%s: NULL weight, weight-gradient or workspace pointer", who);
  MOE_REQUIRE(L->capacity == 0 || (grad_y && x_disp && h && gu_save && grad_x_disp),
              MOE_ERR_INVALID_ARG, "%s: NULL row buffer", who);
  MOE_REQUIRE(aligned16(grad_y) && aligned16(x_disp) && aligned16(h) && aligned16(gu_save) &&
                  aligned16(W1) && aligned16(W2) && aligned16(grad_x_disp) && aligned16(dW1) &&
                  aligned16(dW2),
              MOE_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", who);
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t err = launch_experts_backward(grad_y, x_disp, h, gu_save, *L, H, I, W1, W2, grad_x_disp,
                                            dW1, dW2, workspace, stream, g_o_given);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, who);
}

}  // namespace

extern "C" {

moe_status moe_combine_backward_scaled(const moe_bf16* grad_out, const moe_bf16* o_save,
                                       const moe_layout* L, int32_t H, moe_bf16* g_o, float* grad_w,
                                       moe_stream_t stream) {
  return combine_backward_impl("moe_combine_backward_scaled", grad_out, o_save, L, H, g_o, grad_w, stream,
                               true);
}

moe_status moe_grouped_experts_backward_scaled(const moe_bf16* g_o, const moe_bf16* x_disp,
                                               const moe_bf16* h, const moe_bf16* gu_save,
                                               const moe_layout* L, int32_t H, int32_t I,
                                               const moe_bf16* W1, const moe_bf16* W2,
                                               moe_bf16* grad_x_disp, float* dW1, float* dW2,
                                               void* workspace, moe_stream_t stream) {
  return experts_backward_impl("moe_grouped_experts_backward_scaled", g_o, x_disp, h, gu_save, L, H, I, W1,
                               W2, grad_x_disp, dW1, dW2, workspace, stream, true);
}

moe_status moe_combine_backward(const moe_bf16* grad_out, const moe_bf16* o_save,
                                const moe_layout* L, int32_t H, moe_bf16* grad_y, float* grad_w,
                                moe_stream_t stream) {
  return combine_backward_impl("moe_combine_backward", grad_out, o_save, L, H, grad_y, grad_w, stream,
                               false);
}


moe_status moe_dispatch_backward(const moe_bf16* grad_x_disp, const float* grad_w,
                                 const moe_layout* L, int32_t H, moe_bf16* grad_x,
                                 float* grad_probs, moe_stream_t stream) {
  moe_status st = check_layout(L);
  if (st != MOE_OK) return st;
  if ((st = check_hidden(H)) != MOE_OK) return st;
  MOE_REQUIRE(L->T == 0 || (grad_x_disp && grad_x), MOE_ERR_INVALID_ARG,
              "moe_dispatch_backward: NULL pointer");
  MOE_REQUIRE(aligned16(grad_x_disp) && aligned16(grad_x) && aligned16(grad_probs),
              MOE_ERR_INVALID_ARG, "moe_dispatch_backward: pointers must be 16-byte aligned");
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t err = launch_combine(grad_x_disp, *L, H, grad_x, grad_w, grad_probs, stream);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_dispatch_backward launch");
}

moe_status moe_router_topk(const float* logits, int32_t T, int32_t E, int32_t K, int64_t* topk_idx,
                           float* topk_probs, uint8_t* routing_map, float* probs,
                           int8_t* winner_slot, moe_stream_t stream) {
  moe_status st = check_routing_shape(T, K, E);
  if (st != MOE_OK) return st;
  MOE_REQUIRE(T == 0 || (logits && topk_idx && topk_probs), MOE_ERR_INVALID_ARG,
              "moe_router_topk: NULL logits or top-k output");
  const bool mh = routing_map || probs || winner_slot;
  MOE_REQUIRE(!mh || (routing_map && probs && winner_slot), MOE_ERR_INVALID_ARG,
              "moe_router_topk: give all three multihot outputs or none");
  MOE_REQUIRE(aligned16(routing_map) && aligned16(probs) && aligned16(winner_slot),
              MOE_ERR_INVALID_ARG, "moe_router_topk: multihot outputs must be 16-byte aligned");
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t err = launch_router_topk(logits, T, K, E, topk_idx, topk_probs,
                                       mh ? routing_map : nullptr, probs, winner_slot, stream);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_router_topk launch");
}

moe_status moe_router_topk_backward(const float* grad_topk_probs, const float* topk_probs,
                                    const int64_t* topk_idx, int32_t T, int32_t E, int32_t K,
                                    float* grad_logits, moe_stream_t stream) {
  moe_status st = check_routing_shape(T, K, E);
  if (st != MOE_OK) return st;
  MOE_REQUIRE(T == 0 || (grad_topk_probs && topk_probs && topk_idx && grad_logits),
              MOE_ERR_INVALID_ARG, "moe_router_topk_backward: NULL pointer");
  MOE_REQUIRE(aligned16(grad_logits), MOE_ERR_INVALID_ARG,
              "moe_router_topk_backward: grad_logits must be 16-byte aligned");
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t err = launch_router_topk_backward(grad_topk_probs, topk_probs, topk_idx, T, K, E,
                                                grad_logits, stream);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_router_topk_backward launch");
}

moe_status moe_route_to_multihot_backward(const float* grad_probs, const int64_t* topk_idx,
                                          const int8_t* winner_slot, int32_t T, int32_t K,
                                          int32_t E, float* grad_topk_probs, moe_stream_t stream) {
  moe_status st = check_routing_shape(T, K, E);
  if (st != MOE_OK) return st;
  MOE_REQUIRE(T == 0 || (grad_probs && topk_idx && winner_slot && grad_topk_probs),
              MOE_ERR_INVALID_ARG, "moe_route_to_multihot_backward: NULL pointer");
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t err = launch_multihot_backward(grad_probs, topk_idx, winner_slot, T, K, E,
                                             grad_topk_probs, stream);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_route_to_multihot_backward launch");
}

moe_status moe_experts_backward_workspace_bytes(int64_t capacity, int32_t H, int32_t I,
                                                size_t* bytes) {
  MOE_REQUIRE(bytes != nullptr, MOE_ERR_INVALID_ARG, "bytes is NULL");
  MOE_REQUIRE(capacity >= 0 && H > 0 && I > 0, MOE_ERR_INVALID_ARG, "bad capacity / H / I");
  *bytes = experts_backward_workspace(capacity, H, I);
  return MOE_OK;
}

moe_status moe_grouped_experts_backward(const moe_bf16* grad_y, const moe_bf16* x_disp,
                                        const moe_bf16* h, const moe_bf16* gu_save,
                                        const moe_layout* L, int32_t H, int32_t I,
                                        const moe_bf16* W1, const moe_bf16* W2,
                                        moe_bf16* grad_x_disp, float* dW1, float* dW2,
                                        void* workspace, moe_stream_t stream) {
  return experts_backward_impl("moe_grouped_experts_backward", grad_y, x_disp, h, gu_save, L, H, I, W1, W2,
                               grad_x_disp, dW1, dW2, workspace, stream, false);
}

}  // extern "C"
