// ws_noalloc.cu -- ws_gemv_bf16_noalloc: the GEMV entry point for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they need a GEMV:
// code that runs while a stream is being captured into a CUDA graph (an
// allocation there would break or end the capture), serving loops that must
// not take an allocator lock or grow the memory footprint after start-up,
// and hosts that hand out only memory they allocated themselves.  The regular
// ws_gemv_bf16 asks such callers for a workspace whenever the schedule splits
// K; this variant instead keeps the split-K partial sums and tickets in a
// fixed array of device memory that belongs to the library.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes, so
// every GPU that loads the library holds it until the process exits.  Host
// code may not use the array's name as a device pointer (on the host it names
// a stand-in object); its device address is looked up once per device with
// cudaGetSymbolAddress, on the first call made with that device current, and
// passed to the kernel.  The looked-up address is kept until the process
// exits; a cudaDeviceReset while the library is loaded is not supported (the
// module, and with it the array, may be reloaded at another address).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "wsgemv.h"
#include "ws_common.cuh"

namespace ws {

constexpr size_t kNoAllocScratchBytes = 1u << 20;  // 1 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array for the current device (set up on
// first use with that device current), or null with the reason in `why`.
static void* noalloc_scratch_ptr(char* why, size_t why_len) {
  static std::mutex mu;
  static void* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    snprintf(why, why_len, "no current CUDA device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
      snprintf(why, why_len, "cudaGetSymbolAddress of the scratch array failed: %s",
               cudaGetErrorString(e));
      return nullptr;
    }
    cache[dev] = ptr;
  }
  return cache[dev];
}

}  // namespace ws

using namespace ws;

extern "C" ws_status ws_gemv_bf16_noalloc(const void* W, const void* x, float* y, int M, int K,
                                          int B, ws_stream_t stream) {
  if (M <= 0 || K <= 0 || K % 8 != 0 || B < 1 || B > kMaxBatch) {
    set_error("bad shape M=%d K=%d B=%d (need M>0, K>0, K%%8==0, 1<=B<=16)", M, K, B);
    return WS_ERR_SHAPE;
  }
  const void* ptrs[3] = {W, x, y};
  for (const void* q : ptrs) {
    if (!q) {
      set_error("null device pointer");
      return WS_ERR_ARG;
    }
    if ((uintptr_t)q & 15u) {
      set_error("device pointer %p is not 16-byte aligned", q);
      return WS_ERR_ALIGN;
    }
  }
  GemvParams p;
  init_gemv_params(p, K, B);
  p.nseg = 1;
  p.seg[0].W0 = static_cast<const uint16_t*>(W);
  p.seg[0].out = y;
  p.seg[0].M = M;
  p.x = x;
  p.x_dtype = DT_BF16;
  p.prologue = PRO_NONE;
  p.epilogue = EPI_F32;
  char why[256];
  if (!plan_gemv(p, 0, why, sizeof why)) {
    set_error("%s", why);
    return WS_ERR_SHAPE;
  }
  size_t off_tickets = 0, off_part = 0;
  const size_t need = workspace_layout(p, &off_tickets, &off_part, nullptr, nullptr, nullptr);
  if (need > kNoAllocScratchBytes) {
    set_error("M=%d K=%d B=%d needs %zu bytes of split-K scratch; the fixed scratch array "
              "holds %zu bytes (use ws_gemv_bf16 with a workspace)",
              M, K, B, need, kNoAllocScratchBytes);
    return WS_ERR_SHAPE;
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (need > 0) {
    void* scratch = noalloc_scratch_ptr(why, sizeof why);
    if (!scratch) {
      set_error("%s", why);
      return WS_ERR_CUDA;
    }
    if (!bind_workspace(p, scratch, kNoAllocScratchBytes)) {
      set_error("internal: scratch binding failed");
      return WS_ERR_ARG;
    }
    // The tickets must start at zero; the previous call left them zeroed
    // unless it failed part way, so clear them on the stream first.
    const cudaError_t e = cudaMemsetAsync(static_cast<char*>(scratch) + off_tickets, 0,
                                          (size_t)p.sc.RG * 4, st);
    if (e != cudaSuccess) {
      set_error("clearing the scratch tickets failed: %s", cudaGetErrorString(e));
      return WS_ERR_CUDA;
    }
  }
  const cudaError_t e = launch_gemv(p, st, tuning().launch_pdl != 0);
  if (e != cudaSuccess) {
    set_error("launch failed: %s", cudaGetErrorString(e));
    return WS_ERR_CUDA;
  }
  return WS_OK;
}
