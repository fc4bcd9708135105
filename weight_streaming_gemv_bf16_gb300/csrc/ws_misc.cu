// ws_misc.cu -- the library's small kernels: standalone RMSNorm, row argmax,
// the L2 prefetch kernel, roofline/latency probes and the bounded-wait test.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>

#include "wsgemv.h"
#include "ws_common.cuh"
#include "ws_device.cuh"

namespace ws {

// ---------------------------------------------------------------------------
// RMSNorm of [R][N] rows, one warp per row ("GPU Kernel Optimization",
// Architecture: mean square, rsqrt and weight multiply in one launch).  fp32
// arithmetic, one rounding to the storage type.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ void unpack8(const uint4 u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (DT == DT_F16) {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
      v[2 * j] = __low2float(h);
      v[2 * j + 1] = __high2float(h);
    } else {
      v[2 * j] = bf16lo(w[j]);
      v[2 * j + 1] = bf16hi(w[j]);
    }
  }
}

template <int DT>
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (DT == DT_F16) {
      const __half2 h = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
      w[j] = *reinterpret_cast<const uint32_t*>(&h);
    } else {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * j]));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * j + 1]));
      w[j] = lo | (hi << 16);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int DT>
__global__ void __launch_bounds__(256) k_rmsnorm(const uint16_t* __restrict__ x,
                                                 const uint16_t* __restrict__ gamma,
                                                 uint16_t* __restrict__ y, int R, int N,
                                                 float eps) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= R) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)warp * N);
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  uint4* yr = reinterpret_cast<uint4*>(y + (size_t)warp * N);
  const int nch = N >> 3;
  float ss = 0.f;
  for (int c = lane; c < nch; c += 32) {
    float v[8];
    unpack8<DT>(xr[c], v);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(v[j], v[j], ss);
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / (float)N + eps);
  for (int c = lane; c < nch; c += 32) {
    float v[8], g[8];
    unpack8<DT>(xr[c], v);
    unpack8<DT>(g4[c], g);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = v[j] * r * g[j];
    yr[c] = pack8<DT>(v);
  }
}

// ---------------------------------------------------------------------------
// Row argmax: CB CTAs per row scan column ranges, write (value, index)
// partials, and the last CTA of the row (ticket) combines them.  Ties go to
// the lower index, so the order the CTAs finish in does not matter.
// ---------------------------------------------------------------------------
static int argmax_cols_per_row_blocks(int cols) {
  int cb = (cols + 8191) / 8192;
  if (cb < 1) cb = 1;
  if (cb > 64) cb = 64;
  return cb;
}

__global__ void __launch_bounds__(256) k_argmax_rows(const float* __restrict__ v, int32_t* idx,
                                                     int rows, int cols, float* pv, int* pi,
                                                     unsigned* tickets) {
  __shared__ float sv[8];
  __shared__ int si[8];
  __shared__ int last;
  const int row = blockIdx.y;
  const int cb = blockIdx.x, CB = gridDim.x;
  const int c0 = (int)((long long)cb * cols / CB);
  const int c1 = (int)((long long)(cb + 1) * cols / CB);
  const float* vr = v + (size_t)row * cols;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int c = c0 + threadIdx.x; c < c1; c += blockDim.x) {
    const float x = vr[c];
    if (arg_better(x, c, bv, bi)) {
      bv = x;
      bi = c;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (arg_better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (arg_better(sv[w], si[w], bv, bi)) {
        bv = sv[w];
        bi = si[w];
      }
    pv[(size_t)row * CB + cb] = bv;
    pi[(size_t)row * CB + cb] = bi;
    __threadfence();
    const unsigned old = atomicAdd(&tickets[row], 1u);
    last = old == (unsigned)(CB - 1);
    if (last) atomicExch(&tickets[row], 0u);
  }
  __syncthreads();
  if (last && threadIdx.x == 0) {
    __threadfence();
    float fv = -INFINITY;
    int fi = 0x7fffffff;
    for (int c = 0; c < CB; ++c) {
      const float x = __ldcg(&pv[(size_t)row * CB + c]);
      const int xi = __ldcg(&pi[(size_t)row * CB + c]);
      if (arg_better(x, xi, fv, fi)) {
        fv = x;
        fi = xi;
      }
    }
    idx[row] = fi;
  }
}

// ---------------------------------------------------------------------------
// L2 prefetch ("Making small PyTorch ops faster on a laptop GPU", "Prefetching
// the next layer while this one runs"): grid-stride over the range, one
// prefetch every `stride` bytes, never a write.  The bulk mode asks the TMA
// unit to prefetch `stride`-byte chunks into L2.
// ---------------------------------------------------------------------------
__global__ void k_l2_prefetch(const char* __restrict__ p, long long bytes, int stride, int mode) {
  const long long nthr = (long long)gridDim.x * blockDim.x;
  const long long step = nthr * stride;
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (mode == 3) {
    for (long long off = t * stride; off < bytes; off += step) {
      long long n = bytes - off < stride ? bytes - off : stride;
      n &= ~15ll;
      if (n > 0) bulk_prefetch_l2(p + off, (uint32_t)n);
    }
  } else if (mode == 2) {
    for (long long off = t * stride; off < bytes; off += step) prefetch_l2_evict_last(p + off);
  } else {
    for (long long off = t * stride; off < bytes; off += step) prefetch_l2(p + off);
  }
}

// ---------------------------------------------------------------------------
// Probes: a read-only streaming kernel (read roofline) and an empty / one-load
// kernel (launch-latency floor).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(512) k_read_probe(const uint4* __restrict__ p, long long n16,
                                                    uint32_t* sink) {
  const long long nthr = (long long)gridDim.x * blockDim.x;
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  constexpr int U = 8;
  for (; i + (U - 1) * nthr < n16; i += U * nthr) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = ld_stream(p + i + u * nthr);
#pragma unroll
    for (int u = 0; u < U; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += nthr) {
    const uint4 v = ld_stream(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ uint32_t s[16];
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t a = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) a ^= s[w];
    sink[blockIdx.x] = a;
  }
}

__global__ void k_empty_probe(int touch, const uint32_t* ptr, uint32_t* sink) {
  if (touch && threadIdx.x == 0) sink[0] = __ldcg(ptr);
}

__global__ void k_test_bounded_wait(unsigned long long timeout_ns, int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Nothing ever arrives: phase 0 never completes, so the wait must run out.
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, timeout_ns) && err)
    atomicExch(err, DERR_TIMEOUT);
}

// Word copies between device-accessible buffers, for a step's inputs read
// from pinned host memory and its result written back (the host buffers
// reached through their device mapping): up to two (dst, src, bytes) pairs,
// bytes a multiple of 4, 4-byte aligned.  SMs move the few kilobytes of a
// decode step's inputs with one launch instead of a copy-engine transfer
// per buffer.
// Launched as a programmatic dependent of the kernel before it, it waits
// for that kernel's results before copying; the kernel after it may start
// (and stream its weights) at once, and waits for the copy before it reads.
__global__ void __launch_bounds__(256) k_copy_words(uint32_t* d0, const uint32_t* s0, long long n0,
                                                    uint32_t* d1, const uint32_t* s1, long long n1) {
  pdl_launch_dependents();
  pdl_wait();
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = t; i < n0; i += stride) d0[i] = s0[i];
  for (long long i = t; i < n1; i += stride) d1[i] = s1[i];
}

cudaError_t launch_copy_words(void* d0, const void* s0, size_t b0, void* d1, const void* s1,
                              size_t b1, cudaStream_t stream, bool pdl) {
  const long long n0 = (long long)(b0 / 4), n1 = (long long)(b1 / 4);
  const long long n = n0 > n1 ? n0 : n1;
  int blocks = (int)((n + 255) / 256);
  if (blocks < 1) blocks = 1;
  if (blocks > 148) blocks = 148;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_copy_words, static_cast<uint32_t*>(d0),
                            static_cast<const uint32_t*>(s0), n0, static_cast<uint32_t*>(d1),
                            static_cast<const uint32_t*>(s1), n1);
}

size_t argmax_rows_workspace(int rows, int cols) {
  if (rows <= 0 || cols <= 0) return 0;
  const size_t cb = (size_t)argmax_cols_per_row_blocks(cols);
  const size_t a = ((size_t)rows * cb * 4 + 255) / 256 * 256;
  const size_t t = ((size_t)rows * 4 + 255) / 256 * 256;
  return 2 * a + t;
}

}  // namespace ws

using namespace ws;

static bool al16(const void* q) { return ((uintptr_t)q & 15u) == 0; }

static ws_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("launch failed: %s", cudaGetErrorString(e));
    return WS_ERR_CUDA;
  }
  return WS_OK;
}

extern "C" {

ws_status ws_rmsnorm(const void* x, const void* gamma, void* y, int R, int N, int dtype, float eps,
                     ws_stream_t stream) {
  if (R <= 0 || N <= 0 || N % 8 != 0) {
    set_error("bad shape R=%d N=%d (need R>0, N>0, N%%8==0)", R, N);
    return WS_ERR_SHAPE;
  }
  if (!x || !gamma || !y) {
    set_error("null device pointer");
    return WS_ERR_ARG;
  }
  if (!al16(x) || !al16(gamma) || !al16(y)) {
    set_error("device pointers must be 16-byte aligned");
    return WS_ERR_ALIGN;
  }
  const int blocks = (R + 7) / 8;
  cudaStream_t st = (cudaStream_t)stream;
  const uint16_t* xx = static_cast<const uint16_t*>(x);
  const uint16_t* gg = static_cast<const uint16_t*>(gamma);
  uint16_t* yy = static_cast<uint16_t*>(y);
  if (dtype == WS_DTYPE_F16) {
    k_rmsnorm<DT_F16><<<blocks, 256, 0, st>>>(xx, gg, yy, R, N, eps);
  } else if (dtype == WS_DTYPE_BF16) {
    k_rmsnorm<DT_BF16><<<blocks, 256, 0, st>>>(xx, gg, yy, R, N, eps);
  } else {
    set_error("dtype must be WS_DTYPE_F16 or WS_DTYPE_BF16");
    return WS_ERR_ARG;
  }
  return launch_status();
}

ws_status ws_argmax_rows(const float* logits, int32_t* idx, int rows, int cols, void* workspace,
                         size_t workspace_bytes, ws_stream_t stream) {
  if (rows <= 0 || cols <= 0 || rows > 65535) {
    set_error("bad shape rows=%d cols=%d", rows, cols);
    return WS_ERR_SHAPE;
  }
  if (!logits || !idx || !workspace) {
    set_error("null device pointer");
    return WS_ERR_ARG;
  }
  if (!al16(workspace)) {
    set_error("workspace must be 16-byte aligned");
    return WS_ERR_ALIGN;
  }
  const size_t need = argmax_rows_workspace(rows, cols);
  if (workspace_bytes < need) {
    set_error("workspace too small: need %zu bytes, got %zu", need, workspace_bytes);
    return WS_ERR_ARG;
  }
  const int cb = argmax_cols_per_row_blocks(cols);
  const size_t a = ((size_t)rows * cb * 4 + 255) / 256 * 256;
  char* base = static_cast<char*>(workspace);
  float* pv = reinterpret_cast<float*>(base);
  int* pi = reinterpret_cast<int*>(base + a);
  unsigned* tickets = reinterpret_cast<unsigned*>(base + 2 * a);
  k_argmax_rows<<<dim3(cb, rows), 256, 0, (cudaStream_t)stream>>>(logits, idx, rows, cols, pv,
                                                                   pi, tickets);
  return launch_status();
}

ws_status ws_l2_prefetch(const void* ptr, size_t bytes, ws_prefetch_plan plan,
                         ws_stream_t stream) {
  if (plan.mode == WS_PREFETCH_NONE || bytes == 0) return WS_OK;
  if (!ptr) {
    set_error("null pointer");
    return WS_ERR_ARG;
  }
  if (plan.mode < WS_PREFETCH_L2 || plan.mode > WS_PREFETCH_BULK || plan.blocks <= 0 ||
      plan.threads <= 0 || plan.threads > 1024 || plan.stride_bytes <= 0) {
    set_error("bad prefetch plan (mode %d, blocks %d, threads %d, stride %d)", plan.mode,
              plan.blocks, plan.threads, plan.stride_bytes);
    return WS_ERR_ARG;
  }
  if (plan.mode == WS_PREFETCH_BULK && (!al16(ptr) || plan.stride_bytes % 16 != 0)) {
    set_error("bulk prefetch needs a 16-byte aligned pointer and stride");
    return WS_ERR_ALIGN;
  }
  k_l2_prefetch<<<plan.blocks, plan.threads, 0, (cudaStream_t)stream>>>(
      static_cast<const char*>(ptr), (long long)bytes, plan.stride_bytes, plan.mode);
  return launch_status();
}

ws_status ws_read_probe(const void* ptr, size_t bytes, int blocks, uint32_t* sink,
                        ws_stream_t stream) {
  if (!ptr || !sink || blocks <= 0 || bytes < 16) {
    set_error("bad read-probe arguments");
    return WS_ERR_ARG;
  }
  if (!al16(ptr)) {
    set_error("read probe needs a 16-byte aligned pointer");
    return WS_ERR_ALIGN;
  }
  k_read_probe<<<blocks, 512, 0, (cudaStream_t)stream>>>(static_cast<const uint4*>(ptr),
                                                          (long long)(bytes / 16), sink);
  return launch_status();
}

ws_status ws_empty_probe(int touch, const uint32_t* ptr, uint32_t* sink, ws_stream_t stream) {
  if (touch && (!ptr || !sink)) {
    set_error("one-load probe needs ptr and sink");
    return WS_ERR_ARG;
  }
  k_empty_probe<<<1, 32, 0, (cudaStream_t)stream>>>(touch, ptr, sink);
  return launch_status();
}

ws_status ws_test_bounded_wait(unsigned long long timeout_ns, ws_stream_t stream) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) {
    set_error("timeout must be in (0, 10 s]");
    return WS_ERR_ARG;
  }
  int* err = device_error_ptr();
  if (!err) {
    set_error("device error flag unavailable");
    return WS_ERR_CUDA;
  }
  k_test_bounded_wait<<<1, 32, 0, (cudaStream_t)stream>>>(timeout_ns, err);
  return launch_status();
}

}  // extern "C"
