// ws_attention.cu -- decode attention over a key-value cache, one new token
// per batch row ("Making small PyTorch ops faster on a laptop GPU", "A full
// decode step is a different story": append the new key and value, an FP32
// softmax, the cache split across blocks, the last block to finish merging
// the partial results; "One Token, Kernel by Kernel", "The fix: Part 10's
// split-KV kernel": the (batch, head, slot, dimension) cache layout, the
// valid length read on the GPU at run time so that a CUDA graph can be
// replayed, one key-value head read once for all of its query heads).
//
// Design for GB300: one CTA of 128 threads per (chunk of 128 cached slots,
// key-value head, batch row).  Scores: thread t takes slot t of the chunk,
// reads its key row (256 bytes) once and forms the dot products with the G
// query heads of the group (queries in shared memory).  Softmax over the
// chunk in fp32 (max and sum over the CTA).  Values: thread t takes dimension
// t and walks the chunk's slots (each slot's 256-byte value row read by the
// CTA in one coalesced pass), accumulating G outputs.  Every chunk writes
// (acc, max, sum) for its G heads; the last chunk of the (row, head) to
// finish (an atomic ticket, reset for the next replay) rescales and adds
// them in chunk order.  Chunks past the valid length exit at once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "wsgemv.h"
#include "ws_common.cuh"
#include "ws_device.cuh"

namespace ws {

constexpr int kAttnChunk = 128;  // cached slots per CTA
constexpr int kAttnDim = 128;    // head dimension: one thread per dimension
constexpr int kDerrBadPos = 2;   // device error flag: a position outside the cache

struct AttnParams {
  const float* q;      // [B][nh * 128]
  const float* k_new;  // [B][nkv * 128]
  const float* v_new;
  uint16_t* k_cache;   // bf16 [B][nkv][S][128]
  uint16_t* v_cache;
  const int* pos;      // [B]: slot of the new token
  float* out_f32;      // optional [B][nh * 128]
  uint16_t* out_bf16;  // optional bf16 [B][nh * 128]
  int nh, nkv, S;
  float scale;         // 1 / sqrt(128)
  float* part;         // [B][nkv][S / 128][G][128 + 2]: acc, max, sum
  unsigned* tickets;   // [B][nkv]
  int* err;
};

__device__ __forceinline__ uint16_t to_bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

template <int G>
__global__ void __launch_bounds__(kAttnChunk) k_decode_attention(const __grid_constant__ AttnParams a) {
  const int chunk = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int pos = a.pos[b];
  if (pos < 0 || pos >= a.S) {  // no access outside the cache
    if (t == 0 && chunk == 0) atomicExch(a.err, kDerrBadPos);
    return;
  }
  const int n_valid = pos + 1;
  const int nchunks = (n_valid + kAttnChunk - 1) / kAttnChunk;
  if (chunk >= nchunks) return;

  __shared__ float qs[G][kAttnDim];
  __shared__ float ps[kAttnChunk][G];
  __shared__ float red[kAttnChunk / 32][G];
  __shared__ float mx[G], sm[G];
  __shared__ int last;

  const size_t row0 = (size_t)(b * a.nkv + g) * a.S;  // first slot of this head's cache
  const size_t kvn = (size_t)(b * a.nkv + g) * kAttnDim;
  // the new token's key and value go to slot pos (the chunk that holds it)
  if (pos / kAttnChunk == chunk) {
    a.k_cache[(row0 + pos) * kAttnDim + t] = to_bf16_bits(a.k_new[kvn + t]);
    a.v_cache[(row0 + pos) * kAttnDim + t] = to_bf16_bits(a.v_new[kvn + t]);
  }
#pragma unroll
  for (int h = 0; h < G; ++h) qs[h][t] = a.q[(size_t)b * a.nh * kAttnDim + (g * G + h) * kAttnDim + t];
  __syncthreads();  // queries, and the appended row, visible to the CTA

  // scores: thread t takes slot j
  const int j = chunk * kAttnChunk + t;
  float s[G];
#pragma unroll
  for (int h = 0; h < G; ++h) s[h] = 0.f;
  if (j <= pos) {
    const uint4* kr = reinterpret_cast<const uint4*>(a.k_cache + (row0 + j) * kAttnDim);
#pragma unroll 4
    for (int c = 0; c < kAttnDim / 8; ++c) {
      const uint4 u = kr[c];  // coherent load: slot pos may have been written above
      const float kv[8] = {bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y),
                           bf16lo(u.z), bf16hi(u.z), bf16lo(u.w), bf16hi(u.w)};
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) s[h] = fmaf(kv[e], qs[h][c * 8 + e], s[h]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] *= a.scale;
  } else {
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] = -INFINITY;
  }
  // the chunk's maximum and sum of exponentials per head
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float m = s[h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp][h] = m;
  }
  __syncthreads();
  if (t < G) {
    float m = red[0][t];
#pragma unroll
    for (int w = 1; w < kAttnChunk / 32; ++w) m = fmaxf(m, red[w][t]);
    mx[t] = m;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float p = j <= pos ? expf(s[h] - mx[h]) : 0.f;
    ps[t][h] = p;
    const float w = warp_sum(p);
    if (lane == 0) red[warp][h] = w;
  }
  __syncthreads();
  if (t < G) {
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnChunk / 32; ++w) l += red[w][t];
    sm[t] = l;
  }

  // values: thread t takes dimension t over the chunk's valid slots
  const int nj = min(kAttnChunk, n_valid - chunk * kAttnChunk);
  const uint16_t* vr = a.v_cache + (row0 + (size_t)chunk * kAttnChunk) * kAttnDim + t;
  float acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll 4
  for (int i = 0; i < nj; ++i) {
    const float v = __uint_as_float((uint32_t)vr[(size_t)i * kAttnDim] << 16);
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = fmaf(ps[i][h], v, acc[h]);
  }
  __syncthreads();  // sm written

  // this chunk's partials, then the ticket of the (row, head)
  const int maxc = a.S / kAttnChunk;
  float* pp = a.part + ((size_t)(b * a.nkv + g) * maxc + chunk) * G * (kAttnDim + 2);
#pragma unroll
  for (int h = 0; h < G; ++h) pp[h * (kAttnDim + 2) + t] = acc[h];
  if (t < G) {
    pp[t * (kAttnDim + 2) + kAttnDim] = mx[t];
    pp[t * (kAttnDim + 2) + kAttnDim + 1] = sm[t];
  }
  __threadfence();
  __syncthreads();
  if (t == 0) {
    unsigned* tk = a.tickets + b * a.nkv + g;
    const unsigned old = atomicAdd(tk, 1u);
    last = old == (unsigned)(nchunks - 1);
    if (last) atomicExch(tk, 0u);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();

  // merge in chunk order: out = sum_c e^(m_c - M) acc_c / sum_c e^(m_c - M) l_c
  const float* base = a.part + (size_t)(b * a.nkv + g) * maxc * G * (kAttnDim + 2);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
    for (int c = 0; c < nchunks; ++c)
      M = fmaxf(M, __ldcg(base + ((size_t)c * G + h) * (kAttnDim + 2) + kAttnDim));
    float L = 0.f, O = 0.f;
    for (int c = 0; c < nchunks; ++c) {
      const float* pc = base + ((size_t)c * G + h) * (kAttnDim + 2);
      const float w = expf(__ldcg(pc + kAttnDim) - M);
      L = fmaf(w, __ldcg(pc + kAttnDim + 1), L);
      O = fmaf(w, __ldcg(pc + t), O);
    }
    const float o = O / L;
    const size_t oi = (size_t)b * a.nh * kAttnDim + (g * G + h) * kAttnDim + t;
    if (a.out_f32) a.out_f32[oi] = o;
    if (a.out_bf16) a.out_bf16[oi] = to_bf16_bits(o);
  }
}

typedef void (*AttnKernel)(const AttnParams);

static AttnKernel pick_attention(int G) {
  switch (G) {
    case 1: return k_decode_attention<1>;
    case 2: return k_decode_attention<2>;
    case 4: return k_decode_attention<4>;
    case 6: return k_decode_attention<6>;
    case 8: return k_decode_attention<8>;
    default: return nullptr;
  }
}

static size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Workspace layout: tickets [B][nkv] (256-byte aligned), then the partials.
static size_t attention_workspace(int B, int nh, int nkv, int s_max, size_t* off_part) {
  const int G = nh / nkv;
  const size_t tk = align256((size_t)B * nkv * 4);
  if (off_part) *off_part = tk;
  return tk + (size_t)B * nkv * (s_max / kAttnChunk) * G * (kAttnDim + 2) * 4;
}

}  // namespace ws

using namespace ws;

extern "C" {

size_t ws_attention_workspace_bytes(int B, int n_heads, int n_kv_heads, int head_dim, int s_max) {
  if (B < 1 || B > kMaxBatch || n_kv_heads < 1 || n_heads % n_kv_heads || head_dim != kAttnDim ||
      s_max < kAttnChunk || s_max % kAttnChunk)
    return 0;
  return attention_workspace(B, n_heads, n_kv_heads, s_max, nullptr);
}

ws_status ws_decode_attention(const float* q, const float* k_new, const float* v_new,
                              void* k_cache, void* v_cache, const int32_t* pos, float* out_f32,
                              void* out_bf16, int B, int n_heads, int n_kv_heads, int head_dim,
                              int s_max, void* workspace, size_t workspace_bytes,
                              ws_stream_t stream) {
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !pos || (!out_f32 && !out_bf16) ||
      !workspace) {
    set_error("null argument");
    return WS_ERR_ARG;
  }
  if (B < 1 || B > kMaxBatch || n_kv_heads < 1 || n_heads % n_kv_heads || head_dim != kAttnDim ||
      s_max < kAttnChunk || s_max % kAttnChunk) {
    set_error("decode attention: B 1..%d, head_dim %d, n_heads a multiple of n_kv_heads, "
              "s_max a multiple of %d", kMaxBatch, kAttnDim, kAttnChunk);
    return WS_ERR_SHAPE;
  }
  AttnKernel k = pick_attention(n_heads / n_kv_heads);
  if (!k) {
    set_error("decode attention: %d query heads per key-value head (1, 2, 4, 6 or 8)",
              n_heads / n_kv_heads);
    return WS_ERR_SHAPE;
  }
  if (((uintptr_t)k_cache & 15u) || ((uintptr_t)v_cache & 15u)) {
    set_error("decode attention: caches must be 16-byte aligned");
    return WS_ERR_ALIGN;
  }
  size_t off_part = 0;
  const size_t need = attention_workspace(B, n_heads, n_kv_heads, s_max, &off_part);
  if (workspace_bytes < need) {
    set_error("workspace too small: need %zu bytes, got %zu", need, workspace_bytes);
    return WS_ERR_ARG;
  }
  cudaStream_t st = (cudaStream_t)stream;
  AttnParams a;
  memset(&a, 0, sizeof a);
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = static_cast<uint16_t*>(k_cache);
  a.v_cache = static_cast<uint16_t*>(v_cache);
  a.pos = pos;
  a.out_f32 = out_f32;
  a.out_bf16 = static_cast<uint16_t*>(out_bf16);
  a.nh = n_heads;
  a.nkv = n_kv_heads;
  a.S = s_max;
  a.scale = 1.0f / sqrtf((float)kAttnDim);
  a.tickets = static_cast<unsigned*>(workspace);
  a.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + off_part);
  a.err = device_error_ptr();
  // the tickets are zero on entry (a zero-filled workspace; the last chunk of
  // every (row, head) resets its own ticket, rows with a bad position take none)
  const dim3 grid(s_max / kAttnChunk, n_kv_heads, B);
  k<<<grid, kAttnChunk, 0, st>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("launch failed: %s", cudaGetErrorString(e));
    return WS_ERR_CUDA;
  }
  return WS_OK;
}

}  // extern "C"
