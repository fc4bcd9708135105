// ws_attention.cu -- decode attention over a key-value cache, one new token
// per batch row ("Making small PyTorch ops faster on a laptop GPU", "A full
// decode step is a different story": append the new key and value, an FP32
// softmax, the cache split across blocks, the last block to finish merging
// the partial results; "One Token, Kernel by Kernel", "The fix: Part 10's
// split-KV kernel": the (batch, head, slot, dimension) cache layout, the
// valid length read on the GPU at run time so that a CUDA graph can be
// replayed, one key-value head read once for all of its query heads).
//
// Design for GB300: one CTA of 256 threads per (chunk of 128 cached slots,
// key-value head, batch row).  The chunk's key and value rows (32 KB each,
// contiguous in the cache) land in shared memory by two bulk async copies on
// one mbarrier, so a CTA has its whole chunk in flight at once; the new
// token's row is written to the cache and to shared memory by the CTA's
// threads (the copies stop short of it).  Scores: two threads per slot (one
// per half of the head dimension, in different warps), reading the key row
// by 16-byte columns in a per-slot rotated order and the queries from a
// padded copy, so neither read has bank conflicts.  Softmax over the chunk in
// fp32.  Values: warp w takes slots 16w..16w+15, lane l dimensions 4l..4l+3,
// all G heads; the eight warps' sums are added in shared memory.  A chunk
// writes (acc, max, sum) per head; the last chunk of each group of 16 to
// finish (an atomic ticket, reset by that chunk for the next replay) merges
// the group in chunk order, and with more than one group the last group
// merges the groups.  A (row, head) with a single chunk writes its output
// directly.  Chunks past the valid length exit at once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "wsgemv.h"
#include "ws_common.cuh"
#include "ws_device.cuh"

namespace ws {

constexpr int kAttnChunk = 128;           // cached slots per CTA
constexpr int kAttnDim = 128;             // head dimension
constexpr int kAttnThreads = 256;
constexpr int kAttnGroup = 16;            // chunks merged by one first-level merge
constexpr int kPartStride = kAttnDim + 2;  // one partial result: acc[128], max, sum
constexpr int kQPad = kAttnDim + kAttnDim / 8;  // padded query row: 16 bytes after every 128
constexpr int kDerrBadPos = 2;            // device error flag: a position outside the cache

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
  float* part0;        // [B][nkv][S / 128][G][130]: per chunk
  float* part1;        // [B][nkv][groups][G][130]: per group of 16 chunks
  unsigned* tick0;     // [B][nkv][groups]
  unsigned* tick1;     // [B][nkv]
  int* err;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ uint16_t to_bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

template <int G>
struct AttnSmem {
  static constexpr int kKV = kAttnChunk * kAttnDim * 2;  // bytes of one chunk of keys
  static constexpr int kQ = G * kQPad * 4;
  static constexpr int kS = 2 * G * kAttnChunk * 4;      // half-dimension scores, then p
  static constexpr int bytes = 2 * kKV + kQ + kS;
};

// Online merge of n partial results (acc, max, sum) in entry order for the
// heads hp, hp + 2, ... and dimension d: M = max m_c, L = sum e^(m_c - M) l_c,
// O = sum e^(m_c - M) acc_c.
template <int G>
__device__ __forceinline__ void merge_partials(const float* src, int n, int d, int hp,
                                               float (&O)[(G + 1) / 2], float (&M)[(G + 1) / 2],
                                               float (&L)[(G + 1) / 2]) {
#pragma unroll
  for (int i = 0; i < (G + 1) / 2; ++i) {
    const int h = hp + 2 * i;
    float m_run = -INFINITY, l_run = 0.f, o_run = 0.f;
    if (h < G) {
#pragma unroll 8
      for (int c = 0; c < n; ++c) {
        const float* e = src + ((size_t)c * G + h) * kPartStride;
        const float m = __ldcg(e + kAttnDim), l = __ldcg(e + kAttnDim + 1), x = __ldcg(e + d);
        const float mn = fmaxf(m_run, m);
        const float r = expf(m_run - mn), w = expf(m - mn);
        l_run = fmaf(l_run, r, w * l);
        o_run = fmaf(o_run, r, w * x);
        m_run = mn;
      }
    }
    O[i] = o_run;
    M[i] = m_run;
    L[i] = l_run;
  }
}

template <int G>
__device__ __forceinline__ void write_output(const AttnParams& a, int b, int g, int d, int hp,
                                             const float (&O)[(G + 1) / 2],
                                             const float (&L)[(G + 1) / 2]) {
#pragma unroll
  for (int i = 0; i < (G + 1) / 2; ++i) {
    const int h = hp + 2 * i;
    if (h >= G) break;
    const float o = O[i] / L[i];
    const size_t oi = ((size_t)b * a.nh + g * G + h) * kAttnDim + d;
    if (a.out_f32) a.out_f32[oi] = o;
    if (a.out_bf16) a.out_bf16[oi] = to_bf16_bits(o);
  }
}

template <int G>
__device__ __forceinline__ void write_partial(float* dst, int d, int hp,
                                              const float (&O)[(G + 1) / 2],
                                              const float (&M)[(G + 1) / 2],
                                              const float (&L)[(G + 1) / 2]) {
#pragma unroll
  for (int i = 0; i < (G + 1) / 2; ++i) {
    const int h = hp + 2 * i;
    if (h >= G) break;
    dst[h * kPartStride + d] = O[i];
    if (d == 0) {
      dst[h * kPartStride + kAttnDim] = M[i];
      dst[h * kPartStride + kAttnDim + 1] = L[i];
    }
  }
}

template <int G>
__global__ void __launch_bounds__(kAttnThreads)
    k_decode_attention(const __grid_constant__ AttnParams a) {
  constexpr int HPT = (G + 1) / 2;  // heads per thread in the combine and merge steps
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

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* Ks = smem;
  unsigned char* Vs = smem + AttnSmem<G>::kKV;
  float* qs = reinterpret_cast<float*>(smem + 2 * AttnSmem<G>::kKV);
  float* sp = reinterpret_cast<float*>(smem + 2 * AttnSmem<G>::kKV + AttnSmem<G>::kQ);
  __shared__ uint64_t bar;
  __shared__ float red[kAttnThreads / 32][G];
  __shared__ float mx[G], sm[G];
  __shared__ int last;

  const int c0 = chunk * kAttnChunk;
  const int nv = min(kAttnChunk, n_valid - c0);  // valid slots of this chunk
  const int nk = min(kAttnChunk, pos - c0);      // of them already cached (all but pos)
  const size_t row0 = (size_t)(b * a.nkv + g) * a.S + c0;  // first slot of the chunk
  if (t == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (nk > 0) {
      const uint64_t pol = l2_policy_evict_normal();
      mbar_arrive_expect_tx(&bar, 2u * nk * kAttnDim * 2);
      bulk_copy_g2s(Ks, a.k_cache + row0 * kAttnDim, nk * kAttnDim * 2, &bar, pol);
      bulk_copy_g2s(Vs, a.v_cache + row0 * kAttnDim, nk * kAttnDim * 2, &bar, pol);
    }
  }
  // the new token's key and value: slot pos of the cache and row nk of the chunk
  if (nk < kAttnChunk) {
    const int d = t & (kAttnDim - 1);
    const bool is_v = t >= kAttnDim;
    const float* src = is_v ? a.v_new : a.k_new;
    const uint16_t u = to_bf16_bits(src[(size_t)(b * a.nkv + g) * kAttnDim + d]);
    (is_v ? a.v_cache : a.k_cache)[(row0 + nk) * kAttnDim + d] = u;
    reinterpret_cast<uint16_t*>(is_v ? Vs : Ks)[nk * kAttnDim + d] = u;
  }
  for (int i = t; i < G * kAttnDim; i += kAttnThreads) {
    const int h = i / kAttnDim, d = i % kAttnDim;
    qs[h * kQPad + d + (d / 32) * 4] = a.q[((size_t)b * a.nh + g * G + h) * kAttnDim + d];
  }
  __syncthreads();  // mbarrier initialised, queries and the new row visible
  bool ok = nk == 0 || mbar_wait_bounded(&bar, 0, a.timeout_ns);
  if (__syncthreads_or(!ok)) {
    if (t == 0) {
      atomicExch(a.err, (int)DERR_TIMEOUT);
      mbar_wait_bounded(&bar, 0, a.timeout_ns);  // no copy may land after the CTA exits
    }
    return;
  }

  // scores: warp w, lane l -> slot 32 (w % 4) + l, dimension half w / 4
  {
    const int p = warp >> 2, s = ((warp & 3) << 5) | lane;
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.f;
    if (s < nv) {
      const unsigned char* kr = Ks + s * kAttnDim * 2;
      const float4* q4 = reinterpret_cast<const float4*>(qs);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int col = p * 8 + ((c + s) & 7);  // 16-byte column: 8 dimensions
        const uint4 u = *reinterpret_cast<const uint4*>(kr + col * 16);
        const float kv[8] = {bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y),
                             bf16lo(u.z), bf16hi(u.z), bf16lo(u.w), bf16hi(u.w)};
        const int qi = (col * 8 + (col >> 2) * 4) >> 2;  // padded float4 index
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 qa = q4[h * (kQPad / 4) + qi], qb = q4[h * (kQPad / 4) + qi + 1];
          acc[h] = fmaf(kv[0], qa.x, acc[h]);
          acc[h] = fmaf(kv[1], qa.y, acc[h]);
          acc[h] = fmaf(kv[2], qa.z, acc[h]);
          acc[h] = fmaf(kv[3], qa.w, acc[h]);
          acc[h] = fmaf(kv[4], qb.x, acc[h]);
          acc[h] = fmaf(kv[5], qb.y, acc[h]);
          acc[h] = fmaf(kv[6], qb.z, acc[h]);
          acc[h] = fmaf(kv[7], qb.w, acc[h]);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) sp[(p * G + h) * kAttnChunk + s] = acc[h];
  }
  __syncthreads();

  // softmax over the chunk: warps 0..3, thread t = slot t
  float sc[G];
  if (t < kAttnChunk) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      sc[h] = t < nv ? (sp[h * kAttnChunk + t] + sp[(G + h) * kAttnChunk + t]) * a.scale
                     : -INFINITY;
      float m = sc[h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) red[warp][h] = m;
    }
  }
  __syncthreads();
  if (t < G) mx[t] = fmaxf(fmaxf(red[0][t], red[1][t]), fmaxf(red[2][t], red[3][t]));
  __syncthreads();
  float* ps = sp;  // p[slot][G] over the scores, all of which are read
  if (t < kAttnChunk) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float pj = t < nv ? expf(sc[h] - mx[h]) : 0.f;
      ps[t * G + h] = pj;
      const float w = warp_sum(pj);
      if (lane == 0) red[warp][h] = w;
    }
  }
  __syncthreads();
  if (t < G) sm[t] = (red[0][t] + red[1][t]) + (red[2][t] + red[3][t]);

  // values: warp w takes slots 16w..16w+15, lane l dimensions 4l..4l+3
  float av[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < 4; ++e) av[h][e] = 0.f;
  {
    const int s1 = min(warp * 16 + 16, nv);
#pragma unroll 4
    for (int s = warp * 16; s < s1; ++s) {
      const uint2 u = *reinterpret_cast<const uint2*>(Vs + s * kAttnDim * 2 + lane * 8);
      const float v[4] = {bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y)};
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pj = ps[s * G + h];
#pragma unroll
        for (int e = 0; e < 4; ++e) av[h][e] = fmaf(pj, v[e], av[h][e]);
      }
    }
  }
  // the eight warps' sums: through the key buffer, no longer read
  float* racc = reinterpret_cast<float*>(Ks);  // [8][G][128]
#pragma unroll
  for (int h = 0; h < G; ++h)
    *reinterpret_cast<float4*>(racc + (warp * G + h) * kAttnDim + lane * 4) =
        make_float4(av[h][0], av[h][1], av[h][2], av[h][3]);
  __syncthreads();  // also: sm written
  const int d = t & (kAttnDim - 1), hp = t >> 7;
  float O[HPT], M[HPT], L[HPT];
#pragma unroll
  for (int i = 0; i < HPT; ++i) {
    const int h = hp + 2 * i;
    float o = 0.f;
    if (h < G) {
#pragma unroll
      for (int w = 0; w < kAttnThreads / 32; ++w) o += racc[(w * G + h) * kAttnDim + d];
    }
    O[i] = o;
    M[i] = h < G ? mx[h] : 0.f;
    L[i] = h < G ? sm[h] : 1.f;
  }
  if (nchunks == 1) {
    write_output<G>(a, b, g, d, hp, O, L);
    return;
  }

  // this chunk's partials, then the ticket of its group
  const int maxc = a.S / kAttnChunk, maxg = (maxc + kAttnGroup - 1) / kAttnGroup;
  const size_t bg = (size_t)b * a.nkv + g;
  float* base0 = a.part0 + bg * maxc * G * kPartStride;
  write_partial<G>(base0 + (size_t)chunk * G * kPartStride, d, hp, O, M, L);
  const int grp = chunk / kAttnGroup, ngroups = (nchunks + kAttnGroup - 1) / kAttnGroup;
  const int gsize = min(kAttnGroup, nchunks - grp * kAttnGroup);
  __threadfence();
  __syncthreads();
  if (t == 0) {
    unsigned* tk = a.tick0 + bg * maxg + grp;
    const unsigned old = atomicAdd(tk, 1u);
    last = old == (unsigned)(gsize - 1);
    if (last) atomicExch(tk, 0u);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  merge_partials<G>(base0 + (size_t)grp * kAttnGroup * G * kPartStride, gsize, d, hp, O, M, L);
  if (ngroups == 1) {
    write_output<G>(a, b, g, d, hp, O, L);
    return;
  }

  // the group's merged result, then the ticket of the (row, head)
  float* base1 = a.part1 + bg * maxg * G * kPartStride;
  write_partial<G>(base1 + (size_t)grp * G * kPartStride, d, hp, O, M, L);
  __threadfence();
  __syncthreads();
  if (t == 0) {
    unsigned* tk = a.tick1 + bg;
    const unsigned old = atomicAdd(tk, 1u);
    last = old == (unsigned)(ngroups - 1);
    if (last) atomicExch(tk, 0u);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  merge_partials<G>(base1, ngroups, d, hp, O, M, L);
  write_output<G>(a, b, g, d, hp, O, L);
}

typedef void (*AttnKernel)(const AttnParams);

template <int G>
static cudaError_t launch_attention(const AttnParams& a, dim3 grid, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(
        k_decode_attention<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnSmem<G>::bytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k_decode_attention<G><<<grid, kAttnThreads, AttnSmem<G>::bytes, st>>>(a);
  return cudaGetLastError();
}

static size_t align256(size_t v) { return (v + 255) / 256 * 256; }

struct AttnLayout {
  size_t tick1, part0, part1, total;
};

// Workspace: tickets per group [B][nkv][groups], tickets per (row, head)
// [B][nkv], partials per chunk, partials per group (each 256-byte aligned).
static AttnLayout attention_workspace(int B, int nh, int nkv, int s_max) {
  const int G = nh / nkv, maxc = s_max / kAttnChunk;
  const int maxg = (maxc + kAttnGroup - 1) / kAttnGroup;
  const size_t bg = (size_t)B * nkv;
  AttnLayout l;
  l.tick1 = align256(bg * maxg * 4);
  l.part0 = l.tick1 + align256(bg * 4);
  l.part1 = l.part0 + align256(bg * maxc * G * kPartStride * 4);
  l.total = l.part1 + bg * maxg * G * kPartStride * 4;
  return l;
}

}  // namespace ws

using namespace ws;

extern "C" {

size_t ws_attention_workspace_bytes(int B, int n_heads, int n_kv_heads, int head_dim, int s_max) {
  if (B < 1 || B > kMaxBatch || n_kv_heads < 1 || n_heads % n_kv_heads || head_dim != kAttnDim ||
      s_max < kAttnChunk || s_max % kAttnChunk)
    return 0;
  return attention_workspace(B, n_heads, n_kv_heads, s_max).total;
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
  const int G = n_heads / n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 6 && G != 8) {
    set_error("decode attention: %d query heads per key-value head (1, 2, 4, 6 or 8)", G);
    return WS_ERR_SHAPE;
  }
  if (((uintptr_t)k_cache & 15u) || ((uintptr_t)v_cache & 15u)) {
    set_error("decode attention: caches must be 16-byte aligned");
    return WS_ERR_ALIGN;
  }
  const AttnLayout lay = attention_workspace(B, n_heads, n_kv_heads, s_max);
  if (workspace_bytes < lay.total) {
    set_error("workspace too small: need %zu bytes, got %zu", lay.total, workspace_bytes);
    return WS_ERR_ARG;
  }
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
  char* w = static_cast<char*>(workspace);
  a.tick0 = reinterpret_cast<unsigned*>(w);
  a.tick1 = reinterpret_cast<unsigned*>(w + lay.tick1);
  a.part0 = reinterpret_cast<float*>(w + lay.part0);
  a.part1 = reinterpret_cast<float*>(w + lay.part1);
  a.err = device_error_ptr();
  a.timeout_ns = tuning().timeout_ns;
  // the tickets are zero on entry (a zero-filled workspace; the last arrival
  // at every ticket resets it, rows with a bad position take none)
  const dim3 grid(s_max / kAttnChunk, n_kv_heads, B);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  switch (G) {
    case 1: e = launch_attention<1>(a, grid, st); break;
    case 2: e = launch_attention<2>(a, grid, st); break;
    case 4: e = launch_attention<4>(a, grid, st); break;
    case 6: e = launch_attention<6>(a, grid, st); break;
    default: e = launch_attention<8>(a, grid, st); break;
  }
  if (e != cudaSuccess) {
    set_error("launch failed: %s", cudaGetErrorString(e));
    return WS_ERR_CUDA;
  }
  return WS_OK;
}

}  // extern "C"
