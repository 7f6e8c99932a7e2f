// Chunked prefill ("Megakernels", "Chunked prefill for long prompts"): a
// chunk of prompt rows at consecutive positions goes through every layer
// together. The projections are tensor-core GEMMs over the chunk's rows
// (gemm_tc.cuh); the kernels here do the per-row work between them and the
// causal attention of the rows over the cache (earlier chunks and the rows of
// this chunk up to each row's own position):
//
//   embedding gather + input RMSNorm (layer 0)   pf_embed_norm_kernel
//   RMSNorm of the residual rows                  pf_norm_kernel
//   per-head Q/K RMSNorm, RoPE, K/V cache append  pf_qk_rope_kv_kernel
//   causal grouped-query attention                pf_attn_kernel
//   SwiGLU of the gate/up rows                    pf_swiglu_kernel
//
// The residual rows stay float32; each GEMM operand row (normalised rows,
// attention output, SwiGLU output) is written as a pair of bfloat16 rows,
// value and remainder (v = hi + lo to ~2^-17 relative), which the GEMM
// multiplies into one accumulator: the chunk's projections see the same
// float32 activations as the single-token path.
#pragma once
#include <cstdint>

#include "attention.cuh"
#include "gemv_stream.cuh"
#include "ptx.cuh"

namespace wsg {

constexpr int kPfThreads = 256;

// v as bfloat16 value and remainder: hi = nearest(v), lo = nearest(v - hi).
__device__ __forceinline__ void pf_split(float v, uint16_t* hi, uint16_t* lo, size_t i) {
  const uint16_t h = f32_to_bf16_rn(v);
  hi[i] = h;
  lo[i] = f32_to_bf16_rn(v - bf16_to_f32(h));
}

// Sum over the block (kPfThreads threads); every thread gets the total.
__device__ __forceinline__ float pf_block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kPfThreads / 32; ++w) t += red[w];
  __syncthreads();
  return t;
}

// Row r: h = E[token of position p0 + r] into X, x = RMSNorm(h) * g into (A, A2).
template <typename WT>
__global__ void __launch_bounds__(kPfThreads) pf_embed_norm_kernel(const int32_t* tok, int p0, const void* embed,
                                                                    int vocab, const float* g, float eps, int H,
                                                                    float* X, uint16_t* A, uint16_t* A2, uint32_t* err) {
  __shared__ float red[kPfThreads / 32];
  const int r = blockIdx.x;
  int t = tok[p0 + r];
  if (t < 0 || t >= vocab) {
    if (threadIdx.x == 0) atomicOr(err, ERR_BAD_TOKEN);
    t = 0;
  }
  const WT* row = static_cast<const WT*>(embed) + static_cast<size_t>(t) * H;
  float* x = X + static_cast<size_t>(r) * H;
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += kPfThreads) {
    const float h = load_f32<WT>(row, i);
    x[i] = h;
    ss = fmaf(h, h, ss);
  }
  const float inv = 1.0f / sqrtf(pf_block_sum(ss, red) / static_cast<float>(H) + eps);
  const size_t base = static_cast<size_t>(r) * H;
  for (int i = threadIdx.x; i < H; i += kPfThreads) pf_split(x[i] * inv * g[i], A, A2, base + i);
}

// Row r: (A, A2) = RMSNorm(X[r]) * g.
__global__ void __launch_bounds__(kPfThreads) pf_norm_kernel(const float* X, const float* g, float eps, int H,
                                                              uint16_t* A, uint16_t* A2) {
  __shared__ float red[kPfThreads / 32];
  const int r = blockIdx.x;
  const float* x = X + static_cast<size_t>(r) * H;
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += kPfThreads) ss = fmaf(x[i], x[i], ss);
  const float inv = 1.0f / sqrtf(pf_block_sum(ss, red) / static_cast<float>(H) + eps);
  const size_t base = static_cast<size_t>(r) * H;
  for (int i = threadIdx.x; i < H; i += kPfThreads) pf_split(x[i] * inv * g[i], A, A2, base + i);
}

// One warp per (row, head) over the n_q + 2 n_kv heads of the row's raw
// projections (row stride W = (n_q + 2 n_kv) d): q heads are normalised
// (g_q), rotated and written back in place; k heads are normalised (g_k),
// rotated, rounded to the cache type and appended at position p0 + row; v
// heads are rounded and appended.
template <typename KT>
__global__ void __launch_bounds__(128) pf_qk_rope_kv_kernel(float* qkv, int p0, int n_q, int n_kv, int d,
                                                             const float* g_q, const float* g_k, float eps,
                                                             const float* rope_cos, const float* rope_sin, void* kc,
                                                             void* vc, int max_seq) {
  __shared__ float buf[4][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x, h = blockIdx.y * 4 + warp;
  const int nh = n_q + 2 * n_kv;
  if (h >= nh) return;
  const int W = nh * d, p = p0 + r, half = d >> 1;
  float* v = qkv + static_cast<size_t>(r) * W + static_cast<size_t>(h) * d;
  float* s = buf[warp];
  if (h >= n_q + n_kv) {  // value head: append
    const int gv = h - n_q - n_kv;
    for (int e = lane; e < d; e += 32)
      store1<KT>(vc, (static_cast<size_t>(gv) * max_seq + p) * d + e, v[e]);
    return;
  }
  const bool is_q = h < n_q;
  const float* g = is_q ? g_q : g_k;
  float ss = 0.f;
  for (int e = lane; e < d; e += 32) {
    const float x = v[e];
    s[e] = x;
    ss = fmaf(x, x, ss);
  }
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
  for (int e = lane; e < d; e += 32) s[e] = s[e] * inv * g[e];
  __syncwarp();
  const float* cs = rope_cos + static_cast<size_t>(p) * half;
  const float* sn = rope_sin + static_cast<size_t>(p) * half;
  for (int i = lane; i < half; i += 32) {
    const float a = s[i], b = s[i + half], c = cs[i], sv = sn[i];
    const float lo = a * c - b * sv, hi = a * sv + b * c;
    if (is_q) {
      v[i] = lo;
      v[i + half] = hi;
    } else {
      const int gk = h - n_q;
      store1<KT>(kc, (static_cast<size_t>(gk) * max_seq + p) * d + i, lo);
      store1<KT>(kc, (static_cast<size_t>(gk) * max_seq + p) * d + i + half, hi);
    }
  }
}

// Causal grouped-query attention of up to 8 chunk rows (one warp each) for
// key/value head g and its n_q/n_kv query heads: keys 0..p (p the row's
// position) in tiles of 32 keys staged in shared memory and shared by the
// block's rows; online softmax per warp and head. Output as value and
// remainder into (AO, AO2)[row][(g * group + h) * d + e].
constexpr int kPfAttnRows = 8, kPfAttnKeys = 32;

template <typename KT, int GMAX>
__global__ void __launch_bounds__(kPfAttnRows * 32) pf_attn_kernel(const float* qkv, int n, int p0, int n_q, int n_kv,
                                                                    int d, const void* kc, const void* vc, int max_seq,
                                                                    float scale, uint16_t* AO, uint16_t* AO2) {
  __shared__ __align__(16) float Ks[kPfAttnKeys][128];
  __shared__ __align__(16) float Vs[kPfAttnKeys][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x, r0 = blockIdx.y * kPfAttnRows;
  const int group = n_q / n_kv, W = (n_q + 2 * n_kv) * d;
  const int row = r0 + warp;
  const bool live = row < n;
  const int p = p0 + row;
  const int pmax = p0 + min(n, r0 + kPfAttnRows) - 1;
  const bool active = 4 * lane < d;
  const size_t head_base = static_cast<size_t>(g) * max_seq * d;

  float4 q[GMAX];
  float m[GMAX], l[GMAX];
  float4 o[GMAX];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    q[h] = make_float4(0, 0, 0, 0);
    if (h < group && live && active)
      q[h] = *reinterpret_cast<const float4*>(qkv + static_cast<size_t>(row) * W + (g * group + h) * d + 4 * lane);
    m[h] = -INFINITY;
    l[h] = 0.f;
    o[h] = make_float4(0, 0, 0, 0);
  }

  for (int t0 = 0; t0 <= pmax; t0 += kPfAttnKeys) {
    __syncthreads();
    // stage keys/values t0 .. min(t0 + 31, pmax): 4 elements per thread per step
    const int nk = min(kPfAttnKeys, pmax - t0 + 1);
    for (int i = threadIdx.x; i < nk * (d >> 2); i += kPfAttnRows * 32) {
      const int kk = i / (d >> 2), e = (i - kk * (d >> 2)) * 4;
      const size_t idx = head_base + static_cast<size_t>(t0 + kk) * d + e;
      *reinterpret_cast<float4*>(&Ks[kk][e]) = load4<KT>(kc, idx);
      *reinterpret_cast<float4*>(&Vs[kk][e]) = load4<KT>(vc, idx);
    }
    __syncthreads();
    if (!live) continue;
    const int kend = min(nk, p - t0 + 1);  // keys of this tile the row sees
    for (int j = 0; j < kend; j += 8) {
      float4 kk[8], vv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        kk[u] = vv[u] = make_float4(0, 0, 0, 0);
        if (j + u < kend && active) {
          kk[u] = *reinterpret_cast<const float4*>(&Ks[j + u][4 * lane]);
          vv[u] = *reinterpret_cast<const float4*>(&Vs[j + u][4 * lane]);
        }
      }
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        if (h >= group) break;
        float sc[8];
        float mx = m[h];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float dot = q[h].x * kk[u].x + q[h].y * kk[u].y + q[h].z * kk[u].z + q[h].w * kk[u].w;
          sc[u] = (j + u < kend) ? warp_sum(dot) * scale : -INFINITY;
          mx = fmaxf(mx, sc[u]);
        }
        const float corr = expf(m[h] - mx);
        l[h] *= corr;
        o[h].x *= corr;
        o[h].y *= corr;
        o[h].z *= corr;
        o[h].w *= corr;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float pw = expf(sc[u] - mx);
          l[h] += pw;
          o[h].x = fmaf(pw, vv[u].x, o[h].x);
          o[h].y = fmaf(pw, vv[u].y, o[h].y);
          o[h].z = fmaf(pw, vv[u].z, o[h].z);
          o[h].w = fmaf(pw, vv[u].w, o[h].w);
        }
        m[h] = mx;
      }
    }
  }
  if (!live || !active) return;
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    if (h >= group) break;
    const float il = 1.0f / l[h];
    const size_t at = static_cast<size_t>(row) * n_q * d + (g * group + h) * d + 4 * lane;
    pf_split(o[h].x * il, AO, AO2, at);
    pf_split(o[h].y * il, AO, AO2, at + 1);
    pf_split(o[h].z * il, AO, AO2, at + 2);
    pf_split(o[h].w * il, AO, AO2, at + 3);
  }
}

// (AI, AI2)[r][j] = silu(GU[r][j]) * GU[r][I + j] as value and remainder.
__global__ void pf_swiglu_kernel(const float* GU, int n, int I, uint16_t* AI, uint16_t* AI2) {
  const size_t total = static_cast<size_t>(n) * I;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t r = i / I, j = i - r * I;
    const float* gu = GU + r * 2 * I;
    pf_split(silu_f32(gu[j]) * gu[I + j], AI, AI2, i);
  }
}

// Small control writes after a chunk: ctrl[0] = value; every kv_ready count of
// the persistent engine = value2 (when kv_ready is not NULL).
__global__ void pf_control_kernel(int32_t* ctrl, int32_t value, uint32_t* kv_ready, int n_ready, uint32_t value2) {
  if (threadIdx.x == 0 && blockIdx.x == 0) ctrl[0] = value;
  if (kv_ready)
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_ready; i += gridDim.x * blockDim.x) kv_ready[i] = value2;
}

// Copy one float row (the chunk's last residual row into the head's input).
__global__ void pf_copy_row_kernel(const float* src, float* dst, int H) {
  for (int i = threadIdx.x; i < H; i += blockDim.x) dst[i] = src[i];
}

}  // namespace wsg
