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
//   causal grouped-query attention                pf_attn_tmem_kernel
//                                                 (prefill_attn_tc.cuh: bfloat16
//                                                 cache, head size 128),
//                                                 pf_attn_tc_kernel (other
//                                                 bfloat16 heads), pf_attn_kernel
// (SwiGLU runs in the gate/up GEMM's epilogue.)
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
  pdl_trigger();
  pdl_wait();  // inputs come from the previous kernel
  __shared__ float red[kPfThreads / 32];
  const int r = blockIdx.x;
  const float* x = X + static_cast<size_t>(r) * H;
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += kPfThreads) ss = fmaf(x[i], x[i], ss);
  const float inv = 1.0f / sqrtf(pf_block_sum(ss, red) / static_cast<float>(H) + eps);
  const size_t base = static_cast<size_t>(r) * H;
  for (int i = threadIdx.x; i < H; i += kPfThreads) pf_split(x[i] * inv * g[i], A, A2, base + i);
}

// Row r: (A, A2) = RMSNorm(X[r]) * g, for H % 4 == 0 and H <= 4096: each
// thread keeps its (up to four) 4-element pieces in registers between the sum
// of squares and the scaled, split write.
constexpr int kPfNormPieces = 4;
__global__ void __launch_bounds__(kPfThreads) pf_norm4_kernel(const float* X, const float* g, float eps, int H,
                                                               uint16_t* A, uint16_t* A2) {
  pdl_trigger();
  pdl_wait();  // inputs come from the previous kernel
  __shared__ float red[kPfThreads / 32];
  const int r = blockIdx.x, n4 = H >> 2;
  const float4* x = reinterpret_cast<const float4*>(X + static_cast<size_t>(r) * H);
  float4 xv[kPfNormPieces];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kPfNormPieces; ++k) {
    const int i = threadIdx.x + k * kPfThreads;
    xv[k] = i < n4 ? x[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    ss = fmaf(xv[k].x, xv[k].x, fmaf(xv[k].y, xv[k].y, fmaf(xv[k].z, xv[k].z, fmaf(xv[k].w, xv[k].w, ss))));
  }
  ss = warp_sum(ss);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kPfThreads / 32; ++w) t += red[w];
  const float inv = 1.0f / sqrtf(t / static_cast<float>(H) + eps);
  uint2* a = reinterpret_cast<uint2*>(A + static_cast<size_t>(r) * H);
  uint2* a2 = reinterpret_cast<uint2*>(A2 + static_cast<size_t>(r) * H);
  const float4* g4 = reinterpret_cast<const float4*>(g);
#pragma unroll
  for (int k = 0; k < kPfNormPieces; ++k) {
    const int i = threadIdx.x + k * kPfThreads;
    if (i < n4) {
      const float4 gv = g4[i];
      const float y0 = xv[k].x * inv * gv.x, y1 = xv[k].y * inv * gv.y, y2 = xv[k].z * inv * gv.z,
                  y3 = xv[k].w * inv * gv.w;
      const uint16_t h0 = f32_to_bf16_rn(y0), h1 = f32_to_bf16_rn(y1), h2 = f32_to_bf16_rn(y2),
                     h3 = f32_to_bf16_rn(y3);
      const uint16_t l0 = f32_to_bf16_rn(y0 - bf16_to_f32(h0)), l1 = f32_to_bf16_rn(y1 - bf16_to_f32(h1)),
                     l2 = f32_to_bf16_rn(y2 - bf16_to_f32(h2)), l3 = f32_to_bf16_rn(y3 - bf16_to_f32(h3));
      a[i] = make_uint2(h0 | (static_cast<uint32_t>(h1) << 16), h2 | (static_cast<uint32_t>(h3) << 16));
      a2[i] = make_uint2(l0 | (static_cast<uint32_t>(l1) << 16), l2 | (static_cast<uint32_t>(l3) << 16));
    }
  }
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
  pdl_trigger();
  pdl_wait();  // inputs come from the previous kernel
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

// pf_qk_rope_kv_kernel for head size d = 32 EPL (EPL = 1, 2 or 4), one warp
// per (row, head) with the head in registers, EPL consecutive elements per
// lane: RoPE pairs element i with i + d / 2, which lane l ^ 16 holds. Eight
// warps per block over the n (n_q + 2 n_kv) (row, head) pairs.
template <typename KT, int EPL>
__global__ void __launch_bounds__(256) pf_qk_rope_kv_vec_kernel(float* qkv, int n, int p0, int n_q, int n_kv,
                                                                 const float* g_q, const float* g_k, float eps,
                                                                 const float* rope_cos, const float* rope_sin,
                                                                 void* kc, void* vc, int max_seq) {
  pdl_trigger();
  pdl_wait();  // inputs come from the previous kernel
  static_assert(EPL == 1 || EPL == 2 || EPL == 4, "head size 32, 64 or 128");
  constexpr int d = 32 * EPL, half = d / 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nh = n_q + 2 * n_kv;
  const int gw = blockIdx.x * 8 + warp;
  if (gw >= n * nh) return;
  const int r = gw / nh, h = gw - r * nh;
  const int p = p0 + r;
  float* v = qkv + static_cast<size_t>(r) * nh * d + static_cast<size_t>(h) * d + lane * EPL;
  float x[EPL];
  if constexpr (EPL == 4) {
    const float4 t = *reinterpret_cast<const float4*>(v);
    x[0] = t.x, x[1] = t.y, x[2] = t.z, x[3] = t.w;
  } else if constexpr (EPL == 2) {
    const float2 t = *reinterpret_cast<const float2*>(v);
    x[0] = t.x, x[1] = t.y;
  } else {
    x[0] = v[0];
  }
  auto store_cache = [&](void* base, int head, const float* y) {
    const size_t at = (static_cast<size_t>(head) * max_seq + p) * d + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) store1<KT>(base, at + e, y[e]);
  };
  if (h >= n_q + n_kv) {  // value head: append
    store_cache(vc, h - n_q - n_kv, x);
    return;
  }
  const bool is_q = h < n_q;
  const float* g = (is_q ? g_q : g_k) + lane * EPL;
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) ss = fmaf(x[e], x[e], ss);
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
  const int ci = (lane & 15) * EPL;
  const float* cs = rope_cos + static_cast<size_t>(p) * half + ci;
  const float* sn = rope_sin + static_cast<size_t>(p) * half + ci;
  float y[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const float own = x[e] * inv * g[e];
    const float other = __shfl_xor_sync(0xffffffffu, own, 16);
    // lanes 0-15 hold a = element i, lanes 16-31 b = element i + d/2
    y[e] = lane < 16 ? own * cs[e] - other * sn[e] : other * sn[e] + own * cs[e];
  }
  if (is_q) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] = y[e];
  } else {
    store_cache(kc, h - n_q, y);
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
  pdl_trigger();
  pdl_wait();  // Q, keys and values come from the previous kernels
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

// ---- causal attention on the tensor cores (bfloat16 cache) ----
//
// Flash-attention form with warp-level BF16 MMAs (m16n8k16, FP32
// accumulation): a warp owns 16 query vectors, the group's query heads of
// 16/group consecutive chunk rows (vector v = row * group + head), all on key
// head g. Tiles of 64 keys and their values are copied row-major into padded
// shared-memory rows with cp.async (zero-filled past the last key any row of
// the block sees), two tiles in flight, so a tile's copies overlap the
// previous tile's MMAs; the value operand of O += P V is read transposed with
// ldmatrix.trans. Per tile the warp forms S = Q K^T, masks keys past each
// row's position, updates the running max and sum, and accumulates O += P V.
// Q and P enter the MMAs as bfloat16 value + remainder pairs (two MMAs each),
// keys and values are the cache's bfloat16, so scores and outputs keep
// float32 precision. Needs head_dim % 16 == 0 and n_q / n_kv dividing 16.
constexpr int kPfTcWarps = 4, kPfTcKeys = 64;

// Dynamic shared memory of pf_attn_tc_kernel<D>: two stages of key and value
// tiles, rows padded by 8 elements (conflict-free fragment and ldmatrix reads).
constexpr size_t pf_attn_tc_smem(int D) { return 2ull * 2 * kPfTcKeys * (D + 8) * sizeof(uint16_t); }

__device__ __forceinline__ void mma_bf16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte asynchronous copy global -> shared; src_bytes 0 fills zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Two transposed 8x8 bfloat16 matrices: lanes 0-7 give the row addresses of
// the first, lanes 8-15 of the second; thread t receives, per matrix, the
// elements (2 (t % 4), t / 4) and (2 (t % 4) + 1, t / 4), low half first.
__device__ __forceinline__ void ldmatrix_x2_trans(uint32_t& r0, uint32_t& r1, const void* row_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(smem_u32(row_addr)));
}

// Two floats as a packed bfloat16 pair (low half: x) for value and remainder.
__device__ __forceinline__ void pack_split(float x, float y, uint32_t* hi, uint32_t* lo) {
  const uint16_t hx = f32_to_bf16_rn(x), hy = f32_to_bf16_rn(y);
  const uint16_t lx = f32_to_bf16_rn(x - bf16_to_f32(hx)), ly = f32_to_bf16_rn(y - bf16_to_f32(hy));
  *hi = static_cast<uint32_t>(hx) | (static_cast<uint32_t>(hy) << 16);
  *lo = static_cast<uint32_t>(lx) | (static_cast<uint32_t>(ly) << 16);
}

template <int D>
__global__ void __launch_bounds__(kPfTcWarps * 32) pf_attn_tc_kernel(const float* qkv, int n, int p0, int n_q, int n_kv,
                                                                      const uint16_t* kc, const uint16_t* vc,
                                                                      int max_seq, float scale, uint16_t* AO,
                                                                      uint16_t* AO2) {
  constexpr int KS = D / 16;  // k-steps of S = Q K^T
  pdl_trigger();
  pdl_wait();  // Q, keys and values come from the previous kernels
  constexpr int NT = D / 8;   // n-tiles of O
  constexpr int RS = D + 8;   // padded row length (elements)
  extern __shared__ __align__(16) uint16_t pf_tc_smem[];
  uint16_t* Kst = pf_tc_smem;                              // [2][kPfTcKeys][RS]
  uint16_t* Vst = pf_tc_smem + 2 * kPfTcKeys * RS;         // [2][kPfTcKeys][RS]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int g = blockIdx.x;
  const int group = n_q / n_kv, rpw = 16 / group;  // rows per warp
  const int r0 = blockIdx.y * kPfTcWarps * rpw;
  const int rw = r0 + warp * rpw;                 // first row of this warp
  const int W = (n_q + 2 * n_kv) * D;
  const int blk_rows = min(n - r0, kPfTcWarps * rpw);
  const int pmax = p0 + r0 + blk_rows - 1;         // last key any row of the block sees
  const int pmax_w = p0 + min(n, rw + rpw) - 1;     // ... and of this warp
  // this thread's two query vectors: rows of the C fragments
  const int v0 = gid, v1 = gid + 8;
  const int row0 = rw + v0 / group, row1 = rw + v1 / group;
  const int pos0 = p0 + row0, pos1 = p0 + row1;
  const size_t kv_base = static_cast<size_t>(g) * max_seq * D;
  // copies of one tile (keys t0.. into stage st): 16-byte pieces, zero past pmax
  auto stage_tile = [&](int t0, int st) {
    for (int i = threadIdx.x; i < kPfTcKeys * (D / 8); i += kPfTcWarps * 32) {
      const int kk = i / (D / 8), e = (i - kk * (D / 8)) * 8;
      const bool in = t0 + kk <= pmax;
      const size_t at = kv_base + static_cast<size_t>(in ? t0 + kk : 0) * D + e;
      cp_async16(Kst + (st * kPfTcKeys + kk) * RS + e, kc + at, in ? 16u : 0u);
      cp_async16(Vst + (st * kPfTcKeys + kk) * RS + e, vc + at, in ? 16u : 0u);
    }
    cp_async_commit();
  };
  stage_tile(0, 0);  // the first tile's copies overlap the Q set-up

  // Q fragments (value and remainder), zero for rows past the chunk
  uint32_t qh[KS][4], ql[KS][4];
  {
    auto qptr = [&](int v) -> const float* {
      const int row = rw + v / group;
      return row < n ? qkv + static_cast<size_t>(row) * W + (g * group + v % group) * D : nullptr;
    };
    const float* q0 = qptr(v0);
    const float* q1 = qptr(v1);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int c = ks * 16 + 2 * tig;
      pack_split(q0 ? q0[c] : 0.f, q0 ? q0[c + 1] : 0.f, &qh[ks][0], &ql[ks][0]);
      pack_split(q1 ? q1[c] : 0.f, q1 ? q1[c + 1] : 0.f, &qh[ks][1], &ql[ks][1]);
      pack_split(q0 ? q0[c + 8] : 0.f, q0 ? q0[c + 9] : 0.f, &qh[ks][2], &ql[ks][2]);
      pack_split(q1 ? q1[c + 8] : 0.f, q1 ? q1[c + 9] : 0.f, &qh[ks][3], &ql[ks][3]);
    }
  }
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int t0 = 0, it = 0; t0 <= pmax; t0 += kPfTcKeys, ++it) {
    const int st = it & 1;
    // the next tile's copies go into the other stage, freed by the barrier
    // that ended the previous iteration
    if (t0 + kPfTcKeys <= pmax) {
      stage_tile(t0 + kPfTcKeys, st ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint16_t* Ks = Kst + st * kPfTcKeys * RS;
    const uint16_t* Vs = Vst + st * kPfTcKeys * RS;
    if (t0 > pmax_w) {  // no row of this warp sees these keys
      __syncthreads();
      continue;
    }
    // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
    float sc[kPfTcKeys / 8][4];
#pragma unroll
    for (int j = 0; j < kPfTcKeys / 8; ++j) {
      sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
      const uint16_t* krow = Ks + (j * 8 + gid) * RS;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow + ks * 16 + 2 * tig);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(krow + ks * 16 + 8 + 2 * tig);
        mma_bf16_16816(sc[j], qh[ks][0], qh[ks][1], qh[ks][2], qh[ks][3], b0, b1);
        mma_bf16_16816(sc[j], ql[ks][0], ql[ks][1], ql[ks][2], ql[ks][3], b0, b1);
      }
    }
    // mask, scale, running max
    float mx0 = m0, mx1 = m1;
#pragma unroll
    for (int j = 0; j < kPfTcKeys / 8; ++j) {
      const int t = t0 + j * 8 + 2 * tig;
      sc[j][0] = t <= pos0 ? sc[j][0] * scale : -INFINITY;
      sc[j][1] = t + 1 <= pos0 ? sc[j][1] * scale : -INFINITY;
      sc[j][2] = t <= pos1 ? sc[j][2] * scale : -INFINITY;
      sc[j][3] = t + 1 <= pos1 ? sc[j][3] * scale : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(sc[j][0], sc[j][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[j][2], sc[j][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    // rows with no visible key yet keep max -inf: use 0 as the reference so exp() gives 0
    const float ref0 = mx0 == -INFINITY ? 0.f : mx0, ref1 = mx1 == -INFINITY ? 0.f : mx1;
    const float c0 = expf(m0 - ref0), c1 = expf(m1 - ref1);
    m0 = mx0;
    m1 = mx1;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < kPfTcKeys / 8; ++j) {
      sc[j][0] = expf(sc[j][0] - ref0);
      sc[j][1] = expf(sc[j][1] - ref0);
      sc[j][2] = expf(sc[j][2] - ref1);
      sc[j][3] = expf(sc[j][3] - ref1);
      s0 += sc[j][0] + sc[j][1];
      s1 += sc[j][2] + sc[j][3];
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    l0 = l0 * c0 + s0;
    l1 = l1 * c1 + s1;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      o[j][0] *= c0;
      o[j][1] *= c0;
      o[j][2] *= c1;
      o[j][3] *= c1;
    }
    // O += P V: 4 k-steps of 16 keys; P from the score fragments (value + remainder)
#pragma unroll
    for (int kk = 0; kk < kPfTcKeys / 16; ++kk) {
      uint32_t ah[4], al[4];
      pack_split(sc[2 * kk][0], sc[2 * kk][1], &ah[0], &al[0]);
      pack_split(sc[2 * kk][2], sc[2 * kk][3], &ah[1], &al[1]);
      pack_split(sc[2 * kk + 1][0], sc[2 * kk + 1][1], &ah[2], &al[2]);
      pack_split(sc[2 * kk + 1][2], sc[2 * kk + 1][3], &ah[3], &al[3]);
      // value rows kk*16 .. kk*16+15, columns j*8 ..: lane r < 16 points at row kk*16 + r
      const uint16_t* vrow = Vs + (kk * 16 + (lane & 15)) * RS;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        uint32_t b0, b1;
        ldmatrix_x2_trans(b0, b1, vrow + j * 8);
        mma_bf16_16816(o[j], ah[0], ah[1], ah[2], ah[3], b0, b1);
        mma_bf16_16816(o[j], al[0], al[1], al[2], al[3], b0, b1);
      }
    }
    __syncthreads();  // this stage is refilled two tiles on
  }
  // O / L as value and remainder
  const float i0 = 1.0f / l0, i1 = 1.0f / l1;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int c = j * 8 + 2 * tig;
    if (row0 < n) {
      const size_t at = static_cast<size_t>(row0) * n_q * D + (g * group + v0 % group) * D + c;
      pf_split(o[j][0] * i0, AO, AO2, at);
      pf_split(o[j][1] * i0, AO, AO2, at + 1);
    }
    if (row1 < n) {
      const size_t at = static_cast<size_t>(row1) * n_q * D + (g * group + v1 % group) * D + c;
      pf_split(o[j][2] * i1, AO, AO2, at);
      pf_split(o[j][3] * i1, AO, AO2, at + 1);
    }
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
