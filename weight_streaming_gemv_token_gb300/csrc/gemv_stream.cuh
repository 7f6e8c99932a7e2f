// Weight-streaming GEMV engine: y = W x for one activation vector.
//
// The matrix-vector products of the decode step read every weight exactly
// once per token ("Our Kernel Benchmark Was Measuring the System Cache",
// Summary: production decode streams every weight once per token), so the
// kernel is built to keep HBM busy:
//
//  * one CTA per SM; each CTA owns a contiguous range of output rows, handed
//    out in balanced units so no CTA gets more than one unit above average;
//  * each row is cut into segments of at most a few KB; warp w of the CTA
//    takes segments w, w + NW, w + 2NW, ... and streams them through its own
//    RING-byte shared-memory ring (as many slots as segments fit, up to
//    NSMAX) with bulk (TMA) copies completed on mbarriers; the copies carry
//    an L2 evict-first policy;
//  * the first copies of every warp, and for matrices that fit in L2 an L2
//    prefetch of the CTA's whole weight slice, are issued before the kernel
//    waits on its predecessor (programmatic dependent launch), so the weight
//    stream of this kernel overlaps the tail and the prologue of the chain;
//  * the activation vector is staged once per CTA in shared memory, with an
//    optional fused RMSNorm prologue;
//  * per-segment partial dots are reduced in a fixed order, so results are
//    bit-reproducible run to run;
//  * fused epilogues: plain store, residual add, SwiGLU on (gate, up) row
//    pairs, and logits + two-pass lowest-ID argmax + position advance.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace wsg {

enum Pro : int {
  PRO_X = 0,           // x read from memory (XT), no norm
  PRO_NORM = 1,        // x = RMSNorm(h) * g, h f32
  PRO_EMBED_NORM = 2,  // h = embed[token]; x = RMSNorm(h) * g; CTA 0 stores h
};

enum Epi : int {
  EPI_STORE = 0,   // y[row] = v
  EPI_RESID = 1,   // y[row] += v
  EPI_SWIGLU = 2,  // logical rows (2i, 2i+1) = (gate_i, up_i): y[i] = silu(gate_i) * up_i
  EPI_ARGMAX = 3,  // y[row] = v (if y); greedy token of all rows -> tok[pos+1]; ctrl[0] = pos+1
};

struct RowMap {
  const char* base[3];
  int32_t split1, split2;  // logical rows [0,split1) -> base[0], [split1,split2) -> base[1], rest -> base[2]
  int32_t interleave;      // nonzero: logical row 2i -> base[0] row i, 2i+1 -> base[1] row i
};

struct GemvArgs {
  RowMap w;
  int32_t out, in;
  int32_t row_bytes, seg_bytes, segs_per_row, row_unit;
  const void* x;
  const float* norm_g;
  float eps;
  const void* embed;
  const int32_t* tok;
  int32_t* ctrl;
  float* h_out;
  float* y;
  int32_t vocab;
  float* part_val;
  int32_t* part_idx;
  uint32_t* counter;
  int32_t* tok_w;
  uint32_t* err;
  int32_t l2_prefetch;  // nonzero: prefetch this CTA's whole weight slice into L2 up front
};

__device__ __forceinline__ const char* row_ptr(const RowMap& m, int row, int row_bytes) {
  if (m.interleave) return m.base[row & 1] + static_cast<size_t>(row >> 1) * row_bytes;
  if (row < m.split1) return m.base[0] + static_cast<size_t>(row) * row_bytes;
  if (row < m.split2) return m.base[1] + static_cast<size_t>(row - m.split1) * row_bytes;
  return m.base[2] + static_cast<size_t>(row - m.split2) * row_bytes;
}

template <typename T>
__device__ __forceinline__ float load_f32(const void* p, int i);
template <>
__device__ __forceinline__ float load_f32<float>(const void* p, int i) {
  return static_cast<const float*>(p)[i];
}
template <>
__device__ __forceinline__ float load_f32<uint16_t>(const void* p, int i) {
  return bf16_to_f32(static_cast<const uint16_t*>(p)[i]);
}

// Position of element i of the activation vector in the shared staging array.
// bf16 weights read 8 columns per 16-byte load; their x is staged as two float4
// planes (columns 8g..8g+3 in plane 0, 8g+4..8g+7 in plane 1) so that the
// 32 lanes of a warp hit distinct banks.
template <typename WT>
__device__ __forceinline__ int xs_index(int i, int in);
template <>
__device__ __forceinline__ int xs_index<float>(int i, int) {
  return i;
}
template <>
__device__ __forceinline__ int xs_index<uint16_t>(int i, int in) {
  const int g = i >> 3, r = i & 7;
  return r < 4 ? 4 * g + r : 4 * ((in >> 3) + g) + (r - 4);
}

// Partial dot of one segment held in shared memory with the matching x.
template <typename WT>
__device__ __forceinline__ float seg_dot(const unsigned char* seg, const float* xs, int e0, int bytes, int in, int lane);

template <>
__device__ __forceinline__ float seg_dot<float>(const unsigned char* seg, const float* xs, int e0, int bytes, int,
                                                int lane) {
  const float4* w4 = reinterpret_cast<const float4*>(seg);
  const float4* x4 = reinterpret_cast<const float4*>(xs + e0);
  const int n4 = bytes >> 4;
  float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
  for (int i = lane; i < n4; i += 32) {
    const float4 w = w4[i], x = x4[i];
    a0 = fmaf(w.x, x.x, a0);
    a1 = fmaf(w.y, x.y, a1);
    a0 = fmaf(w.z, x.z, a0);
    a1 = fmaf(w.w, x.w, a1);
  }
  return a0 + a1;
}

template <>
__device__ __forceinline__ float seg_dot<uint16_t>(const unsigned char* seg, const float* xs, int e0, int bytes, int in,
                                                   int lane) {
  const uint4* w8 = reinterpret_cast<const uint4*>(seg);
  const float4* xa = reinterpret_cast<const float4*>(xs) + (e0 >> 3);
  const float4* xb = reinterpret_cast<const float4*>(xs) + (in >> 3) + (e0 >> 3);
  const int n8 = bytes >> 4;
  float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
  for (int i = lane; i < n8; i += 32) {
    const uint4 w = w8[i];
    const float4 p = xa[i], q = xb[i];
    a0 = fmaf(__uint_as_float(w.x << 16), p.x, a0);
    a1 = fmaf(__uint_as_float(w.x & 0xFFFF0000u), p.y, a1);
    a0 = fmaf(__uint_as_float(w.y << 16), p.z, a0);
    a1 = fmaf(__uint_as_float(w.y & 0xFFFF0000u), p.w, a1);
    a0 = fmaf(__uint_as_float(w.z << 16), q.x, a0);
    a1 = fmaf(__uint_as_float(w.z & 0xFFFF0000u), q.y, a1);
    a0 = fmaf(__uint_as_float(w.w << 16), q.z, a0);
    a1 = fmaf(__uint_as_float(w.w & 0xFFFF0000u), q.w, a1);
  }
  return a0 + a1;
}

// Dots of nr (<= 4) consecutive whole rows held in shared memory with the same
// x: each x chunk is read from shared memory once for all rows. Lane partials
// are returned in v[0..3] (zero past nr).
template <typename WT>
__device__ __forceinline__ void rows_dot(const unsigned char* seg, int row_bytes, int nr, const float* xs, int in,
                                         int lane, float (&v)[4]);

template <>
__device__ __forceinline__ void rows_dot<float>(const unsigned char* seg, int row_bytes, int nr, const float* xs, int,
                                                int lane, float (&v)[4]) {
  const int n4 = row_bytes >> 4;
  const float4* x4 = reinterpret_cast<const float4*>(xs);
#pragma unroll
  for (int r = 0; r < 4; ++r) v[r] = 0.f;
#pragma unroll 2
  for (int i = lane; i < n4; i += 32) {
    const float4 x = x4[i];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (r < nr) {
        const float4 w = reinterpret_cast<const float4*>(seg + static_cast<size_t>(r) * row_bytes)[i];
        v[r] = fmaf(w.x, x.x, fmaf(w.y, x.y, fmaf(w.z, x.z, fmaf(w.w, x.w, v[r]))));
      }
    }
  }
}

template <>
__device__ __forceinline__ void rows_dot<uint16_t>(const unsigned char* seg, int row_bytes, int nr, const float* xs,
                                                   int in, int lane, float (&v)[4]) {
  const int n8 = row_bytes >> 4;
  const float4* xa = reinterpret_cast<const float4*>(xs);
  const float4* xb = reinterpret_cast<const float4*>(xs) + (in >> 3);
#pragma unroll
  for (int r = 0; r < 4; ++r) v[r] = 0.f;
#pragma unroll 2
  for (int i = lane; i < n8; i += 32) {
    const float4 p = xa[i], q = xb[i];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (r < nr) {
        const uint4 w = reinterpret_cast<const uint4*>(seg + static_cast<size_t>(r) * row_bytes)[i];
        float t = v[r];
        t = fmaf(__uint_as_float(w.x << 16), p.x, t);
        t = fmaf(__uint_as_float(w.x & 0xFFFF0000u), p.y, t);
        t = fmaf(__uint_as_float(w.y << 16), p.z, t);
        t = fmaf(__uint_as_float(w.y & 0xFFFF0000u), p.w, t);
        t = fmaf(__uint_as_float(w.z << 16), q.x, t);
        t = fmaf(__uint_as_float(w.z & 0xFFFF0000u), q.y, t);
        t = fmaf(__uint_as_float(w.w << 16), q.z, t);
        t = fmaf(__uint_as_float(w.w & 0xFFFF0000u), q.w, t);
        v[r] = t;
      }
    }
  }
}

// (v, i) beats (bv, bi) under "largest value, lowest index on ties"; NaN never beats.
__device__ __forceinline__ bool argmax_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// Shared memory bytes the kernel needs for a given problem.
template <int NW, int NSMAX, int RING>
__host__ __device__ constexpr size_t gemv_ring_bytes() {
  return static_cast<size_t>(NW) * RING + static_cast<size_t>(NW) * NSMAX * 8;
}

inline size_t gemv_smem_bytes(size_t ring_bytes, int in, int max_rows, int segs_per_row) {
  size_t b = ring_bytes;
  b += ((static_cast<size_t>(in) * 4 + 15) / 16) * 16;                        // x staging
  b += ((static_cast<size_t>(max_rows) * segs_per_row * 4 + 15) / 16) * 16;   // partial dots
  b += 64 * 8;                                                               // reductions
  return b;
}

// Row epilogues after the per-segment partial dots are complete: store,
// residual add, or logits with the two argmax passes (the last CTA to
// finish, detected with an atomic counter, reduces every CTA's best).
template <int EPI>
__device__ __forceinline__ void rows_epilogue(const GemvArgs& a, const float* part, float* red, int nrows, int spr,
                                                int r0, int pos, int c, int G, int tid, int warp, int lane, int NT,
                                                int NW) {
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int r = tid; r < nrows; r += NT) {
    float v = 0.f;
    for (int j = 0; j < spr; ++j) v += part[r * spr + j];
    const int row = r0 + r;
    if constexpr (EPI == EPI_STORE) a.y[row] = v;
    if constexpr (EPI == EPI_RESID) a.y[row] += v;
    if constexpr (EPI == EPI_ARGMAX) {
      if (a.y) a.y[row] = v;
      if (argmax_better(v, row, bv, bi)) {
        bv = v;
        bi = row;
      }
    }
  }
  if constexpr (EPI == EPI_ARGMAX) {
  // Pass 1: this CTA's best (value, index).
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (argmax_better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  int* redi = reinterpret_cast<int*>(red + 32);
  __syncthreads();
  if (lane == 0) {
    red[warp] = bv;
    redi[warp] = bi;
  }
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) {
    for (int w = 1; w < NW; ++w)
      if (argmax_better(red[w], redi[w], bv, bi)) {
        bv = red[w];
        bi = redi[w];
      }
    a.part_val[c] = bv;
    a.part_idx[c] = bi;
    __threadfence();
    const uint32_t prev = atomicAdd(a.counter, 1u);
    s_last = (prev == static_cast<uint32_t>(G - 1));
  }
  __syncthreads();
  if (!s_last) return;
  // Pass 2 (last CTA to finish): best over all CTAs, lowest index on ties.
  __threadfence();
  float gv = -INFINITY;
  int gi = 0x7fffffff;
  for (int k = tid; k < G; k += NT) {
    const float v = __ldcg(a.part_val + k);
    const int i = __ldcg(a.part_idx + k);
    if (argmax_better(v, i, gv, gi)) {
      gv = v;
      gi = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, gv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, gi, o);
    if (argmax_better(ov, oi, gv, gi)) {
      gv = ov;
      gi = oi;
    }
  }
  __syncthreads();
  if (lane == 0) {
    red[warp] = gv;
    redi[warp] = gi;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < NW; ++w)
      if (argmax_better(red[w], redi[w], gv, gi)) {
        gv = red[w];
        gi = redi[w];
      }
    if (gi == 0x7fffffff) {  // every logit was NaN
      gi = 0;
      atomicOr(a.err, ERR_ARGMAX_NAN);
    }
    a.tok_w[pos + 1] = gi;
    a.ctrl[0] = pos + 1;
    *a.counter = 0u;
    __threadfence();
  }
  }
}

// Issue L2 prefetches covering this CTA's weight rows [r0, r0 + nrows).
__device__ __forceinline__ void prefetch_rows_l2(const RowMap& m, int r0, int nrows, int row_bytes) {
  auto piece = [&](const char* p, long long bytes) {
    for (long long off = 0; off < bytes; off += 32768)
      bulk_prefetch_l2(p + off, static_cast<uint32_t>(bytes - off < 32768 ? bytes - off : 32768));
  };
  if (m.interleave) {
    piece(m.base[0] + static_cast<size_t>(r0 >> 1) * row_bytes, static_cast<long long>(nrows >> 1) * row_bytes);
    piece(m.base[1] + static_cast<size_t>(r0 >> 1) * row_bytes, static_cast<long long>(nrows >> 1) * row_bytes);
    return;
  }
  const int r1 = r0 + nrows;
  const int lo[3] = {0, m.split1, m.split2};
  const int hi[3] = {m.split1, m.split2, 0x7fffffff};
  for (int k = 0; k < 3; ++k) {
    const int a = r0 > lo[k] ? r0 : lo[k];
    const int b = r1 < hi[k] ? r1 : hi[k];
    if (a < b) piece(m.base[k] + static_cast<size_t>(a - lo[k]) * row_bytes, static_cast<long long>(b - a) * row_bytes);
  }
}

// NW warps per CTA; each warp streams its segments through a ring of RING
// bytes cut into slots of a.seg_bytes (at most NSMAX slots).
template <typename WT, typename XT, int PRO, int EPI, int NW, int NSMAX, int RING>
__global__ void __launch_bounds__(NW * 32, 2) gemv_stream_kernel(const GemvArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int NT = NW * 32;
  unsigned char* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(NW) * RING);
  float* xs = reinterpret_cast<float*>(smem + gemv_ring_bytes<NW, NSMAX, RING>());
  float* part = xs + ((a.in + 3) & ~3);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int spr = a.segs_per_row;
  const int nunits = a.out / a.row_unit;
  const int G = gridDim.x, c = blockIdx.x;
  const int u0 = static_cast<int>(static_cast<int64_t>(c) * nunits / G);
  const int u1 = static_cast<int>(static_cast<int64_t>(c + 1) * nunits / G);
  const int r0 = u0 * a.row_unit;
  const int nrows = (u1 - u0) * a.row_unit;
  const int nseg = nrows * spr;
  float* red = part + ((nrows * spr + 3) & ~3);
  const int njobs = nseg > warp ? (nseg - warp + NW - 1) / NW : 0;
  const int ns = min(NSMAX, RING / a.seg_bytes);

  uint64_t* mybars = bars + warp * NSMAX;
  unsigned char* myring = ring + static_cast<size_t>(warp) * RING;
  const uint64_t pol = l2_policy_evict_first();

  auto issue = [&](int it) {
    const int k = warp + it * NW;
    const int row = r0 + k / spr, j = k % spr;
    const int off = j * a.seg_bytes;
    const uint32_t bytes = static_cast<uint32_t>(min(a.seg_bytes, a.row_bytes - off));
    const int slot = it % ns;
    mbar_arrive_expect_tx(&mybars[slot], bytes);
    bulk_g2s(myring + static_cast<size_t>(slot) * a.seg_bytes, row_ptr(a.w, row, a.row_bytes) + off, bytes,
             &mybars[slot], pol);
  };

  // Weights never depend on earlier kernels: start streaming them at once,
  // into this warp's ring and (for matrices that fit in L2) into L2.
  if (lane == 0) {
    for (int s = 0; s < ns; ++s) mbar_init(&mybars[s], 1);
    fence_mbar_init();
    const int first = njobs < ns ? njobs : ns;
    for (int it = 0; it < first; ++it) issue(it);
  }
  if (tid == 0 && a.l2_prefetch && nrows > 0) prefetch_rows_l2(a.w, r0, nrows, a.row_bytes);
  __syncwarp();
  pdl_trigger();
  pdl_wait();

  // ---- activation vector (and fused RMSNorm) ----
  int pos = 0;
  if (PRO == PRO_EMBED_NORM || EPI == EPI_ARGMAX) pos = a.ctrl[0];
  if (PRO == PRO_X) {
    for (int i = tid; i < a.in; i += NT) xs[xs_index<WT>(i, a.in)] = load_f32<XT>(a.x, i);
  } else {
    const void* src = a.x;
    bool src_is_w = false;
    if (PRO == PRO_EMBED_NORM) {
      int t = a.tok[pos];
      if (t < 0 || t >= a.vocab) {
        if (tid == 0) atomicOr(a.err, ERR_BAD_TOKEN);
        t = 0;
      }
      src = static_cast<const WT*>(a.embed) + static_cast<size_t>(t) * a.in;
      src_is_w = true;
    }
    float ss = 0.f;
    for (int i = tid; i < a.in; i += NT) {
      const float v = src_is_w ? load_f32<WT>(src, i) : static_cast<const float*>(src)[i];
      if (PRO == PRO_EMBED_NORM && c == 0) a.h_out[i] = v;
      xs[xs_index<WT>(i, a.in)] = v;
      ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (warp == 0) {
      float t = lane < NW ? red[lane] : 0.f;
      t = warp_sum(t);
      if (lane == 0) red[NW] = 1.0f / sqrtf(t / static_cast<float>(a.in) + a.eps);
    }
    __syncthreads();
    const float inv = red[NW];
    for (int i = tid; i < a.in; i += NT) {
      const int k = xs_index<WT>(i, a.in);
      xs[k] = xs[k] * inv * a.norm_g[i];
    }
  }
  __syncthreads();

  // ---- stream this warp's segments ----
  int fail_it = -1;
  for (int it = 0; it < njobs; ++it) {
    const int slot = it % ns;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&mybars[slot], (it / ns) & 1));
    if (!ok) {
      fail_it = it;
      break;
    }
    const int k = warp + it * NW;
    const int j = k % spr;
    const int off = j * a.seg_bytes;
    const int bytes = min(a.seg_bytes, a.row_bytes - off);
    float v = seg_dot<WT>(myring + static_cast<size_t>(slot) * a.seg_bytes, xs, off / static_cast<int>(sizeof(WT)),
                          bytes, a.in, lane);
    v = warp_sum(v);
    if (lane == 0) part[k] = v;
    __syncwarp();
    if (lane == 0 && it + ns < njobs) {
      fence_proxy_async_smem();
      issue(it + ns);
    }
  }
  if (fail_it >= 0) {
    if (lane == 0) atomicOr(a.err, ERR_MBAR_TIMEOUT);
    // Drain copies still in flight into this warp's ring before the CTA exits.
    const int last = min(njobs, fail_it + ns);
    for (int it = fail_it + 1; it < last; ++it) mbar_wait(&mybars[it % ns], (it / ns) & 1);
  }
  __syncthreads();

  // ---- epilogue ----
  if constexpr (EPI == EPI_SWIGLU) {
    for (int i = tid; i < nrows / 2; i += NT) {
      float g = 0.f, u = 0.f;
      for (int j = 0; j < spr; ++j) g += part[(2 * i) * spr + j];
      for (int j = 0; j < spr; ++j) u += part[(2 * i + 1) * spr + j];
      a.y[r0 / 2 + i] = silu_f32(g) * u;
    }
  } else {
    rows_epilogue<EPI>(a, part, red, nrows, spr, r0, pos, c, G, tid, warp, lane, NT, NW);
  }
}

}  // namespace wsg
