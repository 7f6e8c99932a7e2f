// 4-bit groupwise-affine GEMV streamed by bulk copies ("Our Kernel Benchmark
// Was Measuring the System Cache", Summary and "Why it mattered, concretely":
// the one-token matvec and its two-token variant, measured cold).
//
//  * Each CTA owns a contiguous range of rows. Its codes ([rows][in/8] u32)
//    and its scales and biases ([rows][in/64] fp16) are three contiguous
//    byte ranges, so one producer lane streams them with plain 1D bulk copies
//    into a ring of stages of up to RC = 8 * R rows (one full/empty mbarrier
//    pair per stage). The copies start before the kernel waits on its predecessor
//    (programmatic dependent launch): the weights of a launch do not depend
//    on earlier kernels, only x does.
//  * 8 consumer warps: warp w takes rows w, w + 8, ... (R of them) of every
//    stage, lane l the 32-column chunks l, l + 32, ... of those rows; one
//    16-byte shared load brings a row's 32 codes of a chunk, and a chunk is
//    half of a 64-column group, so it has one scale s and bias b. The CTA is
//    sized for two per SM: large matrices run two per SM, small ones one, so
//    the next launch's CTAs can start their copies beside it.
//  * Integer dot products. Per chunk and token, x is written in 16-bit fixed
//    point with the power-of-two step u = 2^(e-14), 2^e <= max|x| < 2^(e+1):
//    xi = rint(x / u) clamped to [-32768, 32767], split into a signed high
//    byte and an unsigned low byte (xi = 256 hi + lo). A bfloat16 x whose
//    exponent is at least e - 7 is represented exactly (|xi| <= 32640, the
//    clamp never acts); smaller ones are within u/2, i.e. 2^-15 of the
//    chunk's largest |x|. A float32 x is within u/2 as well, or within u where
//    the clamp acts (only values within 2^-16 of 2^(e+1)). The codes need no
//    conversion:
//    lo = word & 0x0F0F0F0F holds the even columns' codes and
//    hi = word & 0xF0F0F0F0 16 times the odd columns' codes, one per byte, so
//    four 4-way byte dot products (dp4a) per word accumulate exact integer sums
//    against the matching x byte planes, and
//    16 sum q xi = 16 (256 He + Le) + 256 Ho + Lo (below 2^28).
//    The chunk adds s * u/16 * (that sum) + b * X to the row, X the chunk's
//    float sum of x. All staged once per CTA.
//  * A warp owns whole rows: a butterfly reduce-scatter over its lanes gives
//    each row's sum, which one lane stores. No cross-warp sums: results are
//    bit-reproducible.
//
//  * The rows may come from up to three matrices (segments; the 4-bit decoder
//    runs Q/K/V, and gate/up, as one launch): each segment gets its own run of
//    CTAs, in proportion to its rows, and writes its own range of y.
//  * x prologues (XM): bfloat16 x read as is (the standalone product); float32
//    x; x = RMSNorm(h) * g from a float32 residual row h; x = silu(gate) * up
//    from float32 gate/up rows. The float32 forms go straight into the
//    fixed-point planes: the decoder's activations are never rounded to a
//    16-bit float. Epilogues: y = W x or y += W x (residual add).
//
// Every mbarrier wait is bounded; on a timeout the CTA raises an abort flag,
// the producer waits (bounded) for its copies in flight, and the error word
// records the cause.
#pragma once
#include <cuda_fp16.h>

#include <cstdint>
#include <string>

#include "common.h"
#include "gemv_stream.cuh"  // silu_f32
#include "megakernel.cuh"   // reduce_scatter
#include "ptx.cuh"

namespace wsg {

constexpr int kQ4Warps = 8;                     // consumer warps
constexpr int kQ4Threads = kQ4Warps * 32 + 32;  // plus a producer warp
constexpr int kQ4MaxStages = 16;
constexpr int kQ4MaxSegs = 3;

enum Q4X : int {
  Q4X_BF16 = 0,    // x bf16 [ntok][x_ld]
  Q4X_F32 = 1,     // x f32 [ntok][x_ld]
  Q4X_NORM = 2,    // x = h * rsqrt(mean(h^2) + eps) * g, h f32 [ntok][x_ld]
  Q4X_SWIGLU = 3,  // x = silu(gu[j]) * gu[in + j], gu f32 [ntok][x_ld]
};

enum Q4Epi : int {
  Q4E_STORE = 0,  // y = W x
  Q4E_ADD = 1,    // y += W x
};

struct Q4Seg {
  const uint32_t* codes;  // [rows][in/8]
  const uint16_t* scale;  // fp16 [rows][in/64]
  const uint16_t* bias;   // fp16 [rows][in/64]
  int32_t rows;
  int32_t y_off;          // first row of y this segment writes
  int32_t cta0;           // first CTA of this segment (segment 0: 0)
};

struct Q4Args {
  Q4Seg seg[kQ4MaxSegs];
  int32_t nseg;
  const void* x;          // per the x prologue; row t starts at x + t * x_ld elements
  int32_t x_ld;
  const float* norm_g;    // Q4X_NORM: gain [in]
  float eps;
  float* y;               // y[t * ldy + y_off + row]
  int32_t ldy, in;
  int32_t nstages;        // ring depth
  int32_t srows;          // row capacity of a stage: min(RC, most rows of a CTA)
  uint32_t stage_bytes;   // one stage: srows rows of codes, then of scales, then of biases (multiple of 128)
  uint32_t* err;
};

// Host description of one bulk 4-bit launch (gemv.cu builds the Q4Args).
struct Q4Launch {
  Q4Seg seg[kQ4MaxSegs];  // rows, y_off and pointers; cta0 is chosen by the launcher
  int32_t nseg;
  int32_t xm, epi, ntok;  // Q4X_*, Q4E_*, 1 or 2
  const void* x;
  int32_t x_ld;
  const float* norm_g;
  float eps;
  float* y;
  int32_t ldy, in;
  bool pdl;
  uint32_t* err;
};

// A 4-bit projection of the decoder (prologue / epilogue pairs NORM+STORE,
// F32+ADD, SWIGLU+ADD). DEC_EINVAL when the shape does not fit the bulk kernel.
dec_status launch_q4_fused(const Q4Launch& q, cudaStream_t st, std::string* err);

__device__ __forceinline__ void q4_consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kQ4Warps * 32) : "memory");
}

// 4-way byte dot products: c + sum_k a.byte[k] * b.byte[k], a unsigned and b
// signed (us) or both unsigned (uu).
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Word m (columns 32 ch + 8 m .. + 7, float32 values xv) of
// token t's byte planes of chunk ch: four consecutive lanes hold the four words
// of a chunk and reduce its largest |x| and its sum by shuffles, so every lane
// of the warp calls this (valid: the item exists).
__device__ __forceinline__ void q4_item_planes(const float (&xv)[8], int t, int ch, int m, int nch, bool valid,
                                               uint4* xq, float2* xu) {
  float mx = 0.f, X = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    mx = fmaxf(mx, fabsf(xv[j]));
    X += xv[j];
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    X += __shfl_xor_sync(0xffffffffu, X, o);
  }
  int e = 0;
  if (mx > 0.f) {
    frexpf(mx, &e);  // mx = f 2^e, f in [0.5, 1): 2^(e-1) <= mx < 2^e
    e -= 1;
  }
  uint32_t he = 0, le = 0, ho = 0, lo = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    // |x| < 2^(e+1) puts x / u below 2^15; a float32 x within 2^-16 of that
    // rounds to 32768, one past the signed 16-bit range, hence the clamp
    const int xe = mx > 0.f ? min(static_cast<int>(rintf(scalbnf(xv[2 * k], 14 - e))), 32767) : 0;
    const int xo = mx > 0.f ? min(static_cast<int>(rintf(scalbnf(xv[2 * k + 1], 14 - e))), 32767) : 0;
    he |= (static_cast<uint32_t>(xe >> 8) & 0xFFu) << (8 * k);
    le |= (static_cast<uint32_t>(xe) & 0xFFu) << (8 * k);
    ho |= (static_cast<uint32_t>(xo >> 8) & 0xFFu) << (8 * k);
    lo |= (static_cast<uint32_t>(xo) & 0xFFu) << (8 * k);
  }
  if (valid) {
    uint32_t* w = reinterpret_cast<uint32_t*>(xq + t * 4 * nch + ch) + m;  // word m of plane 0
    w[0] = he;
    w[4 * nch] = le;
    w[8 * nch] = ho;
    w[12 * nch] = lo;
    if (m == 0) xu[t * nch + ch] = make_float2(mx > 0.f ? scalbnf(1.0f, e - 18) : 0.f, X);
  }
}

// Consumers (threads 0 .. kQ4Warps * 32 - 1): per chunk of 32 columns and
// token, the fixed-point step, the byte planes and the float sum of x, built
// by the x prologue XM; ends with a consumer barrier.
template <int NTOK, int XM>
__device__ __forceinline__ void q4_stage_x(const void* xp, int x_ld, const float* norm_g, float eps, int in, uint4* xq,
                                           float2* xu, float* s_rs, int tid) {
  const int warp = tid >> 5, lane = tid & 31, nch = in >> 5;
  // One token of at most 8 columns per thread: the first pass reads exactly
  // this thread's staging item (columns 8 tid .. 8 tid + 7) and keeps it.
  constexpr bool kOne = XM == Q4X_NORM && NTOK == 1;
  const bool keep = kOne && in <= 8 * kQ4Warps * 32;
  float hv[8];
  if (XM == Q4X_NORM) {
    // 1 / RMS of each token's h, summed in a fixed order
    const float* h = static_cast<const float*>(xp);
    for (int t = 0; t < NTOK; ++t) {
      float ss = 0.f;
      if (keep) {
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
        if (8 * tid < in) {
          v0 = __ldcg(reinterpret_cast<const float4*>(h + 8 * tid));
          v1 = __ldcg(reinterpret_cast<const float4*>(h + 8 * tid + 4));
        }
        hv[0] = v0.x, hv[1] = v0.y, hv[2] = v0.z, hv[3] = v0.w;
        hv[4] = v1.x, hv[5] = v1.y, hv[6] = v1.z, hv[7] = v1.w;
#pragma unroll
        for (int j = 0; j < 8; ++j) ss = fmaf(hv[j], hv[j], ss);
      } else {
        for (int i = 4 * tid; i < in; i += 4 * kQ4Warps * 32) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(h + static_cast<size_t>(t) * x_ld + i));
          ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
        }
      }
      ss = warp_sum(ss);
      if (lane == 0) s_rs[t * kQ4Warps + warp] = ss;
    }
    q4_consumer_sync();
  }
  float rs[NTOK];
  if (XM == Q4X_NORM) {
#pragma unroll
    for (int t = 0; t < NTOK; ++t) {
      float ss = 0.f;
      for (int w = 0; w < kQ4Warps; ++w) ss += s_rs[t * kQ4Warps + w];
      rs[t] = rsqrtf(ss / static_cast<float>(in) + eps);
    }
  }
  // x: per chunk and token, the fixed point step, the byte planes and the
  // float sum. Four consecutive lanes per chunk, lane m taking the 8 columns
  // of word m and building that word of all four planes; the butterfly max
  // and sum over the four lanes leave the same value in each.
  {
    const int items = NTOK * nch * 4;
    for (int it0 = warp * 32; it0 < items; it0 += kQ4Warps * 32) {
      const int it = it0 + lane;
      const bool valid = it < items;
      const int t = valid ? it / (nch * 4) : 0, rem = it - t * nch * 4, ch = rem >> 2, m = rem & 3;
      const int col = 32 * ch + 8 * m;
      float xv[8];
      if (XM == Q4X_BF16) {
        uint4 u = make_uint4(0, 0, 0, 0);
        if (valid)
          u = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(xp) + static_cast<size_t>(t) * x_ld +
                                                    col));
        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          xv[2 * k] = __uint_as_float(uw[k] << 16);              // column 8m + 2k
          xv[2 * k + 1] = __uint_as_float(uw[k] & 0xFFFF0000u);  // column 8m + 2k + 1
        }
      } else {
        const float* xr = static_cast<const float*>(xp) + static_cast<size_t>(t) * x_ld + col;
        float f[8];
        if (keep) {  // item it == tid: this thread's columns from the first pass
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = hv[j];
        } else {
          float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
          if (valid) {
            v0 = __ldcg(reinterpret_cast<const float4*>(xr));
            v1 = __ldcg(reinterpret_cast<const float4*>(xr + 4));
          }
          f[0] = v0.x, f[1] = v0.y, f[2] = v0.z, f[3] = v0.w;
          f[4] = v1.x, f[5] = v1.y, f[6] = v1.z, f[7] = v1.w;
        }
        if (XM == Q4X_NORM) {
          float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0;
          if (valid) {
            g0 = __ldg(reinterpret_cast<const float4*>(norm_g + col));
            g1 = __ldg(reinterpret_cast<const float4*>(norm_g + col + 4));
          }
          const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          float r = rs[0];
#pragma unroll
          for (int tt = 1; tt < NTOK; ++tt)
            if (t == tt) r = rs[tt];
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = (f[j] * r) * g[j];
        } else if (XM == Q4X_SWIGLU) {
          float4 u0 = make_float4(0.f, 0.f, 0.f, 0.f), u1 = u0;
          if (valid) {
            u0 = __ldcg(reinterpret_cast<const float4*>(xr + in));
            u1 = __ldcg(reinterpret_cast<const float4*>(xr + in + 4));
          }
          const float up[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = silu_f32(f[j]) * up[j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) xv[j] = f[j];
      }
      q4_item_planes(xv, t, ch, m, nch, valid, xq, xu);
    }
  }
  q4_consumer_sync();
}

// Consumers: add the chunk's row sums (rows w, w + 8, ... of warp w; lane
// partials) for every token to acc[i * NTOK + t]. base: the chunk's codes
// [rows][cb], then scales and biases [rows][sbb] at sbase and bbase.
template <int R, int NTOK>
__device__ __forceinline__ void q4_chunk_dot(const unsigned char* base, const unsigned char* sbase,
                                             const unsigned char* bbase, int rows, uint32_t cb, uint32_t sbb, int nch,
                                             const uint4* xq, const float2* xu, int warp, int lane,
                                             float (&acc)[R * NTOK]) {
    for (int ch = lane; ch < nch; ch += 32) {
      uint4 q[R];
      float s[R], b[R];
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const int rr = warp + kQ4Warps * i;
        if (rr < rows) {
          q[i] = *reinterpret_cast<const uint4*>(base + rr * cb + 16 * ch);
          s[i] = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(sbase + rr * sbb + 2 * (ch >> 1))));
          b[i] = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(bbase + rr * sbb + 2 * (ch >> 1))));
        } else {
          q[i] = make_uint4(0, 0, 0, 0);
          s[i] = b[i] = 0.f;
        }
      }
#pragma unroll
      for (int t = 0; t < NTOK; ++t) {
        const uint4 phe = xq[(t * 4 + 0) * nch + ch], ple = xq[(t * 4 + 1) * nch + ch];
        const uint4 pho = xq[(t * 4 + 2) * nch + ch], plo = xq[(t * 4 + 3) * nch + ch];
        const float2 xs = xu[t * nch + ch];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          int he = 0, ho = 0;
          uint32_t le = 0, lo = 0;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t w = m == 0 ? q[i].x : m == 1 ? q[i].y : m == 2 ? q[i].z : q[i].w;
            const uint32_t ev = w & 0x0F0F0F0Fu;  // q of columns 8m, 8m+2, 8m+4, 8m+6
            const uint32_t od = w & 0xF0F0F0F0u;  // 16 q of columns 8m+1, 8m+3, 8m+5, 8m+7
            const uint32_t xhe = m == 0 ? phe.x : m == 1 ? phe.y : m == 2 ? phe.z : phe.w;
            const uint32_t xle = m == 0 ? ple.x : m == 1 ? ple.y : m == 2 ? ple.z : ple.w;
            const uint32_t xho = m == 0 ? pho.x : m == 1 ? pho.y : m == 2 ? pho.z : pho.w;
            const uint32_t xlo = m == 0 ? plo.x : m == 1 ? plo.y : m == 2 ? plo.z : plo.w;
            he = dp4a_us(ev, xhe, he);
            le = dp4a_uu(ev, xle, le);
            ho = dp4a_us(od, xho, ho);
            lo = dp4a_uu(od, xlo, lo);
          }
          // 16 sum q xi, exact (below 2^28 in magnitude)
          const int tot = 16 * (256 * he + static_cast<int>(le)) + 256 * ho + static_cast<int>(lo);
          acc[i * NTOK + t] = fmaf(s[i] * xs.x, static_cast<float>(tot), fmaf(b[i], xs.y, acc[i * NTOK + t]));
        }
      }
    }
}

// Shared memory: [ring: nstages x stage_bytes][xq: NTOK][4][nch] uint4 (the byte
// planes of chunk c: high bytes of the even columns, low bytes of the even
// columns, high and low bytes of the odd columns; word m of a plane holds
// columns 32c + 8m + (0, 2, 4, 6) or + (1, 3, 5, 7))[xu: NTOK][nch] float2
// (u / 16, X)][full: nstages][empty: nstages] mbarriers.
template <int R, int NTOK, int XM = Q4X_BF16, int EPI = Q4E_STORE>
__global__ void __launch_bounds__(kQ4Threads, 2) gemv_q4_bulk_kernel(const Q4Args a) {
  constexpr int RC = kQ4Warps * R;
  constexpr int NV = R * NTOK;  // row sums per lane before the reduction
  constexpr int kLogNV = NV == 1 ? 0 : NV == 2 ? 1 : NV == 4 ? 2 : NV == 8 ? 3 : 4;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_abort;
  __shared__ float s_rs[kQ4Warps * NTOK];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int in = a.in, nch = in >> 5;
  const uint32_t cb = static_cast<uint32_t>(in) >> 1;   // code bytes per row
  const uint32_t sbb = static_cast<uint32_t>(in) >> 5;  // scale (or bias) bytes per row
  const int S = a.nstages;
  unsigned char* ring = smem;
  uint4* xq = reinterpret_cast<uint4*>(smem + static_cast<size_t>(S) * a.stage_bytes);
  float2* xu = reinterpret_cast<float2*>(xq + NTOK * 4 * nch);
  uint64_t* full = reinterpret_cast<uint64_t*>(xu + NTOK * nch);
  uint64_t* empty = full + S;
  volatile int* vabort = &s_abort;
  // this CTA's segment, and its rows [r0, r0 + n) of that segment
  int k = 0;
  while (k + 1 < a.nseg && static_cast<int>(blockIdx.x) >= a.seg[k + 1].cta0) ++k;
  const Q4Seg sg = a.seg[k];
  const int c = blockIdx.x - sg.cta0;
  const int G = (k + 1 < a.nseg ? a.seg[k + 1].cta0 : static_cast<int>(gridDim.x)) - sg.cta0;
  const int r0 = static_cast<int>(static_cast<long long>(c) * sg.rows / G);
  const int n = static_cast<int>(static_cast<long long>(c + 1) * sg.rows / G) - r0;
  const int nst = (n + RC - 1) / RC;
  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kQ4Warps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();

  // ---- producer: one lane streams the CTA's stages ----
  if (warp == kQ4Warps) {
    if (lane != 0) return;
    const uint64_t pol = l2_policy_evict_first();
    const char* codes = reinterpret_cast<const char*>(sg.codes);
    const char* sc = reinterpret_cast<const char*>(sg.scale);
    const char* bi = reinterpret_cast<const char*>(sg.bias);
    int issued = 0;
    for (int st = 0; st < nst; ++st) {
      const int slot = st % S;
      if (st >= S && !mbar_wait(&empty[slot], ((st / S) - 1) & 1)) {
        *vabort = 1;
        atomicOr(a.err, ERR_MBAR_TIMEOUT);
      }
      if (*vabort) break;
      const int row = r0 + st * RC, rows = min(RC, n - st * RC);
      unsigned char* dst = ring + static_cast<size_t>(slot) * a.stage_bytes;
      mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(rows) * (cb + 2 * sbb));
      bulk_g2s(dst, codes + static_cast<size_t>(row) * cb, rows * cb, &full[slot], pol);
      bulk_g2s(dst + a.srows * cb, sc + static_cast<size_t>(row) * sbb, rows * sbb, &full[slot], pol);
      bulk_g2s(dst + a.srows * (cb + sbb), bi + static_cast<size_t>(row) * sbb, rows * sbb, &full[slot], pol);
      ++issued;
    }
    // After an abort: shared memory must outlive the copies already issued.
    if (*vabort)
      for (int k = max(0, issued - S); k < issued; ++k) mbar_wait(&full[k % S], (k / S) & 1);
    return;
  }

  // ---- consumers ----
  // x may come from the previous kernel, and y may still be read by it.
  pdl_wait();
  q4_stage_x<NTOK, XM>(a.x, a.x_ld, a.norm_g, a.eps, in, xq, xu, s_rs, tid);

  bool ok = true;
  for (int st = 0; st < nst && ok; ++st) {
    const int slot = st % S;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], (st / S) & 1));
    if (!ok) {
      if (lane == 0) atomicOr(a.err, ERR_MBAR_TIMEOUT);
      *vabort = 1;
      break;
    }
    const int rows = min(RC, n - st * RC);
    const unsigned char* base = ring + static_cast<size_t>(slot) * a.stage_bytes;
    const unsigned char* sbase = base + a.srows * cb;
    const unsigned char* bbase = sbase + a.srows * sbb;
    float acc[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[v] = 0.f;
    q4_chunk_dot<R, NTOK>(base, sbase, bbase, rows, cb, sbb, nch, xq, xu, warp, lane, acc);
    // every lane's reads of the stage are in registers: release it
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    const float v = reduce_scatter<NV>(acc, lane);
    const int vi = lane >> (5 - kLogNV), i = vi / NTOK, t = vi - i * NTOK;
    const int rr = warp + kQ4Warps * i;
    if ((lane & ((32 >> kLogNV) - 1)) == 0 && rr < rows) {
      float* yp = a.y + static_cast<size_t>(t) * a.ldy + sg.y_off + r0 + st * RC + rr;
      if (EPI == Q4E_ADD)
        *yp += v;
      else
        *yp = v;
    }
  }
}

}  // namespace wsg
