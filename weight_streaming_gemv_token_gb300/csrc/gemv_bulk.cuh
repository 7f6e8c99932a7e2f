// Standalone GEMV y = W x for float32 or bfloat16 W ("Our Kernel Benchmark
// Was Measuring the System Cache", Summary: the product whose cold weight
// stream is measured), streamed by plain bulk copies:
//
//  * each CTA owns a contiguous range of rows, which is one contiguous byte
//    range of the row-major W; a producer lane copies it stage by stage
//    (srows rows per stage, one 1D bulk copy) into a ring of shared memory
//    (one full/empty mbarrier pair per stage), starting before the kernel
//    waits on its predecessor (programmatic dependent launch): W never
//    depends on earlier kernels, only x does;
//  * the CTA is sized so two fit on an SM: large matrices run two per SM,
//    small ones one, so the next launch's CTAs can start their copies beside
//    it and its weight stream overlaps this launch's tail;
//  * 8 consumer warps: warp w takes rows w, w + 8, ... (R of them) of every
//    stage; lane l reads 16 bytes of the row per pass (4 float32 or 8
//    bfloat16 weights) and the matching float32 x from shared memory, with
//    packed FP32 FMAs (even / odd columns); a butterfly reduce-scatter over
//    the warp gives each row's sum, stored by one lane. No cross-warp sums:
//    bit-reproducible.
//
// Every mbarrier wait is bounded; on a timeout the CTA raises an abort flag,
// the producer waits (bounded) for its copies in flight, and the error word
// records the cause.
#pragma once
#include <cstdint>

#include "megakernel.cuh"  // reduce_scatter
#include "ptx.cuh"

namespace wsg {

constexpr int kGbWarps = 8;                     // consumer warps
constexpr int kGbThreads = kGbWarps * 32 + 32;  // plus a producer warp
constexpr int kGbMaxStages = 16;

struct GbArgs {
  const void* W;  // [out][in], row bytes a multiple of 16
  const void* x;  // [in], float32 (W float32) or bfloat16 (W bfloat16)
  float* y;       // [out]
  int32_t out, in;
  int32_t nstages;       // ring depth
  int32_t srows;         // rows per stage (at most 8 R)
  uint32_t stage_bytes;  // srows rows, rounded up to 128
  uint32_t* err;
};

__device__ __forceinline__ void gb_consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGbWarps * 32) : "memory");
}

// Shared memory: [ring: nstages x stage_bytes][x: float32, laid out per pass
// p of E * 32 columns as [p][E / 4][32 lanes] float4][full: nstages][empty: nstages].
template <typename WT, int R>
__global__ void __launch_bounds__(kGbThreads, 2) gemv_bulk_kernel(const GbArgs a) {
  constexpr int E = 16 / static_cast<int>(sizeof(WT));  // weights per 16 bytes
  constexpr int H = E / 4;                              // float4 of x per lane and pass
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int in = a.in, np = (in + 32 * E - 1) / (32 * E);  // passes per row
  const uint32_t rb = static_cast<uint32_t>(in) * sizeof(WT);
  const int S = a.nstages, SR = a.srows;
  unsigned char* ring = smem;
  float4* xs = reinterpret_cast<float4*>(smem + static_cast<size_t>(S) * a.stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(xs + np * H * 32);
  uint64_t* empty = full + S;
  volatile int* vabort = &s_abort;
  const int c = blockIdx.x, G = gridDim.x;
  const int r0 = static_cast<int>(static_cast<long long>(c) * a.out / G);
  const int n = static_cast<int>(static_cast<long long>(c + 1) * a.out / G) - r0;
  const int nst = (n + SR - 1) / SR;
  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGbWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();

  // ---- producer: one lane streams the CTA's rows ----
  if (warp == kGbWarps) {
    if (lane != 0) return;
    const uint64_t pol = l2_policy_evict_first();
    const char* src = static_cast<const char*>(a.W) + static_cast<size_t>(r0) * rb;
    int issued = 0;
    for (int st = 0; st < nst; ++st) {
      const int slot = st % S;
      if (st >= S && !mbar_wait(&empty[slot], ((st / S) - 1) & 1)) {
        *vabort = 1;
        atomicOr(a.err, ERR_MBAR_TIMEOUT);
      }
      if (*vabort) break;
      const int rows = min(SR, n - st * SR);
      mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(rows) * rb);
      bulk_g2s(ring + static_cast<size_t>(slot) * a.stage_bytes, src + static_cast<size_t>(st) * SR * rb,
               static_cast<uint32_t>(rows) * rb, &full[slot], pol);
      ++issued;
    }
    // After an abort: shared memory must outlive the copies already issued.
    if (*vabort)
      for (int k = max(0, issued - S); k < issued; ++k) mbar_wait(&full[k % S], (k / S) & 1);
    return;
  }

  // ---- consumers ----
  // x (it may come from the previous kernel) as float32 in the pass layout:
  // column 32 E p + E l + 4 h + j sits in float4 (p H + h) * 32 + l, element j.
  pdl_wait();
  for (int i = tid; i < np * H * 32; i += kGbWarps * 32) {
    const int l = i & 31, ph = i >> 5, p = ph / H, h = ph - p * H;
    const int col = 32 * E * p + E * l + 4 * h;
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = col + j < in ? load_f32<WT>(static_cast<const WT*>(a.x), col + j) : 0.f;
    xs[i] = make_float4(v[0], v[1], v[2], v[3]);
  }
  gb_consumer_sync();

  bool ok = true;
  for (int st = 0; st < nst && ok; ++st) {
    const int slot = st % S;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], (st / S) & 1));
    if (!ok) {
      if (lane == 0) atomicOr(a.err, ERR_MBAR_TIMEOUT);
      *vabort = 1;
      break;
    }
    const int rows = min(SR, n - st * SR);
    const unsigned char* base = ring + static_cast<size_t>(slot) * a.stage_bytes;
    float ae[R], ao[R];  // even / odd columns of each row
#pragma unroll
    for (int i = 0; i < R; ++i) ae[i] = ao[i] = 0.f;
    for (int p = 0; p < np; ++p) {
      const int col = 32 * E * p + E * lane;
      if (col < in) {
        float4 xv[H];
#pragma unroll
        for (int h = 0; h < H; ++h) xv[h] = xs[(p * H + h) * 32 + lane];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const int rr = warp + kGbWarps * i;
          if (rr < rows) {
            const uint4 w = *reinterpret_cast<const uint4*>(base + rr * rb + static_cast<uint32_t>(col) * sizeof(WT));
            if constexpr (E == 4) {
              ffma2(ae[i], ao[i], __uint_as_float(w.x), __uint_as_float(w.y), xv[0].x, xv[0].y);
              ffma2(ae[i], ao[i], __uint_as_float(w.z), __uint_as_float(w.w), xv[0].z, xv[0].w);
            } else {
              ffma2(ae[i], ao[i], __uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), xv[0].x, xv[0].y);
              ffma2(ae[i], ao[i], __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u), xv[0].z, xv[0].w);
              ffma2(ae[i], ao[i], __uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u), xv[H - 1].x,
                    xv[H - 1].y);
              ffma2(ae[i], ao[i], __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u), xv[H - 1].z,
                    xv[H - 1].w);
            }
          }
        }
      }
    }
    // every lane's reads of the stage are in registers: release it
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    float acc[R];
#pragma unroll
    for (int i = 0; i < R; ++i) acc[i] = ae[i] + ao[i];
    constexpr int kLogR = R == 1 ? 0 : R == 2 ? 1 : R == 4 ? 2 : 3;
    const float v = reduce_scatter<R>(acc, lane);
    const int i = lane >> (5 - kLogR), rr = warp + kGbWarps * i;
    if ((lane & ((32 >> kLogR) - 1)) == 0 && rr < rows) a.y[r0 + st * SR + rr] = v;
  }
}

}  // namespace wsg
