// Standalone GEMV y = W x ("Our Kernel Benchmark Was Measuring the System
// Cache", Summary: the product whose cold weight stream is measured), built
// from the persistent decode kernel's machinery as a single stage:
//
//  * each CTA owns a contiguous range of rows; the columns are cut into
//    8 (or 16) parts and consumer warp w owns parts w (and w + 8) of every
//    row (split-K), holding the matching x elements in registers;
//  * a producer warp streams each warp's parts as tiled TMA boxes (R rows x
//    one part) into the warp's byte ring (full/empty mbarrier per box in
//    flight), starting before the kernel waits on its predecessor
//    (programmatic dependent launch): weights never depend on earlier kernels,
//    so a launch's stream overlaps the previous launch's tail, and shared
//    memory is sized for two CTAs per SM so the next launch's CTAs can start;
//  * per box every lane accumulates one partial per row, a butterfly
//    reduce-scatter makes per-warp row sums, and the 8 warp sums of a row are
//    added in a fixed order (bit-reproducible) into y.
#pragma once
#include <cuda.h>

#include <cstdint>

#include "megakernel.cuh"

namespace wsg {

constexpr int kGtWarps = 8, kGtThreads = kGtWarps * 32 + 32, kGtQ = 8, kGtPartRows = 256;

struct GtArgs {
  const void* x;
  float* y;
  int32_t out, in;
  MkGeom gm;
  int32_t ring_bytes;  // per consumer warp, multiple of 128
  uint32_t* err;
};

template <typename WT>
__global__ void __launch_bounds__(kGtThreads, 2) gemv_tma_kernel(const __grid_constant__ CUtensorMap mapW,
                                                                 const GtArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_abort;
  const uint32_t RB = static_cast<uint32_t>(a.ring_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(kGtWarps) * RB);
  uint64_t* empty = full + kGtWarps * kGtQ;
  float* part = reinterpret_cast<float*>(empty + kGtWarps * kGtQ);  // [kGtPartRows][8]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;
  const int u0 = static_cast<int>(static_cast<long long>(c) * a.out / G);
  const int u1 = static_cast<int>(static_cast<long long>(c + 1) * a.out / G);
  const int nrows = u1 - u0;
  const MkGeom& gm = a.gm;
  const int R = gm.R, pw = gm.pw, cw = gm.cw;
  const int ng = (nrows + R - 1) / R;
  const int wpp = mk_wpp(gm), np = kGtWarps / wpp;  // warps per part, parts
  // boxes of warp w: its part's boxes of the row groups with index % wpp == w / np
  auto boxes_of = [&](int w) { const int sub = w / np; return (ng > sub ? (ng - sub + wpp - 1) / wpp : 0) * pw; };
  const uint32_t B = (static_cast<uint32_t>(gm.box_bytes) + 127u) & ~127u;
  volatile int* vabort = &s_abort;
  if (tid < kGtWarps * kGtQ) {
    mbar_init(&full[tid], 1);
    mbar_init(&empty[tid], 1);
    fence_mbar_init();
  }
  if (tid == 0) s_abort = 0;
  __syncthreads();
  pdl_trigger();

  if (warp == kGtWarps) {
    // ---- producer: lane w feeds warp w's byte ring (the decode kernel's placement rule) ----
    const int w = lane;
    const bool active = w < kGtWarps;
    uint64_t* wfull = full + (active ? w : 0) * kGtQ;
    uint64_t* wempty = empty + (active ? w : 0) * kGtQ;
    unsigned char* wring = smem + static_cast<size_t>(active ? w : 0) * RB;
    const uint64_t pol = l2_policy_evict_first();
    uint32_t vhead = 0, phead = 0;
    uint32_t qv[kGtQ];
#pragma unroll
    for (int i = 0; i < kGtQ; ++i) qv[i] = 0;
    int issued = 0, retired = 0;
    const int total = active ? boxes_of(w) : 0;
    const int wpart = w % np, wsub = w / np;
    uint64_t idle_since = 0;
    while (__any_sync(0xffffffffu, issued < total || retired < issued)) {
      bool progress = false;
      while (retired < issued && mbar_test(&wempty[retired % kGtQ], (retired / kGtQ) & 1)) {
#pragma unroll
        for (int i = 0; i + 1 < kGtQ; ++i) qv[i] = qv[i + 1];
        ++retired;
        progress = true;
      }
      while (issued < total && issued - retired < kGtQ) {
        uint32_t v = vhead, ph = phead;
        if (ph + B > RB) {
          v += RB - ph;
          ph = 0;
        }
        const int n = issued - retired;
        if (n > 0 && v + B - qv[0] > RB) break;
        const int li = pw == 2 ? (issued >> 1) : issued, pj = issued - li * pw;
        const int rg = wsub + wpp * li;
        const int q = issued % kGtQ;
        mbar_arrive_expect_tx(&wfull[q], static_cast<uint32_t>(gm.box_bytes));
        tma_load_2d(wring + ph, &mapW, (wpart + np * pj) * cw, u0 + rg * R, &wfull[q], pol);
#pragma unroll
        for (int i = 0; i < kGtQ; ++i)
          if (i == n) qv[i] = v;
        vhead = v + B;
        phead = ph + B;
        ++issued;
        progress = true;
      }
      if (__any_sync(0xffffffffu, progress)) {
        idle_since = 0;
        continue;
      }
      if (*vabort) break;
      const uint64_t now = globaltimer_ns();
      if (idle_since == 0) {
        idle_since = now;
      } else if (now - idle_since > WSG_WAIT_LIMIT_NS) {
        if (lane == 0) {
          *vabort = 1;
          atomicOr(a.err, ERR_MBAR_TIMEOUT);
        }
        break;
      }
      __nanosleep(64);
    }
    if (*vabort && active)
      for (int k = max(retired, issued - kGtQ); k < issued; ++k) mbar_wait(&wfull[k % kGtQ], (k / kGtQ) & 1);
    return;
  }

  // ---- consumers ----
  pdl_wait();  // x may come from the previous kernel, and y is written below
  uint64_t* mfull = full + warp * kGtQ;
  uint64_t* mempty = empty + warp * kGtQ;
  const unsigned char* myring = smem + static_cast<size_t>(warp) * RB;
  // this lane's x elements: part j (warp % np + np j), 128-column chunk k, 4 columns
  const int mypart = warp % np, mysub = warp / np;
  float4 xr[kMkXr];
#pragma unroll
  for (int q = 0; q < kMkXr; ++q) {
    const int j = q >> 1, k = q & 1, off = 4 * lane + 128 * k;
    const int col = (mypart + np * j) * cw + off;
    xr[q] = (j < pw && k < gm.kc && off < cw && col < a.in) ? ldg4<WT>(a.x, col) : make_float4(0, 0, 0, 0);
  }
  int cq = 0;
  uint32_t cph = 0, chead = 0;
  bool ok = true;
  auto run = [&](auto kc_tag) {
    constexpr int KC = decltype(kc_tag)::value;
    constexpr int RM = kMkRowsMax / KC;  // rows per box, at most
    constexpr int kSh = RM == 32 ? 0 : RM == 16 ? 1 : RM == 8 ? 2 : 3;
    using W = MkW4<WT>;
    for (int cg = 0; cg < ng; cg += gm.gchunk) {
      const int ce = min(ng, cg + gm.gchunk);
      for (int rg = cg + (((mysub - cg) % wpp) + wpp) % wpp; rg < ce; rg += wpp) {
        const int nr = min(R, nrows - rg * R);
        float acc[RM], acc2[RM];  // even / odd columns of each row
#pragma unroll
        for (int r = 0; r < RM; ++r) acc[r] = acc2[r] = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (j >= pw) break;
          if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(&mfull[cq], cph));
            if (!ok) {
              if (lane == 0) atomicOr(a.err, ERR_MBAR_TIMEOUT);
              *vabort = 1;
            }
          }
          if (ok) {
            const uint32_t boff = chead + B > RB ? 0u : chead;
            chead = boff + B;
            const unsigned char* buf = myring + boff;
#pragma unroll
            for (int k = 0; k < KC; ++k) {
              const int off = 4 * lane + 128 * k;
              if (off < cw) {
                const float4 x = xr[2 * j + k];
#pragma unroll
                for (int r = 0; r < RM; ++r)
                  if (r < nr) W::dot2(W::lds(buf, r * cw + off), x, acc[r], acc2[r]);
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&mempty[cq]);
            if (++cq == kGtQ) {
              cq = 0;
              cph ^= 1u;
            }
          }
        }
#pragma unroll
        for (int r = 0; r < RM; ++r) acc[r] += acc2[r];
        const float v = reduce_scatter<RM>(acc, lane);
        const int r = lane >> kSh;
        if (ok && (lane & ((1 << kSh) - 1)) == 0 && r < nr) part[((rg - cg) * R + r) * kGtWarps + warp] = v;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kGtWarps * 32) : "memory");
      if (*vabort) return;
      const int r0 = cg * R, r1 = min(nrows, ce * R);
      for (int lr = r0 + tid; lr < r1; lr += kGtWarps * 32) {
        // the partials of the warps that own the row's group, in a fixed order
        const float* p = part + (lr - r0) * kGtWarps + ((lr / R) % wpp) * np;
        float v = p[0];
        for (int w = 1; w < np; ++w) v += p[w];
        a.y[u0 + lr] = v;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kGtWarps * 32) : "memory");
    }
  };
  if (gm.kc == 1)
    run(std::integral_constant<int, 1>{});
  else
    run(std::integral_constant<int, 2>{});
}

}  // namespace wsg
