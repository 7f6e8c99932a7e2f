// Persistent decode megakernel: whole token-to-logits forwards in one launch.
//
// "Megakernels" (the page's opening and "GPU-wide end-to-end generation")
// puts a complete forward in one dispatch, but its single-threadgroup version
// leaves most of the GPU idle, and its GPU-wide version splits the forward into
// 227 ordered dispatches. This kernel keeps the whole GPU busy inside one
// launch: one CTA per SM, co-resident by cooperative launch.
//
//  * Every weight segment (at most 8 KB) this CTA will read, over all stages
//    of all requested steps (QKV, O, gate/up, down of every layer, then the
//    vocabulary slice), is assigned to one of its 8 consumer warps: segment j
//    of a stage goes to warp j mod 8. Each consumer warp owns a private ring
//    of shared-memory slots. Lane w of a ninth, producer warp walks a cursor
//    through consumer w's future segments (across stage, layer and step
//    boundaries) and issues a bulk copy into ring w whenever a slot is free
//    (full/empty mbarrier pair per slot). Weights never depend on
//    activations, so the rings hold the next stages' weights while the
//    consumers wait at a barrier, and HBM keeps streaming.
//  * Per stage the CTA stages the activation vector (with the fused RMSNorm),
//    each warp reduces its segments to partial dots, the partials are summed
//    in a fixed order, the fused epilogue runs, and the CTAs meet at a grid
//    barrier before the next stage reads what this one wrote.
//  * Attention runs between QKV and O on n_kv x nsplit CTAs (the same body as
//    the standalone attention kernel: Q/K norm, RoPE, KV append, key-parallel
//    splits merged by the last CTA).
//  * The head (final RMSNorm, vocabulary GEMV, two-pass argmax) writes the
//    next token, which the next step's embedding gather reads after a barrier.
//
// Every wait is bounded. On a timeout the CTA raises an abort flag, stops
// issuing, waits (bounded) for the copies already in flight, and the error
// word records the cause.
#pragma once
#include <cstdint>

#include "attention.cuh"
#include "gemv_stream.cuh"
#include "ptx.cuh"

namespace wsg {

constexpr int kMkWarps = 8;                      // consumer warps
constexpr int kMkConsumers = kMkWarps * 32;
constexpr int kMkThreads = kMkConsumers + 32;    // plus one producer warp
constexpr int kMkSlot = 8192;         // bytes per ring slot
constexpr int kMkLayerPtrs = 12;      // pointers per layer in the shared layer table
constexpr int kMkWarpSlotsMax = 8;    // ring slots per warp, upper bound

enum : uint32_t { ERR_GRID_BARRIER_TIMEOUT = 1u << 4 };

struct MkLayer {
  const void *wq, *wk, *wv, *wo, *wg, *wu, *wd;
  const float *g_in, *g_post, *g_q, *g_k;
};

// Streaming geometry of one matrix shape.
struct MkGeom {
  int32_t row_bytes;  // in * sizeof(weight)
  int32_t spr;        // segments per row (> 1 when a row is longer than a slot)
  int32_t seg_bytes;  // bytes per segment of a split row (multiple of 16)
  int32_t rps;        // whole rows per segment when spr == 1
};

struct MkArgs {
  const MkLayer* layers;  // device array [L]
  const void* embed;
  const float* g_final;
  int32_t L, H, I, n_q, n_kv, d, V;
  float eps;
  MkGeom gq, go, gg, gd, gv;  // QKV, O, gate/up, down, vocabulary
  float* h;
  float* qkv;
  float* attn;
  float* act;
  float* logits;  // may be NULL
  int32_t* tok;
  int32_t* ctrl;
  uint32_t* err;
  float* mval;
  int32_t* midx;
  uint32_t* mcnt;
  uint32_t* bar;  // [0] grid barrier arrivals, [1] CTAs finished
  AttnArgs at;    // kc / vc point at layer 0's cache
  size_t kv_layer_bytes;
  int32_t wslots;  // ring slots per warp (<= kMkWarpSlotsMax)
  int32_t xs_floats, part_floats;
  int32_t pos0, nsteps;
  int32_t head_every, head_last;  // head on every step / on the last step
  uint64_t* trace;  // optional: [G][L + 1][5][4] globaltimer stamps of the first forward
};

// Trace points per stage: entry, activations staged, segments consumed, barrier passed.
constexpr int kMkTraceStages = 5, kMkTraceEvents = 4;
// Per-segment trace of warp 0 of CTA 0 (first kMkTraceSegs segments of the first
// forward), after the stage trace: wait begins, data ready, dot reduced, next copy issued.
constexpr int kMkTraceSegs = 512, kMkTraceSegEvents = 4;

enum MkStageKind : int { MK_QKV = 0, MK_O = 1, MK_GU = 2, MK_DOWN = 3, MK_VOCAB = 4 };

// This CTA's share of one stage type: partition units [u0, u1) (rows, or
// gate/up row pairs), balanced so no CTA has more than one unit above average.
struct MkRange {
  int u0, u1;
};

__device__ __forceinline__ int mk_units(const MkArgs& a, int st) {
  return st == MK_QKV ? (a.n_q + 2 * a.n_kv) * a.d : st == MK_GU ? a.I : st == MK_VOCAB ? a.V : a.H;
}

__device__ __forceinline__ MkRange mk_range(const MkArgs& a, int st, int c, int G) {
  const long long units = mk_units(a, st);
  return MkRange{static_cast<int>(c * units / G), static_cast<int>((c + 1) * units / G)};
}

// One stage's weight segments for this CTA: up to three contiguous row pieces
// (QKV spans the three source matrices; gate/up streams the gate rows, then
// the up rows, of the same units). Held in registers: pieces are chosen by
// comparisons, never by array indexing.
struct MkStage {
  const char *b0, *b1, *b2;  // first row of each piece
  int nr0, nr1, nr2;         // rows per piece
  int l1, l2;                // local index of the first row of pieces 1 and 2 (piece 0 starts at 0)
  int c1, c2, n;             // segments: piece 0 [0, c1), piece 1 [c1, c2), piece 2 [c2, n)
  int u0, nloc;
};

__device__ __forceinline__ int mk_segs(const MkGeom& gm, int nrows) {
  return gm.spr > 1 ? nrows * gm.spr : (nrows + gm.rps - 1) / gm.rps;
}

__device__ __forceinline__ const MkGeom& mk_geom(const MkArgs& a, int st) {
  return st == MK_QKV ? a.gq : st == MK_O ? a.go : st == MK_GU ? a.gg : st == MK_DOWN ? a.gd : a.gv;
}

// Stage geometry of this CTA with tensors named by index into a layer's
// pointer table (0 wq, 1 wk, 2 wv, 3 wo, 4 wg, 5 wu, 6 wd; 7: the embedding),
// so it is computed once per launch and combined with any layer's pointers.
struct MkStageT {
  int t0, t1, t2;        // tensor of each piece
  int row0, row1, row2;  // first row of each piece within its tensor
  int nr0, nr1, nr2, l1, l2, c1, c2, n, u0, nloc;
};

__device__ __forceinline__ MkStageT mk_stage_t(const MkArgs& a, int st, MkRange r) {
  const MkGeom& gm = mk_geom(a, st);
  MkStageT s;
  s.u0 = r.u0;
  s.t1 = s.t2 = 0;
  s.row1 = s.row2 = 0;
  s.nr1 = s.nr2 = 0;
  s.l1 = s.l2 = 0;
  if (st == MK_QKV) {
    const int qw = a.n_q * a.d, kvw = a.n_kv * a.d;
    const int q0 = min(r.u0, qw), q1 = min(r.u1, qw);
    const int k0 = min(max(r.u0, qw), qw + kvw), k1 = min(max(r.u1, qw), qw + kvw);
    const int v0 = max(r.u0, qw + kvw), v1 = max(r.u1, qw + kvw);
    s.t0 = 0, s.row0 = q0, s.nr0 = q1 - q0;
    s.t1 = 1, s.row1 = k0 - qw, s.nr1 = k1 - k0, s.l1 = k0 - r.u0;
    s.t2 = 2, s.row2 = v0 - qw - kvw, s.nr2 = v1 - v0, s.l2 = v0 - r.u0;
    s.nloc = r.u1 - r.u0;
  } else if (st == MK_GU) {
    s.t0 = 4, s.row0 = r.u0, s.nr0 = r.u1 - r.u0;
    s.t1 = 5, s.row1 = r.u0, s.nr1 = r.u1 - r.u0, s.l1 = r.u1 - r.u0;
    s.nloc = 2 * (r.u1 - r.u0);
  } else {
    s.t0 = st == MK_O ? 3 : st == MK_DOWN ? 6 : 7;
    s.row0 = r.u0;
    s.nr0 = r.u1 - r.u0;
    s.nloc = r.u1 - r.u0;
  }
  s.c1 = mk_segs(gm, s.nr0);
  s.c2 = s.c1 + mk_segs(gm, s.nr1);
  s.n = s.c2 + mk_segs(gm, s.nr2);
  return s;
}

// Bind a stage template to one layer's tensors (lp: that layer's pointer table).
__device__ __forceinline__ MkStage mk_bind(const MkStageT& t, const MkGeom& gm, const void* const* lp,
                                          const void* embed) {
  auto ptr = [&](int id) { return static_cast<const char*>(id == 7 ? embed : lp[id]); };
  const size_t rb = static_cast<size_t>(gm.row_bytes);
  MkStage s;
  s.b0 = ptr(t.t0) + t.row0 * rb;
  s.b1 = ptr(t.t1) + t.row1 * rb;
  s.b2 = ptr(t.t2) + t.row2 * rb;
  s.nr0 = t.nr0, s.nr1 = t.nr1, s.nr2 = t.nr2;
  s.l1 = t.l1, s.l2 = t.l2;
  s.c1 = t.c1, s.c2 = t.c2, s.n = t.n;
  s.u0 = t.u0, s.nloc = t.nloc;
  return s;
}

struct MkSeg {
  const char* src;
  int bytes;
  int lrow;  // first local row
  int part;  // segment index within its row (split rows)
  int nr;    // rows in this segment
  int off;   // byte offset within the row
};

__device__ __forceinline__ MkSeg mk_seg(const MkStage& s, const MkGeom& gm, int j) {
  const bool p0 = j < s.c1, p1 = !p0 && j < s.c2;
  const int jj = j - (p0 ? 0 : p1 ? s.c1 : s.c2);
  const char* base = p0 ? s.b0 : p1 ? s.b1 : s.b2;
  const int lbase = p0 ? 0 : p1 ? s.l1 : s.l2;
  MkSeg r;
  if (gm.spr > 1) {
    const int row = jj / gm.spr, part = jj - row * gm.spr;
    r.off = part * gm.seg_bytes;
    r.bytes = min(gm.seg_bytes, gm.row_bytes - r.off);
    r.src = base + static_cast<size_t>(row) * gm.row_bytes + r.off;
    r.lrow = lbase + row;
    r.part = part;
    r.nr = 1;
  } else {
    const int nrows = p0 ? s.nr0 : p1 ? s.nr1 : s.nr2;
    const int row = jj * gm.rps;
    r.nr = min(gm.rps, nrows - row);
    r.off = 0;
    r.bytes = r.nr * gm.row_bytes;
    r.src = base + static_cast<size_t>(row) * gm.row_bytes;
    r.lrow = lbase + row;
    r.part = 0;
  }
  return r;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ bool mk_head_on(const MkArgs& a, int step) {
  return a.head_every || (a.head_last && step == a.nsteps - 1);
}

// Widest activation vector the staging code holds in registers (16 per thread).
constexpr int kMkMaxWidth = 16 * kMkConsumers;

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kMkConsumers) : "memory"); }

struct ConsumerSync {  // barrier over the consumer warps only
  __device__ __forceinline__ void operator()() const { consumer_sync(); }
};

template <typename WT, typename KT, int GMAX>
__global__ void __launch_bounds__(kMkThreads, 1) decode_megakernel(const MkArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red[64];
  __shared__ int redi[32];
  __shared__ int s_abort, s_last;
  __shared__ MkStageT s_stage[5];
  const int R = a.wslots;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(kMkWarps) * R * kMkSlot);
  uint64_t* empty = full + kMkWarps * kMkWarpSlotsMax;
  float* xs = reinterpret_cast<float*>(empty + kMkWarps * kMkWarpSlotsMax);
  float* part = xs + a.xs_floats;
  float* ascratch = xs;  // the attention stage reuses the GEMV staging area
  const void** lptr = reinterpret_cast<const void**>(part + a.part_floats);  // [L][kMkLayerPtrs]
  volatile int* vabort = &s_abort;
  auto ring_of = [&](int w) { return smem + static_cast<size_t>(w) * R * kMkSlot; };

  // ---- per-launch tables: every layer's tensor pointers, this CTA's stage geometry ----
  for (int i = tid; i < a.L * kMkLayerPtrs; i += kMkThreads) {
    const int l = i / kMkLayerPtrs, k = i - l * kMkLayerPtrs;
    const MkLayer* p = a.layers + l;
    const void* v = nullptr;
    switch (k) {
      case 0: v = p->wq; break;
      case 1: v = p->wk; break;
      case 2: v = p->wv; break;
      case 3: v = p->wo; break;
      case 4: v = p->wg; break;
      case 5: v = p->wu; break;
      case 6: v = p->wd; break;
      case 7: v = p->g_in; break;
      case 8: v = p->g_post; break;
      case 9: v = p->g_q; break;
      case 10: v = p->g_k; break;
      default: break;
    }
    lptr[i] = v;
  }
  if (tid < 5) s_stage[tid] = mk_stage_t(a, tid, mk_range(a, tid, c, G));
  if (tid == 0) {
    s_abort = 0;
    s_last = 0;
  }
  if (tid < kMkWarps * R) {
    const int w = tid / R, s = tid - w * R;
    mbar_init(&full[w * kMkWarpSlotsMax + s], 1);
    mbar_init(&empty[w * kMkWarpSlotsMax + s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto layer_ptrs = [&](int l) { return lptr + l * kMkLayerPtrs; };

  // ------------------------------------------------------------------ producer ----
  if (warp == kMkWarps) {
    // Lane w feeds consumer warp w's ring. The warp stays converged: every
    // pass, each lane tests (without blocking) whether its next slot is free,
    // and all lanes that can issue do so together.
    const int w = lane;
    uint64_t* wfull = full + (w < kMkWarps ? w : 0) * kMkWarpSlotsMax;
    uint64_t* wempty = empty + (w < kMkWarps ? w : 0) * kMkWarpSlotsMax;
    unsigned char* wring = ring_of(w < kMkWarps ? w : 0);
    const uint64_t pol = l2_policy_evict_first();
    int cstep = 0, clayer = 0, cst = MK_QKV, cj = 0;
    bool cdone = w >= kMkWarps;
    MkStage cs{};
    auto advance = [&]() {
      if (cst == MK_VOCAB) {
        ++cstep;
        clayer = 0;
        cst = MK_QKV;
      } else if (cst == MK_DOWN) {
        if (clayer + 1 < a.L) {
          ++clayer;
          cst = MK_QKV;
        } else if (mk_head_on(a, cstep)) {
          cst = MK_VOCAB;
        } else {
          ++cstep;
          clayer = 0;
          cst = MK_QKV;
        }
      } else {
        ++cst;
      }
    };
    auto settle = [&]() {  // first stage, from the current one, with a segment for consumer w
      while (true) {
        if (cstep >= a.nsteps) {
          cdone = true;
          return;
        }
        cs = mk_bind(s_stage[cst], mk_geom(a, cst), layer_ptrs(cst == MK_VOCAB ? 0 : clayer), a.embed);
        cj = w;
        if (cj < cs.n) return;
        advance();
      }
    };
    if (!cdone) settle();
    int issued = 0;
    uint64_t idle_since = 0;
    while (__any_sync(0xffffffffu, !cdone)) {
      bool can = false;
      if (!cdone) {
        const int slot = issued % R;
        can = issued < R || mbar_test(&wempty[slot], ((issued / R) - 1) & 1);
        if (can) {
          const MkSeg sg = mk_seg(cs, mk_geom(a, cst), cj);
          mbar_arrive_expect_tx(&wfull[slot], static_cast<uint32_t>(sg.bytes));
          bulk_g2s(wring + static_cast<size_t>(slot) * kMkSlot, sg.src, static_cast<uint32_t>(sg.bytes),
                   &wfull[slot], pol);
          ++issued;
          cj += kMkWarps;
          if (cj >= cs.n) {
            advance();
            settle();
          }
        }
      }
      if (__any_sync(0xffffffffu, can)) {
        idle_since = 0;
        continue;
      }
      // nothing to issue this pass: back off, bounded
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
    // After an abort: wait (bounded) until the copies already issued have landed.
    if (*vabort && w < kMkWarps)
      for (int n = max(0, issued - R); n < issued; ++n) mbar_wait(&wfull[n % R], (n / R) & 1);
    return;
  }

  // ------------------------------------------------------------------ consumers ----
  uint64_t* mfull = full + warp * kMkWarpSlotsMax;
  uint64_t* mempty = empty + warp * kMkWarpSlotsMax;
  const unsigned char* myring = ring_of(warp);
  int consumed = 0;
  uint32_t sync_target = 0;
  const int qw = a.n_q * a.d;

  auto grid_sync = [&]() -> bool {
    consumer_sync();
    if (tid == 0) {
      sync_target += G;
      // release: the consumers' writes (ordered before by the named barrier)
      // become visible to every CTA that acquires the count
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.bar) : "memory");
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(a.bar) < sync_target) {
        if (globaltimer_ns() - t0 > WSG_WAIT_LIMIT_NS) {
          *vabort = 1;
          atomicOr(a.err, ERR_GRID_BARRIER_TIMEOUT);
          break;
        }
      }
    }
    consumer_sync();
    return !*vabort;
  };

  // Stage the activation vector: plain copy, or RMSNorm(src) * gain. Values
  // and gains are loaded together (one memory round trip) into registers.
  auto stage_x = [&](const float* src, const WT* wsrc, int in, const float* gain, bool store_h) {
    constexpr int K = kMkMaxWidth / kMkConsumers;
    float v[K], gn[K];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int i = tid + k * kMkConsumers;
      v[k] = 0.f;
      gn[k] = 1.f;
      if (i < in) {
        v[k] = wsrc ? load_f32<WT>(wsrc, i) : __ldcg(src + i);
        if (gain) gn[k] = __ldg(gain + i);
      }
    }
#pragma unroll
    for (int k = 0; k < K; ++k) ss = fmaf(v[k], v[k], ss);
    float inv = 1.f;
    if (gain) {
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
      consumer_sync();
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kMkWarps; ++w) t += red[w];
      inv = 1.0f / sqrtf(t / static_cast<float>(in) + a.eps);
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int i = tid + k * kMkConsumers;
      if (i < in) {
        if (store_h) a.h[i] = v[k];
        xs[xs_index<WT>(i, in)] = gain ? v[k] * inv * gn[k] : v[k];
      }
    }
    consumer_sync();
  };

  uint64_t* segtrace = nullptr;
  if (a.trace && c == 0 && warp == 0)
    segtrace = a.trace + static_cast<size_t>(G) * (a.L + 1) * kMkTraceStages * kMkTraceEvents;
  auto segstamp = [&](int ev) {
    if (segtrace && lane == 0 && consumed < kMkTraceSegs) segtrace[consumed * kMkTraceSegEvents + ev] = clock64();
  };

  // This warp's segments of one stage, in ring order, into part[].
  auto consume = [&](const MkStage& sl, const MkGeom& gm, int in) -> bool {
    for (int j = warp; j < sl.n; j += kMkWarps) {
      const int slot = consumed % R;
      segstamp(0);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&mfull[slot], (consumed / R) & 1));
      segstamp(1);
      if (!ok) {
        if (lane == 0) atomicOr(a.err, ERR_MBAR_TIMEOUT);
        *vabort = 1;
        break;
      }
      const MkSeg sg = mk_seg(sl, gm, j);
      const unsigned char* buf = myring + static_cast<size_t>(slot) * kMkSlot;
      if (sg.nr == 1) {
        float v = seg_dot<WT>(buf, xs, sg.off / static_cast<int>(sizeof(WT)), sg.bytes, in, lane);
        v = warp_sum(v);
        if (lane == 0) part[sg.lrow * gm.spr + sg.part] = v;
      } else {
        // several whole rows: all lane partials first (each x chunk read once),
        // then one interleaved reduction
        float v[4];
        for (int r0 = 0; r0 < sg.nr; r0 += 4) {
          rows_dot<WT>(buf + static_cast<size_t>(r0) * gm.row_bytes, gm.row_bytes, min(4, sg.nr - r0), xs, in, lane, v);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int r = 0; r < 4; ++r) v[r] += __shfl_xor_sync(0xffffffffu, v[r], o);
          if (lane == 0)
            for (int r = 0; r < 4 && r0 + r < sg.nr; ++r) part[sg.lrow + r0 + r] = v[r];
        }
      }
      segstamp(2);
      // The slot's data reached registers before the shuffles above; hand the
      // slot back to the producer.
      __syncwarp();
      if (lane == 0) mbar_arrive(&mempty[slot]);
      segstamp(3);
      ++consumed;
    }
    consumer_sync();
    return !*vabort;
  };

  auto row_value = [&](const MkGeom& gm, int lr) {
    float v = 0.f;
    for (int k = 0; k < gm.spr; ++k) v += part[lr * gm.spr + k];
    return v;
  };

  auto stamp = [&](int step, int l, int st, int ev) {
    if (a.trace && step == 0 && tid == 0)
      a.trace[((static_cast<size_t>(c) * (a.L + 1) + l) * kMkTraceStages + st) * kMkTraceEvents + ev] =
          globaltimer_ns();
  };

  bool ok = true;
  for (int step = 0; step < a.nsteps && ok; ++step) {
    const int pos = a.pos0 + step;
    for (int l = 0; l < a.L && ok; ++l) {
      const void* const* lp = layer_ptrs(l);
      const float* g_in = static_cast<const float*>(lp[7]);
      const float* g_post = static_cast<const float*>(lp[8]);
      // ---- QKV with the input RMSNorm (layer 0: of the token's embedding row) ----
      {
        stamp(step, l, 0, 0);
        const MkStage sl = mk_bind(s_stage[MK_QKV], a.gq, lp, a.embed);
        if (l == 0) {
          int t = __ldcg(a.tok + pos);
          if (t < 0 || t >= a.V) {
            if (tid == 0) atomicOr(a.err, ERR_BAD_TOKEN);
            t = 0;
          }
          stage_x(nullptr, static_cast<const WT*>(a.embed) + static_cast<size_t>(t) * a.H, a.H, g_in, c == 0);
        } else {
          stage_x(a.h, nullptr, a.H, g_in, false);
        }
        stamp(step, l, 0, 1);
        // Keys and values before pos do not depend on this token: pull this
        // CTA's attention range of them into L2 while QKV runs.
        if (tid == 0 && c < a.n_kv * a.at.nsplit_max) {
          int t0, t1, ns;
          if (attn_split_range(a.at, c / a.n_kv, pos, &t0, &t1, &ns)) {
            t1 = min(t1, pos);
            if (t1 > t0) {
              const size_t eb = a.kv_layer_bytes / (static_cast<size_t>(a.n_kv) * a.at.max_seq * a.d);
              const size_t off = static_cast<size_t>(l) * a.kv_layer_bytes +
                                 ((static_cast<size_t>(c % a.n_kv) * a.at.max_seq + t0) * a.d) * eb;
              const uint32_t bytes = static_cast<uint32_t>(static_cast<size_t>(t1 - t0) * a.d * eb);
              bulk_prefetch_l2(static_cast<const char*>(a.at.kc) + off, bytes);
              bulk_prefetch_l2(static_cast<const char*>(a.at.vc) + off, bytes);
            }
          }
        }
        if (!(ok = consume(sl, a.gq, a.H))) break;
        for (int lr = tid; lr < sl.nloc; lr += kMkConsumers) a.qkv[sl.u0 + lr] = row_value(a.gq, lr);
        stamp(step, l, 0, 2);
        if (!(ok = grid_sync())) break;
        stamp(step, l, 0, 3);
      }
      // ---- attention (Q/K norm, RoPE, KV append, key-parallel splits) ----
      {
        AttnArgs at = a.at;
        at.g_q = static_cast<const float*>(lp[9]);
        at.g_k = static_cast<const float*>(lp[10]);
        at.kc = static_cast<char*>(a.at.kc) + static_cast<size_t>(l) * a.kv_layer_bytes;
        at.vc = static_cast<char*>(a.at.vc) + static_cast<size_t>(l) * a.kv_layer_bytes;
        stamp(step, l, 1, 0);
        if (c < a.n_kv * at.nsplit_max)
          attn_decode_body<KT, GMAX, kMkConsumers, ConsumerSync, 4>(at, c % a.n_kv, c / a.n_kv, pos, ascratch, tid,
                                                                    ConsumerSync{}, &s_last);
        stamp(step, l, 1, 2);
        if (!(ok = grid_sync())) break;
        stamp(step, l, 1, 3);
      }
      // ---- O projection + residual ----
      {
        stamp(step, l, 2, 0);
        const MkStage sl = mk_bind(s_stage[MK_O], a.go, lp, a.embed);
        stage_x(a.attn, nullptr, qw, nullptr, false);
        stamp(step, l, 2, 1);
        if (!(ok = consume(sl, a.go, qw))) break;
        for (int lr = tid; lr < sl.nloc; lr += kMkConsumers) {
          const int row = sl.u0 + lr;
          a.h[row] = __ldcg(a.h + row) + row_value(a.go, lr);
        }
        stamp(step, l, 2, 2);
        if (!(ok = grid_sync())) break;
        stamp(step, l, 2, 3);
      }
      // ---- gate/up with the post-attention RMSNorm, SwiGLU ----
      {
        stamp(step, l, 3, 0);
        const MkStage sl = mk_bind(s_stage[MK_GU], a.gg, lp, a.embed);
        stage_x(a.h, nullptr, a.H, g_post, false);
        stamp(step, l, 3, 1);
        if (!(ok = consume(sl, a.gg, a.H))) break;
        const int np = sl.nloc >> 1;
        for (int i = tid; i < np; i += kMkConsumers)
          a.act[sl.u0 + i] = silu_f32(row_value(a.gg, i)) * row_value(a.gg, np + i);
        stamp(step, l, 3, 2);
        if (!(ok = grid_sync())) break;
        stamp(step, l, 3, 3);
      }
      // ---- down projection + residual ----
      {
        stamp(step, l, 4, 0);
        const MkStage sl = mk_bind(s_stage[MK_DOWN], a.gd, lp, a.embed);
        stage_x(a.act, nullptr, a.I, nullptr, false);
        stamp(step, l, 4, 1);
        if (!(ok = consume(sl, a.gd, a.I))) break;
        for (int lr = tid; lr < sl.nloc; lr += kMkConsumers) {
          const int row = sl.u0 + lr;
          a.h[row] = __ldcg(a.h + row) + row_value(a.gd, lr);
        }
        stamp(step, l, 4, 2);
        if (!(ok = grid_sync())) break;
        stamp(step, l, 4, 3);
      }
    }
    if (!ok || !mk_head_on(a, step)) continue;
    // ---- head: final RMSNorm, tied vocabulary projection, two-pass argmax ----
    stamp(step, a.L, 0, 0);
    const MkStage sl = mk_bind(s_stage[MK_VOCAB], a.gv, layer_ptrs(0), a.embed);
    stage_x(a.h, nullptr, a.H, a.g_final, false);
    stamp(step, a.L, 0, 1);
    if (!(ok = consume(sl, a.gv, a.H))) break;
    stamp(step, a.L, 0, 2);
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int lr = tid; lr < sl.nloc; lr += kMkConsumers) {
      const int row = sl.u0 + lr;
      const float v = row_value(a.gv, lr);
      if (a.logits) a.logits[row] = v;
      if (argmax_better(v, row, bv, bi)) {
        bv = v;
        bi = row;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (argmax_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      red[warp] = bv;
      redi[warp] = bi;
    }
    consumer_sync();
    if (tid == 0) {
      for (int w = 1; w < kMkWarps; ++w)
        if (argmax_better(red[w], redi[w], bv, bi)) {
          bv = red[w];
          bi = redi[w];
        }
      a.mval[c] = bv;
      a.midx[c] = bi;
      __threadfence();
      if (atomicAdd(a.mcnt, 1u) == static_cast<uint32_t>(G - 1)) {
        __threadfence();
        float gv = -INFINITY;
        int gi = 0x7fffffff;
        for (int k = 0; k < G; ++k) {
          const float v = __ldcg(a.mval + k);
          const int i = __ldcg(a.midx + k);
          if (argmax_better(v, i, gv, gi)) {
            gv = v;
            gi = i;
          }
        }
        if (gi == 0x7fffffff) {  // every logit was NaN
          gi = 0;
          atomicOr(a.err, ERR_ARGMAX_NAN);
        }
        a.tok[pos + 1] = gi;
        *a.mcnt = 0u;
        __threadfence();
      }
    }
    stamp(step, a.L, 1, 0);
    if (step + 1 < a.nsteps) ok = grid_sync();  // the next step reads the new token
  }

  // ---- exit: the last CTA out resets the barrier counters and publishes the position ----
  consumer_sync();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.bar + 1, 1u) == static_cast<uint32_t>(G - 1)) {
      a.bar[0] = 0u;
      a.bar[1] = 0u;
      a.ctrl[0] = a.pos0 + a.nsteps;
      __threadfence();
    }
  }
}

}  // namespace wsg
