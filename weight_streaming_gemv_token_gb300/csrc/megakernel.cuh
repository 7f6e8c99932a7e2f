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
//    in a fixed order and the fused epilogue writes the outputs. Stages hand
//    data to each other through exchange words: 64-bit (tag, value) pairs
//    written in one store. A reader polls the words it needs until they carry
//    the tag of the producing stage, so readiness and data arrive together
//    and no grid-wide barrier is needed. Each buffer's next version can only
//    be written after every reader of the current version has read it (the
//    forward's own data dependencies order them), and a CTA with no rows in a
//    stage reads nothing for it.
//  * Attention runs between QKV and O on n_kv x nsplit CTAs (the same body as
//    the standalone attention kernel: Q/K norm, RoPE, KV append, key-parallel
//    splits merged by the last CTA).
//  * The head (final RMSNorm, vocabulary GEMV, two-pass argmax) publishes the
//    next token as an exchange word for the next step's embedding gather.
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

enum : uint32_t { ERR_EXCHANGE_TIMEOUT = 1u << 4 };

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
  // Cross-CTA exchanges: 64-bit (tag, value) words, each written in one store,
  // so a reader that sees the expected tag also has the value.
  uint64_t* ll_h;     // residual stream [H]
  uint64_t* ll_qkv;   // raw q, k, v [(n_q + 2 n_kv) d]
  uint64_t* ll_attn;  // attention output [n_q d]
  uint64_t* ll_act;   // SwiGLU activations [I]
  uint64_t* ll_tok;   // next token [1]
  uint64_t* ll_apart; // attention split partials [n_kv][nsplit_max][group][d + 2]
  uint32_t* kv_ready; // [L][n_kv]: positions appended to the cache (release-stored)
  uint32_t epoch;     // per-launch tag prefix (nonzero; 12 bits)
  AttnArgs at;        // kc / vc point at layer 0's cache
  size_t kv_layer_bytes;
  int32_t wslots;  // ring slots per warp (<= kMkWarpSlotsMax)
  int32_t xs_floats, part_floats, hown_floats;
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

// ---- flag-in-data exchange ----
__device__ __forceinline__ uint32_t mk_tag(const MkArgs& a, int step, int l, int st) {
  return (a.epoch << 20) | static_cast<uint32_t>((step * (a.L + 1) + l) * 5 + st + 1);
}

__device__ __forceinline__ void ll_store(uint64_t* p, float v, uint32_t tag) {
  const uint64_t w = (static_cast<uint64_t>(tag) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

// Release store: this thread's earlier writes (and, through a CTA barrier,
// the CTA's) are visible to whoever reads the tag.
__device__ __forceinline__ void ll_store_release(uint64_t* p, float v, uint32_t tag) {
  const uint64_t w = (static_cast<uint64_t>(tag) << 32) | __float_as_uint(v);
  asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ uint64_t ll_load(const uint64_t* p) {
  uint64_t w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Value of an exchange word once its tag is `tag`; bounded poll. On timeout
// raises the abort flag, records the error and returns 0.
__device__ __forceinline__ float ll_wait(const uint64_t* p, uint32_t tag, uint64_t w, volatile int* abort,
                                         uint32_t* err) {
  if (static_cast<uint32_t>(w >> 32) == tag) return __uint_as_float(static_cast<uint32_t>(w));
  const uint64_t t0 = globaltimer_ns();
  for (int it = 0;; ++it) {
    w = ll_load(p);
    if (static_cast<uint32_t>(w >> 32) == tag) return __uint_as_float(static_cast<uint32_t>(w));
    if ((it & 63) == 63) {
      if (*abort) return 0.f;
      if (globaltimer_ns() - t0 > WSG_WAIT_LIMIT_NS) {
        *abort = 1;
        atomicOr(err, ERR_EXCHANGE_TIMEOUT);
        return 0.f;
      }
    }
  }
}

// Attention input/output through the exchange words; the cache rows this CTA
// appends are published with a release store of the per-head position count.
// Splits of one head hand their partial (O, M, L) to split 0 as exchange words.
struct AttnLlIo {
  static constexpr bool kPolledMerge = true;
  const uint64_t* qkv;
  uint64_t* out;
  uint64_t* part;      // [n_kv][nsplit_max][group][d + 2] partial words
  uint32_t* kv_ready;  // this layer's [n_kv]
  uint32_t tag_in, tag_out;
  volatile int* abort;
  uint32_t* err;
  uint64_t* trace_slot;  // this CTA's [4] stamps of the stage, or NULL
  __device__ __forceinline__ void mark(int ev) const {
    if (trace_slot) trace_slot[ev] = globaltimer_ns();
  }
  // Poll the N words addr(0..N) (nullptr: none) until each carries `tag`;
  // all stale words are reloaded together, one round trip per round.
  template <int N, typename Addr>
  __device__ __forceinline__ void poll(Addr addr, uint32_t tag, uint64_t* w) const {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const uint64_t* p = addr(k);
      w[k] = p ? ll_load(p) : (static_cast<uint64_t>(tag) << 32);
    }
    const uint64_t t0 = globaltimer_ns();
    for (int round = 0;; ++round) {
      bool stale = false;
#pragma unroll
      for (int k = 0; k < N; ++k) stale |= static_cast<uint32_t>(w[k] >> 32) != tag;
      if (!stale) break;
      if ((round & 63) == 63) {
        if (*abort) break;
        if (globaltimer_ns() - t0 > WSG_WAIT_LIMIT_NS) {
          *abort = 1;
          atomicOr(err, ERR_EXCHANGE_TIMEOUT);
          break;
        }
      }
#pragma unroll
      for (int k = 0; k < N; ++k)
        if (static_cast<uint32_t>(w[k] >> 32) != tag) w[k] = ll_load(addr(k));
    }
  }
  // q of the head group, k and v of head g.
  __device__ __forceinline__ void load_all(float* qn, float* kn, float* vn, int qbase, int kbase, int vbase, int nq_el,
                                           int d, int tid, int nt) const {
    constexpr int NQ = 4;  // q elements per thread: group * d <= 8 * 128 over 256 threads
    uint64_t w[NQ + 2];
    poll<NQ + 2>(
        [&](int k) -> const uint64_t* {
          if (k < NQ) return tid + k * nt < nq_el ? qkv + qbase + tid + k * nt : nullptr;
          return tid < d ? qkv + (k == NQ ? kbase : vbase) + tid : nullptr;
        },
        tag_in, w);
#pragma unroll
    for (int k = 0; k < NQ; ++k)
      if (tid + k * nt < nq_el) qn[tid + k * nt] = __uint_as_float(static_cast<uint32_t>(w[k]));
    if (tid < d) {
      kn[tid] = __uint_as_float(static_cast<uint32_t>(w[NQ]));
      vn[tid] = __uint_as_float(static_cast<uint32_t>(w[NQ + 1]));
    }
  }
  __device__ __forceinline__ void store_out(int i, float v) const { ll_store(out + i, v, tag_out); }
  __device__ __forceinline__ void store_part(size_t i, float v) const { ll_store(part + i, v, tag_out); }
  // Splits k < cnt at base + k * stride: element e of O, then M and L.
  template <int KC>
  __device__ __forceinline__ void poll_parts(size_t base, size_t stride, int cnt, int e, int d, float* ov, float* mv,
                                             float* lv) const {
    uint64_t w[3 * KC];
    const uint64_t* p0 = part + base;
    poll<3 * KC>(
        [&](int j) -> const uint64_t* {
          const int k = j / 3, r = j - 3 * k;
          return k < cnt ? p0 + k * stride + (r == 0 ? e : d + r - 1) : nullptr;
        },
        tag_out, w);
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      ov[k] = __uint_as_float(static_cast<uint32_t>(w[3 * k]));
      mv[k] = __uint_as_float(static_cast<uint32_t>(w[3 * k + 1]));
      lv[k] = __uint_as_float(static_cast<uint32_t>(w[3 * k + 2]));
    }
  }
  __device__ __forceinline__ void publish_kv(int g, int pos) const {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(kv_ready + g), "r"(static_cast<uint32_t>(pos + 1))
                 : "memory");
  }
};

// Bounded wait until *p >= v, with acquire semantics.
__device__ __forceinline__ bool wait_at_least(const uint32_t* p, uint32_t v, volatile int* abort, uint32_t* err) {
  const uint64_t t0 = globaltimer_ns();
  for (int it = 0;; ++it) {
    uint32_t x;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(x) : "l"(p) : "memory");
    if (x >= v) return true;
    if ((it & 63) == 63) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > WSG_WAIT_LIMIT_NS) {
        *abort = 1;
        atomicOr(err, ERR_EXCHANGE_TIMEOUT);
        return false;
      }
    }
  }
}

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
  float* hown = reinterpret_cast<float*>(lptr + a.L * kMkLayerPtrs);  // this CTA's rows of h
  int consumed = 0;
  const int qw = a.n_q * a.d;
  const MkRange rH = mk_range(a, MK_O, c, G);  // O and down own the same rows of h

  // Stage an activation vector from exchange words (tag `tag`) into xs:
  // plain copy, or RMSNorm * gain. All loads are issued first, then only the
  // words not yet carrying the tag are polled.
  auto stage_ll = [&](const uint64_t* src, uint32_t tag, int in, const float* gain) {
    constexpr int K = kMkMaxWidth / kMkConsumers;
    uint64_t wv[K];
    float gn[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int i = tid + k * kMkConsumers;
      wv[k] = 0;
      gn[k] = 1.f;
      if (i < in) {
        wv[k] = ll_load(src + i);
        if (gain) gn[k] = __ldg(gain + i);
      }
    }
    // Poll in rounds: every round reloads all of this thread's words that do
    // not yet carry the tag, together (one round trip per round).
    {
      const uint64_t t0 = globaltimer_ns();
      for (int round = 0;; ++round) {
        bool stale = false;
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const int i = tid + k * kMkConsumers;
          if (i < in && static_cast<uint32_t>(wv[k] >> 32) != tag) stale = true;
        }
        if (!stale) break;
        if ((round & 63) == 63) {
          if (*vabort) break;
          if (globaltimer_ns() - t0 > WSG_WAIT_LIMIT_NS) {
            *vabort = 1;
            atomicOr(a.err, ERR_EXCHANGE_TIMEOUT);
            break;
          }
        }
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const int i = tid + k * kMkConsumers;
          if (i < in && static_cast<uint32_t>(wv[k] >> 32) != tag) wv[k] = ll_load(src + i);
        }
      }
    }
    float v[K];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      v[k] = __uint_as_float(static_cast<uint32_t>(wv[k]));
      ss = fmaf(v[k], v[k], ss);
    }
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
      if (i < in) xs[xs_index<WT>(i, in)] = gain ? v[k] * inv * gn[k] : v[k];
    }
    consumer_sync();
  };

  // Layer 0: RMSNorm of the token's embedding row.
  auto stage_embed = [&](int t, const float* gain) {
    constexpr int K = kMkMaxWidth / kMkConsumers;
    const WT* row = static_cast<const WT*>(a.embed) + static_cast<size_t>(t) * a.H;
    float v[K], gn[K];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int i = tid + k * kMkConsumers;
      v[k] = i < a.H ? load_f32<WT>(row, i) : 0.f;
      gn[k] = i < a.H ? __ldg(gain + i) : 1.f;
      ss = fmaf(v[k], v[k], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    consumer_sync();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kMkWarps; ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / static_cast<float>(a.H) + a.eps);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int i = tid + k * kMkConsumers;
      if (i < a.H) xs[xs_index<WT>(i, a.H)] = v[k] * inv * gn[k];
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

  // Trace events per stage: 0 entry, 1 inputs staged, 2 outputs published.
  auto stamp = [&](int step, int l, int st, int ev) {
    if (a.trace && step == 0 && tid == 0)
      a.trace[((static_cast<size_t>(c) * (a.L + 1) + l) * kMkTraceStages + st) * kMkTraceEvents + ev] =
          globaltimer_ns();
  };

  const bool attn_cta = c < a.n_kv * a.at.nsplit_max;
  bool ok = true;
  for (int step = 0; step < a.nsteps && ok; ++step) {
    const int pos = a.pos0 + step;
    // The token: written by the host before the launch, or published by the
    // previous step's head.
    int tok;
    if (step > 0 && a.head_every) {
      const uint64_t* p = a.ll_tok;
      tok = __float_as_int(ll_wait(p, mk_tag(a, step - 1, a.L, 0), ll_load(p), vabort, a.err));
    } else {
      tok = __ldcg(a.tok + pos);
    }
    if (tok < 0 || tok >= a.V) {
      if (tid == 0) atomicOr(a.err, ERR_BAD_TOKEN);
      tok = 0;
    }
    if (step > 0 && !a.head_every) {
      // Body-only steps take their token from the host, so nothing else would
      // order this step's writes after the previous step's reads: read the
      // previous step's final residual words (written by every CTA that owns
      // rows of h) before writing anything.
      for (int i = tid; i < a.H; i += kMkConsumers) {
        const uint64_t* p = a.ll_h + i;
        ll_wait(p, mk_tag(a, step - 1, a.L - 1, MK_DOWN), ll_load(p), vabort, a.err);
      }
      consumer_sync();
    }
    for (int l = 0; l < a.L && ok && !*vabort; ++l) {
      const void* const* lp = layer_ptrs(l);
      const float* g_in = static_cast<const float*>(lp[7]);
      const float* g_post = static_cast<const float*>(lp[8]);
      // ---- QKV with the input RMSNorm (layer 0: of the token's embedding row) ----
      {
        stamp(step, l, 0, 0);
        const MkStage sl = mk_bind(s_stage[MK_QKV], a.gq, lp, a.embed);
        if (sl.nloc > 0) {
          if (l == 0)
            stage_embed(tok, g_in);
          else
            stage_ll(a.ll_h, mk_tag(a, step, l - 1, MK_DOWN), a.H, g_in);
        }
        stamp(step, l, 0, 1);
        // Keys and values before pos do not depend on this token: make sure the
        // rows of earlier positions are published (acquire) and pull this
        // CTA's attention range of them into L2 while QKV runs.
        if (tid == 0 && attn_cta && pos > 0)
          wait_at_least(a.kv_ready + l * a.n_kv + c % a.n_kv, static_cast<uint32_t>(pos), vabort, a.err);
        if (tid == 0 && attn_cta) {
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
        const uint32_t tg = mk_tag(a, step, l, MK_QKV);
        for (int lr = tid; lr < sl.nloc; lr += kMkConsumers) ll_store(a.ll_qkv + sl.u0 + lr, row_value(a.gq, lr), tg);
        stamp(step, l, 0, 2);
      }
      // ---- attention (Q/K norm, RoPE, KV append, key-parallel splits) ----
      if (attn_cta) {
        consumer_sync();  // the attention scratch overlaps the staging area the QKV epilogue read
        AttnArgs at = a.at;
        at.g_q = static_cast<const float*>(lp[9]);
        at.g_k = static_cast<const float*>(lp[10]);
        at.kc = static_cast<char*>(a.at.kc) + static_cast<size_t>(l) * a.kv_layer_bytes;
        at.vc = static_cast<char*>(a.at.vc) + static_cast<size_t>(l) * a.kv_layer_bytes;
        stamp(step, l, 1, 0);
        attn_decode_body<KT, GMAX, kMkConsumers, ConsumerSync, (GMAX <= 2 ? 4 : 2), AttnLlIo>(
            at, c % a.n_kv, c / a.n_kv, pos, ascratch, tid, ConsumerSync{}, &s_last,
            AttnLlIo{a.ll_qkv, a.ll_attn, a.ll_apart, a.kv_ready + l * a.n_kv, mk_tag(a, step, l, MK_QKV),
                     mk_tag(a, step, l, 1),
                     vabort, a.err,
                     (a.trace && step == 0)
                         ? a.trace + ((static_cast<size_t>(c) * (a.L + 1) + l) * kMkTraceStages + 1) * kMkTraceEvents
                         : nullptr});
        stamp(step, l, 1, 2);
        consumer_sync();
      }
      // ---- O projection + residual ----
      {
        stamp(step, l, 2, 0);
        const MkStage sl = mk_bind(s_stage[MK_O], a.go, lp, a.embed);
        if (sl.nloc > 0) stage_ll(a.ll_attn, mk_tag(a, step, l, 1), qw, nullptr);
        stamp(step, l, 2, 1);
        if (!(ok = consume(sl, a.go, qw))) break;
        const uint32_t tg = mk_tag(a, step, l, MK_O);
        for (int lr = tid; lr < sl.nloc; lr += kMkConsumers) {
          const int row = sl.u0 + lr;
          const float prev = l == 0 ? load_f32<WT>(static_cast<const WT*>(a.embed) + static_cast<size_t>(tok) * a.H, row)
                                    : hown[lr];
          const float hn = prev + row_value(a.go, lr);
          hown[lr] = hn;
          ll_store(a.ll_h + row, hn, tg);
        }
        stamp(step, l, 2, 2);
      }
      // ---- gate/up with the post-attention RMSNorm, SwiGLU ----
      {
        stamp(step, l, 3, 0);
        const MkStage sl = mk_bind(s_stage[MK_GU], a.gg, lp, a.embed);
        if (sl.nloc > 0) stage_ll(a.ll_h, mk_tag(a, step, l, MK_O), a.H, g_post);
        stamp(step, l, 3, 1);
        if (!(ok = consume(sl, a.gg, a.H))) break;
        const int np = sl.nloc >> 1;
        const uint32_t tg = mk_tag(a, step, l, MK_GU);
        for (int i = tid; i < np; i += kMkConsumers)
          ll_store(a.ll_act + sl.u0 + i, silu_f32(row_value(a.gg, i)) * row_value(a.gg, np + i), tg);
        stamp(step, l, 3, 2);
      }
      // ---- down projection + residual ----
      {
        stamp(step, l, 4, 0);
        const MkStage sl = mk_bind(s_stage[MK_DOWN], a.gd, lp, a.embed);
        if (sl.nloc > 0) stage_ll(a.ll_act, mk_tag(a, step, l, MK_GU), a.I, nullptr);
        stamp(step, l, 4, 1);
        if (!(ok = consume(sl, a.gd, a.I))) break;
        const uint32_t tg = mk_tag(a, step, l, MK_DOWN);
        for (int lr = tid; lr < sl.nloc; lr += kMkConsumers) {
          const float hn = hown[lr] + row_value(a.gd, lr);
          hown[lr] = hn;
          ll_store(a.ll_h + sl.u0 + lr, hn, tg);
        }
        stamp(step, l, 4, 2);
      }
      consumer_sync();  // hown is rewritten by the next layer's O stage
    }
    (void)rH;
    if (!ok || *vabort || !mk_head_on(a, step)) continue;
    // ---- head: final RMSNorm, tied vocabulary projection, two-pass argmax ----
    stamp(step, a.L, 0, 0);
    const MkStage sl = mk_bind(s_stage[MK_VOCAB], a.gv, layer_ptrs(0), a.embed);
    if (sl.nloc > 0) stage_ll(a.ll_h, mk_tag(a, step, a.L - 1, MK_DOWN), a.H, a.g_final);
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
        ll_store_release(a.ll_tok, __int_as_float(gi), mk_tag(a, step, a.L, 0));
      }
    }
    stamp(step, a.L, 1, 0);
    consumer_sync();
  }

  // ---- exit: publish the position for the host-side mirror ----
  if (tid == 0 && c == 0) a.ctrl[0] = a.pos0 + a.nsteps;
}

}  // namespace wsg
