// Persistent decode megakernel: whole token-to-logits forwards in one launch.
//
// "Megakernels" (the page's opening and "GPU-wide end-to-end generation")
// puts a complete forward in one dispatch, but its single-threadgroup version
// leaves most of the GPU idle, and its GPU-wide version splits the forward into
// 227 ordered dispatches. This kernel keeps the whole GPU busy inside one
// launch: one CTA per SM, co-resident by cooperative launch.
//
//  * GEMV stages (QKV, O, gate/up, down of every layer, then the vocabulary
//    slice) give each CTA a contiguous range of output rows and split every
//    row's columns across the CTA's 8 consumer warps (split-K): warp w owns
//    the column parts w (and w + 8) of every row, holds the matching
//    activation elements in registers for the whole stage, and reads only
//    weights from shared memory. All warps get the same work, whatever the
//    row count.
//  * Weights arrive as tiled TMA boxes (R rows x one column part) through a
//    private byte ring per consumer warp. Lane w of a producer warp walks a
//    cursor through consumer w's future boxes (across stage, layer and step
//    boundaries) and issues each box as soon as the ring has room for it
//    (full/empty mbarrier per box in flight; a box never straddles the ring's
//    end). The consumer derives each box's ring offset from the same
//    placement rule, so no offsets are exchanged. Weights never depend on
//    activations, so the rings hold the next stages' weights while the
//    consumers wait for their inputs, and HBM keeps streaming. The producer
//    sits in a warpgroup of its own that gives registers back (setmaxnreg),
//    so the consumer warps run with 224 registers per thread; a tiled copy
//    that waits for room in the copy engine never stalls a consumer.
//  * Per box, every lane accumulates its column chunk into one partial per
//    row; a butterfly reduce-scatter turns the R lane partials into row sums
//    (16 or 32 rows in log2(32) shuffle steps), the 8 warp partials of a row
//    meet in shared memory and are added in a fixed order, so results are
//    bit-reproducible. Fused epilogues store the outputs.
//  * Stages hand data to each other through exchange words: 64-bit
//    (tag, value) pairs written in one store. A reader polls the words it
//    needs until they carry the tag of the producing stage, so readiness and
//    data arrive together and no grid-wide barrier is needed. Each buffer's
//    next version can only be written after every reader of the current
//    version has read it (the forward's own data dependencies order them), and
//    a CTA with no rows in a stage reads nothing for it. Each thread polls
//    exactly the activation elements its lane multiplies, and the input
//    RMSNorm is applied to them in registers.
//  * Attention runs between QKV and O on n_kv x nsplit CTAs (the same body as
//    the standalone attention kernel: Q/K norm, RoPE, KV append, key-parallel
//    splits, here merged by split 0 from exchange words).
//  * The head (final RMSNorm, vocabulary GEMV, two-pass argmax) publishes the
//    next token as an exchange word for the next step's embedding gather.
//
// Every wait is bounded. On a timeout the CTA raises an abort flag, stops
// issuing, waits (bounded) for the copies already in flight, and the error
// word records the cause.
#pragma once
#include <cstdint>
#include <type_traits>

#include "attention.cuh"
#include "gemv_stream.cuh"
#include "ptx.cuh"

namespace wsg {

constexpr int kMkWarps = 8;                      // consumer warps
constexpr int kMkConsumers = kMkWarps * 32;
constexpr int kMkThreads = kMkConsumers + 128;   // plus a producer warpgroup (one active warp)
constexpr int kMkProducerRegs = 56;   // registers per thread after setmaxnreg: producer warpgroup
constexpr int kMkConsumerRegs = 224;  // consumer warpgroups (2 x 128 x 224 + 128 x 56 = 384 x 168)
constexpr int kMkSlot = 8192;         // bytes per ring slot
constexpr int kMkLayerPtrs = 12;      // pointers per layer in the shared layer table
constexpr int kMkQ = 8;               // boxes in flight per warp, at most (one mbarrier each)
constexpr int kMkMapsPerLayer = 7;    // tensor maps per layer: wq wk wv wo wg wu wd
constexpr int kMkMapBytes = 128;      // one CUtensorMap
constexpr int kMkXr = 4;              // float4 of x per lane: parts per warp (<= 2) x 128-column chunks (<= 2)
constexpr int kMkRowsMax = 16;       // rows of one-chunk part per box (the consumer unrolls over them)
constexpr int kMkPartRows = 256;      // row capacity of the shared partials of one epilogue chunk (at least)

enum : uint32_t { ERR_EXCHANGE_TIMEOUT = 1u << 4 };

struct MkLayer {
  const void *wq, *wk, *wv, *wo, *wg, *wu, *wd;
  const float *g_in, *g_post, *g_q, *g_k;
};

// Split-K streaming geometry of one matrix shape. The columns are cut into
// 8 * pw parts of cw columns (the last ones may reach past the row end: the
// copies fill zeros there); warp w owns parts w and, when pw == 2, w + 8.
// Boxes of R rows x cw columns stream through the warps' rings.
struct MkGeom {
  int32_t cw;         // columns per part (weights: a multiple of 16 bytes)
  int32_t pw;         // parts per warp: 1 or 2
  int32_t kc;         // 128-column chunks of a part: 1 or 2 (a lane covers 4 columns of each)
  int32_t R;          // rows per box
  int32_t box_bytes;  // R * cw * element size
  int32_t gchunk;     // row groups per epilogue chunk
  int32_t wpp;        // warps per part: 1, or 2 (one-part stages over 4 parts: warp w takes
                      // part w % 4 and the row groups whose index has the parity of w / 4)
};

// Column part of warp w, and which of the part's warps it is (its row groups
// are those with index % wpp == sub).
__device__ __forceinline__ int mk_part(const MkGeom& g, int w) { return g.wpp == 2 ? (w & 3) : w; }
__device__ __forceinline__ int mk_sub(const MkGeom& g, int w) { return g.wpp == 2 ? (w >> 2) : 0; }
__device__ __forceinline__ int mk_wpp(const MkGeom& g) { return g.wpp == 2 ? 2 : 1; }

struct MkArgs {
  const MkLayer* layers;  // device array [L]
  const void* maps;       // tensor maps [L][7] then the embedding's (128 bytes each, 64-byte aligned)
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
  int32_t ring_bytes;  // bytes of each warp's ring (a multiple of 128, at least one slot)
  int32_t xs_floats, part_floats, hown_floats;
  int32_t pos0, nsteps;
  int32_t head_every, head_last;  // head on every step / on the last step
  int32_t first_tok;   // >= 0: the first step's token (else read from tok[pos0])
  int32_t* host_next;  // optional (host memory mapped to the device): the last step's greedy token
  uint64_t* trace;  // optional: [G][L + 1][5][4] globaltimer stamps of the first forward
  uint64_t xwait_ns;  // limit of a wait for another CTA's words (exchange words, cache counts)
};

// Trace points per stage: entry, activations staged, segments consumed, barrier passed.
constexpr int kMkTraceStages = 5, kMkTraceEvents = 4;
// Per-box trace of every consumer warp of CTA 0 (first kMkTraceSegs boxes of
// each, from the launch's start), after the stage trace: [warp][box][event],
// events: wait begins, data ready, dot done (SM clock), and the %globaltimer
// stamp of the wait's beginning (to place the box among the stage events).
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

__device__ __forceinline__ const MkGeom& mk_geom(const MkArgs& a, int st) {
  return st == MK_QKV ? a.gq : st == MK_O ? a.go : st == MK_GU ? a.gg : st == MK_DOWN ? a.gd : a.gv;
}

// One stage's rows for this CTA: up to three contiguous row pieces (QKV spans
// the three source matrices; gate/up takes the gate rows, then the up rows,
// of the same units), each cut into row groups of R rows (one box per group
// and column part). Tensors are named by index: 0 wq, 1 wk, 2 wv, 3 wo,
// 4 wg, 5 wu, 6 wd, 7 the embedding; computed once per launch.
struct MkStageT {
  int t0, t1, t2;        // tensor of each piece
  int row0, row1, row2;  // first row of each piece within its tensor
  int nr0, nr1, nr2;     // rows per piece
  int l1, l2;            // local index of the first row of pieces 1 and 2 (piece 0 starts at 0)
  int g1, g2, ng;        // row groups: piece 0 [0, g1), piece 1 [g1, g2), piece 2 [g2, ng)
  int u0, nloc;
};

__device__ __forceinline__ MkStageT mk_stage_t(const MkArgs& a, int st, MkRange r) {
  const MkGeom& gm = mk_geom(a, st);
  MkStageT s;
  s.u0 = r.u0;
  s.t1 = s.t2 = 0;
  s.row1 = s.row2 = 0;
  s.nr1 = s.nr2 = 0;
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
    s.l2 = s.nloc;
  } else {
    s.t0 = st == MK_O ? 3 : st == MK_DOWN ? 6 : 7;
    s.row0 = r.u0;
    s.nr0 = r.u1 - r.u0;
    s.nloc = r.u1 - r.u0;
    s.l1 = s.l2 = s.nloc;
  }
  auto groups = [&](int n) { return (n + gm.R - 1) / gm.R; };
  s.g1 = groups(s.nr0);
  s.g2 = s.g1 + groups(s.nr1);
  s.ng = s.g2 + groups(s.nr2);
  return s;
}

// Row group rg of a stage: its tensor, first row in that tensor, rows, and
// the local index of its first row.
struct MkGroup {
  int t, y, nr, lrow;
};

__device__ __forceinline__ MkGroup mk_group(const MkStageT& s, int R, int rg) {
  const bool p0 = rg < s.g1, p1 = !p0 && rg < s.g2;
  const int gl = rg - (p0 ? 0 : p1 ? s.g1 : s.g2);
  MkGroup g;
  g.t = p0 ? s.t0 : p1 ? s.t1 : s.t2;
  g.y = (p0 ? s.row0 : p1 ? s.row1 : s.row2) + gl * R;
  g.nr = min(R, (p0 ? s.nr0 : p1 ? s.nr1 : s.nr2) - gl * R);
  g.lrow = (p0 ? 0 : p1 ? s.l1 : s.l2) + gl * R;
  return g;
}

// Slot of local row lr among the partials of the chunk that starts at row group cg.
__device__ __forceinline__ int mk_slot(const MkStageT& s, int R, int cg, int lr) {
  const bool p0 = lr < s.l1, p1 = !p0 && lr < s.l2;
  const int q = lr - (p0 ? 0 : p1 ? s.l1 : s.l2);
  const int rg = (p0 ? 0 : p1 ? s.g1 : s.g2) + q / R;
  return (rg - cg) * R + q % R;
}

__device__ __forceinline__ const void* mk_map(const MkArgs& a, int layer, int t) {
  const int i = t == 7 ? a.L * kMkMapsPerLayer : layer * kMkMapsPerLayer + t;
  return static_cast<const char*>(a.maps) + static_cast<size_t>(i) * kMkMapBytes;
}

// Raw weight words of four consecutive elements (f32: float4, bf16: uint2).
template <typename WT>
struct MkW4;
template <>
struct MkW4<float> {
  using T = float4;
  __device__ __forceinline__ static T zero() { return make_float4(0, 0, 0, 0); }
  __device__ __forceinline__ static T lds(const unsigned char* buf, int i) {
    return *reinterpret_cast<const float4*>(buf + static_cast<size_t>(i) * 4);
  }
  __device__ __forceinline__ static float dot(const T& w, const float4& x, float acc) {
    return fmaf(w.x, x.x, fmaf(w.y, x.y, fmaf(w.z, x.z, fmaf(w.w, x.w, acc))));
  }
  // even / odd columns into two accumulators, two products per instruction
  __device__ __forceinline__ static void dot2(const T& w, const float4& x, float& ae, float& ao) {
    ffma2(ae, ao, w.x, w.y, x.x, x.y);
    ffma2(ae, ao, w.z, w.w, x.z, x.w);
  }
};
template <>
struct MkW4<uint16_t> {
  using T = uint2;
  __device__ __forceinline__ static T zero() { return make_uint2(0, 0); }
  __device__ __forceinline__ static T lds(const unsigned char* buf, int i) {
    return *reinterpret_cast<const uint2*>(buf + static_cast<size_t>(i) * 2);
  }
  __device__ __forceinline__ static float dot(const T& w, const float4& x, float acc) {
    return fmaf(__uint_as_float(w.x << 16), x.x,
                fmaf(__uint_as_float(w.x & 0xFFFF0000u), x.y,
                     fmaf(__uint_as_float(w.y << 16), x.z, fmaf(__uint_as_float(w.y & 0xFFFF0000u), x.w, acc))));
  }
  __device__ __forceinline__ static void dot2(const T& w, const float4& x, float& ae, float& ao) {
    ffma2(ae, ao, __uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), x.x, x.y);
    ffma2(ae, ao, __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u), x.z, x.w);
  }
};

// Four consecutive elements at index i of a global row (16-byte aligned for
// f32, 8-byte for bf16).
template <typename WT>
__device__ __forceinline__ float4 ldg4(const void* row, int i);
template <>
__device__ __forceinline__ float4 ldg4<float>(const void* row, int i) {
  return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(row) + i));
}
template <>
__device__ __forceinline__ float4 ldg4<uint16_t>(const void* row, int i) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(row) + i));
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xFFFF0000u));
}

// Butterfly reduce-scatter of N (1 to 32, a power of two) per-lane values over the warp:
// at each step a lane keeps half of its values and adds the partner's copy of
// them; the remaining steps are plain sums. Returns the full 32-lane sum of
// value lane >> (5 - log2 N), held by every lane of that group.
template <int N>
__device__ __forceinline__ float reduce_scatter(float (&a)[N], int lane) {
  static_assert(N == 1 || N == 2 || N == 4 || N == 8 || N == 16 || N == 32, "at most 32 values, a power of two");
  int o = 16;
#pragma unroll
  for (int m = N; m > 1; m >>= 1, o >>= 1) {
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < m / 2; ++i) {
      const float send = hi ? a[i] : a[i + m / 2];
      const float keep = hi ? a[i + m / 2] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float v = a[0];
#pragma unroll
  for (int r = 32 / N / 2; r > 0; r >>= 1) v += __shfl_xor_sync(0xffffffffu, v, r);
  return v;
}


// Warpgroup-wide register reallocation (every thread of the warpgroup executes it).
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ bool mk_head_on(const MkArgs& a, int step) {
  return a.head_every || (a.head_last && step == a.nsteps - 1);
}

// Widest activation vector a stage can take (16 elements per consumer thread).
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

// Whether a bounded poll reads the clock in its round r: in round 1 (by then
// at least one load has followed the start time) and every 64th round after,
// so a limit shorter than a round trip ends any wait that one reload did not
// satisfy.
__device__ __forceinline__ bool poll_check_due(int r) { return r == 1 || (r & 63) == 63; }

// Value of an exchange word once its tag is `tag`; bounded poll. On timeout
// raises the abort flag, records the error and returns 0.
__device__ __forceinline__ float ll_wait(const uint64_t* p, uint32_t tag, uint64_t w, volatile int* abort,
                                         uint32_t* err, uint64_t limit_ns) {
  if (static_cast<uint32_t>(w >> 32) == tag) return __uint_as_float(static_cast<uint32_t>(w));
  const uint64_t t0 = globaltimer_ns();
  for (int it = 0;; ++it) {
    w = ll_load(p);
    if (static_cast<uint32_t>(w >> 32) == tag) return __uint_as_float(static_cast<uint32_t>(w));
    if (poll_check_due(it)) {
      if (*abort) return 0.f;
      if (globaltimer_ns() - t0 > limit_ns) {
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
  uint64_t wait_ns;      // limit of a wait for another CTA's words
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
      if (poll_check_due(round)) {
        if (*abort) break;
        if (globaltimer_ns() - t0 > wait_ns) {
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
  // One round for split 0's merge: element e of head h's O of splits 1 ..
  // nsplit - 1 into ov[0 .. nsplit - 2], and word `ml` (< 0: none) of the
  // splits' (M, L) pairs, ordered split, head, M then L, into *mlv. gbase:
  // word offset of (head g, split 0, query head 0); a split's block of group
  // heads is group (d + 2) words long.
  template <int KO>
  __device__ __forceinline__ void poll_merge(size_t gbase, int nsplit, int group, int h, int e, int d, int ml,
                                             float* ov, float* mlv) const {
    uint64_t w[KO + 1];
    const uint64_t* pg = part + gbase;
    const size_t hs = static_cast<size_t>(d) + 2, ss = static_cast<size_t>(group) * hs;
    poll<KO + 1>(
        [&](int j) -> const uint64_t* {
          if (j < KO) return j < nsplit - 1 ? pg + (j + 1) * ss + h * hs + e : nullptr;
          if (ml < 0) return nullptr;
          const int k = 1 + ml / (2 * group), hh = (ml >> 1) % group;
          return pg + k * ss + hh * hs + d + (ml & 1);
        },
        tag_out, w);
#pragma unroll
    for (int j = 0; j < KO; ++j) ov[j] = __uint_as_float(static_cast<uint32_t>(w[j]));
    *mlv = __uint_as_float(static_cast<uint32_t>(w[KO]));
  }
  __device__ __forceinline__ void publish_kv(int g, int pos) const {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(kv_ready + g), "r"(static_cast<uint32_t>(pos + 1))
                 : "memory");
  }
};

// Bounded wait until *p >= v, with acquire semantics.
__device__ __forceinline__ bool wait_at_least(const uint32_t* p, uint32_t v, volatile int* abort, uint32_t* err,
                                              uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (int it = 0;; ++it) {
    uint32_t x;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(x) : "l"(p) : "memory");
    if (x >= v) return true;
    if (poll_check_due(it)) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
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

// Issue cursor of one warp's ring: the next box to request, walking the
// stages of every layer of every step (and the head where it runs) in the
// order the warp consumes them. The current stage's rows are copied to
// registers when the cursor enters it.
struct MkCursor {
  int step, layer, st;  // stage being issued
  int j, n;             // next box of the stage, boxes in the stage
  int t0, t1, t2, row0, row1, row2, g1, g2;
  int pw, cw, R, box_bytes;
  int part, sub, wpp;   // this lane's warp: its column part, row-group parity, warps per part
  bool done;
};

template <typename WT, typename KT, int GMAX>
__global__ void __launch_bounds__(kMkThreads, 1) decode_megakernel(const MkArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red[64];
  __shared__ int redi[32];
  __shared__ int s_abort, s_last;
  __shared__ MkStageT s_stage[5];
  const uint32_t RB = static_cast<uint32_t>(a.ring_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;
  // per consumer warp: ring bytes; after all rings, kMkQ full and kMkQ empty
  // barriers per warp (one pair per box in flight)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(kMkWarps) * RB);
  uint64_t* empty = full + kMkWarps * kMkQ;
  float* xs = reinterpret_cast<float*>(empty + kMkWarps * kMkQ);
  float* part = xs + a.xs_floats;  // [rows of an epilogue chunk][8 warps]
  float* ascratch = xs;            // attention scratch
  const void** lptr = reinterpret_cast<const void**>(part + a.part_floats);  // [L][kMkLayerPtrs]
  volatile int* vabort = &s_abort;

  // ---- per-launch tables: every layer's tensor pointers, this CTA's stage rows ----
  for (int i = tid; i < a.L * kMkLayerPtrs; i += kMkThreads) {
    const int l = i / kMkLayerPtrs, k = i - l * kMkLayerPtrs;
    const MkLayer* p = a.layers + l;
    const void* v = nullptr;
    switch (k) {
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
  if (tid < kMkWarps * kMkQ) {
    mbar_init(&full[tid], 1);
    mbar_init(&empty[tid], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto layer_ptrs = [&](int l) { return lptr + l * kMkLayerPtrs; };

  // Issue cursor over the stages, in the order the consumers run them; the
  // current stage's rows are copied to registers when the cursor enters it.
  MkCursor cur;
  cur.step = 0;
  cur.layer = 0;
  cur.st = MK_QKV;
  cur.done = false;
  auto cur_next_stage = [&]() {
    if (cur.st == MK_VOCAB) {
      ++cur.step;
      cur.layer = 0;
      cur.st = MK_QKV;
    } else if (cur.st == MK_DOWN) {
      if (cur.layer + 1 < a.L) {
        ++cur.layer;
        cur.st = MK_QKV;
      } else if (mk_head_on(a, cur.step)) {
        cur.st = MK_VOCAB;
      } else {
        ++cur.step;
        cur.layer = 0;
        cur.st = MK_QKV;
      }
    } else {
      ++cur.st;
    }
  };
  auto cur_settle = [&]() {  // first stage, from the current one, with boxes for this CTA
    while (true) {
      if (cur.step >= a.nsteps) {
        cur.done = true;
        return;
      }
      const MkStageT& t = s_stage[cur.st];
      const MkGeom& gm = mk_geom(a, cur.st);
      cur.j = 0;
      cur.wpp = mk_wpp(gm);
      cur.part = mk_part(gm, lane);
      cur.sub = mk_sub(gm, lane);
      cur.n = (t.ng > cur.sub ? (t.ng - cur.sub + cur.wpp - 1) / cur.wpp : 0) * gm.pw;  // this warp's row groups
      if (cur.n > 0) {
        cur.t0 = t.t0, cur.t1 = t.t1, cur.t2 = t.t2;
        cur.row0 = t.row0, cur.row1 = t.row1, cur.row2 = t.row2;
        cur.g1 = t.g1, cur.g2 = t.g2;
        cur.pw = gm.pw, cur.cw = gm.cw, cur.R = gm.R, cur.box_bytes = gm.box_bytes;
        return;
      }
      cur_next_stage();
    }
  };

  // Keys and values of positions before pos do not depend on the token:
  // pull this CTA's attention range of them into L2 ahead of the attention
  // stage. A prefetch is only a hint (L2 is where writes become visible), so
  // it needs no ordering; the attention stage acquires the rows before reading
  // them. Issued by the producer warp, whose copies share the copy engine's
  // queue, so no consumer warp waits for room in it. The rows of layer l + 1
  // are final while layer l runs, so they are requested as soon as the issue
  // cursor leaves layer l's QKV stage: a layer ahead of their attention, while
  // the latency-bound projection stages leave HBM time unused.
  auto prefetch_attn = [&](int step, int l) {
    if (!(c < a.n_kv * a.at.nsplit_max) || step >= a.nsteps) return;
    const int pos = a.pos0 + step;
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
  };

  // Next (step, layer) whose attention range to prefetch, as step * L + layer.
  int pf_next = 0;
  auto prefetch_ahead = [&]() {
    if (cur.done) return;
    const int here = cur.step * a.L + cur.layer;
    // at a layer's QKV stage its own range is due (if not requested yet);
    // past it, the next layer's
    const int want = cur.st == MK_QKV ? here : here + 1;
    while (pf_next <= want) {
      prefetch_attn(pf_next / a.L, pf_next % a.L);
      ++pf_next;
    }
  };

  // ------------------------------------------------------------------ producer ----
  if (warp >= kMkWarps) {
    setmaxnreg_dec<kMkProducerRegs>();
    if (warp > kMkWarps) return;  // the rest of the warpgroup only gives its registers back
    // Lane w feeds consumer warp w's ring. Boxes sit at increasing virtual
    // byte offsets (skipping the ring's tail where a box would straddle its
    // end); a box may be issued when at most kMkQ boxes are in flight and it
    // ends within RB bytes of the start of the oldest box not yet released.
    // The warp stays converged: every pass, each lane retires the boxes its
    // consumer has released (non-blocking tests) and issues what fits.
    const int w = lane;
    const bool active = w < kMkWarps;
    uint64_t* wfull = full + (active ? w : 0) * kMkQ;
    uint64_t* wempty = empty + (active ? w : 0) * kMkQ;
    unsigned char* wring = smem + static_cast<size_t>(active ? w : 0) * RB;
    const uint64_t pol = l2_policy_evict_first();
    if (active) cur_settle();
    cur.done = cur.done || !active;
    // lane 0's cursor requests the attention ranges (every CTA has QKV rows,
    // so it passes every layer's QKV stage)
    if (lane == 0) prefetch_ahead();
    uint32_t vhead = 0, phead = 0;  // virtual and ring offset of the next box
    uint32_t qv[kMkQ];              // virtual offsets of the boxes in flight, oldest first
#pragma unroll
    for (int i = 0; i < kMkQ; ++i) qv[i] = 0;
    int issued = 0, retired = 0;
    uint64_t idle_since = 0;
    while (__any_sync(0xffffffffu, !cur.done || retired < issued)) {
      bool progress = false;
      // retire released boxes
      while (retired < issued && mbar_test(&wempty[retired % kMkQ], (retired / kMkQ) & 1)) {
#pragma unroll
        for (int i = 0; i + 1 < kMkQ; ++i) qv[i] = qv[i + 1];
        ++retired;
        progress = true;
      }
      // issue what fits
      while (!cur.done && issued - retired < kMkQ) {
        const uint32_t B = (static_cast<uint32_t>(cur.box_bytes) + 127u) & ~127u;
        uint32_t v = vhead, ph = phead;
        if (ph + B > RB) {
          v += RB - ph;
          ph = 0;
        }
        const int n = issued - retired;
        if (n > 0 && v + B - qv[0] > RB) break;  // not free yet
        const int li = cur.pw == 2 ? (cur.j >> 1) : cur.j, pj = cur.j - li * cur.pw;
        const int rg = cur.sub + cur.wpp * li;  // row group of this box
        const bool p0 = rg < cur.g1, p1 = !p0 && rg < cur.g2;
        const int gl = rg - (p0 ? 0 : p1 ? cur.g1 : cur.g2);
        const int t = p0 ? cur.t0 : p1 ? cur.t1 : cur.t2;
        const int y = (p0 ? cur.row0 : p1 ? cur.row1 : cur.row2) + gl * cur.R;
        const int q = issued % kMkQ;
        mbar_arrive_expect_tx(&wfull[q], static_cast<uint32_t>(cur.box_bytes));
        tma_load_2d(wring + ph, mk_map(a, cur.layer, t), (cur.part + (kMkWarps / cur.wpp) * pj) * cur.cw, y, &wfull[q],
                    pol);
#pragma unroll
        for (int i = 0; i < kMkQ; ++i)
          if (i == n) qv[i] = v;
        vhead = v + B;
        phead = ph + B;
        ++issued;
        progress = true;
        if (++cur.j >= cur.n) {
          cur_next_stage();
          cur_settle();
          if (lane == 0) prefetch_ahead();
        }
      }
      if (__any_sync(0xffffffffu, progress)) {
        idle_since = 0;
        continue;
      }
      // nothing to do this pass: back off, bounded
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
    if (*vabort && active)
      for (int k = max(retired, issued - kMkQ); k < issued; ++k) mbar_wait(&wfull[k % kMkQ], (k / kMkQ) & 1);
    return;
  }

  // ------------------------------------------------------------------ consumers ----
  setmaxnreg_inc<kMkConsumerRegs>();
  uint64_t* mfull = full + warp * kMkQ;
  uint64_t* mempty = empty + warp * kMkQ;
  const unsigned char* myring = smem + static_cast<size_t>(warp) * RB;
  // Ring position of the next box to read: its barrier, phase parity, and the
  // ring offset where the previous box ended (the producer's placement rule).
  int cq = 0;
  uint32_t cph = 0, chead = 0;
  int consumed = 0;
  float* hown = reinterpret_cast<float*>(lptr + a.L * kMkLayerPtrs);  // this CTA's rows of h

  const int qw = a.n_q * a.d;

  // Input column of this thread's x register q (part q / 2 of its warp,
  // 128-column chunk q % 2), or -1.
  auto xcol = [&](const MkGeom& gm, int q, int in) {
    const int j = q >> 1, k = q & 1, off = 4 * lane + 128 * k;
    const int col = (mk_part(gm, warp) + (kMkWarps / mk_wpp(gm)) * j) * gm.cw + off;
    return (j < gm.pw && k < gm.kc && off < gm.cw && col < in) ? col : -1;
  };
  // CTA-wide RMSNorm scale from per-thread sums of squares.
  auto norm_scale = [&](float ss, int in) {
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    consumer_sync();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kMkWarps; ++w) t += red[w];
    return 1.0f / sqrtf(t / static_cast<float>(in) + a.eps);
  };

  // Stage the activation vector from exchange words (tag `tag`) into this
  // thread's x registers: plain, or RMSNorm * gain. Threads poll the words
  // coalesced (thread t: words t, t + 256, ...; all requested first, then only
  // the stale ones reloaded together, one round trip per round), pass them
  // through shared memory, and after one barrier each lane picks up the
  // elements its warp's column parts need.
  auto stage_x = [&](const uint64_t* src, uint32_t tag, int in, const float* gain, const MkGeom& gm,
                     float4 (&xr)[kMkXr]) {
    constexpr int K = kMkMaxWidth / kMkConsumers;
    // the gain of this lane's columns does not depend on the exchange: request
    // it before polling so its latency is not on the stage's critical path
    float4 gv[kMkXr];
#pragma unroll
    for (int q = 0; q < kMkXr; ++q) {
      const int col = xcol(gm, q, in);
      gv[q] = (gain && col >= 0) ? __ldg(reinterpret_cast<const float4*>(gain + col)) : make_float4(0, 0, 0, 0);
    }
    uint64_t wv[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int i = tid + k * kMkConsumers;
      wv[k] = i < in ? ll_load(src + i) : (static_cast<uint64_t>(tag) << 32);
    }
    {
      const uint64_t t0 = globaltimer_ns();
      for (int round = 0;; ++round) {
        bool stale = false;
#pragma unroll
        for (int k = 0; k < K; ++k) stale |= static_cast<uint32_t>(wv[k] >> 32) != tag;
        if (!stale) break;
        if (poll_check_due(round)) {
          if (*vabort) break;
          if (globaltimer_ns() - t0 > a.xwait_ns) {
            *vabort = 1;
            atomicOr(a.err, ERR_EXCHANGE_TIMEOUT);
            break;
          }
        }
#pragma unroll
        for (int k = 0; k < K; ++k)
          if (static_cast<uint32_t>(wv[k] >> 32) != tag) wv[k] = ll_load(src + tid + k * kMkConsumers);
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int i = tid + k * kMkConsumers;
      if (i < in) {
        const float v = __uint_as_float(static_cast<uint32_t>(wv[k]));
        xs[i] = v;
        ss = fmaf(v, v, ss);
      }
    }
    if (gain) {
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
    }
    consumer_sync();
    float inv = 1.f;
    if (gain) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kMkWarps; ++w) t += red[w];
      inv = 1.0f / sqrtf(t / static_cast<float>(in) + a.eps);
    }
#pragma unroll
    for (int q = 0; q < kMkXr; ++q) {
      const int col = xcol(gm, q, in);
      xr[q] = make_float4(0, 0, 0, 0);
      if (col >= 0) {
        const float4 v = *reinterpret_cast<const float4*>(xs + col);
        if (gain) {
          const float4 g = gv[q];
          xr[q] = make_float4(v.x * inv * g.x, v.y * inv * g.y, v.z * inv * g.z, v.w * inv * g.w);
        } else {
          xr[q] = v;
        }
      }
    }
  };

  // Layer 0: RMSNorm of the token's embedding row.
  auto stage_embed = [&](int t, const float* gain, const MkGeom& gm, float4 (&xr)[kMkXr]) __attribute__((always_inline)) {
    const WT* row = static_cast<const WT*>(a.embed) + static_cast<size_t>(t) * a.H;
    float ss = 0.f;
    float4 gv[kMkXr];
#pragma unroll
    for (int q = 0; q < kMkXr; ++q) {
      const int col = xcol(gm, q, a.H);
      xr[q] = col >= 0 ? ldg4<WT>(row, col) : make_float4(0, 0, 0, 0);
      gv[q] = col >= 0 ? __ldg(reinterpret_cast<const float4*>(gain + col)) : make_float4(0, 0, 0, 0);
      ss = fmaf(xr[q].x, xr[q].x, fmaf(xr[q].y, xr[q].y, fmaf(xr[q].z, xr[q].z, fmaf(xr[q].w, xr[q].w, ss))));
    }
    // with two warps per part both hold the same columns: count them once
    const float inv = norm_scale(mk_sub(gm, warp) == 0 ? ss : 0.f, a.H);
#pragma unroll
    for (int q = 0; q < kMkXr; ++q) {
      xr[q].x = xr[q].x * inv * gv[q].x;
      xr[q].y = xr[q].y * inv * gv[q].y;
      xr[q].z = xr[q].z * inv * gv[q].z;
      xr[q].w = xr[q].w * inv * gv[q].w;
    }
  };

  uint64_t* segtrace = nullptr;
  if (a.trace && c == 0)
    segtrace = a.trace + static_cast<size_t>(G) * (a.L + 1) * kMkTraceStages * kMkTraceEvents +
               static_cast<size_t>(warp) * kMkTraceSegs * kMkTraceSegEvents;
  auto segstamp = [&](int ev) {
    if (segtrace && lane == 0 && consumed < kMkTraceSegs) {
      segtrace[consumed * kMkTraceSegEvents + ev] = clock64();
      if (ev == 0) segtrace[consumed * kMkTraceSegEvents + 3] = globaltimer_ns();
    }
  };

  // Sum of the 8 warp partials of local row lr (chunk starting at row group cg).
  auto row_value = [&](const MkStageT& st, const MkGeom& gm, int cg, int lr) {
    const int slot = mk_slot(st, gm.R, cg, lr);
    const float* p = part + slot * kMkWarps;
    if (gm.wpp != 2) {
      float v = p[0];
#pragma unroll
      for (int w = 1; w < kMkWarps; ++w) v += p[w];
      return v;
    }
    // two warps per part: the row's partials are those of the warps of its parity
    p += ((cg + slot / gm.R) & 1) * (kMkWarps / 2);
    float v = p[0];
#pragma unroll
    for (int w = 1; w < kMkWarps / 2; ++w) v += p[w];
    return v;
  };


  // This warp's boxes of one stage, in ring order: lane partials per row,
  // reduce-scatter, warp partials into part[]; after each chunk of row groups
  // the epilogue epi(cg, ce) reads the row sums of groups [cg, ce). KC
  // (128-column chunks per part) is a template constant so every register
  // array is indexed statically; the stage's piece sizes are copied to
  // registers once, so the loop reads shared memory only for weights and the
  // ring barriers. After a failed wait the warp skips its data work but keeps
  // every barrier of the stage, so the CTA leaves the stage together at the
  // next chunk boundary.
  uint64_t boxes_done_ns = 0;  // trace: when the CTA's warps finished a stage's first chunk of boxes
  auto consume_kc = [&](auto kc_tag, const MkStageT& st, const MkGeom& gm, const float4(&xr)[kMkXr],
                        auto&& epi) -> bool {
    constexpr int KC = decltype(kc_tag)::value;
    constexpr int RM = kMkRowsMax / KC;  // rows per box, at most
    constexpr int kSh = RM == 32 ? 0 : RM == 16 ? 1 : RM == 8 ? 2 : 3;
    using W = MkW4<WT>;
    const int R = gm.R, pw = gm.pw, cw = gm.cw, gchunk = gm.gchunk;
    const int ng = st.ng, g1 = st.g1, g2 = st.g2, nr0 = st.nr0, nr1 = st.nr1, nr2 = st.nr2;
    bool ok = true;
    for (int cg = 0; cg < ng; cg += gchunk) {
      const int ce = min(ng, cg + gchunk);
      const int wpp = mk_wpp(gm), sub = mk_sub(gm, warp);
      for (int rg = cg + (((sub - cg) % wpp) + wpp) % wpp; rg < ce; rg += wpp) {
        const bool p0 = rg < g1, p1 = !p0 && rg < g2;
        const int nr = min(R, (p0 ? nr0 : p1 ? nr1 : nr2) - (rg - (p0 ? 0 : p1 ? g1 : g2)) * R);
        float acc[RM], acc2[RM];  // even / odd columns of each row
#pragma unroll
        for (int r = 0; r < RM; ++r) acc[r] = acc2[r] = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (j >= pw) break;
          if (ok) {
            segstamp(0);
            ok = __all_sync(0xffffffffu, mbar_wait(&mfull[cq], cph));
            segstamp(1);
            if (!ok) {
              if (lane == 0) atomicOr(a.err, ERR_MBAR_TIMEOUT);
              *vabort = 1;
            }
          }
          if (ok) {
            const uint32_t B = (static_cast<uint32_t>(gm.box_bytes) + 127u) & ~127u;
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
            segstamp(2);
            // every lane's reads of the box completed (their values are in
            // registers): release its bytes to the producer
            __syncwarp();
            if (lane == 0) mbar_arrive(&mempty[cq]);
            ++consumed;
            if (++cq == kMkQ) {
              cq = 0;
              cph ^= 1u;
            }
          }
        }
#pragma unroll
        for (int r = 0; r < RM; ++r) acc[r] += acc2[r];
        const float v = reduce_scatter<RM>(acc, lane);
        const int r = lane >> kSh;
        if (ok && (lane & ((1 << kSh) - 1)) == 0 && r < nr) part[((rg - cg) * R + r) * kMkWarps + warp] = v;
      }
      consumer_sync();
      if (*vabort) return false;
      if (a.trace && tid == 0 && cg == 0) boxes_done_ns = globaltimer_ns();
      epi(cg, ce);
      consumer_sync();
    }
    return !*vabort;
  };
  auto consume = [&](const MkStageT& st, const MkGeom& gm, const float4(&xr)[kMkXr], auto&& epi)
                     __attribute__((always_inline)) -> bool {
    if (gm.kc == 1) return consume_kc(std::integral_constant<int, 1>{}, st, gm, xr, epi);
    return consume_kc(std::integral_constant<int, 2>{}, st, gm, xr, epi);
  };

  // Trace events per stage: 0 entry, 1 inputs staged, 2 outputs published, 3 (projections)
  // every warp of the CTA done with the boxes / (attention) key loop done.
  auto stamp = [&](int step, int l, int st, int ev) {
    if (a.trace && step == 0 && tid == 0)
      a.trace[((static_cast<size_t>(c) * (a.L + 1) + l) * kMkTraceStages + st) * kMkTraceEvents + ev] =
          globaltimer_ns();
  };

  const bool attn_cta = c < a.n_kv * a.at.nsplit_max;
  bool ok = true;
  float4 xr[kMkXr];
  for (int step = 0; step < a.nsteps && ok; ++step) {
    const int pos = a.pos0 + step;
    // The token: written by the host before the launch, or published by the
    // previous step's head.
    int tok;
    if (step > 0 && a.head_every) {
      const uint64_t* p = a.ll_tok;
      tok = __float_as_int(ll_wait(p, mk_tag(a, step - 1, a.L, 0), ll_load(p), vabort, a.err, a.xwait_ns));
    } else if (step == 0 && a.first_tok >= 0) {
      tok = a.first_tok;  // passed with the launch: no copy ahead of it
      if (c == 0 && tid == 0) a.tok[pos] = tok;
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
        ll_wait(p, mk_tag(a, step - 1, a.L - 1, MK_DOWN), ll_load(p), vabort, a.err, a.xwait_ns);
      }
      consumer_sync();
    }
    for (int l = 0; l < a.L && ok && !*vabort; ++l) {
      const void* const* lp = layer_ptrs(l);
      const float* g_in = static_cast<const float*>(lp[7]);
      const float* g_post = static_cast<const float*>(lp[8]);
      // The four projections of the layer run through one copy of the staging,
      // consume and epilogue code (a loop over the stage kind, its inputs and
      // epilogue picked at run time): five unrolled copies of the consumer's
      // dot loop do not stay in the instruction cache together.
      for (int sid = MK_QKV; sid <= MK_DOWN; ++sid) {
        if (sid == MK_O && attn_cta) {
          // ---- attention (Q/K norm, RoPE, KV append, key-parallel splits) ----
          AttnArgs at = a.at;
          at.g_q = static_cast<const float*>(lp[9]);
          at.g_k = static_cast<const float*>(lp[10]);
          at.kc = static_cast<char*>(a.at.kc) + static_cast<size_t>(l) * a.kv_layer_bytes;
          at.vc = static_cast<char*>(a.at.vc) + static_cast<size_t>(l) * a.kv_layer_bytes;
          stamp(step, l, 1, 0);
          {
            // Cache rows below pos were appended by earlier forwards: every
            // thread acquires their published count before reading them, so
            // no barrier is needed; the wait overlaps the one for q/k/v. Every
            // active split acquires, the one appending row pos included, so
            // each published count covers all rows below it.
            int t0, t1, ns;
            if (pos > 0 && attn_split_range(a.at, c / a.n_kv, pos, &t0, &t1, &ns))
              wait_at_least(a.kv_ready + l * a.n_kv + c % a.n_kv, static_cast<uint32_t>(pos), vabort, a.err, a.xwait_ns);
          }
          attn_decode_body<KT, GMAX, kMkConsumers, ConsumerSync, (GMAX <= 2 ? kAttnChunk<KT> / 2 : 8), AttnLlIo>(
              at, c % a.n_kv, c / a.n_kv, pos, ascratch, tid, ConsumerSync{}, &s_last,
              AttnLlIo{a.ll_qkv, a.ll_attn, a.ll_apart, a.kv_ready + l * a.n_kv, mk_tag(a, step, l, MK_QKV),
                       mk_tag(a, step, l, 1), vabort, a.err, a.xwait_ns,
                       (a.trace && step == 0)
                           ? a.trace + ((static_cast<size_t>(c) * (a.L + 1) + l) * kMkTraceStages + 1) * kMkTraceEvents
                           : nullptr});
          stamp(step, l, 1, 2);
          consumer_sync();  // the attention scratch is reused by the next layer's attention
        }
        const int ts = sid == MK_QKV ? 0 : sid + 1;  // trace stage (1 is attention)
        const MkStageT& st = s_stage[sid];
        const MkGeom& gm = sid == MK_QKV ? a.gq : sid == MK_O ? a.go : sid == MK_GU ? a.gg : a.gd;
        stamp(step, l, ts, 0);
        if (st.nloc > 0) {
          if (sid == MK_QKV && l == 0) {
            stage_embed(tok, g_in, gm, xr);  // the token's embedding row, with the input RMSNorm
          } else {
            // QKV: previous layer's residual (input RMSNorm); O: attention output;
            // GU: residual after attention (post-attention RMSNorm); DOWN: SwiGLU output
            const uint64_t* src = sid == MK_QKV ? a.ll_h : sid == MK_O ? a.ll_attn : sid == MK_GU ? a.ll_h : a.ll_act;
            const uint32_t tin = sid == MK_QKV ? mk_tag(a, step, l - 1, MK_DOWN)
                                 : sid == MK_O  ? mk_tag(a, step, l, 1)
                                 : sid == MK_GU ? mk_tag(a, step, l, MK_O)
                                                : mk_tag(a, step, l, MK_GU);
            const int n = sid == MK_O ? qw : sid == MK_DOWN ? a.I : a.H;
            const float* gain = sid == MK_QKV ? g_in : sid == MK_GU ? g_post : nullptr;
            stage_x(src, tin, n, gain, gm, xr);
          }
        }
        stamp(step, l, ts, 1);
        const uint32_t tg = mk_tag(a, step, l, sid);
        ok = consume(st, gm, xr, [&](int cg, int) {
          if (sid == MK_QKV) {
            for (int lr = tid; lr < st.nloc; lr += kMkConsumers) ll_store(a.ll_qkv + st.u0 + lr, row_value(st, gm, cg, lr), tg);
          } else if (sid == MK_GU) {
            const int np = st.nloc >> 1;
            for (int i = tid; i < np; i += kMkConsumers)
              ll_store(a.ll_act + st.u0 + i, silu_f32(row_value(st, gm, cg, i)) * row_value(st, gm, cg, np + i), tg);
          } else {
            // O and DOWN: residual add into this CTA's rows of h (layer 0's O adds
            // to the embedding row)
            for (int lr = tid; lr < st.nloc; lr += kMkConsumers) {
              const int row = st.u0 + lr;
              const float prev = (sid == MK_O && l == 0)
                                     ? load_f32<WT>(static_cast<const WT*>(a.embed) + static_cast<size_t>(tok) * a.H, row)
                                     : hown[lr];
              const float hn = prev + row_value(st, gm, cg, lr);
              hown[lr] = hn;
              ll_store(a.ll_h + row, hn, tg);
            }
          }
        });
        if (!ok) break;
        stamp(step, l, ts, 2);
        if (a.trace && step == 0 && tid == 0)
          a.trace[((static_cast<size_t>(c) * (a.L + 1) + l) * kMkTraceStages + ts) * kMkTraceEvents + 3] = boxes_done_ns;
      }
    }
    if (!ok || *vabort || !mk_head_on(a, step)) continue;
    // ---- head: final RMSNorm, tied vocabulary projection, two-pass argmax ----
    stamp(step, a.L, 0, 0);
    const MkStageT& st = s_stage[MK_VOCAB];
    if (st.nloc > 0) stage_x(a.ll_h, mk_tag(a, step, a.L - 1, MK_DOWN), a.H, a.g_final, a.gv, xr);
    stamp(step, a.L, 0, 1);
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    if (!(ok = consume(st, a.gv, xr, [&](int cg, int ce) {
          const int r0 = cg * a.gv.R, r1 = min(st.nloc, ce * a.gv.R);
          for (int lr = r0 + tid; lr < r1; lr += kMkConsumers) {
            const int row = st.u0 + lr;
            const float v = row_value(st, a.gv, cg, lr);
            if (a.logits) a.logits[row] = v;
            if (argmax_better(v, row, bv, bi)) {
              bv = v;
              bi = row;
            }
          }
        })))
      break;
    stamp(step, a.L, 0, 2);
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
        if (a.host_next && step == a.nsteps - 1) *a.host_next = gi;  // read by the host after the launch
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
