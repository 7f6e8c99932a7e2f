// Persistent decode megakernel: whole token-to-logits forwards in one launch.
//
// "Megakernels" (the page's opening and "GPU-wide end-to-end generation")
// puts a complete forward in one dispatch, but its single-threadgroup version
// leaves most of the GPU idle, and its GPU-wide version splits the forward into
// 227 ordered dispatches. This kernel keeps the whole GPU busy inside one
// launch: one CTA per SM, co-resident by cooperative launch.
//
//  * Every weight segment (at most 4 KB) this CTA will read, over all stages
//    of all requested steps (QKV, O, gate/up, down of every layer, then the
//    vocabulary slice), is assigned to one of its 8 warps: segment j of a
//    stage goes to warp j mod 8. Each warp owns a private ring of 4 KB
//    shared-memory slots and keeps it full: lane 0 walks a cursor through the
//    warp's future segments (across stage, layer and step boundaries) and
//    issues a bulk copy for the next one each time a slot is consumed.
//    Weights never depend on activations, so the rings hold the next stages'
//    weights while the CTA waits at a barrier and HBM keeps streaming.
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

constexpr int kMkWarps = 8;
constexpr int kMkThreads = kMkWarps * 32;
constexpr int kMkSlot = 4096;         // bytes per ring slot
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
};

enum MkStage : int { MK_QKV = 0, MK_O = 1, MK_GU = 2, MK_DOWN = 3, MK_VOCAB = 4 };

struct MkPiece {
  const char* base;  // first row of the piece
  int nrows;
  int local0;  // index of its first row among the CTA's local rows
};

struct MkSlice {
  MkPiece p[3];
  int np;
  int nloc;  // local rows
  int u0;    // first partition unit (row, or gate/up pair)
  int nseg;
};

__device__ __forceinline__ int mk_piece_segs(const MkGeom& gm, int nrows) {
  return gm.spr > 1 ? nrows * gm.spr : (nrows + gm.rps - 1) / gm.rps;
}

__device__ __forceinline__ const MkGeom& mk_geom(const MkArgs& a, int st) {
  return st == MK_QKV ? a.gq : st == MK_O ? a.go : st == MK_GU ? a.gg : st == MK_DOWN ? a.gd : a.gv;
}

// This CTA's rows of one stage: balanced contiguous units, cut at source boundaries.
__device__ __forceinline__ MkSlice mk_slice(const MkArgs& a, const MkLayer& lw, int st, int c, int G) {
  MkSlice s;
  s.np = 0;
  const MkGeom& gm = mk_geom(a, st);
  const int qw = a.n_q * a.d, kvw = a.n_kv * a.d;
  int units = st == MK_QKV ? qw + 2 * kvw : st == MK_GU ? a.I : st == MK_VOCAB ? a.V : a.H;
  const int u0 = static_cast<int>(static_cast<int64_t>(c) * units / G);
  const int u1 = static_cast<int>(static_cast<int64_t>(c + 1) * units / G);
  s.u0 = u0;
  auto add = [&](const void* base, int first_row, int nrows, int local0) {
    if (nrows <= 0) return;
    s.p[s.np].base = static_cast<const char*>(base) + static_cast<size_t>(first_row) * gm.row_bytes;
    s.p[s.np].nrows = nrows;
    s.p[s.np].local0 = local0;
    ++s.np;
  };
  if (st == MK_QKV) {
    const int lo[3] = {0, qw, qw + kvw}, hi[3] = {qw, qw + kvw, qw + 2 * kvw};
    const void* b[3] = {lw.wq, lw.wk, lw.wv};
    for (int k = 0; k < 3; ++k) {
      const int x0 = max(u0, lo[k]), x1 = min(u1, hi[k]);
      add(b[k], x0 - lo[k], x1 - x0, x0 - u0);
    }
    s.nloc = u1 - u0;
  } else if (st == MK_GU) {
    add(lw.wg, u0, u1 - u0, 0);
    add(lw.wu, u0, u1 - u0, u1 - u0);
    s.nloc = 2 * (u1 - u0);
  } else {
    const void* b = st == MK_O ? lw.wo : st == MK_DOWN ? lw.wd : a.embed;
    add(b, u0, u1 - u0, 0);
    s.nloc = u1 - u0;
  }
  s.nseg = 0;
  for (int k = 0; k < s.np; ++k) s.nseg += mk_piece_segs(gm, s.p[k].nrows);
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

__device__ __forceinline__ MkSeg mk_seg(const MkSlice& s, const MkGeom& gm, int j) {
  int k = 0;
  while (k + 1 < s.np) {
    const int n = mk_piece_segs(gm, s.p[k].nrows);
    if (j < n) break;
    j -= n;
    ++k;
  }
  const MkPiece& p = s.p[k];
  MkSeg r;
  if (gm.spr > 1) {
    const int row = j / gm.spr, part = j - row * gm.spr;
    r.off = part * gm.seg_bytes;
    r.bytes = min(gm.seg_bytes, gm.row_bytes - r.off);
    r.src = p.base + static_cast<size_t>(row) * gm.row_bytes + r.off;
    r.lrow = p.local0 + row;
    r.part = part;
    r.nr = 1;
  } else {
    const int row = j * gm.rps;
    r.nr = min(gm.rps, p.nrows - row);
    r.off = 0;
    r.bytes = r.nr * gm.row_bytes;
    r.src = p.base + static_cast<size_t>(row) * gm.row_bytes;
    r.lrow = p.local0 + row;
    r.part = 0;
  }
  return r;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ bool mk_head_on(const MkArgs& a, int step) {
  return a.head_every || (a.head_last && step == a.nsteps - 1);
}

// Walks one warp's segments in consumption order: steps, layers, stages
// (QKV, O, gate/up, down, then the vocabulary on head steps), segment j of a
// stage for j = warp, warp + 8, ...
struct MkCursor {
  int step, layer, stage, j;
  bool done;
  MkSlice sl;
};

__device__ __forceinline__ void mk_cursor_settle(MkCursor& k, const MkArgs& a, int c, int G, int warp) {
  while (true) {
    if (k.step >= a.nsteps) {
      k.done = true;
      return;
    }
    k.sl = mk_slice(a, a.layers[k.stage == MK_VOCAB ? 0 : k.layer], k.stage, c, G);
    k.j = warp;
    if (k.j < k.sl.nseg) return;
    // next stage
    if (k.stage == MK_VOCAB) {
      ++k.step;
      k.layer = 0;
      k.stage = MK_QKV;
    } else if (k.stage == MK_DOWN) {
      if (k.layer + 1 < a.L) {
        ++k.layer;
        k.stage = MK_QKV;
      } else if (mk_head_on(a, k.step)) {
        k.stage = MK_VOCAB;
      } else {
        ++k.step;
        k.layer = 0;
        k.stage = MK_QKV;
      }
    } else {
      ++k.stage;
    }
  }
}

__device__ __forceinline__ void mk_cursor_next(MkCursor& k, const MkArgs& a, int c, int G, int warp) {
  k.j += kMkWarps;
  if (k.j < k.sl.nseg) return;
  if (k.stage == MK_VOCAB) {
    ++k.step;
    k.layer = 0;
    k.stage = MK_QKV;
  } else if (k.stage == MK_DOWN) {
    if (k.layer + 1 < a.L) {
      ++k.layer;
      k.stage = MK_QKV;
    } else if (mk_head_on(a, k.step)) {
      k.stage = MK_VOCAB;
    } else {
      ++k.step;
      k.layer = 0;
      k.stage = MK_QKV;
    }
  } else {
    ++k.stage;
  }
  mk_cursor_settle(k, a, c, G, warp);
}

template <typename WT, typename KT, int GMAX>
__global__ void __launch_bounds__(kMkThreads, 1) decode_megakernel(const MkArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red[64];
  __shared__ int redi[32];
  __shared__ int s_abort, s_last;
  const int R = a.wslots;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;
  unsigned char* myring = smem + static_cast<size_t>(warp) * R * kMkSlot;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(kMkWarps) * R * kMkSlot);
  uint64_t* mybars = bars + warp * kMkWarpSlotsMax;
  float* xs = reinterpret_cast<float*>(bars + kMkWarps * kMkWarpSlotsMax);
  float* part = xs + a.xs_floats;
  float* ascratch = xs;  // the attention stage reuses the GEMV staging area
  volatile int* vabort = &s_abort;

  // ---- each warp primes its ring ----
  MkCursor cur;
  int issued = 0;    // lane 0: segments issued into this warp's ring
  int consumed = 0;  // all lanes: segments consumed
  const uint64_t pol = l2_policy_evict_first();
  auto issue_one = [&]() {  // lane 0 only; requires issued < consumed + R
    const MkGeom& gm = mk_geom(a, cur.stage);
    const MkSeg sg = mk_seg(cur.sl, gm, cur.j);
    const int slot = issued % R;
    mbar_arrive_expect_tx(&mybars[slot], static_cast<uint32_t>(sg.bytes));
    bulk_g2s(myring + static_cast<size_t>(slot) * kMkSlot, sg.src, static_cast<uint32_t>(sg.bytes), &mybars[slot], pol);
    ++issued;
    mk_cursor_next(cur, a, c, G, warp);
  };
  if (tid == 0) {
    s_abort = 0;
    s_last = 0;
  }
  if (lane == 0) {
    for (int s = 0; s < R; ++s) mbar_init(&mybars[s], 1);
    fence_mbar_init();
    cur.step = 0;
    cur.layer = 0;
    cur.stage = MK_QKV;
    cur.done = false;
    mk_cursor_settle(cur, a, c, G, warp);
    while (!cur.done && issued < R) issue_one();
  }
  __syncthreads();

  uint32_t sync_target = 0;
  const int qw = a.n_q * a.d;

  auto grid_sync = [&]() -> bool {
    __syncthreads();
    if (tid == 0) {
      sync_target += G;
      __threadfence();
      atomicAdd(a.bar, 1u);
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(a.bar) < sync_target) {
        if (globaltimer_ns() - t0 > WSG_WAIT_LIMIT_NS) {
          *vabort = 1;
          atomicOr(a.err, ERR_GRID_BARRIER_TIMEOUT);
          break;
        }
      }
    }
    __syncthreads();
    return !*vabort;
  };

  // Stage the activation vector: plain copy, or RMSNorm(src) * gain.
  auto stage_x = [&](const float* src, const WT* wsrc, int in, const float* gain, bool store_h) {
    float ss = 0.f;
    for (int i = tid; i < in; i += kMkThreads) {
      const float v = wsrc ? load_f32<WT>(wsrc, i) : __ldcg(src + i);
      if (store_h) a.h[i] = v;
      xs[xs_index<WT>(i, in)] = v;
      ss = fmaf(v, v, ss);
    }
    if (gain) {
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kMkWarps; ++w) t += red[w];
      const float inv = 1.0f / sqrtf(t / static_cast<float>(in) + a.eps);
      for (int i = tid; i < in; i += kMkThreads) {
        const int k = xs_index<WT>(i, in);
        xs[k] = xs[k] * inv * gain[i];
      }
    }
    __syncthreads();
  };

  // This warp's segments of one stage, in ring order, into part[].
  auto consume = [&](const MkSlice& sl, const MkGeom& gm, int in) -> bool {
    for (int j = warp; j < sl.nseg; j += kMkWarps) {
      const int slot = consumed % R;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&mybars[slot], (consumed / R) & 1));
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
        for (int r = 0; r < sg.nr; ++r) {
          float v = seg_dot<WT>(buf + static_cast<size_t>(r) * gm.row_bytes, xs, 0, gm.row_bytes, in, lane);
          v = warp_sum(v);
          if (lane == 0) part[sg.lrow + r] = v;
        }
      }
      __syncwarp();
      ++consumed;
      if (lane == 0 && !cur.done && !*vabort) {
        fence_proxy_async_smem();
        issue_one();
      }
    }
    __syncthreads();
    return !*vabort;
  };

  auto row_value = [&](const MkGeom& gm, int lr) {
    float v = 0.f;
    for (int k = 0; k < gm.spr; ++k) v += part[lr * gm.spr + k];
    return v;
  };

  bool ok = true;
  for (int step = 0; step < a.nsteps && ok; ++step) {
    const int pos = a.pos0 + step;
    for (int l = 0; l < a.L && ok; ++l) {
      const MkLayer lw = a.layers[l];
      // ---- QKV with the input RMSNorm (layer 0: of the token's embedding row) ----
      {
        const MkSlice sl = mk_slice(a, lw, MK_QKV, c, G);
        if (l == 0) {
          int t = __ldcg(a.tok + pos);
          if (t < 0 || t >= a.V) {
            if (tid == 0) atomicOr(a.err, ERR_BAD_TOKEN);
            t = 0;
          }
          stage_x(nullptr, static_cast<const WT*>(a.embed) + static_cast<size_t>(t) * a.H, a.H, lw.g_in, c == 0);
        } else {
          stage_x(a.h, nullptr, a.H, lw.g_in, false);
        }
        if (!(ok = consume(sl, a.gq, a.H))) break;
        for (int lr = tid; lr < sl.nloc; lr += kMkThreads) a.qkv[sl.u0 + lr] = row_value(a.gq, lr);
        if (!(ok = grid_sync())) break;
      }
      // ---- attention (Q/K norm, RoPE, KV append, key-parallel splits) ----
      {
        AttnArgs at = a.at;
        at.g_q = lw.g_q;
        at.g_k = lw.g_k;
        at.kc = static_cast<char*>(a.at.kc) + static_cast<size_t>(l) * a.kv_layer_bytes;
        at.vc = static_cast<char*>(a.at.vc) + static_cast<size_t>(l) * a.kv_layer_bytes;
        if (c < a.n_kv * at.nsplit_max)
          attn_decode_body<KT, GMAX, kMkThreads>(at, c % a.n_kv, c / a.n_kv, pos, ascratch, tid, CtaSync{}, &s_last);
        if (!(ok = grid_sync())) break;
      }
      // ---- O projection + residual ----
      {
        const MkSlice sl = mk_slice(a, lw, MK_O, c, G);
        stage_x(a.attn, nullptr, qw, nullptr, false);
        if (!(ok = consume(sl, a.go, qw))) break;
        for (int lr = tid; lr < sl.nloc; lr += kMkThreads) {
          const int row = sl.u0 + lr;
          a.h[row] = __ldcg(a.h + row) + row_value(a.go, lr);
        }
        if (!(ok = grid_sync())) break;
      }
      // ---- gate/up with the post-attention RMSNorm, SwiGLU ----
      {
        const MkSlice sl = mk_slice(a, lw, MK_GU, c, G);
        stage_x(a.h, nullptr, a.H, lw.g_post, false);
        if (!(ok = consume(sl, a.gg, a.H))) break;
        const int np = sl.nloc >> 1;
        for (int i = tid; i < np; i += kMkThreads)
          a.act[sl.u0 + i] = silu_f32(row_value(a.gg, i)) * row_value(a.gg, np + i);
        if (!(ok = grid_sync())) break;
      }
      // ---- down projection + residual ----
      {
        const MkSlice sl = mk_slice(a, lw, MK_DOWN, c, G);
        stage_x(a.act, nullptr, a.I, nullptr, false);
        if (!(ok = consume(sl, a.gd, a.I))) break;
        for (int lr = tid; lr < sl.nloc; lr += kMkThreads) {
          const int row = sl.u0 + lr;
          a.h[row] = __ldcg(a.h + row) + row_value(a.gd, lr);
        }
        if (!(ok = grid_sync())) break;
      }
    }
    if (!ok || !mk_head_on(a, step)) continue;
    // ---- head: final RMSNorm, tied vocabulary projection, two-pass argmax ----
    const MkSlice sl = mk_slice(a, a.layers[0], MK_VOCAB, c, G);
    stage_x(a.h, nullptr, a.H, a.g_final, false);
    if (!(ok = consume(sl, a.gv, a.H))) break;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int lr = tid; lr < sl.nloc; lr += kMkThreads) {
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
    __syncthreads();
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
    if (step + 1 < a.nsteps) ok = grid_sync();  // the next step reads the new token
  }

  // ---- after an abort: wait (bounded) for this warp's copies still in flight ----
  if (*vabort && lane == 0) {
    for (int g = consumed; g < issued; ++g) mbar_wait(&mybars[g % R], (g / R) & 1);
  }
  __syncthreads();

  // ---- exit: the last CTA out resets the barrier counters and publishes the position ----
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
