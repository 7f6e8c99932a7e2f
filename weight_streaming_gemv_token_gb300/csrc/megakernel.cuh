// Persistent decode megakernel: whole token-to-logits forwards in one launch.
//
// "Megakernels" (the page's opening and "GPU-wide end-to-end generation")
// puts a complete forward in one dispatch, but its single-threadgroup version
// leaves most of the GPU idle, and its GPU-wide version splits the forward into
// 227 ordered dispatches. This kernel keeps the whole GPU busy inside one
// launch: one CTA per SM, co-resident by cooperative launch.
//
//  * Warp 8 of each CTA is a producer. One lane streams, in order, every
//    weight segment this CTA will need for all stages of all requested steps
//    (QKV, O, gate/up, down of every layer, then the vocabulary slice) into a
//    ring of 4 KB shared-memory slots with bulk copies. Weights never depend
//    on activations, so the producer runs ahead across stage and layer
//    boundaries, limited only by free slots; HBM keeps streaming while the
//    consumers wait at barriers.
//  * Warps 0-7 are consumers. Per stage they stage the activation vector (with
//    the fused RMSNorm), take the stage's segments round-robin, reduce partial
//    dots in a fixed order, run the fused epilogue, and meet the other CTAs at
//    a grid barrier before the next stage reads what this one wrote.
//  * Attention runs between QKV and O on n_kv x nsplit CTAs (the same body as
//    the standalone attention kernel: Q/K norm, RoPE, KV append, key-parallel
//    splits merged by the last CTA).
//  * The head (final RMSNorm, vocabulary GEMV, two-pass argmax) writes the
//    next token, which the next step's embedding gather reads after a barrier.
//
// Every wait is bounded. On a timeout the CTA raises an abort flag, the
// producer stops issuing, the consumers wait (bounded) for the copies already
// in flight, and the error word records the cause.
#pragma once
#include <cstdint>

#include "attention.cuh"
#include "gemv_stream.cuh"
#include "ptx.cuh"

namespace wsg {

constexpr int kMkConsumerWarps = 8;
constexpr int kMkConsumers = kMkConsumerWarps * 32;
constexpr int kMkThreads = kMkConsumers + 32;
constexpr int kMkSlot = 4096;      // bytes per ring slot
constexpr int kMkSlotsMax = 64;    // ring depth limit (barrier array size)

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
  int32_t slots;  // ring slots in use (<= kMkSlotsMax)
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

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kMkConsumers) : "memory"); }

struct ConsumerSync {
  __device__ __forceinline__ void operator()() const { consumer_sync(); }
};

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct MkShared {
  int abort;          // set on any timeout
  int issued;         // segments the producer has issued
  int producer_done;  // producer has stopped issuing
  int s_last;
};

template <typename WT, typename KT, int GMAX>
__global__ void __launch_bounds__(kMkThreads, 1) decode_megakernel(const MkArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ MkShared sh;
  __shared__ float red[64];
  __shared__ int redi[32];
  const int S = a.slots;
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * kMkSlot);
  uint64_t* empty = full + kMkSlotsMax;
  float* xs = reinterpret_cast<float*>(empty + kMkSlotsMax);
  float* part = xs + a.xs_floats;
  float* ascratch = xs;  // the attention stage reuses the GEMV staging area

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;
  volatile MkShared* vsh = &sh;

  if (tid == 0) {
    sh.abort = 0;
    sh.issued = 0;
    sh.producer_done = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  auto head_on = [&](int step) { return a.head_every || (a.head_last && step == a.nsteps - 1); };

  // ------------------------------------------------------------- producer ----
  if (warp == kMkConsumerWarps) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int g = 0;
      bool stop = false;
      auto stream_stage = [&](const MkSlice& sl, const MkGeom& gm) {
        for (int j = 0; j < sl.nseg && !stop; ++j, ++g) {
          const int slot = g % S;
          if (g >= S && !mbar_wait(&empty[slot], ((g / S) - 1) & 1)) {
            vsh->abort = 1;
            atomicOr(a.err, ERR_MBAR_TIMEOUT);
            stop = true;
            break;
          }
          if (vsh->abort) {
            stop = true;
            break;
          }
          const MkSeg sg = mk_seg(sl, gm, j);
          mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(sg.bytes));
          bulk_g2s(ring + static_cast<size_t>(slot) * kMkSlot, sg.src, static_cast<uint32_t>(sg.bytes), &full[slot],
                   pol);
          vsh->issued = g + 1;
        }
      };
      for (int step = 0; step < a.nsteps && !stop; ++step) {
        for (int l = 0; l < a.L && !stop; ++l) {
          const MkLayer lw = a.layers[l];
          for (int st = MK_QKV; st <= MK_DOWN && !stop; ++st) stream_stage(mk_slice(a, lw, st, c, G), mk_geom(a, st));
        }
        if (!stop && head_on(step)) stream_stage(mk_slice(a, a.layers[0], MK_VOCAB, c, G), a.gv);
      }
      vsh->producer_done = 1;
    }
    return;
  }

  // ------------------------------------------------------------- consumers ----
  const int ctid = tid;  // 0 .. kMkConsumers-1
  int gbase = 0;         // global index of the current stage's first segment
  uint32_t sync_target = 0;
  const int qw = a.n_q * a.d;
  const int group = a.n_q / a.n_kv;

  auto grid_sync = [&]() -> bool {
    consumer_sync();
    if (ctid == 0) {
      sync_target += G;
      __threadfence();
      atomicAdd(a.bar, 1u);
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(a.bar) < sync_target) {
        if (vsh->abort) break;
        if (globaltimer_ns() - t0 > WSG_WAIT_LIMIT_NS) {
          vsh->abort = 1;
          atomicOr(a.err, ERR_GRID_BARRIER_TIMEOUT);
          break;
        }
      }
    }
    consumer_sync();
    return !vsh->abort;
  };

  // Stage the activation vector: plain copy, or RMSNorm(src) * gain.
  auto stage_x = [&](const float* src, const WT* wsrc, int in, const float* gain, bool store_h) {
    float ss = 0.f;
    for (int i = ctid; i < in; i += kMkConsumers) {
      const float v = wsrc ? load_f32<WT>(wsrc, i) : __ldcg(src + i);
      if (store_h) a.h[i] = v;
      xs[xs_index<WT>(i, in)] = v;
      ss = fmaf(v, v, ss);
    }
    if (gain) {
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
      consumer_sync();
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kMkConsumerWarps; ++w) t += red[w];
      const float inv = 1.0f / sqrtf(t / static_cast<float>(in) + a.eps);
      for (int i = ctid; i < in; i += kMkConsumers) {
        const int k = xs_index<WT>(i, in);
        xs[k] = xs[k] * inv * gain[i];
      }
    }
    consumer_sync();
  };

  // Consume this CTA's segments of one stage into part[].
  auto consume = [&](const MkSlice& sl, const MkGeom& gm, int in) -> bool {
    const int rchunks = gm.row_bytes >> 4;  // 16-byte chunks per row
    for (int j = warp; j < sl.nseg; j += kMkConsumerWarps) {
      const int g = gbase + j;
      const int slot = g % S;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], (g / S) & 1));
      if (!ok) {
        if (lane == 0) {
          vsh->abort = 1;
          atomicOr(a.err, ERR_MBAR_TIMEOUT);
        }
        return false;
      }
      const MkSeg sg = mk_seg(sl, gm, j);
      const unsigned char* buf = ring + static_cast<size_t>(slot) * kMkSlot;
      if (sg.nr == 1) {
        float v = seg_dot<WT>(buf, xs, sg.off / static_cast<int>(sizeof(WT)), sg.bytes, in, lane);
        v = warp_sum(v);
        if (lane == 0) part[sg.lrow * gm.spr + sg.part] = v;
      } else {
        for (int r = 0; r < sg.nr; ++r) {
          float v = seg_dot<WT>(buf + static_cast<size_t>(r) * gm.row_bytes, xs, 0, rchunks << 4, in, lane);
          v = warp_sum(v);
          if (lane == 0) part[sg.lrow + r] = v;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    gbase += sl.nseg;
    consumer_sync();
    return !vsh->abort;
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
            if (ctid == 0) atomicOr(a.err, ERR_BAD_TOKEN);
            t = 0;
          }
          stage_x(nullptr, static_cast<const WT*>(a.embed) + static_cast<size_t>(t) * a.H, a.H, lw.g_in, c == 0);
        } else {
          stage_x(a.h, nullptr, a.H, lw.g_in, false);
        }
        if (!(ok = consume(sl, a.gq, a.H))) break;
        for (int lr = ctid; lr < sl.nloc; lr += kMkConsumers) a.qkv[sl.u0 + lr] = row_value(a.gq, lr);
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
          attn_decode_body<KT, GMAX, kMkConsumers>(at, c % a.n_kv, c / a.n_kv, pos, ascratch, ctid, ConsumerSync{},
                                                   &sh.s_last);
        if (!(ok = grid_sync())) break;
      }
      // ---- O projection + residual ----
      {
        const MkSlice sl = mk_slice(a, lw, MK_O, c, G);
        stage_x(a.attn, nullptr, qw, nullptr, false);
        if (!(ok = consume(sl, a.go, qw))) break;
        for (int lr = ctid; lr < sl.nloc; lr += kMkConsumers) {
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
        for (int i = ctid; i < np; i += kMkConsumers) a.act[sl.u0 + i] = silu_f32(row_value(a.gg, i)) * row_value(a.gg, np + i);
        if (!(ok = grid_sync())) break;
      }
      // ---- down projection + residual ----
      {
        const MkSlice sl = mk_slice(a, lw, MK_DOWN, c, G);
        stage_x(a.act, nullptr, a.I, nullptr, false);
        if (!(ok = consume(sl, a.gd, a.I))) break;
        for (int lr = ctid; lr < sl.nloc; lr += kMkConsumers) {
          const int row = sl.u0 + lr;
          a.h[row] = __ldcg(a.h + row) + row_value(a.gd, lr);
        }
        if (!(ok = grid_sync())) break;
      }
    }
    if (!ok || !head_on(step)) continue;
    // ---- head: final RMSNorm, tied vocabulary projection, two-pass argmax ----
    const MkSlice sl = mk_slice(a, a.layers[0], MK_VOCAB, c, G);
    stage_x(a.h, nullptr, a.H, a.g_final, false);
    if (!(ok = consume(sl, a.gv, a.H))) break;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int lr = ctid; lr < sl.nloc; lr += kMkConsumers) {
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
    if (ctid == 0) {
      for (int w = 1; w < kMkConsumerWarps; ++w)
        if (argmax_better(red[w], redi[w], bv, bi)) {
          bv = red[w];
          bi = redi[w];
        }
      a.mval[c] = bv;
      a.midx[c] = bi;
      __threadfence();
      sh.s_last = atomicAdd(a.mcnt, 1u) == static_cast<uint32_t>(G - 1);
      if (sh.s_last) {
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

  // ---- drain after an abort: wait for the copies already issued ----
  if (vsh->abort) {
    if (ctid == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (!vsh->producer_done && globaltimer_ns() - t0 < WSG_WAIT_LIMIT_NS) {
      }
      const int issued = vsh->issued;
      for (int s = 0; s < S && s < issued; ++s) {
        const int last = issued - 1 - ((issued - 1 - s) % S);  // last segment issued into slot s
        mbar_wait(&full[s], (last / S) & 1);
      }
    }
    consumer_sync();
  }

  // ---- exit: the last CTA out resets the barrier counters and publishes the position ----
  if (ctid == 0) {
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
