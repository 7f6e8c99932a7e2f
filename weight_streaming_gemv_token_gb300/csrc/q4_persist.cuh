// Persistent 4-bit decode kernel: whole forwards of the 4-bit configuration in
// one cooperative launch ("Megakernels", opening and "GPU-wide end-to-end
// generation": the forward in one dispatch, the GPU kept busy; "Our Kernel
// Benchmark Was Measuring the System Cache", Summary: the 4-bit matvec).
//
// A 4-bit layer streams only 8.6 MB, so launched stage by stage the forward
// is bound by launch-to-launch latency, not by bytes. Here one CTA per SM runs
// every stage of every step:
//
//  * Every 4-bit matrix is cut into G row slices, one per CTA (slice c of a
//    matrix with n rows: rows [c n / G, (c + 1) n / G)). A producer lane walks
//    the fixed schedule of the call (per step: per layer Q, K, V, O, gate,
//    up, down, then the vocabulary slice when the step has a head) and
//    streams each slice in chunks of 8 R rows (codes, then scales, then
//    biases, 1D bulk copies) into a ring of stages, as far ahead as the ring
//    allows: weights never depend on activations, so they stream across
//    stage, layer and step boundaries while the consumers wait for inputs.
//  * Eight consumer warps run the stages in the same order. A GEMV stage
//    builds the bfloat16 x it needs (RMSNorm of the residual, the attention
//    output, or silu(gate) * up) in 16-bit fixed point, as the bulk 4-bit
//    kernel does, consumes its chunks with integer dot products, and stores
//    or adds its rows. Attention runs on n_kv x nsplit CTAs with the float
//    decoders' body (Q/K norm, RoPE, KV append, key splits merged by the last
//    split to finish).
//  * Dependent stages are separated by a grid barrier (all CTAs are resident:
//    cooperative launch) on a 64-bit arrival counter that only grows: each CTA
//    adds 1 with release semantics and polls with acquire loads until the
//    count reaches the barrier's multiple of G (every launch passes the same
//    number of barriers per CTA, so a launch starts at a multiple of G; its
//    first arrival tells each CTA that base).
//  * The head: each CTA stores its logits slice and the best (value, lowest
//    index) of it; after a barrier every CTA reduces the G candidates itself,
//    so the next step's embedding row needs no further barrier.
//
// Every wait is bounded: an mbarrier or barrier wait that gives up sets an
// error bit and the abort word, which every other wait also watches; the
// producer then waits (bounded) for its copies in flight.
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

#include "attention.cuh"
#include "gemv_q4.cuh"
#include "megakernel.cuh"  // setmaxnreg_inc / setmaxnreg_dec
#include "ptx.cuh"

namespace wsg {

constexpr int kQ4pR = 4;                     // rows per warp per chunk
constexpr int kQ4pRC = kQ4Warps * kQ4pR;     // rows per chunk
constexpr int kQ4pMaxStages = 32;
// 8 consumer warps (two warpgroups) and a producer warpgroup of which one lane
// works; the producer group gives registers back so the consumers (whose
// attention body holds a chunk of keys and values in registers) run with 224:
// 2 x 128 x 224 + 128 x 56 = 384 x 168, the launch's registers.
constexpr int kQ4pThreads = kQ4Warps * 32 + 128;
constexpr int kQ4pProducerRegs = 56;
constexpr int kQ4pConsumerRegs = 224;

enum : uint32_t { ERR_GRID_BARRIER_TIMEOUT = 1u << 6 };

struct Q4PLayer {
  Q4Seg q, k, v, o, gate, up, down;  // rows and pointers (y_off, cta0 unused)
  const float *g_in, *g_post, *g_q, *g_k;
};

struct Q4PArgs {
  const Q4PLayer* layers;  // device [L]
  Q4Seg head;              // the tied embedding as the vocabulary matrix [V][H]
  const float* g_final;
  int32_t L, H, I, qw, kvw, V;
  float eps;
  AttnArgs at;             // kc / vc of layer 0, rotary table, partials, counters, split rule
  size_t kv_layer_bytes;   // one layer's K (or V) cache
  float* h;                // [H]
  float* qkv;              // [qw + 2 kvw]
  float* attn;             // [qw]
  float* gu;               // [2 I]: gate, then up
  float* logits;           // [V]
  float* mval;             // [G] head candidates
  int32_t* midx;
  int32_t* tok;            // token stream [max_seq + 1]
  int32_t* ctrl;           // ctrl[0]: position
  int32_t* host_next;      // optional mapped host word: the last step's greedy token
  unsigned long long* bar;  // [0] arrivals (only grows), [1] abort
  int32_t pos0, nsteps, head_every, head_last, first_tok;
  int32_t nstages;
  uint32_t stage_bytes;    // multiple of 128
  uint32_t attn_bytes;     // attention scratch in shared memory (multiple of 16)
  uint32_t* err;
  uint64_t xwait_ns;       // limit of a grid-barrier wait
  uint64_t* trace;         // optional: [G][L + 1][5][4] globaltimer stamps of the first forward
};

// Threads 0..255 of every CTA; ends with all of this CTA's consumers past the
// barrier. `target` is the count that releases this barrier (0 before the
// first: it is set from the first arrival). Returns false if the barrier (or
// another CTA) gave up.
__device__ __forceinline__ bool q4p_grid_sync(unsigned long long* bar, unsigned long long G, unsigned long long& target,
                                              volatile int* vabort, uint32_t* err, int tid, uint64_t limit_ns) {
  q4_consumer_sync();
  if (tid == 0 && !*vabort) {
    unsigned long long old;
    asm volatile("atom.add.release.gpu.global.u64 %0, [%1], 1;" : "=l"(old) : "l"(bar) : "memory");
    if (target == 0) target = old - old % G;  // the launch's base
    target += G;
    const uint64_t t0 = globaltimer_ns();
    for (int it = 0;; ++it) {
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(bar) : "memory");
      if (v >= target) break;
      if (it == 1 || (it & 63) == 63) {  // the clock on the first re-poll, then every 64th
        unsigned long long ab;
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(ab) : "l"(bar + 1) : "memory");
        if (ab) {
          *vabort = 1;
          break;
        }
        if (globaltimer_ns() - t0 > limit_ns) {
          atomicOr(err, ERR_GRID_BARRIER_TIMEOUT);
          atomicExch(bar + 1, 1ull);
          *vabort = 1;
          break;
        }
      }
    }
  }
  q4_consumer_sync();
  return !*vabort;
}

__device__ __forceinline__ void q4p_slice(int rows, int c, int G, int* r0, int* n) {
  *r0 = static_cast<int>(static_cast<long long>(c) * rows / G);
  *n = static_cast<int>(static_cast<long long>(c + 1) * rows / G) - *r0;
}

struct Q4pSync {  // the attention body's barrier: the consumer warps only
  __device__ __forceinline__ void operator()() const { q4_consumer_sync(); }
};

// Shared memory: [ring: nstages x stage_bytes][xq: 4 x (in_max/32) uint4]
// [xu: in_max/32 float2][attention scratch][full: nstages][empty: nstages].
template <typename KT, int GMAX>
__global__ void __launch_bounds__(kQ4pThreads, 1) q4_persist_kernel(const Q4PArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_abort, s_last;
  __shared__ float s_rs[kQ4Warps];
  __shared__ float s_bv[kQ4Warps];
  __shared__ int s_bi[kQ4Warps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;
  const int S = a.nstages;
  const int in_max = max(a.H, max(a.qw, a.I));
  unsigned char* ring = smem;
  uint4* xq = reinterpret_cast<uint4*>(smem + static_cast<size_t>(S) * a.stage_bytes);
  float2* xu = reinterpret_cast<float2*>(xq + 4 * (in_max >> 5));
  float* asmem = reinterpret_cast<float*>(xu + (in_max >> 5));
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<unsigned char*>(asmem) + a.attn_bytes);
  uint64_t* empty = full + S;
  volatile int* vabort = &s_abort;
  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kQ4Warps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  auto has_head = [&](int step) { return a.head_every || (a.head_last && step == a.nsteps - 1); };

  // ---- producer: one lane streams every chunk of the call, in schedule order ----
  if (warp >= kQ4Warps) {
    setmaxnreg_dec<kQ4pProducerRegs>();
    if (warp > kQ4Warps || lane != 0) return;
    const uint64_t pol = l2_policy_evict_first();
    int st = 0;
    auto put = [&](const Q4Seg& sg, int in) {
      int r0, n;
      q4p_slice(sg.rows, c, G, &r0, &n);
      const uint32_t cb = static_cast<uint32_t>(in) >> 1, sbb = static_cast<uint32_t>(in) >> 5;
      for (int j = 0; j < n; j += kQ4pRC, ++st) {
        const int slot = st % S, rows = min(kQ4pRC, n - j);
        if (st >= S && !mbar_wait(&empty[slot], ((st / S) - 1) & 1)) {
          atomicOr(a.err, ERR_MBAR_TIMEOUT);
          *vabort = 1;
        }
        if (*vabort) return false;
        unsigned char* dst = ring + static_cast<size_t>(slot) * a.stage_bytes;
        const size_t row = static_cast<size_t>(r0 + j);
        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(rows) * (cb + 2 * sbb));
        bulk_g2s(dst, reinterpret_cast<const char*>(sg.codes) + row * cb, rows * cb, &full[slot], pol);
        bulk_g2s(dst + rows * cb, reinterpret_cast<const char*>(sg.scale) + row * sbb, rows * sbb, &full[slot], pol);
        bulk_g2s(dst + rows * (cb + sbb), reinterpret_cast<const char*>(sg.bias) + row * sbb, rows * sbb, &full[slot],
                 pol);
      }
      return true;
    };
    bool ok = true;
    for (int step = 0; step < a.nsteps && ok; ++step) {
      for (int l = 0; l < a.L && ok; ++l) {
        const Q4PLayer& w = a.layers[l];
        ok = put(w.q, a.H);
        // This CTA's attention keys and values of the earlier positions (they
        // do not depend on the token): into L2 while the layer's projections
        // run. A prefetch is only a hint; the attention reads them after the
        // grid barriers that order it after their writes.
        if (ok && c < a.at.n_kv * a.at.nsplit_max) {
          int t0, t1, ns;
          const int pos = a.pos0 + step;
          if (attn_split_range(a.at, c % a.at.nsplit_max, pos, &t0, &t1, &ns) && min(t1, pos) > t0) {
            const size_t rb = static_cast<size_t>(a.at.d) * sizeof(KT);
            const size_t off = static_cast<size_t>(l) * a.kv_layer_bytes +
                               (static_cast<size_t>(c / a.at.nsplit_max) * a.at.max_seq + t0) * rb;
            const uint32_t bytes = static_cast<uint32_t>(static_cast<size_t>(min(t1, pos) - t0) * rb);
            bulk_prefetch_l2(static_cast<const char*>(a.at.kc) + off, bytes);
            bulk_prefetch_l2(static_cast<const char*>(a.at.vc) + off, bytes);
          }
        }
        ok = ok && put(w.k, a.H) && put(w.v, a.H) && put(w.o, a.qw) && put(w.gate, a.H) && put(w.up, a.H) &&
             put(w.down, a.I);
      }
      if (ok && has_head(step)) ok = put(a.head, a.H);
    }
    // After an abort: shared memory must outlive the copies already issued.
    if (!ok)
      for (int k = max(0, st - S); k < st; ++k) mbar_wait(&full[k % S], (k / S) & 1);
    return;
  }

  // ---- consumers ----
  setmaxnreg_inc<kQ4pConsumerRegs>();
  unsigned long long target = 0;
  int st = 0;
  bool ok = true;
  // One GEMV stage over the CTA's slice of sg (input width in; x already
  // staged): y[y_off + row] = (or +=) the row's product.
  auto consume = [&](const Q4Seg& sg, int in, float* y, int y_off, bool add) {
    int r0, n;
    q4p_slice(sg.rows, c, G, &r0, &n);
    const uint32_t cb = static_cast<uint32_t>(in) >> 1, sbb = static_cast<uint32_t>(in) >> 5;
    const int nch = in >> 5;
    for (int j = 0; j < n && ok; j += kQ4pRC, ++st) {
      const int slot = st % S, rows = min(kQ4pRC, n - j);
      ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], (st / S) & 1));
      if (!ok) {
        if (lane == 0) {
          atomicOr(a.err, ERR_MBAR_TIMEOUT);
          atomicExch(a.bar + 1, 1ull);
        }
        *vabort = 1;
        break;
      }
      const unsigned char* base = ring + static_cast<size_t>(slot) * a.stage_bytes;
      float acc[kQ4pR];
#pragma unroll
      for (int v = 0; v < kQ4pR; ++v) acc[v] = 0.f;
      q4_chunk_dot<kQ4pR, 1>(base, base + rows * cb, base + rows * (cb + sbb), rows, cb, sbb, nch, xq, xu, warp, lane,
                             acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      const float v = reduce_scatter<kQ4pR>(acc, lane);
      const int i = lane >> 3, rr = warp + kQ4Warps * i;
      if ((lane & 7) == 0 && rr < rows) {
        float* yp = y + y_off + r0 + j + rr;
        *yp = add ? __ldcg(yp) + v : v;
      }
    }
  };
  auto sync_all = [&]() { ok = ok && q4p_grid_sync(a.bar, static_cast<unsigned long long>(G), target, vabort, a.err, tid, a.xwait_ns); };

  const int attn_ctas = a.at.n_kv * a.at.nsplit_max;
  // Trace of the first forward (tid 0 of every CTA): per layer and stage (QKV,
  // attention, O, gate/up, down; the head as layer L, stage 0), the stage's
  // entry, its x staged, its products done, and the grid barrier after it.
  auto stamp = [&](int step, int l, int st, int ev) {
    if (a.trace && step == 0 && tid == 0) a.trace[((static_cast<size_t>(c) * (a.L + 1) + l) * 5 + st) * 4 + ev] = globaltimer_ns();
  };
  int gi = 0;  // the previous step's greedy token
  for (int step = 0; step < a.nsteps && ok; ++step) {
    const int pos = a.pos0 + step;
    // embedding row of this step's token: this CTA's slice of h
    {
      int token;
      if (step == 0 && a.first_tok >= 0)
        token = a.first_tok;
      else if (step > 0 && a.head_every)
        token = gi;
      else
        token = __ldcg(a.tok + pos);
      if (token < 0 || token >= a.V) {
        if (tid == 0) atomicOr(a.err, ERR_BAD_TOKEN);
        token = 0;
      }
      if (c == 0 && tid == 0) a.tok[pos] = token;
      int r0, n;
      q4p_slice(a.H, c, G, &r0, &n);
      const unsigned char* E = reinterpret_cast<const unsigned char*>(a.head.codes);
      const uint32_t* codes = reinterpret_cast<const uint32_t*>(E) + static_cast<size_t>(token) * (a.H / 8);
      const __half* sc = reinterpret_cast<const __half*>(a.head.scale) + static_cast<size_t>(token) * (a.H / 64);
      const __half* bi = reinterpret_cast<const __half*>(a.head.bias) + static_cast<size_t>(token) * (a.H / 64);
      for (int j = r0 + tid; j < r0 + n; j += kQ4Warps * 32) {
        const uint32_t q = (__ldg(codes + (j >> 3)) >> (4 * (j & 7))) & 0xFu;
        a.h[j] = __fadd_rn(__fmul_rn(__half2float(sc[j >> 6]), static_cast<float>(q)), __half2float(bi[j >> 6]));
      }
    }
    sync_all();
    for (int l = 0; l < a.L && ok; ++l) {
      const Q4PLayer& w = a.layers[l];
      // Q, K, V with the input RMSNorm
      stamp(step, l, 0, 0);
      q4_stage_x<1, Q4X_NORM>(a.h, a.H, w.g_in, a.eps, a.H, xq, xu, s_rs, tid);
      stamp(step, l, 0, 1);
      consume(w.q, a.H, a.qkv, 0, false);
      consume(w.k, a.H, a.qkv, a.qw, false);
      consume(w.v, a.H, a.qkv, a.qw + a.kvw, false);
      stamp(step, l, 0, 2);
      sync_all();
      stamp(step, l, 0, 3);
      if (!ok) break;
      // attention
      stamp(step, l, 1, 0);
      if (c < attn_ctas) {
        AttnArgs at = a.at;
        at.g_q = w.g_q;
        at.g_k = w.g_k;
        at.kc = static_cast<unsigned char*>(a.at.kc) + static_cast<size_t>(l) * a.kv_layer_bytes;
        at.vc = static_cast<unsigned char*>(a.at.vc) + static_cast<size_t>(l) * a.kv_layer_bytes;
        attn_decode_body<KT, GMAX, kQ4Warps * 32, Q4pSync, GMAX <= 2 ? kAttnChunk<KT> / 2 : 8>(
            at, c / a.at.nsplit_max, c % a.at.nsplit_max, pos, asmem, tid, Q4pSync{}, &s_last,
            AttnPlainIo{a.qkv, a.attn});
      }
      stamp(step, l, 1, 2);
      sync_all();
      stamp(step, l, 1, 3);
      if (!ok) break;
      // O + residual
      stamp(step, l, 2, 0);
      q4_stage_x<1, Q4X_F32>(a.attn, a.qw, nullptr, 0.f, a.qw, xq, xu, s_rs, tid);
      stamp(step, l, 2, 1);
      consume(w.o, a.qw, a.h, 0, true);
      stamp(step, l, 2, 2);
      sync_all();
      stamp(step, l, 2, 3);
      if (!ok) break;
      // gate / up with the post-attention RMSNorm
      stamp(step, l, 3, 0);
      q4_stage_x<1, Q4X_NORM>(a.h, a.H, w.g_post, a.eps, a.H, xq, xu, s_rs, tid);
      stamp(step, l, 3, 1);
      consume(w.gate, a.H, a.gu, 0, false);
      consume(w.up, a.H, a.gu, a.I, false);
      stamp(step, l, 3, 2);
      sync_all();
      stamp(step, l, 3, 3);
      if (!ok) break;
      // down (SwiGLU prologue) + residual
      stamp(step, l, 4, 0);
      q4_stage_x<1, Q4X_SWIGLU>(a.gu, 2 * a.I, nullptr, 0.f, a.I, xq, xu, s_rs, tid);
      stamp(step, l, 4, 1);
      consume(w.down, a.I, a.h, 0, true);
      stamp(step, l, 4, 2);
      sync_all();
      stamp(step, l, 4, 3);
    }
    if (!ok) break;
    if (!has_head(step)) {
      if (c == 0 && tid == 0) a.ctrl[0] = pos + 1;
      continue;
    }
    // head: final RMSNorm, this CTA's logits slice and its best candidate
    stamp(step, a.L, 0, 0);
    q4_stage_x<1, Q4X_NORM>(a.h, a.H, a.g_final, a.eps, a.H, xq, xu, s_rs, tid);
    stamp(step, a.L, 0, 1);
    consume(a.head, a.H, a.logits, 0, false);
    stamp(step, a.L, 0, 2);
    q4_consumer_sync();
    {
      int r0, n;
      q4p_slice(a.V, c, G, &r0, &n);
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int r = r0 + tid; r < r0 + n; r += kQ4Warps * 32) {
        const float v = __ldcg(a.logits + r);
        if (argmax_better(v, r, bv, bi)) {
          bv = v;
          bi = r;
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
        s_bv[warp] = bv;
        s_bi[warp] = bi;
      }
      q4_consumer_sync();
      if (tid == 0) {
        for (int k = 1; k < kQ4Warps; ++k)
          if (argmax_better(s_bv[k], s_bi[k], bv, bi)) {
            bv = s_bv[k];
            bi = s_bi[k];
          }
        a.mval[c] = bv;
        a.midx[c] = bi;
      }
    }
    sync_all();
    if (!ok) break;
    // every CTA reduces the candidates (lowest index on ties)
    {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int k = tid; k < G; k += kQ4Warps * 32) {
        const float v = __ldcg(a.mval + k);
        const int i = __ldcg(a.midx + k);
        if (argmax_better(v, i, bv, bi)) {
          bv = v;
          bi = i;
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
      q4_consumer_sync();  // earlier readers of s_bv / s_bi are done
      if (lane == 0) {
        s_bv[warp] = bv;
        s_bi[warp] = bi;
      }
      q4_consumer_sync();
      bv = s_bv[0];
      bi = s_bi[0];
      for (int k = 1; k < kQ4Warps; ++k)
        if (argmax_better(s_bv[k], s_bi[k], bv, bi)) {
          bv = s_bv[k];
          bi = s_bi[k];
        }
      if (bi == 0x7fffffff) {  // every logit was NaN
        bi = 0;
        if (c == 0 && tid == 0) atomicOr(a.err, ERR_ARGMAX_NAN);
      }
      gi = bi;
    }
    if (c == 0 && tid == 0) {
      a.tok[pos + 1] = gi;
      a.ctrl[0] = pos + 1;
      if (a.host_next && step == a.nsteps - 1) *a.host_next = gi;
    }
    // the candidates are rewritten only after the next step's barriers
  }
}

}  // namespace wsg
