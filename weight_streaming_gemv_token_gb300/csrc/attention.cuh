// Decode attention for one token with the Q/K RMSNorm, RoPE and KV-cache
// append fused in front ("Megakernels", "What runs in the DSL": per-head Q/K
// RMSNorm -> RoPE -> grouped-query attention + KV update; "GPU-wide end-to-end
// generation": attention distributed over heads; "Chunked prefill for long
// prompts": single-token decode keeps a key-parallel attention path).
//
// Grid: (n_kv, nsplit_max). CTA (g, s) serves key/value head g and the
// n_q/n_kv query heads that read it, over one contiguous range of key
// positions (key-parallel split). Every CTA normalises and rotates the
// current token's q and k itself (a few hundred floats), so no separate
// kernel is needed; the CTA whose range holds the current position writes
// its k and v into the cache and uses the same stored values for the current
// key. Each warp runs an online softmax over its keys; warps merge in shared
// memory; splits merge through a last-CTA-done reduction (partials in the
// workspace, an atomic counter that the last CTA resets), with no spinning.
#pragma once
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace wsg {

struct AttnArgs {
  const float* qkv;  // q [n_q*d], k [n_kv*d], v [n_kv*d] (raw projections)
  const float* g_q;
  const float* g_k;
  float eps;
  const float* rope_cos;  // [max_seq][d/2]
  const float* rope_sin;
  const int32_t* ctrl;  // ctrl[0] = position of the current token
  void* kc;             // this layer's cache, [n_kv][max_seq][d]
  void* vc;
  int32_t max_seq, n_q, n_kv, d;
  float* out;  // [n_q*d]
  float* part;  // [n_kv][nsplit_max][group][d+2]
  uint32_t* counter;  // [n_kv]
  int32_t nsplit_max, tmin;
  float scale;  // 1/sqrt(d)
  uint32_t* err;
  int32_t pos_add;  // attn_decode_kernel: the row's position is ctrl[0] + pos_add
};

template <typename KT>
__device__ __forceinline__ float4 load4(const void* base, size_t idx);
template <>
__device__ __forceinline__ float4 load4<float>(const void* base, size_t idx) {
  return __ldcg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx));
}
template <>
__device__ __forceinline__ float4 load4<uint16_t>(const void* base, size_t idx) {
  const uint2 u = __ldcg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + idx));
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xFFFF0000u));
}

// The elements of a 16-byte piece of a cache row, and of 4 elements of a
// value row, as floats.
template <typename KT>
__device__ __forceinline__ void unpack_piece(const uint4& u, float* f);
template <>
__device__ __forceinline__ void unpack_piece<float>(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void unpack_piece<uint16_t>(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <typename KT, typename R>
__device__ __forceinline__ float4 unpack_row(const R& u);
template <>
__device__ __forceinline__ float4 unpack_row<float, uint4>(const uint4& u) {
  return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
}
template <>
__device__ __forceinline__ float4 unpack_row<uint16_t, uint2>(const uint2& u) {
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xFFFF0000u));
}

template <typename KT>
__device__ __forceinline__ float round_store(float v);
template <>
__device__ __forceinline__ float round_store<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float round_store<uint16_t>(float v) {
  return bf16_to_f32(f32_to_bf16_rn(v));
}

template <typename KT>
__device__ __forceinline__ void store1(void* base, size_t idx, float v);
template <>
__device__ __forceinline__ void store1<float>(void* base, size_t idx, float v) {
  static_cast<float*>(base)[idx] = v;
}
template <>
__device__ __forceinline__ void store1<uint16_t>(void* base, size_t idx, float v) {
  static_cast<uint16_t*>(base)[idx] = f32_to_bf16_rn(v);
}

// RMSNorm over d elements held in shared memory, then RoPE at position pos,
// in place; one warp. g, cs, sn: the gain and the cos/sin row, in shared memory.
// With round_k the result is also rounded to the cache's element type (the
// key is stored, and attended to, at that precision).
template <typename KT>
__device__ __forceinline__ void norm_rope_warp(float* v, const float* g, float eps, int d, const float* cs,
                                               const float* sn, int lane, bool round_k) {
  float ss = 0.f;
  for (int e = lane; e < d; e += 32) ss = fmaf(v[e], v[e], ss);
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
  for (int e = lane; e < d; e += 32) v[e] = v[e] * inv * g[e];
  __syncwarp();
  const int half = d >> 1;
  for (int i = lane; i < half; i += 32) {
    const float a = v[i], b = v[i + half], c = cs[i], s = sn[i];
    float lo = a * c - b * s, hi = a * s + b * c;
    if (round_k) {
      lo = round_store<KT>(lo);
      hi = round_store<KT>(hi);
    }
    v[i] = lo;
    v[i + half] = hi;
  }
  __syncwarp();
}

constexpr int kAttnWarps = 8;

struct CtaSync {  // barrier over the whole CTA
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};
// Keys one warp scores per round trip (a chunk): every load of a chunk, its
// key rows and value rows, is issued at once; the rows then take 64 + 64
// registers per lane for 128-element heads.
template <typename KT>
constexpr int kAttnChunk = sizeof(KT) == 2 ? 32 : 16;

inline size_t attn_smem_bytes(int group, int d) {
  // qn[group][d], kn[d], vn[d], per-warp (m, l)[group] and o[group][d], then
  // the tables gain_q[d], gain_k[d], cos[d/2], sin[d/2]
  return sizeof(float) * (static_cast<size_t>(group) * d + 2 * d + kAttnWarps * group * 2 +
                          static_cast<size_t>(kAttnWarps) * group * d + 3 * static_cast<size_t>(d)) +
         16;
}

// Key range [t0, t1) of split s for the token at position pos (keys 0..pos);
// false if split s has no keys. Splits hold at least tmin keys where possible
// and number at most nsplit_max.
__device__ __forceinline__ bool attn_split_range(const AttnArgs& a, int s, int pos, int* t0, int* t1, int* nsplit_out) {
  const int n = pos + 1;
  int nsplit = (n + a.tmin - 1) / a.tmin;
  if (nsplit > a.nsplit_max) nsplit = a.nsplit_max;
  const int per = (n + nsplit - 1) / nsplit;
  nsplit = (n + per - 1) / per;
  *nsplit_out = nsplit;
  if (s >= nsplit) return false;
  *t0 = s * per;
  *t1 = min(n, *t0 + per);
  return true;
}

// How the attention body reads the raw q/k/v projections and writes its
// output: directly from / to the buffers of AttnArgs (kernel-boundary
// ordering; splits merged by the last CTA to finish), or through another
// exchange (see the persistent kernel).
struct AttnPlainIo {
  static constexpr bool kPolledMerge = false;
  const float* qkv;
  float* out;
  // q of this head group into qn[group*d], k and v of head g into kn[d], vn[d]
  // (elements tid, tid + nt, ...).
  __device__ __forceinline__ void load_all(float* qn, float* kn, float* vn, int qbase, int kbase, int vbase, int nq_el,
                                           int d, int tid, int nt) const {
    for (int i = tid; i < nq_el; i += nt) qn[i] = __ldcg(qkv + qbase + i);
    for (int i = tid; i < d; i += nt) {
      kn[i] = __ldcg(qkv + kbase + i);
      vn[i] = __ldcg(qkv + vbase + i);
    }
  }
  __device__ __forceinline__ void store_out(int i, float v) const { out[i] = v; }
  // Called by one thread, after a CTA barrier that follows the cache append
  // of position pos of head g.
  __device__ __forceinline__ void publish_kv(int, int) const {}
  // Trace hook (thread 0): 1 = current q/k/v received by the CTA, 3 = key loop done.
  __device__ __forceinline__ void mark(int) const {}
  // Polled split merge (unused here).
  __device__ __forceinline__ void store_part(size_t, float) const {}
  template <int KC>
  __device__ __forceinline__ void poll_parts(size_t, size_t, int, int, int, float*, float*, float*) const {}
  template <int KO>
  __device__ __forceinline__ void poll_merge(size_t, int, int, int, int, int, int, float*, float*) const {}
};

// Split 0 merges up to this many other splits in one polling round (their
// O words in registers, their (M, L) pairs through shared memory).
constexpr int kAttnMergeOne = 24;

template <typename KT, int GMAX, int NT, typename Sync, int CK = kAttnChunk<KT>, typename Io = AttnPlainIo>
__device__ __forceinline__ void attn_decode_body(const AttnArgs& a, int g, int s, int pos, float* asmem, int tid,
                                                 Sync sync, int* s_last, Io io = Io{}) {
  static_assert(NT == kAttnWarps * 32, "the split layout assumes kAttnWarps warps");
  const int warp = tid >> 5, lane = tid & 31;
  const int d = a.d, group = a.n_q / a.n_kv, half = d >> 1;
  const int n = pos + 1;
  int t0, t1, nsplit;
  if (!attn_split_range(a, s, pos, &t0, &t1, &nsplit)) return;

  float* qn = asmem;                       // [group][d]
  float* kn = qn + group * d;              // [d]
  float* vn = kn + d;                      // [d]
  float* wm = vn + d;                      // [warps][group]
  float* wl = wm + kAttnWarps * group;     // [warps][group]
  float* wo = wl + kAttnWarps * group;     // [warps][group][d]
  float* tab = wo + kAttnWarps * group * d;  // gain_q[d], gain_k[d], cos[d/2], sin[d/2]

  const int kraw = a.n_q * d + g * d;
  const int vraw = a.n_q * d + a.n_kv * d + g * d;
  // Each warp takes a contiguous run of this CTA's keys, CK at a time.
  // Scores: 4 lanes per key, 8 keys per pass; lane (4 kq + sub) reads the
  // 16-byte pieces sub, sub + 4, ... of its key's row (a key's 4 lanes read
  // 64 contiguous bytes per load), dots them with q from shared memory, and
  // two shuffles add the 4 partial dots. Values: lane owns the 4 elements
  // [4 lane, 4 lane + 4) of every value row (one coalesced row per load),
  // weighted by the key's probability, shuffled from the key's lanes.
  static_assert(CK % 8 == 0, "a chunk is whole passes of 8 keys");
  constexpr int PE = 16 / static_cast<int>(sizeof(KT));  // elements per 16-byte piece
  constexpr int NPL = 128 / PE / 4;                        // pieces per lane per row (d <= 128)
  constexpr int NPASS = CK / 8;
  using VRow = typename std::conditional<sizeof(KT) == 2, uint2, uint4>::type;  // 4 elements
  const bool active = 4 * lane < d;
  const int kq = lane >> 2, sub = lane & 3;
  const int npieces = d / PE;
  const int per_w = (t1 - t0 + kAttnWarps - 1) / kAttnWarps;
  const int w0 = t0 + warp * per_w;
  const int w1 = min(t1, w0 + per_w);
  const size_t head_base = static_cast<size_t>(g) * a.max_seq * d;
  const unsigned char* kbytes = static_cast<const unsigned char*>(a.kc) + head_base * sizeof(KT);
  const unsigned char* vbytes = static_cast<const unsigned char*>(a.vc) + head_base * sizeof(KT);
  const size_t row_bytes = static_cast<size_t>(d) * sizeof(KT);
  uint4 kr[NPASS][NPL];
  VRow vr[CK];
  // The current position's row is not read from the cache (it is written by
  // this kernel): its key and value come from shared memory instead.
  // Keys and values of the chunk at cb into registers. In the loop the next
  // chunk's keys are requested once this chunk's scores are done, and its
  // values once this chunk's values are accumulated, so each chunk's loads
  // overlap the previous chunk's work without more registers.
  auto issue_k = [&](int cb) {
#pragma unroll
    for (int ps = 0; ps < NPASS; ++ps) {
      const int t = cb + ps * 8 + kq;
      const bool ok = t < w1 && t != pos;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int pc = i * 4 + sub;
        kr[ps][i] = (ok && pc < npieces)
                        ? __ldcg(reinterpret_cast<const uint4*>(kbytes + static_cast<size_t>(t) * row_bytes) + pc)
                        : make_uint4(0, 0, 0, 0);
      }
    }
  };
  auto issue_v = [&](int cb) {
#pragma unroll
    for (int j = 0; j < CK; ++j) {
      const int t = cb + j;
      VRow z{};
      vr[j] = (t < w1 && t != pos && active)
                  ? __ldcg(reinterpret_cast<const VRow*>(vbytes + static_cast<size_t>(t) * row_bytes) + lane)
                  : z;
    }
  };
  auto issue = [&](int cb) {
    issue_k(cb);
    issue_v(cb);
  };
  // Nothing below depends on this token until its q/k/v arrive: the gains,
  // the RoPE row and the first chunk of cached keys/values are requested
  // before waiting for them.
  float tv[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = tid + k * NT;
    const float* cs = a.rope_cos + static_cast<size_t>(pos) * half;
    const float* sn = a.rope_sin + static_cast<size_t>(pos) * half;
    tv[k] = i < d ? __ldg(a.g_q + i)
                  : i < 2 * d ? __ldg(a.g_k + i - d)
                              : i < 2 * d + half ? __ldg(cs + i - 2 * d) : i < 3 * d ? __ldg(sn + i - 2 * d - half) : 0.f;
  }
  if (w0 < w1) issue(w0);
  io.load_all(qn, kn, vn, (g * group) * d, kraw, vraw, group * d, d, tid, NT);
  for (int i = tid; i < d; i += NT) vn[i] = round_store<KT>(vn[i]);
#pragma unroll
  for (int k = 0; k < 2; ++k)
    if (tid + k * NT < 3 * d) tab[tid + k * NT] = tv[k];
  sync();
  if (tid == 0) io.mark(1);
  // Current token: RMSNorm -> RoPE of each q head and of k (k rounded to the cache type).
  for (int h = warp; h <= group; h += kAttnWarps)
    norm_rope_warp<KT>(h < group ? qn + h * d : kn, h < group ? tab : tab + d, a.eps, d, tab + 2 * d, tab + 2 * d + half,
                       lane, h == group);
  sync();
  if (t1 == n) {  // this CTA's range holds the current position: append to the cache
    for (int i = tid; i < d; i += NT) {
      store1<KT>(a.kc, head_base + static_cast<size_t>(pos) * d + i, kn[i]);
      store1<KT>(a.vc, head_base + static_cast<size_t>(pos) * d + i, vn[i]);
    }
  }

  float m[GMAX], l[GMAX];
  float4 o[GMAX];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
    o[h] = make_float4(0, 0, 0, 0);
  }

  for (int cb = w0; cb < w1; cb += CK) {
    // scores of this lane's key in every pass, for every head
    float sc[NPASS][GMAX];
#pragma unroll
    for (int ps = 0; ps < NPASS; ++ps) {
      const int t = cb + ps * 8 + kq;
      const bool cur = t == pos;
      float acc[GMAX];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) acc[h] = 0.f;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int pc = i * 4 + sub;
        if (pc < npieces) {
          float kf[PE];
          unpack_piece<KT>(kr[ps][i], kf);
          if (cur) {
#pragma unroll
            for (int e = 0; e < PE; e += 4) {
              const float4 c4 = *reinterpret_cast<const float4*>(kn + pc * PE + e);
              kf[e] = c4.x;
              kf[e + 1] = c4.y;
              kf[e + 2] = c4.z;
              kf[e + 3] = c4.w;
            }
          }
#pragma unroll
          for (int h = 0; h < GMAX; ++h) {
            if (h >= group) break;
#pragma unroll
            for (int e = 0; e < PE; e += 4) {
              const float4 q4 = *reinterpret_cast<const float4*>(qn + h * d + pc * PE + e);
              acc[h] = fmaf(q4.x, kf[e], acc[h]);
              acc[h] = fmaf(q4.y, kf[e + 1], acc[h]);
              acc[h] = fmaf(q4.z, kf[e + 2], acc[h]);
              acc[h] = fmaf(q4.w, kf[e + 3], acc[h]);
            }
          }
        }
      }
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
        acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 2);
        sc[ps][h] = t < w1 ? acc[h] * a.scale : -INFINITY;
      }
    }
    if (cb + CK < w1) issue_k(cb + CK);
    // online softmax over the chunk; pr = this lane's key's probability per pass
    float pr[NPASS][GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      if (h >= group) break;
      float mx = sc[0][h];
#pragma unroll
      for (int ps = 1; ps < NPASS; ++ps) mx = fmaxf(mx, sc[ps][h]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float mn = fmaxf(m[h], mx);
      const float corr = expf(m[h] - mn);
      float ls = 0.f;
#pragma unroll
      for (int ps = 0; ps < NPASS; ++ps) {
        pr[ps][h] = expf(sc[ps][h] - mn);
        ls += pr[ps][h];
      }
      ls += __shfl_xor_sync(0xffffffffu, ls, 4);
      ls += __shfl_xor_sync(0xffffffffu, ls, 8);
      ls += __shfl_xor_sync(0xffffffffu, ls, 16);
      l[h] = fmaf(l[h], corr, ls);
      o[h].x *= corr;
      o[h].y *= corr;
      o[h].z *= corr;
      o[h].w *= corr;
      m[h] = mn;
    }
#pragma unroll
    for (int j = 0; j < CK; ++j) {
      if (cb + j >= w1) break;
      float4 v = unpack_row<KT>(vr[j]);
      if (cb + j == pos && active) v = *reinterpret_cast<const float4*>(vn + 4 * lane);
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        if (h >= group) break;
        const float pj = __shfl_sync(0xffffffffu, pr[j >> 3][h], (j & 7) * 4);
        o[h].x = fmaf(pj, v.x, o[h].x);
        o[h].y = fmaf(pj, v.y, o[h].y);
        o[h].z = fmaf(pj, v.z, o[h].z);
        o[h].w = fmaf(pj, v.w, o[h].w);
      }
    }
    if (cb + CK < w1) issue_v(cb + CK);
  }

  if (tid == 0) io.mark(3);
  // Merge the warps of this CTA.
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    if (h >= group) break;
    if (lane == 0) {
      wm[warp * group + h] = m[h];
      wl[warp * group + h] = l[h];
    }
    if (active) *reinterpret_cast<float4*>(wo + (warp * group + h) * d + 4 * lane) = o[h];
  }
  sync();
  const bool merger = Io::kPolledMerge && nsplit > 1 && s == 0;
  // Split 0 in one round: every thread one output element (group * d <= NT),
  // the other splits' (M, L) pairs fitting in the q/k/v scratch (dead now).
  const bool one_round = merger && group * d <= NT && nsplit - 1 <= kAttnMergeOne &&
                         2 * (nsplit - 1) * group <= (group + 2) * d && 2 * (nsplit - 1) * group <= NT;
  if constexpr (Io::kPolledMerge) {
    if (one_round) {
      const int h = tid / d, e = tid - h * d;
      const bool have = tid < group * d;
      // this split's own (M, L, O) of element (h, e) from the warps
      float M = -INFINITY, L = 0.f, O = 0.f;
      if (have) {
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, wm[w * group + h]);
        for (int w = 0; w < kAttnWarps; ++w) {
          const float f = expf(wm[w * group + h] - M);
          L += wl[w * group + h] * f;
          O += wo[(w * group + h) * d + e] * f;
        }
      }
      const int nml = 2 * (nsplit - 1) * group;
      float ov[kAttnMergeOne], mlv;
      io.template poll_merge<kAttnMergeOne>(static_cast<size_t>(g) * a.nsplit_max * group * (d + 2), nsplit, group,
                                           have ? h : 0, have ? e : 0, d, tid < nml ? tid : -1, ov, &mlv);
      float* sml = qn;  // [split - 1][head][M, L]
      if (tid < nml) sml[tid] = mlv;
      sync();
      if (have) {
        float Mx = M;
        for (int k = 1; k < nsplit; ++k) Mx = fmaxf(Mx, sml[((k - 1) * group + h) * 2]);
        const float f0 = expf(M - Mx);
        float Lx = L * f0, Ox = O * f0;
#pragma unroll
        for (int j = 0; j < kAttnMergeOne; ++j) {
          if (j + 1 >= nsplit) break;
          const float f = expf(sml[(j * group + h) * 2] - Mx);
          Lx = fmaf(sml[(j * group + h) * 2 + 1], f, Lx);
          Ox = fmaf(ov[j], f, Ox);
        }
        io.store_out((g * group + h) * d + e, Ox / Lx);
      }
    }
  }
  for (int idx = one_round ? group * d : tid; idx < group * d; idx += NT) {
    const int h = idx / d, e = idx - h * d;
    float M = -INFINITY;
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, wm[w * group + h]);
    float L = 0.f, O = 0.f;
    for (int w = 0; w < kAttnWarps; ++w) {
      const float f = expf(wm[w * group + h] - M);
      L += wl[w * group + h] * f;
      O += wo[(w * group + h) * d + e] * f;
    }
    const size_t pbase = ((static_cast<size_t>(g) * a.nsplit_max) * group + h) * (d + 2);  // split 0 of (g, h)
    const size_t pstride = static_cast<size_t>(group) * (d + 2);                       // next split
    if (nsplit == 1) {
      io.store_out((g * group + h) * d + e, O / L);
    } else if constexpr (Io::kPolledMerge) {
      if (!merger) {
        // (O, M, L) of this split as exchange words; split 0 merges them
        const size_t pb = pbase + s * pstride;
        io.store_part(pb + e, O);
        if (e == 0) {
          io.store_part(pb + d, M);
          io.store_part(pb + d + 1, L);
        }
      } else {
        // split 0: fold in the other splits in order, eight at a time (their
        // words requested together, then polled; sixteen at a time spills)
        constexpr int KC = 8;
        for (int k0 = 1; k0 < nsplit; k0 += KC) {
          float ov[KC], mv[KC], lv[KC];
          io.template poll_parts<KC>(pbase + k0 * pstride, pstride, min(KC, nsplit - k0), e, d, ov, mv, lv);
#pragma unroll
          for (int k = 0; k < KC; ++k) {
            if (k0 + k >= nsplit) break;
            const float Mn = fmaxf(M, mv[k]);
            const float fa = expf(M - Mn), fb = expf(mv[k] - Mn);
            L = L * fa + lv[k] * fb;
            O = O * fa + ov[k] * fb;
            M = Mn;
          }
        }
        io.store_out((g * group + h) * d + e, O / L);
      }
    } else {
      float* p = a.part + pbase + s * pstride;
      p[e] = O;
      if (e == 0) {
        p[d] = M;
        p[d + 1] = L;
      }
    }
  }
  // The appended row was written before the barrier above.
  if (tid == NT - 1 && t1 == n) io.publish_kv(g, pos);
  if (nsplit == 1 || Io::kPolledMerge) return;

  // Split merge: the last CTA of this key/value head to finish combines all splits.
  __threadfence();
  sync();
  if (tid == 0) *s_last = (atomicAdd(a.counter + g, 1u) == static_cast<uint32_t>(nsplit - 1));
  sync();
  if (!*s_last) return;
  __threadfence();
  for (int idx = tid; idx < group * d; idx += NT) {
    const int h = idx / d, e = idx - h * d;
    float M = -INFINITY;
    for (int k = 0; k < nsplit; ++k) {
      const float* p = a.part + ((static_cast<size_t>(g) * a.nsplit_max + k) * group + h) * (d + 2);
      M = fmaxf(M, __ldcg(p + d));
    }
    float L = 0.f, O = 0.f;
    for (int k = 0; k < nsplit; ++k) {
      const float* p = a.part + ((static_cast<size_t>(g) * a.nsplit_max + k) * group + h) * (d + 2);
      const float f = expf(__ldcg(p + d) - M);
      L += __ldcg(p + d + 1) * f;
      O += __ldcg(p + e) * f;
    }
    io.store_out((g * group + h) * d + e, O / L);
  }
  if (tid == 0) a.counter[g] = 0u;
}

template <typename KT, int GMAX>
__global__ void __launch_bounds__(kAttnWarps * 32) attn_decode_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) float asmem[];
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();
  const int pos = a.ctrl[0] + a.pos_add;
  if (pos < 0 || pos >= a.max_seq) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(a.err, ERR_BAD_POSITION);
    return;
  }
  if (threadIdx.x == 0) {  // this CTA's cached rows (before pos) into L2 at once
    int t0, t1, ns;
    if (attn_split_range(a, blockIdx.y, pos, &t0, &t1, &ns) && min(t1, pos) > t0) {
      const size_t rb = static_cast<size_t>(a.d) * sizeof(KT);
      const size_t off = (static_cast<size_t>(blockIdx.x) * a.max_seq + t0) * rb;
      const uint32_t bytes = static_cast<uint32_t>((min(t1, pos) - t0) * rb);
      bulk_prefetch_l2(static_cast<const char*>(a.kc) + off, bytes);
      bulk_prefetch_l2(static_cast<const char*>(a.vc) + off, bytes);
    }
  }
  attn_decode_body<KT, GMAX, kAttnWarps * 32, CtaSync, GMAX <= 2 ? kAttnChunk<KT> : kAttnChunk<KT> / 2>(a, blockIdx.x, blockIdx.y, pos, asmem, threadIdx.x, CtaSync{}, &s_last,
                                              AttnPlainIo{a.qkv, a.out});
}

}  // namespace wsg
