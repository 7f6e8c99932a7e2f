// Causal attention of a prefill chunk on the 5th-generation tensor cores
// ("Megakernels", "Chunked prefill for long prompts": the chunk's rows attend
// to the cache, earlier chunks and the chunk itself up to each row's own
// position). Bfloat16 cache, head size 128.
//
// A CTA owns 128 query vectors of one key/value head g: the group's query
// heads of 128 / group consecutive chunk rows (vector v = row * group + head),
// one per tensor-memory lane, and walks the key tiles of 128 positions from 0
// up to the last position any of its rows sees (flash-attention form). Q and
// the probabilities P stay in tensor memory and enter the products as the A
// operand from there; shared memory holds only key and value tiles, so each
// MMA reads one 4 KB operand slice from shared memory:
//
//   warp 0      one thread streams each tile's keys and values (two 128 x 64
//               boxes each, 128-byte swizzle) from the whole-cache tensor maps
//               into 3-stage key and value rings;
//   warp 1      one thread issues S_j = Q K_j^T (M 128, N 128, into one of two
//               score buffers in tensor memory) one tile ahead, then, once the
//               probabilities of tile j have replaced its scores in that
//               buffer, O += P_j V_j (M 128, N 128; the value tile is read in
//               its stored, value-contiguous layout as an MN-major operand);
//   warps 2-9   two threads per vector, each on half of the tile's keys
//               (warps w and w + 4 share the tensor-memory lanes of w % 4):
//               read 64 scores (tcgen05.ld), mask keys past the vector's
//               position, exchange the half maxima, exponentiate against a
//               reference maximum, add to a running half sum and write the
//               half probability row over the scores (tcgen05.st).
//
// The running maximum is a reference that moves only when a tile's maximum
// passes it by more than 2^8: probabilities stay below 256, and the rare move
// rescales the output accumulator in tensor memory (read, scale, write back)
// after the previous P V product has completed. O / sum is exact in any
// reference, so the result is the softmax-weighted sum of the values.
//
// Precision: Q (float32) and P enter the products as bfloat16 value +
// remainder pairs (two MMAs into the same accumulator), keys and values are
// the cache's bfloat16, accumulation is FP32: scores and outputs keep about 16
// mantissa bits, as in the single-token path's float32 attention. The output
// is written as a bfloat16 value + remainder pair, the O projection's operand.
//
// Tensor memory (512 columns, one CTA per SM): score / probability buffers at
// columns 0 and 128 (probabilities: value at +0..63, remainder at +64..127,
// two bfloat16 per column), O at 256, Q value at 384 and remainder at 448.
//
// Launched as a programmatic dependent of the previous kernel (RoPE and the
// cache append of this chunk's rows): barrier and tensor-memory set-up run
// before the dependency wait, everything that reads Q or the cache after it.
//
// Every wait is bounded; on a timeout the CTA records ERR_TC_TIMEOUT, stops,
// waits for its issued MMAs and frees its tensor memory.
#pragma once
#include <cuda.h>

#include <cstdint>

#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace wsg {

constexpr int kAtD = 128;                                // head size
constexpr int kAtBM = 128;                               // query vectors per CTA (tensor-memory lanes)
constexpr int kAtBN = 128;                               // keys per tile
constexpr int kAtKStages = 3, kAtVStages = 3;            // key / value tiles in flight
constexpr int kAtSoftWarps = 8;                          // two per lane quarter of tensor memory
constexpr int kAtThreads = 32 * (2 + kAtSoftWarps);      // TMA warp, MMA warp, softmax warps
constexpr uint32_t kAtKBytes = kAtBN * kAtD * 2;         // a key (or value) tile: 32 KB, two 64-column boxes
constexpr uint32_t kAtBoxBytes = kAtKBytes / 2;          // 128 keys x 64 columns
constexpr uint32_t kAtTmemCols = 512;                    // S / P buffers at 0 and 128, O at 256, Q at 384
constexpr uint32_t kAtTmO = 256, kAtTmQ = 384;
constexpr float kAtRescaleLog2 = 8.f;                    // reference moves past this margin (log2 units)
constexpr size_t kAtSmem = (kAtKStages + kAtVStages) * kAtKBytes + 1024;

struct PfAttnArgs {
  const float* qkv;  // [n][(n_q + 2 n_kv) D] chunk rows: Q after its norm and RoPE, then K, V
  uint16_t* AO;      // [n][n_q D] attention output, bfloat16 value
  uint16_t* AO2;     // ... and remainder
  uint32_t* err;
  int n, p0;         // chunk rows, position of row 0
  int n_q, n_kv;
  int kv_row0;       // row of (this layer, head 0, position 0) in the cache tensor maps
  int max_seq;       // cache rows per head
  float scale_log2;  // softmax scale (1 / sqrt(D)) times log2(e)
};

// Shared-memory descriptor of an MN-major operand with 128-byte swizzle:
// 64 contiguous MN elements per 128-byte row, rows along K; lbo = bytes
// between 64-element groups along MN, sbo = bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t tc_desc_sw128_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// D (+)= A B with A (M x 16, two bfloat16 per column, lane = row) in tensor
// memory at a_tmem and B from the shared-memory descriptor db; kind::f16,
// FP32 accumulator at tensor-memory address d (accumulate when acc != 0).
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d, uint32_t a_tmem, uint64_t db, uint32_t idesc,
                                              uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(db), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive columns of this warp's 32 lanes from registers (one each).
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Two floats as packed bfloat16 value and remainder pairs (low half: x),
// each rounded to nearest even by the conversion instruction.
__device__ __forceinline__ void at_pack_split(float x, float y, uint32_t* hi, uint32_t* lo) {
  uint32_t h, l;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(y), "f"(x));
  const float rx = x - __uint_as_float(h << 16), ry = y - __uint_as_float(h & 0xFFFF0000u);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(l) : "f"(ry), "f"(rx));
  *hi = h;
  *lo = l;
}

// 2^x (ex2.approx: a few ulp; results below 2^-126 flush to zero, -inf gives 0).
__device__ __forceinline__ float at_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Grid: (n_kv, ceil(n / (128 / group))), kAtThreads threads, kAtSmem bytes of
// dynamic shared memory. kmap / vmap: the whole K / V cache as a 2D bfloat16
// tensor [layers * n_kv * max_seq][128] in 128-row x 64-column boxes with
// 128-byte swizzle.
__global__ void __launch_bounds__(kAtThreads, 1)
    pf_attn_tmem_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const PfAttnArgs a) {
  extern __shared__ __align__(1024) unsigned char at_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(at_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* Ks = sm;                                   // key stages: box 0 (columns 0-63), box 1
  unsigned char* Vs = Ks + kAtKStages * kAtKBytes;          // value stages, the same
  __shared__ __align__(8) uint64_t k_full[kAtKStages], k_empty[kAtKStages], v_full[kAtVStages], v_empty[kAtVStages];
  // o_done[b]: completions of the P V products of tiles j = b, b + 2, ...; a
  // parity wait on a barrier is only sound while the completion before the one
  // awaited has happened, which for the product of tile j means that of tile
  // j - 2 (done once S_j, issued after it, is)
  __shared__ __align__(8) uint64_t s_full[2], p_full[2], o_done[2], drain;
  __shared__ __align__(8) uint64_t pair_bar[4];  // the two softmax warps of a lane quarter
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  __shared__ float xch[2][2][kAtBM];  // softmax: [exchange parity][half][vector] half maxima, then half sums
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x;
  const int group = a.n_q / a.n_kv, rows = kAtBM / group;
  const int r0 = (gridDim.y - 1 - blockIdx.y) * rows;  // the blocks with the most keys start first
  const int last_row = min(a.n, r0 + rows) - 1;
  const int T = (a.p0 + last_row) / kAtBN + 1;           // key tiles this CTA walks
  volatile int* vfail = &s_fail;

  if (tid == 0) {
    for (int s = 0; s < kAtKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kAtVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], kAtSoftWarps);
      mbar_init(&o_done[b], 1);
    }
    mbar_init(&drain, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&pair_bar[i], 64);
    s_fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "n"(kAtTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();
  pdl_wait();  // Q and this chunk's cache rows come from the previous kernels
  const uint32_t tmem = tmem_base;
  const int q = warp & 3, half = (warp - 2) >> 2;  // softmax warps: lane quarter, half of the keys / of D
  const int v = q * 32 + lane;
  const int row = r0 + v / group;
  const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);  // this warp's lanes
  if (warp >= 2) {
    // Q row v as bfloat16 value and remainder into tensor memory: this thread
    // converts elements 64 half .. 64 half + 63 (32 columns of each part)
    uint32_t qh[32], ql[32];
    if (row < a.n) {
      const int W = (a.n_q + 2 * a.n_kv) * kAtD;
      const float4* src = reinterpret_cast<const float4*>(a.qkv + static_cast<size_t>(row) * W +
                                                          (g * group + v % group) * kAtD + half * (kAtD / 2));
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float4 x = src[k];
        at_pack_split(x.x, x.y, &qh[2 * k], &ql[2 * k]);
        at_pack_split(x.z, x.w, &qh[2 * k + 1], &ql[2 * k + 1]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) qh[k] = ql[k] = 0u;
    }
    tc_st32(tl + kAtTmQ + half * 32, qh);
    tc_st32(tl + kAtTmQ + 64 + half * 32, ql);
    tc_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  auto fail = [&]() {
    *vfail = 1;
    atomicOr(a.err, ERR_TC_TIMEOUT);
  };

  if (warp == 0) {
    // ---- TMA: keys and values of tile j into stage j % 3 of their rings ----
    if (lane == 0) {
      const int y0 = a.kv_row0 + g * a.max_seq;
      for (int j = 0; j < T && !*vfail; ++j) {
        const int y = y0 + j * kAtBN;
        const int sk = j % kAtKStages, sv = j % kAtVStages;
        if (j >= kAtKStages && !mbar_wait(&k_empty[sk], ((j / kAtKStages) - 1) & 1)) {
          fail();
          break;
        }
        unsigned char* kd = Ks + static_cast<size_t>(sk) * kAtKBytes;
        mbar_arrive_expect_tx(&k_full[sk], kAtKBytes);
        tma_load_2d_map(kd, &kmap, 0, y, &k_full[sk]);
        tma_load_2d_map(kd + kAtBoxBytes, &kmap, 64, y, &k_full[sk]);
        if (j >= kAtVStages && !mbar_wait(&v_empty[sv], ((j / kAtVStages) - 1) & 1)) {
          fail();
          break;
        }
        unsigned char* vd = Vs + static_cast<size_t>(sv) * kAtKBytes;
        mbar_arrive_expect_tx(&v_full[sv], kAtKBytes);
        tma_load_2d_map(vd, &vmap, 0, y, &v_full[sv]);
        tma_load_2d_map(vd + kAtBoxBytes, &vmap, 64, y, &v_full[sv]);
      }
    }
  } else if (warp == 1) {
    // ---- MMA: S one tile ahead of P V ----
    if (lane == 0) {
      constexpr uint32_t idS = tc_idesc(kAtBM, kAtBN);
      constexpr uint32_t idO = tc_idesc(kAtBM, kAtD) | (1u << 16);  // B (values) MN-major
      auto issue_s = [&](int j) -> bool {
        const int s = j % kAtKStages;
        if (!mbar_wait(&k_full[s], (j / kAtKStages) & 1)) return false;
        tc_fence_after();
        const uint32_t kb = smem_u32(Ks + static_cast<size_t>(s) * kAtKBytes);
        const uint32_t d = tmem + static_cast<uint32_t>((j & 1) * kAtBN);
#pragma unroll
        for (int kk = 0; kk < kAtD / 16; ++kk) {
          const uint64_t db = tc_desc_sw128(kb + (kk >> 2) * kAtBoxBytes + (kk & 3) * 32);
#pragma unroll
          for (int part = 0; part < 2; ++part)
            tc_mma_f16_ts(d, tmem + kAtTmQ + part * 64 + kk * 8, db, idS, (kk | part) != 0);
        }
        tc_commit(&k_empty[s]);  // the key stage is free once these MMAs have read it
        tc_commit(&s_full[j & 1]);
        return true;
      };
      bool ok = issue_s(0);
      for (int j = 0; ok && j < T; ++j) {
        // S_{j+1} goes into the buffer of P_{j-1}: issued after P_{j-1} V_{j-1},
        // it overwrites those probabilities only once that product has read them
        if (j + 1 < T && !issue_s(j + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1)) {
          ok = false;
          break;
        }
        const int s = j % kAtVStages;
        if (!mbar_wait(&v_full[s], (j / kAtVStages) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t vb = smem_u32(Vs + static_cast<size_t>(s) * kAtKBytes);
        const uint32_t pb = tmem + static_cast<uint32_t>((j & 1) * kAtBN);
#pragma unroll
        for (int kk = 0; kk < kAtBN / 16; ++kk) {
          // keys 16 kk .. 16 kk + 15: two 8-row groups 1024 bytes apart; value
          // columns 64 .. 127 in the second box
          const uint64_t db = tc_desc_sw128_mn(vb + kk * 2048, kAtBoxBytes, 1024);
#pragma unroll
          for (int part = 0; part < 2; ++part)
            tc_mma_f16_ts(tmem + kAtTmO, pb + part * 64 + kk * 8, db, idO, (j | kk | part) != 0);
        }
        tc_commit(&v_empty[s]);  // the value stage is free once these MMAs have read it
        tc_commit(&o_done[j & 1]);  // O holds tiles 0..j
      }
      if (!ok) fail();
      // every MMA this thread issued has completed before tensor memory is freed
      tc_commit(&drain);
      if (!mbar_wait(&drain, 0)) fail();
    }
  } else {
    // ---- softmax: two threads per vector (tensor-memory lane), half a tile each ----
    const int pos = a.p0 + min(row, last_row);  // rows past the chunk reuse the last row's keys
    const uint32_t to = tl + kAtTmO + half * (kAtD / 2);  // this thread's half of O
    const float c = a.scale_log2;
    float m_ref = -INFINITY, lsum = 0.f;  // reference (log2 units, shared by the pair), half sum
    bool ok = true;
    // exchange k of the pair: both threads of every vector have written
    // xch[k & 1] (and finished their tensor-memory reads before it)
    auto pair_done = [&](int k) {
      tc_fence_before();
      mbar_arrive(&pair_bar[q]);
      const bool r = __all_sync(0xffffffffu, mbar_wait(&pair_bar[q], k & 1));
      tc_fence_after();
      return r;
    };
    for (int j = 0; j < T; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tb = tl + static_cast<uint32_t>((j & 1) * kAtBN);
      uint32_t s0[32], s1[32];
      tc_ld32(s0, tb + half * 64);
      tc_ld32(s1, tb + half * 64 + 32);
      tc_wait_ld();
      // keys t0 .. t0 + 63 of this half; k <= lim are visible
      const int lim = pos - (j * kAtBN + half * 64);
      float x[64];
      if (__all_sync(0xffffffffu, lim >= 63)) {
#pragma unroll
        for (int k = 0; k < 64; ++k) x[k] = __uint_as_float(k < 32 ? s0[k] : s1[k - 32]);
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k) x[k] = k <= lim ? __uint_as_float(k < 32 ? s0[k] : s1[k - 32]) : -INFINITY;
      }
      float mh[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) mh[k] = fmaxf(x[k], x[k + 32]);
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k) mh[k] = fmaxf(mh[k], mh[k + w]);
      xch[j & 1][half][v] = mh[0];
      if (!pair_done(j)) {
        ok = false;
        break;
      }
      const float mx = fmaxf(mh[0], xch[j & 1][half ^ 1][v]) * c;
      const bool move = mx > m_ref + kAtRescaleLog2;
      if (__any_sync(0xffffffffu, move)) {
        const float nref = move ? mx : m_ref;
        const float f = nref == m_ref ? 1.f : at_exp2(m_ref - nref);  // 0 on the first move
        lsum *= f;
        if (j > 0) {
          // O holds tiles 0..j-1 once P_{j-1} V_{j-1} has completed (P_{j-3}
          // V_{j-3} had, before S_j that this thread has read)
          if (!__all_sync(0xffffffffu, mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < kAtD / 2; c0 += 32) {
            uint32_t o[32];
            tc_ld32(o, to + c0);
            tc_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
            tc_st32(to + c0, o);
          }
        }
        m_ref = nref;
      }
      // probabilities over the scores: value at columns 32 half .., remainder at 64 + 32 half ..
      uint32_t ph[32], pl[32];
      float sh[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float p0 = at_exp2(fmaf(x[2 * k], c, -m_ref)), p1 = at_exp2(fmaf(x[2 * k + 1], c, -m_ref));
        sh[k] = p0 + p1;
        at_pack_split(p0, p1, &ph[k], &pl[k]);
      }
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k) sh[k] += sh[k + w];
      lsum += sh[0];
      tc_st32(tb + half * 32, ph);
      tc_st32(tb + 64 + half * 32, pl);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[j & 1]);
    }
    if (ok && !__all_sync(0xffffffffu, mbar_wait(&o_done[(T - 1) & 1], ((T - 1) >> 1) & 1))) ok = false;
    xch[T & 1][half][v] = lsum;
    if (!pair_done(T)) ok = false;  // (after a failure the pair may be out of step: bounded either way)
    if (ok) {
      tc_fence_after();
      const float inv = 1.0f / (lsum + xch[T & 1][half ^ 1][v]);
      const bool store = row < a.n;
      const size_t at = static_cast<size_t>(row) * a.n_q * kAtD + static_cast<size_t>(g * group + v % group) * kAtD +
                        half * (kAtD / 2);
#pragma unroll 1
      for (int c0 = 0; c0 < kAtD / 2; c0 += 32) {
        uint32_t o[32];
        tc_ld32(o, to + c0);
        tc_wait_ld();
        if (store) {
          uint32_t h[16], l[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            at_pack_split(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv, &h[k], &l[k]);
          uint4* dh = reinterpret_cast<uint4*>(a.AO + at + c0);
          uint4* dl = reinterpret_cast<uint4*>(a.AO2 + at + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            dh[k] = make_uint4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]);
            dl[k] = make_uint4(l[4 * k], l[4 * k + 1], l[4 * k + 2], l[4 * k + 3]);
          }
        }
      }
    }
    if (!ok && lane == 0) fail();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kAtTmemCols) : "memory");
}

}  // namespace wsg
