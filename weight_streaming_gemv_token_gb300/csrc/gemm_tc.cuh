// Tensor-core GEMM for the chunked-prefill projections ("Megakernels",
// "Chunked prefill for long prompts": the chunk's rows turn every projection
// into a dense matrix product): C[M][N] (float32) = A[M][K] . W[N][K]^T, or
// C += that product, with A (activation rows) and W (weights, row-major
// [out][in]) in bfloat16 and FP32 accumulation.
//
// Tiles of C are 128 x 256, 128 x 128 or 128 x 64, computed with tcgen05.mma
// (cta_group::1, kind::f16, BF16 inputs, FP32 accumulator in tensor memory);
// one launch may cover up to three weight matrices side by side in N (Q, K
// and V, or gate and up). The kernel is persistent: one CTA per SM walks the
// tiles blockIdx.x, blockIdx.x + gridDim.x, ...
//  * warp 0: a TMA thread streams 128 x 64 tiles of A and W (128-byte swizzle)
//    of every K block of every tile into a 3- or 4-stage shared-memory ring
//    (full mbarrier per stage, completed by the copies' transaction bytes);
//  * warp 1: an MMA thread issues four K = 16 MMAs per stage from shared-
//    memory descriptors into one of two accumulator buffers in tensor memory
//    (alternating by tile), releases each stage with tcgen05.commit on its
//    empty mbarrier and, after a tile's last stage, commits the buffer full;
//  * warps 2-5: each reads its quarter of the accumulator lanes (32 rows) with
//    tcgen05.ld, stores (or adds, or SwiGLUs) the rows and marks the buffer
//    empty, while the MMA thread already fills the other buffer with the next
//    tile: a tile's epilogue overlaps the next tile's main loop.
// TC_SWIGLU (128- or 256-column tiles): tile j takes rows BN/2 j .. BN/2 j +
// BN/2 - 1 of the gate weights (mapB0, BN/2-row boxes) and the same rows of
// the up weights (mapB1) as one W tile, so accumulator columns 0..BN/2-1 hold
// gate and BN/2..BN-1 up of the same BN/2 outputs; the epilogue writes
// silu(gate) * up for them as a bfloat16 value + remainder pair (the next
// GEMM's activation operand), and the gate/up product never goes to memory.
// With SPLIT the activation operand comes as two bfloat16 matrices, A = hi +
// lo (hi the nearest bfloat16 of a float32 value, lo the nearest bfloat16 of
// the remainder), and both products go into the same accumulator: the rows
// keep about 16 mantissa bits, so the product matches float32 activations
// times bfloat16 weights to ~2^-17 relative per term.
// Rows of A past M and columns of K past K read as zeros (the tensor maps'
// bounds), so any M, N and K (K % 8 == 0) work. Every wait is bounded; on a
// timeout the CTA records an error bit, skips the accumulator read, frees its
// tensor memory and returns.
#pragma once
#include <cuda.h>

#include <cstdint>

#include "gemv_stream.cuh"  // silu_f32
#include "ptx.cuh"

namespace wsg {

// Tiles of C are kTcBM x BN, BN = 256 (kTcBN), 128 or 64 (for grids that
// would not fill the GPU with wider tiles).
// Warps: 0 TMA, 1 MMA (and tensor-memory allocation), 2-5 epilogue.
constexpr int kTcBM = 128, kTcBN = 256, kTcBK = 64, kTcEpiWarps = 4, kTcThreads = 32 * (2 + kTcEpiWarps);
constexpr uint32_t kTcABytes = kTcBM * kTcBK * 2;  // 16 KB
template <int BN>
constexpr uint32_t tc_b_bytes() {
  return BN * kTcBK * 2;
}
// stage: A tile (and with SPLIT the A-remainder tile), then the W tile
template <bool SPLIT, int BN>
constexpr uint32_t tc_stage_bytes() {
  return (SPLIT ? 2 : 1) * kTcABytes + tc_b_bytes<BN>();
}
// four stages where they fit in 200 KB, else three
template <bool SPLIT, int BN>
constexpr int tc_stages() {
  return 4 * tc_stage_bytes<SPLIT, BN>() <= 200u * 1024u ? 4 : 3;
}
template <bool SPLIT, int BN>
constexpr size_t tc_smem_bytes() {
  return tc_stages<SPLIT, BN>() * tc_stage_bytes<SPLIT, BN>() + 1024;  // plus alignment slack
}

enum : uint32_t { ERR_TC_TIMEOUT = 1u << 5 };

// Epilogues: store C, add into C, or (TC_SWIGLU) the gate/up product's
// SwiGLU written as bfloat16 value + remainder (see the kernel).
enum TcEpi : int { TC_STORE = 0, TC_ADD = 1, TC_SWIGLU = 2 };

struct TcArgs {
  float* C;
  int32_t ldc;   // row stride of C in elements
  int32_t col0;  // column of C where this product's column 0 goes
  int32_t M, N, K;
  // Up to three weight matrices side by side in N: columns [0, nb1) come from
  // mapB0, [nb1, nb2) from mapB1, [nb2, N) from mapB2 (nb1, nb2 multiples of
  // the tile width, so no tile straddles two of them).
  int32_t nb1, nb2;
  // TC_SWIGLU: act / act2 [M][ld_act] receive the value and remainder of silu(gate) * up
  uint16_t* act;
  uint16_t* act2;
  int32_t ld_act;
  uint32_t* err;
};

// Shared-memory matrix descriptor of a K-major tile with 128-byte swizzle:
// rows of 128 bytes, 8-row groups 1024 bytes apart, descriptor version 1.
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;            // leading byte offset (unused with this swizzle)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;    // stride byte offset: one 8-row group
  d |= static_cast<uint64_t>(1) << 46;            // descriptor version
  d |= static_cast<uint64_t>(2) << 61;            // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: FP32 accumulator, BF16 A and B, both
// K-major, N and M as encoded by the instruction (N >> 3, M >> 4).
constexpr uint32_t tc_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d_map(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 32 consecutive accumulator columns of this warp's 32 lanes (one register each).
__device__ __forceinline__ void tc_ld32(uint32_t (&v)[32], uint32_t taddr) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

// Epilogue of one tile for one warp: its 32 rows (TMEM lanes at tbase), every
// column of the tile; `row` is this lane's row of C.
template <int EPI, int BN>
__device__ __forceinline__ void tc_epilogue(const TcArgs& a, uint32_t tbase, int row, int n0) {
  if constexpr (EPI == TC_SWIGLU) {
    {
      const int half = a.N / 2;  // outputs of the whole product
#pragma unroll 1
      for (int c0 = 0; c0 < BN / 2; c0 += 32) {
        uint32_t gv[32], uv[32];
        const uint32_t taddr = tbase + static_cast<uint32_t>(c0);
        tc_ld32(gv, taddr);
        tc_ld32(uv, taddr + BN / 2);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const int col0 = n0 / 2 + c0;
        if (row < a.M) {
          uint16_t* h = a.act + static_cast<size_t>(row) * a.ld_act + col0;
          uint16_t* l = a.act2 + static_cast<size_t>(row) * a.ld_act + col0;
          uint32_t hp[16], lp[16];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float v = silu_f32(__uint_as_float(gv[j])) * __uint_as_float(uv[j]);
            const uint16_t hb = f32_to_bf16_rn(v), lb = f32_to_bf16_rn(v - bf16_to_f32(hb));
            if (j & 1) {
              hp[j >> 1] |= static_cast<uint32_t>(hb) << 16;
              lp[j >> 1] |= static_cast<uint32_t>(lb) << 16;
            } else {
              hp[j >> 1] = hb;
              lp[j >> 1] = lb;
            }
          }
          if (col0 + 32 <= half && ((reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(l)) & 15u) == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              reinterpret_cast<uint4*>(h)[q] = make_uint4(hp[4 * q], hp[4 * q + 1], hp[4 * q + 2], hp[4 * q + 3]);
              reinterpret_cast<uint4*>(l)[q] = make_uint4(lp[4 * q], lp[4 * q + 1], lp[4 * q + 2], lp[4 * q + 3]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (col0 + j < half) {
                h[j] = static_cast<uint16_t>(hp[j >> 1] >> (16 * (j & 1)));
                l[j] = static_cast<uint16_t>(lp[j >> 1] >> (16 * (j & 1)));
              }
          }
        }
      }
    }
  } else {
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      uint32_t v[32];
      const uint32_t taddr = tbase + static_cast<uint32_t>(c0);
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
          "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
          : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
            "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
            "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
            "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
          : "r"(taddr));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      if (row < a.M) {
        float* crow = a.C + static_cast<size_t>(row) * a.ldc + a.col0;
        const int nb = n0 + c0;
        if (nb + 32 <= a.N && ((reinterpret_cast<uintptr_t>(crow + nb) & 15u) == 0)) {
          // the row's 32 columns in 16-byte pieces
          float4* c4 = reinterpret_cast<float4*>(crow + nb);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float4 x = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                   __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
            if (EPI == TC_ADD) {
              const float4 y = c4[j];
              x.x += y.x;
              x.y += y.y;
              x.z += y.z;
              x.w += y.w;
            }
            c4[j] = x;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = nb + j;
            if (col < a.N) {
              const float x = __uint_as_float(v[j]);
              if (EPI == TC_ADD)
                crow[col] += x;
              else
                crow[col] = x;
            }
          }
        }
      }
    }
  }
}

template <int EPI, bool SPLIT, int BN>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapA2,
                        const __grid_constant__ CUtensorMap mapB0, const __grid_constant__ CUtensorMap mapB1,
                        const __grid_constant__ CUtensorMap mapB2, const TcArgs a) {
  static_assert(BN == 64 || BN == 128 || BN == 256, "64-, 128- or 256-column tiles");
  static_assert(EPI != TC_SWIGLU || BN >= 128, "the SwiGLU epilogue pairs BN/2 gate and BN/2 up columns");
  constexpr int kTcStages = tc_stages<SPLIT, BN>();
  constexpr uint32_t kStage = tc_stage_bytes<SPLIT, BN>();
  constexpr uint32_t kBOff = (SPLIT ? 2 : 1) * kTcABytes;  // W tile offset within a stage
  constexpr uint32_t kTmemCols = 2 * BN;                   // two FP32 accumulators of 128 lanes x BN columns
  extern __shared__ __align__(1024) unsigned char tc_raw[];
  unsigned char* tsm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kTcStages], empty[kTcStages], tfull[2], tempty[2], drain;
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntn = (a.N + BN - 1) / BN, ntiles = ntn * ((a.M + kTcBM - 1) / kTcBM);
  const int KB = (a.K + kTcBK - 1) / kTcBK;
  volatile int* vfail = &s_fail;

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kTcEpiWarps);
    }
    mbar_init(&drain, 1);
    s_fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();  // the next launch may start its own set-up and weight loads
  const uint32_t tmem = tmem_base;
  auto fail = [&]() {
    *vfail = 1;
    atomicOr(a.err, ERR_TC_TIMEOUT);
  };

  if (warp == 0) {
    // ---- TMA: A and W tiles of every K block of every tile into the stage ring ----
    // The weights never depend on earlier kernels: the first ring's worth of
    // W tiles is requested before waiting for the kernel this launch follows
    // (programmatic dependent launch), the activation tiles after it.
    if (lane == 0) {
      auto tile_of = [&](int t, int* n0, int* m0, const CUtensorMap** mapB, int* wn0) {
        *n0 = (t % ntn) * BN;
        *m0 = (t / ntn) * kTcBM;
        *mapB = *n0 < a.nb1 ? &mapB0 : *n0 < a.nb2 ? &mapB1 : &mapB2;
        *wn0 = *n0 - (*n0 < a.nb1 ? 0 : *n0 < a.nb2 ? a.nb1 : a.nb2);  // first row of the tile in its weight
      };
      auto load_w = [&](unsigned char* st, int kb, int n0, const CUtensorMap* mapB, int wn0, uint64_t* bar) {
        if constexpr (EPI == TC_SWIGLU) {
          tma_load_2d_map(st + kBOff, &mapB0, kb * kTcBK, n0 / 2, bar);
          tma_load_2d_map(st + kBOff + tc_b_bytes<BN / 2>(), &mapB1, kb * kTcBK, n0 / 2, bar);
        } else {
          tma_load_2d_map(st + kBOff, mapB, kb * kTcBK, wn0, bar);
        }
      };
      uint32_t pre = 0;  // stages whose W tiles went out before the wait
      for (int t = blockIdx.x; t < ntiles && pre < static_cast<uint32_t>(kTcStages); t += gridDim.x) {
        int n0, m0, wn0;
        const CUtensorMap* mapB;
        tile_of(t, &n0, &m0, &mapB, &wn0);
        for (int kb = 0; kb < KB && pre < static_cast<uint32_t>(kTcStages); ++kb, ++pre) {
          mbar_arrive_expect_tx(&full[pre], kStage);
          load_w(tsm + static_cast<size_t>(pre) * kStage, kb, n0, mapB, wn0, &full[pre]);
        }
      }
      pdl_wait();
      uint32_t gk = 0;  // k blocks issued by this CTA (ring position)
      for (int t = blockIdx.x; t < ntiles && !*vfail; t += gridDim.x) {
        int n0, m0, wn0;
        const CUtensorMap* mapB;
        tile_of(t, &n0, &m0, &mapB, &wn0);
        for (int kb = 0; kb < KB; ++kb, ++gk) {
          const int s = gk % kTcStages;
          if (gk >= kTcStages && !mbar_wait(&empty[s], ((gk / kTcStages) - 1) & 1)) {
            fail();
            break;
          }
          if (*vfail) break;
          unsigned char* st = tsm + static_cast<size_t>(s) * kStage;
          if (gk >= pre) {
            mbar_arrive_expect_tx(&full[s], kStage);
            load_w(st, kb, n0, mapB, wn0, &full[s]);
          }
          tma_load_2d_map(st, &mapA, kb * kTcBK, m0, &full[s]);
          if (SPLIT) tma_load_2d_map(st + kTcABytes, &mapA2, kb * kTcBK, m0, &full[s]);
        }
      }
      // a stage whose W tile went out ahead must not be left pending at exit
      for (uint32_t k = gk; k < pre; ++k) mbar_wait(&full[k], 0);
    } else {
      pdl_wait();
    }
  } else if (warp == 1) {
    // ---- MMA: four K = 16 steps per stage into the tile's accumulator buffer ----
    if (lane == 0) {
      constexpr uint32_t idesc = tc_idesc(kTcBM, BN);
      uint32_t gk = 0;
      int li = 0;  // tiles of this CTA so far
      for (int t = blockIdx.x; t < ntiles && !*vfail; t += gridDim.x, ++li) {
        const int b = li & 1;
        // the epilogue has drained this buffer (its tile two back)
        if (li >= 2 && !mbar_wait(&tempty[b], ((li >> 1) - 1) & 1)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++gk) {
          const int s = gk % kTcStages;
          if (!mbar_wait(&full[s], (gk / kTcStages) & 1)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(tsm + static_cast<size_t>(s) * kStage);
          const uint32_t sb = sa + kBOff;
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk) {
            const uint64_t db = tc_desc_sw128(sb + kk * 32);
#pragma unroll
            for (int part = 0; part < (SPLIT ? 2 : 1); ++part) {
              const uint64_t da = tc_desc_sw128(sa + part * kTcABytes + kk * 32);
              const uint32_t acc = (kb | kk | part) != 0;
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                  "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                  "l"(da), "l"(db), "r"(idesc), "r"(acc)
                  : "memory");
            }
          }
          // the stage's shared memory is free once these MMAs have read it
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                           smem_u32(&empty[s]))
                       : "memory");
        }
        if (!ok) break;
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(&tfull[b]))
                     : "memory");
      }
      // every MMA this thread issued has completed before tensor memory is freed
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                       smem_u32(&drain))
                   : "memory");
      if (!mbar_wait(&drain, 0)) fail();
    }
  } else {
    // ---- epilogue warps: warp w reads TMEM lanes (rows) 32 (w % 4) .. 32 (w % 4) + 31 ----
    pdl_wait();  // C (and the SwiGLU output) may be read or written by the kernel before
    const int q = warp & 3;
    int li = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++li) {
      const int b = li & 1;
      const bool have = mbar_wait(&tfull[b], (li >> 1) & 1);
      if (!__all_sync(0xffffffffu, have)) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const int n0 = (t % ntn) * BN, m0 = (t / ntn) * kTcBM;
      const int row = m0 + q * 32 + lane;
      const uint32_t tbase = tmem + static_cast<uint32_t>(b * BN) + (static_cast<uint32_t>(q * 32) << 16);
      tc_epilogue<EPI, BN>(a, tbase, row, n0);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
}

}  // namespace wsg
