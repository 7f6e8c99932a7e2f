// Standalone matrix-vector products: gemv (float32 / bfloat16 weights) and
// gemv_q4 (4-bit groupwise-affine weights, one or two tokens).
//
// "Our Kernel Benchmark Was Measuring the System Cache" measures exactly
// these products cold: every call streams a weight matrix that is not in
// cache. gemv uses the bulk-copy streaming engine of gemv_stream.cuh; gemv_q4
// dequantises in registers.
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "common.h"
#include "gemv_bulk.cuh"
#include "gemv_q4.cuh"
#include "gemv_stream.cuh"
#include "gemv_tma.cuh"

namespace wsg {

std::string& thread_error() {
  static thread_local std::string s;
  return s;
}

// Device error word of the context-free entry points (gemv, gemv_q4,
// gemm_bf16, greedy_head_noalloc); gemv_device_errors reads and clears it.
__device__ uint32_t g_gemv_err;

dec_status device_info(DeviceInfo* out, std::string* err) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  WSG_CUDA_TRY(err, cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(err, DEC_EDEVICE, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev].device != dev) {
    cudaDeviceProp p;
    WSG_CUDA_TRY(err, cudaGetDeviceProperties(&p, dev));
    if (p.major != 10 || p.minor != 3)
      return fail(err, DEC_EDEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev, p.major,
                  p.minor);
    void* ew = nullptr;
    WSG_CUDA_TRY(err, cudaGetSymbolAddress(&ew, g_gemv_err));
    cache[dev].sms = p.multiProcessorCount;
    cache[dev].major = p.major;
    cache[dev].minor = p.minor;
    cache[dev].smem_optin = p.sharedMemPerBlockOptin;
    cache[dev].smem_per_sm = p.sharedMemPerMultiprocessor;
    cache[dev].err = static_cast<uint32_t*>(ew);
    cache[dev].device = dev;  // last: marks the entry complete
  }
  *out = cache[dev];
  return DEC_OK;
}

namespace {

constexpr int kNW = 8, kNSMAX = 8, kRING = 12288, kSEGMAX = 4096;
// Matrices up to this size are prefetched into L2 whole at kernel start.
constexpr long long kL2PrefetchMax = 64ll << 20;

// Lift a kernel's dynamic shared memory limit to the device maximum, once per device.
template <typename K>
cudaError_t smem_once(K kern, const DeviceInfo& di, bool* done) {
  if (done[di.device]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(di.smem_optin));
  if (e == cudaSuccess) done[di.device] = true;
  return e;
}

__global__ void fill_zero_kernel(float* y, int n) {
  pdl_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) y[i] = 0.f;
}

// Any-alignment fallback: one warp per row, element loads, float32 accumulation,
// lane partials reduced by a fixed shuffle tree.
template <typename WT, typename XT>
__global__ void gemv_plain_kernel(const WT* __restrict__ W, const XT* __restrict__ x, float* __restrict__ y, int out,
                                  int in) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < out; row += warps) {
    const WT* w = W + static_cast<size_t>(row) * in;
    float acc = 0.f;
    for (int j = lane; j < in; j += 32) acc = fmaf(load_f32<WT>(w, j), load_f32<XT>(x, j), acc);
    acc = warp_sum(acc);
    if (lane == 0) y[row] = acc;
  }
}

// ---- 4-bit groupwise-affine GEMV ----
//
// Lane l of a warp handles 32-column chunks c = l, l+32, ... of R rows at a
// time; one 16-byte load brings a chunk's 32 codes. Each code q becomes the
// float 0.5 + q/256 with one byte permute (exponent byte 0x3F, code in the
// third byte), so S = sum (0.5 + q/256) x = X/2 + (sum q x)/256 over the chunk
// and the chunk's contribution s*sum(q x) + b*X equals 256 s S + (b - 128 s) X,
// with X the chunk's column sum of x (staged once per CTA). A chunk is half of
// a 64-column group, so it has a single (s, b).
//
// Work items of a warp are (row batch, chunk slot) pairs; the codes and scales
// of item i+1 are loaded while item i is computed, and item 0 is loaded before
// the kernel waits on its predecessor (programmatic dependent launch).
template <int R>
struct Q4Item {
  uint4 q[R];
  float s[R], b[R];
};

template <int R>
__device__ __forceinline__ void q4_load(Q4Item<R>& it, const uint32_t* __restrict__ codes, const __half* __restrict__ sc,
                                        const __half* __restrict__ bi, int rb, int c, int out, int nch,
                                        int words_per_row, int groups_per_row) {
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int row = rb + r;
    if (row < out && c < nch) {
      const uint32_t* p = codes + static_cast<size_t>(row) * words_per_row + 4 * c;
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(it.q[r].x), "=r"(it.q[r].y), "=r"(it.q[r].z), "=r"(it.q[r].w)
                   : "l"(p));
      it.s[r] = __half2float(sc[static_cast<size_t>(row) * groups_per_row + (c >> 1)]);
      it.b[r] = __half2float(bi[static_cast<size_t>(row) * groups_per_row + (c >> 1)]);
    } else {
      it.q[r] = make_uint4(0, 0, 0, 0);
      it.s[r] = it.b[r] = 0.f;
    }
  }
}

template <int R, int NTOK>
__global__ void __launch_bounds__(256) gemv_q4_kernel(const uint32_t* __restrict__ codes,
                                                      const __half* __restrict__ sc, const __half* __restrict__ bi,
                                                      const uint16_t* __restrict__ x, float* __restrict__ y, int out,
                                                      int in) {
  extern __shared__ float4 q4_smem[];
  const int nch = in >> 5;
  float4* xs4 = q4_smem;                                         // [NTOK][8][nch]
  float* xsum = reinterpret_cast<float*>(xs4 + NTOK * 8 * nch);  // [NTOK][nch]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int words_per_row = in >> 3, groups_per_row = in >> 6;
  const int cpl = (nch + 31) >> 5;  // chunk slots per lane per row batch
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const int gw = blockIdx.x * (blockDim.x >> 5) + warp;
  const int nbatch = (out + R - 1) / R;
  const int my_batches = gw < nbatch ? (nbatch - gw + warps_total - 1) / warps_total : 0;
  const int nitems = my_batches * cpl;

  Q4Item<R> cur;
  if (nitems > 0) q4_load<R>(cur, codes, sc, bi, gw * R, lane, out, nch, words_per_row, groups_per_row);
  pdl_trigger();
  pdl_wait();
  for (int idx = tid; idx < NTOK * nch * 8; idx += blockDim.x) {
    const int t = idx / (nch * 8), rem = idx - t * nch * 8, c = rem >> 3, k = rem & 7;
    const uint16_t* xp = x + static_cast<size_t>(t) * in + 32 * c + 4 * k;
    xs4[(t * 8 + k) * nch + c] = make_float4(bf16_to_f32(xp[0]), bf16_to_f32(xp[1]), bf16_to_f32(xp[2]),
                                             bf16_to_f32(xp[3]));
  }
  for (int idx = tid; idx < NTOK * nch; idx += blockDim.x) {
    const int t = idx / nch, c = idx - t * nch;
    const uint16_t* xp = x + static_cast<size_t>(t) * in + 32 * c;
    float s = 0.f;
    for (int j = 0; j < 32; ++j) s += bf16_to_f32(xp[j]);
    xsum[t * nch + c] = s;
  }
  __syncthreads();

  float acc[R][NTOK];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int t = 0; t < NTOK; ++t) acc[r][t] = 0.f;

#pragma unroll 1
  for (int i = 0; i < nitems; ++i) {
    const int k = i / cpl, j = i - k * cpl;
    const int rb = (gw + k * warps_total) * R;
    const int c = lane + 32 * j;
    Q4Item<R> nxt;
    if (i + 1 < nitems) {
      const int k2 = (i + 1) / cpl, j2 = (i + 1) - k2 * cpl;
      q4_load<R>(nxt, codes, sc, bi, (gw + k2 * warps_total) * R, lane + 32 * j2, out, nch, words_per_row,
                 groups_per_row);
    }
    if (c < nch) {
#pragma unroll
      for (int t = 0; t < NTOK; ++t) {
        float xv[32];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const float4 v = xs4[(t * 8 + kk) * nch + c];
          xv[4 * kk] = v.x;
          xv[4 * kk + 1] = v.y;
          xv[4 * kk + 2] = v.z;
          xv[4 * kk + 3] = v.w;
        }
        const float X = xsum[t * nch + c];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t wd[4] = {cur.q[r].x, cur.q[r].y, cur.q[r].z, cur.q[r].w};
          float S0 = 0.f, S1 = 0.f;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t lo = wd[m] & 0x0F0F0F0Fu;         // codes 0,2,4,6 of the word
            const uint32_t hi = (wd[m] >> 4) & 0x0F0F0F0Fu;  // codes 1,3,5,7
            S0 = fmaf(__uint_as_float(__byte_perm(lo, 0x3F000000u, 0x7044)), xv[8 * m + 0], S0);
            S1 = fmaf(__uint_as_float(__byte_perm(hi, 0x3F000000u, 0x7044)), xv[8 * m + 1], S1);
            S0 = fmaf(__uint_as_float(__byte_perm(lo, 0x3F000000u, 0x7144)), xv[8 * m + 2], S0);
            S1 = fmaf(__uint_as_float(__byte_perm(hi, 0x3F000000u, 0x7144)), xv[8 * m + 3], S1);
            S0 = fmaf(__uint_as_float(__byte_perm(lo, 0x3F000000u, 0x7244)), xv[8 * m + 4], S0);
            S1 = fmaf(__uint_as_float(__byte_perm(hi, 0x3F000000u, 0x7244)), xv[8 * m + 5], S1);
            S0 = fmaf(__uint_as_float(__byte_perm(lo, 0x3F000000u, 0x7344)), xv[8 * m + 6], S0);
            S1 = fmaf(__uint_as_float(__byte_perm(hi, 0x3F000000u, 0x7344)), xv[8 * m + 7], S1);
          }
          const float S = S0 + S1;
          acc[r][t] = fmaf(256.f * cur.s[r], S, fmaf(cur.b[r] - 128.f * cur.s[r], X, acc[r][t]));
        }
      }
    }
    if (j == cpl - 1) {  // this row batch is complete
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
          const float v = warp_sum(acc[r][t]);
          if (lane == 0 && rb + r < out) y[static_cast<size_t>(t) * out + rb + r] = v;
          acc[r][t] = 0.f;
        }
    }
    if (i + 1 < nitems) cur = nxt;
  }
}

int g_q4_rows[3] = {0, 0, 0};  // rows per warp for ntok = 1, 2 (index by ntok); 0: chosen per launch

template <int R, int NTOK>
dec_status launch_q4_r(const uint32_t* codes, const uint16_t* s, const uint16_t* b, const uint16_t* x, float* y,
                       int out, int in, cudaStream_t st, const DeviceInfo& di) {
  auto kern = gemv_q4_kernel<R, NTOK>;
  const size_t smem = static_cast<size_t>(NTOK) * (in >> 5) * (8 * sizeof(float4) + sizeof(float));
  if (smem > di.smem_optin) return fail(nullptr, DEC_EINVAL, "gemv_q4: in=%d needs %zu B of shared memory", in, smem);
  static bool done[64] = {};
  WSG_CUDA_TRY(nullptr, smem_once(kern, di, done));
  // Resident CTAs per SM, cached per (device, in).
  static int occ_dev[64] = {}, occ_in[64] = {}, occ_val[64] = {};
  int per_sm = 0;
  if (occ_dev[di.device] == di.device + 1 && occ_in[di.device] == in) {
    per_sm = occ_val[di.device];
  } else {
    WSG_CUDA_TRY(nullptr, cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem));
    occ_dev[di.device] = di.device + 1;
    occ_in[di.device] = in;
    occ_val[di.device] = per_sm;
  }
  if (per_sm < 1) per_sm = 1;
  const long long warps_needed = (static_cast<long long>(out) + R - 1) / R;
  long long grid = static_cast<long long>(di.sms) * per_sm;
  const long long grid_needed = (warps_needed + 7) / 8;
  if (grid > grid_needed) grid = grid_needed;
  if (grid < 1) grid = 1;
  WSG_CUDA_TRY(nullptr, launch_k(kern, dim3(static_cast<unsigned>(grid)), dim3(256), smem, st, true, codes,
                                 reinterpret_cast<const __half*>(s), reinterpret_cast<const __half*>(b), x, y, out,
                                 in));
  return DEC_OK;
}

// Bulk-copy 4-bit GEMV (gemv_q4.cuh): one CTA per SM (two when the rows
// give each more than four stages), split between the segments in proportion
// to their rows; a ring of as many stages of 8 R rows as the CTA needs and
// shared memory holds. Needs in % 512 == 0 (every row range's scales are then
// a multiple of 16 bytes) and 16-byte aligned codes, scales, biases and x;
// *used is false when the shape does not fit.
template <int R, int NTOK, int XM, int EPI>
dec_status launch_q4_bulk_r(const Q4Launch& q, cudaStream_t st, const DeviceInfo& di, std::string* err, bool* used) {
  *used = false;
  auto kern = gemv_q4_bulk_kernel<R, NTOK, XM, EPI>;
  static size_t static_smem[64] = {};
  static bool lifted[64] = {};
  if (!lifted[di.device]) {
    cudaFuncAttributes fa{};
    WSG_CUDA_TRY(err, cudaFuncGetAttributes(&fa, kern));
    WSG_CUDA_TRY(err, cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(di.smem_optin - fa.sharedSizeBytes)));
    static_smem[di.device] = fa.sharedSizeBytes;
    lifted[di.device] = true;
  }
  constexpr int RC = kQ4Warps * R;
  long long total = 0;
  for (int k = 0; k < q.nseg; ++k) total += q.seg[k].rows;
  // One CTA per SM while each has at most 4 stages of rows (small matrices:
  // the next launch's CTAs then fit beside them), else two per SM.
  long long G = total < di.sms ? total : di.sms;
  if (total > 4ll * RC * di.sms) G = 2ll * di.sms;
  if (G < q.nseg) G = q.nseg;
  Q4Args a = {};
  a.nseg = q.nseg;
  long long rows_max = 0, c0 = 0;
  for (int k = 0; k < q.nseg; ++k) {
    a.seg[k] = q.seg[k];
    a.seg[k].cta0 = static_cast<int32_t>(c0);
    // CTAs of segment k: its share of G, at least one, leaving one for each later segment
    long long ck = k + 1 == q.nseg ? G - c0 : (G * q.seg[k].rows + total / 2) / total;
    if (ck < 1) ck = 1;
    if (k + 1 < q.nseg && ck > G - c0 - (q.nseg - 1 - k)) ck = G - c0 - (q.nseg - 1 - k);
    if (ck > q.seg[k].rows && q.seg[k].rows > 0) ck = q.seg[k].rows;
    const long long rk = (q.seg[k].rows + ck - 1) / ck;
    if (rk > rows_max) rows_max = rk;
    c0 += ck;
  }
  const int in = q.in;
  const long long nst = (rows_max + RC - 1) / RC;
  const long long srows = rows_max < RC ? rows_max : RC;  // rows a stage holds
  const long long stage = (srows * (in / 2 + in / 16) + 127) / 128 * 128;
  const long long xbytes = static_cast<long long>(NTOK) * (in / 32) * (4 * 16 + 8);
  // shared memory for two CTAs per SM
  const long long budget = static_cast<long long>(di.smem_per_sm / 2) - 1024 -
                           static_cast<long long>(static_smem[di.device]) - xbytes - 2ll * kQ4MaxStages * 8;
  long long S = budget > 0 ? budget / stage : 0;
  if (S > kQ4MaxStages) S = kQ4MaxStages;
  if (S > nst) S = nst;
  if (S < 1) return DEC_OK;
  a.x = q.x;
  a.x_ld = q.x_ld;
  a.norm_g = q.norm_g;
  a.eps = q.eps;
  a.y = q.y;
  a.ldy = q.ldy;
  a.in = in;
  a.nstages = static_cast<int>(S);
  a.srows = static_cast<int>(srows);
  a.stage_bytes = static_cast<uint32_t>(stage);
  a.err = q.err;
  const size_t smem = static_cast<size_t>(S * stage + xbytes + 2 * S * 8);
  WSG_CUDA_TRY(err, launch_k(kern, dim3(static_cast<unsigned>(c0)), dim3(kQ4Threads), smem, st, q.pdl, a));
  *used = true;
  return DEC_OK;
}

template <int NTOK, int XM, int EPI>
dec_status launch_q4_bulk_x(int R, const Q4Launch& q, cudaStream_t st, const DeviceInfo& di, std::string* err,
                            bool* used) {
  // a smaller R when a stage of the requested one does not fit
  for (int r = R; r >= 1 && !*used; r >>= 1) {
    dec_status e = DEC_OK;
    switch (r) {
      case 1: e = launch_q4_bulk_r<1, NTOK, XM, EPI>(q, st, di, err, used); break;
      case 2: e = launch_q4_bulk_r<2, NTOK, XM, EPI>(q, st, di, err, used); break;
      case 4: e = launch_q4_bulk_r<4, NTOK, XM, EPI>(q, st, di, err, used); break;
      default: e = launch_q4_bulk_r<8, NTOK, XM, EPI>(q, st, di, err, used); break;
    }
    if (e != DEC_OK) return e;
  }
  return DEC_OK;
}

template <int NTOK>
dec_status launch_q4_bulk(int R, const uint32_t* codes, const uint16_t* s, const uint16_t* b, const uint16_t* x,
                          float* y, int out, int in, cudaStream_t st, const DeviceInfo& di, bool* used) {
  *used = false;
  if (in % 512 || in > 16384 || !aligned16(s) || !aligned16(b) || !aligned16(x)) return DEC_OK;
  Q4Launch q = {};
  q.seg[0] = {codes, s, b, out, 0, 0};
  q.nseg = 1;
  q.x = x;
  q.x_ld = in;
  q.y = y;
  q.ldy = out;
  q.in = in;
  q.ntok = NTOK;
  q.pdl = true;
  q.err = di.err;
  if (!q.err) return fail(nullptr, DEC_ECUDA, "gemv_q4: device error word unavailable");
  return launch_q4_bulk_x<NTOK, Q4X_BF16, Q4E_STORE>(R, q, st, di, nullptr, used);
}

template <int NTOK>
dec_status launch_q4(int R, const uint32_t* codes, const uint16_t* s, const uint16_t* b, const uint16_t* x, float* y,
                     int out, int in, cudaStream_t st, const DeviceInfo& di) {
  {
    bool used = false;
    const dec_status e = launch_q4_bulk<NTOK>(R, codes, s, b, x, y, out, in, st, di, &used);
    if (e != DEC_OK || used) return e;
  }
  switch (R) {
    case 1: return launch_q4_r<1, NTOK>(codes, s, b, x, y, out, in, st, di);
    case 2: return launch_q4_r<2, NTOK>(codes, s, b, x, y, out, in, st, di);
    case 4: return launch_q4_r<4, NTOK>(codes, s, b, x, y, out, in, st, di);
    default: return launch_q4_r<8, NTOK>(codes, s, b, x, y, out, in, st, di);
  }
}

// Split-K geometry of one matrix for gemv_tma_kernel (the persistent decode
// kernel's rules): 8 column parts (16 when a part would exceed 256 columns; 4
// parts of two warps each when 8 would be at most 128 columns), 16-byte
// aligned; R rows per box minimising the busiest warp's bytes plus a fixed cost
// per box; boxes fit one 8 KB slot.
MkGeom plan_gemv_tma(int out, int in, int elem, int G) {
  MkGeom m{};
  m.wpp = 1;  // one warp per column part (two for narrow inputs, below)
  const int align = 16 / elem;
  auto width = [&](int parts) {
    const int cw = (in + parts - 1) / parts;
    return (cw + align - 1) / align * align;
  };
  m.pw = 1;
  m.cw = width(kGtWarps);
  if (m.cw > 256) {
    m.pw = 2;
    m.cw = width(2 * kGtWarps);
  } else if (m.cw <= 128) {
    m.wpp = 2;  // 4 parts of up to 256 columns, two warps each (alternate row groups)
    m.cw = width(kGtWarps / 2);
  }
  m.kc = (m.cw + 127) / 128;
  const int rmax = std::min(kMkRowsMax / m.kc, kMkSlot / (m.cw * elem));
  const int lo = out / G, hi = (out + G - 1) / G;  // rows of the CTAs
  long long best = -1;
  for (int R = 1; R <= rmax; ++R) {
    long long worst = 0;  // the busiest warp's boxes
    for (int nr : {lo, hi})
      worst = std::max(worst, static_cast<long long>(((nr + R - 1) / R + m.wpp - 1) / m.wpp) *
                                  (static_cast<long long>(R) * m.cw * elem + 2048));
    if (best < 0 || worst <= best) {
      best = worst;
      m.R = R;
    }
  }
  m.box_bytes = m.R * m.cw * elem;
  m.gchunk = std::max(1, kGtPartRows / m.R);
  return m;
}

template <typename WT>
dec_status launch_gemv_tma(const void* W, const void* x, float* y, int out, int in, cudaStream_t st,
                           const DeviceInfo& di, bool* used) {
  *used = false;
  const int elem = static_cast<int>(sizeof(WT));
  if (in > kMkMaxWidth || (in * elem) % 16 || !aligned16(W) ||
      (reinterpret_cast<uintptr_t>(x) % (4 * elem)) != 0)
    return DEC_OK;
  const int G = out < di.sms ? out : di.sms;
  const MkGeom gm = plan_gemv_tma(out, in, elem, G);
  // shared memory: byte rings, then full/empty barriers, then the partials;
  // sized for two CTAs per SM when the rings still hold a slot each
  const size_t fixed = 2 * static_cast<size_t>(kGtWarps) * kGtQ * 8 + static_cast<size_t>(kGtPartRows) * kGtWarps * 4;
  size_t per_cta = di.smem_per_sm / 2 - 1024 - 256;
  if (per_cta < fixed + static_cast<size_t>(kGtWarps) * kMkSlot) per_cta = di.smem_optin - 256;
  size_t ring = (per_cta - fixed) / kGtWarps / 128 * 128;
  if (ring > 8 * static_cast<size_t>(kMkSlot)) ring = 8 * static_cast<size_t>(kMkSlot);
  if (ring < static_cast<size_t>(kMkSlot)) return DEC_OK;
  const size_t smem = static_cast<size_t>(kGtWarps) * ring + fixed;
  alignas(64) CUtensorMap map;
  dec_status s = encode_map_2d(&map, W, out, in, elem, gm.cw, gm.R, false, nullptr);
  if (s != DEC_OK) return s;
  static bool lifted[64] = {};
  auto kern = gemv_tma_kernel<WT>;
  if (!lifted[di.device]) {  // dynamic limit: the device maximum minus the kernel's static shared memory
    cudaFuncAttributes fa{};
    WSG_CUDA_TRY(nullptr, cudaFuncGetAttributes(&fa, kern));
    WSG_CUDA_TRY(nullptr, cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(di.smem_optin - fa.sharedSizeBytes)));
    lifted[di.device] = true;
  }
  GtArgs a;
  a.x = x;
  a.y = y;
  a.out = out;
  a.in = in;
  a.gm = gm;
  a.ring_bytes = static_cast<int>(ring);
  a.err = di.err;
  if (!a.err) return fail(nullptr, DEC_ECUDA, "gemv: device error word unavailable");
  WSG_CUDA_TRY(nullptr, launch_k(kern, dim3(G), dim3(kGtThreads), smem, st, true, map, a));
  *used = true;
  return DEC_OK;
}

// Bulk-copy GEMV (gemv_bulk.cuh): one CTA per SM while each has at most 4
// stages of rows (the next launch's CTAs then fit beside them), else two per
// SM; stages of up to 8 R rows, as many as the CTA needs and two CTAs' share
// of shared memory holds. Needs 16-byte aligned W and row bytes a multiple of
// 16; *used is false when the shape does not fit.
template <typename WT, int R>
dec_status launch_gemv_bulk_r(const void* W, const void* x, float* y, int out, int in, cudaStream_t st,
                              const DeviceInfo& di, bool* used) {
  *used = false;
  auto kern = gemv_bulk_kernel<WT, R>;
  static size_t static_smem[64] = {};
  static bool lifted[64] = {};
  if (!lifted[di.device]) {
    cudaFuncAttributes fa{};
    WSG_CUDA_TRY(nullptr, cudaFuncGetAttributes(&fa, kern));
    WSG_CUDA_TRY(nullptr, cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(di.smem_optin - fa.sharedSizeBytes)));
    static_smem[di.device] = fa.sharedSizeBytes;
    lifted[di.device] = true;
  }
  constexpr int E = 16 / static_cast<int>(sizeof(WT));
  constexpr int RC = kGbWarps * R;
  const long long rb = static_cast<long long>(in) * sizeof(WT);
  int G = out < di.sms ? out : di.sms;
  if (static_cast<long long>(out) > 4ll * RC * di.sms) G = 2 * di.sms;
  const long long rows_max = (static_cast<long long>(out) + G - 1) / G;
  const long long np = (in + 32 * E - 1) / (32 * E);
  const long long xbytes = np * 32 * E * 4;
  const long long budget = static_cast<long long>(di.smem_per_sm / 2) - 1024 -
                           static_cast<long long>(static_smem[di.device]) - xbytes - 2ll * kGbMaxStages * 8;
  if (budget < rb) return DEC_OK;
  long long srows = RC;
  if (srows > rows_max) srows = rows_max;
  if (srows > budget / rb) srows = budget / rb;
  const long long stage = (srows * rb + 127) / 128 * 128;
  const long long nst = (rows_max + srows - 1) / srows;
  long long S = budget / stage;
  if (S > kGbMaxStages) S = kGbMaxStages;
  if (S > nst) S = nst;
  if (S < 1) return DEC_OK;
  GbArgs a;
  a.W = W;
  a.x = x;
  a.y = y;
  a.out = out;
  a.in = in;
  a.nstages = static_cast<int>(S);
  a.srows = static_cast<int>(srows);
  a.stage_bytes = static_cast<uint32_t>(stage);
  a.err = di.err;
  if (!a.err) return fail(nullptr, DEC_ECUDA, "gemv: device error word unavailable");
  const size_t smem = static_cast<size_t>(S * stage + xbytes + 2 * S * 8);
  WSG_CUDA_TRY(nullptr, launch_k(kern, dim3(G), dim3(kGbThreads), smem, st, true, a));
  *used = true;
  return DEC_OK;
}

// Used when every SM gets at least 16 rows and 96 KB of the matrix. Fewer,
// longer rows, and the smaller matrices whose time is mostly the launch
// handover, measured faster on the split-K kernel (its 8 warps share every
// row, x sits in registers). Rows per warp: 1 while the matrix runs one CTA
// per SM (stages of 8 rows, the finest pipeline), else a stage of 8 R rows
// near 32 KB (float32 rows of 1024: R = 1).
template <typename WT>
dec_status launch_gemv_bulk(const void* W, const void* x, float* y, int out, int in, cudaStream_t st,
                            const DeviceInfo& di, bool* used) {
  *used = false;
  const long long rb = static_cast<long long>(in) * sizeof(WT);
  if (rb % 16 || !aligned16(W) || rb > (1ll << 20) || out < 16ll * di.sms ||
      static_cast<long long>(out) * rb < 96ll * 1024 * di.sms)
    return DEC_OK;
  if (static_cast<long long>(out) <= 4ll * kGbWarps * di.sms)
    return launch_gemv_bulk_r<WT, 1>(W, x, y, out, in, st, di, used);
  const long long r = 32768 / (kGbWarps * rb);
  if (r >= 4) return launch_gemv_bulk_r<WT, 4>(W, x, y, out, in, st, di, used);
  if (r >= 2) return launch_gemv_bulk_r<WT, 2>(W, x, y, out, in, st, di, used);
  return launch_gemv_bulk_r<WT, 1>(W, x, y, out, in, st, di, used);
}

template <typename WT, typename XT>
dec_status launch_gemv(const void* W, const void* x, float* y, int out, int in, cudaStream_t st,
                       const DeviceInfo& di) {
  {
    bool used = false;
    const dec_status s = launch_gemv_bulk<WT>(W, x, y, out, in, st, di, &used);
    if (s != DEC_OK || used) return s;
  }
  {
    bool used = false;
    const dec_status s = launch_gemv_tma<WT>(W, x, y, out, in, st, di, &used);
    if (s != DEC_OK || used) return s;
  }
  const int row_bytes_ok = (static_cast<long long>(in) * sizeof(WT)) % 16 == 0;
  const long long row_bytes = static_cast<long long>(in) * sizeof(WT);
  if (row_bytes_ok && aligned16(W) && row_bytes < (1ll << 30)) {
    GemvArgs a = {};
    a.w.base[0] = a.w.base[1] = a.w.base[2] = static_cast<const char*>(W);
    a.w.split1 = a.w.split2 = out;
    a.out = out;
    a.in = in;
    a.row_bytes = static_cast<int>(row_bytes);
    int spr = static_cast<int>((row_bytes + kSEGMAX - 1) / kSEGMAX);
    int seg = static_cast<int>(((row_bytes + spr - 1) / spr + 15) / 16 * 16);
    spr = static_cast<int>((row_bytes + seg - 1) / seg);
    a.seg_bytes = seg;
    a.segs_per_row = spr;
    a.row_unit = 1;
    a.x = x;
    a.err = nullptr;
    int grid = out < di.sms ? out : di.sms;
    int max_rows = (out + grid - 1) / grid;
    // Keep the partial-dot array within shared memory by adding CTAs if needed.
    while (static_cast<size_t>(max_rows) * spr * 4 > 64 * 1024) {
      grid *= 2;
      max_rows = (out + grid - 1) / grid;
    }
    const size_t smem = gemv_smem_bytes(gemv_ring_bytes<kNW, kNSMAX, kRING>(), in, max_rows, spr);
    if (smem <= di.smem_optin) {
      auto kern = gemv_stream_kernel<WT, XT, PRO_X, EPI_STORE, kNW, kNSMAX, kRING>;
      static bool done[64] = {};
      a.err = di.err;
      if (!a.err) return fail(nullptr, DEC_ECUDA, "gemv: device error word unavailable");
      a.y = y;
      a.l2_prefetch = static_cast<long long>(out) * row_bytes <= kL2PrefetchMax;
      WSG_CUDA_TRY(nullptr, smem_once(kern, di, done));
      WSG_CUDA_TRY(nullptr, launch_k(kern, dim3(grid), dim3(kNW * 32), smem, st, true, a));
      return DEC_OK;
    }
  }
  const int blocks = static_cast<int>((static_cast<long long>(out) + 7) / 8);
  const int grid = blocks < di.sms * 8 ? blocks : di.sms * 8;
  WSG_CUDA_TRY(nullptr, launch_k(gemv_plain_kernel<WT, XT>, dim3(grid), dim3(256), 0, st, true,
                                 static_cast<const WT*>(W), static_cast<const XT*>(x), y, out, in));
  return DEC_OK;
}

}  // namespace
}  // namespace wsg

using namespace wsg;

extern "C" dec_status gemv(int32_t wdtype, const void* d_W, const void* d_x, float* d_y, int32_t out, int32_t in,
                           void* stream) {
  if (out < 0 || in < 0) return fail(nullptr, DEC_EINVAL, "gemv: negative size out=%d in=%d", out, in);
  if (wdtype != DEC_F32 && wdtype != DEC_BF16) return fail(nullptr, DEC_EINVAL, "gemv: wdtype %d", wdtype);
  if (out == 0) return DEC_OK;
  if (!d_y || (in > 0 && (!d_W || !d_x))) return fail(nullptr, DEC_EINVAL, "gemv: NULL pointer");
  DeviceInfo di;
  dec_status st = device_info(&di, nullptr);
  if (st != DEC_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (in == 0) {
    const int grid = (out + 255) / 256 < di.sms * 4 ? (out + 255) / 256 : di.sms * 4;
    WSG_CUDA_TRY(nullptr, launch_k(fill_zero_kernel, dim3(grid), dim3(256), 0, s, true, d_y, out));
    return DEC_OK;
  }
  if (wdtype == DEC_F32) return launch_gemv<float, float>(d_W, d_x, d_y, out, in, s, di);
  return launch_gemv<uint16_t, uint16_t>(d_W, d_x, d_y, out, in, s, di);
}

extern "C" dec_status gemv_q4(const uint32_t* d_codes, const uint16_t* d_scale, const uint16_t* d_bias,
                              const uint16_t* d_x, float* d_y, int32_t out, int32_t in, int32_t ntok, void* stream) {
  if (out < 0 || in < 0) return fail(nullptr, DEC_EINVAL, "gemv_q4: negative size out=%d in=%d", out, in);
  if (ntok != 1 && ntok != 2) return fail(nullptr, DEC_EINVAL, "gemv_q4: ntok must be 1 or 2, got %d", ntok);
  if (in % 64) return fail(nullptr, DEC_EINVAL, "gemv_q4: in=%d is not a multiple of 64", in);
  if (out == 0) return DEC_OK;
  if (!d_y) return fail(nullptr, DEC_EINVAL, "gemv_q4: NULL output");
  DeviceInfo di;
  dec_status st = device_info(&di, nullptr);
  if (st != DEC_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (in == 0) {
    const long long n = static_cast<long long>(out) * ntok;
    const int grid = static_cast<int>((n + 255) / 256 < di.sms * 4 ? (n + 255) / 256 : di.sms * 4);
    WSG_CUDA_TRY(nullptr, launch_k(fill_zero_kernel, dim3(grid), dim3(256), 0, s, true, d_y, static_cast<int>(n)));
    return DEC_OK;
  }
  if (!d_codes || !d_scale || !d_bias || !d_x) return fail(nullptr, DEC_EINVAL, "gemv_q4: NULL pointer");
  if (!aligned16(d_codes)) return fail(nullptr, DEC_EINVAL, "gemv_q4: codes must be 16-byte aligned");
  int R = g_q4_rows[ntok];
  if (R == 0) {
    // automatic: one row per warp when a CTA has at most one warp's worth of
    // rows (out <= 8 per SM), else four (the cold-sweep optimum of large shapes);
    // the per-warp fallback kernel keeps its own optimum (1 row, 2 for two tokens)
    const bool bulk = in % 512 == 0 && in <= 16384 && aligned16(d_scale) && aligned16(d_bias) && aligned16(d_x);
    R = bulk ? (static_cast<long long>(out) <= 8ll * di.sms ? 1 : 4) : ntok;
  }
  if (ntok == 1) return launch_q4<1>(R, d_codes, d_scale, d_bias, d_x, d_y, out, in, s, di);
  return launch_q4<2>(R, d_codes, d_scale, d_bias, d_x, d_y, out, in, s, di);
}

extern "C" int32_t gemv_q4_rows_per_warp(int32_t ntok, int32_t r) {
  if (ntok != 1 && ntok != 2) return -1;
  if (r != -1 && r != 0 && r != 1 && r != 2 && r != 4 && r != 8) return -1;
  if (r > 0) g_q4_rows[ntok] = r;
  if (r == -1) g_q4_rows[ntok] = 0;
  return g_q4_rows[ntok];
}

namespace wsg {

dec_status launch_q4_fused(const Q4Launch& q, cudaStream_t st, std::string* err) {
  DeviceInfo di;
  const dec_status ds = device_info(&di, err);
  if (ds != DEC_OK) return ds;
  if (q.in % 512 || q.in > 16384 || q.nseg < 1 || q.nseg > kQ4MaxSegs || (q.ntok != 1 && q.ntok != 2))
    return fail(err, DEC_EINVAL, "4-bit projection: in=%d (a multiple of 512 up to 16384), %d segments, %d tokens",
                q.in, q.nseg, q.ntok);
  long long total = 0;
  for (int k = 0; k < q.nseg; ++k) total += q.seg[k].rows;
  // one row per warp when a CTA has at most one warp's worth of rows, else four
  const int R = total <= 8ll * di.sms ? 1 : 4;
  bool used = false;
  dec_status e;
  const int key = (q.xm * 2 + q.epi) * 2 + (q.ntok - 1);
  switch (key) {
    case (Q4X_NORM * 2 + Q4E_STORE) * 2 + 0: e = launch_q4_bulk_x<1, Q4X_NORM, Q4E_STORE>(R, q, st, di, err, &used); break;
    case (Q4X_NORM * 2 + Q4E_STORE) * 2 + 1: e = launch_q4_bulk_x<2, Q4X_NORM, Q4E_STORE>(R, q, st, di, err, &used); break;
    case (Q4X_F32 * 2 + Q4E_ADD) * 2 + 0: e = launch_q4_bulk_x<1, Q4X_F32, Q4E_ADD>(R, q, st, di, err, &used); break;
    case (Q4X_F32 * 2 + Q4E_ADD) * 2 + 1: e = launch_q4_bulk_x<2, Q4X_F32, Q4E_ADD>(R, q, st, di, err, &used); break;
    case (Q4X_SWIGLU * 2 + Q4E_ADD) * 2 + 0: e = launch_q4_bulk_x<1, Q4X_SWIGLU, Q4E_ADD>(R, q, st, di, err, &used); break;
    case (Q4X_SWIGLU * 2 + Q4E_ADD) * 2 + 1: e = launch_q4_bulk_x<2, Q4X_SWIGLU, Q4E_ADD>(R, q, st, di, err, &used); break;
    default: return fail(err, DEC_EINVAL, "4-bit projection: prologue %d with epilogue %d is not built", q.xm, q.epi);
  }
  if (e != DEC_OK) return e;
  if (!used) return fail(err, DEC_EINVAL, "4-bit projection: in=%d does not fit in shared memory", q.in);
  return DEC_OK;
}

}  // namespace wsg

extern "C" dec_status gemv_device_errors(int32_t clear, uint32_t* bits) {
  if (!bits) return fail(nullptr, DEC_EINVAL, "gemv_device_errors: NULL output");
  WSG_CUDA_TRY(nullptr, cudaDeviceSynchronize());
  WSG_CUDA_TRY(nullptr, cudaMemcpyFromSymbol(bits, g_gemv_err, sizeof(uint32_t)));
  if (clear) {
    const uint32_t z = 0;
    WSG_CUDA_TRY(nullptr, cudaMemcpyToSymbol(g_gemv_err, &z, sizeof(uint32_t)));
  }
  return DEC_OK;
}
