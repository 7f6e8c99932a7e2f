// Decoder runtime: the batch-1 token-to-logits forward, on two engines.
//
// Step structure ("Megakernels", "GPU-wide end-to-end generation" lists eight
// ordered stages per layer plus embedding, final norm and vocabulary
// projection, then two argmax passes). Here fusion leaves five stages per
// layer and one for the head:
//
//   layer l:  QKV GEMV      (input RMSNorm fused as prologue; layer 0 also
//                            gathers the embedding row of the token)
//             attention     (per-head Q/K RMSNorm, RoPE and KV append fused)
//             O GEMV        (residual add fused as epilogue)
//             gate/up GEMV  (post-attention RMSNorm prologue, SwiGLU epilogue)
//             down GEMV     (residual add epilogue)
//   head:     vocab GEMV    (final RMSNorm prologue; logits; both argmax
//                            passes; next token and position advance)
//
// The persistent engine (the default) runs these stages for any number of
// forwards inside one cooperative launch (megakernel.cuh; q4_persist.cuh for
// 4-bit weights). The staged engine launches one kernel per stage, captured
// once as a CUDA graph: token and position live in device memory, so the same
// instantiated graph replays for every step, and kernels after the first
// carry a programmatic dependent-launch edge, so each GEMV starts streaming
// its weights while its predecessor finishes and waits only before reading
// activations. Chunked prefill (prefill.cuh, gemm_tc.cuh) runs prompt rows
// together on the tensor cores.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "attention.cuh"
#include "common.h"
#include "gemv_q4.cuh"
#include "gemv_stream.cuh"
#include "gemm_tc_host.h"
#include "megakernel.cuh"
#include "prefill.cuh"
#include "prefill_attn_tc.cuh"
#include "q4_persist.cuh"

namespace wsg {
void* mk_kernel_f32(bool kv_bf16, bool group_le2);
void* mk_kernel_bf16(bool kv_bf16, bool group_le2);
}  // namespace wsg

using namespace wsg;

namespace {

constexpr int kNW = 8, kNSMAX = 8, kRING = 12288, kSEGMAX = 4096;
constexpr long long kL2PrefetchMax = 64ll << 20;  // whole-matrix L2 prefetch up to this size
constexpr int kArgmaxPartsMax = 4096;
constexpr int kSplitMax = 64;
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
size_t dtype_bytes(int dt) { return dt == DEC_F32 ? 4 : 2; }

struct Layout {
  size_t ctrl, err, tok, h, qkv, attn, act, logits, q4gu, q4next, q4bar, q4layers, apart, acnt, mval, midx, mcnt, ll_h, ll_qkv, ll_attn,
      ll_act,
      ll_tok, ll_apart, kv_ready, mk_layers, mk_maps, rope_cos, rope_sin, kc, vc;
  // chunked prefill (chunk_cap > 0): rows padded to a multiple of 128
  size_t pf_x, pf_ah, pf_ah2, pf_qkv, pf_ao, pf_ao2, pf_ai, pf_ai2;  // *2: bfloat16 remainders
  int pf_rows;
  size_t total;
};

bool config_ok(const dec_config* c, std::string* why) {
  auto bad = [&](const char* m) {
    if (why) *why = m;
    return false;
  };
  if (!c) return bad("NULL config");
  if (c->layers < 1 || c->hidden < 1 || c->inter < 1 || c->n_q < 1 || c->n_kv < 1 || c->head_dim < 1 || c->vocab < 1)
    return bad("every geometry field must be positive");
  if (c->n_q % c->n_kv) return bad("n_q must be a multiple of n_kv");
  if (c->n_q / c->n_kv > 8) return bad("at most 8 query heads per key/value head");
  if (c->head_dim % 8 || c->head_dim > 128) return bad("head_dim must be a multiple of 8 and <= 128");
  if (c->hidden % 8 || c->inter % 8 || (c->n_q * c->head_dim) % 8)
    return bad("hidden, inter and n_q*head_dim must be multiples of 8");
  if (c->wdtype != DEC_F32 && c->wdtype != DEC_BF16 && c->wdtype != DEC_Q4G64)
    return bad("wdtype must be DEC_F32, DEC_BF16 or DEC_Q4G64");
  if (c->wdtype == DEC_Q4G64) {
    if (c->chunk_cap != 0) return bad("4-bit weights (DEC_Q4G64) take prompts one token at a time (chunk_cap 0)");
    const int w[3] = {c->hidden, c->inter, c->n_q * c->head_dim};
    for (int x : w)
      if (x % 512 || x > 16384)
        return bad("4-bit weights: hidden, inter and n_q*head_dim must be multiples of 512, at most 16384");
  }
  if (c->kvdtype != DEC_F32 && c->kvdtype != DEC_BF16) return bad("kvdtype must be DEC_F32 or DEC_BF16");
  if (c->max_seq < 1) return bad("max_seq must be >= 1");
  if (c->chunk_cap < 0) return bad("chunk_cap must be >= 0");
  if (c->chunk_cap > 0 && c->wdtype != DEC_BF16)
    return bad("batched prefill (chunk_cap > 0) runs bfloat16 tensor-core projections: wdtype must be DEC_BF16");
  if (c->engine != DEC_ENGINE_PERSISTENT && c->engine != DEC_ENGINE_STAGED) return bad("unknown engine");
  if (!(c->eps >= 0.f) || !(c->rope_theta > 0.f)) return bad("eps >= 0 and rope_theta > 0 required");
  return true;
}

Layout make_layout(const dec_config& c) {
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  const size_t qw = static_cast<size_t>(c.n_q) * c.head_dim, kvw = static_cast<size_t>(c.n_kv) * c.head_dim;
  const int group = c.n_q / c.n_kv;
  const bool q4 = c.wdtype == DEC_Q4G64;
  const size_t rows = q4 ? 2 : 1;  // the 4-bit configuration's verify step runs two rows
  L.ctrl = take(64 * 4);
  L.err = take(16);
  L.tok = take((static_cast<size_t>(c.max_seq) + 1) * 4);
  L.h = take(rows * c.hidden * 4);
  L.qkv = take(rows * (qw + 2 * kvw) * 4);
  L.attn = take(rows * qw * 4);
  L.act = take(static_cast<size_t>(c.inter) * 4);
  L.logits = take(rows * c.vocab * 4);
  L.q4gu = take(q4 ? rows * 2 * c.inter * 4 : 0);  // gate then up, per row
  L.q4next = take(16);
  L.q4bar = take(16);  // persistent 4-bit kernel: grid barrier words (cleared by dec_reset)
  L.apart = take(static_cast<size_t>(c.n_kv) * kSplitMax * group * (c.head_dim + 2) * 4);
  L.acnt = take(static_cast<size_t>(c.n_kv) * 4);
  L.mval = take(kArgmaxPartsMax * 4);
  L.midx = take(kArgmaxPartsMax * 4);
  L.mcnt = take(16);
  // persistent-engine exchange words (64-bit tag/value) and per-head cache positions
  L.ll_h = take(static_cast<size_t>(c.hidden) * 8);
  L.ll_qkv = take((qw + 2 * kvw) * 8);
  L.ll_attn = take(qw * 8);
  L.ll_act = take(static_cast<size_t>(c.inter) * 8);
  L.ll_tok = take(8);
  L.ll_apart = take(static_cast<size_t>(c.n_kv) * kSplitMax * group * (c.head_dim + 2) * 8);
  L.kv_ready = take(static_cast<size_t>(c.layers) * c.n_kv * 4);
  L.mk_layers = take(static_cast<size_t>(c.layers) * sizeof(MkLayer));
  L.mk_maps = take((static_cast<size_t>(c.layers) * kMkMapsPerLayer + 1) * kMkMapBytes);
  L.q4layers = take(q4 ? static_cast<size_t>(c.layers) * sizeof(Q4PLayer) : 0);
  L.rope_cos = take(static_cast<size_t>(c.max_seq) * (c.head_dim / 2) * 4);
  L.rope_sin = take(static_cast<size_t>(c.max_seq) * (c.head_dim / 2) * 4);
  L.pf_rows = c.chunk_cap > 0 ? (c.chunk_cap + 127) / 128 * 128 : 0;
  {
    const size_t R = static_cast<size_t>(L.pf_rows);
    L.pf_x = take(R * c.hidden * 4);
    L.pf_ah = take(R * c.hidden * 2);
    L.pf_ah2 = take(R * c.hidden * 2);
    L.pf_qkv = take(R * (qw + 2 * kvw) * 4);
    L.pf_ao = take(R * qw * 2);
    L.pf_ao2 = take(R * qw * 2);
    L.pf_ai = take(R * c.inter * 2);
    L.pf_ai2 = take(R * c.inter * 2);
  }
  const size_t cache = static_cast<size_t>(c.layers) * kvw * c.max_seq * dtype_bytes(c.kvdtype);
  L.kc = take(cache);
  L.vc = take(cache);
  L.total = o;
  return L;
}

struct Plan {  // launch shape of one decoder GEMV
  int grid = 0, seg = 0, spr = 0;
  size_t smem = 0;
  bool l2pf = false;
};

Plan plan_gemv(int out, int in, int elem, int row_unit, int sms, int max_grid) {
  Plan p;
  const long long rb = static_cast<long long>(in) * elem;
  int spr = static_cast<int>((rb + kSEGMAX - 1) / kSEGMAX);
  p.seg = static_cast<int>(((rb + spr - 1) / spr + 15) / 16 * 16);
  p.spr = static_cast<int>((rb + p.seg - 1) / p.seg);
  const int units = out / row_unit;
  p.grid = units < sms ? units : sms;
  if (p.grid > max_grid) p.grid = max_grid;
  int max_rows = (units + p.grid - 1) / p.grid * row_unit;
  while (static_cast<size_t>(max_rows) * p.spr * 4 > 64 * 1024 && p.grid * 2 <= max_grid) {
    p.grid *= 2;
    max_rows = (units + p.grid - 1) / p.grid * row_unit;
  }
  p.smem = gemv_smem_bytes(gemv_ring_bytes<kNW, kNSMAX, kRING>(), in, max_rows, p.spr);
  p.l2pf = static_cast<long long>(out) * rb <= kL2PrefetchMax;
  return p;
}

__global__ void advance_kernel(int32_t* ctrl) {
  pdl_wait();
  if (threadIdx.x == 0) ctrl[0] += 1;
}

}  // namespace

struct dec_ctx {
  dec_config cfg{};
  DeviceInfo di{};
  char* ws = nullptr;
  size_t ws_bytes = 0;
  Layout L{};
  cudaStream_t stream = nullptr;
  cudaStream_t cap = nullptr;
  bool have_weights = false;
  dec_weights w{};
  std::vector<dec_layer_weights> layers;
  int32_t pos = 0;
  int32_t* h_tok = nullptr;   // pinned [max_seq + 1], one slot per position
  int32_t* h_next = nullptr;  // pinned, two slots
  int32_t* d_h_next = nullptr;  // h_next as the device addresses it (mapped)
  cudaGraphExec_t g_full = nullptr, g_body = nullptr;
  cudaGraphExec_t g_verify = nullptr;  // 4-bit configuration: two rows through the head
  Plan p_qkv, p_o, p_gu, p_down, p_vocab;
  size_t attn_smem = 0;
  int nsplit_max = 1;
  MkArgs mk{};          // persistent-engine arguments (per-call fields filled at launch)
  uint64_t* trace = nullptr;  // caller's stage-trace buffer (persistent engine), or NULL
  uint32_t epoch = 0;         // tag prefix of the last persistent launch (1..4095)
  size_t mk_smem = 0;
  int mk_grid = 0;
  Q4PArgs q4p{};  // persistent 4-bit kernel: argument template (per-call fields filled at launch)
  size_t q4p_smem = 0;
  uint64_t xwait_ns = WSG_WAIT_LIMIT_NS;  // persistent engines: limit of a wait on another CTA
  // chunked prefill: tensor maps of the GEMM operands (activation rows: normed
  // input, attention output, SwiGLU output, then their bfloat16 remainders;
  // weights: 7 per layer)
  struct alignas(64) Map128 {
    unsigned char b[128];
  };
  Map128 pf_amap[6];
  std::vector<Map128> pf_wmap256;  // weights in 256-row boxes (256-column tiles)
  std::vector<Map128> pf_wmap;     // weights in 128-row boxes (128-column tiles; gate/up of 256-column ones)
  std::vector<Map128> pf_wmap64;  // the same in 64-row boxes (64-column tiles)
  // the whole K and V cache [layers * n_kv * max_seq][128] in 64 x 64 boxes
  // (bfloat16 cache, head size 128: pf_attn_tmem_kernel)
  Map128 pf_kvmap[2];
  bool pf_attn_tmem = false;
  std::string err;

  template <typename T>
  T* at(size_t off) const {
    return reinterpret_cast<T*>(ws + off);
  }
  size_t kv_layer_elems() const { return static_cast<size_t>(cfg.n_kv) * cfg.max_seq * cfg.head_dim; }
};

namespace {

template <typename WT, int PRO, int EPI>
dec_status launch_dec_gemv(dec_ctx* c, const Plan& p, const GemvArgs& a, cudaStream_t st, bool pdl) {
  auto kern = gemv_stream_kernel<WT, float, PRO, EPI, kNW, kNSMAX, kRING>;
  WSG_CUDA_TRY(&c->err, launch_k(kern, dim3(p.grid), dim3(kNW * 32), p.smem, st, pdl, a));
  return DEC_OK;
}

// Raise the dynamic shared-memory limit of every kernel a step launches (once,
// outside stream capture).
template <typename WT>
dec_status prepare_kernels(dec_ctx* c) {
  std::string* e = &c->err;
  WSG_CUDA_TRY(e, allow_smem(gemv_stream_kernel<WT, float, PRO_EMBED_NORM, EPI_STORE, kNW, kNSMAX, kRING>, c->p_qkv.smem));
  WSG_CUDA_TRY(e, allow_smem(gemv_stream_kernel<WT, float, PRO_NORM, EPI_STORE, kNW, kNSMAX, kRING>, c->p_qkv.smem));
  WSG_CUDA_TRY(e, allow_smem(gemv_stream_kernel<WT, float, PRO_X, EPI_RESID, kNW, kNSMAX, kRING>,
                             c->p_o.smem > c->p_down.smem ? c->p_o.smem : c->p_down.smem));
  WSG_CUDA_TRY(e, allow_smem(gemv_stream_kernel<WT, float, PRO_NORM, EPI_SWIGLU, kNW, kNSMAX, kRING>, c->p_gu.smem));
  WSG_CUDA_TRY(e, allow_smem(gemv_stream_kernel<WT, float, PRO_NORM, EPI_ARGMAX, kNW, kNSMAX, kRING>, c->p_vocab.smem));
  WSG_CUDA_TRY(e, allow_smem(attn_decode_kernel<float, 2>, c->attn_smem));
  WSG_CUDA_TRY(e, allow_smem(attn_decode_kernel<float, 8>, c->attn_smem));
  WSG_CUDA_TRY(e, allow_smem(attn_decode_kernel<uint16_t, 2>, c->attn_smem));
  WSG_CUDA_TRY(e, allow_smem(attn_decode_kernel<uint16_t, 8>, c->attn_smem));
  return DEC_OK;
}

GemvArgs base_args(dec_ctx* c, const Plan& p, int out, int in) {
  GemvArgs a = {};
  a.out = out;
  a.in = in;
  a.row_bytes = in * static_cast<int>(dtype_bytes(c->cfg.wdtype));
  a.seg_bytes = p.seg;
  a.segs_per_row = p.spr;
  a.l2_prefetch = p.l2pf;
  a.row_unit = 1;
  a.eps = c->cfg.eps;
  a.vocab = c->cfg.vocab;
  a.ctrl = c->at<int32_t>(c->L.ctrl);
  a.tok = c->at<int32_t>(c->L.tok);
  a.err = c->at<uint32_t>(c->L.err);
  return a;
}

RowMap single(const void* p, int out) {
  RowMap m = {};
  m.base[0] = m.base[1] = m.base[2] = static_cast<const char*>(p);
  m.split1 = m.split2 = out;
  return m;
}

template <typename WT>
dec_status enqueue_step_t(dec_ctx* c, cudaStream_t st, bool full) {
  const dec_config& g = c->cfg;
  const int H = g.hidden, I = g.inter, d = g.head_dim;
  const int qw = g.n_q * d, kvw = g.n_kv * d;
  const int group = g.n_q / g.n_kv;
  dec_status s;
  for (int l = 0; l < g.layers; ++l) {
    const dec_layer_weights& lw = c->layers[l];
    // QKV projection with the input RMSNorm (layer 0: of the embedding row).
    {
      GemvArgs a = base_args(c, c->p_qkv, qw + 2 * kvw, H);
      a.w.base[0] = static_cast<const char*>(lw.w_q);
      a.w.base[1] = static_cast<const char*>(lw.w_k);
      a.w.base[2] = static_cast<const char*>(lw.w_v);
      a.w.split1 = qw;
      a.w.split2 = qw + kvw;
      a.norm_g = lw.g_in;
      a.y = c->at<float>(c->L.qkv);
      if (l == 0) {
        a.embed = c->w.embed;
        a.h_out = c->at<float>(c->L.h);
        s = launch_dec_gemv<WT, PRO_EMBED_NORM, EPI_STORE>(c, c->p_qkv, a, st, false);
      } else {
        a.x = c->at<float>(c->L.h);
        s = launch_dec_gemv<WT, PRO_NORM, EPI_STORE>(c, c->p_qkv, a, st, true);
      }
      if (s != DEC_OK) return s;
    }
    // Attention with Q/K norm, RoPE and the KV append.
    {
      AttnArgs a = {};
      a.qkv = c->at<float>(c->L.qkv);
      a.g_q = lw.g_q;
      a.g_k = lw.g_k;
      a.eps = g.eps;
      a.rope_cos = c->at<float>(c->L.rope_cos);
      a.rope_sin = c->at<float>(c->L.rope_sin);
      a.ctrl = c->at<int32_t>(c->L.ctrl);
      const size_t off = static_cast<size_t>(l) * c->kv_layer_elems() * dtype_bytes(g.kvdtype);
      a.kc = c->ws + c->L.kc + off;
      a.vc = c->ws + c->L.vc + off;
      a.max_seq = g.max_seq;
      a.n_q = g.n_q;
      a.n_kv = g.n_kv;
      a.d = d;
      a.out = c->at<float>(c->L.attn);
      a.part = c->at<float>(c->L.apart);
      a.counter = c->at<uint32_t>(c->L.acnt);
      a.nsplit_max = c->nsplit_max;
      a.tmin = 64;
      a.scale = 1.0f / sqrtf(static_cast<float>(d));
      a.err = c->at<uint32_t>(c->L.err);
      cudaError_t e;
      if (g.kvdtype == DEC_F32) {
        auto k = (group <= 2) ? attn_decode_kernel<float, 2> : attn_decode_kernel<float, 8>;
        e = launch_k(k, dim3(g.n_kv, c->nsplit_max), dim3(kAttnWarps * 32), c->attn_smem, st, true, a);
      } else {
        auto k = (group <= 2) ? attn_decode_kernel<uint16_t, 2> : attn_decode_kernel<uint16_t, 8>;
        e = launch_k(k, dim3(g.n_kv, c->nsplit_max), dim3(kAttnWarps * 32), c->attn_smem, st, true, a);
      }
      WSG_CUDA_TRY(&c->err, e);
    }
    // Output projection + residual.
    {
      GemvArgs a = base_args(c, c->p_o, H, qw);
      a.w = single(lw.w_o, H);
      a.x = c->at<float>(c->L.attn);
      a.y = c->at<float>(c->L.h);
      if ((s = launch_dec_gemv<WT, PRO_X, EPI_RESID>(c, c->p_o, a, st, true)) != DEC_OK) return s;
    }
    // Gate/up projection (rows interleaved gate_i, up_i) with RMSNorm and SwiGLU.
    {
      GemvArgs a = base_args(c, c->p_gu, 2 * I, H);
      a.w.base[0] = static_cast<const char*>(lw.w_gate);
      a.w.base[1] = static_cast<const char*>(lw.w_up);
      a.w.base[2] = a.w.base[0];
      a.w.interleave = 1;
      a.row_unit = 2;
      a.x = c->at<float>(c->L.h);
      a.norm_g = lw.g_post;
      a.y = c->at<float>(c->L.act);
      if ((s = launch_dec_gemv<WT, PRO_NORM, EPI_SWIGLU>(c, c->p_gu, a, st, true)) != DEC_OK) return s;
    }
    // Down projection + residual.
    {
      GemvArgs a = base_args(c, c->p_down, H, I);
      a.w = single(lw.w_down, H);
      a.x = c->at<float>(c->L.act);
      a.y = c->at<float>(c->L.h);
      if ((s = launch_dec_gemv<WT, PRO_X, EPI_RESID>(c, c->p_down, a, st, true)) != DEC_OK) return s;
    }
  }
  if (full) {
    GemvArgs a = base_args(c, c->p_vocab, g.vocab, H);
    a.w = single(c->w.embed, g.vocab);
    a.x = c->at<float>(c->L.h);
    a.norm_g = c->w.g_final;
    a.y = c->at<float>(c->L.logits);
    a.part_val = c->at<float>(c->L.mval);
    a.part_idx = c->at<int32_t>(c->L.midx);
    a.counter = c->at<uint32_t>(c->L.mcnt);
    a.tok_w = c->at<int32_t>(c->L.tok);
    if ((s = launch_dec_gemv<WT, PRO_NORM, EPI_ARGMAX>(c, c->p_vocab, a, st, true)) != DEC_OK) return s;
  } else {
    WSG_CUDA_TRY(&c->err, launch_k(advance_kernel, dim3(1), dim3(32), 0, st, true, c->at<int32_t>(c->L.ctrl)));
  }
  return DEC_OK;
}


// ---- 4-bit configuration ----
//
// Every projection (Q/K/V, O, gate/up, down and the tied vocabulary head) is a
// 4-bit groupwise-affine matrix ("Our Kernel Benchmark Was Measuring the
// System Cache", Summary: the 4-bit matvec and its two-token variant) streamed
// by gemv_q4_bulk_kernel, whose prologue builds the bfloat16 x it consumes
// (RMSNorm, SwiGLU or a plain rounding of the float32 attention output) and
// whose epilogue stores or adds into the residual. A weight pointer points at
// one buffer holding codes [rows][in/8] u32, then scales and then biases
// [rows][in/64] fp16. Per layer: QKV (one launch over the three matrices),
// attention once per row, O (+= residual), gate/up (one launch over both),
// down (+= residual); then the head and the argmax. The verify step runs two
// rows at positions p and p + 1 through the same launches (two-token x).

Q4Seg q4_seg(const void* blob, int rows, int in, int y_off) {
  const char* b = static_cast<const char*>(blob);
  const size_t code_bytes = static_cast<size_t>(rows) * in / 2, sb = static_cast<size_t>(rows) * (in / 64) * 2;
  Q4Seg s{};
  s.codes = reinterpret_cast<const uint32_t*>(b);
  s.scale = reinterpret_cast<const uint16_t*>(b + code_bytes);
  s.bias = reinterpret_cast<const uint16_t*>(b + code_bytes + sb);
  s.rows = rows;
  s.y_off = y_off;
  return s;
}

// h[t] = the dequantised embedding row of the token at position ctrl[0] + t:
// w = s * q + b (product, then sum, each rounded to float32).
__global__ void q4_embed_kernel(const int32_t* __restrict__ tok, const int32_t* __restrict__ ctrl,
                                const unsigned char* __restrict__ E, int V, int H, float* __restrict__ h,
                                uint32_t* err) {
  pdl_wait();
  const int t = blockIdx.x;
  int token = tok[ctrl[0] + t];
  if (token < 0 || token >= V) {
    if (threadIdx.x == 0) atomicOr(err, ERR_BAD_TOKEN);
    token = 0;
  }
  const uint32_t* codes = reinterpret_cast<const uint32_t*>(E) + static_cast<size_t>(token) * (H / 8);
  const __half* sc = reinterpret_cast<const __half*>(E + static_cast<size_t>(V) * H / 2) + static_cast<size_t>(token) * (H / 64);
  const __half* bi = sc + static_cast<size_t>(V) * (H / 64);
  for (int j = threadIdx.x; j < H; j += blockDim.x) {
    const uint32_t q = (codes[j >> 3] >> (4 * (j & 7))) & 0xFu;
    h[static_cast<size_t>(t) * H + j] =
        __fadd_rn(__fmul_rn(__half2float(sc[j >> 6]), static_cast<float>(q)), __half2float(bi[j >> 6]));
  }
}

// Greedy token of each of the ntok logit rows (lowest ID on ties): CTA (b, t)
// reduces a slice of row t to one candidate; the last CTA to finish reduces the
// candidates, writes next[t], the token after the last row into the token
// stream, and advances the position by ntok.
constexpr int kQ4ArgmaxThreads = 256;
__global__ void __launch_bounds__(kQ4ArgmaxThreads) q4_argmax_kernel(const float* __restrict__ logits, int V, int ntok,
                                                                     float* part_val, int32_t* part_idx,
                                                                     uint32_t* counter, int32_t* tok, int32_t* ctrl,
                                                                     int32_t* next, uint32_t* err) {
  __shared__ float sv[kQ4ArgmaxThreads / 32];
  __shared__ int si[kQ4ArgmaxThreads / 32];
  __shared__ int s_last;
  pdl_wait();
  const int P = gridDim.x, b = blockIdx.x, t = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto block_best = [&](float& bv, int& bi) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (argmax_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    __syncthreads();
    if (lane == 0) {
      sv[warp] = bv;
      si[warp] = bi;
    }
    __syncthreads();
    bv = sv[0];
    bi = si[0];
    for (int w = 1; w < kQ4ArgmaxThreads / 32; ++w)
      if (argmax_better(sv[w], si[w], bv, bi)) {
        bv = sv[w];
        bi = si[w];
      }
  };
  const float* row = logits + static_cast<size_t>(t) * V;
  const int i0 = static_cast<int>(static_cast<long long>(b) * V / P), i1 = static_cast<int>(static_cast<long long>(b + 1) * V / P);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = i0 + tid; i < i1; i += kQ4ArgmaxThreads) {
    const float v = __ldcg(row + i);
    if (argmax_better(v, i, bv, bi)) {
      bv = v;
      bi = i;
    }
  }
  block_best(bv, bi);
  if (tid == 0) {
    part_val[t * P + b] = bv;
    part_idx[t * P + b] = bi;
    __threadfence();
    s_last = atomicAdd(counter, 1u) == static_cast<uint32_t>(P * ntok - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int pos = ctrl[0];
  int last = 0;
  for (int tt = 0; tt < ntok; ++tt) {
    float gv = -INFINITY;
    int gi = 0x7fffffff;
    for (int k = tid; k < P; k += kQ4ArgmaxThreads) {
      const float v = __ldcg(part_val + tt * P + k);
      const int i = __ldcg(part_idx + tt * P + k);
      if (argmax_better(v, i, gv, gi)) {
        gv = v;
        gi = i;
      }
    }
    block_best(gv, gi);
    if (gi == 0x7fffffff) {  // every logit of the row was NaN
      gi = 0;
      if (tid == 0) atomicOr(err, ERR_ARGMAX_NAN);
    }
    if (tid == 0) next[tt] = gi;
    last = gi;
  }
  if (tid == 0) {
    tok[pos + ntok] = last;
    ctrl[0] = pos + ntok;
    *counter = 0u;
    __threadfence();
  }
}

dec_status enqueue_step_q4(dec_ctx* c, cudaStream_t st, bool full, int ntok) {
  const dec_config& g = c->cfg;
  const int H = g.hidden, I = g.inter, d = g.head_dim;
  const int qw = g.n_q * d, kvw = g.n_kv * d, qkvw = qw + 2 * kvw;
  const int group = g.n_q / g.n_kv;
  float* h = c->at<float>(c->L.h);
  float* qkv = c->at<float>(c->L.qkv);
  float* attn = c->at<float>(c->L.attn);
  float* gu = c->at<float>(c->L.q4gu);
  uint32_t* err = c->at<uint32_t>(c->L.err);
  auto base = [&](int xm, int epi, const void* x, int x_ld, const float* gain, float* y, int ldy, int in) {
    Q4Launch q = {};
    q.xm = xm;
    q.epi = epi;
    q.ntok = ntok;
    q.x = x;
    q.x_ld = x_ld;
    q.norm_g = gain;
    q.eps = g.eps;
    q.y = y;
    q.ldy = ldy;
    q.in = in;
    q.pdl = true;
    q.err = err;
    return q;
  };
  WSG_CUDA_TRY(&c->err, launch_k(q4_embed_kernel, dim3(ntok), dim3(256), 0, st, false, c->at<int32_t>(c->L.tok),
                                 c->at<int32_t>(c->L.ctrl), static_cast<const unsigned char*>(c->w.embed), g.vocab, H,
                                 h, err));
  dec_status s;
  for (int l = 0; l < g.layers; ++l) {
    const dec_layer_weights& lw = c->layers[l];
    {
      Q4Launch q = base(Q4X_NORM, Q4E_STORE, h, H, lw.g_in, qkv, qkvw, H);
      q.seg[0] = q4_seg(lw.w_q, qw, H, 0);
      q.seg[1] = q4_seg(lw.w_k, kvw, H, qw);
      q.seg[2] = q4_seg(lw.w_v, kvw, H, qw + kvw);
      q.nseg = 3;
      if ((s = launch_q4_fused(q, st, &c->err)) != DEC_OK) return s;
    }
    for (int t = 0; t < ntok; ++t) {
      AttnArgs a = {};
      a.qkv = qkv + static_cast<size_t>(t) * qkvw;
      a.g_q = lw.g_q;
      a.g_k = lw.g_k;
      a.eps = g.eps;
      a.rope_cos = c->at<float>(c->L.rope_cos);
      a.rope_sin = c->at<float>(c->L.rope_sin);
      a.ctrl = c->at<int32_t>(c->L.ctrl);
      a.pos_add = t;
      const size_t off = static_cast<size_t>(l) * c->kv_layer_elems() * dtype_bytes(g.kvdtype);
      a.kc = c->ws + c->L.kc + off;
      a.vc = c->ws + c->L.vc + off;
      a.max_seq = g.max_seq;
      a.n_q = g.n_q;
      a.n_kv = g.n_kv;
      a.d = d;
      a.out = attn + static_cast<size_t>(t) * qw;
      a.part = c->at<float>(c->L.apart);
      a.counter = c->at<uint32_t>(c->L.acnt);
      a.nsplit_max = c->nsplit_max;
      a.tmin = 64;
      a.scale = 1.0f / sqrtf(static_cast<float>(d));
      a.err = err;
      cudaError_t e;
      if (g.kvdtype == DEC_F32) {
        auto k = (group <= 2) ? attn_decode_kernel<float, 2> : attn_decode_kernel<float, 8>;
        e = launch_k(k, dim3(g.n_kv, c->nsplit_max), dim3(kAttnWarps * 32), c->attn_smem, st, true, a);
      } else {
        auto k = (group <= 2) ? attn_decode_kernel<uint16_t, 2> : attn_decode_kernel<uint16_t, 8>;
        e = launch_k(k, dim3(g.n_kv, c->nsplit_max), dim3(kAttnWarps * 32), c->attn_smem, st, true, a);
      }
      WSG_CUDA_TRY(&c->err, e);
    }
    {
      Q4Launch q = base(Q4X_F32, Q4E_ADD, attn, qw, nullptr, h, H, qw);
      q.seg[0] = q4_seg(lw.w_o, H, qw, 0);
      q.nseg = 1;
      if ((s = launch_q4_fused(q, st, &c->err)) != DEC_OK) return s;
    }
    {
      Q4Launch q = base(Q4X_NORM, Q4E_STORE, h, H, lw.g_post, gu, 2 * I, H);
      q.seg[0] = q4_seg(lw.w_gate, I, H, 0);
      q.seg[1] = q4_seg(lw.w_up, I, H, I);
      q.nseg = 2;
      if ((s = launch_q4_fused(q, st, &c->err)) != DEC_OK) return s;
    }
    {
      Q4Launch q = base(Q4X_SWIGLU, Q4E_ADD, gu, 2 * I, nullptr, h, H, I);
      q.seg[0] = q4_seg(lw.w_down, H, I, 0);
      q.nseg = 1;
      if ((s = launch_q4_fused(q, st, &c->err)) != DEC_OK) return s;
    }
  }
  if (!full) {
    WSG_CUDA_TRY(&c->err, launch_k(advance_kernel, dim3(1), dim3(32), 0, st, true, c->at<int32_t>(c->L.ctrl)));
    return DEC_OK;
  }
  {
    Q4Launch q = base(Q4X_NORM, Q4E_STORE, h, H, c->w.g_final, c->at<float>(c->L.logits), g.vocab, H);
    q.seg[0] = q4_seg(c->w.embed, g.vocab, H, 0);
    q.nseg = 1;
    if ((s = launch_q4_fused(q, st, &c->err)) != DEC_OK) return s;
  }
  const int P = std::min(c->di.sms, kArgmaxPartsMax / 2);
  WSG_CUDA_TRY(&c->err, launch_k(q4_argmax_kernel, dim3(P, ntok), dim3(kQ4ArgmaxThreads), 0, st, true,
                                 static_cast<const float*>(c->at<float>(c->L.logits)), g.vocab, ntok,
                                 c->at<float>(c->L.mval), c->at<int32_t>(c->L.midx), c->at<uint32_t>(c->L.mcnt),
                                 c->at<int32_t>(c->L.tok), c->at<int32_t>(c->L.ctrl), c->at<int32_t>(c->L.q4next),
                                 err));
  return DEC_OK;
}

// ---- chunked prefill ----

// Rows p0..p0+n-1 (tokens already in the token stream) through every layer
// together: per-row kernels (prefill.cuh) between tensor-core GEMMs over the
// chunk's rows (gemm_tc.cuh); the last row optionally through the head.
template <typename KT>
dec_status run_chunk_prefill_t(dec_ctx* c, int p0, int n, bool is_last) {
  const dec_config& g = c->cfg;
  const Layout& L = c->L;
  const int H = g.hidden, I = g.inter, d = g.head_dim;
  const int qw = g.n_q * d, kvw = g.n_kv * d, W = qw + 2 * kvw;
  const int group = g.n_q / g.n_kv;
  cudaStream_t st = c->stream;
  float* X = c->at<float>(L.pf_x);
  uint16_t* AH = c->at<uint16_t>(L.pf_ah);
  uint16_t* AH2 = c->at<uint16_t>(L.pf_ah2);
  float* QKV = c->at<float>(L.pf_qkv);
  uint16_t* AO = c->at<uint16_t>(L.pf_ao);
  uint16_t* AO2 = c->at<uint16_t>(L.pf_ao2);
  uint16_t* AI = c->at<uint16_t>(L.pf_ai);
  uint16_t* AI2 = c->at<uint16_t>(L.pf_ai2);
  uint32_t* err = c->at<uint32_t>(L.err);
  const float* rc = c->at<float>(L.rope_cos);
  const float* rs = c->at<float>(L.rope_sin);
  dec_status s;
  // weight map `wm` in boxes of the tile width (gemm_plan picks the width)
  auto wmap = [&](int wm, int bn) {
    return bn == 64 ? c->pf_wmap64[wm].b : bn == 128 ? c->pf_wmap[wm].b : c->pf_wmap256[wm].b;
  };
  // C[:, col0..col0+N) (=, or += with accumulate) rows . W^T with operand
  // maps `amap` and amap + 3 (value and remainder of: 0 normed input, 1
  // attention output, 2 SwiGLU output) and weight map `wm`
  auto gemm = [&](int amap, int wm, float* C, int ldc, int col0, int N, int K, bool acc) {
    const int bn = gemm_plan(n, N, K, c->di.sms, 0, true);
    const void* mb[1] = {wmap(wm, bn)};
    return launch_gemm_bf16(c->pf_amap[amap].b, c->pf_amap[amap + 3].b, mb, nullptr, 1, bn, C, ldc, col0, n, N, K, acc,
                            err, st, &c->err);
  };
  // Several weights side by side in one launch (Q, K, V): one grid over all
  // their columns fills the GPU better than a launch per weight. Their widths
  // are whole 128-column tiles; 256-column tiles where they are whole ones.
  auto gemm_multi = [&](int amap, const int* wms, const int* widths, int nw, float* C, int ldc, int K) {
    const void* mb[3];
    int nb[2] = {0, 0}, N = 0, orb = 0;
    for (int i = 0; i < nw; ++i) {
      N += widths[i];
      if (i + 1 < nw) orb |= N;  // the boundary after weight i
    }
    const int align = orb & -orb;  // largest power of two dividing every boundary (0: none)
    const int bn = gemm_plan(n, N, K, c->di.sms, align, true);
    for (int i = 0, acc = 0; i < nw; ++i) {
      mb[i] = wmap(wms[i], bn);
      acc += widths[i];
      if (i + 1 < nw) nb[i] = acc;
    }
    return launch_gemm_bf16(c->pf_amap[amap].b, c->pf_amap[amap + 3].b, mb, nb, nw, bn, C, ldc, 0, n, N, K, false, err,
                            st, &c->err);
  };
  const bool fuse_qkv = qw % kGemmTileN == 0 && kvw % kGemmTileN == 0;
  // RMSNorm of the residual rows into the next GEMM's operand pair
  const bool norm4 = H % 4 == 0 && H <= 4 * kPfNormPieces * kPfThreads;
  auto norm = [&](const float* Xr, const float* gain, float eps, int Hn, uint16_t* A, uint16_t* A2) {
    return norm4 && (reinterpret_cast<uintptr_t>(gain) & 15u) == 0
               ? launch_k(pf_norm4_kernel, dim3(n), dim3(kPfThreads), 0, st, true, Xr, gain, eps, Hn, A, A2)
               : launch_k(pf_norm_kernel, dim3(n), dim3(kPfThreads), 0, st, true, Xr, gain, eps, Hn, A, A2);
  };
  pf_embed_norm_kernel<uint16_t><<<n, kPfThreads, 0, st>>>(c->at<int32_t>(L.tok), p0, c->w.embed, g.vocab,
                                                           c->layers[0].g_in, g.eps, H, X, AH, AH2, err);
  WSG_CUDA_TRY(&c->err, cudaGetLastError());
  for (int l = 0; l < g.layers; ++l) {
    const dec_layer_weights& lw = c->layers[l];
    const int wm = l * kMkMapsPerLayer;
    if (l > 0) {
      WSG_CUDA_TRY(&c->err, norm(X, lw.g_in, g.eps, H, AH, AH2));
      WSG_CUDA_TRY(&c->err, cudaGetLastError());
    }
    if (fuse_qkv) {
      const int wms[3] = {wm + 0, wm + 1, wm + 2}, widths[3] = {qw, kvw, kvw};
      if ((s = gemm_multi(0, wms, widths, 3, QKV, W, H)) != DEC_OK) return s;
    } else {
      if ((s = gemm(0, wm + 0, QKV, W, 0, qw, H, false)) != DEC_OK) return s;
      if ((s = gemm(0, wm + 1, QKV, W, qw, kvw, H, false)) != DEC_OK) return s;
      if ((s = gemm(0, wm + 2, QKV, W, qw + kvw, kvw, H, false)) != DEC_OK) return s;
    }
    const size_t off = static_cast<size_t>(l) * c->kv_layer_elems() * dtype_bytes(g.kvdtype);
    void* kc = c->ws + L.kc + off;
    void* vc = c->ws + L.vc + off;
    if (d == 128 || d == 64 || d == 32) {
      auto rk = d == 128 ? pf_qk_rope_kv_vec_kernel<KT, 4>
                         : d == 64 ? pf_qk_rope_kv_vec_kernel<KT, 2> : pf_qk_rope_kv_vec_kernel<KT, 1>;
      const long long pairs = static_cast<long long>(n) * (g.n_q + 2 * g.n_kv);
      WSG_CUDA_TRY(&c->err, launch_k(rk, dim3(static_cast<unsigned>((pairs + 7) / 8)), dim3(256), 0, st, true, QKV, n,
                                     p0, g.n_q, g.n_kv, static_cast<const float*>(lw.g_q),
                                     static_cast<const float*>(lw.g_k), g.eps, rc, rs, kc, vc, g.max_seq));
    } else {
      WSG_CUDA_TRY(&c->err, launch_k(pf_qk_rope_kv_kernel<KT>, dim3(n, (g.n_q + 2 * g.n_kv + 3) / 4), dim3(128), 0,
                                     st, true, QKV, p0, g.n_q, g.n_kv, d, static_cast<const float*>(lw.g_q),
                                     static_cast<const float*>(lw.g_k), g.eps, rc, rs, kc, vc, g.max_seq));
    }
    WSG_CUDA_TRY(&c->err, cudaGetLastError());
    // A chunk that does not end the prompt stops after the last layer's K/V
    // write: later rows read only the cache, so that layer's attention output,
    // O projection and MLP would feed nothing. The terminal chunk runs it all.
    if (l == g.layers - 1 && !is_last) break;
    const float scale = 1.0f / std::sqrt(static_cast<float>(d));
    bool tc = false;
    if (c->pf_attn_tmem) {  // bfloat16 cache, head size 128: tcgen05 attention
      static bool lifted[64] = {};  // per device
      if (!lifted[c->di.device]) {
        WSG_CUDA_TRY(&c->err, cudaFuncSetAttribute(pf_attn_tmem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kAtSmem)));
        lifted[c->di.device] = true;
      }
      PfAttnArgs aa;
      aa.qkv = QKV;
      aa.AO = AO;
      aa.AO2 = AO2;
      aa.err = err;
      aa.n = n;
      aa.p0 = p0;
      aa.n_q = g.n_q;
      aa.n_kv = g.n_kv;
      aa.kv_row0 = l * g.n_kv * g.max_seq;
      aa.max_seq = g.max_seq;
      aa.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
      const int rows = kAtBM / group;
      WSG_CUDA_TRY(&c->err, launch_k(pf_attn_tmem_kernel, dim3(g.n_kv, (n + rows - 1) / rows), dim3(kAtThreads),
                                     kAtSmem, st, true, *reinterpret_cast<const CUtensorMap*>(c->pf_kvmap[0].b),
                                     *reinterpret_cast<const CUtensorMap*>(c->pf_kvmap[1].b), aa));
      tc = true;
    } else if constexpr (sizeof(KT) == 2) {  // bfloat16 cache, other head sizes or groups: warp-level MMAs
      void (*tk)(const float*, int, int, int, int, const uint16_t*, const uint16_t*, int, float, uint16_t*, uint16_t*) =
          d == 128 ? pf_attn_tc_kernel<128> : d == 64 ? pf_attn_tc_kernel<64> : d == 32 ? pf_attn_tc_kernel<32>
                                                                            : d == 16 ? pf_attn_tc_kernel<16> : nullptr;
      if (tk && 16 % group == 0) {
        const int rows_per_block = kPfTcWarps * (16 / group);
        const size_t smem = pf_attn_tc_smem(d);
        static bool lifted[64][4] = {};  // per device, per head size
        const int hs = d == 128 ? 0 : d == 64 ? 1 : d == 32 ? 2 : 3;
        if (!lifted[c->di.device][hs]) {
          WSG_CUDA_TRY(&c->err, cudaFuncSetAttribute(tk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     static_cast<int>(smem)));
          lifted[c->di.device][hs] = true;
        }
        WSG_CUDA_TRY(&c->err, launch_k(tk, dim3(g.n_kv, (n + rows_per_block - 1) / rows_per_block),
                                       dim3(kPfTcWarps * 32), smem, st, true, static_cast<const float*>(QKV), n, p0,
                                       g.n_q, g.n_kv, static_cast<const uint16_t*>(kc),
                                       static_cast<const uint16_t*>(vc), g.max_seq, scale, AO, AO2));
        tc = true;
      }
    }
    if (!tc) {
      auto ak = group <= 2 ? pf_attn_kernel<KT, 2> : pf_attn_kernel<KT, 8>;
      WSG_CUDA_TRY(&c->err, launch_k(ak, dim3(g.n_kv, (n + kPfAttnRows - 1) / kPfAttnRows), dim3(kPfAttnRows * 32), 0,
                                     st, true, static_cast<const float*>(QKV), n, p0, g.n_q, g.n_kv, d,
                                     static_cast<const void*>(kc), static_cast<const void*>(vc), g.max_seq, scale, AO,
                                     AO2));
    }
    WSG_CUDA_TRY(&c->err, cudaGetLastError());
    if ((s = gemm(1, wm + 3, X, H, 0, H, qw, true)) != DEC_OK) return s;  // O projection + residual
    WSG_CUDA_TRY(&c->err, norm(X, lw.g_post, g.eps, H, AH, AH2));
    WSG_CUDA_TRY(&c->err, cudaGetLastError());
    // gate/up with SwiGLU in the GEMM's epilogue: a tile pairs bn/2 gate and bn/2 up outputs
    const int gbn = gemm_plan(n, 2 * I, H, c->di.sms, 256, true) == 256 ? 256 : 128;
    const void* gmap = gbn == 256 ? c->pf_wmap[wm + 4].b : c->pf_wmap64[wm + 4].b;
    const void* umap = gbn == 256 ? c->pf_wmap[wm + 5].b : c->pf_wmap64[wm + 5].b;
    if ((s = launch_gemm_swiglu(c->pf_amap[0].b, c->pf_amap[3].b, gmap, umap, gbn, AI,
                                AI2, I, n, I, H, err, st, &c->err)) != DEC_OK)
      return s;
    if ((s = gemm(2, wm + 6, X, H, 0, H, I, true)) != DEC_OK) return s;  // down projection + residual
  }
  // Position word (the head's position, or the next one) and, for the
  // persistent engine, the appended cache rows published to its readers.
  uint32_t* kvr = g.engine == DEC_ENGINE_PERSISTENT ? c->at<uint32_t>(L.kv_ready) : nullptr;
  pf_control_kernel<<<1, 256, 0, st>>>(c->at<int32_t>(L.ctrl), is_last ? p0 + n - 1 : p0 + n, kvr,
                                       g.layers * g.n_kv, static_cast<uint32_t>(p0 + n));
  WSG_CUDA_TRY(&c->err, cudaGetLastError());
  if (is_last) {
    pf_copy_row_kernel<<<1, 256, 0, st>>>(X + static_cast<size_t>(n - 1) * H, c->at<float>(L.h), H);
    WSG_CUDA_TRY(&c->err, cudaGetLastError());
    GemvArgs a = base_args(c, c->p_vocab, g.vocab, H);
    a.w = single(c->w.embed, g.vocab);
    a.x = c->at<float>(L.h);
    a.norm_g = c->w.g_final;
    a.y = c->at<float>(L.logits);
    a.part_val = c->at<float>(L.mval);
    a.part_idx = c->at<int32_t>(L.midx);
    a.counter = c->at<uint32_t>(L.mcnt);
    a.tok_w = c->at<int32_t>(L.tok);
    if ((s = launch_dec_gemv<uint16_t, PRO_NORM, EPI_ARGMAX>(c, c->p_vocab, a, st, false)) != DEC_OK) return s;
  }
  return DEC_OK;
}

dec_status run_chunk_prefill(dec_ctx* c, int p0, int n, bool is_last) {
  return c->cfg.kvdtype == DEC_F32 ? run_chunk_prefill_t<float>(c, p0, n, is_last)
                                   : run_chunk_prefill_t<uint16_t>(c, p0, n, is_last);
}

// ---- persistent engine ----

// Rows of each piece of stage st for CTA c of G (the kernel's partition,
// mirrored on the host to plan box heights and partial capacity).
void mk_pieces(const dec_config& g, int st, int c, int G, int nr[3]) {
  const long long qw = static_cast<long long>(g.n_q) * g.head_dim, kvw = static_cast<long long>(g.n_kv) * g.head_dim;
  const long long units = st == MK_QKV ? qw + 2 * kvw : st == MK_GU ? g.inter : st == MK_VOCAB ? g.vocab : g.hidden;
  const long long u0 = c * units / G, u1 = (c + 1) * units / G;
  nr[0] = nr[1] = nr[2] = 0;
  if (st == MK_QKV) {
    auto clampr = [](long long x, long long lo, long long hi) { return std::min(std::max(x, lo), hi); };
    nr[0] = static_cast<int>(clampr(u1, 0, qw) - clampr(u0, 0, qw));
    nr[1] = static_cast<int>(clampr(u1, qw, qw + kvw) - clampr(u0, qw, qw + kvw));
    nr[2] = static_cast<int>(std::max(u1, qw + kvw) - std::max(u0, qw + kvw));
  } else if (st == MK_GU) {
    nr[0] = nr[1] = static_cast<int>(u1 - u0);
  } else {
    nr[0] = static_cast<int>(u1 - u0);
  }
}

// Split-K geometry of stage st (input width `in`): 8 column parts, one per
// consumer warp (16 when a part would exceed 256 columns, the TMA box limit;
// 4, two warps each, when 8 parts would be at most 128 columns), each 16-byte
// aligned; R rows per box chosen to minimise the busiest warp's streamed
// bytes plus a fixed cost per box; boxes fit one ring slot.
MkGeom mk_geom_for(const dec_config& g, int st, int in, int elem, int G) {
  MkGeom m{};
  const int align = 16 / elem;
  auto width = [&](int parts) {
    const int cw = (in + parts - 1) / parts;
    return (cw + align - 1) / align * align;
  };
  m.pw = 1;
  m.wpp = 1;
  m.cw = width(kMkWarps);
  if (m.cw > 256) {
    m.pw = 2;
    m.cw = width(2 * kMkWarps);
  } else if (m.cw <= 128) {
    // narrow inputs: 4 parts of up to 256 columns, two warps each (alternate
    // row groups). A box then holds fewer, longer rows for the same bytes,
    // so a warp reduces fewer rows per byte.
    m.wpp = 2;
    m.cw = width(kMkWarps / 2);
  }
  m.kc = (m.cw + 127) / 128;
  // rows per box: the consumer unrolls over at most kMkRowsMax rows of a
  // one-chunk part (its code stays small enough to stay in the instruction cache)
  const int rmax = std::min(kMkRowsMax / m.kc, kMkSlot / (m.cw * elem));
  constexpr long long kBoxCost = 2048;
  long long best = -1;
  for (int R = 1; R <= rmax; ++R) {
    // the busiest warp of the busiest CTA: its boxes' bytes plus a fixed cost
    // per box (a copy of a few KB runs below the streaming rate of larger ones)
    long long worst = 0;
    for (int c = 0; c < G; ++c) {
      int nr[3];
      mk_pieces(g, st, c, G, nr);
      long long ng = 0;
      for (int p = 0; p < 3; ++p) ng += (nr[p] + R - 1) / R;
      const long long cost =
          (ng + m.wpp - 1) / m.wpp * m.pw * (static_cast<long long>(R) * m.cw * elem + kBoxCost);
      worst = std::max(worst, cost);
    }
    if (best < 0 || worst <= best) {
      best = worst;
      m.R = R;
    }
  }
  m.box_bytes = m.R * m.cw * elem;
  return m;
}

// Most row groups x R over the CTAs (shared partial rows the stage needs in one chunk).
int mk_group_rows(const dec_config& g, int st, const MkGeom& m, int G) {
  int most = 0;
  for (int c = 0; c < G; ++c) {
    int nr[3];
    mk_pieces(g, st, c, G, nr);
    int ng = 0;
    for (int p = 0; p < 3; ++p) ng += (nr[p] + m.R - 1) / m.R;
    most = std::max(most, ng * m.R);
  }
  return most;
}

// Tensor map of a row-major [rows][in] weight matrix with boxes of m.R rows x m.cw columns.
dec_status encode_map(CUtensorMap* out, const void* base, int rows, int in, int wdtype, const MkGeom& m,
                      std::string* err) {
  return encode_map_2d(out, base, rows, in, static_cast<int>(dtype_bytes(wdtype)), m.cw, m.R, false, err);
}

// Persistent kernel instance for the configuration (defined per weight dtype in
// megakernel_f32.cu / megakernel_bf16.cu).
void* mk_kernel(const dec_config& g) {
  const bool g2 = g.n_q / g.n_kv <= 2;
  return g.wdtype == DEC_F32 ? mk_kernel_f32(g.kvdtype == DEC_BF16, g2) : mk_kernel_bf16(g.kvdtype == DEC_BF16, g2);
}

// Plan the persistent engine: ring depth, staging sizes, argument template.
dec_status plan_persistent(dec_ctx* c) {
  const dec_config& g = c->cfg;
  const int elem = static_cast<int>(dtype_bytes(g.wdtype));
  const int qw = g.n_q * g.head_dim, kvw = g.n_kv * g.head_dim;
  const int G = c->di.sms;
  MkArgs& a = c->mk;
  a = MkArgs{};
  a.L = g.layers;
  a.H = g.hidden;
  a.I = g.inter;
  a.n_q = g.n_q;
  a.n_kv = g.n_kv;
  a.d = g.head_dim;
  a.V = g.vocab;
  a.eps = g.eps;
  if (std::max(g.hidden, std::max(qw, g.inter)) > kMkMaxWidth)
    return fail(&c->err, DEC_EINVAL, "persistent engine: widths above %d need the staged engine", kMkMaxWidth);
  a.gq = mk_geom_for(g, MK_QKV, g.hidden, elem, G);
  a.go = mk_geom_for(g, MK_O, qw, elem, G);
  a.gg = mk_geom_for(g, MK_GU, g.hidden, elem, G);
  a.gd = mk_geom_for(g, MK_DOWN, g.inter, elem, G);
  a.gv = mk_geom_for(g, MK_VOCAB, g.hidden, elem, G);
  (void)kvw;
  auto cdiv = [](long long x, long long y) { return static_cast<int>((x + y - 1) / y); };
  // Shared partials: every layer stage in one chunk; the vocabulary in chunks.
  int prows = kMkPartRows;
  prows = std::max(prows, mk_group_rows(g, MK_QKV, a.gq, G));
  prows = std::max(prows, mk_group_rows(g, MK_O, a.go, G));
  prows = std::max(prows, mk_group_rows(g, MK_GU, a.gg, G));
  prows = std::max(prows, mk_group_rows(g, MK_DOWN, a.gd, G));
  for (MkGeom* m : {&a.gq, &a.go, &a.gg, &a.gd, &a.gv}) m->gchunk = std::max(1, prows / m->R);
  a.part_floats = prows * kMkWarps;
  // staging of one activation vector; the attention scratch shares it
  a.xs_floats = std::max(static_cast<int>((attn_smem_bytes(g.n_q / g.n_kv, g.head_dim) + 15) / 16 * 4),
                         (std::max(g.hidden, std::max(qw, g.inter)) + 3) / 4 * 4);
  a.hown_floats = (cdiv(g.hidden, G) + 3) / 4 * 4;
  const size_t fixed = 2 * kMkWarps * kMkQ * sizeof(uint64_t) +  // full and empty barriers
                       4 * static_cast<size_t>(a.xs_floats + a.part_floats) +
                       static_cast<size_t>(g.layers) * kMkLayerPtrs * sizeof(void*) + 4 * static_cast<size_t>(a.hown_floats);
  const size_t static_smem = 64 * 4 + 32 * 4 + 8 + 5 * sizeof(MkStageT) + 256;
  if (fixed + static_smem + static_cast<size_t>(kMkWarps) * kMkSlot > c->di.smem_optin)
    return fail(&c->err, DEC_EINVAL, "persistent engine: staging needs %zu B of shared memory", fixed);
  // every warp's ring: what is left, in 128-byte units, at most 8 slots' worth
  const size_t ring = std::min<size_t>(8 * kMkSlot, (c->di.smem_optin - fixed - static_smem) / kMkWarps / 128 * 128);
  a.ring_bytes = static_cast<int>(ring);
  c->mk_smem = static_cast<size_t>(kMkWarps) * ring + fixed;
  c->mk_grid = G;
  void* k = mk_kernel(g);
  WSG_CUDA_TRY(&c->err, cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(c->mk_smem)));
  int per_sm = 0;
  WSG_CUDA_TRY(&c->err, cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kMkThreads, c->mk_smem));
  if (per_sm < 1) return fail(&c->err, DEC_EINVAL, "persistent engine: kernel does not fit on an SM");
  // The warpgroups re-split the registers the block is launched with
  // (setmaxnreg); the new split must fit in them, or the raise would wait forever.
  cudaFuncAttributes fa{};
  WSG_CUDA_TRY(&c->err, cudaFuncGetAttributes(&fa, k));
  if (static_cast<long long>(fa.numRegs) * kMkThreads <
      static_cast<long long>(kMkConsumerRegs) * kMkConsumers + static_cast<long long>(kMkProducerRegs) * 128)
    return fail(&c->err, DEC_EINVAL, "persistent engine: launched with %d registers per thread, too few for the split",
                fa.numRegs);
  a.h = c->at<float>(c->L.h);
  a.qkv = c->at<float>(c->L.qkv);
  a.attn = c->at<float>(c->L.attn);
  a.act = c->at<float>(c->L.act);
  a.logits = c->at<float>(c->L.logits);
  a.tok = c->at<int32_t>(c->L.tok);
  a.ctrl = c->at<int32_t>(c->L.ctrl);
  a.err = c->at<uint32_t>(c->L.err);
  a.mval = c->at<float>(c->L.mval);
  a.midx = c->at<int32_t>(c->L.midx);
  a.mcnt = c->at<uint32_t>(c->L.mcnt);
  a.ll_h = c->at<uint64_t>(c->L.ll_h);
  a.ll_qkv = c->at<uint64_t>(c->L.ll_qkv);
  a.ll_attn = c->at<uint64_t>(c->L.ll_attn);
  a.ll_act = c->at<uint64_t>(c->L.ll_act);
  a.ll_tok = c->at<uint64_t>(c->L.ll_tok);
  a.ll_apart = c->at<uint64_t>(c->L.ll_apart);
  a.kv_ready = c->at<uint32_t>(c->L.kv_ready);
  a.layers = c->at<MkLayer>(c->L.mk_layers);
  a.maps = c->ws + c->L.mk_maps;
  AttnArgs& at = a.at;
  at.qkv = a.qkv;
  at.eps = g.eps;
  at.rope_cos = c->at<float>(c->L.rope_cos);
  at.rope_sin = c->at<float>(c->L.rope_sin);
  at.ctrl = a.ctrl;
  at.kc = c->ws + c->L.kc;
  at.vc = c->ws + c->L.vc;
  at.max_seq = g.max_seq;
  at.n_q = g.n_q;
  at.n_kv = g.n_kv;
  at.d = g.head_dim;
  at.out = a.attn;
  at.part = c->at<float>(c->L.apart);
  at.counter = c->at<uint32_t>(c->L.acnt);
  at.nsplit_max = std::max(1, std::min(kSplitMax, G / g.n_kv));
  at.tmin = 64;
  at.scale = 1.0f / std::sqrt(static_cast<float>(g.head_dim));
  at.err = a.err;
  a.kv_layer_bytes = c->kv_layer_elems() * dtype_bytes(g.kvdtype);
  return DEC_OK;
}

// nsteps forwards at positions pos0.. in one cooperative launch.
void* q4p_kernel(const dec_config& g) {
  const bool g2 = g.n_q / g.n_kv <= 2;
  if (g.kvdtype == DEC_BF16)
    return g2 ? reinterpret_cast<void*>(q4_persist_kernel<uint16_t, 2>)
              : reinterpret_cast<void*>(q4_persist_kernel<uint16_t, 8>);
  return g2 ? reinterpret_cast<void*>(q4_persist_kernel<float, 2>) : reinterpret_cast<void*>(q4_persist_kernel<float, 8>);
}

// Plan the persistent 4-bit kernel: one CTA per SM, a ring of as many chunk
// stages as shared memory holds after the x planes and the attention scratch.
dec_status plan_q4_persistent(dec_ctx* c) {
  const dec_config& g = c->cfg;
  const int G = c->di.sms;
  const int qw = g.n_q * g.head_dim, kvw = g.n_kv * g.head_dim;
  const struct {
    int rows, in;
  } mats[8] = {{qw, g.hidden}, {kvw, g.hidden}, {g.hidden, qw}, {g.inter, g.hidden}, {g.hidden, g.inter},
               {g.vocab, g.hidden}, {kvw, g.hidden}, {g.inter, g.hidden}};
  size_t stage = 0;
  for (const auto& m : mats) {
    const long long rmax = std::min<long long>(kQ4pRC, (m.rows + G - 1) / G);
    stage = std::max(stage, static_cast<size_t>(rmax) * (m.in / 2 + m.in / 16));
  }
  stage = (stage + 127) / 128 * 128;
  const int in_max = std::max(g.hidden, std::max(qw, g.inter));
  const size_t fixed = static_cast<size_t>(in_max / 32) * (4 * 16 + 8) +
                       (attn_smem_bytes(g.n_q / g.n_kv, g.head_dim) + 15) / 16 * 16;
  void* k = q4p_kernel(g);
  cudaFuncAttributes fa{};
  WSG_CUDA_TRY(&c->err, cudaFuncGetAttributes(&fa, k));
  const long long budget = static_cast<long long>(c->di.smem_optin) - static_cast<long long>(fa.sharedSizeBytes) -
                           static_cast<long long>(fixed) - 1024;
  long long S = budget > 0 ? budget / static_cast<long long>(stage + 16) : 0;
  if (S > kQ4pMaxStages) S = kQ4pMaxStages;
  if (S < 2) return fail(&c->err, DEC_EINVAL, "persistent 4-bit engine: a %zu-byte chunk stage does not fit", stage);
  c->q4p_smem = static_cast<size_t>(S) * (stage + 16) + fixed;
  WSG_CUDA_TRY(&c->err, cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(c->q4p_smem)));
  int per_sm = 0;
  WSG_CUDA_TRY(&c->err, cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kQ4pThreads, c->q4p_smem));
  if (per_sm < 1) return fail(&c->err, DEC_EINVAL, "persistent 4-bit engine: no CTA fits on an SM");
  if (g.n_kv * c->nsplit_max > G) return fail(&c->err, DEC_EINVAL, "persistent 4-bit engine: attention CTAs exceed the grid");
  Q4PArgs& a = c->q4p;
  a = Q4PArgs{};
  a.layers = c->at<Q4PLayer>(c->L.q4layers);
  a.L = g.layers;
  a.H = g.hidden;
  a.I = g.inter;
  a.qw = qw;
  a.kvw = kvw;
  a.V = g.vocab;
  a.eps = g.eps;
  AttnArgs& at = a.at;
  at.eps = g.eps;
  at.rope_cos = c->at<float>(c->L.rope_cos);
  at.rope_sin = c->at<float>(c->L.rope_sin);
  at.kc = c->ws + c->L.kc;
  at.vc = c->ws + c->L.vc;
  at.max_seq = g.max_seq;
  at.n_q = g.n_q;
  at.n_kv = g.n_kv;
  at.d = g.head_dim;
  at.part = c->at<float>(c->L.apart);
  at.counter = c->at<uint32_t>(c->L.acnt);
  at.nsplit_max = c->nsplit_max;
  at.tmin = 64;
  at.scale = 1.0f / sqrtf(static_cast<float>(g.head_dim));
  at.err = c->at<uint32_t>(c->L.err);
  a.kv_layer_bytes = c->kv_layer_elems() * dtype_bytes(g.kvdtype);
  a.h = c->at<float>(c->L.h);
  a.qkv = c->at<float>(c->L.qkv);
  a.attn = c->at<float>(c->L.attn);
  a.gu = c->at<float>(c->L.q4gu);
  a.logits = c->at<float>(c->L.logits);
  a.mval = c->at<float>(c->L.mval);
  a.midx = c->at<int32_t>(c->L.midx);
  a.tok = c->at<int32_t>(c->L.tok);
  a.ctrl = c->at<int32_t>(c->L.ctrl);
  a.bar = c->at<unsigned long long>(c->L.q4bar);
  a.nstages = static_cast<int32_t>(S);
  a.stage_bytes = static_cast<uint32_t>(stage);
  a.attn_bytes = static_cast<uint32_t>((attn_smem_bytes(g.n_q / g.n_kv, g.head_dim) + 15) / 16 * 16);
  a.err = c->at<uint32_t>(c->L.err);
  return DEC_OK;
}

dec_status run_q4_persistent(dec_ctx* c, int pos0, int nsteps, bool head_every, bool head_last, int32_t first_tok,
                             int32_t* host_next) {
  Q4PArgs a = c->q4p;
  a.head = q4_seg(c->w.embed, c->cfg.vocab, c->cfg.hidden, 0);
  a.g_final = c->w.g_final;
  a.pos0 = pos0;
  a.nsteps = nsteps;
  a.head_every = head_every ? 1 : 0;
  a.head_last = head_last ? 1 : 0;
  a.first_tok = first_tok;
  a.host_next = host_next;
  a.xwait_ns = c->xwait_ns;
  a.trace = c->trace;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c->di.sms);
  cfg.blockDim = dim3(kQ4pThreads);
  cfg.dynamicSmemBytes = c->q4p_smem;
  cfg.stream = c->stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  WSG_CUDA_TRY(&c->err, cudaLaunchKernelExC(&cfg, q4p_kernel(c->cfg), args));
  return DEC_OK;
}

dec_status run_persistent(dec_ctx* c, int pos0, int nsteps, bool head_every, bool head_last, int32_t first_tok = -1,
                          int32_t* host_next = nullptr) {
  if (c->cfg.wdtype == DEC_Q4G64) return run_q4_persistent(c, pos0, nsteps, head_every, head_last, first_tok, host_next);
  MkArgs a = c->mk;
  a.first_tok = first_tok;
  a.host_next = host_next;
  a.embed = c->w.embed;
  a.g_final = c->w.g_final;
  a.pos0 = pos0;
  a.nsteps = nsteps;
  a.head_every = head_every ? 1 : 0;
  a.head_last = head_last ? 1 : 0;
  a.trace = c->trace;
  a.xwait_ns = c->xwait_ns;
  c->epoch = c->epoch % 4095 + 1;  // exchange tags never repeat between consecutive launches
  a.epoch = c->epoch;
  if (static_cast<long long>(nsteps) * (c->cfg.layers + 1) * 5 + 1 >= (1ll << 20))
    return fail(&c->err, DEC_EINVAL, "persistent engine: %d steps exceed one launch's tag space", nsteps);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c->mk_grid);
  cfg.blockDim = dim3(kMkThreads);
  cfg.dynamicSmemBytes = c->mk_smem;
  cfg.stream = c->stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  WSG_CUDA_TRY(&c->err, cudaLaunchKernelExC(&cfg, mk_kernel(c->cfg), args));
  return DEC_OK;
}

dec_status capture(dec_ctx* c, bool full, cudaGraphExec_t* out, int ntok = 1) {
  WSG_CUDA_TRY(&c->err, cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal));
  dec_status s = c->cfg.wdtype == DEC_Q4G64 ? enqueue_step_q4(c, c->cap, full, ntok)
                 : c->cfg.wdtype == DEC_F32 ? enqueue_step_t<float>(c, c->cap, full)
                                            : enqueue_step_t<uint16_t>(c, c->cap, full);
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(c->cap, &graph);
  if (s != DEC_OK) {
    if (graph) cudaGraphDestroy(graph);
    return s;
  }
  if (e != cudaSuccess) return fail(&c->err, DEC_ECUDA, "graph capture failed: %s", cudaGetErrorString(e));
  e = cudaGraphInstantiate(out, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return fail(&c->err, DEC_ECUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
  return DEC_OK;
}

dec_status ensure_graphs(dec_ctx* c, bool full) {
  if (full && !c->g_full) return capture(c, true, &c->g_full);
  if (!full && !c->g_body) return capture(c, false, &c->g_body);
  return DEC_OK;
}

dec_status run_steps(dec_ctx* c, bool full, int n) {
  dec_status s = ensure_graphs(c, full);
  if (s != DEC_OK) return s;
  for (int i = 0; i < n; ++i) WSG_CUDA_TRY(&c->err, cudaGraphLaunch(full ? c->g_full : c->g_body, c->stream));
  return DEC_OK;
}

dec_status put_tokens(dec_ctx* c, const int32_t* toks, int n) {
  for (int i = 0; i < n; ++i) {
    if (toks[i] < 0 || toks[i] >= c->cfg.vocab)
      return fail(&c->err, DEC_EINVAL, "token %d at row %d is outside [0, %d)", toks[i], i, c->cfg.vocab);
  }
  std::memcpy(c->h_tok + c->pos, toks, sizeof(int32_t) * n);
  WSG_CUDA_TRY(&c->err, cudaMemcpyAsync(c->at<int32_t>(c->L.tok) + c->pos, c->h_tok + c->pos, sizeof(int32_t) * n,
                                        cudaMemcpyHostToDevice, c->stream));
  return DEC_OK;
}

dec_status finish_head(dec_ctx* c, int32_t last_pos, float* d_logits, int32_t* h_next) {
  if (d_logits)
    WSG_CUDA_TRY(&c->err, cudaMemcpyAsync(d_logits, c->at<float>(c->L.logits), sizeof(float) * c->cfg.vocab,
                                          cudaMemcpyDeviceToDevice, c->stream));
  if (h_next) {
    WSG_CUDA_TRY(&c->err, cudaMemcpyAsync(c->h_next, c->at<int32_t>(c->L.tok) + last_pos + 1, sizeof(int32_t),
                                          cudaMemcpyDeviceToHost, c->stream));
    WSG_CUDA_TRY(&c->err, cudaStreamSynchronize(c->stream));
    *h_next = *c->h_next;
  }
  return DEC_OK;
}

}  // namespace

extern "C" size_t dec_workspace_bytes(const dec_config* cfg) {
  if (!config_ok(cfg, nullptr)) return 0;
  return make_layout(*cfg).total;
}

extern "C" dec_status dec_create(const dec_config* cfg, void* d_workspace, size_t workspace_bytes, void* stream,
                                 dec_ctx** out) {
  std::string why;
  if (!out) return fail(nullptr, DEC_EINVAL, "dec_create: NULL output handle");
  *out = nullptr;
  if (!config_ok(cfg, &why)) return fail(nullptr, DEC_EINVAL, "dec_create: %s", why.c_str());
  if (!d_workspace || (reinterpret_cast<uintptr_t>(d_workspace) % kAlign))
    return fail(nullptr, DEC_EINVAL, "dec_create: workspace must be non-NULL and 256-byte aligned");
  const Layout L = make_layout(*cfg);
  if (workspace_bytes < L.total)
    return fail(nullptr, DEC_ENOMEM, "dec_create: workspace has %zu bytes, %zu needed", workspace_bytes, L.total);
  DeviceInfo di;
  dec_status s = device_info(&di, nullptr);
  if (s != DEC_OK) return s;

  dec_ctx* c = new (std::nothrow) dec_ctx();
  if (!c) return fail(nullptr, DEC_ENOMEM, "dec_create: out of host memory");
  c->cfg = *cfg;
  c->di = di;
  c->ws = static_cast<char*>(d_workspace);
  c->ws_bytes = workspace_bytes;
  c->L = L;
  c->stream = static_cast<cudaStream_t>(stream);
  auto bail = [&](dec_status st) {
    dec_destroy(c);
    return st;
  };
  cudaError_t e = cudaStreamCreateWithFlags(&c->cap, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaMallocHost(&c->h_tok, sizeof(int32_t) * (cfg->max_seq + 1));
  if (e == cudaSuccess) e = cudaHostAlloc(&c->h_next, 2 * sizeof(int32_t), cudaHostAllocMapped);
  if (e == cudaSuccess) e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->d_h_next), c->h_next, 0);
  if (e != cudaSuccess) return bail(fail(nullptr, DEC_ECUDA, "dec_create: %s", cudaGetErrorString(e)));

  // Rotary table: angle = p * theta^(-2i/d), evaluated in double, stored float32.
  const int half = cfg->head_dim / 2;
  std::vector<float> cs(static_cast<size_t>(cfg->max_seq) * half), sn(cs.size());
  for (int i = 0; i < half; ++i) {
    const double inv = std::pow(static_cast<double>(cfg->rope_theta), -2.0 * i / cfg->head_dim);
    for (int p = 0; p < cfg->max_seq; ++p) {
      const double ang = static_cast<double>(p) * inv;
      cs[static_cast<size_t>(p) * half + i] = static_cast<float>(std::cos(ang));
      sn[static_cast<size_t>(p) * half + i] = static_cast<float>(std::sin(ang));
    }
  }
  e = cudaMemcpy(c->ws + L.rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(c->ws + L.rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(c->ws, 0, L.rope_cos);           // control, activations, partials
  if (e == cudaSuccess) e = cudaMemset(c->ws + L.kc, 0, L.total - L.kc);  // caches
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return bail(fail(nullptr, DEC_ECUDA, "dec_create: %s", cudaGetErrorString(e)));

  const int welem = static_cast<int>(dtype_bytes(cfg->wdtype));
  const int qw = cfg->n_q * cfg->head_dim, kvw = cfg->n_kv * cfg->head_dim;
  c->p_qkv = plan_gemv(qw + 2 * kvw, cfg->hidden, welem, 1, di.sms, di.sms);
  c->p_o = plan_gemv(cfg->hidden, qw, welem, 1, di.sms, di.sms);
  c->p_gu = plan_gemv(2 * cfg->inter, cfg->hidden, welem, 2, di.sms, di.sms);
  c->p_down = plan_gemv(cfg->hidden, cfg->inter, welem, 1, di.sms, di.sms);
  c->p_vocab = plan_gemv(cfg->vocab, cfg->hidden, welem, 1, di.sms, kArgmaxPartsMax);
  for (const Plan* p : {&c->p_qkv, &c->p_o, &c->p_gu, &c->p_down, &c->p_vocab})
    if (p->smem > di.smem_optin)
      return bail(fail(nullptr, DEC_EINVAL, "dec_create: a projection needs %zu B of shared memory (max %zu)", p->smem,
                       di.smem_optin));
  c->attn_smem = attn_smem_bytes(cfg->n_q / cfg->n_kv, cfg->head_dim);
  if (L.pf_rows > 0) {
    const dec_status ms[6] = {
        encode_gemm_operand(c->pf_amap[0].b, c->ws + L.pf_ah, L.pf_rows, cfg->hidden, 128, &c->err),
        encode_gemm_operand(c->pf_amap[1].b, c->ws + L.pf_ao, L.pf_rows, qw, 128, &c->err),
        encode_gemm_operand(c->pf_amap[2].b, c->ws + L.pf_ai, L.pf_rows, cfg->inter, 128, &c->err),
        encode_gemm_operand(c->pf_amap[3].b, c->ws + L.pf_ah2, L.pf_rows, cfg->hidden, 128, &c->err),
        encode_gemm_operand(c->pf_amap[4].b, c->ws + L.pf_ao2, L.pf_rows, qw, 128, &c->err),
        encode_gemm_operand(c->pf_amap[5].b, c->ws + L.pf_ai2, L.pf_rows, cfg->inter, 128, &c->err)};
    for (dec_status m : ms)
      if (m != DEC_OK) {
        thread_error() = c->err;
        return bail(m);
      }
    const long long kv_rows = static_cast<long long>(cfg->layers) * cfg->n_kv * cfg->max_seq;
    if (cfg->kvdtype == DEC_BF16 && cfg->head_dim == kAtD && kAtBM % (cfg->n_q / cfg->n_kv) == 0 &&
        kv_rows + kAtBN < (1ll << 31)) {
      for (int i = 0; i < 2; ++i) {
        const dec_status m = encode_map_2d(c->pf_kvmap[i].b, c->ws + (i ? L.vc : L.kc), kv_rows, kAtD, 2, 64, kAtBN,
                                           true, &c->err);
        if (m != DEC_OK) {
          thread_error() = c->err;
          return bail(m);
        }
      }
      c->pf_attn_tmem = true;
    }
  }
  c->nsplit_max = di.sms / cfg->n_kv;
  if (c->nsplit_max < 1) c->nsplit_max = 1;
  if (c->nsplit_max > kSplitMax) c->nsplit_max = kSplitMax;
  s = cfg->wdtype == DEC_F32 ? prepare_kernels<float>(c) : prepare_kernels<uint16_t>(c);
  if (s == DEC_OK && cfg->engine == DEC_ENGINE_PERSISTENT)
    s = cfg->wdtype == DEC_Q4G64 ? plan_q4_persistent(c) : plan_persistent(c);
  if (s != DEC_OK) {
    thread_error() = c->err;
    return bail(s);
  }
  *out = c;
  return DEC_OK;
}

extern "C" dec_status dec_load_weights(dec_ctx* c, const dec_weights* w) {
  if (!c) return fail(nullptr, DEC_EINVAL, "dec_load_weights: NULL context");
  if (!w || !w->embed || !w->g_final || !w->layers) return fail(&c->err, DEC_EINVAL, "dec_load_weights: NULL pointer");
  auto ok = [](const void* p) { return p && aligned16(p); };
  if (!ok(w->embed) || !ok(w->g_final)) return fail(&c->err, DEC_EINVAL, "dec_load_weights: embed/g_final misaligned");
  for (int l = 0; l < c->cfg.layers; ++l) {
    const dec_layer_weights& x = w->layers[l];
    const void* ps[] = {x.w_q, x.w_k, x.w_v, x.w_o, x.w_gate, x.w_up, x.w_down, x.g_in, x.g_post, x.g_q, x.g_k};
    for (const void* p : ps)
      if (!ok(p)) return fail(&c->err, DEC_EINVAL, "dec_load_weights: layer %d has a NULL or misaligned tensor", l);
  }
  c->layers.assign(w->layers, w->layers + c->cfg.layers);
  c->w = *w;
  c->w.layers = c->layers.data();
  std::vector<MkLayer> tab(c->cfg.layers);
  for (int l = 0; l < c->cfg.layers; ++l) {
    const dec_layer_weights& x = c->layers[l];
    tab[l] = MkLayer{x.w_q, x.w_k, x.w_v, x.w_o, x.w_gate, x.w_up, x.w_down, x.g_in, x.g_post, x.g_q, x.g_k};
  }
  WSG_CUDA_TRY(&c->err, cudaMemcpyAsync(c->ws + c->L.mk_layers, tab.data(), tab.size() * sizeof(MkLayer),
                                        cudaMemcpyHostToDevice, c->stream));
  if (c->cfg.wdtype == DEC_Q4G64 && c->cfg.engine == DEC_ENGINE_PERSISTENT) {
    // the persistent 4-bit kernel's layer table: each matrix as (codes, scales, biases, rows)
    const dec_config& g = c->cfg;
    const int qw = g.n_q * g.head_dim, kvw = g.n_kv * g.head_dim;
    std::vector<Q4PLayer> q4t(g.layers);
    for (int l = 0; l < g.layers; ++l) {
      const dec_layer_weights& x = c->layers[l];
      q4t[l] = Q4PLayer{q4_seg(x.w_q, qw, g.hidden, 0),       q4_seg(x.w_k, kvw, g.hidden, 0),
                        q4_seg(x.w_v, kvw, g.hidden, 0),      q4_seg(x.w_o, g.hidden, qw, 0),
                        q4_seg(x.w_gate, g.inter, g.hidden, 0), q4_seg(x.w_up, g.inter, g.hidden, 0),
                        q4_seg(x.w_down, g.hidden, g.inter, 0), x.g_in, x.g_post, x.g_q, x.g_k};
    }
    WSG_CUDA_TRY(&c->err, cudaMemcpyAsync(c->ws + c->L.q4layers, q4t.data(), q4t.size() * sizeof(Q4PLayer),
                                          cudaMemcpyHostToDevice, c->stream));
    WSG_CUDA_TRY(&c->err, cudaStreamSynchronize(c->stream));
  }
  std::vector<CUtensorMap> maps;
  if (c->cfg.engine == DEC_ENGINE_PERSISTENT && c->cfg.wdtype != DEC_Q4G64) {
    // Tiled-copy descriptors of every weight matrix for the persistent engine.
    const dec_config& g = c->cfg;
    const int qw = g.n_q * g.head_dim, kvw = g.n_kv * g.head_dim;
    maps.resize(static_cast<size_t>(g.layers) * kMkMapsPerLayer + 1);
    for (int l = 0; l < g.layers; ++l) {
      const dec_layer_weights& x = c->layers[l];
      CUtensorMap* m = maps.data() + static_cast<size_t>(l) * kMkMapsPerLayer;
      const struct {
        const void* p;
        int rows, in;
        const MkGeom* gm;
      } t[kMkMapsPerLayer] = {{x.w_q, qw, g.hidden, &c->mk.gq},     {x.w_k, kvw, g.hidden, &c->mk.gq},
                              {x.w_v, kvw, g.hidden, &c->mk.gq},    {x.w_o, g.hidden, qw, &c->mk.go},
                              {x.w_gate, g.inter, g.hidden, &c->mk.gg}, {x.w_up, g.inter, g.hidden, &c->mk.gg},
                              {x.w_down, g.hidden, g.inter, &c->mk.gd}};
      for (int k = 0; k < kMkMapsPerLayer; ++k) {
        const dec_status st = encode_map(m + k, t[k].p, t[k].rows, t[k].in, g.wdtype, *t[k].gm, &c->err);
        if (st != DEC_OK) return st;
      }
    }
    const dec_status st = encode_map(maps.data() + maps.size() - 1, c->w.embed, g.vocab, g.hidden, g.wdtype, c->mk.gv, &c->err);
    if (st != DEC_OK) return st;
    static_assert(sizeof(CUtensorMap) == kMkMapBytes, "tensor map size");
    WSG_CUDA_TRY(&c->err, cudaMemcpyAsync(c->ws + c->L.mk_maps, maps.data(), maps.size() * sizeof(CUtensorMap),
                                          cudaMemcpyHostToDevice, c->stream));
  }
  if (c->L.pf_rows > 0) {
    // Tensor-core GEMM operand maps of every weight matrix (chunked prefill).
    const dec_config& g = c->cfg;
    const int qw = g.n_q * g.head_dim, kvw = g.n_kv * g.head_dim;
    c->pf_wmap256.resize(static_cast<size_t>(g.layers) * kMkMapsPerLayer);
    c->pf_wmap.resize(static_cast<size_t>(g.layers) * kMkMapsPerLayer);
    c->pf_wmap64.resize(static_cast<size_t>(g.layers) * kMkMapsPerLayer);
    for (int l = 0; l < g.layers; ++l) {
      const dec_layer_weights& x = c->layers[l];
      const struct {
        const void* p;
        int rows, K;
      } t[kMkMapsPerLayer] = {{x.w_q, qw, g.hidden},    {x.w_k, kvw, g.hidden},      {x.w_v, kvw, g.hidden},
                              {x.w_o, g.hidden, qw},    {x.w_gate, g.inter, g.hidden}, {x.w_up, g.inter, g.hidden},
                              {x.w_down, g.hidden, g.inter}};
      for (int k = 0; k < kMkMapsPerLayer; ++k) {
        const size_t i = static_cast<size_t>(l) * kMkMapsPerLayer + k;
        dec_status st = encode_gemm_operand(c->pf_wmap256[i].b, t[k].p, t[k].rows, t[k].K, 256, &c->err);
        if (st == DEC_OK) st = encode_gemm_operand(c->pf_wmap[i].b, t[k].p, t[k].rows, t[k].K, 128, &c->err);
        if (st == DEC_OK) st = encode_gemm_operand(c->pf_wmap64[i].b, t[k].p, t[k].rows, t[k].K, 64, &c->err);
        if (st != DEC_OK) return st;
      }
    }
  }
  WSG_CUDA_TRY(&c->err, cudaStreamSynchronize(c->stream));
  // Graphs bake in the weight pointers: drop any captured with older ones.
  if (c->g_full) cudaGraphExecDestroy(c->g_full);
  if (c->g_body) cudaGraphExecDestroy(c->g_body);
  if (c->g_verify) cudaGraphExecDestroy(c->g_verify);
  c->g_full = c->g_body = c->g_verify = nullptr;
  c->have_weights = true;
  return DEC_OK;
}

extern "C" dec_status dec_reset(dec_ctx* c) {
  if (!c) return fail(nullptr, DEC_EINVAL, "dec_reset: NULL context");
  // Earlier asynchronous copies may still read the pinned token slots.
  WSG_CUDA_TRY(&c->err, cudaStreamSynchronize(c->stream));
  c->pos = 0;
  // control words, counters, activations and partials (everything before the layer table)
  WSG_CUDA_TRY(&c->err, cudaMemsetAsync(c->ws, 0, c->L.mk_layers, c->stream));
  WSG_CUDA_TRY(&c->err, cudaMemsetAsync(c->ws + c->L.kc, 0, c->L.total - c->L.kc, c->stream));
  return DEC_OK;
}

extern "C" dec_status dec_set_wait_limit(dec_ctx* c, uint64_t ns) {
  if (!c) return fail(nullptr, DEC_EINVAL, "dec_set_wait_limit: NULL context");
  c->xwait_ns = ns == 0 ? WSG_WAIT_LIMIT_NS : ns;
  return DEC_OK;
}

extern "C" dec_status dec_rewind(dec_ctx* c, int32_t pos) {
  if (!c) return fail(nullptr, DEC_EINVAL, "dec_rewind: NULL context");
  if (pos < 0 || pos > c->pos) return fail(&c->err, DEC_EINVAL, "dec_rewind: position %d outside [0, %d]", pos, c->pos);
  c->pos = pos;
  // The position word, and (persistent engine) the appended-row counts its
  // attention waits on: rows below pos stay valid, rows from pos on are
  // rewritten before anything reads them.
  uint32_t* kvr = c->cfg.engine == DEC_ENGINE_PERSISTENT ? c->at<uint32_t>(c->L.kv_ready) : nullptr;
  pf_control_kernel<<<1, 256, 0, c->stream>>>(c->at<int32_t>(c->L.ctrl), pos, kvr, c->cfg.layers * c->cfg.n_kv,
                                              static_cast<uint32_t>(pos));
  WSG_CUDA_TRY(&c->err, cudaGetLastError());
  return DEC_OK;
}

extern "C" dec_status dec_step(dec_ctx* c, int32_t token, uint32_t flags, float* d_logits, int32_t* h_next) {
  if (!c) return fail(nullptr, DEC_EINVAL, "dec_step: NULL context");
  if (flags & ~DEC_SKIP_LOGITS) return fail(&c->err, DEC_EINVAL, "dec_step: unknown flags 0x%x", flags);
  const bool full = !(flags & DEC_SKIP_LOGITS);
  if (!full && (d_logits || h_next))
    return fail(&c->err, DEC_EINVAL, "dec_step: DEC_SKIP_LOGITS with a logits or token output");
  if (!c->have_weights) return fail(&c->err, DEC_ESTATE, "dec_step: weights not loaded");
  if (c->pos >= c->cfg.max_seq)
    return fail(&c->err, DEC_ECAPACITY, "dec_step: position %d reached max_seq %d", c->pos, c->cfg.max_seq);
  const bool persistent = c->cfg.engine == DEC_ENGINE_PERSISTENT;
  dec_status s = persistent ? DEC_OK : ensure_graphs(c, full);
  if (s != DEC_OK) return s;
  if (token < 0 || token >= c->cfg.vocab)
    return fail(&c->err, DEC_EINVAL, "token %d is outside [0, %d)", token, c->cfg.vocab);
  const int32_t p = c->pos;
  if (persistent) {
    // The token goes in with the launch and the greedy token comes back through
    // mapped host memory: no copies around the kernel.
    c->h_tok[p] = token;
    int32_t* hn = nullptr;
    if (full && h_next) {
      *c->h_next = -1;
      hn = c->d_h_next;
    }
    if ((s = run_persistent(c, p, 1, full, false, token, hn)) != DEC_OK) return s;
    c->pos += 1;
    if (!full) return DEC_OK;
    if (d_logits)
      WSG_CUDA_TRY(&c->err, cudaMemcpyAsync(d_logits, c->at<float>(c->L.logits), sizeof(float) * c->cfg.vocab,
                                            cudaMemcpyDeviceToDevice, c->stream));
    if (h_next) {
      WSG_CUDA_TRY(&c->err, cudaStreamSynchronize(c->stream));
      *h_next = *static_cast<volatile int32_t*>(c->h_next);
    }
    return DEC_OK;
  }
  if ((s = put_tokens(c, &token, 1)) != DEC_OK) return s;
  if ((s = run_steps(c, full, 1)) != DEC_OK) return s;
  c->pos += 1;
  if (full) return finish_head(c, p, d_logits, h_next);
  return DEC_OK;
}

extern "C" dec_status dec_prefill_chunk(dec_ctx* c, const int32_t* h_tokens, int32_t n, int32_t is_last,
                                        float* d_logits, int32_t* h_next) {
  if (!c) return fail(nullptr, DEC_EINVAL, "dec_prefill_chunk: NULL context");
  if (!h_tokens || n < 1) return fail(&c->err, DEC_EINVAL, "dec_prefill_chunk: need n >= 1 tokens");
  if (!is_last && (d_logits || h_next))
    return fail(&c->err, DEC_EINVAL, "dec_prefill_chunk: outputs requested from a non-final chunk");
  if (!c->have_weights) return fail(&c->err, DEC_ESTATE, "dec_prefill_chunk: weights not loaded");
  if (static_cast<long long>(c->pos) + n > c->cfg.max_seq)
    return fail(&c->err, DEC_ECAPACITY, "dec_prefill_chunk: %d rows at position %d exceed max_seq %d", n, c->pos,
                c->cfg.max_seq);
  if (c->cfg.chunk_cap > 0 && n <= c->cfg.chunk_cap) {  // batched: tensor-core projections
    dec_status s = put_tokens(c, h_tokens, n);
    if (s != DEC_OK) return s;
    const int32_t p0 = c->pos;
    if ((s = run_chunk_prefill(c, p0, n, is_last != 0)) != DEC_OK) return s;
    c->pos += n;
    if (is_last) return finish_head(c, p0 + n - 1, d_logits, h_next);
    return DEC_OK;
  }
  const bool persistent = c->cfg.engine == DEC_ENGINE_PERSISTENT;
  dec_status s = DEC_OK;
  if (!persistent) {
    s = ensure_graphs(c, false);
    if (s == DEC_OK && is_last) s = ensure_graphs(c, true);
  }
  if (s != DEC_OK) return s;
  if ((s = put_tokens(c, h_tokens, n)) != DEC_OK) return s;
  const int32_t p0 = c->pos;
  if (persistent) {
    if ((s = run_persistent(c, p0, n, false, is_last != 0)) != DEC_OK) return s;
  } else {
    const int body = is_last ? n - 1 : n;
    if ((s = run_steps(c, false, body)) != DEC_OK) return s;
    if (is_last && (s = run_steps(c, true, 1)) != DEC_OK) return s;
  }
  c->pos += n;
  if (is_last) return finish_head(c, p0 + n - 1, d_logits, h_next);
  return DEC_OK;
}

extern "C" dec_status dec_verify2(dec_ctx* c, const int32_t* h_tokens, float* d_logits, int32_t* h_next) {
  if (!c) return fail(nullptr, DEC_EINVAL, "dec_verify2: NULL context");
  if (!h_tokens) return fail(&c->err, DEC_EINVAL, "dec_verify2: NULL tokens");
  if (c->cfg.wdtype != DEC_Q4G64) return fail(&c->err, DEC_EINVAL, "dec_verify2: needs the 4-bit configuration");
  if (!c->have_weights) return fail(&c->err, DEC_ESTATE, "dec_verify2: weights not loaded");
  if (c->pos + 2 > c->cfg.max_seq)
    return fail(&c->err, DEC_ECAPACITY, "dec_verify2: positions %d, %d exceed max_seq %d", c->pos, c->pos + 1,
                c->cfg.max_seq);
  if (!c->g_verify) {
    const dec_status s = capture(c, true, &c->g_verify, 2);
    if (s != DEC_OK) return s;
  }
  dec_status s = put_tokens(c, h_tokens, 2);
  if (s != DEC_OK) return s;
  WSG_CUDA_TRY(&c->err, cudaGraphLaunch(c->g_verify, c->stream));
  c->pos += 2;
  if (d_logits)
    WSG_CUDA_TRY(&c->err, cudaMemcpyAsync(d_logits, c->at<float>(c->L.logits), 2 * sizeof(float) * c->cfg.vocab,
                                          cudaMemcpyDeviceToDevice, c->stream));
  if (h_next) {
    WSG_CUDA_TRY(&c->err, cudaMemcpyAsync(c->h_next, c->at<int32_t>(c->L.q4next), 2 * sizeof(int32_t),
                                          cudaMemcpyDeviceToHost, c->stream));
    WSG_CUDA_TRY(&c->err, cudaStreamSynchronize(c->stream));
    h_next[0] = c->h_next[0];
    h_next[1] = c->h_next[1];
  }
  return DEC_OK;
}

extern "C" dec_status dec_generate(dec_ctx* c, int32_t token, int32_t n, int32_t* d_tokens_out) {
  if (!c) return fail(nullptr, DEC_EINVAL, "dec_generate: NULL context");
  if (n < 1 || !d_tokens_out) return fail(&c->err, DEC_EINVAL, "dec_generate: need n >= 1 and an output buffer");
  if (!c->have_weights) return fail(&c->err, DEC_ESTATE, "dec_generate: weights not loaded");
  if (static_cast<long long>(c->pos) + n > c->cfg.max_seq)
    return fail(&c->err, DEC_ECAPACITY, "dec_generate: %d steps at position %d exceed max_seq %d", n, c->pos,
                c->cfg.max_seq);
  const bool persistent = c->cfg.engine == DEC_ENGINE_PERSISTENT;
  dec_status s = persistent ? DEC_OK : ensure_graphs(c, true);
  if (s != DEC_OK) return s;
  if ((s = put_tokens(c, &token, 1)) != DEC_OK) return s;
  s = persistent ? run_persistent(c, c->pos, n, true, false) : run_steps(c, true, n);
  if (s != DEC_OK) return s;
  WSG_CUDA_TRY(&c->err, cudaMemcpyAsync(d_tokens_out, c->at<int32_t>(c->L.tok) + c->pos + 1, sizeof(int32_t) * n,
                                        cudaMemcpyDeviceToDevice, c->stream));
  c->pos += n;
  return DEC_OK;
}

extern "C" dec_status dec_get_kv(const dec_ctx* c, int32_t layer, const void** d_k, const void** d_v,
                                 int32_t* n_valid) {
  if (!c) return fail(nullptr, DEC_EINVAL, "dec_get_kv: NULL context");
  if (layer < 0 || layer >= c->cfg.layers) return fail(nullptr, DEC_EINVAL, "dec_get_kv: layer %d", layer);
  const size_t off = static_cast<size_t>(layer) * c->kv_layer_elems() * dtype_bytes(c->cfg.kvdtype);
  if (d_k) *d_k = c->ws + c->L.kc + off;
  if (d_v) *d_v = c->ws + c->L.vc + off;
  if (n_valid) *n_valid = c->pos;
  return DEC_OK;
}

extern "C" int32_t dec_position(const dec_ctx* c) { return c ? c->pos : -1; }

extern "C" size_t dec_trace_bytes(const dec_ctx* c) {
  if (!c || c->cfg.engine != DEC_ENGINE_PERSISTENT) return 0;
  const size_t G = c->cfg.wdtype == DEC_Q4G64 ? static_cast<size_t>(c->di.sms) : static_cast<size_t>(c->mk_grid);
  return (G * (c->cfg.layers + 1) * kMkTraceStages * kMkTraceEvents +
          static_cast<size_t>(kMkWarps) * kMkTraceSegs * kMkTraceSegEvents) *
         sizeof(uint64_t);
}

extern "C" dec_status dec_set_trace(dec_ctx* c, uint64_t* d_trace, size_t bytes) {
  if (!c) return fail(nullptr, DEC_EINVAL, "dec_set_trace: NULL context");
  if (c->cfg.engine != DEC_ENGINE_PERSISTENT)
    return fail(&c->err, DEC_EINVAL, "dec_set_trace: tracing records the persistent engine only");
  if (d_trace && bytes < dec_trace_bytes(c))
    return fail(&c->err, DEC_EINVAL, "dec_set_trace: buffer has %zu bytes, %zu needed", bytes, dec_trace_bytes(c));
  c->trace = d_trace;
  return DEC_OK;
}

extern "C" dec_status dec_device_errors(dec_ctx* c, int32_t clear, uint32_t* bits) {
  if (!c || !bits) return fail(nullptr, DEC_EINVAL, "dec_device_errors: NULL argument");
  WSG_CUDA_TRY(&c->err, cudaStreamSynchronize(c->stream));
  WSG_CUDA_TRY(&c->err, cudaMemcpy(bits, c->ws + c->L.err, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  if (clear) WSG_CUDA_TRY(&c->err, cudaMemset(c->ws + c->L.err, 0, sizeof(uint32_t)));
  return DEC_OK;
}

extern "C" void dec_destroy(dec_ctx* c) {
  if (!c) return;
  if (c->stream || c->cap) cudaStreamSynchronize(c->stream);
  if (c->g_full) cudaGraphExecDestroy(c->g_full);
  if (c->g_verify) cudaGraphExecDestroy(c->g_verify);
  if (c->g_body) cudaGraphExecDestroy(c->g_body);
  if (c->cap) cudaStreamDestroy(c->cap);
  if (c->h_tok) cudaFreeHost(c->h_tok);
  if (c->h_next) cudaFreeHost(c->h_next);
  delete c;
}

extern "C" const char* dec_last_error(const dec_ctx* c) {
  if (c) return c->err.c_str();
  return thread_error().c_str();
}
