/*
 * wsg.h - C ABI of the weight-streaming decode library (GB300, sm_103a).
 *
 * The library computes the batch-1 token-to-logits forward of a
 * Qwen3-shaped decoder and the standalone matrix-vector products that
 * dominate it. All arithmetic runs in this library's CUDA kernels.
 *
 * Sources (page title, section):
 *   "Megakernels", "What runs in the DSL": the forward pass
 *       token ID -> embedding; per layer RMSNorm -> Q/K/V projections ->
 *       per-head Q/K RMSNorm -> RoPE -> grouped-query attention + KV update
 *       -> output projection -> residual add -> RMSNorm -> gate/up
 *       projections -> SwiGLU -> down projection -> residual add; then final
 *       RMSNorm -> tied vocabulary projection -> logits.
 *   "Megakernels", "GPU-wide end-to-end generation": greedy argmax on the
 *       GPU with ties broken by lowest token ID; the host reads the ID;
 *       prompt tokens processed one at a time skip only the final norm and
 *       vocabulary projection; the first output comes from the final prompt
 *       row.
 *   "Megakernels", "Chunked prefill for long prompts": a chunk is a run of
 *       consecutive positions of the single request; every row attends to
 *       its whole causal prefix; only the final valid row reaches the
 *       vocabulary projection.
 *   "Our Kernel Benchmark Was Measuring the System Cache", "Summary": the
 *       4-bit matrix-vector product and its two-token variant.
 *
 * Conventions for every call:
 *   - Pointers named d_* are device pointers, h_* host pointers. All device
 *     memory belongs to the caller; the library never frees it.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream. Calls are asynchronous on that stream unless stated.
 *   - Every call returns a dec_status. On failure nothing has been enqueued
 *     and dec_last_error() describes the cause. No call aborts the process.
 *   - Device-side problems that can only be seen while kernels run (a token
 *     ID outside the vocabulary, an all-NaN logit vector, a bounded wait
 *     that gave up) set bits of a device error word, read with
 *     dec_device_errors() or gemv_device_errors().
 */
#ifndef WSG_H
#define WSG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DEC_OK = 0,
  DEC_EINVAL = 1,     /* bad argument: NULL, size, alignment, dtype */
  DEC_ESTATE = 2,     /* call out of order (e.g. step before weights) */
  DEC_ECAPACITY = 3,  /* position or chunk beyond the configured capacity */
  DEC_ENOMEM = 4,     /* workspace too small, or a host allocation failed */
  DEC_ECUDA = 5,      /* a CUDA runtime call failed (message has the name) */
  DEC_EDEVICE = 6     /* device is not an sm_103 GPU */
} dec_status;

typedef enum { DEC_F32 = 0, DEC_BF16 = 1, DEC_Q4G64 = 2 } dec_dtype;

/* Device error bits (dec_device_errors / gemv_device_errors). */
#define DEC_DEVERR_WAIT_TIMEOUT 0x1u /* a bounded mbarrier wait gave up */
#define DEC_DEVERR_ARGMAX_NAN 0x2u   /* all logits NaN; token 0 was returned */
#define DEC_DEVERR_BAD_TOKEN 0x4u    /* a token ID outside [0, vocab) was read as 0 */
#define DEC_DEVERR_BAD_POSITION 0x8u /* a position reached the KV capacity; the step did nothing */
#define DEC_DEVERR_EXCHANGE_TIMEOUT 0x10u /* persistent engine: a wait for another CTA's words gave up */
#define DEC_DEVERR_GEMM_TIMEOUT 0x20u     /* chunked prefill: a tensor-core GEMM pipeline wait gave up */
#define DEC_DEVERR_BARRIER_TIMEOUT 0x40u  /* persistent 4-bit engine: a grid barrier gave up (dec_reset clears it) */

/* dec_config.engine */
#define DEC_ENGINE_PERSISTENT 0 /* one cooperative launch runs whole forwards (default) */
#define DEC_ENGINE_STAGED 1     /* five kernels per layer, replayed as a CUDA graph */

/* dec_step flags */
#define DEC_SKIP_LOGITS 0x1u /* body only: no final norm, vocabulary projection or argmax */

/* Decoder geometry and storage ("Megakernels", "What runs in the DSL").
 * Requirements: layers, hidden, inter, n_q, n_kv, head_dim, vocab > 0;
 * n_q % n_kv == 0; head_dim a multiple of 8 and <= 128; hidden, inter and
 * n_q*head_dim multiples of 8; wdtype DEC_F32, DEC_BF16 or DEC_Q4G64 (the
 * 4-bit configuration: chunk_cap 0, hidden, inter and n_q*head_dim
 * multiples of 512 up to 16384; its persistent engine separates stages
 * with grid barriers, and its staged engine is the faster of the two);
 * kvdtype DEC_F32
 * or DEC_BF16; max_seq >= 1 is the KV capacity in positions; chunk_cap is
 * the largest row count of one dec_prefill_chunk call that runs batched
 * (0: prompts are processed one token at a time). engine selects the
 * execution of decode steps: DEC_ENGINE_PERSISTENT runs each call's forwards
 * inside one persistent kernel (one CTA per SM, a producer warp streaming
 * weights through shared memory ahead of the consumers, grid barriers
 * between dependent stages); DEC_ENGINE_STAGED launches the per-stage
 * kernels as a CUDA graph. Both compute the same forward. Decode attention
 * at position p splits the p + 1 cached keys of each key/value head into
 * nsplit = min(ceil((p + 1) / 64), min(64, SMs / n_kv)) key-parallel ranges
 * of ceil((p + 1) / nsplit) keys (the last one shorter), whose partial
 * softmax sums are merged in split order. */
typedef struct {
  int32_t layers, hidden, inter, n_q, n_kv, head_dim, vocab;
  float eps;        /* RMSNorm epsilon, e.g. 1e-6 */
  float rope_theta; /* RoPE base, e.g. 1e6 */
  int32_t wdtype;   /* dec_dtype of projections and the tied embedding */
  int32_t kvdtype;  /* dec_dtype of the KV cache */
  int32_t max_seq;
  int32_t chunk_cap;
  int32_t engine;   /* DEC_ENGINE_*: how steps are executed */
} dec_config;

/* One layer's tensors, device pointers, row-major [out][in] in wdtype.
 * With DEC_Q4G64 each matrix pointer (and embed) points at one buffer
 * holding the codes [out][in/8] uint32 (code j of word w at bits
 * [4j, 4j+4), column 8w+j), then the scales and then the biases
 * [out][in/64] fp16: w = s * q + b per 64-column group.
 * w_q [n_q*head_dim][hidden], w_k and w_v [n_kv*head_dim][hidden],
 * w_o [hidden][n_q*head_dim], w_gate and w_up [inter][hidden],
 * w_down [hidden][inter]; gains are float32: g_in and g_post [hidden],
 * g_q and g_k [head_dim] (one per layer, shared by all heads). Every
 * pointer must be 16-byte aligned. */
typedef struct {
  const void *w_q, *w_k, *w_v, *w_o, *w_gate, *w_up, *w_down;
  const float *g_in, *g_post, *g_q, *g_k;
} dec_layer_weights;

/* embed: [vocab][hidden] in wdtype, also the vocabulary head (tied).
 * layers: HOST array of cfg.layers entries (copied by dec_load_weights). */
typedef struct {
  const void* embed;
  const float* g_final;
  const dec_layer_weights* layers;
} dec_weights;

typedef struct dec_ctx dec_ctx;

/* Bytes of device workspace dec_create needs for cfg (KV cache, rotary
 * table, activations, argmax and attention partials, prefill scratch).
 * The cache holds keys and values in the selected dtype ("Megakernels",
 * "What runs in the DSL"), sized for max_seq positions, i.e. the P + N - 1
 * entries a generation leaves ("GPU-wide end-to-end generation").
 * Returns 0 if cfg is invalid. */
size_t dec_workspace_bytes(const dec_config* cfg);

/* Creates a decoder on the current CUDA device ("Megakernels", "What runs
 * in the DSL": the host precomputes the rotary constants once, before any
 * forward). d_workspace (>= 256-byte aligned, at least
 * dec_workspace_bytes(cfg) bytes) must stay allocated until dec_destroy.
 * Builds the rotary table and clears the cache; returns after that work has
 * finished. stream: the stream later calls run on.
 * Errors: DEC_EINVAL (cfg, NULL, alignment), DEC_ENOMEM (workspace too
 * small), DEC_EDEVICE (not sm_103), DEC_ECUDA. */
dec_status dec_create(const dec_config* cfg, void* d_workspace, size_t workspace_bytes, void* stream,
                      dec_ctx** out);

/* Registers the caller's weight tensors ("Megakernels", "What runs in the
 * DSL": the projections, norm gains and the tied embedding of the forward;
 * no copy: they must outlive the context). Errors: DEC_EINVAL on a NULL or
 * misaligned pointer, DEC_ECUDA. */
dec_status dec_load_weights(dec_ctx* ctx, const dec_weights* w);

/* Position back to 0 and every cache entry invalidated (the cache is
 * zeroed). Timed by the pages' protocol ("Benchmark methodology",
 * "Long-document chunked prefill": timing starts before cache reset). */
dec_status dec_reset(dec_ctx* ctx);

/* Moves the position back to pos (0 <= pos <= current position): cache
 * entries 0..pos-1 stay valid, the next forward runs at position pos and
 * overwrites slot pos. This is how a fixed-context timing trial repeats one
 * token at a fixed cache slot ("Megakernels", "Fixed-context methodology").
 * Asynchronous on the context's stream. Errors: DEC_EINVAL (NULL, pos
 * outside [0, position]), DEC_ECUDA. */
dec_status dec_rewind(dec_ctx* ctx, int32_t pos);

/* One forward of `token` at the current position p ("Megakernels", "What
 * runs in the DSL" for the forward; "GPU-wide end-to-end generation" for the
 * greedy argmax with lowest-ID ties and the host reading the token ID);
 * writes K/V at p and advances the position to p+1.
 * Without DEC_SKIP_LOGITS: final RMSNorm, tied vocabulary projection and
 * argmax (lowest ID on ties) run too. d_logits (nullable, float32[vocab])
 * receives the logits; h_next (nullable) receives the greedy token, and
 * then the call synchronizes the stream to read it. On the persistent engine
 * the token is passed with the launch and the greedy token is written by the
 * kernel into mapped page-locked host memory (no copy calls per step).
 * With DEC_SKIP_LOGITS: only the body runs; d_logits and h_next must be NULL.
 * Errors: DEC_ESTATE (no weights), DEC_ECAPACITY (p == max_seq),
 * DEC_EINVAL (token outside [0, vocab), bad flags). */
dec_status dec_step(dec_ctx* ctx, int32_t token, uint32_t flags, float* d_logits, int32_t* h_next);

/* Two-token verify step of the 4-bit configuration (cfg.wdtype ==
 * DEC_Q4G64): one forward of h_tokens[0] at position p and h_tokens[1] at
 * p+1, where row 1 attends to row 0's cache entry, both through the final
 * norm, the vocabulary projection and the argmax; every projection runs the
 * two-token 4-bit matrix-vector product ("Our Kernel Benchmark Was Measuring
 * the System Cache", Summary: the 4-bit matvec and its two-token variant,
 * the shape of checking a drafted token). d_logits (nullable) receives
 * float32[2][vocab]; h_next (nullable) receives int32[2], the greedy token
 * after each row, and then the call synchronizes the stream to read them.
 * Writes cache entries p and p+1 and advances the position to p+2; the
 * token stream holds h_next[1] at p+2. A caller whose draft h_tokens[1]
 * differs from h_next[0] rewinds to p+1 (dec_rewind) and continues from
 * h_next[0].
 * Errors: DEC_EINVAL (NULL, token outside [0, vocab), not the 4-bit
 * configuration), DEC_ESTATE (no weights), DEC_ECAPACITY (p + 2 > max_seq). */
dec_status dec_verify2(dec_ctx* ctx, const int32_t* h_tokens, float* d_logits, int32_t* h_next);

/* Prompt rows h_tokens[0..n) at positions p..p+n-1 ("Chunked prefill for
 * long prompts"). If cfg.chunk_cap > 0 and n <= chunk_cap the rows run
 * batched (tensor-core projections, causal attention over cache + chunk);
 * otherwise, or with chunk_cap == 0, one token at a time.
 * is_last != 0: the final row also runs the final norm, the vocabulary
 * projection and the argmax; d_logits / h_next as in dec_step (h_next
 * synchronizes). is_last == 0: d_logits and h_next must be NULL.
 * Errors: DEC_EINVAL (n < 1, token out of range), DEC_ECAPACITY
 * (p + n > max_seq), DEC_ESTATE. */
dec_status dec_prefill_chunk(dec_ctx* ctx, const int32_t* h_tokens, int32_t n, int32_t is_last, float* d_logits,
                             int32_t* h_next);

/* n greedy forwards without host involvement ("Megakernels", "GPU-wide
 * end-to-end generation": token IDs in, generated IDs out, the cache
 * advancing by one entry per forward and the next token chosen on the GPU
 * by the lowest-ID argmax; there the host reads each ID before the next
 * forward, here the ID stays on the device): the first input is `token` at
 * the current position, each later input is the previous output. Writes
 * the n outputs to d_tokens_out (device int32[n]). Asynchronous.
 * Errors: DEC_ECAPACITY (p + n > max_seq), DEC_EINVAL, DEC_ESTATE. */
dec_status dec_generate(dec_ctx* ctx, int32_t token, int32_t n, int32_t* d_tokens_out);

/* Read access to one layer's cache ("Benchmark methodology", "Long-document
 * chunked prefill": validation checks every valid K/V entry of every layer):
 * device pointers to K and V, each laid out [n_kv][max_seq][head_dim] in
 * kvdtype, and the number of valid positions. Keys are stored after Q/K-norm
 * and RoPE, values raw. Errors: DEC_EINVAL (NULL, layer out of range). */
dec_status dec_get_kv(const dec_ctx* ctx, int32_t layer, const void** d_k, const void** d_v, int32_t* n_valid);

/* Current position (number of valid cache entries; after a P-token prompt
 * and N outputs it is P + N - 1, the count "Megakernels", "GPU-wide
 * end-to-end generation" validates). -1 if ctx is NULL. */
int32_t dec_position(const dec_ctx* ctx);

/* Stage tracing of the persistent engines. The pages give no tracing API;
 * "Our Kernel Benchmark Was Measuring the System Cache", "Key takeaways",
 * warns that a synchronizing profiler only bounds a kernel's time from
 * below, so the engines stamp their own stages on the device instead.
 * dec_trace_bytes: size of the trace buffer (0 for the staged engine). dec_set_trace: with a non-NULL
 * device buffer of at least that size, every later persistent launch writes,
 * for its first forward, one %globaltimer stamp (nanoseconds) per
 * [cta][layer 0..layers][stage 0..4][event 0..3] as uint64. Stages 0-4 of a
 * layer are QKV, attention, O, gate/up, down; the extra layer index `layers`
 * holds the head (stage 0: vocabulary GEMV, stage 1 event 0: argmax done).
 * Float engine events: 0 stage entry, 1 inputs received and staged (includes
 * waiting for the producing stage), 2 outputs published, 3 every warp done
 * with the stage's weight boxes (attention: key loop done). 4-bit engine
 * events: 0 stage entry, 1 input vector staged in fixed point, 2 products
 * (attention: the attention body) done, 3 the grid barrier after the stage
 * passed; its head has events 0-2 of stage 0 only. After that block, [8][512][4] uint64 for each consumer warp of
 * CTA 0 and the first 512 weight boxes it consumes in the launch: SM clock
 * stamps (clock64) when the box's wait begins, when its data is ready and
 * when its dot products are issued, then the %globaltimer stamp of the wait's
 * beginning. NULL turns tracing off. */
size_t dec_trace_bytes(const dec_ctx* ctx);
dec_status dec_set_trace(dec_ctx* ctx, uint64_t* d_trace, size_t bytes);

/* Limit, in nanoseconds, of every wait of the persistent engines on another
 * CTA's results (exchange words, appended-row counts, grid barriers); 0
 * restores the default of 2 s. The pages give no API for this: the forward
 * runs as ordered stages with no host waits between them ("Megakernels",
 * "GPU-wide end-to-end generation"), so such waits are where a broken
 * launch would otherwise stall. A wait that runs out makes the launch give
 * up: the kernel sets DEC_DEVERR_EXCHANGE_TIMEOUT (float engine) or
 * DEC_DEVERR_BARRIER_TIMEOUT (4-bit engine), waits for its own copies in
 * flight (those waits keep a fixed 2 s limit) and returns; that call's
 * outputs, tokens and cache entries are then undefined, and dec_reset
 * restores a usable state. A limit of a few microseconds makes ordinary
 * forwards give up, which is how the tests exercise that path. The staged
 * engine has no such waits. Takes effect at the next launch.
 * Errors: DEC_EINVAL (NULL). */
dec_status dec_set_wait_limit(dec_ctx* ctx, uint64_t ns);

/* Synchronizes the context's stream and returns (and, if clear != 0,
 * clears) the device error bits DEC_DEVERR_* listed above, among them an
 * all-NaN logit vector at the argmax (the lowest-ID argmax of "Megakernels",
 * "GPU-wide end-to-end generation" has no answer there) and waits that gave
 * up. A set bit marks the affected call's outputs as invalid, as a failed check
 * invalidates a run in "Benchmark methodology", "Long-document chunked
 * prefill". Errors: DEC_EINVAL (NULL), DEC_ECUDA. */
dec_status dec_device_errors(dec_ctx* ctx, int32_t clear, uint32_t* bits);

/* Frees host-side state and CUDA graphs. The workspace stays the caller's
 * (the pages give no API; this is the counterpart of dec_create, which
 * follows "Megakernels", "What runs in the DSL"). */
void dec_destroy(dec_ctx* ctx);

/* Message for the last failed call on ctx (ctx == NULL: last failure of a
 * context-free call on this thread). Never NULL. The pages give no API; the
 * calls above report every failure with a status and this message instead
 * of aborting or continuing silently ("Benchmark methodology", "Long-document
 * chunked prefill": a failed check discards the whole run rather than
 * leaving a partial result that looks successful). */
const char* dec_last_error(const dec_ctx* ctx);

/* y = W x ("Our Kernel Benchmark Was Measuring the System Cache":
 * the matrix-vector product of the decode step).
 * wdtype DEC_F32: W float32 [out][in], x float32 [in];
 * wdtype DEC_BF16: W bfloat16 [out][in], x bfloat16 [in].
 * y float32 [out]; products accumulated in float32, partial sums reduced
 * in a fixed order (bit-reproducible). out, in >= 0 (out == 0: no work;
 * in == 0: y = 0). Any alignment is accepted; 16-byte aligned W with
 * in*sizeof(elem) a multiple of 16 takes the bulk-copy streaming path.
 * Ordering: the call is a programmatic dependent of the previous kernel on
 * `stream` and starts streaming W before that kernel has finished (x and y
 * only after), so W, a weight matrix, must not be written by the kernel
 * enqueued immediately before the call; anything earlier is ordered.
 * Errors: DEC_EINVAL, DEC_ECUDA. */
dec_status gemv(int32_t wdtype, const void* d_W, const void* d_x, float* d_y, int32_t out, int32_t in, void* stream);

/* y[t] = W x[t] for a 4-bit groupwise-affine W ("Our Kernel Benchmark Was
 * Measuring the System Cache", Summary and "Why it mattered, concretely":
 * the one-token matvec and the two-token variant). Each group of 64
 * consecutive columns of a row has an fp16 scale s and bias b, and
 * w = s*q + b for the 4-bit code q.
 * d_codes: uint32 [out][in/8], code j of word w in bits [4j, 4j+4), column
 * 8w+j; d_scale, d_bias: fp16 bits [out][in/64]; d_x: bfloat16 [ntok][in];
 * d_y: float32 [ntok][out]. ntok is 1 or 2; in % 64 == 0; d_codes 16-byte
 * aligned. With in % 512 == 0 (in <= 16384) and 16-byte aligned scales,
 * biases and x, the bulk-copy kernel runs: integer dot products of the codes
 * with x in 16-bit fixed point per 32 columns (step a power of two, error at
 * most 2^-15 of the 32 columns' largest |x|), float32 sums per row, fixed
 * order. Otherwise a per-warp kernel dequantises to float32. Both are
 * bit-reproducible. Like gemv, the call may start reading the codes, scales
 * and biases before the previous kernel on `stream` has finished (x and y
 * only after it): they must not be written by the kernel enqueued
 * immediately before the call. Errors: DEC_EINVAL, DEC_ECUDA. */
dec_status gemv_q4(const uint32_t* d_codes, const uint16_t* d_scale, const uint16_t* d_bias, const uint16_t* d_x,
                   float* d_y, int32_t out, int32_t in, int32_t ntok, void* stream);

/* Rows of W each warp of gemv_q4 handles per pass (1, 2, 4 or 8), for the
 * given ntok ("Our Kernel Benchmark Was Measuring the System Cache", "Why it
 * mattered, concretely": tuned on the cold number). r > 0 sets it, r == -1
 * returns to the automatic choice (the default: 1 when out <= 8 x the SM
 * count, else 4), r == 0 only reads it. Returns the setting in effect (0:
 * automatic), or -1 for a bad argument. Process-wide. */
int32_t gemv_q4_rows_per_warp(int32_t ntok, int32_t r);

/* Lossless bfloat16 storage of float32 weights ("Megakernels", "Lossless
 * decode-weight storage"): d_dst[i] = high 16 bits of d_src[i] for n
 * elements (device pointers, any alignment), and *h_bad (host) = how many
 * elements that storage does not hold exactly (low 16 bits non-zero, or not
 * finite). With *h_bad == 0 the bfloat16 copy widens back to the same
 * float32 bits, so a decoder created with wdtype DEC_BF16 over such copies
 * computes the float32 model's forward on half the weight bytes. Runs on
 * `stream` and synchronizes it to read the count. Calls on one device must
 * not overlap (they share the count). Errors: DEC_EINVAL, DEC_ECUDA. */
dec_status pack_bf16_exact(const float* d_src, uint16_t* d_dst, int64_t n, void* stream, int64_t* h_bad);

/* Reads (and if clear != 0 clears) the device error bits of the
 * context-free calls (gemv, gemv_q4, gemm_bf16, greedy_head_noalloc) on the
 * current device; synchronizes the device. The bits mean what they mean for
 * dec_device_errors (the argmax rule of "Megakernels", "GPU-wide end-to-end
 * generation"; bounded waits that gave up). Errors: DEC_EINVAL (NULL),
 * DEC_ECUDA. */
dec_status gemv_device_errors(int32_t clear, uint32_t* bits);

/* Greedy head for callers that cannot allocate device memory. The operation
 * is the decode step's head: the final RMSNorm and tied vocabulary
 * projection of "Megakernels", "What runs in the DSL", then the lowest-ID
 * argmax of "GPU-wide end-to-end generation"; the pages have no entry point
 * that runs it alone without allocating. Some callers cannot call cudaMalloc: code
 * running inside a host framework that owns every device allocation, or a
 * generation loop that must not risk the device synchronisation an
 * allocation can cause. This call computes x = RMSNorm(h) * gain (eps as
 * given), logits = E x and the greedy token (lowest ID among equal maxima)
 * with the same kernel as the decoder's head, but keeps that kernel's
 * scratch (per-CTA argmax partials, a counter, a position word) in a
 * fixed 8448-byte device array inside the library instead of a workspace.
 * wdtype DEC_F32 or DEC_BF16: d_embed [vocab][hidden] in that dtype (16-byte
 * aligned, rows a multiple of 16 bytes); d_h and d_gain float32 [hidden];
 * d_logits float32 [vocab] or NULL; d_token receives the int32 token.
 * Limits: at most 1024 CTAs of argmax partials (vocab x hidden beyond that is
 * rejected with DEC_EINVAL) and hidden small enough for the shared-memory
 * staging (DEC_EINVAL beyond it). The array persists on every device that
 * loaded the library until exit and is shared by all calls: calls that
 * overlap on the GPU (other streams, other threads) race on it and must be
 * serialised by the caller. The first call on a device looks up the array's
 * address and sets the kernel's shared-memory limit (under a lock, so first
 * calls from several host threads are safe); make that first call before any
 * stream capture. Device-side errors of the call (an all-NaN logit vector,
 * which returns token 0; a bounded wait that gave up) set bits of the
 * context-free error word that gemv_device_errors reads and clears.
 * Allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 * Errors: DEC_EINVAL, DEC_EDEVICE, DEC_ECUDA. */
dec_status greedy_head_noalloc(int32_t wdtype, const void* d_embed, const float* d_h, const float* d_gain, float eps,
                               int32_t vocab, int32_t hidden, float* d_logits, int32_t* d_token, void* stream);

/* Chunked-prefill projection GEMM as a standalone call ("Megakernels",
 * "Chunked prefill for long prompts": a chunk of prompt rows turns each
 * projection into a dense matrix product, run on the tensor cores):
 * C[m][n] = sum_k A[m][k] * W[n][k] for m < M, n < N (accumulate != 0:
 * C[m][n] += that sum). A [M][K] and W [N][K] are bfloat16, row-major,
 * 16-byte aligned (W is a weight matrix in the decoder's [out][in] layout);
 * C is float32 with row stride ldc >= N. Products are exact in FP32 and
 * accumulated in FP32 (tcgen05 tensor cores; 128-row tiles 256, 128 or 64
 * columns wide, chosen per call by the operand bytes the busiest SM
 * streams). K must be a multiple of 8. Asynchronous on `stream`; like gemv
 * the call may start reading W before the previous kernel on `stream` has
 * finished (A and C only after it), so W must not be written by the kernel
 * enqueued immediately before it. Device errors (a bounded wait that gave
 * up) are reported by gemv_device_errors.
 * Errors: DEC_EINVAL (sizes, alignment), DEC_EDEVICE, DEC_ECUDA. */
dec_status gemm_bf16(const uint16_t* d_A, const uint16_t* d_W, float* d_C, int32_t M, int32_t N, int32_t K,
                     int32_t ldc, int32_t accumulate, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* WSG_H */
