/*
 * blk.h — C ABI of the GB300 decoder-block library (libblk.so).
 *
 * One call runs one Qwen2-style decoder block forward (or a stack of them)
 * on one GPU, for one sequence (batch 1) or, with blk_decode_batch and
 * blk_decode_batch_stack, for B sequences of one new token each.  The block
 * is the one printed as TopOp pseudo-code in
 * "An MLIR-based LLM compilation method" (TopOp/TpuOp paper translation),
 * §3.1 Listing 1 (no history) and Listing 2 (with history K/V):
 *
 *   xn   = RMSNorm(x) * ln1_g                  y = x / sqrt(mean(x^2) + eps)
 *   q,k,v= xn Wq^T (+bq), xn Wk^T (+bk), xn Wv^T (+bv)
 *   cos,sin gathered by position_ids from a precomputed table
 *   q,k  = RoPE(q), RoPE(k)                    rotate_half pairs (i, i + D/2),
 *                                              angle = pos * theta^(-2i/D)
 *   attn = FAttention(q, [history K; k], [history V; v])
 *          softmax(q.k / sqrt(D)), causal in cache-slot order, q head h reads
 *          kv head h / (n_heads / n_kv_heads)
 *   h    = x + attn Wo^T
 *   out  = h + W_down (silu(RMSNorm(h) W_gate^T) * (RMSNorm(h) W_up^T))
 *   returns (out, k, v)                        k after RoPE, v as projected
 *
 * and its three statically shaped phases of that paper's §4.1: prefill
 * (T new tokens, no history), prefill_kv (T new tokens after cache_len
 * history slots), decode (one token after cache_len slots).
 *
 * Data types: every activation, weight and cache element is IEEE binary16
 * (fp16), passed as `void*` / `const void*`; position_ids are int64.
 * Arithmetic is fp32 on the GPU (fp16 tensor-core inputs, fp32 accumulate).
 *
 * Ownership: the caller owns every buffer passed in (weights, inputs, outputs,
 * KV cache, workspace) and every pointer named "device" must be device memory
 * on the handle's GPU, 16-byte aligned.  The library allocates device memory
 * only in blk_create (a RoPE table and a status word), never on the hot path.
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and never synchronize, trap or abort; the one exception is the
 * setup call blk_set_rope_yarn, which waits for the device before it
 * replaces the rotation table.
 *
 * KV cache: one K and one V buffer per layer, each [n_kv_heads][max_ctx][head_dim]
 * (the buddy-mlir runtime's per-layer [1, kv_heads, max_len, head_dim] cache of
 * its §6.4.3).  A call reads slots [0, cache_len), writes slots
 * [cache_len, cache_len + T) in place, and leaves every other slot untouched.
 * Slots are the cache's order; position_ids drive RoPE only.  Batched decode
 * takes B such caches back to back per layer, [B][n_kv_heads][max_ctx][head_dim].
 */
#ifndef BLK_H
#define BLK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (0 = success, negative = failure). */
#define BLK_OK 0
#define BLK_ERR_NULL (-1)            /* a required pointer is NULL              */
#define BLK_ERR_ALIGN (-2)           /* a device pointer is not 16-byte aligned */
#define BLK_ERR_SHAPE (-3)           /* unsupported or inconsistent shape       */
#define BLK_ERR_CACHE_OVERFLOW (-4)  /* cache_len + T > max_ctx, or cache_len<0 */
#define BLK_ERR_WORKSPACE (-5)       /* ws_bytes below blk_workspace_bytes()    */
#define BLK_ERR_CUDA (-6)            /* a CUDA runtime call or launch failed    */
#define BLK_ERR_DEVICE_TIMEOUT (-7)  /* a bounded device-side wait gave up      */
#define BLK_ERR_POSITION (-8)        /* a position id outside [0, max_ctx)      */
#define BLK_ERR_DEVICE (-9)          /* the current GPU is not sm_103 (GB300)   */
#define BLK_ERR_SCRATCH_LIMIT (-10)  /* shape needs more scratch than
                                        blk_decode_static's fixed array holds   */
#define BLK_ERR_TOKEN (-11)          /* a token id outside [0, vocab)           */

/* Block shape.  Supported: head_dim 64 or 128; n_heads % n_kv_heads == 0 with
 * group size n_heads / n_kv_heads in {1, 2, 4, 6, 8, 16}; hidden a multiple
 * of 64, intermediate a multiple of 8, both at most 16384; n_heads*head_dim
 * a multiple of 64; max_ctx >= 1. */
typedef struct {
  int32_t hidden;
  int32_t n_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t intermediate;
  float rms_eps;      /* 1e-6 for every shape here                          */
  float rope_theta;   /* 10000                                              */
  int64_t max_ctx;    /* cache slots per head; also bounds position_ids     */
  int32_t has_qkv_bias;
} blk_config;

/* Device pointers to one layer's fp16 weights.  Matrices are [out, in]
 * row-major (PyTorch nn.Linear layout): wq [n_heads*D, hidden],
 * wk/wv [n_kv_heads*D, hidden], wo [hidden, n_heads*D],
 * w_gate/w_up [intermediate, hidden], w_down [hidden, intermediate];
 * ln1_g/ln2_g [hidden]; bq/bk/bv [out] or NULL when !has_qkv_bias. */
typedef struct {
  const void *ln1_g, *wq, *wk, *wv, *bq, *bk, *bv, *wo, *ln2_g, *w_gate,
      *w_up, *w_down;
} blk_weights;

typedef struct blk_handle_s* blk_handle;

/* Option bits for blk_set_flags. */
#define BLK_FLAG_CHAIN 1u
/* BLK_FLAG_CHAIN: the caller promises that the stream work enqueued just
 * before each call never writes that call's weights or KV-cache history
 * (true for a layer stack run back to back).  The first kernel of each call
 * then starts streaming weights while the previous kernel is still running
 * (programmatic dependent launch).  Off by default: the first kernel then
 * waits for all earlier stream work. */

/* Sliding-window attention (the "swa" layer forward of the ds4.c study
 * notes, Part 4, which names the variant without its window; the reading
 * here is the plain one): with window W > 0 the query in cache slot p
 * attends slots [max(0, p - W + 1), p], the last W slots including its own,
 * in every phase and entry point of the handle; W = 0 (the default) is full
 * causal attention.  Slots before a query's window are never read for its
 * result.  Returns BLK_OK, BLK_ERR_NULL or BLK_ERR_SHAPE (W < 0). */
int blk_set_window(blk_handle h, int64_t window);

/* YaRN RoPE (the ds4.c study notes, Part 4, "Trace 1: YaRN frequency
 * scaling" and the RoPE tail-rotation listing), for the handle's whole
 * rotation table: every phase and entry point then rotates q and k with it.
 * With D = head_dim, pair i (rotate_half partners i, i + D/2) at position p:
 *   a      = p * rope_theta^(-2i/D)                       (the original angle)
 *   low    = corr_dim(beta_fast), high = corr_dim(beta_slow),
 *            corr_dim(n) = D ln(n_ctx_orig / (2 pi n)) / (2 ln rope_theta)
 *   ramp_i = 1 - clamp((i - low) / max(0.001, high - low), 0, 1)  (the notes' ramp)
 *   r_i    = ramp_i * ext_factor
 *   angle  = freq_scale * a * (1 - r_i) + a * r_i
 *   cos, sin are multiplied by m = attn_factor * (1 + 0.1 ln(1/freq_scale))
 *            when ext_factor != 0, else by attn_factor
 * The notes elide the blend and never define m; the two are the readings
 * above, the YaRN method's interpolation by parts and its attention
 * temperature (q . k is scaled by m^2).  freq_scale = 1, ext_factor = 0,
 * attn_factor = 1 is plain RoPE. */
typedef struct {
  double freq_scale;   /* 1/s, in (0, 1]                                          */
  double ext_factor;   /* in [0, 1]; the notes use 1 on scaled layers, 0 elsewhere */
  double attn_factor;  /* > 0                                                      */
  double beta_fast;    /* > 0, rotations over n_ctx_orig where the ramp starts (32) */
  double beta_slow;    /* > 0, ... where it ends (1)                               */
  int64_t n_ctx_orig;  /* >= 1, the original training context                      */
} blk_yarn;

/* Sets YaRN RoPE for the handle (y = NULL: back to plain RoPE).  Rebuilds the
 * handle's cos/sin table on the host in f64 and copies it to the device; it
 * first waits for all work on the device (the table may be in use), so it is
 * a setup call, not one for the hot path.  Allocates nothing.  Returns
 * BLK_OK, BLK_ERR_NULL, BLK_ERR_SHAPE (a field out of range) or BLK_ERR_CUDA
 * (including: the current device is not the handle's). */
int blk_set_rope_yarn(blk_handle h, const blk_yarn* y);

/* Creates a handle for `cfg` on the current CUDA device: validates the shape,
 * builds the fp32 cos/sin table [max_ctx][head_dim/2] (angles in f64) and a
 * status word.  Returns BLK_OK, BLK_ERR_NULL, BLK_ERR_SHAPE, BLK_ERR_DEVICE or
 * BLK_ERR_CUDA. */
int blk_create(const blk_config* cfg, blk_handle* out);

/* Frees the handle's device memory.  NULL is ignored. */
void blk_destroy(blk_handle h);

int blk_set_flags(blk_handle h, uint32_t flags);

/* Workspace bytes enough for every call with T <= max_T new tokens (decode
 * needs max_T = 1).  0 on a bad handle or max_T < 1. */
size_t blk_workspace_bytes(blk_handle h, int64_t max_T);

/* prefill (Listing 1): T new tokens, no history (cache_len = 0).
 *   x      device fp16 [T, hidden]
 *   pos    device int64 [T]
 *   k_cache, v_cache  device fp16 [n_kv_heads, max_ctx, head_dim]; slots
 *          [0, T) written
 *   out    device fp16 [T, hidden]
 *   k_new, v_new  device fp16 [T, n_kv_heads, head_dim], or NULL
 *   ws     device workspace of ws_bytes >= blk_workspace_bytes(h, T); its
 *          contents need no initialisation and are garbage afterwards
 * x, pos, out and ws must not overlap the caches or each other. */
int blk_prefill(blk_handle h, const blk_weights* w, const void* x,
                const int64_t* pos, int64_t T, void* k_cache, void* v_cache,
                void* out, void* k_new, void* v_new, void* ws,
                size_t ws_bytes, void* stream);

/* prefill_kv (Listing 2): T new tokens after cache_len history slots; new
 * row t attends slots [0, cache_len + t].  Arguments as blk_prefill. */
int blk_prefill_kv(blk_handle h, const blk_weights* w, const void* x,
                   const int64_t* pos, int64_t T, int64_t cache_len,
                   void* k_cache, void* v_cache, void* out, void* k_new,
                   void* v_new, void* ws, size_t ws_bytes, void* stream);

/* A whole layer stack for T new tokens (prefill when cache_len = 0, else
 * prefill_kv on cache_len history slots) in one call: layer l's output is
 * layer l+1's input, w[l], k_caches[l], v_caches[l] are layer l's weights and
 * caches (as for blk_prefill / blk_prefill_kv), x is the first layer's
 * input and out the last layer's output (device fp16 [T, hidden]); no k_new
 * / v_new (the caches hold them).  Rows pass between layers through two
 * buffers at the end of ws, and each layer's last kernel also writes the next
 * layer's RMSNorm 1, so the result equals one call per layer bit for bit
 * with one launch fewer per layer.  Every layer's arguments are checked
 * before anything is enqueued.  ws_bytes >=
 * blk_prefill_stack_workspace_bytes(h, T).  Returns what blk_prefill_kv
 * returns. */
size_t blk_prefill_stack_workspace_bytes(blk_handle h, int64_t max_T);
int blk_prefill_stack(blk_handle h, const blk_weights* w, int n_layers, void* const* k_caches,
                      void* const* v_caches, const void* x, const int64_t* pos, int64_t T,
                      int64_t cache_len, void* out, void* ws, size_t ws_bytes, void* stream);

/* decode (§4.1): one token after cache_len slots; attends [0, cache_len].
 *   x [1, hidden], pos [1], out [1, hidden], k_new/v_new [1, n_kv_heads, D].
 * One launch of the persistent decode kernel (weight streaming, HBM-bound).
 * Supported when hidden, intermediate and n_heads*head_dim are at most 12288
 * and the group size is at most 16 (BLK_ERR_SHAPE otherwise). */
int blk_decode(blk_handle h, const blk_weights* w, const void* x,
               const int64_t* pos, int64_t cache_len, void* k_cache,
               void* v_cache, void* out, void* k_new, void* v_new, void* ws,
               size_t ws_bytes, void* stream);

/* decode through a stack of n_layers blocks of this shape, in order: layer
 * l's output is layer l+1's input, all at the same cache_len and position.
 * This is the decode call of the buddy-mlir runtime's forward_decode (one
 * token through every layer, each with its own cache; §6.4.6 of that page),
 * done as one launch per 16 layers.
 *   w          host array [n_layers] of weight structs
 *   k_caches, v_caches  host arrays [n_layers] of device cache pointers
 *   k_new, v_new        host arrays [n_layers] of device [1, n_kv_heads, D]
 *                       pointers (entries may be NULL), or NULL
 *   x, out     device fp16 [1, hidden]; out may alias x
 *   ws         blk_workspace_bytes(h, 1) bytes
 * Same return codes as blk_decode. */
int blk_decode_stack(blk_handle h, const blk_weights* w, int n_layers,
                     void* const* k_caches, void* const* v_caches,
                     const void* x, const int64_t* pos, int64_t cache_len,
                     void* out, void* const* k_new, void* const* v_new,
                     void* ws, size_t ws_bytes, void* stream);

/* blk_decode_static — decode without a workspace argument, for callers that
 * cannot allocate device memory.  (The paper has no counterpart: this entry
 * point exists only for such callers.)
 *
 * Some callers may not call cudaMalloc or any allocating routine: a plugin
 * running inside a host framework whose memory manager owns all device memory
 * and rejects outside allocations, or a latency-critical serving loop, where
 * cudaMalloc / cudaFree can synchronize the whole device.  This entry point
 * takes the same inputs and outputs as blk_decode but uses, as its scratch, a
 * fixed array of BLK_STATIC_SCRATCH_BYTES (1 MiB) compiled into the library
 * as a __device__ variable.  Every GPU that loads the library holds that
 * array until the process exits.  It allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * Limit: a shape whose decode scratch (the same bytes blk_decode would need
 * from its workspace) exceeds BLK_STATIC_SCRATCH_BYTES is rejected with
 * BLK_ERR_SCRATCH_LIMIT before anything is enqueued.  The 1.5B shape needs
 * about 0.3 MiB and the hidden-4096 / 32-head shape about 0.8 MiB; a
 * hidden-12288 / 96-head / 6-kv-head shape needs about 1.1 MiB and is
 * rejected.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture begins.
 *
 * Sharing: all calls on a device share the one array and it keeps the last
 * call's contents (the kernels clear what must start at zero).  Calls whose
 * work overlaps on the GPU — on different streams, or from different
 * handles — race on the array; serialize them (one stream, or events).
 * Return codes are those of blk_decode plus BLK_ERR_SCRATCH_LIMIT.  When
 * several apply, BLK_ERR_NULL (a NULL handle, w, x, pos, cache or out) comes
 * first, then BLK_ERR_SCRATCH_LIMIT, then blk_decode's other checks. */
#define BLK_STATIC_SCRATCH_BYTES ((size_t)1 << 20)
int blk_decode_static(blk_handle h, const blk_weights* w, const void* x,
                      const int64_t* pos, int64_t cache_len, void* k_cache,
                      void* v_cache, void* out, void* k_new, void* v_new,
                      void* stream);

/* Synchronizes `stream`, then reports and clears the handle's device status
 * word: BLK_OK, BLK_ERR_DEVICE_TIMEOUT, BLK_ERR_POSITION (a kernel clamped
 * an out-of-range position id), BLK_ERR_TOKEN (blk_embed met an id outside
 * the vocabulary), or BLK_ERR_CUDA if the stream failed. */
int blk_check(blk_handle h, void* stream);

/* Diagnostics of the failure path: launches one kernel that waits for the
 * device int at `flag` (4-byte aligned) to become non-zero, bounded by
 * limit_ns (1 us .. 2 s) of %globaltimer, exactly like the kernels' own
 * waits.  If the limit passes first, the next blk_check reports
 * BLK_ERR_DEVICE_TIMEOUT and the context stays usable.  Returns BLK_OK,
 * BLK_ERR_NULL, BLK_ERR_ALIGN, BLK_ERR_SHAPE (limit out of range) or
 * BLK_ERR_CUDA. */
int blk_wait_probe(blk_handle h, const void* flag, uint64_t limit_ns, void* stream);

/* Per-kernel timing, for benchmarks.  While on, every kernel a call enqueues
 * is bracketed by CUDA events recorded on the call's stream (this keeps
 * consecutive kernels from overlapping, so time the whole step with timing
 * off).  blk_timing_collect synchronizes `stream` and adds the elapsed time
 * of every bracketed launch since the previous collect to a per-kernel total;
 * at most 1024 launches are held between two collects (later ones are not
 * timed and blk_timing_collect returns BLK_ERR_WORKSPACE).  blk_timing_read
 * returns the totals of kernel id `kernel` (0 <= kernel < BLK_N_KERNELS) and
 * its name; BLK_ERR_SHAPE for an unknown id. */
#define BLK_N_KERNELS 16
int blk_timing(blk_handle h, int on);
int blk_timing_collect(blk_handle h, void* stream);
int blk_timing_read(blk_handle h, int kernel, double* total_ms,
                    int64_t* launches, const char** name);

/* Decode timeline, for performance work.  With a device buffer set, every
 * decode launch (blk_decode, blk_decode_stack) has thread 0 of each CTA write
 * %globaltimer nanoseconds when each phase of each layer starts (after its
 * grid barrier) and when its work ends: uint64 entries at
 * [(cta * n_layers + layer) * 6 + phase] * 2 + {0 = start, 1 = end}, phases
 * QKV, attention, split combine, o_proj, gate/up, down; n_layers counts the
 * layers of one launch (at most 16).  Entries past `bytes` are not written.
 * NULL turns tracing off (the default).  Returns BLK_OK or BLK_ERR_NULL. */
int blk_set_trace(blk_handle h, void* device_buffer, size_t bytes);

/* ---- batched decode --------------------------------------------------------
 * One decode step of the block for B independent sequences (one new token
 * each): the decode phase of the TopOp decoder block (§4 "three-phase
 * split") applied per sequence, with the weights read once for all B rows.
 *   x        device fp16 [B, hidden]; pos: device int64 [B] position_ids
 *   cache_lens device int64 [B]: sequence b's history length L_b; its new K/V
 *            go to slot L_b and it attends to slots [0, L_b] of its own cache
 *   max_cache_len  an upper bound of the cache_lens (host value, sizes the
 *            attention's split of the slots); max_cache_len + 1 <= max_ctx
 *   k_cache, v_cache  device fp16 [B, n_kv_heads, max_ctx, head_dim]
 *   out      device fp16 [B, hidden]; k_new, v_new  [B, n_kv_heads, head_dim]
 *            or NULL
 * Equals blk_decode on each sequence within the tolerance (the projections
 * run on tcgen05 MMAs with K split: up to 128 sequences with the weight rows
 * as the MMA's M side, one CTA per 128-row tile and split; more sequences on
 * the 2-SM GEMMs with B rows; the attention is a split-K flash decode per
 * sequence).  A cache length outside
 * [0, max_ctx) skips that sequence's K/V write and attention, and reports
 * BLK_ERR_POSITION from the next blk_check.  Returns BLK_OK, BLK_ERR_NULL,
 * BLK_ERR_ALIGN, BLK_ERR_SHAPE (B outside [1, 4096], more than 16 query heads
 * per kv head), BLK_ERR_CACHE_OVERFLOW (max_cache_len), BLK_ERR_WORKSPACE or
 * BLK_ERR_CUDA.  Asynchronous on `stream`.  The cache lengths are read on the
 * device, so one captured CUDA graph serves consecutive steps.
 * blk_decode_batch_workspace_bytes: enough for every call with B <= max_B
 * sequences; 0 on a bad handle or max_B outside [1, 4096]. */
size_t blk_decode_batch_workspace_bytes(blk_handle h, int64_t max_B);
int blk_decode_batch(blk_handle h, const blk_weights* w, const void* x, const int64_t* pos,
                     const int64_t* cache_lens, int64_t B, int64_t max_cache_len, void* k_cache,
                     void* v_cache, void* out, void* k_new, void* v_new, void* ws,
                     size_t ws_bytes, void* stream);

/* Batched decode through a stack of n_layers blocks of this shape, in order:
 * layer l's output rows are layer l+1's input rows, every layer at the same
 * positions and cache lengths (the batched counterpart of blk_decode_stack).
 *   w                    host array [n_layers] of weight structs
 *   k_caches, v_caches   host arrays [n_layers] of device caches, each
 *                        [B, n_kv_heads, max_ctx, head_dim] as for blk_decode_batch
 *   x, out               device fp16 [B, hidden]; out must not alias x
 *   ws                   blk_decode_batch_stack_workspace_bytes(h, max_B) bytes
 *                        or more, for any max_B >= B (the one-layer workspace
 *                        plus two [B, hidden] fp16 buffers between layers)
 * No k_new / v_new: the new K/V are in each layer's cache slot.  Every
 * layer's arguments are checked before anything is enqueued.  Returns the
 * codes of blk_decode_batch, BLK_ERR_NULL for a NULL array and BLK_ERR_SHAPE
 * for n_layers < 1. */
size_t blk_decode_batch_stack_workspace_bytes(blk_handle h, int64_t max_B);
int blk_decode_batch_stack(blk_handle h, const blk_weights* w, int n_layers,
                           void* const* k_caches, void* const* v_caches, const void* x,
                           const int64_t* pos, const int64_t* cache_lens, int64_t B,
                           int64_t max_cache_len, void* out, void* ws, size_t ws_bytes,
                           void* stream);

/* ---- around the block stack: embedding in, next token out ----------------
 * The inference flow of the MLIR-compilation page (§2.3 "LLM inference
 * overview"): input tokens -> word embedding -> the blocks -> LM head ->
 * logits -> sampling; the buddy-mlir DeepSeek-R1 page (§6.4.4, §6.4.6) picks
 * the next token greedily, the index of the largest logit of the last valid
 * position (vocabulary 151936).
 *
 * blk_embed: x[t, :] = table[ids[t], :] for t < T (fp16 rows copied bit for
 * bit).  table: device fp16 [vocab, hidden], 16-byte aligned; ids: device
 * int64 [T]; x: device fp16 [T, hidden], 16-byte aligned.  An id outside
 * [0, vocab) gives a zero row and BLK_ERR_TOKEN from the next blk_check.
 * Returns BLK_OK, BLK_ERR_NULL, BLK_ERR_ALIGN, BLK_ERR_SHAPE (T <= 0,
 * vocab <= 0) or BLK_ERR_CUDA.  Asynchronous on `stream`. */
int blk_embed(blk_handle h, const void* table, int64_t vocab, const int64_t* ids, int64_t T,
              void* x, void* stream);

/* Bytes of workspace blk_lm_head needs (a few KB: per-SM argmax candidates). */
size_t blk_lm_head_workspace_bytes(blk_handle h);

/* Final RMSNorm, LM head and greedy argmax for T (1..8) hidden rows:
 *   y[t] = RMSNorm(x[t]) * norm_g (eps of the handle's config, y rounded to
 *          fp16), logits[t][v] = sum_i w_lm[v][i] * y[t][i] (fp32 accumulation),
 *   tokens[t] = the lowest v with the largest logits[t][v].
 * x: device fp16 [T, hidden] (16-byte aligned); norm_g: device fp16
 * [hidden]; w_lm: device fp16 [vocab, hidden] row-major (16-byte aligned;
 * hidden <= 4096); logits: device fp32 [T, vocab] or NULL; tokens: device
 * int64 [T]; ws: device workspace of blk_lm_head_workspace_bytes() bytes.
 * Returns BLK_OK, BLK_ERR_NULL, BLK_ERR_ALIGN, BLK_ERR_SHAPE (T outside
 * [1, 8], vocab < 1 or >= 2^31 - 16, hidden > 4096), BLK_ERR_WORKSPACE or
 * BLK_ERR_CUDA.  Asynchronous on `stream`; two kernel launches. */
int blk_lm_head(blk_handle h, const void* x, int64_t T, const void* norm_g, const void* w_lm,
                int64_t vocab, float* logits, int64_t* tokens, void* ws, size_t ws_bytes,
                void* stream);

/* ---- weight-only quantized projections ------------------------------------
 * The TpuOp dialect of "An MLIR-based LLM compilation method" (§2.2) carries
 * INT8 and W4A16 weights with scales and zero points, and its lowering (§3.2)
 * takes GPTQ / AWQ-style formats; activations stay fp16.  Here the seven
 * matrices of a layer (wq, wk, wv, wo, w_gate, w_up, w_down; each [out, in])
 * are quantized per output row:
 *   BLK_WFMT_I8  w[o][i] = scale[o] * q[o][i]
 *                q: int8 [out, in], scale: fp16 [out]
 *   BLK_WFMT_U4  w[o][i] = scale[o][i / group] * (c(o, i) - zero[o][i / group])
 *                c: 4-bit codes 0..15, two per byte along `in`, the even i in
 *                the low nibble: uint8 [out, in / 2]; scale: fp16
 *                [out, in / group]; zero: uint8 [out, in / group], 0..15
 * Gains and q/k/v biases stay fp16, as in blk_weights.  The kernels form
 * each weight as the fp16 product fp16(scale * (code - zero)) (exact code
 * arithmetic, one rounding) and accumulate in fp32.
 * Shape rules (BLK_ERR_SHAPE otherwise): INT8 needs hidden, n_heads*head_dim
 * and intermediate multiples of 16; int4 needs them multiples of 32 and of
 * `group`, a power of two of at least 16.  Decode also needs the scales of one
 * projection phase to fit the kernel's staging area (about 5000 entries per
 * SM: every shape here fits at group 128). */
#define BLK_WFMT_F16 0
#define BLK_WFMT_I8 1
#define BLK_WFMT_U4 2
typedef struct {
  const void* q;      /* codes (device, 16-byte aligned)                      */
  const void* scale;  /* fp16 scales (device, 2-byte aligned)                 */
  const void* zero;   /* uint8 zero points (device), BLK_WFMT_U4 only         */
} blk_qmatrix;
typedef struct {
  int32_t format;     /* BLK_WFMT_I8 or BLK_WFMT_U4                           */
  int32_t group;      /* BLK_WFMT_U4: columns per scale and zero point        */
  const void *ln1_g, *bq, *bk, *bv, *ln2_g;   /* fp16, as in blk_weights     */
  blk_qmatrix wq, wk, wv, wo, w_gate, w_up, w_down;
} blk_qweights;

/* Workspace bytes enough for every quantized call with T <= max_T: decode
 * needs blk_workspace_bytes(h, 1); prefill and prefill_kv also hold the
 * layer's weights formed as fp16 (the first part of the workspace) before
 * the fp16 tensor-core GEMMs run on them.  0 on a bad handle or max_T < 1. */
size_t blk_qworkspace_bytes(blk_handle h, int64_t max_T);

/* The three phases with quantized weights; arguments, caches, outputs and
 * return codes as blk_prefill / blk_prefill_kv / blk_decode /
 * blk_decode_stack, with the workspace sized by blk_qworkspace_bytes.
 * Decode streams the codes themselves (the persistent kernel forms the
 * weights in registers, so a step reads about half (INT8) or a quarter
 * (int4) of the fp16 bytes); prefill and prefill_kv first write the layer's
 * fp16 weights into the workspace (one extra kernel), then run as
 * blk_prefill. */
int blk_prefill_q(blk_handle h, const blk_qweights* w, const void* x, const int64_t* pos,
                  int64_t T, void* k_cache, void* v_cache, void* out, void* k_new, void* v_new,
                  void* ws, size_t ws_bytes, void* stream);
int blk_prefill_kv_q(blk_handle h, const blk_qweights* w, const void* x, const int64_t* pos,
                     int64_t T, int64_t cache_len, void* k_cache, void* v_cache, void* out,
                     void* k_new, void* v_new, void* ws, size_t ws_bytes, void* stream);
int blk_decode_q(blk_handle h, const blk_qweights* w, const void* x, const int64_t* pos,
                 int64_t cache_len, void* k_cache, void* v_cache, void* out, void* k_new,
                 void* v_new, void* ws, size_t ws_bytes, void* stream);
int blk_decode_stack_q(blk_handle h, const blk_qweights* w, int n_layers,
                       void* const* k_caches, void* const* v_caches, const void* x,
                       const int64_t* pos, int64_t cache_len, void* out, void* const* k_new,
                       void* const* v_new, void* ws, size_t ws_bytes, void* stream);

/* Static description of a status code. */
const char* blk_status_str(int status);

#ifdef __cplusplus
}
#endif
#endif /* BLK_H */
