/*
 * gdn.h -- C ABI of the GB300 (sm_103a) batched-prefill library for one
 * Gated DeltaNet (GDN) layer with Q4_K weights.
 *
 * The layer (one call of gdn_prefill) runs five steps, as the pages on the
 * subject describe them:
 *   1. the fused input projection: Q4_K weight superblocks decoded straight to
 *      int8 rows with one fp32 scale per row, activations quantised to int8
 *      rows, an integer tensor-core product and an fp32 rescale
 *      (sparkinfer PR #464 "fused Q4K/Q6K->int8 dequant + token-parallel GDN
 *      conv ...", Summary, "Fused Q4_K/Q6_K -> int8-row dequant");
 *   2. the token-parallel causal 4-tap conv with SiLU and per-head L2 norm
 *      (same page, "Token-parallel GDN conv");
 *   3. the gated delta rule per value head, chunk-parallel (WY/UT form) with the
 *      state carried across chunks ("Verbs Are Fast" epic #3598, parked
 *      ticket "chunk-resident delta-rule scan vs the WY-chunked (tensor-core)
 *      form"; CRUX parity spike #4220, technique table row 1);
 *   4. the gated RMSNorm with a SiLU(z) gate (CRUX parity spike #4220,
 *      technique table row 2: "gated-norm");
 *   5. the output projection, quantised like step 1.
 *
 * Conventions shared by every entry point:
 *   - Pointers named "host" are host memory; every other pointer is device
 *     memory on the current CUDA device, owned by the caller.  The library
 *     never allocates or frees device memory, and keeps none across calls
 *     with one exception: the static scratch array of
 *     gdn_delta_rule_noalloc (GDN_NOALLOC_SCRATCH_BYTES on every device
 *     that loads the library, held until the process exits).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Device
 *     work is enqueued asynchronously on it; the call returns when the work is
 *     enqueued.  A fault inside a kernel shows up at gdn_sync_status().
 *     gdn_delta_rule and gdn_prefill run the delta rule of long inputs (more
 *     than 64 chunks) on two streams of the library, forked from `stream`
 *     and joined back to it within the call, so the work stays ordered on
 *     `stream` and a stream capture records it; the first such call on a
 *     device creates the two streams and two events, kept until exit.
 *   - Return value: GDN_OK (0) or a negative GDN_E* code; the message of the
 *     last failure on the calling thread is gdn_last_error().  A failing call
 *     enqueues nothing unless the code is GDN_ECUDA (a launch that failed).
 *   - There is no fallback path: an unsupported shape is an error, never a
 *     slower route.
 *   - bf16 and fp16 tensors are passed as their 16-bit patterns.
 *   - "codes" tensors carry int8 quantisation codes q (|q| <= 127) stored in
 *     fp16 bit patterns.  Every such q is exact in fp16, and sm_103a's
 *     tensor cores multiply fp16 operands (they have no int8 MMA kind), so the
 *     integer product is taken on fp16 operands with fp32 accumulation, exact
 *     in segments of <= 1024 terms (1024 * 127^2 < 2^24), and the segments are
 *     summed as int32.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_OK 0
#define GDN_EINVAL (-1)   /* null pointer, size out of range, unsupported shape or alignment */
#define GDN_ENOMEM (-2)   /* workspace smaller than one ubatch of tokens needs */
#define GDN_ECUDA (-3)    /* a CUDA call or kernel launch failed */
#define GDN_ETIMEOUT (-4) /* a bounded device-side wait ran out; the kernel returned early */
#define GDN_ERANGE (-5)   /* a value beyond the fp16 operand range (|x| > 65504) reached the recurrence */
#define GDN_EINDEX (-6)   /* debug library only: a kernel's index check failed (the store was skipped) */

#define GDN_W_Q4K 0 /* weights are GGUF Q4_K superblocks, activations bf16 */
#define GDN_W_F32 1 /* weights and activations fp32, no quantisation anywhere */

#define GDN_CHUNK 64 /* tokens per chunk of the chunked delta rule */
#define GDN_MAX_SEQS 256 /* sequences per gdn_prefill_batch or gdn_decode call */
#define GDN_DECODE_GEMV_TOKENS 8 /* tokens per launch of the decode step's fused weight-decode GEMV (dp4a form; the Q4_K tensor-core form takes twice as many) */

/*
 * One GDN layer.  Sizes: Hk = n_qk_heads, Hv = n_v_heads (a multiple of Hk,
 * at most 8 Hk and 64; value head h reads key head h / (Hv/Hk)), dk = dv (64 or 128),
 * C_qk = Hk*dk, C_v = Hv*dv, C_conv = 2*C_qk + C_v,
 * R_in = 2*C_qk + 2*C_v + 2*Hv (rows of the fused input projection, in the
 * order q | k | v | z | beta | alpha).  hidden is a multiple of 256, and so
 * is C_v for Q4_K layers (it is the K extent of the output projection).
 */
typedef struct gdn_layer {
    int32_t hidden;
    int32_t n_qk_heads;
    int32_t n_v_heads;
    int32_t dk;
    int32_t dv;
    int32_t conv_taps; /* must be 4 */
    int32_t wtype;     /* GDN_W_Q4K or GDN_W_F32 */
    int32_t q6k_mask;  /* GDN_W_Q4K layers: bit 0 set = w_in is Q6_K, bit 1 set = w_out is
                          Q6_K (210-byte blocks, see q6k_pack); 0 = both Q4_K.  0 for F32. */
    const void *w_in;  /* Q4_K: [R_in][hidden/256] blocks of 144 B (210 B if Q6_K), 16-byte aligned;
                          F32: fp32 [R_in][hidden] */
    const void *w_out; /* Q4_K: [hidden][C_v/256] blocks (Q6_K likewise); F32: fp32 [hidden][C_v] */
    const float *conv_w;  /* [C_conv][4]; tap 3 multiplies the current token */
    const float *A_log;   /* [Hv] */
    const float *dt_bias; /* [Hv] */
    const float *norm_w;  /* [dv], shared by all value heads */
    /* Optional per-token gates for this call, both or neither: [N][Hv] each,
     * log a_t and b_t drawn directly.  NULL: log a = -exp(A_log) *
     * softplus(alpha + dt_bias) and b = sigmoid(beta) from the projection. */
    const float *gate_log_a;
    const float *gate_b;
    float eps_l2;  /* L2 norm of q and k: x / sqrt(sum x^2 + eps_l2) */
    float eps_rms; /* gated RMSNorm: o / sqrt(mean o^2 + eps_rms) */
    float q_scale; /* multiplies q after its L2 norm (dk^-1/2 for the model family) */
    float reserved1;
} gdn_layer;

/*
 * q4k_pack -- encode fp32 weights into GGUF Q4_K blocks (host only, no GPU).
 * w: host fp32 [rows][cols], cols a multiple of 256.  blocks: host output,
 * rows * cols/256 * 144 bytes.  Per 32-weight sub-block the range
 * [min(0, min w), max w] is split into 15 steps; d and dmin are the largest
 * step and min over the superblock divided by 63, rounded to fp16; the 6-bit
 * indices and 4-bit codes are nearest-even roundings in fp32, clamped.
 * The pages give no encoder (they only decode); this is the plain min-max one.
 * Returns GDN_EINVAL for null pointers, rows < 0 or cols % 256 != 0.
 */
int q4k_pack(const float *w, int64_t rows, int64_t cols, void *blocks);

/*
 * q4k_deq_i8 -- step 1a as its own call: decode Q4_K rows in registers and
 * quantise each row straight to int8 with one fp32 scale, no bf16 scratch
 * (sparkinfer PR #464, Summary, "Fused Q4_K/Q6_K -> int8-row dequant":
 * "decodes superblocks in registers and writes int8 + per-row scale
 * directly"; Correctness paragraph: from "the exact fp32 dequant").
 * The decoded weight is fma(d*sc, q, -(dmin*m)) in fp32 (one rounding);
 * row_scale = amax/127 and q = clamp(rne(w/row_scale), -127, 127), IEEE fp32.
 * blocks: device [rows][cols/256][144 B], 16-byte aligned.  q: device int8
 * [rows][cols], 8-byte aligned.  row_scale: device fp32 [rows].
 * 256 <= cols <= 16384, cols % 256 == 0, rows >= 1.
 */
int q4k_deq_i8(const void *blocks, int64_t rows, int64_t cols, int8_t *q, float *row_scale, void *stream);

/*
 * q6k_pack -- encode fp32 weights into GGUF Q6_K blocks (host only, no GPU),
 * the second weight format of the fused dequant (sparkinfer PR #464,
 * Summary, "Fused Q4_K/Q6_K -> int8-row dequant").  w: host fp32
 * [rows][cols], cols a multiple of 256.  blocks: host output, rows *
 * cols/256 * 210 bytes, each ql[128] | qh[64] | int8 scales[16] | fp16 d.
 * Per 16-weight sub-block step = max|w| / 31; d = the largest step / 127
 * rounded to fp16; scale = clamp(rne(step / d), 0, 127); 6-bit codes q + 32
 * with q = clamp(rne(w / (d*scale)), -32, 31), all in IEEE fp32.  The pages
 * give no encoder; this is the plain absmax one.
 * Returns GDN_EINVAL for null pointers, rows < 0 or cols % 256 != 0.
 */
int q6k_pack(const float *w, int64_t rows, int64_t cols, void *blocks);

/*
 * q6k_deq_i8 -- q4k_deq_i8 for Q6_K rows: decode in registers (the exact
 * fp32 value d*scale*(c - 32)) and quantise each row straight to int8 with one
 * fp32 scale, row_scale = amax/127 and q = clamp(rne(w/row_scale), -127, 127)
 * in IEEE fp32.  blocks: device [rows][cols/256][210 B], 16-byte aligned base.
 * q: device int8 [rows][cols], 8-byte aligned.  row_scale: device fp32 [rows].
 * 256 <= cols <= 16384, cols % 256 == 0, rows >= 1.
 */
int q6k_deq_i8(const void *blocks, int64_t rows, int64_t cols, int8_t *q, float *row_scale, void *stream);

/*
 * gdn_workspace_size -- bytes of device workspace gdn_prefill needs to run
 * `ubatch_tokens` tokens per internal pass (the decoded weights plus every
 * per-token intermediate of one pass).  0 for an invalid layer.
 */
size_t gdn_workspace_size(const gdn_layer *layer, int64_t ubatch_tokens);

/*
 * gdn_prefill -- the whole layer over N prompt tokens, optionally extending a
 * saved state ("Qwen3.5 on CPU prefills one token at a time" #5475: a prompt
 * that extends the held tokens prefills only the suffix from the held state).
 *   x          Q4_K layers: bf16 [N][hidden]; F32 layers: fp32 [N][hidden]
 *   state_in   fp32 [Hv][dv][dk], the recurrent state S before token 0;
 *              NULL = zero state
 *   state_out  fp32 [Hv][dv][dk], S after token N-1; may equal state_in
 *   conv_state fp32 [C_conv][3], in/out: the last 3 raw conv inputs per
 *              channel, oldest first.  Read before token 0 (NULL state_in
 *              with a non-NULL conv_state still reads it), written after.
 *   y          Q4_K layers: bf16 [N][hidden]; F32 layers: fp32 [N][hidden]
 *   workspace  device scratch of ws_bytes >= gdn_workspace_size(layer, 1);
 *              the tokens run in passes of as many tokens as it holds, with
 *              the state and conv tail carried between passes (exact: a pass
 *              boundary is the same as an extend).  256-byte aligned.
 * N >= 1.  Returns GDN_ENOMEM if the workspace holds less than one token.
 */
int gdn_prefill(const gdn_layer *layer, const void *x, int64_t n_tokens, const float *state_in,
                float *state_out, float *conv_state, void *y, void *workspace, size_t ws_bytes,
                void *stream);

/*
 * gdn_prefill_batch -- the whole layer over several independent sequences in
 * one call (variable lengths, each with its own recurrent state and conv
 * tail): the projections run once over the tokens of all sequences, and the
 * state passes of the sequences run side by side (the pages' decode kernels
 * put heads x sequences on the grid: "CRUX parity spike" #4220, technique
 * table row 1).  Each sequence is chunked from its own first token, so its
 * results are bitwise those of a gdn_prefill call on that sequence alone.
 *   x           bf16 (Q4_K) or fp32 (F32) [T][hidden]: the sequences' tokens
 *               one after another, T = cu_seqlens[n_seqs]
 *   cu_seqlens  HOST int64 [n_seqs + 1]: cu_seqlens[0] = 0, non-decreasing;
 *               sequence i holds tokens [cu_seqlens[i], cu_seqlens[i+1]).  A
 *               sequence may be empty: its state is passed through.
 *   n_seqs      1 .. GDN_MAX_SEQS
 *   state_in    fp32 [n_seqs][Hv][dv][dk] or NULL (all zero)
 *   state_out   fp32 [n_seqs][Hv][dv][dk]; may equal state_in
 *   conv_state  fp32 [n_seqs][C_conv][3], in/out, one tail per sequence
 *   y           as x
 *   layer->gate_log_a, gate_b   when given: device [T][Hv]
 *   workspace   device, 256-byte aligned, ws_bytes >=
 *               gdn_batch_workspace_size(layer, T, n_seqs); the call runs in
 *               one pass (GDN_ENOMEM when the workspace is smaller)
 */
size_t gdn_batch_workspace_size(const gdn_layer *layer, int64_t n_tokens, int n_seqs);
int gdn_prefill_batch(const gdn_layer *layer, const void *x, const int64_t *cu_seqlens, int n_seqs,
                      const float *state_in, float *state_out, float *conv_state, void *y, void *workspace,
                      size_t ws_bytes, void *stream);

/*
 * gdn_decode -- the decode step: one new token for each of n_seqs sequences,
 * each with its own state and conv tail, updated in place ("Qwen3.5 speed:
 * prefill and decode parity with llama.cpp" #5305, the decode side of the
 * same layer; the state layout is gdn_prefill's, so a sequence prefills and
 * then decodes on the same buffers).
 *   x          bf16 (Q4_K) or fp32 (F32) [n_seqs][hidden], token s of sequence s
 *   state      fp32 [n_seqs][Hv][dv][dk], in/out
 *   conv_state fp32 [n_seqs][C_conv][3], in/out
 *   y          as x
 *   layer->gate_log_a, gate_b   when given: device [n_seqs][Hv]
 *   workspace  device, 256-byte aligned, ws_bytes >= gdn_decode_workspace_size(
 *              layer, n_seqs)
 * The tokens are quantised to int8 rows as in gdn_prefill; the projections
 * read the Q4_K / Q6_K weights once and take, per weight sub-block, integer
 * dot products of the 4- or 6-bit codes with the tokens' codes, scaled by the
 * sub-block's d*sc (and dmin*m) in fp32: the product of the int8 activations
 * with the exactly decoded weights (no re-quantisation of the weights, unlike
 * the prefill's int8 weight rows), within fp32 rounding.  The conv, SiLU,
 * L2 norms, gates, one token of the recurrence (S <- a S (I - b k k^T) +
 * b v k^T, o = S q) and the gated RMSNorm run in fp32 in one kernel per
 * (value head, sequence), with none of the prefill's fp16 operand roundings;
 * each token (before the input projection) and its gated-norm output with
 * the RMS of each head (before the output projection) are quantised once by
 * a small packing kernel.  Five launches in all, each started while the one
 * before it ends (programmatic dependent launches: the projections' weight
 * copies begin before their inputs exist).  A decoded token therefore
 * agrees with a prefill of it within the stated tolerances, not bit for bit.
 * A sequence's results do not depend on the other sequences of the call: a
 * batch decodes each sequence bit for bit as that sequence alone (with Q4_K
 * the several-token projections run on the tensor cores and one token on
 * dp4a, in the same fp32 operations).
 * 1 <= n_seqs <= GDN_MAX_SEQS.
 */
size_t gdn_decode_workspace_size(const gdn_layer *layer, int n_seqs);
int gdn_decode(const gdn_layer *layer, const void *x, int n_seqs, float *state, float *conv_state, void *y,
               void *workspace, size_t ws_bytes, void *stream);

/*
 * gdn_decode_gemv -- the decode step's projection as its own call:
 * out[t][r] = sx[t] * sum_k xc[t][k] * W[r][k], W the exactly decoded Q4_K
 * (q6k = 0) or Q6_K (q6k = 1) rows [rows][cols/256 blocks] (16-byte aligned),
 * xc the int8 codes of n tokens as fp16 patterns [n][cols] (16-byte aligned),
 * sx [n]; integer dot products per weight sub-block, fp32 sums; a token's
 * result does not depend on n or on the other tokens, bit for bit.  Rows r <
 * n_bf16 go to out_bf16[t*ld_bf16 + r] (bf16), the others to out_f32[t*ld_f32 +
 * r - n_bf16].  256 <= cols <= 16384, cols % 256 == 0, 1 <= n <= GDN_MAX_SEQS.
 */
int gdn_decode_gemv(const void *blocks, int q6k, int64_t rows, int64_t cols, const uint16_t *xc, const float *sx,
                    int64_t n, uint16_t *out_bf16, int64_t ld_bf16, int64_t n_bf16, float *out_f32, int64_t ld_f32,
                    void *stream);

/*
 * gdn_prefill_host -- gdn_prefill fed from, and writing to, host memory: the
 * prompt arrives from the host and the layer output goes back to it, as for
 * an engine whose activations live in host memory between layers.  The
 * tokens run in passes of B tokens; the host-to-device copy of pass p+1 and
 * the device-to-host copy of pass p-1 run on two copy streams of the library
 * while pass p computes (two device staging slots each of x, y and the
 * drawn gates), so the copies hide behind the compute except for the first
 * input and the last output.  Those ends are short: when N > B, B is a
 * multiple of 8 * GDN_CHUNK and N holds the ramps, the passes are B/8, 3B/8,
 * passes of at most B, 3B/8 and B/8 (a pass's copy-in takes about a third of
 * its compute time, so each pass's input arrives while one a third its size
 * computes); otherwise passes of B, the first and the last B/4 when B is a
 * multiple of 4 * GDN_CHUNK and N > B.  Every pass boundary is a chunk
 * boundary (an exact extend), so the results are bitwise those of
 * gdn_prefill.
 *   x_host     page-locked host memory (cudaHostAlloc / cudaHostRegister):
 *              bf16 (Q4_K) or fp32 (F32) [N][hidden]
 *   y_host     page-locked host memory, same type and shape as x_host;
 *              complete once `stream` has reached the end of the call
 *   layer->gate_log_a, gate_b   when given: page-locked HOST memory [N][Hv]
 *   state_in, state_out, conv_state   device memory, as in gdn_prefill
 *   pass_tokens  tokens per pass (rounded down to whole chunks of GDN_CHUNK
 *              when at least one chunk); 0 = as many as the workspace holds;
 *              never more than the workspace holds
 *   workspace  device, 256-byte aligned, ws_bytes >=
 *              gdn_host_workspace_size(layer, 1); gdn_host_workspace_size(
 *              layer, B) holds passes of B tokens
 * Host buffers that are not page-locked are rejected (GDN_EINVAL): pageable
 * copies would serialise with the host thread and defeat the overlap.  The
 * first call on a device creates two copy streams and nine events, kept
 * until exit; the copy streams are forked from `stream` and joined back to
 * it within the call.  Calls from several host threads are serialised while
 * they enqueue.
 */
size_t gdn_host_workspace_size(const gdn_layer *layer, int64_t pass_tokens);
int gdn_prefill_host(const gdn_layer *layer, const void *x_host, int64_t n_tokens, const float *state_in,
                     float *state_out, float *conv_state, void *y_host, int64_t pass_tokens, void *workspace,
                     size_t ws_bytes, void *stream);

/*
 * gdn_prefill_ckpt -- gdn_prefill that also keeps recurrent-state checkpoints:
 * every ckpt_every tokens of the prompt, the state and conv state a prefill
 * of that prefix would leave, so that a later prompt sharing the prefix (a
 * second turn, a retried request) resumes from it instead of prefilling it
 * again ("Qwen3.5 on CPU prefills one token at a time" #5475: a prompt that
 * extends the held tokens prefills only the suffix, and the same page's "Not
 * in scope here" names cross-request reuse of the state as its own issue).
 *   ckpt_every  a positive multiple of GDN_CHUNK
 *   ckpt_state  fp32 [N / ckpt_every][Hv][dv][dk]: snapshot k holds S after
 *               token (k+1)*ckpt_every - 1
 *   ckpt_conv   fp32 [N / ckpt_every][C_conv][3]: the conv state at the same
 *               point (raw inputs of tokens p-3, p-2, p-1, p = (k+1)*ckpt_every)
 * Both may be NULL when N < ckpt_every.  Snapshots are bitwise the state_out and
 * conv_state of gdn_prefill over that prefix (the same chunks, the same
 * arithmetic).  Other arguments as gdn_prefill; the workspace must hold at
 * least GDN_CHUNK tokens unless it holds all N.
 */
int gdn_prefill_ckpt(const gdn_layer *layer, const void *x, int64_t n_tokens, const float *state_in, float *state_out,
                     float *conv_state, void *y, int64_t ckpt_every, float *ckpt_state, float *ckpt_conv,
                     void *workspace, size_t ws_bytes, void *stream);

/*
 * gdn_attn_prefill -- prefill of the hybrid model's full-attention layers:
 * causal softmax attention with grouped key/value heads (the pages' flash
 * attention for those layers, "Qwen3.5 speed: prefill and decode parity with
 * llama.cpp" #5305, sub-ticket #4442: at 32k tokens the prefill falls because
 * they run "cuBLAS f32 with a materialised score matrix", "CRUX parity spike"
 * #4220, long-context finding 2).  For query head h (key/value head h /
 * (n_q_heads / n_kv_heads)) and query i at position nk - nq + i:
 *     o_i = sum_{j <= nk - nq + i} softmax_j(scale * q_i . k_j) v_j
 * (nq = nk: a fresh prefill; nq < nk: queries extending held keys).
 *   q  bf16 [nq][n_q_heads][head_dim], k and v bf16 [nk][n_kv_heads][head_dim],
 *      o bf16 [nq][n_q_heads][head_dim], all 16-byte aligned
 *   head_dim 64, 128 or 256; scale <= 0 means head_dim^-1/2
 *   workspace >= gdn_attn_workspace_size(nk, n_kv_heads, head_dim) bytes (V^T)
 * Products on tcgen05 tensor cores with bf16 operands and fp32 accumulation;
 * the probabilities enter the second product rounded to bf16; the softmax is
 * fp32.  A bounded wait that runs out is reported as GDN_ETIMEOUT.
 */
size_t gdn_attn_workspace_size(int64_t nk, int n_kv_heads, int head_dim);
int gdn_attn_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t nq, int64_t nk, int n_q_heads,
                     int n_kv_heads, int head_dim, float scale, uint16_t *o, void *workspace, size_t ws_bytes,
                     void *stream);

/*
 * gdn_sync_status -- wait for `stream`, then report (and clear) the device
 * error words the kernels set: GDN_OK, GDN_ETIMEOUT (a bounded wait ran out),
 * GDN_ERANGE (a value beyond the fp16 operand range of the recurrence: the
 * results of that call are not valid) or GDN_ECUDA (a CUDA error from the
 * stream).
 */
int gdn_sync_status(void *stream);

/* gdn_last_error -- message of the last failure on this thread ("" if none). */
const char *gdn_last_error(void);

/*
 * gdn_set_stage_events -- instrumentation for per-stage timing.  While set,
 * every gdn_prefill call on this thread records events[i] (cudaEvent_t
 * handles created by the caller) on its stream after stage i of its first
 * pass: 0 entry, 1 weight decode, 2 activation quantisation, 3 input
 * projection, 4 conv (+ conv state), 5 delta rule, 6 gated norm, 7 output
 * projection.  n_events must be 0 (turns it off, events may be NULL) or
 * GDN_N_STAGE_EVENTS.  The events are not owned by the library.
 */
#define GDN_N_STAGE_EVENTS 8
int gdn_set_stage_events(void *const *events, int n_events);

/* ---------------------------------------------------------------------------
 * Stage entry points.  Each runs exactly the kernel gdn_prefill runs for its
 * step, on caller-provided buffers, so that every step can be checked on its
 * own.  Shapes and layouts are those gdn_prefill uses internally.
 * ------------------------------------------------------------------------- */

/*
 * gdn_q4k_deq_codes -- step 1a as gdn_prefill runs it: like q4k_deq_i8 but
 * the int8 codes are written as fp16 bit patterns (codes: [rows][cols],
 * 16-byte aligned), the operand form of the tensor-core product.
 */
int gdn_q4k_deq_codes(const void *blocks, int64_t rows, int64_t cols, uint16_t *codes,
                      float *row_scale, void *stream);

/* gdn_q6k_deq_codes -- gdn_q4k_deq_codes for Q6_K rows (q6k_deq_i8's codes as fp16 patterns). */
int gdn_q6k_deq_codes(const void *blocks, int64_t rows, int64_t cols, uint16_t *codes,
                      float *row_scale, void *stream);

/*
 * gdn_quant_rows -- step 1b (and the quantisation of step 4's output): per row
 * of a bf16 matrix x [rows][cols], scale = amax/127 and codes =
 * clamp(rne(x/scale), -127, 127) in IEEE fp32, written as fp16 patterns.
 * 8 <= cols <= 16384, cols % 8 == 0, x and codes 16-byte aligned.
 */
int gdn_quant_rows(const uint16_t *x, int64_t rows, int64_t cols, uint16_t *codes, float *scale,
                   void *stream);

/*
 * gdn_gemm_codes -- steps 1c and 5: out[m][n] = ((float)sum_k A[m][k]*B[n][k]
 * * sa[m]) * sb[n] with A, B int8 codes in fp16 patterns ([M][K], [Nn][K]
 * row-major, 16-byte aligned), the integer sum exact, the rescale in fp32
 * (nearest-even at each step).  Columns n < n_bf16 go to out_bf16[m*ld_bf16 +
 * n] rounded to bf16; columns n >= n_bf16 go to out_f32[m*ld_f32 + n - n_bf16]
 * (either pointer may be NULL if no column lands there).  K % 64 == 0,
 * 64 <= K <= 65536; M, Nn >= 1.  tcgen05 tensor cores, TMEM accumulators,
 * TMA-fed shared memory.
 */
int gdn_gemm_codes(const uint16_t *a, const float *sa, const uint16_t *b, const float *sb, int64_t M,
                   int64_t Nn, int64_t K, uint16_t *out_bf16, int64_t ld_bf16, int64_t n_bf16,
                   float *out_f32, int64_t ld_f32, void *stream);

/*
 * gdn_gemm_f32 -- steps 1c and 5 of an F32 layer: out[m][n] = sum_k
 * A[m][k]*B[n][k] in fp32, split into bf16 and fp32 columns as gdn_gemm_codes.
 */
int gdn_gemm_f32(const float *a, const float *b, int64_t M, int64_t Nn, int64_t K, uint16_t *out_bf16,
                 int64_t ld_bf16, int64_t n_bf16, float *out_f32, int64_t ld_f32, void *stream);

/*
 * gdn_conv -- step 2: causal 4-tap depthwise conv over the q|k|v channels of
 * the projection (qkvz: bf16 [N][ld_qkvz], channel c at column c), SiLU, L2
 * norm of each q and k head (q then scaled by q_scale), written as fp16
 * (rounded to nearest; the operand type of gdn_delta_rule's tensor cores)
 * into qkv [N][C_conv] (16-byte aligned); a value beyond the fp16 range is
 * reported as GDN_ERANGE by gdn_sync_status.  conv_state [C_conv][3] holds the raw inputs before token 0
 * (read only here).  When gates are not drawn (layer gate pointers NULL) it
 * also writes log_a, b [N][Hv] from beta | alpha (ba: fp32 [N][ld_ba],
 * beta at column h, alpha at column Hv + h); otherwise ba, log_a, b unused.
 */
int gdn_conv(const gdn_layer *layer, const uint16_t *qkvz, int64_t ld_qkvz, int64_t n_tokens,
             const float *conv_state, const float *ba, int64_t ld_ba, uint16_t *qkv, float *log_a,
             float *b, void *stream);

/*
 * gdn_conv_state_update -- after gdn_conv: conv_state <- the last 3 raw conv
 * inputs (x_{N-3}, x_{N-2}, x_{N-1}), taken from qkvz or, for N < 3, from the
 * old conv_state.
 */
int gdn_conv_state_update(const gdn_layer *layer, const uint16_t *qkvz, int64_t ld_qkvz,
                          int64_t n_tokens, float *conv_state, void *stream);

/*
 * gdn_delta_rule -- step 3: the gated delta rule
 *     S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,   o_t = S_t q_t
 * per value head, in chunks of GDN_CHUNK tokens (WY/UT form), products on
 * tensor cores with fp16 operands and fp32 accumulation; the state stays
 * fp32.  qkv: fp16 [N][C_conv] as written by gdn_conv (16-byte aligned);
 * log_a, b: fp32 [N][Hv]; state_in / state_out fp32 [Hv][dv][dk] (state_in
 * NULL = zero; may alias); o: fp16 [N][C_v] (16-byte aligned; rounded to
 * nearest; |o| <= max|S| for |q| <= dk^-1/2).  scratch: 16-byte aligned device
 * bytes >= gdn_delta_rule_scratch_size(layer, N).  An intermediate or output
 * outside the fp16 range (T, A T, the state's fp16 image, R, Delta or o) is
 * reported as GDN_ERANGE by gdn_sync_status; o and the state are then not to
 * be used.
 */
int gdn_delta_rule(const gdn_layer *layer, const uint16_t *qkv, const float *log_a, const float *b,
                   int64_t n_tokens, const float *state_in, float *state_out, uint16_t *o,
                   void *scratch, size_t scratch_bytes, void *stream);
size_t gdn_delta_rule_scratch_size(const gdn_layer *layer, int64_t n_tokens);

/*
 * gdn_delta_rule_noalloc -- the same computation as gdn_delta_rule, for
 * callers that must not allocate device memory: for example a plug-in whose
 * host engine owns every device allocation through its own pool and forbids
 * its plug-ins to call cudaMalloc, or a loop that cannot afford the implicit
 * device synchronisation of cudaMalloc/cudaFree.  The pages have no
 * counterpart to this entry point; it exists only for such callers.
 *   - No scratch argument: the scratch lives in one file-scope device array of
 *     GDN_NOALLOC_SCRATCH_BYTES (48 MiB), which every GPU that loads this
 *     library holds until the process exits.  The call itself allocates
 *     nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *   - A call whose gdn_delta_rule_scratch_size(layer, n_tokens) exceeds that
 *     size returns GDN_EINVAL with a message (e.g. at most 3904 tokens, 61
 *     chunks of 64, for 32 value heads over 16 key heads of d = 128).
 *   - A call outside a stream capture looks up the array's device address
 *     (cudaGetSymbolAddress) with the current device, so a cudaDeviceReset,
 *     which may move the array, is followed; a call inside a capture reuses
 *     the address found by that device's last call outside one.  Make the
 *     first call on each device before any stream capture (inside one, a
 *     device that has no address yet gets GDN_EINVAL).
 *   - Every call shares the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero: each call writes every scratch
 *     entry it reads).  Calls that overlap on the GPU (other streams, other
 *     host threads) race on it: serialise them.
 * Arguments, layouts and results are those of gdn_delta_rule.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (48u << 20)
int gdn_delta_rule_noalloc(const gdn_layer *layer, const uint16_t *qkv, const float *log_a, const float *b,
                           int64_t n_tokens, const float *state_in, float *state_out, uint16_t *o,
                           void *stream);

/*
 * gdn_test_delta_wait_timeout -- a test of the bounded device waits (the
 * pages' lesson that an infrastructure failure must surface as a failure,
 * not as a result: sparkinfer PR #464, eval-bot thread).  Runs only the
 * delta rule's prep kernel of gdn_delta_rule on these inputs, with its copy
 * of the [Q; K] tile never issued, so the kernel's wait for that copy runs
 * out after wait_ns nanoseconds (1 us .. 100 ms).  The kernel records the
 * timeout in its error word, frees its tensor memory and returns; nothing
 * faults and the context stays usable.  gdn_sync_status() then reports
 * GDN_ETIMEOUT once (reading clears the word) and the next call runs
 * normally.  Writes only into `scratch` (gdn_delta_rule_scratch_size bytes).
 */
int gdn_test_delta_wait_timeout(const gdn_layer *layer, const uint16_t *qkv, const float *log_a, const float *b,
                                int64_t n_tokens, void *scratch, size_t scratch_bytes, uint64_t wait_ns,
                                void *stream);

/*
 * gdn_gated_norm -- step 4: per token and value head
 * o_hat = o / sqrt(mean(o^2) + eps_rms) * norm_w * SiLU(z), o fp16 [N][C_v]
 * (8-byte aligned) as gdn_delta_rule writes it, z bf16 at z[t*ld_z + h*dv + i].  Q4_K layers: each token row of o_hat (all C_v
 * values) is quantised like gdn_quant_rows into codes [N][C_v] + scale [N]
 * (out_f32 unused).  F32 layers: o_hat is written to out_f32 [N][C_v].
 */
int gdn_gated_norm(const gdn_layer *layer, const uint16_t *o, const uint16_t *z, int64_t ld_z,
                   int64_t n_tokens, uint16_t *codes, float *scale, float *out_f32, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
