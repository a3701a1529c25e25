// C ABI of the GDN prefill library: argument checks, workspace layout, the
// ubatch loop of gdn_prefill, and the stage entry points.
//
// The batched-prefill entry of the pages refuses what it cannot run instead of
// falling back (sparkinfer PR #464, discussion: "if (!s.gguf || !c.hybrid ||
// !c.dense_ffn || n <= 0) return -1;"), and a prefill whose workspace is sized
// by end position rather than by the tokens in flight collapsed to one token
// at a time ("CRUX parity spike" #4220, part 2, the 512-row workspace).  Here
// every unsupported input returns a negative status, and the workspace is
// sized per ubatch of tokens: when it holds fewer than N tokens the call runs
// in passes, each an exact extend of the previous one.
#include "common.cuh"
#include "streams.h"

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

namespace gdn {
cudaError_t launch_q4k_deq_i8(const void*, int64_t, int64_t, int8_t*, float*, cudaStream_t);
cudaError_t launch_q4k_deq_codes(const void*, int64_t, int64_t, uint16_t*, float*, cudaStream_t);
cudaError_t launch_q6k_deq_i8(const void*, int64_t, int64_t, int8_t*, float*, cudaStream_t);
cudaError_t launch_q6k_deq_codes(const void*, int64_t, int64_t, uint16_t*, float*, cudaStream_t);
cudaError_t launch_q4k_deq_codes2(const void*, int64_t, int64_t, uint16_t*, float*, const void*, int64_t, int64_t,
                                  uint16_t*, float*, cudaStream_t);
cudaError_t launch_quant_rows(const uint16_t*, int64_t, int64_t, uint16_t*, float*, cudaStream_t);
cudaError_t launch_gemm_codes(const uint16_t*, const float*, const uint16_t*, const float*, int64_t, int64_t, int64_t,
                              uint16_t*, int64_t, int64_t, float*, int64_t, cudaStream_t);
cudaError_t launch_gemm_f32(const float*, const float*, int64_t, int64_t, int64_t, uint16_t*, int64_t, int64_t, float*,
                            int64_t, cudaStream_t);
cudaError_t launch_conv(const gdn_layer&, const uint16_t*, int64_t, int64_t, const float*, const float*, int64_t,
                        uint16_t*, float*, float*, cudaStream_t, const int64_t* cu_seqlens = nullptr, int n_seqs = 1);
cudaError_t launch_conv_state(const gdn_layer&, const uint16_t*, int64_t, int64_t, float*, cudaStream_t,
                              const int64_t* cu_seqlens = nullptr, int n_seqs = 1);
cudaError_t launch_delta(const gdn_layer&, const uint16_t*, const float*, const float*, int64_t, const float*, float*,
                         uint16_t*, void*, cudaStream_t, bool overlap, const TokenRangeHook* after_state,
                         const int64_t* cu_seqlens = nullptr, int n_seqs = 1, const DeltaCkpt* ckpt = nullptr,
                         const DeltaFault* fault = nullptr);
cudaError_t launch_conv_ckpt(const gdn_layer&, const uint16_t*, int64_t, int64_t, int64_t, int64_t, float*, cudaStream_t);
size_t delta_scratch_bytes(int hv, int hk, int d, int64_t n);
cudaError_t launch_gated_norm(const gdn_layer&, const uint16_t*, const uint16_t*, int64_t, int64_t, uint16_t*, float*,
                              float*, cudaStream_t);
cudaError_t launch_gemv_dot(const void*, bool, int64_t, int64_t, const uint16_t*, const uint32_t*, int64_t, const float*,
                            int64_t, uint16_t*, int64_t, int64_t, float*, int64_t, cudaStream_t, float*, const uint16_t*,
                            int64_t, int, int);
cudaError_t launch_decode_pack(const void*, bool, int64_t, int64_t, const float*, int, int, int, float, uint32_t*, float*,
                               cudaStream_t);
int64_t decode_pack_stride(int64_t);
cudaError_t launch_decode_mid(const gdn_layer&, const uint16_t*, int64_t, const float*, int64_t, const float*, int64_t,
                              float*, float*, float*, cudaStream_t);
cudaError_t launch_decode_rms_apply(const gdn_layer&, float*, const float*, int64_t, cudaStream_t);
constexpr int DECODE_MID_SPLIT = 4;   // row blocks per value head in the decode step's middle kernel
int read_and_clear_decode_error();
cudaError_t launch_attn(const uint16_t*, const uint16_t*, const uint16_t*, int64_t, int64_t, int, int, int, float, uint16_t*,
                        void*, cudaStream_t);
size_t attn_workspace_bytes(int64_t nk, int hkv, int d);
int read_and_clear_attn_error();
int read_and_clear_gemm_error();
int read_and_clear_delta_error();
int read_and_clear_q4k_error();
int read_and_clear_q6k_error();
int read_and_clear_quant_error();
int read_and_clear_conv_error();
int read_and_clear_norm_error();
}  // namespace gdn

using namespace gdn;

namespace {

thread_local std::string t_last_error;
thread_local cudaEvent_t t_stage_events[GDN_N_STAGE_EVENTS];
thread_local bool t_stage_events_on = false;

// Record stage event i on the stream (first pass only), when instrumentation is on.
cudaError_t mark(int i, bool first_pass, cudaStream_t st) {
    if (!t_stage_events_on || !first_pass) return cudaSuccess;
    return cudaEventRecord(t_stage_events[i], st);
}

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(GDN_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define GDN_LAUNCH(expr, what)                               \
    do {                                                     \
        cudaError_t e_ = (expr);                             \
        if (e_ != cudaSuccess) return cuda_fail(e_, what);   \
    } while (0)

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Sizes {
    int64_t H, hk, hv, d, c_qk, c_v, c_conv, n_bf16, r_in;
};

int check_layer(const gdn_layer* L, Sizes* s) {
    if (!L) return fail(GDN_EINVAL, "layer is NULL");
    if (L->conv_taps != 4) return fail(GDN_EINVAL, "conv_taps must be 4 (got %d)", L->conv_taps);
    if (L->wtype != GDN_W_Q4K && L->wtype != GDN_W_F32) return fail(GDN_EINVAL, "unknown wtype %d", L->wtype);
    if (L->dk != L->dv || (L->dk != 64 && L->dk != 128)) return fail(GDN_EINVAL, "dk = dv in {64, 128} required (got %d, %d)", L->dk, L->dv);
    if (L->n_qk_heads < 1 || L->n_v_heads < 1 || L->n_v_heads % L->n_qk_heads)
        return fail(GDN_EINVAL, "n_v_heads must be a positive multiple of n_qk_heads (got %d, %d)", L->n_v_heads, L->n_qk_heads);
    if (L->n_v_heads > 64) return fail(GDN_EINVAL, "n_v_heads <= 64 required (got %d)", L->n_v_heads);
    if (L->n_v_heads / L->n_qk_heads > 8) return fail(GDN_EINVAL, "at most 8 value heads per key head (got %d)", L->n_v_heads / L->n_qk_heads);
    if (L->hidden < 256 || L->hidden > 16384 || L->hidden % 256)
        return fail(GDN_EINVAL, "hidden must be a multiple of 256 in [256, 16384] (got %d)", L->hidden);
    s->H = L->hidden;
    s->hk = L->n_qk_heads;
    s->hv = L->n_v_heads;
    s->d = L->dk;
    s->c_qk = s->hk * s->d;
    s->c_v = s->hv * s->d;
    s->c_conv = 2 * s->c_qk + s->c_v;
    s->n_bf16 = 2 * s->c_qk + 2 * s->c_v;
    s->r_in = s->n_bf16 + 2 * s->hv;
    if (s->c_v > 16384 || (L->wtype == GDN_W_Q4K && s->c_v % 256))
        return fail(GDN_EINVAL, "n_v_heads * dv must be <= 16384 (and a multiple of 256 for Q4_K) (got %lld)", (long long)s->c_v);
    if (!L->w_in || !L->w_out || !L->conv_w || !L->A_log || !L->dt_bias || !L->norm_w)
        return fail(GDN_EINVAL, "a layer weight pointer is NULL");
    if ((L->gate_log_a == nullptr) != (L->gate_b == nullptr)) return fail(GDN_EINVAL, "gate_log_a and gate_b: both or neither");
    if (!aligned(L->w_in, 16) || !aligned(L->w_out, 16) || !aligned(L->conv_w, 16))
        return fail(GDN_EINVAL, "w_in, w_out and conv_w must be 16-byte aligned");
    if (L->q6k_mask & ~3) return fail(GDN_EINVAL, "q6k_mask: only bits 0 (w_in) and 1 (w_out) are defined");
    if (L->q6k_mask && L->wtype != GDN_W_Q4K) return fail(GDN_EINVAL, "q6k_mask needs a quantised (GDN_W_Q4K) layer");
    return GDN_OK;
}

// Workspace layout for a pass of B tokens.  Every buffer starts on 256 bytes.
struct Workspace {
    uint16_t* wc_in; float* ws_in;    // decoded W_in codes [r_in][H], scales [r_in]
    uint16_t* wc_out; float* ws_out;  // decoded W_out codes [H][c_v], scales [H]
    uint16_t* xc; float* sx;          // x codes [B][H], scales [B]
    uint16_t* qkvz;                   // projection, bf16 [B][n_bf16]
    float* ba;                        // projection, fp32 [B][2 hv]
    uint16_t* qkv;                    // conv output, fp16 [B][c_conv]
    float* log_a; float* b;           // gates [B][hv]
    uint16_t* o;                      // recurrence output, fp16 [B][c_v]
    uint16_t* oc; float* so;          // gated-norm codes [B][c_v], scales [B]  (Q4_K)
    float* ohat;                      // gated-norm output [B][c_v]               (F32)
    void* delta; size_t delta_bytes;  // chunked delta-rule scratch
    size_t total;
};

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// delta_chunks: chunks the delta-rule scratch holds (default: those of B
// tokens in one sequence).
Workspace carve(const gdn_layer* L, const Sizes& s, int64_t B, void* base, int64_t delta_chunks = -1) {
    Workspace w{};
    uint8_t* p = static_cast<uint8_t*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) -> void* {
        void* r = p ? static_cast<void*>(p + off) : nullptr;
        off += up256(bytes);
        return r;
    };
    const bool q4k = L->wtype == GDN_W_Q4K;
    if (q4k) {
        w.wc_in = static_cast<uint16_t*>(take(s.r_in * s.H * 2));
        w.ws_in = static_cast<float*>(take(s.r_in * 4));
        w.wc_out = static_cast<uint16_t*>(take(s.H * s.c_v * 2));
        w.ws_out = static_cast<float*>(take(s.H * 4));
        w.xc = static_cast<uint16_t*>(take(B * s.H * 2));
        w.sx = static_cast<float*>(take(B * 4));
        w.oc = static_cast<uint16_t*>(take(B * s.c_v * 2));
        w.so = static_cast<float*>(take(B * 4));
    } else {
        w.ohat = static_cast<float*>(take(B * s.c_v * 4));
    }
    w.qkvz = static_cast<uint16_t*>(take(B * s.n_bf16 * 2));
    w.ba = static_cast<float*>(take(B * 2 * s.hv * 4));
    w.qkv = static_cast<uint16_t*>(take(B * s.c_conv * 2));
    w.log_a = static_cast<float*>(take(B * s.hv * 4));
    w.b = static_cast<float*>(take(B * s.hv * 4));
    w.o = static_cast<uint16_t*>(take(B * s.c_v * 2));
    w.delta_bytes = delta_scratch_bytes(static_cast<int>(s.hv), static_cast<int>(s.hk), static_cast<int>(s.d),
                                        delta_chunks < 0 ? B : delta_chunks * GDN_CHUNK);
    w.delta = take(w.delta_bytes);
    w.total = off;
    return w;
}

// One pass of nb tokens (steps 1b to 5) on device buffers: x [nb][H] -> y
// [nb][H], the state read from st_in and written to state_out, the conv tail
// carried in place.  gla / gb: this pass's drawn gates (device [nb][hv]) or
// NULL.  The weight codes in w must already be decoded.
// Snapshots of a prefill with checkpoints: every `every` tokens (a multiple
// of GDN_CHUNK) of the prompt, the state and the conv state.
struct Ckpt {
    int64_t every;
    float* state;   // [n/every][hv][d][d]
    float* conv;    // [n/every][c_conv][3]
};

// u0: the pass's first token within the prompt (for the snapshots; a
// multiple of GDN_CHUNK when ck is given).
int run_pass(const gdn_layer* layer, const Sizes& s, const Workspace& w, const void* x, int64_t nb, const float* gla,
             const float* gb, const float* st_in, float* state_out, float* conv_state, void* y, bool first,
             cudaStream_t st, const Ckpt* ck = nullptr, int64_t u0 = 0) {
    const bool q4k = layer->wtype == GDN_W_Q4K;
    if (q4k) {
        GDN_LAUNCH(launch_quant_rows(static_cast<const uint16_t*>(x), nb, s.H, w.xc, w.sx, st), "quantise x");
        GDN_LAUNCH(mark(2, first, st), "stage event");
        cudaError_t e = launch_gemm_codes(w.xc, w.sx, w.wc_in, w.ws_in, nb, s.r_in, s.H, w.qkvz, s.n_bf16, s.n_bf16,
                                          w.ba, 2 * s.hv, st);
        if (e != cudaSuccess) return cuda_fail(e, "input projection");
    } else {
        GDN_LAUNCH(mark(2, first, st), "stage event");
        GDN_LAUNCH(launch_gemm_f32(static_cast<const float*>(x), static_cast<const float*>(layer->w_in), nb, s.r_in, s.H,
                                   w.qkvz, s.n_bf16, s.n_bf16, w.ba, 2 * s.hv, st),
                   "input projection");
    }
    GDN_LAUNCH(mark(3, first, st), "stage event");
    gdn_layer lu = *layer;
    lu.gate_log_a = gla;
    lu.gate_b = gb;
    GDN_LAUNCH(launch_conv(lu, w.qkvz, s.n_bf16, nb, conv_state, w.ba, 2 * s.hv, w.qkv, w.log_a, w.b, st), "conv");
    GDN_LAUNCH(launch_conv_state(lu, w.qkvz, s.n_bf16, nb, conv_state, st), "conv state");
    if (ck) GDN_LAUNCH(launch_conv_ckpt(lu, w.qkvz, s.n_bf16, u0, nb, ck->every, ck->conv, st), "conv-state snapshots");
    GDN_LAUNCH(mark(4, first, st), "stage event");
    const float* la = gla ? gla : w.log_a;
    const float* bb = gb ? gb : w.b;
    // The gated norm of each token segment of the delta rule runs as soon as
    // that segment's state pass is done, beside the later segments.
    const uint16_t* z = w.qkvz + s.c_conv;
    const TokenRangeHook norm_hook = [&](int64_t t0, int64_t t1, cudaStream_t cs) {
        return launch_gated_norm(lu, w.o + t0 * s.c_v, z + t0 * s.n_bf16, s.n_bf16, t1 - t0,
                                 w.oc ? w.oc + t0 * s.c_v : nullptr, w.so ? w.so + t0 : nullptr,
                                 w.ohat ? w.ohat + t0 * s.c_v : nullptr, cs);
    };
    const DeltaCkpt dck{ck ? ck->state : nullptr, ck ? static_cast<int>(ck->every / GDN_CHUNK) : 1,
                        static_cast<int>(u0 / GDN_CHUNK)};
    GDN_LAUNCH(launch_delta(lu, w.qkv, la, bb, nb, st_in, state_out, w.o, w.delta, st, true, &norm_hook, nullptr, 1,
                            ck ? &dck : nullptr),
               "delta rule and gated norm");
    GDN_LAUNCH(mark(5, first, st), "stage event");
    GDN_LAUNCH(mark(6, first, st), "stage event");
    if (q4k) {
        cudaError_t e = launch_gemm_codes(w.oc, w.so, w.wc_out, w.ws_out, nb, s.H, s.c_v, static_cast<uint16_t*>(y), s.H,
                                          s.H, nullptr, 0, st);
        if (e != cudaSuccess) return cuda_fail(e, "output projection");
    } else {
        GDN_LAUNCH(launch_gemm_f32(w.ohat, static_cast<const float*>(layer->w_out), nb, s.H, s.c_v, nullptr, 0, 0,
                                   static_cast<float*>(y), s.H, st),
                   "output projection");
    }
    GDN_LAUNCH(mark(7, first, st), "stage event");
    return GDN_OK;
}

// Tokens per pass for a workspace of ws_bytes: all n if they fit, else the
// largest count that fits, rounded down to whole chunks when at least one
// chunk fits.  0 if not even one token fits.
int64_t pass_tokens_for(const gdn_layer* layer, const Sizes& s, int64_t n, size_t ws_bytes,
                        size_t (*extra)(const gdn_layer*, const Sizes&, int64_t)) {
    auto need = [&](int64_t B) { return carve(layer, s, B, nullptr).total + (extra ? extra(layer, s, B) : 0); };
    if (need(1) > ws_bytes) return 0;
    if (need(n) <= ws_bytes) return n;
    int64_t lo = 1, hi = n;  // need(lo) fits, need(hi) does not
    while (hi - lo > 1) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (need(mid) <= ws_bytes) lo = mid; else hi = mid;
    }
    return lo >= GDN_CHUNK ? lo - lo % GDN_CHUNK : lo;
}

// Step 1a for both weight matrices: each decoded from its own format (Q4_K,
// or Q6_K where the layer's q6k_mask says so) to int8 codes + row scales.
// Two Q4_K matrices share one launch.
int decode_weights(const gdn_layer* L, const Sizes& s, const Workspace& w, cudaStream_t st) {
    const bool in6 = L->q6k_mask & 1, out6 = L->q6k_mask & 2;
    if (!in6 && !out6) {
        GDN_LAUNCH(launch_q4k_deq_codes2(L->w_in, s.r_in, s.H, w.wc_in, w.ws_in, L->w_out, s.H, s.c_v, w.wc_out,
                                         w.ws_out, st),
                   "dequant W_in, W_out");
        return GDN_OK;
    }
    GDN_LAUNCH(in6 ? launch_q6k_deq_codes(L->w_in, s.r_in, s.H, w.wc_in, w.ws_in, st)
                   : launch_q4k_deq_codes(L->w_in, s.r_in, s.H, w.wc_in, w.ws_in, st),
               "dequant W_in");
    GDN_LAUNCH(out6 ? launch_q6k_deq_codes(L->w_out, s.H, s.c_v, w.wc_out, w.ws_out, st)
                    : launch_q4k_deq_codes(L->w_out, s.H, s.c_v, w.wc_out, w.ws_out, st),
               "dequant W_out");
    return GDN_OK;
}

// Device staging of gdn_prefill_host beyond the pass workspace: two slots each
// of x, y and (when the gates are drawn) log a and b.
size_t host_stage_bytes(const gdn_layer* L, const Sizes& s, int64_t B) {
    const size_t esz = L->wtype == GDN_W_Q4K ? 2 : 4;
    size_t t = 4 * up256(B * s.H * esz);
    if (L->gate_log_a) t += 4 * up256(B * s.hv * 4);
    return t;
}

// Workspace of one decode step of B tokens (one per sequence).
struct DecodeWs {
    uint16_t* qkvz; float* ba;        // projection [B][n_bf16] bf16, [B][2 hv] fp32
    float* ohat;                      // gated output [B][c_v] fp32 (RMS applied when it is packed)
    float* psum;                      // partial sums of o^2 [B][hv][DECODE_MID_SPLIT]
    uint32_t* xp; float* sx;          // packed codes of x [B][H] and of o_hat [B][c_v] with row scales
    uint32_t* op; float* so;          // (Q4_K / Q6_K layers)
    size_t total;
};

DecodeWs carve_decode(const gdn_layer* L, const Sizes& s, int64_t B, void* base) {
    DecodeWs w{};
    uint8_t* p = static_cast<uint8_t*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) -> void* {
        void* r = p ? static_cast<void*>(p + off) : nullptr;
        off += up256(bytes);
        return r;
    };
    w.qkvz = static_cast<uint16_t*>(take(B * s.n_bf16 * 2));
    w.ba = static_cast<float*>(take(B * 2 * s.hv * 4));
    w.ohat = static_cast<float*>(take(B * s.c_v * 4));
    w.psum = static_cast<float*>(take(B * s.hv * DECODE_MID_SPLIT * 4));
    if (L->wtype == GDN_W_Q4K) {
        w.xp = static_cast<uint32_t*>(take(B * decode_pack_stride(s.H) * 4));
        w.sx = static_cast<float*>(take(B * 4));
        w.op = static_cast<uint32_t*>(take(B * decode_pack_stride(s.c_v) * 4));
        w.so = static_cast<float*>(take(B * 4));
    }
    w.total = off;
    return w;
}

// GDN_OK if p is page-locked host memory (cudaHostAlloc or cudaHostRegister).
int check_pinned(const void* p, const char* what) {
    cudaPointerAttributes a{};
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return fail(GDN_EINVAL, "gdn_prefill_host: %s: %s", what, cudaGetErrorString(e));
    }
    if (a.type != cudaMemoryTypeHost)
        return fail(GDN_EINVAL, "gdn_prefill_host: %s must be page-locked host memory (cudaHostAlloc or cudaHostRegister)",
                    what);
    return GDN_OK;
}

}  // namespace

extern "C" {

const char* gdn_last_error(void) { return t_last_error.c_str(); }

int gdn_set_stage_events(void* const* events, int n_events) {
    if (n_events == 0) {
        t_stage_events_on = false;
        return GDN_OK;
    }
    if (n_events != GDN_N_STAGE_EVENTS || !events) return fail(GDN_EINVAL, "gdn_set_stage_events: n_events must be 0 or %d", GDN_N_STAGE_EVENTS);
    for (int i = 0; i < GDN_N_STAGE_EVENTS; ++i) {
        if (!events[i]) return fail(GDN_EINVAL, "gdn_set_stage_events: event %d is NULL", i);
        t_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
    }
    t_stage_events_on = true;
    return GDN_OK;
}

int q4k_deq_i8(const void* blocks, int64_t rows, int64_t cols, int8_t* q, float* row_scale, void* stream) {
    if (!blocks || !q || !row_scale) return fail(GDN_EINVAL, "q4k_deq_i8: NULL pointer");
    if (rows < 1 || rows > 0x7fffffff || cols < 256 || cols > 16384 || cols % 256)
        return fail(GDN_EINVAL, "q4k_deq_i8: rows >= 1 and cols a multiple of 256 in [256, 16384] required");
    if (!aligned(blocks, 16) || !aligned(q, 8)) return fail(GDN_EINVAL, "q4k_deq_i8: blocks 16-byte and q 8-byte alignment required");
    GDN_LAUNCH(launch_q4k_deq_i8(blocks, rows, cols, q, row_scale, static_cast<cudaStream_t>(stream)), "q4k_deq_i8");
    return GDN_OK;
}

int gdn_q4k_deq_codes(const void* blocks, int64_t rows, int64_t cols, uint16_t* codes, float* row_scale, void* stream) {
    if (!blocks || !codes || !row_scale) return fail(GDN_EINVAL, "gdn_q4k_deq_codes: NULL pointer");
    if (rows < 1 || rows > 0x7fffffff || cols < 256 || cols > 16384 || cols % 256)
        return fail(GDN_EINVAL, "gdn_q4k_deq_codes: rows >= 1 and cols a multiple of 256 in [256, 16384] required");
    if (!aligned(blocks, 16) || !aligned(codes, 16)) return fail(GDN_EINVAL, "gdn_q4k_deq_codes: 16-byte alignment required");
    GDN_LAUNCH(launch_q4k_deq_codes(blocks, rows, cols, codes, row_scale, static_cast<cudaStream_t>(stream)), "gdn_q4k_deq_codes");
    return GDN_OK;
}

int q6k_deq_i8(const void* blocks, int64_t rows, int64_t cols, int8_t* q, float* row_scale, void* stream) {
    if (!blocks || !q || !row_scale) return fail(GDN_EINVAL, "q6k_deq_i8: NULL pointer");
    if (rows < 1 || rows > 0x7fffffff || cols < 256 || cols > 16384 || cols % 256)
        return fail(GDN_EINVAL, "q6k_deq_i8: rows >= 1 and cols a multiple of 256 in [256, 16384] required");
    if (!aligned(blocks, 16) || !aligned(q, 8)) return fail(GDN_EINVAL, "q6k_deq_i8: blocks 16-byte and q 8-byte alignment required");
    GDN_LAUNCH(launch_q6k_deq_i8(blocks, rows, cols, q, row_scale, static_cast<cudaStream_t>(stream)), "q6k_deq_i8");
    return GDN_OK;
}

int gdn_q6k_deq_codes(const void* blocks, int64_t rows, int64_t cols, uint16_t* codes, float* row_scale, void* stream) {
    if (!blocks || !codes || !row_scale) return fail(GDN_EINVAL, "gdn_q6k_deq_codes: NULL pointer");
    if (rows < 1 || rows > 0x7fffffff || cols < 256 || cols > 16384 || cols % 256)
        return fail(GDN_EINVAL, "gdn_q6k_deq_codes: rows >= 1 and cols a multiple of 256 in [256, 16384] required");
    if (!aligned(blocks, 16) || !aligned(codes, 16)) return fail(GDN_EINVAL, "gdn_q6k_deq_codes: 16-byte alignment required");
    GDN_LAUNCH(launch_q6k_deq_codes(blocks, rows, cols, codes, row_scale, static_cast<cudaStream_t>(stream)),
               "gdn_q6k_deq_codes");
    return GDN_OK;
}

int gdn_quant_rows(const uint16_t* x, int64_t rows, int64_t cols, uint16_t* codes, float* scale, void* stream) {
    if (!x || !codes || !scale) return fail(GDN_EINVAL, "gdn_quant_rows: NULL pointer");
    if (rows < 1 || rows > 0x7fffffff || cols < 8 || cols > 16384 || cols % 8)
        return fail(GDN_EINVAL, "gdn_quant_rows: rows >= 1 and cols a multiple of 8 in [8, 16384] required");
    if (!aligned(x, 16) || !aligned(codes, 16)) return fail(GDN_EINVAL, "gdn_quant_rows: 16-byte alignment required");
    GDN_LAUNCH(launch_quant_rows(x, rows, cols, codes, scale, static_cast<cudaStream_t>(stream)), "gdn_quant_rows");
    return GDN_OK;
}

int gdn_gemm_codes(const uint16_t* a, const float* sa, const uint16_t* b, const float* sb, int64_t M, int64_t Nn,
                   int64_t K, uint16_t* out_bf16, int64_t ld_bf16, int64_t n_bf16, float* out_f32, int64_t ld_f32,
                   void* stream) {
    if (!a || !sa || !b || !sb) return fail(GDN_EINVAL, "gdn_gemm_codes: NULL operand");
    if (M < 1 || Nn < 1 || M > 0x7fffffff || Nn > 0x7fffffff || K < 64 || K > 65536 || K % 64)
        return fail(GDN_EINVAL, "gdn_gemm_codes: M, N >= 1 and K a multiple of 64 in [64, 65536] required");
    if (n_bf16 < 0) return fail(GDN_EINVAL, "gdn_gemm_codes: n_bf16 < 0");
    if (n_bf16 > 0 && (!out_bf16 || ld_bf16 < (n_bf16 < Nn ? n_bf16 : Nn))) return fail(GDN_EINVAL, "gdn_gemm_codes: bf16 output");
    if (n_bf16 < Nn && (!out_f32 || ld_f32 < Nn - n_bf16)) return fail(GDN_EINVAL, "gdn_gemm_codes: fp32 output");
    if (!aligned(a, 16) || !aligned(b, 16)) return fail(GDN_EINVAL, "gdn_gemm_codes: operands must be 16-byte aligned");
    cudaError_t e = launch_gemm_codes(a, sa, b, sb, M, Nn, K, out_bf16, ld_bf16, n_bf16, out_f32, ld_f32,
                                      static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue) return fail(GDN_EINVAL, "gdn_gemm_codes: tensor map rejected (alignment or driver entry point)");
    if (e != cudaSuccess) return cuda_fail(e, "gdn_gemm_codes");
    return GDN_OK;
}

int gdn_gemm_f32(const float* a, const float* b, int64_t M, int64_t Nn, int64_t K, uint16_t* out_bf16, int64_t ld_bf16,
                 int64_t n_bf16, float* out_f32, int64_t ld_f32, void* stream) {
    if (!a || !b) return fail(GDN_EINVAL, "gdn_gemm_f32: NULL operand");
    if (M < 1 || Nn < 1 || K < 1 || M > 0x7fffffff || Nn > 0x7fffffff || K > 0x7fffffff) return fail(GDN_EINVAL, "gdn_gemm_f32: sizes");
    if (n_bf16 < 0) return fail(GDN_EINVAL, "gdn_gemm_f32: n_bf16 < 0");
    if (n_bf16 > 0 && !out_bf16) return fail(GDN_EINVAL, "gdn_gemm_f32: bf16 output");
    if (n_bf16 < Nn && !out_f32) return fail(GDN_EINVAL, "gdn_gemm_f32: fp32 output");
    GDN_LAUNCH(launch_gemm_f32(a, b, M, Nn, K, out_bf16, ld_bf16, n_bf16, out_f32, ld_f32, static_cast<cudaStream_t>(stream)),
               "gdn_gemm_f32");
    return GDN_OK;
}

int gdn_conv(const gdn_layer* layer, const uint16_t* qkvz, int64_t ld_qkvz, int64_t n_tokens, const float* conv_state,
             const float* ba, int64_t ld_ba, uint16_t* qkv, float* log_a, float* b, void* stream) {
    Sizes s;
    int r = check_layer(layer, &s);
    if (r) return r;
    if (n_tokens < 1 || n_tokens > 0x7fffffff) return fail(GDN_EINVAL, "gdn_conv: n_tokens >= 1 required");
    if (!qkvz || !conv_state || !qkv) return fail(GDN_EINVAL, "gdn_conv: NULL pointer");
    if (!aligned(qkv, 16)) return fail(GDN_EINVAL, "gdn_conv: qkv must be 16-byte aligned");
    if (ld_qkvz < s.c_conv || ld_qkvz % 4 || !aligned(qkvz, 8)) return fail(GDN_EINVAL, "gdn_conv: qkvz layout");
    if (layer->gate_log_a == nullptr && (!ba || !log_a || !b || ld_ba < 2 * s.hv)) return fail(GDN_EINVAL, "gdn_conv: gate buffers");
    GDN_LAUNCH(launch_conv(*layer, qkvz, ld_qkvz, n_tokens, conv_state, ba, ld_ba, qkv, log_a, b, static_cast<cudaStream_t>(stream)),
               "gdn_conv");
    return GDN_OK;
}

int gdn_conv_state_update(const gdn_layer* layer, const uint16_t* qkvz, int64_t ld_qkvz, int64_t n_tokens,
                          float* conv_state, void* stream) {
    Sizes s;
    int r = check_layer(layer, &s);
    if (r) return r;
    if (n_tokens < 1 || !qkvz || !conv_state || ld_qkvz < s.c_conv) return fail(GDN_EINVAL, "gdn_conv_state_update: arguments");
    GDN_LAUNCH(launch_conv_state(*layer, qkvz, ld_qkvz, n_tokens, conv_state, static_cast<cudaStream_t>(stream)),
               "gdn_conv_state_update");
    return GDN_OK;
}

size_t gdn_delta_rule_scratch_size(const gdn_layer* layer, int64_t n_tokens) {
    Sizes s;
    if (check_layer(layer, &s) || n_tokens < 1) return 0;
    return delta_scratch_bytes(static_cast<int>(s.hv), static_cast<int>(s.hk), static_cast<int>(s.d), n_tokens);
}

int gdn_delta_rule(const gdn_layer* layer, const uint16_t* qkv, const float* log_a, const float* b, int64_t n_tokens,
                   const float* state_in, float* state_out, uint16_t* o, void* scratch, size_t scratch_bytes, void* stream) {
    Sizes s;
    int r = check_layer(layer, &s);
    if (r) return r;
    if (n_tokens < 1 || n_tokens > 0x7fffffff) return fail(GDN_EINVAL, "gdn_delta_rule: n_tokens >= 1 required");
    if (!qkv || !log_a || !b || !state_out || !o || !scratch) return fail(GDN_EINVAL, "gdn_delta_rule: NULL pointer");
    if (!aligned(qkv, 16) || !aligned(scratch, 16) || !aligned(o, 16)) return fail(GDN_EINVAL, "gdn_delta_rule: qkv, scratch and o 16-byte alignment required");
    if (scratch_bytes < delta_scratch_bytes(static_cast<int>(s.hv), static_cast<int>(s.hk), static_cast<int>(s.d), n_tokens))
        return fail(GDN_ENOMEM, "gdn_delta_rule: scratch too small");
    GDN_LAUNCH(launch_delta(*layer, qkv, log_a, b, n_tokens, state_in, state_out, o, scratch, static_cast<cudaStream_t>(stream),
                            true, nullptr),
               "gdn_delta_rule");
    return GDN_OK;
}

int gdn_test_delta_wait_timeout(const gdn_layer* layer, const uint16_t* qkv, const float* log_a, const float* b,
                                int64_t n_tokens, void* scratch, size_t scratch_bytes, uint64_t wait_ns, void* stream) {
    Sizes s;
    int r = check_layer(layer, &s);
    if (r) return r;
    if (n_tokens < 1 || n_tokens > 0x7fffffff) return fail(GDN_EINVAL, "gdn_test_delta_wait_timeout: n_tokens >= 1 required");
    if (!qkv || !log_a || !b || !scratch) return fail(GDN_EINVAL, "gdn_test_delta_wait_timeout: NULL pointer");
    if (!aligned(qkv, 16) || !aligned(scratch, 16))
        return fail(GDN_EINVAL, "gdn_test_delta_wait_timeout: qkv and scratch 16-byte alignment required");
    if (wait_ns < 1000 || wait_ns > 100000000ull)
        return fail(GDN_EINVAL, "gdn_test_delta_wait_timeout: wait_ns in [1 us, 100 ms] required");
    if (scratch_bytes < delta_scratch_bytes(static_cast<int>(s.hv), static_cast<int>(s.hk), static_cast<int>(s.d), n_tokens))
        return fail(GDN_ENOMEM, "gdn_test_delta_wait_timeout: scratch too small");
    const DeltaFault fault{wait_ns};
    // the prep alone writes no state and no output: state_out and o are unused
    GDN_LAUNCH(launch_delta(*layer, qkv, log_a, b, n_tokens, nullptr, nullptr, nullptr, scratch,
                            static_cast<cudaStream_t>(stream), false, nullptr, nullptr, 1, nullptr, &fault),
               "gdn_test_delta_wait_timeout");
    return GDN_OK;
}

int gdn_gated_norm(const gdn_layer* layer, const uint16_t* o, const uint16_t* z, int64_t ld_z, int64_t n_tokens,
                   uint16_t* codes, float* scale, float* out_f32, void* stream) {
    Sizes s;
    int r = check_layer(layer, &s);
    if (r) return r;
    if (n_tokens < 1 || n_tokens > 0x7fffffff || !o || !z) return fail(GDN_EINVAL, "gdn_gated_norm: arguments");
    if (ld_z < s.c_v || ld_z % 4 || !aligned(z, 8) || !aligned(o, 8)) return fail(GDN_EINVAL, "gdn_gated_norm: layout");
    if (layer->wtype == GDN_W_Q4K && (!codes || !scale || !aligned(codes, 8))) return fail(GDN_EINVAL, "gdn_gated_norm: codes");
    if (layer->wtype == GDN_W_F32 && !out_f32) return fail(GDN_EINVAL, "gdn_gated_norm: out_f32");
    GDN_LAUNCH(launch_gated_norm(*layer, o, z, ld_z, n_tokens, codes, scale, out_f32, static_cast<cudaStream_t>(stream)),
               "gdn_gated_norm");
    return GDN_OK;
}

size_t gdn_workspace_size(const gdn_layer* layer, int64_t ubatch_tokens) {
    Sizes s;
    if (check_layer(layer, &s) || ubatch_tokens < 1) return 0;
    return carve(layer, s, ubatch_tokens, nullptr).total;
}

static int prefill_impl(const gdn_layer* layer, const void* x, int64_t n_tokens, const float* state_in, float* state_out,
                        float* conv_state, void* y, void* workspace, size_t ws_bytes, void* stream, const Ckpt* ck) {
    Sizes s;
    int r = check_layer(layer, &s);
    if (r) return r;
    if (n_tokens < 1 || n_tokens > 0x7fffffff) return fail(GDN_EINVAL, "gdn_prefill: n_tokens >= 1 required (got %lld)", (long long)n_tokens);
    if (!x || !state_out || !conv_state || !y || !workspace) return fail(GDN_EINVAL, "gdn_prefill: NULL pointer");
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(workspace, 256)) return fail(GDN_EINVAL, "gdn_prefill: x, y 16-byte and workspace 256-byte alignment required");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Largest pass that fits: the workspace grows linearly in B.
    const int64_t B = pass_tokens_for(layer, s, n_tokens, ws_bytes, nullptr);
    if (B < 1)
        return fail(GDN_ENOMEM, "gdn_prefill: workspace %zu B < %zu B needed for one token", ws_bytes,
                    carve(layer, s, 1, nullptr).total);
    if (ck && B < n_tokens && B % GDN_CHUNK)
        return fail(GDN_ENOMEM, "gdn_prefill_ckpt: with snapshots the workspace must hold %d tokens or all of them",
                    GDN_CHUNK);
    Workspace w = carve(layer, s, B, workspace);
    const bool q4k = layer->wtype == GDN_W_Q4K;
    GDN_LAUNCH(mark(0, true, st), "stage event");
    if (q4k && (r = decode_weights(layer, s, w, st))) return r;
    GDN_LAUNCH(mark(1, true, st), "stage event");
    for (int64_t u0 = 0; u0 < n_tokens; u0 += B) {
        const int64_t nb = (n_tokens - u0) < B ? (n_tokens - u0) : B;
        const size_t esz = q4k ? 2 : 4;
        const float* gla = layer->gate_log_a ? layer->gate_log_a + u0 * s.hv : nullptr;
        const float* gb = layer->gate_b ? layer->gate_b + u0 * s.hv : nullptr;
        r = run_pass(layer, s, w, static_cast<const uint8_t*>(x) + u0 * s.H * esz, nb, gla, gb,
                     u0 == 0 ? state_in : state_out, state_out, conv_state, static_cast<uint8_t*>(y) + u0 * s.H * esz,
                     u0 == 0, st, ck, u0);
        if (r) return r;
    }
    return GDN_OK;
}

int gdn_prefill(const gdn_layer* layer, const void* x, int64_t n_tokens, const float* state_in, float* state_out,
                float* conv_state, void* y, void* workspace, size_t ws_bytes, void* stream) {
    return prefill_impl(layer, x, n_tokens, state_in, state_out, conv_state, y, workspace, ws_bytes, stream, nullptr);
}

int gdn_prefill_ckpt(const gdn_layer* layer, const void* x, int64_t n_tokens, const float* state_in, float* state_out,
                     float* conv_state, void* y, int64_t ckpt_every, float* ckpt_state, float* ckpt_conv,
                     void* workspace, size_t ws_bytes, void* stream) {
    if (ckpt_every < GDN_CHUNK || ckpt_every % GDN_CHUNK)
        return fail(GDN_EINVAL, "gdn_prefill_ckpt: ckpt_every must be a positive multiple of %d (got %lld)", GDN_CHUNK,
                    (long long)ckpt_every);
    if (n_tokens >= ckpt_every && (!ckpt_state || !ckpt_conv)) return fail(GDN_EINVAL, "gdn_prefill_ckpt: NULL snapshot buffer");
    if ((ckpt_state && !aligned(ckpt_state, 16)) || (ckpt_conv && !aligned(ckpt_conv, 4)))
        return fail(GDN_EINVAL, "gdn_prefill_ckpt: snapshot buffers misaligned");
    const Ckpt ck{ckpt_every, ckpt_state, ckpt_conv};
    return prefill_impl(layer, x, n_tokens, state_in, state_out, conv_state, y, workspace, ws_bytes, stream,
                        n_tokens >= ckpt_every ? &ck : nullptr);
}

size_t gdn_host_workspace_size(const gdn_layer* layer, int64_t pass_tokens) {
    Sizes s;
    if (check_layer(layer, &s) || pass_tokens < 1) return 0;
    return carve(layer, s, pass_tokens, nullptr).total + host_stage_bytes(layer, s, pass_tokens);
}

int gdn_prefill_host(const gdn_layer* layer, const void* x_host, int64_t n_tokens, const float* state_in,
                     float* state_out, float* conv_state, void* y_host, int64_t pass_tokens, void* workspace,
                     size_t ws_bytes, void* stream) {
    Sizes s;
    int r = check_layer(layer, &s);
    if (r) return r;
    if (n_tokens < 1 || n_tokens > 0x7fffffff)
        return fail(GDN_EINVAL, "gdn_prefill_host: n_tokens >= 1 required (got %lld)", (long long)n_tokens);
    if (pass_tokens < 0) return fail(GDN_EINVAL, "gdn_prefill_host: pass_tokens >= 0 required");
    if (!x_host || !state_out || !conv_state || !y_host || !workspace) return fail(GDN_EINVAL, "gdn_prefill_host: NULL pointer");
    if (!aligned(workspace, 256)) return fail(GDN_EINVAL, "gdn_prefill_host: workspace 256-byte alignment required");
    if ((r = check_pinned(x_host, "x_host")) || (r = check_pinned(y_host, "y_host"))) return r;
    const bool gates = layer->gate_log_a != nullptr;
    if (gates && ((r = check_pinned(layer->gate_log_a, "gate_log_a")) || (r = check_pinned(layer->gate_b, "gate_b"))))
        return r;
    int64_t B = pass_tokens_for(layer, s, n_tokens, ws_bytes, host_stage_bytes);
    if (B < 1)
        return fail(GDN_ENOMEM, "gdn_prefill_host: workspace %zu B < %zu B needed for one token", ws_bytes,
                    carve(layer, s, 1, nullptr).total + host_stage_bytes(layer, s, 1));
    if (pass_tokens > 0 && pass_tokens < B) B = pass_tokens >= GDN_CHUNK ? pass_tokens - pass_tokens % GDN_CHUNK : pass_tokens;
    const bool q4k = layer->wtype == GDN_W_Q4K;
    const size_t esz = q4k ? 2 : 4;
    Workspace w = carve(layer, s, B, workspace);
    uint8_t* stage = static_cast<uint8_t*>(workspace) + w.total;
    const size_t xb = up256(B * s.H * esz), gbytes = up256(B * s.hv * 4);
    uint8_t* xs[2] = {stage, stage + xb};
    uint8_t* ys[2] = {stage + 2 * xb, stage + 3 * xb};
    float* gas[2] = {nullptr, nullptr};
    float* gbs[2] = {nullptr, nullptr};
    if (gates)
        for (int i = 0; i < 2; ++i) {
            gas[i] = reinterpret_cast<float*>(stage + 4 * xb + (2 * i) * gbytes);
            gbs[i] = reinterpret_cast<float*>(stage + 4 * xb + (2 * i + 1) * gbytes);
        }
    // Pass boundaries, every one a chunk boundary.  The copy-in of the first
    // pass and the copy-out of the last are the ones nothing hides, so those
    // passes are short.  A pass's copy-in takes about a third of the time its
    // tokens take to compute, so when B is a whole number of 8 chunks and the
    // prompt holds the ramps, the passes grow B/8, 3B/8, up to B, and shrink
    // 3B/8, B/8 again (the ragged tail, if any, in the last one); otherwise
    // passes of B, the first and the last B/4 when B is a whole number of 4
    // chunks and there is more than one pass.
    std::vector<int64_t> bounds{0};
    const int64_t e1 = B / 8, e2 = 3 * (B / 8);
    const int64_t n_whole = n_tokens - n_tokens % GDN_CHUNK;
    if (n_tokens > B && B % (8 * GDN_CHUNK) == 0 && n_whole >= 2 * (e1 + e2)) {
        int64_t t = 0;
        for (int64_t len : {e1, e2}) bounds.push_back(t += len);
        const int64_t mid = n_whole - 2 * (e1 + e2);
        if (mid > 0) {
            const int64_t k = (mid + B - 1) / B;
            const int64_t m = ((mid + k - 1) / k + GDN_CHUNK - 1) / GDN_CHUNK * GDN_CHUNK;
            for (int64_t left = mid; left > 0; left -= m) bounds.push_back(t += left < m ? left : m);
        }
        bounds.push_back(t += e2);
        bounds.push_back(n_tokens);
    } else {
        const int64_t qb = B / 4;
        const bool short_ends = n_tokens > B && B % (4 * GDN_CHUNK) == 0;
        int64_t t = short_ends ? qb : (B < n_tokens ? B : n_tokens);
        bounds.push_back(t);
        while (t < n_tokens) {
            int64_t next = t + B < n_tokens ? t + B : n_tokens;
            if (short_ends && next == n_tokens && n_tokens - t > qb) {
                // a short last pass, split on a chunk boundary
                const int64_t split = t + (n_tokens - t - qb) / GDN_CHUNK * GDN_CHUNK;
                if (split > t) next = split;
            }
            t = next;
            bounds.push_back(t);
        }
    }
    const int64_t np = static_cast<int64_t>(bounds.size()) - 1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(copy_streams_mutex());
    CopyStreams* cs = nullptr;
    cudaError_t e = copy_streams(&cs);
    if (e != cudaSuccess) return cuda_fail(e, "gdn_prefill_host: copy streams");
    GDN_LAUNCH(cudaEventRecord(cs->fork, st), "gdn_prefill_host: fork");
    GDN_LAUNCH(cudaStreamWaitEvent(cs->h2d, cs->fork, 0), "gdn_prefill_host: fork");
    GDN_LAUNCH(cudaStreamWaitEvent(cs->d2h, cs->fork, 0), "gdn_prefill_host: fork");

    // Host-to-device copy of pass p into slot p % 2, once pass p - 2 (the
    // previous user of the slot) is done with it.
    auto copy_in = [&](int64_t p) -> int {
        const int64_t u0 = bounds[p], nb = bounds[p + 1] - bounds[p];
        const int slot = static_cast<int>(p & 1);
        if (p >= 2) GDN_LAUNCH(cudaStreamWaitEvent(cs->h2d, cs->pass_done[slot], 0), "gdn_prefill_host: slot wait");
        GDN_LAUNCH(cudaMemcpyAsync(xs[slot], static_cast<const uint8_t*>(x_host) + u0 * s.H * esz, nb * s.H * esz,
                                   cudaMemcpyHostToDevice, cs->h2d),
                   "gdn_prefill_host: copy x");
        if (gates) {
            GDN_LAUNCH(cudaMemcpyAsync(gas[slot], layer->gate_log_a + u0 * s.hv, nb * s.hv * 4, cudaMemcpyHostToDevice,
                                       cs->h2d),
                       "gdn_prefill_host: copy gate_log_a");
            GDN_LAUNCH(cudaMemcpyAsync(gbs[slot], layer->gate_b + u0 * s.hv, nb * s.hv * 4, cudaMemcpyHostToDevice,
                                       cs->h2d),
                       "gdn_prefill_host: copy gate_b");
        }
        GDN_LAUNCH(cudaEventRecord(cs->in_ready[slot], cs->h2d), "gdn_prefill_host: event");
        return GDN_OK;
    };
    auto pipeline = [&]() -> int {
        GDN_LAUNCH(mark(0, true, st), "stage event");
        int rr = q4k ? decode_weights(layer, s, w, st) : GDN_OK;
        if (rr) return rr;
        GDN_LAUNCH(mark(1, true, st), "stage event");
        if ((rr = copy_in(0))) return rr;
        for (int64_t p = 0; p < np; ++p) {
            const int64_t u0 = bounds[p], nb = bounds[p + 1] - bounds[p];
            const int slot = static_cast<int>(p & 1);
            if (p + 1 < np && (rr = copy_in(p + 1))) return rr;
            GDN_LAUNCH(cudaStreamWaitEvent(st, cs->in_ready[slot], 0), "gdn_prefill_host: input wait");
            if (p >= 2) GDN_LAUNCH(cudaStreamWaitEvent(st, cs->out_free[slot], 0), "gdn_prefill_host: output wait");
            rr = run_pass(layer, s, w, xs[slot], nb, gas[slot], gbs[slot], p == 0 ? state_in : state_out, state_out,
                          conv_state, ys[slot], p == 0, st);
            if (rr) return rr;
            GDN_LAUNCH(cudaEventRecord(cs->pass_done[slot], st), "gdn_prefill_host: event");
            GDN_LAUNCH(cudaStreamWaitEvent(cs->d2h, cs->pass_done[slot], 0), "gdn_prefill_host: output wait");
            GDN_LAUNCH(cudaMemcpyAsync(static_cast<uint8_t*>(y_host) + u0 * s.H * esz, ys[slot], nb * s.H * esz,
                                       cudaMemcpyDeviceToHost, cs->d2h),
                       "gdn_prefill_host: copy y");
            GDN_LAUNCH(cudaEventRecord(cs->out_free[slot], cs->d2h), "gdn_prefill_host: event");
        }
        return GDN_OK;
    };
    r = pipeline();
    // Join both copy streams back into the caller's stream on every path.
    const cudaError_t j[4] = {cudaEventRecord(cs->join_h2d, cs->h2d), cudaStreamWaitEvent(st, cs->join_h2d, 0),
                              cudaEventRecord(cs->join_d2h, cs->d2h), cudaStreamWaitEvent(st, cs->join_d2h, 0)};
    if (r) return r;
    for (cudaError_t je : j)
        if (je != cudaSuccess) return cuda_fail(je, "gdn_prefill_host: join");
    return GDN_OK;
}

size_t gdn_batch_workspace_size(const gdn_layer* layer, int64_t n_tokens, int n_seqs) {
    Sizes s;
    if (check_layer(layer, &s) || n_tokens < 0 || n_seqs < 1 || n_seqs > GDN_MAX_SEQS) return 0;
    // every sequence's last chunk may be partial: at most n/64 + n_seqs chunks
    return carve(layer, s, n_tokens > 0 ? n_tokens : 1, nullptr, n_tokens / GDN_CHUNK + n_seqs).total;
}

int gdn_prefill_batch(const gdn_layer* layer, const void* x, const int64_t* cu_seqlens, int n_seqs,
                      const float* state_in, float* state_out, float* conv_state, void* y, void* workspace,
                      size_t ws_bytes, void* stream) {
    Sizes s;
    int r = check_layer(layer, &s);
    if (r) return r;
    if (n_seqs < 1 || n_seqs > GDN_MAX_SEQS)
        return fail(GDN_EINVAL, "gdn_prefill_batch: 1 <= n_seqs <= %d required (got %d)", GDN_MAX_SEQS, n_seqs);
    if (!cu_seqlens) return fail(GDN_EINVAL, "gdn_prefill_batch: cu_seqlens is NULL");
    if (cu_seqlens[0] != 0) return fail(GDN_EINVAL, "gdn_prefill_batch: cu_seqlens[0] must be 0");
    int64_t n_chunks = 0;
    for (int i = 0; i < n_seqs; ++i) {
        if (cu_seqlens[i + 1] < cu_seqlens[i])
            return fail(GDN_EINVAL, "gdn_prefill_batch: cu_seqlens must not decrease (sequence %d)", i);
        n_chunks += (cu_seqlens[i + 1] - cu_seqlens[i] + GDN_CHUNK - 1) / GDN_CHUNK;
    }
    const int64_t T = cu_seqlens[n_seqs];
    if (T > 0x7fffffff) return fail(GDN_EINVAL, "gdn_prefill_batch: more than 2^31 - 1 tokens");
    if (!state_out || !conv_state || !workspace) return fail(GDN_EINVAL, "gdn_prefill_batch: NULL pointer");
    if (T > 0 && (!x || !y)) return fail(GDN_EINVAL, "gdn_prefill_batch: NULL x or y");
    if ((x && !aligned(x, 16)) || (y && !aligned(y, 16)) || !aligned(workspace, 256))
        return fail(GDN_EINVAL, "gdn_prefill_batch: x, y 16-byte and workspace 256-byte alignment required");
    const size_t need = carve(layer, s, T > 0 ? T : 1, nullptr, n_chunks).total;
    if (ws_bytes < need)
        return fail(GDN_ENOMEM, "gdn_prefill_batch: workspace %zu B < %zu B for %lld tokens in %d sequences", ws_bytes,
                    need, (long long)T, n_seqs);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // An empty sequence passes its state through unchanged (its conv state is
    // left as it is by the conv-state kernel).
    const size_t sbytes = static_cast<size_t>(s.hv) * s.d * s.d * 4;
    for (int i = 0; i < n_seqs; ++i) {
        if (cu_seqlens[i + 1] != cu_seqlens[i]) continue;
        float* so = state_out + static_cast<size_t>(i) * sbytes / 4;
        if (!state_in)
            GDN_LAUNCH(cudaMemsetAsync(so, 0, sbytes, st), "gdn_prefill_batch: zero state");
        else if (state_in != state_out)
            GDN_LAUNCH(cudaMemcpyAsync(so, state_in + static_cast<size_t>(i) * sbytes / 4, sbytes,
                                       cudaMemcpyDeviceToDevice, st),
                       "gdn_prefill_batch: copy state");
    }
    if (T == 0) return GDN_OK;

    Workspace w = carve(layer, s, T, workspace, n_chunks);
    const bool q4k = layer->wtype == GDN_W_Q4K;
    GDN_LAUNCH(mark(0, true, st), "stage event");
    if (q4k && (r = decode_weights(layer, s, w, st))) return r;
    GDN_LAUNCH(mark(1, true, st), "stage event");
    // steps 1b, 1c: all tokens of all sequences in one product
    if (q4k) {
        GDN_LAUNCH(launch_quant_rows(static_cast<const uint16_t*>(x), T, s.H, w.xc, w.sx, st), "quantise x");
        GDN_LAUNCH(mark(2, true, st), "stage event");
        cudaError_t e = launch_gemm_codes(w.xc, w.sx, w.wc_in, w.ws_in, T, s.r_in, s.H, w.qkvz, s.n_bf16, s.n_bf16,
                                          w.ba, 2 * s.hv, st);
        if (e != cudaSuccess) return cuda_fail(e, "input projection");
    } else {
        GDN_LAUNCH(mark(2, true, st), "stage event");
        GDN_LAUNCH(launch_gemm_f32(static_cast<const float*>(x), static_cast<const float*>(layer->w_in), T, s.r_in, s.H,
                                   w.qkvz, s.n_bf16, s.n_bf16, w.ba, 2 * s.hv, st),
                   "input projection");
    }
    GDN_LAUNCH(mark(3, true, st), "stage event");
    // step 2 per sequence (its own conv state), in one launch
    GDN_LAUNCH(launch_conv(*layer, w.qkvz, s.n_bf16, T, conv_state, w.ba, 2 * s.hv, w.qkv, w.log_a, w.b, st, cu_seqlens,
                           n_seqs),
               "conv");
    GDN_LAUNCH(launch_conv_state(*layer, w.qkvz, s.n_bf16, T, conv_state, st, cu_seqlens, n_seqs), "conv state");
    GDN_LAUNCH(mark(4, true, st), "stage event");
    // step 3: every sequence chunked from its first token, all in parallel; step 4 after it
    const float* la = layer->gate_log_a ? layer->gate_log_a : w.log_a;
    const float* bb = layer->gate_b ? layer->gate_b : w.b;
    const uint16_t* z = w.qkvz + s.c_conv;
    const TokenRangeHook norm_hook = [&](int64_t t0, int64_t t1, cudaStream_t cs) {
        return launch_gated_norm(*layer, w.o + t0 * s.c_v, z + t0 * s.n_bf16, s.n_bf16, t1 - t0,
                                 w.oc ? w.oc + t0 * s.c_v : nullptr, w.so ? w.so + t0 : nullptr,
                                 w.ohat ? w.ohat + t0 * s.c_v : nullptr, cs);
    };
    GDN_LAUNCH(launch_delta(*layer, w.qkv, la, bb, T, state_in, state_out, w.o, w.delta, st, true, &norm_hook, cu_seqlens,
                            n_seqs),
               "delta rule and gated norm");
    GDN_LAUNCH(mark(5, true, st), "stage event");
    GDN_LAUNCH(mark(6, true, st), "stage event");
    // step 5
    if (q4k) {
        cudaError_t e = launch_gemm_codes(w.oc, w.so, w.wc_out, w.ws_out, T, s.H, s.c_v, static_cast<uint16_t*>(y), s.H,
                                          s.H, nullptr, 0, st);
        if (e != cudaSuccess) return cuda_fail(e, "output projection");
    } else {
        GDN_LAUNCH(launch_gemm_f32(w.ohat, static_cast<const float*>(layer->w_out), T, s.H, s.c_v, nullptr, 0, 0,
                                   static_cast<float*>(y), s.H, st),
                   "output projection");
    }
    GDN_LAUNCH(mark(7, true, st), "stage event");
    return GDN_OK;
}

size_t gdn_decode_workspace_size(const gdn_layer* layer, int n_seqs) {
    Sizes s;
    if (check_layer(layer, &s) || n_seqs < 1 || n_seqs > GDN_MAX_SEQS) return 0;
    return carve_decode(layer, s, n_seqs, nullptr).total;
}

int gdn_decode(const gdn_layer* layer, const void* x, int n_seqs, float* state, float* conv_state, void* y,
               void* workspace, size_t ws_bytes, void* stream) {
    Sizes s;
    int r = check_layer(layer, &s);
    if (r) return r;
    if (n_seqs < 1 || n_seqs > GDN_MAX_SEQS)
        return fail(GDN_EINVAL, "gdn_decode: 1 <= n_seqs <= %d required (got %d)", GDN_MAX_SEQS, n_seqs);
    if (!x || !state || !conv_state || !y || !workspace) return fail(GDN_EINVAL, "gdn_decode: NULL pointer");
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(state, 16) || !aligned(workspace, 256))
        return fail(GDN_EINVAL, "gdn_decode: x, y, state 16-byte and workspace 256-byte alignment required");
    const DecodeWs w = carve_decode(layer, s, n_seqs, workspace);
    if (ws_bytes < w.total) return fail(GDN_ENOMEM, "gdn_decode: workspace %zu B < %zu B", ws_bytes, w.total);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool q4k = layer->wtype == GDN_W_Q4K;
    const int64_t B = n_seqs;
    // Q4_K / Q6_K layers, five launches, each a programmatic dependent of the
    // one before (it starts while that one ends and waits for it before it
    // reads its results; the projections' weight copies start earlier):
    //   steps 1b + 1c: x quantised to packed int8 rows once, then the weight
    //   rows read once against them;
    //   steps 2-4 per (value head, row block, sequence): conv, norms, gates,
    //   one token of the recurrence, gated output o_hat (fp32) and o^2 sums;
    //   step 5: o_hat with the RMS of each head packed once, then the output
    //   weights; that kernel also moves the conv tails up by one token.
    // F32 layers: plain products.
    if (q4k) {
        GDN_LAUNCH(launch_decode_pack(x, false, B, s.H, nullptr, 0, 0, 0, 0.0f, w.xp, w.sx, st), "decode: pack x");
        GDN_LAUNCH(launch_gemv_dot(layer->w_in, layer->q6k_mask & 1, s.r_in, s.H, nullptr, w.xp, decode_pack_stride(s.H),
                                   w.sx, B, w.qkvz, s.n_bf16, s.n_bf16, w.ba, 2 * s.hv, st, nullptr, nullptr, 0, 0, 0),
                   "decode: input projection");
    } else {
        GDN_LAUNCH(launch_gemm_f32(static_cast<const float*>(x), static_cast<const float*>(layer->w_in), B, s.r_in, s.H,
                                   w.qkvz, s.n_bf16, s.n_bf16, w.ba, 2 * s.hv, st),
                   "decode: input projection");
    }
    GDN_LAUNCH(launch_decode_mid(*layer, w.qkvz, s.n_bf16, w.ba, 2 * s.hv, conv_state, B, state, w.ohat, w.psum, st),
               "decode: conv, recurrence and gated norm");
    if (q4k) {
        GDN_LAUNCH(launch_decode_pack(w.ohat, true, B, s.c_v, w.psum, static_cast<int>(s.hv), static_cast<int>(s.d),
                                      DECODE_MID_SPLIT, layer->eps_rms, w.op, w.so, st),
                   "decode: pack o_hat");
        GDN_LAUNCH(launch_gemv_dot(layer->w_out, layer->q6k_mask & 2, s.H, s.c_v, nullptr, w.op,
                                   decode_pack_stride(s.c_v), w.so, B, static_cast<uint16_t*>(y), s.H, s.H, nullptr, 0,
                                   st, conv_state, w.qkvz, s.n_bf16, static_cast<int>(s.c_conv), n_seqs),
                   "decode: conv state and output projection");
    } else {
        GDN_LAUNCH(launch_decode_rms_apply(*layer, w.ohat, w.psum, B, st), "decode: gated-norm RMS");
        std::vector<int64_t> cu(static_cast<size_t>(B) + 1);
        for (int64_t i = 0; i <= B; ++i) cu[static_cast<size_t>(i)] = i;
        GDN_LAUNCH(launch_conv_state(*layer, w.qkvz, s.n_bf16, B, conv_state, st, cu.data(), n_seqs), "decode: conv state");
        GDN_LAUNCH(launch_gemm_f32(w.ohat, static_cast<const float*>(layer->w_out), B, s.H, s.c_v, nullptr, 0, 0,
                                   static_cast<float*>(y), s.H, st),
                   "decode: output projection");
    }
    return GDN_OK;
}

int gdn_decode_gemv(const void* blocks, int q6k, int64_t rows, int64_t cols, const uint16_t* xc, const float* sx,
                   int64_t n, uint16_t* out_bf16, int64_t ld_bf16, int64_t n_bf16, float* out_f32, int64_t ld_f32,
                   void* stream) {
    if (!blocks || !xc || !sx) return fail(GDN_EINVAL, "gdn_decode_gemv: NULL operand");
    if (q6k != 0 && q6k != 1) return fail(GDN_EINVAL, "gdn_decode_gemv: q6k must be 0 or 1");
    if (rows < 1 || rows > 0x7fffffff || cols < 256 || cols > 16384 || cols % 256 || n < 1 || n > GDN_MAX_SEQS)
        return fail(GDN_EINVAL, "gdn_decode_gemv: rows >= 1, cols a multiple of 256 in [256, 16384], 1 <= n <= %d",
                    GDN_MAX_SEQS);
    if (n_bf16 < 0) return fail(GDN_EINVAL, "gdn_decode_gemv: n_bf16 < 0");
    if (n_bf16 > 0 && (!out_bf16 || ld_bf16 < (n_bf16 < rows ? n_bf16 : rows))) return fail(GDN_EINVAL, "gdn_decode_gemv: bf16 output");
    if (n_bf16 < rows && (!out_f32 || ld_f32 < rows - n_bf16)) return fail(GDN_EINVAL, "gdn_decode_gemv: fp32 output");
    if (!aligned(blocks, 16) || !aligned(xc, 16)) return fail(GDN_EINVAL, "gdn_decode_gemv: 16-byte alignment required");
    GDN_LAUNCH(launch_gemv_dot(blocks, q6k == 1, rows, cols, xc, nullptr, 0, sx, n, out_bf16, ld_bf16, n_bf16, out_f32,
                               ld_f32, static_cast<cudaStream_t>(stream), nullptr, nullptr, 0, 0, 0),
               "gdn_decode_gemv");
    return GDN_OK;
}

size_t gdn_attn_workspace_size(int64_t nk, int n_kv_heads, int head_dim) {
    if (nk < 1 || n_kv_heads < 1 || (head_dim != 64 && head_dim != 128 && head_dim != 256)) return 0;
    return attn_workspace_bytes(nk, n_kv_heads, head_dim);
}

int gdn_attn_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t nq, int64_t nk, int n_q_heads,
                     int n_kv_heads, int head_dim, float scale, uint16_t* o, void* workspace, size_t ws_bytes,
                     void* stream) {
    if (!q || !k || !v || !o || !workspace) return fail(GDN_EINVAL, "gdn_attn_prefill: NULL pointer");
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(GDN_EINVAL, "gdn_attn_prefill: head_dim must be 64, 128 or 256 (got %d)", head_dim);
    if (n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads || n_q_heads > 256)
        return fail(GDN_EINVAL, "gdn_attn_prefill: n_q_heads a multiple of n_kv_heads, at most 256 (got %d, %d)",
                    n_q_heads, n_kv_heads);
    if (nq < 1 || nk < nq || nk > 0x7fffffff)
        return fail(GDN_EINVAL, "gdn_attn_prefill: 1 <= nq <= nk < 2^31 required (got %lld, %lld)", (long long)nq,
                    (long long)nk);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(workspace, 16))
        return fail(GDN_EINVAL, "gdn_attn_prefill: 16-byte alignment required");
    if (ws_bytes < attn_workspace_bytes(nk, n_kv_heads, head_dim))
        return fail(GDN_ENOMEM, "gdn_attn_prefill: workspace %zu B < %zu B", ws_bytes,
                    attn_workspace_bytes(nk, n_kv_heads, head_dim));
    const float sc = scale > 0.0f ? scale : 1.0f / sqrtf(static_cast<float>(head_dim));
    cudaError_t e = launch_attn(q, k, v, nq, nk, n_q_heads, n_kv_heads, head_dim, sc, o, workspace,
                                static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue) return fail(GDN_EINVAL, "gdn_attn_prefill: tensor map rejected");
    if (e != cudaSuccess) return cuda_fail(e, "gdn_attn_prefill");
    return GDN_OK;
}

int gdn_sync_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gdn_sync_status");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "gdn_sync_status");
    // every unit's error word is read (and cleared) once
    const int gcode = read_and_clear_gemm_error();
    const int acode = read_and_clear_attn_error();
    const int dcode = read_and_clear_delta_error();
    const int rcode = read_and_clear_decode_error();
    const int ccode = read_and_clear_conv_error();
    const int ncode = read_and_clear_norm_error();
    const int words[] = {read_and_clear_q4k_error(), read_and_clear_q6k_error(), read_and_clear_quant_error(),
                         gcode, ccode, dcode, ncode, rcode, acode};
    const char* units[] = {"Q4_K decode", "Q6_K decode", "activation quantisation", "projection", "conv",
                           "delta-rule", "gated-norm", "decode-step", "attention"};
    for (int i = 0; i < static_cast<int>(sizeof(words) / sizeof(words[0])); ++i)
        if (words[i] == ERR_INDEX)
            return fail(GDN_EINDEX, "an index check of the %s kernel failed (the store was skipped; debug library)",
                        units[i]);
    if (gcode == ERR_WAIT_TIMEOUT) return fail(GDN_ETIMEOUT, "a bounded wait in the projection kernel ran out");
    if (acode == ERR_WAIT_TIMEOUT) return fail(GDN_ETIMEOUT, "a bounded wait in the attention kernel ran out");
    if (ncode == ERR_WAIT_TIMEOUT) return fail(GDN_ETIMEOUT, "a bounded wait in the gated-norm kernel ran out");
    if (dcode == ERR_WAIT_TIMEOUT) return fail(GDN_ETIMEOUT, "a bounded wait in the delta-rule kernel ran out");
    if (rcode == ERR_WAIT_TIMEOUT) return fail(GDN_ETIMEOUT, "a bounded wait in a decode-step kernel ran out");
    if (rcode == ERR_RANGE) return fail(GDN_ERANGE, "a decode-step output o exceeded the fp16 range (|x| > 65504)");
    if (ccode == ERR_RANGE || dcode == ERR_RANGE)
        return fail(GDN_ERANGE, "a %s value exceeded the fp16 operand range (|x| > 65504)",
                    ccode == ERR_RANGE ? "q, k or v" : "delta-rule intermediate (T, A T, S, R or Delta)");
    return GDN_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gdn_delta_rule_noalloc: the delta rule with its scratch in a static device
// array, for callers that must not allocate device memory.  The array's host
// name is only a stand-in; its device address is looked up once per device
// (with that device current) and passed to the kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 256;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kMaxDevices] = {};
}  // namespace

extern "C" int gdn_delta_rule_noalloc(const gdn_layer* layer, const uint16_t* qkv, const float* log_a, const float* b,
                                      int64_t n_tokens, const float* state_in, float* state_out, uint16_t* o,
                                      void* stream) {
    Sizes s;
    int r = check_layer(layer, &s);
    if (r) return r;
    if (n_tokens < 1 || n_tokens > 0x7fffffff) return fail(GDN_EINVAL, "gdn_delta_rule_noalloc: n_tokens >= 1 required");
    if (!qkv || !log_a || !b || !state_out || !o) return fail(GDN_EINVAL, "gdn_delta_rule_noalloc: NULL pointer");
    if (!aligned(qkv, 16) || !aligned(o, 16)) return fail(GDN_EINVAL, "gdn_delta_rule_noalloc: qkv and o 16-byte alignment required");
    const size_t need = delta_scratch_bytes(static_cast<int>(s.hv), static_cast<int>(s.hk), static_cast<int>(s.d), n_tokens);
    if (need > GDN_NOALLOC_SCRATCH_BYTES) {
        const size_t per_chunk = delta_scratch_bytes(static_cast<int>(s.hv), static_cast<int>(s.hk), static_cast<int>(s.d), 1);
        return fail(GDN_EINVAL,
                    "gdn_delta_rule_noalloc: %lld tokens need %zu bytes of scratch, more than the static %u bytes "
                    "(at most %lld tokens for this layer)",
                    (long long)n_tokens, need, GDN_NOALLOC_SCRATCH_BYTES,
                    (long long)(GDN_NOALLOC_SCRATCH_BYTES / per_chunk) * GDN_CHUNK);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "gdn_delta_rule_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(GDN_EINVAL, "gdn_delta_rule_noalloc: device ordinal %d out of range", dev);
    // Outside a stream capture the address is looked up on every call (a
    // cudaDeviceReset reloads the module and may move the array); inside one,
    // the address of this device's last call outside a capture is used.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap);
    if (e != cudaSuccess) return cuda_fail(e, "gdn_delta_rule_noalloc: cudaStreamIsCapturing");
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (cap == cudaStreamCaptureStatusNone) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return cuda_fail(e, "gdn_delta_rule_noalloc: cudaGetSymbolAddress");
            g_noalloc_addr[dev] = p;
        } else if (!g_noalloc_addr[dev]) {
            return fail(GDN_EINVAL, "gdn_delta_rule_noalloc: the first call on a device must come before any stream capture");
        }
        scratch = g_noalloc_addr[dev];
    }
    GDN_LAUNCH(launch_delta(*layer, qkv, log_a, b, n_tokens, state_in, state_out, o, scratch,
                            static_cast<cudaStream_t>(stream), false, nullptr),
               "gdn_delta_rule_noalloc");
    return GDN_OK;
}
