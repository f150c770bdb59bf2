/*
 * gf.h — C-ABI of libgf, a GB300 (sm_103a) engine for the batch-size-1
 * decode step of Llama-style transformers with bf16, int8 weight-only and
 * int4 grouped (G = 32, 64, 128) weight-only linear layers (the workload of
 * the gpt-fast README, sections "Benchmarks" and "Quantization").
 *
 * Conventions for every call below:
 *  - Return value: 0 (GF_OK) or a gf_status code; gf_last_error() returns a
 *    message for the calling thread.  Arguments are checked on the host before
 *    anything is launched; a failed check launches nothing.
 *  - Tensor pointers are DEVICE pointers owned by the caller, 16-byte aligned
 *    (GF_EALIGN otherwise).  The library keeps no reference to them after the
 *    call returns, except for gf_model / gf_kv handles, which the library owns
 *    and which are freed with gf_model_destroy / gf_kv_destroy.
 *  - bf16 is the upper half of an IEEE binary32 (round-to-nearest-even on
 *    conversion), passed as 16-bit words.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous on that stream unless stated; errors raised inside a kernel
 *    (a bounded wait that gave up) are reported by gf_device_error().
 *  - K must be a multiple of 8 (bf16), 16 (int8) or 32 (int4, and of its
 *    group size G), and at most GF_KMAX; otherwise GF_EINVAL.
 */
#ifndef GF_H_
#define GF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GF_OK = 0,
  GF_EINVAL = 1,        /* bad size, dtype or null pointer */
  GF_EALIGN = 2,        /* pointer not 16-byte aligned */
  GF_ECUDA = 3,         /* a CUDA runtime call failed */
  GF_ENOMEM = 4,        /* device allocation failed (model / kv creation only) */
  GF_EUNSUPPORTED = 5,  /* shape outside what the kernels handle */
  GF_EDEVICE = 6        /* a kernel gave up a bounded wait (see gf_device_error) */
} gf_status;

typedef enum { GF_W_BF16 = 0, GF_W_INT8 = 1, GF_W_INT4G32 = 2 } gf_wdtype;
typedef enum { GF_Y_BF16 = 0, GF_Y_F32 = 1 } gf_ydtype;

#define GF_KMAX 14336
#define GF_TILE_ROWS 32

typedef void* gf_stream; /* cudaStream_t */

const char* gf_last_error(void);
int gf_version(void);

/* Size in bytes of a packed weight buffer for an N x K matrix of `wdtype`
 * (the device layout below; int4 with G = 32), or -1 for a bad argument. */
long long gf_packed_bytes(int wdtype, int N, int K);

/*
 * Device layout of the weights ("offline weight repack"; the kernels load
 * boxes of 32 rows x 128 bytes of it with the tensor-memory accelerator,
 * which lays each box out in shared memory with the 128-byte swizzle, so the
 * matrices keep their logical row-major order in memory):
 *  - bf16: the matrix itself, [N][K] 16-bit values.
 *  - int8: [N][K] bytes, the offset code q + 128.
 *  - int4 (group G): [N][K/2] bytes, byte i of a row = code 2i in the low
 *    nibble, code 2i+1 in the high nibble; then, from byte
 *    round_up(N K / 2, 256), the scale/zero words [K/G][Np] (32 bits each,
 *    s | z << 16, bf16 scale and zero of (row, group); Np = N rounded up to 32,
 *    the padding rows zero).  gf_packed_bytes_w4g() gives the size.
 */
long long gf_packed_bytes_w4g(int N, int K, int G);

/* int8 weight-only quantisation (gpt-fast README, "Int8 weight-only
 * quantization"): per output row n, s_n = bf16(max_k |W[n,k]| / 127) (fp32
 * divide) and q = clamp(rint(W / s_n), -127, 127) (fp32 divide, ties to
 * even); an all-zero row gets s = 0, q = 0.
 * W: bf16 [N][K] row-major.  packed: gf_packed_bytes(GF_W_INT8, N, K) bytes
 * in the device layout.  s: bf16 [N]. */
int gf_quantize_w8(const void* W, int N, int K, void* packed, void* s, gf_stream stream);

/* int4 weight-only grouped quantisation, group G along K (gpt-fast README,
 * "Int4 weight-only quantization", --groupsize): per row and group
 * z = min (bf16, exact), s = bf16((max - min) / 15) (fp32 subtract and
 * divide), q = clamp(rint((W - min) / s), 0, 15) (fp32); s == 0 gives q = 0.
 * The dequantised weight is q s + z.  packed (gf_packed_bytes_w4g bytes)
 * receives codes, s and z in the device layout.  G must be 32, 64 or 128 and
 * divide K (GF_EUNSUPPORTED otherwise). */
int gf_quantize_w4g(const void* W, int N, int K, int G, void* packed, gf_stream stream);

/* bf16 weights into the device layout (a copy: the layout is the matrix). */
int gf_repack_bf16(const void* W, int N, int K, void* packed, gf_stream stream);

/* Inverses of the above, for bit-exact checks: packed -> logical.
 * gf_unpack_w8: q int8 [N][K].  gf_unpack_w4g: q uint8 [N][K] (one code per
 * byte), s, z bf16 [N][K/G].  gf_unpack_bf16: W bf16 [N][K]. */
int gf_unpack_w8(const void* packed, int N, int K, void* q, gf_stream stream);
int gf_unpack_w4g(const void* packed, int N, int K, int G, void* q, void* s, void* z,
                  gf_stream stream);
int gf_unpack_bf16(const void* packed, int N, int K, void* W, gf_stream stream);

/* Matrix-vector products y = x W^T of the pages' linear layers at batch
 * size 1: y[n] = sum_k x[k] What[n,k], fp32 accumulation, What = W (bf16),
 * q s_n (int8) or q s + z (int4, group G = 32, 64 or 128).  x: bf16 [K].
 * y: [N] bf16 (rounded to nearest even) or fp32, by ydtype.  Weights stream
 * through shared memory by tensor-memory-accelerator copies; codes are
 * dequantised in registers, one output row per lane.
 * Input range (int8, int4): the codes are read as subnormal floats and the
 * inputs staged multiplied by powers of two up to 2^85, so |x[k]| must stay
 * below 2^43 (larger inputs overflow to inf); inputs below about 2^-60 in
 * magnitude lose relative precision gradually.  bf16 has no such limit. */
int gf_gemv_bf16(const void* x, const void* Wpacked, int N, int K, void* y, int ydtype,
                 gf_stream stream);
int gf_gemv_w8(const void* x, const void* qpacked, const void* s, int N, int K, void* y,
               int ydtype, gf_stream stream);
int gf_gemv_w4g(const void* x, const void* qpacked, int N, int K, int G, void* y, int ydtype,
                gf_stream stream);

/* gf_gemv_bf16 behind a gate, to exercise the bounded device waits: every
 * CTA of the launch first waits until the device word *d_gate (read with
 * acquire semantics) is at least the launch's CTA count (min(ceil(N / 32),
 * SMs); any value >= 65536 opens the gate), for at most wait_ns
 * nanoseconds (0 < wait_ns <= 1e10) in place of the library's 2 s limit.
 * A CTA that gives up records GF_DEVERR_WAIT_GRID in the device error word
 * (gf_device_error), writes nothing to y, waits for its own copies in flight
 * and returns; the launch completes and the context stays usable.  With the
 * gate open the result is that of gf_gemv_bf16.  Nothing in the decode path
 * calls this; it exists for tests of the wait limits and for callers that
 * order a GEMV after a device-side event of their own. */
int gf_gemv_bf16_gated(const void* x, const void* Wpacked, int N, int K, void* y, int ydtype,
                       const unsigned* d_gate, unsigned long long wait_ns, gf_stream stream);

/* Single-query attention of the decode step (the KV-cache attention the
 * gpt-fast model runs at every generated token): for each of Hq heads,
 * o_h = sum_t p_t v_t over positions t = 0..pos (inclusive), p = softmax of
 * q_h . k_t / sqrt(hd), kv head = h / (Hq / Hkv).  q: bf16 [Hq][hd];
 * kcache, vcache: bf16 [Hkv][Tmax][hd]; out: bf16 [Hq][hd].  The position
 * range is split across CTAs and merged with a log-sum-exp combine; the
 * caller provides `ws` of at least gf_attn_workspace_bytes() bytes (scratch,
 * contents undefined after the call).  hd must be 64 or 128, Hq % Hkv == 0,
 * Hq / Hkv <= 4, 0 <= pos < Tmax. */
size_t gf_attn_workspace_bytes(int Hq, int Hkv, int hd);
int gf_decode_attn(const void* q, const void* kcache, const void* vcache, int Hq, int Hkv, int hd,
                   int Tmax, int pos, void* out, void* ws, size_t ws_bytes, gf_stream stream);

/* Decode attention that allocates nothing: the same computation and result
 * as gf_decode_attn, for callers that cannot allocate device memory (a
 * plug-in that only receives tensor pointers from a host framework owning all
 * device memory, or a latency-critical loop that must not call into the CUDA
 * allocator, which can synchronise the device).  The pages have no
 * counterpart of this call; it exists only for such callers.
 * Scratch: a static device array of GF_NOALLOC_ATTN_SCRATCH bytes in the
 * library, held by every GPU that loads the library until the process exits.
 * Shapes needing more (Hq * ceil(SMs / Hkv) * (hd + 2) * 4 bytes, plus 4 per kv
 * head rounded up to 256)
 * return GF_EINVAL with the size in gf_last_error().  Every call looks up
 * the array's device address in the current context (cudaGetSymbolAddress, a
 * host call that allocates nothing), so the address stays right after a
 * context is re-created.  Every call shares the one array: calls
 * that overlap on the same GPU (for example from two streams at once) race
 * and give wrong results; serialise them.  No cudaMalloc / cudaFree is made. */
#define GF_NOALLOC_ATTN_SCRATCH (2 << 20)
int gf_decode_attn_noalloc(const void* q, const void* kcache, const void* vcache, int Hq, int Hkv, int hd,
                           int Tmax, int pos, void* out, gf_stream stream);

/* ------------------------------------------------------ decode step ---- */
typedef struct {
  int d;           /* model width */
  int n_layers;
  int n_heads;     /* query heads */
  int n_kv_heads;  /* key/value heads (grouped-query when < n_heads) */
  int head_dim;    /* 64 or 128 */
  int ffn;         /* SwiGLU hidden width (per expert for MoE) */
  int vocab;
  int n_experts;   /* 0 = dense FFN; else a top-2 mixture of experts */
  float eps;       /* RMSNorm epsilon */
  double theta;    /* RoPE base */
  int group_size;  /* int4 weights: group size along K, 32, 64 or 128 (0 = 32) */
} gf_model_config;

/* Weights as bf16 device arrays owned by the caller (read during
 * gf_model_create only).  Per-layer entries are arrays of n_layers pointers
 * (MoE expert entries: n_layers * n_experts, layer-major).
 *  wqkv  [(Hq + 2 Hkv) hd][d]: rows of Wq, then Wk, then Wv
 *  wo    [d][Hq hd]
 *  wgu   [2 ffn][d]: row 2j = gate row j, row 2j+1 = up row j
 *  wd    [d][ffn]
 *  router [n_experts][d] (MoE only; kept bf16) */
typedef struct {
  const void* embed;    /* [vocab][d], kept bf16 */
  const void* g_final;  /* [d] */
  const void* lm_head;  /* [vocab][d] */
  const void* const* wqkv;
  const void* const* wo;
  const void* const* wgu;
  const void* const* wd;
  const void* const* g_attn;
  const void* const* g_ffn;
  const void* const* router;
} gf_weights;

typedef struct gf_model gf_model;
typedef struct gf_kv gf_kv;

/* Quantises (or repacks) every linear weight, lm_head included, into
 * library-owned device buffers.  Synchronous.  GF_ENOMEM if they do not fit. */
int gf_model_create(const gf_model_config* cfg, int wdtype, const gf_weights* w, gf_model** out);
int gf_model_destroy(gf_model* m);
/* Bytes the model streams per token: linear weights + scales + norm gains +
 * one embedding row (the KV bytes depend on the position and are added by
 * the caller: 2 n_layers Hkv hd 2 (pos+1)). */
long long gf_model_weight_bytes(const gf_model* m);

/* KV cache (bf16 [layer][Hkv][Tmax][hd] for K and for V), RoPE table,
 * scratch and the decode program, for contexts of up to Tmax positions. */
int gf_kv_create(gf_model* m, int Tmax, gf_kv** out);
int gf_kv_destroy(gf_kv* kv);
/* Clears the cache for a new context without allocating: zeroes every K and V
 * row and the engine's step counters (asynchronous on `stream`).  The
 * position lives with the caller (the device int32 passed as d_pos to
 * gf_decode_step / gf_verify_k): set it to 0 to start again from position 0. */
int gf_kv_reset(gf_kv* kv, gf_stream stream);
/* Device pointers of the K and V caches (for tests that pre-fill them). */
int gf_kv_cache_ptrs(gf_kv* kv, void** kcache, void** vcache);

/* Device pointers of the step's activations after the last layer that ran,
 * all fp32: q [Hq hd] (after RoPE), attention output [Hq hd], SwiGLU output
 * [ffn], residual [d] (for tests of intermediate values). */
int gf_kv_activation_ptrs(gf_kv* kv, void** q, void** attn, void** h, void** resid);

/* One decode step at position *d_pos (device int32): embeds *d_token, runs
 * every layer (RMSNorm, q/k/v, RoPE, KV append, attention, o, residual,
 * RMSNorm, SwiGLU or top-2 MoE, residual), the final RMSNorm and lm_head,
 * with fp32 activations and a bf16 KV cache,
 * writes fp32 logits [vocab] to d_logits and their argmax (lowest index on
 * ties) to *d_argmax, then advances *d_pos by one.  One kernel launch on
 * every SM; nothing is copied to the host. */
int gf_decode_step(gf_model* m, gf_kv* kv, const int32_t* d_token, int32_t* d_pos,
                   float* d_logits, int32_t* d_argmax, gf_stream stream);

/* Decode step with a phase trace: as gf_decode_step, and for every phase of
 * the step's program and every CTA, eight 64-bit words are written to d_trace
 * ([phase][cta][8]): %globaltimer ns at phase entry, after the grid barrier,
 * after input staging, after the phase's work, at phase close, and when the
 * CTA's producer finished issuing the phase's copies; then the number of
 * consumer slot waits that found the slot still in flight and of producer
 * waits that found no free slot.  gf_trace_bytes() gives the buffer size. */
size_t gf_trace_bytes(const gf_kv* kv);
int gf_decode_step_traced(gf_model* m, gf_kv* kv, const int32_t* d_token, int32_t* d_pos, float* d_logits,
                          int32_t* d_argmax, unsigned long long* d_trace, gf_stream stream);

/* Speculative verification (gpt-fast README, "Speculative sampling"):
 * d_tokens holds k+1 ids [last accepted token, draft_1 .. draft_k], fed at
 * positions *d_pos .. *d_pos + k in one pass.  With a_i the argmax of row i,
 * n = the largest n <= k with a_{i-1} == draft_i for all i <= n is written to
 * *d_n_accepted, a_n to *d_next_token, and *d_pos advances by n + 1.  KV rows
 * of all k+1 positions are written (rows past the accepted ones are
 * overwritten by later steps).  d_logits, if not NULL, receives the fp32
 * logits [k+1][vocab].  1 <= k+1 <= 8. */
int gf_verify_k(gf_model* m, gf_kv* kv, const int32_t* d_tokens, int k, int32_t* d_pos,
                int32_t* d_n_accepted, int32_t* d_next_token, float* d_logits, gf_stream stream);

/* Batched prefill (gpt-fast README, "Generate text": the prompt before the
 * first generated token): the n device tokens d_tokens are fed at positions
 * *d_pos .. *d_pos + n - 1 in passes of up to 8 rows, each ONE stream of the
 * weights (the verify pass with every row accepted): the K/V rows of all n
 * positions are written and *d_pos advances by n on the device.  The argmax
 * of the last row (the first generated token) goes to *d_next_token and, if
 * d_logits is not NULL (16-byte aligned, [vocab] fp32), that row's logits.
 * The result equals n gf_decode_step calls up to the accumulation order.
 * n >= 1; *d_pos + n <= Tmax (a pass past the cache records
 * GF_DEVERR_BAD_TOKEN and writes nothing, as gf_verify_k). */
int gf_prefill(gf_model* m, gf_kv* kv, const int32_t* d_tokens, int n, int32_t* d_pos,
               int32_t* d_next_token, float* d_logits, gf_stream stream);

/* Greedy generation (gpt-fast README, "Generate text", at batch size 1): the
 * n_prompt host tokens h_prompt are fed one per gf_decode_step from position
 * 0 of kv (earlier contents are overwritten), then n_new tokens are
 * generated, each the argmax of the step fed the one before; they are
 * written to the host array h_out[n_new].  Token ids stay on the device
 * between steps; the call returns after the last one (the stream is
 * synchronised).  n_prompt >= 1, n_new >= 1, n_prompt + n_new <= Tmax.
 * Allocates and frees n_prompt + n_new + 8 ints of device memory. */
int gf_generate(gf_model* m, gf_kv* kv, const int32_t* h_prompt, int n_prompt, int n_new, int32_t* h_out,
                gf_stream stream);

/* Counters of a speculative generation: verify passes, draft tokens
 * proposed (rounds * k), draft tokens the target accepted. */
typedef struct {
  int rounds;
  int drafted;
  int accepted;
} gf_spec_stats;

/* Speculative greedy generation (README, "Speculative sampling"; the draft is
 * the int8 or int4 copy of the target in the README's example): the prompt
 * is fed to both models as in gf_generate.  Then, per round, from the current
 * token t at position p: the draft runs k gf_decode_step calls (t and its own
 * argmaxes at p .. p + k - 1) proposing d_1..d_k; gf_verify_k on the target
 * checks [t, d_1..d_k] at p .. p + k and accepts the longest prefix d_1..d_n
 * equal to its own greedy choices, with next token a_n; d_1..d_n and a_n are
 * emitted, the target's position advances to p + n + 1 and the draft's is
 * set to the same (after one more draft step over d_k when n = k).  The
 * emitted tokens equal gf_generate's on the target wherever the verify pass
 * and the decode step take the same argmax.  h_out receives n_new tokens;
 * *stats (if not NULL) the counters.  1 <= k <= 7, equal vocabularies,
 * distinct KV handles, n_prompt + n_new + k + 1 <= both Tmax.  Synchronises
 * the stream once per round (to read n); returns GF_EDEVICE if a verify pass
 * reports an impossible count (a device error). */
int gf_generate_speculative(gf_model* target, gf_kv* tkv, gf_model* draft, gf_kv* dkv, const int32_t* h_prompt,
                            int n_prompt, int n_new, int k, int32_t* h_out, gf_spec_stats* stats,
                            gf_stream stream);

/* Codes of the device error word: the first failure a launch records. */
enum {
  GF_DEVERR_NONE = 0,
  GF_DEVERR_WAIT_FULL = 1,      /* a consumer warp gave up waiting for a weight slot */
  GF_DEVERR_WAIT_EMPTY = 2,     /* a producer gave up waiting for a free ring slot */
  GF_DEVERR_WAIT_GRID = 3,      /* a CTA gave up waiting at a grid barrier or gate */
  GF_DEVERR_WAIT_CTA = 4,       /* a warp gave up waiting at a CTA barrier */
  GF_DEVERR_DRAIN = 5,          /* a producer gave up waiting for its last copies */
  GF_DEVERR_BAD_PROGRAM = 6,    /* a phase the kernel does not run */
  GF_DEVERR_BAD_POS = 7,        /* *d_pos outside the KV cache */
  GF_DEVERR_BAD_TOKEN = 8,      /* a token id outside the vocabulary */
  GF_DEVERR_WAIT_ROUTER = 9,    /* a producer gave up waiting for the expert choice */
  GF_DEVERR_WAIT_COMBINE = 10,  /* a tile's combine buffer was not handed on in time */
  GF_DEVERR_WAIT_HEAD = 11      /* a kernel gave up waiting for a head's q/k/v rows or output */
};

/* Reads and clears the device error word of the engine (GF_DEVERR_NONE, or
 * the GF_DEVERR_* code of the first wait that gave up or input a kernel
 * refused).  Synchronises the device.  The word is shared by
 * every call in the process.  The library keeps per-device state (the
 * addresses of its device variables, kernel attributes) for the life of the
 * process: do not use it again on a device after cudaDeviceReset. */
int gf_device_error(void);

/* Device-to-device copy at full bandwidth (16-byte vector loads and stores),
 * used as the measured HBM ceiling.  bytes % 16 == 0. */
int gf_copy_ceiling(const void* src, void* dst, size_t bytes, gf_stream stream);

#ifdef __cplusplus
}
#endif
#endif
