// gf_internal.cuh — shared definitions of the sm_103a engine: the weight
// layout and slot geometry of the bulk copies, the phase program executed by
// the persistent kernel, the shared-memory map, and host-side helpers.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gf.h"

namespace gf {

// ------------------------------------------------------------- layout ----
// Device layout of a weight matrix: slots of 32 rows (one per lane of a
// consumer warp) by 256 bytes of each row, stored one after another (tile t,
// K-slot b at slot t * nb + b), each contiguous so that one bulk copy moves
// it into a shared-memory ring entry.  A slot is 128-byte lines: line
// h * 32 + r (h = 0, 1) holds bytes [256 b + 128 h, 256 b + 128 h + 128) of
// row 32 t + r (zero past the row or the matrix), then for int4 lines 64 + g
// hold the scale/zero words s | z << 16 of the 32 rows for group
// 512 b / G + g.  Inside every line the 16-byte units are stored swizzled:
// unit u of line L at unit u ^ (L & 7), so that the 32 lanes' 16-byte reads of
// one unit of their rows (and their 4-byte reads of one scale line) hit all
// 32 banks.
constexpr int TR = GF_TILE_ROWS;  // rows per tile
constexpr int KMAX = GF_KMAX;
enum { DT_BF16 = 0, DT_INT8 = 1, DT_INT4 = 2 };

__host__ __device__ constexpr int per_chunk(int dt) { return dt == DT_BF16 ? 8 : dt == DT_INT8 ? 16 : 32; }
// K values per slot (256 bytes of each row)
__host__ __device__ constexpr int slot_k(int dt) { return dt == DT_BF16 ? 128 : dt == DT_INT8 ? 256 : 512; }
constexpr int LINE = 128;                    // bytes of a line (the swizzle span)
constexpr int CODE_BYTES = 2 * TR * LINE;    // code lines of a slot
constexpr int SLOT_CHUNKS = 16;              // 16-byte chunks of each row in a slot
__host__ __device__ inline long long round_up(long long a, long long m) { return (a + m - 1) / m * m; }
__host__ __device__ inline int slot_bytes(int dt, int G) { return CODE_BYTES + (dt == DT_INT4 ? (512 / G) * LINE : 0); }
__host__ __device__ inline int k_slots(int dt, int K) { return (K + slot_k(dt) - 1) / slot_k(dt); }
__host__ __device__ inline long long packed_bytes(int dt, int N, int K, int G) {
  return (long long)((N + TR - 1) / TR) * k_slots(dt, K) * slot_bytes(dt, G);
}
// byte of the packed buffer holding byte `kb` of row n's codes
__host__ __device__ inline long long code_addr(int dt, int K, int G, int n, long long kb) {
  const int nb = k_slots(dt, K), b = (int)(kb >> 8), r = n % TR, line = (int)((kb >> 7) & 1) * TR + r;
  const int unit = (int)((kb >> 4) & 7) ^ (line & 7);
  return ((long long)(n / TR) * nb + b) * slot_bytes(dt, G) + (long long)line * LINE + unit * 16 + (kb & 15);
}
// byte of the packed buffer holding the int4 scale/zero word of (row n, group g)
__host__ __device__ inline long long sz_addr(int K, int G, int n, int g) {
  const int nb = k_slots(DT_INT4, K), gps = 512 / G, b = g / gps, gl = g % gps, r = n % TR;
  const int unit = (r >> 2) ^ (gl & 7);  // line 64 + gl: (64 + gl) & 7 == gl & 7
  return ((long long)(n / TR) * nb + b) * slot_bytes(DT_INT4, G) + CODE_BYTES + (long long)gl * LINE + unit * 16 +
         (r & 3) * 4;
}

// ------------------------------------------------------- engine sizes ----
constexpr int NCW = 8;                       // consumer warps per CTA
constexpr int NPROD = 4;                     // producer warps (lane 0 of each issues copies)
constexpr int NTHREADS = (NCW + NPROD) * 32;
constexpr int SLOT_BYTES = 10240;            // ring entry: a slot of any type
// Slot X of the CTA's stream (counted over the whole program) belongs to
// consumer warp X % NCW and uses ring entry X % NSLOT.  NSLOT is a multiple
// of NCW, so every ring entry always belongs to the same warp (two entries
// per warp): the previous use of the entry a warp waits on is that warp's
// own, already consumed slot, and the mbarrier parity it waits for is never
// ambiguous.
constexpr int NSLOT = 2 * NCW;
constexpr int NTB = 4;                       // tile combine buffers (round-robin, guarded)
constexpr int OFF_RING = 0;                  // 128-aligned: a slot's lines map to whole bank rows
constexpr int OFF_X = OFF_RING + NSLOT * SLOT_BYTES;     // fp32 x (staged with the dequantisation powers)
constexpr int OFF_XSUM = OFF_X + KMAX * 4;               // fp32 sums of x per chunk (int8) / group (int4)
constexpr int OFF_TB = OFF_XSUM + (KMAX / 16) * 4;       // [NTB][NCW][TR] partial row sums
constexpr int OFF_TBC = OFF_TB + NTB * NCW * TR * 4;     // [NTB] arrival counters, then [NTB] guards
constexpr int OFF_BAR = OFF_TBC + 2 * NTB * 4;           // mbarriers
constexpr int OFF_MISC = OFF_BAR + (2 * NSLOT + 2) * 8;
// red[128] f32, bcast[192] i32 (fixed slots below 64, the verify argmax
// merge from 64), moew[64] f32, FFN counters [16] i32
constexpr int MISC_BYTES = 2048;
constexpr int OFF_PHB = OFF_MISC + MISC_BYTES;
constexpr int PHB_BYTES = 256;            // one phase descriptor (two buffers)
constexpr int SMEM_USED = OFF_PHB + 2 * PHB_BYTES;
constexpr int SMEM_BYTES = SMEM_USED + 128;  // + slack to align the base to 128
static_assert(SLOT_BYTES % 16 == 0 && SLOT_BYTES >= CODE_BYTES + 16 * LINE, "slot geometry");
static_assert(OFF_BAR % 8 == 0 && OFF_PHB % 16 == 0, "shared-memory alignment");
static_assert(NSLOT % NCW == 0 && NSLOT % NPROD == 0, "ring entries must map to a fixed warp and producer");
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
constexpr int ATT_POS_PER_SLOT = 16;         // positions a warp scores at once (and a slot's most)
// positions of K and V in one ring entry: 8 for head dim 128, 16 for 64
__host__ __device__ constexpr int att_slot_pos(int hd) { return SLOT_BYTES / (4 * hd) >= 16 ? 16 : 8; }
constexpr int FFN_HN = 8;                    // SwiGLU output buffers of a PH_FFN phase (tiles in flight)
constexpr int FFN_MAX_D = 4096;              // widest model the fused FFN handles
// Down projection of a PH_FFN phase: per gate/up tile, the 16 matching
// columns of every output row (a column-sliced copy), split into NCW row
// ranges of RW rows (warp w always owns rows w RW .. w RW + RW - 1, so its
// partial outputs need no synchronisation), each streamed as P pieces of at
// most PR rows (one slot each, as even as the slot size allows).  Row bytes
// per slot: int4 8 code + 4 scale, int8 16, bf16 32.
struct FfnSplit {
  int RW, PR, P;
};
__host__ __device__ inline int ffn_row_bytes(int dt) { return dt == DT_INT4 ? 12 : dt == DT_INT8 ? 16 : 32; }
__host__ __device__ inline FfnSplit ffn_split(int dt, int d) {
  FfnSplit s;
  s.RW = (int)round_up((d + NCW - 1) / NCW, 32);
  const int maxr = SLOT_BYTES / ffn_row_bytes(dt) / 32 * 32;
  s.P = (s.RW + maxr - 1) / maxr;
  s.PR = (int)round_up((s.RW + s.P - 1) / s.P, 32);
  return s;
}
// rows [r0, r1) of piece k of warp w (empty when r0 >= r1)
__host__ __device__ inline void ffn_piece(const FfnSplit& s, int d, int w, int k, int& r0, int& r1) {
  r0 = w * s.RW + k * s.PR;
  r1 = r0 + s.PR;
  const int wend = (w + 1) * s.RW;
  if (r1 > wend) r1 = wend;
  if (r1 > d) r1 = d;
}
constexpr int MAX_GQ = 4;                    // q heads per kv head (GQA group)
constexpr int MAX_M = 8;                     // rows of a verify pass
constexpr int VTG = 8;                       // tiles per group of a multi-row GEMV phase

// --------------------------------------------------------------- phases --
// PH_FFN: a dense FFN in one phase -- the gate/up GEMV (rows interleaved) and,
// per gate/up tile, the matching 16-column slice of the down projection
// (column-sliced copy W2), accumulated per CTA and added to the residual.
// PH_OSPLIT: the o projection split by K-slot: unit (tile, K-slot) waits for
// the attention of the slot's heads, stages those heads' outputs, and adds its
// 32 partial row sums to the residual -- no grid barrier after the attention.
enum PhaseKind { PH_GEMV = 0, PH_ATTN = 1, PH_FFN = 2, PH_OSPLIT = 3 };
enum XSrc { X_NONE = 0, X_BF16 = 1, X_NORM = 2, X_EMBED_NORM = 3, X_F32 = 4 };
enum Epi {
  EPI_STORE_BF16 = 0,
  EPI_STORE_F32 = 1,
  EPI_QKV = 2,       // RoPE q and k; q -> fp32 q buffer, k, v -> bf16 cache row at pos
  EPI_RESID = 3,     // resid[n] += y
  EPI_SWIGLU = 4,    // h[n/2] = silu(gate) * up (fp32)
  EPI_LOGITS = 5,    // logits[n] = y (fp32), running argmax
  EPI_MOE_SWIGLU = 6,  // h[slot * F + n/2] = silu(gate) * up for the slot's expert
  EPI_MOE_RESID = 7    // resid[n] += w[slot] * y
};
// Mixture-of-experts role of a GEMV phase: MOE_GU runs the router and then the
// gate/up rows of the two chosen experts (2 * N_e rows); MOE_DOWN0 / 1 run the
// down projection of the first / second chosen expert.
enum MoeMode { MOE_NONE = 0, MOE_GU = 1, MOE_DOWN0 = 2, MOE_DOWN1 = 3, MOE_DOWNU = 4 };
// In a verify pass (several rows) MOE_GU streams the union of the experts the
// rows chose (each expert once, in index order) and MOE_DOWNU the down
// projections of that union.
enum ErrCode {
  ERR_NONE = 0,
  ERR_WAIT_FULL = 1,
  ERR_WAIT_EMPTY = 2,
  ERR_WAIT_GRID = 3,
  ERR_WAIT_CTA = 4,
  ERR_DRAIN = 5,
  ERR_BAD_PROGRAM = 6,
  ERR_BAD_POS = 7,    // *d_pos outside [0, Tmax)
  ERR_BAD_TOKEN = 8,  // token id outside [0, vocab)
  ERR_WAIT_ROUTER = 9, // the producer gave up waiting for the expert choice
  ERR_WAIT_COMBINE = 10, // a tile combine buffer was not handed on in time
  ERR_WAIT_HEAD = 11   // an attention unit gave up waiting for its head's q/k/v rows
};

struct alignas(16) Phase {
  int kind;
  int wait_bar;    // grid barrier to wait on before the phase (-1: none)
  int signal_bar;  // grid barrier to arrive on after the phase (-1: none)
  int rot;         // unit rotation across CTAs
  // GEMV
  int dtype, N, K, G;      // G: int4 group size
  int epi;
  int pad0;
  const uint8_t* W;        // packed matrix (experts back to back)
  unsigned* attd;          // [Hkv] attention of each kv group finished (PH_ATTN signals, PH_OSPLIT waits)
  const uint16_t* s8;      // int8 row scales
  const uint8_t* W2;       // PH_FFN: column-sliced down projection
  const uint16_t* s8b;     // PH_FFN: its int8 row scales
  int N2;                  // PH_FFN: rows of the down projection (the model width)
  int xsrc;
  const void* xptr;        // bf16 or fp32 vector, or the fp32 residual for X_NORM
  const uint16_t* gain;    // RMSNorm gain
  float eps;
  void* out;               // epilogue target
  int q_rows, kv_rows;     // EPI_QKV split
  // attention (also used by EPI_QKV)
  void* qbuf;              // q: fp32 (q_f32) or bf16 [Hq][hd]
  uint16_t* kc;            // cache base for this layer [Hkv][Tmax][hd]
  uint16_t* vc;
  void* attn_out;          // fp32 (out_f32) or bf16 [Hq][hd]
  int q_f32, out_f32;
  int Hq, Hkv, hd, Tmax;
  float* part;             // [Hq][nch_max][hd + 2] partials
  unsigned* tick;          // [Hkv] combine tickets
  unsigned* headc;         // [Hkv] q/k/v tiles of each kv group finished (nullptr: no wait)
  int stream_cur;          // 1: the row at pos is in memory before launch (standalone)
  // mixture of experts
  int moe;                 // MoeMode
  int n_experts;
  const uint16_t* router;  // [n_experts][K] bf16 (MOE_GU)
  // multi-row (verify) input addressing: row m, expert segment e of X_F32
  int x_mstride;           // floats between rows
  long long x_sstride;     // floats between experts (MOE_DOWNU)
  long long out_mstride;   // elements between rows of the epilogue target
};
static_assert(sizeof(Phase) % 16 == 0 && sizeof(Phase) <= PHB_BYTES, "phase descriptor copies");

// Split of a decode attention over positions 0..T-1 into nch chunks of CH
// positions per kv head (CH a multiple of the slot size, chunks of at least
// ATT_MIN_CHUNK positions so that short contexts stay in one CTA and skip the
// cross-CTA merge), aiming at about `target` units in all.  Kernel and host
// use this one definition.
constexpr int ATT_MIN_CHUNK = 256;           // positions per chunk, at least
__host__ __device__ inline void attn_split(int T, int Hkv, int target, int& CH, int& nch) {
  int want = (target + Hkv - 1) / Hkv;
  if (want < 1) want = 1;
  const int maxch = (T + ATT_MIN_CHUNK - 1) / ATT_MIN_CHUNK;
  nch = want < maxch ? want : maxch;
  CH = ((T + nch - 1) / nch + ATT_POS_PER_SLOT - 1) / ATT_POS_PER_SLOT * ATT_POS_PER_SLOT;
  nch = (T + CH - 1) / CH;
}

struct Params {
  const Phase* prog;   // device program (nullptr: use `single`)
  int nphases;
  int dtype;           // weight type of the program's GEMV phases (selects the kernel)
  Phase single;
  const int* d_pos;    // current position (nullptr: use pos_const)
  int pos_const;
  int nctas;           // CTAs taking part (grid size)
  int unit_target;     // attention split target (normally the SM count)
  unsigned* bars;      // grid barrier counters (zeroed before launch)
  int* err;
  const float2* rope;  // [Tmax][hd/2] cos, sin
  float* resid;        // fp32 residual [d]
  const uint16_t* embed;
  const int* token;
  float* logits;
  int* argmax;
  float* amax_val;     // [nctas]
  int* amax_idx;       // [nctas]
  unsigned* amax_tick;
  int* pos_inc;        // advanced by one at the end (nullptr: no)
  int vocab;
  int tmax;            // positions must lie in [0, tmax) (0: not checked)
  unsigned long long* trace;  // [nphases][nctas][TRACE_W] timestamps and counters (nullptr: off)
  unsigned long long wait_ns;  // limit of every bounded wait (0: the default, 2 s)
  // speculative verification (tokens != nullptr): rows m = 0..M-1 are
  // tokens[m] at pos + m, 1 <= M <= MAX_M
  int M;               // rows of the pass (1 for a decode step)
  const int* tokens;   // [M] token ids (verify)
  int* n_accepted;     // verify outputs
  int prefill;         // verify program as a prefill pass: every row accepted (n = M - 1)
  int* next_token;
  float* hbuf_moe;     // verify MoE: [MAX_M][8][ffn] SwiGLU outputs per row and expert
};
// Trace record of one CTA in one phase (ns of %globaltimer, then counters):
// 0 phase entered, 1 grid barrier passed, 2 input staged, 3 units done,
// 4 phase closed, 5 producer finished issuing the phase, 6 consumer slot
// waits that found the slot empty, 7 producer waits that found no free slot.
constexpr int TRACE_W = 8;

// A launch is a verification pass when it carries its rows' tokens.
__host__ __device__ __forceinline__ bool verifying(const Params& P) { return P.tokens != nullptr; }

// ------------------------------------------------------------ host side --
void set_error(const char* fmt, ...);
long long cols_bytes(int dt, int N, int K);
int pack_cols(int dt, const void* packed, int N, int K, int G, void* out, cudaStream_t s);
int quantize_rows(int dt, const void* W, int N, int K, int G, void* packed, void* s8, cudaStream_t s);
int cuda_fail(cudaError_t e, const char* what);
#define GF_CUDA(call)                                        \
  do {                                                       \
    cudaError_t e_ = (call);                                 \
    if (e_ != cudaSuccess) return gf::cuda_fail(e_, #call);  \
  } while (0)
inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
int device_sms();
int launch_engine(const Params& p, int grid, bool cooperative, cudaStream_t s);
int* device_err_ptr();

}  // namespace gf
