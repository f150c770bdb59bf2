// gf_internal.cuh — shared definitions of the sm_103a engine: tile layout
// arithmetic, PTX wrappers (mbarrier, bulk asynchronous copy, acquire/release
// loads), the phase program executed by the persistent kernel, and host-side
// error helpers.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gf.h"

namespace gf {

// ------------------------------------------------------------- layout ----
constexpr int TR = GF_TILE_ROWS;  // rows per tile
constexpr int KBLK = 32;          // chunks per K-block (one per lane)
constexpr int KMAX = GF_KMAX;
enum { DT_BF16 = 0, DT_INT8 = 1, DT_INT4 = 2 };

__host__ __device__ inline int per_chunk(int dt) { return dt == DT_BF16 ? 8 : dt == DT_INT8 ? 16 : 32; }

__host__ __device__ inline long long block_bytes(int dt, int Rt, int Lb) {
  long long b = (long long)Rt * Lb * 16;
  if (dt == DT_INT4) b += ((long long)Rt * Lb * 4 + 15) / 16 * 16;
  return b;
}
// Bytes of a full tile (TR rows, all K-blocks).  With TR a multiple of 4 the
// int4 scale words need no padding, so this is TR times the row bytes.
__host__ __device__ inline long long full_tile_bytes(int dt, int C) {
  return (long long)TR * C * (dt == DT_INT4 ? 20 : 16);
}
__host__ __device__ inline long long packed_bytes(int dt, int N, int K) {
  int C = K / per_chunk(dt);
  long long total = (long long)(N / TR) * full_tile_bytes(dt, C);
  if (N % TR) {
    int Rt = N % TR;
    for (int c0 = 0; c0 < C; c0 += KBLK) total += block_bytes(dt, Rt, C - c0 < KBLK ? C - c0 : KBLK);
  }
  return total;
}
// Byte offset of K-block b of the tile holding row-tile t (rows Rt), and of
// chunk (r, l) inside it.
__host__ __device__ inline long long block_offset(int dt, int C, int t, int Rt, int b) {
  return (long long)t * full_tile_bytes(dt, C) + (long long)b * block_bytes(dt, Rt, KBLK);
}

// ------------------------------------------------------- engine sizes ----
constexpr int NCW = 7;                       // consumer warps per CTA
constexpr int NTHREADS = (NCW + 1) * 32;     // + one producer warp
constexpr int HROWS = 16;                    // rows of a slot: half a tile
constexpr int SLOT_BYTES = 10240;            // codes of 16 rows x 32 chunks + int4 scale words
constexpr int SLOT_SZ_OFF = 8192;            // int4 scale words inside a slot
// Slot X of the CTA's stream (counted over the whole program) belongs to
// consumer warp X % NCW and uses ring entry X % NSLOT.  NSLOT is a multiple
// of NCW, so every ring entry always belongs to the same warp: the previous
// use of the entry a warp waits on is that warp's own, already consumed slot,
// and the mbarrier phase parity it waits for is never ambiguous.
constexpr int NSLOT = 14;
// Half-tile combine buffers, used round-robin by half-tile number; a guard
// word per buffer holds the number of the half-tile allowed to use it next.
constexpr int NTB = 16;
constexpr int OFF_RING = 0;
constexpr int OFF_X = OFF_RING + NSLOT * SLOT_BYTES;     // fp32 x, swizzled
constexpr int OFF_XSUM = OFF_X + KMAX * 4;               // fp32 sums of x per chunk (int8) / group (int4)
constexpr int OFF_TB = OFF_XSUM + (KMAX / 16) * 4 + 256;  // [NTB][NCW][HROWS] partial row sums
constexpr int OFF_TBC = OFF_TB + NTB * NCW * HROWS * 4;  // [NTB] arrival counters, then [NTB] guards
constexpr int OFF_BAR = OFF_TBC + 2 * NTB * 4;           // mbarriers
constexpr int OFF_MISC = OFF_BAR + 320;
constexpr int OFF_PHB = OFF_MISC + 1024;  // red[64] f32, bcast[64] i32, moew[64] f32, spare
constexpr int PHB_BYTES = 256;            // one phase descriptor (two buffers)
constexpr int SMEM_BYTES = OFF_PHB + 2 * PHB_BYTES;
static_assert(OFF_PHB % 16 == 0, "phase descriptor buffers take 16-byte copies");
static_assert(NSLOT % NCW == 0, "ring entries must map to a fixed warp");
static_assert((2 * NSLOT + 1) * 8 <= 320, "mbarrier area");
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
constexpr int ATT_POS_PER_SLOT = 16;
constexpr int FFN_HN = 8;                    // SwiGLU output buffers of a PH_FFN phase (tiles in flight)
// Slots of a down slice in a PH_FFN phase: nsl slots of DR rows, as full as
// the slot size allows (DR a multiple of 8, so every bulk copy is 16-byte
// sized and aligned; the last slot may hold fewer rows), int4 scale words
// right after a slot's DR rows of codes.
constexpr int FFN_MAXSL = 32;                // most down slots per tile
__host__ __device__ inline void ffn_split(int dt, int d, int& nsl, int& DR) {
  const int rowb = dt == DT_INT4 ? 12 : dt == DT_INT8 ? 16 : 32;  // slot bytes per row
  const int maxr = (SLOT_BYTES / rowb) / 8 * 8;
  nsl = (d + maxr - 1) / maxr;
  DR = ((d + nsl - 1) / nsl + 7) / 8 * 8;
}
// shared floats a PH_FFN phase needs above its input: partial outputs, SwiGLU
// buffers and their counters, the down slots' turn counters
__host__ __device__ constexpr int ffn_smem_floats(int d) { return d + FFN_HN * 16 + FFN_HN + 2 * FFN_MAXSL; }
constexpr int MAX_GQ = 4;                    // q heads per kv head (GQA group)
constexpr int MAX_M = 8;                     // rows of a verify pass
constexpr int VTG = 4;                       // tiles per group of a multi-row GEMV phase

// --------------------------------------------------------------- phases --
// PH_FFN: a dense FFN in one phase -- the gate/up GEMV (rows interleaved) and,
// per gate/up tile, the matching 16-column slice of the down projection
// (column-sliced copy W2), accumulated per CTA and added to the residual.
enum PhaseKind { PH_GEMV = 0, PH_ATTN = 1, PH_FFN = 2 };
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
  ERR_WAIT_COMBINE = 10 // a half-tile combine buffer was not handed on in time
};

struct alignas(16) Phase {
  int kind;
  int wait_bar;    // grid barrier to wait on before the phase (-1: none)
  int signal_bar;  // grid barrier to arrive on after the phase (-1: none)
  int rot;         // unit rotation across CTAs
  // GEMV
  int dtype, N, K;
  int epi;
  const uint8_t* W;        // packed weights
  const uint16_t* s8;      // int8 row scales
  const uint8_t* W2;       // PH_FFN: column-sliced down projection [N2][N/2]
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
  int stream_cur;          // 1: the row at pos is in memory before launch (standalone)
  // mixture of experts
  int moe;                 // MoeMode
  int n_experts;
  long long expert_stride; // bytes between consecutive experts' packed matrices
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
  // speculative verification (tokens != nullptr): rows m = 0..M-1 are
  // tokens[m] at pos + m, 1 <= M <= MAX_M
  int M;               // rows of the pass (1 for a decode step)
  const int* tokens;   // [M] token ids (verify)
  int* n_accepted;     // verify outputs
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
int pack_cols(int dt, const void* packed, int N, int K, void* out, cudaStream_t s);
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
