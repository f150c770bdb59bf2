// engine.cu — the persistent phase engine of libgf (sm_103a).
//
// One CTA per SM runs a program of phases (a single GEMV or attention for the
// standalone calls; every layer of a decode step for gf_decode_step).  In
// each CTA one producer thread streams the CTA's weight blocks (and KV-cache
// rows) from HBM into a ring of shared-memory slots with bulk asynchronous
// copies (cp.async.bulk, completion counted on an mbarrier, L2 evict-first
// hint), running ahead across phase boundaries because the weight stream does
// not depend on activations.  Eight consumer warps wait for each slot,
// dequantise int8 / int4 codes in registers against an fp32 copy of the input
// vector held in shared memory, and release the slot.  Dependent phases are
// separated by grid barriers (cooperative launch); every wait in the kernel is
// bounded by a 2-second clock, after which the kernel records an error code,
// drains its own copies in flight and returns.
//
// The decode step computed here is the batch-size-1 autoregressive step of
// the gpt-fast README ("Benchmarks", "Quantization"): RMSNorm, q/k/v, RoPE,
// KV append, single-query attention, o projection, residual, RMSNorm, SwiGLU,
// residual, final RMSNorm, lm_head, greedy argmax.
#include <math.h>

#include "gf_internal.cuh"

namespace gf {

__device__ int g_err_word;

// ------------------------------------------------------------- PTX glue --
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ int ld_relaxed(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

constexpr uint64_t WAIT_NS = 2000000000ull;

__device__ __noinline__ bool mbar_wait_slow(uint64_t* b, uint32_t parity, int* err, int code) {
  const uint64_t t0 = gtimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(b, parity)) return true;
    if ((it & 31) == 0) {
      if (ld_relaxed(err)) return false;
      if (gtimer() - t0 > WAIT_NS) {
        atomicCAS(err, 0, code);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, int* err, int code) {
  if (mbar_test(b, parity)) return true;
  return mbar_wait_slow(b, parity, err, code);
}

__device__ __noinline__ bool grid_wait(const unsigned* bar, unsigned target, int* err) {
  const uint64_t t0 = gtimer();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire(bar) >= target) return true;
    __nanosleep(40);
    if ((it & 15) == 15) {
      if (ld_relaxed(err)) return false;
      if (gtimer() - t0 > WAIT_NS) {
        atomicCAS(err, 0, ERR_WAIT_GRID);
        return false;
      }
    }
  }
}
__device__ __forceinline__ void grid_arrive(unsigned* bar) {
  __threadfence();
  atomicAdd(bar, 1u);
}

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
__device__ __forceinline__ float rbf(float f) { return bf2f(f2bf(f)); }

// ---------------------------------------------------------- shared state --
struct Smem {
  uint8_t* ring;
  float* xs;       // fp32 input vector, swizzled per chunk
  float4* xsum;    // per-chunk sums of the input vector
  uint64_t* full;  // [NSLOT]
  uint64_t* empty; // [NSLOT]
  uint64_t* cbar;  // consumer-warps barrier
  float* red;      // [64] reduction scratch
  int* bcast;      // [8] broadcast ints
};

__device__ __forceinline__ Smem smem_layout(uint8_t* base) {
  Smem s;
  s.ring = base + OFF_RING;
  s.xs = reinterpret_cast<float*>(base + OFF_X);
  s.xsum = reinterpret_cast<float4*>(base + OFF_XSUM);
  s.full = reinterpret_cast<uint64_t*>(base + OFF_BAR);
  s.empty = s.full + NSLOT;
  s.cbar = s.empty + NSLOT;
  s.red = reinterpret_cast<float*>(base + OFF_MISC);
  s.bcast = reinterpret_cast<int*>(base + OFF_MISC + 256);
  return s;
}

__device__ __forceinline__ int first_unit(int cta, int rot, int G) { return ((cta - rot) % G + G) % G; }

__device__ __forceinline__ void attn_split(int T, int Hkv, int target, int& CH, int& nch) {
  int want = (target + Hkv - 1) / Hkv;
  if (want < 1) want = 1;
  int maxch = (T + 31) / 32;
  nch = want < maxch ? want : maxch;
  CH = ((T + nch - 1) / nch + 31) / 32 * 32;
  nch = (T + CH - 1) / CH;
}

__device__ __forceinline__ const Phase& phase_at(const Params& P, int i) { return P.prog ? P.prog[i] : P.single; }

// ============================================================ producer ====
struct Prod {
  uint32_t it;
  uint64_t pol;
  uint32_t blocked;
};

__device__ __forceinline__ bool prod_slot(const Smem& S, Prod& pr, int* err, uint8_t*& dst, uint64_t*& fb) {
  const uint32_t slot = pr.it % NSLOT, use = pr.it / NSLOT;
  if (use > 0 && !mbar_test(&S.empty[slot], (use - 1) & 1u)) {
    ++pr.blocked;
    if (!mbar_wait_slow(&S.empty[slot], (use - 1) & 1u, err, ERR_WAIT_EMPTY)) return false;
  }
  dst = S.ring + slot * SLOT_BYTES;
  fb = &S.full[slot];
  ++pr.it;
  return true;
}

__device__ void producer(const Params& P, const Smem& S, int cta, int pos) {
  Prod pr;
  pr.it = 0;
  pr.blocked = 0;
  pr.pol = evict_first_policy();
  int* err = P.err;
  const int G = P.nctas;
  bool ok = true;
  for (int pi = 0; pi < P.nphases && ok; ++pi) {
    const Phase& ph = phase_at(P, pi);
    if (ph.kind == PH_GEMV) {
      const int dt = ph.dtype, C = ph.K / per_chunk(dt);
      const int ntiles = (ph.N + TR - 1) / TR, nb = (C + KBLK - 1) / KBLK;
      for (int t = first_unit(cta, ph.rot, G); t < ntiles && ok; t += G) {
        const int Rt = min(TR, ph.N - t * TR);
        for (int b = 0; b < nb; ++b) {
          const int Lb = min(KBLK, C - b * KBLK);
          const uint32_t bytes = (uint32_t)block_bytes(dt, Rt, Lb);
          uint8_t* dst;
          uint64_t* fb;
          if (!(ok = prod_slot(S, pr, err, dst, fb))) break;
          mbar_expect_tx(fb, bytes);
          bulk_g2s(dst, ph.W + block_offset(dt, C, t, Rt, b), bytes, fb, pr.pol);
        }
      }
    } else if (ph.kind == PH_ATTN) {
      const int T = pos + 1, Ts = ph.stream_cur ? T : T - 1;
      int CH, nch;
      attn_split(T, ph.Hkv, P.unit_target, CH, nch);
      const int nunits = ph.Hkv * nch;
      const uint32_t rowb = (uint32_t)ph.hd * 2;
      for (int u = first_unit(cta, ph.rot, G); u < nunits && ok; u += G) {
        const int h = u / nch, c = u % nch;
        const int p0 = c * CH, p1 = min(p0 + CH, T), pe = min(p1, Ts);
        for (int p = p0; p < pe; p += ATT_POS_PER_SLOT) {
          const int np = min(ATT_POS_PER_SLOT, pe - p);
          uint8_t* dst;
          uint64_t* fb;
          if (!(ok = prod_slot(S, pr, err, dst, fb))) break;
          const size_t off = ((size_t)h * ph.Tmax + p) * ph.hd;
          mbar_expect_tx(fb, 2u * np * rowb);
          bulk_g2s(dst, ph.kc + off, np * rowb, fb, pr.pol);
          bulk_g2s(dst + ATT_POS_PER_SLOT * rowb, ph.vc + off, np * rowb, fb, pr.pol);
        }
      }
    }
    if (P.trace) {
      unsigned long long* tr = P.trace + ((size_t)pi * G + cta) * TRACE_W;
      tr[5] = gtimer();
      tr[7] = pr.blocked;
      pr.blocked = 0;
    }
  }
  // Drain: never leave the CTA with bulk copies still writing its shared
  // memory.  The last min(it, NSLOT) slots are the only ones that can be in
  // flight; wait for each one's completion (bounded).
  const uint32_t n = pr.it < (uint32_t)NSLOT ? pr.it : (uint32_t)NSLOT;
  for (uint32_t k = 0; k < n; ++k) {
    const uint32_t i = pr.it - 1 - k, slot = i % NSLOT, use = i / NSLOT;
    const uint64_t t0 = gtimer();
    while (!mbar_test(&S.full[slot], use & 1u)) {
      if (gtimer() - t0 > WAIT_NS) {
        atomicCAS(err, 0, ERR_DRAIN);
        break;
      }
    }
  }
}

// ============================================================ consumers ===
struct Cons {
  uint32_t it;      // ring position
  uint32_t cphase;  // parity of the consumer barrier
  int warp, lane, ctid;
  uint32_t starved; // slot waits that found the slot not yet filled (warp 0)
};

// all consumer warps meet; false if the wait gave up
__device__ __forceinline__ bool cta_sync(const Smem& S, Cons& cs, int* err) {
  __syncwarp();
  mbar_arrive(S.cbar);
  int ok = 1;
  if (cs.lane == 0) ok = mbar_wait(S.cbar, cs.cphase, err, ERR_WAIT_CTA);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok && cs.lane) mbar_test(S.cbar, cs.cphase);  // acquire for this lane (phase already complete)
  cs.cphase ^= 1u;
  return ok != 0;
}

__device__ __forceinline__ bool slot_acquire(const Smem& S, Cons& cs, int* err, const uint8_t*& base) {
  const uint32_t slot = cs.it % NSLOT, par = (cs.it / NSLOT) & 1u;
  int ok = 1;
  if (cs.lane == 0 && !mbar_test(&S.full[slot], par)) {
    ++cs.starved;
    ok = mbar_wait_slow(&S.full[slot], par, err, ERR_WAIT_FULL);
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok && cs.lane) mbar_test(&S.full[slot], par);
  base = S.ring + slot * SLOT_BYTES;
  return ok != 0;
}
__device__ __forceinline__ void slot_release(const Smem& S, Cons& cs) {
  __syncwarp();
  if (cs.lane == 0) mbar_arrive(&S.empty[cs.it % NSLOT]);
  ++cs.it;
}

// ------------------------------------------------------ input staging ----
__device__ __forceinline__ int swz(int g, int U) { return ((g * U) >> 3) & (U - 1); }

// Stages the phase's input vector into shared memory (fp32, swizzled per
// chunk) with per-chunk sums used by the int8 / int4 dequantisation.
__device__ bool stage_x(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta) {
  const int K = ph.K, dt = ph.dtype, E = per_chunk(dt), U = E / 4, C = K / E;
  const int NT = NCW * 32;
  float r = 1.0f;
  const float* res = nullptr;
  const uint16_t* emb = nullptr;
  if (ph.xsrc == X_NORM || ph.xsrc == X_EMBED_NORM) {
    if (ph.xsrc == X_NORM) {
      res = reinterpret_cast<const float*>(ph.xptr);
    } else {
      emb = P.embed + (size_t)(*P.token) * K;
    }
    float ss = 0.0f;
    for (int k = cs.ctid * 4; k < K; k += NT * 4) {
      float4 v;
      if (res) {
        v = __ldcg(reinterpret_cast<const float4*>(res + k));
      } else {
        const uint2 h = *reinterpret_cast<const uint2*>(emb + k);
        v = make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xFFFF0000u), __uint_as_float(h.y << 16),
                        __uint_as_float(h.y & 0xFFFF0000u));
        if (cta == 0) *reinterpret_cast<float4*>(P.resid + k) = v;
      }
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (cs.lane == 0) S.red[cs.warp] = ss;
    if (!cta_sync(S, cs, P.err)) return false;
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) tot += S.red[w];
    r = 1.0f / sqrtf(tot / (float)K + ph.eps);
  }
  float4* xs4 = reinterpret_cast<float4*>(S.xs);
  for (int g = cs.ctid; g < C; g += NT) {
    const int k0 = g * E;
    float se = 0.0f, so = 0.0f;
    for (int u = 0; u < U; ++u) {
      float v[4];
      if (ph.xsrc == X_BF16) {
        const uint2 h = __ldcg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(ph.xptr) + k0 + 4 * u));
        v[0] = __uint_as_float(h.x << 16);
        v[1] = __uint_as_float(h.x & 0xFFFF0000u);
        v[2] = __uint_as_float(h.y << 16);
        v[3] = __uint_as_float(h.y & 0xFFFF0000u);
      } else {
        float4 a;
        if (res) {
          a = __ldcg(reinterpret_cast<const float4*>(res + k0 + 4 * u));
        } else {
          const uint2 h = *reinterpret_cast<const uint2*>(emb + k0 + 4 * u);
          a = make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xFFFF0000u), __uint_as_float(h.y << 16),
                          __uint_as_float(h.y & 0xFFFF0000u));
        }
        const uint2 gg = *reinterpret_cast<const uint2*>(ph.gain + k0 + 4 * u);
        v[0] = rbf(a.x * r * __uint_as_float(gg.x << 16));
        v[1] = rbf(a.y * r * __uint_as_float(gg.x & 0xFFFF0000u));
        v[2] = rbf(a.z * r * __uint_as_float(gg.y << 16));
        v[3] = rbf(a.w * r * __uint_as_float(gg.y & 0xFFFF0000u));
      }
      se += v[0] + v[2];
      so += v[1] + v[3];
      xs4[g * U + (u ^ swz(g, U))] = make_float4(v[0], v[1], v[2], v[3]);
    }
    if (dt == DT_INT4) S.xsum[g] = make_float4(-se, -so, se + so, 0.0f);
    else if (dt == DT_INT8) S.xsum[g] = make_float4(-1.5f * se, -1.5f * so, 0.0f, 0.0f);
  }
  return cta_sync(S, cs, P.err);
}

// ------------------------------------------------------ GEMV compute -----
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// int4: view i of a code word (rotated right by 8i) carries code k = 8j+2i in
// bits 15..18 and k = 8j+2i+1 in bits 19..22.  OR-ing the exponent of 1.0f
// turns them into 1 + q/256 and 1 + q/16 exactly; the per-group offsets are
// removed through the staged sums (accumulator initialised to -sum x).
__device__ __forceinline__ float2 dot_int4(const uint4 c, const float2* x2, float2 acc) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = i ? __funnelshift_r(w[j], w[j], 8 * i) : w[j];
      const float lo = __uint_as_float((v & 0x00078000u) | 0x3F800000u);
      const float hi = __uint_as_float((v & 0x00780000u) | 0x3F800000u);
      acc = ffma2(make_float2(lo, hi), x2[4 * j + i], acc);
    }
  }
  return acc;
}
// int8: view i carries code k = 4j+i in bits 15..22; XOR with 0x3FC00000 sets
// the exponent of 1.0f and flips the sign bit, giving 1 + (q + 128)/256.
__device__ __forceinline__ float2 dot_int8(const uint4 c, const float2* x2, float2 acc) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float f[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = i ? __funnelshift_r(w[j], w[j], 8 * i) : w[j];
      f[i] = __uint_as_float((v & 0x007F8000u) ^ 0x3FC00000u);
    }
    acc = ffma2(make_float2(f[0], f[1]), x2[2 * j], acc);
    acc = ffma2(make_float2(f[2], f[3]), x2[2 * j + 1], acc);
  }
  return acc;
}
__device__ __forceinline__ float2 dot_bf16(const uint4 c, const float2* x2, float2 acc) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 4; ++j)
    acc = ffma2(make_float2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u)), x2[j], acc);
  return acc;
}

// Sum of each of the warp's 4 rows over the 32 lanes; lane l ends with row
// 2*bit4(l) + bit3(l).
__device__ __forceinline__ float warp_rows4(const float v[4], int lane) {
  const bool h16 = lane & 16;
  float k0 = h16 ? v[2] : v[0], k1 = h16 ? v[3] : v[1];
  const float s0 = h16 ? v[0] : v[2], s1 = h16 ? v[1] : v[3];
  k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  const bool h8 = lane & 8;
  float keep = h8 ? k1 : k0;
  const float send = h8 ? k0 : k1;
  keep += __shfl_xor_sync(0xffffffffu, send, 8);
  keep += __shfl_xor_sync(0xffffffffu, keep, 4);
  keep += __shfl_xor_sync(0xffffffffu, keep, 2);
  keep += __shfl_xor_sync(0xffffffffu, keep, 1);
  return keep;
}

struct ArgMax {
  float v;
  int i;
};
__device__ __forceinline__ void amax_merge(ArgMax& a, float v, int i) {
  if (v > a.v || (v == a.v && i < a.i)) {
    a.v = v;
    a.i = i;
  }
}

template <int DT>
__device__ bool gemv_unit(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int t, int pos, ArgMax& am) {
  constexpr int E = DT == DT_BF16 ? 8 : DT == DT_INT8 ? 16 : 32;
  constexpr int U = E / 4;
  const int C = ph.K / E, nb = (C + KBLK - 1) / KBLK;
  const int Rt = min(TR, ph.N - t * TR);
  const int lane = cs.lane, w = cs.warp;
  float yacc[RPW] = {0.f, 0.f, 0.f, 0.f};
  float2 acc2[RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i) acc2[i] = make_float2(0.f, 0.f);
  const float4* xs4 = reinterpret_cast<const float4*>(S.xs);

  for (int b = 0; b < nb; ++b) {
    const int Lb = min(KBLK, C - b * KBLK);
    const uint8_t* base;
    if (!slot_acquire(S, cs, P.err, base)) return false;
    if (lane < Lb) {
      const int g = b * KBLK + lane;
      float4 xv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) xv[u] = xs4[g * U + (u ^ swz(g, U))];
      const float2* x2 = reinterpret_cast<const float2*>(xv);
      float4 xsm = make_float4(0.f, 0.f, 0.f, 0.f);
      if (DT != DT_BF16) xsm = S.xsum[g];
      uint4 code[RPW];
      uint32_t sz[RPW];
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        const int r = w * RPW + i;
        if (r < Rt) {
          code[i] = *reinterpret_cast<const uint4*>(base + (r * Lb + lane) * 16);
          if (DT == DT_INT4) sz[i] = *reinterpret_cast<const uint32_t*>(base + Rt * Lb * 16 + (r * Lb + lane) * 4);
        }
      }
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        const int r = w * RPW + i;
        if (r < Rt) {
          if (DT == DT_INT4) {
            const float2 a = dot_int4(code[i], x2, make_float2(xsm.x, xsm.y));
            const float Sq = fmaf(256.0f, a.x, 16.0f * a.y);
            const float s = __uint_as_float(sz[i] << 16), z = __uint_as_float(sz[i] & 0xFFFF0000u);
            yacc[i] = fmaf(s, Sq, fmaf(z, xsm.z, yacc[i]));
          } else if (DT == DT_INT8) {
            acc2[i] = __fadd2_rn(acc2[i], make_float2(xsm.x, xsm.y));
            acc2[i] = dot_int8(code[i], x2, acc2[i]);
          } else {
            acc2[i] = dot_bf16(code[i], x2, acc2[i]);
          }
        }
      }
    }
    slot_release(S, cs);
  }

  float v[RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i) v[i] = DT == DT_INT4 ? yacc[i] : acc2[i].x + acc2[i].y;
  float y = warp_rows4(v, lane);
  const int ri = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
  const int row = w * RPW + ri;
  const int n = t * TR + row;
  const bool own = (lane & 7) == 0 && row < Rt;
  if (DT == DT_INT8 && own) y *= 256.0f * bf2f(ph.s8[n]);
  // pair partner (rows 2i, 2i+1 sit in lanes l and l^8)
  const float yp = __shfl_xor_sync(0xffffffffu, y, 8);
  if (!own) return true;
  switch (ph.epi) {
    case EPI_STORE_BF16:
      reinterpret_cast<uint16_t*>(ph.out)[n] = f2bf(y);
      break;
    case EPI_STORE_F32:
      reinterpret_cast<float*>(ph.out)[n] = y;
      break;
    case EPI_RESID: {
      float* res = reinterpret_cast<float*>(ph.out);
      res[n] = __ldcg(res + n) + rbf(y);
      break;
    }
    case EPI_SWIGLU: {
      if ((ri & 1) == 0) {  // even row = gate j, odd row = up j
        const float gt = rbf(y), up = rbf(yp);
        const float h = gt / (1.0f + expf(-gt)) * up;
        reinterpret_cast<uint16_t*>(ph.out)[n >> 1] = f2bf(h);
      }
      break;
    }
    case EPI_QKV: {
      const int hd = ph.hd;
      if (n < ph.q_rows + ph.kv_rows) {
        if ((ri & 1) == 0) {
          const bool isq = n < ph.q_rows;
          const int nn = isq ? n : n - ph.q_rows;
          const int d = nn % hd;
          const float2 cssn = P.rope[(size_t)pos * (hd / 2) + d / 2];
          const float a = rbf(y), bq = rbf(yp);
          const uint16_t o0 = f2bf(a * cssn.x - bq * cssn.y);
          const uint16_t o1 = f2bf(a * cssn.y + bq * cssn.x);
          uint16_t* dst = isq ? const_cast<uint16_t*>(ph.qbuf) + n
                              : ph.kc + (((size_t)(nn / hd)) * ph.Tmax + pos) * hd + d;
          dst[0] = o0;
          dst[1] = o1;
        }
      } else {
        const int nn = n - ph.q_rows - ph.kv_rows;
        const int d = nn % hd;
        ph.vc[(((size_t)(nn / hd)) * ph.Tmax + pos) * hd + d] = f2bf(y);
      }
      break;
    }
    case EPI_LOGITS:
      P.logits[n] = y;
      amax_merge(am, y, n);
      break;
    default:
      break;
  }
  return true;
}

// ----------------------------------------------------------- attention ---
template <int HD>
__device__ bool attn_unit(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int u, int nch, int CH, int pos) {
  constexpr int DPL = HD / 32;
  const int gq = ph.Hq / ph.Hkv;
  const int kvh = u / nch, c = u % nch;
  const int T = pos + 1, Ts = ph.stream_cur ? T : T - 1;
  const int p0 = c * CH, p1 = min(p0 + CH, T), pe = min(p1, Ts);
  const int lane = cs.lane, w = cs.warp;
  float* qs = S.xs;                       // [gq][HD], pre-scaled by 1/sqrt(HD)
  float* sc = S.xs + MAX_GQ * HD;         // [NCW][gq][HD + 2]
  const float scale = rsqrtf((float)HD);
  for (int i = cs.ctid; i < gq * HD; i += NCW * 32)
    qs[i] = bf2f(__ldcg(ph.qbuf + (size_t)kvh * gq * HD + i)) * scale;
  if (!cta_sync(S, cs, P.err)) return false;

  float m[MAX_GQ], l[MAX_GQ], o[MAX_GQ][DPL];
#pragma unroll
  for (int j = 0; j < MAX_GQ; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[j][d] = 0.f;
  }
  auto consume = [&](const uint16_t* krow, const uint16_t* vrow, bool global) {
    float kf[DPL], vf[DPL];
#pragma unroll
    for (int d = 0; d < DPL; d += 2) {
      const uint32_t kk = global ? __ldcg(reinterpret_cast<const unsigned*>(krow + lane * DPL + d))
                                 : *reinterpret_cast<const uint32_t*>(krow + lane * DPL + d);
      const uint32_t vv = global ? __ldcg(reinterpret_cast<const unsigned*>(vrow + lane * DPL + d))
                                 : *reinterpret_cast<const uint32_t*>(vrow + lane * DPL + d);
      kf[d] = __uint_as_float(kk << 16);
      kf[d + 1] = __uint_as_float(kk & 0xFFFF0000u);
      vf[d] = __uint_as_float(vv << 16);
      vf[d + 1] = __uint_as_float(vv & 0xFFFF0000u);
    }
#pragma unroll
    for (int j = 0; j < MAX_GQ; ++j) {
      if (j < gq) {
        float dot = 0.f;
#pragma unroll
        for (int d = 0; d < DPL; ++d) dot = fmaf(qs[j * HD + lane * DPL + d], kf[d], dot);
#pragma unroll
        for (int of = 16; of; of >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, of);
        const float mn = fmaxf(m[j], dot);
        const float corr = expf(m[j] - mn), p = expf(dot - mn);
        l[j] = fmaf(l[j], corr, p);
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[j][d] = fmaf(o[j][d], corr, p * vf[d]);
        m[j] = mn;
      }
    }
  };
  const uint32_t rowe = HD;  // elements per cache row
  for (int p = p0; p < pe; p += ATT_POS_PER_SLOT) {
    const int np = min(ATT_POS_PER_SLOT, pe - p);
    const uint8_t* base;
    if (!slot_acquire(S, cs, P.err, base)) return false;
    const uint16_t* kb = reinterpret_cast<const uint16_t*>(base);
    const uint16_t* vb = kb + ATT_POS_PER_SLOT * rowe;
    for (int q = w * 4; q < w * 4 + 4; ++q)
      if (q < np) consume(kb + q * rowe, vb + q * rowe, false);
    slot_release(S, cs);
  }
  if (w == 0) {
    for (int p = max(pe, p0); p < p1; ++p) {
      const size_t off = ((size_t)kvh * ph.Tmax + p) * HD;
      consume(ph.kc + off, ph.vc + off, true);
    }
  }
  // combine the warps of this CTA
#pragma unroll
  for (int j = 0; j < MAX_GQ; ++j) {
    if (j < gq) {
      float* dst = sc + (w * gq + j) * (HD + 2);
#pragma unroll
      for (int d = 0; d < DPL; ++d) dst[2 + lane * DPL + d] = o[j][d];
      if (lane == 0) {
        dst[0] = m[j];
        dst[1] = l[j];
      }
    }
  }
  if (!cta_sync(S, cs, P.err)) return false;
  const int stride = HD + 2;
  for (int i = cs.ctid; i < gq * HD; i += NCW * 32) {
    const int j = i / HD, d = i % HD;
    float M = -INFINITY;
    for (int ww = 0; ww < NCW; ++ww) M = fmaxf(M, sc[(ww * gq + j) * stride]);
    float L = 0.f, O = 0.f;
    for (int ww = 0; ww < NCW; ++ww) {
      const float* s = sc + (ww * gq + j) * stride;
      const float e = s[1] > 0.f ? expf(s[0] - M) : 0.f;
      L = fmaf(s[1], e, L);
      O = fmaf(s[2 + d], e, O);
    }
    const int h = kvh * gq + j;
    float* part = ph.part + ((size_t)h * nch + c) * stride;
    part[2 + d] = O;
    if (d == 0) {
      part[0] = M;
      part[1] = L;
    }
  }
  __threadfence();
  if (!cta_sync(S, cs, P.err)) return false;
  if (cs.ctid == 0) {
    const unsigned old = atomicAdd(ph.tick + kvh, 1u);
    S.bcast[0] = (old == (unsigned)(nch - 1));
  }
  if (!cta_sync(S, cs, P.err)) return false;
  if (S.bcast[0]) {
    __threadfence();
    for (int i = cs.ctid; i < gq * HD; i += NCW * 32) {
      const int j = i / HD, d = i % HD, h = kvh * gq + j;
      const float* pb = ph.part + (size_t)h * nch * stride;
      float M = -INFINITY;
      for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(pb + cc * stride));
      float L = 0.f, O = 0.f;
      for (int cc = 0; cc < nch; ++cc) {
        const float e = expf(__ldcg(pb + cc * stride) - M);
        L = fmaf(__ldcg(pb + cc * stride + 1), e, L);
        O = fmaf(__ldcg(pb + cc * stride + 2 + d), e, O);
      }
      ph.attn_out[(size_t)h * HD + d] = f2bf(O / L);
    }
    if (cs.ctid == 0) ph.tick[kvh] = 0u;
  }
  return true;
}

// ------------------------------------------------------ argmax finish ----
__device__ bool argmax_finish(const Params& P, const Smem& S, Cons& cs, int cta, ArgMax am) {
  // warp reduce, then CTA, then across CTAs through the last-arriving CTA
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float v = __shfl_xor_sync(0xffffffffu, am.v, o);
    const int i = __shfl_xor_sync(0xffffffffu, am.i, o);
    amax_merge(am, v, i);
  }
  if (cs.lane == 0) {
    S.red[cs.warp] = am.v;
    S.bcast[cs.warp] = am.i;  // bcast has room for 8 ints
  }
  if (!cta_sync(S, cs, P.err)) return false;
  if (cs.ctid == 0) {
    ArgMax b = {S.red[0], S.bcast[0]};
    for (int w = 1; w < NCW; ++w) amax_merge(b, S.red[w], S.bcast[w]);
    P.amax_val[cta] = b.v;
    P.amax_idx[cta] = b.i;
    __threadfence();
    const unsigned old = atomicAdd(P.amax_tick, 1u);
    if (old == (unsigned)(P.nctas - 1)) {
      __threadfence();
      ArgMax g = {-INFINITY, 0x7fffffff};
      for (int k = 0; k < P.nctas; ++k) amax_merge(g, __ldcg(P.amax_val + k), __ldcg(P.amax_idx + k));
      *P.argmax = g.i;
      *P.amax_tick = 0u;
      if (P.pos_inc) *P.pos_inc = *P.pos_inc + 1;
    }
  }
  return true;
}

// ============================================================== kernel ====
__global__ void __launch_bounds__(NTHREADS, 1) k_engine(const __grid_constant__ Params P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Smem S = smem_layout(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, cta = blockIdx.x;
  if (tid == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], NCW);
    }
    mbar_init(S.cbar, NCW * 32);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int pos = P.d_pos ? *P.d_pos : P.pos_const;
  // Reject a position or token that would index outside the cache, the RoPE
  // table or the embedding.  Every thread reads the same values, so the whole
  // CTA leaves together before any copy is issued.
  if (P.tmax > 0 && (pos < 0 || pos >= P.tmax)) {
    if (tid == 0) atomicCAS(P.err, 0, ERR_BAD_POS);
    return;
  }
  if (P.token && (*P.token < 0 || *P.token >= P.vocab)) {
    if (tid == 0) atomicCAS(P.err, 0, ERR_BAD_TOKEN);
    return;
  }

  if (warp == NCW) {
    if (lane == 0) producer(P, S, cta, pos);
    return;
  }

  Cons cs;
  cs.it = 0;
  cs.cphase = 0;
  cs.warp = warp;
  cs.lane = lane;
  cs.ctid = tid;
  cs.starved = 0;
  const int G = P.nctas;
  ArgMax am = {-INFINITY, 0x7fffffff};
  bool any_logits = false;

  for (int pi = 0; pi < P.nphases; ++pi) {
    const Phase& ph = phase_at(P, pi);
    unsigned long long* tr = (P.trace && tid == 0) ? P.trace + ((size_t)pi * G + cta) * TRACE_W : nullptr;
    if (tr) tr[0] = gtimer();
    if (ph.wait_bar >= 0) {
      int ok = 1;
      if (tid == 0) ok = grid_wait(P.bars + ph.wait_bar, (unsigned)G, P.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return;
      if (!cta_sync(S, cs, P.err)) return;
    }
    if (tr) tr[1] = gtimer();
    if (ph.kind == PH_GEMV) {
      if (!stage_x(ph, P, S, cs, cta)) return;
      if (tr) tr[2] = gtimer();
      const int ntiles = (ph.N + TR - 1) / TR;
      for (int t = first_unit(cta, ph.rot, G); t < ntiles; t += G) {
        bool ok;
        if (ph.dtype == DT_INT4) ok = gemv_unit<DT_INT4>(ph, P, S, cs, t, pos, am);
        else if (ph.dtype == DT_INT8) ok = gemv_unit<DT_INT8>(ph, P, S, cs, t, pos, am);
        else ok = gemv_unit<DT_BF16>(ph, P, S, cs, t, pos, am);
        if (!ok) return;
      }
      if (ph.epi == EPI_LOGITS) any_logits = true;
    } else if (ph.kind == PH_ATTN) {
      const int T = pos + 1;
      int CH, nch;
      attn_split(T, ph.Hkv, P.unit_target, CH, nch);
      const int nunits = ph.Hkv * nch;
      for (int u = first_unit(cta, ph.rot, G); u < nunits; u += G) {
        const bool ok = ph.hd == 128 ? attn_unit<128>(ph, P, S, cs, u, nch, CH, pos)
                                     : attn_unit<64>(ph, P, S, cs, u, nch, CH, pos);
        if (!ok) return;
      }
    }
    if (tr) {
      if (ph.kind != PH_GEMV) tr[2] = tr[1];
      tr[3] = gtimer();
      tr[6] = cs.starved;
    }
    cs.starved = 0;
    // every warp of this CTA has finished the phase (its global writes made)
    if (!cta_sync(S, cs, P.err)) return;
    if (ph.signal_bar >= 0 && tid == 0) grid_arrive(P.bars + ph.signal_bar);
    if (tr) tr[4] = gtimer();
  }
  if (any_logits) argmax_finish(P, S, cs, cta, am);
}

int launch_engine(const Params& p, int grid, bool cooperative, cudaStream_t s) {
  static bool attr_set[64] = {false};
  int dev = 0;
  GF_CUDA(cudaGetDevice(&dev));
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    GF_CUDA(cudaFuncSetAttribute(k_engine, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    attr_set[dev] = true;
  }
  if (cooperative) {
    void* args[] = {const_cast<Params*>(&p)};
    GF_CUDA(cudaLaunchCooperativeKernel((const void*)k_engine, dim3(grid), dim3(NTHREADS), args, SMEM_BYTES, s));
  } else {
    k_engine<<<grid, NTHREADS, SMEM_BYTES, s>>>(p);
    GF_CUDA(cudaGetLastError());
  }
  return GF_OK;
}

int* device_err_ptr() {
  static int* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
    cached[dev] = (int*)p;
  }
  return cached[dev];
}

// ------------------------------------------------- standalone launches ----
static Params base_params() {
  Params p;
  memset(&p, 0, sizeof p);
  p.nphases = 1;
  p.single.wait_bar = -1;
  p.single.signal_bar = -1;
  return p;
}

static int gemv_common(const char* fn, int dt, const void* x, const void* Wp, const void* s8, int N, int K, void* y,
                       int ydt, cudaStream_t stream) {
  if (!x || !Wp || !y || N <= 0 || K <= 0 || K % per_chunk(dt) || (dt == DT_INT8 && !s8) ||
      (ydt != GF_Y_BF16 && ydt != GF_Y_F32)) {
    set_error("%s: bad arguments (N=%d, K=%d, ydtype=%d)", fn, N, K, ydt);
    return GF_EINVAL;
  }
  if (K > KMAX) {
    set_error("%s: K=%d exceeds GF_KMAX=%d", fn, K, KMAX);
    return GF_EUNSUPPORTED;
  }
  if (!aligned16(x) || !aligned16(Wp) || !aligned16(y) || (s8 && !aligned16(s8))) {
    set_error("%s: pointers must be 16-byte aligned", fn);
    return GF_EALIGN;
  }
  Params p = base_params();
  Phase& ph = p.single;
  ph.kind = PH_GEMV;
  ph.dtype = dt;
  ph.N = N;
  ph.K = K;
  ph.W = (const uint8_t*)Wp;
  ph.s8 = (const uint16_t*)s8;
  ph.xsrc = X_BF16;
  ph.xptr = x;
  ph.epi = ydt == GF_Y_BF16 ? EPI_STORE_BF16 : EPI_STORE_F32;
  ph.out = y;
  const int ntiles = (N + TR - 1) / TR, sms = device_sms();
  const int grid = ntiles < sms ? ntiles : sms;
  p.nctas = grid;
  p.unit_target = sms;
  p.err = device_err_ptr();
  if (!p.err) {
    set_error("%s: cannot resolve the device error word", fn);
    return GF_ECUDA;
  }
  return launch_engine(p, grid, false, stream);
}

}  // namespace gf

using namespace gf;

extern "C" {

int gf_gemv_bf16(const void* x, const void* Wpacked, int N, int K, void* y, int ydtype, gf_stream stream) {
  return gemv_common("gf_gemv_bf16", DT_BF16, x, Wpacked, nullptr, N, K, y, ydtype, (cudaStream_t)stream);
}
int gf_gemv_w8(const void* x, const void* qpacked, const void* s, int N, int K, void* y, int ydtype, gf_stream stream) {
  return gemv_common("gf_gemv_w8", DT_INT8, x, qpacked, s, N, K, y, ydtype, (cudaStream_t)stream);
}
int gf_gemv_w4g(const void* x, const void* qpacked, int N, int K, int G, void* y, int ydtype, gf_stream stream) {
  if (G != 32) {
    set_error("gf_gemv_w4g: only group size 32 is supported (got %d)", G);
    return GF_EUNSUPPORTED;
  }
  return gemv_common("gf_gemv_w4g", DT_INT4, x, qpacked, nullptr, N, K, y, ydtype, (cudaStream_t)stream);
}

size_t gf_attn_workspace_bytes(int Hq, int Hkv, int hd) {
  if (Hq <= 0 || Hkv <= 0 || hd <= 0) return 0;
  const int sms = device_sms() > 0 ? device_sms() : 1;
  const int nch_max = (sms + Hkv - 1) / Hkv;
  return (size_t)Hq * nch_max * (hd + 2) * sizeof(float) + 256;
}

int gf_decode_attn(const void* q, const void* kcache, const void* vcache, int Hq, int Hkv, int hd, int Tmax, int pos,
                   void* out, void* ws, size_t ws_bytes, gf_stream stream) {
  if (!q || !kcache || !vcache || !out || !ws || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Hq / Hkv > MAX_GQ ||
      (hd != 64 && hd != 128) || pos < 0 || pos >= Tmax) {
    set_error("gf_decode_attn: bad arguments (Hq=%d Hkv=%d hd=%d Tmax=%d pos=%d)", Hq, Hkv, hd, Tmax, pos);
    return GF_EINVAL;
  }
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out) || !aligned16(ws)) {
    set_error("gf_decode_attn: pointers must be 16-byte aligned");
    return GF_EALIGN;
  }
  const size_t need = gf_attn_workspace_bytes(Hq, Hkv, hd);
  if (ws_bytes < need) {
    set_error("gf_decode_attn: workspace of %zu bytes is below the %zu needed", ws_bytes, need);
    return GF_EINVAL;
  }
  const int sms = device_sms();
  Params p = base_params();
  Phase& ph = p.single;
  ph.kind = PH_ATTN;
  ph.qbuf = (const uint16_t*)q;
  ph.kc = (uint16_t*)kcache;
  ph.vc = (uint16_t*)vcache;
  ph.attn_out = (uint16_t*)out;
  ph.Hq = Hq;
  ph.Hkv = Hkv;
  ph.hd = hd;
  ph.Tmax = Tmax;
  ph.stream_cur = 1;
  const size_t part_bytes = need - 256;
  ph.part = (float*)ws;
  ph.tick = (unsigned*)((uint8_t*)ws + part_bytes);
  GF_CUDA(cudaMemsetAsync(ph.tick, 0, Hkv * sizeof(unsigned), (cudaStream_t)stream));
  // same split rule as the kernel: units = Hkv * nch
  const int T = pos + 1;
  int want = (sms + Hkv - 1) / Hkv, maxch = (T + 31) / 32;
  int nch = want < maxch ? want : maxch;
  const int CH = ((T + nch - 1) / nch + 31) / 32 * 32;
  nch = (T + CH - 1) / CH;
  const int units = Hkv * nch;
  const int grid = units < sms ? units : sms;
  p.nctas = grid;
  p.unit_target = sms;
  p.pos_const = pos;
  p.err = device_err_ptr();
  if (!p.err) {
    set_error("gf_decode_attn: cannot resolve the device error word");
    return GF_ECUDA;
  }
  return launch_engine(p, grid, false, (cudaStream_t)stream);
}

}  // extern "C"
