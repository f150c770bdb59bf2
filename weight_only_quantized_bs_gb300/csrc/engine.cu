// engine.cu — the persistent phase engine of libgf (sm_103a).
//
// One CTA per SM (8 consumer warps, 4 producer warps) runs a program of
// phases: a single GEMV or attention for the standalone calls; every layer of
// a decode step, or of a k-draft verification, for gf_decode_step /
// gf_verify_k.  Lane 0 of each producer warp streams every fourth of the
// CTA's weight slots and KV-cache slots from HBM into a ring of 16
// shared-memory entries, running ahead across phase boundaries because the
// weight stream does not depend on activations.  A weight slot is 32 rows x
// 256 code bytes of each row (plus, for int4, the rows' scale/zero words),
// stored contiguously in the swizzled layout of gf_internal.cuh and moved by
// one bulk asynchronous copy (cp.async.bulk, the copy engine's linear mode)
// with an L2 evict-first hint; a KV slot is up to 16 positions of K and of V.
// Completion is counted on an mbarrier per entry.  Slot X of the stream
// belongs to consumer warp X mod 8 (two ring entries per warp).  The warp's
// lanes are 8 row lanes x 4 K quarters: each lane dequantises the int8 /
// int4 codes of four rows over a quarter of the slot's K range in registers
// against the fp32 input staged in shared memory, and the quarters meet in
// two shuffles.  A tile's partial sums from the warps that held its K-slots
// meet in shared memory, where the last warp to arrive adds them in K order
// and runs the epilogue.  Dependent phases are separated by grid barriers
// (cooperative launch) or by per-head completion counters (q/k/v rows ->
// attention -> o projection); every wait in the kernel is bounded by a clock
// (2 s by default), after which the kernel records an error code, drains its
// own copies in flight and returns.
//
// The decode step computed here is the batch-size-1 autoregressive step of
// the gpt-fast README ("Benchmarks", "Quantization"): RMSNorm, q/k/v, RoPE,
// KV append, single-query attention, o projection, residual, RMSNorm, SwiGLU,
// residual, final RMSNorm, lm_head, greedy argmax.
#include <math.h>
#include <string.h>

#include "gf_internal.cuh"

namespace gf {

__device__ int g_err_word;

// ------------------------------------------------------------- PTX glue --
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
// asynchronous 16-byte global -> shared copy (completion: cp_async_wait_all)
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sdst)), "l"(gsrc) : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

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
// non-blocking probe (never suspends), used only to count stalls for the trace
__device__ __forceinline__ bool mbar_probe(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
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
// one-dimensional bulk copy (KV rows, column-sliced down projection)
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

// try_wait that may suspend the thread for up to 20 us; the hardware wakes it
// as soon as the phase completes, so the hint adds no latency but keeps a
// waiting warp from spinning on issue slots the compute warps need.
__device__ __forceinline__ bool mbar_test_sleep(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

// The limit of every bounded wait of a launch (Params::wait_ns, else 2 s).
__device__ __forceinline__ uint64_t wait_limit(const Params& P) { return P.wait_ns ? P.wait_ns : 2000000000ull; }

__device__ __noinline__ bool mbar_wait_slow(uint64_t* b, uint32_t parity, int* err, int code, uint64_t lim) {
  const uint64_t t0 = gtimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_sleep(b, parity)) return true;
    if ((it & 3) == 0) {
      if (ld_relaxed(err)) return false;
      if (gtimer() - t0 > lim) {
        atomicCAS(err, 0, code);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, int* err, int code, uint64_t lim) {
  if (mbar_test(b, parity)) return true;
  return mbar_wait_slow(b, parity, err, code, lim);
}

// Waits until *ctr >= target (acquire); bounded.
__device__ __noinline__ bool counter_wait(const unsigned* ctr, unsigned target, int* err, int code, uint64_t lim) {
  const uint64_t t0 = gtimer();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire(ctr) >= target) return true;
    __nanosleep(40);
    if ((it & 15) == 15) {
      if (ld_relaxed(err)) return false;
      if (gtimer() - t0 > lim) {
        atomicCAS(err, 0, code);
        return false;
      }
    }
  }
}
__device__ __forceinline__ void grid_arrive(unsigned* bar) {
  __threadfence();
  atomicAdd(bar, 1u);
}

// Bounded wait of one lane on a shared-memory word reaching `want` (==) or
// at least `want` (ge); false if it gave up.
__device__ __noinline__ bool smem_wait(const int* w, int want, bool ge, int* err, uint64_t lim) {
  volatile const int* p = w;
  const uint64_t t0 = gtimer();
  while (ge ? (*p < want) : (*p != want)) {
    __nanosleep(32);
    if (gtimer() - t0 > lim) {
      atomicCAS(err, 0, ERR_WAIT_COMBINE);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// ---------------------------------------------------------- shared state --
struct Smem {
  uint8_t* ring;
  float* xs;        // fp32 input vector (times the dequantisation powers)
  float* xsum;      // sums of x over each int4 group / int8 chunk (times 2^-64)
  float* tb;        // [NTB][NCW][TR] partial row sums of tiles
  int* tbc;         // [NTB] arrival counters
  int* tbg;         // [NTB] tile allowed to use the buffer next
  uint64_t* full;   // [NSLOT]
  uint64_t* empty;  // [NSLOT]
  uint64_t* cbar;   // consumer-warps barrier
  float* red;       // [64] reduction scratch; [32..39] router logits, [40..41] expert weights
  int* bcast;       // [64] broadcast ints; [32..33] chosen experts, [34] phase they were chosen in,
                    // [48..55] verify: union of the rows' experts, [56] its size
  float* moew;      // [MAX_M][8] verify: weight of expert e for row m (0 if not chosen)
  int* ffnc;        // [2][FFN_HN] PH_FFN: SwiGLU buffer rounds written, down pieces finished (zero between phases)
  Phase* phb;       // [2] the consumers' copies of the current and next phase descriptor
};

__device__ __forceinline__ Smem smem_layout(uint8_t* raw) {
  // slots start on 128-byte boundaries, so that a line's units map to banks
  // as the swizzle assumes
  const uint32_t a = smem_u32(raw);
  uint8_t* base = raw + ((128u - (a & 127u)) & 127u);
  Smem s;
  s.ring = base + OFF_RING;
  s.xs = reinterpret_cast<float*>(base + OFF_X);
  s.xsum = reinterpret_cast<float*>(base + OFF_XSUM);
  s.tb = reinterpret_cast<float*>(base + OFF_TB);
  s.tbc = reinterpret_cast<int*>(base + OFF_TBC);
  s.tbg = s.tbc + NTB;
  s.full = reinterpret_cast<uint64_t*>(base + OFF_BAR);
  s.empty = s.full + NSLOT;
  s.cbar = s.empty + NSLOT;
  s.red = reinterpret_cast<float*>(base + OFF_MISC);
  s.bcast = reinterpret_cast<int*>(base + OFF_MISC + 512);
  s.moew = reinterpret_cast<float*>(base + OFF_MISC + 1280);
  s.ffnc = reinterpret_cast<int*>(base + OFF_MISC + 1536);
  static_assert(NCW * MAX_M <= 128 && 64 + NCW * MAX_M <= 192 && 1536 + 2 * FFN_HN * 4 <= MISC_BYTES,
                "misc shared-memory areas");
  s.phb = reinterpret_cast<Phase*>(base + OFF_PHB);
  return s;
}

__device__ __forceinline__ int first_unit(int cta, int rot, int G) { return ((cta - rot) % G + G) % G; }
__device__ __forceinline__ int units_of(int first, int n, int G) { return first < n ? (n - first + G - 1) / G : 0; }

__device__ __forceinline__ const Phase& phase_at(const Params& P, int i) { return P.prog ? P.prog[i] : P.single; }

// ------------------------------------------------ attention units -------
// Units of an attention phase: for each query row m (one in a decode step,
// M in a verify pass) the kv heads times the chunks of that row's positions
// 0..pos+m.  Positions below `Ts` come through the ring; the rest (rows
// written during this launch) are read from global memory.
struct AttnUnit {
  int m, kvh, c, nch, T, Ts, p0, p1;
};
__device__ int attn_units(const Phase& ph, const Params& P, int pos, int u, AttnUnit* out) {
  const bool ver = verifying(P);
  const int M = ver ? P.M : 1;
  int base = 0;
  for (int m = 0; m < M; ++m) {
    const int T = pos + m + 1;
    int CH, nch;
    attn_split(T, ph.Hkv, P.unit_target, CH, nch);
    const int n = ph.Hkv * nch;
    if (u >= base && u < base + n && out) {
      const int v = u - base;
      out->m = m;
      out->kvh = v / nch;
      out->c = v % nch;
      out->nch = nch;
      out->T = T;
      out->Ts = ver ? pos : (ph.stream_cur ? T : T - 1);
      out->p0 = out->c * CH;
      out->p1 = min(out->p0 + CH, T);
      return 0;
    }
    base += n;
  }
  return base;
}

// Segments of a GEMV phase: the matrices it covers (several experts for MoE),
// as expert indices into the tall matrix of all experts.
__device__ __forceinline__ int gemv_segments(const Phase& ph, const Params& P, const Smem& S, int& Ns, int* eseg) {
  volatile int* bc = S.bcast;
  if (ph.moe == MOE_NONE) {
    Ns = ph.N;
    eseg[0] = 0;
    return 1;
  }
  if (verifying(P)) {  // verify: the union of the rows' experts
    const int n = bc[56];
    Ns = ph.N;
    for (int k = 0; k < n; ++k) eseg[k] = bc[48 + k];
    return n;
  }
  if (ph.moe == MOE_GU) {
    Ns = ph.N / 2;
    eseg[0] = bc[32];
    eseg[1] = bc[33];
    return 2;
  }
  Ns = ph.N;
  eseg[0] = bc[32 + ph.moe - MOE_DOWN0];
  return 1;
}

// Slot order of a multi-row (verify) GEMV phase: the CTA's tiles in groups of
// up to VTG tiles of one segment; per group, K-slot by K-slot, the group's
// tiles.  Consumers walk the same order.
struct TileGroups {
  int first, G, ntiles, tps;
};
__device__ __forceinline__ int group_end(const TileGroups& tg, int i0) {
  const int t0 = tg.first + i0 * tg.G, seg = t0 / tg.tps;
  int i1 = i0 + 1;
  while (i1 - i0 < VTG) {
    const int t = tg.first + i1 * tg.G;
    if (t >= tg.ntiles || t / tg.tps != seg) break;
    ++i1;
  }
  return i1;
}

// ============================================================ producer ====
// NPROD producer threads (lane 0 of the last NPROD warps) walk the same slot
// stream; producer p issues the slots X with X % NPROD == p, which use the
// ring entries of that residue only.  One thread can issue a bulk copy only
// every few hundred nanoseconds, which alone would cap the stream below the
// HBM rate; four issue in parallel (measured: the bf16 step, which waits on
// its copies, runs about 5 % faster with four than with two).
struct Prod {
  uint32_t it;
  uint64_t pol;
  uint32_t blocked;
  uint64_t lim;
  uint32_t pid;
};

// Advances the stream by one slot.  1: this producer's slot (dst and fb set,
// its copies to be issued); 0: another producer's slot; -1: a wait gave up.
__device__ __forceinline__ int prod_slot(const Smem& S, Prod& pr, int* err, uint8_t*& dst, uint64_t*& fb) {
  const uint32_t x = pr.it++;
  if (x % NPROD != pr.pid) return 0;
  const uint32_t slot = x % NSLOT, use = x / NSLOT;
  if (use > 0) {
    if (!mbar_probe(&S.empty[slot], (use - 1) & 1u)) ++pr.blocked;
    if (!mbar_wait(&S.empty[slot], (use - 1) & 1u, err, ERR_WAIT_EMPTY, pr.lim)) return -1;
  }
  dst = S.ring + slot * SLOT_BYTES;
  fb = &S.full[slot];
  return 1;
}

// One GEMV slot: tile lt of segment (expert) e (tiles per expert tps), K-slot b.
__device__ __forceinline__ bool produce_gemv_slot(const Phase& ph, const Params& P, const Smem& S, Prod& pr, int e,
                                                  int tps, int lt, int b) {
  const int dt = ph.dtype, nb = k_slots(dt, ph.K), sb = slot_bytes(dt, ph.G);
  uint8_t* dst;
  uint64_t* fb;
  const int r = prod_slot(S, pr, P.err, dst, fb);
  if (r <= 0) return r == 0;
  mbar_expect_tx(fb, (uint32_t)sb);
  bulk_g2s(dst, ph.W + (((size_t)e * tps + lt) * nb + b) * sb, (uint32_t)sb, fb, pr.pol);
  return true;
}

// The producer needs the two experts of a MOE_GU phase before it can stream
// their weights: consumer thread 0 publishes them in shared memory, tagged
// with the phase index.  Bounded wait.
__device__ bool wait_experts(const Smem& S, int* err, int pi, uint64_t lim) {
  volatile int* seq = S.bcast + 34;
  const uint64_t t0 = gtimer();
  for (uint32_t it = 0;; ++it) {
    if (*seq == pi + 1) {
      __threadfence_block();
      return true;
    }
    __nanosleep(64);
    if ((it & 31) == 31) {
      if (ld_relaxed(err)) return false;
      if (gtimer() - t0 > lim) {
        atomicCAS(err, 0, ERR_WAIT_ROUTER);
        return false;
      }
    }
  }
}

__device__ bool produce_gemv_m(const Phase& ph, const Params& P, const Smem& S, Prod& pr, int cta, int pi) {
  if (ph.moe == MOE_GU && !wait_experts(S, P.err, pi, pr.lim)) return false;
  const int nb = k_slots(ph.dtype, ph.K);
  int Ns;
  int eseg[8];
  const int nseg = gemv_segments(ph, P, S, Ns, eseg);
  TileGroups tg;
  tg.tps = (Ns + TR - 1) / TR;
  tg.ntiles = nseg * tg.tps;
  tg.G = P.nctas;
  tg.first = first_unit(cta, ph.rot, P.nctas);
  for (int i0 = 0; tg.first + i0 * tg.G < tg.ntiles;) {
    const int i1 = group_end(tg, i0);
    for (int b = 0; b < nb; ++b) {
      for (int i = i0; i < i1; ++i) {
        const int t = tg.first + i * tg.G;
        if (!produce_gemv_slot(ph, P, S, pr, eseg[t / tg.tps], tg.tps, t % tg.tps, b)) return false;
      }
    }
    i0 = i1;
  }
  return true;
}

// Slot order of a GEMV phase (producer and consumers walk it identically):
// for each of the CTA's tiles t, the K-slots b in order.  PH_FFN: per tile its
// gate/up K-slots, then the down pieces of the previous tile (NCW * P slots;
// the piece at stream position X carries rows of warp X % NCW).
__device__ void producer(const Params& P, const Smem& S, int cta, int pos, int pid) {
  Prod pr;
  pr.it = 0;
  pr.blocked = 0;
  pr.pid = (uint32_t)pid;
  pr.pol = evict_first_policy();
  pr.lim = wait_limit(P);
  int* err = P.err;
  const int G = P.nctas;
  bool ok = true;
  for (int pi = 0; pi < P.nphases && ok; ++pi) {
    const Phase& ph = phase_at(P, pi);
    if (ph.kind == PH_GEMV && verifying(P)) {
      ok = produce_gemv_m(ph, P, S, pr, cta, pi);
    } else if (ph.kind == PH_GEMV) {
      if (ph.moe == MOE_GU && !(ok = wait_experts(S, err, pi, pr.lim))) break;
      const int nb = k_slots(ph.dtype, ph.K);
      int Ns;
      int eseg[8];
      gemv_segments(ph, P, S, Ns, eseg);
      const int nseg = ph.moe == MOE_GU ? 2 : 1;
      const int tps = (Ns + TR - 1) / TR, ntiles = nseg * tps;
      for (int t = first_unit(cta, ph.rot, G); t < ntiles && ok; t += G)
        for (int b = 0; b < nb && ok; ++b) ok = produce_gemv_slot(ph, P, S, pr, eseg[t / tps], tps, t % tps, b);
    } else if (ph.kind == PH_OSPLIT) {
      const int nb = k_slots(ph.dtype, ph.K), tps = (ph.N + TR - 1) / TR;
      for (int u = first_unit(cta, ph.rot, G); u < tps * nb && ok; u += G)
        ok = produce_gemv_slot(ph, P, S, pr, 0, tps, u / nb, u % nb);
    } else if (ph.kind == PH_FFN) {
      const int dt = ph.dtype, nb = k_slots(dt, ph.K);
      const int tps = ph.N / TR, d = ph.N2;
      const FfnSplit fs = ffn_split(dt, d);
      const int ND = NCW * fs.P;
      // the down slice of local tile t: ND pieces
      auto down_slice = [&](int t) {
        for (int m = 0; m < ND && ok; ++m) {
          const int w = (int)(pr.it % NCW), k = m / NCW;
          int r0, r1;
          ffn_piece(fs, d, w, k, r0, r1);
          uint8_t* dst;
          uint64_t* fb;
          const int rs = prod_slot(S, pr, err, dst, fb);
          if (rs < 0) {
            ok = false;
            break;
          }
          if (rs == 0) continue;
          if (r0 >= r1) {  // an empty slot: completed by the arrival alone
            mbar_arrive(fb);
            continue;
          }
          const uint32_t nr = (uint32_t)(r1 - r0);
          if (dt == DT_INT4) {
            const uint8_t* g = ph.W2 + (size_t)(t >> 1) * d * 20;
            mbar_expect_tx(fb, nr * 12u);
            bulk_g2s(dst, g + (size_t)(t & 1) * d * 8 + (size_t)r0 * 8, nr * 8u, fb, pr.pol);
            bulk_g2s(dst + (size_t)fs.PR * 8, g + (size_t)d * 16 + (size_t)r0 * 4, nr * 4u, fb, pr.pol);
          } else if (dt == DT_INT8) {
            mbar_expect_tx(fb, nr * 16u);
            bulk_g2s(dst, ph.W2 + ((size_t)t * d + r0) * 16, nr * 16u, fb, pr.pol);
          } else {
            const uint8_t* g = ph.W2 + (size_t)t * d * 32;
            mbar_expect_tx(fb, nr * 32u);
            bulk_g2s(dst, g + (size_t)r0 * 16, nr * 16u, fb, pr.pol);
            bulk_g2s(dst + (size_t)fs.PR * 16, g + (size_t)d * 16 + (size_t)r0 * 16, nr * 16u, fb, pr.pol);
          }
        }
      };
      int prev = -1;
      for (int t = first_unit(cta, ph.rot, G); t < tps && ok; t += G) {
        for (int b = 0; b < nb && ok; ++b) ok = produce_gemv_slot(ph, P, S, pr, 0, tps, t, b);
        if (prev >= 0 && ok) down_slice(prev);
        prev = t;
      }
      if (prev >= 0 && ok) down_slice(prev);
    } else if (ph.kind == PH_ATTN) {
      const uint32_t rowb = (uint32_t)ph.hd * 2;
      const int nunits = attn_units(ph, P, pos, -1, nullptr);
      for (int u = first_unit(cta, ph.rot, G); u < nunits && ok; u += G) {
        AttnUnit au;
        attn_units(ph, P, pos, u, &au);
        const int hh = au.kvh;
        const int p0 = au.p0, p1 = au.p1, pe = min(p1, au.Ts);
        const int aps = att_slot_pos(ph.hd);
        for (int p = p0; p < pe; p += aps) {
          const int np = min(aps, pe - p);
          uint8_t* dst;
          uint64_t* fb;
          const int rs = prod_slot(S, pr, err, dst, fb);
          if (rs < 0) {
            ok = false;
            break;
          }
          if (rs == 0) continue;
          const size_t off = ((size_t)hh * ph.Tmax + p) * ph.hd;
          mbar_expect_tx(fb, 2u * np * rowb);
          bulk_g2s(dst, ph.kc + off, np * rowb, fb, pr.pol);
          bulk_g2s(dst + aps * rowb, ph.vc + off, np * rowb, fb, pr.pol);
        }
      }
    }
    if (P.trace && pid == 0) {
      unsigned long long* tr = P.trace + ((size_t)pi * G + cta) * TRACE_W;
      tr[5] = gtimer();
      tr[7] = pr.blocked;
      pr.blocked = 0;
    }
  }
  // Drain: never leave the CTA with copies still writing its shared memory.
  // Of this producer's slots, only those among the last min(it, NSLOT) can be
  // in flight; wait for each one's completion (bounded).
  const uint32_t n = pr.it < (uint32_t)NSLOT ? pr.it : (uint32_t)NSLOT;
  for (uint32_t k = 0; k < n; ++k) {
    const uint32_t i = pr.it - 1 - k, slot = i % NSLOT, use = i / NSLOT;
    if (i % NPROD != pr.pid) continue;
    const uint64_t t0 = gtimer();
    while (!mbar_test_sleep(&S.full[slot], use & 1u)) {
      if (gtimer() - t0 > pr.lim) {
        atomicCAS(err, 0, ERR_DRAIN);
        break;
      }
    }
  }
}

// ============================================================ consumers ===
struct Cons {
  uint32_t it;       // ring position of the phase's first slot
  uint32_t cphase;   // parity of the consumer barrier
  uint32_t useq;     // tiles seen so far (combine-buffer index)
  int warp, lane, ctid;
  uint32_t starved;  // slot waits that found the slot still in flight (warp 0)
  float rnorm;       // RMSNorm factor of the staged input (1 if none)
  bool wnorm;        // staged per warp: the RMSNorm factor is formed at the combine from S.red
  uint64_t lim;      // limit of the bounded waits
};

// all consumer warps meet; false if the wait gave up
__device__ __forceinline__ bool cta_sync(const Smem& S, Cons& cs, int* err) {
  __syncwarp();
  mbar_arrive(S.cbar);
  int ok = 1;
  if (cs.lane == 0) ok = mbar_wait(S.cbar, cs.cphase, err, ERR_WAIT_CTA, cs.lim);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok && cs.lane) mbar_test(S.cbar, cs.cphase);  // acquire for this lane (phase already complete)
  cs.cphase ^= 1u;
  return ok != 0;
}

// Every lane waits on the slot's barrier itself (each lane's completed wait
// orders its reads of the slot after the copy).
__device__ __forceinline__ bool slot_acquire(const Smem& S, Cons& cs, uint32_t it, int* err, const uint8_t*& base) {
  const uint32_t slot = it % NSLOT, par = (it / NSLOT) & 1u;
  if (cs.warp == 0 && cs.lane == 0 && !mbar_probe(&S.full[slot], par)) ++cs.starved;
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&S.full[slot], par, err, ERR_WAIT_FULL, cs.lim));
  base = S.ring + slot * SLOT_BYTES;
  return ok;
}
__device__ __forceinline__ void slot_release(const Smem& S, const Cons& cs, uint32_t it) {
  __syncwarp();
  if (cs.lane == 0) mbar_arrive(&S.empty[it % NSLOT]);
}

// Dequantisation through subnormals.  A code c held in bits p..p+3 (int4)
// or p..p+7 (int8, offset to c + 128) of a 32-bit word whose other bits are
// clear reads, as an IEEE binary32, exactly c * 2^(p - 149): a subnormal, or
// with bit 23 set a number of the smallest normal binade, whose spacing is
// the same, so the value stays linear in c.  That holds for every p up to 20
// (int4) or 16 (int8); the codes of a word's top byte are taken from the word
// shifted right by 8.  The staged input carries the inverse power (each x is
// multiplied by 2^(85 - p) for the position p its code is read from), so a
// fused multiply-add adds c * x * 2^-64 with one rounding, as with ordinary
// fp32 operands: one AND per code, one packed FMA per two codes, no bias to
// remove.  Products and partial sums are normal numbers for any input above
// about 2^-60 in magnitude; the 2^-64 is undone in the epilogue (exact).
// FMAs must keep subnormal operands (no flush-to-zero), which is the default.
constexpr float DQ_UP = 18446744073709551616.0f;  // 2^64
constexpr float DQ_DOWN = 1.0f / DQ_UP;           // 2^-64

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }  // normal range
// multipliers of the staged inputs, per component of float4 number u of a chunk
__device__ __forceinline__ float4 dq_mult(int dt, int u) {
  if (dt == DT_INT4)
    return (u & 1) ? make_float4(pow2f(69), pow2f(65), pow2f(69), pow2f(65))
                   : make_float4(pow2f(85), pow2f(81), pow2f(77), pow2f(73));
  if (dt == DT_INT8) return make_float4(pow2f(85), pow2f(77), pow2f(69), pow2f(69));
  return make_float4(1.0f, 1.0f, 1.0f, 1.0f);
}
__device__ __forceinline__ float4 dq_inv(int dt, int u) {
  if (dt == DT_INT4)
    return (u & 1) ? make_float4(pow2f(-69), pow2f(-65), pow2f(-69), pow2f(-65))
                   : make_float4(pow2f(-85), pow2f(-81), pow2f(-77), pow2f(-73));
  if (dt == DT_INT8) return make_float4(pow2f(-85), pow2f(-77), pow2f(-69), pow2f(-69));
  return make_float4(1.0f, 1.0f, 1.0f, 1.0f);
}
// ------------------------------------------------------ input staging ----
__device__ __forceinline__ float4 bf4(uint2 h) {
  return make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xFFFF0000u), __uint_as_float(h.y << 16),
                     __uint_as_float(h.y & 0xFFFF0000u));
}

// Stores float4 number k4 of x multiplied by the powers of two that the
// subnormal dequantisation of int4 / int8 codes expects, and the sums the
// epilogues need: for int4 the sum of x over each group of G (G / 4
// consecutive lanes hold one group; k4 runs over whole warps of consecutive
// float4), for int8 128 times the sum over each 16-wide chunk (4 lanes),
// both times 2^-64.
__device__ __forceinline__ void stage_store(const Smem& S, const Cons& cs, int dt, int G, int k4, bool ok, float4 a) {
  const float4 m = dq_mult(dt, k4 & 7);
  if (ok) reinterpret_cast<float4*>(S.xs)[k4] = make_float4(a.x * m.x, a.y * m.y, a.z * m.z, a.w * m.w);
  if (dt != DT_BF16) {
    float sg = a.x + a.y + a.z + a.w;
    const int span = dt == DT_INT4 ? G / 4 : 4;  // lanes per group / chunk
    for (int o = 1; o < span; o <<= 1) sg += __shfl_xor_sync(0xffffffffu, sg, o);
    if (ok && (cs.lane & (span - 1)) == 0) S.xsum[(4 * k4) / (dt == DT_INT4 ? G : 16)] =
        sg * (dt == DT_INT4 ? DQ_DOWN : 128.0f * DQ_DOWN);
  }
}

// Per-warp staging.  When the K-slots of a phase's tiles are a multiple of
// the warp count, slot (tile, b) always belongs to warp (phase start + b) mod
// NCW, so each warp stages only the input slices of its own K-slots (zero past
// K): no CTA-wide barrier before the GEMV starts.  For an RMSNorm input each
// warp leaves the sum of squares of its slices in S.red[warp]; the combining
// warp of a tile forms 1/rms from all of them (every warp contributes to
// every tile, so all are written by then).  Used for every non-MoE GEMV and
// fused-FFN phase of the decode step whose K-slots divide evenly.
__device__ __forceinline__ bool warp_stageable(const Phase& ph) {
  return ph.moe == MOE_NONE && k_slots(ph.dtype, ph.K) % NCW == 0 && ph.xsrc != X_NONE;
}
__device__ void stage_x_warp(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta) {
  const int K = ph.K, dt = ph.dtype, G = ph.G, K4 = K / 4, SK4 = slot_k(dt) / 4, nb = k_slots(dt, K);
  const bool norm = ph.xsrc == X_NORM || ph.xsrc == X_EMBED_NORM;
  const bool f32 = ph.xsrc == X_F32 || ph.xsrc == X_NORM;
  const uint16_t* emb = ph.xsrc == X_EMBED_NORM ? P.embed + (size_t)(*P.token) * K : nullptr;
  const uint2* src16 = emb ? reinterpret_cast<const uint2*>(emb) : reinterpret_cast<const uint2*>(ph.xptr);
  const float4* src32 = reinterpret_cast<const float4*>(ph.xptr);
  const uint2* gain = reinterpret_cast<const uint2*>(ph.gain);
  // this lane's float4: runs of 32 in the warp's K-slots b0, b0 + NCW, ...
  const int b0 = (cs.warp - (int)(cs.it % NCW) + NCW) % NCW, per = SK4 / 32;
  const int n = (nb - b0 + NCW - 1) / NCW * per;
  float ss = 0.f;
  constexpr int BATCH = 4;  // loads in flight per lane before the first is used
  for (int j0 = 0; j0 < n; j0 += BATCH) {  // warp-uniform trip count
    float4 a[BATCH];
    uint2 g[BATCH];
    int fs[BATCH];
#pragma unroll
    for (int q = 0; q < BATCH; ++q) {
      const int j = j0 + q;
      fs[q] = ((b0 + (j / per) * NCW) * SK4) + (j % per) * 32 + cs.lane;
      const bool in = j < n && fs[q] < K4;
      a[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      g[q] = make_uint2(0u, 0u);
      if (in) {
        if (f32) {
          a[q] = __ldcg(src32 + fs[q]);
        } else {
          const uint2 h = __ldcg(src16 + fs[q]);
          a[q].x = __uint_as_float(h.x);
          a[q].y = __uint_as_float(h.y);
        }
        if (norm) g[q] = gain[fs[q]];
      }
    }
#pragma unroll
    for (int q = 0; q < BATCH; ++q) {
      if (j0 + q >= n) break;  // uniform
      const int f = fs[q];
      const bool in = f < K4;
      float4 v = f32 ? a[q] : bf4(make_uint2(__float_as_uint(a[q].x), __float_as_uint(a[q].y)));
      if (!in) v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (norm) {
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        if (emb && cta == 0 && in) reinterpret_cast<float4*>(P.resid)[f] = v;
        const float4 gg = bf4(g[q]);
        v = make_float4(v.x * gg.x, v.y * gg.y, v.z * gg.z, v.w * gg.w);
      }
      stage_store(S, cs, dt, G, f, true, v);
    }
  }
  cs.rnorm = 1.0f;
  cs.wnorm = norm;
  if (norm) {
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (cs.lane == 0) S.red[cs.warp] = ss;
  }
  __syncwarp();
}
// 1 / rms of a warp-staged RMSNorm input (after every warp staged its part)
__device__ __forceinline__ float warp_rnorm(const Phase& ph, const Smem& S) {
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < NCW; ++w) tot += S.red[w];
  return 1.0f / sqrtf(tot / (float)ph.K + ph.eps);
}

// Stages the phase's input vector into shared memory as fp32, zero from K up
// to the end of the last K-slot (the slots' padding codes are zero, and the
// products with them must be exactly zero).  For an
// RMSNorm input only the gain is applied here: the factor 1/rms needs the
// whole vector, and as the GEMV is linear it is applied to the outputs in
// the epilogue instead (cs.rnorm, 1 for other inputs), which keeps the
// reduction off the path.  fp32 inputs (X_F32, X_NORM) are fetched with
// per-thread asynchronous copies into the x area (the gain into the top of
// that area), then converted in place: gain, 1/rms partial sums, the
// dequantisation powers and the group sums.  Warp w copies and converts the
// runs of 32 float4 starting at 32 w + 256 i: its lanes' copies are complete
// and visible to the warp after wait_all and __syncwarp.  The copies use the
// load/store path, not the bulk-copy engine, whose queue holds the
// producer's weight prefetches.  bf16 inputs (standalone GEMVs, the embedding
// row) are loaded into registers first.
__device__ bool stage_x(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta) {
  const int K = ph.K, dt = ph.dtype, G = ph.G, K4 = K / 4;
  const int KP4 = (int)round_up(K, slot_k(dt)) / 4;  // staged float4, with the zero tail
  const bool norm = ph.xsrc == X_NORM || ph.xsrc == X_EMBED_NORM;
  float4* xs4 = reinterpret_cast<float4*>(S.xs);
  float ss = 0.0f;
  if ((ph.xsrc == X_F32 || ph.xsrc == X_NORM) && ((uintptr_t)ph.xptr & 15) == 0 &&
      (!norm || (KP4 * 16 + K * 2 <= KMAX * 4 && ((uintptr_t)ph.gain & 7) == 0))) {
    uint2* gs = reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(S.xs) + KMAX * 4 - K * 2);
    const float4* src = reinterpret_cast<const float4*>(ph.xptr);
    const uint2* gsrc = reinterpret_cast<const uint2*>(ph.gain);
#pragma unroll 1
    for (int f = cs.warp * 32 + cs.lane; f < K4; f += NCW * 32) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(xs4 + f)), "l"(src + f) : "memory");
      if (norm) asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(gs + f)), "l"(gsrc + f) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    cp_async_wait_all();
    __syncwarp();
#pragma unroll 1
    for (int base = cs.warp * 32; base < KP4; base += NCW * 32) {  // warp-uniform trip count
      const int f = base + cs.lane;
      const bool in = f < K4;
      float4 a = in ? xs4[f] : make_float4(0.f, 0.f, 0.f, 0.f);
      if (norm) {
        ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
        const float4 g = bf4(in ? gs[f] : make_uint2(0u, 0u));
        a = make_float4(a.x * g.x, a.y * g.y, a.z * g.z, a.w * g.w);
      }
      __syncwarp();  // every lane has read the run before any lane overwrites it
      stage_store(S, cs, dt, G, f, f < KP4, a);
    }
  } else {
    // bf16 vector or embedding row (optionally normalised), or an unaligned
    // fp32 vector: loads into registers, one run of 32 float4 per warp at a time
    const uint16_t* emb = ph.xsrc == X_EMBED_NORM ? P.embed + (size_t)(*P.token) * K : nullptr;
#pragma unroll 1
    for (int base = cs.warp * 32; base < KP4; base += NCW * 32) {
      const int f = base + cs.lane;
      const bool in = f < K4;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (in) {
        if (ph.xsrc == X_F32 || ph.xsrc == X_NORM) {
          const float* x = reinterpret_cast<const float*>(ph.xptr) + 4 * f;
          a = make_float4(__ldcg(x), __ldcg(x + 1), __ldcg(x + 2), __ldcg(x + 3));
        } else {
          const uint2* src = emb ? reinterpret_cast<const uint2*>(emb) : reinterpret_cast<const uint2*>(ph.xptr);
          a = bf4(__ldcg(src + f));
        }
      }
      if (norm) {
        ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
        if (emb && cta == 0 && in) reinterpret_cast<float4*>(P.resid)[f] = a;
        const float4 g = bf4(in ? reinterpret_cast<const uint2*>(ph.gain)[f] : make_uint2(0u, 0u));
        a = make_float4(a.x * g.x, a.y * g.y, a.z * g.z, a.w * g.w);
      }
      stage_store(S, cs, dt, G, f, f < KP4, a);
    }
  }
  if (norm) {
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (cs.lane == 0) S.red[cs.warp] = ss;
  }
  if (!cta_sync(S, cs, P.err)) return false;
  cs.rnorm = 1.0f;
  cs.wnorm = false;
  if (norm) {
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) tot += S.red[w];
    cs.rnorm = 1.0f / sqrtf(tot / (float)K + ph.eps);
  }
  return true;
}

// ------------------------------------------------------ GEMV compute -----
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ float2 bits2(uint32_t a, uint32_t b) { return make_float2(__uint_as_float(a), __uint_as_float(b)); }
__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }

// One 32-bit word of codes of one row against its staged inputs (natural k
// order, as pairs), accumulated into acc.
// int4: the word holds 8 consecutive codes in nibbles 0..7.
__device__ __forceinline__ float2 word_int4(const uint32_t w, float4 xa, float4 xb, float2 acc) {
  const uint32_t h = w >> 8;
  acc = ffma2(bits2(w & 0x0000000Fu, w & 0x000000F0u), lo2(xa), acc);
  acc = ffma2(bits2(w & 0x00000F00u, w & 0x0000F000u), hi2(xa), acc);
  acc = ffma2(bits2(w & 0x000F0000u, w & 0x00F00000u), lo2(xb), acc);
  acc = ffma2(bits2(h & 0x000F0000u, h & 0x00F00000u), hi2(xb), acc);
  return acc;
}
// int8: 4 consecutive codes, one byte each, stored as the offset code c + 128.
__device__ __forceinline__ float2 word_int8(const uint32_t w, float4 x, float2 acc) {
  const uint32_t h = w >> 8;
  acc = ffma2(bits2(w & 0x000000FFu, w & 0x0000FF00u), lo2(x), acc);
  acc = ffma2(bits2(w & 0x00FF0000u, h & 0x00FF0000u), hi2(x), acc);
  return acc;
}
// bf16: 2 consecutive weights (low half first).
__device__ __forceinline__ float2 word_bf16(const uint32_t w, float2 x, float2 acc) {
  return ffma2(bits2(w << 16, w & 0xFFFF0000u), x, acc);
}

// Lane `lane`'s 16-byte chunk u of a GEMV slot (row lane: line
// (u >> 3) * 32 + lane, swizzled).
__device__ __forceinline__ uint4 slot_chunk(const uint8_t* base, int lane, int u) {
  return *reinterpret_cast<const uint4*>(base + (u >> 3) * (TR * LINE) + lane * LINE + (((u & 7) ^ (lane & 7)) << 4));
}
// The int4 scale/zero word of group g of the slot for row `lane` (line 64 + g,
// swizzled).
__device__ __forceinline__ uint32_t slot_sz(const uint8_t* base, int lane, int g) {
  return *reinterpret_cast<const uint32_t*>(base + CODE_BYTES + g * LINE + ((((lane >> 2) ^ (g & 7)) << 4) | ((lane & 3) << 2)));
}
__device__ __forceinline__ float sum4(float2 a, float2 b, float2 c, float2 d) {
  return ((a.x + a.y) + (b.x + b.y)) + ((c.x + c.y) + (d.x + d.y));
}

__device__ __forceinline__ float fold_sz(uint32_t sz, float dot, float xsum, float v) {
  return fmaf(__uint_as_float(sz << 16), dot, fmaf(__uint_as_float(sz & 0xFFFF0000u), xsum, v));
}

// The work of one lane on one GEMV slot.  A warp's lanes are 8 row lanes x 4
// K quarters: lane (rr = lane & 7, kq = lane >> 3) takes rows rr + 8 i
// (i = 0..3) over the quarter's chunks 4 kq .. 4 kq + 3, so each input chunk
// it reads from shared memory (x, the slot's inputs from its first K value)
// serves four rows: a quarter of the input reads of one row per lane, and
// sixteen independent accumulator chains.  Per row i: int4 v[i] += s *
// (codes . x) + z * (sum of x) per group of G (a group never straddles a
// quarter); int8 / bf16 acc[i][] collect the dot product (int8: bias, the
// 128 * sum of x over the lane's chunks, is removed at the end).
template <int DT>
__device__ __forceinline__ void slot_dot(const uint8_t* base, int lane, int G, const float* x, const float* xs,
                                         float* v, float2 (*acc)[2], float& bias) {
  const float4* x4 = reinterpret_cast<const float4*>(x);
  const float2 z2 = make_float2(0.f, 0.f);
  const int rr = lane & 7, kq = lane >> 3;
  if (DT == DT_INT4) {
    const int cpg = G >> 5;
    float ga[4] = {0.f, 0.f, 0.f, 0.f};  // the running group's code . x, per row
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int u = kq * 4 + c;
      const float4* xu = x4 + u * 8;
      const float4 x0 = xu[0], x1 = xu[1], x2 = xu[2], x3 = xu[3], x4_ = xu[4], x5 = xu[5], x6 = xu[6], x7 = xu[7];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = rr + 8 * i;
        const uint4 q = slot_chunk(base, r, u);
        const float2 a0 = word_int4(q.x, x0, x1, z2), a1 = word_int4(q.y, x2, x3, z2);
        const float2 a2 = word_int4(q.z, x4_, x5, z2), a3 = word_int4(q.w, x6, x7, z2);
        const float sa = sum4(a0, a1, a2, a3);
        if (cpg == 1) {
          v[i] = fold_sz(slot_sz(base, r, u), sa, xs[u], v[i]);
        } else {
          ga[i] += sa;
          if (((c + 1) & (cpg - 1)) == 0) {  // group end
            const int g = u / cpg;
            v[i] = fold_sz(slot_sz(base, r, g), ga[i], xs[g], v[i]);
            ga[i] = 0.f;
          }
        }
      }
    }
  } else if (DT == DT_INT8) {
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int u = kq * 4 + c;
      const float4* xu = x4 + u * 4;
      const float4 x0 = xu[0], x1 = xu[1], x2 = xu[2], x3 = xu[3];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 q = slot_chunk(base, rr + 8 * i, u);
        acc[i][0] = word_int8(q.x, x0, acc[i][0]);
        acc[i][1] = word_int8(q.y, x1, acc[i][1]);
        acc[i][0] = word_int8(q.z, x2, acc[i][0]);
        acc[i][1] = word_int8(q.w, x3, acc[i][1]);
      }
      bias += xs[u];
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int u = kq * 4 + c;
      const float4 x0 = x4[u * 2], x1 = x4[u * 2 + 1];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 q = slot_chunk(base, rr + 8 * i, u);
        acc[i][0] = word_bf16(q.x, lo2(x0), acc[i][0]);
        acc[i][1] = word_bf16(q.y, hi2(x0), acc[i][1]);
        acc[i][0] = word_bf16(q.z, lo2(x1), acc[i][0]);
        acc[i][1] = word_bf16(q.w, hi2(x1), acc[i][1]);
      }
    }
  }
}

// The row sums of a lane's four rows over the warp's K-slots of a tile, added
// over the four K quarters; returns the total of row `lane` (lane l =
// (rr, kq) holds row rr + 8 kq among its four).
template <int DT>
__device__ __forceinline__ float rows_total(const float* v, float2 (*acc)[2], float bias, int lane) {
  float t[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    t[i] = DT == DT_INT4 ? v[i] : ((acc[i][0].x + acc[i][0].y) + (acc[i][1].x + acc[i][1].y)) - bias;
    t[i] += __shfl_xor_sync(0xffffffffu, t[i], 8);
    t[i] += __shfl_xor_sync(0xffffffffu, t[i], 16);
  }
  const int kq = lane >> 3;
  return kq == 0 ? t[0] : kq == 1 ? t[1] : kq == 2 ? t[2] : t[3];
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

// Epilogue of one output row n (value y); every lane calls it, lane r for
// row r of the tile; yp is the value of row n ^ 1 (its lane's partner).
__device__ __forceinline__ void gemv_epilogue(const Phase& ph, const Params& P, const Smem& S, int seg, int n, float y,
                                              float yp, int pos, float2 rp, ArgMax& am) {
  switch (ph.epi) {
    case EPI_STORE_BF16:
      reinterpret_cast<uint16_t*>(ph.out)[n] = f2bf(y);
      break;
    case EPI_STORE_F32:
      reinterpret_cast<float*>(ph.out)[n] = y;
      break;
    case EPI_RESID:
      // one writer per row and phase, phases ordered by grid barriers: the
      // fire-and-forget add is deterministic and hides the load latency
      atomicAdd(reinterpret_cast<float*>(ph.out) + n, y);
      break;
    case EPI_SWIGLU:
      if ((n & 1) == 0) reinterpret_cast<float*>(ph.out)[n >> 1] = y / (1.0f + expf(-y)) * yp;  // gate, up
      break;
    case EPI_QKV: {
      const int hd = ph.hd;
      if (n < ph.q_rows + ph.kv_rows) {
        if ((n & 1) == 0) {
          const bool isq = n < ph.q_rows;
          const int nn = isq ? n : n - ph.q_rows;
          const int d = nn % hd;
          const float o0 = y * rp.x - yp * rp.y, o1 = y * rp.y + yp * rp.x;  // (cos, sin) of the pair
          if (isq) {
            float* q = reinterpret_cast<float*>(ph.qbuf) + n;
            q[0] = o0;
            q[1] = o1;
          } else {
            uint16_t* k = ph.kc + ((size_t)(nn / hd) * ph.Tmax + pos) * hd + d;
            k[0] = f2bf(o0);
            k[1] = f2bf(o1);
          }
        }
      } else {
        const int nn = n - ph.q_rows - ph.kv_rows;
        ph.vc[((size_t)(nn / hd) * ph.Tmax + pos) * hd + nn % hd] = f2bf(y);
      }
      break;
    }
    case EPI_LOGITS:
      P.logits[n] = y;
      amax_merge(am, y, n);
      break;
    case EPI_MOE_SWIGLU:  // rows of a segment: gate j, up j interleaved; F = rows / 2
      if ((n & 1) == 0) reinterpret_cast<float*>(ph.out)[(size_t)seg * (ph.N / 4) + (n >> 1)] = y / (1.0f + expf(-y)) * yp;
      break;
    case EPI_MOE_RESID:
      atomicAdd(reinterpret_cast<float*>(ph.out) + n, S.red[40 + ph.moe - MOE_DOWN0] * y);
      break;
    default:
      break;
  }
}

// kv group whose q/k/v rows tile lt (32 rows of the stacked q/k/v matrix) holds
__device__ __forceinline__ int qkv_group(const Phase& ph, int lt) {
  const int n0 = lt * TR, gq = ph.Hq / ph.Hkv;
  if (n0 < ph.q_rows) return n0 / ph.hd / gq;
  if (n0 < ph.q_rows + ph.kv_rows) return (n0 - ph.q_rows) / ph.hd;
  return (n0 - ph.q_rows - ph.kv_rows) / ph.hd;
}

// One tile (32 rows lt*32.. of segment seg; its nb K-slots are the CTA's
// local slots j0 ..) for the calling warp: its K-slots, the deposit, and for
// the last contributing warp the combine.  Returns -1 if a wait gave up, 1
// for the combining warp (lane r holds in tot the sum of row lt*32 + r,
// already multiplied by the row's output factor, and in rp its RoPE pair),
// else 0.
template <int DT>
__device__ __forceinline__ int gemv_tile(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int seg, int Ns,
                                         int lt, uint32_t j0, int pos, float& tot, float2& rp) {
  const int nb = k_slots(DT, ph.K);
  const int lane = cs.lane, w = cs.warp;
  const int own0 = (int)((cs.it + j0) % NCW);  // owner of K-slot 0
  const int bfirst = (w - own0 + NCW) % NCW;   // this warp's first K-slot
  if (bfirst >= nb) return 0;
  const int ncontrib = nb < NCW ? nb : NCW;
  const int n = lt * TR + lane;
  // the epilogue's own inputs, fetched now so that their latency is hidden
  // behind the K-slots
  float pf = cs.rnorm * (DT == DT_BF16 ? 1.0f : DQ_UP);  // RMSNorm, 2^64, int8 row scale
  rp = make_float2(1.f, 0.f);
  if (n < Ns) {
    if (DT == DT_INT8) {
      const uint16_t* s8 = ph.s8;
      if (ph.moe != MOE_NONE) s8 += (size_t)S.bcast[32 + (ph.moe == MOE_GU ? seg : ph.moe - MOE_DOWN0)] * Ns;
      pf *= bf2f(s8[n]);
    }
    if (ph.epi == EPI_QKV && n < ph.q_rows + ph.kv_rows) {
      const int nn = n < ph.q_rows ? n : n - ph.q_rows;
      rp = P.rope[(size_t)pos * (ph.hd / 2) + (nn % ph.hd) / 2];
    }
  }
  float vr[4] = {0.f, 0.f, 0.f, 0.f}, bias = 0.0f;
  float2 acc[4][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = make_float2(0.f, 0.f);
  for (int b = bfirst; b < nb; b += NCW) {
    const uint32_t it = cs.it + j0 + (uint32_t)b;
    const uint8_t* base;
    if (!slot_acquire(S, cs, it, P.err, base)) return -1;
    const int k0 = b * slot_k(DT);
    slot_dot<DT>(base, lane, ph.G, S.xs + k0, S.xsum + (DT == DT_INT4 ? k0 / ph.G : k0 / 16), vr, acc, bias);
    slot_release(S, cs, it);
  }
  const float v = rows_total<DT>(vr, acc, bias, lane);
  // deposit this warp's 32 row sums, then the last contributor combines
  const int buf = (int)(cs.useq % NTB);
  float* tb = S.tb + (size_t)buf * NCW * TR;
  // the buffer's previous tile has been combined (bounded wait; in practice
  // it was long ago)
  int ok = 1;
  if (lane == 0) {
    ok = smem_wait(S.tbg + buf, (int)cs.useq, false, P.err, cs.lim);
    __threadfence_block();
  }
  if (!__shfl_sync(0xffffffffu, ok, 0)) return -1;
  tb[w * TR + lane] = v;
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    __threadfence_block();
    last = atomicAdd(S.tbc + buf, 1) == ncontrib - 1;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return 0;
  __threadfence_block();
  float t = 0.0f;
  for (int c = 0; c < ncontrib; ++c) t += tb[((own0 + c) % NCW) * TR + lane];  // K order
  __syncwarp();
  if (lane == 0) {
    S.tbc[buf] = 0;
    __threadfence_block();
    *reinterpret_cast<volatile int*>(S.tbg + buf) = (int)(cs.useq + NTB);  // hand the buffer on
  }
  tot = t * pf * (cs.wnorm ? warp_rnorm(ph, S) : 1.0f);
  return 1;
}

// One GEMV phase for this CTA: its tiles (round-robin over the CTAs); the
// combining warp of a tile runs the epilogue.
template <int DT>
__device__ bool gemv_phase(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta, int pos, ArgMax& am) {
  const int G = P.nctas, nb = k_slots(DT, ph.K);
  int Ns;
  int eseg[8];
  gemv_segments(ph, P, S, Ns, eseg);
  const int nseg = ph.moe == MOE_GU ? 2 : 1;
  const int tps = (Ns + TR - 1) / TR, ntiles = nseg * tps;
  const int lane = cs.lane;
  uint32_t j = 0;  // slot index within the phase
  for (int t = first_unit(cta, ph.rot, G); t < ntiles; t += G, ++cs.useq, j += (uint32_t)nb) {
    const int seg = t / tps, lt = t % tps;
    float tot;
    float2 rp;
    const int k = gemv_tile<DT>(ph, P, S, cs, seg, Ns, lt, j, pos, tot, rp);
    if (k < 0) return false;
    if (k == 0) continue;
    const int n = lt * TR + lane;
    const float yp = __shfl_xor_sync(0xffffffffu, tot, 1);
    if (n < Ns) gemv_epilogue(ph, P, S, seg, n, tot, yp, pos, rp, am);
    if (ph.headc) {
      // this tile's q/k/v rows are written: release them to the tile's kv
      // group (the warp barrier orders every lane's stores before lane 0's
      // release, so the waiting attention unit's acquire sees them all)
      __syncwarp();
      if (lane == 0)
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ph.headc + qkv_group(ph, lt)) : "memory");
    }
  }
  cs.it += j;
  return true;
}

// The o projection split by K-slot (PH_OSPLIT).  The CTA's units (tile,
// K-slot), round-robin over the CTAs, are one slot each, so each runs on one
// warp alone: it waits (bounded) until the attention of every kv group with a
// head in the K-slot has published its outputs, stages those SK inputs (fp32
// attention outputs, times the dequantisation powers, with their group sums)
// in its own shared-memory area, runs the slot, and adds the 32 partial row
// sums to the residual.  The FFN behind it waits for all of them at its grid
// barrier.
template <int DT>
__device__ bool osplit_phase(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta) {
  constexpr int SK = slot_k(DT), PL = SK / 32;  // inputs per slot, per lane
  const int G = P.nctas, nb = k_slots(DT, ph.K), tps = (ph.N + TR - 1) / TR;
  const int first = first_unit(cta, ph.rot, G), nu = units_of(first, tps * nb, G);
  const int lane = cs.lane, w = cs.warp, gq = ph.Hq / ph.Hkv;
  float* xw = S.xs + w * (512 + 32);  // this warp's inputs
  float* xsw = xw + 512;              // and their group / chunk sums
  const float* attn = reinterpret_cast<const float*>(ph.xptr);
  for (int k = 0; k < nu; ++k) {
    const uint32_t it = cs.it + (uint32_t)k;
    if ((int)(it % NCW) != w) continue;
    const int u = first + k * G, lt = u / nb, b = u % nb;
    // the kv groups of the slot's heads, one lane each, polled together
    const int h0 = b * SK / ph.hd, h1 = min((b * SK + SK - 1) / ph.hd, ph.Hq - 1);
    const int g = h0 / gq + lane;
    const bool mine = g <= h1 / gq;
    const bool ok = !mine || counter_wait(ph.attd + g, 1u, P.err, ERR_WAIT_HEAD, cs.lim);
    if (!__all_sync(0xffffffffu, ok)) return false;
    __syncwarp();  // the polling lanes' acquires order every lane's reads below
    // inputs b*SK .. b*SK + SK - 1: lane l holds PL consecutive ones
    float sg = 0.f;
#pragma unroll
    for (int q = 0; q < PL / 4; ++q) {
      const int f4 = lane * (PL / 4) + q, k4 = (b * SK) / 4 + f4;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (4 * k4 < ph.K) a = __ldcg(reinterpret_cast<const float4*>(attn) + k4);
      const float4 mu = dq_mult(DT, f4 & 7);
      reinterpret_cast<float4*>(xw)[f4] = make_float4(a.x * mu.x, a.y * mu.y, a.z * mu.z, a.w * mu.w);
      sg += (a.x + a.y) + (a.z + a.w);
    }
    if (DT != DT_BF16) {  // sums per int4 group / int8 chunk of 16
      const int span = DT == DT_INT4 ? ph.G / PL : 16 / PL;  // lanes per group / chunk
      for (int o = 1; o < span; o <<= 1) sg += __shfl_xor_sync(0xffffffffu, sg, o);
      if ((lane & (span - 1)) == 0) xsw[lane / span] = sg * (DT == DT_INT4 ? DQ_DOWN : 128.0f * DQ_DOWN);
    }
    __syncwarp();
    const uint8_t* base;
    if (!slot_acquire(S, cs, it, P.err, base)) return false;
    float vr[4] = {0.f, 0.f, 0.f, 0.f}, bias = 0.f;
    float2 acc[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = make_float2(0.f, 0.f);
    slot_dot<DT>(base, lane, ph.G, xw, xsw, vr, acc, bias);
    slot_release(S, cs, it);
    const float v = rows_total<DT>(vr, acc, bias, lane);
    const int n = lt * TR + lane;
    if (n < ph.N) {
      float f = DT == DT_BF16 ? 1.0f : DQ_UP;
      if (DT == DT_INT8) f *= bf2f(ph.s8[n]);
      atomicAdd(reinterpret_cast<float*>(ph.out) + n, v * f);
    }
    __syncwarp();  // the warp's inputs are read before the next unit restages them
  }
  cs.it += (uint32_t)nu;
  return true;
}

// One row of a down piece (16 columns: the SwiGLU outputs of one gate/up
// tile), its codes (q0, q1: int4 in q0.x/y, int8 in q0, bf16 in q0 and q1)
// and int4 scale/zero word, against those outputs,
// staged as the subnormal dequantisation reads them (xr; xz: their sum for
// the int4 zeros, or 128 times it for the int8 offset), without the 2^64 and
// int8 row scale that the phase end applies.
template <int DT>
__device__ __forceinline__ float down_row(uint4 q0, uint4 q1, uint32_t sz, const float4* xr, float xz) {
  if (DT == DT_INT4) {
    const float2 a0 = word_int4(q0.x, xr[0], xr[1], make_float2(0.f, 0.f));
    const float2 a1 = word_int4(q0.y, xr[2], xr[3], make_float2(0.f, 0.f));
    return fmaf(__uint_as_float(sz << 16), (a0.x + a1.x) + (a0.y + a1.y), __uint_as_float(sz & 0xFFFF0000u) * xz);
  } else if (DT == DT_INT8) {
    float2 a0 = word_int8(q0.x, xr[0], make_float2(0.f, 0.f));
    float2 a1 = word_int8(q0.z, xr[2], make_float2(0.f, 0.f));
    a0 = word_int8(q0.y, xr[1], a0);
    a1 = word_int8(q0.w, xr[3], a1);
    return ((a0.x + a1.x) + (a0.y + a1.y)) - xz;
  } else {
    float2 a0 = word_bf16(q0.x, lo2(xr[0]), make_float2(0.f, 0.f));
    float2 a1 = word_bf16(q1.x, lo2(xr[2]), make_float2(0.f, 0.f));
    a0 = word_bf16(q0.y, hi2(xr[0]), a0);
    a1 = word_bf16(q1.y, hi2(xr[2]), a1);
    a0 = word_bf16(q0.z, lo2(xr[1]), a0);
    a1 = word_bf16(q1.z, lo2(xr[3]), a1);
    a0 = word_bf16(q0.w, hi2(xr[1]), a0);
    a1 = word_bf16(q1.w, hi2(xr[3]), a1);
    return (a0.x + a1.x) + (a0.y + a1.y);
  }
}


// A dense FFN in one phase (PH_FFN).  For each of this CTA's gate/up tiles
// (round-robin): its K-slots as in a GEMV phase, whose combining warp writes
// silu(gate) * up of the tile's 16 pairs into a shared buffer instead of
// memory; then (one tile behind, so that those outputs are ready) the tile's
// 16-column slice of the down projection, one piece per warp: warp w always
// gets the rows w RW .., lane l rows l, l + 32, ..., and adds their products
// with the 16 outputs into the CTA's partial down outputs in shared memory
// (each row has one writer: no atomics, no ordering between warps).  At the
// end the CTA adds its partial outputs to the residual (vector atomics): the
// down projection needs no phase, no grid barrier and no staging of its own.
template <int DT>
__device__ bool ffn_phase(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta, int pos) {
  const int G = P.nctas, nb = k_slots(DT, ph.K);
  const int tps = ph.N / TR, d = ph.N2;
  const FfnSplit fs = ffn_split(DT, d);
  const int ND = NCW * fs.P;
  const int lane = cs.lane, w = cs.warp;
  float* hb = S.xs + round_up(ph.K, slot_k(DT));          // [FFN_HN][16] SwiGLU outputs of the tiles in flight
  int* hcnt = S.ffnc;                                     // [FFN_HN] rounds of each buffer written
  int* dcnt = hcnt + FFN_HN;                              // [FFN_HN] down pieces of each buffer finished
  float* dacc = hb + FFN_HN * 16;                         // [d] this CTA's partial down outputs
  // each warp zeroes the rows it owns (the counters are zero between phases)
  for (int i = w * fs.RW + lane; i < min((w + 1) * fs.RW, d); i += 32) dacc[i] = 0.0f;
  __syncwarp();
  const int first = first_unit(cta, ph.rot, G), nt = units_of(first, tps, G);
  const uint32_t X0 = cs.it;
  // the down pieces of local tile i for this warp
  auto down = [&](int i) -> bool {
    const int e = i % FFN_HN;
    const uint32_t pd = (i + 1 < nt) ? (uint32_t)((i + 2) * nb + i * ND) : (uint32_t)(nt * nb + i * ND);
    const int m0 = (w - (int)((X0 + pd) % NCW) + NCW) % NCW;
    // this tile's SwiGLU outputs (bounded wait)
    int ok = 1;
    if (lane == 0) {
      ok = smem_wait(hcnt + e, i / FFN_HN + 1, true, P.err, cs.lim);
      __threadfence_block();
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
    // the outputs as the subnormal dequantisation reads them (natural k order)
    float4 xr[4];
    float hs = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 t4 = reinterpret_cast<const float4*>(hb)[e * 4 + c];
      const float4 m = dq_mult(DT, DT == DT_INT4 ? c & 1 : 0);
      xr[c] = make_float4(t4.x * m.x, t4.y * m.y, t4.z * m.z, t4.w * m.w);
      hs += (t4.x + t4.y) + (t4.z + t4.w);
    }
    const float xz = DT == DT_INT4 ? hs * DQ_DOWN : DT == DT_INT8 ? 128.0f * hs * DQ_DOWN : 0.0f;
    for (int k = 0; k < fs.P; ++k) {
      const uint32_t it = X0 + pd + (uint32_t)(m0 + k * NCW);
      const uint8_t* base;
      if (!slot_acquire(S, cs, it, P.err, base)) return false;
      int r0, r1;
      ffn_piece(fs, d, w, k, r0, r1);
      const int nr = r1 - r0;
#pragma unroll 4
      for (int rl = lane; rl < nr; rl += 32) {
        uint4 q0, q1 = make_uint4(0u, 0u, 0u, 0u);
        uint32_t sz = 0u;
        if (DT == DT_INT4) {
          const uint2 t = reinterpret_cast<const uint2*>(base)[rl];
          q0 = make_uint4(t.x, t.y, 0u, 0u);
          sz = reinterpret_cast<const uint32_t*>(base + (size_t)fs.PR * 8)[rl];
        } else {
          q0 = reinterpret_cast<const uint4*>(base)[rl];
          if (DT == DT_BF16) q1 = reinterpret_cast<const uint4*>(base + (size_t)fs.PR * 16)[rl];
        }
        dacc[r0 + rl] += down_row<DT>(q0, q1, sz, xr, xz);
      }
      slot_release(S, cs, it);
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      atomicAdd(dcnt + e, 1);
    }
    return true;
  };
  for (int i = 0; i < nt; ++i, ++cs.useq) {
    const int t = first + i * G;
    const uint32_t pg = (uint32_t)(i * nb + (i > 0 ? (i - 1) * ND : 0));
    float tot;
    float2 rp;
    const int k = gemv_tile<DT>(ph, P, S, cs, 0, ph.N, t, pg, pos, tot, rp);
    if (k < 0) return false;
    if (k == 1) {
      const int e = i % FFN_HN;
      // the buffer's previous round has been read by every warp (bounded)
      int ok = 1;
      if (lane == 0) {
        ok = smem_wait(dcnt + e, NCW * (i / FFN_HN), true, P.err, cs.lim);
        __threadfence_block();
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      const float up = __shfl_xor_sync(0xffffffffu, tot, 1);
      if ((lane & 1) == 0) hb[e * 16 + (lane >> 1)] = tot / (1.0f + expf(-tot)) * up;
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        *reinterpret_cast<volatile int*>(hcnt + e) = i / FFN_HN + 1;
      }
    }
    // the previous tile's down slice follows this tile's gate/up slots
    if (i > 0 && !down(i - 1)) return false;
  }
  if (nt > 0 && !down(nt - 1)) return false;
  cs.it += (uint32_t)(nt * (nb + ND));
  // every warp's partial outputs are in dacc: add them to the residual
  if (!cta_sync(S, cs, P.err)) return false;
  if (cs.ctid < 2 * FFN_HN) S.ffnc[cs.ctid] = 0;  // for the next FFN phase
  if (nt > 0) {
    float4* out = reinterpret_cast<float4*>(ph.out);
    for (int n4 = cs.ctid; n4 < d / 4; n4 += NCW * 32) {
      float4 v = reinterpret_cast<const float4*>(dacc)[n4];
      if (DT != DT_BF16) {
        float f[4] = {DQ_UP, DQ_UP, DQ_UP, DQ_UP};
        if (DT == DT_INT8) {
          const uint2 s2 = *reinterpret_cast<const uint2*>(ph.s8b + 4 * n4);
          f[0] *= __uint_as_float(s2.x << 16);
          f[1] *= __uint_as_float(s2.x & 0xFFFF0000u);
          f[2] *= __uint_as_float(s2.y << 16);
          f[3] *= __uint_as_float(s2.y & 0xFFFF0000u);
        }
        v = make_float4(v.x * f[0], v.y * f[1], v.z * f[2], v.w * f[3]);
      }
      atomicAdd(out + n4, v);
    }
  }
  return true;
}

// ----------------------------------------------------------- attention ---
// One unit = one query row x one kv head x one chunk of positions.  Each slot
// (16 positions of K and V) belongs to the warp given by its stream index.  A
// warp takes the positions of a slot at once: lane l holds dims
// l*DPL .. l*DPL+DPL-1 (DPL = HD/32) of every position; it forms the 16
// partial dot products of its dims, a reduce-scatter over the lanes leaves
// lane l with the score of position l/2, and the block updates the warp's
// online softmax (m, l, o) once per q head: one rescale, one exponential per
// position, and the V sum weighted by each position's probability broadcast
// from its lane.  The warps merge in shared memory; a head split over several
// chunks merges its chunks' (m, l, o) in the CTA that finishes last
// (log-sum-exp combine).
// Sums each of 16 per-lane values over the 32 lanes; afterwards lane l holds
// the total of value l >> 1.
__device__ __forceinline__ float warp_rows16(float v[16], int lane) {
#pragma unroll
  for (int s = 16, n = 16; s >= 2; s >>= 1, n >>= 1) {
    const bool hi = lane & s;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float keep = hi ? v[k + n / 2] : v[k];
      const float send = hi ? v[k] : v[k + n / 2];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}
// Rows of one block, this lane's dims (bf16 pairs): NP positions of K or V.
template <int HD, int NP>
struct AttnRows {
  uint32_t w[NP][HD / 64];
};
// Loads positions 0..np-1 of NP rows (HD bf16 each, consecutive) starting at
// R; rows past np are zero.  GLOBAL: rows written during this launch, read
// around the L1 cache.
template <int HD, int NP, bool GLOBAL>
__device__ __forceinline__ void attn_rows(AttnRows<HD, NP>& r, const uint16_t* R, int np, int lane) {
  constexpr int DPL = HD / 32;
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const uint16_t* src = R + (size_t)i * HD + lane * DPL;
    if constexpr (DPL == 4) {
      uint2 t = make_uint2(0u, 0u);
      if (i < np) t = GLOBAL ? __ldcg(reinterpret_cast<const uint2*>(src)) : *reinterpret_cast<const uint2*>(src);
      r.w[i][0] = t.x;
      r.w[i][1] = t.y;
    } else {
      uint32_t t = 0u;
      if (i < np) t = GLOBAL ? __ldcg(reinterpret_cast<const unsigned*>(src)) : *reinterpret_cast<const uint32_t*>(src);
      r.w[i][0] = t;
    }
  }
}
// Scores of a block of np positions (K rows kr) for the gq q heads (q: this
// lane's dims of each head, pre-scaled by 1/sqrt(HD)); updates m and l and
// returns in pr[jj] the probability of position lane/2 (0 past np) and in
// cr[jj] the factor that rescales the head's running output.
template <int HD, int NP, int NG>
__device__ __forceinline__ void attn_scores(const AttnRows<HD, NP>& kr, int np, int gq, const float (*q)[HD / 32],
                                            float* m, float* l, float* pr, float* cr, int lane) {
  constexpr int DPL = HD / 32;
  const bool valid = (lane >> 1) < np;
#pragma unroll
  for (int jj = 0; jj < NG; ++jj) {
    pr[jj] = 0.f;
    cr[jj] = 1.f;
    if (jj < gq) {
      float part[ATT_POS_PER_SLOT];
#pragma unroll
      for (int i = 0; i < ATT_POS_PER_SLOT; ++i) {
        float d = 0.f;
        if (i < NP) {
#pragma unroll
          for (int e = 0; e < DPL / 2; ++e) {
            d = fmaf(q[jj][2 * e], __uint_as_float(kr.w[i][e] << 16), d);
            d = fmaf(q[jj][2 * e + 1], __uint_as_float(kr.w[i][e] & 0xFFFF0000u), d);
          }
        }
        part[i] = d;
      }
      float sc = warp_rows16(part, lane);  // score of position lane / 2 (all lanes shuffle)
      if (!valid) sc = -INFINITY;
      float mx = sc;
#pragma unroll
      for (int of = 2; of < 32; of <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, of));
      const float mn = fmaxf(m[jj], mx);
      cr[jj] = expf(m[jj] - mn);  // 0 while the state is empty (m = -inf)
      pr[jj] = valid ? expf(sc - mn) : 0.f;
      float ps = 0.5f * pr[jj];  // each position sits in two lanes
#pragma unroll
      for (int of = 1; of < 32; of <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, of);
      l[jj] = fmaf(l[jj], cr[jj], ps);
      m[jj] = mn;
    }
  }
}
// o = o * cr + sum_i pr_i v_i for each head (V rows vr).
template <int HD, int NP, int NG>
__device__ __forceinline__ void attn_values(const AttnRows<HD, NP>& vr, int gq, const float* pr, const float* cr,
                                            float (*o)[HD / 32]) {
  constexpr int DPL = HD / 32;
#pragma unroll
  for (int jj = 0; jj < NG; ++jj) {
    if (jj < gq) {
#pragma unroll
      for (int d = 0; d < DPL; ++d) o[jj][d] *= cr[jj];
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const float pi = __shfl_sync(0xffffffffu, pr[jj], 2 * i);
#pragma unroll
        for (int e = 0; e < DPL / 2; ++e) {
          o[jj][2 * e] = fmaf(pi, __uint_as_float(vr.w[i][e] << 16), o[jj][2 * e]);
          o[jj][2 * e + 1] = fmaf(pi, __uint_as_float(vr.w[i][e] & 0xFFFF0000u), o[jj][2 * e + 1]);
        }
      }
    }
  }
}

// The outputs of kv group kvh's heads are written (by this CTA's threads):
// publish that for the o projection units waiting on the group (PH_OSPLIT).
// The CTA barrier orders every thread's stores before thread 0's release.
__device__ __forceinline__ bool attn_done(const Phase& ph, const Smem& S, Cons& cs, const Params& P, int kvh) {
  if (!ph.attd) return true;
  if (!cta_sync(S, cs, P.err)) return false;
  if (cs.ctid == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ph.attd + kvh) : "memory");
  return true;
}

// NG: the largest number of q heads per kv head this copy handles (1, 2 or
// 4); the per-head loops and registers are sized by it, so a model with one
// q head per kv head runs a quarter of the code.
template <int HD, int NG, bool VER>
__device__ bool attn_unit(const Phase& ph, const Params& P, const Smem& S, Cons& cs, const AttnUnit& au, int pos,
                          uint32_t& j) {
  constexpr int DPL = HD / 32;
  const int gq = ph.Hq / ph.Hkv;
  const int kvh = au.kvh, c = au.c, nch = au.nch;
  const int p0 = au.p0, p1 = au.p1, pe = min(p1, au.Ts);
  const int lane = cs.lane, w = cs.warp;
  const size_t qrow = (size_t)au.m * ph.Hq * HD;  // this unit's query / output row
  float* qs = S.xs;                       // [gq][HD], pre-scaled by 1/sqrt(HD)
  float* sc = S.xs + MAX_GQ * HD;         // [NCW][gq][HD + 2]
  constexpr int APS = att_slot_pos(HD);  // positions of K and V in a slot
  const int nslots = pe > p0 ? (pe - p0 + APS - 1) / APS : 0;
  // the q/k/v rows of this kv group written during this launch (by the
  // q/k/v tiles of every CTA, in the same phase): bounded wait on the group's
  // tile count
  if (ph.headc) {
    int ok = 1;
    if (cs.ctid == 0)
      ok = counter_wait(ph.headc + kvh, (unsigned)((gq + 2) * (HD / TR)), P.err, ERR_WAIT_HEAD, cs.lim);
    S.bcast[1] = ok;
    if (!cta_sync(S, cs, P.err) || !S.bcast[1]) return false;
  }
  // positions not streamed (rows written during this launch, at most 8) go
  // to the warp after the last slot's owner, which loads them right away
  const int pg = max(pe, p0);
  const int gw = (int)((cs.it + j + (uint32_t)nslots) % NCW);
  const bool has_g = (w == gw) && pg < p1;
  // rows written during this launch: a verify pass's own rows (at most
  // MAX_M) or a decode step's current row
  constexpr int NPG = VER ? MAX_M : 1;
  AttnRows<HD, NPG> gk, gv;
  if (has_g) {
    const size_t off = ((size_t)kvh * ph.Tmax + pg) * HD;
    attn_rows<HD, NPG, true>(gk, ph.kc + off, p1 - pg, lane);
    attn_rows<HD, NPG, true>(gv, ph.vc + off, p1 - pg, lane);
  }
  const float scale = rsqrtf((float)HD);
  for (int i = cs.ctid; i < gq * HD; i += NCW * 32) {
    const size_t qi = qrow + (size_t)kvh * gq * HD + i;
    const float qv = ph.q_f32 ? __ldcg(reinterpret_cast<const float*>(ph.qbuf) + qi)
                              : bf2f(__ldcg(reinterpret_cast<const uint16_t*>(ph.qbuf) + qi));
    qs[i] = qv * scale;
  }
  if (!cta_sync(S, cs, P.err)) return false;

  float q[NG][DPL], m[NG], l[NG], o[NG][DPL];
#pragma unroll
  for (int jj = 0; jj < NG; ++jj) {
    m[jj] = -INFINITY;
    l[jj] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
      q[jj][d] = jj < gq ? qs[jj * HD + lane * DPL + d] : 0.f;
      o[jj][d] = 0.f;
    }
  }
  float pr[NG], cr[NG];
  if (has_g) {
    attn_scores<HD, NPG, NG>(gk, p1 - pg, gq, q, m, l, pr, cr, lane);
    attn_values<HD, NPG, NG>(gv, gq, pr, cr, o);
  }
  for (int k = (w - (int)((cs.it + j) % NCW) + NCW) % NCW; k < nslots; k += NCW) {
    const uint32_t it = cs.it + j + (uint32_t)k;
    const int np = min(APS, pe - (p0 + k * APS));
    const uint8_t* base;
    if (!slot_acquire(S, cs, it, P.err, base)) return false;
    const uint16_t* kb = reinterpret_cast<const uint16_t*>(base);
    {
      AttnRows<HD, APS> kr;
      attn_rows<HD, APS, false>(kr, kb, np, lane);
      attn_scores<HD, APS, NG>(kr, np, gq, q, m, l, pr, cr, lane);
    }
    {
      AttnRows<HD, APS> vr;
      attn_rows<HD, APS, false>(vr, kb + APS * HD, np, lane);
      slot_release(S, cs, it);  // the slot's rows are in registers
      attn_values<HD, APS, NG>(vr, gq, pr, cr, o);
    }
  }
  j += (uint32_t)nslots;
  // the warps of this CTA merge in shared memory
#pragma unroll
  for (int jj = 0; jj < NG; ++jj) {
    if (jj < gq) {
      float* dst = sc + (w * gq + jj) * (HD + 2);
#pragma unroll
      for (int d = 0; d < DPL; ++d) dst[2 + lane * DPL + d] = o[jj][d];
      if (lane == 0) {
        dst[0] = m[jj];
        dst[1] = l[jj];
      }
    }
  }
  if (!cta_sync(S, cs, P.err)) return false;
  const int stride = HD + 2;
  for (int i = cs.ctid; i < gq * HD; i += NCW * 32) {
    const int jj = i / HD, d = i % HD;
    float M = -INFINITY;
    for (int ww = 0; ww < NCW; ++ww) M = fmaxf(M, sc[(ww * gq + jj) * stride]);
    float L = 0.f, O = 0.f;
    for (int ww = 0; ww < NCW; ++ww) {
      const float* s = sc + (ww * gq + jj) * stride;
      const float e = s[1] > 0.f ? expf(s[0] - M) : 0.f;
      L = fmaf(s[1], e, L);
      O = fmaf(s[2 + d], e, O);
    }
    const int hq = kvh * gq + jj;
    if (nch == 1) {  // the whole head was here
      if (ph.out_f32) reinterpret_cast<float*>(ph.attn_out)[qrow + (size_t)hq * HD + d] = O / L;
      else reinterpret_cast<uint16_t*>(ph.attn_out)[qrow + (size_t)hq * HD + d] = f2bf(O / L);
    } else {
      float* part = ph.part + (((size_t)au.m * ph.Hq + hq) * nch + c) * stride;
      part[2 + d] = O;
      if (d == 0) {
        part[0] = M;
        part[1] = L;
      }
    }
  }
  if (nch == 1) return attn_done(ph, S, cs, P, kvh);
  __threadfence();
  if (!cta_sync(S, cs, P.err)) return false;
  unsigned* tick = ph.tick + (size_t)au.m * ph.Hkv + kvh;
  if (cs.ctid == 0) {
    const unsigned old = atomicAdd(tick, 1u);
    S.bcast[0] = (old == (unsigned)(nch - 1));
  }
  if (!cta_sync(S, cs, P.err)) return false;
  if (S.bcast[0]) {
    __threadfence();
    for (int i = cs.ctid; i < gq * HD; i += NCW * 32) {
      const int jj = i / HD, d = i % HD, hq = kvh * gq + jj;
      const float* pb = ph.part + ((size_t)au.m * ph.Hq + hq) * nch * stride;
      float M = -INFINITY;
      for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(pb + cc * stride));
      float L = 0.f, O = 0.f;
      for (int cc = 0; cc < nch; ++cc) {
        const float e = expf(__ldcg(pb + cc * stride) - M);
        L = fmaf(__ldcg(pb + cc * stride + 1), e, L);
        O = fmaf(__ldcg(pb + cc * stride + 2 + d), e, O);
      }
      if (ph.out_f32) reinterpret_cast<float*>(ph.attn_out)[qrow + (size_t)hq * HD + d] = O / L;
      else reinterpret_cast<uint16_t*>(ph.attn_out)[qrow + (size_t)hq * HD + d] = f2bf(O / L);
    }
    if (cs.ctid == 0) *tick = 0u;
    return attn_done(ph, S, cs, P, kvh);
  }
  return true;
}

// Attention runs out of line, on copies of the consumer state, so that its
// register needs (per-position rows, softmax state of up to four heads) do
// not push the GEMV loops' values out to local memory.
struct AttnRet {
  uint32_t j, cphase, starved;
  int ok;
};
template <int HD, int NG, bool VER>
__device__ __noinline__ AttnRet attn_call(const Phase& ph, const Params& P, const Smem S, Cons cs, const AttnUnit au,
                                          int pos, uint32_t j) {
  AttnRet r;
  r.ok = attn_unit<HD, NG, VER>(ph, P, S, cs, au, pos, j);
  r.j = j;
  r.cphase = cs.cphase;
  r.starved = cs.starved;
  return r;
}

// ========================================================= verify pass ====
// A speculative-verification pass (gpt-fast README, "Speculative sampling")
// feeds M rows (the last accepted token and the drafts) at positions
// pos..pos+M-1 through every layer with ONE stream of the weights.  GEMV
// phases then work K-slot by K-slot over groups of up to VTG tiles: the CTA
// stages the K-slot's inputs of all M rows (fp32, times the dequantisation
// powers), each slot's owner warp dequantises its codes once (lane r: row r)
// and multiplies them with the M rows, and adds its rows' M sums into a
// shared accumulator (each (row, m) has one writer per K-slot, K-slots in
// order: deterministic); the group's epilogues then run per (row, m).
// A multi-row GEMV stages its M input rows VKB K values at a time (one
// staging round covers VKB / slot_k K-slots: 2 int4, 4 int8, 8 bf16), so
// that every round keeps all consumer warps busy and the rounds' staging
// latency and barriers are paid K / VKB times per tile group.
constexpr int VKB = 1024;
struct VS {
  float* xk;    // [MAX_M][VKB] inputs of the current round
  float* xgk;   // [MAX_M][64] sums of the inputs per int4 group / int8 chunk, as S.xsum
  float* acc;   // [VTG * TR][MAX_M] row sums of the tile group
  float* rfac;  // [MAX_M] RMSNorm factors
};
__device__ __forceinline__ VS vsmem(const Smem& S) {
  VS v;
  v.xk = S.xs;
  v.xgk = v.xk + MAX_M * VKB;
  v.acc = v.xgk + MAX_M * 64;
  v.rfac = v.acc + VTG * TR * MAX_M;
  return v;
}
static_assert(MAX_M * VKB + MAX_M * 64 + VTG * TR * MAX_M + MAX_M <= KMAX, "verify staging area");
static_assert(VKB / 32 <= 64 && VKB / 16 <= 64, "verify group sums per row");

// Row m of the phase's input, element k: the source a decode step would read.
__device__ __forceinline__ float4 vin4(const Phase& ph, const Params& P, const VS& V, int m, int e, int k4) {
  if (ph.xsrc == X_F32) {
    const float* x = reinterpret_cast<const float*>(ph.xptr) + (size_t)m * ph.x_mstride + (size_t)e * ph.x_sstride;
    return __ldcg(reinterpret_cast<const float4*>(x) + k4);
  }
  float4 a;
  if (ph.xsrc == X_EMBED_NORM) a = bf4(*reinterpret_cast<const uint2*>(P.embed + (size_t)P.tokens[m] * ph.K + 4 * k4));
  else a = __ldcg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(ph.xptr) + (size_t)m * ph.K) + k4);
  const float4 g = bf4(reinterpret_cast<const uint2*>(ph.gain)[k4]);
  const float r = V.rfac[m];
  return make_float4(a.x * r * g.x, a.y * r * g.y, a.z * r * g.z, a.w * r * g.w);
}

// RMSNorm factors of the M rows (and, for the first layer, the residual rows
// written from the embedding by CTA 0).
__device__ bool verify_norm(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta) {
  const VS V = vsmem(S);
  const int K4 = ph.K / 4;
  for (int m = cs.warp; m < P.M; m += NCW) {
    float ss = 0.f;
    for (int k4 = cs.lane; k4 < K4; k4 += 32) {
      float4 a;
      if (ph.xsrc == X_EMBED_NORM) {
        a = bf4(*reinterpret_cast<const uint2*>(P.embed + (size_t)P.tokens[m] * ph.K + 4 * k4));
        if (cta == 0) reinterpret_cast<float4*>(P.resid + (size_t)m * ph.K)[k4] = a;
      } else {
        a = __ldcg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(ph.xptr) + (size_t)m * ph.K) + k4);
      }
      ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (cs.lane == 0) V.rfac[m] = 1.0f / sqrtf(ss / (float)ph.K + ph.eps);
  }
  return cta_sync(S, cs, P.err);
}

// Router of a verify pass: logits for every (row, expert), top-2 per row,
// weights into moew (0 for experts a row did not choose), and the union of
// the chosen experts in index order for the producer.
__device__ bool verify_route(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int pi) {
  const VS V = vsmem(S);
  const int K4 = ph.K / 4, E = ph.n_experts;
  float* rl = S.moew;  // logits first, weights after
  for (int q = cs.warp; q < P.M * E; q += NCW) {
    const int m = q / E, e = q % E;
    const uint2* wr = reinterpret_cast<const uint2*>(ph.router + (size_t)e * ph.K);
    float acc = 0.f;
    for (int k4 = cs.lane; k4 < K4; k4 += 32) {
      const float4 x = vin4(ph, P, V, m, 0, k4);
      const float4 wv = bf4(wr[k4]);
      acc = fmaf(x.x, wv.x, fmaf(x.y, wv.y, fmaf(x.z, wv.z, fmaf(x.w, wv.w, acc))));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (cs.lane == 0) rl[m * 8 + e] = acc;
  }
  if (!cta_sync(S, cs, P.err)) return false;
  if (cs.ctid == 0) {
    unsigned used = 0u;
    for (int m = 0; m < P.M; ++m) {
      float* r = rl + m * 8;
      int e1 = 0;
      for (int e = 1; e < E; ++e)
        if (r[e] > r[e1]) e1 = e;
      int e2 = e1 == 0 ? 1 : 0;
      for (int e = 0; e < E; ++e)
        if (e != e1 && r[e] > r[e2]) e2 = e;
      const float b = expf(r[e2] - r[e1]);
      const float w1 = 1.0f / (1.0f + b), w2 = b / (1.0f + b);
      for (int e = 0; e < 8; ++e) r[e] = e == e1 ? w1 : e == e2 ? w2 : 0.0f;
      used |= (1u << e1) | (1u << e2);
    }
    int n = 0;
    for (int e = 0; e < E; ++e)
      if (used & (1u << e)) S.bcast[48 + n++] = e;
    S.bcast[56] = n;
    __threadfence_block();
    *reinterpret_cast<volatile int*>(S.bcast + 34) = pi + 1;  // releases the producer
  }
  return cta_sync(S, cs, P.err);
}

// Epilogue of row n (value y, partner row n ^ 1 value yp) for input row m.
__device__ __forceinline__ void gemv_epilogue_m(const Phase& ph, const Params& P, const Smem& S, int e, int n, int m,
                                                float y, float yp, int pos, ArgMax* am) {
  switch (ph.epi) {
    case EPI_STORE_F32:
      reinterpret_cast<float*>(ph.out)[(size_t)m * ph.out_mstride + n] = y;
      break;
    case EPI_RESID:
      atomicAdd(reinterpret_cast<float*>(ph.out) + (size_t)m * ph.out_mstride + n, y);
      break;
    case EPI_SWIGLU:
      if ((n & 1) == 0) reinterpret_cast<float*>(ph.out)[(size_t)m * ph.out_mstride + (n >> 1)] = y / (1.0f + expf(-y)) * yp;
      break;
    case EPI_MOE_SWIGLU:  // h of (row m, expert e)
      if ((n & 1) == 0)
        reinterpret_cast<float*>(ph.out)[((size_t)m * 8 + e) * ph.out_mstride + (n >> 1)] = y / (1.0f + expf(-y)) * yp;
      break;
    case EPI_MOE_RESID: {
      const float wgt = S.moew[m * 8 + e];
      if (wgt != 0.0f) atomicAdd(reinterpret_cast<float*>(ph.out) + (size_t)m * ph.out_mstride + n, wgt * y);
      break;
    }
    case EPI_QKV: {
      const int hd = ph.hd, p = pos + m;
      if (n < ph.q_rows + ph.kv_rows) {
        if ((n & 1) == 0) {
          const bool isq = n < ph.q_rows;
          const int nn = isq ? n : n - ph.q_rows;
          const int d = nn % hd;
          const float2 cs = P.rope[(size_t)p * (hd / 2) + d / 2];
          const float o0 = y * cs.x - yp * cs.y, o1 = y * cs.y + yp * cs.x;
          if (isq) {
            float* q = reinterpret_cast<float*>(ph.qbuf) + (size_t)m * ph.q_rows + n;
            q[0] = o0;
            q[1] = o1;
          } else {
            uint16_t* k = ph.kc + ((size_t)(nn / hd) * ph.Tmax + p) * hd + d;
            k[0] = f2bf(o0);
            k[1] = f2bf(o1);
          }
        }
      } else {
        const int nn = n - ph.q_rows - ph.kv_rows;
        ph.vc[((size_t)(nn / hd) * ph.Tmax + p) * hd + nn % hd] = f2bf(y);
      }
      break;
    }
    case EPI_LOGITS:
      P.logits[(size_t)m * P.vocab + n] = y;
      amax_merge(am[m], y, n);
      break;
    default:
      break;
  }
}

template <int DT>
__device__ bool gemv_phase_m(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta, int pos, int pi,
                             ArgMax* am) {
  constexpr int SK = slot_k(DT);  // K values per slot
  const VS V = vsmem(S);
  const int M = P.M, K = ph.K, Gq = ph.G;
  const int nb = k_slots(DT, K);
  const int lane = cs.lane, w = cs.warp;
  if ((ph.xsrc == X_NORM || ph.xsrc == X_EMBED_NORM) && !verify_norm(ph, P, S, cs, cta)) return false;
  if (ph.moe == MOE_GU && !verify_route(ph, P, S, cs, pi)) return false;
  int Ns;
  int eseg[8];
  const int nseg = gemv_segments(ph, P, S, Ns, eseg);
  TileGroups tg;
  tg.tps = (Ns + TR - 1) / TR;
  tg.ntiles = nseg * tg.tps;
  tg.G = P.nctas;
  tg.first = first_unit(cta, ph.rot, P.nctas);
  for (int i = cs.ctid; i < VTG * TR * MAX_M; i += NCW * 32) V.acc[i] = 0.f;
  const float4* xk4 = reinterpret_cast<const float4*>(V.xk);
  uint32_t j = 0;
  for (int i0 = 0; tg.first + i0 * tg.G < tg.ntiles;) {
    const int i1 = group_end(tg, i0);
    const int seg = (tg.first + i0 * tg.G) / tg.tps, e = eseg[seg];
    constexpr int KR = VKB / SK, PM = VKB / 4;  // K-slots and float4 per row of a round
    for (int b0 = 0; b0 < nb; b0 += KR) {
      const int b1 = min(nb, b0 + KR);
      // stage the round's inputs of the M rows, zero past K (one row per
      // iteration, whole warps of consecutive float4, so that group sums
      // shuffle within a warp)
      constexpr int VB = 4;  // rows whose loads are in flight together
      static_assert(PM == NCW * 32, "one staging pass per row");
      for (int m0 = 0; m0 < M; m0 += VB) {
        const int f4 = cs.ctid;
        const bool inK = b0 * (SK / 4) + f4 < K / 4;
        float4 a[VB];
#pragma unroll
        for (int r = 0; r < VB; ++r) {
          a[r] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (m0 + r < M && inK) a[r] = vin4(ph, P, V, m0 + r, e, b0 * (SK / 4) + f4);
        }
        const float4 mu = dq_mult(DT, f4 & 7);
#pragma unroll
        for (int r = 0; r < VB; ++r) {
          const int m = m0 + r;
          if (m >= M) break;  // uniform
          reinterpret_cast<float4*>(V.xk)[m * PM + f4] =
              make_float4(a[r].x * mu.x, a[r].y * mu.y, a[r].z * mu.z, a[r].w * mu.w);
          if (DT != DT_BF16) {  // group / chunk sums as in stage_store
            float sg = a[r].x + a[r].y + a[r].z + a[r].w;
            const int span = DT == DT_INT4 ? Gq / 4 : 4;
            for (int o = 1; o < span; o <<= 1) sg += __shfl_xor_sync(0xffffffffu, sg, o);
            if ((lane & (span - 1)) == 0)
              V.xgk[m * 64 + (4 * f4) / (DT == DT_INT4 ? Gq : 16)] = sg * (DT == DT_INT4 ? DQ_DOWN : 128.0f * DQ_DOWN);
          }
        }
      }
      if (!cta_sync(S, cs, P.err)) return false;
      for (int b = b0; b < b1; ++b) {
      const int kb = (b - b0) * SK;  // the K-slot's first input within the round
      for (int i = i0; i < i1; ++i, ++j) {
        const uint32_t it = cs.it + j;
        if ((int)(it % NCW) != w) continue;
        const uint8_t* base;
        if (!slot_acquire(S, cs, it, P.err, base)) return false;
        float2 a[MAX_M];
        float v[MAX_M];
#pragma unroll
        for (int m = 0; m < MAX_M; ++m) {
          a[m] = make_float2(0.f, 0.f);
          v[m] = 0.f;
        }
        const int cpg = DT == DT_INT4 ? Gq / 32 : 1;
#pragma unroll 1
        for (int u = 0; u < SLOT_CHUNKS; ++u) {
          const uint4 qv = slot_chunk(base, lane, u);
          const uint32_t wq[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
          for (int jw = 0; jw < 4; ++jw) {
            const uint32_t wv = wq[jw];
            if (DT == DT_INT4) {  // the subnormal reading of word_int4
              const uint32_t hv = wv >> 8;
              const float2 c0 = bits2(wv & 0x0000000Fu, wv & 0x000000F0u), c1 = bits2(wv & 0x00000F00u, wv & 0x0000F000u);
              const float2 c2 = bits2(wv & 0x000F0000u, wv & 0x00F00000u), c3 = bits2(hv & 0x000F0000u, hv & 0x00F00000u);
#pragma unroll
              for (int m = 0; m < MAX_M; ++m) {
                if (m < M) {
                  const float4* xm = xk4 + m * PM + kb / 4 + u * 8 + 2 * jw;
                  const float4 xa = xm[0], xb = xm[1];
                  a[m] = ffma2(c0, lo2(xa), a[m]);
                  a[m] = ffma2(c1, hi2(xa), a[m]);
                  a[m] = ffma2(c2, lo2(xb), a[m]);
                  a[m] = ffma2(c3, hi2(xb), a[m]);
                }
              }
            } else if (DT == DT_INT8) {  // as word_int8
              const uint32_t hv = wv >> 8;
              const float2 c0 = bits2(wv & 0x000000FFu, wv & 0x0000FF00u), c1 = bits2(wv & 0x00FF0000u, hv & 0x00FF0000u);
#pragma unroll
              for (int m = 0; m < MAX_M; ++m) {
                if (m < M) {
                  const float4 xa = xk4[m * PM + kb / 4 + u * 4 + jw];
                  a[m] = ffma2(c0, lo2(xa), a[m]);
                  a[m] = ffma2(c1, hi2(xa), a[m]);
                }
              }
            } else {
              const float2 c0 = bits2(wv << 16, wv & 0xFFFF0000u);
#pragma unroll
              for (int m = 0; m < MAX_M; ++m) {
                if (m < M) {
                  const float4 xa = xk4[m * PM + kb / 4 + u * 2 + (jw >> 1)];
                  a[m] = ffma2(c0, (jw & 1) ? hi2(xa) : lo2(xa), a[m]);
                }
              }
            }
          }
          if (DT == DT_INT4) {
            if ((u + 1) % cpg == 0) {  // group end: scale and zero
              const int gi = u / cpg;
              const uint32_t sz = slot_sz(base, lane, gi);
#pragma unroll
              for (int m = 0; m < MAX_M; ++m) {
                v[m] = fmaf(__uint_as_float(sz << 16), a[m].x + a[m].y,
                            fmaf(__uint_as_float(sz & 0xFFFF0000u), V.xgk[m * 64 + kb / Gq + gi], v[m]));
                a[m] = make_float2(0.f, 0.f);
              }
            }
          } else if (DT == DT_INT8) {
#pragma unroll
            for (int m = 0; m < MAX_M; ++m) v[m] -= V.xgk[m * 64 + kb / 16 + u];
          }
        }
        slot_release(S, cs, it);
        // several warps hold K-slots of the same tile in one round
        float* accr = V.acc + ((i - i0) * TR + lane) * MAX_M;
#pragma unroll
        for (int m = 0; m < MAX_M; ++m) {
          if (m < M) atomicAdd(accr + m, DT == DT_INT4 ? v[m] : (a[m].x + a[m].y) + v[m]);
        }
      }
      }
      if (!cta_sync(S, cs, P.err)) return false;
    }
    // epilogues of the group: one thread per (row pair, m)
    const uint16_t* s8 = ph.s8;
    if (DT == DT_INT8 && ph.moe != MOE_NONE) s8 += (size_t)e * Ns;
    for (int q = cs.ctid; q < (i1 - i0) * (TR / 2) * M; q += NCW * 32) {
      const int m = q % M, pr = q / M, gi = pr / (TR / 2), r = (pr % (TR / 2)) * 2;
      const int t = tg.first + (i0 + gi) * tg.G, lt = t % tg.tps;
      const int Rt = min(TR, Ns - lt * TR);
      for (int k = 0; k < 2; ++k) {
        if (r + k >= Rt) break;
        const int n = lt * TR + r + k;
        float y = V.acc[(gi * TR + r + k) * MAX_M + m];
        float yp = (r + (k ^ 1) < Rt) ? V.acc[(gi * TR + r + (k ^ 1)) * MAX_M + m] : 0.f;
        if (DT == DT_INT4) {
          y *= DQ_UP;
          yp *= DQ_UP;
        } else if (DT == DT_INT8) {
          y *= DQ_UP * bf2f(s8[n]);
          if (r + (k ^ 1) < Rt) yp *= DQ_UP * bf2f(s8[n ^ 1]);
        }
        gemv_epilogue_m(ph, P, S, e, n, m, y, yp, pos, am);
      }
    }
    if (!cta_sync(S, cs, P.err)) return false;
    for (int q = cs.ctid; q < VTG * TR * MAX_M; q += NCW * 32) V.acc[q] = 0.f;
    if (!cta_sync(S, cs, P.err)) return false;
    i0 = i1;
  }
  cs.it += j;
  return true;
}

// Argmax of every row of a verify pass, then the greedy acceptance: with a_m
// the argmax of row m and d_i = tokens[i] the drafts, n = the largest n with
// a_{i-1} == d_i for all i <= n; next token a_n; the position advances by n+1.
__device__ bool verify_finish(const Params& P, const Smem& S, Cons& cs, int cta, ArgMax* am) {
  for (int m = 0; m < P.M; ++m) {
    ArgMax a = am[m];
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float v = __shfl_xor_sync(0xffffffffu, a.v, o);
      const int i = __shfl_xor_sync(0xffffffffu, a.i, o);
      amax_merge(a, v, i);
    }
    if (cs.lane == 0) {
      S.red[cs.warp * MAX_M + m] = a.v;
      S.bcast[64 + cs.warp * MAX_M + m] = a.i;
    }
  }
  if (!cta_sync(S, cs, P.err)) return false;
  if (cs.warp == 0) {
    int last = 0;
    if (cs.lane == 0) {
      for (int m = 0; m < P.M; ++m) {
        ArgMax b = {S.red[m], S.bcast[64 + m]};
        for (int w = 1; w < NCW; ++w) amax_merge(b, S.red[w * MAX_M + m], S.bcast[64 + w * MAX_M + m]);
        P.amax_val[cta * MAX_M + m] = b.v;
        P.amax_idx[cta * MAX_M + m] = b.i;
      }
      __threadfence();
      last = atomicAdd(P.amax_tick, 1u) == (unsigned)(P.nctas - 1);
    }
    if (__shfl_sync(0xffffffffu, last, 0)) {
      // the last CTA merges every CTA's candidates: 32 lanes load in parallel
      __threadfence();
      int a[MAX_M];
      for (int m = 0; m < P.M; ++m) {
        ArgMax g = {-INFINITY, 0x7fffffff};
        for (int k = cs.lane; k < P.nctas; k += 32)
          amax_merge(g, __ldcg(P.amax_val + k * MAX_M + m), __ldcg(P.amax_idx + k * MAX_M + m));
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float v = __shfl_xor_sync(0xffffffffu, g.v, o);
          const int i = __shfl_xor_sync(0xffffffffu, g.i, o);
          amax_merge(g, v, i);
        }
        a[m] = g.i;
      }
      if (cs.lane == 0) {
      int n = 0;
      if (P.prefill) n = P.M - 1;  // a prompt: every row is the caller's
      else
        while (n < P.M - 1 && a[n] == P.tokens[n + 1]) ++n;
      *P.n_accepted = n;
      *P.next_token = a[n];
      *P.amax_tick = 0u;
      int* pos = const_cast<int*>(P.d_pos);
      *pos = *pos + n + 1;
      }
    }
  }
  return true;
}

// ------------------------------------------------------- MoE router -----
// Top-2 router of a mixture-of-experts layer ("Efficiently implementing the
// Mixtral 8x7B model with gpt-fast"; gpt-fast README, "Mixtral 8x7B"):
// logits r_e = x . Wr[e] over the staged (normalised) input, the two largest
// (lower index first on ties), weights = softmax over those two.  Every CTA
// computes the same logits in the same order, so all agree on the experts.
__device__ bool route_experts(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int pi) {
  const int K = ph.K, K4 = K / 4;
  const float4* xs4 = reinterpret_cast<const float4*>(S.xs);
  for (int e = cs.warp; e < ph.n_experts; e += NCW) {
    const uint2* wr = reinterpret_cast<const uint2*>(ph.router + (size_t)e * K);
    float acc = 0.0f;
    for (int k4 = cs.lane; k4 < K4; k4 += 32) {
      const float4 xm = xs4[k4], iv = dq_inv(ph.dtype, k4 & 7);
      const float4 x = make_float4(xm.x * iv.x, xm.y * iv.y, xm.z * iv.z, xm.w * iv.w);
      const float4 wv = bf4(wr[k4]);
      acc = fmaf(x.x, wv.x, fmaf(x.y, wv.y, fmaf(x.z, wv.z, fmaf(x.w, wv.w, acc))));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (cs.lane == 0) S.red[32 + e] = acc * cs.rnorm;
  }
  if (!cta_sync(S, cs, P.err)) return false;
  if (cs.ctid == 0) {
    int e1 = 0;
    for (int e = 1; e < ph.n_experts; ++e)
      if (S.red[32 + e] > S.red[32 + e1]) e1 = e;
    int e2 = e1 == 0 ? 1 : 0;
    for (int e = 0; e < ph.n_experts; ++e)
      if (e != e1 && S.red[32 + e] > S.red[32 + e2]) e2 = e;
    const float b = expf(S.red[32 + e2] - S.red[32 + e1]);  // r2 <= r1
    S.red[40] = 1.0f / (1.0f + b);
    S.red[41] = b / (1.0f + b);
    S.bcast[32] = e1;
    S.bcast[33] = e2;
    __threadfence_block();
    *reinterpret_cast<volatile int*>(S.bcast + 34) = pi + 1;  // releases the producer
  }
  return cta_sync(S, cs, P.err);
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
    S.bcast[cs.warp] = am.i;
  }
  if (!cta_sync(S, cs, P.err)) return false;
  if (cs.warp == 0) {
    int last = 0;
    if (cs.lane == 0) {
      ArgMax b = {S.red[0], S.bcast[0]};
      for (int w = 1; w < NCW; ++w) amax_merge(b, S.red[w], S.bcast[w]);
      P.amax_val[cta] = b.v;
      P.amax_idx[cta] = b.i;
      __threadfence();
      last = atomicAdd(P.amax_tick, 1u) == (unsigned)(P.nctas - 1);
    }
    if (__shfl_sync(0xffffffffu, last, 0)) {
      // the last CTA merges every CTA's candidate: 32 lanes load in parallel
      __threadfence();
      ArgMax g = {-INFINITY, 0x7fffffff};
      for (int k = cs.lane; k < P.nctas; k += 32) amax_merge(g, __ldcg(P.amax_val + k), __ldcg(P.amax_idx + k));
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float v = __shfl_xor_sync(0xffffffffu, g.v, o);
        const int i = __shfl_xor_sync(0xffffffffu, g.i, o);
        amax_merge(g, v, i);
      }
      if (cs.lane == 0) {
        *P.argmax = g.i;
        *P.amax_tick = 0u;
        if (P.pos_inc) *P.pos_inc = *P.pos_inc + 1;
      }
    }
  }
  return true;
}

// ============================================================== kernel ====
// One instantiation per weight type DT and pass kind: VER, the verification
// pass (multi-row GEMV phases); otherwise the decode step (single-row GEMV,
// fused FFN, split o projection).  Splitting them keeps each kernel's
// register budget to its own code paths and its code small: the code that
// runs once per phase (staging, attention, epilogues) otherwise misses the
// instruction cache every time.
template <int DT, bool VER>
__global__ void __launch_bounds__(NTHREADS, 1) k_engine(const __grid_constant__ Params P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Smem S = smem_layout(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, cta = blockIdx.x;
  if (tid == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], 1);
    }
    mbar_init(S.cbar, NCW * 32);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < NTB) {
    S.tbc[tid] = 0;
    S.tbg[tid] = tid;
  }
  if (tid == 0) S.bcast[34] = 0;
  if (tid < 2 * FFN_HN) S.ffnc[tid] = 0;
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
  if (VER) {
    bool bad = P.M < 1 || P.M > MAX_M || pos + P.M > P.tmax;
    for (int m = 0; m < P.M; ++m) bad |= P.tokens[m] < 0 || P.tokens[m] >= P.vocab;
    if (bad) {
      if (tid == 0) atomicCAS(P.err, 0, ERR_BAD_TOKEN);
      return;
    }
  }

  if (warp >= NCW) {
    if (lane == 0) producer(P, S, cta, pos, warp - NCW);
    return;
  }

  Cons cs;
  cs.it = 0;
  cs.cphase = 0;
  cs.useq = 0;
  cs.warp = warp;
  cs.lane = lane;
  cs.ctid = tid;
  cs.starved = 0;
  cs.rnorm = 1.0f;
  cs.wnorm = false;
  cs.lim = wait_limit(P);
  const int G = P.nctas;
  ArgMax am = {-INFINITY, 0x7fffffff};
  ArgMax amv[VER ? MAX_M : 1];
#pragma unroll
  for (int m = 0; m < (VER ? MAX_M : 1); ++m) amv[m] = am;
  bool any_logits = false;

  // The consumers read phase descriptors from shared memory: the copy of
  // phase pi + 1 is requested at the start of phase pi (16 threads, 16 bytes
  // each) and completes before that phase's closing CTA barrier, so its L2
  // latency never sits on a phase's critical path.
  constexpr int PH16 = (int)(sizeof(Phase) / 16);
  if (P.prog) {
    if (tid < PH16) {
      cp_async16(reinterpret_cast<uint4*>(S.phb) + tid, reinterpret_cast<const uint4*>(P.prog) + tid);
      cp_async_wait_all();
    }
    if (!cta_sync(S, cs, P.err)) return;
  }
  for (int pi = 0; pi < P.nphases; ++pi) {
    const Phase& ph = P.prog ? S.phb[pi & 1] : P.single;
    if (P.prog && pi + 1 < P.nphases && tid < PH16)
      cp_async16(reinterpret_cast<uint4*>(S.phb + ((pi + 1) & 1)) + tid,
                 reinterpret_cast<const uint4*>(P.prog + pi + 1) + tid);
    unsigned long long* tr = (P.trace && tid == 0) ? P.trace + ((size_t)pi * G + cta) * TRACE_W : nullptr;
    if (tr) tr[0] = gtimer();
    if (ph.wait_bar >= 0) {
      int ok = 1;
      if (tid == 0) ok = counter_wait(P.bars + ph.wait_bar, (unsigned)G, P.err, ERR_WAIT_GRID, cs.lim);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return;
      if (!cta_sync(S, cs, P.err)) return;
    }
    if (tr) tr[1] = gtimer();
    if (ph.kind == PH_GEMV) {
      bool ok;
      if (ph.dtype != DT) {
        if (tid == 0) atomicCAS(P.err, 0, ERR_BAD_PROGRAM);
        return;
      }
      if (VER) {
        if (tr) tr[2] = gtimer();
        ok = gemv_phase_m<DT>(ph, P, S, cs, cta, pos, pi, amv);
      } else {
        if (warp_stageable(ph)) stage_x_warp(ph, P, S, cs, cta);
        else if (!stage_x(ph, P, S, cs, cta)) return;
        if (ph.moe == MOE_GU && !route_experts(ph, P, S, cs, pi)) return;
        if (tr) tr[2] = gtimer();
        ok = gemv_phase<DT>(ph, P, S, cs, cta, pos, am);
      }
      if (!ok) return;
      if (ph.epi == EPI_LOGITS) any_logits = true;
    } else if (ph.kind == PH_OSPLIT && !VER && ph.dtype == DT) {
      if (tr) tr[2] = tr[1];
      if (!osplit_phase<DT>(ph, P, S, cs, cta)) return;
    } else if (ph.kind == PH_FFN && !VER && ph.dtype == DT) {
      if (warp_stageable(ph)) stage_x_warp(ph, P, S, cs, cta);
      else if (!stage_x(ph, P, S, cs, cta)) return;
      if (tr) tr[2] = gtimer();
      if (!ffn_phase<DT>(ph, P, S, cs, cta, pos)) return;
    } else if (ph.kind == PH_ATTN) {
      if (tr) tr[2] = tr[1];
      const int nunits = attn_units(ph, P, pos, -1, nullptr);
      uint32_t j = 0;
      for (int u = first_unit(cta, ph.rot, G); u < nunits; u += G) {
        AttnUnit au;
        attn_units(ph, P, pos, u, &au);
        const int gq = ph.Hq / ph.Hkv;
        const AttnRet r =
            ph.hd == 128 ? (gq == 1   ? attn_call<128, 1, VER>(ph, P, S, cs, au, pos, j)
                            : gq == 2 ? attn_call<128, 2, VER>(ph, P, S, cs, au, pos, j)
                                      : attn_call<128, MAX_GQ, VER>(ph, P, S, cs, au, pos, j))
                         : (gq == 1   ? attn_call<64, 1, VER>(ph, P, S, cs, au, pos, j)
                            : gq == 2 ? attn_call<64, 2, VER>(ph, P, S, cs, au, pos, j)
                                      : attn_call<64, MAX_GQ, VER>(ph, P, S, cs, au, pos, j));
        j = r.j;
        cs.cphase = r.cphase;
        cs.starved = r.starved;
        if (!r.ok) return;
      }
      cs.it += j;
    } else {
      if (tid == 0) atomicCAS(P.err, 0, ERR_BAD_PROGRAM);
      return;
    }
    if (tr) {
      tr[3] = gtimer();
      tr[6] = cs.starved;
    }
    cs.starved = 0;
    if (tid < PH16) cp_async_wait_all();  // the next phase's descriptor has landed
    // Past the barrier below, lanes of warp 0 may start the next phase and
    // overwrite this descriptor's buffer with the one after it: what is read
    // of it later is read before the barrier.
    const int sbar = ph.signal_bar;
    // every warp of this CTA has finished the phase (its global writes made)
    if (!cta_sync(S, cs, P.err)) return;
    if (sbar >= 0 && tid == 0) grid_arrive(P.bars + sbar);
    if (tr) tr[4] = gtimer();
  }
  if (any_logits) {
    if (VER) verify_finish(P, S, cs, cta, amv);
    else argmax_finish(P, S, cs, cta, am);
  }
}

// The kernel instantiation of a launch: weight type p.dtype, decode or verify.
static const void* engine_fn(int dt, bool ver) {
  static const void* fns[3][2] = {{(const void*)k_engine<DT_BF16, false>, (const void*)k_engine<DT_BF16, true>},
                                  {(const void*)k_engine<DT_INT8, false>, (const void*)k_engine<DT_INT8, true>},
                                  {(const void*)k_engine<DT_INT4, false>, (const void*)k_engine<DT_INT4, true>}};
  return fns[dt][ver];
}

int launch_engine(const Params& p, int grid, bool cooperative, cudaStream_t s) {
  static bool attr_set[64][3][2] = {};
  int dev = 0;
  GF_CUDA(cudaGetDevice(&dev));
  const bool ver = verifying(p);
  if (p.dtype < 0 || p.dtype > 2) {
    set_error("engine launch: bad weight type %d", p.dtype);
    return GF_EINVAL;
  }
  const void* fn = engine_fn(p.dtype, ver);
  if (dev >= 0 && dev < 64 && !attr_set[dev][p.dtype][ver]) {
    GF_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    attr_set[dev][p.dtype][ver] = true;
  }
  void* args[] = {const_cast<Params*>(&p)};
  if (cooperative) GF_CUDA(cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(NTHREADS), args, SMEM_BYTES, s));
  else GF_CUDA(cudaLaunchKernel(fn, dim3(grid), dim3(NTHREADS), args, SMEM_BYTES, s));
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

static int gemv_common(const char* fn, int dt, const void* x, const void* Wp, const void* s8, int N, int K, int G,
                       void* y, int ydt, cudaStream_t stream, const unsigned* gate = nullptr,
                       unsigned long long wait_ns = 0) {
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
  p.dtype = dt;
  Phase& ph = p.single;
  ph.kind = PH_GEMV;
  ph.dtype = dt;
  ph.N = N;
  ph.K = K;
  ph.G = G;
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
  if (gate) {  // every CTA first waits for the gate word to reach the CTA count
    ph.wait_bar = 0;
    p.bars = const_cast<unsigned*>(gate);
    p.wait_ns = wait_ns;
  }
  return launch_engine(p, grid, false, stream);
}

}  // namespace gf

using namespace gf;

extern "C" {

int gf_gemv_bf16(const void* x, const void* Wpacked, int N, int K, void* y, int ydtype, gf_stream stream) {
  return gemv_common("gf_gemv_bf16", DT_BF16, x, Wpacked, nullptr, N, K, 32, y, ydtype, (cudaStream_t)stream);
}
int gf_gemv_w8(const void* x, const void* qpacked, const void* s, int N, int K, void* y, int ydtype, gf_stream stream) {
  return gemv_common("gf_gemv_w8", DT_INT8, x, qpacked, s, N, K, 32, y, ydtype, (cudaStream_t)stream);
}
int gf_gemv_w4g(const void* x, const void* qpacked, int N, int K, int G, void* y, int ydtype, gf_stream stream) {
  if ((G != 32 && G != 64 && G != 128) || K % G) {
    set_error("gf_gemv_w4g: group size must be 32, 64 or 128 and divide K (G=%d, K=%d)", G, K);
    return GF_EUNSUPPORTED;
  }
  return gemv_common("gf_gemv_w4g", DT_INT4, x, qpacked, nullptr, N, K, G, y, ydtype, (cudaStream_t)stream);
}

int gf_gemv_bf16_gated(const void* x, const void* Wpacked, int N, int K, void* y, int ydtype, const unsigned* d_gate,
                       unsigned long long wait_ns, gf_stream stream) {
  if (!d_gate || ((uintptr_t)d_gate & 3) || wait_ns == 0 || wait_ns > 10000000000ull) {
    set_error("gf_gemv_bf16_gated: need a 4-byte aligned gate word and 0 < wait_ns <= 1e10");
    return GF_EINVAL;
  }
  return gemv_common("gf_gemv_bf16_gated", DT_BF16, x, Wpacked, nullptr, N, K, 32, y, ydtype, (cudaStream_t)stream,
                     d_gate, wait_ns);
}

size_t gf_attn_workspace_bytes(int Hq, int Hkv, int hd) {
  if (Hq <= 0 || Hkv <= 0 || hd <= 0) return 0;
  const int sms = device_sms() > 0 ? device_sms() : 1;
  const int nch_max = (sms + Hkv - 1) / Hkv;
  // partials, then one combine ticket per kv head
  return (size_t)Hq * nch_max * (hd + 2) * sizeof(float) + ((size_t)Hkv * sizeof(unsigned) + 255) / 256 * 256;
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
  ph.qbuf = const_cast<void*>(q);
  ph.kc = (uint16_t*)kcache;
  ph.vc = (uint16_t*)vcache;
  ph.attn_out = out;
  ph.Hq = Hq;
  ph.Hkv = Hkv;
  ph.hd = hd;
  ph.Tmax = Tmax;
  ph.stream_cur = 1;
  const int nch_max = (sms + Hkv - 1) / Hkv;
  const size_t part_bytes = (size_t)Hq * nch_max * (hd + 2) * sizeof(float);
  ph.part = (float*)ws;
  ph.tick = (unsigned*)((uint8_t*)ws + part_bytes);
  GF_CUDA(cudaMemsetAsync(ph.tick, 0, Hkv * sizeof(unsigned), (cudaStream_t)stream));
  int CH, nch;
  attn_split(pos + 1, Hkv, sms, CH, nch);
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
