// engine.cu — the persistent phase engine of libgf (sm_103a).
//
// One CTA per SM runs a program of phases (a single GEMV or attention for the
// standalone calls; every layer of a decode step for gf_decode_step).  In
// each CTA one producer thread streams the CTA's weight half-tiles (16 rows x
// one K-block) and KV-cache rows from HBM into a ring of 16 shared-memory
// slots with bulk asynchronous copies (cp.async.bulk, completion counted on
// an mbarrier, L2 evict-first hint), running ahead across phase boundaries
// because the weight stream does not depend on activations.  Each slot
// belongs to one of eight consumer warps (stream index mod 8, so a ring entry
// always serves the same warp), which dequantises the
// int8 / int4 codes of its 16 rows in registers against an fp32 copy of the
// input vector held in shared memory and releases the slot; the K-block
// partial sums of a half-tile meet in shared memory, where the last warp to
// arrive adds them in a fixed order and runs the epilogue.  Dependent phases
// are separated by grid barriers (cooperative launch); every wait in the
// kernel is bounded by a 2-second clock, after which the kernel records an
// error code, drains its own copies in flight and returns.
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
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_plain(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
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

__device__ __noinline__ bool mbar_wait_slow(uint64_t* b, uint32_t parity, int* err, int code) {
  const uint64_t t0 = gtimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_sleep(b, parity)) return true;
    if ((it & 3) == 0) {
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
  float* xs;        // fp32 input vector, swizzled per chunk
  float* xsum;      // sum of x over each 32-wide group (int4 zero offsets)
  float* tb;        // [NTB][NCW][HROWS] partial row sums of half-tiles
  int* tbc;         // [NTB] arrival counters
  int* tbg;         // [NTB] half-tile allowed to use the buffer next
  uint64_t* full;   // [NSLOT]
  uint64_t* empty;  // [NSLOT]
  uint64_t* cbar;   // consumer-warps barrier
  uint64_t* xbar;   // completion of the bulk copy of a phase's input vector
  float* red;       // [64] reduction scratch; [32..39] router logits, [40..41] expert weights
  int* bcast;       // [64] broadcast ints; [32..33] chosen experts, [34] phase they were chosen in,
                    // [48..55] verify: union of the rows' experts, [56] its size
  float* moew;      // [MAX_M][8] verify: weight of expert e for row m (0 if not chosen)
  Phase* phb;       // [2] the consumers' copies of the current and next phase descriptor
};

__device__ __forceinline__ Smem smem_layout(uint8_t* base) {
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
  s.xbar = s.cbar + 1;
  s.red = reinterpret_cast<float*>(base + OFF_MISC);
  s.bcast = reinterpret_cast<int*>(base + OFF_MISC + 256);
  s.moew = reinterpret_cast<float*>(base + OFF_MISC + 512);
  s.phb = reinterpret_cast<Phase*>(base + OFF_PHB);
  return s;
}

__device__ __forceinline__ int first_unit(int cta, int rot, int G) { return ((cta - rot) % G + G) % G; }

__device__ __forceinline__ const Phase& phase_at(const Params& P, int i) { return P.prog ? P.prog[i] : P.single; }

// ============================================================ producer ====
struct Prod {
  uint32_t it;
  uint64_t pol;
  uint32_t blocked;
};

__device__ __forceinline__ bool prod_slot(const Smem& S, Prod& pr, int* err, uint8_t*& dst, uint64_t*& fb) {
  const uint32_t slot = pr.it % NSLOT, use = pr.it / NSLOT;
  if (use > 0) {
    if (!mbar_probe(&S.empty[slot], (use - 1) & 1u)) ++pr.blocked;
    if (!mbar_wait(&S.empty[slot], (use - 1) & 1u, err, ERR_WAIT_EMPTY)) return false;
  }
  dst = S.ring + slot * SLOT_BYTES;
  fb = &S.full[slot];
  ++pr.it;
  return true;
}

// The producer needs the two experts of a MOE_GU phase before it can stream
// their weights: consumer thread 0 publishes them in shared memory, tagged
// with the phase index.  Bounded wait.
__device__ bool wait_experts(const Smem& S, int* err, int pi) {
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
      if (gtimer() - t0 > WAIT_NS) {
        atomicCAS(err, 0, ERR_WAIT_ROUTER);
        return false;
      }
    }
  }
}

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

// Segments of a GEMV phase: the matrices it covers (several experts for MoE).
__device__ __forceinline__ int gemv_segments(const Phase& ph, const Params& P, const Smem& S, int& Ns,
                                             const uint8_t** wseg, int* eseg) {
  volatile int* bc = S.bcast;
  if (ph.moe == MOE_NONE) {
    Ns = ph.N;
    wseg[0] = ph.W;
    eseg[0] = 0;
    return 1;
  }
  if (verifying(P)) {  // verify: the union of the rows' experts
    const int n = bc[56];
    Ns = ph.N;
    for (int k = 0; k < n; ++k) {
      eseg[k] = bc[48 + k];
      wseg[k] = ph.W + (size_t)eseg[k] * ph.expert_stride;
    }
    return n;
  }
  if (ph.moe == MOE_GU) {
    Ns = ph.N / 2;
    for (int k = 0; k < 2; ++k) {
      eseg[k] = bc[32 + k];
      wseg[k] = ph.W + (size_t)eseg[k] * ph.expert_stride;
    }
    return 2;
  }
  Ns = ph.N;
  eseg[0] = bc[32 + ph.moe - MOE_DOWN0];
  wseg[0] = ph.W + (size_t)eseg[0] * ph.expert_stride;
  return 1;
}

// Slot order of a multi-row (verify) GEMV phase: the CTA's tiles in groups of
// up to VTG tiles of one segment; per group, K-block by K-block, the group's
// tiles and their halves.  Consumers walk the same order.
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

__device__ bool wait_experts(const Smem& S, int* err, int pi);

__device__ bool produce_gemv_m(const Phase& ph, const Params& P, const Smem& S, Prod& pr, int cta, int pi) {
  int* err = P.err;
  if (ph.moe == MOE_GU && !wait_experts(S, err, pi)) return false;
  const int dt = ph.dtype, C = ph.K / per_chunk(dt), nb = (C + KBLK - 1) / KBLK;
  int Ns;
  const uint8_t* wseg[8];
  int eseg[8];
  const int nseg = gemv_segments(ph, P, S, Ns, wseg, eseg);
  TileGroups tg;
  tg.tps = (Ns + TR - 1) / TR;
  tg.ntiles = nseg * tg.tps;
  tg.G = P.nctas;
  tg.first = first_unit(cta, ph.rot, P.nctas);
  for (int i0 = 0; tg.first + i0 * tg.G < tg.ntiles;) {
    const int i1 = group_end(tg, i0);
    for (int b = 0; b < nb; ++b) {
      const int Lb = min(KBLK, C - b * KBLK);
      for (int i = i0; i < i1; ++i) {
        const int t = tg.first + i * tg.G, seg = t / tg.tps, lt = t % tg.tps;
        const int Rt = min(TR, Ns - lt * TR);
        for (int h = 0; h * HROWS < Rt; ++h) {
          const int r0 = h * HROWS, rh = min(HROWS, Rt - r0);
          const uint8_t* blk = wseg[seg] + block_offset(dt, C, lt, Rt, b);
          const uint32_t cb = (uint32_t)(rh * Lb * 16);
          const uint32_t sb = dt == DT_INT4 ? (uint32_t)((rh * Lb * 4 + 15) / 16 * 16) : 0u;
          uint8_t* dst;
          uint64_t* fb;
          if (!prod_slot(S, pr, err, dst, fb)) return false;
          mbar_expect_tx(fb, cb + sb);
          bulk_g2s(dst, blk + (size_t)r0 * Lb * 16, cb, fb, pr.pol);
          if (sb) bulk_g2s(dst + SLOT_SZ_OFF, blk + (size_t)Rt * Lb * 16 + (size_t)r0 * Lb * 4, sb, fb, pr.pol);
        }
      }
    }
    i0 = i1;
  }
  return true;
}

// Slot order of a GEMV phase (producer and consumers walk it identically):
// for each of the CTA's tiles t, for each half h of the tile's rows, the
// K-blocks b in order.
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
    if (ph.kind == PH_GEMV && verifying(P)) {
      ok = produce_gemv_m(ph, P, S, pr, cta, pi);
    } else if (ph.kind == PH_GEMV) {
      const int dt = ph.dtype, C = ph.K / per_chunk(dt);
      // a phase covers nseg matrices of Ns rows each (two experts for MOE_GU)
      const int nseg = ph.moe == MOE_GU ? 2 : 1, Ns = ph.N / nseg;
      const int tps = (Ns + TR - 1) / TR, ntiles = nseg * tps, nb = (C + KBLK - 1) / KBLK;
      const uint8_t* wseg[2] = {ph.W, ph.W};
      if (ph.moe != MOE_NONE) {
        if (ph.moe == MOE_GU && !(ok = wait_experts(S, err, pi))) break;
        volatile int* sel = S.bcast + 32;
        if (ph.moe == MOE_GU) {
          wseg[0] = ph.W + (size_t)sel[0] * ph.expert_stride;
          wseg[1] = ph.W + (size_t)sel[1] * ph.expert_stride;
        } else {
          wseg[0] = ph.W + (size_t)sel[ph.moe - MOE_DOWN0] * ph.expert_stride;
        }
      }
      for (int t = first_unit(cta, ph.rot, G); t < ntiles && ok; t += G) {
        const int seg = t / tps, lt = t % tps;
        const int Rt = min(TR, Ns - lt * TR);
        for (int h = 0; h * HROWS < Rt && ok; ++h) {
          const int r0 = h * HROWS, rh = min(HROWS, Rt - r0);
          for (int b = 0; b < nb; ++b) {
            const int Lb = min(KBLK, C - b * KBLK);
            const uint8_t* blk = wseg[seg] + block_offset(dt, C, lt, Rt, b);
            const uint32_t cb = (uint32_t)(rh * Lb * 16);
            const uint32_t sb = dt == DT_INT4 ? (uint32_t)((rh * Lb * 4 + 15) / 16 * 16) : 0u;
            uint8_t* dst;
            uint64_t* fb;
            if (!(ok = prod_slot(S, pr, err, dst, fb))) break;
            mbar_expect_tx(fb, cb + sb);
            bulk_g2s(dst, blk + (size_t)r0 * Lb * 16, cb, fb, pr.pol);
            if (sb) bulk_g2s(dst + SLOT_SZ_OFF, blk + (size_t)Rt * Lb * 16 + (size_t)r0 * Lb * 4, sb, fb, pr.pol);
          }
        }
      }
    } else if (ph.kind == PH_FFN) {
      // per gate/up tile: its two half-tiles' K-blocks, then the rows of the
      // matching 16-column slice of the down projection
      const int dt = ph.dtype, C = ph.K / per_chunk(dt), nb = (C + KBLK - 1) / KBLK;
      const int tps = ph.N / TR, d = ph.N2;
      int nsl, DR;
      ffn_split(dt, d, nsl, DR);
      // an empty slot: completed by the arrival alone
      auto empty_slot = [&]() {
        uint8_t* dst;
        uint64_t* fb;
        if ((ok = prod_slot(S, pr, err, dst, fb))) mbar_arrive(fb);
      };
      // the down slice of a tile follows the next tile's gate/up blocks, so
      // that its SwiGLU outputs are ready when its rows arrive
      auto down_slice = [&](int t) {
        for (int k = 0; k < nsl && ok; ++k) {
          const int r0 = k * DR, nr = min(DR, d - r0);
          if (nr <= 0) {
            empty_slot();
            continue;
          }
          const uint8_t* src;
          const uint8_t* szs = nullptr;
          uint32_t cb;
          if (dt == DT_INT4) {
            const uint8_t* g = ph.W2 + (size_t)(t >> 1) * d * 20;
            src = g + (size_t)(t & 1) * d * 8 + (size_t)r0 * 8;
            szs = g + (size_t)d * 16 + (size_t)r0 * 4;
            cb = (uint32_t)nr * 8;
          } else {
            const int rb = dt == DT_INT8 ? 16 : 32;
            src = ph.W2 + ((size_t)t * d + r0) * rb;
            cb = (uint32_t)(nr * rb);
          }
          uint8_t* dst;
          uint64_t* fb;
          if (!(ok = prod_slot(S, pr, err, dst, fb))) break;
          mbar_expect_tx(fb, cb + (szs ? (uint32_t)nr * 4 : 0u));
          bulk_g2s(dst, src, cb, fb, pr.pol);
          if (szs) bulk_g2s(dst + (size_t)DR * 8, szs, (uint32_t)nr * 4, fb, pr.pol);
        }
      };
      int prev = -1;
      for (int t = first_unit(cta, ph.rot, G); t < tps && ok; t += G) {
        for (int h = 0; h < 2 && ok; ++h) {
          for (int b = 0; b < nb && ok; ++b) {
            const int Lb = min(KBLK, C - b * KBLK);
            const uint8_t* blk = ph.W + block_offset(dt, C, t, TR, b);
            const uint32_t cb = (uint32_t)(HROWS * Lb * 16);
            const uint32_t sb = dt == DT_INT4 ? (uint32_t)(HROWS * Lb * 4) : 0u;
            uint8_t* dst;
            uint64_t* fb;
            if (!(ok = prod_slot(S, pr, err, dst, fb))) break;
            mbar_expect_tx(fb, cb + sb);
            bulk_g2s(dst, blk + (size_t)h * HROWS * Lb * 16, cb, fb, pr.pol);
            if (sb) bulk_g2s(dst + SLOT_SZ_OFF, blk + (size_t)TR * Lb * 16 + (size_t)h * HROWS * Lb * 4, sb, fb, pr.pol);
          }
        }
        if (prev >= 0) down_slice(prev);
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
        for (int p = p0; p < pe; p += ATT_POS_PER_SLOT) {
          const int np = min(ATT_POS_PER_SLOT, pe - p);
          uint8_t* dst;
          uint64_t* fb;
          if (!(ok = prod_slot(S, pr, err, dst, fb))) break;
          const size_t off = ((size_t)hh * ph.Tmax + p) * ph.hd;
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
    while (!mbar_test_sleep(&S.full[slot], use & 1u)) {
      if (gtimer() - t0 > WAIT_NS) {
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
  uint32_t useq;     // half-tiles seen so far (combine-buffer index)
  int warp, lane, ctid;
  uint32_t starved;  // slot waits that found the slot still in flight (warp 0)
  float rnorm;       // RMSNorm factor of the staged input (1 if none)
  uint32_t xphase;   // parity of the input-copy barrier
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

// Every lane waits on the slot's barrier itself (each lane's completed wait
// orders its reads of the slot after the copy).
__device__ __forceinline__ bool slot_acquire(const Smem& S, Cons& cs, uint32_t it, int* err, const uint8_t*& base) {
  const uint32_t slot = it % NSLOT, par = (it / NSLOT) & 1u;
  if (cs.warp == 0 && cs.lane == 0 && !mbar_probe(&S.full[slot], par)) ++cs.starved;
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&S.full[slot], par, err, ERR_WAIT_FULL));
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
__device__ __forceinline__ int swz(int g, int U) { return ((g * U) >> 3) & (U - 1); }

__device__ __forceinline__ float4 bf4(uint2 h) {
  return make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xFFFF0000u), __uint_as_float(h.y << 16),
                     __uint_as_float(h.y & 0xFFFF0000u));
}

// Stores float4 number k4 of x (swizzled per chunk so that the 32 lanes of a
// warp read their chunks without bank conflicts), multiplied by the powers of
// two that the subnormal dequantisation of int4 / int8 codes expects, and the
// chunk sums the epilogues need: for int4 the sum of x over each 32-wide group
// (8 consecutive threads hold one group), for int8 128 times the sum over each
// 16-wide chunk (4 threads), both times 2^-64.
__device__ __forceinline__ void stage_store(const Smem& S, const Cons& cs, int dt, int U, int k4, bool ok, float4 a) {
  const int g = k4 / U, u = k4 % U;
  const float4 m = dq_mult(dt, u);
  if (ok)
    reinterpret_cast<float4*>(S.xs)[g * U + (u ^ swz(g, U))] = make_float4(a.x * m.x, a.y * m.y, a.z * m.z, a.w * m.w);
  if (dt != DT_BF16) {
    float sg = a.x + a.y + a.z + a.w;
    sg += __shfl_xor_sync(0xffffffffu, sg, 1);
    sg += __shfl_xor_sync(0xffffffffu, sg, 2);
    if (dt == DT_INT4) sg += __shfl_xor_sync(0xffffffffu, sg, 4);
    if (ok && (cs.lane & (U - 1)) == 0) S.xsum[g] = sg * (dt == DT_INT4 ? DQ_DOWN : 128.0f * DQ_DOWN);
  }
}

// Stages the phase's input vector into shared memory as fp32.  Thread t
// handles float4 numbers t + 224 i; all of its loads are issued before any is
// used, so staging costs about one L2 round trip.  For an RMSNorm input only
// the gain is applied here: the factor 1/rms needs the whole vector, and as
// the GEMV is linear it is applied to the outputs in the epilogue instead
// (cs.rnorm, 1 for other inputs), which keeps the reduction off the path.
__device__ bool stage_x_regs(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta) {
  constexpr int NT = NCW * 32, MAXIT = (KMAX / 4 + NT - 1) / NT;
  const int K = ph.K, dt = ph.dtype, U = per_chunk(dt) / 4, K4 = K / 4;
  const bool norm = ph.xsrc == X_NORM || ph.xsrc == X_EMBED_NORM;
  const uint16_t* emb = ph.xsrc == X_EMBED_NORM ? P.embed + (size_t)(*P.token) * K : nullptr;
  float4 a[MAXIT];
  uint2 gk[MAXIT];
  // one load loop per source, each load writing its own register, so that
  // nothing waits for a load before the next is issued
#pragma unroll
  for (int t = 0; t < MAXIT; ++t) {
    const int k4 = cs.ctid + t * NT;
    gk[t] = make_uint2(0x3F803F80u, 0x3F803F80u);  // bf16 ones
    if (norm && k4 < K4) gk[t] = reinterpret_cast<const uint2*>(ph.gain)[k4];
  }
  if (ph.xsrc == X_F32 || ph.xsrc == X_NORM) {
    const float4* src = reinterpret_cast<const float4*>(ph.xptr);
#pragma unroll
    for (int t = 0; t < MAXIT; ++t) {
      const int k4 = cs.ctid + t * NT;
      a[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k4 < K4) a[t] = __ldcg(src + k4);
    }
  } else {
    const uint2* src = emb ? reinterpret_cast<const uint2*>(emb) : reinterpret_cast<const uint2*>(ph.xptr);
    uint2 h[MAXIT];
#pragma unroll
    for (int t = 0; t < MAXIT; ++t) {
      const int k4 = cs.ctid + t * NT;
      h[t] = make_uint2(0u, 0u);
      if (k4 < K4) h[t] = __ldcg(src + k4);
    }
#pragma unroll
    for (int t = 0; t < MAXIT; ++t) a[t] = bf4(h[t]);
  }
  // keep every load above the shared-memory stores below (the compiler
  // cannot tell that they do not alias), so that all are in flight at once
  asm volatile("" ::: "memory");
  float ss = 0.0f;
#pragma unroll
  for (int t = 0; t < MAXIT; ++t) {
    const int k4 = cs.ctid + t * NT;
    if (t * NT < K4) {  // warp-uniform: the chunk sums shuffle within the warp
      if (norm) {
        ss += a[t].x * a[t].x + a[t].y * a[t].y + a[t].z * a[t].z + a[t].w * a[t].w;
        if (emb && cta == 0 && k4 < K4) reinterpret_cast<float4*>(P.resid)[k4] = a[t];
        const float4 g = bf4(gk[t]);
        a[t] = make_float4(a[t].x * g.x, a[t].y * g.y, a[t].z * g.z, a[t].w * g.w);
      }
      stage_store(S, cs, dt, U, k4, k4 < K4, a[t]);
    }
  }
  if (norm) {
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (cs.lane == 0) S.red[cs.warp] = ss;
  }
  if (!cta_sync(S, cs, P.err)) return false;
  cs.rnorm = 1.0f;
  if (norm) {
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) tot += S.red[w];
    cs.rnorm = 1.0f / sqrtf(tot / (float)K + ph.eps);
  }
  return true;
}

// Stages an fp32 input vector (X_F32, or X_NORM with its bf16 gain) with
// per-thread asynchronous copies into the x area (the gain into the top of
// that area), then converts it in place with a short loop: gain, 1/rms
// partial sums, the dequantisation multipliers, the per-chunk swizzle and the
// chunk sums.  Warp w copies and converts the runs of 32 float4 starting at
// 32 w + 224 i (whole chunks): its lanes' copies are complete and visible to
// the warp after wait_all and __syncwarp, and all lanes load a run before any
// lane stores into it, so the in-place permutation inside a chunk is safe.
// The copies use the load/store path, not the bulk-copy engine, whose queue
// holds the producer's weight prefetches.  Other inputs (bf16 vectors, the
// embedding row) go through stage_x_regs.
__device__ bool stage_x(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta) {
  const int K = ph.K, dt = ph.dtype, U = per_chunk(dt) / 4, K4 = K / 4;
  const bool norm = ph.xsrc == X_NORM;
  const bool fast = (ph.xsrc == X_F32 || norm) && (!norm || (K * 6 <= KMAX * 4 && ((uintptr_t)ph.gain & 7) == 0)) &&
                    ((uintptr_t)ph.xptr & 15) == 0;
  if (!fast) return stage_x_regs(ph, P, S, cs, cta);
  float4* xs4 = reinterpret_cast<float4*>(S.xs);
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
  float ss = 0.0f;
#pragma unroll 1
  for (int base = cs.warp * 32; base < K4; base += NCW * 32) {  // warp-uniform trip count
    const int f = base + cs.lane;
    const bool in = f < K4;
    float4 a = in ? xs4[f] : make_float4(0.f, 0.f, 0.f, 0.f);
    if (norm) {
      ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
      const float4 g = bf4(in ? gs[f] : make_uint2(0u, 0u));
      a = make_float4(a.x * g.x, a.y * g.y, a.z * g.z, a.w * g.w);
    }
    __syncwarp();  // every lane has read the run before any lane overwrites it
    stage_store(S, cs, dt, U, f, in, a);
  }
  if (norm) {
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (cs.lane == 0) S.red[cs.warp] = ss;
  }
  if (!cta_sync(S, cs, P.err)) return false;
  cs.rnorm = 1.0f;
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

// One 32-bit word of codes of one row against its staged inputs x (natural
// k order, as pairs), accumulated into acc.
// int4: the word holds 8 consecutive codes in nibbles 0..7.
__device__ __forceinline__ float2 word_int4(const uint32_t w, const float2* x, float2 acc) {
  const uint32_t h = w >> 8;
  acc = ffma2(bits2(w & 0x0000000Fu, w & 0x000000F0u), x[0], acc);
  acc = ffma2(bits2(w & 0x00000F00u, w & 0x0000F000u), x[1], acc);
  acc = ffma2(bits2(w & 0x000F0000u, w & 0x00F00000u), x[2], acc);
  acc = ffma2(bits2(h & 0x000F0000u, h & 0x00F00000u), x[3], acc);
  return acc;
}
// int8: 4 consecutive codes, one byte each, stored as the offset code c + 128.
__device__ __forceinline__ float2 word_int8(const uint32_t wq, const float2* x, float2 acc) {
  const uint32_t w = wq, h = w >> 8;
  acc = ffma2(bits2(w & 0x000000FFu, w & 0x0000FF00u), x[0], acc);
  acc = ffma2(bits2(w & 0x00FF0000u, h & 0x00FF0000u), x[1], acc);
  return acc;
}
// bf16: 2 consecutive weights (low half first).
__device__ __forceinline__ float2 word_bf16(const uint32_t w, const float2* x, float2 acc) {
  return ffma2(bits2(w << 16, w & 0xFFFF0000u), x[0], acc);
}

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

// Epilogue of one output row n (value y); lanes 0..15 call it together, each
// with its own row of the half-tile; yp is the value of row n ^ 1.
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

// The work of one lane on one slot of Lb chunks per row: its chunk (number g
// of the row) of every row of the slot.  One copy of this code serves every
// slot width, which keeps the engine's hot code small.
template <int DT>
__device__ __forceinline__ void slot_rows(const uint8_t* base, int Lb, int lane, int g, const float4* xs4, const Smem& S,
                                          float* v, float2* acc, float& bias) {
  constexpr int E = DT == DT_BF16 ? 8 : DT == DT_INT8 ? 16 : 32;
  constexpr int U = E / 4;
  const int L = Lb;
  // The four words of the chunk go by in a run-time loop (a small loop body
  // stays in the instruction cache); in step jw lane l reads word
  // (jw + l / 8) % 4, so that the 32 lanes' 4-byte loads hit 32 banks.
  const int sw = swz(g, U);
  const uint32_t* wrow = reinterpret_cast<const uint32_t*>(base) + lane * 4;
  float2 a[HROWS];  // int4: this chunk's sums; int8 / bf16: running sums
#pragma unroll
  for (int r = 0; r < HROWS; ++r) a[r] = DT == DT_INT4 ? make_float2(0.f, 0.f) : acc[r];
#pragma unroll 1
  for (int jw = 0; jw < 4; ++jw) {
    const int ws = (jw + (lane >> 3)) & 3;
    float2 xr[4];
    if (DT == DT_INT4) {
      const float4 xa = xs4[g * U + ((2 * ws) ^ sw)], xb = xs4[g * U + ((2 * ws + 1) ^ sw)];
      xr[0] = make_float2(xa.x, xa.y);
      xr[1] = make_float2(xa.z, xa.w);
      xr[2] = make_float2(xb.x, xb.y);
      xr[3] = make_float2(xb.z, xb.w);
    } else if (DT == DT_INT8) {
      const float4 xa = xs4[g * U + (ws ^ sw)];
      xr[0] = make_float2(xa.x, xa.y);
      xr[1] = make_float2(xa.z, xa.w);
    } else {
      const float4 xa = xs4[g * U + ((ws >> 1) ^ sw)];
      xr[0] = (ws & 1) ? make_float2(xa.z, xa.w) : make_float2(xa.x, xa.y);
    }
#pragma unroll
    for (int r = 0; r < HROWS; ++r) {
      const uint32_t wv = wrow[r * L * 4 + ws];
      if (DT == DT_INT4) a[r] = word_int4(wv, xr, a[r]);
      else if (DT == DT_INT8) a[r] = word_int8(wv, xr, a[r]);
      else a[r] = word_bf16(wv, xr, a[r]);
    }
  }
  if (DT == DT_INT4) {
    const float xg = S.xsum[g];
    const uint32_t* szp = reinterpret_cast<const uint32_t*>(base + SLOT_SZ_OFF) + lane;
#pragma unroll
    for (int r = 0; r < HROWS; ++r) {
      const uint32_t sz = szp[r * L];
      v[r] = fmaf(__uint_as_float(sz << 16), a[r].x + a[r].y, fmaf(__uint_as_float(sz & 0xFFFF0000u), xg, v[r]));
    }
  } else {
    if (DT == DT_INT8) bias += S.xsum[g];
#pragma unroll
    for (int r = 0; r < HROWS; ++r) acc[r] = a[r];
  }
}

// Waits until combine buffer buf may take half-tile cs.useq (the last
// combiner of half-tile useq - NTB hands it on).  Bounded.
__device__ __forceinline__ bool tb_claim(const Smem& S, const Cons& cs, int buf, int* err) {
  int ok = 1;
  if (cs.lane == 0) {
    volatile int* g = S.tbg + buf;
    if (*g != (int)cs.useq) {
      const uint64_t t0 = gtimer();
      while (*g != (int)cs.useq) {
        __nanosleep(32);
        if (gtimer() - t0 > WAIT_NS) {
          atomicCAS(err, 0, ERR_WAIT_COMBINE);
          ok = 0;
          break;
        }
      }
    }
    __threadfence_block();
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// One GEMV phase for this CTA.  Slot X of the stream (in producer order)
// belongs to warp X % NCW.  A warp accumulates its K-blocks of a half-tile in
// registers (16 rows per lane), reduces them over the lanes, and deposits the
// 16 row sums in the half-tile's combine buffer; the last contributing warp
// adds the deposits in warp order and runs the epilogue.
// One half-tile (16 rows r0.. of tile lt of segment seg; its nb K-blocks are
// the CTA's local slots j0 ..) for the calling warp: its K-blocks, the lane
// reduction, the deposit, and for the last contributing warp the combine.
// Returns -1 if a wait gave up, 1 for the combining warp (lanes r < 16 hold
// in tot the row sum of row r0 + r, already multiplied by the row's output
// factor, and in rp its RoPE pair), else 0.
template <int DT>
__device__ __forceinline__ int gemv_half(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int seg, int lt,
                                         int r0, int Rt, uint32_t j0, int pos, float& tot, float2& rp) {
  constexpr int E = DT == DT_BF16 ? 8 : DT == DT_INT8 ? 16 : 32;
  const int C = ph.K / E, nb = (C + KBLK - 1) / KBLK;
  const int nseg = ph.moe == MOE_GU ? 2 : 1, Ns = ph.N / nseg;
  const int lane = cs.lane, w = cs.warp;
  const int own0 = (int)((cs.it + j0) % NCW);  // owner of K-block 0
  const int bfirst = (w - own0 + NCW) % NCW;   // this warp's first K-block
  const int ncontrib = nb < NCW ? nb : NCW;
  if (bfirst >= nb) return 0;
  const float4* xs4 = reinterpret_cast<const float4*>(S.xs);
  // int8 row scales of the segment's matrix (the chosen expert's, for MoE)
  const uint16_t* s8 = ph.s8;
  if (DT == DT_INT8 && ph.moe != MOE_NONE)
    s8 += (size_t)S.bcast[32 + (ph.moe == MOE_GU ? seg : ph.moe - MOE_DOWN0)] * Ns;
  // the epilogue's own inputs, fetched now so that their latency is hidden
  // behind the K-blocks: lane r < 16 for row r0 + r
  float pf = cs.rnorm * (DT == DT_BF16 ? 1.0f : DQ_UP);  // RMSNorm, 2^64, int8 row scale
  rp = make_float2(1.f, 0.f);
  {
    const int n = lt * TR + r0 + lane;
    if (lane < HROWS && r0 + lane < Rt) {
      if (DT == DT_INT8) pf *= bf2f(s8[n]);
      if (ph.epi == EPI_QKV && n < ph.q_rows + ph.kv_rows) {
        const int nn = n < ph.q_rows ? n : n - ph.q_rows;
        rp = P.rope[(size_t)pos * (ph.hd / 2) + (nn % ph.hd) / 2];
      }
    }
  }
  // int4: v[r] collects s * (codes . x) + z * (sum of x) per group, x 2^-64;
  // int8 / bf16: acc[r] collects the row's dot product over the blocks
  float v[HROWS];
  float2 acc[HROWS];
#pragma unroll
  for (int r = 0; r < HROWS; ++r) {
    v[r] = 0.0f;
    acc[r] = make_float2(0.f, 0.f);
  }
  float bias = 0.0f;  // int8: 128 * sum x * 2^-64 over this lane's chunks
  for (int b = bfirst; b < nb; b += NCW) {
    const uint32_t it = cs.it + j0 + (uint32_t)b;
    const uint8_t* base;
    if (!slot_acquire(S, cs, it, P.err, base)) return -1;
    const int Lb = min(KBLK, C - b * KBLK);
    // lane l takes chunk l of every row of the slot (rows past the tile read
    // in-bounds stale bytes of the slot and are discarded)
    if (lane < Lb) slot_rows<DT>(base, Lb, lane, b * KBLK + lane, xs4, S, v, acc, bias);
    slot_release(S, cs, it);
  }
  if (DT != DT_INT4) {
#pragma unroll
    for (int r = 0; r < HROWS; ++r) v[r] = (acc[r].x + acc[r].y) - bias;
  }
  // deposit this warp's 16 row sums, then the last contributor combines
  const float y = warp_rows16(v, lane);
  const int buf = (int)(cs.useq % NTB);
  float* tb = S.tb + (size_t)buf * NCW * HROWS;
  // the buffer's previous half-tile has been combined (bounded wait; in
  // practice it was long ago)
  if (!tb_claim(S, cs, buf, P.err)) return -1;
  if ((lane & 1) == 0) tb[w * HROWS + (lane >> 1)] = y;
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
  if (lane < HROWS) {
    for (int ww = 0; ww < NCW; ++ww) {
      const int bw = (ww - own0 + NCW) % NCW;
      if (bw < nb) t += tb[ww * HROWS + lane];
    }
  }
  __syncwarp();
  if (lane == 0) {
    S.tbc[buf] = 0;
    __threadfence_block();
    *reinterpret_cast<volatile int*>(S.tbg + buf) = (int)(cs.useq + NTB);  // hand the buffer on
  }
  tot = t * pf;
  return 1;
}

// One GEMV phase for this CTA: its tiles (round-robin over the CTAs), two
// half-tiles each; the combining warp of a half-tile runs the epilogue.
template <int DT>
__device__ bool gemv_phase(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta, int pos, ArgMax& am) {
  constexpr int E = DT == DT_BF16 ? 8 : DT == DT_INT8 ? 16 : 32;
  const int G = P.nctas;
  const int C = ph.K / E, nb = (C + KBLK - 1) / KBLK;
  const int nseg = ph.moe == MOE_GU ? 2 : 1, Ns = ph.N / nseg;
  const int tps = (Ns + TR - 1) / TR, ntiles = nseg * tps;
  const int lane = cs.lane;
  uint32_t j = 0;  // slot index within the phase
  for (int t = first_unit(cta, ph.rot, G); t < ntiles; t += G) {
    const int seg = t / tps, lt = t % tps;
    const int Rt = min(TR, Ns - lt * TR);
    for (int h = 0; h * HROWS < Rt; ++h, ++cs.useq, j += (uint32_t)nb) {
      float tot;
      float2 rp;
      const int k = gemv_half<DT>(ph, P, S, cs, seg, lt, h * HROWS, Rt, j, pos, tot, rp);
      if (k < 0) return false;
      if (k == 0) continue;
      const int r = h * HROWS + lane, n = lt * TR + r;
      const float yp = __shfl_xor_sync(0xffffffffu, tot, 1);
      if (lane < HROWS && r < Rt) gemv_epilogue(ph, P, S, seg, n, tot, yp, pos, rp, am);
    }
  }
  cs.it += j;
  return true;
}

// One row of a down slot (DR rows of 16 columns: the SwiGLU outputs of one
// gate/up tile) against those outputs, staged as the subnormal
// dequantisation reads them (xr; xz: their sum for the int4 zeros, or 128
// times it for the int8 offset), without the 2^64 and int8 row scale that the
// phase end applies.
template <int DT>
__device__ __forceinline__ float down_row(const uint8_t* base, int rl, int DR, const float2* xr, float xz) {
  if (DT == DT_INT4) {
    const uint2 q = reinterpret_cast<const uint2*>(base)[rl];
    const uint32_t sz = reinterpret_cast<const uint32_t*>(base + (size_t)DR * 8)[rl];
    const float2 a0 = word_int4(q.x, xr, make_float2(0.f, 0.f));
    const float2 a1 = word_int4(q.y, xr + 4, make_float2(0.f, 0.f));
    return fmaf(__uint_as_float(sz << 16), (a0.x + a1.x) + (a0.y + a1.y), __uint_as_float(sz & 0xFFFF0000u) * xz);
  } else if (DT == DT_INT8) {
    const uint4 q = reinterpret_cast<const uint4*>(base)[rl];
    float2 a0 = word_int8(q.x, xr, make_float2(0.f, 0.f));
    float2 a1 = word_int8(q.z, xr + 4, make_float2(0.f, 0.f));
    a0 = word_int8(q.y, xr + 2, a0);
    a1 = word_int8(q.w, xr + 6, a1);
    return ((a0.x + a1.x) + (a0.y + a1.y)) - xz;
  } else {
    const uint4 q0 = reinterpret_cast<const uint4*>(base)[2 * rl], q1 = reinterpret_cast<const uint4*>(base)[2 * rl + 1];
    float2 a0 = word_bf16(q0.x, xr, make_float2(0.f, 0.f));
    float2 a1 = word_bf16(q1.x, xr + 4, make_float2(0.f, 0.f));
    a0 = word_bf16(q0.y, xr + 1, a0);
    a1 = word_bf16(q1.y, xr + 5, a1);
    a0 = word_bf16(q0.z, xr + 2, a0);
    a1 = word_bf16(q1.z, xr + 6, a1);
    a0 = word_bf16(q0.w, xr + 3, a0);
    a1 = word_bf16(q1.w, xr + 7, a1);
    return (a0.x + a1.x) + (a0.y + a1.y);
  }
}

// A dense FFN in one phase (PH_FFN).  For each of this CTA's gate/up tiles
// (round-robin): the two half-tiles as in a GEMV phase, whose combining warps
// write silu(gate) * up of their 8 pairs into a shared buffer instead of
// memory; then the tile's 16-column slice of the down projection, split into
// slots of rows: lane l takes rows l, l + 32, ... of a slot, multiplies the
// slot's codes by the 16 SwiGLU outputs (dequantised as in the GEMV) and adds
// into the CTA's partial down outputs in shared memory.  At the end the CTA
// adds its partial outputs to the residual (vector atomics): the down
// projection needs no phase, no grid barrier and no staging of its own.
template <int DT>
__device__ bool ffn_phase(const Phase& ph, const Params& P, const Smem& S, Cons& cs, int cta, int pos) {
  constexpr int E = DT == DT_BF16 ? 8 : DT == DT_INT8 ? 16 : 32;
  const int G = P.nctas, C = ph.K / E, nb = (C + KBLK - 1) / KBLK;
  const int tps = ph.N / TR, d = ph.N2;
  int nsl, DR;
  ffn_split(DT, d, nsl, DR);
  const int lane = cs.lane, w = cs.warp;
  // The CTA's partial down outputs.  int8 / bf16 slots add in turn with plain
  // adds (below), into two buffers where they fit (local tile kp into buffer
  // kp % nbuf); int4 slots, whose tiles span fewer slots, use shared atomic
  // adds into one buffer (measured faster on this path; the order of the adds
  // then varies, the sum only by rounding).
  constexpr bool ORDERED = DT != DT_INT4;
  const int nbuf = ORDERED && ph.K + d + ffn_smem_floats(d) <= KMAX ? 2 : 1;
  float* dacc = S.xs + ph.K;   // [nbuf][d]
  float* hb = dacc + nbuf * d;  // [FFN_HN][16] SwiGLU outputs of the tiles in flight
  int* hcnt = reinterpret_cast<int*>(hb + FFN_HN * 16);  // [FFN_HN] half-tiles finished per buffer
  // dturn[b][k]: tiles of buffer b whose down slot k has been added; the
  // buffer's next tile waits for it, so each row of a buffer is added to by
  // one warp at a time, tile after tile (plain adds, a fixed order), while
  // with two buffers consecutive tiles never wait for each other
  int* dturn = hcnt + FFN_HN;  // [2][FFN_MAXSL]
  for (int i = cs.ctid; i < nbuf * d; i += NCW * 32) dacc[i] = 0.0f;
  if (cs.ctid < FFN_HN) hcnt[cs.ctid] = 0;
  if (cs.ctid < 2 * FFN_MAXSL) dturn[cs.ctid] = 0;
  if (!cta_sync(S, cs, P.err)) return false;
  uint32_t j = 0;
  int kt = 0;  // this CTA's tiles so far
  // the down slice of local tile kp (buffer e), slots j .. j + nsl - 1
  auto down = [&](int kp) -> bool {
    const int e = kp % FFN_HN, target = 2 * (kp / FFN_HN + 1);
    for (int k = (w - (int)((cs.it + j) % NCW) + NCW) % NCW; k < nsl; k += NCW) {
      // this tile's SwiGLU outputs (both half-tiles combined; bounded wait)
      int ok = 1;
      if (lane == 0) {
        volatile int* c = hcnt + e;
        if (*c < target) {
          const uint64_t t0 = gtimer();
          while (*c < target) {
            __nanosleep(32);
            if (gtimer() - t0 > WAIT_NS) {
              atomicCAS(P.err, 0, ERR_WAIT_COMBINE);
              ok = 0;
              break;
            }
          }
        }
        __threadfence_block();
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      float hv[16];
#pragma unroll
      for (int c = 0; c < 16; c += 4) {
        const float4 t4 = reinterpret_cast<const float4*>(hb)[e * 4 + c / 4];
        hv[c] = t4.x;
        hv[c + 1] = t4.y;
        hv[c + 2] = t4.z;
        hv[c + 3] = t4.w;
      }
      // the inputs as the subnormal dequantisation reads them (natural k order)
      float2 xr[8];
      float hs = 0.0f;
#pragma unroll
      for (int c = 0; c < 16; c += 4) {
        const float4 m = dq_mult(DT, DT == DT_INT4 ? (c >> 2) & 1 : 0);
        xr[c / 2] = make_float2(hv[c] * m.x, hv[c + 1] * m.y);
        xr[c / 2 + 1] = make_float2(hv[c + 2] * m.z, hv[c + 3] * m.w);
        hs += (hv[c] + hv[c + 1]) + (hv[c + 2] + hv[c + 3]);
      }
      const float xz = DT == DT_INT4 ? hs * DQ_DOWN : DT == DT_INT8 ? 128.0f * hs * DQ_DOWN : 0.0f;
      const uint32_t it = cs.it + j + (uint32_t)k;
      const uint8_t* base;
      if (!slot_acquire(S, cs, it, P.err, base)) return false;
      // the buffer's previous tile has added its slot k (bounded wait)
      const int bsel = kp % nbuf, turn = kp / nbuf;
      float* acc = dacc + bsel * d;
      int* tp = dturn + bsel * FFN_MAXSL + k;
      if (ORDERED && lane == 0) {
        volatile int* c = tp;
        if (*c != turn) {
          const uint64_t t0 = gtimer();
          while (*c != turn) {
            __nanosleep(32);
            if (gtimer() - t0 > WAIT_NS) {
              atomicCAS(P.err, 0, ERR_WAIT_COMBINE);
              ok = 0;
              break;
            }
          }
        }
        __threadfence_block();
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      const int r0 = k * DR, nr = min(DR, d - r0);
      if (!ORDERED) {
#pragma unroll 4
        for (int i = 0; i * 32 < nr; ++i) {
          const int rl = lane + 32 * i;
          if (rl < nr) atomicAdd(acc + r0 + rl, down_row<DT>(base, rl, DR, xr, xz));
        }
      }
      // groups of four rows per lane: their loads (codes, scales and the
      // partial outputs, which no other warp touches now) go out first
      for (int i0 = 0; ORDERED && i0 * 32 < nr; i0 += 4) {
        float c[4], a0[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int rl = lane + 32 * (i0 + u);
          c[u] = 0.f;
          a0[u] = 0.f;
          if (rl < nr) {
            a0[u] = acc[r0 + rl];
            c[u] = down_row<DT>(base, rl, DR, xr, xz);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int rl = lane + 32 * (i0 + u);
          if (rl < nr) acc[r0 + rl] = a0[u] + c[u];
        }
      }
      __syncwarp();
      if (ORDERED && lane == 0) {
        __threadfence_block();
        *reinterpret_cast<volatile int*>(tp) = turn + 1;
      }
      slot_release(S, cs, it);
    }
    j += (uint32_t)nsl;
    return true;
  };
  for (int t = first_unit(cta, ph.rot, G); t < tps; t += G, ++kt) {
    const int e = kt % FFN_HN;
    for (int h = 0; h < 2; ++h, ++cs.useq, j += (uint32_t)nb) {
      float tot;
      float2 rp;
      const int k = gemv_half<DT>(ph, P, S, cs, 0, t, h * HROWS, TR, j, pos, tot, rp);
      if (k < 0) return false;
      if (k == 0) continue;
      const float up = __shfl_xor_sync(0xffffffffu, tot, 1);
      if (lane < HROWS && (lane & 1) == 0) hb[e * 16 + h * 8 + (lane >> 1)] = tot / (1.0f + expf(-tot)) * up;
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        atomicAdd(hcnt + e, 1);
      }
    }
    // the previous tile's down slice follows this tile's gate/up blocks
    if (kt > 0 && !down(kt - 1)) return false;
  }
  if (kt > 0 && !down(kt - 1)) return false;
  cs.it += j;
  // every warp's partial outputs are in dacc: add them to the residual
  if (!cta_sync(S, cs, P.err)) return false;
  if (kt > 0) {
    float4* out = reinterpret_cast<float4*>(ph.out);
    for (int n4 = cs.ctid; n4 < d / 4; n4 += NCW * 32) {
      float4 v = reinterpret_cast<const float4*>(dacc)[n4];
      if (nbuf == 2) {
        const float4 v1 = reinterpret_cast<const float4*>(dacc + d)[n4];
        v = make_float4(v.x + v1.x, v.y + v1.y, v.z + v1.z, v.w + v1.w);
      }
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
// (16 positions of K and V) belongs to the warp given by its stream index.
// A warp takes the 16 positions of a block at once: lane l holds dims
// l*DPL .. l*DPL+DPL-1 (DPL = HD/32) of every position; it forms the 16
// partial dot products of its dims, a reduce-scatter over the lanes leaves
// lane l with the score of position l/2, and the block updates the warp's
// online softmax (m, l, o) once per q head: one rescale, one exponential per
// position, and the V sum weighted by each position's probability broadcast
// from its lane.  The warps merge in shared memory; a head split over several
// chunks merges its chunks' (m, l, o) in the CTA that finishes last
// (log-sum-exp combine).
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
template <int HD, int NP>
__device__ __forceinline__ void attn_scores(const AttnRows<HD, NP>& kr, int np, int gq, const float (*q)[HD / 32],
                                            float* m, float* l, float* pr, float* cr, int lane) {
  constexpr int DPL = HD / 32;
  const bool valid = (lane >> 1) < np;
#pragma unroll
  for (int jj = 0; jj < MAX_GQ; ++jj) {
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
template <int HD, int NP>
__device__ __forceinline__ void attn_values(const AttnRows<HD, NP>& vr, int gq, const float* pr, const float* cr,
                                            float (*o)[HD / 32]) {
  constexpr int DPL = HD / 32;
#pragma unroll
  for (int jj = 0; jj < MAX_GQ; ++jj) {
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

template <int HD>
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
  const int nslots = pe > p0 ? (pe - p0 + ATT_POS_PER_SLOT - 1) / ATT_POS_PER_SLOT : 0;
  // positions not streamed (rows written during this launch, at most 8) go
  // to the warp after the last slot's owner, which loads them right away
  const int pg = max(pe, p0);
  const int gw = (int)((cs.it + j + (uint32_t)nslots) % NCW);
  const bool has_g = (w == gw) && pg < p1;
  // rows written during this launch: a verify pass's own rows (at most
  // MAX_M) or a decode step's current row
  constexpr int NPG = MAX_M;
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

  float q[MAX_GQ][DPL], m[MAX_GQ], l[MAX_GQ], o[MAX_GQ][DPL];
#pragma unroll
  for (int jj = 0; jj < MAX_GQ; ++jj) {
    m[jj] = -INFINITY;
    l[jj] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
      q[jj][d] = jj < gq ? qs[jj * HD + lane * DPL + d] : 0.f;
      o[jj][d] = 0.f;
    }
  }
  float pr[MAX_GQ], cr[MAX_GQ];
  if (has_g) {
    attn_scores<HD, NPG>(gk, p1 - pg, gq, q, m, l, pr, cr, lane);
    attn_values<HD, NPG>(gv, gq, pr, cr, o);
  }
  for (int k = (w - (int)((cs.it + j) % NCW) + NCW) % NCW; k < nslots; k += NCW) {
    const uint32_t it = cs.it + j + (uint32_t)k;
    const int np = min(ATT_POS_PER_SLOT, pe - (p0 + k * ATT_POS_PER_SLOT));
    const uint8_t* base;
    if (!slot_acquire(S, cs, it, P.err, base)) return false;
    const uint16_t* kb = reinterpret_cast<const uint16_t*>(base);
    {
      AttnRows<HD, ATT_POS_PER_SLOT> kr;
      attn_rows<HD, ATT_POS_PER_SLOT, false>(kr, kb, np, lane);
      attn_scores<HD, ATT_POS_PER_SLOT>(kr, np, gq, q, m, l, pr, cr, lane);
    }
    {
      AttnRows<HD, ATT_POS_PER_SLOT> vr;
      attn_rows<HD, ATT_POS_PER_SLOT, false>(vr, kb + ATT_POS_PER_SLOT * HD, np, lane);
      slot_release(S, cs, it);  // the slot's rows are in registers
      attn_values<HD, ATT_POS_PER_SLOT>(vr, gq, pr, cr, o);
    }
  }
  j += (uint32_t)nslots;
  // the warps of this CTA merge in shared memory
#pragma unroll
  for (int jj = 0; jj < MAX_GQ; ++jj) {
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
  if (nch == 1) return true;
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
  }
  return true;
}

// ========================================================= verify pass ====
// A speculative-verification pass (gpt-fast README, "Speculative sampling")
// feeds M rows (the last accepted token and the drafts) at positions
// pos..pos+M-1 through every layer with ONE stream of the weights.  GEMV
// phases then work K-block by K-block over groups of up to VTG tiles: the
// CTA stages the K-block's inputs of all M rows (fp32, swizzled per chunk),
// each slot's owner warp dequantises its codes once and multiplies them with
// the M rows, reduces over its lanes and adds the row sums into a shared
// accumulator (each (row, m) has one writer per K-block, K-blocks in order:
// deterministic); the group's epilogues then run per (row, m).
struct VS {
  float* xk;    // [MAX_M][KBLK chunks][E] inputs of the current K-block
  float* xgk;   // [MAX_M][KBLK] chunk sums of the inputs, as S.xsum
  float* acc;   // [VTG * TR][MAX_M] row sums of the tile group
  float* rfac;  // [MAX_M] RMSNorm factors
};
__device__ __forceinline__ VS vsmem(const Smem& S) {
  VS v;
  v.xk = S.xs;
  v.xgk = v.xk + MAX_M * KBLK * 32;
  v.acc = v.xgk + MAX_M * KBLK;
  v.rfac = v.acc + VTG * TR * MAX_M;
  return v;
}

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
  constexpr int E = DT == DT_BF16 ? 8 : DT == DT_INT8 ? 16 : 32;
  constexpr int U = E / 4;
  constexpr int WP = E / 8;  // input pairs per 32-bit word of codes
  const VS V = vsmem(S);
  const int M = P.M;
  const int C = ph.K / E, nb = (C + KBLK - 1) / KBLK;
  const int lane = cs.lane, w = cs.warp;
  if ((ph.xsrc == X_NORM || ph.xsrc == X_EMBED_NORM) && !verify_norm(ph, P, S, cs, cta)) return false;
  if (ph.moe == MOE_GU && !verify_route(ph, P, S, cs, pi)) return false;
  int Ns;
  const uint8_t* wseg[8];
  int eseg[8];
  const int nseg = gemv_segments(ph, P, S, Ns, wseg, eseg);
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
    for (int b = 0; b < nb; ++b) {
      const int Lb = min(KBLK, C - b * KBLK);
      // stage the K-block's inputs of the M rows
      const int per_m = KBLK * U;  // float4 per row
      for (int q0 = 0; q0 < MAX_M * per_m; q0 += NCW * 32) {
        const int q = q0 + cs.ctid, m = q / per_m, f4 = q % per_m, l = f4 / U, u = f4 % U;
        const bool ok = m < M && l < Lb;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ok) a = vin4(ph, P, V, m, e, (b * KBLK + l) * U + u);
        const float4 mu = dq_mult(DT, u);
        if (ok)
          reinterpret_cast<float4*>(V.xk)[m * per_m + l * U + (u ^ swz(l, U))] =
              make_float4(a.x * mu.x, a.y * mu.y, a.z * mu.z, a.w * mu.w);
        if (DT != DT_BF16) {  // chunk sums as in stage_store
          float sg = a.x + a.y + a.z + a.w;
          sg += __shfl_xor_sync(0xffffffffu, sg, 1);
          sg += __shfl_xor_sync(0xffffffffu, sg, 2);
          if (DT == DT_INT4) sg += __shfl_xor_sync(0xffffffffu, sg, 4);
          if (ok && (lane & (U - 1)) == 0) V.xgk[m * KBLK + l] = sg * (DT == DT_INT4 ? DQ_DOWN : 128.0f * DQ_DOWN);
        }
      }
      if (!cta_sync(S, cs, P.err)) return false;
      for (int i = i0; i < i1; ++i) {
        const int t = tg.first + i * tg.G, lt = t % tg.tps;
        const int Rt = min(TR, Ns - lt * TR);
        for (int h = 0; h * HROWS < Rt; ++h, ++j) {
          const uint32_t it = cs.it + j;
          if ((int)(it % NCW) != w) continue;
          const uint8_t* base;
          if (!slot_acquire(S, cs, it, P.err, base)) return false;
          const bool lane_ok = lane < Lb;
          const int sw = swz(lane, U);
          const uint32_t* wbase = reinterpret_cast<const uint32_t*>(base) + lane * 4;
#pragma unroll 1
          for (int rb = 0; rb < HROWS; rb += 4) {
            float2 a[4][MAX_M];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
              for (int m = 0; m < MAX_M; ++m) a[r][m] = make_float2(0.f, 0.f);
#pragma unroll 1
            for (int jw0 = 0; jw0 < 4; ++jw0) {
              const int jw = (jw0 + (lane >> 3)) & 3;  // per-lane word order: conflict-free loads
              float2 xp[MAX_M][WP];
#pragma unroll
              for (int m = 0; m < MAX_M; ++m) {
                if (m < M) {
                  const float4* xm = xk4 + m * (KBLK * U) + lane * U;
                  if (DT == DT_INT4) {
                    const float4 xa = xm[(2 * jw) ^ sw], xb = xm[(2 * jw + 1) ^ sw];
                    xp[m][0] = make_float2(xa.x, xa.y);
                    xp[m][1 % WP] = make_float2(xa.z, xa.w);
                    xp[m][2 % WP] = make_float2(xb.x, xb.y);
                    xp[m][3 % WP] = make_float2(xb.z, xb.w);
                  } else if (DT == DT_INT8) {
                    const float4 xa = xm[jw ^ sw];
                    xp[m][0] = make_float2(xa.x, xa.y);
                    xp[m][1 % WP] = make_float2(xa.z, xa.w);
                  } else {
                    const float4 xa = xm[(jw >> 1) ^ sw];
                    xp[m][0] = (jw & 1) ? make_float2(xa.z, xa.w) : make_float2(xa.x, xa.y);
                  }
                } else {
#pragma unroll
                  for (int i2 = 0; i2 < WP; ++i2) xp[m][i2] = make_float2(0.f, 0.f);
                }
              }
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                const uint32_t wv = wbase[(rb + r) * Lb * 4 + jw];
                float2 qv[WP];
                if (DT == DT_INT4) {  // the subnormal reading of word_int4
                  const uint32_t hv = wv >> 8;
                  qv[0] = bits2(wv & 0x0000000Fu, wv & 0x000000F0u);
                  qv[1 % WP] = bits2(wv & 0x00000F00u, wv & 0x0000F000u);
                  qv[2 % WP] = bits2(wv & 0x000F0000u, wv & 0x00F00000u);
                  qv[3 % WP] = bits2(hv & 0x000F0000u, hv & 0x00F00000u);
                } else if (DT == DT_INT8) {  // as word_int8
                  const uint32_t w8 = wv, hv = w8 >> 8;
                  qv[0] = bits2(w8 & 0x000000FFu, w8 & 0x0000FF00u);
                  qv[1 % WP] = bits2(w8 & 0x00FF0000u, hv & 0x00FF0000u);
                } else {
                  qv[0] = bits2(wv << 16, wv & 0xFFFF0000u);
                }
#pragma unroll
                for (int m = 0; m < MAX_M; ++m)
#pragma unroll
                  for (int i2 = 0; i2 < WP; ++i2) a[r][m] = ffma2(qv[i2], xp[m][i2], a[r][m]);
              }
            }
            // per (row, m) contributions, then a reduce-scatter over the lanes:
            // lane l ends with the total of row l >> 3 of the batch, input row l & 7
            float v[32];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              uint32_t sz = 0u;
              if (DT == DT_INT4) sz = reinterpret_cast<const uint32_t*>(base + SLOT_SZ_OFF)[(rb + r) * Lb + lane];
#pragma unroll
              for (int m = 0; m < MAX_M; ++m) {
                float c;
                if (DT == DT_INT4) {
                  c = fmaf(__uint_as_float(sz << 16), a[r][m].x + a[r][m].y,
                           __uint_as_float(sz & 0xFFFF0000u) * V.xgk[m * KBLK + lane]);
                } else if (DT == DT_INT8) {
                  c = (a[r][m].x + a[r][m].y) - V.xgk[m * KBLK + lane];
                } else {
                  c = a[r][m].x + a[r][m].y;
                }
                v[r * 8 + m] = (lane_ok && m < M) ? c : 0.0f;
              }
            }
#pragma unroll
            for (int sft = 16, n = 32; sft >= 1; sft >>= 1, n >>= 1) {
              const bool hi = lane & sft;
#pragma unroll
              for (int k = 0; k < n / 2; ++k) {
                const float keep = hi ? v[k + n / 2] : v[k];
                const float send = hi ? v[k] : v[k + n / 2];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, send, sft);
              }
            }
            const int rr = h * HROWS + rb + (lane >> 3), m = lane & 7;
            if (m < M) V.acc[((i - i0) * TR + rr) * MAX_M + m] += v[0];
          }
          slot_release(S, cs, it);
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
      S.red[cs.warp * 8 + m] = a.v;  // red has 64 floats: warps x rows <= 7 x 8
      S.bcast[cs.warp * 8 + m] = a.i;
    }
  }
  if (!cta_sync(S, cs, P.err)) return false;
  if (cs.ctid == 0) {
    for (int m = 0; m < P.M; ++m) {
      ArgMax b = {S.red[m], S.bcast[m]};
      for (int w = 1; w < NCW; ++w) amax_merge(b, S.red[w * 8 + m], S.bcast[w * 8 + m]);
      P.amax_val[cta * MAX_M + m] = b.v;
      P.amax_idx[cta * MAX_M + m] = b.i;
    }
    __threadfence();
    const unsigned old = atomicAdd(P.amax_tick, 1u);
    if (old == (unsigned)(P.nctas - 1)) {
      __threadfence();
      int a[MAX_M];
      for (int m = 0; m < P.M; ++m) {
        ArgMax g = {-INFINITY, 0x7fffffff};
        for (int k = 0; k < P.nctas; ++k)
          amax_merge(g, __ldcg(P.amax_val + k * MAX_M + m), __ldcg(P.amax_idx + k * MAX_M + m));
        a[m] = g.i;
      }
      int n = 0;
      while (n < P.M - 1 && a[n] == P.tokens[n + 1]) ++n;
      *P.n_accepted = n;
      *P.next_token = a[n];
      *P.amax_tick = 0u;
      int* pos = const_cast<int*>(P.d_pos);
      *pos = *pos + n + 1;
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
  const int K = ph.K, U = per_chunk(ph.dtype) / 4, K4 = K / 4;
  const float4* xs4 = reinterpret_cast<const float4*>(S.xs);
  for (int e = cs.warp; e < ph.n_experts; e += NCW) {
    const uint2* wr = reinterpret_cast<const uint2*>(ph.router + (size_t)e * K);
    float acc = 0.0f;
    for (int k4 = cs.lane; k4 < K4; k4 += 32) {
      const int g = k4 / U, u = k4 % U;
      const float4 xm = xs4[g * U + (u ^ swz(g, U))], iv = dq_inv(ph.dtype, u);
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
      mbar_init(&S.empty[i], 1);
    }
    mbar_init(S.cbar, NCW * 32);
    mbar_init(S.xbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < NTB) {
    S.tbc[tid] = 0;
    S.tbg[tid] = tid;
  }
  if (tid == 0) S.bcast[34] = 0;
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
  if (verifying(P)) {
    bool bad = P.M < 1 || P.M > MAX_M || pos + P.M > P.tmax;
    for (int m = 0; m < P.M; ++m) bad |= P.tokens[m] < 0 || P.tokens[m] >= P.vocab;
    if (bad) {
      if (tid == 0) atomicCAS(P.err, 0, ERR_BAD_TOKEN);
      return;
    }
  }

  if (warp == NCW) {
    if (lane == 0) producer(P, S, cta, pos);
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
  cs.xphase = 0;
  const int G = P.nctas;
  ArgMax am = {-INFINITY, 0x7fffffff};
  ArgMax amv[MAX_M];
#pragma unroll
  for (int m = 0; m < MAX_M; ++m) amv[m] = am;
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
      if (tid == 0) ok = grid_wait(P.bars + ph.wait_bar, (unsigned)G, P.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return;
      if (!cta_sync(S, cs, P.err)) return;
    }
    if (tr) tr[1] = gtimer();
    if (ph.kind == PH_GEMV && verifying(P)) {
      if (tr) tr[2] = gtimer();
      bool ok;
      if (ph.dtype == DT_INT4) ok = gemv_phase_m<DT_INT4>(ph, P, S, cs, cta, pos, pi, amv);
      else if (ph.dtype == DT_INT8) ok = gemv_phase_m<DT_INT8>(ph, P, S, cs, cta, pos, pi, amv);
      else ok = gemv_phase_m<DT_BF16>(ph, P, S, cs, cta, pos, pi, amv);
      if (!ok) return;
      if (ph.epi == EPI_LOGITS) any_logits = true;
    } else if (ph.kind == PH_GEMV) {
      if (!stage_x(ph, P, S, cs, cta)) return;
      if (ph.moe == MOE_GU && !route_experts(ph, P, S, cs, pi)) return;
      if (tr) tr[2] = gtimer();
      bool ok;
      if (ph.dtype == DT_INT4) ok = gemv_phase<DT_INT4>(ph, P, S, cs, cta, pos, am);
      else if (ph.dtype == DT_INT8) ok = gemv_phase<DT_INT8>(ph, P, S, cs, cta, pos, am);
      else ok = gemv_phase<DT_BF16>(ph, P, S, cs, cta, pos, am);
      if (!ok) return;
      if (ph.epi == EPI_LOGITS) any_logits = true;
    } else if (ph.kind == PH_FFN) {
      if (!stage_x(ph, P, S, cs, cta)) return;
      if (tr) tr[2] = gtimer();
      bool ok;
      if (ph.dtype == DT_INT4) ok = ffn_phase<DT_INT4>(ph, P, S, cs, cta, pos);
      else if (ph.dtype == DT_INT8) ok = ffn_phase<DT_INT8>(ph, P, S, cs, cta, pos);
      else ok = ffn_phase<DT_BF16>(ph, P, S, cs, cta, pos);
      if (!ok) return;
    } else if (ph.kind == PH_ATTN) {
      if (tr) tr[2] = tr[1];
      const int nunits = attn_units(ph, P, pos, -1, nullptr);
      uint32_t j = 0;
      for (int u = first_unit(cta, ph.rot, G); u < nunits; u += G) {
        AttnUnit au;
        attn_units(ph, P, pos, u, &au);
        const bool ok = ph.hd == 128 ? attn_unit<128>(ph, P, S, cs, au, pos, j)
                                     : attn_unit<64>(ph, P, S, cs, au, pos, j);
        if (!ok) return;
      }
      cs.it += j;
    }
    if (tr) {
      tr[3] = gtimer();
      tr[6] = cs.starved;
    }
    cs.starved = 0;
    if (tid < PH16) cp_async_wait_all();  // the next phase's descriptor has landed
    // every warp of this CTA has finished the phase (its global writes made)
    if (!cta_sync(S, cs, P.err)) return;
    if (ph.signal_bar >= 0 && tid == 0) grid_arrive(P.bars + ph.signal_bar);
    if (tr) tr[4] = gtimer();
  }
  if (any_logits) {
    if (verifying(P)) verify_finish(P, S, cs, cta, amv);
    else argmax_finish(P, S, cs, cta, am);
  }
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
