// model.cu — host side of the decode step: library-owned quantised weights
// (gf_model), the KV cache with its RoPE table and
// scratch (gf_kv), and the phase program that the persistent engine runs once
// per token.
#include <math.h>
#include <string.h>

#include <vector>

#include "gf_internal.cuh"

struct gf_model {
  gf_model_config cfg;
  int wdtype;
  int G;  // int4 group size
  // One matrix in the device layout; the experts of a layer are packed one
  // after another in one buffer (expert e at e * packed_bytes(N, K)).
  struct Mat {
    uint8_t* packed = nullptr;
    uint16_t* s8 = nullptr;
    int N = 0, K = 0, E = 1;
  };
  std::vector<Mat> qkv, o, gu, dn;  // per layer
  std::vector<uint8_t*> dn_cols;    // dense: column-sliced copy of dn for the fused FFN phase
  bool ffn_fused = false;
  std::vector<uint16_t*> g_attn, g_ffn, router;
  Mat lm;
  uint16_t* embed = nullptr;
  uint16_t* g_final = nullptr;
  std::vector<void*> allocs;
  long long weight_bytes = 0;
};

struct gf_kv {
  gf_model* m = nullptr;
  int Tmax = 0;
  uint16_t *kc = nullptr, *vc = nullptr;
  float2* rope = nullptr;
  float *qbuf = nullptr, *attn = nullptr, *h = nullptr;
  float* resid = nullptr;      // [MAX_M][d] (row 0: decode)
  float* part = nullptr;
  float* hmoe = nullptr;       // verify MoE: [MAX_M][8][ffn]
  float* vlogits = nullptr;    // verify: [MAX_M][vocab] when the caller passes no logits
  int32_t* vscratch = nullptr; // [16] prefill: the pass's accepted count
  gf::Phase* vprog = nullptr;  // verify program
  int nvphases = 0;
  float* amax_val = nullptr;
  int* amax_idx = nullptr;
  unsigned* counters = nullptr;  // bars, attention tickets, q/k/v head counters, the argmax ticket
  size_t counter_bytes = 0;
  unsigned *bars = nullptr, *ticks = nullptr, *headc = nullptr, *attd = nullptr, *amax_tick = nullptr;
  gf::Phase* prog = nullptr;
  int nphases = 0;
  int sms = 0;
  size_t cache_elems = 0;
  std::vector<void*> allocs;
};

namespace gf {

static int dev_alloc(std::vector<void*>& list, void** p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(p, (bytes + 255) / 256 * 256);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_error("device allocation of %zu bytes failed: %s", bytes, cudaGetErrorString(e));
    return GF_ENOMEM;
  }
  list.push_back(*p);
  return GF_OK;
}

static void free_all(std::vector<void*>& list) {
  for (void* p : list) cudaFree(p);
  list.clear();
}

// E matrices of N x K (E = 1: a single matrix) quantised into one buffer,
// expert e from srcs[e].
static int make_mat(gf_model* m, const void* const* srcs, int E, int N, int K, gf_model::Mat& out) {
  out.N = N;
  out.K = K;
  out.E = E;
  const int dt = m->wdtype, G = m->G;
  const long long pb = packed_bytes(dt, N, K, G);
  int rc = dev_alloc(m->allocs, (void**)&out.packed, (size_t)(pb * E));
  if (rc) return rc;
  if (dt == DT_INT8 && (rc = dev_alloc(m->allocs, (void**)&out.s8, (size_t)E * N * 2))) return rc;
  GF_CUDA(cudaMemset(out.packed, 0, (size_t)(pb * E)));  // padding rows and K-slots read as zero
  for (int e = 0; e < E && !rc; ++e) {
    if (!srcs[e]) {
      set_error("gf_model_create: null weight pointer");
      return GF_EINVAL;
    }
    rc = quantize_rows(dt, srcs[e], N, K, G, out.packed + (size_t)(pb * e), out.s8 ? out.s8 + (size_t)e * N : nullptr,
                       nullptr);
  }
  return rc;
}

// bytes one token streams from a matrix (one expert of a tall one): the
// method's codes and scales, not the layout's padding
static long long mat_stream_bytes(const gf_model* m, const gf_model::Mat& a) {
  const int dt = m->wdtype;
  long long b = dt == DT_BF16 ? 2LL * a.N * a.K : dt == DT_INT8 ? (long long)a.N * a.K : (long long)a.N * a.K / 2;
  if (dt == DT_INT8) b += 2LL * a.N;
  if (dt == DT_INT4) b += 4LL * a.N * (a.K / m->G);
  return b;
}

static int copy_vec(gf_model* m, const void* src, size_t elems, uint16_t** out) {
  int rc = dev_alloc(m->allocs, (void**)out, elems * 2);
  if (rc) return rc;
  GF_CUDA(cudaMemcpy(*out, src, elems * 2, cudaMemcpyDeviceToDevice));
  return GF_OK;
}

static int check_cfg(const gf_model_config* c, int wdtype) {
  if (!c || c->d <= 0 || c->n_layers <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->ffn <= 0 || c->vocab <= 0 ||
      c->n_heads % c->n_kv_heads || c->n_heads / c->n_kv_heads > MAX_GQ || (c->head_dim != 64 && c->head_dim != 128) ||
      c->d % 32 || c->ffn % 32 || c->d > KMAX || c->ffn > KMAX || c->n_heads * c->head_dim > KMAX ||
      !(c->eps > 0) || !(c->theta > 0)) {
    set_error("gf_model_create: unsupported configuration");
    return GF_EINVAL;
  }
  if (c->n_experts == 1 || c->n_experts < 0 || c->n_experts > 8) {
    set_error("gf_model_create: n_experts must be 0 (dense) or 2..8");
    return GF_EUNSUPPORTED;
  }
  const int G = c->group_size ? c->group_size : 32;
  if (wdtype == DT_INT4 && ((G != 32 && G != 64 && G != 128) || c->d % G || c->ffn % G ||
                            (c->n_heads * c->head_dim) % G)) {
    set_error("gf_model_create: int4 group size %d must be 32, 64 or 128 and divide d, ffn and the head width", G);
    return GF_EUNSUPPORTED;
  }
  return GF_OK;
}

}  // namespace gf

using namespace gf;

extern "C" {

int gf_model_create(const gf_model_config* cfg, int wdtype, const gf_weights* w, gf_model** out) {
  int rc = check_cfg(cfg, wdtype);
  if (rc) return rc;
  if (!w || !out || wdtype < 0 || wdtype > 2 || !w->embed || !w->g_final || !w->lm_head || !w->wqkv || !w->wo ||
      !w->wgu || !w->wd || !w->g_attn || !w->g_ffn || (cfg->n_experts && !w->router)) {
    set_error("gf_model_create: null weights or bad dtype");
    return GF_EINVAL;
  }
  gf_model* m = new gf_model();
  m->cfg = *cfg;
  m->wdtype = wdtype;
  m->G = cfg->group_size ? cfg->group_size : 32;
  const gf_model_config& c = *cfg;
  const int hd = c.head_dim, qkvN = (c.n_heads + 2 * c.n_kv_heads) * hd;
  m->qkv.resize(c.n_layers);
  m->o.resize(c.n_layers);
  m->gu.resize(c.n_layers);
  m->dn.resize(c.n_layers);
  m->g_attn.resize(c.n_layers);
  m->g_ffn.resize(c.n_layers);
  m->router.resize(c.n_layers);
  m->dn_cols.resize(c.n_layers, nullptr);
  const int E = c.n_experts;
  // dense FFNs run as one phase when the partial down outputs fit in shared
  // memory beside the staged input
  m->ffn_fused = !E && round_up(c.d, slot_k(wdtype)) + c.d + FFN_HN * 16 + 2 * FFN_HN <= KMAX && c.d % 16 == 0;
  for (int l = 0; l < c.n_layers && !rc; ++l) {
    if (!w->wqkv[l] || !w->wo[l] || !w->g_attn[l] || !w->g_ffn[l] || (E && !w->router[l])) {
      set_error("gf_model_create: null weight pointer in layer %d", l);
      rc = GF_EINVAL;
      break;
    }
    if ((rc = make_mat(m, &w->wqkv[l], 1, qkvN, c.d, m->qkv[l]))) break;
    if ((rc = make_mat(m, &w->wo[l], 1, c.d, c.n_heads * hd, m->o[l]))) break;
    m->weight_bytes += mat_stream_bytes(m, m->qkv[l]) + mat_stream_bytes(m, m->o[l]);
    if (E) {
      if ((rc = make_mat(m, w->wgu + (size_t)l * E, E, 2 * c.ffn, c.d, m->gu[l]))) break;
      if ((rc = make_mat(m, w->wd + (size_t)l * E, E, c.d, c.ffn, m->dn[l]))) break;
      if ((rc = copy_vec(m, w->router[l], (size_t)E * c.d, &m->router[l]))) break;
      // a token streams two experts and the router
      m->weight_bytes += 2 * (mat_stream_bytes(m, m->gu[l]) + mat_stream_bytes(m, m->dn[l])) + (long long)E * c.d * 2;
    } else {
      if (!w->wgu[l] || !w->wd[l]) {
        set_error("gf_model_create: null weight pointer in layer %d", l);
        rc = GF_EINVAL;
        break;
      }
      if ((rc = make_mat(m, &w->wgu[l], 1, 2 * c.ffn, c.d, m->gu[l]))) break;
      if ((rc = make_mat(m, &w->wd[l], 1, c.d, c.ffn, m->dn[l]))) break;
      m->weight_bytes += mat_stream_bytes(m, m->gu[l]) + mat_stream_bytes(m, m->dn[l]);
      if (m->ffn_fused) {
        // the decode step streams this copy instead of dn (same bytes); the
        // verify pass keeps using dn
        if ((rc = dev_alloc(m->allocs, (void**)&m->dn_cols[l], (size_t)cols_bytes(wdtype, c.d, c.ffn)))) break;
        if ((rc = pack_cols(wdtype, m->dn[l].packed, c.d, c.ffn, m->G, m->dn_cols[l], nullptr))) break;
      }
    }
    if ((rc = copy_vec(m, w->g_attn[l], c.d, &m->g_attn[l]))) break;
    if ((rc = copy_vec(m, w->g_ffn[l], c.d, &m->g_ffn[l]))) break;
    m->weight_bytes += 2LL * c.d * 2;
  }
  if (!rc) rc = make_mat(m, &w->lm_head, 1, c.vocab, c.d, m->lm);
  if (!rc) m->weight_bytes += mat_stream_bytes(m, m->lm);
  if (!rc) rc = copy_vec(m, w->embed, (size_t)c.vocab * c.d, &m->embed);
  if (!rc) rc = copy_vec(m, w->g_final, c.d, &m->g_final);
  if (!rc) {
    m->weight_bytes += (long long)c.d * 2 /* g_final */ + (long long)c.d * 2 /* one embedding row */;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) rc = cuda_fail(e, "gf_model_create");
  }
  if (rc) {
    free_all(m->allocs);
    delete m;
    return rc;
  }
  *out = m;
  return GF_OK;
}

int gf_model_destroy(gf_model* m) {
  if (!m) return GF_EINVAL;
  free_all(m->allocs);
  delete m;
  return GF_OK;
}

long long gf_model_weight_bytes(const gf_model* m) { return m ? m->weight_bytes : -1; }

int gf_kv_create(gf_model* m, int Tmax, gf_kv** out) {
  if (!m || !out || Tmax <= 0) {
    set_error("gf_kv_create: bad arguments");
    return GF_EINVAL;
  }
  const gf_model_config& c = m->cfg;
  const int hd = c.head_dim, L = c.n_layers, Hq = c.n_heads, Hkv = c.n_kv_heads;
  gf_kv* kv = new gf_kv();
  kv->m = m;
  kv->Tmax = Tmax;
  kv->sms = device_sms();
  const int G = kv->sms;
  int rc = GF_OK;
  const size_t cache_elems = (size_t)L * Hkv * Tmax * hd;
  kv->cache_elems = cache_elems;
  const int nch_max = (G + Hkv - 1) / Hkv;
  const int E = c.n_experts;
  const int ppl = E ? 6 : m->ffn_fused ? 4 : 5;  // phases per layer
  const int nph = ppl * L + 1;
  const int nbars = nph;
  const size_t nticks = (size_t)L * MAX_M * Hkv;
  const size_t nheadc = (size_t)L * Hkv;
  kv->counter_bytes = (nbars + nticks + 2 * nheadc + 1) * sizeof(unsigned);
  do {
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->kc, cache_elems * 2))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->vc, cache_elems * 2))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->rope, (size_t)Tmax * (hd / 2) * sizeof(float2)))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->qbuf, (size_t)MAX_M * Hq * hd * 4))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->attn, (size_t)MAX_M * Hq * hd * 4))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->h, (size_t)MAX_M * c.ffn * 4 * (c.n_experts ? 2 : 1)))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->resid, (size_t)MAX_M * c.d * 4))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->part, (size_t)MAX_M * Hq * nch_max * (hd + 2) * 4))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->amax_val, (size_t)G * MAX_M * 4))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->amax_idx, (size_t)G * MAX_M * 4))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->vlogits, (size_t)MAX_M * c.vocab * 4))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->vscratch, 16 * sizeof(int32_t)))) break;
    if (c.n_experts && (rc = dev_alloc(kv->allocs, (void**)&kv->hmoe, (size_t)MAX_M * 8 * c.ffn * 4))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->counters, kv->counter_bytes))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->prog, (size_t)nph * sizeof(Phase)))) break;
    if ((rc = dev_alloc(kv->allocs, (void**)&kv->vprog, (size_t)(5 * L + 1) * sizeof(Phase)))) break;
  } while (0);
  if (rc) {
    free_all(kv->allocs);
    delete kv;
    return rc;
  }
  kv->bars = kv->counters;
  kv->ticks = kv->counters + nbars;
  kv->headc = kv->ticks + nticks;
  kv->attd = kv->headc + nheadc;
  kv->amax_tick = kv->attd + nheadc;
  cudaError_t e = cudaMemset(kv->kc, 0, cache_elems * 2);
  if (e == cudaSuccess) e = cudaMemset(kv->vc, 0, cache_elems * 2);
  if (e == cudaSuccess) e = cudaMemset(kv->counters, 0, kv->counter_bytes);

  // RoPE table: angle pos * theta^(-2i/hd), evaluated in double on the host
  std::vector<float2> rope((size_t)Tmax * (hd / 2));
  for (int p = 0; p < Tmax; ++p)
    for (int i = 0; i < hd / 2; ++i) {
      const double a = (double)p * pow(c.theta, -2.0 * i / hd);
      rope[(size_t)p * (hd / 2) + i] = make_float2((float)cos(a), (float)sin(a));
    }
  if (e == cudaSuccess) e = cudaMemcpy(kv->rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice);

  // The program, per dense layer: q/k/v (with RoPE and the KV append),
  // attention and the o projection in one stretch without a grid barrier (each
  // attention unit waits for its kv group's q/k/v tiles, each o unit for the
  // attention of its heads), then the FFN; lm_head at the end.
  std::vector<Phase> ph(nph);
  std::vector<char> chained(nph, 0);  // 1: follows its predecessor without a grid barrier
  memset(ph.data(), 0, ph.size() * sizeof(Phase));
  long long cum_units = 0;
  const int Gq = m->G;
  auto gemv = [&](Phase& p, const gf_model::Mat& mat) {
    p.kind = PH_GEMV;
    p.dtype = m->wdtype;
    p.N = mat.N;
    p.K = mat.K;
    p.G = Gq;
    p.W = mat.packed;
    p.s8 = mat.s8;
    p.rot = (int)(cum_units % G);
    cum_units += (mat.N + TR - 1) / TR;
  };
  for (int l = 0; l < L; ++l) {
    Phase* P = &ph[ppl * l];
    uint16_t* kcl = kv->kc + (size_t)l * Hkv * Tmax * hd;
    uint16_t* vcl = kv->vc + (size_t)l * Hkv * Tmax * hd;
    // q/k/v with RoPE and the KV append
    gemv(P[0], m->qkv[l]);
    P[0].xsrc = l == 0 ? X_EMBED_NORM : X_NORM;
    P[0].xptr = kv->resid;
    P[0].gain = m->g_attn[l];
    P[0].eps = c.eps;
    P[0].epi = EPI_QKV;
    P[0].q_rows = Hq * hd;
    P[0].kv_rows = Hkv * hd;
    P[0].qbuf = kv->qbuf;
    P[0].kc = kcl;
    P[0].vc = vcl;
    P[0].hd = hd;
    P[0].Hq = Hq;
    P[0].Hkv = Hkv;
    P[0].Tmax = Tmax;
    P[0].headc = kv->headc + (size_t)l * Hkv;
    // attention over positions 0..pos (the units start on CTAs that hold
    // fewer q/k/v tiles: the rotation continues after the q/k/v tiles)
    P[1].kind = PH_ATTN;
    P[1].qbuf = kv->qbuf;
    P[1].kc = kcl;
    P[1].vc = vcl;
    P[1].attn_out = kv->attn;
    P[1].q_f32 = 1;
    P[1].out_f32 = 1;
    P[1].Hq = Hq;
    P[1].Hkv = Hkv;
    P[1].hd = hd;
    P[1].Tmax = Tmax;
    P[1].part = kv->part;
    P[1].tick = kv->ticks + (size_t)l * MAX_M * Hkv;
    P[1].headc = kv->headc + (size_t)l * Hkv;
    P[1].attd = kv->attd + (size_t)l * Hkv;
    P[1].stream_cur = 0;
    P[1].rot = (int)(cum_units % G);
    chained[ppl * l + 1] = 1;
    // o projection split by K-slot, each unit added to the residual
    gemv(P[2], m->o[l]);
    P[2].kind = PH_OSPLIT;
    P[2].xsrc = X_F32;
    P[2].xptr = kv->attn;
    P[2].out = kv->resid;
    P[2].attd = kv->attd + (size_t)l * Hkv;
    P[2].Hq = Hq;
    P[2].Hkv = Hkv;
    P[2].hd = hd;
    cum_units += (long long)((c.d + TR - 1) / TR) * (k_slots(m->wdtype, Hq * hd) - 1);  // units, not tiles
    chained[ppl * l + 2] = 1;
    if (!E && m->ffn_fused) {
      // gate/up + SwiGLU + down + residual in one phase
      gemv(P[3], m->gu[l]);
      P[3].kind = PH_FFN;
      P[3].xsrc = X_NORM;
      P[3].xptr = kv->resid;
      P[3].gain = m->g_ffn[l];
      P[3].eps = c.eps;
      P[3].epi = EPI_SWIGLU;
      P[3].out = kv->resid;
      P[3].W2 = m->dn_cols[l];
      P[3].s8b = m->dn[l].s8;
      P[3].N2 = c.d;
    } else if (!E) {
      // gate/up + SwiGLU
      gemv(P[3], m->gu[l]);
      P[3].xsrc = X_NORM;
      P[3].xptr = kv->resid;
      P[3].gain = m->g_ffn[l];
      P[3].eps = c.eps;
      P[3].epi = EPI_SWIGLU;
      P[3].out = kv->h;
      // down + residual
      gemv(P[4], m->dn[l]);
      P[4].xsrc = X_F32;
      P[4].xptr = kv->h;
      P[4].epi = EPI_RESID;
      P[4].out = kv->resid;
    } else {
      // router + gate/up of the two chosen experts (2 x 2 ffn rows)
      gf_model::Mat two = m->gu[l];
      two.N = 2 * m->gu[l].N;
      gemv(P[3], two);
      P[3].moe = MOE_GU;
      P[3].n_experts = E;
      P[3].router = m->router[l];
      P[3].xsrc = X_NORM;
      P[3].xptr = kv->resid;
      P[3].gain = m->g_ffn[l];
      P[3].eps = c.eps;
      P[3].epi = EPI_MOE_SWIGLU;
      P[3].out = kv->h;
      // down projection of each chosen expert, weighted into the residual
      for (int k = 0; k < 2; ++k) {
        Phase& D = P[4 + k];
        gemv(D, m->dn[l]);
        D.moe = k == 0 ? MOE_DOWN0 : MOE_DOWN1;
        D.n_experts = E;
        D.xsrc = X_F32;
        D.xptr = kv->h + (size_t)k * c.ffn;
        D.epi = EPI_MOE_RESID;
        D.out = kv->resid;
      }
    }
  }
  Phase& lm = ph[nph - 1];
  gemv(lm, m->lm);
  lm.xsrc = X_NORM;
  lm.xptr = kv->resid;
  lm.gain = m->g_final;
  lm.eps = c.eps;
  lm.epi = EPI_LOGITS;
  // grid barriers: phase i waits on barrier i - 1, which phase i - 1 signals,
  // unless it is chained to its predecessor
  for (int i = 0; i < nph; ++i) {
    ph[i].wait_bar = (i == 0 || chained[i]) ? -1 : i - 1;
    ph[i].signal_bar = (i == nph - 1 || chained[i + 1]) ? -1 : i;
  }
  kv->nphases = nph;
  if (e == cudaSuccess) e = cudaMemcpy(kv->prog, ph.data(), ph.size() * sizeof(Phase), cudaMemcpyHostToDevice);

  // The verify program: the same layers over up to MAX_M rows, each GEMV
  // phase reading its rows' inputs at a row stride, every phase behind a grid
  // barrier; a MoE layer streams the union of the rows' experts (gate/up,
  // then down) once.
  const int nvph = 5 * L + 1;
  std::vector<Phase> vp(nvph);
  memset(vp.data(), 0, vp.size() * sizeof(Phase));
  cum_units = 0;
  for (int l = 0; l < L; ++l) {
    Phase* P = &vp[5 * l];
    const Phase* D = &ph[ppl * l];
    P[0] = D[0];  // q/k/v: rows m at pos + m
    P[0].headc = nullptr;
    P[0].out_mstride = 0;
    P[1] = D[1];  // attention of each row
    P[1].headc = nullptr;
    P[1].attd = nullptr;
    gemv(P[2], m->o[l]);  // o, all rows, behind a grid barrier
    P[2].xsrc = X_F32;
    P[2].xptr = kv->attn;
    P[2].epi = EPI_RESID;
    P[2].out = kv->resid;
    P[2].x_mstride = Hq * hd;
    P[2].out_mstride = c.d;
    if (!E) {
      // gate/up + SwiGLU, then down + residual, as separate phases
      gemv(P[3], m->gu[l]);
      P[3].xsrc = X_NORM;
      P[3].xptr = kv->resid;
      P[3].gain = m->g_ffn[l];
      P[3].eps = c.eps;
      P[3].epi = EPI_SWIGLU;
      P[3].out = kv->h;
      P[3].out_mstride = c.ffn;
      gemv(P[4], m->dn[l]);
      P[4].xsrc = X_F32;
      P[4].xptr = kv->h;
      P[4].x_mstride = c.ffn;
      P[4].epi = EPI_RESID;
      P[4].out = kv->resid;
      P[4].out_mstride = c.d;
    } else {
      P[3] = D[3];  // router + gate/up of the union of experts
      P[3].N = m->gu[l].N;
      P[3].out = kv->hmoe;
      P[3].out_mstride = c.ffn;
      P[4] = D[4];  // down projections of the union, weighted per row
      P[4].moe = MOE_DOWNU;
      P[4].xptr = kv->hmoe;
      P[4].x_mstride = 8 * c.ffn;
      P[4].x_sstride = c.ffn;
      P[4].out_mstride = c.d;
    }
  }
  vp[nvph - 1] = ph[nph - 1];
  for (int i = 0; i < nvph; ++i) {
    vp[i].wait_bar = i == 0 ? -1 : i - 1;
    vp[i].signal_bar = i == nvph - 1 ? -1 : i;
  }
  kv->nvphases = nvph;
  if (e == cudaSuccess) e = cudaMemcpy(kv->vprog, vp.data(), vp.size() * sizeof(Phase), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    rc = cuda_fail(e, "gf_kv_create");
    free_all(kv->allocs);
    delete kv;
    return rc;
  }
  *out = kv;
  return GF_OK;
}

int gf_kv_reset(gf_kv* kv, gf_stream stream) {
  if (!kv) {
    set_error("gf_kv_reset: null handle");
    return GF_EINVAL;
  }
  cudaStream_t s = (cudaStream_t)stream;
  GF_CUDA(cudaMemsetAsync(kv->kc, 0, kv->cache_elems * 2, s));
  GF_CUDA(cudaMemsetAsync(kv->vc, 0, kv->cache_elems * 2, s));
  GF_CUDA(cudaMemsetAsync(kv->counters, 0, kv->counter_bytes, s));
  return GF_OK;
}

int gf_kv_destroy(gf_kv* kv) {
  if (!kv) return GF_EINVAL;
  free_all(kv->allocs);
  delete kv;
  return GF_OK;
}

int gf_kv_cache_ptrs(gf_kv* kv, void** kcache, void** vcache) {
  if (!kv || !kcache || !vcache) {
    set_error("gf_kv_cache_ptrs: null argument");
    return GF_EINVAL;
  }
  *kcache = kv->kc;
  *vcache = kv->vc;
  return GF_OK;
}

static int decode_launch(gf_model* m, gf_kv* kv, const int32_t* d_token, int32_t* d_pos, float* d_logits,
                         int32_t* d_argmax, unsigned long long* d_trace, cudaStream_t stream);

size_t gf_trace_bytes(const gf_kv* kv) {
  return kv ? (size_t)kv->nphases * kv->sms * TRACE_W * sizeof(unsigned long long) : 0;
}

int gf_kv_activation_ptrs(gf_kv* kv, void** q, void** attn, void** h, void** resid) {
  if (!kv || !q || !attn || !h || !resid) {
    set_error("gf_kv_activation_ptrs: null argument");
    return GF_EINVAL;
  }
  *q = kv->qbuf;
  *attn = kv->attn;
  *h = kv->h;
  *resid = kv->resid;
  return GF_OK;
}

int gf_decode_step_traced(gf_model* m, gf_kv* kv, const int32_t* d_token, int32_t* d_pos, float* d_logits,
                          int32_t* d_argmax, unsigned long long* d_trace, gf_stream stream) {
  if (!d_trace || !aligned16(d_trace)) {
    set_error("gf_decode_step_traced: trace buffer must be a 16-byte aligned device pointer");
    return GF_EINVAL;
  }
  return decode_launch(m, kv, d_token, d_pos, d_logits, d_argmax, d_trace, (cudaStream_t)stream);
}

int gf_decode_step(gf_model* m, gf_kv* kv, const int32_t* d_token, int32_t* d_pos, float* d_logits,
                   int32_t* d_argmax, gf_stream stream) {
  return decode_launch(m, kv, d_token, d_pos, d_logits, d_argmax, nullptr, (cudaStream_t)stream);
}

static int decode_launch(gf_model* m, gf_kv* kv, const int32_t* d_token, int32_t* d_pos, float* d_logits,
                         int32_t* d_argmax, unsigned long long* d_trace, cudaStream_t stream) {
  if (!m || !kv || kv->m != m || !d_token || !d_pos || !d_logits || !d_argmax) {
    set_error("gf_decode_step: bad arguments");
    return GF_EINVAL;
  }
  if (!aligned16(d_logits)) {
    set_error("gf_decode_step: logits must be 16-byte aligned");
    return GF_EALIGN;
  }
  cudaStream_t s = (cudaStream_t)stream;
  GF_CUDA(cudaMemsetAsync(kv->counters, 0, kv->counter_bytes, s));
  Params p;
  memset(&p, 0, sizeof p);
  p.prog = kv->prog;
  p.nphases = kv->nphases;
  p.dtype = m->wdtype;
  p.d_pos = d_pos;
  p.nctas = kv->sms;
  p.unit_target = kv->sms;
  p.bars = kv->bars;
  p.err = device_err_ptr();
  p.rope = kv->rope;
  p.resid = kv->resid;
  p.embed = m->embed;
  p.token = d_token;
  p.logits = d_logits;
  p.argmax = d_argmax;
  p.amax_val = kv->amax_val;
  p.amax_idx = kv->amax_idx;
  p.amax_tick = kv->amax_tick;
  p.pos_inc = d_pos;
  p.vocab = m->cfg.vocab;
  p.tmax = kv->Tmax;
  p.trace = d_trace;
  p.M = 1;
  if (!p.err) {
    set_error("gf_decode_step: cannot resolve the device error word");
    return GF_ECUDA;
  }
  return launch_engine(p, kv->sms, true, s);
}

static int verify_launch(gf_model* m, gf_kv* kv, const int32_t* d_tokens, int k, int32_t* d_pos,
                         int32_t* d_n_accepted, int32_t* d_next_token, float* d_logits, int prefill,
                         cudaStream_t stream);

int gf_verify_k(gf_model* m, gf_kv* kv, const int32_t* d_tokens, int k, int32_t* d_pos, int32_t* d_n_accepted,
                int32_t* d_next_token, float* d_logits, gf_stream stream) {
  if (!m || !kv || kv->m != m || !d_tokens || !d_pos || !d_n_accepted || !d_next_token || k < 0 || k + 1 > MAX_M) {
    set_error("gf_verify_k: bad arguments (k must be 0..%d)", MAX_M - 1);
    return GF_EINVAL;
  }
  if (d_logits && !aligned16(d_logits)) {
    set_error("gf_verify_k: logits must be 16-byte aligned");
    return GF_EALIGN;
  }
  return verify_launch(m, kv, d_tokens, k, d_pos, d_n_accepted, d_next_token, d_logits, 0, (cudaStream_t)stream);
}

int gf_prefill(gf_model* m, gf_kv* kv, const int32_t* d_tokens, int n, int32_t* d_pos, int32_t* d_next_token,
               float* d_logits, gf_stream stream) {
  if (!m || !kv || kv->m != m || !d_tokens || !d_pos || !d_next_token || n < 1) {
    set_error("gf_prefill: bad arguments (n=%d)", n);
    return GF_EINVAL;
  }
  if (d_logits && !aligned16(d_logits)) {
    set_error("gf_prefill: logits must be 16-byte aligned");
    return GF_EALIGN;
  }
  cudaStream_t s = (cudaStream_t)stream;
  // passes of up to MAX_M rows; the last pass's last row gives the next
  // token and (if asked) the logits
  for (int c0 = 0; c0 < n; c0 += MAX_M) {
    const int M = n - c0 < MAX_M ? n - c0 : MAX_M;
    const int rc = verify_launch(m, kv, d_tokens + c0, M - 1, d_pos, kv->vscratch, d_next_token, kv->vlogits, 1, s);
    if (rc) return rc;
    if (d_logits && c0 + M == n)
      GF_CUDA(cudaMemcpyAsync(d_logits, kv->vlogits + (size_t)(M - 1) * m->cfg.vocab,
                              (size_t)m->cfg.vocab * sizeof(float), cudaMemcpyDeviceToDevice, s));
  }
  return GF_OK;
}

static int verify_launch(gf_model* m, gf_kv* kv, const int32_t* d_tokens, int k, int32_t* d_pos,
                         int32_t* d_n_accepted, int32_t* d_next_token, float* d_logits, int prefill,
                         cudaStream_t stream) {
  cudaStream_t s = stream;
  GF_CUDA(cudaMemsetAsync(kv->counters, 0, kv->counter_bytes, s));
  Params p;
  memset(&p, 0, sizeof p);
  p.prog = kv->vprog;
  p.nphases = kv->nvphases;
  p.dtype = m->wdtype;
  p.d_pos = d_pos;
  p.nctas = kv->sms;
  p.unit_target = kv->sms;
  p.bars = kv->bars;
  p.err = device_err_ptr();
  p.rope = kv->rope;
  p.resid = kv->resid;
  p.embed = m->embed;
  p.logits = d_logits ? d_logits : kv->vlogits;
  p.amax_val = kv->amax_val;
  p.amax_idx = kv->amax_idx;
  p.amax_tick = kv->amax_tick;
  p.vocab = m->cfg.vocab;
  p.tmax = kv->Tmax;
  p.M = k + 1;
  p.tokens = d_tokens;
  p.n_accepted = d_n_accepted;
  p.next_token = d_next_token;
  p.prefill = prefill;
  p.hbuf_moe = kv->hmoe;
  if (!p.err) {
    set_error("gf_verify_k: cannot resolve the device error word");
    return GF_ECUDA;
  }
  return launch_engine(p, kv->sms, true, s);
}

}  // extern "C"

// ============================================================ generation ===
// Host loops over the decode and verify launches: plain greedy generation
// (gpt-fast README, "Generate text": a prompt, then greedy tokens at batch
// size 1) and speculative generation (README, "Speculative sampling": a draft
// model -- the int8 or int4 copy of the target -- proposes k tokens, the
// target checks them in one pass and keeps the longest prefix equal to its
// own greedy choices plus its next token).  The loops only order launches,
// copy token ids and positions, and count; every step of the arithmetic runs
// in the engine.
namespace {

struct DevInts {  // one small device array, freed on scope exit
  int32_t* p = nullptr;
  ~DevInts() {
    if (p) cudaFree(p);
  }
};

// Feeds the prompt one token per step from position 0; the argmax of the
// last step is written to *d_first (the first generated token), the other
// steps' to *d_junk.
int feed_prompt(gf_model* m, gf_kv* kv, const int32_t* d_prompt, int n, int32_t* d_pos, int32_t* d_first,
                int32_t* d_junk, cudaStream_t s) {
  GF_CUDA(cudaMemsetAsync(d_pos, 0, sizeof(int32_t), s));
  for (int i = 0; i < n; ++i) {
    const int rc = decode_launch(m, kv, d_prompt + i, d_pos, kv->vlogits, i == n - 1 ? d_first : d_junk, nullptr, s);
    if (rc) return rc;
  }
  return GF_OK;
}

}  // namespace

extern "C" {

int gf_generate(gf_model* m, gf_kv* kv, const int32_t* h_prompt, int n_prompt, int n_new, int32_t* h_out,
                gf_stream stream) {
  if (!m || !kv || kv->m != m || !h_prompt || !h_out || n_prompt < 1 || n_new < 1 ||
      (long long)n_prompt + n_new > kv->Tmax) {
    set_error("gf_generate: bad arguments (n_prompt=%d, n_new=%d, Tmax=%d)", n_prompt, n_new, kv ? kv->Tmax : 0);
    return GF_EINVAL;
  }
  cudaStream_t s = (cudaStream_t)stream;
  // [0] position, [1] junk argmax, [8..) the prompt then the generated tokens
  DevInts d;
  const size_t nints = 8 + (size_t)n_prompt + n_new;
  GF_CUDA(cudaMalloc(&d.p, nints * sizeof(int32_t)));
  int32_t* seq = d.p + 8;
  GF_CUDA(cudaMemcpyAsync(seq, h_prompt, (size_t)n_prompt * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  int rc = feed_prompt(m, kv, seq, n_prompt, d.p, seq + n_prompt, d.p + 1, s);
  if (rc) return rc;
  // generated token j (j >= 1) is the argmax of the step fed token j - 1
  for (int j = 1; j < n_new; ++j) {
    int32_t* in = seq + n_prompt + j - 1;
    if ((rc = decode_launch(m, kv, in, d.p, kv->vlogits, in + 1, nullptr, s))) return rc;
  }
  GF_CUDA(cudaMemcpyAsync(h_out, seq + n_prompt, (size_t)n_new * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  GF_CUDA(cudaStreamSynchronize(s));
  return GF_OK;
}

int gf_generate_speculative(gf_model* target, gf_kv* tkv, gf_model* draft, gf_kv* dkv, const int32_t* h_prompt,
                            int n_prompt, int n_new, int k, int32_t* h_out, gf_spec_stats* stats,
                            gf_stream stream) {
  if (!target || !tkv || tkv->m != target || !draft || !dkv || dkv->m != draft || tkv == dkv || !h_prompt ||
      !h_out || n_prompt < 1 || n_new < 1 || k < 1 || k + 1 > MAX_M ||
      target->cfg.vocab != draft->cfg.vocab ||
      (long long)n_prompt + n_new + k + 1 > (tkv->Tmax < dkv->Tmax ? tkv->Tmax : dkv->Tmax)) {
    set_error("gf_generate_speculative: bad arguments (k must be 1..%d, the vocabularies equal, "
              "n_prompt + n_new + k + 1 <= both Tmax)", MAX_M - 1);
    return GF_EINVAL;
  }
  cudaStream_t s = (cudaStream_t)stream;
  // [0] target position, [1] draft position, [2] accepted, [3] next token,
  // [4] junk argmax, [8..8+k] the verify rows (current token, k drafts),
  // [16..) the prompt
  DevInts d;
  GF_CUDA(cudaMalloc(&d.p, (16 + (size_t)n_prompt) * sizeof(int32_t)));
  int32_t *pos_t = d.p, *pos_d = d.p + 1, *n_acc = d.p + 2, *nxt = d.p + 3, *junk = d.p + 4, *rows = d.p + 8;
  int32_t* prompt = d.p + 16;
  GF_CUDA(cudaMemcpyAsync(prompt, h_prompt, (size_t)n_prompt * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  int rc = feed_prompt(target, tkv, prompt, n_prompt, pos_t, rows, junk, s);
  if (!rc) rc = feed_prompt(draft, dkv, prompt, n_prompt, pos_d, junk, junk, s);
  if (rc) return rc;
  gf_spec_stats st = {0, 0, 0};
  int emitted = 0, p = n_prompt;  // rows[0] is the token at position p
  int32_t h[16];
  while (emitted < n_new) {
    // the draft proposes rows[1..k] from rows[0], positions p .. p + k - 1
    for (int j = 0; j < k; ++j)
      if ((rc = decode_launch(draft, dkv, rows + j, pos_d, dkv->vlogits, rows + j + 1, nullptr, s))) return rc;
    // the target checks rows[0..k] at positions p .. p + k in one pass
    if ((rc = gf_verify_k(target, tkv, rows, k, pos_t, n_acc, nxt, nullptr, s))) return rc;
    GF_CUDA(cudaMemcpyAsync(h, d.p, 16 * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    GF_CUDA(cudaStreamSynchronize(s));
    const int n = h[2];
    if (n < 0 || n > k || h[0] != p + n + 1) {
      set_error("gf_generate_speculative: the verify pass returned n=%d at position %d (device error %d)", n,
                h[0], gf_device_error());
      return GF_EDEVICE;
    }
    if (st.rounds == 0) h_out[emitted++] = h[8];  // the target's token after the prompt
    for (int j = 1; j <= n && emitted < n_new; ++j) h_out[emitted++] = h[8 + j];
    if (emitted < n_new) h_out[emitted++] = h[3];
    ++st.rounds;
    st.drafted += k;
    st.accepted += n;
    // the draft's cache must hold rows[0..n] at p .. p + n: with all k
    // accepted it has not yet seen rows[k]; otherwise step back
    if (n == k) {
      if ((rc = decode_launch(draft, dkv, rows + k, pos_d, dkv->vlogits, junk, nullptr, s))) return rc;
    } else {
      const int32_t back = p + n + 1;
      GF_CUDA(cudaMemcpyAsync(pos_d, &back, sizeof back, cudaMemcpyHostToDevice, s));
    }
    GF_CUDA(cudaMemcpyAsync(rows, nxt, sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
    p += n + 1;
  }
  GF_CUDA(cudaStreamSynchronize(s));
  if (stats) *stats = st;
  return GF_OK;
}

}  // extern "C"
