// attn_noalloc.cu — gf_decode_attn_noalloc: the decode attention of
// gf_decode_attn for callers that cannot allocate device memory, e.g. a
// plug-in handed only tensor pointers by a host framework that owns every
// device allocation, or a latency-critical loop that must not enter the CUDA
// allocator (cudaMalloc / cudaFree can synchronise the device).  Its scratch
// (the per-chunk softmax partials and the combine tickets) lives in the
// file-scope array below instead of a caller-provided workspace.
#include <string.h>

#include "gf_internal.cuh"

namespace gf {

// Every GPU that loads this library holds these bytes until the process exits.
static __device__ __align__(256) unsigned char g_attn_scratch[GF_NOALLOC_ATTN_SCRATCH];

// Host code cannot use g_attn_scratch as a device address (in host code the
// name is a stand-in).  The real address is looked up on every call, in the
// current context: a host call that allocates nothing, and stays right after
// the context (and with it the module) has been re-created.
static void* scratch_addr() {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
  if (e != cudaSuccess) {
    set_error("gf_decode_attn_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    return nullptr;
  }
  return p;
}

}  // namespace gf

using namespace gf;

extern "C" {

int gf_decode_attn_noalloc(const void* q, const void* kcache, const void* vcache, int Hq, int Hkv, int hd, int Tmax,
                           int pos, void* out, gf_stream stream) {
  if (!q || !kcache || !vcache || !out || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Hq / Hkv > MAX_GQ ||
      (hd != 64 && hd != 128) || pos < 0 || pos >= Tmax) {
    set_error("gf_decode_attn_noalloc: bad arguments (Hq=%d Hkv=%d hd=%d Tmax=%d pos=%d)", Hq, Hkv, hd, Tmax, pos);
    return GF_EINVAL;
  }
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out)) {
    set_error("gf_decode_attn_noalloc: pointers must be 16-byte aligned");
    return GF_EALIGN;
  }
  const int sms = device_sms();
  if (sms <= 0) {
    set_error("gf_decode_attn_noalloc: cannot query the device");
    return GF_ECUDA;
  }
  // same scratch shape as gf_decode_attn: partials, then one ticket per kv head
  const int nch_max = (sms + Hkv - 1) / Hkv;
  const size_t part_bytes = (size_t)Hq * nch_max * (hd + 2) * sizeof(float);
  const size_t need = part_bytes + ((size_t)Hkv * sizeof(unsigned) + 255) / 256 * 256;
  if (need > (size_t)GF_NOALLOC_ATTN_SCRATCH) {
    set_error("gf_decode_attn_noalloc: needs %zu bytes of scratch for Hq=%d Hkv=%d hd=%d; the static scratch holds "
              "%d bytes (use gf_decode_attn with a workspace instead)",
              need, Hq, Hkv, hd, GF_NOALLOC_ATTN_SCRATCH);
    return GF_EINVAL;
  }
  unsigned char* base = (unsigned char*)scratch_addr();
  if (!base) return GF_ECUDA;
  int* err = device_err_ptr();
  if (!err) {
    set_error("gf_decode_attn_noalloc: cannot resolve the device error word");
    return GF_ECUDA;
  }

  Params p;
  memset(&p, 0, sizeof p);
  p.nphases = 1;
  Phase& ph = p.single;
  ph.kind = PH_ATTN;
  ph.wait_bar = -1;
  ph.signal_bar = -1;
  ph.qbuf = const_cast<void*>(q);
  ph.kc = (uint16_t*)kcache;
  ph.vc = (uint16_t*)vcache;
  ph.attn_out = out;
  ph.Hq = Hq;
  ph.Hkv = Hkv;
  ph.hd = hd;
  ph.Tmax = Tmax;
  ph.stream_cur = 1;
  ph.part = (float*)base;
  ph.tick = (unsigned*)(base + part_bytes);
  // The array keeps the previous call's contents: the combine tickets must
  // start at zero (the partials are always written before they are read).
  GF_CUDA(cudaMemsetAsync(ph.tick, 0, (size_t)Hkv * sizeof(unsigned), (cudaStream_t)stream));
  int CH, nch;
  attn_split(pos + 1, Hkv, sms, CH, nch);
  const int units = Hkv * nch;
  const int grid = units < sms ? units : sms;
  p.nctas = grid;
  p.unit_target = sms;
  p.pos_const = pos;
  p.err = err;
  return launch_engine(p, grid, false, (cudaStream_t)stream);
}

}  // extern "C"
