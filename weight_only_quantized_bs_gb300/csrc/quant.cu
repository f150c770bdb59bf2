// quant.cu — offline weight preparation: int8 and int4 grouped weight-only
// quantisation written straight into the device layout (slots of 32 rows x
// 256 bytes, int4 scale/zero words after each slot's codes), the bf16 repack
// into the same slots, the inverse unpack kernels used for bit-exact layout
// checks, and the column-sliced copy of a down projection for the fused FFN.
//
// Quantisation follows the gpt-fast README, section "Quantization" (int8
// weight-only; int4 weight-only with --groupsize 32 / 64 / 128), read as: int8
// symmetric per output row, s = bf16(max|w| / 127); int4 per row and G-wide K
// group, z = min, s = bf16((max - min) / 15), codes 0..15.  Every quotient is
// an IEEE fp32 division and every rounding to an integer is rint (ties to
// even), so the codes are bit-identical to any IEEE implementation of the
// same steps.
#include "gf_internal.cuh"

namespace gf {

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ int warp_id_global() { return (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); }
__device__ __forceinline__ int warps_total() { return (int)((gridDim.x * blockDim.x) >> 5); }

// int8: one warp per output row; codes [N][K] stored as q + 128.
__global__ void __launch_bounds__(256) k_quant_w8(const uint16_t* __restrict__ W, int N, int K,
                                                  uint8_t* __restrict__ P, uint16_t* __restrict__ S) {
  const int lane = threadIdx.x & 31, C = K / 16;
  for (int n = warp_id_global(); n < N; n += warps_total()) {
    const uint16_t* row = W + (size_t)n * K;
    float mx = 0.0f;
    for (int k = lane; k < K; k += 32) mx = fmaxf(mx, fabsf(bf2f(row[k])));
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const uint16_t sb = f2bf(mx / 127.0f);
    const float sv = bf2f(sb);
    if (lane == 0) S[n] = sb;
    for (int c = lane; c < C; c += 32) {
      const uint4 raw0 = *reinterpret_cast<const uint4*>(row + c * 16);
      const uint4 raw1 = *reinterpret_cast<const uint4*>(row + c * 16 + 8);
      const uint32_t h[8] = {raw0.x, raw0.y, raw0.z, raw0.w, raw1.x, raw1.y, raw1.z, raw1.w};
      uint32_t words[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int k = 4 * j + i;
          const uint16_t wb = (uint16_t)(h[k >> 1] >> ((k & 1) * 16));
          int code = 0;
          if (sv != 0.0f) {
            code = (int)rintf(bf2f(wb) / sv);
            code = max(-127, min(127, code));
          }
          word |= (uint32_t)(code + 128) << (8 * i);  // offset binary
        }
        words[j] = word;
      }
      *reinterpret_cast<uint4*>(P + code_addr(DT_INT8, K, 32, n, (long long)c * 16)) =
          make_uint4(words[0], words[1], words[2], words[3]);
    }
  }
}

// bf16: 16-byte chunks moved into their slots.
__global__ void __launch_bounds__(256) k_repack_bf16(const uint16_t* __restrict__ W, int N, int K,
                                                     uint8_t* __restrict__ P) {
  const int lane = threadIdx.x & 31, C = K / 8;
  for (int n = warp_id_global(); n < N; n += warps_total())
    for (int c = lane; c < C; c += 32)
      *reinterpret_cast<uint4*>(P + code_addr(DT_BF16, K, 32, n, (long long)c * 16)) =
          *reinterpret_cast<const uint4*>(W + (size_t)n * K + c * 8);
}

// int4, group G (a multiple of 32): one warp per output row, one lane per
// group.  Codes two per byte (code 2i low nibble of byte i of the row) and
// the scale/zero word of each (row, group), in their slots.
__global__ void __launch_bounds__(256) k_quant_w4g(const uint16_t* __restrict__ W, int N, int K, int G,
                                                   uint8_t* __restrict__ P) {
  const int lane = threadIdx.x & 31, ng = K / G;
  for (int n = warp_id_global(); n < N; n += warps_total()) {
    const uint16_t* row = W + (size_t)n * K;
    for (int g = lane; g < ng; g += 32) {
      const uint16_t* w = row + (size_t)g * G;
      // running min / max in index order, strict comparisons (so a signed
      // zero is kept exactly as the first one met)
      float mn = bf2f(w[0]), mx = mn;
      for (int i = 1; i < G; ++i) {
        const float v = bf2f(w[i]);
        if (v < mn) mn = v;
        if (v > mx) mx = v;
      }
      const float range = mx - mn;
      const uint16_t sb = f2bf(range / 15.0f);
      const float sv = bf2f(sb);
      const uint16_t zb = f2bf(mn);
      for (int c = 0; c < G; c += 32) {
        uint32_t words[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t word = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            int code = 0;
            if (sv != 0.0f) {
              code = (int)rintf((bf2f(w[c + 8 * j + i]) - mn) / sv);
              code = max(0, min(15, code));
            }
            word |= (uint32_t)code << (4 * i);
          }
          words[j] = word;
        }
        *reinterpret_cast<uint4*>(P + code_addr(DT_INT4, K, G, n, ((long long)g * G + c) / 2)) =
            make_uint4(words[0], words[1], words[2], words[3]);
      }
      *reinterpret_cast<uint32_t*>(P + sz_addr(K, G, n, g)) = (uint32_t)sb | ((uint32_t)zb << 16);
    }
  }
}

// device layout -> logical (for layout checks)
__global__ void __launch_bounds__(256) k_unpack(int dt, const uint8_t* __restrict__ P, int N, int K, int G,
                                                void* __restrict__ Q, uint16_t* __restrict__ S, uint16_t* __restrict__ Z) {
  const int lane = threadIdx.x & 31, E = per_chunk(dt), C = K / E;
  for (int n = warp_id_global(); n < N; n += warps_total()) {
    for (int c = lane; c < C; c += 32) {
      const uint4 v = *reinterpret_cast<const uint4*>(P + code_addr(dt, K, G, n, (long long)c * 16));
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      if (dt == DT_BF16) {
        *reinterpret_cast<uint4*>((uint16_t*)Q + (size_t)n * K + c * 8) = v;
      } else if (dt == DT_INT8) {  // offset binary back to two's complement
        *reinterpret_cast<uint4*>((uint8_t*)Q + (size_t)n * K + c * 16) =
            make_uint4(v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u);
      } else {
        uint8_t* q = (uint8_t*)Q + (size_t)n * K + c * 32;
        for (int j = 0; j < 4; ++j) {
          for (int i = 0; i < 8; ++i) q[8 * j + i] = (uint8_t)((wv[j] >> (4 * i)) & 15u);
        }
      }
    }
    if (dt == DT_INT4) {
      for (int g = lane; g < K / G; g += 32) {
        const uint32_t sz = *reinterpret_cast<const uint32_t*>(P + sz_addr(K, G, n, g));
        S[(size_t)n * (K / G) + g] = (uint16_t)sz;
        Z[(size_t)n * (K / G) + g] = (uint16_t)(sz >> 16);
      }
    }
  }
}

static int check_w(const char* fn, int dt, const void* W, int N, int K) {
  if (!W || N <= 0 || K <= 0 || K % per_chunk(dt) || K > KMAX * 64) {
    set_error("%s: bad arguments (N=%d, K=%d; K must be a multiple of %d)", fn, N, K, per_chunk(dt));
    return GF_EINVAL;
  }
  if (!aligned16(W)) {
    set_error("%s: pointers must be 16-byte aligned", fn);
    return GF_EALIGN;
  }
  return GF_OK;
}

static bool group_ok(int G, int K) { return (G == 32 || G == 64 || G == 128) && K % G == 0; }

static int grid_for_rows(int N) {
  int sms = device_sms();
  int blocks = (N + 7) / 8;
  return blocks < sms * 16 ? blocks : sms * 16;
}

// Quantises (or repacks) W [N][K] into `packed` (packed_bytes bytes, already
// zeroed: the padding of ragged tiles and K-slots must read as zero); int8
// row scales into s8.
int quantize_rows(int dt, const void* W, int N, int K, int G, void* packed, void* s8, cudaStream_t s) {
  if (dt == DT_BF16) {
    k_repack_bf16<<<grid_for_rows(N), 256, 0, s>>>((const uint16_t*)W, N, K, (uint8_t*)packed);
  } else if (dt == DT_INT8) {
    k_quant_w8<<<grid_for_rows(N), 256, 0, s>>>((const uint16_t*)W, N, K, (uint8_t*)packed, (uint16_t*)s8);
  } else {
    k_quant_w4g<<<grid_for_rows(N), 256, 0, s>>>((const uint16_t*)W, N, K, G, (uint8_t*)packed);
  }
  GF_CUDA(cudaGetLastError());
  return GF_OK;
}

// Column-sliced copy of a matrix in the device layout, for a down projection
// fused behind its gate/up GEMV.  int4: per group of 32 columns, the rows'
// 8 code bytes of columns 0..15, then of columns 16..31, then the rows'
// scale/zero words (of the group that holds those columns); int8: per 16
// columns, the rows' 16 code bytes; bf16: per 16 columns, the rows' first 8
// values (16 bytes), then their last 8.  One thread per (row, 16 columns).
__global__ void __launch_bounds__(256) k_pack_cols(int dt, const uint8_t* __restrict__ P, int N, int K, int G,
                                                   uint8_t* __restrict__ out) {
  const int nsl = K / 16;
  const long long total = (long long)N * nsl;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(i % N), j = (int)(i / N);
    if (dt == DT_INT4) {
      const uint2 w = *reinterpret_cast<const uint2*>(P + code_addr(DT_INT4, K, G, n, (long long)j * 8));
      uint8_t* g = out + (size_t)(j >> 1) * N * 20;
      *reinterpret_cast<uint2*>(g + (size_t)(j & 1) * N * 8 + (size_t)n * 8) = w;
      if ((j & 1) == 0)
        *reinterpret_cast<uint32_t*>(g + (size_t)N * 16 + (size_t)n * 4) =
            *reinterpret_cast<const uint32_t*>(P + sz_addr(K, G, n, 16 * j / G));
    } else if (dt == DT_INT8) {
      *reinterpret_cast<uint4*>(out + ((size_t)j * N + n) * 16) =
          *reinterpret_cast<const uint4*>(P + code_addr(DT_INT8, K, 32, n, (long long)j * 16));
    } else {
      uint8_t* o = out + (size_t)j * N * 32;
      *reinterpret_cast<uint4*>(o + (size_t)n * 16) =
          *reinterpret_cast<const uint4*>(P + code_addr(DT_BF16, K, 32, n, (long long)j * 32));
      *reinterpret_cast<uint4*>(o + (size_t)N * 16 + (size_t)n * 16) =
          *reinterpret_cast<const uint4*>(P + code_addr(DT_BF16, K, 32, n, (long long)j * 32 + 16));
    }
  }
}

long long cols_bytes(int dt, int N, int K) {
  return dt == DT_INT4 ? (long long)(K / 32) * N * 20 : (long long)(K / 16) * N * (dt == DT_INT8 ? 16 : 32);
}

int pack_cols(int dt, const void* packed, int N, int K, int G, void* out, cudaStream_t s) {
  if (K % 32 || N <= 0) {
    set_error("column-sliced copy: K must be a multiple of 32 (got %d)", K);
    return GF_EINVAL;
  }
  const long long total = (long long)N * (K / 16);
  const int blocks = (int)((total + 255) / 256 < 65535 ? (total + 255) / 256 : 65535);
  k_pack_cols<<<blocks, 256, 0, s>>>(dt, (const uint8_t*)packed, N, K, G, (uint8_t*)out);
  GF_CUDA(cudaGetLastError());
  return GF_OK;
}

}  // namespace gf

using namespace gf;

extern "C" {

long long gf_packed_bytes_w4g(int N, int K, int G) {
  if (N <= 0 || K <= 0 || K % 32 || !group_ok(G, K)) return -1;
  return packed_bytes(DT_INT4, N, K, G);
}

int gf_quantize_w8(const void* W, int N, int K, void* packed, void* s, gf_stream stream) {
  int rc = check_w("gf_quantize_w8", DT_INT8, W, N, K);
  if (rc) return rc;
  if (!packed || !s) { set_error("gf_quantize_w8: null output"); return GF_EINVAL; }
  if (!aligned16(packed) || !aligned16(s)) { set_error("gf_quantize_w8: outputs must be 16-byte aligned"); return GF_EALIGN; }
  GF_CUDA(cudaMemsetAsync(packed, 0, (size_t)packed_bytes(DT_INT8, N, K, 32), (cudaStream_t)stream));
  return quantize_rows(DT_INT8, W, N, K, 32, packed, s, (cudaStream_t)stream);
}

int gf_quantize_w4g(const void* W, int N, int K, int G, void* packed, gf_stream stream) {
  int rc = check_w("gf_quantize_w4g", DT_INT4, W, N, K);
  if (rc) return rc;
  if (!group_ok(G, K)) {
    set_error("gf_quantize_w4g: group size must be 32, 64 or 128 and divide K (G=%d, K=%d)", G, K);
    return GF_EUNSUPPORTED;
  }
  if (!packed) { set_error("gf_quantize_w4g: null output"); return GF_EINVAL; }
  if (!aligned16(packed)) { set_error("gf_quantize_w4g: output must be 16-byte aligned"); return GF_EALIGN; }
  GF_CUDA(cudaMemsetAsync(packed, 0, (size_t)packed_bytes(DT_INT4, N, K, G), (cudaStream_t)stream));
  return quantize_rows(DT_INT4, W, N, K, G, packed, nullptr, (cudaStream_t)stream);
}

int gf_repack_bf16(const void* W, int N, int K, void* packed, gf_stream stream) {
  int rc = check_w("gf_repack_bf16", DT_BF16, W, N, K);
  if (rc) return rc;
  if (!packed) { set_error("gf_repack_bf16: null output"); return GF_EINVAL; }
  if (!aligned16(packed)) { set_error("gf_repack_bf16: output must be 16-byte aligned"); return GF_EALIGN; }
  GF_CUDA(cudaMemsetAsync(packed, 0, (size_t)packed_bytes(DT_BF16, N, K, 32), (cudaStream_t)stream));
  return quantize_rows(DT_BF16, W, N, K, 32, packed, nullptr, (cudaStream_t)stream);
}

static int unpack_common(const char* fn, int dt, const void* packed, int N, int K, int G, void* q, void* s, void* z,
                         gf_stream stream) {
  int rc = check_w(fn, dt, packed, N, K);
  if (rc) return rc;
  if (!q || (dt == DT_INT4 && (!s || !z))) { set_error("%s: null output", fn); return GF_EINVAL; }
  if (!aligned16(q)) { set_error("%s: outputs must be 16-byte aligned", fn); return GF_EALIGN; }
  k_unpack<<<grid_for_rows(N), 256, 0, (cudaStream_t)stream>>>(dt, (const uint8_t*)packed, N, K, G, q, (uint16_t*)s,
                                                                 (uint16_t*)z);
  GF_CUDA(cudaGetLastError());
  return GF_OK;
}

int gf_unpack_w8(const void* packed, int N, int K, void* q, gf_stream stream) {
  return unpack_common("gf_unpack_w8", DT_INT8, packed, N, K, 32, q, nullptr, nullptr, stream);
}
int gf_unpack_w4g(const void* packed, int N, int K, int G, void* q, void* s, void* z, gf_stream stream) {
  if (!group_ok(G, K)) {
    set_error("gf_unpack_w4g: group size must be 32, 64 or 128 and divide K (G=%d, K=%d)", G, K);
    return GF_EUNSUPPORTED;
  }
  return unpack_common("gf_unpack_w4g", DT_INT4, packed, N, K, G, q, s, z, stream);
}
int gf_unpack_bf16(const void* packed, int N, int K, void* W, gf_stream stream) {
  return unpack_common("gf_unpack_bf16", DT_BF16, packed, N, K, 32, W, nullptr, nullptr, stream);
}

}  // extern "C"
