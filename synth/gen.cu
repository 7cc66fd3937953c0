// libsynth: fills seeded synthetic inputs (weights, tokens, paged KV) on the
// host (OpenMP) or on the device (CUDA), from the one definition in gen.h.
// Input preparation only: nothing here computes any part of the decode step.
#include <cuda_runtime.h>
#include <stdint.h>
#include "gen.h"

namespace {

__global__ void k_fill_normal(uint16_t* out, int64_t n, syn_keys k, int64_t start,
                              double mean, double scale) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (; i < n; i += stride) out[i] = syn_normal_bf16(k, (uint64_t)(start + i), mean, scale);
}

__global__ void k_fill_uniform(int32_t* out, int64_t n, syn_keys k, int64_t start, uint32_t hi) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (; i < n; i += stride) out[i] = syn_uniform_int(k, (uint64_t)(start + i), hi);
}

// Element (pos, g, e) of a request's logical [n_tok, nkv, d] cache goes to
// row e, slot pos % ps of block (page_table[pos / ps], g): each page holds its
// head's [d, page_size] block transposed (one row per dimension), the blocks
// `hs` elements apart (d * ps when the pool holds one kind, 2 * d * ps for
// the K or V half of an interleaved pool).
__global__ void k_fill_kv_paged(uint16_t* pool, const int32_t* page_table, int64_t n_tok, int nkv,
                                int ps, int d, int64_t hs, syn_keys k, double scale) {
  int64_t n = n_tok * nkv * d;
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (; i < n; i += stride) {
    int64_t e = i % d;
    int64_t g = (i / d) % nkv;
    int64_t pos = i / ((int64_t)d * nkv);
    int64_t page = page_table[pos / ps];
    int64_t dst = (page * nkv + g) * hs + e * ps + pos % ps;
    pool[dst] = syn_normal_bf16(k, (uint64_t)i, 0.0, scale);
  }
}

int grid_for(int64_t n) {
  int64_t b = (n + 255) / 256;
  if (b > 152 * 64) b = 152 * 64;
  if (b < 1) b = 1;
  return (int)b;
}

}  // namespace

extern "C" {

// Returns 0 on success, a cudaError_t value otherwise.
int synth_fill_normal_bf16(void* out, int64_t n, uint64_t seed, uint32_t stream, int64_t start,
                           double mean, double scale, int on_device, void* cuda_stream) {
  syn_keys k = syn_make_keys(seed, stream);
  uint16_t* o = (uint16_t*)out;
  if (n <= 0) return 0;
  if (on_device) {
    k_fill_normal<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(o, n, k, start, mean, scale);
    return (int)cudaGetLastError();
  }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) o[i] = syn_normal_bf16(k, (uint64_t)(start + i), mean, scale);
  return 0;
}

int synth_fill_uniform_int(int32_t* out, int64_t n, uint64_t seed, uint32_t stream, int64_t start,
                           uint32_t hi, int on_device, void* cuda_stream) {
  syn_keys k = syn_make_keys(seed, stream);
  if (n <= 0) return 0;
  if (on_device) {
    k_fill_uniform<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(out, n, k, start, hi);
    return (int)cudaGetLastError();
  }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = syn_uniform_int(k, (uint64_t)(start + i), hi);
  return 0;
}

// page_table: n_pages_used entries covering positions [0, n_tok); device pointer
// when on_device, host pointer otherwise.  Pool layout [pages][nkv][d][page_size]
// with the (page, head) blocks head_stride elements apart.
int synth_fill_kv_paged(void* pool, const int32_t* page_table, int64_t n_tok, int nkv, int page_size,
                        int d, int64_t head_stride, uint64_t seed, uint32_t stream, double scale,
                        int on_device, void* cuda_stream) {
  syn_keys k = syn_make_keys(seed, stream);
  uint16_t* p = (uint16_t*)pool;
  int64_t n = n_tok * nkv * d;
  if (n <= 0) return 0;
  if (on_device) {
    k_fill_kv_paged<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(p, page_table, n_tok, nkv,
                                                                         page_size, d, head_stride, k, scale);
    return (int)cudaGetLastError();
  }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    int64_t e = i % d;
    int64_t g = (i / d) % nkv;
    int64_t pos = i / ((int64_t)d * nkv);
    int64_t page = page_table[pos / page_size];
    p[(page * nkv + g) * head_stride + e * page_size + pos % page_size] =
        syn_normal_bf16(k, (uint64_t)i, 0.0, scale);
  }
  return 0;
}

}  // extern "C"
