/* Counter-based synthetic-input generator, shared verbatim by the host (C) and
 * device (CUDA) builds of libsynth.so so both produce the same bits.
 *
 * It holds none of the decode step's arithmetic: it only turns
 * (seed, stream, element index) into an input value.
 *
 * Definition (all integer, then two correctly rounded IEEE double operations):
 *   k1..k4 = keys derived from (seed, stream) with fmix32 (MurmurHash3's
 *            32-bit finaliser, a bijection on 32-bit words)
 *   lo, hi = low / high 32 bits of the element index
 *   u1 = fmix32(fmix32(lo ^ k1) ^ hi ^ k2)
 *   u2 = fmix32(fmix32(lo ^ k3) ^ hi ^ k4)
 *   S  = four 16-bit halves of u1, u2 summed     (Irwin-Hall sum of 4 uniforms)
 *   z  = (S - 131070) * scale                      (scale = sigma / sd(S))
 *   value = bf16_rne(float_rn(mean + z))
 * Because u1 (and u2) is a bijection of lo for a fixed hi, every 16-bit half
 * is exactly uniform over any aligned block of 2^32 indices.
 * Uniform integers in [0, n) are (u1 * n) >> 32.
 */
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define SYN_HD __host__ __device__ __forceinline__
#else
#define SYN_HD static inline
#endif

SYN_HD uint32_t syn_fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}

typedef struct { uint32_t k1, k2, k3, k4; } syn_keys;

SYN_HD syn_keys syn_make_keys(uint64_t seed, uint32_t stream) {
  syn_keys k;
  uint32_t s_lo = (uint32_t)seed, s_hi = (uint32_t)(seed >> 32);
  uint32_t base = syn_fmix32(syn_fmix32(s_lo ^ 0x9e3779b9u) ^ s_hi ^ stream);
  k.k1 = syn_fmix32(base ^ 0x243f6a88u);
  k.k2 = syn_fmix32(base ^ 0x85a308d3u);
  k.k3 = syn_fmix32(base ^ 0x13198a2eu);
  k.k4 = syn_fmix32(base ^ 0x03707344u);
  return k;
}

SYN_HD uint32_t syn_u1(syn_keys k, uint64_t i) {
  uint32_t lo = (uint32_t)i, hi = (uint32_t)(i >> 32);
  return syn_fmix32(syn_fmix32(lo ^ k.k1) ^ hi ^ k.k2);
}

SYN_HD uint32_t syn_u2(syn_keys k, uint64_t i) {
  uint32_t lo = (uint32_t)i, hi = (uint32_t)(i >> 32);
  return syn_fmix32(syn_fmix32(lo ^ k.k3) ^ hi ^ k.k4);
}

/* Round a float to bfloat16 bits, round-to-nearest-even (inputs are finite). */
SYN_HD uint16_t syn_f32_to_bf16(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t u = v.u;
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

SYN_HD double syn_dmul(double a, double b) {
#if defined(__CUDA_ARCH__)
  return __dmul_rn(a, b);
#else
  volatile double r = a * b; /* keeps the host from contracting into an FMA */
  return r;
#endif
}

SYN_HD double syn_dadd(double a, double b) {
#if defined(__CUDA_ARCH__)
  return __dadd_rn(a, b);
#else
  volatile double r = a + b;
  return r;
#endif
}

/* Approximately normal bf16 value with the given mean and scale. */
SYN_HD uint16_t syn_normal_bf16(syn_keys k, uint64_t i, double mean, double scale) {
  uint32_t a = syn_u1(k, i), b = syn_u2(k, i);
  int32_t s = (int32_t)((a & 0xffffu) + (a >> 16) + (b & 0xffffu) + (b >> 16)) - 131070;
  double z = syn_dmul((double)s, scale);
  double v = syn_dadd(mean, z);
  return syn_f32_to_bf16((float)v);
}

SYN_HD int32_t syn_uniform_int(syn_keys k, uint64_t i, uint32_t n) {
  return (int32_t)(((uint64_t)syn_u1(k, i) * (uint64_t)n) >> 32);
}
