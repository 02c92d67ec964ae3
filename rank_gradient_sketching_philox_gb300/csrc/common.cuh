// Device helpers shared by the library's kernels: Philox4x32-10, BF16 bit
// handling and stochastic rounding, launch bookkeeping.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sketch.h"

namespace rgs {

// Purpose word (counter word 3) of each Philox stream.
constexpr uint32_t kTagSR = 0u;
constexpr uint32_t kTagRademacher = 1u;
constexpr uint32_t kTagGaussian = 2u;

struct Philox4 {
  uint32_t w0, w1, w2, w3;
};

// Philox4x32-10 of Salmon, Moraes, Dror and Shaw ("Parallel random numbers:
// as easy as 1, 2, 3", SC'11): ten rounds of the two-multiplier S-box with a
// Weyl key schedule; the key is bumped before every round but the first.
__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;  // one wide multiply gives both halves
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t lo0 = (uint32_t)p0, hi0 = (uint32_t)(p0 >> 32);
    const uint32_t lo1 = (uint32_t)p1, hi1 = (uint32_t)(p1 >> 32);
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    const uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return Philox4{c0, c1, c2, c3};
}

// Philox4x32-10 with the round keys taken from a table (rk0[i] = k0 + i*W0,
// rk1[i] = k1 + i*W1, filled on the host): when the table lives in a kernel's
// parameters, each round's XOR reads its key straight from the constant bank.
__device__ __forceinline__ Philox4 philox4x32_10_rk(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                    const uint32_t* rk0, const uint32_t* rk1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ rk0[round];
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ rk1[round];
    c1 = (uint32_t)p1;
    c3 = (uint32_t)p0;
    c0 = n0;
    c2 = n2;
  }
  return Philox4{c0, c1, c2, c3};
}

// philox4x32_10_rk for NB counters (blk[b], c1, c2, c3) that differ only in
// the first word, computed round by round across the blocks so that their
// independent chains interleave.  The first round's product of c2 is the same
// for every block and is formed once.
template <int NB>
__device__ __forceinline__ void philox4x32_10_rk_multi(const uint32_t (&blk)[NB], uint32_t c1, uint32_t c2,
                                                       uint32_t c3, const uint32_t* rk0, const uint32_t* rk1,
                                                       uint32_t (&out)[NB][4]) {
  const uint64_t q = (uint64_t)0xCD9E8D57u * c2;
  const uint32_t n0 = (uint32_t)(q >> 32) ^ c1 ^ rk0[0];
  uint32_t x0[NB], x1[NB], x2[NB], x3[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * blk[b];
    x0[b] = n0;
    x1[b] = (uint32_t)q;
    x2[b] = (uint32_t)(p0 >> 32) ^ c3 ^ rk1[0];
    x3[b] = (uint32_t)p0;
  }
#pragma unroll
  for (int round = 1; round < 10; ++round) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const uint64_t p0 = (uint64_t)0xD2511F53u * x0[b];
      const uint64_t p1 = (uint64_t)0xCD9E8D57u * x2[b];
      const uint32_t m0 = (uint32_t)(p1 >> 32) ^ x1[b] ^ rk0[round];
      const uint32_t m2 = (uint32_t)(p0 >> 32) ^ x3[b] ^ rk1[round];
      x1[b] = (uint32_t)p1;
      x3[b] = (uint32_t)p0;
      x0[b] = m0;
      x2[b] = m2;
    }
  }
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    out[b][0] = x0[b];
    out[b][1] = x1[b];
    out[b][2] = x2[b];
    out[b][3] = x3[b];
  }
}

// Round-key table of philox4x32_10_rk for a 64-bit seed.
__host__ __device__ inline void philox_round_keys(uint64_t seed, uint32_t* rk0, uint32_t* rk1) {
  uint32_t a = (uint32_t)(seed & 0xFFFFFFFFull), b = (uint32_t)(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    rk0[i] = a;
    rk1[i] = b;
    a += 0x9E3779B9u;
    b += 0xBB67AE85u;
  }
}

// acc + lo*lo + hi*hi for the two BF16 halves of w (low half first), each step
// one fused multiply-add with BF16 multiplicands (exact products, one rounding),
// so no unpacking to fp32 first.
__device__ __forceinline__ float sq_acc_bf16x2(uint32_t w, float acc) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "fma.rn.f32.bf16 %0, lo, lo, %0;\n\t"
      "fma.rn.f32.bf16 %0, hi, hi, %0;\n\t}"
      : "+f"(acc)
      : "r"(w));
  return acc;
}

// min of a, b and c that returns NaN when any is NaN (PTX three-input min.NaN).
__device__ __forceinline__ float fmin3_nan(float a, float b, float c) {
  float r;
  asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Integer multiply-adds (the multiplier pipe, leaving the ALU pipe to the rest):
// mad_lo = low 32 bits of a*b + c, mad_hi = high 32 bits of a*b, plus c.
__device__ __forceinline__ uint32_t mad_lo(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t mad_hi(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// min of a and b that returns NaN when either is NaN (PTX min.NaN).
__device__ __forceinline__ float fmin_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Block `block` of the stream (seed, layer, step, tag).
__device__ __forceinline__ Philox4 stream_block(uint64_t seed, uint32_t layer, uint32_t step,
                                                uint32_t tag, uint32_t block) {
  return philox4x32_10(block, step, layer, tag, (uint32_t)(seed & 0xFFFFFFFFull),
                       (uint32_t)(seed >> 32));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) {
  return __uint_as_float(h << 16);
}

// Stochastic rounding of v to BF16 with 16 random bits: add them below the
// kept mantissa and truncate, so the magnitude rounds up with probability
// (dropped bits) / 2^16.  NaN becomes the canonical quiet NaN.
__device__ __forceinline__ uint32_t sr_bf16_bits(float v, uint32_t rand16) {
  const uint32_t b = __float_as_uint(v);
  const uint32_t r = (b + rand16) >> 16;
  return (v != v) ? 0x7FC0u : r;
}

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) {
  return (a + b - 1) / b;
}

}  // namespace rgs
