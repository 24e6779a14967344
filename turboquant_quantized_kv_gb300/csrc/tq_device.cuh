// Device helpers shared by the libtq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq.h"

namespace tq {

constexpr int kD = TQ_HEAD_DIM;       // 128
constexpr int kBlock = TQ_BLOCK_SIZE;  // 16

// Tables of one codebook passed by value to kernels (constant bank).
struct Codebook {
  float c[16];
  float b[15];
};

__device__ __forceinline__ void flag_status(unsigned* status, unsigned bits) {
  if (status) atomicOr(status, bits);
}

// prmt.b32 with the full selector semantics (bit 3 of a selector nibble
// replicates the sign bit of the selected byte).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

template <typename T>
__device__ __forceinline__ float load_elem(const T* p);
template <>
__device__ __forceinline__ float load_elem<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void store_elem(T* p, float v);
template <>
__device__ __forceinline__ void store_elem<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_elem<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Loads 32 consecutive elements starting at p (16-byte aligned) into fp32 registers.
template <typename T>
__device__ __forceinline__ void load32(const T* p, float (&x)[32]);
template <>
__device__ __forceinline__ void load32<float>(const float* p, float (&x)[32]) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4 v = __ldg(q + i);
    x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
  }
}
template <>
__device__ __forceinline__ void load32<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[32]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 v = __ldg(q + i);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
      x[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
}

// Unnormalised Walsh-Hadamard transform of 128 values spread over the 4
// consecutive lanes of a quad (lane q holds coordinates [32q, 32q + 32)):
// 5 butterfly stages inside the registers, 2 across lanes.
__device__ __forceinline__ void fwht128_quad(float (&x)[32], int q) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & h) == 0) {
        float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
    }
  }
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    const bool upper = (q & m) != 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float o = __shfl_xor_sync(0xffffffffu, x[i], m);
      x[i] = upper ? (o - x[i]) : (x[i] + o);
    }
  }
}

// The same transform with packed fp32 pairs (sm_100+ f32x2 arithmetic): bit 0 of
// the coordinate inside each pair, bits 1..4 as pair butterflies, bits 5 and 6
// across the quad as x <- partner + s x with s = -1 on the upper lane.
__device__ __forceinline__ void fwht128_quad_f2(float (&x)[32], int q) {
  float2 v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = make_float2(x[2 * j] + x[2 * j + 1], x[2 * j] - x[2 * j + 1]);
  const float2 m1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if ((j & h) == 0) {
        const float2 a = v[j], b = v[j + h];
        v[j] = __fadd2_rn(a, b);
        v[j + h] = __ffma2_rn(b, m1, a);
      }
    }
  }
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    const float sgn = (q & m) ? -1.0f : 1.0f;
    const float2 s2 = make_float2(sgn, sgn);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, v[j].x, m), __shfl_xor_sync(0xffffffffu, v[j].y, m));
      v[j] = __ffma2_rn(v[j], s2, o);
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    x[2 * j] = v[j].x;
    x[2 * j + 1] = v[j].y;
  }
}

__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  return v;
}

// Magnitude count #{k : P_k <= a} over the positive boundaries
// P_k = b[2^(B-1) + k], k < 2^(B-1) - 1, by an unrolled binary search.
template <int BITS>
__device__ __forceinline__ int pos_count(float a, const Codebook& cb) {
  constexpr int H = 1 << (BITS - 1);
  if constexpr (BITS == 2) {
    return a >= cb.b[H] ? 1 : 0;
  } else if constexpr (BITS == 3) {
    const bool c1 = a >= cb.b[H + 1];
    const float t = c1 ? cb.b[H + 2] : cb.b[H];
    const bool c2 = a >= t;
    return (c1 ? 2 : 0) + (c2 ? 1 : 0);
  } else {
    const bool c1 = a >= cb.b[H + 3];
    const float t2 = c1 ? cb.b[H + 5] : cb.b[H + 1];
    const bool c2 = a >= t2;
    const float t3 = c1 ? (c2 ? cb.b[H + 6] : cb.b[H + 4]) : (c2 ? cb.b[H + 2] : cb.b[H]);
    const bool c3 = a >= t3;
    return (c1 ? 4 : 0) + (c2 ? 2 : 0) + (c3 ? 1 : 0);
  }
}

// Code of one rotated coordinate: idx = #{i : y >= beta_i} for an
// antisymmetric boundary table (beta_{2^B-2-i} = -beta_i, middle 0).
// y >= 0: idx = 2^(B-1) + #{P_k <= y}.  y < 0: idx = 2^(B-1) - 1 - #{P_k < |y|},
// and P_k < |y| <=> P_k <= prevfloat(|y|).  Returns the code; *mag gets the
// magnitude index (|c[idx]| = c[2^(B-1) + mag]).
template <int BITS>
__device__ __forceinline__ uint32_t quantize_coord(float y, const Codebook& cb, int* mag) {
  constexpr uint32_t H = 1u << (BITS - 1);
  constexpr uint32_t M = (1u << BITS) - 1u;
  const bool neg = y < 0.0f;
  uint32_t ab = __float_as_uint(y) & 0x7FFFFFFFu;
  ab -= neg ? 1u : 0u;
  const int cnt = pos_count<BITS>(__uint_as_float(ab), cb);
  *mag = cnt;
  return ((H + (uint32_t)cnt) ^ (neg ? M : 0u)) & M;
}

// Packs 32 codes (code k at bits [BITS k, BITS k + BITS)) into BITS words.
template <int BITS>
__device__ __forceinline__ void pack32(const uint32_t (&code)[32], uint32_t (&w)[BITS]) {
  if constexpr (BITS == 4) {  // code pairs to bytes, bytes to words
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t by[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) by[j] = code[8 * k + 2 * j] + (code[8 * k + 2 * j + 1] << 4);
      w[k] = __byte_perm(__byte_perm(by[0], by[1], 0x0040u), __byte_perm(by[2], by[3], 0x0040u), 0x5410u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < BITS; ++i) w[i] = 0u;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int bit = BITS * k;
      w[bit >> 5] |= code[k] << (bit & 31);
      if ((bit & 31) + BITS > 32) w[(bit >> 5) + 1] |= code[k] >> (32 - (bit & 31));
    }
  }
}

}  // namespace tq
