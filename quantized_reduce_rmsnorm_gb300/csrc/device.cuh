// device.cuh -- device helpers shared by the libfcomm kernels (sm_103a).
//
// Data movement: 256-bit (v8.u32) global loads/stores, a Blackwell addition,
// so one warp instruction moves 1 KB of contiguous data; streamed inputs are
// read through the non-coherent path without L1 allocation and streamed
// outputs are written with the evict-first (.cs) policy.
//
// Arithmetic that must be bit-identical to the definition (quantizer,
// dequantizer, fixed-order sum, residual add) uses the explicit round-to-
// nearest intrinsics (__fmul_rn, __fadd_rn, IEEE division and the RNE
// float->int conversion), which the compiler never contracts into FMA.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fc {

constexpr int kMaxP = 8;
constexpr unsigned kFull = 0xFFFFFFFFu;

struct V8 {
  uint32_t w[8];
};

// ----------------------------------------------------------- global I/O --
__device__ __forceinline__ V8 ld256_stream(const void* p) {
  V8 r;
  asm("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
        "=r"(r.w[6]), "=r"(r.w[7])
      : "l"(p));
  return r;
}

// Cached load for data every CTA re-reads (gamma).
__device__ __forceinline__ V8 ld256_keep(const void* p) {
  V8 r;
  asm("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
        "=r"(r.w[6]), "=r"(r.w[7])
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld128_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ld64_stream(const void* p) {
  uint2 r;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ float ldf_stream(const float* p) {
  float r;
  asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint16_t ld16(const void* p) {
  return *reinterpret_cast<const uint16_t*>(p);
}

__device__ __forceinline__ void st256(void* p, const V8& v) {
  asm volatile("st.global.cs.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
               "r"(v.w[7])
               : "memory");
}

__device__ __forceinline__ void st128(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st64(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void stf(float* p, float v) {
  asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// ----------------------------------------------------------------- bf16 --
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats -> two bf16 (round to nearest even) in one 32-bit word, lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}

// 16 bf16 (one V8) -> 16 floats
__device__ __forceinline__ void unpack16(const V8& v, float f[16]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf_lo(v.w[i]);
    f[2 * i + 1] = bf_hi(v.w[i]);
  }
}

// ------------------------------------------------------- code unpacking --
// INT8 code k of a 32-bit word, as float (exact).
__device__ __forceinline__ float i8_at(uint32_t w, int k) {
  return __int2float_rn(static_cast<int>(static_cast<int8_t>((w >> (8 * k)) & 0xFFu)));
}

// INT4 code k (0..7) of a 32-bit word, as float (exact): the code is placed
// in the mantissa of 2^23 and 2^23 is subtracted.
__device__ __forceinline__ float u4_at(uint32_t w, int k) {
  return __uint_as_float(0x4B000000u | ((w >> (4 * k)) & 0xFu)) - 8388608.0f;
}

// ------------------------------------------------------- group reductions --
// Reductions across the `lpg` lanes (a power of two, 1..32) holding one group.
// Every lane of the warp must call these (inactive lanes with neutral data).
__device__ __forceinline__ float group_max(float v, int lpg) {
  for (int m = 1; m < lpg; m <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
  return v;
}
__device__ __forceinline__ float group_min(float v, int lpg) {
  for (int m = 1; m < lpg; m <<= 1) v = fminf(v, __shfl_xor_sync(kFull, v, m));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
  return v;
}

// ------------------------------------------------------------ quantizers --
// INT8 symmetric on this lane's 16 values of a group spread over lpg lanes.
// Writes the 16 codes packed in q[4] and returns the group's scale.
//   s = max|x| / 127;  q = clamp(rne(x / s), -127, 127);  s == 0 -> q = 0.
__device__ __forceinline__ float quant_i8_lane(const float v[16], int lpg, uint32_t q[4]) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(v[i]));
  a = group_max(a, lpg);
  const float s = __fdiv_rn(a, 127.0f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      int c = 0;
      if (s != 0.0f) {
        c = __float2int_rn(__fdiv_rn(v[4 * j + k], s));
        c = max(-127, min(127, c));
      }
      w |= (static_cast<uint32_t>(c) & 0xFFu) << (8 * k);
    }
    q[j] = w;
  }
  return s;
}

// INT4 asymmetric: lo = min, hi = max (a zero extreme taken as +0),
// s = (hi - lo) / 15, z = lo, q = clamp(rne((x - lo) / s), 0, 15).
// Element 2i in the low nibble of byte i.  Returns s, writes z.
__device__ __forceinline__ float quant_i4_lane(const float v[16], int lpg, uint32_t q[2],
                                               float& z) {
  float lo = v[0], hi = v[0];
#pragma unroll
  for (int i = 1; i < 16; ++i) {
    lo = fminf(lo, v[i]);
    hi = fmaxf(hi, v[i]);
  }
  lo = group_min(lo, lpg);
  hi = group_max(hi, lpg);
  if (lo == 0.0f) lo = 0.0f;  // -0 -> +0
  if (hi == 0.0f) hi = 0.0f;
  const float s = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
  z = lo;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      int c = 0;
      if (s != 0.0f) {
        c = __float2int_rn(__fdiv_rn(__fsub_rn(v[8 * j + k], lo), s));
        c = max(0, min(15, c));
      }
      w |= static_cast<uint32_t>(c) << (4 * k);
    }
    q[j] = w;
  }
  return s;
}

// Dequantizers: d = q * s (INT8), d = q * s + z (INT4; multiply, then add).
__device__ __forceinline__ void dequant_i8_lane(const uint32_t q[4], float s, float d[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) d[i] = __fmul_rn(i8_at(q[i >> 2], i & 3), s);
}
__device__ __forceinline__ void dequant_i4_lane(const uint32_t q[2], float s, float z,
                                                float d[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) d[i] = __fadd_rn(__fmul_rn(u4_at(q[i >> 3], i & 7), s), z);
}

}  // namespace fc
