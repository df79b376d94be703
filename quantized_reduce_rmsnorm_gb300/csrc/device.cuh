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

#include <type_traits>

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

// Streamed load on the coherent path (for a tensor the kernel may also
// write, e.g. a residual that aliases residual_out), without L1 allocation.
__device__ __forceinline__ V8 ld256_coherent(const void* p) {
  V8 r;
  asm volatile("ld.global.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
                 "=r"(r.w[6]), "=r"(r.w[7])
               : "l"(p)
               : "memory");
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

// Single words and bytes on the coherent path, for a warp patching codes it
// stored earlier in the same kernel: ld_u32 for a word the thread stored
// itself (program order), ld_u32_l2 for one another lane of the warp stored
// (read from L2, after a warp barrier).
__device__ __forceinline__ uint32_t ld_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_u32_l2(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_u8(uint8_t* p, uint32_t v) {
  asm volatile("st.global.u8 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void stf(float* p, float v) {
  asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// --------------------------------------------- TMA bulk copies, mbarrier --
// 1-D bulk copies (cp.async.bulk, the TMA engine without a tensor map) from
// this GPU's global memory into the CTA's own shared memory; completion is
// counted in bytes on an mbarrier.  No multicast.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for phase `parity` of the barrier, giving up after ~2^31 clock
// cycles (about a second): returns false then, so no wait can hang the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > (1ll << 31)) return false;
  return true;
}

// --------------------------------------------- programmatic dependent launch --
// Every kernel here is launched with programmatic stream serialization
// (launch_pdl): it may be scheduled while the previous kernel in its stream
// is still finishing.  pdl_begin() waits until that previous kernel has
// completed and its writes are visible (griddepcontrol.wait; a no-op for a
// launch without the attribute).  No global memory is read or written
// before it; the only thing a kernel may issue earlier is prefetch_l2 of its
// first tiles (below), which returns no data.  pdl_begin() then lets the next
// kernel in the stream be scheduled as resources free up
// (griddepcontrol.launch_dependents).
// A dependent grid is scheduled only once every CTA of this grid has issued
// that instruction (or finished), i.e. has started, so its CTAs never hold a
// slot that a CTA of this grid still needs in order to start.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Asks the TMA engine to bring [p, p + bytes) into L2 (cp.async.bulk.prefetch;
// p and bytes multiples of 16).  Nothing comes back to the SM.  The staged
// kernels issue it for their first tiles before pdl_begin(), so those tiles'
// DRAM latency overlaps the tail of the previous kernel in the stream (whose
// last CTAs are still running when this kernel's first CTAs become resident).
// It cannot make a later load see stale data: the loads that use the data
// are issued after pdl_begin(), when the previous kernel's writes are visible,
// and L2, which serves them, is this GPU's point of coherence for global
// memory -- a line prefetched before a write is updated by that write.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
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

// Mixed-precision arithmetic (sm_100 and later): one operand is the bf16 in
// the low or high half of a 32-bit word, converted exactly to binary32 inside
// the instruction, so the result is the same single IEEE rounding as the
// binary32 operation on the unpacked value, without the unpacking.
//   add_bf_{lo,hi}(w, c)     = fl(bf16(w) + c)
//   fma_bf_{lo,hi}(w, g, c)  = fl(bf16(w) * bf16(g) + c)   (both halves alike)
__device__ __forceinline__ float add_bf_lo(uint32_t w, float c) {
  float d;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n add.rn.f32.bf16 %0, l, %2;\n}"
      : "=f"(d) : "r"(w), "f"(c));
  return d;
}
__device__ __forceinline__ float add_bf_hi(uint32_t w, float c) {
  float d;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n add.rn.f32.bf16 %0, h, %2;\n}"
      : "=f"(d) : "r"(w), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_bf_lo(uint32_t w, uint32_t g, float c) {
  float d;
  asm("{\n .reg .b16 l, h, gl, gh;\n mov.b32 {l, h}, %1;\n mov.b32 {gl, gh}, %2;\n"
      " fma.rn.f32.bf16 %0, l, gl, %3;\n}"
      : "=f"(d) : "r"(w), "r"(g), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_bf_hi(uint32_t w, uint32_t g, float c) {
  float d;
  asm("{\n .reg .b16 l, h, gl, gh;\n mov.b32 {l, h}, %1;\n mov.b32 {gl, gh}, %2;\n"
      " fma.rn.f32.bf16 %0, h, gh, %3;\n}"
      : "=f"(d) : "r"(w), "r"(g), "f"(c));
  return d;
}

// Three-input minimum / maximum (sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// -------------------------------------------------- packed fp32 pairs --
// Blackwell issues two binary32 operations per instruction on a register
// pair (.f32x2); each half is an IEEE round-to-nearest operation.  The
// compiler may fuse a packed multiply whose product has one use with a
// following packed add into one fused multiply-add, so a packed multiply is
// used only where that cannot change a result (the tolerance-checked RMSNorm
// output).  Packed adds and packed fused multiply-adds cannot be contracted
// any further, so exact chains are written with them: a product that must be
// rounded on its own is formed as fma(2^23 + q, s, -2^23 * s), whose exact
// value is q * s (see the dequantizers).
__device__ __forceinline__ float2 padd(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 psub(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " sub.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 pmul(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 pfma(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
__device__ __forceinline__ float2 dup2(float a) { return make_float2(a, a); }

// ------------------------------------------------------- code unpacking --
// Codes become floats without an int->float conversion: the code is placed
// in the low mantissa bits of 2^23 with a byte permute and 2^23 (+128 for the
// sign-flipped INT8 bytes) is subtracted; both steps are exact.
constexpr float kTwo23 = 8388608.0f;            // 2^23, bits 0x4B000000
constexpr float kTwo23p128 = 8388736.0f;        // 2^23 + 128
constexpr uint32_t kTwo23Bits = 0x4B000000u;

// The same for a byte selector known at compile time, kept opaque to the
// compiler: measured on GB300 (executed-instruction counts), the INT4
// dequantizer issues 51 instead of 70 instructions per 16 codes when its
// byte permutes and nibble masks are written this way, all permutes of a
// word first and the packed arithmetic after.
template <int SEL>
__device__ __forceinline__ float prmt_two23(uint32_t a) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0x4B000000, %2;" : "=r"(r) : "r"(a), "n"(SEL));
  return __uint_as_float(r);
}
// The eight 4-bit codes of w spread one per byte: codes 0, 2, 4, 6 in ev,
// codes 1, 3, 5, 7 in od.
__device__ __forceinline__ void spread_nibbles(uint32_t w, uint32_t& ev, uint32_t& od) {
  asm("{\n .reg .b32 t;\n and.b32 %0, %2, 0x0F0F0F0F;\n shr.u32 t, %2, 4;\n and.b32 %1, t, 0x0F0F0F0F;\n}"
      : "=r"(ev), "=r"(od) : "r"(w));
}

// byte k of w as the low byte of 2^23's bit pattern
__device__ __forceinline__ float byte_in_two23(uint32_t w, int k) {
  return __uint_as_float(__byte_perm(w, kTwo23Bits, 0x7540u | static_cast<uint32_t>(k)));
}

// acc[i] += q_i * s for the 16 INT8 codes in w[4] (code i = byte i%4 of w[i/4]).
// With b = q + 128 (exact, from the sign-flipped byte in the low bits of
// 2^23), fma(b, s, -128 * s) has the exact value q * s and rounds it once, so
// it equals fl(q * s) (for s < 2^100, where 128 * s is exact and finite;
// larger scales take the plain product).  Packed in pairs.
__device__ __forceinline__ void dequant_i8_acc(const uint32_t w[4], float s, float acc[16]) {
  if (s < 1.2676506e30f) {  // 2^100
    const float2 S = dup2(s), N = dup2(__fmul_rn(-128.0f, s)), M = dup2(-kTwo23);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t x = w[j] ^ 0x80808080u;  // int8 -> q + 128
#pragma unroll
      for (int k = 0; k < 4; k += 2) {
        const float2 b = padd(make_float2(byte_in_two23(x, k), byte_in_two23(x, k + 1)), M);
        const float2 t = padd(make_float2(acc[4 * j + k], acc[4 * j + k + 1]), pfma(b, S, N));
        acc[4 * j + k] = t.x, acc[4 * j + k + 1] = t.y;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t x = w[j] ^ 0x80808080u;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float q = __fadd_rn(byte_in_two23(x, k), -kTwo23p128);
        acc[4 * j + k] = __fadd_rn(acc[4 * j + k], __fmul_rn(q, s));
      }
    }
  }
}

// acc[i] += (q_i * s) + z for the 16 INT4 codes in w[2] (code i = nibble i%8 of w[i/8]).
// With U = 2^23 + q (the code in the low bits of 2^23) and nms = -2^23 * s
// (exact while 2^23 * s does not overflow, i.e. s < 2^100 here),
// fma(U, s, nms) rounds the exact value q*s once: it equals the separately
// rounded product fl(q*s).  Larger scales take the plain product.
// The fused form runs on packed pairs (codes 2k and 2k + 1 are neighbours).
template <bool FUSED>
__device__ __forceinline__ void dequant_i4_acc_t(const uint32_t w[2], float s, float z,
                                                 float acc[16]) {
  const float nms = __fmul_rn(-kTwo23, s);
  const float2 S = dup2(s), N = dup2(nms), Z = dup2(z);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t ev, od;  // codes 8j + 2k, codes 8j + 2k + 1
    spread_nibbles(w[j], ev, od);
    float u0[4], u1[4];
    u0[0] = prmt_two23<0x7540>(ev), u1[0] = prmt_two23<0x7540>(od);
    u0[1] = prmt_two23<0x7541>(ev), u1[1] = prmt_two23<0x7541>(od);
    u0[2] = prmt_two23<0x7542>(ev), u1[2] = prmt_two23<0x7542>(od);
    u0[3] = prmt_two23<0x7543>(ev), u1[3] = prmt_two23<0x7543>(od);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float* a = acc + 8 * j + 2 * k;
      if (FUSED) {
        const float2 d = padd(pfma(make_float2(u0[k], u1[k]), S, N), Z);
        const float2 t = padd(make_float2(a[0], a[1]), d);
        a[0] = t.x, a[1] = t.y;
      } else {
        const float p0 = __fmul_rn(__fadd_rn(u0[k], -kTwo23), s);
        const float p1 = __fmul_rn(__fadd_rn(u1[k], -kTwo23), s);
        a[0] = __fadd_rn(a[0], __fadd_rn(p0, z));
        a[1] = __fadd_rn(a[1], __fadd_rn(p1, z));
      }
    }
  }
}
__device__ __forceinline__ void dequant_i4_acc(const uint32_t w[2], float s, float z,
                                               float acc[16]) {
  if (s < 1.2676506e30f)  // 2^100: 2^23 * s stays finite
    dequant_i4_acc_t<true>(w, s, z, acc);
  else
    dequant_i4_acc_t<false>(w, s, z, acc);
}

// RMSNorm's inverse root mean square, 1/sqrt(ss/H + eps), for an output held
// to one bf16 ulp: ss * (1/H) and the hardware reciprocal square root
// (a few binary32 ulps) instead of two IEEE divisions and a square root.
__device__ __forceinline__ float inv_rms(float ss, float inv_h, float eps) {
  return rsqrtf(__fadd_rn(__fmul_rn(ss, inv_h), eps));
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
// Codes are rne(fl(v / s)), v = x (INT8) or v = fl(x - lo) (INT4): an IEEE
// division per element by definition.  Computed without one:
//  1. r ~ 1/s from the hardware reciprocal (relative error <= 2^-23).  With
//     r_hi = fl(r (1 + 2^-20)) and r_lo = fl(r (1 - 2^-20)), the exact
//     products v r_hi and v r_lo bracket fl(v/s) strictly (fl(v/s) is within
//     2^-24 of v/s relative, and (1 + 2^-20)(1 - 2^-23)(1 - 2^-24) > 1 +
//     2^-24).  u = fma(v, r_x, M) with M = 1.5*2^23 (INT8) or 2^23 (INT4)
//     rounds the product to the nearest integer and leaves it in the low
//     mantissa bits of u (which also pack directly into bytes/nibbles).
//  2. If both products round to the same integer c, no half-integer lies
//     strictly between them, hence none between fl(v/s) and them, and
//     rne(fl(v/s)) = c.
//  3. Otherwise (a half-integer lies between the two products: the element
//     sits next to one; bf16 inputs put about 0.2% of the elements there)
//     the element is flagged, and the exact pass gives it its code by the
//     definition, the IEEE quotient rounded to the nearest even integer.
//     (An exact resolution next to the half-integer m through D = v - m*s,
//     which fma gives exactly, took more instructions per flagged element.)
//  4. Groups where the bound v * r <= 127.25 (INT8) / 15.25 (INT4) fails or
//     s < 2^-100 flag every element, i.e. take the IEEE division for all of
//     them (never seen on finite activations; it keeps denormal scales
//     exact).
constexpr float kMagicI8 = 12582912.0f;         // 1.5 * 2^23, bits 0x4B400000
constexpr float kTwoM100 = 7.888609052210118e-31f;  // 2^-100

// fl(x / 15) and fl(x / 127) for the scales, without a division: with
// zh = fl(1/y) and zl = fl(1/y - zh), q = fma(x, zh, fl(x * zl)) is the
// correctly rounded quotient (the method of Brisebarre, Muller and Raina,
// "Accelerating correctly rounded floating-point division when the divisor
// is known in advance", IEEE Trans. Computers 53(8), 2004).  For y = 15 and
// y = 127 this was checked against the IEEE quotient for every binary32
// significand; the check scales to every x >= 2^-98 (quotient and x * zl
// stay normal).  Smaller x take the division.
constexpr uint32_t kInv15Hi = 0x3D888889u, kInv15Lo = 0xB16EEEEFu;
constexpr uint32_t kInv127Hi = 0x3C010204u, kInv127Lo = 0x2E010204u;
template <uint32_t HI, uint32_t LO>
__device__ __forceinline__ float div_by_const(float x, float y) {
  if (!(x >= __uint_as_float(0x0E800000u))) return __fdiv_rn(x, y);  // below 2^-98 (or 0)
  return __fmaf_rn(x, __uint_as_float(HI), __fmul_rn(x, __uint_as_float(LO)));
}
__device__ __forceinline__ float div15(float x) { return div_by_const<kInv15Hi, kInv15Lo>(x, 15.0f); }
__device__ __forceinline__ float div127(float x) { return div_by_const<kInv127Hi, kInv127Lo>(x, 127.0f); }

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ uint32_t low_bytes4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, d, 0x0040u), 0x5410u);
}

// Lane-local group statistics on the 16 bf16 inputs packed in w[8] with
// bf16x2 min/max (exact: selections of input values), as pairwise trees so
// the dependency chains stay short.
__device__ __forceinline__ __nv_bfloat162 bf2(uint32_t w) {
  return *reinterpret_cast<const __nv_bfloat162*>(&w);
}
__device__ __forceinline__ float bf16_absmax16(const uint32_t w[8]) {
  __nv_bfloat162 m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = __hmax2(__habs2(bf2(w[2 * i])), __habs2(bf2(w[2 * i + 1])));
  const __nv_bfloat162 r = __hmax2(__hmax2(m[0], m[1]), __hmax2(m[2], m[3]));
  return fmaxf(__low2float(r), __high2float(r));
}
__device__ __forceinline__ void bf16_minmax16(const uint32_t w[8], float& lo, float& hi) {
  __nv_bfloat162 mn[4], mx[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    mn[i] = __hmin2(bf2(w[2 * i]), bf2(w[2 * i + 1]));
    mx[i] = __hmax2(bf2(w[2 * i]), bf2(w[2 * i + 1]));
  }
  const __nv_bfloat162 a = __hmin2(__hmin2(mn[0], mn[1]), __hmin2(mn[2], mn[3]));
  const __nv_bfloat162 b = __hmax2(__hmax2(mx[0], mx[1]), __hmax2(mx[2], mx[3]));
  lo = fminf(__low2float(a), __high2float(a));
  hi = fmaxf(__low2float(b), __high2float(b));
}

// Tree reductions over 16 floats (max of |v|, min and max).
// (Three-input steps: 16 -> 6 -> 2 -> 1.)
__device__ __forceinline__ float absmax16(const float v[16]) {
  float a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = fabsf(v[i]);
  const float m0 = fmax3(a[0], a[1], a[2]), m1 = fmax3(a[3], a[4], a[5]);
  const float m2 = fmax3(a[6], a[7], a[8]), m3 = fmax3(a[9], a[10], a[11]);
  const float m4 = fmax3(a[12], a[13], a[14]);
  return fmaxf(fmax3(m0, m1, m2), fmax3(m3, m4, a[15]));
}
__device__ __forceinline__ void minmax16(const float v[16], float& lo, float& hi) {
  const float a0 = fmin3(v[0], v[1], v[2]), a1 = fmin3(v[3], v[4], v[5]);
  const float a2 = fmin3(v[6], v[7], v[8]), a3 = fmin3(v[9], v[10], v[11]);
  const float a4 = fmin3(v[12], v[13], v[14]);
  const float b0 = fmax3(v[0], v[1], v[2]), b1 = fmax3(v[3], v[4], v[5]);
  const float b2 = fmax3(v[6], v[7], v[8]), b3 = fmax3(v[9], v[10], v[11]);
  const float b4 = fmax3(v[12], v[13], v[14]);
  lo = fminf(fmin3(a0, a1, a2), fmin3(a3, a4, v[15]));
  hi = fmaxf(fmax3(b0, b1, b2), fmax3(b3, b4, v[15]));
}

// Rounds the 16 quotients v[i] / s; ub[i] gets the bits of M + code (the
// code in its low byte or nibble; the code itself is M + code - M).  group_ok:
// fl(vmax * r) is within the code range and s >= 2^-100 (else every element
// takes the division); s == 0 is passed as r == 0 with group_ok set, which
// yields codes 0.  Every lane of the warp must call this.
// Flagged elements (next to a half-integer, or in a group outside the fast
// path's bounds) are settled after the fast path:
// round_codes returns a 16-bit mask of the lane's elements that need it (bit
// 8b + w for element 4w + b, gathered by byte permutes), settle_codes ORs
// the masks over the warp and one uniform loop
// visits only the element indices set in some lane, each lane computing
// that element's code by division (steps 3 and 4).  pick(i) supplies the
// lane's v_i, put(i, u) stores its exact code (u = bits of M + code).
template <bool SIGNED>
__device__ __forceinline__ uint32_t round_codes(const float v[16], float r, bool group_ok,
                                                uint32_t ub[16]) {
  // Flags from two roundings of every quotient, v * fl(r (1 + 2^-20)) and
  // v * fl(r (1 - 2^-20)), which bracket fl(v / s) strictly (see the
  // requantizers below): where both round to the same integer it is
  // rne(fl(v / s)); where they differ the element lies within 2^-13 of a
  // half-integer and is flagged.  The difference of the two roundings is 0 or
  // +-1.0, whose byte 2 is 0x80: byte permutes gather it into the mask.
  // (Measured on GB300: 6 fewer instructions per 16 values than flags from
  // the residual c - v r.)
  const float magic = SIGNED ? kMagicI8 : 8388608.0f;
  const float2 RH = dup2(__fmul_rn(r, 1.00000095367431640625f)),
               RL = dup2(__fmul_rn(r, 0.99999904632568359375f)), M = dup2(magic);
  float2 dd[8];
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const float2 x = make_float2(v[i], v[i + 1]);
    const float2 a = pfma(x, RH, M), b = pfma(x, RL, M);
    ub[i] = __float_as_uint(a.x), ub[i + 1] = __float_as_uint(a.y);
    dd[i / 2] = psub(a, b);
  }
  uint32_t flag = 0;  // bit w of byte b: element 4w + b flagged
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t s0 = __byte_perm(__float_as_uint(dd[2 * w].x), __float_as_uint(dd[2 * w].y), 0x0062u);
    const uint32_t s1 = __byte_perm(__float_as_uint(dd[2 * w + 1].x), __float_as_uint(dd[2 * w + 1].y), 0x0062u);
    flag |= (__byte_perm(s0, s1, 0x5410u) >> (7 - w)) & (0x01010101u << w);
  }
  return group_ok ? flag : 0x0F0F0F0Fu;
}

// The code by its definition: the IEEE quotient, rounded to the nearest
// even integer, clamped to the code range.
template <bool SIGNED>
__device__ __forceinline__ float code_by_division(float v, float s) {
  const float q = rintf(__fdiv_rn(v, s));
  return SIGNED ? fminf(127.0f, fmaxf(-127.0f, q)) : fminf(15.0f, fmaxf(0.0f, q));
}

template <bool SIGNED, class Pick, class Put>
__device__ __forceinline__ void settle_codes(uint32_t mask, float s, Pick pick, Put put) {
  const float magic = SIGNED ? kMagicI8 : 8388608.0f;
  uint32_t todo = __reduce_or_sync(kFull, mask);
  while (todo) {  // warp-uniform
    const int pos = __ffs(todo) - 1;
    todo &= todo - 1;
    const int i = 4 * (pos & 7) + (pos >> 3);
    const float res = code_by_division<SIGNED>(pick(i), s);
    if ((mask >> pos) & 1u) put(i, __float_as_uint(__fadd_rn(res, magic)));
  }
}

// pick / put over the register arrays (a switch on the warp-uniform index)
struct RegSettle {
  const float* v;
  uint32_t* ub;
  __device__ __forceinline__ float operator()(int i) const {
    switch (i) {
#define FC_PICK(k) \
  case k: return v[k];
      FC_PICK(0) FC_PICK(1) FC_PICK(2) FC_PICK(3) FC_PICK(4) FC_PICK(5) FC_PICK(6) FC_PICK(7)
      FC_PICK(8) FC_PICK(9) FC_PICK(10) FC_PICK(11) FC_PICK(12) FC_PICK(13) FC_PICK(14) FC_PICK(15)
#undef FC_PICK
    }
    return 0.0f;
  }
  __device__ __forceinline__ void operator()(int i, uint32_t rb) const {
    switch (i) {
#define FC_PUT(k) \
  case k: ub[k] = rb; break;
      FC_PUT(0) FC_PUT(1) FC_PUT(2) FC_PUT(3) FC_PUT(4) FC_PUT(5) FC_PUT(6) FC_PUT(7)
      FC_PUT(8) FC_PUT(9) FC_PUT(10) FC_PUT(11) FC_PUT(12) FC_PUT(13) FC_PUT(14) FC_PUT(15)
#undef FC_PUT
    }
  }
};

// The exact pass over register arrays, unrolled over the 16 element
// positions: position i is visited (a warp-uniform branch) when it is
// flagged in any lane of the warp, every lane computes element i's exact
// code, and lanes that flagged it keep it.  Registers are indexed at
// compile time, so a visit costs the exact code alone.  Measured on GB300
// (with the earlier exact resolution next to the half-integer) it pays
// where flagged elements are dense -- the requantized sum of two INT4 slabs,
// whose quotients sit on or next to half-integers often (fused kernel, 64 MB
// messages: 68 -> 60 us) -- and costs time in the larger kernels of more
// slabs, which keep the index loop (settle_codes).
template <bool SIGNED>
__device__ __forceinline__ void settle_codes_regs(uint32_t mask, float s, const float v[16], uint32_t ub[16]) {
  const uint32_t any = __reduce_or_sync(kFull, mask);
  if (!any) return;
  const float magic = SIGNED ? kMagicI8 : 8388608.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t bit = 1u << (8 * (i & 3) + (i >> 2));  // element 4w + b is mask bit 8b + w
    if (any & bit) {
      const float res = code_by_division<SIGNED>(v[i], s);
      if (mask & bit) ub[i] = __float_as_uint(__fadd_rn(res, magic));
    }
  }
}

// Where the quantizers settle the flagged elements: SettleHere, in this call,
// over the register arrays (the fused kernels' requantization); DeferSettle,
// not at all: the flag mask (bit 8b + w for element 4w + b) goes to *mask
// and the caller settles those elements later and patches the stored codes
// (the sender, once per staged tile for all its chunks).
struct SettleHere {};
struct DeferSettle {
  uint32_t* mask;
};

// INT8 symmetric on this lane's 16 values of a group spread over lpg lanes:
//   s = max|x| / 127;  q = clamp(rne(x / s), -127, 127);  s == 0 -> q = 0.
// Writes the codes packed in q[4]; with DEQ also d[i] = q_i * s.  Returns s.
// With BFW, the lane's max|x| is taken from the packed bf16 inputs bw[8].
// UNROLLED: the exact pass over registers is settle_codes_regs (else the
// index loop, settle_codes).
template <bool DEQ, bool BFW = false, class Settle = SettleHere, bool UNROLLED = false>
__device__ __forceinline__ float quant_i8(const float v[16], int lpg, uint32_t q[4], float d[16],
                                          const uint32_t* bw = nullptr, Settle settle = Settle()) {
  float a = BFW ? bf16_absmax16(bw) : absmax16(v);
  a = group_max(a, lpg);
  const float s = div127(a);
  uint32_t ub[16];  // low byte: the code
  const float r = s == 0.0f ? 0.0f : rcp_approx(s);
  const bool ok = s == 0.0f || (__fmul_rn(a, r) <= 127.25f && s >= kTwoM100);
  const uint32_t mask = round_codes<true>(v, r, ok, ub);
  if constexpr (std::is_same<Settle, DeferSettle>::value) {
    *settle.mask = mask;
  } else {
    if (UNROLLED)
      settle_codes_regs<true>(mask, s, v, ub);
    else
      settle_codes<true>(mask, s, RegSettle{v, ub}, RegSettle{v, ub});
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) q[j] = low_bytes4(ub[4 * j], ub[4 * j + 1], ub[4 * j + 2], ub[4 * j + 3]);
  if (DEQ) {
    if (s < 1.2676506e30f) {  // u - 2^22 = 2^23 + q exactly; fma(2^23 + q, s, -2^23 s) = fl(q s)
      const float2 C = dup2(-4194304.0f), S = dup2(s), N = dup2(__fmul_rn(-kTwo23, s));
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float2 t = pfma(padd(make_float2(__uint_as_float(ub[i]), __uint_as_float(ub[i + 1])), C), S, N);
        d[i] = t.x, d[i + 1] = t.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) d[i] = __fmul_rn(__fsub_rn(__uint_as_float(ub[i]), kMagicI8), s);
    }
  }
  return s;
}

// INT4 asymmetric: lo = min, hi = max (a zero extreme taken as +0),
// s = (hi - lo) / 15, z = lo, q = clamp(rne((x - lo) / s), 0, 15).
// Element 2i in the low nibble of byte i.  Returns s, writes z; with DEQ also
// d[i] = (q_i * s) + z.  With BFW, the lane's min and max come from the
// packed bf16 inputs bw[8].
template <bool DEQ, bool BFW = false, class Settle = SettleHere, bool UNROLLED = false>
__device__ __forceinline__ float quant_i4(const float v[16], int lpg, uint32_t q[2], float& z,
                                          float d[16], const uint32_t* bw = nullptr,
                                          Settle settle = Settle()) {
  float lo, hi;
  if (BFW)
    bf16_minmax16(bw, lo, hi);
  else
    minmax16(v, lo, hi);
  lo = __fadd_rn(group_min(lo, lpg), 0.0f);  // -0 + 0 = +0; other values unchanged
  hi = __fadd_rn(group_max(hi, lpg), 0.0f);
  const float span = __fsub_rn(hi, lo);
  const float s = div15(span);
  z = lo;
  uint32_t ub[16];
  float num[16];  // fl(x - lo)
  if (BFW) {
#pragma unroll
    for (int i = 0; i < 8; ++i) num[2 * i] = add_bf_lo(bw[i], -lo), num[2 * i + 1] = add_bf_hi(bw[i], -lo);
  } else {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const float2 n = padd(make_float2(v[i], v[i + 1]), dup2(-lo));
      num[i] = n.x, num[i + 1] = n.y;
    }
  }
  const float r = s == 0.0f ? 0.0f : rcp_approx(s);
  const bool ok = s == 0.0f || (__fmul_rn(span, r) <= 15.25f && s >= kTwoM100);
  const uint32_t mask = round_codes<false>(num, r, ok, ub);
  if constexpr (std::is_same<Settle, DeferSettle>::value) {
    *settle.mask = mask;
  } else {
    if (UNROLLED)
      settle_codes_regs<false>(mask, s, num, ub);
    else
      settle_codes<false>(mask, s, RegSettle{num, ub}, RegSettle{num, ub});
  }
  // Nibble packing by multiply-adds: ub = 0x4B000000 + code with code in
  // [0, 15] wherever the fast path holds, so sum_i ub[8j+i] * 16^i is the
  // packed word plus 0x4B000000 * 0x11111111 = 0xFB000000 (mod 2^32).
  // (Groups outside the fast path have every nibble rewritten by the exact
  // pass.)
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t w = ub[8 * j + 7];
#pragma unroll
    for (int i = 6; i >= 1; --i) w = w * 16u + ub[8 * j + i];
    q[j] = w * 16u + (ub[8 * j] - 0xFB000000u);
  }
  if (DEQ) {  // d = fl(fl(q * s) + z); fl(q * s) = fma(2^23 + q, s, -2^23 * s) for s < 2^100
    if (s < 1.2676506e30f) {
      const float2 S = dup2(s), N = dup2(__fmul_rn(-kTwo23, s)), Z = dup2(z);
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float2 t =
            padd(pfma(make_float2(__uint_as_float(ub[i]), __uint_as_float(ub[i + 1])), S, N), Z);
        d[i] = t.x, d[i + 1] = t.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        d[i] = __fadd_rn(__fmul_rn(__fsub_rn(__uint_as_float(ub[i]), kTwo23), s), z);
    }
  }
  return s;
}

// ------------------------------------------------ requantizers (fp32 in) --
// The requantization of the reduced sums (fp32 values) in kernels that sum
// eight slabs.  It uses the same two roundings as round_codes (steps
// 1-3 above) but flags nothing per element: the codes of both roundings are
// packed side by side and compared word by word, and only a warp in which
// some word differs builds the per-element mask and settles it.  With four or
// more slabs an element next to a half-integer is rare (0.05% of the prefill
// sums, against 0.3% for two slabs, where the mask of round_codes is cheaper),
// so the common case costs one extra rounding and packing per element (with
// four slabs the extra live values made the compact build spill).
// Measured on GB300 (executed instructions per 16 values, quantize and
// dequantize, random groups): INT4 139 -> 116, INT8 127 -> 96; checked
// bit-identical to the earlier near-half-integer scheme on 2^20 chunks of
// random, tie-dense and near-tie groups, and against the oracle by the GPU
// tests.

// The exact pass over register arrays with a natural-order mask (bit i =
// element i): position i is visited, unrolled, when any lane of the warp
// flagged it.
__device__ __forceinline__ void settle_unrolled(uint32_t mask, float s, const float v[16], bool is_signed,
                                                uint32_t ub[16]) {
  const uint32_t any = __reduce_or_sync(kFull, mask);
  const float magic = is_signed ? kMagicI8 : kTwo23;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (any & (1u << i)) {
      const float res = is_signed ? code_by_division<true>(v[i], s) : code_by_division<false>(v[i], s);
      if (mask & (1u << i)) ub[i] = __float_as_uint(__fadd_rn(res, magic));
    }
  }
}

// Eight 4-bit codes (ub = bits of 2^23 + code) packed into nibbles by a
// multiply-add chain (see quant_i4).
__device__ __forceinline__ uint32_t pack_nibbles8(const uint32_t* ub) {
  uint32_t w = ub[7];
#pragma unroll
  for (int i = 6; i >= 1; --i) w = w * 16u + ub[i];
  return w * 16u + (ub[0] - 0xFB000000u);
}

constexpr float kRcpUp = 1.00000095367431640625f;    // 1 + 2^-20
constexpr float kRcpDown = 0.99999904632568359375f;  // 1 - 2^-20

// INT4 asymmetric requantization of this lane's 16 fp32 values of a group
// spread over lpg lanes: lo = min, hi = max (a zero extreme taken as +0),
// s = (hi - lo) / 15, z = lo, q = clamp(rne((v - lo) / s), 0, 15).  Writes the
// packed codes q[2], z, and d = fl(fl(q s) + z); returns s.  Every lane of the
// warp must call it.
__device__ __forceinline__ float requant_i4(const float v[16], int lpg, uint32_t q[2], float& z,
                                            float d[16]) {
  float lo, hi;
  minmax16(v, lo, hi);
  lo = __fadd_rn(group_min(lo, lpg), 0.0f);  // -0 + 0 = +0; other values unchanged
  hi = __fadd_rn(group_max(hi, lpg), 0.0f);
  const float span = __fsub_rn(hi, lo);
  const float s = div15(span);
  z = lo;
  float num[16];  // fl(v - lo)
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const float2 n = padd(make_float2(v[i], v[i + 1]), dup2(-lo));
    num[i] = n.x, num[i + 1] = n.y;
  }
  const float r = s == 0.0f ? 0.0f : rcp_approx(s);
  const bool ok = s == 0.0f || (__fmul_rn(span, r) <= 15.25f && s >= kTwoM100);
  const float2 RH = dup2(__fmul_rn(r, kRcpUp)), RL = dup2(__fmul_rn(r, kRcpDown)), M = dup2(kTwo23);
  uint32_t u1[16];
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const float2 a = pfma(make_float2(num[i], num[i + 1]), RH, M);
    u1[i] = __float_as_uint(a.x), u1[i + 1] = __float_as_uint(a.y);
  }
  q[0] = pack_nibbles8(u1), q[1] = pack_nibbles8(u1 + 8);
  // the codes from r_lo, folded into packed words as they come (high code
  // first), so only a pair of them is live at a time
  uint32_t diff = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t w = 0;
#pragma unroll
    for (int k = 3; k >= 0; --k) {
      const float2 b = pfma(make_float2(num[8 * j + 2 * k], num[8 * j + 2 * k + 1]), RL, M);
      w = w * 16u + __float_as_uint(b.y);
      w = w * 16u + __float_as_uint(b.x);
    }
    diff |= q[j] ^ (w - 0xFB000000u);
  }
  if (__any_sync(kFull, diff != 0u || !ok)) {  // rare: settle the flagged elements
    uint32_t mask = 0xFFFFu;
    if (ok) {
      mask = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        mask |= (u1[i] != __float_as_uint(__fmaf_rn(num[i], __fmul_rn(r, kRcpDown), kTwo23)) ? 1u : 0u) << i;
    }
    settle_unrolled(mask, s, num, false, u1);
    q[0] = pack_nibbles8(u1), q[1] = pack_nibbles8(u1 + 8);
  }
  if (s < 1.2676506e30f) {  // fl(q s) = fma(2^23 + q, s, -2^23 s), exact for s < 2^100
    const float2 S = dup2(s), N = dup2(__fmul_rn(-kTwo23, s)), Z = dup2(z);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const float2 t =
          padd(pfma(make_float2(__uint_as_float(u1[i]), __uint_as_float(u1[i + 1])), S, N), Z);
      d[i] = t.x, d[i + 1] = t.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) d[i] = __fadd_rn(__fmul_rn(__fsub_rn(__uint_as_float(u1[i]), kTwo23), s), z);
  }
  return s;
}

// INT8 symmetric requantization of this lane's 16 fp32 values of a group
// spread over lpg lanes: s = max|v| / 127, q = clamp(rne(v / s), -127, 127);
// writes q[4] and d = fl(q s); returns s.  Every lane must call it.
__device__ __forceinline__ float requant_i8(const float v[16], int lpg, uint32_t q[4], float d[16]) {
  const float a = group_max(absmax16(v), lpg);
  const float s = div127(a);
  const float r = s == 0.0f ? 0.0f : rcp_approx(s);
  const bool ok = s == 0.0f || (__fmul_rn(a, r) <= 127.25f && s >= kTwoM100);
  const float2 RH = dup2(__fmul_rn(r, kRcpUp)), RL = dup2(__fmul_rn(r, kRcpDown)), M = dup2(kMagicI8);
  uint32_t u1[16], diff = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // four codes at a time: both roundings, packed and compared
    const float2 a0 = pfma(make_float2(v[4 * j], v[4 * j + 1]), RH, M);
    const float2 a1 = pfma(make_float2(v[4 * j + 2], v[4 * j + 3]), RH, M);
    const float2 b0 = pfma(make_float2(v[4 * j], v[4 * j + 1]), RL, M);
    const float2 b1 = pfma(make_float2(v[4 * j + 2], v[4 * j + 3]), RL, M);
    u1[4 * j] = __float_as_uint(a0.x), u1[4 * j + 1] = __float_as_uint(a0.y);
    u1[4 * j + 2] = __float_as_uint(a1.x), u1[4 * j + 3] = __float_as_uint(a1.y);
    q[j] = low_bytes4(u1[4 * j], u1[4 * j + 1], u1[4 * j + 2], u1[4 * j + 3]);
    diff |= q[j] ^ low_bytes4(__float_as_uint(b0.x), __float_as_uint(b0.y), __float_as_uint(b1.x),
                              __float_as_uint(b1.y));
  }
  if (__any_sync(kFull, diff != 0u || !ok)) {  // rare: settle the flagged elements
    uint32_t mask = 0xFFFFu;
    if (ok) {
      mask = 0;
      const float rl = __fmul_rn(r, kRcpDown);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        mask |= (u1[i] != __float_as_uint(__fmaf_rn(v[i], rl, kMagicI8)) ? 1u : 0u) << i;
    }
    settle_unrolled(mask, s, v, true, u1);
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = low_bytes4(u1[4 * j], u1[4 * j + 1], u1[4 * j + 2], u1[4 * j + 3]);
  }
  if (s < 1.2676506e30f) {  // u - 2^22 = 2^23 + q exactly; fma(2^23 + q, s, -2^23 s) = fl(q s)
    const float2 C = dup2(-4194304.0f), S = dup2(s), N = dup2(__fmul_rn(-kTwo23, s));
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const float2 t = pfma(padd(make_float2(__uint_as_float(u1[i]), __uint_as_float(u1[i + 1])), C), S, N);
      d[i] = t.x, d[i + 1] = t.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) d[i] = __fmul_rn(__fsub_rn(__uint_as_float(u1[i]), kMagicI8), s);
  }
  return s;
}

}  // namespace fc
