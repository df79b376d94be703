// fused.cu -- the fused quantized All-Reduce + residual add + RMSNorm.
//
// One CTA owns one token row at a time (persistent CTAs stride over rows),
// because RMSNorm needs the whole row before any output can be written:
//   pass 1: for each 16-element chunk of the row, read the P slabs' codes
//           (or bf16 / tagged blocks), sum the dequantized values in slab
//           order, requantize the group (the all-gather payload), dequantize
//           it, add the residual, round to bf16 (written as residual_out and
//           kept in registers), accumulate the sum of squares;
//   block reduction of the sum of squares;
//   pass 2: y = bf16((h * inv_rms) * gamma) from the registers.
// Nothing but y, residual_out and the optional payload leaves the SM; the
// reduced fp32 row never touches HBM.
#include <climits>

#include "device.cuh"
#include "internal.h"

namespace fc {

namespace {

constexpr int kMaxThreads = 512;

// Sum of squares over the CTA; `red` is double-buffered by row parity so
// that one barrier per row suffices.
__device__ __forceinline__ float block_sum(float v, float (*red)[32], int parity) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  if (lane == 0) red[parity][wid] = v;
  __syncthreads();
  float t = 0.0f;
  for (int w = 0; w < nw; ++w) t += red[parity][w];
  return t;
}

__device__ __forceinline__ float inv_rms(float ss, int H, float eps) {
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(H)), eps)));
}

// ------------------------------------------------ BF16 / INT8 / INT4 path --
template <int FMT, int NCH>
__global__ void __launch_bounds__(kMaxThreads) k_fused(FusedArgs a) {
  __shared__ float red[2][32];
  const int tid = threadIdx.x, lane = tid & 31;
  const int nthr = blockDim.x;
  const int cpr = a.H >> 4;  // chunks per row
  const int lpg = a.G >> 4;
  const int P = a.P;
  int parity = 0;

  for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, parity ^= 1) {
    uint32_t hb[NCH][8];
    float2 ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
      const int c = k * nthr + tid;
      const bool act = c < cpr;
      const int64_t gc = row * cpr + c;  // global chunk index
      const int64_t g = gc >> a.lpg_shift;
      float acc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = 0.0f;

      // ---- loads: every slab's chunk, then the residual
      V8 rv;
      if (FMT == kBF16) {
        V8 xv[kMaxP];
#pragma unroll
        for (int p = 0; p < kMaxP; ++p)
          if (p < P && act) xv[p] = ld256_stream(static_cast<const uint16_t*>(a.s.codes[p]) + gc * 16);
        if (act) rv = ld256_stream(static_cast<const uint16_t*>(a.res_in) + gc * 16);
#pragma unroll
        for (int p = 0; p < kMaxP; ++p) {
          if (p < P && act) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float2 t = padd(make_float2(acc[2 * i], acc[2 * i + 1]),
                                    make_float2(bf_lo(xv[p].w[i]), bf_hi(xv[p].w[i])));
              acc[2 * i] = t.x, acc[2 * i + 1] = t.y;
            }
          }
        }
      } else {
        uint32_t qv[kMaxP][FMT == kINT8 ? 4 : 2];
        float sc[kMaxP], zp[kMaxP];
#pragma unroll
        for (int p = 0; p < kMaxP; ++p) {
          if (p < P && act) {
            if (FMT == kINT8) {
              const uint4 w = ld128_stream(static_cast<const int8_t*>(a.s.codes[p]) + gc * 16);
              qv[p][0] = w.x, qv[p][1] = w.y, qv[p][2] = w.z, qv[p][3] = w.w;
            } else {
              const uint2 w = ld64_stream(static_cast<const uint8_t*>(a.s.codes[p]) + gc * 8);
              qv[p][0] = w.x, qv[p][1] = w.y;
              zp[p] = ldf_stream(a.s.zeros[p] + g);
            }
            sc[p] = ldf_stream(a.s.scales[p] + g);
          }
        }
        if (act) rv = ld256_stream(static_cast<const uint16_t*>(a.res_in) + gc * 16);
        // ---- fixed-order sum of the dequantized slabs
#pragma unroll
        for (int p = 0; p < kMaxP; ++p) {
          if (p < P && act) {
            if (FMT == kINT8)
              dequant_i8_acc(qv[p], sc[p], acc);
            else
              dequant_i4_acc(qv[p], sc[p], zp[p], acc);
          }
        }
        // ---- requantize the reduced group (all-gather payload) and
        //      dequantize it in place (every lane joins the group shuffles)
        if (FMT == kINT8) {
          uint32_t q[4];
          const float s = quant_i8<true>(acc, lpg, q, acc);
          if (act && a.rq_codes) {
            st128(static_cast<int8_t*>(a.rq_codes) + gc * 16, make_uint4(q[0], q[1], q[2], q[3]));
            if ((lane & (lpg - 1)) == 0) stf(a.rq_scales + g, s);
          }
        } else {
          uint32_t q[2];
          float z;
          const float s = quant_i4<true>(acc, lpg, q, z, acc);
          if (act && a.rq_codes) {
            st64(static_cast<uint8_t*>(a.rq_codes) + gc * 8, make_uint2(q[0], q[1]));
            if ((lane & (lpg - 1)) == 0) {
              stf(a.rq_scales + g, s);
              stf(a.rq_zeros + g, z);
            }
          }
        }
      }

      // ---- residual add, bf16 rounding, sum of squares
      if (act) {
        V8 hv;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hb[k][i] = hv.w[i] = pack_bf2(__fadd_rn(acc[2 * i], bf_lo(rv.w[i])),
                                        __fadd_rn(acc[2 * i + 1], bf_hi(rv.w[i])));
        }
        st256(static_cast<uint16_t*>(a.res_out) + gc * 16, hv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 h = make_float2(bf_lo(hb[k][i]), bf_hi(hb[k][i]));
          ss2 = pfma(h, h, ss2);
        }
      }
    }

    const float ss = __fadd_rn(ss2.x, ss2.y);
    const float inv = inv_rms(block_sum(ss, red, parity), a.H, a.eps);

    // ---- y = bf16((h * inv) * gamma)
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
      const int c = k * nthr + tid;
      if (c < cpr) {
        const V8 gv = ld256_keep(static_cast<const uint16_t*>(a.gamma) + c * 16);
        V8 yv;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 y = pmul(pmul(make_float2(bf_lo(hb[k][i]), bf_hi(hb[k][i])), dup2(inv)),
                                make_float2(bf_lo(gv.w[i]), bf_hi(gv.w[i])));
          yv.w[i] = pack_bf2(y.x, y.y);
        }
        st256(static_cast<uint16_t*>(a.y) + (row * cpr + c) * 16, yv);
      }
    }
  }
}

// ------------------------------------------------------ tagged bf16 path --
// A unit is 4 blocks = 24 elements of one row (48 bytes of residual / gamma /
// outputs, 16-byte aligned).  Each block's tag is checked in the same
// 16-byte load that brings its payload; a failing block is not summed.
template <int NU>
__global__ void __launch_bounds__(kMaxThreads) k_fused_tagged(FusedArgs a) {
  __shared__ float red[2][32];
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const int H = a.H;
  const int nb = (H + 5) / 6;
  const int units = (nb + 3) >> 2;
  const int P = a.P;
  const uint32_t epoch = a.epoch;
  int parity = 0;

  for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, parity ^= 1) {
    uint32_t hb[NU][12];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < NU; ++k) {
      const int u = k * nthr + tid;
      const bool act = u < units;
      const bool full = act && 24 * u + 24 <= H;
      float acc[24];
#pragma unroll
      for (int i = 0; i < 24; ++i) acc[i] = 0.0f;
      int64_t first_bad = LLONG_MAX;
#pragma unroll
      for (int p = 0; p < kMaxP; ++p) {
        if (p < P && act) {
          const uint4* bl = static_cast<const uint4*>(a.s.codes[p]) + row * nb + 4 * u;
          uint4 b[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            b[j] = (4 * u + j < nb) ? ld128_stream(bl + j) : make_uint4(0, 0, 0, epoch);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (b[j].w == epoch) {
              acc[6 * j + 0] = __fadd_rn(acc[6 * j + 0], bf_lo(b[j].x));
              acc[6 * j + 1] = __fadd_rn(acc[6 * j + 1], bf_hi(b[j].x));
              acc[6 * j + 2] = __fadd_rn(acc[6 * j + 2], bf_lo(b[j].y));
              acc[6 * j + 3] = __fadd_rn(acc[6 * j + 3], bf_hi(b[j].y));
              acc[6 * j + 4] = __fadd_rn(acc[6 * j + 4], bf_lo(b[j].z));
              acc[6 * j + 5] = __fadd_rn(acc[6 * j + 5], bf_hi(b[j].z));
            } else {
              const int64_t idx = (static_cast<int64_t>(p) * a.rows + row) * nb + 4 * u + j;
              first_bad = idx < first_bad ? idx : first_bad;
            }
          }
        }
      }
      if (first_bad != LLONG_MAX && a.status) {
        atomicCAS(a.status, 0, 3 /* FC_ERR_STALE_BLOCK */);
        atomicMin(a.status + 1, first_bad < INT_MAX ? static_cast<int>(first_bad) : INT_MAX - 1);
      }
      // residual
      const uint16_t* rr = static_cast<const uint16_t*>(a.res_in) + row * H + 24 * u;
      uint32_t rw[12];
      if (full) {
        const uint4 r0 = ld128_stream(rr), r1 = ld128_stream(rr + 8), r2 = ld128_stream(rr + 16);
        rw[0] = r0.x, rw[1] = r0.y, rw[2] = r0.z, rw[3] = r0.w;
        rw[4] = r1.x, rw[5] = r1.y, rw[6] = r1.z, rw[7] = r1.w;
        rw[8] = r2.x, rw[9] = r2.y, rw[10] = r2.z, rw[11] = r2.w;
      } else {
#pragma unroll
        for (int i = 0; i < 12; ++i) {
          const int e = 24 * u + 2 * i;
          const uint32_t lo = (act && e < H) ? ld16(rr + 2 * i) : 0u;
          const uint32_t hi = (act && e + 1 < H) ? ld16(rr + 2 * i + 1) : 0u;
          rw[i] = lo | (hi << 16);
        }
      }
#pragma unroll
      for (int i = 0; i < 12; ++i)
        hb[k][i] = pack_bf2(__fadd_rn(acc[2 * i], bf_lo(rw[i])),
                            __fadd_rn(acc[2 * i + 1], bf_hi(rw[i])));
      uint16_t* ro = static_cast<uint16_t*>(a.res_out) + row * H + 24 * u;
      if (full) {
        st128(ro, make_uint4(hb[k][0], hb[k][1], hb[k][2], hb[k][3]));
        st128(ro + 8, make_uint4(hb[k][4], hb[k][5], hb[k][6], hb[k][7]));
        st128(ro + 16, make_uint4(hb[k][8], hb[k][9], hb[k][10], hb[k][11]));
      } else if (act) {
#pragma unroll
        for (int i = 0; i < 24; ++i)
          if (24 * u + i < H) ro[i] = static_cast<uint16_t>(hb[k][i >> 1] >> (16 * (i & 1)));
      }
      if (act) {
#pragma unroll
        for (int i = 0; i < 12; ++i) {
          const float h0 = bf_lo(hb[k][i]), h1 = bf_hi(hb[k][i]);
          ss = __fmaf_rn(h0, h0, ss);
          ss = __fmaf_rn(h1, h1, ss);
        }
      }
    }

    const float inv = inv_rms(block_sum(ss, red, parity), H, a.eps);

#pragma unroll
    for (int k = 0; k < NU; ++k) {
      const int u = k * nthr + tid;
      if (u >= units) continue;
      const bool full = 24 * u + 24 <= H;
      const uint16_t* gp = static_cast<const uint16_t*>(a.gamma) + 24 * u;
      uint32_t gw[12];
      if (full) {
        const uint4 g0 = *reinterpret_cast<const uint4*>(gp),
                    g1 = *reinterpret_cast<const uint4*>(gp + 8),
                    g2 = *reinterpret_cast<const uint4*>(gp + 16);
        gw[0] = g0.x, gw[1] = g0.y, gw[2] = g0.z, gw[3] = g0.w;
        gw[4] = g1.x, gw[5] = g1.y, gw[6] = g1.z, gw[7] = g1.w;
        gw[8] = g2.x, gw[9] = g2.y, gw[10] = g2.z, gw[11] = g2.w;
      } else {
#pragma unroll
        for (int i = 0; i < 12; ++i) {
          const int e = 24 * u + 2 * i;
          const uint32_t lo = e < H ? ld16(gp + 2 * i) : 0u;
          const uint32_t hi = e + 1 < H ? ld16(gp + 2 * i + 1) : 0u;
          gw[i] = lo | (hi << 16);
        }
      }
      uint32_t yw[12];
#pragma unroll
      for (int i = 0; i < 12; ++i)
        yw[i] = pack_bf2(__fmul_rn(__fmul_rn(bf_lo(hb[k][i]), inv), bf_lo(gw[i])),
                         __fmul_rn(__fmul_rn(bf_hi(hb[k][i]), inv), bf_hi(gw[i])));
      uint16_t* yo = static_cast<uint16_t*>(a.y) + row * H + 24 * u;
      if (full) {
        st128(yo, make_uint4(yw[0], yw[1], yw[2], yw[3]));
        st128(yo + 8, make_uint4(yw[4], yw[5], yw[6], yw[7]));
        st128(yo + 16, make_uint4(yw[8], yw[9], yw[10], yw[11]));
      } else {
#pragma unroll
        for (int i = 0; i < 24; ++i)
          if (24 * u + i < H) yo[i] = static_cast<uint16_t>(yw[i >> 1] >> (16 * (i & 1)));
      }
    }
  }
}

// ---------------------------------------------------------------- launch --
struct OccEntry {
  const void* fn;
  int threads;
  int dev;
  int blocks;
};

int occupancy(const void* fn, int threads) {
  static OccEntry cache[64];
  static int n = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < n; ++i)
    if (cache[i].fn == fn && cache[i].threads == threads && cache[i].dev == dev)
      return cache[i].blocks;
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, 0) != cudaSuccess || b < 1)
    b = 1;
  if (n < 64) cache[n++] = OccEntry{fn, threads, dev, b};
  return b;
}

template <typename K>
cudaError_t launch_rows(K kernel, int threads, const FusedArgs& a, int max_ctas, cudaStream_t st) {
  int64_t grid = static_cast<int64_t>(num_sms()) * occupancy(reinterpret_cast<const void*>(kernel), threads);
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  if (grid > a.rows) grid = a.rows;
  kernel<<<static_cast<int>(grid), threads, 0, st>>>(a);
  return cudaGetLastError();
}

int round_warp(int t) { return (t + 31) & ~31; }

template <int FMT>
cudaError_t launch_fmt(const FusedArgs& a, int max_ctas, cudaStream_t st) {
  // chunks per thread: the smallest power of two keeping the CTA at <= 256
  // threads (<= 512 for very wide rows).
  const int cpr = a.H >> 4;
  int nch = 1;
  while (nch < 8 && (cpr + nch - 1) / nch > 256) nch <<= 1;
  const int threads = round_warp((cpr + nch - 1) / nch);
  if (threads > kMaxThreads) return cudaErrorInvalidConfiguration;
  switch (nch) {
    case 1: return launch_rows(k_fused<FMT, 1>, threads, a, max_ctas, st);
    case 2: return launch_rows(k_fused<FMT, 2>, threads, a, max_ctas, st);
    case 4: return launch_rows(k_fused<FMT, 4>, threads, a, max_ctas, st);
    default: return launch_rows(k_fused<FMT, 8>, threads, a, max_ctas, st);
  }
}

cudaError_t launch_tagged(const FusedArgs& a, int max_ctas, cudaStream_t st) {
  const int nb = (a.H + 5) / 6;
  const int units = (nb + 3) / 4;
  int nu = 1;
  while (nu < 8 && (units + nu - 1) / nu > 256) nu <<= 1;
  const int threads = round_warp((units + nu - 1) / nu);
  if (threads > kMaxThreads) return cudaErrorInvalidConfiguration;
  switch (nu) {
    case 1: return launch_rows(k_fused_tagged<1>, threads, a, max_ctas, st);
    case 2: return launch_rows(k_fused_tagged<2>, threads, a, max_ctas, st);
    case 4: return launch_rows(k_fused_tagged<4>, threads, a, max_ctas, st);
    default: return launch_rows(k_fused_tagged<8>, threads, a, max_ctas, st);
  }
}

}  // namespace

cudaError_t launch_fused(int fmt, const FusedArgs& a, int max_ctas, int path, cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  if (path != kPathStream && fused_tma_eligible(fmt, a)) return launch_fused_tma(fmt, a, max_ctas, st);
  if (path == kPathTma) return cudaErrorNotSupported;
  switch (fmt) {
    case kBF16: return launch_fmt<kBF16>(a, max_ctas, st);
    case kINT8: return launch_fmt<kINT8>(a, max_ctas, st);
    case kINT4: return launch_fmt<kINT4>(a, max_ctas, st);
    case kTAGGED: return launch_tagged(a, max_ctas, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fc
