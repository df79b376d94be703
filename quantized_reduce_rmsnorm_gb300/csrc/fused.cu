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
//   pass 2: y = bf16(fl(h * gamma) * inv_rms) from the registers.
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


// ------------------------------------------------ BF16 / INT8 / INT4 path --
template <int FMT, int NCH>
__global__ void __launch_bounds__(kMaxThreads) k_fused(FusedArgs a) {
  pdl_begin();
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
              acc[2 * i] = add_bf_lo(xv[p].w[i], acc[2 * i]);
              acc[2 * i + 1] = add_bf_hi(xv[p].w[i], acc[2 * i + 1]);
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
          hb[k][i] = hv.w[i] = pack_bf2(add_bf_lo(rv.w[i], acc[2 * i]),
                                        add_bf_hi(rv.w[i], acc[2 * i + 1]));
        }
        st256(static_cast<uint16_t*>(a.res_out) + gc * 16, hv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ss2.x = fma_bf_lo(hb[k][i], hb[k][i], ss2.x);
          ss2.y = fma_bf_hi(hb[k][i], hb[k][i], ss2.y);
        }
      }
    }

    const float ss = __fadd_rn(ss2.x, ss2.y);
    const float inv = inv_rms(block_sum(ss, red, parity), 1.0f / static_cast<float>(a.H), a.eps);

    // ---- y = bf16(fl(h * gamma) * inv); h * gamma is exact in binary32
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
      const int c = k * nthr + tid;
      if (c < cpr) {
        const V8 gv = ld256_keep(static_cast<const uint16_t*>(a.gamma) + c * 16);
        V8 yv;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 y = pmul(make_float2(fma_bf_lo(hb[k][i], gv.w[i], -0.0f),
                                            fma_bf_hi(hb[k][i], gv.w[i], -0.0f)),
                                dup2(inv));
          yv.w[i] = pack_bf2(y.x, y.y);
        }
        st256(static_cast<uint16_t*>(a.y) + (row * cpr + c) * 16, yv);
      }
    }
  }
}

// ------------------------------------------------------ tagged bf16 path --
// One warp per token row, one lane per 16-byte block.  Per group of 32
// blocks: each slab's block arrives in one 16-byte load (a warp reads 512
// contiguous bytes per slab) and its tag is checked in that same load; a
// block that fails is not summed.  The residual and the outputs move as
// three 4-byte words per lane (6 bf16 at a 12-byte stride).  The row's sum
// of squares is a warp reduction, so warps never wait for each other; pass 2
// reads h back from residual_out, which this lane has just written (the row
// is still in L2).
__device__ __forceinline__ uint32_t ld32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.u32 %0, [%1];" : "=r"(r) : "l"(p) : "memory");
  return r;
}
__device__ __forceinline__ uint32_t ld32_nc(const void* p) {
  uint32_t r;
  asm("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ void st32(void* p, uint32_t v) {
  asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 6 bf16 (3 words) of row element e0.. of a row of length H; full: e0 + 6 <= H.
template <bool NC>
__device__ __forceinline__ void load6(const uint16_t* row, int e0, int H, bool full, uint32_t w[3]) {
  if (full) {
#pragma unroll
    for (int k = 0; k < 3; ++k) w[k] = NC ? ld32_nc(row + e0 + 2 * k) : ld32(row + e0 + 2 * k);
  } else {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int e = e0 + 2 * k;
      const uint32_t lo = e < H ? ld16(row + e) : 0u;
      const uint32_t hi = e + 1 < H ? ld16(row + e + 1) : 0u;
      w[k] = lo | (hi << 16);
    }
  }
}
__device__ __forceinline__ void store6(uint16_t* row, int e0, int H, bool full, const uint32_t w[3]) {
  if (full) {
#pragma unroll
    for (int k = 0; k < 3; ++k) st32(row + e0 + 2 * k, w[k]);
  } else {
#pragma unroll
    for (int k = 0; k < 6; ++k)
      if (e0 + k < H) row[e0 + k] = static_cast<uint16_t>(w[k >> 1] >> (16 * (k & 1)));
  }
}

// Async copies (cp.async, 16 bytes per lane, completion tracked per thread
// in commit groups) into a warp's own shared-memory ring: the loads need no
// registers, so two block groups of every slab stay in flight per warp while
// a third is summed.
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Block groups in a warp's ring, and the CTAs per SM its registers are
// bounded for: two slabs, three groups and four CTAs (62 registers); four
// slabs, three and three; eight slabs, two groups and three CTAs (70
// registers; three groups would leave room for two).  Measured on GB300
// against three groups and unbounded registers everywhere (back-to-back
// calls, same box): eight slabs 91.1 -> 86.7 us (H = 4096), 94.3 -> 90.6 us
// (H = 8192), 63.2 -> 59.8 us (the 2048-row token-split subset); two slabs
// 72.0 -> 70.6 us.
template <int PMAX>
__host__ __device__ constexpr int tag_stages() { return PMAX <= 4 ? 3 : 2; }
template <int PMAX>
constexpr int tag_min_ctas() { return PMAX <= 2 ? 4 : 3; }  // CTAs per SM the registers are bounded for
constexpr int kTagWarps = 8;
// A row is shared by kTagRowWarps warps, each streaming a contiguous share of
// its block groups; their sums of squares meet in shared memory at one CTA
// barrier per kTagRowsPerCta rows, and persistent CTAs walk the row pairs.
// Measured on GB300 (token split, two 2048-row subsets of 5120 on two
// streams, both consumer calls): a warp per row (the last of two waves of
// CTAs two-thirds full) 122.8 us; two warps per row 123.4 us; four 116.2 us;
// eight 119.6 us.
constexpr int kTagRowWarps = 4;
constexpr int kTagRowsPerCta = kTagWarps / kTagRowWarps;
template <int PMAX>
__host__ __device__ constexpr int tag_stage_bytes() { return PMAX * 32 * 16 + 384; }  // 32 blocks per slab + residual

template <int PMAX>
__global__ void __launch_bounds__(256, tag_min_ctas<PMAX>()) k_fused_tagged(FusedArgs a) {
  pdl_begin();
  extern __shared__ __align__(16) uint8_t tsmem[];
  __shared__ float red[2][kTagRowsPerCta][kTagRowWarps];  // per-warp sums of squares
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int slot = wid / kTagRowWarps, part = wid % kTagRowWarps;
  const int H = a.H;
  const int nb = (H + 5) / 6;
  const int gpr = (nb + 31) >> 5;
  const int P = a.P;
  const uint32_t epoch = a.epoch;
  constexpr int kStage = tag_stage_bytes<PMAX>();
  constexpr int kTagStages = tag_stages<PMAX>();
  uint8_t* ring = tsmem + wid * (kTagStages * kStage);
  // this warp's block groups of every row: a contiguous share of the row
  const int g0 = part * gpr / kTagRowWarps, g1 = (part + 1) * gpr / kTagRowWarps;

  int it = 0;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kTagRowsPerCta; base < a.rows;
       base += static_cast<int64_t>(gridDim.x) * kTagRowsPerCta, ++it) {
    const int64_t row = base + slot;
    const bool live = row < a.rows;  // warp-uniform
    const uint16_t* rr = static_cast<const uint16_t*>(a.res_in) + row * H;
    uint16_t* ro = static_cast<uint16_t*>(a.res_out) + row * H;
    float ss = 0.0f;
    int64_t first_bad = LLONG_MAX;
    if (live) {
      // every lane copies its own block of each slab and 16 bytes of the
      // group's residual chunk (384 bytes = 32 lanes x 6 bf16, 16-byte aligned)
      auto issue = [&](int gi) {
        if (gi < g1) {
          uint8_t* st = ring + ((gi - g0) % kTagStages) * kStage;
          const int j = gi * 32 + lane;
          if (j < nb) {
#pragma unroll
            for (int p = 0; p < PMAX; ++p)
              if (p < P)
                cp_async16(st + (p * 32 + lane) * 16, static_cast<const uint4*>(a.s.codes[p]) + row * nb + j);
          }
          const int rbytes = 2 * H - 384 * gi < 384 ? 2 * H - 384 * gi : 384;
          if (16 * lane < rbytes)
            cp_async16(st + PMAX * 512 + 16 * lane, reinterpret_cast<const uint8_t*>(rr) + 384 * gi + 16 * lane);
        }
        cp_async_commit();  // one commit group per block group (possibly empty)
      };
#pragma unroll
      for (int k = 0; k < kTagStages - 1; ++k) issue(g0 + k);
      for (int gi = g0; gi < g1; ++gi) {
        issue(gi + kTagStages - 1);
        cp_async_wait<kTagStages - 1>();  // this lane's copies of group gi have landed
        __syncwarp();                     // and every lane's (the residual chunk is shared)
        const uint8_t* st = ring + ((gi - g0) % kTagStages) * kStage;
        const int j = gi * 32 + lane;
        if (j < nb) {
          const int e0 = 6 * j;
          const bool full = e0 + 6 <= H;
          float acc[6] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int p = 0; p < PMAX; ++p) {
            if (p < P) {
              const uint4 bp = *reinterpret_cast<const uint4*>(st + (p * 32 + lane) * 16);
              if (bp.w == epoch) {
                const uint32_t w[3] = {bp.x, bp.y, bp.z};
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                  const float2 t = padd(make_float2(acc[2 * k], acc[2 * k + 1]),
                                        make_float2(bf_lo(w[k]), bf_hi(w[k])));
                  acc[2 * k] = t.x, acc[2 * k + 1] = t.y;
                }
              } else {
                const int64_t idx = (static_cast<int64_t>(p) * a.rows + row) * nb + j;
                first_bad = idx < first_bad ? idx : first_bad;
              }
            }
          }
          const uint8_t* rs = st + PMAX * 512 + 12 * lane;  // this lane's 6 residual values
          uint32_t rw[3];
          if (full) {
#pragma unroll
            for (int k = 0; k < 3; ++k) rw[k] = *reinterpret_cast<const uint32_t*>(rs + 4 * k);
          } else {
#pragma unroll
            for (int k = 0; k < 3; ++k) {
              const int e = e0 + 2 * k;
              const uint32_t lo = e < H ? *reinterpret_cast<const uint16_t*>(rs + 4 * k) : 0u;
              const uint32_t hi = e + 1 < H ? *reinterpret_cast<const uint16_t*>(rs + 4 * k + 2) : 0u;
              rw[k] = lo | (hi << 16);
            }
          }
          uint32_t hw[3];
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            const float2 h = padd(make_float2(acc[2 * k], acc[2 * k + 1]),
                                  make_float2(bf_lo(rw[k]), bf_hi(rw[k])));
            hw[k] = pack_bf2(h.x, h.y);
            const float h0 = bf_lo(hw[k]), h1 = bf_hi(hw[k]);
            ss = __fmaf_rn(h0, h0, ss);
            ss = __fmaf_rn(h1, h1, ss);
          }
          store6(ro, e0, H, full, hw);
        }
        __syncwarp();  // every lane is done with this slot before it is refilled
      }
      cp_async_wait<0>();
    }
    ss = warp_sum(ss);
    // first failing block of this warp's share (lanes agree via a min-reduction)
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      const int64_t o = __shfl_xor_sync(kFull, first_bad, m);
      first_bad = o < first_bad ? o : first_bad;
    }
    if (lane == 0 && first_bad != LLONG_MAX && a.status) {
      atomicCAS(a.status, 0, 3 /* FC_ERR_STALE_BLOCK */);
      atomicMin(a.status + 1, first_bad < INT_MAX ? static_cast<int>(first_bad) : INT_MAX - 1);
    }
    // the row's sum of squares from its warps' shares, in share order
    if (lane == 0) red[it & 1][slot][part] = ss;
    __syncthreads();
    if (!live) continue;
    float tot = 0.0f;
#pragma unroll
    for (int q = 0; q < kTagRowWarps; ++q) tot += red[it & 1][slot][q];
    const float inv = inv_rms(tot, 1.0f / static_cast<float>(H), a.eps);
    // pass 2 in batches of kOutBatch block groups: all their loads (h, which
    // this lane wrote above and is in L2, and gamma) are issued before any
    // is used, so the L2 latency is paid once per batch
    constexpr int kOutBatch = 4;
    for (int gb = g0; gb < g1; gb += kOutBatch) {
      uint32_t hw[kOutBatch][3], gw[kOutBatch][3];
#pragma unroll
      for (int u = 0; u < kOutBatch; ++u) {
        const int j = (gb + u) * 32 + lane;
        if (gb + u < g1 && j < nb) {
          const int e0 = 6 * j;
          load6<false>(ro, e0, H, e0 + 6 <= H, hw[u]);
          load6<true>(static_cast<const uint16_t*>(a.gamma), e0, H, e0 + 6 <= H, gw[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kOutBatch; ++u) {
        const int j = (gb + u) * 32 + lane;
        if (gb + u < g1 && j < nb) {
          const int e0 = 6 * j;
          uint32_t yw[3];
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            const float2 y = pmul(make_float2(fma_bf_lo(hw[u][k], gw[u][k], -0.0f),
                                              fma_bf_hi(hw[u][k], gw[u][k], -0.0f)),
                                  dup2(inv));
            yw[k] = pack_bf2(y.x, y.y);
          }
          store6(static_cast<uint16_t*>(a.y) + row * H, e0, H, e0 + 6 <= H, yw);
        }
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
  return launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(threads), 0, st, a);
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

template <int PMAX>
int tagged_occupancy() {
  constexpr int smem = kTagWarps * tag_stages<PMAX>() * tag_stage_bytes<PMAX>();
  static int occ = 0;
  if (!occ) {
    cudaFuncSetAttribute(k_fused_tagged<PMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_fused_tagged<PMAX>, kTagWarps * 32, smem) !=
            cudaSuccess || occ < 1)
      occ = 1;
  }
  return occ;
}

template <int PMAX>
cudaError_t launch_tagged_p(const FusedArgs& a, int max_ctas, cudaStream_t st) {
  constexpr int smem = kTagWarps * tag_stages<PMAX>() * tag_stage_bytes<PMAX>();
  int64_t grid = static_cast<int64_t>(num_sms()) * tagged_occupancy<PMAX>();
  const int64_t need = (a.rows + kTagRowsPerCta - 1) / kTagRowsPerCta;
  if (grid > need) grid = need;
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  return launch_pdl(k_fused_tagged<PMAX>, dim3(static_cast<unsigned>(grid)), dim3(kTagWarps * 32), smem,
                    st, a);
}

cudaError_t launch_tagged(const FusedArgs& a, int max_ctas, cudaStream_t st) {
  if (a.P <= 2) return launch_tagged_p<2>(a, max_ctas, st);
  if (a.P <= 4) return launch_tagged_p<4>(a, max_ctas, st);
  return launch_tagged_p<8>(a, max_ctas, st);
}

}  // namespace

// Rows the chosen fused kernel processes concurrently on the current device.
int64_t fused_wave_rows(int fmt, const FusedArgs& a) {
  if (fmt == kTAGGED) {
    const int occ = a.P <= 2 ? tagged_occupancy<2>() : a.P <= 4 ? tagged_occupancy<4>() : tagged_occupancy<8>();
    return static_cast<int64_t>(num_sms()) * occ * kTagRowsPerCta;  // kTagRowWarps warps per row
  }
  if (fused_tma_eligible(fmt, a)) return fused_tma_wave_rows(fmt, a);
  if (fmt == kINT8T || fmt == kINT4T) return 0;
  const int cpr = a.H >> 4;
  int nch = 1;
  while (nch < 8 && (cpr + nch - 1) / nch > 256) nch <<= 1;
  const int threads = round_warp((cpr + nch - 1) / nch);
  const void* k = nullptr;
  if (fmt == kBF16) k = reinterpret_cast<const void*>(k_fused<kBF16, 1>);
  else if (fmt == kINT8) k = reinterpret_cast<const void*>(k_fused<kINT8, 1>);
  else k = reinterpret_cast<const void*>(k_fused<kINT4, 1>);
  return static_cast<int64_t>(num_sms()) * occupancy(k, threads);
}

cudaError_t launch_fused(int fmt, const FusedArgs& a, int max_ctas, int path, cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  if (fmt == kINT8T || fmt == kINT4T) {  // staged kernel only
    if (path == kPathStream || !fused_tma_eligible(fmt, a)) return cudaErrorNotSupported;
    return launch_fused_tma(fmt, a, max_ctas, st);
  }
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
