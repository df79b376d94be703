// fused_tma.cu -- the fused reduce + requant + residual add + RMSNorm with
// TMA-staged rows.
//
// Same arithmetic as k_fused (fused.cu), different data movement: one CTA
// owns one token row at a time, and one elected thread streams the CTA's
// NEXT row -- every slab's codes, scales and zero-points (or bf16 data) and
// the residual -- into a ring of NSTAGE shared-memory stages with 1-D bulk
// copies (cp.async.bulk) that complete on an mbarrier.  While those bytes
// are in flight, all threads work on the current row out of shared memory.
// The bf16 row h (residual + reduced value) goes to a shared-memory row
// buffer, so nothing row-sized is held in registers and
// occupancy is set by shared memory alone.
//
// Stage layout (every piece a multiple of 16 bytes, 16-byte aligned):
//   [codes of slab 0..P-1][scales 0..P-1][zeros 0..P-1 (INT4)][residual]
#include <climits>

#include "device.cuh"
#include "internal.h"

namespace fc {

namespace {

constexpr int kTmaThreadsMax = 512;  // threads per CTA at most
constexpr int kGammaRegChunks = 2;   // gamma chunks a thread keeps in registers

struct TmaGeom {
  int cb;           // code (or bf16 data) bytes of one slab row
  int sb;           // scale bytes of one slab row (0 for bf16)
  int zb;           // zero-point bytes of one slab row (INT4 only)
  int stage_bytes;  // P * (cb + sb + zb) + 2H
  int gamma_off;    // byte offset of the h row buffer in dynamic smem
  int stage_off;    // byte offset of stage 0
};

template <int FMT>
__device__ __forceinline__ void issue_row(const FusedArgs& a, const TmaGeom& g, uint8_t* st,
                                          uint64_t* bar, int64_t row) {
  mbar_expect_tx(bar, static_cast<uint32_t>(g.stage_bytes));
  const int P = a.P;
  for (int p = 0; p < P; ++p) {
    bulk_load(st + p * g.cb, static_cast<const uint8_t*>(a.s.codes[p]) + row * g.cb, g.cb, bar);
    if (FMT == kINT8 || FMT == kINT4)
      bulk_load(st + P * g.cb + p * g.sb,
                reinterpret_cast<const uint8_t*>(a.s.scales[p]) + row * g.sb, g.sb, bar);
    if (FMT == kINT4)
      bulk_load(st + P * (g.cb + g.sb) + p * g.zb,
                reinterpret_cast<const uint8_t*>(a.s.zeros[p]) + row * g.zb, g.zb, bar);
  }
  bulk_load(st + P * (g.cb + g.sb + g.zb), static_cast<const uint8_t*>(a.res_in) + row * 2 * a.H,
            2 * a.H, bar);
}

template <int FMT, int NSTAGE, int PMAX>
__global__ void __launch_bounds__(kTmaThreadsMax) k_fused_tma(FusedArgs a, TmaGeom g) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float red[2][32];
  __shared__ uint64_t bar[NSTAGE];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  const int nthr = blockDim.x;
  const int H = a.H, cpr = H >> 4, P = a.P;
  const int lpg = a.G >> 4, sh = a.lpg_shift;
  // h (the bf16 row) lives in its own buffer: each thread reads back only the
  // chunks it wrote, so it needs no barrier and frees the stage early.
  uint16_t* hbuf = reinterpret_cast<uint16_t*>(smem + g.gamma_off);
  uint8_t* stage0 = smem + g.stage_off;
  const int64_t row0 = blockIdx.x, rstride = gridDim.x;
  if (row0 >= a.rows) return;
  // tagged quantized formats decode to the plain ones
  constexpr int BASE = FMT == kINT8T ? kINT8 : FMT == kINT4T ? kINT4 : FMT;
  constexpr bool QTAG = FMT == kINT8T || FMT == kINT4T;
  const int64_t bpr = g.cb / 16;  // tagged blocks per row and slab

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bar[s], 1);
    mbar_init_fence();
    for (int s = 0; s < NSTAGE; ++s)
      if (row0 + s * rstride < a.rows)
        issue_row<FMT>(a, g, stage0 + s * g.stage_bytes, &bar[s], row0 + s * rstride);
  }
  __syncthreads();

  // gamma of this thread's first chunks, read once: every row uses the same chunks
  uint32_t greg[kGammaRegChunks][8];
#pragma unroll
  for (int j = 0; j < kGammaRegChunks; ++j) {
    const int c = tid + j * nthr;
    if (c < cpr) {
      const V8 gv = ld256_keep(static_cast<const uint16_t*>(a.gamma) + c * 16);
#pragma unroll
      for (int k = 0; k < 8; ++k) greg[j][k] = gv.w[k];
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) greg[j][k] = 0u;
    }
  }

  bool all_ok = true;
  int i = 0;
  for (int64_t row = row0; row < a.rows; row += rstride, ++i) {
    const int s = i % NSTAGE;
    const uint8_t* st = stage0 + s * g.stage_bytes;
    const bool ok = mbar_wait_bounded(&bar[s], (i / NSTAGE) & 1);
    const uint8_t* codes = st;
    const float* scales = reinterpret_cast<const float*>(st + P * g.cb);
    const float* zeros = reinterpret_cast<const float*>(st + P * (g.cb + g.sb));
    const uint4* rrow = reinterpret_cast<const uint4*>(st + P * (g.cb + g.sb + g.zb));

    // ---- pass 1: reduce, requantize, dequantize, residual add (h -> hbuf).
    // Every thread runs the same number of iterations so whole warps join
    // the group shuffles; lanes past the row end feed zeros (their groups
    // hold no real element) and touch no memory.
    float2 ss2 = make_float2(0.0f, 0.0f);
    int64_t first_bad = LLONG_MAX;
    for (int cbase = 0; cbase < cpr; cbase += nthr) {
      const int c = cbase + tid;
      const bool act = c < cpr;
      float acc[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
#pragma unroll
      for (int p = 0; p < PMAX; ++p) {
        if (p < P && act) {
          if (FMT == kBF16) {
            const uint4* x = reinterpret_cast<const uint4*>(codes + p * g.cb) + 2 * c;
            const uint4 x0 = x[0], x1 = x[1];
            const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float2 t = padd(make_float2(acc[2 * k], acc[2 * k + 1]),
                                    make_float2(bf_lo(w[k]), bf_hi(w[k])));
              acc[2 * k] = t.x, acc[2 * k + 1] = t.y;
            }
          } else if (FMT == kINT8T) {
            // group c>>3, lane k = c&7: code bytes 16k.. = words o.. of blocks b0, b0+1
            const int gl = c >> 3, k = c & 7, b0 = (4 * k) / 3, o = 4 * k - 3 * b0;
            const uint4* gb = reinterpret_cast<const uint4*>(codes + p * g.cb) + gl * kBlocksPerGroupI8;
            const uint4 B0 = gb[b0], B1 = gb[b0 + 1], BS = gb[kBlocksPerGroupI8 - 1];
            if (B0.w == a.epoch && B1.w == a.epoch && BS.w == a.epoch) {
              const uint32_t W[6] = {B0.x, B0.y, B0.z, B1.x, B1.y, B1.z};
              const uint32_t w[4] = {o == 0 ? W[0] : o == 1 ? W[1] : W[2],
                                     o == 0 ? W[1] : o == 1 ? W[2] : W[3],
                                     o == 0 ? W[2] : o == 1 ? W[3] : W[4],
                                     o == 0 ? W[3] : o == 1 ? W[4] : W[5]};
              dequant_i8_acc(w, __uint_as_float(BS.z), acc);
            } else {
              const int64_t base = (static_cast<int64_t>(p) * a.rows + row) * bpr + gl * kBlocksPerGroupI8;
              const int64_t bad = base + (B0.w != a.epoch ? b0 : B1.w != a.epoch ? b0 + 1 : kBlocksPerGroupI8 - 1);
              first_bad = bad < first_bad ? bad : first_bad;
            }
          } else if (FMT == kINT4T) {
            // group c>>1: block 0 = {codes 0-3, 4-7, 8-11}, block 1 = {codes 12-15, scale, zero}
            const int gl = c >> 1, k = c & 1;
            const uint4* gb = reinterpret_cast<const uint4*>(codes + p * g.cb) + gl * kBlocksPerGroupI4;
            const uint4 B0 = gb[0], B1 = gb[1];
            if (B0.w == a.epoch && B1.w == a.epoch) {
              const uint32_t w[2] = {k ? B0.z : B0.x, k ? B1.x : B0.y};
              dequant_i4_acc(w, __uint_as_float(B1.y), __uint_as_float(B1.z), acc);
            } else {
              const int64_t bad = (static_cast<int64_t>(p) * a.rows + row) * bpr + gl * kBlocksPerGroupI4 +
                                  (B0.w != a.epoch ? 0 : 1);
              first_bad = bad < first_bad ? bad : first_bad;
            }
          } else if (FMT == kINT8) {
            const uint4 q = reinterpret_cast<const uint4*>(codes + p * g.cb)[c];
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
            dequant_i8_acc(w, scales[p * (g.sb >> 2) + (c >> sh)], acc);
          } else {
            const uint2 q = reinterpret_cast<const uint2*>(codes + p * g.cb)[c];
            const uint32_t w[2] = {q.x, q.y};
            const int gi = p * (g.sb >> 2) + (c >> sh);
            dequant_i4_acc(w, scales[gi], zeros[gi], acc);
          }
        }
      }
      const int64_t gc = row * cpr + c;
      const int64_t gg = gc >> sh;
      if (BASE == kINT8) {
        uint32_t q[4];
        const float s8 = quant_i8<true>(acc, lpg, q, acc);
        if (act && a.rq_codes) {
          st128(static_cast<int8_t*>(a.rq_codes) + gc * 16, make_uint4(q[0], q[1], q[2], q[3]));
          if ((lane & (lpg - 1)) == 0) stf(a.rq_scales + gg, s8);
        }
      } else if (BASE == kINT4) {
        uint32_t q[2];
        float z;
        const float s4 = quant_i4<true>(acc, lpg, q, z, acc);
        if (act && a.rq_codes) {
          st64(static_cast<uint8_t*>(a.rq_codes) + gc * 8, make_uint2(q[0], q[1]));
          if ((lane & (lpg - 1)) == 0) {
            stf(a.rq_scales + gg, s4);
            stf(a.rq_zeros + gg, z);
          }
        }
      }
      if (act) {
        // h = bf16(fl(o + R)) straight from the packed residual; sum of h^2
        // straight from the packed h
        const uint4 r0 = rrow[2 * c], r1 = rrow[2 * c + 1];
        const uint32_t rw[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        V8 hv;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          hv.w[k] = pack_bf2(add_bf_lo(rw[k], acc[2 * k]), add_bf_hi(rw[k], acc[2 * k + 1]));
        uint4* hp = reinterpret_cast<uint4*>(hbuf) + 2 * c;
        hp[0] = make_uint4(hv.w[0], hv.w[1], hv.w[2], hv.w[3]);
        hp[1] = make_uint4(hv.w[4], hv.w[5], hv.w[6], hv.w[7]);
        st256(static_cast<uint16_t*>(a.res_out) + gc * 16, hv);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          ss2.x = fma_bf_lo(hv.w[k], hv.w[k], ss2.x);
          ss2.y = fma_bf_hi(hv.w[k], hv.w[k], ss2.y);
        }
      }
    }

    if (QTAG) {  // the row's first failing block (if any) -> status
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
        const int64_t o2 = __shfl_xor_sync(kFull, first_bad, m);
        first_bad = o2 < first_bad ? o2 : first_bad;
      }
      if (lane == 0 && first_bad != LLONG_MAX && a.status) {
        atomicCAS(a.status, 0, 3 /* FC_ERR_STALE_BLOCK */);
        atomicMin(a.status + 1, first_bad < INT_MAX ? static_cast<int>(first_bad) : INT_MAX - 1);
      }
    }
    // ---- the row's only barrier: sum of squares + vote on the staged copy
    float v = warp_sum(__fadd_rn(ss2.x, ss2.y));
    if (lane == 0) red[i & 1][wid] = v;
    all_ok = __syncthreads_and(ok) != 0;
    if (!all_ok) break;
    float tot = 0.0f;
    for (int w = 0; w < nw; ++w) tot += red[i & 1][w];
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, static_cast<float>(H)), a.eps)));

    // every thread is past its reads of stage s: refill it NSTAGE rows ahead
    if (tid == 0) {
      const int64_t nrow = row + NSTAGE * rstride;
      if (nrow < a.rows) {
        fence_proxy_async_smem();
        issue_row<FMT>(a, g, stage0 + s * g.stage_bytes, &bar[s], nrow);
      }
    }

    // ---- pass 2: y = bf16(fl(h * gamma) * inv); h * gamma is exact in binary32
    auto out_chunk = [&](int c, const uint32_t gw[8]) {
      const uint4* hp = reinterpret_cast<const uint4*>(hbuf) + 2 * c;
      const uint4 h0 = hp[0], h1 = hp[1];
      const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
      V8 yv;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 y = pmul(make_float2(fma_bf_lo(hw[k], gw[k], -0.0f), fma_bf_hi(hw[k], gw[k], -0.0f)),
                              dup2(inv));
        yv.w[k] = pack_bf2(y.x, y.y);
      }
      st256(static_cast<uint16_t*>(a.y) + (row * cpr + c) * 16, yv);
    };
#pragma unroll
    for (int j = 0; j < kGammaRegChunks; ++j)
      if (tid + j * nthr < cpr) out_chunk(tid + j * nthr, greg[j]);
    for (int c = tid + kGammaRegChunks * nthr; c < cpr; c += nthr) {
      const V8 gv = ld256_keep(static_cast<const uint16_t*>(a.gamma) + c * 16);
      out_chunk(c, gv.w);
    }
  }
  if (!all_ok && tid == 0) {
    // a staged copy did not land within the bound: report it and give the
    // copies still in flight one more bounded wait before the CTA exits
    if (a.status) atomicExch(a.status, 2 /* FC_ERR_CUDA */);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_wait_bounded(&bar[s], 0);
      mbar_wait_bounded(&bar[s], 1);
    }
  }
}

int geometry(int fmt, const FusedArgs& a, TmaGeom& g) {
  const int H = a.H, P = a.P;
  if (fmt == kBF16) {
    g.cb = 2 * H, g.sb = 0, g.zb = 0;
  } else if (fmt == kINT8T) {
    g.cb = (H / 128) * kBlocksPerGroupI8 * 16, g.sb = 0, g.zb = 0;
  } else if (fmt == kINT4T) {
    g.cb = (H / 32) * kBlocksPerGroupI4 * 16, g.sb = 0, g.zb = 0;
  } else {
    g.cb = fmt == kINT8 ? H : H / 2;
    g.sb = (H / a.G) * 4;
    g.zb = fmt == kINT4 ? g.sb : 0;
  }
  if (g.cb % 16 || g.sb % 16 || g.zb % 16) return 0;
  g.stage_bytes = P * (g.cb + g.sb + g.zb) + 2 * H;
  g.gamma_off = 0;
  g.stage_off = (2 * H + 127) & ~127;
  return 1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch shape of one instantiation: threads per CTA and resident CTAs per SM.
struct TmaShape {
  int nstage = 0, threads = 0, occ = 0, smem = 0;
};

// Threads per CTA, from the work a thread does per row and barrier (measured
// on GB300 across the message-size sweep): where a chunk carries little
// arithmetic (INT4, INT8 with up to four slabs) two 16-element chunks per
// thread and row; where it carries more (INT8 with more slabs) or the row is
// plain bf16, up to 256 threads, i.e. one chunk per thread for rows up to
// 4096 elements.
int tma_threads(int fmt, int P, int H) {
  const int cpr = H >> 4;
  const bool heavy = fmt == kBF16 || ((fmt == kINT8 || fmt == kINT8T) && P > 4);
  int t = heavy ? (cpr < 256 ? cpr : 256) : (cpr + 1) / 2;
  t = (t + 31) & ~31;
  return t < 32 ? 32 : (t > kTmaThreadsMax ? kTmaThreadsMax : t);
}

template <int FMT, int NSTAGE, int PMAX>
TmaShape shape_t(const FusedArgs& a, const TmaGeom& g) {
  TmaShape sh;
  sh.nstage = NSTAGE;
  sh.smem = g.stage_off + NSTAGE * g.stage_bytes;
  if (sh.smem > kTmaSmemLimit) return sh;
  auto kern = k_fused_tma<FMT, NSTAGE, PMAX>;
  static int configured_smem[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  dev = dev < 64 ? dev : 63;
  if (configured_smem[dev] < sh.smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, sh.smem) != cudaSuccess)
      return sh;
    configured_smem[dev] = sh.smem;
  }
  sh.threads = tma_threads(FMT, a.P, a.H);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&sh.occ, kern, sh.threads, sh.smem) != cudaSuccess)
    sh.occ = 0;
  return sh;
}

// A two-row ring (the next row streams in while this one is computed).  For
// the quantized formats, when that ring leaves room for a single CTA per SM,
// two single-stage CTAs (which overlap each other's copies and row
// barriers) were measured faster; for bf16 rows the two-row ring stays.
template <int FMT, int PMAX>
TmaShape choose_shape(const FusedArgs& a, const TmaGeom& g) {
  const TmaShape two = shape_t<FMT, 2, PMAX>(a, g);
  if (FMT == kBF16 && two.occ >= 1) return two;
  const TmaShape one = shape_t<FMT, 1, PMAX>(a, g);
  if (two.occ >= 1 && (two.occ >= 2 || one.occ <= two.occ)) return two;
  return one;
}

template <int FMT, int PMAX>
cudaError_t launch_tma_p(const FusedArgs& a, const TmaGeom& g, int max_ctas, cudaStream_t st) {
  const TmaShape sh = choose_shape<FMT, PMAX>(a, g);
  if (sh.occ < 1) return cudaErrorInvalidConfiguration;
  int64_t grid = static_cast<int64_t>(num_sms()) * sh.occ;
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  if (grid > a.rows) grid = a.rows;
  const dim3 gr(static_cast<unsigned>(grid));
  if (sh.nstage == 2)
    k_fused_tma<FMT, 2, PMAX><<<gr, sh.threads, sh.smem, st>>>(a, g);
  else
    k_fused_tma<FMT, 1, PMAX><<<gr, sh.threads, sh.smem, st>>>(a, g);
  return cudaGetLastError();
}

// The slab loop is unrolled to PMAX (2, 4 or 8) slots, so no instruction is
// spent on slots beyond P when P is 2, 4 or 8.
template <int FMT>
cudaError_t launch_tma_fmt(const FusedArgs& a, const TmaGeom& g, int max_ctas, cudaStream_t st) {
  if (a.P <= 2) return launch_tma_p<FMT, 2>(a, g, max_ctas, st);
  if (a.P <= 4) return launch_tma_p<FMT, 4>(a, g, max_ctas, st);
  return launch_tma_p<FMT, 8>(a, g, max_ctas, st);
}

}  // namespace

bool fused_tma_eligible(int fmt, const FusedArgs& a) {
  if (fmt != kBF16 && fmt != kINT8 && fmt != kINT4 && fmt != kINT8T && fmt != kINT4T) return false;
  TmaGeom g;
  if (!geometry(fmt, a, g)) return false;
  if (g.stage_off + g.stage_bytes > kTmaSmemLimit) return false;
  for (int p = 0; p < a.P; ++p) {
    if (!aligned16(a.s.codes[p])) return false;
    if ((fmt == kINT8 || fmt == kINT4) && !aligned16(a.s.scales[p])) return false;
    if (fmt == kINT4 && !aligned16(a.s.zeros[p])) return false;
  }
  return aligned16(a.res_in) && aligned16(a.gamma);
}

template <int FMT>
int64_t wave_fmt(const FusedArgs& a, const TmaGeom& g) {
  const TmaShape sh = a.P <= 2 ? choose_shape<FMT, 2>(a, g)
                      : a.P <= 4 ? choose_shape<FMT, 4>(a, g)
                                 : choose_shape<FMT, 8>(a, g);
  return static_cast<int64_t>(num_sms()) * (sh.occ > 0 ? sh.occ : 1);  // a CTA per row
}

int64_t fused_tma_wave_rows(int fmt, const FusedArgs& a) {
  TmaGeom g;
  geometry(fmt, a, g);
  if (fmt == kBF16) return wave_fmt<kBF16>(a, g);
  if (fmt == kINT8) return wave_fmt<kINT8>(a, g);
  if (fmt == kINT8T) return wave_fmt<kINT8T>(a, g);
  if (fmt == kINT4T) return wave_fmt<kINT4T>(a, g);
  return wave_fmt<kINT4>(a, g);
}

cudaError_t launch_fused_tma(int fmt, const FusedArgs& a, int max_ctas, cudaStream_t st) {
  TmaGeom g;
  geometry(fmt, a, g);
  switch (fmt) {
    case kBF16: return launch_tma_fmt<kBF16>(a, g, max_ctas, st);
    case kINT8: return launch_tma_fmt<kINT8>(a, g, max_ctas, st);
    case kINT8T: return launch_tma_fmt<kINT8T>(a, g, max_ctas, st);
    case kINT4T: return launch_tma_fmt<kINT4T>(a, g, max_ctas, st);
    default: return launch_tma_fmt<kINT4>(a, g, max_ctas, st);
  }
}

}  // namespace fc
