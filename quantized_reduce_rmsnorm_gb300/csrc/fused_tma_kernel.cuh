// fused_tma_kernel.cuh -- the TMA-staged fused kernel (template), shared by
// the one-CTA-per-row launches (fused_tma.cu) and the thread-block-cluster
// launches that split rows across CTAs (fused_tma_cluster.cu).
//
// Same arithmetic as k_fused (fused.cu), different data movement: one CTA
// (or, with CL > 1, one cluster of CL CTAs, each owning a contiguous segment
// of the row) works on one token row at a time, and one elected thread
// streams the CTA's NEXT rows -- every slab's codes, scales and zero-points
// (or bf16 data) and the residual, for its segment -- into a ring of NSTAGE
// shared-memory stages with 1-D bulk copies (cp.async.bulk) that complete on
// an mbarrier.  While those bytes are in flight, all threads work on the
// current row out of shared memory.  The bf16 row h (residual + reduced
// value) goes to a shared-memory row buffer, so nothing row-sized is held in
// registers and occupancy is set by shared memory alone.
//
// Stage layout (every piece a multiple of 16 bytes, 16-byte aligned):
//   [codes of slab 0..P-1][scales 0..P-1][zeros 0..P-1 (INT4)][residual]
#pragma once

#include <climits>

#include "device.cuh"
#include "internal.h"

namespace fc {

constexpr int kTmaThreadsMax = 512;  // threads per CTA at most
constexpr int kGammaRegChunks = 2;   // gamma chunks a thread keeps in registers

// A CTA's share of a row is a segment of cps chunks (the whole row when the
// CTA is not in a cluster); segment r of a row starts r * cb code bytes,
// r * sb scale bytes and r * 32 * cps residual bytes into it.
struct TmaGeom {
  int cb;           // code (or bf16 data, or tagged block) bytes of one slab's segment
  int sb;           // scale bytes of one slab's segment (0 for bf16 and tagged)
  int zb;           // zero-point bytes of one slab's segment (INT4 only)
  int row_cb;       // code bytes of one slab row (its row stride)
  int row_sb;       // scale (and zero-point) bytes of one slab row
  int cps;          // chunks (16 elements) in the segment
  int stage_bytes;  // P * (cb + sb + zb) + 32 * cps
  int gamma_off;    // byte offset of the h segment buffer in dynamic smem
  int stage_off;    // byte offset of stage 0
};

// The compact build (fused_tma_compact.cu): resident CTAs per SM of the
// instantiation for (fmt, P, nstage) at `threads` threads and `smem` bytes
// (0 when it cannot run), and its launch.
int fused_tma_compact_occupancy(int fmt, int P, int nstage, int threads, int smem);
cudaError_t launch_fused_tma_compact(int fmt, int nstage, const FusedArgs& a, const TmaGeom& g,
                                     int threads, int smem, int64_t grid, cudaStream_t st);

// The compact build with the residual left out of the stage, for shapes of
// the quantized formats (fused_tma_rg.cu): resident CTAs per SM of the
// instantiation for (fmt, P, nstage, sub, with or without the h row buffer)
// at `threads` threads and `smem` bytes (0 when that combination is not
// built), and its launch.
int fused_tma_rg_occupancy(int fmt, int P, int nstage, int sub, bool hb, int threads, int smem);
cudaError_t launch_fused_tma_rg(int fmt, int nstage, int sub, bool hb, const FusedArgs& a, const TmaGeom& g,
                                int threads, int smem, int64_t grid, cudaStream_t st);

namespace {

template <int FMT, bool RG = false>
__device__ __forceinline__ void issue_row(const FusedArgs& a, const TmaGeom& g, uint8_t* st,
                                          uint64_t* bar, int64_t row, int rank) {
  mbar_expect_tx(bar, static_cast<uint32_t>(g.stage_bytes));
  const int P = a.P;
  const int64_t co = row * g.row_cb + static_cast<int64_t>(rank) * g.cb;
  const int64_t so = row * g.row_sb + static_cast<int64_t>(rank) * g.sb;
  for (int p = 0; p < P; ++p) {
    bulk_load(st + p * g.cb, static_cast<const uint8_t*>(a.s.codes[p]) + co, g.cb, bar);
    if (FMT == kINT8 || FMT == kINT4)
      bulk_load(st + P * g.cb + p * g.sb, reinterpret_cast<const uint8_t*>(a.s.scales[p]) + so, g.sb,
                bar);
    if (FMT == kINT4)
      bulk_load(st + P * (g.cb + g.sb) + p * g.zb, reinterpret_cast<const uint8_t*>(a.s.zeros[p]) + so,
                g.zb, bar);
  }
  if (!RG)
    bulk_load(st + P * (g.cb + g.sb + g.zb),
              static_cast<const uint8_t*>(a.res_in) + row * 2 * a.H + static_cast<int64_t>(rank) * 32 * g.cps,
              32 * g.cps, bar);
}

// L2 prefetch of the bytes issue_row copies (issued before pdl_begin()).
template <int FMT>
__device__ __forceinline__ void prefetch_row(const FusedArgs& a, const TmaGeom& g, int64_t row, int rank) {
  const int P = a.P;
  const int64_t co = row * g.row_cb + static_cast<int64_t>(rank) * g.cb;
  const int64_t so = row * g.row_sb + static_cast<int64_t>(rank) * g.sb;
  for (int p = 0; p < P; ++p) {
    prefetch_l2(static_cast<const uint8_t*>(a.s.codes[p]) + co, g.cb);
    if (FMT == kINT8 || FMT == kINT4) prefetch_l2(reinterpret_cast<const uint8_t*>(a.s.scales[p]) + so, g.sb);
    if (FMT == kINT4) prefetch_l2(reinterpret_cast<const uint8_t*>(a.s.zeros[p]) + so, g.zb);
  }
  prefetch_l2(static_cast<const uint8_t*>(a.res_in) + row * 2 * a.H + static_cast<int64_t>(rank) * 32 * g.cps,
              32 * g.cps);
}

// Thread-block clusters: the CTA's rank, a barrier over the whole cluster
// (release/acquire: shared-memory writes before it are visible to every CTA
// after it), and stores into a peer CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
__device__ __forceinline__ uint32_t peer_smem(const void* p, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_u32(p)), "r"(rank));
  return d;
}
__device__ __forceinline__ void st_peer_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_peer_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// CL: CTAs per row (a cluster of CL CTAs shares each row, CTA r owning
// chunks [r * cps, (r + 1) * cps); 1: a CTA per row).
// COMPACT: built for at most 256 threads and three CTAs per SM (about 80
// registers, a few values spilled), for shapes where shared memory admits
// more CTAs than the full register budget does.
// SUB: sub-stages per stage (CL == 1 only).  With SUB > 1 the geometry g
// describes one of SUB equal segments of the row, each stage is SUB
// segment-sized sub-stages on their own mbarriers, and the CTA's threads take
// one segment per pass-1 iteration (blockDim.x == g.cps): a sub-stage is
// refilled with the next row as soon as every thread is past it, instead of
// after the whole row, so the next row's bytes have longer to land.
// RG: the residual is not staged; each thread loads its chunk of it straight
// from global memory before the chunk's slab loop, whose work hides the
// load.  Its stage is 2 * H bytes smaller, which is what lets a second CTA
// per SM fit for eight tagged INT8 slabs at H = 8192, and a sixth for two
// tagged INT4 slabs at H = 4096.
// HB: h is kept in the shared-memory row buffer (else pass 2 reads each
// chunk back from residual_out, which this thread has just written and L2
// still holds: 2 * H bytes less shared memory per CTA, for one more CTA per
// SM where that buffer is what keeps it out).
template <int FMT, int NSTAGE, int PMAX, int CL = 1, bool COMPACT = false, int SUB = 1, bool RG = false,
          bool HB = true>
__global__ void __launch_bounds__(COMPACT ? 256 : kTmaThreadsMax, COMPACT ? 3 : 1)
    k_fused_tma(FusedArgs a, TmaGeom g) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float red[2][32];
  static_assert(CL == 1 || SUB == 1, "sub-stages are for a CTA per row");
  __shared__ uint64_t bar[NSTAGE * SUB];
  __shared__ float cl_tot[2][CL];       // per-CTA sums of squares of the row (cluster)
  __shared__ uint32_t cl_ok[2][CL];     // per-CTA "staged copy arrived" votes
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  const int nthr = blockDim.x;
  const int H = a.H, cpr = H >> 4, P = a.P;
  const int rank = CL > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int cps = SUB * g.cps, c0 = rank * cps;  // this CTA's chunks of every row
  const float inv_h = 1.0f / static_cast<float>(H);
  const int lpg = a.G >> 4, sh = a.lpg_shift;
  // h (the bf16 row) lives in its own buffer: each thread reads back only the
  // chunks it wrote, so it needs no barrier and frees the stage early.
  uint16_t* hbuf = reinterpret_cast<uint16_t*>(smem + g.gamma_off);
  uint8_t* stage0 = smem + g.stage_off;
  const int64_t row0 = blockIdx.x / CL, rstride = gridDim.x / CL;
  if (row0 >= a.rows) return;  // whole clusters leave together
  // tagged quantized formats decode to the plain ones
  constexpr int BASE = FMT == kINT8T ? kINT8 : FMT == kINT4T ? kINT4 : FMT;
  constexpr bool QTAG = FMT == kINT8T || FMT == kINT4T;
  const int64_t bpr = g.row_cb / 16;           // tagged blocks per row and slab
  const int64_t seg_blk = rank * (g.cb / 16);  // ... before this CTA's segment

  // tid 0's last copy into each (sub-)stage x: bit x of `used`, its phase
  // parity in `ppar`.  On a timeout tid 0 waits once for each of these: a
  // wait on the parity of the last phase returns at once if that copy has
  // landed (no later copy was issued into the stage) and otherwise waits for
  // it, bounded.  Kept in shared memory (only tid 0 touches them).
  __shared__ uint32_t used, ppar;
  auto note_issue = [&](int x, int iter) {
    used |= 1u << x;
    ppar = (ppar & ~(1u << x)) | (static_cast<uint32_t>((iter / NSTAGE) & 1) << x);
  };
  if (tid == 0) used = 0, ppar = 0;
  if (tid == 0) {
    for (int s = 0; s < NSTAGE * SUB; ++s) mbar_init(&bar[s], 1);
    mbar_init_fence();
    for (int s = 0; s < NSTAGE; ++s)
      if (row0 + s * rstride < a.rows)
        for (int j = 0; j < SUB; ++j) prefetch_row<FMT>(a, g, row0 + s * rstride, SUB > 1 ? j : rank);
  }
  if (blockIdx.x == 0 && tid == 32) prefetch_l2(a.gamma, static_cast<uint32_t>(2 * H));  // every CTA reads it
  pdl_begin();
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s)
      if (row0 + s * rstride < a.rows)
        for (int j = 0; j < SUB; ++j) {
          issue_row<FMT, RG>(a, g, stage0 + (s * SUB + j) * g.stage_bytes, &bar[s * SUB + j], row0 + s * rstride,
                         SUB > 1 ? j : rank);
          note_issue(s * SUB + j, s);
        }
  }
  __syncthreads();
  if (CL > 1) cluster_barrier();  // every CTA of the cluster runs before any peer store

  // gamma of this thread's first chunks, read once: every row uses the same chunks
  // (the compact eight-slab build without a staged residual reads gamma per
  // row from L1 instead: registers are what bounds its CTAs per SM)
  constexpr int GRC = RG && COMPACT && PMAX == 8 ? 0 : kGammaRegChunks;
  uint32_t greg[GRC > 0 ? GRC : 1][8];
#pragma unroll
  for (int j = 0; j < GRC; ++j) {
    const int c = tid + j * nthr;
    if (c < cps) {
      const V8 gv = ld256_keep(static_cast<const uint16_t*>(a.gamma) + (c0 + c) * 16);
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
    const uint32_t par = (i / NSTAGE) & 1;
    bool ok = SUB > 1 ? true : mbar_wait_bounded(&bar[s], par);

    // ---- pass 1: reduce, requantize, dequantize, residual add (h -> hbuf).
    // Every thread runs the same number of iterations so whole warps join
    // the group shuffles; lanes past the row end feed zeros (their groups
    // hold no real element) and touch no memory.
    float2 ss2 = make_float2(0.0f, 0.0f);
    int64_t first_bad = LLONG_MAX;
    for (int cbase = 0; cbase < cps; cbase += nthr) {
      const int c = cbase + tid;  // chunk of the CTA's part of the row
      const bool act = c < cps;
      const int j = SUB > 1 ? cbase / nthr : 0;  // its sub-stage
      if (SUB > 1) ok = mbar_wait_bounded(&bar[s * SUB + j], par) && ok;
      const int cs = c - j * g.cps;  // chunk within the (sub-)stage
      const uint8_t* st = stage0 + (s * SUB + j) * g.stage_bytes;
      const uint8_t* codes = st;
      const float* scales = reinterpret_cast<const float*>(st + P * g.cb);
      const float* zeros = reinterpret_cast<const float*>(st + P * (g.cb + g.sb));
      const uint4* rrow = reinterpret_cast<const uint4*>(st + P * (g.cb + g.sb + g.zb));
      V8 rv;  // RG: this chunk's residual, loaded while the slabs are summed
      if (RG && act) rv = ld256_coherent(static_cast<const uint16_t*>(a.res_in) + (row * cpr + c0 + c) * 16);
      float acc[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
#pragma unroll
      for (int p = 0; p < PMAX; ++p) {
        if (p < P && act) {
          if (FMT == kBF16) {
            const uint4* x = reinterpret_cast<const uint4*>(codes + p * g.cb) + 2 * cs;
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
            const uint4* gb = reinterpret_cast<const uint4*>(codes + p * g.cb) + (cs >> 3) * kBlocksPerGroupI8;
            const uint4 B0 = gb[b0], B1 = gb[b0 + 1], BS = gb[kBlocksPerGroupI8 - 1];
            if (B0.w == a.epoch && B1.w == a.epoch && BS.w == a.epoch) {
              const uint32_t W[6] = {B0.x, B0.y, B0.z, B1.x, B1.y, B1.z};
              const uint32_t w[4] = {o == 0 ? W[0] : o == 1 ? W[1] : W[2],
                                     o == 0 ? W[1] : o == 1 ? W[2] : W[3],
                                     o == 0 ? W[2] : o == 1 ? W[3] : W[4],
                                     o == 0 ? W[3] : o == 1 ? W[4] : W[5]};
              dequant_i8_acc(w, __uint_as_float(BS.z), acc);
            } else {
              const int64_t base = (static_cast<int64_t>(p) * a.rows + row) * bpr + seg_blk + gl * kBlocksPerGroupI8;
              const int64_t bad = base + (B0.w != a.epoch ? b0 : B1.w != a.epoch ? b0 + 1 : kBlocksPerGroupI8 - 1);
              first_bad = bad < first_bad ? bad : first_bad;
            }
          } else if (FMT == kINT4T) {
            // group c>>1: block 0 = {codes 0-3, 4-7, 8-11}, block 1 = {codes 12-15, scale, zero}
            const int gl = c >> 1, k = c & 1;
            const uint4* gb = reinterpret_cast<const uint4*>(codes + p * g.cb) + (cs >> 1) * kBlocksPerGroupI4;
            const uint4 B0 = gb[0], B1 = gb[1];
            if (B0.w == a.epoch && B1.w == a.epoch) {
              const uint32_t w[2] = {k ? B0.z : B0.x, k ? B1.x : B0.y};
              dequant_i4_acc(w, __uint_as_float(B1.y), __uint_as_float(B1.z), acc);
            } else {
              const int64_t bad = (static_cast<int64_t>(p) * a.rows + row) * bpr + seg_blk + gl * kBlocksPerGroupI4 +
                                  (B0.w != a.epoch ? 0 : 1);
              first_bad = bad < first_bad ? bad : first_bad;
            }
          } else if (FMT == kINT8) {
            const uint4 q = reinterpret_cast<const uint4*>(codes + p * g.cb)[cs];
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
            dequant_i8_acc(w, scales[p * (g.sb >> 2) + (cs >> sh)], acc);
          } else {
            const uint2 q = reinterpret_cast<const uint2*>(codes + p * g.cb)[cs];
            const uint32_t w[2] = {q.x, q.y};
            const int gi = p * (g.sb >> 2) + (cs >> sh);
            dequant_i4_acc(w, scales[gi], zeros[gi], acc);
          }
        }
      }
      const int64_t gc = row * cpr + c0 + c;
      const int64_t gg = gc >> sh;
      if (BASE == kINT8) {
        uint32_t q[4];
        // sums of up to four slabs sit next to half-integers often enough that
        // flags as a mask pay (and the compact builds have no registers for the
        // alternative); eight: flags by comparing packed words
        const float s8 = PMAX >= 8 ? requant_i8(acc, lpg, q, acc)
                                   : quant_i8<true, false, SettleHere, (PMAX <= 2)>(acc, lpg, q, acc);
        if (act && a.rq_codes) {
          st128(static_cast<int8_t*>(a.rq_codes) + gc * 16, make_uint4(q[0], q[1], q[2], q[3]));
          if ((lane & (lpg - 1)) == 0) stf(a.rq_scales + gg, s8);
        }
      } else if (BASE == kINT4) {
        uint32_t q[2];
        float z;
        const float s4 = PMAX >= 8 ? requant_i4(acc, lpg, q, z, acc)
                                   : quant_i4<true, false, SettleHere, (PMAX <= 2)>(acc, lpg, q, z, acc);
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
        uint32_t rw[8];
        if (RG) {
#pragma unroll
          for (int k = 0; k < 8; ++k) rw[k] = rv.w[k];
        } else {
          const uint4 r0 = rrow[2 * cs], r1 = rrow[2 * cs + 1];
          rw[0] = r0.x, rw[1] = r0.y, rw[2] = r0.z, rw[3] = r0.w;
          rw[4] = r1.x, rw[5] = r1.y, rw[6] = r1.z, rw[7] = r1.w;
        }
        V8 hv;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          hv.w[k] = pack_bf2(add_bf_lo(rw[k], acc[2 * k]), add_bf_hi(rw[k], acc[2 * k + 1]));
        if (HB) {
          uint4* hp = reinterpret_cast<uint4*>(hbuf) + 2 * c;
          hp[0] = make_uint4(hv.w[0], hv.w[1], hv.w[2], hv.w[3]);
          hp[1] = make_uint4(hv.w[4], hv.w[5], hv.w[6], hv.w[7]);
        }
        st256(static_cast<uint16_t*>(a.res_out) + gc * 16, hv);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          ss2.x = fma_bf_lo(hv.w[k], hv.w[k], ss2.x);
          ss2.y = fma_bf_hi(hv.w[k], hv.w[k], ss2.y);
        }
      }
      if (SUB > 1 && j < SUB - 1) {
        // every thread is past sub-stage j: refill it with the next row's segment
        __syncthreads();
        if (tid == 0 && ok) {
          const int64_t nrow = row + NSTAGE * rstride;
          if (nrow < a.rows) {
            fence_proxy_async_smem();
            issue_row<FMT, RG>(a, g, stage0 + (s * SUB + j) * g.stage_bytes, &bar[s * SUB + j], nrow, j);
            note_issue(s * SUB + j, i + NSTAGE);
          }
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
    float tot = 0.0f;
    for (int w = 0; w < nw; ++w) tot += red[i & 1][w];
    if (CL > 1) {
      // every CTA's partial sum and vote into every CTA's slots, one cluster
      // barrier, then the same rank-ordered sum in every CTA
      if (tid == 0)
        for (int r = 0; r < CL; ++r) {
          st_peer_f32(peer_smem(&cl_tot[i & 1][rank], r), tot);
          st_peer_u32(peer_smem(&cl_ok[i & 1][rank], r), all_ok ? 1u : 0u);
        }
      cluster_barrier();
      tot = 0.0f;
      for (int r = 0; r < CL; ++r) {
        tot += cl_tot[i & 1][r];
        all_ok = all_ok && cl_ok[i & 1][r] != 0u;
      }
    }
    if (!all_ok) break;
    const float inv = inv_rms(tot, inv_h, a.eps);

    // every thread is past its reads of stage s (its last sub-stage): refill
    // it NSTAGE rows ahead
    if (tid == 0) {
      const int64_t nrow = row + NSTAGE * rstride;
      if (nrow < a.rows) {
        fence_proxy_async_smem();
        issue_row<FMT, RG>(a, g, stage0 + (s * SUB + SUB - 1) * g.stage_bytes, &bar[s * SUB + SUB - 1], nrow,
                       SUB > 1 ? SUB - 1 : rank);
        note_issue(s * SUB + SUB - 1, i + NSTAGE);
      }
    }


    // ---- pass 2: y = bf16(fl(h * gamma) * inv); h * gamma is exact in binary32
    auto out_chunk = [&](int c, const uint32_t gw[8]) {
      uint32_t hw[8];
      if (HB) {
        const uint4* hp = reinterpret_cast<const uint4*>(hbuf) + 2 * c;
        const uint4 h0 = hp[0], h1 = hp[1];
        hw[0] = h0.x, hw[1] = h0.y, hw[2] = h0.z, hw[3] = h0.w;
        hw[4] = h1.x, hw[5] = h1.y, hw[6] = h1.z, hw[7] = h1.w;
      } else {  // this thread's own store of the chunk, read back through L2
        const V8 hv = ld256_coherent(static_cast<const uint16_t*>(a.res_out) + (row * cpr + c0 + c) * 16);
#pragma unroll
        for (int k = 0; k < 8; ++k) hw[k] = hv.w[k];
      }
      V8 yv;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 y = pmul(make_float2(fma_bf_lo(hw[k], gw[k], -0.0f), fma_bf_hi(hw[k], gw[k], -0.0f)),
                              dup2(inv));
        yv.w[k] = pack_bf2(y.x, y.y);
      }
      st256(static_cast<uint16_t*>(a.y) + (row * cpr + c0 + c) * 16, yv);
    };
#pragma unroll
    for (int j = 0; j < GRC; ++j)
      if (tid + j * nthr < cps) out_chunk(tid + j * nthr, greg[j]);
    for (int c = tid + GRC * nthr; c < cps; c += nthr) {
      const V8 gv = ld256_keep(static_cast<const uint16_t*>(a.gamma) + (c0 + c) * 16);
      out_chunk(c, gv.w);
    }
  }
  if (!all_ok && tid == 0) {
    // a staged copy did not land within the bound: report it and give each
    // copy still in flight one bounded wait, with its own phase parity,
    // before the CTA exits
    if (a.status) atomicExch(a.status, 2 /* FC_ERR_CUDA */);
    for (int x = 0; x < NSTAGE * SUB; ++x)
      if ((used >> x) & 1u) mbar_wait_bounded(&bar[x], (ppar >> x) & 1u);
  }
}

// Stage geometry for rows cut into cl segments (cl = 1: whole rows); 0 when a
// segment's pieces are not whole groups or not multiples of 16 bytes.
int geometry(int fmt, const FusedArgs& a, TmaGeom& g, int cl = 1) {
  const int H = a.H, P = a.P, cpr = H >> 4;
  if (cl < 1 || cpr % cl) return 0;
  g.cps = cpr / cl;
  const int hs = 16 * g.cps;  // elements in a segment
  if (fmt == kBF16) {
    g.row_cb = 2 * H, g.row_sb = 0;
    g.cb = 2 * hs, g.sb = 0, g.zb = 0;
  } else if (fmt == kINT8T || fmt == kINT4T) {
    const int G = fmt == kINT8T ? 128 : 32, nbg = fmt == kINT8T ? kBlocksPerGroupI8 : kBlocksPerGroupI4;
    if (hs % G) return 0;
    g.row_cb = (H / G) * nbg * 16, g.row_sb = 0;
    g.cb = (hs / G) * nbg * 16, g.sb = 0, g.zb = 0;
  } else {
    if (hs % a.G) return 0;
    g.row_cb = fmt == kINT8 ? H : H / 2;
    g.row_sb = (H / a.G) * 4;
    g.cb = fmt == kINT8 ? hs : hs / 2;
    g.sb = (hs / a.G) * 4;
    g.zb = fmt == kINT4 ? g.sb : 0;
  }
  if (g.cb % 16 || g.sb % 16 || g.zb % 16) return 0;
  g.stage_bytes = P * (g.cb + g.sb + g.zb) + 2 * hs;
  g.gamma_off = 0;
  g.stage_off = (2 * hs + 127) & ~127;
  return 1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


}  // namespace

}  // namespace fc
