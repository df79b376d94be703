// quant.cu -- streaming kernels: group quantize / requantize, fixed-order
// dequant-sum (reduce-scatter stage), tagged-block packing.
//
// Work unit: a "chunk" of 16 consecutive elements handled by one lane; a
// group of G elements spans G/16 adjacent lanes, so every per-group
// reduction is a few xor-shuffles.  A warp covers 32 consecutive chunks
// (512 elements, 1 KB of bf16), so every load and store instruction of a
// warp touches one contiguous span.  Grids are persistent: a multiple of the
// SM count, each warp striding over warp tiles, with two tiles in flight per
// iteration.
#include <atomic>
#include <mutex>

#include "device.cuh"
#include "internal.h"

namespace fc {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 2;

// ------------------------------------------------------- quantize kernel --
template <int FMT, bool IN_F32, int DEQ>
__global__ void __launch_bounds__(kThreads) k_quantize(QuantJob job, int64_t chunks,
                                                       int lpg_shift) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int lpg = 1 << lpg_shift;
  const int64_t tiles = (chunks + 31) >> 5;
  const int64_t gwarp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;

  const int64_t total = tiles * job.P;
  for (int64_t t0 = gwarp; t0 < total; t0 += nwarps * kUnroll) {
    float v[kUnroll][16];
    uint32_t bw[kUnroll][8];  // the bf16 inputs, packed
    int64_t cc[kUnroll];
    int pp[kUnroll];
    bool act[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      // tile t of the flattened (slab, tile) space; slab found by subtraction (P <= 8)
      int64_t t = t0 + u * nwarps;
      int p = 0;
      while (p < job.P - 1 && t >= tiles) t -= tiles, ++p;
      const int64_t c = t * 32 + lane;
      cc[u] = c;
      pp[u] = p;
      act[u] = t0 + u * nwarps < total && c < chunks;
      if (act[u]) {
        if (IN_F32) {
          const float* x = static_cast<const float*>(job.x[p]) + c * 16;
          V8 a = ld256_stream(x), b = ld256_stream(x + 8);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v[u][i] = __uint_as_float(a.w[i]);
            v[u][8 + i] = __uint_as_float(b.w[i]);
          }
        } else {
          const V8 x = ld256_stream(static_cast<const uint16_t*>(job.x[p]) + c * 16);
#pragma unroll
          for (int i = 0; i < 8; ++i) bw[u][i] = x.w[i];
          unpack16(x, v[u]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[u][i] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) bw[u][i] = 0u;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = cc[u];
      const int p = pp[u];
      float d[16];
      if (FMT == kINT8) {
        uint32_t q[4];
        const float s = quant_i8<DEQ != kDeqNone, !IN_F32>(v[u], lpg, q, d, bw[u]);
        if (act[u] && job.codes[p]) {
          st128(static_cast<int8_t*>(job.codes[p]) + c * 16, make_uint4(q[0], q[1], q[2], q[3]));
          if ((lane & (lpg - 1)) == 0) stf(job.scales[p] + (c >> lpg_shift), s);
        }
      } else {
        uint32_t q[2];
        float z;
        const float s = quant_i4<DEQ != kDeqNone, !IN_F32>(v[u], lpg, q, z, d, bw[u]);
        if (act[u] && job.codes[p]) {
          st64(static_cast<uint8_t*>(job.codes[p]) + c * 8, make_uint2(q[0], q[1]));
          if ((lane & (lpg - 1)) == 0) {
            stf(job.scales[p] + (c >> lpg_shift), s);
            stf(job.zeros[p] + (c >> lpg_shift), z);
          }
        }
      }
      if (DEQ != kDeqNone && act[u]) {
        if (DEQ == kDeqBF16) {
          V8 o;
#pragma unroll
          for (int i = 0; i < 8; ++i) o.w[i] = pack_bf2(d[2 * i], d[2 * i + 1]);
          st256(static_cast<uint16_t*>(job.deq) + c * 16, o);
        } else {
          V8 o0, o1;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o0.w[i] = __float_as_uint(d[i]);
            o1.w[i] = __float_as_uint(d[8 + i]);
          }
          float* out = static_cast<float*>(job.deq) + c * 16;
          st256(out, o0);
          st256(out + 8, o1);
        }
      }
    }
  }
}

// --------------------------------------------- TMA-streamed quantize kernel --
// Sender-side quantization of bf16 slabs with the input streamed by the TMA
// engine.  Every warp is autonomous: it owns a private ring of kWStages
// shared-memory tiles of kWTile elements, its lane 0 issues the bulk copies
// (cp.async.bulk, completing on the tile's mbarrier) kWStages-1 tiles ahead,
// and its 32 lanes quantize the current tile out of shared memory and store
// codes and scales directly.  Warps never wait for each other: no CTA-wide
// barrier is used.  Tiles cover the flattened (slab, tile) space.
// TILE: elements per warp tile.  Measured on GB300: for large calls (prefill,
// 4 x 8192 x 8192) 2048-element tiles in a two-deep ring (three CTAs per SM)
// beat 1024-element tiles four deep by 8% -- half the per-tile waits and
// cursor steps; calls with fewer 2048-element tiles than resident warps
// (decode) keep the smaller tiles, which spread over more warps.  Both use
// 8 KB of ring per warp.
template <int TILE, int STAGES>
struct WRing {
  static constexpr int kStages = STAGES;
  static constexpr int kBytes = kStages * TILE * 2;
};
template <int TILE>
constexpr int default_stages() { return TILE == 1024 ? 4 : 2; }
static_assert(WRing<1024, 4>::kBytes == WRing<2048, 2>::kBytes, "one shared-memory size for both tilings");
static_assert(WRing<1536, 2>::kBytes <= WRing<2048, 2>::kBytes, "1536-element tiles fit the same budget");
constexpr int kQWarps = kThreads / 32;

// TAGGED: the codes and scales go out as self-synchronizing blocks carrying
// job.epoch: every group's payload (INT8 g128: 128 code bytes + scale = 11
// pieces of 12 bytes; INT4 g32: 16 code bytes + scale + zero = 2 pieces) in
// words 0..2 of a 16-byte block, the epoch in word 3.
// LPG: lanes per group when known at compile time (the two standard group
// sizes), 0 to take it from lpg_shift.
template <int FMT, bool TAGGED = false, int LPG = 0, int TILE = 2048, int STAGES = default_stages<TILE>()>
__global__ void __launch_bounds__(kThreads, STAGES == 1 ? 4 : 3)
    k_quantize_tma(QuantJob job, int lpg_shift, int64_t tiles_per_slab) {
  constexpr int kWTile = TILE, kWStages = STAGES;
  constexpr int kRingBytes = WRing<TILE, STAGES>::kBytes;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bars[kQWarps][STAGES];
  // INT8 tagged: a warp assembles its 4 groups' payloads (33 words each) here
  __shared__ uint32_t qstage[TAGGED && FMT == kINT8 ? kQWarps : 1][4][33];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int lpg = LPG ? LPG : 1 << lpg_shift;
  const int64_t total = tiles_per_slab * job.P;
  const int64_t w0 = static_cast<int64_t>(blockIdx.x) * kQWarps + wid;
  const int64_t wstride = static_cast<int64_t>(gridDim.x) * kQWarps;
  if (w0 >= total) return;  // whole warp
  uint8_t* ring = smem + wid * kRingBytes;
  uint64_t* bar = bars[wid];

  // A cursor over the flattened (slab, tile) space that only moves forward by
  // wstride tiles: (slab p, tile tt of that slab).
  struct Cursor {
    int p;
    int64_t tt;
  };
  auto advance = [&](Cursor cur, int64_t by) {
    cur.tt += by;
    while (cur.tt >= tiles_per_slab && cur.p < job.P - 1) cur.tt -= tiles_per_slab, ++cur.p;
    return cur;
  };
  auto issue = [&](Cursor cur, int st) {
    const int64_t e0 = cur.tt * kWTile;
    const int64_t rem = job.n - e0;
    const int ne = static_cast<int>(rem < kWTile ? rem : kWTile);
    mbar_expect_tx(&bar[st], static_cast<uint32_t>(ne * 2));
    bulk_load(ring + st * (kWTile * 2), static_cast<const uint16_t*>(job.x[cur.p]) + e0, ne * 2,
              &bar[st]);
  };

  const Cursor first = advance(Cursor{0, 0}, w0);
  Cursor ahead = first;  // lane 0's issue cursor, kWStages - 1 tiles ahead
  if (lane == 0) {
    for (int s = 0; s < kWStages; ++s) mbar_init(&bar[s], 1);
    mbar_init_fence();
    // the first tiles into L2 while the previous kernel finishes
    Cursor pf = first;
    for (int s = 0; s < kWStages - 1 && w0 + s * wstride < total; ++s, pf = advance(pf, wstride)) {
      const int64_t e0 = pf.tt * kWTile, rem = job.n - e0;
      prefetch_l2(static_cast<const uint16_t*>(job.x[pf.p]) + e0,
                  static_cast<uint32_t>((rem < kWTile ? rem : kWTile) * 2));
    }
  }
  pdl_begin();
  if (lane == 0) {
    for (int s = 0; s < kWStages - 1; ++s) {
      if (w0 + s * wstride < total) issue(ahead, s);
      ahead = advance(ahead, wstride);
    }
  }
  __syncwarp();

  int k = 0;
  bool ok = true;
  Cursor cur = first;
  for (int64_t t = w0; t < total; t += wstride, ++k, cur = advance(cur, wstride)) {
    const int st = k % kWStages;
    if (lane == 0) {
      // refill the stage the warp finished with last iteration (after __syncwarp)
      if (t + (kWStages - 1) * wstride < total) {
        fence_proxy_async_smem();
        issue(ahead, (k + kWStages - 1) % kWStages);
      }
      ahead = advance(ahead, wstride);
    }
    if (!__all_sync(kFull, mbar_wait_bounded(&bar[st], (k / kWStages) & 1))) {
      ok = false;  // a tile never landed (about a second): stop, outputs incomplete
      if (lane == 0) {
        if (job.status) atomicExch(job.status, 2 /* FC_ERR_CUDA */);
        // the copies still in flight: this iteration's and the ones issued
        // ahead of it, each waited for once with its own phase parity
        for (int j = 0; j < kWStages; ++j)
          if (t + j * wstride < total)
            mbar_wait_bounded(&bar[(k + j) % kWStages], ((k + j) / kWStages) & 1);
      }
      break;
    }
    const int p = cur.p;
    const int64_t e0 = cur.tt * kWTile;
    const int64_t rem = job.n - e0;
    const int ne = static_cast<int>(rem < kWTile ? rem : kWTile);
    const uint4* tile = reinterpret_cast<const uint4*>(ring + st * (kWTile * 2));
    const int nch = ne >> 4;
    // each chunk's flag mask, scale and minimum, settled once for the whole
    // tile below
    constexpr int kNJ = kWTile / 16 / 32;
    uint32_t mk[kNJ];
    float sj[kNJ], zj[kNJ];
#pragma unroll
    for (int j = 0; j < kNJ; ++j) mk[j] = 0u, sj[j] = 0.0f, zj[j] = 0.0f;
#pragma unroll
    for (int j = 0; j < kNJ; ++j) {
      const int cl = j * 32 + lane;
      const bool act = cl < nch;
      uint32_t bw[8];
      if (act) {
        const uint4 a = tile[2 * cl], b = tile[2 * cl + 1];
        bw[0] = a.x, bw[1] = a.y, bw[2] = a.z, bw[3] = a.w;
        bw[4] = b.x, bw[5] = b.y, bw[6] = b.z, bw[7] = b.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) bw[i] = 0u;
      }
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[2 * i] = bf_lo(bw[i]), v[2 * i + 1] = bf_hi(bw[i]);
      const int64_t c = (e0 >> 4) + cl;  // global chunk of slab p
      float d[16];
      if (FMT == kINT8) {
        uint32_t q[4];
        float s;
        s = quant_i8<false, true>(v, lpg, q, d, bw, DeferSettle{&mk[j]});
        sj[j] = s;
        if (TAGGED) {
          // lpg == 8: lane = (group in warp) * 8 + k; stage the payload, then
          // one lane per block writes it (11 blocks per group, 44 per warp)
          uint32_t* pl = qstage[wid][lane >> 3];
#pragma unroll
          for (int i = 0; i < 4; ++i) pl[4 * (lane & 7) + i] = q[i];
          if ((lane & 7) == 0) pl[32] = __float_as_uint(s);
          __syncwarp();
          const int64_t g0 = ((e0 >> 4) + j * 32) >> 3;  // first group of this warp chunk
          const int ngr = min(4, (nch - j * 32 + 7) >> 3);
          uint4* out = static_cast<uint4*>(job.codes[p]);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int bi = r * 32 + lane;
            const int gr = bi / kBlocksPerGroupI8, b = bi - gr * kBlocksPerGroupI8;
            if (bi < 44 && gr < ngr) {
              const uint32_t* w = qstage[wid][gr] + 3 * b;
              st128(out + (g0 + gr) * kBlocksPerGroupI8 + b, make_uint4(w[0], w[1], w[2], job.epoch));
            }
          }
          __syncwarp();
        } else if (act) {
          st128(static_cast<int8_t*>(job.codes[p]) + c * 16, make_uint4(q[0], q[1], q[2], q[3]));
          if ((lane & (lpg - 1)) == 0) stf(job.scales[p] + (c >> lpg_shift), s);
        }
      } else {
        uint32_t q[2];
        float z, s;
        s = quant_i4<false, true>(v, lpg, q, z, d, bw, DeferSettle{&mk[j]});
        sj[j] = s, zj[j] = z;
        if (TAGGED) {
          // lpg == 2: the even lane writes block 0 {its two code words, the odd
          // lane's first}, the odd lane block 1 {its second, scale, zero}
          const uint32_t other = __shfl_xor_sync(kFull, q[0], 1);
          if (act) {
            uint4* out = static_cast<uint4*>(job.codes[p]) + (c >> 1) * kBlocksPerGroupI4;
            if ((lane & 1) == 0)
              st128(out, make_uint4(q[0], q[1], other, job.epoch));
            else
              st128(out + 1, make_uint4(q[1], __float_as_uint(s), __float_as_uint(z), job.epoch));
          }
        } else if (act) {
          st64(static_cast<uint8_t*>(job.codes[p]) + c * 8, make_uint2(q[0], q[1]));
          if ((lane & (lpg - 1)) == 0) {
            stf(job.scales[p] + (c >> lpg_shift), s);
            stf(job.zeros[p] + (c >> lpg_shift), z);
          }
        }
      }
    }
    {
      // The exact pass for the whole tile: each lane settles its flagged
      // elements of all its chunks in turn (re-read from the staged tile,
      // which lane 0 refills only after this), and patches the stored codes.
      // Once per tile instead of once per chunk, the warp loops about half as
      // often (flags are sparse: most lanes hold at most one per tile).
      // Tagged INT4 blocks hold an odd lane's first code word in its even
      // neighbour's block; the warp barrier orders that store before the
      // patch.
      if (TAGGED) __syncwarp();
      const uint16_t* t16 = reinterpret_cast<const uint16_t*>(tile);
      auto pending = [&]() {
        uint32_t m = 0u;
#pragma unroll
        for (int j = 0; j < kNJ; ++j) m |= mk[j];
        return m;
      };
      while (__any_sync(kFull, pending() != 0u)) {
        if (pending() != 0u) {
          int js = 0;
#pragma unroll
          for (int j = kNJ - 1; j >= 0; --j)
            if (mk[j]) js = j;
          uint32_t m = 0u;
          float s = 0.0f, z = 0.0f;
#pragma unroll
          for (int j = 0; j < kNJ; ++j)
            if (j == js) m = mk[j], s = sj[j], z = zj[j], mk[j] &= mk[j] - 1u;
          const int pos = __ffs(m) - 1;
          const int i = 4 * (pos & 7) + (pos >> 3);  // mask bit 8b + w is element 4w + b
          const int cl = js * 32 + lane;
          const uint32_t xb = t16[16 * cl + i];
          const int64_t c = (e0 >> 4) + cl;
          uint8_t* out = static_cast<uint8_t*>(job.codes[p]);
          if (FMT == kINT8) {
            const int code = __float2int_rn(code_by_division<true>(__uint_as_float(xb << 16), s));
            // plain: 16 code bytes per chunk; tagged: payload word 4k + i/4 of
            // the group (k = chunk within the group), three words per block
            const int pw = 4 * (cl & 7) + (i >> 2);
            uint8_t* bp = TAGGED ? out + ((c >> 3) * kBlocksPerGroupI8 + pw / 3) * 16 + (pw % 3) * 4 + (i & 3)
                                 : out + c * 16 + i;
            st_u8(bp, static_cast<uint32_t>(code) & 0xFFu);
          } else {
            const int code = __float2int_rn(code_by_division<false>(add_bf_lo(xb, -z), s));
            // plain: two code words per chunk; tagged: block 0 = {even lane's
            // words, odd lane's first}, block 1 = {odd lane's second, ...}
            const int k = i >> 3;
            const int wi = !TAGGED ? 0 : (cl & 1) == 0 ? k : (k == 0 ? 2 : 4);
            uint32_t* wp = TAGGED ? reinterpret_cast<uint32_t*>(out + (c >> 1) * kBlocksPerGroupI4 * 16) + wi
                                  : reinterpret_cast<uint32_t*>(out + c * 8) + k;
            const int sh = 4 * (i & 7);
            const uint32_t old = TAGGED ? ld_u32_l2(wp) : ld_u32(wp);
            st_u32(wp, (old & ~(0xFu << sh)) | (static_cast<uint32_t>(code) << sh));
          }
        }
      }
    }
    __syncwarp();  // every lane is done with stage st before lane 0 refills it
  }
  (void)ok;
}

// --------------------------------------------------------- reduce kernel --
// out[i] = ((0 + deq_0(i)) + deq_1(i)) + ... + deq_{P-1}(i)   (fp32, slab order)
template <int FMT>
__global__ void __launch_bounds__(kThreads) k_reduce(Slabs s, int P, int lpg_shift, int64_t c0,
                                                     int64_t c1, float* out) {
  pdl_begin();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t c = c0 + static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; c < c1;
       c += stride) {
    const int64_t g = c >> lpg_shift;
    uint32_t q[kMaxP][4];
    float sc[kMaxP], zp[kMaxP];
#pragma unroll
    for (int p = 0; p < kMaxP; ++p) {
      if (p < P) {
        if (FMT == kINT8) {
          uint4 w = ld128_stream(static_cast<const int8_t*>(s.codes[p]) + c * 16);
          q[p][0] = w.x, q[p][1] = w.y, q[p][2] = w.z, q[p][3] = w.w;
        } else {
          uint2 w = ld64_stream(static_cast<const uint8_t*>(s.codes[p]) + c * 8);
          q[p][0] = w.x, q[p][1] = w.y;
          zp[p] = ldf_stream(s.zeros[p] + g);
        }
        sc[p] = ldf_stream(s.scales[p] + g);
      }
    }
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int p = 0; p < kMaxP; ++p) {
      if (p < P) {
        if (FMT == kINT8)
          dequant_i8_acc(q[p], sc[p], acc);
        else
          dequant_i4_acc(q[p], sc[p], zp[p], acc);
      }
    }
    V8 o0, o1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o0.w[i] = __float_as_uint(acc[i]);
      o1.w[i] = __float_as_uint(acc[8 + i]);
    }
    st256(out + c * 16, o0);
    st256(out + c * 16 + 8, o1);
  }
}

// ---------------------------------------------------- tagged-block packing --
// One lane per 16-byte block, one warp per 32 consecutive blocks of a row:
// the warp reads 384 contiguous input bytes (three 4-byte loads per lane)
// and writes 512 contiguous output bytes (one 16-byte store per lane), two
// block groups in flight per iteration.  blockIdx.y selects the slab, so all
// P producers pack in one launch.
constexpr int kPackUnroll = 2;

struct PackJob {
  const uint16_t* x[8];
  uint4* blocks[8];
};

__device__ __forceinline__ uint32_t ld32_stream(const void* p) {
  uint32_t r;
  asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__global__ void __launch_bounds__(kThreads) k_pack_tagged(PackJob job, int64_t rows, int H, int nb,
                                                          uint32_t epoch) {
  pdl_begin();
  const uint16_t* __restrict__ x = job.x[blockIdx.y];
  uint4* blocks = job.blocks[blockIdx.y];
  const int lane = threadIdx.x & 31;
  const uint32_t gpr = static_cast<uint32_t>((nb + 31) >> 5);  // block groups per row
  const int64_t items = rows * gpr;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  // (row, group) cursors, advanced by nw items without dividing again
  const int64_t step_rows = nw / gpr;
  const uint32_t step_g = static_cast<uint32_t>(nw - step_rows * gpr);
  auto advance = [&](int64_t& row, uint32_t& g) {
    row += step_rows;
    g += step_g;
    if (g >= gpr) g -= gpr, ++row;
  };
  int64_t row0 = w0 / gpr;
  uint32_t g0 = static_cast<uint32_t>(w0 - row0 * gpr);
  for (int64_t it0 = w0; it0 < items; it0 += nw * kPackUnroll) {
    uint32_t wv[kPackUnroll][3];
    int64_t blk[kPackUnroll];
    bool act[kPackUnroll];
    int64_t row = row0;
    uint32_t g = g0;
#pragma unroll
    for (int u = 0; u < kPackUnroll; ++u) {
      if (u) advance(row, g);
      const int64_t it = it0 + u * nw;
      const int j = static_cast<int>(g) * 32 + lane;
      act[u] = it < items && j < nb;
      blk[u] = row * nb + j;
      if (act[u]) {
        const uint16_t* xr = x + row * H;
        const int e0 = 6 * j;
        if (e0 + 6 <= H) {
#pragma unroll
          for (int k = 0; k < 3; ++k) wv[u][k] = ld32_stream(xr + e0 + 2 * k);
        } else {
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            const int e = e0 + 2 * k;
            const uint32_t lo = e < H ? ld16(xr + e) : 0u;
            const uint32_t hi = e + 1 < H ? ld16(xr + e + 1) : 0u;
            wv[u][k] = lo | (hi << 16);
          }
        }
      }
    }
    advance(row, g);
    row0 = row, g0 = g;
#pragma unroll
    for (int u = 0; u < kPackUnroll; ++u)
      if (act[u]) st128(blocks + blk[u], make_uint4(wv[u][0], wv[u][1], wv[u][2], epoch));
  }
}

// log2 of the lanes per group (G / 16; G is a power of two in [16, 512])
int log2_lanes(int G) {
  int sh = 0;
  while ((16 << sh) < G) ++sh;
  return sh;
}

// Persistent grid: enough blocks for the work, at most 8 x 256-thread
// blocks (2048 threads, the per-SM maximum) per SM.
int grid_for(int64_t work_items, int per_block) {
  const int64_t need = (work_items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  return static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
}

template <int FMT, bool IN_F32, int DEQ>
cudaError_t launch_quantize_t(const QuantJob& job, cudaStream_t st) {
  const int64_t chunks = job.n / 16;
  const int64_t tiles = (chunks + 31) / 32;
  const int64_t warps_needed = (tiles * job.P + kUnroll - 1) / kUnroll;
  const int grid = grid_for(warps_needed * 32, kThreads);
  return launch_pdl(k_quantize<FMT, IN_F32, DEQ>, dim3(grid), dim3(kThreads), 0, st, job, chunks,
                    log2_lanes(job.G));
}

}  // namespace

// SM count of the current device, queried once per device (thread-safe: a
// racing first query stores the same value).
int num_sms() {
  static std::atomic<int> sms[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  int v = sms[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (v < 1) v = 1;
    sms[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

namespace {
constexpr int kOccMemoMax = 512;
OccKey g_occ_keys[kOccMemoMax];
int g_occ_vals[kOccMemoMax];
int g_occ_n = 0;
std::mutex g_occ_mu;
bool same_key(const OccKey& a, const OccKey& b) {
  return a.fn == b.fn && a.dev == b.dev && a.threads == b.threads && a.smem == b.smem &&
         a.cluster == b.cluster;
}
}  // namespace

bool occ_memo_find(const OccKey& k, int* value) {
  std::lock_guard<std::mutex> lock(g_occ_mu);
  for (int i = 0; i < g_occ_n; ++i)
    if (same_key(g_occ_keys[i], k)) {
      *value = g_occ_vals[i];
      return true;
    }
  return false;
}

cudaError_t raise_smem_limit(const void* fn, int smem) {
  static std::mutex mu;
  static const void* fns[kOccMemoMax];
  static int devs[kOccMemoMax], lims[kOccMemoMax];
  static int n = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  int i = 0;
  while (i < n && !(fns[i] == fn && devs[i] == dev)) ++i;
  if (i < n && lims[i] >= smem) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (i == n && n < kOccMemoMax) fns[n] = fn, devs[n] = dev, ++n;
  if (i < n) lims[i] = smem;
  return cudaSuccess;
}

void occ_memo_store(const OccKey& k, int value) {
  std::lock_guard<std::mutex> lock(g_occ_mu);
  for (int i = 0; i < g_occ_n; ++i)
    if (same_key(g_occ_keys[i], k)) return;
  if (g_occ_n < kOccMemoMax) {  // a full memo only means later misses are re-queried
    g_occ_keys[g_occ_n] = k;
    g_occ_vals[g_occ_n] = value;
    ++g_occ_n;
  }
}

template <int FMT, bool TAGGED, int LPG, int TILE, int STAGES = default_stages<TILE>()>
cudaError_t launch_quantize_tma_t(const QuantJob& job, cudaStream_t st) {
  constexpr int kWTile = TILE;
  const int smem = kQWarps * WRing<TILE, STAGES>::kBytes;
  auto kern = k_quantize_tma<FMT, TAGGED, LPG, TILE, STAGES>;
  const int occ = occupancy_memo(reinterpret_cast<const void*>(kern), kThreads, smem, 1, [&] {
    int o = 0;
    if (raise_smem_limit(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, kThreads, smem) != cudaSuccess)
      return 0;
    return o;
  });
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int64_t tps = (job.n + kWTile - 1) / kWTile;
  int64_t grid = static_cast<int64_t>(num_sms()) * occ;
  const int64_t need = (tps * job.P + kQWarps - 1) / kQWarps;
  if (grid > need) grid = need;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), smem, st, job,
                    log2_lanes(job.G), tps);
}

// INT8 g128 (8 lanes per group) and INT4 g32 (2 lanes) are specialised
// Tile size: the elements the busiest warp streams, ceil(tiles / resident
// warps) * tile, bound a call too small to fill the GPU several times over.
// 1536-element tiles (three chunks a lane, two deep) are taken where they
// make that strictly smaller than both other sizes: a decode step's eight
// 64 x 8192 slabs are 4096 tiles of 1024 for 3648 resident warps (2048
// elements on the busiest), or 2731 of 1536 (1536).
template <int FMT, bool TAGGED, int LPG>
cudaError_t launch_quantize_tma_tile(const QuantJob& job, cudaStream_t st) {
  // resident warps: three CTAs of kQWarps per SM
  const int64_t warps = static_cast<int64_t>(num_sms()) * 3 * kQWarps;
  auto busiest = [&](int64_t tile) { return ((job.n + tile - 1) / tile * job.P + warps - 1) / warps * tile; };
  const int64_t b1 = busiest(1024), b15 = busiest(1536), b2 = busiest(2048);
  if (b15 < b1 && b15 < b2) return launch_quantize_tma_t<FMT, TAGGED, LPG, 1536>(job, st);
  const int64_t big_tiles = (job.n + 2047) / 2048 * job.P;
  if (big_tiles < warps)
    return launch_quantize_tma_t<FMT, TAGGED, LPG, 1024>(job, st);
  return launch_quantize_tma_t<FMT, TAGGED, LPG, 2048>(job, st);
}

template <int FMT, bool TAGGED = false>
cudaError_t launch_quantize_tma(const QuantJob& job, cudaStream_t st) {
  constexpr int kStdLanes = FMT == kINT8 ? 8 : 2;
  if (TAGGED || job.G == 16 * kStdLanes) return launch_quantize_tma_tile<FMT, TAGGED, kStdLanes>(job, st);
  return launch_quantize_tma_tile<FMT, false, 0>(job, st);
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cudaError_t launch_quantize(int fmt, bool in_f32, int deq, const QuantJob& job, cudaStream_t st) {
  if (job.n == 0) return cudaSuccess;
  if (!in_f32) {
    // bf16 slabs: TMA-streamed input (16-byte aligned slabs, which the ABI guarantees)
    bool ok = true;
    for (int p = 0; p < job.P; ++p) ok = ok && aligned_to(job.x[p], 16) && job.codes[p];
    if (ok) return fmt == kINT8 ? launch_quantize_tma<kINT8>(job, st) : launch_quantize_tma<kINT4>(job, st);
  }
  if (fmt == kINT8) {
    if (!in_f32) return launch_quantize_t<kINT8, false, kDeqNone>(job, st);
    if (deq == kDeqBF16) return launch_quantize_t<kINT8, true, kDeqBF16>(job, st);
    if (deq == kDeqF32) return launch_quantize_t<kINT8, true, kDeqF32>(job, st);
    return launch_quantize_t<kINT8, true, kDeqNone>(job, st);
  }
  if (!in_f32) return launch_quantize_t<kINT4, false, kDeqNone>(job, st);
  if (deq == kDeqBF16) return launch_quantize_t<kINT4, true, kDeqBF16>(job, st);
  if (deq == kDeqF32) return launch_quantize_t<kINT4, true, kDeqF32>(job, st);
  return launch_quantize_t<kINT4, true, kDeqNone>(job, st);
}

cudaError_t launch_quantize_tagged(int fmt, const QuantJob& job, cudaStream_t st) {
  if (job.n == 0) return cudaSuccess;
  return fmt == kINT8T ? launch_quantize_tma<kINT8, true>(job, st)
                       : launch_quantize_tma<kINT4, true>(job, st);
}

cudaError_t launch_reduce(int fmt, const Slabs& s, int P, int G, int64_t c0, int64_t c1,
                          float* out, cudaStream_t st) {
  if (c1 <= c0) return cudaSuccess;
  const int grid = grid_for(c1 - c0, kThreads);
  return launch_pdl(fmt == kINT8 ? k_reduce<kINT8> : k_reduce<kINT4>, dim3(grid), dim3(kThreads), 0, st,
                    s, P, log2_lanes(G), c0, c1, out);
}

cudaError_t launch_pack_tagged(const void* const* x, void* const* blocks, int P, int64_t rows,
                               int H, uint32_t epoch, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int nb = (H + 5) / 6;
  PackJob job{};
  for (int p = 0; p < P; ++p) {
    job.x[p] = static_cast<const uint16_t*>(x[p]);
    job.blocks[p] = static_cast<uint4*>(blocks[p]);
  }
  const int64_t lanes = rows * ((nb + 31) / 32) * 32;
  int grid = grid_for((lanes + kPackUnroll - 1) / kPackUnroll, kThreads);
  grid = (grid + P - 1) / P;  // the P slabs share the resident-CTA budget
  return launch_pdl(k_pack_tagged, dim3(grid, P), dim3(kThreads), 0, st, job, rows, H, nb, epoch);
}

// The two status words of a call, {FC_OK, no index}, written after the
// previous kernel in the stream has finished (it may write them too) and
// before the call's own kernel reads or writes them.  A one-thread kernel
// launched with programmatic dependent launch, like the kernels it precedes:
// the next kernel may be scheduled as soon as this one starts, so its
// prologue (barrier set-up, L2 prefetch of its first tiles) still overlaps
// the previous kernel's tail, and its griddepcontrol.wait returns only after
// this kernel, and therefore the one before it, has completed.  Two memset
// nodes in its place break that chain.
__global__ void k_reset_status(int32_t* s) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  s[0] = 0;           // FC_OK
  s[1] = 0x7F7F7F7F;  // no block index
}

cudaError_t launch_reset_status(int32_t* d_status, cudaStream_t st) {
  return launch_pdl(k_reset_status, dim3(1), dim3(1), 0, st, d_status);
}

}  // namespace fc
