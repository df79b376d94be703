// gather.cu -- the standalone quantized all-gather.
//
// flash-comm (abstract) names an all-gather collective beside the
// All-Reduce, and Flash Communication ("Core ideas") builds the All-Reduce's
// second step from one: every rank holds the quantized payload of one shard
// of the tensor (the contiguous groups it reduced), every rank receives all
// shards and dequantizes them.  On one GPU the P shards are P buffers in HBM
// and the call writes the whole dequantized tensor: a pure streaming kernel,
// each lane one 16-element chunk (one 16-byte INT8 / 8-byte INT4 load, or
// the chunk's words of the 16-byte tagged blocks, whose epochs are checked in
// the same loads), written as bf16 (round to nearest even) or fp32.
#include <climits>

#include "device.cuh"
#include "internal.h"

namespace fc {

namespace {

constexpr int kGatherThreads = 256;

template <int FMT, bool OUT_F32>
__global__ void __launch_bounds__(kGatherThreads) k_allgather(GatherJob j) {
  pdl_begin();
  constexpr bool TAGGED = FMT == kINT8T || FMT == kINT4T;
  constexpr int BASE = FMT == kINT8T ? kINT8 : FMT == kINT4T ? kINT4 : FMT;
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kGatherThreads;
  int64_t first_bad = LLONG_MAX;
  // warp-uniform trip count: every lane reaches the final shuffles
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kGatherThreads + (threadIdx.x & ~31);
       base < j.chunks; base += stride) {
    const int64_t c = base + lane;
    if (c >= j.chunks) continue;
    int p = 0;
    while (p < j.P - 1 && c >= j.first[p + 1]) ++p;  // the shard holding chunk c
    const int64_t lc = c - j.first[p];               // its chunk in that shard
    const int64_t lg = lc >> j.lpg_shift;            // its group in that shard
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = -0.0f;  // -0 + d == d for every d
    bool ok = true;
    if (!TAGGED) {
      if (BASE == kINT8) {
        const uint4 q = ld128_stream(static_cast<const int8_t*>(j.codes[p]) + lc * 16);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        dequant_i8_acc(w, ldf_stream(j.scales[p] + lg), acc);
      } else {
        const uint2 q = ld64_stream(static_cast<const uint8_t*>(j.codes[p]) + lc * 8);
        const uint32_t w[2] = {q.x, q.y};
        dequant_i4_acc(w, ldf_stream(j.scales[p] + lg), ldf_stream(j.zeros[p] + lg), acc);
      }
    } else if (BASE == kINT8) {
      // group lg, lane k = lc & 7: code bytes 16k.. are words o.. of blocks b0, b0 + 1
      const int k = static_cast<int>(lc & 7), b0 = (4 * k) / 3, o = 4 * k - 3 * b0;
      const uint4* gb = static_cast<const uint4*>(j.codes[p]) + lg * kBlocksPerGroupI8;
      const uint4 B0 = ld128_stream(gb + b0), B1 = ld128_stream(gb + b0 + 1);
      const uint4 BS = ld128_stream(gb + kBlocksPerGroupI8 - 1);
      if (B0.w == j.epoch && B1.w == j.epoch && BS.w == j.epoch) {
        const uint32_t W[6] = {B0.x, B0.y, B0.z, B1.x, B1.y, B1.z};
        const uint32_t w[4] = {o == 0 ? W[0] : o == 1 ? W[1] : W[2],
                               o == 0 ? W[1] : o == 1 ? W[2] : W[3],
                               o == 0 ? W[2] : o == 1 ? W[3] : W[4],
                               o == 0 ? W[3] : o == 1 ? W[4] : W[5]};
        dequant_i8_acc(w, __uint_as_float(BS.z), acc);
      } else {
        ok = false;
        const int64_t bad = j.blk0[p] + lg * kBlocksPerGroupI8 +
                            (B0.w != j.epoch ? b0 : B1.w != j.epoch ? b0 + 1 : kBlocksPerGroupI8 - 1);
        first_bad = bad < first_bad ? bad : first_bad;
      }
    } else {
      // group lg: block 0 = {codes 0-3, 4-7, 8-11}, block 1 = {codes 12-15, scale, zero}
      const int k = static_cast<int>(lc & 1);
      const uint4* gb = static_cast<const uint4*>(j.codes[p]) + lg * kBlocksPerGroupI4;
      const uint4 B0 = ld128_stream(gb), B1 = ld128_stream(gb + 1);
      if (B0.w == j.epoch && B1.w == j.epoch) {
        const uint32_t w[2] = {k ? B0.z : B0.x, k ? B1.x : B0.y};
        dequant_i4_acc(w, __uint_as_float(B1.y), __uint_as_float(B1.z), acc);
      } else {
        ok = false;
        const int64_t bad = j.blk0[p] + lg * kBlocksPerGroupI4 + (B0.w != j.epoch ? 0 : 1);
        first_bad = bad < first_bad ? bad : first_bad;
      }
    }
    if (!ok) continue;  // a chunk read from a stale block is not written
    if (OUT_F32) {
      V8 o0, o1;
#pragma unroll
      for (int i = 0; i < 8; ++i) o0.w[i] = __float_as_uint(acc[i]), o1.w[i] = __float_as_uint(acc[8 + i]);
      float* out = static_cast<float*>(j.out) + c * 16;
      st256(out, o0);
      st256(out + 8, o1);
    } else {
      V8 o;
#pragma unroll
      for (int i = 0; i < 8; ++i) o.w[i] = pack_bf2(acc[2 * i], acc[2 * i + 1]);
      st256(static_cast<uint16_t*>(j.out) + c * 16, o);
    }
  }
  if (TAGGED) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      const int64_t o2 = __shfl_xor_sync(kFull, first_bad, m);
      first_bad = o2 < first_bad ? o2 : first_bad;
    }
    if (lane == 0 && first_bad != LLONG_MAX && j.status) {
      atomicCAS(j.status, 0, 3 /* FC_ERR_STALE_BLOCK */);
      atomicMin(j.status + 1, first_bad < INT_MAX ? static_cast<int>(first_bad) : INT_MAX - 1);
    }
  }
}

template <int FMT>
cudaError_t launch_fmt(bool out_f32, const GatherJob& j, cudaStream_t st) {
  // persistent: 8 CTAs of 8 warps per SM of the current device at most, fewer
  // when the tensor is small
  const int64_t sms = num_sms();
  int64_t grid = (j.chunks + kGatherThreads - 1) / kGatherThreads;
  if (grid > 8 * sms) grid = 8 * sms;
  if (grid < 1) grid = 1;
  const dim3 gr(static_cast<unsigned>(grid));
  if (out_f32) return launch_pdl(k_allgather<FMT, true>, gr, dim3(kGatherThreads), 0, st, j);
  return launch_pdl(k_allgather<FMT, false>, gr, dim3(kGatherThreads), 0, st, j);
}

}  // namespace

cudaError_t launch_allgather(int fmt, bool out_f32, const GatherJob& j, cudaStream_t st) {
  if (j.chunks == 0) return cudaSuccess;
  switch (fmt) {
    case kINT8: return launch_fmt<kINT8>(out_f32, j, st);
    case kINT4: return launch_fmt<kINT4>(out_f32, j, st);
    case kINT8T: return launch_fmt<kINT8T>(out_f32, j, st);
    case kINT4T: return launch_fmt<kINT4T>(out_f32, j, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fc
