// internal.h -- launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fc {

enum Fmt : int {
  kBF16 = 0, kINT8 = 1, kINT4 = 2, kTAGGED = 3, kF32 = 4,
  kINT8T = 5,  // INT8 g128 groups in epoch-tagged 16-byte blocks (11 per group)
  kINT4T = 6   // INT4 g32 groups in epoch-tagged 16-byte blocks (2 per group)
};
// 16-byte blocks per quantization group of the tagged quantized formats.
constexpr int kBlocksPerGroupI8 = 11, kBlocksPerGroupI4 = 2;

// Dequantized output of a requantization: none, bf16 or fp32.
enum DeqOut : int { kDeqNone = 0, kDeqBF16 = 1, kDeqF32 = 2 };

// P slabs as device pointers (passed to kernels by value).
struct Slabs {
  const void* codes[8];
  const float* scales[8];
  const float* zeros[8];
};

// Group quantization of P tensors of n elements each (bf16 or fp32 input),
// optionally writing the dequantized values (single tensor only).
struct QuantJob {
  const void* x[8];
  void* codes[8];
  float* scales[8];
  float* zeros[8];
  void* deq;  // NULL, bf16 or fp32 [n] (P == 1 only)
  int32_t* status;  // NULL, or word 0 set to FC_ERR_CUDA if a staged copy never lands
  uint32_t epoch;  // tagged quantized output only
  int64_t n;  // elements per tensor (multiple of G)
  int P;
  int G;
};

struct FusedArgs {
  Slabs s;
  const void* res_in;
  void* res_out;
  const void* gamma;
  void* y;
  void* rq_codes;  // NULL: the requantized payload is not stored
  float* rq_scales;
  float* rq_zeros;
  int32_t* status;  // tagged only; NULL allowed
  int64_t rows;
  int H;
  int G;
  int lpg_shift;  // log2(G / 16)
  int P;
  float eps;
  uint32_t epoch;
};

int num_sms();

// Launches kern<<<grid, block, smem, st>>>(args...) with programmatic stream
// serialization: the kernel may be scheduled while the previous kernel in st
// is finishing (each kernel starts with pdl_begin(), which waits for it), so
// back-to-back calls lose no launch gap.  Returns the launch status.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       const Args&... args) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Host-side memo of occupancy answers (resident CTAs, or clusters, per SM)
// for one kernel at one launch shape on the current device.  Each answer is
// queried once and then reused, so a call's host cost is its launch and not
// the occupancy calculator.  Thread-safe.
struct OccKey {
  const void* fn;
  int dev, threads, smem, cluster;
};
bool occ_memo_find(const OccKey& k, int* value);
void occ_memo_store(const OccKey& k, int value);
// Raises kernel fn's dynamic shared-memory limit on the current device to at
// least smem bytes; never lowers it, so every earlier launch shape of the
// kernel stays valid.
cudaError_t raise_smem_limit(const void* fn, int smem);
// query() runs on a miss; it raises the kernel's shared-memory limit where
// needed, and since the limit never drops, a remembered answer stays valid.
template <class Q>
int occupancy_memo(const void* fn, int threads, int smem, int cluster, Q query) {
  OccKey k{fn, 0, threads, smem, cluster};
  cudaGetDevice(&k.dev);
  int v = 0;
  if (occ_memo_find(k, &v)) return v;
  v = query();
  occ_memo_store(k, v);
  return v;
}

// Dynamic shared memory a TMA-staged fused CTA may use (GB300: 227 KB per CTA).
constexpr int kTmaSmemLimit = 224 * 1024;

// Fused-kernel choice: automatic, the register-streaming kernel, or the
// TMA-staged kernel.
enum FusedPath : int { kPathAuto = 0, kPathStream = 1, kPathTma = 2 };
bool fused_tma_eligible(int fmt, const FusedArgs& a);
cudaError_t launch_fused_tma(int fmt, const FusedArgs& a, int max_ctas, cudaStream_t st);
// Row-starved calls: each row shared by a cluster of CTAs (segments of the
// row); cudaErrorNotSupported when the row cannot be cut into such segments.
cudaError_t launch_fused_tma_cluster(int fmt, const FusedArgs& a, cudaStream_t st);
int64_t fused_tma_wave_rows(int fmt, const FusedArgs& a);
// Rows the fused kernel that a call would launch processes concurrently.
int64_t fused_wave_rows(int fmt, const FusedArgs& a);

// in_f32: input is fp32 (requantization) instead of bf16; deq_kind: a DeqOut.
cudaError_t launch_quantize(int fmt, bool in_f32, int deq_kind, const QuantJob& job,
                            cudaStream_t st);
// Sender quantization of P bf16 slabs straight into epoch-tagged blocks
// (fmt kINT8T / kINT4T; job.codes[p] are the block arrays).
cudaError_t launch_quantize_tagged(int fmt, const QuantJob& job, cudaStream_t st);
// {FC_OK, no index} into a call's two status words, ordered after the previous
// kernel in the stream and before the call's kernel (quant.cu).
cudaError_t launch_reset_status(int32_t* d_status, cudaStream_t st);
// Sum of dequantized slabs over the 16-element chunks [c0, c1).
// Standalone all-gather: shard p holds chunks [first[p], first[p+1]) of the
// whole tensor (16-element chunks), indexed from its own chunk 0; for the
// tagged formats codes[p] are its blocks and blk0[p] the global index of its
// first block (for stale reports).
struct GatherJob {
  const void* codes[8];
  const float* scales[8];
  const float* zeros[8];
  int64_t first[9];
  int64_t blk0[8];
  void* out;
  int32_t* status;
  int64_t chunks;
  int P, lpg_shift;
  uint32_t epoch;
};
cudaError_t launch_allgather(int fmt, bool out_f32, const GatherJob& j, cudaStream_t st);

cudaError_t launch_reduce(int fmt, const Slabs& s, int P, int G, int64_t c0, int64_t c1,
                          float* out, cudaStream_t st);
cudaError_t launch_pack_tagged(const void* const* x, void* const* blocks, int P, int64_t rows,
                               int H, uint32_t epoch, cudaStream_t st);
cudaError_t launch_fused(int fmt, const FusedArgs& a, int max_ctas, int path, cudaStream_t st);

}  // namespace fc
