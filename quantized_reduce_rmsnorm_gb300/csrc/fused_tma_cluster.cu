// fused_tma_cluster.cu -- the TMA-staged fused kernel for calls with too few
// rows to occupy the GPU (decode-sized batches): each row is shared by a
// thread-block cluster of CL CTAs, each CTA staging and processing its own
// contiguous segment of the row; the row's sum of squares is completed across
// the cluster through distributed shared memory (fused_tma_kernel.cuh).
#include "fused_tma_kernel.cuh"

namespace fc {

namespace {

template <int FMT, int PMAX, int CL>
cudaError_t launch_cl(const FusedArgs& a, const TmaGeom& g, cudaStream_t st) {
  auto kern = k_fused_tma<FMT, 1, PMAX, CL>;
  const int smem = g.stage_off + g.stage_bytes;
  // one chunk per thread (the segments are short), at least two warps
  int threads = (g.cps + 31) & ~31;
  threads = threads < 64 ? 64 : (threads > kTmaThreadsMax ? kTmaThreadsMax : threads);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const int clusters = occupancy_memo(reinterpret_cast<const void*>(kern), threads, smem, CL, [&] {
    int c = 0;
    if (raise_smem_limit(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&c, kern, &cfg) != cudaSuccess)
      return 0;
    return c;
  });
  if (clusters < 1) return cudaErrorNotSupported;
  const int64_t n = a.rows < clusters ? a.rows : clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(n * CL));
  cudaLaunchAttribute at2[2] = {at[0], {}};  // + programmatic stream serialization (launch_pdl)
  at2[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at2[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at2;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a, g);
}

template <int FMT, int CL>
cudaError_t launch_p(const FusedArgs& a, const TmaGeom& g, cudaStream_t st) {
  if (a.P <= 2) return launch_cl<FMT, 2, CL>(a, g, st);
  if (a.P <= 4) return launch_cl<FMT, 4, CL>(a, g, st);
  return launch_cl<FMT, 8, CL>(a, g, st);
}

template <int CL>
cudaError_t launch_fmt(int fmt, const FusedArgs& a, const TmaGeom& g, cudaStream_t st) {
  switch (fmt) {
    case kBF16: return launch_p<kBF16, CL>(a, g, st);
    case kINT8: return launch_p<kINT8, CL>(a, g, st);
    case kINT8T: return launch_p<kINT8T, CL>(a, g, st);
    case kINT4T: return launch_p<kINT4T, CL>(a, g, st);
    default: return launch_p<kINT4, CL>(a, g, st);
  }
}

}  // namespace

// Rows split over clusters of 8 (or 4) CTAs when the segments are whole groups
// of 16-byte multiples; cudaErrorNotSupported when neither cut is possible
// (the caller then launches a CTA per row).
cudaError_t launch_fused_tma_cluster(int fmt, const FusedArgs& a, cudaStream_t st) {
  TmaGeom g;
  if (geometry(fmt, a, g, 8) && g.stage_off + g.stage_bytes <= kTmaSmemLimit)
    return launch_fmt<8>(fmt, a, g, st);
  if (geometry(fmt, a, g, 4) && g.stage_off + g.stage_bytes <= kTmaSmemLimit)
    return launch_fmt<4>(fmt, a, g, st);
  return cudaErrorNotSupported;
}

}  // namespace fc
