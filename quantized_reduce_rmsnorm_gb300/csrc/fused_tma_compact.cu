// fused_tma_compact.cu -- the compact build of the TMA-staged fused kernel
// (fused_tma_kernel.cuh): at most 256 threads and three CTAs' worth of
// registers per SM.  fused_tma.cu launches it instead of the full build when
// shared memory admits more CTAs per SM than the full build's registers do
// (measured on GB300: INT4 rows of two slabs 0.57 -> 0.64 of the HBM peak,
// INT8 rows of four slabs at H = 8192 0.73 -> 0.88); elsewhere its spills
// only cost time.
#include "fused_tma_kernel.cuh"

namespace fc {

namespace {

template <int FMT, int NS, int PMAX>
int occ_t(int threads, int smem) {
  auto kern = k_fused_tma<FMT, NS, PMAX, 1, true>;
  return occupancy_memo(reinterpret_cast<const void*>(kern), threads, smem, 1, [&] {
    int o = 0;
    if (raise_smem_limit(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, threads, smem) != cudaSuccess)
      return 0;
    return o;
  });
}

template <int FMT, int NS>
int occ_p(int P, int threads, int smem) {
  if (P <= 2) return occ_t<FMT, NS, 2>(threads, smem);
  if (P <= 4) return occ_t<FMT, NS, 4>(threads, smem);
  return occ_t<FMT, NS, 8>(threads, smem);
}

template <int NS>
int occ_fmt(int fmt, int P, int threads, int smem) {
  switch (fmt) {
    case kBF16: return occ_p<kBF16, NS>(P, threads, smem);
    case kINT8: return occ_p<kINT8, NS>(P, threads, smem);
    case kINT8T: return occ_p<kINT8T, NS>(P, threads, smem);
    case kINT4T: return occ_p<kINT4T, NS>(P, threads, smem);
    default: return occ_p<kINT4, NS>(P, threads, smem);
  }
}

template <int FMT, int NS>
cudaError_t launch_p(const FusedArgs& a, const TmaGeom& g, int threads, int smem, int64_t grid,
                     cudaStream_t st) {
  const dim3 gr(static_cast<unsigned>(grid));
  if (a.P <= 2) return launch_pdl(k_fused_tma<FMT, NS, 2, 1, true>, gr, dim3(threads), smem, st, a, g);
  if (a.P <= 4) return launch_pdl(k_fused_tma<FMT, NS, 4, 1, true>, gr, dim3(threads), smem, st, a, g);
  return launch_pdl(k_fused_tma<FMT, NS, 8, 1, true>, gr, dim3(threads), smem, st, a, g);
}

template <int NS>
cudaError_t launch_fmt(int fmt, const FusedArgs& a, const TmaGeom& g, int threads, int smem,
                       int64_t grid, cudaStream_t st) {
  switch (fmt) {
    case kBF16: return launch_p<kBF16, NS>(a, g, threads, smem, grid, st);
    case kINT8: return launch_p<kINT8, NS>(a, g, threads, smem, grid, st);
    case kINT8T: return launch_p<kINT8T, NS>(a, g, threads, smem, grid, st);
    case kINT4T: return launch_p<kINT4T, NS>(a, g, threads, smem, grid, st);
    default: return launch_p<kINT4, NS>(a, g, threads, smem, grid, st);
  }
}

}  // namespace

int fused_tma_compact_occupancy(int fmt, int P, int nstage, int threads, int smem) {
  if (threads > 256 || smem > kTmaSmemLimit) return 0;
  return nstage == 2 ? occ_fmt<2>(fmt, P, threads, smem) : occ_fmt<1>(fmt, P, threads, smem);
}

cudaError_t launch_fused_tma_compact(int fmt, int nstage, const FusedArgs& a, const TmaGeom& g,
                                     int threads, int smem, int64_t grid, cudaStream_t st) {
  return nstage == 2 ? launch_fmt<2>(fmt, a, g, threads, smem, grid, st)
                     : launch_fmt<1>(fmt, a, g, threads, smem, grid, st);
}

}  // namespace fc
