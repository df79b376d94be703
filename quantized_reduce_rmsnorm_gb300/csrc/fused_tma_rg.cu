// fused_tma_rg.cu -- the compact build of the TMA-staged fused kernel
// (fused_tma_kernel.cuh) with the residual left out of the stage (RG), for
// the shapes whose staged residual makes shared memory, not the compact
// build's registers, bound the CTAs per SM (or leaves room only for a
// one-row stage).  A tagged slab row is 16/12 the bytes of the plain payload,
// so most of them are tagged.  Built for (fused_tma.cu chooses):
//   two slabs (INT8 g128, tagged INT4 g32 or INT8 g128): a two-row ring;
//   four tagged INT8 slabs: a one-row stage, whole or as two half-row
//     sub-stages;
//   eight INT4 slabs (plain or tagged): a one-row stage; for eight tagged
//     INT4 slabs also without the h row buffer (pass 2 reads h back from
//     residual_out), as a one-row stage or two half-row sub-stages;
//   eight INT8 slabs: two half-row sub-stages without the h row buffer, or
//     at H = 4096 a one-row stage as 128-thread CTAs;
//   rows of 8192 of two or four plain slabs in calls of eight waves or more:
//     128-thread CTAs without the h row buffer (a two-row ring for two
//     slabs, a one-row stage for four).
#include "fused_tma_kernel.cuh"

namespace fc {

namespace {

// HB: the shared-memory h row buffer (false: pass 2 reads h back from
// residual_out through L2).
template <int FMT, int NS, int PMAX, int SUB, bool HB>
constexpr bool rg_built() {
  if (HB) {
    if (FMT == kINT4T) return (PMAX == 2 && NS == 2 && SUB == 1) || (PMAX == 8 && NS == 1 && SUB == 1);
    if (FMT == kINT8T) return (PMAX == 2 && NS == 2 && SUB == 1) || (PMAX == 4 && NS == 1);
    if (FMT == kINT4) return PMAX == 8 && NS == 1 && SUB == 1;
    if (FMT == kINT8) return PMAX == 2 && NS == 2 && SUB == 1;
    return false;
  }
  // without the h row buffer: eight slabs (one-row stage or half-row
  // sub-stages), and the 128-thread CTAs of plain rows of 8192 (two-row
  // rings for two slabs, one-row stages for four)
  if (FMT == kINT4T) return PMAX == 8 && NS == 1;
  if (FMT == kINT8)
    return (PMAX == 8 && NS == 1) || (PMAX == 2 && NS == 2 && SUB == 1) || (PMAX == 4 && NS == 1 && SUB == 1);
  if (FMT == kINT4) return (PMAX == 2 && NS == 2 && SUB == 1) || (PMAX == 4 && NS == 1 && SUB == 1);
  return false;
}

template <int FMT, int NS, int PMAX, int SUB, bool HB>
int occ_t(int threads, int smem) {
  if constexpr (!rg_built<FMT, NS, PMAX, SUB, HB>()) {
    return 0;
  } else {
    auto kern = k_fused_tma<FMT, NS, PMAX, 1, true, SUB, true, HB>;
    return occupancy_memo(reinterpret_cast<const void*>(kern), threads, smem, 1, [&] {
      int o = 0;
      if (raise_smem_limit(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, threads, smem) != cudaSuccess)
        return 0;
      return o;
    });
  }
}

template <int FMT, int NS, int SUB, bool HB>
int occ_p(int P, int threads, int smem) {
  if (P <= 2) return occ_t<FMT, NS, 2, SUB, HB>(threads, smem);
  if (P <= 4) return occ_t<FMT, NS, 4, SUB, HB>(threads, smem);
  return occ_t<FMT, NS, 8, SUB, HB>(threads, smem);
}

template <int FMT, bool HB>
int occ_fmt(int P, int nstage, int sub, int threads, int smem) {
  if (nstage == 2) return sub == 1 ? occ_p<FMT, 2, 1, HB>(P, threads, smem) : 0;
  return sub == 1 ? occ_p<FMT, 1, 1, HB>(P, threads, smem) : occ_p<FMT, 1, 2, HB>(P, threads, smem);
}

template <int FMT, int NS, int PMAX, int SUB, bool HB>
cudaError_t launch_t(const FusedArgs& a, const TmaGeom& g, int threads, int smem, int64_t grid,
                     cudaStream_t st) {
  if constexpr (!rg_built<FMT, NS, PMAX, SUB, HB>()) {
    return cudaErrorInvalidConfiguration;
  } else {
    return launch_pdl(k_fused_tma<FMT, NS, PMAX, 1, true, SUB, true, HB>, dim3(static_cast<unsigned>(grid)),
                      dim3(threads), smem, st, a, g);
  }
}

template <int FMT, int NS, int SUB, bool HB>
cudaError_t launch_p(const FusedArgs& a, const TmaGeom& g, int threads, int smem, int64_t grid,
                     cudaStream_t st) {
  if (a.P <= 2) return launch_t<FMT, NS, 2, SUB, HB>(a, g, threads, smem, grid, st);
  if (a.P <= 4) return launch_t<FMT, NS, 4, SUB, HB>(a, g, threads, smem, grid, st);
  return launch_t<FMT, NS, 8, SUB, HB>(a, g, threads, smem, grid, st);
}

template <int FMT, bool HB>
cudaError_t launch_fmt(int nstage, int sub, const FusedArgs& a, const TmaGeom& g, int threads, int smem,
                       int64_t grid, cudaStream_t st) {
  if (nstage == 2)
    return sub == 1 ? launch_p<FMT, 2, 1, HB>(a, g, threads, smem, grid, st) : cudaErrorInvalidConfiguration;
  return sub == 1 ? launch_p<FMT, 1, 1, HB>(a, g, threads, smem, grid, st)
                  : launch_p<FMT, 1, 2, HB>(a, g, threads, smem, grid, st);
}

template <bool HB>
int occ_any(int fmt, int P, int nstage, int sub, int threads, int smem) {
  switch (fmt) {
    case kINT4T: return occ_fmt<kINT4T, HB>(P, nstage, sub, threads, smem);
    case kINT8T: return occ_fmt<kINT8T, HB>(P, nstage, sub, threads, smem);
    case kINT4: return occ_fmt<kINT4, HB>(P, nstage, sub, threads, smem);
    case kINT8: return occ_fmt<kINT8, HB>(P, nstage, sub, threads, smem);
    default: return 0;
  }
}

template <bool HB>
cudaError_t launch_any(int fmt, int nstage, int sub, const FusedArgs& a, const TmaGeom& g, int threads,
                       int smem, int64_t grid, cudaStream_t st) {
  switch (fmt) {
    case kINT4T: return launch_fmt<kINT4T, HB>(nstage, sub, a, g, threads, smem, grid, st);
    case kINT8T: return launch_fmt<kINT8T, HB>(nstage, sub, a, g, threads, smem, grid, st);
    case kINT4: return launch_fmt<kINT4, HB>(nstage, sub, a, g, threads, smem, grid, st);
    case kINT8: return launch_fmt<kINT8, HB>(nstage, sub, a, g, threads, smem, grid, st);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace

int fused_tma_rg_occupancy(int fmt, int P, int nstage, int sub, bool hb, int threads, int smem) {
  if (threads > 256 || smem > kTmaSmemLimit) return 0;
  return hb ? occ_any<true>(fmt, P, nstage, sub, threads, smem) : occ_any<false>(fmt, P, nstage, sub, threads, smem);
}

cudaError_t launch_fused_tma_rg(int fmt, int nstage, int sub, bool hb, const FusedArgs& a, const TmaGeom& g,
                                int threads, int smem, int64_t grid, cudaStream_t st) {
  return hb ? launch_any<true>(fmt, nstage, sub, a, g, threads, smem, grid, st)
            : launch_any<false>(fmt, nstage, sub, a, g, threads, smem, grid, st);
}

}  // namespace fc
