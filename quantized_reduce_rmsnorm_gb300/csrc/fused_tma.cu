// fused_tma.cu -- launches of the TMA-staged fused kernel
// (fused_tma_kernel.cuh): one CTA per row at a time, the launch shape chosen
// from the row length, format and slab count; row-starved calls go to the
// cluster launches of fused_tma_cluster.cu.
#include "fused_tma_kernel.cuh"

namespace fc {

namespace {

// Launch shape of one instantiation: threads per CTA and resident CTAs per SM.
struct TmaShape {
  int nstage = 0, threads = 0, occ = 0, smem = 0;
  bool compact = false;  // the compact build (fused_tma_compact.cu)
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
  sh.threads = tma_threads(FMT, a.P, a.H);
  sh.occ = occupancy_memo(reinterpret_cast<const void*>(kern), sh.threads, sh.smem, 1, [&] {
    int o = 0;
    if (raise_smem_limit(reinterpret_cast<const void*>(kern), sh.smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, sh.threads, sh.smem) != cudaSuccess)
      return 0;
    return o;
  });
  return sh;
}

// A two-row ring (the next row streams in while this one is computed).  For
// the quantized formats, when that ring leaves room for a single CTA per SM,
// two single-stage CTAs (which overlap each other's copies and row
// barriers) were measured faster; for bf16 rows the two-row ring stays.
template <int FMT, int PMAX>
TmaShape choose_full(const FusedArgs& a, const TmaGeom& g) {
  const TmaShape two = shape_t<FMT, 2, PMAX>(a, g);
  if (FMT == kBF16 && two.occ >= 1) return two;
  const TmaShape one = shape_t<FMT, 1, PMAX>(a, g);
  if (two.occ >= 1 && (two.occ >= 2 || one.occ <= two.occ)) return two;
  return one;
}

// For the quantized formats the compact build replaces that choice where it
// holds more CTAs per SM (shared memory, not registers, then bounds the
// count); bf16 rows measured slower with it.
template <int FMT, int PMAX>
TmaShape choose_shape(const FusedArgs& a, const TmaGeom& g) {
  TmaShape best = choose_full<FMT, PMAX>(a, g);
  if (FMT == kBF16 || best.threads < 1 || best.threads > 256) return best;
  for (int ns = 2; ns >= 1; --ns) {
    const int smem = g.stage_off + ns * g.stage_bytes;
    const int occ = fused_tma_compact_occupancy(FMT, a.P, ns, best.threads, smem);
    if (occ > best.occ) {
      best.nstage = ns, best.occ = occ, best.smem = smem, best.compact = true;
      break;
    }
  }
  return best;
}

// Two half-row sub-stages in place of a one-row stage (k_fused_tma's SUB):
// for the quantized formats (plain or in tagged blocks) with a one-stage
// ring whose row is exactly two passes of 256 threads (H = 8192), when the
// half-row pieces are whole groups of 16-byte multiples.  Measured on GB300
// against the one-row stage: prefill (INT4, P=4) 132.7 -> 126.9 us, its
// tagged form 146.5 -> 137.3 us, INT8 with two slabs at 64 MB 0.75 -> 0.84
// of the HBM peak, 16 MB messages up to +0.13; rows of 4096 (128 threads,
// smaller copies) were slower with it (INT4 P=8 0.64 -> 0.56) and keep the
// one-row stage.  Returns the half-row geometry in g2 (its h buffer sized
// for the whole row) and the occupancy of that build, 0 when not applicable.
template <int FMT, int PMAX, bool COMPACT>
int sub_shape(const FusedArgs& a, const TmaShape& sh, TmaGeom& g2) {
  if (FMT != kINT8 && FMT != kINT4 && FMT != kINT8T && FMT != kINT4T) return 0;
  if (sh.nstage != 1 || sh.threads != 256 || (a.H >> 4) != 2 * sh.threads) return 0;
  if (!geometry(FMT, a, g2, 2)) return 0;
  g2.stage_off = (2 * a.H + 127) & ~127;
  const int smem = g2.stage_off + 2 * g2.stage_bytes;
  if (smem > kTmaSmemLimit) return 0;
  auto kern = k_fused_tma<FMT, 1, PMAX, 1, COMPACT, 2>;
  return occupancy_memo(reinterpret_cast<const void*>(kern), sh.threads, smem, 1, [&] {
    int o = 0;
    if (raise_smem_limit(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, sh.threads, smem) != cudaSuccess)
      return 0;
    return o;
  });
}

// The half-row sub-stages without the residual in them (k_fused_tma's RG),
// for eight slabs at H = 8192 where it raises the CTAs per SM:
// * tagged INT8: its 104 KB row of tagged blocks plus the residual and h left
//   room for one CTA per SM (which then took a two-row ring); without the
//   residual two fit (64 MB 0.51 -> 0.67 of the measured HBM peak);
// * INT4: 64 KB with the residual and h held two CTAs per SM; without the
//   residual, the compact build (gamma read per row from L1, no spills) runs
//   three (64 MB 0.65 -> 0.71, 256 MB 0.68 -> 0.74).
// Returns that occupancy (0 when not applicable), the geometry in g3 and the
// build in compact.
template <int FMT, int PMAX>
int rg_shape(const FusedArgs& a, const TmaShape& sh, TmaGeom& g3, bool& compact) {
  compact = false;
  if constexpr (PMAX != 8 || (FMT != kINT8T && FMT != kINT4)) {
    return 0;
  } else {
    if (sh.threads != 256 || (a.H >> 4) != 2 * sh.threads) return 0;  // (any ring depth)
    if (!geometry(FMT, a, g3, 2)) return 0;
    g3.stage_bytes -= 32 * g3.cps;  // no residual in the stage
    g3.stage_off = (2 * a.H + 127) & ~127;
    const int smem = g3.stage_off + 2 * g3.stage_bytes;
    if (smem > kTmaSmemLimit) return 0;
    auto occ_of = [&](auto kern) {
      return occupancy_memo(reinterpret_cast<const void*>(kern), sh.threads, smem, 1, [&] {
        int o = 0;
        if (raise_smem_limit(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, sh.threads, smem) != cudaSuccess)
          return 0;
        return o;
      });
    };
    const int of = occ_of(k_fused_tma<FMT, 1, PMAX, 1, false, 2, true>);
    const int oc = FMT == kINT4 ? occ_of(k_fused_tma<FMT, 1, PMAX, 1, true, 2, true>) : 0;
    compact = oc > of;
    return compact ? oc : of;
  }
}

// The residual-free compact build (fused_tma_rg.cu) for shapes of the
// quantized formats whose staged residual makes shared memory bound the CTAs
// per SM below what the compact build's registers allow, or leaves room only
// for a one-row stage (most of them tagged: a tagged slab row is 16/12 the
// bytes of the plain payload).  Among the
// builds of fused_tma_rg.cu (a two-row ring; a one-row stage; two half-row
// sub-stages) the plan with the most CTAs per SM, then the deepest ring, is
// returned when it beats the current plan (occ_now CTAs per SM, a ring of
// depth_now half rows: 4 two-row ring, 3 half-row sub-stages, 2 one row):
// more CTAs per SM, or as many with a two-row ring in place of a one-row
// stage.  Measured on GB300 against the staged residual (64 MB messages,
// fraction of the measured HBM peak): eight INT4 slabs at H = 4096
// 0.71 -> 0.79 (five -> six CTAs; 32 MB 0.64 -> 0.71); four tagged INT8 slabs
// 0.75 -> 0.82 at H = 4096 (five -> six) and H = 8192 (two -> three); two
// tagged INT4 slabs at H = 4096 0.65 -> 0.67 (five -> six); eight tagged INT4
// slabs at H = 4096 0.66 -> 0.68 (four -> five); two tagged INT8 slabs at
// H = 4096 0.77 -> 0.80 (a two-row ring).  Slower, and not taken: a two-row
// ring in place of half-row sub-stages at the same count (two slabs,
// H = 8192; +4-6% at 16 MB) or of a one-row stage for four plain INT4 slabs
// (+2-7%), and an L2 prefetch of each row's residual (eight INT4 slabs at
// H = 8192, 64 MB: 88 -> 109 us).  Eight tagged INT4 slabs also drop the h
// row buffer (pass 2 reads h back from residual_out through L2), for a
// third CTA per SM at H = 8192 and a sixth at 4096: 64 MB 0.70 -> 0.72 and
// 0.70 -> 0.75, 256 MB 0.73 -> 0.76 and 0.76 -> 0.80; so do eight plain INT8
// slabs at H = 8192 (two -> three CTAs): 16 MB 0.67 -> 0.70, 64 MB
// 0.84 -> 0.94, 256 MB 0.90 -> 0.98.  At equal resident warps the smaller
// CTA is taken: eight INT8 slabs at H = 4096 as six 128-thread CTAs (two
// chunks a thread, no h row buffer) in place of three of 256: 64 MB
// 0.76 -> 0.93, 256 MB 0.82 -> 0.97, 16 MB 0.61 -> 0.67 (a CTA barrier waits
// on four warps, not eight).
struct RgPlan {
  int occ = 0, nstage = 0, sub = 0, smem = 0, threads = 0;
  bool hb = true;  // h in the shared-memory row buffer (else read back from residual_out)
  TmaGeom g{};
};
template <int FMT>
RgPlan rg_plan(const FusedArgs& a, int threads, int occ_now, int depth_now) {
  RgPlan best;
  int best_depth = 0;
  if (FMT == kBF16) return best;
  // Candidates (stages, sub-stages, h row buffer, threads halved), those
  // with the h row buffer first, so that where two tie the build that keeps
  // h on chip is taken.  256-thread builds of the plain formats are also
  // tried at 128 threads (twice the chunks a thread), as six four-warp CTAs
  // per SM in place of three eight-warp ones; not those of the tagged
  // formats: four tagged INT4 slabs at H = 8192 so built ran as fast alone,
  // but the prefill-qtagged step, back to back, went 245 -> 303 us with
  // unchanged per-stage times.
  const int cands[10][4] = {{2, 1, 1, 0}, {1, 2, 1, 0}, {1, 1, 1, 0}, {2, 1, 0, 0}, {1, 2, 0, 0}, {1, 1, 0, 0},
                            {2, 1, 1, 1}, {1, 1, 1, 1}, {2, 1, 0, 1}, {1, 1, 0, 1}};
  for (const auto& c : cands) {
    const int ns = c[0], sub = c[1];
    const bool hb = c[2] != 0;
    const int thr = c[3] ? threads / 2 : threads;
    if (c[3] && (threads != 256 || FMT == kINT4T || FMT == kINT8T)) continue;
    if (sub == 2 && (thr != 256 || (a.H >> 4) != 2 * thr)) continue;
    TmaGeom g;
    if (!geometry(FMT, a, g, sub)) continue;
    g.stage_bytes -= 32 * g.cps;  // no residual in the stage
    g.stage_off = hb ? (2 * a.H + 127) & ~127 : 0;
    const int smem = g.stage_off + ns * sub * g.stage_bytes;
    if (smem > kTmaSmemLimit) continue;
    const int occ = fused_tma_rg_occupancy(FMT, a.P, ns, sub, hb, thr, smem);
    const int depth = ns == 2 ? 4 : sub == 2 ? 3 : 2;
    // compared by resident warps, then ring depth, then the smaller CTA
    const int w = occ * thr, bw = best.occ * best.threads;
    if (w > bw || (w == bw && occ > 0 && (depth > best_depth || (depth == best_depth && thr < best.threads)))) {
      best.occ = occ, best.nstage = ns, best.sub = sub, best.smem = smem, best.g = g, best.hb = hb;
      best.threads = thr;
      best_depth = depth;
    }
  }
  const int64_t warps_now = static_cast<int64_t>(occ_now) * threads, warps = static_cast<int64_t>(best.occ) * best.threads;
  if (!(warps > warps_now || (warps == warps_now && (best_depth >= depth_now + 2 || best.threads < threads))))
    best.occ = 0;
  // Taken for calls of eight waves or more only:
  // * two plain INT8 slabs carry the least work per chunk to hide the threads'
  //   residual loads behind: at H = 4096 the build measured faster from 64 MB
  //   (0.80 -> 0.92 of the measured HBM peak), slower at 16 and 32 MB
  //   (0.74 -> 0.65, 0.87 -> 0.83);
  // * 128-thread CTAs with four chunks a thread (rows of 8192) take twice as
  //   long per row: faster on long calls (256 MB, two or four INT4 or INT8
  //   slabs, 4-9%; prefill fused 119 -> 112 us), slower at 16 and 64 MB
  //   (2-26%).
  const bool long_only = (FMT == kINT8 && a.P <= 2) || (best.threads < threads && (a.H >> 4) > 2 * best.threads);
  if (long_only && a.rows < 8 * static_cast<int64_t>(num_sms()) * best.occ) best.occ = 0;
  return best;
}

template <int FMT, int PMAX>
cudaError_t launch_tma_p(const FusedArgs& a, const TmaGeom& g, int max_ctas, cudaStream_t st) {
  const TmaShape sh = choose_shape<FMT, PMAX>(a, g);
  if (sh.occ < 1) return cudaErrorInvalidConfiguration;
  // a batch too small to give every SM a CTA (decode): share each row among
  // a cluster of CTAs instead, not under a CTA budget, which caps CTAs.
  // Measured on GB300 (back-to-back calls, a CTA per row -> clusters): rows
  // of 8192, 8..128 of them, 0.4-2.2 us faster (eight INT8 slabs, 64 rows:
  // 7.8 -> 6.4 us); 192 rows 6.5 -> 10.6 us slower (more clusters than fit
  // at once); plain rows of 4096 slower at every count (64 rows, eight INT8
  // slabs: 5.2 -> 6.5 us), tagged ones faster (INT4, two slabs, 32 rows:
  // 10.8 -> 9.4 us); a single row gains nothing.
  constexpr bool kTagged = FMT == kINT8T || FMT == kINT4T;
  if (max_ctas == 0 && a.rows >= 8 && a.rows <= 128 && (a.H >= 8192 || kTagged) &&
      2 * a.rows <= static_cast<int64_t>(num_sms()) * sh.occ) {
    const cudaError_t e = launch_fused_tma_cluster(FMT, a, st);
    if (e != cudaErrorNotSupported) return e;
  }
  int64_t grid = static_cast<int64_t>(num_sms()) * sh.occ;
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  if (grid > a.rows) grid = a.rows;
  if constexpr (PMAX == 8 && (FMT == kINT8T || FMT == kINT4)) {
    TmaGeom g3;
    bool compact = false;
    const int occ3 = rg_shape<FMT, PMAX>(a, sh, g3, compact);
    // only for more rows than one wave of the staged build: a lone row per
    // CTA ran slower there (a row of gamma from L2, not registers; 256 rows
    // of eight INT4 slabs 9.8 -> 12.3 us)
    if (occ3 > sh.occ && a.rows > static_cast<int64_t>(num_sms()) * sh.occ) {
      int64_t grid3 = static_cast<int64_t>(num_sms()) * occ3;
      if (max_ctas > 0 && grid3 > max_ctas) grid3 = max_ctas;
      if (grid3 > a.rows) grid3 = a.rows;
      const dim3 gr3(static_cast<unsigned>(grid3));
      const int smem3 = g3.stage_off + 2 * g3.stage_bytes;
      if (compact) return launch_pdl(k_fused_tma<FMT, 1, PMAX, 1, true, 2, true>, gr3, dim3(sh.threads), smem3, st, a, g3);
      return launch_pdl(k_fused_tma<FMT, 1, PMAX, 1, false, 2, true>, gr3, dim3(sh.threads), smem3, st, a, g3);
    }
  }
  {
    TmaGeom g2;
    const int occ2 = sh.compact ? sub_shape<FMT, PMAX, true>(a, sh, g2) : sub_shape<FMT, PMAX, false>(a, sh, g2);
    const bool sub2 = occ2 >= sh.occ && occ2 > 0;
    if constexpr (FMT != kBF16) {
      // only for more rows than one wave of the current plan (as above), and
      // not under a CTA cap below that wave: there the CTAs per SM these
      // plans add do not count, and the 128-thread ones make each CTA slower
      const int64_t wave = static_cast<int64_t>(num_sms()) * sh.occ;
      if (a.rows > wave && (max_ctas == 0 || max_ctas >= wave)) {
        const RgPlan rp = rg_plan<FMT>(a, sh.threads, sub2 ? occ2 : sh.occ,
                                              sub2 ? 3 : 2 * sh.nstage);
        if (rp.occ > 0) {
          int64_t grid4 = static_cast<int64_t>(num_sms()) * rp.occ;
          if (max_ctas > 0 && grid4 > max_ctas) grid4 = max_ctas;
          if (grid4 > a.rows) grid4 = a.rows;
          return launch_fused_tma_rg(FMT, rp.nstage, rp.sub, rp.hb, a, rp.g, rp.threads, rp.smem, grid4, st);
        }
      }
    }
    if (sub2) {
      const int smem2 = g2.stage_off + 2 * g2.stage_bytes;
      if (sh.compact)
        return launch_pdl(k_fused_tma<FMT, 1, PMAX, 1, true, 2>, dim3(static_cast<unsigned>(grid)),
                          dim3(sh.threads), smem2, st, a, g2);
      return launch_pdl(k_fused_tma<FMT, 1, PMAX, 1, false, 2>, dim3(static_cast<unsigned>(grid)),
                        dim3(sh.threads), smem2, st, a, g2);
    }
  }
  if (sh.compact)
    return launch_fused_tma_compact(FMT, sh.nstage, a, g, sh.threads, sh.smem, grid, st);
  const dim3 gr(static_cast<unsigned>(grid));
  if (sh.nstage == 2) return launch_pdl(k_fused_tma<FMT, 2, PMAX>, gr, dim3(sh.threads), sh.smem, st, a, g);
  return launch_pdl(k_fused_tma<FMT, 1, PMAX>, gr, dim3(sh.threads), sh.smem, st, a, g);
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

// CTAs per SM of the plan launch_tma_p takes for a call of a.rows rows
// (the cluster launch aside): the same choices in the same order.
template <int FMT, int PMAX>
int plan_occ(const FusedArgs& a, const TmaGeom& g) {
  const TmaShape sh = choose_shape<FMT, PMAX>(a, g);
  if (sh.occ < 1) return 1;
  const bool more = a.rows > static_cast<int64_t>(num_sms()) * sh.occ;
  if constexpr (PMAX == 8 && (FMT == kINT8T || FMT == kINT4)) {
    TmaGeom g3;
    bool compact = false;
    const int occ3 = rg_shape<FMT, PMAX>(a, sh, g3, compact);
    if (occ3 > sh.occ && more) return occ3;
  }
  if constexpr (FMT != kBF16) {
    if (more) {
      TmaGeom g2;
      const int occ2 = sh.compact ? sub_shape<FMT, PMAX, true>(a, sh, g2) : sub_shape<FMT, PMAX, false>(a, sh, g2);
      const bool sub2 = occ2 >= sh.occ && occ2 > 0;
      const RgPlan rp = rg_plan<FMT>(a, sh.threads, sub2 ? occ2 : sh.occ, sub2 ? 3 : 2 * sh.nstage);
      if (rp.occ > 0) return rp.occ;
    }
  }
  return sh.occ;
}

template <int FMT>
int64_t wave_fmt(const FusedArgs& a, const TmaGeom& g) {
  const int occ = a.P <= 2 ? plan_occ<FMT, 2>(a, g) : a.P <= 4 ? plan_occ<FMT, 4>(a, g) : plan_occ<FMT, 8>(a, g);
  return static_cast<int64_t>(num_sms()) * occ;  // a CTA per row
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
