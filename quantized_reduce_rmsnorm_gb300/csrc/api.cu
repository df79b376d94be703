// api.cu -- the libfcomm C ABI: argument validation and kernel dispatch.
// Every entry point validates all arguments before it launches anything,
// never allocates, frees or synchronizes, and launches on the caller's
// stream.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <algorithm>

#include "fcomm.h"
#include "internal.h"

namespace {

thread_local char g_msg[512] = "";

fc_status fail(fc_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return st;
}

fc_status ok() {
  g_msg[0] = '\0';
  return FC_OK;
}

fc_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(FC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool quantized(int fmt) { return fmt == FC_FMT_INT8_SYM || fmt == FC_FMT_INT4_ASYM; }
bool qtagged(int fmt) { return fmt == FC_FMT_INT8_TAGGED || fmt == FC_FMT_INT4_TAGGED; }
int base_fmt(int fmt) {
  return fmt == FC_FMT_INT8_TAGGED ? FC_FMT_INT8_SYM : fmt == FC_FMT_INT4_TAGGED ? FC_FMT_INT4_ASYM : fmt;
}

// Common shape/spec checks.  needs_group: the format is quantized.
fc_status check_shape(fc_qspec spec, int64_t rows, int64_t hidden, bool quant_only) {
  if (rows < 0) return fail(FC_ERR_INVALID, "rows must be >= 0 (got %lld)", (long long)rows);
  if (hidden <= 0 || hidden % 16 != 0)
    return fail(FC_ERR_INVALID, "hidden must be a positive multiple of 16 (got %lld)",
                (long long)hidden);
  if (hidden > 65536) return fail(FC_ERR_UNSUPPORTED, "hidden > 65536 is not supported");
  if (quant_only && !quantized(spec.fmt))
    return fail(FC_ERR_INVALID, "format %d is not a quantized format", spec.fmt);
  if (qtagged(spec.fmt)) {
    const int want = spec.fmt == FC_FMT_INT8_TAGGED ? 128 : 32;
    if (spec.group != want)
      return fail(FC_ERR_UNSUPPORTED, "the tagged quantized format needs group %d (got %d)", want,
                  spec.group);
    if (hidden % want != 0)
      return fail(FC_ERR_INVALID, "hidden (%lld) must be a multiple of group (%d)",
                  (long long)hidden, want);
  } else if (quantized(spec.fmt)) {
    const int G = spec.group;
    if (G < 16 || G > 512 || (G & (G - 1)) != 0)
      return fail(FC_ERR_INVALID, "group must be a power of two in [16, 512] (got %d)", G);
    if (hidden % G != 0)
      return fail(FC_ERR_INVALID, "hidden (%lld) must be a multiple of group (%d)",
                  (long long)hidden, G);
  } else if (spec.fmt != FC_FMT_BF16 && spec.fmt != FC_FMT_BF16_TAGGED) {
    return fail(FC_ERR_INVALID, "unknown format %d", spec.fmt);
  }
  return FC_OK;
}

fc_status check_ptr(const void* p, size_t align, const char* name) {
  if (!p) return fail(FC_ERR_INVALID, "%s must not be NULL", name);
  if (!aligned(p, align)) return fail(FC_ERR_INVALID, "%s must be %zu-byte aligned", name, align);
  return FC_OK;
}

fc_status check_qtensor(const fc_qtensor& t, int fmt, const char* name) {
  char buf[64];
  snprintf(buf, sizeof buf, "%s.codes", name);
  if (fc_status s = check_ptr(t.codes, 16, buf)) return s;
  if (quantized(fmt)) {
    snprintf(buf, sizeof buf, "%s.scales", name);
    if (fc_status s = check_ptr(t.scales, 4, buf)) return s;
    if (fmt == FC_FMT_INT4_ASYM) {
      snprintf(buf, sizeof buf, "%s.zeros", name);
      if (fc_status s = check_ptr(t.zeros, 4, buf)) return s;
    }
  } else if (fmt == FC_FMT_BF16 && !aligned(t.codes, 32)) {
    return fail(FC_ERR_INVALID, "%s.codes (bf16 data) must be 32-byte aligned", name);
  }
  return FC_OK;
}

}  // namespace

namespace {

#include "rates.inc"

// One call's device time from a measured table (rates.inc): encoding f
// (table order), P slabs, rows x hidden bf16 partial sums.  The table's
// hidden (4096 or 8192) nearest to `hidden`; message bytes interpolated
// log-linearly between the measured sizes 16 KB .. 256 MB (the 16 KB time
// below them, proportional to bytes above); P linearly between 2, 4 and 8.
// 0 where the table holds 0 (bf16 has no sender).
double table_us(const double (&t)[6][3][2][15], int f, int P, int64_t rows, int64_t hidden) {
  const int h = hidden > 6144 ? 1 : 0;
  const double M = 2.0 * static_cast<double>(rows) * static_cast<double>(hidden);
  auto at = [&](int pi) {
    const double* v = t[f][pi][h];
    const double m0 = 16384.0;
    if (v[0] <= 0.0) return 0.0;
    if (M <= m0) return v[0];
    const double x = std::log2(M / m0);
    if (x >= 14.0) return v[14] * M / (m0 * 16384.0);
    const int i = static_cast<int>(x);
    const double fr = x - i;
    return std::exp2((1.0 - fr) * std::log2(v[i]) + fr * std::log2(v[i + 1]));
  };
  if (P <= 2) return at(0);
  if (P <= 4) return at(0) + (at(1) - at(0)) * (P - 2) / 2.0;
  return at(1) + (at(2) - at(1)) * (P - 4) / 4.0;
}

// The encodings, in the order of the measured table.
struct Cand {
  int fmt, group, bits;
  bool tagged;
};
const Cand kCands[6] = {
    {FC_FMT_BF16, 0, 16, false},       {FC_FMT_BF16_TAGGED, 0, 16, true},
    {FC_FMT_INT8_SYM, 128, 8, false},  {FC_FMT_INT8_TAGGED, 128, 8, true},
    {FC_FMT_INT4_ASYM, 32, 4, false},  {FC_FMT_INT4_TAGGED, 32, 4, true},
};

// Estimated us of one all-reduce step in encoding f: this GPU's measured
// fused call and sender call (interpolated), plus, with a link model, the
// wire time of the two-step reduce (2 (P-1)/P of a slab's payload per rank)
// and two readiness barriers for the untagged encodings.  Payload per slab:
// bf16 2E; INT8 g128 E + 4E/128; INT4 g32 E/2 + 8E/32; the tagged encodings
// carry 12 payload bytes in every 16.
double estimate_us(int f, int64_t rows, int64_t hidden, int P, const fc_link_model* link) {
  double t = table_us(kFusedUs, f, P, rows, hidden) + table_us(kSenderUs, f, P, rows, hidden);
  if (link) {
    const double E = static_cast<double>(rows) * static_cast<double>(hidden);
    const double base = f < 2 ? 2 * E : f < 4 ? E + 4 * E / 128 : E / 2 + 8 * E / 32;
    const double payload = kCands[f].tagged ? base * 16 / 12 : base;
    t += 2.0 * (P - 1) / P * payload / (link->link_gbps * 1e3);
    if (!kCands[f].tagged) t += 2.0 * link->barrier_us;
  }
  return t;
}

}  // namespace

extern "C" {

const char* fc_status_string(fc_status s) {
  switch (s) {
    case FC_OK: return "FC_OK";
    case FC_ERR_INVALID: return "FC_ERR_INVALID";
    case FC_ERR_CUDA: return "FC_ERR_CUDA";
    case FC_ERR_STALE_BLOCK: return "FC_ERR_STALE_BLOCK";
    case FC_ERR_UNSUPPORTED: return "FC_ERR_UNSUPPORTED";
  }
  return "FC_ERR_UNKNOWN";
}

const char* fc_last_error(void) { return g_msg; }

const char* fc_version(void) { return "libfcomm 0.1 sm_103a"; }

size_t fc_tagged_bytes(int64_t rows, int64_t hidden) {
  if (rows < 0 || hidden <= 0) return 0;
  return static_cast<size_t>(rows) * static_cast<size_t>((hidden + 5) / 6) * 16u;
}

size_t fc_codes_bytes(fc_qspec spec, int64_t rows, int64_t hidden) {
  if (rows < 0 || hidden <= 0) return 0;
  const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(hidden);
  switch (spec.fmt) {
    case FC_FMT_BF16: return 2 * n;
    case FC_FMT_INT8_SYM: return n;
    case FC_FMT_INT4_ASYM: return n / 2;
    case FC_FMT_BF16_TAGGED: return fc_tagged_bytes(rows, hidden);
    case FC_FMT_INT8_TAGGED: return n / 128 * 11 * 16;
    case FC_FMT_INT4_TAGGED: return n / 32 * 2 * 16;
    default: return 0;
  }
}

size_t fc_groups(fc_qspec spec, int64_t rows, int64_t hidden) {
  if (!(quantized(spec.fmt) || qtagged(spec.fmt)) || spec.group <= 0 || rows < 0 || hidden <= 0)
    return 0;
  return static_cast<size_t>(rows) * static_cast<size_t>(hidden) / static_cast<size_t>(spec.group);
}

fc_status fc_shard_range(fc_qspec spec, int64_t rows, int64_t hidden, int P, int shard,
                         int64_t* g0, int64_t* g1) {
  if (fc_status s = check_shape(spec, rows, hidden, true)) return s;
  if (P < 1 || shard < 0 || shard >= P || !g0 || !g1)
    return fail(FC_ERR_INVALID, "need 0 <= shard < P and non-NULL outputs");
  const int64_t ng = rows * hidden / spec.group;
  const int64_t per = (ng + P - 1) / P;
  int64_t a = per * shard, b = a + per;
  if (a > ng) a = ng;
  if (b > ng) b = ng;
  *g0 = a;
  *g1 = b;
  return ok();
}

// {FC_OK, 0x7F7F7F7F} into an optional two-word device status, ordered before
// the call's kernel on its stream (a one-thread kernel, so the launches of a
// stream still overlap one another's prologue and tail).
fc_status reset_status(int32_t* d_status, cudaStream_t st) {
  if (!d_status) return ok();
  if (!aligned(d_status, 4)) return fail(FC_ERR_INVALID, "d_status must be 4-byte aligned");
  return cuda_status(fc::launch_reset_status(d_status, st), "d_status reset");
}

fc_status fc_group_quantize_multi(const void* const* x_bf16, int P, int64_t rows, int64_t hidden,
                                  fc_qspec spec, const fc_qtensor* out, int32_t* d_status,
                                  fc_stream_t stream) {
  if (fc_status s = check_shape(spec, rows, hidden, true)) return s;
  if (P < 1 || P > 8) return fail(FC_ERR_INVALID, "P must be in [1, 8] (got %d)", P);
  if (rows == 0) return ok();
  if (!x_bf16 || !out) return fail(FC_ERR_INVALID, "x_bf16 and out must not be NULL");
  fc::QuantJob job{};
  for (int p = 0; p < P; ++p) {
    if (fc_status s = check_ptr(x_bf16[p], 32, "x_bf16[p]")) return s;
    if (fc_status s = check_qtensor(out[p], spec.fmt, "out[p]")) return s;
    job.x[p] = x_bf16[p];
    job.codes[p] = out[p].codes;
    job.scales[p] = out[p].scales;
    job.zeros[p] = out[p].zeros;
  }
  job.n = rows * hidden;
  job.P = P;
  job.G = spec.group;
  job.status = d_status;
  if (fc_status s = reset_status(d_status, (cudaStream_t)stream)) return s;
  return cuda_status(fc::launch_quantize(spec.fmt, false, fc::kDeqNone, job, (cudaStream_t)stream),
                     "fc_group_quantize launch");
}

fc_status fc_group_quantize_tagged(const void* const* x_bf16, int P, int64_t rows,
                                   int64_t hidden, fc_qspec spec, uint32_t epoch,
                                   void* const* blocks, int32_t* d_status, fc_stream_t stream) {
  if (!qtagged(spec.fmt))
    return fail(FC_ERR_INVALID, "format %d is not a tagged quantized format", spec.fmt);
  if (fc_status s = check_shape(spec, rows, hidden, false)) return s;
  if (P < 1 || P > 8) return fail(FC_ERR_INVALID, "P must be in [1, 8] (got %d)", P);
  if (rows == 0) return ok();
  if (!x_bf16 || !blocks) return fail(FC_ERR_INVALID, "x_bf16 and blocks must not be NULL");
  fc::QuantJob job{};
  for (int p = 0; p < P; ++p) {
    if (fc_status s = check_ptr(x_bf16[p], 32, "x_bf16[p]")) return s;
    if (fc_status s = check_ptr(blocks[p], 16, "blocks[p]")) return s;
    job.x[p] = x_bf16[p];
    job.codes[p] = blocks[p];
  }
  job.n = rows * hidden;
  job.P = P;
  job.G = spec.group;
  job.epoch = epoch;
  job.status = d_status;
  if (fc_status s = reset_status(d_status, (cudaStream_t)stream)) return s;
  return cuda_status(fc::launch_quantize_tagged(spec.fmt, job, (cudaStream_t)stream),
                     "fc_group_quantize_tagged launch");
}

fc_status fc_group_quantize(const void* x_bf16, int64_t rows, int64_t hidden, fc_qspec spec,
                            fc_qtensor out, int32_t* d_status, fc_stream_t stream) {
  return fc_group_quantize_multi(&x_bf16, 1, rows, hidden, spec, &out, d_status, stream);
}

fc_status fc_reduce_dequant_sum(const fc_qtensor* slabs, int P, int64_t rows, int64_t hidden,
                                fc_qspec spec, int shard, float* out_f32, fc_stream_t stream) {
  if (fc_status s = check_shape(spec, rows, hidden, true)) return s;
  if (P < 2 || P > 8) return fail(FC_ERR_INVALID, "P must be in [2, 8] (got %d)", P);
  if (shard < -1 || shard >= P)
    return fail(FC_ERR_INVALID, "shard must be -1 or in [0, P) (got %d)", shard);
  if (rows == 0) return ok();
  if (!slabs) return fail(FC_ERR_INVALID, "slabs must not be NULL");
  if (fc_status s = check_ptr(out_f32, 32, "out_f32")) return s;
  fc::Slabs sl{};
  for (int p = 0; p < P; ++p) {
    if (fc_status s = check_qtensor(slabs[p], spec.fmt, "slabs[p]")) return s;
    sl.codes[p] = slabs[p].codes;
    sl.scales[p] = slabs[p].scales;
    sl.zeros[p] = slabs[p].zeros;
  }
  const int64_t lpg = spec.group / 16;
  int64_t c0 = 0, c1 = rows * hidden / 16;
  if (shard >= 0) {
    int64_t g0, g1;
    fc_shard_range(spec, rows, hidden, P, shard, &g0, &g1);
    c0 = g0 * lpg;
    c1 = g1 * lpg;
  }
  return cuda_status(fc::launch_reduce(spec.fmt, sl, P, spec.group, c0, c1, out_f32,
                                       (cudaStream_t)stream),
                     "fc_reduce_dequant_sum launch");
}

fc_status fc_requant_gather(const float* reduced_f32, int64_t rows, int64_t hidden, fc_qspec spec,
                            fc_qtensor requant_out, void* out, int32_t out_dtype,
                            fc_stream_t stream) {
  if (fc_status s = check_shape(spec, rows, hidden, true)) return s;
  if (rows == 0) return ok();
  if (fc_status s = check_ptr(reduced_f32, 32, "reduced_f32")) return s;
  if (requant_out.codes)
    if (fc_status s = check_qtensor(requant_out, spec.fmt, "requant_out")) return s;
  int deq = fc::kDeqNone;
  if (out) {
    if (out_dtype != FC_FMT_BF16 && out_dtype != FC_FMT_F32)
      return fail(FC_ERR_INVALID, "out_dtype must be FC_FMT_BF16 or FC_FMT_F32");
    if (fc_status s = check_ptr(out, 32, "out")) return s;
    deq = out_dtype == FC_FMT_BF16 ? fc::kDeqBF16 : fc::kDeqF32;
  }
  fc::QuantJob job{};
  job.x[0] = reduced_f32;
  job.codes[0] = requant_out.codes;
  job.scales[0] = requant_out.scales;
  job.zeros[0] = requant_out.zeros;
  job.deq = out;
  job.n = rows * hidden;
  job.P = 1;
  job.G = spec.group;
  return cuda_status(fc::launch_quantize(spec.fmt, true, deq, job, (cudaStream_t)stream),
                     "fc_requant_gather launch");
}

fc_status fc_allgather_dequant(const fc_qtensor* shards, int P, int64_t rows, int64_t hidden,
                               fc_qspec spec, int32_t out_dtype, void* out, uint32_t expected_epoch,
                               int32_t* d_status, fc_stream_t stream) {
  if (fc_status s = check_shape(spec, rows, hidden, false)) return s;
  if (!quantized(spec.fmt) && !qtagged(spec.fmt))
    return fail(FC_ERR_INVALID, "format %d is not a quantized format", spec.fmt);
  if (P < 1 || P > 8) return fail(FC_ERR_INVALID, "P must be in [1, 8] (got %d)", P);
  if (out_dtype != FC_FMT_BF16 && out_dtype != FC_FMT_F32)
    return fail(FC_ERR_INVALID, "out_dtype must be FC_FMT_BF16 or FC_FMT_F32");
  if (rows == 0) return ok();
  if (!shards) return fail(FC_ERR_INVALID, "shards must not be NULL");
  if (fc_status s = check_ptr(out, 32, "out")) return s;
  if (d_status && !aligned(d_status, 4)) return fail(FC_ERR_INVALID, "d_status must be 4-byte aligned");
  const bool tagged = qtagged(spec.fmt);
  const int G = spec.group, lpg = G / 16;
  const int nbg = spec.fmt == FC_FMT_INT8_TAGGED ? fc::kBlocksPerGroupI8 : fc::kBlocksPerGroupI4;
  const int64_t ng = rows * hidden / G, per = (ng + P - 1) / P;
  fc::GatherJob j{};
  int64_t blk = 0;
  for (int p = 0; p < P; ++p) {
    const int64_t g0 = std::min<int64_t>(p * per, ng), g1 = std::min<int64_t>(g0 + per, ng);
    j.first[p] = g0 * lpg;
    j.blk0[p] = blk;
    if (g1 > g0) {  // an empty shard needs no buffers
      const size_t calign = tagged || spec.fmt == FC_FMT_INT8_SYM ? 16 : 8;
      if (fc_status s = check_ptr(shards[p].codes, calign, "shards[p].codes")) return s;
      if (!tagged) {
        if (fc_status s = check_ptr(shards[p].scales, 4, "shards[p].scales")) return s;
        if (spec.fmt == FC_FMT_INT4_ASYM)
          if (fc_status s = check_ptr(shards[p].zeros, 4, "shards[p].zeros")) return s;
      }
      if (tagged) blk += (g1 - g0) * nbg;
    }
    j.codes[p] = shards[p].codes;
    j.scales[p] = shards[p].scales;
    j.zeros[p] = shards[p].zeros;
  }
  j.first[P] = ng * lpg;
  j.chunks = ng * lpg;
  j.P = P;
  j.lpg_shift = 0;
  while ((1 << j.lpg_shift) < lpg) ++j.lpg_shift;
  j.out = out;
  j.epoch = expected_epoch;
  cudaStream_t st = (cudaStream_t)stream;
  j.status = d_status;
  if (fc_status s = reset_status(d_status, st)) return s;
  return cuda_status(fc::launch_allgather(spec.fmt, out_dtype == FC_FMT_F32, j, st),
                     "fc_allgather_dequant launch");
}

fc_status fc_pack_tagged_multi(const void* const* x_bf16, int P, int64_t rows, int64_t hidden,
                               uint32_t epoch, void* const* blocks, fc_stream_t stream) {
  fc_qspec spec{FC_FMT_BF16_TAGGED, 0};
  if (fc_status s = check_shape(spec, rows, hidden, false)) return s;
  if (P < 1 || P > 8) return fail(FC_ERR_INVALID, "P must be in [1, 8] (got %d)", P);
  if (rows == 0) return ok();
  if (!x_bf16 || !blocks) return fail(FC_ERR_INVALID, "x_bf16 and blocks must not be NULL");
  for (int p = 0; p < P; ++p) {
    if (fc_status s = check_ptr(x_bf16[p], 32, "x_bf16[p]")) return s;
    if (fc_status s = check_ptr(blocks[p], 16, "blocks[p]")) return s;
  }
  return cuda_status(fc::launch_pack_tagged(x_bf16, blocks, P, rows, static_cast<int>(hidden),
                                            epoch, (cudaStream_t)stream),
                     "fc_pack_tagged launch");
}

fc_status fc_pack_tagged(const void* x_bf16, int64_t rows, int64_t hidden, uint32_t epoch,
                         void* blocks, fc_stream_t stream) {
  return fc_pack_tagged_multi(&x_bf16, 1, rows, hidden, epoch, &blocks, stream);
}

fc_status fc_allreduce_residual_rmsnorm_ex(const fc_qtensor* slabs, int P, int64_t rows,
                                           int64_t hidden, fc_qspec spec,
                                           const void* residual_in, void* residual_out,
                                           const void* gamma, float eps, fc_qtensor requant_out,
                                           void* y, uint32_t expected_epoch, int32_t* d_status,
                                           const fc_launch_opts* opts, fc_stream_t stream) {
  if (fc_status s = check_shape(spec, rows, hidden, false)) return s;
  if (P < 2 || P > 8) return fail(FC_ERR_INVALID, "P must be in [2, 8] (got %d)", P);
  if (opts && opts->max_ctas < 0) return fail(FC_ERR_INVALID, "max_ctas must be >= 0");
  if (opts && (opts->kernel < 0 || opts->kernel > 2))
    return fail(FC_ERR_INVALID, "kernel must be 0 (auto), 1 (streaming) or 2 (TMA-staged)");
  if (rows == 0) return ok();
  if (!slabs) return fail(FC_ERR_INVALID, "slabs must not be NULL");
  if (!(eps >= 0.0f) || eps > 1.0f) return fail(FC_ERR_INVALID, "eps must be in [0, 1]");
  if (fc_status s = check_ptr(residual_in, 32, "residual_in")) return s;
  if (fc_status s = check_ptr(residual_out, 32, "residual_out")) return s;
  if (fc_status s = check_ptr(gamma, 32, "gamma")) return s;
  if (fc_status s = check_ptr(y, 32, "y")) return s;
  if (opts && opts->max_ctas < 0) return fail(FC_ERR_INVALID, "max_ctas must be >= 0");
  fc::FusedArgs a{};
  for (int p = 0; p < P; ++p) {
    if (fc_status s = check_qtensor(slabs[p], spec.fmt, "slabs[p]")) return s;
    a.s.codes[p] = slabs[p].codes;
    a.s.scales[p] = slabs[p].scales;
    a.s.zeros[p] = slabs[p].zeros;
  }
  if ((quantized(spec.fmt) || qtagged(spec.fmt)) && requant_out.codes) {
    if (fc_status s = check_qtensor(requant_out, base_fmt(spec.fmt), "requant_out")) return s;
    a.rq_codes = requant_out.codes;
    a.rq_scales = requant_out.scales;
    a.rq_zeros = requant_out.zeros;
  }
  if (d_status && !aligned(d_status, 4)) return fail(FC_ERR_INVALID, "d_status must be 4-byte aligned");
  a.res_in = residual_in;
  a.res_out = residual_out;
  a.gamma = gamma;
  a.y = y;
  a.rows = rows;
  a.H = static_cast<int>(hidden);
  a.G = (quantized(spec.fmt) || qtagged(spec.fmt)) ? spec.group : 16;
  a.lpg_shift = 0;
  while ((16 << a.lpg_shift) < a.G) ++a.lpg_shift;
  a.P = P;
  a.eps = eps;
  a.epoch = expected_epoch;
  cudaStream_t st = (cudaStream_t)stream;
  a.status = d_status;
  if (fc_status s = reset_status(d_status, st)) return s;
  const int path = opts ? opts->kernel : 0;
  const cudaError_t e = fc::launch_fused(spec.fmt, a, opts ? opts->max_ctas : 0, path, st);
  if (e == cudaErrorNotSupported)
    return fail(FC_ERR_UNSUPPORTED,
                "the TMA-staged kernel (the only one for tagged quantized formats) does not support "
                "this shape/alignment");
  return cuda_status(e, "fc_allreduce_residual_rmsnorm launch");
}

fc_status fc_allreduce_residual_rmsnorm(const fc_qtensor* slabs, int P, int64_t rows,
                                        int64_t hidden, fc_qspec spec, const void* residual_in,
                                        void* residual_out, const void* gamma, float eps,
                                        fc_qtensor requant_out, void* y, uint32_t expected_epoch,
                                        int32_t* d_status, fc_stream_t stream) {
  return fc_allreduce_residual_rmsnorm_ex(slabs, P, rows, hidden, spec, residual_in, residual_out,
                                          gamma, eps, requant_out, y, expected_epoch, d_status,
                                          nullptr, stream);
}

fc_status fc_token_split(int P, int64_t rows, int64_t hidden, fc_qspec spec, int64_t* split,
                         int64_t* wave_rows) {
  if (fc_status s = check_shape(spec, rows, hidden, false)) return s;
  if (P < 2 || P > 8) return fail(FC_ERR_INVALID, "P must be in [2, 8] (got %d)", P);
  if (!split) return fail(FC_ERR_INVALID, "split must not be NULL");
  fc::FusedArgs a{};
  a.P = P;
  a.H = static_cast<int>(hidden);
  a.G = (quantized(spec.fmt) || qtagged(spec.fmt)) ? spec.group : 16;
  a.rows = rows;
  // shape-only query: the kernel choice assumes 16-byte aligned tensors
  static const uint4 aligned_probe[1] = {};
  for (int p = 0; p < P; ++p) {
    a.s.codes[p] = aligned_probe;
    a.s.scales[p] = reinterpret_cast<const float*>(aligned_probe);
    a.s.zeros[p] = reinterpret_cast<const float*>(aligned_probe);
  }
  a.res_in = a.gamma = aligned_probe;
  const int64_t w = fc::fused_wave_rows(spec.fmt, a);
  if (w <= 0) return fail(FC_ERR_CUDA, "could not query the fused kernel's occupancy");
  if (wave_rows) *wave_rows = w;
  int64_t s = rows / 2;
  if (rows > w) {
    // the whole-wave split nearest the middle: the first subset fills whole
    // waves and the pair needs no more waves than one unsplit call
    const int64_t k = (rows / 2 + w / 2) / w;
    const int64_t cand = (k < 1 ? 1 : k) * w;
    if (cand < rows) s = cand;
  }
  *split = s;
  return ok();
}

fc_status fc_protocol_estimate(int64_t rows, int64_t hidden, int P, fc_qspec spec,
                               const fc_link_model* link, double* est_us) {
  if (rows <= 0 || hidden <= 0 || hidden % 128 != 0)
    return fail(FC_ERR_INVALID, "need rows > 0 and hidden a positive multiple of 128");
  if (P < 2 || P > 8) return fail(FC_ERR_INVALID, "P must be in [2, 8] (got %d)", P);
  if (!est_us) return fail(FC_ERR_INVALID, "est_us must not be NULL");
  if (link && (!(link->link_gbps > 0.0) || !(link->barrier_us >= 0.0)))
    return fail(FC_ERR_INVALID, "link_gbps must be > 0 and barrier_us >= 0");
  int f = -1;
  switch (spec.fmt) {
    case FC_FMT_BF16: f = 0; break;
    case FC_FMT_BF16_TAGGED: f = 1; break;
    case FC_FMT_INT8_SYM: f = spec.group == 128 ? 2 : -1; break;
    case FC_FMT_INT8_TAGGED: f = spec.group == 128 ? 3 : -1; break;
    case FC_FMT_INT4_ASYM: f = spec.group == 32 ? 4 : -1; break;
    case FC_FMT_INT4_TAGGED: f = spec.group == 32 ? 5 : -1; break;
    default: break;
  }
  if (f < 0) return fail(FC_ERR_UNSUPPORTED, "no measured rates for format %d group %d", spec.fmt, spec.group);
  *est_us = estimate_us(f, rows, hidden, P, link);
  return ok();
}

fc_status fc_select_protocol(int64_t rows, int64_t hidden, int P, int min_bits,
                             const fc_link_model* link, fc_qspec* choice, double* est_us) {
  if (rows <= 0 || hidden <= 0 || hidden % 128 != 0)
    return fail(FC_ERR_INVALID, "need rows > 0 and hidden a positive multiple of 128");
  if (P < 2 || P > 8) return fail(FC_ERR_INVALID, "P must be in [2, 8] (got %d)", P);
  if (min_bits != 4 && min_bits != 8 && min_bits != 16)
    return fail(FC_ERR_INVALID, "min_bits must be 4, 8 or 16 (got %d)", min_bits);
  if (!choice) return fail(FC_ERR_INVALID, "choice must not be NULL");
  if (link && (!(link->link_gbps > 0.0) || !(link->barrier_us >= 0.0)))
    return fail(FC_ERR_INVALID, "link_gbps must be > 0 and barrier_us >= 0");
  double best = 1e300;
  int pick = -1;
  for (int i = 0; i < 6; ++i) {
    if (kCands[i].bits < min_bits) continue;
    const double t = estimate_us(i, rows, hidden, P, link);
    if (t < best) best = t, pick = i;
  }
  choice->fmt = kCands[pick].fmt;
  choice->group = kCands[pick].group;
  if (est_us) *est_us = best;
  return ok();
}

}  // extern "C"
