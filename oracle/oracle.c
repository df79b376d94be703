/*
 * oracle.c -- plain CPU oracle (TEST INFRASTRUCTURE ONLY; see oracle.h).
 *
 * Written from the definitions of the method, one step per function, in
 * plain scalar loops.  No blocking, fusion or reordering: each element is
 * visited in index order, each slab in slab order.  Build with
 *   gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 * so that every float expression below is exactly one binary32 operation
 * rounded to nearest-even (no fused multiply-add, no excess precision).
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 -- */

float or_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* bf16 keeps the top 16 bits of a binary32; round to nearest, ties to the
 * even 16-bit result.  Inputs here are finite (NaN is out of contract). */
uint16_t or_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* binary64 -> bf16 with a single rounding: first to binary32 rounding to
 * odd (sticky last bit), then to bf16 to nearest-even.  Rounding to odd at
 * a precision at least two bits wider than the target makes the second
 * rounding equal to one direct rounding (Boldo and Melquiond, "Emulation of
 * FMA and correctly rounded sums: proved algorithms using rounding to odd",
 * IEEE Trans. Computers 2008). */
uint16_t or_f64_to_bf16(double d) {
  float f = (float)d;
  if ((double)f != d) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 1u) == 0u) {
      if (fabs((double)f) < fabs(d))
        u += 1u; /* step away from zero, toward d */
      else
        u -= 1u; /* step toward zero, toward d */
      memcpy(&f, &u, 4);
    }
  }
  return or_f32_to_bf16(f);
}

void or_bf16_to_f32_array(const uint16_t* b, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = or_bf16_to_f32(b[i]);
}

void or_f32_to_bf16_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = or_f32_to_bf16(x[i]);
}

/* ---------------------------------------------------------- quantizers -- */
/* [FC] "Main contributions" 2: activations are quantized to low bit-width
 * in fine-grained groups before they are communicated.  Formats: INT8
 * symmetric with one fp32 scale per group of G, and INT4 asymmetric with an
 * fp32 scale and an fp32 offset (the group minimum) per group of G. */

/* INT8 symmetric: s = max|x| / 127, q = clamp(rne(x / s), -127, 127).
 * A group whose scale is zero (all zeros) gets s = 0 and codes 0. */
void or_quant_i8s(const float* x, int64_t n, int G, int8_t* q, float* s) {
  int64_t ng = n / G;
  for (int64_t g = 0; g < ng; ++g) {
    const float* xg = x + g * G;
    float a = 0.0f;
    for (int k = 0; k < G; ++k) {
      float v = fabsf(xg[k]);
      if (v > a) a = v;
    }
    float sc = a / 127.0f;
    s[g] = sc;
    for (int k = 0; k < G; ++k) {
      int code = 0;
      if (sc != 0.0f) {
        float t = xg[k] / sc;
        float r = nearbyintf(t); /* default rounding mode: nearest, ties to even */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        code = (int)r;
      }
      q[g * G + k] = (int8_t)code;
    }
  }
}

void or_dequant_i8s(const int8_t* q, const float* s, int64_t n, int G, float* d) {
  for (int64_t i = 0; i < n; ++i) d[i] = (float)q[i] * s[i / G];
}

/* INT4 asymmetric: lo = min x, hi = max x (a zero extreme is taken as +0),
 * s = (hi - lo) / 15, z = lo, q = clamp(rne((x - lo) / s), 0, 15).
 * Codes are packed two per byte: element 2i in the low nibble of byte i,
 * element 2i+1 in the high nibble. */
void or_quant_i4a(const float* x, int64_t n, int G, uint8_t* packed, float* s, float* z) {
  int64_t ng = n / G;
  for (int64_t i = 0; i < n / 2; ++i) packed[i] = 0;
  for (int64_t g = 0; g < ng; ++g) {
    const float* xg = x + g * G;
    float lo = xg[0], hi = xg[0];
    for (int k = 1; k < G; ++k) {
      if (xg[k] < lo) lo = xg[k];
      if (xg[k] > hi) hi = xg[k];
    }
    if (lo == 0.0f) lo = 0.0f; /* -0 -> +0 */
    if (hi == 0.0f) hi = 0.0f;
    float sc = (hi - lo) / 15.0f;
    s[g] = sc;
    z[g] = lo;
    for (int k = 0; k < G; ++k) {
      int code = 0;
      if (sc != 0.0f) {
        float t = (xg[k] - lo) / sc;
        float r = nearbyintf(t);
        if (r > 15.0f) r = 15.0f;
        if (r < 0.0f) r = 0.0f;
        code = (int)r;
      }
      int64_t e = g * G + k;
      packed[e / 2] |= (uint8_t)(code << ((e & 1) ? 4 : 0));
    }
  }
}

static float deq_i4_one(const uint8_t* packed, const float* s, const float* z, int64_t e, int G) {
  int code = (packed[e / 2] >> ((e & 1) ? 4 : 0)) & 0xF;
  float m = (float)code * s[e / G];
  return m + z[e / G]; /* two roundings: multiply, then add */
}

void or_dequant_i4a(const uint8_t* packed, const float* s, const float* z, int64_t n, int G,
                    float* d) {
  for (int64_t i = 0; i < n; ++i) d[i] = deq_i4_one(packed, s, z, i, G);
}

/* ------------------------------------------------------- fixed-order sum -- */
/* [FL] abstract: the reduction order is decoupled from the order in which
 * data arrives, so the result is the same on every GPU.  Reading: the sum
 * always runs over slabs 0, 1, ..., P-1 from an fp32 zero. */
void or_reduce_sum(const float* const* d, int P, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) {
    float acc = 0.0f;
    for (int p = 0; p < P; ++p) acc = acc + d[p][i];
    out[i] = acc;
  }
}

/* ------------------------------------------------------ two-step reduce -- */
/* [FC] "Main contributions" 2 / "Core ideas": the All-Reduce runs in two
 * steps.  Step 1 (reduce-scatter): the owner of shard j dequantizes shard j
 * of every slab, sums it, and requantizes the sum.  Step 2 (all-gather):
 * every rank receives all requantized shards and dequantizes them. */
static float deq_one(int fmt, const void* codes, const float* s, const float* z, int64_t e,
                     int G) {
  if (fmt == OR_FMT_INT8_SYM) return (float)((const int8_t*)codes)[e] * s[e / G];
  return deq_i4_one((const uint8_t*)codes, s, z, e, G);
}

int or_two_step(int fmt, const void* const* codes, const float* const* scales,
                const float* const* zeros, int P, int64_t n, int G, int shards, float* reduced,
                void* rq_codes, float* rq_scales, float* rq_zeros, float* gathered) {
  if (fmt != OR_FMT_INT8_SYM && fmt != OR_FMT_INT4_ASYM) return -1;
  if (P < 1 || G < 1 || n < 0 || n % G != 0 || shards < 1) return -1;
  if (fmt == OR_FMT_INT4_ASYM && (G % 2) != 0) return -1;
  int64_t ng = n / G;
  float* red = reduced ? reduced : (float*)malloc(sizeof(float) * (size_t)(n ? n : 1));
  size_t cbytes = fmt == OR_FMT_INT8_SYM ? (size_t)n : (size_t)(n / 2);
  void* rc = rq_codes ? rq_codes : malloc(cbytes ? cbytes : 1);
  float* rs = rq_scales ? rq_scales : (float*)malloc(sizeof(float) * (size_t)(ng ? ng : 1));
  float* rz = rq_zeros ? rq_zeros : (float*)malloc(sizeof(float) * (size_t)(ng ? ng : 1));
  int64_t per = (ng + shards - 1) / shards;

  /* step 1: every shard owner reduces and requantizes its own shard */
  for (int j = 0; j < shards; ++j) {
    int64_t g0 = (int64_t)j * per, g1 = g0 + per;
    if (g1 > ng) g1 = ng;
    if (g0 >= g1) continue;
    int64_t e0 = g0 * G, e1 = g1 * G;
    for (int64_t e = e0; e < e1; ++e) {
      float acc = 0.0f;
      for (int p = 0; p < P; ++p)
        acc = acc + deq_one(fmt, codes[p], scales[p], zeros ? zeros[p] : NULL, e, G);
      red[e] = acc;
    }
    if (fmt == OR_FMT_INT8_SYM)
      or_quant_i8s(red + e0, e1 - e0, G, (int8_t*)rc + e0, rs + g0);
    else
      or_quant_i4a(red + e0, e1 - e0, G, (uint8_t*)rc + e0 / 2, rs + g0, rz + g0);
  }
  /* step 2: gather every requantized shard and dequantize it */
  if (gathered)
    for (int64_t e = 0; e < n; ++e) gathered[e] = deq_one(fmt, rc, rs, rz, e, G);

  if (!reduced) free(red);
  if (!rq_codes) free(rc);
  if (!rq_scales) free(rs);
  if (!rq_zeros) free(rz);
  return 0;
}

/* ------------------------------------------------- standalone all-gather -- */
/* [FL] abstract (the all-gather collective) and [FC] "Core ideas" (its
 * second step): each of P ranks holds the quantized payload of one shard --
 * the contiguous groups [j*per, min((j+1)*per, n_g)), per = ceil(n_g/P), the
 * same partition as the reduce-scatter -- indexed from the shard's own first
 * group.  Every rank receives all shards and dequantizes them. */
int or_allgather_dequant(int fmt, const void* const* codes, const float* const* scales,
                         const float* const* zeros, int P, int64_t n, int G, float* out) {
  if (fmt != OR_FMT_INT8_SYM && fmt != OR_FMT_INT4_ASYM) return -1;
  if (P < 1 || G < 1 || n < 0 || n % G != 0) return -1;
  if (fmt == OR_FMT_INT4_ASYM && (G % 2) != 0) return -1;
  int64_t ng = n / G;
  int64_t per = (ng + P - 1) / P;
  for (int j = 0; j < P; ++j) {
    int64_t g0 = (int64_t)j * per, g1 = g0 + per;
    if (g1 > ng) g1 = ng;
    if (g0 >= g1) continue; /* an empty shard */
    int64_t local_n = (g1 - g0) * G;
    for (int64_t e = 0; e < local_n; ++e)
      out[g0 * G + e] = deq_one(fmt, codes[j], scales[j], zeros ? zeros[j] : NULL, e, G);
  }
  return 0;
}

/* ------------------------------------------------ residual add, RMSNorm -- */
/* [TW] abstract: the RMSNorm that follows each tensor-parallel All-Reduce is
 * fused into it.  h = bf16(o + R) is the new residual stream (the sum is the
 * fp32 accumulator's precision); RMSNorm normalizes that bf16 h:
 *   y_k = h_k / sqrt((1/H) sum_k h_k^2 + eps) * gamma_k. */
void or_residual_rmsnorm(const float* o, const uint16_t* r, const uint16_t* gamma, int64_t T,
                         int64_t H, float eps, uint16_t* h_out, uint16_t* y_out) {
  for (int64_t t = 0; t < T; ++t) {
    const float* ot = o + t * H;
    const uint16_t* rt = r + t * H;
    uint16_t* ht = h_out + t * H;
    for (int64_t k = 0; k < H; ++k) {
      float hf = ot[k] + or_bf16_to_f32(rt[k]);
      ht[k] = or_f32_to_bf16(hf);
    }
    double ss = 0.0;
    for (int64_t k = 0; k < H; ++k) {
      double v = (double)or_bf16_to_f32(ht[k]);
      ss = ss + v * v;
    }
    double inv = 1.0 / sqrt(ss / (double)H + (double)eps);
    for (int64_t k = 0; k < H; ++k) {
      double v = (double)or_bf16_to_f32(ht[k]);
      double g = (double)or_bf16_to_f32(gamma[k]);
      y_out[t * H + k] = or_f64_to_bf16((v * inv) * g);
    }
  }
}

/* ------------------------------------------------------ tagged blocks --- */
/* [FL] abstract: each data block carries evidence of its own readiness and
 * the receiver validates the blocks it needs directly.  Reading: a 16-byte
 * block carries 6 bf16 values and a 32-bit epoch, so payload and tag arrive
 * in one 16-byte access; blocks never straddle token rows. */
int64_t or_tagged_blocks_per_row(int64_t H) { return (H + 5) / 6; }

void or_pack_tagged(const uint16_t* x, int64_t T, int64_t H, uint32_t epoch, uint32_t* blocks) {
  int64_t nb = or_tagged_blocks_per_row(H);
  for (int64_t t = 0; t < T; ++t)
    for (int64_t j = 0; j < nb; ++j) {
      uint32_t* w = blocks + 4 * (t * nb + j);
      for (int k = 0; k < 3; ++k) {
        int64_t e0 = 6 * j + 2 * k, e1 = e0 + 1;
        uint32_t lo = e0 < H ? x[t * H + e0] : 0u;
        uint32_t hi = e1 < H ? x[t * H + e1] : 0u;
        w[k] = lo | (hi << 16);
      }
      w[3] = epoch;
    }
}

int64_t or_validate_tagged(const uint32_t* blocks, int64_t nblocks, uint32_t epoch) {
  for (int64_t b = 0; b < nblocks; ++b)
    if (blocks[4 * b + 3] != epoch) return b;
  return -1;
}

void or_unpack_tagged(const uint32_t* blocks, int64_t T, int64_t H, uint16_t* x) {
  int64_t nb = or_tagged_blocks_per_row(H);
  for (int64_t t = 0; t < T; ++t)
    for (int64_t e = 0; e < H; ++e) {
      const uint32_t* w = blocks + 4 * (t * nb + e / 6);
      int64_t k = (e % 6) / 2;
      x[t * H + e] = (uint16_t)((e % 2) ? (w[k] >> 16) : (w[k] & 0xFFFFu));
    }
}

/* --------------------------------------------- tagged quantized payloads -- */
/* [FL] abstract (readiness evidence in every block) applied to [FC]'s
 * quantized groups: the payload a rank sends for one group is carried by
 * ceil(payload/12) self-validating 16-byte blocks. */
static int qt_payload_bytes(int fmt, int G) {
  return fmt == OR_FMT_INT8_SYM ? G + 4 : G / 2 + 8;
}

int or_qtagged_blocks_per_group(int fmt, int G) { return (qt_payload_bytes(fmt, G) + 11) / 12; }

void or_pack_qtagged(int fmt, const void* codes, const float* scales, const float* zeros,
                     int64_t n, int G, uint32_t epoch, uint32_t* blocks) {
  int64_t ng = n / G;
  int nbg = or_qtagged_blocks_per_group(fmt, G);
  int cb = fmt == OR_FMT_INT8_SYM ? G : G / 2;
  uint8_t payload[12 * 64];
  for (int64_t g = 0; g < ng; ++g) {
    memset(payload, 0, sizeof payload);
    memcpy(payload, (const uint8_t*)codes + g * cb, (size_t)cb);
    memcpy(payload + cb, &scales[g], 4);
    if (fmt == OR_FMT_INT4_ASYM) memcpy(payload + cb + 4, &zeros[g], 4);
    for (int b = 0; b < nbg; ++b) {
      uint32_t* w = blocks + 4 * (g * nbg + b);
      memcpy(w, payload + 12 * b, 12);
      w[3] = epoch;
    }
  }
}

int64_t or_unpack_qtagged(int fmt, const uint32_t* blocks, int64_t n, int G, uint32_t epoch,
                          void* codes, float* scales, float* zeros) {
  int64_t ng = n / G;
  int nbg = or_qtagged_blocks_per_group(fmt, G);
  int cb = fmt == OR_FMT_INT8_SYM ? G : G / 2;
  int64_t bad = -1;
  uint8_t payload[12 * 64];
  for (int64_t g = 0; g < ng; ++g) {
    for (int b = 0; b < nbg; ++b) {
      const uint32_t* w = blocks + 4 * (g * nbg + b);
      if (w[3] != epoch && bad < 0) bad = g * nbg + b;
      memcpy(payload + 12 * b, w, 12);
    }
    memcpy((uint8_t*)codes + g * cb, payload, (size_t)cb);
    memcpy(&scales[g], payload + cb, 4);
    if (fmt == OR_FMT_INT4_ASYM && zeros) memcpy(&zeros[g], payload + cb + 4, 4);
  }
  return bad;
}

/* --------------------------------------------------------- whole path --- */
int or_allreduce_residual_rmsnorm(int fmt, const uint16_t* const* slabs, int P, int64_t T,
                                  int64_t H, int G, const uint16_t* r, const uint16_t* gamma,
                                  float eps, void* rq_codes, float* rq_scales, float* rq_zeros,
                                  uint16_t* h_out, uint16_t* y_out) {
  int64_t n = T * H;
  if (P < 1 || T < 0 || H < 1) return -1;
  float* o = (float*)malloc(sizeof(float) * (size_t)(n ? n : 1));
  float* xf = (float*)malloc(sizeof(float) * (size_t)(n ? n : 1));
  int rc = 0;
  if (fmt == OR_FMT_BF16 || fmt == OR_FMT_BF16_TAGGED) {
    for (int64_t i = 0; i < n; ++i) o[i] = 0.0f;
    for (int p = 0; p < P; ++p) {
      or_bf16_to_f32_array(slabs[p], n, xf);
      for (int64_t i = 0; i < n; ++i) o[i] = o[i] + xf[i];
    }
  } else if (fmt == OR_FMT_INT8_SYM || fmt == OR_FMT_INT4_ASYM) {
    if (G < 1 || H % G != 0) {
      free(o);
      free(xf);
      return -1;
    }
    int64_t ng = n / G;
    void* codes[8];
    float* sc[8];
    float* zp[8];
    if (P > 8) {
      free(o);
      free(xf);
      return -1;
    }
    for (int p = 0; p < P; ++p) {
      codes[p] = malloc((size_t)(n ? n : 1));
      sc[p] = (float*)malloc(sizeof(float) * (size_t)(ng ? ng : 1));
      zp[p] = (float*)malloc(sizeof(float) * (size_t)(ng ? ng : 1));
      or_bf16_to_f32_array(slabs[p], n, xf);
      if (fmt == OR_FMT_INT8_SYM)
        or_quant_i8s(xf, n, G, (int8_t*)codes[p], sc[p]);
      else
        or_quant_i4a(xf, n, G, (uint8_t*)codes[p], sc[p], zp[p]);
    }
    rc = or_two_step(fmt, (const void* const*)codes, (const float* const*)sc,
                     (const float* const*)zp, P, n, G, P, NULL, rq_codes, rq_scales, rq_zeros, o);
    for (int p = 0; p < P; ++p) {
      free(codes[p]);
      free(sc[p]);
      free(zp[p]);
    }
  } else {
    rc = -1;
  }
  if (rc == 0) or_residual_rmsnorm(o, r, gamma, T, H, eps, h_out, y_out);
  free(o);
  free(xf);
  return rc;
}
