/*
 * oracle.h -- plain, slow, single-threaded CPU oracle for the quantized
 * reduce + residual-add + RMSNorm path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (libfcomm) never links, loads or calls it, and shares no source with it.
 *
 * Sources followed (pages, by title and section):
 *  [FC]  "Flash Communication: Reducing Tensor Parallelization Bottleneck for
 *        Fast Large Language Model Inference" (arXiv 2412.04964), summary,
 *        "Main contributions" item 2 and "Core ideas": low-bit fine-grained
 *        quantization of activations and a two-step All-Reduce.
 *  [FL]  flash-comm, abstract: self-synchronizing blocks that carry evidence
 *        of readiness; reduction order decoupled from transport order.
 *  [TW]  "TokenWeave: Efficient Compute-Communication Overlap for Distributed
 *        LLM Inference" (arXiv 2505.11329), abstract: RMSNorm fused after the
 *        All-Reduce; token splitting into two subsets.
 *
 * Precision: the quantizer, the dequantizer, the fixed-order sum and the
 * residual add are defined in binary32 (fp32 scales, fp32 accumulation): each
 * operation here is one IEEE-754 binary32 operation rounded to nearest-even,
 * compiled with -ffp-contract=off (no fused multiply-add).  RMSNorm, whose
 * output only has to agree to one bf16 ulp, is evaluated in binary64 and
 * rounded once to bf16.
 *
 * Parity pins: every function here is checked by the CPU tests against
 * closed forms, brute force, invariants or a library routine; none is
 * "parity unpinned".
 */
#ifndef QRR_ORACLE_H
#define QRR_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* formats (same numbering as the product's public header, restated here) */
#define OR_FMT_BF16 0
#define OR_FMT_INT8_SYM 1
#define OR_FMT_INT4_ASYM 2
#define OR_FMT_BF16_TAGGED 3

float or_bf16_to_f32(uint16_t b);
uint16_t or_f32_to_bf16(float f);   /* round to nearest even */
uint16_t or_f64_to_bf16(double d);  /* one rounding, to nearest even */
void or_bf16_to_f32_array(const uint16_t* b, int64_t n, float* out);
void or_f32_to_bf16_array(const float* x, int64_t n, uint16_t* out);

/* Group quantizers over n elements in groups of G consecutive elements. */
void or_quant_i8s(const float* x, int64_t n, int G, int8_t* q, float* s);
void or_dequant_i8s(const int8_t* q, const float* s, int64_t n, int G, float* d);
void or_quant_i4a(const float* x, int64_t n, int G, uint8_t* packed, float* s, float* z);
void or_dequant_i4a(const uint8_t* packed, const float* s, const float* z, int64_t n, int G,
                    float* d);

/* acc = 0; for p = 0..P-1: acc = acc + d_p   (slab order is the reduction order) */
void or_reduce_sum(const float* const* d, int P, int64_t n, float* out);

/* Two-step reduce of P quantized slabs (fmt INT8_SYM or INT4_ASYM), split into
 * `shards` contiguous shards of ceil(n_g/shards) groups.  Outputs (any may be
 * NULL): reduced fp32 sum, requantized payload, gathered dequantized fp32.
 * Returns 0, or -1 on a bad argument. */
int or_two_step(int fmt, const void* const* codes, const float* const* scales,
                const float* const* zeros, int P, int64_t n, int G, int shards,
                float* reduced, void* rq_codes, float* rq_scales, float* rq_zeros,
                float* gathered);

/* Standalone all-gather: shard j (of P) holds the payload of groups
 * [j*per, min((j+1)*per, n_g)), per = ceil(n_g/P), indexed from its own first
 * group (codes[j], scales[j], zeros[j]; zeros may be NULL for INT8).  out gets
 * the n dequantized values of the whole tensor.  Returns 0, or -1 on a bad
 * argument. */
int or_allgather_dequant(int fmt, const void* const* codes, const float* const* scales,
                         const float* const* zeros, int P, int64_t n, int G, float* out);

/* Residual add and RMSNorm over T rows of H: h = bf16(o + R) (fp32 add),
 * y = bf16(h / sqrt(mean(h^2) + eps) * gamma) (binary64). */
void or_residual_rmsnorm(const float* o, const uint16_t* r, const uint16_t* gamma, int64_t T,
                         int64_t H, float eps, uint16_t* h_out, uint16_t* y_out);

/* Self-validating 16-byte blocks: per row, ceil(H/6) blocks; block j of a
 * row holds row elements 6j..6j+5 as bf16 in words 0..2 (element 6j+2k in
 * the low half of word k, zero past the row end) and the epoch in word 3. */
int64_t or_tagged_blocks_per_row(int64_t H);
void or_pack_tagged(const uint16_t* x, int64_t T, int64_t H, uint32_t epoch, uint32_t* blocks);
/* returns -1 when every block carries `epoch`, else the first bad block index */
int64_t or_validate_tagged(const uint32_t* blocks, int64_t nblocks, uint32_t epoch);
void or_unpack_tagged(const uint32_t* blocks, int64_t T, int64_t H, uint16_t* x);

/* Self-synchronizing quantized payloads: every quantization group's payload
 * (INT8: its G code bytes then the fp32 scale; INT4: its G/2 packed code
 * bytes, the fp32 scale, the fp32 zero-point), zero-padded to a multiple of
 * 12 bytes, is cut into 12-byte pieces; each goes into a 16-byte block as
 * words 0..2 (little-endian payload bytes) with the epoch in word 3.  Groups
 * follow each other in row-major order. */
int or_qtagged_blocks_per_group(int fmt, int G);
void or_pack_qtagged(int fmt, const void* codes, const float* scales, const float* zeros,
                     int64_t n, int G, uint32_t epoch, uint32_t* blocks);
/* Unpacks codes/scales/zeros (zeros may be NULL for INT8) and returns -1 when
 * every block carries `epoch`, else the first bad block index. */
int64_t or_unpack_qtagged(int fmt, const uint32_t* blocks, int64_t n, int G, uint32_t epoch,
                          void* codes, float* scales, float* zeros);

/* Whole path from bf16 partial-sum slabs (the CPU baseline):
 * quantize each slab (sender side), two-step reduce with P shards, gather,
 * residual add, RMSNorm.  fmt BF16: plain fp32 sum of the bf16 slabs, no
 * quantization.  Writes h (residual out) and y; rq_* may be NULL. */
int or_allreduce_residual_rmsnorm(int fmt, const uint16_t* const* slabs, int P, int64_t T,
                                  int64_t H, int G, const uint16_t* r, const uint16_t* gamma,
                                  float eps, void* rq_codes, float* rq_scales, float* rq_zeros,
                                  uint16_t* h_out, uint16_t* y_out);

#ifdef __cplusplus
}
#endif
#endif
