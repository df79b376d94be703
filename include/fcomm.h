/*
 * fcomm.h -- C ABI of libfcomm: the data-parallel compute of a quantized
 * tensor-parallel All-Reduce followed by residual add and RMSNorm, on one
 * GB300 (sm_103a).
 *
 * The method (pages, by title and section):
 *  - "Flash Communication: Reducing Tensor Parallelization Bottleneck for
 *    Fast Large Language Model Inference" (arXiv 2412.04964), summary,
 *    "Main contributions" item 2 and "Core ideas": activations are quantized
 *    to low bit-width in fine-grained groups before they are sent, and the
 *    All-Reduce runs in two steps (reduce-scatter of quantized shards, then
 *    all-gather of the requantized reduced shards).
 *  - flash-comm, abstract: self-synchronizing transfers in which every data
 *    block carries evidence of its readiness and the receiver validates the
 *    blocks it needs directly; the reduction order is decoupled from the
 *    transport order so every GPU gets the same result.
 *  - "TokenWeave: Efficient Compute-Communication Overlap for Distributed LLM
 *    Inference" (arXiv 2505.11329), abstract: the RMSNorm after each
 *    All-Reduce is fused into it, and a batch's tokens are split into two
 *    subsets whose work overlaps.
 *
 * On one GPU the P tensor-parallel ranks are P "slabs" (partial sums) in the
 * same HBM.  Slab order is the reduction order.
 *
 * Conventions for every entry point:
 *  - Ownership: the caller owns all memory.  Tensor arguments are DEVICE
 *    pointers; fc_qtensor / slab arrays themselves are HOST arrays of device
 *    pointers.  The library never allocates device memory, never frees and
 *    never synchronizes; every call is asynchronous on `stream` (NULL = the
 *    legacy default stream).
 *  - Layout: tensors are row-major [rows, hidden]; groups are `group`
 *    consecutive elements of one row (hidden % group == 0).  INT8 codes are
 *    int8[rows*hidden]; INT4 codes are uint8[rows*hidden/2] with element 2i
 *    in the low nibble of byte i and 2i+1 in the high nibble.  Scales and
 *    zero-points are fp32[rows*hidden/group], group-major.
 *  - Alignment: bf16 and fp32 tensors 32 bytes, codes and tagged blocks 16
 *    bytes, scales and zero-points 4 bytes.  Violations return
 *    FC_ERR_INVALID.
 *  - Errors: argument errors are returned before anything is launched
 *    (FC_ERR_INVALID, FC_ERR_UNSUPPORTED); a failed launch returns
 *    FC_ERR_CUDA.  fc_last_error() gives a message for the calling thread's
 *    last failure.  Data-dependent errors (a stale tagged block) are only
 *    reported through the optional device status words, so no call blocks.
 *  - rows == 0 is valid and launches nothing.
 *  - Launch: every kernel is launched with programmatic stream serialization
 *    (programmatic dependent launch, sm_90 and later).  It may be scheduled
 *    while the previous kernel in the stream is finishing, but waits for it
 *    to complete, and for its writes to become visible, before touching any
 *    memory, so stream order is kept.  It also lets the next kernel in the
 *    stream be scheduled early: a kernel the caller launches next with the
 *    same attribute must execute griddepcontrol.wait
 *    (cudaGridDependencySynchronize) before it reads this call's outputs.
 *    A kernel launched without the attribute, and any copy, event or
 *    host synchronization, is ordered as usual.
 */
#ifndef FCOMM_H
#define FCOMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st* fc_stream_t;

typedef enum {
  FC_OK = 0,
  FC_ERR_INVALID = 1,     /* bad argument: null/misaligned pointer, bad size or format */
  FC_ERR_CUDA = 2,        /* a CUDA call or kernel launch failed */
  FC_ERR_STALE_BLOCK = 3, /* device status only: a tagged block carried a wrong epoch */
  FC_ERR_UNSUPPORTED = 4  /* a valid request the library does not implement */
} fc_status;

typedef enum {
  FC_FMT_BF16 = 0,        /* unquantized bf16 payload */
  FC_FMT_INT8_SYM = 1,    /* INT8 symmetric: scale = absmax/127, codes in [-127, 127] */
  FC_FMT_INT4_ASYM = 2,   /* INT4 asymmetric: scale = (max-min)/15, zero = min, codes in [0, 15] */
  FC_FMT_BF16_TAGGED = 3, /* bf16 in epoch-tagged 16-byte blocks */
  FC_FMT_F32 = 4,         /* output dtype only (fc_requant_gather) */
  FC_FMT_INT8_TAGGED = 5, /* INT8 g128 groups as self-synchronizing blocks (11 per group) */
  FC_FMT_INT4_TAGGED = 6  /* INT4 g32 groups as self-synchronizing blocks (2 per group) */
} fc_format;

/* Quantization spec.  group: 16..512, a multiple of 16 (INT8 uses 128 and
 * INT4 uses 32 in the reference workloads).  Ignored for BF16 and TAGGED. */
typedef struct {
  int32_t fmt;   /* fc_format */
  int32_t group; /* elements per group */
} fc_qspec;

/* One quantized tensor: device pointers.  For FC_FMT_BF16 / FC_FMT_BF16_TAGGED
 * slabs, `codes` is the bf16 data / the tagged blocks and scales/zeros are
 * unused.  `zeros` is used by INT4 only. */
typedef struct {
  void* codes;
  float* scales;
  float* zeros;
} fc_qtensor;

/* ---------------------------------------------------------------- sizes -- */
/* Bytes of codes for rows x hidden elements (INT8: n, INT4: n/2, BF16: 2n,
 * TAGGED: fc_tagged_bytes).  0 for an invalid spec. */
size_t fc_codes_bytes(fc_qspec spec, int64_t rows, int64_t hidden);
/* Number of groups (= fp32 scales, = fp32 zero-points) for rows x hidden. */
size_t fc_groups(fc_qspec spec, int64_t rows, int64_t hidden);
/* Bytes of the tagged form of rows x hidden bf16: rows * ceil(hidden/6) * 16.
 * Each row is cut into ceil(hidden/6) blocks of 16 bytes: block j carries row
 * elements 6j..6j+5 as bf16 in 32-bit words 0..2 (element 6j+2k in the low
 * half of word k, zero past the row end) and the 32-bit epoch in word 3.
 * Blocks never straddle rows, so any row range is a contiguous block range. */
size_t fc_tagged_bytes(int64_t rows, int64_t hidden);
/* Group range [g0, g1) of shard `shard` when the groups are split into P
 * contiguous shards of ceil(n_groups/P) groups (the reduce-scatter partition
 * of the two-step All-Reduce).  Returns FC_ERR_INVALID on bad arguments. */
fc_status fc_shard_range(fc_qspec spec, int64_t rows, int64_t hidden, int P, int shard,
                         int64_t* g0, int64_t* g1);

/* ------------------------------------------------------------- compute -- */

/* Group-quantize one bf16 slab (the sender side of the quantized All-Reduce;
 * Flash Communication, "Main contributions" 2).
 *  x_bf16: [rows, hidden] bf16.  out: codes + scales (+ zeros for INT4), sized
 *  by fc_codes_bytes / fc_groups.  spec.fmt: INT8_SYM or INT4_ASYM.
 * Per group (fp32, IEEE division, round-to-nearest-even codes, no FMA):
 *  INT8: s = max|x|/127; q = clamp(rne(x/s), -127, 127); s == 0 -> codes 0.
 *  INT4: lo = min, hi = max (a zero extreme is +0); s = (hi-lo)/15; z = lo;
 *        q = clamp(rne((x-lo)/s), 0, 15); s == 0 -> codes 0.
 * d_status (optional, two int32 words of device memory, 4-byte aligned) is
 * set by this call to {FC_OK, 0x7F7F7F7F}; word 0 becomes FC_ERR_CUDA if a
 * shared-memory staging copy of the input fails to land within its bounded
 * wait (about a second), in which case the outputs are incomplete. */
fc_status fc_group_quantize(const void* x_bf16, int64_t rows, int64_t hidden, fc_qspec spec,
                            fc_qtensor out, int32_t* d_status, fc_stream_t stream);

/* Self-synchronizing quantized payloads (flash-comm, abstract: every block
 * carries evidence of its readiness; applied to Flash Communication's
 * fine-grained quantized groups).  spec.fmt FC_FMT_INT8_TAGGED (group 128) or
 * FC_FMT_INT4_TAGGED (group 32); other groups return FC_ERR_UNSUPPORTED.
 * Each group's payload -- INT8: its 128 code bytes then the fp32 scale (132
 * bytes); INT4: its 16 packed code bytes, the fp32 scale, the fp32 zero-point
 * (24 bytes) -- is cut into 12-byte pieces carried as words 0..2 of 16-byte
 * blocks whose word 3 is `epoch`: 11 blocks per INT8 group, 2 per INT4 group,
 * groups in row-major order (fc_codes_bytes gives the size).  The codes and
 * scales are exactly those fc_group_quantize computes.  P slabs (1..8, host
 * arrays of device pointers) in one launch.  The consumer is
 * fc_allreduce_residual_rmsnorm with the same spec: slabs[p].codes = blocks,
 * every block checked against expected_epoch, stale blocks reported through
 * d_status like FC_FMT_BF16_TAGGED (block index counted over the blocks of
 * slab 0's rows, then slab 1's, ...); its requant_out (optional) is the plain
 * INT8/INT4 payload.  d_status: optional, as for fc_group_quantize. */
fc_status fc_group_quantize_tagged(const void* const* x_bf16, int P, int64_t rows,
                                   int64_t hidden, fc_qspec spec, uint32_t epoch,
                                   void* const* blocks, int32_t* d_status, fc_stream_t stream);

/* Quantize P bf16 slabs in one launch; slab p reads x_bf16[p] and writes
 * out[p] (host arrays of P entries, 1 <= P <= 8).  Same result as P calls of
 * fc_group_quantize.  d_status: optional, as for fc_group_quantize. */
fc_status fc_group_quantize_multi(const void* const* x_bf16, int P, int64_t rows,
                                  int64_t hidden, fc_qspec spec, const fc_qtensor* out,
                                  int32_t* d_status, fc_stream_t stream);

/* Reduce-scatter stage math of the two-step All-Reduce (Flash Communication,
 * "Main contributions" 2; flash-comm abstract for the fixed order):
 *  out_f32[i] = ((0 + deq_0(i)) + deq_1(i)) + ... + deq_{P-1}(i), fp32,
 *  slab order, where deq(i) = q*s (INT8) or q*s + z (INT4, two roundings).
 *  slabs: host array of P (2..8) quantized slabs; out_f32: the whole
 *  [rows, hidden] fp32 tensor.  shard = -1 writes every element; shard j in
 *  [0, P) writes only shard j's groups (fc_shard_range). */
fc_status fc_reduce_dequant_sum(const fc_qtensor* slabs, int P, int64_t rows, int64_t hidden,
                                fc_qspec spec, int shard, float* out_f32, fc_stream_t stream);

/* All-gather half of the two-step All-Reduce (Flash Communication, "Core
 * ideas": every reduced shard is requantized and sent to every rank, which
 * dequantizes it).  Requantize a reduced fp32 tensor (same quantizer as
 * fc_group_quantize, applied to the fp32 values) into requant_out (the
 * all-gather payload), and write its dequantization to `out` as out_dtype
 * FC_FMT_BF16 (round to nearest even) or FC_FMT_F32.  requant_out.codes may
 * be NULL (payload not stored); out may be NULL (no dequantized output).
 * The kernel reads its input with plain loads (no staging copy, no wait),
 * so it has no status word. */
fc_status fc_requant_gather(const float* reduced_f32, int64_t rows, int64_t hidden, fc_qspec spec,
                            fc_qtensor requant_out, void* out, int32_t out_dtype,
                            fc_stream_t stream);

/* Producer side of the self-validating block format (flash-comm, abstract):
 * pack [rows, hidden] bf16 into fc_tagged_bytes(rows, hidden) bytes of
 * 16-byte blocks carrying `epoch`. */
fc_status fc_pack_tagged(const void* x_bf16, int64_t rows, int64_t hidden, uint32_t epoch,
                         void* blocks, fc_stream_t stream);

/* Pack P bf16 slabs (host arrays of P device pointers, 1 <= P <= 8) in one
 * launch: slab p reads x_bf16[p] and writes blocks[p].  Same result as P
 * calls of fc_pack_tagged. */
fc_status fc_pack_tagged_multi(const void* const* x_bf16, int P, int64_t rows, int64_t hidden,
                               uint32_t epoch, void* const* blocks, fc_stream_t stream);

/* The fused path: quantized All-Reduce + residual add + RMSNorm (Flash
 * Communication two-step reduce; TokenWeave fused AllReduce-RMSNorm).
 * For every row, in one kernel:
 *   o   = two-step result: INT8/INT4: dequant(requant(sum_p deq_p)),
 *         BF16/TAGGED: sum_p float(x_p) (fp32, slab order, from +0);
 *   h   = bf16(o + float(residual_in))          -> residual_out
 *   y_k = bf16((float(h_k) * inv) * float(gamma_k)),
 *         inv = 1 / sqrt(sum_k h_k^2 / hidden + eps)  (fp32)
 * slabs: host array of P (2..8) slabs in spec.fmt (INT8/INT4 quantized as by
 *   fc_group_quantize; BF16 data; TAGGED blocks from fc_pack_tagged).
 * residual_in, residual_out (may be the same pointer), y: [rows, hidden] bf16;
 * gamma: [hidden] bf16.  requant_out: INT8/INT4 only, optional (codes == NULL:
 * not written): the requantized reduced tensor, i.e. the all-gather payload.
 * expected_epoch: TAGGED only.  Every block of every slab is checked against
 * expected_epoch before it is summed; a block that fails is not summed.
 * d_status (optional, two int32 words of device memory) is set by this call
 * to {FC_OK, 0x7F7F7F7F}; if any tagged block fails it becomes
 * {FC_ERR_STALE_BLOCK, index of the first failing block, counting blocks
 * row-major over slab 0, then slab 1, ..., within this call's rows}; rows
 * with a failing block have unspecified outputs.  Nothing waits for data: on
 * one GPU the producer has finished by stream order, so a wrong tag is an
 * error, not a retry.  If a shared-memory staging copy of the TMA-staged
 * kernel fails to complete within its bounded wait (about a second), word 0
 * becomes FC_ERR_CUDA and the outputs are unspecified. */
fc_status fc_allreduce_residual_rmsnorm(const fc_qtensor* slabs, int P, int64_t rows,
                                        int64_t hidden, fc_qspec spec, const void* residual_in,
                                        void* residual_out, const void* gamma, float eps,
                                        fc_qtensor requant_out, void* y, uint32_t expected_epoch,
                                        int32_t* d_status, fc_stream_t stream);

/* Launch options for the fused path.  max_ctas > 0 caps the grid at that
 * many CTAs (persistent CTAs loop over rows), so the fused kernel can run on
 * a few SMs beside other work (TokenWeave, abstract: communication and
 * RMSNorm on only 2-8 SMs).  0 = size the grid to the whole GPU. */
typedef struct {
  int32_t max_ctas;
  /* 0: automatic; 1: the register-streaming kernel; 2: the TMA-staged kernel
   * (rows staged in shared memory by bulk copies; needs every per-row piece
   * to be a multiple of 16 bytes and 16-byte aligned tensors, else the call
   * returns FC_ERR_UNSUPPORTED).  All give bit-identical results. */
  int32_t kernel;
} fc_launch_opts;

fc_status fc_allreduce_residual_rmsnorm_ex(const fc_qtensor* slabs, int P, int64_t rows,
                                           int64_t hidden, fc_qspec spec,
                                           const void* residual_in, void* residual_out,
                                           const void* gamma, float eps, fc_qtensor requant_out,
                                           void* y, uint32_t expected_epoch, int32_t* d_status,
                                           const fc_launch_opts* opts, fc_stream_t stream);

/* Standalone quantized all-gather (flash-comm, abstract: the all-gather
 * collective; Flash Communication, "Core ideas": the second step of the
 * two-step All-Reduce, in which every rank receives all requantized shards
 * and dequantizes them).  Shard p (of P, 1..8) holds the payload of the
 * contiguous groups [p*per, min((p+1)*per, n_g)), per = ceil(n_g/P) -- the
 * partition of fc_shard_range -- indexed from its own first group: for
 * FC_FMT_INT8_SYM / FC_FMT_INT4_ASYM, shards[p] = {codes, scales, zeros}
 * (codes 16-byte aligned for INT8, 8-byte for INT4; scales and zeros 4-byte);
 * for FC_FMT_INT8_TAGGED / FC_FMT_INT4_TAGGED, shards[p].codes is its
 * epoch-tagged blocks (16-byte aligned; fc_group_quantize_tagged's layout) and
 * every block is checked against expected_epoch before use.  An empty shard
 * (p*per >= n_g) may have NULL buffers.  out: the whole [rows, hidden] tensor,
 * out_dtype FC_FMT_BF16 (round to nearest even) or FC_FMT_F32, 32-byte
 * aligned; element e = dequant of e's code (INT8: q*s; INT4: q*s + z, two
 * roundings).  d_status (optional, two int32 words, reset by the call):
 * {FC_OK, 0x7F7F7F7F}, or {FC_ERR_STALE_BLOCK, first stale block index}
 * counting shard 0's blocks, then shard 1's, ...; the outputs of a group
 * with a stale block are unspecified (the chunks read from it are not
 * written), every other group's are exact. */
fc_status fc_allgather_dequant(const fc_qtensor* shards, int P, int64_t rows, int64_t hidden,
                               fc_qspec spec, int32_t out_dtype, void* out, uint32_t expected_epoch,
                               int32_t* d_status, fc_stream_t stream);

/* Wave-aware token split (TokenWeave, abstract: the batch's tokens are
 * divided into two approximately equal subsets in a wave-aware manner; the
 * work of one overlaps the other's).  A "wave" is the number of rows the
 * fused kernel that fc_allreduce_residual_rmsnorm would launch for this
 * shape processes concurrently on the current GPU (SMs x resident rows per
 * SM, from the kernel's occupancy; returned in *wave_rows, may be NULL).
 * *split receives the first subset's row count: the multiple of the wave
 * nearest rows/2 (so the first subset is whole waves and the two subsets
 * together take no more waves than one unsplit call), or rows/2 when rows is
 * at most one wave.  Host-side query; launches nothing, allocates nothing. */
fc_status fc_token_split(int P, int64_t rows, int64_t hidden, fc_qspec spec, int64_t* split,
                         int64_t* wave_rows);

/* Cost-guided protocol choice (flash-comm, abstract: a selector adapts the
 * readiness encoding to the message size and the number of GPUs, balancing
 * synchronization overhead against additional data-transfer cost).  One-GPU
 * analogue: for P ranks reducing rows x hidden bf16 partial sums, estimate
 * one all-reduce step for every encoding whose bit width is >= min_bits (16:
 * bf16 only; 8: + INT8 g128; 4: + INT4 g32), plain and tagged:
 *   t = fused(format) + sender(format)                      (this GPU)
 *     + 2 (P-1)/P * payload(format) / link_gbps              (wire, optional)
 *     + (untagged ? 2 * barrier_us : 0)                      (readiness)
 * where fused and sender are the steady-state device times of one call
 * measured on GB300 by the message-size sweep (every encoding, P in {2, 4,
 * 8}, hidden 4096 and 8192, messages 16 KB .. 256 MB, compiled into the
 * library), interpolated log-linearly in the message size (proportional to
 * it above 256 MB), linearly in P, at the nearest measured hidden size;
 * tagged encodings carry 16/12 of the payload and need no barrier.  link ==
 * NULL models one GPU (no wire, no barrier).  *choice receives the fastest
 * encoding (group 128 for INT8, 32 for INT4), *est_us its estimate.
 * Host-only; no GPU needed; hidden must be a multiple of 128. */
typedef struct {
  double link_gbps;  /* per-GPU interconnect bandwidth, GB/s (> 0) */
  double barrier_us; /* cost of one all-rank readiness barrier, us (>= 0) */
} fc_link_model;

fc_status fc_select_protocol(int64_t rows, int64_t hidden, int P, int min_bits,
                             const fc_link_model* link, fc_qspec* choice, double* est_us);

/* The estimate fc_select_protocol makes for one encoding `spec` (BF16,
 * BF16_TAGGED, INT8_SYM or INT8_TAGGED with group 128, INT4_ASYM or
 * INT4_TAGGED with group 32; other specs return FC_ERR_UNSUPPORTED), in
 * *est_us.  Host-only. */
fc_status fc_protocol_estimate(int64_t rows, int64_t hidden, int P, fc_qspec spec,
                               const fc_link_model* link, double* est_us);

/* --------------------------------------------------------------- misc --- */
const char* fc_status_string(fc_status s);
/* Message describing the calling thread's last non-OK status ("" if none). */
const char* fc_last_error(void);
/* Library version, e.g. "libfcomm 0.1 sm_103a". */
const char* fc_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FCOMM_H */
