/*
 * qgemv.h -- C ABI of the block-quantized weight mat-vec library for GB300 (sm_103a).
 *
 * The operation (Track 2 Audit & Optimization Report: M5 Metal Kernels for
 * Multi-Token Speculative Decode, section 1 item 1, the multi-token gemv over
 * ntok activation rows; opus-mtp-turbo Track 1 report, item 3):
 *
 *     y[t][o] = sum_i dequant(W)[o][i] * x[t][i],   t < ntok <= 4,  o < n_out,  i < n_in
 *
 * and, for a vocabulary-sized head, the per-token argmax of y fused into the
 * same kernel (perf(speculative): cut the MTP drafter's per-step cost,
 * "Phase 2", item 2a).  The effective-bandwidth metric the library is built
 * for is weight bytes / kernel time (Where the time goes on an M2 Max,
 * "Dense K-quants are integer-ALU bound at small batches").
 *
 * Conventions for every call:
 *   - Device buffers (W, x, y, argmax, workspace) are allocated and owned by
 *     the caller.  qgemv and qgemv_argmax never allocate, free or synchronize;
 *     they enqueue one kernel on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and return.
 *   - Arguments are validated on the host before anything is launched.  A
 *     failed check returns a negative qg_status and launches nothing.  No
 *     call ever traps, asserts or exits.
 *   - The calls are reentrant and thread-safe.  The tile override (below) is
 *     process-wide.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight formats.  Byte counts per 32 weights: Q8_0 34, Q4_0 18, AFFINE4_G64 18, BF16 64,
 * Q5_0 22. */
typedef enum {
    QG_Q8_0 = 0,        /* 32-weight blocks: fp16 d + 32 int8 q; w = q*d                         */
    QG_Q4_0 = 1,        /* 32-weight blocks: fp16 d + 16 B of nibbles; w = (q-8)*d                */
    QG_AFFINE4_G64 = 2, /* 64-weight groups: 4-bit q, fp16 scale s, fp16 bias b; w = q*s + b      */
    QG_BF16 = 3,        /* plain bf16                                                             */
    QG_Q5_0 = 4         /* 32-weight blocks: fp16 d + 32 fifth bits + 16 B of nibbles; w = (q-16)*d */
} qg_fmt;

typedef int qg_status;
#define QG_OK            0
#define QG_EINVAL       (-1)  /* bad format, size, ntok or null pointer                 */
#define QG_EALIGN       (-2)  /* a pointer is not aligned as required                     */
#define QG_EUNSUPPORTED (-3)  /* valid but outside what the kernels handle (e.g. n_in too large) */
#define QG_EWORKSPACE   (-4)  /* argmax workspace missing or too small                  */
#define QG_ECUDA        (-5)  /* the CUDA runtime reported an error at launch             */

/* A static, human-readable string for a status code.  The status codes are this
 * library's own error contract (validation before launch, no trap or exit); the
 * pages have no counterpart. */
const char* qg_strerror(qg_status status);

/* ABI version of this header (incremented on incompatible change). */
int qg_abi_version(void);

/* ------------------------------------------------------------------ sizes and layouts
 * Canonical layout: the format's stored bytes, row-major, exactly the weight bytes
 * of the bandwidth metric (Where the time goes on an M2 Max, "Dense K-quants are
 * integer-ALU bound at small batches": effective bandwidth = weight bytes / time,
 * scales included).  The byte counts match the pages where they print them: Q8_0's
 * 34 bytes per 32 weights reproduces the (time, GB/s) rows of the Track 2 Audit &
 * Optimization Report's table 2.1 (e.g. 2560 x 40525 = 110.2 MB); the affine 4-bit
 * g64 head's 715.2 MB is the split of perf(speculative): cut the MTP drafter's
 * per-step cost, "The cost model" (weights 635.7 + scales 39.7 + biases 39.7 MB).
 * The pages name the formats but print no block layout: the layouts below are the
 * formats' usual ones (Q8_0 / Q4_0 / Q5_0 blocks of 32, MLX-style affine planes).
 *   Q8_0:  per 32-block: little-endian fp16 d, then 32 int8 q.
 *   Q4_0:  per 32-block: fp16 d, then 16 bytes; byte j holds element j in its low
 *          nibble and element j+16 in its high nibble.
 *   AFFINE4_G64: three planes, one after the other: uint32 words [n_out][n_in/8]
 *          (element k of a word at bits [4k,4k+4)), fp16 scales [n_out][n_in/64],
 *          fp16 biases [n_out][n_in/64].
 *   BF16:  bf16 [n_out][n_in].
 *   Q5_0:  per 32-block: fp16 d, a little-endian uint32 whose bit j is bit 4 of
 *          element j's code, then the 16 bytes of low nibbles in the Q4_0 order.
 * Device layout: what qgemv reads.  Rows are stored one after the other, so
 * the first k rows of a packed matrix are themselves a packed k-row matrix (a
 * reduced draft vocabulary that is a prefix of the head needs no copy).  A row
 * is a run of steps; a step is 512 bytes of codes followed by the scales of
 * exactly those codes, zero-padded to a 16-byte multiple (only the last step
 * of a row can be shorter).  No padding at all when the codes of a row are a
 * multiple of 512 bytes (n_in a multiple of 512 for Q8_0, 1024 for the 4-bit
 * formats, 256 for BF16), so then qg_packed_bytes == qg_canonical_bytes.
 *   codes:  Q8_0 q+128 (uint8); Q4_0, Q5_0 (low nibbles) and AFFINE4_G64 uint32
 *           words of 8 consecutive elements (element k at bits [4k,4k+4)); BF16 raw.
 *   scales: Q8_0 / Q4_0 one fp16 d per 32 weights; AFFINE4_G64 one (fp16 s,
 *           fp16 b) pair per 64 weights; Q5_0 one (uint32 fifth bits, fp16 d)
 *           record of 6 bytes per 32 weights, the fifth bit of block element e at
 *           bit 8b + g of the uint32, g = 2*(e/8) + e%2 and b = (e%8)/2 (shifting
 *           the word by 4 - g and masking 0x10101010 puts a group's fifth bits at
 *           bit 4 of its code bytes).
 * Sizes return 0 for invalid arguments. */
size_t  qg_canonical_bytes(qg_fmt fmt, int64_t n_out, int64_t n_in);
size_t  qg_packed_bytes(qg_fmt fmt, int64_t n_out, int64_t n_in);
int64_t qg_row_stride(qg_fmt fmt, int64_t n_in);     /* device-layout bytes per row */

/* --------------------------------------------------------------------- host packer
 * The pages give no encoder for any format (they time and name Q8_0, Q4_0 and
 * Q5_0 draft weights: opus-mtp-turbo Track 1 report, item 3, and the M2 Max page's
 * format table; the drafter issue's 4-bit head).  The quantizers below are the
 * rules of the workloads this library is measured on (d = max|w|/127 for Q8_0;
 * d = m/-8 with m the value of largest magnitude for Q4_0; min/max fit of s and
 * b per 64 for the affine format); what those rules leave open (rounding, nibble
 * order, which d the codes use) is stated per format.
 * All three work on host memory, use several CPU threads, and return QG_EINVAL on
 * a null pointer, n_out < 1, or n_in not a multiple of the block (32 for Q8_0,
 * Q4_0 and Q5_0; 64 for AFFINE4_G64; 16 for BF16, the kernels' 16-weight chunk).
 *
 * qg_quantize: fp32 W [n_out][n_in] -> canonical bytes (qg_canonical_bytes).
 *   Q8_0: d = max|w|/127 (fp32), stored fp16 (nearest even); q = roundf(w/d) with
 *         the fp32 d, clamped to [-127,127]; d = 0, q = 0 for an all-zero block.
 *   Q4_0: m = the signed value of largest |w| (first on ties); d = m/-8 (fp32),
 *         stored fp16; q = clamp(roundf(w/d)+8, 0, 15); d = 0, q = 8 when m == 0.
 *   AFFINE4_G64: s = fp16((max-min)/15), b = fp16(min); q = clamp(roundf((w-b)/s),
 *         0, 15) in fp32 with the fp16 s and b; q = 0 when s == 0.
 *   BF16: round to nearest even.
 *   Q5_0: as Q4_0 with 5-bit codes: d = m/-16 (fp32), stored fp16;
 *         q = clamp(roundf(w/d)+16, 0, 31); d = 0, q = 16 when m == 0.
 * qg_to_device_layout: canonical bytes -> device layout (qg_packed_bytes).
 * qg_pack: fp32 W -> device layout directly (same bytes as the two steps). */
qg_status qg_quantize(qg_fmt fmt, const float* W_host, int64_t n_out, int64_t n_in,
                      void* canonical_host);
qg_status qg_to_device_layout(qg_fmt fmt, const void* canonical_host, int64_t n_out,
                              int64_t n_in, void* packed_host);
qg_status qg_pack(qg_fmt fmt, const float* W_host, int64_t n_out, int64_t n_in,
                  void* packed_host);

/* --------------------------------------------------------------------------- qgemv
 * y[t][o] = sum_i dequant(W)[o][i] * x[t][i] for t < ntok, o < n_out.
 *   W     device, device layout (qg_packed_bytes(fmt, n_out, n_in) bytes), 16-B aligned.
 *   x     device, fp32 [ntok][n_in] row-major, 16-B aligned.
 *   y     device, fp32 [ntok][n_out] row-major, 4-B aligned; fully overwritten.
 *   ntok  1..4.   n_out >= 1.   n_in a positive multiple of the block (as above)
 *         and small enough that ntok*n_in fp32 values fit in one SM's shared
 *         memory (QG_EUNSUPPORTED otherwise; n_in <= 12288 always fits at ntok 4, and
 *         16384 for Q8_0, Q4_0 and AFFINE4_G64, whose x is staged as 16-bit integers).
 * Each output is an fp32 sum over n_in whose order depends only on the matrix
 * (fmt, n_out, n_in; see the split under tile selection): row t of an ntok=k
 * call is bitwise equal to the ntok=1 call on x[t], for every geometry, grid
 * and launch option (a forced split override changes the order).
 * Asynchronous on `stream`; returns QG_ECUDA if the launch is rejected. */
qg_status qgemv(qg_fmt fmt, const void* W, int64_t n_out, int64_t n_in,
                const float* x, float* y, int ntok, void* stream);

/* ----------------------------------------------------------------- qgemv_argmax
 * The same mat-vec fused with the per-token argmax over the n_out outputs
 * (vocabulary-sized LM heads): argmax[t] = the lowest o with y[t][o] equal to
 * max_o y[t][o].  A NaN output never wins; argmax[t] = -1 if every output is NaN.
 *   y          device fp32 [ntok][n_out], or NULL to skip writing the logits.
 *              When written, the logits are bitwise those qgemv produces, and
 *              argmax is the first-index argmax of exactly these values.
 *   argmax     device int32 [ntok], 4-B aligned.
 *   workspace  device, >= qgemv_argmax_workspace_bytes(n_out, ntok) bytes,
 *              16-B aligned, ZEROED by the caller once before its first use
 *              (cudaMemset).  Each call leaves it zeroed again for the next
 *              call; calls sharing one workspace must be serialized on one
 *              stream.
 * Same size rules as qgemv; QG_EWORKSPACE if the workspace is NULL or small. */
size_t    qgemv_argmax_workspace_bytes(int64_t n_out, int ntok);
qg_status qgemv_argmax(qg_fmt fmt, const void* W, int64_t n_out, int64_t n_in,
                       const float* x, float* y, int32_t* argmax, int ntok,
                       void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------ draft vocabulary given as an id list
 * A drafter may score only a listed subset of the LM head's rows ("Where the
 * time goes on an M2 Max", section "MTP draft vocabulary subset": the listed rows
 * are copied once into a small head) and map its argmax back to full-vocabulary
 * ids ("perf(speculative): cut the MTP drafter's per-step cost", Phase 2 item 2b:
 * a reduced draft vocabulary plus a d2t index mapping).  A list that is a row
 * prefix needs neither call: pass the first rows of the head to qgemv_argmax.
 *
 * qg_gather_rows: W_out (device layout, n_ids rows, qg_packed_bytes(fmt, n_ids,
 *   n_in) bytes, caller-allocated, 16-byte aligned, not overlapping W) receives
 *   row ids[j] of W (device layout, n_out rows, 16-byte aligned) as its row j.
 *   ids: n_ids int32 in device memory (4-byte aligned), any order, repeats
 *   allowed.  An id outside [0, n_out) gives a zero row and sets
 *   QG_DEVICE_BAD_ROW_ID in the device status word (qg_device_status); nothing
 *   outside W is read.  Asynchronous on `stream`; run it once per list, off the
 *   per-token path.  Errors: QG_EINVAL (format, shape, null pointer, n_ids < 1 or
 *   >= 2^31), QG_EALIGN, QG_ECUDA.
 *
 * qgemv_argmax_ids: qgemv_argmax over the gathered head W_sub (n_sub rows):
 *   y, if not NULL, receives the small head's logits [ntok][n_sub]; argmax[t]
 *   receives ids[j*], the full-vocabulary id of the winning row j* (the lowest j
 *   on ties; -1 when every logit is NaN).  ids: the n_sub int32 ids W_sub was
 *   gathered with, in device memory, read once per token at the end.  Workspace,
 *   ownership and errors as qgemv_argmax, plus QG_EINVAL for ids == NULL and
 *   QG_EALIGN for misaligned ids. */
#define QG_DEVICE_BAD_ROW_ID 2u
qg_status qg_gather_rows(qg_fmt fmt, const void* W, int64_t n_out, int64_t n_in,
                         const int32_t* ids, int64_t n_ids, void* W_out, void* stream);
qg_status qgemv_argmax_ids(qg_fmt fmt, const void* W_sub, int64_t n_sub, int64_t n_in,
                           const float* x, float* y, int32_t* argmax, int ntok,
                           const int32_t* ids, void* workspace, size_t workspace_bytes,
                           void* stream);

/* ------------------------------------------------------------ routed experts
 * The routed-expert projections of a mixture-of-experts layer at ntok <= 4 (Track
 * 2 Audit & Optimization Report, M5 Metal kernels, section 1 item 2, and table
 * 2.2): a plan groups the step's (token, choice) pairs by expert, and each
 * projection multiplies every group's expert once by the group's ne = 1..4 rows,
 * so each active expert's weights are read once per projection.
 *
 * qg_expert_plan: ids = device int32 [ntok][topk] (4-byte aligned), the expert of
 *   token t's choice j; pair i = t * topk + j; 1 <= ntok * topk <= 1024.  Writes
 *   the plan, qg_expert_plan_ints(ntok * topk) device int32 (caller-allocated,
 *   4-byte aligned), for G = ntok * topk slots:
 *     plan[0]                      n_groups
 *     plan[1 + g], g = 0..G        group_start: group g holds slots
 *                                  [group_start[g], group_start[g + 1]); entries
 *                                  n_groups..G hold G
 *     plan[2 + G + g], g < G       group_expert (-1 from n_groups on)
 *     plan[2 + 2G + s], s < G      slot_pair: the pair i in slot s
 *     plan[2 + 3G + s], s < G      slot_token = slot_pair / topk
 *     plan[2 + 4G + i], i < G      pair_slot: the slot of pair i
 *   Groups come in increasing expert id; a group's slots hold its pairs in
 *   increasing i; an expert with more than four pairs continues in the next
 *   group, four pairs at a time (the pages' plan has one group per expert; with
 *   ntok <= 4 and distinct experts per token the two agree).  An id outside
 *   [0, n_experts) sets QG_DEVICE_BAD_PLAN and writes n_groups = 0 (the rest of the
 *   plan is then unspecified).  One CTA, asynchronous on `stream`.  Errors:
 *   QG_EINVAL (null pointer, ntok, topk or n_experts < 1, ntok * topk > 1024),
 *   QG_EALIGN, QG_ECUDA.
 *
 * qgemv_experts: for every slot s of group g with e = group_expert[g],
 *     y[s][o] = sum_i dequant(W_e)[o][i] * x_row(s)[i],   o < n_out,
 *   where W_e = rows [e * n_out, (e + 1) * n_out) of W, the n_experts matrices
 *   stacked and packed as one (n_experts * n_out)-row matrix in the device layout
 *   (16-byte aligned), and x_row(s) = x[slot_token[s]] (the gate / up projections
 *   read the step's token rows) or, with QG_EXPERTS_X_BY_SLOT in flags, x[s] (the
 *   down projection reads one activation row per slot).  x: device fp32 [n_x][n_in],
 *   16-byte aligned.  y: device fp32 [n_slots][n_out], 4-byte aligned.  plan: as
 *   written by qg_expert_plan for n_slots = ntok * topk (or by the caller to the
 *   same layout).  The kernel reads n_groups and the groups from device memory;
 *   a plan entry out of range (n_groups > n_slots, a group of 0 or more than 4
 *   slots, an expert outside the stack, a row outside x) skips that group and
 *   sets QG_DEVICE_BAD_PLAN.  Each output is bitwise the same for every ne, group
 *   and geometry, and equals qgemv's on the expert's rows whenever that call does
 *   not split (qg_describe_tile shows split=1).
 *   QG_EXPERTS_SWIGLU in flags (a gate / up projection whose expert rows come in
 *   pairs, row 2j = gate j, row 2j + 1 = up j; n_out even): instead of the n_out
 *   projections, y[s][j] = silu(gate_j) * up_j with silu(v) = v / (1 + exp(-v)),
 *   fp32, y [n_slots][n_out / 2] — the down projection's input, with no separate
 *   activation launch.  QG_EUNSUPPORTED if a tile override forces an odd rpw.
 *   QG_EXPERTS_PLAN_READY in flags: the caller promises the plan is complete when
 *   this launch begins; the launch then reads it and starts its weight copies
 *   before waiting for the previous kernel (under early start, this overlaps the
 *   previous kernel's tail).  It holds without early start whenever the plan's
 *   writer precedes on the stream; under early start when the writer is at least
 *   two launches back and every launch in between is a qgemv_experts call (each
 *   lets its dependents begin only after its own wait) — e.g. plan, gate/up, down
 *   with the flag on the down call.  Errors: QG_EINVAL (format, shape,
 *   n_experts * n_out >= 2^31, n_slots outside 1..1024, n_x < 1, unknown flags,
 *   odd n_out with QG_EXPERTS_SWIGLU,
 *   n_x < n_slots with QG_EXPERTS_X_BY_SLOT, null pointer), QG_EALIGN,
 *   QG_EUNSUPPORTED, QG_ECUDA.  The geometry follows qg_set_tile_override's rpw,
 *   depth, warps and ctas (rpw 1, 2 or 4; the split does not apply) and gw: the CTAs
 *   are dealt to groups in proportion to gw + the group's token count (default 4;
 *   0 = equal shares; equal anyway when every group has one token).
 *   W_next (optional, NULL = none): the stack of the projection that comes next
 *   (same fmt and n_experts; next_n_out rows of next_n_in per expert, device
 *   layout, 16-byte aligned), e.g. the down projection while gate/up runs.  The
 *   launch prefetches each active expert's rows of it into L2 (a hint: no result
 *   changes, nothing is written), so the next launch starts on cached weights.
 *   Errors for it: QG_EINVAL (shape), QG_EALIGN. */
#define QG_DEVICE_BAD_PLAN 4u
#define QG_EXPERTS_X_BY_SLOT 1u
#define QG_EXPERTS_PLAN_READY 2u
#define QG_EXPERTS_SWIGLU 4u
/* qg_describe_expert_tile: the geometry qgemv_experts would use for one expert's
 * shape, written as qg_describe_tile does.
 *
 * qgemv_expert_layer: the whole routed-expert layer in ONE launch, for callers that
 * want one call instead of three.  It is the SLOWER path: on GB300 it measured 4-6%
 * slower than qg_expert_plan + qgemv_experts x 2 with early start (a barrier waits
 * for the slowest CTA just as the next launch would, and the single kernel holds
 * both projections' registers); prefer the three calls where speed matters.  (No
 * counterpart launch structure on the pages; the same arithmetic as qg_expert_plan +
 * qgemv_experts(gate/up, QG_EXPERTS_SWIGLU) + qgemv_experts(down, X_BY_SLOT), and
 * bitwise the same act and y).  Every CTA builds the plan from ids in shared memory
 * (the plan is also written to `plan`, qg_expert_plan_ints(ntok * topk) int32),
 * computes its groups' act = silu(gate) * up ([n_slots][d_ff], device fp32, 16-byte
 * aligned) while prefetching the same experts' down rows into L2, starts its first
 * down copies, waits at a barrier of its group's CTAs for the group's act, then
 * computes its groups' y = W_down . act ([n_slots][d_model], fp32, 4-byte aligned).
 *   W_gate_up: n_experts stacked [2 d_ff][d_model] matrices, rows interleaved gate /
 *   up (row 2j = gate j); W_down: n_experts stacked [d_model][d_ff]; both device
 *   layout, 16-byte aligned, same fmt.  x: [ntok][d_model] fp32, 16-byte aligned.
 *   ids: [ntok][topk] int32 (1 <= ntok * topk <= 1024).
 *   workspace: >= qgemv_expert_layer_workspace_bytes() bytes, 16-byte aligned,
 *   ZEROED by the caller once; each launch leaves it zeroed.  Launches sharing a
 *   workspace must be serialized (one stream).  After QG_DEVICE_WAIT_TIMEOUT,
 *   zero it again.
 *   The grid is one persistent wave, launched cooperatively: the driver starts it
 *   only when every CTA can be resident at once (early start is added when enabled
 *   and the driver accepts the pair; otherwise the launch is cooperative only).  The
 *   barriers' waits stay bounded as a guard: should a wait run out, the launch sets
 *   QG_DEVICE_WAIT_TIMEOUT and its y is not valid, so a caller that cannot rule that
 *   out checks qg_device_status after the call.  Errors: QG_EINVAL (shapes,
 *   ntok * topk, null pointers), QG_EALIGN, QG_EWORKSPACE, QG_EUNSUPPORTED,
 *   QG_ECUDA; a routed id outside [0, n_experts) sets QG_DEVICE_BAD_PLAN and the
 *   launch computes nothing. */
size_t    qgemv_expert_layer_workspace_bytes(void);
qg_status qgemv_expert_layer(qg_fmt fmt, const void* W_gate_up, const void* W_down, int64_t n_experts,
                             int64_t d_model, int64_t d_ff, const float* x, int ntok, const int32_t* ids,
                             int topk, int32_t* plan, float* act, float* y, void* workspace,
                             size_t workspace_bytes, void* stream);
size_t    qg_expert_plan_ints(int64_t n_pairs);
qg_status qg_expert_plan(const int32_t* ids, int ntok, int topk, int n_experts, int32_t* plan,
                         void* stream);
qg_status qgemv_experts(qg_fmt fmt, const void* W, int64_t n_experts, int64_t n_out, int64_t n_in,
                        const float* x, int64_t n_x, unsigned int flags, const int32_t* plan,
                        int64_t n_slots, float* y, const void* W_next, int64_t next_n_out,
                        int64_t next_n_in, void* stream);
qg_status qg_describe_expert_tile(qg_fmt fmt, int64_t n_out, int64_t n_in, char* buf, size_t len);

/* ------------------------------------------------------- qgemv_argmax_noalloc
 * No counterpart on the source pages: an addition for callers that cannot call
 * cudaMalloc, such as a plugin inside a host framework that owns every device
 * allocation, or a decode loop that must never hit the device allocator (which
 * can synchronize the device).  Same computation, arguments and rules as
 * qgemv_argmax, but without a workspace: the scratch it needs (a ticket and one
 * partial maximum per CTA and token) is a fixed array inside this library,
 * 32 KiB + 16 bytes, present on every GPU that loads the library until the
 * process exits.  It allocates nothing and calls no allocating routine.
 *   - The first call on a device looks up that array's device address for the
 *     current device (a one-time set-up, repeated only if the device's context
 *     changes, e.g. after cudaDeviceReset); make that first call before any
 *     stream capture.
 *   - Each call clears the ticket (cudaMemsetAsync on `stream`) before its
 *     kernel; the array otherwise keeps the last call's contents.
 *   - All calls on a device share the one array: calls that overlap on the GPU
 *     (different streams, no ordering between them) race and give wrong
 *     results.  Serialize them, e.g. on one stream.
 *   - A launch that would need partials for more than 1024 CTAs is refused
 *     with QG_EWORKSPACE (possible only with a tile override of many CTAs per
 *     SM); otherwise the errors are those of qgemv_argmax. */
qg_status qgemv_argmax_noalloc(qg_fmt fmt, const void* W, int64_t n_out, int64_t n_in,
                               const float* x, float* y, int32_t* argmax, int ntok,
                               void* stream);

/* --------------------------------------------------------------- tile selection
 * The kernel geometry (rows per warp, ring stages per warp, warps per CTA, CTAs
 * per SM) is chosen per (fmt, n_out, n_in, ntok) by a table measured on GB300
 * with a heuristic fallback (the Track 2 audit's per-shape, per-ntok tile
 * rules are the prior art).  The reduction order never depends on this choice.
 *
 * The split P (1..8) is chosen per (fmt, n_out, n_in) only: a row's steps are
 * cut into P segments, one per warp of a team, and the segments' sums are added
 * in segment order.  P fixes the reduction order, so it never depends on ntok
 * or the geometry: for a given matrix every ntok and every geometry give
 * bitwise the same rows.  (P = 1 for n_out >= 8192 or at most 6 steps of 512
 * code bytes per row; otherwise one segment per four steps, at most 4.)
 *
 * qg_set_tile_override: force a geometry for later calls, e.g.
 * "rpw=4,depth=4,warps=8,ctas=2,pre=1,split=2,gw=4" (any subset of the keys; rpw in
 * {1,2,3,4,5,6,8}: 1, 2, 4 for every ntok, 8 for ntok <= 3, 6 for ntok 2-4,
 * 3 and 5 for ntok 4 (QG_EUNSUPPORTED otherwise); where rpw * ntok > 20 a CTA
 * has at most 12 warps; depth in
 * {2..16}, warps in {1..16}, ctas in {1..8}, pre in {1..16}: the ring stages each
 * warp requests before the wait for the previous kernel, the rest once x is
 * staged (capped at depth), split in {1..8}, gw in {0..64}: the expert calls'
 * group weighting).  The
 * split is capped at one segment per step and
 * lowered until one team fits in shared memory at ntok = 4 (so it stays the
 * same for every ntok); warps are rounded to whole teams; the ring depth, then
 * the warp count, then the rows per warp are lowered if the CTA would not fit
 * in shared memory.  Forcing a split changes the reduction order of that
 * matrix (results stay within rounding of the default).
 * NULL or "" clears it.  The environment variable QGEMV_TILE, read at the
 * first call, sets the same override.  Returns QG_EINVAL on a malformed spec
 * (the override is unchanged).
 *
 * qg_describe_tile: writes the geometry a call would use into buf as
 * "rpw=..,depth=..,warps=..,ctas=..,pre=..,split=..,grid=.." (NUL-terminated,
 * truncated to len). */
qg_status qg_set_tile_override(const char* spec);
qg_status qg_describe_tile(qg_fmt fmt, int64_t n_out, int64_t n_in, int ntok,
                           char* buf, size_t len);

/* ------------------------------------------------------------- launch options
 * QG_LAUNCH_EARLY_START: launch with programmatic dependent launch.  Each kernel
 * lets the next kernel in the stream start as soon as SMs free up, and a kernel
 * that starts early begins copying its weights W before the previous kernel
 * has finished; it waits for that kernel to complete before it reads x or
 * writes y, argmax or the workspace.  So back-to-back calls (a decode chain of
 * projections) overlap one call's weight stream with the previous call's tail.
 * Enable it only when W is not written by work still in flight in the stream
 * (model weights are written once, before decoding).  Process-wide; default
 * off; the environment variable QGEMV_EARLY_START=1 turns it on at first use.
 * Unknown flags give QG_EINVAL. */
#define QG_LAUNCH_EARLY_START 1u
qg_status qg_set_launch_options(unsigned int flags);

/* ------------------------------------------------------------ device status
 * Every wait inside the kernels (on the mbarrier that counts a TMA copy into
 * shared memory) is bounded.  If a wait gives up, the kernel sets
 * QG_DEVICE_WAIT_TIMEOUT in a per-device status word, stops issuing copies,
 * drains the copies it already issued (again bounded) and exits normally; its
 * outputs are then not valid.  qg_gather_rows sets QG_DEVICE_BAD_ROW_ID when a
 * listed id is outside the head; qg_expert_plan and qgemv_experts set
 * QG_DEVICE_BAD_PLAN on a routed id or plan entry out of range.  qg_device_status copies the current device's
 * word into *status (synchronously: it waits for the device) and, if `clear`,
 * resets it to 0. */
#define QG_DEVICE_WAIT_TIMEOUT 1u
qg_status qg_device_status(int clear, unsigned int* status);

/* Test hook: `polls` = polls of an mbarrier before a wait gives up (0 restores
 * the default, about 4 million); `extra_tx_bytes` > 0 adds that many bytes to
 * the first expected transaction of every warp, so that wait can never
 * complete and the timeout path runs.  Process-wide; for tests only. */
qg_status qg_set_wait_limit(uint32_t polls, uint32_t extra_tx_bytes);

/* Profiling hook: per-CTA phase timestamps of the mat-vec kernel.  With `buf`
 * non-null (device memory of `slots` * QG_PHASE_SLOT_WORDS uint64, 8-byte aligned,
 * owned by the caller), every later qgemv / qgemv_argmax launch on this process
 * takes the next slot (a process-wide counter modulo `slots`, advanced at launch
 * time, so the launches of a captured graph keep distinct slots) and thread 0 of
 * CTA b writes the QG_PHASE_WORDS words at slot * QG_PHASE_SLOT_WORDS +
 * b * QG_PHASE_WORDS: [0] %globaltimer (ns) at entry, [1] %globaltimer when the
 * CTA's warps are done, [2] %smid; then the SM clock (%clock, 32 bits): [6] at
 * entry, [3] when warp 0 has issued its first copies, [4] after the wait for the
 * previous kernel, [5] after x is staged, [7] when warp 0 has finished its row
 * groups, [8] when every warp is done, and [9..15] when warp 0's ring stages 0..6
 * have landed, polled in order before the wait for the previous kernel (0 for
 * stages warp 0 did not fill).  The
 * launch then also ends with a CTA barrier.  `buf` = NULL turns the hook off
 * (the default); the results are unchanged either way.  The buffer must stay
 * allocated until the hook is off and every launch that recorded into it has
 * completed; launches captured into a CUDA graph while it is on keep their slots
 * and record on every replay.  QG_EINVAL if slots < 1 with a non-null buf, QG_EALIGN if buf is not
 * 8-byte aligned.  For profiling only; the expert calls do not record. */
#define QG_PHASE_WORDS 16
#define QG_PHASE_SLOT_WORDS (4096 * QG_PHASE_WORDS)
qg_status qg_set_phase_record(unsigned long long* buf, int64_t slots);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
