/*
 * fsdp.h - C ABI of the GB300 FSDP FlatParameter shard step.
 *
 * One GPU holds W virtual data-parallel ranks. For one FSDP unit the step is:
 * flatten the unit's tensors into one padded 1-D FlatParameter, reduce-scatter
 * the W bf16 full gradients (fp32 sum in fixed rank order, divided by W),
 * update each owned rank's fp32 master/exp_avg/exp_avg_sq shard with Adam in
 * place, cast the result to bf16, and all-gather the bf16 shards into the full
 * bf16 FlatParameter.
 *
 * The steps are labelled throughout the sources as follows:
 *   a1  flatten layout: tensor offsets, padding to a multiple of W, shard length
 *   a2  pack / unpack: tensors into the flat buffer (pad zeroed) and back
 *   a3  reduce-scatter: fp32 fold of the W bf16 rows in rank order, divided
 *       by W, at the rank's shard
 *   a4  Adam on a shard, in place (fp32 master, exp_avg, exp_avg_sq)
 *   a5  bf16 cast of the updated master shard
 *   a6  all-gather: the bf16 shards into the full FlatParameter
 *   a7  the fused step: a3 -> a4 -> a5 -> a6 in one pass
 *   a8  hybrid sharding (F | W): shard within groups of F, W / F replicas
 *   a9  closed-form memory and communication accountant
 *
 * Sources, cited by page title and section:
 *   [notes] "NOTE-003: PyTorch FSDP" (reading notes on the FSDP paper)
 *   [math]  "transformer math: FSDP"
 *   [gloss] glossary entry "fully sharded data parallel fsdp"
 *
 * Conventions for every call:
 *   - The caller owns all memory of the data. No call allocates, and the
 *     library keeps no state about the data between calls (it caches the SM
 *     count and kernel occupancy per device; fsdp_pipeline_step and
 *     fsdp_offload_step create and release CUDA events within a call; a
 *     per-device status word records a device wait that ran out, see
 *     fsdp_device_status). One fixed device array is part of the library's
 *     device code: the staging pool of fsdp_pipeline_step_noalloc, of
 *     FSDP_NOALLOC_STAGING_BYTES. The CUDA runtime reserves it on every GPU
 *     where it loads the library's device code, whether or not that entry
 *     point is ever called, and keeps it until the process exits.
 *   - Diagnostic calls that drive failure paths on purpose are declared in
 *     fsdp_test.h, not here.
 *   - "device" pointers point to CUDA global memory of the current device;
 *     pointer arrays themselves (const T* const*) are HOST arrays of device
 *     pointers and are read before the call returns.
 *   - Optimizer-state offload ([gloss] "CPU Offload"): the fp32 master,
 *     exp_avg and exp_avg_sq pointers of fsdp_shard_step(_grouped),
 *     fsdp_adam_shard_step and fsdp_pipeline_step may instead point to
 *     page-locked host memory mapped into the device's address space
 *     (cudaHostAlloc, or cudaHostRegister with cudaHostRegisterMapped, at an
 *     address the device can use as is). The kernels then read and write the
 *     state over the host link; nothing else changes. fsdp_offload_step
 *     instead copies the state between host memory and device slots.
 *   - bf16 values are passed as their uint16_t bit patterns; fp32 as float.
 *   - Every GPU call is asynchronous on `stream` (0 = legacy default stream).
 *     Inputs must stay unchanged, and outputs untouched, until the stream has
 *     passed the call.
 *   - Return value: FSDP_OK (0) or a negative status (below). All arguments
 *     are validated on the host before anything is launched; on a negative
 *     status nothing was launched (except FSDP_ECUDA from a failed launch).
 *     Kernels never trap.
 *   - Results are deterministic: the same inputs give bit-identical outputs.
 *   - Sizes are int64_t element counts; all device index arithmetic is 64-bit.
 */
#ifndef FSDP_GB300_H
#define FSDP_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st *fsdp_stream_t;

#define FSDP_OK 0
#define FSDP_EINVAL (-1) /* null pointer, bad size, W outside [1,64], F not dividing W,
                            rank outside [0,W), inconsistent layout, step < 1,
                            weight_decay != 0, ... */
#define FSDP_EALIAS (-2) /* an output overlaps an input or another output */
#define FSDP_ECUDA (-3)  /* a CUDA call or launch failed (cudaGetLastError) */
#define FSDP_ENOSPACE (-4) /* the work does not fit the fixed staging capacity of
                              fsdp_pipeline_step_noalloc */

#define FSDP_MAX_WORLD 64

#define FSDP_DTYPE_F32 0  /* 4-byte elements (fp32 master) */
#define FSDP_DTYPE_BF16 1 /* 2-byte elements (bf16 bits) */

/* Layout of one FlatParameter. [math] "The sharding unit: FlatParameter and the
 * wrapping policy": the unit's tensors are flattened into one 1-D buffer that is
 * split evenly over the ranks, each rank holding one contiguous slice.
 * [notes] "Key results": sharding factor F (F = W full shard, F = 1 DDP,
 * 1 < F < W hybrid). */
typedef struct {
  int64_t numel;        /* P: real elements (sum of tensor numels) */
  int64_t padded_numel; /* ceil(P / W) * W: zero padding at the end */
  int64_t shard_numel;  /* S = padded_numel / F: one rank's slice */
  int32_t world_size;   /* W, 1..64 */
  int32_t shard_factor; /* F, divides W; R = W / F replica groups */
  int32_t n_tensors;
} fsdp_layout_t;

/* Adam hyper-parameters (Kingma & Ba 2015, Algorithm 1; the pages name the
 * optimizer only: [math] "Why FSDP exists", [gloss] "Optimizer Step").
 * Each per-element fp32 scalar (lr, beta1, beta2, eps, 1-beta1, 1-beta2,
 * 1-beta1^step, 1-beta2^step) is formed in double and rounded once to fp32. */
typedef struct {
  double lr;
  double beta1;        /* in [0, 1) */
  double beta2;        /* in [0, 1) */
  double eps;          /* >= 0, added outside the square root */
  double weight_decay; /* must be 0 (the method uses none) */
  int64_t step;        /* t >= 1: the step being taken */
} fsdp_adam_t;

/* a1. Flatten layout (host only, no GPU).
 * [math] "The sharding unit: FlatParameter and the wrapping policy".
 * numels: n_tensors element counts (>= 0) in the order the tensors are packed
 * (row-major, concatenated, no padding between tensors).
 * offsets_out: caller-owned array of n_tensors + 1 entries; offsets_out[i] is
 * tensor i's first flat element, offsets_out[n_tensors] = P.
 * out: the layout. Padding is to a multiple of W for every F, so the layout is
 * the same for all sharding factors. EINVAL: n_tensors < 1, a negative numel,
 * W outside [1,64], F < 1 or F not dividing W, a null pointer. */
int fsdp_flatten_layout(const int64_t *numels, int32_t n_tensors, int32_t world_size,
                        int32_t shard_factor, int64_t *offsets_out, fsdp_layout_t *out);

/* a2. Pack tensors into the flat buffer (one launch), zero-filling the pad.
 * [math] "The sharding unit: FlatParameter and the wrapping policy": a unit's
 * parameters are flattened into one contiguous 1-D buffer (row-major, in the
 * listed order) that splits evenly over the ranks.
 * tensors: host array of n_tensors device pointers (contiguous tensors of the
 * element type `dtype`); offsets: the host array fsdp_flatten_layout wrote;
 * flat_out: device buffer of padded_numel elements. Pad elements become +0.0
 * (all-zero bits). EINVAL: a bad layout, dtype or offsets, a null pointer;
 * EALIAS if flat_out overlaps a tensor. */
int fsdp_pack_flat(const void *const *tensors, const fsdp_layout_t *layout,
                   const int64_t *offsets, int32_t dtype, void *flat_out, fsdp_stream_t stream);

/* a2. Unpack: copy each tensor's range of the flat buffer back out (pad dropped).
 * [math] "The sharding unit: FlatParameter and the wrapping policy": the
 * tensors are views of their ranges of the FlatParameter; this is the inverse
 * of fsdp_pack_flat. flat: device buffer of padded_numel elements of `dtype`;
 * tensors_out: host array of n_tensors device pointers, tensor i receives
 * elements [offsets[i], offsets[i+1]). EINVAL as for fsdp_pack_flat; EALIAS if
 * a tensor overlaps the flat buffer or another tensor. */
int fsdp_unpack_flat(const void *flat, const fsdp_layout_t *layout, const int64_t *offsets,
                     int32_t dtype, void *const *tensors_out, fsdp_stream_t stream);

/* a3. Reduce-scatter for one rank.
 * [math] "The backward cycle: all-gather, grads, reduce-scatter"; [gloss]
 * "Mixed Precision" (reduce_dtype fp32).
 * grads: host array of W device pointers, grads[k] = rank k's bf16 full
 * gradient, padded_numel elements (pad elements are expected to be zero).
 * rank: in [0, W); it keeps position p = rank mod F, i.e. elements [p*S, (p+1)*S).
 * grad_shard_out: device fp32 [S]:
 *   out[j] = ((((0 + g_0[pS+j]) + g_1[pS+j]) + ... ) + g_{W-1}[pS+j]) / W
 * a left fold in rank order over all W ranks, one fp32 rounding per add, IEEE
 * division. EALIAS if the output overlaps a gradient row. */
int fsdp_reduce_scatter(const uint16_t *const *grads, const fsdp_layout_t *layout,
                        int32_t rank, float *grad_shard_out, fsdp_stream_t stream);

/* a3 for the owned ranks [rank_begin, rank_end) in one launch (the same
 * definition and passages as fsdp_reduce_scatter; one GPU holding several
 * ranks reduces all of their slices at once).
 * grads: as in fsdp_reduce_scatter. grad_shards_out: rank_end - rank_begin
 * device pointers, fp32 [S] each, indexed by r - rank_begin; rank r's output
 * is fsdp_reduce_scatter of rank r bit for bit (ranks at the same position of
 * different groups get identical copies). EINVAL: a bad layout or rank range,
 * a null pointer; EALIAS: an output overlaps a gradient row or another
 * output. */
int fsdp_reduce_scatter_ranks(const uint16_t *const *grads, const fsdp_layout_t *layout,
                              int32_t rank_begin, int32_t rank_end, float *const *grad_shards_out,
                              fsdp_stream_t stream);

/* a4 + a5. Adam on one shard, in place, and its bf16 cast.
 * [math] "Why FSDP exists" (fp32 master, fp32 momentum and variance) and "The
 * backward cycle" (the optimizer updates the local slice in place).
 * master, exp_avg, exp_avg_sq: device fp32 [n], updated in place:
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g*g;
 *   p = p - lr * ((m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps))
 * every operation one fp32 rounding (no fused multiply-add).
 * grad_shard: device fp32 [n] (read only). bf16_shard_out: device bf16 [n],
 * round-to-nearest-even of the new master, or NULL for none. n >= 0. */
int fsdp_adam_shard_step(float *master, float *exp_avg, float *exp_avg_sq,
                         const float *grad_shard, int64_t n, const fsdp_adam_t *adam,
                         uint16_t *bf16_shard_out, fsdp_stream_t stream);

/* One shard of fsdp_adam_shard_step_grouped (same meaning as the arguments of
 * fsdp_adam_shard_step). */
typedef struct {
  float *master;            /* device fp32 [n], in place */
  float *exp_avg;           /* device fp32 [n], in place */
  float *exp_avg_sq;        /* device fp32 [n], in place */
  const float *grad_shard;  /* device fp32 [n], read only */
  uint16_t *bf16_shard_out; /* device bf16 [n], or NULL */
  int64_t n;                /* >= 0 */
} fsdp_adam_shard_t;

/* a4 + a5 over several shards (e.g. the shards of every rank a GPU holds, or
 * of several units) in one launch, with the same definition and passages as
 * fsdp_adam_shard_step and one set of hyper-parameters. Each shard's results
 * equal fsdp_adam_shard_step on it bit for bit. n_shards == 0 is a no-op.
 * EINVAL: n_shards < 0, a negative n, a null state or gradient pointer of a
 * non-empty shard, bad hyper-parameters; EALIAS: an output overlaps a
 * gradient or another output (of any shard). */
int fsdp_adam_shard_step_grouped(const fsdp_adam_shard_t *shards, int32_t n_shards,
                                 const fsdp_adam_t *adam, fsdp_stream_t stream);

/* a6. All-gather (unshard) one group.
 * [math] "The forward cycle: all-gather, compute, reshard".
 * shards: host array of F device pointers, shards[k] = bf16 [S] of position k;
 * full_out: device bf16 [padded_numel]; full_out[k*S + j] = shards[k][j].
 * A shard that already is the view full_out + k*S is left in place. */
int fsdp_all_gather(const uint16_t *const *shards, const fsdp_layout_t *layout,
                    uint16_t *full_out, fsdp_stream_t stream);

/* a7 / a8. Fused shard step of one unit for the owned ranks [rank_begin, rank_end):
 * reduce-scatter -> Adam -> bf16 cast -> all-gather in one launch, with no fp32
 * gradient written to memory.
 * Rank r belongs to group g = r / F (contiguous ranks form a group) at position
 * p = r mod F ([gloss] "Hybrid Sharding", "HSDP": shard within a group,
 * replicate across groups).
 *   grads:        W device pointers, bf16 [padded_numel] each (as in a3). For
 *                 every F all W ranks are summed in global rank order, so every
 *                 F gives bit-identical parameters.
 *   master, exp_avg, exp_avg_sq:
 *                 rank_end - rank_begin device pointers, fp32 [S] each, indexed
 *                 by r - rank_begin; updated in place (a4).
 *   other_shards: NULL when every group that contains an owned rank is fully
 *                 owned (all-ranks mode); otherwise W device pointers indexed by
 *                 rank, bf16 [S]: the already-updated shards of the non-owned
 *                 ranks in those groups (local-rank mode; entries of owned
 *                 ranks and of other groups are ignored and may be NULL).
 *   full_out:     R = W / F device pointers indexed by group, bf16 [padded_numel];
 *                 every group containing an owned rank is written completely:
 *                 owned positions with the new bf16 shard, the others copied
 *                 from other_shards (skipped when other_shards[r] already is
 *                 full_out[g] + p*S). Entries of other groups are ignored.
 * Positions owned by several replicas are reduced once and the result applied
 * to every replica. EALIAS: an output overlaps an input or another output.
 * padded_numel == 0 is a no-op. */
int fsdp_shard_step(const uint16_t *const *grads, const fsdp_layout_t *layout,
                    int32_t rank_begin, int32_t rank_end, float *const *master,
                    float *const *exp_avg, float *const *exp_avg_sq,
                    const uint16_t *const *other_shards, uint16_t *const *full_out,
                    const fsdp_adam_t *adam, fsdp_stream_t stream);

/* Arguments of one unit for fsdp_shard_step_grouped (same meaning as above). */
typedef struct {
  const fsdp_layout_t *layout;
  const uint16_t *const *grads;
  float *const *master;
  float *const *exp_avg;
  float *const *exp_avg_sq;
  const uint16_t *const *other_shards;
  uint16_t *const *full_out;
} fsdp_unit_args_t;

/* a7 over several units (e.g. one per transformer block, [math] "The sharding
 * unit": transformer_auto_wrap_policy makes each block a unit) in one launch
 * when they fit the launch's descriptor table, else in as few as needed.
 * The launch runs every unit's fused step first and then every unit's gather
 * of the other ranks' shards (the two touch disjoint memory, so the order
 * does not change any result). When many of the segments lie off 16-byte
 * alignment (shard lengths not a multiple of 8) and the aligned ones alone
 * fill the TMA form, the aligned segments go in a first launch and the
 * others in a second (again no result changes). All units share W, F, the owned rank range
 * and the hyper-parameters. Units must not share output memory.
 * n_units == 0 is a no-op. */
int fsdp_shard_step_grouped(const fsdp_unit_args_t *units, int32_t n_units, int32_t rank_begin,
                            int32_t rank_end, const fsdp_adam_t *adam, fsdp_stream_t stream);

/* Host only: the number of kernel launches fsdp_shard_step_grouped would make
 * for these arguments (validated exactly as the call validates them; nothing is
 * launched). *launches_out is written on FSDP_OK. */
int fsdp_shard_step_grouped_launches(const fsdp_unit_args_t *units, int32_t n_units,
                                     int32_t rank_begin, int32_t rank_end,
                                     int32_t *launches_out);

/* As fsdp_shard_step_grouped_launches, and *tma_launches_out (if not NULL)
 * receives how many of those launches use the TMA form of the kernel (bulk
 * copies into a shared-memory pipeline; chosen for W = 8 launches made of
 * one-replica step segments, and copies, for W = 16 ones whose gradient rows
 * do not all lie a multiple of 2 KB apart, and for launches of copies only, each with
 * enough chunks to fill every SM's pipeline and at most one eighth of its step
 * and of its copy chunks off 16-byte alignment), *tma_interleaved_out (if not
 * NULL) how many of the W = 8 TMA launches stage their step chunks in four
 * interleaved rounds of quarter-chunk copies (chosen when a launch's gradient
 * rows span 3 GiB or more of addresses).
 * Needs no GPU, but reads the SM count of the current device when one is
 * present. */
int fsdp_shard_step_grouped_plan(const fsdp_unit_args_t *units, int32_t n_units,
                                 int32_t rank_begin, int32_t rank_end, int32_t *launches_out,
                                 int32_t *tma_launches_out, int32_t *tma_interleaved_out);

/* The current device's sticky status word, read after all work of the
 * device, on every stream, has finished (the call synchronizes the device). Bit 0 is
 * set when a bounded wait of the TMA form ran out (2 s on one mbarrier): the
 * block that saw it stopped early, so the outputs of that launch are not
 * valid. This does not happen in a correct run. clear != 0 resets the word
 * after reading it. EINVAL: status_out NULL; ECUDA: the read failed. */
int fsdp_device_status(int32_t clear, uint32_t *status_out);

/* Pipelined step of one rank over many units (full sharding, F = W), with a
 * bounded pool of staging slots for the incoming gradients.
 * [notes] "Key results" (backward prefetching: issue the next unit's
 * collective before the current one finishes), [math] "Overlap: prefetching to
 * hide the collectives" and "Per-unit memory and communication, in numbers"
 * (transient = 2 U (1 + prefetch) bytes of bf16 per rank).
 * For unit u in order, slot s = u mod n_slots:
 *   on `copy`:    wait until the unit that last used slot s has been stepped,
 *                 then copy its W x S gradient slices into slot s;
 *   on `compute`: wait for that copy, run the fused local-rank step of `rank`
 *                 reading the gradients from slot s (reduce-scatter, Adam,
 *                 bf16 cast, all-gather of the other shards into full_out),
 *                 then copy the new bf16 shard to shard_out if given.
 * With n_slots = 1 (prefetch 0) copies and steps alternate; with n_slots = 2
 * (prefetch 1) the copy of unit u+1 overlaps the step of unit u.
 * The first and the last unit go through the same cycle in pieces of at most
 * 4,194,304 shard elements (whole 2048-element chunks; one 2D copy of the W
 * slices' ranges, one step and one shard_out copy per piece; each piece takes
 * the next slot), so that the first step starts before a whole unit has
 * arrived and little remains after the last copy in. Results do not depend on
 * the pieces.
 * staging: device bf16 buffer of n_slots x slot_numel elements, caller-owned,
 * slot_numel >= padded_numel of every unit (its W x S slices); n_slots in
 * [1, 8]; its contents are overwritten. The pool's size is the transient
 * gradient budget: 2 * n_slots * slot_numel bytes.
 * The call's copies start after the work queued on `compute` before the call
 * (so inputs written there, and a previous call's steps, come first); when the
 * call returns, `compute` is ordered after everything the call queued on both
 * streams, so later work on `compute` sees the results (order later work on
 * `copy` after `compute` yourself). The two streams may be the same stream (no
 * overlap). The call can be captured into a CUDA graph from `compute`.
 * Results are bit-identical to fsdp_shard_step_grouped on the same values.
 * EINVAL: F != W, a unit with
 * another W, bad rank, n_slots outside [1,8], a slot too small, null pointers;
 * EALIAS: outputs overlapping inputs, the staging pool or each other. */
typedef struct {
  const fsdp_layout_t *layout;
  const uint16_t *grad_slices;         /* W x S bf16 (row k = rank k's gradient at the
                                          owned slice), host (pinned) or device memory */
  float *master;                       /* device fp32 [S] of the owned rank, in place */
  float *exp_avg;                      /* device fp32 [S] */
  float *exp_avg_sq;                   /* device fp32 [S] */
  const uint16_t *const *other_shards; /* W device pointers by rank; the owned rank's entry
                                          is ignored */
  uint16_t *full_out;                  /* device bf16 [padded_numel] */
  uint16_t *shard_out;                 /* bf16 [S] (host or device) or NULL */
} fsdp_pipeline_unit_t;

int fsdp_pipeline_step(const fsdp_pipeline_unit_t *units, int32_t n_units, int32_t rank,
                       uint16_t *staging, int64_t slot_numel, int32_t n_slots,
                       const fsdp_adam_t *adam, fsdp_stream_t compute, fsdp_stream_t copy);

/* Staged optimizer-state offload: one rank's step over many units (full
 * sharding, F = W) with that rank's fp32 master, exp_avg and exp_avg_sq
 * shards in host memory.
 * [gloss] "CPU Offload" (optimizer state held in CPU memory and brought to the
 * GPU for the update); [math] "The backward cycle: all-gather, grads,
 * reduce-scatter" (the per-unit step it wraps).
 * For unit u in order, slot s = u mod n_slots of `staging`:
 *   on `h2d`:     wait until the unit that last used slot s is back in host
 *                 memory, then copy the unit's master, exp_avg, exp_avg_sq
 *                 (S fp32 each) into slot s;
 *   on `compute`: wait for those copies, run the fused local-rank step of
 *                 `rank` on the state in slot s (reduce-scatter of the rank's
 *                 slice of the W gradient rows, Adam, bf16 cast into full_out,
 *                 all-gather of the other ranks' shards into full_out);
 *   on `d2h`:     wait for the step, copy the three updated shards back to
 *                 host memory.
 * With n_slots >= 2 the copy in of unit u+1, the step of unit u and the copy
 * back of unit u-1 overlap, so both directions of the host link are busy at
 * once (the zero-copy form of the conventions above moves the same state by
 * kernel loads and stores instead).
 * staging: device fp32 buffer of n_slots x 3 x slot_numel, caller-owned,
 * contents overwritten; slot_numel >= shard_numel of every unit (a multiple
 * of 4 keeps every slot array 16-byte aligned, the vector path). n_slots in
 * [1, 8]. master/exp_avg/exp_avg_sq: host memory, page-locked for the copies
 * to overlap (pageable memory works but each copy then waits for the host);
 * device memory also works. The call's copies start after the work queued
 * on `compute` before the call; when the call returns, `compute` is ordered
 * after everything the call queued, the last copy back included, so later work
 * on `compute` sees the updated state. The streams may coincide (no overlap).
 * The call can be captured into a CUDA graph from `compute`. Results are
 * bit-identical to fsdp_shard_step_grouped with the same state in HBM.
 * EINVAL: F != W, a unit with another W, bad rank, n_slots outside [1,8], a
 * slot too small, null pointers; EALIAS: outputs (state, full_out, staging)
 * overlapping inputs or each other. */
typedef struct {
  const fsdp_layout_t *layout;
  const uint16_t *const *grads;        /* W device bf16 rows of padded_numel (rank k's
                                          gradient); the step reads the owned slice */
  float *master;                       /* fp32 [S] of the owned rank, host memory, in place */
  float *exp_avg;                      /* fp32 [S], host memory, in place */
  float *exp_avg_sq;                   /* fp32 [S], host memory, in place */
  const uint16_t *const *other_shards; /* W device pointers by rank; the owned rank's entry
                                          is ignored */
  uint16_t *full_out;                  /* device bf16 [padded_numel] */
} fsdp_offload_unit_t;

int fsdp_offload_step(const fsdp_offload_unit_t *units, int32_t n_units, int32_t rank, float *staging,
                      int64_t slot_numel, int32_t n_slots, const fsdp_adam_t *adam,
                      fsdp_stream_t compute, fsdp_stream_t h2d, fsdp_stream_t d2h);

/* Allocation-free form of fsdp_pipeline_step. (The FSDP pages have no
 * counterpart: this exists for callers, not for the method.)
 * For callers that cannot allocate device memory where they step the
 * optimizer: processes whose device memory is owned entirely by another
 * allocator (a framework's caching allocator, or a fixed arena carved out at
 * start-up), and loops that must not call cudaMalloc because it can
 * synchronize the device and stall the very streams the pipeline overlaps.
 * They pass only inputs and outputs; the staging pool is a fixed array of
 * FSDP_NOALLOC_STAGING_BYTES inside the library's device code, which the CUDA
 * runtime reserves on a GPU when it loads that code there and keeps until the
 * process exits. The call itself allocates nothing.
 * Same arguments and results as fsdp_pipeline_step, with slot_numel = the
 * largest padded_numel among the units rounded up to a multiple of 8 (so every
 * slot starts 16-byte aligned). FSDP_ENOSPACE (nothing launched) if
 * n_slots * slot_numel * 2 exceeds FSDP_NOALLOC_STAGING_BYTES.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture. Every
 * call on a device uses the same array: calls whose work overlaps on the GPU
 * (different streams without ordering between them) race on it and give
 * wrong results. Each unit's slot is filled completely before it is read, so
 * nothing needs clearing between calls. */
#define FSDP_NOALLOC_STAGING_BYTES (64ll << 20)

int fsdp_pipeline_step_noalloc(const fsdp_pipeline_unit_t *units, int32_t n_units, int32_t rank,
                               int32_t n_slots, const fsdp_adam_t *adam, fsdp_stream_t compute,
                               fsdp_stream_t copy);

/* Gather of any per-rank state into the full flat buffer of a group, for the
 * full state dict. [gloss] "Checkpoint/Resume": FULL_STATE_DICT gathers the
 * full model (on rank 0) instead of saving one piece per rank.
 * shards: F device pointers, shards[k] = S elements of position k, element
 * type `dtype` (FSDP_DTYPE_F32 for master / exp_avg / exp_avg_sq, FSDP_DTYPE_BF16
 * for parameters); full_out: padded_numel elements, full_out[k*S + j] =
 * shards[k][j]. A shard that already is the view full_out + k*S is left in
 * place. fsdp_unpack_flat then splits full_out into the unit's tensors. */
int fsdp_all_gather_state(const void *const *shards, const fsdp_layout_t *layout, int32_t dtype,
                          void *full_out, fsdp_stream_t stream);

/* ZeRO stage 1 step of one rank ([gloss] "ZeRO Stages": stage 1 shards only
 * the optimizer state; every rank keeps the full model and the full averaged
 * gradient; [notes] "Key results": F = 1 reduces to an all-reduce).
 * Two launches on `stream`: (1) the all-reduce average of the W bf16 gradients
 * over the whole padded buffer into avg_grad_out (fp32 [padded_numel], the
 * same fixed-order fold and division as the reduce-scatter); (2) Adam on the
 * rank's slice avg_grad_out[rank*S, (rank+1)*S) of its fp32 master/exp_avg/
 * exp_avg_sq [S] with the bf16 result written to full_out + rank*S, and the
 * other ranks' bf16 shards copied into full_out (other_shards by rank, the
 * owned entry ignored). Requires F = W. Results equal fsdp_shard_step of the
 * same rank bit for bit; avg_grad_out equals fsdp_reduce_scatter with F = 1. */
int fsdp_zero1_step(const uint16_t *const *grads, const fsdp_layout_t *layout, int32_t rank,
                    float *avg_grad_out, float *master, float *exp_avg, float *exp_avg_sq,
                    const uint16_t *const *other_shards, uint16_t *full_out, const fsdp_adam_t *adam,
                    fsdp_stream_t stream);

/* ZeRO-stage accountant (host only). Per-GPU persistent bytes with the 16
 * bytes per parameter of [math] "Why FSDP exists" split as 2 (bf16 weights)
 * + 2 (bf16 gradients) + 12 (fp32 master, m, v), and [gloss] "ZeRO Stages":
 *   stage 0 (DDP): 2P + 2P + 12P
 *   stage 1: 2P + 2P + 12P/N      (optimizer state sharded)
 *   stage 2: 2P + 2P/N + 12P/N    (+ gradients sharded)
 *   stage 3: 2P/N + 2P/N + 12P/N  (+ parameters sharded: FSDP full sharding)
 * comm_elems per rank per step (pages' rounded form, [math] "Per-unit memory
 * and communication"): 2P for stages 0-2 (an all-reduce, or reduce-scatter +
 * all-gather), 3P for stage 3. reduction_vs_ddp = 16P / total_bytes. */
typedef struct {
  double weights_bytes;
  double grads_bytes;
  double optimizer_bytes;
  double total_bytes;
  double reduction_vs_ddp;
  double comm_elems;
} fsdp_zero_account_t;

int fsdp_account_zero(double P, int32_t N, int32_t stage, fsdp_zero_account_t *out);

/* a9. Closed-form accountant (host only).
 * [math] "Why FSDP exists": ~16 bytes per parameter (bf16 weight + bf16 grad +
 * fp32 master + two fp32 Adam moments); DDP keeps 16P on every GPU.
 * [math] "Per-unit memory and communication, in numbers":
 *   persistent = 16 P / N, transient = 2 U (1 + prefetch); a ring all-gather or
 *   reduce-scatter moves ~P per rank, an all-reduce ~2P; FSDP pays
 *   AG(fwd) + AG(bwd) + RS(bwd) ~ 3P against DDP's ~2P; bf16 on the wire.
 * With sharding factor F over N ranks (R = N / F groups): persistent 16 P / F;
 * the three collectives run inside a group and the gradient slice P/F is
 * all-reduced across the R groups:
 *   comm_elems_ring = 3 (F-1)/F P + 2 (R-1)/R P/F
 *   comm_elems      = 3P [F > 1] + 2 P/F [R > 1]   (the pages' rounded form)
 * P, U: total parameters and parameters of the largest unit; prefetch >= 0
 * units gathered ahead. EINVAL: N < 1, F < 1, F not dividing N, negatives. */
typedef struct {
  double persistent_bytes;     /* 16 P / F */
  double ddp_persistent_bytes; /* 16 P */
  double transient_bytes;      /* 2 U (1 + prefetch) */
  double peak_bytes;           /* persistent + transient */
  double comm_elems;           /* per rank per step, rounded form */
  double comm_elems_ring;      /* per rank per step, exact ring form */
  double ddp_comm_elems;       /* 2P */
  double ddp_comm_elems_ring;  /* 2 (N-1)/N P */
  double comm_bytes;           /* 2 bytes per element */
  double ddp_comm_bytes;
} fsdp_account_t;

int fsdp_account(double P, double U, int32_t N, int32_t F, int32_t prefetch,
                 fsdp_account_t *out);

/* Text of a status code (static storage). */
const char *fsdp_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FSDP_GB300_H */
