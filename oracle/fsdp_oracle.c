/*
 * CPU oracle of the FSDP FlatParameter shard step.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against. Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the library
 * under fully_sharded_gb300/ never links, loads or calls it, and the two share
 * no code. Single-threaded loops, no blocking, no fusion, no reordering.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (no FMA contraction: every fp32 operation below rounds once, IEEE RNE).
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
 * Sources (web pages on PyTorch FSDP; cited by page and section):
 *   [notes]   "NOTE-003: PyTorch FSDP" (reading notes on the FSDP paper)
 *   [math]    "transformer math: FSDP" (FlatParameter, cycles, budgets, worked example)
 *   [gloss]   glossary entry "fully sharded data parallel fsdp"
 * The Adam update itself is not written out on any of the pages (they say
 * only "Adam"); it follows Kingma & Ba 2015, Algorithm 1, weight decay 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_EINVAL (-1)
#define ORA_ENOMEM (-2)

/* ---------------------------------------------------------------------------
 * a1  FlatParameter layout.
 * [math] "The sharding unit: FlatParameter and the wrapping policy": the
 * parameters of a unit are flattened into one 1-D buffer that is split evenly
 * over the N ranks, each rank holding one contiguous 1/N slice. Even split =
 * pad the flat length up to a multiple of the world size W.
 * [notes] "Key results" / "Concepts": with sharding factor F the slice is 1/F
 * of the buffer (F = W full sharding, F = 1 replication, 1 < F < W hybrid).
 * The pad is a multiple of W for every F, so the layout is the same for all F.
 * ------------------------------------------------------------------------- */
int ora_flatten_layout(const int64_t *numels, int32_t n_tensors, int32_t world_size,
                       int32_t shard_factor, int64_t *offsets_out, int64_t *sizes_out)
{
    if (n_tensors < 1 || world_size < 1 || shard_factor < 1) return ORA_EINVAL;
    if (world_size % shard_factor != 0) return ORA_EINVAL;
    int64_t off = 0;
    for (int32_t i = 0; i < n_tensors; ++i) {
        if (numels[i] < 0) return ORA_EINVAL;
        offsets_out[i] = off;           /* row-major tensors, concatenated in order */
        off += numels[i];
    }
    offsets_out[n_tensors] = off;
    int64_t P = off;
    int64_t W = world_size;
    int64_t padded = ((P + W - 1) / W) * W;
    sizes_out[0] = P;                   /* real elements */
    sizes_out[1] = padded;              /* padded FlatParameter length */
    sizes_out[2] = padded / shard_factor; /* shard length S */
    return ORA_OK;
}

/* a2  pack: copy each tensor to its offset, zero the padding (+0.0 bits). */
void ora_pack(const void *const *tensors, const int64_t *numels, int32_t n_tensors,
              int32_t elem_size, int64_t padded_numel, void *flat)
{
    unsigned char *dst = (unsigned char *)flat;
    int64_t off = 0;
    for (int32_t i = 0; i < n_tensors; ++i) {
        const unsigned char *src = (const unsigned char *)tensors[i];
        for (int64_t b = 0; b < numels[i] * elem_size; ++b) dst[off * elem_size + b] = src[b];
        off += numels[i];
    }
    for (int64_t b = off * elem_size; b < padded_numel * elem_size; ++b) dst[b] = 0;
}

/* a2  unpack: the inverse copy, padding dropped. */
void ora_unpack(const void *flat, const int64_t *numels, int32_t n_tensors,
                int32_t elem_size, void *const *tensors)
{
    const unsigned char *src = (const unsigned char *)flat;
    int64_t off = 0;
    for (int32_t i = 0; i < n_tensors; ++i) {
        unsigned char *dst = (unsigned char *)tensors[i];
        for (int64_t b = 0; b < numels[i] * elem_size; ++b) dst[b] = src[off * elem_size + b];
        off += numels[i];
    }
}

/* ---------------------------------------------------------------------------
 * bfloat16 <-> fp32.  [gloss] "Mixed Precision": parameters in BF16,
 * reductions in FP32.  bf16 is the upper half of an fp32 bit pattern.
 * ------------------------------------------------------------------------- */
static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* a5  fp32 -> bf16, round to nearest, ties to even, by the integer method:
 * add 0x7FFF plus the lowest kept bit, then drop the low 16 bits. A NaN keeps
 * its sign and upper payload and is made quiet. */
uint16_t ora_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u = u + 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void ora_bf16_rne_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ora_bf16_rne(x[i]);
}

/* ---------------------------------------------------------------------------
 * a3  reduce-scatter (the reduction part).
 * [math] "The backward cycle: all-gather, grads, reduce-scatter": the
 * collective sums the full gradients of all ranks (the data-parallel average)
 * and each rank keeps the reduced slice matching its own parameter slice.
 * [gloss] "Mixed Precision": reduce_dtype = FP32.
 * Definition used: out[j] = (((0 + g_0[j]) + g_1[j]) + ... + g_{W-1}[j]) / W,
 * each g widened from bf16 to fp32, the sum a left fold in rank order, one
 * fp32 rounding per addition, then one IEEE fp32 division by W.
 * ------------------------------------------------------------------------- */
void ora_fold_mean(const uint16_t *const *rows, int32_t n_rows, int64_t n, float *out)
{
    for (int64_t j = 0; j < n; ++j) {
        float acc = 0.0f;
        for (int32_t k = 0; k < n_rows; ++k) {
            float x = bf16_to_f32(rows[k][j]);
            acc = acc + x;
        }
        out[j] = acc / (float)n_rows;
    }
}

/* The slice kept by `rank`: position p = rank mod F inside its group, elements
 * [p*S, (p+1)*S) of every rank's padded gradient, S = padded / F. All W ranks
 * are summed for every F (hybrid: one global fold, see ora_shard_step). */
int ora_reduce_scatter(const uint16_t *const *grads, int32_t world_size, int32_t shard_factor,
                       int64_t padded_numel, int32_t rank, float *out)
{
    if (world_size < 1 || shard_factor < 1 || world_size % shard_factor) return ORA_EINVAL;
    if (rank < 0 || rank >= world_size || padded_numel % world_size) return ORA_EINVAL;
    int64_t S = padded_numel / shard_factor;
    int32_t p = rank % shard_factor;
    const uint16_t **rows = (const uint16_t **)malloc(sizeof(*rows) * (size_t)world_size);
    if (!rows) return ORA_ENOMEM;
    for (int32_t k = 0; k < world_size; ++k) rows[k] = grads[k] + (int64_t)p * S;
    ora_fold_mean(rows, world_size, S, out);
    free(rows);
    return ORA_OK;
}

/* ---------------------------------------------------------------------------
 * a4  Adam on the local shard, in place; a5 the bf16 copy of the result.
 * [math] "Why FSDP exists": fp32 master copy plus Adam's fp32 momentum and
 * variance; "The backward cycle": the optimizer updates the local slice in
 * place. [gloss] "Optimizer Step": each GPU updates its own shard, no
 * communication.
 * Kingma & Ba 2015, Algorithm 1, weight decay 0, step t >= 1:
 *   m <- b1 m + (1 - b1) g
 *   v <- b2 v + (1 - b2) g^2
 *   mhat = m / (1 - b1^t),  vhat = v / (1 - b2^t)
 *   p <- p - lr * mhat / (sqrt(vhat) + eps)
 * The hyper-parameters arrive as double (the values a user writes, e.g.
 * 0.999); each fp32 scalar used per element (lr, b1, b2, eps, 1-b1, 1-b2,
 * 1-b1^t, 1-b2^t) is formed in double and rounded once to fp32. Everything
 * per element is fp32 with one rounding per operation.
 * ------------------------------------------------------------------------- */
void ora_adam(float *param, float *exp_avg, float *exp_avg_sq, const float *grad, int64_t n,
              double lr_d, double beta1_d, double beta2_d, double eps_d, int64_t step,
              uint16_t *bf16_out)
{
    const float lr = (float)lr_d, beta1 = (float)beta1_d, beta2 = (float)beta2_d;
    const float eps = (float)eps_d;
    const float one_minus_b1 = (float)(1.0 - beta1_d);
    const float one_minus_b2 = (float)(1.0 - beta2_d);
    const float bias_corr1 = (float)(1.0 - pow(beta1_d, (double)step));
    const float bias_corr2 = (float)(1.0 - pow(beta2_d, (double)step));
    for (int64_t i = 0; i < n; ++i) {
        float g = grad[i];
        float m = beta1 * exp_avg[i] + one_minus_b1 * g;
        float v = beta2 * exp_avg_sq[i] + one_minus_b2 * (g * g);
        float m_hat = m / bias_corr1;
        float v_hat = v / bias_corr2;
        float denom = sqrtf(v_hat) + eps;
        float p = param[i] - lr * (m_hat / denom);
        exp_avg[i] = m;
        exp_avg_sq[i] = v;
        param[i] = p;
        if (bf16_out) bf16_out[i] = ora_bf16_rne(p);
    }
}

/* ---------------------------------------------------------------------------
 * a6  all-gather (unshard).
 * [math] "The forward cycle: all-gather, compute, reshard": every rank
 * contributes its slice and each rank ends with the full unit parameters.
 * full[k*S + j] = shard_k[j], k = 0..F-1: a plain copy.
 * ------------------------------------------------------------------------- */
void ora_all_gather(const uint16_t *const *shards, int32_t n_shards, int64_t shard_numel,
                    uint16_t *full)
{
    for (int32_t k = 0; k < n_shards; ++k)
        for (int64_t j = 0; j < shard_numel; ++j) full[(int64_t)k * shard_numel + j] = shards[k][j];
}

/* ---------------------------------------------------------------------------
 * a7/a8  one unit's step for the owned ranks [rank_begin, rank_end), as the
 * plain sequence a3 -> a4 -> a5 -> a6 (no fusion).
 * Rank r sits in group g = r / F at position p = r mod F ([gloss] "HSDP":
 * shard within a group, replicate across groups; contiguous ranks form a
 * group). For each owned rank: reduce-scatter its slice (all W ranks, global
 * rank order), Adam on its own master/m/v, bf16 result written to slice p of
 * its group's full buffer. Then every group holding an owned rank gathers the
 * slices of its non-owned positions from other_shards[rank].
 * master/exp_avg/exp_avg_sq are indexed by r - rank_begin; full_out by group;
 * other_shards by rank (NULL entries allowed where unused).
 * ------------------------------------------------------------------------- */
int ora_shard_step(const uint16_t *const *grads, int32_t world_size, int32_t shard_factor,
                   int64_t padded_numel, int32_t rank_begin, int32_t rank_end,
                   float *const *master, float *const *exp_avg, float *const *exp_avg_sq,
                   const uint16_t *const *other_shards, uint16_t *const *full_out,
                   double lr, double beta1, double beta2, double eps, int64_t step)
{
    const int32_t W = world_size, F = shard_factor;
    if (W < 1 || F < 1 || W % F || padded_numel % W) return ORA_EINVAL;
    if (rank_begin < 0 || rank_end > W || rank_begin >= rank_end) return ORA_EINVAL;
    const int64_t S = padded_numel / F;
    float *g = (float *)malloc(sizeof(float) * (size_t)(S > 0 ? S : 1));
    uint16_t *sh = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(S > 0 ? S : 1));
    if (!g || !sh) { free(g); free(sh); return ORA_ENOMEM; }
    for (int32_t r = rank_begin; r < rank_end; ++r) {
        const int32_t grp = r / F, p = r % F, o = r - rank_begin;
        ora_reduce_scatter(grads, W, F, padded_numel, r, g);
        ora_adam(master[o], exp_avg[o], exp_avg_sq[o], g, S, lr, beta1, beta2, eps, step, sh);
        memcpy(full_out[grp] + (int64_t)p * S, sh, sizeof(uint16_t) * (size_t)S);
    }
    for (int32_t grp = 0; grp < W / F; ++grp) {
        int has_owned = 0;
        for (int32_t p = 0; p < F; ++p) {
            int32_t r = grp * F + p;
            if (r >= rank_begin && r < rank_end) has_owned = 1;
        }
        if (!has_owned) continue;
        for (int32_t p = 0; p < F; ++p) {
            int32_t r = grp * F + p;
            if (r >= rank_begin && r < rank_end) continue;
            if (!other_shards || !other_shards[r]) { free(g); free(sh); return ORA_EINVAL; }
            memcpy(full_out[grp] + (int64_t)p * S, other_shards[r], sizeof(uint16_t) * (size_t)S);
        }
    }
    free(g);
    free(sh);
    return ORA_OK;
}

/* ---------------------------------------------------------------------------
 * a9  closed-form memory and communication accountant.
 * [math] "Why FSDP exists": about 16 bytes per parameter (2 bf16 weight,
 *   2 bf16 grad, 4 fp32 master, 4 + 4 Adam moments); DDP holds 16P per GPU,
 *   sharding over N ranks holds 16P/N.
 * [math] "Per-unit memory and communication, in numbers":
 *   persistent = 16 P / N, transient = 2 U (1 + prefetch);
 *   a ring all-gather or reduce-scatter moves about P per rank, an
 *   all-reduce about 2P; FSDP = all-gather (fwd) + all-gather (bwd) +
 *   reduce-scatter (bwd) = 3P against DDP's 2P; bytes are 2 per element.
 * [notes] "Key results": F = 1 is DDP (all-reduce), F = W full sharding.
 * With F ranks per group and R = N/F groups (hybrid), state is sharded over F
 * (16 P / F), the three collectives run inside a group and the gradient slice
 * (P/F) is all-reduced across the R groups. Ring volumes per rank:
 *   ring  = 3 (F-1)/F P + 2 (R-1)/R P/F
 *   pages' rounded form = 3P [F > 1] + 2 P/F [R > 1]
 * (F = N gives 3P and 3(N-1)/N P; F = 1 gives 2P and 2(N-1)/N P.)
 * out[]: 0 persistent, 1 ddp_persistent, 2 transient, 3 peak,
 *        4 comm_elems (rounded), 5 comm_elems_ring,
 *        6 ddp_comm_elems (rounded), 7 ddp_comm_elems_ring,
 *        8 comm_bytes (rounded), 9 ddp_comm_bytes (rounded).
 * ------------------------------------------------------------------------- */
int ora_account(double P, double U, int32_t N, int32_t F, int32_t prefetch, double *out)
{
    if (N < 1 || F < 1 || N % F || prefetch < 0 || P < 0 || U < 0) return ORA_EINVAL;
    const double R = (double)(N / F);
    const double Fd = (double)F, Nd = (double)N;
    out[0] = 16.0 * P / Fd;
    out[1] = 16.0 * P;
    out[2] = 2.0 * U * (1.0 + (double)prefetch);
    out[3] = out[0] + out[2];
    out[4] = (F > 1 ? 3.0 * P : 0.0) + (R > 1.0 ? 2.0 * P / Fd : 0.0);
    out[5] = 3.0 * (Fd - 1.0) / Fd * P + 2.0 * (R - 1.0) / R * P / Fd;
    out[6] = 2.0 * P;
    out[7] = 2.0 * (Nd - 1.0) / Nd * P;
    out[8] = 2.0 * out[4];
    out[9] = 2.0 * out[6];
    return ORA_OK;
}

/* ---------------------------------------------------------------------------
 * ZeRO stages, per GPU persistent bytes.
 * [math] "Why FSDP exists": per parameter a 2-byte weight, a 2-byte gradient,
 *   a 4-byte fp32 master and 4 + 4 bytes of Adam moments.
 * [gloss] "ZeRO Stages": stage 1 shards the optimizer state over the N ranks,
 *   stage 2 also the gradients, stage 3 also the parameters (= FSDP).
 * out[]: 0 weights, 1 grads, 2 optimizer (master + moments), 3 total,
 *        4 16P / total, 5 communication elements per rank per step
 *        ([math] "Per-unit memory and communication": an all-reduce ~2P,
 *        FSDP's three collectives ~3P).
 * ------------------------------------------------------------------------- */
int ora_account_zero(double P, int32_t N, int32_t stage, double *out)
{
    if (N < 1 || stage < 0 || stage > 3 || P < 0) return ORA_EINVAL;
    double n = (double)N;
    double weights = 2.0 * P, grads = 2.0 * P, optim = (4.0 + 4.0 + 4.0) * P;
    if (stage >= 1) optim = optim / n;
    if (stage >= 2) grads = grads / n;
    if (stage >= 3) weights = weights / n;
    out[0] = weights;
    out[1] = grads;
    out[2] = optim;
    out[3] = weights + grads + optim;
    out[4] = out[3] > 0 ? 16.0 * P / out[3] : 1.0;
    out[5] = stage == 3 ? 3.0 * P : 2.0 * P;
    return ORA_OK;
}
