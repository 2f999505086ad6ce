"""Planted mistakes: each altered copy of the oracle must fail at least one pin.

A plausible slip anywhere in the oracle (a dropped term, a wrong sign, index or
order, a transposed operand) has to be caught by the pins, or the pins do not
prove the oracle. Each mutant below is the oracle source with one line
changed, compiled to a temporary library on the CPU.
"""
import os

import pytest

import oracle
import oracle_pins as pins

MUTANTS = {
    "fold_reversed": ("for (int32_t k = 0; k < n_rows; ++k) {",
                      "for (int32_t k = n_rows - 1; k >= 0; --k) {"),
    "fold_no_divide": ("out[j] = acc / (float)n_rows;", "out[j] = acc;"),
    "fold_drops_last_rank": ("for (int32_t k = 0; k < n_rows; ++k) {",
                             "for (int32_t k = 0; k < n_rows - (n_rows > 1); ++k) {"),
    "rs_wrong_position": ("int32_t p = rank % shard_factor;", "int32_t p = rank / shard_factor;"),
    "adam_eps_inside_sqrt": ("float denom = sqrtf(v_hat) + eps;", "float denom = sqrtf(v_hat + eps);"),
    "adam_no_bias_correction": ("float m_hat = m / bias_corr1;", "float m_hat = m;"),
    "adam_no_v_bias_correction": ("float v_hat = v / bias_corr2;", "float v_hat = v;"),
    "adam_betas_swapped": ("float v = beta2 * exp_avg_sq[i] + one_minus_b2 * (g * g);",
                           "float v = beta1 * exp_avg_sq[i] + one_minus_b1 * (g * g);"),
    "adam_sign_flipped": ("float p = param[i] - lr * (m_hat / denom);",
                          "float p = param[i] + lr * (m_hat / denom);"),
    "adam_step_off_by_one": ("const float bias_corr1 = (float)(1.0 - pow(beta1_d, (double)step));",
                             "const float bias_corr1 = (float)(1.0 - pow(beta1_d, (double)(step + 1)));"),
    "adam_grad_not_squared": ("one_minus_b2 * (g * g);", "one_minus_b2 * g;"),
    "cast_truncates": ("u = u + 0x7FFFu + lsb;", "u = u;"),
    "cast_ties_up": ("u = u + 0x7FFFu + lsb;", "u = u + 0x8000u;"),
    "layout_pad_to_F": ("int64_t W = world_size;", "int64_t W = shard_factor;"),
    "pack_pad_not_zero": ("for (int64_t b = off * elem_size; b < padded_numel * elem_size; ++b) dst[b] = 0;",
                          "for (int64_t b = off * elem_size; b < padded_numel * elem_size; ++b) dst[b] = 1;"),
    "gather_interleaved": ("full[(int64_t)k * shard_numel + j] = shards[k][j];",
                           "full[(int64_t)j * n_shards + k] = shards[k][j];"),
    "step_wrong_group": ("memcpy(full_out[grp] + (int64_t)p * S, sh, sizeof(uint16_t) * (size_t)S);",
                         "memcpy(full_out[0] + (int64_t)p * S, sh, sizeof(uint16_t) * (size_t)S);"),
    "account_4P": ("out[4] = (F > 1 ? 3.0 * P : 0.0)", "out[4] = (F > 1 ? 4.0 * P : 0.0)"),
    "account_no_prefetch": ("out[2] = 2.0 * U * (1.0 + (double)prefetch);", "out[2] = 2.0 * U;"),
    "account_persist_over_N": ("out[0] = 16.0 * P / Fd;", "out[0] = 16.0 * P / Nd;"),
    "account_ring_AR_over_F": ("+ 2.0 * (R - 1.0) / R * P / Fd;", "+ 2.0 * (R - 1.0) / R * P;"),
    "zero_stage2_shards_weights": ("if (stage >= 2) grads = grads / n;", "if (stage >= 2) weights = weights / n;"),
    "zero_optimizer_8_bytes": ("optim = (4.0 + 4.0 + 4.0) * P;", "optim = (4.0 + 4.0) * P;"),
    "zero_stage3_comm_2P": ("out[5] = stage == 3 ? 3.0 * P : 2.0 * P;", "out[5] = 2.0 * P;"),
    "adam_bias_corrections_swapped": ("float m_hat = m / bias_corr1;", "float m_hat = m / bias_corr2;"),
    "adam_m_drops_one_minus_b1": ("float m = beta1 * exp_avg[i] + one_minus_b1 * g;",
                                  "float m = beta1 * exp_avg[i] + g;"),
    "adam_lr_squared": ("float p = param[i] - lr * (m_hat / denom);",
                        "float p = param[i] - lr * lr * (m_hat / denom);"),
    "cast_lsb_wrong_bit": ("uint32_t lsb = (u >> 16) & 1u;", "uint32_t lsb = (u >> 15) & 1u;"),
    "cast_nan_not_quieted": ("return (uint16_t)((u >> 16) | 0x0040u);", "return (uint16_t)(u >> 16);"),
    "fold_rounds_to_bf16": ("acc = acc + x;", "acc = bf16_to_f32(ora_bf16_rne(acc + x));"),
    "layout_shard_over_W": ("sizes_out[2] = padded / shard_factor;", "sizes_out[2] = padded / world_size;"),
    "pack_tensors_overlap": ("        off += numels[i];\n    }\n    for (int64_t b = off",
                             "        off += numels[i] > 0 ? numels[i] - 1 : 0;\n    }\n    for (int64_t b = off"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(before) >= 1, "mutation site not found: %s" % name
    mutated = src.replace(before, after, 1)
    path = os.path.join(tmp_path, "mut.c")
    with open(path, "w") as f:
        f.write(mutated)
    so = oracle.compile_oracle(path, os.path.join(tmp_path, "libmut.so"))
    mut = oracle.Oracle(so)
    caught = None
    for pin in pins.ALL_PINS:  # the first pin that fails is enough
        try:
            pin(mut)
        except (AssertionError, ValueError, IndexError):
            caught = pin.__name__
            break
    assert caught, "no pin catches the planted mistake %s" % name
