"""Synthetic workloads: tensor shapes per FSDP unit, value distributions and stream keys.

Shapes only (no trained weights, no model code); the FlatParameter layout of
each unit is computed by the library (or by the oracle in the tests), not here.

  tiny_mlp     one unit: 64x32, 32, 32x16, 16 (2,608 params); W = 4;
               master N(0, 0.02), grads N(0, 1e-2), m = v = 0; 3 steps
  llama_block  one unit = one Llama-style block: q,k,v,o 4096x4096,
               gate/up 11008x4096, down 4096x11008, two RMSNorm 4096
               (202,383,360 params); W = 8; master N(0, 0.02),
               grads N(0, 1e-3), m and v |N(0, 1e-4)|
  gpt2_small   12 GPT-2 blocks (d = 768, ff = 3072) + root unit (wte 50257x768,
               wpe 1024x768, ln_f; lm_head tied): 124,439,808 params, W = 8;
               master N(0, 0.02), grads N(0, 1e-3), m = v = 0
  hybrid       the Llama block with W = 16 and F in {1, 4, 16}; same draws as llama_block
  llama7b      32 Llama blocks + root unit (embed 32000x4096, untied lm_head,
               final norm): 6,738,415,616 params, W = 8, one rank's step
               (local-rank mode); same draws as llama_block
"""
from __future__ import annotations

from dataclasses import dataclass, field

from . import (KIND_EXP_AVG, KIND_EXP_AVG_SQ, KIND_GRAD, KIND_MASTER, KIND_SHARD, stream_key)

SEED = 0

TINY_MLP_UNIT = [(64, 32), (32,), (32, 16), (16,)]

LLAMA_BLOCK_UNIT = [(4096, 4096)] * 4 + [(11008, 4096), (11008, 4096), (4096, 11008), (4096,), (4096,)]

GPT2_BLOCK_UNIT = [
    (768,), (768,),            # ln_1 weight, bias
    (768, 2304), (2304,),      # attn.c_attn weight, bias
    (768, 768), (768,),        # attn.c_proj weight, bias
    (768,), (768,),            # ln_2 weight, bias
    (768, 3072), (3072,),      # mlp.c_fc weight, bias
    (3072, 768), (768,),       # mlp.c_proj weight, bias
]
GPT2_ROOT_UNIT = [(50257, 768), (1024, 768), (768,), (768,)]  # wte, wpe, ln_f weight, bias

LLAMA7B_ROOT_UNIT = [(32000, 4096), (32000, 4096), (4096,)]  # embed, lm_head, final norm


def numels(unit_shapes):
    out = []
    for s in unit_shapes:
        n = 1
        for d in s:
            n *= d
        out.append(n)
    return out


@dataclass
class Workload:
    name: str
    config_id: int
    units: list                  # list of unit shape lists
    world_size: int
    shard_factors: tuple = ()     # () = (W,)
    sigma_master: float = 0.02
    sigma_grad: float = 1e-3
    sigma_state: float = 0.0      # 0 = zero Adam state
    steps: int = 1
    notes: str = ""
    extra: dict = field(default_factory=dict)

    def factors(self):
        return self.shard_factors or (self.world_size,)


TINY_MLP = Workload("tiny_mlp", 1, [TINY_MLP_UNIT], 4, sigma_grad=1e-2, steps=3)
LLAMA_BLOCK = Workload("llama_block", 2, [LLAMA_BLOCK_UNIT], 8, sigma_state=1e-4)
GPT2_SMALL = Workload("gpt2_small", 3, [GPT2_BLOCK_UNIT] * 12 + [GPT2_ROOT_UNIT], 8)
HYBRID = Workload("hybrid", 4, [LLAMA_BLOCK_UNIT], 16, shard_factors=(1, 4, 16), sigma_state=1e-4)
LLAMA7B = Workload("llama7b", 5, [LLAMA_BLOCK_UNIT] * 32 + [LLAMA7B_ROOT_UNIT], 8, sigma_state=1e-4)

ALL = {w.name: w for w in (TINY_MLP, LLAMA_BLOCK, GPT2_SMALL, HYBRID, LLAMA7B)}


# -------------------------------------------------------------- stream keys

def key_master(wl: Workload, unit: int) -> int:
    return stream_key(SEED, wl.config_id, unit, KIND_MASTER)


def key_exp_avg(wl: Workload, unit: int) -> int:
    return stream_key(SEED, wl.config_id, unit, KIND_EXP_AVG)


def key_exp_avg_sq(wl: Workload, unit: int) -> int:
    return stream_key(SEED, wl.config_id, unit, KIND_EXP_AVG_SQ)


def key_grad(wl: Workload, unit: int, rank: int, step: int) -> int:
    """A rank's full gradient of a unit (or of a gradient-pool slot) at a step."""
    return stream_key(SEED, wl.config_id, unit, KIND_GRAD, rank, step)


def key_shard(wl: Workload, unit: int) -> int:
    """bf16 parameters the other ranks contribute to the all-gather (local-rank mode)."""
    return stream_key(SEED, wl.config_id, unit, KIND_SHARD)
