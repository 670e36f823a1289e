"""Synthetic workloads shaped like the pages' examples (harness only).

Each workload fixes: the tensor list that is flattened, the number N of
simulated data-parallel ranks (N resident gradient replicas on one GPU), the
bucket size in elements, the gradient format, the gradient recipe for the
seeded generator, the optimizer hyperparameters and the number of steps.
All values are synthetic; no dataset or trained weights are involved.
"""
from dataclasses import dataclass, field, replace
from typing import List, Optional, Tuple


def gpt2_small_numels() -> List[int]:
    """GPT-2 small (124M) parameter list in module order: token and position
    embeddings, 12 blocks of (ln_1 w/b, qkv w/b, attn proj w/b, ln_2 w/b,
    mlp fc w/b, mlp proj w/b), final layer norm w/b."""
    d, v, ctx = 768, 50257, 1024
    out = [v * d, ctx * d]
    for _ in range(12):
        out += [d, d, d * 3 * d, 3 * d, d * d, d, d, d, d * 4 * d, 4 * d, 4 * d * d, d]
    out += [d, d]
    return out


def llama_2b_numels() -> List[int]:
    """Llama-style list: tied embedding 128256 x 2048, 16 blocks of
    (attention RMSNorm, q, k, v, o 2048 x 2048, MLP RMSNorm, gate, up
    2048 x 8192, down 8192 x 2048), final RMSNorm."""
    d, v, f = 2048, 128256, 8192
    out = [v * d]
    for _ in range(16):
        out += [d, d * d, d * d, d * d, d * d, d, d * f, d * f, f * d]
    out += [d]
    return out


@dataclass
class Workload:
    name: str
    numels: List[int]
    n_ranks: int
    bucket_elems: int = 0
    is_bf16: bool = True
    seed: int = 0
    sigma: float = 1e-3
    bias_sigma: float = 0.0
    outliers: bool = False
    init_scale: float = 1.0
    dynamic_scale: bool = False
    growth_interval: int = 2000
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    max_grad_norm: float = 0.0
    steps: int = 3
    rank_lo: int = 0
    rank_hi: Optional[int] = None           # None = all ranks
    # (step, rank, element, 16-bit pattern) written into one replica element
    # (of the step's last micro-batch)
    inject: Optional[Tuple[int, int, int, int]] = None
    # micro-batches per optimizer step, accumulated in fp32 before the reduce
    n_micro: int = 1

    @property
    def psi(self) -> int:
        return sum(self.numels)

    @property
    def ranks(self) -> Tuple[int, int]:
        return self.rank_lo, (self.n_ranks if self.rank_hi is None else self.rank_hi)

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)

    def gen_step(self, step: int, micro: int) -> int:
        """Generator step index of micro-batch `micro` (1-based) of optimizer
        step `step`: the step itself when there is one micro-batch."""
        return step if self.n_micro == 1 else step * 64 + micro


FP16_POS_INF = 0x7C00
BF16_POS_INF = 0x7F80

# A 1,000,003-parameter flat model (odd, forces padding), 4 ranks, fp16
# gradients with a static loss scale of 1024, 3 steps.
TINY_FLAT = Workload("tiny_flat_1M_n4_fp16", [1_000_003], 4, 0, False, 0, 1e-3,
                     init_scale=1024.0, steps=3)

# GPT-2 small list, 8 ranks, 25M-element buckets, bf16, 10 steps.
GPT2_SMALL = Workload("gpt2_small_124M_n8_bf16", gpt2_small_numels(), 8, 25_000_000, True,
                      1, 1e-3, steps=10)

# 1.5B flat parameters, 8 ranks, fp16 gradients N(0,1e-4) under a dynamic loss
# scale starting at 65536, global-norm clip 1.0, 5 steps; step 3 puts +inf in
# rank 5's gradient at element floor(psi/3).
FLAT_1P5B = Workload("flat_1p5B_n8_fp16_clip", [1_500_000_000], 8, 0, False, 2, 1e-4,
                     init_scale=65536.0, dynamic_scale=True, max_grad_norm=1.0, steps=5,
                     inject=(3, 5, 1_500_000_000 // 3, FP16_POS_INF))

# Rank 0's owned slice (137,656,250 elements) of an 8.81B-parameter model at
# 64 ranks: 64 bf16 replicas of the slice, N(0,1e-3) plus a per-rank bias
# N(0,1e-5), 5 steps.
STAGE3_SLICE = Workload("stage3_slice_8p81B_n64_bf16", [8_810_000_000], 64, 0, True, 3, 1e-3,
                        bias_sigma=1e-5, steps=5, rank_lo=0, rank_hi=1)

# Llama-style 1.34B list, 16 ranks, 50M-element buckets, bf16 with 0.1%
# outliers x100, global-norm clip 1.0, weight decay 0.1, 5 steps.
LLAMA_2B = Workload("llama_2B_n16_bf16_clip", llama_2b_numels(), 16, 50_000_000, True, 4,
                    1e-3, outliers=True, weight_decay=0.1, max_grad_norm=1.0, steps=5)

ALL = [TINY_FLAT, GPT2_SMALL, FLAT_1P5B, STAGE3_SLICE, LLAMA_2B]


# ------------------------------------------------------ stage-3 FSDP units ----

@dataclass
class UnitWorkload:
    """A tensor list wrapped into stage-3 FSDP units (forward order), the
    number N of simulated ranks and the unit alignment grain in elements."""
    name: str
    numels: List[int]
    unit_of_tensor: List[int]
    n_units: int
    n_ranks: int
    align_elems: int = 1
    seed: int = 0


def _blocks_with_root(numels: List[int], root: List[int], per_block: int) -> Tuple[List[int], int]:
    """Unit ids for a list laid out as root tensors + equal blocks: unit 0 is
    the root (embeddings, final norm, head), unit b + 1 is block b."""
    uot = []
    body = [k for k in range(len(numels)) if k not in root]
    assert len(body) % per_block == 0
    ids = {}
    for i, k in enumerate(body):
        ids[k] = 1 + i // per_block
    for k in range(len(numels)):
        uot.append(0 if k in root else ids[k])
    return uot, 1 + len(body) // per_block


def gpt2_small_units(n_ranks=8, align_elems=1) -> UnitWorkload:
    """GPT-2 small: one unit per transformer block, the root unit holding the
    token and position embeddings and the final layer norm."""
    numels = gpt2_small_numels()
    uot, n_units = _blocks_with_root(numels, [0, 1, len(numels) - 2, len(numels) - 1], 12)
    return UnitWorkload("gpt2_small_124M_units_n%d_a%d" % (n_ranks, align_elems), numels, uot,
                        n_units, n_ranks, align_elems, seed=5)


def llama_2b_units(n_ranks=16, align_elems=1) -> UnitWorkload:
    """The Llama-style list: one unit per block, the root unit holding the
    tied embedding and the final norm."""
    numels = llama_2b_numels()
    uot, n_units = _blocks_with_root(numels, [0, len(numels) - 1], 9)
    return UnitWorkload("llama_2B_units_n%d_a%d" % (n_ranks, align_elems), numels, uot, n_units,
                        n_ranks, align_elems, seed=6)


def stage3_8p81b_units(n_ranks=64, align_elems=1) -> UnitWorkload:
    """The 8.81B-parameter data-parallel share at 64 ranks, wrapped one block
    per unit: blocks of 110,000,000 parameters (220 MB gathered in BF16) and
    a root unit with the remaining 10,000,000 (80 blocks + root = 8.81e9)."""
    numels = [10_000_000] + [110_000_000] * 80
    return UnitWorkload("stage3_8p81B_units_n%d_a%d" % (n_ranks, align_elems), numels,
                        list(range(81)), 81, n_ranks, align_elems, seed=7)
