"""Seeded synthetic workloads for the sharded optimizer step.

This module only describes inputs: unit-size lists, hyper-parameters and
seeded random tensors.  It holds none of the method's arithmetic (no layout,
no reduction, no update), so both the CUDA path and the CPU oracle may take
their inputs from it.

Gradient buffers are generated at full padded length; padding entries are
filled with random values too, because the step must ignore them.
"""
import math

import numpy as np
import torch

BF16, F32 = "bf16", "f32"


# ------------------------------------------------------------------ unit lists
def toy_units():
    """One unit of P = 1000 weights ("ZeRO and FSDP sharding", Code, main)."""
    return [1000]


def gpt2_block(d: int) -> int:
    """Parameters of one GPT-2 block of width d: attention 4d^2+4d, MLP 8d^2+5d, two LayerNorms 4d."""
    return 12 * d * d + 13 * d


def gpt2l_units():
    """GPT-2 Large (n_layer 36, n_embd 1280, vocab 50257, context 1024) wrapped per block:
    token embedding, 36 blocks, then position embedding + final LayerNorm.
    Psi = 774,030,080 ("ZeRO: Three Ledgers, Zero Redundancy", section 4: Psi = 0.774B)."""
    d = 1280
    return [50257 * d] + [gpt2_block(d)] * 36 + [1024 * d + 2 * d]


def gpt_1p3b_units():
    """24 GPT-2-style blocks of width 2048 plus the token embedding (Psi = 1,311,524,864)."""
    d = 2048
    return [50257 * d] + [gpt2_block(d)] * 24


def gated_block(d: int, ffn: int) -> int:
    """Attention 4d^2, gated MLP 3 d ffn, two norms 2d (no biases)."""
    return 4 * d * d + 3 * d * ffn + 2 * d


def llm_4b_units():
    """32 blocks of d=3072, ffn=8192 plus one embedding unit of 122,368 x 3072 (Psi = 3,999,989,760)."""
    d, ffn = 3072, 8192
    return [gated_block(d, ffn)] * 32 + [122368 * d]


def finewrap_units(n_units=4096, lo_log2=10, hi_log2=22, seed=4):
    """n_units sizes drawn log-uniformly from [2^lo, 2^hi): floor(2^(lo + (hi-lo) u)), u ~ U[0,1)."""
    u = np.random.default_rng(seed).random(n_units)
    return [int(math.floor(2.0 ** (lo_log2 + (hi_log2 - lo_log2) * x))) for x in u]


# ------------------------------------------------------------------ configurations
# lr/b1/b2/eps/wd are the pages' toy constants ("ZeRO and FSDP sharding", Code).
HP = dict(lr=0.01, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)

CONFIGS = {
    "toy": dict(desc="pages' toy ZeRO-2: N=4, P=1000, fp32 grads w-target, 50 steps, fp32 gather",
                units=toy_units, N=4, gdtype=F32, pdtype=F32, stage=2, steps=50, max_norm=0.0),
    "gpt2l": dict(desc="GPT-2-Large-shaped ZeRO-1: N=8, 38 units, Psi=774,030,080, bf16 grads N(0,1e-3)",
                  units=gpt2l_units, N=8, gdtype=BF16, pdtype=BF16, stage=1, steps=20, max_norm=0.0,
                  grad_sigma=1e-3, master_sigma=0.02),
    "1p3b_clip": dict(desc="1.3B ZeRO-2 + global-norm clip 1.0: N=8, 25 units, bf16 grads N(0,1e-2), "
                           "0.1% outliers x100, 10 steps",
                      units=gpt_1p3b_units, N=8, gdtype=BF16, pdtype=BF16, stage=2, steps=10, max_norm=1.0,
                      grad_sigma=1e-2, outlier_frac=1e-3, outlier_scale=100.0, master_sigma=0.02),
    "finewrap": dict(desc="fine-wrap stress: N=16, 4096 log-uniform units in [2^10, 2^22), bf16 grads N(0,1e-3)",
                     units=finewrap_units, N=16, gdtype=BF16, pdtype=BF16, stage=2, steps=3, max_norm=0.0,
                     grad_sigma=1e-3, master_sigma=0.02),
    "finewrap600": dict(desc="fine-wrap stress at the stated ~600M total: N=16, 4096 log-uniform units in "
                             "[2^10, 2^20) (same seed), Psi=638,561,671, bf16 grads N(0,1e-3)",
                        units=lambda: finewrap_units(hi_log2=20), N=16, gdtype=BF16, pdtype=BF16, stage=2, steps=3,
                        max_norm=0.0, grad_sigma=1e-3, master_sigma=0.02),
    "gpt2l_prof": dict(desc="profiling case: the first two GPT-2-Large units (token embedding + one block, "
                            "84,006,400 params), N=8, bf16 grads N(0,1e-3); 3.5 GB of traffic per step",
                       units=lambda: gpt2l_units()[:2], N=8, gdtype=BF16, pdtype=BF16, stage=1, steps=3, max_norm=0.0,
                       grad_sigma=1e-3, master_sigma=0.02),
    "1p3b_clip_prof": dict(desc="profiling case: two 1.3B blocks (100,716,544 params), N=8, clip 1.0, bf16 grads "
                                "N(0,1e-2) with 0.1% outliers x100; about 3.5 GB resident",
                           units=lambda: gpt_1p3b_units()[1:3], N=8, gdtype=BF16, pdtype=BF16, stage=2, steps=3,
                           max_norm=1.0, grad_sigma=1e-2, outlier_frac=1e-3, outlier_scale=100.0, master_sigma=0.02),
    "finewrap_prof": dict(desc="profiling case: 128 fine-wrap units (same law, seed 4), N=16, bf16 grads "
                               "N(0,1e-3); about 3 GB resident",
                          units=lambda: finewrap_units(n_units=128), N=16, gdtype=BF16, pdtype=BF16, stage=2, steps=3,
                          max_norm=0.0, grad_sigma=1e-3, master_sigma=0.02),
    "finewrap600_prof": dict(desc="profiling case: the first 512 units of finewrap600 (same law and seed, "
                                  "88,946,467 params), N=16, bf16 grads N(0,1e-3); about 4 GB resident",
                             units=lambda: finewrap_units(n_units=512, hi_log2=20), N=16, gdtype=BF16, pdtype=BF16,
                             stage=2, steps=3, max_norm=0.0, grad_sigma=1e-3, master_sigma=0.02),
    "4b_z3_prof": dict(desc="profiling case: one 4B block (d=3072, ffn=8192: 113,252,352 params), N=8, ZeRO-3, "
                            "bf16 grads N(0,1e-3); about 3.6 GB resident",
                       units=lambda: llm_4b_units()[:1], N=8, gdtype=BF16, pdtype=BF16, stage=3, steps=3,
                       max_norm=0.0, grad_sigma=1e-3, master_sigma=0.02),
    "beyond_2p32": dict(desc="index-width case: N=2, units of 2^31+3, 7, 2^31+2^24+5 and 1 elements "
                             "(4,311,744,532 padded positions: full positions beyond 2^32, shard positions "
                             "beyond 2^31), bf16 grads N(0,1e-2) with 0.1% outliers x100, clip 1.0; "
                             "about 103 GB resident with the ZeRO-3 param shards",
                        units=lambda: [2 ** 31 + 3, 7, 2 ** 31 + 2 ** 24 + 5, 1], N=2, gdtype=BF16, pdtype=BF16,
                        stage=2, steps=2, max_norm=1.0, grad_sigma=1e-2, outlier_frac=1e-3, outlier_scale=100.0,
                        master_sigma=0.02),
    "4b_z3": dict(desc="4B ZeRO-3: N=8, 33 units, bf16 grads N(0,1e-3), per-unit bf16 all-gather",
                  units=llm_4b_units, N=8, gdtype=BF16, pdtype=BF16, stage=3, steps=3, max_norm=0.0,
                  grad_sigma=1e-3, master_sigma=0.02),
}


# ------------------------------------------------------------------ tensors
def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def toy_targets(N=4, P=1000, device="cpu"):
    """target[r][i] = (7 i + 13 r) mod 11 as fp32 ("ZeRO and FSDP sharding", Code, main)."""
    i = torch.arange(P, device=device, dtype=torch.int64)
    return torch.stack([((i * 7 + r * 13) % 11).to(torch.float32) for r in range(N)])


def make_grads(n_ranks, length, dtype=BF16, sigma=1e-3, device="cpu", seed=1, outlier_frac=0.0,
               outlier_scale=1.0, out=None):
    """[n_ranks, length] gradient buffers; rank r draws N(0, sigma^2) from seed + r, and a
    Bernoulli(outlier_frac) subset is multiplied by outlier_scale.  Values are drawn in fp32
    and stored in `dtype` (round to nearest even by torch)."""
    tdt = torch.bfloat16 if dtype == BF16 else torch.float32
    if out is None:
        out = torch.empty(n_ranks, length, dtype=tdt, device=device)
    chunk = 1 << 28
    for r in range(n_ranks):
        gen = _gen(device, seed + r)
        for s in range(0, length, chunk):
            e = min(length, s + chunk)
            x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32) * sigma
            if outlier_frac > 0.0:
                mask = torch.rand(e - s, generator=gen, device=device) < outlier_frac
                x = torch.where(mask, x * outlier_scale, x)
            out[r, s:e].copy_(x)
            del x
    return out


def make_state(n_ranks, length, sigma=0.02, device="cpu", seed=1000, out=None):
    """Per-rank fp32 master ~ N(0, sigma^2) and zero m, v, each [n_ranks, length]
    (written into `out` = (master, m, v) when given)."""
    gen = _gen(device, seed)
    if out is None:
        out = tuple(torch.empty(n_ranks, length, dtype=torch.float32, device=device) for _ in range(3))
    master, m, v = out
    chunk = 1 << 28
    for r in range(n_ranks):
        for s in range(0, length, chunk):
            e = min(length, s + chunk)
            master[r, s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32) * sigma
    m.zero_()
    v.zero_()
    return master, m, v


def wide_range_f32(shape, seed, nonneg=False, subnormal_frac=0.3, wide_frac=0.3, sigma=1e-3):
    """Seeded fp32 values spanning the whole finite range, as a float32 numpy array.

    A subnormal_frac share has a zero exponent field (subnormals and zeros), a
    wide_frac share has an exponent field drawn uniformly from 1..254 (up to
    about 3.4e38), and the rest is N(0, sigma^2).  Signs are random unless
    nonneg.  Built from bit fields, so every value is finite."""
    rng = np.random.default_rng(seed)
    n = int(np.prod(shape))
    mant = rng.integers(0, 1 << 23, n, dtype=np.uint32)
    kind = rng.random(n)
    exp = rng.integers(1, 255, n, dtype=np.uint32)
    exp[kind < subnormal_frac] = 0
    bits = (exp << 23) | mant
    if not nonneg:
        bits |= rng.integers(0, 2, n, dtype=np.uint32) << 31
    x = bits.view(np.float32).copy()
    normal = kind >= subnormal_frac + wide_frac
    g = rng.normal(0.0, sigma, int(normal.sum()))
    x[normal] = (np.abs(g) if nonneg else g).astype(np.float32)
    return x.reshape(shape)
