"""Seeded synthetic inputs for the attention workloads.

This module holds no attention arithmetic: it only draws random tensors, so both
the oracle side (tests) and the CUDA side may use it.

Recipe (all workloads): a CPU ``torch.Generator`` seeded with ``seed``; fp32
standard normal draws in the order Q, K, V, dO; each then rounded to bf16
(round to nearest even).  Layout ``[B, N, H, d]``.  The grouped-query workload
adds outliers: one channel index c in [0, d) is drawn by a CPU generator of its
own seeded with the same seed (``outlier_channel``: channel 44 for seed 0 and
d = 128), and Q[..., c] and K[..., c] are multiplied by 20 before the bf16
rounding (1% of d=128 channels, rounded to one channel, shared by all heads and
tokens).

Large workloads can be drawn on the GPU instead (``device='cuda'``, a CUDA
generator with the same seed); those values differ from the CPU draws and are
used only where the reference values are computed from the very same tensors.
"""

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    outliers: bool = False
    seed: int = 0
    decode: bool = False
    window: tuple = None  # (left, right): query i sees keys i - left .. i + right (negative: unbounded)
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def scale(self):
        return 1.0 / (self.d ** 0.5)


# The five workloads of the benchmark plan, by what they are.
TINY = Workload("tiny_b1_h1_n256_d64", 1, 1, 1, 256, 256, 64, False)
MHA_N2048_D64 = Workload("mha_b4_h16_n2048_d64", 4, 16, 16, 2048, 2048, 64, False)
CAUSAL_N4096_D128 = Workload("causal_b2_h16_n4096_d128", 2, 16, 16, 4096, 4096, 128, True)
GQA_N8192_D128 = Workload("gqa_causal_b1_hq32_hkv8_n8192_d128_outliers", 1, 32, 8, 8192, 8192, 128,
                          True, outliers=True)
DECODE_Q1 = Workload("decode_b8_hq32_hkv8_q1_kv131072_d128", 8, 32, 8, 1, 131072, 128, False, decode=True)
DECODE_Q4 = Workload("decode_b8_hq32_hkv8_q4_kv131072_d128", 8, 32, 8, 4, 131072, 128, False, decode=True)
# Causal sliding window: every query sees itself and the 4095 keys before it.
WINDOW_N16384_W4096 = Workload("window_causal_b1_hq32_hkv8_n16384_w4096_d128", 1, 32, 8, 16384, 16384, 128,
                               True, window=(4095, 0))

# Packed variable-length sequences (SFT-like, long-tailed lengths): extra["n_seqs"]
# sequences, lengths varlen_lengths(n_seqs, Nq, seed), in [total, H, d] tensors, causal.
VARLEN_T32768_D128 = Workload("varlen_causal_b24_hq32_hkv8_total32768_d128", 1, 32, 8, 32768, 32768, 128, True,
                              extra={"n_seqs": 24})

# Block-sparse: each 128-row query tile lists its own key tile, the seven before it
# and tile 0 (a local window plus a global prefix), causal.
BLOCKSPARSE_N16384 = Workload("blocksparse_causal_b1_hq32_hkv8_n16384_d128_local8_global1", 1, 32, 8, 16384, 16384,
                              128, True, extra={"local_tiles": 8, "global_tiles": 1})

ALL = [TINY, MHA_N2048_D64, CAUSAL_N4096_D128, GQA_N8192_D128, DECODE_Q1, DECODE_Q4, WINDOW_N16384_W4096,
       VARLEN_T32768_D128, BLOCKSPARSE_N16384]


def local_global_tiles(n_tiles, local, glob):
    """Block table of the local + global pattern: query tile i lists key tiles
    max(0, i - local + 1) .. i and 0 .. glob - 1 (as a [n_tiles, n_tiles] bool list of lists)."""
    return [[(i - local < j <= i) or (j < glob and j <= i) for j in range(n_tiles)] for i in range(n_tiles)]


def varlen_lengths(n_seqs, total, lo=64, hi=8192, seed=0):
    """n_seqs lengths summing to ``total``, long-tailed: Pareto(1.2) draws of a CPU
    generator seeded with ``seed``, scaled and clipped to [lo, hi], the rounding
    remainder spread over the sequences below hi."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    u = torch.rand(n_seqs, generator=gen, dtype=torch.float64)
    raw = (1.0 - u) ** (-1.0 / 1.2)                            # Pareto(1.2) on [1, inf)
    lens = [int(min(hi, max(lo, round(float(r) * total / float(raw.sum()))))) for r in raw]
    i = 0
    while sum(lens) != total:                                  # fix the rounding, one token at a time
        step = 1 if sum(lens) < total else -1
        if lo <= lens[i] + step <= hi:
            lens[i] += step
        i = (i + 1) % n_seqs
    return lens


def make(w, device="cpu", with_do=True, seed=None):
    """Draw (q, k, v, do) bf16 tensors for workload ``w`` on ``device``.

    Returns a dict with keys q, k, v, do (do is None when ``with_do`` is False
    or for decode workloads), and ``outlier_channel`` (int or None).
    """
    seed = w.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def draw(n, h):
        return torch.randn((w.B, n, h, w.d), generator=gen, dtype=torch.float32, device=device)

    q = draw(w.Nq, w.Hq)
    k = draw(w.Nk, w.Hkv)
    v = draw(w.Nk, w.Hkv)
    do = draw(w.Nq, w.Hq) if (with_do and not w.decode) else None
    ch = None
    if w.outliers:
        ch = outlier_channel(w.d, seed)
        q[..., ch] *= 20.0
        k[..., ch] *= 20.0
    out = {
        "q": q.to(torch.bfloat16),
        "k": k.to(torch.bfloat16),
        "v": v.to(torch.bfloat16),
        "do": None if do is None else do.to(torch.bfloat16),
        "outlier_channel": ch,
    }
    return out


def outlier_channel(d, seed=0):
    """The outlier channel of a workload: one index in [0, d) drawn by its own CPU
    generator seeded with ``seed``, so every draw of the workload (CPU or CUDA
    tensors, with or without dO) scales the same channel."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    return int(torch.randint(0, d, (1,), generator=gen).item())


def hadamard_signs(d, seed=0):
    """d random signs (+1.0 / -1.0, float32) for the random Hadamard rotation: a CPU
    generator seeded with ``seed`` draws d bits."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    bits = torch.randint(0, 2, (d,), generator=gen)
    return (1.0 - 2.0 * bits).to(torch.float32)


def shape_inputs(B, Hq, Hkv, Nq, Nk, d, seed=0, device="cpu", with_do=True):
    """Draw (q, k, v, do) for an arbitrary shape with the same recipe (no outliers)."""
    w = Workload("custom", B, Hq, Hkv, Nq, Nk, d, False, seed=seed)
    return make(w, device=device, with_do=with_do)
