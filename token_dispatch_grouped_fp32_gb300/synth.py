"""Seeded synthetic inputs for one MoE layer forward.

This module only draws random tensors of the workloads' shapes; it holds none
of the layer's arithmetic.  The test suite and the benchmark use it to feed the
same bytes to the CUDA library and to the CPU oracle.

Workloads (all seeded; x ~ N(0, 1); router and expert weights ~ N(0, 1/d);
the tiny fp32 case draws its down projection from N(0, 1/f)):

=================  =====  ====  ===  ==  =====  =====  ======================
name               T      d     E    k   f      dtype  notes
=================  =====  ====  ===  ==  =====  =====  ======================
tiny_fp32          64     128   8    2   256    f32    parity case
mixtral            4096   4096  8    2   14336  bf16   Mixtral-8x7B shape
gptoss_decode      64     2880  128  4   2880   bf16   gpt-oss-120b, decode
gptoss_prefill     8192   2880  128  4   2880   bf16   gpt-oss-120b, prefill
qwen3_zipf         16384  2048  128  8   768    bf16   Zipf-skewed routing
deepseek           8192   7168  256  8   2048   bf16   DeepSeek-V3 routed experts
mixtral_norenorm   4096   4096  8    2   14336  bf16   top-k weights kept as
                                                       softmax probabilities
mixtral_dense      1024   4096  8    8   14336  bf16   k = E: the dense soft
                                                       mixture of all experts
=================  =====  ====  ===  ==  =====  =====  ======================

The router weight is always fp32 (E x d, nn.Linear layout).  The packed
gate/up weight is E x d x 2f (gate in the first f columns) and the down weight
E x f x d, both in the activation dtype.  Renormalised top-k weights except in
the two workloads that say otherwise.

Skewed routing (qwen3_zipf): a seeded random permutation gives each expert a
rank r in 1..E, and a per-expert logit offset 3 * r**-1.2 is added to the
router logits (rank 1 gets +3), so expert loads are heavily imbalanced.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    f: int
    dtype: str  # "f32" or "bf16"
    seed: int
    renorm: bool = True
    zipf: bool = False
    scale_inputs: bool = False  # routing weights on the expert inputs
    down_std_from_f: bool = False

    def with_tokens(self, T: int) -> "Workload":
        return replace(self, T=int(T))

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def pairs(self) -> int:
        return self.T * self.k


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_fp32", 64, 128, 8, 2, 256, "f32", 0, down_std_from_f=True),
        Workload("mixtral", 4096, 4096, 8, 2, 14336, "bf16", 1),
        Workload("gptoss_decode", 64, 2880, 128, 4, 2880, "bf16", 2),
        Workload("gptoss_prefill", 8192, 2880, 128, 4, 2880, "bf16", 3),
        Workload("qwen3_zipf", 16384, 2048, 128, 8, 768, "bf16", 4, zipf=True),
        Workload("deepseek", 8192, 7168, 256, 8, 2048, "bf16", 5),
        Workload("mixtral_norenorm", 4096, 4096, 8, 2, 14336, "bf16", 6, renorm=False),
        Workload("mixtral_dense", 1024, 4096, 8, 8, 14336, "bf16", 7, renorm=False),
    ]
}


def zipf_logit_bias(E: int, gen: torch.Generator, s: float = 1.2, top: float = 3.0):
    """Per-expert additive logit offset top * rank**-s over a random ranking."""
    perm = torch.randperm(E, generator=gen, device=gen.device)
    rank = torch.empty(E, dtype=torch.float64, device=gen.device)
    rank[perm] = torch.arange(1, E + 1, dtype=torch.float64, device=gen.device)
    return (top * rank.pow(-s)).to(torch.float32)


def make_inputs(w: Workload, device: str | torch.device = "cpu", weights: bool = True):
    """Draw (x, Wr, Wgu, Wd, bias) for workload ``w`` on ``device``.

    The draw order is fixed (x, Wr, Wgu, Wd, then the skew permutation), and
    each tensor is drawn in fp32 and then cast to the workload dtype, so a
    given (workload, seed, device type) always yields the same bytes.  With
    ``weights=False`` only x, Wr and bias are drawn (the router-only tests).
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    act = w.torch_dtype
    x = torch.randn(w.T, w.d, generator=gen, device=device).to(act)
    Wr = torch.randn(w.E, w.d, generator=gen, device=device) * (1.0 / w.d) ** 0.5
    Wgu = Wd = None
    if weights:
        Wgu = (torch.randn(w.E, w.d, 2 * w.f, generator=gen, device=device)
               * (1.0 / w.d) ** 0.5).to(act)
        dstd = (1.0 / w.f) ** 0.5 if w.down_std_from_f else (1.0 / w.d) ** 0.5
        Wd = (torch.randn(w.E, w.f, w.d, generator=gen, device=device) * dstd).to(act)
    bias = zipf_logit_bias(w.E, gen) if w.zipf else None
    return {"x": x.contiguous(), "Wr": Wr.contiguous(),
            "Wgu": None if Wgu is None else Wgu.contiguous(),
            "Wd": None if Wd is None else Wd.contiguous(), "bias": bias}


def make_expert_weights_chunked(w: Workload, device, chunk_experts: int = 8):
    """Like make_inputs' expert weights, but drawn expert-chunk by expert-chunk
    in fp32 so the fp32 temporaries stay small for the 20+ GB workloads.

    Uses its own generator stream (seed + 1000), so its bytes differ from
    make_inputs'; callers use one or the other for a given run.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed + 1000)
    act = w.torch_dtype
    Wgu = torch.empty(w.E, w.d, 2 * w.f, dtype=act, device=device)
    Wd = torch.empty(w.E, w.f, w.d, dtype=act, device=device)
    s_d = (1.0 / w.d) ** 0.5
    s_dn = (1.0 / w.f) ** 0.5 if w.down_std_from_f else s_d
    for e0 in range(0, w.E, chunk_experts):
        e1 = min(w.E, e0 + chunk_experts)
        Wgu[e0:e1] = (torch.randn(e1 - e0, w.d, 2 * w.f, generator=gen, device=device) * s_d).to(act)
        Wd[e0:e1] = (torch.randn(e1 - e0, w.f, w.d, generator=gen, device=device) * s_dn).to(act)
    return Wgu, Wd


def make_logits(T: int, E: int, seed: int, device="cpu", ties: str | None = None):
    """A seeded fp32 logit buffer [T, E] for the routing tests.

    ties=None: N(0, 1) entries.  ties="coarse": entries drawn from a handful
    of values so many rows hold exact ties.  ties="all_equal": every entry 0.5.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    if ties == "all_equal":
        return torch.full((T, E), 0.5, dtype=torch.float32, device=device)
    L = torch.randn(T, E, generator=gen, device=device)
    if ties == "coarse":
        L = torch.round(L * 2.0) / 2.0
    return L.contiguous()
