"""Seeded synthetic inputs for the routed MoE expert layer.

This module is shared by the CUDA path's tests and bench and by the CPU
oracle. It holds the workload shapes and the input recipe only: it does no
routing, no expert arithmetic and no reduction of the layer.

Recipe (one CPU ``torch.Generator`` per workload, seed 0, drawn in this fixed
order): x, W_r, the expert rank permutation for the bias, W_gate, W_up, W_down,
dY. Every value is drawn in fp32; tensors stored as bf16 are round-to-nearest-
even casts of those fp32 draws.

* x  ~ N(0, 1)                       bf16 [T, d]
* W_r ~ N(0, 0.02)                   fp32 [d, E]   (std 0.02: the random-init
  convention of prime-rl PR #3885, §Changes, "debug.random_init")
* W_gate, W_up ~ N(0, 1/sqrt(d))     bf16 [E, d, f]
* W_down ~ N(0, 1/sqrt(f))           bf16 [E, f, d]
* dY ~ N(0, 1)                       bf16 [T, d]
* bias (skewed workloads only)       fp32 [E]: b_e = -tau * s * ln(r_e), with
  r = a seeded permutation of 1..E (a Zipf(s)-shaped popularity ranking) and
  tau read from ``zipf_tau.json`` (written by ``oracle/calibrate_zipf.py``).

Weights are never zero: zero-initialised weights make expert kernels run
unrealistically fast (prime-rl PR #3885, §Changes, "debug.random_init").
"""
from __future__ import annotations

import json
import math
import os
from dataclasses import dataclass, replace
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
TAU_FILE = os.path.join(_HERE, "zipf_tau.json")


@dataclass(frozen=True)
class Workload:
    """Shape of one MoE layer problem.

    T tokens of width d, E experts of ffn width f, top-k routing.
    ``zipf_s`` set -> a per-expert router bias that skews the load.
    ``align`` is the padding multiple of each expert's row group.
    """

    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    zipf_s: Optional[float] = None
    align: int = 128
    backward: bool = True
    seed: int = 0
    note: str = ""

    @property
    def P(self) -> int:
        """Token-expert pairs."""
        return self.T * self.k

    @property
    def R_cap(self) -> int:
        """Row capacity of the padded expert-grouped layout (an upper bound
        of sum_e ceil(n_e/align)*align that needs no knowledge of n_e)."""
        return self.P + self.E * (self.align - 1)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads. Shapes follow the pages' systems:
#  * GPT-OSS 20B on B300 (Halo "Performance", §Rough numbers: batch 4 x 4096),
#  * Qwen3-30B-A3B (Halo "Performance", §Levers that help, grouped GEMM row),
#  * a 512-expert top-10 layer of hidden size 2560 with 9.375 MiB bf16 experts
#    (PocketLLM "Qwen4-Exp Heterogeneous TP4 Performance", §Runtime
#    architecture), which fixes f = 640,
#  * small-M experts bound by weight bandwidth (Halo "Performance", §Levers
#    that do not help here).
CONFIGS = {
    "tiny": Workload("tiny", T=256, d=128, f=256, E=8, k=2,
                     note="tiny MoE layer, fits in L2: a correctness case"),
    "gptoss20b": Workload("gptoss20b", T=16384, d=2880, f=2880, E=32, k=4,
                          note="GPT-OSS-20B-shaped layer, batch 4 x 4096, near-uniform load"),
    "qwen3_30b": Workload("qwen3_30b", T=8192, d=2048, f=768, E=128, k=8, zipf_s=1.1,
                          note="Qwen3-30B-A3B-shaped layer, Zipf(1.1) router bias"),
    "fine512": Workload("fine512", T=8192, d=2560, f=640, E=512, k=10, zipf_s=1.2,
                        note="fine-grained 512-expert top-10 layer, Zipf(1.2) router bias"),
}
# a smaller case of the GPT-OSS-20B-shaped layer (one sequence of 4096 tokens)
# for ncu captures, whose replays save and restore device memory
CONFIGS["gptoss20b_T4096"] = Workload("gptoss20b_T4096", T=4096, d=2880, f=2880, E=32, k=4,
                                      note="GPT-OSS-20B-shaped layer, one 4096-token sequence")
# half the bench batch (2 x 4096 tokens, 1024 rows per expert): a profiling size
CONFIGS["gptoss20b_T8192"] = Workload("gptoss20b_T8192", T=8192, d=2880, f=2880, E=32, k=4,
                                      note="GPT-OSS-20B-shaped layer, batch 2 x 4096")
# the fine-grained expert shape (d = 2560, f = 640, top-10, ~160 rows per
# expert) over 128 experts instead of 512: a profiling size (a few GB on the device)
CONFIGS["fine_E128_T2048"] = Workload("fine_E128_T2048", T=2048, d=2560, f=640, E=128, k=10,
                                      note="fine-grained expert shape, 128 experts, 2048 tokens")
for _T in (128, 512, 1024, 2048):
    CONFIGS[f"smallm_T{_T}"] = Workload(
        f"smallm_T{_T}", T=_T, d=2048, f=768, E=128, k=8, backward=False,
        note="small-M weight-bound sweep, forward only")
# decode: one and eight tokens through the same layer shape (every selected
# expert's weights streamed for one or two rows)
for _T in (1, 8):
    CONFIGS[f"decode_T{_T}"] = Workload(
        f"decode_T{_T}", T=_T, d=2048, f=768, E=128, k=8, align=16, backward=False,
        note="decode, forward only")


def zipf_tau(name: str) -> float:
    """Bias temperature for a skewed workload, as calibrated on the oracle."""
    with open(TAU_FILE) as fh:
        table = json.load(fh)
    return float(table[name]["tau"])


def _normal(gen: torch.Generator, shape, std: float) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.float32)
    t.normal_(0.0, std, generator=gen)
    return t


def generate(wl: Workload, tau: Optional[float] = None, with_dy: bool = True,
             router_only: bool = False) -> dict:
    """Draw the inputs of ``wl`` on the CPU.

    Returns a dict of CPU tensors: x (bf16), w_router (fp32), bias (fp32 or
    None), w_gate, w_up, w_down (bf16), dy (bf16, when ``with_dy``), and
    ``tau`` (float or None). ``tau`` overrides the stored temperature (used by
    the calibration script). ``router_only`` stops after the bias (the draw
    order makes that prefix identical to a full draw).
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(wl.seed)
    out: dict = {}
    out["x"] = _normal(gen, (wl.T, wl.d), 1.0).to(torch.bfloat16)
    out["w_router"] = _normal(gen, (wl.d, wl.E), 0.02)
    if wl.zipf_s is not None:
        rank = torch.randperm(wl.E, generator=gen).to(torch.float64) + 1.0
        if tau is None:
            tau = zipf_tau(wl.name)
        out["bias"] = (-tau * wl.zipf_s * torch.log(rank)).to(torch.float32)
        out["tau"] = float(tau)
    else:
        out["bias"] = None
        out["tau"] = None
    if router_only:
        return out
    out["w_gate"] = _normal(gen, (wl.E, wl.d, wl.f), 1.0 / math.sqrt(wl.d)).to(torch.bfloat16)
    out["w_up"] = _normal(gen, (wl.E, wl.d, wl.f), 1.0 / math.sqrt(wl.d)).to(torch.bfloat16)
    out["w_down"] = _normal(gen, (wl.E, wl.f, wl.d), 1.0 / math.sqrt(wl.f)).to(torch.bfloat16)
    if with_dy:
        out["dy"] = _normal(gen, (wl.T, wl.d), 1.0).to(torch.bfloat16)
    return out


def generate_device(wl: Workload, device, with_dy: bool = True) -> dict:
    """Inputs for timing runs, with the large tensors drawn on the device.

    x, W_r and the bias are the CPU recipe's own (the prefix ``generate``
    draws first), so the routing, and with it every expert's row count, is
    the one the parity tests check. The expert weights and dY are drawn from
    the same distributions by a device generator seeded with ``wl.seed``
    (drawing billions of values on the host takes minutes; the kernels'
    timing does not depend on the values, only that they are not zero).
    Returns device tensors with the keys of ``generate``."""
    out = generate(wl, router_only=True)
    out = {k_: (v.to(device) if isinstance(v, torch.Tensor) else v) for k_, v in out.items()}
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed)

    def draw(shape, std):
        t = torch.empty(shape, dtype=torch.float32, device=device)
        t.normal_(0.0, std, generator=gen)
        return t.to(torch.bfloat16)

    out["w_gate"] = draw((wl.E, wl.d, wl.f), 1.0 / math.sqrt(wl.d))
    out["w_up"] = draw((wl.E, wl.d, wl.f), 1.0 / math.sqrt(wl.d))
    out["w_down"] = draw((wl.E, wl.f, wl.d), 1.0 / math.sqrt(wl.f))
    if with_dy:
        out["dy"] = draw((wl.T, wl.d), 1.0)
    return out


def stride97_topk(T: int, k: int, E: int) -> torch.Tensor:
    """Exactly balanced routing for the small-M variant: pair p = t*k + j goes
    to expert (97 * p) mod E (prime-rl PR #3885, §Changes, "Spread balanced
    routing": experts strided by 97). Returns int32 [T, k]."""
    p = torch.arange(T * k, dtype=torch.int64)
    return ((p * 97) % E).to(torch.int32).reshape(T, k)
