"""Seeded synthetic inputs for the MoE layer workloads.

This module is the one place both the CUDA path's callers and the CPU oracle draw
their inputs from.  It holds none of the layer's arithmetic (no routing, sorting,
quantisation or expert math): it only draws random numbers with a seeded
``torch.Generator`` and arranges them into the workloads' shapes.

Values depend on the device the generator runs on (torch's CPU and CUDA generators
produce different streams for the same seed), so a test that compares the two paths
draws once and hands the same tensors to both.

Workloads (shapes follow the pages' own test and validation shapes; the pages'
lm_eval / OLMoE runs need datasets and trained weights, which these stand in for):

* ``tiny``      T=64,  H=256,  I=512,  E=8,   K=2, BF16, no shared expert; logits N(0,1).
* ``mid``       T=512, H=2048, I=1408, E=64,  K=8, BF16; logits N(0,1) + 8 on experts
  0-3 (the MoonEP page's "--skew 8" at S=512, H=2048, top-8 of 64); each slot turned
  into padding (-1) with probability 0.1.
* ``decode``    T=128, H=7168, I=2048, E=256, K=8, one shared expert, FP8 E4M3 with
  128x128 weight / 1x128 activation block scales; logits i.i.d. U(0,1).
* ``prefill``   T=8192 tokens in a power-of-two bucket of 16384 rows (rows past 8192 are
  padding), H=7168, I=2048, E=256, K=8, one shared expert, BF16; logits N(0,1) plus a
  per-expert bias -1.1*ln(rank+1) over a seeded permutation rank (Zipf(1.1) popularity).
* ``prefill_small`` the prefill shapes with E=32 and T=2048 tokens in a 4096-row bucket
  (about 4 GB on the device), for hardware-counter profiles.
* ``decode_small`` the decode shapes with E=64 (2.8 GB of E4M3 weights), for
  hardware-counter profiles of the FP8 kernels.
* ``prefill_fq`` the prefill workload with the combine's constant-scale FP8
  fake-quant; the scale comes from a calibration batch drawn with seed + 1.
* ``prefill_fq4`` the same with the NVFP4 combine fake-quant (per-tensor scale 448*6/amax
  from the same calibration batch).

x ~ N(0, 1) in BF16.  Expert weights ~ N(0, std = 1/sqrt(fan_in)) in BF16 (fan_in = H for
the gate/up rows, I for the down rows); W13 holds gate rows [0, I) then up rows [I, 2I).
"""
import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int            # rows of the (possibly bucketed) batch
    T_valid: int      # real tokens; rows >= T_valid are padding
    H: int
    I: int
    E: int
    K: int
    shared: bool
    dtype: str        # "bf16" or "e4m3"
    logits: str       # "normal" | "skew" | "uniform" | "zipf"
    slot_pad: float   # probability that a slot is padding
    fake_quant: bool = False
    graph: bool = False
    fq_format: str = "e4m3"   # the combine fake-quant's format: "e4m3" or "nvfp4"


WORKLOADS = {
    "tiny": Workload("tiny", 64, 64, 256, 512, 8, 2, False, "bf16", "normal", 0.0),
    "mid": Workload("mid", 512, 512, 2048, 1408, 64, 8, False, "bf16", "skew", 0.1),
    "decode": Workload("decode", 128, 128, 7168, 2048, 256, 8, True, "e4m3", "uniform", 0.0),
    "prefill": Workload("prefill", 16384, 8192, 7168, 2048, 256, 8, True, "bf16", "zipf", 0.0),
    # prefill shapes with fewer experts and tokens (about 4 GB on the device): the case
    # full hardware-counter profiles are taken on
    "prefill_small": Workload("prefill_small", 4096, 2048, 7168, 2048, 32, 8, True, "bf16", "zipf", 0.0),
    # decode shapes with 64 experts (2.8 GB of E4M3 weights): the FP8 kernels' profiling case
    "decode_small": Workload("decode_small", 128, 128, 7168, 2048, 64, 8, True, "e4m3", "uniform", 0.0),
    "prefill_fq": Workload("prefill_fq", 16384, 8192, 7168, 2048, 256, 8, True, "bf16", "zipf",
                           0.0, fake_quant=True, graph=True),
    "prefill_fq4": Workload("prefill_fq4", 16384, 8192, 7168, 2048, 256, 8, True, "bf16", "zipf",
                            0.0, fake_quant=True, graph=True, fq_format="nvfp4"),
}


def scaled(w: Workload, **kw) -> Workload:
    """A copy of a workload with some sizes changed (for small test cases)."""
    return replace(w, **kw)


def _gen(device, seed, *tags):
    s = int(seed)
    for t in tags:
        s = (s * 1000003 + int(t)) % (2 ** 62)
    return torch.Generator(device=device).manual_seed(s)


def router_logits(w: Workload, seed: int, device="cpu") -> torch.Tensor:
    """float32 [T, E] router logits with the workload's distribution."""
    g = _gen(device, seed, 1)
    if w.logits == "uniform":
        return torch.rand(w.T, w.E, generator=g, device=device, dtype=torch.float32)
    l = torch.randn(w.T, w.E, generator=g, device=device, dtype=torch.float32)
    if w.logits == "skew":
        l[:, :4] += 8.0
    elif w.logits == "zipf":
        rank = torch.randperm(w.E, generator=g, device=device)
        bias = torch.tensor([-1.1 * math.log(r + 1.0) for r in range(w.E)],
                            dtype=torch.float32, device=device)
        l += bias[rank]
    return l


def hidden(w: Workload, seed: int, device="cpu") -> torch.Tensor:
    """BF16 [T, H] token activations, N(0, 1)."""
    g = _gen(device, seed, 2)
    return torch.randn(w.T, w.H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def slot_padding(w: Workload, seed: int, device="cpu") -> torch.Tensor:
    """bool [T, K]: True where a slot is turned into padding (probability slot_pad)."""
    g = _gen(device, seed, 3)
    u = torch.rand(w.T, w.K, generator=g, device=device)
    return u < w.slot_pad


def _normal_bf16(shape, std, g, device):
    return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def expert_w13(w: Workload, seed: int, e: int, device="cpu") -> torch.Tensor:
    """BF16 [2I, H] gate+up weights of routed expert e (e == E: the shared expert)."""
    return _normal_bf16((2 * w.I, w.H), 1.0 / math.sqrt(w.H), _gen(device, seed, 4, e), device)


def expert_w2(w: Workload, seed: int, e: int, device="cpu") -> torch.Tensor:
    """BF16 [H, I] down weights of routed expert e (e == E: the shared expert)."""
    return _normal_bf16((w.H, w.I), 1.0 / math.sqrt(w.I), _gen(device, seed, 5, e), device)


def expert_weights(w: Workload, seed: int, device="cpu"):
    """(w13 [E, 2I, H], w2 [E, H, I], shared_w13 [2I, H] | None, shared_w2 [H, I] | None)."""
    w13 = torch.empty(w.E, 2 * w.I, w.H, dtype=torch.bfloat16, device=device)
    w2 = torch.empty(w.E, w.H, w.I, dtype=torch.bfloat16, device=device)
    for e in range(w.E):
        w13[e] = expert_w13(w, seed, e, device)
        w2[e] = expert_w2(w, seed, e, device)
    s13 = expert_w13(w, seed, w.E, device) if w.shared else None
    s2 = expert_w2(w, seed, w.E, device) if w.shared else None
    return w13, w2, s13, s2


def bf16_bits(t: torch.Tensor):
    """A BF16 tensor's bit patterns as a numpy uint16 array (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
