"""Seeded synthetic inputs for the denoising step.

This module draws weights, caches and canvases; it holds none of the method's
arithmetic.  Both the device path and the CPU oracle take their inputs from
here.  Distributions (the one-layer synthetic stand-in):

* E, Wq, Wk, Wv, Wo, W1 ~ N(0, 1/d); W2 ~ N(0, 1/F)    (all stored [out][in])
* prefix K/V cache ~ N(0, 1), keys taken as already rotated
* alpha (per-position logit sharpness) = exp(U(ln 0.5, ln 64))
* canvas tokens uniform over [0, V); self-conditioning z = 0
* MoE (optional): router Wr ~ N(0, 1/d) for moe_hot experts and N(0, 1/d) / 64 for
  the rest; expert We1 ~ N(0, 1/d), We2 ~ N(0, 1/Fe)
* everything rounded to bf16 (round to nearest even) unless fp32 is asked for

Workloads are named by what they are, with their sizes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Dims:
    V: int
    d: int
    C: int
    B: int
    Hq: int
    Hkv: int
    hd: int
    F: int
    P: int          # prefix length in the cache when the step runs
    cap: int = 0    # cache capacity in rows (0: equal to P)
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    L: int = 1      # attention layers (Wq, Wk, Wv, Wo and the caches stacked [L, ...] when L > 1)
    n_exp: int = 0  # routed experts of the per-layer MoE FFN (0: no MoE)
    top_k: int = 0  # experts per token
    Fe: int = 0     # expert hidden width (the shared expert has the same shape)
    moe_hot: int = 0  # experts with full-spread router logits (0: all); the rest near zero

    def __post_init__(self):
        if self.cap == 0:
            object.__setattr__(self, "cap", self.P)

    @property
    def M(self) -> int:
        return self.B * self.C


# name -> (dims, seed, description)
WORKLOADS = {
    "tiny_v512_c16": (Dims(V=512, d=64, C=16, B=1, Hq=2, Hkv=1, hd=32, F=128, P=32), 0,
                      "tiny single step, V=512 d=64 C=16 P=32, 2 q / 1 kv heads, hd 32, FFW 128"),
    "step_v32k_c256_p2k": (Dims(V=32768, d=1024, C=256, B=1, Hq=8, Hkv=2, hd=128, F=1024, P=2048), 1,
                           "single step, V=32768 d=1024 C=256 P=2048, 8 q / 2 kv heads"),
    "loop_v262k_c256_p8k": (Dims(V=262144, d=2816, C=256, B=1, Hq=16, Hkv=8, hd=128, F=1024, P=8192), 2,
                            "annealed 48-step canvas loop, V=262144 d=2816 C=256 P=8192, 16 q / 8 kv heads"),
    "prefix_p131k_v32k_c256": (Dims(V=32768, d=1024, C=256, B=1, Hq=8, Hkv=8, hd=128, F=1024, P=131072), 3,
                               "attention-heavy single step, P=131072, 8 q / 8 kv heads, V=32768 d=1024"),
    "blocks_b8_v32k_p4k": (Dims(V=32768, d=1024, C=256, B=8, Hq=8, Hkv=2, hd=128, F=1024, P=4096,
                                cap=4096 + 4 * 256), 4,
                           "multi-block generation: 8 canvases x 4 blocks, P 4096 -> 5120"),
}


def workload(name: str) -> tuple[Dims, int]:
    d, s, _ = WORKLOADS[name]
    return d, s


def with_prefix(dims: Dims, P: int) -> Dims:
    return replace(dims, P=P, cap=max(dims.cap, P))


def make_weights(dims: Dims, seed: int, device="cpu", dtype=torch.bfloat16):
    """Model weights and prefix cache.  Returns a dict of tensors on `device`."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    kw = dict(generator=g, device=device, dtype=torch.float32)
    sd, sf = 1.0 / math.sqrt(dims.d), 1.0 / math.sqrt(dims.F)
    nq, nkv = dims.Hq * dims.hd, dims.Hkv * dims.hd

    def draw(shape, scale):
        t = torch.randn(shape, **kw)
        if scale != 1.0:
            t.mul_(scale)
        return t.to(dtype)

    L = dims.L
    lead = () if L == 1 else (L,)
    w = {}
    w["E"] = draw((dims.V, dims.d), sd)
    w["Wq"] = draw(lead + (nq, dims.d), sd)
    w["Wk"] = draw(lead + (nkv, dims.d), sd)
    w["Wv"] = draw(lead + (nkv, dims.d), sd)
    w["Wo"] = draw(lead + (dims.d, nq), sd)
    w["W1"] = draw((dims.F, dims.d), sd)
    w["W2"] = draw((dims.d, dims.F), sf)
    Kc = torch.zeros(lead + (dims.B, dims.Hkv, dims.cap, dims.hd), device=device, dtype=dtype)
    Vc = torch.zeros_like(Kc)
    if dims.P > 0:
        Kc[..., : dims.P, :] = draw(lead + (dims.B, dims.Hkv, dims.P, dims.hd), 1.0)
        Vc[..., : dims.P, :] = draw(lead + (dims.B, dims.Hkv, dims.P, dims.hd), 1.0)
    w["Kc"], w["Vc"] = Kc, Vc
    if dims.n_exp > 0:
        # router rows of the "hot" experts ~ N(0, 1/d) (logits of unit spread), the other
        # experts' rows scaled by 1/64 (logits near zero, rarely in a top-k): a canvas then
        # activates about moe_hot experts; experts W1 ~ N(0, 1/d), W2 ~ N(0, 1/Fe), expert
        # index n_exp being the shared expert
        NE = dims.n_exp
        Wr = torch.randn(lead + (NE, dims.d), **kw).mul_(sd)
        We1 = draw(lead + (NE + 1, dims.Fe, dims.d), sd)
        We2 = draw(lead + (NE + 1, dims.d, dims.Fe), 1.0 / math.sqrt(dims.Fe))
        hot = dims.moe_hot if 0 < dims.moe_hot < NE else NE
        if hot < NE:
            cold = torch.randperm(NE, generator=g, device=device)[hot:]
            Wr[..., cold, :] *= 1.0 / 64
        w["Wr"], w["We1"], w["We2"] = Wr.to(dtype), We1, We2
    return w


def make_canvas(dims: Dims, seed: int, device="cpu", dtype=torch.bfloat16, alpha_range=(0.5, 64.0)):
    """Canvas tokens x [B, C] int32, z [B, C, d] zeros, alpha [B, C] float32."""
    g = torch.Generator(device=device).manual_seed(int(seed) + 7919)
    x = torch.randint(0, dims.V, (dims.B, dims.C), generator=g, device=device, dtype=torch.int64)
    lo, hi = math.log(alpha_range[0]), math.log(alpha_range[1])
    u = torch.rand((dims.B, dims.C), generator=g, device=device, dtype=torch.float32)
    alpha = torch.exp(lo + (hi - lo) * u)
    z = torch.zeros((dims.B, dims.C, dims.d), device=device, dtype=dtype)
    return x.to(torch.int32), z, alpha


def to_numpy_f32(w: dict) -> dict:
    """float32 numpy copies (exact for bf16 values) for the oracle."""
    return {k: v.detach().to("cpu", torch.float32).numpy() for k, v in w.items()}
