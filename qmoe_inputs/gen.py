"""Seeded input generators for the NVFP4 W4A16 MoE layer.

Workloads follow the synthetic recipes of the NVFP4 MoE pages (DeepSeek-class
decode and prefill shapes): activations x ~ N(0, 1) rounded to bf16, router
logits ~ N(0, 1) with top-k by value and a softmax over the chosen k, and expert
weights ~ N(0, 0.02) encoded to NVFP4 per expert matrix.  The skewed prefill
recipe draws each token's k experts without replacement from a Zipf(1.2) law over
a random permutation of the experts (Gumbel-top-k, slot order = draw order) and
takes routing weights as a softmax of N(0, 1) over the k slots.

NVFP4 encoding of one expert matrix W [N][K] (fp32), applied per expert:
  gscale = amax|W| / (6 * 448)
  scale  = E4M3 round-to-nearest-even of (amax of the 16-element K block) / 6 / gscale,
           saturated at 448; a block whose scale is 0 gets all-zero codes
  code   = nearest E2M1 value of W / (scale * gscale), ties to the even code,
           saturated at 6, sign kept (a negative zero is stored as +0)
  bytes  = two codes per byte along K, the even K element in the low nibble.

The generators run with torch on any device; the same bytes feed the CPU oracle
and the GPU kernels, so nothing here can affect parity.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    M: int
    H: int
    I: int
    E: int
    top_k: int
    seed: int
    routing: str = "softmax"  # "softmax" (top-k of N(0,1) logits) or "zipf"
    zipf_s: float = 1.2


CONFIGS = [
    LayerConfig("tiny_m4_h256_i128_e8_k2", 4, 256, 128, 8, 2, 0),
    LayerConfig("decode_m16_h7168_i2048_e256_k8", 16, 7168, 2048, 256, 8, 1),
    LayerConfig("decode_m1_h7168_i3072_e32_k8", 1, 7168, 3072, 32, 8, 2),
    LayerConfig("prefill_zipf_m2048_h4096_i1536_e128_k8", 2048, 4096, 1536, 128, 8, 3, "zipf"),
    LayerConfig("prefill_m8192_h7168_i2048_e256_k8", 8192, 7168, 2048, 256, 8, 4),
]


# Smaller cases of the same kernels for profiler captures (inputs still larger than L2).
PROFILE_CONFIGS = [
    LayerConfig("decode_m16_h7168_i2048_e32_k8", 16, 7168, 2048, 32, 8, 1),
    LayerConfig("prefill_m1024_h7168_i2048_e16_k8", 1024, 7168, 2048, 16, 8, 4),
]


@dataclasses.dataclass
class LayerInputs:
    cfg: LayerConfig
    x: torch.Tensor             # [M][H] bf16
    topk_ids: torch.Tensor      # [M][top_k] int32
    topk_weights: torch.Tensor  # [M][top_k] fp32
    w13: torch.Tensor           # [E][2I][H/2] uint8
    s13: torch.Tensor           # [E][2I][H/16] uint8 (E4M3 bits)
    gs13: torch.Tensor          # [E] fp32
    w2: torch.Tensor            # [E][H][I/2] uint8
    s2: torch.Tensor            # [E][H][I/16] uint8 (E4M3 bits)
    gs2: torch.Tensor           # [E] fp32

    def to(self, device) -> "LayerInputs":
        kw = {f.name: getattr(self, f.name) for f in dataclasses.fields(self)}
        for k, v in kw.items():
            if isinstance(v, torch.Tensor):
                kw[k] = v.to(device)
        return LayerInputs(**kw)


# E2M1 encoding boundaries on |w| / (scale * gscale).  A value exactly on a
# boundary goes to the code with an even mantissa bit: 0.25 -> 0, 0.75 -> 1.0,
# 1.25 -> 1.0, 1.75 -> 2.0, 2.5 -> 2.0, 3.5 -> 4.0, 5.0 -> 4.0.
_BOUNDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)
_TIE_GOES_UP = (False, True, False, True, False, True, False)


def _e2m1_encode(r: torch.Tensor) -> torch.Tensor:
    """Nearest-E2M1 code (4 bits, sign in bit 3) of real values r, ties to even."""
    a = r.abs()
    mag = torch.zeros_like(a, dtype=torch.int32)
    for b, up in zip(_BOUNDS, _TIE_GOES_UP):
        mag += (a >= b).int() if up else (a > b).int()
    neg = (r < 0) & (mag > 0)
    return (mag | (neg.int() << 3)).to(torch.uint8)


def quantize_nvfp4(w: torch.Tensor):
    """Encode one fp32 matrix [N][K] to (codes [N][K/2] u8, scales [N][K/16] u8, gscale)."""
    n, k = w.shape
    assert k % 16 == 0
    w = w.float()
    amax = w.abs().max()
    gscale = (amax / (6.0 * 448.0)).float()
    if float(gscale) == 0.0:
        gscale = torch.ones((), dtype=torch.float32, device=w.device)
    blk = w.view(n, k // 16, 16)
    bmax = blk.abs().amax(dim=-1)
    sreal = (bmax / 6.0 / gscale).clamp(max=448.0)
    s8 = sreal.to(torch.float8_e4m3fn)
    sdec = s8.float()
    denom = (sdec * gscale).unsqueeze(-1)
    r = torch.where(denom > 0, blk / torch.where(denom > 0, denom, torch.ones_like(denom)),
                    torch.zeros_like(blk))
    codes = _e2m1_encode(r).view(n, k)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()
    return packed, s8.view(torch.uint8).contiguous(), gscale.reshape(())


def _routing(cfg: LayerConfig, g: torch.Generator, device):
    M, E, k = cfg.M, cfg.E, cfg.top_k
    if cfg.routing == "softmax":
        logits = torch.randn(M, E, generator=g, device=device)
        vals, ids = torch.topk(logits, k, dim=1)
        wts = torch.softmax(vals, dim=1)
    elif cfg.routing == "zipf":
        perm = torch.randperm(E, generator=g, device=device)
        ranks = torch.arange(1, E + 1, device=device, dtype=torch.float64)
        logp_rank = (-cfg.zipf_s * torch.log(ranks)).float()
        logp = torch.empty(E, device=device)
        logp[perm] = logp_rank
        u = torch.rand(M, E, generator=g, device=device).clamp_(1e-20, 1.0 - 1e-7)
        gumbel = -torch.log(-torch.log(u))
        _, ids = torch.topk(logp.unsqueeze(0) + gumbel, k, dim=1)
        wts = torch.softmax(torch.randn(M, k, generator=g, device=device), dim=1)
    else:
        raise ValueError(cfg.routing)
    return ids.to(torch.int32).contiguous(), wts.float().contiguous()


def expert_seed(seed: int, e: int) -> int:
    """Seed of expert e's weight draws: each expert has its own stream, so any subset
    of experts can be generated alone with the same bytes."""
    return (seed + 1) * 1_000_003 + 7919 * (e + 1)


def make_inputs(cfg: LayerConfig, device="cpu", seed: Optional[int] = None,
                weight_std: float = 0.02, token_seed: Optional[int] = None,
                experts=None) -> LayerInputs:
    """Draw one layer's inputs with the config's recipe on `device`.

    `token_seed` (default: the config seed) seeds x and the routing; weights are
    drawn per expert from expert_seed(seed, e).  With `experts` given, only those
    experts' weights are drawn and the others are left as zero bytes."""
    device = torch.device(device)
    seed = cfg.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(seed if token_seed is None else token_seed)
    M, H, I, E = cfg.M, cfg.H, cfg.I, cfg.E
    x = torch.randn(M, H, generator=g, device=device).to(torch.bfloat16)
    ids, wts = _routing(cfg, g, device)
    w13 = torch.zeros(E, 2 * I, H // 2, dtype=torch.uint8, device=device)
    s13 = torch.zeros(E, 2 * I, H // 16, dtype=torch.uint8, device=device)
    w2 = torch.zeros(E, H, I // 2, dtype=torch.uint8, device=device)
    s2 = torch.zeros(E, H, I // 16, dtype=torch.uint8, device=device)
    gs13 = torch.ones(E, dtype=torch.float32, device=device)
    gs2 = torch.ones(E, dtype=torch.float32, device=device)
    for e in (range(E) if experts is None else sorted(set(int(v) for v in experts))):
        ge = torch.Generator(device=device)
        ge.manual_seed(expert_seed(seed, e))
        wa = torch.randn(2 * I, H, generator=ge, device=device) * weight_std
        w13[e], s13[e], gs13[e] = quantize_nvfp4(wa)
        del wa
        wb = torch.randn(H, I, generator=ge, device=device) * weight_std
        w2[e], s2[e], gs2[e] = quantize_nvfp4(wb)
        del wb
    return LayerInputs(cfg, x.contiguous(), ids, wts, w13, s13, gs13, w2, s2, gs2)


def config_by_name(name: str) -> LayerConfig:
    for c in CONFIGS + PROFILE_CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)
