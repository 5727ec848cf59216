"""Seeded synthetic inputs for the LatentMoE layer forward.

This module only draws random tensors of the right shapes, scales and
dtypes. It holds none of the layer's arithmetic, so the CUDA path and the
float64 oracle can both be fed from it without sharing any computation.

Shapes follow the layer statement on the pages:
- MAI-Base-1 shape ("The Training and RL Infrastructure Behind
  MAI-Thinking-1", section "The model the systems run", MoE row): hidden
  6656, latent 3072, 512 experts, top-8, expert FFN 10240.
- MAI-Base-2 shape ("MAI-Base-2: Microsoft's 2.8T base model, and whether
  its compute numbers add up", section "The model"): hidden 8704, latent
  4096, top-7 plus one shared expert that is not down/up projected. The
  expert count is reduced from 512 to 256 to fit one GPU, and the expert and
  shared FFN widths (10240) are assumed, since the pages do not give them.

Every tensor comes from its own ``torch.Generator`` whose seed is derived
from (base seed, tensor name, expert index), so one expert's weights can be
regenerated on their own. CPU and CUDA generators produce different
streams: a test that compares the two paths generates once and hands the
same tensors to both.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int          # tokens
    d: int          # hidden width
    l: int          # latent width
    E: int          # routed experts
    k: int          # experts per token
    F: int          # expert FFN width
    Fs: int = 0     # shared-expert FFN width (0 = no shared expert)
    router_std: Optional[float] = None   # None: N(0, 1/d) like every other weight
    zipf_bias: bool = False              # per-expert router bias for skewed loads

    @property
    def slots(self) -> int:
        return self.T * self.k


CONFIGS: Dict[str, LayerConfig] = {
    "tiny": LayerConfig("tiny", T=128, d=256, l=128, E=16, k=2, F=256),
    "mid": LayerConfig("mid", T=4096, d=2048, l=1024, E=64, k=4, F=2048,
                       router_std=0.02),
    "imbalanced": LayerConfig("imbalanced", T=4096, d=2048, l=1024, E=64, k=4,
                              F=2048, router_std=0.02, zipf_bias=True),
    "mai-base-1": LayerConfig("mai-base-1", T=16384, d=6656, l=3072, E=512,
                              k=8, F=10240),
    "mai-base-2": LayerConfig("mai-base-2", T=8192, d=8704, l=4096, E=256,
                              k=7, F=10240, Fs=10240),
    # 1/16 of the MAI-Base-1 layer (32 experts, 1024 tokens): same widths and
    # the same ~256 slots per expert, ~6 GB of weights; small enough for a
    # full profiler capture.
    "mai-base-1-slice": LayerConfig("mai-base-1-slice", T=1024, d=6656, l=3072,
                                    E=32, k=8, F=10240),
    # 1/16 of the MAI-Base-2-like layer (16 experts, 512 tokens) with its
    # full-width shared expert: the profiler proxy for that shape.
    "mai-base-2-slice": LayerConfig("mai-base-2-slice", T=512, d=8704, l=4096,
                                    E=16, k=7, F=10240, Fs=10240),
    # MAI-Base-1's dense GEMMs at full size (T=16384, d=6656, l=3072) with 8
    # tiny experts (F=256, every token on all of them): ~3 GB on the device,
    # the profiler proxy for the down- and up-projection kernels.
    "mai-base-1-dense": LayerConfig("mai-base-1-dense", T=16384, d=6656, l=3072, E=8, k=8,
                                    F=256),
    # The same for the MAI-Base-2-like layer with its full-width shared expert
    # (T=8192, d=8704, l=4096, F_s=10240).
    "mai-base-2-dense": LayerConfig("mai-base-2-dense", T=8192, d=8704, l=4096, E=8, k=7,
                                    F=256, Fs=10240),
    # The MAI-Base-1 router at full size (T=16384, d=6656, E=512, top-8) with
    # 128-wide experts: the profiler proxy for the router kernel alone.
    "mai-base-1-router": LayerConfig("mai-base-1-router", T=16384, d=6656, l=128,
                                     E=512, k=8, F=128),
}


def derive_seed(base: int, name: str, index: int = -1) -> int:
    """A 63-bit seed from (base, tensor name, index); stable across runs."""
    h = zlib.crc32(f"{base}:{name}:{index}".encode())
    return (base * 1_000_003 + h * 2_654_435_761 + index + 1) & ((1 << 63) - 1)


def _gen(device: torch.device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, seed: int, device) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 on ``device`` and rounded to bf16 (RNE)."""
    device = torch.device(device)
    t = torch.randn(shape, generator=_gen(device, seed), device=device,
                    dtype=torch.float32)
    return t.mul_(std).to(torch.bfloat16)


def zipf_router_bias(E: int, seed: int) -> torch.Tensor:
    """b_e = 1.5 * ln(1 / rank_e^1.2), rank = 1 + a seeded permutation of E.

    Drawn on the CPU with its own generator so that it does not depend on
    the device; returned as fp32.
    """
    perm = torch.randperm(E, generator=_gen(torch.device("cpu"), seed))
    rank = (perm + 1).to(torch.float64)
    b = 1.5 * torch.log(1.0 / rank.pow(1.2))
    return b.to(torch.float32)


def make_x(cfg: LayerConfig, seed: int = 0, device="cpu", T: Optional[int] = None):
    T = cfg.T if T is None else T
    return normal_bf16((T, cfg.d), 1.0, derive_seed(seed, "x"), device)


def make_expert(cfg: LayerConfig, e: int, seed: int = 0, device="cpu"):
    """(w_g [F,l], w_u [F,l], w_d [l,F]) of expert ``e``, bf16."""
    wg = normal_bf16((cfg.F, cfg.l), 1.0 / math.sqrt(cfg.l), derive_seed(seed, "w_g", e), device)
    wu = normal_bf16((cfg.F, cfg.l), 1.0 / math.sqrt(cfg.l), derive_seed(seed, "w_u", e), device)
    wd = normal_bf16((cfg.l, cfg.F), 1.0 / math.sqrt(cfg.F), derive_seed(seed, "w_d", e), device)
    return wg, wu, wd


def make_weights(cfg: LayerConfig, seed: int = 0, device="cpu",
                 experts: bool = True) -> Dict[str, Optional[torch.Tensor]]:
    """All weights in torch nn.Linear layout [out, in], bf16.

    Keys: w_r [E,d], b_r [E] fp32 or None, w_dn [l,d], w_g/w_u [E,F,l],
    w_d [E,l,F], w_up [d,l], w_gs/w_us [Fs,d] and w_ds [d,Fs] (None when
    Fs == 0). With ``experts=False`` the stacked expert tensors are left out
    (None); ``make_expert`` regenerates any one of them.
    """
    device = torch.device(device)
    rstd = cfg.router_std if cfg.router_std is not None else 1.0 / math.sqrt(cfg.d)
    w: Dict[str, Optional[torch.Tensor]] = {
        "w_r": normal_bf16((cfg.E, cfg.d), rstd, derive_seed(seed, "w_r"), device),
        "b_r": zipf_router_bias(cfg.E, derive_seed(seed, "b_r")).to(device) if cfg.zipf_bias else None,
        "w_dn": normal_bf16((cfg.l, cfg.d), 1.0 / math.sqrt(cfg.d), derive_seed(seed, "w_dn"), device),
        "w_up": normal_bf16((cfg.d, cfg.l), 1.0 / math.sqrt(cfg.l), derive_seed(seed, "w_up"), device),
        "w_g": None, "w_u": None, "w_d": None,
        "w_gs": None, "w_us": None, "w_ds": None,
    }
    if experts:
        wg = torch.empty((cfg.E, cfg.F, cfg.l), dtype=torch.bfloat16, device=device)
        wu = torch.empty_like(wg)
        wd = torch.empty((cfg.E, cfg.l, cfg.F), dtype=torch.bfloat16, device=device)
        for e in range(cfg.E):
            a, b, c = make_expert(cfg, e, seed, device)
            wg[e].copy_(a)
            wu[e].copy_(b)
            wd[e].copy_(c)
            del a, b, c
        w["w_g"], w["w_u"], w["w_d"] = wg, wu, wd
    if cfg.Fs > 0:
        w["w_gs"] = normal_bf16((cfg.Fs, cfg.d), 1.0 / math.sqrt(cfg.d), derive_seed(seed, "w_gs"), device)
        w["w_us"] = normal_bf16((cfg.Fs, cfg.d), 1.0 / math.sqrt(cfg.d), derive_seed(seed, "w_us"), device)
        w["w_ds"] = normal_bf16((cfg.d, cfg.Fs), 1.0 / math.sqrt(cfg.Fs), derive_seed(seed, "w_ds"), device)
    return w


def sample_tokens(T: int, n: int, seed: int = 1):
    """Seeded token subset used where the oracle runs on a sample."""
    g = _gen(torch.device("cpu"), seed)
    return torch.randperm(T, generator=g)[:n].sort().values
