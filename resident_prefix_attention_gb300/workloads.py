"""Seeded synthetic workloads for resident-prefix replay attention.

This module only draws inputs: shapes, random tensors, page permutations,
outlier positions and response lengths.  It holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle can consume its output
without sharing any of the method's code.

Workload shapes follow the LongStraw explainer ("longstraw-2m-rl", section
"Two incompatible architectures, same transaction": CP8-sharded KV pages,
reverse replay of response blocks) and "Serial replay makes G a schedule"
(one resident prompt shared by G serially replayed responses).  Head counts,
head_dim and page size are not on the pages; they are fixed here.

Recipe (every draw comes from one ``torch.Generator`` seeded with ``seed``):
  1. (group only) response lengths R_g ~ U{r_min..r_max}, G draws
  2. q       [R, Hq, d]   ~ N(0,1) -> bf16 (round to nearest even)
  3. k_prompt[P, Hkv, d]  ~ N(0,1) -> bf16
  4. v_prompt[P, Hkv, d]  ~ N(0,1) -> bf16
  5. k_resp  [R, Hkv, d]  ~ N(0,1) -> bf16
  6. v_resp  [R, Hkv, d]  ~ N(0,1) -> bf16
  7. dO      [R, Hq, d]   ~ N(0,1) -> bf16
  8. page permutation: randperm(num_pages) (identity when not shuffled)
  9. outliers: round(frac * P) distinct prompt positions whose K rows (all
     kv heads) are multiplied by 8 (exact in bf16).
For the group workload steps 2, 5, 6, 7 repeat per response g in order.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    P: int                      # prompt length (resident, stop-gradient)
    R: int                      # response length (max length for 'group')
    Hq: int
    Hkv: int
    d: int
    page_size: int
    shards: int                 # contiguous prompt KV shards, LSE-merged
    blocks: int = 1             # response blocks replayed in reverse
    shuffle: bool = True        # seeded random physical page order
    outlier_frac: float = 0.0   # fraction of prompt keys scaled x8
    G: int = 1                  # responses sharing the prompt
    r_min: int = 0              # group: response length range (inclusive)
    r_max: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def prompt_pages(self) -> int:
        return self.P // self.page_size

    @property
    def resp_pages(self) -> int:
        return -(-self.R // self.page_size)

    @property
    def num_pages(self) -> int:
        return self.prompt_pages + self.resp_pages

    @property
    def block_rows(self) -> int:
        return self.R // self.blocks


CONFIGS = {
    "tiny": Config("tiny", P=1024, R=256, Hq=4, Hkv=1, d=64, page_size=64,
                   shards=1, shuffle=False),
    "mid": Config("mid", P=32768, R=2048, Hq=32, Hkv=8, d=128, page_size=256,
                  shards=8),
    "long": Config("long", P=262144, R=4096, Hq=32, Hkv=8, d=128,
                   page_size=256, shards=16, blocks=4),
    "2M": Config("2M", P=2093056, R=4096, Hq=32, Hkv=8, d=128, page_size=256,
                 shards=8, outlier_frac=0.001),
    "group": Config("group", P=1048576, R=4096, Hq=32, Hkv=8, d=128,
                    page_size=256, shards=8, G=8, r_min=512, r_max=4096),
    # The 2M workload cut to one kv head (and its 4 query heads): the same
    # key stream per kv head, the same CTAs per stream and per wave, with
    # 1.07 GB of K/V instead of 8.6 GB.  Used for hardware-counter
    # captures, whose DRAM traffic scales to 2M by the kv-head count.
    "2M_kv1": Config("2M_kv1", P=2093056, R=4096, Hq=4, Hkv=1, d=128,
                     page_size=256, shards=8, outlier_frac=0.001),
}


def make_config(base: str = "mid", **overrides) -> Config:
    """A named workload with some fields replaced (smaller parity cases)."""
    c = dataclasses.asdict(CONFIGS[base])
    c.update(overrides)
    if "name" not in overrides:
        c["name"] = base + "*"
    return Config(**c)


@dataclasses.dataclass
class Response:
    q: torch.Tensor         # [R, Hq, d] bf16
    k: torch.Tensor         # [R, Hkv, d] bf16
    v: torch.Tensor         # [R, Hkv, d] bf16
    dO: torch.Tensor        # [R, Hq, d] bf16


@dataclasses.dataclass
class Workload:
    cfg: Config
    k_prompt: torch.Tensor  # [P, Hkv, d] bf16
    v_prompt: torch.Tensor  # [P, Hkv, d] bf16
    responses: List[Response]
    page_table: torch.Tensor  # [num_pages] int32, logical -> physical
    outliers: torch.Tensor    # [n_outliers] int64 prompt positions


def _randn_bf16(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def make_workload(cfg: Config, seed: int = 0, device: str = "cpu",
                  lengths: Optional[List[int]] = None) -> Workload:
    """Draw one workload; ``device`` selects the generator (cpu or cuda)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    if cfg.G > 1 and cfg.r_min > 0:
        if lengths is None:
            lengths = torch.randint(cfg.r_min, cfg.r_max + 1, (cfg.G,),
                                    generator=gen, device=device).tolist()
    elif lengths is None:
        lengths = [cfg.R] * cfg.G
    P, Hq, Hkv, d = cfg.P, cfg.Hq, cfg.Hkv, cfg.d
    # Draw order follows the module docstring.  For G responses the prompt
    # sits between the first response's q and its k/v, then responses
    # 2..G repeat q, k, v, dO.
    responses: List[Response] = []
    q0 = _randn_bf16((lengths[0], Hq, d), gen, device)
    k_prompt = _randn_bf16((P, Hkv, d), gen, device)
    v_prompt = _randn_bf16((P, Hkv, d), gen, device)
    for gi, R in enumerate(lengths):
        q = q0 if gi == 0 else _randn_bf16((R, Hq, d), gen, device)
        k = _randn_bf16((R, Hkv, d), gen, device)
        v = _randn_bf16((R, Hkv, d), gen, device)
        dO = _randn_bf16((R, Hq, d), gen, device)
        responses.append(Response(q, k, v, dO))
    npages = cfg.prompt_pages + (-(-max(lengths) // cfg.page_size))
    if cfg.shuffle:
        perm = torch.randperm(npages, generator=gen, device=device)
    else:
        perm = torch.arange(npages, device=device)
    n_out = int(round(cfg.outlier_frac * P))
    if n_out > 0:
        outliers = torch.randperm(P, generator=gen, device=device)[:n_out]
        k_prompt[outliers] = k_prompt[outliers] * 8
    else:
        outliers = torch.zeros(0, dtype=torch.int64, device=device)
    return Workload(cfg, k_prompt, v_prompt, responses,
                    perm.to(torch.int32), outliers)


# ------------------------------------------------------------ latent pages
# The latent-page variant (MLA-style resident state: the GLM bullet of "Two
# incompatible architectures, same transaction").  Each position stores one
# latent row [c (d_c), r (d_r)] shared by every query head; queries are the
# absorbed q~ of width d_c + d_r, outputs and output gradients have width
# d_c.  The widths are not on the pages; d_c = 128, d_r = 64 here.
#
# Recipe (one torch.Generator seeded with ``seed``):
#   1. q      [R, Hq, d_c + d_r] ~ N(0,1) -> bf16
#   2. prompt latent rows [P, d_c + d_r] ~ N(0,1) -> bf16
#   3. response latent rows [R, d_c + d_r] ~ N(0,1) -> bf16
#   4. dO     [R, Hq, d_c] ~ N(0,1) -> bf16
#   5. page permutation (identity when not shuffled)
#   6. outliers: round(frac * P) distinct prompt positions whose rotary part
#      r is multiplied by 8 (exact in bf16).  Only r is scaled: c is also
#      the value, and the outliers are meant to sharpen the scores, not to
#      change the values' range.
@dataclasses.dataclass(frozen=True)
class LatentConfig:
    name: str
    P: int
    R: int
    Hq: int
    page_size: int
    shards: int
    d_c: int = 128
    d_r: int = 64
    blocks: int = 1
    shuffle: bool = True
    outlier_frac: float = 0.0
    G: int = 1                  # responses sharing the prompt
    r_min: int = 0              # group: response length range (inclusive)
    r_max: int = 0

    @property
    def d_l(self) -> int:
        return self.d_c + self.d_r

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_l)

    @property
    def prompt_pages(self) -> int:
        return self.P // self.page_size

    @property
    def num_pages(self) -> int:
        return self.prompt_pages + (-(-self.R // self.page_size))

    @property
    def block_rows(self) -> int:
        return self.R // self.blocks


LATENT_CONFIGS = {
    "latent_tiny": LatentConfig("latent_tiny", P=1024, R=256, Hq=32,
                                page_size=128, shards=2, shuffle=False),
    "latent_mid": LatentConfig("latent_mid", P=32768, R=1024, Hq=32,
                               page_size=256, shards=8, blocks=2),
    "latent_long": LatentConfig("latent_long", P=524288, R=1024, Hq=32,
                                page_size=256, shards=8),
    "latent": LatentConfig("latent", P=2093056, R=4096, Hq=32,
                           page_size=256, shards=8, outlier_frac=0.001),
    "latent_group": LatentConfig("latent_group", P=1048576, R=4096, Hq=32,
                                 page_size=256, shards=8, G=8, r_min=512,
                                 r_max=4096),
}


def make_latent_config(base: str = "latent_mid", **overrides) -> LatentConfig:
    c = dataclasses.asdict(LATENT_CONFIGS[base])
    c.update(overrides)
    if "name" not in overrides:
        c["name"] = base + "*"
    return LatentConfig(**c)


@dataclasses.dataclass
class LatentWorkload:
    cfg: LatentConfig
    q: torch.Tensor          # [R, Hq, d_c + d_r] bf16
    lat_prompt: torch.Tensor  # [P, d_c + d_r] bf16
    lat_resp: torch.Tensor    # [R, d_c + d_r] bf16
    dO: torch.Tensor         # [R, Hq, d_c] bf16
    page_table: torch.Tensor  # [num_pages] int32
    outliers: torch.Tensor


def make_latent_workload(cfg: LatentConfig, seed: int = 0,
                         device: str = "cpu") -> LatentWorkload:
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = _randn_bf16((cfg.R, cfg.Hq, cfg.d_l), gen, device)
    lat_prompt = _randn_bf16((cfg.P, cfg.d_l), gen, device)
    lat_resp = _randn_bf16((cfg.R, cfg.d_l), gen, device)
    dO = _randn_bf16((cfg.R, cfg.Hq, cfg.d_c), gen, device)
    if cfg.shuffle:
        perm = torch.randperm(cfg.num_pages, generator=gen, device=device)
    else:
        perm = torch.arange(cfg.num_pages, device=device)
    n_out = int(round(cfg.outlier_frac * cfg.P))
    if n_out > 0:
        outliers = torch.randperm(cfg.P, generator=gen, device=device)[:n_out]
        lat_prompt[outliers, cfg.d_c:] = lat_prompt[outliers, cfg.d_c:] * 8
    else:
        outliers = torch.zeros(0, dtype=torch.int64, device=device)
    return LatentWorkload(cfg, q, lat_prompt, lat_resp, dO,
                          perm.to(torch.int32), outliers)


@dataclasses.dataclass
class LatentResponse:
    q: torch.Tensor          # [R, Hq, d_c + d_r] bf16
    lat: torch.Tensor        # [R, d_c + d_r] bf16
    dO: torch.Tensor         # [R, Hq, d_c] bf16


@dataclasses.dataclass
class LatentGroup:
    cfg: LatentConfig
    lat_prompt: torch.Tensor  # [P, d_c + d_r] bf16
    responses: List[LatentResponse]
    page_table: torch.Tensor  # prompt pages + one response slot, int32


def make_latent_group(cfg: LatentConfig, seed: int = 0,
                      device: str = "cpu") -> LatentGroup:
    """G responses of one latent prompt.  Recipe (one generator): lengths
    R_g ~ U{r_min..r_max}; the prompt's latent rows; then per response q~,
    latent rows and dO~ (each ~N(0,1) -> bf16); the page permutation of the
    prompt pages plus one response slot of ceil(max R_g / page_size)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    lengths = torch.randint(cfg.r_min, cfg.r_max + 1, (cfg.G,),
                            generator=gen, device=device).tolist()
    lat_prompt = _randn_bf16((cfg.P, cfg.d_l), gen, device)
    responses = []
    for R in lengths:
        q = _randn_bf16((R, cfg.Hq, cfg.d_l), gen, device)
        lat = _randn_bf16((R, cfg.d_l), gen, device)
        dO = _randn_bf16((R, cfg.Hq, cfg.d_c), gen, device)
        responses.append(LatentResponse(q, lat, dO))
    npages = cfg.prompt_pages + (-(-max(lengths) // cfg.page_size))
    perm = torch.randperm(npages, generator=gen, device=device)
    return LatentGroup(cfg, lat_prompt, responses, perm.to(torch.int32))
