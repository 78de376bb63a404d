"""Seeded synthetic workloads for the fused-MoE layer.

This module only draws random numbers; it holds none of the layer's arithmetic,
so both the CUDA path and the CPU oracle can take their inputs from it.

Recipe (seed 0 unless stated; draw order: logits, a1, w13, w2, shared w13/w2,
residual, RMSNorm weight):

* router logits ~ N(0, 1), fp32, [T, E];
* activations a1 ~ N(0, 1), bf16, [T, H];
* bf16 expert weights ~ N(0, 1/fan_in): w13 [E, 2I, H] (fan_in H, rows 0..I-1
  the gate, rows I..2I-1 the up projection), w2 [E, H, I] (fan_in I);
* fp8 expert weights: E4M3 codes of N(0, 64^2) draws (torch's cast) with one
  fp32 scale per 128x128 block, scale = U(0.75, 1.25) / (64 sqrt(fan_in)), so the
  dequantised weights have the N(0, 1/fan_in) scale of the bf16 ones;
* NVFP4 expert weights: uniform random bytes (two E2M1 codes each, so every
  code is equally likely), E4M3 scale codes uniform in [0x40, 0x50) (values
  2 .. 7.5) per 16 elements, and one fp32 global scale per expert and matrix,
  U(0.75, 1.25) / (13.2 sqrt(fan_in)), so the dequantised weights have about the
  N(0, 1/fan_in) scale of the bf16 ones (E2M1 codes have rms 2.93, the scales
  about 4.5); the activations' global scale is 2^-8 and the intermediate's
  2^-7 (a1 ~ N(0, 1) and h = silu(g) u with g, u of unit scale keep every
  group's scale code below the E4M3 maximum);
* shared expert (when present): bf16 weights drawn like the routed ones;
* finalize-only workloads: expert rows y ~ N(0, 1) bf16 [T*k, H], logits over k
  experts ~ N(0, 1) (softmax of them gives the top-k weights), distinct random
  expert ids of 256, shared and residual rows ~ N(0, 1) bf16, RMSNorm weight
  gamma ~ U(0.5, 1.5) rounded to bf16, eps 1e-6.

Large tensors can be drawn directly on a CUDA device (torch's Philox stream);
the bits then differ from a CPU draw of the same seed, so a check that needs the
same bits on both sides copies the device tensors to the host.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional

import torch


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    top_k: int
    quant: str = "bf16"            # "bf16"; "fp8" (E4M3 G(128) activations, 128x128 block weights);
                                   # "fp8_token" / "fp8_tensor" (per-token / per-tensor activation scales);
                                   # "nvfp4" (E2M1 + E4M3 per 16 + fp32 global scales, every operand)
    scoring: str = "softmax"       # "softmax" (renormalised top-k) or "sigmoid" (top-1)
    weight_on_input: bool = False  # apply the top-k weight to a1 in prepare (top_k == 1)
    shared_I: int = 0              # intermediate size of the bf16 shared expert, 0 = none
    finalize_only: bool = False    # workload of the finalize kernel alone
    residual: bool = False
    rms: bool = False
    nvfp4: bool = False
    activation: str = "silu"       # between the expert GEMMs; *_no_mul: w13 holds I rows
    single_launch: bool = False    # the whole step as one launch (moe_layer_fused)
    description: str = ""


def _cfgs():
    c = {}
    c["tiny"] = LayerConfig("tiny", 16, 256, 512, 8, 2,
                            description="tiny MoE layer T16 H256 I512 E8 top2 bf16")
    c["mixtral"] = LayerConfig("mixtral", 512, 4096, 14336, 8, 2,
                               description="Mixtral-8x7B-like layer T512 H4096 I14336 E8 top2 bf16")
    c["deepseek"] = LayerConfig("deepseek", 4096, 7168, 2048, 256, 8, quant="fp8", shared_I=2048,
                                description="DeepSeek-V3-like layer T4096 H7168 I2048 E256 top8 fp8 + bf16 shared I2048")
    # prefill sweeps where the expert GEMMs are tensor-bound (hundreds to thousands of rows per expert)
    for T in (4096, 8192):
        c[f"mixtral_T{T}"] = LayerConfig(f"mixtral_T{T}", T, 4096, 14336, 8, 2,
                                         description=f"Mixtral-8x7B-like layer T{T} H4096 I14336 E8 top2 bf16 (prefill)")
    # Qwen3-MoE-like layers: the Qwen3-30B-A3B expert shape (128 experts of intermediate size 768
    # over hidden 2048, top-8, no shared expert, softmax top-k renormalised), ~256 rows per expert
    c["qwen3"] = LayerConfig("qwen3", 4096, 2048, 768, 128, 8,
                             description="Qwen3-MoE-like layer T4096 H2048 I768 E128 top8 bf16")
    c["qwen3_fp8"] = LayerConfig("qwen3_fp8", 4096, 2048, 768, 128, 8, quant="fp8",
                                 description="Qwen3-MoE-like layer T4096 H2048 I768 E128 top8 fp8 G(128)")
    # the Llama-4-Scout-like shared expert alone at T=512: one dense expert of 512 rows, where the
    # expert GEMMs are tensor-bound (top-1 over one expert: every weight is 1)
    c["llama_shared512"] = LayerConfig("llama_shared512", 512, 5120, 8192, 1, 1,
                                       description="Llama-4-Scout-like shared expert alone T512 H5120 I8192 "
                                                   "(one dense expert, bf16)")
    c["deepseek_T16384"] = LayerConfig("deepseek_T16384", 16384, 7168, 2048, 256, 8, quant="fp8", shared_I=2048,
                                       description="DeepSeek-V3-like layer T16384 H7168 I2048 E256 top8 fp8 + bf16 shared (prefill)")
    # same per-expert shape as the DeepSeek-V3-like layer (~128 rows per expert), a quarter of the
    # experts: a small case for detailed profiles of the fp8 kernels
    c["deepseek_e64"] = LayerConfig("deepseek_e64", 1024, 7168, 2048, 64, 8, quant="fp8", shared_I=2048,
                                    description="DeepSeek-V3-shaped experts T1024 H7168 I2048 E64 top8 fp8 + bf16 shared")
    # the per-token ("A") and per-tensor ("T") activation formats on the same shape
    for q in ("token", "tensor"):
        c[f"deepseek_e64_{q}"] = LayerConfig(f"deepseek_e64_{q}", 1024, 7168, 2048, 64, 8, quant=f"fp8_{q}",
                                             shared_I=2048,
                                             description=f"DeepSeek-V3-shaped experts T1024 H7168 I2048 E64 top8 fp8 "
                                                         f"per-{q} activation scales + bf16 shared")
    c["mixtral_swigluoai"] = LayerConfig("mixtral_swigluoai", 512, 4096, 14336, 8, 2, activation="swigluoai",
                                         description="Mixtral-8x7B-like layer T512 H4096 I14336 E8 top2 bf16, "
                                                     "clamped SwiGLU (swigluoai)")
    for T in (128, 512):
        c[f"finalize{T}"] = LayerConfig(f"finalize{T}", T, 7168, 0, 256, 4, finalize_only=True,
                                        residual=True, rms=True, nvfp4=True, shared_I=1,
                                        description=f"finalize kernel T{T} H7168 top4 + shared + residual + RMSNorm")
    # every expert operand in NVFP4 (E2M1 + E4M3 per 16 + fp32 global scales)
    c["mixtral_nvfp4"] = LayerConfig("mixtral_nvfp4", 512, 4096, 14336, 8, 2, quant="nvfp4",
                                     description="Mixtral-8x7B-like layer T512 H4096 I14336 E8 top2 NVFP4 experts")
    c["llama1_nvfp4"] = LayerConfig("llama1_nvfp4", 1, 5120, 8192, 16, 1, scoring="sigmoid", weight_on_input=True,
                                    shared_I=8192, quant="nvfp4",
                                    description="Llama-4-Scout-like layer T1 H5120 I8192 E16 top1 sigmoid-on-input, "
                                                "NVFP4 experts + bf16 shared I8192")
    for T in (1, 8, 64, 512):
        c[f"llama{T}"] = LayerConfig(f"llama{T}", T, 5120, 8192, 16, 1, scoring="sigmoid",
                                     weight_on_input=True, shared_I=8192,
                                     description=f"Llama-4-Scout-like layer T{T} H5120 I8192 E16 top1 sigmoid-on-input + shared I8192")
    # the same layers as one launch (route, align, prepare, experts, finalize in one kernel)
    for T in (1, 8, 64):
        c[f"llama{T}_fused"] = LayerConfig(f"llama{T}_fused", T, 5120, 8192, 16, 1, scoring="sigmoid",
                                           weight_on_input=True, shared_I=8192, single_launch=True,
                                           description=f"Llama-4-Scout-like layer T{T} H5120 I8192 E16 top1 "
                                                       f"sigmoid-on-input + shared I8192, one launch")
    c["mixtral_fused"] = LayerConfig("mixtral_fused", 512, 4096, 14336, 8, 2, single_launch=True,
                                     description="Mixtral-8x7B-like layer T512 H4096 I14336 E8 top2 bf16, one launch")
    return c


CONFIGS: Dict[str, LayerConfig] = _cfgs()


def scaled(cfg: LayerConfig, **kw) -> LayerConfig:
    """A copy of `cfg` with some sizes replaced (smaller parity cases)."""
    d = dict(cfg.__dict__)
    d.update(kw)
    return LayerConfig(**d)


@dataclass
class LayerInputs:
    cfg: LayerConfig
    logits: torch.Tensor
    a1: Optional[torch.Tensor] = None
    w13: Optional[torch.Tensor] = None
    w13_scale: Optional[torch.Tensor] = None
    w2: Optional[torch.Tensor] = None
    w2_scale: Optional[torch.Tensor] = None
    shared_w13: Optional[torch.Tensor] = None
    shared_w2: Optional[torch.Tensor] = None
    residual: Optional[torch.Tensor] = None
    rms_weight: Optional[torch.Tensor] = None
    # finalize-only workload
    y: Optional[torch.Tensor] = None
    topk_ids: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)

    def to(self, device) -> "LayerInputs":
        mv = lambda v: v.to(device) if isinstance(v, torch.Tensor) else v
        d = {k: mv(v) for k, v in self.__dict__.items()}
        d["extra"] = {k: mv(v) for k, v in self.extra.items()}
        return LayerInputs(**d)


def _bf16_weights(gen, E, N, K, device):
    out = torch.empty((E, N, K), dtype=torch.bfloat16, device=device)
    std = 1.0 / math.sqrt(K)
    for e in range(E):
        out[e] = (torch.randn((N, K), generator=gen, device=device) * std).to(torch.bfloat16)
    return out


def _fp8_weights(gen, E, N, K, device):
    assert N % 128 == 0 and K % 128 == 0
    codes = torch.empty((E, N, K), dtype=torch.uint8, device=device)
    for e in range(E):
        codes[e] = (torch.randn((N, K), generator=gen, device=device) * 64.0).to(torch.float8_e4m3fn).view(torch.uint8)
    u = torch.rand((E, N // 128, K // 128), generator=gen, device=device) * 0.5 + 0.75
    scale = (u / (64.0 * math.sqrt(K))).to(torch.float32)
    return codes, scale


def _nvfp4_weights(gen, E, N, K, device):
    assert K % 16 == 0
    packed = torch.empty((E, N, K // 2), dtype=torch.uint8, device=device)
    sf = torch.empty((E, N, K // 16), dtype=torch.uint8, device=device)
    for e in range(E):
        packed[e] = torch.randint(0, 256, (N, K // 2), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
        sf[e] = torch.randint(0x40, 0x50, (N, K // 16), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
    u = torch.rand((E,), generator=gen, device=device) * 0.5 + 0.75
    gscale = (u / (13.2 * math.sqrt(K))).to(torch.float32)
    return packed, sf, gscale


NVFP4_A1_GSCALE = 2.0 ** -8
NVFP4_H_GSCALE = 2.0 ** -7


def make_logits(cfg: LayerConfig, seed: int = 0, device="cpu") -> torch.Tensor:
    """The router logits of `make_inputs(cfg, seed, device)` (its first draw) alone."""
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(seed)
    ncol = cfg.top_k if cfg.finalize_only else cfg.E
    return torch.randn((cfg.T, ncol), generator=gen, device=torch.device(device), dtype=torch.float32)


def make_inputs(cfg: LayerConfig, seed: int = 0, device="cpu") -> LayerInputs:
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
    if cfg.finalize_only:
        logits = torch.randn((T, k), generator=gen, device=dev, dtype=torch.float32)
        y = torch.randn((T * k, H), generator=gen, device=dev).to(torch.bfloat16)
        ids = torch.argsort(torch.rand((T, E), generator=gen, device=dev), dim=1)[:, :k].to(torch.int32).contiguous()
        shared = torch.randn((T, H), generator=gen, device=dev).to(torch.bfloat16)
        residual = torch.randn((T, H), generator=gen, device=dev).to(torch.bfloat16)
        gamma = (torch.rand((H,), generator=gen, device=dev) + 0.5).to(torch.bfloat16)
        return LayerInputs(cfg, logits, y=y, topk_ids=ids, residual=residual, rms_weight=gamma,
                           extra={"shared": shared})
    logits = torch.randn((T, E), generator=gen, device=dev, dtype=torch.float32)
    a1 = torch.randn((T, H), generator=gen, device=dev).to(torch.bfloat16)
    inp = LayerInputs(cfg, logits, a1=a1)
    rows13 = I if cfg.activation.endswith("_no_mul") else 2 * I
    if cfg.quant == "nvfp4":
        inp.w13, inp.w13_scale, g13 = _nvfp4_weights(gen, E, rows13, H, dev)
        inp.w2, inp.w2_scale, g2 = _nvfp4_weights(gen, E, H, I, dev)
        inp.extra.update(w13_gscale=g13, w2_gscale=g2, a1_gscale=NVFP4_A1_GSCALE, h_gscale=NVFP4_H_GSCALE)
    elif cfg.quant != "bf16":
        inp.w13, inp.w13_scale = _fp8_weights(gen, E, rows13, H, dev)
        inp.w2, inp.w2_scale = _fp8_weights(gen, E, H, I, dev)
    else:
        inp.w13 = _bf16_weights(gen, E, rows13, H, dev)
        inp.w2 = _bf16_weights(gen, E, H, I, dev)
    if cfg.shared_I:
        inp.shared_w13 = _bf16_weights(gen, 1, 2 * cfg.shared_I, H, dev)
        inp.shared_w2 = _bf16_weights(gen, 1, H, cfg.shared_I, dev)
    if cfg.residual:
        inp.residual = torch.randn((T, H), generator=gen, device=dev).to(torch.bfloat16)
    if cfg.rms:
        inp.rms_weight = (torch.rand((H,), generator=gen, device=dev) + 0.5).to(torch.bfloat16)
    return inp
