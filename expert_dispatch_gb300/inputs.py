"""Seeded synthetic inputs for the MoE layer forward.

This module draws random tensors and nothing else: it holds none of the
layer's arithmetic (no routing, no scoring, no FFN), so both the CUDA path and
the CPU oracle can take their inputs from it without sharing any of the
method.  Every workload is defined by its shapes and value distributions:

* activations x ~ N(0, 1), one row per token;
* router weights Wr[E, d] and expert weights Wg[E+S, I, d], Wu[E+S, I, d],
  Wd[E+S, d, I] ~ N(0, 1/fan_in) (std 1/sqrt(fan_in)), stored in the
  workload's dtype (fp32, or bf16 rounded from fp32 draws).  The expert index
  is the outermost dimension, so each expert is one contiguous slab;
* sigmoid-family workloads draw a per-expert selection bias ~ U(-0.1, 0.1);
* the skewed workload offsets every router logit of expert e by
  log(Zipf_s(e)) = -s*log(e+1) - log(H_{E,s}), s = 1.2, which makes the
  lowest-numbered experts an order of magnitude hotter than the mean.

Rows of x can be redrawn (``redraw_rows``) from a fresh generator seeded
``seed + 1 + round``; the test suite uses this to keep top-k score margins
above 1e-3 so that no routing decision is a near-tie.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

GATE_SOFTMAX = 0
GATE_SIGMOID = 1


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    d: int
    E: int
    I: int
    k: int
    S: int = 0
    gate: int = GATE_SOFTMAX
    norm_topk: int = 0
    routed_scaling: float = 1.0
    dtype: str = "bf16"  # storage dtype of x and of all weights
    sel_bias_range: float = 0.0  # sigmoid family: selection bias ~ U(-r, r)
    zipf_s: float = 0.0  # > 0: skewed router logits, offset log Zipf_s(e)
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_T(self, T: int) -> "LayerConfig":
        return LayerConfig(self.name.split("@")[0] + "@T%d" % T, T, self.d, self.E, self.I,
                           self.k, self.S, self.gate, self.norm_topk, self.routed_scaling,
                           self.dtype, self.sel_bias_range, self.zipf_s, dict(self.extra))


# The five workloads (shapes of the catalogued Qwen-, DeepSeek- and Kimi-layout
# MoE layers; synthetic values).
TINY_FP32 = LayerConfig("tiny_fp32_T64_d256_E16_I128_top2", T=64, d=256, E=16, I=128, k=2,
                        dtype="f32")
QWEN_T512 = LayerConfig("qwen_layout_T512_d4096_E256_I1536_top8", T=512, d=4096, E=256,
                        I=1536, k=8)
DEEPSEEK_PREFILL = LayerConfig("deepseek_layout_prefill_T4096_d7168_E256_I2048_top8_shared1",
                               T=4096, d=7168, E=256, I=2048, k=8, S=1, gate=GATE_SIGMOID,
                               norm_topk=1, routed_scaling=2.5, sel_bias_range=0.1)
SKEWED_ZIPF = LayerConfig("skewed_zipf1.2_T16384_d4096_E256_I1536_top8", T=16384, d=4096,
                          E=256, I=1536, k=8, zipf_s=1.2)
KIMI_DECODE = LayerConfig("kimi_layout_decode_d7168_E384_I2048_top8_shared1", T=64, d=7168,
                          E=384, I=2048, k=8, S=1, gate=GATE_SIGMOID, norm_topk=1,
                          routed_scaling=2.827, sel_bias_range=0.1)
DECODE_TS = (1, 8, 32, 64)

CONFIGS = {
    "tiny_fp32": TINY_FP32,
    "qwen_t512": QWEN_T512,
    "deepseek_prefill": DEEPSEEK_PREFILL,
    "skewed_zipf": SKEWED_ZIPF,
    "kimi_decode": KIMI_DECODE,
}


def _normal(shape, std, g, device, dtype):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(dtype)


def make_inputs(cfg: LayerConfig, seed: int = 0, device="cpu") -> dict:
    """Draw one layer's tensors.  Large weights are drawn expert by expert."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = cfg.torch_dtype
    nE = cfg.E + cfg.S
    x = _normal((cfg.T, cfg.d), 1.0, g, device, dt)
    Wr = _normal((cfg.E, cfg.d), 1.0 / math.sqrt(cfg.d), g, device, dt)
    Wg = torch.empty((nE, cfg.I, cfg.d), dtype=dt, device=device)
    Wu = torch.empty((nE, cfg.I, cfg.d), dtype=dt, device=device)
    Wd = torch.empty((nE, cfg.d, cfg.I), dtype=dt, device=device)
    for e in range(nE):
        Wg[e] = _normal((cfg.I, cfg.d), 1.0 / math.sqrt(cfg.d), g, device, dt)
        Wu[e] = _normal((cfg.I, cfg.d), 1.0 / math.sqrt(cfg.d), g, device, dt)
        Wd[e] = _normal((cfg.d, cfg.I), 1.0 / math.sqrt(cfg.I), g, device, dt)
    sel_bias = None
    if cfg.sel_bias_range > 0:
        r = cfg.sel_bias_range
        sel_bias = (torch.rand((cfg.E,), generator=g, device=device, dtype=torch.float32) * 2 - 1) * r
    logit_bias = None
    if cfg.zipf_s > 0:
        e1 = torch.arange(1, cfg.E + 1, dtype=torch.float64)
        h = torch.sum(e1 ** (-cfg.zipf_s))
        logit_bias = (-cfg.zipf_s * torch.log(e1) - torch.log(h)).to(torch.float32).to(device)
    return {"x": x, "Wr": Wr, "Wg": Wg, "Wu": Wu, "Wd": Wd, "sel_bias": sel_bias,
            "logit_bias": logit_bias}


def redraw_rows(x: torch.Tensor, rows, seed: int, round_: int) -> None:
    """Replace rows of x (in place) with fresh N(0,1) draws from seed + 1 + round_."""
    rows = torch.as_tensor(rows, dtype=torch.long)
    if rows.numel() == 0:
        return
    g = torch.Generator(device=x.device)
    g.manual_seed(seed + 1 + round_)
    fresh = torch.randn((rows.numel(), x.shape[1]), generator=g, device=x.device,
                        dtype=torch.float32).to(x.dtype)
    x[rows.to(x.device)] = fresh


def random_residual(cfg: LayerConfig, seed: int, device="cpu") -> torch.Tensor:
    """An fp32 residual stream [T, d] ~ N(0, 1) for tests of the residual add."""
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed + 7919)
    return torch.randn((cfg.T, cfg.d), generator=g, device=device, dtype=torch.float32)
