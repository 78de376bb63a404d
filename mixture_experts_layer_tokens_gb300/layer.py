"""One fused-MoE layer step composed from the C-ABI calls, with every buffer
allocated once up front (PyTorch allocates, the library computes).

Step: moe_route -> moe_align -> moe_prepare -> moe_experts [-> shared expert via
  moe_experts with one expert and the identity permutation] -> moe_finalize, on the
caller's stream.  The shared expert needs no routing: when it runs as calls of its own
and neither its GEMMs nor the routed experts' split units across CTAs (whose waits
assume every CTA of the launch resident, which two concurrent launches cannot
promise), it runs on a second stream forked at the start of the step and joined
before the finalize, so its GEMMs overlap the routing, quantisation, gather and the
routed experts' GEMMs (which take their units from a counter, so CTAs that start
late because the shared expert still holds their SMs take fewer units).
NVFP4 layers use moe_prepare_nvfp4 and moe_experts_nvfp4 (the shared expert
stays bf16).  Single-launch layers run the whole step as one moe_layer_fused launch.

The shared expert sees the unweighted bf16 input, as the shared-expert row of
the flashinfer finalize fusion is added unscaled.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import moe
from .inputs import LayerConfig, LayerInputs


class MoELayer:
    def __init__(self, inp: LayerInputs, stream: Optional[torch.cuda.Stream] = None):
        cfg = self.cfg = inp.cfg
        assert not cfg.finalize_only
        self.inp = inp
        dev = inp.logits.device
        T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
        self.scoring = moe.MOE_SCORING_SIGMOID if cfg.scoring == "sigmoid" else moe.MOE_SCORING_SOFTMAX_RENORM
        self.topk_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.topk_weights = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.al = moe.Alignment(T, k, E, dev)
        self.nvfp4 = cfg.quant == "nvfp4"
        fp8 = cfg.quant != "bf16" and not self.nvfp4
        # bf16 without weight-on-input: prepare is the passthrough (a1q is a1)
        self.passthrough = cfg.quant == "bf16" and not cfg.weight_on_input
        self.y = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
        if self.nvfp4:
            # packed codes and one E4M3 scale code per 16 elements; fp32 global scales on the device
            self.a1q = torch.empty((T, H // 2), dtype=torch.uint8, device=dev)
            self.a1q_scale = torch.empty((T, H // 16), dtype=torch.uint8, device=dev)
            self.g_a = torch.tensor([inp.extra["a1_gscale"]], dtype=torch.float32, device=dev)
            self.g_h = torch.tensor([inp.extra["h_gscale"]], dtype=torch.float32, device=dev)
            self.ws = torch.empty(max(moe.workspace_size_nvfp4(T, H, I, E, k), 16), dtype=torch.uint8, device=dev)
        else:
            self.a1q = None if self.passthrough else torch.empty(
                (T, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
            self.a1q_scale = (torch.empty(moe.scale_shape(cfg.quant, T, H), dtype=torch.float32, device=dev)
                              if fp8 else None)
            self.ws = torch.empty(max(moe.workspace_size(T, H, I, E, k, cfg.quant), 16), dtype=torch.uint8,
                                  device=dev)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.shared = None
        if cfg.shared_I:
            self.shared = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
            ids0 = torch.zeros((T, 1), dtype=torch.int32, device=dev)
            self.al_shared = moe.moe_align(ids0, 1, stream=stream)
            self.ws_shared = torch.empty(max(moe.workspace_size(T, H, cfg.shared_I, 1, 1, "bf16"), 16),
                                         dtype=torch.uint8, device=dev)
            self.side = torch.cuda.Stream(device=dev)
            self.ev_fork = torch.cuda.Event()
            self.ev_join = torch.cuda.Event()
        # the whole step as one launch: a bf16 SiLU layer whose shared expert (if any) has the
        # routed experts' I
        self.single = cfg.single_launch
        if self.single:
            assert cfg.quant == "bf16" and cfg.activation == "silu" and cfg.shared_I in (0, I)
            self.ws_fused = torch.empty(max(moe.layer_fused_workspace_size(T, H, I, E, k, cfg.shared_I > 0), 16),
                                        dtype=torch.uint8, device=dev)
        # a bf16 layer whose shared expert has the routed experts' I and activation runs both
        # in the same GEMM launches (moe_experts_multi)
        self.fused_shared = (cfg.shared_I == I and cfg.quant == "bf16" and cfg.activation == "silu")
        # the shared expert on the second stream: its own calls, neither they (one expert, T
        # rows: split only for T <= 16) nor the routed experts (fp8 never; bf16 and NVFP4
        # at most 16 slots per expert) split units
        routed_splits = cfg.quant in ("bf16", "nvfp4") and T * k <= 16 * E
        self.shared_side = bool(cfg.shared_I) and not self.fused_shared and T > 16 and not routed_splits
        if self.fused_shared:
            a_dummy = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
            self.ws_multi = torch.empty(max(moe.workspace_size_multi(
                [moe.experts_problem(a_dummy, None, inp.w13, None, inp.w2, None, self.al, self.y),
                 moe.experts_problem(a_dummy, None, inp.shared_w13, None, inp.shared_w2, None, self.al_shared,
                                     self.shared, identity=True)], H, "bf16"), 16), dtype=torch.uint8, device=dev)

    def forward(self, logits: torch.Tensor, a1: torch.Tensor, stream=None) -> torch.Tensor:
        cfg, inp = self.cfg, self.inp
        if self.single:
            return moe.moe_layer_fused(
                logits, a1, inp.w13, inp.w2, cfg.top_k, self.scoring, cfg.weight_on_input,
                shared_w13=inp.shared_w13[0] if cfg.shared_I else None,
                shared_w2=inp.shared_w2[0] if cfg.shared_I else None, residual=inp.residual,
                rms_weight=inp.rms_weight, eps=1e-6, topk_ids=self.topk_ids, topk_weights=self.topk_weights,
                output=self.out, ws=self.ws_fused, stream=stream)
        main = stream if stream is not None else torch.cuda.current_stream()
        if self.shared_side:
            self.ev_fork.record(main)
            self.side.wait_event(self.ev_fork)
            moe.moe_experts(a1, None, inp.shared_w13, None, inp.shared_w2, None, self.al_shared, "bf16",
                            out=self.shared, ws=self.ws_shared, identity=True, stream=self.side)
            self.ev_join.record(self.side)
        moe.moe_route(logits, cfg.top_k, self.scoring, self.topk_ids, self.topk_weights, stream=stream)
        moe.moe_align(self.topk_ids, cfg.E, out=self.al, stream=stream)
        if self.passthrough:
            a1q, a1q_scale = a1, None
        elif self.nvfp4:
            a1q, a1q_scale = moe.moe_prepare_nvfp4(a1, self.topk_weights, cfg.top_k, cfg.weight_on_input, self.g_a,
                                                   self.a1q, self.a1q_scale, stream=stream)
        else:
            a1q, a1q_scale = moe.moe_prepare(a1, self.topk_weights, cfg.top_k, cfg.weight_on_input, cfg.quant,
                                             self.a1q, self.a1q_scale, stream=stream)
        shared = self.experts(a1q, a1q_scale, a1, stream, shared_launched=self.shared_side)
        if self.shared_side:
            main.wait_event(self.ev_join)
        moe.moe_finalize(self.y, self.topk_weights, cfg.top_k, cfg.weight_on_input, shared=shared,
                         residual=inp.residual, rms_weight=inp.rms_weight, output=self.out, stream=stream)
        return self.out

    def experts(self, a1q, a1q_scale, a1, stream=None, shared_launched=False):
        """The routed experts into self.y and the shared expert (if any) into
        self.shared -- one moe_experts_multi call when they can share launches;
        shared_launched: the step has already run the shared expert (second stream).
        Returns the shared-expert rows or None."""
        cfg, inp = self.cfg, self.inp
        if self.shared is not None and self.fused_shared:
            moe.moe_experts_multi(
                [moe.experts_problem(a1q, a1q_scale, inp.w13, inp.w13_scale, inp.w2, inp.w2_scale, self.al, self.y),
                 moe.experts_problem(a1, None, inp.shared_w13, None, inp.shared_w2, None, self.al_shared, self.shared,
                                     identity=True)], cfg.H, "bf16", self.ws_multi, stream=stream)
            return self.shared
        if self.nvfp4:
            moe.moe_experts_nvfp4(a1q, a1q_scale, self.g_a, inp.w13, inp.w13_scale, inp.extra["w13_gscale"], inp.w2,
                                  inp.w2_scale, inp.extra["w2_gscale"], self.g_h, self.al, out=self.y, ws=self.ws,
                                  stream=stream, activation=cfg.activation)
        else:
            moe.moe_experts(a1q, a1q_scale, inp.w13, inp.w13_scale, inp.w2, inp.w2_scale, self.al, cfg.quant,
                            activation=cfg.activation, out=self.y, ws=self.ws, stream=stream)
        if self.shared is None:
            return None
        if shared_launched:
            return self.shared
        return moe.moe_experts(a1, None, inp.shared_w13, None, inp.shared_w2, None, self.al_shared, "bf16",
                               out=self.shared, ws=self.ws_shared, identity=True, stream=stream)


class FinalizeStep:
    """The finalize-only workload: route over k logits, then finalize to bf16
    and to NVFP4."""

    def __init__(self, inp: LayerInputs):
        cfg = self.cfg = inp.cfg
        assert cfg.finalize_only
        self.inp = inp
        dev = inp.logits.device
        T, H, k = cfg.T, cfg.H, cfg.top_k
        self.topk_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.topk_weights = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.out_fp4 = torch.empty((T, H // 2), dtype=torch.uint8, device=dev)
        self.out_sf = torch.empty((T, H // 16), dtype=torch.uint8, device=dev)

    def weights(self, stream=None):
        moe.moe_route(self.inp.logits, self.cfg.top_k, moe.MOE_SCORING_SOFTMAX_RENORM, self.topk_ids,
                      self.topk_weights, stream=stream)
        return self.topk_weights

    def finalize(self, nvfp4: bool, stream=None):
        inp = self.inp
        if nvfp4:
            return moe.moe_finalize(inp.y, self.topk_weights, self.cfg.top_k, False, shared=inp.extra["shared"],
                                    residual=inp.residual, rms_weight=inp.rms_weight, eps=1e-6,
                                    out_dtype=moe.MOE_DT_NVFP4, out_global_scale=1.0, output=self.out_fp4,
                                    out_scale=self.out_sf, topk_ids=inp.topk_ids, stream=stream)
        return moe.moe_finalize(inp.y, self.topk_weights, self.cfg.top_k, False, shared=inp.extra["shared"],
                                residual=inp.residual, rms_weight=inp.rms_weight, eps=1e-6,
                                out_dtype=moe.MOE_DT_BF16, output=self.out, topk_ids=inp.topk_ids, stream=stream)
