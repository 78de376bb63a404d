"""Plain, slow CPU oracle of the single-GPU fused-MoE layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import or run anything in ``oracle/``.  The CUDA library never calls it and
shares no code with it: no kernels, headers, constants or helpers.

Arithmetic is float64 (torch CPU and numpy) unless the step fixes a narrower
precision; every narrowing is written out where the step stores its result.

The pages define the layer as a modular pipeline, prepare -> experts ->
finalize, run on one device without dispatch or combine:

* "[vLLM] MoE Oracle & Prepare/Finalize" blog, section "No DP/EP: the simplest
  case" (the ``MoEPrepareAndFinalizeNoDPEPModular`` class): prepare multiplies a1
  by the top-k weight when ``apply_router_weight_on_input`` (top-k must be 1),
  then quantises the input; finalize hands the expert rows and top-k weights to
  a weight-and-reduce step.
* "Fused MoE Kernel Features" (vLLM design doc), section "Fused MoE Modular
  All2All backends": prepare returns the quantised type, finalize takes and
  returns the original activation type in the standard (token-major) format;
  with no quantisation type the kernels run in bf16.  Section "Fused Experts
  Kernels": the experts apply an activation between two GEMMs (SiLU-and-mul is
  the default SwiGLU); quantisation format "G(128)" means one scale per token
  per 128-channel block.
* "[flashinfer] MoE Finalize + AllReduce fusion" page, introduction: finalize
  multiplies the top-k expert rows by their routing scales and sums them,
  optionally adds the shared-expert row, then (after the all-reduce, absent on
  one GPU) adds the residual, applies RMSNorm and optionally packs NVFP4.

* "Fused MoE Kernel Features", section "Fused MoE Modular All2All backends": the
  prepare output comes in a "standard" or a "batched" format (the batched
  functions at the end of this file state the layout read for it).
* "Fused MoE Kernel Features", experts table: besides bf16 and fp8 (formats
  G(128), A, T), nvfp4 is a quantisation type of the experts; the NVFP4 experts
  below take every operand in the finalize page's NVFP4 encoding.

Where the pages leave a step open (router, alignment, scale formats, finalize
order, the NVFP4 experts' global scales and intermediate) each function below
states the plain reading it takes.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against invariants, closed forms, brute force or library routines.  The whole
layer composed of them has no printed worked example on the pages, so parity of
the composition rests on the per-step pins.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import codecs

F64 = torch.float64
AMAX_FLOOR = float(np.float32(1e-10))  # the amax clamp, as an fp32 number


def _np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().to(torch.float64).numpy() if t.is_floating_point() else t.detach().cpu().numpy()
    return np.asarray(t)


def to_bf16_tensor(x64: np.ndarray) -> torch.Tensor:
    """fp64 array -> bf16 torch tensor with a single round-to-nearest-even step."""
    r = codecs.round_bf16(x64)
    return torch.from_numpy(np.ascontiguousarray(r)).to(torch.float32).to(torch.bfloat16)  # exact


# =========================================================================== route
def route_softmax_renorm(logits: torch.Tensor, top_k: int):
    """Top-k routing with softmax weights renormalised over the selected experts.

    The pages take ``topk_ids``/``topk_weights`` as given (prepare and finalize
    arguments in the "No DP/EP" listing); the router is read as: rank experts
    by the fp32 logit, larger first, equal logits to the lower expert index; weight_j = exp(l_j - l_max) / sum over the selected
    experts of exp(l_i - l_max), which equals the full softmax renormalised over
    the top-k.  Weights are computed in fp64 and stored as fp32.
    """
    L = _np(logits)  # fp32 values held exactly in fp64
    T, E = L.shape
    assert 1 <= top_k <= E
    ids = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float32)
    for t in range(T):
        order = sorted(range(E), key=lambda i: (-L[t, i], i))[:top_k]
        ids[t] = order
        sel = L[t, order]
        e = np.exp(sel - sel[0])  # sel[0] is the largest selected logit
        w[t] = (e / e.sum()).astype(np.float32)
    return torch.from_numpy(ids), torch.from_numpy(w)


def route_sigmoid_top1(logits: torch.Tensor):
    """Top-1 routing with weight sigmoid(logit) (Llama-4-like router).

    The "Fused MoE Kernel Features" page notes that Llama-type models with
    top-k == 1 apply the top-k weight to the input activation; the weight
    itself is read as sigmoid of the selected logit, not renormalised.
    Argmax ties go to the lower expert index.
    """
    L = _np(logits)
    T, E = L.shape
    ids = np.empty((T, 1), dtype=np.int32)
    w = np.empty((T, 1), dtype=np.float32)
    for t in range(T):
        best = 0
        for i in range(1, E):
            if L[t, i] > L[t, best]:
                best = i
        ids[t, 0] = best
        w[t, 0] = np.float32(1.0 / (1.0 + math.exp(-L[t, best])))
    return torch.from_numpy(ids), torch.from_numpy(w)


# =========================================================================== align
@dataclass
class Alignment:
    expert_offsets: torch.Tensor  # [E+1] int32, offsets[E] = S = T*k
    sorted_slot: torch.Tensor     # [S] int32, value f = t*k + j
    inv_slot: torch.Tensor        # [S] int32, inv_slot[sorted_slot[p]] = p
    tile_map: torch.Tensor        # [num_tiles, 2] int32: (expert, first row)
    num_tiles: int


def align(topk_ids: torch.Tensor, num_experts: int, block_m: int) -> Alignment:
    """Per-expert grouping of the token slots (the "alignment and permutation").

    Reading: slot f = t*k + j is the j-th choice of token t; the
    slots are sorted by the key (expert id, f), so each expert's rows are
    contiguous and in ascending slot order; expert_offsets is the exclusive
    prefix sum of the per-expert counts (unpadded, so offsets[E] = T*k); the
    tile map lists, expert by expert, the first row of each block_m-row tile.
    """
    flat = [int(v) for v in _np(topk_ids).reshape(-1)]
    S = len(flat)
    order = sorted(range(S), key=lambda f: (flat[f], f))
    counts = [0] * num_experts
    for e in flat:
        counts[e] += 1
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    inv = [0] * S
    for p, f in enumerate(order):
        inv[f] = p
    tiles = []
    for e in range(num_experts):
        r = offsets[e]
        while r < offsets[e + 1]:
            tiles.append((e, r))
            r += block_m
    tm = torch.tensor(tiles, dtype=torch.int32).reshape(-1, 2)
    return Alignment(torch.tensor(offsets, dtype=torch.int32), torch.tensor(order, dtype=torch.int32),
                     torch.tensor(inv, dtype=torch.int32), tm, len(tiles))


# =========================================================================== prepare
def quantize_fp8_g128(x64: np.ndarray, group: int = 128):
    """Per-row, per-128-column fp8 E4M3 quantisation ("G(128)" format).

    Reading: for each row and each 128-column group,
    s = fp32(max(amax, fp32(1e-10)) / 448) and q = e4m3_rn_satfinite(fp32(x / s)).
    The scale is stored as the fp32 value used for dequantisation, x ~ q * s.
    x must hold values exactly representable in fp32 (bf16 inputs are).
    Returns (codes uint8 [R, C], scales fp32 [R, C/128]).
    """
    R, C = x64.shape
    assert C % group == 0
    g = x64.reshape(R, C // group, group)
    amax = np.abs(g).max(axis=2)
    s = codecs.round_fp32(np.maximum(amax, AMAX_FLOOR) / 448.0)  # IEEE fp32 division
    ratio = codecs.round_fp32(g / s[:, :, None])               # IEEE fp32 division
    q = codecs.e4m3_encode(ratio).reshape(R, C)
    return q, s.astype(np.float32)


def dequant_fp8_g128(q: np.ndarray, s: np.ndarray, group: int = 128) -> np.ndarray:
    R, C = q.shape
    return (codecs.e4m3_decode(q).reshape(R, C // group, group) * s.astype(np.float64)[:, :, None]).reshape(R, C)


# The "A" (per activation token) and "T" (per tensor) quantisation formats of the
# "Fused MoE Kernel Features" tables (table key: "A - Per activation token",
# "T - Per tensor"), read with the G(128) rule above: one scale per row over all
# its columns, or one scale over the whole tensor.
def quantize_fp8_token(x64: np.ndarray):
    """"A" format: s_r = fp32(max(amax_r, fp32(1e-10)) / 448) over row r,
    q = e4m3_rn_satfinite(fp32(x / s_r)).  Returns (codes [R, C], scales fp32 [R])."""
    amax = np.abs(x64).max(axis=1) if x64.shape[1] else np.zeros(x64.shape[0])
    s = codecs.round_fp32(np.maximum(amax, AMAX_FLOOR) / 448.0)
    q = codecs.e4m3_encode(codecs.round_fp32(x64 / s[:, None]))
    return q, s.astype(np.float32)


def quantize_fp8_tensor(x64: np.ndarray):
    """"T" format: one s = fp32(max(amax, fp32(1e-10)) / 448) over all elements.
    Returns (codes [R, C], scale fp32 [1])."""
    amax = float(np.abs(x64).max()) if x64.size else 0.0
    s = codecs.round_fp32(max(amax, AMAX_FLOOR) / 448.0)
    q = codecs.e4m3_encode(codecs.round_fp32(x64 / s))
    return q, np.array([s], dtype=np.float32)


def dequant_fp8(q: np.ndarray, s: np.ndarray, quant: str) -> np.ndarray:
    """codes x scale for the three fp8 formats (rows of q, with their scales)."""
    if quant == "fp8":
        return dequant_fp8_g128(q, s)
    v = codecs.e4m3_decode(q)
    if quant == "fp8_token":
        return v * s.astype(np.float64)[:, None]
    if quant == "fp8_tensor":
        return v * float(s[0])
    raise ValueError(quant)


def prepare(a1: torch.Tensor, topk_weights: torch.Tensor, apply_router_weight_on_input: bool, quant: str):
    """Prepare step of the no-DP/EP prepare/finalize ("[vLLM] MoE Oracle &
    Prepare/Finalize" blog, "No DP/EP" section).

    With ``apply_router_weight_on_input`` (allowed only for top-k == 1) the
    input is first multiplied by the top-k weight cast to the activation type:
    a1 = bf16(a1 * bf16(w)).  Then the input is quantised: ``quant == 'bf16'``
    is "no quantisation type", a passthrough; ``quant == 'fp8'`` is the
    per-token G(128) E4M3 format; ``'fp8_token'`` and ``'fp8_tensor'`` the "A"
    and "T" formats.  Returns (a1q, a1q_scale or None) with a1q a bf16 tensor or
    a uint8 tensor of E4M3 codes.
    """
    x = _np(a1)
    if apply_router_weight_on_input:
        w = _np(topk_weights)
        assert w.shape[1] == 1, "apply_router_weight_on_input needs top_k == 1"
        wb = codecs.round_bf16(w[:, 0])
        x = codecs.round_bf16(x * wb[:, None])
    if quant == "bf16":
        return to_bf16_tensor(x), None
    if quant == "fp8":
        q, s = quantize_fp8_g128(x)
        return torch.from_numpy(q), torch.from_numpy(s)
    if quant == "fp8_token":
        q, s = quantize_fp8_token(x)
        return torch.from_numpy(q), torch.from_numpy(s)
    if quant == "fp8_tensor":
        q, s = quantize_fp8_tensor(x)
        return torch.from_numpy(q), torch.from_numpy(s)
    raise ValueError(quant)


# =========================================================================== experts
_E4M3_TABLE = codecs.e4m3_decode(np.arange(256))  # value of every code


def dequant_weight_block(w_codes: np.ndarray, w_scale: np.ndarray, block: int = 128) -> np.ndarray:
    """[N, K] E4M3 codes with [N/128, K/128] fp32 block scales -> fp64 [N, K]."""
    N, K = w_codes.shape
    v = _E4M3_TABLE[w_codes].reshape(N // block, block, K // block, block)
    return (v * w_scale.astype(np.float64)[:, None, :, None]).reshape(N, K)


def silu_and_mul(gu: torch.Tensor) -> torch.Tensor:
    """act(x) = silu(x[:, :I]) * x[:, I:], silu(g) = g / (1 + exp(-g)).

    The "Fused Experts Kernels" table names SiLU (the SwiGLU gate) as the
    activation between the two expert GEMMs; the gate half comes first."""
    I = gu.shape[1] // 2
    g, u = gu[:, :I], gu[:, I:]
    return g / (1.0 + torch.exp(-g)) * u


# The activation column of the "Fused Experts Kernels" table (vLLM design doc)
# lists silu, gelu, swigluoai, silu_no_mul and gelu_no_mul (triton row) and
# gelu_tanh (cpu_moe row) without formulas.  Readings taken here:
# * gated forms (silu, gelu, gelu_tanh): h = act(g) * u with g, u the gate and
#   up halves of x = A w13^T (w13 rows 0..I-1 gate, I..2I-1 up);
# * *_no_mul forms: w13 holds the I gate rows only and h = act(g);
# * gelu is the exact form g * Phi(g) = g/2 (1 + erf(g / sqrt 2)); gelu_tanh is
#   the usual tanh approximation g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)));
# * swigluoai is the clamped SwiGLU of the gpt-oss models as published with them:
#   g' = min(g, 7), u' = clamp(u, -7, 7), h = (u' + 1) * g' * sigmoid(1.702 g'),
#   with the same gate-then-up layout of w13 as the other gated forms.
ACTIVATIONS = ("silu", "gelu", "gelu_tanh", "swigluoai", "silu_no_mul", "gelu_no_mul")
SWIGLUOAI_ALPHA = 1.702
SWIGLUOAI_LIMIT = 7.0


def activation_is_gated(activation: str) -> bool:
    if activation not in ACTIVATIONS:
        raise ValueError(f"unknown activation {activation!r}")
    return not activation.endswith("_no_mul")


def activation(x: torch.Tensor, name: str) -> torch.Tensor:
    """h = act(x) between the two expert GEMMs, fp64, by the readings above.
    Gated forms take x = [g | u] ([rows, 2I]); *_no_mul forms take x = g ([rows, I])."""
    if activation_is_gated(name):
        I = x.shape[1] // 2
        g, u = x[:, :I], x[:, I:]
    else:
        g, u = x, None
    if name == "swigluoai":
        gc = torch.clamp(g, max=SWIGLUOAI_LIMIT)
        uc = torch.clamp(u, min=-SWIGLUOAI_LIMIT, max=SWIGLUOAI_LIMIT)
        return (uc + 1.0) * gc / (1.0 + torch.exp(-SWIGLUOAI_ALPHA * gc))
    if name in ("silu", "silu_no_mul"):
        a = g / (1.0 + torch.exp(-g))
    elif name in ("gelu", "gelu_no_mul"):
        a = 0.5 * g * (1.0 + torch.erf(g / math.sqrt(2.0)))
    else:  # gelu_tanh
        a = 0.5 * g * (1.0 + torch.tanh(math.sqrt(2.0 / math.pi) * (g + 0.044715 * g ** 3)))
    return a if u is None else a * u


def expert_rows(A64: torch.Tensor, W13: torch.Tensor, W2: torch.Tensor, quant: str,
                act: str = "silu") -> torch.Tensor:
    """One expert on a block of (already dequantised) input rows.

    g, u = A W13[:I]^T, A W13[I:]^T (fp64); h = silu(g) * u (or the activation
    ``act``, see ``activation``), stored the way the intermediate is stored
    (bf16, or re-quantised to fp8 G(128) when the activations are fp8);
    y = h W2^T in fp64, stored bf16.  Returns fp64 values of the stored bf16 y."""
    h = silu_and_mul(A64 @ W13.T) if act == "silu" else activation(A64 @ W13.T, act)
    hn = h.numpy()
    if quant == "bf16":
        h_st = codecs.round_bf16(hn)
    elif quant == "fp8":
        q, s = quantize_fp8_g128(codecs.round_fp32(hn))
        h_st = dequant_fp8_g128(q, s)
    elif quant == "fp8_token":
        # reading: with the "A" format the intermediate is stored in the activation
        # type (bf16) and quantised per row like the input
        q, s = quantize_fp8_token(codecs.round_bf16(hn))
        h_st = dequant_fp8(q, s, quant)
    else:
        raise ValueError(f"{quant}: the per-tensor intermediate needs all experts (see experts())")
    return _expert_out(h_st, W2)


def _expert_out(h_st: np.ndarray, W2: torch.Tensor) -> torch.Tensor:
    y = torch.from_numpy(h_st) @ W2.T
    return torch.from_numpy(codecs.round_bf16(y.numpy()))


def _weights64(w, w_scale, e, quant):
    if quant == "bf16":
        return torch.from_numpy(_np(w[e]))
    return torch.from_numpy(dequant_weight_block(_np(w[e]).astype(np.uint8), _np(w_scale[e])))


def _act64(a1q, a1q_scale, rows, quant):
    if quant == "bf16":
        return torch.from_numpy(_np(a1q)[rows])
    sc = _np(a1q_scale)
    return torch.from_numpy(dequant_fp8(_np(a1q)[rows].astype(np.uint8), sc if quant == "fp8_tensor" else sc[rows],
                                        quant))


def experts(a1q, a1q_scale, w13, w13_scale, w2, w2_scale, al: Alignment, top_k: int, quant: str,
            act: str = "silu") -> torch.Tensor:
    """Grouped expert computation: for every expert e and every sorted row
    p in [offsets[e], offsets[e+1]), slot f = sorted_slot[p] of token t = f // k
    gets y[f] = expert_e(a1q[t]).  Output: the unweighted expert rows in
    token-major order [T*k, H] (fp64 holding bf16 values), the layout finalize
    takes ("fused_expert_output" in the "No DP/EP" listing)."""
    offs = _np(al.expert_offsets)
    order = _np(al.sorted_slot)
    S = int(offs[-1])
    H = a1q.shape[1]
    y = torch.zeros((S, H), dtype=F64)
    if quant == "fp8_tensor":
        # reading: the "T" intermediate is h of every expert stored in bf16, then one
        # scale over all of it
        hs, used = [], []
        for e in range(len(offs) - 1):
            p0, p1 = int(offs[e]), int(offs[e + 1])
            if p0 == p1:
                continue
            slots = order[p0:p1]
            A = _act64(a1q, a1q_scale, slots // top_k, quant)
            W13 = _weights64(w13, w13_scale, e, quant)
            h = silu_and_mul(A @ W13.T) if act == "silu" else activation(A @ W13.T, act)
            hs.append(codecs.round_bf16(h.numpy()))
            used.append((e, slots))
        if not hs:
            return y
        q, s = quantize_fp8_tensor(np.concatenate(hs, 0))
        h_all = dequant_fp8(q, s, quant)
        r = 0
        for (e, slots), h in zip(used, hs):
            n = h.shape[0]
            y[torch.from_numpy(slots.astype(np.int64))] = _expert_out(
                h_all[r:r + n], _weights64(w2, w2_scale, e, quant))
            r += n
        return y
    for e in range(len(offs) - 1):
        p0, p1 = int(offs[e]), int(offs[e + 1])
        if p0 == p1:
            continue
        slots = order[p0:p1]
        A = _act64(a1q, a1q_scale, slots // top_k, quant)
        y[torch.from_numpy(slots.astype(np.int64))] = expert_rows(
            A, _weights64(w13, w13_scale, e, quant), _weights64(w2, w2_scale, e, quant), quant, act)
    return y


def token_expert_rows(a1q, a1q_scale, w13, w13_scale, w2, w2_scale, topk_ids, t: int, quant: str,
                      act: str = "silu") -> torch.Tensor:
    """The k expert rows of one token, y[t*k + j] for j < k (used to check
    sampled tokens of full-size layers one by one)."""
    ids = _np(topk_ids)[t]
    A = _act64(a1q, a1q_scale, np.array([t]), quant)
    return torch.cat([expert_rows(A, _weights64(w13, w13_scale, int(e), quant),
                                  _weights64(w2, w2_scale, int(e), quant), quant, act) for e in ids], 0)


def dense_mlp(x: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor) -> torch.Tensor:
    """Shared expert: one SwiGLU MLP over all tokens on the unweighted bf16 a1
    (the optional shared-expert row of the flashinfer finalize page).  Output
    fp64 holding bf16 values."""
    return expert_rows(torch.from_numpy(_np(x)), torch.from_numpy(_np(w13)), torch.from_numpy(_np(w2)), "bf16")


# =========================================================================== finalize
def nvfp4_quantize(x64: np.ndarray, global_scale: float):
    """NVFP4 packing of rows of x: 16-element groups, each with one E4M3 scale.

    Reading: sf = e4m3_rn_satfinite(amax / (6 g)); codes
    q_i = e2m1_rn_satfinite(x_i / (sf g)) (q = 0 when sf = 0); element 2i in
    the low nibble.  Returns (packed uint8 [R, C/2], scale codes uint8 [R, C/16])."""
    R, C = x64.shape
    g = x64.reshape(R, C // 16, 16)
    amax = np.abs(g).max(axis=2)
    sf_code = codecs.e4m3_encode(amax / (6.0 * global_scale))
    sf = codecs.e4m3_decode(sf_code)
    denom = (sf * global_scale)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(denom > 0, g / np.where(denom > 0, denom, 1.0), 0.0)
    codes = codecs.e2m1_encode(ratio).reshape(R, C)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, sf_code


def nvfp4_dequantize(packed: np.ndarray, sf_code: np.ndarray, global_scale: float) -> np.ndarray:
    R, Ch = packed.shape
    codes = np.empty((R, Ch * 2), dtype=np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    v = codecs.e2m1_decode(codes).reshape(R, -1, 16)
    return (v * (codecs.e4m3_decode(sf_code) * global_scale)[:, :, None]).reshape(R, Ch * 2)


@dataclass
class FinalizeOut:
    out: np.ndarray                      # fp64 unrounded output (after RMSNorm when given)
    out_bf16: torch.Tensor               # bf16 rounding of `out`
    residual_out: torch.Tensor           # bf16(sum before the norm)
    nvfp4: Optional[tuple] = None        # (packed, scale codes) when requested


def finalize(fused_expert_output, topk_weights, top_k: int, apply_router_weight_on_input: bool,
             shared=None, residual=None, rms_weight=None, eps: float = 1e-6,
             nvfp4_global_scale: Optional[float] = None) -> FinalizeOut:
    """Finalize: top-k weight-and-reduce, + shared row, + residual, RMSNorm, NVFP4.

    o_t = sum_j w_tj * y[t*k + j] (the weights are skipped when they were
    applied on the input) + shared_t + residual_t, in fp64.  Then, when an
    RMSNorm weight is given, o_t <- o_t / sqrt(mean_h(o_t^2) + eps) * gamma.
    The order follows the flashinfer finalize page's introduction with its
    all-reduce step removed (one GPU).  residual_out is bf16 of the sum before
    the norm.  NVFP4 packs the unrounded normalised values."""
    y = _np(fused_expert_output)
    S, H = y.shape
    T = S // top_k
    y = y.reshape(T, top_k, H)
    if apply_router_weight_on_input:
        o = y.sum(axis=1)
    else:
        w = _np(topk_weights).reshape(T, top_k)
        o = (w[:, :, None] * y).sum(axis=1)
    if shared is not None:
        o = o + _np(shared)
    if residual is not None:
        o = o + _np(residual)
    res_out = to_bf16_tensor(o)
    if rms_weight is not None:
        gmm = _np(rms_weight)
        o = o / np.sqrt((o * o).mean(axis=1, keepdims=True) + eps) * gmm[None, :]
    fo = FinalizeOut(out=o, out_bf16=to_bf16_tensor(o), residual_out=res_out)
    if nvfp4_global_scale is not None:
        fo.nvfp4 = nvfp4_quantize(o, nvfp4_global_scale)
    return fo


# =========================================================================== NVFP4 experts
# Reading: the "Fused MoE Kernel Features" experts table lists nvfp4 as the
# quantisation type of the cutlass_fp4 experts (formats A, T; SiLU) and of the
# trtllm experts (G(16)).  NVFP4 is the encoding the flashinfer finalize page's
# packed output uses: E2M1 pairs, one E4M3 scale per 16 elements, and one fp32
# global scale per tensor ("T").  Every tensor of the experts here is in that
# encoding: the activations (one global scale), each expert's weight matrices
# (one global scale per expert and matrix) and the intermediate h between the
# GEMMs (one global scale), which is stored in the activation type (bf16) and
# then quantised, as the "A"/"T" fp8 formats do.

def nvfp4_quantize_fp32(x: np.ndarray, global_scale: float):
    """NVFP4 packing with each decision step in fp32, the precision the kernels
    quantise in: s6 = fp32(6 g); sf = e4m3_rn_satfinite(fp32(amax / s6));
    d = fp32(sf g); q_i = e2m1_rn_satfinite(fp32(x_i / d)) (q = 0 when d = 0).
    x must hold fp32 values (bf16 inputs do); g an fp32 number > 0.  Returns
    (packed uint8 [R, C/2], element 2i in the low nibble; scale codes [R, C/16])."""
    R, C = x.shape
    g32 = float(np.float32(global_scale))
    grp = np.asarray(x, dtype=np.float64).reshape(R, C // 16, 16)
    amax = np.abs(grp).max(axis=2)
    s6 = float(np.float32(6.0 * g32))
    sf_code = codecs.e4m3_encode(codecs.round_fp32(amax / s6))
    d = codecs.round_fp32(codecs.e4m3_decode(sf_code) * g32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(d > 0, codecs.round_fp32(grp / np.where(d > 0, d, 1.0)), 0.0)
    codes = codecs.e2m1_encode(ratio).reshape(R, C)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, sf_code.astype(np.uint8)


def prepare_nvfp4(a1: torch.Tensor, topk_weights, apply_router_weight_on_input: bool, global_scale: float):
    """Prepare into NVFP4: the optional weight on the input exactly as
    ``prepare``, then ``nvfp4_quantize_fp32`` of the bf16 rows with the
    activations' global scale.  Returns (packed [T, H/2], scale codes [T, H/16])
    as uint8 tensors."""
    x = _np(a1)
    if apply_router_weight_on_input:
        w = _np(topk_weights)
        assert w.shape[1] == 1, "apply_router_weight_on_input needs top_k == 1"
        x = codecs.round_bf16(x * codecs.round_bf16(w[:, 0])[:, None])
    packed, sf = nvfp4_quantize_fp32(x, global_scale)
    return torch.from_numpy(packed), torch.from_numpy(sf)


def experts_nvfp4(a1q, a1q_sf, a1_gscale: float, w13, w13_sf, w13_gscale, w2, w2_sf, w2_gscale,
                  h_gscale: float, al: Alignment, top_k: int, act: str = "silu", return_h: bool = False):
    """Grouped experts with every operand in NVFP4 (see the reading above).

    For expert e and its rows (token t of slot f as in ``experts``):
    A = dequant(a1q[t]; g_a), W13 = dequant(w13[e]; g13[e]) in fp64;
    h = act(A W13^T) (fp64), stored bf16, then h_q = nvfp4_quantize_fp32(h; g_h);
    y[f] = bf16(dequant(h_q; g_h) . dequant(w2[e]; g2[e])^T).
    w13 [E, 2I, H/2] (*_no_mul: [E, I, H/2]) with w13_sf [E, rows, H/16];
    w2 [E, H, I/2] with w2_sf [E, H, I/16]; w13_gscale, w2_gscale [E].
    Returns y [T*k, H] (fp64 holding bf16 values); with ``return_h`` also the
    unrounded fp64 h of every sorted row [S, I] (S = offsets[E])."""
    offs = _np(al.expert_offsets)
    order = _np(al.sorted_slot)
    S = int(offs[-1])
    aq, asf = _np(a1q).astype(np.uint8), _np(a1q_sf).astype(np.uint8)
    H = aq.shape[1] * 2
    g13 = _np(w13_gscale).astype(np.float64).reshape(-1)
    g2 = _np(w2_gscale).astype(np.float64).reshape(-1)
    y = torch.zeros((S, H), dtype=F64)
    h_all = None
    for e in range(len(offs) - 1):
        p0, p1 = int(offs[e]), int(offs[e + 1])
        if p0 == p1:
            continue
        slots = order[p0:p1]
        t = slots // top_k
        A = nvfp4_dequantize(aq[t], asf[t], a1_gscale)
        W13 = nvfp4_dequantize(_np(w13[e]).astype(np.uint8), _np(w13_sf[e]).astype(np.uint8), g13[e])
        h = activation(torch.from_numpy(A @ W13.T), act).numpy()
        if return_h:
            if h_all is None:
                h_all = np.zeros((S, h.shape[1]))
            h_all[p0:p1] = h
        hq, hsf = nvfp4_quantize_fp32(codecs.round_bf16(h), h_gscale)
        W2 = nvfp4_dequantize(_np(w2[e]).astype(np.uint8), _np(w2_sf[e]).astype(np.uint8), g2[e])
        y[torch.from_numpy(slots.astype(np.int64))] = _expert_out(nvfp4_dequantize(hq, hsf, h_gscale),
                                                                  torch.from_numpy(W2))
    return (y, h_all) if return_h else y


# =========================================================================== batched activation format
# "Fused MoE Kernel Features" (vLLM design doc), section "Fused MoE Modular All2All
# backends": the prepare step outputs its activations in one of two formats, "standard"
# or "batched"; every prepare takes standard activations in and every finalize gives
# standard activations back, so a finalize takes the format its prepare produced.  The
# "Fused Experts Kernels" table lists batched entry points beside the standard ones
# (batched triton, batched deep gemm, cutlass batched fp8, naive batched).  The pages
# leave the layout itself to another document.  Reading taken here: the batched
# activations are one slab per expert, [E, max_tokens, H]; expert e's slab holds, in
# ascending slot order f = t*k + j, the prepared rows of the tokens that chose e, and
# expert_num_tokens[e] counts them; rows past the count hold nothing (zeros here).  The
# experts compute every counted row of every slab into an output slab of the same layout
# (unweighted bf16 rows); the finalize reads the row of slot f at (the expert of f, the
# rank of f among that expert's slots) and reduces like the standard finalize.

def batched_positions(topk_ids, num_experts: int):
    """The place of every slot in the batched layout: (expert of f, rank of f among the
    slots of that expert, counting in ascending f), and the per-expert counts."""
    ids = _np(topk_ids).reshape(-1).astype(np.int64)
    counts = np.zeros(num_experts, dtype=np.int64)
    rank = np.empty(len(ids), dtype=np.int64)
    for f in range(len(ids)):
        e = ids[f]
        rank[f] = counts[e]
        counts[e] += 1
    return ids, rank, counts


def prepare_batched(a1, topk_ids, topk_weights, apply_router_weight_on_input: bool, quant: str,
                    num_experts: int, max_tokens: int):
    """Prepare into the batched format: the standard prepare of every token (``prepare``),
    then token t's prepared row placed at (expert, rank) of each of its slots.  Returns
    (a1q_b [E, max_tokens, H] of the prepared type, scales in the same per-row layout --
    G(128): [E, max_tokens, H/128], "A": [E, max_tokens], "T": the tensor's [1]; None for
    bf16 -- and expert_num_tokens [E] int32).  A count above max_tokens is an error."""
    a1q, sc = prepare(a1, topk_weights, apply_router_weight_on_input, quant)
    ids, rank, counts = batched_positions(topk_ids, num_experts)
    if len(counts) and counts.max() > max_tokens:
        raise ValueError(f"an expert receives {int(counts.max())} slots, more than max_tokens = {max_tokens}")
    k = _np(topk_ids).shape[1]
    H = a1q.shape[1]
    q = torch.zeros((num_experts, max_tokens, H), dtype=a1q.dtype)
    s = None
    if quant == "fp8":
        s = torch.zeros((num_experts, max_tokens, H // 128), dtype=torch.float32)
    elif quant == "fp8_token":
        s = torch.zeros((num_experts, max_tokens), dtype=torch.float32)
    elif quant == "fp8_tensor":
        s = sc.clone()
    for f in range(len(ids)):
        q[ids[f], rank[f]] = a1q[f // k]
        if quant in ("fp8", "fp8_token"):
            s[ids[f], rank[f]] = sc[f // k]
    return q, s, torch.from_numpy(counts.astype(np.int32))


def experts_batched(a1q_b, a1q_b_scale, expert_num_tokens, w13, w13_scale, w2, w2_scale, quant: str,
                    act: str = "silu") -> torch.Tensor:
    """The experts on the batched format: slab e's first expert_num_tokens[e] rows through
    expert e (``expert_rows``: GEMM1, activation, the intermediate stored as in the
    standard path, GEMM2), written at the same place of an [E, max_tokens, H] output
    (fp64 holding bf16 values; uncounted rows zero).  "T": one intermediate scale over
    the counted rows of every slab, as ``experts`` does over every expert's rows."""
    E, M, H = a1q_b.shape
    counts = _np(expert_num_tokens).astype(np.int64)
    y = torch.zeros((E, M, H), dtype=F64)
    sc = None if a1q_b_scale is None else _np(a1q_b_scale)

    def rows_of(e):
        n = int(counts[e])
        if quant == "bf16":
            return torch.from_numpy(_np(a1q_b[e])[:n])
        if quant == "fp8_tensor":
            return torch.from_numpy(dequant_fp8(_np(a1q_b[e])[:n].astype(np.uint8), sc, quant))
        return torch.from_numpy(dequant_fp8(_np(a1q_b[e])[:n].astype(np.uint8), sc[e][:n], quant))

    if quant == "fp8_tensor":
        hs, used = [], []
        for e in range(E):
            if counts[e]:
                x = rows_of(e) @ _weights64(w13, w13_scale, e, quant).T
                h = silu_and_mul(x) if act == "silu" else activation(x, act)
                hs.append(codecs.round_bf16(h.numpy()))
                used.append(e)
        if not hs:
            return y
        q, s = quantize_fp8_tensor(np.concatenate(hs, 0))
        h_all = dequant_fp8(q, s, quant)
        r = 0
        for e, h in zip(used, hs):
            n = h.shape[0]
            y[e, :n] = _expert_out(h_all[r:r + n], _weights64(w2, w2_scale, e, quant))
            r += n
        return y
    for e in range(E):
        if counts[e]:
            y[e, :int(counts[e])] = expert_rows(rows_of(e), _weights64(w13, w13_scale, e, quant),
                                                _weights64(w2, w2_scale, e, quant), quant, act)
    return y


def unbatch(y_b, topk_ids) -> torch.Tensor:
    """Token-major expert rows [T*k, H] from a batched output: row f is the output row at
    (the expert of f, the rank of f) -- what the finalize reads for slot f."""
    E = y_b.shape[0]
    ids, rank, _ = batched_positions(topk_ids, E)
    yb = y_b if isinstance(y_b, torch.Tensor) else torch.from_numpy(np.asarray(y_b))
    return yb[torch.from_numpy(ids), torch.from_numpy(rank)].to(F64)


def finalize_batched(y_b, topk_ids, topk_weights, top_k: int, apply_router_weight_on_input: bool, **kw) -> FinalizeOut:
    """The finalize of the batched format: ``finalize`` of the rows ``unbatch`` reads."""
    return finalize(unbatch(y_b, topk_ids), topk_weights, top_k, apply_router_weight_on_input, **kw)
