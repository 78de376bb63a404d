"""Thin ctypes binding of the fused-MoE C ABI (``include/moe.h``).

Every function here checks tensor dtypes/devices, passes ``data_ptr()`` values
and the current torch CUDA stream to the C entry point of the same name, and
turns a non-OK status into :class:`MoeError`.  All arithmetic happens in the
CUDA library; there is no fallback path.  PyTorch only provides device memory
and streams.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = range(6)
MOE_DT_BF16, MOE_DT_FP8_E4M3, MOE_DT_NVFP4, MOE_DT_FP32 = range(4)
MOE_SCORING_SOFTMAX_RENORM, MOE_SCORING_SIGMOID = 0, 1
MOE_BLOCK_M = 128
# moe_activation_t, by the names of the "Fused Experts Kernels" table
ACTIVATIONS = {"silu": 0, "gelu": 1, "gelu_tanh": 2, "swigluoai": 3, "silu_no_mul": 4, "gelu_no_mul": 5}

# (name, argtypes, restype) of every exported entry point
_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class QuantConfig(ctypes.Structure):
    _fields_ = [("act", ctypes.c_int), ("act_group", ctypes.c_int), ("weight", ctypes.c_int),
                ("w_block_n", ctypes.c_int), ("w_block_k", ctypes.c_int)]


QC_BF16 = QuantConfig(MOE_DT_BF16, 0, MOE_DT_BF16, 0, 0)
QC_FP8 = QuantConfig(MOE_DT_FP8_E4M3, 128, MOE_DT_FP8_E4M3, 128, 128)
MOE_GROUP_TOKEN, MOE_GROUP_TENSOR = -1, -2
# quant names: "bf16"; "fp8" (G(128) activations); "fp8_token" ("A"); "fp8_tensor" ("T")
QUANT_CONFIGS = {
    "bf16": QC_BF16,
    "fp8": QC_FP8,
    "fp8_token": QuantConfig(MOE_DT_FP8_E4M3, MOE_GROUP_TOKEN, MOE_DT_FP8_E4M3, 128, 128),
    "fp8_tensor": QuantConfig(MOE_DT_FP8_E4M3, MOE_GROUP_TENSOR, MOE_DT_FP8_E4M3, 128, 128),
}


def _qc(quant: str) -> QuantConfig:
    if quant not in QUANT_CONFIGS:
        raise ValueError(f"unknown quantisation {quant!r}")
    return QUANT_CONFIGS[quant]


def scale_shape(quant: str, T: int, H: int):
    """Shape of a1q_scale for each fp8 format (None for bf16)."""
    return {"bf16": None, "fp8": (T, H // 128), "fp8_token": (T,), "fp8_tensor": (1,)}[quant]
_QCP = ctypes.POINTER(QuantConfig)


class ExpertsProblem(ctypes.Structure):
    """moe_experts_problem: one expert problem of a moe_experts_multi call."""
    _fields_ = [("a1q", ctypes.c_void_p), ("a1q_scale", ctypes.c_void_p), ("w13", ctypes.c_void_p),
                ("w13_scale", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("w2_scale", ctypes.c_void_p),
                ("expert_offsets", ctypes.c_void_p), ("sorted_slot", ctypes.c_void_p), ("tile_map", ctypes.c_void_p),
                ("num_tiles", ctypes.c_void_p), ("T", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
                ("top_k", ctypes.c_int), ("fused_expert_output", ctypes.c_void_p)]


_EPP = ctypes.POINTER(ExpertsProblem)

SIGNATURES = {
    "moe_route": ([_P, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_align": ([_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _Z, _P], _I),
    "moe_align_workspace_size": ([_I, _I, _I], _Z),
    "moe_align_noalloc": ([_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
    "moe_tile_map_capacity": ([_I, _I, _I], _I),
    "moe_prepare": ([_P, _P, _P, _I, _I, _I, _I, _QCP, _P, _P, _P], _I),
    "moe_experts": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _QCP, _P, _P, _Z, _P], _I),
    "moe_experts_act": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _QCP, _I, _P, _P, _Z, _P], _I),
    "moe_experts_multi": ([_EPP, _I, _I, _QCP, _I, _P, _Z, _P], _I),
    "moe_workspace_size_multi": ([_EPP, _I, _I, _QCP], _Z),
    "moe_workspace_size": ([_I, _I, _I, _I, _I, _QCP], _Z),
    "moe_workspace_intermediate": ([_I, _I, _I, _I, _I, _QCP, _P, _P, _P], _I),
    "moe_workspace_intermediate_nvfp4": ([_I, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_prepare_nvfp4": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_experts_nvfp4": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P,
                           _Z, _P], _I),
    "moe_workspace_size_nvfp4": ([_I, _I, _I, _I, _I], _Z),
    "moe_layer_fused": ([_P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _F, _P, _P, _P, _P, _Z, _P], _I),
    "moe_layer_fused_workspace_size": ([_I, _I, _I, _I, _I, _I], _Z),
    "moe_finalize": ([_P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _P, _F, _P, _P], _I),
    "moe_prepare_batched_workspace_size": ([_I, _I, _QCP], _Z),
    "moe_prepare_batched": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _QCP, _P, _P, _P, _P, _Z, _P], _I),
    "moe_workspace_size_batched": ([_I, _I, _I, _I, _QCP], _Z),
    "moe_experts_batched": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _QCP, _I, _P, _P, _Z, _P], _I),
    "moe_finalize_batched": ([_P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _P, _F, _P, _P], _I),
    "moe_device_status": ([_I], _I),
    "moe_selftest_wait_timeout": ([ctypes.c_uint64, _P], _I),
    "moe_selftest_row_division": ([ctypes.c_longlong, ctypes.c_uint32, _P, _P], _I),
    "moe_status_string": ([_I], ctypes.c_char_p),
}

_lib_handle = None


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} (status {status})")


def lib():
    """Load libmoe.so (built by ``mixture_experts_layer_tokens_gb300.build``).

    Raises if the library is missing: there is no CPU or PyTorch fallback."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m mixture_experts_layer_tokens_gb300.build` (nvcc, sm_103a)")
        h = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(h, name)
            f.argtypes = args
            f.restype = res
        _lib_handle = h
    return _lib_handle


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: Optional[torch.Tensor], dtype, name: str, cuda: bool = True):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if cuda and not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")


# ------------------------------------------------------------------ entry points
def moe_route(logits: torch.Tensor, top_k: int, scoring: int = MOE_SCORING_SOFTMAX_RENORM,
              topk_ids: Optional[torch.Tensor] = None, topk_weights: Optional[torch.Tensor] = None,
              stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    _need(logits, torch.float32, "logits")
    T, E = logits.shape
    if topk_ids is None:
        topk_ids = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    if topk_weights is None:
        topk_weights = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    _need(topk_ids, torch.int32, "topk_ids")
    _need(topk_weights, torch.float32, "topk_weights")
    _check("moe_route", lib().moe_route(_ptr(logits), T, E, top_k, scoring, _ptr(topk_ids), _ptr(topk_weights),
                                        _stream(stream)))
    return topk_ids, topk_weights


def align_workspace_size(T: int, top_k: int, E: int) -> int:
    return int(lib().moe_align_workspace_size(T, top_k, E))


def tile_map_capacity(num_slots: int, E: int, block_m: int = MOE_BLOCK_M) -> int:
    return int(lib().moe_tile_map_capacity(num_slots, E, block_m))


class Alignment:
    """Device buffers written by moe_align."""

    def __init__(self, T: int, top_k: int, E: int, device, block_m: int = MOE_BLOCK_M):
        S = T * top_k
        self.T, self.top_k, self.E, self.block_m = T, top_k, E, block_m
        self.expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=device)
        self.sorted_slot = torch.empty(max(S, 1), dtype=torch.int32, device=device)
        self.inv_slot = torch.empty(max(S, 1), dtype=torch.int32, device=device)
        self.tile_map = torch.empty((max(tile_map_capacity(S, E, block_m), 1), 2), dtype=torch.int32, device=device)
        self.num_tiles = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws = torch.empty(max(align_workspace_size(T, top_k, E), 16), dtype=torch.uint8, device=device)


def moe_align(topk_ids: torch.Tensor, E: int, block_m: int = MOE_BLOCK_M, out: Optional[Alignment] = None,
              stream=None) -> Alignment:
    _need(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    al = out if out is not None else Alignment(T, k, E, topk_ids.device, block_m)
    _check("moe_align", lib().moe_align(_ptr(topk_ids), T, k, E, block_m, _ptr(al.expert_offsets),
                                        _ptr(al.sorted_slot), _ptr(al.inv_slot), _ptr(al.tile_map),
                                        _ptr(al.num_tiles), _ptr(al.ws), al.ws.numel(), _stream(stream)))
    return al


ALIGN_NOALLOC_SCRATCH_BYTES = 256 * 1024


def moe_align_noalloc(topk_ids: torch.Tensor, E: int, out: Alignment, block_m: int = MOE_BLOCK_M,
                      stream=None) -> Alignment:
    """moe_align for callers that cannot allocate device memory at call time:
    the library's own fixed scratch array stands in for the workspace (out.ws
    is not used).  Calls that overlap on the GPU race on that array."""
    _need(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    _check("moe_align_noalloc", lib().moe_align_noalloc(
        _ptr(topk_ids), T, k, E, block_m, _ptr(out.expert_offsets), _ptr(out.sorted_slot), _ptr(out.inv_slot),
        _ptr(out.tile_map), _ptr(out.num_tiles), _stream(stream)))
    return out


def moe_prepare(a1: torch.Tensor, topk_weights: Optional[torch.Tensor], top_k: int,
                apply_router_weight_on_input: bool, quant: str, a1q: Optional[torch.Tensor] = None,
                a1q_scale: Optional[torch.Tensor] = None, topk_ids: Optional[torch.Tensor] = None,
                stream=None):
    """quant: "bf16" (no quantisation), "fp8" (E4M3, per-token 128-group scales
    [T, H/128]), "fp8_token" (one scale per token [T]) or "fp8_tensor" (one scale
    [1]).  Passing ``a1q=a1`` with bf16 and no weight is the passthrough (nothing runs)."""
    _need(a1, torch.bfloat16, "a1")
    _need(topk_weights, torch.float32, "topk_weights")
    T, H = a1.shape
    qc = _qc(quant)
    fp8 = quant != "bf16"
    if a1q is None:
        a1q = torch.empty((T, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=a1.device)
    if fp8 and a1q_scale is None:
        a1q_scale = torch.empty(scale_shape(quant, T, H), dtype=torch.float32, device=a1.device)
    _need(a1q, torch.uint8 if fp8 else torch.bfloat16, "a1q")
    _need(a1q_scale, torch.float32, "a1q_scale")
    _check("moe_prepare", lib().moe_prepare(_ptr(a1), _ptr(topk_weights), _ptr(topk_ids), T, H, top_k,
                                            int(bool(apply_router_weight_on_input)), ctypes.byref(qc), _ptr(a1q),
                                            _ptr(a1q_scale), _stream(stream)))
    return a1q, a1q_scale


def workspace_size(T: int, H: int, I: int, E: int, top_k: int, quant: str) -> int:
    return int(lib().moe_workspace_size(T, H, I, E, top_k, ctypes.byref(_qc(quant))))


def experts_intermediate(ws: torch.Tensor, T: int, H: int, I: int, E: int, top_k: int, quant: str):
    """Views into a moe_experts workspace of the intermediate h that the call left
    there (``moe_workspace_intermediate``): h [S, I] (bf16, or uint8 E4M3 codes for the
    fp8 formats) and its fp32 scales -- G(128): [I/128, S] (transposed, row stride
    s_pad), "A"/"T": [S] -- or None for bf16.  S = T * top_k rows in expert order."""
    off, soff, stride = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_int()
    _check("moe_workspace_intermediate", lib().moe_workspace_intermediate(
        T, H, I, E, top_k, ctypes.byref(_qc(quant)), ctypes.byref(off), ctypes.byref(soff), ctypes.byref(stride)))
    S = T * top_k
    fp8 = quant != "bf16"
    esz = 1 if fp8 else 2
    h = ws[off.value:off.value + S * I * esz]
    h = h.view(S, I) if fp8 else h.view(torch.bfloat16).view(S, I)
    if not fp8:
        return h, None
    if quant == "fp8":
        n = (I // 128) * stride.value
        sc = ws[soff.value:soff.value + 4 * n].view(torch.float32).view(I // 128, stride.value)[:, :S]
    else:
        sc = ws[soff.value:soff.value + 4 * S].view(torch.float32)
    return h, sc


def experts_intermediate_nvfp4(ws: torch.Tensor, T: int, H: int, I: int, E: int, top_k: int):
    """Views into a moe_experts_nvfp4 workspace (``moe_workspace_intermediate_nvfp4``):
    the bf16 h [S, I] of the first GEMM and its NVFP4 codes [S, I/2] and scale codes
    [S, I/16] that the second GEMM read."""
    hb, hq, hsf = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check("moe_workspace_intermediate_nvfp4", lib().moe_workspace_intermediate_nvfp4(
        T, H, I, E, top_k, ctypes.byref(hb), ctypes.byref(hq), ctypes.byref(hsf)))
    S = T * top_k
    return (ws[hb.value:hb.value + S * I * 2].view(torch.bfloat16).view(S, I),
            ws[hq.value:hq.value + S * I // 2].view(S, I // 2),
            ws[hsf.value:hsf.value + S * I // 16].view(S, I // 16))


def moe_experts(a1q: torch.Tensor, a1q_scale: Optional[torch.Tensor], w13: torch.Tensor,
                w13_scale: Optional[torch.Tensor], w2: torch.Tensor, w2_scale: Optional[torch.Tensor],
                al: Alignment, quant: str, out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                identity: bool = False, stream=None, activation: str = "silu") -> torch.Tensor:
    """Grouped expert MLPs (``moe_experts_act``; SiLU-and-mul by default, see
    ``ACTIVATIONS``; the *_no_mul activations take w13 [E, I, H]).
    ``identity=True`` (E == 1, top_k == 1) passes a NULL sorted_slot: rows are
    the tokens in order."""
    if activation not in ACTIVATIONS:
        raise ValueError(f"unknown activation {activation!r}")
    fp8 = quant != "bf16"
    _need(a1q, torch.uint8 if fp8 else torch.bfloat16, "a1q")
    _need(w13, torch.uint8 if fp8 else torch.bfloat16, "w13")
    _need(w2, torch.uint8 if fp8 else torch.bfloat16, "w2")
    for t, n in ((a1q_scale, "a1q_scale"), (w13_scale, "w13_scale"), (w2_scale, "w2_scale")):
        _need(t, torch.float32, n)
    T, H = a1q.shape
    E, rows13, _ = w13.shape
    I = rows13 if activation.endswith("_no_mul") else rows13 // 2
    k = al.top_k
    if out is None:
        out = torch.empty((T * k, H), dtype=torch.bfloat16, device=a1q.device)
    _need(out, torch.bfloat16, "fused_expert_output")
    if ws is None:
        ws = torch.empty(max(workspace_size(T, H, I, E, k, quant), 16), dtype=torch.uint8, device=a1q.device)
    qc = _qc(quant)
    _check("moe_experts_act", lib().moe_experts_act(
        _ptr(a1q), _ptr(a1q_scale), _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(al.expert_offsets),
        None if identity else _ptr(al.sorted_slot), _ptr(al.tile_map), _ptr(al.num_tiles), T, H, I, E, k,
        ctypes.byref(qc), ACTIVATIONS[activation], _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def experts_problem(a1q: torch.Tensor, a1q_scale: Optional[torch.Tensor], w13: torch.Tensor,
                    w13_scale: Optional[torch.Tensor], w2: torch.Tensor, w2_scale: Optional[torch.Tensor],
                    al: Alignment, out: torch.Tensor, identity: bool = False,
                    activation: str = "silu") -> ExpertsProblem:
    """One problem of moe_experts_multi (``identity``: NULL sorted_slot, E == 1, top_k == 1)."""
    T = a1q.shape[0]
    E, rows13, _ = w13.shape
    I = rows13 if activation.endswith("_no_mul") else rows13 // 2
    prob = ExpertsProblem(_ptr(a1q), _ptr(a1q_scale), _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale),
                          _ptr(al.expert_offsets), None if identity else _ptr(al.sorted_slot), _ptr(al.tile_map),
                          _ptr(al.num_tiles), T, I, E, al.top_k, _ptr(out))
    # the struct holds raw device pointers: keep the tensors alive as long as it is
    prob._tensors = (a1q, a1q_scale, w13, w13_scale, w2, w2_scale, al, out)
    return prob


def workspace_size_multi(problems, H: int, quant: str) -> int:
    arr = (ExpertsProblem * len(problems))(*problems)
    return int(lib().moe_workspace_size_multi(arr, len(problems), H, ctypes.byref(_qc(quant))))


def moe_experts_multi(problems, H: int, quant: str, ws: torch.Tensor, activation: str = "silu", stream=None):
    """Several expert problems (``experts_problem``) in the same GEMM launches."""
    if activation not in ACTIVATIONS:
        raise ValueError(f"unknown activation {activation!r}")
    arr = (ExpertsProblem * len(problems))(*problems)
    _check("moe_experts_multi", lib().moe_experts_multi(arr, len(problems), H, ctypes.byref(_qc(quant)),
                                                        ACTIVATIONS[activation], _ptr(ws), ws.numel(),
                                                        _stream(stream)))


def _gscale(g, device, name):
    """A global scale as the device fp32 tensor the C ABI takes (a Python number is copied)."""
    if isinstance(g, torch.Tensor):
        _need(g, torch.float32, name)
        return g
    return torch.tensor([float(g)], dtype=torch.float32, device=device)


def moe_prepare_nvfp4(a1: torch.Tensor, topk_weights: Optional[torch.Tensor], top_k: int,
                      apply_router_weight_on_input: bool, a1_gscale, a1q: Optional[torch.Tensor] = None,
                      a1q_sf: Optional[torch.Tensor] = None, stream=None):
    """NVFP4 prepare: a1 [T, H] bf16 -> (a1q [T, H/2] codes, a1q_sf [T, H/16] scale
    codes) with global scale ``a1_gscale`` (number or [1] fp32 device tensor)."""
    _need(a1, torch.bfloat16, "a1")
    _need(topk_weights, torch.float32, "topk_weights")
    T, H = a1.shape
    g = _gscale(a1_gscale, a1.device, "a1_gscale")
    if a1q is None:
        a1q = torch.empty((T, H // 2), dtype=torch.uint8, device=a1.device)
    if a1q_sf is None:
        a1q_sf = torch.empty((T, H // 16), dtype=torch.uint8, device=a1.device)
    _need(a1q, torch.uint8, "a1q")
    _need(a1q_sf, torch.uint8, "a1q_sf")
    _check("moe_prepare_nvfp4", lib().moe_prepare_nvfp4(
        _ptr(a1), _ptr(topk_weights), T, H, top_k, int(bool(apply_router_weight_on_input)), _ptr(g), _ptr(a1q),
        _ptr(a1q_sf), _stream(stream)))
    return a1q, a1q_sf


def workspace_size_nvfp4(T: int, H: int, I: int, E: int, top_k: int) -> int:
    return int(lib().moe_workspace_size_nvfp4(T, H, I, E, top_k))


def moe_experts_nvfp4(a1q: torch.Tensor, a1q_sf: torch.Tensor, a1_gscale, w13: torch.Tensor,
                      w13_sf: torch.Tensor, w13_gscale: torch.Tensor, w2: torch.Tensor, w2_sf: torch.Tensor,
                      w2_gscale: torch.Tensor, h_gscale, al: Alignment, out: Optional[torch.Tensor] = None,
                      ws: Optional[torch.Tensor] = None, identity: bool = False, stream=None,
                      activation: str = "silu") -> torch.Tensor:
    """Grouped expert MLPs with NVFP4 operands (``moe_experts_nvfp4``): packed codes
    a1q [T, H/2], w13 [E, 2I, H/2] (*_no_mul: [E, I, H/2]), w2 [E, H, I/2] with
    their scale codes (one per 16 elements) and fp32 global scales."""
    if activation not in ACTIVATIONS:
        raise ValueError(f"unknown activation {activation!r}")
    for t, n in ((a1q, "a1q"), (a1q_sf, "a1q_sf"), (w13, "w13"), (w13_sf, "w13_sf"), (w2, "w2"), (w2_sf, "w2_sf")):
        _need(t, torch.uint8, n)
    _need(w13_gscale, torch.float32, "w13_gscale")
    _need(w2_gscale, torch.float32, "w2_gscale")
    T, H = a1q.shape[0], a1q.shape[1] * 2
    E, rows13, _ = w13.shape
    I = rows13 if activation.endswith("_no_mul") else rows13 // 2
    k = al.top_k
    ga = _gscale(a1_gscale, a1q.device, "a1_gscale")
    gh = _gscale(h_gscale, a1q.device, "h_gscale")
    if out is None:
        out = torch.empty((T * k, H), dtype=torch.bfloat16, device=a1q.device)
    _need(out, torch.bfloat16, "fused_expert_output")
    if ws is None:
        ws = torch.empty(max(workspace_size_nvfp4(T, H, I, E, k), 16), dtype=torch.uint8, device=a1q.device)
    _check("moe_experts_nvfp4", lib().moe_experts_nvfp4(
        _ptr(a1q), _ptr(a1q_sf), _ptr(ga), _ptr(w13), _ptr(w13_sf), _ptr(w13_gscale), _ptr(w2), _ptr(w2_sf),
        _ptr(w2_gscale), _ptr(gh), _ptr(al.expert_offsets), None if identity else _ptr(al.sorted_slot),
        _ptr(al.tile_map), _ptr(al.num_tiles), T, H, I, E, k, ACTIVATIONS[activation], _ptr(out), _ptr(ws),
        ws.numel(), _stream(stream)))
    return out


def layer_fused_workspace_size(T: int, H: int, I: int, E: int, top_k: int, has_shared: bool) -> int:
    return int(lib().moe_layer_fused_workspace_size(T, H, I, E, top_k, int(bool(has_shared))))


def moe_layer_fused(logits: torch.Tensor, a1: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor, top_k: int,
                    scoring: int = MOE_SCORING_SOFTMAX_RENORM, apply_router_weight_on_input: bool = False,
                    shared_w13: Optional[torch.Tensor] = None, shared_w2: Optional[torch.Tensor] = None,
                    residual: Optional[torch.Tensor] = None, rms_weight: Optional[torch.Tensor] = None,
                    eps: float = 1e-6, topk_ids: Optional[torch.Tensor] = None,
                    topk_weights: Optional[torch.Tensor] = None, output: Optional[torch.Tensor] = None,
                    ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The whole bf16 layer step in one launch (``moe_layer_fused``): w13 [E, 2I, H],
    w2 [E, H, I]; shared_w13 [2I, H] / shared_w2 [H, I] (or [1, ...]) for a shared expert."""
    _need(logits, torch.float32, "logits")
    for t, n in ((a1, "a1"), (w13, "w13"), (w2, "w2"), (shared_w13, "shared_w13"), (shared_w2, "shared_w2"),
                 (residual, "residual"), (rms_weight, "rms_weight")):
        _need(t, torch.bfloat16, n)
    T, H = a1.shape
    E, rows13, _ = w13.shape
    I = rows13 // 2
    dev = a1.device
    if topk_ids is None:
        topk_ids = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty((T, top_k), dtype=torch.float32, device=dev)
    if output is None:
        output = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = torch.empty(max(layer_fused_workspace_size(T, H, I, E, top_k, shared_w13 is not None), 16),
                         dtype=torch.uint8, device=dev)
    _check("moe_layer_fused", lib().moe_layer_fused(
        _ptr(logits), _ptr(a1), T, H, I, E, top_k, scoring, int(bool(apply_router_weight_on_input)), _ptr(w13),
        _ptr(w2), _ptr(shared_w13), _ptr(shared_w2), _ptr(residual), _ptr(rms_weight), eps, _ptr(topk_ids),
        _ptr(topk_weights), _ptr(output), _ptr(ws), ws.numel(), _stream(stream)))
    return output


def moe_finalize(fused_expert_output: torch.Tensor, topk_weights: Optional[torch.Tensor], top_k: int,
                 apply_router_weight_on_input: bool = False, shared: Optional[torch.Tensor] = None,
                 residual: Optional[torch.Tensor] = None, rms_weight: Optional[torch.Tensor] = None,
                 eps: float = 1e-6, out_dtype: int = MOE_DT_BF16, out_global_scale: float = 1.0,
                 output: Optional[torch.Tensor] = None, out_scale: Optional[torch.Tensor] = None,
                 residual_out: Optional[torch.Tensor] = None, topk_ids: Optional[torch.Tensor] = None,
                 stream=None):
    _need(fused_expert_output, torch.bfloat16, "fused_expert_output")
    _need(topk_weights, torch.float32, "topk_weights")
    for t, n in ((shared, "shared"), (residual, "residual"), (rms_weight, "rms_weight"),
                 (residual_out, "residual_out")):
        _need(t, torch.bfloat16, n)
    S, H = fused_expert_output.shape
    T = S // top_k
    dev = fused_expert_output.device
    if output is None:
        if out_dtype == MOE_DT_NVFP4:
            output = torch.empty((T, H // 2), dtype=torch.uint8, device=dev)
        else:
            output = torch.empty((T, H), dtype=torch.float32 if out_dtype == MOE_DT_FP32 else torch.bfloat16,
                                 device=dev)
    if out_dtype == MOE_DT_NVFP4 and out_scale is None:
        out_scale = torch.empty((T, H // 16), dtype=torch.uint8, device=dev)
    _check("moe_finalize", lib().moe_finalize(
        _ptr(output), _ptr(fused_expert_output), _ptr(topk_weights), _ptr(topk_ids), _ptr(shared), _ptr(residual),
        _ptr(rms_weight), float(eps), T, H, top_k, int(bool(apply_router_weight_on_input)), out_dtype,
        _ptr(out_scale), float(out_global_scale), _ptr(residual_out), _stream(stream)))
    return output, out_scale


def moe_device_status(clear: bool = True) -> int:
    return int(lib().moe_device_status(int(clear)))


def moe_selftest_row_division(n: int, seed: int, stream=None) -> int:
    """Run the library's self-test of the requantisation division (see moe.h) on n
    pairs; returns how many results differ from the IEEE division."""
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    _check("moe_selftest_row_division",
           lib().moe_selftest_row_division(int(n), int(seed) & 0xFFFFFFFF, _ptr(cnt), _stream(stream)))
    return int(cnt.item())


def moe_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Launch the library's self-test of a device-side wait that runs out (see moe.h):
    afterwards moe_device_status() reports MOE_ERR_TIMEOUT."""
    _check("moe_selftest_wait_timeout", lib().moe_selftest_wait_timeout(int(limit_ns), _stream(stream)))


# ------------------------------------------------------------------ batched activation format
def batched_scale_shape(quant: str, E: int, M: int, H: int):
    """Shape of a1q_b_scale in the batched format (None for bf16)."""
    return {"bf16": None, "fp8": (E, M, H // 128), "fp8_token": (E, M), "fp8_tensor": (1,)}[quant]


def moe_prepare_batched(a1: torch.Tensor, topk_weights: Optional[torch.Tensor], al: "Alignment", E: int,
                        max_tokens: int, apply_router_weight_on_input: bool, quant: str, stream=None):
    """Prepare into the batched format (``moe_prepare_batched``): returns (a1q_b
    [E, max_tokens, H], a1q_b_scale or None, expert_num_tokens [E] int32)."""
    _need(a1, torch.bfloat16, "a1")
    T, H = a1.shape
    fp8 = quant != "bf16"
    qb = torch.empty((E, max_tokens, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=a1.device)
    shp = batched_scale_shape(quant, E, max_tokens, H)
    sb = None if shp is None else torch.empty(shp, dtype=torch.float32, device=a1.device)
    counts = torch.empty((E,), dtype=torch.int32, device=a1.device)
    qc = _qc(quant)
    nws = int(lib().moe_prepare_batched_workspace_size(T, H, ctypes.byref(qc)))
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=a1.device)
    _check("moe_prepare_batched", lib().moe_prepare_batched(
        _ptr(a1), _ptr(topk_weights), _ptr(al.expert_offsets), _ptr(al.sorted_slot), T, H, al.top_k, E, max_tokens,
        int(apply_router_weight_on_input), ctypes.byref(qc), _ptr(qb), _ptr(sb), _ptr(counts), _ptr(ws), ws.numel(),
        _stream(stream)))
    return qb, sb, counts


def workspace_size_batched(E: int, max_tokens: int, H: int, I: int, quant: str) -> int:
    return int(lib().moe_workspace_size_batched(E, max_tokens, H, I, ctypes.byref(_qc(quant))))


def moe_experts_batched(a1q_b: torch.Tensor, a1q_b_scale: Optional[torch.Tensor], w13: torch.Tensor,
                        w13_scale: Optional[torch.Tensor], w2: torch.Tensor, w2_scale: Optional[torch.Tensor],
                        expert_num_tokens: torch.Tensor, quant: str, out: Optional[torch.Tensor] = None,
                        ws: Optional[torch.Tensor] = None, activation: str = "silu", stream=None) -> torch.Tensor:
    """The experts on the batched format (``moe_experts_batched``): out [E, max_tokens, H] bf16."""
    if activation not in ACTIVATIONS:
        raise ValueError(f"unknown activation {activation!r}")
    E, M, H = a1q_b.shape
    _, rows13, _ = w13.shape
    I = rows13 if activation.endswith("_no_mul") else rows13 // 2
    _need(expert_num_tokens, torch.int32, "expert_num_tokens")
    if out is None:
        out = torch.empty((E, M, H), dtype=torch.bfloat16, device=a1q_b.device)
    if ws is None:
        ws = torch.empty(max(workspace_size_batched(E, M, H, I, quant), 16), dtype=torch.uint8, device=a1q_b.device)
    _check("moe_experts_batched", lib().moe_experts_batched(
        _ptr(a1q_b), _ptr(a1q_b_scale), _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(expert_num_tokens),
        E, M, H, I, ctypes.byref(_qc(quant)), ACTIVATIONS[activation], _ptr(out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def moe_finalize_batched(out_b: torch.Tensor, topk_weights: Optional[torch.Tensor], topk_ids: torch.Tensor,
                         al: "Alignment", apply_router_weight_on_input: bool, shared=None, residual=None,
                         rms_weight=None, eps: float = 1e-6, output: Optional[torch.Tensor] = None,
                         residual_out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """moe_finalize reading each slot's row from a batched output [E, max_tokens, H]
    (``moe_finalize_batched``); bf16 output [T, H]."""
    E, M, H = out_b.shape
    T, k = topk_ids.shape
    if output is None:
        output = torch.empty((T, H), dtype=torch.bfloat16, device=out_b.device)
    _check("moe_finalize_batched", lib().moe_finalize_batched(
        _ptr(output), _ptr(out_b), M, _ptr(topk_weights), _ptr(topk_ids), _ptr(al.inv_slot), _ptr(al.expert_offsets),
        _ptr(shared), _ptr(residual), _ptr(rms_weight), eps, T, H, k, int(apply_router_weight_on_input), MOE_DT_BF16,
        None, 1.0, _ptr(residual_out), _stream(stream)))
    return output
