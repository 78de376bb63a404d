"""C-ABI checks that need no GPU: the library loads, exports every entry point
the header declares, and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_tokens_gb300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_entry_point(moelib):
    names = _declared()
    assert "moe_route" in names and "moe_finalize" in names and len(names) >= 10
    for n in names:
        assert hasattr(moelib, n), n
    assert set(names) == set(moe.SIGNATURES)


def test_status_strings(moelib):
    assert moe.status_string(moe.MOE_OK) == "ok"
    assert "workspace" in moe.status_string(moe.MOE_ERR_WORKSPACE)
    assert moe.status_string(99) == "unknown status"


def test_sizes(moelib):
    assert moe.tile_map_capacity(0, 8) == 0
    assert moe.tile_map_capacity(32768, 256) == 510
    assert moe.tile_map_capacity(10, 8) == 8    # at most one tile per non-empty expert
    assert moe.tile_map_capacity(5, 8) == 5
    assert moe.tile_map_capacity(1024, 8) == (1024 + 8 * 127) // 128
    assert moe.align_workspace_size(4096, 8, 256) == 16 * 256 * 4
    fp8 = moe.workspace_size(4096, 7168, 2048, 256, 8, "fp8")
    S = 32768
    assert fp8 >= S * 7168 + S * 2048 + (7168 // 128 + 2048 // 128) * S * 4
    assert moe.workspace_size(512, 4096, 14336, 8, 2, "bf16") >= 1024 * 4096 * 2 + 1024 * 14336 * 2


P = ctypes.c_void_p
FAKE = P(256)  # never dereferenced: every call below fails its host-side checks


def test_route_rejects_bad_arguments(moelib):
    L = moelib
    assert L.moe_route(FAKE, 4, 0, 1, 0, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG        # E = 0
    assert L.moe_route(FAKE, 4, 8, 9, 0, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG        # k > E
    assert L.moe_route(FAKE, 4, 64, 33, 0, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG      # k > 32
    assert L.moe_route(FAKE, 4, 2048, 2, 0, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG     # E > 1024
    assert L.moe_route(FAKE, 4, 8, 2, 1, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG        # sigmoid needs k 1
    assert L.moe_route(FAKE, 4, 8, 2, 7, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG        # scoring
    assert L.moe_route(None, 4, 8, 2, 0, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG        # null logits
    assert L.moe_route(None, 0, 8, 2, 0, None, None, None) == moe.MOE_OK                     # T = 0: no-op


def test_align_rejects_bad_arguments(moelib):
    L = moelib
    ok = [FAKE, 16, 2, 8, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None]
    bad = list(ok); bad[3] = 0
    assert L.moe_align(*bad) == moe.MOE_ERR_INVALID_ARG
    bad = list(ok); bad[3] = 4096
    assert L.moe_align(*bad) == moe.MOE_ERR_INVALID_ARG
    bad = list(ok); bad[4] = 0
    assert L.moe_align(*bad) == moe.MOE_ERR_INVALID_ARG
    bad = list(ok); bad[10] = None
    assert L.moe_align(*bad) == moe.MOE_ERR_WORKSPACE
    bad = list(ok); bad[11] = 4
    assert L.moe_align(*bad) == moe.MOE_ERR_WORKSPACE
    bad = list(ok); bad[6] = None
    assert L.moe_align(*bad) == moe.MOE_ERR_INVALID_ARG


def test_prepare_rejects_bad_arguments(moelib):
    L = moelib
    qb, q8 = ctypes.byref(moe.QC_BF16), ctypes.byref(moe.QC_FP8)
    # apply_router_weight_on_input needs top_k == 1 (the pages' `assert topk == 1`)
    assert L.moe_prepare(FAKE, FAKE, None, 4, 256, 2, 1, qb, FAKE, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_prepare(FAKE, FAKE, None, 4, 200, 1, 0, q8, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG  # H%128
    assert L.moe_prepare(FAKE, FAKE, None, 4, 256, 1, 0, q8, FAKE, None, None) == moe.MOE_ERR_INVALID_ARG  # scale
    assert L.moe_prepare(P(258), FAKE, None, 4, 256, 1, 1, qb, FAKE, None, None) == moe.MOE_ERR_INVALID_ARG  # align
    nv = moe.QuantConfig(moe.MOE_DT_NVFP4, 16, moe.MOE_DT_NVFP4, 0, 0)
    assert L.moe_prepare(FAKE, FAKE, None, 4, 256, 1, 0, ctypes.byref(nv), FAKE, FAKE, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_prepare(FAKE, FAKE, None, 4, 256, 1, 0, None, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG


def test_experts_rejects_bad_arguments(moelib):
    L = moelib
    qb, q8 = ctypes.byref(moe.QC_BF16), ctypes.byref(moe.QC_FP8)

    def call(T=16, H=256, I=512, E=8, k=2, qc=qb, ws=FAKE, wsb=1 << 30, slot=FAKE, sc=FAKE):
        return L.moe_experts(FAKE, sc, FAKE, sc, FAKE, sc, FAKE, slot, FAKE, FAKE, T, H, I, E, k, qc,
                             FAKE, ws, wsb, None)

    assert call(H=200) == moe.MOE_ERR_INVALID_ARG
    assert call(I=100) == moe.MOE_ERR_INVALID_ARG
    assert call(k=9) == moe.MOE_ERR_INVALID_ARG
    assert call(ws=None) == moe.MOE_ERR_WORKSPACE
    assert call(wsb=1000) == moe.MOE_ERR_WORKSPACE
    assert call(slot=None) == moe.MOE_ERR_INVALID_ARG            # identity needs E == 1 and k == 1
    assert call(qc=q8, sc=None) == moe.MOE_ERR_INVALID_ARG        # fp8 needs scales
    mixed = moe.QuantConfig(moe.MOE_DT_FP8_E4M3, 128, moe.MOE_DT_BF16, 0, 0)
    assert call(qc=ctypes.byref(mixed)) == moe.MOE_ERR_UNSUPPORTED
    assert call(T=0) == moe.MOE_OK


def test_finalize_rejects_bad_arguments(moelib):
    L = moelib

    def call(T=4, H=256, k=2, won=0, odt=moe.MOE_DT_BF16, sc=FAKE, g=1.0, w=FAKE, eps=1e-6):
        return L.moe_finalize(FAKE, FAKE, w, None, None, None, None, eps, T, H, k, won, odt, sc, g, None, None)

    assert call(H=12) == moe.MOE_ERR_INVALID_ARG
    assert call(k=0) == moe.MOE_ERR_INVALID_ARG
    assert call(odt=moe.MOE_DT_FP8_E4M3) == moe.MOE_ERR_INVALID_ARG
    assert call(odt=moe.MOE_DT_NVFP4, H=264) == moe.MOE_ERR_INVALID_ARG
    assert call(odt=moe.MOE_DT_NVFP4, g=0.0) == moe.MOE_ERR_INVALID_ARG
    assert call(odt=moe.MOE_DT_NVFP4, sc=None) == moe.MOE_ERR_INVALID_ARG
    assert call(w=None) == moe.MOE_ERR_INVALID_ARG
    assert call(eps=-1.0) == moe.MOE_ERR_INVALID_ARG
    assert call(T=0) == moe.MOE_OK


def test_experts_act_rejects_unknown_activation(moelib):
    L = moelib
    qb = ctypes.byref(moe.QC_BF16)

    def call(act, T=16):
        return L.moe_experts_act(FAKE, None, FAKE, None, FAKE, None, FAKE, FAKE, FAKE, FAKE, T, 256, 512, 8, 2, qb,
                                 act, FAKE, FAKE, 1 << 30, None)

    assert call(-1) == moe.MOE_ERR_UNSUPPORTED
    assert call(6) == moe.MOE_ERR_UNSUPPORTED
    assert call(moe.ACTIVATIONS["gelu"], T=0) == moe.MOE_OK   # nothing to do, no launch
    assert sorted(moe.ACTIVATIONS.values()) == list(range(6))


def test_experts_multi_rejects_what_it_cannot_fuse(moelib):
    L = moelib
    P = moe.ExpertsProblem

    def prob(I, T=4):
        return P(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, T, I, 8, 1, FAKE)

    two = (P * 2)(prob(256), prob(512))
    assert L.moe_experts_multi(two, 2, 256, ctypes.byref(moe.QC_BF16), 0, FAKE, 1 << 30, None) == \
        moe.MOE_ERR_UNSUPPORTED                      # the second GEMM's depth differs
    same = (P * 2)(prob(256), prob(256))
    assert L.moe_experts_multi(same, 2, 256, ctypes.byref(moe.QC_FP8), 0, FAKE, 1 << 30, None) == \
        moe.MOE_ERR_UNSUPPORTED                      # fp8 problems run one per call
    assert L.moe_experts_multi(same, 3, 256, ctypes.byref(moe.QC_BF16), 0, FAKE, 1 << 30, None) == \
        moe.MOE_ERR_INVALID_ARG
    empty = (P * 2)(prob(256, T=0), prob(512, T=0))
    assert L.moe_experts_multi(empty, 2, 256, ctypes.byref(moe.QC_BF16), 0, FAKE, 1 << 30, None) == moe.MOE_OK


def test_nvfp4_entry_points_reject_bad_arguments(moelib):
    L = moelib
    G = FAKE  # a global-scale pointer

    def experts(T=16, H=256, I=512, E=8, k=2, act=0, ws=FAKE, wsb=1 << 30, slot=FAKE, a=FAKE, asf=FAKE, out=FAKE):
        return L.moe_experts_nvfp4(a, asf, G, FAKE, FAKE, G, FAKE, FAKE, G, G, FAKE, slot, FAKE, FAKE, T, H, I, E,
                                   k, act, out, ws, wsb, None)

    assert experts(H=384) == moe.MOE_ERR_INVALID_ARG            # H % 256
    assert experts(I=128) == moe.MOE_ERR_INVALID_ARG            # I % 256
    assert experts(k=9) == moe.MOE_ERR_INVALID_ARG              # top_k > E
    assert experts(act=6) == moe.MOE_ERR_UNSUPPORTED            # unknown activation
    assert experts(a=None) == moe.MOE_ERR_INVALID_ARG
    assert experts(asf=P(264)) == moe.MOE_ERR_INVALID_ARG       # scale rows not 16-byte aligned
    assert experts(slot=None) == moe.MOE_ERR_INVALID_ARG        # identity needs E == 1 and k == 1
    assert experts(ws=None) == moe.MOE_ERR_WORKSPACE
    assert experts(wsb=1000) == moe.MOE_ERR_WORKSPACE
    assert experts(T=0, a=None, asf=None, out=None) == moe.MOE_OK

    def prepare(T=4, H=256, k=1, weight=0, w=FAKE, g=G, a1=FAKE):
        return L.moe_prepare_nvfp4(a1, w, T, H, k, weight, g, FAKE, FAKE, None)

    assert prepare(H=24) == moe.MOE_ERR_INVALID_ARG             # H % 16
    assert prepare(weight=1, k=2) == moe.MOE_ERR_INVALID_ARG    # weight on the input needs top_k == 1
    assert prepare(weight=1, w=None) == moe.MOE_ERR_INVALID_ARG
    assert prepare(g=None) == moe.MOE_ERR_INVALID_ARG
    assert prepare(a1=P(264)) == moe.MOE_ERR_INVALID_ARG        # bf16 rows not 16-byte aligned
    assert prepare(T=0, a1=None) == moe.MOE_OK


def test_nvfp4_workspace_size(moelib):
    assert moe.workspace_size_nvfp4(512, 384, 14336, 8, 2) == 0        # H % 256
    assert moe.workspace_size_nvfp4(512, 4096, 14000, 8, 2) == 0       # I % 256
    S, H, I = 1024, 4096, 14336
    # gathered codes and scale rows, bf16 h, h codes and scales
    need = S * H // 2 + S * H // 16 + S * I * 2 + S * I // 2 + S * I // 16
    assert moe.workspace_size_nvfp4(512, H, I, 8, 2) >= need
    assert moe.workspace_size_nvfp4(0, H, I, 8, 2) > 0                 # flags and partials only


def test_layer_fused_rejects_what_it_cannot_run(moelib):
    L = moelib

    def call(T=4, H=256, I=256, E=8, k=2, scoring=0, woi=0, sh13=FAKE, sh2=FAKE, ws=FAKE, wsb=1 << 30, a1=FAKE):
        return L.moe_layer_fused(FAKE, a1, T, H, I, E, k, scoring, woi, FAKE, FAKE, sh13, sh2, None, None,
                                 ctypes.c_float(1e-6), FAKE, FAKE, FAKE, ws, wsb, None)

    assert call(T=1025) == moe.MOE_ERR_UNSUPPORTED               # T * top_k > 2048
    assert call(E=512) == moe.MOE_ERR_UNSUPPORTED                # E > 256
    assert call(H=200) == moe.MOE_ERR_INVALID_ARG                # H % 128
    assert call(scoring=1) == moe.MOE_ERR_INVALID_ARG            # sigmoid needs top_k 1
    assert call(woi=1) == moe.MOE_ERR_INVALID_ARG                # weight on the input needs top_k 1
    assert call(sh2=None) == moe.MOE_ERR_INVALID_ARG             # shared weights: both or neither
    assert call(a1=P(264)) == moe.MOE_ERR_INVALID_ARG            # not 16-byte aligned
    assert call(ws=None) == moe.MOE_ERR_WORKSPACE
    assert call(T=0, a1=None) == moe.MOE_OK
    assert moe.layer_fused_workspace_size(4, 256, 256, 8, 2, True) > moe.layer_fused_workspace_size(4, 256, 256, 8, 2,
                                                                                                   False)
