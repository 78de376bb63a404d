"""Host-side logic that needs no GPU: the binding's argument handling and the
bench's traffic records (only while the recorded kernel sources match)."""
import importlib.util
import json
import os

import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_quant_and_activation_names():
    assert set(moe.QUANT_CONFIGS) == {"bf16", "fp8", "fp8_token", "fp8_tensor"}
    assert moe.QUANT_CONFIGS["fp8_token"].act_group == moe.MOE_GROUP_TOKEN == -1
    assert moe.QUANT_CONFIGS["fp8_tensor"].act_group == moe.MOE_GROUP_TENSOR == -2
    assert moe.scale_shape("fp8", 5, 256) == (5, 2)
    assert moe.scale_shape("fp8_token", 5, 256) == (5,)
    assert moe.scale_shape("fp8_tensor", 5, 256) == (1,)
    with pytest.raises(ValueError):
        moe._qc("int8")


def test_experts_problem_keeps_its_tensors_alive():
    a = torch.zeros(4, 256, dtype=torch.bfloat16)
    w13 = torch.zeros(2, 512, 256, dtype=torch.bfloat16)
    w2 = torch.zeros(2, 256, 256, dtype=torch.bfloat16)
    out = torch.zeros(4, 256, dtype=torch.bfloat16)

    class Al:  # the fields experts_problem reads
        expert_offsets = sorted_slot = tile_map = num_tiles = torch.zeros(4, dtype=torch.int32)
        top_k = 1
    p = moe.experts_problem(a, None, w13, None, w2, None, Al(), out)
    assert (p.T, p.I, p.E, p.top_k) == (4, 256, 2, 1)
    assert p.w13 == w13.data_ptr() and any(t is w13 for t in p._tensors)
    q = moe.experts_problem(a, None, w13[:, :256], None, w2, None, Al(), out, activation="gelu_no_mul")
    assert q.I == 256


def test_traffic_record_only_while_sources_match(tmp_path):
    b = _bench()
    rec = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
    for name, e in rec["workloads"].items():
        assert e["unit"] in b.UNIT_SOURCES and e["bytes_per_call"] > 0
    # a record whose hash matches the unit's current sources is reported, a stale one is not
    digest = b.sources_digest(b.UNIT_SOURCES["finalize"])
    fake = {"workloads": {"w_ok": {"unit": "finalize", "bytes_per_call": 123, "sources_sha256": digest},
                          "w_stale": {"unit": "finalize", "bytes_per_call": 456, "sources_sha256": "0" * 64}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(fake))
    assert b.measured_traffic("w_ok", str(path)) == 123
    assert b.measured_traffic("w_stale", str(path)) is None
    assert b.measured_traffic("absent", str(path)) is None


def test_graph_kernel_count_without_a_graph_is_none():
    b = _bench()

    class NoGraph:
        def raw_cuda_graph(self):
            raise RuntimeError("no graph")
    assert b.graph_kernel_nodes(NoGraph()) is None


def test_traffic_digest_ignores_comments_and_formatting_only():
    import bench
    a = 'int f(int x) { return x + 1; }  // one\n/* block\n comment */\nconst char* s = "a // b /* c */";\n'
    b = 'int f(int x) {\n  return x + 1;\n}\nconst char* s = "a // b /* c */";\n'
    c = 'int f(int x) { return x + 2; }\nconst char* s = "a // b /* c */";\n'
    assert bench.code_only(a) == bench.code_only(b)           # comments and layout do not count
    assert bench.code_only(a) != bench.code_only(c)           # code does
    assert '"a // b /* c */"' in bench.code_only(a)           # string literals are kept whole


def test_nvfp4_inputs_are_seeded_codes_in_their_ranges():
    from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, NVFP4_A1_GSCALE, NVFP4_H_GSCALE, make_inputs, scaled
    cfg = scaled(CONFIGS["mixtral_nvfp4"], T=4, H=256, I=256, E=3)
    a, b = make_inputs(cfg, seed=5), make_inputs(cfg, seed=5)
    assert torch.equal(a.w13, b.w13) and torch.equal(a.w2_scale, b.w2_scale)      # seeded
    assert a.w13.shape == (3, 512, 128) and a.w13_scale.shape == (3, 512, 16)
    assert a.w2.shape == (3, 256, 128) and a.w2_scale.shape == (3, 256, 16)
    for sf in (a.w13_scale, a.w2_scale):
        assert int(sf.min()) >= 0x40 and int(sf.max()) < 0x50                    # E4M3 2 .. 7.5
    assert a.extra["w13_gscale"].shape == (3,) and (a.extra["w13_gscale"] > 0).all()
    assert a.extra["a1_gscale"] == NVFP4_A1_GSCALE and a.extra["h_gscale"] == NVFP4_H_GSCALE


def test_bench_accounting_of_the_formats():
    import numpy as np
    import bench
    from mixture_experts_layer_tokens_gb300.inputs import CONFIGS
    counts = np.array([1, 0, 2, 1, 0, 0, 1, 1])
    b16, f16 = bench.experts_algorithmic(CONFIGS["mixtral"], counts)
    b4, f4 = bench.experts_algorithmic(CONFIGS["mixtral_nvfp4"], counts)
    touched, H, I = 5, 4096, 14336
    assert f16 == f4 == 2.0 * 3 * 512 * 2 * H * I                           # the same FLOPs
    weights = touched * 3 * H * I                                          # of the experts that got rows
    assert 2.0 < b16 / weights < 2.1                                        # 2 B per bf16 weight + activations
    assert 0.5625 < b4 / weights < 0.7                                      # 9/16 B per NVFP4 weight + activations
    assert bench.tensor_ratio("bf16") == 1 and bench.tensor_ratio("fp8") == 2 and bench.tensor_ratio("nvfp4") == 6
