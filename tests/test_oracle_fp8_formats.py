"""Pins of the oracle's "A" (per token) and "T" (per tensor) fp8 formats.

They reduce to the pinned G(128) quantiser where the formats coincide, keep the
e4m3 format's error bound, put every row's largest element on the top code, are
invariant under power-of-two rescaling, and the "T" intermediate of a layer is
one scale over all experts' rows."""
import numpy as np
import pytest
import torch

from oracle import codecs, moe_ref


def _x(R, C, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return codecs.round_bf16((torch.randn(R, C, generator=g, dtype=torch.float64) * scale).numpy())


def test_per_token_with_one_group_is_g128():
    x = _x(37, 128, 1, 3.0)
    q1, s1 = moe_ref.quantize_fp8_token(x)
    q2, s2 = moe_ref.quantize_fp8_g128(x)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2[:, 0])


def test_per_tensor_with_one_row_is_per_token():
    x = _x(1, 640, 2)
    q1, s1 = moe_ref.quantize_fp8_tensor(x)
    q2, s2 = moe_ref.quantize_fp8_token(x)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_per_tensor_scale_is_the_largest_row_scale():
    x = _x(50, 256, 3) * np.linspace(0.1, 4.0, 50)[:, None]
    _, st = moe_ref.quantize_fp8_tensor(x)
    _, sr = moe_ref.quantize_fp8_token(x)
    assert st[0] == sr.max()


@pytest.mark.parametrize("fmt", ["token", "tensor"])
def test_largest_element_takes_the_top_code_and_error_is_bounded(fmt):
    x = _x(64, 512, 4, 7.0)
    q, s = (moe_ref.quantize_fp8_token if fmt == "token" else moe_ref.quantize_fp8_tensor)(x)
    d = moe_ref.dequant_fp8(q, s, "fp8_" + fmt)
    sr = s.astype(np.float64)[:, None] if fmt == "token" else float(s[0])
    # e4m3 keeps 3 fraction bits: half a step is 2^-4 of a normal value; subnormal steps are 2^-9 s
    assert np.all(np.abs(d - x) <= 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * sr + 1e-12)
    top = np.abs(x).argmax(axis=1) if fmt == "token" else None
    if fmt == "token":
        assert np.all((q[np.arange(64), top] & 0x7F) == 0x7E)  # +-448
    else:
        r, c = np.unravel_index(np.abs(x).argmax(), x.shape)
        assert (q[r, c] & 0x7F) == 0x7E


@pytest.mark.parametrize("fmt", ["token", "tensor"])
def test_power_of_two_rescaling_keeps_the_codes(fmt):
    f = moe_ref.quantize_fp8_token if fmt == "token" else moe_ref.quantize_fp8_tensor
    x = _x(20, 256, 5)
    q1, s1 = f(x)
    q2, s2 = f(x * 8.0)
    assert np.array_equal(q1, q2) and np.array_equal(s2, s1 * 8)


def test_zero_rows():
    x = np.zeros((3, 256))
    x[1, 5] = 2.0
    q, s = moe_ref.quantize_fp8_token(x)
    assert np.all(q[0] == 0) and np.all(q[2] == 0)
    assert s[0] == np.float32(np.float32(1e-10) / np.float32(448.0))


def test_layer_tensor_format_uses_one_scale_over_all_experts():
    # every expert's h rows are quantised with the scale of the largest |h| of the
    # whole layer: doubling one expert's w2 changes only that expert's rows, but
    # making one expert's h larger changes the codes of the others
    g = torch.Generator().manual_seed(6)
    T, H, I, E, k = 24, 256, 128, 3, 1
    a1 = torch.randn(T, H, generator=g).to(torch.bfloat16)
    w13 = (torch.randn(E, 2 * I, H, generator=g) / 16)
    w2 = (torch.randn(E, H, I, generator=g) / 11)
    # block-quantise the weights 128x128 the way the harness does
    def block_q(w):
        out_q, out_s = [], []
        for e in range(w.shape[0]):
            x = w[e].double().numpy()
            N, K = x.shape
            blk = np.abs(x.reshape(N // 128, 128, K // 128, 128)).max(axis=(1, 3))
            s = codecs.round_fp32(np.maximum(blk, moe_ref.AMAX_FLOOR) / 448.0)
            q = codecs.e4m3_encode(codecs.round_fp32(x / np.repeat(np.repeat(s, 128, 0), 128, 1)))
            out_q.append(q)
            out_s.append(s.astype(np.float32))
        return torch.from_numpy(np.stack(out_q)), torch.from_numpy(np.stack(out_s))
    q13, s13 = block_q(w13)
    q2, s2 = block_q(w2)
    ids = torch.arange(T, dtype=torch.int32).remainder(E)[:, None].contiguous()
    al = moe_ref.align(ids, E, 128)
    a1q, sc = moe_ref.prepare(a1, None, False, "fp8_tensor")
    y = moe_ref.experts(a1q, sc, q13, s13, q2, s2, al, k, "fp8_tensor")
    s13b = s13.clone()
    s13b[0] *= 64  # expert 0's h grows far beyond the others': the shared h scale grows
    yb = moe_ref.experts(a1q, sc, q13, s13b, q2, s2, al, k, "fp8_tensor")
    rows1 = (ids[:, 0] == 1).nonzero()[:, 0]
    assert not torch.equal(y[rows1], yb[rows1])     # expert 1's rows see the larger common scale
    # with the "A" format each row keeps its own scale: expert 1's rows do not move
    a1t, sct = moe_ref.prepare(a1, None, False, "fp8_token")
    yt = moe_ref.experts(a1t, sct, q13, s13, q2, s2, al, k, "fp8_token")
    ytb = moe_ref.experts(a1t, sct, q13, s13b, q2, s2, al, k, "fp8_token")
    assert torch.equal(yt[rows1], ytb[rows1])
