"""Pins of the oracle's 8-bit T2 quantiser (CPU only).

"Not All Thoughts Need HBM", Methodology 1 and Results 4: T2 holds tokens at
8 bits and they are still read.
"""
import json
import os

import numpy as np
import torch

from oracle import dequantize, quantize_rows, to_storage
from oracle.quant import bf16_round


def test_hand_worked_rows(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "quant_examples.json")))
    for row in g["rows"]:
        codes, scale = quantize_rows(np.array([row["x"]], dtype=np.float32))
        assert float(scale[0]) == row["scale"]
        assert codes[0].tolist() == row["codes"]


def test_absmax_maps_to_127_and_error_is_half_a_step():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((200, 512)) * rng.lognormal(0, 1, (200, 1))).astype(np.float32)
    codes, scale = quantize_rows(x)
    i = np.argmax(np.abs(x), axis=1)
    top = codes[np.arange(200), i]
    assert np.all(np.abs(top) == 127)
    assert np.all(np.sign(top) == np.sign(x[np.arange(200), i]))
    err = np.abs(x.astype(np.float64) - dequantize(codes, scale))
    assert np.all(err <= scale[:, None].astype(np.float64) * (0.5 + 1e-6))


def test_zero_row_and_fp16_scale():
    codes, scale = quantize_rows(np.zeros((2, 8), dtype=np.float32), "f16")
    assert scale.dtype == np.float16 and np.all(scale == 0) and np.all(codes == 0)
    x = np.array([[1.0, -0.5, 0.25]], dtype=np.float32)
    codes, scale = quantize_rows(x, "f16")
    # 1/127 rounds to the float16 0.007873535..., and 1 / that is 127.008 -> 127
    assert scale[0] == np.float16(1.0 / 127.0)
    assert codes[0].tolist() == [127, -64, 32]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(100000).astype(np.float32) * 10
    bits = x.view(np.uint32)
    x = np.concatenate([x, ((bits & 0xFFFF0000) | 0x8000).view(np.float32)])  # exact ties
    ours = bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_promotion_value_is_storage_rounded_product():
    codes = np.array([[127, -3, 0]], dtype=np.int8)
    scale = np.array([0.1], dtype=np.float32)
    v32 = to_storage(codes, scale, "f32")
    assert v32[0, 0] == float(np.float32(127) * np.float32(0.1))
    vb = to_storage(codes, scale, "bf16")
    ref = torch.tensor([127 * np.float32(0.1)], dtype=torch.float32).to(torch.bfloat16).float()
    assert vb[0, 0] == float(ref[0])
