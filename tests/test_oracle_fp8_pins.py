"""Pins for the oracle's fp8 K/V path (E4M3 codes, one scale per key block and
KV head), against facts fixed outside the oracle:
  * a hand-worked table of E4M3 codes and roundings (tests/golden/e4m3_codes.json,
    worked from the format's definition);
  * torch's float8_e4m3fn dtype, a library implementation of the same format,
    on every code and on many random values inside the finite range;
  * properties of the quantizer (the block maximum maps to +-448, error within
    half a unit in the last place) and of the attention over fp8 K/V, which must
    equal the bf16 Main Branch when K and V already lie on the fp8 grid with a
    power-of-two scale.
The fp8 support itself: the atlas record of the report, provenance of section
4.2 (the kernels handle fp8 as well; no format is given, the reading is stated
in the oracle).  No GPU is needed.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads.configs import small

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_codes.json")


def test_e4m3_golden_table():
    d = json.load(open(GOLDEN))
    for r in d["values"]:
        v = oracle.e4m3_value(int(r["code"], 16))
        assert v == r["value"] and math.copysign(1.0, v) == math.copysign(1.0, r["value"]), r
    for c in d["nan_codes"]:
        assert math.isnan(oracle.e4m3_value(int(c, 16)))
    for r in d["rounding"]:
        assert oracle.e4m3_code(r["x"]) == int(r["code"], 16), r


def test_e4m3_values_match_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], (hex(c), v, ref[c])


def test_e4m3_codes_match_torch_rounding():
    rng = np.random.default_rng(0)
    # magnitudes over the whole finite range, including subnormals and exact midpoints between codes
    mids = []
    for c in range(0, 0x7E):
        mids.append(0.5 * (oracle.e4m3_value(c) + oracle.e4m3_value(c + 1)))
    x = np.concatenate([rng.standard_normal(4000) * 30, np.exp(rng.uniform(-12, 6, 4000)), np.array(mids),
                        -np.array(mids), rng.uniform(-448, 448, 2000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_code(v) for v in x], np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_e4m3_codes_round_trip_and_order():
    vals = [oracle.e4m3_value(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))          # non-negative codes are ordered
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.e4m3_code(oracle.e4m3_value(c)) == c     # every finite code encodes to itself


def _fp8_case(seed=0, seqs=((5, 300), (17, 17), (40, 200)), hq=8, hkv=2, d=16, block=128):
    cfg = small("fp8", seqs, hq=hq, hkv=hkv, head_dim=d, d_idx=8, block=block, topk=3, n_topics=3, seed=seed)
    return cfg, workloads.generate(cfg)


def test_quantizer_scale_and_error_bound():
    cfg, x = _fp8_case()
    codes, scales = oracle.quantize_fp8(x.cu_k, x.k, block=cfg.block)
    kf = x.k.float().numpy()
    cu = x.cu_k.numpy()
    row = 0
    for s in range(len(cu) - 1):
        for b0 in range(int(cu[s]), int(cu[s + 1]), cfg.block):
            b1 = min(b0 + cfg.block, int(cu[s + 1]))
            for g in range(cfg.hkv):
                blk = kf[b0:b1, g]
                amax = np.float32(np.abs(blk).max())
                assert scales[row, g] == np.float32(amax / np.float32(448.0))
                c = codes[b0:b1, g]
                deq = np.vectorize(oracle.e4m3_value)(c) * np.float64(scales[row, g])
                # the element of largest magnitude lands on +-448 exactly
                j = np.unravel_index(np.abs(blk).argmax(), blk.shape)
                assert c[j] in (0x7E, 0xFE)
                # half a unit in the last place: 2^-4 relative for normals, 2^-10 * scale below 2^-6 * scale
                err = np.abs(deq - blk)
                bound = np.maximum(np.abs(blk) * 2.0 ** -4, 2.0 ** -10 * scales[row, g]) * (1 + 1e-6)
                assert np.all(err <= bound)
            row += 1
    assert row == scales.shape[0] == oracle.key_blocks(x.cu_k, cfg.block)


def test_quantizer_zero_block_has_unit_scale():
    cfg, x = _fp8_case(seed=1, seqs=((3, 130),))
    k = x.k.clone()
    k[:128] = 0.0
    codes, scales = oracle.quantize_fp8(x.cu_k, k, block=cfg.block)
    assert np.all(scales[0] == 1.0) and np.all(codes[:128] == 0)


def test_attention_fp8_equals_bf16_attention_on_the_fp8_grid():
    """K and V drawn from E4M3 values times a power of two f / 8 that differs between key blocks and heads,
    with every (block, head) holding an element of magnitude 56 f: its scale is then exactly 56 f / 448 =
    f / 8, quantization is exact, and the fp8 Main Branch must equal the bf16 one."""
    cfg, x = _fp8_case(seed=2, seqs=((60, 400), (33, 33), (9, 250)))
    rng = np.random.default_rng(3)
    grid = np.array([oracle.e4m3_value(c) for c in range(0x7F)], np.float64)
    cu = x.cu_k.numpy()
    f_of = {}  # (scale row, head) -> f

    def on_grid(shape):
        v = grid[rng.integers(0, 0x70, size=shape)] * rng.choice([-1.0, 1.0], size=shape) / 8.0
        row = 0
        for s in range(len(cu) - 1):
            for b0 in range(int(cu[s]), int(cu[s + 1]), cfg.block):
                b1 = min(b0 + cfg.block, int(cu[s + 1]))
                for g in range(cfg.hkv):
                    f = 2.0 ** -((row + 2 * g) % 5)
                    f_of[(row, g)] = f
                    v[b0:b1, g] *= f
                    v[b0, g, g % shape[2]] = 56.0 * f * (1 if row % 2 else -1)
                row += 1
        return v

    k = on_grid(x.k.shape)
    v = on_grid(x.v.shape)
    kb = torch.from_numpy(k).to(torch.bfloat16)
    vb = torch.from_numpy(v).to(torch.bfloat16)
    assert np.array_equal(kb.double().numpy(), k) and np.array_equal(vb.double().numpy(), v)
    k8, ks = oracle.quantize_fp8(x.cu_k, kb, block=cfg.block)
    v8, vs = oracle.quantize_fp8(x.cu_k, vb, block=cfg.block)
    for (row, g), f in f_of.items():
        assert ks[row, g] == f / 8 and vs[row, g] == f / 8
    assert len(set(ks[:, 0].tolist())) > 1   # the scales differ between key blocks
    ref = oracle.forward(x.cu_q, x.cu_k, x.q, kb, vb, x.q_idx, x.k_idx, block=cfg.block, topk=cfg.topk)
    o8, l8 = oracle.attention_fp8(x.cu_q, x.cu_k, x.q, k8, v8, ks, vs, ref["idx"], block=cfg.block)
    np.testing.assert_array_equal(o8, ref["o"])
    np.testing.assert_array_equal(l8, ref["lse"])


def test_attention_fp8_is_close_to_bf16_attention():
    """On ordinary inputs the fp8 Main Branch differs from the bf16 one by the quantization error only."""
    cfg, x = _fp8_case(seed=4)
    k8, ks = oracle.quantize_fp8(x.cu_k, x.k, block=cfg.block)
    v8, vs = oracle.quantize_fp8(x.cu_k, x.v, block=cfg.block)
    ref = oracle.forward(x.cu_q, x.cu_k, x.q, x.k, x.v, x.q_idx, x.k_idx, block=cfg.block, topk=cfg.topk)
    o8, l8 = oracle.attention_fp8(x.cu_q, x.cu_k, x.q, k8, v8, ks, vs, ref["idx"], block=cfg.block)
    assert np.abs(o8 - ref["o"]).max() < 0.15 and np.abs(l8 - ref["lse"]).max() < 0.15
    assert np.abs(o8 - ref["o"]).max() > 0.0   # the quantization does change the result
