"""Pins for the oracle's q8_0 encoder (the cache write of the walk).

* Hand-worked blocks (tests/golden/q8_0_encode.txt): exact halves rounding
  away from zero, power-of-two scales, the zero block, a subnormal and an
  overflowing fp16 scale.
* The fp16 rounding of the scale against numpy's float32 -> float16
  conversion (round to nearest even) over normal, subnormal and overflowing
  magnitudes.
* The input generator's independent encoder (synth.encode_q8_0) on random
  blocks, bit for bit.
* Round trip: dequantised codes lie within half a step (plus the fp16
  rounding of the scale) of the inputs, and the absmax gets code +-127.
* Planted mistakes (ties to even; dividing by the fp16-rounded scale) fail:
  edited copies of the oracle's source (tests/oracle_mutants.py).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import oracle_mutants as mutants

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q8_0_encode.txt")


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _golden():
    cases = []
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        left, right = line.split("->")
        parts = left.split()
        name, scale = parts[0], int(parts[1], 16)
        vals = np.zeros(32, dtype=np.float32)
        if len(parts) > 2:
            for kv in parts[2].split(","):
                k, v = kv.split(":")
                vals[int(k)] = float(v)
        codes = np.zeros(32, dtype=np.int8)
        if right.strip():
            for kv in right.strip().split(","):
                k, v = kv.split(":")
                codes[int(k)] = int(v)
        cases.append((name, scale, vals, codes))
    return cases


def _golden_ok():
    cases = _golden()
    x = np.stack([c[2] for c in cases])
    bits = _bf16_bits(x)
    # every golden value is exact in bf16
    assert np.array_equal(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy(), x)
    out = oracle.quantize_q8_0(bits)
    ok = True
    for i, (name, scale, _, codes) in enumerate(cases):
        ok &= int(out[i, 0]) | (int(out[i, 1]) << 8) == scale
        ok &= np.array_equal(out[i, 2:].view(np.int8), codes)
    return bool(ok)


def test_golden_encodings():
    assert len(_golden()) >= 8
    assert _golden_ok()


def test_scale_rounding_matches_float16_conversion():
    # blocks whose absmax is 127 * s give d = s exactly when s*127 is exact
    # and fp32(s*127)/127 == s; compare the stored scale with numpy's RNE
    rng = np.random.default_rng(5)
    mags = np.concatenate([2.0 ** rng.uniform(-30, 20, 4000),      # subnormal .. overflow
                           [6.0e-8, 6.1e-5, 65504.0, 65519.0, 65520.0, 1e-9]])
    x = np.zeros((len(mags), 32), dtype=np.float32)
    x[:, 0] = (mags * 127.0).astype(np.float32)
    bits = _bf16_bits(x)
    amax = torch.from_numpy(bits[:, 0].view(np.int16)).view(torch.bfloat16).float().numpy()
    d32 = (np.abs(amax) / np.float32(127.0)).astype(np.float32)
    with np.errstate(over="ignore"):            # scales past 65504 become infinity
        want = d32.astype(np.float16).view(np.uint16)
    out = oracle.quantize_q8_0(bits)
    got = out[:, 0].astype(np.uint16) | (out[:, 1].astype(np.uint16) << 8)
    assert np.array_equal(got, want)


def _random_blocks(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 32)).astype(np.float32) * rng.uniform(0.01, 10, (n, 1)).astype(np.float32)
    x[:5] = 0.0                   # zero blocks
    x[5, :] = 1e-38               # subnormal-range values
    return x


def _matches_generator():
    x = _random_blocks(4096, 1)
    bits = _bf16_bits(x)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float()
    want = synth.encode_q8_0(xb).numpy()
    got = oracle.quantize_q8_0(bits)
    return np.array_equal(got, want)


def test_matches_the_input_generator_encoder():
    assert _matches_generator()


def test_round_trip_bound_and_absmax_code():
    x = _random_blocks(2048, 2)
    bits = _bf16_bits(x)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    q8 = oracle.quantize_q8_0(bits)
    f64, _, _ = oracle.dequant_q8_0(q8)
    amax = np.abs(xb).max(1)
    d = amax / 127
    dh = q8[:, 0].astype(np.uint16) | (q8[:, 1].astype(np.uint16) << 8)
    d16 = dh.view(np.float16).astype(np.float64)
    bound = d / 2 + 127 * np.abs(d16 - d) + 1e-300
    assert np.all(np.abs(f64 - xb) <= bound[:, None] * (1 + 1e-6))
    codes = q8[:, 2:].view(np.int8).astype(int)
    nz = amax > 0
    assert np.all(np.abs(codes[nz]).max(1) == 127)


@pytest.mark.parametrize("n", [15, 16])
def test_pins_catch_planted_encoder_mistake(n):
    with mutants.c_mutant(n):
        caught = not (_golden_ok() and _matches_generator())
    assert caught, mutants.C_MUTANTS[n][0]
