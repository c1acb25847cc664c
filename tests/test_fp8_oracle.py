"""Pins of the FP8 (e4m3, per-128 fp32 scale) KV oracle, on the CPU.

* e4m3 codes whose values the format's definition fixes (1.0 = 0x38, the
  largest finite 448 = 0x7E, the smallest subnormal 2^-9 = 0x01, NaN = 0x7F);
  order and sign symmetry over all 256 codes; torch's own float8_e4m3fn
  conversion as a library cross-check;
* the 528-byte row layout, from a row built by hand;
* decode over an FP8 cache whose values are exactly representable in bf16
  equals the (pinned) dense oracle over the bf16 cache of the same values;
* slips planted in the decoder or the layout fail one of these pins.
"""
import math

import numpy as np
import pytest
import torch

import oracle.fp8 as f8
from oracle import gqa_paged_decode_oracle
from paged_kv_gqa_split_gb300 import workloads as wl

KNOWN = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0x30: 0.5, 0x7E: 448.0, 0xFE: -448.0, 0x08: 2.0 ** -6,
         0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x0F: 1.875 * 2.0 ** -6, 0x77: 240.0, 0x78: 256.0, 0x7D: 416.0,
         0xB8: -1.0, 0x81: -(2.0 ** -9)}


def test_known_codes():
    for code, val in KNOWN.items():
        assert f8.e4m3_decode([code])[0] == val, hex(code)
    assert np.isnan(f8.e4m3_decode([0x7F, 0xFF])).all()
    assert math.copysign(1.0, f8.e4m3_decode([0x80])[0]) == -1.0


def test_order_and_sign_symmetry():
    pos = f8.e4m3_decode(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0)
    neg = f8.e4m3_decode(np.arange(0x80, 0xFF))
    assert np.array_equal(neg, -pos)


def test_matches_torch_float8_conversion():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = f8.e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])


def test_row_layout_by_hand():
    row = np.zeros((2, f8.ROW_BYTES), dtype=np.uint8)
    row[1, 2 * 128 + 5] = 0x40                              # head 2, dim 5: 2.0
    row[1, 3 * 128 + 127] = 0xB8                            # head 3, dim 127: -1.0
    scales = np.array([[1, 1, 1, 1], [3.0, 7.0, 0.25, 0.5]], dtype="<f4")
    row[:, 512:] = scales.view(np.uint8).reshape(2, 16)
    deq = f8.dequantize_rows(row)
    assert deq.shape == (2, 4, 128)
    assert deq[1, 2, 5] == 0.5 and deq[1, 3, 127] == -0.5
    assert np.count_nonzero(deq) == 2


def _exact_fp8_problem(lens, seed):
    """FP8 rows with power-of-two scales: every dequantized value is exact in bf16."""
    g = torch.Generator().manual_seed(seed)
    dense = wl.make_workload(lens, seed)
    p = dense.num_pages
    codes = torch.randint(0, 0x7F, (p, 4, 128), generator=g)
    codes = codes | (torch.randint(0, 2, (p, 4, 128), generator=g) << 7)       # both signs, no NaN
    scale = torch.pow(2.0, torch.randint(-3, 4, (p, 4), generator=g).double()).float()
    rows = torch.empty((p, f8.ROW_BYTES), dtype=torch.uint8)
    rows[:, :512] = codes.reshape(p, 512).to(torch.uint8)
    rows[:, 512:] = scale.contiguous().view(torch.uint8).reshape(p, 16)
    vals = torch.from_numpy(np.vectorize(lambda c: float(KNOWN_TABLE[c]))(codes.numpy())) * scale[:, :, None].double()
    bf = vals.to(torch.bfloat16)
    assert torch.equal(bf.double(), vals)                                      # exact in bf16
    return dense, rows, bf[:, None]


# e4m3 values written out from the definition once more, by construction of
# the bits (exponent and mantissa fields), for the table used above
KNOWN_TABLE = {}
for c in range(256):
    s, e, m = c >> 7, (c >> 3) & 15, c & 7
    if e == 15 and m == 7:
        continue
    v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
    KNOWN_TABLE[c] = -v if s else v


@pytest.mark.parametrize("lens,seed", [([5, 0, 40, 1], 81), ([300, 17], 82)])
def test_equals_dense_oracle_on_exact_values(lens, seed):
    dense, rows, bf = _exact_fp8_problem(lens, seed)
    o, l = f8.gqa_paged_decode_fp8_oracle(dense.q, rows, rows, dense.kv_indptr, dense.kv_indices, dense.sm_scale)
    od, ld = gqa_paged_decode_oracle(dense.q, bf, bf, dense.kv_indptr, dense.kv_indices, dense.sm_scale)
    assert np.array_equal(np.isneginf(l), np.isneginf(ld))
    assert np.allclose(o, od, rtol=1e-13, atol=1e-13)
    fin = np.isfinite(ld)
    assert np.allclose(l[fin], ld[fin], rtol=0, atol=1e-12)


def test_quantized_workload_is_close_to_its_source():
    """The generator's rows dequantize to within e4m3's half-ulp of the bf16 source."""
    w = wl.make_workload([50, 7], seed=83)
    rows = wl.quantize_fp8_rows(w.k_cache)
    deq = f8.dequantize_rows(rows)
    src = w.k_cache[:, 0].double().numpy()
    amax = np.abs(src).max(axis=2, keepdims=True)
    assert np.all(np.abs(deq - src) <= amax / 448.0 * 2.0 ** -4 * np.maximum(np.abs(src) / (amax / 448.0), 2.0 ** -6)
                  + 1e-12)


@pytest.mark.parametrize("slip", ["bias8", "subnormal_shift", "scale_of_next_head", "nan_as_max"])
def test_pins_catch_planted_mistakes(monkeypatch, slip):
    good_decode, good_deq = f8.e4m3_decode, f8.dequantize_rows

    def bad_decode(codes):
        b = np.asarray(codes, dtype=np.int64) & 0xFF
        sign = np.where(b >> 7, -1.0, 1.0)
        e = (b >> 3) & 0xF
        m = (b & 7).astype(np.float64)
        bias = 8.0 if slip == "bias8" else 7.0
        normal = sign * (1.0 + m / 8.0) * np.exp2(e - bias)
        sub = sign * (m / 8.0) * 2.0 ** (-7 if slip == "subnormal_shift" else -6)
        out = np.where(e == 0, sub, normal)
        if slip == "nan_as_max":
            return out
        return np.where((b & 0x7F) == 0x7F, np.nan, out)

    def bad_deq(cache):
        raw = np.ascontiguousarray(np.asarray(cache), dtype=np.uint8).reshape(-1, f8.ROW_BYTES)
        vals = f8.e4m3_decode(raw[:, :512]).reshape(-1, 4, 128)
        scales = raw[:, 512:].copy().view("<f4").astype(np.float64)
        return vals * np.roll(scales, 1, axis=1)[:, :, None]

    if slip == "scale_of_next_head":
        monkeypatch.setattr(f8, "dequantize_rows", bad_deq)
    else:
        monkeypatch.setattr(f8, "e4m3_decode", bad_decode)
    failed = False
    try:
        test_known_codes()
        test_order_and_sign_symmetry()
        test_row_layout_by_hand()
        test_equals_dense_oracle_on_exact_values([5, 0, 40, 1], 81)
    except AssertionError:
        failed = True
    finally:
        monkeypatch.setattr(f8, "e4m3_decode", good_decode)
        monkeypatch.setattr(f8, "dequantize_rows", good_deq)
    assert failed, slip
