"""Pins of the oracle's FP8 cache-writer functions against things other than themselves.

The rule ("DeepSeek V4 Flash는 단일 AMD MI300X에서 실행됩니다", section 두 가지 핵심 정확성 수정
사항, FP8 형식 불일치: the indexer cache is FP8 E4M3 and the format's largest value sets the
scale): scale = fp32(absmax / 448), code = E4M3FN(clamp(fp32(x / scale), +-448)), nearest with
ties to the even code; scale 0 gives codes 0; the query scale folds into w as fp32(w * qscale).
Pins: hand-worked codes and rows (tests/golden/e4m3_quant_hand.json), the round trip of every
finite code through the (separately pinned) decoder, torch's own float8_e4m3fn cast on every
tie point and its neighbours, the torch-based input generator on random rows, numpy's float32
multiply for the fold, and invariants (the row maximum maps to +-448, order is kept).
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from sparse_attention_lightning_indexer_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_quant_hand.json")


@pytest.fixture(scope="module")
def hand():
    with open(GOLDEN) as f:
        return json.load(f)


def test_hand_encodings(hand):
    for case in hand["encode"]:
        assert orc.encode_e4m3(case["y"]) == case["code"], case


def test_hand_rows(hand):
    for case in hand["rows"]:
        codes, scale = orc.quantize_rows(np.array([case["x"]], dtype=np.float32))
        assert codes[0].tolist() == case["codes"], case
        assert scale[0] == np.float32(case["scale"]), case


def test_every_finite_code_round_trips():
    for c in range(256):
        if c & 0x7F == 0x7F:  # NaN
            continue
        assert orc.encode_e4m3(orc.decode_e4m3(c)) == c, hex(c)


def _torch_cast(y):
    return torch.tensor(np.asarray(y, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_matches_torch_cast_on_ties_and_neighbours():
    vals = np.array(sorted({orc.decode_e4m3(c) for c in range(0x7F)}), dtype=np.float64)
    mids = (vals[:-1] + vals[1:]) / 2  # exact in fp32: adjacent E4M3 values are dyadic
    pts = np.concatenate([vals, mids]).astype(np.float32)
    pts = np.concatenate([pts, np.nextafter(pts, np.float32(np.inf)),
                          np.nextafter(pts, np.float32(0))])
    pts = pts[np.abs(pts) <= 448]
    pts = np.concatenate([pts, -pts])
    want = _torch_cast(pts)
    got = np.array([orc.encode_e4m3(float(y)) for y in pts], dtype=np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(pts[i]), int(got[i]), int(want[i])) for i in bad[:5]]


def test_matches_torch_cast_on_random_values():
    rng = np.random.default_rng(5)
    y = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1, 20000),
                        rng.normal(0, 1e-3, 20000)]).astype(np.float32)
    got = np.array([orc.encode_e4m3(float(v)) for v in y], dtype=np.uint8)
    assert np.array_equal(got, _torch_cast(y))


def test_saturation():
    for y in (448.0, 448.5, 463.99, 464.0, 479.0, 1e6, 3.4e38):
        assert orc.encode_e4m3(y) == 0x7E and orc.encode_e4m3(-y) == 0xFE


@pytest.mark.parametrize("seed", [0, 1])
def test_rows_match_the_input_generator(seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(3000, 128, generator=g) * torch.exp(torch.randn(3000, 1, generator=g) * 4)
    x[7] = 0.0
    x[11, :5] = -0.0
    tc, ts = inputs.quantize_e4m3_rows(x)
    codes, scales = orc.quantize_rows(x.numpy())
    assert np.array_equal(codes, tc.numpy())
    assert np.array_equal(scales.view(np.uint32), ts.numpy().view(np.uint32))


def test_row_invariants():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((500, 128)) * np.exp(rng.standard_normal((500, 1)) * 3)).astype(np.float32)
    codes, scales = orc.quantize_rows(x)
    dec = np.vectorize(orc.decode_e4m3)(codes)
    amax = np.abs(x).argmax(axis=1)
    assert np.all(np.abs(dec[np.arange(500), amax]) == 448.0)  # the row maximum maps to +-448
    assert np.all(np.sign(dec) * np.sign(x) >= 0)              # signs kept
    order = np.argsort(x, axis=1, kind="stable")
    assert np.all(np.diff(np.take_along_axis(dec, order, axis=1), axis=1) >= 0)  # monotone
    # reconstruction within half a code step: |code*scale - x| <= 2^-4 |x| (normal range)
    big = np.abs(x) / scales[:, None] >= 2.0 ** -6
    err = np.abs(dec * scales[:, None] - x)
    assert np.all(err[big] <= 2.0 ** -4 * np.abs(x[big]) * 1.0001)


def test_fold_matches_float32_multiply():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((257, 64)).astype(np.float32)
    qs = np.abs(rng.standard_normal(257)).astype(np.float32) * np.float32(1e-3)
    want = (w * qs[:, None]).astype(np.float32)  # numpy: IEEE float32 multiply
    assert np.array_equal(orc.fold_qscale(w, qs).view(np.uint32), want.view(np.uint32))


def test_workload_codes_follow_the_rule():
    # The FP8 workloads' codes and scales are this rule applied to their fp32 draws.
    prob = inputs.make("w", T=64, S=3000, pos_offset=2936, seed=3, dtype=inputs.FP8_E4M3)
    qf, kf, w = inputs.draw_f32(64, 3000, 3)
    kc, ks = orc.quantize_rows(kf.numpy())
    assert np.array_equal(kc, prob.k.numpy()) and np.array_equal(ks, prob.kscale.numpy())
    qc, qs = orc.quantize_rows(qf.reshape(64, -1).numpy())
    assert np.array_equal(qc.reshape(64, 64, 128), prob.q.numpy())
    assert np.array_equal(orc.fold_qscale(w.numpy(), qs), prob.w.numpy())
