"""Host-side arithmetic of bench.py (no GPU): algorithmic work and the all-bytes figure."""
import pytest

import bench
from sparse_attention_lightning_indexer_gb300 import inputs


class _P:  # the fields bench reads from a problem, without drawing its tensors
    def __init__(self, T, S, pos, dtype, topk=512):
        self.T, self.S, self.pos_offset, self.dtype, self.topk = T, S, pos, dtype, topk


def test_causal_pairs_and_flops():
    # T = S = 4 from position 0: rows see 1, 2, 3, 4 keys
    flops, key_bytes, pairs = bench.algorithmic(_P(4, 4, 0, inputs.BF16))
    assert pairs == 10
    assert flops == 2 * 64 * 128 * 10
    assert key_bytes == 4 * 256
    # a decode row at the last position sees every key; FP8 keys carry a 4-byte scale
    flops, key_bytes, pairs = bench.algorithmic(_P(1, 262144, 262143, inputs.FP8_E4M3))
    assert pairs == 262144 and key_bytes == 262144 * 132


def test_all_bytes_counts_inputs_and_outputs_once():
    # decode sequence: q 64x128 codes, w 64 fp32, keys + scales, 512 (idx, score)
    assert bench.all_bytes(_P(1, 262144, 262143, inputs.FP8_E4M3)) == (
        64 * 128 + 64 * 4 + 262144 * 132 + 512 * 8)
    # 64k bf16 prefill: q 1 GiB + w 16 MiB + keys 16 MiB + outputs 256 MiB
    assert bench.all_bytes(_P(65536, 65536, 0, inputs.BF16)) == pytest.approx(
        2**30 + 2**24 + 2**24 + 2**28)


@pytest.mark.parametrize("T,n", [(65536, 104), (65536, 1), (7, 7), (7, 20), (1, 16)])
def test_reference_rows_are_spread_evenly(T, n):
    import numpy as np
    for phase in (0.0, 0.37, 0.999):
        rows = bench.even_rows(T, n, phase)
        m = min(n, T)
        assert len(rows) == m and rows.min() >= 0 and rows.max() < T
        assert np.all(np.diff(rows) > 0)
        # row i is the floor of a point of the i-th of m equal strata of [0, T): the causal row
        # lengths' mix
        i = np.arange(m)
        assert np.all(rows >= i * T // m) and np.all(rows * m < (i + 1) * T)
