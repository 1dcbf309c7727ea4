"""Seeded synthetic inputs for the Lightning Indexer workloads.

This module is shared by the oracle tests, the GPU parity tests and the benchmark. It only
draws and encodes inputs; it holds none of the indexer's arithmetic (no score, no ReLU, no
selection). Everything is drawn on the CPU with ``torch.Generator`` so the oracle reads the very
same host buffers that are copied to the device.

Recipe (per workload):
  * q, k drawn N(0, sigma^2) per element with sigma = 128^-1/2; w drawn N(0, (1/64)^2).
  * bf16 workloads round q and k to bf16 (round-to-nearest-even, torch's cast).
  * FP8 workloads quantise each token row (q over all heads and dims of a token, k per key) with
    scale = absmax / 448 into OCP E4M3FN codes (clamped to +-448, torch's RNE cast); an all-zero
    row gets scale 0 and code 0. The q scale is folded into the head weights,
    w'[t,j] = fp32(w[t,j] * qscale[t]), which is exact in the indexer score because ReLU is
    positively homogeneous.
  * Planted workload: 16 random unit "topic" vectors u_m. One query in eight (seeded subset) gets
    a topic m(t) and q[t,j] += a * sign(w[t,j]) * u_m; in every aligned 1024-key block 32 random
    positions get a random topic m and k[s] += a * u_m. The amplitude ``a`` comes from the normal
    model of the inputs alone, not from any score: with x = q_j . k ~ N(0, D sigma^4) the base
    score std is s_I = sqrt(H sigma_w^2 Var(x) / 2); with c = H E|w| / 2 a same-topic pair gains
    c a^2, while the topic term a sign(w_j) (u . k), shared by all heads of a planted query, adds
    a common-mode std of c a sigma. Solving c a^2 = 3 sqrt(s_I^2 + c^2 a^2 sigma^2) for a^2
    puts same-topic keys three (model) standard deviations above the planted query's row.
  * Each tensor has its own generator, seeded from (workload seed, tensor tag), so two workloads
    with the same seed share the same key cache.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

H_I = 64
D_I = 128
TOPK = 512
SIGMA_QK = 128 ** -0.5
SIGMA_W = 1.0 / 64.0
E4M3_MAX = 448.0

BF16 = 0
FP8_E4M3 = 1

_TAGS = {"q": 1, "k": 2, "w": 3, "plant": 4}
_CHUNK = 1 << 24  # elements drawn per randn call (bounds the fp32 temporaries)


def _gen(seed: int, tag: str) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed) * 1009 + _TAGS[tag])
    return g


def _randn(shape, g: torch.Generator, std: float) -> torch.Tensor:
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.float32)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = torch.randn(hi - lo, generator=g, dtype=torch.float32)
    out.mul_(std)
    return out.view(*shape)


def quantize_e4m3_rows(x: torch.Tensor):
    """Per-row absmax/448 E4M3FN quantisation of x [R, C] (fp32). Returns (codes u8, scale f32)."""
    absmax = x.abs().amax(dim=1)
    scale = (absmax / E4M3_MAX).to(torch.float32)
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    y = (x / safe[:, None]).clamp_(-E4M3_MAX, E4M3_MAX)
    y = torch.where(scale[:, None] > 0, y, torch.zeros_like(y))
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


@dataclass
class Problem:
    """One indexer call's inputs, as CPU tensors in the library's layouts.

    q: [T, H, D] (bf16, or uint8 E4M3 codes); w: [T, H] fp32; k: [S, D] (bf16 or uint8);
    kscale: [S] fp32 for FP8, else None.
    """
    name: str
    dtype: int
    q: torch.Tensor
    w: torch.Tensor
    k: torch.Tensor
    kscale: torch.Tensor | None
    T: int
    S: int
    pos_offset: int
    topk: int = TOPK
    meta: dict = field(default_factory=dict)

    def n_visible(self, t: int) -> int:
        return min(self.pos_offset + t, self.S - 1) + 1

    def codes(self):
        """(q, k) as numpy code arrays: uint16 bit patterns for bf16, uint8 for E4M3."""
        if self.dtype == BF16:
            return (self.q.view(torch.int16).numpy().view("uint16"),
                    self.k.view(torch.int16).numpy().view("uint16"))
        return self.q.numpy(), self.k.numpy()


def draw_f32(T: int, S: int, seed: int, H: int = H_I, D: int = D_I, parts=("q", "k", "w")):
    """The fp32 draws of a workload before any rounding: q [T, H, D], k [S, D], w [T, H]
    (None for a part not in ``parts``). These are the inputs of the FP8 cache writer; ``make``
    rounds or quantises these same draws."""
    qf = _randn((T, H, D), _gen(seed, "q"), SIGMA_QK) if "q" in parts else None
    kf = _randn((S, D), _gen(seed, "k"), SIGMA_QK) if "k" in parts else None
    w = _randn((T, H), _gen(seed, "w"), SIGMA_W) if "w" in parts else None
    return qf, kf, w


def planted_amplitude(H: int = H_I, D: int = D_I, sigma: float = SIGMA_QK,
                      sigma_w: float = SIGMA_W, n_sigma: float = 3.0) -> float:
    """Topic amplitude that lifts a same-topic pair by n_sigma score std (normal model only)."""
    var_x = D * sigma ** 4
    var_i = H * sigma_w ** 2 * var_x / 2.0
    c = H * sigma_w * math.sqrt(2.0 / math.pi) / 2.0
    # c^2 a^4 = n^2 (var_i + c^2 sigma^2 a^2)  ->  quadratic in a^2.
    b = n_sigma ** 2 * sigma ** 2
    a2 = (b + math.sqrt(b * b + 4.0 * n_sigma ** 2 * var_i / c ** 2)) / 2.0
    return math.sqrt(a2)


def make(name: str, T: int, S: int, pos_offset: int, seed: int, dtype: int = BF16,
         planted: bool = False, H: int = H_I, D: int = D_I, topk: int = TOPK) -> Problem:
    """Draw one workload. Shapes and distributions follow the module recipe."""
    if T < 0 or S < 1 or pos_offset < 0:
        raise ValueError("bad shape")
    qf, kf, w = draw_f32(T, S, seed, H, D)
    meta = {"seed": seed}
    if planted:
        a = planted_amplitude(H, D)
        g = _gen(seed, "plant")
        topics = torch.randn(16, D, generator=g, dtype=torch.float64)
        topics = (topics / topics.norm(dim=1, keepdim=True)).to(torch.float32)
        n_q = T // 8
        q_rows = torch.randperm(T, generator=g)[:n_q]
        q_topic = torch.randint(0, 16, (n_q,), generator=g)
        sgn = torch.sign(w[q_rows])  # [n_q, H]
        qf[q_rows] += a * sgn[:, :, None] * topics[q_topic][:, None, :]
        k_pos, k_topic = [], []
        for blk in range(0, S - S % 1024, 1024):
            pos = torch.randperm(1024, generator=g)[:32] + blk
            k_pos.append(pos)
            k_topic.append(torch.randint(0, 16, (32,), generator=g))
        if k_pos:
            k_pos_t = torch.cat(k_pos)
            k_topic_t = torch.cat(k_topic)
            kf[k_pos_t] += a * topics[k_topic_t]
            meta.update(planted_keys=k_pos_t, planted_key_topic=k_topic_t)
        meta.update(amplitude=a, planted_queries=q_rows, planted_query_topic=q_topic)
    if dtype == BF16:
        q = qf.to(torch.bfloat16)
        k = kf.to(torch.bfloat16)
        kscale = None
    elif dtype == FP8_E4M3:
        qc, qscale = quantize_e4m3_rows(qf.view(T, H * D))
        q = qc.view(T, H, D)
        k, kscale = quantize_e4m3_rows(kf)
        w = (w * qscale[:, None]).to(torch.float32)
        meta["qscale"] = qscale
    else:
        raise ValueError("dtype")
    return Problem(name, dtype, q.contiguous(), w.contiguous(), k.contiguous(),
                   None if kscale is None else kscale.contiguous(), T, S, pos_offset, topk, meta)


# The six workload shapes (name -> constructor). The first five are single indexer calls.
WORKLOADS = {
    "tiny_1k": dict(T=1024, S=1024, pos_offset=0, seed=0, dtype=BF16),
    "planted_16k": dict(T=16384, S=16384, pos_offset=0, seed=1, dtype=BF16, planted=True),
    "prefill_64k": dict(T=65536, S=65536, pos_offset=0, seed=2, dtype=BF16),
    "fp8_prefill_128k": dict(T=131072, S=131072, pos_offset=0, seed=3, dtype=FP8_E4M3),
    "chunk_2048_at_260096": dict(T=2048, S=262144, pos_offset=260096, seed=4, dtype=FP8_E4M3),
}
DECODE_BATCH = dict(B=8, S=262144, pos=262143, seed=4)


def workload(name: str) -> Problem:
    return make(name, **WORKLOADS[name])


def decode_batch(B: int = 8, S: int = 262144, pos: int = 262143, seed: int = 4,
                 T: int = 1) -> list[Problem]:
    """Independent decode sequences: sequence b is drawn with seed + b (its own FP8 cache)."""
    return [make(f"decode_b{b}", T, S, pos - (T - 1), seed + b, dtype=FP8_E4M3)
            for b in range(B)]


def sample_rows(T: int, seed: int, n_random: int = 256, head: int = 16, tail: int = 16):
    """Row sample for full-size checks: all t < head, n_random seeded rows and the last tail."""
    g = torch.Generator()
    g.manual_seed(10_007 + seed)
    rows = set(range(min(head, T)))
    rows.update(range(max(0, T - tail), T))
    if T > 0:
        rows.update(torch.randint(0, T, (n_random,), generator=g).tolist())
    return sorted(rows)
