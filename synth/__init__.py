"""Seeded synthetic inputs for the MoE layer workloads.

Shared by the tests and ``bench.py``; it feeds both the CUDA path and the
oracle the same bytes.  It holds none of the layer's arithmetic: every array
is drawn directly in its storage format (bf16 bit patterns, float32, E2M1 /
E4M3 / UE8M0 codes) from fixed distributions, so no quantiser or rounding
rule of the method lives here.

Workloads (the pages' decode shape T=8, H=7168, I=2048, E=256, K=6 and four
variants):

* ``tiny``     T=8,     H=512,  I=256,  E=16,  K=4, softmax,               align 16, MXFP4
* ``decode``   T=8,     H=7168, I=2048, E=256, K=6, sqrt(softplus)+bias,   align 16, MXFP4
* ``batched``  T=128,   same dims, + per-expert gate offset N(0,1),        align 64, MXFP4
* ``prefill``  T=4096,  same dims, uniform gate weights,                   align 256, MXFP4
* ``skewed``   T=16384, same dims, Zipf(1.1) popularity via gate bias,     align 128, NVFP4

Distributions:
* hidden: float32 N(0,1), kept as its top 16 bits (a bfloat16 pattern).
* W_gate: float32 N(0, 1/H) (``prefill``: uniform with the same variance).
* e_score_correction_bias: float32 N(0, 0.1) (all but ``tiny``).
* MXFP4 weights: each E2M1 code has a uniform sign and a magnitude code drawn
  from MAG_P below; each UE8M0 block scale is 2**-7 or 2**-6 with equal
  odds.  The resulting weight RMS is about 0.02, the spread of the
  N(0, 0.02) weights the workloads name.
* NVFP4 weights: same E2M1 codes; each per-16 E4M3 scale code is uniform in
  [0x30, 0x48) (0.5 .. 3.75); one float32 tensor scale per expert matrix,
  uniform in [0.0058, 0.0068), for the same RMS.
* INT8 weights (any workload with ``fmt="int8"``): int8 codes in [-127, 127]
  with probabilities proportional to exp(-c**2 / (2 * 40**2)) (a discretised
  normal of spread 40, drawn through a 16-bit lookup table), and one float32
  scale per output channel uniform in [4.5e-4, 5.5e-4), again an RMS of
  about 0.02.  ``fmt="int8b"``: the same codes with one float32 scale per
  256 x 256 block, uniform in the same range.
Each expert's weights come from their own generator, seeded by
(seed, matrix, expert), so any expert can be regenerated alone.
"""
from dataclasses import dataclass
from typing import Optional

import numpy as np

# Probabilities of the E2M1 magnitude codes 0..7 (values 0, .5, 1, 1.5, 2, 3, 4, 6).
MAG_P = (0.16, 0.24, 0.20, 0.14, 0.11, 0.09, 0.05, 0.01)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    K: int
    align: int
    score_fn: str            # "softmax" or "sqrt_softplus"
    fmt: str                 # "mxfp4", "nvfp4" or "int8"
    e_bias: bool             # e_score_correction_bias present
    gate_offset: str         # "none", "normal" (N(0,1) per expert), "zipf"
    gate_uniform: bool = False
    renormalize: bool = True
    seed: int = 0
    wide_scales: bool = False  # per-stage tests: weight block scales over a wide code range


WORKLOADS = {
    "tiny": Workload("tiny", 8, 512, 256, 16, 4, 16, "softmax", "mxfp4", False, "none", seed=1000),
    "decode": Workload("decode", 8, 7168, 2048, 256, 6, 16, "sqrt_softplus", "mxfp4", True, "none", seed=1001),
    "batched": Workload("batched", 128, 7168, 2048, 256, 6, 64, "sqrt_softplus", "mxfp4", True, "normal", seed=1002),
    "prefill": Workload("prefill", 4096, 7168, 2048, 256, 6, 256, "sqrt_softplus", "mxfp4", True, "none",
                        gate_uniform=True, seed=1003),
    "skewed": Workload("skewed", 16384, 7168, 2048, 256, 6, 128, "sqrt_softplus", "nvfp4", True, "zipf", seed=1004),
}


def custom(name="custom", **kw) -> Workload:
    base = dict(T=8, H=512, I=256, E=16, K=4, align=16, score_fn="softmax", fmt="mxfp4",
                e_bias=False, gate_offset="none", seed=7)
    base.update(kw)
    return Workload(name, **base)


def _rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(list(key)))


def _nibble_lut() -> np.ndarray:
    """uint8 draw -> E2M1 code: bit 0 is the sign, bits 1..7 pick the magnitude by MAG_P."""
    cum = np.cumsum(np.array(MAG_P) * 128.0)
    lut = np.zeros(256, dtype=np.uint8)
    for u in range(256):
        sign = u & 1
        v = (u >> 1) + 0.5
        mag = int(np.searchsorted(cum, v, side="right"))
        lut[u] = (sign << 3) | min(mag, 7)
    return lut


_NIB = _nibble_lut()
_u = np.arange(65536)
_BYTE = (_NIB[_u & 0xFF] | (_NIB[_u >> 8] << 4)).astype(np.uint8)   # uint16 draw -> packed byte
del _u


def fp4_codes(rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """[rows, cols/2] packed E2M1 bytes (element 2j in the low nibble)."""
    n = rows * (cols // 2)
    r = np.frombuffer(rng.bytes(2 * n), dtype=np.uint16)
    return _BYTE[r].reshape(rows, cols // 2)


def _i8_lut() -> np.ndarray:
    """uint16 draw -> int8 code with probabilities proportional to exp(-c^2 / (2 * 40^2)), |c| <= 127."""
    c = np.arange(-127, 128)
    cum = np.cumsum(np.exp(-(c / 40.0) ** 2 / 2.0))
    cum *= 65536.0 / cum[-1]
    idx = np.searchsorted(cum, np.arange(65536) + 0.5, side="right")
    return c[np.minimum(idx, c.size - 1)].astype(np.int8)


_I8 = _i8_lut()


def i8_codes(rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """[rows, cols] int8 weight codes (discretised normal, spread 40)."""
    r = np.frombuffer(rng.bytes(2 * rows * cols), dtype=np.uint16)
    return _I8[r].reshape(rows, cols)


def i8_channel_scales(rng: np.random.Generator, rows: int) -> np.ndarray:
    """[rows] float32 per-output-channel scales uniform in [4.5e-4, 5.5e-4)."""
    return rng.uniform(4.5e-4, 5.5e-4, size=rows).astype(np.float32)


def i8_block_scales(rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """[rows/256, cols/256] float32 scales of 256 x 256 weight blocks, uniform in [4.5e-4, 5.5e-4)."""
    return rng.uniform(4.5e-4, 5.5e-4, size=(rows // 256, cols // 256)).astype(np.float32)


def mx_scales(rng: np.random.Generator, rows: int, cols: int, wide: bool = False) -> np.ndarray:
    """[rows, cols/32] UE8M0 bytes, 120 or 121 (2**-7 or 2**-6); ``wide``: uniform over 97..131
    (2**-30 .. 2**4)."""
    if wide:
        return rng.integers(97, 132, size=(rows, cols // 32), dtype=np.uint8).astype(np.uint8)
    return (120 + rng.integers(0, 2, size=(rows, cols // 32), dtype=np.uint8)).astype(np.uint8)


def nv_scales(rng: np.random.Generator, rows: int, cols: int, wide: bool = False) -> np.ndarray:
    """[rows, cols/16] E4M3 bytes uniform in [0x30, 0x48); ``wide``: uniform over every positive
    finite non-zero code 0x01 .. 0x7E (subnormal 2**-9 up to 448)."""
    if wide:
        return rng.integers(0x01, 0x7F, size=(rows, cols // 16), dtype=np.uint8).astype(np.uint8)
    return (0x30 + rng.integers(0, 0x18, size=(rows, cols // 16), dtype=np.uint8)).astype(np.uint8)


def expert_weights(w: Workload, e: int) -> dict:
    """Weights of expert e in the logical layouts: W13 [2I, H] (rows 0..I-1 gate, I..2I-1 up), W2 [H, I].

    FP4 formats: ``*_q`` packed E2M1 [N, Kd/2], ``*_sf`` block scales, ``*_ts`` NVFP4 tensor scale.
    INT8: ``*_q`` int8 [N, Kd], ``*_sf`` float32 channel scales [N], ``*_ts`` None.
    INT8 with [256, 256] blocks ("int8b"): ``*_sf`` float32 block scales [N/256, Kd/256].
    """
    out = {}
    for mat, (rows, cols) in (("w13", (2 * w.I, w.H)), ("w2", (w.H, w.I))):
        rng = _rng(w.seed, 1 if mat == "w13" else 2, e)
        if w.fmt in ("int8", "int8b"):
            out[mat + "_q"] = i8_codes(rng, rows, cols)
            out[mat + "_sf"] = i8_channel_scales(rng, rows) if w.fmt == "int8" else i8_block_scales(rng, rows, cols)
            out[mat + "_ts"] = None
            continue
        out[mat + "_q"] = fp4_codes(rng, rows, cols)
        if w.fmt == "mxfp4":
            out[mat + "_sf"] = mx_scales(rng, rows, cols, w.wide_scales)
            out[mat + "_ts"] = None
        else:
            out[mat + "_sf"] = nv_scales(rng, rows, cols, w.wide_scales)
            out[mat + "_ts"] = np.float32(rng.uniform(0.0058, 0.0068))
    return out


def all_expert_weights(w: Workload, threads: int = 16) -> dict:
    """Stacked [E, ...] weight arrays for every expert (experts generated in parallel threads)."""
    from concurrent.futures import ThreadPoolExecutor
    first = expert_weights(w, 0)
    out = {k: np.empty((w.E,) + first[k].shape, dtype=first[k].dtype)
           for k in ("w13_q", "w13_sf", "w2_q", "w2_sf")}
    ts = {"w13_ts": np.zeros(w.E, np.float32), "w2_ts": np.zeros(w.E, np.float32)}

    def fill(e):
        p = first if e == 0 else expert_weights(w, e)
        for k in out:
            out[k][e] = p[k]
        if w.fmt == "nvfp4":
            ts["w13_ts"][e] = p["w13_ts"]
            ts["w2_ts"][e] = p["w2_ts"]

    with ThreadPoolExecutor(max(1, threads)) as ex:
        list(ex.map(fill, range(w.E)))
    if w.fmt == "nvfp4":
        out.update(ts)
    else:
        out["w13_ts"] = None
        out["w2_ts"] = None
    return out


def bf16_bits_from_normal(rng: np.random.Generator, shape, scale=1.0) -> np.ndarray:
    x = (rng.standard_normal(size=shape) * scale).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def layer_inputs(w: Workload, T: Optional[int] = None) -> dict:
    """hidden [T,H] bf16 bits, w_gate [E,H] f32, gate_bias [E] f32 or None, e_score_bias [E] f32 or None."""
    T = w.T if T is None else T
    rng = _rng(w.seed, 0)
    hidden = bf16_bits_from_normal(rng, (T, w.H))
    if w.gate_uniform:
        a = np.sqrt(3.0 / w.H)
        w_gate = rng.uniform(-a, a, size=(w.E, w.H)).astype(np.float32)
    else:
        w_gate = (rng.standard_normal(size=(w.E, w.H)) / np.sqrt(w.H)).astype(np.float32)
    e_bias = (rng.standard_normal(size=w.E) * 0.1).astype(np.float32) if w.e_bias else None
    if w.gate_offset == "normal":
        gate_bias = rng.standard_normal(size=w.E).astype(np.float32)
    elif w.gate_offset == "zipf":
        # popularity p_e proportional to rank**-1.1 over a seeded permutation of the experts,
        # injected as gate bias beta * ln(p_e / p_max) with beta = 1
        perm = rng.permutation(w.E)
        rank = np.empty(w.E, dtype=np.float64)
        rank[perm] = np.arange(1, w.E + 1)
        gate_bias = (-1.1 * np.log(rank)).astype(np.float32)
    else:
        gate_bias = None
    return dict(hidden=hidden, w_gate=w_gate, gate_bias=gate_bias, e_score_bias=e_bias)


# --- stage inputs drawn directly (for per-stage tests that must not feed one stage's
# --- GPU output into the next stage's oracle)

def e4m3_codes(rng: np.random.Generator, shape, wide: bool = False) -> np.ndarray:
    """E4M3 codes with uniform sign, exponent field uniform in 3..14, uniform mantissa (no NaN).

    ``wide``: every non-NaN code with equal odds (zeros, subnormals and the top binade up to 448)."""
    if wide:
        c = rng.integers(0, 254, size=shape, dtype=np.int32)      # 254 non-NaN codes
        c = c + (c >= 0x7F) + (c >= 0xFE)                         # skip 0x7F and 0xFF
        return c.astype(np.uint8)
    s = rng.integers(0, 2, size=shape, dtype=np.uint8)
    e = rng.integers(3, 15, size=shape, dtype=np.uint8)
    m = rng.integers(0, 8, size=shape, dtype=np.uint8)
    return ((s << 7) | (e << 3) | m).astype(np.uint8)


def act_scale_codes(rng: np.random.Generator, shape, wide: bool = False) -> np.ndarray:
    """UE8M0 activation scales in 2**-10 .. 2**-6; ``wide``: uniform over 2**-120 .. 2**10."""
    if wide:
        return rng.integers(7, 138, size=shape, dtype=np.uint8).astype(np.uint8)
    return (117 + rng.integers(0, 5, size=shape, dtype=np.uint8)).astype(np.uint8)


def topk_ids_random(rng: np.random.Generator, T: int, E: int, K: int, skew: float = 0.0) -> np.ndarray:
    """Distinct expert ids per token; with skew > 0 expert e is drawn with weight (e+1)**-skew."""
    p = np.arange(1, E + 1, dtype=np.float64) ** (-skew)
    p /= p.sum()
    out = np.empty((T, K), dtype=np.int32)
    for t in range(T):
        out[t] = rng.choice(E, size=K, replace=False, p=p)
    return out


def topk_weights_random(rng: np.random.Generator, T: int, K: int) -> np.ndarray:
    w = rng.uniform(0.05, 1.0, size=(T, K)).astype(np.float32)
    return w


def bf16_rows(rng: np.random.Generator, rows: int, cols: int, scale=1.0) -> np.ndarray:
    return bf16_bits_from_normal(rng, (rows, cols), scale)
