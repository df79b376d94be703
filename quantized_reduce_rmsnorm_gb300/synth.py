"""Seeded synthetic inputs: partial-sum activation slabs, residual, gamma.

This module only draws random numbers and rounds them to bf16 storage; it
holds none of the method's arithmetic.  Both the CUDA path (through the
binding) and the CPU oracle (in the tests) consume exactly the bits it
returns, so the two sides always see identical inputs.

Random streams: numpy's Philox-4x64 counter-based generator keyed by
(seed, stream, row chunk).  Rows are drawn in chunks of ``ROW_CHUNK`` rows so a
sample of rows can be regenerated without drawing the whole tensor.  bf16
storage is produced by torch's float32 -> bfloat16 conversion (round to
nearest even) and handed out as uint16 bit patterns.

Workloads (tensor-parallel activations standing in for the pages' LLaMA-class
models; no dataset or weights are involved):

* ``decode-tiny``: P=2 slabs, 1 token x hidden 4096, N(0,1); INT8 symmetric g128.
* ``decode``: P=8, 64 x 8192, Student-t (3 degrees of freedom) with 0.1% of the
  channels scaled x50; INT8 symmetric g128.
* ``prefill``: P=4, 8192 x 8192, N(0,1) with 0.5% of the channels scaled x20;
  INT4 asymmetric g32.
* ``token-split``: P=8, 4096 x 5120 bf16, N(0,1), sent as epoch-tagged 16-byte
  blocks, processed as two subsets of 2048 rows.
* ``sweep``: message 16 KB .. 256 MB, hidden 4096 or 8192, P in {2,4,8},
  format in {bf16, INT8 g128, INT4 g32}, N(0,1).
* ``decode-qtagged`` / ``prefill-qtagged``: decode / prefill with the quantized
  groups sent as self-synchronizing (epoch-tagged) 16-byte blocks.

Every workload: residual N(0,1), gamma N(1, 0.1), eps 1e-5.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import os

import numpy as np
import torch

ROW_CHUNK = 64

# stream ids
_S_RESIDUAL, _S_GAMMA, _S_OUTLIER = 100, 101, 102

FMT_BF16, FMT_INT8_SYM, FMT_INT4_ASYM, FMT_BF16_TAGGED = 0, 1, 2, 3
FMT_INT8_TAGGED, FMT_INT4_TAGGED = 5, 6
FMT_NAMES = {FMT_BF16: "bf16", FMT_INT8_SYM: "int8_sym_g128",
             FMT_INT4_ASYM: "int4_asym_g32", FMT_BF16_TAGGED: "bf16_tagged",
             FMT_INT8_TAGGED: "int8_sym_g128_tagged", FMT_INT4_TAGGED: "int4_asym_g32_tagged"}
QUANTIZED = (FMT_INT8_SYM, FMT_INT4_ASYM, FMT_INT8_TAGGED, FMT_INT4_TAGGED)
QTAGGED = (FMT_INT8_TAGGED, FMT_INT4_TAGGED)


def base_format(fmt: int) -> int:
    """The plain quantized format a tagged quantized format carries."""
    return {FMT_INT8_TAGGED: FMT_INT8_SYM, FMT_INT4_TAGGED: FMT_INT4_ASYM}.get(fmt, fmt)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    P: int
    T: int
    H: int
    fmt: int
    group: int
    dist: str = "normal"          # "normal" or "student_t3"
    outlier_frac: float = 0.0     # fraction of hidden channels scaled
    outlier_scale: float = 1.0
    splits: int = 1               # token subsets run on separate streams
    eps: float = 1e-5

    @property
    def n_outliers(self) -> int:
        return int(round(self.outlier_frac * self.H))


WORKLOADS = {
    "decode-tiny": Workload("decode-tiny", P=2, T=1, H=4096, fmt=FMT_INT8_SYM, group=128),
    "decode": Workload("decode", P=8, T=64, H=8192, fmt=FMT_INT8_SYM, group=128,
                       dist="student_t3", outlier_frac=0.001, outlier_scale=50.0),
    "prefill": Workload("prefill", P=4, T=8192, H=8192, fmt=FMT_INT4_ASYM, group=32,
                        outlier_frac=0.005, outlier_scale=20.0),
    "token-split": Workload("token-split", P=8, T=4096, H=5120, fmt=FMT_BF16_TAGGED, group=0,
                            splits=2),
    # the decode and prefill workloads with self-synchronizing quantized payloads
    "decode-qtagged": Workload("decode-qtagged", P=8, T=64, H=8192, fmt=FMT_INT8_TAGGED,
                               group=128, dist="student_t3", outlier_frac=0.001,
                               outlier_scale=50.0),
    "prefill-qtagged": Workload("prefill-qtagged", P=4, T=8192, H=8192, fmt=FMT_INT4_TAGGED,
                                group=32, outlier_frac=0.005, outlier_scale=20.0),
}


SWEEP_FORMATS = ((FMT_BF16, 0), (FMT_INT8_SYM, 128), (FMT_INT4_ASYM, 32))
# the self-synchronizing encodings of the same payloads (rates for the
# protocol selector; the sweep's figure of merit is the untagged three)
SWEEP_TAGGED_FORMATS = ((FMT_BF16_TAGGED, 0), (FMT_INT8_TAGGED, 128), (FMT_INT4_TAGGED, 32))


def sweep_points(formats=SWEEP_FORMATS):
    """(message bytes, H, T, P, fmt, group) of the message-size sweep."""
    pts = []
    for i in range(15):
        msg = (16 << 10) << i
        for H in (4096, 8192):
            T = msg // (2 * H)
            for P in (2, 4, 8):
                for fmt, G in formats:
                    pts.append((msg, H, T, P, fmt, G))
    return pts


def sweep_workload(H, T, P, fmt, G) -> Workload:
    return Workload(f"sweep-h{H}-t{T}-p{P}-{FMT_NAMES[fmt]}", P=P, T=T, H=H, fmt=fmt, group=G)


def _rng(seed: int, stream: int, chunk: int) -> np.random.Generator:
    key = np.array([seed & 0xFFFFFFFFFFFFFFFF, (stream << 32) | chunk], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def _to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _draw(rng: np.random.Generator, n: int, dist: str) -> np.ndarray:
    if dist == "normal":
        return rng.standard_normal(n, dtype=np.float32)
    if dist == "student_t3":
        return rng.standard_t(3, n).astype(np.float32)
    raise ValueError(dist)


def outlier_channels(w: Workload, seed: int = 0) -> np.ndarray:
    """Sorted hidden-channel indices scaled by w.outlier_scale (same for all slabs and rows)."""
    k = w.n_outliers
    if k == 0:
        return np.zeros(0, np.int64)
    return np.sort(_rng(seed, _S_OUTLIER, 0).choice(w.H, size=k, replace=False))


def _rows_tensor(w: Workload, seed: int, stream: int, rows: np.ndarray, dist: str,
                 outliers: np.ndarray) -> np.ndarray:
    """bf16 bits [len(rows), H] of the given rows of one [T, H] stream."""
    out = np.empty((len(rows), w.H), np.uint16)
    rows = np.asarray(rows, np.int64)

    def fill(c):
        r0 = int(c) * ROW_CHUNK
        nr = min(ROW_CHUNK, w.T - r0)
        x = _draw(_rng(seed, stream, int(c)), nr * w.H, dist).reshape(nr, w.H)
        if len(outliers):
            x[:, outliers] *= np.float32(w.outlier_scale)
        sel = np.nonzero(rows // ROW_CHUNK == c)[0]
        out[sel] = _to_bf16_bits(x[rows[sel] - r0])

    chunks = np.unique(rows // ROW_CHUNK)
    if len(chunks) > 4:
        # each chunk has its own counter-based stream, so the result does not
        # depend on how chunks are scheduled over threads
        with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, chunks))
    else:
        for c in chunks:
            fill(c)
    return out


def slab(w: Workload, p: int, seed: int = 0, rows=None) -> np.ndarray:
    """Partial-sum slab p as bf16 bits [T, H] (or the given rows)."""
    rows = np.arange(w.T) if rows is None else np.asarray(rows)
    return _rows_tensor(w, seed, p, rows, w.dist, outlier_channels(w, seed))


def residual(w: Workload, seed: int = 0, rows=None) -> np.ndarray:
    rows = np.arange(w.T) if rows is None else np.asarray(rows)
    return _rows_tensor(w, seed, _S_RESIDUAL, rows, "normal", np.zeros(0, np.int64))


def gamma(w: Workload, seed: int = 0) -> np.ndarray:
    g = 1.0 + 0.1 * _rng(seed, _S_GAMMA, 0).standard_normal(w.H, dtype=np.float32)
    return _to_bf16_bits(g.astype(np.float32))


def make_inputs(w: Workload, seed: int = 0, rows=None) -> dict:
    """All host inputs of one workload: dict(slabs=[...], residual, gamma)."""
    return dict(slabs=[slab(w, p, seed, rows) for p in range(w.P)],
                residual=residual(w, seed, rows), gamma=gamma(w, seed))
