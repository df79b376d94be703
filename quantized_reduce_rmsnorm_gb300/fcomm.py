"""Thin Python binding of libfcomm (ctypes): argument marshalling only.

Every step of the path runs in libfcomm's CUDA kernels; this module only
turns torch tensors into device pointers and the current torch stream into a
cudaStream_t, calls the C entry point of the same name, and raises FcommError
on a non-OK status.  There is no CPU fallback: if the library cannot be
built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import build as _build

FMT_BF16, FMT_INT8_SYM, FMT_INT4_ASYM, FMT_BF16_TAGGED, FMT_F32 = 0, 1, 2, 3, 4
FMT_INT8_TAGGED, FMT_INT4_TAGGED = 5, 6
FC_OK, FC_ERR_INVALID, FC_ERR_CUDA, FC_ERR_STALE_BLOCK, FC_ERR_UNSUPPORTED = 0, 1, 2, 3, 4
STATUS_NO_INDEX = 0x7F7F7F7F

# Names exported by the C ABI (include/fcomm.h)
EXPORTS = (
    "fc_codes_bytes", "fc_groups", "fc_tagged_bytes", "fc_shard_range", "fc_group_quantize",
    "fc_group_quantize_multi", "fc_reduce_dequant_sum", "fc_requant_gather", "fc_pack_tagged",
    "fc_pack_tagged_multi", "fc_group_quantize_tagged",
    "fc_allreduce_residual_rmsnorm", "fc_allreduce_residual_rmsnorm_ex", "fc_status_string",
    "fc_last_error", "fc_version", "fc_token_split", "fc_select_protocol", "fc_allgather_dequant",
    "fc_protocol_estimate",
)


class FcommError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_STATUS_NAMES = {0: "FC_OK", 1: "FC_ERR_INVALID", 2: "FC_ERR_CUDA", 3: "FC_ERR_STALE_BLOCK",
                 4: "FC_ERR_UNSUPPORTED"}


class QSpec(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("group", ctypes.c_int32)]

    def __repr__(self):
        return f"QSpec(fmt={self.fmt}, group={self.group})"


class QTensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zeros", ctypes.c_void_p)]


class LinkModel(ctypes.Structure):
    _fields_ = [("link_gbps", ctypes.c_double), ("barrier_us", ctypes.c_double)]


class LaunchOpts(ctypes.Structure):
    _fields_ = [("max_ctas", ctypes.c_int32), ("kernel", ctypes.c_int32)]


KERNEL_AUTO, KERNEL_STREAM, KERNEL_TMA = 0, 1, 2


INT8_G128 = QSpec(FMT_INT8_SYM, 128)
INT4_G32 = QSpec(FMT_INT4_ASYM, 32)
BF16 = QSpec(FMT_BF16, 0)
BF16_TAGGED = QSpec(FMT_BF16_TAGGED, 0)
INT8_G128_TAGGED = QSpec(FMT_INT8_TAGGED, 128)
INT4_G32_TAGGED = QSpec(FMT_INT4_TAGGED, 32)

_lib = None


def lib_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None):
    """Load libfcomm.so (building it with nvcc if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or _build.build()
    lib = ctypes.CDLL(p)
    P, i64, i32, u32, f32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32,
                             ctypes.c_float)
    QS, QT = QSpec, QTensor
    sigs = {
        "fc_codes_bytes": (ctypes.c_size_t, [QS, i64, i64]),
        "fc_groups": (ctypes.c_size_t, [QS, i64, i64]),
        "fc_tagged_bytes": (ctypes.c_size_t, [i64, i64]),
        "fc_shard_range": (i32, [QS, i64, i64, i32, i32, ctypes.POINTER(i64),
                                 ctypes.POINTER(i64)]),
        "fc_group_quantize": (i32, [P, i64, i64, QS, QT, P, P]),
        "fc_group_quantize_multi": (i32, [P, i32, i64, i64, QS, P, P, P]),
        "fc_reduce_dequant_sum": (i32, [P, i32, i64, i64, QS, i32, P, P]),
        "fc_requant_gather": (i32, [P, i64, i64, QS, QT, P, i32, P]),
        "fc_allgather_dequant": (i32, [ctypes.POINTER(QT), i32, i64, i64, QS, i32, P, u32, P, P]),
        "fc_pack_tagged": (i32, [P, i64, i64, u32, P, P]),
        "fc_pack_tagged_multi": (i32, [P, i32, i64, i64, u32, P, P]),
        "fc_group_quantize_tagged": (i32, [P, i32, i64, i64, QS, u32, P, P, P]),
        "fc_allreduce_residual_rmsnorm": (
            i32, [P, i32, i64, i64, QS, P, P, P, f32, QT, P, u32, P, P]),
        "fc_allreduce_residual_rmsnorm_ex": (
            i32, [P, i32, i64, i64, QS, P, P, P, f32, QT, P, u32, P, P, P]),
        "fc_status_string": (ctypes.c_char_p, [i32]),
        "fc_last_error": (ctypes.c_char_p, []),
        "fc_version": (ctypes.c_char_p, []),
        "fc_token_split": (i32, [i32, i64, i64, QS, ctypes.POINTER(i64), ctypes.POINTER(i64)]),
        "fc_select_protocol": (i32, [i64, i64, i32, i32, P, ctypes.POINTER(QSpec),
                                     ctypes.POINTER(ctypes.c_double)]),
        "fc_protocol_estimate": (i32, [i64, i64, i32, QS, P, ctypes.POINTER(ctypes.c_double)]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != FC_OK:
        raise FcommError(status, _lib.fc_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libfcomm takes CUDA tensors (device memory)")
    if not t.is_contiguous():
        raise ValueError("libfcomm takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _qt(q) -> QTensor:
    """(codes, scales, zeros) tuple of tensors (or None entries) -> QTensor."""
    if q is None:
        return QTensor(None, None, None)
    codes, scales, zeros = (tuple(q) + (None, None, None))[:3]
    return QTensor(_ptr(codes), _ptr(scales), _ptr(zeros))


class Bound:
    """One libfcomm call with its arguments marshalled once.

    Calling it launches the entry point again with the same device pointers
    on `stream` (default: the current torch stream), with no per-call
    argument conversion: the host cost of a call is the C entry point
    itself.  The object holds a reference to every tensor it was bound to,
    so their memory cannot be freed and handed to another tensor while the
    bound call exists.  For the calls that carry an epoch (tagged formats),
    `epoch` may be changed between calls."""
    __slots__ = ("_fn", "_args", "_si", "_ei", "_keep")

    def __init__(self, fn, args, stream_index, epoch_index=None, keep=()):
        self._fn, self._args, self._si, self._ei, self._keep = fn, list(args), stream_index, \
            epoch_index, keep

    @property
    def epoch(self) -> int:
        return self._args[self._ei].value

    @epoch.setter
    def epoch(self, e: int):
        self._args[self._ei] = ctypes.c_uint32(e & 0xFFFFFFFF)

    def __call__(self, stream=None):
        a = self._args
        a[self._si] = _stream(stream)
        st = self._fn(*a)
        if st != FC_OK:
            _check(st)


def _rows_hidden(x: torch.Tensor):
    if x.dim() != 2:
        raise ValueError("expected a [rows, hidden] tensor")
    return x.shape[0], x.shape[1]


# ----------------------------------------------------------------- sizes ---
def codes_bytes(spec: QSpec, rows: int, hidden: int) -> int:
    return load().fc_codes_bytes(spec, rows, hidden)


def groups(spec: QSpec, rows: int, hidden: int) -> int:
    return load().fc_groups(spec, rows, hidden)


def tagged_bytes(rows: int, hidden: int) -> int:
    return load().fc_tagged_bytes(rows, hidden)


def shard_range(spec: QSpec, rows: int, hidden: int, P: int, shard: int):
    g0, g1 = ctypes.c_int64(), ctypes.c_int64()
    _check(load().fc_shard_range(spec, rows, hidden, P, shard, ctypes.byref(g0), ctypes.byref(g1)))
    return g0.value, g1.value


def alloc_qtensor(spec: QSpec, rows: int, hidden: int, device="cuda"):
    """Caller-owned (codes, scales, zeros) torch tensors for a quantized tensor."""
    nb = codes_bytes(spec, rows, hidden)
    ng = groups(spec, rows, hidden)
    codes = torch.empty(nb, dtype=torch.uint8, device=device)
    scales = torch.empty(ng, dtype=torch.float32, device=device)
    zeros = torch.empty(ng, dtype=torch.float32, device=device) if spec.fmt == FMT_INT4_ASYM \
        else None
    return codes, scales, zeros


# --------------------------------------------------------------- compute ---
def group_quantize(x: torch.Tensor, spec: QSpec, out, stream=None,
                   d_status: Optional[torch.Tensor] = None):
    """Quantize one [rows, hidden] bf16 slab into out = (codes, scales[, zeros]);
    d_status: optional int32[2] device status words (see fcomm.h)."""
    rows, hidden = _rows_hidden(x)
    _check(load().fc_group_quantize(_ptr(x), rows, hidden, spec, _qt(out), _ptr(d_status),
                                    _stream(stream)))


def bind_group_quantize_multi(xs: Sequence[torch.Tensor], spec: QSpec, outs,
                              d_status: Optional[torch.Tensor] = None) -> Bound:
    rows, hidden = _rows_hidden(xs[0])
    xp = (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])
    qo = (QTensor * len(outs))(*[_qt(o) for o in outs])
    return Bound(load().fc_group_quantize_multi,
                 [xp, len(xs), rows, hidden, spec, qo, ctypes.c_void_p(_ptr(d_status)), None], 7,
                 keep=(tuple(xs), tuple(outs), d_status))


def group_quantize_multi(xs: Sequence[torch.Tensor], spec: QSpec, outs, stream=None,
                         d_status: Optional[torch.Tensor] = None):
    bind_group_quantize_multi(xs, spec, outs, d_status)(stream)


def reduce_dequant_sum(slabs, spec: QSpec, rows: int, hidden: int, out: torch.Tensor,
                       shard: int = -1, stream=None):
    """out[rows, hidden] fp32 = fixed-order sum of the dequantized slabs (or one shard)."""
    qs = (QTensor * len(slabs))(*[_qt(s) for s in slabs])
    _check(load().fc_reduce_dequant_sum(qs, len(slabs), rows, hidden, spec, shard, _ptr(out),
                                        _stream(stream)))


def requant_gather(reduced: torch.Tensor, spec: QSpec, requant_out=None,
                   out: Optional[torch.Tensor] = None, out_dtype: int = FMT_BF16, stream=None):
    rows, hidden = _rows_hidden(reduced)
    _check(load().fc_requant_gather(_ptr(reduced), rows, hidden, spec, _qt(requant_out),
                                    _ptr(out), out_dtype, _stream(stream)))


def allgather_dequant(shards, spec: QSpec, rows: int, hidden: int, out: torch.Tensor,
                      expected_epoch: int = 0, d_status: Optional[torch.Tensor] = None,
                      stream=None):
    """Standalone quantized all-gather: shards = P (codes, scales, zeros) tuples
    (or tagged-block tensors), shard p holding groups [p*per, min((p+1)*per,
    n_g)) from its own index 0; out = the whole dequantized [rows, hidden]
    tensor (bf16 or fp32, by its dtype)."""
    qs = (QTensor * len(shards))(*[_qt(s if isinstance(s, (tuple, list)) else (s,))
                                   for s in shards])
    od = FMT_F32 if out.dtype == torch.float32 else FMT_BF16
    _check(load().fc_allgather_dequant(qs, len(shards), rows, hidden, spec, od, _ptr(out),
                                       expected_epoch, _ptr(d_status), _stream(stream)))


def bind_allgather_dequant(shards, spec: QSpec, rows: int, hidden: int, out: torch.Tensor,
                           expected_epoch: int = 0, d_status: Optional[torch.Tensor] = None) -> Bound:
    """allgather_dequant with its arguments marshalled once (fcomm.Bound)."""
    qs = (QTensor * len(shards))(*[_qt(s if isinstance(s, (tuple, list)) else (s,))
                                   for s in shards])
    od = FMT_F32 if out.dtype == torch.float32 else FMT_BF16
    return Bound(load().fc_allgather_dequant,
                 [qs, len(shards), rows, hidden, spec, od, ctypes.c_void_p(_ptr(out)),
                  ctypes.c_uint32(expected_epoch & 0xFFFFFFFF), ctypes.c_void_p(_ptr(d_status)),
                  None], 9,
                 epoch_index=7, keep=(shards, out, d_status, qs))


def shard_views(q, spec: QSpec, rows: int, hidden: int, P: int):
    """The P shard payloads (views, no copy) of a whole payload q = (codes,
    scales, zeros) or tagged blocks, in the partition fc_allgather_dequant reads."""
    ng = groups(spec, rows, hidden)
    per = -(-ng // P)
    if spec.fmt in (FMT_INT8_TAGGED, FMT_INT4_TAGGED):
        nbg = 11 if spec.fmt == FMT_INT8_TAGGED else 2
        b = q if isinstance(q, torch.Tensor) else q[0]
        return [b[min(j * per, ng) * nbg * 16:min((j + 1) * per, ng) * nbg * 16] for j in range(P)]
    cb = spec.group if spec.fmt == FMT_INT8_SYM else spec.group // 2
    codes, scales, zeros = (tuple(q) + (None, None, None))[:3]
    out = []
    for j in range(P):
        g0, g1 = min(j * per, ng), min((j + 1) * per, ng)
        if g1 <= g0:
            out.append((None, None, None))
            continue
        out.append((codes[g0 * cb:g1 * cb], scales[g0:g1], None if zeros is None else zeros[g0:g1]))
    return out


def pack_tagged(x: torch.Tensor, epoch: int, blocks: torch.Tensor, stream=None):
    rows, hidden = _rows_hidden(x)
    _check(load().fc_pack_tagged(_ptr(x), rows, hidden, epoch, _ptr(blocks), _stream(stream)))


def bind_group_quantize_tagged(xs: Sequence[torch.Tensor], spec: QSpec, epoch: int,
                               blocks: Sequence[torch.Tensor],
                               d_status: Optional[torch.Tensor] = None) -> Bound:
    rows, hidden = _rows_hidden(xs[0])
    xp = (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])
    bp = (ctypes.c_void_p * len(blocks))(*[_ptr(b) for b in blocks])
    return Bound(load().fc_group_quantize_tagged,
                 [xp, len(xs), rows, hidden, spec, ctypes.c_uint32(epoch), bp,
                  ctypes.c_void_p(_ptr(d_status)), None], 8, 5,
                 keep=(tuple(xs), tuple(blocks), d_status))


def group_quantize_tagged(xs: Sequence[torch.Tensor], spec: QSpec, epoch: int,
                          blocks: Sequence[torch.Tensor], stream=None,
                          d_status: Optional[torch.Tensor] = None):
    """Quantize P bf16 slabs straight into self-synchronizing blocks."""
    bind_group_quantize_tagged(xs, spec, epoch, blocks, d_status)(stream)


def bind_pack_tagged_multi(xs: Sequence[torch.Tensor], epoch: int,
                           blocks: Sequence[torch.Tensor]) -> Bound:
    rows, hidden = _rows_hidden(xs[0])
    xp = (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])
    bp = (ctypes.c_void_p * len(blocks))(*[_ptr(b) for b in blocks])
    return Bound(load().fc_pack_tagged_multi,
                 [xp, len(xs), rows, hidden, ctypes.c_uint32(epoch), bp, None], 6, 4,
                 keep=(tuple(xs), tuple(blocks)))


def pack_tagged_multi(xs: Sequence[torch.Tensor], epoch: int, blocks: Sequence[torch.Tensor],
                      stream=None):
    bind_pack_tagged_multi(xs, epoch, blocks)(stream)


def allreduce_residual_rmsnorm(slabs, spec: QSpec, rows: int, hidden: int,
                               residual_in: torch.Tensor, residual_out: torch.Tensor,
                               gamma: torch.Tensor, eps: float, y: torch.Tensor,
                               requant_out=None, expected_epoch: int = 0,
                               d_status: Optional[torch.Tensor] = None, max_ctas: int = 0,
                               kernel: int = KERNEL_AUTO, stream=None):
    """The fused quantized All-Reduce + residual add + RMSNorm.

    slabs: list of P (codes, scales, zeros) tuples (INT8/INT4), or of bf16
    tensors / tagged-block tensors (BF16 / BF16_TAGGED)."""
    bind_allreduce_residual_rmsnorm(slabs, spec, rows, hidden, residual_in, residual_out, gamma,
                                    eps, y, requant_out, expected_epoch, d_status, max_ctas,
                                    kernel)(stream)


def bind_allreduce_residual_rmsnorm(slabs, spec: QSpec, rows: int, hidden: int,
                                    residual_in: torch.Tensor, residual_out: torch.Tensor,
                                    gamma: torch.Tensor, eps: float, y: torch.Tensor,
                                    requant_out=None, expected_epoch: int = 0,
                                    d_status: Optional[torch.Tensor] = None, max_ctas: int = 0,
                                    kernel: int = KERNEL_AUTO) -> Bound:
    """allreduce_residual_rmsnorm with its arguments marshalled once (Bound)."""
    qs = (QTensor * len(slabs))(*[_qt(s if isinstance(s, (tuple, list)) else (s,))
                                  for s in slabs])
    opts = LaunchOpts(max_ctas, kernel)
    P = ctypes.c_void_p
    args = [qs, len(slabs), rows, hidden, spec, P(_ptr(residual_in)), P(_ptr(residual_out)),
            P(_ptr(gamma)), ctypes.c_float(eps), _qt(requant_out), P(_ptr(y)),
            ctypes.c_uint32(expected_epoch), P(_ptr(d_status)), ctypes.byref(opts), None]
    return Bound(load().fc_allreduce_residual_rmsnorm_ex, args, 14, 11,
                 keep=(opts, tuple(slabs), residual_in, residual_out, gamma, y, requant_out,
                       d_status))


def token_split(spec: QSpec, P: int, rows: int, hidden: int):
    """(first subset's rows, wave rows) of the wave-aware token split."""
    sp, wv = ctypes.c_int64(), ctypes.c_int64()
    _check(load().fc_token_split(P, rows, hidden, spec, ctypes.byref(sp), ctypes.byref(wv)))
    return sp.value, wv.value


def select_protocol(rows: int, hidden: int, P: int, min_bits: int,
                    link_gbps: Optional[float] = None, barrier_us: float = 0.0):
    """(QSpec, estimated us) of the cost-guided format choice."""
    link = LinkModel(link_gbps, barrier_us) if link_gbps is not None else None
    choice, est = QSpec(), ctypes.c_double()
    _check(load().fc_select_protocol(rows, hidden, P, min_bits,
                                     ctypes.byref(link) if link is not None else None,
                                     ctypes.byref(choice), ctypes.byref(est)))
    return choice, est.value


def version() -> str:
    return load().fc_version().decode()


def protocol_estimate(rows: int, hidden: int, P: int, spec: QSpec,
                      link_gbps: Optional[float] = None, barrier_us: float = 0.0) -> float:
    """The selector's estimated us of one step in encoding `spec`."""
    link = LinkModel(link_gbps, barrier_us) if link_gbps is not None else None
    est = ctypes.c_double()
    _check(load().fc_protocol_estimate(rows, hidden, P, spec,
                                       ctypes.byref(link) if link is not None else None,
                                       ctypes.byref(est)))
    return est.value
