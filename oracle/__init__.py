"""CPU oracle for the quantized reduce + residual-add + RMSNorm path.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product package never imports
this module, and this module never imports the product package.

The arithmetic lives in ``oracle.c`` (plain scalar C, one binary32 operation
per float expression, no fused multiply-add); this file only compiles it with
gcc and marshals numpy arrays into it.  Each function cites the page and
section it follows:

* "Flash Communication: Reducing Tensor Parallelization Bottleneck for Fast
  Large Language Model Inference" (arXiv 2412.04964), summary, "Main
  contributions" item 2 and "Core ideas": fine-grained low-bit quantization of
  activations, two-step All-Reduce.
* flash-comm, abstract: self-synchronizing blocks; reduction order fixed
  independently of arrival order.
* "TokenWeave: Efficient Compute-Communication Overlap for Distributed LLM
  Inference" (arXiv 2505.11329), abstract: RMSNorm fused after the All-Reduce.

No function here is "parity unpinned": tests/test_oracle_pins.py pins each one
to closed forms, brute force, invariants or an independent library routine.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

FMT_BF16, FMT_INT8_SYM, FMT_INT4_ASYM, FMT_BF16_TAGGED = 0, 1, 2, 3

def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle C source into a shared library (strict IEEE binary32)."""
    stale = force or not os.path.exists(out) or max(
        os.path.getmtime(src), os.path.getmtime(_HDR)) > os.path.getmtime(out)
    if stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fexcess-precision=standard", "-I", _HERE, "-fPIC", "-shared", src,
               "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _signatures():
    P, i64, i32, u32, f32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                             ctypes.c_uint32, ctypes.c_float)
    return {
        "or_bf16_to_f32_array": (None, [P, i64, P]),
        "or_f32_to_bf16": (ctypes.c_uint16, [f32]),
        "or_f32_to_bf16_array": (None, [P, i64, P]),
        "or_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
        "or_quant_i8s": (None, [P, i64, i32, P, P]),
        "or_dequant_i8s": (None, [P, P, i64, i32, P]),
        "or_quant_i4a": (None, [P, i64, i32, P, P, P]),
        "or_dequant_i4a": (None, [P, P, P, i64, i32, P]),
        "or_reduce_sum": (None, [P, i32, i64, P]),
        "or_two_step": (i32, [i32, P, P, P, i32, i64, i32, i32, P, P, P, P, P]),
        "or_allgather_dequant": (i32, [i32, P, P, P, i32, i64, i32, P]),
        "or_residual_rmsnorm": (None, [P, P, P, i64, i64, f32, P, P]),
        "or_tagged_blocks_per_row": (i64, [i64]),
        "or_pack_tagged": (None, [P, i64, i64, u32, P]),
        "or_validate_tagged": (i64, [P, i64, u32]),
        "or_unpack_tagged": (None, [P, i64, i64, P]),
        "or_qtagged_blocks_per_group": (i32, [i32, i32]),
        "or_pack_qtagged": (None, [i32, P, P, P, i64, i32, u32, P]),
        "or_unpack_qtagged": (i64, [i32, P, i64, i32, u32, P, P, P]),
        "or_allreduce_residual_rmsnorm": (
            i32, [i32, P, i32, i64, i64, i32, P, P, f32, P, P, P, P, P]),
    }


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptrs(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


class Oracle:
    """numpy front end of one compiled copy of the oracle library."""

    def __init__(self, lib_path: str):
        self.lib = ctypes.CDLL(lib_path)
        for name, (res, args) in _signatures().items():
            fn = getattr(self.lib, name)
            fn.restype = res
            fn.argtypes = args

    # -------------------------------------------------------------- bf16 ---
    def bf16_to_f32(self, b):
        b = _c(b, np.uint16)
        out = np.empty(b.shape, np.float32)
        self.lib.or_bf16_to_f32_array(_p(b), b.size, _p(out))
        return out

    def f32_to_bf16(self, x):
        x = _c(x, np.float32)
        fn = self.lib.or_f32_to_bf16
        return np.array([fn(float(v)) for v in x.ravel()], np.uint16).reshape(x.shape)

    def f32_to_bf16_array(self, x):
        """Same rounding as f32_to_bf16, one C loop over the whole array."""
        x = _c(x, np.float32)
        out = np.empty(x.shape, np.uint16)
        self.lib.or_f32_to_bf16_array(_p(x), x.size, _p(out))
        return out

    def f64_to_bf16(self, x):
        x = _c(x, np.float64)
        fn = self.lib.or_f64_to_bf16
        return np.array([fn(float(v)) for v in x.ravel()], np.uint16).reshape(x.shape)

    # -------------------------------------------------------- quantizers ---
    def quant_i8s(self, x, G=128):
        """INT8 symmetric group quantizer: (codes int8[n], scales f32[n/G])."""
        x = _c(x, np.float32).ravel()
        q = np.empty(x.size, np.int8)
        s = np.empty(x.size // G, np.float32)
        self.lib.or_quant_i8s(_p(x), x.size, G, _p(q), _p(s))
        return q, s

    def dequant_i8s(self, q, s, G=128):
        q = _c(q, np.int8).ravel()
        s = _c(s, np.float32)
        d = np.empty(q.size, np.float32)
        self.lib.or_dequant_i8s(_p(q), _p(s), q.size, G, _p(d))
        return d

    def quant_i4a(self, x, G=32):
        """INT4 asymmetric group quantizer: (packed u8[n/2], scales, zeros)."""
        x = _c(x, np.float32).ravel()
        q = np.empty(x.size // 2, np.uint8)
        s = np.empty(x.size // G, np.float32)
        z = np.empty(x.size // G, np.float32)
        self.lib.or_quant_i4a(_p(x), x.size, G, _p(q), _p(s), _p(z))
        return q, s, z

    def dequant_i4a(self, q, s, z, G=32):
        q = _c(q, np.uint8).ravel()
        s, z = _c(s, np.float32), _c(z, np.float32)
        d = np.empty(q.size * 2, np.float32)
        self.lib.or_dequant_i4a(_p(q), _p(s), _p(z), d.size, G, _p(d))
        return d

    def quantize(self, fmt, x, G):
        """(codes, scales, zeros-or-None) of fp32 values x."""
        if fmt == FMT_INT8_SYM:
            q, s = self.quant_i8s(x, G)
            return q, s, None
        if fmt == FMT_INT4_ASYM:
            return self.quant_i4a(x, G)
        raise ValueError(fmt)

    def dequantize(self, fmt, q, s, z, G):
        if fmt == FMT_INT8_SYM:
            return self.dequant_i8s(q, s, G)
        if fmt == FMT_INT4_ASYM:
            return self.dequant_i4a(q, s, z, G)
        raise ValueError(fmt)

    # ------------------------------------------------------------ reduce ---
    def reduce_sum(self, ds):
        """Fixed-order fp32 sum of equally sized fp32 arrays (list order)."""
        ds = [_c(d, np.float32).ravel() for d in ds]
        out = np.empty(ds[0].size, np.float32)
        self.lib.or_reduce_sum(_ptrs(ds), len(ds), out.size, _p(out))
        return out

    def two_step(self, fmt, slabs, G, shards=None):
        """Two-step reduce of quantized slabs [(codes, scales, zeros), ...].

        Returns dict(reduced, codes, scales, zeros, gathered)."""
        P = len(slabs)
        shards = P if shards is None else shards
        cdt = np.int8 if fmt == FMT_INT8_SYM else np.uint8
        codes = [_c(c, cdt).ravel() for c, _, _ in slabs]
        scales = [_c(s, np.float32) for _, s, _ in slabs]
        n = codes[0].size if fmt == FMT_INT8_SYM else codes[0].size * 2
        ng = n // G
        zeros = [(_c(z, np.float32) if z is not None else np.zeros(ng, np.float32))
                 for _, _, z in slabs]
        red = np.empty(n, np.float32)
        rq = np.empty(n if fmt == FMT_INT8_SYM else n // 2, cdt)
        rs = np.empty(ng, np.float32)
        rz = np.zeros(ng, np.float32)
        gath = np.empty(n, np.float32)
        rc = self.lib.or_two_step(fmt, _ptrs(codes), _ptrs(scales), _ptrs(zeros), P, n, G,
                                  shards, _p(red), _p(rq), _p(rs), _p(rz), _p(gath))
        if rc != 0:
            raise ValueError("or_two_step rejected its arguments")
        return dict(reduced=red, codes=rq, scales=rs,
                    zeros=rz if fmt == FMT_INT4_ASYM else None, gathered=gath)

    def allgather_dequant(self, fmt, shards, n, G):
        """Standalone all-gather: shards = [(codes, scales, zeros), ...], shard j
        holding groups [j*per, min((j+1)*per, n_g)) from its own index 0.
        Returns the n dequantized fp32 values of the whole tensor."""
        P = len(shards)
        cdt = np.int8 if fmt == FMT_INT8_SYM else np.uint8
        keep = []
        for c, s_, z in shards:
            keep.append((_c(c, cdt).ravel() if c is not None else np.zeros(1, cdt),
                         _c(s_, np.float32) if s_ is not None else np.zeros(1, np.float32),
                         _c(z, np.float32) if z is not None else np.zeros(1, np.float32)))
        out = np.empty(n, np.float32)
        rc = self.lib.or_allgather_dequant(fmt, _ptrs([k[0] for k in keep]), _ptrs([k[1] for k in keep]),
                                           _ptrs([k[2] for k in keep]), P, n, G, _p(out))
        if rc != 0:
            raise ValueError("or_allgather_dequant rejected its arguments")
        return out

    # ---------------------------------------------------- residual, norm ---
    def residual_rmsnorm(self, o, r_bf16, gamma_bf16, T, H, eps=1e-5):
        """(h_bf16, y_bf16) as uint16 arrays of shape [T, H]."""
        o = _c(o, np.float32).ravel()
        r = _c(r_bf16, np.uint16).ravel()
        g = _c(gamma_bf16, np.uint16).ravel()
        h = np.empty(T * H, np.uint16)
        y = np.empty(T * H, np.uint16)
        self.lib.or_residual_rmsnorm(_p(o), _p(r), _p(g), T, H, eps, _p(h), _p(y))
        return h.reshape(T, H), y.reshape(T, H)

    # ------------------------------------------------------------ tagged ---
    def tagged_blocks_per_row(self, H):
        return int(self.lib.or_tagged_blocks_per_row(H))

    def pack_tagged(self, x_bf16, T, H, epoch):
        """uint32 words [T * blocks_per_row * 4] of 16-byte tagged blocks."""
        x = _c(x_bf16, np.uint16).ravel()
        out = np.empty(T * self.tagged_blocks_per_row(H) * 4, np.uint32)
        self.lib.or_pack_tagged(_p(x), T, H, epoch, _p(out))
        return out

    def validate_tagged(self, blocks, epoch):
        """-1 when every block carries epoch, else the first bad block index."""
        b = _c(blocks, np.uint32).ravel()
        return int(self.lib.or_validate_tagged(_p(b), b.size // 4, epoch))

    def unpack_tagged(self, blocks, T, H):
        b = _c(blocks, np.uint32).ravel()
        x = np.empty(T * H, np.uint16)
        self.lib.or_unpack_tagged(_p(b), T, H, _p(x))
        return x.reshape(T, H)

    # ------------------------------------------- tagged quantized payloads ---
    def qtagged_blocks_per_group(self, fmt, G):
        return int(self.lib.or_qtagged_blocks_per_group(fmt, G))

    def pack_qtagged(self, fmt, q, s, z, G, epoch):
        """uint32 words of the self-synchronizing quantized payload blocks."""
        cdt = np.int8 if fmt == FMT_INT8_SYM else np.uint8
        q = _c(q, cdt).ravel()
        s = _c(s, np.float32)
        n = q.size if fmt == FMT_INT8_SYM else q.size * 2
        zz = _c(z, np.float32) if z is not None else np.zeros(s.size, np.float32)
        out = np.empty((n // G) * self.qtagged_blocks_per_group(fmt, G) * 4, np.uint32)
        self.lib.or_pack_qtagged(fmt, _p(q), _p(s), _p(zz), n, G, epoch, _p(out))
        return out

    def unpack_qtagged(self, fmt, blocks, n, G, epoch):
        """(codes, scales, zeros-or-None, first bad block or -1)."""
        b = _c(blocks, np.uint32).ravel()
        q = np.empty(n if fmt == FMT_INT8_SYM else n // 2, np.int8 if fmt == FMT_INT8_SYM else np.uint8)
        s = np.empty(n // G, np.float32)
        z = np.empty(n // G, np.float32)
        bad = self.lib.or_unpack_qtagged(fmt, _p(b), n, G, epoch, _p(q), _p(s), _p(z))
        return q, s, (z if fmt == FMT_INT4_ASYM else None), int(bad)

    # -------------------------------------------------------- whole path ---
    def allreduce_residual_rmsnorm(self, fmt, slabs_bf16, r_bf16, gamma_bf16, T, H, G=0,
                                   eps=1e-5, want_payload=True):
        """Whole path from bf16 slabs: dict(h, y[, codes, scales, zeros])."""
        slabs = [_c(s, np.uint16).ravel() for s in slabs_bf16]
        P = len(slabs)
        r = _c(r_bf16, np.uint16).ravel()
        g = _c(gamma_bf16, np.uint16).ravel()
        n = T * H
        h = np.empty(n, np.uint16)
        y = np.empty(n, np.uint16)
        rq = rs = rz = None
        if want_payload and fmt in (FMT_INT8_SYM, FMT_INT4_ASYM):
            rq = np.empty(n if fmt == FMT_INT8_SYM else n // 2,
                          np.int8 if fmt == FMT_INT8_SYM else np.uint8)
            rs = np.empty(n // G, np.float32)
            rz = np.zeros(n // G, np.float32)
        rc = self.lib.or_allreduce_residual_rmsnorm(fmt, _ptrs(slabs), P, T, H, G, _p(r), _p(g),
                                                    eps, _p(rq), _p(rs), _p(rz), _p(h), _p(y))
        if rc != 0:
            raise ValueError("or_allreduce_residual_rmsnorm rejected its arguments")
        out = dict(h=h.reshape(T, H), y=y.reshape(T, H))
        if rq is not None:
            out.update(codes=rq, scales=rs, zeros=rz if fmt == FMT_INT4_ASYM else None)
        return out


_default = None


def default() -> Oracle:
    """The oracle compiled from this directory's oracle.c."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def __getattr__(name):
    # module-level shortcuts: oracle.quant_i8s(...) == oracle.default().quant_i8s(...)
    if not name.startswith("_") and hasattr(Oracle, name):
        return getattr(default(), name)
    raise AttributeError(name)
