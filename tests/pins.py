"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a closed form, a hand-derived worked example under
``tests/golden/``, brute force in exact rational arithmetic, an invariant of
the method, or an independent library routine (torch's bf16 conversion and
RMSNorm).  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on deliberately broken copies and
requires each copy to fail at least one check.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import torch

FMT_INT8_SYM, FMT_INT4_ASYM = 1, 2
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (t.strip() for t in line.split("=", 1))
            vals[k] = [int(t, 0) if t.startswith(("0x", "-0x")) else float(t) for t in v.split()]
    return vals


# ----------------------------------------------------------- helpers ------
def _f32_neighbours(v):
    v = np.float32(v)
    return (np.nextafter(v, np.float32(-np.inf)), np.nextafter(v, np.float32(np.inf)))


def is_nearest_f32(v, exact: Fraction) -> bool:
    """v is a binary32 value nearest to the exact rational (ties: either)."""
    e = abs(Fraction(float(v)) - exact)
    return all(e <= abs(Fraction(float(w)) - exact) for w in _f32_neighbours(v))


def nearest_int_even(fr: Fraction) -> int:
    """Round an exact rational to the nearest integer, ties to even."""
    fl = math.floor(fr)
    rem = fr - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


def bf16_bits_to_float(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def torch_bf16_bits(x32):
    t = torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_ulp(v):
    """ulp of bf16 values v (float array): 2^(exponent - 7), normal range."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def nearest_bf16_exact(d: float) -> int:
    """bf16 bits nearest to the double d (ties to even), by exact rationals."""
    fr = Fraction(d)
    f = np.float32(d)  # a binary32 within one float ulp of d
    b = int(np.array([f], np.float32).view(np.uint32)[0] >> 16)
    cands = {(b + k) & 0xFFFF for k in (-2, -1, 0, 1, 2)}
    best = None
    for c in sorted(cands):
        val = Fraction(float(bf16_bits_to_float([c])[0]))
        err = abs(val - fr)
        key = (err, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


# ---------------------------------------------------------------- bf16 ----
def check_bf16_rne(orc):
    """fp32 -> bf16 equals torch's conversion (an independent library
    routine), including constructed ties in both directions."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 3 * 2 ** -9,
                     1 + 2 ** -8 + 2 ** -20, 0.0, -0.0], np.float32)
    x = np.concatenate([x, ties])
    assert np.array_equal(orc.f32_to_bf16(x), torch_bf16_bits(x))
    assert np.array_equal(orc.f32_to_bf16_array(x), torch_bf16_bits(x))
    assert list(orc.f32_to_bf16(ties[:2])) == [0x3F80, 0x3F82]


def check_f64_bf16_single_rounding(orc):
    """binary64 -> bf16 rounds once: values just off a bf16 midpoint by less
    than a binary32 ulp must round away from the midpoint."""
    mid = 1 + 2 ** -8
    vals = [mid, mid + 2 ** -40, mid - 2 ** -40, -(mid + 2 ** -40), 1 + 3 * 2 ** -8 - 2 ** -45]
    got = orc.f64_to_bf16(np.array(vals))
    assert list(got) == [0x3F80, 0x3F81, 0x3F80, 0xBF81, 0x3F81]
    rng = np.random.default_rng(12)
    rand = rng.standard_normal(3000) * np.exp(rng.uniform(-30, 30, 3000))
    got = orc.f64_to_bf16(rand)
    want = np.array([nearest_bf16_exact(float(d)) for d in rand], np.uint16)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- INT8 ----
def check_int8_golden(orc):
    g = load_golden("int8_sym_tiny.txt")
    G = int(g["G"][0])
    q, s = orc.quant_i8s(np.array(g["x"], np.float32), G)
    assert list(q) == [int(v) for v in g["q"]]
    assert list(s) == g["s"]
    assert list(orc.dequant_i8s(q, s, G)) == g["d"]


def _groups(rng, ng, G, outlier=True):
    x = rng.standard_normal((ng, G)).astype(np.float32)
    if outlier:
        x[:, rng.integers(0, G)] *= 50
    x *= np.exp(rng.uniform(-8, 8, (ng, 1))).astype(np.float32)
    return torch_bf16_bits(x).astype(np.uint16)


def check_int8_bound_and_extremes(orc):
    """|dequant(q(x)) - x| <= s/2 (plus fp32 rounding), |q| = 127 at the
    absmax element, codes within [-127, 127]."""
    rng = np.random.default_rng(13)
    G = 128
    xb = _groups(rng, 600, G)
    x = bf16_bits_to_float(xb).reshape(-1, G)
    q, s = orc.quant_i8s(x.ravel(), G)
    d = orc.dequant_i8s(q, s, G).reshape(-1, G).astype(np.float64)
    q = q.reshape(-1, G)
    slack = np.abs(x).max(1, keepdims=True).astype(np.float64) * 2.0 ** -21
    assert np.all(np.abs(d - x) <= s[:, None] / 2 + slack)
    am = np.abs(x).argmax(1)
    assert np.all(np.abs(q[np.arange(len(q)), am]) == 127)
    assert q.min() >= -127


def check_int8_exact_rational(orc):
    """Brute force in exact rationals: the scale is the binary32 nearest to
    absmax/127 and each code is the integer nearest to x/scale."""
    rng = np.random.default_rng(14)
    G = 16
    x = bf16_bits_to_float(_groups(rng, 40, G)).reshape(-1, G)
    q, s = orc.quant_i8s(x.ravel(), G)
    q = q.reshape(-1, G)
    for g in range(len(x)):
        a = max(abs(Fraction(float(v))) for v in x[g])
        assert is_nearest_f32(s[g], a / 127)
        for k in range(G):
            want = nearest_int_even(Fraction(float(x[g, k])) / Fraction(float(s[g])))
            assert q[g, k] == max(-127, min(127, want))


# ---------------------------------------------------------------- INT4 ----
def check_int4_golden(orc):
    g = load_golden("int4_asym_tiny.txt")
    G = int(g["G"][0])
    q, s, z = orc.quant_i4a(np.array(g["x"], np.float32), G)
    assert list(q) == [int(v) for v in g["packed"]]
    assert list(s) == g["s"] and list(z) == g["z"]
    assert list(orc.dequant_i4a(q, s, z, G)) == g["d"]


def unpack_nibbles(packed):
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.size * 2, np.int64)
    out[0::2] = p & 0xF
    out[1::2] = p >> 4
    return out


def check_int4_bound_and_extremes(orc):
    """|d - x| <= s/2 (plus fp32 rounding); code 0 at the minimum, 15 at the
    maximum; zero-point = group minimum; scale nearest to (hi-lo)/15."""
    rng = np.random.default_rng(15)
    G = 32
    x = bf16_bits_to_float(_groups(rng, 800, G)).reshape(-1, G)
    x[::7] += 3.0  # groups that are not centred on zero
    q, s, z = orc.quant_i4a(x.ravel(), G)
    c = unpack_nibbles(q).reshape(-1, G)
    d = orc.dequant_i4a(q, s, z, G).reshape(-1, G).astype(np.float64)
    mag = np.abs(x).max(1, keepdims=True).astype(np.float64)
    assert np.all(np.abs(d - x) <= s[:, None] / 2 + mag * 2.0 ** -20)
    rows = np.arange(len(x))
    assert np.all(c[rows, x.argmin(1)] == 0) and np.all(c[rows, x.argmax(1)] == 15)
    assert np.array_equal(z, x.min(1))
    for g in range(0, len(x), 37):
        dh = np.float32(x[g].max()) - np.float32(x[g].min())
        assert is_nearest_f32(dh, Fraction(float(x[g].max())) - Fraction(float(x[g].min())))
        assert is_nearest_f32(s[g], Fraction(float(dh)) / 15)
        for k in range(G):
            num = np.float32(x[g, k]) - np.float32(z[g])
            want = nearest_int_even(Fraction(float(num)) / Fraction(float(s[g])))
            assert c[g, k] == max(0, min(15, want))


def check_quant_degenerate(orc):
    """Constant groups dequantize exactly (INT4) and zero groups give scale 0
    and codes 0 (both formats); signed zeros give a +0 scale and zero-point."""
    x = np.array([2.5] * 32 + [0.0] * 32 + [-0.0] * 16 + [0.0] * 16 + [-3.0] * 32, np.float32)
    q, s, z = orc.quant_i4a(x, 32)
    assert np.array_equal(orc.dequant_i4a(q, s, z, 32), x + np.float32(0))
    assert list(s) == [0.0, 0.0, 0.0, 0.0]
    assert np.all(np.signbit(z) == [False, False, False, True])
    q8, s8 = orc.quant_i8s(np.zeros(256, np.float32), 128)
    assert not q8.any() and list(s8) == [0.0, 0.0]


# -------------------------------------------------------------- reduce ----
def check_reduce_integer_exact(orc):
    """Integer-valued slabs (|v| <= 2^10): every partial sum is exact in fp32,
    so the sum equals the int64 sum whatever the order."""
    rng = np.random.default_rng(16)
    for P in (2, 3, 8):
        iv = rng.integers(-1024, 1025, (P, 4099))
        got = orc.reduce_sum([v.astype(np.float32) for v in iv])
        assert np.array_equal(got.astype(np.int64), iv.sum(0))


def check_reduce_order_fixed(orc):
    """The sum runs over slabs 0..P-1 from +0: (1e8 + 1) - 1e8 = 0 in fp32
    while (1e8 - 1e8) + 1 = 1, and an all -0 column sums to +0."""
    a = np.array([1e8, 1e8, -0.0], np.float32)
    b = np.array([1.0, -1e8, -0.0], np.float32)
    c = np.array([-1e8, 1.0, -0.0], np.float32)
    got = orc.reduce_sum([a, b, c])
    assert got[0] == 0.0 and got[1] == 1.0
    assert got[2] == 0.0 and not np.signbit(got[2])


# ------------------------------------------------------------ two-step ----
def check_two_step_equals_direct(orc):
    """Requantizing each shard of the sum and gathering equals dequant-sum-
    requant of the unsharded tensor, bit for bit, for every partition; and
    the reduced sum equals the fixed-order sum of the dequantized slabs."""
    rng = np.random.default_rng(17)
    for fmt, G in ((FMT_INT8_SYM, 128), (FMT_INT4_ASYM, 32)):
        for P in (2, 3, 8):
            n = G * 37
            slabs = []
            for _ in range(P):
                x = bf16_bits_to_float(_groups(rng, 37, G))
                slabs.append(orc.quantize(fmt, x, G))
            direct = orc.two_step(fmt, slabs, G, shards=1)
            deq = [orc.dequantize(fmt, *sl, G) for sl in slabs]
            assert np.array_equal(direct["reduced"], orc.reduce_sum(deq))
            rq = orc.quantize(fmt, direct["reduced"], G)
            assert np.array_equal(direct["codes"], rq[0])
            assert np.array_equal(direct["gathered"], orc.dequantize(fmt, *rq, G))
            for shards in (2, 3, P, 7, 37):
                two = orc.two_step(fmt, slabs, G, shards=shards)
                for k in ("reduced", "codes", "scales", "gathered"):
                    assert np.array_equal(two[k].view(np.uint8), direct[k].view(np.uint8)), k
                if fmt == FMT_INT4_ASYM:
                    assert np.array_equal(two["zeros"].view(np.uint32),
                                          direct["zeros"].view(np.uint32))
            assert n == direct["reduced"].size


def check_allgather_golden(orc):
    g = load_golden("allgather_tiny.txt")
    for fmt, pre, cdt in ((FMT_INT8_SYM, "i8", np.int8), (FMT_INT4_ASYM, "i4", np.uint8)):
        G, P = int(g[pre + "_G"][0]), int(g[pre + "_P"][0])
        shards = []
        for j in range(P):
            c = np.array([int(v) for v in g[f"{pre}_shard{j}_codes"]], np.int64).astype(cdt)
            sc = np.array(g[f"{pre}_shard{j}_scales"], np.float32)
            z = np.array(g[f"{pre}_shard{j}_zeros"], np.float32) if fmt == FMT_INT4_ASYM else None
            shards.append((c, sc, z))
        want = np.array(g[pre + "_out"], np.float32)
        got = orc.allgather_dequant(fmt, shards, want.size, G)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def check_allgather_equals_dequant_of_slices(orc):
    """Gathering the shard slices of a payload dequantizes the whole payload,
    for every shard count (incl. more shards than groups, i.e. empty shards),
    and gathering the shards of the two-step reduce's requantized payload gives
    its gathered result."""
    rng = np.random.default_rng(29)
    for fmt, G in ((FMT_INT8_SYM, 128), (FMT_INT4_ASYM, 32), (FMT_INT4_ASYM, 16)):
        ng = 37
        x = bf16_bits_to_float(_groups(rng, ng, G))
        q, s, z = orc.quantize(fmt, x, G)
        cb = G if fmt == FMT_INT8_SYM else G // 2
        whole = orc.dequantize(fmt, q, s, z, G)
        for P in (1, 2, 3, 5, 8, 40):
            per = -(-ng // P)
            shards = []
            for j in range(P):
                g0, g1 = min(j * per, ng), min((j + 1) * per, ng)
                shards.append((q[g0 * cb:g1 * cb], s[g0:g1], None if z is None else z[g0:g1]))
            got = orc.allgather_dequant(fmt, shards, x.size, G)
            assert np.array_equal(got.view(np.uint32), whole.view(np.uint32)), (fmt, G, P)
        slabs = [orc.quantize(fmt, bf16_bits_to_float(_groups(rng, ng, G)), G) for _ in range(3)]
        two = orc.two_step(fmt, slabs, G, shards=3)
        per = -(-ng // 3)
        shards = [(two["codes"][j * per * cb:min((j + 1) * per, ng) * cb],
                   two["scales"][j * per:min((j + 1) * per, ng)],
                   None if two["zeros"] is None else two["zeros"][j * per:min((j + 1) * per, ng)])
                  for j in range(3)]
        got = orc.allgather_dequant(fmt, shards, x.size, G)
        assert np.array_equal(got.view(np.uint32), two["gathered"].view(np.uint32))


# ------------------------------------------------------ residual, norm ----
def check_residual_add(orc):
    """h = bf16(o + R) equals torch's fp32 add and bf16 conversion."""
    rng = np.random.default_rng(18)
    T, H = 3, 256
    o = (rng.standard_normal(T * H) * 4).astype(np.float32)
    r = torch_bf16_bits(rng.standard_normal(T * H).astype(np.float32))
    g = torch_bf16_bits(np.ones(H, np.float32))
    h, _ = orc.residual_rmsnorm(o, r, g, T, H)
    want = torch_bf16_bits(torch.from_numpy(o).add(torch.from_numpy(bf16_bits_to_float(r))).numpy())
    assert np.array_equal(h.ravel(), want)


def check_rmsnorm_constant_rows(orc):
    """Closed form: a row with every h_k = c gives y_k = c / sqrt(c^2 + eps) *
    gamma_k, rounded once to bf16."""
    H = 64
    rng = np.random.default_rng(19)
    gam = torch_bf16_bits((1 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    gf = bf16_bits_to_float(gam).astype(np.float64)
    for c in (1.0, -3.0, 0.0078125, 40.0):
        o = np.full(H, c, np.float32)
        r = np.zeros(H, np.uint16)
        for eps in (1e-5, 0.25):
            h, y = orc.residual_rmsnorm(o, r, gam, 1, H, eps=eps)
            assert np.all(bf16_bits_to_float(h) == np.float32(c))
            e = float(np.float32(eps))
            want = [nearest_bf16_exact(c / math.sqrt(c * c + e) * gk) for gk in gf]
            assert list(y.ravel()) == want
    o = np.zeros(H, np.float32)
    _, y = orc.residual_rmsnorm(o, np.zeros(H, np.uint16), gam, 1, H)
    assert not y.any()


def check_rmsnorm_vs_torch(orc):
    """Random rows: y agrees with torch.nn.functional.rms_norm in float64
    (an independent implementation) to one bf16 rounding."""
    rng = np.random.default_rng(20)
    T, H = 4, 1024
    o = (rng.standard_normal(T * H) * 3).astype(np.float32)
    r = torch_bf16_bits(rng.standard_normal(T * H).astype(np.float32))
    gam = torch_bf16_bits((1 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    h, y = orc.residual_rmsnorm(o, r, gam, T, H)
    hf = torch.from_numpy(bf16_bits_to_float(h).astype(np.float64)).reshape(T, H)
    gf = torch.from_numpy(bf16_bits_to_float(gam).astype(np.float64))
    ref = torch.nn.functional.rms_norm(hf, (H,), gf, eps=float(np.float32(1e-5))).numpy()
    yf = bf16_bits_to_float(y).astype(np.float64)
    assert np.all(np.abs(yf - ref) <= 0.5 * bf16_ulp(ref) * (1 + 1e-9))
    rms = np.sqrt((bf16_bits_to_float(y).astype(np.float64) / gf.numpy()) ** 2).mean()
    assert 0.7 < rms < 1.0  # mean |y/gamma| of a unit-RMS row of normals ~ sqrt(2/pi)


# -------------------------------------------------------------- tagged ----
def check_tagged_golden_and_roundtrip(orc):
    g = load_golden("tagged_tiny.txt")
    T, H, ep = int(g["T"][0]), int(g["H"][0]), int(g["epoch"][0])
    x = np.array(g["x"], np.uint16)
    w = orc.pack_tagged(x, T, H, ep)
    assert list(w) == [int(v) for v in g["words"]]
    assert np.array_equal(orc.unpack_tagged(w, T, H).ravel(), x)
    rng = np.random.default_rng(21)
    for T, H in ((3, 5120), (2, 6), (1, 1), (4, 13)):
        xb = rng.integers(0, 1 << 16, T * H).astype(np.uint16)
        w = orc.pack_tagged(xb, T, H, 77)
        assert w.size == T * ((H + 5) // 6) * 4
        assert np.array_equal(orc.unpack_tagged(w, T, H).ravel(), xb)
        assert orc.validate_tagged(w, 77) == -1


def check_tagged_stale(orc):
    rng = np.random.default_rng(22)
    T, H = 3, 100
    xb = rng.integers(0, 1 << 16, T * H).astype(np.uint16)
    w = orc.pack_tagged(xb, T, H, 9)
    nb = w.size // 4
    for bad in (0, 17, nb - 1):
        w2 = w.copy()
        w2[4 * bad + 3] = 8
        assert orc.validate_tagged(w2, 9) == bad
    w2 = w.copy()
    w2[4 * 40 + 3] = 1
    w2[4 * 20 + 3] = 1
    assert orc.validate_tagged(w2, 9) == 20
    assert orc.validate_tagged(w, 10) == 0


def check_qtagged_golden_roundtrip_and_stale(orc):
    g = load_golden("qtagged_int4_tiny.txt")
    G, ep = int(g["G"][0]), int(g["epoch"][0])
    q = np.array(g["codes"], np.uint8)
    w = orc.pack_qtagged(FMT_INT4_ASYM, q, np.array(g["scale"], np.float32),
                         np.array(g["zero"], np.float32), G, ep)
    assert list(w) == [int(v) for v in g["words"]]
    assert orc.qtagged_blocks_per_group(FMT_INT8_SYM, 128) == 11
    assert orc.qtagged_blocks_per_group(FMT_INT4_ASYM, 32) == 2
    rng = np.random.default_rng(24)
    for fmt, G in ((FMT_INT8_SYM, 128), (FMT_INT4_ASYM, 32), (FMT_INT8_SYM, 64)):
        x = bf16_bits_to_float(_groups(rng, 12, G))
        q, s, z = orc.quantize(fmt, x, G)
        w = orc.pack_qtagged(fmt, q, s, z, G, 77)
        q2, s2, z2, bad = orc.unpack_qtagged(fmt, w, x.size, G, 77)
        assert bad == -1 and np.array_equal(q2, q) and np.array_equal(s2, s)
        if z is not None:
            assert np.array_equal(z2, z)
        w2 = w.copy()
        nb = orc.qtagged_blocks_per_group(fmt, G)
        w2[4 * (3 * nb + 1) + 3] = 76
        assert orc.unpack_qtagged(fmt, w2, x.size, G, 77)[3] == 3 * nb + 1


# --------------------------------------------------------- whole path -----
def check_whole_path_composition(orc):
    """The whole path equals its pinned steps composed by hand."""
    rng = np.random.default_rng(23)
    T, H = 5, 256
    r = torch_bf16_bits(rng.standard_normal(T * H).astype(np.float32))
    gam = torch_bf16_bits((1 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    for fmt, G, P in ((FMT_INT8_SYM, 128, 3), (FMT_INT4_ASYM, 32, 4), (0, 0, 2)):
        slabs = [torch_bf16_bits(rng.standard_normal(T * H).astype(np.float32))
                 for _ in range(P)]
        got = orc.allreduce_residual_rmsnorm(fmt, slabs, r, gam, T, H, G)
        xs = [bf16_bits_to_float(s) for s in slabs]
        if fmt:
            two = orc.two_step(fmt, [orc.quantize(fmt, x, G) for x in xs], G, shards=P)
            o = two["gathered"]
            assert np.array_equal(got["codes"], two["codes"])
            assert np.array_equal(got["scales"], two["scales"])
        else:
            o = orc.reduce_sum(xs)
        h, y = orc.residual_rmsnorm(o, r, gam, T, H)
        assert np.array_equal(got["h"], h) and np.array_equal(got["y"], y)


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
