"""GPU parity: libfcomm (through its C ABI) against the CPU oracle, element by
element, on the same seeded inputs.

Bar: codes, scales, zero-points, fp32 sums and residual_out bit-exact; y
(RMSNorm output, bf16) within one bf16 ulp of the oracle, the ulp of the
oracle's value's binade (gpu_util.bf16_ulp).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import quantized_reduce_rmsnorm_gb300 as fc
from quantized_reduce_rmsnorm_gb300 import synth
from gpu_util import (assert_bits_equal, assert_y_close, bf16_float, dev, dev_bf16, host,
                      host_bits)

pytestmark = pytest.mark.gpu

I8, I4, BF, TG = synth.FMT_INT8_SYM, synth.FMT_INT4_ASYM, synth.FMT_BF16, synth.FMT_BF16_TAGGED
I8T, I4T = synth.FMT_INT8_TAGGED, synth.FMT_INT4_TAGGED


def spec_of(fmt, G):
    return fc.QSpec(fmt, G)


def small(name, **kw):
    """A workload of the given shape family (sizes the oracle finishes quickly)."""
    base = synth.WORKLOADS.get(name)
    if base is None:
        base = synth.Workload(name, P=2, T=1, H=4096, fmt=I8, group=128)
    return synth.Workload(**{**base.__dict__, "name": name, **kw})


def quantize_on_gpu(w, inp):
    spec = spec_of(w.fmt, w.group)
    xs = [dev_bf16(s) for s in inp["slabs"]]
    outs = [fc.alloc_qtensor(spec, w.T, w.H) for _ in range(w.P)]
    fc.group_quantize_multi(xs, spec, outs)
    return outs


def oracle_quant(orc, w, slab_bits):
    return orc.quantize(w.fmt, bf16_float(slab_bits).ravel(), w.group)


# ------------------------------------------------------------- quantize ---
QUANT_CASES = [
    ("decode-tiny", {}),
    ("decode", {}),
    ("prefill", {"T": 48}),
    ("i8-g32-ragged", {"P": 3, "T": 7, "H": 1184, "fmt": I8, "group": 32}),
    ("i4-g64", {"P": 2, "T": 5, "H": 4160, "fmt": I4, "group": 64, "outlier_frac": 0.01,
                "outlier_scale": 100.0}),
    ("i8-g512", {"P": 2, "T": 3, "H": 2048, "fmt": I8, "group": 512}),
    ("i4-g16", {"P": 2, "T": 3, "H": 1040, "fmt": I4, "group": 16}),
]


@pytest.mark.parametrize("name,kw", QUANT_CASES, ids=[c[0] for c in QUANT_CASES])
def test_group_quantize_bit_exact(orc, name, kw):
    w = small(name, **kw)
    inp = synth.make_inputs(w, seed=1)
    outs = quantize_on_gpu(w, inp)
    torch.cuda.synchronize()
    for p in range(w.P):
        q, s, z = oracle_quant(orc, w, inp["slabs"][p])
        assert_bits_equal(host(outs[p][0]), q, f"codes slab {p}")
        assert_bits_equal(host(outs[p][1]), s, f"scales slab {p}")
        if w.fmt == I4:
            assert_bits_equal(host(outs[p][2]), z, f"zeros slab {p}")


def test_group_quantize_single_matches_multi():
    w = small("decode", T=8)
    inp = synth.make_inputs(w, seed=2)
    spec = spec_of(w.fmt, w.group)
    multi = quantize_on_gpu(w, inp)
    for p in range(w.P):
        one = fc.alloc_qtensor(spec, w.T, w.H)
        fc.group_quantize(dev_bf16(inp["slabs"][p]), spec, one)
        torch.cuda.synchronize()
        assert torch.equal(one[0], multi[p][0]) and torch.equal(one[1], multi[p][1])


@pytest.mark.parametrize("fmt,G", [(I8, 128), (I4, 32)])
def test_quantize_degenerate_groups(orc, fmt, G):
    """All-zero groups, constant groups, signed zeros, one huge outlier, ties,
    and groups whose scale is below 2^-100 or subnormal (every element of
    those takes the division)."""
    H = 512
    x = np.zeros((6, H), np.float32)
    x[1, :] = 2.5                                  # constant row
    x[2, :G] = -0.0
    x[2, G:2 * G:2] = -0.0
    x[2, G + 1:2 * G:2] = 0.0                      # mixed signed zeros
    x[2, 2 * G:] = np.arange(H - 2 * G) * 0.5      # exact ties after scaling
    x[3, :] = np.linspace(-3, 3, H)
    x[3, 7] = 3.0e30                               # one huge outlier
    x[4, :] = np.linspace(-1, 1, H) * 1e-33        # scales below 2^-100
    x[5, :] = np.linspace(-1, 1, H) * 3e-39        # bf16 subnormals
    x[5, ::3] = np.float32(2.0 ** -126) * 1.5
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    spec = spec_of(fmt, G)
    out = fc.alloc_qtensor(spec, 6, H)
    fc.group_quantize(dev_bf16(bits), spec, out)
    torch.cuda.synchronize()
    q, s, z = orc.quantize(fmt, bf16_float(bits).ravel(), G)
    assert_bits_equal(host(out[0]), q, "codes")
    assert_bits_equal(host(out[1]), s, "scales")
    if fmt == I4:
        assert_bits_equal(host(out[2]), z, "zeros")


# --------------------------------------------------------------- reduce ---
REDUCE_CASES = [(I8, 128, 2), (I8, 128, 3), (I8, 128, 8), (I4, 32, 2), (I4, 32, 4),
                (I4, 32, 8), (I8, 64, 5)]


@pytest.mark.parametrize("fmt,G,P", REDUCE_CASES)
def test_reduce_dequant_sum_bit_exact(orc, fmt, G, P):
    w = synth.Workload("reduce", P=P, T=9, H=2048, fmt=fmt, group=G, outlier_frac=0.01,
                       outlier_scale=30.0)
    inp = synth.make_inputs(w, seed=3)
    outs = quantize_on_gpu(w, inp)
    red = torch.empty(w.T, w.H, dtype=torch.float32, device="cuda")
    fc.reduce_dequant_sum(outs, spec_of(fmt, G), w.T, w.H, red)
    torch.cuda.synchronize()
    slabs = [oracle_quant(orc, w, s) for s in inp["slabs"]]
    want = orc.two_step(fmt, slabs, G)
    assert_bits_equal(host(red), want["reduced"], "reduced fp32")


@pytest.mark.parametrize("fmt,G", [(I4, 32), (I8, 128)])
def test_reduce_huge_scales(orc, fmt, G):
    """Groups whose scale exceeds 2^100 (outliers near 1e34) take the plain
    dequantization product; the rest the fused one.  Both bit-exact."""
    w = synth.Workload("huge", P=3, T=4, H=1024, fmt=fmt, group=G, outlier_frac=0.05,
                       outlier_scale=1.0e34)
    inp = synth.make_inputs(w, seed=23)
    outs = quantize_on_gpu(w, inp)
    red = torch.empty(w.T, w.H, device="cuda")
    fc.reduce_dequant_sum(outs, spec_of(fmt, G), w.T, w.H, red)
    torch.cuda.synchronize()
    slabs = [oracle_quant(orc, w, s) for s in inp["slabs"]]
    assert max(float(np.max(sl[1])) for sl in slabs) > 2.0 ** 100
    assert_bits_equal(host(red), orc.two_step(fmt, slabs, G)["reduced"], "reduced fp32")


@pytest.mark.parametrize("fmt,G,P", [(I8, 128, 3), (I4, 32, 8)])
def test_reduce_shards_write_only_their_range(orc, fmt, G, P):
    w = synth.Workload("shards", P=P, T=5, H=1024, fmt=fmt, group=G)
    inp = synth.make_inputs(w, seed=4)
    outs = quantize_on_gpu(w, inp)
    spec = spec_of(fmt, G)
    slabs = [oracle_quant(orc, w, s) for s in inp["slabs"]]
    want = orc.two_step(fmt, slabs, G)["reduced"]
    full = torch.full((w.T, w.H), float("nan"), device="cuda")
    for j in range(P):
        part = torch.full((w.T, w.H), float("nan"), device="cuda")
        fc.reduce_dequant_sum(outs, spec, w.T, w.H, part, shard=j)
        fc.reduce_dequant_sum(outs, spec, w.T, w.H, full, shard=j)
        g0, g1 = fc.shard_range(spec, w.T, w.H, P, j)
        torch.cuda.synchronize()
        got = host(part).ravel()
        assert np.all(np.isnan(got[:g0 * G])) and np.all(np.isnan(got[g1 * G:]))
        assert_bits_equal(got[g0 * G:g1 * G], want[g0 * G:g1 * G], f"shard {j}")
    assert_bits_equal(host(full), want, "all shards")


# ---------------------------------------------------------- requant/gather --
@pytest.mark.parametrize("fmt,G", [(I8, 128), (I4, 32), (I8, 32), (I4, 128)])
@pytest.mark.parametrize("out_dtype", [fc.FMT_BF16, fc.FMT_F32])
def test_requant_gather_bit_exact(orc, fmt, G, out_dtype):
    rng = np.random.default_rng(5)
    T, H = 6, 2048
    red = (rng.standard_normal((T, H)) * np.exp(rng.uniform(-5, 5, (T, 1)))).astype(np.float32)
    red[2, :G] = 0.0
    red[3, G:2 * G] = 1.25
    spec = spec_of(fmt, G)
    rq = fc.alloc_qtensor(spec, T, H)
    out = torch.empty(T, H, dtype=torch.bfloat16 if out_dtype == fc.FMT_BF16 else torch.float32,
                      device="cuda")
    fc.requant_gather(dev(red), spec, rq, out, out_dtype)
    torch.cuda.synchronize()
    q, s, z = orc.quantize(fmt, red.ravel(), G)
    d = orc.dequantize(fmt, q, s, z, G)
    assert_bits_equal(host(rq[0]), q, "codes")
    assert_bits_equal(host(rq[1]), s, "scales")
    if fmt == I4:
        assert_bits_equal(host(rq[2]), z, "zeros")
    if out_dtype == fc.FMT_F32:
        assert_bits_equal(host(out), d, "gathered fp32")
    else:
        assert_bits_equal(host_bits(out), orc.f32_to_bf16_array(d), "gathered bf16")


def _near_ties(fmt, G, rng):
    """fp32 groups whose quotients x/s sit exactly on, or a few ulps around,
    half-integers: the cases where rounding x*(1/s) could disagree with
    rounding fl(x/s), so the kernels must take their exact division path."""
    groups = []
    for s0 in (3.0, 0.5, float(np.float32(1.0) / np.float32(127.0)), 1.0e-3, 7.0e4):
        s0 = np.float32(s0)
        if fmt == I8:
            k = rng.integers(-127, 127, G).astype(np.float32)
            x = ((k + np.float32(0.5)) * s0).astype(np.float32)
            x[0] = np.float32(127) * s0          # absmax fixes s = fl(127 s0 / 127)
        else:
            k = rng.integers(0, 15, G).astype(np.float32)
            x = ((k + np.float32(0.5)) * s0).astype(np.float32)
            x[0], x[1] = np.float32(0), np.float32(15) * s0   # lo = 0, hi = 15 s0
        nud = rng.integers(-3, 4, G)
        for i in range(2, G):
            for _ in range(abs(nud[i])):
                x[i] = np.nextafter(x[i], np.float32(np.inf) if nud[i] > 0 else np.float32(-np.inf))
        groups.append(x)
    return np.concatenate(groups)


@pytest.mark.parametrize("fmt,G", [(I8, 128), (I4, 32), (I8, 16), (I4, 64)])
def test_quantizer_near_half_integer_quotients(orc, fmt, G):
    rng = np.random.default_rng(21)
    red = np.concatenate([_near_ties(fmt, G, rng) for _ in range(8)])
    T = red.size // (4 * G)
    red = red[:T * 4 * G].reshape(T, 4 * G)
    spec = spec_of(fmt, G)
    rq = fc.alloc_qtensor(spec, T, 4 * G)
    out = torch.empty(T, 4 * G, dtype=torch.float32, device="cuda")
    fc.requant_gather(dev(red), spec, rq, out, fc.FMT_F32)
    torch.cuda.synchronize()
    q, s, z = orc.quantize(fmt, red.ravel(), G)
    assert_bits_equal(host(rq[0]), q, "codes")
    assert_bits_equal(host(rq[1]), s, "scales")
    assert_bits_equal(host(out), orc.dequantize(fmt, q, s, z, G), "dequantized")


@pytest.mark.parametrize("fmt,G,P", [(I8, 128, 8), (I4, 32, 4), (I4, 32, 3)])
def test_two_step_chain_equals_oracle(orc, fmt, G, P):
    """quantize -> reduce-scatter math per shard -> requant -> gather on the
    GPU equals the oracle's two-step result (which equals the direct one)."""
    w = synth.Workload("chain", P=P, T=16, H=4096, fmt=fmt, group=G, dist="student_t3")
    inp = synth.make_inputs(w, seed=6)
    spec = spec_of(fmt, G)
    outs = quantize_on_gpu(w, inp)
    red = torch.empty(w.T, w.H, device="cuda")
    for j in range(P):
        fc.reduce_dequant_sum(outs, spec, w.T, w.H, red, shard=j)
    rq = fc.alloc_qtensor(spec, w.T, w.H)
    gath = torch.empty(w.T, w.H, device="cuda")
    fc.requant_gather(red, spec, rq, gath, fc.FMT_F32)
    torch.cuda.synchronize()
    want = orc.two_step(fmt, [oracle_quant(orc, w, s) for s in inp["slabs"]], G, shards=P)
    assert_bits_equal(host(rq[0]), want["codes"], "payload codes")
    assert_bits_equal(host(rq[1]), want["scales"], "payload scales")
    assert_bits_equal(host(gath), want["gathered"], "gathered")


# ------------------------------------------------------------------ fused --
def run_fused(w, inp, seed_payload=True, max_ctas=0, alias=False, epoch=7, kernel=0):
    """Quantize (or pack) the slabs on the GPU, run the fused call; returns host arrays."""
    spec = spec_of(w.fmt, w.group)
    if w.fmt in (I8, I4):
        slabs = quantize_on_gpu(w, inp)
    elif w.fmt == BF:
        slabs = [dev_bf16(s) for s in inp["slabs"]]
    else:
        slabs = []
        for s in inp["slabs"]:
            blk = torch.empty(fc.tagged_bytes(w.T, w.H), dtype=torch.uint8, device="cuda")
            fc.pack_tagged(dev_bf16(s), epoch, blk)
            slabs.append(blk)
    r_in = dev_bf16(inp["residual"])
    r_out = r_in if alias else torch.empty_like(r_in)
    gam = dev_bf16(inp["gamma"])
    y = torch.empty_like(r_in)
    rq = fc.alloc_qtensor(spec, w.T, w.H) if (w.fmt in (I8, I4) and seed_payload) else None
    st = torch.zeros(2, dtype=torch.int32, device="cuda") if w.fmt == TG else None
    fc.allreduce_residual_rmsnorm(slabs, spec, w.T, w.H, r_in, r_out, gam, w.eps, y,
                                  requant_out=rq, expected_epoch=epoch, d_status=st,
                                  max_ctas=max_ctas, kernel=kernel)
    torch.cuda.synchronize()
    res = dict(h=host_bits(r_out), y=host_bits(y))
    if rq is not None:
        res.update(codes=host(rq[0]), scales=host(rq[1]),
                   zeros=host(rq[2]) if rq[2] is not None else None)
    if st is not None:
        res["status"] = host(st)
    return res


def oracle_fused(orc, w, inp):
    fmt = BF if w.fmt == TG else synth.base_format(w.fmt)
    return orc.allreduce_residual_rmsnorm(fmt, inp["slabs"], inp["residual"], inp["gamma"],
                                          w.T, w.H, w.group, w.eps)


def check_fused(orc, w, got, want):
    assert_bits_equal(got["h"], want["h"], "residual_out")
    exact = assert_y_close(got["y"], want["y"])
    assert exact > 0.99, f"only {exact:.4f} of y bit-exact"
    if "codes" in got:
        assert_bits_equal(got["codes"], want["codes"], "payload codes")
        assert_bits_equal(got["scales"], want["scales"], "payload scales")
        if w.fmt == I4:
            assert_bits_equal(got["zeros"], want["zeros"], "payload zeros")


FUSED_CASES = [
    ("decode-tiny", {}),
    ("decode", {}),
    ("prefill", {"T": 24}),
    ("token-split", {"T": 40}),
    ("bf16-p3", {"P": 3, "T": 5, "H": 4096, "fmt": BF, "group": 0}),
    ("i8-ragged-h", {"P": 3, "T": 11, "H": 1152, "fmt": I8, "group": 128}),
    ("i4-ragged-h", {"P": 5, "T": 9, "H": 4128, "fmt": I4, "group": 32}),
    ("i4-wide-h", {"P": 2, "T": 3, "H": 16384, "fmt": I4, "group": 32}),
    ("i8-wide-h", {"P": 2, "T": 2, "H": 32768, "fmt": I8, "group": 128}),
    ("tagged-ragged-h", {"P": 2, "T": 6, "H": 1040, "fmt": TG, "group": 0}),
    ("tagged-h16", {"P": 4, "T": 3, "H": 16, "fmt": TG, "group": 0}),
    ("i8-h16", {"P": 2, "T": 5, "H": 16, "fmt": I8, "group": 16}),
]


@pytest.mark.parametrize("fmt,G", [(I4, 32), (I8, 128)])
@pytest.mark.parametrize("P", [2, 4, 8])
@pytest.mark.parametrize("kernel", [fc.KERNEL_STREAM, fc.KERNEL_AUTO], ids=["stream", "auto"])
def test_fused_tiny_sums(orc, fmt, G, P, kernel):
    """Slabs near 1e-33 (and their sums): every requantization scale is below
    2^-100, so every element of the payload takes the division, in each
    build's exact pass (two, four and eight slabs)."""
    w = synth.Workload("tiny", P=P, T=6, H=8192, fmt=fmt, group=G, outlier_frac=1.0,
                       outlier_scale=1.0e-33)
    inp = synth.make_inputs(w, seed=29)
    want = oracle_fused(orc, w, inp)
    assert float(np.max(want["scales"])) < 2.0 ** -100
    check_fused(orc, w, run_fused(w, inp, kernel=kernel), want)


@pytest.mark.parametrize("kernel", [fc.KERNEL_STREAM, fc.KERNEL_AUTO], ids=["stream", "auto"])
@pytest.mark.parametrize("name,kw", FUSED_CASES, ids=[c[0] for c in FUSED_CASES])
def test_fused_matches_oracle(orc, name, kw, kernel):
    w = small(name, **kw)
    inp = synth.make_inputs(w, seed=8)
    got = run_fused(w, inp, kernel=kernel)
    check_fused(orc, w, got, oracle_fused(orc, w, inp))
    if w.fmt == TG:
        assert list(got["status"]) == [fc.FC_OK, fc.STATUS_NO_INDEX]


TMA_CASES = [
    ("prefill", {"T": 40}),
    ("decode", {"T": 16}),
    ("decode-tiny", {}),
    ("bf16-p8", {"P": 8, "T": 9, "H": 5120, "fmt": BF, "group": 0}),
    ("i4-ragged-h", {"P": 3, "T": 13, "H": 4224, "fmt": I4, "group": 32}),  # 132 groups/row
    ("i8-cpr-not-warp-multiple", {"P": 2, "T": 7, "H": 1152, "fmt": I8, "group": 32}),
    ("i4-wide-h", {"P": 2, "T": 5, "H": 16384, "fmt": I4, "group": 32}),
    # short rows, many per CTA at max_ctas 1 and 3
    ("i4-short-rows", {"P": 2, "T": 37, "H": 4096, "fmt": I4, "group": 32}),
    ("i8-short-rows", {"P": 2, "T": 29, "H": 2048, "fmt": I8, "group": 128}),
    # single-stage rings of the compact build (shared memory admits 3 CTAs per SM)
    ("i8-p4-wide", {"P": 4, "T": 9, "H": 8192, "fmt": I8, "group": 128}),
    # eight INT4 slabs at H = 8192: the build without the h buffer (capped grids)
    ("i4-p8-h8192", {"P": 8, "T": 9, "H": 8192, "fmt": I4, "group": 32}),
]


@pytest.mark.parametrize("name,kw", TMA_CASES, ids=[c[0] for c in TMA_CASES])
def test_fused_tma_kernel_matches_oracle(orc, name, kw):
    """The TMA-staged kernel, forced, on shapes it supports (incl. rows whose
    chunk count is not a multiple of the warp size, and 1- and 2-stage rings)."""
    w = small(name, **kw)
    inp = synth.make_inputs(w, seed=18)
    want = oracle_fused(orc, w, inp)
    check_fused(orc, w, run_fused(w, inp, kernel=fc.KERNEL_TMA), want)
    for cap in (1, 3):
        check_fused(orc, w, run_fused(w, inp, kernel=fc.KERNEL_TMA, max_ctas=cap), want)


def test_fused_tma_kernel_rejects_unsupported_shape():
    w = small("i8-h16", P=2, T=5, H=16, fmt=I8, group=16)   # 4-byte scale rows
    inp = synth.make_inputs(w, seed=19)
    with pytest.raises(fc.FcommError) as e:
        run_fused(w, inp, kernel=fc.KERNEL_TMA)
    assert e.value.status == fc.FC_ERR_UNSUPPORTED


def test_fused_in_place_residual_and_capped_grid(orc):
    w = small("prefill", T=20)
    inp = synth.make_inputs(w, seed=9)
    want = oracle_fused(orc, w, inp)
    for kernel in (fc.KERNEL_STREAM, fc.KERNEL_TMA):
        check_fused(orc, w, run_fused(w, inp, alias=True, kernel=kernel), want)
        for cap in (1, 2, 8):
            check_fused(orc, w, run_fused(w, inp, max_ctas=cap, kernel=kernel), want)


RG_PLAIN = [(I4, 32, 8, 320, 8192), (I4, 32, 8, 800, 4096), (I8, 128, 2, 7300, 4096), (I8, 128, 8, 320, 8192),
            (I8, 128, 8, 480, 4096), (I4, 32, 2, 7300, 8192), (I4, 32, 4, 7300, 8192), (I8, 128, 4, 7300, 8192),
            (I8, 128, 2, 7300, 8192),
            # slab counts between the built ones take the build for the next one up
            (I4, 32, 6, 800, 4096), (I8, 128, 5, 480, 4096), (I4, 32, 3, 7300, 8192), (I8, 128, 7, 320, 8192)]


@pytest.mark.parametrize("fmt,G,P,T,H", RG_PLAIN,
                         ids=[f"{synth.FMT_NAMES[f]}-p{p}-h{h}" for f, _, p, _, h in RG_PLAIN])
def test_fused_in_place_residual_free_stage(orc, fmt, G, P, T, H):
    """Shapes with more rows than one wave of the staged build whose stage
    leaves the residual out (each thread loads its residual chunk from global
    memory): eight INT4 slabs at H = 8192 (half-row sub-stages) and at
    H = 4096 (one-row stage), two INT8 slabs at H = 4096 (a two-row ring,
    taken from eight waves of rows), eight INT8 slabs at H = 8192 (half-row
    sub-stages without the h row buffer: pass 2 reads h back from
    residual_out) and at H = 4096 (one-row stage without the h row buffer,
    128-thread CTAs), and the 128-thread CTAs without the h row buffer for
    rows of 8192 in calls of eight waves or more (two INT4 or INT8 slabs:
    two-row rings; four: one-row stages).  residual_out aliasing the
    residual, and capped grids,
    still give the oracle's bits."""
    w = synth.Workload("rg-rows", P=P, T=T, H=H, fmt=fmt, group=G)
    inp = synth.make_inputs(w, seed=31)
    want = oracle_fused(orc, w, inp)
    check_fused(orc, w, run_fused(w, inp, alias=True), want)
    check_fused(orc, w, run_fused(w, inp), want)
    for cap in (3, 200):
        check_fused(orc, w, run_fused(w, inp, max_ctas=cap), want)


def test_fused_without_payload(orc):
    w = small("decode", T=4)
    inp = synth.make_inputs(w, seed=10)
    got = run_fused(w, inp, seed_payload=False)
    want = oracle_fused(orc, w, inp)
    assert_bits_equal(got["h"], want["h"], "residual_out")
    assert_y_close(got["y"], want["y"])


def test_fused_degenerate_rows(orc):
    """All-zero slabs and residual (y = 0), constant rows, zero gamma."""
    w = synth.Workload("degenerate", P=2, T=3, H=1024, fmt=I8, group=128)
    inp = synth.make_inputs(w, seed=11)
    inp["slabs"] = [s.copy() for s in inp["slabs"]]
    for s in inp["slabs"]:
        s[0] = 0
        s[1] = 0x3FC0  # 1.5
    inp["residual"] = inp["residual"].copy()
    inp["residual"][0] = 0
    inp["residual"][1] = 0
    inp["gamma"] = inp["gamma"].copy()
    inp["gamma"][:8] = 0
    got = run_fused(w, inp)
    want = oracle_fused(orc, w, inp)
    check_fused(orc, w, got, want)
    assert not got["y"][0].any()


def test_tagged_pack_bit_exact(orc):
    for T, H in ((3, 5120), (4, 1040), (2, 16), (5, 4096)):
        rng = np.random.default_rng(T * H)
        x = rng.integers(0, 1 << 16, (T, H)).astype(np.uint16)
        blk = torch.empty(fc.tagged_bytes(T, H), dtype=torch.uint8, device="cuda")
        fc.pack_tagged(dev_bf16(x), 0xABCD1234, blk)
        torch.cuda.synchronize()
        assert_bits_equal(host(blk).view(np.uint32), orc.pack_tagged(x, T, H, 0xABCD1234),
                          f"tagged blocks {T}x{H}")


def test_tagged_pack_multi_equals_oracle(orc):
    T, H, P = 7, 1040, 3
    rng = np.random.default_rng(77)
    xs = [rng.integers(0, 1 << 16, (T, H)).astype(np.uint16) for _ in range(P)]
    blks = [torch.empty(fc.tagged_bytes(T, H), dtype=torch.uint8, device="cuda") for _ in range(P)]
    fc.pack_tagged_multi([dev_bf16(x) for x in xs], 12345, blks)
    torch.cuda.synchronize()
    for p in range(P):
        assert_bits_equal(host(blks[p]).view(np.uint32), orc.pack_tagged(xs[p], T, H, 12345),
                          f"slab {p}")


def test_tagged_stale_block_is_reported(orc):
    """Blocks built on the host by the oracle; one or two tags corrupted
    before upload: the call reports FC_ERR_STALE_BLOCK and the first index,
    and never hangs.  Clean blocks give FC_OK and oracle-equal outputs."""
    w = synth.Workload("stale", P=4, T=6, H=1000 // 16 * 16, fmt=TG, group=0)
    inp = synth.make_inputs(w, seed=12)
    ep = 41
    blocks = [orc.pack_tagged(s, w.T, w.H, ep) for s in inp["slabs"]]
    nb = orc.tagged_blocks_per_row(w.H)
    spec = spec_of(TG, 0)
    r_in, gam = dev_bf16(inp["residual"]), dev_bf16(inp["gamma"])
    r_out, y = torch.empty_like(r_in), torch.empty_like(r_in)
    st = torch.full((2,), -5, dtype=torch.int32, device="cuda")

    def call(bl, epoch=ep):
        fc.allreduce_residual_rmsnorm([dev(b.view(np.int32)) for b in bl], spec, w.T, w.H, r_in, r_out, gam,
                                      w.eps, y, expected_epoch=epoch, d_status=st)
        torch.cuda.synchronize()
        return list(host(st))

    assert call(blocks) == [fc.FC_OK, fc.STATUS_NO_INDEX]
    want = oracle_fused(orc, w, inp)
    assert_bits_equal(host_bits(r_out), want["h"], "residual_out")
    assert_y_close(host_bits(y), want["y"])

    bad = [b.copy() for b in blocks]
    bad[2][4 * (3 * nb + 17) + 3] = ep - 1          # slab 2, row 3, block 17
    bad[3][4 * 5 + 3] = ep + 1                      # slab 3, row 0, block 5
    first = (2 * w.T + 3) * nb + 17
    assert call(bad) == [fc.FC_ERR_STALE_BLOCK, first]
    bad[1][4 * (5 * nb + nb - 1) + 3] = 0           # slab 1, last block of the last row
    assert call(bad) == [fc.FC_ERR_STALE_BLOCK, (1 * w.T + 5) * nb + nb - 1]
    assert call(blocks, epoch=ep + 1) == [fc.FC_ERR_STALE_BLOCK, 0]
    assert call(blocks) == [fc.FC_OK, fc.STATUS_NO_INDEX]


def test_token_split_two_streams_equals_one_call(orc):
    """Two subsets of rows on two streams give the same bits as one call."""
    w = small("token-split", T=64)
    inp = synth.make_inputs(w, seed=13)
    spec = spec_of(TG, 0)
    blocks = []
    for s in inp["slabs"]:
        b = torch.empty(fc.tagged_bytes(w.T, w.H), dtype=torch.uint8, device="cuda")
        fc.pack_tagged(dev_bf16(s), 3, b)
        blocks.append(b)
    r_in, gam = dev_bf16(inp["residual"]), dev_bf16(inp["gamma"])
    r_out, y = torch.empty_like(r_in), torch.empty_like(r_in)
    half = w.T // 2
    bpr = fc.tagged_bytes(1, w.H)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    st = torch.zeros(2, 2, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    for i, s in enumerate(streams):
        r0, r1 = i * half, (i + 1) * half
        fc.allreduce_residual_rmsnorm([b[r0 * bpr:r1 * bpr] for b in blocks], spec, half, w.H,
                                      r_in[r0:r1], r_out[r0:r1], gam, w.eps, y[r0:r1],
                                      expected_epoch=3, d_status=st[i], stream=s)
    torch.cuda.synchronize()
    assert host(st).tolist() == [[0, fc.STATUS_NO_INDEX]] * 2
    want = oracle_fused(orc, w, inp)
    assert_bits_equal(host_bits(r_out), want["h"], "residual_out")
    assert_y_close(host_bits(y), want["y"])


def test_wave_aware_token_split(orc):
    """The split is whole waves of the fused kernel (nearest the middle), and
    the two-stream step with it gives the same bits as with an even split."""
    from quantized_reduce_rmsnorm_gb300.pipeline import Pipeline
    for spec, P, T, H in ((fc.BF16_TAGGED, 8, 4096, 5120), (fc.INT4_G32, 4, 3000, 8192),
                          (fc.INT8_G128, 8, 64, 8192), (fc.BF16, 2, 10000, 4096)):
        split, wave = fc.token_split(spec, P, T, H)
        assert wave > 0 and 0 < split < T
        if T > wave:
            assert split % wave == 0
            assert abs(split - T / 2) <= wave / 2 + 1
        else:
            assert split == T // 2
    w = small("token-split", T=600)
    inp = synth.make_inputs(w, seed=31)
    outs = []
    for mode in ("even", "wave"):
        pipe = Pipeline(w, inp, split=mode)
        pipe.step()
        outs.append(pipe.outputs())
    assert np.array_equal(outs[0]["h"], outs[1]["h"]) and np.array_equal(outs[0]["y"], outs[1]["y"])
    want = oracle_fused(orc, w, inp)
    assert_bits_equal(outs[1]["h"], want["h"], "residual_out")


@pytest.mark.parametrize("fmt,G,P,H", [(I8, 128, 8, 8192), (I4, 32, 4, 8192), (I4, 32, 3, 4096)])
@pytest.mark.parametrize("mode", ["even", "wave"])
def test_quantized_token_split_every_element(orc, fmt, G, P, H, mode):
    """Two token subsets of a quantized workload, each a fused call on its own
    stream over its rows' codes, scales and zero-points: every element
    against the oracle, at the even and the wave-aware boundary (a row count
    past one wave, so the two differ)."""
    from quantized_reduce_rmsnorm_gb300.pipeline import Pipeline
    _, wave = fc.token_split(spec_of(fmt, G), P, 4096, H)
    w = synth.Workload("qsplit", P=P, T=wave + wave // 3 + 7, H=H, fmt=fmt, group=G, splits=2)
    inp = synth.make_inputs(w, seed=41)
    pipe = Pipeline(w, inp, split=mode)
    assert 0 < pipe.bounds[1] < w.T
    pipe.step()
    pipe.step()
    check_every_element(orc, w, pipe, inp)


# ---------------------------------------- self-synchronizing quantized payloads --
QT_CASES = [("decode-qtagged", {"T": 12}), ("prefill-qtagged", {"T": 10}),
            ("i8t-p3", {"P": 3, "T": 5, "H": 1152, "fmt": I8T, "group": 128}),
            ("i4t-p5", {"P": 5, "T": 7, "H": 4128, "fmt": I4T, "group": 32}),
            # enough rows for a CTA per row: the build without the h buffer
            ("i8t-p8-h8192-rows", {"P": 8, "T": 160, "H": 8192, "fmt": I8T, "group": 128}),
            # more rows than one wave: the residual-free stages of the tagged
            # formats (two-row rings for two slabs; one-row stages for eight
            # INT4 and four INT8 slabs, as two half-row sub-stages at H = 8192;
            # eight INT4 slabs without the h row buffer)
            ("i4t-p2-h4096-rows", {"P": 2, "T": 1000, "H": 4096, "fmt": I4T, "group": 32}),
            ("i4t-p2-h8192-rows", {"P": 2, "T": 480, "H": 8192, "fmt": I4T, "group": 32}),
            ("i4t-p8-h4096-rows", {"P": 8, "T": 640, "H": 4096, "fmt": I4T, "group": 32}),
            # eight tagged INT4 slabs at H = 8192: half-row sub-stages without the
            # h row buffer (pass 2 reads h back from residual_out)
            ("i4t-p8-h8192-rows", {"P": 8, "T": 320, "H": 8192, "fmt": I4T, "group": 32}),
            # four tagged INT4 slabs at H = 8192 (the prefill-qtagged rows)
            ("i4t-p4-h8192-rows", {"P": 4, "T": 480, "H": 8192, "fmt": I4T, "group": 32}),
            ("i4t-p6-h8192-rows", {"P": 6, "T": 320, "H": 8192, "fmt": I4T, "group": 32}),
            ("i8t-p3-h4096-rows", {"P": 3, "T": 800, "H": 4096, "fmt": I8T, "group": 128}),
            ("i8t-p2-h4096-rows", {"P": 2, "T": 1000, "H": 4096, "fmt": I8T, "group": 128}),
            ("i8t-p2-h8192-rows", {"P": 2, "T": 480, "H": 8192, "fmt": I8T, "group": 128}),
            ("i8t-p4-h4096-rows", {"P": 4, "T": 800, "H": 4096, "fmt": I8T, "group": 128}),
            ("i8t-p4-h8192-rows", {"P": 4, "T": 320, "H": 8192, "fmt": I8T, "group": 128})]


@pytest.mark.parametrize("name,kw", QT_CASES, ids=[c[0] for c in QT_CASES])
def test_quantized_tagged_producer_and_consumer(orc, name, kw):
    """Producer: the blocks equal the oracle's packing of the oracle's codes.
    Consumer: the fused path equals the oracle (same math as untagged)."""
    from quantized_reduce_rmsnorm_gb300.pipeline import Pipeline
    w = small(name, **kw)
    inp = synth.make_inputs(w, seed=41)
    pipe = Pipeline(w, inp)
    pipe.step()
    got = pipe.outputs()
    base = synth.base_format(w.fmt)
    for p in range(w.P):
        q, s, z = oracle_quant(orc, synth.Workload(**{**w.__dict__, "fmt": base}), inp["slabs"][p])
        want = orc.pack_qtagged(base, q, s, z, w.group, pipe.epoch)
        assert_bits_equal(host(pipe.blocks[p]).view(np.uint32), want, f"blocks slab {p}")
    check_fused(orc, synth.Workload(**{**w.__dict__, "fmt": base}), got, oracle_fused(orc, w, inp))
    assert got["status"].tolist() == [[fc.FC_OK, fc.STATUS_NO_INDEX]]


@pytest.mark.parametrize("H", [1024, 8192])
@pytest.mark.parametrize("T", [4, 8], ids=["cta-per-row", "cluster-per-row"])
@pytest.mark.parametrize("fmt,G,nbg", [(I8T, 128, 11), (I4T, 32, 2)])
@pytest.mark.parametrize("P", [3, 8])
def test_quantized_tagged_stale_blocks(orc, fmt, G, nbg, T, H, P):
    """Blocks built on the host by the oracle, one tag corrupted before upload
    (4 rows: a CTA per row, whose 8192-element rows are staged as two half-row
    sub-stages; 8 rows of 8192: each row shared by a cluster of CTAs, whose
    segments offset the block index, while 8 rows of 1024 take a CTA per row;
    eight INT8 slabs at H = 8192 take the build whose stage holds no
    residual)."""
    check_stale_blocks(orc, fmt, G, nbg, T, H, P, ((1, 2, 5), (2, 3, None), (0, 0, nbg - 1)))


@pytest.mark.parametrize("fmt,G,nbg,T,H,P", [(I4T, 32, 2, 1000, 4096, 2), (I8T, 128, 11, 320, 8192, 4),
                                              (I4T, 32, 2, 320, 8192, 8)],
                         ids=["i4t-p2-two-row-ring", "i8t-p4-half-rows", "i4t-p8-no-h-buffer"])
def test_quantized_tagged_stale_blocks_residual_free(orc, fmt, G, nbg, T, H, P):
    """The residual-free stages of the tagged formats (more rows than one
    wave) report the first stale block too: in the first row, a middle row
    and the last row."""
    check_stale_blocks(orc, fmt, G, nbg, T, H, P, ((1, T - 1, 3), (0, T // 2, None), (P - 1, 0, 0)))


def check_stale_blocks(orc, fmt, G, nbg, T, H, P, sites):
    """sites: (slab, row, block) to corrupt one at a time (block None: the
    row's last block); each call must report that block's flat index."""
    base = synth.base_format(fmt)
    w = synth.Workload("qtstale", P=P, T=T, H=H, fmt=fmt, group=G)
    inp = synth.make_inputs(w, seed=42)
    ep = 5
    blocks = []
    for s_ in inp["slabs"]:
        q, s, z = orc.quantize(base, bf16_float(s_).ravel(), G)
        blocks.append(orc.pack_qtagged(base, q, s, z, G, ep))
    spec = spec_of(fmt, G)
    r_in, gam = dev_bf16(inp["residual"]), dev_bf16(inp["gamma"])
    r_out, y = torch.empty_like(r_in), torch.empty_like(r_in)
    st = torch.full((2,), -1, dtype=torch.int32, device="cuda")

    def call(bl):
        fc.allreduce_residual_rmsnorm([dev(b.view(np.int32)) for b in bl], spec, w.T, w.H, r_in, r_out,
                                      gam, w.eps, y, expected_epoch=ep, d_status=st)
        torch.cuda.synchronize()
        return list(host(st))

    assert call(blocks) == [fc.FC_OK, fc.STATUS_NO_INDEX]
    want = oracle_fused(orc, w, inp)
    assert_bits_equal(host_bits(r_out), want["h"], "residual_out")
    # residual_out aliasing the residual (builds without the h row buffer
    # read h back from it)
    r_al = r_in.clone()
    fc.allreduce_residual_rmsnorm([dev(b.view(np.int32)) for b in blocks], spec, w.T, w.H, r_al, r_al, gam,
                                  w.eps, y, expected_epoch=ep, d_status=st)
    torch.cuda.synchronize()
    assert list(host(st)) == [fc.FC_OK, fc.STATUS_NO_INDEX]
    assert_bits_equal(host_bits(r_al), want["h"], "residual_out in place")
    assert_y_close(host_bits(y), want["y"])
    bpr = (w.H // G) * nbg
    for slab, row, blk in sites:
        blk = bpr - 1 if blk is None else blk
        bad = [b.copy() for b in blocks]
        bad[slab][4 * (row * bpr + blk) + 3] = ep + 1
        assert call(bad) == [fc.FC_ERR_STALE_BLOCK, (slab * w.T + row) * bpr + blk]


def test_quantized_tagged_rejects_other_groups():
    x = torch.zeros(2, 4096, dtype=torch.bfloat16, device="cuda")
    b = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(fc.FcommError) as e:
        fc.group_quantize_tagged([x], fc.QSpec(I8T, 64), 1, [b])
    assert e.value.status == fc.FC_ERR_UNSUPPORTED


# --------------------------------------------------- full-size, sampled rows --
# ----------------------------------------------------- standalone gather ---
def _gather_shards_host(orc, fmt, G, T, H, P, seed):
    """The oracle's payload of a seeded bf16 tensor, cut into P shards."""
    w = synth.Workload("gather", P=1, T=T, H=H, fmt=fmt, group=G, outlier_frac=0.01,
                       outlier_scale=30.0)
    x = bf16_float(synth.make_inputs(w, seed=seed)["slabs"][0]).ravel()
    q, s, z = orc.quantize(fmt, x, G)
    ng = x.size // G
    per = -(-ng // P)
    cb = G if fmt == I8 else G // 2
    shards = []
    for j in range(P):
        g0, g1 = min(j * per, ng), min((j + 1) * per, ng)
        shards.append((q[g0 * cb:g1 * cb], s[g0:g1], None if z is None else z[g0:g1]))
    return x.size, shards


def _dev_shards(shards):
    return [(None, None, None) if c.size == 0 else
            (dev(c.view(np.uint8)), dev(s_), None if z is None else dev(z)) for c, s_, z in shards]


GATHER_CASES = [(I8, 128, 1), (I8, 128, 3), (I8, 128, 8), (I4, 32, 2), (I4, 32, 5), (I4, 32, 8),
                (I8, 32, 4), (I4, 16, 3), (I4, 128, 8)]


@pytest.mark.parametrize("fmt,G,P", GATHER_CASES)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_allgather_dequant_bit_exact(orc, fmt, G, P, out_dtype):
    """Ragged shards (the group count is not a multiple of P) of a payload the
    oracle built on the host; fp32 output bit-exact, bf16 = its RNE rounding."""
    T, H = 7, 1152
    n, shards = _gather_shards_host(orc, fmt, G, T, H, P, seed=60 + P)
    want = orc.allgather_dequant(fmt, shards, n, G)
    out = torch.empty(T, H, dtype=out_dtype, device="cuda")
    fc.allgather_dequant(_dev_shards(shards), spec_of(fmt, G), T, H, out)
    torch.cuda.synchronize()
    if out_dtype == torch.float32:
        assert_bits_equal(host(out), want, "gathered fp32")
    else:
        assert_bits_equal(host_bits(out), orc.f32_to_bf16_array(want), "gathered bf16")


def test_allgather_more_shards_than_groups(orc):
    """P = 8 shards of a 5-group tensor: shards 5..7 are empty (NULL buffers)."""
    T, H, G = 1, 640, 128
    n, shards = _gather_shards_host(orc, I8, G, T, H, 8, seed=70)
    assert [c.size for c, _, _ in shards][5:] == [0, 0, 0]
    out = torch.empty(T, H, dtype=torch.float32, device="cuda")
    fc.allgather_dequant(_dev_shards(shards), spec_of(I8, G), T, H, out)
    torch.cuda.synchronize()
    assert_bits_equal(host(out), orc.allgather_dequant(I8, shards, n, G), "gathered")


@pytest.mark.parametrize("fmt,G,nbg", [(I8T, 128, 11), (I4T, 32, 2)])
def test_allgather_tagged_shards_and_stale_blocks(orc, fmt, G, nbg):
    """Self-synchronizing shards (blocks built by the oracle on the host): every
    group bit-exact; a corrupted tag is reported with its index (shard 0's
    blocks first), and every group but the stale block's stays exact."""
    base = synth.base_format(fmt)
    T, H, P, ep = 5, 1024, 3, 9
    n, shards = _gather_shards_host(orc, base, G, T, H, P, seed=80)
    blocks = [orc.pack_qtagged(base, c, s_, z, G, ep) for c, s_, z in shards]
    want = orc.allgather_dequant(base, shards, n, G)
    spec = spec_of(fmt, G)
    st = torch.full((2,), -1, dtype=torch.int32, device="cuda")

    def call(bl):
        out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        fc.allgather_dequant([dev(b.view(np.int32)) for b in bl], spec, T, H, out,
                             expected_epoch=ep, d_status=st)
        torch.cuda.synchronize()
        return host(out).ravel(), list(host(st))

    got, status = call(blocks)
    assert status == [fc.FC_OK, fc.STATUS_NO_INDEX]
    assert_bits_equal(got, want, "gathered")
    nblk = [b.size // 4 for b in blocks]
    for shard, blk in ((1, 3), (2, nblk[2] - 1), (0, 0)):
        bad = [b.copy() for b in blocks]
        bad[shard][4 * blk + 3] = ep + 1
        got, status = call(bad)
        assert status == [fc.FC_ERR_STALE_BLOCK, sum(nblk[:shard]) + blk]
        g = sum(nblk[:shard]) // nbg + blk // nbg  # the global group of the stale block
        keep = np.ones(n, bool)
        keep[g * G:(g + 1) * G] = False
        assert_bits_equal(got[keep], want[keep], "gathered, other groups")


def test_allgather_full_size_sampled(orc):
    """A prefill-sized INT4 payload (8192 x 8192, P = 4 shards) of random codes,
    scales and zero-points drawn on the host; sampled rows against the oracle."""
    T, H, G, P = 8192, 8192, 32, 4
    rng = np.random.default_rng(90)
    ng = T * H // G
    codes = rng.integers(0, 256, T * H // 2, dtype=np.uint8)
    scales = (rng.random(ng, dtype=np.float32) * 0.5).astype(np.float32)
    zeros = rng.standard_normal(ng).astype(np.float32)
    spec = spec_of(I4, G)
    whole = (dev(codes), dev(scales), dev(zeros))
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    fc.allgather_dequant(fc.shard_views(whole, spec, T, H, P), spec, T, H, out)
    torch.cuda.synchronize()
    gpb = H // G
    for r in (0, 1, 2047, 2048, 4095, 6000, 8191):
        want = orc.dequantize(I4, codes[r * H // 2:(r + 1) * H // 2], scales[r * gpb:(r + 1) * gpb],
                              zeros[r * gpb:(r + 1) * gpb], G)
        assert_bits_equal(host_bits(out[r]), orc.f32_to_bf16_array(want), f"row {r}")


def _row_ranges(T, parts):
    return [(T * k // parts, T * (k + 1) // parts) for k in range(parts) if T * (k + 1) // parts > T * k // parts]


def _host_threads():
    import os
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_fused_all(orc, w, inp):
    """The oracle's whole path over every row: the rows are cut into
    contiguous ranges, each one unmodified oracle call on its own host thread
    (rows are independent, and tests/test_bench_host.py checks that ranges
    give the bits of one call).  Returns dict(h, y[, codes, scales, zeros])
    over all rows, flat in row-major order."""
    import concurrent.futures as cf
    fmt = BF if w.fmt == TG else synth.base_format(w.fmt)
    parts = _row_ranges(w.T, min(w.T, 4 * _host_threads()))

    def one(rr):
        r0, r1 = rr
        return orc.allreduce_residual_rmsnorm(fmt, [s[r0:r1] for s in inp["slabs"]],
                                              inp["residual"][r0:r1], inp["gamma"], r1 - r0, w.H,
                                              w.group, w.eps)
    with cf.ThreadPoolExecutor(_host_threads()) as ex:
        outs = list(ex.map(one, parts))
    res = {k: np.concatenate([o[k].ravel() for o in outs]) for k in ("h", "y")}
    for k in ("codes", "scales", "zeros"):
        if outs[0].get(k) is not None:
            res[k] = np.concatenate([o[k].ravel() for o in outs])
    return res


def oracle_quant_all(orc, fmt, slab_bits, G, T):
    """The oracle's quantizer over a whole slab, in contiguous row ranges on
    host threads (groups never straddle rows).  (codes, scales, zeros)."""
    import concurrent.futures as cf
    parts = _row_ranges(T, min(T, 4 * _host_threads()))

    def one(rr):
        return orc.quantize(fmt, bf16_float(slab_bits[rr[0]:rr[1]]).ravel(), G)
    with cf.ThreadPoolExecutor(_host_threads()) as ex:
        outs = list(ex.map(one, parts))
    cat = lambda i: None if outs[0][i] is None else np.concatenate([o[i] for o in outs])
    return cat(0), cat(1), cat(2)


def check_every_element(orc, w, pipe, inp):
    """Every output of a Pipeline step against the oracle: residual_out
    bit-exact, y within one bf16 ulp, the all-gather payload bit-exact, and
    every slab's sender output (codes, scales, zero-points, or tagged
    blocks with the step's epoch) bit-exact."""
    got = pipe.outputs()
    want = oracle_fused_all(orc, w, inp)
    assert_bits_equal(got["h"], want["h"], "residual_out")
    assert_y_close(got["y"], want["y"])
    if w.fmt in (I8, I4, I8T, I4T):
        assert_bits_equal(got["codes"], want["codes"], "payload codes")
        assert_bits_equal(got["scales"], want["scales"], "payload scales")
        if w.fmt in (I4, I4T):
            assert_bits_equal(got["zeros"], want["zeros"], "payload zeros")
    base = synth.base_format(w.fmt)
    for p in range(w.P):
        if w.fmt in (I8, I4, I8T, I4T):
            q, s_, z = oracle_quant_all(orc, base, inp["slabs"][p], w.group, w.T)
            if w.fmt in (I8, I4):
                assert_bits_equal(host(pipe.codes[p][0]), q, f"sender codes, slab {p}")
                assert_bits_equal(host(pipe.codes[p][1]), s_, f"sender scales, slab {p}")
                if w.fmt == I4:
                    assert_bits_equal(host(pipe.codes[p][2]), z, f"sender zeros, slab {p}")
            else:
                blk = orc.pack_qtagged(base, q, s_, z, w.group, pipe.epoch)
                assert_bits_equal(host(pipe.blocks[p]).view(np.uint32), blk, f"sender blocks, slab {p}")
        elif w.fmt == TG:
            blk = orc.pack_tagged(inp["slabs"][p], w.T, w.H, pipe.epoch)
            assert_bits_equal(host(pipe.blocks[p]).view(np.uint32), blk, f"producer blocks, slab {p}")
    if w.fmt in (I8T, I4T):
        assert got["status"].tolist() == [[fc.FC_OK, fc.STATUS_NO_INDEX]]
    if w.fmt == TG:
        assert got["status"].tolist() == [[fc.FC_OK, fc.STATUS_NO_INDEX]] * w.splits


FULL_SIZE = ["decode", "prefill", "token-split", "prefill-qtagged", "decode-tiny", "decode-qtagged",
             "sweep-256M-h8192-p8-int4"]


@pytest.mark.parametrize("name", FULL_SIZE)
def test_full_size_every_element(orc, name):
    """The full-size workloads through the same Pipeline.step() the
    benchmark times (token-split: two subsets on two streams; a second step
    with a new epoch for the tagged formats), every element compared with
    the oracle; also the largest sweep point (a 256 MB message, eight INT4
    slabs of 16384 x 8192)."""
    from quantized_reduce_rmsnorm_gb300.pipeline import Pipeline
    if name.startswith("sweep"):
        w, seed = synth.sweep_workload(8192, 16384, 8, I4, 32), 3
    else:
        w, seed = synth.WORKLOADS[name], 0
    inp = synth.make_inputs(w, seed=seed)
    pipe = Pipeline(w, inp)
    pipe.step()
    pipe.step()
    check_every_element(orc, w, pipe, inp)
    del pipe
    torch.cuda.empty_cache()


def test_rows_zero_launches_nothing():
    spec = fc.INT8_G128
    t = torch.empty(0, 4096, dtype=torch.bfloat16, device="cuda")
    fc.group_quantize(t, spec, fc.alloc_qtensor(spec, 0, 4096))
    torch.cuda.synchronize()


def test_invalid_arguments_rejected_before_launch():
    spec = fc.INT8_G128
    x = torch.zeros(2, 4096, dtype=torch.bfloat16, device="cuda")
    out = fc.alloc_qtensor(spec, 2, 4096)
    bad = torch.zeros(2 * 4096 + 8, dtype=torch.bfloat16, device="cuda")[8:].view(2, 4096)
    with pytest.raises(fc.FcommError) as e:
        fc.group_quantize(bad, spec, out)            # 16-byte but not 32-byte aligned
    assert e.value.status == fc.FC_ERR_INVALID
    with pytest.raises(fc.FcommError):
        fc.group_quantize(x, fc.QSpec(fc.FMT_INT8_SYM, 96), out)   # group not a power of 2
    with pytest.raises(fc.FcommError):
        fc.allreduce_residual_rmsnorm([out], spec, 2, 4096, x, x, x[0], 1e-5, x)  # P = 1


def test_bound_call_epoch_and_repeat(orc):
    """A bound fused call (arguments marshalled once) gives the same bits as
    the plain call, again on a second launch, and a changed epoch makes
    every block stale (first index 0) without touching the rest."""
    w = small("tagged-bound", P=3, T=5, H=1040, fmt=TG, group=0)
    inp = synth.make_inputs(w, seed=53)
    xs = [dev_bf16(s) for s in inp["slabs"]]
    blocks = [torch.empty(fc.tagged_bytes(w.T, w.H), dtype=torch.uint8, device="cuda")
              for _ in range(w.P)]
    fc.pack_tagged_multi(xs, 7, blocks)
    res, gam = dev_bf16(inp["residual"]), dev_bf16(inp["gamma"])
    h, y = torch.empty_like(res), torch.empty_like(res)
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    call = fc.bind_allreduce_residual_rmsnorm(blocks, fc.BF16_TAGGED, w.T, w.H, res, h, gam,
                                              w.eps, y, expected_epoch=7, d_status=st)
    want = oracle_fused(orc, w, inp)
    for _ in range(2):
        h.zero_(), y.zero_()
        call()
        torch.cuda.synchronize()
        assert host(st).tolist() == [fc.FC_OK, fc.STATUS_NO_INDEX]
        check_fused(orc, w, {"h": host_bits(h), "y": host_bits(y)}, want)
    call.epoch = 8
    assert call.epoch == 8
    call()
    torch.cuda.synchronize()
    assert host(st).tolist() == [fc.FC_ERR_STALE_BLOCK, 0]


def test_launch_shapes_alternate(orc):
    """Calls whose staged kernels need different shared memory, in the order
    large, small, large (the second large call reuses remembered launch
    shapes), all match the oracle."""
    for H in (16384, 1024, 16384):
        w = small(f"i8-h{H}", P=4, T=3, H=H, fmt=I8, group=128)
        inp = synth.make_inputs(w, seed=H)
        outs = quantize_on_gpu(w, inp)
        res, gam = dev_bf16(inp["residual"]), dev_bf16(inp["gamma"])
        h, y = torch.empty_like(res), torch.empty_like(res)
        fc.allreduce_residual_rmsnorm(outs, fc.INT8_G128, w.T, w.H, res, h, gam, w.eps, y,
                                      kernel=fc.KERNEL_TMA)
        torch.cuda.synchronize()
        check_fused(orc, w, {"h": host_bits(h), "y": host_bits(y)}, oracle_fused(orc, w, inp))


@pytest.mark.parametrize("name", ["decode", "prefill", "bf16-graph"])
def test_graph_replay_matches_step(orc, name):
    """A step captured into a CUDA graph (the kernels keep their programmatic
    dependent launch edges) and replayed twice writes the same bits as the
    launched step, and matches the oracle."""
    from quantized_reduce_rmsnorm_gb300.pipeline import Pipeline
    kw = {"T": 24} if name != "bf16-graph" else {"P": 3, "T": 7, "H": 4096, "fmt": BF, "group": 0}
    w = small(name, **kw)
    inp = synth.make_inputs(w, seed=61)
    direct = Pipeline(w, inp)
    direct.step()
    want = direct.outputs()
    pipe = Pipeline(w, inp)
    pipe.capture()
    for _ in range(2):
        pipe.residual_out.zero_(), pipe.y.zero_()
        pipe.replay()
        got = pipe.outputs()
        for k in want:
            if want[k] is not None:
                assert_bits_equal(got[k], want[k], f"graph replay: {k}")
    check_fused(orc, w, got, oracle_fused(orc, w, inp))


def test_graph_capture_refuses_tagged():
    from quantized_reduce_rmsnorm_gb300.pipeline import Pipeline
    w = small("token-split", T=12)
    pipe = Pipeline(w, synth.make_inputs(w, seed=1))
    with pytest.raises(ValueError):
        pipe.capture()


@pytest.mark.parametrize("fmt,G", [(I4, 32), (I8, 128)])
@pytest.mark.parametrize("P", [2, 4])
@pytest.mark.parametrize("kernel", [fc.KERNEL_AUTO, fc.KERNEL_STREAM], ids=["auto", "stream"])
def test_fused_dense_exact_ties(orc, fmt, G, P, kernel):
    """Requantized sums whose quotients are exact half-integers for a large
    share of elements: every slab holds integers in [0, 15] (INT4) or
    [-127, 127] (INT8), and every group of every slab holds both extremes at
    the same positions, so the reduced group spans P times the slab range and
    its scale is P times the slab scale.  The exact pass then settles dense
    ties (INT4 with two slabs: every odd sum), in the staged kernel and in the
    streaming kernel."""
    T, H = 6, 2048
    rng = np.random.default_rng(P * 10 + fmt)
    lo, hi = (0, 15) if fmt == I4 else (-127, 127)
    slabs = []
    for _ in range(P):
        x = rng.integers(lo, hi + 1, size=(T, H)).astype(np.float32)
        x.reshape(T, H // G, G)[:, :, 0] = lo
        x.reshape(T, H // G, G)[:, :, 1] = hi
        slabs.append(orc.f32_to_bf16_array(x.ravel()).reshape(T, H))
    base = synth.make_inputs(synth.Workload("ties", P=P, T=T, H=H, fmt=fmt, group=G), seed=5)
    inp = dict(slabs=slabs, residual=base["residual"], gamma=base["gamma"])
    w = synth.Workload("ties", P=P, T=T, H=H, fmt=fmt, group=G)
    want = oracle_fused(orc, w, inp)
    q = want["codes"].view(np.uint8)
    if fmt == I4 and P == 2:  # a large share of the quotients were exact ties
        assert np.mean(((q & 0xF) % 2 == 0)) > 0.55
    check_fused(orc, w, run_fused(w, inp, kernel=kernel), want)


SWEEP_PARITY = [(msg, H, P, fmt, G) for msg in (16 << 10, 1 << 20, 16 << 20) for H in (4096, 8192)
                for P in (2, 4, 8) for fmt, G in ((BF, 0), (I8, 128), (I4, 32))]


@pytest.mark.parametrize("msg,H,P,fmt,G", SWEEP_PARITY,
                         ids=[f"{m >> 10}K-h{h}-p{p}-{synth.FMT_NAMES[f]}" for m, h, p, f, _ in SWEEP_PARITY])
def test_sweep_point_every_element(orc, msg, H, P, fmt, G):
    """Message-size sweep shapes (every H, P and format at 16 KB, 1 MB and
    16 MB messages) through the same Pipeline.step() as the benchmark, with
    seeded N(0,1) inputs; every element against the oracle."""
    from quantized_reduce_rmsnorm_gb300.pipeline import Pipeline
    T = msg // (2 * H)
    w = synth.sweep_workload(H, T, P, fmt, G)
    inp = synth.make_inputs(w, seed=3)
    pipe = Pipeline(w, inp)
    pipe.step()
    check_every_element(orc, w, pipe, inp)


@pytest.mark.parametrize("fmt,G,tagged", [(I8, 128, False), (I4, 32, False), (I8T, 128, True)])
def test_sender_status_word_reset_to_ok(orc, fmt, G, tagged):
    """The sender calls set their optional status word to {FC_OK, 0x7F7F7F7F}
    (a staged copy that never lands would turn word 0 into FC_ERR_CUDA; that
    path needs a fault to trigger and is not run), and the codes are still
    the oracle's."""
    w = small("status", P=3, T=5, H=2048, fmt=fmt, group=G)
    inp = synth.make_inputs(w, seed=71)
    xs = [dev_bf16(s) for s in inp["slabs"]]
    st = torch.full((2,), -5, dtype=torch.int32, device="cuda")
    spec = spec_of(fmt, G)
    if tagged:
        blocks = [torch.empty(fc.codes_bytes(spec, w.T, w.H), dtype=torch.uint8, device="cuda")
                  for _ in range(w.P)]
        fc.group_quantize_tagged(xs, spec, 4, blocks, d_status=st)
    else:
        outs = [fc.alloc_qtensor(spec, w.T, w.H) for _ in range(w.P)]
        fc.group_quantize_multi(xs, spec, outs, d_status=st)
    torch.cuda.synchronize()
    assert host(st).tolist() == [fc.FC_OK, fc.STATUS_NO_INDEX]
    base = synth.base_format(fmt)
    for p in range(w.P):
        q, s_, z = orc.quantize(base, bf16_float(inp["slabs"][p]).ravel(), G)
        if tagged:
            assert_bits_equal(host(blocks[p]).view(np.uint32), orc.pack_qtagged(base, q, s_, z, G, 4),
                              f"blocks slab {p}")
        else:
            assert_bits_equal(host(outs[p][0]), q, f"codes slab {p}")
            assert_bits_equal(host(outs[p][1]), s_, f"scales slab {p}")


def test_protocol_selector_pick_within_5pct_of_measured_fastest():
    """One GPU (no link model): the selector's pick, from the measured rates
    compiled into the library, is within 5% of the encoding measured fastest
    here (sender + fused steady device time), at shapes on and off the
    measured grid; the estimate errors are reported."""
    import bench
    for r in bench.selector_check([(192, 8192, 4), (768, 8192, 8), (512, 8192, 3)], calls=50, reps=3):
        print(r["rows"], r["hidden"], r["P"], "pick", r["pick"], "fastest", r["fastest"],
              "errors", r["est_error"])
        assert r["pick_over_fastest"] <= 1.05, r
