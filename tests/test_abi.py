"""CPU checks of the C ABI: the library loads, exports every symbol the
header declares, sizes and shard ranges are right, and bad arguments are
rejected before anything touches a GPU."""
import ctypes
import os
import re

import pytest

import quantized_reduce_rmsnorm_gb300 as fc

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "fcomm.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fc_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = fc.fcomm.load()
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), f"{n} declared in fcomm.h but not exported"
    assert set(names) == set(fc.fcomm.EXPORTS)


def test_version_and_status_strings():
    lib = fc.fcomm.load()
    assert "sm_103a" in fc.version()
    assert lib.fc_status_string(3) == b"FC_ERR_STALE_BLOCK"


def test_sizes():
    assert fc.codes_bytes(fc.INT8_G128, 64, 8192) == 64 * 8192
    assert fc.codes_bytes(fc.INT4_G32, 8192, 8192) == 8192 * 8192 // 2
    assert fc.codes_bytes(fc.BF16, 3, 16) == 96
    assert fc.groups(fc.INT4_G32, 8192, 8192) == 8192 * 8192 // 32
    assert fc.groups(fc.BF16, 8192, 8192) == 0
    assert fc.tagged_bytes(2048, 5120) == 2048 * 854 * 16
    assert fc.tagged_bytes(1, 6) == 16 and fc.tagged_bytes(1, 7) == 32


@pytest.mark.parametrize("P", [2, 3, 4, 8])
def test_shard_ranges_partition_the_groups(P):
    ng = fc.groups(fc.INT8_G128, 7, 1152)
    ranges = [fc.shard_range(fc.INT8_G128, 7, 1152, P, j) for j in range(P)]
    per = -(-ng // P)
    assert ranges[0][0] == 0 and ranges[-1][1] == ng
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    assert all(0 <= b - a <= per for a, b in ranges)


def _status(call):
    lib = fc.fcomm.load()
    return call(lib), lib.fc_last_error().decode()


@pytest.mark.parametrize("hidden,group,fmt", [
    (100, 128, 1),     # hidden not a multiple of 16
    (4096, 96, 1),     # group not a power of two
    (4096, 8, 2),      # group below 16
    (4000, 128, 1),    # hidden not a multiple of group
    (4096, 128, 9),    # unknown format
    (4096, 128, 0),    # bf16 is not a quantized format
])
def test_quantize_rejects_bad_specs(hidden, group, fmt):
    st, msg = _status(lambda L: L.fc_group_quantize(None, 4, hidden, fc.QSpec(fmt, group),
                                                    fc.QTensor(), None, None))
    assert st == fc.FC_ERR_INVALID and msg


def test_pointer_checks_precede_any_launch():
    q = fc.QTensor(64, 128, None)
    st, msg = _status(lambda L: L.fc_group_quantize(None, 4, 4096, fc.INT8_G128, q, None, None))
    assert st == fc.FC_ERR_INVALID and "NULL" in msg
    st, msg = _status(lambda L: L.fc_group_quantize(48, 4, 4096, fc.INT8_G128, q, None, None))
    assert st == fc.FC_ERR_INVALID and "aligned" in msg
    bad = fc.QTensor(64, 130, None)   # scales not 4-byte aligned
    st, msg = _status(lambda L: L.fc_group_quantize(64, 4, 4096, fc.INT8_G128, bad, None, None))
    assert st == fc.FC_ERR_INVALID and "scales" in msg
    nozeros = fc.QTensor(64, 128, None)
    st, msg = _status(lambda L: L.fc_group_quantize(64, 4, 4096, fc.INT4_G32, nozeros, None, None))
    assert st == fc.FC_ERR_INVALID and "zeros" in msg


def test_fused_rejects_bad_p_eps_and_opts():
    slabs = (fc.QTensor * 9)(*[fc.QTensor(64, 128, 256)] * 9)
    q = fc.QTensor()
    lib = fc.fcomm.load()
    for P in (0, 1, 9):
        st = lib.fc_allreduce_residual_rmsnorm(slabs, P, 4, 4096, fc.INT8_G128, 64, 64, 64,
                                               1e-5, q, 64, 0, None, None)
        assert st == fc.FC_ERR_INVALID
    st = lib.fc_allreduce_residual_rmsnorm(slabs, 2, 4, 4096, fc.INT8_G128, 64, 64, 64,
                                           -1.0, q, 64, 0, None, None)
    assert st == fc.FC_ERR_INVALID
    opts = fc.LaunchOpts(-1)
    st = lib.fc_allreduce_residual_rmsnorm_ex(slabs, 2, 4, 4096, fc.INT8_G128, 64, 64, 64,
                                              1e-5, q, 64, 0, None, ctypes.byref(opts), None)
    assert st == fc.FC_ERR_INVALID


def test_reduce_rejects_bad_shard():
    slabs = (fc.QTensor * 2)(*[fc.QTensor(64, 128, 256)] * 2)
    lib = fc.fcomm.load()
    for shard in (-2, 2):
        st = lib.fc_reduce_dequant_sum(slabs, 2, 4, 4096, fc.INT8_G128, shard, 64, None)
        assert st == fc.FC_ERR_INVALID


def test_rows_zero_is_a_no_op():
    lib = fc.fcomm.load()
    st = lib.fc_group_quantize(None, 0, 4096, fc.INT8_G128, fc.QTensor(), None, None)
    assert st == fc.FC_OK


def test_product_package_never_imports_the_oracle():
    pkg = os.path.dirname(fc.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(root, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", txt, re.M), f
                assert "liboracle" not in txt and "oracle.h" not in txt, f


def test_protocol_selector_trades_barriers_against_bytes():
    """One GPU (no wire, no barrier): plain bf16, since quantizing costs
    compute and saves nothing.  With a link, large messages quantize; with a
    slow barrier, small messages take a tagged encoding and large ones do not;
    the bit-width floor is always respected."""
    F = fc.fcomm
    for bits in (4, 8, 16):
        c, t = fc.select_protocol(8192, 8192, 4, bits)
        assert c.fmt == F.FMT_BF16 and t > 0
    c, _ = fc.select_protocol(8192, 8192, 8, 4, link_gbps=100.0, barrier_us=0.0)
    assert c.fmt == F.FMT_INT4_ASYM
    small, _ = fc.select_protocol(1, 4096, 8, 8, link_gbps=450.0, barrier_us=8.0)
    large, _ = fc.select_protocol(16384, 8192, 8, 8, link_gbps=450.0, barrier_us=8.0)
    assert small.fmt in (F.FMT_INT8_TAGGED, F.FMT_BF16_TAGGED)
    assert large.fmt in (F.FMT_INT8_SYM, F.FMT_INT4_ASYM, F.FMT_BF16)
    for bits in (4, 8, 16):
        for rows in (1, 64, 4096):
            c, _ = fc.select_protocol(rows, 8192, 4, bits, link_gbps=100.0, barrier_us=5.0)
            width = {F.FMT_BF16: 16, F.FMT_BF16_TAGGED: 16, F.FMT_INT8_SYM: 8,
                     F.FMT_INT8_TAGGED: 8, F.FMT_INT4_ASYM: 4, F.FMT_INT4_TAGGED: 4}[c.fmt]
            assert width >= bits
    with pytest.raises(fc.FcommError):
        fc.select_protocol(1, 4096, 8, 3)


def test_allgather_rejects_bad_arguments():
    lib = fc.fcomm.load()
    shards = (fc.QTensor * 8)(*[fc.QTensor(64, 128, 256)] * 8)
    for P in (0, 9):
        assert lib.fc_allgather_dequant(shards, P, 4, 4096, fc.INT8_G128, 0, 64, 0, None,
                                        None) == fc.FC_ERR_INVALID
    # bf16 is not a quantized payload; out_dtype must be bf16 or f32
    assert lib.fc_allgather_dequant(shards, 2, 4, 4096, fc.BF16, 0, 64, 0, None, None) == \
        fc.FC_ERR_INVALID
    assert lib.fc_allgather_dequant(shards, 2, 4, 4096, fc.INT8_G128, 1, 64, 0, None, None) == \
        fc.FC_ERR_INVALID
    # misaligned output, NULL codes of a non-empty shard
    assert lib.fc_allgather_dequant(shards, 2, 4, 4096, fc.INT8_G128, 0, 48, 0, None, None) == \
        fc.FC_ERR_INVALID
    bad = (fc.QTensor * 2)(fc.QTensor(64, 128, 256), fc.QTensor(None, 128, 256))
    assert lib.fc_allgather_dequant(bad, 2, 4, 4096, fc.INT8_G128, 0, 64, 0, None, None) == \
        fc.FC_ERR_INVALID
    assert "shards" in lib.fc_last_error().decode()
    # an empty shard may have NULL buffers (checked before any launch: rows = 0)
    assert lib.fc_allgather_dequant(bad, 2, 0, 4096, fc.INT8_G128, 0, 64, 0, None, None) == fc.FC_OK


def test_bound_call_reuses_marshalled_arguments():
    """fcomm.Bound passes the arguments it was built with, substitutes the
    stream on every call, lets the epoch change between calls and raises on a
    non-OK status (checked with a stand-in for the C entry point)."""
    fc.fcomm.load()
    seen = []

    def entry(*args):
        seen.append(args)
        return fc.FC_OK if len(seen) < 3 else fc.FC_ERR_INVALID

    b = fc.fcomm.Bound(entry, ["slabs", 4, ctypes.c_uint32(7), None], 3, 2)
    b(stream=11)
    b.epoch = 8
    b(stream=12)
    assert seen[0][:2] == ("slabs", 4) and seen[0][2].value == 7 and seen[0][3] == 11
    assert seen[1][2].value == 8 and seen[1][3] == 12 and b.epoch == 8
    b.epoch = 2 ** 32 + 5  # epochs are u32
    assert b.epoch == 5
    with pytest.raises(fc.FcommError):
        b(stream=13)


def test_kernel_hash_ignores_comments_only():
    """The hash that ties the committed ncu traffic to the kernel code sees
    code changes and not comment changes."""
    import bench
    src = "int a; // one\n/* two\n three */ int b;  \n\nint c;\n"
    assert bench.code_only(src) == "int a;\n int b;\nint c;"
    assert bench.code_only(src) == bench.code_only(src.replace("one", "uno").replace("three", "tres"))
    assert bench.code_only(src) != bench.code_only(src.replace("int c", "int d"))
    assert len(bench.source_hash()) == 16


def test_bound_call_keeps_its_tensors_alive(monkeypatch):
    """A bound call holds every tensor it was bound to: dropping the caller's
    own references must not free memory the call will touch again (the
    allocator would hand it to the next tensor).  Binding launches nothing,
    so host tensors serve here, with the binding's device-memory check
    relaxed for the test."""
    import gc
    import weakref

    import torch
    monkeypatch.setattr(fc.fcomm, "_ptr", lambda t: None if t is None else t.data_ptr())
    x = [torch.zeros(2, 128, dtype=torch.bfloat16) for _ in range(2)]
    outs = [fc.alloc_qtensor(fc.INT8_G128, 2, 128, "cpu") for _ in range(2)]
    res, gam = torch.zeros(2, 128, dtype=torch.bfloat16), torch.ones(128, dtype=torch.bfloat16)
    r_out, y = torch.empty_like(res), torch.empty_like(res)
    pay = fc.alloc_qtensor(fc.INT8_G128, 2, 128, "cpu")
    send = fc.bind_group_quantize_multi(x, fc.INT8_G128, outs)
    fuse = fc.bind_allreduce_residual_rmsnorm(outs, fc.INT8_G128, 2, 128, res, r_out, gam, 1e-5, y,
                                              requant_out=pay)
    refs = [weakref.ref(t) for t in x + [o[0] for o in outs] + [o[1] for o in outs]
            + [res, r_out, gam, y, pay[0], pay[1]]]
    del x, outs, res, gam, r_out, y, pay
    gc.collect()
    assert all(r() is not None for r in refs)
    del send, fuse
    gc.collect()
    assert all(r() is None for r in refs)


def test_bound_sender_passes_its_status_word(monkeypatch):
    """The sender calls marshal their optional status word into the C call
    (checked with a stand-in for the entry point, binding host tensors): a
    staged copy that never lands is then reported in it, not lost."""
    import torch
    monkeypatch.setattr(fc.fcomm, "_ptr", lambda t: None if t is None else t.data_ptr())
    seen = []

    class FakeLib:
        def fc_group_quantize_multi(self, *args):
            seen.append(("multi", args))
            return fc.FC_OK

        def fc_group_quantize_tagged(self, *args):
            seen.append(("tagged", args))
            return fc.FC_OK

    out = [fc.alloc_qtensor(fc.INT8_G128, 2, 128, "cpu")]
    monkeypatch.setattr(fc.fcomm, "load", lambda path=None: FakeLib())
    x = [torch.zeros(2, 128, dtype=torch.bfloat16)]
    st = torch.zeros(2, dtype=torch.int32)
    fc.bind_group_quantize_multi(x, fc.INT8_G128, out, d_status=st)(stream=5)
    fc.bind_group_quantize_tagged(x, fc.INT8_G128_TAGGED, 3, [torch.zeros(64, dtype=torch.uint8)],
                                  d_status=st)(stream=6)
    (k1, a1), (k2, a2) = seen
    assert k1 == "multi" and a1[6].value == st.data_ptr() and a1[7] == 5
    assert k2 == "tagged" and a2[7].value == st.data_ptr() and a2[8] == 6 and a2[5].value == 3


def test_bound_allgather_marshals_once(monkeypatch):
    """The bound all-gather passes the shards, the output, the epoch, the
    status word and the stream of each call (stand-in entry point, host
    tensors), and holds the tensors it was bound to."""
    import torch
    monkeypatch.setattr(fc.fcomm, "_ptr", lambda t: None if t is None else t.data_ptr())
    seen = []

    class FakeLib:
        def fc_allgather_dequant(self, *args):
            seen.append(args)
            return fc.FC_OK

    whole = fc.alloc_qtensor(fc.INT8_G128, 4, 256, "cpu")
    shards = fc.shard_views(whole, fc.INT8_G128, 4, 256, 3)
    monkeypatch.setattr(fc.fcomm, "load", lambda path=None: FakeLib())
    out = torch.zeros(4, 256, dtype=torch.float32)
    st = torch.zeros(2, dtype=torch.int32)
    call = fc.bind_allgather_dequant(shards, fc.INT8_G128, 4, 256, out, expected_epoch=9, d_status=st)
    call(stream=4)
    call.epoch = 10
    call(stream=5)
    (a1, a2) = seen
    assert a1[1] == 3 and a1[2] == 4 and a1[3] == 256 and a1[5] == fc.FMT_F32
    assert a1[6].value == out.data_ptr() and a1[8].value == st.data_ptr()
    assert a1[7].value == 9 and a1[9] == 4 and a2[7].value == 10 and a2[9] == 5
    assert a1[0][0].codes == shards[0][0].data_ptr() and a1[0][2].scales == shards[2][1].data_ptr()
    assert any(t is out for t in call._keep)


def _rates_table():
    """kFusedUs and kSenderUs parsed from the committed rates.inc."""
    import numpy as np
    path = os.path.join(os.path.dirname(fc.fcomm.__file__), "csrc", "rates.inc")
    text = open(path).read()
    tabs = {}
    for name in ("kFusedUs", "kSenderUs"):
        body = text.split(name + "[6][3][2][15] = {", 1)[1].split("};", 1)[0]
        vals = [float(v) for v in re.findall(r"[-+]?\d+\.\d+", body)]
        tabs[name] = np.array(vals).reshape(6, 3, 2, 15)
    return tabs


def test_protocol_estimate_reads_the_measured_table():
    """At measured points the estimate is the table's fused + sender time;
    between sizes it lies between its neighbours; above 256 MB it grows in
    proportion to the bytes; P between 4 and 8 interpolates linearly."""
    t = _rates_table()
    specs = [fc.BF16, fc.BF16_TAGGED, fc.INT8_G128, fc.INT8_G128_TAGGED, fc.INT4_G32,
             fc.INT4_G32_TAGGED]
    for f, spec in enumerate(specs):
        for pi, P in enumerate((2, 4, 8)):
            for hi, H in enumerate((4096, 8192)):
                for m in (0, 6, 14):
                    rows = ((16 << 10) << m) // (2 * H)
                    if rows == 0:
                        continue
                    want = t["kFusedUs"][f, pi, hi, m] + t["kSenderUs"][f, pi, hi, m]
                    assert abs(fc.protocol_estimate(rows, H, P, spec) - want) < 1e-6 * want + 1e-9
        # between 1 MB and 2 MB (H = 8192: 64 and 128 rows)
        lo = fc.protocol_estimate(64, 8192, 4, spec)
        hi_ = fc.protocol_estimate(128, 8192, 4, spec)
        mid = fc.protocol_estimate(96, 8192, 4, spec)
        assert min(lo, hi_) - 1e-9 <= mid <= max(lo, hi_) + 1e-9
        big = fc.protocol_estimate(16384, 8192, 8, spec)
        assert abs(fc.protocol_estimate(32768, 8192, 8, spec) - 2 * big) < 1e-6 * big
        e4, e8 = fc.protocol_estimate(1024, 8192, 4, spec), fc.protocol_estimate(1024, 8192, 8, spec)
        assert abs(fc.protocol_estimate(1024, 8192, 6, spec) - (e4 + e8) / 2) < 1e-6 * e8
    with pytest.raises(fc.FcommError):
        fc.protocol_estimate(64, 8192, 4, fc.QSpec(fc.FMT_INT8_SYM, 64))
