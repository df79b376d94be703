"""CPU checks of bench.py's host-side measurement: the oracle timed on several
host threads runs it over contiguous row ranges, which must give exactly the
rows one call gives (rows are independent in every step of the path)."""
import numpy as np

import bench
from quantized_reduce_rmsnorm_gb300 import synth


def test_oracle_row_ranges_equal_one_call(orc):
    for fmt, G in ((synth.FMT_INT4_ASYM, 32), (synth.FMT_INT8_SYM, 128), (synth.FMT_BF16, 0)):
        w = synth.Workload("rows", P=3, T=13, H=512, fmt=fmt, group=G)
        inp = synth.make_inputs(w, seed=9)
        whole = orc.allreduce_residual_rmsnorm(fmt, inp["slabs"], inp["residual"], inp["gamma"],
                                               w.T, w.H, G, w.eps)
        for r0, r1 in ((0, 5), (5, 6), (6, 13)):
            part = orc.allreduce_residual_rmsnorm(fmt, [s[r0:r1] for s in inp["slabs"]],
                                                  inp["residual"][r0:r1], inp["gamma"], r1 - r0,
                                                  w.H, G, w.eps)
            assert np.array_equal(part["h"], whole["h"][r0:r1])
            assert np.array_equal(part["y"], whole["y"][r0:r1])
            if "codes" in whole:
                per_row = whole["codes"].size // w.T
                assert np.array_equal(part["codes"], whole["codes"][r0 * per_row:r1 * per_row])


def test_oracle_sample_on_threads():
    w = synth.Workload("rows", P=2, T=24, H=1024, fmt=synth.FMT_INT8_SYM, group=128)
    inp = synth.make_inputs(w, seed=2)
    for threads in (1, 3):
        gbs, dt, rows, passes = bench.oracle_sample(w, inp, 0.01, threads=threads)
        assert gbs > 0 and dt > 0 and 1 <= rows <= w.T and passes >= 1
    assert bench.host_cores() >= 1


def test_spread_is_median_and_deciles():
    med, p10, p90 = bench.spread([5.0, 1.0, 3.0, 2.0, 4.0])
    assert med == 3.0 and abs(p10 - 1.4) < 1e-12 and abs(p90 - 4.6) < 1e-12


def test_parse_size_units():
    assert bench.parse_size("16K") == 16 << 10
    assert bench.parse_size("256m") == 256 << 20
    assert bench.parse_size("1G") == 1 << 30
    assert bench.parse_size("4096") == 4096


class _Args:
    def __init__(self, sweep="full", sizes="", formats="", only=""):
        self.sweep, self.sizes, self.formats, self.only = sweep, sizes, formats, only


def test_sweep_selection_counts_and_filters():
    # 15 sizes x 2 hidden x 3 P: 90 shapes per encoding
    assert len(bench.sweep_selection(_Args())) == 90 * 3
    assert len(bench.sweep_selection(_Args(formats="bf16,int8,int4,bf16t,int8t,int4t"))) == 90 * 6
    quick = bench.sweep_selection(_Args(sweep="quick"))
    assert {p[0] for p in quick} == {16 << 10, 1 << 20, 16 << 20, 64 << 20, 256 << 20}
    sized = bench.sweep_selection(_Args(sizes="16M,32M", formats="int4"))
    assert len(sized) == 2 * 2 * 3 and all(p[4] == synth.FMT_INT4_ASYM for p in sized)
    one = bench.sweep_selection(_Args(only="64M:8192:8:int4,16K:4096:2:int8t", formats="int4,int8t"))
    assert sorted((p[0], p[1], p[3], p[4]) for p in one) == sorted(
        [(64 << 20, 8192, 8, synth.FMT_INT4_ASYM), (16 << 10, 4096, 2, synth.FMT_INT8_TAGGED)])
    for msg, H, T, P, fmt, G in bench.sweep_selection(_Args(formats="int8,int4")):
        assert T * H * 2 == msg and G == (128 if fmt == synth.FMT_INT8_SYM else 32)


def test_sweep_report_counts_points_below_the_bar(tmp_path, capsys):
    import json
    rows = []
    for msg, frac in ((16 << 20, 0.65), (64 << 20, 0.9), (256 << 20, 0.69)):
        rows.append(dict(sweep=True, message_bytes=msg, hidden=8192, tokens=msg // 16384, P=4,
                         format="int4_asym_g32", fused_us=1.0, fused_us_p10=0.9, fused_us_p90=1.1,
                         fused_frac=frac, fused_frac_nominal=frac * 0.85, fused_held_us=1.2, sets=2,
                         inputs_cold=True, sender_us=2.0, sender_us_p10=1.9, sender_us_p90=2.1,
                         sender_frac=0.8))
    p = tmp_path / "s.jsonl"
    p.write_text("noise\n" + "\n".join(json.dumps(r) for r in rows) + "\n")
    bench.sweep_report(str(p))
    out = capsys.readouterr().out
    assert out.count("| int4_asym_g32 |") == 3
    assert "2 of 3 points below 0.70" in out and "1 of 2 points below 0.70" in out
    assert "0.650 / 0.690 / 0.900" in out


def test_code_only_ignores_comments_and_blank_lines():
    a = "int f() { // one\n  return 1; /* two\n three */}\n\n"
    b = "int f() {\n\n  return 1; }   \n"
    assert bench.code_only(a) == bench.code_only(b) == "int f() {\n  return 1; }"
    assert bench.code_only("x = 1; // c\n") == "x = 1;"


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_gbs(10**9, 1, 1.0) == 1000.0
    assert bench.whole_job_gbs(10**9, 4, 2.0) == 2000.0
