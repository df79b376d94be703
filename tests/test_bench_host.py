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
        gbs, dt, rows = bench.oracle_sample(w, inp, 0.01, threads=threads)
        assert gbs > 0 and dt > 0 and 1 <= rows <= w.T
    assert bench.host_cores() >= 1
