"""The read-ceiling probe the benchmark places the score pass against
(long_context_decode_subset_b300/read_ceiling.cu): it runs, reports both of
its figures for the requested byte count, and those figures are plausible
for a read of that many bytes (neither faster than any HBM could deliver nor
absurdly slow)."""
import pytest

import bench
from long_context_decode_subset_b300 import build

pytestmark = pytest.mark.gpu


def test_read_ceiling_reports_both_figures():
    build.build_ceiling()
    nbytes = 64 << 20
    ceil = bench.read_ceiling([nbytes])
    assert ceil is not None and nbytes in ceil
    plain_us, ring_us = ceil[nbytes]
    for us in (plain_us, ring_us):
        gbs = nbytes / (us * 1e-6) / 1e9
        assert 200.0 < gbs < 10000.0, (us, gbs)
    rec = bench.ceiling_record(ceil, float(nbytes), 2.0 * min(plain_us, ring_us))
    assert rec["kernel_frac"] == 0.5

