"""Host-side pieces of bench.py that need no GPU: the oracle baseline lines
every workload reports beside its GPU number."""
import math

import bench


def test_oracle_rate_runs_every_part_once_within_zero_budget():
    rate, done, used = bench._oracle_attention_rate([(16, 40), (8, 24)], 64, budget_s=0.0)
    assert done == 2 and used > 0
    assert math.isclose(rate, 4.0 * 64 * (16 * 40 + 8 * 24) / used, rel_tol=1e-12)


def test_oracle_line_fields():
    line = bench._oracle_line(2.5e12, 3, 1.25, "a sample")
    assert line == {"value": 2.5, "unit": bench.UNIT, "cores": line["cores"], "kind": "oracle",
                    "sample": "3 heads of a sample (float64 numpy), 1.2 s",
                    "cpu_model": line["cpu_model"], "blas_threads": line["blas_threads"]}
    assert line["cores"] >= 1
    assert line["blas_threads"] is not None
    ms = bench._oracle_line(1e12, 1, 1.0, "x", value=12.5, unit="ms/layer")
    assert ms["value"] == 12.5 and ms["unit"] == "ms/layer"
