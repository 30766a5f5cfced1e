"""bench.py's accuracy report (INT2 g32 against INT4 g64 on the same seeds):
every sampled row of the CUDA path within the parity tolerances of the
oracle's stored answers, on inputs whose fingerprints match the stored ones."""
from __future__ import annotations

import pytest

from tests.gpu_common import MASS_TOL, O_TOL

pytestmark = pytest.mark.gpu


def test_accuracy_report_within_tolerance():
    import torch

    import bench
    from quantized_kv_cache_quantize_gb300 import synth

    rep = bench.accuracy_report(synth.inputs(synth.WORKLOADS["w4_int2"]), torch.device("cuda", 0),
                                reps=2)
    for name in bench.ACCURACY_WORKLOADS:
        e = rep[name]
        assert e["inputs_match_refs"], name
        for corr in ("none", "taylor", "exact"):
            assert e[corr]["err_o"] <= O_TOL, (name, corr, e[corr])
            assert e[corr]["err_ps"] <= MASS_TOL and e[corr]["err_pr"] <= MASS_TOL, (name, corr, e[corr])
        assert e["attention_tflops"] > 0
