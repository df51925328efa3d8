"""CUDA path vs oracle at the workloads' full sizes (all layers, all decode steps, the
launch configuration the benchmark times), checked on seeded samples of units."""
import pytest

import synth
from _fullsize import run_fullsize

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wid", [2, 3, 4, 5])
def test_fullsize_sampled_units(wid):
    spec = synth.workload(wid)
    rep = run_fullsize(spec, steps=spec.steps, n_samples=3, seed=wid)
    print(f"workload {wid} ({spec.name}): units={rep.units} excused={rep.excused} "
          f"codes={rep.codes_compared} decode_err={rep.decode_err:.2e} "
          f"score_err={rep.score_err:.2e} checked={rep.decode_checked}")
    assert rep.decode_checked > 0
