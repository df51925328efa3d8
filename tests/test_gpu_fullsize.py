"""CUDA path vs oracle at the workloads' full sizes (all layers, all decode steps, the
launch configuration the benchmark times): selection and decode on at least 8
sampled units per workload, the stored codes and window of every kv head of every
layer (a subset of layers for the quantize-only workload) bit-exact."""
import pytest

import synth
from _fullsize import run_fullsize

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wid", [2, 3, 4, 5])
def test_fullsize_sampled_units(wid):
    spec = synth.workload(wid)
    rep = run_fullsize(spec, steps=spec.steps, n_samples=8, seed=wid)
    print(f"workload {wid} ({spec.name}): sampled={rep.units} store_units={rep.store_units} "
          f"excused={rep.excused} rebuilt={rep.rebuilt_units} codes={rep.codes_compared} "
          f"decode_err={rep.decode_err:.2e} score_err={rep.score_err:.2e} "
          f"checked={rep.decode_checked}")
    assert rep.decode_checked > 0
