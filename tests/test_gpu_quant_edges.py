"""Group quantization at the edges of its arithmetic, CUDA path vs oracle, bit for bit.

The quantizer forms each code's quotient without a divide instruction when a
group's S and Z are finite and its quotients stay small, adds no clamp when every
code of the block lies in [0, 2^b - 1], and otherwise takes the clamped or the
exact (divide) path. Workload data never leave the first case, so these groups do:
  * tiny values (~1e-6, ranges down to ~2e-7): S and Z are fp16 subnormals, S
    rounds by up to half its size (or to 0), so quotients run past 2^b - 1/2 (the
    clamped path) or every code is 0;
  * constant groups: S == 0 (every code 0);
  * a range beyond fp16: one element of 3e38 makes S = +inf (the divide path:
    every other element's quotient is 0);
  * ordinary groups beside them in the same blocks.
Codes, scales, zero-points and the window are compared with the oracle."""
import numpy as np
import pytest
import torch

from _parity import Report, check_export, kvc
from oracle import OracleCache

pytestmark = pytest.mark.gpu


def _bf16(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).float().numpy()


def _rows(n_groups: int, alpha: int, d: int, rng, along_tokens: bool) -> np.ndarray:
    n = 32 * n_groups + alpha
    x = rng.standard_normal((n, d)).astype(np.float32)
    for g in range(n_groups):
        r0 = 32 * g
        if along_tokens:       # key groups: one channel over the group's 32 tokens
            x[r0:r0 + 32, 0:24] = 1e-6 * (1 + rng.random((32, 24)))            # tiny
            x[r0:r0 + 32, 24:32] = 5e-7 + 2.4e-7 * rng.random((32, 8))         # tinier
            x[r0:r0 + 32, 40:48] = np.float32(0.375)                             # constant
            if g == 0:
                x[r0:r0 + 32, 56:64] = 1000 * rng.standard_normal((32, 8))
                x[r0 + 5, 56:64] = 3e38                                           # S = inf
        else:                  # value groups: one token over 32 channels
            x[r0:r0 + 8, 0:32] = 1e-6 * (1 + rng.random((8, 32)))
            x[r0 + 8:r0 + 12, 32:64] = 5e-7 + 2.4e-7 * rng.random((4, 32))
            x[r0 + 12:r0 + 16, 64:96] = np.float32(-1.25)
            if g == 0:
                x[r0 + 16:r0 + 18, 96:128] = 1000 * rng.standard_normal((2, 32))
                x[r0 + 16, 100] = 3e38
                x[r0 + 17, 127] = 3e38
    return _bf16(x)


@pytest.mark.parametrize("bits", [2, 4])
def test_edge_groups_match_oracle(bits):
    K = kvc()
    d, n_groups, alpha, window = 128, 3, 16, 32
    rng = np.random.default_rng(77 + bits)
    k = _rows(n_groups, alpha, d, rng, True)
    v = _rows(n_groups, alpha, d, rng, False)
    n = k.shape[0]
    assert np.isfinite(k).all() and np.isfinite(v).all()
    kb = torch.from_numpy(k).to(torch.bfloat16)[None, None]
    vb = torch.from_numpy(v).to(torch.bfloat16)[None, None]
    dims = K.make_dims(1, 1, 1, 1, d, n, alpha, 7, bits, 32, window, 1)
    budgets = K.kvc_plan_budgets(dims, "none", 0)
    cache = K.kvc_prefill_compress(dims, budgets, 0, None, kb.cuda(), vb.cuda())
    ex = K.kvc_export_layer(cache, 0)
    torch.cuda.synchronize()
    oc = OracleCache(1, 1, 1, d, bits, 32, window)
    with np.errstate(over="ignore", invalid="ignore"):
        oc.prefill(kb.double().numpy(), vb.double().numpy(), alpha, budget=None, q_obs=None,
                   pool_kernel=7)
    st = oc.heads[0][0]
    # the edge cases are present: subnormal and infinite scales, zero scales
    for S in (st.kS, st.vS):
        s = S.astype(np.float32)
        assert np.isinf(s).any() and (s == 0).any()
        assert ((s > 0) & (s < np.float32(6.103515625e-05))).any()
    rep = Report()
    check_export(ex, oc, [(0, 0)], rep)
    assert rep.codes_compared == 32 * n_groups
    cache.close()
