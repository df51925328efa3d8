"""Group quantization at exact rounding ties, CUDA path vs oracle.

With bf16 inputs and fp16 scale / zero-point, the fp32 quotient (x - Z) / S is
either an exact half-integer or far (relative to fp32 precision) from one, so the
ties are where the code's round-half-to-even matters and where a quotient taken
through the reciprocal could differ from the IEEE division. These groups put
every non-extreme element on a tie (k + 1/2) * S, with scales of few mantissa
bits so that every value is exact in bf16, and compare codes, scales,
zero-points and the window bit for bit.
"""
import numpy as np
import pytest
import torch

from _parity import Report, check_export, kvc
from oracle import OracleCache

pytestmark = pytest.mark.gpu

SCALES = np.array([0.5, 0.625, 0.75, 0.875, 1.25, 0.15625, 0.1875, 2.5], np.float32)


def _tie_rows(n_groups: int, d: int, bits: int, along_tokens: bool, rng) -> np.ndarray:
    """[32 * n_groups, d] float32 values, every quantization group (32 tokens of
    one channel when along_tokens, else 32 channels of one token) holding its
    minimum, its maximum and 30 elements on rounding ties."""
    top = 2 ** bits - 1
    out = np.empty((32 * n_groups, d), np.float32)
    n_lines = d if along_tokens else 32 * n_groups    # one group line per channel / token
    per_line = n_groups if along_tokens else d // 32
    for line in range(n_lines):
        for gi in range(per_line):
            s0 = SCALES[(line + 3 * gi) % len(SCALES)]
            k = rng.integers(0, top, size=32).astype(np.float32)
            vals = (k + 0.5) * s0
            vals[0], vals[1] = 0.0, top * s0
            if (line + gi) % 2:
                vals -= top * s0                     # an all-negative group
            perm = rng.permutation(32)
            vals = vals[perm]
            if along_tokens:
                out[32 * gi:32 * gi + 32, line] = vals
            else:
                out[line, 32 * gi:32 * gi + 32] = vals
    exact = torch.from_numpy(out).to(torch.bfloat16).float().numpy()
    assert np.array_equal(exact, out), "tie values must be exact in bf16"
    return out


@pytest.mark.parametrize("d,bits", [(128, 2), (128, 4), (64, 2), (64, 4)])
def test_rounding_ties_match_oracle(d, bits):
    K = kvc()
    rng = np.random.default_rng(1000 + d + bits)
    n_groups, alpha, window = 3, 16, 32
    n = 32 * n_groups + alpha
    k = np.concatenate([_tie_rows(n_groups, d, bits, True, rng),
                        rng.standard_normal((alpha, d)).astype(np.float32)])
    v = np.concatenate([_tie_rows(n_groups, d, bits, False, rng),
                        rng.standard_normal((alpha, d)).astype(np.float32)])
    kb = torch.from_numpy(k).to(torch.bfloat16)[None, None]
    vb = torch.from_numpy(v).to(torch.bfloat16)[None, None]
    dims = K.make_dims(1, 1, 1, 1, d, n, alpha, 7, bits, 32, window, 1)
    budgets = K.kvc_plan_budgets(dims, "none", 0)
    assert budgets[0] >= n - alpha                   # quantize only: every token kept
    cache = K.kvc_prefill_compress(dims, budgets, 0, None, kb.cuda(), vb.cuda())
    ex = K.kvc_export_layer(cache, 0)
    torch.cuda.synchronize()
    oc = OracleCache(1, 1, 1, d, bits, 32, window)
    oc.prefill(kb.double().numpy(), vb.double().numpy(), alpha, budget=None, q_obs=None,
               pool_kernel=7)
    rep = Report()
    check_export(ex, oc, [(0, 0)], rep)
    assert rep.codes_compared == 32 * n_groups
    cache.close()
