"""The causal conv1d update (gdn_causal_conv1d_update; torch-to-nnef page,
CausalConvUpdateReified) against the fp64 oracle, element by element.

Tolerances: per tensor max|x - y| / max|y|, 1e-5 for fp32 (a K-term fp32 sum
and one SiLU) and 2e-2 for bf16 inputs (the output is rounded to bf16); the
carried state is a copy of input samples and must match exactly.
"""

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_06_gb300 import workloads as wl
from parity_util import check, np64

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_delta_rule_06_gb300 import build

    build.build()


def _run(B, C, S, K, dtype, seed, in_place=False):
    from gated_delta_rule_06_gb300 import ops

    x = wl.make_conv_inputs(B, C, S, K, dtype, seed)
    xd = {n: t.cuda() for n, t in x.items()}
    st = xd["conv_state"].clone()
    out, fs = ops.causal_conv1d_update(xd["hidden"], st, xd["weight"],
                                       final_state=st if in_place else None)
    torch.cuda.synchronize()
    o_r, f_r = oracle.causal_conv1d_update(x["hidden"], x["conv_state"], x["weight"])
    check("out", out, o_r, TOL[dtype])
    np.testing.assert_array_equal(np64(fs), f_r)
    if in_place:
        assert fs.data_ptr() == st.data_ptr()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("S,K", [(1, 4), (1, 1), (7, 4), (130, 3), (5, 16), (2, 9)])
def test_conv1d_update(S, K, dtype):
    _run(3, 200, S, K, dtype, seed=S * 31 + K)


def test_conv1d_update_in_place_decode_width():
    """Decode shape of the 9B layer's mixed projection (C = 2 * 16 * 128 + 32 * 128),
    B = 64, S = 1, K = 4, state updated in place."""
    _run(64, 2 * 16 * 128 + 32 * 128, 1, 4, torch.bfloat16, seed=5, in_place=True)


def test_conv1d_rejects_bad_shapes():
    from gated_delta_rule_06_gb300 import ops

    x = wl.make_conv_inputs(1, 8, 1, 17, torch.float32, 1)
    xd = {n: t.cuda() for n, t in x.items()}
    with pytest.raises(ops.GdnError):
        ops.causal_conv1d_update(xd["hidden"], xd["conv_state"], xd["weight"])
