"""The softmax loops compute a fixed share of their exponentials with a
polynomial on the FMA pipes instead of the MUFU instruction.  Its accuracy is
checked here against fp64 exp2 (and the MUFU instruction's own results) on
the range the kernels feed it: arguments x = s * scale * log2(e) - reference
that are at most a few units above 0 and down to -inf for masked entries."""
import numpy as np
import pytest
import torch

import prefix_tree_block_gb300 as pt
from parity import ensure_built

pytestmark = pytest.mark.gpu

POLY_REL = 1e-4  # design bound 7.8e-5 (degree-3 minimax of 2^f on [-1/2, 1/2])


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _inputs():
    rng = np.random.default_rng(11)
    x = rng.uniform(-125.0, 8.0, 1 << 20).astype(np.float32)
    edges = np.array([0.0, -0.0, 1e-7, -1e-7, 0.5, -0.5, 0.4999999, -0.5000001, 1.0, -1.0, 7.9, -124.9, -125.0],
                     np.float32)
    return np.concatenate([x, edges])


def test_poly_exp2_relative_error():
    x = _inputs()
    y = pt.debug_exp2(torch.from_numpy(x).cuda(), 1).cpu().numpy().astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1.0)
    assert rel.max() <= POLY_REL, f"max relative error {rel.max():.3e} at x={x[rel.argmax()]}"


def test_poly_exp2_underflow_and_masked():
    x = np.array([-125.01, -125.5, -126.0, -126.4, -126.6, -127.0, -127.5, -130.0, -200.0, -1e30, -np.inf], np.float32)
    y = pt.debug_exp2(torch.from_numpy(x).cuda(), 1).cpu().numpy()
    assert np.all(np.isfinite(y)) and np.all(y >= 0.0) and np.all(y <= 2.0 ** -124)


def test_poly_agrees_with_mufu():
    x = _inputs()
    xt = torch.from_numpy(x).cuda()
    ym = pt.debug_exp2(xt, 0).cpu().numpy().astype(np.float64)
    yp = pt.debug_exp2(xt, 1).cpu().numpy().astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.abs(ym / ref - 1.0).max() <= 1e-5  # the MUFU instruction itself
    assert np.abs(yp / ym - 1.0).max() <= POLY_REL + 1e-5


def test_debug_exp2_rejects_bad_method():
    lib = pt.load_library()
    assert lib.pt_debug_exp2(None, None, 0, 2, None) == pt.PT_ERR_INVALID_ARG
