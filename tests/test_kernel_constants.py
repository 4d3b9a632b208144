"""Constants of the CUDA kernels that come from a derivation committed beside
them: checked against that derivation on the CPU (no GPU)."""
import os

import numpy as np
import pytest


def test_bf16_erfc_coefficients_match_their_fit():
    """The degree-5 erfc polynomial the bf16 GeLU kernels use (ZR_ERFC_SHORT_P,
    shared by the scalar and the packed forms) is the one
    csrc/erfc_fit.py derives (least squares on Chebyshev nodes), and its
    measured relative error stays below 2^-16."""
    pytest.importorskip("scipy")
    import importlib.util
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    csrc = os.path.join(root, "broadcast_elementwise_shape_gb300", "csrc")
    spec = importlib.util.spec_from_file_location("erfc_fit", os.path.join(csrc, "erfc_fit.py"))
    fit = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(fit)
    coef = fit.fit()[::-1]  # highest power first
    src = open(os.path.join(csrc, "zr_kernels.cuh")).read()
    body = src[src.index("#define ZR_ERFC_SHORT_P"):]
    body = body[:body.index("__device__")]
    lits = [float(np.float32(v)) for v in re.findall(r"(-?\d+\.\d+)f", body)]
    assert lits == [float(c) for c in coef]
    t = np.linspace(fit.T_MIN, 1.0, 20001)
    err = np.max(np.abs(fit.horner32(np.asarray(coef[::-1], np.float32), t) - fit.target(t)))
    assert err < 2.0 ** -16
