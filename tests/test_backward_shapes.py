"""CPU check of the backward parity shapes: each is a valid layer for the
library's config check, and the oracle's backward runs on its seeded inputs
with gradients of the right shapes and finite values, so a GPU run never
meets a shape its reference cannot handle."""
import numpy as np
import pytest

import mixture_experts_routed_gb300 as moe
import oracle
from backward_shapes import SHAPES
from workloads import make_inputs


@pytest.mark.parametrize("name", list(SHAPES))
def test_backward_shape_is_valid_and_differentiable(name):
    cfg = SHAPES[name]
    assert moe.check_config(cfg) == 0
    host = oracle.inputs_to_numpy(make_inputs(cfg))
    fwd = oracle.forward(cfg, host)
    g = oracle.backward(cfg, host, fwd, np.ones((cfg.T, cfg.d)))
    for key, shape in (("dx", (cfg.T, cfg.d)), ("dWg", (cfg.d, cfg.E)), ("dbias", (cfg.E,)),
                       ("dW1", (cfg.E, cfg.d, cfg.f)), ("dW2", (cfg.E, cfg.f, cfg.d))):
        assert g[key].shape == shape, key
        assert np.all(np.isfinite(g[key])), key
