"""The OpenMP build of the oracle (used only to time the CPU baseline on
every host core) gives the single-threaded build's results bit for bit: it
shares out loops over independent output elements, and each element keeps
its own plain summation order."""

from fractions import Fraction

import numpy as np
import pytest

import dv_inputs
import oracle
from oracle import build as oracle_build

RAGGED = dv_inputs.LayerConfig("ragged_f16", 264, 5, 32, 1000, 24, 37, 3, "f16",
                               Fraction(1, 7), k_heads_fixed=3)


@pytest.fixture(scope="module", autouse=True)
def _omp_build():
    if oracle_build.build_omp() is None:
        pytest.skip("no OpenMP in this compiler")


@pytest.mark.parametrize("cfg,B", [(dv_inputs.CONFIGS["tiny"], 1),
                                   (dv_inputs.CONFIGS["tiny"].with_(dtype="f16"), 3),
                                   (RAGGED, 3)])
@pytest.mark.parametrize("threads", [3, 4])
def test_threaded_oracle_is_bit_identical(cfg, B, threads):
    w = oracle.numpy_weights(dv_inputs.make_weights(cfg, 2, "cpu", norm_affine=True))
    kc, vc = dv_inputs.make_kv(cfg, B, 2, "cpu")
    x = dv_inputs.make_x(cfg, B, 2, "cpu").numpy()
    xp = dv_inputs.make_x(cfg, B, 3, "cpu").numpy()
    D = oracle.desc_from_config(cfg)
    args = (D, w, x, cfg.k_heads, cfg.k_neurons, kc.numpy(), vc.numpy(), cfg.kv_len)
    r1 = oracle.layer_decode(*args, x_pred=xp)
    rt = oracle.layer_decode(*args, x_pred=xp, threads=threads)
    assert oracle.threads_used(threads) == threads
    for key in ("s_h", "s_n", "idx_h", "idx_n", "u_h", "u_n", "h1", "y", "k_cache", "v_cache"):
        assert np.array_equal(r1[key], rt[key]), key
