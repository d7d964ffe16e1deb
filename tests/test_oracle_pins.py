"""The fp64 oracle against what the definition of attention fixes (closed
forms, library routines, invariants).  CPU only."""
import pytest

from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(oracle_mod, check):
    check(oracle_mod.attn_fwd)


def test_oracle_weights(oracle_mod):
    pins.check_weights(oracle_mod.attn_weights)


def test_rows_entry_matches_whole_head(oracle_mod):
    """The row-sampling entry point computes the same rows as the whole-head
    one (it is how the large workloads are checked)."""
    import numpy as np
    from tiled_attention_tk_gb300.inputs import make_qkv
    q, k, v = make_qkv(1, 1, 300, 64, 17)
    rows = [0, 1, 127, 128, 129, 255, 299]
    for causal in (False, True):
        O, L = oracle_mod.attn_fwd(q, k, v, causal, 0.125)
        Or, Lr = oracle_mod.attn_fwd_rows(q[0, 0], k[0, 0], v[0, 0], rows, causal, 0.125)
        assert np.array_equal(Or, O[0, 0, rows])
        assert np.array_equal(Lr, L[0, 0, rows])
    # 130 queries at the end of 300 keys
    qs = q[:, :, :130].contiguous()
    rows = [0, 1, 127, 128, 129]
    for causal in (False, True):
        O, L = oracle_mod.attn_fwd(qs, k, v, causal, 0.125)
        Or, Lr = oracle_mod.attn_fwd_rows(qs[0, 0], k[0, 0], v[0, 0], rows, causal, 0.125)
        assert np.array_equal(Or, O[0, 0, rows])
        assert np.array_equal(Lr, L[0, 0, rows])


def test_thread_count_does_not_change_results(oracle_mod):
    import numpy as np
    from tiled_attention_tk_gb300.inputs import make_qkv
    q, k, v = make_qkv(2, 2, 65, 32, 23)
    O1, L1 = oracle_mod.attn_fwd(q, k, v, True, 0.2, threads=1)
    assert oracle_mod.last_threads() == 1
    O4, L4 = oracle_mod.attn_fwd(q, k, v, True, 0.2, threads=4)
    assert np.array_equal(O1, O4) and np.array_equal(L1, L4)


def test_oracle_rejects_bad_arguments(oracle_mod):
    import numpy as np
    z = np.zeros((1, 1, 4, 8), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.attn_fwd(z, z, np.zeros((1, 1, 5, 8), dtype=np.uint16), False, 1.0)
    with pytest.raises(RuntimeError):
        oracle_mod.attn_fwd_rows(z[0, 0], z[0, 0], z[0, 0], [4], False, 1.0)
    # causal with fewer keys than queries: some query would see no key
    with pytest.raises(RuntimeError):
        oracle_mod.attn_fwd(z, z[:, :, :3].copy(), z[:, :, :3].copy(), True, 1.0)
    oracle_mod.attn_fwd(z, z[:, :, :3].copy(), z[:, :, :3].copy(), False, 1.0)


def test_oracle_regression_fixture(oracle_mod):
    """The oracle still gives the values frozen in tests/golden (written by
    tests/golden/make_golden.py from the oracle alone) up to a few ulps,
    which a different libm may move."""
    import json
    import os
    import numpy as np
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_regression.json")
    doc = json.load(open(path))
    shape = tuple(doc["shape"])
    q, k, v = (np.array(doc[n], dtype=np.uint16).reshape(shape)
               for n in ("q_bits", "k_bits", "v_bits"))
    for case in doc["cases"]:
        O, L = oracle_mod.attn_fwd(q, k, v, case["causal"], case["scale"])
        O_ref = np.array([float(x) for x in case["O"]]).reshape(O.shape)
        L_ref = np.array([float(x) for x in case["LSE"]]).reshape(L.shape)
        assert np.max(np.abs(O - O_ref)) <= 1e-13
        assert np.max(np.abs(L - L_ref)) <= 1e-13


from tests import oracle_bwd_pins as bwd_pins  # noqa: E402


@pytest.mark.parametrize("check", bwd_pins.ALL_BWD_CHECKS, ids=lambda c: c.__name__)
def test_oracle_bwd_pin(oracle_mod, check):
    check(oracle_mod.attn_bwd)


def test_oracle_bwd_thread_count(oracle_mod):
    import numpy as np
    from tiled_attention_tk_gb300.inputs import make_qkv
    q, k, v = make_qkv(1, 2, 40, 16, 51)
    do = make_qkv(1, 2, 40, 16, 52)[0]
    a = oracle_mod.attn_bwd(q, k, v, do, True, 0.25, threads=1)
    b = oracle_mod.attn_bwd(q, k, v, do, True, 0.25, threads=3)
    for x, y in zip(a, b):
        assert np.max(np.abs(x - y)) <= 1e-13


from tests import oracle_gemm_pins as gemm_pins  # noqa: E402


@pytest.mark.parametrize("check", gemm_pins.GEMM_CHECKS, ids=lambda c: c.__name__)
def test_oracle_gemm_pin(oracle_mod, check):
    check(oracle_mod.gemm)


from tests import oracle_based_pins as based_pins  # noqa: E402


@pytest.mark.parametrize("check", based_pins.BASED_CHECKS, ids=lambda c: c.__name__)
def test_oracle_based_pin(oracle_mod, check):
    check(oracle_mod.based)


from tests import oracle_hedgehog_pins as hh_pins  # noqa: E402


@pytest.mark.parametrize("check", hh_pins.HEDGEHOG_CHECKS, ids=lambda c: c.__name__)
def test_oracle_hedgehog_pin(oracle_mod, check):
    check(oracle_mod.hedgehog)
