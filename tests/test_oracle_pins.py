"""The CPU oracle checked against what the Gated DeltaNet-2 page and plain
mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
import pins


def _c(q, k, v, b, w, g, S0):
    return oracle.forward(q, k, v, b, w, g, S0, nthreads=2)


def _np(q, k, v, b, w, g, S0):
    return oracle.forward_np(q, k, v, b, w, g, S0)


IMPLS = {"c": _c, "numpy": _np}


@pytest.mark.parametrize("impl", sorted(IMPLS))
@pytest.mark.parametrize("pin", sorted(pins.PINS))
def test_pin(impl, pin):
    err = pins.PINS[pin](IMPLS[impl])
    assert err < pins.TOL, f"{impl} oracle fails pin {pin}: rel err {err:.3e}"


def test_golden_files_present():
    names = [n for n, _ in pins.golden_cases()]
    assert len(names) >= 2, names


def test_c_matches_numpy():
    rng = np.random.default_rng(7)
    for (B, T, H, dk, dv) in ((2, 33, 3, 8, 8), (1, 17, 2, 16, 4), (3, 5, 1, 3, 9)):
        p = pins.rand_problem(rng, B=B, T=T, H=H, dk=dk, dv=dv, b_hi=2.0)
        oc, Sc = _c(*p)
        on, Sn = _np(*p)
        assert pins.rel_err(oc, on) < 1e-12
        assert pins.rel_err(Sc, Sn) < 1e-12


def test_thread_count_does_not_change_result():
    rng = np.random.default_rng(8)
    p = pins.rand_problem(rng, B=3, T=20, H=5, dk=8, dv=6)
    o1, S1 = oracle.forward(*p, nthreads=1)
    o7, S7 = oracle.forward(*p, nthreads=7)
    assert np.array_equal(o1, o7) and np.array_equal(S1, S7)


def test_empty_sequence_returns_initial_state():
    rng = np.random.default_rng(9)
    q, k, v, b, w, g, S0 = pins.rand_problem(rng, B=2, T=0, H=2, dk=4, dv=4)
    o, ST = oracle.forward(q, k, v, b, w, g, S0)
    assert o.shape == (2, 0, 2, 4)
    assert np.array_equal(ST, S0)
    o, ST = oracle.forward(q, k, v, b, w, g, None)
    assert np.array_equal(ST, np.zeros_like(S0))


def test_decode_step_is_one_token_of_forward():
    rng = np.random.default_rng(10)
    q, k, v, b, w, g, S0 = pins.rand_problem(rng, B=2, T=1, H=3, dk=6, dv=5)
    o, ST = oracle.forward(q, k, v, b, w, g, S0)
    od, Sd = oracle.decode_step(q[:, 0], k[:, 0], v[:, 0], b[:, 0], w[:, 0], g[:, 0], S0)
    assert np.array_equal(od, o[:, 0]) and np.array_equal(Sd, ST)


def test_bf16_inputs_upcast_exactly():
    torch = pytest.importorskip("torch")
    x = torch.randn(3, 4).to(torch.bfloat16)
    up = oracle._f64(x)
    assert up.dtype == np.float64
    assert np.array_equal(up, x.float().numpy().astype(np.float64))


def test_bad_shapes_raise():
    rng = np.random.default_rng(11)
    q, k, v, b, w, g, S0 = pins.rand_problem(rng, B=1, T=3, H=1, dk=4, dv=4)
    with pytest.raises(ValueError):
        oracle.forward(q, k[:, :2], v, b, w, g, S0)
    with pytest.raises(ValueError):
        oracle.forward(q, k, v, b, w, g, S0[..., :3])


def test_segment_transfer_decomposition():
    """The algebra behind the chunk-parallel scan of the GPU prefill: for a
    segment of tokens, the run from S_start equals the run from zero plus the
    start state pushed through the segment's transfer, where the transfer M and
    the readout responses r_t come from the run that starts at the identity with
    no writes (w = 0):  S_end = M S_start + N  and  o_t = o_t^0 + S_start^T r_t.
    Chaining two segments this way must reproduce the unsplit run."""
    rng = np.random.default_rng(21)
    B, T, H, dk, dv, T1 = 2, 23, 2, 6, 5, 9
    q, k, v, b, w, g, S0 = pins.rand_problem(rng, B=B, T=T, H=H, dk=dk, dv=dv, b_hi=2.0)
    g = 0.05 * g   # slow decay: the start state stays visible through the segment
    o_ref, S_ref = _c(q, k, v, b, w, g, S0)
    eye = np.broadcast_to(np.eye(dk), (B, H, dk, dk)).copy()
    zeros_k = np.zeros((B, T - T1, H, dk))
    sl = slice(T1, None)
    # segment 0 from S0, segment 1 from zero and from the identity
    o0, S1 = _c(q[:, :T1], k[:, :T1], v[:, :T1], b[:, :T1], w[:, :T1], g[:, :T1], S0)
    oz, N = _c(q[:, sl], k[:, sl], v[:, sl], b[:, sl], w[:, sl], g[:, sl], None)
    r, M = _c(q[:, sl], k[:, sl], zeros_k, b[:, sl], zeros_k, g[:, sl], eye)
    S_end = np.einsum("bhij,bhjd->bhid", M, S1) + N
    o1 = oz + np.einsum("bthj,bhjd->bthd", r, S1)
    assert pins.rel_err(S_end, S_ref) < 1e-12
    assert pins.rel_err(np.concatenate([o0, o1], axis=1), o_ref) < 1e-12
    # a plausible slip -- the transposed transfer -- breaks it
    S_bad = np.einsum("bhji,bhjd->bhid", M, S1) + N
    assert pins.rel_err(S_bad, S_ref) > 1e-3
