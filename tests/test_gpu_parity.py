"""GPU path vs the CPU oracle, through the C ABI, on seeded inputs.

Tolerances: apply_A and precond within 1e-12 relative max-norm; the PCG
solution within 1e-8 relative 2-norm at equal iteration count; iteration
counts to the 1e-10 residual within +-1.
"""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import matrix_free_pcg_gb300 as mf  # noqa: E402

DEV = torch.device("cuda:0")
OP_TOL = 1e-12
SOL_TOL = 1e-8


def rel_maxdiff(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def case(nx, ny, nz, varying, graded, a_v=1e3, seed=0):
    h = W.layer_thickness(nz, graded)
    ah = W.horizontal_coefficient(nx, ny, varying)
    prob = oracle.Problem(nx, ny, nz, ah=ah, a_v=a_v, mass=1.0, h=h)
    kw = dict(a_h_field=ah if varying else None, a_h=1.0, a_v=a_v, mass=1.0, dz=h)
    return prob, kw, np.random.default_rng(seed).uniform(-1, 1, nx * ny * nz)


SHAPES = [
    (37, 29, 16, True, True),     # 1073 columns: 33 full tiles + a ragged one
    (37, 29, 16, False, False),
    (33, 5, 7, True, True),       # odd nz: scalar path
    (64, 48, 64, False, True),
    (17, 19, 130, True, True),    # nz not a multiple of 16
    (5, 3, 1, False, False),      # single level
    (1, 1, 3, True, True),        # one column, self-neighbour in i and j
    (3, 1, 2, False, True),
    (2, 2, 4, True, False),
    (7, 5, 500, True, False),     # too tall for the staged tile: direct path
    # nz = 32, 64, 128 with 16-byte aligned vectors: the standalone solve
    # keeps its forward pass in tensor memory
    (37, 29, 32, True, True),     # ragged last tile
    (40, 9, 128, True, True),     # 360 columns: 11 full tiles + 8 columns
    (20, 20, 64, False, False),
    (256, 256, 32, True, True),   # 2048 tiles: more than one per warp of the grid
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:3])) +
                         ("v" if s[3] else "c") + ("g" if s[4] else "u"))
def test_apply_A_matches_oracle(shape):
    prob, kw, x = case(*shape)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        y = s.apply_A(torch.from_numpy(x).to(DEV)).cpu().numpy()
    assert rel_maxdiff(y, oracle.apply_A(prob, x)) <= OP_TOL


@pytest.mark.parametrize("tmem", [True, False], ids=["tmem", "global_w"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:3])) +
                         ("v" if s[3] else "c") + ("g" if s[4] else "u"))
def test_precond_matches_oracle(shape, tmem):
    # both column-solve kernel families: w in tensor memory (where it
    # applies) and w in global memory
    prob, kw, r = case(*shape)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        mf.pcg_test_tensor_memory(s.ctx, tmem)
        z = s.precond(torch.from_numpy(r).to(DEV)).cpu().numpy()
    assert rel_maxdiff(z, oracle.precond(prob, r)) <= OP_TOL


def test_unaligned_pointers_take_the_scalar_path():
    prob, kw, x = case(16, 12, 8, True, True)
    n = prob.n
    buf_x = torch.zeros(n + 1, dtype=torch.float64, device=DEV)
    buf_y = torch.zeros(n + 1, dtype=torch.float64, device=DEV)
    xv, yv = buf_x[1:], buf_y[1:]          # 8-byte aligned views
    xv.copy_(torch.from_numpy(x))
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        s.apply_A(xv, yv)
        z = s.precond(xv, buf_y[1:]).cpu().numpy()
        y2 = s.apply_A(xv).cpu().numpy()
    assert rel_maxdiff(y2, oracle.apply_A(prob, x)) <= OP_TOL
    assert rel_maxdiff(z, oracle.precond(prob, x)) <= OP_TOL


SOLVE_CASES = [
    (37, 29, 16, True, True, 1e3),
    (33, 5, 7, True, True, 1e2),
    (40, 36, 64, False, True, 1e4),
    (17, 19, 130, True, True, 1e5),
    (6, 5, 500, False, False, 1e3),
    (45, 26, 32, True, True, 1e4),   # the column layout's tensor-memory sweep at nz = 32
]


def configure(s, mode):
    """mode: "column"; "tiled" (Thomas column solves, stored factors, batched
    loop); "tiled_recompute" (Thomas, factors rebuilt per sweep);
    "tiled_split" (substructured column solves, blocks chosen automatically);
    "tiled_persistent" (Thomas, stored factors, one cooperative kernel);
    "column_global_w" (the column layout without tensor memory).
    The row-tiled modes form A z as r + (A - M) z wherever that applies (the
    default); a "_stencil" suffix selects the full 7-point stencil."""
    stencil = mode.endswith("_stencil")
    mode = mode[: -len("_stencil")] if stencil else mode
    # "column_global_w": the column layout with its preconditioner sweep on the
    # kernels that keep w in global memory instead of tensor memory
    mf.pcg_test_tensor_memory(s.ctx, mode != "column_global_w")
    mode = "column" if mode == "column_global_w" else mode
    s.set_layout("column" if mode == "column" else "tiled")
    s.set_factors("recompute" if mode == "tiled_recompute" else "stored")
    s.set_loop("persistent" if mode == "tiled_persistent" else "batched")
    s.set_substructuring(0 if mode == "tiled_split" else 1)
    s.set_az_form("stencil" if stencil else "auto")
    if mode == "tiled_persistent":
        assert s.loop == "persistent"
    # the residual form needs Thomas column solves (no substructuring)
    thomas = s.substructuring == 1
    assert s.az_form == ("residual" if thomas and not stencil else "stencil")


MODES = ["column", "column_stencil", "column_global_w", "tiled", "tiled_stencil",
         "tiled_recompute", "tiled_split", "tiled_persistent", "tiled_persistent_stencil"]


@pytest.mark.parametrize("layout", MODES)
@pytest.mark.parametrize("cfg", SOLVE_CASES, ids=lambda c: "x".join(map(str, c[:3])))
def test_solve_matches_oracle(cfg, layout):
    nx, ny, nz, varying, graded, a_v = cfg
    prob, kw, b = case(nx, ny, nz, varying, graded, a_v=a_v, seed=3)
    x_ref, it_ref, hist_ref, st_ref = oracle.pcg(prob, b, rtol=1e-10, maxit=500)
    assert st_ref == oracle.OK
    with mf.Solver(nx, ny, nz, **kw) as s:
        configure(s, layout)
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        iters, hist, st = s.solve(bd, x, rtol=1e-10, maxit=500)
        assert st == mf.PCG_OK
        assert abs(iters - it_ref) <= 1
        np.testing.assert_allclose(hist[: min(iters, it_ref) + 1],
                                   hist_ref[: min(iters, it_ref) + 1], rtol=1e-6, atol=1e-13)
        # compare the iterates at the oracle's iteration count
        x.zero_()
        it2, _, st2 = s.solve(bd, x, rtol=0.0, maxit=it_ref)
        assert (it2, st2) == (it_ref, mf.PCG_OK)
        xs = x.cpu().numpy()
    assert np.linalg.norm(xs - x_ref) <= SOL_TOL * np.linalg.norm(x_ref)


@pytest.mark.parametrize("layout", MODES)
def test_solve_is_bitwise_repeatable(layout):
    prob, kw, b = case(40, 36, 64, True, True, a_v=1e4, seed=5)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        configure(s, layout)
        bd = torch.from_numpy(b).to(DEV)
        x1, x2 = torch.zeros_like(bd), torch.zeros_like(bd)
        i1, h1, _ = s.solve(bd, x1, rtol=1e-10)
        i2, h2, _ = s.solve(bd, x2, rtol=1e-10)
    assert i1 == i2
    assert np.array_equal(h1, h2)
    assert torch.equal(x1, x2)


UPDATE_SOLVE_CASES = [
    # nx, ny, nz, varying, graded, a_v, solver set-up
    (30, 20, 32, True, True, 1e3, "default"),
    (37, 29, 16, False, False, 1e2, "default"),     # cluster loop
    (64, 48, 64, True, True, 1e4, "column"),
    (40, 36, 33, True, True, 1e4, "multigrid"),
    (96, 80, 24, True, True, 1e3, "persistent"),
]


def _setup(s, how):
    if how == "column":
        s.set_layout("column")
    elif how == "multigrid":
        s.set_preconditioner("multigrid")
    elif how == "persistent":
        s.set_loop("persistent")


@pytest.mark.parametrize("cfg", UPDATE_SOLVE_CASES, ids=lambda c: "x".join(map(str, c[:3])) +
                         "-" + c[6])
def test_update_solve_host_equals_update_then_solve(cfg):
    # the one-call form (b copied in on a second stream while the set-up of
    # the new coefficients runs) gives the two-call form's results bit for
    # bit, and the oracle's for the new coefficients
    nx, ny, nz, varying, graded, a_v, how = cfg
    prob, kw, b = case(nx, ny, nz, varying, graded, a_v=a_v, seed=31)
    ah2 = prob.ah * 1.5 if varying else 0.75
    kw2 = dict(kw, a_h_field=ah2 if varying else None, a_h=1.0 if varying else ah2,
               a_v=2.0 * a_v, mass=0.5)
    prob2 = oracle.Problem(nx, ny, nz, ah=ah2, a_v=2.0 * a_v, mass=0.5, h=prob.h)
    bh = torch.from_numpy(b).pin_memory()
    with mf.Solver(nx, ny, nz, **kw) as s:
        _setup(s, how)
        x1 = torch.full((prob.n,), float("nan"), dtype=torch.float64).pin_memory()
        i1, h1, st1 = s.update_solve_host(bh, x1, rtol=1e-10, x0=None, **kw2)
        x2 = np.full(prob.n, np.nan)                # pageable output and input
        i2, h2, st2 = s.update_solve_host(b, x2, rtol=1e-10, x0=None, **kw2)
    if how == "multigrid":
        x_ref, it_ref, _, _ = oracle.mg_pcg(prob2, b, rtol=1e-10)
    else:
        x_ref, it_ref, _, _ = oracle.pcg(prob2, b, rtol=1e-10)
    with mf.Solver(nx, ny, nz, **kw) as s:
        _setup(s, how)
        s.update_coeffs(**kw2)
        x3 = np.zeros(prob.n)
        i3, h3, st3 = s.solve_host(b, x3, rtol=1e-10, x0=None)
        # the iterate at the oracle's count
        x4 = np.zeros(prob.n)
        i4, _, st4 = s.update_solve_host(b, x4, rtol=0.0, maxit=it_ref, x0=None, **kw2)
    assert st1 == st2 == st3 == mf.PCG_OK and i1 == i2 == i3
    assert np.array_equal(h1, h3) and np.array_equal(h2, h3)
    assert np.array_equal(x1.numpy(), x3) and np.array_equal(x2, x3)
    assert abs(i1 - it_ref) <= 1 and (i4, st4) == (it_ref, mf.PCG_OK)
    assert np.linalg.norm(x4 - x_ref) <= SOL_TOL * np.linalg.norm(x_ref)


@pytest.mark.parametrize("layout", ["tiled", "column"])
def test_update_solve_host_async_matches_the_synchronous_call(layout):
    # a sequence of solves whose solution copies run behind the next solve:
    # every solution, count and history bit for bit the synchronous call's,
    # with separate output buffers, with one shared buffer (the last solution
    # after the wait) and with initial guesses copied in on the second stream
    nx, ny, nz = 37, 29, 32
    prob, kw, _ = case(nx, ny, nz, True, True, a_v=1e4, seed=40)
    n = prob.n
    rng = np.random.default_rng(41)
    steps = []
    for i in range(5):
        coef = dict(kw, a_h_field=prob.ah * (1.0 + 0.1 * i), a_v=1e4 * (1 + i), mass=1.0)
        x0 = rng.standard_normal(n) if i % 2 else None
        steps.append((torch.from_numpy(rng.uniform(-1, 1, n)).pin_memory(), x0, coef))
    ref = []
    with mf.Solver(nx, ny, nz, **kw) as s:
        s.set_layout(layout)
        for bh, x0, coef in steps:
            x = torch.empty(n, dtype=torch.float64).pin_memory()
            it, h, st = s.update_solve_host(bh, x, rtol=1e-10, x0=x0, **coef)
            ref.append((it, h, st, x.numpy().copy()))
    with mf.Solver(nx, ny, nz, **kw) as s:
        s.set_layout(layout)
        outs = [torch.full((n,), float("nan"), dtype=torch.float64).pin_memory() for _ in steps]
        got = [s.update_solve_host_async(bh, x, rtol=1e-10, x0=x0, **coef)
               for (bh, x0, coef), x in zip(steps, outs)]
        s.host_wait()
        for (it, h, st), x, (it_r, h_r, st_r, x_r) in zip(got, outs, ref):
            assert (it, st) == (it_r, st_r) and np.array_equal(h, h_r)
            assert np.array_equal(x.numpy(), x_r)
        # one shared output buffer: after the wait it holds the last solution
        shared = torch.full((n,), float("nan"), dtype=torch.float64).pin_memory()
        for bh, x0, coef in steps:
            s.update_solve_host_async(bh, shared, rtol=1e-10, x0=x0, **coef)
        s.host_wait()
        assert np.array_equal(shared.numpy(), ref[-1][3])
        # a synchronous call right after asynchronous ones waits for their copies
        bh, x0, coef = steps[0]
        s.update_solve_host_async(steps[1][0], outs[1], rtol=1e-10, x0=steps[1][1], **steps[1][2])
        x = torch.empty(n, dtype=torch.float64).pin_memory()
        s.update_solve_host(bh, x, rtol=1e-10, x0=x0, **coef)
        assert np.array_equal(x.numpy(), ref[0][3])
        assert np.array_equal(outs[1].numpy(), ref[1][3])


@pytest.mark.parametrize("layout", ["tiled", "column"])
def test_update_solve_host_async_chain_from_the_last_solution(layout):
    # each solve of a sequence starts from the previous solution, passed as x0
    # while that solution's copy to the host (16 MB, page-locked) may still be
    # running: the copy-in waits for it.  A constant a_h, whose update does not
    # wait for the device, starts the copy-in at once; the outputs start as
    # NaN, so a copy-in that overtook the copy-out would show.
    nx, ny, nz = 128, 128, 128
    h = W.layer_thickness(nz, True)
    n = nx * ny * nz
    rng = np.random.default_rng(46)
    steps = [(torch.from_numpy(rng.uniform(-1, 1, n)).pin_memory(),
              dict(a_h=1.0 + 0.25 * i, a_v=1e3 * (1 + i), mass=1.0, dz=h)) for i in range(4)]
    kw = dict(a_h=1.0, a_v=1e3, mass=1.0, dz=h)

    def chain(solve):
        with mf.Solver(nx, ny, nz, **kw) as s:
            s.set_layout(layout)
            prev = torch.zeros(n, dtype=torch.float64).pin_memory()
            outs, res = [], []
            for bh, coef in steps:
                x = torch.full((n,), float("nan"), dtype=torch.float64).pin_memory()
                res.append(solve(s, bh, x, prev, coef))
                outs.append(x)
                prev = x
            s.host_wait()
        return res, [x.numpy() for x in outs]

    ref, x_ref = chain(lambda s, bh, x, x0, coef: s.update_solve_host(bh, x, rtol=1e-8, x0=x0,
                                                                      **coef))
    got, x_got = chain(lambda s, bh, x, x0, coef: s.update_solve_host_async(bh, x, rtol=1e-8,
                                                                            x0=x0, **coef))
    for (it, h_, st), (it_r, h_r, st_r), x, x_r in zip(got, ref, x_got, x_ref):
        assert st_r == mf.PCG_OK and (it, st) == (it_r, st_r) and np.array_equal(h_, h_r)
        assert np.array_equal(x, x_r)


def test_update_solve_host_initial_guess_and_errors():
    prob, kw, b = case(30, 26, 24, True, True, a_v=1e3, seed=32)
    x0 = np.random.default_rng(33).standard_normal(prob.n)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        x = np.full(prob.n, np.nan)
        it, hist, st = s.update_solve_host(b, x, rtol=1e-9, x0=x0, **kw)
        x_ref, it_ref, _, _ = oracle.pcg(prob, b, x0=x0, rtol=1e-9)
        assert st == mf.PCG_OK and abs(it - it_ref) <= 1
        assert np.linalg.norm(x - x_ref) <= 1e-7 * np.linalg.norm(x_ref)
        xio = x0.copy()                             # x0 and x the same buffer
        it2, hist2, st2 = s.update_solve_host(b, xio, rtol=1e-9, x0=xio, **kw)
        assert (it2, st2) == (it, st) and np.array_equal(xio, x) and np.array_equal(hist2, hist)
        # stopped at maxit: the last iterate comes back
        it3, _, st3 = s.update_solve_host(b, x, rtol=1e-9, maxit=3, x0=None, **kw)
        assert (it3, st3) == (3, mf.PCG_ENOTCONV) and np.all(np.isfinite(x))
        bad = b.copy()
        bad[11] = np.nan
        _, _, st4 = s.update_solve_host(bad, x, rtol=1e-9, x0=None, **kw)
        assert st4 == mf.PCG_EBREAKDOWN
        for args, kwargs in [((b, b), dict(x0=None)),          # b and x overlap
                             ((b, x), dict(x0=b))]:            # b and x0 overlap
            with pytest.raises(mf.PCGError) as e:
                s.update_solve_host(*args, rtol=1e-9, **kwargs, **kw)
            assert e.value.status == mf.PCG_EINVAL
        with pytest.raises(mf.PCGError) as e:
            s.update_solve_host(b, x, rtol=1e-9, **dict(kw, mass=0.0))
        assert e.value.status == mf.PCG_EINVAL
        # the context still solves normally afterwards
        it5, _, st5 = s.update_solve_host(b, x, rtol=1e-9, x0=x0, **kw)
        assert (it5, st5) == (it, st)
        # a zero initial guess from the host call is not carried into the next
        # device solve, whose x0 is read as usual
        s.update_solve_host(b, x, rtol=1e-9, x0=None, **kw)
        xd = torch.from_numpy(x0).to(DEV)
        it6, _, st6 = s.solve(torch.from_numpy(b).to(DEV), xd, rtol=1e-9)
        assert (it6, st6) == (it, st)
        assert np.linalg.norm(xd.cpu().numpy() - x_ref) <= 1e-7 * np.linalg.norm(x_ref)
    # a context made with a constant a_h takes no field, and solves nothing
    prob_c, kw_c, b_c = case(16, 12, 8, False, True, a_v=1e2, seed=34)
    with mf.Solver(prob_c.nx, prob_c.ny, prob_c.nz, **kw_c) as s:
        xc = np.full(prob_c.n, 7.0)
        with pytest.raises(mf.PCGError) as e:
            s.update_solve_host(b_c, xc, x0=None, **dict(kw_c, a_h_field=np.ones(16 * 12)))
        assert e.value.status == mf.PCG_EINVAL and np.all(xc == 7.0)


def test_solve_host_equals_solve_device():
    prob, kw, b = case(30, 20, 32, True, True, a_v=1e3, seed=6)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        bd = torch.from_numpy(b).to(DEV)
        xd = torch.zeros_like(bd)
        i1, h1, st1 = s.solve(bd, xd, rtol=1e-10)
        bh = torch.from_numpy(b).pin_memory()
        xh = torch.zeros(prob.n, dtype=torch.float64).pin_memory()
        i2, h2, st2 = s.solve_host(bh, xh, rtol=1e-10)
        xn = np.zeros(prob.n)                       # pageable host memory works too
        i3, _, _ = s.solve_host(b, xn, rtol=1e-10)
        # zero initial guess without a host buffer for it; the output buffer's
        # old contents (a previous solution) are not read
        i4, _, st4 = s.solve_host(bh, xh, rtol=1e-10, x0=None)
        # separate initial guess == the same guess passed in/out
        x0 = 0.5 * xh.numpy()
        xo = np.full(prob.n, np.nan)
        i5, _, st5 = s.solve_host(b, xo, rtol=1e-10, x0=x0)
        xio = x0.copy()
        i6, _, st6 = s.solve_host(b, xio, rtol=1e-10)
        with pytest.raises(mf.PCGError) as e:
            mf.pcg_solve_host_x0(s.ctx, prob.n, b, b, xn, 1e-10, 10)   # x0 overlaps b
        assert e.value.status == mf.PCG_EINVAL
    assert (i1, st1) == (i2, st2) == (i3, mf.PCG_OK) == (i4, st4)
    assert np.array_equal(xd.cpu().numpy(), xh.numpy())
    assert np.array_equal(xh.numpy(), xn)
    assert (i5, st5) == (i6, st6) and st5 == mf.PCG_OK
    assert np.array_equal(xo, xio)
    assert np.linalg.norm(xo - xn) <= 1e-8 * np.linalg.norm(xn)


@pytest.mark.parametrize("layout", ["column", "tiled", "tiled_persistent"])
def test_status_semantics_match_oracle(layout):
    prob, kw, b = case(20, 18, 16, True, True, a_v=1e3, seed=7)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        configure(s, layout)
        bd = torch.from_numpy(b).to(DEV)
        _, it_ref, _, _ = oracle.pcg(prob, b, rtol=1e-8)
        x = torch.zeros_like(bd)
        it, hist, st = s.solve(bd, x, rtol=1e-8, maxit=it_ref - 2)
        assert (it, st) == (it_ref - 2, mf.PCG_ENOTCONV)
        x.zero_()
        it, hist, st = s.solve(bd, x, rtol=0.0, maxit=3)
        assert (it, st, len(hist)) == (3, mf.PCG_OK, 4)
        x.zero_()
        it, hist, st = s.solve(torch.zeros_like(bd), x, rtol=1e-10)
        assert (it, st) == (0, mf.PCG_OK) and hist[0] == 0.0 and float(x.abs().max()) == 0.0
        x.zero_()
        it, hist, st = s.solve(bd, x, rtol=1e-10, maxit=0)
        assert (it, st) == (0, mf.PCG_ENOTCONV)
        bad = bd.clone()
        bad[123] = float("nan")
        x.zero_()
        it, hist, st = s.solve(bad, x, rtol=1e-10)
        assert st == mf.PCG_EBREAKDOWN
        assert "breakdown" in mf.pcg_last_error(s.ctx)
        # restart from a non-zero iterate: x carries the state, as in the oracle
        x0 = np.random.default_rng(11).standard_normal(prob.n)
        x.copy_(torch.from_numpy(x0))
        it, hist, st = s.solve(bd, x, rtol=1e-8)
        x_ref, it_ref, _, st_ref = oracle.pcg(prob, b, x0=x0, rtol=1e-8)
        assert st == mf.PCG_OK and abs(it - it_ref) <= 1
        assert np.linalg.norm(x.cpu().numpy() - x_ref) <= 1e-6 * np.linalg.norm(x_ref)
        with pytest.raises(mf.PCGError) as e:
            s.solve(bd, bd, rtol=1e-10)
        assert e.value.status == mf.PCG_EINVAL


def test_zero_horizontal_coupling_converges_in_one_iteration():
    nx, ny, nz = 12, 10, 24
    h = W.layer_thickness(nz, True)
    b = np.random.default_rng(9).uniform(-1, 1, nx * ny * nz)
    with mf.Solver(nx, ny, nz, a_h=0.0, a_v=1e3, mass=1.0, dz=h) as s:
        x = torch.zeros(nx * ny * nz, dtype=torch.float64, device=DEV)
        it, hist, st = s.solve(torch.from_numpy(b).to(DEV), x, rtol=1e-10)
    assert (it, st) == (1, mf.PCG_OK)


def test_update_coeffs_and_streams():
    prob, kw, x = case(24, 20, 32, True, True, a_v=1e3, seed=8)
    prob2 = oracle.Problem(prob.nx, prob.ny, prob.nz, ah=prob.ah * 2.0, a_v=5e4, mass=0.5,
                           h=prob.h)
    stream = torch.cuda.Stream()
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        s.update_coeffs(a_h_field=prob2.ah, a_v=5e4, mass=0.5, dz=prob.h)
        s.set_stream(stream)
        xd = torch.from_numpy(x).to(DEV)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            y = torch.empty_like(xd)
            s.apply_A(xd, y)
        stream.synchronize()
        assert rel_maxdiff(y.cpu().numpy(), oracle.apply_A(prob2, x)) <= OP_TOL
        # a field context may drop back to a constant a_h
        s.update_coeffs(a_h=0.7, a_v=5e4, mass=0.5, dz=prob.h)
        prob3 = oracle.Problem(prob.nx, prob.ny, prob.nz, ah=0.7, a_v=5e4, mass=0.5, h=prob.h)
        with torch.cuda.stream(stream):
            z = s.precond(xd)
        stream.synchronize()
        assert rel_maxdiff(z.cpu().numpy(), oracle.precond(prob3, x)) <= OP_TOL
    with mf.Solver(8, 8, 8, a_h=1.0, a_v=10.0) as s:
        with pytest.raises(mf.PCGError) as e:
            s.update_coeffs(a_h_field=np.ones(64), a_v=10.0)
        assert e.value.status == mf.PCG_EINVAL


@pytest.mark.parametrize("layout", ["column", "tiled"])
def test_kernel_timing_counts_launches(layout):
    prob, kw, b = case(40, 40, 64, True, True, a_v=1e4, seed=10)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        configure(s, layout)
        s.enable_timing(True)
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        it, _, _ = s.solve(bd, x, rtol=1e-10)
        t = s.kernel_times()
        info = s.launch_info()
    # one residual launch in either layout (the row-tiled one writes r, x0, p
    # and q at its own positions in it)
    assert t["residual"][1] == 1 and t["finalize"][1] == 1
    # the batched row-tiled loop runs its first iteration with the first-
    # iteration sweeps, timed under kinds of their own
    first = 1 if layout == "tiled" else 0
    assert t["precond_first"][1] == first and t["spmv_first"][1] == first
    assert t["precond_fused"][1] + first >= it + 1 and t["spmv_fused"][1] + first >= it
    # sweeps enqueued after convergence return at once and are launched but
    # not timed: at most two polling batches of 16 iterations
    worked = sum(v[1] for v in t.values())
    assert worked <= info["last_solve_launches"] <= worked + 2 * 2 * 16
    assert all(v[0] >= 0 for v in t.values())


def test_layouts_agree_and_switch_back_and_forth():
    prob, kw, b = case(45, 33, 64, True, True, a_v=1e4, seed=12)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        s.set_substructuring(1)  # Thomas column solves in both layouts
        s.set_az_form("stencil")  # and the same arithmetic for A z
        bd = torch.from_numpy(b).to(DEV)
        xs = {}
        for layout in ["tiled", "column", "tiled"]:
            s.set_layout(layout)
            x = torch.zeros_like(bd)
            it, hist, st = s.solve(bd, x, rtol=0.0, maxit=12)
            assert (it, st) == (12, mf.PCG_OK)
            xs.setdefault(layout, []).append(x.cpu().numpy())
        with pytest.raises(mf.PCGError):
            mf.pcg_set_layout(s.ctx, 7)
    assert np.array_equal(xs["tiled"][0], xs["tiled"][1])
    xc, xt = xs["column"][0], xs["tiled"][0]
    assert np.linalg.norm(xt - xc) <= 1e-12 * np.linalg.norm(xc)


@pytest.mark.parametrize("form", ["residual", "stencil"])
@pytest.mark.parametrize("cfg", [c for c in SOLVE_CASES if c[3]], ids=lambda c: "x".join(map(str, c[:3])))
def test_recomputed_factors_give_the_stored_iterates_bit_for_bit(cfg, form):
    # the sweeps rebuild the diagonal, the weights and the Thomas factors with
    # the set-up's rounding, so nothing but the data source differs
    nx, ny, nz, varying, graded, a_v = cfg
    prob, kw, b = case(nx, ny, nz, varying, graded, a_v=a_v, seed=7)
    with mf.Solver(nx, ny, nz, **kw) as s:
        s.set_loop("batched")  # the same loop (and reduction trees) for both
        s.set_substructuring(1)
        s.set_az_form(form)
        assert s.az_form == form
        bd = torch.from_numpy(b).to(DEV)
        out = {}
        for mode in ["stored", "recompute", "stored"]:
            s.set_factors(mode)
            x = torch.zeros_like(bd)
            it, hist, st = s.solve(bd, x, rtol=1e-10, maxit=500)
            assert st == mf.PCG_OK
            out.setdefault(mode, []).append((it, hist, x.cpu().numpy()))
    (i0, h0, x0), (i2, h2, x2) = out["stored"]
    (i1, h1, x1), = out["recompute"]
    assert i0 == i1 == i2
    assert np.array_equal(h0, h1) and np.array_equal(h0, h2)
    assert np.array_equal(x0, x1) and np.array_equal(x0, x2)


@pytest.mark.parametrize("loop", ["batched", "persistent"])
@pytest.mark.parametrize("cfg", SOLVE_CASES, ids=lambda c: "x".join(map(str, c[:3])))
def test_residual_form_of_Az_agrees_with_the_stencil(cfg, loop):
    # A z = r + (A - M) z holds exactly for the z of M z = r; in floating
    # point the two forms differ by rounding, which the iteration carries: the
    # same iteration count within one and solutions far inside the solver's
    # 1e-8 parity bound
    nx, ny, nz, varying, graded, a_v = cfg
    prob, kw, b = case(nx, ny, nz, varying, graded, a_v=a_v, seed=13)
    out = {}
    with mf.Solver(nx, ny, nz, **kw) as s:
        s.set_substructuring(1)
        s.set_loop(loop)
        bd = torch.from_numpy(b).to(DEV)
        for form in ["stencil", "residual"]:
            s.set_az_form(form)
            assert s.az_form == form
            x = torch.zeros_like(bd)
            it, hist, st = s.solve(bd, x, rtol=1e-10, maxit=500)
            assert st == mf.PCG_OK
            out[form] = (it, hist, x.cpu().numpy())
    (i0, h0, x0), (i1, h1, x1) = out["stencil"], out["residual"]
    assert abs(i0 - i1) <= 1
    m = min(i0, i1) + 1
    np.testing.assert_allclose(h1[:m], h0[:m], rtol=1e-6, atol=1e-13)
    assert np.linalg.norm(x1 - x0) <= 1e-9 * np.linalg.norm(x0)
    # the true residual of the residual-form solution meets the tolerance as
    # well as the stencil form's does (to a factor 2 of rounding)
    tr = [np.linalg.norm(b - oracle.apply_A(prob, xx)) / np.linalg.norm(b) for xx in (x0, x1)]
    assert tr[1] <= max(2.0 * tr[0], 1e-10)


def test_az_form_resolution_and_arguments():
    prob, kw, b = case(20, 12, 16, True, True, a_v=1e3, seed=8)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        assert s.az_form == "residual"          # the default: row-tiled, Thomas
        s.set_az_form("stencil")
        assert s.az_form == "stencil"
        s.set_az_form("residual")
        s.set_substructuring(2)                 # substructured solves: the stencil
        assert s.az_form == "stencil"
        s.set_substructuring(1)
        assert s.az_form == "residual"
        s.set_layout("column")                  # the column layout has both forms
        assert s.az_form == "residual"
        s.set_az_form("stencil")
        assert s.az_form == "stencil"
        with pytest.raises(mf.PCGError) as e:
            mf.pcg_set_az_form(s.ctx, 3)
        assert e.value.status == mf.PCG_EINVAL


def test_factor_mode_arguments_and_column_layout():
    prob, kw, b = case(20, 12, 16, True, True, a_v=1e3, seed=8)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        with pytest.raises(mf.PCGError) as e:
            mf.pcg_set_factors(s.ctx, 2)
        assert e.value.status == mf.PCG_EINVAL
        bd = torch.from_numpy(b).to(DEV)
        xs = []
        s.set_layout("column")
        for mode in ["stored", "recompute"]:   # the column layout always reads stored factors
            s.set_factors(mode)
            x = torch.zeros_like(bd)
            s.solve(bd, x, rtol=1e-10)
            xs.append(x.cpu().numpy())
    assert np.array_equal(xs[0], xs[1])


# ---- substructured column solves (parallel in k)

SPLIT_CASES = [  # nx, ny, nz, varying, graded, a_v, blocks per column
    (32, 32, 16, False, False, 1e2, 8),    # the 32x32x16 operator
    (37, 29, 16, True, True, 1e3, 4),      # ragged last tile
    (33, 5, 7, True, True, 1e2, 4),        # odd nz: blocks of one level
    (40, 36, 64, False, True, 1e4, 2),
    (17, 19, 130, True, True, 1e5, 16),
    (7, 5, 400, True, False, 1e3, 16),     # blocks of about 24 levels, 221 KB of shared tiles
]


def column_cond(prob):
    """Largest 2-norm condition number of the column blocks of M (eq. (19)),
    over the smallest and the largest horizontal face sum of the grid."""
    nz, h = prob.nz, np.asarray(prob.h)
    ah = np.asarray(prob.ah).reshape(prob.ny, prob.nx)
    faces = 0.5 * (ah + np.roll(ah, -1, 1)) + 0.5 * (ah + np.roll(ah, 1, 1)) \
        + 0.5 * (ah + np.roll(ah, -1, 0)) + 0.5 * (ah + np.roll(ah, 1, 0))
    t = np.array([prob.a_v / (0.5 * (h[k] + h[k + 1])) for k in range(nz - 1)])
    conds = []
    for sf in (faces.min(), faces.max()):
        d = h * (prob.mass + sf)
        d[:-1] += t
        d[1:] += t
        T = np.diag(d) - np.diag(t, 1) - np.diag(t, -1)
        conds.append(np.linalg.cond(T))
    return max(conds)


@pytest.mark.parametrize("cfg", SPLIT_CASES, ids=lambda c: "x".join(map(str, c[:3])) + "P%d" % c[6])
def test_substructured_solve_matches_oracle(cfg):
    nx, ny, nz, varying, graded, a_v, nb = cfg
    prob, kw, b = case(nx, ny, nz, varying, graded, a_v=a_v, seed=11)
    # one iteration: x_1 = alpha M^{-1} b, so x_1 carries the preconditioner's
    # error, which for a different elimination order is bounded by a few units
    # of cond(T) * eps of the column blocks T
    tol1 = max(OP_TOL, column_cond(prob) * np.finfo(float).eps)
    x1_ref, _, _, _ = oracle.pcg(prob, b, rtol=0.0, maxit=1)
    x_ref, it_ref, hist_ref, st_ref = oracle.pcg(prob, b, rtol=1e-10, maxit=500)
    assert st_ref == oracle.OK
    with mf.Solver(nx, ny, nz, **kw) as s:
        s.set_substructuring(nb)
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        assert s.solve(bd, x, rtol=0.0, maxit=1)[0] == 1
        x1 = x.cpu().numpy()
        x.zero_()
        iters, hist, st = s.solve(bd, x, rtol=1e-10, maxit=500)
        assert st == mf.PCG_OK and abs(iters - it_ref) <= 1
        np.testing.assert_allclose(hist[: min(iters, it_ref) + 1],
                                   hist_ref[: min(iters, it_ref) + 1], rtol=1e-6, atol=1e-13)
        x.zero_()
        assert s.solve(bd, x, rtol=0.0, maxit=it_ref)[:1] == (it_ref,)
        xs = x.cpu().numpy()
    assert rel_maxdiff(x1, x1_ref) <= tol1, (rel_maxdiff(x1, x1_ref), tol1)
    assert np.linalg.norm(xs - x_ref) <= SOL_TOL * np.linalg.norm(x_ref)


def test_substructuring_arguments():
    prob, kw, b = case(20, 12, 7, True, True, a_v=1e3, seed=9)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        for bad in (-1, 3, 32, 8):   # 8 blocks need nz >= 15
            with pytest.raises(mf.PCGError) as e:
                s.set_substructuring(bad)
            assert e.value.status == mf.PCG_EINVAL
        bd = torch.from_numpy(b).to(DEV)
        out = []
        # with the automatic loop these 8 tiles run the cluster loop, which
        # needs (and beats) Thomas column solves; with the batched loop they
        # are substructured (fewer tiles than half the SMs): 4 blocks
        s.set_substructuring(0)
        assert (s.substructuring, s.loop) == (1, "cluster")
        s.set_loop("batched")
        for nb in (4, 1, 2, 0, 4):
            s.set_substructuring(nb)
            assert s.substructuring == (4 if nb == 0 else nb)
            x = torch.zeros_like(bd)
            it, _, st = s.solve(bd, x, rtol=1e-10)
            assert st == mf.PCG_OK
            out.append((nb, it, x.cpu().numpy()))
    assert np.array_equal(out[0][2], out[4][2])   # switching back is exact
    for nb, it, x in out[1:4]:
        assert abs(it - out[0][1]) <= 1


def test_substructuring_refuses_columns_too_tall_for_its_shared_tiles():
    # 2 x 500 levels x 32 columns of doubles exceed a block's shared memory:
    # an explicit request is refused, the automatic choice falls back to
    # Thomas, and neither leaves an error behind for the next launch
    prob, kw, b = case(6, 5, 500, False, False, a_v=1e3, seed=13)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        assert s.substructuring == 1
        with pytest.raises(mf.PCGError) as e:
            s.set_substructuring(2)
        assert e.value.status == mf.PCG_EINVAL
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        it, _, st = s.solve(bd, x, rtol=1e-10)
        assert st == mf.PCG_OK and s.substructuring == 1


# ---- coefficient changes and degenerate grids in every solver mode

def fixed_iterate_matches(s, prob, b, iters=6):
    """Iterate after a fixed number of iterations against the oracle's."""
    x_ref, it_ref, _, st_ref = oracle.pcg(prob, b, rtol=0.0, maxit=iters)
    bd = torch.from_numpy(b).to(DEV)
    x = torch.zeros_like(bd)
    it, _, st = s.solve(bd, x, rtol=0.0, maxit=iters)
    assert (it, st) == (it_ref, mf.PCG_OK) and st_ref == oracle.OK
    xs = x.cpu().numpy()
    return np.linalg.norm(xs - x_ref) <= SOL_TOL * np.linalg.norm(x_ref)


@pytest.mark.parametrize("mode", ["column", "tiled", "tiled_recompute", "tiled_split2"])
def test_solves_follow_coefficient_updates(mode):
    # field -> another field -> constant a_h -> the first field again: the
    # per-cell tables of every layout (diagonal, weights, factors, blocks)
    # must follow each update
    prob, kw, b = case(37, 21, 24, True, True, a_v=1e4, seed=14)
    ah2 = W.horizontal_coefficient(37, 21, True)[::-1].copy() * 1.5
    steps = [
        (dict(a_h_field=ah2, a_v=3e3, mass=0.5, dz=prob.h), ah2, 3e3, 0.5),
        (dict(a_h=0.8, a_v=1e4, mass=1.0, dz=prob.h), 0.8, 1e4, 1.0),
        (kw, prob.ah, kw["a_v"], 1.0),
    ]
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        if mode == "column":
            s.set_layout("column")
        s.set_factors("recompute" if mode == "tiled_recompute" else "stored")
        s.set_substructuring(2 if mode == "tiled_split2" else 1)
        assert fixed_iterate_matches(s, prob, b)
        for coeffs, ah, a_v, mass in steps:
            s.update_coeffs(**coeffs)
            p2 = oracle.Problem(prob.nx, prob.ny, prob.nz, ah=ah, a_v=a_v, mass=mass, h=prob.h)
            assert fixed_iterate_matches(s, p2, b), coeffs.keys()


DEGENERATE = [  # nx, ny, nz, varying, graded: self-neighbours, single columns, single levels
    (1, 1, 9, True, True),
    (1, 7, 12, True, False),
    (7, 1, 12, False, True),
    (3, 1, 2, True, True),
    (33, 1, 5, True, True),     # one full tile and one column in the next
    (40, 2, 1, True, False),    # a single level: M is diagonal
]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("cfg", DEGENERATE, ids=lambda c: "x".join(map(str, c[:3])))
def test_degenerate_grids_solve_like_the_oracle(cfg, mode):
    nx, ny, nz, varying, graded = cfg
    prob, kw, b = case(nx, ny, nz, varying, graded, a_v=1e3, seed=15)
    x_ref, it_ref, _, st_ref = oracle.pcg(prob, b, rtol=1e-10, maxit=500)
    assert st_ref == oracle.OK
    with mf.Solver(nx, ny, nz, **kw) as s:
        configure(s, mode)
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        it, _, st = s.solve(bd, x, rtol=1e-10, maxit=500)
        assert st == mf.PCG_OK and abs(it - it_ref) <= 1
        x.zero_()
        assert s.solve(bd, x, rtol=0.0, maxit=it_ref)[0] == it_ref
        xs = x.cpu().numpy()
    assert np.linalg.norm(xs - x_ref) <= SOL_TOL * np.linalg.norm(x_ref)


# ---- the persistent solve loop (one cooperative kernel per solve)

def test_persistent_loop_choice_and_timing():
    prob, kw, b = case(30, 26, 24, True, True, a_v=1e3, seed=16)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        s.set_substructuring(1)
        assert s.loop == "cluster"             # 25 tiles fit one cluster: the automatic choice
        s.set_az_form("stencil")               # the cluster loop has the residual form only
        assert s.loop == "persistent"          # 25 tiles: the next automatic choice
        s.set_az_form("auto")
        s.set_loop("batched")
        assert s.loop == "batched"
        s.set_loop("persistent")
        s.set_factors("recompute")             # not for rebuilt factors ...
        assert s.loop == "batched"
        s.set_factors("stored")
        s.set_substructuring(2)                # ... nor for substructured columns
        assert s.loop == "batched"
        s.set_substructuring(1)
        assert s.loop == "persistent"
        with pytest.raises(mf.PCGError):
            mf.pcg_set_loop(s.ctx, 5)
        s.enable_timing(True)
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        it, _, st = s.solve(bd, x, rtol=1e-10)
        t = s.kernel_times()
        assert st == mf.PCG_OK and t["loop"][1] == 1 and t["loop"][0] > 0
        assert t["precond_fused"][1] == 0 and t["spmv_fused"][1] == 0
        assert s.launch_info()["last_solve_launches"] == 3   # residual, loop, final update


def test_persistent_loop_automatic_choice_on_mid_grids():
    # 1000 tiles (6.6 per SM): persistent by the cell-count rule, and equal to
    # the oracle's iterate; 2048 tiles with 6.55 M cells: batched
    prob, kw, b = case(200, 160, 24, True, True, a_v=1e3, seed=19)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        assert s.loop == "persistent"
        x_ref, it_ref, _, _ = oracle.pcg(prob, b, rtol=1e-10)
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        it, _, st = s.solve(bd, x, rtol=1e-10)
        assert st == mf.PCG_OK and abs(it - it_ref) <= 1
        x.zero_()
        it2, _, st2 = s.solve(bd, x, rtol=0.0, maxit=it_ref)
        assert (it2, st2) == (it_ref, mf.PCG_OK)
        assert np.linalg.norm(x.cpu().numpy() - x_ref) <= SOL_TOL * np.linalg.norm(x_ref)
    with mf.Solver(256, 256, 100, a_h=1.0, a_v=1e3) as s:
        assert s.loop == "batched"
    with mf.Solver(256, 256, 96, a_h=1.0, a_v=1e3) as s:      # 6 * 2^20 cells
        assert s.loop == "persistent"


@pytest.mark.parametrize("cfg", SOLVE_CASES, ids=lambda c: "x".join(map(str, c[:3])))
def test_persistent_and_batched_loops_agree(cfg):
    # the same sweeps in the same arithmetic; only the reduction trees differ
    nx, ny, nz, varying, graded, a_v = cfg
    prob, kw, b = case(nx, ny, nz, varying, graded, a_v=a_v, seed=17)
    with mf.Solver(nx, ny, nz, **kw) as s:
        bd = torch.from_numpy(b).to(DEV)
        out = {}
        for mode in ["tiled", "tiled_persistent"]:
            configure(s, mode)
            x = torch.zeros_like(bd)
            it, hist, st = s.solve(bd, x, rtol=1e-10)
            out[mode] = (it, st, hist, x.cpu().numpy())
    (i1, s1, h1, x1), (i2, s2, h2, x2) = out["tiled"], out["tiled_persistent"]
    assert s1 == s2 == mf.PCG_OK and abs(i1 - i2) <= 1
    n = min(i1, i2) + 1
    np.testing.assert_allclose(h1[:n], h2[:n], rtol=1e-6, atol=1e-13)
    assert np.linalg.norm(x1 - x2) <= SOL_TOL * np.linalg.norm(x1)


@pytest.mark.parametrize("loop", ["persistent", "batched"])
def test_two_contexts_solve_concurrently_on_two_streams(loop):
    # each context captures its graphs on a private stream and launches on
    # the caller's; concurrent solves give the sequential results bit for bit
    cases = [case(30, 26, 24, True, True, a_v=1e3, seed=18),
             case(41, 17, 16, False, True, a_v=1e4, seed=19)]
    solvers = [mf.Solver(p.nx, p.ny, p.nz, **kw) for p, kw, _ in cases]
    try:
        bs = [torch.from_numpy(b).to(DEV) for _, _, b in cases]
        ref = []
        for s, bd in zip(solvers, bs):
            s.set_substructuring(1)
            s.set_loop(loop)
            x = torch.zeros_like(bd)
            it, _, st = s.solve(bd, x, rtol=1e-10)
            ref.append((it, st, x.cpu().numpy()))
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        xs = [torch.zeros_like(bd) for bd in bs]
        for s, st_ in zip(solvers, streams):
            s.set_stream(st_)
        torch.cuda.synchronize()
        import threading
        out = [None, None]

        def run(i):
            with torch.cuda.stream(streams[i]):
                out[i] = solvers[i].solve(bs[i], xs[i], rtol=1e-10)

        threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        torch.cuda.synchronize()
        for i in range(2):
            it, _, st = out[i]
            assert (it, st) == ref[i][:2]
            assert np.array_equal(xs[i].cpu().numpy(), ref[i][2])
    finally:
        for s in solvers:
            s.close()


@pytest.mark.parametrize("mode", ["column", "tiled", "tiled_persistent"])
def test_very_tall_columns(mode):
    # 1500 levels: the row-tiled sweeps stream any height in register chunks;
    # the column layout takes its unstaged preconditioner sweep
    prob, kw, b = case(5, 3, 1500, True, False, a_v=1e3, seed=20)
    x_ref, it_ref, _, st_ref = oracle.pcg(prob, b, rtol=1e-10, maxit=500)
    assert st_ref == oracle.OK
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        configure(s, mode)
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        it, _, st = s.solve(bd, x, rtol=1e-10, maxit=500)
        assert st == mf.PCG_OK and abs(it - it_ref) <= 1
        x.zero_()
        assert s.solve(bd, x, rtol=0.0, maxit=it_ref)[0] == it_ref
        xs = x.cpu().numpy()
    assert np.linalg.norm(xs - x_ref) <= SOL_TOL * np.linalg.norm(x_ref)


def test_persistent_barrier_wait_runs_out_and_the_context_recovers():
    # the barriers count one arrival that never comes: the first wait runs out
    # after its poll limit (about a second), the solve reports PCG_ETIMEOUT,
    # and the next solve on the same context is normal
    import time
    prob, kw, b = case(30, 26, 24, True, True, a_v=1e3, seed=21)
    _, it_ref, _, _ = oracle.pcg(prob, b, rtol=1e-10)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        s.set_loop("persistent")
        s.set_substructuring(1)
        assert s.loop == "persistent"
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        mf.pcg_test_barrier_absent(s.ctx, 1)
        t0 = time.perf_counter()
        with pytest.raises(mf.PCGError) as e:
            s.solve(bd, x, rtol=1e-10)
        assert e.value.status == mf.PCG_ETIMEOUT
        assert "bounded device wait" in mf.pcg_last_error(s.ctx)
        assert time.perf_counter() - t0 < 60.0
        mf.pcg_test_barrier_absent(s.ctx, 0)
        x.zero_()
        it, _, st = s.solve(bd, x, rtol=1e-10)
        assert st == mf.PCG_OK and abs(it - it_ref) <= 1


CLUSTER_CASES = [
    # nx, ny, nz, varying, graded, a_v: grids whose vectors fit one cluster
    (37, 29, 16, True, True, 1e3),
    (33, 5, 7, True, True, 1e2),
    (32, 32, 16, False, False, 1e2),
    (30, 26, 24, True, True, 1e4),
    (1, 1, 40, True, True, 1e3),
    (64, 3, 9, False, True, 1e3),
]


@pytest.mark.parametrize("cfg", CLUSTER_CASES, ids=lambda c: "x".join(map(str, c[:3])))
def test_cluster_loop_matches_oracle(cfg):
    nx, ny, nz, varying, graded, a_v = cfg
    prob, kw, b = case(nx, ny, nz, varying, graded, a_v=a_v, seed=17)
    x_ref, it_ref, hist_ref, st_ref = oracle.pcg(prob, b, rtol=1e-10, maxit=500)
    assert st_ref == oracle.OK
    with mf.Solver(nx, ny, nz, **kw) as s:
        s.set_substructuring(1)
        s.set_loop("cluster")
        assert s.loop == "cluster"
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        iters, hist, st = s.solve(bd, x, rtol=1e-10, maxit=500)
        assert st == mf.PCG_OK and abs(iters - it_ref) <= 1
        m = min(iters, it_ref) + 1
        np.testing.assert_allclose(hist[:m], hist_ref[:m], rtol=1e-6, atol=1e-13)
        x2 = torch.zeros_like(bd)
        i2, h2, _ = s.solve(bd, x2, rtol=1e-10, maxit=500)
        assert i2 == iters and np.array_equal(h2, hist) and torch.equal(x, x2)  # repeatable
        x.zero_()
        it3, _, st3 = s.solve(bd, x, rtol=0.0, maxit=it_ref)
        assert (it3, st3) == (it_ref, mf.PCG_OK)
        xs = x.cpu().numpy()
        # the persistent loop computes the same iterates up to rounding
        s.set_loop("persistent")
        assert s.loop == "persistent"
        xp = torch.zeros_like(bd)
        s.solve(bd, xp, rtol=0.0, maxit=it_ref)
    assert np.linalg.norm(xs - x_ref) <= SOL_TOL * np.linalg.norm(x_ref)
    assert np.linalg.norm(xs - xp.cpu().numpy()) <= 1e-10 * np.linalg.norm(x_ref)


def test_cluster_loop_status_semantics_and_timing():
    prob, kw, b = case(20, 18, 16, True, True, a_v=1e3, seed=18)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        s.set_substructuring(1)
        assert s.loop == "cluster"
        bd = torch.from_numpy(b).to(DEV)
        _, it_ref, _, _ = oracle.pcg(prob, b, rtol=1e-8)
        x = torch.zeros_like(bd)
        it, _, st = s.solve(bd, x, rtol=1e-8, maxit=it_ref - 2)
        assert (it, st) == (it_ref - 2, mf.PCG_ENOTCONV)
        x.zero_()
        it, hist, st = s.solve(bd, x, rtol=0.0, maxit=3)
        assert (it, st, len(hist)) == (3, mf.PCG_OK, 4)
        x.zero_()
        it, hist, st = s.solve(torch.zeros_like(bd), x, rtol=1e-10)
        assert (it, st) == (0, mf.PCG_OK) and float(x.abs().max()) == 0.0
        bad = bd.clone()
        bad[40] = float("nan")
        x.zero_()
        _, _, st = s.solve(bad, x, rtol=1e-10)
        assert st == mf.PCG_EBREAKDOWN
        x0 = np.random.default_rng(19).standard_normal(prob.n)
        x.copy_(torch.from_numpy(x0))
        it, _, st = s.solve(bd, x, rtol=1e-8)
        x_ref, it_ref2, _, _ = oracle.pcg(prob, b, x0=x0, rtol=1e-8)
        assert st == mf.PCG_OK and abs(it - it_ref2) <= 1
        assert np.linalg.norm(x.cpu().numpy() - x_ref) <= 1e-6 * np.linalg.norm(x_ref)
        s.enable_timing(True)
        x.zero_()
        it, _, st = s.solve(bd, x, rtol=1e-10)
        t = s.kernel_times()
        assert st == mf.PCG_OK and t["loop"][1] == 1 and t["loop"][0] > 0
        assert s.launch_info()["last_solve_launches"] == 3   # residual, loop, final update
        # a grid too large for one cluster runs persistent when the cluster loop is asked for
    with mf.Solver(128, 128, 64, a_h=1.0, a_v=1e3) as s:
        s.set_substructuring(1)
        s.set_loop("cluster")
        assert s.loop == "persistent"


@pytest.mark.parametrize("bad", [float("nan"), -0.25, float("inf")], ids=["nan", "negative", "inf"])
@pytest.mark.parametrize("api", ["update_coeffs", "update_solve_host", "update_solve_host_async"])
def test_rejected_field_leaves_the_context_as_it_was(bad, api):
    # the field of an update is checked on the device in a staging copy:
    # a bad value is named by its index, and the context keeps its old
    # coefficients (a solve gives the same bits as before the attempt)
    prob, kw, b = case(37, 29, 16, True, True, a_v=1e3, seed=41)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        bd = torch.from_numpy(b).to(DEV)
        x1 = torch.zeros_like(bd)
        i1, h1, _ = s.solve(bd, x1, rtol=1e-10)
        field = np.array(kw["a_h_field"], dtype=np.float64).ravel().copy() * 2.0
        where = 517
        field[where] = bad
        new = dict(kw, a_h_field=field.reshape(prob.ny, prob.nx))
        with pytest.raises(mf.PCGError) as e:
            if api == "update_coeffs":
                s.update_coeffs(**new)
            else:
                xh = np.zeros(prob.n)
                getattr(s, api)(b, xh, **new)
        assert e.value.status == mf.PCG_EINVAL
        assert "a_h_field[%d]" % where in mf.pcg_last_error(s.ctx)
        s.host_wait()
        x2 = torch.zeros_like(bd)
        i2, h2, _ = s.solve(bd, x2, rtol=1e-10)
        assert i1 == i2 and np.array_equal(h1, h2) and torch.equal(x1, x2)
        # and a good field after the rejected one is taken
        field[where] = 1.0
        s.update_coeffs(**dict(kw, a_h_field=field.reshape(prob.ny, prob.nx)))
        prob2 = oracle.Problem(prob.nx, prob.ny, prob.nz, ah=field.reshape(prob.ny, prob.nx),
                               a_v=prob.a_v, mass=prob.mass, h=prob.h)
        y = s.apply_A(bd).cpu().numpy()
    assert rel_maxdiff(y, oracle.apply_A(prob2, b)) <= OP_TOL


@pytest.mark.parametrize("mode", ["tiled", "column", "tiled_persistent"])
def test_solve_from_zero_never_reads_x(mode):
    # pcg_solve_from_zero: the same bits as pcg_solve from an x filled with
    # +0.0, whatever x held before (here NaN)
    prob, kw, b = case(37, 29, 16, True, True, a_v=1e3, seed=43)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        configure(s, mode)
        bd = torch.from_numpy(b).to(DEV)
        x1 = torch.zeros_like(bd)
        i1, h1, st1 = s.solve(bd, x1, rtol=1e-10)
        x2 = torch.full_like(bd, float("nan"))
        i2, h2, st2 = s.solve_from_zero(bd, x2, rtol=1e-10)
    assert st1 == st2 == mf.PCG_OK and i1 == i2
    assert np.array_equal(h1, h2) and torch.equal(x1, x2)


@pytest.mark.parametrize("mode", MODES + ["tiled_cluster", "tiled_multigrid"])
def test_solves_write_work_vectors_before_reading_them(mode):
    # The context's work vectors filled with NaN, as memory that an earlier
    # user left behind may hold: a solve from x0 = 0 with b = 0, a solve
    # allowed no iteration (x = x0) and a full solve give the same bits as
    # without the fill.  The batched row-tiled start leaves p unwritten, so a
    # solve that stops before its first direction must not read it.
    prob, kw, b = case(20, 18, 16, True, True, a_v=1e3, seed=53)
    x0 = np.random.default_rng(54).standard_normal(prob.n)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        if mode == "tiled_cluster":
            configure(s, "tiled")
            s.set_loop("cluster")
            assert s.loop == "cluster"
        elif mode == "tiled_multigrid":
            configure(s, "tiled")
            s.set_preconditioner("multigrid")
        else:
            configure(s, mode)
        bd = torch.from_numpy(b).to(DEV)
        x0d = torch.from_numpy(x0).to(DEV)
        runs = []
        for poison in (False, True):
            out = []
            for rhs, guess, maxit in ((torch.zeros_like(bd), None, 500), (bd, x0d, 0),
                                      (bd, None, 500)):
                if poison:
                    mf.pcg_test_poison_work(s.ctx)
                x = torch.zeros_like(bd) if guess is None else guess.clone()
                it, hist, st = s.solve(rhs, x, rtol=1e-10, maxit=maxit)
                out.append((it, st, hist, x.cpu().numpy()))
            runs.append(out)
    (z_it, z_st, _, z_x), (m_it, m_st, _, m_x), (f_it, f_st, _, _) = runs[1]
    assert (z_it, z_st) == (0, mf.PCG_OK) and np.array_equal(z_x, np.zeros(prob.n))
    assert (m_it, m_st) == (0, mf.PCG_ENOTCONV) and np.array_equal(m_x, x0)
    assert f_st == mf.PCG_OK and f_it > 1
    for a, c in zip(runs[0], runs[1]):
        assert a[:2] == c[:2]
        assert np.array_equal(a[2], c[2]) and np.array_equal(a[3], c[3])
