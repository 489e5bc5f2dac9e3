"""Out-of-bounds writes and read-only inputs, on the GPU.

The caller's vectors are cut from larger buffers whose bands on either side
hold a signalling-NaN bit pattern; after every entry point the bands must be
bit for bit intact, and the read-only inputs unchanged.  The vectors start at
16-byte-aligned addresses and at addresses that are only 8-byte aligned (the
kernels take vector loads only where the alignment allows).  Also: an
allocation failure reported as PCG_ENOMEM, after which the next context works.
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
BAND = 2048
PATTERN = 0x7FF4DEADBEEF0001  # a signalling NaN


def guarded(values, misalign):
    """(buffer, view): `values` in a view of a device buffer with guard bands."""
    n = values.numel()
    off = BAND + (1 if misalign else 0)
    buf = torch.empty(n + 2 * BAND + 1, dtype=torch.float64, device=DEV)
    buf.view(torch.int64).fill_(PATTERN)
    view = buf[off:off + n]
    view.copy_(values)
    return buf, view, off


def bands_intact(buf, off, n):
    bits = buf.view(torch.int64)
    return bool(torch.all(bits[:off] == PATTERN)) and bool(torch.all(bits[off + n:] == PATTERN))


def case(nx, ny, nz, varying, graded, a_v, seed):
    h = W.layer_thickness(nz, graded)
    ah = W.horizontal_coefficient(nx, ny, varying)
    prob = oracle.Problem(nx, ny, nz, ah=ah, a_v=a_v, mass=1.0, h=h)
    kw = dict(a_h_field=ah if varying else None, a_h=1.0, a_v=a_v, mass=1.0, dz=h)
    return prob, kw, np.random.default_rng(seed).uniform(-1, 1, nx * ny * nz)


GUARD_CASES = [
    # nx, ny, nz, varying, graded, a_v, set-up
    (37, 29, 16, True, True, 1e3, "default"),      # cluster loop, ragged last tile
    (33, 5, 7, True, True, 1e2, "column"),         # odd nz, column layout
    (100, 60, 20, False, True, 1e3, "persistent"),
    (48, 40, 33, True, True, 1e4, "batched"),
    (40, 36, 33, True, True, 1e4, "multigrid"),
    (64, 48, 64, True, True, 1e4, "split"),        # substructured columns
]


def configure(s, how):
    if how == "column":
        s.set_layout("column")
    elif how == "persistent":
        s.set_loop("persistent")
    elif how == "batched":
        s.set_loop("batched")
    elif how == "multigrid":
        s.set_preconditioner("multigrid")
    elif how == "split":
        s.set_substructuring(4)


@pytest.mark.parametrize("misalign", [False, True], ids=["aligned", "misaligned"])
@pytest.mark.parametrize("cfg", GUARD_CASES, ids=lambda c: "x".join(map(str, c[:3])) + "-" + c[6])
def test_entry_points_stay_inside_the_callers_vectors(cfg, misalign):
    nx, ny, nz, varying, graded, a_v, how = cfg
    prob, kw, b = case(nx, ny, nz, varying, graded, a_v, seed=41)
    n = prob.n
    bt = torch.from_numpy(b).to(DEV)
    with mf.Solver(nx, ny, nz, **kw) as s:
        configure(s, how)
        bbuf, bv, boff = guarded(bt, misalign)
        # y = A x
        ybuf, yv, yoff = guarded(torch.zeros_like(bt), misalign)
        mf.pcg_apply_A(s.ctx, n, bv, yv)
        torch.cuda.synchronize()
        assert bands_intact(ybuf, yoff, n) and bands_intact(bbuf, boff, n)
        assert torch.equal(bv, bt)
        assert np.max(np.abs(yv.cpu().numpy() - oracle.apply_A(prob, b))) <= \
            1e-12 * np.max(np.abs(oracle.apply_A(prob, b)))
        # z = M^{-1} r (and the V-cycle with the multigrid preconditioner)
        zbuf, zv, zoff = guarded(torch.zeros_like(bt), misalign)
        mf.pcg_precond(s.ctx, n, bv, zv)
        torch.cuda.synchronize()
        assert bands_intact(zbuf, zoff, n) and torch.equal(bv, bt)
        if how == "multigrid":
            vbuf, vv, voff = guarded(torch.zeros_like(bt), misalign)
            mf.pcg_mg_vcycle(s.ctx, n, bv, vv)
            torch.cuda.synchronize()
            assert bands_intact(vbuf, voff, n) and torch.equal(bv, bt)
        # the solve: b read only, x in and out
        xbuf, xv, xoff = guarded(torch.zeros_like(bt), misalign)
        it, _, st = mf.pcg_solve(s.ctx, n, bv, xv, 1e-10, 500, history=True)
        torch.cuda.synchronize()
        assert st == mf.PCG_OK
        assert bands_intact(xbuf, xoff, n) and bands_intact(bbuf, boff, n)
        assert torch.equal(bv, bt)
        if how == "multigrid":
            x_ref, it_ref, _, _ = oracle.mg_pcg(prob, b, rtol=1e-10)
        else:
            x_ref, it_ref, _, _ = oracle.pcg(prob, b, rtol=1e-10)
        assert abs(it - it_ref) <= 1
        # the iterate at the oracle's count, into the same guarded vector
        xv.zero_()
        it2, _, st2 = mf.pcg_solve(s.ctx, n, bv, xv, 0.0, it_ref, history=False)
        torch.cuda.synchronize()
        assert (it2, st2) == (it_ref, mf.PCG_OK) and bands_intact(xbuf, xoff, n)
        assert np.linalg.norm(xv.cpu().numpy() - x_ref) <= 1e-8 * np.linalg.norm(x_ref)


def test_allocation_failure_is_reported_and_the_next_context_works():
    # 2^39 cells: 4.4 TB per vector, far beyond the device
    with pytest.raises(mf.PCGError) as e:
        mf.Solver(1 << 15, 1 << 15, 512, a_h=1.0, a_v=1.0)
    assert e.value.status == mf.PCG_ENOMEM
    assert "allocation" in mf.pcg_last_error(None)
    prob, kw, b = case(37, 29, 16, True, True, 1e3, seed=42)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        it, _, st = s.solve(bd, x, rtol=1e-10)
        _, it_ref, _, _ = oracle.pcg(prob, b, rtol=1e-10)
        assert st == mf.PCG_OK and abs(it - it_ref) <= 1
