"""Long oracle runs for the full-size parity tests, in background threads.

The oracle's whole-grid solves on the two largest workloads take minutes of
one host core each (the 1024x1024x128 solve to 1e-10, 50 fixed iterations on
2048x2048x64).  The C oracle releases the GIL for the length of a call, so
these runs go in daemon threads as soon as collection has selected a test
that needs them (tests/conftest.py) and overlap with the GPU tests that run
meanwhile; the tests that need a result wait for it here.  Nothing in this
module touches the GPU or the CUDA path: inputs come from the seeded
generators, results from the oracle alone.
"""
import threading
import time

import oracle
import workloads as W

# workload -> maxit of the oracle run (None: the workload's own stopping rule)
RUNS = {
    "graded_varcoef_1024x1024x128": None,   # to rtol 1e-10 (converged count, iterate)
    "bumps_2048x2048x64": 50,               # exactly 50 iterations
}

_lock = threading.Lock()
_jobs = {}


class _Job:
    def __init__(self, name):
        self.name = name
        self.result = None
        self.error = None
        self.seconds = None
        self.thread = threading.Thread(target=self._run, name="oracle-" + name, daemon=True)

    def _run(self):
        try:
            w = W.WORKLOADS[self.name]
            h, ah, vec = W.make_inputs(w)
            prob = oracle.Problem(w.nx, w.ny, w.nz, ah=ah, a_v=w.a_v, mass=w.mass, h=h)
            b = oracle.apply_A(prob, vec) if w.rhs == "manufactured" else vec
            fixed = RUNS[self.name]
            t0 = time.perf_counter()
            if fixed is None:
                x, it, hist, st = oracle.pcg(prob, b, rtol=w.rtol, maxit=w.maxit)
            else:
                x, it, hist, st = oracle.pcg(prob, b, rtol=0.0, maxit=fixed)
            self.seconds = time.perf_counter() - t0
            self.result = {"x": x, "iters": it, "hist": hist, "status": st}
        except BaseException as e:  # handed to the waiting test
            self.error = e


def start(names):
    """Start the oracle runs of `names` (each at most once per process)."""
    with _lock:
        for name in names:
            if name in RUNS and name not in _jobs:
                job = _Job(name)
                _jobs[name] = job
                job.thread.start()


def result(name, timeout=1800.0):
    """The oracle run of `name`: dict(x, iters, hist, status); waits for it."""
    start([name])
    job = _jobs[name]
    job.thread.join(timeout)
    if job.thread.is_alive():
        raise TimeoutError("oracle run of %s still going after %.0f s" % (name, timeout))
    if job.error is not None:
        raise job.error
    return job.result
