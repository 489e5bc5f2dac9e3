import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")
    config.addinivalue_line("markers", "oracle_run(name): compares with a long oracle run on "
                                       "workload `name` (started in the background after "
                                       "collection, see tests/oracle_refs.py)")


def pytest_collection_finish(session):
    """Start the long oracle runs that the selected tests need, so that they
    overlap with the tests that run before them."""
    names = []
    for item in session.items:
        for m in item.iter_markers("oracle_run"):
            names.extend(m.args)
    if not names:
        return
    try:
        import torch
        if not torch.cuda.is_available():
            return  # the tests that would wait for them are skipped
    except ImportError:
        return
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import oracle_refs
    oracle_refs.start(sorted(set(names)))
