import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle


def load_golden(name):
    import json

    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        return json.load(f)


def build_product_library():
    """Run pagedattention_decode_pkv_gb300/build.py by path: importing it as a
    submodule would load the package (and a stale libpkv.so) first."""
    import importlib.util

    path = os.path.join(ROOT, "pagedattention_decode_pkv_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_pkv_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build_library()


@pytest.fixture(scope="session")
def pkv():
    """The product binding; builds libpkv.so in-tree first if needed (nvcc, sm_103a)."""
    build_product_library()
    import pagedattention_decode_pkv_gb300 as mod

    return mod


@pytest.fixture(scope="session")
def cuda_dev(pkv):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


# ------------------------------------------------------------------ accuracy margins
# Every attention comparison against the oracle goes through attn_error, which
# returns the max absolute error (what the bars bound) and records it with the
# max relative error for the end-of-session summary.  The relative error is
# taken over the elements whose reference magnitude is at least 1 % of the
# largest one: near-zero outputs of a flat softmax carry no relative meaning.
_ERRS = []  # (test id, max abs, max rel, bar)
_CURRENT = {"id": None}


@pytest.fixture(autouse=True)
def _track_test(request):
    _CURRENT["id"] = request.node.nodeid
    yield


def attn_error(out, ref) -> float:
    import torch

    if ref.numel() == 0:
        return 0.0
    got = out.detach().cpu().double()
    want = ref.detach().cpu().double()
    d = (got - want).abs()
    mabs = d.max().item()
    mag = want.abs()
    big = mag >= 0.01 * mag.max()
    rel = (d[big] / mag[big]).max().item() if bool(big.any()) else 0.0
    bar = 1e-5 if out.dtype == torch.float32 else 2e-2
    _ERRS.append((_CURRENT["id"], mabs, rel, bar))
    return mabs


def pytest_terminal_summary(terminalreporter):
    if not _ERRS:
        return
    import json

    by_file = {}
    for tid, a, r, bar in _ERRS:
        f = tid.split("::")[0]
        w = by_file.setdefault(f, [0, 0.0, 0.0, 0.0])
        w[0] += 1
        w[1] = max(w[1], a / bar)
        w[2] = max(w[2], a)
        w[3] = max(w[3], r)
    tr = terminalreporter
    tr.write_sep("-", "attention error vs the binary64 oracle (max abs / bar, max abs, max rel)")
    for f, (n, m, a, r) in sorted(by_file.items()):
        tr.write_line(f"{f}: {n} comparisons, worst {m:.3f} of the bar, max abs {a:.3g}, max rel {r:.3g}")
    path = os.environ.get("PKV_ACCURACY_REPORT")
    if path:
        with open(path, "w") as fh:
            json.dump([{"test": t, "max_abs": a, "max_rel": r, "bar": b} for t, a, r, b in _ERRS], fh, indent=0)
