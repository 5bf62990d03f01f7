import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


# The five workloads' parity tests: their err (rounding allowance of the
# output dtype subtracted) and plain (max |X - ref| / max |ref|) per tensor.
WORKLOAD_TESTS = {
    "test_prefill_tiny_fp32": "tiny (fp32, T=256, H=2, d=64)",
    "test_prefill_single_sequence_workload": "single (bf16, T=8192, H=32)",
    "test_prefill_varlen_workload": "varlen (bf16, 16 seqs, H=32)",
    "test_prefill_long_context_workload": "long (bf16, T=1M, H=32)",
    "test_decode_workload_first_steps_full": "decode (B=256, 8 steps)",
    "test_decode_workload_1024_steps_sampled_sequences": "decode (1024 steps, seqs 0-7)",
}


def pytest_terminal_summary(terminalreporter):
    try:
        import parity
    except Exception:  # pragma: no cover
        return
    recs = parity.RECORDS
    if not recs:
        return
    path = os.environ.get("KDA_PARITY_LOG")
    if path:
        import json
        with open(path, "w") as f:
            json.dump([dict(test=t, name=n, err=e, plain=p, tol=tol)
                       for t, n, e, p, tol in recs], f, indent=1)
    rows = {}
    for test, name, e, p, tol in recs:
        fn = test.split("::")[-1]
        if fn not in WORKLOAD_TESTS:
            continue
        key = (WORKLOAD_TESTS[fn], name.split(" step")[0])
        old = rows.get(key, (0.0, 0.0, tol))
        rows[key] = (max(old[0], e), max(old[1], p), tol)
    if not rows:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity on the workloads: err (dtype rounding allowed) / plain")
    for (wl, name), (e, p, tol) in rows.items():
        tr.write_line("%-32s %-40s err %.2e  plain %.2e  tol %.0e" % (wl, name, e, p, tol))
