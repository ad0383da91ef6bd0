"""The bounds-checking build (compiled with -DQGEMV_BOUNDS_CHECK): every
entry point on small and odd shapes gives the oracle's results with no failed
index check, and a planted out-of-extent store is skipped and recorded, the
context staying usable.  It stands in for a memory checker, which cannot run
here.  The library is built and exercised in a child process, since the
binding picks the library when it is imported."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounds_checking_build_runs_clean_and_catches_a_planted_store():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_gemv_quantize_gb300 import build

    build.build(debug=True)
    env = dict(os.environ, QGEMV_BOUNDS_CHECK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_bounds_child.py")], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=1200)
    assert p.returncode == 0, p.stderr[-3000:]
    res = json.loads(p.stdout.strip().splitlines()[-1])
    print(len(res["cases"]), "cases;", "planted:", res["planted"])
    assert res["bounds_build"] is True
    assert res["fail"] == [], res["fail"]
    assert len(res["cases"]) >= 60
    count, site = res["planted"]
    assert count >= 1 and site == 620
    assert res["after_planted_ok"] and res["after_planted_records"] == [0, 0]
    assert res["timeouts"] == 0
