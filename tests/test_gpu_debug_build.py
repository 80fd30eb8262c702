"""The bounds-checked debug build of the library (-DHE_DEBUG: each computed
global access of the step kernels is checked, a failed check records an error
the host returns as HE_EDEVICE) runs the parity cases of several shapes and
options, and the allocation-free attention entry point, clean: no check fails
and every result matches the oracle (or, for the entry point, the step).  It stands
in for compute-sanitizer, which this pool does not offer."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_debug_build_runs_clean():
    from lsh_pre_attention_decode_b300 import _build
    _build.build(debug=True)  # (nothing to do when the build is current)
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([ROOT, HERE, env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, os.path.join(HERE, "_debug_build_cases.py")], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.count("ok ") == 10, r.stdout
