"""Race detection without a sanitizer: the same parity cases run against a
build in which the MMA thread waits for every MMA group to complete before it
moves on (CPATTN_SERIALIZE_MMA).  That stretches one side of every
producer/consumer hand-off in the pipeline; a protocol whose correctness
depends on timing (e.g. an ambiguous mbarrier parity wait) fails here."""
import os
import subprocess
import sys

import pytest

from long_context_chunked_gb300 import build as cpbuild

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_under_serialized_mma():
    lib = cpbuild.build(serialized=True)
    env = dict(os.environ, CPATTN_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_prefill.py"), "-k",
                        "tiny_full or edges_full or equal_keys or repeatable"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
