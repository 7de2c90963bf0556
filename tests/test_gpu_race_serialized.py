"""Race detection without a sanitizer: the same parity cases run against a
build in which the MMA thread waits for every MMA group to complete before it
moves on (CPATTN_SERIALIZE_MMA).  That stretches one side of every
producer/consumer hand-off in the pipeline; a protocol whose correctness
depends on timing (e.g. an ambiguous mbarrier parity wait) fails here.  The
selection spans every pipeline form: paired (2-SM MMA) and
unpaired kernels, the two-query-tile kernel, split-KV pieces, GQA-packed units, the fused KV write, the
fp16 V cache forms (with and without the chunk's V staged in fp16, whose prefill starts as a
programmatic dependent of the staging), and inputs that rescale O on every tile."""
import os
import subprocess
import sys

import pytest

from long_context_chunked_gb300 import build as cpbuild

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_under_serialized_mma():
    lib = cpbuild.build(variant="serialized")
    env = dict(os.environ, CPATTN_LIBRARY=lib)
    t = lambda f: os.path.join(ROOT, "tests", f)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        t("test_gpu_prefill.py"), t("test_gpu_pairing.py"),
                        t("test_gpu_splitkv.py"), t("test_gpu_gqa_packing.py"),
                        t("test_gpu_prefill_write_kv.py"), t("test_gpu_v_f16.py"),
                        t("test_gpu_pingpong.py"), "-k",
                        "tiny_full or edges_full or equal_keys or repeatable or rescale "
                        "or pairing_mode_parity or forced_split or packed_parity "
                        "or test_prefill_write_kv or test_parity or test_pairing_modes "
                        "or test_split_kv or test_fused_write_kv or pingpong_parity "
                        "or pingpong_split or pingpong_fused"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    import re
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and " failed" not in r.stdout, r.stdout[-2000:]
    print("serialized MMA:", r.stdout.strip().splitlines()[-1])
    assert int(m.group(1)) >= 90, r.stdout[-2000:]  # the selection above, not a subset
