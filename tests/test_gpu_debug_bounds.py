"""The bounds-checking debug build (libzr_debug.so, ZR_DEBUG_BOUNDS).

Every global row index that a kernel derives from the device-built plans
(pack and reconstruction segments, group member ranges, attention query
blocks and key tiles) is checked before the access in that build; a failed
check skips the access and records its site in the status words, which
zr_check_status reports.  The outer test builds the variant and reruns a set
of the parity tests against it in a child process (ZR_LIBRARY selects the
library there): they must pass unchanged, i.e. the checks raise no false
alarm on valid batches (small, ragged, left-padded, unpadded, prompt-less,
response-less, odd widths and head counts) and the results equal the
oracle's.  No test feeds the kernels a corrupt plan: an out-of-range access
is what the checks prevent, and is not provoked on the GPU.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# parity tests rerun on the debug build: every copy kernel, both attention
# directions on every small layout, and one full-size attention case
SUBSET = ("group_pack_reconstruct_small or row_widths or reconstruct_backward_small or "
          "pack_rows_backward_small or reconstruct_pack_backward_small or dense_parity or "
          "reduced_qwen or pipeline-unpad or loaded_library")


def test_loaded_library_is_debug_build():
    """Runs only in the child process, against the debug build."""
    if not os.environ.get("ZR_LIBRARY"):
        pytest.skip("runs in the debug-build child process")
    from prompt_deduplicated_shared_gb300 import zr
    assert zr.LIB_PATH == os.environ["ZR_LIBRARY"]
    assert zr.debug_bounds()


def test_debug_build_passes_parity_without_false_alarms():
    if os.environ.get("ZR_LIBRARY"):
        pytest.skip("already in the child process")
    sys.path.insert(0, ROOT)
    import __graft_entry__  # noqa: F401  (the normal build, for the imports below)
    from prompt_deduplicated_shared_gb300 import build as zr_build
    from prompt_deduplicated_shared_gb300 import zr
    assert not zr.debug_bounds()  # the normal build checks nothing
    lib = zr_build.build(debug_bounds=True)
    env = dict(os.environ, ZR_LIBRARY=lib)
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu", "-k", SUBSET,
         "tests/test_gpu_dedup.py", "tests/test_gpu_attention.py", "tests/test_gpu_debug_bounds.py"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail
