"""The checked build: libkvq3_checked.so, compiled with KVQ3_CHECKED, carries
in-kernel bounds checks (pool ranges of the writes and the read-back, the
source and destination of every bulk copy, the stage reads of each decode
step, the workspace slots of the split-K merge and the combine) that report
KVQ3_DEV_CHECK in the status word and skip the access; they never trap.
This runs the write, read-back and decode parity tests against the oracle
through that library in a child process (KVQ3_LIBRARY selects it); every one
of them requires a zero status word, so a check that fires fails them."""
import importlib.util
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _checked_library() -> str:
    path = os.path.join(ROOT, "hadamard_rotated_bit_kvq3_gb300", "_build.py")
    spec = importlib.util.spec_from_file_location("kvq3_build_checked", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build(checked=True)


def test_parity_through_the_checked_build():
    lib = _checked_library()
    assert os.path.exists(lib)
    env = dict(os.environ, KVQ3_LIBRARY=lib)
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", "test_gpu_parity.py"), os.path.join(ROOT, "tests", "test_gpu_asym.py"),
           "-k", "write or decode or dequant or tiny"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    print(p.stdout[-2000:])
    assert p.returncode == 0, p.stdout[-4000:] + p.stderr[-2000:]
    # the child really loaded the checked library
    probe = subprocess.run([sys.executable, "-c", "import hadamard_rotated_bit_kvq3_gb300 as K; print(K.LIB_PATH)"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.stdout.strip() == lib
