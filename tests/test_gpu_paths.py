"""Both engine paths at every token count.

By default an engine layer launch with 8 or more tokens per expert runs on
tcgen05 and smaller ones on the CUDA cores, and the standalone GEMM calls
run on tcgen05 at every row count.  The library reads MOEQ_MMA_MIN_TOKENS once
per process, so these tests re-run the GEMM and reduced-layer parity tests
in child processes:
  * with the crossover at 1, every launch runs on tcgen05 (one-token
    experts, ragged K tails, split-K at every size);
  * with it at 17, every launch runs on the CUDA cores (16-token experts on
    the shared-memory accumulation mode).
Layers without the per-pair y output run the multi-token kernel unless
MOEQ_MTOK_KERNEL=0 (with MOEQ_TOKEN_KERNEL=0) hands them to the persistent
engine; the crossover children set both, a third child re-runs the
one-token layer tests, the full-size one included, and the reduced ones on
the engine, and a fourth the one-token ones on the one-token kernel
(MOEQ_MTOK_MIN_TOKENS=2).
The children use the same oracle comparisons and tolerances as the default
run."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("crossover", ["1", "17"])
def test_parity_with_forced_path(crossover):
    env = dict(os.environ, MOEQ_MMA_MIN_TOKENS=crossover, MOEQ_TOKEN_KERNEL="0", MOEQ_MTOK_KERNEL="0")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(HERE, "test_gpu_gemm.py"), os.path.join(HERE, "test_gpu_layer.py"),
           "-k", "not full_size and not full_m1 and not multi_token"]
    r = subprocess.run(cmd, env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"crossover {crossover}:\n{r.stdout[-3000:]}\n{r.stderr[-2000:]}"


def test_parity_one_token_on_the_persistent_engine():
    env = dict(os.environ, MOEQ_TOKEN_KERNEL="0", MOEQ_MTOK_KERNEL="0")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(HERE, "test_gpu_layer.py"), "-k", "m1 or reduced"]
    r = subprocess.run(cmd, env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"engine one-token path:\n{r.stdout[-3000:]}\n{r.stderr[-2000:]}"


def test_parity_one_token_on_the_one_token_kernel():
    env = dict(os.environ, MOEQ_MTOK_MIN_TOKENS="2")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(HERE, "test_gpu_layer.py"), os.path.join(HERE, "test_gpu_graph.py"),
           os.path.join(HERE, "test_gpu_stack.py"), os.path.join(HERE, "test_gpu_dense.py"),
           "-k", "m1 or (reduced and 1-) or graph or stack or (dense and 1-)"]
    r = subprocess.run(cmd, env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"one-token kernel path:\n{r.stdout[-3000:]}\n{r.stderr[-2000:]}"
