"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle (on the CPU, never in the
real one) and runs the pin suite against the copy; the suite must fail.  The mistakes
are the ones a restatement of the method could plausibly make: a wrong GQA head map, a
dropped softmax scale, a strict causal test, positions counted from the wrong origin,
values taken from K, a wrong slot offset, and a mask that forgets the request test.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "gqa_head_map": ("kvh = h // group\n            s = (Q[:, h, :]", "kvh = h % n_kv_heads\n            s = (Q[:, h, :]"),
    "dropped_scale": ("s = (Q[:, h, :] @ K[:, kvh, :].T) * scale ", "s = (Q[:, h, :] @ K[:, kvh, :].T) "),
    "strict_causal": ("visible = key_pos[None, :] <= pos[:, None]", "visible = key_pos[None, :] < pos[:, None]"),
    "position_origin": ("pos = np.array([ctx + j for j in js])", "pos = np.array([ctx + j - 1 for j in js])"),
    "values_from_k": ("out[[start + j for j in js], h, :] = w @ V[:, kvh, :]",
                      "out[[start + j for j in js], h, :] = w @ K[:, kvh, :]"),
    "slot_offset": ("off = p % block_size\n    return", "off = (p + 1) % block_size\n    return"),
    "mask_without_request": ("return (q_seq[:, None] == key_seq[None, :]) & (key_pos[None, :] <= q_pos[:, None])",
                             "return (key_pos[None, :] <= q_pos[:, None])"),
}


def _sandbox(tmp, mutated_source):
    os.makedirs(os.path.join(tmp, "oracle"))
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), os.path.join(tmp, "oracle", "__init__.py"))
    with open(os.path.join(tmp, "oracle", "paged_step.py"), "w") as f:
        f.write(mutated_source)
    pkg = os.path.join(tmp, "continuous_batching_paged_step_gb300")
    os.makedirs(pkg)
    open(os.path.join(pkg, "__init__.py"), "w").close()
    shutil.copy(os.path.join(ROOT, "continuous_batching_paged_step_gb300", "workloads.py"), pkg)
    os.makedirs(os.path.join(tmp, "tests"))
    shutil.copy(os.path.join(ROOT, "tests", "test_oracle_pins.py"), os.path.join(tmp, "tests"))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(tmp, "tests", "golden"))


def _run_pins(tmp):
    env = dict(os.environ, PYTHONPATH=tmp)
    return subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                           "--rootdir", tmp, os.path.join(tmp, "tests", "test_oracle_pins.py")],
                          cwd=tmp, env=env, capture_output=True, text=True)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "paged_step.py")).read()
    old, new = MUTATIONS[name]
    assert old in src, f"mutation site for {name} not found"
    _sandbox(str(tmp_path), src.replace(old, new, 1))
    r = _run_pins(str(tmp_path))
    assert r.returncode != 0, f"pins did not catch {name}:\n{r.stdout[-2000:]}"


def test_unmutated_copy_passes(tmp_path):
    _sandbox(str(tmp_path), open(os.path.join(ROOT, "oracle", "paged_step.py")).read())
    r = _run_pins(str(tmp_path))
    assert r.returncode == 0, r.stdout[-3000:]
