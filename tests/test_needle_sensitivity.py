"""The needle step's comparison is sharp enough to see one lost or repeated KV block.

With N(0, 1) inputs a long row's attention is nearly uniform and a missing 16-key block
moves its output by less than the tolerance.  On the needle step (chosen keys dominate
every row that sees them) the oracle run on a history with one block dropped or
repeated must fail the parity comparison against the true oracle output.  The mistake is
planted in the oracle's input history, on the CPU; the GPU parity test
(test_parity_sensitive_gpu.py) runs the CUDA path on the same step against the true
oracle.
"""
import numpy as np
import pytest

import oracle
from continuous_batching_paged_step_gb300 import workloads as wl

import parity_helpers as ss


@pytest.fixture(scope="module")
def needle():
    inp = wl.make_inputs(wl.long_context_step())
    ni, pos = wl.plant_needles(inp)
    rows = ss.compare_rows(ni)
    want = oracle.step_reference(ni, rows=rows)
    return ni, pos, rows, want


def _picks(inp, pos):
    """(request, block) pairs: first, middle and last cached block holding a needle, in
    every request whose history has at least three such blocks."""
    out = []
    for r, ps in enumerate(pos):
        c = int(inp.context_lens[r])
        bl = sorted(set(p // inp.spec.block_size for p in ps if p < c))
        if len(bl) >= 3:
            out += [(r, bl[0]), (r, bl[len(bl) // 2]), (r, bl[-1])]
    return out


@pytest.mark.parametrize("mode", ["drop", "dup"])
def test_one_block_more_or_less_fails_the_comparison(needle, mode):
    ni, pos, rows, want = needle
    picks = _picks(ni, pos)
    assert len(picks) >= 60
    kinds = set()
    for r, b in picks:
        rr = ss.rows_of_request(ni, r, rows)
        got = ss.mutated_reference(ni, r, b, mode, rr)
        mx, mn = ss.errors(got[rr], want[rr])
        assert not ss.within_tolerance(got[rr], want[rr]), \
            f"request {r} block {b} {mode}: max {mx:.3g} mean {mn:.3g} passes the comparison"
        kinds.add(ni.spec.q_lens[r] > 1)
    assert kinds == {False, True}    # decode rows and prefill chunks both covered


def test_needles_dominate(needle):
    # Every decode row's output is (nearly) the mean of its needles' values: the needle
    # keys carry essentially all of the softmax weight.
    ni, pos, rows, want = needle
    spec = ni.spec
    cu = ni.cu_seqlens_q
    checked = 0
    for r in range(spec.num_reqs):
        if spec.q_lens[r] != 1 or len(pos[r]) < 3:
            continue
        vals = []
        for t in pos[r]:
            arr, i = wl._key_row(ni, r, t, "v")
            vals.append(oracle.bf16_to_f64(arr[i]).reshape(spec.n_kv_heads, spec.head_dim))
        mean_v = np.mean(vals, axis=0)                     # [n_kv, d]
        o = want[int(cu[r])].reshape(spec.n_kv_heads, 4, spec.head_dim)
        assert np.abs(o - mean_v[:, None, :]).max() < 0.1
        checked += 1
    assert checked >= 20


def test_late_peak_moves_the_running_max():
    # On the late-peak step the largest score of a decode row lies in its last quarter
    # and exceeds the first block's largest score by far more than 2^8 in base-2 units,
    # so the kernels' lazily moved maximum has to move mid-row.
    spec = wl.long_context_step()
    inp = wl.plant_late_peak(wl.make_inputs(spec))
    ks, _ = oracle.request_histories(inp, None)
    cu = inp.cu_seqlens_q
    n = 0
    for r in range(spec.num_reqs):
        c = spec.ctx_lens[r]
        if spec.q_lens[r] != 1 or c < 1024:
            continue
        q = oracle.bf16_to_f64(inp.q[int(cu[r])]).reshape(32, 128)[0]
        k = oracle.bf16_to_f64(ks[r]).reshape(-1, 8, 128)[:, 0, :]
        s = (k @ q) / np.sqrt(128.0) * np.log2(np.e)
        assert np.argmax(s) >= 3 * (c + 1) // 4
        assert s.max() - s[:16].max() > 3 * 8
        n += 1
    assert n >= 10
