"""Host-side checks of the trace scheduler (no GPU): budget and ordering rules, block
accounting through the C-ABI allocator, and the step counts the pages print for static
versus continuous batching."""
import numpy as np
import pytest

from continuous_batching_paged_step_gb300 import workloads as wl

FAKE_K, FAKE_V = 0x7F0000000000, 0x7F8000000000


@pytest.fixture(scope="module")
def kp():
    from continuous_batching_paged_step_gb300 import build
    build.build()
    from continuous_batching_paged_step_gb300 import kvpaged
    return kvpaged


def _sched(kp, trace, ts, pool_blocks):
    from continuous_batching_paged_step_gb300.trace import Scheduler
    h = kp.kv_pool_create(FAKE_K, FAKE_V, num_blocks=pool_blocks)
    shared = [int(b) for b in kp.kv_block_alloc(h, ts.shared_prefix // 16)]
    s = Scheduler(trace, ts, shared, lambda n: kp.kv_block_alloc(h, n), lambda ids: kp.kv_block_ref(h, ids),
                  lambda ids: kp.kv_block_free(h, ids))
    return h, s


def _replay(s, max_steps=100000):
    plans = []
    while not s.finished() and s.step < max_steps:
        p = s.plan()
        plans.append([(rs.req.rid, c, q, rs.state) for rs, c, q in p.entries])
        s.commit(p)
    return plans


def test_trace_rules_and_block_accounting(kp):
    ts = wl.TraceSpec(name="t", n_requests=60, arrivals_per_step=3.0, shared_prefix=64, prompt_median=40,
                      prompt_cap=300, output_median=12, output_range=(3, 40), budget=128, pool_blocks=4096, seed=7)
    trace = wl.make_trace(ts)
    h, s = _sched(kp, trace, ts, ts.pool_blocks)
    try:
        free0 = kp.kv_pool_num_free(h)
        plans = _replay(s)
        assert s.finished() and len(s.done) == len(trace)
        admitted = []
        for plan in plans:
            assert sum(q for _, _, q, _ in plan) <= ts.budget
            kinds = [q == 1 and st == "decode" for _, _, q, st in plan]
            # decode rows come first in the pack
            assert kinds == sorted(kinds, reverse=True)
            admitted += [rid for rid, c, q, st in plan if c == ts.shared_prefix]
        assert admitted == sorted(admitted)          # FCFS
        for rs in s.done:
            r = rs.req
            assert rs.generated == r.output_len
            # chunks are contiguous from the end of the shared prefix and cover the prompt and
            # every generated token but the last
            pos = ts.shared_prefix
            for start, n in rs.chunks:
                assert start == pos
                pos += n
            assert pos == ts.shared_prefix + r.prompt_len + r.output_len - 1
            assert rs.admitted >= r.arrival
        # every request's own blocks came back; the shared prefix is held once
        assert kp.kv_pool_num_free(h) == free0
        assert all(kp.kv_block_refcount(h, b) == 1 for b in s.shared_blocks)
    finally:
        kp.kv_pool_destroy(h)


def test_shared_prefix_refcount_while_running(kp):
    ts = wl.TraceSpec(name="t", n_requests=5, arrivals_per_step=10.0, shared_prefix=32, prompt_median=10,
                      prompt_cap=20, output_median=5, output_range=(5, 5), budget=1000, pool_blocks=256, seed=3)
    trace = wl.make_trace(ts)
    h, s = _sched(kp, trace, ts, ts.pool_blocks)
    try:
        p = s.plan()
        n_admitted = sum(1 for rs, c, q in p.entries if c == ts.shared_prefix)
        # the system holds one reference and every running request one more
        assert all(kp.kv_block_refcount(h, b) == 1 + n_admitted for b in s.shared_blocks)
    finally:
        kp.kv_pool_destroy(h)


def test_figure_11_2_static_vs_continuous(kp):
    # Page "11.2 连续批处理与 PagedAttention", section 11.2.2, Figure 11-2: 8 requests
    # occupying A2 B5 C3 D8 E4 F3 G5 H6 steps on 4 rows.  Static batching: 14 steps, 64 % of
    # the 56 cells useful, E starts at step 9; continuous batching: 12 steps, 75 % useful,
    # E starts at step 3.
    from continuous_batching_paged_step_gb300.trace import static_batch_steps
    steps = [2, 5, 3, 8, 4, 3, 5, 6]
    assert static_batch_steps(steps, 4) == 14
    assert round(sum(steps) / (14 * 4), 2) == 0.64
    ts = wl.TraceSpec(name="fig", n_requests=8, shared_prefix=0, budget=10000, max_num_seqs=4, pool_blocks=256)
    # one-token prompts (a request's first step is its prefill, which yields its first
    # token) and as many output tokens as the figure's steps
    trace = [wl.TraceRequest(i, 0, 1, n) for i, n in enumerate(steps)]
    h, s = _sched(kp, trace, ts, ts.pool_blocks)
    try:
        _replay(s)
        total = max(rs.finished for rs in s.done) + 1
        assert total == 12
        assert round(sum(steps) / (total * 4), 2) == 0.75
        e = next(rs for rs in s.done if rs.req.rid == 4)
        assert e.admitted + 1 == 3                 # steps counted from 1 on the page
        # the static schedule starts E with the second wave
        assert max(steps[:4]) + 1 == 9
    finally:
        kp.kv_pool_destroy(h)


def test_static_batching_useful_fraction():
    # Page "11.2", section 11.2.1: outputs of 10, 50, 200 and 2,000 tokens in one static
    # batch of 4 use 2,260 of 8,000 request-steps, 28.25 %.
    from continuous_batching_paged_step_gb300.trace import static_batch_steps
    lens = [10, 50, 200, 2000]
    steps = static_batch_steps(lens, 4)
    assert steps == 2000 and sum(lens) / (steps * 4) == pytest.approx(0.2825, abs=1e-12)


def test_default_trace_shape():
    tr = wl.make_trace(wl.TraceSpec())
    p = np.array([r.prompt_len for r in tr])
    o = np.array([r.output_len for r in tr])
    assert len(tr) == 512 and p.max() <= 4096 and o.min() >= 10 and o.max() <= 2000
    assert 200 <= np.median(p) <= 320 and 70 <= np.median(o) <= 130
    assert [r.arrival for r in tr] == sorted(r.arrival for r in tr)
