"""The decode runner's rotating plan buffers (host logic, no GPU).

Each one-call decode step writes its plan (slots, copy pairs, table, lengths)
into one of a few pinned host buffer sets, and its kernels read that set in
place later, on the device's schedule. A set must therefore not be written
again before the kernels that read it have run. The runner marks, at every
step, the work enqueued so far with an event and waits on the mark left on
the set it is about to write. These tests drive that logic with a fake event
and stream that log the order of records, waits, plan writes and launches,
and check the rule on the log for one, two and three sets."""

import pytest

from paged_kv_cache_40_gb300.engine import DecodeBatchRunner


class _Log:
    def __init__(self):
        self.items = []


class _FakeEvent:
    def __init__(self, log, name):
        self.log, self.name, self.recorded = log, name, None

    def record(self, stream):
        # the mark covers every launch enqueued so far on the stream
        self.recorded = len(stream.launched)
        self.log.items.append(("record", self.name, self.recorded))

    def synchronize(self):
        self.log.items.append(("wait", self.name, self.recorded))


class _FakeStream:
    def __init__(self):
        self.launched = []


def _runner(sets):
    log, stream = _Log(), _FakeStream()
    r = object.__new__(DecodeBatchRunner)
    r._plan_sets = [object() for _ in range(sets)]
    r._plan_marks = [_FakeEvent(log, i) for i in range(sets)]
    r._plan_marked = [False] * sets
    r._plan_next = 0
    r._plan_stream = stream
    return r, log, stream


@pytest.mark.parametrize("sets", [1, 2, 3])
def test_a_set_is_written_only_after_its_readers_ran(sets):
    r, log, stream = _runner(sets)
    last_launch_of = {}   # set -> index of the launch that read it last
    done = set()          # launches known complete (covered by a waited mark)
    for step in range(12):
        k = r._take_plan_set()
        # the marks waited on since the previous step say which launches are complete
        for kind, _, upto in log.items:
            if kind == "wait":
                done.update(range(upto))
        log.items.clear()
        if k in last_launch_of:
            assert last_launch_of[k] in done, (
                f"step {step} rewrites set {k} while launch {last_launch_of[k]} may read it")
        # the step writes set k, then enqueues the kernels that read it
        stream.launched.append(k)
        last_launch_of[k] = len(stream.launched) - 1
    assert r._plan_next == 12


@pytest.mark.parametrize("sets", [2, 3])
def test_no_wait_before_every_set_was_used(sets):
    """The first use of each set waits on nothing (the host may run ahead by
    `sets` - 1 steps), and every later step waits exactly once."""
    r, log, stream = _runner(sets)
    waits = []
    for step in range(3 * sets):
        r._take_plan_set()
        waits.append(sum(1 for kind, *_ in log.items if kind == "wait"))
        log.items.clear()
        stream.launched.append(step)
    assert waits[:sets] == [0] * sets
    assert waits[sets:] == [1] * (2 * sets)
