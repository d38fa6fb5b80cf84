"""The decode plan's run table for the merged-output decode, checked on the
host against a direct walk of the plan's own schedule: within a worker, the
consecutive items of one request form a run; a run holding all of its
request's nonempty items writes the request's result (-2 on its last item),
any other run writes a part, and a request's parts take consecutive slots in
worker order, listed with the request for the merge.  Requests with no rows
are listed with no parts (their result is O = 0, LSE = -inf)."""

import pytest

import context_long_attention_gb300 as cp


def check_runs(plan):
    B = plan.R
    pairs = plan.pairs
    work = plan.work
    woff = plan.worker_off
    run_out = plan.run_out
    rows = lambda it: int(pairs[int(work[it, 0]), 0])  # noqa: E731
    req = lambda it: int(work[it, 0]) % B  # noqa: E731
    items_of = [0] * B
    for it in range(plan.n_seg):
        if rows(it) > 0:
            items_of[req(it)] += 1
    runs = []  # (request, [items]) in worker order
    for w in range(plan.n_tiles):
        cur = None
        for it in range(int(woff[w]), int(woff[w + 1])):
            if rows(it) == 0:
                assert run_out[it] == -3
                continue
            if cur is not None and cur[0] == req(it):
                cur[1].append(it)
            else:
                cur = (req(it), [it])
                runs.append(cur)
    slots = {}
    for b, its in runs:
        for it in its[:-1]:
            assert run_out[it] == -1
        last = int(run_out[its[-1]])
        if len(its) == items_of[b]:
            assert last == -2
        else:
            assert last >= 0
            slots.setdefault(b, []).append(last)
    listed = {int(b): (int(f), int(n)) for b, f, n in plan.merge_list}
    n_slots = 0
    for b in range(B):
        if b in slots:
            first, n = listed[b]
            assert slots[b] == list(range(first, first + n))
            n_slots += n
        elif items_of[b] == 0:
            assert listed[b] == (0, 0) or listed[b][1] == 0
        else:
            assert b not in listed
    assert plan.n_merge_parts == n_slots
    assert sorted(s for v in slots.values() for s in v) == list(range(n_slots))


@pytest.mark.parametrize("C,ctx,nw", [
    (8, [131072] * 4, 152),
    (8, [1024] * 300, 152),
    (8, [0, 5, 40000, 3, 0, 9000, 131072, 1], 7),
    (4, [257], 1),
    (16, [70000, 1500, 0, 222222], 37),
    (1, [5000, 0, 300], 3),
])
def test_run_table(C, ctx, nw):
    check_runs(cp.cp_decode_plan(C, ctx, n_workers=nw))


@pytest.mark.parametrize("layout", [0, 1])
def test_run_table_layouts_and_rows(layout):
    check_runs(cp.cp_decode_plan_ex(8, [3000, 17, 3, 60000], layout=layout, s_q=3, n_workers=11))
