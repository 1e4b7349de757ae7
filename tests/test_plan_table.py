"""The measured plan table (csrc/arf_plan_table.inc) on the CPU: every row is
a plan arf_plan_check accepts, the rows of one shape cover disjoint M ranges,
and arf_plan_for_caps returns each row's plan, with the row's grid rule, at
both ends of its range for a device with the row's capabilities."""
import all_reduce_residual_gb300 as arf
from all_reduce_residual_gb300 import plan_table as pt


def _caps(r):
    return arf.DeviceCaps(num_sms=r["num_sms"], max_cluster=r["max_cluster"],
                          max_threads_per_sm=r["max_threads_per_sm"], max_smem_per_block=r["max_smem_per_block"])


def test_table_parses():
    rows = pt.read_table()
    for r in rows:
        assert 1 <= r["m_lo"] <= r["m_hi"] <= (1 << 40) // r["H"], r
        assert r["pattern"] in (arf.ARF_ALLREDUCE, arf.ARF_AR_RESIDUAL_RMSNORM)
        assert r["dtype"] in (arf.ARF_BF16, arf.ARF_FP16)


def test_ranges_are_disjoint_and_contiguous():
    by_key = {}
    for r in pt.read_table():
        key = tuple(r[f] for f in pt.FIELDS[:8])
        by_key.setdefault(key, []).append((r["m_lo"], r["m_hi"]))
    for key, rs in by_key.items():
        rs.sort()
        assert rs[0][0] == 1, key
        for (a_lo, a_hi), (b_lo, b_hi) in zip(rs, rs[1:]):
            assert b_lo == a_hi + 1, (key, rs)


def _fields(p):
    return (p.path, p.threads, p.vpt, p.cluster, p.grid, p.w_spec, p.stages)


def test_planner_returns_each_row_plan():
    """At both ends of each row's range (and inside it) the planner returns the
    row's plan; where that plan is not legal for the M (the flat kAllReduce
    range of rows with H % 8 != 0 needs M * H to be a multiple of 8) it
    returns the closed-form rules' plan instead."""
    for r in pt.read_table():
        caps = _caps(r)
        for M in sorted({r["m_lo"], r["m_lo"] + 1, min(r["m_hi"], 4 * r["m_lo"]), r["m_hi"]} - {r["m_hi"] + 1}):
            if M > r["m_hi"]:
                continue
            row = arf.Plan(*pt.row_plan_fields(r, M))
            legal = arf.arf_plan_check(caps, row, r["pattern"], r["W"], M, r["H"], r["dtype"]) == arf.ARF_OK
            want = arf.Plan()
            if legal:
                want = row
            else:
                assert arf.arf_plan_rules(caps, r["pattern"], r["W"], M, r["H"], r["dtype"], want) == arf.ARF_OK
            got = arf.Plan()
            st = arf.arf_plan_for_caps(caps, r["pattern"], r["W"], M, r["H"], r["dtype"], got)
            assert st == arf.ARF_OK, (r, M)
            assert _fields(got) == _fields(want), (r, M, got)
            assert arf.arf_plan_check(caps, got, r["pattern"], r["W"], M, r["H"], r["dtype"]) == arf.ARF_OK


def test_other_devices_keep_the_rules():
    """A device whose capabilities differ from the table's gets the rule plan."""
    for r in pt.read_table()[:20]:
        caps = _caps(r)
        other = arf.DeviceCaps(num_sms=caps.num_sms - 4, max_cluster=caps.max_cluster,
                               max_threads_per_sm=caps.max_threads_per_sm, max_smem_per_block=caps.max_smem_per_block)
        got = arf.Plan()
        assert arf.arf_plan_for_caps(other, r["pattern"], r["W"], r["m_lo"], r["H"], r["dtype"], got) == arf.ARF_OK
        assert arf.arf_plan_check(other, got, r["pattern"], r["W"], r["m_lo"], r["H"], r["dtype"]) == arf.ARF_OK
