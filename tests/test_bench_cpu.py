"""Host-side arithmetic of the benchmark on CPU: the attend kernel's
algorithmic bytes (the roofline numerator) counted by hand for small
workloads, the splits-per-request decoding of a work plan, and the parsing
of nvidia-smi clock samples (only those inside the timed region count; the
throttle reasons that were active are reported).  No GPU is involved."""

import datetime
import os

import numpy as np

import bench
import mla_decode_paged_gb300 as mla
from mla_decode_paged_gb300 import workloads as W
from tests import _plan

PARTIAL = 512 * 2 + 4          # one partial row: bf16 o + f32 lse


def test_attend_bytes_by_hand_round_robin():
    """Two requests of 64 and 100 tokens, 12 heads, qlen 1, 4 splits of 25
    tokens: 3 + 4 used splits, one unused split whose LSE is still written."""
    inp = W.make_inputs(0, "cpu")
    assert inp.lengths.tolist() == [64, 100]
    s = bench._plan_stats(inp, 4, 25)
    kv = 164 * 576 + 164 * 4            # KV rows + one page index per token
    meta = 3 * 4                        # indptr
    q = 2 * 12 * 576 * 2                # bf16 query, real heads
    part = 7 * 12 * PARTIAL + 1 * 12 * 4
    assert s["attend_bytes"] == kv + meta + q + part
    assert s["used_units"] == 7 and s["kv_tokens"] == 164
    assert s["attend_flops"] == 2 * 164 * 12 * (576 + 512)


def test_attend_bytes_with_fp8_query_and_block_tables():
    """Block tables of 16 rows: one index per block plus last_page_len per
    request; an fp8 query moves one byte per element."""
    inp = W.make_inputs(0, "cpu")
    s = bench._plan_stats(inp, 4, 25, page_size=16, q_bytes=1)
    blocks = -(-64 // 16) + -(-100 // 16)
    expect = 164 * 576 + 4 * blocks + 4 * 2 + 3 * 4 + 2 * 12 * 576 + 7 * 12 * PARTIAL + 12 * 4
    assert s["attend_bytes"] == expect


def test_attend_bytes_with_a_work_plan():
    """With a plan the used splits are the plan's, and the plan itself is
    read once."""
    inp = W.make_inputs(0, "cpu")
    plan, used = mla.plan_units(inp.lengths, 1, 12, 4, sm_count=2)
    n_r = bench._plan_splits(plan, 2)
    cuts = _plan.ranges(plan, 2)
    assert n_r.tolist() == [len(c) for c in cuts] and max(n_r) == used
    s = bench._plan_stats(inp, used, 0, plan=plan)
    unused = int((used - n_r).sum())
    expect = (164 * 580 + 3 * 4 + 2 * 12 * 576 * 2 + int(n_r.sum()) * 12 * PARTIAL + unused * 12 * 4
              + 4 * plan.numel())
    assert s["attend_bytes"] == expect


def test_attend_bytes_count_empty_requests_once():
    """An empty request reads no KV and writes one LSE row per split slot
    (all -inf) and no partial rows."""
    inp = W.make_inputs(4, "cpu", lengths=[0, 300])
    s = bench._plan_stats(inp, 2, 200)
    rows = 8 * 12                       # qlen 8 x 12 heads per request
    expect = (300 * 580 + 3 * 4 + 2 * rows * 576 * 2
              + 2 * rows * PARTIAL      # request 1: two used splits
              + 2 * rows * 4)           # request 0: its two LSE slots
    assert s["attend_bytes"] == expect


def _line(t, mhz, reasons=("Not Active",) * 4):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return "%s, 0, %d, 2070, 181.13, 0x0000000000000000, %s\n" % (ts, mhz, ", ".join(reasons))


class _Proc:
    def terminate(self):
        pass

    def wait(self):
        return 0


def test_clock_samples_inside_the_timed_region_only(tmp_path):
    c = bench.Clocks(0, str(tmp_path))
    assert os.path.dirname(c.path) == str(tmp_path)
    t0 = 1_800_000_000.0
    with open(c.path, "w") as f:
        f.write(_line(t0, 1000))                                    # before the region
        for k in range(5):
            f.write(_line(t0 + 1 + 0.2 * k, 2070 - k))
        f.write(_line(t0 + 1.4, 1965, ("Not Active", "Not Active", "Not Active", "Active")))
        f.write("garbage line\n")
        f.write(_line(t0 + 5, 500, ("Active",) * 4))                 # after the region
    c.proc, c.f = _Proc(), open(os.devnull, "w")
    c.r0, c.r1 = t0 + 0.9, t0 + 2.0
    r = c.stop()
    assert r["samples"] == 8 and r["samples_in_region"] == 6     # the garbage line is skipped
    assert r["sm_mhz"] == np.median([2070, 2069, 2068, 2067, 2066, 1965])
    assert r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"]


def test_clocks_without_nvidia_smi_say_so(tmp_path):
    c = bench.Clocks(0, str(tmp_path))
    c.proc = None
    assert c.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_smaller_case_of_a_workload():
    """--requests N: the same workload's shapes and distributions with N
    requests, under its own name (so no full-size ncu traffic is taken for
    it); without it the workload as stated."""
    full = bench._spec("ragged_r256_q8_h12")
    small = bench._spec("ragged_r256_q8_h12", 64)
    assert full.requests == 256 and full.name == "ragged_r256_q8_h12"
    assert small.requests == 64 and small.name == "ragged_r256_q8_h12:r64"
    assert (small.qlen, small.heads, small.lengths, small.kv_scale, small.seed) == \
        (full.qlen, full.heads, full.lengths, full.kv_scale, full.seed)
    assert small.zero_requests == full.zero_requests
    assert bench._spec("ragged_r256_q8_h12", 4).zero_requests == 4
    assert bench._ncu_traffic(small.name) is None
