"""Pins against numbers the pages print for worked examples (tests/golden/page_figures.json, each
entry with its citation): the memory that a materialised score matrix would take, the
list-scheduling example behind the heaviest-first launch order of causal CTAs, and the exp2
emulation's exponent-field trick and polynomial error bound.  CPU only."""
import heapq
import json
import os
import re
import sys

import numpy as np

from workloads import Workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "page_figures.json")))
CSRC = os.path.join(ROOT, "exact_attention_13_gb300", "csrc")


def test_score_matrix_and_output_bytes():
    g = GOLDEN["score_matrix_memory"]
    w = Workload("page", 1, 1, g["N"], g["d"], False, "bf16", 0)
    assert w.score_matrix_bytes(g["elem_bytes"]) == g["score_matrix_bytes"]
    assert w.rows * w.d * g["elem_bytes"] == g["output_bytes"]


def test_long_context_probabilities_against_row_statistics():
    g = GOLDEN["long_context_memory"]
    w = Workload("page", 1, g["H"], g["N"], 128, False, "bf16", 0)
    p_bytes = w.H * w.score_matrix_bytes(g["elem_bytes"])
    stat_bytes = w.rows * g["stat_bytes_per_row"]   # the one fp32 LSE per row this library keeps
    assert p_bytes == g["p_bytes"]
    assert stat_bytes == g["stat_bytes"]
    assert p_bytes // stat_bytes == g["ratio"]


def list_schedule_makespan(durations, n_sm):
    """Greedy list scheduling: tasks go, in the given order, to the SM that frees up first (how the
    hardware hands CTAs of one launch to SMs)."""
    free = [0.0] * n_sm
    heapq.heapify(free)
    for t in durations:
        heapq.heappush(free, heapq.heappop(free) + t)
    return max(free)


def test_lpt_worked_example():
    g = GOLDEN["lpt_worked_example"]
    assert list_schedule_makespan(g["dispatch_order"], g["n_sm"]) == g["makespan"]
    # longest first, the order the causal launch uses, finishes at the lower bound sum / n_sm
    lpt = sorted(g["dispatch_order"], reverse=True)
    assert list_schedule_makespan(lpt, g["n_sm"]) == sum(lpt) / g["n_sm"]


def causal_cta_order(bh, n, tile=128):
    """Key blocks per CTA in launch order for the causal grid (bh, ceil(n / 256)): heads fastest,
    query blocks from the last to the first; a CTA holds two 128-row tiles and runs as long as
    its second tile, which sees one key block more than the first."""
    mblocks = (n + 2 * tile - 1) // (2 * tile)
    order = []
    for y in range(mblocks):
        mblock = mblocks - 1 - y
        for _ in range(bh):
            row1 = mblock * 2 * tile + tile
            last_row = min(row1 + tile, n) - 1 if row1 < n else min(row1, n) - 1
            order.append(last_row // tile + 1)
    return order


def test_causal_work_table_and_launch_order():
    g = GOLDEN["causal_work_table"]
    # block m of 128 queries sees key blocks 0..m
    n = g["query_blocks"] * 128
    assert [m + 1 for m in range(g["query_blocks"])] == g["kv_blocks_per_mblock"]
    order = causal_cta_order(4, n)
    assert order == sorted(order, reverse=True)                 # heaviest first
    assert order[0] == g["query_blocks"] and order[-1] == 2
    # and on 3 SMs it finishes no later than the same CTAs launched lightest first
    assert list_schedule_makespan(order, 3) <= list_schedule_makespan(sorted(order), 3)


def test_exp2_exponent_field_example():
    g = GOLDEN["exp2_exponent_field"]
    bits = np.array([g["value"]], dtype=np.float32).view(np.uint32)[0]
    assert (bits >> 23) & 0xFF == g["exponent_field"] == g["n"] + 127
    # bits(2^n q) = bits(q) + (n << 23) for q in [1, 2) and every normal result
    q = np.float32(1.6875)
    for n in range(-126, 128):
        want = np.float32(np.ldexp(np.float64(q), n)).view(np.uint32)
        assert want == np.uint32(int(q.view(np.uint32)) + (n << 23)), n


def test_exp2_polynomial_meets_page_bound_and_matches_kernel_constants():
    g = GOLDEN["exp2_poly_error"]
    sys.path.insert(0, CSRC)
    try:
        import fit_exp2_poly as fit
    finally:
        sys.path.remove(CSRC)
    coef = [np.float32(c) for c in fit.remez(g["degree"])]
    max_rel, _ = fit.fp32_horner_error(coef)
    assert max_rel <= g["max_rel_error"], max_rel
    # the kernel's constants are the fitted fp32 coefficients
    src = open(os.path.join(CSRC, "sm103_ptx.cuh")).read()
    kernel = [np.float32(float(re.search(rf"kA{i} = ([0-9.e+-]+)f;", src).group(1)))
              for i in (1, 2, 3)]
    assert kernel == coef, (kernel, coef)
