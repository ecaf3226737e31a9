"""The benchmark's algorithmic flop counts against the per-workload totals
worked out independently for the hot path: forward 4d per (row, visible
key) per query head, backward 2d(3 prompt pairs + 5 response pairs); and
the latent-page rule 2(d_l + d_c) forward, 2(2 d_l + d_c) per pair plus
2(d_l + d_c) per response pair backward."""
import math
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from resident_prefix_attention_gb300 import workloads as W  # noqa: E402


@pytest.mark.parametrize("name,total", [("tiny", 7.89e8), ("mid", 2.869e12),
                                        ("long", 4.446e13),
                                        ("2M", 3.516e14)])
def test_step_flops_match_the_worked_totals(name, total):
    cfg = W.CONFIGS[name]
    fl = bench.step_flops(cfg, cfg.R)
    assert math.isclose(fl["fwd"] + fl["bwd"], total, rel_tol=2e-3)


def test_2M_split_and_dq_kernel_share():
    cfg = W.CONFIGS["2M"]
    fl = bench.step_flops(cfg, cfg.R)
    assert math.isclose(fl["fwd"], 1.406e14, rel_tol=1e-3)
    assert math.isclose(fl["bwd"], 2.110e14, rel_tol=1e-3)
    # the dQ pass runs three products over every visible pair
    assert math.isclose(fl["dq"], 1.5 * fl["fwd"], rel_tol=1e-12)


def test_latent_step_flops_by_hand():
    cfg = W.LATENT_CONFIGS["latent"]
    R, P, Hq, dl, dc = cfg.R, cfg.P, cfg.Hq, cfg.d_l, cfg.d_c
    pairs_r = R * (R + 1) // 2
    pairs = R * P + pairs_r
    fl = bench.latent_step_flops(cfg, R)
    assert fl["fwd"] == 2 * (dl + dc) * pairs * Hq
    assert fl["dq"] == 2 * (2 * dl + dc) * pairs * Hq
    assert fl["bwd"] == (2 * (2 * dl + dc) * pairs + 2 * (dl + dc) * pairs_r) * Hq
    assert math.isclose(fl["fwd"] + fl["bwd"], 4.57e14, rel_tol=2e-3)


def test_block_list_replays_in_reverse_and_covers_the_response():
    blocks = bench.block_list(1000, 3)
    assert [b[0] for b in blocks] == [666, 333, 0]
    assert sum(n for _, n in blocks) == 1000


def test_tensor_rate_from_the_clock():
    """The tensor core's rate is 8192 flop per clock per SM: at 152 SMs and
    2070 MHz that is 2577.5 TFLOP/s, at 1900 MHz 2365.8."""
    clocks = {"sm_mhz": 1900.0, "sm_max_mhz": 2070.0}
    tp = bench.tensor_peaks(clocks)
    scale = tp["sms"] / 152
    assert math.isclose(tp["at_max_clock"], 2577.53088 * scale, rel_tol=1e-9)
    assert math.isclose(tp["at_sampled_clock"], 2365.8496 * scale,
                        rel_tol=1e-9)
    peaks = {"bf16": 1890.7, "bf16_sustained": 1684.3, "source": "measured"}
    r = bench.tensor_roofline("attn_bwd_dq", 1000.0, peaks, clocks, None)
    assert math.isclose(r["frac"], 1000.0 / 1684.3)
    assert math.isclose(r["frac_at_clock"], 1000.0 / tp["at_sampled_clock"])
    pc = bench.peak_pcts(1000.0, peaks, clocks)
    assert math.isclose(pc["pct_nominal_dense_bf16"], 100 * 1000 / 2250)
    assert math.isclose(pc["pct_bf16_peak_burst"], 100 * 1000 / 1890.7)
