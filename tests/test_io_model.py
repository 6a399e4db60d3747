"""The page-2 traffic/time model reproduces every number the page prints."""
import json
import os

from oracle.io_model import io_model

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "io_model_page2.json")


def test_io_model_reproduces_printed_accounting():
    g = json.load(open(GOLDEN))
    x, p = g["inputs"], g["printed"]
    r = io_model(x["N"], x["d"], x["M"], x["bytes_per_elem"], x["hbm_bytes_per_s"], x["flops_per_s"])
    assert round(r["score_entries"] / 1e6, 1) == p["score_entries_millions_1dp"]
    assert round(r["standard_elems"] / 1e6, 1) == p["standard_elems_millions_1dp"]
    assert round(r["flash_elems"] / 1e6, 1) == p["flash_elems_millions_1dp"]
    assert round(r["traffic_reduction"], 1) == p["traffic_reduction_1dp"]
    assert int(r["standard_total_s"] * 1e6) == p["standard_total_us_int"]
    assert int(r["standard_wait_s"] * 1e6) == p["standard_wait_us_int"]
    assert int(r["compute_s"] * 1e6) == p["compute_us_int"]
    assert round(r["flash_total_s"] * 1e6) == p["flash_total_us_int"]
    assert round(r["flash_wait_s"] * 1e6) == p["flash_wait_us_int"]
    assert round(r["speedup"], 1) == p["speedup_1dp"]
    assert round(100 * r["standard_wait_frac"]) == p["standard_wait_pct_int"]
    assert round(100 * r["flash_wait_frac"]) == p["flash_wait_pct_int"]


def test_io_model_limits():
    # flash traffic grows ~linearly in N at fixed d, M; standard ~quadratically
    a, b = io_model(4096, 128, 65536), io_model(8192, 128, 65536)
    assert 3.8 < b["standard_elems"] / a["standard_elems"] < 4.0
    assert b["traffic_reduction"] > a["traffic_reduction"]
