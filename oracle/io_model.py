"""The HBM-traffic and time model printed on the attention-lab page (test infrastructure).

Source: "01 · FlashAttention — Never materialize the N×N score matrix"
(divagr.com attention lab), step 5 "The payoff" and its "show the
accounting" panel:

- standard attention moves 2 N^2 + 4 N d elements across HBM,
- FlashAttention moves 4 N d + 2 N^2 d^2 / M elements, M = elements that fit
  in on-chip SRAM,
- time = elements * bytes_per_element / HBM bandwidth (waiting) plus the
  layer's matmul FLOPs / math throughput (computing), the compute part being
  identical for both schedules.  The page's 55 us at N = 8192, d = 128 and
  312 TFLOP/s fixes the FLOP count at 2 N^2 d.

The page prints, for N = 8192, d = 128, M = 64K elements, 2-byte elements,
2 TB/s and 312 TFLOP/s: 67.1M score entries per head, 138.4M vs 37.7M
elements (3.7x), 138/55/193 us vs 38/55/93 us (2.1x), 72% vs 41% waiting.
"""
from __future__ import annotations


def io_model(N: int, d: int, M: int, bytes_per_elem: int = 2, hbm_bytes_per_s: float = 2e12,
             flops_per_s: float = 312e12) -> dict:
    """Traffic (elements) and modelled time (seconds) of both schedules."""
    std_elems = 2 * N * N + 4 * N * d
    flash_elems = 4 * N * d + 2 * N * N * d * d / M
    flops = 2 * N * N * d
    compute_s = flops / flops_per_s
    std_wait = std_elems * bytes_per_elem / hbm_bytes_per_s
    flash_wait = flash_elems * bytes_per_elem / hbm_bytes_per_s
    std_total = std_wait + compute_s
    flash_total = flash_wait + compute_s
    return {
        "score_entries": N * N,
        "standard_elems": std_elems,
        "flash_elems": flash_elems,
        "traffic_reduction": std_elems / flash_elems,
        "compute_s": compute_s,
        "standard_wait_s": std_wait,
        "flash_wait_s": flash_wait,
        "standard_total_s": std_total,
        "flash_total_s": flash_total,
        "speedup": std_total / flash_total,
        "standard_wait_frac": std_wait / std_total,
        "flash_wait_frac": flash_wait / flash_total,
    }
