"""Roofline time-limit oracle (test infrastructure only).

Restates the burn "autotune" page, section "roofline and the hundred thousand
launches": the time limit of a problem is the larger of (operations / peak
compute) and (bytes / peak bandwidth), divided by the level's threshold
(Balanced: 0.8, i.e. 80 % of peak is good enough), plus one launch overhead.
Operations are m*n*(2k-1) (k multiplies and k-1 adds per output, the page's
compute_ops); bytes are both inputs read once plus the output written once.
The page's worked 1024^2 f32 decision pins it: limit 300281 ns.
"""
from __future__ import annotations


def compute_ops(M: int, N: int, K: int, batch: int = 1) -> int:
    return M * N * max(0, 2 * K - 1) * batch


def bytes_moved(M: int, N: int, K: int, ea: int, eb: int, ec: int, batch: int = 1) -> int:
    return (M * K * ea + K * N * eb + M * N * ec) * batch


def time_limit_s(ops: float, peak_ops_per_s: float, nbytes: float, peak_bytes_per_s: float,
                 threshold: float = 0.8, launch_overhead_s: float = 0.0) -> float:
    return max(ops / peak_ops_per_s, nbytes / peak_bytes_per_s) / threshold + launch_overhead_s
