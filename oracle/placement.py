"""Placement arithmetic -- oracle.

* Tile rows: [DAK] section 4.1 "Data Partition" cuts A (M x K) along M into tile rows of
  m x K. T = ceil(M / m) tile rows; an offload ratio x puts h tile rows in host memory.
  The page does not say how x is rounded to whole tiles; the reading used here is
  h = ceil(x * T), so that at least the fraction x of the rows leaves HBM (the capacity
  constraint), with tile rows 0 .. h-1 on the host (Fig. 5a shows tile row 0 on the host).
* Requests: [DAK] section 5 splits the KV cache by request; h_r = ceil(x * B) requests
  go to the host, requests 0 .. h_r-1.
* Global ratio: [DAK-explainer], section on why offloading is more than moving overflow
  to the CPU: x_global >= max(0, (M - H) / M) for footprint M and HBM capacity H,
  workspace ignored.
* Host-link traffic: [DAK] section 4.3.2 and Table 1: host memory is not cached in the GPU
  L2, so every CTA that reads a host tile moves its bytes over the link again. With
  output tiles n_tile columns wide, each host tile row is read once per column tile:
  traffic = host_bytes * ceil(N / n_tile).

Parity pins (tests/test_oracle_planner.py, placement section): Table 1's five rows (98 MiB host matrix,
n_tile = 256), Fig. 10's and Fig. 14's global ratios from footprint and H = 96 GB, and
the tile-count edge cases (x = 0, x = 1, ragged last tile).
"""
import math


def n_tiles(M: int, tile_m: int) -> int:
    return -(-int(M) // int(tile_m))


def n_host_tiles(x: float, M: int, tile_m: int) -> int:
    """h = ceil(x * T) tile rows on the host, clamped to [0, T]."""
    T = n_tiles(M, tile_m)
    h = math.ceil(x * T - 1e-12)
    return max(0, min(T, h))


def n_host_requests(x: float, batch: int) -> int:
    h = math.ceil(x * batch - 1e-12)
    return max(0, min(batch, h))


def global_ratio(footprint: float, hbm_capacity: float) -> float:
    """x_global = max(0, (M - H) / M)."""
    if footprint <= 0:
        return 0.0
    return max(0.0, (footprint - hbm_capacity) / footprint)


def host_link_traffic(host_bytes: float, N: int, n_tile: int) -> float:
    """Bytes crossing the host link when every column tile re-reads the host rows."""
    return float(host_bytes) * (-(-int(N) // int(n_tile)))


def tier_roofline(total_bytes: float, x: float, b_host: float, b_hbm: float) -> float:
    """Tier-aggregate roofline R(x) = C / max(x C / B_host, (1 - x) C / B_hbm) in bytes/s.

    [DAK] section 4.2.1: for a memory-bound operation the memory time is the slower of
    the two concurrent transfers, T_mem = max(T_h, T_g)."""
    t = max(x * total_bytes / b_host, (1.0 - x) * total_bytes / b_hbm)
    return total_bytes / t if t > 0 else float("inf")
