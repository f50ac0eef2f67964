"""Oracle of the variant-selection rules -- TEST INFRASTRUCTURE ONLY.

Source [LBG]: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
Optimization via Neural Networks" (press summary page).  Section 2: the
search space is three tile sizes (large, medium, small) times three pipeline
stage counts (2, 3, 4), nine templates; each (M, N, K) sample of the dataset is
labelled with the index of the fastest template.  Section 3: the selector's
inputs are M, N, K and the SM count.  Section 4: the selected template is
compared with a default template.

Readings where the page is silent:
  - variant index = 3 * tile + stage level, tile 0 = small, 1 = medium,
    2 = large, stage level 0, 1, 2.  The page's three stage counts are 2, 3
    and 4 (Ampere multistage templates); on GB300 the levels keep those counts
    for the small and medium tiles and are 4, 5 and 6 for the large tile,
    which is 256 x 256 on a pair of CTAs and halves the shared memory a stage
    costs each SM.  Index 0 is small/2 stages, index 8 is large/6 stages.
  - the default template (not named on the page) is the large tile at the
    middle stage level, index 7.
  - label: the argmin of the measured times, the lowest index on exact ties.
  - the library's stored choice adds a no-regression guard: keep the default
    unless the label beats it by more than ``keep_within`` (2 %).
  - the dispatch also measures the library's shape-route kernels as
    candidates beside the nine variants and keeps the fastest under the same
    guard; a shape with such a measured pick runs it, any other shape follows
    the library's fixed shape rules.
  - a shape missing from the table takes the entry of the nearest swept
    shape of the same bit width and SM count, distance = sum over M, N, K of
    |log2(x) - log2(x')|, ties to the earlier entry in (M, N, K) order; an
    empty table gives the default.
"""
from __future__ import annotations

import math

NUM_VARIANTS = 9
TILES = ("small", "medium", "large")
STAGE_COUNTS = ((2, 3, 4), (2, 3, 4), (4, 5, 6))  # per tile class, levels 0..2
DEFAULT_VARIANT = 3 * 2 + 1  # large tile, middle stage level


def variant_index(tile: int, stages: int) -> int:
    return 3 * tile + STAGE_COUNTS[tile].index(stages)


def variant_of(index: int) -> tuple[int, int]:
    """(tile class, pipeline stages) of a variant index."""
    return index // 3, STAGE_COUNTS[index // 3][index % 3]


def label(times) -> int:
    """Index of the fastest variant; lowest index on exact ties (section 2)."""
    if len(times) != NUM_VARIANTS:
        raise ValueError("need one time per variant")
    best = 0
    for i, t in enumerate(times):
        if t < times[best]:
            best = i
    return best


def table_choice(times, default: int = DEFAULT_VARIANT, keep_within: float = 0.02) -> int:
    """The stored choice: the label, unless the default is within keep_within of it."""
    lab = label(times)
    if times[default] <= times[lab] * (1.0 + keep_within):
        return default
    return lab


def candidate_choice(times, default_index: int = DEFAULT_VARIANT,
                     keep_within: float = 0.02) -> int:
    """The same guard over any list of measured candidates (the nine variants
    first, then the shape-route kernels): the fastest, lowest index on exact
    ties, unless the default is within keep_within of it."""
    best = 0
    for i, t in enumerate(times):
        if t < times[best]:
            best = i
    if times[default_index] <= times[best] * (1.0 + keep_within):
        return default_index
    return best


def dispatch(entry, rule):
    """The kernel a call runs: the table's measured (route, param) for the
    exact shape when there is one that runs the operands, else the rule's."""
    return entry if entry is not None else rule


def nearest(entries, M: int, N: int, K: int, default: int = DEFAULT_VARIANT) -> int:
    """Variant for (M, N, K) from a list of ((M', N', K'), variant) entries."""
    best, best_d = default, None
    for (m, n, k), v in sorted(entries, key=lambda e: e[0]):
        d = abs(math.log2(M) - math.log2(m)) + abs(math.log2(N) - math.log2(n)) + \
            abs(math.log2(K) - math.log2(k))
        if best_d is None or d < best_d - 1e-12:
            best, best_d = v, d
    return best
