"""The stream-K schedule (cfa_sched.cuh) checked on the host.

The persistent forward and dQ kernels split the (query block, key tile)
iterations of every window and KV head evenly over the grid; the same header
compiles for the host, and tests/native/sched_check.cpp walks every CTA's
range and checks coverage, ordering, the head/tail flags and the part lists
the split merges use.  Configurations span the benchmark layers, GQA group
sizes, ragged and empty windows and grids larger than the work.

The same checker also runs the cu_seqlens validation every kernel performs
before it derives a row index from a window (window_valid / seqlens_valid):
well-formed arrays pass, and each malformed one -- a non-zero start, a
decrease, a wrong total, a window longer than the host maximum -- is rejected,
so inconsistent host sizes never reach a load or a store on the GPU.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "native", "sched_check.cpp")
INC = os.path.join(ROOT, "frozen_prefix_chunk_gb300", "csrc")


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path_factory.mktemp("sched") / "sched_check")
    subprocess.check_call([cxx, "-O1", "-std=c++17", "-x", "c++", "-I", INC, SRC, "-o", exe])
    return exe


VARLEN8_LP = [7328, 14558, 6267, 22159, 13492, 16783, 15051, 21922]

CASES = [
    # G, hkv, g, q_per_cta, setup, [(lp, lc), ...]
    (152, 8, 4, 2, 2, [(16128, 256)]),                  # 8B layer, forward tiling
    (152, 8, 4, 1, 2, [(16128, 256)]),                  # 8B layer, dQ tiling
    (149, 8, 4, 1, 2, [(16128, 256)]),                  # dQ beside dK/dV on 3 SMs
    (152, 8, 4, 2, 2, [(lp, 256) for lp in VARLEN8_LP]),
    (150, 8, 4, 1, 2, [(lp, 256) for lp in VARLEN8_LP]),
    (152, 8, 4, 2, 2, [(62976, 512)]),                  # 63k window
    (152, 8, 2, 2, 2, [(1536, 512)]),                   # 1.7B layer
    (152, 1, 2, 1, 2, [(256, 64)]),                     # tiny: fewer iterations than CTAs
    (152, 2, 4, 2, 0, [(5, 37), (0, 100), (700, 0), (128, 256)]),
    (152, 2, 4, 1, 3, [(5, 37), (0, 100), (700, 0), (128, 256)]),
    (7, 4, 1, 2, 2, [(129, 130), (4096, 3)]),
    (13, 2, 3, 1, 2, [(257, 77), (1000, 200)]),
    (152, 1, 8, 2, 2, [(1000, 200)]),
    (1, 2, 4, 2, 2, [(300, 1), (0, 64)]),
    (64, 4, 4, 1, 5, [(1000, 512), (300, 256)]),        # CTA boundaries inside setup iterations
    (40, 8, 4, 1, 4, [(2000, 256), (500, 128), (64, 64)]),
]


# Row mode (every window with the same chunk length; the rows divide the
# grid): G, hkv, g, q_per_cta, setup, nrow, windows
ROW_CASES = [
    (152, 8, 4, 2, 2, 8, [(62976, 512)]),               # 63k window, forward
    (144, 8, 4, 1, 2, 16, [(62976, 512)]),              # 63k window, dQ beside dK/dV on 8 SMs
    (152, 8, 4, 2, 2, 4, [(lp, 256) for lp in VARLEN8_LP]),
    (144, 8, 4, 1, 2, 8, [(lp, 256) for lp in VARLEN8_LP]),
    (152, 8, 4, 2, 2, 4, [(16128, 256)]),               # 8B layer (row mode is legal there too)
    (12, 2, 4, 1, 3, 4, [(5, 128), (0, 128), (700, 128), (128, 128)]),  # short and empty prefixes
    (16, 1, 8, 2, 2, 8, [(100, 256)]),                  # two CTAs per row, tiny rows
    (48, 1, 8, 2, 2, 8, [(0, 256)]),                    # fewer iterations than CTAs in a row
]


def _run(checker, G, hkv, g, qpc, setup, nrow, wins):
    args = [str(x) for x in (G, hkv, g, qpc, setup, nrow, len(wins))]
    for lp, lc in wins:
        args += [str(lp), str(lc)]
    return subprocess.run([checker] + args, capture_output=True, text=True)


@pytest.mark.parametrize("case", ROW_CASES, ids=[str(i) for i in range(len(ROW_CASES))])
def test_row_mode_schedule_covers_every_tile_once(checker, case):
    r = _run(checker, *case)
    assert r.returncode == 0 and r.stdout.startswith("OK"), r.stdout + r.stderr


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_schedule_covers_every_tile_once(checker, case):
    G, hkv, g, qpc, setup, wins = case
    args = [str(x) for x in (G, hkv, g, qpc, setup, 1, len(wins))]
    for lp, lc in wins:
        args += [str(lp), str(lc)]
    r = subprocess.run([checker] + args, capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.startswith("OK"), r.stdout + r.stderr


# (total_lp, total_lc, max_lp, max_lc, cu_seqlens_prefix, cu_seqlens_chunk, valid)
SEQ_CASES = [
    (16128, 256, 16128, 256, [0, 16128], [0, 256], True),
    (700, 393, 700, 256, [0, 5, 5, 705 - 5, 700], [0, 37, 137, 137, 393], True),  # empty windows
    (0, 64, 0, 64, [0, 0], [0, 64], True),                           # no prefix
    (300, 0, 300, 0, [0, 300], [0, 0], True),                        # no chunk rows
    (16128, 256, 16128, 256, [1, 16128], [0, 256], False),           # prefix does not start at 0
    (16128, 256, 16128, 256, [0, 16128], [4, 256], False),           # chunk does not start at 0
    (16128, 256, 16128, 256, [0, 16000], [0, 256], False),           # prefix total differs
    (16128, 256, 16128, 256, [0, 16128], [0, 255], False),           # chunk total differs
    (1000, 200, 1000, 200, [0, 600, 500, 1000], [0, 50, 100, 200], False),  # prefix decreases
    (1000, 200, 1000, 200, [0, 300, 600, 1000], [0, 150, 100, 200], False),  # chunk decreases
    (1000, 200, 400, 200, [0, 300, 800, 1000], [0, 50, 100, 200], False),    # window over max_lp
    (1000, 200, 1000, 64, [0, 300, 600, 1000], [0, 50, 120, 200], False),    # window over max_lc
    (1000, 200, 1000, 200, [0, -5, 600, 1000], [0, 50, 100, 200], False),    # negative entry
    (2147483647, 64, 2147483647, 64, [0, 2147483647], [0, 64], True),        # int32 extremes
    (5, 64, 5, 64, [0, -2147483648 + 2, 5], [0, 32, 64], False),              # wrap-around
]


@pytest.mark.parametrize("case", SEQ_CASES, ids=[str(i) for i in range(len(SEQ_CASES))])
def test_cu_seqlens_validation(checker, case):
    tlp, tlc, mlp, mlc, cp, cc, valid = case
    args = ["seq", str(tlp), str(tlc), str(mlp), str(mlc), str(len(cp) - 1)]
    args += [str(x) for x in cp] + [str(x) for x in cc]
    r = subprocess.run([checker] + args, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == ("VALID" if valid else "INVALID"), (case, r.stdout)
