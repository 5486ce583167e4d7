"""The work-stealing group arithmetic of the device scheduler (pgt_sched.cuh, WsGroups:
32-bit formulas for each group's share of the tiles) against oracle.schedule's plain
definitions, on the host: tests/ws_groups_host.cu is compiled with nvcc and run on the CPU."""
import itertools
import os
import shutil
import subprocess

import pytest

from oracle import schedule as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NVCC = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"


@pytest.fixture(scope="module")
def prog(tmp_path_factory):
    if not os.path.exists(NVCC):
        pytest.skip("nvcc not found")
    out = str(tmp_path_factory.mktemp("wsg") / "ws_groups_host")
    cmd = [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1",
           "-I", os.path.join(ROOT, "persistent_gemm_tile_gb300", "csrc"), "-I", os.path.join(ROOT, "include"),
           "-o", out, os.path.join(ROOT, "tests", "ws_groups_host.cu")]
    subprocess.run(cmd, check=True, capture_output=True, timeout=300)
    return out


def device_groups(prog, cases, full=1):
    text = "".join(f"{T} {P} {G} {lay} {full}\n" for (T, P, G, lay) in cases)
    out = subprocess.run([prog], input=text, capture_output=True, text=True, check=True, timeout=120).stdout
    blocks, cur = [], []
    for line in out.splitlines():
        if line == "end":
            blocks.append(cur)
            cur = []
        else:
            _, rest = line.split(":")
            cur.append([int(x) for x in rest.split()])
    return blocks


def test_group_tiles_equal_the_oracle(prog):
    cases = [(T, P, G, lay)
             for T, P, G, lay in itertools.product((0, 1, 5, 37, 76, 240, 304, 1000, 1024), (1, 3, 7, 8, 19, 76, 152),
                                                   (1, 2, 3, 4, 8, 16), (S.WS_RANGES, S.WS_STRIPED))
             if G <= P]
    got = device_groups(prog, cases)
    assert len(got) == len(cases)
    for (T, P, G, lay), g in zip(cases, got):
        assert g == S.ws_group_tiles(T, G, lay, P), (T, P, G, lay)


@pytest.mark.parametrize("G", [3, 64])
def test_group_ranges_at_the_limits(prog, G):
    """P = 65535 (the host's limit for work stealing) and T up to 2^31 - 1: the 32-bit
    products stay exact.  Each group's size, first and last tile against the oracle's
    range bounds."""
    P = 65535
    for T in (2 ** 31 - 1, 2 ** 31 - 7, 32768 * P - 1, 3 * P + 11):  # 32768 P - 1: remainder P - 1
        got = device_groups(prog, [(T, P, G, S.WS_RANGES)], full=0)[0]
        want = [[n, s if n else -1, s + n - 1 if n else -1] for (s, n) in S.ws_partition(T, G, P)]
        assert got == want, T


def test_group_stripes_at_the_worker_limit(prog):
    P, G, T = 65535, 3, 3 * 65535 + 11
    got = device_groups(prog, [(T, P, G, S.WS_STRIPED)], full=0)[0]
    want = [[len(g), g[0], g[-1]] for g in S.ws_group_tiles(T, G, S.WS_STRIPED, P)]
    assert got == want
