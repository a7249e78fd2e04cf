"""The K-split planner (choose_split in csrc/launch.h), compiled with the host
compiler against synthetic device descriptions: every plan it returns must
be feasible and consistent, forced splits must be honoured, and the costed
choices measured on GB300 must come out as measured (no GPU needed)."""
import json
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "w4a16_int4_weight_gemv_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")

DRIVER = r'''
#include <cstdio>
#include "launch.h"
using namespace w4a16;
// args: sms smem_optin smem_per_sm ntiles units warps max_ctas_per_sm forced split_cost
//       smem_per_unit smem_fixed max_clusters
int main(int argc, char** argv) {
    if (argc != 13) return 2;
    int v[12];
    for (int i = 0; i < 12; ++i) v[i] = atoi(argv[i + 1]);
    DeviceInfo dev{v[0], v[1], v[2]};
    const int per_unit = v[9], fixed = v[10], mc = v[11];
    SplitChoice c = choose_split(
        dev, v[3], v[4], v[5], v[6], v[7], v[8],
        [&](int upc, int tg, int wpt, int tpg, int S) { return fixed + per_unit * upc + 64 * tg * wpt * tpg * (S > 1 ? 2 : 1); },
        [&](int S, int) { return mc / S; });
    printf("{\"wpt\": %d, \"S\": %d, \"ctas\": %d, \"tpg\": %d, \"upc\": %d, \"smem\": %d}\n",
           c.wpt, c.S, c.ctas, c.tiles_per_group, c.units_per_cta, c.smem_bytes);
    return 0;
}
'''


@pytest.fixture(scope="module")
def planner(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime.h")):
        pytest.skip("g++ or the CUDA headers are missing")
    d = tmp_path_factory.mktemp("planner")
    src, exe = d / "driver.cpp", d / "driver"
    src.write_text(DRIVER)
    r = subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, "-I", INCLUDE, "-I", CUDA_INC,
                        str(src), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr

    def run(ntiles, units, warps=16, forced=0, split_cost=1, sms=152, optin=232448,
            per_sm=233472, max_ctas=1, per_unit=1024, fixed=4096, max_clusters=152):
        out = subprocess.run([str(exe)] + [str(a) for a in (
            sms, optin, per_sm, ntiles, units, warps, max_ctas, forced, split_cost, per_unit,
            fixed, max_clusters)], capture_output=True, text=True, check=True).stdout
        return json.loads(out)
    return run


CASES = [(20480, 4), (1024, 4), (3584, 4), (1024, 14), (64, 1), (1, 1), (7, 64), (896, 8)]


@pytest.mark.parametrize("ntiles,units", CASES)
def test_plans_are_feasible_and_cover_the_work(planner, ntiles, units):
    p = planner(ntiles, units)
    f = p["wpt"] * p["S"]
    assert p["ctas"] >= 1 and 1 <= p["S"] <= 8 and 16 % p["wpt"] == 0
    assert f <= 32 and (f & (f - 1)) == 0
    assert p["ctas"] % p["S"] == 0 and p["ctas"] <= 152          # one CTA per SM at most
    assert p["smem"] <= 232448
    # every K unit lies in one CTA's slice, every tile in some group
    assert p["upc"] * p["S"] >= units
    clusters, groups = p["ctas"] // p["S"], 16 // p["wpt"]
    assert clusters * groups * p["tpg"] >= ntiles
    if p["S"] > 1:
        assert clusters <= 152 // p["S"]


@pytest.mark.parametrize("forced", [1, 2, 4, 8, 16, 32])
def test_forced_split_is_honoured(planner, forced):
    p = planner(1024, 64, forced=forced)
    assert p["wpt"] * p["S"] == forced
    assert p["S"] <= 8 and p["wpt"] <= 16


def test_measured_choices(planner):
    # one token, 1024-k spans, 16 warps: the vocabulary head (20480 8-row
    # tiles of 4 spans) runs fastest unsplit once a split tile's reduction is
    # charged; square (1024 tiles x 4), up (3584 x 4) and down (1024 x 14)
    # keep an in-CTA split of two -- all as measured
    p = planner(20480, 4)
    assert p["wpt"] * p["S"] == 1
    for ntiles, units in ((1024, 4), (3584, 4), (1024, 14)):
        p = planner(ntiles, units)
        assert (p["wpt"], p["S"]) == (2, 1), (ntiles, units, p)
    # without the reduction charge the vocabulary head would be split
    p = planner(20480, 4, split_cost=0)
    assert p["wpt"] * p["S"] > 1


def test_infeasible_shared_memory_gives_no_plan(planner):
    # a K slice that can never fit one CTA's shared memory: no CTA at all
    p = planner(1024, 64, per_unit=1 << 20)
    assert p["ctas"] == 0
