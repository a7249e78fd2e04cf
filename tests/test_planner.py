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


# Kernel 4 (fp16 warp-MMA): choose_hmma_plan picks between 8-warp CTAs (two
# per SM) and 16-warp CTAs (one per SM), each with its cluster K split, WPT
# and ring depth.  Occupancy is modelled as the device does it: CTAs per SM
# limited by shared memory (1 KB reserved per CTA) and by the register file
# (16 warps of 124-register threads).
HMMA_DRIVER = r'''
#include <cstdio>
#include "launch.h"
using namespace w4a16;
// args: M N K forced_S
int main(int argc, char** argv) {
    if (argc != 5) return 2;
    const int M = atoi(argv[1]), N = atoi(argv[2]), K = atoi(argv[3]), forced = atoi(argv[4]);
    DeviceInfo dev{152, 232448, 233472};
    auto occ = [&](int warps) {
        return [&dev, warps](int S, int smem) {
            int per_sm = dev.smem_per_sm / (smem + 1024);
            const int reg_cap = 16 / warps;
            if (per_sm > reg_cap) per_sm = reg_cap;
            return per_sm * dev.sms / S;
        };
    };
    HmmaChoice c = choose_hmma_plan(dev, M, N, K, forced, occ(kHmmaWarpsPaired), occ(kHmmaWarpsWide));
    const HmmaLayout L = hmma_layout(c.warps > 0 ? c.warps : 8, M, c.steps_per_rank > 0 ? c.steps_per_rank : 1,
                                     c.S > 0 ? c.S : 1, c.max_tiles, c.depth > 0 ? c.depth : 2);
    printf("{\"warps\": %d, \"S\": %d, \"nclusters\": %d, \"sps\": %d, \"max_tiles\": %d, \"wpt\": %d, "
           "\"depth\": %d, \"smem\": %d, \"per_sm\": %d, \"layout_total\": %d}\n",
           c.warps, c.S, c.nclusters, c.steps_per_rank, c.max_tiles, c.wpt, c.depth, c.smem_bytes,
           c.per_sm, L.total);
    return 0;
}
'''


@pytest.fixture(scope="module")
def hmma_planner(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime.h")):
        pytest.skip("g++ or the CUDA headers are missing")
    d = tmp_path_factory.mktemp("hmma_planner")
    src, exe = d / "driver.cpp", d / "driver"
    src.write_text(HMMA_DRIVER)
    r = subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, "-I", INCLUDE, "-I", CUDA_INC,
                        str(src), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr

    def run(M, N, K, forced=0):
        out = subprocess.run([str(exe), str(M), str(N), str(K), str(forced)],
                             capture_output=True, text=True, check=True).stdout
        return json.loads(out)
    return run


HMMA_SHAPES = [(1, 4096, 4096), (1, 14336, 4096), (1, 4096, 14336), (1, 163840, 4096),
               (1, 28672, 4096), (1, 1, 512), (1, 17, 512), (2, 257, 2048), (8, 150, 4096),
               (8, 14336, 4096), (4, 4096, 14336), (1, 64, 14336), (8, 33, 8192),
               (16, 14336, 4096), (12, 28672, 4096), (16, 8192, 8192), (9, 200, 4096)]


@pytest.mark.parametrize("M,N,K", HMMA_SHAPES)
def test_hmma_plans_are_feasible_and_cover_the_work(hmma_planner, M, N, K):
    p = hmma_planner(M, N, K)
    assert p["warps"] in (8, 16) and p["nclusters"] >= 1
    S, wpt = p["S"], p["wpt"]
    assert S in (1, 2, 4, 8) and (K // 512) % S == 0 and p["sps"] * S == K // 512
    assert wpt in (1, 2, 4, 8, 16) and p["warps"] % wpt == 0
    assert 2 <= p["depth"] <= 6
    ntiles = (N + 15) // 16
    assert p["nclusters"] * p["max_tiles"] >= ntiles            # every tile has a cluster
    assert p["nclusters"] <= ntiles
    assert p["smem"] == p["layout_total"] <= 232448             # the layout the kernel uses
    # the residency the plan claims is what the modelled occupancy gives
    fit = min(233472 // (p["smem"] + 1024), 16 // p["warps"])
    assert p["per_sm"] <= fit
    assert p["nclusters"] * S <= 152 * fit


def test_hmma_measured_width_choices(hmma_planner):
    # measured on GB300, one token: 8-warp pairs for the short runs (square,
    # MLP up and down), 16-warp CTAs for the 28672 x 4096 projection and the
    # vocabulary head
    for shape in ((1, 4096, 4096), (1, 14336, 4096), (1, 4096, 14336)):
        p = hmma_planner(*shape)
        assert p["warps"] == 8 and p["per_sm"] == 2, (shape, p)
    for shape in ((1, 28672, 4096), (1, 163840, 4096)):
        p = hmma_planner(*shape)
        assert p["warps"] == 16 and p["per_sm"] == 1, (shape, p)


def test_hmma_measured_split_choices(hmma_planner):
    # the K splits that timed fastest on GB300 for one token: in-CTA parts
    # rather than clusters where K allows (square 4 parts; the vocabulary head
    # and 81920 x 4096 two parts, where four or eight cost part 0 more adds
    # than they save), and a cluster pair with two parts each for the MLP down
    # projection (4096 x 14336), which keeps two CTAs per SM
    def split(shape):
        p = hmma_planner(*shape)
        return p["S"], p["wpt"]
    assert split((1, 4096, 4096)) == (1, 4)
    assert split((1, 163840, 4096)) == (1, 2)
    assert split((1, 81920, 4096)) == (1, 2)
    assert split((1, 4096, 14336)) == (2, 2)


@pytest.mark.parametrize("M,N,K", [(1, 28672, 4096), (2, 6000, 14336), (3, 28672, 4096),
                                   (8, 12000, 4096)])
def test_hmma_wide_parity_shapes_plan_16_warps(hmma_planner, M, N, K):
    # the GPU parity cases of the 16-warp instantiations rely on these plans
    assert hmma_planner(M, N, K)["warps"] == 16


@pytest.mark.parametrize("forced", [1, 2, 4, 8])
def test_hmma_forced_cluster_split(hmma_planner, forced):
    p = hmma_planner(1, 4096, 8192, forced)
    assert p["S"] == forced
    # a split that does not divide K / 512 gives no plan
    assert hmma_planner(1, 4096, 1536, 4)["nclusters"] == 0


def test_hmma_sixteen_token_plans_take_short_slices(hmma_planner):
    # 9..16 tokens (two MMA tiles): K slices of at most 2048 k where they fit,
    # one CTA per SM; the MLP down projection (28 steps of 512 k) has no
    # plan at 4096 rows (the library then takes the bf16 kernel)
    for shape, S in (((16, 14336, 4096), 2), ((12, 28672, 4096), 2), ((16, 8192, 8192), 4)):
        p = hmma_planner(*shape)
        assert p["S"] == S and p["sps"] <= 4 and p["per_sm"] == 1, (shape, p)
    assert hmma_planner(16, 4096, 14336)["nclusters"] == 0
    # where no short slice fits, any slice that does (a small matrix)
    assert hmma_planner(16, 33, 14336)["nclusters"] > 0
