"""The pair kernels' launch planner (csrc/pair_plan.h) at several device sizes, on the CPU.

The planner sizes the K split and the pipeline depth from the device it launches on (SM
count and shared memory per SM are queried at run time, not compiled in). A host C++
client compiles the planner header without CUDA and prints its plans; each plan must keep
its launch resident on that device (or fall back to the unsplit plan), split the K blocks
evenly, and fit the block's shared-memory limit -- and a smaller device must not be given a
larger split than it can hold.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "fp8_block_scaled_router_gb300", "csrc")

K_MAX_STAGES = 8


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_client")
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC, os.path.join(HERE, "plan_client.cpp"),
                    "-o", exe], check=True, capture_output=True, text=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=60).stdout
    rows = []
    for line in out.splitlines():
        sms, per_sm, mode, nkb, units, K, split, nst, smem, resident = (int(v) for v in line.split())
        rows.append(dict(sms=sms, per_sm=per_sm, mode=mode, nkb=nkb, units=units, K=K, split=split, nst=nst,
                         smem=smem, resident=resident))
    assert len(rows) == 7 * 12
    return rows


def test_plans_are_valid_on_every_device(plans):
    for r in plans:
        assert r["nkb"] % r["split"] == 0, r
        per = r["nkb"] // r["split"]
        assert 1 <= r["nst"] <= min(per, K_MAX_STAGES), r
        assert r["smem"] <= r["per_sm"] - 1024 or r["split"] == 1, r
        cluster = {3: 8, 11: 4}.get(r["mode"], r["split"])
        fits = r["units"] * cluster <= r["resident"]
        # a split is only chosen when the whole launch is resident at once
        assert r["split"] == 1 or fits, r


def test_smaller_devices_get_no_larger_split(plans):
    by_case = {}
    for r in plans:
        if r["per_sm"] != 233472:
            continue
        by_case.setdefault((r["mode"], r["nkb"], r["units"]), []).append((r["sms"], r["split"]))
    for case, v in by_case.items():
        v.sort()
        splits = [s for _, s in v]
        assert splits == sorted(splits), (case, v)


def test_decode_gate_up_plan_on_the_full_part_and_a_small_one(plans):
    dec = {r["sms"]: r for r in plans if r["mode"] == 1 and r["units"] == 48 and r["per_sm"] == 233472}
    # 152 SMs: every K block of a unit on its own CTA of an 8-CTA cluster (384 CTAs resident)
    assert dec[152]["split"] == 8 and 48 * 8 <= dec[152]["resident"]
    # 8 SMs cannot hold a split launch: the unsplit plan with two stages
    assert dec[8]["split"] == 1 and dec[8]["nst"] == 2
    assert dec[38]["split"] < dec[152]["split"]


TMEM_COLS = {10: 256, 11: 128}  # MXFP4 gate/up, down: columns one CTA allocates


def test_mxfp4_plans_keep_tmem_within_the_sm(plans):
    """No more MXFP4 CTAs of one launch fit on an SM (by shared memory, even without the
    per-block reserve) than its 512 TMEM columns hold, on every device."""
    for r in plans:
        if r["mode"] not in TMEM_COLS:
            continue
        per_sm = r["per_sm"] // r["smem"]
        assert per_sm * TMEM_COLS[r["mode"]] <= 512, r


def test_mxfp4_decode_plan_splits_on_the_full_part(plans):
    mx = {r["sms"]: r for r in plans if r["mode"] == 10 and r["units"] == 24 and r["per_sm"] == 233472}
    assert mx[152]["split"] == 8 and 24 * 8 <= mx[152]["resident"]
    tiny = [r for r in plans if r["mode"] == 10 and r["nkb"] == 2 and r["per_sm"] == 233472 and r["sms"] == 152]
    assert tiny and tiny[0]["split"] == 2 and tiny[0]["nst"] == 1
