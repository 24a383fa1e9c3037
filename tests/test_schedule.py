"""The GEMM's kernel choice and schedule, on CPU: fp8lin_gemm_describe_for
runs the same host planning as fp8lin_gemm (tile shape, waves, K split of
few-tile products and of the last wave of long-K products) for a device of a
given SM count, without a GPU.  The expected lines are the ones the GB300
(152 SMs) printed through fp8lin_gemm_describe."""
import ctypes
import random
import re

import pytest

import quantised_gemm_gb300 as q

GB300_SMS = 152


@pytest.fixture(scope="module", autouse=True)
def _built():
    from quantised_gemm_gb300 import build as qb
    qb.build()


LINE = re.compile(
    r"^(?P<kernel>[a-z0-9_]+<[0-9, ]+>): (?P<swap>swap-AB \(D\^T = B\.A\^T\), )?"
    r"(?P<rows>\d+)x(?P<bn>\d+) tiles, (?P<tiles>\d+) tiles on (?P<used>\d+) of (?P<slots>\d+) "
    r"(?P<unit>CTAs|CTA pairs), (?P<sched>.+)$")


@pytest.mark.parametrize("mnk,kernel,sched", [
    ((16, 4096, 4096), "gemm_fp8_kernel<16, 8, 1>", "K split 4 ways"),
    ((48, 208, 160), "gemm_fp8_kernel<64, 8, 1>", "whole tiles"),
    ((128, 4096, 4096), "gemm_fp8_kernel<256, 4, 0>", "K split 8 ways"),
    ((128, 1600, 512), "gemm_fp8_kernel<256, 4, 0>", "whole tiles"),
    ((96, 128, 512), "gemm_fp8_kernel<128, 6, 0>", "whole tiles"),
    ((384, 1600, 1600), "gemm_fp8_pair_kernel<256, 6, 8>", "whole tiles"),
    ((512, 128, 1024), "gemm_fp8_pair_kernel<128, 8, 8>", "whole tiles"),
    ((4096, 4096, 65536), "gemm_fp8_pair_kernel<256, 6, 4>", "last 28 tiles K split 2 ways"),
    ((4096, 4096, 4096), "gemm_fp8_pair_kernel<256, 6, 4>", "whole tiles"),
    ((4096, 4096, 1024), "gemm_fp8_pair_kernel<256, 6, 8>", "whole tiles"),
    ((512, 10240, 12288), "gemm_fp8_pair_kernel<256, 6, 4>", "last 4 tiles K split 8 ways"),
])
def test_kernel_and_schedule_on_gb300(mnk, kernel, sched):
    desc = q.gemm_describe_for(*mnk, GB300_SMS)
    assert desc.startswith(kernel + ":") and desc.endswith(sched), desc


def test_headline_products_exactly():
    # the three products of the 65536-token step of the 4096 x 4096 Linear
    assert q.gemm_describe_for(65536, 4096, 4096, GB300_SMS) == (
        "gemm_fp8_pair_kernel<256, 6, 4>: 256x256 tiles, 4096 tiles on 76 of 76 CTA pairs, "
        "whole tiles")
    assert q.gemm_describe_for(4096, 4096, 65536, GB300_SMS) == (
        "gemm_fp8_pair_kernel<256, 6, 4>: 256x256 tiles, 256 tiles on 76 of 76 CTA pairs, "
        "last 28 tiles K split 2 ways")


def _check_line(M, N, K, sms):
    desc = q.gemm_describe_for(M, N, K, sms)
    m = LINE.match(desc)
    assert m, desc
    rows, bn = int(m["rows"]), int(m["bn"])
    tiles, used, slots = int(m["tiles"]), int(m["used"]), int(m["slots"])
    swap = m["swap"] is not None
    pair = m["unit"] == "CTA pairs"
    tm, tn = (N, M) if swap else (M, N)
    assert tiles == -(-tm // rows) * -(-tn // bn), desc
    assert slots == (sms // 2 if pair else sms), desc
    assert rows == (256 if pair else 128), desc
    assert swap == (M <= 64), desc
    assert 1 <= used <= slots, desc
    sched = m["sched"]
    if sched == "whole tiles":
        assert used == min(tiles, slots), desc
    else:
        s = re.match(r"^(?:last (\d+) tiles )?K split (\d+) ways$", sched)
        assert s, desc
        ways = int(s[2])
        assert ways >= 2, desc
        split = int(s[1]) if s[1] else tiles
        assert 1 <= split <= tiles, desc
        # the slices of a split tile run side by side, never more than the slots
        assert split * ways <= slots, desc
        assert used == min(tiles - split + split * ways, slots), desc
        if s[1]:
            # a tail split: whole waves first, the last one at most half full
            assert split == tiles % slots and 0 < split <= slots // 2, desc
        else:
            assert tiles < slots, desc            # few-tile split: under one wave
    return desc


def test_schedule_invariants_random_shapes():
    rng = random.Random(1234)
    for _ in range(400):
        M = 16 * rng.randint(1, 4096)
        N = 16 * rng.randint(1, 1024)
        K = 16 * rng.randint(1, 8192)
        for sms in (GB300_SMS, 148, 132):
            _check_line(M, N, K, sms)


@pytest.mark.parametrize("sms", [152, 148, 132, 2])
def test_schedule_invariants_pinned_shapes(sms):
    for mnk in [(16, 4096, 4096), (256, 4096, 4096), (4096, 4096, 4096), (65536, 4096, 4096),
                (4096, 4096, 65536), (12288, 4800, 1600), (1600, 1600, 12288),
                (8192, 14336, 4096), (4096, 14336, 8192)]:
        _check_line(*mnk, sms)


def test_describe_for_rejects_bad_arguments():
    lib = q.library()
    buf = ctypes.create_string_buffer(64)
    assert lib.fp8lin_gemm_describe_for(-1, 16, 16, 152, buf, len(buf)) == 1   # EINVAL
    assert lib.fp8lin_gemm_describe_for(16, 16, 16, 1, buf, len(buf)) == 1
    assert lib.fp8lin_gemm_describe_for(16, 16, 16, 152, None, 64) == 1
    assert lib.fp8lin_gemm_describe_for(16, 16, 16, 152, buf, 0) == 1
    small = ctypes.create_string_buffer(8)          # truncated, still terminated
    assert lib.fp8lin_gemm_describe_for(65536, 4096, 4096, 152, small, len(small)) == 0
    assert small.value == b"gemm_fp"


GROUP = re.compile(
    r"^(?P<use>grouped|separate): (?P<t0>\d+) \+ (?P<t1>\d+) tiles \(K blocks (?P<kb0>\d+), "
    r"(?P<kb1>\d+)\), d = (?P<d>\d+); busiest pair (?P<g>\d+) K blocks grouped, (?P<a>\d+) alone; "
    r"(?P<epi>4|8) epilogue warps$")


def _backward_group(M, K, N, sms=GB300_SMS):
    """The plan for a Linear's backward: dX = dY8 . W8 ([M, K], K loop N) and
    dW = dY8^T . x8 ([N, K], K loop M)."""
    return q.gemm_group_describe_for((M, K, N), (N, K, M), sms)


@pytest.mark.parametrize("mkn,use,tiles,kb", [
    ((4096, 4096, 4096), "grouped", (256, 256), (32, 32)),      # 3.37 + 3.37 rounds -> 7 rounds
    ((12288, 1600, 1600), "grouped", (49, 336), (96, 13)),     # dW's long loop first
    ((65536, 4096, 4096), "separate", (256, 4096), (512, 32)),  # 2.4% estimated: not enough
    ((8192, 4096, 14336), "separate", (512, 896), (112, 64)),
    ((12288, 1600, 4800), "grouped", (133, 336), (96, 38)),
    ((1040, 784, 512), "grouped", (8, 20), (9, 4)),            # under one round
])
def test_group_plan_on_gb300(mkn, use, tiles, kb):
    desc = _backward_group(*mkn)
    m = GROUP.match(desc)
    assert m, desc
    assert m["use"] == use
    assert (int(m["t0"]), int(m["t1"])) == tiles and (int(m["kb0"]), int(m["kb1"])) == kb


def test_group_plan_separate_when_not_both_pair256():
    # dX of a 16-token step runs on the swapped narrow tiles
    assert _backward_group(16, 4096, 4096).startswith("separate: not both")


def test_group_deal_covers_every_tile_once():
    rng = random.Random(4321)
    shapes = [(4096, 4096, 4096), (12288, 1600, 4800), (12288, 1600, 1600), (12288, 6400, 1600),
              (8192, 4096, 14336), (8192, 14336, 4096), (65536, 4096, 4096), (256, 4096, 4096)]
    shapes += [(256 * rng.randint(1, 64), 256 * rng.randint(1, 32), 256 * rng.randint(1, 64))
               for _ in range(150)]
    shapes += [(16 * rng.randint(17, 1024), 16 * rng.randint(17, 512), 16 * rng.randint(1, 2048))
               for _ in range(150)]
    for M, K, N in shapes:
        for sms in (GB300_SMS, 148, 132, 4):
            desc = _backward_group(M, K, N, sms)
            assert "DEAL BROKEN" not in desc, (M, K, N, sms, desc)
            m = GROUP.match(desc)
            if m is None:
                assert desc.startswith("separate: not both"), desc
                continue
            assert int(m["kb0"]) >= int(m["kb1"]), desc              # problem 0: the longer loop
            units, kb_min = int(m["t0"]) + int(m["t1"]), int(m["kb1"])
            assert m["epi"] == ("4" if units >= sms // 2 and kb_min >= 12 else "8"), desc
            assert (m["use"] == "grouped") == (int(m["g"]) * 100 < int(m["a"]) * 92), desc
            # the busiest pair does at least its share of all K blocks
            total = int(m["t0"]) * int(m["kb0"]) + int(m["t1"]) * int(m["kb1"])
            assert int(m["g"]) * (sms // 2) >= total, desc


def test_group_describe_rejects_bad_arguments():
    lib = q.library()
    buf = ctypes.create_string_buffer(64)
    assert lib.fp8lin_gemm_group_describe_for(0, 16, 16, 16, 16, 16, 152, buf, len(buf)) == 1
    assert lib.fp8lin_gemm_group_describe_for(16, 16, 16, 16, 16, 16, 1, buf, len(buf)) == 1
    assert lib.fp8lin_gemm_group_describe_for(16, 16, 16, 16, 16, 16, 152, None, 64) == 1
    assert lib.fp8lin_gemm_group_describe_for(16, 16, 16, 16, 16, 16, 152, buf, 0) == 1


@pytest.mark.parametrize("mnk,epi", [
    ((65536, 4096, 4096), 4),    # 54 rounds of 32 K blocks: the epilogue hides
    ((4096, 4096, 2048), 4),     # 16 K blocks a tile
    ((4096, 4096, 1024), 8),     # 8: the epilogue shows
    ((4096, 4096, 256), 8),
    ((256, 4096, 4096), 8),      # a few tiles split along K
    ((384, 1600, 1600), 8),      # under one round
])
def test_pair_kernel_epilogue_warps(mnk, epi):
    desc = q.gemm_describe_for(*mnk, GB300_SMS)
    assert desc.startswith("gemm_fp8_pair_kernel<256, 6, %d>:" % epi), desc
