"""Host-side logic of bench.py (no GPU): closed-form work counts against the
oracle, and the multi-process aggregation (barrier + max over ranks) on a
world_size-2 gloo group."""
import os
import socket
import time

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle as O


@pytest.mark.parametrize("S,C", [(64, 2), (128, 4), (256, 8), (96, 3)])
@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
def test_exact_pairs_closed_form_matches_oracle(S, C, layout):
    if layout == "zigzag" and S % (2 * C):
        pytest.skip("zigzag needs S % 2C == 0")
    pos = O.positions(S, C, O.ZIGZAG if layout == "zigzag" else O.CONTIGUOUS)
    want = O.pair_counts(pos).sum(axis=1).tolist()
    assert bench.exact_pairs_per_rank(S, C, layout) == want


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms = [3.0, 5.0][rank]                      # rank 1 is the slow replica
        m = bench.max_over_ranks(ms, world, device="cpu")
        value = bench.job_throughput(1e9, world, m)
        out[rank] = (m, value)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        m, value = out[r]
        assert m == 5.0                              # max over ranks
        assert value == pytest.approx(2e9 / 5e-3)    # units of all ranks over the slowest time


def test_single_rank_is_identity():
    assert bench.max_over_ranks(7.0, 1) == 7.0
    assert bench.job_throughput(10.0, 1, 1000.0) == pytest.approx(10.0)


def test_code_hash_ignores_comments_only():
    """The recorded-traffic check hashes kernel code with comments and
    whitespace removed: a comment edit keeps the hash, a code edit changes it."""
    import bench
    src = 'int f(int a) {  // twice\n  /* body */ return a * 2; }\nconst char *s = "x // y";\n'
    same = 'int f(int a) { // doubled\n  return a * 2;   /* note */ }\nconst char *s = "x // y";\n'
    other = 'int f(int a) { return a * 3; }\nconst char *s = "x // y";\n'
    strings = 'int f(int a) { return a * 2; }\nconst char *s = "x // z";\n'
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)
    assert bench._code_only(src) != bench._code_only(strings)  # string literals are code
    assert len(bench.attn_source_hash()) == 16


def test_tile_counts_brute_force():
    """The sweep's per-rank tile counts equal a per-element brute force of the
    kernel's tile rules (issue a key tile for a 256-row block if any of its keys
    is visible to any of the block's queries; run it unmasked for a 128-row
    query tile if every key is visible to every query of the tile)."""
    import numpy as np
    import bench
    import oracle as O
    for C, S, layout in ((2, 1024, O.ZIGZAG), (4, 2048, O.ZIGZAG), (4, 2048, O.CONTIGUOUS), (3, 1536, O.CONTIGUOUS)):
        pos = O.positions(S, C, layout)
        got = bench.tile_counts_per_rank(pos)
        s = S // C
        for r in range(C):
            c = {"issued": 0, "skipped": 0, "unmasked": 0, "masked": 0}
            for st in range(C):
                kp = pos[(r - st) % C]
                for qb in range(0, s, 256):
                    for kt in range(0, s, 128):
                        vis = kp[kt:kt + 128][None, :] <= pos[r][qb:qb + 256][:, None]
                        if vis.any():
                            c["issued"] += 1
                            for qt in range(qb, min(qb + 256, s), 128):
                                allv = (kp[kt:kt + 128][None, :] <= pos[r][qt:qt + 128][:, None]).all()
                                c["unmasked" if allv else "masked"] += 1
                        else:
                            c["skipped"] += 1
            assert got[r] == c, (C, S, layout, r, got[r], c)


def _smi_line(t, sm, power_cap=False):
    """One line of `nvidia-smi --query-gpu=<ClockSampler.FIELDS> --format=csv,noheader,nounits`."""
    stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t)) + ".%03d" % int(round((t % 1) * 1000) % 1000)
    cap = "Active" if power_cap else "Not Active"
    return f"{stamp}, 0, {sm}, 2070, 950.5, 0x0000000000000004, Not Active, Not Active, Not Active, {cap}"


def test_clock_samples_kept_inside_timed_region():
    t0 = 1_700_000_000.0
    # idle before (low clock), loaded and power-capped inside, idle after
    lines = [_smi_line(t0 + 0.05 * k, 2070 if 4 <= k < 8 else 345, power_cap=(k == 5)) for k in range(12)]
    lines.append("garbage line")
    samples = bench.ClockSampler.parse(lines)
    assert len(samples) == 12
    assert abs(samples[3][0] - (t0 + 0.15)) < 2e-3
    got = bench.ClockSampler.summarise(samples, (t0 + 0.19, t0 + 0.36))
    assert got["samples_in_timed_region"] == 4 and got["samples"] == 4
    assert got["sm_mhz"] == 2070 and got["sm_max_mhz"] == 2070 and got["reasons"] == ["sw_power_cap"]
    # a window no sample fell in: every sample is used, and that is reported
    got = bench.ClockSampler.summarise(samples, (t0 + 100, t0 + 101))
    assert got["samples_in_timed_region"] == 0 and got["samples"] == 12
