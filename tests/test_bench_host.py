"""Host-side logic of bench.py (no GPU): the multi-rank timing reduction over
world size 2 (gloo on CPU), the reference arm's rank handling, and the
algorithmic byte / flop accounting against the pages' own figures."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from tests import oracle_pins


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(dist)
    m = bench.max_over_ranks(dist, 10.0 + rank)       # rank-dependent "time"
    r, w, _ = bench.dist_env()
    ref = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0, "cpu_seconds": 0.2})(),
                              r, w) if r != 0 else None
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": m, "rank": r, "world": w, "ref_is_none": ref is None}, f)
    dist.destroy_process_group()


def test_two_rank_max_and_barrier(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert all(x["max"] == 11.0 for x in res)          # max over ranks, seen by all
    assert [x["rank"] for x in res] == [0, 1] and all(x["world"] == 2 for x in res)
    assert res[1]["ref_is_none"]                         # only rank 0 runs the reference


def test_algorithmic_accounting():
    # 1,794 B per (token, head) and two 64 KB states per head: 718 MB per call
    assert bench.BYTES_PER_TOKEN_HEAD == 1794
    assert abs(bench.prefill_bytes() / 1e6 - 718.0) < 0.5
    # decode: 815 MB of traffic per step of 64 x 96 heads
    assert abs(bench.DEC_BYTES_PER_UNIT * 64 * 96 / 1e6 - 815.0) < 1.0
    # the pages put the cost near 127 thousand FLOPs per token (head dim 128,
    # chunk 64): the triangle-aware count used here is within 5 % of that
    g = oracle_pins.golden("kda_cost.json")
    per_token = bench.prefill_flops(g["chunk"], T_=1, H_=1, d=g["d"])
    assert abs(per_token / g["flops_per_token_about"] - 1.0) < 0.05
    # one state is 64x the KV of a token (snapshot break-even, p4)
    assert g["state_numbers_per_head"] // g["kv_numbers_per_token"] == \
        g["snapshot_break_even_tokens"]


def test_reference_arm_line(capsys):
    rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3",
                     "--cpu-seconds", "0.2"])
    assert rc == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
    assert line["metric"] == bench.METRIC


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_code_hash_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("// head\n__global__ void k(int* x) { x[0] = 1; /* one */ }\n")
    h = bench.code_sha16(str(a))
    a.write_text("// another head\n__global__ void k(int* x) {\n  x[0] = 1;  // one\n}\n")
    assert bench.code_sha16(str(a)) == h
    a.write_text("__global__ void k(int* x) { x[0] = 2; }\n")
    assert bench.code_sha16(str(a)) != h


def test_measured_traffic_follows_the_code(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.code_sha16(str(src))
    (prof / "k.md").write_text(
        "notes\n"
        f"traffic: kernel=k bytes_per_launch=1234 source=k.cu code_sha16={h}\n"
        "traffic: kernel=old bytes_per_launch=99 source=k.cu code_sha16=0000000000000000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic() == {"k": 1234.0}
    src.write_text("__global__ void k() { int a = 0; }\n")   # the kernel changed
    assert bench.measured_traffic() == {}


def test_nvml_sampler_summary():
    """The clock summary from (SM MHz, clock-event reason bits) samples: the
    median of the loaded samples, and the named reasons that were set."""
    import bench
    nv = bench.NvmlSampler.__new__(bench.NvmlSampler)
    nv.max_mhz = 2070.0
    nv.samples = []
    assert nv.summary() is None
    nv.samples = [(2070.0, 0), (2055.0, 0x4), (2070.0, 0x1), (400.0, 0)]
    s = nv.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 4
    assert s["reasons"] == ["sw_power_cap"]
    nv.samples = [(1500.0, 0x8 | 0x40)]
    assert nv.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
