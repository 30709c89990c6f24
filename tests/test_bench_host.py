"""Host-side logic of bench.py: clock-record parsing, the max-over-ranks
timing reduction on world_size 2 (gloo, CPU) and the reference arm's JSON."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_clock_summary_parses_reasons():
    c = bench.ClockSampler(0)
    c.lines = ["0, 1900, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active",
               "0, 1950, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1800, 2070, 980.0, 0x0, Not Active, Active, Not Active, Not Active",
               "garbage"]
    s = c.summary()
    assert s["sm_mhz"] == 1900 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    dist.init_process_group("gloo", rank=rank, world_size=2)
    v = bench.max_over_ranks(dist, 10.0 + rank * 5.0, "cpu")
    bench.barrier(dist)
    q.put((rank, v))
    dist.destroy_process_group()


def test_max_over_ranks_world2_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = dict(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
    assert got == {0: 15.0, 1: 15.0}


def test_reference_arm_prints_one_json_line(tmp_path):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--workload", "tiny-gqa-s1k",
                        "--cpu-seconds", "1"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True, env=env,
                       timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_recorded_traffic_follows_kernel_sources(monkeypatch):
    """The committed ncu DRAM record is reported only for the kernel sources it
    was taken on; any other source hash gives null traffic."""
    rec = json.load(open(os.path.join(ROOT, "profiles", "roofline_traffic.json")))
    ent = rec["kernels"]["ring_bwd_kernel"]["llama3-8b-s128k"]["rank-major"]
    # the small-case capture scaled by tile iterations: Hkv * G * nt(nt+1)/2, nt = S/128
    from head_context_attention_gb300 import inputs
    w = inputs.WORKLOADS["llama3-8b-s128k"]
    tiles = lambda S: w.hkv * (w.hq // w.hkv) * (S // 128) * (S // 128 + 1) // 2
    small = ent["measured_s16384"]
    assert small["tile_iterations"] == tiles(16384)
    want = (small["dram_read_bytes"] + small["dram_write_bytes"]) * tiles(w.seqlen) / tiles(16384)
    assert ent["dram_bytes_per_launch"] == round(want)
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["source_sha256"])
    assert bench.recorded_traffic("ring_bwd_kernel", "llama3-8b-s128k") == ent["dram_bytes_per_launch"]
    assert bench.recorded_traffic("ring_bwd_kernel", "no-such-workload") is None
    assert bench.recorded_traffic("ring_bwd_kernel", "llama3-8b-s128k", "no-such-layout") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 64)
    assert bench.recorded_traffic("ring_bwd_kernel", "llama3-8b-s128k") is None


@pytest.mark.parametrize("placement", [0, 1])
@pytest.mark.parametrize("seqlen,cp", [(1024, 4), (131072, 16), (96, 3)])
def test_rank_pairs_match_the_oracle_schedule(placement, seqlen, cp):
    """The bench's per-rank work count (closed form) equals the oracle's count
    over the rank's token positions."""
    from head_context_attention_gb300 import inputs
    from oracle import schedule
    w = inputs.WORKLOADS["tiny-gqa-s1k"].with_(seqlen=seqlen, cp=cp, ring_inner=cp, ring_outer=1)
    for c in range(cp):
        assert bench.rank_pairs(w, placement, c) == schedule.pair_work(seqlen, cp, c, placement)


def test_kernel_source_hash_ignores_comments(tmp_path, monkeypatch):
    src = tmp_path / "head_context_attention_gb300" / "csrc"
    src.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES:
        (src / f).write_text("int a = 1;  // one\n\nint b = 2;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (src / bench.KERNEL_SOURCES[0]).write_text("// a new comment\nint a = 1;  // changed\n   \nint b = 2;\n")
    assert bench.kernel_source_hash() == h0
    (src / bench.KERNEL_SOURCES[0]).write_text("int a = 3;\nint b = 2;\n")
    assert bench.kernel_source_hash() != h0


def test_huge_page_share_reads_the_buffer_mappings():
    """The e2e record's huge-page share: a fraction for buffers that start a
    mapping (as loong_host_alloc's do), None for memory that does not."""
    import mmap

    import torch

    if not os.path.exists("/proc/self/smaps"):
        pytest.skip("no /proc/self/smaps")
    m = mmap.mmap(-1, 4 << 20)
    t = torch.frombuffer(m, dtype=torch.uint8)
    t.fill_(1)
    share = bench.huge_page_share([t])
    assert share is not None and 0.0 <= share <= 1.0
    assert bench.huge_page_share([torch.empty(16)[8:]]) is None
    del t
    m.close()
