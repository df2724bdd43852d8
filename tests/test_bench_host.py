"""Host-side logic of bench.py without a GPU: byte accounting, the clock
summary, max-over-ranks timing with two gloo ranks, and the oracle arm."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_byte_accounting():
    T, E = 8192, 2304
    assert bench.bytes_per_launch("topk_fwd", T, E, 4) == T * E * 13
    assert bench.bytes_per_launch("topk_fwd", T, E, 2, bias=True) == T * E * 9 + 4 * E
    assert bench.bytes_per_launch("topk_bwd", T, E, 4) == T * E * 13
    assert bench.bytes_per_launch("aux_fwd", T, E, 4, "softmax") == T * E * 9
    assert bench.bytes_per_launch("aux_fwd", T, E, 4, "sigmoid") == T * E * 13
    assert bench.bytes_per_launch("aux_bwd", T, E, 4) == T * E * 12
    # the headline figure of the router forward: 8192 x 2304 fp32 moves 245 MB
    assert abs(bench.bytes_per_launch("topk_fwd", T, E, 4) / 1e6 - 245.4) < 0.1


def test_clock_summary_parses_samples():
    c = bench.ClockSampler(0)
    c.out = "\n".join([
        "1965, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "1980, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
        "345, 2070, 100.0, 0x1, Not Active, Not Active, Not Active, Not Active",
    ])
    s = c.summary()
    assert s["sm_mhz"] == pytest.approx(1972.5)
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    c.out = ""
    assert c.summary()["samples"] == 0


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    v = bench.max_over_ranks(1.0 + rank * 2.5, world)
    bench.barrier(world)
    q.put((rank, v))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get() for _ in range(2))
    assert got == {0: 3.5, 1: 3.5}


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_next_row_byte_accounting():
    T, E, K = 8192, 2304, 36
    assert bench.next_row_bytes("compact_fwd", T, E, K, 4) == T * E * 4 + T * K * 12
    assert bench.next_row_bytes("expert_maps", T, E, K, 4) == T * K * 16 + (E + 1) * 4
    assert bench.next_row_bytes("aux_loss_fwd", T, E, K, 4) == T * E * 5 + E * 4 + 4
    assert bench.next_row_bytes("aux_loss_bwd", T, E, K, 4) == T * E * 4 + E * 4 + 4
    with pytest.raises(ValueError):
        bench.next_row_bytes("nope", T, E, K, 4)


def test_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    csrc = tmp_path / "score_top_expert_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = 'int f(int a) { return a / 2; }  // halve\n/* block */ const char* s = "//x /*y*/";\n'
    (csrc / "k.cu").write_text(src)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (csrc / "k.cu").write_text("// a new comment\n" + src.replace("// halve", "// half of a"))
    assert bench.kernel_source_hash() == h0
    (csrc / "k.cu").write_text(src.replace("a / 2", "a / 3"))
    assert bench.kernel_source_hash() != h0
    (csrc / "k.cu").write_text(src.replace('"//x /*y*/"', '"//x"'))
    assert bench.kernel_source_hash() != h0  # string literals are code


def test_traffic_needs_a_matching_hash(tmp_path, monkeypatch):
    f = tmp_path / "traffic.json"
    f.write_text('{"kernel_source_hash": "0000", "kernels": {"topk_fwd@w": '
                 '{"dram_bytes_per_launch": 5}}}')
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0000")
    assert bench.traffic_for("topk_fwd", "w") == 5
    assert bench.traffic_for("aux_fwd", "w") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "1111")
    assert bench.traffic_for("topk_fwd", "w") is None
