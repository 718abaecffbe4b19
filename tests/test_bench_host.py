"""Host logic of bench.py on CPU: the multi-rank timing reduction (gloo, world
size 2), the FLOP/byte accounting, the reference arm's rank handling, and the
source-signature guard on stored DRAM figures."""

import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
rank = int(os.environ["RANK"]); world = int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:{port}", rank=rank, world_size=world)
bench.barrier(world)
got = bench.max_over_ranks(1.5 + rank, world)
bench.barrier(world)
print("RESULT", rank, got, flush=True)
dist.destroy_process_group()
"""


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    port = _free_port()
    script = tmp_path / "worker.py"
    script.write_text(WORKER.format(root=ROOT, port=port))
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err
    results = sorted(line.split()[1:] for out, _ in outs for line in out.splitlines()
                     if line.startswith("RESULT"))
    assert results == [["0", "2.5"], ["1", "2.5"]]


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)


def test_flop_and_byte_accounting():
    # 4*B*H*N^2*d, halved for causal
    assert bench.prefill_flops(4, 16, 2048, 128, True) == 4 * 4 * 16 * 2048 ** 2 * 128 / 2
    assert bench.prefill_flops(1, 1, 10, 64, False) == 4 * 100 * 64
    rows = np.array([[0, 0, 0], [0, 0, 9]], np.int64)
    assert bench.rows_flops(rows, 64, True, 10) == 4 * 64 * (1 + 10)
    assert bench.rows_flops(rows, 64, False, 10) == 4 * 64 * 20


def test_reference_arm_only_rank_zero_prints(capsys):
    class A:
        steps, warmup, ref_rows, gpus = 1, 3, 64, 2

    bench.run_reference(A, world=2, rank=1)
    assert capsys.readouterr().out == ""


def test_reference_arm_line(capsys):
    class A:
        steps, warmup, ref_rows, gpus = 1, 3, 64, 1

    bench.run_reference(A, world=1, rank=0)
    import json

    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == "TFLOPS" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["higher_is_better"] is True and line["metric"] == bench.METRIC


def test_clock_summary_parsing():
    c = bench.ClockSampler(0)
    c.out = ("0, 2032, 2032, 900.0, 0x0, Not Active, Not Active, Not Active, Active\n"
             "0, 1900, 2032, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    s = c.summary()
    assert s["sm_mhz"] == 1966.0 and s["sm_max_mhz"] == 2032.0 and s["reasons"] == ["sw_power_cap"]


def test_decode_side_bytes():
    """q/O/LSE/lengths/page-table bytes and the split partials of 256-token splits."""
    got = bench.decode_side_bytes([512, 300, 0], H=2, d=128, max_pages=32)
    assert got["q"] == got["o"] == 3 * 2 * 128 * 2
    assert got["lse"] == 3 * 2 * 4 and got["seqlens"] == 12 and got["page_table"] == 3 * 32 * 4
    assert got["split_partials_written"] == got["split_partials_read"] == (2 + 2 + 0) * 2 * 129 * 4


def test_traffic_figures_need_a_matching_source_signature(tmp_path, monkeypatch):
    """A stored DRAM figure is reported only while its kernel family's source signature matches
    the current sources; stale, unknown and comment lines are ignored."""
    from io_aware_attention_03_b300 import build as b

    good = b.source_signature("prefill")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        f"# kernel bytes signature\nprefill 123 {good}\ndecode 456 000000000000\n"
        f"unknown 7 {good}\n# prefill 9 {good}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic() == {"prefill": 123.0}


def test_source_signature_ignores_comments_and_layout_only():
    """The signature hashes code with comments and whitespace removed: a comment or a line
    break does not change it, a changed token does."""
    from io_aware_attention_03_b300 import build as b

    code = "int f(int x) {\n  return x + 1;  // one\n}\n/* block */"
    same = "int f(int x)\n{ return x + 1; }  // another comment"
    other = "int f(int x) { return x + 2; }"
    assert b._code_only(code) == b._code_only(same)
    assert b._code_only(code) != b._code_only(other)

