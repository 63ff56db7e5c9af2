"""Host logic of bench.py that needs no GPU: the whole-job throughput and the
max-over-ranks reduction of the timed region (two gloo ranks on CPU), the
algorithmic byte/FLOP counts against the GEMV page's Table 1, the L2 rotation
rule, and the reference arm's rank handling."""
import json
import os
import socket

import pytest

import bench
from tma_pipelined_tensor_tn_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gemv_bytes_and_flops_match_the_page():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "gemv_table1.json")))
    assert bench.gemv_bytes(g["N"], g["K"]) == g["bytes"]["total"]
    assert 2 * g["N"] * g["K"] == g["flops"]


def test_gemm_counts():
    assert bench.gemm_flops(4096, 4096, 4096) == 2 * 4096 ** 3
    assert bench.gemm_bytes(4096, 4096, 4096) == 2 * 3 * 4096 ** 2


def test_whole_job_value_counts_every_rank():
    # 2 ranks x 10 steps x 5 units in 4 s (the slowest rank's time) = 25 units/s
    assert bench.whole_job_value(5, 10, 2, 4.0) == 25.0


def test_l2_rotation_exceeds_four_times_l2():
    """A set is read again only after at least 4 x L2 bytes of sets (the
    smallest such count)."""
    l2 = 129 * 2 ** 20
    for per_set in (int(bench.gemm_bytes()), int(bench.gemv_bytes()), 10 ** 6):
        n = inputs.l2_rotation_count(per_set, l2)
        assert n >= 2 and n * per_set >= 4 * l2
        assert (n - 1) * per_set < 4 * l2 or n == 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 10.0 - rank, 3.0 * rank]
        got = bench.max_over_ranks(mine)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump(got, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_traffic_capture_survives_comment_edits_not_code_edits():
    src = 'int f(int a) {  // sum\n  /* the body */\n  return a + 1;\n}\n'
    reworded = 'int f(int a) {  // the sum, reworded\n  return a + 1;  /* note */\n}\n'
    changed = 'int f(int a) {  // sum\n  return a + 2;\n}\n'
    assert bench._code_only(src) == bench._code_only(reworded)
    assert bench._code_only(src) != bench._code_only(changed)
    # every committed capture names a kernel whose sources the bench knows
    with open(os.path.join(os.path.dirname(bench.__file__), "profiles", "dram_traffic.json")) as f:
        keys = json.load(f)
    assert keys and all(k.split("@")[0] in bench.KERNEL_SOURCES for k in keys)


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert json.load(open(tmp_path / f"r{r}.json")) == [2.0, 10.0, 3.0]


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks([1, 2.5]) == [1.0, 2.5]


def test_reference_arm_only_rank0_reports(capsys):
    class A:
        steps, warmup = 1, 3
    assert bench.run_reference(A(), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
