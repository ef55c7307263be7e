"""Host-side logic of bench.py (no GPU): work counts, the step's new keys,
whole-job aggregation, max over ranks with two gloo ranks, clock parsing."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

import bench
import workloads


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_work_counts_against_brute_force(idx):
    w = workloads.config(idx, small=True)
    c = bench.work_counts(w)
    pages = 0
    for r, s in enumerate(w.dec_seq_lens):
        for i in range(w.query_len):
            pos = int(s) - w.query_len + i
            pages += (pos // 128 if pos >= 0 else 0) * w.num_heads
    dec = pages
    for s, q in zip(w.pre_seq_lens, w.pre_query_lens):
        for i in range(int(q)):
            pos = int(s) - int(q) + i
            pages += (pos // 128 if pos >= 0 else 0) * w.num_heads
    assert c["pages_scored"] == pages and c["dec_pages_scored"] == dec
    assert c["pre_flops"] == (pages - dec) * 2 * 128 * 128


def test_full_size_work_matches_the_stated_figures():
    c = bench.work_counts(workloads.config(4))
    assert c["pre_flops"] == 8904704 * 8 * 2 * 128 * 128          # 2.334 TFLOP per step
    assert c["dec_bytes"] == 16 * 1023 * (9216 + 4) + 16 * (64 * 128 + 64 * 64 + 4)


def test_step_new_tokens():
    w = workloads.config(4, small=True)
    new = bench.step_new_tokens(w)
    assert len(new) == w.num_decode_reqs * w.query_len + int(w.pre_query_lens.sum())
    seq = w.seq_lens.astype(np.int64)
    ends = np.cumsum(seq)
    assert new[w.query_len - 1] == ends[0] - 1                  # last token of request 0
    assert new[-1] == ends[-1] - 1


def test_aggregate_uses_slowest_rank():
    assert bench.aggregate([100, 100], [1.0, 2.0]) == 100.0


def _ranks(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    v = bench.max_over_ranks(1.0 + rank, world, torch.device("cpu"))
    q.put((rank, v))
    tdist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_ranks, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.0, 1: 2.0}


def test_clock_summary_parsing():
    c = bench.ClockSampler(0)
    c.lines = ["1965, 2070, 900.1, Not Active, Not Active, Not Active, Active",
               "1980, 2070, 950.0, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    s = c.summary()
    assert s["sm_mhz"] == pytest.approx(1972.5) and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 2


def test_traffic_needs_current_kernel_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "profiles")
    src = tmp_path / "sparse_attention_block_nvfp4_gb300" / "csrc"
    os.makedirs(src)
    for rel in bench.KERNEL_SOURCES:
        (tmp_path / "sparse_attention_block_nvfp4_gb300" / rel).write_text("x")
    hp, hd = bench.kernel_hash("prefill"), bench.kernel_hash("decode")
    (tmp_path / "profiles" / "traffic.txt").write_text(
        f"prefill long_mixed {hp} 12345\nprefill long_mixed deadbeef 1\ndecode long_mixed {hd} 678\n")
    assert bench.recorded_traffic("prefill", "long_mixed") == 12345.0
    assert bench.recorded_traffic("decode", "long_mixed") == 678.0
    # a change to one kernel's own source voids only that kernel's record
    (tmp_path / "sparse_attention_block_nvfp4_gb300" / "csrc" / "prefill.cu").write_text("changed")
    assert bench.recorded_traffic("prefill", "long_mixed") is None
    assert bench.recorded_traffic("decode", "long_mixed") == 678.0
    # a shared header voids both
    (tmp_path / "sparse_attention_block_nvfp4_gb300" / "csrc" / "ptx.cuh").write_text("changed")
    assert bench.recorded_traffic("decode", "long_mixed") is None


def test_kernel_deps_cover_every_included_header():
    """Each timed kernel's hash covers its .cu and every header it includes
    (directly or through another header), so that a change to any of them
    voids the kernel's committed DRAM-traffic record."""
    import re
    base = os.path.join(bench.ROOT, "sparse_attention_block_nvfp4_gb300")

    def closure(rel):
        seen, todo = set(), [rel]
        while todo:
            r = todo.pop()
            if r in seen:
                continue
            seen.add(r)
            text = open(os.path.join(base, r)).read()
            for inc in re.findall(r'^\s*#\s*include\s+"([^"]+)"', text, re.M):
                todo.append(os.path.normpath(os.path.join(os.path.dirname(r), inc)))
        return seen

    for kernel, deps in bench.KERNEL_DEPS.items():
        assert deps[0].endswith(".cu"), kernel
        missing = closure(deps[0]) - set(deps)
        assert not missing, f"{kernel}: {sorted(missing)} not in its hashed sources"
