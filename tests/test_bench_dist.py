"""Host logic of `bench.py --gpus N`: with N > 1 every rank runs an independent
replica, the timed value is the slowest rank's time, and the reported
throughput is the work of all ranks over that time.  Checked with two gloo
ranks on the CPU (no GPU involved)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, local, w = bench.dist_setup()
    try:
        mine = 10.0 + 5.0 * r                     # rank 1 is the slow one
        slowest = bench.max_over_ranks(mine, w)
        bench.barrier(w)
        gbs = bench.whole_job_gbs(1e9, steps=2, world=w, max_ms=slowest)
        q.put((r, local, w, slowest, gbs))
    finally:
        import torch.distributed as dist
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[2] == 2 for r in res)
    assert all(r[3] == pytest.approx(15.0) for r in res)
    # 2 ranks x 2 steps x 1 GB over 15 ms
    assert all(r[4] == pytest.approx(2 * 2 * 1.0 / 0.015) for r in res)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.dist_setup() == (0, 0, 1)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_byte_model_matches_the_per_element_totals():
    import bench
    c = bench.code_bytes_per_elem(4)
    assert c == 0.53125
    P, n = 4, 1 << 20
    assert bench.call_model_bytes(P, n, 4, True, False) == pytest.approx(P * n * (12 + 2 * c))
    assert bench.call_model_bytes(P, n, 4, False, False) == pytest.approx(P * n * (4 + 2 * c))
    assert bench.call_model_bytes(P, n, 8, True, False) == pytest.approx(P * n * (12 + 2 * 1.03125))
    # the fused gather skips one read of the gather codes
    assert bench.call_model_bytes(P, n, 4, True, True) == pytest.approx(P * n * (12 + 2 * c) - n * c)
    # a bf16 state moves 4 B per element instead of 8 (13.06 -> 9.06 B at 4-bit)
    assert bench.call_model_bytes(P, n, 4, True, False, 2) == pytest.approx(P * n * (8 + 2 * c))
    assert (bench.call_model_bytes(P, n, 4, True, False) -
            bench.call_model_bytes(P, n, 4, True, False, 2)) == pytest.approx(4 * P * n)


def test_profiled_traffic_belongs_to_one_configuration(tmp_path, monkeypatch):
    """A DRAM-traffic figure from ncu is reported only for the configuration it
    was captured on, and only while the kernel sources are unchanged; a capture
    of a smaller case of that configuration is scaled by the element ratio."""
    import json
    import bench
    (tmp_path / "profiles").mkdir()
    f32 = bench.traffic_key("p4_2048x4096", 4, 128, "f32", 0, "fused")
    bf16 = bench.traffic_key("p4_2048x4096", 4, 128, "bf16", 0, "fused")
    big = bench.traffic_key("p8_1gib", 4, 128, "f32", 0, "fused")
    rec = {f32: {"push_kernel": {"dram_bytes_per_launch": 100, "source_hash": "h1"}},
           bf16: {"push_kernel": {"dram_bytes_per_launch": 60, "source_hash": "h1"}},
           big: {"push_kernel": {"dram_bytes_per_launch": 1000, "source_hash": "h1",
                                 "captured_elements": 8 * 2048 * 4096, "capture": "x.md"}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel="": "h1")
    n2 = 4 * 2048 * 4096
    assert bench.profiled_traffic("push_kernel", f32, n2) == (100, None)
    assert bench.profiled_traffic("push_kernel", bf16, n2) == (60, None)
    assert bench.profiled_traffic("reduce_kernel", f32, n2) == (None, None)
    scaled, note = bench.profiled_traffic("push_kernel", big, 8 * 131072 * 4096)
    assert scaled == 64 * 1000 and "scaled by 64" in note
    assert bench.profiled_traffic("push_kernel", big, 8 * 2048 * 4096) == (1000, None)
    for other in (bench.traffic_key("p4_2048x4096", 8, 128, "f32", 0, "fused"),
                  bench.traffic_key("p4_2048x4096", 4, 64, "f32", 0, "fused"),
                  bench.traffic_key("p4_2048x4096", 4, 128, "f32", 1, "fused"),
                  bench.traffic_key("p4_2048x4096", 4, 128, "f32", 0, "unfused"),
                  bench.traffic_key("p4_8192x4096", 4, 128, "f32", 0, "fused")):
        assert bench.profiled_traffic("push_kernel", other, n2) == (None, None)
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel="": "h2")   # sources changed
    assert bench.profiled_traffic("push_kernel", f32, n2) == (None, None)


def test_also_specs_and_host_cpu_info():
    import bench
    assert bench.parse_also("4", 4) == (4, 4)
    assert bench.parse_also("3b8", 4) == (3, 8)
    info = bench.host_cpu_info()
    assert info["nproc"] >= 1 and isinstance(info["cpu_model"], str)
    assert bench.shape_of(3) == ("p8_1gib", 8, 512 * 2 ** 20)
    assert bench.shape_of(3, 2048) == ("p8_1gib@2048x4096", 8, 2048 * 4096)


def test_oracle_sample_threads_give_the_single_thread_result():
    """Splitting the sampled positions over threads changes nothing but the time:
    same state and the same tie count as one thread."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor
    import bench

    class A:
        workload, bits, g, quantizer, state, decay, tokens = 1, 4, 128, 0, "f32", 1.0, 0
    one, many = bench.oracle_sample(A()), bench.oracle_sample(A())
    with ThreadPoolExecutor(3) as pool:
        for _ in range(3):
            one.step()
            many.step(pool, 3)
    assert one.e.keys() == many.e.keys() == {"fwd"}
    assert np.array_equal(one.e["fwd"].view(np.uint32), many.e["fwd"].view(np.uint32))
    assert one.ties == many.ties


def test_uncompensated_runs_and_oracle_sample_states():
    """--uncompensated turns every call of the sequence into one without state;
    the oracle sample then holds no state, and in a mixed sequence (the P=2
    workload: one uncompensated call, then compensated ones) it leaves the
    state untouched on the uncompensated call and keeps the forward and
    backward states apart (the P=4, 32768x1024 workload)."""
    import numpy as np
    import bench

    class A:
        workload, bits, g, quantizer, state, decay, tokens, calls = 1, 4, 128, 0, "f32", 1.0, 0, 0
        uncompensated, fused, tile, persistent, graph = False, True, True, False, False
    a = A()
    mixed = bench.workload_sequence(a)
    assert [c.state for c in mixed] == ["none"] + ["fwd"] * 8
    assert bench.state_key(a) == "f32"
    s = bench.oracle_sample(a, seq=mixed)
    s.step()                                   # the uncompensated call
    assert not s.e["fwd"].any()
    s.step()
    assert s.e["fwd"].any()
    a.uncompensated = True
    none = bench.workload_sequence(a)
    assert [c.state for c in none] == ["none"] * 9 and bench.state_key(a) == "none"
    s = bench.oracle_sample(a, seq=none)
    assert s.e == {}
    s.step()
    s.step()
    cfg = bench.workload_config(a, 1, none)
    assert cfg["compensated"] is False and cfg["state"] == {"format": "none"}
    a.uncompensated, a.calls = False, 3
    assert len(bench.workload_sequence(a)) == 3
    assert len(bench.workload_sequence(a, 2)) == 64   # another workload: all of its calls
    a.workload, a.calls = 5, 0
    seq5 = bench.workload_sequence(a)
    assert {c.state for c in seq5} == {"fwd", "bwd"}


def test_reference_arm_reports_the_gpu_arms_config():
    """`--impl reference` times the oracle on the host cores for the GPU arm's
    workload and options, and reports the same config dict, with its sample
    described beside it, so the two lines pair up."""
    import bench
    from bit_error_compensated_gb300.workloads import call_sequence
    args = bench.main.__globals__["argparse"].Namespace(
        workload=1, bits=4, g=128, quantizer=0, state="f32", decay=1.0, tokens=0, calls=0,
        fused=True, persistent=False, tile=False, graph=False, steps=2, warmup=1)
    line = bench.run_reference(args, 0, 1)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"] == bench.workload_config(args, 1, call_sequence(1, steps=1))
    assert "sample" in line and line["sample"] == line["cpu_baseline"]["sample"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == cb["nproc"] >= 1 and cb["cpu_model"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_kernel_source_hash_follows_code_not_comments(tmp_path, monkeypatch):
    """A committed ncu figure stays valid through comment-only edits and edits
    to other kernels, and is dropped by any change to its kernel's code."""
    import shutil
    import bench
    csrc = tmp_path / "bit_error_compensated_gb300" / "csrc"
    shutil.copytree(os.path.join(bench.ROOT, "bit_error_compensated_gb300", "csrc"), csrc)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    push0, reduce0 = bench.kernel_source_hash("push_kernel"), bench.kernel_source_hash("reduce_kernel")
    f = csrc / "k_push.cu"
    f.write_text(f.read_text() + "\n// a comment\n/* and a block\n comment */\n")
    assert bench.kernel_source_hash("push_kernel") == push0
    f.write_text(f.read_text() + "\nnamespace echo { constexpr int kUnused = 1; }\n")
    assert bench.kernel_source_hash("push_kernel") != push0
    assert bench.kernel_source_hash("reduce_kernel") == reduce0
    q = csrc / "quant.cuh"
    q.write_text(q.read_text() + "\nnamespace echo { constexpr int kAlsoUnused = 2; }\n")
    assert bench.kernel_source_hash("reduce_kernel") != reduce0


def test_first_calls_parity_compares_the_sampled_outputs():
    """The bench's check of the timed configuration's first calls against the
    oracle on the sampled positions, driven here by a stand-in for the GPU
    call that runs the oracle's whole call on the CPU: no mismatch, over two
    calls that carry the state; then a stand-in that changes one output bit
    at a sampled position is caught."""
    import numpy as np
    import torch
    import bench
    import oracle
    from bit_error_compensated_gb300.workloads import call_sequence, rank_inputs

    class A:
        workload, bits, g, quantizer, state, decay, tokens = 2, 4, 128, 0, "f32", 1.0, 8
    seq = call_sequence(2)[:3]
    P, n = 4, 8 * 4096
    xs = torch.stack([rank_inputs(2, c, "cpu", tokens=8) for c in seq])
    out = torch.empty((P, n), dtype=torch.bfloat16)

    def calls(flip=None):
        e = np.zeros((P, n), np.float32)
        made = []

        def make(k):
            def call(stream):
                x = xs[k].view(torch.int16).numpy().view(np.uint16)
                y = oracle.allreduce(x, 128, 4, e=e)["out"].copy()
                if flip is not None and len(made) == 1:       # the second call
                    y[:, flip] ^= 1
                out.view(torch.int16).copy_(torch.from_numpy(y.view(np.int16)))
                made.append(k)
            return call
        return [make(k) for k in range(len(seq))]

    r = bench.first_calls_parity(A(), xs, seq, calls(), out, None)
    assert r["calls"] == 2 and r["output_mismatches"] == 0
    assert r["outputs_compared"] == 2 * P * r["sampled_groups"] * 128
    s = bench.oracle_sample(A(), xs, seq)
    sampled = int(s.idx_t[5])
    r = bench.first_calls_parity(A(), xs, seq, calls(flip=sampled), out, None)
    assert r["output_mismatches"] == P
