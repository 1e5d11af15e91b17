"""Host-side logic of bench.py that needs no GPU: the max-over-ranks timing
reduction of the replica mode (world size 2, gloo), the clock-sample parser
and the oracle slice sizing."""
import os
import socket
import time

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    q.put((rank, bench.max_over_ranks(1.5 + rank, world)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_clock_sampler_parses_nvidia_smi_lines():
    s = bench.ClockSampler(0)
    now = time.monotonic()
    s.lines = [
        # idle, before the timed region began: left out of the summary
        (now - 5.0, "0, 1980, 2070, 180.0, 0x0, Not Active, Not Active, "
                    "Not Active, Not Active"),
        (now - 1.0, "0, 1650, 2070, 1361.2, 0x4, Not Active, Not Active, "
                    "Not Active, Active"),
        (now - 0.9, "0, 1605, 2070, 1370.0, 0x4, Not Active, Not Active, "
                    "Not Active, Active"),
        (now - 0.8, "garbage"),
    ]
    s.t0 = now - 2.0

    class FinishedProcess:  # stand-in for the nvidia-smi child process
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s.proc = FinishedProcess()
    out = s.stop()
    assert out["sm_mhz"] == pytest.approx(1627.5)
    assert out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 2


def test_oracle_slice_is_bounded():
    from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
    for name, w in W.WORKLOADS.items():
        n = bench.oracle_tokens(w)
        assert 16 <= n <= max(16, w.tokens)
        assert (12 if w.backward else 4) * n * w.hidden * w.ffn <= 1.6e12


def test_attention_reference_arm_runs_the_oracle_on_cpu():
    """bench.py --impl reference on an attention workload: the fp64 oracle
    on a bounded one-sequence sample, same metric, a valid JSON line."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"),
                        "--impl", "reference", "--workload", "attn_tiny_d64",
                        "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s"
    assert line["metric"].startswith("TP-attention")
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


class _FakeEvent:
    """A CUDA event stand-in: record() reads a scripted clock (ms)."""
    clock = []

    def __init__(self, enable_timing=True):
        self.t = None

    def record(self, stream=None):
        self.t = _FakeEvent.clock.pop(0)

    def elapsed_time(self, other):
        return other.t - self.t


class _FakeTorch:
    class cuda:
        Event = _FakeEvent

        @staticmethod
        def synchronize():
            pass


def test_timed_steps_reports_mean_and_per_step_stats():
    # events at 0, 2, 5, 6, 10 ms: steps of 2, 3, 1, 4 ms
    _FakeEvent.clock = [0.0, 2.0, 5.0, 6.0, 10.0]
    calls = []
    ms, st = bench.timed_steps(_FakeTorch, None, lambda: calls.append(1), 4)
    assert len(calls) == 4
    assert ms == 2.5
    assert st == {"median": 2.5, "min": 1.0, "max": 4.0}


def test_oracle_one_core_runs_in_a_single_threaded_child():
    from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
    r = bench.oracle_one_core(W.WORKLOADS["tiny_fp32"], 16)
    assert "error" not in r, r
    assert r["threads"] == 1 and r["value"] > 0
    assert r["sample"].startswith("first 16 of 32 tokens")


def test_l2_flush_only_where_the_weights_fit_in_l2():
    import torch
    # GPT-3-13B MLP weights (A and B in bf16) exceed L2: no flush, no
    # allocation
    assert bench.l2_flusher(torch, 4 * 5120 * 20480) is None
    assert "no flush" in bench.l2_note(None)
    assert "flushed" in bench.l2_note(lambda: None)
    # GPT-2-medium's do not (a flush would be made on the device)
    assert 4 * 1024 * 4096 < bench.L2_BYTES


def test_roofline_peak_is_burst_for_short_regions():
    # a 20-step region of the GPT-3-13B step lasts ~0.12 s: burst peak
    # whatever its clock samples show; a region of a second or more is held
    # to the sustained figure
    assert bench._kernel_peak(0.12, 1885.6, 1707.6) == (1885.6, "burst")
    assert bench._kernel_peak(bench.SUSTAINED_REGION_S, 1885.6, 1707.6) == \
        (1707.6, "sustained")
