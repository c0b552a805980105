"""Host logic of bench.py on CPU: the FLOP accounting (exact visible pairs)
against brute force, and the multi-process launch path (``--gpus N`` without
a torchrun environment) driven end to end with the CPU stand-in compute."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _brute(Lq, Lk, causal, window, n_sink):
    """Visible pairs by enumerating the mask the pages define: causal
    bottom-right (key j <= i + Lk - Lq), window of W keys ending at the
    diagonal, sink keys always visible where causal allows."""
    off = Lk - Lq
    n = 0
    for i in range(Lq):
        for j in range(Lk):
            vis = True
            if causal and j > i + off:
                vis = False
            if vis and window > 0 and not (j > i + off - window or j < n_sink):
                vis = False
            n += vis
    return n


@pytest.mark.parametrize("Lq,Lk,causal,window,n_sink", [
    (7, 7, False, 0, 0), (7, 7, True, 0, 0), (5, 9, True, 0, 0), (9, 5, True, 0, 0),
    (20, 20, True, 4, 0), (20, 20, True, 4, 1), (20, 20, True, 4, 3), (13, 30, True, 6, 2),
    (30, 13, True, 6, 2), (16, 16, True, 16, 1), (16, 16, True, 40, 5), (1, 1, True, 1, 1),
    (0, 5, True, 0, 0), (5, 0, True, 0, 0),
])
def test_visible_pairs_brute_force(Lq, Lk, causal, window, n_sink):
    assert bench.visible_pairs(Lq, Lk, causal, window, n_sink) == _brute(Lq, Lk, causal, window,
                                                                          n_sink)


def test_visible_pairs_closed_forms():
    S = 8192
    assert bench.visible_pairs(S, S, True) == S * (S + 1) // 2
    assert bench.visible_pairs(S, S, False) == S * S
    # window of W keys plus one sink key: rows past the window see W + 1 keys
    W = 1024
    expect = sum(min(i + 1, W) + (1 if i >= W else 0) for i in range(S))
    assert bench.visible_pairs(S, S, True, W, 1) == expect


def test_prefill_flop_convention():
    assert bench.prefill_flops(1, 16, 8192, 8192, 128, True) == 2.0 * 16 * 8192 * 8192 * 128
    assert bench.prefill_flops(4, 16, 2048, 2048, 128, False) == 4.0 * 4 * 16 * 2048 ** 2 * 128


def test_decode_kv_bytes():
    assert bench.decode_kv_bytes([1, 2, 3], 8, 128) == 6 * 8 * 128 * 4


def test_reread_model():
    # (Q + O) + (K + V) x ceil(Sq / 128): one head, S = 256 -> two query tiles
    assert bench.reread_model_bytes(1, 1, 1, 256, 256, 128) == 2 * 2 * 256 * 128 * (1 + 2)


@pytest.mark.parametrize("world", [2, 3])
def test_gpus_flag_launches_ranks(world):
    """`bench.py --gpus N` started without WORLD_SIZE re-launches itself with N
    ranks; rank 0 prints one line with n_gpus == N, the whole-job value
    formed from the slowest rank's time."""
    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", str(world),
                        "--stub", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=240, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["n_gpus"] == world and line["stub"]
    # the last rank sleeps longest: 3 steps x 2 ms x world at least
    assert line["rank_seconds_max"] >= 3 * 0.002 * world
    assert np.isclose(line["value"], world * 3 * 1.0e12 / line["rank_seconds_max"] / 1e12)


def test_single_rank_stub_runs_in_process():
    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--stub", "--steps", "2"],
                       capture_output=True, text=True, env=env, timeout=120, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][0])
    assert line["n_gpus"] == 1
