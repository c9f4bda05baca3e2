"""Host logic of bench.py: the max-over-ranks timing reduction across two
gloo processes (the N > 1 replicas path, on CPU) and the algorithmic-byte
accounting the roofline uses."""

import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        q.put((rank, bench.max_over_ranks(1.5 + rank, ws)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 2.5, 1: 2.5}


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_algorithmic_bytes():
    w = workloads.WORKLOADS["sample_b64_g4_v128256_bf16_s0.7"]
    n = np.array([4] * 10 + [1] * 54)
    ab = bench.algorithmic_bytes(w, n)
    assert ab["stream"] == 64 * 5 * 128256 * 2 + 64 * 4 * 6
    assert ab["final"] == 54 * 128256 * 6 + 10 * 128256 * 2
    g = workloads.WORKLOADS["greedy_b512_g4_v128256_bf16"]
    assert bench.algorithmic_bytes(g, np.zeros(512, int)) == {"stream": 512 * 5 * 128256 * 2, "final": 0}
    t = workloads.WORKLOADS["topk50_topp0.9_b256_g8_v152064_bf16"]
    assert bench.algorithmic_bytes(t, np.zeros(256, int))["final"] == 0
    # q as bf16 draft logits: the draft rows once more, q elements at 2 bytes
    ql = workloads.WORKLOADS["sample_qlogits_b64_g4_v128256_bf16"]
    ab = bench.algorithmic_bytes(ql, n)
    assert ab["stream"] == 64 * 5 * 128256 * 2 + 64 * 4 * (2 + 2) + 64 * 4 * 128256 * 2
    assert ab["final"] == 54 * 128256 * (2 + 2) + 10 * 128256 * 2
    # deterministic drafts read no q
    dt = workloads.WORKLOADS["sample_det_b64_g4_v128256_bf16"]
    ab = bench.algorithmic_bytes(dt, n)
    assert ab["stream"] == 64 * 5 * 128256 * 2 + 64 * 4 * 2
    assert ab["final"] == 64 * 128256 * 2


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_reference_arm_fields(name):
    """The reference arm's JSON line (oracle on host cores) for a tiny run."""
    import json
    import subprocess

    if workloads.WORKLOADS[name].B * workloads.WORKLOADS[name].V > 10 ** 6:
        pytest.skip("large workload: input generation is slow on CPU")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", name,
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == name


def test_kept_counts_match_the_oracle_keep_set():
    """The bench's count of kept candidates (torch) equals the size of the
    oracle's top-k then top-p keep set, row by row."""
    from oracle import svref
    import torch

    g = torch.Generator().manual_seed(5)
    rows = (torch.randn(12, 3000, generator=g) * 2).to(torch.bfloat16)
    for k, tp in [(50, 0.9), (0, 0.5), (7, 1.0), (3000, 0.99)]:
        got = bench.kept_counts(rows, 0.8, k, tp).numpy()
        want = [len(svref.truncation_keep_set(r, 0.8, k, tp)[0]) for r in rows.float().numpy()]
        assert list(got) == want, (k, tp)


def test_algorithmic_bytes_counts_kept_q_reads():
    t = workloads.WORKLOADS["topk50_topp0.9_b256_g8_v152064_bf16"]
    base = bench.algorithmic_bytes(t, np.zeros(256, int))["stream"]
    assert bench.algorithmic_bytes(t, np.zeros(256, int), kept_rejected=1000)["stream"] == base + 4000
    # top-p alone: row n's logits again, q at the kept tokens of rejected rows
    tp = workloads.WORKLOADS["topp0.9_b64_g4_v128256_bf16"]
    ab = bench.algorithmic_bytes(tp, np.zeros(64, int), kept_rejected=1000)
    assert ab["stream"] == 64 * 5 * 128256 * 2 + 64 * 4 * 6
    assert ab["final"] == 64 * 128256 * 2 + 4000


def test_q_bytes_read_in_place():
    """q bytes the kernels read when q stays in host memory (the e2e arm):
    q(d_i) at every tested position, then row n's kept candidates
    (truncated) or the whole row n (untruncated) of each rejected sequence."""
    import torch

    w = workloads.WORKLOADS["sample_b64_g4_v128256_bf16_s0.7"]
    n = np.array([4] * 10 + [1] * 54)
    assert bench.q_bytes_read(w, n, {}, 0) == (64 * 4 + 54 * 128256) * 4
    t = workloads.WORKLOADS["topk50_topp0.9_b256_g8_v152064_bf16"]
    assert bench.q_bytes_read(t, np.zeros(256, int), {}, 1000) == (256 * 8 + 1000) * 4
    for name in ("greedy_b512_g4_v128256_bf16", "sample_det_b64_g4_v128256_bf16", "sample_qlogits_b64_g4_v128256_bf16"):
        assert bench.q_bytes_read(workloads.WORKLOADS[name], n, {}, 0) == 0
    r = workloads.WORKLOADS["sample_ragged_b64_g8_v128256_bf16"]
    gb = torch.tensor([8] * 32 + [2] * 32, dtype=torch.int32)
    nr = np.array([8] * 32 + [0] * 32)
    assert bench.q_bytes_read(r, nr, {"gamma_b": gb}, 0) == (32 * 8 + 32 * 2 + 32 * 128256) * 4
