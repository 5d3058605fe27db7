"""Context-parallel FLARE (latent_query_split_gb300.cp) over two ranks.

The appendix on context parallelism splits the tokens over ranks: each rank
computes its partial (O_r, L_r), the ranks merge them by the cross-rank
log-sum-exp rule, the decode is local; in the backward the gradient of the
replicated Z and the query gradient are summed over the ranks. Two gloo
ranks run cp_fwd and cp_bwd on slices of one problem and every result is
compared with the fp64 oracle on the unsplit problem.

The CPU tests run the exchanges with oracle stand-ins for the library's
local steps; the GPU tests run the library itself, both ranks on cuda:0
(their kernels never wait on each other: the exchange goes through host
memory).
"""
import json
import os
import socket
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from latent_query_split_gb300 import cp  # noqa: E402
from parity import ATOL, L_ATOL, REL  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(mode, case, world=2):
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, os.path.join(HERE, "cp_worker.py"), str(r),
                               str(world), str(port), mode, case],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(world)]
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=300)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        assert p.returncode == 0, err[-3000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    return sorted(outs, key=lambda o: o["rank"])


def _check(outs, atol, rel):
    for o in outs:
        assert o["same_on_ranks"] == [True, True, True], o
        for name in ("Z", "Y", "dQ", "dK", "dV"):
            err, scale = o[name]
            assert err <= atol and err <= rel * scale + 1e-30, (o["rank"], name, err, scale)
        assert o["L"][0] <= L_ATOL, (o["rank"], o["L"])


def test_token_range_covers_once():
    for N, W in ((301, 2), (5, 4), (3, 4), (0, 2), (1 << 20, 8)):
        ranges = [cp.token_range(N, W, r) for r in range(W)]
        assert ranges[0][0] == 0 and ranges[-1][1] == N
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
        lens = [e - s for s, e in ranges]
        assert max(lens) - min(lens) <= 1


def test_local_offsets_clip_global_shards():
    off = [0, 100, 100, 250, 301]
    assert cp.local_offsets(off, 0, 151) == [0, 100, 100, 151, 151]
    assert cp.local_offsets(off, 151, 301) == [0, 0, 0, 99, 150]
    # the ranks' pieces of every shard add up to the shard
    for W in (2, 3, 4):
        pieces = [cp.local_offsets(off, *cp.token_range(301, W, r)) for r in range(W)]
        for s in range(4):
            assert sum(p[s + 1] - p[s] for p in pieces) == off[s + 1] - off[s]
    with pytest.raises(ValueError):
        cp.local_offsets([0, 5, 3], 0, 3)


@pytest.mark.parametrize("case", ["small", "onepad"])
def test_two_rank_exchanges_match_unsplit_oracle(case):
    outs = _run("oracle", case)
    assert outs[0]["slice"][1] == outs[1]["slice"][0]
    _check(outs, atol=1e-10, rel=1e-10)


@pytest.mark.gpu
@pytest.mark.parametrize("case,dtype", [("gpu_bf16", "bf16"), ("gpu_f32", "f32"),
                                        ("gpu_m256", "bf16")])
def test_two_rank_library_matches_unsplit_oracle(cuda_device, case, dtype):
    _check(_run("gpu", case), ATOL[dtype], REL[dtype])
