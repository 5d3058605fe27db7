"""One rank of the context-parallel checks (tests/test_cp.py).

Run as `python cp_worker.py RANK WORLD PORT MODE CASE`. Every rank draws the
same global problem from the case's seed, keeps its own token slice
(latent_query_split_gb300.cp.token_range) with the global shards clipped to it
(cp.local_offsets), runs cp_fwd and cp_bwd over a gloo process group and
compares its results with the fp64 oracle run on the whole, unsplit problem:
Z, L and dQ in full, Y, dK and dV on its own slice. MODE "oracle" runs the
local steps with oracle stand-ins on the CPU (the exchanges are what is
checked); MODE "gpu" runs them in the library on cuda:0, with the ranks'
partials staged through host memory by gloo. Prints one JSON line.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
sys.path.insert(0, ROOT)
sys.path.insert(0, HERE)

# B, H, M, N, D, dtype, global shard offsets, padding fraction, seed
CASES = {
    "small": (2, 2, 16, 301, 8, "f64", [0, 100, 100, 250, 301], 0.1, 11),
    "onepad": (1, 2, 8, 64, 8, "f64", [0, 64], 0.0, 12),     # rank 1's slice all padding
    "gpu_bf16": (2, 2, 128, 3001, 64, "bf16", [0, 700, 700, 2000, 3001], 0.05, 13),
    "gpu_f32": (1, 2, 16, 1000, 32, "f32", [0, 250, 500, 750, 1000], 0.05, 14),
    "gpu_m256": (1, 2, 256, 2600, 64, "bf16", [0, 1000, 2600], 0.05, 15),
}


class OracleOps:
    """The library's local steps written with the fp64 oracle (test stand-ins
    with the binding's signatures), so the exchanges run on a CPU host."""

    @staticmethod
    def _t(x, like):
        import torch
        return torch.from_numpy(x).to(like.device)

    @staticmethod
    def flare_encoder_fwd(Q, K, V, mask, off, **kw):
        import oracle
        Z, L = oracle.encode(Q, K, V, mask)
        return None, None, OracleOps._t(Z, K), OracleOps._t(L, K)

    @staticmethod
    def flare_lse_merge(O_r, L_r, Z=None, L=None, **kw):
        import oracle
        Z, L = oracle.lse_merge(O_r, L_r)
        return OracleOps._t(Z, O_r), OracleOps._t(L, O_r)

    @staticmethod
    def flare_decode_fwd(Q, Z, K, Y=None, **kw):
        import oracle
        return OracleOps._t(oracle.decode(Q, Z, K), K)

    @staticmethod
    def flare_decode_bwd(Q, Z, K, dY, **kw):
        import oracle
        return tuple(OracleOps._t(x, K) for x in oracle.decode_bwd(Q, Z, K, dY))

    @staticmethod
    def flare_encoder_bwd_accumulate(Q, K, V, mask, off, Z, L, dZ, dQ, dK, **kw):
        import oracle
        dQe, dKe, dV = oracle.encode_bwd(Q, K, V, mask, Z, L, dZ)
        return dQ + OracleOps._t(dQe, K), dK + OracleOps._t(dKe, K), OracleOps._t(dV, K)


def main():
    rank, world, port = (int(x) for x in sys.argv[1:4])
    mode, case = sys.argv[4], sys.argv[5]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    from latent_query_split_gb300 import cp

    def max_err(dev, ref):
        # (max |dev - ref| over finite reference entries, max |ref|), in fp64;
        # the -inf entries must coincide
        d = dev.detach().cpu().double().numpy()
        r = np.asarray(ref, dtype=np.float64)
        assert d.shape == r.shape and not np.isnan(d).any()
        assert np.array_equal(np.isneginf(d), np.isneginf(r))
        fin = ~np.isneginf(r)
        if not fin.any():
            return 0.0, 0.0
        return float(np.abs(d[fin] - r[fin]).max()), float(np.abs(r[fin]).max())

    B, H, M, N, D, dtype, off, pad, seed = CASES[case]
    g = torch.Generator().manual_seed(seed)
    dt = {"f64": torch.float64, "f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    Q = (torch.randn((H, M, D), generator=g) * 0.5).to(dt)
    K = torch.randn((B, N, H, D), generator=g).to(dt)
    V = torch.randn((B, N, H, D), generator=g).to(dt)
    dY = torch.randn((B, N, H, D), generator=g).to(dt)
    mask = (torch.rand((B, N), generator=g) > pad).to(torch.uint8)
    if case == "onepad":
        mask[:, N // 2:] = 0
    # the unsplit problem, in fp64
    Zo, Lo, Yo = oracle.flare_fwd(Q, K, V, mask)
    dQo, dKo, dVo = oracle.flare_bwd(Q, K, V, mask, Zo, Lo, dY)

    dist.init_process_group("gloo", rank=rank, world_size=world)
    ex = cp.Exchange()
    n0, n1 = cp.token_range(N, world, rank)
    loff = cp.local_offsets(off, n0, n1)
    dev = torch.device("cuda:0") if mode == "gpu" else torch.device("cpu")
    sl = lambda x: x[:, n0:n1].contiguous().to(dev)      # noqa: E731
    Qd, Kd, Vd, dYd, md = Q.to(dev), sl(K), sl(V), sl(dY), sl(mask)
    kw = {} if mode == "gpu" else {"ops": OracleOps}
    Y, Z, L = cp.cp_fwd(ex, Qd, Kd, Vd, md, loff, **kw)
    dQ, dK, dV = cp.cp_bwd(ex, Qd, Kd, Vd, md, loff, Z, L, dYd, **kw)
    if mode == "gpu":
        from latent_query_split_gb300 import flare
        flare.flare_device_status()
    # every rank holds the same global Z, L and dQ, bit for bit
    same = [bool(torch.equal(t.cpu(), ex.all_gather(t)[0].cpu())) for t in (Z, L, dQ)]
    res = {"rank": rank, "slice": [n0, n1], "local_offsets": loff, "same_on_ranks": same}
    for name, a, b in (("Z", Z, Zo), ("Y", Y, Yo[:, n0:n1]), ("dQ", dQ, dQo),
                       ("dK", dK, dKo[:, n0:n1]), ("dV", dV, dVo[:, n0:n1])):
        res[name] = max_err(a, b)
    res["L"] = max_err(L, Lo)
    dist.barrier()
    dist.destroy_process_group()
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
