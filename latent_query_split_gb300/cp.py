"""Context-parallel FLARE mixer across the ranks of a torch.distributed group.

Follows the appendix on context parallelism of "FLARE++: Low-rank attention
with dynamic attention routing": every rank holds one contiguous slice of the
tokens (its own shards of K, V, the mask and the output gradient) and a
replica of the latent queries. The forward runs the local primitive on the
rank's tokens, which returns the rank's normalised partial output O_r and row
log-normaliser L_r; the ranks exchange those partials (their size does not
depend on N) and every rank merges them by the cross-rank log-sum-exp rule of
eq. 23, so every rank holds the same global (Z, L); the decode is local. The
backward paragraphs give the exchanges of the backward: the gradient of the
replicated Z is summed over the ranks before the encoder backward, which
then runs locally with the global Z and L, and the query gradient is summed
over the ranks at the end.

The page's exchange is an all-reduce max of L_r followed by two all-reduce
sums; here it is one all-gather of (O_r, L_r) followed by the library's merge
kernel on every rank, which computes the same rule in a fixed rank order (so
every rank gets bit-identical Z and L).

Every arithmetic step runs in the library's kernels (the `flare` binding);
this module only moves tensors between ranks with torch.distributed. Over
the gloo backend device tensors are staged through host memory.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import torch
import torch.distributed as dist

from . import flare


def token_range(N: int, world: int, rank: int) -> Tuple[int, int]:
    """Token slice [start, end) of rank `rank` when N tokens are split into
    `world` contiguous slices whose lengths differ by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    base, rem = divmod(N, world)
    start = rank * base + min(rank, rem)
    return start, start + base + (1 if rank < rem else 0)


def local_offsets(shard_offsets: Sequence[int], start: int, end: int) -> List[int]:
    """Offsets, relative to `start`, of the global shards clipped to the token
    slice [start, end): one entry per global shard (shards outside the slice
    become empty), so shard r of every rank is a piece of global shard r."""
    off = [int(x) for x in shard_offsets]
    if off[0] != 0 or any(b < a for a, b in zip(off, off[1:])):
        raise ValueError("shard offsets must start at 0 and not decrease")
    if not 0 <= start <= end <= off[-1]:
        raise ValueError(f"slice [{start}, {end}) outside [0, {off[-1]})")
    return [min(max(x, start), end) - start for x in off]


class Exchange:
    """The collectives of the context-parallel path over one process group.

    all_gather stacks every rank's tensor in rank order; all_reduce_sum_
    replaces a tensor by its sum over the ranks. With the gloo backend a
    device tensor goes through host memory (gloo moves host buffers); with
    NCCL it stays on the device."""

    def __init__(self, group=None):
        if not dist.is_initialized():
            raise RuntimeError("torch.distributed is not initialised")
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.host_staging = dist.get_backend(group) == "gloo"

    def _out(self, t: torch.Tensor) -> torch.Tensor:
        return t.cpu() if (self.host_staging and t.is_cuda) else t

    def all_gather(self, t: torch.Tensor) -> torch.Tensor:
        """[world, *t.shape] on t's device, rank r's tensor at index r."""
        src = self._out(t.contiguous())
        parts = [torch.empty_like(src) for _ in range(self.world)]
        dist.all_gather(parts, src, group=self.group)
        return torch.stack(parts).to(t.device)

    def all_reduce_sum_(self, t: torch.Tensor) -> torch.Tensor:
        """In place: t <- sum over the ranks of t."""
        buf = self._out(t)
        dist.all_reduce(buf, op=dist.ReduceOp.SUM, group=self.group)
        if buf is not t:
            t.copy_(buf)
        return t


def cp_fwd(ex: Exchange, Q, K, V, mask=None, shard_offsets=None, *, Y=None, Z=None, L=None,
           workspace=None, kernel: str = "auto", stream=None, ops=flare):
    """FLARE forward of one rank: K, V [B, N_rank, H, D] (and mask
    [B, N_rank]) are this rank's token slice, shard_offsets its local shard
    offsets; Q is replicated. Returns (Y [B, N_rank, H, D], Z, L), Z and L
    global and identical on every rank (written into Y, Z, L when given).
    The collectives run on torch's current stream: pass stream=None, or make
    `stream` current around the call.

    `ops` names the module whose functions run the local steps: the compiled
    library binding, which is the only implementation; a test on a host
    without a GPU passes stand-ins with the same signatures to check the
    exchanges."""
    N = K.shape[1]
    off = [0, N] if shard_offsets is None else list(shard_offsets)
    # the local primitive: this rank's (O_r, L_r), all of its shards merged
    _, _, Z_r, L_r = ops.flare_encoder_fwd(Q, K, V, mask, off, workspace=workspace,
                                           kernel=kernel, stream=stream)
    # cross-rank log-sum-exp merge (eq. 23): exchange the partials, merge in rank order
    Z, L = ops.flare_lse_merge(ex.all_gather(Z_r), ex.all_gather(L_r), Z=Z, L=L, stream=stream)
    Y = ops.flare_decode_fwd(Q, Z, K, Y=Y, kernel=kernel, stream=stream)
    return Y, Z, L


def cp_bwd(ex: Exchange, Q, K, V, mask, shard_offsets, Z, L, dY, *, workspace=None,
           kernel: str = "auto", stream=None, ops=flare):
    """FLARE mixer backward of one rank from the global (Z, L) of cp_fwd and
    this rank's output gradient dY [B, N_rank, H, D]. Returns (dQ, dK, dV):
    dQ [B, H, M, D] summed over every rank's tokens (identical on every
    rank), dK, dV this rank's token gradients. Streams and `ops` as for
    cp_fwd."""
    N = K.shape[1]
    off = [0, N] if shard_offsets is None else list(shard_offsets)
    # the decode's shares of dQ and dK, and this rank's contribution to dZ
    dQ, dZ, dK = ops.flare_decode_bwd(Q, Z, K, dY, workspace=workspace, kernel=kernel,
                                      stream=stream)
    # Z is replicated: its gradient is the sum over the ranks' decodes
    ex.all_reduce_sum_(dZ)
    # the encoder with the global (Z, L, dZ) adds its local shares of dQ, dK
    dQ, dK, dV = ops.flare_encoder_bwd_accumulate(Q, K, V, mask, off, Z, L, dZ, dQ, dK,
                                                  workspace=workspace, kernel=kernel,
                                                  stream=stream)
    # Q is replicated: its gradient is summed over the ranks
    ex.all_reduce_sum_(dQ)
    return dQ, dK, dV
