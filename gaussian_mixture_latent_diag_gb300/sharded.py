"""One head's sequence sharded over N across ranks (torch.distributed).

Rank r of a process group holds a contiguous block of the sequence positions
of every (b, h) it serves, in rank order.  GMA needs one small exchange per
head to stitch the shards together ("Gaussian Mixture Attention: Linear-Time
Sequence Mixing via Probabilistic Latent Routing", arXiv 2606.18283):

* bidirectional -- the latent memory (Eqs. (5)-(6)) is a sum over positions, so
  the memories of the key/value shards add up to the memory of the whole
  sequence; every rank then reads that total with its own queries (Eq. (7));
* causal -- the prefix memories of Eq. (8b) at a shard boundary are the sum of
  the memories of all earlier shards, so rank r continues from the exclusive
  prefix (over ranks 0..r-1) of the shard memories.

The exchange is one all_gather of each rank's [B, H, K, d_v + 1] memory
(16.6 KB per head at K = d_v = 64) followed by a sum in rank order, so every
rank computes bitwise the same total whatever the collective's internal
reduction order.  All arithmetic -- the per-shard steps and the rank-order sum
-- runs in libgma.so's kernels (``CudaOps``); this module only moves tensors.
The orchestration takes any object with the same four methods, which is how
its host logic is tested on CPU ranks.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


class CudaOps:
    """The per-shard steps in libgma.so's kernels: on the tensor cores wherever
    the memory calls have tensor-core kernels (bf16, d_r in {32, 64}, d_v = 64,
    K <= 64: the sizes of the 64-wide family, where the unsharded forward runs
    on the tensor cores too, so a sharded call has the unsharded call's
    accuracy), else on the CUDA cores.  The 128-wide tensor-core kernels serve
    only the whole-sequence forwards, so their sizes shard on the CUDA cores."""

    @staticmethod
    def _path(X, V, mu, causal=0):
        import ctypes
        from . import PATH_SIMT, PATH_TC, _native
        code = _native.GMA_BF16 if X.dtype == torch.bfloat16 else _native.GMA_F32
        N, d_r = X.shape[-2:]
        # the library's own answer: the memory calls' workspace query with
        # GMA_PATH_TC is 0 where they have no tensor-core kernels
        opt = _native.options(path=PATH_TC)
        nb = _native.load().gma_latent_memory_workspace_size(1, 1, max(N, 1), d_r, V.shape[-1], mu.shape[1], code,
                                                             ctypes.byref(opt))
        return PATH_TC if nb > 0 else PATH_SIMT

    def latent_memory(self, K, V, mu, sigma2, log_pi):
        from . import latent_memory
        return latent_memory(K, V, mu, sigma2, log_pi, path=self._path(K, V, mu))

    def read_memory(self, Q, mu, sigma2, log_pi, Vt, Z, eps):
        from . import read_memory
        return read_memory(Q, mu, sigma2, log_pi, Vt, Z, eps=eps, path=self._path(Q, Vt, mu))

    def forward_causal_carry(self, Q, K, V, mu, sigma2, log_pi, Vt_in, Z_in, eps):
        from . import forward_causal_carry
        return forward_causal_carry(Q, K, V, mu, sigma2, log_pi, Vt_in, Z_in, eps=eps, want_state=False,
                                    path=self._path(Q, V, mu, causal=1))[0]

    def combine(self, packed, count):
        """Rows 0..count-1 of a [P, n] packed array summed in row order (gma_combine_memories)."""
        from . import combine_memories
        return combine_memories(packed, count)


def pack_memories(parts):
    """[P, n] array of the shards' memories, row r = [Vt_r | Z_r] flattened (a copy)."""
    return torch.stack([torch.cat([vt.reshape(-1), z.reshape(-1)]) for vt, z in parts])


def combine_total(parts, ops=None):
    """Sum of the (Vt, Z) memories of every shard, in shard order (ops.combine)."""
    ops = ops or CudaOps()
    Vt0, Z0 = parts[0]
    flat = ops.combine(pack_memories(parts), len(parts))
    n = Vt0.numel()
    return flat[:n].view_as(Vt0), flat[n:].view_as(Z0)


def combine_exclusive(parts, rank: int, ops=None):
    """Sum of the memories of shards 0..rank-1 in shard order; (None, None) for
    rank 0 (an empty prefix)."""
    if rank == 0:
        return None, None
    return combine_total(parts[:rank], ops)


def gather_memories(Vt, Z, group=None):
    """all_gather of every rank's (Vt, Z), returned in rank order."""
    world = dist.get_world_size(group)
    packed = torch.cat([Vt.reshape(-1), Z.reshape(-1)])
    bufs = [torch.empty_like(packed) for _ in range(world)]
    dist.all_gather(bufs, packed, group=group)
    n = Vt.numel()
    return [(b[:n].view_as(Vt), b[n:].view_as(Z)) for b in bufs]


def forward_bidir_sharded(Q, K, V, mu, sigma2, log_pi, eps=1e-6, group=None, ops=None):
    """Bidirectional GMA of a sequence sharded over N: this rank's Q, K, V
    [B, H, n_r, d] are its block of positions; returns its block of O."""
    ops = ops or CudaOps()
    Vt, Z = ops.latent_memory(K, V, mu, sigma2, log_pi)
    Vt, Z = combine_total(gather_memories(Vt, Z, group), ops)
    return ops.read_memory(Q, mu, sigma2, log_pi, Vt, Z, eps)


def forward_causal_sharded(Q, K, V, mu, sigma2, log_pi, eps=1e-6, group=None, ops=None):
    """Causal GMA of a sequence sharded over N (rank r holds the r-th block of
    positions): continues from the memories of all earlier ranks' blocks."""
    ops = ops or CudaOps()
    Vt, Z = ops.latent_memory(K, V, mu, sigma2, log_pi)
    carry_v, carry_z = combine_exclusive(gather_memories(Vt, Z, group), dist.get_rank(group), ops)
    return ops.forward_causal_carry(Q, K, V, mu, sigma2, log_pi, carry_v, carry_z, eps)
