"""ZeRO-2 split of the gradient step across data-parallel ranks, one GPU each.

"Parallelisms" -- ZeRO-2: rank r owns the r-th 1/R shard of every bucket's
gradient, optimizer state and fp32 master weight.  "Parallelism Starts With
the Bottleneck" -- Allreduce equals reducescatter plus allgather: the
all-reduce of data parallelism becomes a reduce-scatter before the owner's
update and an all-gather of the updated parameters after it.

Per bucket b (padded size N_b, shard size n_b = N_b / R, offset off_b):

1. exchange -- rank r sends slice q of its bucket gradient,
   g[off_b + q*n_b : off_b + (q+1)*n_b], to rank q and receives slice r of
   every rank's bucket gradient (an all-to-all of bf16 slices, as point-to-
   point sends and receives).  The sum is NOT taken inside the collective:
   the received slices are summed by the owner in rank order 0..R-1 in fp32,
   so every rank gets the bits of the single-device step;
2. update -- dpg_reduce_scatter_adam on the shard plan (dpg_plan_shards),
   with the R received slice buffers in rank order as its replicas: fp32 sum,
   x fp32(1/G), Adam on the rank's master/m/v shard, bf16 cast into the
   rank's parameter shard;
3. all-gather -- every rank's bf16 shard of bucket b into the bucket's slice
   of every rank's full parameter buffer.

G, the global valid-token count, needs every rank's counts: they are
all-gathered first.  Steps 1-3 run per bucket range, so a caller can start a
bucket's exchange as soon as the backward has produced it.

With K microbatches per step ("Distributed Training and Parallelism" -- Data
parallelism and the global gradient: accumulate locally, reduce once), each
rank first adds all K microbatches into its fp32 buffer (dpg_accumulate, the
first with first=True) and the exchange carries fp32 slices
(grad_dtype=torch.float32).  The owner's rank-ordered sum of those slices is
the single-device accumulation path's: there too each replica's accumulator
and its last microbatch are added in binary32 before the rank-ordered sum.

Every collective here is a torch.distributed call on the caller's process
group (NCCL for CUDA tensors, gloo for CPU tensors); no kernel of the library
ever reads another GPU's memory.  The local update is the library's CUDA
entry point; a caller may pass its own update function (same arguments) to
run the same exchange elsewhere.
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence

import numpy as np

from . import (HParams, Plan, dpg_plan_shards, dpg_reduce_scatter_adam)


class ShardedStep:
    """Buffers and collectives of one rank's part of the ZeRO-2 split.

    plan: the global bucket plan (R = world size).  The rank's own buffers:
      recv[s]      bf16 (fp32 with grad_dtype=torch.float32), shard-plan
                   layout: slices of this rank's shard received from rank s
                   (padding zero);
      param_shard  bf16, shard-plan layout: this rank's updated parameters.
    The fp32 master/m/v shards (shard-plan layout, shard.total_padded
    elements each) belong to the caller.
    """

    def __init__(self, plan: Plan, rank: int, world: int, device, group=None,
                 update_fn: Optional[Callable] = None, grad_dtype=None):
        import torch
        grad_dtype = torch.bfloat16 if grad_dtype is None else grad_dtype
        if grad_dtype not in (torch.bfloat16, torch.float32):
            raise ValueError(f"gradients are exchanged as bf16 or fp32, not {grad_dtype}")
        if plan.R != world:
            raise ValueError(f"the plan's R ({plan.R}) must equal the world size ({world})")
        if not 0 <= rank < world:
            raise ValueError(f"rank {rank} outside [0, {world})")
        self.plan, self.rank, self.world, self.group = plan, rank, world, group
        self.device = device
        self.shard = dpg_plan_shards(plan)
        self.off = [int(x) for x in plan.bucket_offset]
        self.n = [int(x) for x in plan.shard_numel]
        self.soff = [int(x) for x in self.shard.bucket_offset]
        S = self.shard.total_padded
        self.recv = [torch.zeros(S, dtype=grad_dtype, device=device) for _ in range(world)]
        self.param_shard = torch.zeros(S, dtype=torch.bfloat16, device=device)
        self.update_fn = update_fn or dpg_reduce_scatter_adam

    # -- layout ------------------------------------------------------------
    def global_slice(self, b: int, q: int):
        """Elements [lo, hi) of bucket b's shard q in the global flat layout."""
        lo = self.off[b] + q * self.n[b]
        return lo, lo + self.n[b]

    def shard_slice(self, b: int):
        """Elements [lo, hi) of bucket b's shard in the shard-plan layout."""
        return self.soff[b], self.soff[b] + self.n[b]

    def state_from_global(self, full):
        """This rank's shard (shard-plan layout) of a global flat fp32 array:
        for initialising master weights from a replicated copy."""
        import torch
        out = torch.zeros(self.shard.total_padded, dtype=full.dtype, device=full.device)
        for b in range(self.plan.n_buckets):
            lo, hi = self.global_slice(b, self.rank)
            a, z = self.shard_slice(b)
            out[a:z].copy_(full[lo:hi])
        return out

    # -- collectives ---------------------------------------------------------
    def all_tokens(self, local_counts) -> np.ndarray:
        """Every rank's valid-token counts (K per rank), replica-major: the
        R*K counts that G sums ("Distributed Training and Parallelism" -- Data
        parallelism and the global gradient: normalise by the global count)."""
        import torch
        import torch.distributed as dist
        mine = torch.as_tensor(np.asarray(local_counts, np.int64).reshape(-1))
        if self.device is not None and torch.device(self.device).type == "cuda":
            mine = mine.to(self.device)
        out = torch.empty(self.world * mine.numel(), dtype=torch.int64, device=mine.device)
        dist.all_gather_into_tensor(out, mine, group=self.group)
        return out.cpu().numpy()

    def bucket_groups(self, n_groups: int):
        """[b0, b1) ranges of about equal padded size, in bucket order."""
        n_groups = max(1, min(int(n_groups), self.plan.n_buckets))
        ends = np.cumsum(self.plan.bucket_padded)
        total = int(ends[-1]) if len(ends) else 0
        cuts = [0]
        for g in range(1, n_groups):
            b = int(np.searchsorted(ends, total * g / n_groups)) + 1
            if cuts[-1] < b < self.plan.n_buckets:
                cuts.append(b)
        cuts.append(self.plan.n_buckets)
        return list(zip(cuts[:-1], cuts[1:]))

    def exchange(self, grad_flat, b0: int = 0, b1: Optional[int] = None, wait: bool = True):
        """Step 1 for buckets [b0, b1): slice q of this rank's bucket gradient
        to rank q; slice `rank` of every rank's into recv[src].  wait=False
        returns the pending works instead of waiting for them."""
        import torch.distributed as dist
        if grad_flat.dtype != self.recv[0].dtype:
            raise ValueError(f"gradient buffer is {grad_flat.dtype}, the exchange carries "
                             f"{self.recv[0].dtype}")
        b1 = self.plan.n_buckets if b1 is None else b1
        ops = []
        for b in range(b0, b1):
            a, z = self.shard_slice(b)
            for q in range(self.world):
                lo, hi = self.global_slice(b, q)
                if q == self.rank:
                    self.recv[q][a:z].copy_(grad_flat[lo:hi])
                    continue
                ops.append(dist.P2POp(dist.isend, grad_flat[lo:hi], q, group=self.group))
                ops.append(dist.P2POp(dist.irecv, self.recv[q][a:z], q, group=self.group))
        works = dist.batch_isend_irecv(ops) if ops else []
        if not wait:
            return works
        for w in works:
            w.wait()
        return []

    def update(self, tokens, hp: HParams, master, exp_avg, exp_avg_sq, *, bucket_sqnorm=None,
               bucket_nonfinite=None, b0: int = 0, b1: Optional[int] = None, stream=None):
        """Step 2 for buckets [b0, b1): the fused update of this rank's shard
        from the received slices (norms: this rank's shard of each bucket)."""
        b1 = self.plan.n_buckets if b1 is None else b1
        self.update_fn(self.shard, self.recv, tokens, hp, master, exp_avg, exp_avg_sq,
                       [self.param_shard], bucket_sqnorm=bucket_sqnorm,
                       bucket_nonfinite=bucket_nonfinite, b0=b0, b1=b1, stream=stream)

    def allgather(self, param_flat, b0: int = 0, b1: Optional[int] = None, wait: bool = True):
        """Step 3 for buckets [b0, b1): every rank's bf16 shard of bucket b
        into param_flat's bucket slice (shard q at slice q).  wait=False
        returns the pending works instead of waiting for them."""
        import torch.distributed as dist
        b1 = self.plan.n_buckets if b1 is None else b1
        works = []
        for b in range(b0, b1):
            a, z = self.shard_slice(b)
            lo, hi = self.off[b], self.off[b] + self.world * self.n[b]
            w = dist.all_gather_into_tensor(param_flat[lo:hi], self.param_shard[a:z],
                                            group=self.group, async_op=not wait)
            if w is not None:
                works.append(w)
        return works

    def step(self, grad_flat, local_counts, hp: HParams, master, exp_avg, exp_avg_sq,
             param_flat, *, bucket_sqnorm=None, bucket_nonfinite=None, stream=None,
             groups: int = 1):
        """The whole split step over every bucket: tokens, exchange, update,
        all-gather.  With groups > 1 the buckets are cut into that many ranges
        and pipelined ("Distributed Training and Parallelism" -- Hide
        communication): the exchange of range g + 1 is in flight while range
        g is updated, and range g's all-gather while range g + 1 is; the
        results are the same bits."""
        tokens = self.all_tokens(local_counts)
        kw = dict(bucket_sqnorm=bucket_sqnorm, bucket_nonfinite=bucket_nonfinite, stream=stream)
        if groups <= 1:
            self.exchange(grad_flat)
            self.update(tokens, hp, master, exp_avg, exp_avg_sq, **kw)
            self.allgather(param_flat)
            return tokens
        cuts = self.bucket_groups(groups)
        pending = self.exchange(grad_flat, *cuts[0], wait=False)
        gathers = []
        for g, (b0, b1) in enumerate(cuts):
            nxt = (self.exchange(grad_flat, *cuts[g + 1], wait=False)
                   if g + 1 < len(cuts) else [])
            for w in pending:
                w.wait()
            self.update(tokens, hp, master, exp_avg, exp_avg_sq, b0=b0, b1=b1, **kw)
            gathers += self.allgather(param_flat, b0, b1, wait=False)
            pending = nxt
        for w in gathers:
            w.wait()
        return tokens


def loopback_receive(step: ShardedStep, grads: Sequence, b0: int = 0, b1: Optional[int] = None):
    """Fill step.recv as the exchange would, from every rank's gradient
    buffer held in one process (grads[s] = rank s's flat gradient): the same
    slices, copied locally.  For checking one rank's update on one device."""
    b1 = step.plan.n_buckets if b1 is None else b1
    for b in range(b0, b1):
        a, z = step.shard_slice(b)
        lo, hi = step.global_slice(b, step.rank)
        for s in range(step.world):
            step.recv[s][a:z].copy_(grads[s][lo:hi])
